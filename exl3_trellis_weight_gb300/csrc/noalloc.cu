// noalloc.cu -- exl3_encode_tiles_noalloc: the trellis encode for callers that
// cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: plug-ins that run inside a host
// application which owns every byte of device memory through its own pool, and
// latency-critical loops where an allocation (which can synchronise the whole
// device) is not acceptable.  They cannot provide the encoder's workspace either
// if they have no pool of their own to carve it from.  For them the decision
// rows of the encoder live in one file-scope device array instead.
//
// The array holds the decision rows of up to kNoAllocMaxBlocks persistent encode
// blocks (3 MiB each, 24 MiB in total).  It is created when the library's code
// is loaded on a device and stays allocated on every device that loads the
// library until the process exits.  Its host-side name is only a stand-in: the
// device address is looked up with cudaGetSymbolAddress once per device (again
// after that device's context was destroyed and re-created).
#include <mutex>

#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kNoAllocMaxBlocks = EXL3_NOALLOC_MAX_BLOCKS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_noalloc_scratch[(size_t)kNoAllocMaxBlocks *
                                                            kEncodeBlockScratchBytes /
                                                            sizeof(uint32_t)];

std::mutex g_mu;

// Per device: the context the address was looked up in, and the address.  A
// device's primary context is destroyed by cudaDeviceReset and the array's
// address in the next context may differ, so the cache is keyed by the
// driver's unique context id (0 = not looked up yet).
struct ScratchSlot {
    unsigned long long ctx_id;
    uint32_t *addr;
};
ScratchSlot g_slot[kMaxDevices] = {};

typedef int (*PFN_ctx_get_current)(void **ctx);                   // cuCtxGetCurrent
typedef int (*PFN_ctx_get_id)(void *ctx, unsigned long long *id);  // cuCtxGetId

// The current context's unique id through the driver entry points the runtime
// hands out (no link against libcuda); 0 when there is no current context yet.
exl3_status current_context_id(unsigned long long *id) {
    static PFN_ctx_get_current get_current = nullptr;
    static PFN_ctx_get_id get_id = nullptr;
    if (!get_current || !get_id) {
        void *p1 = nullptr, *p2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 4000,
                                                          cudaEnableDefault, &q1);
        cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000,
                                                          cudaEnableDefault, &q2);
        if (e1 != cudaSuccess || e2 != cudaSuccess || q1 != cudaDriverEntryPointSuccess ||
            q2 != cudaDriverEntryPointSuccess || !p1 || !p2)
            return set_error(EXL3_ERR_CUDA, "driver entry points cuCtxGetCurrent/cuCtxGetId "
                                            "are not available");
        get_current = reinterpret_cast<PFN_ctx_get_current>(p1);
        get_id = reinterpret_cast<PFN_ctx_get_id>(p2);
    }
    void *ctx = nullptr;
    if (get_current(&ctx) != 0)
        return set_error(EXL3_ERR_CUDA, "cuCtxGetCurrent failed");
    *id = 0;
    if (ctx && get_id(ctx, id) != 0)
        return set_error(EXL3_ERR_CUDA, "cuCtxGetId failed");
    return EXL3_OK;
}

// Device address of the scratch array for the current device (set-up on the
// first call per device and context).
exl3_status scratch_address(uint32_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(EXL3_ERR_UNSUPPORTED, "device index %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_mu);
    unsigned long long ctx = 0;
    exl3_status st = current_context_id(&ctx);
    if (st != EXL3_OK)
        return st;
    if (ctx == 0 || g_slot[dev].ctx_id != ctx || !g_slot[dev].addr) {
        void *p = nullptr;
        // also makes the device's primary context current when none was yet
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_check(e, "cudaGetSymbolAddress(noalloc scratch)");
        st = current_context_id(&ctx);
        if (st != EXL3_OK)
            return st;
        g_slot[dev].ctx_id = ctx;
        g_slot[dev].addr = static_cast<uint32_t *>(p);
    }
    *out = g_slot[dev].addr;
    return EXL3_OK;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" EXL3_API exl3_status exl3_encode_tiles_noalloc(const float *Y, int64_t rows,
                                                          int64_t cols, int K, float scale,
                                                          uint16_t *codes, float *tile_cost,
                                                          int blocks, void *stream) {
    if (!Y || !codes)
        return set_error(EXL3_ERR_INVALID_ARG, "Y and codes must not be NULL");
    if (((uintptr_t)Y % 4) || ((uintptr_t)codes % 4) || ((uintptr_t)tile_cost % 4))
        return set_error(EXL3_ERR_INVALID_ARG, "Y, codes and tile_cost must be 4-byte aligned");
    if (rows <= 0 || cols <= 0)
        return set_error(EXL3_ERR_INVALID_ARG, "rows and cols must be positive");
    if (rows % 16 || cols % 16)
        return set_error(EXL3_ERR_UNSUPPORTED, "rows=%lld cols=%lld must be multiples of 16",
                         (long long)rows, (long long)cols);
    if (rows > (1ll << 24) || cols > (1ll << 24) || rows * cols > (1ll << 34))
        return set_error(EXL3_ERR_INVALID_ARG, "matrix %lldx%lld is too large", (long long)rows,
                         (long long)cols);
    if (K < 1 || K > 4)
        return set_error(EXL3_ERR_UNSUPPORTED, "K=%d is not built (K in {1,2,3,4})", K);
    if (!(scale > 0.0f) || !(scale < __builtin_inff()) || !(1.0f / scale < __builtin_inff()))
        return set_error(EXL3_ERR_INVALID_ARG, "scale and 1 / scale must be positive and finite");
    if (blocks < 0 || blocks > kNoAllocMaxBlocks)
        return set_error(EXL3_ERR_WORKSPACE,
                         "blocks=%d exceeds the static scratch: at most %d blocks (%zu bytes each)",
                         blocks, kNoAllocMaxBlocks, kEncodeBlockScratchBytes);
    uint32_t *scratch = nullptr;
    exl3_status st = scratch_address(&scratch);
    if (st != EXL3_OK)
        return st;
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    int64_t grid = blocks == 0 ? kNoAllocMaxBlocks : blocks;
    if (grid > n_tiles)
        grid = n_tiles;
    EncodeLaunch el{};
    el.Y = Y;
    el.rows = rows;
    el.cols = cols;
    el.K = K;
    el.T = 256;
    el.row_tiles = 0;
    el.inv_scale = 1.0f / scale;
    el.inv_scale_dev = nullptr;
    el.codes = reinterpret_cast<uint32_t *>(codes);
    el.tile_cost = tile_cost;
    el.scratch = scratch;   // every decision row is written before it is read
    el.grid = (int)grid;
    return launch_encode_unprofiled(el, (cudaStream_t)stream);
}
