"""exl3_encode_tiles_noalloc through the C ABI (gpu).

This entry point is for callers that must not allocate device memory, such as
plug-ins inside an application that owns all device memory through its own
pool, or latency-critical loops that cannot afford an allocation.  It keeps the
encoder's decision rows in a static device array of the library instead of a
caller workspace.  Its codes and tile costs must equal those of
exl3_encode_tiles and of the CPU oracle bit for bit, on consecutive calls that
reuse the same static array.  The file is named so that pytest collects it
last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exl3_trellis_weight_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_BLOCKS = 8   # EXL3_NOALLOC_MAX_BLOCKS in include/exl3.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for -m gpu tests")
    import __graft_entry__
    __graft_entry__.build()
    import exl3_trellis_weight_gb300 as ex
    L = ex.lib()
    L.exl3_encode_tiles_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    L.exl3_encode_tiles_noalloc.restype = ctypes.c_int
    return ex, L


def _noalloc(L, Y, K, scale, blocks):
    rows, cols = Y.shape
    codes = torch.empty(rows // 16, cols // 16, 16 * K, dtype=torch.int16, device=Y.device)
    cost = torch.empty((rows // 16) * (cols // 16), dtype=torch.float32, device=Y.device)
    st = L.exl3_encode_tiles_noalloc(ctypes.c_void_p(Y.data_ptr()), rows, cols, K,
                                     ctypes.c_float(scale), ctypes.c_void_p(codes.data_ptr()),
                                     ctypes.c_void_p(cost.data_ptr()), blocks,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.exl3_last_error()
    return codes, cost


def test_noalloc_matches_workspace_encode_on_consecutive_calls(lib):
    ex, L = lib
    dev = torch.device("cuda:0")
    cases = [  # (rows, cols, K, scale, blocks, seed): second call reuses the static rows
        (128, 256, 2, 1.0, 0, 1),
        (96, 160, 4, 0.8, 3, 2),
        (64, 96, 1, 1.1, 5, 3),
        (48, 112, 3, 0.9, 0, 4),
    ]
    for rows, cols, K, scale, blocks, seed in cases:
        Yc = inputs.iid_f32(rows, cols, seed)
        Y = Yc.to(dev)
        codes_n, cost_n = _noalloc(L, Y, K, scale, blocks)
        codes_w, cost_w = ex.encode_tiles(Y, K, scale, want_cost=True)
        torch.cuda.synchronize()
        assert torch.equal(codes_n, codes_w)
        assert np.array_equal(cost_n.cpu().numpy().view(np.uint32),
                              cost_w.cpu().numpy().view(np.uint32))
        # and against the oracle: targets fl(Y * fl32(1 / scale))
        inv = float(np.float32(1.0) / np.float32(scale))
        st, costs_o = oracle.encode_matrix(Yc.numpy(), K, inv)
        codes_o = np.stack([oracle.pack(s, K) for s in st])
        assert np.array_equal(codes_n.cpu().numpy().view(np.uint16).reshape(-1, 16 * K), codes_o)
        assert np.array_equal(cost_n.cpu().numpy().view(np.uint32), costs_o.view(np.uint32))


def test_noalloc_rejects_more_blocks_than_the_static_array_holds(lib):
    _, L = lib
    Y = torch.zeros(16, 16, device="cuda:0")
    codes = torch.empty(1, 1, 32, dtype=torch.int16, device="cuda:0")
    st = L.exl3_encode_tiles_noalloc(ctypes.c_void_p(Y.data_ptr()), 16, 16, 2, ctypes.c_float(1.0),
                                     ctypes.c_void_p(codes.data_ptr()), None, MAX_BLOCKS + 1, None)
    assert st == 3   # EXL3_ERR_WORKSPACE
    assert b"at most" in L.exl3_last_error()


def test_noalloc_rejects_an_unbuilt_k(lib):
    """K outside {1, 2, 3, 4} returns EXL3_ERR_UNSUPPORTED and enqueues nothing."""
    _, L = lib
    Y = torch.zeros(16, 16, device="cuda:0")
    codes = torch.full((1, 1, 80), 7, dtype=torch.int16, device="cuda:0")
    st = L.exl3_encode_tiles_noalloc(ctypes.c_void_p(Y.data_ptr()), 16, 16, 5, ctypes.c_float(1.0),
                                     ctypes.c_void_p(codes.data_ptr()), None, 0, None)
    assert st == 2   # EXL3_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((codes == 7).all())
