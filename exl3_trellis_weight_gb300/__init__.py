"""EXL3 trellis tile encoder for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libexl3.so`` (``include/exl3.h``).
Functions take torch CUDA tensors, check shapes and dtypes, and pass raw
device pointers plus the current CUDA stream to the library; every step of
the computation runs in the library's kernels.  There is no CPU fallback: if
the shared library is missing or CUDA is unavailable, the calls raise.

Entry points (same names as the C ABI, without the ``exl3_`` prefix):
  rotate, encode_tiles, decode_tiles, mse, quantize, gss_scale
plus the workspace queries.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "Exl3Error", "lib", "lib_path", "rotate", "encode_tiles", "decode_tiles", "mse",
    "encode_rows", "decode_rows",
    "quantize", "gss_scale", "scale_search", "scale_search_workspace_bytes", "encode_workspace_bytes", "encode_workspace_min_bytes",
    "quantize_workspace_bytes", "gss_workspace_bytes", "mse_workspace_bytes",
    "supports_k", "rotate_last_kernel", "profile_enable", "profile_read", "wait_timeouts", "EXL3_F32", "EXL3_BF16",
]

EXL3_F32 = 0
EXL3_BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libexl3.so")
_lock = threading.Lock()
_lib = None


class Exl3Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libexl3.so (built by ``exl3_trellis_weight_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise Exl3Error(-1, f"libexl3.so not built at {_LIB_PATH}; run "
                                "python -c 'import __graft_entry__ as g; g.build()'")
        L = ctypes.CDLL(_LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        f32, f64, sz = ctypes.c_float, ctypes.c_double, ctypes.c_size_t
        L.exl3_status_str.argtypes = [i32]
        L.exl3_status_str.restype = ctypes.c_char_p
        L.exl3_last_error.restype = ctypes.c_char_p
        L.exl3_version.restype = i32
        L.exl3_supports_k.argtypes = [i32]
        L.exl3_supports_k.restype = i32
        L.exl3_rotate.argtypes = [P, i32, i64, i64, P, P, i32, P, P]
        L.exl3_encode_workspace_bytes.argtypes = [i64, i32]
        L.exl3_encode_workspace_bytes.restype = sz
        L.exl3_encode_workspace_min_bytes.argtypes = [i32]
        L.exl3_encode_workspace_min_bytes.restype = sz
        L.exl3_encode_tiles.argtypes = [P, i64, i64, i32, f32, P, P, P, sz, P]
        L.exl3_decode_tiles.argtypes = [P, i64, i64, i32, f32, P, P]
        L.exl3_encode_rows.argtypes = [P, i64, i32, i32, f32, P, P, P, sz, P]
        L.exl3_decode_rows.argtypes = [P, i64, i32, i32, f32, P, P]
        L.exl3_mse_workspace_bytes.argtypes = [i64, i64]
        L.exl3_mse_workspace_bytes.restype = sz
        L.exl3_mse.argtypes = [P, i32, P, i64, i64, P, P, sz, P]
        L.exl3_quantize_workspace_bytes.argtypes = [i64, i64, i32]
        L.exl3_quantize_workspace_bytes.restype = sz
        L.exl3_quantize.argtypes = [P, i32, i64, i64, P, P, i32, f64, P, P, P, P, P, P, sz, P]
        L.exl3_gss_workspace_bytes.argtypes = [i64, i64, i32]
        L.exl3_gss_workspace_bytes.restype = sz
        L.exl3_gss_scale.argtypes = [P, i32, i64, i64, P, P, i32, f64, f64, i32,
                                     P, P, P, P, P, P, sz, P]
        L.exl3_scale_search_workspace_bytes.argtypes = [i64, i64, i32]
        L.exl3_scale_search_workspace_bytes.restype = sz
        L.exl3_scale_search.argtypes = [P, i32, i64, i64, P, P, i32, P, P, P, P, sz, P]
        L.exl3_block_ldl_workspace_bytes.argtypes = [i64]
        L.exl3_block_ldl_workspace_bytes.restype = sz
        L.exl3_block_ldl.argtypes = [P, i64, f64, i32, P, P, P, sz, P]
        L.exl3_ldlq_workspace_bytes.argtypes = [i64, i64, i32]
        L.exl3_ldlq_workspace_bytes.restype = sz
        L.exl3_ldlq.argtypes = [P, i64, i64, P, i32, f32, P, P, P, sz, P]
        L.exl3_regularize_workspace_bytes.argtypes = [i64, i64]
        L.exl3_regularize_workspace_bytes.restype = sz
        L.exl3_regularize.argtypes = [P, i32, i64, i64, P, P, i32, P, P, P, P, sz, P]
        L.exl3_profile_enable.argtypes = [i32]
        L.exl3_profile_enable.restype = None
        L.exl3_profile_read.argtypes = [P, P, P]
        L.exl3_wait_timeouts.argtypes = [P]
        L.exl3_rotate_last_kernel.argtypes = []
        L.exl3_rotate_last_kernel.restype = i32
        for name in ("exl3_regularize", "exl3_block_ldl", "exl3_ldlq", "exl3_scale_search", "exl3_encode_rows", "exl3_decode_rows", "exl3_profile_read", "exl3_wait_timeouts", "exl3_rotate", "exl3_encode_tiles", "exl3_decode_tiles", "exl3_mse",
                     "exl3_quantize", "exl3_gss_scale"):
            getattr(L, name).restype = i32
        _lib = L
        return L


def _check(status: int):
    if status != 0:
        L = lib()
        raise Exl3Error(status, f"{L.exl3_status_str(status).decode()}: "
                                f"{L.exl3_last_error().decode()}")


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (no CPU fallback)")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return EXL3_F32
    if t.dtype == torch.bfloat16:
        return EXL3_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _workspace(nbytes: int, device, ws=None):
    """A caller-supplied workspace is passed through as is: the library accepts
    anything from its per-call minimum up (fewer encode blocks when smaller)
    and returns EXL3_ERR_WORKSPACE below that."""
    torch = _torch()
    if ws is not None:
        _need_cuda(ws)
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def profile_enable(on: bool = True) -> None:
    """exl3_profile_enable: bracket each encode launch with CUDA events, count launches."""
    lib().exl3_profile_enable(int(bool(on)))


def profile_read():
    """exl3_profile_read -> (encode_ms_total, encode_launches, kernel_launches); waits
    for the recorded events and clears them."""
    ms = ctypes.c_double(0.0)
    ne = ctypes.c_int64(0)
    nk = ctypes.c_int64(0)
    _check(lib().exl3_profile_read(ctypes.byref(ms), ctypes.byref(ne), ctypes.byref(nk)))
    return ms.value, ne.value, nk.value


def wait_timeouts() -> int:
    """exl3_wait_timeouts -> number of bounded device waits that expired since
    the last call (the TMA forward rotation's waits on its tile loads);
    synchronises the device and resets the count.  A nonzero count means the
    launches concerned produced void results."""
    n = ctypes.c_uint(0)
    st = lib().exl3_wait_timeouts(ctypes.byref(n))
    if st not in (0, 5):
        _check(st)
    return int(n.value)


def rotate_last_kernel() -> int:
    """exl3_rotate_last_kernel: 1 TMA forward, 2 shared-memory forward, 3 warp-shuffle
    kernel, 0 none -- the kernel the calling thread's last rotation launched."""
    return int(lib().exl3_rotate_last_kernel())


def supports_k(K: int) -> bool:
    return bool(lib().exl3_supports_k(K))


def encode_workspace_bytes(n_tiles: int, K: int) -> int:
    return int(lib().exl3_encode_workspace_bytes(n_tiles, K))


def encode_workspace_min_bytes(K: int) -> int:
    return int(lib().exl3_encode_workspace_min_bytes(K))


def quantize_workspace_bytes(rows: int, cols: int, K: int) -> int:
    return int(lib().exl3_quantize_workspace_bytes(rows, cols, K))


def gss_workspace_bytes(rows: int, cols: int, K: int) -> int:
    return int(lib().exl3_gss_workspace_bytes(rows, cols, K))


def mse_workspace_bytes(rows: int, cols: int) -> int:
    return int(lib().exl3_mse_workspace_bytes(rows, cols))


def rotate(W, su, sv, inverse: bool = False, out=None):
    """exl3_rotate: blockwise randomized Hadamard rotation -> fp32 [rows, cols]."""
    torch = _torch()
    _need_cuda(W, su, sv, out)
    rows, cols = W.shape
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.float32, device=W.device)
    _check(lib().exl3_rotate(_ptr(W), _dt(W), rows, cols, _ptr(su), _ptr(sv), int(bool(inverse)),
                             _ptr(out), _stream(W.device)))
    return out


def encode_tiles(Y, K: int, scale: float = 1.0, codes=None, tile_cost=None,
                 want_cost: bool = False, ws=None):
    """exl3_encode_tiles -> codes uint16 [rows/16, cols/16, 16K] (and per-tile cost)."""
    torch = _torch()
    _need_cuda(Y, codes, tile_cost)
    rows, cols = Y.shape
    n = (rows // 16) * (cols // 16)
    if codes is None:
        codes = torch.empty(rows // 16, cols // 16, 16 * K, dtype=torch.int16, device=Y.device)
    if want_cost and tile_cost is None:
        tile_cost = torch.empty(n, dtype=torch.float32, device=Y.device)
    ws = _workspace(encode_workspace_bytes(n, K), Y.device, ws)
    _check(lib().exl3_encode_tiles(_ptr(Y), rows, cols, K, ctypes.c_float(scale), _ptr(codes),
                                   _ptr(tile_cost), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(Y.device)))
    return (codes, tile_cost) if want_cost or tile_cost is not None else codes


def encode_rows(Y, K: int, scale: float = 1.0, codes=None, row_cost=None,
                want_cost: bool = False, ws=None):
    """exl3_encode_rows: each row of Y[n_rows, T] is one tile -> codes uint16 [n_rows, T*K/16]."""
    torch = _torch()
    _need_cuda(Y, codes, row_cost)
    n_rows, T = Y.shape
    if codes is None:
        codes = torch.empty(n_rows, T * K // 16, dtype=torch.int16, device=Y.device)
    if want_cost and row_cost is None:
        row_cost = torch.empty(n_rows, dtype=torch.float32, device=Y.device)
    ws = _workspace(encode_workspace_bytes(n_rows, K), Y.device, ws)
    _check(lib().exl3_encode_rows(_ptr(Y), n_rows, T, K, ctypes.c_float(scale), _ptr(codes),
                                  _ptr(row_cost), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(Y.device)))
    return (codes, row_cost) if want_cost or row_cost is not None else codes


def decode_rows(codes, n_rows: int, T: int, K: int, scale: float = 1.0, out=None):
    """exl3_decode_rows -> fp32 [n_rows, T]."""
    torch = _torch()
    _need_cuda(codes, out)
    if out is None:
        out = torch.empty(n_rows, T, dtype=torch.float32, device=codes.device)
    _check(lib().exl3_decode_rows(_ptr(codes), n_rows, T, K, ctypes.c_float(scale), _ptr(out),
                                  _stream(codes.device)))
    return out


def decode_tiles(codes, rows: int, cols: int, K: int, scale: float = 1.0, out=None):
    """exl3_decode_tiles -> fp32 [rows, cols] = v(state) * scale."""
    torch = _torch()
    _need_cuda(codes, out)
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.float32, device=codes.device)
    _check(lib().exl3_decode_tiles(_ptr(codes), rows, cols, K, ctypes.c_float(scale), _ptr(out),
                                   _stream(codes.device)))
    return out


def mse(W, What, out=None, ws=None):
    """exl3_mse -> device fp64 scalar tensor (fixed-order reduction)."""
    torch = _torch()
    _need_cuda(W, What, out)
    rows, cols = W.shape
    if out is None:
        out = torch.empty((), dtype=torch.float64, device=W.device)
    ws = _workspace(mse_workspace_bytes(rows, cols), W.device, ws)
    _check(lib().exl3_mse(_ptr(W), _dt(W), _ptr(What), rows, cols, _ptr(out), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(W.device)))
    return out


def quantize(W, su, sv, K: int, g: float = 1.0, codes=None, want_What: bool = False, ws=None):
    """exl3_quantize: one full rotate/encode/decode/inverse/MSE pass at relative scale g.

    Returns dict(codes, scale (device f32), mse (device f64), sigma (device f64), What|None).
    """
    torch = _torch()
    _need_cuda(W, su, sv, codes)
    rows, cols = W.shape
    dev = W.device
    if codes is None:
        codes = torch.empty(rows // 16, cols // 16, 16 * K, dtype=torch.int16, device=dev)
    scale = torch.empty((), dtype=torch.float32, device=dev)
    m = torch.empty((), dtype=torch.float64, device=dev)
    sigma = torch.empty((), dtype=torch.float64, device=dev)
    What = torch.empty(rows, cols, dtype=torch.float32, device=dev) if want_What else None
    ws = _workspace(quantize_workspace_bytes(rows, cols, K), dev, ws)
    _check(lib().exl3_quantize(_ptr(W), _dt(W), rows, cols, _ptr(su), _ptr(sv), K,
                               ctypes.c_double(g), _ptr(codes), _ptr(scale), _ptr(m), _ptr(sigma),
                               _ptr(What), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(dev)))
    return dict(codes=codes, scale=scale, mse=m, sigma=sigma, What=What)


def scale_search_workspace_bytes(rows: int, cols: int, K: int) -> int:
    return int(lib().exl3_scale_search_workspace_bytes(rows, cols, K))


def scale_search(W, su, sv, K: int, want_history: bool = True, ws=None):
    """exl3_scale_search: grid + parabola search for the relative scale on a tile
    sample.  Returns dict(g, scale, history) as device tensors (history [27, 2])."""
    torch = _torch()
    _need_cuda(W, su, sv)
    rows, cols = W.shape
    dev = W.device
    g = torch.empty((), dtype=torch.float64, device=dev)
    scale = torch.empty((), dtype=torch.float32, device=dev)
    hist = torch.empty(54, dtype=torch.float64, device=dev) if want_history else None
    ws = _workspace(scale_search_workspace_bytes(rows, cols, K), dev, ws)
    _check(lib().exl3_scale_search(_ptr(W), _dt(W), rows, cols, _ptr(su), _ptr(sv), K, _ptr(g),
                                   _ptr(scale), _ptr(hist), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(dev)))
    return dict(g=g, scale=scale, history=None if hist is None else hist.view(27, 2))


def block_ldl_workspace_bytes(n: int) -> int:
    return int(lib().exl3_block_ldl_workspace_bytes(n))


def block_ldl(H, sigma_reg: float = 0.01, max_retries: int = 10, M=None, ws=None):
    """exl3_block_ldl: M = L blockdiag(L_bb)^-1 (strictly lower block part, fp32)
    of the damped Cholesky factor of H (fp64 [n, n]).  Returns (M, retries);
    raises Exl3Error (EXL3_ERR_NUMERIC) when every damping attempt fails."""
    torch = _torch()
    _need_cuda(H, M)
    if H.dtype != torch.float64:
        raise ValueError("H must be float64")
    n = H.shape[0]
    if M is None:
        M = torch.empty(n, n, dtype=torch.float32, device=H.device)
    ws = _workspace(block_ldl_workspace_bytes(n), H.device, ws)
    retries = ctypes.c_int(-1)
    _check(lib().exl3_block_ldl(_ptr(H), n, ctypes.c_double(sigma_reg), int(max_retries), _ptr(M),
                                ctypes.byref(retries), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(H.device)))
    return M, retries.value


def ldlq_workspace_bytes(rows: int, cols: int, K: int) -> int:
    return int(lib().exl3_ldlq_workspace_bytes(rows, cols, K))


def ldlq(R, M, K: int, scale: float, want_q: bool = True, codes=None, ws=None):
    """exl3_ldlq: span-by-span trellis coding of R (fp32 [rows, cols], input
    channels down the rows) with error feedback through M.  Returns
    dict(codes [rows/16, cols/16, 16K] int16, Q fp32 [rows, cols] | None)."""
    torch = _torch()
    _need_cuda(R, M, codes)
    rows, cols = R.shape
    dev = R.device
    if codes is None:
        codes = torch.empty(rows // 16, cols // 16, 16 * K, dtype=torch.int16, device=dev)
    Q = torch.empty(rows, cols, dtype=torch.float32, device=dev) if want_q else None
    ws = _workspace(ldlq_workspace_bytes(rows, cols, K), dev, ws)
    _check(lib().exl3_ldlq(_ptr(R), rows, cols, _ptr(M), K, ctypes.c_float(scale), _ptr(codes),
                           _ptr(Q), _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return dict(codes=codes, Q=Q)


def regularize_workspace_bytes(rows: int, cols: int) -> int:
    return int(lib().exl3_regularize_workspace_bytes(rows, cols))


def regularize(W, h, sv, apply_out: int = -1, W_out=None, ws=None):
    """exl3_regularize: output-channel normalisation with the skew heuristic.
    Returns dict(W_out fp32 [rows, cols], sv_out fp32 [cols],
    info fp64 [4] = (skew, applied, zeros, global rms))."""
    torch = _torch()
    _need_cuda(W, h, sv, W_out)
    rows, cols = W.shape
    dev = W.device
    if W_out is None:
        W_out = torch.empty(rows, cols, dtype=torch.float32, device=dev)
    sv_out = torch.empty(cols, dtype=torch.float32, device=dev)
    info = torch.empty(4, dtype=torch.float64, device=dev)
    ws = _workspace(regularize_workspace_bytes(rows, cols), dev, ws)
    _check(lib().exl3_regularize(_ptr(W), _dt(W), rows, cols, _ptr(h), _ptr(sv), int(apply_out),
                                 _ptr(W_out), _ptr(sv_out), _ptr(info), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(dev)))
    return dict(W_out=W_out, sv_out=sv_out, info=info)


def gss_scale(W, su, sv, K: int, lo: float = 0.5, hi: float = 2.0, n_eval: int = 12,
              best_codes=None, want_history: bool = False, ws=None):
    """exl3_gss_scale: device-resident golden-section search over g in [lo, hi].

    Returns dict(codes, scale, g, mse, history|None) as device tensors.
    """
    torch = _torch()
    _need_cuda(W, su, sv, best_codes)
    rows, cols = W.shape
    dev = W.device
    if best_codes is None:
        best_codes = torch.empty(rows // 16, cols // 16, 16 * K, dtype=torch.int16, device=dev)
    scale = torch.empty((), dtype=torch.float32, device=dev)
    g = torch.empty((), dtype=torch.float64, device=dev)
    m = torch.empty((), dtype=torch.float64, device=dev)
    hist = torch.empty(2 * n_eval, dtype=torch.float64, device=dev) if want_history else None
    ws = _workspace(gss_workspace_bytes(rows, cols, K), dev, ws)
    _check(lib().exl3_gss_scale(_ptr(W), _dt(W), rows, cols, _ptr(su), _ptr(sv), K,
                                ctypes.c_double(lo), ctypes.c_double(hi), int(n_eval),
                                _ptr(best_codes), _ptr(scale), _ptr(g), _ptr(m), _ptr(hist),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return dict(codes=best_codes, scale=scale, g=g, mse=m, history=hist)
