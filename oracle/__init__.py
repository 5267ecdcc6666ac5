"""Plain CPU oracle for the EXL3 trellis tile encoder.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` are the only callers.  The product
library never imports this package and shares no code with it.

The arithmetic lives in ``exl3_oracle.c`` (plain scalar C, fp32 without FMA
contraction, fp64 reductions); this module only builds it with gcc, loads it
with ctypes and marshals numpy arrays.  Tiles are spread over host threads:
ctypes releases the GIL for the duration of each foreign call.

Each function cites the passage it follows on the page "EXL3 Intel Arc
Quantizer", section "Core Implemented Architecture", items 1, 4, 5, 7 and 10.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exl3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libexl3_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

STATE_BITS = 16
TILE_STEPS = 256


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, u32, i64, f32 = ctypes.c_int, ctypes.c_uint32, ctypes.c_int64, ctypes.c_float
        L.ora_round_fp16.argtypes = [f32]
        L.ora_round_fp16.restype = f32
        L.ora_round_fp16_array.argtypes = [P, P, i64]
        L.ora_mul1_value.argtypes = [u32]
        L.ora_mul1_value.restype = f32
        L.ora_mul1_table.argtypes = [P, i32]
        L.ora_mul1_constant.restype = f32
        L.ora_mul1_multiplier.restype = u32
        L.ora_viterbi_forward.argtypes = [P, i32, i32, i32, P, i32, u32, P, P, P]
        L.ora_traceback.argtypes = [P, i32, i32, i32, i32, u32, P]
        L.ora_final_argmin.argtypes = [P, P, i32, i32]
        L.ora_final_argmin.restype = u32
        L.ora_encode_tile.argtypes = [P, i32, i32, i32, P, P, P, P]
        L.ora_encode_matrix.argtypes = [P, i64, i64, i32, f32, P, i64, i64, P, P]
        L.ora_pack.argtypes = [P, i32, i32, P]
        L.ora_unpack_states.argtypes = [P, i32, i32, i32, P]
        L.ora_decode_values.argtypes = [P, i32, P, f32, P]
        L.ora_rotate_forward.argtypes = [P, i64, i64, P, P, P]
        L.ora_rotate_inverse.argtypes = [P, i64, i64, P, P, P]
        L.ora_tile_sumsq.argtypes = [P, P, i64, i64, P]
        L.ora_tree_sum.argtypes = [P, i64]
        L.ora_tree_sum.restype = ctypes.c_double
        f64 = ctypes.c_double
        L.ora_cholesky.argtypes = [P, i64, f64, P]
        L.ora_cholesky.restype = i32
        L.ora_cholesky_damped.argtypes = [P, i64, f64, i32, P]
        L.ora_cholesky_damped.restype = i32
        L.ora_block_fold.argtypes = [P, i64, P]
        L.ora_ldlq_feedback.argtypes = [P, P, i64, i64, i64, P]
        L.ora_block_sumsq_cols.argtypes = [P, i64, i64, i32, P]
        _lib = L
        return L


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------
# codebook (item 5: procedural mul1 levels in fp16)
# --------------------------------------------------------------------------

def round_fp16(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty_like(x)
    _load().ora_round_fp16_array(_p(x), _p(out), x.size)
    return out


_mul1_cache: dict[int, np.ndarray] = {}


def mul1_table(L: int = STATE_BITS) -> np.ndarray:
    """v(s) for s in [0, 2^L): the mul1 decode of each state (fp32 holding fp16)."""
    if L not in _mul1_cache:
        out = np.empty(1 << L, dtype=np.float32)
        _load().ora_mul1_table(_p(out), 1 << L)
        _mul1_cache[L] = out
    return _mul1_cache[L]


def mul1_constant() -> float:
    return float(np.float32(_load().ora_mul1_constant()))


def mul1_multiplier() -> int:
    return int(_load().ora_mul1_multiplier())


# --------------------------------------------------------------------------
# Viterbi primitives (items 1 and 4)
# --------------------------------------------------------------------------

def viterbi_forward(y, L: int, K: int, cb, constrained: bool = False, pre_state: int = 0):
    """Forward ACS pass.  Returns (dec[T, 2^(L-K)] uint8, final_cost, penult_cost)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    cb = np.ascontiguousarray(cb, dtype=np.float32)
    T = y.size
    G = 1 << (L - K)
    dec = np.empty((T, G), dtype=np.uint8)
    fc = np.empty(G, dtype=np.float32)
    pen = np.empty(G, dtype=np.float32)
    _load().ora_viterbi_forward(_p(y), T, L, K, _p(cb), int(bool(constrained)),
                                int(pre_state), _p(dec), _p(fc), _p(pen))
    return dec, fc, pen


def traceback(dec, L: int, K: int, t_last: int, t_first: int, last_state: int) -> np.ndarray:
    dec = np.ascontiguousarray(dec, dtype=np.uint8)
    states = np.zeros(dec.shape[0], dtype=np.uint32)
    _load().ora_traceback(_p(dec), L, K, t_last, t_first, int(last_state), _p(states))
    return states


def final_argmin(dec_last_row, final_cost, L: int, K: int) -> int:
    d = np.ascontiguousarray(dec_last_row, dtype=np.uint8)
    c = np.ascontiguousarray(final_cost, dtype=np.float32)
    return int(_load().ora_final_argmin(_p(d), _p(c), L, K))


def encode_tile(y, K: int, L: int = STATE_BITS, cb=None):
    """Two-pass tail-biting encode of one tile.  Returns (states, cost, end_state)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    if cb is None:
        cb = mul1_table(L)
    cb = np.ascontiguousarray(cb, dtype=np.float32)
    T = y.size
    states = np.empty(T, dtype=np.uint32)
    cost = np.empty(1, dtype=np.float32)
    end = np.empty(1, dtype=np.uint32)
    _load().ora_encode_tile(_p(y), T, L, K, _p(cb), _p(states), _p(cost), _p(end))
    return states, float(cost[0]), int(end[0])


def encode_matrix(Y, K: int, inv_scale: float = 1.0, tiles=None, threads: int | None = None):
    """Encode the 16x16 tiles of an fp32 [rows, cols] matrix (targets Y * inv_scale).

    ``tiles``: optional array of tile indices (row-major tile order); default all.
    Returns (states[n, 256] uint32, costs[n] float32) in the order of ``tiles``.
    """
    Y = np.ascontiguousarray(Y, dtype=np.float32)
    rows, cols = Y.shape
    n_all = (rows // 16) * (cols // 16)
    idx = np.arange(n_all, dtype=np.int64) if tiles is None else np.asarray(tiles, dtype=np.int64)
    cb = mul1_table(STATE_BITS)
    states = np.empty((idx.size, 256), dtype=np.uint32)
    costs = np.empty(idx.size, dtype=np.float32)
    lib = _load()
    inv = np.float32(inv_scale)

    def work(i):
        t = int(idx[i])
        st = np.empty(256, dtype=np.uint32)
        c = np.empty(1, dtype=np.float32)
        lib.ora_encode_matrix(_p(Y), rows, cols, K, ctypes.c_float(inv), _p(cb), t, t + 1,
                              _p(st), _p(c))
        states[i] = st
        costs[i] = c[0]

    nthr = threads or default_threads()
    if nthr == 1 or idx.size <= 1:
        for i in range(idx.size):
            work(i)
    else:
        with ThreadPoolExecutor(max_workers=nthr) as ex:
            list(ex.map(work, range(idx.size)))
    return states, costs


# --------------------------------------------------------------------------
# packing (item 5: MSB-first stream, SWAP16) and decode
# --------------------------------------------------------------------------

def pack(states, K: int) -> np.ndarray:
    states = np.ascontiguousarray(states, dtype=np.uint32)
    T = states.size
    out = np.empty(T * K // 16, dtype=np.uint16)
    _load().ora_pack(_p(states), T, K, _p(out))
    return out


def unpack_states(words, K: int, L: int = STATE_BITS, T: int = TILE_STEPS) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint16)
    assert words.size == T * K // 16
    out = np.empty(T, dtype=np.uint32)
    _load().ora_unpack_states(_p(words), T, K, L, _p(out))
    return out


def decode_values(states, scale: float, cb=None) -> np.ndarray:
    states = np.ascontiguousarray(states, dtype=np.uint32)
    if cb is None:
        cb = mul1_table(STATE_BITS)
    out = np.empty(states.size, dtype=np.float32)
    _load().ora_decode_values(_p(states), states.size, _p(cb), ctypes.c_float(np.float32(scale)),
                              _p(out))
    return out


def codes_from_states(states, rows: int, cols: int, K: int) -> np.ndarray:
    """Per-tile packed codes laid out [rows/16, cols/16, 16K] (uint16)."""
    n = (rows // 16) * (cols // 16)
    assert states.shape == (n, 256)
    out = np.empty((n, 16 * K), dtype=np.uint16)
    for t in range(n):
        out[t] = pack(states[t], K)
    return out.reshape(rows // 16, cols // 16, 16 * K)


def decode_matrix(codes, rows: int, cols: int, K: int, scale: float) -> np.ndarray:
    """Packed codes [rows/16, cols/16, 16K] -> fp32 [rows, cols] = fl(v(s) * scale)."""
    codes = np.asarray(codes, dtype=np.uint16).reshape(-1, 16 * K)
    tr, tc = rows // 16, cols // 16
    out = np.empty((rows, cols), dtype=np.float32)
    for t in range(tr * tc):
        st = unpack_states(codes[t], K)
        v = decode_values(st, scale).reshape(16, 16)
        r0, c0 = (t // tc) * 16, (t % tc) * 16
        out[r0:r0 + 16, c0:c0 + 16] = v
    return out


# --------------------------------------------------------------------------
# rotation (item 7)
# --------------------------------------------------------------------------

def rotate_forward(W, su, sv) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    su = np.ascontiguousarray(su, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    rows, cols = W.shape
    out = np.empty_like(W)
    _load().ora_rotate_forward(_p(W), rows, cols, _p(su), _p(sv), _p(out))
    return out


def rotate_inverse(Q, su, sv) -> np.ndarray:
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    su = np.ascontiguousarray(su, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    rows, cols = Q.shape
    out = np.empty_like(Q)
    _load().ora_rotate_inverse(_p(Q), rows, cols, _p(su), _p(sv), _p(out))
    return out


# --------------------------------------------------------------------------
# fixed-order fp64 reductions (item 10)
# --------------------------------------------------------------------------

def tile_sumsq(x, ref=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    out = np.empty((rows // 16) * (cols // 16), dtype=np.float64)
    r = None if ref is None else np.ascontiguousarray(ref, dtype=np.float32)
    _load().ora_tile_sumsq(_p(x), None if r is None else _p(r), rows, cols, _p(out))
    return out


def tree_sum(v) -> float:
    v = np.ascontiguousarray(v, dtype=np.float64)
    return float(_load().ora_tree_sum(_p(v), v.size))


def rms(R) -> float:
    """sigma_R = sqrt(tree(tile sums of R^2) / n) in fp64."""
    R = np.asarray(R, dtype=np.float32)
    return math.sqrt(tree_sum(tile_sumsq(R)) / R.size)


def mse(W, What) -> float:
    W = np.asarray(W, dtype=np.float32)
    return tree_sum(tile_sumsq(W, What)) / W.size


def scale_for(g: float, sigma: float) -> tuple[float, float]:
    """(s, inv_s): s = fl32(g * sigma) (product in fp64), inv_s = fl32(1 / s).
    An all-zero matrix (sigma == 0) is coded at sigma = 1."""
    if sigma == 0.0:
        sigma = 1.0
    s = np.float32(float(g) * float(sigma))
    inv = np.float32(1.0) / s
    return float(s), float(inv)


from .gss import golden_section_search, evaluate_matrix  # noqa: E402,F401
