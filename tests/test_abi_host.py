"""Host-side checks of the C ABI (not gpu): the library loads, exports every
symbol include/exl3.h declares, and rejects bad arguments before touching the
GPU.  Only invalid-argument paths are exercised, with fake pointers that the
library never dereferences."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ex():
    import __graft_entry__
    from exl3_trellis_weight_gb300 import build
    build.build()
    import exl3_trellis_weight_gb300 as ex
    ex.lib()
    return ex


def _declared():
    src = open(os.path.join(ROOT, "include", "exl3.h")).read()
    return sorted(set(re.findall(r"EXL3_API[^;(]*?\b(exl3_\w+)\s*\(", src)))


def test_header_declares_the_path(ex):
    names = _declared()
    for n in ["exl3_rotate", "exl3_encode_tiles", "exl3_decode_tiles", "exl3_gss_scale",
              "exl3_quantize", "exl3_mse", "exl3_scale_search"]:
        assert n in names


def test_every_declared_symbol_is_exported(ex):
    L = ex.lib()
    for n in _declared():
        assert hasattr(L, n), n


def test_status_strings(ex):
    L = ex.lib()
    assert L.exl3_status_str(0) == b"EXL3_OK"
    assert L.exl3_status_str(3) == b"EXL3_ERR_WORKSPACE"
    assert L.exl3_status_str(5) == b"EXL3_ERR_TIMEOUT"
    assert L.exl3_status_str(6) == b"EXL3_ERR_NUMERIC"
    assert L.exl3_status_str(99) == b"EXL3_ERR_UNKNOWN"
    assert L.exl3_version() >= 100


def test_supported_k(ex):
    assert [ex.supports_k(k) for k in range(0, 6)] == [False, True, True, True, True, False]


FAKE = ctypes.c_void_p(0x10000000)      # 256-byte aligned, never dereferenced


def test_encode_rejects_bad_arguments(ex):
    L = ex.lib()
    ws_min = ex.encode_workspace_min_bytes(2)
    assert ws_min > 0
    args = dict(Y=FAKE, rows=64, cols=64, K=2, scale=ctypes.c_float(1.0), codes=FAKE,
                cost=None, ws=FAKE, ws_bytes=ws_min, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.exl3_encode_tiles(a["Y"], a["rows"], a["cols"], a["K"], a["scale"], a["codes"],
                                   a["cost"], a["ws"], a["ws_bytes"], a["stream"])

    assert call(K=0) == 2 and call(K=5) == 2               # unsupported K
    assert call(K=1, ws_bytes=ws_min - 256) == 3           # below one block slice
    assert call(rows=40) == 2 and call(cols=24) == 2       # not multiples of 16
    assert call(rows=0) == 1 and call(cols=-16) == 1
    assert call(Y=None) == 1 and call(codes=None) == 1
    assert call(codes=ctypes.c_void_p(0x10000002)) == 1    # misaligned
    assert call(scale=ctypes.c_float(0.0)) == 1
    assert call(scale=ctypes.c_float(float("inf"))) == 1
    assert call(scale=ctypes.c_float(float("nan"))) == 1
    assert call(scale=ctypes.c_float(1e-45)) == 1          # 1 / scale overflows to inf
    assert call(ws_bytes=ws_min - 1) == 3                   # workspace too small
    assert call(ws=None) == 1
    assert call(ws=ctypes.c_void_p(0x10000010)) == 1        # workspace not 256-aligned
    assert b"workspace" in L.exl3_last_error()


def test_rotate_and_quantize_reject_bad_arguments(ex):
    L = ex.lib()
    # rows/cols must be multiples of 128 for the rotation
    assert L.exl3_rotate(FAKE, 1, 64, 128, FAKE, FAKE, 0, ctypes.c_void_p(0x20000000), None) == 2
    assert L.exl3_rotate(FAKE, 7, 128, 128, FAKE, FAKE, 0, ctypes.c_void_p(0x20000000), None) == 1
    assert L.exl3_rotate(FAKE, 1, 128, 128, FAKE, FAKE, 1, ctypes.c_void_p(0x20000000), None) == 1
    assert L.exl3_rotate(FAKE, 0, 128, 128, None, FAKE, 0, ctypes.c_void_p(0x20000000), None) == 1
    # overlapping output
    assert L.exl3_rotate(FAKE, 1, 128, 128, FAKE, FAKE, 0, ctypes.c_void_p(0x10000100), None) == 1
    ws = ex.quantize_workspace_bytes(256, 256, 2)
    assert ws > 0
    q = lambda **kw: L.exl3_quantize(FAKE, 1, kw.get("rows", 256), 256, FAKE, FAKE, kw.get("K", 2),
                                     ctypes.c_double(kw.get("g", 1.0)), FAKE, FAKE, FAKE, None, None,
                                     FAKE, kw.get("ws", ws), None)
    assert q(K=3, g=-1.0) == 1
    assert q(g=float("nan")) == 1
    assert q(rows=200) == 2
    assert q(K=7) == 2
    assert q(ws=1000) == 3
    gws = ex.gss_workspace_bytes(256, 256, 2)
    gs = lambda lo, hi, n, w=gws: L.exl3_gss_scale(FAKE, 1, 256, 256, FAKE, FAKE, 2,
                                                   ctypes.c_double(lo), ctypes.c_double(hi), n,
                                                   FAKE, FAKE, FAKE, FAKE, None, FAKE, w, None)
    assert gs(0.5, 2.0, 1) == 1
    assert gs(0.5, 2.0, 65) == 1
    assert gs(2.0, 0.5, 12) == 1
    assert gs(0.0, 2.0, 12) == 1
    assert gs(0.5, 2.0, 12, w=100) == 3
    sws = ex.scale_search_workspace_bytes(256, 256, 2)
    sc = lambda rows, cols, K, w=sws, g=FAKE: L.exl3_scale_search(FAKE, 1, rows, cols, FAKE, FAKE, K,
                                                                  g, None, None, FAKE, w, None)
    assert sc(256, 200, 2) == 2          # cols not a multiple of 128
    assert sc(256, 256, 5) == 2
    assert sc(256, 256, 2, g=None) == 1
    assert sc(256, 256, 2, w=100) == 3
    assert sc(32768, 128, 2) == 2        # beyond the 32736-row limit


def test_ldl_and_ldlq_reject_bad_arguments(ex):
    L = ex.lib()
    wl = ex.block_ldl_workspace_bytes(64)
    ldl = lambda n=64, H=FAKE, M=FAKE, sig=0.01, r=10, w=wl: L.exl3_block_ldl(
        H, n, ctypes.c_double(sig), r, M, None, FAKE, w, None)
    assert ldl(n=40) == 2 and ldl(n=0) == 2 and ldl(n=32784) == 2
    assert ldl(H=None) == 1
    assert ldl(M=ctypes.c_void_p(0x10000004)) == 1          # M must be 16-byte aligned
    assert ldl(sig=-1.0) == 1 and ldl(sig=float("inf")) == 1
    assert ldl(r=-1) == 1 and ldl(r=101) == 1
    assert ldl(w=wl - 1) == 3
    assert ex.block_ldl_workspace_bytes(64) >= 64 * 64 * 8
    assert ex.block_ldl_workspace_bytes(40) == 0
    wq = ex.ldlq_workspace_bytes(64, 128, 2)
    lq = lambda rows=64, cols=128, K=2, s=1.0, w=wq, codes=FAKE: L.exl3_ldlq(
        FAKE, rows, cols, FAKE, K, ctypes.c_float(s), codes, None, FAKE, w, None)
    assert lq(rows=40) == 2 and lq(cols=8) == 2
    assert lq(rows=1 << 20, cols=1 << 15) == 1             # 2^35 elements
    assert lq(K=5) == 2
    assert lq(s=0.0) == 1 and lq(s=float("nan")) == 1
    assert lq(codes=None) == 1
    assert lq(w=64 * 128 * 4) == 3
    assert ex.ldlq_workspace_bytes(64, 128, 0) == 0
    # every K needs at least one encode block slice on top of the fixed part
    w1 = ex.ldlq_workspace_bytes(64, 128, 1)
    fixed = w1 - (w1 - 64 * 128 * 4) // ex.encode_workspace_min_bytes(1) * ex.encode_workspace_min_bytes(1)
    assert lq(K=1, w=fixed + ex.encode_workspace_min_bytes(1) - 256) == 3


def test_regularize_rejects_bad_arguments(ex):
    L = ex.lib()
    w = ex.regularize_workspace_bytes(64, 32)
    rg = lambda rows=64, cols=32, dt=1, W=FAKE, Wo=ctypes.c_void_p(0x20000000), ap=-1, ws=w: \
        L.exl3_regularize(W, dt, rows, cols, FAKE, FAKE, ap, Wo, FAKE, None, FAKE, ws, None)
    assert rg(rows=0) == 2 and rg(cols=0) == 2 and rg(rows=65537) == 2
    assert rg(dt=7) == 1
    assert rg(W=None) == 1
    assert rg(ap=2) == 1 and rg(ap=-2) == 1
    assert rg(Wo=FAKE) == 1                     # in place needs an fp32 W
    assert rg(dt=0, Wo=FAKE, ws=100) == 3       # fp32 in place is fine; workspace too small
    assert ex.regularize_workspace_bytes(64, 32) > 32 * 32 * 8
    assert ex.regularize_workspace_bytes(0, 32) == 0


def test_workspace_queries_scale_with_work(ex):
    a = ex.encode_workspace_bytes(10, 2)
    b = ex.encode_workspace_bytes(100000, 2)
    assert 0 < a <= b
    assert a == 10 * ex.encode_workspace_min_bytes(2)
    assert ex.encode_workspace_bytes(100, 0) == 0
    assert all(ex.encode_workspace_min_bytes(k) == ex.encode_workspace_min_bytes(2) for k in (1, 3, 4))
    assert ex.quantize_workspace_bytes(4096, 4096, 2) > 4096 * 4096 * 4
    assert ex.gss_workspace_bytes(4096, 4096, 2) > ex.quantize_workspace_bytes(4096, 4096, 2)
    assert ex.scale_search_workspace_bytes(4096, 4096, 2) > 4096 * 4096 * 4
    assert ex.scale_search_workspace_bytes(4096, 4096, 0) == 0


def test_rows_reject_bad_lengths(ex):
    L = ex.lib()
    ws_min = ex.encode_workspace_min_bytes(2)
    enc = lambda n, T, K, ws=ws_min: L.exl3_encode_rows(FAKE, n, T, K, ctypes.c_float(1.0), FAKE,
                                                        None, FAKE, ws, None)
    assert enc(10, 161, 2) == 2          # odd T
    assert enc(10, 258, 2) == 2          # T > 256
    assert enc(10, 8, 4) == 2            # T < 16
    assert enc(10, 48, 3) == 2           # T*K not a multiple of 32
    assert enc(0, 160, 2) == 1
    assert enc(10, 160, 5) == 2
    assert enc(10, 160, 2, ws=ws_min - 1) == 3
    dec = lambda n, T, K: L.exl3_decode_rows(FAKE, n, T, K, ctypes.c_float(1.0), FAKE, None)
    assert dec(10, 161, 2) == 2 and dec(-1, 160, 2) == 1
