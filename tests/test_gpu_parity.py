"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Codes, decoded values, rotations and tile costs must be bit-exact; the scale
and the MSE are compared within 1e-6 relative (the fixed reduction order makes
them exact in practice, and the tests also record that).  Inputs come from the
seeded generators in exl3_trellis_weight_gb300.inputs and reach both sides as
the same bytes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from exl3_trellis_weight_gb300 import inputs  # noqa: E402

REL_TOL = 1e-6


@pytest.fixture(scope="module")
def ex():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for -m gpu tests")
    import __graft_entry__
    __graft_entry__.build()
    import exl3_trellis_weight_gb300 as ex
    return ex


DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _no_expired_waits(ex):
    """No bounded device wait (the TMA rotation's) may give up in any test."""
    yield
    assert ex.wait_timeouts() == 0


def _np_codes(codes_t, K):
    return codes_t.detach().cpu().numpy().view(np.uint16).reshape(-1, 16 * K)


def _oracle_codes(Y, K, inv_scale, tiles=None):
    st, costs = oracle.encode_matrix(Y, K, inv_scale, tiles=tiles)
    return np.stack([oracle.pack(s, K) for s in st]), costs


def _tiles_of(rows, cols):
    return (rows // 16) * (cols // 16)


# ---------------------------------------------------------------------------
# encode: small cases, all tiles
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def rot128():
    (_, W, _, _, _), = inputs.workload("rot128_iid_k2")
    return W.numpy()


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_encode_rot128_bit_exact(ex, rot128, K):
    Y = rot128
    codes, cost = ex.encode_tiles(torch.from_numpy(Y).to(DEV), K, scale=1.0, want_cost=True)
    torch.cuda.synchronize()
    want, wcost = _oracle_codes(Y, K, 1.0)
    got = _np_codes(codes, K)
    assert np.array_equal(got, want)
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), wcost.view(np.uint32))


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("blocks", [None, 1, 4])
def test_encode_ragged_tiles_and_small_grids(ex, K, blocks):
    """15 tiles (3x5, not a multiple of the pair pipeline); 1 block walks all
    15 (odd count, drain phase), 4 blocks take 4/4/4/3."""
    rng = np.random.default_rng(10 + K)
    Y = rng.standard_normal((48, 80)).astype(np.float32) * 0.7
    ws = None
    if blocks is not None:
        # the minimum workspace is one block slice
        ws = torch.empty(blocks * ex.encode_workspace_min_bytes(K), dtype=torch.uint8, device=DEV)
    codes, cost = ex.encode_tiles(torch.from_numpy(Y).to(DEV), K, scale=0.7, want_cost=True, ws=ws)
    torch.cuda.synchronize()
    inv = float(np.float32(1.0) / np.float32(0.7))
    want, wcost = _oracle_codes(Y, K, inv)
    assert np.array_equal(_np_codes(codes, K), want)
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), wcost.view(np.uint32))


def _edge_inputs():
    rng = np.random.default_rng(5)
    cb = oracle.mul1_table()
    yield "zeros", np.zeros((16, 64), np.float32)
    yield "constant", np.full((16, 64), 0.37, np.float32)
    yield "tiny", (rng.standard_normal((16, 64)) * 1e-30).astype(np.float32)
    yield "outliers", np.where(rng.random((16, 64)) < 0.05, 1e4, rng.standard_normal((16, 64))).astype(np.float32)
    # targets exactly on codebook levels: many exact ties between paths
    yield "levels", cb[rng.integers(0, 65536, (16, 64))].astype(np.float32)
    yield "two_levels", np.where(rng.random((16, 64)) < 0.5, cb[1], cb[2]).astype(np.float32)


@pytest.mark.parametrize("name,Y", list(_edge_inputs()), ids=[n for n, _ in _edge_inputs()])
@pytest.mark.parametrize("K", [1, 2, 4])
def test_encode_edge_inputs_bit_exact(ex, name, Y, K):
    codes, cost = ex.encode_tiles(torch.from_numpy(Y).to(DEV), K, scale=1.0, want_cost=True)
    torch.cuda.synchronize()
    want, wcost = _oracle_codes(Y, K, 1.0)
    assert np.array_equal(_np_codes(codes, K), want), name
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), wcost.view(np.uint32)), name


def test_encode_single_tile_and_repeatability(ex):
    rng = np.random.default_rng(99)
    Y = rng.standard_normal((16, 16)).astype(np.float32)
    a = ex.encode_tiles(torch.from_numpy(Y).to(DEV), 3)
    b = ex.encode_tiles(torch.from_numpy(Y).to(DEV), 3)
    torch.cuda.synchronize()
    want, _ = _oracle_codes(Y, 3, 1.0)
    assert np.array_equal(_np_codes(a, 3), want)
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# decode, rotation, MSE
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_decode_random_codes_bit_exact(ex, K):
    rows, cols = 512, 1024 if K == 4 else 256
    rng = np.random.default_rng(K)
    n = _tiles_of(rows, cols)
    codes = rng.integers(0, 1 << 16, (n, 16 * K), dtype=np.uint64).astype(np.uint16)
    scale = 0.0123
    got = ex.decode_tiles(torch.from_numpy(codes.view(np.int16)).to(DEV).reshape(rows // 16, cols // 16, 16 * K),
                          rows, cols, K, scale)
    torch.cuda.synchronize()
    want = oracle.decode_matrix(codes, rows, cols, K, scale)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))
    if K == 4:
        # 2^20 windows: (nearly) every state's level went through the comparison
        states = np.concatenate([oracle.unpack_states(codes[t], K) for t in range(0, n, 1)])
        assert np.unique(states).size > 65000


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_rotate_forward_and_inverse_bit_exact(ex, dt):
    rows, cols = 256, 384
    W = inputs.linear_bf16(rows, cols, seed=3, std=0.02)
    if dt == "f32":
        W = (W.float() + torch.randn(rows, cols, generator=torch.Generator().manual_seed(4)) * 1e-3)
    su, sv = inputs.sign_pair(rows, cols, 3)
    R = ex.rotate(W.to(DEV), su.to(DEV), sv.to(DEV))
    torch.cuda.synchronize()
    Wf = W.float().numpy()
    want = oracle.rotate_forward(Wf, su.numpy(), sv.numpy())
    assert np.array_equal(R.cpu().numpy().view(np.uint32), want.view(np.uint32))
    back = ex.rotate(R, su.to(DEV), sv.to(DEV), inverse=True)
    torch.cuda.synchronize()
    want_b = oracle.rotate_inverse(want, su.numpy(), sv.numpy())
    assert np.array_equal(back.cpu().numpy().view(np.uint32), want_b.view(np.uint32))


def test_rotate_in_place_fp32(ex):
    rows, cols = 128, 256
    W = torch.randn(rows, cols, generator=torch.Generator().manual_seed(8))
    su, sv = inputs.sign_pair(rows, cols, 8)
    want = oracle.rotate_forward(W.numpy(), su.numpy(), sv.numpy())
    Wd = W.to(DEV)
    ex.rotate(Wd, su.to(DEV), sv.to(DEV), out=Wd)
    torch.cuda.synchronize()
    assert np.array_equal(Wd.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_rotate_forward_unaligned_views(ex, dt):
    """Inputs and outputs that are not 16-byte aligned take the shuffle-based
    kernel; 16-byte aligned fp32 inputs the shared-memory one; 16-byte aligned
    bf16 inputs the TMA one, also from a base that is only 16-byte aligned: all
    give the oracle's bits, including non-unit sign vectors (su, sv multiplied as
    given)."""
    rows, cols = 128, 384
    W = inputs.linear_bf16(rows, cols, seed=11, std=0.02)
    if dt == "f32":
        W = W.float()
    su = inputs.signs(rows, 12) * 0.75
    sv = inputs.signs(cols, 13) * 1.25
    want = oracle.rotate_forward(W.float().numpy(), su.numpy(), sv.numpy())
    n = rows * cols
    buf = torch.empty(n + 8, dtype=W.dtype, device=DEV)
    Wu = buf[1:1 + n].view(rows, cols)                  # element offset 1: 2 or 4 bytes
    Wu.copy_(W.to(DEV))
    obuf = torch.empty(n + 8, dtype=torch.float32, device=DEV)
    out_u = obuf[2:2 + n].view(rows, cols)              # 8-byte offset
    buf16 = torch.empty(n + 8, dtype=W.dtype, device=DEV)
    W16 = buf16[(8 if dt == "bf16" else 4):][:n].view(rows, cols)   # 16-byte offset
    W16.copy_(W.to(DEV))
    obuf16 = torch.empty(n + 8, dtype=torch.float32, device=DEV)
    out16 = obuf16[4:4 + n].view(rows, cols)            # 16-byte offset
    def kernel_for(src, out):
        al16 = src.data_ptr() % 16 == 0 and (out is None or out.data_ptr() % 16 == 0)
        if not al16:
            return 3                                     # warp-shuffle kernel
        return 1 if dt == "bf16" else 2                  # TMA (bf16) / shared-memory (fp32)

    for src, out in ((W.to(DEV), None), (Wu, None), (W.to(DEV), out_u), (Wu, out_u),
                     (W16, out16), (W16, None), (W.to(DEV), out16)):
        R = ex.rotate(src, su.to(DEV), sv.to(DEV), out=out)
        assert ex.rotate_last_kernel() == kernel_for(src, out)
        torch.cuda.synchronize()
        assert np.array_equal(R.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_mse_fixed_order(ex, dt):
    rows, cols = 256, 512
    W = inputs.linear_bf16(rows, cols, seed=11)
    if dt == "f32":
        W = W.float()
    What = (W.float() + torch.randn(rows, cols, generator=torch.Generator().manual_seed(12)) * 1e-3)
    m = ex.mse(W.to(DEV), What.to(DEV))
    torch.cuda.synchronize()
    want = oracle.mse(W.float().numpy(), What.numpy())
    got = float(m.item())
    assert abs(got - want) <= REL_TOL * want
    assert got == want   # same per-tile order and tree


# ---------------------------------------------------------------------------
# full chain and golden-section search
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols,K,seed", [(256, 256, 2, 21), (128, 256, 3, 22), (256, 128, 4, 23),
                                              (128, 128, 1, 24)])
def test_quantize_chain_matches_oracle(ex, rows, cols, K, seed):
    W = inputs.linear_bf16(rows, cols, seed=seed, std=0.02, outlier_frac=0.001)
    su, sv = inputs.sign_pair(rows, cols, seed)
    res = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K, g=1.1, want_What=True)
    torch.cuda.synchronize()
    ref = oracle.evaluate_matrix(W.float().numpy(), su.numpy(), sv.numpy(), K, 1.1)
    assert np.array_equal(_np_codes(res["codes"], K), ref["codes"].reshape(-1, 16 * K))
    assert float(res["scale"].item()) == ref["scale"]
    assert float(res["sigma"].item()) == ref["sigma"]
    assert np.array_equal(res["What"].cpu().numpy().view(np.uint32), ref["What"].view(np.uint32))
    got = float(res["mse"].item())
    assert abs(got - ref["mse"]) <= REL_TOL * ref["mse"]


def test_quantize_zero_matrix(ex):
    W = torch.zeros(128, 128, dtype=torch.bfloat16)
    su, sv = inputs.sign_pair(128, 128, 1)
    res = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), 2, g=1.0)
    torch.cuda.synchronize()
    ref = oracle.evaluate_matrix(W.float().numpy(), su.numpy(), sv.numpy(), 2, 1.0)
    assert np.array_equal(_np_codes(res["codes"], 2), ref["codes"].reshape(-1, 32))
    assert float(res["scale"].item()) == ref["scale"] == 1.0
    assert float(res["mse"].item()) == ref["mse"]


def test_quantize_small_workspace_same_result(ex):
    rows, cols, K = 256, 256, 2
    W = inputs.linear_bf16(rows, cols, seed=31)
    su, sv = inputs.sign_pair(rows, cols, 31)
    full = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(_tiles_of(rows, cols), sms)
    fixed = ex.quantize_workspace_bytes(rows, cols, K) - grid * ex.encode_workspace_min_bytes(K)
    ws = torch.empty(fixed + 3 * ex.encode_workspace_min_bytes(K), dtype=torch.uint8, device=DEV)
    small = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(full["codes"], small["codes"])
    assert float(full["mse"].item()) == float(small["mse"].item())


@pytest.mark.parametrize("K,seed", [(2, 41), (1, 42), (3, 43), (4, 44)])
def test_gss_matches_oracle_search(ex, K, seed):
    rows, cols = 128, 128
    W = inputs.linear_bf16(rows, cols, seed=seed, std=0.02)
    su, sv = inputs.sign_pair(rows, cols, seed)
    res = ex.gss_scale(W.to(DEV), su.to(DEV), sv.to(DEV), K, 0.5, 2.0, 12, want_history=True)
    torch.cuda.synchronize()
    Wf, sun, svn = W.float().numpy(), su.numpy(), sv.numpy()
    cache = {}

    def f(g):
        cache[g] = oracle.evaluate_matrix(Wf, sun, svn, K, g)
        return cache[g]["mse"]

    best_g, best_f, hist = oracle.golden_section_search(f, 0.5, 2.0, 12)
    h = res["history"].cpu().numpy().reshape(-1, 2)
    assert np.array_equal(h[:, 0], np.array([x for x, _ in hist]))
    assert np.allclose(h[:, 1], np.array([y for _, y in hist]), rtol=REL_TOL, atol=0)
    assert float(res["g"].item()) == best_g
    assert abs(float(res["mse"].item()) - best_f) <= REL_TOL * best_f
    assert float(res["scale"].item()) == cache[best_g]["scale"]
    assert np.array_equal(_np_codes(res["codes"], K), cache[best_g]["codes"].reshape(-1, 16 * K))


# ---------------------------------------------------------------------------
# full workload sizes, launch configuration of the benchmark, sampled tiles
# ---------------------------------------------------------------------------

def _sample_tiles(n, k, seed):
    rng = np.random.default_rng(seed)
    fixed = np.array([0, 1, n - 1, n // 2, n - 2], dtype=np.int64)
    return np.unique(np.concatenate([fixed, rng.choice(n, k, replace=False)]))


def _check_full(ex, W, su, sv, K, n_sample, seed):
    rows, cols = W.shape
    res = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K, g=1.0)
    torch.cuda.synchronize()
    Wf = W.float().numpy()
    R = oracle.rotate_forward(Wf, su.numpy(), sv.numpy())
    sigma = oracle.rms(R)
    s, inv = oracle.scale_for(1.0, sigma)
    assert float(res["sigma"].item()) == sigma
    assert float(res["scale"].item()) == s
    idx = _sample_tiles(_tiles_of(rows, cols), n_sample, seed)
    want, _ = _oracle_codes(R, K, inv, tiles=idx)
    got = _np_codes(res["codes"], K)[idx]
    assert np.array_equal(got, want)
    # the decoded weights of the sampled tiles (rotated domain, fl(v * s))
    Yhat = ex.decode_tiles(res["codes"], rows, cols, K, s)
    torch.cuda.synchronize()
    Yh = Yhat.cpu().numpy()
    tc = cols // 16
    for t, words in zip(idx, want):
        vals = oracle.decode_values(oracle.unpack_states(words, K), s).reshape(16, 16)
        r0, c0 = (t // tc) * 16, (t % tc) * 16
        assert np.array_equal(Yh[r0:r0 + 16, c0:c0 + 16], vals)
    return res


def test_full_linear4096_k2_sampled(ex):
    (_, W, su, sv, K), = inputs.workload("linear4096_k2")
    res = _check_full(ex, W, su, sv, K, 48, 1)
    m = float(res["mse"].item())
    assert 0 < m < float(W.float().var())


@pytest.mark.parametrize("wl,proj,band", [("linear4096_k2", None, 17), ("mlp12288_t5_k4", None, 61),
                                          ("layer4096_k3", "gate", 40)])
def test_full_size_one_whole_band(ex, wl, proj, band):
    """Every tile of one 128-row band (2,048 tiles) of a full-size workload, coded in
    the benchmark's launch configuration, equals the oracle bit for bit."""
    (_, W, su, sv, K), = [w for w in inputs.workload(wl) if proj is None or w[0] == proj]
    rows, cols = W.shape
    res = ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K, g=1.0)
    torch.cuda.synchronize()
    R = oracle.rotate_forward(W.float().numpy(), su.numpy(), sv.numpy())
    s, inv = oracle.scale_for(1.0, oracle.rms(R))
    assert float(res["scale"].item()) == s
    tc = cols // 16
    idx = np.arange(band * 8 * tc, (band + 1) * 8 * tc, dtype=np.int64)
    assert idx[-1] < _tiles_of(rows, cols)
    want, _ = _oracle_codes(R, K, inv, tiles=idx)
    assert np.array_equal(_np_codes(res["codes"], K)[idx], want)


def test_full_mlp12288_k4_sampled(ex):
    (_, W, su, sv, K), = inputs.workload("mlp12288_t5_k4")
    _check_full(ex, W, su, sv, K, 24, 2)


def test_full_linear4096_k1_sampled(ex):
    """K=1 (one block per tile, cost row updated in place) at full size, the bench's
    launch configuration."""
    (_, W, su, sv, _), = inputs.workload("linear4096_k2")
    _check_full(ex, W, su, sv, 1, 24, 5)


@pytest.mark.parametrize("proj", ["q", "k", "v", "o", "gate", "up", "down"])
def test_full_layer_k3_sampled(ex, proj):
    for lab, W, su, sv, K in inputs.workload("layer4096_k3"):
        if lab == proj:
            _check_full(ex, W, su, sv, K, 16, 3)


def test_full_gss4096_k2(ex):
    """12-evaluation search on 4096x4096: the state machine reproduces the
    oracle's points given the measured MSEs; the best codes equal a fresh
    quantize at the best g; sampled tiles match the oracle at that scale."""
    (_, W, su, sv, K), = inputs.workload("gss4096_k2")
    Wd, sud, svd = W.to(DEV), su.to(DEV), sv.to(DEV)
    res = ex.gss_scale(Wd, sud, svd, K, 0.5, 2.0, 12, want_history=True)
    torch.cuda.synchronize()
    h = res["history"].cpu().numpy().reshape(-1, 2)
    lookup = {float(x): float(y) for x, y in h}
    best_g, best_f, hist = oracle.golden_section_search(lambda g: lookup[g], 0.5, 2.0, 12)
    assert [x for x, _ in hist] == [float(x) for x in h[:, 0]]
    assert float(res["g"].item()) == best_g and float(res["mse"].item()) == best_f
    again = ex.quantize(Wd, sud, svd, K, g=best_g)
    torch.cuda.synchronize()
    assert torch.equal(again["codes"], res["codes"])
    assert float(again["mse"].item()) == best_f
    R = oracle.rotate_forward(W.float().numpy(), su.numpy(), sv.numpy())
    s, inv = oracle.scale_for(best_g, oracle.rms(R))
    assert float(res["scale"].item()) == s
    # 16 sampled tiles plus every tile of one whole 128-row band at the chosen scale
    tc = W.shape[1] // 16
    band = np.arange(23 * 8 * tc, 24 * 8 * tc, dtype=np.int64)
    idx = np.unique(np.concatenate([_sample_tiles(_tiles_of(*W.shape), 16, 4), band]))
    want, _ = _oracle_codes(R, K, inv, tiles=idx)
    assert np.array_equal(_np_codes(res["codes"], K)[idx], want)


def test_profile_counts_launches(ex):
    rows, cols, K = 256, 256, 2
    W = inputs.linear_bf16(rows, cols, seed=51)
    su, sv = inputs.sign_pair(rows, cols, 51)
    ex.profile_enable(True)
    ex.quantize(W.to(DEV), su.to(DEV), sv.to(DEV), K)
    ms, n_enc, n_all = ex.profile_read()
    ex.profile_enable(False)
    assert n_enc == 1 and ms > 0
    assert n_all >= 7


# ---------------------------------------------------------------------------
# rows of T targets (non-256 tile lengths)
# ---------------------------------------------------------------------------

ROW_CASES = [(160, 1), (160, 2), (160, 3), (160, 4), (16, 2), (48, 2), (96, 3), (64, 4), (256, 2),
             (32, 4), (64, 1)]


@pytest.mark.parametrize("T,K", ROW_CASES)
def test_encode_rows_bit_exact(ex, T, K):
    rng = np.random.default_rng(T * 10 + K)
    n_rows = 37
    Y = rng.standard_normal((n_rows, T)).astype(np.float32)
    codes, cost = ex.encode_rows(torch.from_numpy(Y).to(DEV), K, 1.3, want_cost=True)
    torch.cuda.synchronize()
    inv = np.float32(1.0) / np.float32(1.3)
    got = codes.cpu().numpy().view(np.uint16)
    for r in range(n_rows):
        st, c, _ = oracle.encode_tile((Y[r] * inv).astype(np.float32), K)
        assert np.array_equal(got[r], oracle.pack(st, K)), (T, K, r)
    want_cost = np.array([oracle.encode_tile((Y[r] * inv).astype(np.float32), K)[1]
                          for r in range(n_rows)], dtype=np.float32)
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), want_cost.view(np.uint32))
    # decode through the library matches the oracle's decode of the same words
    dec = ex.decode_rows(codes, n_rows, T, K, 1.3)
    torch.cuda.synchronize()
    want = np.stack([oracle.decode_values(oracle.unpack_states(got[r], K, T=T), 1.3)
                     for r in range(n_rows)])
    assert np.array_equal(dec.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_encode_rows_one_block_many_rows(ex):
    """All rows through one persistent block: odd count, pipeline drain."""
    T, K, n_rows = 160, 2, 9
    rng = np.random.default_rng(77)
    Y = rng.standard_normal((n_rows, T)).astype(np.float32)
    ws = torch.empty(ex.encode_workspace_min_bytes(K), dtype=torch.uint8, device=DEV)
    codes = ex.encode_rows(torch.from_numpy(Y).to(DEV), K, 1.0, ws=ws)
    torch.cuda.synchronize()
    got = codes.cpu().numpy().view(np.uint16)
    for r in range(n_rows):
        st, _, _ = oracle.encode_tile(Y[r], K)
        assert np.array_equal(got[r], oracle.pack(st, K))


# ---------------------------------------------------------------------------
# grid-and-parabola scale search
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols,K,seed", [(128, 256, 2, 61), (256, 128, 3, 62), (128, 128, 4, 63),
                                              (128, 128, 1, 64)])
def test_scale_search_matches_oracle(ex, rows, cols, K, seed):
    from oracle import scale_search as ss
    W = inputs.linear_bf16(rows, cols, seed=seed, std=0.02, outlier_frac=0.002)
    su, sv = inputs.sign_pair(rows, cols, seed)
    res = ex.scale_search(W.to(DEV), su.to(DEV), sv.to(DEV), K)
    torch.cuda.synchronize()
    R = oracle.rotate_forward(W.float().numpy(), su.numpy(), sv.numpy())
    ref = ss.grid_scale_search(R, K)
    h = res["history"].cpu().numpy()
    want = np.array(ref["coarse"] + ref["fine"] +
                    [ref["refined"] if ref["refined"] is not None else (-1.0, -1.0)])
    assert np.array_equal(h, want)
    assert float(res["g"].item()) == ref["g"]
    assert float(res["scale"].item()) == oracle.scale_for(ref["g"], ref["sigma"])[0]


def test_scale_search_full_size_properties(ex):
    from oracle import scale_search as ss
    (_, W, su, sv, K), = inputs.workload("linear4096_k2")
    res = ex.scale_search(W.to(DEV), su.to(DEV), sv.to(DEV), K)
    torch.cuda.synchronize()
    h = res["history"].cpu().numpy()
    g = float(res["g"].item())
    fine = h[19:26]
    assert 0.01 <= g <= 1.975
    # the chosen g is a fine point or the accepted refinement
    if h[26, 0] >= 0 and h[26, 1] < fine[:, 1].min():
        assert g == h[26, 0]
    else:
        assert g == fine[np.argmin(fine[:, 1]), 0]
    # the oracle's whole search on the same matrix: every (g, MSE) point exact
    R = oracle.rotate_forward(W.float().numpy(), su.numpy(), sv.numpy())
    ref = ss.grid_scale_search(R, K)
    want = np.array(ref["coarse"] + ref["fine"] +
                    [ref["refined"] if ref["refined"] is not None else (-1.0, -1.0)])
    assert np.array_equal(h, want)
    assert g == ref["g"]


# ---------------------------------------------------------------------------
# block LDL factorisation and LDLQ error feedback
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,seed", [(16, 1), (48, 2), (256, 3), (1024, 4)])
def test_block_ldl_matches_oracle(ex, n, seed):
    from oracle import ldlq as OL
    H = inputs.spd_hessian(n, seed)
    M, a = ex.block_ldl(H.to(DEV))
    Mo, ao, _ = OL.block_ldl(H.numpy())
    assert a == ao == 0
    assert np.array_equal(M.cpu().numpy(), Mo)


def test_block_ldl_damping_retries_and_failure(ex):
    from oracle import ldlq as OL
    n = 64
    eigs = np.linspace(0.5, 2.0, n)
    for need in (1, 3):
        e = eigs.copy()
        e[0] = -(need - 0.5) * 2 * 0.01 * e.mean()    # half a damping step short
        e[0] = -(need - 0.5) * 2 * 0.01 * e.mean()    # of `need` retries
        H = inputs.spectral_hessian(n, e, seed=5)
        M, a = ex.block_ldl(H.to(DEV))
        Mo, ao, _ = OL.block_ldl(H.numpy())
        assert a == ao == need
        assert np.array_equal(M.cpu().numpy(), Mo)
    e = eigs.copy()
    e[0] = -1.0
    H = inputs.spectral_hessian(n, e, seed=6)
    with pytest.raises(ex.Exl3Error) as err:
        ex.block_ldl(H.to(DEV))
    assert err.value.status == 6
    # the library stays usable after the failure
    M, a = ex.block_ldl(inputs.spd_hessian(n, 1).to(DEV))
    assert a == 0


@pytest.mark.parametrize("n,cols,K,seed", [(256, 256, 2, 31), (128, 512, 3, 32), (192, 64, 4, 33),
                                           (128, 128, 1, 34), (32, 16, 2, 35), (512, 1024, 2, 36)])
def test_ldlq_matches_oracle(ex, n, cols, K, seed):
    from oracle import ldlq as OL
    H = inputs.spd_hessian(n, seed, rho=0.95)
    Mo, _, _ = OL.block_ldl(H.numpy())
    R = inputs.iid_f32(n, cols, seed + 100)
    s = float(np.float32(oracle.rms(R.numpy())))
    M, _ = ex.block_ldl(H.to(DEV))
    res = ex.ldlq(R.to(DEV), M, K, s)
    torch.cuda.synchronize()
    ref = OL.ldlq(R.numpy(), Mo, K, s)
    assert np.array_equal(res["codes"].cpu().numpy().view(np.uint16), ref["codes"])
    assert np.array_equal(res["Q"].cpu().numpy(), ref["Q"])


def test_ldlq_small_workspace_and_no_q(ex):
    from oracle import ldlq as OL
    n, cols, K = 96, 256, 2
    H = inputs.spd_hessian(n, 41, rho=0.95)
    Mo, _, _ = OL.block_ldl(H.numpy())
    R = inputs.iid_f32(n, cols, 42)
    s = 0.75
    M, _ = ex.block_ldl(H.to(DEV))
    fixed = ex.ldlq_workspace_bytes(n, cols, K) - 16 * ex.encode_workspace_min_bytes(K)
    ws = torch.empty(fixed + ex.encode_workspace_min_bytes(K), dtype=torch.uint8, device=DEV)
    res = ex.ldlq(R.to(DEV), M, K, s, want_q=False, ws=ws)
    torch.cuda.synchronize()
    ref = OL.ldlq(R.numpy(), Mo, K, s)
    assert res["Q"] is None
    assert np.array_equal(res["codes"].cpu().numpy().view(np.uint16), ref["codes"])


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_ldlq_launches_straddle_span_rows(ex, K):
    """A workspace of five encode blocks on a 16-tile-wide matrix: each launch codes
    5 tiles (K >= 3: 10, a pair per block), so launches start in the middle of a span
    row and cover the end of one row and the start of the next, and the target and
    code rings wrap; codes and Q bit-exact against the oracle."""
    from oracle import ldlq as OL
    n, cols = 128, 256
    H = inputs.spd_hessian(n, 60 + K, rho=0.95)
    Mo, _, _ = OL.block_ldl(H.numpy())
    R = inputs.iid_f32(n, cols, 70 + K)
    s = float(np.float32(oracle.rms(R.numpy())))
    M, _ = ex.block_ldl(H.to(DEV))
    emin = ex.encode_workspace_min_bytes(K)
    fixed = ex.ldlq_workspace_bytes(n, cols, K) - 16 * emin
    ws = torch.empty(fixed + 5 * emin, dtype=torch.uint8, device=DEV)
    res = ex.ldlq(R.to(DEV), M, K, s, ws=ws)
    torch.cuda.synchronize()
    ref = OL.ldlq(R.numpy(), Mo, K, s)
    assert np.array_equal(res["codes"].cpu().numpy().view(np.uint16), ref["codes"])
    assert np.array_equal(res["Q"].cpu().numpy(), ref["Q"])


def test_ldlq_full_size_properties(ex):
    """4096 x 4096 K=2 with a 4096-channel synthetic Hessian: the factor is
    bit-exact against the oracle's (all 16.8 M entries) and block-diagonalises
    H; the two bottom spans (which read nothing above them) match the oracle's
    LDLQ of R's bottom 32 rows with M's bottom-right 32 x 32 block; the feedback
    lowers the Hessian-weighted error against plain coding."""
    from oracle import ldlq as OL
    n, cols, K = 4096, 4096, 2
    Hc = inputs.spd_hessian(n, 50, rho=0.95)
    H = Hc.to(DEV)
    M, a = ex.block_ldl(H)
    assert a == 0
    Mo, ao, _ = OL.block_ldl(Hc.numpy())
    assert ao == 0
    assert np.array_equal(M.cpu().numpy(), Mo)
    U = M.double() + torch.eye(n, dtype=torch.float64, device=DEV)
    Y = torch.linalg.solve_triangular(U, H, upper=False)
    Z = torch.linalg.solve_triangular(U, Y.T.contiguous(), upper=False)   # U^-1 H U^-T
    blk = torch.zeros(n, n, dtype=torch.bool, device=DEV)
    for b in range(n // 16):
        blk[16 * b:16 * b + 16, 16 * b:16 * b + 16] = True
    assert Z[~blk].abs().max().item() <= 1e-4 * Z[blk].abs().max().item()
    R = inputs.iid_f32(n, cols, 51)
    s = float(np.float32(oracle.rms(R.numpy())))
    Rd = R.to(DEV)
    res = ex.ldlq(Rd, M, K, s)
    torch.cuda.synchronize()
    bottom = res["codes"][-1:].cpu().numpy().view(np.uint16).reshape(-1, 16 * K)
    want, _ = _oracle_codes(R.numpy()[n - 16:], K, float(np.float32(1.0) / np.float32(s)))
    assert np.array_equal(bottom, want)
    ref = OL.ldlq(R.numpy()[n - 32:], Mo[n - 32:, n - 32:], K, s)
    assert np.array_equal(res["codes"][-2:].cpu().numpy().view(np.uint16), ref["codes"])
    assert np.array_equal(res["Q"][n - 32:].cpu().numpy(), ref["Q"])
    plain = ex.ldlq(Rd, torch.zeros_like(M), K, s)
    E1 = (Rd - res["Q"]).double()
    E0 = (Rd - plain["Q"]).double()
    l1 = ((H @ E1) * E1).sum().item()
    l0 = ((H @ E0) * E0).sum().item()
    assert l1 < 0.8 * l0


# ---------------------------------------------------------------------------
# output-channel regularisation
# ---------------------------------------------------------------------------

def _reg_case(rows, cols, seed, kind):
    g = np.random.default_rng(seed)
    W = inputs.linear_bf16(rows, cols, seed=seed, std=0.02, outlier_frac=0.001)
    W = (W.float() * torch.from_numpy(g.uniform(0.05, 4.0, cols).astype(np.float32))).to(torch.bfloat16)
    h = inputs.hessian_diag(rows, seed).numpy().copy()
    if kind == "spiky":
        h[::40] *= 1e4
    sv = inputs.signs(cols, seed + 2)
    return W, torch.from_numpy(h), sv


@pytest.mark.parametrize("rows,cols,seed,kind,apply_out", [
    (256, 384, 61, "flat", -1), (256, 384, 62, "spiky", -1), (128, 64, 63, "flat", 0),
    (512, 16, 64, "spiky", 1), (100, 33, 65, "flat", -1), (7, 5, 66, "flat", -1),
    (20000, 16, 67, "spiky", -1)])      # 20000 rows: the sort runs in global memory
def test_regularize_matches_oracle(ex, rows, cols, seed, kind, apply_out):
    from oracle import regularize as OR
    W, h, sv = _reg_case(rows, cols, seed, kind)
    W[:, 3 % cols] = 0
    r = ex.regularize(W.to(DEV), h.to(DEV), sv.to(DEV), apply_out=apply_out)
    torch.cuda.synchronize()
    ref = OR.regularize(W.float().numpy(), h.numpy(), sv.numpy(), apply_out=apply_out)
    info = r["info"].cpu().numpy()
    assert info[0] == ref["skew"]
    assert bool(info[1]) == ref["apply_out"] and not info[2]
    assert info[3] == ref["rms"]
    if apply_out < 0 and rows >= 100:      # with 7 rows the top 2 % is one channel
        assert ref["apply_out"] == (kind == "flat")
    assert np.array_equal(r["sv_out"].cpu().numpy(), ref["sv_out"])
    assert np.array_equal(r["W_out"].cpu().numpy(), ref["W_out"])


def test_regularize_extreme_bf16_magnitudes(ex):
    """bf16 values whose squares leave fp32's normal range (tiny, subnormal and
    huge) take the binary64 square: S_c still matches the oracle exactly."""
    from oracle import regularize as OR
    vals = torch.tensor([1e-30, 3e-39, 1e-20, 0.5, 3e25, -2e30, 7.0, 0.0], dtype=torch.float32)
    W = vals.repeat(64, 4).reshape(64, 32).to(torch.bfloat16)
    h = torch.ones(64)
    sv = torch.ones(32)
    r = ex.regularize(W.to(DEV), h.to(DEV), sv.to(DEV), apply_out=1)
    torch.cuda.synchronize()
    ref = OR.regularize(W.float().numpy(), h.numpy(), sv.numpy(), apply_out=1)
    assert np.array_equal(r["sv_out"].cpu().numpy(), ref["sv_out"])
    assert np.array_equal(r["W_out"].cpu().numpy(), ref["W_out"])


def test_regularize_all_zero_and_in_place(ex):
    from oracle import regularize as OR
    Z = torch.zeros(64, 48, device=DEV)
    r = ex.regularize(Z, torch.ones(64, device=DEV), torch.ones(48, device=DEV))
    info = r["info"].cpu().numpy()
    assert info[2] == 1.0 and not r["sv_out"].any().item() and not r["W_out"].any().item()
    W, h, sv = _reg_case(256, 128, 70, "flat")
    Wf = W.float().to(DEV)
    r = ex.regularize(Wf, h.to(DEV), sv.to(DEV), W_out=Wf)
    torch.cuda.synchronize()
    ref = OR.regularize(W.float().numpy(), h.numpy(), sv.numpy())
    assert np.array_equal(Wf.cpu().numpy(), ref["W_out"])


def test_regularize_full_size_and_round_trip(ex):
    """12288 x 4096 bf16 (a 12288-input projection) against the oracle, then the
    chain regularise -> quantize -> decode -> inverse rotation with sv_out."""
    from oracle import regularize as OR
    W, h, sv = _reg_case(12288, 4096, 71, "flat")
    r = ex.regularize(W.to(DEV), h.to(DEV), sv.to(DEV))
    torch.cuda.synchronize()
    ref = OR.regularize(W.float().numpy(), h.numpy(), sv.numpy())
    assert np.array_equal(r["sv_out"].cpu().numpy(), ref["sv_out"])
    assert np.array_equal(r["W_out"].cpu().numpy(), ref["W_out"])
    # round trip on a smaller slab, compared with the oracle's chain
    Ws, hs, svs = _reg_case(256, 512, 72, "flat")
    su = inputs.signs(256, 73)
    r = ex.regularize(Ws.to(DEV), hs.to(DEV), svs.to(DEV))
    q = ex.quantize(r["W_out"], su.to(DEV), svs.to(DEV), 3, 1.0)
    s = float(q["scale"].item())
    Qd = ex.decode_tiles(q["codes"], 256, 512, 3, s)
    What = ex.rotate(Qd, su.to(DEV), r["sv_out"], inverse=True)
    torch.cuda.synchronize()
    ref = OR.regularize(Ws.float().numpy(), hs.numpy(), svs.numpy())
    Rn = oracle.rotate_forward(ref["W_out"], su.numpy(), svs.numpy())
    assert s == oracle.scale_for(1.0, oracle.rms(Rn))[0]
    codes_o = oracle.codes_from_states(oracle.encode_matrix(Rn, 3, 1.0 / np.float32(s))[0], 256, 512, 3)
    Qo = oracle.decode_matrix(codes_o, 256, 512, 3, s)
    What_o = oracle.rotate_inverse(Qo, su.numpy(), ref["sv_out"])
    assert np.array_equal(What.cpu().numpy(), What_o)
    Wd = Ws.float().numpy().astype(np.float64)
    rel = np.sum((What_o - Wd) ** 2) / np.sum(Wd ** 2)
    assert rel < 0.05          # K=3 keeps the relative error near 2^-6


# ---------------------------------------------------------------------------
# non-finite weights are rejected on the device
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 2])
def test_quantize_rejects_non_finite_weight(ex, K):
    import math
    W = inputs.linear_bf16(256, 256, seed=80)
    su, sv = (t.to(DEV) for t in inputs.sign_pair(256, 256, 80))
    for bad in (float("nan"), float("inf")):
        Wb = W.clone()
        Wb[17, 33] = bad
        codes = torch.full((16, 16, 16 * K), 0x1234, dtype=torch.int16, device=DEV)
        r = ex.quantize(Wb.to(DEV), su, sv, K, 1.0, codes=codes)
        torch.cuda.synchronize()
        assert math.isnan(r["scale"].item()) and math.isnan(r["mse"].item())
        assert not math.isfinite(r["sigma"].item())
        assert bool((codes == 0x1234).all().item())          # no tile was coded
    # the context stays usable: a clean call matches the oracle
    r = ex.quantize(W.to(DEV), su, sv, K, 1.0)
    torch.cuda.synchronize()
    R = oracle.rotate_forward(W.float().numpy(), su.cpu().numpy(), sv.cpu().numpy())
    s, inv = oracle.scale_for(1.0, oracle.rms(R))
    assert float(r["scale"].item()) == s
    want, _ = _oracle_codes(R, K, inv)
    assert np.array_equal(_np_codes(r["codes"], K), want)


# ---------------------------------------------------------------------------
# CUDA graph capture: the quantize chain and the GSS enqueue no host syncs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 2])
def test_quantize_and_gss_replay_from_cuda_graph(ex, K):
    rows, cols = 256, 256
    W = inputs.linear_bf16(rows, cols, seed=90)
    su, sv = (t.to(DEV) for t in inputs.sign_pair(rows, cols, 90))
    Wd = W.to(DEV)
    ws = torch.empty(ex.gss_workspace_bytes(rows, cols, K), dtype=torch.uint8, device=DEV)
    direct = ex.quantize(Wd, su, sv, K, 1.3, ws=ws)
    gdirect = ex.gss_scale(Wd, su, sv, K, 0.5, 2.0, 6, ws=ws)
    torch.cuda.synchronize()
    codes = torch.zeros_like(direct["codes"])
    gcodes = torch.zeros_like(gdirect["codes"])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        q = ex.quantize(Wd, su, sv, K, 1.3, codes=codes, ws=ws)
        gs = ex.gss_scale(Wd, su, sv, K, 0.5, 2.0, 6, best_codes=gcodes, ws=ws)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(codes, direct["codes"])
        assert float(q["mse"].item()) == float(direct["mse"].item())
        assert torch.equal(gcodes, gdirect["codes"])
        assert float(gs["g"].item()) == float(gdirect["g"].item())
        codes.zero_()
        gcodes.zero_()


def test_ldlq_scale_search_regularize_replay_from_cuda_graph(ex):
    """The other asynchronous entry points capture and replay bit for bit too
    (exl3_block_ldl reads a device flag back and is called outside the graph)."""
    n, cols, K = 128, 256, 2
    H = inputs.spd_hessian(n, 91, rho=0.95).to(DEV)
    M, _ = ex.block_ldl(H)
    R = inputs.iid_f32(n, cols, 92).to(DEV)
    W = inputs.linear_bf16(n, cols, seed=93).to(DEV)
    su, sv = (t.to(DEV) for t in inputs.sign_pair(n, cols, 93))
    h = inputs.hessian_diag(n, 94).to(DEV)
    wl = torch.empty(ex.ldlq_workspace_bytes(n, cols, K), dtype=torch.uint8, device=DEV)
    ws = torch.empty(ex.scale_search_workspace_bytes(n, cols, K), dtype=torch.uint8, device=DEV)
    wr = torch.empty(ex.regularize_workspace_bytes(n, cols), dtype=torch.uint8, device=DEV)
    d_lq = ex.ldlq(R, M, K, 0.9, ws=wl)
    d_ss = ex.scale_search(W, su, sv, K, ws=ws)
    d_rg = ex.regularize(W, h, sv, ws=wr)
    torch.cuda.synchronize()
    codes = torch.zeros_like(d_lq["codes"])
    Wout = torch.zeros_like(d_rg["W_out"])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lq = ex.ldlq(R, M, K, 0.9, codes=codes, ws=wl)
        ss = ex.scale_search(W, su, sv, K, ws=ws)
        rg = ex.regularize(W, h, sv, W_out=Wout, ws=wr)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(codes, d_lq["codes"]) and torch.equal(lq["Q"], d_lq["Q"])
    assert torch.equal(ss["history"], d_ss["history"])
    assert torch.equal(Wout, d_rg["W_out"]) and torch.equal(rg["sv_out"], d_rg["sv_out"])


def test_concurrent_streams_do_not_interfere(ex):
    """Two quantize calls (K=2 and K=1) enqueued on two streams at once, each with
    its own workspace, give the results of the same calls made one after the
    other: the library keeps no device state outside the caller's buffers."""
    mats = []
    for seed, K in ((101, 2), (102, 1)):
        W = inputs.linear_bf16(256, 256, seed=seed).to(DEV)
        su, sv = (t.to(DEV) for t in inputs.sign_pair(256, 256, seed))
        ws = torch.empty(ex.quantize_workspace_bytes(256, 256, K), dtype=torch.uint8, device=DEV)
        mats.append((W, su, sv, K, ws))
    seq = [ex.quantize(W, su, sv, K, 1.0, ws=ws) for W, su, sv, K, ws in mats]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    par = []
    for rep in range(3):
        outs = []
        for st, (W, su, sv, K, ws) in zip(streams, mats):
            with torch.cuda.stream(st):
                outs.append(ex.quantize(W, su, sv, K, 1.0, ws=ws))
        torch.cuda.synchronize()
        par.append(outs)
    for outs in par:
        for a, b in zip(outs, seq):
            assert torch.equal(a["codes"], b["codes"])
            assert float(a["mse"].item()) == float(b["mse"].item())
