"""Every tile of the full-size workloads, bit for bit against the oracle (gpu).

The oracle's results on the full matrices take hours of CPU time, so they are
stored as digests (tests/golden/full_digests.json, written by
tests/golden/make_full_digests.py from ``oracle/`` and the seeded generators
only).  Each test first checks that this host drew the same input bytes as the
host that wrote the digests, then runs the CUDA path through the C ABI in the
launch configuration the benchmark times (one persistent block per SM) and
compares:
  * sigma_R and the scale exactly, the MSE within 1e-6 relative;
  * the rotated matrix R and the reconstruction W-hat (SHA-256 of all bytes);
  * per 128-row band, the packed codes and the fp32 tile costs (a mismatch
    names the band).
Workloads: 4096x4096 bf16 K=2 with 0.1 % outliers; 12288x4096 Student-t K=4;
the seven projections of the 4096/12288 decoder layer at K=3; and the
12-evaluation golden-section search on 4096x4096 K=2, where every evaluated g
must match exactly and every evaluation's codes bit for bit (pages "EXL3 Intel
Arc Quantizer", Current Status: bit-exact CPU and GPU encoders; and
"alpha2beta/JEV-9B-EXL3-K2", section 2: golden-section scale search).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import digests as D  # noqa: E402
from exl3_trellis_weight_gb300 import inputs  # noqa: E402

REL_TOL = 1e-6
DEV = "cuda:0"
MATRIX_KEYS = ["linear4096_k2", "mlp12288_t5_k4",
               "layer4096_k3/q", "layer4096_k3/k", "layer4096_k3/v", "layer4096_k3/o",
               "layer4096_k3/gate", "layer4096_k3/up", "layer4096_k3/down"]
GSS_KEY = "gss4096_k2"


@pytest.fixture(scope="module")
def ex():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is required for -m gpu tests")
    import __graft_entry__
    __graft_entry__.build()
    import exl3_trellis_weight_gb300 as ex
    return ex


@pytest.fixture(scope="module")
def store():
    return D.load()


@pytest.fixture(autouse=True)
def _no_expired_waits(ex):
    yield
    assert ex.wait_timeouts() == 0


def _matrix(key):
    name, _, proj = key.partition("/")
    for lab, W, su, sv, K in inputs.workload(name):
        if not proj or lab == proj:
            return W, su, sv, K
    raise KeyError(key)


def _entry(store, key, W, su, sv):
    assert key in store, f"no stored oracle digests for {key}"
    e = store[key]
    assert D.input_digests(W, su, sv) == e["inputs"], \
        f"{key}: this host drew different input bytes than the host that wrote the digests"
    return e


def _compare_evaluation(ex, key, e, Wd, sud, svd, K, g):
    """quantize at relative scale g, then the rotation and an encode with tile
    costs at the same scale; compare everything the oracle stored."""
    rows, cols = Wd.shape
    q = ex.quantize(Wd, sud, svd, K, g, want_What=True)
    R = ex.rotate(Wd, sud, svd)
    scale = float(q["scale"].item())
    codes, cost = ex.encode_tiles(R, K, scale, want_cost=True)
    torch.cuda.synchronize()
    assert float(q["sigma"].item()) == D.unhex(e["sigma"]), f"{key} g={g}: sigma"
    assert scale == D.unhex(e["scale"]), f"{key} g={g}: scale"
    m, mo = float(q["mse"].item()), D.unhex(e["mse"])
    assert abs(m - mo) <= REL_TOL * mo, f"{key} g={g}: mse {m!r} vs oracle {mo!r}"
    assert D.sha(R.cpu().numpy()) == e["R"], f"{key}: rotated matrix differs"
    assert torch.equal(codes, q["codes"])
    got = D.band_digests(codes.cpu().numpy(), cost.cpu().numpy(), rows, cols, K)
    bad_codes = [b for b, (x, y) in enumerate(zip(got, e["bands"])) if x[0] != y[0]]
    bad_costs = [b for b, (x, y) in enumerate(zip(got, e["bands"])) if x[1] != y[1]]
    assert len(got) == len(e["bands"])
    assert not bad_codes, f"{key} g={g}: codes differ in 128-row bands {bad_codes}"
    assert not bad_costs, f"{key} g={g}: tile costs differ in 128-row bands {bad_costs}"
    assert D.sha(q["What"].cpu().numpy()) == e["What"], f"{key} g={g}: reconstruction differs"
    return q


def test_every_full_size_workload_has_stored_digests(store):
    missing = [k for k in MATRIX_KEYS + [GSS_KEY] if k not in store]
    assert not missing, f"run tests/golden/make_full_digests.py for {missing}"


@pytest.mark.parametrize("key", MATRIX_KEYS)
def test_full_matrix_every_tile_bit_exact(ex, store, key):
    W, su, sv, K = _matrix(key)
    e = _entry(store, key, W, su, sv)
    assert (e["rows"], e["cols"], e["K"]) == (W.shape[0], W.shape[1], K)
    Wd, sud, svd = W.to(DEV), su.to(DEV), sv.to(DEV)
    _compare_evaluation(ex, key, e, Wd, sud, svd, K, 1.0)


def test_full_gss_search_path_and_every_evaluation_bit_exact(ex, store):
    W, su, sv, K = _matrix(GSS_KEY)
    e = _entry(store, GSS_KEY, W, su, sv)
    Wd, sud, svd = W.to(DEV), su.to(DEV), sv.to(DEV)
    n = e["n_eval"]
    res = ex.gss_scale(Wd, sud, svd, K, D.unhex(e["lo"]), D.unhex(e["hi"]), n, want_history=True)
    hist = res["history"].view(n, 2).cpu().numpy()
    for i, ev in enumerate(e["evals"]):
        assert hist[i, 0] == D.unhex(ev["g"]), f"evaluation {i}: g"
        mo = D.unhex(ev["mse"])
        assert abs(hist[i, 1] - mo) <= REL_TOL * mo, f"evaluation {i}: mse"
    best_g = D.unhex(e["best_g"])
    assert float(res["g"].item()) == best_g
    assert abs(float(res["mse"].item()) - D.unhex(e["best_mse"])) <= REL_TOL * D.unhex(e["best_mse"])
    best = [ev for ev in e["evals"] if D.unhex(ev["g"]) == best_g][0]
    assert float(res["scale"].item()) == D.unhex(best["scale"])
    rows, cols = W.shape
    got = D.band_digests(res["codes"].cpu().numpy(), None, rows, cols, K)
    bad = [b for b, (x, y) in enumerate(zip(got, best["bands"])) if x[0] != y[0]]
    assert not bad, f"codes at the chosen g differ in 128-row bands {bad}"
    # every evaluation of the search, each a full quantization, bit for bit
    for ev in e["evals"]:
        _compare_evaluation(ex, GSS_KEY, ev, Wd, sud, svd, K, D.unhex(ev["g"]))
