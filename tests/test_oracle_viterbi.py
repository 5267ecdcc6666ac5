"""Pins for the oracle's Viterbi search by exhaustive enumeration (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture items 1 and 4:
forward add-compare-select over 2^(L-K) tracked states with candidates
sigma = (k << (L-K)) | e and predecessor sigma >> K, strict-< first-branch
tie-breaking, and the two-pass tail-biting closure.  The oracle is written for
any state width L and length T, so small trellises can be enumerated.
"""
import itertools

import numpy as np
import pytest

import oracle
from tests.brute import all_paths, path_costs, lexmin_from_end

CASES = [(4, 1, 6), (4, 2, 4), (6, 2, 6), (6, 3, 4), (8, 2, 5), (8, 3, 4), (6, 1, 8)]


def _rand_case(L, K, T, seed, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        cb = rng.integers(-3, 4, size=1 << L).astype(np.float32)
        y = rng.integers(-3, 4, size=T).astype(np.float32)
    else:
        cb = rng.standard_normal(1 << L).astype(np.float32)
        y = rng.standard_normal(T).astype(np.float32)
    return y, cb


@pytest.mark.parametrize("L,K,T", CASES)
@pytest.mark.parametrize("seed", [0, 1])
def test_free_start_cost_equals_enumeration(L, K, T, seed):
    y, cb = _rand_case(L, K, T, seed)
    dec, fc, pen = oracle.viterbi_forward(y, L, K, cb, constrained=False)
    paths = all_paths(L, K, T)
    costs = path_costs(paths, y, cb)
    # every full end state: fl(cost_{T-2}(s>>K) + q_{T-1}(s)) equals the best path into s
    mask = (1 << L) - 1
    for s in range(1 << L):
        sel = paths[:, -1] == s
        d = np.float32(y[-1] - cb[s])
        mine = np.float32(pen[s >> K] + np.float32(d * d))
        assert mine == costs[sel].min()
    # tracked final row = min over the group of full states sharing the low bits
    for g in range(1 << (L - K)):
        sel = (paths[:, -1] & ((1 << (L - K)) - 1)) == g
        assert fc[g] == costs[sel].min()
    # the traced path from the final argmin has the minimal cost
    s_star = oracle.final_argmin(dec[-1], fc, L, K)
    st = oracle.traceback(dec, L, K, T - 1, 0, s_star)
    assert path_costs(st[None, :].astype(np.int64), y, cb)[0] == costs.min()


@pytest.mark.parametrize("L,K,T", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_ties_resolve_to_lexicographically_smallest_from_end(L, K, T, seed):
    # integer codebook and targets: all sums are exact, so ties are real ties
    y, cb = _rand_case(L, K, T, seed, integer=True)
    dec, fc, _ = oracle.viterbi_forward(y, L, K, cb)
    s_star = oracle.final_argmin(dec[-1], fc, L, K)
    st = oracle.traceback(dec, L, K, T - 1, 0, s_star)
    paths = all_paths(L, K, T)
    costs = path_costs(paths, y, cb)
    best = paths[costs == costs.min()]
    assert np.array_equal(st.astype(np.int64), best[lexmin_from_end(best)])


@pytest.mark.parametrize("L,K,T", CASES)
@pytest.mark.parametrize("seed", [0, 3])
def test_constrained_start_and_forced_end_equal_enumeration(L, K, T, seed):
    rng = np.random.default_rng(100 + seed)
    y, cb = _rand_case(L, K, T, seed)
    pre = int(rng.integers(0, 1 << L))
    dec, fc, pen = oracle.viterbi_forward(y, L, K, cb, constrained=True, pre_state=pre)
    paths = all_paths(L, K, T, start_pred=pre)
    costs = path_costs(paths, y, cb)
    for end in range(1 << L):
        sel = paths[:, -1] == end
        d = np.float32(y[-1] - cb[end])
        mine = np.float32(pen[end >> K] + np.float32(d * d))
        if not sel.any():
            assert np.isinf(mine)
            continue
        assert mine == costs[sel].min()
        if np.isfinite(mine):
            st = oracle.traceback(dec, L, K, T - 1, 0, end)
            assert path_costs(st[None, :].astype(np.int64), y, cb)[0] == mine
            assert (st[0] >> K) == (pre & ((1 << (L - K)) - 1))


@pytest.mark.parametrize("L,K,T", [(4, 1, 6), (4, 2, 4), (6, 2, 6), (6, 3, 4), (8, 2, 6)])
def test_two_pass_encode_ring_closure_and_bound(L, K, T):
    for seed in range(4):
        y, cb = _rand_case(L, K, T, seed)
        st, cost, end = oracle.encode_tile(y, K, L=L, cb=cb)
        lowmask = (1 << (L - K)) - 1
        # ring closure: last state is end_state, first state's predecessor is end_state
        assert st[-1] == end
        assert (st[0] >> K) == (end & lowmask)
        # consecutive states share L-K bits
        for t in range(1, T):
            assert (st[t] >> K) == (st[t - 1] & lowmask)
        # reported cost is the left-to-right fp32 sum along the path
        assert path_costs(st[None, :].astype(np.int64), y, cb)[0] == np.float32(cost)
        # never better than the best tail-biting (circular) path
        paths = all_paths(L, K, T)
        circ = (paths[:, 0] >> K) == (paths[:, -1] & lowmask)
        assert np.float32(cost) >= path_costs(paths[circ], y, cb).min()
        # pass 1 alone: end_state is on an optimal free path of the rolled targets
        yr = np.roll(y, -(T // 2))
        dec, fc, _ = oracle.viterbi_forward(yr, L, K, cb)
        s_star = oracle.final_argmin(dec[-1], fc, L, K)
        p1 = oracle.traceback(dec, L, K, T - 1, T // 2 - 1, s_star)
        assert p1[T // 2 - 1] == end


def test_planted_mistakes_are_caught_by_enumeration():
    """A wrong predecessor index or a non-strict tie rule changes the result on
    some small case; the enumeration above would flag it."""
    L, K, T = 6, 2, 6
    found_tie_case = False
    for seed in range(40):
        y, cb = _rand_case(L, K, T, seed, integer=True)
        paths = all_paths(L, K, T)
        costs = path_costs(paths, y, cb)
        best = paths[costs == costs.min()]
        want = best[lexmin_from_end(best)]
        # "last branch wins ties" variant, written here directly
        G, NK = 1 << (L - K), 1 << K
        prev = np.zeros(G, np.float32)
        decs = []
        for t in range(T):
            cur = np.empty(G, np.float32)
            dk = np.empty(G, np.int64)
            for g in range(G):
                best_c, best_k = None, 0
                for k in range(NK):
                    sig = (k << (L - K)) | g
                    c = np.float32(prev[sig >> K] + np.float32((y[t] - cb[sig]) ** 2))
                    if best_c is None or c <= best_c:
                        best_c, best_k = c, k
                cur[g], dk[g] = best_c, best_k
            decs.append(dk)
            prev = cur
        if len(best) > 1:
            g_star = int(np.argmin(prev))
            s = (int(decs[-1][g_star]) << (L - K)) | g_star
            wrong = [s]
            for t in range(T - 1, 0, -1):
                g = s >> K
                s = (int(decs[t - 1][g]) << (L - K)) | g
                wrong.append(s)
            if not np.array_equal(np.array(wrong[::-1]), want):
                found_tie_case = True
                break
    assert found_tie_case


def test_random_trellises_match_enumeration():
    """Randomised breadth for the enumeration pins: random state widths, bits per
    step, lengths, codebooks (continuous or small integers, so ties occur) and
    targets; the oracle's tracked final row equals the best enumerated path into
    every group, and its traced path has the minimal cost."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(L=st.integers(3, 6), K=st.integers(1, 3), T=st.integers(2, 6),
               seed=st.integers(0, 2**31 - 1), integer=st.booleans())
    def check(L, K, T, seed, integer):
        hyp.assume(K < L and (1 << L) * (1 << (K * (T - 1))) <= 1 << 14)
        rng = np.random.default_rng(seed)
        if integer:
            cb = rng.integers(-3, 4, 1 << L).astype(np.float32)
            y = rng.integers(-3, 4, T).astype(np.float32)
        else:
            cb = rng.standard_normal(1 << L).astype(np.float32)
            y = rng.standard_normal(T).astype(np.float32)
        dec, fc, pen = oracle.viterbi_forward(y, L, K, cb, constrained=False)
        paths = all_paths(L, K, T)
        costs = path_costs(paths, y, cb)
        low = (1 << (L - K)) - 1
        for g in range(1 << (L - K)):
            assert fc[g] == costs[(paths[:, -1] & low) == g].min()
        s_star = oracle.final_argmin(dec[-1], fc, L, K)
        stt = oracle.traceback(dec, L, K, T - 1, 0, s_star)
        assert path_costs(stt[None, :].astype(np.int64), y, cb)[0] == costs.min()

    check()
