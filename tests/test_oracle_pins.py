"""Pins for the float64 oracle: each function is checked against something other
than itself -- values a page prints, closed forms, invariants, brute force on tiny
inputs, and independent library routines (torch SDPA in float64, scipy).

Sources (cited by page title and section):
  * "手写 Flash Attention：从算法原理到高性能实现", section 2.2 "Online Softmax"
    (the worked row [2, 1, 5, 3], block 2) -- tests/golden/worked_row_2153.json;
  * CS336 lecture 5 "05_flash_attention.py", part 1 (online softmax demo: randn(10)*5,
    block 3) and part 2 (flash forward demo: n=100, d=32, blocks 16x24, float64);
  * "Flash Attention" (blog.cyberangel.work), sections "Online Softmax" and "平行化"
    (the merge operator is associative and commutative).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_row_2153.json")


def _sdpa64(Q, K, V, scale, causal):
    """torch's own scaled_dot_product_attention in float64 on the CPU (library routine).

    With is_causal and Nq != Nk torch aligns the mask top-left (query i sees key j <= i),
    the reading the oracle takes."""
    q, k, v = (torch.from_numpy(np.asarray(a, np.float64)) for a in (Q, K, V))
    return F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale).numpy()


def _lse64(Q, K, scale, causal):
    S = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    if causal:
        Nq, Nk = S.shape[-2:]
        S = np.where(np.arange(Nk)[None, :] > np.arange(Nq)[:, None], -np.inf, S)
    return scipy.special.logsumexp(S, axis=-1)


# --------------------------------------------------------------------------- worked row
def test_worked_row_intermediates(oracle_mod):
    g = json.load(open(GOLDEN))
    x, block, pr = g["x"], g["block"], g["printed"]
    tol = 0.5 * 10 ** (-g["printed_decimals"]) + 1e-12
    m, l, mt, lt = oracle_mod.online_softmax(x, block)
    assert len(mt) == 2
    assert mt[0] == pr["block1_max"]
    assert abs(lt[0] - pr["block1_sum"]) <= tol
    assert mt[1] == pr["block2_new_max"] == m
    rebased = lt[0] * math.exp(mt[0] - mt[1])
    assert abs(rebased - pr["block1_sum_rebased"]) <= tol
    assert abs((lt[1] - rebased) - pr["block2_sum"]) <= tol
    assert abs(l - pr["total_sum"]) <= tol
    # block-local softmax of the first block as printed
    loc = np.exp(np.array(x[:2]) - mt[0]) / lt[0]
    assert np.all(np.abs(loc - pr["block1_local_softmax"]) <= tol)


def test_worked_row_final_softmax_and_errata(oracle_mod):
    """The attention oracle on a row whose scores are exactly [2,1,5,3] (d=4, scale=1,
    V = identity, so O is the probability row)."""
    g = json.load(open(GOLDEN))
    x = np.array(g["x"])
    Q = np.zeros((1, 1, 1, 4)); Q[0, 0, 0, 0] = 1.0
    K = np.zeros((1, 1, 4, 4)); K[0, 0, :, 0] = x
    V = np.eye(4)[None, None]
    O, L = oracle_mod.attention(Q, K, V, 1.0, False)
    p = O[0, 0, 0]
    # closed form of this row
    e = [math.exp(v - 5.0) for v in g["x"]]
    exact = [v / sum(e) for v in e]
    assert np.allclose(p, exact, rtol=0, atol=1e-15)
    assert np.allclose(p, [0.041371, 0.015219, 0.830953, 0.112457], atol=5e-7)
    assert abs(L[0, 0, 0] - (5.0 + math.log(sum(e)))) < 1e-14
    assert abs(L[0, 0, 0] - 5.18518) < 5e-6
    tol = 0.5 * 10 ** (-g["printed_decimals"]) + 1e-12
    for k, ok in enumerate(g["final_softmax_entries_correct_on_page"]):
        matches = abs(p[k] - g["printed"]["final_softmax"][k]) <= tol
        assert matches == ok, f"entry {k}: oracle {p[k]:.6f}, page {g['printed']['final_softmax'][k]}"


# --------------------------------------------------------------------------- online softmax
@pytest.mark.parametrize("block", [1, 2, 3, 4, 7, 10, 64])
def test_online_softmax_matches_logsumexp(oracle_mod, block):
    rng = np.random.default_rng(0)
    x = rng.standard_normal(10) * 5          # the CS336 demo's distribution
    m, l, _, _ = oracle_mod.online_softmax(x, block)
    assert m == x.max()
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-12
    # softmax from the statistics equals scipy's softmax
    assert np.allclose(np.exp(x - m) / l, scipy.special.softmax(x), rtol=1e-13, atol=0)


def test_online_softmax_large_values_no_overflow(oracle_mod):
    """Entries above 709 overflow exp() in double without the max shift."""
    x = np.array([1000.0, 999.0, 1001.0, -5.0, 998.5])
    m, l, _, _ = oracle_mod.online_softmax(x, 2)
    assert math.isfinite(l)
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-12


# --------------------------------------------------------------------------- merge operator
def test_merge_two_singletons_closed_form(oracle_mod):
    # (x1,1,v1) (+) (x2,1,v2): m = max, d = 1 + e^{-|x1-x2|}, o = v_max + e^{-|x1-x2|} v_min
    v1, v2 = np.array([1.0, -2.0, 0.5]), np.array([3.0, 4.0, -1.0])
    m, d, o = oracle_mod.merge((0.3, 1.0, v1), (1.7, 1.0, v2))
    w = math.exp(0.3 - 1.7)
    assert m == 1.7
    assert abs(d - (1.0 + w)) < 1e-15
    assert np.allclose(o, v2 + w * v1, rtol=0, atol=1e-15)
    # commutative
    m2, d2, o2 = oracle_mod.merge((1.7, 1.0, v2), (0.3, 1.0, v1))
    assert (m2, d2) == (m, d) and np.array_equal(o2, o)


def test_merge_identity(oracle_mod):
    v = np.array([0.25, -1.5])
    st = (2.5, 3.0, v)
    for a, b in [((-np.inf, 0.0, np.zeros(2)), st), (st, (-np.inf, 0.0, np.zeros(2)))]:
        m, d, o = oracle_mod.merge(a, b)
        assert m == 2.5 and d == 3.0 and np.array_equal(o, v)


@pytest.mark.parametrize("causal", [False, True])
def test_merge_any_blocking_any_order_equals_definition(oracle_mod, causal):
    """Cut a row's keys into blocks of every size, merge the block states in random
    tree orders: (m, d, o~) is the same, and o~/d, m + ln d equal the attention oracle."""
    rng = np.random.default_rng(7)
    Nk, d, Nq = 100, 32, 100
    Q = rng.standard_normal((1, 1, Nq, d))
    K = rng.standard_normal((1, 1, Nk, d))
    V = rng.standard_normal((1, 1, Nk, d))
    scale = 1 / math.sqrt(d)
    O, L = oracle_mod.attention(Q, K, V, scale, causal)
    for i in [0, 1, 37, 99]:
        ref = None
        for bs in [1, 2, 3, 16, 24, 128]:
            states = [oracle_mod.block_state(Q[0, 0, i], K[0, 0], V[0, 0], i, j0, min(Nk, j0 + bs),
                                             scale, causal) for j0 in range(0, Nk, bs)]
            for trial in range(3):
                work = list(states)
                rng.shuffle(work)
                while len(work) > 1:          # random merge tree
                    a = work.pop(rng.integers(len(work)))
                    b = work.pop(rng.integers(len(work)))
                    work.append(oracle_mod.merge(a, b))
                m, den, o = work[0]
                if ref is None:
                    ref = (m, den, o)
                assert m == ref[0]
                assert abs(den - ref[1]) <= 1e-12 * abs(ref[1])
                assert np.allclose(o, ref[2], rtol=1e-12, atol=1e-12)
                assert np.allclose(o / den, O[0, 0, i], rtol=1e-12, atol=1e-13)
                assert abs(m + math.log(den) - L[0, 0, i]) < 1e-12


# --------------------------------------------------------------------------- attention definition
@pytest.mark.parametrize("shape,causal", [
    ((1, 1, 100, 100, 32), False),     # CS336 part 2 demo shape (float64, n=100, d=32)
    ((1, 1, 100, 100, 32), True),
    ((2, 4, 512, 512, 64), False),     # the P4 test shape B=2,H=4,N=512,D=64
    ((2, 4, 512, 512, 64), True),
    ((3, 2, 37, 53, 16), False),       # cross attention, Nq != Nk
    ((3, 2, 53, 37, 16), True),        # causal, top-left aligned, Nq > Nk
    ((1, 2, 29, 61, 8), True),         # causal, Nq < Nk
])
def test_attention_matches_torch_sdpa_float64(oracle_mod, shape, causal):
    B, H, Nq, Nk, d = shape
    rng = np.random.default_rng(sum(shape) + causal)
    Q = rng.standard_normal((B, H, Nq, d))
    K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d))
    scale = 1 / math.sqrt(d)
    O, L = oracle_mod.attention(Q, K, V, scale, causal)
    assert np.allclose(O, _sdpa64(Q, K, V, scale, causal), rtol=1e-12, atol=1e-12)
    assert np.allclose(L, _lse64(Q, K, scale, causal), rtol=1e-13, atol=1e-12)


def test_attention_brute_force_tiny(oracle_mod):
    """Pure-Python naive softmax (no max shift, exact fsum) on tiny rows, both masks,
    several scales (including 0: uniform attention)."""
    rng = np.random.default_rng(11)
    for (Nq, Nk, d) in [(1, 1, 1), (3, 5, 2), (5, 3, 4), (8, 8, 3)]:
        for causal in (False, True):
            for scale in (0.0, 0.37, 1.0):
                Q = rng.standard_normal((1, 1, Nq, d))
                K = rng.standard_normal((1, 1, Nk, d))
                V = rng.standard_normal((1, 1, Nk, d))
                O, L = oracle_mod.attention(Q, K, V, scale, causal)
                for i in range(Nq):
                    vis = [j for j in range(Nk) if not (causal and j > i)]
                    w = [math.exp(scale * math.fsum(Q[0, 0, i, c] * K[0, 0, j, c] for c in range(d)))
                         for j in vis]
                    den = math.fsum(w)
                    for c in range(d):
                        o = math.fsum(w[t] * V[0, 0, j, c] for t, j in enumerate(vis)) / den
                        assert abs(O[0, 0, i, c] - o) < 1e-13
                    assert abs(L[0, 0, i] - math.log(den)) < 1e-13


def test_causal_row0_is_v0(oracle_mod):
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((2, 3, 40, 16)); K = rng.standard_normal((2, 3, 40, 16))
    V = rng.standard_normal((2, 3, 40, 16))
    scale = 0.25
    O, L = oracle_mod.attention(Q, K, V, scale, True)
    assert np.array_equal(O[:, :, 0], V[:, :, 0])
    # L_0 = scale * <q_0, k_0> (one visible key): same summation order as a dot product
    dots = np.einsum("bhd,bhd->bh", Q[:, :, 0], K[:, :, 0])
    assert np.allclose(L[:, :, 0], scale * dots, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_is_uniform_average(oracle_mod, causal):
    rng = np.random.default_rng(5)
    Nq, Nk, d = 30, 45, 8
    Q = np.zeros((1, 2, Nq, d))
    K = rng.standard_normal((1, 2, Nk, d)); V = rng.standard_normal((1, 2, Nk, d))
    O, L = oracle_mod.attention(Q, K, V, 0.5, causal)
    for i in range(Nq):
        n = min(i + 1, Nk) if causal else Nk
        assert np.allclose(O[:, :, i], V[:, :, :n].mean(axis=2), rtol=0, atol=1e-14)
        assert np.allclose(L[:, :, i], math.log(n), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value(oracle_mod):
    rng = np.random.default_rng(9)
    Nq, Nk, d = 4, 16, 8
    Q = rng.standard_normal((1, 1, Nq, d)); K = rng.standard_normal((1, 1, Nk, d)) * 0.01
    V = rng.standard_normal((1, 1, Nk, d))
    for i in range(Nq):
        K[0, 0, 3 + i] = 60.0 * Q[0, 0, i]     # key 3+i dominates row i by a wide margin
    O, _ = oracle_mod.attention(Q, K, V, 1.0, False)
    for i in range(Nq):
        assert np.allclose(O[0, 0, i], V[0, 0, 3 + i], atol=1e-9)


def test_probs_rows_sum_to_one_and_match_softmax(oracle_mod):
    rng = np.random.default_rng(13)
    Nq, Nk, d = 33, 47, 16
    Q = rng.standard_normal((Nq, d)) * 2; K = rng.standard_normal((Nk, d)) * 2
    for causal in (False, True):
        P = oracle_mod.probs(Q, K, 0.25, causal)
        assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        S = 0.25 * (Q @ K.T)
        if causal:
            S = np.where(np.arange(Nk)[None, :] > np.arange(Nq)[:, None], -np.inf, S)
            assert np.all(P[np.arange(Nk)[None, :] > np.arange(Nq)[:, None]] == 0.0)
        assert np.allclose(P, scipy.special.softmax(S, axis=1), rtol=1e-13, atol=1e-16)


def test_output_in_convex_hull_and_permutation_invariance(oracle_mod):
    rng = np.random.default_rng(17)
    B, H, Nq, Nk, d = 1, 2, 20, 31, 8
    Q = rng.standard_normal((B, H, Nq, d)); K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d))
    O, L = oracle_mod.attention(Q, K, V, 0.3, False)
    lo, hi = V.min(axis=2, keepdims=True), V.max(axis=2, keepdims=True)
    assert np.all(O >= lo - 1e-14) and np.all(O <= hi + 1e-14)
    perm = rng.permutation(Nk)
    O2, L2 = oracle_mod.attention(Q, K[:, :, perm], V[:, :, perm], 0.3, False)
    assert np.allclose(O2, O, rtol=1e-13, atol=1e-14) and np.allclose(L2, L, rtol=1e-14, atol=1e-14)
    # the causal output is NOT permutation invariant (a transposed or missing mask would be)
    Oc, _ = oracle_mod.attention(Q, K, V, 0.3, True)
    Oc2, _ = oracle_mod.attention(Q, K[:, :, perm], V[:, :, perm], 0.3, True)
    assert not np.allclose(Oc, Oc2)


def test_rows_api_matches_full(oracle_mod):
    rng = np.random.default_rng(19)
    B, H, Nq, Nk, d = 2, 3, 17, 23, 8
    Q = rng.standard_normal((B, H, Nq, d)); K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d))
    for causal in (False, True):
        O, L = oracle_mod.attention(Q, K, V, 0.4, causal, nthreads=3)
        rows = np.array([0, 5, 16, 17, 40, B * H * Nq - 1])
        Or, Lr = oracle_mod.attention_rows(Q, K, V, 0.4, causal, rows)
        assert np.array_equal(Or, O.reshape(-1, d)[rows])
        assert np.array_equal(Lr, L.reshape(-1)[rows])


def test_thread_count_does_not_change_result(oracle_mod):
    rng = np.random.default_rng(23)
    Q = rng.standard_normal((2, 2, 50, 16)); K = rng.standard_normal((2, 2, 70, 16))
    V = rng.standard_normal((2, 2, 70, 16))
    O1, L1 = oracle_mod.attention(Q, K, V, 0.25, True, nthreads=1)
    O4, L4 = oracle_mod.attention(Q, K, V, 0.25, True, nthreads=4)
    assert np.array_equal(O1, O4) and np.array_equal(L1, L4)
