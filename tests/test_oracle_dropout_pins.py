"""Pins for the dropout part of the float64 oracle.

The "Flash Attention" page, "Algorithm 2", adds dropout to the forward pass
(P_dropped = dropout(P, p), O = P_dropped V; the forward also returns the generator state
R) and "Algorithm 4" regenerates the mask Z from R in the backward pass
(dV += (P o Z)^T dO, dP = dP_dropped o Z). The pages name no generator: the library uses
Philox-4x32-10 (Salmon et al., SC'11) with the counter layout stated in the oracle and in
include/fa_fwd.h. What fixes each piece here, other than the oracle itself:
  * the generator: the published known-answer vectors (tests/golden/philox4x32_10_kat.json)
    and Triton's independent tl.philox run by its CPU interpreter;
  * the counter layout and the 8-bit threshold: mask bits worked out by hand from the
    first known-answer vector, and the layout checked against Triton's words;
  * the dropout arithmetic: p = 0 gives the plain forward exactly, L does not depend on
    the mask, the mean over seeds converges to the undropped output (unbiased, within a
    CLT bound), the kept fraction is binomial, a one-hot V reads the mask out of O, and
    the backward matches central differences and torch autograd of the masked forward.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
KAT = os.path.join(HERE, "golden", "philox4x32_10_kat.json")


def _h(x):
    return int(x, 16)


def test_philox_known_answer_vectors(oracle_mod):
    with open(KAT) as f:
        vecs = json.load(f)["vectors"]
    assert len(vecs) == 3
    for v in vecs:
        out = oracle_mod.philox4x32_10([_h(x) for x in v["ctr"]], [_h(x) for x in v["key"]])
        assert [int(x) for x in out] == [_h(x) for x in v["out"]], v


def _triton_words(items):
    pytest.importorskip("triton")
    r = subprocess.run([sys.executable, os.path.join(HERE, "philox_triton_ref.py")],
                       input=json.dumps(items), capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        pytest.skip("Triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1]
                    if r.stderr.strip() else "Triton interpreter unavailable")
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_philox_matches_triton_and_mask_layout(oracle_mod):
    """Triton's tl.philox (an independent implementation) gives the same words as the
    oracle for arbitrary counters and 64-bit seeds, and the oracle's mask follows the
    stated layout: counter (j >> 4, i, bh, offset), word (j >> 2) & 3, byte
    2 (j & 1) + ((j >> 1) & 1), keep iff x >= t."""
    rng = np.random.default_rng(11)
    B, H, Nq, Nk = 2, 3, 5, 37
    seed, offset = (1 << 63) + 987654321, 77
    p = 0.3
    t = oracle_mod.dropout_threshold(p)
    items = []
    for bh in range(B * H):
        for i in range(Nq):
            for g in range((Nk + 15) // 16):
                items.append([g, i, bh, offset, seed])
    extra = [[int(x) for x in rng.integers(0, 2**32, 4)] + [int(rng.integers(0, 2**63))]
             for _ in range(8)]
    words = _triton_words(items + extra)
    for it, w in zip(extra, words[len(items):]):
        assert [int(x) for x in oracle_mod.philox4x32_10(it[:4], [it[4] & 0xFFFFFFFF, it[4] >> 32])] == w
    expect = np.zeros((B, H, Nq, Nk), np.uint8)
    k = 0
    for bh in range(B * H):
        for i in range(Nq):
            for g in range((Nk + 15) // 16):
                w = words[k]
                k += 1
                for j in range(16 * g, min(Nk, 16 * g + 16)):
                    word = w[(j >> 2) & 3]
                    x = (word >> (8 * (2 * (j & 1) + ((j >> 1) & 1)))) & 0xFF
                    expect[bh // H, bh % H, i, j] = 1 if x >= t else 0
    got = oracle_mod.dropout_keep(B, H, Nq, Nk, p, seed, offset)
    assert np.array_equal(got, expect)


def test_mask_bits_from_the_first_known_answer_vector(oracle_mod):
    """seed 0, offset 0, head 0, row 0, keys 0..15 use counter (0, 0, 0, 0) under key
    (0, 0), whose words are 6627e8d5 e169c58d bc57ac4c 9b00dbd8. Taking bytes 0, 2, 1, 3 of
    each word in turn, the keys draw
    d5 27 e8 66 | 8d 69 c5 e1 | 4c 57 ac bc | d8 00 db 9b."""
    x = [0xd5, 0x27, 0xe8, 0x66, 0x8d, 0x69, 0xc5, 0xe1,
         0x4c, 0x57, 0xac, 0xbc, 0xd8, 0x00, 0xdb, 0x9b]
    assert oracle_mod.dropout_threshold(0.5) == 128
    got = oracle_mod.dropout_keep(1, 1, 1, 16, 0.5, 0, 0)[0, 0, 0]
    assert got.tolist() == [1, 0, 1, 0, 1, 0, 1, 1, 0, 0, 1, 1, 1, 0, 1, 1]
    # a threshold equal to a draw keeps that key (x >= t), one above drops it
    for t in (0x66, 0x67, 0x27, 0x28, 1, 0, 255):
        p = t / 256.0
        assert oracle_mod.dropout_threshold(p) == t
        got = oracle_mod.dropout_keep(1, 1, 1, 16, p, 0, 0)[0, 0, 0]
        assert got.tolist() == [1 if v >= t else 0 for v in x], t


def test_threshold_rounding_and_range(oracle_mod):
    assert oracle_mod.dropout_threshold(0.0) == 0
    assert oracle_mod.dropout_threshold(0.1) == 26            # 25.6 rounds up
    assert oracle_mod.dropout_threshold(0.5) == 128
    assert oracle_mod.dropout_threshold(1 - 2.0 ** -8) == 255
    assert oracle_mod.dropout_threshold(1.5 / 256) == 2        # ties round up
    for bad in (1.0, 1 - 2.0 ** -9, 1.5, -1e-9, float("nan"), float("inf")):
        assert oracle_mod.dropout_threshold(bad) == -1, bad
    with pytest.raises(ValueError):
        oracle_mod.dropout_keep(1, 1, 1, 1, 1.0, 0, 0)


def _qkv(seed, B, H, Nq, Nk, d):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, H, Nq, d)), rng.standard_normal((B, H, Nk, d)),
            rng.standard_normal((B, H, Nk, d)))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_probability_is_the_plain_forward(oracle_mod, causal):
    Q, K, V = _qkv(1, 2, 2, 33, 41, 8)
    O0, L0 = oracle_mod.attention(Q, K, V, 0.35, causal)
    O1, L1 = oracle_mod.attention_dropout(Q, K, V, 0.35, causal, 0.0, 1234, 5)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


@pytest.mark.parametrize("causal", [False, True])
def test_logsumexp_does_not_depend_on_the_mask(oracle_mod, causal):
    Q, K, V = _qkv(2, 1, 3, 20, 29, 8)
    _, L0 = oracle_mod.attention(Q, K, V, 0.5, causal)
    for p, seed in ((0.1, 1), (0.6, 2), (0.9, 3)):
        _, L1 = oracle_mod.attention_dropout(Q, K, V, 0.5, causal, p, seed, 0)
        assert np.array_equal(L0, L1)


def test_one_hot_values_read_the_mask_out_of_the_output(oracle_mod):
    """Q = 0 makes every probability 1/Nk; with V_j = e_j (Nk = d) the output is
    O_ij = keep_ij * 256 / (256 - t) / Nk, so O reveals the mask element by element."""
    B, H, Nq, Nk = 2, 2, 9, 16
    Q = np.zeros((B, H, Nq, Nk))
    K = np.random.default_rng(3).standard_normal((B, H, Nk, Nk))
    V = np.broadcast_to(np.eye(Nk), (B, H, Nk, Nk)).copy()
    p, seed, off = 0.4, 99, 3
    t = oracle_mod.dropout_threshold(p)
    O, _ = oracle_mod.attention_dropout(Q, K, V, 1.0, False, p, seed, off)
    keep = oracle_mod.dropout_keep(B, H, Nq, Nk, p, seed, off)
    assert np.allclose(O, keep * (256.0 / (256 - t)) / Nk, rtol=0, atol=1e-15)


def test_kept_fraction_is_binomial(oracle_mod):
    B, H, Nq, Nk = 1, 2, 256, 300
    for p, seed, off in ((0.1, 5, 0), (0.5, 6, 1), (0.85, 7, 2)):
        keep = oracle_mod.dropout_keep(B, H, Nq, Nk, p, seed, off)
        n = keep.size
        q = (256 - oracle_mod.dropout_threshold(p)) / 256.0
        assert abs(keep.mean() - q) < 6 * math.sqrt(q * (1 - q) / n), (p, keep.mean())
        # different offsets and seeds give different masks
        other = oracle_mod.dropout_keep(B, H, Nq, Nk, p, seed, off + 1)
        assert (other != keep).mean() > 0.5 * 2 * q * (1 - q)


def test_dropout_is_unbiased_over_seeds(oracle_mod):
    """E[P_dropped] = P ("dropout" of Algorithm 2 scales kept entries by 1/(1-p)), so the
    mean of O over independent masks converges to the plain O. Var[O_ic] =
    sum_j P_ij^2 V_jc^2 (1/(1-p) - 1) per mask; the bound is 6 standard errors."""
    Q, K, V = _qkv(4, 1, 1, 6, 12, 4)
    scale, p, n = 0.6, 0.35, 3000
    O0, _ = oracle_mod.attention(Q, K, V, scale, False)
    acc = np.zeros_like(O0)
    for s in range(n):
        O1, _ = oracle_mod.attention_dropout(Q, K, V, scale, False, p, 1000 + s, 0, nthreads=1)
        acc += O1
    mean = acc / n
    P = oracle_mod.probs(Q[0, 0], K[0, 0], scale, False)
    q = (256 - oracle_mod.dropout_threshold(p)) / 256.0
    var = (P ** 2) @ (V[0, 0] ** 2) * (1.0 / q - 1.0)
    se = np.sqrt(var / n)
    assert np.all(np.abs(mean[0, 0] - O0[0, 0]) < 6 * se + 1e-12)


def _masked_forward_torch(Q, K, V, scale, causal, Z):
    """Algorithm 2 in torch float64 with the mask Z (already scaled) as a constant."""
    S = scale * Q @ K.transpose(-1, -2)
    if causal:
        Nq, Nk = S.shape[-2:]
        S = S.masked_fill(torch.arange(Nk)[None, :] > torch.arange(Nq)[:, None], float("-inf"))
    return (torch.softmax(S, dim=-1) * Z) @ V


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_forward_and_backward_match_torch_autograd(oracle_mod, causal):
    B, H, Nq, Nk, d = 2, 2, 23, 31, 8
    Q, K, V = _qkv(8, B, H, Nq, Nk, d)
    dO = np.random.default_rng(9).standard_normal((B, H, Nq, d))
    scale, p, seed, off = 0.45, 0.3, 4242, 1
    q = (256 - oracle_mod.dropout_threshold(p)) / 256.0
    Z = torch.from_numpy(oracle_mod.dropout_keep(B, H, Nq, Nk, p, seed, off).astype(np.float64) / q)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    O_t = _masked_forward_torch(tq, tk, tv, scale, causal, Z)
    O_t.backward(torch.from_numpy(dO))
    O, _ = oracle_mod.attention_dropout(Q, K, V, scale, causal, p, seed, off)
    assert np.allclose(O, O_t.detach().numpy(), rtol=0, atol=1e-12)
    dQ, dK, dV = oracle_mod.attention_bwd_dropout(Q, K, V, dO, scale, causal, p, seed, off)
    for g, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        assert np.allclose(g, ref.numpy(), rtol=0, atol=1e-11)


def test_dropout_backward_central_differences(oracle_mod):
    """With the mask fixed by (seed, offset) the dropout forward is a smooth function of
    Q, K, V; the backward must be the gradient of sum(O o dO)."""
    B, H, Nq, Nk, d = 1, 1, 5, 7, 3
    Q, K, V = _qkv(10, B, H, Nq, Nk, d)
    dO = np.random.default_rng(12).standard_normal((B, H, Nq, d))
    scale, p, seed, off = 0.8, 0.4, 77, 0
    dQ, dK, dV = oracle_mod.attention_bwd_dropout(Q, K, V, dO, scale, False, p, seed, off)

    def loss(Qx, Kx, Vx):
        return float((oracle_mod.attention_dropout(Qx, Kx, Vx, scale, False, p, seed, off)[0] * dO).sum())

    h = 1e-6
    args = [Q.copy(), K.copy(), V.copy()]
    for which, g in ((0, dQ), (1, dK), (2, dV)):
        for idx in np.ndindex(*args[which].shape):
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            dn = loss(*args)
            args[which][idx] += h
            assert abs((up - dn) / (2 * h) - g[idx]) < 1e-7, (which, idx)


def test_zero_probability_backward_is_the_plain_backward(oracle_mod):
    Q, K, V = _qkv(13, 1, 2, 17, 19, 8)
    dO = np.random.default_rng(14).standard_normal(Q.shape)
    a = oracle_mod.attention_bwd(Q, K, V, dO, 0.3, True)
    b = oracle_mod.attention_bwd_dropout(Q, K, V, dO, 0.3, True, 0.0, 5, 5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
