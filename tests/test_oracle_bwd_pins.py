"""Pins for the float64 backward oracle (CS336 lecture 5 "05_flash_attention.py", part 3;
"Flash Attention" page, Algorithm 4 and its derivation): torch autograd in float64
(library routine), central finite differences of the forward oracle on tiny inputs, and
closed forms (sum over keys of dK is zero; sum over keys of dV equals the sum over queries
of dO; causal row 0 has zero dQ)."""
import math

import numpy as np
import pytest
import torch


def _torch_grads(Q, K, V, dO, scale, causal):
    q, k, v = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        Nq, Nk = s.shape[-2:]
        s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("shape,causal", [
    ((1, 1, 100, 100, 32), False), ((1, 1, 100, 100, 32), True),
    ((2, 3, 37, 53, 16), False), ((2, 2, 53, 37, 16), True), ((1, 2, 29, 61, 8), True),
])
def test_bwd_matches_torch_autograd_float64(oracle_mod, shape, causal):
    B, H, Nq, Nk, d = shape
    rng = np.random.default_rng(sum(shape) + 7 * causal)
    Q = rng.standard_normal((B, H, Nq, d)); K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d)); dO = rng.standard_normal((B, H, Nq, d))
    scale = 1 / math.sqrt(d)
    dQ, dK, dV = oracle_mod.attention_bwd(Q, K, V, dO, scale, causal)
    tq, tk, tv = _torch_grads(Q, K, V, dO, scale, causal)
    assert np.allclose(dQ, tq, rtol=1e-11, atol=1e-12)
    assert np.allclose(dK, tk, rtol=1e-11, atol=1e-12)
    assert np.allclose(dV, tv, rtol=1e-11, atol=1e-12)


def test_bwd_central_differences(oracle_mod):
    """d/dx of sum(O * G) by central differences of the FORWARD oracle."""
    rng = np.random.default_rng(3)
    for causal in (False, True):
        Nq, Nk, d = 3, 4, 2
        Q = rng.standard_normal((1, 1, Nq, d)); K = rng.standard_normal((1, 1, Nk, d))
        V = rng.standard_normal((1, 1, Nk, d)); G = rng.standard_normal((1, 1, Nq, d))
        scale = 0.7
        dQ, dK, dV = oracle_mod.attention_bwd(Q, K, V, G, scale, causal)
        h = 1e-6

        def loss(Qx, Kx, Vx):
            O, _ = oracle_mod.attention(Qx, Kx, Vx, scale, causal)
            return float((O * G).sum())

        for X, g, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
            for idx in np.ndindex(X.shape):
                args = [Q.copy(), K.copy(), V.copy()]
                args[which][idx] += h
                up = loss(*args)
                args[which][idx] -= 2 * h
                dn = loss(*args)
                assert abs((up - dn) / (2 * h) - g[idx]) < 1e-7, (which, idx)


def test_bwd_closed_forms(oracle_mod):
    rng = np.random.default_rng(5)
    B, H, Nq, Nk, d = 2, 2, 30, 45, 8
    Q = rng.standard_normal((B, H, Nq, d)); K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d)); dO = rng.standard_normal((B, H, Nq, d))
    for causal in (False, True):
        dQ, dK, dV = oracle_mod.attention_bwd(Q, K, V, dO, 0.4, causal)
        # each row of dS sums to zero, hence the sum over keys of dK vanishes
        assert np.allclose(dK.sum(axis=2), 0.0, atol=1e-12)
        # each row of P sums to one, hence sum_j dV_j = sum_i dO_i
        assert np.allclose(dV.sum(axis=2), dO.sum(axis=2), atol=1e-12)
        if causal:  # row 0 attends to key 0 only: P = 1, dS = 0
            assert np.allclose(dQ[:, :, 0], 0.0, atol=1e-14)
