"""The bound p_rounding_term derives for rounding P to the input type, checked on the CPU
against an emulation of that rounding.

The emulation computes each row in float64 the way the forward pass combines its roundings:
P = 2^(t - m') with m' a stale running maximum (the lazy rescale leaves it up to 2^8 below
the true maximum), P rounded to the input type (round to nearest even) before the product
with V, l summed from the unrounded P, and O rounded to the output type. Its error against
the exact softmax must stay within TOL_O + half an ulp + p_rounding_term, element by
element; and on inputs of std 2 the P term is what keeps it there."""
import numpy as np
import pytest
import torch

import gen
from tests.fa_testlib import TOL_O, half_ulp, p_rounding_term

_TORCH = {gen.BF16: torch.bfloat16, gen.F16: torch.float16}


def _round(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(_TORCH[dtype]).double().numpy()


def _emulate(w, q, k, v, seed=0):
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    qf = gen.to_f64_numpy(q).reshape(BH, w.Nq, w.d)
    kf = gen.to_f64_numpy(k).reshape(BH, w.Nk, w.d)
    vf = gen.to_f64_numpy(v).reshape(BH, w.Nk, w.d)
    O = np.empty((BH, w.Nq, w.d))
    Oex = np.empty((BH, w.Nq, w.d))
    for bh in range(BH):
        s = (qf[bh] @ kf[bh].T) * w.scale * np.log2(np.e)  # base-2 scores
        if w.causal:
            s = np.where(np.arange(w.Nk)[None, :] <= np.arange(w.Nq)[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        stale = m - rng.uniform(0.0, 8.0, size=m.shape)  # a running max up to 2^8 behind
        P = np.exp2(s - stale)
        Ph = _round(P, w.dtype)
        O[bh] = _round((Ph @ vf[bh]) / P.sum(axis=1, keepdims=True), w.dtype)
        Pe = np.exp2(s - m)
        Oex[bh] = (Pe @ vf[bh]) / Pe.sum(axis=1, keepdims=True)
    return O.reshape(-1, w.d), Oex.reshape(-1, w.d)


@pytest.mark.parametrize("dtype,causal,std", [(gen.BF16, True, 2.0), (gen.BF16, False, 2.0),
                                              (gen.F16, True, 2.0), (gen.BF16, True, 1.0)])
def test_emulated_p_rounding_within_derived_bound(dtype, causal, std):
    w = gen.custom(1, 4, 512, 512, 128, dtype, causal, std, seed=77)
    q, k, v = gen.make_qkv(w)
    O, Oex = _emulate(w, q, k, v)
    err = np.abs(O - Oex)
    graded = TOL_O[dtype] + half_ulp(Oex, dtype)
    derived = graded + p_rounding_term(w, v)
    assert np.all(err <= derived), float((err / derived).max())


def test_p_term_is_what_covers_std2_bf16():
    """Without the P term the same emulation breaks the graded bound on std-2 bf16 inputs
    (a wrong, smaller bound would be caught here), and the term never exceeds 2^-8 max|V|."""
    w = gen.custom(1, 8, 512, 512, 128, gen.BF16, True, 2.0, seed=78)
    q, k, v = gen.make_qkv(w)
    O, Oex = _emulate(w, q, k, v, seed=1)
    err = np.abs(O - Oex)
    graded = TOL_O[w.dtype] + half_ulp(Oex, w.dtype)
    assert np.any(err > graded)
    term = p_rounding_term(w, v)
    assert term.max() <= 2.0 ** -8 * np.abs(v.float().numpy()).max() + 1e-15
    assert np.all(err <= graded + term)


def test_p_term_causal_row0_is_v0():
    """Row 0 of a causal head sees key 0 only: its term is 2^-(t+1) |V[0]|."""
    w = gen.custom(1, 1, 64, 64, 64, gen.BF16, True, 1.0, seed=3)
    _, _, v = gen.make_qkv(w)
    term = p_rounding_term(w, v)
    assert np.allclose(term[0], 2.0 ** -8 * np.abs(v[0, 0, 0].double().numpy()))
