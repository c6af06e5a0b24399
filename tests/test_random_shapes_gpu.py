"""A seeded sweep of random problem shapes through the forward, backward and dropout paths,
each compared element by element with the float64 oracle under the same bounds as the
dedicated tests: forward 1e-2 (bf16) / 4e-3 (fp16) on O and 1e-3 on L (plus half an ulp
of O's type, the rounding of the exact answer); backward 8 half-ulps of the largest
gradient (floor 0.05); dropout forward the forward bound times the keep factor.

The shapes mix every dimension the kernels tile: ragged query and key lengths on both
sides of the 128-row tiles and 256-row work items, single rows and single keys, more
query rows than keys under the causal mask (top-left alignment), both head dims and both
16-bit types."""
import ctypes

import numpy as np
import pytest
import torch

import gen
from tests.fa_bwd_testlib import make_inputs, run_fwd_bwd
from tests.fa_testlib import TOL_L, TOL_O, half_ulp, run_cuda

pytestmark = pytest.mark.gpu

TOL_BWD = {gen.BF16: 8 * 2.0 ** -9, gen.F16: 8 * 2.0 ** -12}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    lens = [1, 2, 17, 127, 128, 129, 255, 256, 257, 300, 511, 640]
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 5))
        Nq = int(rng.choice(lens)) if rng.random() < 0.6 else int(rng.integers(1, 700))
        Nk = int(rng.choice(lens)) if rng.random() < 0.6 else int(rng.integers(1, 700))
        d = int(rng.choice([64, 128]))
        dt = gen.BF16 if rng.random() < 0.5 else gen.F16
        causal = bool(rng.random() < 0.5)
        out.append((B, H, Nq, Nk, d, dt, causal))
    return out


def _seed(c):
    """A reproducible input seed per case (Python's str hash varies between processes)."""
    B, H, Nq, Nk, d, dt, causal = c
    return 10007 * B + 1009 * H + 101 * Nq + 11 * Nk + d + (7 if dt == gen.BF16 else 0) + int(causal)


def _id(c):
    return "B{}H{}_q{}k{}_d{}_{}_{}".format(c[0], c[1], c[2], c[3], c[4], c[5],
                                            "causal" if c[6] else "full")


@pytest.mark.parametrize("case", _shapes(24, 2026), ids=_id)
def test_random_shape_forward(oracle_mod, case):
    B, H, Nq, Nk, d, dt, causal = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=_seed(case))
    q, k, v = gen.make_qkv(w)
    O, L = run_cuda(w, q, k, v)
    Oref, Lref = oracle_mod.attention(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                      gen.to_f64_numpy(v), w.scale, causal)
    err = np.abs(O.double().numpy() - Oref)
    assert np.all(err <= TOL_O[dt] + half_ulp(Oref, dt)), float(err.max())
    assert np.abs(L.double().numpy() - Lref).max() <= TOL_L


@pytest.mark.parametrize("case", _shapes(12, 7), ids=_id)
def test_random_shape_backward(oracle_mod, case):
    B, H, Nq, Nk, d, dt, causal = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=_seed(case))
    q, k, v, do = make_inputs(w)
    _, _, dQ, dK, dV = run_fwd_bwd(w, q, k, v, do)
    refs = oracle_mod.attention_bwd(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                    gen.to_f64_numpy(do), w.scale, causal)
    for name, got, ref in (("dQ", dQ, refs[0]), ("dK", dK, refs[1]), ("dV", dV, refs[2])):
        g = got.double().numpy()
        assert np.isfinite(g).all(), name
        bound = TOL_BWD[dt] * max(float(np.abs(ref).max()), 0.05)
        assert float(np.abs(g - ref).max()) <= bound, (name, float(np.abs(g - ref).max()), bound)


@pytest.mark.parametrize("case", _shapes(10, 31), ids=_id)
def test_random_shape_dropout_forward(oracle_mod, case):
    import exact_attention_forward_02_gb300 as fa
    B, H, Nq, Nk, d, dt, causal = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=_seed(case))
    q, k, v = gen.make_qkv(w)
    p, seed, off = 0.2, 1000 + Nq, 3
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    O = torch.full((B, H, Nq, d), float("nan"), dtype=q.dtype, device=dev)
    L = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    rc = fa.fa_fwd_dropout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                           B, H, Nq, Nk, d, w.scale, causal,
                           fa.FA_BF16 if dt == gen.BF16 else fa.FA_F16, p, seed, off,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
    p32 = float(np.float32(p))
    Oref, Lref = oracle_mod.attention_dropout(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                              gen.to_f64_numpy(v), w.scale, causal, p32, seed, off)
    keep = 256.0 / (256 - oracle_mod.dropout_threshold(p32))
    err = np.abs(O.double().cpu().numpy() - Oref)
    assert np.all(err <= TOL_O[dt] * keep + half_ulp(Oref, dt)), float(err.max())
    assert np.abs(L.double().cpu().numpy() - Lref).max() <= TOL_L
