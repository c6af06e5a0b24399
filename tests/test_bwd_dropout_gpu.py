"""GPU parity of the dropout backward pass (fa_bwd_dropout after fa_fwd_dropout) against the
float64 dropout backward oracle.

"Flash Attention" page, "Algorithm 4": the backward regenerates the forward's mask Z from
its generator state and uses dV = (P o Z)^T dO and dP = (dO V^T) o Z. Tolerance: the
backward's (8 half-ulps of the largest gradient, floor 0.05), with the largest gradient
taken from the oracle, which already carries the keep factor 256 / (256 - t) of Z."""
import ctypes

import numpy as np
import pytest
import torch

import gen
from tests.fa_bwd_testlib import make_inputs, run_fwd_bwd

pytestmark = pytest.mark.gpu

TOL_REL = {gen.BF16: 8 * 2.0 ** -9, gen.F16: 8 * 2.0 ** -12}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()


def _f32(p):
    return float(np.float32(p))


def run_drop_fwd_bwd(w, q, k, v, do, p, seed, offset):
    import exact_attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    O = torch.empty((w.B, w.H, w.Nq, w.d), dtype=q.dtype, device=dev)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    dt = fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16
    st = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = fa.fa_fwd_dropout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                           w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt, p, seed, offset, st)
    assert rc == 0, fa.strerror(rc)
    dQ = torch.full_like(qd, float("nan"))
    dK = torch.full_like(kd, float("nan"))
    dV = torch.full_like(vd, float("nan"))
    nws = fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    rc = fa.fa_bwd_dropout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), dod.data_ptr(),
                           L.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), w.B, w.H, w.Nq,
                           w.Nk, w.d, w.scale, w.causal, dt, p, seed, offset, ws.data_ptr(), nws, st)
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize(dev)
    assert fa.fa_last_status() == 0
    return O.cpu(), L.cpu(), dQ.cpu(), dK.cpu(), dV.cpu()


CASES = [
    (1, 1, 128, 128, 64, gen.F16, False, 0.1),
    (1, 1, 128, 128, 64, gen.F16, True, 0.5),
    (1, 2, 256, 256, 128, gen.BF16, False, 0.2),
    (1, 2, 256, 256, 128, gen.BF16, True, 0.1),
    (2, 3, 300, 257, 64, gen.F16, False, 0.3),      # ragged tails in both sequences
    (1, 2, 257, 300, 128, gen.BF16, True, 0.1),     # causal, Nq < Nk
    (1, 2, 700, 130, 64, gen.F16, True, 0.6),       # causal, Nq > Nk
    (2, 4, 1024, 1024, 128, gen.BF16, True, 0.1),
    (1, 2, 1000, 4097, 64, gen.F16, False, 0.1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}_{}_p{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full", c[7]))
def test_dropout_bwd_matches_oracle(oracle_mod, case):
    B, H, Nq, Nk, d, dt, causal, p = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=4000 + sum(case[:5]))
    q, k, v, do = make_inputs(w)
    seed, off = 99 + Nq, 7
    O, L, dQ, dK, dV = run_drop_fwd_bwd(w, q, k, v, do, p, seed, off)
    rq, rk, rv = oracle_mod.attention_bwd_dropout(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                                  gen.to_f64_numpy(v), gen.to_f64_numpy(do), w.scale,
                                                  causal, _f32(p), seed, off)
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.double().numpy()
        assert np.isfinite(g).all(), name
        err = float(np.abs(g - ref).max())
        bound = TOL_REL[dt] * max(float(np.abs(ref).max()), 0.05)
        print(w.describe(), "p", p, name, "max err", err, "bound", bound)
        assert err <= bound, (name, err, bound)


@pytest.mark.parametrize("name", ["b2h8_n4096_d128_full", "b2h8_n8192_d128_causal"])
def test_dropout_bwd_full_size_workloads(oracle_mod, name):
    """The dropout backward of the two benchmark workloads at full size (p = 0.1, as
    `bench.py --bwd --dropout 0.1` runs it): every element of dQ, dK and dV."""
    w = gen.WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    p, seed, off = 0.1, 1234, 1
    O, L, dQ, dK, dV = run_drop_fwd_bwd(w, q, k, v, do, p, seed, off)
    rq, rk, rv = oracle_mod.attention_bwd_dropout(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                                  gen.to_f64_numpy(v), gen.to_f64_numpy(do), w.scale,
                                                  w.causal, _f32(p), seed, off)
    for gname, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.double().numpy()
        assert np.isfinite(g).all(), gname
        err = float(np.abs(g - ref).max())
        bound = TOL_REL[w.dtype] * max(float(np.abs(ref).max()), 0.05)
        print(name, gname, "max err", err, "bound", bound)
        assert err <= bound, (gname, err, bound)


def test_zero_probability_is_fa_bwd_and_bad_probability():
    import exact_attention_forward_02_gb300 as fa
    w = gen.custom(1, 2, 300, 300, 128, gen.BF16, True, 1.0, seed=12)
    q, k, v, do = make_inputs(w)
    a = run_fwd_bwd(w, q, k, v, do)
    b = run_drop_fwd_bwd(w, q, k, v, do, 0.0, 5, 6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    P = 1 << 20
    for bad in (1.0, -0.5, float("nan")):
        rc = fa.fa_bwd_dropout(P, P, P, P, P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_F16,
                               bad, 0, 0, P, 1 << 20, None)
        assert rc == fa.FA_ERR_DROPOUT


def test_dropout_bwd_deterministic():
    w = gen.custom(2, 3, 333, 333, 128, gen.BF16, False, 1.0, seed=13)
    q, k, v, do = make_inputs(w)
    a = run_drop_fwd_bwd(w, q, k, v, do, 0.25, 1, 2)
    b = run_drop_fwd_bwd(w, q, k, v, do, 0.25, 1, 2)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
