"""GPU parity of the backward pass (fa_bwd) against the float64 backward oracle.

Tolerance (derived from the arithmetic; the forward's target tolerances do not cover
gradients): P and dS are rounded to the input type before the products that use them,
and dQ, dK, dV are rounded to it on output. Each rounding is at most half an ulp, 2^-9
relative for bf16 and 2^-12 for fp16. The bound is 8 such half-ulps of the largest
gradient magnitude: max |g - g64| <= 8 * 2^-(m+1) * max(max |g64|, 0.05) (1.6e-2 bf16,
2e-3 fp16). The floor of 0.05 covers gradients that are exactly zero (one key: P = 1, so
dS = 0), where only the rounding of D = rowsum(dO o O) from the 16-bit O is left."""
import pytest
import torch

import gen
from tests.fa_bwd_testlib import grad_errors, make_inputs, run_fwd_bwd

pytestmark = pytest.mark.gpu

TOL_REL = {gen.BF16: 8 * 2.0 ** -9, gen.F16: 8 * 2.0 ** -12}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()


CASES = [
    (1, 1, 128, 128, 64, gen.F16, False),
    (1, 1, 128, 128, 64, gen.F16, True),
    (1, 1, 1, 1, 128, gen.BF16, False),
    (1, 2, 2, 2, 64, gen.BF16, True),
    (1, 2, 256, 256, 128, gen.BF16, False),
    (1, 2, 256, 256, 128, gen.BF16, True),
    (2, 3, 300, 257, 64, gen.F16, False),      # ragged tails in both sequences
    (1, 2, 257, 300, 128, gen.BF16, True),     # causal, Nq < Nk (top-left)
    (1, 2, 700, 130, 64, gen.F16, True),       # causal, Nq > Nk
    (2, 4, 1024, 1024, 128, gen.BF16, True),
    (1, 2, 1000, 4097, 64, gen.F16, False),    # the cross-attention shape, fewer heads
    (3, 70, 256, 384, 128, gen.BF16, False),   # more work items than SMs in both kernels
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
def test_bwd_matches_oracle(case):
    B, H, Nq, Nk, d, dt, causal = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=3000 + sum(case[:5]))
    q, k, v, do = make_inputs(w)
    O, L, dQ, dK, dV = run_fwd_bwd(w, q, k, v, do)
    errs = grad_errors(w, q, k, v, do, dQ, dK, dV)
    print(w.describe(), errs)
    for name, e in errs.items():
        assert e["finite"], name
        assert e["max_abs_err"] <= TOL_REL[dt] * max(e["max_abs_ref"], 0.05), (name, e)


@pytest.mark.parametrize("name", ["b2h8_n4096_d128_full", "b2h8_n8192_d128_causal"])
def test_bwd_full_size_workloads(name):
    """The backward of the two benchmark workloads at full size, as `bench.py --bwd` runs
    it: every element of dQ, dK and dV against the float64 oracle."""
    w = gen.WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    O, L, dQ, dK, dV = run_fwd_bwd(w, q, k, v, do)
    errs = grad_errors(w, q, k, v, do, dQ, dK, dV)
    print(w.name, errs)
    for gname, e in errs.items():
        assert e["finite"], gname
        assert e["max_abs_err"] <= TOL_REL[w.dtype] * max(e["max_abs_ref"], 0.05), (gname, e)


def test_bwd_deterministic():
    w = gen.custom(2, 3, 500, 500, 128, gen.BF16, True, 1.0, seed=99)
    q, k, v, do = make_inputs(w)
    a = run_fwd_bwd(w, q, k, v, do)
    b = run_fwd_bwd(w, q, k, v, do)
    for x, y in zip(a[2:], b[2:]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bwd_workspace_checks():
    import ctypes

    import exact_attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    x = torch.zeros(1 * 1 * 128 * 64, dtype=torch.float16, device=dev)
    L = torch.zeros(128, dtype=torch.float32, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = x.data_ptr()
    need = fa.fa_bwd_workspace_bytes(1, 1, 128, 128, 64)
    assert need >= 128 * 4
    small = torch.zeros(need // 2, dtype=torch.uint8, device=dev)
    args = (p, p, p, p, p, L.data_ptr(), p, p, p, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_F16)
    assert fa.fa_bwd(*args, small.data_ptr(), small.numel(), st) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd(*args, 0, 0, st) == fa.FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
