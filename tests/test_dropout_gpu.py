"""GPU parity of the dropout forward (fa_fwd_dropout) and its mask (fa_dropout_mask)
against the float64 oracle.

"Flash Attention" page, "Algorithm 2": O = dropout(softmax(S), p) V. The mask is integer
work, so it is compared bit for bit: directly (fa_dropout_mask against the oracle's
mask), and through the attention kernel itself, where Q = 0 makes every probability equal
and weighted one-hot values make O spell out the kept bits. The outputs on random inputs
are compared with the oracle's dropout forward under the forward's tolerances scaled by
the keep factor 256 / (256 - t): every term of O is multiplied by it, and so is the
rounding error of P that the forward's tolerance covers."""
import ctypes

import numpy as np
import pytest
import torch

import gen
from tests.fa_testlib import TOL_L, TOL_O, half_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()


def _fa():
    import exact_attention_forward_02_gb300 as fa
    return fa


def _f32(p):
    """The probability as the C ABI sees it (a float)."""
    return float(np.float32(p))


def keep_factor(p):
    import oracle
    t = oracle.dropout_threshold(_f32(p))
    return 256.0 / (256 - t)


def run_dropout(w, q, k, v, p, seed, offset, nan_fill=True):
    fa = _fa()
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fill = float("nan") if nan_fill else 0.0
    O = torch.full((w.B, w.H, w.Nq, w.d), fill, dtype=q.dtype, device=dev)
    L = torch.full((w.B, w.H, w.Nq), fill, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream(dev)
    rc = fa.fa_fwd_dropout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                           w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                           fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16, p, seed, offset,
                           ctypes.c_void_p(st.cuda_stream))
    assert rc == 0, f"fa_fwd_dropout rc={rc} ({fa.strerror(rc)})"
    torch.cuda.synchronize(dev)
    assert fa.fa_last_status() == 0
    return O.cpu(), L.cpu()


def gpu_mask(B, H, Nq, Nk, p, seed, offset):
    fa = _fa()
    keep = torch.full((B, H, Nq, Nk), 7, dtype=torch.uint8, device="cuda:0")
    rc = fa.fa_dropout_mask(keep.data_ptr(), B, H, Nq, Nk, p, seed, offset,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize()
    return keep.cpu().numpy()


MASK_CASES = [
    (1, 1, 1, 16, 0.5, 0, 0),
    (2, 3, 37, 45, 0.1, 12345, 7),
    (1, 2, 300, 257, 0.5, (1 << 63) + 99, 0xFFFFFFFF),
    (4, 12, 5, 4097, 0.9, 2**32 + 5, 3),
    (1, 1, 64, 64, 1 - 2.0 ** -8, 1, 1),
    (2, 2, 129, 33, 0.0, 3, 4),
]


@pytest.mark.parametrize("case", MASK_CASES, ids=lambda c: "B{}H{}_q{}k{}_p{:.3g}".format(*c[:5]))
def test_mask_kernel_is_bit_exact(oracle_mod, case):
    B, H, Nq, Nk, p, seed, off = case
    got = gpu_mask(B, H, Nq, Nk, p, seed, off)
    ref = oracle_mod.dropout_keep(B, H, Nq, Nk, _f32(p), seed, off)
    assert np.array_equal(got, ref), int((got != ref).sum())


@pytest.mark.parametrize("d,dtype,causal", [(64, gen.F16, False), (128, gen.BF16, False),
                                            (64, gen.BF16, True), (128, gen.F16, True)])
def test_attention_kernel_applies_the_exact_mask(oracle_mod, d, dtype, causal):
    """Q = 0: every visible key has probability 1 / n_visible. V_j = 2^(j div d) e_(j mod d)
    over Nk = 4d keys (four K/V tiles at d = 128, two at d = 64): then
    O_ic * n_visible / keep_factor = sum_q 2^q keep(i, c + q d), an integer in [0, 15] that
    the 16-bit output holds exactly enough to read back."""
    B, H, Nq, Nk = 1, 3, 300, 4 * d
    p, seed, off = 0.37, 2024, 11
    w = gen.custom(B, H, Nq, Nk, d, dtype, causal, 1.0, seed=0)
    tdt = gen.torch_dtype(dtype)
    q = torch.zeros((B, H, Nq, d), dtype=tdt)
    k = torch.randn((B, H, Nk, d), generator=torch.Generator().manual_seed(1)).to(tdt)
    v = torch.zeros((B, H, Nk, d), dtype=tdt)
    for j in range(Nk):
        v[:, :, j, j % d] = float(2 ** (j // d))
    O, L = run_dropout(w, q, k, v, p, seed, off)
    keep = oracle_mod.dropout_keep(B, H, Nq, Nk, _f32(p), seed, off).astype(np.int64)
    rows = np.arange(Nq)
    nvis = np.minimum(rows + 1, Nk) if causal else np.full(Nq, Nk)
    if causal:
        keep = keep * (np.arange(Nk)[None, None, None, :] <= rows[None, None, :, None])
    expect = sum(keep[..., qq * d:(qq + 1) * d] << qq for qq in range(4))
    got = O.double().numpy() * nvis[None, None, :, None] / keep_factor(p)
    n = np.rint(got).astype(np.int64)
    assert np.all(np.abs(got - n) < 0.25), float(np.abs(got - n).max())
    assert np.array_equal(n, expect), int((n != expect).sum())
    assert np.allclose(L.double().numpy(), np.log(nvis)[None, None, :], atol=TOL_L)


def _rand(w, seed):
    g = torch.Generator().manual_seed(seed)
    tdt = gen.torch_dtype(w.dtype)
    q = torch.randn((w.B, w.H, w.Nq, w.d), generator=g).to(tdt)
    k = torch.randn((w.B, w.H, w.Nk, w.d), generator=g).to(tdt)
    v = torch.randn((w.B, w.H, w.Nk, w.d), generator=g).to(tdt)
    return q, k, v


def _check(w, O, L, Oref, Lref, p):
    Ok = O.double().numpy().reshape(-1, w.d)
    Lk = L.double().numpy().reshape(-1)
    Or = np.asarray(Oref).reshape(-1, w.d)
    Lr = np.asarray(Lref).reshape(-1)
    assert np.all(np.isfinite(Ok)) and np.all(np.isfinite(Lk))
    tol = TOL_O[w.dtype] * keep_factor(p)
    err = np.abs(Ok - Or)
    assert np.all(err <= tol + half_ulp(Or, w.dtype)), float(err.max())
    assert np.abs(Lk - Lr).max() <= TOL_L
    return float(err.max())


PARITY = [
    (1, 1, 128, 128, 64, gen.F16, False, 0.1),
    (1, 1, 128, 128, 64, gen.F16, True, 0.5),
    (2, 3, 300, 257, 64, gen.F16, False, 0.2),
    (1, 2, 257, 600, 128, gen.BF16, True, 0.1),
    (2, 2, 1000, 1000, 128, gen.BF16, False, 0.3),
    (1, 4, 700, 130, 128, gen.BF16, True, 0.6),
    (1, 2, 1000, 4097, 64, gen.F16, False, 0.1),
]


@pytest.mark.parametrize("case", PARITY, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}_{}_p{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full", c[7]))
def test_dropout_forward_matches_oracle(oracle_mod, case):
    B, H, Nq, Nk, d, dt, causal, p = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=0)
    q, k, v = _rand(w, 500 + Nq + Nk)
    seed, off = 77 + Nq, 5
    O, L = run_dropout(w, q, k, v, p, seed, off)
    Oref, Lref = oracle_mod.attention_dropout(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                              gen.to_f64_numpy(v), w.scale, causal, _f32(p), seed,
                                              off)
    print(w.describe(), "p", p, "max err", _check(w, O, L, Oref, Lref, p))


@pytest.mark.parametrize("name", ["b2h8_n8192_d128_causal", "b2h8_n4096_d128_full"])
def test_dropout_full_size_whole_output(oracle_mod, name):
    """The two benchmark workloads at full size with p = 0.1: every element of O and L
    against the oracle, which draws the same mask."""
    w = gen.WORKLOADS[name]
    q, k, v = gen.make_qkv(w)
    p, seed, off = 0.1, 31337, 2
    O, L = run_dropout(w, q, k, v, p, seed, off)
    Oref, Lref = oracle_mod.attention_dropout(gen.to_f64_numpy(q), gen.to_f64_numpy(k),
                                              gen.to_f64_numpy(v), w.scale, w.causal, _f32(p),
                                              seed, off)
    print(name, "max err", _check(w, O, L, Oref, Lref, p))


def test_zero_probability_is_fa_fwd_and_determinism():
    fa = _fa()
    w = gen.custom(2, 2, 300, 300, 128, gen.BF16, True, 1.0, seed=0)
    q, k, v = _rand(w, 9)
    from tests.fa_testlib import run_cuda
    O0, L0 = run_cuda(w, q, k, v)
    O1, L1 = run_dropout(w, q, k, v, 0.0, 5, 6)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
    Oa, La = run_dropout(w, q, k, v, 0.25, 5, 6)
    Ob, Lb = run_dropout(w, q, k, v, 0.25, 5, 6)
    Oc, _ = run_dropout(w, q, k, v, 0.25, 5, 7)
    assert torch.equal(Oa, Ob) and torch.equal(La, Lb)
    assert torch.equal(La, L0)  # the logsumexp ignores the mask
    assert not torch.equal(Oa, Oc)
    for bad in (1.0, -0.1, float("nan"), float("inf")):
        rc = fa.fa_fwd_dropout(1, 1, 1, 1, 1, 1, 1, 1, 1, 64, 1.0, 0, fa.FA_F16, bad, 0, 0, None)
        assert rc == fa.FA_ERR_DROPOUT, (bad, rc)
        assert fa.fa_dropout_mask(1, 1, 1, 1, 1, bad, 0, 0, None) == fa.FA_ERR_DROPOUT
