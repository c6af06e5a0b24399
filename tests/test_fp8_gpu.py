"""GPU parity of the E4M3 forward pass (fa_fwd_fp8) against the float64 oracle.

The oracle evaluates the definition on the exactly decoded inputs with the descales
applied: O = softmax(scale (q_descale Q)(k_descale K)^T) (v_descale V). The kernel rounds
the probabilities fed to the second product to E4M3 (3 mantissa bits), so its error bound
is derived from that rounding, row by row:
    |O_ic - O64_ic| <= 2^-4 * v_descale * sum_j P_ij |V_jc|  + half an ulp of O's type
(each P_ij carries a relative rounding error of at most 2^-4, half an E4M3 ulp; l is summed
from the unrounded fp32 values) plus 1e-3 for the fp32 arithmetic and the approximate
exp2. L does not see that rounding and keeps the forward's 1e-3 bound.

A second test makes every probability an exact power of two (scores that are integers in
log2 units), so the E4M3 rounding is exact and the output must match the oracle to the
output rounding: this pins the packing of P (four keys per TMEM column) and the V^T
operand key by key."""
import ctypes
import math

import numpy as np
import pytest
import torch

import gen
from tests.fa_testlib import TOL_L, half_ulp

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


def run_fp8(q, k, v, scale, causal, qd=1.0, kd=1.0, vd=1.0, out=gen.BF16):
    fa = _fa()
    dev = torch.device("cuda:0")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    qg, kg, vg = (t.contiguous().view(torch.uint8).to(dev) for t in (q, k, v))
    O = torch.full((B, H, Nq, d), float("nan"), dtype=gen.torch_dtype(out), device=dev)
    L = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    nws = fa.fa_fwd_fp8_workspace_bytes(B, H, Nk, d)
    ws = torch.full((nws,), 0xAB, dtype=torch.uint8, device=dev)  # garbage: must be overwritten
    rc = fa.fa_fwd_fp8(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), O.data_ptr(), L.data_ptr(),
                       B, H, Nq, Nk, d, scale, causal, qd, kd, vd,
                       fa.FA_BF16 if out == gen.BF16 else fa.FA_F16, ws.data_ptr(), nws,
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, f"fa_fwd_fp8 rc={rc} ({fa.strerror(rc)})"
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
    return O.cpu(), L.cpu()


def _f64(t):
    return gen.to_f64_numpy(t)


def _probs64(Q, K, scale, causal, rows):
    """P of the selected query rows of one head (float64), for the error bound only."""
    S = scale * Q[rows] @ K.T
    if causal:
        S = np.where(np.arange(K.shape[0])[None, :] > rows[:, None], -np.inf, S)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    return P / P.sum(axis=1, keepdims=True)


def check(q, k, v, O, L, scale, causal, qd, kd, vd, out, rows=None):
    import oracle
    Q, K, V = _f64(q) * qd, _f64(k) * kd, _f64(v) * vd
    B, H, Nq, d = Q.shape
    if rows is None:
        Oref, Lref = oracle.attention(Q, K, V, scale, causal)
        Oref, Lref = Oref.reshape(-1, d), Lref.reshape(-1)
        rows = np.arange(B * H * Nq)
    else:
        Oref, Lref = oracle.attention_rows(Q, K, V, scale, causal, rows)
    Ok = O.double().numpy().reshape(-1, d)[rows]
    Lk = L.double().numpy().reshape(-1)[rows]
    assert np.all(np.isfinite(Ok)) and np.all(np.isfinite(Lk))
    bound = np.empty_like(Oref)
    for bh in np.unique(rows // Nq):
        sel = np.nonzero(rows // Nq == bh)[0]
        P = _probs64(Q.reshape(B * H, Nq, d)[bh], K.reshape(B * H, -1, d)[bh], scale, causal,
                     rows[sel] % Nq)
        bound[sel] = 2.0 ** -4 * (P @ np.abs(V.reshape(B * H, -1, d)[bh]))
    tol = bound + half_ulp(Oref, out) + 1e-3
    err = np.abs(Ok - Oref)
    assert np.all(err <= tol), (float(err.max()), float((err / tol).max()))
    assert np.abs(Lk - Lref).max() <= TOL_L
    return float(err.max()), float(np.sqrt((err ** 2).mean())), float(bound.mean())


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.float32).to(torch.float8_e4m3fn)


@pytest.mark.parametrize("causal", [False, True])
def test_dyadic_probabilities_are_exact(oracle_mod, causal):
    """Q = e_0, K_j = k_j e_0 with k_j in {0, -1, ..., -7} and scale = ln 2: every score is
    an integer in log2 units, every probability relative to the row max a power of two,
    exactly representable in E4M3. V_j = (1 + j div 128) e_(perm(j mod 128)) spreads the
    keys of the four K/V tiles over the columns with distinct weights."""
    B, H, Nq, Nk, d = 1, 2, 300, 500, 128
    rng = np.random.default_rng(17)
    Q = np.zeros((B, H, Nq, d)); Q[..., 0] = 1.0
    K = np.zeros((B, H, Nk, d)); K[..., 0] = -rng.integers(0, 8, size=(B, H, Nk))
    V = np.zeros((B, H, Nk, d))
    perm = rng.permutation(d)
    for j in range(Nk):
        V[:, :, j, perm[j % d]] = 1 + j // d
    q, k, v = _e4m3(Q), _e4m3(K), _e4m3(V)
    assert np.array_equal(_f64(k), K) and np.array_equal(_f64(v), V)
    scale = math.log(2.0)
    O, L = run_fp8(q, k, v, scale, causal)
    Oref, Lref = oracle_mod.attention(Q, K, V, scale, causal)
    err = np.abs(O.double().numpy() - Oref)
    assert np.all(err <= half_ulp(Oref, gen.BF16) + 1e-6), float(err.max())
    assert np.abs(L.double().numpy() - Lref).max() <= TOL_L


CASES = [
    # B, H, Nq, Nk, causal, q_descale, k_descale, v_descale, out
    (1, 1, 128, 128, False, 1.0, 1.0, 1.0, gen.BF16),
    (1, 1, 128, 128, True, 1.0, 1.0, 1.0, gen.F16),
    (2, 3, 300, 257, False, 0.5, 2.0, 0.25, gen.BF16),
    (1, 2, 257, 600, True, 0.37, 1.3, 1.7, gen.BF16),
    (2, 2, 1000, 1000, False, 1.0, 1.0, 1.0, gen.BF16),
    (1, 4, 700, 130, True, 1.0, 1.0, 0.1, gen.F16),
    (1, 2, 1000, 4097, False, 0.25, 0.25, 4.0, gen.BF16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_{}_d{}-{}-{}_{}".format(
    c[0], c[1], c[2], c[3], "causal" if c[4] else "full", c[5], c[6], c[7], c[8]))
def test_fp8_matches_oracle(oracle_mod, case):
    B, H, Nq, Nk, causal, qd, kd, vd, out = case
    w = gen.custom(B, H, Nq, Nk, 128, gen.FP8, causal, seed=600 + Nq + Nk)
    q, k, v = gen.make_qkv(w)
    O, L = run_fp8(q, k, v, w.scale, causal, qd, kd, vd, out)
    print(w.describe(), "max err, rms err, mean bound", check(q, k, v, O, L, w.scale, causal, qd, kd, vd, out))


@pytest.mark.parametrize("name", sorted(gen.FP8_WORKLOADS))
def test_fp8_full_size_whole_output(oracle_mod, name):
    """The E4M3 versions of the two benchmark workloads at full size: every element of O and
    L against the oracle on the decoded inputs, with the bound of the E4M3 rounding of P."""
    w = gen.FP8_WORKLOADS[name]
    q, k, v = gen.make_qkv(w)
    O, L = run_fp8(q, k, v, w.scale, w.causal)
    print(name, "max err, rms err, mean bound",
          check(q, k, v, O, L, w.scale, w.causal, 1.0, 1.0, 1.0, gen.BF16))


def test_fp8_errors_and_determinism():
    fa = _fa()
    P = 1 << 20
    base = (P, P, P, P, P, 1, 1, 128, 128)
    assert fa.fa_fwd_fp8(*base, 64, 0.1, 0, 1.0, 1.0, 1.0, fa.FA_BF16, P, 1 << 20, None) == fa.FA_ERR_HEAD_DIM
    assert fa.fa_fwd_fp8(*base, 128, 0.1, 0, 0.0, 1.0, 1.0, fa.FA_BF16, P, 1 << 20, None) == fa.FA_ERR_SCALE
    assert fa.fa_fwd_fp8(*base, 128, 0.1, 0, 1.0, float("nan"), 1.0, fa.FA_BF16, P, 1 << 20, None) == fa.FA_ERR_SCALE
    assert fa.fa_fwd_fp8(*base, 128, 0.1, 0, 1.0, 1.0, 1.0, fa.FA_BF16, P, 16, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_fp8(*base, 128, 0.1, 0, 1.0, 1.0, 1.0, 5, P, 1 << 20, None) == fa.FA_ERR_DTYPE
    w = gen.custom(2, 2, 333, 444, 128, gen.FP8, True, seed=5)
    q, k, v = gen.make_qkv(w)
    a = run_fp8(q, k, v, w.scale, True)
    b = run_fp8(q, k, v, w.scale, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
