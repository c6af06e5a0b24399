"""GPU parity of the workspace entry point (fa_fwd_ws): full attention whose key range is
split across CTAs (stream-K) and merged with the online-softmax combine, against the
float64 oracle; repeated calls on one workspace (its counters must return to zero)."""
import ctypes

import numpy as np
import pytest
import torch

import gen
from tests.fa_testlib import compare, oracle_whole, run_cuda_ws

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()
    return fa


def run_ws(w, q, k, v, ws=None, calls=1):
    import exact_attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    nbytes = fa.fa_fwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, w.causal)
    if ws is None:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(calls):
        O = torch.full((w.B, w.H, w.Nq, w.d), float("nan"), dtype=q.dtype, device=dev)
        L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=dev)
        rc = fa.fa_fwd_ws(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                          w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                          fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16,
                          ws.data_ptr(), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, fa.strerror(rc)
        torch.cuda.synchronize()
        assert fa.fa_last_status() == 0
        outs.append((O.cpu(), L.cpu()))
    return outs, nbytes


CASES = [
    (1, 1, 128, 128, 64, gen.F16),
    (1, 1, 128, 8192, 128, gen.BF16),      # one item, 64 tiles: split across 64 CTAs
    (1, 2, 1000, 4097, 64, gen.F16),       # ragged key tail inside split pieces
    (2, 3, 1000, 1000, 64, gen.F16),
    (1, 3, 300, 257, 128, gen.BF16),
    (1, 1, 3, 300, 128, gen.F16),
    (2, 40, 512, 640, 128, gen.BF16),      # 160 items on 152 SMs
    (4, 12, 1000, 4097, 64, gen.F16),      # the cross-attention workload's shape
    (8, 64, 256, 256, 64, gen.F16),        # 512 items of 2 K/V tiles: ranges span several
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}".format(*c))
def test_streamk_full_compare_and_reuse(case):
    import oracle
    B, H, Nq, Nk, d, dt = case
    w = gen.custom(B, H, Nq, Nk, d, dt, False, 1.0, seed=2000 + sum(case[:5]))
    q, k, v = gen.make_qkv(w)
    outs, nbytes = run_ws(w, q, k, v, calls=3)
    Oref, Lref = oracle.attention(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                  w.scale, w.causal)
    for O, L in outs:
        r = compare(w, O, L, Oref, Lref)
        print(w.describe(), "workspace", nbytes, r)
        assert r["raw_ok"], r
    # the same workspace reused without re-zeroing gives the same bits every time
    for O, L in outs[1:]:
        assert torch.equal(O.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(L, outs[0][1])


@pytest.mark.parametrize("name", ["b2h8_n4096_d128_full", "b4h12_q1000_k4097_d64_cross"])
def test_streamk_full_size_whole_output(name):
    """The two full-attention workloads at full size, launched as the benchmark launches
    them (fa_fwd_ws, two calls on one workspace): every element against the oracle."""
    w = gen.WORKLOADS[name]
    (q, k, v), (Oref, Lref) = oracle_whole(name)
    outs, nbytes = run_cuda_ws(w, q, k, v, calls=2)
    assert nbytes > 0
    for O, L in outs:
        r = compare(w, O, L, Oref, Lref)
        print(w.name, r)
        assert r["raw_ok"], r
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


def test_streamk_agrees_with_plain_path():
    from tests.fa_testlib import run_cuda
    w = gen.custom(2, 5, 777, 1500, 128, gen.BF16, False, 1.0, seed=77)
    q, k, v = gen.make_qkv(w)
    (O1, L1), = run_ws(w, q, k, v)[0]
    O2, L2 = run_cuda(w, q, k, v)
    assert (O1.double() - O2.double()).abs().max().item() <= 2e-2
    assert (L1 - L2).abs().max().item() <= 1e-5


def test_workspace_errors_and_causal_ignores_it():
    import exact_attention_forward_02_gb300 as fa
    from tests.fa_testlib import run_cuda
    dev = torch.device("cuda:0")
    w = gen.custom(1, 1, 128, 4096, 128, gen.BF16, False, 1.0, seed=3)
    q, k, v = (t.to(dev) for t in gen.make_qkv(w))
    O = torch.empty((1, 1, 128, 128), dtype=torch.bfloat16, device=dev)
    L = torch.empty((1, 1, 128), dtype=torch.float32, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    need = fa.fa_fwd_workspace_bytes(1, 1, 128, 4096, 128, False)
    assert need > 0
    small = torch.zeros(need - 256, dtype=torch.uint8, device=dev)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(), 1, 1, 128, 4096, 128,
            w.scale)
    assert fa.fa_fwd_ws(*args, 0, fa.FA_BF16, small.data_ptr(), small.numel(), st) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_ws(*args, 0, fa.FA_BF16, 0, 0, st) == fa.FA_ERR_WORKSPACE
    # causal attention needs no workspace: NULL is accepted and the result matches fa_fwd
    assert fa.fa_fwd_workspace_bytes(1, 1, 128, 4096, 128, True) == 0
    assert fa.fa_fwd_ws(*args, 1, fa.FA_BF16, 0, 0, st) == 0
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
    wc = gen.custom(1, 1, 128, 4096, 128, gen.BF16, True, 1.0, seed=3)
    O2, L2 = run_cuda(wc, *gen.make_qkv(wc))
    assert torch.equal(O.cpu().view(torch.int16), O2.view(torch.int16))


@pytest.mark.parametrize("shape", [(2, 8, 4096, 4096, 128), (4, 12, 1000, 4097, 64), (1, 1, 128, 8192, 128)])
def test_workspace_size_is_the_documented_layout(shape):
    """fa_fwd_workspace_bytes = the partial states [CTA][slot 2][Q tile 2][d + 2][128 rows]
    fp32 (O~, m and l) and one int counter per (work item, Q tile), each part rounded up to 256 bytes,
    with one CTA per SM (or per K/V tile when there are fewer)."""
    import exact_attention_forward_02_gb300 as fa
    B, H, Nq, Nk, d = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_items = -(-Nq // 256) * B * H
    n_kv = -(-Nk // 128)
    G = min(n_items * n_kv, sms)
    up = lambda x: -(-x // 256) * 256  # noqa: E731
    expect = up(G * 2 * 2 * (d + 2) * 128 * 4) + up(n_items * 2 * 4)
    if n_items % sms == 0:
        expect = 0
    assert fa.fa_fwd_workspace_bytes(B, H, Nq, Nk, d, False) == expect
