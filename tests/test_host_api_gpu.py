"""fa_fwd_host (host buffers, copies overlapped with the computation) against fa_fwd on the
same inputs: the same kernel computes every row the same way, so the results must be
bit-identical, for pinned and for pageable host memory, whatever the chunking of heads."""
import ctypes

import pytest
import torch

import gen
from tests.fa_testlib import run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()


def run_host(w, q, k, v, pinned=True):
    import exact_attention_forward_02_gb300 as fa
    hq, hk, hv = (t.contiguous().pin_memory() if pinned else t.contiguous() for t in (q, k, v))
    O = torch.full((w.B, w.H, w.Nq, w.d), float("nan"), dtype=q.dtype)
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32)
    if pinned:
        O, L = O.pin_memory(), L.pin_memory()
    nws = fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda:0")
    st = torch.cuda.current_stream()
    rc = fa.fa_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), O.data_ptr(), L.data_ptr(),
                        w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                        fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16, ws.data_ptr(), nws,
                        ctypes.c_void_p(st.cuda_stream))
    assert rc == 0, fa.strerror(rc)
    st.synchronize()
    assert fa.fa_last_status() == 0
    return O, L


# Chunks hold enough heads for 8 MiB per tensor (the smaller of Q and K), capped at the
# head count; the last chunk has a quarter of that (at least one head).
CASES = [
    (1, 1, 128, 128, 64, gen.F16, False),       # one chunk of one head
    (2, 3, 300, 257, 64, gen.F16, True),        # small heads: 5 + 1
    (2, 8, 1000, 1000, 128, gen.BF16, True),    # 12 + 4
    (3, 7, 257, 600, 128, gen.BF16, False),     # 16 + 5
    (1, 13, 129, 131, 64, gen.F16, False),      # 10 + 3
    (3, 7, 8192, 8192, 128, gen.BF16, True),    # 2 MiB heads: 4 4 4 4 4 1, the 4-slot ring wraps
    (1, 6, 8192, 4096, 128, gen.BF16, False),   # 1 MiB K/V heads: 5 + 1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_api_is_fa_fwd(case, pinned):
    B, H, Nq, Nk, d, dt, causal = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=70 + H)
    q, k, v = gen.make_qkv(w)
    O0, L0 = run_cuda(w, q, k, v)
    O1, L1 = run_host(w, q, k, v, pinned)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)


def test_host_api_full_size_workload():
    w = gen.WORKLOADS["b2h8_n8192_d128_causal"]
    q, k, v = gen.make_qkv(w)
    O0, L0 = run_cuda(w, q, k, v)
    O1, L1 = run_host(w, q, k, v, True)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)


def test_host_api_full_size_full_attention():
    """The full N=4096 workload through fa_fwd_host (chunks of 8, 6 and 2 heads): every
    element of O and L against the oracle, and bit for bit against fa_fwd."""
    from tests.fa_testlib import compare, oracle_whole
    w = gen.WORKLOADS["b2h8_n4096_d128_full"]
    (q, k, v), (Oref, Lref) = oracle_whole(w.name)
    O1, L1 = run_host(w, q, k, v, True)
    r = compare(w, O1, L1, Oref, Lref)
    assert r["raw_ok"], r
    O0, L0 = run_cuda(w, q, k, v)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
