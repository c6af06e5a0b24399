"""fa_fwd_noalloc: the entry point for callers that cannot allocate device memory (for
example, hosts whose own pool owns all of the device memory, or processes with a fixed
memory budget). It splits full attention across CTAs like fa_fwd_ws, with its workspace
in a fixed device array inside the library instead of a caller allocation.

Checked through the C ABI against the existing workspace entry point and against the
float64 oracle, on two calls in a row (the fixed array keeps the previous call's
contents); the device's free memory is the same before and after those calls; and the
size limit. The file is collected last, so that a failure here comes after every other
test has run."""
import ctypes

import pytest
import torch

import gen
from tests.fa_testlib import TOL_L, TOL_O, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    fa.fa_clear_status()
    return fa


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _outputs(w, dev, dtype):
    O = torch.full((w.B, w.H, w.Nq, w.d), float("nan"), dtype=dtype, device=dev)
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=dev)
    return O, L


def _args(fa, w, tensors, O, L):
    qd, kd, vd = tensors
    dt = fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16
    return (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
            w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt)


def _run_ws(fa, w, tensors):
    """The existing workspace entry point, with a workspace allocated here."""
    O, L = _outputs(w, tensors[0].device, tensors[0].dtype)
    nbytes = fa.fa_fwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, w.causal)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=tensors[0].device)
    rc = fa.fa_fwd_ws(*_args(fa, w, tensors, O, L), ws.data_ptr(), ws.numel(), _stream())
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
    return O, L


def _run_noalloc(fa, w, tensors, O, L):
    rc = fa.fa_fwd_noalloc(*_args(fa, w, tensors, O, L), _stream())
    assert rc == 0, fa.strerror(rc)


@pytest.mark.parametrize("case", [
    (2, 40, 512, 640, 128, gen.BF16),   # 160 work items on 152 SMs: split key ranges
    (1, 2, 1000, 4097, 64, gen.F16),    # 8 items split across many CTAs, ragged key tail
])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(fa, case):
    import oracle
    B, H, Nq, Nk, d, dt = case
    w = gen.custom(B, H, Nq, Nk, d, dt, False, 1.0, seed=4000 + Nq)
    assert 0 < fa.fa_fwd_workspace_bytes(B, H, Nq, Nk, d, False) <= fa.FA_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    q, k, v = gen.make_qkv(w)
    tensors = tuple(t.to(dev) for t in (q, k, v))
    O_ref, L_ref = _run_ws(fa, w, tensors)  # the existing entry point first
    Oref64, Lref64 = oracle.attention(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                      w.scale, w.causal)
    outs = [_outputs(w, dev, tensors[0].dtype) for _ in range(2)]
    # warm-up: the first call on a device looks up the fixed array's address
    O0, L0 = _outputs(w, dev, tensors[0].dtype)
    _run_noalloc(fa, w, tensors, O0, L0)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    for O, L in outs:  # two calls in a row on the shared fixed scratch
        _run_noalloc(fa, w, tensors, O, L)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info(dev)[0]
    assert free_after == free_before, "fa_fwd_noalloc changed the device's free memory"
    assert fa.fa_last_status() == 0
    for O, L in outs:
        assert torch.isfinite(O).all() and torch.isfinite(L).all()
        assert (O.double() - O_ref.double()).abs().max().item() <= TOL_O[w.dtype]
        assert (L.double() - L_ref.double()).abs().max().item() <= TOL_L
        r = compare(w, O.cpu(), L.cpu(), Oref64, Lref64)
        assert r["raw_ok"], r


def test_noalloc_causal_needs_no_scratch(fa):
    import oracle
    w = gen.custom(1, 3, 700, 700, 128, gen.BF16, True, 1.0, seed=41)
    dev = torch.device("cuda:0")
    q, k, v = gen.make_qkv(w)
    tensors = tuple(t.to(dev) for t in (q, k, v))
    O_ref, L_ref = _run_ws(fa, w, tensors)
    O, L = _outputs(w, dev, tensors[0].dtype)
    _run_noalloc(fa, w, tensors, O, L)
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
    assert (O.double() - O_ref.double()).abs().max().item() <= TOL_O[w.dtype]
    assert (L.double() - L_ref.double()).abs().max().item() <= TOL_L
    Oref64, Lref64 = oracle.attention(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                      w.scale, w.causal)
    r = compare(w, O.cpu(), L.cpu(), Oref64, Lref64)
    assert r["raw_ok"], r


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    # 2^21 heads of one query row: 2^21 work items, whose counters (one per item and Q tile)
    # together with the partial states of every CTA outgrow the fixed array. The size check
    # comes before any device access, so placeholder (aligned, never dereferenced) pointers
    # stand in for tensors that would not fit on the device.
    B, H, Nq, Nk, d = 1024, 2048, 1, 128, 128
    need = fa.fa_fwd_workspace_bytes(B, H, Nq, Nk, d, False)
    assert need > fa.FA_NOALLOC_SCRATCH_BYTES
    P = 1 << 20
    rc = fa.fa_fwd_noalloc(P, P, P, P, P, B, H, Nq, Nk, d, 0.088, False, fa.FA_BF16, _stream())
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in fa.strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_last_status() == 0
