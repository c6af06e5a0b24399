"""The range-checked build (libfa_debug.so, compiled with FA_DEBUG) on the GPU.

That build checks, on the device, every stream-K workspace access (the partial states a CTA
stores, the per-item counters, the pieces a merging CTA reads) against the workspace's
layout, and the coordinates of every TMA tile copy against the tensors' extents; a
violation records FA_ERR_BOUNDS and the access is skipped (a load is only recorded). Here:
no check fires on the shapes whose partial states and tiles cover the edges (ragged key
tails, one item over 64 CTAs, more items than SMs, the full-size workloads), the results
are bit-identical to the release build's, and a workspace cut through the test hook makes
the checks fire, with every access still inside the real workspace, and leaves the library
usable."""
import ctypes

import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_02_gb300 as fa
    rel = fa.load_library(fa.LIB_PATH)
    dbg = fa.load_library(fa.DEBUG_LIB_PATH)
    assert dbg.fa_clear_status() == 0 and rel.fa_clear_status() == 0
    assert dbg.fa_debug_cap_workspace(-1) == 1
    yield fa, rel, dbg
    dbg.fa_debug_cap_workspace(-1)


def _dtype(fa, w):
    return fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16


def _run(fa, lib, w, qkv, entry):
    """One call of `entry` ("fa_fwd" or "fa_fwd_ws") of the given library build; O and L
    start as NaN so that a skipped store shows."""
    dev = torch.device("cuda:0")
    q, k, v = qkv
    O = torch.full((w.B, w.H, w.Nq, w.d), float("nan"), dtype=q.dtype, device=dev)
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(),
            w.B, w.H, w.Nq, w.Nk, w.d, w.scale, int(w.causal), _dtype(fa, w))
    if entry == "fa_fwd_ws":
        n = max(int(lib.fa_fwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, int(w.causal))), 256)
        ws = torch.zeros(n, dtype=torch.uint8, device=dev)
        rc = lib.fa_fwd_ws(*args, ws.data_ptr(), ws.numel(), st)
    else:
        rc = lib.fa_fwd(*args, st)
    assert rc == 0, fa.strerror(rc)
    status = lib.fa_last_status()
    return O.cpu(), L.cpu(), status


def _same(a, b):
    return torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])


CASES = [
    # (B, H, Nq, Nk, d, dtype, causal, entry)
    (1, 1, 128, 8192, 128, gen.BF16, False, "fa_fwd_ws"),  # one item split over 64 CTAs
    (1, 2, 1000, 4097, 64, gen.F16, False, "fa_fwd_ws"),   # ragged key tail inside pieces
    (2, 40, 512, 640, 128, gen.BF16, False, "fa_fwd_ws"),  # 160 items on the SMs
    (1, 3, 300, 257, 128, gen.BF16, False, "fa_fwd_ws"),
    (1, 1, 3, 300, 128, gen.F16, False, "fa_fwd_ws"),
    (1, 2, 1000, 1000, 128, gen.BF16, True, "fa_fwd"),     # causal, ragged Q tail
    (2, 3, 300, 4097, 64, gen.F16, False, "fa_fwd"),
    (8, 64, 256, 256, 64, gen.F16, False, "fa_fwd_ws"),    # ranges over several short items
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}k{}_d{}_{}_{}_{}".format(
    *c[:6], "causal" if c[6] else "full", c[7]))
def test_no_check_fires_and_results_match_release(libs, case):
    fa, rel, dbg = libs
    B, H, Nq, Nk, d, dt, causal, entry = case
    w = gen.custom(B, H, Nq, Nk, d, dt, causal, 1.0, seed=4100 + Nq + Nk + d)
    dev = torch.device("cuda:0")
    qkv = tuple(t.to(dev) for t in gen.make_qkv(w))
    r = _run(fa, rel, w, qkv, entry)
    g = _run(fa, dbg, w, qkv, entry)
    assert r[2] == 0 and g[2] == 0, (fa.strerror(r[2]), fa.strerror(g[2]))
    assert not torch.isnan(g[0].float()).any() and not torch.isnan(g[1]).any()
    assert _same(r, g)


@pytest.mark.parametrize("name,entry", [("b2h8_n4096_d128_full", "fa_fwd_ws"),
                                        ("b4h12_q1000_k4097_d64_cross", "fa_fwd_ws"),
                                        ("b2h8_n8192_d128_causal", "fa_fwd")])
def test_full_size_workloads_pass_the_checks(libs, name, entry):
    fa, rel, dbg = libs
    w = gen.WORKLOADS[name]
    dev = torch.device("cuda:0")
    qkv = tuple(t.to(dev) for t in gen.make_qkv(w))
    r = _run(fa, rel, w, qkv, entry)
    g = _run(fa, dbg, w, qkv, entry)
    assert r[2] == 0 and g[2] == 0, (fa.strerror(r[2]), fa.strerror(g[2]))
    assert _same(r, g)


def test_cut_workspace_makes_the_checks_fire_and_the_library_recovers(libs):
    """The hook tells the kernel that the partial-state area is 0 floats long: every
    partial-state store is skipped and every piece read is redirected to the workspace's
    start, all inside the real allocation. The status word says FA_ERR_BOUNDS; after the
    cut is removed and the status cleared the same call is right again."""
    fa, rel, dbg = libs
    w = gen.custom(2, 40, 512, 640, 128, gen.BF16, False, 1.0, seed=4242)
    dev = torch.device("cuda:0")
    qkv = tuple(t.to(dev) for t in gen.make_qkv(w))
    ref = _run(fa, rel, w, qkv, "fa_fwd_ws")
    assert ref[2] == 0
    try:
        assert dbg.fa_debug_cap_workspace(0) == 1
        bad = _run(fa, dbg, w, qkv, "fa_fwd_ws")
        assert bad[2] == fa.FA_ERR_BOUNDS, fa.strerror(bad[2])
        # the release build ignores the hook
        assert rel.fa_debug_cap_workspace(0) == 0
        assert _run(fa, rel, w, qkv, "fa_fwd_ws")[2] == 0
    finally:
        dbg.fa_debug_cap_workspace(-1)
        rel.fa_debug_cap_workspace(-1)
    assert dbg.fa_clear_status() == 0
    good = _run(fa, dbg, w, qkv, "fa_fwd_ws")
    assert good[2] == 0 and _same(ref, good)
