"""The C ABI library loads on a machine without a GPU, exports every function that
include/*.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        # every function the header declares: "<type> name(" at the start of a statement
        names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_last_status" in names and "fa_strerror" in names, names


def test_library_exports_every_declared_symbol():
    import exact_attention_forward_02_gb300 as fa
    lib = ctypes.CDLL(fa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in include/*.h but not exported: {missing}"


def test_debug_build_exports_the_same_symbols_and_answers_its_hook():
    """libfa_debug.so (FA_DEBUG: device-side range checks) is the same C ABI; only it takes
    the workspace cut of fa_debug_cap_workspace, which makes no CUDA call."""
    import exact_attention_forward_02_gb300 as fa
    dbg = fa.load_library(fa.DEBUG_LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(dbg, n)]
    assert not missing, f"declared in include/*.h but not exported by the debug build: {missing}"
    assert dbg.fa_debug_cap_workspace(0) == 1
    assert dbg.fa_debug_cap_workspace(-1) == 1
    rel = fa.load_library(fa.LIB_PATH)
    assert rel.fa_debug_cap_workspace(0) == 0
    assert rel.fa_debug_cap_workspace(-1) == 0
    assert "debug" in fa.strerror(fa.FA_ERR_BOUNDS)


def test_status_strings():
    import exact_attention_forward_02_gb300 as fa
    for code, name in fa.STATUS.items():
        assert fa.strerror(code) and "unknown" not in fa.strerror(code), name
    assert "unknown" in fa.strerror(12345)


# Host-side checks run before any CUDA call, so they work without a GPU. Fake pointers
# (never dereferenced) stand in for device memory.
P = 1 << 20  # 16-byte aligned, non-null, never touched


@pytest.mark.parametrize("args,code", [
    ((0, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_NULL"),
    ((P, P, P, P, 0, 1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_NULL"),
    ((P, P, P, P, P, 1, 1, 128, 128, 96, 0.125, 0, 1), "FA_ERR_HEAD_DIM"),
    ((P, P, P, P, P, 1, 1, 128, 128, 256, 0.125, 0, 1), "FA_ERR_HEAD_DIM"),
    ((P, P, P, P, P, -1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_SHAPE"),
    ((P, P, P, P, P, 1, 1, -5, 128, 64, 0.125, 0, 1), "FA_ERR_SHAPE"),
    ((P, P, P, P, P, 1, 1, 128, -1, 64, 0.125, 0, 1), "FA_ERR_SHAPE"),
    ((P, P, P, P, P, 1, 1, 128, 0, 64, 0.125, 0, 1), "FA_ERR_EMPTY_KEYS"),
    ((P, P, P, P, P, 1, 1, 128, 128, 64, float("nan"), 0, 1), "FA_ERR_SCALE"),
    ((P, P, P, P, P, 1, 1, 128, 128, 64, float("inf"), 0, 1), "FA_ERR_SCALE"),
    ((P, P, P, P, P, 1, 1, 128, 128, 64, -0.5, 0, 1), "FA_ERR_SCALE"),
    ((P + 2, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_ALIGN"),
    ((P, P, P + 8, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_ALIGN"),
    ((P, P, P, P, P + 2, 1, 1, 128, 128, 64, 0.125, 0, 1), "FA_ERR_ALIGN"),
    ((P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 2), "FA_ERR_DTYPE"),
    ((P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, -1), "FA_ERR_DTYPE"),
    ((P, P, P, P, P, 70000, 70000, 128, 128, 64, 0.125, 0, 1), "FA_ERR_SHAPE"),
    # nothing to compute: success without touching the pointers (even NULL ones)
    ((0, 0, 0, 0, 0, 0, 4, 128, 128, 64, 0.125, 0, 1), "FA_OK"),
    ((0, 0, 0, 0, 0, 2, 4, 0, 128, 64, 0.125, 1, 1), "FA_OK"),
    ((0, 0, 0, 0, 0, 2, 4, 0, 0, 128, 0.125, 1, 0), "FA_OK"),
])
def test_host_argument_checks(args, code):
    import exact_attention_forward_02_gb300 as fa
    *a, dt = args
    rc = fa.fa_fwd(*a, dt, None)
    assert rc == getattr(fa, code), (rc, fa.strerror(rc))


def test_selftest_rejects_out_of_range_limit():
    import exact_attention_forward_02_gb300 as fa
    assert fa.fa_selftest_wait_timeout(0) == fa.FA_ERR_SHAPE
    assert fa.fa_selftest_wait_timeout(2_000_000) == fa.FA_ERR_SHAPE


def test_wait_limit_setter_checks_its_range_and_makes_no_cuda_call():
    """fa_set_wait_limit_us accepts FA_WAIT_LIMIT_MIN_US..FA_WAIT_LIMIT_MAX_US, rejects the
    rest with FA_ERR_RANGE and then keeps the previous limit; it touches no device."""
    import exact_attention_forward_02_gb300 as fa
    assert fa.fa_get_wait_limit_us() == fa.FA_WAIT_LIMIT_DEFAULT_US == 2_000_000
    try:
        for bad in (0, 99, fa.FA_WAIT_LIMIT_MAX_US + 1, 1 << 63, -1):
            assert fa.fa_set_wait_limit_us(bad) == fa.FA_ERR_RANGE, bad
            assert fa.fa_get_wait_limit_us() == fa.FA_WAIT_LIMIT_DEFAULT_US
        for good in (fa.FA_WAIT_LIMIT_MIN_US, 5_000_000, fa.FA_WAIT_LIMIT_MAX_US):
            assert fa.fa_set_wait_limit_us(good) == fa.FA_OK
            assert fa.fa_get_wait_limit_us() == good
    finally:
        assert fa.fa_set_wait_limit_us(fa.FA_WAIT_LIMIT_DEFAULT_US) == fa.FA_OK
    assert "range" in fa.strerror(fa.FA_ERR_RANGE)


def test_workspace_variant_host_checks():
    """fa_fwd_ws shares fa_fwd's host-side checks; sizes are 0 for invalid or causal calls."""
    import exact_attention_forward_02_gb300 as fa
    assert fa.fa_fwd_ws(0, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1, 0, 0, None) == fa.FA_ERR_NULL
    assert fa.fa_fwd_ws(P, P, P, P, P, 1, 1, 128, 128, 32, 0.125, 0, 1, 0, 0, None) == fa.FA_ERR_HEAD_DIM
    assert fa.fa_fwd_ws(0, 0, 0, 0, 0, 0, 1, 128, 128, 64, 0.125, 0, 1, 0, 0, None) == fa.FA_OK
    # a misaligned workspace is rejected before any CUDA call
    assert fa.fa_fwd_ws(P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1, P + 16, 1 << 20, None) == fa.FA_ERR_ALIGN
    assert fa.fa_fwd_workspace_bytes(1, 1, 128, 128, 64, True) == 0
    assert fa.fa_fwd_workspace_bytes(1, 1, 128, 128, 96, False) == 0
    assert fa.fa_fwd_workspace_bytes(0, 1, 128, 128, 64, False) == 0


def test_backward_host_checks():
    import exact_attention_forward_02_gb300 as fa
    base = (P, P, P, P, P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1)
    assert fa.fa_bwd(0, *base[1:], P, 1 << 20, None) == fa.FA_ERR_NULL
    assert fa.fa_bwd(*base[:4], 0, *base[5:], P, 1 << 20, None) == fa.FA_ERR_NULL      # dO
    assert fa.fa_bwd(*base[:6], P + 2, *base[7:], P, 1 << 20, None) == fa.FA_ERR_ALIGN  # dQ
    assert fa.fa_bwd(*base[:13], 96, *base[14:], P, 1 << 20, None) == fa.FA_ERR_HEAD_DIM
    assert fa.fa_bwd(*base, 0, 0, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd(*base, P + 4, 1 << 20, None) == fa.FA_ERR_ALIGN
    assert fa.fa_bwd_workspace_bytes(2, 3, 100, 50, 64) == 2 * 3 * 100 * 4 + (256 - (2 * 3 * 100 * 4) % 256) % 256
    assert fa.fa_bwd_workspace_bytes(2, 3, 100, 50, 96) == 0


def test_dropout_host_checks():
    import exact_attention_forward_02_gb300 as fa
    base = (P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1)
    for bad in (1.0, 1 - 2.0 ** -17, 2.0, -1e-3, float("nan"), float("inf"), -float("inf")):
        assert fa.fa_fwd_dropout(*base, bad, 1, 2, None) == fa.FA_ERR_DROPOUT, bad
        assert fa.fa_dropout_mask(P, 1, 1, 8, 8, bad, 1, 2, None) == fa.FA_ERR_DROPOUT, bad
    # the forward's own checks still apply with a valid probability
    assert fa.fa_fwd_dropout(0, *base[1:], 0.1, 1, 2, None) == fa.FA_ERR_NULL
    assert fa.fa_fwd_dropout(*base[:9], 96, *base[10:], 0.1, 1, 2, None) == fa.FA_ERR_HEAD_DIM
    assert fa.fa_fwd_dropout(*base[:10], float("nan"), *base[11:], 0.1, 1, 2, None) == fa.FA_ERR_SCALE
    # nothing to do: no-ops that touch no pointer
    assert fa.fa_fwd_dropout(0, 0, 0, 0, 0, 0, 1, 128, 128, 64, 0.125, 0, 1, 0.1, 1, 2, None) == fa.FA_OK
    assert fa.fa_dropout_mask(0, 1, 1, 0, 8, 0.1, 1, 2, None) == fa.FA_OK
    assert fa.fa_dropout_mask(0, 1, 1, 8, 8, 0.1, 1, 2, None) == fa.FA_ERR_NULL
    assert fa.fa_dropout_mask(P, -1, 1, 8, 8, 0.1, 1, 2, None) == fa.FA_ERR_SHAPE


def test_host_buffer_api_host_checks():
    import exact_attention_forward_02_gb300 as fa
    base = (P, P, P, P, P, 1, 1, 128, 128, 64, 0.125, 0, 1)
    need = fa.fa_fwd_host_workspace_bytes(1, 1, 128, 128, 64)
    assert need >= 128 * 64 * 2 * 4 + 128 * 4
    assert fa.fa_fwd_host_workspace_bytes(1, 1, 128, 128, 96) == 0
    assert fa.fa_fwd_host(*base, 0, 0, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_host(*base, P, need - 1, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_host(*base, P + 16, need, None) == fa.FA_ERR_ALIGN
    assert fa.fa_fwd_host(0, *base[1:], P, need, None) == fa.FA_ERR_NULL
    assert fa.fa_fwd_host(*base[:9], 96, *base[10:], P, need, None) == fa.FA_ERR_HEAD_DIM
    # 1 MiB per head and tensor: chunks of 8 heads (8 MiB copies), the last one of 2, so
    # 16 heads run as 8 + 6 + 2 through three slots of 8 heads each (Q, K, V, O and L)
    assert fa.fa_fwd_host_workspace_bytes(2, 8, 4096, 4096, 128) == 3 * (
        8 * (4096 * 128 * 2) * 4 + ((8 * 4096 * 4 + 255) // 256) * 256)
    # 8 MiB per head and tensor: one head per chunk, four slots
    assert fa.fa_fwd_host_workspace_bytes(1, 6, 32768, 32768, 128) == 4 * (
        (32768 * 128 * 2) * 4 + 32768 * 4)
