"""Exact fused attention forward on GB300 (sm_103a): a thin ctypes binding over libfa.so.

The binding only marshals arguments: every step of the computation runs in the CUDA
kernels of ``libfa.so`` (source in ``csrc/``, C ABI in ``include/fa_fwd.h``). There is
no CPU or PyTorch fallback: importing this package fails loudly when the library has
not been built (``python -c "import __graft_entry__ as g; g.build()"``).

Function names follow the C ABI:
    fa_fwd(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, stream) -> status
plus a tensor-level convenience ``attention(q, k, v, causal, scale)`` -> (O, L).
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")
# The same library built with FA_DEBUG: every stream-K workspace access and TMA tile
# coordinate of the forward kernel is range-checked on the device, and a violation is
# recorded as FA_ERR_BOUNDS. Tests load it with load_library; FA_LIBRARY=debug in the
# environment makes it the library this module binds.
DEBUG_LIB_PATH = os.path.join(PKG, "libfa_debug.so")

FA_F16 = 0
FA_BF16 = 1

STATUS = {
    0: "FA_OK", -1: "FA_ERR_NULL", -2: "FA_ERR_HEAD_DIM", -3: "FA_ERR_SHAPE",
    -4: "FA_ERR_EMPTY_KEYS", -5: "FA_ERR_SCALE", -6: "FA_ERR_ALIGN", -7: "FA_ERR_DTYPE",
    -8: "FA_ERR_CUDA", -9: "FA_ERR_TENSOR_MAP", -10: "FA_ERR_DEVICE", -11: "FA_ERR_TIMEOUT",
    -12: "FA_ERR_WORKSPACE", -13: "FA_ERR_SCRATCH_LIMIT", -14: "FA_ERR_DROPOUT",
    -15: "FA_ERR_RANGE", -16: "FA_ERR_BOUNDS",
}
FA_WAIT_LIMIT_DEFAULT_US = 2_000_000
FA_WAIT_LIMIT_MIN_US = 100
FA_WAIT_LIMIT_MAX_US = 3_600_000_000
FA_NOALLOC_SCRATCH_BYTES = 48 << 20
globals().update({v: k for k, v in STATUS.items()})


class FAError(RuntimeError):
    def __init__(self, code: int, what: str = "fa_fwd"):
        self.code = code
        super().__init__(f"{what} failed: {STATUS.get(code, code)} ({strerror(code)})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open one build of the library (release or FA_DEBUG) with its C signatures declared."""
    if not os.path.exists(path):
        raise ImportError(
            f"{os.path.basename(path)} is not built ({path} missing); run __graft_entry__.build() "
            "first. There is no fallback implementation.")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
    lib.fa_fwd_ws.restype = ctypes.c_int
    lib.fa_fwd_ws.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_noalloc.restype = ctypes.c_int
    lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
    lib.fa_fwd_host.restype = ctypes.c_int
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_host_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_fwd_dropout.restype = ctypes.c_int
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong,
        ctypes.c_uint, vp]
    lib.fa_fwd_fp8.restype = ctypes.c_int
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int] + [ctypes.c_float] * 3 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_fp8_workspace_bytes.argtypes = [ctypes.c_int] * 4
    lib.fa_dropout_mask.restype = ctypes.c_int
    lib.fa_dropout_mask.argtypes = [vp] + [ctypes.c_int] * 4 + [
        ctypes.c_float, ctypes.c_ulonglong, ctypes.c_uint, vp]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [vp] * 9 + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_dropout.restype = ctypes.c_int
    lib.fa_bwd_dropout.argtypes = [vp] * 9 + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong,
        ctypes.c_uint, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_workspace_bytes.argtypes = [ctypes.c_int] * 6
    lib.fa_last_status.restype = ctypes.c_int
    lib.fa_last_status.argtypes = []
    lib.fa_stream_status.restype = ctypes.c_int
    lib.fa_stream_status.argtypes = [vp]
    lib.fa_clear_status.restype = ctypes.c_int
    lib.fa_clear_status.argtypes = []
    lib.fa_strerror.restype = ctypes.c_char_p
    lib.fa_strerror.argtypes = [ctypes.c_int]
    lib.fa_selftest_wait_timeout.restype = ctypes.c_int
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_int, vp]
    lib.fa_num_kernel_launches.restype = ctypes.c_longlong
    lib.fa_num_kernel_launches.argtypes = []
    lib.fa_set_wait_limit_us.restype = ctypes.c_int
    lib.fa_set_wait_limit_us.argtypes = [ctypes.c_ulonglong]
    lib.fa_get_wait_limit_us.restype = ctypes.c_ulonglong
    lib.fa_get_wait_limit_us.argtypes = []
    lib.fa_debug_cap_workspace.restype = ctypes.c_int
    lib.fa_debug_cap_workspace.argtypes = [ctypes.c_longlong]
    return lib


_choice = os.environ.get("FA_LIBRARY", "release")
if _choice not in ("release", "debug"):
    raise ImportError(f"FA_LIBRARY must be 'release' or 'debug', not {_choice!r}")
lib = load_library(DEBUG_LIB_PATH if _choice == "debug" else LIB_PATH)


def strerror(code: int) -> str:
    return lib.fa_strerror(int(code)).decode()


def fa_fwd(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, stream) -> int:
    """Direct C-ABI call with raw integer addresses (device pointers) and sizes."""
    return int(lib.fa_fwd(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                          float(scale), int(bool(causal)), int(dtype), stream))


def fa_fwd_ws(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, workspace, workspace_bytes,
              stream) -> int:
    """C-ABI call of the workspace variant (stream-K split of the key range)."""
    return int(lib.fa_fwd_ws(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                             float(scale), int(bool(causal)), int(dtype), workspace,
                             int(workspace_bytes), stream))


def fa_fwd_noalloc(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, stream) -> int:
    """C-ABI call of the allocation-free variant (fixed device scratch, see fa_fwd.h)."""
    return int(lib.fa_fwd_noalloc(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                                  float(scale), int(bool(causal)), int(dtype), stream))


def fa_fwd_host(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                workspace_bytes, stream) -> int:
    """C-ABI call of the forward pass on HOST buffers (device workspace; see fa_fwd.h)."""
    return int(lib.fa_fwd_host(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                               float(scale), int(bool(causal)), int(dtype), workspace,
                               int(workspace_bytes), stream))


def fa_fwd_host_workspace_bytes(B, H, Nq, Nk, d) -> int:
    return int(lib.fa_fwd_host_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(d)))


def fa_fwd_dropout(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, p_drop, seed, offset,
                   stream) -> int:
    """C-ABI call of the forward pass with dropout (mask of (seed, offset), see fa_fwd.h)."""
    return int(lib.fa_fwd_dropout(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                                  float(scale), int(bool(causal)), int(dtype), float(p_drop),
                                  int(seed), int(offset), stream))


def fa_fwd_fp8(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, q_descale, k_descale, v_descale,
               out_dtype, workspace, workspace_bytes, stream) -> int:
    """C-ABI call of the E4M3 forward pass (raw device addresses and sizes)."""
    return int(lib.fa_fwd_fp8(Q, K, V, O, L, int(B), int(H), int(Nq), int(Nk), int(d),
                              float(scale), int(bool(causal)), float(q_descale), float(k_descale),
                              float(v_descale), int(out_dtype), workspace, int(workspace_bytes),
                              stream))


def fa_fwd_fp8_workspace_bytes(B, H, Nk, d) -> int:
    return int(lib.fa_fwd_fp8_workspace_bytes(int(B), int(H), int(Nk), int(d)))


def fa_dropout_mask(keep, B, H, Nq, Nk, p_drop, seed, offset, stream) -> int:
    """C-ABI call writing the keep mask [B,H,Nq,Nk] (bytes) of fa_fwd_dropout."""
    return int(lib.fa_dropout_mask(keep, int(B), int(H), int(Nq), int(Nk), float(p_drop),
                                   int(seed), int(offset), stream))


def fa_fwd_workspace_bytes(B, H, Nq, Nk, d, causal) -> int:
    return int(lib.fa_fwd_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(d),
                                          int(bool(causal))))


def fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
           workspace_bytes, stream) -> int:
    """C-ABI call of the backward pass (raw device addresses and sizes)."""
    return int(lib.fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, int(B), int(H), int(Nq), int(Nk), int(d),
                          float(scale), int(bool(causal)), int(dtype), workspace,
                          int(workspace_bytes), stream))


def fa_bwd_dropout(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, causal, dtype, p_drop,
                   seed, offset, workspace, workspace_bytes, stream) -> int:
    """C-ABI call of the backward pass of fa_fwd_dropout (same p_drop, seed, offset)."""
    return int(lib.fa_bwd_dropout(Q, K, V, O, dO, L, dQ, dK, dV, int(B), int(H), int(Nq), int(Nk),
                                  int(d), float(scale), int(bool(causal)), int(dtype),
                                  float(p_drop), int(seed), int(offset), workspace,
                                  int(workspace_bytes), stream))


def fa_bwd_workspace_bytes(B, H, Nq, Nk, d) -> int:
    return int(lib.fa_bwd_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(d)))


def fa_last_status() -> int:
    return int(lib.fa_last_status())


def fa_stream_status(stream=None) -> int:
    """The device-side status once `stream`'s queued work has finished (that stream only)."""
    return int(lib.fa_stream_status(stream))


def fa_clear_status() -> int:
    return int(lib.fa_clear_status())


def fa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return int(lib.fa_selftest_wait_timeout(int(limit_us), stream))


def fa_num_kernel_launches() -> int:
    return int(lib.fa_num_kernel_launches())


def fa_set_wait_limit_us(limit_us: int) -> int:
    if not 0 <= int(limit_us) < 1 << 64:
        return FA_ERR_RANGE
    return int(lib.fa_set_wait_limit_us(int(limit_us)))


def fa_get_wait_limit_us() -> int:
    return int(lib.fa_get_wait_limit_us())


def attention(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
              stream=None, workspace=None):
    """O, L = attention(q, k, v) for CUDA tensors q [B,H,Nq,d], k/v [B,H,Nk,d] (fp16/bf16).

    Allocates O (like q) and L ([B,H,Nq] fp32) unless given; launches on `stream`
    (a torch.cuda.Stream, default: the current stream) and returns without synchronising.
    `workspace`: a zero-filled uint8 CUDA tensor of at least fa_fwd_workspace_bytes(...)
    bytes enables the stream-K split for full attention (see include/fa_fwd.h).
    """
    import torch

    # Every check runs before anything touches a device: the kernels write through raw
    # pointers, so a caller-supplied `out`, `lse` or `workspace` of the wrong size, type,
    # layout or device would be written out of bounds.
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("q, k, v must be float16 or bfloat16")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H, d")
    if out is not None and (out.dtype != q.dtype or tuple(out.shape) != (B, H, Nq, d)
                            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous [B, H, Nq, d] tensor of q's dtype")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous [B, H, Nq] float32 tensor")
    if workspace is not None and (workspace.dtype != torch.uint8 or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous uint8 tensor")
    tensors = [t for t in (q, k, v, out, lse, workspace) if t is not None]
    if not all(t.is_cuda for t in tensors):
        raise ValueError("q, k, v (and out, lse, workspace when given) must be CUDA tensors")
    if any(t.device != q.device for t in tensors):
        raise ValueError("q, k, v (and out, lse, workspace when given) must be on one device")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_F16
    with torch.cuda.device(q.device):
        if workspace is None:
            rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, H, Nq, Nk, d, scale, causal, dt, ctypes.c_void_p(stream.cuda_stream))
        else:
            rc = fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, Nq, Nk, d, scale, causal, dt,
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise FAError(rc)
    return out, lse
