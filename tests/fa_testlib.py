"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the float64 oracle on the same seeded inputs."""
from __future__ import annotations

import ctypes
import functools

import numpy as np
import torch

import gen

# Tolerances on max |O - O64| by input type, and on max |L - L64| (natural log).
TOL_O = {gen.BF16: 1e-2, gen.F16: 4e-3}
TOL_L = 1e-3
# Mantissa bits of the output types, for half an ulp of the exact result.
_MANT = {gen.BF16: 7, gen.F16: 10}


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of `dtype` numbers around |x| (the error of rounding x to dtype)."""
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    e = np.floor(np.log2(ax))
    return 2.0 ** (e - _MANT[dtype] - 1)


def run_cuda(w: gen.Workload, q, k, v, device="cuda:0", nan_fill=True, stream=None):
    """Launch fa_fwd through the C ABI on host tensors q, k, v; returns host (O, L) and rc."""
    import exact_attention_forward_02_gb300 as fa

    dev = torch.device(device)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fill = float("nan") if nan_fill else 0.0
    O = torch.full((w.B, w.H, w.Nq, w.d), fill, dtype=q.dtype, device=dev)
    L = torch.full((w.B, w.H, w.Nq), fill, dtype=torch.float32, device=dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                   w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                   fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16,
                   ctypes.c_void_p(st.cuda_stream))
    assert rc == 0, f"fa_fwd rc={rc} ({fa.strerror(rc)})"
    torch.cuda.synchronize(dev)
    status = fa.fa_last_status()
    assert status == 0, f"device status {status} ({fa.strerror(status)})"
    return O.cpu(), L.cpu()


def p_rounding_term(w: gen.Workload, v) -> np.ndarray:
    """Per element of O: 2^-(t+1) * max over the keys j visible to row i of |V[j,c]|, t the
    mantissa bits of the input type. P is rounded to the input type before the second
    product (relative error at most 2^-(t+1) per entry, RNE) while l sums the unrounded P,
    so O = sum_j w_j (1 + e_j) V_j moves by sum_j w_j e_j V_j, at most this much. Causal
    rows see keys j <= i (top-left), so the maximum is a prefix maximum of |V|."""
    BH = w.B * w.H
    va = np.abs(v.reshape(BH, w.Nk, w.d).float().numpy())
    if w.causal:
        vmax = np.maximum.accumulate(va, axis=1)[:, np.minimum(np.arange(w.Nq), w.Nk - 1)]
    else:
        vmax = np.broadcast_to(va.max(axis=1, keepdims=True), (BH, w.Nq, w.d))
    return (2.0 ** -(_MANT[w.dtype] + 1)) * vmax.reshape(-1, w.d)


def compare(w: gen.Workload, O, L, Oref, Lref, rows=None, extra=None):
    """Element-wise comparison. O, L: kernel results (torch, host). Oref, Lref: oracle
    float64 (numpy) for all rows, or for the flat rows `rows` when given.

    Returns a dict with the raw maxima and the graded verdicts:
      raw:    max |O - O64| <= TOL_O[dtype] and max |L - L64| <= TOL_L
      graded: |O - O64| <= TOL_O[dtype] + half_ulp(O64) element-wise (the kernel's own
              error budget on top of the unavoidable rounding of the exact answer to
              the output type) and the same L bound.
      derived (when `extra` is given, per element): the graded bound plus `extra`, the
              part of the error that rounding P to the input type can add
              (p_rounding_term).
    """
    Ok = O.double().numpy().reshape(-1, w.d)
    Lk = L.double().numpy().reshape(-1)
    if rows is not None:
        Ok, Lk = Ok[rows], Lk[rows]
    Or = np.asarray(Oref).reshape(-1, w.d)
    Lr = np.asarray(Lref).reshape(-1)
    assert np.all(np.isfinite(Ok)) and np.all(np.isfinite(Lk)), "non-finite output (unwritten row?)"
    err = np.abs(Ok - Or)
    el = np.abs(Lk - Lr)
    tol = TOL_O[w.dtype]
    bound = tol + half_ulp(Or, w.dtype)
    out_extra = {}
    if extra is not None:
        ex = np.asarray(extra).reshape(-1, w.d)
        if rows is not None:
            ex = ex[rows]
        out_extra = {"derived_ok": bool(np.all(err <= bound + ex) and (el.size == 0 or el.max() <= TOL_L)),
                     "over_graded": int((err > bound).sum()),
                     "max_err_over_derived_bound": float((err / (bound + ex)).max()) if err.size else 0.0}
    return {
        **out_extra,
        "max_err_O": float(err.max()) if err.size else 0.0,
        "max_err_L": float(el.max()) if el.size else 0.0,
        "raw_ok": bool((err.size == 0 or err.max() <= tol) and (el.size == 0 or el.max() <= TOL_L)),
        "graded_ok": bool(np.all(err <= bound) and (el.size == 0 or el.max() <= TOL_L)),
        "worst_row": int(np.argmax(err.max(axis=1))) if err.size else -1,
    }


def sample_rows(w: gen.Workload, n_heads: int = 6, n_rand: int = 24, seed: int = 0):
    """Flat row indices covering head boundaries, tile edges and random rows."""
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    heads = sorted(set([0, BH - 1] + list(rng.choice(BH, size=min(BH, n_heads), replace=False))))
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, 257, w.Nq // 2, w.Nq - 2, w.Nq - 1]
    out = []
    for bh in heads:
        rs = [r for r in fixed if 0 <= r < w.Nq]
        rs += list(rng.integers(0, w.Nq, size=n_rand))
        out += [bh * w.Nq + r for r in sorted(set(rs))]
    return np.array(out, dtype=np.int64)


def oracle_rows(w: gen.Workload, q, k, v, rows):
    """The oracle on selected flat rows, slicing one head at a time (so only the heads
    that are sampled are widened to float64)."""
    import oracle

    rows = np.asarray(rows, dtype=np.int64)
    Oref = np.empty((rows.size, w.d))
    Lref = np.empty(rows.size)
    qf = q.reshape(w.B * w.H, w.Nq, w.d)
    kf = k.reshape(w.B * w.H, w.Nk, w.d)
    vf = v.reshape(w.B * w.H, w.Nk, w.d)
    for bh in np.unique(rows // w.Nq):
        sel = np.nonzero(rows // w.Nq == bh)[0]
        local = rows[sel] % w.Nq
        Oh, Lh = oracle.attention_rows(gen.to_f64_numpy(qf[bh])[None, None],
                                       gen.to_f64_numpy(kf[bh])[None, None],
                                       gen.to_f64_numpy(vf[bh])[None, None],
                                       w.scale, w.causal, local)
        Oref[sel] = Oh
        Lref[sel] = Lh
    return Oref, Lref


@functools.lru_cache(maxsize=None)
def oracle_whole(name: str):
    """Inputs and the oracle's whole output of a named workload, computed once per test
    session: (q, k, v) as generated (host tensors) and (O64, L64) for every row. At the
    oracle's rate on a many-core host the largest workload (B=1, H=16, N=32768 causal,
    4.4 TFLOP) takes about a minute; the others a few seconds."""
    import oracle

    w = gen.WORKLOADS[name]
    q, k, v = gen.make_qkv(w)
    Oref, Lref = oracle.attention(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                  w.scale, w.causal)
    return (q, k, v), (Oref, Lref)


def run_cuda_ws(w: gen.Workload, q, k, v, calls=1, device="cuda:0"):
    """fa_fwd_ws (the stream-K split, caller workspace zero-filled once) on host tensors
    q, k, v, `calls` times on the same workspace; returns [(O, L) host tensors] and the
    workspace size."""
    import exact_attention_forward_02_gb300 as fa

    dev = torch.device(device)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    nbytes = fa.fa_fwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, w.causal)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(calls):
        O = torch.full((w.B, w.H, w.Nq, w.d), float("nan"), dtype=q.dtype, device=dev)
        L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=dev)
        rc = fa.fa_fwd_ws(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                          w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                          fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16,
                          ws.data_ptr(), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
        assert rc == 0, fa.strerror(rc)
        torch.cuda.synchronize(dev)
        assert fa.fa_last_status() == 0
        outs.append((O.cpu(), L.cpu()))
    return outs, nbytes
