"""Helpers for the backward parity tests: run fa_fwd then fa_bwd through the C ABI."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import gen


def run_fwd_bwd(w, q, k, v, do, device="cuda:0"):
    """Host tensors in; returns host (O, L, dQ, dK, dV) from the CUDA path."""
    import exact_attention_forward_02_gb300 as fa
    dev = torch.device(device)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    O = torch.empty((w.B, w.H, w.Nq, w.d), dtype=q.dtype, device=dev)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    dt = fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16
    st = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                   w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt, st)
    assert rc == 0, fa.strerror(rc)
    dQ = torch.full_like(qd, float("nan"))
    dK = torch.full_like(kd, float("nan"))
    dV = torch.full_like(vd, float("nan"))
    nws = fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    rc = fa.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), dod.data_ptr(),
                   L.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), w.B, w.H, w.Nq, w.Nk,
                   w.d, w.scale, w.causal, dt, ws.data_ptr(), nws, st)
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize(dev)
    status = fa.fa_last_status()
    assert status == 0, fa.strerror(status)
    return O.cpu(), L.cpu(), dQ.cpu(), dK.cpu(), dV.cpu()


def make_inputs(w):
    q, k, v = gen.make_qkv(w)
    # the upstream gradient: its own seeded N(0,1) draw (tensor id 3), rounded like Q
    rng = np.random.default_rng([int(w.seed), 3])
    do = torch.from_numpy(rng.standard_normal((w.B, w.H, w.Nq, w.d))).to(gen.torch_dtype(w.dtype))
    return q, k, v, do


def grad_errors(w, q, k, v, do, dQ, dK, dV):
    import oracle
    rq, rk, rv = oracle.attention_bwd(gen.to_f64_numpy(q), gen.to_f64_numpy(k), gen.to_f64_numpy(v),
                                      gen.to_f64_numpy(do), w.scale, w.causal)
    out = {}
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.double().numpy()
        out[name] = {"finite": bool(np.isfinite(g).all()),
                     "max_abs_err": float(np.abs(g - ref).max()),
                     "max_abs_ref": float(np.abs(ref).max()),
                     "rel_to_max": float(np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-30))}
    return out
