"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances. The stated bounds: on o, max |o - o*| <= 2e-2 and
mean |o - o*| <= 2e-3; on the final fp32 state, ||S - S*||_F / ||S*||_F <=
1e-3 over the whole final_state tensor. Because outputs are small (mean |o|
is about 1e-2 on these inputs) those absolute bounds alone would let a
missing term slip through, so the tests also bound the relative Frobenius
error of o: 1e-2 for the tensor-core kernel (bf16 rounding of the output is
about 2e-3 of it, the bf16/tf32 operands add about as much) and much tighter
for the fp32 SIMT kernel.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import gated_deltanet_linear_prefill_gb300 as gdn

TOL = {
    # kernel: (max_abs, mean_abs, o_rel_fro, s_rel_fro)
    "tc": (2e-2, 2e-3, 1e-2, 1e-3),
    "simt": (2e-2, 2e-3, 6e-3, 2e-5),
}
TOL_SIMT_F32_OUT = (1e-5, 1e-6, 2e-5, 2e-5)
KERNELS = {"tc": 0, "simt": gdn.GDN_FLAG_SIMT}


def run_lib(w, kernel="tc", device="cuda", flags=0, dirty=True, **kw):
    """Run a workloads.Workload through the library; returns host float64 (o, S)."""
    d = w.to(device)
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device=device)
    fs = torch.empty((d.num_seqs, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device=device)
    if dirty:
        out.fill_(float("nan"))
        fs.fill_(float("nan"))
    gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, initial_state=d.initial_state,
                       state_index=d.state_index, out=out, final_state=fs,
                       max_seqlen=w.max_seqlen, scale=w.scale,
                       flags=KERNELS[kernel] | flags, check_device=True, **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), fs.double().cpu().numpy()


def errors(o, s, o_ref, s_ref):
    do = np.abs(o - o_ref)
    e = {
        "max_abs": float(do.max()) if do.size else 0.0,
        "mean_abs": float(do.mean()) if do.size else 0.0,
        "o_rel_fro": float(np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)),
        "s_rel_fro": float(np.linalg.norm(s - s_ref) / max(np.linalg.norm(s_ref), 1e-30)),
        "nan_o": int(np.isnan(o).sum()),
        "nan_s": int(np.isnan(s).sum()),
    }
    if s.ndim == 4 and s.shape[0] * s.shape[1] > 0:
        num = np.sqrt(((s - s_ref) ** 2).sum(axis=(2, 3)))
        den = np.maximum(np.sqrt((s_ref ** 2).sum(axis=(2, 3))), 1e-30)
        e["s_rel_worst_unit"] = float((num / den).max())
    return e


def check(e, kernel="tc", f32_out=False, label=""):
    tol = TOL_SIMT_F32_OUT if (kernel == "simt" and f32_out) else TOL[kernel]
    log = os.environ.get("GDN_PARITY_LOG")
    if log:  # one JSON line per comparison, for a table of measured errors
        with open(log, "a") as f:
            f.write(json.dumps({"label": label, "kernel": kernel, "tol": tol, **e}) + "\n")
    assert e["nan_o"] == 0 and e["nan_s"] == 0, (label, e)
    assert e["max_abs"] <= tol[0], (label, e)
    assert e["mean_abs"] <= tol[1], (label, e)
    assert e["o_rel_fro"] <= tol[2], (label, e)
    assert e["s_rel_fro"] <= tol[3], (label, e)
