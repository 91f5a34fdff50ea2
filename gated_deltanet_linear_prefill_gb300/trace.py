"""Per-role clock trace of the tensor-core chunk kernel.

Builds the tracing library (build(trace=True): the same sources with
-DGDN_TC_TRACE, include/gdn_trace.h), runs the 74-prompt batch (or its first N
sequences) through it, and prints, for each traced CTA, the chunk period and the
median life of one chunk: when each role reached each of its points, relative to
the moment the state-step group (WG-B) starts splitting that chunk's U'. Times
are CUDA-clock cycles converted with the CTA's own clock rate; the stamps cost
about 10% of the kernel's time, so the absolute period reads a little long.

    python -m gated_deltanet_linear_prefill_gb300.trace [--subset-seqs N] [--ctas 0,77]
    python -m gated_deltanet_linear_prefill_gb300.trace --lengths 96 --heads 1 --ctas 0

The second form traces a random batch of the given lengths (h_qk = h_v = heads,
d 128) and prints every stamp of the CTA from its start: the latency of a short
unit rather than a steady-state period.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np
import torch

from . import GdnDesc, make_desc
from .build import build

# (warp, point) -> what the stamp marks; the chunk index is the chunk the event
# belongs to (WG-B stamps points 2-5 for the chunk after the one it is splitting)
EVENTS = {
    (0, 0): "producer: K/Q ring slot free",
    (0, 1): "producer: K/Q tiles requested",
    (0, 2): "producer: V tile requested",
    (1, 0): "warp 1: top of its chunk loop",
    (1, 1): "warp 1: T_b / T_w written, R and W' accumulators free",
    (1, 2): "warp 1: W' product issued",
    (1, 3): "warp 1: V tile landed",
    (1, 4): "warp 1: U product issued",
    (2, 0): "warp 2: chunk prepared, W' converted, U done",
    (2, 1): "warp 2: state of the previous chunk ready",
    (2, 2): "warp 2: U' = U - W' S product issued",
    (2, 3): "warp 2: bf16 state copy ready, O free",
    (2, 4): "warp 2: U' split into hi / lo",
    (2, 5): "warp 2: state update issued",
    (2, 6): "warp 2: output products issued",
    (3, 0): "warp 3: [K;Q] K^T issued",
    (3, 1): "warp 3: q norms written",
    (4, 0): "WG-A: tiles and [K;Q] K^T in",
    (4, 1): "WG-A: [K;Q] K^T read",
    (4, 2): "WG-A: A and M written",
    (4, 3): "WG-A: previous chunk's U done",
    (4, 4): "WG-A: solve done",
    (4, 5): "WG-A: T_b / T_w ready",
    (12, 0): "WG-B: U' done, split starts",
    (12, 1): "WG-B: split done",
    (12, 2): "WG-B: W' product done, conversion starts",
    (12, 3): "WG-B: W' converted",
    (12, 4): "WG-B: previous state update done, bf16 copy starts",
    (12, 5): "WG-B: bf16 state copy written",
    (12, 6): "WG-B: O done, epilogue starts",
    (12, 7): "WG-B: epilogue done",
}
REF = (12, 0)
WORDS = 16 * 2048 + 4


def load_trace_lib():
    lib = ctypes.CDLL(build(trace=True))
    P = ctypes.c_void_p
    lib.gdn_prefill_varlen.argtypes = [P] * 10 + [ctypes.POINTER(GdnDesc), P]
    lib.gdn_prefill_varlen.restype = ctypes.c_int
    lib.gdn_workspace_bytes.argtypes = [ctypes.POINTER(GdnDesc)]
    lib.gdn_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_trace_set_cta.argtypes = [ctypes.c_int]
    lib.gdn_trace_read.argtypes = [P]
    return lib


def trace_workload(w, ctas, warmup=3):
    """Runs workload `w` through the tracing library; yields (cta, stamps, ghz, cta_us)."""
    lib = load_trace_lib()
    d = w.to("cuda")
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device="cuda")
    fs = torch.empty((w.num_seqs, w.h_v, w.d_k, w.d_v), dtype=torch.float32, device="cuda")
    desc = make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype, initial_state=d.initial_state,
                     max_seqlen=w.max_seqlen)
    ws = torch.empty(max(256, lib.gdn_workspace_bytes(ctypes.byref(desc))), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else 0)

    def call():
        rc = lib.gdn_prefill_varlen(ptr(d.q), ptr(d.k), ptr(d.v), ptr(d.g), ptr(d.beta), ptr(d.cu_seqlens),
                                    ptr(d.initial_state), ptr(d.state_index), ptr(out), ptr(fs),
                                    ctypes.byref(desc), None)
        if rc != 0:
            raise RuntimeError(f"gdn_prefill_varlen returned {rc}")

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    for cta in ctas:
        if lib.gdn_trace_set_cta(int(cta)) or lib.gdn_trace_clear():
            raise RuntimeError("trace set-up failed")
        call()
        buf = np.zeros(WORDS, np.uint64)
        if lib.gdn_trace_read(buf.ctypes.data_as(ctypes.c_void_p)):
            raise RuntimeError("trace read failed")
        buf = buf.astype(np.int64)
        clk0, gt0, clk1, gt1 = buf[16 * 2048:]
        ghz = (clk1 - clk0) / max(1, gt1 - gt0)
        trace_workload.start_clock = int(clk0)
        yield cta, buf[:16 * 2048].reshape(16, 256, 8), ghz, (gt1 - gt0) / 1e3


def report_raw(T, start_clk, ghz, cta, cta_us, file=sys.stdout):
    """Every stamp of one CTA in time order, in us from the CTA's start."""
    print(f"CTA {cta}: {cta_us:.1f} us from start to end, clock {ghz:.3f} GHz", file=file)
    evs = []
    for (wp, pt), name in EVENTS.items():
        for c in range(256):
            if T[wp, c, pt] > 0:
                evs.append(((T[wp, c, pt] - start_clk) / ghz / 1e3, f"chunk {c}: {name}"))
    for t, name in sorted(evs):
        print(f"    {t:8.2f}  {name}", file=file)
    return evs


def report(T, ghz, cta, cta_us, file=sys.stdout):
    """The chunk period and the median life of one chunk, from one CTA's stamps."""
    ref = T[REF[0], :, REF[1]]
    nc = int((ref > 0).sum())
    cs = [c for c in range(4, max(5, nc - 4)) if ref[c] > 0]
    us = lambda cyc: cyc / ghz / 1e3
    period = us((ref[cs[-1]] - ref[cs[0]]) / max(1, cs[-1] - cs[0])) if len(cs) > 1 else float("nan")
    print(f"CTA {cta}: {nc} chunks traced, {cta_us:.1f} us, clock {ghz:.3f} GHz, "
          f"period {period:.2f} us per chunk", file=file)
    rows = []
    for (wp, pt), name in EVENTS.items():
        x = [T[wp, c, pt] - ref[c] for c in cs if T[wp, c, pt] > 0]
        if x:
            rows.append((us(float(np.median(x))), name))
    rows.sort()
    print("  median life of chunk c (us, relative to WG-B starting the split of chunk c):", file=file)
    for t, name in rows:
        print(f"    {t:+7.2f}  {name}", file=file)
    return period, rows


def main(argv=None):
    import workloads
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--subset-seqs", type=int, default=0, help="trace the first N sequences only")
    ap.add_argument("--ctas", default="0,77", help="comma-separated CTAs to trace (one launch each)")
    ap.add_argument("--lengths", default="", help="comma-separated sequence lengths of a random batch")
    ap.add_argument("--heads", type=int, default=1, help="q/k and value heads of the random batch")
    args = ap.parse_args(argv)
    if args.lengths:
        w = workloads.random_workload([int(x) for x in args.lengths.split(",")], h_qk=args.heads,
                                      h_v=args.heads, d_k=128, d_v=128, seed=6, gate_dtype=torch.float32)
    else:
        w = workloads.config(2)
        if args.subset_seqs:
            w = workloads.subset_sequences(w, list(range(args.subset_seqs)))
    print(f"workload {w.name}: {w.num_seqs} sequences, {w.total_tokens} tokens, h_v {w.h_v}")
    for cta, T, ghz, cta_us in trace_workload(w, [int(x) for x in args.ctas.split(",")]):
        if args.lengths:
            report_raw(T, trace_workload.start_clock, ghz, cta, cta_us)
        else:
            report(T, ghz, cta, cta_us)


if __name__ == "__main__":
    main()
