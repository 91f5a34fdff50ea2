"""The per-role clock trace of the chunk kernel (the tracing build, include/gdn_trace.h):
it builds, runs the first 16 prompts of the 74-prompt batch, and its stamps tell a
consistent story (each chunk's products issued after its inputs were ready, a
positive period). Its results are the same bits as the regular library's."""
import numpy as np
import pytest
import torch

import workloads
from gated_deltanet_linear_prefill_gb300 import trace
from tests.parity import run_lib

pytestmark = pytest.mark.gpu


def test_trace_build_runs_and_orders_events():
    w = workloads.subset_sequences(workloads.config(2), list(range(16)))
    (cta, T, ghz, cta_us), = list(trace.trace_workload(w, [0]))
    assert 1.0 < ghz < 2.5 and cta_us > 0
    period, rows = trace.report(T, ghz, cta, cta_us)
    assert 0.5 < period < 50.0
    t = {name: x for x, name in rows}
    order = ["producer: K/Q tiles requested", "warp 3: [K;Q] K^T issued", "WG-A: solve done",
             "WG-A: T_b / T_w ready", "warp 1: U product issued", "warp 2: U' = U - W' S product issued",
             "WG-B: U' done, split starts", "WG-B: split done", "warp 2: state update issued",
             "WG-B: epilogue done"]
    for a, b in zip(order, order[1:]):
        assert t[a] < t[b], (a, b, t[a], t[b])


def test_trace_build_gives_the_same_bits():
    w = workloads.random_workload([300, 129, 64], h_qk=2, h_v=4, d_k=128, d_v=128, seed=81,
                                  gate_dtype=torch.float32, init_sd=0.05)
    o_ref, s_ref = run_lib(w, "tc")
    lib = trace.load_trace_lib()
    d = w.to("cuda")
    import ctypes
    import gated_deltanet_linear_prefill_gb300 as gdn
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device="cuda")
    fs = torch.empty((3, 4, 128, 128), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype, initial_state=d.initial_state)
    ws = torch.empty(max(256, lib.gdn_workspace_bytes(ctypes.byref(desc))), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    p = lambda x: ctypes.c_void_p(x.data_ptr() if x is not None else 0)
    rc = lib.gdn_prefill_varlen(p(d.q), p(d.k), p(d.v), p(d.g), p(d.beta), p(d.cu_seqlens), p(d.initial_state),
                                p(d.state_index), p(out), p(fs), ctypes.byref(desc), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(out.double().cpu().numpy(), o_ref)
    assert np.array_equal(fs.double().cpu().numpy(), s_ref)
