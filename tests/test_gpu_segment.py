"""The segment scan of one long sequence (include/gdn.h, gdn_prefill_varlen).

A single sequence keeps only h_v SMs busy: its chunks form one chain per value
head. The library then cuts it into segments, computes each segment's state map
S -> Phi S + Delta side by side (the gated delta rule is affine in the starting
state), composes the maps and reruns the segments from their true starting
states. These tests hold that path to the oracle at the same bounds as every
other case, compare it with the single-launch path (GDN_FLAG_NO_SEGMENT), and
check that the caller's cu_seqlens and state_index are still checked on the
device and that a dirty workspace changes nothing.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import oracle
import workloads
from tests.parity import check, errors, run_lib

pytestmark = pytest.mark.gpu

SEG_CASES = [
    # T, h_qk, h_v, d, gate dtype, out dtype, initial state
    (4096, 16, 32, 128, torch.bfloat16, torch.bfloat16, "slot"),
    (5001, 2, 4, 128, torch.float32, torch.bfloat16, "none"),
    (9000, 4, 8, 128, torch.float32, torch.float32, "slot"),
    (6000, 1, 4, 64, torch.bfloat16, torch.bfloat16, "index"),
    (4097, 2, 2, 64, torch.float32, torch.float32, "minus1"),
]


def _workload(T, h_qk, h_v, d, gdt, odt, init, seed):
    kw = {}
    if init == "slot":
        kw = dict(init_sd=0.05)
    elif init == "index":
        kw = dict(init_sd=0.05, n_slots=3, state_index=[2])
    elif init == "minus1":
        kw = dict(init_sd=0.05, n_slots=2, state_index=[-1])
    return workloads.random_workload([T], h_qk=h_qk, h_v=h_v, d_k=d, d_v=d, seed=seed, alpha_lo=0.9,
                                     gate_dtype=gdt, out_dtype=odt, name=f"seg_T{T}_h{h_v}_d{d}_{init}", **kw)


@pytest.mark.parametrize("case", SEG_CASES, ids=lambda c: f"T{c[0]}-hv{c[2]}-d{c[3]}-{c[6]}")
def test_segment_scan_against_oracle_and_single_launch(case):
    T, h_qk, h_v, d, gdt, odt, init = case
    w = _workload(T, h_qk, h_v, d, gdt, odt, init, seed=60 + T % 97)
    o_ref, s_ref = oracle.run_workload(w)
    o_seg, s_seg = run_lib(w, "tc")
    o_one, s_one = run_lib(w, "tc", flags=gdn.GDN_FLAG_NO_SEGMENT)
    f32 = odt == torch.float32
    check(errors(o_seg, s_seg, o_ref, s_ref), "tc", f32_out=f32, label=f"segment scan {w.name}")
    check(errors(o_one, s_one, o_ref, s_ref), "tc", f32_out=f32, label=f"one launch {w.name}")
    # the two paths agree far inside the oracle bounds
    e = errors(o_seg, s_seg, o_one, s_one)
    assert e["o_rel_fro"] <= 5e-3 and e["s_rel_fro"] <= 5e-4, e


def test_segment_scan_ran():
    """With a nonzero starting state, the later segments start from composed states,
    so their rounding differs from one launch's: the two results are not the same bits
    (while segment 0, run from the true state in both, is)."""
    w = _workload(8192, 2, 4, 128, torch.float32, torch.float32, "slot", seed=71)
    o_seg, _ = run_lib(w, "tc")
    o_one, _ = run_lib(w, "tc", flags=gdn.GDN_FLAG_NO_SEGMENT)
    assert not np.array_equal(o_seg, o_one)
    assert np.array_equal(o_seg[:64], o_one[:64])


def test_config4_single_launch_every_head():
    """The 16,384-token prompt of the long-prompt workload through one launch (the
    segment scan switched off): the path a caller with a small workspace takes."""
    w = workloads.config(4, layer=0)
    o, s = run_lib(w, "tc", flags=gdn.GDN_FLAG_NO_SEGMENT)
    o_ref, s_ref = oracle.run_workload(w)
    check(errors(o, s, o_ref, s_ref), "tc", label="cfg4 layer 0, one launch")


def _status(w, cu, sidx, init, fill=None):
    d = w.to("cuda")
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device="cuda")
    fs = torch.empty((1, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(d.q, d.v, d.g, cu_d, out_dtype=d.out_dtype, initial_state=init)
    ws = torch.empty(gdn.gdn_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    if fill is not None:
        fill(ws)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    rc = gdn.gdn_prefill_varlen(d.q, d.k, d.v, d.g, d.beta, cu_d, init, sidx, out, fs, desc)
    assert rc == gdn.GDN_OK
    return gdn.gdn_get_device_status(desc), out.cpu(), fs.cpu()


def test_segment_scan_device_checks():
    """The set-up kernel checks what the prep kernel checks for one sequence: the
    caller's cu_seqlens and state_index, reported through the status word."""
    T = 4160
    w = _workload(T, 1, 4, 64, torch.float32, torch.bfloat16, "none", seed=72)
    E = {n: i for i, n in enumerate(gdn.STATUS_NAMES)}
    init = torch.zeros((2, 4, 64, 64), dtype=torch.float32, device="cuda")
    assert _status(w, [0, T], None, None)[0] == gdn.GDN_OK
    assert _status(w, [0, T - 1], None, None)[0] == E["GDN_ERR_SEQLENS"]
    assert _status(w, [1, T], None, None)[0] == E["GDN_ERR_SEQLENS"]
    bad = torch.tensor([2], dtype=torch.int32, device="cuda")
    assert _status(w, [0, T], bad, init)[0] == E["GDN_ERR_STATE_INDEX"]
    ok = torch.tensor([-1], dtype=torch.int32, device="cuda")
    assert _status(w, [0, T], ok, init)[0] == gdn.GDN_OK
    torch.cuda.synchronize()


def test_segment_scan_dirty_workspace():
    """Whatever the workspace held (zeros, 0xFF, random bytes), the same bits."""
    T = 6000
    w = _workload(T, 2, 8, 128, torch.float32, torch.bfloat16, "slot", seed=73)
    d = w.to("cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(78)
    fills = [lambda ws: ws.zero_(), lambda ws: ws.fill_(0xFF),
             lambda ws: ws.copy_(torch.randint(0, 256, ws.shape, generator=gen, device="cuda",
                                               dtype=torch.int32).to(torch.uint8))]
    runs = [_status(w, [0, T], None, d.initial_state, f) for f in fills]
    for st, o, s in runs:
        assert st == gdn.GDN_OK
        assert torch.equal(o, runs[0][1]) and torch.equal(s, runs[0][2])
    o_ref, s_ref = oracle.run_workload(w)
    check(errors(runs[0][1].double().numpy(), runs[0][2].double().numpy(), o_ref, s_ref), "tc",
          label="segment scan dirty workspace")


def test_segment_scan_in_a_cuda_graph():
    """The segmented call (six kernels and a device copy) captures into a CUDA graph;
    replaying it on changed inputs gives the same bits as direct calls."""
    T = 4800
    w1 = _workload(T, 2, 4, 128, torch.float32, torch.bfloat16, "slot", seed=74)
    w2 = _workload(T, 2, 4, 128, torch.float32, torch.bfloat16, "slot", seed=75)
    d1, d2, static = w1.to("cuda"), w2.to("cuda"), w1.to("cuda")
    out = torch.empty(static.v.shape, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((1, 4, 128, 128), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(static.q, static.v, static.g, static.cu_seqlens, initial_state=static.initial_state)
    assert gdn.gdn_segment_plan(desc, torch.cuda.get_device_properties(0).multi_processor_count)[0] == 0
    ws = torch.empty(gdn.gdn_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    assert gdn.gdn_segment_plan(desc, torch.cuda.get_device_properties(0).multi_processor_count)[0] >= 3
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up outside capture
        assert gdn.gdn_prefill_varlen(static.q, static.k, static.v, static.g, static.beta, static.cu_seqlens,
                                      static.initial_state, None, out, fs, desc, s) == gdn.GDN_OK
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rc = gdn.gdn_prefill_varlen(static.q, static.k, static.v, static.g, static.beta, static.cu_seqlens,
                                    static.initial_state, None, out, fs, desc, torch.cuda.current_stream())
    assert rc == gdn.GDN_OK
    for d in (d2, d1):
        for name in ("q", "k", "v", "g", "beta", "initial_state"):
            getattr(static, name).copy_(getattr(d, name))
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_s = gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, initial_state=d.initial_state)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o)
        assert torch.equal(fs, ref_s)


def test_segment_scan_without_final_state():
    """final_state may be NULL: the segmented call still writes every output, the
    same bits as with it."""
    w = _workload(4500, 2, 4, 128, torch.float32, torch.bfloat16, "none", seed=76)
    d = w.to("cuda")
    o1, s1 = gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, check_device=True)
    o2, s2 = gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, want_final_state=False,
                                check_device=True)
    torch.cuda.synchronize()
    assert s2 is None
    assert torch.equal(o1, o2)
