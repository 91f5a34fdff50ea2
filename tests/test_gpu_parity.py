"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every case is compared element by element over every output, the full-size
workloads (74 packed prompts; one 16,384-token prompt) included: they run on
the GPU exactly as the bench launches them, and the oracle computes the whole
batch (a few seconds on the host cores).
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import oracle
import workloads
from tests.parity import check, errors, run_lib

pytestmark = pytest.mark.gpu

KERNELS = ["tc", "simt"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_config0_tiny(kernel):
    w = workloads.config(0)
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, kernel)
    check(errors(o, s, o_ref, s_ref), kernel, f32_out=True, label="cfg0")


@pytest.mark.parametrize("kernel", KERNELS)
def test_config1_single_prompt(kernel):
    w = workloads.config(1)
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, kernel)
    check(errors(o, s, o_ref, s_ref), kernel, label="cfg1")


_ORACLE_CACHE = {}


def _oracle_whole(key, w):
    """The oracle over a whole workload, computed once per test session."""
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.run_workload(w)
    return _ORACLE_CACHE[key]


@pytest.mark.parametrize("kernel", KERNELS)
def test_config2_varlen_full_size_every_sequence(kernel):
    """74 packed prompts at full size, every output element and final state
    against the oracle (all 74 sequences x 32 heads)."""
    w = workloads.config(2)
    o, s = run_lib(w, kernel)
    o_ref, s_ref = _oracle_whole("cfg2", w)
    check(errors(o, s, o_ref, s_ref), kernel, label="cfg2")


@pytest.mark.parametrize("kernel", KERNELS)
def test_config3_prefix_tree_fork(kernel):
    """prefix -> 3 branches -> 7 leaves through gathered states equals the 7
    full root-to-leaf paths, on the GPU and against the oracle."""
    tree = workloads.tree_config()
    rows = tree.rows
    pre = workloads.take_rows(rows, [[tree.segment("prefix")]], "prefix")
    o_p, s_p = run_lib(pre, kernel)
    br = workloads.take_rows(rows, [[tree.segment("branch", b)] for b in range(3)], "branches",
                             initial_state=torch.from_numpy(s_p.astype(np.float32)),
                             state_index=torch.zeros(3, dtype=torch.int32))
    o_b, s_b = run_lib(br, kernel)
    lv = workloads.take_rows(rows, [[tree.segment("leaf", l)] for l in range(7)], "leaves",
                             initial_state=torch.from_numpy(s_b.astype(np.float32)),
                             state_index=torch.tensor(tree.leaf_parent, dtype=torch.int32))
    o_l, s_l = run_lib(lv, kernel)
    paths = workloads.take_rows(rows, [[tree.segment("prefix"),
                                        tree.segment("branch", tree.leaf_parent[l]),
                                        tree.segment("leaf", l)] for l in range(7)], "paths")
    o_f, s_f = run_lib(paths, kernel)
    o_ref, s_ref = oracle.run_workload(paths)
    # the full paths against the oracle
    check(errors(o_f, s_f, o_ref, s_ref), kernel, label="cfg3 paths")
    # the forked leaves against the oracle's full paths (leaf rows) and final states
    cu = paths.cu_seqlens.numpy()
    leaf_rows = np.concatenate([np.arange(cu[l + 1] - tree.leaf_lens[l], cu[l + 1])
                                for l in range(7)])
    check(errors(o_l, s_l, o_ref[leaf_rows], s_ref), kernel, label="cfg3 fork")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("layer", [0, 47])
def test_config4_long_prompt_every_head(kernel, layer):
    """One 16,384-token prompt with a non-zero initial state (layers 0 and 47
    of the 48 input sets), every head against the oracle."""
    w = workloads.config(4, layer=layer)
    o, s = run_lib(w, kernel)
    o_ref, s_ref = _oracle_whole(f"cfg4-{layer}", w)
    check(errors(o, s, o_ref, s_ref), kernel, label=f"cfg4 layer {layer}")


EDGE_LENGTHS = [0, 1, 63, 64, 65, 127, 128, 129, 0, 200, 2]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("h_qk,h_v,d_k,d_v", [(2, 4, 64, 64), (4, 4, 128, 64), (1, 4, 64, 128),
                                              (2, 4, 128, 128)])
def test_edge_lengths_heads_dims(kernel, h_qk, h_v, d_k, d_v):
    """Empty and ragged sequences across chunk boundaries, every supported
    head ratio and head size, gathered states with -1 and shared slots."""
    w = workloads.random_workload(EDGE_LENGTHS, h_qk=h_qk, h_v=h_v, d_k=d_k, d_v=d_v, seed=7,
                                  alpha_lo=0.8, gate_dtype=torch.float32,
                                  out_dtype=torch.bfloat16, init_sd=0.05, n_slots=3,
                                  state_index=[0, 1, 2, -1, 0, 0, 1, 2, -1, 1, 2])
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, kernel)
    check(errors(o, s, o_ref, s_ref), kernel, label=f"edge {h_qk}/{h_v} {d_k}x{d_v}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_fp32_outputs_bf16_gates_custom_scale(kernel):
    w = workloads.random_workload([300, 5, 77], h_qk=2, h_v=4, d_k=128, d_v=128, seed=8,
                                  gate_dtype=torch.bfloat16, out_dtype=torch.float32)
    w.scale = 0.3
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, kernel)
    check(errors(o, s, o_ref, s_ref), kernel, f32_out=True, label="fp32 out")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("gates", ["steep", "wipes", "mixed_sign"])
def test_extreme_gates(kernel, gates):
    """Decays far outside the benchmark range: steep ones (log-decay up to -40
    per token, so chunks end after a few rows), occasional state wipes
    (g = -200) and gates of both signs that still decay on average (a state
    that grows without bound amplifies any rounding). The kernels must still
    match the oracle, with every exponential factor kept in range."""
    w = workloads.random_workload([300, 1, 140], h_qk=2, h_v=4, d_k=128, d_v=128, seed=15,
                                  gate_dtype=torch.float32, out_dtype=torch.float32,
                                  init_sd=0.05)
    rng = np.random.default_rng(16)
    T, H = w.g.shape
    if gates == "steep":
        g = -rng.uniform(0.0, 40.0, (T, H))
    elif gates == "wipes":
        g = np.where(rng.random((T, H)) < 0.03, -200.0, -0.01)
    else:  # both signs (G not monotone inside a chunk), decaying on average
        g = rng.normal(-0.05, 0.15, (T, H))
    w.g = torch.from_numpy(g.astype(np.float32))
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, kernel)
    # the stated bounds (the fp32 SIMT kernel's tighter in-range bounds do not
    # apply to decays of e^-40 per token)
    check(errors(o, s, o_ref, s_ref), "tc", label=f"gates {gates} ({kernel})")


@pytest.mark.parametrize("kernel", KERNELS)
def test_beta_one_stores_v_on_gpu(kernel):
    """b = 1, q = k (unit): o_t = scale v_t at every token, within bf16."""
    w = workloads.random_workload([150, 70], h_qk=1, h_v=2, d_k=128, d_v=128, seed=9,
                                  gate_dtype=torch.float32, out_dtype=torch.float32)
    w.beta.fill_(1.0)
    w.q = w.k.clone()
    o, _ = run_lib(w, kernel)
    ref = w.v.double().numpy() * 128 ** -0.5
    err = np.abs(o - ref).max()
    assert err <= 4e-3 * np.abs(ref).max(), err


@pytest.mark.parametrize("kernel", KERNELS)
def test_permutation_invariance_bitwise(kernel):
    """A sequence's results do not depend on its neighbours or position."""
    w = workloads.random_workload([90, 17, 300, 64, 1], h_qk=2, h_v=4, d_k=128, d_v=128,
                                  seed=10, gate_dtype=torch.float32, init_sd=0.1)
    o, s = run_lib(w, kernel)
    perm = [2, 4, 0, 3, 1]
    pw = workloads.subset_sequences(w, perm)
    o2, s2 = run_lib(pw, kernel)
    cu = w.cu_seqlens.numpy()
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in perm])
    assert np.array_equal(o2, o[rows])
    assert np.array_equal(s2, s[perm])


def test_kernels_agree():
    """The tensor-core kernel and the fp32 SIMT kernel agree within the
    tensor-core tolerance on a mid-size batch."""
    w = workloads.random_workload([700, 333, 64], h_qk=4, h_v=8, d_k=128, d_v=128, seed=11,
                                  gate_dtype=torch.float32, init_sd=0.02)
    o1, s1 = run_lib(w, "tc")
    o2, s2 = run_lib(w, "simt")
    e = errors(o1, s1, o2, s2)
    assert e["o_rel_fro"] <= 1e-2 and e["s_rel_fro"] <= 1e-3, e


def _device_status(w, cu, sidx=None, init=None):
    d = w.to("cuda")
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = torch.empty(d.v.shape, dtype=torch.bfloat16, device="cuda")
    desc = gdn.make_desc(d.q, d.v, d.g, cu_d, initial_state=init)
    ws = torch.empty(gdn.gdn_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    rc = gdn.gdn_prefill_varlen(d.q, d.k, d.v, d.g, d.beta, cu_d, init, sidx, out, None, desc)
    assert rc == gdn.GDN_OK
    return gdn.gdn_get_device_status(desc)


def test_device_detected_errors_are_reported_not_trapped():
    """Malformed cu_seqlens / state_index are found on the device, reported
    through the status word, and leave the context usable."""
    w = workloads.random_workload([50, 50], h_qk=1, h_v=2, d_k=64, d_v=64, seed=12)
    E = {n: i for i, n in enumerate(gdn.STATUS_NAMES)}
    assert _device_status(w, [0, 50, 100]) == gdn.GDN_OK
    assert _device_status(w, [0, 60, 40]) == E["GDN_ERR_SEQLENS"]  # decreasing
    assert _device_status(w, [0, 50, 90]) == E["GDN_ERR_SEQLENS"]  # cu[N] != T
    assert _device_status(w, [4, 50, 100]) == E["GDN_ERR_SEQLENS"]  # cu[0] != 0
    init = torch.zeros((2, 2, 64, 64), dtype=torch.float32, device="cuda")
    bad = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    assert _device_status(w, [0, 50, 100], bad, init) == E["GDN_ERR_STATE_INDEX"]
    ok = torch.tensor([1, -1], dtype=torch.int32, device="cuda")
    assert _device_status(w, [0, 50, 100], ok, init) == gdn.GDN_OK
    torch.cuda.synchronize()  # the context is still usable


def test_cuda_graph_capture_and_replay_with_new_inputs():
    """The call captures into a CUDA graph; replaying it on changed inputs
    gives the same bits as direct calls."""
    w1 = workloads.random_workload([200, 50, 129], h_qk=2, h_v=4, d_k=128, d_v=128, seed=13,
                                   gate_dtype=torch.float32, init_sd=0.1)
    w2 = workloads.random_workload([200, 50, 129], h_qk=2, h_v=4, d_k=128, d_v=128, seed=14,
                                   gate_dtype=torch.float32, init_sd=0.1)
    d1, d2 = w1.to("cuda"), w2.to("cuda")
    static = w1.to("cuda")
    out = torch.empty(static.v.shape, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((3, 4, 128, 128), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(static.q, static.v, static.g, static.cu_seqlens,
                         initial_state=static.initial_state)
    ws = torch.empty(gdn.gdn_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up outside capture
        assert gdn.gdn_prefill_varlen(static.q, static.k, static.v, static.g, static.beta,
                                      static.cu_seqlens, static.initial_state, None, out, fs,
                                      desc, s) == gdn.GDN_OK
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rc = gdn.gdn_prefill_varlen(static.q, static.k, static.v, static.g, static.beta,
                                    static.cu_seqlens, static.initial_state, None, out, fs, desc,
                                    torch.cuda.current_stream())
    assert rc == gdn.GDN_OK
    for d in (d2, d1):
        for name in ("q", "k", "v", "g", "beta", "initial_state"):
            getattr(static, name).copy_(getattr(d, name))
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_s = gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens,
                                          initial_state=d.initial_state)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o)
        assert torch.equal(fs, ref_s)


def test_repeat_runs_bitwise():
    """The persistent kernel hands units to CTAs from an atomic counter, so two runs
    map units to SMs differently; each unit's arithmetic is fixed, so the results
    must be bit-identical (a race in the TMEM / mbarrier pipeline would show here)."""
    w = workloads.config(2)
    o1, s1 = run_lib(w, "tc")
    o2, s2 = run_lib(w, "tc")
    assert np.array_equal(o1, o2)
    assert np.array_equal(s1, s2)
    # the kernels around the prefill as well
    inp = workloads.prep_inputs([300, 0, 129, 64], h_qk=2, d_k=128, h_v=4, d_v=128, K=4, seed=3)
    cuda = lambda t: None if t is None else t.cuda()
    outs = [gdn.input_prep(cuda(inp["x"]), cuda(inp["conv_w"]), cuda(inp["cu_seqlens"]), h_qk=2, d_k=128, h_v=4,
                           d_v=128, a=cuda(inp["a"]), b=cuda(inp["b"]), A_log=cuda(inp["A_log"]),
                           dt_bias=cuda(inp["dt_bias"])) for _ in range(2)]
    for a_, b_ in zip(*outs):
        assert torch.equal(a_, b_)
    z, wt = workloads.norm_inputs(493, 4, 128, seed=4)
    ys = [gdn.gated_rmsnorm(outs[0][2], z.cuda(), wt.cuda()) for _ in range(2)]
    assert torch.equal(ys[0], ys[1])


@pytest.mark.parametrize("lengths", [[65], [80], [96], [65, 72, 80, 88, 91, 94, 96]],
                         ids=["lone65", "lone80", "lone96", "seven_paths"])
def test_short_paths_two_chunks(lengths):
    """Row F4's case: candidate paths of 65-96 tokens (two chunks each), alone and as
    the seven-path batch `bench.py --latency` times, at the long-prompt workload's
    shape (16 q/k and 32 value heads, d 128, bf16 gates), against the oracle."""
    w = workloads.random_workload(lengths, h_qk=16, h_v=32, d_k=128, d_v=128, seed=90 + len(lengths),
                                  gate_dtype=torch.bfloat16, name=f"short paths {lengths}")
    o_ref, s_ref = oracle.run_workload(w)
    o, s = run_lib(w, "tc")
    check(errors(o, s, o_ref, s_ref), "tc", label=f"short paths {lengths}")
