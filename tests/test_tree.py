"""Prefix trees in one launch (gdn_prefill_tree): the oracle's tree pinned to
independent compositions on the CPU, and the CUDA path against it on the GPU.

A tree sequence n continues from the final state of sequence parent[n]
(open-jev-fast README, Phase 2 item 2, "Prefix tree"; System1-Omni PR #186,
"Purpose and summary"); config 3 is the two-level tree of the example request
(shared context -> 3 question branches -> 7 candidate tails).
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import oracle
import workloads
from tests.parity import check, errors


def cfg3_tree():
    t = workloads.tree_config()
    parent = [-1] + [0] * len(t.branch_lens) + [1 + b for b in t.leaf_parent]
    return t, t.rows, np.array(parent, dtype=np.int32)


def random_tree(seed, lengths, parent, *, h_qk=2, h_v=4, d=128, slots=0, roots_slot=None,
                gate_dtype=torch.float32, out_dtype=torch.bfloat16):
    w = workloads.random_workload(lengths, h_qk=h_qk, h_v=h_v, d_k=d, d_v=d, seed=seed,
                                  gate_dtype=gate_dtype, out_dtype=out_dtype)
    if slots:
        rng = np.random.default_rng(seed + 100)
        w.initial_state = torch.from_numpy(
            (rng.standard_normal((slots, h_v, d, d)) * 0.05).astype(np.float32))
        w.state_index = torch.tensor(roots_slot, dtype=torch.int32)
    else:
        w.initial_state, w.state_index = None, None
    return w, np.array(parent, dtype=np.int32)


def oracle_tree(w, parent):
    return oracle.tree(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, parent, w.initial_state,
                       w.state_index, scale=w.scale)


# ---------------------------------------------------------------- CPU: the oracle's tree pinned

def test_oracle_tree_of_roots_is_a_plain_batch():
    w, parent = random_tree(11, [70, 1, 0, 130], [-1, -1, -1, -1], h_v=2, h_qk=2, d=64, slots=3,
                            roots_slot=[2, -1, 0, 1])
    o_t, s_t = oracle_tree(w, parent)
    o_b, s_b = oracle.run_workload(w)
    assert np.array_equal(o_t, o_b) and np.array_equal(s_t, s_b)


def test_oracle_chain_is_one_long_sequence():
    """A sequence cut into a chain (each piece the child of the one before) gives
    the long sequence's outputs and, at its last piece, its final state."""
    w = workloads.random_workload([300], h_qk=2, h_v=2, d_k=64, d_v=64, seed=12,
                                  gate_dtype=torch.float32)
    cuts = [0, 64, 65, 130, 130, 211, 300]
    pieces = workloads.take_rows(w, [[slice(cuts[i], cuts[i + 1])] for i in range(len(cuts) - 1)],
                                 "chain")
    parent = np.arange(-1, len(cuts) - 2, dtype=np.int32)
    o_c, s_c = oracle_tree(pieces, parent)
    o_l, s_l = oracle.run_workload(w)
    assert np.array_equal(o_c, o_l)
    assert np.array_equal(s_c[-1], s_l[0])


def test_oracle_tree_matches_handoff_in_fp32():
    """The hand-off itself: each node run alone from its parent's final state
    (handed over in fp32, as the library's final_state holds it)."""
    t, rows, parent = cfg3_tree()
    o_t, s_t = oracle.tree(rows.q, rows.k, rows.v, rows.g, rows.beta, rows.cu_seqlens, parent,
                           scale=rows.scale)
    cu = rows.cu_seqlens.numpy()
    fs = {}
    for n in range(len(parent)):
        seg = workloads.take_rows(rows, [[slice(int(cu[n]), int(cu[n + 1]))]], "node")
        if parent[n] >= 0:
            seg.initial_state = torch.from_numpy(fs[parent[n]][None].astype(np.float32))
            seg.state_index = torch.tensor([0], dtype=torch.int32)
        o_n, s_n = oracle.run_workload(seg)
        fs[n] = s_n[0]
        assert np.abs(o_n - o_t[cu[n]:cu[n + 1]]).max() <= 1e-6
        assert np.linalg.norm(s_n[0] - s_t[n]) <= 1e-6 * np.linalg.norm(s_t[n])


def test_oracle_tree_rejects_bad_parents():
    w, _ = random_tree(13, [10, 10], [-1, 0], h_v=2, h_qk=2, d=64)
    with pytest.raises(ValueError):
        oracle_tree(w, np.array([-1, 1], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle_tree(w, np.array([-2, 0], dtype=np.int32))


# ---------------------------------------------------------------- GPU: one launch against the oracle

def run_tree(w, parent, **kw):
    d = w.to("cuda")
    out = torch.full(d.v.shape, float("nan"), dtype=d.out_dtype, device="cuda")
    fs = torch.full((d.num_seqs, d.h_v, d.d_k, d.d_v), float("nan"), dtype=torch.float32,
                    device="cuda")
    gdn.prefill_tree(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens,
                     torch.from_numpy(parent).to("cuda"), initial_state=d.initial_state,
                     state_index=d.state_index, out=out, final_state=fs, max_seqlen=w.max_seqlen,
                     scale=w.scale, check_device=True, **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), fs.double().cpu().numpy()


@pytest.mark.gpu
def test_config3_tree_in_one_launch():
    t, rows, parent = cfg3_tree()
    o, s = run_tree(rows, parent)
    o_ref, s_ref = oracle.tree(rows.q, rows.k, rows.v, rows.g, rows.beta, rows.cu_seqlens,
                               parent, scale=rows.scale)
    check(errors(o, s, o_ref, s_ref), "tc", label="cfg3 tree")


@pytest.mark.gpu
def test_tree_launch_equals_level_by_level_calls():
    """One launch gives bit for bit what three gdn_prefill_varlen calls give
    (prefix, then branches from its state, then leaves from theirs)."""
    from tests.parity import run_lib
    t, rows, parent = cfg3_tree()
    o, s = run_tree(rows, parent)
    pre = workloads.take_rows(rows, [[t.segment("prefix")]], "prefix")
    o_p, s_p = run_lib(pre)
    br = workloads.take_rows(rows, [[t.segment("branch", b)] for b in range(3)], "branches",
                             initial_state=torch.from_numpy(s_p.astype(np.float32)),
                             state_index=torch.zeros(3, dtype=torch.int32))
    o_b, s_b = run_lib(br)
    lv = workloads.take_rows(rows, [[t.segment("leaf", l)] for l in range(7)], "leaves",
                             initial_state=torch.from_numpy(s_b.astype(np.float32)),
                             state_index=torch.tensor(t.leaf_parent, dtype=torch.int32))
    o_l, s_l = run_lib(lv)
    assert np.array_equal(o, np.concatenate([o_p, o_b, o_l]))
    assert np.array_equal(s, np.concatenate([s_p, s_b, s_l]))


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["forest", "deep_chain_d64_f32", "wide"])
def test_random_trees(case):
    if case == "forest":
        # two trees and a lone root, ragged and empty nodes, roots from initial-state slots
        lengths = [150, 70, 0, 1, 64, 65, 200, 3, 0, 40, 129, 9]
        parent = [-1, 0, 0, 1, -1, 4, 4, 6, 5, -1, 2, 3]
        w, par = random_tree(21, lengths, parent, slots=2, roots_slot=[1, 0, 0, 0, -1, 0, 0, 0, 0,
                                                                       0, 0, 0])
    elif case == "deep_chain_d64_f32":
        lengths = [70, 1, 65, 0, 130, 3, 64, 200]
        w, par = random_tree(22, lengths, list(range(-1, 7)), h_qk=2, h_v=2, d=64,
                             out_dtype=torch.float32)
    else:
        lengths = [300] + [int(x) for x in np.random.default_rng(23).integers(1, 90, 24)]
        w, par = random_tree(23, lengths, [-1] + [0] * 24, h_qk=2, h_v=4, d=128)
    o, s = run_tree(w, par)
    o_ref, s_ref = oracle_tree(w, par)
    check(errors(o, s, o_ref, s_ref), "tc", f32_out=w.out_dtype == torch.float32, label=case)


@pytest.mark.gpu
def test_tree_of_empty_sequences_copies_root_states():
    w, par = random_tree(24, [0, 0, 0, 0], [-1, 0, 1, -1], h_qk=2, h_v=2, d=64, slots=2,
                         roots_slot=[1, 0, 0, -1])
    o, s = run_tree(w, par)
    init = w.initial_state.double().numpy()
    assert np.array_equal(s[0], init[1]) and np.array_equal(s[1], init[1])
    assert np.array_equal(s[2], init[1]) and not s[3].any()


@pytest.mark.gpu
def test_tree_bad_parent_reported_on_device():
    w, _ = random_tree(25, [20, 20, 20], [-1, 0, 0], h_qk=2, h_v=2, d=64)
    with pytest.raises(gdn.GdnError) as e:
        run_tree(w, np.array([-1, 2, 0], dtype=np.int32))  # parent 2 of sequence 1 is not below it
    assert e.value.code == gdn.STATUS_NAMES.index("GDN_ERR_PARENT")


@pytest.mark.gpu
def test_stalled_ready_flags_time_out_and_the_context_survives():
    """Fault injection without a fault: with the work list reversed, a chain of 400
    sequences puts the deepest children in every CTA's hands while their parents wait
    behind them, so no ready flag is ever set. Every bounded wait runs out (2 s), the
    launch reports GDN_ERR_DEVICE_TIMEOUT and returns; the context stays usable and
    the same tree then runs correctly."""
    N = 400
    w = workloads.random_workload([2] * N, h_qk=1, h_v=1, d_k=64, d_v=64, seed=21)
    parent = torch.tensor([-1] + list(range(N - 1)), dtype=torch.int32)
    d = w.to("cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.prefill_tree(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, parent.cuda(),
                         flags=gdn.GDN_FLAG_TEST_CHILD_FIRST, check_device=True)
    assert e.value.code == gdn.STATUS_NAMES.index("GDN_ERR_DEVICE_TIMEOUT")
    o, s = gdn.prefill_tree(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, parent.cuda(), check_device=True)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.tree(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, parent)
    check(errors(o.double().cpu().numpy(), s.double().cpu().numpy(), o_ref, s_ref), "tc", label="tree after stall")
