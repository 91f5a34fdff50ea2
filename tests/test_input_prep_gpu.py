"""Parity of the GDN input prep kernels (through the C ABI) with the fp64 oracle.

Bounds. u = silu(y) is formed in fp32 from y = bias + sum_j w_j x_j (K fused
multiply-adds: error below 4e-6 of sum_j |w_j x_j| + |bias|) with the fast
exponential and division (2e-6 relative), then rounded to bf16 once (2^-9
relative); so |u - u*| <= 2^-8 |u*| + 4e-6 (|bias| + sum_j |w_j x_j|). The gates
use expf / log1pf: g within 1e-5 and beta within 2e-6, relative. The final
windows are copies of input rows: bit-exact.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import oracle
import workloads
from tests.parity import check, errors

pytestmark = pytest.mark.gpu


def run_prep(inp, h_qk, d_k, h_v, d_v, state_index=None, gates=True, want_state=True, parent=None):
    dev = "cuda"
    cuda = lambda t: None if t is None else t.to(dev)
    out = gdn.input_prep(cuda(inp["x"]), cuda(inp["conv_w"]), cuda(inp["cu_seqlens"]), h_qk=h_qk, d_k=d_k,
                         h_v=h_v, d_v=d_v, conv_bias=cuda(inp["conv_bias"]), conv_state=cuda(inp["conv_state"]),
                         state_index=cuda(state_index), a=cuda(inp["a"]) if gates else None,
                         b=cuda(inp["b"]), A_log=cuda(inp["A_log"]), dt_bias=cuda(inp["dt_bias"]),
                         parent=cuda(parent), want_conv_state=want_state)
    torch.cuda.synchronize()
    return out


def reference(inp, state_index=None, seqs=None):
    x = inp["x"].float().numpy()
    w = inp["conv_w"].numpy()
    bias = None if inp["conv_bias"] is None else inp["conv_bias"].numpy()
    st = None if inp["conv_state"] is None else inp["conv_state"].float().numpy()
    si = None if state_index is None else state_index.numpy()
    cu = inp["cu_seqlens"].numpy().astype(np.int64)
    u, fin = oracle.causal_conv_silu(x, w, cu, bias, st, si)
    # the bound's scale: |bias| + sum_j |w_j x_j| over the window (carried rows included)
    K = w.shape[1]
    scale = np.zeros_like(x, dtype=np.float64)
    for n in range(cu.size - 1):
        b, e = int(cu[n]), int(cu[n + 1])
        slot = -1 if st is None else (n if si is None else int(si[n]))
        car = st[slot] if slot >= 0 else np.zeros((K - 1, x.shape[1]))
        seq = np.concatenate([car, x[b:e]])
        for i in range(e - b):
            scale[b + i] = np.sum(np.abs(w.T * seq[i:i + K]), axis=0)
    if bias is not None:
        scale += np.abs(bias)
    g, beta = oracle.gate_params(inp["a"].float().numpy(), inp["b"].float().numpy(), inp["A_log"].numpy(),
                                 inp["dt_bias"].numpy())
    return u, fin, scale, g, beta


def check_u(q, k, v, u_ref, scale, rows=None):
    T = q.shape[0]
    u = torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], dim=1).double().cpu().numpy()
    if rows is not None:
        u = u[rows]
    bound = 2.0 ** -8 * np.abs(u_ref) + 4e-6 * scale + 1e-30
    bad = np.abs(u - u_ref) > bound
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} out of bound; worst excess " \
                          f"{float(np.max(np.abs(u - u_ref) - bound)):.3e}"


def check_gates(g, beta, g_ref, b_ref):
    g = g.double().cpu().numpy()
    beta = beta.double().cpu().numpy()
    assert np.all(np.abs(g - g_ref) <= 1e-5 * np.abs(g_ref) + 1e-30)
    assert np.all(np.abs(beta - b_ref) <= 2e-6 * np.abs(b_ref) + 1e-30)


@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("bias", [False, True])
def test_parity_ragged(K, bias):
    # ragged lengths around the 32-row runs, an empty and a one-row sequence
    lengths = [37, 0, 70, 1, 130, 32, 33]
    inp = workloads.prep_inputs(lengths, h_qk=2, d_k=64, h_v=4, d_v=64, K=K, seed=K * 10 + bias, bias=bias)
    q, k, v, g, beta, fin = run_prep(inp, 2, 64, 4, 64)
    u_ref, fin_ref, scale, g_ref, b_ref = reference(inp)
    check_u(q, k, v, u_ref, scale)
    check_gates(g, beta, g_ref, b_ref)
    np.testing.assert_array_equal(fin.float().cpu().numpy(), fin_ref)


def test_unequal_blocks():
    # q / k blocks of 2 x 64 channels and a v block of 6 x 128: the split at uneven
    # boundaries (thread vectors never straddle a block: every block is a multiple of 8)
    lengths = [129, 3, 200]
    inp = workloads.prep_inputs(lengths, h_qk=2, d_k=64, h_v=6, d_v=128, K=4, seed=12, bias=True)
    q, k, v, g, beta, fin = run_prep(inp, 2, 64, 6, 128)
    assert q.shape == (332, 2, 64) and v.shape == (332, 6, 128) and g.shape == (332, 6)
    u_ref, fin_ref, scale, g_ref, b_ref = reference(inp)
    check_u(q, k, v, u_ref, scale)
    check_gates(g, beta, g_ref, b_ref)
    np.testing.assert_array_equal(fin.float().cpu().numpy(), fin_ref)


def test_carried_windows_and_slots():
    lengths = [0, 2, 1, 65, 40]
    inp = workloads.prep_inputs(lengths, h_qk=1, d_k=128, h_v=2, d_v=128, K=4, seed=3, slots=4, bias=True)
    sidx = torch.tensor([3, -1, 0, 2, 7], dtype=torch.int32)  # 7: out of range -> zeros
    q, k, v, g, beta, fin = run_prep(inp, 1, 128, 2, 128, state_index=sidx)
    si_ref = sidx.clone()
    si_ref[4] = -1
    u_ref, fin_ref, scale, _, _ = reference(inp, state_index=si_ref)
    check_u(q, k, v, u_ref, scale)
    np.testing.assert_array_equal(fin.float().cpu().numpy(), fin_ref)


def test_split_run_equals_one_run():
    # a sequence in two calls, the window carried between them, gives the same rows
    inp = workloads.prep_inputs([100], h_qk=1, d_k=64, h_v=1, d_v=64, K=4, seed=4)
    one = run_prep(inp, 1, 64, 1, 64, gates=False)
    a_ = dict(inp, x=inp["x"][:45], cu_seqlens=torch.tensor([0, 45], dtype=torch.int32))
    first = run_prep(a_, 1, 64, 1, 64, gates=False)
    b_ = dict(inp, x=inp["x"][45:], cu_seqlens=torch.tensor([0, 55], dtype=torch.int32),
              conv_state=first[5].cpu())
    second = run_prep(b_, 1, 64, 1, 64, gates=False)
    for i in range(3):
        assert torch.equal(torch.cat([first[i], second[i]]), one[i])
    assert torch.equal(second[5], one[5])


def test_all_empty_sequences():
    inp = workloads.prep_inputs([0, 0, 0], h_qk=1, d_k=64, h_v=1, d_v=64, K=3, seed=5, slots=3)
    q, k, v, g, beta, fin = run_prep(inp, 1, 64, 1, 64)
    assert q.numel() == 0 and g.numel() == 0
    np.testing.assert_array_equal(fin.float().cpu().numpy(), inp["conv_state"].float().numpy())


def test_prep_then_prefill():
    # the layer's chain: prep, then the prefill on its q, k, v and fp32 gates, against
    # the oracle's prep (rounded to bf16 where the kernel rounds) and recurrence
    lengths = [90, 200, 64]
    h_qk, d_k, h_v, d_v = 2, 128, 4, 128
    inp = workloads.prep_inputs(lengths, h_qk=h_qk, d_k=d_k, h_v=h_v, d_v=d_v, K=4, seed=6)
    q, k, v, g, beta, _ = run_prep(inp, h_qk, d_k, h_v, d_v)
    o, s = gdn.prefill_varlen(q, k, v, g, beta, inp["cu_seqlens"].cuda(), check_device=True)
    torch.cuda.synchronize()
    u_ref, _, _, g_ref, b_ref = reference(inp)
    T = u_ref.shape[0]
    Cq = h_qk * d_k
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()
    q_r = bf(u_ref[:, :Cq]).reshape(T, h_qk, d_k)
    k_r = bf(u_ref[:, Cq:2 * Cq]).reshape(T, h_qk, d_k)
    v_r = bf(u_ref[:, 2 * Cq:]).reshape(T, h_v, d_v)
    o_ref, s_ref = oracle.recurrent(q_r, k_r, v_r, g_ref.astype(np.float32), b_ref.astype(np.float32),
                                    inp["cu_seqlens"].numpy())
    check(errors(o.double().cpu().numpy(), s.double().cpu().numpy(), o_ref, s_ref), "tc", label="prep+prefill")


def test_full_size_sampled_sequences():
    # the 74-prompt batch's shape (62,875 rows of 2 x 16 x 128 + 32 x 128 = 8,192
    # channels) as bench.py launches it; three sequences checked in full
    w = workloads.config(2)
    lengths = w.lengths.tolist()
    inp = workloads.prep_inputs(lengths, h_qk=16, d_k=128, h_v=32, d_v=128, K=4, seed=7)
    q, k, v, g, beta, fin = run_prep(inp, 16, 128, 32, 128)
    cu = inp["cu_seqlens"].numpy().astype(np.int64)
    for n in (0, int(np.argmax(lengths)), len(lengths) - 1):
        b, e = int(cu[n]), int(cu[n + 1])
        sub = dict(inp, x=inp["x"][b:e], a=inp["a"][b:e], b=inp["b"][b:e],
                   cu_seqlens=torch.tensor([0, e - b], dtype=torch.int32))
        u_ref, fin_ref, scale, g_ref, b_ref = reference(sub)
        check_u(q[b:e], k[b:e], v[b:e], u_ref, scale)
        check_gates(g[b:e], beta[b:e], g_ref, b_ref)
        np.testing.assert_array_equal(fin[n].float().cpu().numpy(), fin_ref[0])


def tree_scale(inp, parent, state_index):
    """|bias| + sum_j |w_j x_j| over each row's window along its root-to-node path."""
    x = inp["x"].float().numpy().astype(np.float64)
    w = inp["conv_w"].numpy().astype(np.float64)
    K = w.shape[1]
    st = None if inp["conv_state"] is None else inp["conv_state"].float().numpy()
    cu = inp["cu_seqlens"].numpy().astype(np.int64)
    par = parent.numpy()
    scale = np.zeros_like(x)
    for n in range(cu.size - 1):
        path = [n]
        while par[path[-1]] >= 0:
            path.append(int(par[path[-1]]))
        path.reverse()
        rows = np.concatenate([np.arange(cu[m], cu[m + 1]) for m in path]).astype(np.int64)
        slot = int(state_index[path[0]]) if st is not None else -1
        car = st[slot] if slot >= 0 else np.zeros((K - 1, x.shape[1]))
        seq = np.concatenate([car, x[rows]])
        b, e = int(cu[n]), int(cu[n + 1])
        off = rows.size - (e - b)
        for i in range(e - b):
            scale[b + i] = np.sum(np.abs(w.T * seq[off + i:off + i + K]), axis=0)
    if inp["conv_bias"] is not None:
        scale += np.abs(inp["conv_bias"].numpy())
    return scale


@pytest.mark.parametrize("kind", ["forest", "chain", "wide"])
def test_tree_windows(kind):
    # children continue their parents' rows; empty and short nodes pass the window on
    lengths, parent = {
        "forest": ([40, 2, 0, 70, 1, 33], [-1, 0, 1, 2, -1, 4]),
        "chain": ([1, 0, 2, 130, 1, 5], [-1, 0, 1, 2, 3, 4]),
        "wide": ([100, 3, 0, 64, 7, 1], [-1, 0, 0, 0, 0, 3]),
    }[kind]
    parent = torch.tensor(parent, dtype=torch.int32)
    sidx = torch.tensor([1, -1, -1, -1, 0, -1], dtype=torch.int32)  # roots' carried windows
    inp = workloads.prep_inputs(lengths, h_qk=1, d_k=64, h_v=2, d_v=64, K=4, seed=len(kind), slots=2, bias=True)
    q, k, v, g, beta, fin = run_prep(inp, 1, 64, 2, 64, state_index=sidx, parent=parent)
    u_ref, fin_ref = oracle.causal_conv_silu_tree(inp["x"].float().numpy(), inp["conv_w"].numpy(),
                                                  inp["cu_seqlens"].numpy(), parent.numpy(),
                                                  inp["conv_bias"].numpy(), inp["conv_state"].float().numpy(),
                                                  sidx.numpy())
    check_u(q, k, v, u_ref, tree_scale(inp, parent, sidx))
    np.testing.assert_array_equal(fin.float().cpu().numpy(), fin_ref)


def test_tree_chain_equals_one_sequence_bitwise():
    lens = [7, 1, 0, 2, 150]
    inp = workloads.prep_inputs(lens, h_qk=1, d_k=64, h_v=1, d_v=64, K=4, seed=13, slots=1)
    chain = run_prep(inp, 1, 64, 1, 64, state_index=torch.tensor([0, -1, -1, -1, -1], dtype=torch.int32),
                     parent=torch.tensor([-1, 0, 1, 2, 3], dtype=torch.int32), gates=False)
    one_inp = dict(inp, cu_seqlens=torch.tensor([0, sum(lens)], dtype=torch.int32))
    one = run_prep(one_inp, 1, 64, 1, 64, state_index=torch.tensor([0], dtype=torch.int32), gates=False)
    for i in range(3):
        assert torch.equal(chain[i], one[i])
    assert torch.equal(chain[5][-1], one[5][0])
