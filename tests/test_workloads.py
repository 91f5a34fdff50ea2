"""The synthetic inputs match the recipe the design states (CPU): sizes, dtypes
and the value ranges of every config."""
import numpy as np
import torch

import workloads


def _unit_rows(x):
    n = torch.linalg.vector_norm(x.float(), dim=-1)
    return float((n - 1).abs().max())


def test_config2_recipe():
    w = workloads.config(2)
    lens = w.lengths
    assert w.num_seqs == 74 and w.total_tokens == 62875 and w.max_seqlen == 3080
    assert lens.min() >= 80 and lens.max() <= 3399
    assert (w.h_qk, w.h_v, w.d_k, w.d_v) == (16, 32, 128, 128)
    assert w.q.dtype == w.k.dtype == w.v.dtype == torch.bfloat16
    assert w.g.dtype == w.beta.dtype == torch.float32 and w.out_dtype == torch.bfloat16
    alpha = torch.exp(w.g.double())
    assert float(alpha.min()) >= 0.85 - 1e-6 and float(alpha.max()) <= 1.0
    assert 0.0 < float(w.beta.min()) and float(w.beta.max()) < 1.0
    assert _unit_rows(w.q) < 1e-2 and _unit_rows(w.k) < 1e-2  # unit rows, rounded to bf16
    assert w.initial_state is None


def test_small_configs():
    w0, w1 = workloads.config(0), workloads.config(1)
    assert (w0.total_tokens, w0.h_qk, w0.h_v, w0.d_k) == (128, 2, 2, 64)
    assert w0.g.dtype == torch.bfloat16 and w0.out_dtype == torch.float32
    assert (w1.total_tokens, w1.h_qk, w1.h_v, w1.d_k) == (539, 16, 32, 128)
    assert float(torch.exp(w0.g.float()).min()) >= 0.89


def test_long_config_with_initial_state():
    w = workloads.config(4, layer=0)
    assert w.total_tokens == 16384 and w.num_seqs == 1
    assert float(torch.exp(w.g.double()).min()) >= 0.95 - 1e-6
    s0 = w.initial_state.double()
    assert s0.shape == (1, 32, 128, 128) and abs(float(s0.std()) - 0.02) < 1e-3
    assert torch.equal(w.state_index, torch.tensor([0], dtype=torch.int32))
    assert not torch.equal(workloads.config(4, layer=1).q, w.q)  # one input set per layer


def test_tree_config():
    t = workloads.tree_config()
    assert t.prefix_len == 480
    lens = t.rows.lengths
    assert lens[0] == 480 and len(lens) == 1 + 3 + 7
    assert all(10 <= L <= 30 for L in lens[1:4]) and all(4 <= L <= 40 for L in lens[4:])


def test_seeded_and_distinct():
    a, b = workloads.config(1), workloads.config(1)
    assert torch.equal(a.q, b.q) and torch.equal(a.g, b.g)
    c = workloads.config(1, seed_offset=1)
    assert not torch.equal(a.q, c.q)
