"""The roofline's algorithmic bytes and tensor-core FLOPs in bench.py, checked
against independent counts (CPU)."""
import numpy as np
import torch

import bench
import workloads


def test_algorithmic_bytes_of_the_74_prompt_workload():
    w = workloads.config(2)
    T, N = w.total_tokens, w.num_seqs
    assert (T, N) == (62875, 74)
    # per token: q and k (16 heads x 128, bf16), v (32 x 128, bf16), g and beta
    # (32, fp32), o (32 x 128, bf16)
    per_token = 2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 4 + 32 * 128 * 2
    assert per_token == 24832
    # per sequence: the fp32 final state (32 x 128 x 128); cu_seqlens: N + 1 int32
    expect = per_token * T + N * 32 * 128 * 128 * 4 + 4 * (N + 1)
    assert bench.algorithmic_bytes(w) == expect == 1716501548


def test_algorithmic_bytes_count_gathered_slots_once():
    w = workloads.random_workload([10, 20, 30], h_qk=1, h_v=2, d_k=64, d_v=64, seed=0, init_sd=0.1,
                                  n_slots=2)
    w.state_index = torch.tensor([1, -1, 1], dtype=torch.int32)
    base = workloads.random_workload([10, 20, 30], h_qk=1, h_v=2, d_k=64, d_v=64, seed=0)
    # one distinct slot (slot 1, twice) is read once
    assert bench.algorithmic_bytes(w) - bench.algorithmic_bytes(base) == 1 * 2 * 64 * 64 * 4


def test_tensor_flops_list_every_product():
    lengths = [64, 130, 5]
    h_qk, h_v, dk, dv = 2, 4, 64, 128
    w = workloads.random_workload(lengths, h_qk=h_qk, h_v=h_v, d_k=dk, d_v=dv, seed=1)
    products = []  # (m, k, n): an m x k by k x n product, 2 m k n flops
    for L in lengths:
        chunks = [64] * (L // 64) + ([L % 64] if L % 64 else [])
        for l in chunks:
            for _ in range(h_qk):
                products += [(l, dk, l), (l, dk, l)]  # K K^T and Q K^T
            for _ in range(h_v):
                products += [(l, l, dk),  # W = T_w K
                             (l, l, dv),  # U = T_b V
                             (l, l, dv),  # the intra-chunk output term, with M
                             (l, dk, dv),  # W S
                             (l, dk, dv),  # Q S
                             (dk, l, dv)]  # the state update K^T U'
    expect = sum(2 * m * k * n for m, k, n in products)
    assert bench.chunked_tensor_flops(w) == expect
