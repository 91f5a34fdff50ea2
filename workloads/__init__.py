"""Seeded synthetic inputs for the gated delta rule prefill.

This module is shared by the fp64 oracle (tests, CPU baseline) and by the
CUDA path (tests, bench). It holds none of the method's arithmetic: it only
draws random numbers in a fixed, documented order and rounds them once to
their storage dtypes, so both sides consume the same bits.

Workload shapes follow the pages (Open-Jev / open-jev-fast, see the README of
"open-jev-fast", section "Single inference (example request)", and the
System1-Omni validation page, "Raw HF Transformers comparison"):

* the example request: 539 tokens, 3 questions, 7 candidates;
* the single-candidate workload: 74 prompts of 80 to 3,399 tokens;
* the longest supported prompt: 16,384 tokens;
* the Qwen3.x-27B linear-attention shape: 16 q/k heads, 32 v heads
  (grouped-value attention), head dim 128, 48 linear-attention layers.

Draw order inside every config: lengths, q, k, v, alpha, beta, initial state.
q and k are drawn N(0, 1) and L2-normalised per (token, head) before rounding,
v is N(0, 1), the log-decay is g = log(alpha) with alpha uniform, and
beta = sigmoid(N(0, 1)). Normal draws are made in float32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = ["Workload", "config", "CONFIG_NAMES", "tree_config", "random_workload"]


@dataclasses.dataclass
class Workload:
    """One packed batch of sequences, as the library consumes it.

    Tensors live on the host (CPU torch tensors); callers move them.
    q, k: [T, h_qk, d_k] bf16. v: [T, h_v, d_v] bf16. g, beta: [T, h_v]
    (bf16 or fp32). cu_seqlens: [N+1] int32. initial_state: [slots, h_v, d_k,
    d_v] fp32 or None. state_index: [N] int32 or None.
    """

    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor
    initial_state: Optional[torch.Tensor]
    state_index: Optional[torch.Tensor]
    out_dtype: torch.dtype
    scale: float = 0.0  # 0 means d_k ** -0.5

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def h_qk(self) -> int:
        return int(self.q.shape[1])

    @property
    def h_v(self) -> int:
        return int(self.v.shape[1])

    @property
    def d_k(self) -> int:
        return int(self.q.shape[2])

    @property
    def d_v(self) -> int:
        return int(self.v.shape[2])

    @property
    def lengths(self) -> np.ndarray:
        cu = self.cu_seqlens.numpy().astype(np.int64)
        return cu[1:] - cu[:-1]

    @property
    def max_seqlen(self) -> int:
        lens = self.lengths
        return int(lens.max()) if lens.size else 0

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)

        return dataclasses.replace(
            self, q=mv(self.q), k=mv(self.k), v=mv(self.v), g=mv(self.g), beta=mv(self.beta),
            cu_seqlens=mv(self.cu_seqlens), initial_state=mv(self.initial_state),
            state_index=mv(self.state_index))


def _cu(lengths) -> torch.Tensor:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return torch.from_numpy(cu.astype(np.int32))


def _unit_rows(rng, T, H, d) -> torch.Tensor:
    x = rng.standard_normal((T, H, d), dtype=np.float32)
    x /= np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True)).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def _normal(rng, shape, sd=1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if sd != 1.0:
        x *= np.float32(sd)
    return x


def _gates(rng, T, H, alpha_lo, dtype):
    alpha = rng.uniform(alpha_lo, 1.0, size=(T, H))
    g = np.log(alpha)
    x = rng.standard_normal((T, H))
    beta = 1.0 / (1.0 + np.exp(-x))
    return (torch.from_numpy(g.astype(np.float32)).to(dtype),
            torch.from_numpy(beta.astype(np.float32)).to(dtype))


def random_workload(lengths, *, h_qk, h_v, d_k, d_v, seed, alpha_lo=0.9,
                    gate_dtype=torch.bfloat16, out_dtype=torch.bfloat16,
                    init_sd: Optional[float] = None, n_slots: Optional[int] = None,
                    state_index=None, name="random") -> Workload:
    """A packed batch with the given lengths, drawn in the module's order.

    init_sd: None for no initial state, else the N(0, init_sd) fp32 state
    (n_slots slots, default one per sequence).
    """
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    q = _unit_rows(rng, T, h_qk, d_k)
    k = _unit_rows(rng, T, h_qk, d_k)
    v = torch.from_numpy(_normal(rng, (T, h_v, d_v))).to(torch.bfloat16)
    g, beta = _gates(rng, T, h_v, alpha_lo, gate_dtype)
    init = None
    sidx = None
    if init_sd is not None:
        slots = len(lengths) if n_slots is None else int(n_slots)
        init = torch.from_numpy(_normal(rng, (slots, h_v, d_k, d_v), init_sd))
        if state_index is not None:
            sidx = torch.tensor(list(state_index), dtype=torch.int32)
    return Workload(name, q, k, v, g, beta, _cu(lengths), init, sidx, out_dtype)


def _cfg2_lengths(rng, n=74, lo=80, hi=3399):
    u = rng.uniform(math.log(lo), math.log(hi), size=n)
    return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int64)


def config(idx: int, *, layer: int = 0, seed_offset: int = 0) -> Workload:
    """The five synthetic workloads.

    0: tiny check. 1 sequence, T=128, h_qk=h_v=2, d=64, bf16 inputs (g, beta
       too), fp32 output, zero state, alpha~U(0.90,1), seed 0.
    1: the example request's size as one prompt. T=539, 16/32 heads, d=128,
       bf16 everything (fp32 state), zero state, seed 1.
    2: 74 prompts, lengths round(exp(U(ln 80, ln 3399))) clipped to
       [80, 3399], packed; bf16 q/k/v, fp32 g/beta, bf16 output,
       alpha~U(0.85,1), no initial state, seed 2.
    3: the prefix tree as three packed batches; see tree_config().
    4: one 16,384-token prompt, bf16 inputs, alpha~U(0.95,1), initial state
       N(0, 0.02) fp32 (0.02 read as the standard deviation), state_index=[0],
       seed 4; `layer` selects one of 48 input sets (seed (4, layer)).
    seed_offset shifts the seed (independent replicas on several ranks).
    """
    if idx == 0:
        return random_workload([128], h_qk=2, h_v=2, d_k=64, d_v=64, seed=0 + seed_offset,
                               alpha_lo=0.90, gate_dtype=torch.bfloat16,
                               out_dtype=torch.float32, name="cfg0_tiny_T128_d64")
    if idx == 1:
        return random_workload([539], h_qk=16, h_v=32, d_k=128, d_v=128, seed=1 + seed_offset,
                               alpha_lo=0.90, gate_dtype=torch.bfloat16,
                               out_dtype=torch.bfloat16, name="cfg1_single_T539")
    if idx == 2:
        rng = np.random.default_rng(2 + seed_offset)
        lengths = _cfg2_lengths(rng)
        # continue with the same generator: lengths first, then the tensors
        T = int(lengths.sum())
        q = _unit_rows(rng, T, 16, 128)
        k = _unit_rows(rng, T, 16, 128)
        v = torch.from_numpy(_normal(rng, (T, 32, 128))).to(torch.bfloat16)
        g, beta = _gates(rng, T, 32, 0.85, torch.float32)
        return Workload("cfg2_varlen_74seq", q, k, v, g, beta, _cu(lengths), None, None,
                        torch.bfloat16)
    if idx == 4:
        seed = np.random.SeedSequence([4 + seed_offset, int(layer)])
        rng = np.random.default_rng(seed)
        T = 16384
        q = _unit_rows(rng, T, 16, 128)
        k = _unit_rows(rng, T, 16, 128)
        v = torch.from_numpy(_normal(rng, (T, 32, 128))).to(torch.bfloat16)
        g, beta = _gates(rng, T, 32, 0.95, torch.bfloat16)
        init = torch.from_numpy(_normal(rng, (1, 32, 128, 128), 0.02))
        return Workload(f"cfg4_long_T16384_layer{layer}", q, k, v, g, beta, _cu([T]), init,
                        torch.tensor([0], dtype=torch.int32), torch.bfloat16)
    if idx == 3:
        raise ValueError("config 3 is a tree of three batches: use tree_config()")
    raise ValueError(f"no config {idx}")


CONFIG_NAMES = {0: "cfg0_tiny_T128_d64", 1: "cfg1_single_T539", 2: "cfg2_varlen_74seq",
                3: "cfg3_prefix_tree", 4: "cfg4_long_T16384"}


@dataclasses.dataclass
class Tree:
    """A two-level prefix tree: one shared prefix, branches, leaves.

    rows: the token data of prefix, branches and leaves stacked in that order
    (a Workload whose cu_seqlens lists prefix, then each branch, then each
    leaf). parent[b] of a branch is 0 (the prefix); leaf_parent[l] is its
    branch index.
    """

    rows: Workload
    prefix_len: int
    branch_lens: list
    leaf_lens: list
    leaf_parent: list

    def segment(self, which: str, i: int = 0) -> slice:
        cu = self.rows.cu_seqlens.numpy()
        if which == "prefix":
            j = 0
        elif which == "branch":
            j = 1 + i
        else:
            j = 1 + len(self.branch_lens) + i
        return slice(int(cu[j]), int(cu[j + 1]))


def tree_config(seed: int = 3, prefix_len: int = 480, n_branches: int = 3,
                leaves_per_branch=(3, 1, 3), h_qk=16, h_v=32, d=128,
                alpha_lo=0.90) -> Tree:
    """Config 3: shared context -> 3 question branches -> 7 candidate tails.

    Branch lengths uniform in {10..30}, leaf lengths uniform in {4..40}
    (integers, inclusive), leaves split [3, 1, 3] over the branches (one
    candidate for the yes/no question). bf16 everything, seed 3.
    """
    rng = np.random.default_rng(seed)
    branch_lens = [int(x) for x in rng.integers(10, 31, size=n_branches)]
    n_leaves = int(sum(leaves_per_branch))
    leaf_lens = [int(x) for x in rng.integers(4, 41, size=n_leaves)]
    leaf_parent = [b for b, c in enumerate(leaves_per_branch) for _ in range(c)]
    lengths = [prefix_len] + branch_lens + leaf_lens
    T = int(sum(lengths))
    q = _unit_rows(rng, T, h_qk, d)
    k = _unit_rows(rng, T, h_qk, d)
    v = torch.from_numpy(_normal(rng, (T, h_v, d))).to(torch.bfloat16)
    g, beta = _gates(rng, T, h_v, alpha_lo, torch.bfloat16)
    rows = Workload("cfg3_prefix_tree", q, k, v, g, beta, _cu(lengths), None, None,
                    torch.bfloat16)
    return Tree(rows, prefix_len, branch_lens, leaf_lens, leaf_parent)


def take_rows(w: Workload, segments, name="subset", initial_state=None,
              state_index=None) -> Workload:
    """A new packed batch made of the given row ranges of w (one per sequence).

    Used to build the three calls of a prefix tree and the full root-to-leaf
    paths. segments: list of lists of slices; each inner list is concatenated
    into one sequence.
    """
    idx = []
    lengths = []
    for segs in segments:
        n = 0
        for s in segs:
            idx.extend(range(s.start, s.stop))
            n += s.stop - s.start
        lengths.append(n)
    ii = torch.tensor(idx, dtype=torch.long)
    return Workload(name, w.q[ii], w.k[ii], w.v[ii], w.g[ii], w.beta[ii], _cu(lengths),
                    initial_state, state_index, w.out_dtype, w.scale)


def subset_sequences(w: Workload, seqs) -> Workload:
    """The sequences `seqs` of w (in that order) as their own packed batch,
    with their initial-state slots carried along (state_index kept)."""
    cu = w.cu_seqlens.numpy()
    segs = [[slice(int(cu[n]), int(cu[n + 1]))] for n in seqs]
    sub = take_rows(w, segs, name=w.name + "_subset")
    if w.initial_state is not None:
        if w.state_index is None:
            slot = [int(n) for n in seqs]
        else:
            slot = [int(w.state_index[n]) for n in seqs]
        sub.initial_state = w.initial_state
        sub.state_index = torch.tensor(slot, dtype=torch.int32)
    return sub


def norm_inputs(T: int, h_v: int, d_v: int, *, seed: int, z_dtype=torch.bfloat16):
    """Seeded inputs of the gated RMSNorm that follows the prefill: the output
    gate z [T, h_v, d_v] ~ N(0, 2^2) (it spans SiLU's curved range and both
    tails), stored in z_dtype, and a per-channel weight [d_v] fp32 ~ U(0.5, 1.5)
    (RMSNorm weights sit near their initial value 1)."""
    rng = np.random.default_rng(seed)
    z = torch.from_numpy(_normal(rng, (T, h_v, d_v), sd=2.0)).to(z_dtype)
    w = torch.from_numpy(rng.uniform(0.5, 1.5, d_v).astype(np.float32))
    return z, w


def prep_inputs(lengths, *, h_qk: int, d_k: int, h_v: int, d_v: int, K: int = 4, seed: int,
                slots: int = 0, bias: bool = False):
    """Seeded inputs of the GDN input prep: the packed projection rows x [T, C]
    bf16 ~ N(0, 1) (C = 2 h_qk d_k + h_v d_v); depthwise conv taps [C, K] fp32 ~
    U(-1/sqrt(K), 1/sqrt(K)) (the fan-in scale of a K-tap filter) and, if asked,
    a bias [C] ~ U(-0.1, 0.1); the gate projections a, b [T, h_v] bf16 ~ N(0, 1);
    A_log = ln A with A ~ U(1, 16) and dt_bias = ln(e^dt - 1) with dt
    log-uniform in [1e-3, 1e-1] (Mamba2's initial ranges: the decays alpha have a
    median near 0.94, a tenth below about 0.6 and a tail of strong forgetting);
    with slots > 0, carried windows [slots, K-1, C] bf16 ~ N(0, 1). Returns a
    dict of CPU tensors and cu_seqlens."""
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    C = 2 * h_qk * d_k + h_v * d_v
    bound = 1.0 / np.sqrt(K)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), h_v))
    out = {
        "x": torch.from_numpy(_normal(rng, (T, C))).to(torch.bfloat16),
        "conv_w": torch.from_numpy(rng.uniform(-bound, bound, (C, K)).astype(np.float32)),
        "conv_bias": (torch.from_numpy(rng.uniform(-0.1, 0.1, C).astype(np.float32)) if bias else None),
        "a": torch.from_numpy(_normal(rng, (T, h_v))).to(torch.bfloat16),
        "b": torch.from_numpy(_normal(rng, (T, h_v))).to(torch.bfloat16),
        "A_log": torch.from_numpy(np.log(rng.uniform(1.0, 16.0, h_v)).astype(np.float32)),
        "dt_bias": torch.from_numpy(np.log(np.expm1(dt)).astype(np.float32)),
        "conv_state": (torch.from_numpy(_normal(rng, (slots, K - 1, C))).to(torch.bfloat16) if slots else None),
        "cu_seqlens": _cu(lengths),
    }
    return out
