"""fp64 CPU oracle for the gated delta rule prefill (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline /
reference arm may import this package. The product path (the CUDA library and
its binding) never does, and the two share no code.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision,
pthreads over (sequence, value head) units); this module compiles it with gcc
when the shared object is missing or older than the source, and marshals
arrays. See the C file's header for the definition it follows and the
readings it takes where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into _gdn_oracle.so (gcc -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            common = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      P, P, P, P, P, P, ctypes.c_int, P, ctypes.c_double, ctypes.c_int,
                      ctypes.c_double, P, P, P]
            lib.gdn_oracle_recurrent.argtypes = common + [ctypes.c_int]
            lib.gdn_oracle_recurrent.restype = ctypes.c_int
            lib.gdn_oracle_chunked.argtypes = common + [ctypes.c_int, ctypes.c_int]
            lib.gdn_oracle_chunked.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly to float32 on the host
        import torch
        x = x.detach().to("cpu", torch.float32).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _i64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _run(kind, q, k, v, g, beta, cu_seqlens, initial_state=None, state_index=None,
         scale: float = 0.0, l2norm: bool = True, eps: float = EPS, unit_mask=None,
         chunk: int = 64, n_threads: Optional[int] = None, want_out: bool = True
         ) -> Tuple[Optional[np.ndarray], np.ndarray]:
    lib = _load()
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    cu = _i64(cu_seqlens)
    s0 = _f32(initial_state)
    sidx = _i64(state_index)
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    N = cu.size - 1
    if k.shape != q.shape or v.shape[0] != T or g.shape != (T, h_v) or beta.shape != (T, h_v):
        raise ValueError("inconsistent shapes")
    if int(cu[-1]) != T or int(cu[0]) != 0:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    if not scale:
        scale = float(d_k) ** -0.5
    n_slots = 0 if s0 is None else s0.shape[0]
    mask = None
    if unit_mask is not None:
        mask = np.ascontiguousarray(np.asarray(unit_mask, dtype=np.uint8).reshape(N * h_v))
    out = np.zeros((T, h_v, d_v), dtype=np.float64) if want_out else None
    fs = np.zeros((N, h_v, d_k, d_v), dtype=np.float64)
    nt = default_threads() if n_threads is None else int(n_threads)
    args = [N, _ptr(cu), h_qk, h_v, d_k, d_v, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
            _ptr(s0), n_slots, _ptr(sidx), float(scale), int(bool(l2norm)), float(eps),
            _ptr(mask), _ptr(out), _ptr(fs)]
    if kind == "recurrent":
        rc = lib.gdn_oracle_recurrent(*args, nt)
    else:
        rc = lib.gdn_oracle_chunked(*args, int(chunk), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected the input (code {rc})")
    return out, fs


def recurrent(q, k, v, g, beta, cu_seqlens, initial_state=None, state_index=None, **kw):
    """Token-by-token fp64 recurrence. Returns (out [T,h_v,d_v], final [N,h_v,d_k,d_v])."""
    return _run("recurrent", q, k, v, g, beta, cu_seqlens, initial_state, state_index, **kw)


def chunked(q, k, v, g, beta, cu_seqlens, initial_state=None, state_index=None, chunk=64, **kw):
    """Chunked (WY/UT) fp64 form, for cross-checking the recurrence."""
    return _run("chunked", q, k, v, g, beta, cu_seqlens, initial_state, state_index,
                chunk=chunk, **kw)


def run_workload(w, kind: str = "recurrent", **kw):
    """Run the oracle on a workloads.Workload (host tensors)."""
    fn = recurrent if kind == "recurrent" else chunked
    return fn(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state, w.state_index,
              scale=w.scale, **kw)



def tree(q, k, v, g, beta, cu_seqlens, parent, initial_state=None, state_index=None, **kw):
    """A prefix tree of sequences: sequence n starts from the final state of
    sequence parent[n] (parent[n] in [-1, n)); a sequence with parent -1 starts
    from initial_state[state_index[n]] (or zero) as in ``recurrent``.

    This is the hand-off the open-jev-fast README describes for long prompts
    (Phase 2 item 2, "Prefix tree": the prefix's final recurrent state goes to
    each candidate) and System1-Omni PR #186 runs as compact prefix
    continuations ("Purpose and summary"). Written out without any rounding at
    the hand-off: each sequence's rows are the tail of its full root-to-node
    path (the replicated layout the README uses for linear attention), run by
    the fp64 recurrence from the root's starting state.
    Returns (out [T, h_v, d_v], final [N, h_v, d_k, d_v]).
    """
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    cu = _i64(cu_seqlens)
    par = _i64(parent)
    s0 = _f32(initial_state)
    sidx = _i64(state_index)
    N = cu.size - 1
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    if par is None or par.size != N:
        raise ValueError("parent needs one entry per sequence")
    out = np.zeros((T, h_v, d_v), dtype=np.float64)
    fs = np.zeros((N, h_v, d_k, d_v), dtype=np.float64)
    for n in range(N):
        path = [n]
        while int(par[path[-1]]) >= 0:
            p_ = int(par[path[-1]])
            if p_ >= path[-1]:
                raise ValueError(f"parent[{path[-1]}] = {p_} is not below {path[-1]}")
            path.append(p_)
        if int(par[path[-1]]) < -1:
            raise ValueError(f"parent[{path[-1]}] = {int(par[path[-1]])} is below -1")
        path.reverse()
        root = path[0]
        rows = np.concatenate([np.arange(int(cu[m]), int(cu[m + 1])) for m in path])
        if s0 is not None:
            slot = root if sidx is None else int(sidx[root])
            start = s0[slot][None] if slot >= 0 else None
        else:
            start = None
        o_p, f_p = _run("recurrent", q[rows], k[rows], v[rows], g[rows], beta[rows],
                        np.array([0, rows.size], dtype=np.int64), start,
                        None if start is None else np.array([0], dtype=np.int64), **kw)
        b, e = int(cu[n]), int(cu[n + 1])
        out[b:e] = o_p[rows.size - (e - b):]
        fs[n] = f_p[0]
    return out, fs


def gated_rmsnorm(o, z, weight, eps: float = EPS):
    """Gated RMSNorm of the prefill output, in fp64.

    For every row x = o[..., :] (one token and value head, d_v entries) and its
    gate row z[..., :]:

        y_j = w_j * x_j / sqrt(mean_j(x_j^2) + eps) * silu(z_j),
        silu(z) = z / (1 + e^{-z}).

    The open-jev-fast README lists "gated RMSNorm" among the six fused
    element-wise kernels of its Phase 2 (item 1) and puts it behind the Gated
    DeltaNet core; its item 4 reports that fusing it into that kernel was
    measured and rejected. The README gives no formula: this is the textbook
    RMS normalisation over the value dimension, a per-channel weight w [d_v]
    shared by the value heads, and a SiLU gate, with no rounding before the
    end (the caller rounds y to its storage type).
    o, z: [..., d_v]; weight: [d_v]. Returns y [..., d_v] float64.
    """
    x = np.asarray(o, dtype=np.float64)
    zz = np.asarray(z, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    if zz.shape != x.shape or w.shape != x.shape[-1:]:
        raise ValueError("z must match o, and weight must have d_v entries")
    ms = np.mean(x * x, axis=-1, keepdims=True)
    with np.errstate(over="ignore"):
        silu = zz / (1.0 + np.exp(-zz))
    return w * (x / np.sqrt(ms + float(eps))) * silu


def causal_conv_silu(x, conv_w, cu_seqlens, conv_bias=None, conv_state=None, state_index=None):
    """Causal depthwise convolution over each packed sequence, then SiLU, in fp64.

    The first step of the Gated DeltaNet input prep in the open-jev-fast README
    (Phase 2 item 1: "causal conv, SiLU, q/k/v split, ..."; reference [6] is the
    causal-conv1d kernel). For channel c and row t of a sequence that starts at
    row b, with a window of K taps (conv_w [C, K], tap K-1 on the current row):

        y[t, c] = bias[c] + sum_{j=0}^{K-1} conv_w[c, j] * x[t - (K-1) + j, c]
        u[t, c] = silu(y[t, c]) = y / (1 + e^{-y})

    where a row before b reads the sequence's carried window: conv_state
    [slots, K-1, C] holds the K-1 rows that precede the sequence (oldest first),
    slot state_index[n] (n itself if state_index is None; a negative index, or no
    conv_state, means zeros). The README's prefix-tree item replicates each
    candidate's whole path so that its convolution window sees the prefix's last
    rows; carrying the window into a continuation gives the same rows.
    Returns (u [T, C], final_state [N, K-1, C]): the K-1 last input rows of each
    sequence, oldest first, reaching into its carried window when the sequence
    is shorter than K-1.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(conv_w, dtype=np.float64)
    cu = _i64(cu_seqlens)
    T, C = x.shape
    K = w.shape[1]
    if w.shape[0] != C:
        raise ValueError("conv_w must be [C, K]")
    bias = np.zeros(C) if conv_bias is None else np.asarray(conv_bias, dtype=np.float64)
    N = cu.size - 1
    u = np.zeros((T, C))
    final = np.zeros((N, K - 1, C))
    for n in range(N):
        b, e = int(cu[n]), int(cu[n + 1])
        slot = -1
        if conv_state is not None:
            slot = n if state_index is None else int(np.asarray(state_index)[n])
        carried = (np.asarray(conv_state, dtype=np.float64)[slot] if slot >= 0
                   else np.zeros((K - 1, C)))
        seq = np.concatenate([carried, x[b:e]], axis=0)  # rows -(K-1) .. len-1
        for i in range(e - b):
            y = bias + np.sum(w.T * seq[i:i + K], axis=0)
            with np.errstate(over="ignore"):
                u[b + i] = y / (1.0 + np.exp(-y))
        final[n] = seq[seq.shape[0] - (K - 1):]
    return u, final


def gate_params(a, b, A_log, dt_bias):
    """The per-head gates of the gated delta rule from their projections, in fp64:

        g[t, h]    = -exp(A_log[h]) * softplus(a[t, h] + dt_bias[h]),
        beta[t, h] = 1 / (1 + e^{-b[t, h]}),   softplus(x) = ln(1 + e^x).

    The open-jev-fast README lists gate parameters as the last step of its GDN
    input prep (Phase 2 item 1) but gives no formula. This is the reading taken
    from the model its reference [5] defines ("Gated Delta Networks: Improving
    Mamba2 with Delta Rule"), which keeps Mamba2's decay: a per-head rate
    exp(A_log) times a softplus step, so that alpha = e^g lies in (0, 1), and a
    sigmoid for the writing strength beta. a, b: [T, H]; A_log, dt_bias: [H].
    Returns (g, beta).
    """
    a = np.asarray(a, dtype=np.float64)
    bb = np.asarray(b, dtype=np.float64)
    A = np.asarray(A_log, dtype=np.float64)
    dt = np.asarray(dt_bias, dtype=np.float64)
    softplus = np.logaddexp(0.0, a + dt)  # ln(e^0 + e^x)
    g = -np.exp(A) * softplus
    with np.errstate(over="ignore"):
        beta = 1.0 / (1.0 + np.exp(-bb))
    return g, beta


def causal_conv_silu_tree(x, conv_w, cu_seqlens, parent, conv_bias=None, conv_state=None, state_index=None):
    """``causal_conv_silu`` over a prefix tree of packed sequences: sequence n
    continues sequence parent[n] (parent[n] in [-1, n)), so its window reaches
    into the last rows of its ancestors' path, and a root's into its carried
    window (conv_state[state_index[root]], or zeros). Written out as the
    README's replicated layout (Phase 2 item 2; the prefix-tree item runs each
    candidate over its whole path so that the convolution window matches): each
    node's rows are the tail of its full root-to-node path run as one sequence.
    Returns (u [T, C], final_state [N, K-1, C])."""
    x = np.asarray(x, dtype=np.float64)
    cu = _i64(cu_seqlens)
    par = _i64(parent)
    N = cu.size - 1
    if par is None or par.size != N:
        raise ValueError("parent needs one entry per sequence")
    K = np.asarray(conv_w).shape[1]
    u = np.zeros_like(x)
    final = np.zeros((N, K - 1, x.shape[1]))
    for n in range(N):
        path = [n]
        while int(par[path[-1]]) >= 0:
            p_ = int(par[path[-1]])
            if p_ >= path[-1]:
                raise ValueError(f"parent[{path[-1]}] = {p_} is not below {path[-1]}")
            path.append(p_)
        path.reverse()
        rows = np.concatenate([np.arange(int(cu[m]), int(cu[m + 1])) for m in path]).astype(np.int64)
        root = path[0]
        si = None
        if conv_state is not None:
            si = [root if state_index is None else int(np.asarray(state_index)[root])]
        up, fp = causal_conv_silu(x[rows], conv_w, [0, rows.size], conv_bias, conv_state, si)
        b, e = int(cu[n]), int(cu[n + 1])
        u[b:e] = up[rows.size - (e - b):]
        final[n] = fp[0]
    return u, final
