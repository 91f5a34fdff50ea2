"""Python binding of libgdn.so, the GB300 gated delta rule prefill library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/gdn.h. PyTorch supplies device
memory and streams. The functions named like the C entry points
(``gdn_prefill_varlen``, ``gdn_workspace_bytes``, ``gdn_get_device_status``,
``gdn_status_string``, ``gdn_abi_version``) take the same arguments, with torch
tensors in place of raw pointers; ``prefill_varlen`` is a convenience wrapper
that allocates outputs and the workspace with torch.

There is no fallback: if libgdn.so cannot be built or loaded, or the device is
not sm_103, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = [
    "GdnError", "GdnDesc", "GDN_OK", "GDN_BF16", "GDN_F32", "GDN_FLAG_NO_L2NORM", "GDN_FLAG_SIMT", "GDN_FLAG_NO_SEGMENT",
    "gdn_abi_version", "gdn_workspace_bytes", "gdn_prefill_varlen", "gdn_get_device_status",
    "gdn_status_string", "make_desc", "prefill_varlen", "library_path", "load_library",
    "gdn_gated_rmsnorm", "gated_rmsnorm", "GdnPrepDesc", "gdn_input_prep", "gdn_input_prep_tree", "input_prep",
]

ABI_VERSION = 1
GDN_BF16, GDN_F32 = 0, 1
GDN_OK = 0
GDN_FLAG_NO_L2NORM = 0x1
GDN_FLAG_SIMT = 0x2
GDN_FLAG_TEST_CHILD_FIRST = 0x4  # tests only: fault injection for the bounded waits (include/gdn.h)
GDN_FLAG_NO_SEGMENT = 0x8  # one sequence in one launch even when the segment scan applies
GDN_NOALLOC_MAX_SEQS = 16384  # include/gdn.h
STATUS_NAMES = ["GDN_OK", "GDN_ERR_NULL", "GDN_ERR_SHAPE", "GDN_ERR_DTYPE", "GDN_ERR_ALIGN",
                "GDN_ERR_SEQLENS", "GDN_ERR_STATE_INDEX", "GDN_ERR_ALIAS", "GDN_ERR_WORKSPACE",
                "GDN_ERR_ARCH", "GDN_ERR_CUDA", "GDN_ERR_DEVICE_TIMEOUT", "GDN_ERR_PARENT",
                "GDN_ERR_VALUE", "GDN_ERR_BOUNDS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        super().__init__(f"{where}: {gdn_status_string(code)} ({code})" if where else
                         f"{gdn_status_string(code)} ({code})")


class GdnDesc(ctypes.Structure):
    """Mirror of gdn_desc (include/gdn.h)."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("max_seqlen", ctypes.c_int32),
        ("h_qk", ctypes.c_int32),
        ("h_v", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int),
        ("gate_dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("num_state_slots", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class GdnPrepDesc(ctypes.Structure):
    """Mirror of gdn_prep_desc (include/gdn.h)."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("h_qk", ctypes.c_int32),
        ("h_v", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("conv_width", ctypes.c_int32),
        ("num_state_slots", ctypes.c_int32),
    ]


def library_path() -> str:
    return os.path.join(_HERE, "libgdn.so")


def load_library(build_if_missing: bool = True):
    """Load libgdn.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        if build_if_missing and not _build.up_to_date():
            _build.build()
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libgdn.so is missing at {path}; build it with "
                               "`python -m gated_deltanet_linear_prefill_gb300.build`")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.gdn_abi_version.argtypes = []
        lib.gdn_abi_version.restype = ctypes.c_int
        lib.gdn_workspace_bytes.argtypes = [ctypes.POINTER(GdnDesc)]
        lib.gdn_workspace_bytes.restype = ctypes.c_size_t
        lib.gdn_prefill_varlen.argtypes = [P] * 10 + [ctypes.POINTER(GdnDesc), P]
        lib.gdn_prefill_varlen.restype = ctypes.c_int
        lib.gdn_prefill_varlen_noalloc.argtypes = [P] * 10 + [ctypes.POINTER(GdnDesc), P]
        lib.gdn_prefill_varlen_noalloc.restype = ctypes.c_int
        lib.gdn_tree_workspace_bytes.argtypes = [ctypes.POINTER(GdnDesc)]
        lib.gdn_tree_workspace_bytes.restype = ctypes.c_size_t
        lib.gdn_segment_plan.argtypes = [ctypes.POINTER(GdnDesc), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
        lib.gdn_segment_plan.restype = ctypes.c_int
        lib.gdn_prefill_tree.argtypes = [P] * 11 + [ctypes.POINTER(GdnDesc), P]
        lib.gdn_prefill_tree.restype = ctypes.c_int
        lib.gdn_gated_rmsnorm.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_float, P]
        lib.gdn_gated_rmsnorm.restype = ctypes.c_int
        lib.gdn_input_prep.argtypes = [P] * 16 + [ctypes.POINTER(GdnPrepDesc), P]
        lib.gdn_input_prep.restype = ctypes.c_int
        lib.gdn_input_prep_tree.argtypes = [P] * 17 + [ctypes.POINTER(GdnPrepDesc), P]
        lib.gdn_input_prep_tree.restype = ctypes.c_int
        lib.gdn_get_device_status.argtypes = [ctypes.POINTER(GdnDesc), P]
        lib.gdn_get_device_status.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        if lib.gdn_abi_version() != ABI_VERSION:
            raise RuntimeError(f"libgdn.so ABI {lib.gdn_abi_version()} != binding ABI {ABI_VERSION}")
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {dt}")


def gdn_abi_version() -> int:
    return int(load_library().gdn_abi_version())


def gdn_status_string(code: int) -> str:
    try:
        return load_library().gdn_status_string(int(code)).decode()
    except Exception:  # library unavailable: still name the code
        c = int(code)
        return STATUS_NAMES[c] if 0 <= c < len(STATUS_NAMES) else f"status {c}"


def gdn_workspace_bytes(desc: GdnDesc) -> int:
    return int(load_library().gdn_workspace_bytes(ctypes.byref(desc)))


def gdn_prefill_varlen(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                       final_state, desc: GdnDesc, stream=None) -> int:
    """The C entry point with tensors for pointers; returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      _ptr(cu_seqlens), _ptr(initial_state), _ptr(state_index),
                                      _ptr(out), _ptr(final_state), ctypes.byref(desc),
                                      _stream_handle(stream)))


def gdn_prefill_varlen_noalloc(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                               final_state, desc: GdnDesc, stream=None) -> int:
    """The C entry point that uses the library's static workspace (no
    allocation; desc.workspace is ignored); returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_prefill_varlen_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                              _ptr(cu_seqlens), _ptr(initial_state),
                                              _ptr(state_index), _ptr(out), _ptr(final_state),
                                              ctypes.byref(desc), _stream_handle(stream)))


def gdn_tree_workspace_bytes(desc: GdnDesc) -> int:
    return int(load_library().gdn_tree_workspace_bytes(ctypes.byref(desc)))


def gdn_segment_plan(desc: GdnDesc, sms: int):
    """(segments, rows of segment 0, rows of each later segment) that gdn_prefill_varlen
    takes for this descriptor on `sms` SMs; segments == 0 means one launch."""
    G, a, b = ctypes.c_int32(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = load_library().gdn_segment_plan(ctypes.byref(desc), int(sms), ctypes.byref(G), ctypes.byref(a),
                                         ctypes.byref(b))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_segment_plan")
    return int(G.value), int(a.value), int(b.value)


def gdn_prefill_tree(q, k, v, g, beta, cu_seqlens, parent, initial_state, state_index, out,
                     final_state, desc: GdnDesc, stream=None) -> int:
    """The C tree entry point with tensors for pointers; returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_prefill_tree(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(cu_seqlens), _ptr(parent), _ptr(initial_state),
                                    _ptr(state_index), _ptr(out), _ptr(final_state),
                                    ctypes.byref(desc), _stream_handle(stream)))


def gdn_get_device_status(desc: GdnDesc, stream=None) -> int:
    """Synchronises the stream and returns the device status word's code."""
    return int(load_library().gdn_get_device_status(ctypes.byref(desc), _stream_handle(stream)))


def make_desc(q, v, g, cu_seqlens, *, out_dtype=torch.bfloat16, initial_state=None,
              max_seqlen: int = 0, scale: float = 0.0, flags: int = 0, workspace=None,
              h_qk: Optional[int] = None) -> GdnDesc:
    """A descriptor for tensors shaped as in include/gdn.h. The total token
    count is q's row count (no device read)."""
    d = GdnDesc()
    d.num_seqs = int(cu_seqlens.numel()) - 1
    d.total_tokens = int(q.shape[0])
    d.max_seqlen = int(max_seqlen)
    d.h_qk = int(q.shape[1]) if h_qk is None else int(h_qk)
    d.h_v = int(v.shape[1])
    d.d_k = int(q.shape[2])
    d.d_v = int(v.shape[2])
    d.qkv_dtype = _dtype_code(q.dtype)
    d.gate_dtype = _dtype_code(g.dtype)
    d.out_dtype = _dtype_code(out_dtype)
    d.num_state_slots = 0 if initial_state is None else int(initial_state.shape[0])
    d.scale = float(scale)
    d.flags = int(flags)
    if workspace is not None:
        d.workspace = workspace.data_ptr()
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    return d


def prefill_varlen(q, k, v, g, beta, cu_seqlens, *, initial_state=None, state_index=None,
                   out=None, final_state=None, out_dtype=None, want_final_state: bool = True,
                   max_seqlen: int = 0, scale: float = 0.0, flags: int = 0, workspace=None,
                   stream=None, check_device: bool = False
                   ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Gated delta rule prefill over packed sequences (see include/gdn.h).

    q, k [T, h_qk, d_k] bf16; v [T, h_v, d_v] bf16; g, beta [T, h_v] bf16/fp32;
    cu_seqlens [N+1] int32; initial_state [slots, h_v, d_k, d_v] fp32;
    state_index [N] int32. Returns (out [T, h_v, d_v], final_state
    [N, h_v, d_k, d_v] fp32 or None). Raises GdnError on a non-OK status;
    with check_device=True it also synchronises and checks the device status.
    """
    dev = q.device
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or torch.bfloat16, device=dev)
    N = int(cu_seqlens.numel()) - 1
    if final_state is None and want_final_state:
        final_state = torch.empty((N, v.shape[1], q.shape[2], v.shape[2]), dtype=torch.float32,
                                  device=dev)
    desc = make_desc(q, v, g, cu_seqlens, out_dtype=out.dtype, initial_state=initial_state,
                     max_seqlen=max_seqlen, scale=scale, flags=flags)
    if workspace is None:
        need = gdn_workspace_bytes(desc)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = gdn_prefill_varlen(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                            final_state, desc, stream)
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_prefill_varlen")
    if check_device:
        rc = gdn_get_device_status(desc, stream)
        if rc != GDN_OK:
            raise GdnError(rc, "device status")
    return out, final_state


def prefill_tree(q, k, v, g, beta, cu_seqlens, parent, *, initial_state=None, state_index=None,
                 out=None, final_state=None, out_dtype=None, max_seqlen: int = 0,
                 scale: float = 0.0, flags: int = 0, workspace=None, stream=None,
                 check_device: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """A prefix tree of packed sequences in one launch (see include/gdn.h):
    sequence n continues from the final state of sequence parent[n] (int32 [N],
    parent[n] in [-1, n); -1 starts from initial_state[state_index[n]] or zero).
    Returns (out [T, h_v, d_v], final_state [N, h_v, d_k, d_v] fp32)."""
    dev = q.device
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or torch.bfloat16, device=dev)
    N = int(cu_seqlens.numel()) - 1
    if final_state is None:
        final_state = torch.empty((N, v.shape[1], q.shape[2], v.shape[2]), dtype=torch.float32,
                                  device=dev)
    desc = make_desc(q, v, g, cu_seqlens, out_dtype=out.dtype, initial_state=initial_state,
                     max_seqlen=max_seqlen, scale=scale, flags=flags)
    if workspace is None:
        need = gdn_tree_workspace_bytes(desc)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = gdn_prefill_tree(q, k, v, g, beta, cu_seqlens, parent, initial_state, state_index, out,
                          final_state, desc, stream)
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_prefill_tree")
    if check_device:
        rc = gdn_get_device_status(desc, stream)
        if rc != GDN_OK:
            raise GdnError(rc, "device status")
    return out, final_state


def gdn_gated_rmsnorm(o, z, weight, y, rows: int, d_v: int, x_dtype: int, z_dtype: int, eps: float,
                      stream=None) -> int:
    """The C entry point with tensors for pointers; returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_gated_rmsnorm(_ptr(o), _ptr(z), _ptr(weight), _ptr(y), int(rows), int(d_v),
                                     int(x_dtype), int(z_dtype), float(eps), _stream_handle(stream)))


def gated_rmsnorm(o, z, weight, *, eps: float = 1e-6, out=None, stream=None) -> torch.Tensor:
    """Gated RMSNorm of the prefill output (see include/gdn.h):
    y = weight * o / sqrt(mean(o^2 over d_v) + eps) * silu(z), per row of d_v.

    o [..., d_v] bf16/fp32 (e.g. prefill_varlen's [T, h_v, d_v] output); z the
    same shape, bf16/fp32; weight [d_v] fp32. out (default: new, o's shape and
    type) may be o itself. Raises GdnError on a non-OK status."""
    if out is None:
        out = torch.empty_like(o)
    d_v = int(o.shape[-1])
    rows = o.numel() // d_v if d_v else 0
    if tuple(z.shape) != tuple(o.shape) or tuple(out.shape) != tuple(o.shape) or out.dtype != o.dtype:
        raise ValueError("z and out must have o's shape (and out o's dtype)")
    if tuple(weight.shape) != (d_v,) or weight.dtype != torch.float32:
        raise ValueError("weight must be fp32 with d_v entries")
    for t in (o, z, weight, out):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    rc = gdn_gated_rmsnorm(o, z, weight, out, rows, d_v, _dtype_code(o.dtype), _dtype_code(z.dtype), eps,
                           stream)
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_gated_rmsnorm")
    return out


def gdn_input_prep(x, conv_w, conv_bias, cu_seqlens, conv_state_in, state_index, a, b, A_log, dt_bias,
                   q, k, v, g, beta, conv_state_out, desc: GdnPrepDesc, stream=None) -> int:
    """The C entry point with tensors for pointers; returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_input_prep(_ptr(x), _ptr(conv_w), _ptr(conv_bias), _ptr(cu_seqlens), _ptr(conv_state_in),
                                  _ptr(state_index), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(q),
                                  _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(conv_state_out),
                                  ctypes.byref(desc), _stream_handle(stream)))


def gdn_input_prep_tree(x, conv_w, conv_bias, cu_seqlens, parent, conv_state_in, state_index, a, b, A_log,
                        dt_bias, q, k, v, g, beta, conv_state_out, desc: GdnPrepDesc, stream=None) -> int:
    """The C tree entry point with tensors for pointers; returns the gdn_status code."""
    lib = load_library()
    return int(lib.gdn_input_prep_tree(_ptr(x), _ptr(conv_w), _ptr(conv_bias), _ptr(cu_seqlens), _ptr(parent),
                                       _ptr(conv_state_in), _ptr(state_index), _ptr(a), _ptr(b), _ptr(A_log),
                                       _ptr(dt_bias), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       _ptr(conv_state_out), ctypes.byref(desc), _stream_handle(stream)))


def input_prep(x, conv_w, cu_seqlens, *, h_qk: int, d_k: int, h_v: int, d_v: int, conv_bias=None,
               conv_state=None, state_index=None, a=None, b=None, A_log=None, dt_bias=None,
               parent=None, want_conv_state: bool = True, stream=None):
    """GDN input prep (see include/gdn.h): causal depthwise conv + SiLU over the
    packed rows x [T, C] bf16 (C = 2 h_qk d_k + h_v d_v), split into q, k [T, h_qk,
    d_k] and v [T, h_v, d_v] bf16, and, when a is given, the gates g, beta
    [T, h_v] fp32. conv_w [C, K] fp32; conv_state [slots, K-1, C] bf16. With
    parent (int32 [N], parent[n] in [-1, n)) the sequences form a prefix tree and
    a child's window comes from its ancestors' rows (gdn_input_prep_tree).
    Returns (q, k, v, g, beta, conv_state_out [N, K-1, C] bf16 or None); g and
    beta are None without a. Raises GdnError on a non-OK status."""
    dev = x.device
    T = int(x.shape[0])
    N = int(cu_seqlens.numel()) - 1
    K = int(conv_w.shape[1])
    C = int(x.shape[1])
    if C != 2 * h_qk * d_k + h_v * d_v or tuple(conv_w.shape) != (C, K):
        raise ValueError("x must have 2 h_qk d_k + h_v d_v channels and conv_w must be [C, K]")
    q = torch.empty((T, h_qk, d_k), dtype=torch.bfloat16, device=dev)
    k = torch.empty((T, h_qk, d_k), dtype=torch.bfloat16, device=dev)
    v = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device=dev)
    g = beta = None
    if a is not None:
        g = torch.empty((T, h_v), dtype=torch.float32, device=dev)
        beta = torch.empty((T, h_v), dtype=torch.float32, device=dev)
    cs = torch.empty((N, K - 1, C), dtype=torch.bfloat16, device=dev) if want_conv_state else None
    d = GdnPrepDesc()
    d.num_seqs, d.total_tokens = N, T
    d.h_qk, d.h_v, d.d_k, d.d_v = h_qk, h_v, d_k, d_v
    d.conv_width = K
    d.num_state_slots = 0 if conv_state is None else int(conv_state.shape[0])
    if parent is None:
        rc = gdn_input_prep(x, conv_w, conv_bias, cu_seqlens, conv_state, state_index, a, b, A_log, dt_bias,
                            q, k, v, g, beta, cs, d, stream)
    else:
        rc = gdn_input_prep_tree(x, conv_w, conv_bias, cu_seqlens, parent, conv_state, state_index, a, b, A_log,
                                 dt_bias, q, k, v, g, beta, cs, d, stream)
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_input_prep" if parent is None else "gdn_input_prep_tree")
    return q, k, v, g, beta, cs
