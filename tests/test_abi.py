"""The C-ABI library loads, exports every entry point include/gdn.h declares,
and rejects bad calls on the host before touching the GPU.

No test here launches a kernel: every call made with fake (never dereferenced)
device addresses fails host validation first. That ordering is part of the
contract (host errors are returned before any launch and write nothing).
"""
import ctypes
import os
import re

import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

FAKE = 1 << 20  # an aligned address that is never dereferenced (validation fails first)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted([
        "gdn_abi_version", "gdn_workspace_bytes", "gdn_prefill_varlen", "gdn_prefill_varlen_noalloc",
        "gdn_tree_workspace_bytes", "gdn_prefill_tree", "gdn_get_device_status",
        "gdn_status_string", "gdn_gated_rmsnorm", "gdn_input_prep", "gdn_input_prep_tree",
        "gdn_segment_plan"])


def test_library_exports_every_declared_symbol():
    lib = gdn.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings():
    assert gdn.gdn_abi_version() == 1
    for code, name in enumerate(gdn.STATUS_NAMES):
        assert gdn.gdn_status_string(code).startswith(name)
    assert "unknown" in gdn.gdn_status_string(99)


def test_desc_layout_matches_header():
    # int32, (pad), int64, int32 x5, enum x3, int32, float, uint32, (pad), void*, size_t
    assert ctypes.sizeof(gdn.GdnDesc) == 80
    assert gdn.GdnDesc.workspace.offset == 64


def base_desc(**kw):
    d = gdn.GdnDesc()
    d.num_seqs, d.total_tokens, d.max_seqlen = 2, 100, 0
    d.h_qk, d.h_v, d.d_k, d.d_v = 16, 32, 128, 128
    d.qkv_dtype, d.gate_dtype, d.out_dtype = gdn.GDN_BF16, gdn.GDN_F32, gdn.GDN_BF16
    d.num_state_slots, d.scale, d.flags = 0, 0.0, 0
    d.workspace = FAKE * 64
    d.workspace_bytes = 1 << 16
    for k_, v_ in kw.items():
        setattr(d, k_, v_)
    return d


def call(desc, **ptrs):
    # Fake addresses are only ever passed where no device exists, so that a
    # validation slip can never turn into a launch on bogus memory.
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation calls run only without a device")
    lib = gdn.load_library()
    T = desc.total_tokens if desc else 100
    qb = max(T, 1) * 16 * 128 * 2
    base = dict(q=FAKE, k=FAKE + 4 * qb, v=FAKE + 8 * qb, g=FAKE + 16 * qb, beta=FAKE + 18 * qb,
                cu=FAKE + 20 * qb, init=None, sidx=None, out=FAKE + 32 * qb, fs=None)
    base.update(ptrs)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_prefill_varlen(P(base["q"]), P(base["k"]), P(base["v"]), P(base["g"]),
                                  P(base["beta"]), P(base["cu"]), P(base["init"]),
                                  P(base["sidx"]), P(base["out"]), P(base["fs"]),
                                  ctypes.byref(desc) if desc is not None else None, None)


E = {n: i for i, n in enumerate(gdn.STATUS_NAMES)}


def test_null_desc_and_pointers():
    lib = gdn.load_library()
    assert lib.gdn_workspace_bytes(None) == 0
    assert call(None) == E["GDN_ERR_NULL"]
    assert call(base_desc(), q=None) == E["GDN_ERR_NULL"]
    assert call(base_desc(), cu=None) == E["GDN_ERR_NULL"]
    assert call(base_desc(), out=None) == E["GDN_ERR_NULL"]
    assert lib.gdn_get_device_status(None, None) == E["GDN_ERR_NULL"]


@pytest.mark.parametrize("field,value", [("h_qk", 0), ("h_v", 24), ("d_k", 96), ("d_v", 32),
                                         ("num_seqs", -1), ("total_tokens", -5),
                                         ("max_seqlen", -1)])
def test_shape_errors(field, value):
    d = base_desc(**{field: value})
    if field == "h_v":
        d.h_qk = 16  # 24 is not a multiple of 16
    assert call(d) == E["GDN_ERR_SHAPE"]


def test_initial_state_needs_slots():
    assert call(base_desc(num_state_slots=0), init=FAKE * 200) == E["GDN_ERR_SHAPE"]
    # NULL state_index means slot n for sequence n: fewer slots than sequences is an error
    assert call(base_desc(num_state_slots=1), init=FAKE * 200) == E["GDN_ERR_SHAPE"]


@pytest.mark.parametrize("field,value", [("qkv_dtype", gdn.GDN_F32), ("gate_dtype", 7),
                                         ("out_dtype", 5)])
def test_dtype_errors(field, value):
    assert call(base_desc(**{field: value})) == E["GDN_ERR_DTYPE"]


def test_workspace_errors():
    need = gdn.gdn_workspace_bytes(base_desc())
    assert need >= 256 + 4 * 2
    assert call(base_desc(workspace=None)) == E["GDN_ERR_WORKSPACE"]
    assert call(base_desc(workspace=FAKE * 64 + 16)) == E["GDN_ERR_WORKSPACE"]
    assert call(base_desc(workspace_bytes=need - 1)) == E["GDN_ERR_WORKSPACE"]
    big = base_desc(num_seqs=100000)
    assert gdn.gdn_workspace_bytes(big) >= 256 + 4 * 100000


def test_alignment_errors():
    assert call(base_desc(), q=FAKE + 8) == E["GDN_ERR_ALIGN"]
    assert call(base_desc(), out=FAKE * 40 + 2) == E["GDN_ERR_ALIGN"]
    assert call(base_desc(), g=FAKE * 30 + 2) == E["GDN_ERR_ALIGN"]


def test_alias_errors():
    d = base_desc()
    # out overlapping v
    assert call(d, out=FAKE + 8 * 100 * 16 * 128 * 2 + 64) == E["GDN_ERR_ALIAS"]
    # final_state overlapping initial_state (one slot may feed many sequences)
    d = base_desc(num_state_slots=2)
    assert call(d, init=FAKE * 400, fs=FAKE * 400 + 1024) == E["GDN_ERR_ALIAS"]
    # final_state overlapping the workspace
    d = base_desc()
    assert call(d, fs=d.workspace) == E["GDN_ERR_ALIAS"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path only")
def test_valid_call_without_a_device_reports_cuda_or_arch():
    """With every host check passing and no GPU, the arch query fails cleanly."""
    d = base_desc()
    rc = call(d)
    assert rc in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])


def call_tree(desc, parent=FAKE * 500, **ptrs):
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation calls run only without a device")
    lib = gdn.load_library()
    T = desc.total_tokens if desc else 100
    qb = max(T, 1) * 16 * 128 * 2
    base = dict(q=FAKE, k=FAKE + 4 * qb, v=FAKE + 8 * qb, g=FAKE + 16 * qb, beta=FAKE + 18 * qb,
                cu=FAKE + 20 * qb, init=None, sidx=None, out=FAKE + 32 * qb, fs=FAKE * 600)
    base.update(ptrs)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_prefill_tree(P(base["q"]), P(base["k"]), P(base["v"]), P(base["g"]),
                                P(base["beta"]), P(base["cu"]), P(parent), P(base["init"]),
                                P(base["sidx"]), P(base["out"]), P(base["fs"]),
                                ctypes.byref(desc) if desc is not None else None, None)


def test_tree_workspace_size():
    lib = gdn.load_library()
    assert lib.gdn_tree_workspace_bytes(None) == 0
    d = base_desc(num_seqs=10)
    need = gdn.gdn_tree_workspace_bytes(d)
    assert need >= gdn.gdn_workspace_bytes(d) + 4 * 10 * 32 and need % 256 == 0


def test_tree_host_checks():
    need = gdn.gdn_tree_workspace_bytes(base_desc())
    assert call_tree(None) == E["GDN_ERR_NULL"]
    assert call_tree(base_desc(workspace_bytes=need), parent=None) == E["GDN_ERR_NULL"]
    assert call_tree(base_desc(workspace_bytes=need), fs=None) == E["GDN_ERR_NULL"]
    assert call_tree(base_desc(workspace_bytes=need, flags=gdn.GDN_FLAG_SIMT)) == E["GDN_ERR_SHAPE"]
    # the varlen workspace is not enough for the ready flags
    small = gdn.gdn_workspace_bytes(base_desc())
    assert small < need
    assert call_tree(base_desc(workspace_bytes=small)) == E["GDN_ERR_WORKSPACE"]
    assert call_tree(base_desc(workspace_bytes=need), parent=FAKE * 500 + 2) == E["GDN_ERR_ALIGN"]
    # the output overlapping the parent list
    d = base_desc(workspace_bytes=need)
    out = FAKE + 32 * 100 * 16 * 128 * 2
    assert call_tree(d, parent=out + 64) == E["GDN_ERR_ALIAS"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path only")
def test_valid_tree_call_without_a_device_reports_cuda_or_arch():
    d = base_desc(workspace_bytes=gdn.gdn_tree_workspace_bytes(base_desc()))
    assert call_tree(d) in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])


def call_norm(o=FAKE, z=FAKE * 8, w=FAKE * 16, y=FAKE * 24, rows=1000, d_v=128, xd=gdn.GDN_BF16,
              zd=gdn.GDN_BF16, eps=1e-6):
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation calls run only without a device")
    lib = gdn.load_library()
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_gated_rmsnorm(P(o), P(z), P(w), P(y), rows, d_v, xd, zd, eps, None)


def test_gated_rmsnorm_host_checks():
    assert call_norm(rows=-1) == E["GDN_ERR_SHAPE"]
    for d_v in (0, 32, 96, 512):
        assert call_norm(d_v=d_v) == E["GDN_ERR_SHAPE"]
    assert call_norm(xd=3) == E["GDN_ERR_DTYPE"]
    assert call_norm(zd=-1) == E["GDN_ERR_DTYPE"]
    for eps in (0.0, -1e-6, float("inf"), float("nan")):
        assert call_norm(eps=eps) == E["GDN_ERR_VALUE"]
    # no rows: nothing to do, whatever the pointers
    assert call_norm(rows=0, o=None, z=None, w=None, y=None) == E["GDN_OK"]
    assert call_norm(o=None) == E["GDN_ERR_NULL"]
    assert call_norm(w=None) == E["GDN_ERR_NULL"]
    assert call_norm(y=FAKE * 24 + 8) == E["GDN_ERR_ALIGN"]
    assert call_norm(w=FAKE * 16 + 4) == E["GDN_ERR_ALIGN"]
    # y may be o itself, but not a shifted view of it, nor overlap z or the weights
    assert call_norm(y=FAKE) in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])
    assert call_norm(y=FAKE + 256) == E["GDN_ERR_ALIAS"]
    assert call_norm(y=FAKE * 8 + 1024) == E["GDN_ERR_ALIAS"]
    assert call_norm(w=FAKE * 24 + 512) == E["GDN_ERR_ALIAS"]
    # fp32 o / y are twice as long: y right after a bf16-sized o overlaps an fp32 o
    assert call_norm(y=FAKE + 1000 * 128 * 2, xd=gdn.GDN_F32) == E["GDN_ERR_ALIAS"]
    assert call_norm() in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])


def test_prep_desc_layout_matches_header():
    # int32, (pad), int64, int32 x6
    assert ctypes.sizeof(gdn.GdnPrepDesc) == 40
    assert gdn.GdnPrepDesc.total_tokens.offset == 8 and gdn.GdnPrepDesc.num_state_slots.offset == 36


def prep_desc(**kw):
    d = gdn.GdnPrepDesc()
    d.num_seqs, d.total_tokens = 2, 100
    d.h_qk, d.h_v, d.d_k, d.d_v = 16, 32, 128, 128
    d.conv_width, d.num_state_slots = 4, 0
    for k_, v_ in kw.items():
        setattr(d, k_, v_)
    return d


def call_prep(desc, **ptrs):
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation calls run only without a device")
    lib = gdn.load_library()
    MB = 1 << 22  # 4 MiB apart: x (100 x 8192 bf16 = 1.6 MB) and every other array fit
    base = dict(x=MB, w=2 * MB, bias=None, cu=3 * MB, sin=None, sidx=None, a=4 * MB, b=5 * MB,
                A=6 * MB, dt=7 * MB, q=8 * MB, k=9 * MB, v=10 * MB, g=11 * MB, beta=12 * MB, sout=13 * MB)
    base.update(ptrs)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    order = ["x", "w", "bias", "cu", "sin", "sidx", "a", "b", "A", "dt", "q", "k", "v", "g", "beta", "sout"]
    return lib.gdn_input_prep(*[P(base[n]) for n in order],
                              ctypes.byref(desc) if desc is not None else None, None)


def test_input_prep_host_checks():
    MB = 1 << 22
    assert call_prep(None) == E["GDN_ERR_NULL"]
    for f, val in [("num_seqs", -1), ("total_tokens", -1), ("h_qk", 0), ("d_k", 12), ("d_v", 0),
                   ("conv_width", 1), ("conv_width", 5), ("num_state_slots", -2)]:
        assert call_prep(prep_desc(**{f: val})) == E["GDN_ERR_SHAPE"], f
    assert call_prep(prep_desc(num_seqs=0)) == E["GDN_ERR_SHAPE"]  # rows without a sequence
    assert call_prep(prep_desc(num_seqs=0, total_tokens=0), x=None, cu=None) == E["GDN_OK"]
    # a carried window needs slots (one per sequence without state_index)
    assert call_prep(prep_desc(), sin=14 * MB) == E["GDN_ERR_SHAPE"]
    assert call_prep(prep_desc(num_state_slots=1), sin=14 * MB) == E["GDN_ERR_SHAPE"]
    assert call_prep(prep_desc(), x=None) == E["GDN_ERR_NULL"]
    assert call_prep(prep_desc(), cu=None) == E["GDN_ERR_NULL"]
    assert call_prep(prep_desc(), v=None) == E["GDN_ERR_NULL"]
    assert call_prep(prep_desc(), beta=None) == E["GDN_ERR_NULL"]  # gates asked for (a given)
    assert call_prep(prep_desc(), x=MB + 8) == E["GDN_ERR_ALIGN"]
    assert call_prep(prep_desc(), sout=13 * MB + 4) == E["GDN_ERR_ALIGN"]
    assert call_prep(prep_desc(), g=11 * MB + 2) == E["GDN_ERR_ALIGN"]
    assert call_prep(prep_desc(), w=2 * MB + 4) == E["GDN_ERR_ALIGN"]
    assert call_prep(prep_desc(), a=4 * MB + 1) == E["GDN_ERR_ALIGN"]
    assert call_prep(prep_desc(), q=MB + 4096) == E["GDN_ERR_ALIAS"]     # q over x
    assert call_prep(prep_desc(), v=9 * MB + 1024) == E["GDN_ERR_ALIAS"]  # v over k
    assert call_prep(prep_desc(), g=5 * MB) == E["GDN_ERR_ALIAS"]         # g over b
    # without gates their pointers are ignored (even overlapping ones)
    assert call_prep(prep_desc(), a=None, g=MB, beta=MB) in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])
    assert call_prep(prep_desc()) in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])


def call_prep_tree(desc, parent=(1 << 22) * 15, **ptrs):
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation calls run only without a device")
    lib = gdn.load_library()
    MB = 1 << 22
    base = dict(x=MB, w=2 * MB, bias=None, cu=3 * MB, sin=None, sidx=None, a=4 * MB, b=5 * MB,
                A=6 * MB, dt=7 * MB, q=8 * MB, k=9 * MB, v=10 * MB, g=11 * MB, beta=12 * MB, sout=13 * MB)
    base.update(ptrs)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    order = ["x", "w", "bias", "cu"]
    rest = ["sin", "sidx", "a", "b", "A", "dt", "q", "k", "v", "g", "beta", "sout"]
    return lib.gdn_input_prep_tree(*[P(base[n]) for n in order], P(parent), *[P(base[n]) for n in rest],
                                   ctypes.byref(desc) if desc is not None else None, None)


def test_input_prep_tree_host_checks():
    MB = 1 << 22
    assert call_prep_tree(None) == E["GDN_ERR_NULL"]
    assert call_prep_tree(prep_desc(), parent=None) == E["GDN_ERR_NULL"]
    assert call_prep_tree(prep_desc(num_seqs=0, total_tokens=0), parent=None, x=None, cu=None) == E["GDN_OK"]
    assert call_prep_tree(prep_desc(), parent=15 * MB + 2) == E["GDN_ERR_ALIGN"]
    assert call_prep_tree(prep_desc(), parent=8 * MB + 64) == E["GDN_ERR_ALIAS"]  # parent under q
    assert call_prep_tree(prep_desc()) in (E["GDN_ERR_CUDA"], E["GDN_ERR_ARCH"])


def test_wrappers_reject_bad_shapes_before_any_call():
    # the binding's own checks run before the library is called (CPU tensors are fine)
    o = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdn.gated_rmsnorm(o, torch.zeros(4, 64, dtype=torch.bfloat16), torch.zeros(128))
    with pytest.raises(ValueError):
        gdn.gated_rmsnorm(o, o.clone(), torch.zeros(64))
    with pytest.raises(ValueError):
        gdn.gated_rmsnorm(o, o.clone(), torch.zeros(128, dtype=torch.float64))
    with pytest.raises(ValueError):
        gdn.gated_rmsnorm(o, o.clone(), torch.zeros(128), out=torch.zeros(4, 128))
    x = torch.zeros(10, 2 * 1 * 64 + 2 * 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(ValueError):  # channels do not match the split
        gdn.input_prep(x, torch.zeros(256, 4), cu, h_qk=1, d_k=64, h_v=1, d_v=64)
    with pytest.raises(ValueError):  # taps of the wrong channel count
        gdn.input_prep(x, torch.zeros(128, 4), cu, h_qk=1, d_k=64, h_v=2, d_v=64)


def test_header_is_plain_c_and_cpp():
    # the boundary is a C ABI: the header must compile as C99 and as C++
    import shutil
    import subprocess
    for cc, lang in (("gcc", "c"), ("g++", "c++")):
        if not shutil.which(cc):
            pytest.skip(f"{cc} not found")
        r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Wextra", "-Werror", "-x", lang,
                            *(["-std=c99", "-pedantic"] if lang == "c" else ["-std=c++17"]), HEADER],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def _long_desc(T, h_v=32, d=128, flags=0, big_ws=True):
    d_ = gdn.GdnDesc()
    d_.num_seqs, d_.total_tokens, d_.h_qk, d_.h_v, d_.d_k, d_.d_v = 1, T, 16 if h_v >= 16 else 1, h_v, d, d
    d_.qkv_dtype = d_.gate_dtype = d_.out_dtype = gdn.GDN_BF16
    d_.flags = flags
    if big_ws:
        d_.workspace_bytes = gdn.gdn_workspace_bytes(d_)
    return d_


def _chunks(r):
    return (r + 63) // 64


def test_segment_plan_and_workspace_host_logic():
    """Host logic of the segment scan (no device): which descriptors qualify, the
    workspace they then need, and a plan whose segments tile the sequence and whose
    two-launch makespan (longest-first list scheduling, in chunk periods) beats one
    launch of the whole sequence."""
    sms = 152
    small = gdn.gdn_workspace_bytes(_long_desc(4095))
    big = gdn.gdn_workspace_bytes(_long_desc(16384))
    assert small == 512 and big > 22 * 32 * 128 * 128 * 4  # 2 slots + 13 + 7 states, tables
    assert gdn.gdn_workspace_bytes(_long_desc(16384, flags=gdn.GDN_FLAG_NO_SEGMENT)) == 512
    assert gdn.gdn_workspace_bytes(_long_desc(16384, flags=gdn.GDN_FLAG_SIMT)) == 512
    # a workspace of the small size keeps one launch
    assert gdn.gdn_segment_plan(_long_desc(16384, big_ws=False), sms)[0] == 0
    assert gdn.gdn_segment_plan(_long_desc(4095), sms)[0] == 0
    for T, h_v in [(16384, 32), (4096, 32), (5001, 4), (65536, 32), (9000, 8), (4097, 2)]:
        G, a, b = gdn.gdn_segment_plan(_long_desc(T, h_v), sms)
        assert 3 <= G <= 8, (T, h_v, G)
        last = T - a - (G - 2) * b
        assert a >= 64 and b % 64 == 0 and 1 <= last, (T, G, a, b)
        # launch A: segment 0 and (Delta_j, Phi_j) for j = 1 .. G-2; launch C: segments 1 .. G-1
        def makespan(units):
            import heapq
            load = [0] * sms
            for u in sorted(units, reverse=True):
                heapq.heapreplace(load, load[0] + u)
            return max(load)
        ua = [_chunks(a)] * h_v + [_chunks(b)] * (2 * (G - 2) * h_v)
        uc = [_chunks(b)] * ((G - 2) * h_v) + [_chunks(last)] * h_v
        assert makespan(ua) + makespan(uc) < 0.85 * _chunks(T), (T, h_v, G, a, b)
    assert gdn.gdn_segment_plan(_long_desc(16384), sms) == (4, 2176, 4736)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_segment_plan(_long_desc(16384), 0)


def test_regular_library_has_no_trace_code():
    """The per-role clock trace (include/gdn_trace.h) exists only in the tracing build."""
    lib = gdn.load_library()
    for name in ("gdn_trace_set_cta", "gdn_trace_clear", "gdn_trace_read"):
        assert not hasattr(lib, name), name


def test_bounds_status_is_named():
    assert gdn.STATUS_NAMES[14] == "GDN_ERR_BOUNDS"
    assert b"GDN_ERR_BOUNDS" in gdn.load_library().gdn_status_string(14)
