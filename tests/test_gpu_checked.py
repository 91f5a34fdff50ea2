"""The bounds-checked build (build(checked=True), libgdn_checked.so): every global
index the kernels compute from their inputs is checked against its buffer, and a
failure would report GDN_ERR_BOUNDS and skip the access. It stands in for a memory
checker, which this GPU pool does not run. On every workload here the checked build
reports no violation and writes the same bits as the regular library."""
import ctypes

import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import workloads
from gated_deltanet_linear_prefill_gb300.build import build

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _load(path):
    lib = ctypes.CDLL(path)
    D = ctypes.POINTER(gdn.GdnDesc)
    lib.gdn_prefill_varlen.argtypes = [P] * 10 + [D, P]
    lib.gdn_prefill_varlen.restype = ctypes.c_int
    lib.gdn_prefill_tree.argtypes = [P] * 11 + [D, P]
    lib.gdn_prefill_tree.restype = ctypes.c_int
    lib.gdn_workspace_bytes.argtypes = [D]
    lib.gdn_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_tree_workspace_bytes.argtypes = [D]
    lib.gdn_tree_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_get_device_status.argtypes = [D, P]
    lib.gdn_get_device_status.restype = ctypes.c_int
    return lib


@pytest.fixture(scope="module")
def libs():
    return {"regular": _load(gdn.load_library()._name), "checked": _load(build(checked=True))}


def _ptr(t):
    return P(t.data_ptr() if t is not None else 0)


def _run(lib, w, parent=None, flags=0):
    d = w.to("cuda")
    out = torch.full(d.v.shape, float("nan"), dtype=d.out_dtype, device="cuda")
    fs = torch.full((d.num_seqs, d.h_v, d.d_k, d.d_v), float("nan"), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype, initial_state=d.initial_state,
                         max_seqlen=w.max_seqlen, flags=flags)
    if parent is None:
        need = lib.gdn_workspace_bytes(ctypes.byref(desc))
    else:
        need = lib.gdn_tree_workspace_bytes(ctypes.byref(desc))
    ws = torch.empty(max(256, need), dtype=torch.uint8, device="cuda")
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    if parent is None:
        rc = lib.gdn_prefill_varlen(_ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(d.g), _ptr(d.beta), _ptr(d.cu_seqlens),
                                    _ptr(d.initial_state), _ptr(d.state_index), _ptr(out), _ptr(fs),
                                    ctypes.byref(desc), None)
    else:
        par = torch.tensor(parent, dtype=torch.int32, device="cuda")
        rc = lib.gdn_prefill_tree(_ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(d.g), _ptr(d.beta), _ptr(d.cu_seqlens),
                                  _ptr(par), _ptr(d.initial_state), _ptr(d.state_index), _ptr(out), _ptr(fs),
                                  ctypes.byref(desc), None)
    assert rc == gdn.GDN_OK
    st = lib.gdn_get_device_status(ctypes.byref(desc), None)
    return st, out.cpu(), fs.cpu()


CASES = {
    "edges_d128_gathered": lambda: (workloads.random_workload(
        [0, 1, 63, 64, 65, 127, 128, 129, 0, 200, 2], h_qk=2, h_v=4, d_k=128, d_v=128, seed=7, alpha_lo=0.8,
        gate_dtype=torch.float32, init_sd=0.05, n_slots=3, state_index=[0, 1, 2, -1, 0, 0, 1, 2, -1, 1, 2]), None),
    "edges_d64_f32_out": lambda: (workloads.random_workload(
        [5, 64, 300, 0, 77], h_qk=1, h_v=2, d_k=64, d_v=64, seed=8, gate_dtype=torch.bfloat16,
        out_dtype=torch.float32, init_sd=0.05), None),
    "config0": lambda: (workloads.config(0), None),
    "segment_scan_5001": lambda: (workloads.random_workload(
        [5001], h_qk=2, h_v=4, d_k=128, d_v=128, seed=9, gate_dtype=torch.float32, init_sd=0.05), None),
    "tree_config3": lambda: (workloads.tree_config().rows,
                             [-1] + [0] * len(workloads.tree_config().branch_lens)
                             + [1 + b for b in workloads.tree_config().leaf_parent]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_checked_build_finds_nothing_and_matches(libs, name):
    w, parent = CASES[name]()
    st_c, o_c, s_c = _run(libs["checked"], w, parent)
    st_r, o_r, s_r = _run(libs["regular"], w, parent)
    assert st_c == gdn.GDN_OK, gdn.STATUS_NAMES[st_c] if 0 <= st_c < len(gdn.STATUS_NAMES) else st_c
    assert st_r == gdn.GDN_OK
    assert not torch.isnan(o_c.float()).any() and torch.equal(o_c, o_r), name
    assert torch.equal(s_c, s_r), name
