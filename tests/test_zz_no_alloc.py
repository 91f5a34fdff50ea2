"""gdn_prefill_varlen_noalloc: the entry point that uses the library's static
device workspace instead of a caller buffer.

The GPU test calls it through the C ABI twice in a row, on two different
batches, and compares each call with gdn_prefill_varlen (caller workspace) on
the same inputs: the same kernels run in both, so outputs and final states
must match bit for bit. The file is named to be collected last so that it also
runs after every other test has used the library; it passes alone too (the
first call in a fresh process does the one-time set-up).
"""
import ctypes
import os
import re

import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GDN_ERR_NULL, GDN_ERR_WORKSPACE = 1, 8


def test_limit_matches_header():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    m = re.search(r"#define\s+GDN_NOALLOC_MAX_SEQS\s+(\d+)", text)
    assert m and int(m.group(1)) == gdn.GDN_NOALLOC_MAX_SEQS


def test_rejected_before_any_device_call():
    # Both errors come from the descriptor alone, before the device is touched,
    # so they hold with or without a GPU; nothing is dereferenced.
    lib = gdn.load_library()
    args = [None] * 10
    assert lib.gdn_prefill_varlen_noalloc(*args, None, None) == GDN_ERR_NULL
    d = gdn.GdnDesc()
    d.num_seqs = gdn.GDN_NOALLOC_MAX_SEQS + 1
    d.total_tokens = 0
    assert lib.gdn_prefill_varlen_noalloc(*args, ctypes.byref(d), None) == GDN_ERR_WORKSPACE


def _both(w, flags=0):
    """Run w through gdn_prefill_varlen (own workspace) and the no-alloc entry
    point; return the two (out, final_state) pairs."""
    d = w.to("cuda")
    res = []
    for noalloc in (False, True):
        out = torch.full(d.v.shape, float("nan"), dtype=d.out_dtype, device="cuda")
        fs = torch.full((d.num_seqs, d.h_v, d.d_k, d.d_v), float("nan"), dtype=torch.float32,
                        device="cuda")
        desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=out.dtype,
                             initial_state=d.initial_state, max_seqlen=w.max_seqlen,
                             scale=w.scale, flags=flags)
        if noalloc:
            rc = gdn.gdn_prefill_varlen_noalloc(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens,
                                                d.initial_state, d.state_index, out, fs, desc)
        else:
            ws = torch.empty(max(gdn.gdn_workspace_bytes(desc), 256), dtype=torch.uint8,
                             device="cuda")
            desc.workspace = ws.data_ptr()
            desc.workspace_bytes = ws.numel()
            rc = gdn.gdn_prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens,
                                        d.initial_state, d.state_index, out, fs, desc)
            assert rc == gdn.GDN_OK
            assert gdn.gdn_get_device_status(desc) == gdn.GDN_OK
        assert rc == gdn.GDN_OK, gdn.gdn_status_string(rc)
        torch.cuda.synchronize()
        res.append((out, fs))
    return res


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    # Two batches in a row with different sequence counts, lengths and state
    # gathers: the second call must not see anything the first left behind.
    w1 = workloads.random_workload([130, 64, 0, 257, 1, 63], h_qk=2, h_v=4, d_k=128, d_v=128,
                                   seed=11, init_sd=0.02, n_slots=3,
                                   state_index=[2, 0, -1, 2, 1, 0])
    w2 = workloads.random_workload([500, 7, 192], h_qk=1, h_v=2, d_k=128, d_v=128, seed=12)
    for w in (w1, w2):
        (o_ref, s_ref), (o, s) = _both(w)
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(s, s_ref)
        assert not torch.isnan(s).any()


@pytest.mark.gpu
def test_noalloc_call_allocates_no_device_memory():
    # After one warm-up call (which loads the kernels and looks the static
    # workspace up), further calls leave the device's free memory unchanged.
    w = workloads.random_workload([300, 5, 70], h_qk=2, h_v=4, d_k=128, d_v=128, seed=13)
    d = w.to("cuda")
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device="cuda")
    fs = torch.empty((d.num_seqs, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device="cuda")
    desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=out.dtype, max_seqlen=w.max_seqlen)
    call = lambda: gdn.gdn_prefill_varlen_noalloc(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, None, None,
                                                  out, fs, desc)
    assert call() == gdn.GDN_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert call() == gdn.GDN_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


@pytest.mark.gpu
def test_noalloc_too_many_sequences_writes_nothing():
    n = gdn.GDN_NOALLOC_MAX_SEQS + 1
    cu = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    q = torch.zeros((n, 1, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((n, 1, 64), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((n, 1), dtype=torch.float32, device="cuda")
    out = torch.full_like(v, 7.0)
    desc = gdn.make_desc(q, v, g, cu)
    rc = gdn.gdn_prefill_varlen_noalloc(q, q, v, g, g, cu, None, None, out, None, desc)
    assert rc == GDN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
