"""Parity of the gated RMSNorm kernel (through the C ABI) with the fp64 oracle.

Bound: the kernel works in fp32 and rounds once to y's type. Its fp32
arithmetic (about ten operations, the fast exponential and division of the
SiLU and the reciprocal square root) stays within 2e-6 of the value, relative,
for the |z| <= 20 these inputs hold; rounding y to bf16 adds up to half an ulp,
just under 2^-8 relative for values just above a power of two. The tests allow
2^-8 + 1e-5 (bf16 y) and 1e-5 (fp32 y) relative, plus 1e-30 absolute for the
values near zero that SiLU produces in the negative tail.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_prefill_gb300 as gdn
import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = {torch.bfloat16: 2.0 ** -8 + 1e-5, torch.float32: 1e-5}


def _check(y, o, z, w, eps, rows=None):
    y = y.double().cpu().numpy().reshape(-1, o.shape[-1])
    o_ = o.float().cpu().numpy().reshape(-1, o.shape[-1])
    z_ = z.float().cpu().numpy().reshape(-1, o.shape[-1])
    if rows is not None:
        y, o_, z_ = y[rows], o_[rows], z_[rows]
    ref = oracle.gated_rmsnorm(o_, z_, w.cpu().numpy(), eps)
    tol = RTOL[o.dtype] * np.abs(ref) + 1e-30
    bad = np.abs(y - ref) > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} entries out of bound; worst "
                           f"{float(np.max(np.abs(y - ref) / (np.abs(ref) + 1e-30))):.3e} relative")


@pytest.mark.parametrize("d_v", [64, 128, 256])
@pytest.mark.parametrize("xd,zd", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                   (torch.float32, torch.bfloat16), (torch.float32, torch.float32)])
def test_parity_small(d_v, xd, zd):
    # 1,001 tokens x 3 heads: a ragged last row group and a grid of several waves
    T, H = 1001, 3
    rng = np.random.default_rng(d_v)
    o = torch.from_numpy(rng.standard_normal((T, H, d_v)).astype(np.float32) *
                         rng.uniform(0.01, 3.0, (T, H, 1)).astype(np.float32)).to(xd)
    z, w = workloads.norm_inputs(T, H, d_v, seed=d_v + 1, z_dtype=zd)
    y = gdn.gated_rmsnorm(o.cuda(), z.cuda(), w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    _check(y, o, z, w, 1e-6)


def test_in_place_rows_not_multiple():
    # 201 tokens x 4 heads = 804 rows of 128 (not a multiple of the 2-row groups x 16),
    # y written over o
    rng = np.random.default_rng(8)
    o = torch.from_numpy(rng.standard_normal((201, 4, 128)).astype(np.float32)).to(torch.bfloat16)
    z, w = workloads.norm_inputs(201, 4, 128, seed=10)
    od = o.cuda()
    y = gdn.gated_rmsnorm(od, z.cuda(), w.cuda(), eps=1e-5, out=od)
    torch.cuda.synchronize()
    assert y.data_ptr() == od.data_ptr()
    _check(y, o, z, w, 1e-5)


def test_after_prefill():
    # the layer's chain, prefill then norm, against the oracle's prefill then norm.
    # The prefill's bf16 output is held to 1e-2 relative Frobenius; normalising a
    # row divides by its own RMS, which keeps a row's relative error (up to the
    # error of the RMS itself), so the chain is held to 2e-2.
    wl = workloads.random_workload([70, 130, 1], h_qk=2, h_v=4, d_k=128, d_v=128, seed=9)
    d = wl.to("cuda")
    o, _ = gdn.prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, want_final_state=False,
                              check_device=True)
    z, w = workloads.norm_inputs(o.shape[0], 4, 128, seed=10)
    y = gdn.gated_rmsnorm(o, z.cuda(), w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    o_ref, _ = oracle.run_workload(wl)
    y_ref = oracle.gated_rmsnorm(o_ref, z.float().numpy(), w.numpy(), 1e-6)
    y = y.double().cpu().numpy()
    rel = np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref)
    assert rel <= 2e-2, rel


def test_zero_rows_and_extremes():
    w = torch.ones(128, device="cuda")
    e = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert gdn.gated_rmsnorm(e, e.clone(), w).numel() == 0
    # a zero row stays zero; huge and tiny row scales normalise alike; z at +-60
    o = torch.zeros((4, 128), dtype=torch.float32)
    o[1] = torch.linspace(-1, 1, 128) * 1e15  # squares stay inside fp32
    o[2] = torch.linspace(-1, 1, 128) * 1e-15
    o[3] = torch.linspace(-1, 1, 128)
    z = torch.full((4, 128), 3.0)
    z[3, ::2] = -60.0
    z[3, 1::2] = 60.0
    y = gdn.gated_rmsnorm(o.cuda(), z.cuda(), w, eps=1e-6)
    torch.cuda.synchronize()
    assert torch.all(y[0] == 0)
    assert torch.isfinite(y).all()
    _check(y, o, z, w.cpu(), 1e-6, rows=[1, 3])


def test_full_size_sampled_rows():
    # the 74-prompt workload's output shape [62,875, 32, 128] bf16, as bench.py
    # launches it; 3,000 sampled rows against the oracle
    T, H, D = 62875, 32, 128
    o, _ = workloads.norm_inputs(T, H, D, seed=13)  # a N(0, 2^2) bf16 tensor of o's shape
    z, w = workloads.norm_inputs(T, H, D, seed=11)
    y = gdn.gated_rmsnorm(o.cuda(), z.cuda(), w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    rows = np.random.default_rng(12).choice(T * H, 3000, replace=False)
    rows.sort()
    _check(y, o, z, w, 1e-6, rows=rows)
