"""Pins for the oracle's GDN input prep (CPU): the causal depthwise conv + SiLU
and the gate parameters, each against closed forms and identities.

SiLU is taken off with silu(y) - silu(-y) = y: running the oracle on x and on
-x (with -bias) gives the convolution itself, which shifts, impulses and
splits then pin; a reversed tap order, a window off by one, a leak across
sequences or a wrong carried state each fail one of them.
"""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def conv_only(x, w, cu, bias=None, state=None, sidx=None):
    nb = None if bias is None else -np.asarray(bias)
    ns = None if state is None else -np.asarray(state)
    up, fp = oracle.causal_conv_silu(x, w, cu, bias, state, sidx)
    um, fm = oracle.causal_conv_silu(-np.asarray(x), w, cu, nb, ns, sidx)
    np.testing.assert_allclose(fm, -fp, rtol=0, atol=0)
    return up - um, fp


def test_current_row_tap_is_silu():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((10, 6)) * 3
    w = np.zeros((6, 4))
    w[:, 3] = 1.0
    u, _ = oracle.causal_conv_silu(x, w, [0, 10])
    np.testing.assert_allclose(u[:, 0][x[:, 0] == 0], 0.0)
    np.testing.assert_allclose(u - oracle.causal_conv_silu(-x, w, [0, 10])[0], x, rtol=1e-14)
    # silu(1) = e / (1 + e)
    u1, _ = oracle.causal_conv_silu(np.ones((1, 6)), w, [0, 1])
    np.testing.assert_allclose(u1, math.e / (1 + math.e), rtol=1e-15)


def test_oldest_tap_shifts_by_three_within_each_sequence():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((12, 5))
    w = np.zeros((5, 4))
    w[:, 0] = 1.0
    cu = [0, 7, 7, 12]  # an empty sequence in the middle
    y, _ = conv_only(x, w, cu)
    expect = np.zeros_like(x)
    for b, e in ((0, 7), (7, 12)):
        expect[b + 3:e] = x[b:e - 3]
    np.testing.assert_allclose(y, expect, atol=1e-14)


def test_impulse_response_is_the_taps():
    w = np.array([[0.5, -1.25, 2.0, 0.75], [1.0, 2.0, 3.0, 4.0]])
    x = np.zeros((9, 2))
    x[2, 0] = 1.0
    x[5, 1] = 1.0
    y, _ = conv_only(x, w, [0, 9])
    # an input at row r reaches rows r .. r+3 through taps 3, 2, 1, 0
    np.testing.assert_allclose(y[2:6, 0], [0.75, 2.0, -1.25, 0.5], atol=1e-15)
    np.testing.assert_allclose(y[5:9, 1], [4.0, 3.0, 2.0, 1.0], atol=1e-15)
    assert np.all(y[:2] == 0) and y[6:, 0].sum() == 0


def test_bias_alone():
    bias = np.array([0.3, -2.0, 5.0])
    y, _ = conv_only(np.zeros((4, 3)), np.ones((3, 4)), [0, 4], bias=bias)
    np.testing.assert_allclose(y, np.tile(bias, (4, 1)), rtol=1e-14)


def test_sequences_do_not_mix():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((20, 4))
    w = rng.standard_normal((4, 4))
    cu = [0, 6, 13, 20]
    u, f = oracle.causal_conv_silu(x, w, cu)
    x2 = x.copy()
    x2[6:13] = rng.standard_normal((7, 4)) * 10  # change the middle sequence only
    u2, f2 = oracle.causal_conv_silu(x2, w, cu)
    np.testing.assert_array_equal(u[:6], u2[:6])
    np.testing.assert_array_equal(u[13:], u2[13:])
    np.testing.assert_array_equal(f[[0, 2]], f2[[0, 2]])


def test_split_with_carried_window_equals_one_run():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((17, 8))
    w = rng.standard_normal((8, 4))
    bias = rng.standard_normal(8)
    s0 = rng.standard_normal((2, 3, 8))
    u, f = oracle.causal_conv_silu(x, w, [0, 17], bias, s0, [1])
    for cut in (1, 2, 5, 16):
        ua, fa = oracle.causal_conv_silu(x[:cut], w, [0, cut], bias, s0, [1])
        ub, fb = oracle.causal_conv_silu(x[cut:], w, [0, 17 - cut], bias, fa, [0])
        np.testing.assert_allclose(np.concatenate([ua, ub]), u, rtol=1e-14, atol=1e-15)
        np.testing.assert_array_equal(fb, f)


def test_final_window():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 3))
    s0 = rng.standard_normal((3, 3, 3))
    # sequences of 5, 1 and 0 rows from slots 2, 0 and 1
    _, f = oracle.causal_conv_silu(x, np.ones((3, 4)), [0, 5, 6, 6], None, s0, [2, 0, 1])
    np.testing.assert_array_equal(f[0], x[2:5])
    np.testing.assert_array_equal(f[1], np.concatenate([s0[0][1:], x[5:6]]))
    np.testing.assert_array_equal(f[2], s0[1])
    # a negative slot, or no state, is zeros
    _, f = oracle.causal_conv_silu(x, np.ones((3, 4)), [0, 1, 6], None, s0, [-1, 2])
    np.testing.assert_array_equal(f[0], np.concatenate([np.zeros((2, 3)), x[0:1]]))


def test_gate_closed_forms():
    A_log = np.array([0.0, math.log(3.0), -1.0])
    dt = np.array([0.5, -0.25, 2.0])
    a = np.stack([-dt, -dt + 40.0, -dt - 40.0])  # softplus arguments 0, 40, -40
    g, beta = oracle.gate_params(a, np.zeros((3, 3)), A_log, dt)
    np.testing.assert_allclose(g[0], -np.exp(A_log) * math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(g[1], -np.exp(A_log) * 40.0, rtol=1e-15)  # ln(1 + e^40) = 40 + 4e-18
    np.testing.assert_allclose(g[2], -np.exp(A_log) * math.exp(-40.0), rtol=1e-15)
    assert np.all(beta == 0.5)
    rng = np.random.default_rng(5)
    b = rng.standard_normal((50, 3)) * 5
    a = rng.standard_normal((50, 3)) * 5
    g, beta = oracle.gate_params(a, b, A_log, dt)
    _, beta_neg = oracle.gate_params(a, -b, A_log, dt)
    np.testing.assert_allclose(beta + beta_neg, 1.0, rtol=1e-15)
    assert np.all(g < 0) and np.all(np.exp(g) > 0) and np.all(np.exp(g) < 1)
    # beta is the logistic function: logit(beta) = b
    np.testing.assert_allclose(np.log(beta / (1 - beta)), b, rtol=1e-9, atol=1e-12)


def test_tree_roots_equal_the_plain_batch():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((30, 4))
    w = rng.standard_normal((4, 4))
    s0 = rng.standard_normal((2, 3, 4))
    cu = [0, 10, 30]
    u, f = oracle.causal_conv_silu(x, w, cu, None, s0, [1, 0])
    ut, ft = oracle.causal_conv_silu_tree(x, w, cu, [-1, -1], None, s0, [1, 0])
    np.testing.assert_array_equal(u, ut)
    np.testing.assert_array_equal(f, ft)


def test_tree_chain_equals_one_sequence():
    # a chain of pieces (one of them empty, one shorter than the window) is one sequence
    rng = np.random.default_rng(8)
    lens = [7, 1, 0, 2, 12]
    x = rng.standard_normal((sum(lens), 5))
    w = rng.standard_normal((5, 4))
    b = rng.standard_normal(5)
    s0 = rng.standard_normal((1, 3, 5))
    cu = np.concatenate([[0], np.cumsum(lens)])
    u1, f1 = oracle.causal_conv_silu(x, w, [0, sum(lens)], b, s0, [0])
    ut, ft = oracle.causal_conv_silu_tree(x, w, cu, [-1, 0, 1, 2, 3], b, s0, [0, -1, -1, -1, -1])
    np.testing.assert_allclose(ut, u1, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(ft[-1], f1[0])
    # every node's window is the last three rows of the path up to it
    np.testing.assert_array_equal(ft[0], x[4:7])
    np.testing.assert_array_equal(ft[1], x[5:8])
    np.testing.assert_array_equal(ft[2], ft[1])  # an empty node keeps its parent's window


def test_tree_siblings_share_the_parent_window():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((9, 3))
    w = rng.standard_normal((3, 4))
    cu = [0, 5, 7, 9]  # a prefix of 5 rows and two 2-row children
    u, _ = oracle.causal_conv_silu_tree(x, w, cu, [-1, 0, 0])
    for b in (5, 7):  # each child run alone after the prefix rows
        ua, _ = oracle.causal_conv_silu(np.concatenate([x[:5], x[b:b + 2]]), w, [0, 7])
        np.testing.assert_allclose(u[b:b + 2], ua[5:], rtol=1e-14, atol=1e-15)


def test_recipe_gate_distribution():
    # the synthetic gate parameters (Mamba2's initial ranges, N(0, 1) projections):
    # mostly slow decay (median alpha about 0.94), a tenth below about 0.6 and a
    # tail of strong forgetting, as the input recipe states
    import workloads
    inp = workloads.prep_inputs([4000], h_qk=1, d_k=8, h_v=32, d_v=8, seed=3)
    g, beta = oracle.gate_params(inp["a"].float().numpy(), inp["b"].float().numpy(), inp["A_log"].numpy(),
                                 inp["dt_bias"].numpy())
    alpha = np.exp(g)
    assert 0.0 < alpha.min() and alpha.max() < 1.0
    assert 0.9 < np.median(alpha) < 0.97
    assert 0.5 < np.quantile(alpha, 0.1) < 0.7
    assert alpha.min() < 1e-6
    assert beta.min() > 0.0 and beta.max() < 1.0
