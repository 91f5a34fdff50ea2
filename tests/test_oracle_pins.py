"""Pins for the fp64 oracle: closed forms, exact arithmetic, invariants and
brute force, each written independently of the oracle's own code.

The pages print no numeric example of the gated delta rule, so page-value
parity is unavailable; these pins stand in for it. Every plausible slip in the
oracle (a dropped or reordered decay, a sign, S vs S^T, the q/k head map, the
L2 norm, chunk boundaries, the state gather) makes at least one of them fail.
"""
import numpy as np
import pytest
import sympy as sp

import oracle

RNG = np.random.default_rng(1234)


def f32(x):
    return np.asarray(x, dtype=np.float32)


def rand_case(lengths, h_qk=1, h_v=1, d_k=8, d_v=8, alpha=(0.5, 1.0), beta=(0.0, 2.0),
              s0_sd=None, n_slots=None, unit=True, seed=0):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q = rng.standard_normal((T, h_qk, d_k)).astype(np.float32)
    k = rng.standard_normal((T, h_qk, d_k)).astype(np.float32)
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, h_v, d_v)).astype(np.float32)
    g = np.log(rng.uniform(alpha[0], alpha[1], (T, h_v))).astype(np.float32)
    b = rng.uniform(beta[0], beta[1], (T, h_v)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    s0 = None
    if s0_sd is not None:
        ns = len(lengths) if n_slots is None else n_slots
        s0 = (rng.standard_normal((ns, h_v, d_k, d_v)) * s0_sd).astype(np.float32)
    return dict(q=q, k=k, v=v, g=g, beta=b, cu_seqlens=cu, initial_state=s0)


def run(case, kind="recurrent", **kw):
    c = dict(case)
    fn = oracle.recurrent if kind == "recurrent" else oracle.chunked
    return fn(c.pop("q"), c.pop("k"), c.pop("v"), c.pop("g"), c.pop("beta"), c.pop("cu_seqlens"),
              c.pop("initial_state", None), c.pop("state_index", None), **kw)


def unit(x):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x) + oracle.EPS)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130])
@pytest.mark.parametrize("C,d", [(4, 4), (16, 8), (64, 64), (16, 64), (64, 8)])
def test_chunked_form_equals_recurrence(T, C, d):
    """The chunked WY/UT form equals the token recurrence (any chunk size)."""
    case = rand_case([T], d_k=d, d_v=d, s0_sd=0.5, seed=T * 7 + C)
    o1, s1 = run(case)
    o2, s2 = run(case, "chunked", chunk=C)
    assert np.abs(o1 - o2).max() <= 1e-10 * max(1.0, np.abs(o1).max())
    assert np.linalg.norm(s1 - s2) <= 1e-10 * np.linalg.norm(s1)


def test_chunked_equals_recurrence_varlen_gqa_rectangular():
    """Packed sequences, grouped heads and d_k != d_v through both forms."""
    case = rand_case([5, 0, 70, 33, 1], h_qk=2, h_v=6, d_k=12, d_v=5, s0_sd=1.0, seed=9)
    o1, s1 = run(case)
    for C in (3, 16, 64):
        o2, s2 = run(case, "chunked", chunk=C)
        assert np.abs(o1 - o2).max() <= 1e-10 * np.abs(o1).max()
        assert np.abs(s1 - s2).max() <= 1e-10 * np.abs(s1).max()


# ---------------------------------------------------------------- exact arithmetic
def test_exact_rational_recurrence_matches_the_defining_formula():
    """Three tokens, d_k=3, d_v=2, evaluated exactly with sympy from
    S_t = e^{g_t} (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T, o_t = scale S_t^T q_t.
    The keys are given un-normalised; the L2 normalisation is applied exactly
    (with eps) in sympy as well."""
    rng = np.random.default_rng(5)
    T, dk, dv = 3, 3, 2
    q = f32(rng.standard_normal((T, 1, dk)))
    k = f32(rng.standard_normal((T, 1, dk)))
    v = f32(rng.standard_normal((T, 1, dv)))
    g = f32(np.log(rng.uniform(0.3, 1.0, (T, 1))))
    b = f32(rng.uniform(0.1, 1.9, (T, 1)))
    s0 = f32(rng.standard_normal((1, 1, dk, dv)))
    scale = 0.37
    o, s = oracle.recurrent(q, k, v, g, b, np.array([0, T]), s0, None, scale=scale)

    R = lambda x: sp.Rational(float(x))  # exact value of the float32
    eps = sp.Rational(1, 10 ** 6)
    S = sp.Matrix(dk, dv, lambda i, j: R(s0[0, 0, i, j]))
    for t in range(T):
        kt = sp.Matrix([R(x) for x in k[t, 0]])
        qt = sp.Matrix([R(x) for x in q[t, 0]])
        kt = kt / sp.sqrt((kt.T * kt)[0] + eps)
        qt = qt / sp.sqrt((qt.T * qt)[0] + eps)
        vt = sp.Matrix([R(x) for x in v[t, 0]])
        a = sp.exp(R(g[t, 0]))
        bt = R(b[t, 0])
        S = a * (sp.eye(dk) - bt * kt * kt.T) * S + bt * kt * vt.T
        ot = R(scale) * S.T * qt
        for j in range(dv):
            assert abs(float(sp.N(ot[j], 40)) - o[t, 0, j]) <= 1e-13
    for i in range(dk):
        for j in range(dv):
            assert abs(float(sp.N(S[i, j], 40)) - s[0, 0, i, j]) <= 1e-13


# ---------------------------------------------------------------- closed forms
def test_one_token_closed_form_rectangular_state():
    """S_1 = e^g (I - b k k^T) S_0 + b k v^T with a non-square, non-symmetric S_0."""
    case = rand_case([1], d_k=6, d_v=4, s0_sd=1.0, unit=False, seed=3)
    o, s = run(case)
    kk = unit(case["k"][0, 0])
    qq = unit(case["q"][0, 0])
    a = np.exp(np.float64(case["g"][0, 0]))
    b = np.float64(case["beta"][0, 0])
    S0 = case["initial_state"][0, 0].astype(np.float64)
    S1 = a * (np.eye(6) - b * np.outer(kk, kk)) @ S0 + b * np.outer(kk, case["v"][0, 0])
    np.testing.assert_allclose(s[0, 0], S1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0, 0], 6 ** -0.5 * S1.T @ qq, rtol=0, atol=1e-14)


def test_beta_zero_is_pure_decay():
    """b = 0 writes nothing: S_t = e^{G_t} S_0 and o_t = scale e^{G_t} S_0^T q_t."""
    case = rand_case([40], d_k=8, d_v=5, s0_sd=1.0, seed=4)
    case["beta"][:] = 0.0
    o, s = run(case)
    G = np.cumsum(case["g"][:, 0].astype(np.float64))
    S0 = case["initial_state"][0, 0].astype(np.float64)
    for t in range(40):
        ref = 8 ** -0.5 * np.exp(G[t]) * S0.T @ unit(case["q"][t, 0])
        np.testing.assert_allclose(o[t, 0], ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s[0, 0], np.exp(G[-1]) * S0, rtol=1e-12, atol=1e-15)


def causal_linear_attention(Q, K, V, scale, G=None):
    """Dense (gated) causal linear attention: o_t = scale sum_{j<=t} w_tj (q_t.k_j) v_j,
    w_tj = e^{G_t - G_j} (1 when G is None). Written directly, no recurrence."""
    P = Q @ K.T
    if G is not None:
        P = P * np.exp(G[:, None] - G[None, :])
    return scale * np.tril(P) @ V


@pytest.mark.parametrize("gated", [False, True])
def test_orthonormal_keys_reduce_to_causal_linear_attention(gated):
    """Mutually orthogonal unit keys, b = 1, S_0 = 0: the delta correction sees
    nothing of earlier keys, and the rule is (gated) causal linear attention.
    Keys are signed standard basis vectors, exact in float32."""
    T = d = 16
    rng = np.random.default_rng(11)
    perm = rng.permutation(d)
    sign = rng.choice([-1.0, 1.0], d)
    k = np.zeros((T, 1, d), np.float32)
    k[np.arange(T), 0, perm] = sign
    q = f32(rng.standard_normal((T, 1, d)))
    v = f32(rng.standard_normal((T, 1, 7)))
    g = np.zeros((T, 1), np.float32) if not gated else f32(np.log(rng.uniform(0.5, 1, (T, 1))))
    b = np.ones((T, 1), np.float32)
    o, s = oracle.recurrent(q, k, v, g, b, np.array([0, T]), l2norm=False)
    G = np.cumsum(g[:, 0].astype(np.float64)) if gated else None
    ref = causal_linear_attention(q[:, 0].astype(np.float64), k[:, 0].astype(np.float64),
                                  v[:, 0].astype(np.float64), d ** -0.5, G)
    np.testing.assert_allclose(o[:, 0], ref, rtol=1e-12, atol=1e-13)


def test_small_beta_limit_is_linear_attention():
    """With g = 0 and S_0 = 0, o / b -> causal linear attention as b -> 0, with
    an error of order b: shrinking b tenfold shrinks the error about tenfold."""
    case = rand_case([24], d_k=8, d_v=4, seed=12)
    case["g"][:] = 0.0
    qn = np.stack([unit(x) for x in case["q"][:, 0]])
    kn = np.stack([unit(x) for x in case["k"][:, 0]])
    lin = causal_linear_attention(qn, kn, case["v"][:, 0].astype(np.float64), 8 ** -0.5)
    errs = []
    for b in (1e-3, 1e-4):
        case["beta"][:] = np.float32(b)
        o, _ = run(case)
        errs.append(np.abs(o[:, 0] / np.float64(np.float32(b)) - lin).max())
    ratio = errs[0] / errs[1]
    assert 8.0 < ratio < 12.5, ratio


def test_beta_one_stores_v_exactly():
    """b_t = 1 and a unit key: S_t^T k_t = v_t whatever e^{g_t} and S_{t-1}, so
    with q_t = k_t the output is scale * v_t at every token."""
    case = rand_case([50], d_k=8, d_v=6, s0_sd=2.0, seed=13)
    case["beta"][:] = 1.0
    # exactly unit keys in float32: four entries of +-1/2 at random places
    rng = np.random.default_rng(14)
    k = np.zeros((50, 1, 8), np.float32)
    for t in range(50):
        k[t, 0, rng.choice(8, 4, replace=False)] = rng.choice([-0.5, 0.5], 4)
    case["k"] = k
    case["q"] = k.copy()
    o, _ = oracle.recurrent(case["q"], case["k"], case["v"], case["g"], case["beta"],
                            case["cu_seqlens"], case["initial_state"], l2norm=False)
    np.testing.assert_allclose(o[:, 0], 8 ** -0.5 * case["v"][:, 0].astype(np.float64),
                               rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_fork_equals_full_path():
    """prefix -> branch -> leaf through gathered states equals each root-to-leaf
    path run from scratch (outputs of the leaf rows and final states)."""
    rng = np.random.default_rng(21)
    d, hq, hv = 8, 2, 4
    P, B, L = 37, [5, 9], [3, 11, 6]
    parent = [0, 1, 1]
    full = rand_case([P + sum(B) + sum(L)], h_qk=hq, h_v=hv, d_k=d, d_v=d, seed=22)
    rows = {k_: v_ for k_, v_ in full.items() if k_ not in ("cu_seqlens", "initial_state")}
    seg = {"p": slice(0, P)}
    o = P
    for i, n in enumerate(B):
        seg[f"b{i}"] = slice(o, o + n); o += n
    for i, n in enumerate(L):
        seg[f"l{i}"] = slice(o, o + n); o += n

    def pack(parts):
        idx = np.concatenate([np.arange(s.start, s.stop) for s in parts])
        return {k_: v_[idx] for k_, v_ in rows.items()}

    def call(seqs, s0=None, sidx=None):
        data = [pack(p) for p in seqs]
        cat = {k_: np.concatenate([x[k_] for x in data]) for k_ in rows}
        lens = [sum(s.stop - s.start for s in p) for p in seqs]
        cu = np.concatenate([[0], np.cumsum(lens)])
        return oracle.recurrent(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"], cu,
                                s0, sidx)

    _, sp_ = call([[seg["p"]]])
    _, sb = call([[seg["b0"]], [seg["b1"]]], sp_.astype(np.float32), np.array([0, 0]))
    # the gathered states are rounded to float32 (that is what the library stores):
    # compare against the full path computed from the same float32 hand-offs
    ol, sl = call([[seg[f"l{i}"]] for i in range(3)], sb.astype(np.float32), np.array(parent))
    of, sf = call([[seg["p"], seg[f"b{parent[i]}"], seg[f"l{i}"]] for i in range(3)])
    # full path outputs of the leaf rows
    offs = np.cumsum([0] + [P + B[parent[i]] + L[i] for i in range(3)])
    lo = np.cumsum([0] + L)
    for i in range(3):
        a = of[offs[i] + P + B[parent[i]]: offs[i + 1]]
        b = ol[lo[i]: lo[i + 1]]
        assert np.abs(a - b).max() <= 1e-6 * np.abs(a).max()
        assert np.linalg.norm(sf[i] - sl[i]) <= 1e-6 * np.linalg.norm(sf[i])


def test_fork_exact_in_double():
    """The hand-off is exact when the prefix state is representable: a prefix
    whose final state is exactly float32 (b = 0 keeps S_0, g = 0) makes the
    fork and the full path agree to 1e-12."""
    case = rand_case([20, 15], d_k=6, d_v=6, seed=23)
    q, k, v, g, b = (case[x] for x in ("q", "k", "v", "g", "beta"))
    b[:20] = 0.0
    g[:20] = 0.0
    s0 = f32(np.random.default_rng(3).standard_normal((1, 1, 6, 6)))
    o_full, s_full = oracle.recurrent(q, k, v, g, b, np.array([0, 35]), s0, None)
    _, s_pre = oracle.recurrent(q[:20], k[:20], v[:20], g[:20], b[:20], np.array([0, 20]), s0)
    assert np.array_equal(s_pre.astype(np.float32).astype(np.float64), s_pre)
    o_tail, s_tail = oracle.recurrent(q[20:], k[20:], v[20:], g[20:], b[20:], np.array([0, 15]),
                                      s_pre.astype(np.float32), np.array([0]))
    np.testing.assert_allclose(o_tail, o_full[20:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(s_tail, s_full, rtol=0, atol=1e-12)


def test_packing_and_permutation_invariance():
    """Each sequence's results depend on its own rows only: reordering the
    packed sequences permutes the results and nothing else changes."""
    lens = [13, 0, 40, 7, 1]
    case = rand_case(lens, h_qk=1, h_v=2, d_k=8, d_v=8, s0_sd=1.0, seed=31)
    o, s = run(case)
    perm = [3, 0, 4, 2, 1]
    cu = case["cu_seqlens"]
    idx = np.concatenate([np.arange(cu[p], cu[p + 1]) for p in perm]).astype(np.int64)
    pc = {x: case[x][idx] for x in ("q", "k", "v", "g", "beta")}
    pc["cu_seqlens"] = np.concatenate([[0], np.cumsum([lens[p] for p in perm])])
    pc["initial_state"] = case["initial_state"]
    pc["state_index"] = np.array(perm)
    o2, s2 = run(pc)
    np.testing.assert_array_equal(o2, o[idx])
    np.testing.assert_array_equal(s2, s[perm])


def test_contraction_bound():
    """Unit keys, e^g <= 1 and b in [0, 2]: ||S_t||_2 <= ||S_{t-1}||_2 + b_t ||v_t||,
    checked along a long run one token at a time through the state hand-off."""
    case = rand_case([300], d_k=8, d_v=8, s0_sd=1.0, alpha=(0.9, 1.0), beta=(0, 2), seed=41)
    S = case["initial_state"]
    prev = np.linalg.norm(S[0, 0].astype(np.float64), 2)
    for t in range(300):
        sl = slice(t, t + 1)
        _, s = oracle.recurrent(case["q"][sl], case["k"][sl], case["v"][sl], case["g"][sl],
                                case["beta"][sl], np.array([0, 1]), S, None)
        cur = np.linalg.norm(s[0, 0], 2)
        bound = prev + case["beta"][t, 0] * np.linalg.norm(case["v"][t, 0].astype(np.float64))
        assert cur <= bound * (1 + 1e-6) + 1e-6
        S = s.astype(np.float32)
        prev = np.linalg.norm(S[0, 0].astype(np.float64), 2)


def test_grouped_heads_map_to_contiguous_qk_heads():
    """v head h reads q/k head h // (h_v / h_qk): the same result as a run whose
    q/k heads are explicitly repeated per v head."""
    case = rand_case([30, 17], h_qk=2, h_v=6, d_k=8, d_v=4, s0_sd=0.3, seed=51)
    o, s = run(case)
    rep = dict(case)
    rep["q"] = np.repeat(case["q"], 3, axis=1)
    rep["k"] = np.repeat(case["k"], 3, axis=1)
    o2, s2 = run(rep)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(s, s2)


def test_l2_norm_applied_with_eps():
    """Keys and queries are normalised as x / sqrt(|x|^2 + 1e-6): scaling the
    raw rows changes nothing beyond the eps term; explicit normalisation with
    the norm switched off agrees."""
    case = rand_case([25], d_k=8, d_v=8, s0_sd=0.5, unit=False, seed=61)
    o, s = run(case)
    pre = dict(case)
    pre["q"] = f32(np.stack([unit(x) for x in case["q"][:, 0]])[:, None])
    pre["k"] = f32(np.stack([unit(x) for x in case["k"][:, 0]])[:, None])
    o2, s2 = run(pre, l2norm=False)
    assert np.abs(o - o2).max() <= 1e-6
    big = dict(case)
    big["q"] = case["q"] * np.float32(4.0)
    big["k"] = case["k"] * np.float32(4.0)
    o3, s3 = run(big)
    assert np.abs(o - o3).max() <= 1e-6


def test_state_index_semantics():
    """-1 gathers a zero state; several sequences may gather one slot; a NULL
    index means slot n for sequence n; an index past the slots is rejected;
    a sequence of length 0 returns its gathered state."""
    case = rand_case([10, 0, 10, 10], d_k=4, d_v=4, s0_sd=1.0, n_slots=2, seed=71)
    case["state_index"] = np.array([1, 1, -1, 1])
    o, s = run(case)
    np.testing.assert_array_equal(s[1], case["initial_state"][1].astype(np.float64))
    zero = dict(case)
    zero["initial_state"] = None
    zero["state_index"] = None
    o0, s0 = run(zero)
    np.testing.assert_array_equal(o[10:20], o0[10:20])  # sequence 2 (zero state)
    np.testing.assert_array_equal(s[2], s0[2])
    ident = dict(case)
    ident["state_index"] = None  # sequence n reads slot n
    s1 = case["initial_state"][1]
    ident["initial_state"] = np.stack([s1, s1, np.zeros_like(s1), s1])
    oi, si = run(ident)
    np.testing.assert_array_equal(oi, o)
    np.testing.assert_array_equal(si, s)
    bad = dict(case)
    bad["state_index"] = np.array([0, 1, 2, 0])
    with pytest.raises(ValueError):
        run(bad)


def test_scale_parameter():
    case = rand_case([9], d_k=8, d_v=3, seed=81)
    o1, _ = run(case)
    o2, _ = run(case, scale=0.5)
    np.testing.assert_allclose(o2, o1 * (0.5 / 8 ** -0.5), rtol=1e-13, atol=0)
