"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, a literal matrix-product evaluation of the recurrence on tiny
inputs, special cases that reduce to textbook linear attention, invariants
(linearity, contraction, state hand-off, varlen independence) and a second
formulation (chunked WY form).  CPU only.

A plausible slip in the oracle fails at least one of these:
  sign of the delta-rule correction / order of decay and erase -> brute force
  gate form (sigmoid argument, bound, exp(A_log))               -> prep closed forms
  l2norm epsilon placement / beta sigmoid                       -> prep closed forms
  transposed state layout (init or final)                       -> one-hot / frozen-state pins
  dropped intra-chunk or state term                             -> chunked vs token loop
  sequence boundary handling                                    -> varlen / hand-off pins
"""
import math

import numpy as np
import pytest

import oracle
from kimi_delta_attention_08_gb300 import synth

KD = 128
BF16_NEG_INF = np.uint16(0xFF80)
BF16_POS_INF = np.uint16(0x7F80)


def small(T=40, H=2, lengths=None, init="randn", lb=-5.0, seed=11, state_dtype="fp32"):
    return synth.make("pin", 1, T, H, lengths=lengths, init=init, lower_bound=lb, seed=seed,
                      state_dtype=state_dtype)


def run(w, **kw):
    T = w.tensors
    args = dict(initial_state=T["initial_state"], cu_seqlens=w.cu_seqlens)
    args.update(kw)
    return oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                      w.lower_bound, w.scale, **args)


def rel(a, b):
    d = np.abs(b).max()
    return np.abs(a - b).max() / (d if d > 0 else 1.0)


# ---------------------------------------------------------------- prep -----
def test_prep_closed_forms():
    H = 1
    z = np.zeros((4, H, KD), np.float64)
    q = z.copy()
    q[0, 0, :2] = [3.0, 4.0]                  # |q|^2 = 25
    k = z.copy()                              # row 1: zero vector -> 0
    k[0, 0, 5] = -2.0
    dt = np.zeros((H, KD))
    dt[0, 0] = 0.75
    g = z.copy()
    g[0, 0, 0] = -0.75                        # a = 0 -> sigmoid 1/2
    g[1, 0, 1] = 1e4                          # sigmoid -> 1
    g[2, 0, 2] = -1e4                         # sigmoid -> 0
    g[3, 0, 3] = 1.0                          # a = exp(A_log) * 1 = 2
    A_log = np.array([math.log(2.0)])
    beta = np.array([[0.0], [np.inf], [-np.inf], [math.log(3.0)]])
    lb = -4.0
    qn, kn, la, bs = oracle.prep(q, k, g, beta, A_log, dt, lb)
    assert qn[0, 0, 0] == 3.0 / math.sqrt(25.0 + 1e-6) and qn[0, 0, 1] == 4.0 / math.sqrt(25.0 + 1e-6)
    assert np.all(qn[1:] == 0.0) and np.all(kn[1:] == 0.0)
    assert kn[0, 0, 5] == -2.0 / math.sqrt(4.0 + 1e-6)
    assert la[0, 0, 0] == lb * 0.5
    assert abs(la[1, 0, 1] - lb) < 1e-12 and abs(la[2, 0, 2]) < 1e-12
    assert abs(la[3, 0, 3] - lb / (1.0 + math.exp(-2.0))) < 1e-15
    # channels with g = 0: a = 2 * dt_bias; channel 0 of rows 1.. has dt 0.75 -> a = 1.5
    assert abs(la[1, 0, 0] - lb / (1.0 + math.exp(-1.5))) < 1e-15
    assert bs[0, 0] == 0.5 and bs[1, 0] == 1.0 and bs[2, 0] == 0.0
    assert abs(bs[3, 0] - 0.75) < 1e-15     # sigmoid(log 3) = 3/4
    assert np.all((la <= 0) & (la >= lb))


def test_prep_bf16_decoding():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x3E00, 0x7F80], dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    assert list(vals[:4]) == [1.0, -2.0, 0.0, 0.125] and vals[4] == np.inf


# ------------------------------------------------------- brute force -------
def brute_force(w):
    """Literal S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T, o_t = scale S_t^T q,
    with full K x K matrices (independent of the oracle's rank-1 evaluation)."""
    T = w.tensors
    qn, kn, la, bs = oracle.prep(T["q"].reshape(-1, w.H, KD), T["k"].reshape(-1, w.H, KD),
                                 T["g"].reshape(-1, w.H, KD), T["beta"].reshape(-1, w.H),
                                 T["A_log"], T["dt_bias"], w.lower_bound)
    v = oracle.bf16_bits_to_f64(T["v"]).reshape(-1, w.H, KD)
    init = T["initial_state"]
    out = np.zeros_like(v)
    fin = np.zeros((w.N, w.H, KD, KD))
    I = np.eye(KD)
    for n, (b0, e0) in enumerate(w.seq_bounds()):
        for h in range(w.H):
            S = np.zeros((KD, KD)) if init is None else init[n, h].astype(np.float64).T
            for t in range(b0, e0):
                kk = kn[t, h][:, None]
                S = (I - bs[t, h] * kk @ kk.T) @ np.diag(np.exp(la[t, h])) @ S + bs[t, h] * kk @ v[t, h][None, :]
                out[t, h] = w.scale * S.T @ qn[t, h]
            fin[n, h] = S.T
    return out, fin


@pytest.mark.parametrize("lengths", [None, [3, 0, 5, 1]])
def test_brute_force_tiny(lengths):
    w = small(T=6, H=2, lengths=lengths, seed=3)
    out, fin, _ = run(w)
    bo, bfin = brute_force(w)
    assert rel(out.reshape(bo.shape), bo) < 1e-12
    assert rel(fin, bfin) < 1e-12


# ------------------------------------------------- second formulation -------
@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_chunked_form_equals_token_loop(C):
    w = small(H=2, lengths=[37, 0, 64, 100, 1, 129], seed=5)
    o1, f1, _ = run(w)
    o2, f2, _ = run(w, chunk=C)
    assert rel(o2, o1) < 1e-10 and rel(f2, f1) < 1e-10


def test_chunked_form_slow_decay():
    w = small(T=200, H=1, lb=-0.01, seed=9)
    o1, f1, _ = run(w)
    o2, f2, _ = run(w, chunk=64)
    assert rel(o2, o1) < 1e-10 and rel(f2, f1) < 1e-10


# ------------------------------------------------------ special cases -------
def test_beta_zero_zero_state():
    w = small(T=30, init="none", seed=4)
    w.tensors["beta"][:] = BF16_NEG_INF           # beta = sigmoid(-inf) = 0 exactly
    out, fin, _ = run(w)
    assert np.all(out == 0.0) and np.all(fin == 0.0)


def test_frozen_state_alpha_one_beta_zero():
    """alpha == 1 (lower_bound 0), beta == 0: S_t = S_0 and o_t = scale S_0^T qn_t.
    Also pins the [V, K] layout of the initial state."""
    w = small(T=20, lb=0.0, seed=8)
    w.tensors["beta"][:] = BF16_NEG_INF
    out, fin, _ = run(w)
    T = w.tensors
    qn = oracle.bf16_bits_to_f64(T["q"])[0]
    qn = qn / np.sqrt((qn ** 2).sum(-1, keepdims=True) + 1e-6)
    init = T["initial_state"].astype(np.float64)[0]           # [H, V, K]
    expect = w.scale * np.einsum("hvk,thk->thv", init, qn)
    assert rel(out[0], expect) < 1e-13
    assert np.array_equal(fin[0], init)


def test_linear_attention_limit_small_beta():
    """alpha == 1, S_0 = 0, beta == eps: o_t / eps -> scale sum_{j<=t} (kn_j.qn_t) v_j."""
    w = small(T=24, H=1, lb=0.0, init="none", seed=12)
    raw = np.uint16(0xC1A0)                       # bf16 -20.0
    w.tensors["beta"][:] = raw
    eps = 1.0 / (1.0 + math.exp(20.0))
    out, _, _ = run(w)
    T = w.tensors
    q = oracle.bf16_bits_to_f64(T["q"])[0, :, 0]
    k = oracle.bf16_bits_to_f64(T["k"])[0, :, 0]
    v = oracle.bf16_bits_to_f64(T["v"])[0, :, 0]
    qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6)
    kn = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    att = np.tril(qn @ kn.T)                      # [t, j], j <= t
    lin = w.scale * att @ v
    assert rel(out[0, :, 0] / eps, lin) < 1e-6


def test_exact_linear_attention_onehot_keys():
    """alpha == 1, beta == 1, distinct one-hot keys, S_0 = 0: the erase term
    vanishes and S_t = sum_{j<=t} kn_j v_j^T exactly (causal linear attention).
    Pins the [V, K] layout of the final state too."""
    T_, H = 50, 1
    w = small(T=T_, H=H, lb=0.0, init="none", seed=13)
    k = np.zeros((1, T_, H, KD), np.float32)
    cols = np.random.default_rng(0).permutation(KD)[:T_]
    for t in range(T_):
        k[0, t, 0, cols[t]] = 2.0
    w.tensors["k"] = synth.f32_to_bf16_bits(k)
    w.tensors["beta"][:] = BF16_POS_INF
    out, fin, _ = run(w)
    q = oracle.bf16_bits_to_f64(w.tensors["q"])[0, :, 0]
    v = oracle.bf16_bits_to_f64(w.tensors["v"])[0, :, 0]
    qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6)
    c = 2.0 / math.sqrt(4.0 + 1e-6)               # kn_t = c e_{cols[t]}
    lin = w.scale * np.array([c * sum(qn[t, cols[j]] * v[j] for j in range(t + 1)) for t in range(T_)])
    assert rel(out[0, :, 0], lin) < 1e-13
    S_expect = np.zeros((KD, KD))                  # [V, K]
    for j in range(T_):
        S_expect[:, cols[j]] += c * v[j]
    assert rel(fin[0, 0], S_expect) < 1e-13


# ----------------------------------------------------------- invariants -----
def test_joint_linearity_in_v_and_initial_state():
    w = small(T=33, H=2, seed=21)
    T = w.tensors
    v1 = oracle.bf16_bits_to_f64(T["v"])
    s1 = T["initial_state"].astype(np.float64)
    rng = np.random.default_rng(1)
    v2 = rng.standard_normal(v1.shape)
    s2 = rng.standard_normal(s1.shape)
    a, b = 0.7, -1.3

    def f(v, s):
        return oracle.fwd(T["q"], T["k"], v, T["g"], T["beta"], T["A_log"], T["dt_bias"],
                          w.lower_bound, w.scale, s)[:2]

    o1, F1 = f(v1, s1)
    o2, F2 = f(v2, s2)
    o3, F3 = f(a * v1 + b * v2, a * s1 + b * s2)
    assert rel(o3, a * o1 + b * o2) < 1e-12 and rel(F3, a * F1 + b * F2) < 1e-12


def test_contraction_bound_per_step():
    """||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t|| (transition norm <= 1)."""
    w = small(T=25, H=1, lb=-0.5, seed=22)
    T = w.tensors
    S = T["initial_state"].astype(np.float64)
    _, _, _, bs = oracle.prep(T["q"][0], T["k"][0], T["g"][0], T["beta"][0], T["A_log"],
                              T["dt_bias"], w.lower_bound)
    v = oracle.bf16_bits_to_f64(T["v"])[0]
    for t in range(25):
        sl = slice(t, t + 1)
        _, S2, _ = oracle.fwd(T["q"][:, sl], T["k"][:, sl], T["v"][:, sl], T["g"][:, sl],
                              T["beta"][:, sl], T["A_log"], T["dt_bias"], w.lower_bound, w.scale, S)
        assert np.linalg.norm(S2) <= np.linalg.norm(S) + bs[t, 0] * np.linalg.norm(v[t, 0]) + 1e-12
        S = S2


def test_state_handoff_equals_one_run():
    w = small(T=150, H=2, seed=23)
    T = w.tensors
    o, F, _ = run(w)
    h = 71
    a = {nm: T[nm][:, :h] for nm in ("q", "k", "v", "g", "beta")}
    b = {nm: T[nm][:, h:] for nm in ("q", "k", "v", "g", "beta")}
    oa, Fa, _ = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], T["A_log"], T["dt_bias"],
                           w.lower_bound, w.scale, T["initial_state"])
    ob, Fb, _ = oracle.fwd(b["q"], b["k"], b["v"], b["g"], b["beta"], T["A_log"], T["dt_bias"],
                           w.lower_bound, w.scale, Fa)
    assert rel(np.concatenate([oa, ob], axis=1), o) < 1e-13 and rel(Fb, F) < 1e-13


def test_varlen_equals_independent_runs():
    lengths = [13, 0, 70, 1, 44]
    w = small(H=2, lengths=lengths, seed=24)
    T = w.tensors
    o, F, _ = run(w)
    for n, (b0, e0) in enumerate(w.seq_bounds()):
        sl = slice(b0, e0)
        on, Fn, _ = oracle.fwd(T["q"][:, sl], T["k"][:, sl], T["v"][:, sl], T["g"][:, sl],
                               T["beta"][:, sl], T["A_log"], T["dt_bias"], w.lower_bound,
                               w.scale, T["initial_state"][n:n + 1])
        assert np.array_equal(on, o[:, sl]) and np.array_equal(Fn, F[n:n + 1])
    # the empty sequence keeps its initial state
    assert np.array_equal(F[1], T["initial_state"][1].astype(np.float64))


def test_affine_composition_transition_independent_of_v():
    """S_end = M S_start + B with M independent of V and S_start (pins the
    segment-scan decomposition): M e_i depends only on (q, k, g, beta)."""
    w = small(T=40, H=1, init="none", lb=-0.1, seed=25)
    T = w.tensors
    zero_v = np.zeros_like(oracle.bf16_bits_to_f64(T["v"]))
    rng = np.random.default_rng(2)
    s = rng.standard_normal((1, 1, KD, KD))

    def fin(v, s0):
        return oracle.fwd(T["q"], T["k"], v, T["g"], T["beta"], T["A_log"], T["dt_bias"],
                          w.lower_bound, w.scale, s0)[1]

    B = fin(T["v"], np.zeros_like(s))
    MS = fin(zero_v, s)
    scale = np.abs(MS).max() + np.abs(B).max()
    assert np.abs(fin(T["v"], s) - (MS + B)).max() < 1e-12 * scale
    v2 = rng.standard_normal(zero_v.shape)
    assert np.abs(fin(v2, s) - fin(v2, np.zeros_like(s)) - MS).max() < 1e-12 * scale


# ------------------------------------------- grouped value heads, fp32 gate -----
def gva(T=40, H=2, HV=6, lengths=None, seed=31, g_dtype="bf16", lb=-5.0):
    return synth.make("pin_gva", 1, T, H, lengths=lengths, init="randn", lower_bound=lb,
                      seed=seed, HV=HV, g_dtype=g_dtype)


def repeated_qk(w):
    """The plain (HK = HV) problem with q/k materialised per value head:
    value head h takes q/k head h // (HV / H)."""
    G = w.n_vheads // w.H
    T = w.tensors
    return np.repeat(T["q"], G, axis=-2), np.repeat(T["k"], G, axis=-2)


@pytest.mark.parametrize("lengths", [None, [17, 0, 5, 30]])
def test_grouped_value_heads_equal_repeated_qk(lengths):
    """HV = 3 H: the oracle's own head mapping equals the plain oracle on q/k
    repeated consecutively (h % H instead of h // G fails this), and the literal
    matrix-product recurrence on the same repeated q/k."""
    w = gva(lengths=lengths, T=40 if lengths is None else 0)
    T = w.tensors
    o, F, _ = run(w)
    q2, k2 = repeated_qk(w)
    o2, F2, _ = oracle.fwd(q2, k2, T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                           w.lower_bound, w.scale, T["initial_state"], w.cu_seqlens)
    assert np.array_equal(o, o2) and np.array_equal(F, F2)
    plain = synth.make("pin_gva_plain", 1, w.T, w.n_vheads, lengths=w.lengths, init="randn",
                       seed=w.seed)
    plain.tensors.update({nm: T[nm] for nm in ("v", "g", "beta", "A_log", "dt_bias",
                                                "initial_state")})
    plain.tensors["q"], plain.tensors["k"] = q2, k2
    bo, bfin = brute_force(plain)
    assert rel(o.reshape(bo.shape), bo) < 1e-12 and rel(F, bfin) < 1e-12


def test_grouped_value_heads_chunked_form():
    w = gva(lengths=[37, 64, 1, 90], T=0, seed=32)
    o1, f1, _ = run(w)
    o2, f2, _ = run(w, chunk=16)
    assert rel(o2, o1) < 1e-10 and rel(f2, f1) < 1e-10


def test_fp32_gate_bf16_values_match_bf16_input():
    """An fp32 gate whose values are exactly bf16 gives the bf16-input result bit for bit."""
    w = small(T=30, H=2, seed=33)
    T = w.tensors
    o1, f1, _ = run(w)
    g32 = synth.bf16_bits_to_f32(T["g"])
    o2, f2, _ = oracle.fwd(T["q"], T["k"], T["v"], g32, T["beta"], T["A_log"], T["dt_bias"],
                           w.lower_bound, w.scale, T["initial_state"])
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_fp32_gate_single_token_closed_form():
    """T = 1 with an fp32 gate off the bf16 grid: o = scale (Diag(a) S0 +
    beta kn (v - kn^T Diag(a) S0))^T qn, a = exp(lb sigmoid(exp(A_log)(g + dt_bias)))
    with g read to all 24 bits."""
    w = gva(T=1, H=1, HV=2, seed=34, g_dtype="fp32", lb=-2.0)
    T = w.tensors
    assert not np.array_equal(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(T["g"])), T["g"])
    out, fin, _ = run(w)
    q = oracle.bf16_bits_to_f64(T["q"])[0, 0, 0]
    k = oracle.bf16_bits_to_f64(T["k"])[0, 0, 0]
    qn = q / math.sqrt((q ** 2).sum() + 1e-6)
    kn = k / math.sqrt((k ** 2).sum() + 1e-6)
    for h in range(2):
        g = T["g"][0, 0, h].astype(np.float64)
        a = np.exp(w.lower_bound / (1.0 + np.exp(-math.exp(float(T["A_log"][h])) *
                                                 (g + T["dt_bias"][h].astype(np.float64)))))
        b = 1.0 / (1.0 + math.exp(-float(oracle.bf16_bits_to_f64(T["beta"])[0, 0, h])))
        S0 = T["initial_state"][0, h].astype(np.float64).T          # [K, V]
        v = oracle.bf16_bits_to_f64(T["v"])[0, 0, h]
        aS = a[:, None] * S0
        S1 = aS + b * np.outer(kn, v - kn @ aS)
        assert rel(out[0, 0, h], w.scale * S1.T @ qn) < 1e-13
        assert rel(fin[0, h], S1.T) < 1e-13
