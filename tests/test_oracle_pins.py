"""Pins for the fp64 oracle: checks against facts fixed by the mathematics and
by hand-worked examples, never against the oracle's own formulas retyped.

Each test names the kind of mistake it is there to catch.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.chunked import scan_head_chunked
from gated_deltanet_linear_pre_gb300 import inputs as gin

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))


# ---- conv -------------------------------------------------------------------
def test_conv_hand_worked():
    ex = GOLD["conv"]
    y, h = oracle.conv(ex["x"], ex["w"], ex["hist"])
    np.testing.assert_array_equal(y, ex["y"])
    np.testing.assert_array_equal(h, ex["hist_out"])


def test_conv_impulse_reproduces_reversed_taps():
    # tap-order mistake: a unit impulse at t=0 must read out w[c][3], w[c][2], ...
    rng = np.random.default_rng(0)
    C, T = 8, 6
    w = rng.standard_normal((C, 4))
    x = np.zeros((T, C))
    x[0] = 1.0
    y, _ = oracle.conv(x, w, np.zeros((C, 3)))
    for t in range(4):
        np.testing.assert_array_equal(y[t], w[:, 3 - t])
    np.testing.assert_array_equal(y[4:], 0.0)


def test_conv_history_impulses():
    # history-index mistake: an impulse in hist slot i (i=0 oldest) reaches y[t]
    # through tap m = i - t for t <= i
    rng = np.random.default_rng(1)
    C = 5
    w = rng.standard_normal((C, 4))
    for i in range(3):
        hist = np.zeros((C, 3))
        hist[:, i] = 1.0
        y, _ = oracle.conv(np.zeros((4, C)), w, hist)
        for t in range(4):
            m = i - t
            np.testing.assert_array_equal(y[t], w[:, m] if m >= 0 else 0.0)


@pytest.mark.parametrize("T", [0, 1, 2, 3, 5])
def test_conv_history_out_short_sequences(T):
    # T < 3 must shift the old history: hist_out is the last 3 of (hist ++ x)
    rng = np.random.default_rng(2)
    C = 7
    hist = rng.standard_normal((C, 3))
    x = rng.standard_normal((T, C))
    _, h = oracle.conv(x, rng.standard_normal((C, 4)), hist)
    seq = np.concatenate([hist.T, x], axis=0)  # [3+T, C], oldest first
    np.testing.assert_array_equal(h, seq[-3:].T)


def test_conv_brute_force_small():
    # against the definition as a literal convolution of the history-padded
    # sequence (numpy.convolve with the taps reversed), on tiny random inputs
    rng = np.random.default_rng(3)
    C = 8
    for T in (1, 2, 3, 5):
        x = rng.standard_normal((T, C))
        w = rng.standard_normal((C, 4))
        hist = rng.standard_normal((C, 3))
        y, _ = oracle.conv(x, w, hist)
        for c in range(C):
            padded = np.concatenate([hist[c], x[:, c]])
            full = np.convolve(padded, w[c, ::-1], mode="valid")
            np.testing.assert_allclose(y[:, c], full, rtol=0, atol=1e-14)


# ---- activations --------------------------------------------------------------
def test_activation_special_values():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.silu_scalar(0.0) == 0.0
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16)
    assert oracle.softplus(800.0) == 800.0            # no overflow, asymptote x
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-15)
    assert oracle.sigmoid(-800.0) == 0.0 and oracle.sigmoid(800.0) == 1.0
    for x in (-7.5, -1.0, 0.3, 2.0, 12.0):
        assert oracle.sigmoid(x) == pytest.approx(1.0 / (1.0 + math.exp(-x)), rel=1e-15)
        assert oracle.silu_scalar(x) == pytest.approx(x / (1.0 + math.exp(-x)), rel=1e-15)
        assert oracle.softplus(x) == pytest.approx(math.log1p(math.exp(x)), rel=1e-15)
    # SiLU is x * sigmoid(x), not sigmoid: odd-part identity silu(x) - silu(-x) = x
    for x in (0.7, 3.0):
        assert oracle.silu_scalar(x) - oracle.silu_scalar(-x) == pytest.approx(x, rel=1e-15)


def test_silu_array_matches_scalar():
    x = np.linspace(-10, 10, 41)
    np.testing.assert_array_equal(oracle.silu(x), [oracle.silu_scalar(v) for v in x])


# ---- L2 norm ----------------------------------------------------------------------
def test_l2norm_hand_worked():
    ex = GOLD["l2norm"]
    np.testing.assert_allclose(oracle.l2norm(np.array([ex["x"]]), ex["eps"])[0], ex["y"], rtol=1e-15)


def test_l2norm_unit_norm_and_eps_placement():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((10, 128))
    y = oracle.l2norm(x, 1e-6)
    ss = (x * x).sum(-1)
    # |y|^2 = |x|^2 / (|x|^2 + eps): unit up to the eps effect, direction kept
    np.testing.assert_allclose((y * y).sum(-1), ss / (ss + 1e-6), rtol=1e-14)
    np.testing.assert_allclose(y / np.linalg.norm(y, axis=-1, keepdims=True),
                               x / np.linalg.norm(x, axis=-1, keepdims=True), rtol=1e-14)
    # tiny vectors: eps dominates, y ~ x / sqrt(eps)
    xs = x * 1e-6
    ys = oracle.l2norm(xs, 1e-6)
    np.testing.assert_allclose(ys, xs / np.sqrt((xs * xs).sum(-1, keepdims=True) + 1e-6), rtol=1e-14)
    assert np.abs(ys).max() < 1e-2


# ---- gates ------------------------------------------------------------------------
def test_gates_hand_worked():
    ex = GOLD["gates"]
    g, lam, beta = oracle.gates([[ex["a"]]], [[ex["b"]]], [ex["A_log"]], [ex["dt_bias"]])
    assert lam[0, 0] == pytest.approx(ex["lam"], rel=1e-15)
    assert g[0, 0] == pytest.approx(ex["g"], rel=1e-15)
    assert beta[0, 0] == ex["beta"]


def test_gates_limits():
    # A_log -> -inf or a+dt -> -inf give g -> 1 (no forgetting); large rates give g -> 0
    g, lam, beta = oracle.gates([[0.0, -60.0, 3.0]], [[40.0, -40.0, 0.0]],
                                [-800.0, 0.0, 10.0], [0.0, 0.0, 0.0])
    assert g[0, 0] == 1.0 and lam[0, 0] <= 0.0
    assert g[0, 1] == pytest.approx(1.0, abs=1e-25)
    assert g[0, 2] == 0.0 and lam[0, 2] < -6e4
    assert beta[0, 0] == 1.0 and beta[0, 1] == pytest.approx(math.exp(-40.0), rel=1e-14)
    assert np.all(g <= 1.0) and np.all(lam <= 0.0)


# ---- scan -------------------------------------------------------------------------
def _rand_scan(rng, T, hk, hv, dk, dv, unit_keys=True, S0_std=0.5):
    q = rng.standard_normal((T, hk, dk))
    k = rng.standard_normal((T, hk, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, dv))
    g = rng.uniform(0.5, 1.0, (T, hv))
    beta = rng.uniform(0.0, 1.0, (T, hv))
    S0 = S0_std * rng.standard_normal((hv, dk, dv))
    return q, k, v, g, beta, S0


def test_scan_hand_worked():
    ex = GOLD["scan"]
    dk = ex["dk"]
    q = np.array(ex["q_over_sqrt_dk"])[:, None, :] * math.sqrt(dk)
    k = np.array(ex["k"])[:, None, :]
    v = np.array(ex["v"])[:, None, :]
    g = np.array(ex["g"])[:, None]
    beta = np.array(ex["beta"])[:, None]
    o, S = oracle.scan(q, k, v, g, beta, np.array(ex["S0"])[None])
    np.testing.assert_allclose(o[:, 0], ex["o"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(S[0], ex["S_out"], rtol=1e-14, atol=1e-14)


def test_scan_g0_resets_state():
    # g = 0 forgets everything: S_t = beta k v^T, o = beta (k . q / sqrt(dk)) v
    rng = np.random.default_rng(5)
    T, hk, hv, dk, dv = 6, 1, 1, 16, 24
    q, k, v, g, beta, S0 = _rand_scan(rng, T, hk, hv, dk, dv)
    g[:] = 0.0
    o, S = oracle.scan(q, k, v, g, beta, S0)
    for t in range(T):
        coef = beta[t, 0] * (k[t, 0] @ q[t, 0]) / math.sqrt(dk)
        np.testing.assert_allclose(o[t, 0], coef * v[t, 0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S[0], beta[-1, 0] * np.outer(k[-1, 0], v[-1, 0]), rtol=1e-13, atol=1e-15)


def test_scan_beta0_is_pure_decay():
    rng = np.random.default_rng(6)
    T, hk, hv, dk, dv = 9, 1, 2, 12, 20
    q, k, v, g, beta, S0 = _rand_scan(rng, T, hk, hv, dk, dv)
    beta[:] = 0.0
    o, S = oracle.scan(q, k, v, g, beta, S0)
    for h in range(hv):
        decay = np.cumprod(g[:, h])
        for t in range(T):
            St = decay[t] * S0[h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, 0] / math.sqrt(dk), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[h], decay[-1] * S0[h], rtol=1e-13)


def test_scan_orthonormal_keys_exact_retrieval():
    # g = 1, beta = 1, S0 = 0 and orthonormal keys: every stored value is
    # retrieved exactly, S^T k_i = v_i for all i
    rng = np.random.default_rng(7)
    dk, dv, T = 32, 20, 32
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T[:T][:, None, :]
    v = rng.standard_normal((T, 1, dv))
    q = rng.standard_normal((T, 1, dk))
    o, S = oracle.scan(q, k, v, np.ones((T, 1)), np.ones((T, 1)), np.zeros((1, dk, dv)))
    for i in range(T):
        np.testing.assert_allclose(S[0].T @ k[i, 0], v[i, 0], rtol=0, atol=1e-13)


def test_scan_delta_rule_writes_value_exactly():
    # beta = 1 and |k| = 1: right after step t, S_t^T k_t = v_t for any prior S and g
    rng = np.random.default_rng(8)
    dk, dv = 10, 14
    for T in (1, 2, 5):
        q, k, v, g, beta, S0 = _rand_scan(rng, T, 1, 1, dk, dv)
        beta[:] = 1.0
        _, S = oracle.scan(q, k, v, g, beta, S0)
        np.testing.assert_allclose(S[0].T @ k[-1, 0], v[-1, 0], rtol=0, atol=1e-13)


def test_scan_matches_householder_form():
    # independent formulation: S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    rng = np.random.default_rng(9)
    T, hk, hv, dk, dv = 7, 2, 6, 8, 5
    q, k, v, g, beta, S0 = _rand_scan(rng, T, hk, hv, dk, dv, unit_keys=False)
    o, S = oracle.scan(q, k, v, g, beta, S0)
    for h in range(hv):
        j = h // (hv // hk)            # value head h reads key head h // 3 here
        Sh = S0[h].copy()
        for t in range(T):
            kt = k[t, j]
            Sh = g[t, h] * (np.eye(dk) - beta[t, h] * np.outer(kt, kt)) @ Sh + beta[t, h] * np.outer(kt, v[t, h])
            np.testing.assert_allclose(o[t, h], Sh.T @ q[t, j] / math.sqrt(dk), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S[h], Sh, rtol=1e-12, atol=1e-13)


def test_scan_linear_in_values_from_zero_state():
    rng = np.random.default_rng(10)
    q, k, v, g, beta, _ = _rand_scan(rng, 11, 1, 2, 8, 8)
    S0 = np.zeros((2, 8, 8))
    o1, S1 = oracle.scan(q, k, v, g, beta, S0)
    o3, S3 = oracle.scan(q, k, -3.0 * v, g, beta, S0)
    np.testing.assert_allclose(o3, -3.0 * o1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S3, -3.0 * S1, rtol=1e-13, atol=1e-15)


def test_scan_head_mapping_repeat_interleave():
    # value head h reads key head h // (hv/hk): perturbing key head 1 changes
    # value heads 3, 4, 5 and nothing else
    rng = np.random.default_rng(11)
    T, hk, hv, dk, dv = 5, 4, 12, 8, 8
    q, k, v, g, beta, S0 = _rand_scan(rng, T, hk, hv, dk, dv)
    o1, _ = oracle.scan(q, k, v, g, beta, S0)
    k2 = k.copy()
    k2[:, 1] = rng.standard_normal((T, dk))
    o2, _ = oracle.scan(q, k2, v, g, beta, S0)
    changed = [h for h in range(hv) if not np.array_equal(o1[:, h], o2[:, h])]
    assert changed == [3, 4, 5]


def test_scan_head_subset_matches_full():
    rng = np.random.default_rng(12)
    args = _rand_scan(rng, 9, 2, 6, 8, 8)
    o, S = oracle.scan(*args)
    os_, Ss = oracle.scan(*args, heads=[1, 4])
    np.testing.assert_array_equal(os_[:, [1, 4]], o[:, [1, 4]])
    np.testing.assert_array_equal(Ss[[1, 4]], S[[1, 4]])
    assert np.isnan(os_[:, 0]).all()


@pytest.mark.parametrize("T,chunk", [(37, 64), (37, 8), (130, 64), (200, 16), (64, 64), (1, 64)])
def test_chunked_equals_sequential(T, chunk):
    rng = np.random.default_rng(13 + T)
    dk, dv = 32, 24
    q, k, v, g, beta, S0 = _rand_scan(rng, T, 1, 1, dk, dv)
    g = rng.uniform(0.05, 1.0, (T, 1))
    o, S = oracle.scan(q, k, v, g, beta, S0)
    oc, Sc = scan_head_chunked(q[:, 0], k[:, 0], v[:, 0], np.log(g[:, 0]), beta[:, 0], S0[0], chunk)
    np.testing.assert_allclose(oc, o[:, 0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sc, S[0], rtol=1e-11, atol=1e-12)


def test_chunked_equals_sequential_production_decays():
    # the gates of the production layer: decays down to ~1e-35 per token
    inp = gin.make_layer(21, [150], hist_nonzero=True, S0_std=0.02, dims=(1, 3, 128, 128))
    ref = oracle.layer(inp, hk=1, hv=3, dk=128, dv=128)
    for h in range(3):
        oc, Sc = scan_head_chunked(ref["q"][:, 0], ref["k"][:, 0], ref["v"][:, h], ref["lam"][:, h],
                                   ref["beta"][:, h], inp.S0[0, h])
        np.testing.assert_allclose(oc, ref["o"][:, h], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(Sc, ref["S_out"][0, h], rtol=1e-10, atol=1e-12)


# ---- post -------------------------------------------------------------------------
def test_post_hand_worked():
    ex = GOLD["post"]
    y = oracle.post([ex["o"]], [ex["z"]], ex["gamma"], ex["eps"])
    np.testing.assert_array_equal(y[0], ex["y"])
    z = ex["z_is_large"]
    y2 = oracle.post([ex["o2"]], [[z] * 4], ex["gamma2"], ex["eps"])
    np.testing.assert_allclose(y2[0] / z, ex["y2_over_z"], rtol=1e-15)
    # eps comparable to mean(o^2): it sits inside the square root, added to the mean
    z3 = ex["z3_is_large"]
    y3 = oracle.post([ex["o3"]], [[z3] * 4], ex["gamma3"], ex["eps3"])
    np.testing.assert_allclose(y3[0] / z3, ex["y3_over_z"], rtol=1e-12)


def test_post_scale_invariance_and_rms():
    rng = np.random.default_rng(14)
    o = rng.standard_normal((6, 128))
    z = rng.standard_normal((6, 128))
    gamma = 1 + 0.1 * rng.standard_normal(128)
    y = oracle.post(o, z, gamma, 0.0)
    np.testing.assert_allclose(oracle.post(7.5 * o, z, gamma, 0.0), y, rtol=1e-14)
    # with gamma = 1 and z large, y / z has unit root-mean-square per row
    y1 = oracle.post(o, np.full_like(o, 40.0), np.ones(128), 0.0) / 40.0
    np.testing.assert_allclose(np.sqrt((y1 ** 2).mean(-1)), 1.0, rtol=1e-14)


# ---- whole layer -----------------------------------------------------------------
def test_layer_channel_split_and_unit_norms():
    inp = gin.make_layer(21, [20], hist_nonzero=True, S0_std=0.02, dims=(2, 6, 16, 8))
    ref = oracle.layer(inp, hk=2, hv=6, dk=16, dv=8)
    s = oracle.silu(oracle.conv(inp.qkv, inp.conv_w, inp.hist[0])[0])
    # q | k | v channel order
    np.testing.assert_array_equal(ref["v"].reshape(20, -1), s[:, 64:])
    qn = ref["q"]
    ss = (s[:, :32].reshape(20, 2, 16) ** 2).sum(-1)
    np.testing.assert_allclose((qn ** 2).sum(-1), ss / (ss + 1e-6), rtol=1e-13)


def test_layer_resume_equals_single_call():
    # run(T1) then run(T2) from the returned history and state == run(T1 + T2)
    dims = (2, 6, 16, 8)
    full = gin.make_layer(33, [29], hist_nonzero=True, S0_std=0.02, dims=dims)
    ref = oracle.layer(full, hk=2, hv=6, dk=16, dv=8)
    T1 = 11

    def part(sl, hist, S0):
        return gin.LayerInputs(qkv=full.qkv[sl], conv_w=full.conv_w, hist=hist, a=full.a[sl],
                               b=full.b[sl], A_log=full.A_log, dt_bias=full.dt_bias, z=full.z[sl],
                               gamma=full.gamma, S0=S0,
                               cu_seqlens=np.array([0, sl.stop - sl.start], np.int32), dims=dims)

    r1 = oracle.layer(part(slice(0, T1), full.hist, full.S0), hk=2, hv=6, dk=16, dv=8)
    r2 = oracle.layer(part(slice(T1, 29), r1["hist_out"], r1["S_out"]), hk=2, hv=6, dk=16, dv=8)
    np.testing.assert_array_equal(r2["hist_out"], ref["hist_out"])
    np.testing.assert_allclose(r2["S_out"], ref["S_out"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.concatenate([r1["y"], r2["y"]]), ref["y"], rtol=1e-12, atol=1e-13)


def test_layer_varlen_sequences_are_independent():
    dims = (2, 6, 16, 8)
    batch = gin.make_layer(44, [5, 1, 9], hist_nonzero=True, S0_std=0.02, dims=dims)
    ref = oracle.layer(batch, hk=2, hv=6, dk=16, dv=8)
    cu = batch.cu_seqlens
    for s in range(3):
        sl = slice(int(cu[s]), int(cu[s + 1]))
        one = gin.LayerInputs(qkv=batch.qkv[sl], conv_w=batch.conv_w, hist=batch.hist[s:s + 1],
                              a=batch.a[sl], b=batch.b[sl], A_log=batch.A_log, dt_bias=batch.dt_bias,
                              z=batch.z[sl], gamma=batch.gamma, S0=batch.S0[s:s + 1],
                              cu_seqlens=np.array([0, sl.stop - sl.start], np.int32), dims=dims)
        r = oracle.layer(one, hk=2, hv=6, dk=16, dv=8)
        np.testing.assert_array_equal(r["y"], ref["y"][sl])
        np.testing.assert_array_equal(r["S_out"][0], ref["S_out"][s])
        np.testing.assert_array_equal(r["hist_out"][0], ref["hist_out"][s])
