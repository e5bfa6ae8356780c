"""Pins of the CPU oracle to facts outside itself: closed forms, invariants,
special cases and brute force on tiny inputs. None of these re-types the
oracle's formula; each is chosen so that a plausible mistake (a dropped term, a
wrong sign, a swapped index or operand) fails at least one of them."""
import math

import numpy as np
import pytest

import oracle
import synth
from synth import tiny_config

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------------------
# bf16 rounding of scalars (used by the embedding scale)
# ---------------------------------------------------------------------------
def test_round_to_bf16_closed_forms():
    # sqrt(3840) = 61.9677...; bf16 spacing in [32, 64) is 0.25, so the nearest value is 62.0
    assert oracle.round_to_bf16(math.sqrt(3840)) == 62.0
    # halfway cases go to the even mantissa
    assert oracle.round_to_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_to_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert oracle.round_to_bf16(3.0) == 3.0
    assert oracle.round_to_bf16(1.0 + 2.0 ** -9) == 1.0


def test_round_to_bf16_matches_bit_rounding():
    # two independent implementations (frexp on the oracle side, integer bit
    # arithmetic in the input generator) must agree on random float32 values
    x = RNG.standard_normal(2000).astype(np.float32) * np.float32(50.0)
    bits = synth.f32_to_bf16_bits(x)
    ref = synth.bf16_bits_to_f32(bits).astype(np.float64)
    got = np.array([oracle.round_to_bf16(float(v)) for v in x])
    np.testing.assert_array_equal(got, ref)


def test_embed_scale():
    assert oracle.embed_scale(synth.CONFIGS["gemma3-tower"]) == 62.0
    assert oracle.embed_scale(synth.CONFIGS["smollm2-135m"]) == 1.0
    assert oracle.embed_scale(tiny_config("gemma")) == 4.0  # sqrt(16) is exact in bf16


# ---------------------------------------------------------------------------
# GEMM against a pure-Python triple loop and exact integer cases
# ---------------------------------------------------------------------------
def _triple_loop(x, w):
    P, K = len(x), len(x[0])
    N = len(w)
    out = [[0.0] * N for _ in range(P)]
    for i in range(P):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(x[i][k]) * float(w[j][k])
            out[i][j] = acc
    return np.array(out)


def test_gemm_triple_loop():
    x = RNG.standard_normal((5, 7))
    w = RNG.standard_normal((3, 7))
    np.testing.assert_allclose(oracle.gemm(x, w), _triple_loop(x, w), rtol=1e-13, atol=1e-13)


def test_gemm_exact_integers_identity_onehot():
    x = RNG.integers(-8, 9, size=(6, 16)).astype(np.float64)
    w = RNG.integers(-8, 9, size=(10, 16)).astype(np.float64)
    np.testing.assert_array_equal(oracle.gemm(x, w), _triple_loop(x, w))
    np.testing.assert_array_equal(oracle.gemm(x, np.eye(16)), x)
    onehot = np.zeros((3, 16))
    onehot[0, 2] = onehot[1, 0] = onehot[2, 15] = 1.0
    np.testing.assert_array_equal(oracle.gemm(onehot, w), w[:, [2, 0, 15]].T)


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------
def test_rmsnorm_unit_rms_and_closed_form():
    x = RNG.standard_normal((4, 33)) * 3.0
    y = oracle.rmsnorm(x, np.ones(33), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    c, eps = 0.3, 1e-5
    y = oracle.rmsnorm(np.full((1, 8), c), np.ones(8), eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_scale_invariance_and_weight_columns():
    x = RNG.standard_normal((3, 20))
    w = RNG.standard_normal(20)
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, w, 0.0), oracle.rmsnorm(x, w, 0.0), rtol=1e-13)
    # the weight scales each column: normalising then multiplying column j by w_j
    base = oracle.rmsnorm(x, np.ones(20), 1e-5)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 1e-5), base * w[None, :], rtol=1e-14)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------
def test_rope_frequencies_closed_form():
    cfg = tiny_config("llama", head_dim=4, rope_theta_global=10000.0)
    f = oracle.rope_inv_freq(cfg, 0)
    np.testing.assert_allclose(f, [1.0, 0.01], rtol=1e-15)   # theta^0, theta^(-1/2)


def test_rope_position_zero_identity_and_norm():
    cfg = synth.CONFIGS["smollm2-135m"]
    f = oracle.rope_inv_freq(cfg, 0)
    x = RNG.standard_normal((1, 5, 3, 64))
    pos = np.array([[0, 1, 17, 500, 4095]])
    y = oracle.rope_apply(x, pos, f)
    np.testing.assert_array_equal(y[0, 0], x[0, 0])
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_pairing_and_angle():
    # a unit vector on element j rotates into element j + hd/2 by angle f_j at position 1
    cfg = tiny_config("llama", head_dim=8)
    f = oracle.rope_inv_freq(cfg, 0)
    for j in range(4):
        e = np.zeros((1, 1, 1, 8))
        e[..., j] = 1.0
        y = oracle.rope_apply(e, np.array([[1]]), f)[0, 0, 0]
        expect = np.zeros(8)
        expect[j] = math.cos(f[j])
        expect[j + 4] = math.sin(f[j])
        np.testing.assert_allclose(y, expect, atol=1e-15)


def test_rope_relative_position_property():
    cfg = synth.CONFIGS["llama3-8b"]
    f = oracle.rope_inv_freq(cfg, 0)
    q = RNG.standard_normal((1, 1, 1, 128))
    k = RNG.standard_normal((1, 1, 1, 128))

    def dot(m, n):
        return float(np.sum(oracle.rope_apply(q, np.array([[m]]), f) * oracle.rope_apply(k, np.array([[n]]), f)))

    base = dot(7, 3)
    for shift in (1, 100, 3000):
        assert abs(dot(7 + shift, 3 + shift) - base) < 1e-9 * (1 + abs(base))
    assert abs(dot(7, 3) - dot(3, 7)) > 1e-6  # depends on the sign of m - n


def test_llama3_scaling_bands():
    cfg = synth.CONFIGS["llama3-8b"]
    plain = cfg.with_(rope_scaling="none")
    f0 = oracle.rope_inv_freq(plain, 0)
    f = oracle.rope_inv_freq(cfg, 0)
    lam = 2 * math.pi / f0
    hi = lam < 8192 / 4.0
    lo = lam > 8192 / 1.0
    assert hi.sum() > 0 and lo.sum() > 0 and (~hi & ~lo).sum() > 0
    np.testing.assert_array_equal(f[hi], f0[hi])          # high frequencies untouched
    np.testing.assert_array_equal(f[lo], f0[lo] / 8.0)    # low frequencies divided by the factor
    mid = ~hi & ~lo
    assert np.all(f[mid] < f0[mid]) and np.all(f[mid] > f0[mid] / 8.0)
    assert np.all(np.diff(f) < 0)                         # still strictly decreasing in j


def test_llama3_scaling_band_edges_continuous():
    # the blend weight reaches 1 at wavelength C/b and 0 at C/a: evaluate the rule at
    # frequencies placed just inside each edge of the band through a one-pair head
    cfg = synth.CONFIGS["llama3-8b"]
    C, a, b, s = 8192.0, 1.0, 4.0, 8.0
    for lam, expect_ratio in ((C / b * (1 + 1e-9), 1.0), (C / a * (1 - 1e-9), 1.0 / s),
                              (C / 2.0, (1 - 1 / 3) / s + 1 / 3)):
        f_in = 2 * math.pi / lam
        # hd = 4 with theta chosen so that f_1 = theta^(-1/2) equals f_in
        theta = f_in ** -2.0
        c = cfg.with_(head_dim=4, rope_theta_global=theta)
        got = oracle.rope_inv_freq(c, 0)[1]
        assert abs(got / f_in - expect_ratio) < 1e-6, (lam, got / f_in, expect_ratio)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def _brute_attention(q, k, v, window):
    """Explicit loops and an explicit mask matrix, causal from position 0."""
    S, Hq, hd = q.shape
    Hkv = k.shape[1]
    out = np.zeros_like(q)
    for h in range(Hq):
        g = h * Hkv // Hq
        for i in range(S):
            scores, vals = [], []
            for j in range(S):
                ok = j <= i and (window == 0 or i - j < window)
                if ok:
                    scores.append(sum(q[i, h, d] * k[j, g, d] for d in range(hd)) / math.sqrt(hd))
                    vals.append(v[j, g])
            m = max(scores)
            e = [math.exp(s_ - m) for s_ in scores]
            tot = sum(e)
            out[i, h] = sum(ei / tot * vi for ei, vi in zip(e, vals))
    return out


def _attn(q, k, v, window):
    S = q.shape[0]
    pos = np.arange(S)
    return oracle.attention(q, k, v, pos, pos, window, 1.0 / math.sqrt(q.shape[-1]))


def test_attention_brute_force_gqa_and_window():
    q = RNG.standard_normal((9, 4, 8))
    k = RNG.standard_normal((9, 2, 8))
    v = RNG.standard_normal((9, 2, 8))
    glob = _attn(q, k, v, 0)
    loc = _attn(q, k, v, 4)
    np.testing.assert_allclose(glob, _brute_attention(q, k, v, 0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(loc, _brute_attention(q, k, v, 4), rtol=1e-12, atol=1e-12)
    # the window is not vacuous at S = 9 > W = 4, and vacuous for rows i < W
    assert np.max(np.abs(glob[4:] - loc[4:])) > 1e-3
    np.testing.assert_allclose(glob[:4], loc[:4], rtol=1e-14)


def test_attention_special_cases():
    q = RNG.standard_normal((1, 4, 8))
    k = RNG.standard_normal((1, 2, 8))
    v = RNG.standard_normal((1, 2, 8))
    out = _attn(q, k, v, 0)
    np.testing.assert_allclose(out[0], v[0][[0, 0, 1, 1]], rtol=1e-15)  # one key: output is its value
    # equal keys: uniform weights, output is the running mean of the values
    q = RNG.standard_normal((6, 2, 4))
    k = np.tile(RNG.standard_normal((1, 1, 4)), (6, 1, 1))
    v = RNG.standard_normal((6, 1, 4))
    out = _attn(q, k, v, 0)
    for i in range(6):
        np.testing.assert_allclose(out[i, 0], v[: i + 1, 0].mean(axis=0), rtol=1e-12)
    out_w = _attn(q, k, v, 3)
    np.testing.assert_allclose(out_w[5, 1], v[3:6, 0].mean(axis=0), rtol=1e-12)


def test_attention_causality_and_short_window():
    q = RNG.standard_normal((8, 2, 4))
    k = RNG.standard_normal((8, 1, 4))
    v = RNG.standard_normal((8, 1, 4))
    base = _attn(q, k, v, 0)
    k2, v2 = k.copy(), v.copy()
    k2[5:] += 3.0
    v2[5:] -= 2.0
    np.testing.assert_array_equal(_attn(q, k2, v2, 0)[:5], base[:5])
    np.testing.assert_array_equal(_attn(q, k, v, 8), base)  # S <= W: local == global


# ---------------------------------------------------------------------------
# Activations and softcap
# ---------------------------------------------------------------------------
def test_activations_odd_part_and_limits():
    x = np.linspace(-6, 6, 97)
    for f in (oracle.silu, oracle.gelu_tanh):
        np.testing.assert_allclose(f(x) - f(-x), x, atol=1e-14)  # f(x) - f(-x) = x for x*sigmoid-like gates
        assert f(np.array([0.0]))[0] == 0.0
        assert abs(f(np.array([30.0]))[0] - 30.0) < 1e-9
        assert abs(f(np.array([-30.0]))[0]) < 1e-9
    # SiLU slope at 0 is 1/2; sigmoid(1) = 1 / (1 + 1/e)
    assert abs(oracle.silu(np.array([1e-7]))[0] / 1e-7 - 0.5) < 1e-6
    assert abs(oracle.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_gelu_tanh_close_to_erf_gelu():
    x = np.linspace(-5, 5, 201)
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in x])
    err = np.max(np.abs(oracle.gelu_tanh(x) - exact))
    assert 1e-5 < err < 1e-3  # the tanh form is an approximation, close but not equal


def test_softcap_properties():
    z = np.linspace(-500, 500, 1001)
    c = 30.0
    y = oracle.softcap(z, c)
    assert np.all(np.abs(y) < c) and np.all(np.diff(y) > 0)
    small = np.array([1e-3, -2e-3])
    np.testing.assert_allclose(oracle.softcap(small, c), small - small ** 3 / (3 * c * c), rtol=1e-12)
    assert np.argmax(y) == np.argmax(z)


def test_readouts():
    z = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 1.0, 2.5, 0.0]])
    np.testing.assert_array_equal(oracle.argmax_first(z), [1, 0])
    np.testing.assert_allclose(oracle.top2_margin(z), [0.0, 0.5])
    lp = oracle.log_softmax(z)
    np.testing.assert_allclose(np.exp(lp).sum(axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(lp[1, 0] - lp[1, 1], 2.0, rtol=1e-14)
    np.testing.assert_array_equal(oracle.topk_ids(z, 2), [[1, 2], [0, 2]])


# ---------------------------------------------------------------------------
# Whole forward: an independent brute-force restatement on tiny models
# ---------------------------------------------------------------------------
def _bf(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _brute_forward(cfg, wb, ids):
    """Token-by-token, head-by-head loops over plain lists; written from the
    layer description, independent of the oracle module."""
    H, Hq, Hkv, hd, L = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_layers
    S = len(ids)
    W = {n: _bf(b) for n, b in wb.items()}

    def norm(vec, w):
        r = math.sqrt(sum(t * t for t in vec) / len(vec) + cfg.rms_eps)
        return [vec[i] / r * w[i] for i in range(len(vec))]

    def matvec(M, vec):
        return [sum(M[r][c] * vec[c] for c in range(len(vec))) for r in range(len(M))]

    def freqs(kind):
        theta = cfg.rope_theta_local if kind == 1 else cfg.rope_theta_global
        out = []
        for j in range(hd // 2):
            f = theta ** (-(2.0 * j) / hd)
            if cfg.rope_scaling == "llama3":
                C = cfg.rope_orig_max_pos
                wl = 2 * math.pi / f
                if wl > C / cfg.rope_low_freq_factor:
                    f = f / cfg.rope_factor
                elif wl >= C / cfg.rope_high_freq_factor:
                    t = (C / wl - cfg.rope_low_freq_factor) / (cfg.rope_high_freq_factor - cfg.rope_low_freq_factor)
                    f = t * f + (1 - t) * f / cfg.rope_factor
            out.append(f)
        return out

    def rot(vec, p, fr):
        h2 = hd // 2
        res = list(vec)
        for j in range(h2):
            c, s = math.cos(p * fr[j]), math.sin(p * fr[j])
            res[j] = vec[j] * c - vec[j + h2] * s
            res[j + h2] = vec[j + h2] * c + vec[j] * s
        return res

    def gate(g):
        if cfg.act == "silu":
            return g / (1 + math.exp(-g))
        return 0.5 * g * (1 + math.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)))

    scale = 1.0
    if cfg.embed_scale == "sqrt_hidden_bf16":
        scale = float(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.array([math.sqrt(H)], np.float32)))[0])
    xs = [[W["embed"][t][c] * scale for c in range(H)] for t in ids]
    slots = [[list(r) for r in xs]]
    for l in range(L):
        p = f"L{l}."
        kind = cfg.kinds()[l]
        win = cfg.sliding_window if kind == 1 else 0
        fr = freqs(kind)
        Q, K, V = [], [], []
        for t in range(S):
            u = norm(xs[t], W[p + "attn_norm"])
            qt, kt, vt = matvec(W[p + "wq"], u), matvec(W[p + "wk"], u), matvec(W[p + "wv"], u)
            qh = [qt[h * hd:(h + 1) * hd] for h in range(Hq)]
            kh = [kt[h * hd:(h + 1) * hd] for h in range(Hkv)]
            vh = [vt[h * hd:(h + 1) * hd] for h in range(Hkv)]
            if cfg.qk_norm:
                qh = [norm(a, W[p + "q_norm"]) for a in qh]
                kh = [norm(a, W[p + "k_norm"]) for a in kh]
            Q.append([rot(a, t, fr) for a in qh])
            K.append([rot(a, t, fr) for a in kh])
            V.append(vh)
        new_xs = []
        for t in range(S):
            o = []
            for h in range(Hq):
                g = h // (Hq // Hkv)
                js = [j for j in range(t + 1) if win == 0 or t - j < win]
                sc = [sum(Q[t][h][d] * K[j][g][d] for d in range(hd)) / math.sqrt(hd) for j in js]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                o += [sum(e[n] / z * V[js[n]][g][d] for n in range(len(js))) for d in range(hd)]
            a = matvec(W[p + "wo"], o)
            if cfg.norm_layout == "sandwich":
                a = norm(a, W[p + "post_attn_norm"])
            xt = [xs[t][c] + a[c] for c in range(H)]
            u = norm(xt, W[p + "ffn_norm"])
            if cfg.moe_kinds()[l]:
                # router probabilities, then k times the largest remaining one (lowest expert on ties)
                r = matvec(W[p + "router"], u)
                mx = max(r)
                ex = [math.exp(v - mx) for v in r]
                pr = [v / sum(ex) for v in ex]
                chosen = []
                for _ in range(cfg.n_experts_per_tok):
                    best = None
                    for e in range(cfg.n_experts):
                        if e not in chosen and (best is None or pr[e] > pr[best]):
                            best = e
                    chosen.append(best)
                wsum = sum(pr[e] for e in chosen) if cfg.norm_topk else 1.0
                d = [0.0] * H
                for e in chosen:
                    gg = matvec(W[p + "expert_gate"][e], u)
                    uu = matvec(W[p + "expert_up"][e], u)
                    de = matvec(W[p + "expert_down"][e], [gate(gg[i]) * uu[i] for i in range(len(gg))])
                    d = [d[c] + pr[e] / wsum * de[c] for c in range(H)]
            else:
                gg, uu = matvec(W[p + "w_gate"], u), matvec(W[p + "w_up"], u)
                d = matvec(W[p + "w_down"], [gate(gg[i]) * uu[i] for i in range(len(gg))])
            if cfg.norm_layout == "sandwich":
                d = norm(d, W[p + "post_ffn_norm"])
            new_xs.append([xt[c] + d[c] for c in range(H)])
        xs = new_xs
        slots.append([list(r) for r in xs])
    ys = [norm(xs[t], W["final_norm"]) for t in range(S)]
    slots.append(ys)
    head = W["embed"] if cfg.tied else W["lm_head"]
    logits = [matvec(head, y) for y in ys]
    if cfg.final_softcap > 0:
        c = cfg.final_softcap
        logits = [[c * math.tanh(z / c) for z in row] for row in logits]
    return np.array(slots), np.array(logits)


@pytest.mark.parametrize("kind", ["llama", "llama3", "gemma", "moe", "moe-unnormalised"])
def test_forward_matches_brute_force(kind):
    cfg = tiny_config("moe", norm_topk=False) if kind == "moe-unnormalised" else tiny_config(kind)
    wb = synth.make_weights(cfg, seed=11, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 1, 7, seed=5)
    out = oracle.forward(cfg, wb, ids)
    slots, logits = _brute_forward(cfg, wb, list(ids[0]))
    np.testing.assert_allclose(out["hidden"][:, 0], slots, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["logits"][0], logits, rtol=1e-10, atol=1e-10)


def test_forward_batch_independence_and_causality():
    cfg = tiny_config("gemma")
    wb = synth.make_weights(cfg, seed=3, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 3, 9, seed=8)
    out = oracle.forward(cfg, wb, ids)
    one = oracle.forward(cfg, wb, ids[1:2])
    np.testing.assert_allclose(out["logits"][1], one["logits"][0], rtol=1e-12, atol=1e-13)
    pre = oracle.forward(cfg, wb, ids[:, :5])
    np.testing.assert_allclose(out["logits"][:, :5], pre["logits"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["hidden"][:, :, :5], pre["hidden"], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", ["llama", "llama3", "gemma"])
def test_session_matches_cacheless(kind):
    cfg = tiny_config(kind)
    wb = synth.make_weights(cfg, seed=4, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 2, 11, seed=6)
    full = oracle.forward(cfg, wb, ids)
    sess = oracle.Session(cfg, wb, 2)
    z = sess.prefill(ids[:, :6])
    np.testing.assert_allclose(z, full["logits"][:, 5], rtol=1e-9, atol=1e-12)
    for t in range(6, 11):
        z = sess.decode(ids[:, t])
        np.testing.assert_allclose(z, full["logits"][:, t], rtol=1e-9, atol=1e-12)
    # chunked prefill equals one prefill
    s2 = oracle.Session(cfg, wb, 2)
    s2.prefill(ids[:, :3])
    z2 = s2.prefill(ids[:, 3:11])
    np.testing.assert_allclose(z2, full["logits"][:, 10], rtol=1e-9, atol=1e-12)


def test_greedy_feeds_argmax():
    cfg = tiny_config("llama")
    wb = synth.make_weights(cfg, seed=9, sigma=0.3, norm_mode="random")
    prompt = synth.make_ids(cfg, 2, 4, seed=2)
    g = oracle.greedy(cfg, wb, prompt, 5)
    seq = np.concatenate([prompt, g["ids"][:-1].T], axis=1)
    full = oracle.forward(cfg, wb, seq)
    np.testing.assert_array_equal(np.argmax(full["logits"][:, 3:], axis=-1), g["ids"].T)


def test_store_bf16_matches_scalar_rounding():
    x = RNG.standard_normal(3000) * 37.0
    got = oracle.store_bf16(x)
    want = np.array([oracle.round_to_bf16(float(np.float32(v))) for v in x])
    np.testing.assert_array_equal(got, want)


def test_bf16_storage_mode_is_close_but_not_exact():
    cfg = tiny_config("gemma")
    wb = synth.make_weights(cfg, seed=2, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 1, 8, seed=3)
    ex = oracle.forward(cfg, wb, ids)
    st = oracle.forward(cfg, wb, ids, storage="bf16")
    again = oracle.forward(cfg, wb, ids, storage="exact")
    np.testing.assert_array_equal(ex["logits"], again["logits"])
    d = np.abs(st["logits"] - ex["logits"]).max()
    assert 0 < d < 0.05 * np.abs(ex["logits"]).max()
    np.testing.assert_array_equal(st["hidden"][0], ex["hidden"][0])  # the embedding is not a stored activation


def test_oracle_weights_chunked_linear_matches_whole():
    """OracleWeights.linear widens a large weight a block of output rows at a
    time (the full-size Llama and Gemma heads and FFNs take that branch). Force
    the branch on a small matrix with a ragged last block: every output must
    equal the one-shot float64 product (each element is the same dot product
    over the input), and a wrong block offset would move whole columns."""
    rng = np.random.default_rng(17)
    K, N = 96, 1000
    bits = {"w": synth.normal_bf16(5, 77, (N, K), 0.02), "u": synth.normal_bf16(5, 78, (7, K), 1.0)}
    x = oracle.bf16_to_f64(bits["u"]).reshape(1, 7, K)
    chunked = oracle.OracleWeights(bits, cache_limit_bytes=0)
    assert chunked.cache is None  # the widening-on-read path
    whole = oracle.gemm(x, oracle.bf16_to_f64(bits["w"]))
    for rows in (64, 333, 999, 1000):
        got = chunked.linear(x, "w", rows_per_chunk=rows)
        assert got.shape == (1, 7, N)
        np.testing.assert_allclose(got, whole, rtol=1e-13, atol=1e-15)
    # column j is the dot product with weight row j
    j = int(rng.integers(0, N))
    got = chunked.linear(x, "w", rows_per_chunk=64)
    assert abs(got[0, 3, j] - float(np.dot(x[0, 3], oracle.bf16_to_f64(bits["w"][j])))) < 1e-13


def _round_to_f16_scalar(v: float) -> float:
    """IEEE binary16 rounding of a finite scalar written from the format's
    definition: 11 significant bits for normal numbers (|v| >= 2^-14), a fixed
    spacing of 2^-24 below, ties to even, overflow past 65504 to infinity."""
    if v == 0.0:
        return 0.0
    m, e = math.frexp(v)            # v = m * 2^e, 0.5 <= |m| < 1
    if e - 1 >= -14:
        r = math.ldexp(round(m * 2048.0), e - 11)
    else:
        r = math.ldexp(round(math.ldexp(v, 24)), -24)
    if abs(r) > 65504.0:
        return math.copysign(math.inf, v)
    return r


def test_store_f16_matches_scalar_rounding():
    x = np.concatenate([RNG.standard_normal(3000) * 37.0, RNG.standard_normal(500) * 3e-5,
                        RNG.standard_normal(200) * 2e4, [65504.0, 65519.0, 65520.0, -70000.0, 2.0 ** -24,
                                                        2.0 ** -25, 3 * 2.0 ** -26, 1.0 + 2.0 ** -11]])
    got = oracle.store_f16(x)
    want = np.array([_round_to_f16_scalar(float(np.float32(v))) for v in x])
    np.testing.assert_array_equal(got, want)
    # bf16 values of magnitude in [2^-14, 65504] are binary16 values: storing is exact
    b = oracle.store_bf16(RNG.standard_normal(2000) * 0.02)
    b = b[np.abs(b) >= 2.0 ** -14]
    np.testing.assert_array_equal(oracle.store_f16(b), b)


def test_storage_sites_select_rounding():
    cfg = tiny_config("gemma")
    wb = synth.make_weights(cfg, seed=2, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 1, 8, seed=3)
    ex = oracle.forward(cfg, wb, ids)
    allb = oracle.forward(cfg, wb, ids, storage={s: "bf16" for s in oracle.STORAGE_SITES})
    np.testing.assert_array_equal(allb["logits"], oracle.forward(cfg, wb, ids, storage="bf16")["logits"])
    d16 = np.abs(oracle.forward(cfg, wb, ids, storage="f16")["logits"] - ex["logits"]).max()
    db = np.abs(allb["logits"] - ex["logits"]).max()
    assert 0 < d16 < db / 3  # 3 more significant bits
    # one site at a time moves the result; the head input alone moves only the logits
    for site in oracle.STORAGE_SITES:
        one = oracle.forward(cfg, wb, ids, storage={site: "bf16"})
        assert np.abs(one["logits"] - ex["logits"]).max() > 0, site
        if site == "head_in":
            np.testing.assert_array_equal(one["hidden"], ex["hidden"])
    with pytest.raises(ValueError):
        oracle.forward(cfg, wb, ids, storage={"nope": "bf16"})


# ---------------------------------------------------------------------------
# Mixture-of-experts FFN
# ---------------------------------------------------------------------------
def test_moe_route_closed_forms():
    cfg = tiny_config("moe")  # 4 experts, 2 per token, renormalised
    z = np.array([[0.0, 1.0, 1.0, -2.0], [3.0, 0.0, 0.0, 0.0]])
    ids, w, margin = oracle.moe_route(cfg, z)
    np.testing.assert_array_equal(ids, [[1, 2], [0, 1]])  # equal logits: the lower expert first
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=1e-15)
    p = np.exp(z[1]) / np.exp(z[1]).sum()
    np.testing.assert_allclose(w[1], [p[0] / (p[0] + p[1]), p[1] / (p[0] + p[1])], rtol=1e-14)
    np.testing.assert_allclose(margin, [np.exp(1) / np.exp(z[0]).sum() - 1 / np.exp(z[0]).sum(), 0.0],
                               rtol=1e-14, atol=1e-16)
    # without renormalisation the weights are the softmax probabilities; with k = E they are all of them
    ids2, w2, _ = oracle.moe_route(cfg.with_(norm_topk=False), z)
    np.testing.assert_allclose(w2[1], p[[0, 1]], rtol=1e-14)
    ids3, w3, m3 = oracle.moe_route(cfg.with_(n_experts_per_tok=4, norm_topk=False), z)
    np.testing.assert_allclose(w3.sum(-1), 1.0, rtol=1e-14)
    assert np.all(np.isinf(m3))


def test_moe_single_expert_is_the_dense_ffn():
    """One expert, routed with weight 1: the MoE layer is the dense FFN with
    that expert's matrices."""
    cfg = tiny_config("moe", n_experts=1, n_experts_per_tok=1, expert_intermediate=24, moe_layers=(1, 1))
    wb = synth.make_weights(cfg, seed=12, sigma=0.3, norm_mode="random")
    dense_cfg = cfg.with_(n_experts=0, n_experts_per_tok=0, expert_intermediate=0, moe_layers=())
    db = {k: v for k, v in wb.items() if not k.split(".")[-1] in synth.MOE_TENSORS}
    for l in range(cfg.n_layers):
        db[f"L{l}.w_gate"] = wb[f"L{l}.expert_gate"][0]
        db[f"L{l}.w_up"] = wb[f"L{l}.expert_up"][0]
        db[f"L{l}.w_down"] = wb[f"L{l}.expert_down"][0]
    ids = synth.make_ids(cfg, 2, 6, seed=3)
    a, b = oracle.forward(cfg, wb, ids), oracle.forward(dense_cfg, db, ids)
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a["hidden"], b["hidden"], rtol=1e-12, atol=1e-12)


def test_moe_expert_permutation_and_forced_routing():
    """Relabelling the experts (router rows and expert matrices together)
    leaves the output unchanged; forcing the routing the layer would choose
    anyway changes nothing, and forcing another one does."""
    cfg = tiny_config("moe")
    wb = synth.make_weights(cfg, seed=13, sigma=0.3, norm_mode="random")
    ids = synth.make_ids(cfg, 2, 7, seed=4)
    base = oracle.forward(cfg, wb, ids)
    perm = np.array([2, 0, 3, 1])
    pb = dict(wb)
    for t in synth.MOE_TENSORS:
        pb[f"L1.{t}"] = wb[f"L1.{t}"][perm]
    np.testing.assert_allclose(oracle.forward(cfg, pb, ids)["logits"], base["logits"], rtol=1e-12, atol=1e-12)
    chosen = base["moe"][1]["ids"]
    same = oracle.forward(cfg, wb, ids, moe_forced={1: chosen})
    np.testing.assert_array_equal(same["logits"], base["logits"])
    other = oracle.forward(cfg, wb, ids, moe_forced={1: (chosen + 1) % cfg.n_experts})
    assert np.max(np.abs(other["logits"] - base["logits"])) > 1e-3
