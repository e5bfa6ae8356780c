"""Mixture-of-experts FFN on the device against the oracle ("N7 ·
model/forward-parity", Thm 2: the qwen3moe rung).

Routing is a discrete choice: where two experts' probabilities are within
rounding of each other, fp32 on the device and float64 in the oracle may pick
differently, and both are right. So the parity of the arithmetic is checked
with the device's routing forced to the oracle's choice (its weights still
come from the device's own router), and the routing itself is checked where
the oracle's margin (probability of the k-th minus the (k+1)-th expert) is
clear of that rounding: there the device must choose the same experts.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import cosine, err_scale, weights_to_dev

pytestmark = pytest.mark.gpu

ROUTE_MARGIN = 1e-4  # probability gap above which fp32 and float64 routing of the same input must agree
FORWARD_ROUTE_MARGIN = 1e-2  # the same through the whole forward (router inputs differ by storage rounding)


def _logits(T, E, seed, scale=2.0):
    return synth.normal_f32(seed, T, (T, E), 1.0) * np.float32(scale)


# ---------------------------------------------------------------------------
# routing op
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,norm", [(300, 128, 8, True), (300, 128, 8, False), (65, 8, 2, True),
                                        (130, 16, 16, True), (1, 256, 16, False), (7, 64, 1, True)])
def test_moe_route_vs_oracle(fk, T, E, k, norm):
    import torch
    z = _logits(T, E, seed=71)
    cfg = synth.small_config("moe").with_(n_experts=E, n_experts_per_tok=k, norm_topk=norm)
    ids, w, margin = oracle.moe_route(cfg, z.astype(np.float64))
    out = fk.moe_route(torch.from_numpy(z).cuda(), k, norm_topk=norm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out["ids"].cpu().numpy(), ids)
    np.testing.assert_allclose(out["weights"].cpu().numpy(), w, rtol=2e-6, atol=1e-7)
    m = out["margin"].cpu().numpy()
    if k == E:
        assert np.all(np.isinf(m))
    else:
        np.testing.assert_allclose(m, margin, atol=2e-7)
    assert fk.op_sync_status()[0] == 0


def test_moe_route_ties_and_forced(fk):
    import torch
    E, k = 16, 4
    z = _logits(6, E, seed=72)
    z[0] = 0.0                              # every expert equal: the four lowest ids
    z[1, [3, 9, 12, 14, 15]] = 7.0          # five equal maxima: the four lowest of them
    cfg = synth.small_config("moe").with_(n_experts=E, n_experts_per_tok=k)
    forced = np.array([[5, 1, 0, 2]] * 6, dtype=np.int32)
    forced[3] = [1, 1, 2, 3]                # repeated id: row 3 routes itself
    forced[4] = [0, 1, 2, 16]               # out of range: row 4 routes itself
    zt = torch.from_numpy(z).cuda()
    nat = fk.moe_route(zt, k)
    out = fk.moe_route(zt, k, forced=torch.from_numpy(forced).cuda())
    torch.cuda.synchronize()
    ids, w, _ = oracle.moe_route(cfg, z.astype(np.float64))
    assert list(nat["ids"].cpu().numpy()[0]) == [0, 1, 2, 3]
    assert list(nat["ids"].cpu().numpy()[1]) == [3, 9, 12, 14]
    np.testing.assert_array_equal(nat["ids"].cpu().numpy(), ids)
    got = out["ids"].cpu().numpy()
    for r in (0, 1, 2, 5):
        np.testing.assert_array_equal(got[r], forced[r])
        p = np.exp(z[r].astype(np.float64) - z[r].max())
        p /= p.sum()
        np.testing.assert_allclose(out["weights"].cpu().numpy()[r], p[forced[r]] / p[forced[r]].sum(), rtol=2e-6)
    np.testing.assert_array_equal(got[3], ids[3])
    np.testing.assert_array_equal(got[4], ids[4])
    st, flags = fk.op_sync_status()
    assert st == 7 and flags & fk.DEVERR_EXPERT_IDS, (st, flags)
    assert fk.op_sync_status()[0] == 0  # reading the word cleared it


def test_moe_route_rejects_bad_arguments(fk):
    import torch
    z = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    for k in (0, 9):
        with pytest.raises(fk.FkError) as ei:
            fk.moe_route(z, k)
        assert ei.value.status == 1
    with pytest.raises(fk.FkError):
        fk.moe_route(torch.zeros((4, 264), dtype=torch.float32, device="cuda"), 2)


# ---------------------------------------------------------------------------
# the MoE FFN of one layer
# ---------------------------------------------------------------------------
def _u(cfg, T, seed, f16=False):
    """FFN-norm-like rows: N(0, 1) values stored in the 16-bit site type."""
    import torch
    x = synth.normal_f32(seed, T, (T, cfg.hidden), 1.0)
    t = torch.from_numpy(x).to(torch.float16 if f16 else torch.bfloat16)
    return t.cuda(), t.to(torch.float64).numpy()


def _moe_layer_check(fk, cfg, layer, T, seed, f16=False, tol=4e-3, skew=False):
    import torch
    wb = synth.make_weights(cfg, seed=seed, sigma=0.02)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    u_dev, u = _u(cfg, T, seed + 1, f16)
    W = oracle.OracleWeights(wb)
    storage = "f16" if f16 else "bf16"
    ref = oracle.moe_ffn(cfg, W, layer, u, storage)
    # forced to the oracle's routing: the arithmetic alone
    forced = torch.from_numpy(ref["ids"].astype(np.int32)).cuda()
    got = model.moe_ffn(layer, u_dev, forced=forced)
    torch.cuda.synchronize()
    st, flags = model.sync_status()
    assert st == 0, flags
    np.testing.assert_array_equal(got["ids"].cpu().numpy(), ref["ids"])
    y = got["out"].cpu().numpy()
    e = err_scale(y, ref["out"])
    c = min(cosine(y[t], ref["out"][t]) for t in range(T))
    print(f"{cfg.name} layer {layer} T={T} {storage}: err/max {e:.2e}, worst row cosine {c:.6f}")
    assert e <= tol and c >= 0.9999, (e, c)
    # the device's own routing agrees wherever the choice is clear
    nat = model.moe_ffn(layer, u_dev)
    torch.cuda.synchronize()
    clear = ref["margin"] > ROUTE_MARGIN
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(nat["ids"].cpu().numpy()[clear], ref["ids"][clear])
    np.testing.assert_allclose(nat["margin"].cpu().numpy(), ref["margin"], atol=1e-6)
    same = np.all(nat["ids"].cpu().numpy() == ref["ids"], axis=-1)
    np.testing.assert_array_equal(nat["out"].cpu().numpy()[same], y[same])
    if skew:
        # a skewed routing: even tokens to experts 0..k-1, odd ones to k..2k-1
        # (a few experts with many 128-row tiles, every other expert empty)
        k = cfg.n_experts_per_tok
        sk = (np.arange(k)[None, :] + k * (np.arange(T)[:, None] % 2)).astype(np.int64)
        ref2 = oracle.moe_ffn(cfg, W, layer, u, storage, forced_ids=sk)
        got2 = model.moe_ffn(layer, u_dev, forced=torch.from_numpy(sk.astype(np.int32)).cuda())
        torch.cuda.synchronize()
        y2 = got2["out"].cpu().numpy()
        e2 = err_scale(y2, ref2["out"])
        c2 = min(cosine(y2[t], ref2["out"][t]) for t in range(T))
        print(f"  skewed routing ({2 * k} experts used): err/max {e2:.2e}, worst row cosine {c2:.6f}")
        assert e2 <= tol and c2 >= 0.9999, (e2, c2)
    return e


@pytest.mark.parametrize("T", [1, 63, 300])
def test_moe_ffn_small_vs_oracle(fk, T):
    cfg = synth.small_config("moe")
    _moe_layer_check(fk, cfg, layer=1, T=T, seed=31, skew=T == 300)


def test_moe_ffn_small_f16_sites(fk):
    cfg = synth.small_config("moe").with_(f16_sites=fk.F16_FFN_IN | fk.F16_FFN_ACT)
    _moe_layer_check(fk, cfg, layer=2, T=200, seed=32, f16=True, tol=1e-3)


@pytest.mark.slow
def test_moe_ffn_qwen3_moe_layer_full_width(fk):
    """One MoE layer of the Qwen3-30B-A3B geometry (128 experts of width 768,
    8 per token, hidden 2048) on 2048 tokens: 16384 routed rows over 128
    expert groups of uneven sizes (one to two 128-row tiles each), then a
    skewed routing of 16 experts with eight tiles each and 112 empty ones.
    The vocabulary is cut to 1024: the head plays no part here."""
    import gc
    import torch
    cfg = synth.CONFIGS["qwen3-moe-30b-a3b"].with_(n_layers=1, vocab=1024)
    _moe_layer_check(fk, cfg, layer=0, T=2048, seed=33, skew=True)
    gc.collect()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the forward and the session of a model with MoE layers
# ---------------------------------------------------------------------------
def _forced_tensor(cfg, traces, rows):
    """[n_moe][rows][k] int32 from the oracle's per-layer traces."""
    import torch
    layers = [l for l in range(cfg.n_layers) if cfg.moe_kinds()[l]]
    arr = np.stack([np.asarray(traces[l]["ids"]).reshape(rows, cfg.n_experts_per_tok) for l in layers])
    return torch.from_numpy(arr.astype(np.int32)).cuda()


def _forward_check(fk, cfg, B, S, seed):
    import torch
    wb = synth.make_weights(cfg, seed=seed, sigma=0.02, norm_mode="random")
    ids = synth.make_ids(cfg, B, S, seed=seed + 1)
    ref = oracle.forward(cfg, wb, ids)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=S)
    T = B * S
    n_moe = sum(cfg.moe_kinds())
    k = cfg.n_experts_per_tok
    forced = _forced_tensor(cfg, ref["moe"], T)
    tr_ids = torch.empty((n_moe, T, k), dtype=torch.int32, device="cuda")
    tr_m = torch.empty((n_moe, T), dtype=torch.float32, device="cuda")
    model.set_moe_routing(forced, tr_ids, tr_m, T)
    out = model.forward(ids)
    torch.cuda.synchronize()
    model.set_moe_routing()
    st, flags = model.sync_status()
    assert st == 0, flags
    np.testing.assert_array_equal(tr_ids.cpu().numpy(), forced.cpu().numpy())
    hid = out["hidden"].cpu().numpy().reshape(cfg.n_layers + 2, B, S, cfg.hidden)
    worst = min(cosine(hid[l, b, s], ref["hidden"][l, b, s])
                for l in range(cfg.n_layers + 2) for b in range(B) for s in range(S))
    z = out["logits"].cpu().numpy().reshape(B, S, cfg.vocab)
    last = float(np.max(np.abs(z[:, -1] - ref["logits"][:, -1])))
    print(f"{cfg.name} forward B={B} S={S}: worst cosine {worst:.6f}, last logits max|d| {last:.4f}")
    assert worst >= 0.9999 and last <= 0.05
    decided = oracle.top2_margin(ref["logits"]) > 1e-2
    am = out["argmax"].cpu().numpy().reshape(B, S)
    np.testing.assert_array_equal(am[decided], oracle.argmax_first(ref["logits"])[decided])
    # unforced: the routing agrees with the oracle's wherever it is clear
    model.set_moe_routing(None, tr_ids, tr_m, T)
    out2 = model.forward(ids)
    torch.cuda.synchronize()
    model.set_moe_routing()
    # (the router input carries the forward's bf16 storage rounding, which
    # moves router probabilities by ~1e-4 against the exact oracle; a token
    # routed differently upstream has a different input downstream)
    # The margin separates the k chosen experts from the rest, not their
    # order among themselves: compare the chosen sets.
    got = np.sort(tr_ids.cpu().numpy(), axis=-1)
    agree = np.ones(T, dtype=bool)
    for i, l in enumerate(l for l in range(cfg.n_layers) if cfg.moe_kinds()[l]):
        want = np.sort(np.asarray(ref["moe"][l]["ids"]).reshape(T, k), axis=-1)
        sel = agree & (np.asarray(ref["moe"][l]["margin"]).reshape(T) > FORWARD_ROUTE_MARGIN)
        print(f"  MoE layer {l}: {sel.mean():.2f} of tokens clear, {np.mean(np.all(got[i] == want, -1)):.3f} agree")
        assert sel.mean() > 0.3
        np.testing.assert_array_equal(got[i][sel], want[sel])
        agree &= np.all(got[i] == want, axis=-1)
    # without the hook the same forward as with the trace-only hook
    out3 = model.forward(ids)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out3["logits"].cpu().numpy(), out2["logits"].cpu().numpy())
    return model, wb


def test_moe_forward_small_vs_oracle(fk):
    """small-moe: dense, MoE, MoE layers; two sequences of 150 tokens (three
    64-row routing blocks per call, ragged)."""
    _forward_check(fk, synth.small_config("moe"), B=2, S=150, seed=41)


def test_moe_forward_small_unnormalised_gelu_sandwich(fk):
    """The other branches of the layer: weights not renormalised, the GELU
    gate and the sandwich norm layout around the MoE FFN."""
    cfg = synth.small_config("moe").with_(norm_topk=False, act="gelu_tanh", norm_layout="sandwich",
                                          n_experts_per_tok=3)
    _forward_check(fk, cfg, B=1, S=97, seed=42)


def test_moe_session_prefill_decode(fk):
    """Session prefill in chunks, then decode steps, each forced to the
    oracle session's routing, against the oracle session; then the same
    session unforced: chunked prefill agrees with the cacheless forward."""
    import torch
    cfg = synth.small_config("moe")
    B, P, C, steps = 2, 150, 64, 6
    wb = synth.make_weights(cfg, seed=43, sigma=0.02, norm_mode="random")
    prompt = synth.make_ids(cfg, B, P, seed=44)
    feed = synth.make_ids(cfg, steps, B, seed=45)  # teacher-forced decode ids
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=P + steps)
    sess = model.session(B, P + steps, max_chunk=C)
    osess = oracle.Session(cfg, wb, B)
    n_moe = sum(cfg.moe_kinds())
    k = cfg.n_experts_per_tok
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    worst = 0.0
    for c0 in range(0, P, C):
        chunk = prompt[:, c0:c0 + C]
        zr = osess.prefill(chunk)
        rows = chunk.size
        forced = _forced_tensor(cfg, osess.moe["trace"], rows)
        model.set_moe_routing(forced, None, None, rows)
        sess.prefill(chunk, logits=z)
        torch.cuda.synchronize()
        worst = max(worst, float(np.max(np.abs(z.cpu().numpy() - zr))))
    for t in range(steps):
        zr = osess.decode(feed[t])
        forced = _forced_tensor(cfg, osess.moe["trace"], B)
        model.set_moe_routing(forced, None, None, B)
        sess.decode(torch.from_numpy(feed[t].astype(np.int32)).cuda(), logits=z)
        torch.cuda.synchronize()
        worst = max(worst, float(np.max(np.abs(z.cpu().numpy() - zr))))
    model.set_moe_routing()
    print(f"small-moe session, forced routing: logits max|d| over prefill chunks and decode {worst:.4f}")
    assert worst <= 0.05
    st, flags = model.sync_status()
    assert st == 0, flags
    # a prefill longer than a chunk is refused while the hook is set
    tr = torch.empty((n_moe, B * P, k), dtype=torch.int32, device="cuda")
    model.set_moe_routing(None, tr, None, B * P)
    sess.reset()
    with pytest.raises(fk.FkError):
        sess.prefill(prompt, logits=z)
    model.set_moe_routing()
    # unforced: chunked prefill = the cacheless forward's last position, bit for bit
    sess.reset()
    sess.prefill(prompt, logits=z)
    full = model.forward(prompt, hidden=False)
    torch.cuda.synchronize()
    zl = full["logits"].cpu().numpy().reshape(B, P, cfg.vocab)[:, -1]
    np.testing.assert_array_equal(z.cpu().numpy(), zl)
    # and the captured greedy decode steps run (graphs back on without the hook)
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    for _ in range(3):
        sess.decode(logits=z, next_ids=nxt)
    torch.cuda.synchronize()
    assert model.sync_status()[0] == 0


@pytest.mark.slow
def test_qwen3_moe_two_layer_slice(fk):
    """Two layers of the Qwen3-30B-A3B geometry at full width (QK-norm, 128
    experts, 8 per token, the 151936-word untied head) with f16 activation
    storage, routing forced to the oracle's: the forward-parity gates (hidden
    cosine >= 0.9999 at every slot, last-position logits within 0.05)."""
    import gc
    import torch
    cfg = synth.CONFIGS["qwen3-moe-30b-a3b"].with_(n_layers=2, f16_sites=0x3F)
    B, S = 1, 192
    wb = synth.make_weights(cfg, norm_mode="random")
    ids = synth.make_ids(cfg, B, S, stream=23)
    ref = oracle.forward(cfg, wb, ids, hidden=True, logits="last")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=S)
    T, k = B * S, cfg.n_experts_per_tok
    forced = _forced_tensor(cfg, ref["moe"], T)
    model.set_moe_routing(forced, None, None, T)
    out = model.forward(ids, argmax=False)
    torch.cuda.synchronize()
    model.set_moe_routing()
    st, flags = model.sync_status()
    assert st == 0, flags
    h = out["hidden"].cpu().numpy().reshape(cfg.n_layers + 2, S, cfg.hidden)
    worst = min(cosine(h[l, s], ref["hidden"][l, 0, s]) for l in range(cfg.n_layers + 2) for s in range(S))
    z = out["logits"].cpu().numpy().reshape(S, cfg.vocab)[-1]
    dz = float(np.max(np.abs(z - ref["logits"][0])))
    print(f"qwen3-moe 2-layer slice (f16 storage, forced routing): worst cosine {worst:.6f}, last logits max|d| {dz:.4f}")
    assert worst >= 0.9999 and dz <= 0.05
    del model, out
    gc.collect()
    torch.cuda.empty_cache()
