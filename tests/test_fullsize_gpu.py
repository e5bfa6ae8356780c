"""Parity at the workloads' full sizes.

* SmolLM2-135M shape with KV cache: 8 sequences x 1024 ids prefilled, 64 greedy
  steps ("N7 · model/forward-parity", Thm 1: cached Prefill within 1e-4 of the
  cacheless Forward; greedy ids token-for-token; hidden cosine; argmax).
* Llama-3-8B shape: a 2 x 512 slice against the oracle (prefill + 16 decode
  steps), and the bench's own launch configuration (4 x 4096 prefill, batch-32
  decode at context 2048) through properties that hold at any size: cached ==
  cacheless, prefix (causality) invariance, decode == cacheless forward of the
  extended sequence, bitwise replay.
* Gemma3-style tower: prompts of 1, 9 and 1024 ids ("pegainfer #878",
  Acceptance Criteria: tight gates and exact top-1 on the short cases, the
  distributional gate at the 1024-token window edge, bitwise replay).

Greedy reading (the margin rule of the parity gates): free-running ids must match until a
step where the oracle's top-1/top-2 margin is <= 1e-2 (a near tie, recorded,
not a failure); a teacher-forced pass then checks the argmax of every step
whose margin exceeds 1e-2.

The exact oracle (float64, nothing rounded) is the definition. On the
SmolLM2 shape the device meets every parity gate against it with bf16
activation storage. On the Llama-3-8B and Gemma-style shapes (random weights
with large hidden sizes make attention sharp, which amplifies rounding noise)
bf16 storage of the norm outputs, q/k/v, attention output and FFN activation
moves the result further than those gates allow: the oracle run with exactly
those roundings (storage="bf16") lands 3-6% (hidden state) from the exact
result, and any other bf16 realisation, the device included, lands as far from
it as from the exact one. Storing the same activations as IEEE f16 (3 more
significant bits, fk_config.f16_sites) brings both shapes inside the gates at
the same tensor-core rate, so there the gates are the forward-parity ones, checked
against the exact oracle. The bf16 storage mode keeps gates derived from its
own noise floor: the device's distance from the exact oracle may be at most
1.25x the bf16-storage oracle's, and the argmax must match wherever the exact
margin exceeds what that noise can flip (2.5x that oracle's largest logit
deviation, and never less than 1e-2).
"""
import gc

import numpy as np
import pytest

import oracle
import synth
from helpers import cosine, weights_to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
MARGIN = 1e-2


def _free():
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _greedy_device(fk, model, prompt, steps, forced=None):
    import torch
    B = prompt.shape[0]
    sess = model.session(B, prompt.shape[1] + steps + 1, max_chunk=1024)
    V = model.cfg.vocab
    z = torch.empty((B, V), dtype=torch.float32, device="cuda")
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    sess.prefill(prompt, logits=z, next_ids=nxt)
    first = z.clone()
    ids = [nxt.cpu().numpy().copy()]
    for t in range(steps):
        feed = None if forced is None else torch.from_numpy(np.ascontiguousarray(forced[t], np.int32)).cuda()
        sess.decode(feed, logits=z, next_ids=nxt)
        ids.append(nxt.cpu().numpy().copy())
    return np.stack(ids), first, z


def _rel_err(a, b):
    """Per-position relative L2 distance over the last axis."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)


def _worst_cos(h, href, stride=1):
    L = h.shape[0]
    return min(cosine(h[l, s], href[l, s]) for l in range(L) for s in range(0, h.shape[1], stride))


def _check_greedy(dev_free, dev_forced, ref):
    ids, margins = ref["ids"], ref["margins"]
    near_ties = []
    for b in range(ids.shape[1]):
        mism = np.nonzero(dev_free[:, b] != ids[:, b])[0]
        if len(mism):
            t = mism[0]
            assert margins[t, b] <= MARGIN, f"seq {b}: greedy ids diverge at step {t} with margin {margins[t, b]}"
            near_ties.append((b, int(t), float(margins[t, b])))
    decided = margins > MARGIN
    np.testing.assert_array_equal(dev_forced[decided], ids[decided])
    return near_ties


def test_smollm2_kv_8x1024_greedy64(fk):
    import torch
    cfg = synth.CONFIGS["smollm2-135m"]
    wb = synth.make_weights(cfg)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=1100)
    prompt = synth.make_ids(cfg, 8, 1024)
    steps = 64
    ref = oracle.greedy(cfg, wb, prompt, steps)
    free, first, _ = _greedy_device(fk, model, prompt, steps)
    forced, _, _ = _greedy_device(fk, model, prompt, steps, forced=ref["ids"][:-1])
    near = _check_greedy(free, forced, ref)
    print("near-tie divergences (seq, step, margin):", near)
    # cached prefill == cacheless forward (last position), and vs the oracle
    out = model.forward(prompt, hidden=True, logits=True, argmax=False)
    torch.cuda.synchronize()
    zf = out["logits"].view(8, 1024, -1)[:, -1]
    assert torch.max(torch.abs(first - zf)).item() <= 1e-4
    assert np.max(np.abs(first.cpu().numpy() - ref["first_logits"])) <= 0.05
    # hidden slots of sequence 0 against the oracle
    h_ref = oracle.forward(cfg, wb, prompt[:1], hidden=True, logits="none")["hidden"][:, 0]
    h = out["hidden"].view(cfg.n_layers + 2, 8, 1024, cfg.hidden)[:, 0].cpu().numpy()
    worst = min(cosine(h[l, s], h_ref[l, s]) for l in range(cfg.n_layers + 2) for s in range(0, 1024, 7))
    assert worst >= 0.9999, worst
    st, flags = model.sync_status()
    assert st == 0, flags
    del model, out
    _free()


def _noise_margin(z_ct):
    return max(MARGIN, 2.5 * z_ct)


def _strict_gates(h, h_ref, z_last, z_last_ref, what):
    """The forward-parity gates of "N7 · model/forward-parity", Thm 1 against
    the exact oracle: hidden cosine >= 0.9999 at every slot and position, and
    last-position logits within 0.05."""
    cos = _worst_cos(h, h_ref)
    dz = float(np.max(np.abs(np.asarray(z_last, np.float64) - z_last_ref)))
    print(f"{what}: worst hidden cosine {cos:.6f}, last logits max|d| {dz:.4f}")
    assert cos >= 0.9999, (what, cos)
    assert dz <= 0.05, (what, dz)
    return cos, dz


def test_llama3_8b_slice_vs_oracle(fk):
    """2 x 512 prefill + 16 decode steps of the full Llama-3-8B shape against
    the exact oracle, in both activation storage formats. f16 storage must
    meet the forward-parity gates; bf16 storage is held to its own noise floor
    (the oracle evaluated with exactly the bf16 storage points)."""
    import torch
    cfg = synth.CONFIGS["llama3-8b"]
    wb = synth.make_weights(cfg)
    wdev = weights_to_dev(wb)
    prompt = synth.make_ids(cfg, 2, 512, stream=3)
    steps = 16
    W = oracle.OracleWeights(wb, cache_limit_bytes=80 << 30)
    ex = oracle.forward(cfg, W, prompt[:1], hidden=True, logits="last")
    ct = oracle.forward(cfg, W, prompt[:1], hidden=True, logits="last", storage="bf16")
    ref = oracle.greedy(cfg, W, prompt, steps)
    del W
    gc.collect()

    # ---- f16 activation storage: the forward-parity gates
    model = fk.Model(cfg.with_(f16_sites=0x3F), wdev, max_positions=600)
    forced, first, _ = _greedy_device(fk, model, prompt, steps, forced=ref["ids"][:-1])
    free, _, _ = _greedy_device(fk, model, prompt, steps)
    out = model.forward(prompt, hidden=True, logits=True, argmax=False)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(out["logits"].view(2, 512, -1)[:, -1] - first)).item() <= 1e-4  # cached == cacheless
    h = out["hidden"].view(cfg.n_layers + 2, 2, 512, cfg.hidden)[:, 0].cpu().numpy()
    _strict_gates(h, ex["hidden"][:, 0], first.cpu().numpy(), ref["first_logits"], "llama3-8b f16 storage")
    decided = ref["margins"] > MARGIN
    print(f"f16: argmax checked at {int(decided.sum())}/{decided.size} teacher-forced steps (margin > {MARGIN})")
    np.testing.assert_array_equal(forced[decided], ref["ids"][decided])
    near = _check_greedy(free, forced, ref)
    print("f16: free-running near-tie divergences (seq, step, margin):", near)
    st, flags = model.sync_status()
    assert st == 0, flags
    del model, out
    _free()

    # ---- device ablation of the storage sites: all f16 but one site in bf16
    # (the prefill of sequence 0 against the exact oracle); every site but
    # the LM-head input has to be f16 for both gates on this shape
    sites = {"qkv_in": 0x1, "attn": 0x2, "o_in": 0x4, "ffn_in": 0x8, "ffn_act": 0x10, "head_in": 0x20}
    print("device ablation, llama3-8b 1x512 prefill vs exact: f16 everywhere but <site> in bf16")
    for name, bit in sites.items():
        model = fk.Model(cfg.with_(f16_sites=0x3F & ~bit), wdev, max_positions=600)
        out = model.forward(prompt[:1], hidden=True, logits=True, argmax=False)
        torch.cuda.synchronize()
        h = out["hidden"].view(cfg.n_layers + 2, 512, cfg.hidden).cpu().numpy()
        zl = out["logits"].view(512, -1)[-1].cpu().numpy().astype(np.float64)
        print(f"  {name:8s} bf16: worst cosine {_worst_cos(h, ex['hidden'][:, 0], 3):.6f}, "
              f"last logits max|d| {np.max(np.abs(zl - ex['logits'][0])):.4f}")
        del model, out
        _free()

    # ---- bf16 activation storage: the noise floor of its storage points
    model = fk.Model(cfg, wdev, max_positions=600)
    forced, first, _ = _greedy_device(fk, model, prompt, steps, forced=ref["ids"][:-1])
    out = model.forward(prompt, hidden=True, logits=True, argmax=False)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(out["logits"].view(2, 512, -1)[:, -1] - first)).item() <= 1e-4
    h = out["hidden"].view(cfg.n_layers + 2, 2, 512, cfg.hidden)[:, 0].cpu().numpy()
    z = first.cpu().numpy()
    e_dev = _rel_err(h, ex["hidden"][:, 0]).max()
    e_ct = _rel_err(ct["hidden"][:, 0], ex["hidden"][:, 0]).max()
    z_dev = np.max(np.abs(z - ref["first_logits"]))
    z_ct = np.max(np.abs(ct["logits"][0] - ex["logits"][0]))
    print(f"llama3-8b bf16 storage vs exact: hidden rel err device {e_dev:.4f} contract {e_ct:.4f}; "
          f"last logits max|d| device {z_dev:.4f} contract {z_ct:.4f}; worst cos device "
          f"{_worst_cos(h, ex['hidden'][:, 0], 3):.6f} contract {_worst_cos(ct['hidden'][:, 0], ex['hidden'][:, 0], 3):.6f}")
    assert e_dev <= 1.25 * e_ct and z_dev <= 1.25 * z_ct + 0.01
    assert _worst_cos(h[:2], ex["hidden"][:2, 0], 3) >= 0.9999
    thr = _noise_margin(z_ct)
    decided = ref["margins"] > thr
    print(f"bf16: argmax checked at {int(decided.sum())}/{decided.size} steps (margin > {thr:.3f})")
    np.testing.assert_array_equal(forced[decided], ref["ids"][decided])
    del model, out, wdev
    _free()


def test_llama3_8b_bench_configuration_properties(fk):
    import torch
    cfg = synth.CONFIGS["llama3-8b"]
    wb = synth.make_weights(cfg)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=4096)
    del wb
    prompt = torch.from_numpy(synth.make_ids(cfg, 4, 4096, stream=10)).cuda()
    sess = model.session(4, 4096)
    z = torch.empty((4, cfg.vocab), dtype=torch.float32, device="cuda")
    sess.prefill(prompt, logits=z)
    sess.reset()
    z2 = torch.empty_like(z)
    sess.prefill(prompt, logits=z2)
    torch.cuda.synchronize()
    assert torch.equal(z, z2)  # bitwise replay
    full = model.forward(prompt, hidden=False, logits=True, argmax=False)
    torch.cuda.synchronize()
    lf = full["logits"].view(4, 4096, -1)
    assert torch.max(torch.abs(lf[:, -1] - z)).item() <= 1e-4  # cached == cacheless
    pre = model.forward(prompt[:, :512].contiguous(), hidden=False, logits=True, argmax=False)
    torch.cuda.synchronize()
    d = torch.max(torch.abs(pre["logits"].view(4, 512, -1) - lf[:, :512])).item()
    assert d <= 1e-4, d  # positions < 512 do not see the later tokens
    del full, pre, sess
    _free()
    # batch-32 decode at context 2048 against the cacheless forward of the extended sequences
    ctx_ids = torch.from_numpy(synth.make_ids(cfg, 32, 2049, stream=50)).cuda()
    sd = model.session(32, 2050)
    sd.prefill(ctx_ids[:, :2048].contiguous())
    zd = torch.empty((32, cfg.vocab), dtype=torch.float32, device="cuda")
    sd.decode(ctx_ids[:, 2048].contiguous(), logits=zd)
    full = model.forward(ctx_ids, hidden=False, logits=True, argmax=False)
    torch.cuda.synchronize()
    zf = full["logits"].view(32, 2049, -1)[:, -1]
    # two bf16 paths (split-K decode vs tiled prefill): they differ by the
    # storage noise of the whole stack, which on this shape is ~4% of the hidden
    # state (see the slice test); bound the relative logit distance and the max.
    rel = (torch.linalg.norm(zf - zd, dim=-1) / torch.linalg.norm(zf, dim=-1)).max().item()
    d = torch.max(torch.abs(zf - zd)).item()
    print(f"decode vs cacheless at ctx 2048: rel {rel:.4f} max|d| {d:.4f}")
    assert rel <= 0.06 and d <= 0.5, (rel, d)
    st, flags = model.sync_status()
    assert st == 0, flags
    del model, full, sd
    _free()


def test_gemma3_tower_1_9_1024(fk):
    import torch
    cfg = synth.CONFIGS["gemma3-tower"]
    wb = synth.make_weights(cfg)
    wdev = weights_to_dev(wb)
    P = synth.make_ids(cfg, 1, 1024, stream=4)
    # the 1- and 9-token prompts are prefixes of the 1024-token one (causality)
    ex = oracle.forward(cfg, wb, P, hidden=True, logits="all")
    ct = oracle.forward(cfg, wb, P[:, :9], hidden=True, logits="all", storage="bf16")
    del wb
    gc.collect()
    zx, zc = ex["logits"][0], ct["logits"][0]
    lpr = oracle.log_softmax(zx)
    top64 = oracle.topk_ids(zx, 64)

    def window_edge(model, what):
        """The 1024-token window edge: distributional gate against the exact
        oracle ("pegainfer issue #878", Acceptance Criteria), bitwise replay."""
        out = model.forward(P, hidden=False)
        out2 = model.forward(P, hidden=False)
        torch.cuda.synchronize()
        assert torch.equal(out["logits"], out2["logits"])  # bitwise replay
        z = out["logits"].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(z))
        lp = oracle.log_softmax(z)
        assert np.all(np.isfinite(lp))
        top1 = np.argmax(z, axis=-1) == oracle.argmax_first(zx)
        quarters = [int(top1[q * 256:(q + 1) * 256].sum()) for q in range(4)]
        dlp = np.max(np.abs(np.take_along_axis(lp, top64, -1) - np.take_along_axis(lpr, top64, -1)))
        print(f"{what} window edge: top-1 {int(top1.sum())}/1024, quarters {quarters}, max|dlogprob|@top64 {dlp:.4g}")
        assert top1.sum() >= 802 and min(quarters) >= 179 and dlp <= 16.4
        return z

    # ---- f16 activation storage: the forward-parity gates at 1 and 9 tokens
    model = fk.Model(cfg.with_(f16_sites=0x3F), wdev, max_positions=1024)
    for S in (1, 9):
        out = model.forward(P[:, :S])
        torch.cuda.synchronize()
        z = out["logits"].cpu().numpy()
        assert np.all(np.isfinite(z))
        h = out["hidden"].view(cfg.n_layers + 2, S, cfg.hidden).cpu().numpy()
        _strict_gates(h, ex["hidden"][:, 0, :S], z[S - 1], zx[S - 1], f"gemma f16 storage S={S}")
        assert np.max(np.abs(z - zx[:S])) <= 0.05  # every position, not only the last
        decided = oracle.top2_margin(zx[:S]) > MARGIN
        np.testing.assert_array_equal(out["argmax"].cpu().numpy()[decided], oracle.argmax_first(zx[:S])[decided])
        del out
    z16 = window_edge(model, "f16")
    top1 = np.argmax(z16, axis=-1) == oracle.argmax_first(zx)
    decided = oracle.top2_margin(zx) > MARGIN
    assert np.all(top1[decided]), int((~top1[decided]).sum())  # exact top-1 wherever the margin exceeds 1e-2
    del model
    _free()

    # ---- bf16 activation storage: the noise floor of its storage points
    model = fk.Model(cfg, wdev, max_positions=1024)
    for S in (1, 9):
        out = model.forward(P[:, :S])
        torch.cuda.synchronize()
        z = out["logits"].cpu().numpy()
        assert np.all(np.isfinite(z))
        h = out["hidden"].view(cfg.n_layers + 2, S, cfg.hidden).cpu().numpy()
        e_dev = _rel_err(h, ex["hidden"][:, 0, :S]).max()
        e_ct = _rel_err(ct["hidden"][:, 0, :S], ex["hidden"][:, 0, :S]).max()
        z_dev, z_ct = np.max(np.abs(z - zx[:S])), np.max(np.abs(zc[:S] - zx[:S]))
        print(f"gemma bf16 storage S={S} vs exact: hidden rel err device {e_dev:.4f} contract {e_ct:.4f}; "
              f"logits max|d| device {z_dev:.4f} contract {z_ct:.4f}; worst cos device "
              f"{_worst_cos(h, ex['hidden'][:, 0, :S]):.6f}")
        assert e_dev <= 1.25 * e_ct and z_dev <= 1.25 * z_ct + 0.01
        assert _worst_cos(h[:2], ex["hidden"][:2, 0, :S]) >= 0.9999
        decided = oracle.top2_margin(zx[:S]) > _noise_margin(z_ct)
        np.testing.assert_array_equal(out["argmax"].cpu().numpy()[decided], oracle.argmax_first(zx[:S])[decided])
        del out
    window_edge(model, "bf16")
    del model, wdev
    _free()


def test_gemma3_tower_decode_past_the_window(fk):
    """Gemma-style decode past the 1024-token window: 1100 ids prefilled in
    chunks of 64 (the local layers' ring then holds 1024 + 63 -> 1088
    positions and wraps), then 16 teacher-forced decode steps, every call's
    logits against the exact oracle session ("N7 · model/forward-parity",
    Thm 2: sliding-window non-vacuity; "pegainfer issue #878": beyond the
    window edge). f16 storage: the forward-parity logit and argmax gates on all
    17 calls; bf16 storage: the distributional gate."""
    import os
    import torch
    cfg = synth.CONFIGS["gemma3-tower"]
    wb = synth.make_weights(cfg)
    wdev = weights_to_dev(wb)
    P = synth.make_ids(cfg, 1, 1100, stream=4)
    steps = 16
    ram = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    f64_bytes = sum(int(v.size) for v in wb.values()) * 8  # the widened weights, cached if the host has room
    W = oracle.OracleWeights(wb, cache_limit_bytes=f64_bytes + 1 if ram > f64_bytes + (64 << 30) else (2 << 30))
    osess = oracle.Session(cfg, W, 1)
    zs = [osess.prefill(P)[0]]
    ids = [int(oracle.argmax_first(zs[0]))]
    for t in range(steps):
        zs.append(osess.decode(np.array([ids[-1]]))[0])
        ids.append(int(oracle.argmax_first(zs[-1])))
    zr = np.stack(zs)
    del osess, W, wb
    gc.collect()
    margins = oracle.top2_margin(zr)
    lpr = oracle.log_softmax(zr)
    top64 = oracle.topk_ids(zr, 64)

    def run(model):
        sess = model.session(1, P.shape[1] + steps + 1, max_chunk=64)
        z = torch.empty((1, cfg.vocab), dtype=torch.float32, device="cuda")
        nxt = torch.empty((1,), dtype=torch.int32, device="cuda")
        sess.prefill(P, logits=z, next_ids=nxt)
        rows, am = [z.cpu().numpy()[0].copy()], [int(nxt.item())]
        for t in range(steps):
            sess.decode(torch.tensor([ids[t]], dtype=torch.int32, device="cuda"), logits=z, next_ids=nxt)
            rows.append(z.cpu().numpy()[0].copy())
            am.append(int(nxt.item()))
        st, flags = model.sync_status()
        assert st == 0, flags
        return np.stack(rows).astype(np.float64), np.array(am)

    lib = fk.load()
    for f16 in (0x3F, 0):
        model = fk.Model(cfg.with_(f16_sites=f16), wdev, max_positions=P.shape[1] + steps + 1)
        z, am = run(model)
        assert np.all(np.isfinite(z))
        dz = np.max(np.abs(z - zr), axis=-1)
        lp = oracle.log_softmax(z)
        dlp = np.max(np.abs(np.take_along_axis(lp, top64, -1) - np.take_along_axis(lpr, top64, -1)))
        top1 = am == np.array(ids)
        print(f"gemma decode past the window, f16_sites={f16:#x}: logits max|d| per call max {dz.max():.4f}, "
              f"top-1 {int(top1.sum())}/{len(ids)}, max|dlogprob|@top64 {dlp:.4g}")
        if f16:
            assert dz.max() <= 0.05, dz
            np.testing.assert_array_equal(am[margins > MARGIN], np.array(ids)[margins > MARGIN])
        else:
            assert top1.mean() >= 802 / 1024 and dlp <= 16.4
        del model
        _free()
    del wdev
    _free()
