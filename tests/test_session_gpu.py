"""KV-cached session ("N7", Thm 1: cached Prefill last-position logits agree
with the cacheless Forward within 1e-4; greedy ids token-for-token)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import weights_to_dev

pytestmark = pytest.mark.gpu


def _setup(fk, cfg, norm_mode="random", sigma=0.02):
    wb = synth.make_weights(cfg, norm_mode=norm_mode, sigma=sigma)
    return wb, fk.Model(cfg, weights_to_dev(wb), max_positions=512)


@pytest.mark.parametrize("kind,chunk,f16", [("llama", 48, 0), ("llama3", 48, 0), ("gemma", 48, 0), ("llama", 45, 0),
                                            ("llama3", 37, 0), ("gemma", 45, 0x3F), ("llama3", 48, 0x3F)])
def test_cached_prefill_matches_cacheless(fk, kind, chunk, f16):
    """Chunks of 48 start at positions that are multiples of 8 (the V cache
    takes 16-byte runs); 45 and 37 exercise the unaligned element path."""
    import torch
    cfg = synth.small_config(kind, f16_sites=f16)
    wb, model = _setup(fk, cfg)
    B, S = 2, 100
    ids = synth.make_ids(cfg, B, S)
    full = model.forward(ids, hidden=False)
    sess = model.session(B, 256, max_chunk=chunk)  # three chunks
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    sess.prefill(ids, logits=z, next_ids=nxt)
    torch.cuda.synchronize()
    zf = full["logits"].view(B, S, -1)[:, -1]
    assert torch.max(torch.abs(z - zf)).item() <= 1e-4
    assert sess.length == S


@pytest.mark.parametrize("kind,f16", [("llama", 0), ("llama3", 0), ("gemma", 0), ("llama3", 0x3F), ("gemma", 0x3F),
                                      ("qwen3", 0), ("qwen3", 0x3F), ("mistral", 0)])
def test_decode_matches_oracle(fk, kind, f16):
    import torch
    cfg = synth.small_config(kind, f16_sites=f16)
    wb, model = _setup(fk, cfg)
    B, S, steps = 3, 21, 12
    prompt = synth.make_ids(cfg, B, S)
    ref = oracle.greedy(cfg, wb, prompt, steps)
    sess = model.session(B, 64)
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    sess.prefill(prompt, logits=z, next_ids=nxt)
    got = [nxt.cpu().numpy().copy()]
    for t in range(steps):
        # teacher forcing with the oracle's ids keeps both sides on one path
        feed = torch.from_numpy(ref["ids"][t].astype(np.int32)).cuda()
        sess.decode(feed, logits=z, next_ids=nxt)
        got.append(nxt.cpu().numpy().copy())
    got = np.stack(got)
    decided = ref["margins"] > 1e-2
    np.testing.assert_array_equal(got[decided], ref["ids"][decided])
    np.testing.assert_allclose(z.cpu().numpy(), ref["last_logits"], atol=0.05)


@pytest.mark.parametrize("B,hidden", [(1, 128), (8, 128), (24, 128), (1, 512), (8, 512)])
def test_decode_with_wide_head_matches_cacheless_forward(fk, B, hidden):
    """A vocabulary much wider than the layers: the LM head's split-K GEMM has
    far more feature tiles than the layer GEMMs that share its scratch.
    Several graph-replayed decode steps must each equal the cacheless forward
    of the extended sequences at the new position (every logit written).
    Both sides round the same bf16 activations after different fp32
    summation orders (split-K against tiled GEMMs), so the bound scales with
    the logits' spread, about sqrt(hidden) * 0.02."""
    import torch
    cfg = synth.small_config("llama", vocab=32768, hidden=hidden, intermediate=2 * hidden)
    wb, model = _setup(fk, cfg)
    S, steps = 40, 4
    prompt = synth.make_ids(cfg, B, S)
    sess = model.session(B, 64)
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    sess.prefill(prompt, logits=z, next_ids=nxt)
    seq = [prompt, nxt.cpu().numpy().copy()[:, None]]
    for _ in range(steps):
        z.fill_(float("nan"))
        sess.decode(None, logits=z, next_ids=nxt)
        ext = np.concatenate(seq, axis=1).astype(np.int32)
        full = model.forward(ext, hidden=False)
        zf = full["logits"].view(B, ext.shape[1], -1)[:, -1]
        torch.cuda.synchronize()
        assert torch.isfinite(z).all()
        assert torch.max(torch.abs(z - zf)).item() <= 1e-2 * max(1.0, (hidden / 128) ** 0.5)
        seq.append(nxt.cpu().numpy().copy()[:, None])


def test_graph_decode_equals_launched_decode(fk):
    """Steps fed back from the previous argmax replay a captured CUDA graph;
    feeding the same ids explicitly launches kernel by kernel. Same bits."""
    import torch
    cfg = synth.small_config("llama")
    wb, model = _setup(fk, cfg)
    prompt = synth.make_ids(cfg, 2, 30)
    a, b = model.session(2, 64), model.session(2, 64)
    za, zb = (torch.empty((2, cfg.vocab), dtype=torch.float32, device="cuda") for _ in range(2))
    na, nb = (torch.empty((2,), dtype=torch.int32, device="cuda") for _ in range(2))
    a.prefill(prompt, logits=za, next_ids=na)
    b.prefill(prompt, logits=zb, next_ids=nb)
    for _ in range(8):
        feed = nb.clone()
        a.decode(None, logits=za, next_ids=na)        # graph
        b.decode(feed, logits=zb, next_ids=nb)        # one by one
        torch.cuda.synchronize()
        assert torch.equal(za, zb) and torch.equal(na, nb)
    assert a.length == b.length == 38


@pytest.mark.parametrize("kind,f16", [("gemma", 0), ("gemma", 0x3F), ("llama-window", 0), ("mistral", 0),
                                      ("mistral", 0x3F)])
def test_sliding_window_ring_cache_past_the_window(fk, kind, f16):
    """Sliding-window layers keep a ring of W + max_chunk - 1 positions
    (rounded up to 64): prefill 100 ids in chunks of 16 and decode 40 greedy
    steps past it, so a W = 16 (or 24) window is non-vacuous and the 64-slot
    ring wraps twice; every step against the exact oracle ("N7 ·
    model/forward-parity", Thm 2: sliding-window layers; "pegainfer issue
    #878": the window edge)."""
    import torch
    if kind == "llama-window":
        cfg = synth.small_config("llama", sliding_window=24, layer_kinds=(1, 0))
    else:
        cfg = synth.small_config(kind, f16_sites=f16)
    wb, model = _setup(fk, cfg)
    lib = fk.load()
    B, S, steps, chunk, max_seq = 2, 100, 40, 16, 160
    # the session is smaller than one with every layer global by exactly the
    # ring's savings: 2 caches x B x Hkv x hd x 2 bytes x (global - ring) positions
    all_global = cfg.with_(layer_kinds=tuple(0 for _ in cfg.kinds()))
    m_glob = fk.Model(all_global, model.weights, max_positions=512)
    n_local = sum(1 for k in cfg.kinds() if k == 1)
    ring = (cfg.sliding_window + chunk - 1 + 63) // 64 * 64
    glob = (max_seq + 63) // 64 * 64
    saved = 2 * B * cfg.n_kv_heads * cfg.head_dim * 2 * (glob - ring) * n_local
    assert lib.fk_session_bytes(m_glob.handle, B, max_seq, chunk) - lib.fk_session_bytes(model.handle, B, max_seq,
                                                                                         chunk) == saved
    prompt = synth.make_ids(cfg, B, S, stream=7)
    ref = oracle.greedy(cfg, wb, prompt, steps)
    sess = model.session(B, max_seq, max_chunk=chunk)
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.empty((B,), dtype=torch.int32, device="cuda")
    sess.prefill(prompt, logits=z, next_ids=nxt)
    torch.cuda.synchronize()
    np.testing.assert_allclose(z.cpu().numpy(), ref["first_logits"], atol=0.05)
    got = [nxt.cpu().numpy().copy()]
    worst = 0.0
    for t in range(steps):
        feed = torch.from_numpy(ref["ids"][t].astype(np.int32)).cuda()  # teacher forcing
        sess.decode(feed, logits=z, next_ids=nxt)
        got.append(nxt.cpu().numpy().copy())
    got = np.stack(got)
    decided = ref["margins"] > 1e-2
    np.testing.assert_array_equal(got[decided], ref["ids"][decided])
    np.testing.assert_allclose(z.cpu().numpy(), ref["last_logits"], atol=0.05)
    # free-running greedy from the ring (graph replay) matches the oracle's ids
    sess.reset()
    sess.prefill(prompt, logits=z, next_ids=nxt)
    free = [nxt.cpu().numpy().copy()]
    for t in range(steps):
        sess.decode(None, logits=z, next_ids=nxt)
        free.append(nxt.cpu().numpy().copy())
    free = np.stack(free)
    for b in range(B):
        mism = np.nonzero(free[:, b] != ref["ids"][:, b])[0]
        if len(mism):
            assert ref["margins"][mism[0], b] <= 1e-2, (b, mism[0], ref["margins"][mism[0], b])
    st, flags = model.sync_status()
    assert st == 0, flags
