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


@pytest.mark.parametrize("kind,chunk", [("llama", 48), ("llama3", 48), ("gemma", 48), ("llama", 45), ("llama3", 37)])
def test_cached_prefill_matches_cacheless(fk, kind, chunk):
    """Chunks of 48 start at positions that are multiples of 8 (the V cache
    takes 16-byte runs); 45 and 37 exercise the unaligned element path."""
    import torch
    cfg = synth.small_config(kind)
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


@pytest.mark.parametrize("kind", ["llama", "llama3", "gemma"])
def test_decode_matches_oracle(fk, kind):
    import torch
    cfg = synth.small_config(kind)
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
