"""KV-cached session ("N7", Thm 1: cached Prefill last-position logits agree
with the cacheless Forward within 1e-4; greedy ids token-for-token)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import weights_to_dev

pytestmark = pytest.mark.gpu


def _setup(fk, cfg, norm_mode="random", sigma=0.05):
    wb = synth.make_weights(cfg, norm_mode=norm_mode, sigma=sigma)
    return wb, fk.Model(cfg, weights_to_dev(wb), max_positions=512)


@pytest.mark.parametrize("kind", ["llama", "llama3", "gemma"])
def test_cached_prefill_matches_cacheless(fk, kind):
    import torch
    cfg = synth.small_config(kind)
    wb, model = _setup(fk, cfg)
    B, S = 2, 100
    ids = synth.make_ids(cfg, B, S)
    full = model.forward(ids, hidden=False)
    sess = model.session(B, 256, max_chunk=48)  # three chunks
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
