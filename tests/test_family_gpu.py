"""Family rungs at full width ("N7 · model/forward-parity", Thm 2: the same
forward over the family axes): the Qwen3-8B shape (per-head QK-norm in a
pre-norm layer, RoPE base 1e6, untied 151936-word head) and the Mistral-7B
shape (a sliding window on every layer), each as a two-layer slice of the
full-width model against the exact oracle. Both run with f16 activation
storage and meet the forward-parity gates: hidden cosine >= 0.9999 at every slot
and position, logits within 0.05, argmax exact where the oracle's top-1/top-2
margin exceeds 1e-2. The Mistral slice shrinks the window to 256 so that a
600-token prefill in chunks of 128 makes it non-vacuous and wraps the
sliding-window ring (256 + 127 -> 384 positions), then decodes past it.
"""
import gc

import numpy as np
import pytest

import oracle
import synth
from helpers import cosine, weights_to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
MARGIN = 1e-2
F16_ALL = 0x3F


def _free():
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _worst_cos(h, href):
    return min(cosine(h[l, s], href[l, s]) for l in range(h.shape[0]) for s in range(h.shape[1]))


def test_qwen3_8b_two_layer_slice(fk):
    import torch
    cfg = synth.CONFIGS["qwen3-8b"].with_(n_layers=2, f16_sites=F16_ALL)
    wb = synth.make_weights(cfg, norm_mode="random")  # QK-norm weights away from 1 so their indexing shows
    ids = synth.make_ids(cfg, 1, 300, stream=21)
    ref = oracle.forward(cfg, wb, ids, hidden=True, logits="all")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=300)
    out = model.forward(ids)
    torch.cuda.synchronize()
    h = out["hidden"].view(cfg.n_layers + 2, 300, cfg.hidden).cpu().numpy()
    z = out["logits"].view(300, cfg.vocab).cpu().numpy()
    cos = _worst_cos(h, ref["hidden"][:, 0])
    dz = float(np.max(np.abs(z - ref["logits"][0])))
    print(f"qwen3-8b 2-layer slice (f16 storage): worst cosine {cos:.6f}, logits max|d| {dz:.4f}")
    assert cos >= 0.9999 and dz <= 0.05
    decided = oracle.top2_margin(ref["logits"][0]) > MARGIN
    np.testing.assert_array_equal(out["argmax"].cpu().numpy()[decided], oracle.argmax_first(ref["logits"][0])[decided])
    st, flags = model.sync_status()
    assert st == 0, flags
    del model, out
    _free()


def test_mistral_7b_two_layer_slice_ring(fk):
    import torch
    cfg = synth.CONFIGS["mistral-7b"].with_(n_layers=2, layer_kinds=(1, 1), sliding_window=256, f16_sites=F16_ALL)
    wb = synth.make_weights(cfg, norm_mode="random")
    prompt = synth.make_ids(cfg, 1, 600, stream=22)
    steps = 8
    ref = oracle.greedy(cfg, wb, prompt, steps)
    full = oracle.forward(cfg, wb, prompt, hidden=True, logits="none")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=700)
    out = model.forward(prompt, hidden=True, logits=False, argmax=False)
    torch.cuda.synchronize()
    h = out["hidden"].view(cfg.n_layers + 2, 600, cfg.hidden).cpu().numpy()
    cos = _worst_cos(h, full["hidden"][:, 0])
    sess = model.session(1, 600 + steps + 1, max_chunk=128)
    z = torch.empty((1, cfg.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.empty((1,), dtype=torch.int32, device="cuda")
    sess.prefill(prompt, logits=z, next_ids=nxt)
    torch.cuda.synchronize()
    dz = [float(np.max(np.abs(z.cpu().numpy() - ref["first_logits"])))]
    got = [int(nxt.item())]
    for t in range(steps):
        sess.decode(torch.tensor(ref["ids"][t].astype(np.int32), device="cuda"), logits=z, next_ids=nxt)
        got.append(int(nxt.item()))
    dz.append(float(np.max(np.abs(z.cpu().numpy() - ref["last_logits"]))))
    print(f"mistral-7b 2-layer slice (window 256, f16 storage): worst cosine {cos:.6f}, "
          f"prefill/last decode logits max|d| {dz[0]:.4f}/{dz[1]:.4f}")
    assert cos >= 0.9999 and max(dz) <= 0.05
    decided = ref["margins"][:, 0] > MARGIN
    np.testing.assert_array_equal(np.array(got)[decided], ref["ids"][:, 0][decided])
    st, flags = model.sync_status()
    assert st == 0, flags
    del model, out, sess
    _free()
