"""Device forward vs the float64 oracle ("N7 · model/forward-parity", Thm 1:
hidden-state cosine >= 0.9999 at every slot, last-position logit max|Δ| <=
0.05, per-position argmax equal to the oracle's wherever the oracle's
top-1/top-2 margin exceeds 1e-2; Thm 2 family axes through the small
llama3 and Gemma-style models)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import cosine, weights_to_dev

pytestmark = pytest.mark.gpu

MARGIN = 1e-2


def check_forward(fk, cfg, B, S, norm_mode="ones", sigma=0.02, seed=7):
    import torch
    wb = synth.make_weights(cfg, seed=seed, sigma=sigma, norm_mode=norm_mode)
    ids = synth.make_ids(cfg, B, S, seed=99)
    dev = weights_to_dev(wb)
    model = fk.Model(cfg, dev, max_positions=max(S, 16))
    out = model.forward(ids)
    torch.cuda.synchronize()
    st, flags = model.sync_status()
    assert st == 0, flags
    ref = oracle.forward(cfg, wb, ids)
    hid = out["hidden"].cpu().numpy().reshape(cfg.n_layers + 2, B, S, cfg.hidden)
    worst = min(cosine(hid[l, b, s], ref["hidden"][l, b, s])
                for l in range(cfg.n_layers + 2) for b in range(B) for s in range(S))
    assert worst >= 0.9999, worst
    z = out["logits"].cpu().numpy().reshape(B, S, cfg.vocab)
    zr = ref["logits"]
    last = np.max(np.abs(z[:, -1] - zr[:, -1]))
    assert last <= 0.05, last
    am = out["argmax"].cpu().numpy().reshape(B, S)
    margin = oracle.top2_margin(zr)
    decided = margin > MARGIN
    np.testing.assert_array_equal(am[decided], oracle.argmax_first(zr)[decided])
    # the argmax kernel itself: exact on the device's own logits
    np.testing.assert_array_equal(am, np.argmax(z, axis=-1))
    return {"worst_cos": worst, "last_maxabs": float(last), "decided": float(decided.mean()),
            "logit_err": float(np.max(np.abs(z - zr)))}


SMALL_KINDS = {
    "llama": synth.small_config("llama"),
    "llama3": synth.small_config("llama3"),
    "gemma": synth.small_config("gemma"),
    # sliding window on a head_dim-64 model (the tensor-core prefill attention path)
    "llama-window": synth.small_config("llama", sliding_window=24, layer_kinds=(1, 0)),
    "llama3-window": synth.small_config("llama3", sliding_window=40, layer_kinds=(0, 1)),
    # family rungs: QK-norm in a pre-norm layer (Qwen3), a window on every layer (Mistral)
    "qwen3": synth.small_config("qwen3"),
    "mistral": synth.small_config("mistral"),
}


@pytest.mark.parametrize("kind", sorted(SMALL_KINDS))
@pytest.mark.parametrize("B,S", [(1, 9), (2, 70), (1, 130), (2, 300)])
def test_small_models(fk, kind, B, S):
    cfg = SMALL_KINDS[kind]
    r = check_forward(fk, cfg, B, S, norm_mode="random", sigma=0.02)
    print(kind, B, S, r)


def test_wide_model_k_split_tail(fk):
    """A narrow residual stream with wide projections (Q|K|V 10240 and gate/up
    2 x 20480 outputs over K = 256) at 2 x 1000 tokens: the Q|K|V and gate/up
    GEMMs run 256 x 256 tiles several waves deep with a ragged last row block,
    and attention has 64 query heads over 8 KV heads; every hidden slot
    against the oracle."""
    cfg = synth.small_config("llama3", hidden=256, n_q_heads=64, n_kv_heads=8, head_dim=128, intermediate=20480)
    r = check_forward(fk, cfg, 2, 1000, norm_mode="random", sigma=0.02)
    print(r)


def test_forward_graph_replay(fk):
    """A cacheless forward of few tokens runs eagerly the first time, is
    captured into a CUDA graph the second time it is called with the same
    shape, workspace and outputs, and is replayed after that: every call,
    including ones with new ids, gives the eager result bit for bit."""
    import torch
    cfg = synth.small_config("llama3")
    wb = synth.make_weights(cfg, norm_mode="random", sigma=0.02)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    lib = fk.load()
    B, S = 2, 9
    T = B * S
    wsb = lib.fk_forward_workspace_bytes(model.handle, B, S)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    hid = torch.empty((cfg.n_layers + 2, T, cfg.hidden), dtype=torch.float32, device="cuda")
    z = torch.empty((T, cfg.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty((T,), dtype=torch.int32, device="cuda")

    def run(ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        st = fk.fk_forward(model.handle, ids.ctypes.data, 0, B, S, ws.data_ptr(), wsb, hid.data_ptr(), z.data_ptr(),
                           am.data_ptr(), 0, 0)
        assert st == 0, fk.load().fk_last_error()
        torch.cuda.synchronize()
        return hid.clone(), z.clone(), am.clone()

    ids_a = synth.make_ids(cfg, B, S, seed=99)
    ids_b = synth.make_ids(cfg, B, S, seed=5)
    ref_a = model.forward(ids_a)  # another workspace and outputs: launched one by one
    ref_b = model.forward(ids_b)
    torch.cuda.synchronize()
    for ids, ref in ((ids_a, ref_a), (ids_a, ref_a), (ids_a, ref_a), (ids_b, ref_b), (ids_a, ref_a)):
        h, zz, a = run(ids)  # eager, captured, then replayed
        assert torch.equal(h.view(-1), ref["hidden"].view(-1))
        assert torch.equal(zz, ref["logits"])
        assert torch.equal(a, ref["argmax"])
    st, flags = model.sync_status()
    assert st == 0, flags


def test_forward_graph_cache_many_keys(fk):
    """Five forward shapes called in turn, more than the graphs the model
    keeps: keys are remembered, captured, replayed and replaced in least
    recently used order, and every call equals its eager result bit for bit."""
    import torch
    cfg = synth.small_config("llama")
    wb = synth.make_weights(cfg, norm_mode="random", sigma=0.02)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    lib = fk.load()
    shapes = [(1, 5), (2, 9), (1, 17), (3, 4), (2, 21)]
    bufs = {}
    refs = {}
    for B, S in shapes:
        T = B * S
        wsb = lib.fk_forward_workspace_bytes(model.handle, B, S)
        bufs[(B, S)] = (torch.empty(wsb, dtype=torch.uint8, device="cuda"),
                        torch.empty((T, cfg.vocab), dtype=torch.float32, device="cuda"),
                        torch.empty((T,), dtype=torch.int32, device="cuda"))
        ids = synth.make_ids(cfg, B, S, seed=B * 100 + S)
        refs[(B, S)] = (ids, model.forward(ids, hidden=False))
    torch.cuda.synchronize()
    for rnd in range(4):
        for B, S in (shapes if rnd % 2 == 0 else shapes[::-1]):
            ws, z, am = bufs[(B, S)]
            ids, ref = refs[(B, S)]
            ids = np.ascontiguousarray(ids, dtype=np.int32)
            st = fk.fk_forward(model.handle, ids.ctypes.data, 0, B, S, ws.data_ptr(), ws.numel(), 0, z.data_ptr(),
                               am.data_ptr(), 0, 0)
            assert st == 0, lib.fk_last_error()
            torch.cuda.synchronize()
            assert torch.equal(z, ref["logits"]), (rnd, B, S)
            assert torch.equal(am, ref["argmax"]), (rnd, B, S)


def test_smollm2_shape_9_tokens(fk):
    """The SmolLM2-135M-shaped llama, one sequence of 9 ids, norm weights 1.0."""
    r = check_forward(fk, synth.CONFIGS["smollm2-135m"], 1, 9)
    print(r)


def test_bitwise_replay(fk):
    import torch
    cfg = synth.small_config("gemma")
    wb = synth.make_weights(cfg, norm_mode="random", sigma=0.02)
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    ids = synth.make_ids(cfg, 2, 40)
    a = model.forward(ids)
    b = model.forward(ids)
    torch.cuda.synchronize()
    for k in ("hidden", "logits", "argmax"):
        assert torch.equal(a[k], b[k]), k


def test_token_range_rejected_on_host(fk):
    cfg = synth.small_config("llama")
    model = fk.Model(cfg, weights_to_dev(synth.make_weights(cfg)), max_positions=16)
    ids = synth.make_ids(cfg, 1, 5)
    ids[0, 3] = cfg.vocab
    with pytest.raises(fk.FkError) as ei:
        model.forward(ids)
    assert ei.value.status == 3


def test_token_range_flagged_on_device(fk):
    import torch
    cfg = synth.small_config("llama")
    model = fk.Model(cfg, weights_to_dev(synth.make_weights(cfg)), max_positions=16)
    ids = torch.tensor([[1, 2, cfg.vocab + 5, 3]], dtype=torch.int32, device="cuda")
    model.forward(ids)
    st, flags = model.sync_status()
    assert st == 7 and flags & fk.DEVERR_TOKEN_RANGE
    st, flags = model.sync_status()
    assert st == 0 and flags == 0


# f16 activation storage: every site alone (the plumbing of each storage point:
# a kernel that read or wrote a site in the wrong 16-bit format would fail the
# cosine gate by far), then all sites together
F16_SITES = {"qkv_in": 0x1, "attn": 0x2, "o_in": 0x4, "ffn_in": 0x8, "ffn_act": 0x10, "head_in": 0x20, "all": 0x3F}


@pytest.mark.parametrize("site", sorted(F16_SITES))
@pytest.mark.parametrize("kind", ["llama3", "gemma"])
def test_small_models_f16_storage(fk, kind, site):
    cfg = SMALL_KINDS[kind].with_(f16_sites=F16_SITES[site])
    r = check_forward(fk, cfg, 2, 70, norm_mode="random", sigma=0.02)
    print(kind, site, r)


@pytest.mark.parametrize("kind", ["llama", "llama-window", "llama3-window"])
def test_small_models_f16_storage_all_sites(fk, kind):
    cfg = SMALL_KINDS[kind].with_(f16_sites=F16_SITES["all"])
    for B, S in ((1, 9), (2, 130)):
        check_forward(fk, cfg, B, S, norm_mode="random", sigma=0.02)
