"""Failure detection on the host, without a GPU.

Every rejected call must return its status before anything reaches a device:
the config rules of "pegainfer issue #878", Proposed Plan (geometry validated
at parse, the final-logit softcap validated positive, a parsed layer map), and
the stub contract of "N9 · metalgemm", Thm 2 (no device -> a clear status, no
fallback path).
"""
import ctypes
import math

import pytest

import synth


def _lib():
    import transformer_decoder_forward_bf16_gb300 as fk
    return fk, fk.load()


def _bad_configs():
    base = synth.small_config("gemma")
    moe = synth.small_config("moe")
    return [
        ("softcap negative", base.with_(final_softcap=-1.0), "final_softcap"),
        ("softcap nan", base.with_(final_softcap=math.nan), "final_softcap"),
        ("softcap inf", base.with_(final_softcap=math.inf), "final_softcap"),
        ("layer kind 2", base.with_(layer_kinds=(1, 2, 0)), "layer_kinds"),
        ("local layer without window", base.with_(sliding_window=0), "sliding_window"),
        ("head_dim 96", base.with_(head_dim=96, hidden=192), "head_dim"),
        ("gqa indivisible", base.with_(n_q_heads=3, n_kv_heads=2), "multiple of n_kv_heads"),
        ("group over 8", base.with_(n_q_heads=18, n_kv_heads=2), "8 query heads"),
        ("hidden not multiple of 64", base.with_(hidden=200), "hidden"),
        ("intermediate not multiple of 64", base.with_(intermediate=500), "intermediate"),
        ("vocab not multiple of 8", base.with_(vocab=1001), "vocab"),
        ("rms_eps zero", base.with_(rms_eps=0.0), "rms_eps"),
        ("theta <= 1", base.with_(rope_theta_local=1.0), "theta"),
        ("llama3 low >= high", synth.small_config("llama3").with_(rope_low_freq_factor=4.0), "llama3"),
        ("zero layers", base.with_(n_layers=0, layer_kinds=()), "n_layers"),
        ("experts not multiple of 8", moe.with_(n_experts=12), "n_experts"),
        ("over 256 experts", moe.with_(n_experts=264), "n_experts"),
        ("k above experts", moe.with_(n_experts_per_tok=9), "n_experts_per_tok"),
        ("k above 16", moe.with_(n_experts=32, n_experts_per_tok=17), "n_experts_per_tok"),
        ("expert width", moe.with_(expert_intermediate=100), "expert_intermediate"),
    ]


@pytest.mark.parametrize("name,cfg,needle", _bad_configs(), ids=[c[0] for c in _bad_configs()])
def test_invalid_config_rejected_before_any_device_work(name, cfg, needle):
    fk, lib = _lib()
    ccfg, kinds = fk.config_to_c(cfg)
    assert lib.fk_model_arena_bytes(ctypes.byref(ccfg), 64) == 0
    assert needle in lib.fk_last_error().decode()
    layers = (fk.FkLayerWeights * max(1, cfg.n_layers))()
    w = fk.FkWeights(embed=None, lm_head=None, final_norm=None, layers=layers)
    h = ctypes.c_void_p()
    st = lib.fk_model_create(ctypes.byref(ccfg), ctypes.byref(w), 64, None, 0, ctypes.byref(h))
    assert st == 2, (st, lib.fk_last_error())  # FK_ERR_INVALID_CONFIG
    assert h.value is None


def test_valid_config_sizes_its_arena():
    fk, lib = _lib()
    for cfg in (synth.small_config("gemma"), synth.CONFIGS["llama3-8b"], synth.CONFIGS["gemma3-tower"],
                synth.small_config("moe"), synth.CONFIGS["qwen3-moe-30b-a3b"]):
        ccfg, kinds = fk.config_to_c(cfg)
        assert lib.fk_model_arena_bytes(ctypes.byref(ccfg), 128) > 0, lib.fk_last_error()


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


@pytest.mark.skipif(not _no_gpu(), reason="checks the no-device status; a GPU is present")
def test_no_device_status_without_gpu():
    """A valid request on a machine without an sm_103 GPU returns
    FK_ERR_NO_DEVICE (the stub contract), never a CPU fallback. The fake
    device pointers below are never dereferenced: the device check comes
    first."""
    fk, lib = _lib()
    cfg = synth.small_config("llama")
    ccfg, kinds = fk.config_to_c(cfg)
    fake = 0x7f0000000000
    layers = (fk.FkLayerWeights * cfg.n_layers)()
    for l in range(cfg.n_layers):
        for f, _ in fk.FkLayerWeights._fields_:
            setattr(layers[l], f, fake)
    w = fk.FkWeights(embed=fake, lm_head=None, final_norm=fake, layers=layers)
    need = lib.fk_model_arena_bytes(ctypes.byref(ccfg), 64)
    h = ctypes.c_void_p()
    st = lib.fk_model_create(ctypes.byref(ccfg), ctypes.byref(w), 64, fake, need, ctypes.byref(h))
    assert st == 5, (st, lib.fk_last_error())  # FK_ERR_NO_DEVICE
    assert lib.fk_gemm_bf16(fake, fake, 16, 64, 64, fake, 1, None) == 5
    assert lib.fk_gemm_bf16_splitk_noalloc(fake, fake, 1, 64, 64, fake, 1, None) == 5
    assert lib.fk_attention_decode(fake, fake, fake, 1, 4, 1, 64, 64, 10, 0, fake, None) == 5
    assert lib.fk_debug_set_op_pipe_fault(0, 0) == 5


def test_bad_arguments_rejected_on_host():
    fk, lib = _lib()
    fake = 0x7f0000000000
    # shape and alignment rules are checked before the device is touched
    assert lib.fk_gemm_bf16(fake, fake, 16, 12, 64, fake, 1, None) == 1      # K % 8
    assert lib.fk_gemm_bf16(fake + 8, fake, 16, 64, 64, fake, 1, None) == 1  # misaligned
    assert lib.fk_gemm_bf16(None, fake, 16, 64, 64, fake, 1, None) == 1
    assert lib.fk_attention_decode(fake, fake, fake, 1, 4, 1, 96, 64, 10, 0, fake, None) == 1   # head_dim
    assert lib.fk_attention_decode(fake, fake, fake, 1, 4, 1, 64, 64, 65, 0, fake, None) == 1   # ctx > cap
    assert lib.fk_attention_decode(fake, fake, fake, 1, 3, 2, 64, 64, 10, 0, fake, None) == 1   # GQA
    assert lib.fk_attention_prefill(fake, fake, fake, 1, 10, 0, 4, 1, 64, 60, 0, fake, None) == 1  # cap % 64
    assert lib.fk_debug_set_op_pipe_fault(0, -1) == 1


def test_moe_arena_counts_expert_f16_copies():
    """With f16 FFN sites, the arena holds f16 copies of the router and of
    every expert matrix of each MoE layer (and only the dense FFN of dense
    layers)."""
    fk, lib = _lib()
    cfg = synth.small_config("moe")  # layers: dense, MoE, MoE
    def arena(c):
        ccfg, bufs = fk.config_to_c(c)
        n = lib.fk_model_arena_bytes(ctypes.byref(ccfg), 128)
        assert n > 0, lib.fk_last_error()
        return n
    a0 = arena(cfg.with_(f16_sites=0))
    a1 = arena(cfg.with_(f16_sites=fk.F16_FFN_IN | fk.F16_FFN_ACT))
    H, I, E, Ie = cfg.hidden, cfg.intermediate, cfg.n_experts, cfg.expert_intermediate
    al = lambda b: (b + 255) // 256 * 256
    dense = 3 * al(I * H * 2)
    per_moe = al(E * H * 2) + 3 * al(E * Ie * H * 2)
    assert a1 - a0 == dense + 2 * per_moe


def test_moe_layer_map_without_experts_rejected():
    fk, lib = _lib()
    cfg = synth.small_config("gemma")
    ccfg, bufs = fk.config_to_c(cfg)
    marks = (ctypes.c_uint8 * cfg.n_layers)(*([1] * cfg.n_layers))
    ccfg.moe_layers = ctypes.cast(marks, ctypes.c_void_p)
    assert lib.fk_model_arena_bytes(ctypes.byref(ccfg), 64) == 0
    assert "n_experts is 0" in lib.fk_last_error().decode()
