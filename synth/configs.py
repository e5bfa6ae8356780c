"""Model shapes of the synthetic workloads (data only, no arithmetic).

Each field mirrors one axis of the decoder forward pass described on the pages:
the llama family (SmolLM2-135M shape), llama3 with RoPE scaling, and the
Gemma3-style local/global tower with QK-norm, sandwich norms, a GELU-gated FFN,
a scaled embedding and a final-logit softcap.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta_global: float = 10000.0
    rope_theta_local: float = 10000.0
    rope_scaling: str = "none"          # "none" | "llama3"
    rope_factor: float = 1.0
    rope_low_freq_factor: float = 1.0
    rope_high_freq_factor: float = 4.0
    rope_orig_max_pos: int = 8192
    act: str = "silu"                   # "silu" | "gelu_tanh"
    norm_layout: str = "pre"            # "pre" | "sandwich"
    qk_norm: bool = False
    sliding_window: int = 0             # 0 = no local layers
    layer_kinds: tuple = field(default=())  # per layer: 0 = global, 1 = local (empty = all global)
    embed_scale: str = "none"           # "none" | "sqrt_hidden_bf16"
    final_softcap: float = 0.0          # 0 = off
    tied: bool = True
    f16_sites: int = 0                  # activation storage sites kept as IEEE f16 (bit mask; 0 = all bf16)
    # mixture-of-experts FFN (0 experts = dense FFN on every layer)
    n_experts: int = 0
    n_experts_per_tok: int = 0          # k experts per token
    expert_intermediate: int = 0        # FFN width of one expert
    norm_topk: bool = True              # renormalise the k routing weights to sum 1
    moe_layers: tuple = field(default=())  # per layer: 1 = MoE FFN, 0 = dense (empty = all MoE if n_experts)

    def kinds(self) -> tuple:
        return self.layer_kinds if self.layer_kinds else (0,) * self.n_layers

    def moe_kinds(self) -> tuple:
        if not self.n_experts:
            return (0,) * self.n_layers
        return self.moe_layers if self.moe_layers else (1,) * self.n_layers

    def with_(self, **kw) -> "ModelConfig":
        return replace(self, **kw)


def _gemma_kinds(n_layers: int, period: int = 6) -> tuple:
    # five local layers then one global, repeating: layer l is global iff (l+1) % 6 == 0
    return tuple(0 if (l + 1) % period == 0 else 1 for l in range(n_layers))


SMOLLM2_135M = ModelConfig(
    name="smollm2-135m", n_layers=30, hidden=576, n_q_heads=9, n_kv_heads=3, head_dim=64,
    intermediate=1536, vocab=49152, rms_eps=1e-5, rope_theta_global=100000.0,
    rope_theta_local=100000.0, tied=True)

LLAMA3_8B = ModelConfig(
    name="llama3-8b", n_layers=32, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
    intermediate=14336, vocab=128256, rms_eps=1e-5, rope_theta_global=500000.0,
    rope_theta_local=500000.0, rope_scaling="llama3", rope_factor=8.0, rope_low_freq_factor=1.0,
    rope_high_freq_factor=4.0, rope_orig_max_pos=8192, tied=False)

GEMMA3_TOWER = ModelConfig(
    name="gemma3-tower", n_layers=48, hidden=3840, n_q_heads=16, n_kv_heads=8, head_dim=256,
    intermediate=15360, vocab=262144, rms_eps=1e-6, rope_theta_global=1000000.0,
    rope_theta_local=10000.0, act="gelu_tanh", norm_layout="sandwich", qk_norm=True,
    sliding_window=1024, layer_kinds=_gemma_kinds(48), embed_scale="sqrt_hidden_bf16",
    final_softcap=30.0, tied=True)

# Family shapes of the same kernels ("N7 · model/forward-parity", Thm 2 family
# rungs): Qwen3 puts a per-head RMSNorm on q and k before RoPE in a pre-norm
# layer; Mistral attends through a sliding window on every layer.
QWEN3_8B = ModelConfig(
    name="qwen3-8b", n_layers=36, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
    intermediate=12288, vocab=151936, rms_eps=1e-6, rope_theta_global=1000000.0,
    rope_theta_local=1000000.0, qk_norm=True, tied=False)

MISTRAL_7B = ModelConfig(
    name="mistral-7b", n_layers=32, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
    intermediate=14336, vocab=32000, rms_eps=1e-5, rope_theta_global=10000.0, rope_theta_local=10000.0,
    sliding_window=4096, layer_kinds=(1,) * 32, tied=False)

# Mixture-of-experts rung ("N7", Thm 2: qwen3moe): the Qwen3-30B-A3B geometry,
# 128 experts of width 768 per layer, 8 routed per token, softmax routing
# renormalised over the chosen 8.
QWEN3_MOE_30B = ModelConfig(
    name="qwen3-moe-30b-a3b", n_layers=48, hidden=2048, n_q_heads=32, n_kv_heads=4, head_dim=128,
    intermediate=6144, vocab=151936, rms_eps=1e-6, rope_theta_global=1000000.0, rope_theta_local=1000000.0,
    qk_norm=True, tied=False, n_experts=128, n_experts_per_tok=8, expert_intermediate=768, norm_topk=True)

CONFIGS = {c.name: c for c in (SMOLLM2_135M, LLAMA3_8B, GEMMA3_TOWER, QWEN3_8B, MISTRAL_7B, QWEN3_MOE_30B)}


def tiny_config(kind: str = "llama", **kw) -> ModelConfig:
    """Small models for brute-force checks and fast parity cases."""
    if kind == "llama":
        base = ModelConfig(name="tiny-llama", n_layers=2, hidden=16, n_q_heads=4, n_kv_heads=2,
                           head_dim=4, intermediate=24, vocab=32, rms_eps=1e-5,
                           rope_theta_global=10000.0, rope_theta_local=10000.0)
    elif kind == "llama3":
        base = ModelConfig(name="tiny-llama3", n_layers=2, hidden=32, n_q_heads=4, n_kv_heads=2,
                           head_dim=8, intermediate=40, vocab=48, rms_eps=1e-5,
                           rope_theta_global=500000.0, rope_theta_local=500000.0, rope_scaling="llama3",
                           rope_factor=8.0, rope_low_freq_factor=1.0, rope_high_freq_factor=4.0,
                           rope_orig_max_pos=512, tied=False)
    elif kind == "gemma":
        base = ModelConfig(name="tiny-gemma", n_layers=3, hidden=16, n_q_heads=4, n_kv_heads=2,
                           head_dim=8, intermediate=24, vocab=40, rms_eps=1e-6,
                           rope_theta_global=1000000.0, rope_theta_local=10000.0, act="gelu_tanh",
                           norm_layout="sandwich", qk_norm=True, sliding_window=4,
                           layer_kinds=(1, 1, 0), embed_scale="sqrt_hidden_bf16", final_softcap=30.0)
    elif kind == "moe":
        base = ModelConfig(name="tiny-moe", n_layers=2, hidden=16, n_q_heads=4, n_kv_heads=2, head_dim=4,
                           intermediate=24, vocab=32, rms_eps=1e-6, rope_theta_global=10000.0,
                           rope_theta_local=10000.0, qk_norm=True, tied=False, n_experts=4, n_experts_per_tok=2,
                           expert_intermediate=8, norm_topk=True, moe_layers=(0, 1))
    else:
        raise ValueError(kind)
    return replace(base, **kw)


def small_config(kind: str = "llama", **kw) -> ModelConfig:
    """Small models whose shapes the CUDA kernels accept (head_dim 64/128/256,
    widths multiples of 64), for fast device-vs-oracle parity cases."""
    if kind == "llama":
        base = ModelConfig(name="small-llama", n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=64,
                           intermediate=256, vocab=512, rms_eps=1e-5, rope_theta_global=10000.0,
                           rope_theta_local=10000.0, tied=True)
    elif kind == "llama3":
        base = ModelConfig(name="small-llama3", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=128,
                           intermediate=384, vocab=1024, rms_eps=1e-5, rope_theta_global=500000.0,
                           rope_theta_local=500000.0, rope_scaling="llama3", rope_factor=8.0,
                           rope_low_freq_factor=1.0, rope_high_freq_factor=4.0, rope_orig_max_pos=64, tied=False)
    elif kind == "gemma":
        base = ModelConfig(name="small-gemma", n_layers=3, hidden=256, n_q_heads=2, n_kv_heads=1, head_dim=256,
                           intermediate=512, vocab=1024, rms_eps=1e-6, rope_theta_global=1000000.0,
                           rope_theta_local=10000.0, act="gelu_tanh", norm_layout="sandwich", qk_norm=True,
                           sliding_window=16, layer_kinds=(1, 1, 0), embed_scale="sqrt_hidden_bf16",
                           final_softcap=30.0, tied=True)
    elif kind == "qwen3":
        base = ModelConfig(name="small-qwen3", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                           intermediate=512, vocab=1024, rms_eps=1e-6, rope_theta_global=1000000.0,
                           rope_theta_local=1000000.0, qk_norm=True, tied=False)
    elif kind == "moe":
        # dense, MoE, MoE layers (a hybrid layer map); 8 experts, 2 per token
        base = ModelConfig(name="small-moe", n_layers=3, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                           intermediate=384, vocab=1000, rms_eps=1e-6, rope_theta_global=1000000.0,
                           rope_theta_local=1000000.0, qk_norm=True, tied=False, n_experts=8, n_experts_per_tok=2,
                           expert_intermediate=128, norm_topk=True, moe_layers=(0, 1, 1))
    elif kind == "mistral":
        base = ModelConfig(name="small-mistral", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64,
                           intermediate=384, vocab=1000, rms_eps=1e-5, rope_theta_global=10000.0,
                           rope_theta_local=10000.0, sliding_window=32, layer_kinds=(1, 1), tied=False)
    else:
        raise ValueError(kind)
    return replace(base, **kw)
