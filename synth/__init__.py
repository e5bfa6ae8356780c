"""Seeded synthetic inputs shared by the CPU oracle, the tests and the benchmark.

This module generates inputs only: model shapes, bf16 weight bits and token
ids. It holds none of the forward pass's arithmetic (no norm, no projection, no
attention, no scale), so that the oracle and the CUDA library, which both
consume its output, stay independent of each other.

The generator is counter-based (splitmix64 finaliser + Box-Muller, defined in
``_gen.c``), so any tensor or any slice of it can be regenerated from
``(seed, stream, index)`` alone, on any machine, with any thread count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import ModelConfig, CONFIGS, small_config, tiny_config  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "_gen.c")
_LIB_PATH = os.path.join(_HERE, "_gen.so")
_lib = None
_lock = threading.Lock()

# Default seeds follow the test seeds that "N9 · metalgemm", Thm 1 reports:
# 7 for its random source, 99 and 0x1234567 for its LCG-generated inputs.
SEED_WEIGHTS = 7
SEED_IDS = 99
SEED_GEMM_X = 0x1234567


def build(force: bool = False) -> str:
    """Compile the generator with gcc into ``synth/_gen.so`` (host code only)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                         ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.synth_normal.restype = None
            lib.synth_uniform_ids.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                              ctypes.c_void_p]
            lib.synth_uniform_ids.restype = None
            lib.synth_words.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
            lib.synth_words.restype = None
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, stream: int, shape, sigma: float, mean: float = 0.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, sigma^2) samples, RNE-rounded."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal(seed, stream, n, sigma, mean, out.ctypes.data, None, _threads())
    return out.reshape(shape)


def normal_f32(seed: int, stream: int, shape, sigma: float, mean: float = 0.0) -> np.ndarray:
    """The same samples as :func:`normal_bf16`, before the bf16 rounding."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    out = np.empty(n, dtype=np.float32)
    if n:
        _load().synth_normal(seed, stream, n, sigma, mean, None, out.ctypes.data, _threads())
    return out.reshape(shape)


def uniform_ids(seed: int, stream: int, shape, vocab: int) -> np.ndarray:
    """Token ids uniform in [0, vocab), int32."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_uniform_ids(seed, stream, n, vocab, out.ctypes.data)
    return out.reshape(shape)


def words(seed: int, stream: int, n: int) -> np.ndarray:
    """Raw 64-bit generator words (for tests of the generator itself)."""
    out = np.empty(n, dtype=np.uint64)
    if n:
        _load().synth_words(seed, stream, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: bf16 is the top half of f32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, nearest with ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# ---------------------------------------------------------------------------
# Model weights
# ---------------------------------------------------------------------------
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "post_attn_norm",
                 "ffn_norm", "w_gate", "w_up", "w_down", "post_ffn_norm")
NORM_TENSORS = ("attn_norm", "q_norm", "k_norm", "post_attn_norm", "ffn_norm", "post_ffn_norm")
MOE_TENSORS = ("router", "expert_gate", "expert_up", "expert_down")


def tensor_stream(name: str) -> int:
    """Fixed stream id per weight tensor, so each tensor is reproducible alone."""
    if name == "embed":
        return 1
    if name == "lm_head":
        return 2
    if name == "final_norm":
        return 3
    layer, t = name.split(".", 1)
    if t in MOE_TENSORS:
        return 1_000_000 + 8 * int(layer[1:]) + MOE_TENSORS.index(t)
    return 16 + 16 * int(layer[1:]) + LAYER_TENSORS.index(t)


def weight_shapes(cfg: ModelConfig) -> dict:
    """Shapes of every tensor the model reads (row-major, [out, in] for matrices)."""
    H, hd = cfg.hidden, cfg.head_dim
    shapes = {"embed": (cfg.vocab, H), "final_norm": (H,)}
    if not cfg.tied:
        shapes["lm_head"] = (cfg.vocab, H)
    for l in range(cfg.n_layers):
        p = f"L{l}."
        shapes[p + "attn_norm"] = (H,)
        shapes[p + "wq"] = (cfg.n_q_heads * hd, H)
        shapes[p + "wk"] = (cfg.n_kv_heads * hd, H)
        shapes[p + "wv"] = (cfg.n_kv_heads * hd, H)
        shapes[p + "wo"] = (H, cfg.n_q_heads * hd)
        shapes[p + "ffn_norm"] = (H,)
        if cfg.moe_kinds()[l]:
            E, Ie = cfg.n_experts, cfg.expert_intermediate
            shapes[p + "router"] = (E, H)
            shapes[p + "expert_gate"] = (E, Ie, H)
            shapes[p + "expert_up"] = (E, Ie, H)
            shapes[p + "expert_down"] = (E, H, Ie)
        else:
            shapes[p + "w_gate"] = (cfg.intermediate, H)
            shapes[p + "w_up"] = (cfg.intermediate, H)
            shapes[p + "w_down"] = (H, cfg.intermediate)
        if cfg.qk_norm:
            shapes[p + "q_norm"] = (hd,)
            shapes[p + "k_norm"] = (hd,)
        if cfg.norm_layout == "sandwich":
            shapes[p + "post_attn_norm"] = (H,)
            shapes[p + "post_ffn_norm"] = (H,)
    return shapes


def make_tensor(cfg: ModelConfig, name: str, seed: int = SEED_WEIGHTS, sigma: float = 0.02,
                norm_mode: str = "ones") -> np.ndarray:
    """One weight tensor as bf16 bits. Matrices are N(0, sigma^2); norm weights
    are 1.0 (``norm_mode="ones"``, the configs' setting) or 1 + N(0, 0.1^2)
    (``"random"``, used by small tests so that indexing mistakes show)."""
    shape = weight_shapes(cfg)[name]
    base = name.split(".")[-1]
    if base in NORM_TENSORS or base == "final_norm":
        if norm_mode == "ones":
            return np.full(shape, 0x3F80, dtype=np.uint16)
        return normal_bf16(seed, tensor_stream(name), shape, 0.1, 1.0)
    return normal_bf16(seed, tensor_stream(name), shape, sigma)


def make_weights(cfg: ModelConfig, seed: int = SEED_WEIGHTS, sigma: float = 0.02,
                 norm_mode: str = "ones") -> dict:
    """All weights of ``cfg`` as a dict name -> uint16 array of bf16 bits."""
    return {n: make_tensor(cfg, n, seed, sigma, norm_mode) for n in weight_shapes(cfg)}


def make_ids(cfg: ModelConfig, batch: int, seq: int, seed: int = SEED_IDS, stream: int = 0) -> np.ndarray:
    """Token ids uniform in [0, vocab), shape [batch, seq], int32."""
    return uniform_ids(seed, 1000 + stream, (batch, seq), cfg.vocab)
