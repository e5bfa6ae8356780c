"""Python binding of libfk, the GB300 (sm_103a) decoder-only transformer forward.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libfk.so`` behind the C ABI declared in ``include/fk.h``. PyTorch
is used here only to own device memory and to name streams. There is no CPU
fallback: if the library or a sm_103 GPU is missing, calls raise.

Low-level functions carry the C names (``fk_forward``, ``fk_session_prefill``
...) and take raw pointers; :class:`Model` and :class:`Session` wrap them for
torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, c_double, c_float, c_int32, c_size_t, c_uint32, c_void_p

from . import build as _build

_lib = None
_lock = threading.Lock()

FK_OK = 0
STATUS = {0: "FK_OK", 1: "FK_ERR_INVALID_ARG", 2: "FK_ERR_INVALID_CONFIG", 3: "FK_ERR_TOKEN_RANGE",
          4: "FK_ERR_CONTEXT_FULL", 5: "FK_ERR_NO_DEVICE", 6: "FK_ERR_CUDA", 7: "FK_ERR_DEVICE_FLAG",
          8: "FK_ERR_TIMEOUT", 9: "FK_ERR_WORKSPACE"}
DEVERR_TOKEN_RANGE = 0x1
DEVERR_PIPE_TIMEOUT = 0x2
DEVERR_EXPERT_IDS = 0x4
# activation storage sites stored as IEEE f16 instead of bf16 (fk_config.f16_sites)
F16_QKV_IN, F16_ATTN, F16_O_IN, F16_FFN_IN, F16_FFN_ACT, F16_HEAD_IN = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20
F16_ALL = 0x3F
F16_SITE_BITS = {"qkv_in": F16_QKV_IN, "attn": F16_ATTN, "o_in": F16_O_IN, "ffn_in": F16_FFN_IN,
                 "ffn_act": F16_FFN_ACT, "head_in": F16_HEAD_IN}


class FkError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")


class FkConfig(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("hidden", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("intermediate", c_int32), ("vocab", c_int32), ("rms_eps", c_float),
                ("rope_theta_global", c_double), ("rope_theta_local", c_double), ("rope_scaling", c_int32),
                ("rope_factor", c_float), ("rope_low_freq_factor", c_float), ("rope_high_freq_factor", c_float),
                ("rope_orig_max_pos", c_int32), ("act", c_int32), ("norm_layout", c_int32), ("qk_norm", c_int32),
                ("sliding_window", c_int32), ("layer_kinds", c_void_p), ("embed_scale", c_int32),
                ("final_softcap", c_float), ("tied", c_int32), ("f16_sites", c_uint32),
                ("n_experts", c_int32), ("n_experts_per_tok", c_int32), ("expert_intermediate", c_int32),
                ("norm_topk", c_int32), ("moe_layers", c_void_p)]


class FkLayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "post_attn_norm",
                                        "ffn_norm", "w_gate", "w_up", "w_down", "post_ffn_norm",
                                        "router", "expert_gate", "expert_up", "expert_down")]


class FkWeights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("lm_head", c_void_p), ("final_norm", c_void_p),
                ("layers", POINTER(FkLayerWeights))]


# name -> (restype, argtypes)
_SIGS = {
    "fk_status_string": (ctypes.c_char_p, [c_int32]),
    "fk_last_error": (ctypes.c_char_p, []),
    "fk_version": (ctypes.c_char_p, []),
    "fk_model_arena_bytes": (c_size_t, [POINTER(FkConfig), c_int32]),
    "fk_model_create": (c_int32, [POINTER(FkConfig), POINTER(FkWeights), c_int32, c_void_p, c_size_t,
                                  POINTER(c_void_p)]),
    "fk_model_free": (None, [c_void_p]),
    "fk_forward_workspace_bytes": (c_size_t, [c_void_p, c_int32, c_int32]),
    "fk_forward": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_size_t, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p]),
    "fk_session_bytes": (c_size_t, [c_void_p, c_int32, c_int32, c_int32]),
    "fk_session_create": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_size_t, POINTER(c_void_p)]),
    "fk_session_free": (None, [c_void_p]),
    "fk_session_prefill": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fk_decode_step": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fk_session_reset": (c_int32, [c_void_p]),
    "fk_session_length": (c_int32, [c_void_p]),
    "fk_sync_status": (c_int32, [c_void_p, c_void_p, c_int32, POINTER(c_uint32)]),
    "fk_gemm_bf16": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p]),
    "fk_gemm_bf16_splitk_scratch_bytes": (c_size_t, [c_int32, c_int32, c_int32]),
    "fk_gemm_bf16_splitk": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                      c_size_t, c_void_p]),
    "fk_attention_prefill": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                       c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "fk_attention_decode": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                      c_int32, c_int32, c_void_p, c_void_p]),
    "fk_gemm_bf16_splitk_noalloc_limit": (c_size_t, []),
    "fk_gemm_bf16_splitk_noalloc": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32,
                                              c_void_p]),
    "fk_debug_set_op_pipe_fault": (c_int32, [c_int32, c_int32]),
    "fk_op_rmsnorm": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_float, c_void_p, c_void_p]),
    "fk_op_rope": (c_int32, [c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32,
                             c_void_p]),
    "fk_op_head_argmax": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fk_op_logsoftmax_topk": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p]),
    "fk_op_moe_route": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p]),
    "fk_op_moe_ffn_workspace_bytes": (c_size_t, [c_void_p, c_int32]),
    "fk_op_moe_ffn": (c_int32, [c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_size_t, c_void_p]),
    "fk_model_set_moe_routing": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32]),
    "fk_profile_enable": (None, [c_int32]),
    "fk_profile_reset": (None, []),
    "fk_profile_count": (c_int32, []),
    "fk_profile_get": (c_int32, [c_int32, POINTER(ctypes.c_char_p), POINTER(ctypes.c_int64), POINTER(c_double)]),
}


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_stale: bool = True):
    """Load libfk.so (building it first if it is missing or older than its
    sources). Raises if it cannot be built or loaded: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_stale and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(f"libfk.so is missing at {_build.LIB_PATH}; run build()")
            lib = ctypes.CDLL(_build.LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != FK_OK:
        raise FkError(status, where, load().fk_last_error().decode())


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


# ---------------------------------------------------------------------------
# raw C entry points, same names as the header
# ---------------------------------------------------------------------------
def fk_gemm_bf16(x_ptr, w_ptr, P, K, N, y_ptr, y_fp32, stream_ptr) -> int:
    return load().fk_gemm_bf16(x_ptr, w_ptr, P, K, N, y_ptr, y_fp32, stream_ptr)


def fk_forward(model_ptr, ids_ptr, ids_on_device, batch, seq, ws_ptr, ws_bytes, hidden_ptr, logits_ptr,
               argmax_ptr, margin_ptr, stream_ptr) -> int:
    return load().fk_forward(model_ptr, ids_ptr, ids_on_device, batch, seq, ws_ptr, ws_bytes, hidden_ptr,
                             logits_ptr, argmax_ptr, margin_ptr, stream_ptr)


def fk_session_prefill(sess_ptr, ids_ptr, ids_on_device, seq, logits_ptr, next_ptr, margin_ptr, stream_ptr) -> int:
    return load().fk_session_prefill(sess_ptr, ids_ptr, ids_on_device, seq, logits_ptr, next_ptr, margin_ptr,
                                     stream_ptr)


def fk_decode_step(sess_ptr, ids_ptr, logits_ptr, next_ptr, margin_ptr, stream_ptr) -> int:
    return load().fk_decode_step(sess_ptr, ids_ptr, logits_ptr, next_ptr, margin_ptr, stream_ptr)


def op_sync_status(stream=None, timeout_ms: int = 10000):
    """Drain `stream`, then read and clear the current device's op-level error
    word (set by the op-level entry points): returns (status, flags)."""
    return fk_sync_status(None, _stream_ptr(stream), timeout_ms)


def fk_sync_status(model_ptr, stream_ptr, timeout_ms):
    flags = c_uint32(0)
    st = load().fk_sync_status(model_ptr, stream_ptr, timeout_ms, ctypes.byref(flags))
    return st, flags.value


# ---------------------------------------------------------------------------
# torch conveniences
# ---------------------------------------------------------------------------
def gemm(x, w, out_fp32: bool = False, out=None, stream=None):
    """Y = X · Wᵀ on the tensor cores (bf16 in, fp32 accumulate)."""
    import torch
    P, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((P, N), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=x.device)
    _check(fk_gemm_bf16(_ptr(x), _ptr(w), P, K, N, _ptr(out), 1 if out_fp32 else 0, _stream_ptr(stream)),
           "fk_gemm_bf16")
    return out


def gemm_splitk(x, w, out_fp32: bool = False, out=None, stream=None):
    """Y = X · Wᵀ for few rows (P <= 64) on the weight-streaming split-K kernel."""
    import torch
    P, K = x.shape
    N = w.shape[0]
    lib = load()
    nbytes = lib.fk_gemm_bf16_splitk_scratch_bytes(P, K, N)
    scratch = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((P, N), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=x.device)
    _check(lib.fk_gemm_bf16_splitk(_ptr(x), _ptr(w), P, K, N, _ptr(out), 1 if out_fp32 else 0, _ptr(scratch),
                                   scratch.numel(), _stream_ptr(stream)), "fk_gemm_bf16_splitk")
    return out


def attention_prefill(q, kcache, vcache, seq: int, pos0: int = 0, window: int = 0, out=None, stream=None):
    """Prefill attention: q [B*seq, Hq*hd]; kcache [B, Hkv, cap, hd]; vcache
    transposed [B, Hkv, hd, cap] (bf16)."""
    import torch
    B, Hkv, cap, hd = kcache.shape
    Hq = q.shape[1] // hd
    if out is None:
        out = torch.empty_like(q)
    _check(load().fk_attention_prefill(_ptr(q), _ptr(kcache), _ptr(vcache), B, seq, pos0, Hq, Hkv, hd, cap, window,
                                       _ptr(out), _stream_ptr(stream)), "fk_attention_prefill")
    return out


def attention_decode(q, kcache, vcache, ctx: int, window: int = 0, out=None, stream=None):
    """One decode-attention step: q [B, Hq*hd], kcache [B, Hkv, cap, hd],
    vcache transposed [B, Hkv, hd, cap] (bf16, cap a multiple of 64)."""
    import torch
    B, Hkv, cap, hd = kcache.shape
    Hq = q.shape[1] // hd
    if out is None:
        out = torch.empty_like(q)
    _check(load().fk_attention_decode(_ptr(q), _ptr(kcache), _ptr(vcache), B, Hq, Hkv, hd, cap, ctx, window,
                                      _ptr(out), _stream_ptr(stream)), "fk_attention_decode")
    return out


def rmsnorm(x, w, eps: float, out=None, stream=None):
    """fk_op_rmsnorm: bf16 RMSNorm(x) * w of fp32 rows x [rows, hidden]."""
    import torch
    rows, hidden = x.shape
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=x.device)
    _check(load().fk_op_rmsnorm(_ptr(x), rows, hidden, _ptr(w), eps, _ptr(out), _stream_ptr(stream)),
           "fk_op_rmsnorm")
    return out


def logsoftmax_topk(z, k: int = 64, logprobs: bool = False, stream=None) -> dict:
    """fk_op_logsoftmax_topk on fp32 logit rows z [rows, vocab]: lse, the top-k
    ids (value descending, ties to the lower id), their log-probabilities and
    optionally the whole log-softmax."""
    import torch
    rows, V = z.shape
    dev = z.device
    out = {"lse": torch.empty((rows,), dtype=torch.float32, device=dev),
           "ids": torch.empty((rows, k), dtype=torch.int32, device=dev),
           "top_logprobs": torch.empty((rows, k), dtype=torch.float32, device=dev),
           "logprobs": torch.empty((rows, V), dtype=torch.float32, device=dev) if logprobs else None}
    _check(load().fk_op_logsoftmax_topk(_ptr(z), rows, V, z.stride(0), k, _ptr(out["lse"]), _ptr(out["ids"]),
                                        _ptr(out["top_logprobs"]), _ptr(out["logprobs"]), _stream_ptr(stream)),
           "fk_op_logsoftmax_topk")
    return out


def moe_route(z, k: int, norm_topk: bool = True, forced=None, stream=None) -> dict:
    """fk_op_moe_route on fp32 router logits z [T, E] (CUDA): expert ids and
    weights [T, k] and the routing margin [T]."""
    import torch
    T, E = z.shape
    dev = z.device
    out = {"ids": torch.empty((T, k), dtype=torch.int32, device=dev),
           "weights": torch.empty((T, k), dtype=torch.float32, device=dev),
           "margin": torch.empty((T,), dtype=torch.float32, device=dev)}
    _check(load().fk_op_moe_route(_ptr(z), T, E, z.stride(0), k, int(norm_topk), _ptr(forced), _ptr(out["ids"]),
                                  _ptr(out["weights"]), _ptr(out["margin"]), _stream_ptr(stream)), "fk_op_moe_route")
    return out


def config_to_c(cfg) -> tuple:
    """Fill an FkConfig from any object with the ModelConfig fields; returns
    (struct, buffers) -- keep the buffers alive while the struct is used."""
    kinds = cfg.kinds() if hasattr(cfg, "kinds") else tuple(cfg.layer_kinds)
    kbuf = (ctypes.c_uint8 * max(1, len(kinds)))(*kinds)
    n_exp = int(getattr(cfg, "n_experts", 0))
    moe = cfg.moe_kinds() if hasattr(cfg, "moe_kinds") else (0,) * cfg.n_layers
    mbuf = (ctypes.c_uint8 * max(1, len(moe)))(*moe)
    c = FkConfig(
        n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
        head_dim=cfg.head_dim, intermediate=cfg.intermediate, vocab=cfg.vocab, rms_eps=cfg.rms_eps,
        rope_theta_global=cfg.rope_theta_global, rope_theta_local=cfg.rope_theta_local,
        rope_scaling={"none": 0, "llama3": 1}[cfg.rope_scaling], rope_factor=cfg.rope_factor,
        rope_low_freq_factor=cfg.rope_low_freq_factor, rope_high_freq_factor=cfg.rope_high_freq_factor,
        rope_orig_max_pos=cfg.rope_orig_max_pos, act={"silu": 0, "gelu_tanh": 1}[cfg.act],
        norm_layout={"pre": 0, "sandwich": 1}[cfg.norm_layout], qk_norm=int(cfg.qk_norm),
        sliding_window=cfg.sliding_window, layer_kinds=ctypes.cast(kbuf, c_void_p) if len(kinds) else None,
        embed_scale={"none": 0, "sqrt_hidden_bf16": 1}[cfg.embed_scale], final_softcap=cfg.final_softcap,
        tied=int(cfg.tied), f16_sites=int(getattr(cfg, "f16_sites", 0)),
        n_experts=n_exp, n_experts_per_tok=int(getattr(cfg, "n_experts_per_tok", 0)),
        expert_intermediate=int(getattr(cfg, "expert_intermediate", 0)),
        norm_topk=int(getattr(cfg, "norm_topk", True)),
        moe_layers=ctypes.cast(mbuf, c_void_p) if n_exp and len(moe) else None)
    return c, (kbuf, mbuf)


class Model:
    """A model bound to device weights (a dict name -> bf16 CUDA tensor, names
    as in ``fk_layer_weights``, prefixed ``L{l}.`` per layer)."""

    def __init__(self, cfg, weights: dict, max_positions: int):
        import torch
        lib = load()
        self.cfg = cfg
        self.weights = weights  # keep the tensors alive: the library borrows them
        self._ccfg, self._kinds = config_to_c(cfg)
        n = cfg.n_layers
        self._layers = (FkLayerWeights * n)()
        for l in range(n):
            for f, _ in FkLayerWeights._fields_:
                t = weights.get(f"L{l}.{f}")
                setattr(self._layers[l], f, _ptr(t) if t is not None else None)
        self._cw = FkWeights(embed=_ptr(weights["embed"]), lm_head=_ptr(weights.get("lm_head")) or None,
                             final_norm=_ptr(weights["final_norm"]), layers=self._layers)
        nbytes = lib.fk_model_arena_bytes(ctypes.byref(self._ccfg), max_positions)
        if nbytes == 0:
            raise FkError(2, "fk_model_arena_bytes", lib.fk_last_error().decode())
        dev = weights["embed"].device
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        h = c_void_p()
        _check(lib.fk_model_create(ctypes.byref(self._ccfg), ctypes.byref(self._cw), max_positions,
                                   _ptr(self.arena), nbytes, ctypes.byref(h)), "fk_model_create")
        self.handle = h.value
        self.max_positions = max_positions
        self._ws = None

    def close(self):
        if self.handle:
            load().fk_model_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, ids, hidden: bool = True, logits: bool = True, argmax: bool = True, margin: bool = False,
                stream=None) -> dict:
        """Cacheless forward over ids [B, S] (numpy/CPU int32 = host ids, CUDA
        int32 tensor = device ids). Returns torch tensors on the device."""
        import numpy as np
        import torch
        lib = load()
        on_dev = isinstance(ids, torch.Tensor) and ids.is_cuda
        if not on_dev:
            ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        B, S = ids.shape
        dev = self.arena.device
        cfg = self.cfg
        T = B * S
        wsb = lib.fk_forward_workspace_bytes(self.handle, B, S)
        if self._ws is None or self._ws.numel() < wsb:
            self._ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        out = {
            "hidden": torch.empty((cfg.n_layers + 2, T, cfg.hidden), dtype=torch.float32, device=dev) if hidden else None,
            "logits": torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev) if logits else None,
            "argmax": torch.empty((T,), dtype=torch.int32, device=dev) if argmax else None,
            "margin": torch.empty((T,), dtype=torch.float32, device=dev) if argmax and margin else None,
        }
        ids_ptr = _ptr(ids) if on_dev else ids.ctypes.data
        _check(fk_forward(self.handle, ids_ptr, 1 if on_dev else 0, B, S, _ptr(self._ws), self._ws.numel(),
                          _ptr(out["hidden"]), _ptr(out["logits"]), _ptr(out["argmax"]), _ptr(out["margin"]),
                          _stream_ptr(stream)),
               "fk_forward")
        return out

    def rope(self, layer: int, qkv, batch: int, seq: int, pos0: int, kcache, vcache, stream=None):
        """fk_op_rope: [QK-norm and] RoPE of layer `layer` on qkv rows in
        place; k and transposed v written into the caches."""
        cap = kcache.shape[2]
        _check(load().fk_op_rope(self.handle, layer, _ptr(qkv), batch, seq, pos0, _ptr(kcache), _ptr(vcache), cap,
                                 _stream_ptr(stream)), "fk_op_rope")

    def head_argmax(self, u, margin: bool = True, stream=None) -> dict:
        """fk_op_head_argmax: logits (after the softcap), argmax and top-2
        margin of final-norm rows u [rows, hidden] (bf16)."""
        import torch
        rows = u.shape[0]
        dev = u.device
        out = {"logits": torch.empty((rows, self.cfg.vocab), dtype=torch.float32, device=dev),
               "argmax": torch.empty((rows,), dtype=torch.int32, device=dev),
               "margin": torch.empty((rows,), dtype=torch.float32, device=dev) if margin else None}
        _check(load().fk_op_head_argmax(self.handle, _ptr(u), rows, _ptr(out["logits"]), _ptr(out["argmax"]),
                                        _ptr(out["margin"]), _stream_ptr(stream)), "fk_op_head_argmax")
        return out

    def moe_ffn(self, layer: int, u, forced=None, stream=None) -> dict:
        """fk_op_moe_ffn: the MoE FFN of `layer` on u [T, hidden] (16-bit):
        output fp32 [T, hidden], routing ids [T, k] and margins [T]."""
        import torch
        lib = load()
        T = u.shape[0]
        dev = u.device
        k = self.cfg.n_experts_per_tok
        wsb = lib.fk_op_moe_ffn_workspace_bytes(self.handle, T)
        if wsb == 0:
            raise FkError(1, "fk_op_moe_ffn_workspace_bytes", lib.fk_last_error().decode())
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        out = {"out": torch.empty((T, self.cfg.hidden), dtype=torch.float32, device=dev),
               "ids": torch.empty((T, k), dtype=torch.int32, device=dev),
               "margin": torch.empty((T,), dtype=torch.float32, device=dev)}
        _check(lib.fk_op_moe_ffn(self.handle, layer, _ptr(u), T, _ptr(forced), _ptr(out["out"]), _ptr(out["ids"]),
                                 _ptr(out["margin"]), _ptr(ws), wsb, _stream_ptr(stream)), "fk_op_moe_ffn")
        return out

    def set_moe_routing(self, forced=None, trace_ids=None, trace_margin=None, max_tokens: int = 0):
        """fk_model_set_moe_routing: forced expert ids and routing traces,
        laid out [n_moe_layers][max_tokens][k] (margins [n_moe_layers][max_tokens]);
        all None clears the hook. The tensors must outlive their use."""
        self._moe_hook = (forced, trace_ids, trace_margin)
        _check(load().fk_model_set_moe_routing(self.handle, _ptr(forced), _ptr(trace_ids), _ptr(trace_margin),
                                               max_tokens), "fk_model_set_moe_routing")

    def session(self, batch: int, max_seq: int, max_chunk: int | None = None) -> "Session":
        return Session(self, batch, max_seq, max_chunk or max_seq)

    def sync_status(self, stream=None, timeout_ms: int = 10000):
        return fk_sync_status(self.handle, _stream_ptr(stream), timeout_ms)


class Session:
    """KV-cached prefill + greedy decode for `batch` sequences."""

    def __init__(self, model: Model, batch: int, max_seq: int, max_chunk: int):
        import torch
        lib = load()
        self.model = model
        self.batch = batch
        nbytes = lib.fk_session_bytes(model.handle, batch, max_seq, max_chunk)
        if nbytes == 0:
            raise FkError(1, "fk_session_bytes", lib.fk_last_error().decode())
        self.mem = torch.empty(nbytes, dtype=torch.uint8, device=model.arena.device)
        h = c_void_p()
        _check(lib.fk_session_create(model.handle, batch, max_seq, max_chunk, _ptr(self.mem), nbytes,
                                     ctypes.byref(h)), "fk_session_create")
        self.handle = h.value

    def close(self):
        if self.handle:
            load().fk_session_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, ids, logits=None, next_ids=None, margin=None, stream=None):
        import numpy as np
        import torch
        on_dev = isinstance(ids, torch.Tensor) and ids.is_cuda
        if not on_dev:
            ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        S = ids.shape[1]
        ids_ptr = _ptr(ids) if on_dev else ids.ctypes.data
        _check(fk_session_prefill(self.handle, ids_ptr, 1 if on_dev else 0, S, _ptr(logits), _ptr(next_ids),
                                  _ptr(margin), _stream_ptr(stream)), "fk_session_prefill")

    def decode(self, ids=None, logits=None, next_ids=None, margin=None, stream=None):
        _check(fk_decode_step(self.handle, _ptr(ids), _ptr(logits), _ptr(next_ids), _ptr(margin),
                              _stream_ptr(stream)), "fk_decode_step")

    def reset(self):
        _check(load().fk_session_reset(self.handle), "fk_session_reset")

    @property
    def length(self) -> int:
        return load().fk_session_length(self.handle)


def build_library(force: bool = False) -> str:
    """Compile libfk.so for sm_103a (in-tree)."""
    return _build.build(force=force)
