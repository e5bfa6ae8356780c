"""Float64 CPU oracle of the decoder-only transformer forward pass.

Test infrastructure only (see the package docstring). Every array here is
numpy float64; weights arrive as bf16 bit patterns and are widened exactly.
Sums are left to numpy (``@``, ``sum``, ``mean``) in float64; there is no
blocking, fusion or reordering beyond what each definition states.

Readings taken where the pages are silent or ambiguous (each one is also
listed in the design notes):

* Hidden slots: slot 0 is the embedding output, slot l+1 the residual stream
  after layer l, slot L+1 the final-norm output ("N7 · model/forward-parity",
  Thm 1: one hidden slot per layer, then finalNorm).
* RoPE pairs element j with element j + hd/2 (half split), frequency
  f_j = theta^(-2j/hd), angle = position * f_j, positions 0-based per sequence.
* llama3 RoPE scaling follows the published Llama-3.1 rule (wavelength bands
  set by the original context and the low/high frequency factors).
* Gemma-style layers: local layers use RoPE base 10 000 and a window W where
  query i sees key j iff 0 <= i - j < W; global layers use base 1 000 000.
* QK-norm is an RMSNorm over head_dim per head (weights shared by the heads),
  applied before RoPE. Sandwich norm normalises the attention output and the
  FFN output before each residual add.
* The GELU-gated FFN uses the tanh form of GELU.
* GQA: query head h reads key/value head floor(h / (Hq / Hkv)).
* Softcap z -> c * tanh(z / c) on the float logits, before argmax.
* The embedding scale is bf16(sqrt(hidden)); the product stays in float.
* Argmax ties go to the lowest index.

``storage="bf16"`` evaluates the same definition with the values that the
numerics contract stores in 16 bits rounded where they are stored, to bf16.
The storage sites are: ``qkv_in`` (the norm output feeding the Q/K/V
projection), ``attn`` (the projected q, k, v and q, k after QK-norm and
RoPE), ``o_in`` (the attention output feeding the O projection), ``ffn_in``
(the norm output feeding gate/up), ``ffn_act`` (the gated activation feeding
the down projection) and ``head_in`` (the final-norm output feeding the LM
head). ``storage="f16"`` rounds the same sites to IEEE binary16 instead, and a
dict {site: "exact" | "bf16" | "f16"} chooses per site (unnamed sites stay
exact). Arithmetic stays float64 and the attention probabilities stay
unrounded. ``storage="exact"`` (the default) rounds nothing.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_to_f64", "round_to_bf16", "embed_scale", "rmsnorm", "rope_inv_freq", "rope_apply",
    "attention", "silu", "gelu_tanh", "softcap", "gemm", "OracleWeights", "forward", "Session",
    "argmax_first", "top2_margin", "log_softmax", "topk_ids", "greedy", "store_bf16", "store_f16",
    "STORAGE_SITES", "moe_route", "moe_ffn",
]


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: the bits are the top 16 of a float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(v: float) -> float:
    """Round a finite scalar to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits: write v = m * 2^e with 0.5 <= |m| < 1, keep
    round(m * 2^8) (Python's round is half-to-even) and scale back.
    """
    if v == 0.0:
        return 0.0
    m, e = math.frexp(v)
    return math.ldexp(round(m * 256.0), e - 8)


def store_bf16(x: np.ndarray) -> np.ndarray:
    """Value of x after being stored as bf16: float64 -> float32 (nearest),
    then the float32 bits rounded to the top 16 (nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def store_f16(x: np.ndarray) -> np.ndarray:
    """Value of x after being stored as IEEE binary16: float64 -> float32
    (nearest), then float32 -> binary16 (nearest, ties to even; subnormals
    kept, overflow to infinity)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


STORAGE_SITES = ("qkv_in", "attn", "o_in", "ffn_in", "ffn_act", "head_in")
_FORMATS = {"exact": lambda x: x, "bf16": store_bf16, "f16": store_f16}


class _Rounder:
    """Storage rounding per site (see the module docstring)."""

    def __init__(self, storage):
        if isinstance(storage, str):
            if storage not in _FORMATS:
                raise ValueError(storage)
            storage = {site: storage for site in STORAGE_SITES}
        unknown = set(storage) - set(STORAGE_SITES)
        if unknown:
            raise ValueError(f"unknown storage sites {sorted(unknown)}")
        self.fn = {site: _FORMATS[storage.get(site, "exact")] for site in STORAGE_SITES}

    def __call__(self, site: str, x: np.ndarray) -> np.ndarray:
        return self.fn[site](x)


def _rounder(storage):
    return _Rounder(storage)


# ---------------------------------------------------------------------------
# Ops
# ---------------------------------------------------------------------------
def embed_scale(cfg) -> float:
    """Embedding multiplier: bf16(sqrt(hidden)) for the Gemma3-style tower,
    else 1 ("pegainfer issue #878", Proposed Plan: derive the embedding scale
    and assert it against the recorded bf16-rounded value)."""
    if cfg.embed_scale == "sqrt_hidden_bf16":
        return round_to_bf16(math.sqrt(cfg.hidden))
    return 1.0


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w
    ("N7 · model/forward-parity", Thm 1: the decoder stack's RMSNorm)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_inv_freq(cfg, kind: int) -> np.ndarray:
    """Per-pair rotation frequencies f_j, j < hd/2 ("N7", Thm 1 RoPE; Thm 2
    llama3 "rope scaling" axis; "pegainfer #878" local/global layer kinds).

    kind 0 = global layer (base rope_theta_global), 1 = local (rope_theta_local).
    llama3 scaling: with wavelength lam_j = 2*pi / f_j, original context C,
    low factor a, high factor b and factor s: lam_j < C/b keeps f_j;
    lam_j > C/a gives f_j / s; in between, with t = (C/lam_j - a)/(b - a),
    f = (1 - t) * f_j / s + t * f_j.
    """
    hd = cfg.head_dim
    theta = cfg.rope_theta_local if kind == 1 else cfg.rope_theta_global
    j = np.arange(hd // 2, dtype=np.float64)
    f = theta ** (-2.0 * j / hd)
    if cfg.rope_scaling == "llama3":
        C = float(cfg.rope_orig_max_pos)
        a, b, s = cfg.rope_low_freq_factor, cfg.rope_high_freq_factor, cfg.rope_factor
        lam = 2.0 * math.pi / f
        out = np.empty_like(f)
        for i in range(f.shape[0]):
            if lam[i] < C / b:
                out[i] = f[i]
            elif lam[i] > C / a:
                out[i] = f[i] / s
            else:
                t = (C / lam[i] - a) / (b - a)
                out[i] = (1.0 - t) * f[i] / s + t * f[i]
        f = out
    elif cfg.rope_scaling != "none":
        raise ValueError(cfg.rope_scaling)
    return f


def rope_apply(x: np.ndarray, pos: np.ndarray, inv_freq: np.ndarray) -> np.ndarray:
    """Rotate pairs (j, j + hd/2) of x[..., T, n_heads, hd] by angle pos_t * f_j.

    pos has shape [..., T] (0-based absolute positions)."""
    half = x.shape[-1] // 2
    ang = pos[..., :, None].astype(np.float64) * inv_freq[None, :]      # [..., T, half]
    c = np.cos(ang)[..., :, None, :]
    s = np.sin(ang)[..., :, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray, k_pos: np.ndarray,
              window: int, scale: float) -> np.ndarray:
    """Causal GQA attention for one sequence ("N7", Thm 1: causal multi-head /
    GQA attention; Thm 2 and "pegainfer #878": sliding-window local layers).

    q [Sq, Hq, hd], k/v [Sk, Hkv, hd]; query i may read key j iff
    k_pos_j <= q_pos_i and (window == 0 or q_pos_i - k_pos_j < window).
    Head h reads kv head h // (Hq // Hkv). Softmax is float64.
    """
    Sq, Hq, hd = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    allowed = k_pos[None, :] <= q_pos[:, None]
    if window > 0:
        allowed &= (q_pos[:, None] - k_pos[None, :]) < window
    out = np.empty((Sq, Hq, v.shape[-1]), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) * scale                  # [Sq, Sk]
        s = np.where(allowed, s, -np.inf)
        s = s - np.max(s, axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=-1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU gate of the SwiGLU FFN: g * sigmoid(g) ("N7", Thm 1: SwiGLU FFN)."""
    return g / (1.0 + np.exp(-g))


def gelu_tanh(g: np.ndarray) -> np.ndarray:
    """tanh-form GELU for the GELU-gated FFN of the Gemma3-style tower:
    0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))."""
    return 0.5 * g * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g * g * g)))


def softcap(z: np.ndarray, c: float) -> np.ndarray:
    """Final-logit softcap c * tanh(z / c) ("pegainfer #878": softcap carried
    on the typed config and validated positive)."""
    return c * np.tanh(z / c)


def gemm(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y = X · Wᵀ in float64 ("N9 · metalgemm", Thm 1: the GEMM the device
    lane computes, checked against a float64-accumulated reference)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


# ---------------------------------------------------------------------------
# Weights
# ---------------------------------------------------------------------------
class OracleWeights:
    """Float64 view of a dict of bf16 weight bits. Small models keep the
    widened arrays; large ones widen a tensor each time it is read."""

    def __init__(self, bits: dict, cache_limit_bytes: int = 2 << 30):
        self.bits = bits
        total = sum(int(b.size) for b in bits.values()) * 8
        self.cache = {} if total <= cache_limit_bytes else None

    def __getitem__(self, name: str) -> np.ndarray:
        if self.cache is not None:
            if name not in self.cache:
                self.cache[name] = bf16_to_f64(self.bits[name])
            return self.cache[name]
        return bf16_to_f64(self.bits[name])

    def linear(self, x: np.ndarray, name: str, rows_per_chunk: int = 8192) -> np.ndarray:
        """x · W[name]ᵀ; a large W is widened a block of output rows at a time
        (each output element is still one float64 dot product over the input)."""
        w = self.bits[name]
        if self.cache is not None or w.shape[0] <= rows_per_chunk:
            return gemm(x, self[name])
        out = np.empty(x.shape[:-1] + (w.shape[0],), dtype=np.float64)
        for r0 in range(0, w.shape[0], rows_per_chunk):
            r1 = min(r0 + rows_per_chunk, w.shape[0])
            out[..., r0:r1] = gemm(x, bf16_to_f64(w[r0:r1]))
        return out

    def expert(self, name: str, e: int) -> np.ndarray:
        """Float64 view of expert e of a stacked [E, rows, cols] weight."""
        if self.cache is not None:
            return self[name][e]
        return bf16_to_f64(self.bits[name][e])

    def head_name(self, cfg) -> str:
        return "embed" if cfg.tied else "lm_head"


# ---------------------------------------------------------------------------
# Mixture-of-experts FFN
# ---------------------------------------------------------------------------
def moe_route(cfg, z: np.ndarray):
    """Routing of a mixture-of-experts FFN ("N7 · model/forward-parity", Thm 2:
    the qwen3moe rung): p = softmax of the router logits z [..., E] over the
    experts; the k experts of largest p (ties to the lower index); weights p at
    those experts, renormalised to sum 1 when cfg.norm_topk.

    Returns (ids [..., k], weights [..., k], margin [...]) where margin is the
    gap between the k-th and (k+1)-th largest p (how far the choice is from a
    flip; +inf when k equals the number of experts)."""
    k, E = cfg.n_experts_per_tok, cfg.n_experts
    z = np.asarray(z, dtype=np.float64)
    pz = np.exp(z - np.max(z, axis=-1, keepdims=True))
    pz = pz / np.sum(pz, axis=-1, keepdims=True)
    order = np.argsort(-pz, axis=-1, kind="stable")
    ids = order[..., :k]
    w = np.take_along_axis(pz, ids, -1)
    if cfg.norm_topk:
        w = w / np.sum(w, axis=-1, keepdims=True)
    if k < E:
        srt = np.take_along_axis(pz, order[..., k - 1:k + 1], -1)
        margin = srt[..., 0] - srt[..., 1]
    else:
        margin = np.full(z.shape[:-1], np.inf)
    return ids, w, margin


def moe_ffn(cfg, W: "OracleWeights", l: int, u: np.ndarray, R=None, forced_ids=None) -> dict:
    """The mixture-of-experts FFN of layer l on u [..., H]: router logits
    z = u·W_routerᵀ, routing by moe_route (or the ids in forced_ids [..., k],
    weighted by the same softmax), then out = sum over the chosen experts e of
    w_e · down_e(act(gate_e u) ⊙ up_e u) ("N7", Thm 2: qwen3moe; the expert
    FFN is the SwiGLU FFN of Thm 1 with the expert's own matrices).

    R: the storage rounding of the activation sites (a _Rounder, or a storage
    name as forward() takes; None = exact).

    Returns {"out": [..., H], "ids": [..., k], "margin": [...]}."""
    if R is None or isinstance(R, str):
        R = _rounder(R or "exact")
    p = f"L{l}."
    z = W.linear(u, p + "router")
    ids, w, margin = moe_route(cfg, z)
    if forced_ids is not None:
        ids = np.asarray(forced_ids).reshape(ids.shape)
        pz = np.exp(z - np.max(z, axis=-1, keepdims=True))
        pz = pz / np.sum(pz, axis=-1, keepdims=True)
        w = np.take_along_axis(pz, ids, -1)
        if cfg.norm_topk:
            w = w / np.sum(w, axis=-1, keepdims=True)
    H = u.shape[-1]
    U = u.reshape(-1, H)
    I = ids.reshape(U.shape[0], -1)
    Wt = w.reshape(U.shape[0], -1)
    out = np.zeros_like(U)
    for e in range(cfg.n_experts):
        rows, slots = np.nonzero(I == e)
        if rows.size == 0:
            continue
        ue = U[rows]
        g = ue @ W.expert(p + "expert_gate", e).T
        up = ue @ W.expert(p + "expert_up", e).T
        act = silu(g) if cfg.act == "silu" else gelu_tanh(g)
        y = R("ffn_act", act * up) @ W.expert(p + "expert_down", e).T
        out[rows] += Wt[rows, slots][:, None] * y
    return {"out": out.reshape(u.shape), "ids": ids, "margin": margin}


# ---------------------------------------------------------------------------
# Decoder layer and forward
# ---------------------------------------------------------------------------
def _layer(cfg, W: OracleWeights, l: int, x: np.ndarray, pos: np.ndarray, past_k, past_v, past_pos, R=None,
           moe=None):
    """One decoder layer on x [B, S, H] at positions pos [B, S].

    past_k/past_v [B, P, Hkv, hd] (P may be 0) are this layer's cached keys and
    values at positions past_pos [B, P]. Returns the new x and the keys/values
    of the S new tokens ("N7", Thm 1: RMSNorm, Q/K/V, RoPE, causal GQA
    attention, SwiGLU FFN, residuals; Thm 2: topology-selected norm placement,
    QK-norm, sliding window)."""
    B, S, H = x.shape
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    p = f"L{l}."
    kind = cfg.kinds()[l]
    window = cfg.sliding_window if kind == 1 else 0

    if R is None:
        R = _rounder("exact")
    u = R("qkv_in", rmsnorm(x, W[p + "attn_norm"], cfg.rms_eps))
    q = R("attn", W.linear(u, p + "wq")).reshape(B, S, Hq, hd)
    k = R("attn", W.linear(u, p + "wk")).reshape(B, S, Hkv, hd)
    v = R("attn", W.linear(u, p + "wv")).reshape(B, S, Hkv, hd)
    if cfg.qk_norm:
        q = rmsnorm(q, W[p + "q_norm"], cfg.rms_eps)
        k = rmsnorm(k, W[p + "k_norm"], cfg.rms_eps)
    f = rope_inv_freq(cfg, kind)
    q = R("attn", rope_apply(q, pos, f))
    k = R("attn", rope_apply(k, pos, f))

    keys = np.concatenate([past_k, k], axis=1)
    vals = np.concatenate([past_v, v], axis=1)
    kpos = np.concatenate([past_pos, pos], axis=1)
    o = np.empty((B, S, Hq, hd), dtype=np.float64)
    for b in range(B):
        o[b] = attention(q[b], keys[b], vals[b], pos[b], kpos[b], window, 1.0 / math.sqrt(hd))
    a = W.linear(R("o_in", o).reshape(B, S, Hq * hd), p + "wo")
    if cfg.norm_layout == "sandwich":
        a = rmsnorm(a, W[p + "post_attn_norm"], cfg.rms_eps)
    x = x + a

    u = R("ffn_in", rmsnorm(x, W[p + "ffn_norm"], cfg.rms_eps))
    if cfg.moe_kinds()[l]:
        # moe: {"forced": {layer: ids} or None, "trace": {layer: routing}} (optional)
        forced = (moe or {}).get("forced") or {}
        r = moe_ffn(cfg, W, l, u, R, forced.get(l))
        if moe is not None and "trace" in moe:
            moe["trace"][l] = {"ids": r["ids"], "margin": r["margin"]}
        d = r["out"]
    else:
        g = W.linear(u, p + "w_gate")
        up = W.linear(u, p + "w_up")
        act = silu(g) if cfg.act == "silu" else gelu_tanh(g)
        d = W.linear(R("ffn_act", act * up), p + "w_down")
    if cfg.norm_layout == "sandwich":
        d = rmsnorm(d, W[p + "post_ffn_norm"], cfg.rms_eps)
    x = x + d
    return x, k, v


def _embed(cfg, W: OracleWeights, ids: np.ndarray) -> np.ndarray:
    """Embedding lookup E[id] times the (optional) bf16 embedding scale."""
    ids = np.asarray(ids)
    if ids.size and (ids.min() < 0 or ids.max() >= cfg.vocab):
        raise ValueError("token id out of range")  # "pegainfer #878": ids bounds-checked
    return bf16_to_f64(W.bits["embed"][ids]) * embed_scale(cfg)


def _head(cfg, W: OracleWeights, y: np.ndarray) -> np.ndarray:
    """LM head (tied to the embedding or separate), then the optional softcap."""
    z = W.linear(y, W.head_name(cfg))
    if cfg.final_softcap > 0:
        z = softcap(z, cfg.final_softcap)
    return z


def forward(cfg, weights, ids: np.ndarray, hidden: bool = True, logits: str = "all", storage: str = "exact",
            moe_forced=None) -> dict:
    """Cacheless forward over ids [B, S] ("N7 · model/forward-parity", Thm 1:
    embedding lookup, decoder stack appending one hidden slot per layer, final
    norm, head matmul to logits).

    moe_forced: optional {layer: expert ids [B, S, k]} replacing the routing
    choice of those mixture-of-experts layers (their weights still come from
    this forward's own router softmax).

    Returns {"hidden": [L+2, B, S, H] or None, "logits": [B, S, V] ("all") or
    [B, V] ("last") or None ("none"), "moe": {layer: {"ids", "margin"}} of the
    routing actually used}.
    """
    R = _rounder(storage)
    W = weights if isinstance(weights, OracleWeights) else OracleWeights(weights)
    ids = np.asarray(ids)
    B, S = ids.shape
    Hkv, hd = cfg.n_kv_heads, cfg.head_dim
    x = _embed(cfg, W, ids)
    pos = np.broadcast_to(np.arange(S), (B, S))
    slots = [x] if hidden else None
    empty_kv = np.zeros((B, 0, Hkv, hd))
    empty_pos = np.zeros((B, 0), dtype=np.int64)
    moe = {"forced": moe_forced, "trace": {}}
    for l in range(cfg.n_layers):
        x, _, _ = _layer(cfg, W, l, x, pos, empty_kv, empty_kv, empty_pos, R, moe)
        if hidden:
            slots.append(x)
    y = rmsnorm(x, W["final_norm"], cfg.rms_eps)
    if hidden:
        slots.append(y)
    out = {"hidden": np.stack(slots) if hidden else None, "moe": moe["trace"]}
    if logits == "all":
        out["logits"] = _head(cfg, W, R("head_in", y))
    elif logits == "last":
        out["logits"] = _head(cfg, W, R("head_in", y[:, -1, :]))
    else:
        out["logits"] = None
    return out


class Session:
    """KV-cached prefill and decode for B sequences of equal length ("N7",
    Thm 1: NewSession().Prefill last-position logits agree with the cacheless
    Forward; greedy Generate feeds each argmax back as the next token)."""

    def __init__(self, cfg, weights, batch: int, storage: str = "exact"):
        self.R = _rounder(storage)
        self.cfg = cfg
        self.W = weights if isinstance(weights, OracleWeights) else OracleWeights(weights)
        self.B = batch
        Hkv, hd = cfg.n_kv_heads, cfg.head_dim
        self.k = [np.zeros((batch, 0, Hkv, hd)) for _ in range(cfg.n_layers)]
        self.v = [np.zeros((batch, 0, Hkv, hd)) for _ in range(cfg.n_layers)]
        self.length = 0

    def _run(self, ids: np.ndarray, moe_forced=None) -> np.ndarray:
        cfg, W = self.cfg, self.W
        ids = np.asarray(ids).reshape(self.B, -1)
        S = ids.shape[1]
        pos = np.broadcast_to(np.arange(self.length, self.length + S), (self.B, S))
        past_pos = np.broadcast_to(np.arange(self.length), (self.B, self.length))
        x = _embed(cfg, W, ids)
        self.moe = {"forced": moe_forced, "trace": {}}
        for l in range(cfg.n_layers):
            x, k, v = _layer(cfg, W, l, x, pos, self.k[l], self.v[l], past_pos, self.R, self.moe)
            self.k[l] = np.concatenate([self.k[l], k], axis=1)
            self.v[l] = np.concatenate([self.v[l], v], axis=1)
        self.length += S
        y = self.R("head_in", rmsnorm(x[:, -1, :], W["final_norm"], cfg.rms_eps))
        return _head(cfg, W, y)

    def prefill(self, ids: np.ndarray, moe_forced=None) -> np.ndarray:
        """Append ids [B, S]; return the last-position logits [B, V]. After the
        call, self.moe["trace"] holds the routing of each MoE layer."""
        return self._run(ids, moe_forced)

    def decode(self, ids: np.ndarray, moe_forced=None) -> np.ndarray:
        """Append one token per sequence (ids [B]); return logits [B, V]."""
        return self._run(np.asarray(ids).reshape(self.B, 1), moe_forced)


# ---------------------------------------------------------------------------
# Readouts
# ---------------------------------------------------------------------------
def argmax_first(z: np.ndarray) -> np.ndarray:
    """Per-row argmax over the last axis; ties go to the lowest index."""
    return np.argmax(z, axis=-1)


def top2_margin(z: np.ndarray) -> np.ndarray:
    """Per-row gap between the largest and second-largest value."""
    part = np.partition(z, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def log_softmax(z: np.ndarray) -> np.ndarray:
    """log p = z - max - log(sum(exp(z - max))), float64."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    return z - m - np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True))


def topk_ids(z: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k largest values per row, largest first (ties: lower id first)."""
    order = np.argsort(-np.asarray(z), axis=-1, kind="stable")
    return order[..., :k]


def greedy(cfg, weights, prompt: np.ndarray, n_steps: int, forced: np.ndarray | None = None,
           storage: str = "exact") -> dict:
    """Greedy generation: prefill the prompt [B, S], take next = argmax, then
    n_steps decode steps each feeding the previous id ("N7", Thm 1 witness:
    Generate's greedy ids). With ``forced`` [n_steps, B] the fed ids are those
    instead (teacher forcing) and the argmax of each step is still recorded.

    Returns {"ids": [n_steps + 1, B] argmax per call, "margins": same shape,
    "first_logits": logits of the prefill, "last_logits": logits of the final call}.
    """
    sess = Session(cfg, weights, np.asarray(prompt).shape[0], storage)
    z = sess.prefill(prompt)
    first = z
    ids, margins = [argmax_first(z)], [top2_margin(z)]
    for t in range(n_steps):
        feed = ids[-1] if forced is None else np.asarray(forced[t])
        z = sess.decode(feed)
        ids.append(argmax_first(z))
        margins.append(top2_margin(z))
    return {"ids": np.stack(ids), "margins": np.stack(margins), "first_logits": first, "last_logits": z}
