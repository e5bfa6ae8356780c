/*
 * fk -- decoder-only transformer forward pass (bf16) on one NVIDIA GB300.
 *
 * C ABI. Plain pointers and sizes only; no C++ or framework types cross it.
 *
 * What it computes (the pages' own terms):
 *   "N7 · model/forward-parity", Theorem 1: embedding lookup, the decoder
 *   stack (RMSNorm, Q/K/V projections, RoPE, causal GQA attention, SwiGLU FFN,
 *   residuals), final norm and the (tied) LM head, giving per-layer hidden
 *   states and per-position logits and argmax; a cached session whose prefill
 *   last-position logits equal the cacheless forward; greedy generation.
 *   Theorem 2: family axes -- QK-norm, sliding-window local layers, sandwich
 *   norm placement, llama3 RoPE scaling.
 *   "pegainfer issue #878", Proposed Plan: scaled embedding, layer dispatch
 *   by a parsed local/global layer map, final-logit softcap validated
 *   positive, geometry derived from the config as the one source of buffer
 *   sizes, token ids bounds-checked before upload.
 *   "N9 · metalgemm", Theorem 1: the GEMM Y = X·Wᵀ of the projections.
 *
 * Conventions for every entry point:
 *   - Device pointers ("d_" prefix) point to GPU global memory that the
 *     caller allocated and owns; the library never allocates device memory
 *     and never frees caller memory. Sizes come from the *_bytes queries.
 *     Device buffers must be 256-byte aligned.
 *   - Host pointers ("h_" prefix, or as stated) are read during the call only.
 *   - Work is queued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: outputs are valid once the stream has
 *     synchronised.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and returns a status != FK_OK, with a
 *     message in fk_last_error() (thread-local).
 *   - Device-side faults that can only be seen on the device (a token id read
 *     from device memory that is out of range, a pipeline wait that timed
 *     out) never trap: they set the model's device error word, which
 *     fk_sync_status() reports and clears.
 *   - bf16 tensors are row-major arrays of IEEE bfloat16; fp32 tensors are
 *     row-major float.
 *   - A model may be shared by several sessions; a model or session must not
 *     be used from two host threads at once.
 */
#ifndef FK_H
#define FK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fk_status {
  FK_OK = 0,
  FK_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned buffer */
  FK_ERR_INVALID_CONFIG = 2,  /* model geometry rejected */
  FK_ERR_TOKEN_RANGE = 3,     /* a host token id outside [0, vocab) */
  FK_ERR_CONTEXT_FULL = 4,    /* session would exceed its max_seq */
  FK_ERR_NO_DEVICE = 5,       /* no CUDA device, or not a GB300-class sm_103 device */
  FK_ERR_CUDA = 6,            /* a CUDA runtime or driver call failed */
  FK_ERR_DEVICE_FLAG = 7,     /* the device error word was set (see fk_sync_status) */
  FK_ERR_TIMEOUT = 8,         /* fk_sync_status deadline passed */
  FK_ERR_WORKSPACE = 9        /* a caller buffer is smaller than its *_bytes query */
} fk_status;

/* Bits of the device error word. */
#define FK_DEVERR_TOKEN_RANGE 0x1u   /* a device-resident token id was out of range (clamped) */
#define FK_DEVERR_PIPE_TIMEOUT 0x2u  /* a kernel pipeline wait gave up */
#define FK_DEVERR_EXPERT_IDS 0x4u    /* forced expert ids out of range or repeated (that token routed itself) */

typedef enum { FK_ROPE_NONE = 0, FK_ROPE_LLAMA3 = 1 } fk_rope_scaling;
typedef enum { FK_ACT_SILU = 0, FK_ACT_GELU_TANH = 1 } fk_act;
typedef enum { FK_NORM_PRE = 0, FK_NORM_SANDWICH = 1 } fk_norm_layout;
typedef enum { FK_EMBED_SCALE_NONE = 0, FK_EMBED_SCALE_SQRT_HIDDEN_BF16 = 1 } fk_embed_scale;

/* Activation storage sites (bits of fk_config.f16_sites). Every activation
 * the forward keeps in 16 bits between two kernels is stored as bf16 (8
 * significant bits) unless its site's bit is set, in which case it is stored
 * as IEEE f16 (11 significant bits, range +-65504). A GEMM whose input site is
 * f16 runs on f16 tensor-core operands against an f16 copy of its bf16
 * weights, made once in the model arena (exact for weights of magnitude in
 * [2^-17, 65504]; smaller ones keep an absolute error below 2^-25). All
 * accumulation stays fp32 and the residual stream fp32 either way. The bits:
 *   FK_F16_QKV_IN   norm output feeding the Q/K/V projection
 *   FK_F16_ATTN     q, k, v, the KV cache and the softmax probabilities
 *   FK_F16_O_IN     attention output feeding the O projection
 *   FK_F16_FFN_IN   norm output feeding the gate/up projection
 *   FK_F16_FFN_ACT  gated activation feeding the down projection
 *   FK_F16_HEAD_IN  final-norm output feeding the LM head
 * f16 keeps 3 more significant bits than bf16: on deep models with large
 * hidden sizes the rounding of these activations is what separates the
 * result from the exact forward, so the finer format brings it inside the
 * forward-parity gates ("N7 · model/forward-parity", Thm 1: hidden cosine
 * >= 0.9999, last-position logits within 0.05) at the same tensor-core rate.
 * The price is range: an activation above 65504 in magnitude overflows. */
#define FK_F16_QKV_IN 0x01u
#define FK_F16_ATTN 0x02u
#define FK_F16_O_IN 0x04u
#define FK_F16_FFN_IN 0x08u
#define FK_F16_FFN_ACT 0x10u
#define FK_F16_HEAD_IN 0x20u
#define FK_F16_ALL 0x3Fu

/*
 * Model geometry ("pegainfer #878": one typed config is the single source of
 * every buffer size). Validation rules (FK_ERR_INVALID_CONFIG otherwise):
 *   n_layers >= 1; hidden and intermediate positive multiples of 64;
 *   n_q_heads, n_kv_heads >= 1 with n_q_heads a multiple of n_kv_heads and
 *   at most 8 query heads per kv head; head_dim 64, 128 or 256; vocab a
 *   positive multiple of 8; rms_eps > 0 and finite; rope thetas > 1; llama3
 *   scaling needs factor >= 1, high_freq_factor > low_freq_factor > 0 and
 *   orig_max_pos > 0; act, norm_layout and embed_scale one of their enums;
 *   qk_norm and tied 0 or 1; sliding_window >= 0; layer_kinds entries 0
 *   (global) or 1 (local), local layers only with sliding_window > 0;
 *   final_softcap == 0 (off) or > 0 and finite; f16_sites within FK_F16_ALL.
 * Mixture-of-experts layers ("N7 · model/forward-parity", Thm 2: the qwen3moe
 * rung): n_experts == 0 makes every FFN dense (moe_layers must then be NULL
 * or all 0). Otherwise n_experts is a multiple of 8 up to 256, 1 <=
 * n_experts_per_tok <= min(n_experts, 16), expert_intermediate a positive
 * multiple of 64, norm_topk 0 or 1, moe_layers NULL (every layer MoE) or
 * entries 0 (dense) / 1 (MoE); intermediate is checked only when some layer
 * is dense.
 */
typedef struct fk_config {
  int32_t n_layers;
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  int32_t vocab;
  float rms_eps;
  double rope_theta_global;     /* RoPE base of global layers */
  double rope_theta_local;      /* RoPE base of local (sliding-window) layers */
  int32_t rope_scaling;         /* fk_rope_scaling */
  float rope_factor;            /* llama3: divisor of the low-frequency band */
  float rope_low_freq_factor;   /* llama3: a */
  float rope_high_freq_factor;  /* llama3: b */
  int32_t rope_orig_max_pos;    /* llama3: original context C */
  int32_t act;                  /* fk_act: FFN gate activation */
  int32_t norm_layout;          /* fk_norm_layout */
  int32_t qk_norm;              /* 1 = per-head RMSNorm on q and k before RoPE */
  int32_t sliding_window;       /* W of local layers: query i sees key j iff 0 <= i-j < W */
  const uint8_t* layer_kinds;   /* host, n_layers entries, 0 = global, 1 = local; NULL = all global */
  int32_t embed_scale;          /* fk_embed_scale */
  float final_softcap;          /* c of z -> c*tanh(z/c); 0 = off */
  int32_t tied;                 /* 1 = LM head is the embedding matrix */
  uint32_t f16_sites;           /* FK_F16_* bits: activation sites stored as f16 (0 = all bf16) */
  /* Mixture-of-experts FFN: the router picks the n_experts_per_tok experts of
   * largest softmax probability (ties to the lower expert id) and the FFN
   * output is the sum of their SwiGLU outputs weighted by those
   * probabilities, divided by their sum when norm_topk. */
  int32_t n_experts;            /* 0 = dense FFN on every layer */
  int32_t n_experts_per_tok;    /* k */
  int32_t expert_intermediate;  /* FFN width of one expert */
  int32_t norm_topk;            /* 1 = renormalise the k weights to sum 1 */
  const uint8_t* moe_layers;    /* host, n_layers entries, 1 = MoE FFN; NULL = every layer (if n_experts) */
} fk_config;

/* Per-layer device weights, all bf16. Matrices are [out, in] row-major.
 * q_norm/k_norm [head_dim] are read only when qk_norm; post_attn_norm and
 * post_ffn_norm [hidden] only for FK_NORM_SANDWICH. Norm weights are the
 * effective multipliers (a "1 + w" convention is folded in by the caller). */
typedef struct fk_layer_weights {
  const void* attn_norm;       /* [hidden] */
  const void* wq;              /* [n_q_heads*head_dim, hidden] */
  const void* wk;              /* [n_kv_heads*head_dim, hidden] */
  const void* wv;              /* [n_kv_heads*head_dim, hidden] */
  const void* wo;              /* [hidden, n_q_heads*head_dim] */
  const void* q_norm;          /* [head_dim] */
  const void* k_norm;          /* [head_dim] */
  const void* post_attn_norm;  /* [hidden] */
  const void* ffn_norm;        /* [hidden] */
  const void* w_gate;          /* [intermediate, hidden] */
  const void* w_up;            /* [intermediate, hidden] */
  const void* w_down;          /* [hidden, intermediate] */
  const void* post_ffn_norm;   /* [hidden] */
  /* MoE layers only (w_gate, w_up, w_down are then unused and may be NULL) */
  const void* router;          /* [n_experts, hidden] */
  const void* expert_gate;     /* [n_experts][expert_intermediate, hidden] */
  const void* expert_up;       /* [n_experts][expert_intermediate, hidden] */
  const void* expert_down;     /* [n_experts][hidden, expert_intermediate] */
} fk_layer_weights;

typedef struct fk_weights {
  const void* embed;                /* [vocab, hidden] bf16, device */
  const void* lm_head;              /* [vocab, hidden] bf16, device; ignored (may be NULL) if tied */
  const void* final_norm;           /* [hidden] bf16, device */
  const fk_layer_weights* layers;   /* host array of n_layers entries */
} fk_weights;

typedef struct fk_model fk_model;
typedef struct fk_session fk_session;

/* ---------------------------------------------------------------------------
 * Status and errors
 * ------------------------------------------------------------------------- */
const char* fk_status_string(fk_status s);
/* Message of the last failing call on this host thread ("" if none). */
const char* fk_last_error(void);
/* Library version, e.g. "fk 0.1 sm_103a". */
const char* fk_version(void);

/* ---------------------------------------------------------------------------
 * Model
 * ------------------------------------------------------------------------- */
/* Device arena the model needs (the device error word, RoPE cos/sin tables
 * for positions [0, max_positions) of each layer kind, and the f16 copies of
 * the weights of every GEMM whose input site is f16). Returns 0 if cfg is
 * invalid. */
size_t fk_model_arena_bytes(const fk_config* cfg, int32_t max_positions);

/* Validate cfg, bind the caller's device weights (borrowed: they must outlive
 * the model), fill the arena (synchronously, on the current device) and
 * return a host handle in *out. max_positions bounds every sequence the model
 * will see (sessions' max_seq and forward's seq). */
fk_status fk_model_create(const fk_config* cfg, const fk_weights* w, int32_t max_positions,
                          void* d_arena, size_t arena_bytes, fk_model** out);
void fk_model_free(fk_model* m);

/* ---------------------------------------------------------------------------
 * Cacheless forward ("N7", Thm 1: Forward)
 * ------------------------------------------------------------------------- */
size_t fk_forward_workspace_bytes(const fk_model* m, int32_t batch, int32_t seq);

/* Forward over ids [batch, seq] (positions 0..seq-1 per sequence).
 *   ids: host int32 when ids_on_device == 0 (checked in [0, vocab) before
 *        anything is queued: FK_ERR_TOKEN_RANGE), else device int32 (checked
 *        on the device: out-of-range ids are clamped and set
 *        FK_DEVERR_TOKEN_RANGE).
 *   d_hidden: NULL, or fp32 [n_layers+2][batch*seq][hidden]: slot 0 the
 *        (scaled) embedding, slot l+1 the residual stream after layer l, slot
 *        n_layers+1 the final-norm output.
 *   d_logits: NULL, or fp32 [batch*seq][vocab] (after the softcap, if any).
 *   d_argmax: NULL, or int32 [batch*seq]: lowest index of the row maximum.
 *   d_margin: NULL, or fp32 [batch*seq]: the row maximum minus the largest
 *        other logit (0 on a tie) -- how far the argmax is from a flip ("N7 ·
 *        model/forward-parity", Thm 3: near-tie argmax flips). Needs d_argmax.
 * A host `ids` buffer is copied synchronously before the call returns.
 * Forwards of at most 64 tokens (batch*seq) are launch-bound: the model
 * keeps CUDA graphs of the launches that follow the ids copy, one per batch,
 * seq, workspace and output pointers (the 4 most recent keys), captured on
 * the second call with that key and replayed by later ones (calls
 * on a capturing stream, with kernel timing on, or with FK_NO_GRAPH set in
 * the environment launch one by one). Results are the same either way.
 * Such calls on one model from several host threads are serialised by the
 * model (its graph cache is guarded). */
fk_status fk_forward(fk_model* m, const int32_t* ids, int32_t ids_on_device, int32_t batch, int32_t seq,
                     void* d_ws, size_t ws_bytes, float* d_hidden, float* d_logits, int32_t* d_argmax,
                     float* d_margin, void* stream);

/* ---------------------------------------------------------------------------
 * KV-cached session ("N7", Thm 1: NewSession().Prefill and greedy Generate)
 * batch sequences of equal length. Per layer a K cache [batch][kv_head][cap]
 * [head_dim] and a transposed V cache [batch][kv_head][head_dim][cap] (16-bit,
 * bf16 or f16 as the config stores attention), both cleared when the session
 * is created; position p lives in slot p mod cap. Global layers: cap = max_seq
 * rounded up to 64. Sliding-window layers keep a ring: a query reads at most
 * the last W positions, and a prefill chunk needs the W - 1 positions before
 * it plus its own, so cap = W + max_chunk - 1 rounded up to 64 (at most the
 * global cap); decoding past W reuses the ring.
 * Prefill is processed in chunks of at most max_chunk tokens per sequence.
 * ------------------------------------------------------------------------- */
size_t fk_session_bytes(const fk_model* m, int32_t batch, int32_t max_seq, int32_t max_chunk);
fk_status fk_session_create(fk_model* m, int32_t batch, int32_t max_seq, int32_t max_chunk, void* d_mem,
                            size_t bytes, fk_session** out);
void fk_session_free(fk_session* s);

/* Append ids [batch, seq] (host or device as in fk_forward) after the tokens
 * already in the session. d_last_logits: NULL or fp32 [batch][vocab] of the
 * last position; d_next: NULL or int32 [batch], the greedy next ids (also
 * kept in the session for fk_decode_step); d_margin: NULL or fp32 [batch],
 * the top-1 minus top-2 logit of each next id (as in fk_forward).
 * FK_ERR_CONTEXT_FULL if the session would exceed max_seq. */
fk_status fk_session_prefill(fk_session* s, const int32_t* ids, int32_t ids_on_device, int32_t seq,
                             float* d_last_logits, int32_t* d_next, float* d_margin, void* stream);

/* One greedy decode step: feed d_ids [batch] (device int32), or the session's
 * last greedy ids when d_ids is NULL; write logits / next ids / margins as in
 * prefill. */
fk_status fk_decode_step(fk_session* s, const int32_t* d_ids, float* d_logits, int32_t* d_next, float* d_margin,
                         void* stream);

/* Forget all tokens (length 0); the cache memory is reused. */
fk_status fk_session_reset(fk_session* s);
int32_t fk_session_length(const fk_session* s);

/* Wait up to timeout_ms for `stream` to drain, then read and clear the device
 * error word: FK_OK, FK_ERR_DEVICE_FLAG (bits in *flags if non-NULL), or
 * FK_ERR_TIMEOUT (the stream is still busy; nothing was read). m == NULL reads
 * the current device's op-level word instead, which the op-level entry points
 * below (GEMMs, attention, op hooks) set. */
fk_status fk_sync_status(fk_model* m, void* stream, int32_t timeout_ms, uint32_t* flags);

/* ---------------------------------------------------------------------------
 * Op-level entry points (per-kernel parity; same kernels as the forward)
 * A pipeline timeout inside one of them sets the current device's op-level
 * error word, read with fk_sync_status(NULL, ...).
 * ------------------------------------------------------------------------- */
/* Y[P,N] = X[P,K] · W[N,K]ᵀ, bf16 inputs, fp32 accumulation ("N9 · metalgemm",
 * Thm 1). Y is bf16 (y_fp32 == 0) or fp32. K % 8 == 0, N % 8 == 0 (16-byte
 * rows). No scratch memory. */
fk_status fk_gemm_bf16(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N, void* d_y,
                       int32_t y_fp32, void* stream);

/* The same product for few rows (1 <= P <= 64, the decode and short-prompt
 * regime) on the weight-streaming kernel: the weight tile is the 128-row side
 * of the tensor-core MMA, K is split across CTAs, and the fp32 partial sums
 * (d_scratch, fk_gemm_bf16_splitk_scratch_bytes(P, K, N) bytes) are added in
 * a fixed order, so results are bitwise reproducible. */
size_t fk_gemm_bf16_splitk_scratch_bytes(int32_t P, int32_t K, int32_t N);
fk_status fk_gemm_bf16_splitk(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N, void* d_y,
                              int32_t y_fp32, void* d_scratch, size_t scratch_bytes, void* stream);

/* Prefill attention: seq new queries per sequence at positions
 * pos0..pos0+seq-1 over cached keys/values at positions 0..pos0+seq-1
 * ("N7 · model/forward-parity", Thm 1: causal GQA attention; "pegainfer
 * #878": sliding window, query i sees key j iff 0 <= i-j < window).
 *   d_q:   bf16 [batch*seq][n_q_heads*head_dim] (RoPE applied)
 *   caches as for fk_attention_decode (K [batch][n_kv_heads][cap][head_dim],
 *          V transposed [batch][n_kv_heads][head_dim][cap], cap % 64 == 0,
 *          position p in slot p mod cap, every slot finite); either
 *          pos0 + seq <= cap, or (a sliding-window ring) window > 0 and
 *          window + seq - 1 <= cap
 *   d_out: bf16 [batch*seq][n_q_heads*head_dim]
 * head_dim 64, 128 or 256, on the tensor-core (tcgen05) kernel. No scratch. */
fk_status fk_attention_prefill(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch, int32_t seq,
                               int32_t pos0, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t cap,
                               int32_t window, void* d_out, void* stream);

/* Decode attention of one query per sequence ("N7 · model/forward-parity",
 * Thm 1: causal GQA attention; "pegainfer #878": sliding-window layers).
 *   d_q:      bf16 [batch][n_q_heads*head_dim], the query at position ctx-1
 *   d_kcache: bf16 [batch][n_kv_heads][cap][head_dim], keys at positions
 *             0..ctx-1 (RoPE already applied), position p in slot p mod cap
 *   d_vcache: bf16 [batch][n_kv_heads][head_dim][cap], values transposed
 *             (position fastest); cap a multiple of 64, every slot finite;
 *             ctx <= cap, or (a sliding-window ring) window > 0 and
 *             window <= cap
 *   window:   0 = attend to all ctx keys; W > 0 = only the last W
 *   d_out:    bf16 [batch][n_q_heads*head_dim]
 * Query head h reads kv head h / (n_q_heads/n_kv_heads); scale 1/sqrt(head_dim).
 * Split-KV: the splits of a (sequence, kv head) run as one thread-block
 * cluster and merge their partials in the cluster's shared memory in a fixed
 * order, so results are bitwise reproducible and no scratch memory is used.
 * head_dim is 64, 128 or 256; 1..8 query heads per kv head. */
fk_status fk_attention_decode(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch,
                              int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t cap, int32_t ctx,
                              int32_t window, void* d_out, void* stream);

/* Op hooks: one step of the path alone, on the kernels the forward uses, for
 * per-step parity ("N9 · metalgemm", Thm 1: op-level parity of each device
 * op, not only of the chain).
 *
 * fk_op_rmsnorm ("N7 · model/forward-parity", Thm 1: RMSNorm):
 *   d_out[r] = d_x[r] / sqrt(mean(d_x[r]^2) + eps) * d_w, rounded to bf16.
 *   d_x fp32 [rows][hidden], d_w bf16 [hidden], d_out bf16 [rows][hidden];
 *   hidden a positive multiple of 8, eps > 0. */
fk_status fk_op_rmsnorm(const float* d_x, int32_t rows, int32_t hidden, const void* d_w, float eps, void* d_out,
                        void* stream);

/* fk_op_rope ("N7", Thm 1: RoPE on q and k; Thm 2: QK-norm, llama3 scaling,
 * local/global RoPE bases): for `layer` of model m, on d_qkv bf16
 * [batch*seq][(n_q_heads + 2 n_kv_heads) head_dim] (rows of [q | k | v] heads,
 * token t = b*seq + s at position pos0 + s): [QK-norm with the layer's
 * q_norm/k_norm when the config has qk_norm, then] RoPE with the layer kind's
 * base (and scaling) rotates q in place and writes the rotated k to d_kcache
 * bf16 [batch][n_kv_heads][cap][head_dim] and v, transposed, to d_vcache bf16
 * [batch][n_kv_heads][head_dim][cap] at positions pos0..pos0+seq-1. Other
 * cache positions are untouched. pos0 + seq <= cap, cap % 64 == 0, and
 * pos0 + seq <= the model's max_positions (FK_ERR_CONTEXT_FULL otherwise).
 * d_qkv and the caches hold IEEE f16 instead of bf16 when the model's
 * f16_sites has FK_F16_ATTN. */
fk_status fk_op_rope(fk_model* m, int32_t layer, void* d_qkv, int32_t batch, int32_t seq, int32_t pos0,
                     void* d_kcache, void* d_vcache, int32_t cap, void* stream);

/* fk_op_head_argmax ("N7", Thm 1: head matmul to logits and per-position
 * argmax; "pegainfer #878": final-logit softcap): d_logits fp32
 * [rows][vocab] = softcap(d_u · headᵀ) with the model's (tied or untied)
 * head, d_u bf16 [rows][hidden] (final-norm output); d_argmax (NULL or int32
 * [rows]) the lowest index of each row maximum; d_margin (NULL or fp32 [rows],
 * needs d_argmax) the row maximum minus the largest other logit. d_u is IEEE
 * f16 instead of bf16 when the model's f16_sites has FK_F16_HEAD_IN. */
fk_status fk_op_head_argmax(fk_model* m, const void* d_u, int32_t rows, float* d_logits, int32_t* d_argmax,
                            float* d_margin, void* stream);

/* fk_op_logsoftmax_topk ("pegainfer issue #878", Acceptance Criteria: the
 * distributional gate reads log-probabilities at each position's top-64
 * ids): for each of `rows` fp32 logit rows (d_logits, row stride ld >= vocab):
 *   d_lse (NULL or fp32 [rows]):     lse = max + log(sum(exp(z - max)))
 *   d_top_ids (int32 [rows][k]):     the k largest logits' ids, by value
 *                                    descending, ties to the lower id
 *   d_top_logprobs (fp32 [rows][k]): z[id] - lse at those ids
 *   d_logprobs (NULL or fp32 [rows][vocab]): the whole log-softmax row
 * 1 <= k <= min(128, vocab). Logits must be finite. */
fk_status fk_op_logsoftmax_topk(const float* d_logits, int32_t rows, int32_t vocab, int32_t ld, int32_t k,
                                float* d_lse, int32_t* d_top_ids, float* d_top_logprobs, float* d_logprobs,
                                void* stream);

/* fk_op_moe_route ("N7 · model/forward-parity", Thm 2: qwen3moe routing):
 * for each of T rows of fp32 router logits z (d_logits, row stride ld >= E):
 *   p = softmax(z) over the E experts (fp32);
 *   d_ids (int32 [T][k]): the k experts of largest z -- the order of p --
 *       by value descending, ties to the lower id; or, when d_forced (NULL or
 *       int32 [T][k]) is given, its ids for that row (a row whose forced ids
 *       are out of [0, E) or repeated routes itself instead and sets
 *       FK_DEVERR_EXPERT_IDS in the op-level error word);
 *   d_weights (fp32 [T][k]): p at those ids, divided by their sum when
 *       norm_topk;
 *   d_margin (NULL or fp32 [T]): p of the k-th minus p of the (k+1)-th
 *       largest logit of the row's own ranking (+inf when k == E).
 * 1 <= E <= 256, 1 <= k <= min(E, 16). */
fk_status fk_op_moe_route(const float* d_logits, int32_t T, int32_t E, int32_t ld, int32_t k, int32_t norm_topk,
                          const int32_t* d_forced, int32_t* d_ids, float* d_weights, float* d_margin, void* stream);

/* fk_op_moe_ffn ("N7", Thm 2: the qwen3moe FFN): the mixture-of-experts FFN
 * of MoE layer `layer` of model m on d_u [T][hidden] (the FFN norm output,
 * bf16, or f16 when f16_sites has FK_F16_FFN_IN): router logits u·routerᵀ,
 * routing as fk_op_moe_route (d_forced NULL or int32 [T][k]), then
 *   d_out[t] (fp32 [T][hidden]) = sum_j w[t][j] * down_e(act(gate_e u) * up_e u)
 * over the k chosen experts e = ids[t][j], j ascending, the gated activation
 * stored as bf16 (f16 with FK_F16_FFN_ACT) before the down projection.
 * d_ids (NULL or int32 [T][k]) and d_margin (NULL or fp32 [T]) receive the
 * routing. The workspace (256-byte aligned) holds at least
 * fk_op_moe_ffn_workspace_bytes(m, T) bytes. */
size_t fk_op_moe_ffn_workspace_bytes(const fk_model* m, int32_t T);
fk_status fk_op_moe_ffn(fk_model* m, int32_t layer, const void* d_u, int32_t T, const int32_t* d_forced, float* d_out,
                        int32_t* d_ids, float* d_margin, void* d_ws, size_t ws_bytes, void* stream);

/* Routing hook of the forward, the session prefill and decode. With d_forced
 * set, the i-th MoE layer (counting MoE layers only, from 0) of each later
 * call takes its expert ids from d_forced + i*max_tokens*k (int32
 * [tokens][k], tokens = batch*seq of fk_forward, the chunk of
 * fk_session_prefill, the batch of fk_decode_step, tokens in [batch][seq]
 * order); its weights still come from its own router. d_trace_ids (int32,
 * same layout) and d_trace_margin (fp32 [n_moe_layers][max_tokens]) receive
 * each MoE layer's routing. While the hook is set, calls with more than
 * max_tokens tokens, and prefills longer than the session's max_chunk, fail
 * with FK_ERR_INVALID_ARG, and decode steps run without a CUDA graph. All
 * NULL clears the hook. For parity tests; not for production use. */
fk_status fk_model_set_moe_routing(fk_model* m, const int32_t* d_forced, int32_t* d_trace_ids, float* d_trace_margin,
                                   int32_t max_tokens);

/* Allocation-free fk_gemm_bf16_splitk. The pages have no counterpart: this
 * entry point serves callers that cannot hand the library a scratch buffer --
 * their device memory belongs to another allocator that must remain its only
 * owner, or their path must never enter the driver's allocation code. The
 * split partial sums and arrival counters live in one fixed array of
 * fk_gemm_bf16_splitk_noalloc_limit() bytes (8 MiB) inside the library's
 * device image, which every GPU that loads the library holds until the
 * process exits. Arguments and results are those of fk_gemm_bf16_splitk
 * without the scratch; a shape whose scratch
 * (fk_gemm_bf16_splitk_scratch_bytes) exceeds the limit is rejected with
 * FK_ERR_WORKSPACE before anything is launched. The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 * Every call on a device shares the array and leaves its contents behind;
 * each call clears the counters it needs on its own stream. Calls whose
 * kernels overlap on the GPU (other streams, other host threads) race on the
 * array: serialise them. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make it
 * before any stream capture begins on that device. */
size_t fk_gemm_bf16_splitk_noalloc_limit(void);
fk_status fk_gemm_bf16_splitk_noalloc(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N, void* d_y,
                                      int32_t y_fp32, void* stream);

/* ---------------------------------------------------------------------------
 * Testing hook (failure detection)
 * Sets the test controls of the current device's op-level control block:
 * stall_first_stage != 0 makes fk_gemm_bf16_splitk leave its first pipeline
 * stage unarmed, so the tensor-core issuer's bounded wait on it runs out;
 * wait_limit_us > 0 replaces the 2 s limit of every bounded wait in op-level
 * calls. The kernel then gives up, leaves its output undefined, sets
 * FK_DEVERR_PIPE_TIMEOUT and returns; fk_sync_status(NULL, ...) reports it.
 * (0, 0) restores normal operation. Not for production use.
 * ------------------------------------------------------------------------- */
fk_status fk_debug_set_op_pipe_fault(int32_t stall_first_stage, int32_t wait_limit_us);

/* ---------------------------------------------------------------------------
 * Kernel timing (tracing)
 * When enabled, every kernel launch of the entry points above is bracketed by
 * CUDA events on its stream and filed under a kernel-class name ("gemm_qkv",
 * "attn_prefill", ...). Not for use while a stream is being captured into a
 * CUDA graph. Process-wide; thread-safe.
 * ------------------------------------------------------------------------- */
void fk_profile_enable(int32_t on);
/* Drop every recorded launch. */
void fk_profile_reset(void);
/* Wait for the recorded events, then return the number of kernel classes. */
int32_t fk_profile_count(void);
/* Class i (0 <= i < fk_profile_count()): name (static storage until the next
 * reset), launches and their summed device time in milliseconds. */
fk_status fk_profile_get(int32_t i, const char** name, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* FK_H */
