// The forward pass behind the C ABI: model binding, the layer loop shared by
// the cacheless forward, session prefill and decode, and the LM head.
//
// Per layer, pre-norm layout ("N7 · model/forward-parity", Thm 1):
//   qkv = u·[Wq;Wk;Wv]ᵀ          GEMM, stacked weights, bf16 out
//   q,k <- [QK-norm] RoPE        k, v -> KV cache
//   o   = attention(q, K, V)     causal GQA [sliding window]
//   x'  = x + o·Woᵀ              GEMM, fp32 residual epilogue
//   u   = RMSNorm(x')·w_ffn
//   h   = act(u·Wgᵀ) ⊙ (u·Wuᵀ)   GEMM, gate/up interleaved, fused activation
//   x'' = x' + h·Wdᵀ             GEMM, fp32 residual epilogue
//   u   = RMSNorm(x'')·w_next    (next layer's attn norm, or the final norm)
// Sandwich layout ("N7", Thm 2, gemma3): the O and down GEMMs write fp32 and a
// fused kernel adds RMSNorm(a)·w_post to the residual and normalises the sum.
// Mixture-of-experts layers ("N7", Thm 2, qwen3moe) replace the gated FFN by
// the routed experts of moe.cu, whose output is added to the residual.
#include <chrono>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include <cuda_bf16.h>

#include "fk_internal.h"
#include "fk_ops.h"
#include "fk_launch.h"

using namespace fk;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Scratch {
  int32_t* ids = nullptr;  // [T]
  float* x0 = nullptr;     // [T, H] residual
  float* x1 = nullptr;     // [T, H] residual (mid-layer)
  float* a = nullptr;      // [T, H] sandwich pre-norm outputs
  void* u = nullptr;       // [T, H] bf16 normalised rows
  void* qkv = nullptr;     // [T, Nq + 2 Nkv] bf16
  void* ao = nullptr;      // [T, Nq] bf16 attention output
  void* h = nullptr;       // [T, I] bf16 gated FFN activations
  void* gemv = nullptr;    // split-K counters + partial sums of the few-token GEMMs
  size_t gemv_bytes = 0;
  size_t gemv_counter_bytes = 0;  // leading counters, zero between launches
  void* argmax = nullptr;         // split-row argmax partials + per-row counters (zero between launches)
  float* ssq = nullptr;           // decode of <= 2 tokens: residual rows' group sums of squares for a fused norm
  MoeScratch moe;                 // MoE layers' routing and expert buffers (when the model has any)
};

}  // namespace

struct fk_model {
  fk_config cfg{};
  std::vector<uint8_t> kinds;
  std::vector<fk_layer_weights> layers;
  const void* embed = nullptr;
  const void* head = nullptr;
  const void* final_norm = nullptr;
  int max_pos = 0;
  unsigned* dev_err = nullptr;
  float2* rope[2] = {nullptr, nullptr};  // cos/sin tables per layer kind
  std::vector<GemmWeights> g_qkv, g_o, g_gu, g_down;
  GemmWeights g_head;
  int Nq = 0, Nkv = 0, Nqkv = 0;
  float embed_scale = 1.f;
  float attn_scale = 1.f;
  int sm_count = 0;
  bool has_local = false;
  // mixture-of-experts layers: moe_index[l] = the layer's index among the MoE
  // layers, -1 for a dense layer
  std::vector<uint8_t> moe_kinds;
  std::vector<int> moe_index;
  std::vector<MoeWeights> moe;
  int n_moe = 0;
  // routing hook (fk_model_set_moe_routing)
  const int32_t* moe_forced = nullptr;
  int32_t* moe_trace_ids = nullptr;
  float* moe_trace_margin = nullptr;
  int moe_hook_tokens = 0;
  bool moe_hook() const { return moe_forced || moe_trace_ids || moe_trace_margin; }
  // 1 when the activation storage site (an FK_F16_* bit) holds IEEE f16
  int f16(uint32_t site) const { return (cfg.f16_sites & site) ? 1 : 0; }
  // cacheless forwards of few tokens: the second call with the same shape,
  // workspace and outputs captures the launches after the ids copy into a
  // CUDA graph, which later such calls replay (fk_forward); kFwdGraphs keys
  // are kept
  struct FwdKey {
    int B = 0, S = 0;
    const void* ws = nullptr;
    const void* out[4] = {nullptr, nullptr, nullptr, nullptr};
    bool operator==(const FwdKey& o) const {
      return B == o.B && S == o.S && ws == o.ws && out[0] == o.out[0] && out[1] == o.out[1] &&
             out[2] == o.out[2] && out[3] == o.out[3];
    }
  };
  // a few most recent keys: a caller alternating between output buffers
  // still finds its graphs (least recently used entry replaced)
  static constexpr int kFwdGraphs = 4;
  struct FwdEntry {
    FwdKey key;
    cudaGraphExec_t exec = nullptr;  // null: seen once, not captured yet
    bool used = false;
    unsigned long long last = 0;
  };
  std::mutex fwd_mu;
  cudaStream_t fwd_cap_stream = nullptr;
  FwdEntry fwd[kFwdGraphs];
  unsigned long long fwd_clock = 0;
  ~fk_model() {
    for (FwdEntry& e : fwd)
      if (e.exec) cudaGraphExecDestroy(e.exec);
    if (fwd_cap_stream) cudaStreamDestroy(fwd_cap_stream);
  }
};

struct fk_session {
  fk_model* m = nullptr;
  int B = 0, max_seq = 0, max_chunk = 0;
  int len = 0;
  // per layer l: K cache [B][Hkv][cap_l][hd] at kcache + kv_off[l] bytes, V
  // cache transposed [B][Hkv][hd][cap_l] at vcache + kv_off[l]. Position p
  // lives in slot p mod cap_l: cap_l is max_seq rounded up to 64 on global
  // layers and a ring of W + max_chunk - 1 positions (rounded up to 64, at
  // most the global cap) on sliding-window layers.
  uint8_t* kcache = nullptr;
  uint8_t* vcache = nullptr;
  std::vector<size_t> kv_off;
  std::vector<int> kv_cap;
  size_t kv_bytes = 0;  // bytes of all layers' K caches (= of the V caches)
  Scratch sc;
  int32_t* next_ids = nullptr;  // [B]
  float* logits = nullptr;      // [B, V]
  void* u_last = nullptr;       // [B, H] bf16
  int dec_splits = 1;  // decode attention: CTAs per (sequence, kv head) cluster
  int* d_len = nullptr;          // device copy of len (read by decode kernels)
  bool d_len_valid = false;      // false after reset until the next prefill
  // captured decode step (feeds the previous greedy ids), keyed by outputs
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t graph = nullptr;
  float* graph_logits = nullptr;
  int32_t* graph_next = nullptr;
  float* graph_margin = nullptr;
};

namespace {

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
// 1 for each MoE layer (all layers when moe_layers is NULL and there are experts)
bool is_moe_layer(const fk_config* c, int l) {
  if (c->n_experts <= 0) return false;
  return c->moe_layers ? c->moe_layers[l] == 1 : true;
}

bool has_dense_layer(const fk_config* c) {
  for (int l = 0; l < c->n_layers; ++l)
    if (!is_moe_layer(c, l)) return true;
  return false;
}

fk_status validate_config(const fk_config* c) {
  if (!c) return fail(FK_ERR_INVALID_ARG, "config is NULL");
  auto bad = [](const char* m) { return fail(FK_ERR_INVALID_CONFIG, m); };
  if (c->n_layers < 1) return bad("n_layers must be >= 1");
  if (c->n_experts < 0) return bad("n_experts must be >= 0");
  if (c->n_experts == 0) {
    if (c->moe_layers)
      for (int l = 0; l < c->n_layers; ++l)
        if (c->moe_layers[l]) return bad("moe_layers marks a MoE layer but n_experts is 0");
  } else {
    if (c->n_experts % 8 || c->n_experts > kMoeMaxExperts) return bad("n_experts must be a multiple of 8, at most 256");
    if (c->n_experts_per_tok < 1 || c->n_experts_per_tok > std::min(c->n_experts, kMoeMaxK))
      return bad("n_experts_per_tok must be in [1, min(n_experts, 16)]");
    if (c->expert_intermediate < 64 || c->expert_intermediate % 64)
      return bad("expert_intermediate must be a positive multiple of 64");
    if (c->norm_topk != 0 && c->norm_topk != 1) return bad("norm_topk must be 0 or 1");
    if (c->moe_layers)
      for (int l = 0; l < c->n_layers; ++l)
        if (c->moe_layers[l] > 1) return bad("moe_layers entries must be 0 (dense) or 1 (MoE)");
  }
  if (c->hidden < 64 || c->hidden % 64) return bad("hidden must be a positive multiple of 64");
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads)
    return bad("n_q_heads must be a positive multiple of n_kv_heads");
  if (c->n_q_heads / c->n_kv_heads > 8) return bad("more than 8 query heads per kv head");
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return bad("head_dim must be 64, 128 or 256");
  if (has_dense_layer(c) && (c->intermediate < 64 || c->intermediate % 64))
    return bad("intermediate must be a positive multiple of 64");
  if (c->vocab < 8 || c->vocab % 8) return bad("vocab must be a positive multiple of 8");
  if (!(c->rms_eps > 0.f) || !std::isfinite(c->rms_eps)) return bad("rms_eps must be > 0");
  if (!(c->rope_theta_global > 1.0) || !(c->rope_theta_local > 1.0)) return bad("rope thetas must be > 1");
  if (c->rope_scaling != FK_ROPE_NONE && c->rope_scaling != FK_ROPE_LLAMA3) return bad("unknown rope_scaling");
  if (c->rope_scaling == FK_ROPE_LLAMA3 &&
      (!(c->rope_factor >= 1.f) || !(c->rope_low_freq_factor > 0.f) ||
       !(c->rope_high_freq_factor > c->rope_low_freq_factor) || c->rope_orig_max_pos <= 0))
    return bad("llama3 rope scaling parameters out of range");
  if (c->act != FK_ACT_SILU && c->act != FK_ACT_GELU_TANH) return bad("unknown act");
  if (c->norm_layout != FK_NORM_PRE && c->norm_layout != FK_NORM_SANDWICH) return bad("unknown norm_layout");
  if (c->qk_norm != 0 && c->qk_norm != 1) return bad("qk_norm must be 0 or 1");
  if (c->sliding_window < 0) return bad("sliding_window must be >= 0");
  if (c->embed_scale != FK_EMBED_SCALE_NONE && c->embed_scale != FK_EMBED_SCALE_SQRT_HIDDEN_BF16)
    return bad("unknown embed_scale");
  // "pegainfer #878": the final-logit softcap is validated positive at parse
  if (!std::isfinite(c->final_softcap) || c->final_softcap < 0.f) return bad("final_softcap must be 0 (off) or > 0");
  if (c->tied != 0 && c->tied != 1) return bad("tied must be 0 or 1");
  if (c->f16_sites & ~FK_F16_ALL) return bad("f16_sites has bits outside FK_F16_ALL");
  if (c->layer_kinds) {
    for (int l = 0; l < c->n_layers; ++l) {
      if (c->layer_kinds[l] > 1) return bad("layer_kinds entries must be 0 (global) or 1 (local)");
      if (c->layer_kinds[l] == 1 && c->sliding_window == 0) return bad("local layer without a sliding_window");
    }
  }
  return FK_OK;
}

bool has_local(const fk_config* c) {
  if (!c->layer_kinds) return false;
  for (int l = 0; l < c->n_layers; ++l)
    if (c->layer_kinds[l] == 1) return true;
  return false;
}

// Arena: [control block | rope table global | rope table local | f16 weight copies]
size_t rope_table_bytes(const fk_config* c, int max_pos) {
  return align_up((size_t)max_pos * (c->head_dim / 2) * sizeof(float2));
}

// Bytes of the f16 copies of the weights whose GEMM input site is f16: per
// layer Wq, Wk, Wv (FK_F16_QKV_IN), Wo (FK_F16_O_IN), W_gate, W_up
// (FK_F16_FFN_IN), W_down (FK_F16_FFN_ACT); the head (FK_F16_HEAD_IN).
// MoE layers: the router and the experts' gate/up matrices (FK_F16_FFN_IN),
// the experts' down matrices (FK_F16_FFN_ACT).
size_t f16_copy_bytes(const fk_config* c) {
  const size_t H = c->hidden, I = c->intermediate, Nq = (size_t)c->n_q_heads * c->head_dim,
               Nkv = (size_t)c->n_kv_heads * c->head_dim, E = std::max(c->n_experts, 0),
               Ie = std::max(c->expert_intermediate, 0);
  size_t b = 0;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->f16_sites & FK_F16_QKV_IN) b += align_up(Nq * H * 2) + 2 * align_up(Nkv * H * 2);
    if (c->f16_sites & FK_F16_O_IN) b += align_up(H * Nq * 2);
    if (is_moe_layer(c, l)) {
      if (c->f16_sites & FK_F16_FFN_IN) b += align_up(E * H * 2) + 2 * align_up(E * Ie * H * 2);
      if (c->f16_sites & FK_F16_FFN_ACT) b += align_up(E * H * Ie * 2);
    } else {
      if (c->f16_sites & FK_F16_FFN_IN) b += 2 * align_up(I * H * 2);
      if (c->f16_sites & FK_F16_FFN_ACT) b += align_up(H * I * 2);
    }
  }
  if (c->f16_sites & FK_F16_HEAD_IN) b += align_up((size_t)c->vocab * H * 2);
  return b;
}

// bf16(sqrt(hidden)) by round-to-nearest-even on the float bits ("pegainfer
// #878": derive the embedding scale and assert its recorded bf16 value)
float bf16_round(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  u &= 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, 4);
  return r;
}

// RoPE frequencies f_j (j < hd/2) of one layer kind, in double. llama3
// scaling: wavelength lam = 2*pi/f; lam < C/b keeps f; lam > C/a gives f/s;
// between, t = (C/lam - a)/(b - a) blends f/s and f as (1-t) f/s + t f.
void rope_freqs(const fk_config* c, int kind, std::vector<double>& f) {
  const int half = c->head_dim / 2;
  const double theta = kind == 1 ? c->rope_theta_local : c->rope_theta_global;
  f.resize(half);
  for (int j = 0; j < half; ++j) {
    double fj = std::pow(theta, -2.0 * j / c->head_dim);
    if (c->rope_scaling == FK_ROPE_LLAMA3) {
      const double C = c->rope_orig_max_pos, a = c->rope_low_freq_factor, b = c->rope_high_freq_factor,
                   s = c->rope_factor;
      const double lam = 2.0 * M_PI / fj;
      if (lam > C / a) {
        fj = fj / s;
      } else if (lam >= C / b) {
        const double t = (C / lam - a) / (b - a);
        fj = (1.0 - t) * fj / s + t * fj;
      }
    }
    f[j] = fj;
  }
}

size_t scratch_bytes(const fk_model* m, long T, Scratch* s, uint8_t* base) {
  const fk_config& c = m->cfg;
  size_t off = 0;
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  Scratch t;
  t.ids = reinterpret_cast<int32_t*>(take((size_t)T * 4));
  t.x0 = reinterpret_cast<float*>(take((size_t)T * c.hidden * 4));
  t.x1 = reinterpret_cast<float*>(take((size_t)T * c.hidden * 4));
  if (c.norm_layout == FK_NORM_SANDWICH) t.a = reinterpret_cast<float*>(take((size_t)T * c.hidden * 4));
  t.u = take((size_t)T * c.hidden * 2);
  t.qkv = take((size_t)T * m->Nqkv * 2);
  t.ao = take((size_t)T * m->Nq * 2);
  if (has_dense_layer(&c)) t.h = take((size_t)T * c.intermediate * 2);
  // few-token GEMMs (T <= 64, or decode/short chunks up to that size) need
  // split-K scratch: one counter region sized for the GEMM with the most
  // tiles, then room for the largest GEMM's partial sums
  const int Ms = (int)std::min<long>(T, kSkinnyMaxTokens);
  size_t gb = 0, cb = 0;
  if (!m->g_qkv.empty()) {
    // every layer's GEMMs have the shapes of layer 0's, or of the first
    // dense layer's and the MoE router's
    std::vector<const GemmWeights*> all = {&m->g_qkv[0], &m->g_o[0], &m->g_head};
    for (int l = 0; l < c.n_layers; ++l)
      if (m->moe_index[l] < 0) {
        all.push_back(&m->g_gu[l]);
        all.push_back(&m->g_down[l]);
        break;
      }
    if (m->n_moe) all.push_back(&m->moe[0].router);
    size_t pb = 0;
    for (const GemmWeights* g : all) {
      cb = std::max(cb, skinny_counter_bytes(*g, Ms, m->sm_count));
      pb = std::max(pb, skinny_partial_bytes(*g, Ms, m->sm_count));
    }
    gb = cb + pb;
  }
  t.gemv_bytes = gb;
  t.gemv_counter_bytes = cb;
  t.gemv = gb ? take(gb) : nullptr;
  t.argmax = take(argmax_scratch_bytes());
  t.ssq = reinterpret_cast<float*>(take((size_t)kNormFuseMaxTokens * ((c.hidden + 127) / 128) * 4));
  if (m->n_moe) off += moe_scratch(m->moe[0], T, &t.moe, base ? base + off : nullptr);
  if (s) *s = t;
  return off;
}

struct KV {
  uint8_t* k = nullptr;           // [B][Hkv][cap][hd] per layer
  uint8_t* v = nullptr;           // transposed: [B][Hkv][hd][cap] per layer
  const size_t* off = nullptr;    // per-layer byte offsets (null: one buffer reused by every layer)
  const int* caps = nullptr;      // per-layer capacities (null: `cap` on every layer)
  int cap = 0;                    // positions per (sequence, kv head), a multiple of 64
  size_t bytes = 0;               // bytes of one of k / v (all layers)
  void* kl(int l) const { return k + (off ? off[l] : 0); }
  void* vl(int l) const { return v + (off ? off[l] : 0); }
  int cap_of(int l) const { return caps ? caps[l] : cap; }
};

#define FK_LAUNCH(expr)                                 \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
  } while (0)
#define FK_TRY(expr)                \
  do {                              \
    fk_status _s = (expr);          \
    if (_s != FK_OK) return _s;     \
  } while (0)

// The decoder stack over T = B*S tokens at positions pos0 .. pos0+S-1 of
// each sequence. Reads sc.ids; leaves the final-normed rows (bf16) in sc.u.
// slots (optional): fp32 [L+2][T][H] hidden states. decode: S == 1, attention
// through the split-KV cluster kernel with dsplits CTAs per cluster.
fk_status run_stack(fk_model* m, const Scratch& sc, int B, int S, int pos0, const KV& kv, float* slots,
                    bool decode, int dsplits, cudaStream_t st,
                    const int* d_len = nullptr, const int32_t* ids = nullptr) {
  const fk_config& c = m->cfg;
  const int H = c.hidden, L = c.n_layers, hd = c.head_dim;
  const long T = (long)B * S;
  const bool sandwich = c.norm_layout == FK_NORM_SANDWICH;
  float* x_in = slots ? slots : sc.x0;
  if (m->moe_hook() && T > m->moe_hook_tokens)
    return fail(FK_ERR_INVALID_ARG, "more tokens than the MoE routing hook holds");
  // Layer GEMMs of decode steps stream weights through the split-K kernel.
  // Prefill (any chunk size) keeps the tiled kernel, whose per-element
  // summation order does not depend on the row count: chunked cached prefill
  // then rounds every bf16 activation exactly as the cacheless forward does.
  void* gv = decode ? sc.gemv : nullptr;
  const size_t gvb = decode ? sc.gemv_bytes : 0;
  // Decode steps of one or two sequences run the RMSNorm in front of a dense
  // layer's gate/up projection, and in front of the next layer's QKV
  // projection, inside those GEMMs: the norm kernels and their launch
  // boundaries drop out of the step's dependency chain.
  const bool fuse_norm = decode && !sandwich && T <= kNormFuseMaxTokens;
  NormIn qkv_norm;  // the fused norm of the next QKV projection, when set
  bool qkv_norm_set = false;
  { ProfScope ps(decode ? "embed_norm_dec" : "embed_norm", st);
  FK_LAUNCH(launch_embed_norm(ids ? ids : sc.ids, m->embed, (int)T, H, c.vocab, m->embed_scale, m->layers[0].attn_norm, c.rms_eps,
                              x_in, sc.u, m->dev_err, st, m->f16(FK_F16_QKV_IN))); }
  for (int l = 0; l < L; ++l) {
    const fk_layer_weights& w = m->layers[l];
    const int kind = m->kinds[l];
    const int window = kind == 1 ? c.sliding_window : 0;
    float* x_out = slots ? slots + (size_t)(l + 1) * T * H : sc.x0;
    // A dense pre-norm layer keeps the residual stream in one buffer: the
    // down projection adds into x_out in place (as does the attention output
    // projection when x_out is x_in), which the tiled GEMM turns into TMA
    // reduce-adds instead of residual loads.
    const bool in_place = !sandwich && m->moe_index[l] < 0;
    float* x_mid = in_place ? x_out : sc.x1;
    const void* next_norm = l + 1 < L ? m->layers[l + 1].attn_norm : m->final_norm;
    // the next norm output feeds the next layer's QKV projection, or the LM head
    const int next_f16 = l + 1 < L ? m->f16(FK_F16_QKV_IN) : m->f16(FK_F16_HEAD_IN);
    void* kl = kv.kl(l);
    void* vl = kv.vl(l);
    const int cap = kv.cap_of(l);

    GemmOut o;
    o.epi = EPI_BF16;
    o.out_f16 = m->f16(FK_F16_ATTN);
    o.out = sc.qkv;
    o.ldo = m->Nqkv;
    { ProfScope ps(decode ? "gemm_qkv_dec" : "gemm_qkv", st); FK_TRY(gemm_run(sc.u, (int)T, H, m->g_qkv[l], o, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes, qkv_norm_set ? &qkv_norm : nullptr)); }
    qkv_norm_set = false;
    const bool fuse_ffn_norm = fuse_norm && m->moe_index[l] < 0;
    NormIn ffn_norm;
    ffn_norm.x = x_mid;
    ffn_norm.ldx = H;
    ffn_norm.w = w.ffn_norm;
    ffn_norm.eps = c.rms_eps;
    if (decode) {  // RoPE, cache write and attention in one kernel
      ProfScope ps("attn_decode", st);
      FK_LAUNCH(launch_attention_decode_rope(sc.qkv, m->Nqkv, kl, vl, cap, B, d_len, c.n_q_heads, c.n_kv_heads,
                                             hd, window, m->attn_scale, m->rope[kind], c.qk_norm, w.q_norm, w.k_norm,
                                             c.rms_eps, dsplits, sc.ao, m->dev_err, st, m->f16(FK_F16_ATTN),
                                             m->f16(FK_F16_O_IN)));
    } else {
      { ProfScope ps("rope_qkv", st);
      FK_LAUNCH(launch_rope_qkv(sc.qkv, m->Nqkv, (int)T, S, pos0, c.n_q_heads, c.n_kv_heads, hd,
                                m->rope[kind], c.qk_norm, w.q_norm, w.k_norm, c.rms_eps, kl, vl, cap, st,
                                m->f16(FK_F16_ATTN))); }
      ProfScope ps("attn_prefill", st);
      FK_TRY(attention_prefill_tc(sc.qkv, m->Nqkv, kl, vl, cap, B, S, pos0, c.n_q_heads, c.n_kv_heads, hd, window,
                                  m->attn_scale, sc.ao, m->dev_err, st, m->f16(FK_F16_ATTN), m->f16(FK_F16_O_IN)));
    }
    // attention output projection + residual
    if (sandwich) {
      o.epi = EPI_F32;
      o.out = sc.a;
      o.ldo = H;
      o.softcap = 0.f;
      { ProfScope ps(decode ? "gemm_o_dec" : "gemm_o", st); FK_TRY(gemm_run(sc.ao, (int)T, m->Nq, m->g_o[l], o, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes)); }
      ProfScope ps(decode ? "post_norm_dec" : "post_norm", st);
      FK_LAUNCH(launch_post_norm_residual(sc.a, x_in, x_mid, (int)T, H, w.post_attn_norm, w.ffn_norm, c.rms_eps, sc.u,
                                          st, m->f16(FK_F16_FFN_IN)));
    } else {
      o.epi = EPI_ADD_F32;
      o.out = x_mid;
      o.ldo = H;
      o.res = x_in;
      o.ldr = H;
      if (fuse_ffn_norm && skinny_fused_tail(m->g_o[l], (int)T, m->sm_count, EPI_ADD_F32)) {
        o.ssq = sc.ssq;  // the gate/up projection's fused norm reads the row statistics from here
        ffn_norm.ssq = sc.ssq;
        ffn_norm.n_ssq = (H + 127) / 128;
      }
      { ProfScope ps(decode ? "gemm_o_dec" : "gemm_o", st); FK_TRY(gemm_run(sc.ao, (int)T, m->Nq, m->g_o[l], o, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes)); }
      if (!fuse_ffn_norm) {
        ProfScope ps(decode ? "rmsnorm_dec" : "rmsnorm", st);
        FK_LAUNCH(launch_rmsnorm(x_mid, H, (int)T, H, w.ffn_norm, c.rms_eps, sc.u, H, st, m->f16(FK_F16_FFN_IN)));
      }
    }
    const int mi = m->moe_index[l];
    if (mi >= 0) {
      // mixture-of-experts FFN: out = x_mid + sum of the routed experts (pre-norm) or the sum alone (sandwich)
      const MoeWeights& mw = m->moe[mi];
      const size_t hook_rows = (size_t)m->moe_hook_tokens * mw.k;
      const int32_t* forced = m->moe_forced ? m->moe_forced + (size_t)mi * hook_rows : nullptr;
      int32_t* t_ids = m->moe_trace_ids ? m->moe_trace_ids + (size_t)mi * hook_rows : nullptr;
      float* t_margin = m->moe_trace_margin ? m->moe_trace_margin + (size_t)mi * m->moe_hook_tokens : nullptr;
      // pre-norm: the combine step also makes the next consumer's normalised rows
      NormOut nn;
      nn.w = next_norm;
      nn.eps = c.rms_eps;
      nn.u = sc.u;
      nn.f16 = next_f16;
      FK_TRY(moe_ffn_run(mw, sc.u, (int)T, sc.moe, forced, t_ids, t_margin, sandwich ? sc.a : x_out,
                         sandwich ? nullptr : x_mid, m->dev_err, st, decode, gv, gvb, sc.gemv_counter_bytes,
                         sandwich ? nullptr : &nn));
      if (sandwich) {
        ProfScope ps(decode ? "post_norm_dec" : "post_norm", st);
        FK_LAUNCH(launch_post_norm_residual(sc.a, x_mid, x_out, (int)T, H, w.post_ffn_norm, next_norm, c.rms_eps,
                                            sc.u, st, next_f16));
      }
      x_in = x_out;
      continue;
    }
    // gated FFN
    GemmOut og;
    og.epi = EPI_GLU_BF16;
    og.out_f16 = m->f16(FK_F16_FFN_ACT);
    og.out = sc.h;
    og.ldo = c.intermediate;
    og.act = c.act;
    { ProfScope ps(decode ? "gemm_gate_up_dec" : "gemm_gate_up", st); FK_TRY(gemm_run(sc.u, (int)T, H, m->g_gu[l], og, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes, fuse_ffn_norm ? &ffn_norm : nullptr)); }
    if (sandwich) {
      GemmOut od;
      od.epi = EPI_F32;
      od.out = sc.a;
      od.ldo = H;
      { ProfScope ps(decode ? "gemm_down_dec" : "gemm_down", st); FK_TRY(gemm_run(sc.h, (int)T, c.intermediate, m->g_down[l], od, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes)); }
      ProfScope ps(decode ? "post_norm_dec" : "post_norm", st);
      FK_LAUNCH(launch_post_norm_residual(sc.a, x_mid, x_out, (int)T, H, w.post_ffn_norm, next_norm, c.rms_eps, sc.u,
                                          st, next_f16));
    } else {
      GemmOut od;
      od.epi = EPI_ADD_F32;
      od.out = x_out;
      od.ldo = H;
      od.res = x_mid;
      od.ldr = H;
      const bool down_ssq = fuse_norm && l + 1 < L && skinny_fused_tail(m->g_down[l], (int)T, m->sm_count, EPI_ADD_F32);
      if (down_ssq) od.ssq = sc.ssq;
      { ProfScope ps(decode ? "gemm_down_dec" : "gemm_down", st); FK_TRY(gemm_run(sc.h, (int)T, c.intermediate, m->g_down[l], od, m->dev_err, st, gv, gvb, sc.gemv_counter_bytes)); }
      if (fuse_norm && l + 1 < L) {  // the next QKV projection normalises x_out itself
        qkv_norm.x = x_out;
        qkv_norm.ldx = H;
        qkv_norm.w = next_norm;
        qkv_norm.eps = c.rms_eps;
        qkv_norm.ssq = down_ssq ? sc.ssq : nullptr;
        qkv_norm.n_ssq = (H + 127) / 128;
        qkv_norm_set = true;
      } else {
        ProfScope ps(decode ? "rmsnorm_dec" : "rmsnorm", st);
        FK_LAUNCH(launch_rmsnorm(x_out, H, (int)T, H, next_norm, c.rms_eps, sc.u, H, st, next_f16));
      }
    }
    x_in = x_out;
  }
  if (slots) FK_LAUNCH(launch_rmsnorm_f32(x_in, (int)T, H, m->final_norm, c.rms_eps, slots + (size_t)(L + 1) * T * H, st));
  return FK_OK;
}

fk_status run_head(fk_model* m, const void* u, int R, float* logits, int32_t* argmax, const Scratch& sc,
                   cudaStream_t st, int32_t* argmax2 = nullptr, float* margin = nullptr) {
  GemmOut o;
  o.epi = EPI_F32;
  o.out = logits;
  o.ldo = m->cfg.vocab;
  o.softcap = m->cfg.final_softcap;
  { ProfScope ps("gemm_head", st); FK_TRY(gemm_run(u, R, m->cfg.hidden, m->g_head, o, m->dev_err, st, sc.gemv, sc.gemv_bytes,
                                                   sc.gemv_counter_bytes)); }
  ProfScope ps("argmax", st);
  if (argmax) FK_LAUNCH(launch_argmax(logits, R, m->cfg.vocab, m->cfg.vocab, argmax, st, argmax2, sc.argmax, margin));
  return FK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

fk_status check_ids_host(const int32_t* ids, long n, int vocab) {
  for (long i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= vocab) {
      char buf[128];
      snprintf(buf, sizeof buf, "token id %d at index %ld is outside [0, %d)", ids[i], i, vocab);
      return fail(FK_ERR_TOKEN_RANGE, buf);
    }
  return FK_OK;
}

}  // namespace

// ===========================================================================
// model
// ===========================================================================
extern "C" size_t fk_model_arena_bytes(const fk_config* cfg, int32_t max_positions) {
  if (validate_config(cfg) != FK_OK || max_positions < 1) {
    if (max_positions < 1) set_error("max_positions must be >= 1");
    return 0;
  }
  return kAlign + rope_table_bytes(cfg, max_positions) * (has_local(cfg) ? 2 : 1) + f16_copy_bytes(cfg);
}

extern "C" fk_status fk_model_create(const fk_config* cfg, const fk_weights* w, int32_t max_positions, void* d_arena,
                                     size_t arena_bytes, fk_model** out) {
  if (!out) return fail(FK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  FK_TRY(validate_config(cfg));
  if (!w || !w->embed || !w->final_norm || !w->layers) return fail(FK_ERR_INVALID_ARG, "weights incomplete");
  if (!cfg->tied && !w->lm_head) return fail(FK_ERR_INVALID_ARG, "untied model without lm_head");
  if (max_positions < 1) return fail(FK_ERR_INVALID_ARG, "max_positions must be >= 1");
  const size_t need = fk_model_arena_bytes(cfg, max_positions);
  if (!d_arena || arena_bytes < need) return fail(FK_ERR_WORKSPACE, "model arena too small");
  if (reinterpret_cast<uintptr_t>(d_arena) % kAlign) return fail(FK_ERR_INVALID_ARG, "arena must be 256-byte aligned");
  int sms = 0;
  FK_TRY(check_device(&sms));

  fk_model* m = new fk_model();
  m->cfg = *cfg;
  m->kinds.assign(cfg->n_layers, 0);
  if (cfg->layer_kinds) m->kinds.assign(cfg->layer_kinds, cfg->layer_kinds + cfg->n_layers);
  m->cfg.layer_kinds = m->kinds.data();
  m->has_local = has_local(cfg);
  m->layers.assign(w->layers, w->layers + cfg->n_layers);
  m->embed = w->embed;
  m->head = cfg->tied ? w->embed : w->lm_head;
  m->final_norm = w->final_norm;
  m->max_pos = max_positions;
  m->sm_count = sms;
  m->Nq = cfg->n_q_heads * cfg->head_dim;
  m->Nkv = cfg->n_kv_heads * cfg->head_dim;
  m->Nqkv = m->Nq + 2 * m->Nkv;
  m->embed_scale = cfg->embed_scale == FK_EMBED_SCALE_SQRT_HIDDEN_BF16 ? bf16_round(std::sqrt((float)cfg->hidden)) : 1.f;
  m->moe_kinds.assign(cfg->n_layers, 0);
  m->moe_index.assign(cfg->n_layers, -1);
  for (int l = 0; l < cfg->n_layers; ++l)
    if (is_moe_layer(cfg, l)) {
      m->moe_kinds[l] = 1;
      m->moe_index[l] = m->n_moe++;
    }
  m->cfg.moe_layers = m->moe_kinds.data();
  m->attn_scale = 1.0f / std::sqrt((float)cfg->head_dim);

  auto cleanup = [&](fk_status s) {
    delete m;
    return s;
  };
  // weights: pointers present and 16-byte aligned
  const void* top[3] = {m->embed, m->head, m->final_norm};
  for (const void* p : top)
    if (!aligned16(p)) return cleanup(fail(FK_ERR_INVALID_ARG, "weights must be 16-byte aligned"));
  for (int l = 0; l < cfg->n_layers; ++l) {
    const fk_layer_weights& lw = m->layers[l];
    const void* need_ptrs[] = {lw.attn_norm, lw.wq, lw.wk, lw.wv, lw.wo, lw.ffn_norm};
    for (const void* p : need_ptrs)
      if (!p || !aligned16(p)) return cleanup(fail(FK_ERR_INVALID_ARG, "layer weight missing or misaligned"));
    const bool moe = m->moe_index[l] >= 0;
    const void* ffn_ptrs[4] = {moe ? lw.router : lw.w_gate, moe ? lw.expert_gate : lw.w_up,
                               moe ? lw.expert_up : lw.w_down, moe ? lw.expert_down : lw.w_down};
    for (const void* p : ffn_ptrs)
      if (!p || !aligned16(p))
        return cleanup(fail(FK_ERR_INVALID_ARG, moe ? "MoE layer weight (router or experts) missing or misaligned"
                                                    : "layer weight missing or misaligned"));
    if (cfg->qk_norm && (!lw.q_norm || !lw.k_norm || !aligned16(lw.q_norm) || !aligned16(lw.k_norm)))
      return cleanup(fail(FK_ERR_INVALID_ARG, "qk_norm weights missing"));
    if (cfg->norm_layout == FK_NORM_SANDWICH &&
        (!lw.post_attn_norm || !lw.post_ffn_norm || !aligned16(lw.post_attn_norm) || !aligned16(lw.post_ffn_norm)))
      return cleanup(fail(FK_ERR_INVALID_ARG, "sandwich norm weights missing"));
  }
  // arena: error word + RoPE tables (host double precision -> fp32 cos/sin)
  uint8_t* arena = static_cast<uint8_t*>(d_arena);
  m->dev_err = reinterpret_cast<unsigned*>(arena);
  const size_t tb = rope_table_bytes(cfg, max_positions);
  m->rope[0] = reinterpret_cast<float2*>(arena + kAlign);
  m->rope[1] = m->has_local ? reinterpret_cast<float2*>(arena + kAlign + tb) : m->rope[0];
  const int half = cfg->head_dim / 2;
  std::vector<float2> table((size_t)max_positions * half);
  std::vector<double> f;
  for (int kind = 0; kind < (m->has_local ? 2 : 1); ++kind) {
    rope_freqs(cfg, kind, f);
    for (int p = 0; p < max_positions; ++p)
      for (int j = 0; j < half; ++j) {
        const double ang = (double)p * f[j];
        table[(size_t)p * half + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    cudaError_t e = cudaMemcpy(m->rope[kind], table.data(), table.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "upload rope table"));
  }
  // f16 copies of the weights of GEMMs whose input activations are f16
  const int H = cfg->hidden, I = cfg->intermediate;
  uint8_t* copy_at = arena + kAlign + tb * (m->has_local ? 2 : 1);
  cudaError_t ce = cudaSuccess;
  auto f16_copy = [&](const void* src, size_t elems) -> const void* {
    void* dst = copy_at;
    copy_at += align_up(elems * 2);
    if (ce == cudaSuccess) ce = launch_bf16_to_f16(src, dst, elems, nullptr);
    return dst;
  };
  std::vector<fk_layer_weights> gw(m->layers);  // the matrices the GEMMs read
  for (int l = 0; l < cfg->n_layers; ++l) {
    fk_layer_weights& lw = gw[l];
    if (m->f16(FK_F16_QKV_IN)) {
      lw.wq = f16_copy(lw.wq, (size_t)m->Nq * H);
      lw.wk = f16_copy(lw.wk, (size_t)m->Nkv * H);
      lw.wv = f16_copy(lw.wv, (size_t)m->Nkv * H);
    }
    if (m->f16(FK_F16_O_IN)) lw.wo = f16_copy(lw.wo, (size_t)H * m->Nq);
    if (m->moe_index[l] >= 0) {
      const size_t E = cfg->n_experts, Ie = cfg->expert_intermediate;
      if (m->f16(FK_F16_FFN_IN)) {
        lw.router = f16_copy(lw.router, E * H);
        lw.expert_gate = f16_copy(lw.expert_gate, E * Ie * H);
        lw.expert_up = f16_copy(lw.expert_up, E * Ie * H);
      }
      if (m->f16(FK_F16_FFN_ACT)) lw.expert_down = f16_copy(lw.expert_down, E * H * Ie);
      continue;
    }
    if (m->f16(FK_F16_FFN_IN)) {
      lw.w_gate = f16_copy(lw.w_gate, (size_t)I * H);
      lw.w_up = f16_copy(lw.w_up, (size_t)I * H);
    }
    if (m->f16(FK_F16_FFN_ACT)) lw.w_down = f16_copy(lw.w_down, (size_t)H * I);
  }
  const void* head_mat = m->f16(FK_F16_HEAD_IN) ? f16_copy(m->head, (size_t)cfg->vocab * H) : m->head;
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(nullptr);
  if (ce != cudaSuccess) return cleanup(cuda_fail(ce, "f16 weight copies"));
  // GEMM operands (TMA descriptors of the weights)
  m->g_qkv.resize(cfg->n_layers);
  m->g_o.resize(cfg->n_layers);
  m->g_gu.resize(cfg->n_layers);
  m->g_down.resize(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers; ++l) {
    const fk_layer_weights& lw = gw[l];
    const void* qkv[3] = {lw.wq, lw.wk, lw.wv};
    int rq[3] = {m->Nq, m->Nkv, m->Nkv};
    fk_status s = gemm_weights_init(&m->g_qkv[l], qkv, rq, 3, H, 0, m->f16(FK_F16_QKV_IN));
    const void* wo[1] = {lw.wo};
    int ro[1] = {H};
    if (s == FK_OK) s = gemm_weights_init(&m->g_o[l], wo, ro, 1, m->Nq, 0, m->f16(FK_F16_O_IN));
    if (s != FK_OK) return cleanup(s);
    if (m->moe_index[l] >= 0) {
      MoeWeights mw;
      mw.E = cfg->n_experts;
      mw.k = cfg->n_experts_per_tok;
      mw.Ie = cfg->expert_intermediate;
      mw.H = H;
      mw.norm_topk = cfg->norm_topk;
      mw.act = cfg->act;
      mw.act_f16 = m->f16(FK_F16_FFN_ACT);
      const void* rt[1] = {lw.router};
      int re[1] = {mw.E};
      s = gemm_weights_init(&mw.router, rt, re, 1, H, 0, m->f16(FK_F16_FFN_IN));
      const void* egu[2] = {lw.expert_gate, lw.expert_up};
      if (s == FK_OK) s = gemm_weights_init_grouped(&mw.gate_up, egu, 2, mw.E, mw.Ie, H, 1, m->f16(FK_F16_FFN_IN));
      const void* ed[1] = {lw.expert_down};
      if (s == FK_OK) s = gemm_weights_init_grouped(&mw.down, ed, 1, mw.E, H, mw.Ie, 0, m->f16(FK_F16_FFN_ACT));
      if (s != FK_OK) return cleanup(s);
      m->moe.push_back(mw);
      continue;
    }
    const void* gu[2] = {lw.w_gate, lw.w_up};
    int rg[2] = {I, I};
    s = gemm_weights_init(&m->g_gu[l], gu, rg, 2, H, 1, m->f16(FK_F16_FFN_IN));
    const void* wd[1] = {lw.w_down};
    int rd[1] = {H};
    if (s == FK_OK) s = gemm_weights_init(&m->g_down[l], wd, rd, 1, I, 0, m->f16(FK_F16_FFN_ACT));
    if (s != FK_OK) return cleanup(s);
  }
  {
    const void* hw[1] = {head_mat};
    int rv[1] = {cfg->vocab};
    fk_status s = gemm_weights_init(&m->g_head, hw, rv, 1, H, 0, m->f16(FK_F16_HEAD_IN));
    if (s != FK_OK) return cleanup(s);
  }
  cudaError_t e = cudaMemset(m->dev_err, 0, kCtlWords * sizeof(unsigned));
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "clear error word"));
  *out = m;
  return FK_OK;
}

extern "C" void fk_model_free(fk_model* m) { delete m; }

// ===========================================================================
// cacheless forward
// ===========================================================================
static size_t forward_layout(const fk_model* m, int B, int S, uint8_t* base, Scratch* sc, KV* kv, float** logits) {
  const fk_config& c = m->cfg;
  const long T = (long)B * S;
  size_t off = scratch_bytes(m, T, sc, base);
  const int cap = (S + 63) / 64 * 64;  // attention tiles read whole 64-position blocks
  const size_t kv_elems = (size_t)B * c.n_kv_heads * cap * c.head_dim;
  if (kv) {
    kv->k = base ? base + off : nullptr;
    kv->v = base ? base + off + align_up(kv_elems * 2) : nullptr;
    kv->cap = cap;
    kv->bytes = kv_elems * 2;
  }
  off += 2 * align_up(kv_elems * 2);
  if (logits) *logits = base ? reinterpret_cast<float*>(base + off) : nullptr;
  off += align_up((size_t)T * c.vocab * 4);
  return off;
}

extern "C" size_t fk_forward_workspace_bytes(const fk_model* m, int32_t batch, int32_t seq) {
  if (!m || batch < 1 || seq < 1) return 0;
  return forward_layout(m, batch, seq, nullptr, nullptr, nullptr, nullptr);
}

static bool graphs_disabled() {
  static const bool off = [] {
    const char* e = getenv("FK_NO_GRAPH");
    return e && *e && *e != '0';
  }();
  return off;
}

extern "C" fk_status fk_forward(fk_model* m, const int32_t* ids, int32_t ids_on_device, int32_t batch, int32_t seq,
                                void* d_ws, size_t ws_bytes, float* d_hidden, float* d_logits, int32_t* d_argmax,
                                float* d_margin, void* stream) {
  if (!m || !ids || batch < 1 || seq < 1) return fail(FK_ERR_INVALID_ARG, "fk_forward: bad argument");
  if (seq > m->max_pos) return fail(FK_ERR_CONTEXT_FULL, "seq exceeds the model's max_positions");
  const long T = (long)batch * seq;
  if (!ids_on_device) FK_TRY(check_ids_host(ids, T, m->cfg.vocab));
  const size_t need = fk_forward_workspace_bytes(m, batch, seq);
  if (!d_ws || ws_bytes < need) return fail(FK_ERR_WORKSPACE, "forward workspace too small");
  if (reinterpret_cast<uintptr_t>(d_ws) % kAlign) return fail(FK_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if ((d_hidden && !aligned16(d_hidden)) || (d_logits && !aligned16(d_logits)))
    return fail(FK_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  if (d_margin && !d_argmax) return fail(FK_ERR_INVALID_ARG, "d_margin needs d_argmax");
  FK_TRY(check_device(nullptr));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Scratch sc;
  KV kv;
  float* ws_logits = nullptr;
  forward_layout(m, batch, seq, static_cast<uint8_t*>(d_ws), &sc, &kv, &ws_logits);
  FK_CUDA_TRY(cudaMemcpyAsync(sc.ids, ids, T * sizeof(int32_t),
                              ids_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, st));
  auto enqueue = [&](cudaStream_t s2) -> fk_status {
    if (sc.gemv_counter_bytes) FK_CUDA_TRY(cudaMemsetAsync(sc.gemv, 0, sc.gemv_counter_bytes, s2));
    FK_CUDA_TRY(cudaMemsetAsync(static_cast<uint8_t*>(sc.argmax) + argmax_counter_offset(), 0,
                                argmax_scratch_bytes() - argmax_counter_offset(), s2));
    // attention reads V in 64-position blocks: positions past seq must hold finite values
    if (seq % 64) FK_CUDA_TRY(cudaMemsetAsync(kv.v, 0, kv.bytes, s2));
    FK_TRY(run_stack(m, sc, batch, seq, 0, kv, d_hidden, false, 1, s2));
    if (d_logits || d_argmax)
      FK_TRY(run_head(m, sc.u, (int)T, d_logits ? d_logits : ws_logits, d_argmax, sc, s2, nullptr, d_margin));
    return FK_OK;
  };
  // A forward of few tokens is mostly launch latency: replay it from a graph
  // once the same call has been seen before (the first call runs eagerly, so
  // every lazy set-up is done before a capture). Larger forwards, timed or
  // hooked runs and calls on a capturing stream launch one by one.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  FK_CUDA_TRY(cudaStreamIsCapturing(st, &cs));
  if (T > kSkinnyMaxTokens || cs != cudaStreamCaptureStatusNone || profiling_enabled() || graphs_disabled() ||
      m->moe_hook())
    return enqueue(st);
  fk_model::FwdKey key;
  key.B = batch;
  key.S = seq;
  key.ws = d_ws;
  key.out[0] = d_hidden;
  key.out[1] = d_logits;
  key.out[2] = d_argmax;
  key.out[3] = d_margin;
  std::lock_guard<std::mutex> lock(m->fwd_mu);
  fk_model::FwdEntry* hit = nullptr;
  fk_model::FwdEntry* lru = &m->fwd[0];
  for (fk_model::FwdEntry& e : m->fwd) {
    if (e.used && e.key == key) hit = &e;
    if (!e.used || (lru->used && e.last < lru->last)) lru = &e;
  }
  if (!hit) {  // first call with this key: launched one by one, remembered
    if (lru->exec) cudaGraphExecDestroy(lru->exec);
    *lru = fk_model::FwdEntry();
    lru->key = key;
    lru->used = true;
    lru->last = ++m->fwd_clock;
    return enqueue(st);
  }
  hit->last = ++m->fwd_clock;
  if (!hit->exec) {  // second call: capture
    if (!m->fwd_cap_stream) FK_CUDA_TRY(cudaStreamCreateWithFlags(&m->fwd_cap_stream, cudaStreamNonBlocking));
    FK_CUDA_TRY(cudaStreamBeginCapture(m->fwd_cap_stream, cudaStreamCaptureModeThreadLocal));
    const fk_status es = enqueue(m->fwd_cap_stream);
    cudaGraph_t g = nullptr;
    cudaError_t ce = cudaStreamEndCapture(m->fwd_cap_stream, &g);
    if (es != FK_OK) {
      if (g) cudaGraphDestroy(g);
      return es;
    }
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamEndCapture(forward)");
    ce = cudaGraphInstantiate(&hit->exec, g, 0);
    cudaGraphDestroy(g);
    if (ce != cudaSuccess) {
      hit->exec = nullptr;
      return cuda_fail(ce, "cudaGraphInstantiate(forward)");
    }
  }
  FK_CUDA_TRY(cudaGraphLaunch(hit->exec, st));
  return FK_OK;
}

// ===========================================================================
// sessions
// ===========================================================================
// Cache positions of layer l in a session: max_seq rounded up to 64 on global
// layers. A sliding-window layer reads at most the last W positions before a
// query, so it keeps a ring: position p in slot p mod cap. A prefill chunk of
// C tokens needs the W - 1 positions before it and its own C at once, so the
// ring holds W + max_chunk - 1 positions (rounded up to 64 for the 64-position
// attention tiles), never more than the global capacity.
static int layer_cache_positions(const fk_model* m, int l, int max_seq, int max_chunk) {
  const int global = (max_seq + 63) / 64 * 64;
  if (m->kinds[l] != 1) return global;
  const int ring = (m->cfg.sliding_window + max_chunk - 1 + 63) / 64 * 64;
  return std::min(global, ring);
}

static size_t session_layout(const fk_model* m, int B, int max_seq, int max_chunk, uint8_t* base, fk_session* s) {
  const fk_config& c = m->cfg;
  size_t off = 0;
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  std::vector<size_t> kv_off(c.n_layers);
  std::vector<int> kv_cap(c.n_layers);
  size_t kv_bytes = 0;
  for (int l = 0; l < c.n_layers; ++l) {
    kv_cap[l] = layer_cache_positions(m, l, max_seq, max_chunk);
    kv_off[l] = kv_bytes;
    kv_bytes += align_up((size_t)B * c.n_kv_heads * kv_cap[l] * c.head_dim * 2);
  }
  uint8_t* k = take(kv_bytes);
  uint8_t* v = take(kv_bytes);
  const long T = (long)B * max_chunk;
  Scratch sc;
  const size_t sb = scratch_bytes(m, T, &sc, base ? base + off : nullptr);
  off += sb;
  uint8_t* next = take((size_t)B * 4);
  uint8_t* logits = take((size_t)B * c.vocab * 4);
  uint8_t* ul = take((size_t)B * c.hidden * 2);
  const int splits = decode_attention_splits(B, c.n_kv_heads, c.head_dim, max_seq, m->sm_count);
  uint8_t* dl = take(sizeof(int));
  if (s) {
    s->d_len = reinterpret_cast<int*>(dl);
    s->kcache = k;
    s->vcache = v;
    s->kv_off = kv_off;
    s->kv_cap = kv_cap;
    s->kv_bytes = kv_bytes;
    s->sc = sc;
    s->next_ids = reinterpret_cast<int32_t*>(next);
    s->logits = reinterpret_cast<float*>(logits);
    s->u_last = ul;
    s->dec_splits = splits;
  }
  return off;
}

extern "C" size_t fk_session_bytes(const fk_model* m, int32_t batch, int32_t max_seq, int32_t max_chunk) {
  if (!m || batch < 1 || max_seq < 1 || max_chunk < 1 || max_seq > m->max_pos) {
    set_error("fk_session_bytes: bad argument (batch, max_seq <= max_positions, max_chunk >= 1)");
    return 0;
  }
  return session_layout(m, batch, max_seq, std::min(max_chunk, max_seq), nullptr, nullptr);
}

extern "C" fk_status fk_session_create(fk_model* m, int32_t batch, int32_t max_seq, int32_t max_chunk, void* d_mem,
                                       size_t bytes, fk_session** out) {
  if (!out) return fail(FK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  const size_t need = fk_session_bytes(m, batch, max_seq, max_chunk);
  if (need == 0) return FK_ERR_INVALID_ARG;
  if (!d_mem || bytes < need) return fail(FK_ERR_WORKSPACE, "session memory too small");
  if (reinterpret_cast<uintptr_t>(d_mem) % kAlign) return fail(FK_ERR_INVALID_ARG, "session memory must be 256-byte aligned");
  FK_TRY(check_device(nullptr));
  fk_session* s = new fk_session();
  s->m = m;
  s->B = batch;
  s->max_seq = max_seq;
  s->max_chunk = std::min(max_chunk, max_seq);
  session_layout(m, batch, max_seq, s->max_chunk, static_cast<uint8_t*>(d_mem), s);
  {
    // attention reads whole 64-position blocks of the cache: positions never
    // written must hold finite values
    cudaError_t e = cudaMemset(s->kcache, 0, s->kv_bytes);
    if (e == cudaSuccess) e = cudaMemset(s->vcache, 0, s->kv_bytes);
    if (e != cudaSuccess) {
      delete s;
      return cuda_fail(e, "clear KV cache");
    }
  }
  {
    cudaError_t e = cudaMemset(static_cast<uint8_t*>(s->sc.argmax) + argmax_counter_offset(), 0,
                               argmax_scratch_bytes() - argmax_counter_offset());
    if (e != cudaSuccess) {
      delete s;
      return cuda_fail(e, "clear argmax counters");
    }
  }
  if (s->sc.gemv_counter_bytes) {
    cudaError_t e = cudaMemset(s->sc.gemv, 0, s->sc.gemv_counter_bytes);
    if (e != cudaSuccess) {
      delete s;
      return cuda_fail(e, "clear split-K counters");
    }
  }
  if (m->n_moe) {  // the decode steps' expert GEMMs leave their counters zero after every launch
    cudaError_t e = cudaMemset(s->sc.moe.exp_counters, 0, s->sc.moe.exp_counters_bytes);
    if (e != cudaSuccess) {
      delete s;
      return cuda_fail(e, "clear expert split-K counters");
    }
  }
  *out = s;
  return FK_OK;
}

extern "C" void fk_session_free(fk_session* s) {
  if (!s) return;
  if (s->graph) cudaGraphExecDestroy(s->graph);
  if (s->cap_stream) cudaStreamDestroy(s->cap_stream);
  delete s;
}

extern "C" fk_status fk_session_reset(fk_session* s) {
  if (!s) return fail(FK_ERR_INVALID_ARG, "session is NULL");
  s->len = 0;
  s->d_len_valid = false;
  return FK_OK;
}

extern "C" int32_t fk_session_length(const fk_session* s) { return s ? s->len : -1; }

static fk_status session_head(fk_session* s, const void* u_rows, float* d_logits, int32_t* d_next, float* d_margin,
                              cudaStream_t st) {
  fk_model* m = s->m;
  float* logits = d_logits ? d_logits : s->logits;
  return run_head(m, u_rows, s->B, logits, s->next_ids, s->sc, st, d_next, d_margin);
}

extern "C" fk_status fk_session_prefill(fk_session* s, const int32_t* ids, int32_t ids_on_device, int32_t seq,
                                        float* d_last_logits, int32_t* d_next, float* d_margin, void* stream) {
  if (!s || !ids || seq < 1) return fail(FK_ERR_INVALID_ARG, "fk_session_prefill: bad argument");
  if (s->len + seq > s->max_seq) return fail(FK_ERR_CONTEXT_FULL, "prefill would exceed the session's max_seq");
  if (d_last_logits && !aligned16(d_last_logits)) return fail(FK_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  fk_model* m = s->m;
  if (m->moe_hook() && seq > s->max_chunk)
    return fail(FK_ERR_INVALID_ARG, "prefill in more than one chunk while the MoE routing hook is set");
  if (!ids_on_device) FK_TRY(check_ids_host(ids, (long)s->B * seq, m->cfg.vocab));
  FK_TRY(check_device(nullptr));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KV kv;
  kv.k = s->kcache;
  kv.v = s->vcache;
  kv.off = s->kv_off.data();
  kv.caps = s->kv_cap.data();
  int C = 0;
  for (int c0 = 0; c0 < seq; c0 += C) {
    C = std::min(s->max_chunk, seq - c0);
    FK_CUDA_TRY(cudaMemcpy2DAsync(s->sc.ids, C * sizeof(int32_t), ids + c0, seq * sizeof(int32_t),
                                  C * sizeof(int32_t), s->B,
                                  ids_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, st));
    FK_TRY(run_stack(m, s->sc, s->B, C, s->len, kv, nullptr, false, 1, st));
    s->len += C;
  }
  FK_LAUNCH(launch_gather_last_rows(s->sc.u, m->cfg.hidden, C, m->cfg.hidden, s->B, s->u_last, st));
  FK_LAUNCH(launch_set_int(s->d_len, s->len, st));
  s->d_len_valid = true;
  return session_head(s, s->u_last, d_last_logits, d_next, d_margin, st);
}

// Enqueue one decode step whose positions come from s->d_len (so the same
// launches serve every step, captured or not).
static fk_status enqueue_decode(fk_session* s, const int32_t* d_ids, float* d_logits, int32_t* d_next,
                                float* d_margin, cudaStream_t st) {
  fk_model* m = s->m;
  // every launch of the step may overlap its predecessor's tail (each kernel
  // waits for its predecessor before touching data the predecessor writes)
  PdlScope pdl(true);
  KV kv;
  kv.k = s->kcache;
  kv.v = s->vcache;
  kv.off = s->kv_off.data();
  kv.caps = s->kv_cap.data();
  FK_TRY(run_stack(m, s->sc, s->B, 1, s->len, kv, nullptr, true, s->dec_splits, st,
                   s->d_len, d_ids ? d_ids : s->next_ids));
  FK_TRY(session_head(s, s->sc.u, d_logits, d_next, d_margin, st));
  FK_LAUNCH(launch_inc_int(s->d_len, st));
  return FK_OK;
}


extern "C" fk_status fk_decode_step(fk_session* s, const int32_t* d_ids, float* d_logits, int32_t* d_next,
                                    float* d_margin, void* stream) {
  if (!s) return fail(FK_ERR_INVALID_ARG, "session is NULL");
  if (s->len + 1 > s->max_seq) return fail(FK_ERR_CONTEXT_FULL, "decode would exceed the session's max_seq");
  if (s->len == 0 && !d_ids) return fail(FK_ERR_INVALID_ARG, "no previous greedy ids: prefill first or pass d_ids");
  if (d_logits && !aligned16(d_logits)) return fail(FK_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  FK_TRY(check_device(nullptr));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!s->d_len_valid) {
    FK_LAUNCH(launch_set_int(s->d_len, s->len, st));
    s->d_len_valid = true;
  }
  // Steps that feed back the previous greedy ids are replayed from a CUDA
  // graph captured on the first such call (re-captured if the output
  // buffers change). Steps with caller ids, and steps while kernel timing is
  // on, are launched one by one.
  if (d_ids || profiling_enabled() || graphs_disabled() || s->m->moe_hook()) {
    FK_TRY(enqueue_decode(s, d_ids, d_logits, d_next, d_margin, st));
    s->len += 1;
    return FK_OK;
  }
  if (!s->graph || s->graph_logits != d_logits || s->graph_next != d_next || s->graph_margin != d_margin) {
    if (s->graph) {
      cudaGraphExecDestroy(s->graph);
      s->graph = nullptr;
    }
    if (!s->cap_stream) FK_CUDA_TRY(cudaStreamCreateWithFlags(&s->cap_stream, cudaStreamNonBlocking));
    FK_CUDA_TRY(cudaStreamBeginCapture(s->cap_stream, cudaStreamCaptureModeThreadLocal));
    fk_status es = enqueue_decode(s, nullptr, d_logits, d_next, d_margin, s->cap_stream);
    cudaGraph_t g = nullptr;
    cudaError_t ce = cudaStreamEndCapture(s->cap_stream, &g);
    if (es != FK_OK) {
      if (g) cudaGraphDestroy(g);
      return es;
    }
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamEndCapture(decode step)");
    ce = cudaGraphInstantiate(&s->graph, g, 0);
    cudaGraphDestroy(g);
    if (ce != cudaSuccess) {
      s->graph = nullptr;
      return cuda_fail(ce, "cudaGraphInstantiate(decode step)");
    }
    s->graph_logits = d_logits;
    s->graph_next = d_next;
    s->graph_margin = d_margin;
  }
  FK_CUDA_TRY(cudaGraphLaunch(s->graph, st));
  s->len += 1;
  return FK_OK;
}

// ===========================================================================
// op hooks: one step of the path alone, on the same kernels as the forward
// ===========================================================================
extern "C" fk_status fk_op_rmsnorm(const float* d_x, int32_t rows, int32_t hidden, const void* d_w, float eps,
                                   void* d_out, void* stream) {
  if (!d_x || !d_w || !d_out || rows < 1 || hidden < 8 || hidden % 8)
    return fail(FK_ERR_INVALID_ARG, "fk_op_rmsnorm: need rows >= 1, hidden a positive multiple of 8, non-null buffers");
  if (!(eps > 0.f) || !std::isfinite(eps)) return fail(FK_ERR_INVALID_ARG, "fk_op_rmsnorm: eps must be > 0");
  if (!aligned16(d_x) || !aligned16(d_w) || !aligned16(d_out))
    return fail(FK_ERR_INVALID_ARG, "fk_op_rmsnorm: buffers must be 16-byte aligned");
  FK_TRY(check_device(nullptr));
  FK_LAUNCH(launch_rmsnorm(d_x, hidden, rows, hidden, d_w, eps, d_out, hidden, static_cast<cudaStream_t>(stream), 0));
  return FK_OK;
}

extern "C" fk_status fk_op_rope(fk_model* m, int32_t layer, void* d_qkv, int32_t batch, int32_t seq, int32_t pos0,
                                void* d_kcache, void* d_vcache, int32_t cap, void* stream) {
  if (!m || !d_qkv || !d_kcache || !d_vcache || batch < 1 || seq < 1 || pos0 < 0)
    return fail(FK_ERR_INVALID_ARG, "fk_op_rope: bad argument");
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(FK_ERR_INVALID_ARG, "fk_op_rope: layer out of range");
  if (pos0 + seq > cap || cap % 64) return fail(FK_ERR_INVALID_ARG, "fk_op_rope: need pos0 + seq <= cap, cap % 64 == 0");
  if (pos0 + seq > m->max_pos) return fail(FK_ERR_CONTEXT_FULL, "fk_op_rope: positions beyond the model's max_positions");
  if (!aligned16(d_qkv) || !aligned16(d_kcache) || !aligned16(d_vcache))
    return fail(FK_ERR_INVALID_ARG, "fk_op_rope: buffers must be 16-byte aligned");
  FK_TRY(check_device(nullptr));
  const fk_config& c = m->cfg;
  const fk_layer_weights& w = m->layers[layer];
  const int kind = m->kinds[layer];
  FK_LAUNCH(launch_rope_qkv(d_qkv, m->Nqkv, batch * seq, seq, pos0, c.n_q_heads, c.n_kv_heads, c.head_dim,
                            m->rope[kind], c.qk_norm, w.q_norm, w.k_norm, c.rms_eps, d_kcache, d_vcache, cap,
                            static_cast<cudaStream_t>(stream), m->f16(FK_F16_ATTN)));
  return FK_OK;
}

extern "C" fk_status fk_op_head_argmax(fk_model* m, const void* d_u, int32_t rows, float* d_logits,
                                       int32_t* d_argmax, float* d_margin, void* stream) {
  if (!m || !d_u || !d_logits || rows < 1) return fail(FK_ERR_INVALID_ARG, "fk_op_head_argmax: bad argument");
  if (d_margin && !d_argmax) return fail(FK_ERR_INVALID_ARG, "fk_op_head_argmax: d_margin needs d_argmax");
  if (!aligned16(d_u) || !aligned16(d_logits))
    return fail(FK_ERR_INVALID_ARG, "fk_op_head_argmax: buffers must be 16-byte aligned");
  FK_TRY(check_device(nullptr));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmOut o;
  o.epi = EPI_F32;
  o.out = d_logits;
  o.ldo = m->cfg.vocab;
  o.softcap = m->cfg.final_softcap;
  FK_TRY(gemm_run(d_u, rows, m->cfg.hidden, m->g_head, o, m->dev_err, st));
  if (d_argmax) FK_LAUNCH(launch_argmax(d_logits, rows, m->cfg.vocab, m->cfg.vocab, d_argmax, st, nullptr, nullptr, d_margin));
  return FK_OK;
}

extern "C" fk_status fk_model_set_moe_routing(fk_model* m, const int32_t* d_forced, int32_t* d_trace_ids,
                                              float* d_trace_margin, int32_t max_tokens) {
  if (!m) return fail(FK_ERR_INVALID_ARG, "fk_model_set_moe_routing: model is NULL");
  const bool any = d_forced || d_trace_ids || d_trace_margin;
  if (any && (m->n_moe == 0 || max_tokens < 1))
    return fail(FK_ERR_INVALID_ARG, "fk_model_set_moe_routing: needs a model with MoE layers and max_tokens >= 1");
  m->moe_forced = d_forced;
  m->moe_trace_ids = d_trace_ids;
  m->moe_trace_margin = d_trace_margin;
  m->moe_hook_tokens = any ? max_tokens : 0;
  return FK_OK;
}

static size_t moe_op_bytes(const fk_model* m, int T, MoeScratch* s, uint8_t* base) {
  return moe_scratch(m->moe[0], T, s, base);
}

extern "C" size_t fk_op_moe_ffn_workspace_bytes(const fk_model* m, int32_t T) {
  if (!m || m->n_moe == 0 || T < 1) {
    set_error("fk_op_moe_ffn_workspace_bytes: needs a model with MoE layers and T >= 1");
    return 0;
  }
  return moe_op_bytes(m, T, nullptr, nullptr);
}

extern "C" fk_status fk_op_moe_ffn(fk_model* m, int32_t layer, const void* d_u, int32_t T, const int32_t* d_forced,
                                   float* d_out, int32_t* d_ids, float* d_margin, void* d_ws, size_t ws_bytes,
                                   void* stream) {
  if (!m || !d_u || !d_out || T < 1) return fail(FK_ERR_INVALID_ARG, "fk_op_moe_ffn: bad argument");
  if (layer < 0 || layer >= m->cfg.n_layers || m->moe_index[layer] < 0)
    return fail(FK_ERR_INVALID_ARG, "fk_op_moe_ffn: not a MoE layer");
  if (!aligned16(d_u) || !aligned16(d_out)) return fail(FK_ERR_INVALID_ARG, "fk_op_moe_ffn: buffers must be 16-byte aligned");
  if (!d_ws || ws_bytes < fk_op_moe_ffn_workspace_bytes(m, T))
    return fail(FK_ERR_WORKSPACE, "fk_op_moe_ffn: workspace too small");
  if (reinterpret_cast<uintptr_t>(d_ws) % kAlign) return fail(FK_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  FK_TRY(check_device(nullptr));
  MoeScratch sc;
  moe_op_bytes(m, T, &sc, static_cast<uint8_t*>(d_ws));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // up to kMoeFewMaxTokens tokens: the split-K expert GEMMs (their counters start at zero)
  const bool few = T <= kMoeFewMaxTokens;
  if (few) FK_CUDA_TRY(cudaMemsetAsync(sc.exp_counters, 0, sc.exp_counters_bytes, st));
  return moe_ffn_run(m->moe[m->moe_index[layer]], d_u, T, sc, d_forced, d_ids, d_margin, d_out, nullptr, m->dev_err,
                     st, few);
}

// ===========================================================================
// status
// ===========================================================================
extern "C" fk_status fk_sync_status(fk_model* m, void* stream, int32_t timeout_ms, uint32_t* flags) {
  if (flags) *flags = 0;
  unsigned* word = nullptr;
  if (m) {
    word = m->dev_err;
  } else {
    FK_TRY(check_device(nullptr));
    FK_TRY(op_control_block(&word));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t ev;
  FK_CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
  cudaError_t e = cudaEventRecord(ev, st);
  if (e != cudaSuccess) {
    cudaEventDestroy(ev);
    return cuda_fail(e, "cudaEventRecord");
  }
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    e = cudaEventQuery(ev);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) {
      cudaEventDestroy(ev);
      return cuda_fail(e, "stream reported an error");
    }
    if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms)) {
      cudaEventDestroy(ev);
      return fail(FK_ERR_TIMEOUT, "stream did not drain before the deadline");
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  cudaEventDestroy(ev);
  unsigned h = 0;
  FK_CUDA_TRY(cudaMemcpy(&h, word, sizeof h, cudaMemcpyDeviceToHost));
  if (h) {
    FK_CUDA_TRY(cudaMemset(word, 0, sizeof h));
    if (flags) *flags = h;
    char buf[96];
    snprintf(buf, sizeof buf, "device error word 0x%x", h);
    return fail(FK_ERR_DEVICE_FLAG, buf);
  }
  return FK_OK;
}
