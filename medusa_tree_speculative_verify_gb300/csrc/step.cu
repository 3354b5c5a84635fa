// The whole verify step over a Llama-style backbone, and the prefill that starts a decode.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate() and its steps 二.4 - 二.7: candidates
// from the previous step's root and head top-k, one backbone pass over the flattened tree with the tree mask
// (positions = prefix + depth), posterior evaluation, KV compaction, and the next root / head top-k taken at
// node retrieve[best][acc]. The reference runs the Medusa heads on every tree node and keeps that node's row;
// here they run on that node only (the same consumed value). Every quantity that changes from step to step
// (prefix length, root, head top-k, the accepted path) lives in device memory, so a step needs no host
// synchronisation and can be captured once in a CUDA graph and replayed ("OpenPangu7B-with-Medusa" README, 4:
// static tree tensors and few host-device round trips, here on CUDA graphs).
//
// Kernel sequence of one step (L layers): build_candidates, embed, L x {QKV+RoPE+KV append, tree attention,
// O + residual, gate/up + SiLU-gate, down + residual}, LM head, posterior, KV compaction, heads W1, heads W2.
#include <stdlib.h>

#include <algorithm>
#include <string>
#include <vector>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace {

constexpr int kTok = MV_MAX_NODES;  // token rows of every activation buffer (the largest tree)
constexpr int kChunk = 64;         // prefill chunk: one token group, run as a causal chain

constexpr int kSeqRows = 64;       // rows per sequence when several sequences share a pass

// x[j][:] = float(E[tok[j]][:]), xb = E[tok[j]] (bf16), ssq[s][j] = sum of x^2 over the 128-column slice s.
// With seq_rows > 0, rows j with j % seq_rows >= seq_n are padding between sequences: zeroed, so that what the
// projections compute for them stays finite (no output of a real row depends on them).
__global__ void __launch_bounds__(256) embed_kernel(const int32_t* tokens, const uint16_t* __restrict__ E, int vocab,
                                                    int d, float* x, uint16_t* xb, float* ssq, unsigned int* err,
                                                    int seq_rows, int seq_n) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  if (seq_rows && j % seq_rows >= seq_n) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      x[(size_t)j * d + c] = 0.0f;
      xb[(size_t)j * d + c] = 0;
    }
    for (int s = threadIdx.x; s < (d + 127) / 128; s += blockDim.x) ssq[s * kTok + j] = 0.0f;
    return;
  }
  const int tok = tokens[j];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) mv_set_error(err, 11, MV_DEVERR_INDEX);
    return;
  }
  const int slices = (d + 127) / 128;
  for (int s = warp; s < slices; s += 8) {
    float acc = 0.0f;
    for (int c = s * 128 + lane; c < min(d, s * 128 + 128); c += 32) {
      const uint16_t b = E[(size_t)tok * d + c];
      const float v = __uint_as_float((uint32_t)b << 16);
      x[(size_t)j * d + c] = v;
      xb[(size_t)j * d + c] = b;
      acc += v * v;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) ssq[s * kTok + j] = acc;
  }
}

// After a prefill chunk of c tokens: the last chunk records the root (argmax of its last logits row) and the
// node the heads read (c - 1) in the result; earlier chunks just advance the length.
__global__ void __launch_bounds__(1024) prefill_finish_kernel(const float* logits, int V, int ld, int c,
                                                             int last, int32_t* cur_len,
                                                             mv_posterior_result* res) {
  pdl_trigger();
  pdl_wait();
  if (!last) {
    if (threadIdx.x == 0) *cur_len += c;
    return;
  }
  const float* row = logits + (size_t)(c - 1) * ld;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float v = row[i];
    if (vi_better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (vi_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  __shared__ float sv[32];
  __shared__ int si[32];
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (vi_better(sv[w], si[w], bv, bi)) {
        bv = sv[w];
        bi = si[w];
      }
    res->best = 0;
    res->acc = c - 1;
    res->next_node = c - 1;
    res->next_root = bi;
    res->n_tokens = c;  // the heads kernel commits cur_len += c
  }
}

__global__ void set_int_kernel(int32_t* p, int v) {
  pdl_trigger();
  pdl_wait();
  *p = v;
}

// The Medusa heads' inputs of a batch: for sequence b (one CTA each), h = RMSNorm(x[64 b + result[b].next_node])
// as a bf16 (hi, lo) pair in rows b and 16 + b of h_pair; then cur_len[b] += result[b].n_tokens.
__global__ void __launch_bounds__(256) heads_gather_kernel(const float* x, int d, float eps,
                                                           const mv_posterior_result* res, int32_t* cur_len,
                                                           uint16_t* h_pair, unsigned int* err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  __shared__ float red[8];
  const int node = res[b].next_node;
  if (node < 0 || node >= kSeqRows) {
    if (tid == 0) mv_set_error_detail(err, 15, MV_DEVERR_INDEX, (uint32_t)node);
    return;
  }
  const float* xr = x + (size_t)(b * kSeqRows + node) * d;
  float ss = 0.0f;
  for (int c = tid; c < d; c += 256) ss += xr[c] * xr[c];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = rsqrtf(tot / d + eps);
  for (int c = tid; c < d; c += 256) {
    const float v = xr[c] * inv;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    h_pair[(size_t)b * d + c] = __bfloat16_as_ushort(hi);
    h_pair[(size_t)(16 + b) * d + c] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
  }
  if (tid == 0) cur_len[b] += res[b].n_tokens;
}

// p[b] = v + b * 2^32 for the n sequences of a session (each draws from its own range of counters)
__global__ void set_counters_kernel(uint64_t* p, uint64_t v, int n) {
  pdl_trigger();
  pdl_wait();
  for (int b = 0; b < n; ++b) p[b] = v + ((uint64_t)b << 32);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

struct mv_model {
  mv_model_dims dims;
  int dtype = MV_DTYPE_BF16;  // MV_DTYPE_F32: the fp32 path (f32.cu) on the f_* weights
  int packed;  // projection weights in the packed layout
  const uint16_t* embed;
  std::vector<const uint16_t*> wqkv, wo, w_gate, w_up, w_down;
  const uint16_t* lm_head;
  const uint16_t* w1;
  const uint16_t* w2;
  std::vector<CUtensorMap> m_qkv, m_o, m_gate, m_up, m_down;
  CUtensorMap m_lm;
  // packed models: boxes of two consecutive k-blocks (one load per pipeline stage), and gate + up of a layer as
  // one 4-D map (depth 1 and 2) when the two sit back to back (gu_combined)
  std::vector<CUtensorMap> m_qkv2, m_o2, m_down2, m_gu1, m_gu2;
  CUtensorMap m_lm2;
  int gu_combined = 0;
  // fp32 weights (row-major [out][in])
  const float* f_embed = nullptr;
  std::vector<const float*> f_wqkv, f_wo, f_gate, f_up, f_down;
  const float* f_lm = nullptr;
  const float* f_w1 = nullptr;
  const float* f_w2 = nullptr;
  void* owned = nullptr;  // device memory of a model whose weights the library drew (mv_model_create_random)
};

struct mv_session {
  mv_model* model;
  const mv_tree* tree;
  mv_tree* chain;  // 64-node chain tree for prefill chunks (causal mask)
  uint16_t* kv;
  int s_max, topk;
  int batch;            // sequences verified together (1 .. MV_MAX_BATCH)
  size_t kv_seq_elems;  // elements of one sequence's KV cache
  // device buffers carved from the workspace; the per-sequence state is an array of `batch` entries
  int32_t* cur_len;
  mv_posterior_result* result;
  int32_t* head_topk;   // [batch][n_medusa][topk]
  int32_t* tree_tokens;
  int32_t* cart;
  float* x;
  uint16_t* xb;
  float* ssq;
  uint16_t* q;
  uint16_t* attn;
  uint16_t* act;
  float* logits;
  int ld_logits;
  void* ws_attn;
  void* ws_post;
  void* ws_heads;
  unsigned int* chain_flags;  // phase counters of the projection chains (zero between launches)
  float* xn = nullptr;        // fp32 path: the normalised projection operand [kTok][d]
  float* qkv_f = nullptr;     // fp32 path: [kTok][3 H D] projections, then q [kTok][H][D] (rotated)
  float* q_f = nullptr;
  float* attn_f = nullptr;    // fp32 path: attention output [kTok][H D]
  float* act_f = nullptr;     // fp32 path: SiLU-gate product [kTok][ffn]
  float2* row_max;            // [vocab/128][64]: per LM-head tile and token, max and first argmax
  uint16_t* h_pair;           // [32][d] bf16: the heads' inputs of a batch as (hi, lo) rows
  uint64_t* root_counter;     // per sequence: generator counter of the next sampled root
  mv_root_params root{};      // root rule (MV_ROOT_ARGMAX: the posterior's argmax stands)
  bool fuse_attention = true;  // run each layer's attention inside its projection chain when the shape allows
  int root_epoch = 0;         // bumped by every mv_session_set_root_sampling
  CUtensorMap m_xb, m_attn, m_act, m_kv;
  // the same as one box per pipeline stage, for passes of 1 .. kStageMaps token groups (gemm_act_map_stage)
  static constexpr int kStageMaps = kTok / 64;
  CUtensorMap m_xb2[kStageMaps], m_attn2[kStageMaps], m_act2[kStageMaps];
  bool act_box = false;
  // CUDA graph of n consecutive steps (medusa_verify_steps_graph), captured on first use
  cudaGraphExec_t graph_exec = nullptr;
  cudaStream_t capture_stream = nullptr;
  mv_accept_params graph_prm{};
  int graph_steps = 0;
  int graph_root_epoch = 0;
  bool graph_profiled = false;
  // CUDA graph of one host-buffer step (medusa_verify_step_host with pinned buffers): the seed copies, the step
  // and the result copies, replayed while the parameters and host buffers stay the same
  cudaGraphExec_t host_graph = nullptr;
  mv_accept_params host_prm{};
  int host_root_epoch = 0;
  const void* host_ptrs[3] = {nullptr, nullptr, nullptr};
  // optional per-launch timing (mv_session_profile): event pairs recorded around every launch
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  std::vector<std::pair<int, int>> ev_used;  // (kind, index of the first event of the pair)
  std::vector<std::pair<int, int>> profiled_graph_events;  // the pairs a profiled graph records
  size_t profiled_graph_ev_next = 0;
  size_t ev_next = 0;
};

namespace {

// Records an event on `st` for a profiled launch of `kind`; returns the pool index or -1.
int prof_mark(mv_session* s, cudaStream_t st) {
  if (!s->profiling) return -1;
  if (s->ev_next >= s->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    s->ev_pool.push_back(e);
  }
  const int i = (int)s->ev_next++;
  // external record: inside a stream capture this becomes a real event-record node whose timestamps can be read
  cudaEventRecordWithFlags(s->ev_pool[i], st, cudaEventRecordExternal);
  return i;
}

struct ProfScope {
  mv_session* s;
  cudaStream_t st;
  int kind, first;
  ProfScope(mv_session* s_, cudaStream_t st_, int kind_) : s(s_), st(st_), kind(kind_) { first = prof_mark(s, st); }
  ~ProfScope() {
    const int second = prof_mark(s, st);
    if (first >= 0 && second == first + 1) s->ev_used.push_back({kind, first});
  }
};

}  // namespace

namespace {

struct SessionLayout {
  size_t state, tree_tokens, cart, x, xb, ssq, q, attn, act, logits, attn_ws, post, heads, chain, row_max, h_pair,
      total;
};

SessionLayout session_layout(const mv_model_dims& d, int s_max, int topk, int dtype = MV_DTYPE_BF16) {
  SessionLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const int HD = d.n_heads * d.head_dim;
  const int ldl = (d.vocab + 3) & ~3;
  // cur_len [MV_MAX_BATCH] at 0, root counters at 16, results at 64, head top-k at 512
  static_assert(64 + MV_MAX_BATCH * sizeof(mv_posterior_result) <= 512, "session state layout");
  L.state = take(512 + (size_t)MV_MAX_BATCH * d.n_medusa * topk * 4);
  L.tree_tokens = take(kTok * 4);
  L.cart = take((size_t)kTok * (MV_MAX_DEPTH + 1) * 4);
  if (dtype == MV_DTYPE_F32) {  // fp32 path: every activation in fp32 (xb holds xn, q holds q and qkv)
    L.x = take((size_t)kTok * d.d * 4);
    L.xb = take((size_t)kTok * d.d * 4);
    L.q = take((size_t)kTok * (4 * HD) * 4);
    L.attn = take((size_t)kTok * HD * 4);
    L.act = take((size_t)kTok * d.ffn * 4);
    L.logits = take((size_t)kTok * ldl * 4);
    L.post = take(posterior_ws_bytes(kTok));
    L.heads = take(f32_heads_ws_bytes(d.d, d.n_medusa, d.vocab));
    L.total = o;
    return L;
  }
  L.x = take((size_t)kTok * d.d * 4);
  L.xb = take((size_t)kTok * d.d * 2);
  L.ssq = take((size_t)((d.d + 127) / 128) * kTok * 4);
  L.q = take((size_t)kTok * HD * 2);
  L.attn = take((size_t)kTok * HD * 2);
  L.act = take((size_t)kTok * d.ffn * 2);
  L.logits = take((size_t)kTok * ldl * 4);
  L.attn_ws = take(tree_attn_ws_bytes(d.n_heads, d.head_dim, s_max, kTok));
  L.post = take(posterior_ws_bytes(kTok));
  L.heads = take(heads_ws_bytes(MV_MAX_BATCH, d.d, d.n_medusa, d.vocab, topk));  // B = 1 GEMV or the batched path
  L.chain = take(kGemmChainFlagWords * sizeof(unsigned int));  // zero at creation; each chain launch leaves it so
  L.row_max = take((size_t)((d.vocab + 127) / 128) * kTok * sizeof(float2));  // LM-head tile max / argmax
  L.h_pair = take((size_t)32 * d.d * 2);
  L.total = o;
  return L;
}

bool dims_ok(const mv_model_dims& d) {
  const int D = d.head_dim;
  if (d.d < 8 || (d.d & 7) || d.n_layers < 1 || d.n_heads < 1 || d.ffn < 8 || (d.ffn & 7) || d.vocab < 16 ||
      d.n_medusa < 1 || d.n_medusa > 8)
    return false;
  if (D != 16 && D != 32 && D != 64 && D != 128) return false;
  if (((d.n_heads * D) & 7) || d.d > 8192) return false;
  return d.norm_eps > 0.0f && d.rope_theta > 1.0f;
}

GemmParams base_params(const mv_session* s, int n_tok) {
  GemmParams p{};
  p.n_tok = n_tok;
  p.tok_ld = kTok;  // the stride of the session's sum-of-squares and tile-statistics arrays
  p.packed_a = s->model->packed ? 2 : 0;
  const int groups = (n_tok + 63) / 64;
  p.act_box = s->act_box && groups >= 1 && groups <= mv_session::kStageMaps ? groups : 0;
  p.eps = s->model->dims.norm_eps;
  p.err = mv_error_word();
  return p;
}

// The fp32 model's backbone pass over n tokens of the session's one sequence (see forward below): plain FFMA
// kernels, every intermediate in fp32.
mv_status forward_f32(mv_session* s, const mv_tree* t, const int32_t* d_tokens, int n, bool lm, cudaStream_t st) {
  const mv_model* m = s->model;
  const mv_model_dims& d = m->dims;
  const int H = d.n_heads, D = d.head_dim, HD = H * D;
  const float scale = 1.0f / sqrtf((float)D);
  float* kvf = reinterpret_cast<float*>(s->kv);
  ProfScope ps(s, st, MV_PROF_OTHER);
  mv_status rc = launch_f32_embed(d_tokens, n, m->f_embed, d.vocab, d.d, s->x, st);
  for (int l = 0; l < d.n_layers && rc == MV_OK; ++l) {
    float* kvl = kvf + (size_t)l * 2 * H * s->s_max * D;
    if ((rc = launch_f32_rmsnorm(s->x, n, d.d, d.norm_eps, s->xn, st)) != MV_OK) break;
    if ((rc = launch_f32_linear(s->xn, d.d, m->f_wqkv[l], nullptr, 3 * HD, d.d, n, s->qkv_f, 3 * HD, 0, st)) != MV_OK)
      break;
    if ((rc = launch_f32_rope_append(s->qkv_f, n, H, D, s->s_max, s->cur_len, t->d_position_ids, d.rope_theta,
                                     s->q_f, kvl, st)) != MV_OK)
      break;
    if ((rc = launch_f32_tree_attention(s->q_f, kvl, H, D, s->s_max, n, s->cur_len, t->d_ancestors, scale,
                                        s->attn_f, st)) != MV_OK)
      break;
    if ((rc = launch_f32_linear(s->attn_f, HD, m->f_wo[l], nullptr, d.d, HD, n, s->x, d.d, 1, st)) != MV_OK) break;
    if ((rc = launch_f32_rmsnorm(s->x, n, d.d, d.norm_eps, s->xn, st)) != MV_OK) break;
    if ((rc = launch_f32_linear(s->xn, d.d, m->f_gate[l], m->f_up[l], d.ffn, d.d, n, s->act_f, d.ffn, 2, st)) !=
        MV_OK)
      break;
    rc = launch_f32_linear(s->act_f, d.ffn, m->f_down[l], nullptr, d.d, d.ffn, n, s->x, d.d, 1, st);
  }
  if (rc == MV_OK && lm) {
    rc = launch_f32_rmsnorm(s->x, n, d.d, d.norm_eps, s->xn, st);
    if (rc == MV_OK)
      rc = launch_f32_linear(s->xn, d.d, m->f_lm, nullptr, d.vocab, d.d, n, s->logits, s->ld_logits, 0, st);
  }
  return rc;
}

// One backbone pass over the n tokens (tree nodes or a prefill chunk) of nseq sequences b0 .. b0 + nseq - 1,
// whose ids are at d_tokens (sequence b's at row 64 (b - b0) when nseq > 1). `t` gives the attention mask
// (ancestor words) and positions (depth); each prefix length is read from s->cur_len[b].
mv_status forward(mv_session* s, const mv_tree* t, const int32_t* d_tokens, int n, bool lm, cudaStream_t st,
                  int nseq = 1, int b0 = 0) {
  if (s->model->dtype == MV_DTYPE_F32) return forward_f32(s, t, d_tokens, n, lm, st);
  const mv_model* m = s->model;
  const mv_model_dims& d = m->dims;
  const int HD = d.n_heads * d.head_dim;
  const int ssq_parts = (d.d + 127) / 128;
  const int seq_rows = nseq > 1 ? kSeqRows : 0;
  const int rows = nseq > 1 ? kSeqRows * (nseq - 1) + n : n;  // token rows of the pass, padding included
  mv_status rc;
  {
    ProfScope ps(s, st, MV_PROF_OTHER);
    rc = mv_launch(embed_kernel, dim3(rows), dim3(256), 0, st, d_tokens, m->embed, d.vocab, d.d, s->x, s->xb,
                   s->ssq, mv_error_word(), seq_rows, n) == cudaSuccess
             ? mv_last_launch("embed")
             : MV_ERR_CUDA;
  }
  // the projections, as chain phases: each phase's activations are the previous phase's output
  // packed weights: a0 loads a whole pipeline stage (two k-blocks) when the launch streams two per stage
  const bool two = m->packed && gemm_stage_kblocks(rows) == 2;
  const int gi = std::min(std::max((rows + 63) / 64, 1), (int)mv_session::kStageMaps) - 1;  // stage maps of the pass
  auto qkv_phase = [&](int l) {  // QKV + RoPE + KV append
    GemmPhase g;
    g.epi = EPI_QKV;
    g.a0 = two ? m->m_qkv2[l] : m->m_qkv[l];
    g.a1 = m->m_qkv[l];
    g.b = s->m_xb;
    g.b2 = s->m_xb2[gi];
    GemmParams& p = g.p = base_params(s, rows);
    p.M = 3 * HD;
    p.K = d.d;
    p.ssq = s->ssq;
    p.ssq_parts = ssq_parts;
    p.norm_d = d.d;
    p.q_out = s->q;
    p.kv = s->kv + (size_t)b0 * s->kv_seq_elems;
    p.H = d.n_heads;
    p.D = d.head_dim;
    p.S_max = s->s_max;
    p.layer = l;
    p.cur_len = s->cur_len + b0;
    p.pos_ids = t->d_position_ids;
    p.seq_rows = seq_rows;
    p.seq_n = n;
    p.kv_seq_stride = s->kv_seq_elems;
    p.log2_theta = log2f(d.rope_theta);
    return g;
  };
  auto residual_phase = [&](const CUtensorMap& w, const CUtensorMap* w2, const CUtensorMap& act,
                            const CUtensorMap& act2, int K) {
    GemmPhase g;  // O or down + residual
    g.epi = EPI_RESIDUAL;
    g.a0 = two ? *w2 : w;
    g.a1 = w;
    g.b = act;
    g.b2 = act2;
    GemmParams& p = g.p = base_params(s, rows);
    p.M = d.d;
    p.K = K;
    p.x = s->x;
    p.xb = s->xb;
    p.ssq_out = s->ssq;
    return g;
  };
  auto gate_up_phase = [&](int l) {  // gate/up + SiLU-gate
    GemmPhase g;
    g.epi = EPI_SWIGLU;
    g.a0 = m->m_gate[l];
    g.a1 = m->m_up[l];
    g.b = s->m_xb;
    g.b2 = s->m_xb2[gi];
    GemmParams& p = g.p = base_params(s, rows);
    if (m->gu_combined) {  // gate and up rows of a k-block in one box
      g.a0 = two ? m->m_gu2[l] : m->m_gu1[l];
      g.a1 = m->m_gu1[l];
      p.packed_a = 3;
    } else if (m->packed) {
      p.packed_a = 1;
    }
    p.paired = 1;
    p.F = d.ffn;
    p.M = d.ffn;
    p.K = d.d;
    p.ssq = s->ssq;
    p.ssq_parts = ssq_parts;
    p.norm_d = d.d;
    p.act = s->act;
    return g;
  };
  auto lm_phase = [&]() {  // final RMSNorm (as a column scale) + LM head -> fp32 logits
    GemmPhase g;
    g.epi = EPI_STORE;
    g.a0 = two ? m->m_lm2 : m->m_lm;
    g.a1 = m->m_lm;
    g.b = s->m_xb;
    g.b2 = s->m_xb2[gi];
    GemmParams& p = g.p = base_params(s, rows);
    p.M = d.vocab;
    p.K = d.d;
    p.ssq = s->ssq;
    p.ssq_parts = ssq_parts;
    p.norm_d = d.d;
    p.out_f32 = s->logits;
    p.ld_out = s->ld_logits;
    p.row_max = s->row_max;  // the greedy posterior merges these instead of re-reading the logits
    return g;
  };
  if (rc == MV_OK) {
    GemmPhase g = qkv_phase(0);
    ProfScope ps(s, st, MV_PROF_GEMM_QKV);
    rc = launch_gemm_chain(&g, 1, nullptr, st);
  }
  const float scale = 1.0f / sqrtf((float)d.head_dim);
  // the layer's attention inside its projection chain: one sequence of at most 64 rows, and a cache short enough
  // for the warp-level attention (longer caches take the tcgen05 attention as its own launch, every step)
  const bool try_fuse = s->fuse_attention && nseq == 1 && n <= kSeqRows &&
                        (d.head_dim == 64 || d.head_dim == 128) && s->s_max <= kAttnLongCacheRows;
  for (int l = 0; l < d.n_layers && rc == MV_OK; ++l) {
    const int pl = b0 * 2 * d.n_layers + 2 * l;  // sequence b0's planes of layer l
    // O, gate/up and down of this layer, then the next layer's QKV (or the LM head): one launch
    GemmPhase ch[kGemmMaxPhases];
    int nph = 0;
    ch[nph++] = residual_phase(m->m_o[l], two ? &m->m_o2[l] : nullptr, s->m_attn, s->m_attn2[gi], HD);
    ch[nph++] = gate_up_phase(l);
    ch[nph++] = residual_phase(m->m_down[l], two ? &m->m_down2[l] : nullptr, s->m_act, s->m_act2[gi], d.ffn);
    if (l + 1 < d.n_layers)
      ch[nph++] = qkv_phase(l + 1);
    else if (lm)
      ch[nph++] = lm_phase();
    if (try_fuse) {  // the layer's attention inside the same launch, ahead of the O projection
      GemmAttn ga{};
      ga.kmap = ga.vmap = s->m_kv;
      ga.D = d.head_dim;
      attn::Args& a = ga.args;
      a.q = s->q;
      a.out = s->attn;
      a.anc = t->d_ancestors;
      a.d_prefix = s->cur_len + b0;
      a.H = d.n_heads;
      a.S_max = s->s_max;
      a.n = n;
      a.plane_k = pl;
      a.plane_v = pl + 1;
      a.scale_log2 = scale * 1.4426950408889634f;
      a.err = mv_error_word();
      ProfScope ps(s, st, MV_PROF_GEMM_CHAIN);
      rc = launch_gemm_chain(ch, nph, s->chain_flags, st, false, &ga);
      if (rc != MV_ERR_UNSUPPORTED) continue;
      rc = MV_OK;  // this shape cannot fuse: separate launches below
    }
    {
      ProfScope ps(s, st, MV_PROF_ATTENTION);
      rc = launch_tree_attention_n(s->m_kv, s->m_kv, pl, pl + 1, s->q, d.n_heads, d.head_dim, s->s_max,
                                   s->cur_len + b0, 0, s->s_max - n, t, n, scale, s->attn, s->ws_attn, st, nseq,
                                   2 * d.n_layers);
    }
    if (rc != MV_OK) break;
    ProfScope ps(s, st, MV_PROF_GEMM_CHAIN);
    rc = launch_gemm_chain(ch, nph, s->chain_flags, st);
  }
  return rc;
}

// Medusa heads of sequence b on row result[b].next_node of its block of the pass (x rows from row0), then
// cur_len[b] += result[b].n_tokens.
mv_status run_heads(mv_session* s, int b, int row0, cudaStream_t st) {
  ProfScope ps(s, st, MV_PROF_HEADS);
  const mv_model* m = s->model;
  const mv_model_dims& d = m->dims;
  if (m->dtype == MV_DTYPE_F32)
    return launch_f32_heads(s->x, kTok, s->result + b, d.norm_eps, d.d, d.n_medusa, m->f_w1, m->f_w2, d.vocab,
                            s->topk, s->head_topk + (size_t)b * d.n_medusa * s->topk, s->cur_len + b, s->ws_heads,
                            st);
  return launch_heads(nullptr, s->x + (size_t)row0 * d.d, s->result + b, d.norm_eps, 1, d.d, d.n_medusa, m->w1,
                      m->w2, d.vocab, s->topk, nullptr, s->head_topk + (size_t)b * d.n_medusa * s->topk, nullptr,
                      nullptr, s->cur_len + b, s->ws_heads, st);
}

}  // namespace

extern "C" mv_status mv_model_create(const mv_model_dims* dims, const mv_model_weights* w, mv_model** out) {
  if (!dims || !w || !out) return MV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(*dims)) return MV_ERR_SHAPE;
  const mv_model_dims& d = *dims;
  if (!w->embed || !w->lm_head || !w->medusa_w1 || !w->medusa_w2 || !w->wqkv || !w->wo || !w->w_gate ||
      !w->w_up || !w->w_down)
    return MV_ERR_INVALID_ARG;
  mv_model* m = new mv_model();
  m->dims = d;
  m->packed = w->packed ? 1 : 0;
  m->embed = w->embed;
  m->lm_head = w->lm_head;
  m->w1 = w->medusa_w1;
  m->w2 = w->medusa_w2;
  const int HD = d.n_heads * d.head_dim;
  bool ok = true;
  m->m_qkv.resize(d.n_layers);
  m->m_o.resize(d.n_layers);
  m->m_gate.resize(d.n_layers);
  m->m_up.resize(d.n_layers);
  m->m_down.resize(d.n_layers);
  for (int l = 0; l < d.n_layers && ok; ++l) {
    const uint16_t* ptrs[5] = {w->wqkv[l], w->wo[l], w->w_gate[l], w->w_up[l], w->w_down[l]};
    for (const uint16_t* p : ptrs) ok = ok && p && !(reinterpret_cast<uintptr_t>(p) & 15);
    if (!ok) break;
    m->wqkv.push_back(w->wqkv[l]);
    m->wo.push_back(w->wo[l]);
    m->w_gate.push_back(w->w_gate[l]);
    m->w_up.push_back(w->w_up[l]);
    m->w_down.push_back(w->w_down[l]);
    auto map = [&](CUtensorMap* t, const void* p, int rows, int K, int tr) {
      return m->packed ? gemm_weight_map_packed(t, p, rows, K, tr) : gemm_weight_map(t, p, rows, K, tr);
    };
    ok = map(&m->m_qkv[l], w->wqkv[l], 3 * HD, d.d, 128) && map(&m->m_o[l], w->wo[l], d.d, HD, 128) &&
         map(&m->m_gate[l], w->w_gate[l], d.ffn, d.d, 64) && map(&m->m_up[l], w->w_up[l], d.ffn, d.d, 64) &&
         map(&m->m_down[l], w->w_down[l], d.d, d.ffn, 128);
  }
  ok = ok && (m->packed ? gemm_weight_map_packed(&m->m_lm, w->lm_head, d.vocab, d.d, 128)
                        : gemm_weight_map(&m->m_lm, w->lm_head, d.vocab, d.d, 128));
  if (ok && m->packed) {
    m->m_qkv2.resize(d.n_layers);
    m->m_o2.resize(d.n_layers);
    m->m_down2.resize(d.n_layers);
    m->m_gu1.resize(d.n_layers);
    m->m_gu2.resize(d.n_layers);
    bool gu = true;
    for (int l = 0; l < d.n_layers && ok; ++l) {
      ok = gemm_weight_map_packed_depth(&m->m_qkv2[l], w->wqkv[l], 3 * HD, d.d, 128, 2) &&
           gemm_weight_map_packed_depth(&m->m_o2[l], w->wo[l], d.d, HD, 128, 2) &&
           gemm_weight_map_packed_depth(&m->m_down2[l], w->w_down[l], d.d, d.ffn, 128, 2);
      gu = gu && gemm_weight_map_paired(&m->m_gu1[l], w->w_gate[l], w->w_up[l], d.ffn, d.d, 1) &&
           gemm_weight_map_paired(&m->m_gu2[l], w->w_gate[l], w->w_up[l], d.ffn, d.d, 2);
    }
    ok = ok && gemm_weight_map_packed_depth(&m->m_lm2, w->lm_head, d.vocab, d.d, 128, 2);
    m->gu_combined = gu ? 1 : 0;
  }
  if (!ok) {
    delete m;
    return MV_ERR_SHAPE;
  }
  *out = m;
  return MV_OK;
}

extern "C" mv_status mv_model_create_f32(const mv_model_dims* dims, const mv_model_weights_f32* w, mv_model** out) {
  if (!dims || !w || !out) return MV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(*dims)) return MV_ERR_SHAPE;
  const mv_model_dims& d = *dims;
  if (!w->embed || !w->lm_head || !w->medusa_w1 || !w->medusa_w2 || !w->wqkv || !w->wo || !w->w_gate ||
      !w->w_up || !w->w_down)
    return MV_ERR_INVALID_ARG;
  mv_model* m = new mv_model();
  m->dims = d;
  m->dtype = MV_DTYPE_F32;
  m->packed = 0;
  m->embed = m->lm_head = m->w1 = m->w2 = nullptr;
  m->f_embed = w->embed;
  m->f_lm = w->lm_head;
  m->f_w1 = w->medusa_w1;
  m->f_w2 = w->medusa_w2;
  for (int l = 0; l < d.n_layers; ++l) {
    const float* ptrs[5] = {w->wqkv[l], w->wo[l], w->w_gate[l], w->w_up[l], w->w_down[l]};
    for (const float* p : ptrs)
      if (!p) {
        delete m;
        return MV_ERR_INVALID_ARG;
      }
    m->f_wqkv.push_back(w->wqkv[l]);
    m->f_wo.push_back(w->wo[l]);
    m->f_gate.push_back(w->w_gate[l]);
    m->f_up.push_back(w->w_up[l]);
    m->f_down.push_back(w->w_down[l]);
  }
  *out = m;
  return MV_OK;
}

extern "C" mv_status mv_model_create_random(const mv_model_dims* dims, uint64_t seed, double std, int32_t dtype,
                                            mv_model** out) {
  if (!dims || !out || (dtype != MV_DTYPE_BF16 && dtype != MV_DTYPE_F32) || !(std >= 0.0)) return MV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(*dims)) return MV_ERR_SHAPE;
  const mv_model_dims& d = *dims;
  const int64_t qd = (int64_t)d.n_heads * d.head_dim, L = d.n_layers, K = d.n_medusa;
  const bool bf = dtype == MV_DTYPE_BF16;
  const size_t esz = bf ? 2 : 4;
  // One tensor of the model: [M][Kc] drawn from the named streams of its row segments; the projections of a bf16
  // model in the packed layout (tile_rows), everything else row-major.
  struct T {
    std::vector<std::string> names;
    int64_t M, Kc, seg;
    int tile_rows;
    size_t off, bytes;
  };
  std::vector<T> ts;
  auto add = [&](std::vector<std::string> names, int64_t M, int64_t Kc, int64_t seg, int tr) {
    T t{std::move(names), M, Kc, seg, bf ? tr : 0, 0, 0};
    size_t n = (size_t)M * Kc;
    if (t.tile_rows) {
      size_t b = 0;
      mv_packed_weight_bytes((int32_t)M, (int32_t)Kc, t.tile_rows, &b);
      n = b / 2;
    }
    t.bytes = (n * esz + 255) & ~size_t(255);
    ts.push_back(std::move(t));
  };
  add({"embed"}, d.vocab, d.d, d.vocab, 0);
  for (int l = 0; l < L; ++l) {
    const std::string p = "layer" + std::to_string(l) + ".";
    add({p + "wq", p + "wk", p + "wv"}, 3 * qd, d.d, qd, 128);
    add({p + "wo"}, d.d, qd, d.d, 128);
    add({p + "w_gate"}, d.ffn, d.d, d.ffn, 64);
    add({p + "w_up"}, d.ffn, d.d, d.ffn, 64);
    add({p + "w_down"}, d.d, d.ffn, d.d, 128);
  }
  add({"lm_head"}, d.vocab, d.d, d.vocab, 128);
  std::vector<std::string> w1n, w2n;
  for (int k = 0; k < K; ++k) {
    w1n.push_back("medusa" + std::to_string(k) + ".w1");
    w2n.push_back("medusa" + std::to_string(k) + ".w2");
  }
  add(w1n, K * d.d, d.d, d.d, 0);
  add(w2n, K * d.vocab, d.d, d.vocab, 0);
  size_t total = 0;
  for (T& t : ts) {
    t.off = total;
    total += t.bytes;
  }
  char* base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) {
    cudaGetLastError();
    return MV_ERR_CAPACITY;
  }
  mv_status rc = MV_OK;
  for (const T& t : ts) {
    std::vector<uint64_t> keys;
    for (const std::string& nm : t.names) keys.push_back(mv_stream_key(seed, nm.c_str()));
    rc = launch_gen_normal(base + t.off, dtype, t.M, t.Kc, t.tile_rows, keys.data(), (int)keys.size(), t.seg, std,
                           nullptr);
    if (rc != MV_OK) break;
  }
  if (rc == MV_OK && cudaDeviceSynchronize() != cudaSuccess) rc = MV_ERR_CUDA;
  if (rc != MV_OK) {
    cudaFree(base);
    return rc;
  }
  size_t i = 0;
  auto next = [&]() { return base + ts[i++].off; };
  mv_model* m = nullptr;
  if (bf) {
    std::vector<const mv_bf16*> qkv(L), o(L), g(L), u(L), dn(L);
    const mv_bf16* emb = reinterpret_cast<const mv_bf16*>(next());
    for (int l = 0; l < L; ++l) {
      qkv[l] = reinterpret_cast<const mv_bf16*>(next());
      o[l] = reinterpret_cast<const mv_bf16*>(next());
      g[l] = reinterpret_cast<const mv_bf16*>(next());
      u[l] = reinterpret_cast<const mv_bf16*>(next());
      dn[l] = reinterpret_cast<const mv_bf16*>(next());
    }
    mv_model_weights w{};
    w.embed = emb;
    w.wqkv = qkv.data();
    w.wo = o.data();
    w.w_gate = g.data();
    w.w_up = u.data();
    w.w_down = dn.data();
    w.lm_head = reinterpret_cast<const mv_bf16*>(next());
    w.medusa_w1 = reinterpret_cast<const mv_bf16*>(next());
    w.medusa_w2 = reinterpret_cast<const mv_bf16*>(next());
    w.packed = 1;
    rc = mv_model_create(dims, &w, &m);
  } else {
    std::vector<const float*> qkv(L), o(L), g(L), u(L), dn(L);
    const float* emb = reinterpret_cast<const float*>(next());
    for (int l = 0; l < L; ++l) {
      qkv[l] = reinterpret_cast<const float*>(next());
      o[l] = reinterpret_cast<const float*>(next());
      g[l] = reinterpret_cast<const float*>(next());
      u[l] = reinterpret_cast<const float*>(next());
      dn[l] = reinterpret_cast<const float*>(next());
    }
    mv_model_weights_f32 w{};
    w.embed = emb;
    w.wqkv = qkv.data();
    w.wo = o.data();
    w.w_gate = g.data();
    w.w_up = u.data();
    w.w_down = dn.data();
    w.lm_head = reinterpret_cast<const float*>(next());
    w.medusa_w1 = reinterpret_cast<const float*>(next());
    w.medusa_w2 = reinterpret_cast<const float*>(next());
    rc = mv_model_create_f32(dims, &w, &m);
  }
  if (rc != MV_OK) {
    cudaFree(base);
    return rc;
  }
  m->owned = base;
  *out = m;
  return MV_OK;
}

extern "C" int32_t mv_model_dtype(const mv_model* m) { return m ? m->dtype : -1; }

extern "C" void mv_model_destroy(mv_model* m) {
  if (!m) return;
  if (m->owned) cudaFree(m->owned);
  delete m;
}

extern "C" mv_status mv_session_workspace(const mv_model* m, int32_t s_max, int32_t topk, size_t* bytes) {
  if (!m || !bytes || s_max < 1 || topk < 1 || topk > 16) return MV_ERR_INVALID_ARG;
  *bytes = session_layout(m->dims, s_max, topk, m->dtype).total;
  return MV_OK;
}

extern "C" mv_status mv_batch_session_create(mv_model* m, const mv_tree* tree, int32_t batch, void* kv,
                                             int32_t s_max, int32_t topk, void* ws, size_t ws_bytes,
                                             mv_session** out) {
  if (!m || !tree || !kv || !ws || !out || batch < 1 || batch > MV_MAX_BATCH) return MV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!tree->d_ancestors) return MV_ERR_CUDA;
  const mv_model_dims& d = m->dims;
  if (topk < tree->topk || topk > 16 || tree->depth > d.n_medusa || tree->n_nodes > kTok) return MV_ERR_SHAPE;
  if (batch > 1 && tree->n_nodes > kSeqRows) return MV_ERR_SHAPE;  // one token group per sequence
  if (batch > 1 && m->dtype != MV_DTYPE_BF16) return MV_ERR_UNSUPPORTED;  // the fp32 path runs one sequence
  if (m->dtype == MV_DTYPE_F32 && d.head_dim > 128) return MV_ERR_SHAPE;
  if (s_max < kChunk + 1) return MV_ERR_CAPACITY;
  const SessionLayout L = session_layout(d, s_max, topk, m->dtype);
  if (ws_bytes < L.total) return MV_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(kv)) & 255) return MV_ERR_INVALID_ARG;
  mv_session* s = new mv_session();
  s->model = m;
  s->tree = tree;
  s->kv = static_cast<uint16_t*>(kv);
  s->s_max = s_max;
  s->topk = topk;
  s->batch = batch;
  s->kv_seq_elems = (size_t)d.n_layers * 2 * d.n_heads * s_max * d.head_dim;
  {  // MV_FUSE_ATTN=0 in the environment keeps every attention in its own launch
    const char* e = getenv("MV_FUSE_ATTN");
    s->fuse_attention = !(e && e[0] == '0');
  }
  char* b = static_cast<char*>(ws);
  s->cur_len = reinterpret_cast<int32_t*>(b + L.state);
  s->root_counter = reinterpret_cast<uint64_t*>(b + L.state + 16);
  s->result = reinterpret_cast<mv_posterior_result*>(b + L.state + 64);
  s->head_topk = reinterpret_cast<int32_t*>(b + L.state + 512);
  s->tree_tokens = reinterpret_cast<int32_t*>(b + L.tree_tokens);
  s->cart = reinterpret_cast<int32_t*>(b + L.cart);
  s->x = reinterpret_cast<float*>(b + L.x);
  s->xb = reinterpret_cast<uint16_t*>(b + L.xb);
  s->ssq = reinterpret_cast<float*>(b + L.ssq);
  s->q = reinterpret_cast<uint16_t*>(b + L.q);
  s->attn = reinterpret_cast<uint16_t*>(b + L.attn);
  s->act = reinterpret_cast<uint16_t*>(b + L.act);
  s->logits = reinterpret_cast<float*>(b + L.logits);
  s->ld_logits = (d.vocab + 3) & ~3;
  s->ws_attn = b + L.attn_ws;
  s->ws_post = b + L.post;
  s->ws_heads = b + L.heads;
  s->chain_flags = reinterpret_cast<unsigned int*>(b + L.chain);
  s->row_max = reinterpret_cast<float2*>(b + L.row_max);
  s->h_pair = reinterpret_cast<uint16_t*>(b + L.h_pair);
  const int HD = d.n_heads * d.head_dim;
  bool ok = true;
  if (m->dtype == MV_DTYPE_F32) {  // fp32 buffers over the same regions (see session_layout)
    s->xn = reinterpret_cast<float*>(b + L.xb);
    s->qkv_f = reinterpret_cast<float*>(b + L.q);
    s->q_f = s->qkv_f + (size_t)kTok * 3 * HD;
    s->attn_f = reinterpret_cast<float*>(b + L.attn);
    s->act_f = reinterpret_cast<float*>(b + L.act);
    s->xb = nullptr;
    s->ssq = nullptr;
    s->q = s->attn = s->act = nullptr;
    s->chain_flags = nullptr;
    s->row_max = nullptr;
    s->h_pair = nullptr;
    s->ws_attn = nullptr;
    s->fuse_attention = false;
  } else {
    ok = gemm_act_map(&s->m_xb, s->xb, kTok, d.d) && gemm_act_map(&s->m_attn, s->attn, kTok, HD) &&
         gemm_act_map(&s->m_act, s->act, kTok, d.ffn);
    s->act_box = ok;
    for (int g = 1; g <= mv_session::kStageMaps; ++g)
      s->act_box = s->act_box && gemm_act_map_stage(&s->m_xb2[g - 1], s->xb, kTok, d.d, g) &&
                   gemm_act_map_stage(&s->m_attn2[g - 1], s->attn, kTok, HD, g) &&
                   gemm_act_map_stage(&s->m_act2[g - 1], s->act, kTok, d.ffn, g);
    CUtensorMap vdummy;
    ok = ok && tree_attn_make_maps(&s->m_kv, &vdummy, kv, kv, d.n_heads, d.head_dim, s_max,
                                   2 * d.n_layers * batch, (size_t)d.n_heads * s_max * d.head_dim * 2);
  }
  // 64-node chain (causal) tree for prefill chunks
  s->chain = nullptr;
  if (ok) {
    // the chain is deeper than MV_MAX_DEPTH, so it is built directly rather than through mv_tree_create
    mv_tree* c = new mv_tree();
    c->n_nodes = kChunk;
    c->n_paths = 1;
    c->depth = kChunk - 1;
    c->topk = 1;
    std::vector<int32_t> pos(kChunk);
    std::vector<uint64_t> anc((size_t)kChunk * MV_MASK_WORDS, 0ull);
    for (int i = 0; i < kChunk; ++i) {
      pos[i] = i;
      anc[(size_t)i * MV_MASK_WORDS] = (i == 63) ? ~0ull : ((1ull << (i + 1)) - 1);  // kChunk = 64: one word
    }
    c->h_tree_indices = c->h_retrieve = c->h_parent = nullptr;
    c->h_position_ids = nullptr;
    c->h_ancestors = nullptr;
    c->d_tree_indices = c->d_retrieve = c->d_parent = nullptr;
    c->device = tree->device;
    ok = cudaMalloc(&c->d_position_ids, kChunk * 4) == cudaSuccess &&
         cudaMalloc(&c->d_ancestors, anc.size() * 8) == cudaSuccess &&
         cudaMemcpy(c->d_position_ids, pos.data(), kChunk * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(c->d_ancestors, anc.data(), anc.size() * 8, cudaMemcpyHostToDevice) == cudaSuccess;
    s->chain = c;
  }
  ok = ok && cudaMemset(ws, 0, L.total) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    mv_session_destroy(s);
    return MV_ERR_CUDA;
  }
  *out = s;
  return MV_OK;
}

extern "C" mv_status mv_session_create(mv_model* m, const mv_tree* tree, void* kv, int32_t s_max, int32_t topk,
                                       void* ws, size_t ws_bytes, mv_session** out) {
  return mv_batch_session_create(m, tree, 1, kv, s_max, topk, ws, ws_bytes, out);
}

extern "C" void mv_session_destroy(mv_session* s) {
  if (!s) return;
  if (s->graph_exec) cudaGraphExecDestroy(s->graph_exec);
  if (s->host_graph) cudaGraphExecDestroy(s->host_graph);
  if (s->capture_stream) cudaStreamDestroy(s->capture_stream);
  for (cudaEvent_t e : s->ev_pool) cudaEventDestroy(e);
  if (s->chain) {
    cudaFree(s->chain->d_position_ids);
    cudaFree(s->chain->d_ancestors);
    delete s->chain;
  }
  delete s;
}

extern "C" mv_status mv_session_state(const mv_session* s, mv_session_state_ptrs* out) {
  if (!s || !out) return MV_ERR_INVALID_ARG;
  out->cur_len = s->cur_len;
  out->result = s->result;
  out->head_topk = s->head_topk;
  out->tree_tokens = s->tree_tokens;
  out->cart = s->cart;
  out->logits = s->logits;
  out->ld_logits = s->ld_logits;
  out->hidden = s->x;
  out->root_counter = s->root_counter;
  out->batch = s->batch;
  return MV_OK;
}

extern "C" mv_status mv_prefill_seq(mv_session* s, int32_t b, const int32_t* d_tokens, int32_t n,
                                     mv_stream stream) {
  if (!s || !d_tokens || n < 1 || b < 0 || b >= s->batch) return MV_ERR_INVALID_ARG;
  if (n + kChunk > s->s_max) return MV_ERR_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mv_status rc = mv_launch(set_int_kernel, dim3(1), dim3(1), 0, st, s->cur_len + b, 0) == cudaSuccess
                     ? mv_last_launch("prefill")
                     : MV_ERR_CUDA;
  for (int o = 0; o < n && rc == MV_OK; o += kChunk) {
    const int c = std::min(kChunk, n - o);
    const bool last = o + c == n;
    rc = forward(s, s->chain, d_tokens + o, c, last, st, 1, b);
    if (rc != MV_OK) break;
    rc = mv_launch(prefill_finish_kernel, dim3(1), dim3(1024), 0, st, s->logits, s->model->dims.vocab,
                   s->ld_logits, c, last ? 1 : 0, s->cur_len + b, s->result + b) == cudaSuccess
             ? mv_last_launch("prefill_finish")
             : MV_ERR_CUDA;
    if (rc == MV_OK && last && s->root.mode != MV_ROOT_ARGMAX)  // the root drawn from the prompt's last row
      rc = launch_sample_root(s->logits, s->model->dims.vocab, s->ld_logits, c, s->result + b, nullptr, s->root, 0,
                              s->root_counter + b, st);
  }
  if (rc == MV_OK) rc = run_heads(s, b, 0, st);
  return rc;
}

extern "C" mv_status mv_prefill(mv_session* s, const int32_t* d_tokens, int32_t n, mv_stream stream) {
  if (!s) return MV_ERR_INVALID_ARG;
  if (s->batch != 1) return MV_ERR_UNSUPPORTED;  // a batched session prefills each sequence (mv_prefill_seq)
  return mv_prefill_seq(s, 0, d_tokens, n, stream);
}

extern "C" mv_status mv_session_set_root_sampling(mv_session* s, mv_root_params params, uint64_t counter,
                                                  mv_stream stream) {
  if (!s || !mv_root_params_valid(params)) return MV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mv_launch(set_counters_kernel, dim3(1), dim3(1), 0, st, s->root_counter, counter, s->batch) != cudaSuccess)
    return MV_ERR_CUDA;
  const mv_status rc = mv_last_launch("mv_session_set_root_sampling");
  if (rc != MV_OK) return rc;
  s->root = params;
  ++s->root_epoch;
  return MV_OK;
}

extern "C" mv_status medusa_verify_step(mv_session* s, mv_accept_params prm, mv_stream stream) {
  if (!s) return MV_ERR_INVALID_ARG;
  if (prm.mode != MV_GREEDY && prm.mode != MV_TYPICAL) return MV_ERR_INVALID_ARG;
  if (prm.mode == MV_TYPICAL && !(prm.temperature > 0.0f)) return MV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const mv_tree* t = s->tree;
  const mv_model_dims& d = s->model->dims;
  const int B = s->batch;
  const int K = d.n_medusa;
  const int cart_ld = kSeqRows * (MV_MAX_DEPTH + 1);
  // sequence b's tree tokens, logits and hidden rows start at row 64 b (a batch of one uses rows 0 .. n - 1)
  auto row0 = [&](int b) { return b * kSeqRows; };
  // candidates from the previous step's root (result.next_root) and head top-k
  mv_status rc = MV_OK;
  for (int b = 0; b < B && rc == MV_OK; ++b) {
    ProfScope ps(s, st, MV_PROF_OTHER);
    rc = launch_build_candidates(&s->result[b].next_root, s->head_topk + (size_t)b * K * s->topk, s->topk, t,
                                 s->tree_tokens + row0(b), s->cart + (size_t)b * cart_ld, st);
  }
  // one backbone pass over every sequence's tree: each weight byte is read once for all of them
  if (rc == MV_OK) rc = forward(s, t, s->tree_tokens, t->n_nodes, true, st, B, 0);
  for (int b = 0; b < B && rc == MV_OK; ++b) {
    const float* lg = s->logits + (size_t)row0(b) * s->ld_logits;
    {
      ProfScope ps(s, st, MV_PROF_POSTERIOR);
      // the bf16 path's LM-head projection leaves per-tile max / argmax (greedy then reads no logits row); the
      // fp32 path's posterior reads the rows
      rc = launch_posterior(lg, d.vocab, s->ld_logits, s->tree_tokens + row0(b), t, prm, s->result + b, nullptr,
                            nullptr, s->ws_post, st, s->row_max ? s->row_max + row0(b) : nullptr,
                            s->row_max ? (d.vocab + 127) / 128 : 0, kTok);
    }
    if (rc == MV_OK && s->root.mode != MV_ROOT_ARGMAX) {  // the next root drawn from node retrieve[best][acc]
      ProfScope ps(s, st, MV_PROF_OTHER);
      rc = launch_sample_root(lg, d.vocab, s->ld_logits, t->n_nodes, s->result + b, nullptr, s->root, 0,
                              s->root_counter + b, st);
    }
    if (rc == MV_OK) {
      ProfScope ps(s, st, MV_PROF_KV_COMPACT);
      // an fp32 row of head_dim values moves as 2 head_dim bf16-sized halves: the compaction is a bit copy
      const int e = s->model->dtype == MV_DTYPE_F32 ? 2 : 1;
      rc = launch_kv_compact(s->kv + (size_t)b * s->kv_seq_elems * e, d.n_layers, d.n_heads, s->s_max,
                             d.head_dim * e, s->cur_len + b, 0, s->result + b, nullptr, st);
    }
  }
  if (rc != MV_OK) return rc;
  if (B == 1) return run_heads(s, 0, 0, st);
  // several sequences: their heads' inputs gathered as (hi, lo) rows, then one tensor-core pass over the heads'
  // weights for all of them
  ProfScope ps(s, st, MV_PROF_HEADS);
  if (mv_launch(heads_gather_kernel, dim3(B), dim3(256), 0, st, (const float*)s->x, d.d, d.norm_eps,
                (const mv_posterior_result*)s->result, s->cur_len, s->h_pair, mv_error_word()) != cudaSuccess)
    return MV_ERR_CUDA;
  if ((rc = mv_last_launch("heads_gather")) != MV_OK) return rc;
  const mv_model* m = s->model;
  return launch_heads_rows_pair(s->h_pair, B, d.d, K, m->w1, m->w2, d.vocab, s->topk, s->head_topk, s->ws_heads, st);
}

namespace {

// Enqueues one host-buffer step on `st`: seeds in, the step, result and next seeds out.
mv_status enqueue_host_step(mv_session* s, mv_accept_params prm, const int32_t* h_seeds_in, int32_t* h_result,
                            int32_t* h_seeds_out, cudaStream_t st) {
  const int k = s->model->dims.n_medusa * s->topk;
  if (h_seeds_in) {
    if (cudaMemcpyAsync(&s->result->next_root, h_seeds_in, 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(s->head_topk, h_seeds_in + 1, (size_t)k * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MV_ERR_CUDA;
  }
  mv_status rc = medusa_verify_step(s, prm, st);
  if (rc != MV_OK) return rc;
  if (cudaMemcpyAsync(h_result, s->result, sizeof(mv_posterior_result), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return MV_ERR_CUDA;
  if (h_seeds_out) {  // the next step's seeds: new root, then the head top-k
    if (cudaMemcpyAsync(h_seeds_out, &s->result->next_root, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(h_seeds_out + 1, s->head_topk, (size_t)k * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return MV_ERR_CUDA;
  }
  return MV_OK;
}

// Page-locked host memory (allocated or registered with CUDA): copies from it can be captured in a graph.
bool host_pinned(const void* p) {
  if (!p) return true;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" mv_status medusa_verify_step_host(mv_session* s, mv_accept_params prm, const int32_t* h_seeds_in,
                                             int32_t* h_result, int32_t* h_seeds_out, mv_stream stream) {
  if (!s || !h_result) return MV_ERR_INVALID_ARG;
  if (s->batch != 1) return MV_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s->profiling || !host_pinned(h_seeds_in) || !host_pinned(h_result) || !host_pinned(h_seeds_out)) {
    const mv_status rc = enqueue_host_step(s, prm, h_seeds_in, h_result, h_seeds_out, st);
    if (rc != MV_OK) return rc;
    return cudaStreamSynchronize(st) == cudaSuccess ? MV_OK : MV_ERR_CUDA;
  }
  // pinned buffers: the whole step as one graph launch (captured on first use, replayed while nothing changed)
  const bool same = s->host_graph && s->host_prm.mode == prm.mode && s->host_prm.temperature == prm.temperature &&
                    s->host_prm.eps == prm.eps && s->host_prm.delta == prm.delta &&
                    s->host_root_epoch == s->root_epoch && s->host_ptrs[0] == h_seeds_in &&
                    s->host_ptrs[1] == h_result && s->host_ptrs[2] == h_seeds_out;
  if (!same) {
    if (prm.mode != MV_GREEDY && prm.mode != MV_TYPICAL) return MV_ERR_INVALID_ARG;
    if (prm.mode == MV_TYPICAL && !(prm.temperature > 0.0f)) return MV_ERR_INVALID_ARG;
    if (s->host_graph) {
      cudaGraphExecDestroy(s->host_graph);
      s->host_graph = nullptr;
    }
    if (!s->capture_stream && cudaStreamCreateWithFlags(&s->capture_stream, cudaStreamNonBlocking) != cudaSuccess)
      return MV_ERR_CUDA;
    if (cudaStreamBeginCapture(s->capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return MV_ERR_CUDA;
    const mv_status rc = enqueue_host_step(s, prm, h_seeds_in, h_result, h_seeds_out, s->capture_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s->capture_stream, &g);
    if (rc != MV_OK || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      cudaGetLastError();  // a failed capture leaves nothing behind for later launches to report
      return rc != MV_OK ? rc : MV_ERR_CUDA;
    }
    const cudaError_t ei = cudaGraphInstantiate(&s->host_graph, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) {
      s->host_graph = nullptr;
      return MV_ERR_CUDA;
    }
    s->host_prm = prm;
    s->host_root_epoch = s->root_epoch;
    s->host_ptrs[0] = h_seeds_in;
    s->host_ptrs[1] = h_result;
    s->host_ptrs[2] = h_seeds_out;
  }
  if (cudaGraphLaunch(s->host_graph, st) != cudaSuccess) return MV_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? MV_OK : MV_ERR_CUDA;
}

extern "C" mv_status mv_session_profile(mv_session* s, int32_t enable) {
  if (!s) return MV_ERR_INVALID_ARG;
  s->profiling = enable != 0;
  if (s->profiling) {
    s->ev_used.clear();
    s->ev_next = 0;
  }
  return MV_OK;
}

extern "C" mv_status mv_session_profile_read(mv_session* s, float* ms_by_kind, int32_t* launches_by_kind) {
  if (!s || !ms_by_kind || !launches_by_kind) return MV_ERR_INVALID_ARG;
  for (int k = 0; k < MV_PROF_KINDS; ++k) {
    ms_by_kind[k] = 0.0f;
    launches_by_kind[k] = 0;
  }
  if (s->ev_next > 0 && cudaEventSynchronize(s->ev_pool[s->ev_next - 1]) != cudaSuccess) return MV_ERR_CUDA;
  for (const auto& u : s->ev_used) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, s->ev_pool[u.second], s->ev_pool[u.second + 1]) != cudaSuccess) return MV_ERR_CUDA;
    ms_by_kind[u.first] += ms;
    launches_by_kind[u.first] += 1;
  }
  s->ev_used.clear();
  s->ev_next = 0;
  return MV_OK;
}

extern "C" mv_status medusa_verify_steps_graph(mv_session* s, mv_accept_params prm, int32_t n_steps,
                                               mv_stream stream) {
  if (!s || n_steps < 1 || n_steps > 4096) return MV_ERR_INVALID_ARG;
  if (prm.mode != MV_GREEDY && prm.mode != MV_TYPICAL) return MV_ERR_INVALID_ARG;
  if (prm.mode == MV_TYPICAL && !(prm.temperature > 0.0f)) return MV_ERR_INVALID_ARG;
  const bool same = s->graph_exec && s->graph_steps == n_steps && s->graph_profiled == s->profiling &&
                    s->graph_prm.mode == prm.mode && s->graph_prm.temperature == prm.temperature &&
                    s->graph_prm.eps == prm.eps && s->graph_prm.delta == prm.delta &&
                    s->graph_root_epoch == s->root_epoch;
  if (!same) {
    if (s->graph_exec) {
      cudaGraphExecDestroy(s->graph_exec);
      s->graph_exec = nullptr;
    }
    if (!s->capture_stream && cudaStreamCreateWithFlags(&s->capture_stream, cudaStreamNonBlocking) != cudaSuccess)
      return MV_ERR_CUDA;
    if (s->profiling) {  // the graph records its own events; readings start from this capture
      s->ev_used.clear();
      s->ev_next = 0;
    }
    if (cudaStreamBeginCapture(s->capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return MV_ERR_CUDA;
    mv_status rc = MV_OK;
    for (int i = 0; i < n_steps && rc == MV_OK; ++i) rc = medusa_verify_step(s, prm, s->capture_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s->capture_stream, &g);
    if (rc != MV_OK || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return rc != MV_OK ? rc : MV_ERR_CUDA;
    }
    const cudaError_t ei = cudaGraphInstantiate(&s->graph_exec, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) {
      s->graph_exec = nullptr;
      return MV_ERR_CUDA;
    }
    s->graph_prm = prm;
    s->graph_steps = n_steps;
    s->graph_root_epoch = s->root_epoch;
    s->graph_profiled = s->profiling;
    s->profiled_graph_events = s->ev_used;
    s->profiled_graph_ev_next = s->ev_next;
  }
  if (s->graph_profiled) {  // this replay re-records the captured events
    s->ev_used = s->profiled_graph_events;
    s->ev_next = s->profiled_graph_ev_next;
  }
  return cudaGraphLaunch(s->graph_exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MV_OK : MV_ERR_CUDA;
}
