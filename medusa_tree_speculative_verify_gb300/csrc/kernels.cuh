// Internal launchers shared between the standalone entry points and the whole verify step.
#pragma once

#include "common.cuh"

mv_status launch_build_candidates(const int32_t* d_root, const int32_t* d_head_topk, int ld_topk, const mv_tree* t,
                                  int32_t* d_tree_tokens, int32_t* d_cart, cudaStream_t stream);

size_t posterior_ws_bytes(int n_nodes);
// row_max / n_row_tiles / row_ld: optional per-(128-row tile, node) max and first argmax left by the LM-head
// projection ([n_row_tiles][row_ld] float2, the index as int bits); greedy acceptance then does not read the
// logits rows.
mv_status launch_posterior(const float* logits, int V, int ld, const int32_t* d_tree_tokens, const mv_tree* t,
                           mv_accept_params prm, mv_posterior_result* d_out, float* d_stats, int32_t* d_argmax,
                           void* ws, cudaStream_t stream, const float2* row_max = nullptr, int n_row_tiles = 0,
                           int row_ld = 0);

// One root draw (see sample_root in medusa_verify.h). Row = res->next_node (checked against n_rows) when res is
// set, else row 0; the token goes to res->next_root and/or out_token; with d_counter the draw takes its counter
// from there and stores counter + 1, else it uses `counter`.
bool mv_root_params_valid(const mv_root_params& p);
mv_status launch_sample_root(const float* logits, int V, int ld, int n_rows, mv_posterior_result* res,
                             int32_t* out_token, const mv_root_params& prm, uint64_t counter, uint64_t* d_counter,
                             cudaStream_t stream);

// prefix from d_prefix if non-null, else `prefix`
mv_status launch_kv_compact(mv_bf16* kv, int L, int H, int S_max, int D, const int32_t* d_prefix, int prefix,
                            const mv_posterior_result* d_res, int32_t* d_cur_len, cudaStream_t stream);

// Heads + top-k of B rows given as bf16 (hi, lo) pairs: h_pair [32][d], hi row b and lo row 16 + b (fp32-grade
// input); the weights are read once for all rows (tensor-core projections). out_idx [B][K][topk]. ws:
// heads_ws_bytes(B >= 2, ...).
mv_status launch_heads_rows_pair(const uint16_t* h_pair, int B, int d, int K, const uint16_t* w1, const uint16_t* w2,
                                 int V, int topk, int32_t* out_idx, void* ws, cudaStream_t stream);
size_t heads_ws_bytes(int B, int d, int K, int V, int topk);
// Batch-1 GEMV path, one launch pair per row: h (bf16 [B][d]) or, in step mode (B = 1), x (fp32 rows) + res:
// h = RMSNorm(x[res->next_node]); commit_len (step mode) receives += res->n_tokens.
mv_status launch_heads(const uint16_t* h, const float* x, const mv_posterior_result* res, float norm_eps, int B,
                       int d, int K, const uint16_t* w1, const uint16_t* w2, int V, int topk, const uint16_t* w_lm,
                       int32_t* out_idx, float* out_val, int32_t* out_root, int32_t* commit_len, void* ws,
                       cudaStream_t stream);

// Tree attention over one layer. k/v tensor maps cover [H][S_max][D] planes; prefix from d_prefix if non-null.
// Caches longer than kAttnLongCacheRows rows (head dim 64 or 128) run on the tcgen05 kernel (attention_tc.cu),
// shorter ones on the warp-level kernel; a session takes one of the two for every step, so rows computed in
// different steps (a tree node and the same token decoded alone) come from the same arithmetic. The choice is
// made by capacity because the prefix length lives on the device: a session sized for long contexts spends most
// steps at long prefixes, where the tensor-core kernel is faster (at a 4096-key prefix, 26.6 against 33 us on
// GB300); at short prefixes the warp-level attention inside the projection chain costs less (7 against 16 us).
constexpr int kAttnLongCacheRows = 4096;
mv_status launch_tree_attention_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                   const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                   int max_prefix, const mv_tree* t, int n, float scale, mv_bf16* out,
                                   cudaStream_t stream, int nseq, int seq_planes);
struct TreeAttnPlan {
  int H, D, S_max, n_nodes, splits;
};
size_t tree_attn_ws_bytes(int H, int D, int S_max, int n_nodes);
bool tree_attn_make_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* k_cache, const void* v_cache, int H,
                         int D, int S_max, int planes, size_t plane_stride_bytes);
mv_status launch_tree_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                int max_prefix, const mv_tree* t, float scale, mv_bf16* out, void* ws,
                                cudaStream_t stream);
// nseq > 1: nseq sequences of the same tree (n <= 64 nodes each): sequence b's queries / outputs are rows
// 64 b .. 64 b + n - 1, its cache planes plane_k / plane_v + b * seq_planes, its prefix d_prefix[b].
mv_status launch_tree_attention_n(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                  const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                  int max_prefix, const mv_tree* t, int n, float scale, mv_bf16* out, void* ws,
                                  cudaStream_t stream, int nseq = 1, int seq_planes = 0);

// ---- the fp32 model path (f32.cu): plain FFMA kernels over fp32 weights, activations and KV cache
mv_status launch_f32_embed(const int32_t* tokens, int n, const float* E, int vocab, int d, float* x, cudaStream_t st);
mv_status launch_f32_rmsnorm(const float* x, int n, int d, float eps, float* xn, cudaStream_t st);
// epi: 0 out = in W^T, 1 out += in W^T, 2 out = SiLU(in W^T) * (in W_up^T)
mv_status launch_f32_linear(const float* in, int ld_in, const float* w, const float* w_up, int M, int K, int n,
                            float* out, int ld_out, int epi, cudaStream_t st);
mv_status launch_f32_rope_append(const float* qkv, int n, int H, int D, int S_max, const int32_t* cur_len,
                                 const int32_t* pos_ids, float rope_theta, float* q_out, float* kv_layer,
                                 cudaStream_t st);
mv_status launch_f32_tree_attention(const float* q, const float* kv_layer, int H, int D, int S_max, int n,
                                    const int32_t* cur_len, const uint64_t* anc, float scale, float* out,
                                    cudaStream_t st);
size_t f32_heads_ws_bytes(int d, int K, int V);
// heads on h = RMSNorm(x[res->next_node]) (next_node < n_rows), top-k per head into out_idx [K][topk], then
// cur_len += res->n_tokens
mv_status launch_f32_heads(const float* x, int n_rows, const mv_posterior_result* res, float eps, int d, int K,
                           const float* w1, const float* w2, int V, int topk, int32_t* out_idx, int32_t* cur_len,
                           void* ws, cudaStream_t st);
// The library's random weight generator (see mv_fill_normal): a logical [M][K] matrix whose rows fall in
// segments of seg_rows rows drawn from keys[0..n_keys), written row-major (tile_rows = 0) or in the packed layout.
uint64_t mv_stream_key(uint64_t seed, const char* name);
mv_status launch_gen_normal(void* dst, int dtype, int64_t M, int64_t K, int tile_rows, const uint64_t* keys,
                            int n_keys, int64_t seg_rows, double std, cudaStream_t st);
