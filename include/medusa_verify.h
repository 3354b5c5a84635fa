/*
 * medusa_verify.h -- C ABI of libmedusa_verify.so, the Medusa tree-verify decode step on one GB300 (sm_103a).
 *
 * Sources of the operations (cited by page title and section):
 *   [M5]  "大模型推理 memory bandwidth bound (5) - Medusa" (dtcms.com): 一.1 Medusa heads, 一.2 Tree attention,
 *         一.3 Typical acceptance, 二.2 generate_medusa_buffers(), 二.4 generate_candidates(),
 *         二.5 tree_decoding(), 二.6 evaluate_posterior(), 二.7 update_inference_inputs().
 *   [P3]  "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu" article (lqnn.cn): 4️⃣ tree attention mask.
 *   [OP]  "OpenPangu7B-with-Medusa" README: 4 (static tree tensors, fixed mask, few host-device round trips).
 *
 * Conventions (every entry point):
 *   - Pointers named d_* or documented "device" are device pointers owned by the caller (e.g. PyTorch tensors);
 *     they must stay valid until the stream work completes. Host pointers are read before the call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and is asynchronous; no entry
 *     point synchronises the device except mv_get_error().
 *   - Argument errors are reported synchronously, before anything is launched. Errors found by the kernels
 *     (a bounded wait that expired, an index read from device memory out of range) set a sticky device word
 *     that mv_get_error() returns; the kernels then stop early and leave outputs unspecified.
 *   - bf16 values are IEEE bfloat16 bit patterns (mv_bf16 = uint16_t), ABI-compatible with __nv_bfloat16.
 *   - Workspaces are caller-allocated device memory of at least the size the matching *_workspace() call
 *     returns. They must be zero-filled before their first use; every call leaves the counters it uses in
 *     them back at zero. Calls that share a workspace must be ordered on one stream.
 *   - Not thread-safe per handle.
 *   - The library looks up the device addresses of its own device arrays (the error word, the scratch of
 *     evaluate_posterior_noalloc) once per device and keeps them: do not call cudaDeviceReset on a device the
 *     library has used while the process goes on using the library.
 */
#ifndef MEDUSA_VERIFY_H
#define MEDUSA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mv_bf16;
typedef void* mv_stream; /* cudaStream_t */

typedef enum mv_status {
  MV_OK = 0,
  MV_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum */
  MV_ERR_SHAPE = 2,       /* sizes the kernels do not support or that disagree with a handle */
  MV_ERR_TREE = 3,        /* malformed tree: not prefix-closed, duplicate, rank >= topk, too many nodes */
  MV_ERR_CAPACITY = 4,    /* prefix + tree exceeds the cache, or workspace too small */
  MV_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  MV_ERR_DEVICE = 6,      /* the device error word was set (see mv_get_error) */
  MV_ERR_UNSUPPORTED = 7
} mv_status;

#define MV_MAX_NODES 256 /* tree nodes (root included) */
#define MV_MASK_WORDS 4  /* 64-bit ancestor words per node: the attention mask row of MV_MAX_NODES bits */
#define MV_MAX_DEPTH 8  /* longest root-to-leaf path, root excluded */
#define MV_MAX_BATCH 4  /* sequences of one batched session */

/* ============================================================================================
 * Static token tree  [M5 二.2 generate_medusa_buffers()], [OP 4]
 * ============================================================================================
 * Built once on the host from the choice list (rank tuples, root excluded); a host copy and a device copy
 * (on the current device) are owned by the handle. Node order: root = 0, then the tuples sorted by
 * (length, lexicographic). tree_indices[i] = 0 for the root, 1 + topk*(len-1) + last rank otherwise (index
 * into [root, head-1 top-k, head-2 top-k, ...]). position_ids[i] = depth. retrieve: one row per leaf,
 * leaves in descending node order, root-to-leaf node list padded with -1 to depth+1 entries.
 * ancestors[i][w]: bit b set iff node 64w + b is node i or one of its ancestors (the tree attention mask row;
 * MV_MASK_WORDS words per node, words past the tree's last node zero).
 */
typedef struct mv_tree mv_tree;

typedef struct mv_tree_desc {
  int32_t n_nodes, n_paths, depth, topk;
  const int32_t* tree_indices;   /* host [n_nodes] */
  const int32_t* position_ids;   /* host [n_nodes] */
  const int32_t* retrieve;       /* host [n_paths][depth+1] */
  const int32_t* parent;         /* host [n_nodes], -1 for the root */
  const uint64_t* ancestors;     /* host [n_nodes][MV_MASK_WORDS] */
  const int32_t* d_tree_indices; /* device copies of the above */
  const int32_t* d_position_ids;
  const int32_t* d_retrieve;
  const int32_t* d_parent;
  const uint64_t* d_ancestors;
} mv_tree_desc;

/* ranks: all tuples concatenated; lens[c] = length of tuple c (>= 1). topk: ranks per head (>= 1).
 * Errors: MV_ERR_INVALID_ARG (null / n_choices < 0 / topk < 1), MV_ERR_TREE (see above; also depth >
 * MV_MAX_DEPTH or more than MV_MAX_NODES nodes), MV_ERR_CUDA (device copy failed). *out is set on MV_OK. */
mv_status mv_tree_create(const int32_t* ranks, const int32_t* lens, int32_t n_choices, int32_t topk, mv_tree** out);
mv_status mv_tree_describe(const mv_tree* tree, mv_tree_desc* out);
void mv_tree_destroy(mv_tree* tree);

/* ============================================================================================
 * Medusa heads + per-head top-k  [M5 一.1 Medusa heads, 二.4 generate_candidates()]
 * ============================================================================================
 * For each batch row b and head k:  z = W2_k (SiLU(W1_k h_b) + h_b);  out = the topk largest entries of z
 * (larger value first; equal values: lower token id first). With w_lm != NULL also root[b] = argmax of
 * W_lm h_b (lowest id on ties). Weights are bf16, accumulation fp32, SiLU output and residual kept in fp32.
 *   h      device bf16 [B][d]            w1   device bf16 [K][d][d]  (row = output feature)
 *   w2     device bf16 [K][V][d]         w_lm device bf16 [V][d] or NULL
 *   out_idx device int32 [B][K][topk]    out_val device fp32 [B][K][topk]   out_root device int32 [B] or NULL
 * Limits: 1 <= B <= 16, d % 8 == 0, 8 <= d <= 8192, 1 <= topk <= 16, topk <= V, 1 <= K <= 8.
 * workspace: device memory of medusa_heads_topk_workspace() bytes, 16-byte aligned, zero-filled before its first
 * use; a call leaves its control words zero again, so the same workspace serves later calls on the same stream.
 */
mv_status medusa_heads_topk_workspace(int32_t B, int32_t d, int32_t K, int32_t V, int32_t topk, size_t* bytes);
mv_status medusa_heads_topk(const mv_bf16* h, int32_t B, int32_t d, int32_t K, const mv_bf16* w1,
                            const mv_bf16* w2, int32_t V, int32_t topk, const mv_bf16* w_lm, int32_t* out_idx,
                            float* out_val, int32_t* out_root, void* workspace, size_t ws_bytes, mv_stream stream);

/* ============================================================================================
 * Candidate gather into the tree  [M5 二.4 generate_candidates()]
 * ============================================================================================
 * candidates = [root, head_topk[0][0..topk), head_topk[1][...], ...];  tree_tokens[i] = candidates[tree_indices[i]];
 * cart[p][j] = tree_tokens[retrieve[p][j]], or 0 where retrieve is -1.
 *   d_root device int32 [1]; d_head_topk device int32 [K][ld_topk] (first tree.topk entries of each row used);
 *   d_tree_tokens device int32 [n_nodes]; d_cart device int32 [n_paths][depth+1] or NULL.
 * Limits: K >= tree depth, ld_topk >= tree topk.
 */
mv_status build_candidates(const int32_t* d_root, const int32_t* d_head_topk, int32_t K, int32_t ld_topk,
                           const mv_tree* tree, int32_t* d_tree_tokens, int32_t* d_cart, mv_stream stream);

/* ============================================================================================
 * Tree attention  [M5 一.2 Tree attention, 二.5 tree_decoding()], [P3 4️⃣]
 * ============================================================================================
 * For tree node i and head h:  out[i][h] = softmax_j(scale * q[i][h] . K[h][j]) V[h][j]  over the keys
 * j in [0, prefix_len) (the whole cached prefix) and j = prefix_len + a for every ancestor-or-self a of i.
 * The tree block's keys/values must already be in the cache at rows prefix_len .. prefix_len + n_nodes - 1.
 *   q device bf16 [n_nodes][H][D];  k_cache, v_cache device bf16 [H][S_max][D];  out device bf16 [n_nodes][H][D].
 * Softmax and accumulation in fp32. Limits: D in {16, 32, 64, 128}; prefix_len >= 0;
 * prefix_len + n_nodes <= S_max; 1 <= H <= 256; pointers 16-byte aligned.
 */
mv_status tree_attention_workspace(int32_t H, int32_t D, int32_t S_max, int32_t n_nodes, size_t* bytes);
mv_status tree_attention(const mv_bf16* q, const mv_bf16* k_cache, const mv_bf16* v_cache, int32_t H, int32_t D,
                         int32_t S_max, int32_t prefix_len, const mv_tree* tree, float scale, mv_bf16* out,
                         void* workspace, size_t ws_bytes, mv_stream stream);

/* ============================================================================================
 * Posterior evaluation  [M5 一.3 Typical acceptance, 二.6 evaluate_posterior()]
 * ============================================================================================
 * Per tree node n (row n of logits): greedy: argmax; typical: p = softmax(z/T), H = -sum p log(p + 1e-5),
 * tau = min(eps, delta * exp(-H)). Per path p and position j the candidate tree_tokens[retrieve[p][j+1]] is
 * accepted iff it equals argmax of node retrieve[p][j] (greedy) or p(candidate) > tau (typical). Positions
 * past a path's end (-1) are never accepted. acc_p = leading accepted count; best = greedy: first row with the
 * largest acc; typical: among those rows, largest sum of log p(candidate) over the accepted positions, then
 * first row; acc = 0 -> row 0. The root of the next step is argmax of the logits of node retrieve[best][acc]
 * (the temperature-0 / "fast" root of [M5 二.4]).
 */
typedef enum { MV_GREEDY = 0, MV_TYPICAL = 1 } mv_mode;
typedef struct mv_accept_params {
  int32_t mode;      /* mv_mode */
  float temperature; /* typical only, > 0 (default 0.7) */
  float eps;         /* posterior_threshold, default 0.09 */
  float delta;       /* posterior_alpha, default 0.3 */
} mv_accept_params;

/* Device-resident result of one verification (all int32). */
typedef struct mv_posterior_result {
  int32_t best;                       /* retrieve row of the best path */
  int32_t acc;                        /* accepted candidates on it (0 .. depth) */
  int32_t next_node;                  /* retrieve[best][acc] */
  int32_t next_root;                  /* argmax of that node's logits */
  int32_t n_tokens;                   /* acc + 1 */
  int32_t nodes[MV_MAX_DEPTH + 1];    /* retrieve[best][0..acc] */
  int32_t tokens[MV_MAX_DEPTH + 1];   /* tree_tokens[nodes[j]]: the tokens this step emits */
} mv_posterior_result;

/* logits device fp32 [n_nodes][ld] (ld >= V, ld % 4 == 0, rows 16-byte aligned); d_tree_tokens device int32
 * [n_nodes]; d_out device mv_posterior_result; d_node_stats device fp32 [n_nodes][4] or NULL, receives
 * (max logit, log of the softmax normaliser of z/T relative to that max, entropy H, tau) -- entries 1..3 are
 * 0 in greedy mode; d_node_argmax device int32 [n_nodes] or NULL. */
mv_status evaluate_posterior_workspace(int32_t n_nodes, size_t* bytes);
mv_status evaluate_posterior(const float* logits, int32_t V, int32_t ld, const int32_t* d_tree_tokens,
                             const mv_tree* tree, mv_accept_params params, mv_posterior_result* d_out,
                             float* d_node_stats, int32_t* d_node_argmax, void* workspace, size_t ws_bytes,
                             mv_stream stream);

/* evaluate_posterior without a workspace. The paper has no counterpart: this entry point exists for callers
 * that cannot call cudaMalloc -- code running under another runtime's memory manager that owns every device
 * allocation, or a serving loop that must not touch the device allocator after start-up. It computes exactly
 * what evaluate_posterior computes (same arguments minus the workspace). Its scratch is a fixed 2048-byte
 * __device__ array inside the library (every GPU that loads the library holds it until the process exits),
 * enough for MV_NOALLOC_MAX_NODES tree nodes (a limit of its own, below MV_MAX_NODES); a larger tree is rejected
 * with MV_ERR_CAPACITY. The first call on
 * a device looks up that array's device address (cudaGetSymbolAddress) with the device current; make that
 * first call before any stream capture. Each call clears the array's completion counter on `stream` before
 * its kernel. All calls share the one array, so calls that overlap on the GPU (other streams, other threads)
 * race: order them. Never allocates. */
#define MV_NOALLOC_MAX_NODES 64 /* tree nodes evaluate_posterior_noalloc accepts */
mv_status evaluate_posterior_noalloc(const float* logits, int32_t V, int32_t ld, const int32_t* d_tree_tokens,
                                     const mv_tree* tree, mv_accept_params params, mv_posterior_result* d_out,
                                     float* d_node_stats, int32_t* d_node_argmax, mv_stream stream);

/* ============================================================================================
 * Stochastic root  [M5 二.4 generate_candidates(): get_typical_one_token, get_nucleus_one_token; 一.3]
 * ============================================================================================
 * For temperature > 0 without the "fast" flag the page draws the root token (the first candidate) from the
 * LM logits instead of taking their argmax; 二.1 medusa_generate() defaults top_p = 0.8. The pages do not print
 * the two samplers; this library computes these readings of them:
 *   MV_ROOT_TYPICAL: p = softmax(z / T) restricted to {p > tau}, tau = min(eps, delta * exp(-H)),
 *                    H = -sum p log(p + 1e-5) (the typical-acceptance quantities of 一.3), renormalised;
 *   MV_ROOT_NUCLEUS: the smallest leading set of tokens (logits descending, equal logits by lower index) whose
 *                    probability mass reaches top_p, renormalised;
 *   MV_ROOT_ARGMAX:  the first largest logit (the "fast" root; temperature and the rest are ignored).
 * The draw takes u = (w >> 11) * 2^-53 with w = SplitMix64 word `counter` of the stream with 64-bit `key`
 * (mix(key + (counter + 1) * 0x9E3779B97F4A7C15), Steele, Lea and Flood, OOPSLA 2014) and returns the first
 * token in vocabulary order whose cumulative kept probability exceeds u. Probability masses are summed as
 * fixed-point integers (exp((z - max) / T) * 2^40), so the token does not depend on the order of additions.
 */
typedef enum { MV_ROOT_ARGMAX = 0, MV_ROOT_TYPICAL = 1, MV_ROOT_NUCLEUS = 2 } mv_root_mode;
typedef struct mv_root_params {
  int32_t mode;      /* mv_root_mode */
  float temperature; /* > 0 for TYPICAL / NUCLEUS */
  float eps;         /* TYPICAL: posterior_threshold (0.09), >= 0 */
  float delta;       /* TYPICAL: posterior_alpha (0.3), >= 0 */
  float top_p;       /* NUCLEUS: 0 < top_p <= 1 (0.8) */
  uint32_t reserved; /* 0 */
  uint64_t key;      /* generator key */
} mv_root_params;

/* One draw from the logits row d_logits[0..V) (device fp32) into *d_token (device int32), on one CTA.
 * Errors: MV_ERR_INVALID_ARG (null pointer, V < 1, bad mode, temperature <= 0, top_p outside (0, 1], negative
 * eps / delta). A row whose logits are all NaN gives token 0. */
mv_status sample_root(const float* d_logits, int32_t V, mv_root_params params, uint64_t counter, int32_t* d_token,
                      mv_stream stream);

/* ============================================================================================
 * KV compaction  [M5 二.7 update_inference_inputs()]
 * ============================================================================================
 * For every layer l, K/V plane c and head h:  kv[l][c][h][prefix + j] = (old) kv[l][c][h][prefix + nodes[j]]
 * for j = 0..acc, with acc and nodes from d_res; then *d_cur_len = prefix + acc + 1. Rows are gathered before
 * any is written, so overlapping source/destination rows are safe.
 *   kv device bf16 [L][2][H][S_max][D]; d_cur_len device int32 [1] (may be NULL).
 * Limits: D % 4 == 0, D <= 256, prefix_len + MV_MAX_NODES <= S_max is not required but every accessed row
 * (prefix + nodes[j]) must be < S_max (checked on the device: MV_ERR_DEVICE).
 */
mv_status kv_compact(mv_bf16* kv, int32_t L, int32_t H, int32_t S_max, int32_t D, int32_t prefix_len,
                     const mv_posterior_result* d_res, int32_t* d_cur_len, mv_stream stream);

/* ============================================================================================
 * Projection over up to 256 tokens on the tcgen05 tensor cores  [M5 二.5 tree_decoding()]
 * ============================================================================================
 * out[j][r] = sum_k x[j][k] * w[r][k] for j < n, r < M (fp32 accumulate and output): the kernel every backbone
 * projection of the verify step runs, exposed with a plain-store epilogue.
 *   w device bf16 [M][K] (16-byte aligned), x device bf16 [n][K], out device fp32 [n][ld_out].
 * Limits: 1 <= n <= 256, K % 8 == 0, ld_out >= M, at most 1024 tiles of 128 rows. The tokens go through the
 * tensor cores in groups of 64 (one, two or four per launch), every weight block read once for all of them.
 * workspace / ws_bytes are reserved: the kernel keeps its split-K partial sums in on-chip (distributed shared)
 * memory, mv_linear_bf16_workspace reports 0 bytes and workspace may be null. */
mv_status mv_linear_bf16_workspace(size_t* bytes);
mv_status mv_linear_bf16(const mv_bf16* w, const mv_bf16* x, float* out, int32_t M, int32_t K, int32_t n,
                         int32_t ld_out, void* workspace, size_t ws_bytes, mv_stream stream);
/* The same with w_packed = mv_pack_weight(w, tile_rows = 128). */
mv_status mv_linear_bf16_packed(const mv_bf16* w_packed, const mv_bf16* x, float* out, int32_t M, int32_t K,
                                int32_t n, int32_t ld_out, void* workspace, size_t ws_bytes, mv_stream stream);

/* ============================================================================================
 * Model, decode session, verify step  [M5 二.1 medusa_generate(), 二.3 - 二.7]
 * ============================================================================================
 * A Llama-style decoder: x = E[token]; per layer: x += Wo . attn(RoPE(Wq a), RoPE(Wk a), Wv a) with
 * a = RMSNorm(x); x += Wdown . (SiLU(Wgate a) * (Wup a)) with a = RMSNorm(x); logits = Wlm . RMSNorm(x).
 * RMSNorm gains are 1 (x / sqrt(mean(x^2) + norm_eps)); RoPE pairs (i, i + head_dim/2) with base rope_theta;
 * attention scale 1/sqrt(head_dim); q heads == kv heads. Medusa heads read RMSNorm(x) of the node that is
 * consumed (see medusa_heads_topk).
 * Weights are caller-owned device bf16 matrices [out][in] that must outlive the model handle. */
typedef struct mv_model_dims {
  int32_t d, n_layers, n_heads, head_dim, ffn, vocab, n_medusa;
  float rope_theta, norm_eps;
} mv_model_dims;

typedef struct mv_model_weights {
  const mv_bf16* embed;             /* [vocab][d] */
  const mv_bf16* const* wqkv;       /* host array of n_layers device pointers, each [3*n_heads*head_dim][d]:
                                       the q rows, then the k rows, then the v rows */
  const mv_bf16* const* wo;         /* [d][n_heads*head_dim] per layer */
  const mv_bf16* const* w_gate;     /* [ffn][d] per layer */
  const mv_bf16* const* w_up;       /* [ffn][d] per layer */
  const mv_bf16* const* w_down;     /* [d][ffn] per layer */
  const mv_bf16* lm_head;           /* [vocab][d] */
  const mv_bf16* medusa_w1;         /* [n_medusa][d][d] */
  const mv_bf16* medusa_w2;         /* [n_medusa][vocab][d] */
  int32_t packed;                   /* 0: every matrix row-major as above. 1: wqkv, wo, w_down, lm_head in the
                                       packed layout of mv_pack_weight with tile_rows 128, w_gate and w_up with
                                       tile_rows 64 (embed and the Medusa matrices stay row-major) */
} mv_model_weights;

/* Packed weight layout for the projection kernel: dst[tm][kb][r][c] = src[tm*tile_rows + r][kb*64 + c]
 * (zero where out of range), tile_rows in {64, 128}. Each (tile_rows x 64) block the kernel loads is then one
 * contiguous run of memory. src device bf16 [M][K]; dst device bf16 of mv_packed_weight_bytes() bytes.
 * Asynchronous on `stream`. */
mv_status mv_packed_weight_bytes(int32_t M, int32_t K, int32_t tile_rows, size_t* bytes);
mv_status mv_pack_weight(const mv_bf16* src, mv_bf16* dst, int32_t M, int32_t K, int32_t tile_rows, mv_stream stream);

typedef struct mv_model mv_model;
typedef struct mv_session mv_session;

/* Storage and arithmetic type of a model: its weights, activations and KV cache. */
typedef enum { MV_DTYPE_BF16 = 0, MV_DTYPE_F32 = 1 } mv_dtype;

/* Limits: d % 8 == 0, d <= 8192, head_dim in {16, 32, 64, 128}, ffn % 8 == 0, 1 <= n_medusa <= 8; every
 * pointer 16-byte aligned. MV_ERR_SHAPE otherwise. Builds the weights' TMA descriptors (host only). */
mv_status mv_model_create(const mv_model_dims* dims, const mv_model_weights* weights, mv_model** out);

/* An fp32 model: the same decoder with fp32 weights (row-major [out][in], the layouts of mv_model_weights, never
 * packed), fp32 activations and an fp32 KV cache; every product and sum of its verify step is fp32 (plain FMA on
 * the CUDA cores: a correctness precision for small models, not tuned for speed). Caller-owned device weights that
 * must outlive the handle. Limits as mv_model_create; its sessions take batch 1 only. */
typedef struct mv_model_weights_f32 {
  const float* embed;         /* [vocab][d] */
  const float* const* wqkv;   /* host array of n_layers device pointers, each [3*n_heads*head_dim][d] */
  const float* const* wo;     /* [d][n_heads*head_dim] per layer */
  const float* const* w_gate; /* [ffn][d] per layer */
  const float* const* w_up;   /* [ffn][d] per layer */
  const float* const* w_down; /* [d][ffn] per layer */
  const float* lm_head;       /* [vocab][d] */
  const float* medusa_w1;     /* [n_medusa][d][d] */
  const float* medusa_w2;     /* [n_medusa][vocab][d] */
} mv_model_weights_f32;
mv_status mv_model_create_f32(const mv_model_dims* dims, const mv_model_weights_f32* weights, mv_model** out);

/* A random-init model of `dtype` (MV_DTYPE_BF16 or MV_DTYPE_F32) whose weights the library draws into device
 * memory it allocates (on the current device) and frees in mv_model_destroy. Every matrix and the embedding is
 * N(0, std^2) from mv_fill_normal's generator under `seed`, one stream per tensor name: "embed", "lm_head",
 * "layer<l>.wq", "layer<l>.wk", "layer<l>.wv", "layer<l>.wo", "layer<l>.w_gate", "layer<l>.w_up",
 * "layer<l>.w_down", "medusa<k>.w1", "medusa<k>.w2" (element i = row-major index within the tensor). The
 * projections of a bf16 model are stored in the packed layout. Synchronises the device.
 * Errors: MV_ERR_INVALID_ARG (null, bad dtype, std < 0), MV_ERR_SHAPE (as mv_model_create), MV_ERR_CAPACITY (the
 * allocation failed), MV_ERR_CUDA. */
mv_status mv_model_create_random(const mv_model_dims* dims, uint64_t seed, double std, int32_t dtype,
                                 mv_model** out);
/* MV_DTYPE_BF16 or MV_DTYPE_F32; -1 for NULL. */
int32_t mv_model_dtype(const mv_model* model);
void mv_model_destroy(mv_model* model);

/* The library's generator of random inputs: dst[i] (i < count, device memory of `dtype`) = round(z_i * std) with
 * z_i the Box-Muller normal (Box and Muller, 1958; cosine branch) sqrt(-2 ln u1) cos(2 pi u2) of
 * u1 = ((w_{2i} >> 11) + 1) 2^-53 and u2 = (w_{2i+1} >> 11) 2^-53, w_j the SplitMix64 output (Steele, Lea
 * and Flood, OOPSLA 2014) of key + (j + 1) * 0x9E3779B97F4A7C15, key = mix(fnv1a64(name) ^ mix(seed)) with mix
 * the SplitMix64 output function. Evaluated in float64 without fused multiply-adds, rounded to fp32 and, for bf16, from there to
 * bf16 (round to nearest even both times). Asynchronous on `stream`. */
mv_status mv_fill_normal(void* dst, int32_t dtype, int64_t count, uint64_t seed, const char* name, double std,
                         mv_stream stream);

/* A session binds a model, a tree, a KV cache kv [n_layers][2][n_heads][s_max][head_dim] (of the model's dtype:
 * bf16, or fp32 for an fp32 model; caller-owned, 256-byte aligned, finite values in every row (e.g. zero-filled):
 * a key tile that ends past the tree reads rows beyond it and weights them by zero) and a workspace (caller-owned device memory of mv_session_workspace() bytes, 256-byte
 * aligned; zero-filled by mv_session_create, which is synchronous). The decode state (current length, the
 * last posterior result whose next_root is the next root, the head top-k) lives in the workspace.
 * Limits: tree depth <= n_medusa, tree topk <= topk <= 16, s_max >= 65. */
mv_status mv_session_workspace(const mv_model* model, int32_t s_max, int32_t topk, size_t* bytes);
mv_status mv_session_create(mv_model* model, const mv_tree* tree, void* kv, int32_t s_max, int32_t topk,
                            void* workspace, size_t ws_bytes, mv_session** out);
/* Batch > 1 verify (the pages' code supports only batch 1, 二.1 medusa_generate()): `batch` independent
 * sequences (1 .. MV_MAX_BATCH) of the same tree (at most 64 nodes when batch > 1) in one session, kv
 * [batch][n_layers][2][n_heads][s_max][head_dim]. Each verify step runs one backbone pass over all the
 * sequences' trees, so every weight byte is read once per step for the whole batch; candidates, posterior,
 * root, KV compaction and heads run per sequence. Same workspace size as mv_session_workspace(). A batch of one
 * is mv_session_create. Errors: MV_ERR_INVALID_ARG (batch outside 1 .. MV_MAX_BATCH, null pointers),
 * MV_ERR_SHAPE (as mv_session_create; also a tree over 64 nodes with batch > 1), MV_ERR_UNSUPPORTED (batch > 1 of
 * an fp32 model). */
mv_status mv_batch_session_create(mv_model* model, const mv_tree* tree, int32_t batch, void* kv, int32_t s_max,
                                  int32_t topk, void* workspace, size_t ws_bytes, mv_session** out);
void mv_session_destroy(mv_session* session);

typedef struct mv_session_state_ptrs {
  int32_t* cur_len;             /* device [1]: tokens in the KV cache */
  mv_posterior_result* result;  /* device: the last verification (next_root = the next step's root) */
  int32_t* head_topk;           /* device [n_medusa][topk]: the next step's head candidates */
  int32_t* tree_tokens;         /* device [n_nodes]: the last step's tree tokens */
  int32_t* cart;                /* device [n_paths][depth+1] */
  float* logits;                /* device fp32 [MV_MAX_NODES][ld_logits]: the last forward's LM logits */
  int32_t ld_logits;
  float* hidden;                /* device fp32 [MV_MAX_NODES][d]: the last forward's residual stream (before the
                                   final norm) */
  uint64_t* root_counter;       /* device [batch]: generator counter of each sequence's next sampled root */
  int32_t batch;                /* sequences of the session; the arrays above then hold one entry per sequence:
                                   cur_len[b], result[b], head_topk[b][n_medusa][topk], root_counter[b];
                                   tree_tokens, logits and hidden rows of sequence b start at row 64 b, cart rows
                                   at 64 b (9 entries each) */
} mv_session_state_ptrs;
mv_status mv_session_state(const mv_session* session, mv_session_state_ptrs* out);

/* Prefill [M5 二.3 initialize_medusa()]: runs tokens d_tokens[0..n) causally from position 0 (chunks of 64),
 * then sets the root (argmax of the last logits row), the head top-k (heads on the last token) and
 * cur_len = n. Limits: 1 <= n, n + 64 <= s_max. A batched session returns MV_ERR_UNSUPPORTED (use
 * mv_prefill_seq). */
mv_status mv_prefill(mv_session* session, const int32_t* d_tokens, int32_t n, mv_stream stream);
/* The same for sequence `seq` (0 <= seq < batch) of a session: its cache, length, root and head top-k. */
mv_status mv_prefill_seq(mv_session* session, int32_t seq, const int32_t* d_tokens, int32_t n, mv_stream stream);

/* Root sampling of a session (default MV_ROOT_ARGMAX): the root after mv_prefill and after every verify step
 * is drawn as sample_root() describes from the logits row of node retrieve[best][acc] (the prefill: the
 * prompt's last row), with the counter held in device memory, starting at `counter` (sequence b of a batched
 * session at counter + b * 2^32) and advancing by one per draw. The verify step's acceptance rule stays the one of its mv_accept_params. Enqueues the counter store on
 * `stream`; CUDA graphs captured earlier by medusa_verify_steps_graph are re-captured on their next call.
 * Errors: MV_ERR_INVALID_ARG as for sample_root. */
mv_status mv_session_set_root_sampling(mv_session* session, mv_root_params params, uint64_t counter,
                                       mv_stream stream);

/* One verify step [M5 二.4 - 二.7]: candidates from the state, one backbone pass over the tree (positions
 * cur_len + depth, keys/values appended at cur_len .. cur_len + n_nodes - 1), posterior, KV compaction,
 * heads on node retrieve[best][acc]; the state and result advance; cur_len grows by acc + 1. Asynchronous,
 * no host synchronisation; every step-varying quantity is read from device memory, so the call can be
 * captured in a CUDA graph and replayed. The caller must keep cur_len + n_nodes <= s_max (not checked on the
 * host; the kernels check it and set MV_ERR_DEVICE). */
mv_status medusa_verify_step(mv_session* session, mv_accept_params params, mv_stream stream);

/* The same step driven from host memory: h_seeds_in (nullable) = [root, head_topk[n_medusa][topk]] copied to
 * the device first; afterwards the result (mv_posterior_result, as int32s) is copied to h_result and, if
 * h_seeds_out is not NULL, the next seeds to h_seeds_out. Synchronises `stream` before returning. With
 * page-locked host buffers (and per-launch profiling off) the copies and the step are captured once as a CUDA
 * graph and replayed by later calls with the same params and buffers (re-captured when either changes or the
 * root sampling is set); other buffers take the launches one by one. A batched session returns
 * MV_ERR_UNSUPPORTED. */
mv_status medusa_verify_step_host(mv_session* session, mv_accept_params params, const int32_t* h_seeds_in,
                                  int32_t* h_result, int32_t* h_seeds_out, mv_stream stream);

/* n_steps consecutive verify steps as one CUDA graph: captured (on a library-owned stream) on the first call
 * with these params / n_steps / profiling setting, then replayed on `stream` with a single launch. The graph
 * reads every step-varying quantity from device memory, so each replay continues the decode. Results of the
 * intermediate steps are not kept (the session result holds the last one). With profiling enabled at capture
 * the graph records the per-launch events of all n steps; mv_session_profile_read after a replay returns them. */
mv_status medusa_verify_steps_graph(mv_session* session, mv_accept_params params, int32_t n_steps, mv_stream stream);

/* Per-launch timing of a session's kernels, for benchmarks: while enabled, every launch of medusa_verify_step /
 * mv_prefill is bracketed by CUDA events on its stream (do not enable during CUDA graph capture).
 * mv_session_profile_read waits for the last recorded event, returns the summed milliseconds and launch counts
 * per kind (indices MV_PROF_*) since profiling was enabled or last read, and resets them.
 * The verify step runs each layer's O, gate/up and down projections and the next layer's QKV projection (the
 * LM head after the last layer) as one launch, counted as MV_PROF_GEMM_CHAIN; MV_PROF_GEMM_QKV is then the first
 * layer's QKV projection alone. MV_PROF_GEMM_O / _GATE_UP / _DOWN / _LM stay for launches of a single projection. */
enum {
  MV_PROF_GEMM_QKV = 0, MV_PROF_ATTENTION = 1, MV_PROF_GEMM_O = 2, MV_PROF_GEMM_GATE_UP = 3, MV_PROF_GEMM_DOWN = 4,
  MV_PROF_GEMM_LM = 5, MV_PROF_POSTERIOR = 6, MV_PROF_KV_COMPACT = 7, MV_PROF_HEADS = 8, MV_PROF_OTHER = 9,
  MV_PROF_GEMM_CHAIN = 10, MV_PROF_KINDS = 11
};
mv_status mv_session_profile(mv_session* session, int32_t enable);
mv_status mv_session_profile_read(mv_session* session, float* ms_by_kind, int32_t* launches_by_kind);

/* ============================================================================================
 * Errors
 * ============================================================================================
 * Returns MV_OK if the current device's error word is clear, else MV_ERR_DEVICE and stores the word in *code
 * (high 16 bits: the kernel site, low 16 bits: 1 = bounded wait expired, 2 = index out of range), then clears
 * it. Synchronises the current device. */
mv_status mv_get_error(uint32_t* code);
/* Detail value recorded with the first device error since the last clear (e.g. an offending index); read
 * it before mv_get_error(), which clears both. Synchronous. */
mv_status mv_get_error_detail(uint32_t* detail);
/* Self-test of the device-side failure detection (no counterpart on the pages; a diagnostic, not part of the
 * verify path). One CTA runs the two bounded waits every kernel of the path relies on -- the acquire wait on a
 * device counter that the projection chain uses between phases, and the mbarrier wait of the TMA and bulk-copy
 * rings -- on a counter and a barrier that nothing ever completes, each with a limit of limit_ns nanoseconds
 * instead of the kernels' 2 s. Each wait gives up at its limit; the kernel then sets the device error word (site
 * 20, MV_DEVERR_TIMEOUT; detail bit 0: the counter wait expired, bit 1: the mbarrier wait expired) and returns.
 * d_out: device int32 [4]: [0] 1 if the counter wait succeeded, [1] the same for the mbarrier wait, [2] the
 * counter itself (set to 0), [3] microseconds both waits took. Nothing faults or hangs: read the result with
 * mv_get_error(). Errors: MV_ERR_INVALID_ARG (null or unaligned d_out, limit_ns outside 1 us .. 10 ms). */
mv_status mv_selftest_wait_timeout(uint32_t limit_ns, int32_t* d_out, mv_stream stream);
/* Human-readable name of a status. */
const char* mv_status_string(mv_status s);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_VERIFY_H */
