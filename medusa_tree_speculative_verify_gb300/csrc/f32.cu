// The single-precision model path, and the library's random weight generator.
//
// Models kept in fp32 (weights, activations and KV cache) run the same verify step as the bf16 path -- a
// Llama-style backbone over the flattened tree ("大模型推理 memory bandwidth bound (5) - Medusa", 二.5
// tree_decoding()), tree attention where each node sees the prefix and its own root-to-node path (一.2), the
// Medusa heads z_k = W2_k (SiLU(W1_k h) + h) with their top-k (一.1, 二.4) -- with every product and sum in fp32
// on the CUDA cores. This is the precision of the small correctness configuration whose greedy stream must equal
// plain greedy decoding of the same model token for token ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu",
// 2️⃣). Nothing here is tuned for speed: one warp per output row and token in the projections, one warp per
// (node, head) in the attention. Candidates, the posterior, the root draw and the KV compaction are the
// precision-independent kernels the bf16 path uses.
//
// Random weights: element i of the tensor named `name` under `seed` is the Box-Muller normal (Box and Muller,
// 1958; cosine branch) of SplitMix64 words 2i and 2i + 1 (Steele, Lea and Flood, OOPSLA 2014) of the stream
// keyed by FNV-1a of the name mixed with the seed, scaled by std and rounded once to the storage type.
#include <math.h>

#include <vector>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kW = 8;  // warps per block of the projection and head kernels

MV_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
MV_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// x[j][:] = E[tokens[j]][:]
__global__ void __launch_bounds__(256) f32_embed_kernel(const int32_t* tokens, const float* E, int vocab, int d,
                                                        float* x, unsigned int* err) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  const int tok = tokens[j];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) mv_set_error_detail(err, 30, MV_DEVERR_INDEX, (uint32_t)tok);
    return;
  }
  for (int c = threadIdx.x; c < d; c += blockDim.x) x[(size_t)j * d + c] = E[(size_t)tok * d + c];
}

// xn[j] = x[j] / sqrt(mean(x[j]^2) + eps) (gain 1), one block per row
__global__ void __launch_bounds__(256) f32_rmsnorm_kernel(const float* x, int d, float eps, float* xn) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8];
  const int j = blockIdx.x, tid = threadIdx.x;
  const float* r = x + (size_t)j * d;
  float ss = 0.0f;
  for (int c = tid; c < d; c += 256) ss = fmaf(r[c], r[c], ss);
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  for (int c = tid; c < d; c += 256) xn[(size_t)j * d + c] = r[c] * inv;
}

enum : int { F32_STORE = 0, F32_RESIDUAL = 1, F32_SWIGLU = 2 };

// Row r = blockIdx.x * 8 + warp of the projection for token j = blockIdx.y: s = in[j] . w[r] (and, for
// F32_SWIGLU, s2 = in[j] . w_up[r]); out[j][r] = s, += s, or SiLU(s) * s2.
__global__ void __launch_bounds__(kW * 32) f32_linear_kernel(const float* in, int ld_in, const float* w,
                                                             const float* w_up, int M, int K, float* out,
                                                             int ld_out, int epi) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kW + (threadIdx.x >> 5), j = blockIdx.y;
  if (r >= M) return;
  const float* a = in + (size_t)j * ld_in;
  const float* wr = w + (size_t)r * K;
  float s = 0.0f, s2 = 0.0f;
  if (epi == F32_SWIGLU) {
    const float* ur = w_up + (size_t)r * K;
    for (int k = lane; k < K; k += 32) {
      s = fmaf(a[k], wr[k], s);
      s2 = fmaf(a[k], ur[k], s2);
    }
    s2 = warp_sum(s2);
  } else {
    for (int k = lane; k < K; k += 32) s = fmaf(a[k], wr[k], s);
  }
  s = warp_sum(s);
  if (lane == 0) {
    float* o = out + (size_t)j * ld_out + r;
    if (epi == F32_STORE)
      *o = s;
    else if (epi == F32_RESIDUAL)
      *o += s;
    else
      *o = silu(s) * s2;
  }
}

// Token j's q and k rotated at position cur_len + pos_ids[j] (pair (i, i + D/2) by the angle
// pos * theta^(-2i/D), computed in double), q to q_out [j][H][D], k and v to row cur_len + j of the layer's
// cache planes kvl [2][H][S_max][D].
__global__ void __launch_bounds__(128) f32_rope_append_kernel(const float* qkv, int H, int D, int S_max, int n,
                                                              const int32_t* cur_len, const int32_t* pos_ids,
                                                              double ln_theta, float* q_out, float* kvl,
                                                              unsigned int* err) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  const int P = *cur_len;
  if (P < 0 || P + n > S_max) {
    if (threadIdx.x == 0) mv_set_error_detail(err, 31, MV_DEVERR_INDEX, (uint32_t)P);
    return;
  }
  const int pos = P + pos_ids[j], half = D / 2, HD = H * D;
  const float* row = qkv + (size_t)j * 3 * HD;
  for (int e = threadIdx.x; e < H * half; e += blockDim.x) {
    const int h = e / half, i = e % half;
    double sn, cs;
    sincos((double)pos * exp(-(2.0 * i / D) * ln_theta), &sn, &cs);
    const float c = (float)cs, s = (float)sn;
    const float q0 = row[h * D + i], q1 = row[h * D + i + half];
    const float k0 = row[HD + h * D + i], k1 = row[HD + h * D + i + half];
    float* qo = q_out + ((size_t)j * H + h) * D;
    qo[i] = q0 * c - q1 * s;
    qo[i + half] = q1 * c + q0 * s;
    float* kr = kvl + ((size_t)h * S_max + P + j) * D;
    kr[i] = k0 * c - k1 * s;
    kr[i + half] = k1 * c + k0 * s;
    float* vr = kvl + ((size_t)(H + h) * S_max + P + j) * D;
    vr[i] = row[2 * HD + h * D + i];
    vr[i + half] = row[2 * HD + h * D + i + half];
  }
}

// out[j][h] = sum over the keys node j can see (every prefix row, and tree row P + a for each ancestor-or-self
// a of j) of softmax(scale q.k) v. One warp per (node, head): lane l scores key k0 + l of each chunk of 32 keys,
// the running max and sum are updated per chunk, and lane l accumulates output dims l, l + 32, ...
__global__ void __launch_bounds__(32) f32_tree_attn_kernel(const float* q, const float* kvl, int H, int D,
                                                           int S_max, int n, const int32_t* cur_len,
                                                           const uint64_t* anc, float scale, float* out,
                                                           unsigned int* err) {
  pdl_trigger();
  pdl_wait();
  constexpr int kMaxPerLane = 4;  // head_dim <= 128
  const int j = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
  const int P = *cur_len;
  if (P < 0 || P + n > S_max) {
    if (lane == 0) mv_set_error_detail(err, 32, MV_DEVERR_INDEX, (uint32_t)P);
    return;
  }
  const float* qr = q + ((size_t)j * H + h) * D;
  const float* K = kvl + (size_t)h * S_max * D;
  const float* V = kvl + (size_t)(H + h) * S_max * D;
  const uint64_t* aw = anc + (size_t)j * MV_MASK_WORDS;
  float acc[kMaxPerLane] = {0.0f, 0.0f, 0.0f, 0.0f};
  float m = -INFINITY, l = 0.0f;
  const int nk = P + n;
  for (int k0 = 0; k0 < nk; k0 += 32) {
    const int key = k0 + lane;
    const bool vis = key < P || (key < nk && ((aw[(key - P) >> 6] >> ((key - P) & 63)) & 1ull));
    float s = -INFINITY;
    if (vis) {
      const float* kr = K + (size_t)key * D;
      float dot = 0.0f;
      for (int t = 0; t < D; ++t) dot = fmaf(qr[t], kr[t], dot);
      s = dot * scale;
    }
    const float mn = fmaxf(m, warp_max(s));
    if (mn == -INFINITY) continue;  // nothing visible yet (the same on every lane)
    const float corr = expf(m - mn);
    const float p = vis ? expf(s - mn) : 0.0f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) acc[i] *= corr;
    const int kend = min(32, nk - k0);
    for (int kk = 0; kk < kend; ++kk) {
      const float pk = __shfl_sync(0xffffffffu, p, kk);
      if (pk == 0.0f) continue;  // the same on every lane
      const float* vr = V + (size_t)(k0 + kk) * D;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i < D) acc[i] = fmaf(pk, vr[lane + 32 * i], acc[i]);
    }
    m = mn;
  }
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i)
    if (lane + 32 * i < D) out[((size_t)j * H + h) * D + lane + 32 * i] = acc[i] * inv;
}

// Medusa head k = blockIdx.x on the consumed node: h = RMSNorm(x[res->next_node]), u_k = SiLU(W1_k h) + h.
__global__ void __launch_bounds__(kW * 32) f32_heads_u_kernel(const float* x, const mv_posterior_result* res,
                                                              int n_rows, int d, float eps, const float* w1,
                                                              float* u, unsigned int* err) {
  extern __shared__ float hs[];  // [d]
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, k = blockIdx.x;
  const int node = res->next_node;
  if (node < 0 || node >= n_rows) {
    if (tid == 0) mv_set_error_detail(err, 33, MV_DEVERR_INDEX, (uint32_t)node);
    return;
  }
  const float* xr = x + (size_t)node * d;
  float ss = 0.0f;
  for (int c = tid; c < d; c += kW * 32) ss = fmaf(xr[c], xr[c], ss);
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < kW; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  for (int c = tid; c < d; c += kW * 32) hs[c] = xr[c] * inv;
  __syncthreads();
  const float* wk = w1 + (size_t)k * d * d;
  for (int r = warp; r < d; r += kW) {
    const float* wr = wk + (size_t)r * d;
    float s = 0.0f;
    for (int c = lane; c < d; c += 32) s = fmaf(wr[c], hs[c], s);
    s = warp_sum(s);
    if (lane == 0) u[(size_t)k * d + r] = silu(s) + hs[r];
  }
}

// z[k][v] = W2_k[v] . u_k for row v = blockIdx.x * 8 + warp, head k = blockIdx.y
__global__ void __launch_bounds__(kW * 32) f32_heads_z_kernel(const float* u, const float* w2, int d, int V,
                                                              float* z) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, v = blockIdx.x * kW + (threadIdx.x >> 5), k = blockIdx.y;
  if (v >= V) return;
  const float* wr = w2 + ((size_t)k * V + v) * d;
  const float* uk = u + (size_t)k * d;
  float s = 0.0f;
  for (int c = lane; c < d; c += 32) s = fmaf(wr[c], uk[c], s);
  s = warp_sum(s);
  if (lane == 0) z[(size_t)k * V + v] = s;
}

// Top-k of head k = blockIdx.x's logits z[k] (larger first, equal values by lower id): k rounds of a block
// argmax over the entries ordered after the previous pick. Block 0 then commits cur_len += res->n_tokens.
__global__ void __launch_bounds__(1024) f32_heads_topk_kernel(const float* z, int V, int topk, int32_t* out_idx,
                                                              const mv_posterior_result* res, int32_t* cur_len) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sv[32];
  __shared__ int si[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, k = blockIdx.x;
  const float* zk = z + (size_t)k * V;
  float pv = INFINITY;
  int pi = -1;
  for (int t = 0; t < topk; ++t) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = tid; i < V; i += blockDim.x) {
      const float v = zk[i];
      if (vi_better(pv, pi, v, i) && vi_better(v, i, bv, bi)) {
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
    if (lane == 0) {
      sv[warp] = bv;
      si[warp] = bi;
    }
    __syncthreads();
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (vi_better(sv[w], si[w], bv, bi)) {
        bv = sv[w];
        bi = si[w];
      }
    __syncthreads();
    if (tid == 0) out_idx[(size_t)k * topk + t] = bi == 0x7fffffff ? 0 : bi;
    pv = bv;
    pi = bi;
  }
  if (k == 0 && tid == 0 && cur_len) *cur_len += res->n_tokens;
}

// ------------------------------------------------------------------------------------------------ generator

struct GenSpec {
  uint64_t keys[8];  // stream key of each row segment
  int64_t M, K;      // logical matrix [M][K]
  int64_t seg_rows;  // rows per segment (segment s = row / seg_rows uses keys[s], rows renumbered from 0)
  int tile_rows;     // 0: row-major; 64 / 128: the packed layout [tm][kb][r][64] of mv_pack_weight
  double std;
  int dtype;         // MV_DTYPE_BF16 or MV_DTYPE_F32
};

MV_DEV uint64_t splitmix64_word(uint64_t key, uint64_t i) {  // word i of the stream with key `key`
  uint64_t z = key + (i + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Element e of the destination (in its layout): the normal variate of its logical (row, col) scaled by std.
// Products and sums are explicitly rounded one by one (no fused multiply-add), as the plain evaluation order
// sqrt(-2 ln u1) * cos(2 pi u2) * std in float64, then one rounding to fp32 (and from there to bf16).
__global__ void __launch_bounds__(256) gen_normal_kernel(void* dst, int64_t count, GenSpec g) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t KB = (g.K + 63) / 64;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += stride) {
    int64_t row, col;
    if (g.tile_rows) {
      const int64_t c = e % 64, r = (e / 64) % g.tile_rows, kb = (e / (64 * g.tile_rows)) % KB;
      const int64_t tm = e / (64 * g.tile_rows * KB);
      row = tm * g.tile_rows + r;
      col = kb * 64 + c;
    } else {
      row = e / g.K;
      col = e % g.K;
    }
    float v = 0.0f;
    if (row < g.M && col < g.K) {
      const int64_t seg = row / g.seg_rows;
      const uint64_t i = (uint64_t)((row - seg * g.seg_rows) * g.K + col);
      const uint64_t w0 = splitmix64_word(g.keys[seg], 2 * i), w1 = splitmix64_word(g.keys[seg], 2 * i + 1);
      const double u1 = (double)((w0 >> 11) + 1ull) * 0x1p-53;  // (0, 1]
      const double u2 = (double)(w1 >> 11) * 0x1p-53;           // [0, 1)
      const double rad = sqrt(__dmul_rn(-2.0, log(u1)));
      const double zz = __dmul_rn(rad, cos(__dmul_rn(2.0 * M_PI, u2)));
      // + 0: the mean of N(0, std^2), added like the input generator adds it (so a -0 becomes +0 there too)
      v = __double2float_rn(__dadd_rn(__dmul_rn(zz, g.std), 0.0));
    }
    if (g.dtype == MV_DTYPE_F32)
      static_cast<float*>(dst)[e] = v;
    else
      static_cast<uint16_t*>(dst)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

uint64_t mix64_host(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

uint64_t mv_stream_key(uint64_t seed, const char* name) {
  uint64_t h = 0xCBF29CE484222325ull;  // FNV-1a, 64 bit
  for (const unsigned char* p = reinterpret_cast<const unsigned char*>(name); *p; ++p)
    h = (h ^ *p) * 0x100000001B3ull;
  return mix64_host(h ^ mix64_host(seed));
}

mv_status launch_gen_normal(void* dst, int dtype, int64_t M, int64_t K, int tile_rows, const uint64_t* keys,
                            int n_keys, int64_t seg_rows, double std, cudaStream_t st) {
  if (n_keys < 1 || n_keys > 8 || seg_rows * n_keys < M) return MV_ERR_SHAPE;
  GenSpec g{};
  for (int i = 0; i < n_keys; ++i) g.keys[i] = keys[i];
  g.M = M;
  g.K = K;
  g.seg_rows = seg_rows;
  g.tile_rows = tile_rows;
  g.std = std;
  g.dtype = dtype;
  const int64_t count = tile_rows ? ((M + tile_rows - 1) / tile_rows) * tile_rows * ((K + 63) / 64) * 64 : M * K;
  const int blocks = (int)std::min<int64_t>((count + 255) / 256, (int64_t)mv_sm_count() * 16);
  gen_normal_kernel<<<std::max(blocks, 1), 256, 0, st>>>(dst, count, g);
  return mv_last_launch("gen_normal");
}

extern "C" mv_status mv_fill_normal(void* dst, int32_t dtype, int64_t count, uint64_t seed, const char* name,
                                    double std, mv_stream stream) {
  if (!dst || !name || count < 0 || (dtype != MV_DTYPE_BF16 && dtype != MV_DTYPE_F32)) return MV_ERR_INVALID_ARG;
  if (count == 0) return MV_OK;
  const uint64_t key = mv_stream_key(seed, name);
  return launch_gen_normal(dst, dtype, 1, count, 0, &key, 1, 1, std, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------------ launchers

mv_status launch_f32_embed(const int32_t* tokens, int n, const float* E, int vocab, int d, float* x,
                           cudaStream_t st) {
  if (mv_launch(f32_embed_kernel, dim3(n), dim3(256), 0, st, tokens, E, vocab, d, x, mv_error_word()) !=
      cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("f32_embed");
}

mv_status launch_f32_rmsnorm(const float* x, int n, int d, float eps, float* xn, cudaStream_t st) {
  if (mv_launch(f32_rmsnorm_kernel, dim3(n), dim3(256), 0, st, x, d, eps, xn) != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("f32_rmsnorm");
}

mv_status launch_f32_linear(const float* in, int ld_in, const float* w, const float* w_up, int M, int K, int n,
                            float* out, int ld_out, int epi, cudaStream_t st) {
  if (mv_launch(f32_linear_kernel, dim3((M + kW - 1) / kW, n), dim3(kW * 32), 0, st, in, ld_in, w, w_up, M, K, out,
                ld_out, epi) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("f32_linear");
}

mv_status launch_f32_rope_append(const float* qkv, int n, int H, int D, int S_max, const int32_t* cur_len,
                                 const int32_t* pos_ids, float rope_theta, float* q_out, float* kv_layer,
                                 cudaStream_t st) {
  if (mv_launch(f32_rope_append_kernel, dim3(n), dim3(128), 0, st, qkv, H, D, S_max, n, cur_len, pos_ids,
                log((double)rope_theta), q_out, kv_layer, mv_error_word()) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("f32_rope_append");
}

mv_status launch_f32_tree_attention(const float* q, const float* kv_layer, int H, int D, int S_max, int n,
                                    const int32_t* cur_len, const uint64_t* anc, float scale, float* out,
                                    cudaStream_t st) {
  if (D > 128) return MV_ERR_SHAPE;
  if (mv_launch(f32_tree_attn_kernel, dim3(n, H), dim3(32), 0, st, q, kv_layer, H, D, S_max, n, cur_len, anc, scale,
                out, mv_error_word()) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("f32_tree_attention");
}

size_t f32_heads_ws_bytes(int d, int K, int V) { return ((size_t)K * d + (size_t)K * V) * sizeof(float); }

mv_status launch_f32_heads(const float* x, int n_rows, const mv_posterior_result* res, float eps, int d, int K,
                           const float* w1, const float* w2, int V, int topk, int32_t* out_idx, int32_t* cur_len,
                           void* ws, cudaStream_t st) {
  float* u = static_cast<float*>(ws);
  float* z = u + (size_t)K * d;
  const size_t smem = (size_t)d * sizeof(float);
  if (smem > 48 * 1024) {
    static int flags[64] = {0};
    if (!mv_set_smem_once((const void*)f32_heads_u_kernel, (int)smem, flags)) return MV_ERR_CUDA;
  }
  if (mv_launch(f32_heads_u_kernel, dim3(K), dim3(kW * 32), smem, st, x, res, n_rows, d, eps, w1, u,
                mv_error_word()) != cudaSuccess ||
      mv_launch(f32_heads_z_kernel, dim3((V + kW - 1) / kW, K), dim3(kW * 32), 0, st, (const float*)u, w2, d, V,
                z) != cudaSuccess ||
      mv_launch(f32_heads_topk_kernel, dim3(K), dim3(1024), 0, st, (const float*)z, V, topk, out_idx, res,
                cur_len) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("f32_heads");
}
