// Medusa heads with fused per-head top-k, as split-K GEMVs on the CUDA cores.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.1 Medusa heads: z_k = W2_k (SiLU(W1_k h) + h); 二.4
// generate_candidates(): the per-head top-k of the head logits (torch.topk on logits; the softmax of the head
// formula is monotone and not needed for the ranking).
//
// Both projections are bandwidth-bound GEMVs at batch 1..4 (every weight byte is used once per batch row),
// so they stream the weights with 128-bit non-allocating loads and split the dot products over all 256 threads
// of a CTA: thread t owns the 16-byte slots t, t+256, ... of every row, keeps the matching input-vector entries
// in registers for the whole CTA, and accumulates 8 rows at a time. The 8 x B partial sums are reduced with a
// warp reduce-scatter (31 shuffles for 32 values) and a 8-warp shared-memory sum.
//   heads_w1: u_k = SiLU(W1_k h) + h            (fp32 out, kept in fp32)
//   heads_w2: z_k = W2_k u_k (and W_lm h)       -> per-CTA top-k -> the last CTA of each matrix merges.
// Batches above 4 run in groups of at most 4 rows.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace {

constexpr int kT = 256;  // threads per CTA
constexpr int kR = 8;    // rows per tile

MV_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Warp reduce-scatter of N values (N a power of two <= 32): afterwards lane l holds, in v[0], the sum over the
// warp of value number l / (32 / N).
template <int N, int CNT, int O>
MV_DEV void rs_round(float (&v)[N], int lane) {
  if constexpr (O >= 1) {
    if constexpr (CNT > 1) {
      constexpr int H = CNT / 2;
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = upper ? v[i] : v[i + H];
        const float keep = upper ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      rs_round<N, H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      rs_round<N, 1, O / 2>(v, lane);
    }
  }
}

struct HeadsArgs {
  int d, K, rows, topk, ctas_per_mat;
  const uint16_t* w1;    // [K][d][d]
  const uint16_t* w2;    // [K][V][d]
  const uint16_t* w_lm;  // [V][d] or null (matrix index K of the W2 pass)
  const uint16_t* h;     // bf16 input rows [B][d] (null in step mode)
  const float* x;        // step mode: fp32 residual rows [n][d]; h = RMSNorm(x[res->next_node])
  const mv_posterior_result* res;
  float norm_eps;
  float* u;              // fp32 [B][K][d]: W1 output, W2 input
  float* cand_val;       // [n_mat][ctas_per_mat][B][topk]
  int32_t* cand_idx;
  unsigned int* tickets; // [n_mat]
  int32_t* out_idx;      // [B][K][topk]
  float* out_val;        // [B][K][topk] or null
  int32_t* out_root;     // [B] or null
  int32_t* commit_len;   // step mode: += res->n_tokens
  unsigned int* err;
};

// Fills xin with the CTA's slots of the input vector(s) of matrix `mat`.
template <int B, int NS, bool W2>
MV_DEV float load_inputs(const HeadsArgs& a, int mat, float (&xin)[NS][8][B], float* s_red) {
  const int tid = threadIdx.x, S = a.d >> 3;
  float inv_rms = 1.0f;
  int xrow = 0;
  const bool from_x = a.x != nullptr && (!W2 || mat == a.K);
  if (from_x) {
    xrow = a.res->next_node;
    float ss = 0.0f;
    for (int i = tid; i < a.d; i += kT) {
      const float v = a.x[(size_t)xrow * a.d + i];
      ss += v * v;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) s_red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int w = 0; w < kT / 32; ++w) tot += s_red[w];
    inv_rms = rsqrtf(tot / a.d + a.norm_eps);
    __syncthreads();
  }
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int slot = tid + kT * s;
#pragma unroll
    for (int b = 0; b < B; ++b) {
#pragma unroll
      for (int e = 0; e < 8; ++e) xin[s][e][b] = 0.0f;
      if (slot >= S) continue;
      if (W2 && mat < a.K) {
        const float4* p = reinterpret_cast<const float4*>(a.u + ((size_t)b * a.K + mat) * a.d + slot * 8);
        const float4 v0 = p[0], v1 = p[1];
        xin[s][0][b] = v0.x; xin[s][1][b] = v0.y; xin[s][2][b] = v0.z; xin[s][3][b] = v0.w;
        xin[s][4][b] = v1.x; xin[s][5][b] = v1.y; xin[s][6][b] = v1.z; xin[s][7][b] = v1.w;
      } else if (from_x) {
        const float4* p = reinterpret_cast<const float4*>(a.x + (size_t)xrow * a.d + slot * 8);
        const float4 v0 = p[0], v1 = p[1];
        xin[s][0][b] = v0.x * inv_rms; xin[s][1][b] = v0.y * inv_rms;
        xin[s][2][b] = v0.z * inv_rms; xin[s][3][b] = v0.w * inv_rms;
        xin[s][4][b] = v1.x * inv_rms; xin[s][5][b] = v1.y * inv_rms;
        xin[s][6][b] = v1.z * inv_rms; xin[s][7][b] = v1.w * inv_rms;
      } else {
        const uint4 v = *reinterpret_cast<const uint4*>(a.h + (size_t)b * a.d + slot * 8);
        xin[s][0][b] = bf16lo(v.x); xin[s][1][b] = bf16hi(v.x);
        xin[s][2][b] = bf16lo(v.y); xin[s][3][b] = bf16hi(v.y);
        xin[s][4][b] = bf16lo(v.z); xin[s][5][b] = bf16hi(v.z);
        xin[s][6][b] = bf16lo(v.w); xin[s][7][b] = bf16hi(v.w);
      }
    }
  }
  return inv_rms;
}

// Value of the (normalised) input h at feature `i` of batch row b, for the residual of the W1 pass.
MV_DEV float input_at(const HeadsArgs& a, int b, int i, float inv_rms) {
  if (a.x) return a.x[(size_t)a.res->next_node * a.d + i] * inv_rms;
  return __uint_as_float((uint32_t)a.h[(size_t)b * a.d + i] << 16);
}

// Warp-level top-k over n (value, index) pairs in shared memory; taken entries are set to -inf.
// Returns in lane 0 the selected pairs through the callback.
template <typename F>
MV_DEV void warp_topk(float* val, const int32_t* idx, int n, int stride, int k, F&& emit) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, bp = -1;
    for (int i = lane; i < n; i += 32) {
      const float v = val[i * stride];
      const int id = idx ? idx[i * stride] : i;
      if (v != -INFINITY && (bp < 0 || vi_better(v, id, bv, bi))) {
        bv = v;
        bi = id;
        bp = i;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int op = __shfl_xor_sync(0xffffffffu, bp, o);
      if (op >= 0 && (bp < 0 || vi_better(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
        bp = op;
      }
    }
    if (lane == 0) {
      emit(r, bv, bp < 0 ? -1 : bi);
      if (bp >= 0) val[bp * stride] = -INFINITY;
    }
    __syncwarp();
  }
}

template <int B, int NS, bool W2>
__global__ void __launch_bounds__(kT, 1) heads_kernel(const HeadsArgs a) {
  extern __shared__ float smem[];
  __shared__ float s_red[kR * B * (kT / 32) + 8];
  __shared__ bool s_last;
  pdl_trigger();
  pdl_wait();
  const int mat = blockIdx.y, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.d >> 3;
  if (a.x && a.res->next_node < 0) {
    if (tid == 0) mv_set_error(a.err, 7, MV_DEVERR_INDEX);
    return;
  }
  const int slice = (a.rows + a.ctas_per_mat - 1) / a.ctas_per_mat;
  const int r0 = cta * slice, r1 = min(a.rows, r0 + slice);
  const uint16_t* W = W2 ? (mat == a.K ? a.w_lm : a.w2 + (size_t)mat * a.rows * a.d)
                        : a.w1 + (size_t)mat * a.rows * a.d;

  float xin[NS][8][B];
  const float inv_rms = load_inputs<B, NS, W2>(a, mat, xin, s_red);
  __syncthreads();

  for (int t0 = r0; t0 < r1; t0 += kR) {
    uint4 wv[kR][NS];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const int slot = tid + kT * s;
        if (t0 + r < r1 && slot < S)
          wv[r][s] = ld_stream(W + (size_t)(t0 + r) * a.d + slot * 8);
        else
          wv[r][s] = make_uint4(0, 0, 0, 0);
      }
    }
    float v[kR * B];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float acc = 0.0f;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          const uint4 q = wv[r][s];
          acc = fmaf(bf16lo(q.x), xin[s][0][b], acc);
          acc = fmaf(bf16hi(q.x), xin[s][1][b], acc);
          acc = fmaf(bf16lo(q.y), xin[s][2][b], acc);
          acc = fmaf(bf16hi(q.y), xin[s][3][b], acc);
          acc = fmaf(bf16lo(q.z), xin[s][4][b], acc);
          acc = fmaf(bf16hi(q.z), xin[s][5][b], acc);
          acc = fmaf(bf16lo(q.w), xin[s][6][b], acc);
          acc = fmaf(bf16hi(q.w), xin[s][7][b], acc);
        }
        v[r * B + b] = acc;
      }
    }
    constexpr int N = kR * B;
    rs_round<N, N, 16>(v, lane);
    if ((lane % (32 / N)) == 0) s_red[warp * N + lane / (32 / N)] = v[0];
    __syncthreads();
    if (tid < N) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kT / 32; ++w) sum += s_red[w * N + tid];
      const int r = tid / B, b = tid % B, row = t0 + r;
      if (row < r1) {
        if (!W2)
          a.u[((size_t)b * a.K + mat) * a.d + row] = silu(sum) + input_at(a, b, row, inv_rms);
        else
          smem[(row - r0) * B + b] = sum;
      }
    }
    __syncthreads();
  }
  if (!W2) return;

  // ---- per-CTA top-k of each batch row
  const int n_here = max(0, r1 - r0);
  float* cv = a.cand_val + ((size_t)mat * a.ctas_per_mat + cta) * B * a.topk;
  int32_t* ci = a.cand_idx + ((size_t)mat * a.ctas_per_mat + cta) * B * a.topk;
  if (warp < B) {
    const int b = warp;
    warp_topk(smem + b, nullptr, n_here, B, a.topk, [&](int r, float val, int id) {
      cv[b * a.topk + r] = val;
      ci[b * a.topk + r] = id < 0 ? -1 : r0 + id;
    });
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.tickets + mat, 1u) == (unsigned)(a.ctas_per_mat - 1);
  __syncthreads();
  if (tid == 0 && a.commit_len && cta == 0 && mat == 0) *a.commit_len += a.res->n_tokens;
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of this matrix: merge all CTAs' candidates
  const int C = a.ctas_per_mat * a.topk;
  float* mval = smem;
  int32_t* midx = reinterpret_cast<int32_t*>(smem + (size_t)C * B);
  for (int e = tid; e < C * B; e += kT) {
    const int c = e / (B * a.topk), rem = e % (B * a.topk), b = rem / a.topk, r = rem % a.topk;
    const size_t src = (((size_t)mat * a.ctas_per_mat + c) * B + b) * a.topk + r;
    const int id = __ldcg(a.cand_idx + src);
    mval[(size_t)(c * a.topk + r) * B + b] = id < 0 ? -INFINITY : __ldcg(a.cand_val + src);
    midx[(size_t)(c * a.topk + r) * B + b] = id;
  }
  __syncthreads();
  if (warp < B) {
    const int b = warp;
    warp_topk(mval + b, midx + b, C, B, a.topk, [&](int r, float val, int id) {
      if (mat < a.K) {
        a.out_idx[((size_t)b * a.K + mat) * a.topk + r] = id;
        if (a.out_val) a.out_val[((size_t)b * a.K + mat) * a.topk + r] = val;
      } else if (r == 0 && a.out_root) {
        a.out_root[b] = id;
      }
    });
  }
  if (tid == 0) a.tickets[mat] = 0u;
}

template <int B, int NS>
mv_status launch_pair(HeadsArgs a, int V, bool with_lm, int w2_ctas, cudaStream_t stream) {
  const int sms = mv_sm_count();
  // W1: K matrices of d rows
  HeadsArgs a1 = a;
  a1.rows = a.d;
  a1.ctas_per_mat = max(1, (2 * sms + a.K - 1) / a.K);
  a1.ctas_per_mat = min(a1.ctas_per_mat, max(1, a.d / kR));
  if (mv_launch(heads_kernel<B, NS, false>, dim3(a1.ctas_per_mat, a.K), dim3(kT), 0, stream, a1) != cudaSuccess)
    return MV_ERR_CUDA;
  mv_status s = mv_last_launch("heads_w1");
  if (s != MV_OK) return s;
  // W2: K matrices (+ the LM head) of V rows
  HeadsArgs a2 = a;
  const int n_mat = a.K + (with_lm ? 1 : 0);
  a2.rows = V;
  a2.ctas_per_mat = w2_ctas;
  const int slice = (V + a2.ctas_per_mat - 1) / a2.ctas_per_mat;
  const size_t smem = std::max<size_t>((size_t)slice * B * sizeof(float),
                                       (size_t)a2.ctas_per_mat * a.topk * B * (sizeof(float) + sizeof(int32_t)));
  auto kern = heads_kernel<B, NS, true>;
  static int flags[64] = {0};
  if (!mv_set_smem_once((const void*)kern, (int)smem, flags)) return MV_ERR_CUDA;
  if (mv_launch(kern, dim3(a2.ctas_per_mat, n_mat), dim3(kT), smem, stream, a2) != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("heads_w2");
}

template <int NS>
mv_status launch_group(HeadsArgs a, int B, int V, bool with_lm, int w2_ctas, cudaStream_t stream) {
  if (B == 1) return launch_pair<1, NS>(a, V, with_lm, w2_ctas, stream);
  if (B == 2) return launch_pair<2, NS>(a, V, with_lm, w2_ctas, stream);
  if constexpr (NS <= 2) {
    if (B == 4) return launch_pair<4, NS>(a, V, with_lm, w2_ctas, stream);
  }
  return MV_ERR_SHAPE;
}

}  // namespace


// ---------------------------------------------------------------------------------------------------------
// Batched path (B >= 2): the heads as tcgen05 projections over the B rows, which read every weight once (the
// split-K GEMV above re-reads them per group of rows and its CUDA-core multiply-adds grow with B).
//   t = W1 h                      one projection over the K heads' W1 stacked ([K*d][d]), fp32 out
//   u = SiLU(t) + h               kept to about fp32 precision as a bf16 pair: u_hi = bf16(u), u_lo = bf16(u - u_hi)
//                                 in token rows b and 16 + b of the activations
//   z_k = W2_k u_hi + W2_k u_lo   one projection per head over those 32 rows (one launch, independent phases)
//   top-k of z_k per row; root = argmax of W_lm h
// ---------------------------------------------------------------------------------------------------------
namespace {

constexpr int kHiLo = 16;  // lo rows start here (B <= 16)
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// pair: h (and so t) holds a hi row j and a lo row kHiLo + j per input row, summed here.
__global__ void __launch_bounds__(256) heads_prep_kernel(const float* t, const uint16_t* h, int B, int Kd, int d,
                                                         uint16_t* u, int pair) {
  pdl_wait();
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < (size_t)kHiLo * Kd;
       e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e / Kd), R = (int)(e % Kd);
    uint16_t hi = 0, lo = 0;
    if (j < B) {
      float tv = __ldcg(t + (size_t)j * Kd + R);
      float hv = __bfloat162float(__ushort_as_bfloat16(h[(size_t)j * d + R % d]));
      if (pair) {
        tv += __ldcg(t + (size_t)(kHiLo + j) * Kd + R);
        hv += __bfloat162float(__ushort_as_bfloat16(h[(size_t)(kHiLo + j) * d + R % d]));
      }
      const float uf = silu(tv) + hv;
      const __nv_bfloat16 bh = __float2bfloat16_rn(uf);
      hi = __bfloat16_as_ushort(bh);
      lo = __bfloat16_as_ushort(__float2bfloat16_rn(uf - __bfloat162float(bh)));
    }
    u[(size_t)j * Kd + R] = hi;
    u[(size_t)(kHiLo + j) * Kd + R] = lo;
  }
}

// One CTA per (head or LM row, batch row). The row (hi + lo products summed) is staged in shared memory when it
// fits, then k rounds of a block-wide argmax each take the best entry that comes after the previous pick in the
// order (larger value first, lower id on ties), so nothing has to be marked as taken.
constexpr int kTopThreads = 1024;
constexpr size_t kTopSmemMax = 160 * 1024;

MV_DEV void better_of(float& bv, int& bi, float v, int i) {
  if (bi < 0 || (i >= 0 && vi_better(v, i, bv, bi))) {
    bv = v;
    bi = i;
  }
}

template <bool kStaged>
__global__ void __launch_bounds__(kTopThreads) heads_topk_kernel(const float* zl, int ldz, const float* lm, int V,
                                                                 int K, int topk, int32_t* out_idx, float* out_val,
                                                                 int32_t* out_root) {
  extern __shared__ float row[];  // [V] when staged
  __shared__ float s_v[kTopThreads / 32];
  __shared__ int s_i[kTopThreads / 32];
  pdl_wait();
  const int mat = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_lm = mat == K;
  const int k = is_lm ? 1 : topk;
  const float* z0 = is_lm ? lm + (size_t)b * V : zl + (size_t)b * ldz + (size_t)mat * V;
  const float* z1 = is_lm ? nullptr : zl + (size_t)(kHiLo + b) * ldz + (size_t)mat * V;
  auto zat = [&](int v) { return z1 ? __ldcg(z0 + v) + __ldcg(z1 + v) : __ldcg(z0 + v); };
  if constexpr (kStaged) {
    for (int v = tid; v < V; v += kTopThreads) row[v] = zat(v);
    __syncthreads();
  }
  float pv = INFINITY;  // the previous pick (none yet: every entry comes after it)
  int pi = -1;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = -1;
    for (int v = tid; v < V; v += kTopThreads) {
      const float z = kStaged ? row[v] : zat(v);
      if (pi < 0 || vi_better(pv, pi, z, v)) better_of(bv, bi, z, v);  // z comes after the previous pick
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      better_of(bv, bi, ov, oi);
    }
    if (lane == 0) {
      s_v[warp] = bv;
      s_i[warp] = bi;
    }
    __syncthreads();
    bv = s_v[0];
    bi = s_i[0];
#pragma unroll
    for (int w = 1; w < kTopThreads / 32; ++w) better_of(bv, bi, s_v[w], s_i[w]);
    __syncthreads();  // every thread read this round's partials
    if (tid == 0) {
      if (is_lm) {
        if (out_root) out_root[b] = bi;
      } else {
        out_idx[((size_t)b * K + mat) * topk + r] = bi;
        if (out_val) out_val[((size_t)b * K + mat) * topk + r] = bv;
      }
    }
    pv = bv;
    pi = bi;
    if (bi < 0) break;  // fewer than k entries (cannot happen for topk <= V)
  }
}

size_t heads_gemm_ws_bytes(int B, int d, int K, int V, bool lm) {
  const size_t Kd = (size_t)K * d;
  size_t bytes = 0;
  bytes += align256((size_t)2 * kHiLo * Kd * 4);    // t (hi and lo rows when h is a pair)
  bytes += align256((size_t)2 * kHiLo * Kd * 2);    // u (hi rows, lo rows)
  bytes += align256((size_t)2 * kHiLo * K * V * 4); // z (hi and lo products)
  if (lm) bytes += align256((size_t)B * V * 4);     // LM row
  return bytes + 256;
}

mv_status launch_heads_gemm(const uint16_t* h, int B, int d, int K, const uint16_t* w1, const uint16_t* w2, int V,
                            int topk, const uint16_t* w_lm, int32_t* out_idx, float* out_val, int32_t* out_root,
                            void* ws, cudaStream_t stream, bool pair = false) {
  const int Kd = K * d;
  const int hrows = pair ? 2 * kHiLo : B;  // rows of h (and of t): hi rows, then lo rows from kHiLo
  char* p = static_cast<char*>(ws);
  float* t = reinterpret_cast<float*>(p);
  p += align256((size_t)2 * kHiLo * Kd * 4);
  uint16_t* u = reinterpret_cast<uint16_t*>(p);
  p += align256((size_t)2 * kHiLo * Kd * 2);
  float* zl = reinterpret_cast<float*>(p);
  p += align256((size_t)2 * kHiLo * K * V * 4);
  float* lmz = w_lm ? reinterpret_cast<float*>(p) : nullptr;
  auto base = [&](int n) {
    GemmParams q{};
    q.n_tok = n;
    q.err = mv_error_word();
    return q;
  };
  // t = W1 h (and the LM row, independent of it, in the same launch)
  GemmPhase ph[kGemmMaxPhases];
  int np = 0;
  {
    GemmPhase& g = ph[np++];
    g.epi = EPI_STORE;
    if (!gemm_weight_map(&g.a0, w1, Kd, d, 128) || !gemm_act_map(&g.b, h, hrows, d)) return MV_ERR_CUDA;
    g.a1 = g.a0;
    g.p = base(hrows);
    g.p.M = Kd;
    g.p.K = d;
    g.p.out_f32 = t;
    g.p.ld_out = Kd;
  }
  if (w_lm) {
    GemmPhase& g = ph[np++];
    g.epi = EPI_STORE;
    if (!gemm_weight_map(&g.a0, w_lm, V, d, 128) || !gemm_act_map(&g.b, h, B, d)) return MV_ERR_CUDA;
    g.a1 = g.a0;
    g.p = base(B);
    g.p.M = V;
    g.p.K = d;
    g.p.out_f32 = lmz;
    g.p.ld_out = V;
  }
  mv_status s = launch_gemm_chain(ph, np, nullptr, stream, true);
  if (s != MV_OK) return s;
  // u = SiLU(t) + h as a bf16 (hi, lo) pair
  const int blocks = (int)std::min<size_t>(((size_t)kHiLo * Kd + 255) / 256, (size_t)mv_sm_count() * 8);
  if (mv_launch(heads_prep_kernel, dim3(blocks), dim3(256), 0, stream, t, h, B, Kd, d, u, pair ? 1 : 0) !=
      cudaSuccess)
    return MV_ERR_CUDA;
  if ((s = mv_last_launch("heads_prep")) != MV_OK) return s;
  // z_k = W2_k u for the 32 rows (hi and lo), up to kGemmMaxPhases heads per launch
  for (int k0 = 0; k0 < K; k0 += kGemmMaxPhases) {
    const int nk = std::min(kGemmMaxPhases, K - k0);
    for (int i = 0; i < nk; ++i) {
      const int kk = k0 + i;
      GemmPhase& g = ph[i];
      g.epi = EPI_STORE;
      if (!gemm_weight_map(&g.a0, w2 + (size_t)kk * V * d, V, d, 128) ||
          !gemm_act_map_strided(&g.b, u + (size_t)kk * d, 2 * kHiLo, d, Kd))
        return MV_ERR_CUDA;
      g.a1 = g.a0;
      g.p = base(2 * kHiLo);
      g.p.M = V;
      g.p.K = d;
      g.p.out_f32 = zl + (size_t)kk * V;
      g.p.ld_out = K * V;
    }
    if ((s = launch_gemm_chain(ph, nk, nullptr, stream, true)) != MV_OK) return s;
  }
  const size_t row_bytes = (size_t)V * sizeof(float);
  const dim3 grid(K + (w_lm ? 1 : 0), B);
  cudaError_t e;
  if (row_bytes <= kTopSmemMax) {
    static int flags[64] = {0};
    if (!mv_set_smem_once((const void*)heads_topk_kernel<true>, (int)row_bytes, flags)) return MV_ERR_CUDA;
    e = mv_launch(heads_topk_kernel<true>, grid, dim3(kTopThreads), row_bytes, stream, (const float*)zl, K * V,
                  (const float*)lmz, V, K, topk, out_idx, out_val, out_root);
  } else {
    e = mv_launch(heads_topk_kernel<false>, grid, dim3(kTopThreads), 0, stream, (const float*)zl, K * V,
                  (const float*)lmz, V, K, topk, out_idx, out_val, out_root);
  }
  if (e != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("heads_topk");
}

}  // namespace

mv_status launch_heads_rows_pair(const uint16_t* h_pair, int B, int d, int K, const uint16_t* w1, const uint16_t* w2,
                                 int V, int topk, int32_t* out_idx, void* ws, cudaStream_t stream) {
  if (B < 1 || B > kHiLo) return MV_ERR_SHAPE;
  return launch_heads_gemm(h_pair, B, d, K, w1, w2, V, topk, nullptr, out_idx, nullptr, nullptr, ws, stream, true);
}

int heads_w2_ctas_per_mat(int n_mat, int V) {
  const int sms = mv_sm_count();
  int c = max(1, (2 * sms + n_mat - 1) / n_mat);
  return min(c, max(1, V / 64));
}

size_t heads_ws_bytes(int B, int d, int K, int V, int topk) {
  const int n_mat = K + 1;
  const int c = heads_w2_ctas_per_mat(n_mat, V);
  size_t bytes = 256;                                                   // tickets
  bytes += (size_t)min(B, 4) * K * d * sizeof(float);                   // u
  bytes += (size_t)n_mat * c * min(B, 4) * topk * (sizeof(float) + 4);  // candidates
  bytes += 256;
  if (B >= 2) bytes = std::max(bytes, heads_gemm_ws_bytes(B, d, K, V, true));  // the batched path
  return bytes;
}

mv_status launch_heads(const uint16_t* h, const float* x, const mv_posterior_result* res, float norm_eps, int B,
                       int d, int K, const uint16_t* w1, const uint16_t* w2, int V, int topk, const uint16_t* w_lm,
                       int32_t* out_idx, float* out_val, int32_t* out_root, int32_t* commit_len, void* ws,
                       cudaStream_t stream) {
  const int n_mat = K + 1;
  const int c = heads_w2_ctas_per_mat(n_mat, V);
  char* p = static_cast<char*>(ws);
  HeadsArgs a{};
  a.d = d;
  a.K = K;
  a.topk = topk;
  a.w_lm = w_lm;
  a.x = x;
  a.res = res;
  a.norm_eps = norm_eps;
  a.tickets = reinterpret_cast<unsigned int*>(p);
  a.u = reinterpret_cast<float*>(p + 256);
  a.cand_val = a.u + (size_t)min(B, 4) * K * d;
  a.cand_idx = reinterpret_cast<int32_t*>(a.cand_val + (size_t)n_mat * c * min(B, 4) * topk);
  a.err = mv_error_word();
  const int S = d / 8;
  const int NS = (S + kT - 1) / kT;  // 16-byte slots per thread
  for (int b0 = 0; b0 < B;) {
    int g = B - b0;
    const int gmax = NS <= 2 ? 4 : 2;
    g = g >= gmax ? gmax : (g >= 2 ? 2 : 1);
    HeadsArgs ag = a;
    ag.h = h ? h + (size_t)b0 * d : nullptr;
    ag.out_idx = out_idx + (size_t)b0 * K * topk;
    ag.out_val = out_val ? out_val + (size_t)b0 * K * topk : nullptr;
    ag.out_root = out_root ? out_root + b0 : nullptr;
    ag.commit_len = b0 == 0 ? commit_len : nullptr;
    ag.w1 = w1;
    ag.w2 = w2;
    mv_status s;
    if (NS == 1)
      s = launch_group<1>(ag, g, V, w_lm != nullptr, c, stream);
    else if (NS == 2)
      s = launch_group<2>(ag, g, V, w_lm != nullptr, c, stream);
    else if (NS <= 4)
      s = launch_group<4>(ag, g, V, w_lm != nullptr, c, stream);
    else
      s = MV_ERR_SHAPE;
    if (s != MV_OK) return s;
    b0 += g;
  }
  return MV_OK;
}

extern "C" mv_status medusa_heads_topk_workspace(int32_t B, int32_t d, int32_t K, int32_t V, int32_t topk,
                                                 size_t* bytes) {
  if (!bytes || B < 1 || B > 16 || d < 8 || d > 8192 || (d & 7) || K < 1 || K > 8 || topk < 1 || topk > 16 ||
      V < topk)
    return MV_ERR_SHAPE;
  *bytes = heads_ws_bytes(B, d, K, V, topk);
  return MV_OK;
}

extern "C" mv_status medusa_heads_topk(const mv_bf16* h, int32_t B, int32_t d, int32_t K, const mv_bf16* w1,
                                       const mv_bf16* w2, int32_t V, int32_t topk, const mv_bf16* w_lm,
                                       int32_t* out_idx, float* out_val, int32_t* out_root, void* workspace,
                                       size_t ws_bytes, mv_stream stream) {
  if (!h || !w1 || !w2 || !out_idx || !workspace) return MV_ERR_INVALID_ARG;
  size_t need = 0;
  mv_status s = medusa_heads_topk_workspace(B, d, K, V, topk, &need);
  if (s != MV_OK) return s;
  if (ws_bytes < need) return MV_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(w1) | reinterpret_cast<uintptr_t>(w2) |
       reinterpret_cast<uintptr_t>(w_lm)) & 15)
    return MV_ERR_SHAPE;
  if (B >= 2)  // several rows: the weights are read once by the tensor-core projections
    return launch_heads_gemm(h, B, d, K, w1, w2, V, topk, w_lm, out_idx, out_val, out_root, workspace,
                             static_cast<cudaStream_t>(stream));
  return launch_heads(h, nullptr, nullptr, 0.0f, B, d, K, w1, w2, V, topk, w_lm, out_idx, out_val, out_root,
                      nullptr, workspace, static_cast<cudaStream_t>(stream));
}
