// Medusa heads with fused per-head top-k, as split-K GEMVs on the CUDA cores.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.1 Medusa heads: z_k = W2_k (SiLU(W1_k h) + h); 二.4
// generate_candidates(): the per-head top-k of the head logits (torch.topk on logits; the softmax of the head
// formula is monotone and not needed for the ranking).
//
// One input row (batch 1): both projections are bandwidth-bound GEMVs, every weight byte is used once.
// * Streaming. Each matrix is cut into tiles of R contiguous rows. A CTA (8 compute warps + 1 producer warp)
//   streams tiles through a ring of shared-memory stages with bulk copies (cp.async.bulk, an mbarrier per
//   stage, evict-first L2 policy). The CTAs of all matrices fill the SMs once.
// * Balance. A CTA's first ring-full of tiles is fixed (tile cta, cta + ctas_per_mat, ...) and issued before
//   the wait for the previous kernel, since the weights depend on no earlier kernel; every later tile is
//   claimed from a per-matrix counter, so CTAs that stream faster take more tiles and all finish together.
// * Dot products. The 256 compute threads split each row: thread t owns the 16-byte slots t, t+256, ... and
//   keeps the matching input entries in registers. A warp copies its slots of the stage to registers and
//   releases the stage at once; the R partial sums are then reduced with a warp reduce-scatter and an 8-warp
//   sum through a double-buffered shared array (one barrier of the compute warps per tile).
// * Top-k. W2 row values never go to memory: warp 0 keeps a running top-k list (lane j holds rank j) and a
//   new row enters only if it beats the list's last entry, so the list is ready when the stream ends. Each
//   CTA writes its list; the last CTA of a matrix merges them (warp lists, then one list).
//   heads_w1: u_k = SiLU(W1_k h) + h            (fp32 out, kept in fp32)
//   heads_w2: z_k = W2_k u_k (and W_lm h)       -> top-k per head (and the LM head's argmax)
// Several rows run the tensor-core path further down (one read of the weights for all rows).
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace {

constexpr int kT = 256;                 // compute threads per CTA (8 warps); warp 8 is the producer
constexpr int kThreads = kT + 32;
constexpr int kMaxStages = 4;
constexpr size_t kRing = 192 * 1024;    // shared-memory ring of one CTA
// The 256-byte control block at the start of the workspace (zero-filled before the first call; every pass
// leaves its words zero again): per pass and matrix a ticket (CTAs done) and a tile counter.
constexpr int kCtlWords = 16;  // words per pass and kind (n_mat <= 9)
MV_DEV unsigned int* ctl_ticket(unsigned int* ctl, bool w2, int mat) { return ctl + (w2 ? 2 : 0) * kCtlWords + mat; }
MV_DEV unsigned int* ctl_counter(unsigned int* ctl, bool w2, int mat) {
  return ctl + (w2 ? 3 : 1) * kCtlWords + mat;
}

template <int NS>
__host__ __device__ constexpr int rows_per_tile() { return NS <= 2 ? 8 : 4; }  // R x NS slots per thread held

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

// Barrier of the n threads of named barrier `id`; returns whether pred held for any of them.
MV_DEV bool bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
MV_DEV void bar_compute() { asm volatile("bar.sync 1, %0;" ::"n"(kT) : "memory"); }

struct HeadsArgs {
  int d, K, rows, topk, ctas_per_mat, stages;
  const uint16_t* w1;    // [K][d][d]
  const uint16_t* w2;    // [K][V][d]
  const uint16_t* w_lm;  // [V][d] or null (matrix index K of the W2 pass)
  const uint16_t* h;     // bf16 input row [d] (null in step mode)
  const float* x;        // step mode: fp32 residual rows [n][d]; h = RMSNorm(x[res->next_node])
  const mv_posterior_result* res;
  float norm_eps;
  float* u;              // fp32 [K][d]: W1 output, W2 input
  float* cand_val;       // [n_mat][ctas_per_mat][topk]
  int32_t* cand_idx;
  unsigned int* ctl;     // the control block (tickets, tile counters)
  int32_t* out_idx;      // [K][topk]
  float* out_val;        // [K][topk] or null
  int32_t* out_root;     // [1] or null
  int32_t* commit_len;   // step mode: += res->n_tokens
  unsigned int* err;
};

// Fills xin with the thread's slots of the input vector of matrix `mat`; returns the RMS scale (step mode).
// Called by the 256 compute threads.
template <int NS, bool W2>
MV_DEV float load_inputs(const HeadsArgs& a, int mat, float (&xin)[NS][8], float* s_ss) {
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
    if ((tid & 31) == 0) s_ss[tid >> 5] = ss;
    bar_compute();
    float tot = 0.0f;
    for (int w = 0; w < kT / 32; ++w) tot += s_ss[w];
    inv_rms = rsqrtf(tot / a.d + a.norm_eps);
  }
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int slot = tid + kT * s;
#pragma unroll
    for (int e = 0; e < 8; ++e) xin[s][e] = 0.0f;
    if (slot >= S) continue;
    if (W2 && mat < a.K) {
      const float4* p = reinterpret_cast<const float4*>(a.u + (size_t)mat * a.d + slot * 8);
      const float4 v0 = p[0], v1 = p[1];
      xin[s][0] = v0.x; xin[s][1] = v0.y; xin[s][2] = v0.z; xin[s][3] = v0.w;
      xin[s][4] = v1.x; xin[s][5] = v1.y; xin[s][6] = v1.z; xin[s][7] = v1.w;
    } else if (from_x) {
      const float4* p = reinterpret_cast<const float4*>(a.x + (size_t)xrow * a.d + slot * 8);
      const float4 v0 = p[0], v1 = p[1];
      xin[s][0] = v0.x * inv_rms; xin[s][1] = v0.y * inv_rms; xin[s][2] = v0.z * inv_rms;
      xin[s][3] = v0.w * inv_rms; xin[s][4] = v1.x * inv_rms; xin[s][5] = v1.y * inv_rms;
      xin[s][6] = v1.z * inv_rms; xin[s][7] = v1.w * inv_rms;
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(a.h + slot * 8);
      xin[s][0] = bf16lo(v.x); xin[s][1] = bf16hi(v.x);
      xin[s][2] = bf16lo(v.y); xin[s][3] = bf16hi(v.y);
      xin[s][4] = bf16lo(v.z); xin[s][5] = bf16hi(v.z);
      xin[s][6] = bf16lo(v.w); xin[s][7] = bf16hi(v.w);
    }
  }
  return inv_rms;
}

// Value of the (normalised) input h at feature i, for the residual of the W1 pass.
MV_DEV float input_at(const HeadsArgs& a, int i, float inv_rms) {
  if (a.x) return a.x[(size_t)a.res->next_node * a.d + i] * inv_rms;
  return __uint_as_float((uint32_t)a.h[i] << 16);
}

// A warp's running top-k list: lane j < k holds the entry of rank j (id -1: empty, worse than any entry).
struct TopList {
  float v = -INFINITY;
  int i = -1;
  // Offers each lane's candidate (cv, ci) where `has` holds; the list keeps the k best of all it was offered in
  // the order larger value first, then lower id. A candidate enters only if it beats the list's last entry.
  MV_DEV void offer(float cv, int ci, bool has, int k, int lane) {
    const float lv = __shfl_sync(0xffffffffu, v, k - 1);
    const int li = __shfl_sync(0xffffffffu, i, k - 1);
    unsigned m = __ballot_sync(0xffffffffu, has && (li < 0 || vi_better(cv, ci, lv, li)));
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const float nv = __shfl_sync(0xffffffffu, cv, src);
      const int ni = __shfl_sync(0xffffffffu, ci, src);
      const unsigned b = __ballot_sync(0xffffffffu, lane < k && (i < 0 || vi_better(nv, ni, v, i)));
      if (!b) continue;  // beaten by an entry that came in from this same group
      const int pos = __ffs(b) - 1;
      const float uv = __shfl_up_sync(0xffffffffu, v, 1);
      const int ui = __shfl_up_sync(0xffffffffu, i, 1);
      if (lane > pos) {
        v = uv;
        i = ui;
      } else if (lane == pos) {
        v = nv;
        i = ni;
      }
    }
  }
};

template <int NS, bool W2>
__global__ void __launch_bounds__(kThreads, 1) heads_kernel(const HeadsArgs a) {
  constexpr int R = rows_per_tile<NS>();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ float s_part[2][R * (kT / 32)];
  __shared__ float s_ss[kT / 32];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ int s_tile[kMaxStages];  // tile of each stage; -1: the stream has ended
  __shared__ float s_lv[(kT / 32) * 16];
  __shared__ int s_li[(kT / 32) * 16];
  __shared__ bool s_last;
  const int mat = blockIdx.y, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.d >> 3, nst = a.stages, cpm = a.ctas_per_mat;
  const size_t row_bytes = (size_t)a.d * 2, stage_bytes = R * row_bytes;
  const int n_tiles = (a.rows + R - 1) / R;
  const uint16_t* W = W2 ? (mat == a.K ? a.w_lm : a.w2 + (size_t)mat * a.rows * a.d)
                        : a.w1 + (size_t)mat * a.rows * a.d;
  unsigned int* counter = ctl_counter(a.ctl, W2, mat);
  unsigned int* ticket = ctl_ticket(a.ctl, W2, mat);

  if (tid == kT) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kT / 32);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kT / 32) {
    // ------------------------------------------------------------------ producer (one lane)
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    int pushed = 0;
    bool ended = false, ok = true;
    auto push = [&](int g) {  // g < 0: the end marker
      const int s = pushed % nst;
      s_tile[s] = g;
      if (g < 0) {
        mbar_arrive(&full[s]);
      } else {
        const uint32_t bytes = (uint32_t)(min(R, a.rows - g * R) * row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load_hint(ring + (size_t)s * stage_bytes, W + (size_t)g * R * a.d, bytes, &full[s], pol);
      }
      ++pushed;
      ended = g < 0;
    };
    // the fixed tiles first: they need nothing from earlier kernels
    for (int j = 0; j < nst && !ended; ++j) push(cta + j * cpm < n_tiles ? cta + j * cpm : -1);
    pdl_trigger();
    pdl_wait();
    const bool bad_node = a.x && a.res->next_node < 0;
    while (!ended && !bad_node) {
      const int s = pushed % nst;
      if (!mbar_wait(&empty[s], (uint32_t)((pushed / nst - 1) & 1))) {
        ok = false;
        break;
      }
      const int g = cpm * nst + (int)atomicAdd(counter, 1u);
      push(g < n_tiles ? g : -1);
    }
    if (!ok || bad_node) {  // let the copies in flight land before the CTA leaves
      if (!ok) mv_set_error(a.err, 17, MV_DEVERR_TIMEOUT);
      for (int j = max(0, pushed - nst); j < pushed; ++j)
        if (!mbar_wait(&full[j % nst], (uint32_t)((j / nst) & 1))) break;
    }
    return;
  }

  // -------------------------------------------------------------------- compute warps
  pdl_trigger();
  pdl_wait();
  if (a.x && a.res->next_node < 0) {
    if (tid == 0) mv_set_error(a.err, 7, MV_DEVERR_INDEX);
    return;
  }
  float xin[NS][8];
  const float inv_rms = load_inputs<NS, W2>(a, mat, xin, s_ss);
  TopList top;
  bool timed_out = false;
  for (int t = 0;; ++t) {
    const int s = t % nst;
    const bool ok = mbar_wait(&full[s], (uint32_t)((t / nst) & 1));
    const int g = ok ? s_tile[s] : -1;
    const int nr = g < 0 ? 0 : min(R, a.rows - g * R);
    const uint8_t* st = ring + (size_t)s * stage_bytes;
    uint4 wv[R][NS];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int q = 0; q < NS; ++q) {
        const int slot = tid + kT * q;
        wv[r][q] = (r < nr && slot < S) ? *reinterpret_cast<const uint4*>(st + r * row_bytes + (size_t)slot * 16)
                                        : make_uint4(0, 0, 0, 0);
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp's reads of the stage are done
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < NS; ++q) {
        const uint4 w = wv[r][q];
        acc = fmaf(bf16lo(w.x), xin[q][0], acc);
        acc = fmaf(bf16hi(w.x), xin[q][1], acc);
        acc = fmaf(bf16lo(w.y), xin[q][2], acc);
        acc = fmaf(bf16hi(w.y), xin[q][3], acc);
        acc = fmaf(bf16lo(w.z), xin[q][4], acc);
        acc = fmaf(bf16hi(w.z), xin[q][5], acc);
        acc = fmaf(bf16lo(w.w), xin[q][6], acc);
        acc = fmaf(bf16hi(w.w), xin[q][7], acc);
      }
      v[r] = acc;
    }
    rs_round<R, R, 16>(v, lane);
    if ((lane % (32 / R)) == 0) s_part[t & 1][warp * R + lane / (32 / R)] = v[0];
    // partials written (the other buffer was read one tile ago); leave together at the end or on a timeout
    timed_out |= !ok;
    if (bar_or(1, kT, g < 0)) break;
    if (warp == 0) {
      float sum = 0.0f;
      if (lane < nr) {
#pragma unroll
        for (int w = 0; w < kT / 32; ++w) sum += s_part[t & 1][w * R + lane];
      }
      const int row = g * R + lane;
      if (!W2) {
        if (lane < nr) a.u[(size_t)mat * a.d + row] = silu(sum) + input_at(a, row, inv_rms);
      } else {
        top.offer(sum, row, lane < nr, a.topk, lane);
      }
    }
  }
  if (timed_out) mv_set_error(a.err, 17, MV_DEVERR_TIMEOUT);

  // ---- this CTA's list; the last CTA of the matrix (every tile claimed, every list written) goes on
  const int k = a.topk;
  const size_t cbase = ((size_t)mat * cpm + cta) * k;
  if (W2 && warp == 0 && lane < k) {
    a.cand_val[cbase + lane] = top.v;
    a.cand_idx[cbase + lane] = top.i;
  }
  __threadfence();
  bar_compute();
  if (tid == 0) s_last = atomicAdd(ticket, 1u) == (unsigned)(cpm - 1);
  bar_compute();
  if (W2 && tid == 0 && a.commit_len && cta == 0 && mat == 0) *a.commit_len += a.res->n_tokens;
  if (!s_last) return;
  if (tid == 0) {  // the next call starts from zero
    *ticket = 0u;
    *counter = 0u;
  }
  if (!W2) return;
  __threadfence();

  // ---- last CTA of this matrix: merge all CTAs' lists (a list per warp, then one)
  const int C = cpm * k;
  TopList wl;
  for (int e0 = warp * 32; e0 < C; e0 += kT) {
    const int e = e0 + lane;
    const int id = e < C ? __ldcg(a.cand_idx + (size_t)mat * C + e) : -1;
    const float val = id >= 0 ? __ldcg(a.cand_val + (size_t)mat * C + e) : -INFINITY;
    wl.offer(val, id, id >= 0, k, lane);
  }
  if (lane < k) {
    s_lv[warp * 16 + lane] = wl.v;
    s_li[warp * 16 + lane] = wl.i;
  }
  bar_compute();
  if (warp == 0) {
    TopList fl;
    for (int e0 = 0; e0 < (kT / 32) * 16; e0 += 32) {
      const int e = e0 + lane, j = e % 16;
      const bool has = j < k && s_li[e] >= 0;
      fl.offer(has ? s_lv[e] : -INFINITY, has ? s_li[e] : -1, has, k, lane);
    }
    if (lane < k) {
      if (mat < a.K) {
        a.out_idx[(size_t)mat * k + lane] = fl.i;
        if (a.out_val) a.out_val[(size_t)mat * k + lane] = fl.v;
      } else if (lane == 0 && a.out_root) {
        *a.out_root = fl.i;
      }
    }
  }
}

// CTAs per matrix: the CTAs of all n_mat matrices fill the SMs once.
int heads_ctas_per_mat(int n_mat) { return std::max(1, mv_sm_count() / n_mat); }

template <int NS, bool W2>
mv_status launch_pass(HeadsArgs a, int rows, int n_mat, cudaStream_t stream) {
  constexpr int R = rows_per_tile<NS>();
  a.rows = rows;
  const int n_tiles = (rows + R - 1) / R;
  a.ctas_per_mat = std::min(heads_ctas_per_mat(n_mat), n_tiles);
  const size_t stage = (size_t)R * a.d * 2;
  a.stages = (int)std::min<size_t>(kMaxStages, kRing / stage);
  if (a.stages < 1) return MV_ERR_SHAPE;
  const size_t smem = (size_t)a.stages * stage;
  auto kern = heads_kernel<NS, W2>;
  static int flags[64] = {0};
  if (!mv_set_smem_once((const void*)kern, (int)smem, flags)) return MV_ERR_CUDA;
  if (mv_launch(kern, dim3(a.ctas_per_mat, n_mat), dim3(kThreads), smem, stream, a) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch(W2 ? "heads_w2" : "heads_w1");
}

template <int NS>
mv_status launch_row(const HeadsArgs& a, int V, bool with_lm, cudaStream_t stream) {
  mv_status s = launch_pass<NS, false>(a, a.d, a.K, stream);  // W1: K matrices of d rows
  if (s != MV_OK) return s;
  return launch_pass<NS, true>(a, V, a.K + (with_lm ? 1 : 0), stream);  // W2: K matrices (+ the LM head) of V rows
}

}  // namespace


// ---------------------------------------------------------------------------------------------------------
// Batched path (B >= 2): the heads as tcgen05 projections over the B rows, which read every weight once (the
// GEMV above reads them once per row).
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
  char* p = static_cast<char*>(ws) + 256;  // the batch-1 path's control block stays untouched
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

size_t heads_ws_bytes(int B, int d, int K, int V, int topk) {
  const int c = heads_ctas_per_mat(K);  // the W2 pass without the LM head has the most CTAs per matrix
  size_t bytes = 256;                                                  // control block (tickets, tile counters)
  bytes += (size_t)K * d * sizeof(float);                              // u
  bytes += (size_t)(K + 1) * c * topk * (sizeof(float) + sizeof(int32_t));  // candidates
  bytes += 256;
  if (B >= 2) bytes = std::max(bytes, heads_gemm_ws_bytes(B, d, K, V, true));  // the batched path
  return bytes;
}

mv_status launch_heads(const uint16_t* h, const float* x, const mv_posterior_result* res, float norm_eps, int B,
                       int d, int K, const uint16_t* w1, const uint16_t* w2, int V, int topk, const uint16_t* w_lm,
                       int32_t* out_idx, float* out_val, int32_t* out_root, int32_t* commit_len, void* ws,
                       cudaStream_t stream) {
  const int c = heads_ctas_per_mat(K);
  char* p = static_cast<char*>(ws);
  HeadsArgs a{};
  a.d = d;
  a.K = K;
  a.topk = topk;
  a.w1 = w1;
  a.w2 = w2;
  a.w_lm = w_lm;
  a.x = x;
  a.res = res;
  a.norm_eps = norm_eps;
  a.ctl = reinterpret_cast<unsigned int*>(p);
  a.u = reinterpret_cast<float*>(p + 256);
  a.cand_val = a.u + (size_t)K * d;
  a.cand_idx = reinterpret_cast<int32_t*>(a.cand_val + (size_t)(K + 1) * c * topk);
  a.err = mv_error_word();
  const int NS = (d / 8 + kT - 1) / kT;  // 16-byte slots per thread
  for (int b = 0; b < B; ++b) {  // one row at a time (the same workspace, stream-ordered)
    HeadsArgs ab = a;
    ab.h = h ? h + (size_t)b * d : nullptr;
    ab.out_idx = out_idx + (size_t)b * K * topk;
    ab.out_val = out_val ? out_val + (size_t)b * K * topk : nullptr;
    ab.out_root = out_root ? out_root + b : nullptr;
    ab.commit_len = b == 0 ? commit_len : nullptr;
    mv_status s;
    if (NS == 1)
      s = launch_row<1>(ab, V, w_lm != nullptr, stream);
    else if (NS == 2)
      s = launch_row<2>(ab, V, w_lm != nullptr, stream);
    else if (NS <= 4)
      s = launch_row<4>(ab, V, w_lm != nullptr, stream);
    else
      s = MV_ERR_SHAPE;
    if (s != MV_OK) return s;
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
