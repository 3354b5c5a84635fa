// Backbone projections over the tree tokens on the 5th-generation tensor cores (tcgen05).
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.5 tree_decoding(): the backbone runs once over all tree
// tokens; at 64 tokens every weight byte feeds 64 multiply-adds, so these GEMMs stream the weights from HBM.
//
// Mapping (swap-AB): D[128 weight rows x 64 NT tokens] += W[128 x 64 k] . X[64 NT tokens x 64 k]^T per k-block,
// one tcgen05.mma.cta_group::1.kind::f16 (M=128, N=64 NT, K=16) per 16 k, for NT = 1..4 token groups of 64 (up to
// 256 tokens: larger trees, or one group per sequence of a batch). Operands come from shared memory through TMA
// (128-byte swizzle, K-major), the accumulators live in tensor memory (two buffers, so the epilogue of one tile
// overlaps the MMAs of the next). With one group the chain can also run its layer's tree attention first, on the
// epilogue warps (attn_core.cuh), while the producer streams the first projection's weights.
//
// Work split: split-K inside a thread-block cluster. Cluster q of C CTAs (C = 1, 2, 4 or 8) owns a contiguous range
// of tiles; CTA rank r of the cluster streams k-blocks [r*kbt/C, (r+1)*kbt/C) of each, so the weight bytes of a tile
// are read once. Token t of a token group belongs to CTA t mod C: after each tile every CTA drains its partial
// accumulator from TMEM and stores each value straight into the owning CTA's receive buffer with st.async, counted
// on the owner's mbarrier (no release fence on the sending side). Each owner sums the C slices of its own tokens in
// rank order (deterministic) and runs the fused epilogue on them, so the epilogue is spread over the cluster too:
//   STORE    out[token][row] = acc * s[token]                    (LM head logits, plain projections)
//   RESIDUAL x[token][row] += acc; bf16 copy; per-token sum of squares of the 128-row slice (next RMSNorm)
//   SWIGLU   act[token][f] = SiLU(s*gate) * (s*up), tile = 64 gate rows + the same 64 up rows
//   QKV      q / k / v rows, RoPE on q and k at position prefix + depth, k/v appended to the cache
// s[token] = 1/sqrt(mean(x^2) + eps) of the RMSNorm that precedes the projection (its gains are 1), applied
// to the accumulator instead of the input: x W^T * s = (x * s) W^T.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer + TMEM owner, warps 2..9 = epilogue, two
// per TMEM sub-partition (warp w reads TMEM lanes 32*(w%4) .. +31, the two of a pair take half of the columns
// each). Every mbarrier wait is bounded; on expiry the kernel records MV_DEVERR_TIMEOUT, lets its in-flight copies
// and MMAs land, frees its tensor memory and returns.
#include <float.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace {

constexpr int BM = 128, BN = 64, BK = 64;  // BN: tokens per token group
constexpr int kMaxGroups = 4;              // token groups per launch: up to 256 tokens
constexpr int kTokMax = BN * kMaxGroups;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 8 KB per token group
// Epilogue: 8 warps, two per TMEM sub-partition (warp w reads lanes 32 (w % 4) ..); the two halves of a pair drain
// the two halves of a token group's columns and finish alternate tokens of the CTA's share, so a tile's epilogue --
// the step every phase boundary waits for -- takes half as long as with one warp per sub-partition.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kAcc = 2;  // accumulator buffers in tensor memory (the MMA may run kAcc - 1 tiles ahead)
constexpr int kMaxCluster = 8;  // CTAs per cluster (portable limit)

// Per number of token groups NT (1 to 4): a stage holds one weight block and NT activation blocks, so fewer
// stages fit; one MMA of N = 64 NT per 16 k; the accumulator buffers take 2 x 64 NT TMEM columns (allocated as
// a power of two).
//
// A pipeline stage holds kKps consecutive k-blocks: their weight blocks, then their activation blocks. Two k-blocks
// per stage (32 KB of weights) stream faster than one (16 KB) with the same bytes in flight -- measured on GB300
// with a plain TMA ring of weight + activation stages: 41.8 GB/s per SM at 16 + 8 KB stages, 50.1 GB/s at 32 + 16
// KB -- since every stage costs a full / empty handshake on top of its bytes. As many stages as fit: a stage stays
// held after it lands until its MMAs have read it (eight dependent N = 64 MMAs at one group, about 0.45 us), so the
// depth sets the rate an SM streams at (the same ring with each stage held 0.45 us: 43.9 GB/s per SM with 3
// stages, 45.3 with 4).
template <int NT, bool kAttn = false>
struct Cfg {
  static constexpr int kKps = NT <= 2 ? 2 : 1;  // k-blocks per stage
  static constexpr int kStages = NT == 1 ? 4 : NT == 2 ? 2 : 3;
  static constexpr int kStageBytes = kKps * (kABytes + NT * kBBytes);
  static constexpr int kBOff = kKps * kABytes;  // the activation blocks of a stage start after its weight blocks
  // After the stages: the split-K exchange region, receive buffers of a token group's partials from every CTA of
  // the cluster. One group needs one buffer (a tile's item is finished before the next tile is drained); several
  // groups alternate two, so that one group's exchange overlaps the previous group's reduce.
  static constexpr int kRecv = NT == 1 ? 1 : 2;
  static constexpr size_t kPartBytes = kRecv * (size_t)BM * BN * 4;
  // A fused attention head (kAttn) runs first in the last stage and the receive buffer: the producer fills that
  // stage only once the head is done.
  static_assert(!kAttn || NT == 1, "the layer's attention is fused only into one-group chains");
  static_assert(!kAttn || kStageBytes + kPartBytes >= attn::smem_bytes<128>(), "attention region");
  static constexpr int kTmemCols = kAcc * BN * NT;
  static constexpr int kTmemAlloc = kTmemCols <= 128 ? 128 : kTmemCols <= 256 ? 256 : 512;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kPartBytes + 256;
  // kind::f16 instruction descriptor: D fp32, A/B bf16, both K-major, N = 64 NT, M = 128.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)((BN * NT) >> 3) << 17) |
                                     ((uint32_t)(BM >> 4) << 24);
};

// ---------------------------------------------------------------------------------------------- tcgen05 PTX
MV_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
MV_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
MV_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
MV_DEV void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
MV_DEV void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
MV_DEV void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
MV_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Named barrier 2 over the epilogue warps (barrier 1 belongs to a fused attention's 128 threads).
MV_DEV void epi_bar() { asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory"); }
// OR of `v` over the epilogue threads (named barrier 2), the same answer in every thread.
MV_DEV bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

// Asynchronous 4-byte store into the shared memory of a CTA of the cluster (dst and mbar are shared::cluster
// addresses), counted on that CTA's mbarrier as complete_tx: the value is visible to whoever waits there, with no
// release fence on the storing side.
MV_DEV void st_async_f32(uint32_t dst, float v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst),
               "r"(__float_as_uint(v)), "r"(mbar)
               : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core groups 1024 bytes apart.
MV_DEV uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;             // leading-dimension offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride-dimension offset
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}

// ---------------------------------------------------------------------------------------------- epilogues
// Per-token RMSNorm scale from the sum-of-squares partials (one per 128-row slice of the hidden state).
// Per-CTA constants of the epilogue, loaded once (after the previous kernel finished) into shared memory:
// the per-token RMSNorm scale s[j] = 1/sqrt(sum of the sum-of-squares partials / norm_d + eps) (1 without a
// norm), and for the QKV epilogue the token positions prefix + depth. The 128 epilogue threads split the
// partial sums so the loads are independent and in flight together.
constexpr int kMaxSeq = kTokMax / BN;  // sequences of one pass (one token group each)
template <int NTOK>  // the launch's tokens: 64 per token group
struct EpiConst {
  float scale[NTOK];
  int pos[NTOK];
  float part[2][NTOK];
  int kv_row0[kMaxSeq];  // per sequence; -1: the cache rows would run past S_max (nothing is appended)
};

// i: epilogue thread 0 .. kEpiThreads - 1 (threads 128 and up only take part in the barriers)
template <class EC>
MV_DEV void load_epi_const(const GemmParams& p, EC* ec, int i, int ngroups) {
  const int half = (i >> 6) & 1;  // two threads per token, each summing half of the partials
  for (int g = 0; g < ngroups && i < 128; ++g) {
    const int j = g * BN + (i & (BN - 1));
    float t = 0.0f;
    if (p.ssq) {
      const int q0 = half * ((p.ssq_parts + 1) / 2), q1 = min(p.ssq_parts, q0 + (p.ssq_parts + 1) / 2);
      float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      int q = q0;
      for (; q + 8 <= q1; q += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] += __ldcg(p.ssq + (size_t)(q + u) * p.tok_ld + j);
      }
      for (; q < q1; ++q) acc[0] += __ldcg(p.ssq + (size_t)q * p.tok_ld + j);
      t = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    }
    ec->part[half][j] = t;
    if (half == 0 && p.pos_ids) {
      const int b = p.seq_rows ? j / BN : 0, r = p.seq_rows ? j % BN : j;  // sequences: one group each
      ec->pos[j] = (j < p.n_tok && (!p.seq_rows || r < p.seq_n)) ? p.cur_len[b] + p.pos_ids[r] : 0;
    }
  }
  if (i < kMaxSeq) {
    const int nseq = p.seq_rows ? (p.n_tok + p.seq_rows - 1) / p.seq_rows : 1;
    int r0 = -1;
    if (i < nseq) {
      r0 = p.cur_len ? p.cur_len[i] : 0;
      const int rows = p.seq_rows ? p.seq_n : p.n_tok;
      if (p.kv && (r0 < 0 || r0 + rows > p.S_max)) {  // appending would write past the cache planes
        mv_set_error_detail(p.err, 14, MV_DEVERR_INDEX, (uint32_t)r0);
        r0 = -1;
      }
    }
    ec->kv_row0[i] = r0;
  }
  epi_bar();
  for (int g = 0; g < ngroups && i < 128; ++g) {
    const int j = g * BN + (i & (BN - 1));
    if (half == 0)
      ec->scale[j] = p.ssq ? rsqrtf((ec->part[0][j] + ec->part[1][j]) / (float)p.norm_d + p.eps) : 1.0f;
  }
  epi_bar();
}

// ---- token-major epilogue: thread (warp w, lane l) owns rows 4l..4l+3 of the tile for tokens j = w + 4t
// (t = 0..15), so every global access of the epilogue is one 16-byte (fp32) or 8-byte (bf16) vector per lane and
// a warp covers one token's 128 contiguous rows. Partner rows (RoPE d +- D/2, SwiGLU gate/up) sit in lane l ^ k.
constexpr int kTokPerThread = BN / 4;
constexpr int kChunk = 4;  // tokens per thread finished at once

MV_DEV void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
MV_DEV float4 shfl_xor4(const float4& v, int m) {
  return make_float4(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m),
                     __shfl_xor_sync(0xffffffffu, v.z, m), __shfl_xor_sync(0xffffffffu, v.w, m));
}
MV_DEV uint2 pack_bf16x4(float a, float b, float c, float d) {
  const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
  const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(c)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(d)) << 16);
  return make_uint2(lo, hi);
}
// SiLU for a bf16 result: hardware exp2 and an approximate divide (relative error far below bf16's 2^-9).
MV_DEV float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
// sin and cos of a rotary angle (at most a few thousand radians): Cody-Waite reduction by 2*pi split into a float
// and its remainder, then the hardware sine/cosine on [-pi, pi] (absolute error about 1e-6, below bf16's step).
MV_DEV void rope_sincos(float a, float* s, float* c) {
  const float k = rintf(a * 0.159154943091895336f);  // 1 / (2 pi)
  float r = fmaf(-k, 6.28318548202514648f, a);       // float(2 pi)
  r = fmaf(-k, -1.74845553146951715e-7f, r);         // 2 pi - float(2 pi)
  __sincosf(r, s, c);
}

// This CTA's share of the tile: tokens j = w + 4t for t = r0, r0 + cs, ... (acc[u] holds t = r0 + u * cs, rows
// 4l..4l+3, summed over every K slice of the cluster). Writes the outputs of the launch's epilogue kind.
template <int EPI, int NU, class EC>
MV_DEV void final_epilogue(const GemmParams& p, int tile, int jb, int w, int l, int r0, int cs,
                           float4 (&acc)[NU], const EC* ec) {
  const int ntok = p.n_tok;
  if constexpr (EPI == EPI_STORE) {
    const int R = tile * BM + 4 * l;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.out_f32) & 15) == 0) && ((p.ld_out & 3) == 0) && R + 3 < p.M;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int t = r0 + u * cs;
      if (t >= kTokPerThread) break;
      const int j = jb + w + 4 * t;
      if (j >= ntok) continue;  // uniform over the warp (the shuffles below need every lane)
      const float s = ec->scale[j];
      const float4 v = make_float4(acc[u].x * s, acc[u].y * s, acc[u].z * s, acc[u].w * s);
      if (p.row_max) {  // the tile's max and first argmax for token j (the posterior's greedy statistics)
        float m = -FLT_MAX;
        int mi = 0x7fffffff;
        const float vq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (R + q < p.M && vq[q] > m) {
            m = vq[q];
            mi = R + q;
          }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, m, o);
          const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
          if (om > m || (om == m && oi < mi)) {
            m = om;
            mi = oi;
          }
        }
        if (l == 0) p.row_max[(size_t)tile * p.tok_ld + j] = make_float2(m, __int_as_float(mi));
      }
      if (R >= p.M) continue;
      float* o = p.out_f32 + (size_t)j * p.ld_out + R;
      if (vec) {
        *reinterpret_cast<float4*>(o) = v;
      } else {
        o[0] = v.x;
        if (R + 1 < p.M) o[1] = v.y;
        if (R + 2 < p.M) o[2] = v.z;
        if (R + 3 < p.M) o[3] = v.w;
      }
    }
  } else if constexpr (EPI == EPI_RESIDUAL) {
    // M is a multiple of 4 (host check): a lane's 4 rows are all valid or all past the end
    const int R = tile * BM + 4 * l;
    const bool valid = R < p.M;
    float4 xo[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {  // every residual load in flight before the first use
      const int t = r0 + u * cs;
      if (t >= kTokPerThread) break;
      const int j = jb + w + 4 * t;
      xo[u] = (valid && j < ntok) ? __ldcg(reinterpret_cast<const float4*>(p.x + (size_t)j * p.M + R))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int t = r0 + u * cs;
      if (t >= kTokPerThread) break;
      const int j = jb + w + 4 * t;
      if (j >= ntok) continue;  // uniform over the warp
      float4 xn = xo[u];
      add4(xn, acc[u]);
      float sq = 0.0f;
      if (valid) {
        *reinterpret_cast<float4*>(p.x + (size_t)j * p.M + R) = xn;
        *reinterpret_cast<uint2*>(p.xb + (size_t)j * p.M + R) = pack_bf16x4(xn.x, xn.y, xn.z, xn.w);
        sq = (xn.x * xn.x + xn.y * xn.y) + (xn.z * xn.z + xn.w * xn.w);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, m);
      if (l == 0) p.ssq_out[(size_t)tile * p.tok_ld + j] = sq;  // per-token sum of squares over the tile's rows
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // lanes 0..15: gate rows 4l..4l+3 (features f0 + 4l ..); lanes 16..31: the matching up rows
    const int f = tile * 64 + 4 * l;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int t = r0 + u * cs;
      if (t >= kTokPerThread) break;
      const int j = jb + w + 4 * t;
      if (j >= ntok) continue;  // uniform over the warp
      const float4 up = shfl_xor4(acc[u], 16);
      if (l < 16 && f < p.F) {
        const float s = ec->scale[j];
        const float4 g = acc[u];
        *reinterpret_cast<uint2*>(p.act + (size_t)j * p.F + f) =
            pack_bf16x4(silu_fast(g.x * s) * (up.x * s), silu_fast(g.y * s) * (up.y * s),
                        silu_fast(g.z * s) * (up.z * s), silu_fast(g.w * s) * (up.w * s));
      }
    }
  } else if constexpr (EPI == EPI_QKV) {
    // a tile holds whole heads (D divides 128); rows = [q heads | k heads | v heads] x D
    const int R = tile * BM + 4 * l;
    const bool valid = R < p.M;
    const int HD = p.H * p.D;
    const int half = p.D >> 1;
    // Row R's part (q, k or v), head and dimension. Divisions by run-time sizes cost a long dependent chain at
    // the tile's end, which a phase boundary waits for: with D and H D powers of two (every shape here) they are
    // shifts and masks, with the same results.
    int which, head, dim, dh;  // dh = dim mod D/2
    if (((p.D & (p.D - 1)) | (HD & (HD - 1))) == 0) {
      const int dsh = __ffs(p.D) - 1, hsh = __ffs(HD) - 1;
      which = R >> hsh;
      const int within = R & (HD - 1);
      head = within >> dsh;
      dim = within & (p.D - 1);
      dh = dim & (half - 1);
    } else {
      which = R / HD;
      const int within = R % HD;
      head = within / p.D;
      dim = within % p.D;
      dh = dim % half;
    }
    const bool lo = dim < half;
    // theta^(-2k/D) for the rotary pair index k = (dim + q) mod D/2 of each of the lane's 4 rows. dim is a multiple
    // of 4, so where D/2 is one too k = dim mod D/2 + q. -2 log2(theta) / D is exact for D a power of two, and the
    // exponent then takes one rounding as before: the frequencies are the same bits.
    const float c = -2.0f * p.log2_theta / (float)p.D;
    float inv_freq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) inv_freq[q] = exp2f(c * (float)((half & 3) ? (dim + q) % half : dh + q));
    // q: row j of q_out; k / v: row kv_row0[b] + r of sequence b's cache plane (j = b * seq_rows + r)
    const size_t plane = (size_t)p.layer * 2 + ((which == 1 || which == 2) ? which - 1 : 0);
    uint16_t* const kv_base = p.kv ? p.kv + (plane * p.H + head) * p.S_max * p.D + dim : nullptr;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int t = r0 + u * cs;
      if (t >= kTokPerThread) break;
      const int j = jb + w + 4 * t;
      if (j >= ntok) continue;  // uniform over the warp
      const float4 pr = shfl_xor4(acc[u], p.D >> 3);  // the RoPE partner rows (dim -+ D/2, same head)
      const int b = p.seq_rows ? j / BN : 0, r = p.seq_rows ? j % BN : j;  // sequences: one group each
      if (!valid || (p.seq_rows && r >= p.seq_n)) continue;  // past the weights, or a padding row
      uint16_t* dst;
      if (which == 0) {
        dst = p.q_out + (size_t)j * p.H * p.D + (size_t)head * p.D + dim;
      } else {
        if (ec->kv_row0[b] < 0) continue;
        dst = kv_base + (size_t)b * p.kv_seq_stride + (size_t)(ec->kv_row0[b] + r) * p.D;
      }
      const float s = ec->scale[j];
      float v[4] = {acc[u].x * s, acc[u].y * s, acc[u].z * s, acc[u].w * s};
      if (which < 2) {
        const float pv[4] = {pr.x * s, pr.y * s, pr.z * s, pr.w * s};
        const float pos = (float)ec->pos[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float sn, cs;
          rope_sincos(pos * inv_freq[q], &sn, &cs);
          v[q] = lo ? v[q] * cs - pv[q] * sn : v[q] * cs + pv[q] * sn;
        }
      }
      *reinterpret_cast<uint2*>(dst) = pack_bf16x4(v[0], v[1], v[2], v[3]);
    }
  }
}

struct ChainMaps {
  CUtensorMap a0[kGemmMaxPhases], a1[kGemmMaxPhases], b[kGemmMaxPhases], b2[kGemmMaxPhases];
  CUtensorMap kmap, vmap;  // fused attention: the KV cache planes
};
struct ChainArgs {
  GemmParams ph[kGemmMaxPhases];
  int epi[kGemmMaxPhases];
  int n_phases, csize;
  int indep;            // 1: the phases do not read each other's outputs (no counters, no waits)
  unsigned int* flags;  // [kGemmChainFlagWords]: phase-done counters, the exit counter, the attention counter
  attn::Args attn;      // fused attention (attn_D > 0) of the layer, before phase 0
  int attn_D;
};

// Cluster-wide steps of a fused attention head: only the epilogue warps of the C CTAs take part (the producer
// and MMA warps are busy streaming), so they meet on an mbarrier per step with one remote arrive per CTA.
struct EpiClusterSync {
  uint64_t* rbar;
  uint64_t* dbar;
  int C, i;
  unsigned int* err;
  MV_DEV void step(uint64_t* bar) {
    attn::grp_bar();  // this CTA's attention threads are done with their shared-memory writes / reads
    if (i < C) mbar_arrive_remote(map_rank(smem_u32(bar), (uint32_t)i));
    if (!mbar_wait_cluster(bar, 0u) && i == 0) mv_set_error(err, 16, MV_DEVERR_TIMEOUT);
  }
  bool stepped = false;  // the head took its first step (it has more than one working split)
  MV_DEV void ready() {
    step(rbar);
    stepped = true;
  }
  // The head's last step is taken by the chain itself, after the outputs are published (finish): until then this
  // CTA's partials stay in place, and only the producer's refill of the last stage, where they lie, waits for it.
  MV_DEV void done() {}
  MV_DEV void finish() {
    if (stepped) step(dbar);
  }
};

// *p += 1 with release semantics at GPU scope: every write this thread has made or observed (the other epilogue
// threads' stores, ordered before it by a CTA barrier) is visible to whoever acquires the new count.
MV_DEV void count_release(unsigned int* p) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}

// No thread of this kernel returns early, not even after a bounded wait expired: every CTA must reach the
// end, where the last one out resets the chain's phase counters. A CTA that left before would leave them
// non-zero, and the next launch's waits on them would pass at once and read activations that are not ready.
template <int NT, bool kAttn>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ ChainMaps maps,
                                                           const __grid_constant__ ChainArgs ca) {
  constexpr int kStages = Cfg<NT>::kStages;
  constexpr int kStageBytes = Cfg<NT>::kStageBytes;
  constexpr int kKps = Cfg<NT>::kKps;
  constexpr int kBOff = Cfg<NT>::kBOff;
  constexpr int kTmemAlloc = Cfg<NT>::kTmemAlloc;
  constexpr uint32_t kIdesc = Cfg<NT>::kIdesc;
  constexpr int kRecv = Cfg<NT>::kRecv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* part = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);  // [BN tokens][BM rows], a group
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[kAcc], tempty[kAcc], drain, pfull[2], rfree[2];
  // fused attention: its key/value ring, its cluster steps, and this CTA's head done (the last stage is free)
  __shared__ __align__(8) uint64_t afull[attn::kStages], aready, adone, alocal;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int s_abort;
  __shared__ EpiConst<BN * NT> s_ec;
  // the current phase's parameters and epilogue kind, copied once per phase: the epilogue of a phase's last tile
  // -- the step every phase boundary waits for -- then reads shared memory instead of the kernel parameters
  // through a runtime phase index
  __shared__ GemmParams s_par;
  __shared__ int s_epi;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = ca.csize;                  // CTAs per cluster = K slices per tile (a power of two)
  const int csh = __ffs(C) - 1;            // log2 C: divisions by C are shifts
  const int rank = (int)cluster_rank();    // this CTA's K slice and token share
  // in every phase cluster q owns the contiguous tiles [t0, t1) (adjacent in the packed weight layout)
  const int q = blockIdx.x / C, ncl = gridDim.x / C;
  auto tile_range = [&](const GemmParams& p, int& t0, int& t1) {
    t0 = (int)((long long)q * p.n_tiles / ncl);
    t1 = (int)((long long)(q + 1) * p.n_tiles / ncl);
  };
  unsigned int* err = ca.ph[0].err;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);  // this CTA's arrive with the expected bytes; the cluster's stores complete it
      mbar_init(&rfree[b], C);  // one arrive from every CTA of the cluster: it has consumed this CTA's slice
    }
    mbar_init(&drain, 1);
    for (int s = 0; s < attn::kStages; ++s) mbar_init(&afull[s], 1);
    mbar_init(&aready, C);  // one arrive from every CTA of the cluster per attention step
    mbar_init(&adone, C);
    mbar_init(&alocal, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers are initialised before the first remote arrive
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int ph = 0; ph < ca.n_phases; ++ph) {
        tma_prefetch_desc(&maps.a0[ph]);
        if (ca.ph[ph].paired) tma_prefetch_desc(&maps.a1[ph]);
        tma_prefetch_desc(&maps.b[ph]);
        if (ca.ph[ph].act_box) tma_prefetch_desc(&maps.b2[ph]);
      }
      int it = 0;
      bool ok = true, flag_timeout = false;
      const uint64_t wpol = l2_evict_first_policy();  // weights are read once per step
      for (int ph = 0; ok && ph < ca.n_phases; ++ph) {
        const GemmParams& p = ca.ph[ph];
        const CUtensorMap* am0 = &maps.a0[ph];
        const CUtensorMap* am1 = &maps.a1[ph];
        const CUtensorMap* bm = &maps.b[ph];
        int t0, t1;
        tile_range(p, t0, t1);
        const int kb0 = (rank * p.kbt) >> csh, kb1 = ((rank + 1) * p.kbt) >> csh;  // this CTA's K slice
        // The weights do not depend on anything: their loads run ahead. The activations are the previous
        // kernel's output (phase 0: wait for that grid) or the previous phase's (wait for its counter).
        bool waited = false;
        int pend_s[kStages], pend_kb[kStages], pend_n[kStages];
        int pend = 0;
        auto issue_b = [&](int stage, int kb, int nk) {  // the activation blocks of the NT token groups, nk k-blocks
          if (p.act_box == NT && nk == kKps) {  // every k-block and token group of the stage in one box
            tma_load_3d(stages + (size_t)stage * kStageBytes + kBOff, &maps.b2[ph], &full[stage], 0, 0, kb);
            return;
          }
          for (int u = 0; u < nk; ++u)
#pragma unroll
            for (int g = 0; g < NT; ++g)
              tma_load_2d(stages + (size_t)stage * kStageBytes + kBOff + (u * NT + g) * kBBytes, bm, &full[stage],
                          (kb + u) * BK, g * BN);
        };
        auto release = [&]() -> bool {  // on an expired wait the loads are still issued, so every barrier completes
          bool got = true;
          // Every activation load follows the previous kernel's completion, in any phase: a CTA may have no
          // tile in phase 0 (or the phases may be independent), and a chain that starts early under
          // programmatic launch would otherwise read the previous chain's counters and activations.
          pdl_wait();
          if (ph > 0 && !ca.indep) {
            got = wait_count(ca.flags + ph - 1, gridDim.x);
            flag_timeout |= !got;
            asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes -> TMA reads
          } else if (ph == 0 && ca.attn_D) {  // phase 0's activations are the fused attention's output
            got = wait_count(ca.flags + kGemmAttnFlag, gridDim.x);
            flag_timeout |= !got;
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          waited = true;
          for (int j = 0; j < pend; ++j) issue_b(pend_s[j], pend_kb[j], pend_n[j]);
          return got;
        };
        for (int tile = t0; ok && tile < t1; ++tile) {
          for (int kb = kb0; kb < kb1; kb += kKps, ++it) {
            const int s = it % kStages, r = it / kStages;
            const int nk = min(kKps, kb1 - kb);  // k-blocks of this stage (the last of a tile may hold fewer)
            if (s_abort || !mbar_wait(&empty[s], (uint32_t)((r & 1) ^ 1))) {
              ok = false;
              break;
            }
            // the last stage holds this CTA's attention head until it is done
            if (kAttn && ca.attn_D && it == kStages - 1 && !mbar_wait(&alocal, 0u)) {
              ok = false;
              break;
            }
            uint8_t* a = stages + (size_t)s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(nk * (kABytes + NT * kBBytes)));
            if (p.packed_a >= 2) {  // the stage's weights in one box, or one box per k-block
              const int tb = tile * p.kbt + kb;
              const CUtensorMap* m = nk == kKps ? am0 : am1;
              for (int u = 0; u < (nk == kKps ? 1 : nk); ++u) {
                if (p.packed_a == 3)
                  tma_load_4d_hint(a + u * kABytes, m, &full[s], 0, 0, 0, tb + u, wpol);
                else
                  tma_load_3d_hint(a + u * kABytes, m, &full[s], 0, 0, tb + u, wpol);
              }
            }
            for (int u = 0; u < nk && p.packed_a < 2; ++u) {
              uint8_t* au = a + u * kABytes;
              if (p.packed_a) {  // one contiguous block per matrix
                const int tb = tile * p.kbt + kb + u;
                tma_load_3d_hint(au, am0, &full[s], 0, 0, tb, wpol);
                if (p.paired) tma_load_3d_hint(au + kABytes / 2, am1, &full[s], 0, 0, tb, wpol);
              } else if (p.paired) {
                tma_load_2d_hint(au, am0, &full[s], (kb + u) * BK, tile * 64, wpol);
                tma_load_2d_hint(au + kABytes / 2, am1, &full[s], (kb + u) * BK, tile * 64, wpol);
              } else {
                tma_load_2d_hint(au, am0, &full[s], (kb + u) * BK, tile * BM, wpol);
              }
            }
            if (waited) {
              issue_b(s, kb, nk);
            } else {
              pend_s[pend] = s;
              pend_kb[pend] = kb;
              pend_n[pend] = nk;
              if (++pend == kStages && !release()) {
                ok = false;
                break;
              }
            }
          }
        }
        if (ok && !waited && pend > 0 && !release()) ok = false;
      }
      if (!ok) {
        if (!s_abort) mv_set_error(err, flag_timeout ? 12 : 8, MV_DEVERR_TIMEOUT);
        s_abort = 1;
        // let the copies in flight land: the most recent phase of each stage
        for (int j = max(0, it - kStages); j < it; ++j)
          if (!mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1))) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, n = 0;
      bool ok = true;
      const uint32_t st0 = smem_u32(stages);
      for (int ph = 0; ok && ph < ca.n_phases; ++ph) {
        const GemmParams& p = ca.ph[ph];
        int t0, t1;
        tile_range(p, t0, t1);
        const int kb0 = (rank * p.kbt) >> csh, kb1 = ((rank + 1) * p.kbt) >> csh;
        for (int tile = t0; ok && tile < t1; ++tile, ++n) {
          const int buf = n % kAcc, rr = n / kAcc;
          if (s_abort || !mbar_wait(&tempty[buf], (uint32_t)((rr & 1) ^ 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dt = tmem_base + (uint32_t)(buf * BN * NT);
          for (int kb = kb0; kb < kb1; kb += kKps, ++it) {
            const int s = it % kStages, r = it / kStages;
            const int nk = min(kKps, kb1 - kb);
            if (s_abort || !mbar_wait(&full[s], (uint32_t)(r & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a = st0 + (uint32_t)(s * kStageBytes);
            for (int u = 0; u < nk; ++u) {
              const uint64_t ad = sw128_desc(a + (uint32_t)(u * kABytes));
              const uint64_t bd = sw128_desc(a + (uint32_t)(kBOff + u * NT * kBBytes));
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma(dt, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), kIdesc,
                       (kb > kb0 || u > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(&empty[s]);
          }
          if (!ok) break;
          tc_commit(&tfull[buf]);
        }
      }
      if (!ok) {
        if (!s_abort) mv_set_error(err, 9, MV_DEVERR_TIMEOUT);
        s_abort = 1;
        tc_commit(&drain);  // arrives once every MMA issued so far has completed
        mbar_wait(&drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (kEpiWarps warps)
    // Pipelined over the tiles: iteration n first sums and finishes tile n-1 (its partials were published a
    // whole tile ago, and this runs while the MMA works on tile n), then drains tile n's accumulator from TMEM
    // into this CTA's partial buffer and signals the cluster. At a phase boundary the last tile of the phase is
    // finished, the phase is published (one count per CTA), and this phase's scales wait for every CTA.
    const int sub = warp & 3;                 // TMEM sub-partition this warp may read
    const int row = sub * 32 + lane;          // tile row = TMEM lane
    const int hw = (warp - 2) >> 2;           // which warp of the sub-partition's pair: half of the columns
    const int i = hw * 128 + row;             // epilogue thread 0 .. kEpiThreads - 1
    pdl_wait();                               // the epilogue reads what earlier kernels wrote
    if constexpr (kAttn) {
      if (ca.attn_D) {  // the layer's attention first: cluster q = head q, CTA rank = key split (128 threads)
        const bool head_here = q < ca.attn.H && hw == 0;
        EpiClusterSync sy{&aready, &adone, C, i, err};
        if (head_here) {
          // the last stage and the receive buffer: the producer leaves that stage empty until the head is done,
          // and no CTA stores partials before every head of the layer is done
          uint8_t* region = stages + (size_t)(kStages - 1) * kStageBytes;
          if (ca.attn_D == 128)
            attn::head<128>(ca.attn, &maps.kmap, &maps.vmap, region, afull, rank, q, 0, 0, i, sy);
          else
            attn::head<64>(ca.attn, &maps.kmap, &maps.vmap, region, afull, rank, q, 0, 0, i, sy);
        }
        epi_bar();  // this CTA's attention outputs are stored: publish them
        if (i == 0) count_release(ca.flags + kGemmAttnFlag);
        if (head_here) sy.finish();  // every CTA of the cluster has read this CTA's partials
        // the head's shared-memory accesses come before the bulk copies that refill the last stage
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_bar();
        if (i == 0) mbar_arrive(&alocal);
      }
    }
    // Split-K exchange of a token group ("item" m, receive buffer m % kRecv): token t of a group belongs to CTA t mod C
    // (slot t / C). Every CTA drains its partial accumulator from TMEM and stores each value straight into its
    // owner's receive buffer, slice [sender rank], with st.async counted on the owner's pfull[m % 2]. Each CTA then
    // sums the C slices of its own tokens from its own shared memory (rank order: deterministic) and runs the fused
    // epilogue on them. A sender may reuse a buffer once every owner has consumed the item kRecv before (rfree).
    const int U = kTokPerThread >> csh;  // token slots per owner
    const uint32_t slice_bytes = (uint32_t)(U * 4 * BM * 4);
    const uint32_t recv_s = smem_u32(part);  // [kRecv][C senders][U][4][BM] floats
    if (i == 0)  // items 0 .. kRecv - 1: C slices each
      for (int b = 0; b < kRecv; ++b) mbar_arrive_expect_tx(&pfull[b], (uint32_t)C * slice_bytes);
    bool ok = true;
    int n = 0, m = 0, prev_tile = -1, prev_ph = 0, published = 0;
    // token group g_r of the tile; nr: item number; publish_to: phases before it are finished in this CTA once this
    // item is (they are published right after its stores, ahead of releasing the receive buffer)
    auto finish = [&](int ph_r, int tile_r, int g_r, int nr, int publish_to) {
      const int rb = nr % kRecv;
      const bool all = mbar_wait_cluster(&pfull[rb], (uint32_t)((nr / kRecv) & 1));
      const float* recv = part + (size_t)rb * (C * U * 4 * BM);
      if (epi_any(!all)) {
        if (i == 0) mv_set_error(err, 11, MV_DEVERR_TIMEOUT);
        s_abort = 1;
        ok = false;
        return;
      }
      const GemmParams& pr = s_par;  // phase ph_r's (copied when the phase began in this CTA)
      const int epi = s_epi;
      // this CTA's token share t = rank, rank + C, ..., alternate ones to the two warps of a sub-partition
      // (t0 = rank + hw C, stride 2 C), in chunks of kChunk tokens per thread, each summed over the C partials of
      // the cluster in rank order (16-byte DSMEM loads); only the fused epilogue itself depends on the kind
      const int t0 = rank + hw * C, ts = 2 * C;
      for (int u0 = 0; t0 + u0 * ts < kTokPerThread; u0 += kChunk) {
        float4 acc[kChunk];
        if (C == 4) {
          // clusters of four: two tokens per thread, t0 and t0 + 8 (slots t0 / 4 and t0 / 4 + 2), all eight
          // partials loaded before any is added; the sums of tokens past n_tok are not used by any epilogue
          float4 pa[4], pb[4];
          const int sa = t0 >> 2, sb = (t0 + ts) >> 2;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            pa[c] = reinterpret_cast<const float4*>(recv + ((c * U + sa) * 4 + sub) * BM)[lane];
            pb[c] = reinterpret_cast<const float4*>(recv + ((c * U + sb) * 4 + sub) * BM)[lane];
          }
#pragma unroll
          for (int u = 0; u < kChunk; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            add4(acc[0], pa[c]);
            add4(acc[1], pb[c]);
          }
        }
#pragma unroll
        for (int u = 0; u < kChunk && C != 4; ++u) {
          acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          const int t = t0 + (u0 + u) * ts;
          if (t >= kTokPerThread) break;
          const int j = sub + 4 * t;  // token within the group
          if (g_r * BN + j >= pr.n_tok) continue;
          const int slot = t >> csh;  // this token's place in every sender's slice
          float4 part_c[kMaxCluster];
#pragma unroll
          for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) part_c[c] = reinterpret_cast<const float4*>(recv + ((c * U + slot) * 4 + sub) * BM)[lane];
#pragma unroll
          for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) add4(acc[u], part_c[c]);
        }
        const int r0 = t0 + u0 * ts;
        if (epi == EPI_RESIDUAL)
          final_epilogue<EPI_RESIDUAL, kChunk>(pr, tile_r, g_r * BN, sub, lane, r0, ts, acc, &s_ec);
        else if (epi == EPI_SWIGLU)
          final_epilogue<EPI_SWIGLU, kChunk>(pr, tile_r, g_r * BN, sub, lane, r0, ts, acc, &s_ec);
        else if (epi == EPI_QKV)
          final_epilogue<EPI_QKV, kChunk>(pr, tile_r, g_r * BN, sub, lane, r0, ts, acc, &s_ec);
        else
          final_epilogue<EPI_STORE, kChunk>(pr, tile_r, g_r * BN, sub, lane, r0, ts, acc, &s_ec);
      }
      // the partials were consumed above (stores issued from them): publish the phases this item completes (one
      // count per CTA and phase; the barrier orders every epilogue thread's stores before it), then release the
      // buffers to their owners, one release arrive per CTA of the cluster from C lanes at once
      epi_bar();
      if (publish_to > published) {
        if (i == 0)
          for (int k = published; k < publish_to; ++k) count_release(ca.flags + k);
        published = publish_to;
      }
      // arm this buffer for item nr + kRecv, then tell every sender its slice here may be overwritten
      if (i == 0) mbar_arrive_expect_tx(&pfull[rb], (uint32_t)C * slice_bytes);
      if (i < C) mbar_arrive_remote(map_rank(smem_u32(&rfree[rb]), (uint32_t)i));
    };
    // Drains token group g of TMEM accumulator buffer `buf` and stores it into the owners' receive buffers (item m).
    auto drain_push = [&](int buf, int g) -> bool {
      const int rb = m % kRecv;
      bool free_ok = true;
      if (m >= kRecv)  // item m - kRecv consumed
        free_ok = mbar_wait_cluster(&rfree[rb], (uint32_t)(((m / kRecv) - 1) & 1));
      if (epi_any(!free_ok)) {
        if (i == 0) mv_set_error(err, 10, MV_DEVERR_TIMEOUT);
        s_abort = 1;
        return false;
      }
      float v[BN / 2];  // this warp's half of the group's columns (tokens 32 hw .. 32 hw + 31)
      const uint32_t ta =
          tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(buf * BN * NT + g * BN + hw * (BN / 2));
      tmem_ld32(ta, v);
      tmem_ld_wait();
      if (g == NT - 1) {  // the whole accumulator buffer is read: the MMA may reuse it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      // token j = 32 hw + jj is token t = j / 4 of sub-partition j % 4, owned by CTA t % C at slot t / C
      const uint32_t mine = recv_s + (uint32_t)((rb * C + rank) * U * 4 * BM * 4);  // my slice in every owner
      const uint32_t bar = smem_u32(&pfull[rb]);
#pragma unroll
      for (int jj = 0; jj < BN / 2; ++jj) {
        const int j = hw * (BN / 2) + jj, t = j >> 2, c = t & (C - 1);
        const uint32_t off = (uint32_t)((((t >> csh) * 4 + (j & 3)) * BM + row) * 4);
        st_async_f32(map_rank(mine + off, (uint32_t)c), v[jj], map_rank(bar, (uint32_t)c));
      }
      ++m;
      return true;
    };
    // One loop over this CTA's tiles of every phase, so that each tile is finished at a single place in the code.
    const int NP = ca.n_phases;
    int ph = 0, t0 = 0, t1 = 0, tile = 0, ec_ph = -1;
    tile_range(ca.ph[0], t0, t1);
    tile = t0;
    while (true) {
      while (ph < NP && tile >= t1) {  // the next tile to drain: skip exhausted phases
        if (++ph < NP) {
          tile_range(ca.ph[ph], t0, t1);
          tile = t0;
        }
      }
      // every phase before `upto` is finished in this CTA once the previous tile is: publish them, in order
      const int upto = ca.indep ? 0 : (ph < NP ? ph : NP - 1);
      if (prev_tile >= 0) {
        finish(prev_ph, prev_tile, NT - 1, m - 1, upto);
        prev_tile = -1;
        if (!ok) break;
      }
      if (published < upto) {
        epi_bar();  // every output of those phases written by this CTA
        if (i == 0) {
          for (int k = published; k < upto; ++k) count_release(ca.flags + k);
        }
        published = upto;
      }
      if (ph >= NP) break;
      if (ec_ph != ph) {
        // this phase's scales are sums of squares the previous phase wrote: wait until every CTA finished it
        bool got = true;
        if (ph > 0 && !ca.indep && i == 0) got = wait_count(ca.flags + ph - 1, gridDim.x);
        if (epi_any(!got)) {
          if (i == 0) mv_set_error(err, 12, MV_DEVERR_TIMEOUT);
          s_abort = 1;
          ok = false;
          break;
        }
        load_epi_const(ca.ph[ph], &s_ec, i, NT);  // scales and positions: the same for every tile of the phase
        {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(&ca.ph[ph]);
          uint32_t* dst = reinterpret_cast<uint32_t*>(&s_par);
          for (int k = i; k < (int)(sizeof(GemmParams) / 4); k += kEpiThreads) dst[k] = src[k];
          if (i == 0) s_epi = ca.epi[ph];
        }
        ec_ph = ph;
      }
      const int buf = n % kAcc;
      const bool got = !s_abort && mbar_wait(&tfull[buf], (uint32_t)((n / kAcc) & 1));
      if (epi_any(!got)) {  // uniform over the epilogue warps
        if (i == 0) mv_set_error(err, 10, MV_DEVERR_TIMEOUT);
        s_abort = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      // The tile's token groups (item m = one group of one tile): group g is drained and pushed before group g - 1
      // is finished, so one item's exchange overlaps the other's reduce and epilogue; with several groups the two
      // receive buffers hold items g - 1 and g (drain_push waits until every owner has consumed item g - 2).
      // Across tiles the previous tile's last group is finished first (above): a phase's last item publishes the
      // phase, which the next tile's activations may wait for.
      for (int g = 0; g < NT; ++g) {
        if (!drain_push(buf, g)) {
          ok = false;
          break;
        }
        if (g > 0) {
          finish(ph, tile, g - 1, m - 2, published);
          if (!ok) break;
        }
      }
      if (!ok) break;
      prev_tile = tile;
      prev_ph = ph;
      ++tile;
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another CTA of its cluster may still read its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemAlloc);
  }
  // the last CTA out leaves the chain's counters at zero for the next launch
  if (threadIdx.x == 0 && ca.flags && (ca.n_phases > 1 || ca.attn_D) && !ca.indep) {
    __threadfence();
    if (atomicAdd(ca.flags + kGemmMaxPhases, 1u) == gridDim.x - 1) {
      for (int k = 0; k < kGemmChainFlagWords; ++k) ca.flags[k] = 0u;
      __threadfence();
    }
  }
}

}  // namespace


// Token groups of a launch over n_tok tokens: 1 to 4 (0 when n_tok > 256).
int token_groups(int n_tok) { return n_tok < 1 || n_tok > kTokMax ? 0 : (n_tok + BN - 1) / BN; }

// Kernel variants: v = nt - 1 for nt token groups (0..3), v = 4 for one group with the layer's attention fused.
constexpr int kVariants = 5;
int variant_of(int nt, bool attn) { return attn ? 4 : nt - 1; }
size_t smem_bytes_for(int v) {
  switch (v) {
    case 0: return Cfg<1>::kSmemBytes;
    case 1: return Cfg<2>::kSmemBytes;
    case 2: return Cfg<3>::kSmemBytes;
    case 3: return Cfg<4>::kSmemBytes;
    default: return Cfg<1, true>::kSmemBytes;
  }
}
const void* kernel_for(int v) {
  switch (v) {
    case 0: return (const void*)gemm_kernel<1, false>;
    case 1: return (const void*)gemm_kernel<2, false>;
    case 2: return (const void*)gemm_kernel<3, false>;
    case 3: return (const void*)gemm_kernel<4, false>;
    default: return (const void*)gemm_kernel<1, true>;
  }
}
// Raises the dynamic shared memory limit of a variant once per device.
bool set_smem_for(int v) {
  static int flags[kVariants][64] = {};
  return mv_set_smem_once(kernel_for(v), (int)smem_bytes_for(v), flags[v]);
}

bool gemm_weight_map(CUtensorMap* map, const void* w, int rows, int K, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {(uint32_t)BK, (uint32_t)box_rows};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_weight_map_packed(CUtensorMap* map, const void* w, int rows, int K, int tile_rows) {
  const uint64_t n_blocks = (uint64_t)((rows + tile_rows - 1) / tile_rows) * ((K + BK - 1) / BK);
  const uint64_t dims[3] = {(uint64_t)BK, (uint64_t)tile_rows, n_blocks};
  const uint64_t strides[2] = {(uint64_t)BK * 2, (uint64_t)tile_rows * BK * 2};
  const uint32_t box[3] = {(uint32_t)BK, (uint32_t)tile_rows, 1};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_weight_map_packed_depth(CUtensorMap* map, const void* w, int rows, int K, int tile_rows, int depth) {
  const uint64_t n_blocks = (uint64_t)((rows + tile_rows - 1) / tile_rows) * ((K + BK - 1) / BK);
  const uint64_t dims[3] = {(uint64_t)BK, (uint64_t)tile_rows, n_blocks};
  const uint64_t strides[2] = {(uint64_t)BK * 2, (uint64_t)tile_rows * BK * 2};
  const uint32_t box[3] = {(uint32_t)BK, (uint32_t)tile_rows, (uint32_t)depth};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_weight_map_paired(CUtensorMap* map, const void* gate, const void* up, int F, int K, int depth) {
  const uint64_t n_blocks = (uint64_t)((F + 63) / 64) * ((K + BK - 1) / BK);
  const uint64_t block_bytes = 64ull * BK * 2;  // one packed (64 rows x 64) block of a matrix
  const uintptr_t g = reinterpret_cast<uintptr_t>(gate), u = reinterpret_cast<uintptr_t>(up);
  if (u != g + n_blocks * block_bytes) return false;
  // dims: k within the block, row, matrix (gate, up), block; the box takes both matrices of `depth` blocks
  const uint64_t dims[4] = {(uint64_t)BK, 64, 2, n_blocks};
  const uint64_t strides[3] = {(uint64_t)BK * 2, n_blocks * block_bytes, block_bytes};
  const uint32_t box[4] = {(uint32_t)BK, 64, 2, (uint32_t)depth};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, gate, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

int gemm_stage_kblocks(int n_tok) { return token_groups(n_tok) <= 2 ? 2 : 1; }

bool gemm_act_map_strided(CUtensorMap* map, const void* x, int rows, int K, int ld) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)ld * 2};
  const uint32_t box[2] = {(uint32_t)BK, (uint32_t)BN};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_act_map_stage(CUtensorMap* map, const void* x, int rows, int K, int groups) {
  if (K % BK || groups < 1 || groups > kMaxGroups || rows < BN * groups) return false;
  const uint64_t dims[3] = {(uint64_t)BK, (uint64_t)rows, (uint64_t)(K / BK)};
  const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)BK * 2};
  const uint32_t box[3] = {(uint32_t)BK, (uint32_t)(BN * groups), (uint32_t)gemm_stage_kblocks(BN * groups)};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_act_map(CUtensorMap* map, const void* x, int rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {(uint32_t)BK, (uint32_t)BN};
  return mv_encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// Clusters of c CTAs (one CTA per SM) that can be resident at once on this device, c = 1..kMaxCluster; 0 when
// the size cannot be launched. Asked once per device and size.
int gemm_max_clusters(int c, int v) {
  static int cache[64][kVariants][kMaxCluster + 1];  // 0 = not asked yet, -1 = not launchable
  const int dev = mv_device();
  if (dev < 0 || dev >= 64 || c < 1 || c > kMaxCluster || v < 0 || v >= kVariants) return 0;
  int& slot = cache[dev][v][c];
  if (slot == 0) {
    int n = 0;
    if (set_smem_for(v)) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c * mv_sm_count());
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem_bytes_for(v);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = c;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel_for(v), &cfg);
      if (e != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    slot = n > 0 ? n : -1;
  }
  return slot > 0 ? slot : 0;
}

namespace {
void shape_params(GemmParams& p) {
  p.kbt = (p.K + BK - 1) / BK;
  p.n_tiles = p.paired ? (p.F + 63) / 64 : (p.M + BM - 1) / BM;
}
// One cluster shape for a chain: the cluster size c and count that minimise the summed largest per-CTA share
// of k-blocks, sum over phases of ceil(tiles / clusters) * ceil(kbt / c), with all clusters resident at once
// (ties: the smaller cluster). Every CTA is resident, which the counters between phases rely on.
void plan_chain(GemmParams* p, int n, int v, int* csize, int* ncl_out) {
  int max_tiles = 1, min_kbt = 1 << 30;
  for (int i = 0; i < n; ++i) {
    max_tiles = std::max(max_tiles, p[i].n_tiles);
    min_kbt = std::min(min_kbt, p[i].kbt);
  }
  long long best = -1;
  *csize = 1;
  *ncl_out = std::min(max_tiles, mv_sm_count());
  for (int c = 1; c <= kMaxCluster && c <= min_kbt; c *= 2) {  // powers of two: a group's 16 token slots split evenly
    const int mc = gemm_max_clusters(c, v);
    if (mc < 1) continue;
    const int ncl = std::min(mc, max_tiles);
    long long cost = 0;
    for (int i = 0; i < n; ++i) cost += (long long)((p[i].n_tiles + ncl - 1) / ncl) * ((p[i].kbt + c - 1) / c);
    if (best < 0 || cost < best) {
      best = cost;
      *csize = c;
      *ncl_out = ncl;
    }
  }
}
}  // namespace

void gemm_finish_params(GemmParams& p) {
  shape_params(p);
  plan_chain(&p, 1, variant_of(std::max(1, token_groups(p.n_tok)), false), &p.csize, &p.n_clusters);
  p.grid = p.csize * p.n_clusters;
}

mv_status launch_gemm_chain(GemmPhase* ph, int n, unsigned int* flags, cudaStream_t stream, bool independent,
                            const GemmAttn* attn) {
  if (n < 1 || n > kGemmMaxPhases || (n > 1 && !independent && !flags)) return MV_ERR_INVALID_ARG;
  if (attn && (independent || !flags)) return MV_ERR_INVALID_ARG;
  ChainMaps maps;
  ChainArgs ca;
  memset(&maps, 0, sizeof(maps));
  memset(&ca, 0, sizeof(ca));
  GemmParams ps[kGemmMaxPhases];
  int max_tok = 1;
  for (int i = 0; i < n; ++i) {
    ps[i] = ph[i].p;
    shape_params(ps[i]);
    if (ps[i].n_tiles > kGemmMaxTiles || ps[i].n_tok < 1 || ps[i].n_tok > kTokMax) return MV_ERR_SHAPE;
    if (ps[i].seq_rows && (ps[i].seq_rows != BN || ps[i].seq_n < 1 || ps[i].seq_n > BN)) return MV_ERR_SHAPE;
    if (ph[i].epi < EPI_STORE || ph[i].epi > EPI_QKV) return MV_ERR_INVALID_ARG;
    max_tok = std::max(max_tok, ps[i].n_tok);
  }
  const int nt = token_groups(max_tok);
  for (int i = 0; i < n; ++i) {
    if (ps[i].tok_ld == 0) ps[i].tok_ld = BN * nt;
    if (ps[i].tok_ld < ps[i].n_tok) return MV_ERR_SHAPE;
  }
  const int v = variant_of(nt, attn != nullptr && nt == 1);
  int csize = 1, ncl = 1;
  plan_chain(ps, n, v, &csize, &ncl);
  if (attn && (nt != 1 || csize > attn::kMaxSplits || ncl < attn->args.H || (attn->D != 64 && attn->D != 128) ||
               attn->args.n > attn::kRows || attn->args.seq_rows != 0))
    return MV_ERR_UNSUPPORTED;
  for (int i = 0; i < n; ++i) {
    ps[i].csize = csize;
    ps[i].n_clusters = ncl;
    ps[i].grid = csize * ncl;
    ph[i].p = ps[i];
    ca.ph[i] = ps[i];
    ca.epi[i] = ph[i].epi;
    maps.a0[i] = ph[i].a0;
    maps.a1[i] = ph[i].a1;
    maps.b[i] = ph[i].b;
    if (ps[i].act_box) {
      if (ps[i].act_box != nt || (ps[i].K % BK) != 0) {
        ps[i].act_box = 0;  // a map for another number of token groups, or a ragged last k-block: one box per block
        ca.ph[i].act_box = 0;
        ph[i].p.act_box = 0;
      } else {
        maps.b2[i] = ph[i].b2;
      }
    }
  }
  ca.n_phases = n;
  ca.csize = csize;
  if (attn) {
    ca.attn = attn->args;
    ca.attn.splits = csize;
    ca.attn_D = attn->D;
    maps.kmap = attn->kmap;
    maps.vmap = attn->vmap;
  }
  ca.indep = independent ? 1 : 0;
  ca.flags = independent ? nullptr : flags;
  if (!set_smem_for(v)) return MV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * ncl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(v);
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = csize;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = mv_pdl_enabled() ? 2 : 1;
  cudaError_t e;
  switch (v) {
    case 0: e = cudaLaunchKernelEx(&cfg, gemm_kernel<1, false>, maps, ca); break;
    case 1: e = cudaLaunchKernelEx(&cfg, gemm_kernel<2, false>, maps, ca); break;
    case 2: e = cudaLaunchKernelEx(&cfg, gemm_kernel<3, false>, maps, ca); break;
    case 3: e = cudaLaunchKernelEx(&cfg, gemm_kernel<4, false>, maps, ca); break;
    default: e = cudaLaunchKernelEx(&cfg, gemm_kernel<1, true>, maps, ca); break;
  }
  if (e != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("gemm");
}

mv_status launch_gemm(int epi, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                      const GemmParams& p, cudaStream_t stream) {
  GemmPhase ph;
  ph.epi = epi;
  ph.a0 = a0;
  ph.a1 = a1;
  ph.b = b;
  ph.p = p;
  return launch_gemm_chain(&ph, 1, nullptr, stream);
}

// out[n][ld] (fp32) = X[n][K] . W[M][K]^T, optionally scaled per row of X by 1/sqrt(mean(x^2)+eps) of x_f32.
extern "C" mv_status mv_linear_bf16(const mv_bf16* w, const mv_bf16* x, float* out, int32_t M, int32_t K,
                                    int32_t n, int32_t ld_out, void* workspace, size_t ws_bytes, mv_stream stream) {
  (void)workspace;  // reserved: the kernel needs no global scratch
  (void)ws_bytes;
  if (!w || !x || !out) return MV_ERR_INVALID_ARG;
  if (M < 1 || K < 8 || (K & 7) || n < 1 || n > kTokMax || ld_out < M) return MV_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(x)) & 15) return MV_ERR_SHAPE;
  CUtensorMap a, b;
  if (!gemm_weight_map(&a, w, M, K, BM) || !gemm_act_map(&b, x, n, K)) return MV_ERR_CUDA;
  GemmParams p{};
  p.M = M;
  p.K = K;
  p.n_tok = n;
  p.out_f32 = out;
  p.ld_out = ld_out;
  p.err = mv_error_word();
  gemm_finish_params(p);
  return launch_gemm(EPI_STORE, a, a, b, p, static_cast<cudaStream_t>(stream));
}

// The same projection with w in the packed layout (mv_pack_weight with tile_rows = 128).
extern "C" mv_status mv_linear_bf16_packed(const mv_bf16* w_packed, const mv_bf16* x, float* out, int32_t M,
                                           int32_t K, int32_t n, int32_t ld_out, void* workspace, size_t ws_bytes,
                                           mv_stream stream) {
  (void)workspace;  // reserved: the kernel needs no global scratch
  (void)ws_bytes;
  if (!w_packed || !x || !out) return MV_ERR_INVALID_ARG;
  if (M < 1 || K < 8 || (K & 7) || n < 1 || n > kTokMax || ld_out < M) return MV_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(w_packed) | reinterpret_cast<uintptr_t>(x)) & 15) return MV_ERR_SHAPE;
  CUtensorMap a0, a, b;
  if (!gemm_weight_map_packed_depth(&a0, w_packed, M, K, BM, gemm_stage_kblocks(n)) ||
      !gemm_weight_map_packed(&a, w_packed, M, K, BM) || !gemm_act_map(&b, x, n, K))
    return MV_ERR_CUDA;
  GemmParams p{};
  p.M = M;
  p.K = K;
  p.n_tok = n;
  p.packed_a = 2;
  p.out_f32 = out;
  p.ld_out = ld_out;
  p.err = mv_error_word();
  gemm_finish_params(p);
  return launch_gemm(EPI_STORE, a0, a, b, p, static_cast<cudaStream_t>(stream));
}

extern "C" mv_status mv_linear_bf16_workspace(size_t* bytes) {
  if (!bytes) return MV_ERR_INVALID_ARG;
  *bytes = 0;  // reserved
  return MV_OK;
}
