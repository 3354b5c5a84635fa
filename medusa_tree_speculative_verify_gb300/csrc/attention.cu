// Tree attention: every tree node attends to the whole cached prefix and to its own root-to-node path.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.2 Tree attention and 二.5 tree_decoding(): the tree is
// flattened into a sequence after the prefix; the mask lets node i see only its ancestors and itself
// ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 4️⃣: siblings never see each other). The mask is
// MV_MASK_WORDS 64-bit ancestor words per node; only the key tiles that hold the tree block consult it. Trees
// of more than 64 nodes run as blocks of 64 query rows (grid z); block b needs only the tree keys up to its
// last row, since a node's ancestors precede it.
//
// Layout: q [n][H][D] bf16, K/V caches as planes of [H][S_max][D] bf16. One thread-block cluster per head;
// its CTAs split the head's 64-key tiles (split-KV, so that H x splits fills the GPU at batch 1). 4 warps per
// CTA, each owning 16 of the (up to) 64 tree queries. KV tiles arrive by TMA (128-byte swizzle, 2-stage mbarrier
// ring); Q.K^T and P.V run on the tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate); the softmax is an
// online (running max / sum) softmax in registers. Each CTA leaves its partial (max, sum, output) in its own
// shared memory and, after a cluster barrier, merges a slice of the query rows by reading the partials of the
// whole cluster over distributed shared memory (in rank order, so the result is deterministic).
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 64;   // keys per tile
constexpr int kRows = 64;   // query rows per CTA (tree nodes, padded)
constexpr int kStages = 2;  // 80 KB of shared memory at D = 128: two CTAs share an SM
constexpr int kMinTiles = 2;       // key tiles per split at the longest prefix, at least (sets the cluster size)
constexpr int kTilesPerSplit = 1;  // key tiles per working split at the actual prefix (measured best)
// CTAs per cluster. Measured on GB300: with clusters of 8 (two 81 KB CTAs per SM) a few clusters of a 32-head
// launch only start when others leave (a second wave, +11 us at short prefixes), although the occupancy query
// reports room for all; clusters of 4 start together.
constexpr int kMaxSplits = 4;

MV_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MV_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MV_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a [64 rows][D] bf16 tile. D >= 64: sub-tiles of 64 columns,
// 128-byte rows, 16-byte chunks XOR-swizzled by (row % 8) (the TMA 128B pattern). D < 64: plain rows.
template <int D>
MV_DEV uint32_t tile_off(int r, int c) {
  if constexpr (D >= 64) {
    return (uint32_t)((c >> 3) * (64 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  } else {
    return (uint32_t)(r * (D * 2) + c * 16);
  }
}

// Visibility of the 64 keys key0 .. key0 + 63 for one query row, as bits: keys before the tree block (s < 0
// positions) are all visible, tree key tj = key0 + k - P is visible iff bit tj of the row's ancestor words
// w0..w3 (nodes 0-63, 64-127, 128-191, 192-255) is set; s = key0 - P < 256. Bits past the tree are 0 (a node's
// ancestors precede it).
MV_DEV uint64_t tile_bits(uint64_t w0, uint64_t w1, uint64_t w2, uint64_t w3, int s) {
  if (s <= -64) return ~0ull;
  if (s < 0) return (w0 << -s) | ((1ull << -s) - 1ull);
  const int k = s >> 6, b = s & 63;
  const uint64_t lo = k == 0 ? w0 : k == 1 ? w1 : k == 2 ? w2 : w3;
  const uint64_t hi = k == 0 ? w1 : k == 1 ? w2 : k == 2 ? w3 : 0ull;
  return b == 0 ? lo : (lo >> b) | (hi << (64 - b));
}

struct AttnArgs {
  const uint16_t* q;        // [n][H][D]
  uint16_t* out;            // [n][H][D]
  const uint64_t* anc;      // [n][MV_MASK_WORDS]
  const int32_t* d_prefix;  // device prefix length (one per sequence when seq_rows > 0) or null
  int prefix;               // used when d_prefix is null
  int H, S_max, n, splits, plane_k, plane_v;  // splits = CTAs per cluster (gridDim.x)
  // Several sequences (grid z = sequence): sequence b's queries are rows b * seq_rows + 0 .. n - 1, its cache
  // planes plane_k / plane_v + b * seq_planes, its prefix d_prefix[b]. seq_rows = 0: grid z = blocks of 64 rows
  // of one tree.
  int seq_rows, seq_planes;
  float scale_log2;         // scale * log2(e)
  unsigned int* err;
};

template <int D>
__global__ void __launch_bounds__(kThreads) tree_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap,
                                                             const AttnArgs a) {
  constexpr int kTileBytes = kKeys * D * 2;
  constexpr int kBoxCols = D >= 64 ? 64 : D;
  constexpr int kBoxes = D / kBoxCols;
  constexpr int KS = D / 16;  // k-steps over the head dim
  constexpr int DN = D / 8;   // n-tiles over the head dim
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;                                  // [64][D]
  uint8_t* sk = smem + kTileBytes;                     // kStages x [64][D]
  uint8_t* sv = sk + kStages * kTileBytes;             // kStages x [64][D]
  __shared__ __align__(8) uint64_t full[kStages];
  constexpr int kPo = D + 4;  // row pitch (floats) of the partial output in shared memory

  const int split = blockIdx.x, h = blockIdx.y;  // split = rank in the head's cluster
  const int seq = a.seq_rows ? (int)blockIdx.z : 0;
  // this CTA's query rows: q / out rows qrow0 .. qrow0 + 63, tree nodes row0 .. row0 + 63
  const int row0 = a.seq_rows ? 0 : (int)blockIdx.z * kRows;
  const int qrow0 = a.seq_rows ? seq * a.seq_rows : row0;
  const int plane_k = a.plane_k + seq * a.seq_planes, plane_v = a.plane_v + seq * a.seq_planes;
  const int C = a.splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  pdl_trigger();
  pdl_wait();  // q, the cache and the prefix length come from earlier kernels
  const int P = a.d_prefix ? a.d_prefix[seq] : a.prefix;
  const int n_all = a.n;
  if (P < 0 || P + n_all > a.S_max) {
    if (tid == 0) mv_set_error(a.err, 4, MV_DEVERR_INDEX);
    return;
  }
  const int n = min(kRows, n_all - row0);         // query rows of this block
  const int n_keys = min(n_all, row0 + kRows);    // tree keys any of them can see
  const int total_tiles = (P + n_keys + kKeys - 1) / kKeys;
  // The cluster is sized for the longest prefix. At this prefix only S splits get tiles, about kTilesPerSplit
  // each (a split costs a merge). With S = 1 the first CTA does the whole head and writes it directly; the
  // others leave at once (no cluster barrier is used then). With S > 1 the idle splits still take part in the
  // barriers but contribute nothing to the merge.
  const int S = max(1, min(C, (total_tiles + kTilesPerSplit - 1) / kTilesPerSplit));
  if (S == 1 && split > 0) return;
  const int t_begin = split < S ? (int)((long long)split * total_tiles / S) : 0;
  const int t_end = split < S ? (int)((long long)(split + 1) * total_tiles / S) : 0;
  const int count = t_end - t_begin;

  auto issue = [&](int i) {  // tile t_begin + i into stage i % kStages
    const int st = i % kStages, key0 = (t_begin + i) * kKeys;
    mbar_arrive_expect_tx(&full[st], 2 * kTileBytes);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) {
      tma_load_4d(sk + st * kTileBytes + b * (kKeys * kBoxCols * 2), &kmap, &full[st], b * kBoxCols, key0, h,
                  plane_k);
      tma_load_4d(sv + st * kTileBytes + b * (kKeys * kBoxCols * 2), &vmap, &full[st], b * kBoxCols, key0, h,
                  plane_v);
    }
  };
  // the first key/value tiles are requested before Q is loaded, so the two latencies overlap
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    for (int i = 0; i < kStages && i < count; ++i) issue(i);
  }
  // Q: plain 16-byte loads into the tile layout (rows >= n are zero)
  for (int e = tid; e < kRows * (D / 8); e += kThreads) {
    const int r = e / (D / 8), c = e % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < n) v = *reinterpret_cast<const uint4*>(a.q + ((size_t)(qrow0 + r) * a.H + h) * D + c * 8);
    *reinterpret_cast<uint4*>(sq + tile_off<D>(r, c)) = v;
  }
  __syncthreads();

  // Q fragments for this warp's 16 rows
  uint32_t qa[KS][4];
  const uint32_t sq_base = smem_u32(sq);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int m = lane >> 3;
    const int r = warp * 16 + 8 * (m & 1) + (lane & 7);
    ldsm_x4(sq_base + tile_off<D>(r, 2 * ks + (m >> 1)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
  }
  const int q0 = warp * 16 + g, q1 = q0 + 8;  // rows within the block
  static_assert(MV_MASK_WORDS == 4, "four ancestor words per node");
  const uint64_t* ar0 = a.anc + (size_t)(row0 + q0) * MV_MASK_WORDS;
  const uint64_t* ar1 = a.anc + (size_t)(row0 + q1) * MV_MASK_WORDS;
  const uint64_t a00 = q0 < n ? ar0[0] : 0ull, a01 = q0 < n ? ar0[1] : 0ull, a02 = q0 < n ? ar0[2] : 0ull,
                 a03 = q0 < n ? ar0[3] : 0ull;
  const uint64_t a10 = q1 < n ? ar1[0] : 0ull, a11 = q1 < n ? ar1[1] : 0ull, a12 = q1 < n ? ar1[2] : 0ull,
                 a13 = q1 < n ? ar1[3] : 0ull;

  float o[DN][4];
#pragma unroll
  for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  bool ok = true;
  int stop = 0;  // first tile not consumed (set when a wait expires)

  for (int i = 0; i < count; ++i) {
    const int st = i % kStages;
    const bool got = mbar_wait(&full[st], (uint32_t)((i / kStages) & 1));
    if (__syncthreads_or(!got)) {
      if (tid == 0) mv_set_error(a.err, 4, MV_DEVERR_TIMEOUT);
      ok = false;
      stop = i;
      break;
    }
    const uint32_t kb = smem_u32(sk + st * kTileBytes), vb = smem_u32(sv + st * kTileBytes);
    const int key0 = (t_begin + i) * kKeys;
    // S = Q K^T for 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // pairs of 8-key n-tiles
        const int m = lane >> 3;
        const int key = 16 * np + 8 * (m >> 1) + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + tile_off<D>(key, 2 * ks + (m & 1)), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }
    // mask + running max
    const uint64_t tb0 = tile_bits(a00, a01, a02, a03, key0 - P), tb1 = tile_bits(a10, a11, a12, a13, key0 - P);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 8 * nt + 2 * t4 + e;
        const bool v0 = (tb0 >> k) & 1ull;
        const bool v1 = (tb1 >> k) & 1ull;
        s[nt][e] = v0 ? s[nt][e] * a.scale_log2 : -INFINITY;
        s[nt][2 + e] = v1 ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
    const float base0 = nm0 == -INFINITY ? 0.0f : nm0, base1 = nm1 == -INFINITY ? 0.0f : nm1;
    const float c0 = exp2f(m0 - base0), c1 = exp2f(m1 - base1);
    m0 = nm0;
    m1 = nm1;
    float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base0);
      s[nt][1] = exp2f(s[nt][1] - base0);
      s[nt][2] = exp2f(s[nt][2] - base1);
      s[nt][3] = exp2f(s[nt][3] - base1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * c0 + rs0;
    l1 = l1 * c1 + rs1;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      o[dn][0] *= c0;
      o[dn][1] *= c0;
      o[dn][2] *= c1;
      o[dn][3] *= c1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t p0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t p1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t p2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t p3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < DN / 2; ++dp) {
        const int m = lane >> 3;
        const int key = 16 * kk + 8 * (m & 1) + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + tile_off<D>(key, 2 * dp + (m >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], p0, p1, p2, p3, b0, b1);
        mma_bf16(o[2 * dp + 1], p0, p1, p2, p3, b2, b3);
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (tid == 0 && i + kStages < count) issue(i + kStages);
  }
  if (!ok) {
    // Let the copies already issued land before the pipeline buffers are reused below: tiles [stop, issued)
    // are in flight, each on its stage's barrier at its own phase. Every wait here is bounded too.
    if (tid == 0) {
      const int issued = min(count, stop + kStages);
      for (int j = stop; j < issued; ++j)
        if (!mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1))) break;
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if (S == 1) {  // one split for the head (a short prefix): normalise and write, nothing to merge
    const float i0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, i1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      const int col = 8 * dn + 2 * t4;
      if (q0 < n)
        *reinterpret_cast<uint32_t*>(a.out + ((size_t)(qrow0 + q0) * a.H + h) * D + col) =
            pack_bf16x2(o[dn][0] * i0, o[dn][1] * i0);
      if (q1 < n)
        *reinterpret_cast<uint32_t*>(a.out + ((size_t)(qrow0 + q1) * a.H + h) * D + col) =
            pack_bf16x2(o[dn][2] * i1, o[dn][3] * i1);
    }
    return;
  }

  // ---- this CTA's partial (unnormalised output, running max, sum) into its own shared memory; the CTAs of
  // the cluster (the key splits of this head) then merge it over distributed shared memory, each CTA a slice
  // of the query rows. The pipeline buffers are free once every warp has left the loop.
  __syncthreads();
  float* po = reinterpret_cast<float*>(smem);  // [64][D + 4] (padded rows: conflict-free float2 stores)
  float* pml = po + kRows * kPo;               // [64][2] running max (log2 domain) and sum
  float* pw = pml + kRows * 2;                 // [64][kMaxSplits] merge weights of this CTA's rows
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) {
    const int col = 8 * dn + 2 * t4;
    *reinterpret_cast<float2*>(po + q0 * kPo + col) = make_float2(o[dn][0], o[dn][1]);
    *reinterpret_cast<float2*>(po + q1 * kPo + col) = make_float2(o[dn][2], o[dn][3]);
  }
  if (t4 == 0) {
    pml[q0 * 2 + 0] = m0;
    pml[q0 * 2 + 1] = l0;
    pml[q1 * 2 + 0] = m1;
    pml[q1 * 2 + 1] = l1;
  }
  cluster_sync_all();  // every partial of the head is in place
  const int r0 = split * n / C, r1 = (split + 1) * n / C;  // this CTA's query rows
  const uint32_t ml_s = smem_u32(pml), po_s = smem_u32(po);
  if (tid < r1 - r0) {
    // w_s = 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s' for the row's S splits (rank order)
    const int q = r0 + tid;
    float m[kMaxSplits], l[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      m[s] = -INFINITY;
      l[s] = 0.0f;
      if (s < S) {
        const float2 v = ld_cluster_f2(map_rank(ml_s + (uint32_t)(q * 8), (uint32_t)s));
        m[s] = v.x;
        l[s] = v.y;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) M = fmaxf(M, m[s]);
    const float base = M == -INFINITY ? 0.0f : M;
    float L = 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      m[s] = s < S ? exp2f(m[s] - base) : 0.0f;
      L += m[s] * l[s];
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) pw[tid * kMaxSplits + s] = m[s] * inv;
  }
  __syncthreads();
  for (int e = tid; e < (r1 - r0) * (D / 4); e += kThreads) {
    const int rq = e / (D / 4), c4 = (e % (D / 4)) * 4, q = r0 + rq;
    const uint32_t off = po_s + (uint32_t)((q * kPo + c4) * 4);
    float4 v[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
      if (s < S) v[s] = ld_cluster_f4(map_rank(off, (uint32_t)s));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      if (s < S) {
        const float w = pw[rq * kMaxSplits + s];
        acc.x += w * v[s].x;
        acc.y += w * v[s].y;
        acc.z += w * v[s].z;
        acc.w += w * v[s].w;
      }
    }
    uint2 pk;
    pk.x = pack_bf16x2(acc.x, acc.y);
    pk.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(a.out + ((size_t)(qrow0 + q) * a.H + h) * D + c4) = pk;
  }
  cluster_sync_all();  // no CTA leaves while another may still read its partial
}

// Key splits per head (= CTAs per cluster): enough that each split has about kMinTiles key tiles at the
// longest prefix this launch may see, at most kMaxSplits.
int choose_splits(int max_tiles) {
  return std::max(1, std::min(kMaxSplits, (max_tiles + kMinTiles - 1) / kMinTiles));
}

size_t smem_bytes(int D);

// Clusters of c CTAs of tree_attn_kernel<D> that can be resident at once (asked once per device, D and c).
int max_active_clusters(int D, int c) {
  static int cache[64][4][kMaxSplits + 1];  // 0 = not asked yet, -1 = none
  const int dev = mv_device();
  const int di = D == 16 ? 0 : D == 32 ? 1 : D == 64 ? 2 : 3;
  if (dev < 0 || dev >= 64 || c < 1 || c > kMaxSplits) return 0;
  int& slot = cache[dev][di][c];
  if (slot == 0) {
    const size_t smem = smem_bytes(D);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1024);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = c;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (D) {
#define MV_ATTN_OCC(DD)                                                                                \
  case DD: {                                                                                         \
    static int flags[64] = {0};                                                                      \
    if (mv_set_smem_once((const void*)tree_attn_kernel<DD>, (int)smem, flags))                       \
      e = cudaOccupancyMaxActiveClusters(&n, tree_attn_kernel<DD>, &cfg);                            \
    break;                                                                                           \
  }
      MV_ATTN_OCC(16)
      MV_ATTN_OCC(32)
      MV_ATTN_OCC(64)
      MV_ATTN_OCC(128)
#undef MV_ATTN_OCC
      default:
        break;
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    slot = n > 0 ? n : -1;
  }
  return slot > 0 ? slot : 0;
}

size_t smem_bytes(int D) {
  const size_t pipeline = (size_t)(1 + 2 * kStages) * kKeys * D * 2;
  const size_t merge = ((size_t)kRows * (D + 4) + kRows * 2 + kRows * kMaxSplits) * sizeof(float);
  return 1024 + (pipeline > merge ? pipeline : merge);
}

}  // namespace

size_t tree_attn_ws_bytes(int H, int D, int S_max, int n_nodes) {
  (void)H, (void)D, (void)S_max, (void)n_nodes;
  return 256;  // reserved: the split partials are merged on chip
}

bool tree_attn_make_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* k_cache, const void* v_cache, int H,
                         int D, int S_max, int planes, size_t plane_stride_bytes) {
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)S_max, (uint64_t)H, (uint64_t)planes};
  const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)S_max * D * 2, (uint64_t)plane_stride_bytes};
  const uint32_t box[4] = {(uint32_t)(D >= 64 ? 64 : D), (uint32_t)kKeys, 1, 1};
  const CUtensorMapSwizzle sw = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return mv_encode_tmap(kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k_cache, dims, strides, box, sw) &&
         mv_encode_tmap(vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v_cache, dims, strides, box, sw);
}

mv_status launch_tree_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                int max_prefix, const mv_tree* t, float scale, mv_bf16* out, void* ws,
                                cudaStream_t stream) {
  return launch_tree_attention_n(kmap, vmap, plane_k, plane_v, q, H, D, S_max, d_prefix, prefix, max_prefix, t,
                                 t->n_nodes, scale, out, ws, stream);
}

mv_status launch_tree_attention_n(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                  const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                  int max_prefix, const mv_tree* t, int n, float scale, mv_bf16* out, void* ws,
                                  cudaStream_t stream, int nseq, int seq_planes) {
  (void)ws;  // reserved
  if (n < 1 || n > MV_MAX_NODES || nseq < 1 || (nseq > 1 && (n > kRows || !d_prefix))) return MV_ERR_SHAPE;
  // blocks of 64 query rows of one tree, or one block per sequence
  const int blocks = nseq > 1 ? nseq : (n + kRows - 1) / kRows;
  const int max_tiles = (max_prefix + n + kKeys - 1) / kKeys;
  int splits = choose_splits(max_tiles);
  // all H x blocks clusters resident at once: a cluster that has to wait for another to leave costs a whole
  // second wave
  while (splits > 1 && max_active_clusters(D, splits) < H * blocks) --splits;
  AttnArgs a{};
  a.q = q;
  a.out = out;
  a.anc = t->d_ancestors;
  a.d_prefix = d_prefix;
  a.prefix = prefix;
  a.H = H;
  a.S_max = S_max;
  a.n = n;
  a.splits = splits;
  a.plane_k = plane_k;
  a.plane_v = plane_v;
  a.seq_rows = nseq > 1 ? kRows : 0;
  a.seq_planes = seq_planes;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = mv_error_word();
  const size_t smem = smem_bytes(D);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, H, blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;  // one cluster = the key splits of one head
  at[0].val.clusterDim.x = splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = mv_pdl_enabled() ? 2 : 1;
  cudaError_t e;
  switch (D) {
#define MV_ATTN_CASE(DD)                                                                               \
  case DD: {                                                                                         \
    static int flags[64] = {0};                                                                      \
    if (!mv_set_smem_once((const void*)tree_attn_kernel<DD>, (int)smem, flags)) return MV_ERR_CUDA;  \
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<DD>, kmap, vmap, a);                               \
    break;                                                                                           \
  }
    MV_ATTN_CASE(16)
    MV_ATTN_CASE(32)
    MV_ATTN_CASE(64)
    MV_ATTN_CASE(128)
#undef MV_ATTN_CASE
    default:
      return MV_ERR_SHAPE;
  }
  if (e != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("tree_attention");
}

extern "C" mv_status tree_attention_workspace(int32_t H, int32_t D, int32_t S_max, int32_t n_nodes, size_t* bytes) {
  if (!bytes || H < 1 || H > 256 || S_max < 1 || n_nodes < 1 || n_nodes > MV_MAX_NODES) return MV_ERR_INVALID_ARG;
  if (D != 16 && D != 32 && D != 64 && D != 128) return MV_ERR_SHAPE;
  *bytes = tree_attn_ws_bytes(H, D, S_max, n_nodes);
  return MV_OK;
}

extern "C" mv_status tree_attention(const mv_bf16* q, const mv_bf16* k_cache, const mv_bf16* v_cache, int32_t H,
                                    int32_t D, int32_t S_max, int32_t prefix_len, const mv_tree* tree, float scale,
                                    mv_bf16* out, void* workspace, size_t ws_bytes, mv_stream stream) {
  if (!q || !k_cache || !v_cache || !tree || !out || !workspace) return MV_ERR_INVALID_ARG;
  if (!tree->d_ancestors) return MV_ERR_CUDA;
  size_t need = 0;
  mv_status s = tree_attention_workspace(H, D, S_max, tree->n_nodes, &need);
  if (s != MV_OK) return s;
  if (prefix_len < 0 || prefix_len + tree->n_nodes > S_max) return MV_ERR_CAPACITY;
  if (ws_bytes < need) return MV_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
    return MV_ERR_SHAPE;
  CUtensorMap kmap, vmap;
  if (!tree_attn_make_maps(&kmap, &vmap, k_cache, v_cache, H, D, S_max, 1, (size_t)H * S_max * D * 2))
    return MV_ERR_CUDA;
  return launch_tree_attention(kmap, vmap, 0, 0, q, H, D, S_max, nullptr, prefix_len, prefix_len, tree, scale, out,
                               workspace, static_cast<cudaStream_t>(stream));
}
