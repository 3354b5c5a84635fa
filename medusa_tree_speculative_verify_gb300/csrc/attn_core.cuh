// One head (or one key split of it) of tree attention, shared by the standalone kernel and the projection
// chain that runs the attention of its layer first.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.2 Tree attention and 二.5 tree_decoding(): every tree node
// attends to the whole cached prefix and to its own root-to-node path. 128 threads (4 warps, 16 query rows each)
// handle up to 64 query rows: Q fragments come straight from global memory, key / value tiles of 64 keys arrive
// by TMA (128-byte swizzle, 2-stage mbarrier ring), Q K^T and P V run on mma.sync m16n8k16 (bf16, fp32
// accumulate), the softmax is online in registers, the mask is a 64-bit visibility word per row and key tile. The
// C CTAs of a cluster split the head's key tiles; each leaves its (max, sum, output) partial in its own shared
// memory and, after a cluster-wide step, merges 1/C of the rows over distributed shared memory (rank order:
// deterministic).
#pragma once

#include "common.cuh"

namespace attn {

constexpr int kThreads = 128;  // 4 warps of 16 query rows
constexpr int kKeys = 64;   // keys per tile
constexpr int kRows = 64;   // query rows per CTA (tree nodes, padded)
constexpr int kStages = 2;  // key/value tiles in flight
constexpr int kMinTiles = 2;       // key tiles per split at the longest prefix, at least (sets the cluster size)
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

struct Args {
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

// Shared memory one head() needs: the key/value ring, which the merge buffers overlay afterwards.
template <int D>
constexpr size_t smem_bytes() {
  constexpr size_t ring = (size_t)2 * kStages * kKeys * D * 2;
  constexpr size_t merge = ((size_t)kRows * (D + 4) + kRows * 2) * sizeof(float);
  return ring > merge ? ring : merge;
}

// Named barrier 1 over the 128 attention threads (the standalone kernel's whole CTA, the chain's epilogue warps).
MV_DEV void grp_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
MV_DEV bool grp_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kThreads)
      : "memory");
  return r != 0;
}

// Attention of head h (key split `split` of C = a.splits) for the 64 query rows of block `row0` (one tree) or of
// sequence `seq` (a.seq_rows > 0). smem: smem_bytes<D>() bytes, 1024-byte aligned; full: kStages mbarriers
// initialised with count 1 (this call uses each from phase 0). sync.ready() / sync.done(): steps over the
// attention threads of all C CTAs of the cluster (only reached when the head has more than one working split).
template <int D, class Sync>
MV_DEV void head(const Args& a, const CUtensorMap* kmap, const CUtensorMap* vmap, uint8_t* smem, uint64_t* full,
                 int split, int h, int seq, int row0, int tid, Sync& sync) {
  constexpr int kTileBytes = kKeys * D * 2;
  constexpr int kBoxCols = D >= 64 ? 64 : D;
  constexpr int kBoxes = D / kBoxCols;
  constexpr int KS = D / 16;  // k-steps over the head dim
  constexpr int DN = D / 8;   // n-tiles over the head dim
  constexpr int kPo = D + 4;  // row pitch (floats) of the partial output in shared memory
  uint8_t* sk = smem;                       // kStages x [64][D]
  uint8_t* sv = sk + kStages * kTileBytes;  // kStages x [64][D]
  const int qrow0 = a.seq_rows ? seq * a.seq_rows : row0;  // q / out rows of this block
  const int plane_k = a.plane_k + seq * a.seq_planes, plane_v = a.plane_v + seq * a.seq_planes;
  const int C = a.splits;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int P = a.d_prefix ? a.d_prefix[seq] : a.prefix;
  const int n_all = a.n;
  if (P < 0 || P + n_all > a.S_max) {
    if (tid == 0) mv_set_error(a.err, 4, MV_DEVERR_INDEX);
    return;
  }
  const int n = min(kRows, n_all - row0);         // query rows of this block
  const int n_keys = min(n_all, row0 + kRows);    // tree keys any of them can see
  const int total_tiles = (P + n_keys + kKeys - 1) / kKeys;
  // Key tile t (keys 64 t .. 64 t + 63, absolute positions) goes to split t mod C, whatever the prefix length
  // and the tree size. A query row's result then depends only on the keys it can see: the tiles past its last
  // visible key are fully masked and leave its running max, sum and output exactly as they were, and a split
  // with no visible key adds exact zeros to the merge. So a tree node's row is bit for bit the row the same
  // token gets when it is decoded alone at the same position (a tree of the root only, prefix = its position),
  // and greedy verification emits exactly the library's own autoregressive greedy stream.
  // The cluster is sized for the longest prefix; at this prefix the first S = min(C, tiles) splits get tiles.
  // With S = 1 the first CTA does the whole head and writes it directly (the same arithmetic as a one-split
  // merge); the others leave at once (no cluster barrier is used then). With S > 1 the idle splits still take
  // part in the barriers but contribute nothing to the merge.
  const int S = max(1, min(C, total_tiles));
  if (S == 1 && split > 0) return;
  const int count = split < S ? (total_tiles - split + C - 1) / C : 0;  // tiles split, split + C, ...

  auto issue = [&](int i) {  // tile split + i C into stage i % kStages
    const int st = i % kStages, key0 = (split + i * C) * kKeys;
    mbar_arrive_expect_tx(&full[st], 2 * kTileBytes);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) {
      tma_load_4d(sk + st * kTileBytes + b * (kKeys * kBoxCols * 2), kmap, &full[st], b * kBoxCols, key0, h,
                  plane_k);
      tma_load_4d(sv + st * kTileBytes + b * (kKeys * kBoxCols * 2), vmap, &full[st], b * kBoxCols, key0, h,
                  plane_v);
    }
  };
  // the first key/value tiles are requested before Q is loaded, so the two latencies overlap
  if (tid == 0)
    for (int i = 0; i < kStages && i < count; ++i) issue(i);
  // Q fragments of this warp's 16 rows straight from global memory (rows >= n are zero): thread (g, t4) holds
  // rows g and g + 8, columns 16 ks + 2 t4 (+1) and 16 ks + 8 + 2 t4 (+1), the m16n8k16 A layout
  uint32_t qa[KS][4];
  {
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    const uint32_t* qw0 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)(qrow0 + r0) * a.H + h) * D);
    const uint32_t* qw1 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)(qrow0 + r1) * a.H + h) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = r0 < n ? qw0[8 * ks + t4] : 0u;
      qa[ks][1] = r1 < n ? qw1[8 * ks + t4] : 0u;
      qa[ks][2] = r0 < n ? qw0[8 * ks + 4 + t4] : 0u;
      qa[ks][3] = r1 < n ? qw1[8 * ks + 4 + t4] : 0u;
    }
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
    if (grp_any(!got)) {
      if (tid == 0) mv_set_error(a.err, 4, MV_DEVERR_TIMEOUT);
      ok = false;
      stop = i;
      break;
    }
    const uint32_t kb = smem_u32(sk + st * kTileBytes), vb = smem_u32(sv + st * kTileBytes);
    const int key0 = (split + i * C) * kKeys;
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
    grp_bar();  // every warp is done with this stage
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
  grp_bar();
  float* po = reinterpret_cast<float*>(smem);  // [64][D + 4] (padded rows: conflict-free float2 stores)
  float* pml = po + kRows * kPo;               // [64][2] running max (log2 domain) and sum
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
  sync.ready();  // every partial of the head is in place
  const int r0 = split * n / C, r1 = (split + 1) * n / C;  // this CTA's query rows
  const uint32_t ml_s = smem_u32(pml), po_s = smem_u32(po);
  // Consecutive threads take consecutive 16-byte columns of a row (a warp reads whole rows of the partials),
  // each thread kU elements of the CTA's rows; every split's (max, sum) and partial values of those elements are
  // loaded before any is used. O = sum_s w_s O_s, w_s = 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s' over the row's S
  // splits, in rank order.
  constexpr int kF4 = D / 4, kU = 2;  // float4 per row; elements per thread and pass
  const int total = (r1 - r0) * kF4;
  for (int e0 = tid; e0 < total; e0 += kU * kThreads) {
    float2 ml[kU][kMaxSplits];
    float4 v[kU][kMaxSplits];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kThreads;
      if (e >= total) break;
      const int q = r0 + e / kF4, c4 = (e % kF4) * 4;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        if (sp < S) {
          ml[u][sp] = ld_cluster_f2(map_rank(ml_s + (uint32_t)(q * 8), (uint32_t)sp));
          v[u][sp] = ld_cluster_f4(map_rank(po_s + (uint32_t)((q * kPo + c4) * 4), (uint32_t)sp));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kThreads;
      if (e >= total) break;
      const int q = r0 + e / kF4, c4 = (e % kF4) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp)
        if (sp < S) M = fmaxf(M, ml[u][sp].x);
      const float base = M == -INFINITY ? 0.0f : M;
      float w[kMaxSplits], L = 0.0f;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        w[sp] = sp < S ? exp2f(ml[u][sp].x - base) : 0.0f;
        L += sp < S ? w[sp] * ml[u][sp].y : 0.0f;
      }
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        if (sp < S) {
          const float ws = w[sp] * inv;
          acc.x += ws * v[u][sp].x;
          acc.y += ws * v[u][sp].y;
          acc.z += ws * v[u][sp].z;
          acc.w += ws * v[u][sp].w;
        }
      }
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(a.out + ((size_t)(qrow0 + q) * a.H + h) * D + c4) = pk;
    }
  }
  sync.done();  // no CTA goes on while another may still read its partial
}

}  // namespace attn
