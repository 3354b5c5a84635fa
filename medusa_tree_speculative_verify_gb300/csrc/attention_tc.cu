// Tree attention on the 5th-generation tensor cores (tcgen05), for long cached prefixes.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.2 Tree attention and 二.5 tree_decoding(): every tree node
// attends to the whole cached prefix and to its own root-to-node path. With 64 tree queries every prefix key
// costs 64 x D multiply-adds twice (Q K^T and P V): at a 4096-key prefix that is 2.2 G multiply-adds over 32
// heads, more than the warp-level mma.sync path sustains (its tree_attn kernel is bound by that arithmetic
// there). This kernel runs both products as tcgen05.mma with the accumulators in tensor memory:
//   S = Q K^T   M = 128 query rows (the block's queries, zero-padded), N = 128 keys, K = D; A = Q and B = the key
//               tile, both K-major in shared memory (128-byte swizzle); S in one of two TMEM buffers, so the
//               product of tile i + 1 runs while the softmax reads tile i;
//   O += P V    A = P (bf16, written by the softmax threads in the same K-major layout), B = the value tile read
//               MN-major (the cache rows hold a key's D values contiguously); O stays in TMEM for the whole split.
// One thread per query row (thread r reads TMEM lane r): the row's max, the exponentials and their sum over the
// tile. The reference of the exponentials moves only when the row max grows by more than 2^8 (then O and the sum
// are rescaled in place), so most tiles touch O only through the MMA.
//
// Work split as in the warp-level kernel: key tile t (128 keys at absolute positions 128 t ..) goes to split
// t mod C, and a row's result depends only on the keys it can see (fully masked tiles add exact zeros), so the
// root row is bit for bit the same whatever the tree. The C CTAs of a cluster (the splits of one head) merge
// their (max, sum, unnormalised output) partials over distributed shared memory in rank order.
#include <float.h>

#include <algorithm>

#include "attn_core.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kTcThreads = 128;    // 4 warps: warp w owns TMEM lanes 32 w .. 32 w + 31
constexpr int kTcKeys = 128;       // keys per tile
constexpr int kTcRows = 64;        // query rows per CTA; the MMAs' 128 rows hold them twice (lanes r and r + 64)
constexpr int kTcM = 128;          // MMA rows
constexpr int kTcSplits = 4;       // CTAs per cluster, at most
constexpr uint32_t kTcTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // move the exponent reference when the row max grows by more than this

// Shared memory (bytes from a 1024-byte aligned base). Q: D / 64 regions of [128 rows][64] bf16; P: two buffers
// of 2 regions of [128 rows][64 keys]; K and V rings: 2 stages each of D / 64 regions of [128 keys][64]. The merge
// of the split partials afterwards overlays the rings.
template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kRegion = kTcM * 128;  // 16 KB: 128 rows (or keys) x 64 bf16, 128-byte rows
  static constexpr int kTile = kHalves * kRegion;
  static constexpr int kQ = 0;
  static constexpr int kP = kQ + kHalves * kRegion;  // two buffers of 2 regions (128 keys)
  static constexpr int kK = kP + 4 * kRegion;
  static constexpr int kV = kK + 2 * kTile;
  static constexpr int kEnd = kV + 2 * kTile;
  static constexpr int kPo = D + 4;  // merge: row pitch (floats) of the partial output
  static constexpr int kMergeBytes = (kTcRows * kPo + kTcRows * 2) * 4;
  static_assert(kTcKeys == kTcM, "the key tile fills the regions like the rows");
  static_assert(kK + kMergeBytes <= kEnd, "the merge buffers fit over the rings");
};

// kind::f16, D fp32, A / B bf16, M = 128, N = n; b_mn: B is MN-major (otherwise both K-major)
__host__ __device__ constexpr uint32_t tc_idesc(int n, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

// Shared-memory descriptors, 128-byte swizzle. K-major: rows of 64 bf16 (128 bytes) of consecutive K, 8-row
// groups 1024 bytes apart. MN-major: 128-byte rows of 64 consecutive N elements, one row per K index, 8-row (K)
// groups 1024 bytes apart, and the next 64 N elements `lbo` bytes further.
MV_DEV uint64_t desc_kmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
MV_DEV uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

MV_DEV void tc_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
MV_DEV void tc_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
MV_DEV void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MV_DEV void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MV_DEV void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
MV_DEV void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
MV_DEV void tc_commit_to(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane
MV_DEV void tc_ld32(uint32_t taddr, float* v) {
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
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 consecutive fp32 columns of this thread's TMEM lane, one load and its wait
MV_DEV void tc_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
      "}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
MV_DEV void tc_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 2^x on the special-function unit (denormal results flush to zero: these are probabilities stored as bf16)
MV_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Visibility of the 64 keys starting at s = (first key) - P for a row with ancestor words w0..w3 (tree keys
// past node 255 do not exist: none visible).
MV_DEV uint64_t block_bits(uint64_t w0, uint64_t w1, uint64_t w2, uint64_t w3, int s) {
  return s >= 64 * MV_MASK_WORDS ? 0ull : attn::tile_bits(w0, w1, w2, w3, s);
}

// One (key split, head, query block) per CTA; a cluster = the splits of one head. Warps 0-3 run the softmax (thread
// t reads TMEM lane t), warp 4 issues the copies and the MMAs. mbarriers order the three: kfull / vfull (a key /
// value tile landed), sdone (S of a tile is in TMEM), pfull (the 128 softmax threads wrote P of a tile), odone (P V
// of a tile is done), each used by every second tile (a phase per use, so every wait names the latest phase).
template <int D>
__global__ void __launch_bounds__(kTcThreads + 32, 1) tree_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                        const __grid_constant__ CUtensorMap vmap,
                                                                        const __grid_constant__ CUtensorMap qmap,
                                                                        const attn::Args a) {
  using Ly = TcLayout<D>;
  constexpr int kHalves = Ly::kHalves;
  constexpr uint32_t kIdS = tc_idesc(kTcKeys, false), kIdO = tc_idesc(D, true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Ly::kQ;
  uint8_t* sP = smem + Ly::kP;
  uint8_t* sK = smem + Ly::kK;
  uint8_t* sV = smem + Ly::kV;
  __shared__ __align__(8) uint64_t kfull[2], vfull[2], sdone[2], odone[2], pfull[2], qready, drain;
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int s_abort;
  __shared__ float s_max[2][2][kTcRows];  // per tile parity: each half's row max (then its sum), exchanged
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = (int)blockIdx.x, h = (int)blockIdx.y, C = a.splits;
  const int seq = a.seq_rows ? (int)blockIdx.z : 0;
  const int row0 = a.seq_rows ? 0 : (int)blockIdx.z * kTcRows;  // blocks of 64 query rows of one tree
  const int qrow0 = a.seq_rows ? seq * a.seq_rows : row0;
  const int plane_k = a.plane_k + seq * a.seq_planes, plane_v = a.plane_v + seq * a.seq_planes;
  pdl_trigger();
  if (tid == 0) {
    for (int st = 0; st < 2; ++st) {
      mbar_init(&kfull[st], 1);
      mbar_init(&vfull[st], 1);
      mbar_init(&sdone[st], 1);
      mbar_init(&odone[st], 1);
      mbar_init(&pfull[st], kTcThreads);
    }
    mbar_init(&qready, 1);  // the copies of Q (expected bytes)
    mbar_init(&drain, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tc_alloc(&tmem_sh, kTcTmemCols);
    tc_relinquish();
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = tmem_sh;
  auto release_tmem = [&]() {
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 0) tc_dealloc(tmem, kTcTmemCols);
  };
  pdl_wait();  // q, the cache and the prefix length come from earlier kernels

  const int P = a.d_prefix ? a.d_prefix[seq] : a.prefix;
  const int n_all = a.n;
  if (P < 0 || P + n_all > a.S_max) {  // the same in every CTA of the cluster: all leave here
    if (tid == 0) mv_set_error(a.err, 4, MV_DEVERR_INDEX);
    release_tmem();
    return;
  }
  const int n = min(kTcRows, n_all - row0);       // query rows of this block
  const int n_keys = min(n_all, row0 + kTcRows);  // tree keys any of them can see
  const int total_tiles = (P + n_keys + kTcKeys - 1) / kTcKeys;
  const int S = max(1, min(C, total_tiles));  // splits with tiles at this prefix
  if (S == 1 && split > 0) {  // the first CTA does the whole head and writes it (no cluster step is used)
    release_tmem();
    return;
  }
  const int count = split < S ? (total_tiles - split + C - 1) / C : 0;  // tiles split, split + C, ...
  // a bounded wait that gives up at once after any other wait of this CTA gave up
  auto wait = [&](uint64_t* bar, int use) {
    if (s_abort) return false;
    if (mbar_wait(bar, (uint32_t)(use & 1))) return true;
    s_abort = 1;
    return false;
  };

  // 64-key halves of this split's j-th tile that hold a key some row of the block can see (the prefix, then the
  // tree keys up to the block's last row): a half past them is neither copied nor multiplied by P (its S columns
  // are masked, so O is the same bits), which spares the copy of the empty half of the last tile.
  auto halves = [&](int j) { return (split + j * C) * kTcKeys + 64 < P + n_keys ? 2 : 1; };
  auto issue_k = [&](int j) {  // key tile of this split's j-th tile into stage j % 2
    const int st = j & 1, key0 = (split + j * C) * kTcKeys, nh = halves(j);
    mbar_arrive_expect_tx(&kfull[st], (uint32_t)(nh * kHalves * 64 * 128));
#pragma unroll
    for (int hb = 0; hb < kHalves; ++hb)
      for (int kb = 0; kb < nh; ++kb)
        tma_load_4d(sK + st * Ly::kTile + hb * Ly::kRegion + kb * 64 * 128, &kmap, &kfull[st], hb * 64,
                    key0 + 64 * kb, h, plane_k);
  };
  auto issue_v = [&](int j) {
    const int st = j & 1, key0 = (split + j * C) * kTcKeys, nh = halves(j);
    mbar_arrive_expect_tx(&vfull[st], (uint32_t)(nh * kHalves * 64 * 128));
#pragma unroll
    for (int hb = 0; hb < kHalves; ++hb)
      for (int kb = 0; kb < nh; ++kb)
        tma_load_4d(sV + st * Ly::kTile + hb * Ly::kRegion + kb * 64 * 128, &vmap, &vfull[st], hb * 64,
                    key0 + 64 * kb, h, plane_v);
  };
  // S[j % 2] = Q K(j)^T, then O += P V(j) (P buffer j % 2): issued by warp 4 once their operands are in place
  auto mma_s = [&](int j) {
    const uint32_t d = tmem + ((j & 1) ? kColS1 : kColS0);
    const uint32_t qb = smem_u32(sQ), kb = smem_u32(sK + (j & 1) * Ly::kTile);
#pragma unroll
    for (int hb = 0; hb < kHalves; ++hb)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma_f16(d, desc_kmajor(qb + hb * Ly::kRegion) + (uint64_t)(2 * k),
                   desc_kmajor(kb + hb * Ly::kRegion) + (uint64_t)(2 * k), kIdS, (hb | k) ? 1u : 0u);
    tc_commit_to(&sdone[j & 1]);
  };
  auto mma_o = [&](int j) {
    const uint32_t pb = smem_u32(sP + (j & 1) * 2 * Ly::kRegion), vb = smem_u32(sV + (j & 1) * Ly::kTile);
    const int nh = halves(j);
    for (int c = 0; c < nh; ++c)     // 64-key halves of the tile
#pragma unroll
      for (int k = 0; k < 4; ++k)    // 16 keys each
        tc_mma_f16(tmem + kColO, desc_kmajor(pb + c * Ly::kRegion) + (uint64_t)(2 * k),
                   desc_mnmajor(vb + (uint32_t)((c * 64 + 16 * k) * 128), (uint32_t)Ly::kRegion), kIdO,
                   (j > 0 || c > 0 || k > 0) ? 1u : 0u);
    tc_commit_to(&odone[j & 1]);
  };
  const int r = tid & (kTcRows - 1), kh = tid < kTcThreads ? tid >> 6 : 2;  // query row, key half (2: warp 4)
  const bool valid = tid < kTcThreads && r < n;
  float m_ref = -INFINITY, l = 0.0f;  // exponent reference (log2 domain, the same in both halves), half's sum
  int k_issued = 0, v_issued = 0, k_waited = 0, v_waited = 0;

  if (warp == 4) {
    // ------------------------------------------------------------------ copies and MMAs (one thread)
    // Event-driven: each pass takes every step whose inputs are ready (non-blocking probes of the barrier phase
    // it needs), so S of the next tile goes as soon as its key tile is in and its S buffer is free, whatever the
    // P V of the previous tile is doing. ms / mo: next S / P V product; kl / vl: next key / value copy.
    // S buffer ms % 2 is free once the softmax of tile ms - 2 arrived (mo >= ms - 1: P V of tile ms - 2 was
    // issued after that arrival); key stage kl % 2 once S of tile kl - 2 is done; value stage vl % 2 once P V
    // of tile vl - 2 is done. No barrier can run two phases past a probe: each next use is gated on this thread.
    if (lane == 0) {
      if (count > 0) {
        // Q (rows past the tensor's are zero-filled) into MMA rows 0..63 and again 64..127, with the first tiles
        tma_prefetch_desc(&qmap);
        mbar_arrive_expect_tx(&qready, (uint32_t)(2 * kHalves * kTcRows * 128));
#pragma unroll
        for (int hb = 0; hb < kHalves; ++hb)
#pragma unroll
          for (int dup = 0; dup < 2; ++dup)
            tma_load_3d(sQ + hb * Ly::kRegion + dup * kTcRows * 128, &qmap, &qready, hb * 64, h, qrow0);
        issue_k(k_issued++);
        issue_v(v_issued++);
      }
      bool ok = count == 0 || wait(&qready, 0);
      tc_after();
      int ms = 0, mo = 0;
      uint64_t t_last = mv_globaltimer();
      auto ready = [&](uint64_t* bar, int use) { return mbar_try_wait(bar, (uint32_t)(use & 1)); };
      while (ok && mo < count) {
        bool progress = false;
        if (ms < count && ms <= mo + 1 && ready(&kfull[ms & 1], ms >> 1)) {
          tc_after();
          mma_s(ms++);
          k_waited = ms;
          progress = true;
        }
        if (mo < ms && ready(&pfull[mo & 1], mo >> 1) && ready(&vfull[mo & 1], mo >> 1)) {
          tc_after();
          mma_o(mo++);
          v_waited = mo;
          progress = true;
        }
        if (k_issued < count &&
            (k_issued < 2 || (k_issued - 2 < ms && ready(&sdone[k_issued & 1], (k_issued - 2) >> 1)))) {
          issue_k(k_issued++);
          progress = true;
        }
        if (v_issued < count &&
            (v_issued < 2 || (v_issued - 2 < mo && ready(&odone[v_issued & 1], (v_issued - 2) >> 1)))) {
          issue_v(v_issued++);
          progress = true;
        }
        if (progress) {
          t_last = mv_globaltimer();
        } else if (s_abort || mv_globaltimer() - t_last > MV_WAIT_LIMIT_NS) {
          s_abort = 1;
          ok = false;
        }
      }
      if (!ok) {  // let every MMA issued and every copy in flight finish (bounded) before the buffers are reused
        mv_set_error(a.err, 4, MV_DEVERR_TIMEOUT);
        tc_commit_to(&drain);
        mbar_wait(&drain, 0u);
        if (count > 0) mbar_wait(&qready, 0u);
        for (int j = k_waited; j < k_issued; ++j)
          if (!mbar_wait(&kfull[j & 1], (uint32_t)((j >> 1) & 1))) break;
        for (int j = v_waited; j < v_issued; ++j)
          if (!mbar_wait(&vfull[j & 1], (uint32_t)((j >> 1) & 1))) break;
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax (128 threads)
    // Thread t reads TMEM lane t: query row r = t % 64 of the block, key half kh = t / 64 of every tile. Q rows
    // r and r + 64 of the MMA hold the same query (copied there by the issuing warp), so both halves of the row
    // find its S values in their own lanes; P rows 64..127 stay zero. Rows of Q past the block's queries hold
    // other rows of the q buffer or zeros: their S, P and O rows are neither kept nor stored.
    if (kh == 1) {  // P rows 64..127 of both buffers: zero (their outputs are not used)
#pragma unroll
      for (int c = 0; c < 32; ++c)
        *reinterpret_cast<uint4*>(sP + (c >> 3) * Ly::kRegion + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    static_assert(MV_MASK_WORDS == 4, "four ancestor words per node");
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    if (valid) {
      const uint64_t* ar = a.anc + (size_t)(row0 + r) * MV_MASK_WORDS;
      w0 = ar[0];
      w1 = ar[1];
      w2 = ar[2];
      w3 = ar[3];
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeros of P -> the tensor core
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    for (int i = 0; i < count; ++i) {
      bool got = wait(&sdone[i & 1], i >> 1);
      tc_after();
      const int key0 = (split + i * C) * kTcKeys;
      const uint64_t vb = key0 + kTcKeys <= P ? ~0ull : block_bits(w0, w1, w2, w3, key0 + 64 * kh - P);
      float sv[64];  // this half of the row of S
      tc_ld64(lane_base + ((i & 1) ? kColS1 : kColS0) + 64 * kh, sv);
      float mt = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        if ((vb >> e) & 1ull) mt = fmaxf(mt, sv[e]);
      s_max[i & 1][kh][r] = mt;
      attn::grp_bar();  // named barrier 1 over the 128 softmax threads
      const float m_new = fmaxf(m_ref, fmaxf(mt, s_max[i & 1][kh ^ 1][r]) * a.scale_log2);
      float ref = m_ref;
      if (m_new > -INFINITY && (m_ref == -INFINITY || m_new > m_ref + kRescaleLog2)) ref = m_new;
      const bool move = ref != m_ref;
      const bool had = m_ref > -INFINITY;  // rows that saw no key yet have only exact zeros in O
      const float factor = move ? (had ? exp2f(m_ref - ref) : 0.0f) : 1.0f;
      m_ref = ref;
      l *= factor;
      // rows of O (lanes 0..63, warps 0 and 1) whose reference moved: rescale once the previous P V is done
      // (warp-collective TMEM access: rows that keep their reference store their values back unchanged)
      const bool mine = kh == 0 && move && had;
      if (kh == 0 && __any_sync(0xffffffffu, mine)) {
        if (!wait(&odone[(i - 1) & 1], (i - 1) >> 1)) got = false;  // i > 0: a finite reference saw a tile before
        tc_after();
        const float f = mine ? factor : 1.0f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tc_ld32(lane_base + kColO + 32 * c, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= f;
          tc_st32(lane_base + kColO + 32 * c, ov);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      if (i >= 2 && !wait(&odone[i & 1], (i - 2) >> 1)) got = false;  // P buffer i % 2: the P V of tile i - 2
      // the exponentials against the reference, this half's sum, and its half of the row of P (bf16)
      const float base = ref == -INFINITY ? 0.0f : ref;
      uint8_t* pbuf = sP + (i & 1) * 2 * Ly::kRegion + kh * Ly::kRegion;  // keys 64 kh .. of the tile
      float sum = 0.0f;
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {  // 8 keys per 16-byte chunk
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int k0 = 8 * q8 + e;
          const float p0 = ((vb >> k0) & 1ull) ? fast_exp2(fmaf(sv[k0], a.scale_log2, -base)) : 0.0f;
          const float p1 = ((vb >> (k0 + 1)) & 1ull) ? fast_exp2(fmaf(sv[k0 + 1], a.scale_log2, -base)) : 0.0f;
          sum += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        if (valid)
          *reinterpret_cast<uint4*>(pbuf + r * 128 + ((q8 ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += sum;
      (void)got;  // an expired wait left s_abort set: the issuing warp stops, and the results are not used
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P -> the tensor core
      tc_before();
      mbar_arrive(&pfull[i & 1]);
    }
    // the last P V, then the row's sum: the halves' sums against the same reference
    if (count > 0) wait(&odone[(count - 1) & 1], (count - 1) >> 1);
    s_max[0][kh][r] = l;
    attn::grp_bar();
    l = s_max[0][0][r] + s_max[0][1][r];
  }
  __syncthreads();
  if (s_abort && tid == 0) mv_set_error(a.err, 4, MV_DEVERR_TIMEOUT);
  tc_after();
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  // ---- the split's result: rows 0..63 of O (lanes of warps 0 and 1), unnormalised against m_ref, and (m_ref, l)
  const uint32_t orow = lane_base + kColO;
  uint16_t* out_row = a.out + ((size_t)(qrow0 + r) * a.H + h) * D;
  if (S == 1) {  // one split holds every tile: normalise and write, nothing to merge
    if (kh == 0) {
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tc_ld32(orow + 32 * c, ov);  // count >= 1 here: O was written
        if (valid)
#pragma unroll
          for (int qc = 0; qc < 4; ++qc)
            *reinterpret_cast<uint4*>(out_row + 32 * c + 8 * qc) =
                make_uint4(pack_bf16x2(ov[8 * qc] * inv, ov[8 * qc + 1] * inv),
                           pack_bf16x2(ov[8 * qc + 2] * inv, ov[8 * qc + 3] * inv),
                           pack_bf16x2(ov[8 * qc + 4] * inv, ov[8 * qc + 5] * inv),
                           pack_bf16x2(ov[8 * qc + 6] * inv, ov[8 * qc + 7] * inv));
      }
    }
    release_tmem();
    return;
  }
  // the partial into this CTA's shared memory over the rings (every copy and MMA is done), then the merge: each
  // CTA of the cluster merges a slice of the rows over distributed shared memory, the splits in rank order
  float* po = reinterpret_cast<float*>(smem + Ly::kK);  // [64][D + 4]
  float* pml = po + kTcRows * Ly::kPo;                 // [64][2] exponent reference and sum
  __syncthreads();
  if (kh == 0) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float ov[32];
      if (count > 0) {
        tc_ld32(orow + 32 * c, ov);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0.0f;
      }
      if (valid)
#pragma unroll
        for (int qc = 0; qc < 8; ++qc)
          *reinterpret_cast<float4*>(po + r * Ly::kPo + 32 * c + 4 * qc) =
              make_float4(ov[4 * qc], ov[4 * qc + 1], ov[4 * qc + 2], ov[4 * qc + 3]);
    }
    if (valid) {
      pml[2 * r] = m_ref;
      pml[2 * r + 1] = l;
    }
  }
  release_tmem();
  cluster_sync_all();  // every partial of the head is in place
  const int r0 = split * n / C, r1 = (split + 1) * n / C;  // this CTA's rows of the merge
  const uint32_t ml_s = smem_u32(pml), po_s = smem_u32(po);
  // Consecutive threads take consecutive 16-byte columns of a row (a warp reads whole rows of the partials),
  // each thread kU elements of the CTA's rows; every split's (reference, sum) and partial values of those
  // elements are loaded before any is used. O = sum_s w_s O_s with w_s = 2^(m_s - M) / sum_s' 2^(m_s' - M) l_s',
  // in rank order.
  constexpr int kF4 = D / 4, kU = 4;  // float4 per row; elements per thread and pass
  const int total = (r1 - r0) * kF4;
  for (int e0 = tid; tid < kTcThreads && e0 < total; e0 += kU * kTcThreads) {
    float2 ml[kU][kTcSplits];
    float4 v[kU][kTcSplits];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kTcThreads;
      if (e >= total) break;
      const int q = r0 + e / kF4, c4 = (e % kF4) * 4;
#pragma unroll
      for (int sp = 0; sp < kTcSplits; ++sp) {
        if (sp < S) {
          ml[u][sp] = ld_cluster_f2(map_rank(ml_s + (uint32_t)(q * 8), (uint32_t)sp));
          v[u][sp] = ld_cluster_f4(map_rank(po_s + (uint32_t)((q * Ly::kPo + c4) * 4), (uint32_t)sp));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kTcThreads;
      if (e >= total) break;
      const int q = r0 + e / kF4, c4 = (e % kF4) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < kTcSplits; ++sp)
        if (sp < S) M = fmaxf(M, ml[u][sp].x);
      const float bs = M == -INFINITY ? 0.0f : M;
      float w[kTcSplits], L = 0.0f;
#pragma unroll
      for (int sp = 0; sp < kTcSplits; ++sp) {
        w[sp] = sp < S ? exp2f(ml[u][sp].x - bs) : 0.0f;
        L += sp < S ? w[sp] * ml[u][sp].y : 0.0f;
      }
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kTcSplits; ++sp) {
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
  cluster_sync_all();  // no CTA leaves while another may still read its partial
}
// At least 128 KB, so that one CTA occupies an SM: each CTA allocates all 512 TMEM columns, and two CTAs of a
// cluster on one SM would wait on each other (the allocation of the one, the merge barrier of the other).
size_t tc_smem_bytes(int D) {
  return 1024 + (size_t)std::max(128 * 1024, D == 64 ? TcLayout<64>::kEnd : TcLayout<128>::kEnd);
}

// Clusters of c CTAs of the D-variant that can be resident at once (asked once per device, D and c).
int tc_max_active_clusters(int D, int c) {
  static int cache[64][2][kTcSplits + 1];  // 0 = not asked yet, -1 = none
  const int dev = mv_device();
  if (dev < 0 || dev >= 64 || c < 1 || c > kTcSplits || (D != 64 && D != 128)) return 0;
  int& slot = cache[dev][D == 64 ? 0 : 1][c];
  if (slot == 0) {
    const size_t smem = tc_smem_bytes(D);
    const void* fn = D == 64 ? (const void*)tree_attn_tc_kernel<64> : (const void*)tree_attn_tc_kernel<128>;
    static int flags[2][64] = {};
    int n = 0;
    if (mv_set_smem_once(fn, (int)smem, flags[D == 64 ? 0 : 1])) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1024);
      cfg.blockDim = dim3(kTcThreads + 32);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = c;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    slot = n > 0 ? n : -1;
  }
  return slot > 0 ? slot : 0;
}

}  // namespace

mv_status launch_tree_attention_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, int plane_k, int plane_v,
                                   const mv_bf16* q, int H, int D, int S_max, const int32_t* d_prefix, int prefix,
                                   int max_prefix, const mv_tree* t, int n, float scale, mv_bf16* out,
                                   cudaStream_t stream, int nseq, int seq_planes) {
  if (D != 64 && D != 128) return MV_ERR_UNSUPPORTED;
  if (n < 1 || n > MV_MAX_NODES || nseq < 1 || (nseq > 1 && (n > attn::kRows || !d_prefix))) return MV_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(q) & 15) return MV_ERR_SHAPE;
  // q [rows][H][D] as (d, head, row) boxes of 64 d x one head x 64 rows
  CUtensorMap qmap;
  {
    const int q_rows = nseq > 1 ? nseq * attn::kRows : n;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)q_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)H * D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kTcRows};
    if (!mv_encode_tmap(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
      return MV_ERR_CUDA;
  }
  // blocks of 128 query rows of one tree, or one block per sequence (its rows 64 b ..)
  const int blocks = nseq > 1 ? nseq : (n + kTcRows - 1) / kTcRows;
  const int max_tiles = (max_prefix + n + kTcKeys - 1) / kTcKeys;
  int splits = std::max(1, std::min(kTcSplits, (max_tiles + 1) / 2));  // about two tiles per split, at least
  while (splits > 1 && tc_max_active_clusters(D, splits) < H * blocks) --splits;
  if (tc_max_active_clusters(D, splits) < 1) return MV_ERR_CUDA;
  attn::Args a{};
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
  a.seq_rows = nseq > 1 ? attn::kRows : 0;
  a.seq_planes = seq_planes;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = mv_error_word();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, H, blocks);
  cfg.blockDim = dim3(kTcThreads + 32);
  cfg.dynamicSmemBytes = tc_smem_bytes(D);
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
  const cudaError_t e = D == 64 ? cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<64>, kmap, vmap, qmap, a)
                                : cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<128>, kmap, vmap, qmap, a);
  if (e != cudaSuccess) return MV_ERR_CUDA;
  return mv_last_launch("tree_attention_tc");
}
