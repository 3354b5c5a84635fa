// Stochastic root of a verify step: typical and nucleus one-token draws from one logits row.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.4 generate_candidates(): with temperature > 0 and without
// the "fast" flag the root token is drawn by get_typical_one_token(logits, T, eps, delta) or
// get_nucleus_one_token(logits, T, top_p) (二.1 medusa_generate(): top_p = 0.8). The pages do not print the two
// bodies; this kernel computes the plain readings:
//   typical: p = softmax(z / T) restricted to eta-sampling's allow set {p > tau}, tau = min(eps, delta exp(-H)),
//            H = -sum p log(p + 1e-5) (一.3 Typical acceptance), renormalised;
//   nucleus: the smallest leading set of tokens, logits descending and equal logits by lower index, whose
//            probability mass reaches top_p (a token is kept iff the mass before it is below top_p);
//   draw:    the first token, in vocabulary order, whose cumulative kept mass exceeds u * (kept mass), with
//            u = (w >> 11) 2^-53 and w the SplitMix64 word `counter` under a 64-bit key (Steele, Lea and Flood,
//            "Fast Splittable Pseudorandom Number Generators", OOPSLA 2014).
//
// Rows up to 131072 logits: one cluster of 8 CTAs per draw, the logits in registers (the cluster kernel below).
// Longer rows: one CTA of 512 threads, the row staged in shared memory when it fits (up to 49152 logits),
// otherwise read from global memory (L2) by every pass. Probability masses are fixed-point integers:
// E = round(e 2^40) with e = exp((z - max) / T) <= 1, so every sum is exact and the drawn token does not depend
// on the order of the additions.
//
// The nucleus boundary is found without a sort, in three levels over the row:
//   1. histogram of masses over 2048 bins of x = 16 (max - z) / T (1/16 nat of probability each; x is
//      monotone in z, so bins follow the token order exactly), and the bin where the cumulative mass from the
//      top first reaches ceil(top_p * S);
//   2. the same over 2048 sub-bins of that bin;
//   3. inside that sub-bin, distinct logits one by one from the largest (each a block max and a count; equal
//      logits share one mass, so a tie group is resolved by a count and an index-order scan).
#include <float.h>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kST = 512;           // threads
constexpr int kSW = kST / 32;      // warps
constexpr int kBins = 2048;
constexpr int kStageMaxBytes = 192 * 1024;
constexpr uint32_t kSite = 13;     // device error site

MV_DEV uint64_t splitmix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

MV_DEV uint64_t fixmass(float e) { return (uint64_t)__float2ull_rn(e * 1099511627776.0f); }  // e * 2^40

// Unsigned key with the order of the float (equal floats, +0 and -0 included, give equal keys).
MV_DEV uint32_t order_key(float z) {
  const uint32_t b = __float_as_uint(z == 0.0f ? 0.0f : z);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
MV_DEV float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

struct Scratch {
  float f[kSW];
  int i[kSW];
  unsigned long long u[kSW];
  unsigned long long pre[kSW];  // per-warp exclusive prefixes
  int sel[4];
  unsigned long long selu[4];
};

// Block-wide reductions; every thread gets the result. Each ends with a barrier so the scratch can be reused.
MV_DEV void block_argmax(float& v, int& i, Scratch& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (vi_better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
  if (lane == 0) {
    s.f[w] = v;
    s.i[w] = i;
  }
  __syncthreads();
  v = s.f[0];
  i = s.i[0];
  for (int k = 1; k < kSW; ++k)
    if (vi_better(s.f[k], s.i[k], v, i)) {
      v = s.f[k];
      i = s.i[k];
    }
  __syncthreads();
}

MV_DEV float block_sum(float v, Scratch& s) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) s.f[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
  for (int k = 0; k < kSW; ++k) t += s.f[k];
  __syncthreads();
  return t;
}

MV_DEV unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MV_DEV unsigned long long block_sum_u64(unsigned long long v, Scratch& s) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) s.u[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int k = 0; k < kSW; ++k) t += s.u[k];
  __syncthreads();
  return t;
}

MV_DEV uint32_t block_max_u32(uint32_t v, Scratch& s) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) s.i[threadIdx.x >> 5] = (int)v;
  __syncthreads();
  uint32_t t = 0;
  for (int k = 0; k < kSW; ++k) t = max(t, (uint32_t)s.i[k]);
  __syncthreads();
  return t;
}

MV_DEV unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Warp 0: the first bin b whose cumulative mass a0 + hist[0..b] reaches t (t <= a0 + sum of hist). Writes the
// bin to s.sel[0] and the mass before it to s.selu[0]; (kBins - 1, a0 + everything before it) if none does.
MV_DEV void find_crossing(const unsigned long long* hist, unsigned long long a0, unsigned long long t, Scratch& s) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = kBins / 32;
  unsigned long long mine = 0;
#pragma unroll 4
  for (int k = 0; k < kPer; ++k) mine += hist[lane * kPer + k];
  const unsigned long long incl = warp_incl_scan_u64(mine);
  const unsigned bal = __ballot_sync(0xffffffffu, a0 + incl >= t);
  const int L = bal ? __ffs(bal) - 1 : 31;
  if (lane == L) {
    unsigned long long c = a0 + incl - mine;
    int b = lane * kPer + kPer - 1;
#pragma unroll 1
    for (int k = 0; k < kPer; ++k) {
      const unsigned long long h = hist[lane * kPer + k];
      if (c + h >= t) {
        b = lane * kPer + k;
        break;
      }
      if (k < kPer - 1) c += h;
    }
    s.sel[0] = b;
    s.selu[0] = c;
  }
}

struct SampleArgs {
  const float* logits;
  int V, ld, n_rows;
  mv_posterior_result* res;  // if set: row = res->next_node, and res->next_root receives the token
  int32_t* out_token;        // if set: receives the token
  mv_root_params prm;
  uint64_t counter;
  uint64_t* d_counter;  // if set: the draw uses *d_counter and stores *d_counter + 1
  unsigned int* err;
  int staged;
};

// The whole draw on one CTA of kST threads over the row z (shared or global memory): the path for rows too long
// for the cluster kernel, and that kernel's fallback when the nucleus boundary lies in a bin of too many
// candidates (large groups of equal or nearly equal logits).
MV_DEV void draw_block(const SampleArgs& a, const float* z, unsigned long long* hist, Scratch& sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;

  // pass 1: max and its first index
  float m = -INFINITY;
  int amax = 0x7fffffff;
  for (int i = tid; i < V; i += kST) {
    const float v = z[i];
    if (vi_better(v, i, m, amax)) {
      m = v;
      amax = i;
    }
  }
  block_argmax(m, amax, sc);
  const int mode = a.prm.mode;
  const float inv_t = 1.0f / a.prm.temperature;

  // the kept set: typical -> e * inv_s > tau; nucleus -> (key > kstar) or (key == kstar and index <= istar)
  float inv_s = 0.0f, tau = 0.0f;
  uint32_t kstar = 0u;
  int istar = 0x7fffffff;
  if (mode == MV_ROOT_TYPICAL) {
    float s = 0.0f;
    for (int i = tid; i < V; i += kST) s += expf((z[i] - m) * inv_t);
    inv_s = 1.0f / block_sum(s, sc);
    float h = 0.0f;
    for (int i = tid; i < V; i += kST) {
      const float p = expf((z[i] - m) * inv_t) * inv_s;
      h += p * logf(p + 1e-5f);
    }
    const float H = -block_sum(h, sc);
    tau = fminf(a.prm.eps, a.prm.delta * expf(-H));
  } else if (mode == MV_ROOT_NUCLEUS) {
    unsigned long long sf = 0;
    for (int i = tid; i < V; i += kST) sf += fixmass(expf((z[i] - m) * inv_t));
    const unsigned long long S = block_sum_u64(sf, sc);
    unsigned long long T = (unsigned long long)ceil((double)a.prm.top_p * (double)S);
    if (T > S) T = S;
    if (T == 0) T = 1;  // keep at least the first token
    // level 1: bins of x = 16 (max - z) / T
    for (int b = tid; b < kBins; b += kST) hist[b] = 0ull;
    __syncthreads();
    for (int i = tid; i < V; i += kST) {
      const float zi = z[i];
      const unsigned long long E = fixmass(expf((zi - m) * inv_t));
      if (E) atomicAdd(&hist[(int)fminf((m - zi) * inv_t * 16.0f, (float)(kBins - 1))], E);
    }
    __syncthreads();
    if (warp == 0) find_crossing(hist, 0ull, T, sc);
    __syncthreads();
    const int b1 = sc.sel[0];
    unsigned long long A = sc.selu[0];
    __syncthreads();
    // level 2: sub-bins of bin b1
    for (int b = tid; b < kBins; b += kST) hist[b] = 0ull;
    __syncthreads();
    auto sub_of = [&](float zi, int& bin) {
      const float x = (m - zi) * inv_t * 16.0f;
      bin = (int)fminf(x, (float)(kBins - 1));
      return (int)fminf((x - (float)bin) * (float)kBins, (float)(kBins - 1));
    };
    for (int i = tid; i < V; i += kST) {
      const float zi = z[i];
      int bin;
      const int sb = sub_of(zi, bin);
      if (bin != b1) continue;
      const unsigned long long E = fixmass(expf((zi - m) * inv_t));
      if (E) atomicAdd(&hist[sb], E);
    }
    __syncthreads();
    if (warp == 0) find_crossing(hist, A, T, sc);
    __syncthreads();
    const int b2 = sc.sel[0];
    A = sc.selu[0];
    __syncthreads();
    // level 3: distinct logits of sub-bin (b1, b2), largest first, until the cumulative mass reaches T
    uint32_t kprev = 0xffffffffu;
    bool first = true;
    kstar = 0u;
    istar = -1;
    while (true) {
      uint32_t kmax = 0u;
      for (int i = tid; i < V; i += kST) {
        const float zi = z[i];
        int bin;
        const int sb = sub_of(zi, bin);
        const uint32_t k = order_key(zi);
        if (bin == b1 && sb == b2 && (first || k < kprev)) kmax = max(kmax, k + 1u);  // +1: 0 means none
      }
      kmax = block_max_u32(kmax, sc);
      if (kmax == 0u) {  // the sub-bin ran out (cannot happen with exact sums): keep everything up to kprev
        kstar = kprev;
        istar = 0x7fffffff;
        break;
      }
      const uint32_t kr = kmax - 1u;
      unsigned long long cnt = 0;
      for (int i = tid; i < V; i += kST) cnt += order_key(z[i]) == kr ? 1ull : 0ull;
      cnt = block_sum_u64(cnt, sc);
      const unsigned long long Er = fixmass(expf((key_value(kr) - m) * inv_t));
      if (A + cnt * Er >= T) {
        // the n-th member of the tie group (index order) is the last kept token
        const unsigned long long n = Er == 0 ? cnt : min(cnt, (T - A + Er - 1) / Er);
        kstar = kr;
        const int W = (((V + kSW - 1) / kSW) + 31) & ~31;
        unsigned long long c = 0;
        for (int r = 0; r < W; r += 32) {
          const int i = warp * W + r + lane;
          c += __popc(__ballot_sync(0xffffffffu, i < V && order_key(z[i]) == kr));
        }
        if (lane == 0) sc.u[warp] = c;
        __syncthreads();
        if (tid == 0) {
          unsigned long long p = 0;
          for (int w = 0; w < kSW; ++w) {
            sc.pre[w] = p;
            p += sc.u[w];
          }
          sc.sel[1] = 0x7fffffff;
        }
        __syncthreads();
        const unsigned long long pre = sc.pre[warp];
        if (pre < n && n <= pre + c) {
          unsigned long long q = pre;
          for (int r = 0; r < W; r += 32) {
            const int i = warp * W + r + lane;
            const unsigned bal = __ballot_sync(0xffffffffu, i < V && order_key(z[i]) == kr);
            const unsigned pc = __popc(bal);
            if (q + pc >= n) {
              const int need = (int)(n - q);  // 1-based rank inside this round's ballot
              unsigned bb = bal;
              for (int k = 1; k < need; ++k) bb &= bb - 1;
              if (lane == 0) sc.sel[1] = warp * W + r + __ffs(bb) - 1;
              break;
            }
            q += pc;
          }
        }
        __syncthreads();
        istar = sc.sel[1];
        __syncthreads();
        break;
      }
      A += cnt * Er;
      kprev = kr;
      first = false;
    }
  }

  // the draw: per-warp kept masses over contiguous ranges, then the warp holding the target walks its range
  const int W = (((V + kSW - 1) / kSW) + 31) & ~31;
  auto kept_mass = [&](int i) -> unsigned long long {
    if (i >= V) return 0ull;
    const float zi = z[i];
    const float e = expf((zi - m) * inv_t);
    bool keep;
    if (mode == MV_ROOT_TYPICAL) {
      keep = e * inv_s > tau;
    } else if (mode == MV_ROOT_NUCLEUS) {
      const uint32_t k = order_key(zi);
      keep = k > kstar || (k == kstar && i <= istar);
    } else {
      keep = i == amax;
    }
    return keep ? fixmass(e) : 0ull;
  };
  unsigned long long ws = 0;
  for (int r = 0; r < W; r += 32) ws += kept_mass(warp * W + r + lane);
  ws = warp_sum_u64(ws);
  if (lane == 0) sc.u[warp] = ws;
  __syncthreads();
  if (tid == 0) {
    unsigned long long p = 0;
    for (int w = 0; w < kSW; ++w) {
      sc.pre[w] = p;
      p += sc.u[w];
    }
    const uint64_t ctr = a.d_counter ? *a.d_counter : a.counter;
    const uint64_t word = splitmix64(a.prm.key + (ctr + 1ull) * 0x9E3779B97F4A7C15ull);
    sc.selu[2] = p;                                         // kept mass
    sc.selu[3] = p ? __umul64hi(word & ~0x7ffull, p) : 0ull;  // floor(u * kept mass), u = (word >> 11) 2^-53
    sc.sel[2] = amax;
    if (a.d_counter) *a.d_counter = ctr + 1ull;
  }
  __syncthreads();
  const unsigned long long K = sc.selu[2], target = sc.selu[3];
  const unsigned long long pre = sc.pre[warp];
  if (K && pre <= target && target < pre + sc.u[warp]) {
    unsigned long long c = pre;
    for (int r = 0; r < W; r += 32) {
      const int i = warp * W + r + lane;
      const unsigned long long incl = warp_incl_scan_u64(kept_mass(i));
      const unsigned bal = __ballot_sync(0xffffffffu, c + incl > target);
      if (bal) {
        if (lane == 0) sc.sel[2] = warp * W + r + __ffs(bal) - 1;
        break;
      }
      c += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int tok = (sc.sel[2] >= 0 && sc.sel[2] < V) ? sc.sel[2] : 0;  // a row with no ordered value: token 0
    if (a.res) a.res->next_root = tok;
    if (a.out_token) *a.out_token = tok;
  }
}

// The row of this draw (res->next_node when res is set, checked against n_rows), or nullptr after recording an
// index error.
MV_DEV const float* draw_row(const SampleArgs& a) {
  int row = 0;
  if (a.res) {
    row = a.res->next_node;
    if (row < 0 || row >= a.n_rows) {
      if (threadIdx.x == 0 && cluster_rank() == 0) mv_set_error_detail(a.err, kSite, MV_DEVERR_INDEX, (uint32_t)row);
      return nullptr;
    }
  }
  return a.logits + (size_t)row * a.ld;
}

__global__ void __launch_bounds__(kST, 1) sample_root_kernel(const SampleArgs a) {
  extern __shared__ float4 s_dyn[];
  __shared__ unsigned long long hist[kBins];
  __shared__ Scratch sc;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, V = a.V;
  const float* g = draw_row(a);
  if (!g) return;
  const float* z = g;
  if (a.staged) {
    float* srow = reinterpret_cast<float*>(s_dyn);
    if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
      const int V4 = V >> 2;
      const float4* g4 = reinterpret_cast<const float4*>(g);
      for (int i = tid; i < V4; i += kST) s_dyn[i] = __ldcg(g4 + i);
      for (int i = 4 * V4 + tid; i < V; i += kST) srow[i] = __ldcg(g + i);
    } else {
      for (int i = tid; i < V; i += kST) srow[i] = __ldcg(g + i);
    }
    __syncthreads();
    z = srow;
  }
  draw_block(a, z, hist, sc);
}

// ---------------------------------------------------------------------------------------------- cluster draw
// One draw on a cluster of kRC CTAs: CTA c holds logits [c kRT kRE, (c + 1) kRT kRE) of the row, thread t of it
// kRE consecutive ones in registers. The block-level steps above become cluster-wide through small per-CTA
// tables that every CTA writes into every other CTA's shared memory, one cluster barrier per step:
//   max (all modes);
//   typical: the sum of exp((z - max) / T), then the entropy sum, each in rank order (deterministic);
//   nucleus: the total mass and the level-1 histogram at once: each CTA builds its own histogram, merges the
//            bins [c kSlice, (c + 1) kSlice) of all kRC histograms and publishes the slice total; every CTA then
//            finds the crossing bin from the totals and the owning CTA's merged slice. When that bin holds at
//            most kCap tokens they are copied to every CTA, which ranks them (logit descending, index
//            ascending) and finds the last kept token; otherwise the same is done one level down (sub-bins of
//            the crossing bin), and past that CTA 0 runs the single-CTA draw over the row in global memory;
//   the draw: exact kept masses per CTA, and the CTA holding the target finds the token.
// Every value a step reads from another CTA was written to a table used by that step alone, so a fast CTA that
// has passed a barrier never overwrites what a slower one has still to read.
constexpr int kRC = 8;                // CTAs per cluster
constexpr int kSlice = kBins / kRC;   // merged bins per CTA
constexpr int kCap = 512;             // nucleus candidates ranked in shared memory

MV_DEV unsigned long long ld_cl_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
MV_DEV uint32_t ld_cl_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
MV_DEV void st_cl_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
MV_DEV void st_cl_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
MV_DEV uint32_t atom_cl_add_u32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
// Stores v into slot `rank` of the table at `tab` (a shared-memory array of kRC entries) in every CTA: lanes
// 0 .. kRC - 1 of the calling warp store one copy each.
MV_DEV void publish_u64(unsigned long long* tab, int rank, unsigned long long v) {
  const int lane = threadIdx.x & 31;
  if (lane < kRC) st_cl_u64(map_rank(smem_u32(tab + rank), (uint32_t)lane), v);
}
MV_DEV void publish_u32(uint32_t* tab, int rank, uint32_t v) {
  const int lane = threadIdx.x & 31;
  if (lane < kRC) st_cl_u32(map_rank(smem_u32(tab + rank), (uint32_t)lane), v);
}

// Exclusive prefix of v over the CTA's threads in thread order; *total receives the sum.
MV_DEV unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long* total, Scratch& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned long long incl = warp_incl_scan_u64(v);
  if (lane == 31) s.u[w] = incl;
  __syncthreads();
  unsigned long long pre = 0, t = 0;
  for (int k = 0; k < kSW; ++k) {
    if (k < w) pre += s.u[k];
    t += s.u[k];
  }
  __syncthreads();
  *total = t;
  return pre + incl - v;
}

struct ClusterSmem {
  unsigned long long hist[kBins];  // this CTA's histogram of masses
  uint32_t cnt[kBins];             // and of tokens
  unsigned long long mh[kSlice];   // merged bins of this CTA's slice: inclusive prefix of the masses
  uint32_t mc[kSlice];             // merged token counts
  uint32_t ckey[kCap];             // nucleus candidates (the same list in every CTA)
  int cidx[kCap];
  unsigned long long cmass[kCap];
  uint32_t ccount;                 // slots handed out (CTA 0's copy)
  // one table per step (entry c written by CTA c)
  float tmax[kRC];
  int targ[kRC];
  float tsum[kRC], tent[kRC];
  unsigned long long tslice[2][kRC];  // per nucleus level: slice masses
  uint32_t tcount[2][kRC];            // and token counts
  unsigned long long tkept[kRC];
  int found[4];
  unsigned long long foundu[2];
};

template <int kRE>
__global__ void __launch_bounds__(kST, 1) sample_root_cluster_kernel(const SampleArgs a) {
  __shared__ ClusterSmem sm;
  __shared__ Scratch sc;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31;
  const int rank = (int)cluster_rank();
  const int V = a.V, mode = a.prm.mode;
  const float* g = draw_row(a);
  if (!g) return;  // every CTA of the cluster returns here, before any access to another CTA's shared memory
  // No CTA may touch another's shared memory before that CTA has started: every CTA arrives here and waits just
  // before its first remote store, so the row loads and the local max overlap the wait.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (tid == 0) sm.ccount = 0u;
  const uint64_t ctr = a.d_counter ? *a.d_counter : a.counter;  // every CTA reads it before CTA 0 may advance it

  // this thread's logits: indices i0 .. i0 + kRE - 1
  const int i0 = (rank * kST + tid) * kRE;
  float z[kRE];
  if (i0 + kRE <= V && (reinterpret_cast<uintptr_t>(g + i0) & 15) == 0) {
#pragma unroll
    for (int r = 0; r < kRE; r += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(g + i0 + r));
      z[r] = v.x;
      z[r + 1] = v.y;
      z[r + 2] = v.z;
      z[r + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int r = 0; r < kRE; ++r) z[r] = i0 + r < V ? __ldcg(g + i0 + r) : -INFINITY;
  }

  // step 1: max and its first index
  float m = -INFINITY;
  int amax = 0x7fffffff;
#pragma unroll
  for (int r = 0; r < kRE; ++r)
    if (i0 + r < V && vi_better(z[r], i0 + r, m, amax)) {
      m = z[r];
      amax = i0 + r;
    }
  block_argmax(m, amax, sc);
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
  if (tid < 32 && lane < kRC) {
    st_cl_u32(map_rank(smem_u32(&sm.tmax[rank]), (uint32_t)lane), __float_as_uint(m));
    st_cl_u32(map_rank(smem_u32(&sm.targ[rank]), (uint32_t)lane), (uint32_t)amax);
  }
  cluster_sync_all();
  m = -INFINITY;
  amax = 0x7fffffff;
  for (int c = 0; c < kRC; ++c)
    if (vi_better(sm.tmax[c], sm.targ[c], m, amax)) {
      m = sm.tmax[c];
      amax = sm.targ[c];
    }
  const float inv_t = 1.0f / a.prm.temperature;
  const bool have_max = amax >= 0 && amax < V;
  if (mode == MV_ROOT_ARGMAX) {
    if (rank == 0 && tid == 0) {
      const int tok = have_max ? amax : 0;
      if (a.res) a.res->next_root = tok;
      if (a.out_token) *a.out_token = tok;
      if (a.d_counter) *a.d_counter = ctr + 1ull;
    }
    return;
  }

  float e[kRE];  // exp((z - max) / T); 0 outside the row and for NaN logits
#pragma unroll
  for (int r = 0; r < kRE; ++r) {
    const float v = expf((z[r] - m) * inv_t);
    e[r] = (have_max && i0 + r < V && v == v) ? v : 0.0f;
  }

  // the kept set: typical -> e inv_s > tau; nucleus -> key > kstar, or key == kstar and index <= istar
  float inv_s = 0.0f, tau = 0.0f;
  uint32_t kstar = 0u;
  int istar = 0x7fffffff;
  bool fallback = false;
  if (mode == MV_ROOT_TYPICAL) {
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < kRE; ++r) s += e[r];
    s = block_sum(s, sc);
    if (tid < 32) publish_u32(reinterpret_cast<uint32_t*>(sm.tsum), rank, __float_as_uint(s));
    cluster_sync_all();
    float S = 0.0f;
    for (int c = 0; c < kRC; ++c) S += sm.tsum[c];
    inv_s = 1.0f / S;
    float h = 0.0f;
#pragma unroll
    for (int r = 0; r < kRE; ++r)
      if (i0 + r < V) {
        const float p = e[r] * inv_s;
        h += p * logf(p + 1e-5f);
      }
    h = block_sum(h, sc);
    if (tid < 32) publish_u32(reinterpret_cast<uint32_t*>(sm.tent), rank, __float_as_uint(h));
    cluster_sync_all();
    float Hs = 0.0f;
    for (int c = 0; c < kRC; ++c) Hs += sm.tent[c];
    tau = fminf(a.prm.eps, a.prm.delta * expf(Hs));  // Hs = -H
  } else if (mode == MV_ROOT_NUCLEUS) {
    // one level of the boundary search: histogram of this CTA's tokens selected by `sel` into bins `bin_of`,
    // merged over the cluster; every CTA learns the crossing bin of a0 + cumulative mass >= T, the mass before
    // it and its token count (found[0], foundu[0], found[1])
    // (level 0 also sets T = ceil(top_p S) from the slice totals, S = the total mass)
    unsigned long long T = 1;
    auto level = [&](int lv, unsigned long long a0, auto sel, auto bin_of) {
      for (int b = tid; b < kBins; b += kST) {
        sm.hist[b] = 0ull;
        sm.cnt[b] = 0u;
      }
      if (tid == 0) {  // overwritten by the crossing bin's thread below
        sm.found[0] = kBins - 1;
        sm.foundu[0] = a0;
        sm.found[1] = kCap + 1;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kRE; ++r)
        if (i0 + r < V && sel(z[r])) {
          const int b = bin_of(z[r]);
          const unsigned long long E = fixmass(e[r]);
          if (E) atomicAdd(&sm.hist[b], E);
          atomicAdd(&sm.cnt[b], 1u);
        }
      cluster_sync_all();  // every CTA's histogram is complete
      unsigned long long mine = 0;
      uint32_t n = 0;
      if (tid < kSlice) {
        const uint32_t hb = smem_u32(&sm.hist[rank * kSlice + tid]), cb = smem_u32(&sm.cnt[rank * kSlice + tid]);
#pragma unroll
        for (int c = 0; c < kRC; ++c) {
          mine += ld_cl_u64(map_rank(hb, (uint32_t)c));
          n += ld_cl_u32(map_rank(cb, (uint32_t)c));
        }
      }
      unsigned long long tot;
      const unsigned long long ex = block_excl_scan_u64(mine, &tot, sc);
      if (tid < kSlice) {
        sm.mh[tid] = ex + mine;
        sm.mc[tid] = n;
      }
      const unsigned long long ntot = block_sum_u64(n, sc);
      if (tid < 32) {
        publish_u64(sm.tslice[lv], rank, tot);
        publish_u32(sm.tcount[lv], rank, (uint32_t)ntot);
      }
      cluster_sync_all();  // every slice is merged and its total published
      if (lv == 0) {
        unsigned long long S = 0;
        for (int c = 0; c < kRC; ++c) S += sm.tslice[0][c];
        T = (unsigned long long)ceil((double)a.prm.top_p * (double)S);
        if (T > S) T = S;
        if (T == 0) T = 1;  // keep at least the first token
      }
      unsigned long long base = a0;
      int o = kRC - 1;
      for (int c = 0; c < kRC; ++c) {
        if (base + sm.tslice[lv][c] >= T) {
          o = c;
          break;
        }
        base += sm.tslice[lv][c];
      }
      if (tid < kSlice) {
        const uint32_t ob = map_rank(smem_u32(&sm.mh[0]), (uint32_t)o);
        const unsigned long long inc = ld_cl_u64(ob + 8u * tid);
        const unsigned long long prev = tid ? ld_cl_u64(ob + 8u * (tid - 1)) : 0ull;
        if ((base + inc >= T && base + prev < T) || (tid == kSlice - 1 && base + inc < T)) {
          sm.found[0] = o * kSlice + tid;
          sm.foundu[0] = base + prev;
          sm.found[1] = (int)ld_cl_u32(map_rank(smem_u32(&sm.mc[tid]), (uint32_t)o));
        }
      }
      __syncthreads();
    };
    auto bin1 = [&](float zi) { return (int)fminf((m - zi) * inv_t * 16.0f, (float)(kBins - 1)); };
    auto sub_of = [&](float zi) {
      const float x = (m - zi) * inv_t * 16.0f;
      const int bin = (int)fminf(x, (float)(kBins - 1));
      return (int)fminf((x - (float)bin) * (float)kBins, (float)(kBins - 1));
    };
    level(0, 0ull, [](float) { return true; }, bin1);
    const int b1 = sm.found[0];
    unsigned long long A = sm.foundu[0];
    int n_c = sm.found[1];
    int b2 = -1;
    if (n_c > kCap) {
      level(1, A, [&](float zi) { return bin1(zi) == b1; }, sub_of);
      b2 = sm.found[0];
      A = sm.foundu[0];
      n_c = sm.found[1];
    }
    if (n_c > kCap) {
      fallback = true;
    } else {
      // the candidates: every token of the crossing (sub-)bin, copied to every CTA at one slot per token
      const uint32_t cc = map_rank(smem_u32(&sm.ccount), 0u);
#pragma unroll
      for (int r = 0; r < kRE; ++r) {
        if (!(i0 + r < V) || bin1(z[r]) != b1 || (b2 >= 0 && sub_of(z[r]) != b2)) continue;
        const uint32_t slot = atom_cl_add_u32(cc, 1u);
        if (slot >= (uint32_t)kCap) continue;  // cannot happen: the count was taken over the same tokens
        const uint32_t k = order_key(z[r]);
        const unsigned long long E = fixmass(e[r]);
        for (int c = 0; c < kRC; ++c) {
          st_cl_u32(map_rank(smem_u32(&sm.ckey[slot]), (uint32_t)c), k);
          st_cl_u32(map_rank(smem_u32(&sm.cidx[slot]), (uint32_t)c), (uint32_t)(i0 + r));
          st_cl_u64(map_rank(smem_u32(&sm.cmass[slot]), (uint32_t)c), E);
        }
      }
      cluster_sync_all();  // every candidate is in every CTA
      // the last kept token: the candidate whose mass before it (A + the candidates ranked above it) is below T
      // and reaches T with its own
      if (tid == 0) {
        sm.found[2] = -1;
        sm.found[3] = 0;
      }
      __syncthreads();
      for (int q = tid; q < n_c; q += kST) {
        const uint32_t kq = sm.ckey[q];
        const int iq = sm.cidx[q];
        unsigned long long before = A;
        for (int j = 0; j < n_c; ++j) {
          const uint32_t kj = sm.ckey[j];
          if (kj > kq || (kj == kq && sm.cidx[j] < iq)) before += sm.cmass[j];
        }
        if (before < T && before + sm.cmass[q] >= T) {
          sm.found[2] = iq;
          sm.found[3] = (int)kq;
        }
      }
      __syncthreads();
      if (sm.found[2] >= 0) {
        istar = sm.found[2];
        kstar = (uint32_t)sm.found[3];
      } else {  // cannot happen with exact sums: keep the whole crossing bin
        kstar = 0u;
        istar = 0x7fffffff;
        for (int q = 0; q < n_c; ++q) kstar = q == 0 ? sm.ckey[q] : min(kstar, sm.ckey[q]);
      }
    }
  }
  if (fallback) {  // uniform over the cluster
    // the crossing search above read the owning CTA's merged bins: no CTA may leave before every CTA is done
    cluster_sync_all();
    if (rank == 0) draw_block(a, g, sm.hist, sc);
    return;
  }

  // the draw: exact kept masses of this thread, CTA and cluster, then the CTA holding the target
  auto kept_mass = [&](int r) -> unsigned long long {
    if (!(i0 + r < V)) return 0ull;
    bool keep;
    if (mode == MV_ROOT_TYPICAL) {
      keep = e[r] * inv_s > tau;
    } else {
      const uint32_t k = order_key(z[r]);
      keep = k > kstar || (k == kstar && i0 + r <= istar);
    }
    return keep ? fixmass(e[r]) : 0ull;
  };
  unsigned long long mine = 0;
#pragma unroll
  for (int r = 0; r < kRE; ++r) mine += kept_mass(r);
  unsigned long long cta_tot;
  const unsigned long long ex = block_excl_scan_u64(mine, &cta_tot, sc);
  if (tid < 32) publish_u64(sm.tkept, rank, cta_tot);
  cluster_sync_all();
  unsigned long long K = 0, base = 0;
  for (int c = 0; c < kRC; ++c) {
    if (c < rank) base += sm.tkept[c];
    K += sm.tkept[c];
  }
  const uint64_t word = splitmix64(a.prm.key + (ctr + 1ull) * 0x9E3779B97F4A7C15ull);
  const unsigned long long target = K ? __umul64hi(word & ~0x7ffull, K) : 0ull;  // floor(u K), u = (w >> 11) 2^-53
  if (rank == 0 && tid == 0 && a.d_counter) *a.d_counter = ctr + 1ull;
  int tok = -1;
  if (K == 0) {
    if (rank == 0 && tid == 0) tok = have_max ? amax : 0;
  } else if (base + ex <= target && target < base + ex + mine) {
    unsigned long long c = base + ex;
#pragma unroll
    for (int r = 0; r < kRE; ++r) {
      const unsigned long long E = kept_mass(r);
      if (tok < 0 && c + E > target) tok = i0 + r;
      c += E;
    }
  }
  if (tok >= 0) {
    if (a.res) a.res->next_root = tok;
    if (a.out_token) *a.out_token = tok;
  }
}

bool root_params_ok(const mv_root_params& p) {
  if (p.mode == MV_ROOT_ARGMAX) return true;
  if (p.mode != MV_ROOT_TYPICAL && p.mode != MV_ROOT_NUCLEUS) return false;
  if (!(p.temperature > 0.0f) || !(p.temperature < 1e30f)) return false;
  if (p.mode == MV_ROOT_TYPICAL) return p.eps >= 0.0f && p.delta >= 0.0f && p.eps < 1e30f && p.delta < 1e30f;
  return p.top_p > 0.0f && p.top_p <= 1.0f;
}

}  // namespace

bool mv_root_params_valid(const mv_root_params& p) { return root_params_ok(p); }

mv_status launch_sample_root(const float* logits, int V, int ld, int n_rows, mv_posterior_result* res,
                             int32_t* out_token, const mv_root_params& prm, uint64_t counter, uint64_t* d_counter,
                             cudaStream_t stream) {
  if (!logits || V < 1 || ld < V || n_rows < 1 || !root_params_ok(prm)) return MV_ERR_INVALID_ARG;
  const size_t row_bytes = ((size_t)V * sizeof(float) + 15) & ~size_t(15);
  const int cluster_re = V <= kRC * kST * 8 ? 8 : V <= kRC * kST * 32 ? 32 : 0;  // logits per thread, 0: one CTA
  const bool staged = cluster_re == 0 && row_bytes <= (size_t)kStageMaxBytes;
  static int flags[64] = {};
  if (staged && !mv_set_smem_once((const void*)sample_root_kernel, (int)row_bytes, flags)) return MV_ERR_CUDA;
  SampleArgs a;
  a.logits = logits;
  a.V = V;
  a.ld = ld;
  a.n_rows = n_rows;
  a.res = res;
  a.out_token = out_token;
  a.prm = prm;
  a.counter = counter;
  a.d_counter = d_counter;
  a.err = mv_error_word();
  a.staged = staged ? 1 : 0;
  if (cluster_re) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kRC);
    cfg.blockDim = dim3(kST);
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;  // the whole grid is one cluster
    at[0].val.clusterDim.x = kRC;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = mv_pdl_enabled() ? 2 : 1;
    const cudaError_t e = cluster_re == 8 ? cudaLaunchKernelEx(&cfg, sample_root_cluster_kernel<8>, a)
                                          : cudaLaunchKernelEx(&cfg, sample_root_cluster_kernel<32>, a);
    if (e != cudaSuccess) return MV_ERR_CUDA;
  } else if (mv_launch(sample_root_kernel, dim3(1), dim3(kST), staged ? row_bytes : 0, stream, a) != cudaSuccess) {
    return MV_ERR_CUDA;
  }
  return mv_last_launch("sample_root");
}

extern "C" mv_status sample_root(const float* d_logits, int32_t V, mv_root_params params, uint64_t counter,
                                 int32_t* d_token, mv_stream stream) {
  if (!d_logits || !d_token) return MV_ERR_INVALID_ARG;
  return launch_sample_root(d_logits, V, V, 1, nullptr, d_token, params, counter, nullptr,
                            static_cast<cudaStream_t>(stream));
}
