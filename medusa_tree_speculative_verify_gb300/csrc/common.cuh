// Shared device helpers for the Medusa tree-verify kernels (sm_103a).
//
// * status / error word: every bounded wait or index check that fails writes a
//   code into one device word (first error wins) and the kernel returns early;
//   mv_get_error() reads and clears it.
// * PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and tcgen05.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa_verify.h"

#define MV_DEV __device__ __forceinline__

// error codes written to the device error word (high 16 bits: site, low 16 bits: kind)
enum : uint32_t {
  MV_DEVERR_TIMEOUT = 1,   // a bounded wait expired
  MV_DEVERR_INDEX = 2,     // an index read from device memory was out of range
};

// Device error word of the current device (library-owned, no allocation: a __device__ symbol). The word
// after it holds a detail value of the first error (e.g. the offending index), see mv_get_error_detail().
unsigned int* mv_error_word();
// Host-side helpers.
mv_status mv_last_launch(const char* what);
int mv_sm_count();
int mv_device();
// Sets the dynamic shared-memory limit of `func` once per device (later calls are free, so launches stay
// capturable in CUDA graphs). `flags` must point to a zero-initialised int[64] owned by the caller.
bool mv_set_smem_once(const void* func, int bytes, int* flags);

// Programmatic dependent launch: every kernel of the step is launched with programmatic stream serialization,
// so it may start while the previous kernel drains. pdl_wait() blocks until the previous grid has finished and
// its writes are visible (a no-op when launched without the attribute); work before it may only read data no
// earlier kernel writes (the weights). pdl_trigger() lets the next grid start launching.
MV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Data written by an earlier kernel of the stream is never read through the non-coherent path (__ldg,
// const __restrict__): that path assumes the data is constant for the whole kernel, and under programmatic
// dependent launch a kernel starts while its predecessor is still writing. Such data is read with plain or
// .cg loads after pdl_wait(); only weights and tree buffers (written before any launch) use .nc loads.
MV_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Whether launches use programmatic dependent launch (default on; MV_PDL=0 in the environment turns it off).
bool mv_pdl_enabled();

// Launches `kernel` on `st` with the programmatic-stream-serialization attribute when PDL is enabled.
template <typename... KArgs, typename... Args>
cudaError_t mv_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = mv_pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

MV_DEV void mv_set_error(unsigned int* err, uint32_t site, uint32_t kind) {
  if (err) atomicCAS(err, 0u, (site << 16) | kind);
}
MV_DEV void mv_set_error_detail(unsigned int* err, uint32_t site, uint32_t kind, uint32_t detail) {
  if (err && atomicCAS(err, 0u, (site << 16) | kind) == 0u) err[1] = detail;
}

MV_DEV uint64_t mv_globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound of every spin wait in these kernels (nanoseconds of %globaltimer).
#define MV_WAIT_LIMIT_NS 2000000000ull

MV_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
MV_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MV_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MV_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
MV_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MV_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete; false if limit_ns (default MV_WAIT_LIMIT_NS) passed first.
MV_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = MV_WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = mv_globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (mv_globaltimer() - t0 > limit_ns) return false;
  }
}

// Bounded wait until *p >= target (acquire at GPU scope), the wait on a device counter that other CTAs bump;
// false when limit_ns (default MV_WAIT_LIMIT_NS) passes first.
MV_DEV bool wait_count(const unsigned int* p, unsigned int target, uint64_t limit_ns = MV_WAIT_LIMIT_NS) {
  const uint64_t t0 = mv_globaltimer();
  while (true) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (mv_globaltimer() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
}

// ------------------------------------------------------------------------------------------
// Thread-block clusters: rank, distributed shared memory, remote mbarrier arrives, cluster barrier
// ------------------------------------------------------------------------------------------
MV_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory object in CTA `rank` of this cluster
MV_DEV uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
MV_DEV void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
MV_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded like mbar_wait; acquire at cluster scope (the arrivals come from other CTAs of the cluster)
MV_DEV bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = mv_globaltimer();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (mv_globaltimer() - t0 > MV_WAIT_LIMIT_NS) return false;
  }
}
MV_DEV float2 ld_cluster_f2(uint32_t cluster_addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(cluster_addr) : "memory");
  return v;
}
MV_DEV float4 ld_cluster_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}
// every thread of every CTA of the cluster (all paths reach it: each wait before it is bounded)
MV_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion counted on an mbarrier)
// ------------------------------------------------------------------------------------------
MV_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
MV_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
MV_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Streamed-once data (weights): an L2 policy that evicts these lines first, so that they do not push out data
// that is still to be used (activations, partial sums, the KV cache).
MV_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
MV_DEV void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}
MV_DEV void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                             uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(pol)
      : "memory");
}
// Untiled bulk copy global -> shared of `bytes` (both addresses 16-byte aligned, bytes a multiple of 16),
// counted on `bar` like the tensor copies, with an L2 policy.
MV_DEV void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
MV_DEV void tma_load_4d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2, int c3,
                             uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
      : "memory");
}
MV_DEV void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// ------------------------------------------------------------------------------------------
// small numeric helpers
// ------------------------------------------------------------------------------------------
MV_DEV float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
MV_DEV float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
MV_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}
MV_DEV float silu(float x) { return x / (1.0f + expf(-x)); }

// (value, index) order used by every top-k / argmax here: larger value first, then lower index.
MV_DEV bool vi_better(float va, int ia, float vb, int ib) { return va > vb || (va == vb && ia < ib); }

// Host-side tensor-map encoder (driver entry point fetched through the runtime; no -lcuda).
// Encodes a bf16 / fp32 tiled map with dims[0] innermost. Returns false on failure.
bool mv_encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                    const uint64_t* dims, const uint64_t* strides_bytes /* rank-1 entries */,
                    const uint32_t* box, CUtensorMapSwizzle swizzle);

// Host-side view of a tree handle (defined in tree.cpp).
struct mv_tree {
  int32_t n_nodes, n_paths, depth, topk;
  int32_t* h_tree_indices;
  int32_t* h_position_ids;
  int32_t* h_retrieve;
  int32_t* h_parent;
  uint64_t* h_ancestors;  // [n_nodes][MV_MASK_WORDS]
  int32_t* d_tree_indices;
  int32_t* d_position_ids;
  int32_t* d_retrieve;
  int32_t* d_parent;
  uint64_t* d_ancestors;  // [n_nodes][MV_MASK_WORDS]
  int device;
};
