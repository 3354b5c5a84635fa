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

#include "attn_core.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace {

using attn::kKeys;
using attn::kMaxSplits;
using attn::kMinTiles;
using attn::kRows;
using attn::kThreads;
using AttnArgs = attn::Args;

// The standalone launch: the 128 threads are the whole CTA, so the cluster-wide steps are cluster barriers.
struct ClusterSync {
  MV_DEV void ready() { cluster_sync_all(); }
  MV_DEV void done() { cluster_sync_all(); }
};

template <int D>
__global__ void __launch_bounds__(kThreads) tree_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap,
                                                             const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[attn::kStages];
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < attn::kStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // q, the cache and the prefix length come from earlier kernels
  const int seq = a.seq_rows ? (int)blockIdx.z : 0;
  const int row0 = a.seq_rows ? 0 : (int)blockIdx.z * kRows;  // blocks of 64 query rows of one tree
  ClusterSync sync;
  attn::head<D>(a, &kmap, &vmap, smem, full, (int)blockIdx.x, (int)blockIdx.y, seq, row0, (int)threadIdx.x, sync);
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
  const size_t core = D == 16 ? attn::smem_bytes<16>() : D == 32 ? attn::smem_bytes<32>()
                      : D == 64 ? attn::smem_bytes<64>() : attn::smem_bytes<128>();
  return 1024 + core;
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
  if ((D == 64 || D == 128) && S_max > kAttnLongCacheRows)  // long caches: the tensor-memory kernel
    return launch_tree_attention_tc(kmap, vmap, plane_k, plane_v, q, H, D, S_max, d_prefix, prefix, max_prefix, t,
                                    n, scale, out, stream, nseq, seq_planes);
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
