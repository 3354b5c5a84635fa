// KV compaction after acceptance.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.7 update_inference_inputs(): the accepted path's keys and
// values (rows prefix + nodes[j]) move to rows prefix + j and the length becomes prefix + acc + 1, in every
// layer. One warp owns one (layer, K/V, head) row block: it loads all acc+1 source rows into registers before
// storing any, so a row that is both a source and a destination (e.g. path [0,3,26,56]: source row 3 is the
// destination of j = 3) is read before it is overwritten. Other warps touch other row blocks only.
#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) kv_compact_kernel(uint2* kv, int units, int S_max, int chunks,
                                                                 const int32_t* prefix_dev, int prefix_host,
                                                                 const mv_posterior_result* res, int32_t* cur_len,
                                                                 unsigned int* err) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int prefix = prefix_dev ? *prefix_dev : prefix_host;
  const int acc = res->acc;
  if (acc < 0 || acc > MV_MAX_DEPTH || prefix < 0 || prefix + acc >= S_max) {
    if (threadIdx.x == 0)
      mv_set_error_detail(err, 5, MV_DEVERR_INDEX, ((uint32_t)(acc & 0xff) << 24) | ((uint32_t)prefix & 0xffffff));
    return;
  }
  int src[MV_MAX_DEPTH + 1];
#pragma unroll
  for (int j = 0; j <= MV_MAX_DEPTH; ++j) {
    src[j] = j <= acc ? prefix + res->nodes[j] : -1;
    if (j <= acc && (src[j] < prefix || src[j] >= S_max)) {
      if (lane == 0) mv_set_error_detail(err, 6, MV_DEVERR_INDEX, ((uint32_t)j << 24) | ((uint32_t)src[j] & 0xffffff));
      return;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && cur_len) *cur_len = prefix + acc + 1;
  if (unit >= units) return;
  uint2* base = kv + (size_t)unit * S_max * chunks;
  // chunks <= 64 (D <= 256): at most two 8-byte pieces per lane per row
  uint2 v[MV_MAX_DEPTH + 1][2];
#pragma unroll
  for (int j = 0; j <= MV_MAX_DEPTH; ++j) {
    if (j > acc) break;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int e = lane + 32 * c;
      if (e < chunks) v[j][c] = base[(size_t)src[j] * chunks + e];
    }
  }
#pragma unroll
  for (int j = 0; j <= MV_MAX_DEPTH; ++j) {
    if (j > acc) break;
    if (src[j] == prefix + j) continue;  // already in place
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int e = lane + 32 * c;
      if (e < chunks) base[(size_t)(prefix + j) * chunks + e] = v[j][c];
    }
  }
}

}  // namespace

mv_status launch_kv_compact(mv_bf16* kv, int L, int H, int S_max, int D, const int32_t* d_prefix, int prefix,
                            const mv_posterior_result* d_res, int32_t* d_cur_len, cudaStream_t stream) {
  const int units = L * 2 * H;
  const int blocks = (units + kWarps - 1) / kWarps;
  if (mv_launch(kv_compact_kernel, dim3(blocks), dim3(kWarps * 32), 0, stream, reinterpret_cast<uint2*>(kv), units,
                S_max, D / 4, d_prefix, prefix, d_res, d_cur_len, mv_error_word()) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("kv_compact");
}

extern "C" mv_status kv_compact(mv_bf16* kv, int32_t L, int32_t H, int32_t S_max, int32_t D, int32_t prefix_len,
                                const mv_posterior_result* d_res, int32_t* d_cur_len, mv_stream stream) {
  if (!kv || !d_res) return MV_ERR_INVALID_ARG;
  if (L < 1 || H < 1 || S_max < 1 || D < 4 || (D & 3) || D > 256) return MV_ERR_SHAPE;
  if (prefix_len < 0 || prefix_len >= S_max) return MV_ERR_CAPACITY;
  if (reinterpret_cast<uintptr_t>(kv) & 7) return MV_ERR_SHAPE;
  return launch_kv_compact(kv, L, H, S_max, D, nullptr, prefix_len, d_res, d_cur_len,
                           static_cast<cudaStream_t>(stream));
}
