// One-time weight layout for the projection kernel: [row tile][k-block][tile rows][64].
//
// The projection kernel reads one (tile rows x 64) block of a weight matrix per pipeline stage. In the
// row-major layout such a block is `tile rows` separate 128-byte pieces 2*K bytes apart; in this layout it
// is one contiguous run of tile_rows * 128 bytes, and the k-blocks one CTA streams follow each other in
// memory. The values are unchanged (ragged edges are padded with zeros).
#include <algorithm>

#include "common.cuh"

namespace {

__global__ void __launch_bounds__(256) pack_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int M,
                                                   int K, int tr, int n_kb, size_t total_chunks) {
  // one thread per 16-byte chunk (8 bf16) of the packed output
  for (size_t c = blockIdx.x * (size_t)blockDim.x + threadIdx.x; c < total_chunks;
       c += (size_t)gridDim.x * blockDim.x) {
    const int q = (int)(c & 7);            // chunk within the 64-element row piece
    const size_t rest = c >> 3;
    const int r = (int)(rest % tr);        // row within the tile
    const size_t tb = rest / tr;           // tile-block index = tm * n_kb + kb
    const int kb = (int)(tb % n_kb);
    const int tm = (int)(tb / n_kb);
    const int row = tm * tr + r, k = kb * 64 + q * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < M && k < K) v = src[((size_t)row * K + k) >> 3];
    dst[c] = v;
  }
}

}  // namespace

extern "C" mv_status mv_packed_weight_bytes(int32_t M, int32_t K, int32_t tile_rows, size_t* bytes) {
  if (!bytes || M < 1 || K < 8 || (K & 7) || (tile_rows != 64 && tile_rows != 128)) return MV_ERR_SHAPE;
  const size_t n_tm = (M + tile_rows - 1) / tile_rows, n_kb = (K + 63) / 64;
  *bytes = n_tm * n_kb * tile_rows * 64 * 2;
  return MV_OK;
}

extern "C" mv_status mv_pack_weight(const mv_bf16* src, mv_bf16* dst, int32_t M, int32_t K, int32_t tile_rows,
                                    mv_stream stream) {
  size_t bytes = 0;
  mv_status s = mv_packed_weight_bytes(M, K, tile_rows, &bytes);
  if (s != MV_OK) return s;
  if (!src || !dst) return MV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) return MV_ERR_SHAPE;
  const size_t chunks = bytes / 16;
  const int n_kb = (K + 63) / 64;
  const int blocks = (int)std::min<size_t>((chunks + 255) / 256, (size_t)mv_sm_count() * 16);
  pack_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<const uint4*>(src),
                                                                       reinterpret_cast<uint4*>(dst), M, K,
                                                                       tile_rows, n_kb, chunks);
  return mv_last_launch("pack_weight");
}
