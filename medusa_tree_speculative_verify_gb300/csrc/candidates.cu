// Candidate gather into the static tree.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.4 generate_candidates(): the candidate list is the root
// token followed by every head's top-k (head-major); tree node i takes candidates[tree_indices[i]]; the
// per-path view cart_candidates reads the node tokens through retrieve, with token 0 where retrieve is -1.
// A tree has at most 64 nodes, so one CTA does all of it with no synchronisation: each output is read
// straight from the candidate list.
#include "common.cuh"
#include "kernels.cuh"

namespace {

__device__ __forceinline__ int candidate(int idx, const int32_t* root, const int32_t* head_topk, int topk, int ld) {
  if (idx == 0) return root[0];
  const int k = (idx - 1) / topk, r = (idx - 1) % topk;
  return head_topk[k * ld + r];
}

__global__ void __launch_bounds__(128) build_candidates_kernel(const int32_t* root, const int32_t* head_topk,
                                                               int topk, int ld,
                                                               const int32_t* __restrict__ tree_indices,
                                                               const int32_t* __restrict__ retrieve, int n_nodes,
                                                               int n_cart, int32_t* tree_tokens, int32_t* cart) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < n_nodes; i += blockDim.x)
    tree_tokens[i] = candidate(tree_indices[i], root, head_topk, topk, ld);
  if (cart) {
    for (int e = threadIdx.x; e < n_cart; e += blockDim.x) {
      const int node = retrieve[e];
      cart[e] = node < 0 ? 0 : candidate(tree_indices[node], root, head_topk, topk, ld);
    }
  }
}

}  // namespace

mv_status launch_build_candidates(const int32_t* d_root, const int32_t* d_head_topk, int ld_topk, const mv_tree* t,
                                  int32_t* d_tree_tokens, int32_t* d_cart, cudaStream_t stream) {
  if (mv_launch(build_candidates_kernel, dim3(1), dim3(128), 0, stream, d_root, d_head_topk, t->topk, ld_topk,
                t->d_tree_indices, t->d_retrieve, t->n_nodes, t->n_paths * (t->depth + 1), d_tree_tokens,
                d_cart) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("build_candidates");
}

extern "C" mv_status build_candidates(const int32_t* d_root, const int32_t* d_head_topk, int32_t K,
                                      int32_t ld_topk, const mv_tree* tree, int32_t* d_tree_tokens,
                                      int32_t* d_cart, mv_stream stream) {
  if (!d_root || !d_head_topk || !tree || !d_tree_tokens) return MV_ERR_INVALID_ARG;
  if (!tree->d_tree_indices) return MV_ERR_CUDA;
  if (K < tree->depth || ld_topk < tree->topk) return MV_ERR_SHAPE;
  return launch_build_candidates(d_root, d_head_topk, ld_topk, tree, d_tree_tokens, d_cart,
                                 static_cast<cudaStream_t>(stream));
}
