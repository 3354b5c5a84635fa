// Posterior evaluation over the tree's logits: greedy or typical acceptance, best path, emitted tokens.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.3 Typical acceptance and 二.6 evaluate_posterior().
// The page re-gathers the logits per path ([paths, depth+1, V]) before evaluating; here the per-node statistics
// are computed once per tree node (each node's row is read once) and the per-path walk reads only the
// candidate's own logit.
//
// One CTA per node row: pass 1 (max, first argmax; the softmax normaliser of z/T by online rescaling when the
// row does not fit in registers), pass 2 (typical: the exponentials and their sum), pass 3 (typical: the
// entropy). The node's CTA then decides the acceptance of each of the node's children in the tree (greedy: the
// child's token is the node's argmax; typical: log p(child's token) > log tau) and leaves a flag and the log
// probability. The last CTA to finish (atomic ticket, no waiting) walks the paths over those flags and writes
// the result. Exponentials and logarithms of the typical statistics use the hardware approximations (relative
// error near 2^-22), far below the 1e-3 margins the decisions are held to.
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kBatch = 16;  // float4 per thread per chunk: 512 x 16 x 4 = 32768 logits

struct Stat {
  float m;  // running max of z
  int i;    // first index of the max
  float s;  // sum of exp((z - m) / T)
};

MV_DEV void stat_push(Stat& a, float z, int idx, float inv_t, bool typical) {
  if (z > a.m) {
    if (typical) a.s = a.s * expf((a.m - z) * inv_t) + 1.0f;
    a.m = z;
    a.i = idx;
  } else {
    if (typical) a.s += expf((z - a.m) * inv_t);
    if (z == a.m && idx < a.i) a.i = idx;
  }
}

MV_DEV Stat stat_merge(Stat a, Stat b, float inv_t, bool typical) {
  Stat r;
  if (b.m > a.m || (b.m == a.m && b.i < a.i)) {
    r.m = b.m;
    r.i = b.i;
  } else {
    r.m = a.m;
    r.i = a.i;
  }
  if (typical) {
    const float sa = a.s == 0.0f ? 0.0f : a.s * expf((a.m - r.m) * inv_t);
    const float sb = b.s == 0.0f ? 0.0f : b.s * expf((b.m - r.m) * inv_t);
    r.s = sa + sb;
  } else {
    r.s = 0.0f;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads) posterior_kernel(
    const float* logits, int V, int ld, const int32_t* tree_tokens, const int32_t* __restrict__ retrieve,
    const int32_t* __restrict__ parent, int n_nodes, int n_paths, int width, mv_accept_params prm,
    mv_posterior_result* out, float* node_stats_out, int32_t* node_argmax_out, float* ws_stats, int32_t* ws_argmax,
    int32_t* ws_child_ok, float* ws_child_lp, unsigned int* ticket, unsigned int* err, const float2* row_max,
    int n_row_tiles, int row_ld) {
  pdl_trigger();
  pdl_wait();
  const bool typical = prm.mode == MV_TYPICAL;
  const float inv_t = typical ? 1.0f / prm.temperature : 1.0f;
  const int node = blockIdx.x;
  const float* row = logits + (size_t)node * ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ Stat red[kThreads / 32];
  __shared__ float fred[kThreads / 32];
  __shared__ Stat tot;
  __shared__ bool last;

  // The row (32000 logits) is held in registers, kBatch float4 per thread, all loaded before any is used.
  // pass 1: max and first argmax; pass 2 (typical): e = exp((z - max) / T) kept in place, Z = sum e;
  // pass 3 (typical): H = -sum p log(p + 1e-5) with p = e / Z. Rows longer than 32768 stream in chunks with
  // an online (rescaled) normaliser instead.
  // Greedy with row_max: the LM-head projection already left each 128-row tile's max and first argmax of
  // every token; merging those replaces the pass over the row.
  const bool from_tiles = row_max && !typical;
  const int V4 = from_tiles ? 0 : V >> 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  const bool in_regs = V4 <= kBatch * kThreads;
  float4 buf[kBatch];
  Stat a{-FLT_MAX, 0x7fffffff, 0.0f};
  if (from_tiles) {
    for (int t = tid; t < n_row_tiles; t += kThreads) {
      const float2 e = __ldcg(row_max + (size_t)t * row_ld + node);
      a = stat_merge(a, Stat{e.x, __float_as_int(e.y), 0.0f}, 1.0f, false);
    }
  }
  for (int c0 = 0; c0 < V4; c0 += kBatch * kThreads) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = c0 + tid + u * kThreads;
      buf[u] = i < V4 ? __ldcg(row4 + i) : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
    }
    const bool online = typical && !in_regs;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = c0 + tid + u * kThreads;
      if (i < V4) {
        stat_push(a, buf[u].x, 4 * i + 0, inv_t, online);
        stat_push(a, buf[u].y, 4 * i + 1, inv_t, online);
        stat_push(a, buf[u].z, 4 * i + 2, inv_t, online);
        stat_push(a, buf[u].w, 4 * i + 3, inv_t, online);
      }
    }
  }
  if (!from_tiles)
    for (int i = 4 * V4 + tid; i < V; i += kThreads) stat_push(a, __ldcg(row + i), i, inv_t, typical && !in_regs);
  const bool online = typical && !in_regs;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    Stat b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    a = stat_merge(a, b, inv_t, online);
  }
  if (lane == 0) red[warp] = a;
  __syncthreads();
  if (tid == 0) {
    Stat t = red[0];
    for (int w = 1; w < kThreads / 32; ++w) t = stat_merge(t, red[w], inv_t, online);
    tot = t;
  }
  __syncthreads();
  Stat T = tot;

  float H = 0.0f, tau = 0.0f;
  if (typical) {
    auto block_sum = [&](float v) {
      __syncthreads();
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) fred[warp] = v;
      __syncthreads();
      float s = 0.0f;
      for (int w = 0; w < kThreads / 32; ++w) s += fred[w];
      return s;
    };
    if (in_regs) {  // pass 2: exponentials in place and their sum
      float z = 0.0f;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (tid + u * kThreads < V4) {
          buf[u].x = __expf((buf[u].x - T.m) * inv_t);
          buf[u].y = __expf((buf[u].y - T.m) * inv_t);
          buf[u].z = __expf((buf[u].z - T.m) * inv_t);
          buf[u].w = __expf((buf[u].w - T.m) * inv_t);
          z += (buf[u].x + buf[u].y) + (buf[u].z + buf[u].w);
        }
      }
      for (int i = 4 * V4 + tid; i < V; i += kThreads) z += __expf((__ldcg(row + i) - T.m) * inv_t);
      T.s = block_sum(z);
    }
    const float inv_s = 1.0f / T.s;
    float h = 0.0f;
    auto ent = [&](float p) { h += p * __logf(p + 1e-5f); };
    if (in_regs) {  // pass 3
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (tid + u * kThreads < V4) {
          ent(buf[u].x * inv_s);
          ent(buf[u].y * inv_s);
          ent(buf[u].z * inv_s);
          ent(buf[u].w * inv_s);
        }
      }
    } else {
      for (int c0 = 0; c0 < V4; c0 += kBatch * kThreads) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int i = c0 + tid + u * kThreads;
          buf[u] = i < V4 ? __ldcg(row4 + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (c0 + tid + u * kThreads < V4) {
            ent(__expf((buf[u].x - T.m) * inv_t) * inv_s);
            ent(__expf((buf[u].y - T.m) * inv_t) * inv_s);
            ent(__expf((buf[u].z - T.m) * inv_t) * inv_s);
            ent(__expf((buf[u].w - T.m) * inv_t) * inv_s);
          }
        }
      }
    }
    for (int i = 4 * V4 + tid; i < V; i += kThreads) ent(__expf((__ldcg(row + i) - T.m) * inv_t) * inv_s);
    H = -block_sum(h);
    tau = fminf(prm.eps, prm.delta * expf(-H));
  }

  if (tid == 0) {
    ws_stats[node * 4 + 0] = T.m;
    ws_stats[node * 4 + 1] = T.s;
    ws_stats[node * 4 + 2] = H;
    ws_stats[node * 4 + 3] = tau;
    ws_argmax[node] = T.i;
    if (node_stats_out) {
      node_stats_out[node * 4 + 0] = T.m;
      node_stats_out[node * 4 + 1] = typical ? logf(T.s) : 0.0f;
      node_stats_out[node * 4 + 2] = H;
      node_stats_out[node * 4 + 3] = tau;
    }
    if (node_argmax_out) node_argmax_out[node] = T.i;
  }
  // the acceptance of this node's children: their candidate tokens against this node's distribution
  {
    const float lnz = typical ? logf(T.s) : 0.0f;
    const float ltau = typical ? logf(tau) : 0.0f;
    for (int c = tid; c < n_nodes; c += kThreads) {
      if (__ldg(parent + c) != node) continue;
      const int tok = tree_tokens[c];
      int ok = 0;
      float lp = 0.0f;
      if (tok < 0 || tok >= V) {
        mv_set_error(err, 3, MV_DEVERR_INDEX);
      } else if (typical) {
        lp = (__ldcg(row + tok) - T.m) * inv_t - lnz;  // log p(tok) under softmax(z / T)
        ok = lp > ltau;
      } else {
        ok = tok == T.i;
      }
      ws_child_ok[c] = ok;
      ws_child_lp[c] = lp;
    }
  }
  __syncthreads();  // every child decision of this node is written
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(ticket, 1u) == (unsigned)(n_nodes - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  // ---- last CTA: walk every path (one thread per path), then pick the best
  __shared__ int s_acc[MV_MAX_NODES];
  __shared__ float s_like[MV_MAX_NODES];
  __shared__ int s_bad;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (tid < n_paths) {
    // the path's nodes, then their acceptance flags and log probabilities, each batch of loads in flight at once
    const int32_t* r = retrieve + tid * width;
    int nd[MV_MAX_DEPTH + 1], okv[MV_MAX_DEPTH + 1];
    float lpv[MV_MAX_DEPTH + 1];
#pragma unroll
    for (int j = 0; j <= MV_MAX_DEPTH; ++j) nd[j] = j < width ? __ldg(r + j) : -1;
#pragma unroll
    for (int j = 1; j <= MV_MAX_DEPTH; ++j) {
      const bool in = nd[j] >= 0 && nd[j] < n_nodes;
      if (nd[j] >= n_nodes) s_bad = 1;
      okv[j] = in ? __ldcg(ws_child_ok + nd[j]) : 0;
      lpv[j] = in ? __ldcg(ws_child_lp + nd[j]) : 0.0f;
    }
    int acc = 0;
    float like = 0.0f;
    for (int j = 1; j < width && nd[j] >= 0 && okv[j]; ++j) {
      ++acc;
      like += lpv[j];
    }
    s_acc[tid] = acc;
    s_like[tid] = like;
  }
  __shared__ int s_best, s_bacc;
  __syncthreads();
  if (tid == 0) {
    if (s_bad) mv_set_error(err, 3, MV_DEVERR_INDEX);
    int best = 0;
    for (int p = 1; p < n_paths; ++p) {
      if (s_acc[p] > s_acc[best] || (typical && s_acc[p] == s_acc[best] && s_like[p] > s_like[best])) best = p;
    }
    const int acc = s_acc[best] > 0 ? s_acc[best] : 0;
    if (acc == 0) best = 0;
    s_best = best;
    s_bacc = acc;
    *ticket = 0u;  // leave the counter zeroed for the next call
  }
  __syncthreads();
  // the result, one thread per field (the loads of the best path's nodes and tokens in flight together)
  const int best = s_best, acc = s_bacc;
  const int32_t* r = retrieve + best * width;
  if (tid <= MV_MAX_DEPTH) {
    const int nd = tid <= acc ? __ldg(r + tid) : -1;
    out->nodes[tid] = nd;
    out->tokens[tid] = nd >= 0 ? tree_tokens[nd] : -1;
  } else if (tid == 32) {
    const int nn = __ldg(r + acc);
    out->best = best;
    out->acc = acc;
    out->n_tokens = acc + 1;
    out->next_node = nn;
    out->next_root = __ldcg(ws_argmax + nn);
  }
}

}  // namespace

// ticket, then per node: stats [4], argmax, child flag, child log probability
size_t posterior_ws_bytes(int n_nodes) { return (size_t)n_nodes * 7 * sizeof(float) + 64; }

mv_status launch_posterior(const float* logits, int V, int ld, const int32_t* d_tree_tokens, const mv_tree* t,
                           mv_accept_params prm, mv_posterior_result* d_out, float* d_stats, int32_t* d_argmax,
                           void* ws, cudaStream_t stream, const float2* row_max, int n_row_tiles, int row_ld) {
  char* w = static_cast<char*>(ws);
  unsigned int* ticket = reinterpret_cast<unsigned int*>(w);
  float* ws_stats = reinterpret_cast<float*>(w + 64);
  int32_t* ws_arg = reinterpret_cast<int32_t*>(w + 64 + (size_t)t->n_nodes * 4 * sizeof(float));
  int32_t* ws_ok = ws_arg + t->n_nodes;
  float* ws_lp = reinterpret_cast<float*>(ws_ok + t->n_nodes);
  if (mv_launch(posterior_kernel, dim3(t->n_nodes), dim3(kThreads), 0, stream, logits, V, ld, d_tree_tokens,
                t->d_retrieve, t->d_parent, t->n_nodes, t->n_paths, t->depth + 1, prm, d_out, d_stats, d_argmax,
                ws_stats, ws_arg, ws_ok, ws_lp, ticket, mv_error_word(), row_max, n_row_tiles, row_ld) != cudaSuccess)
    return MV_ERR_CUDA;
  return mv_last_launch("evaluate_posterior");
}

extern "C" mv_status evaluate_posterior_workspace(int32_t n_nodes, size_t* bytes) {
  if (!bytes || n_nodes < 1 || n_nodes > MV_MAX_NODES) return MV_ERR_INVALID_ARG;
  *bytes = posterior_ws_bytes(n_nodes);
  return MV_OK;
}

extern "C" mv_status evaluate_posterior(const float* logits, int32_t V, int32_t ld, const int32_t* d_tree_tokens,
                                        const mv_tree* tree, mv_accept_params params, mv_posterior_result* d_out,
                                        float* d_node_stats, int32_t* d_node_argmax, void* workspace,
                                        size_t ws_bytes, mv_stream stream) {
  if (!logits || !d_tree_tokens || !tree || !d_out || !workspace) return MV_ERR_INVALID_ARG;
  if (!tree->d_retrieve || !tree->d_parent) return MV_ERR_CUDA;
  if (V < 2 || ld < V || (ld & 3) || (reinterpret_cast<uintptr_t>(logits) & 15)) return MV_ERR_SHAPE;
  if (params.mode != MV_GREEDY && params.mode != MV_TYPICAL) return MV_ERR_INVALID_ARG;
  if (params.mode == MV_TYPICAL && !(params.temperature > 0.0f)) return MV_ERR_INVALID_ARG;
  if (ws_bytes < posterior_ws_bytes(tree->n_nodes)) return MV_ERR_CAPACITY;
  return launch_posterior(logits, V, ld, d_tree_tokens, tree, params, d_out, d_node_stats, d_node_argmax,
                          workspace, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------------------------
// Allocation-free variant. Some callers cannot call cudaMalloc: code that runs inside another runtime's memory
// manager (which owns every device allocation and forbids raw ones), or a serving loop that must not touch the
// device allocator once it is running (cudaMalloc may synchronise the device and serialises on a global lock).
// They get the same posterior with its scratch in a fixed array that is part of the library's device image:
// every GPU that loads the library holds these bytes until the process exits.
// ------------------------------------------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxNodes = MV_NOALLOC_MAX_NODES;
constexpr size_t kNoAllocScratchBytes = 2048;  // >= posterior_ws_bytes(kNoAllocMaxNodes) = 64 * 28 + 64 = 1856
static __device__ __align__(256) unsigned char g_posterior_scratch[kNoAllocScratchBytes];

// Device address of g_posterior_scratch on the current device, looked up once per device with that device
// current. In host code the symbol's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress; it is then passed to the kernel like any workspace pointer.
void* noalloc_scratch() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_posterior_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" mv_status evaluate_posterior_noalloc(const float* logits, int32_t V, int32_t ld,
                                                const int32_t* d_tree_tokens, const mv_tree* tree,
                                                mv_accept_params params, mv_posterior_result* d_out,
                                                float* d_node_stats, int32_t* d_node_argmax, mv_stream stream) {
  if (!logits || !d_tree_tokens || !tree || !d_out) return MV_ERR_INVALID_ARG;
  if (!tree->d_retrieve || !tree->d_parent) return MV_ERR_CUDA;
  if (V < 2 || ld < V || (ld & 3) || (reinterpret_cast<uintptr_t>(logits) & 15)) return MV_ERR_SHAPE;
  if (params.mode != MV_GREEDY && params.mode != MV_TYPICAL) return MV_ERR_INVALID_ARG;
  if (params.mode == MV_TYPICAL && !(params.temperature > 0.0f)) return MV_ERR_INVALID_ARG;
  if (tree->n_nodes > kNoAllocMaxNodes || posterior_ws_bytes(tree->n_nodes) > kNoAllocScratchBytes)
    return MV_ERR_CAPACITY;  // more nodes than the fixed scratch array holds
  void* scratch = noalloc_scratch();
  if (!scratch) return MV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the last call left; the completion counter at its start must begin at zero.
  if (cudaMemsetAsync(scratch, 0, 64, st) != cudaSuccess) return MV_ERR_CUDA;
  return launch_posterior(logits, V, ld, d_tree_tokens, tree, params, d_out, d_node_stats, d_node_argmax, scratch,
                          st);
}
