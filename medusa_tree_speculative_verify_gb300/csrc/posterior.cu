// Posterior evaluation over the tree's logits: greedy or typical acceptance, best path, emitted tokens.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 一.3 Typical acceptance and 二.6 evaluate_posterior().
// The page re-gathers the logits per path ([paths, depth+1, V]) before evaluating; here the per-node statistics
// are computed once per tree node (each node's row is read once) and the per-path walk reads only the
// candidate's own logit.
//
// A cluster of two CTAs per node row (128 CTAs at 64 nodes), each reducing half of it held in registers: the
// half's max and first argmax and, for typical acceptance, the exponentials against the half's own max and their
// sum; the two halves exchange (max, argmax, sum) once over distributed shared memory and merge them by
// rescaling, in rank order, so both CTAs hold the same values; typical acceptance then sums the entropy
// -sum p log(p + 1e-5) the same way. The node's first CTA decides the acceptance of each of the node's children
// (greedy: the child's token is the node's argmax; typical: log p(child's token) > log tau) and leaves a flag
// and the log probability. The last CTA to finish (atomic ticket, no waiting) walks the paths over those flags,
// one thread per path with the path's nodes loaded at the start, picks the best path by warp-shuffle argmax and
// writes the result from that path's thread. Exponentials and logarithms of the typical statistics use the
// hardware approximations (relative error near 2^-22), far below the 1e-3 margins the decisions are held to.
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kBatch = 8;  // float4 per thread per chunk: 512 x 8 x 4 = 16384 logits, half of a row

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

// Partial statistics of one half of a row, pushed into both CTAs of the pair (slot = the sender's rank).
struct Xchg {
  Stat st[2];
  float h[2];
};
MV_DEV void push_f32(float* slot, float v) {  // slot: this CTA's entry of a table of the pair
#pragma unroll
  for (uint32_t c = 0; c < 2; ++c)
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(map_rank(smem_u32(slot), c)), "f"(v) : "memory");
}
MV_DEV void push_i32(int* slot, int v) {
#pragma unroll
  for (uint32_t c = 0; c < 2; ++c)
    asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(map_rank(smem_u32(slot), c)), "r"(v) : "memory");
}

MV_DEV Stat shfl_stat(const Stat& a, int o) {
  Stat b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
  return b;
}
// Merge of the CTA's threads' statistics (warp shuffles, then warp 0 over the warps); every thread gets it.
MV_DEV Stat block_stat(Stat a, Stat* red, float inv_t, bool online) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) a = stat_merge(a, shfl_stat(a, o), inv_t, online);
  if (lane == 0) red[warp] = a;
  __syncthreads();
  if (warp == 0) {
    Stat t = lane < kThreads / 32 ? red[lane] : Stat{-FLT_MAX, 0x7fffffff, 0.0f};
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t = stat_merge(t, shfl_stat(t, o), inv_t, online);
    if (lane == 0) red[kThreads / 32] = t;
  }
  __syncthreads();
  return red[kThreads / 32];
}
MV_DEV float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) red[kThreads / 32] = t;
  }
  __syncthreads();
  const float r = red[kThreads / 32];
  __syncthreads();  // red may be reused
  return r;
}

// Whether path (acc_a, like_a, index a) is chosen over (acc_b, like_b, b): more accepted tokens, then (typical)
// the larger likelihood, then the lower index.
MV_DEV bool path_better(int acc_a, float like_a, int a, int acc_b, float like_b, int b, bool typical) {
  if (acc_a != acc_b) return acc_a > acc_b;
  if (typical && like_a != like_b) return like_a > like_b;
  return a < b;
}

__global__ void __launch_bounds__(kThreads) posterior_kernel(
    const float* logits, int V, int ld, const int32_t* tree_tokens, const int32_t* __restrict__ retrieve,
    const int32_t* __restrict__ parent, int n_nodes, int n_paths, int width, mv_accept_params prm,
    mv_posterior_result* out, float* node_stats_out, int32_t* node_argmax_out, float* ws_stats, int32_t* ws_argmax,
    int32_t* ws_child_ok, float* ws_child_lp, unsigned int* ticket, unsigned int* err, const float2* row_max,
    int n_row_tiles, int row_ld) {
  pdl_trigger();
  // No CTA touches its partner's shared memory before the partner has started: arrive now, wait before the first
  // remote store (the row loads and the local reductions overlap the wait).
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const bool typical = prm.mode == MV_TYPICAL;
  const float inv_t = typical ? 1.0f / prm.temperature : 1.0f;
  const int half = (int)cluster_rank();  // which half of the row this CTA reduces
  const int node = blockIdx.x >> 1;
  const float* row = logits + (size_t)node * ld;
  const int tid = threadIdx.x;
  __shared__ Stat red[kThreads / 32 + 1];
  __shared__ float fred[kThreads / 32 + 1];
  __shared__ Xchg xc;
  __shared__ bool last;
  pdl_wait();

  // This CTA's half of the row (float4 units [v0, v1); the scalar tail beyond 4 (V / 4) belongs to the second
  // half) is held in registers, kBatch float4 per thread, all loaded before any is used.
  // Typical: the max of the half, e = exp((z - m_half) / T) kept in place and their sum; the halves exchange
  // (max, first argmax, sum) once and merge them by rescaling (the same value in both CTAs); then the entropy
  // H = -sum p log(p + 1e-5), p = e exp((m_half - m) / T) / Z, exchanged the same way. Greedy: the max and first
  // argmax only. Halves longer than kBatch x kThreads float4 stream in chunks with an online (rescaled) sum.
  // Greedy with row_max: the LM-head projection already left each 128-row tile's max and first argmax of
  // every token; merging those replaces the pass over the row.
  const bool from_tiles = row_max && !typical;
  const int V4all = from_tiles ? 0 : V >> 2;
  const int hv = (V4all + 1) >> 1;
  const int v0 = half ? hv : 0, v1 = half ? V4all : hv, V4 = v1 - v0;
  const float4* row4 = reinterpret_cast<const float4*>(row) + v0;
  const bool in_regs = hv <= kBatch * kThreads;  // the same in both CTAs: they take the same cluster barriers
  const int t0 = from_tiles ? V : 4 * V4all + tid, t1 = half ? V : 0;  // the scalar tail (second half only)
  float4 buf[kBatch];
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = tid + u * kThreads;
      buf[u] = i < V4 ? __ldcg(row4 + i) : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
    }
  }
  // while the row loads are in flight: this thread's tree node (the children decisions: its parent, token and
  // the token's logit) and, in every pair's first CTA (any may be the last to finish), its path of the walk
  const int my_parent = tid < n_nodes ? __ldg(parent + tid) : -1;
  const bool my_child = my_parent == node && half == 0;
  const int my_tok = my_child ? tree_tokens[tid] : 0;
  const float z_tok = my_child && my_tok >= 0 && my_tok < V ? __ldcg(row + my_tok) : 0.0f;
  int nd[MV_MAX_DEPTH + 1];
#pragma unroll
  for (int j = 0; j <= MV_MAX_DEPTH; ++j)
    nd[j] = (half == 0 && tid < n_paths && j < width) ? __ldg(retrieve + tid * width + j) : -1;

  Stat a{-FLT_MAX, 0x7fffffff, 0.0f};
  if (from_tiles) {
    for (int t = tid + half * kThreads; t < n_row_tiles; t += 2 * kThreads) {
      const float2 e = __ldcg(row_max + (size_t)t * row_ld + node);
      a = stat_merge(a, Stat{e.x, __float_as_int(e.y), 0.0f}, 1.0f, false);
    }
  }
  const bool online = typical && !in_regs;
  for (int c0 = 0; c0 < V4; c0 += kBatch * kThreads) {
    if (!in_regs) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = c0 + tid + u * kThreads;
        buf[u] = i < V4 ? __ldcg(row4 + i) : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = c0 + tid + u * kThreads;
      if (i < V4) {
        const int k = 4 * (v0 + i);
        stat_push(a, buf[u].x, k + 0, inv_t, online);
        stat_push(a, buf[u].y, k + 1, inv_t, online);
        stat_push(a, buf[u].z, k + 2, inv_t, online);
        stat_push(a, buf[u].w, k + 3, inv_t, online);
      }
    }
  }
  for (int i = t0; i < t1; i += kThreads) stat_push(a, __ldcg(row + i), i, inv_t, online);
  Stat mine = block_stat(a, red, inv_t, online);
  const float m_half = mine.m;
  if (typical && in_regs) {  // the exponentials against this half's max, in place, and their sum
    float z = 0.0f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (tid + u * kThreads < V4) {
        buf[u].x = __expf((buf[u].x - m_half) * inv_t);
        buf[u].y = __expf((buf[u].y - m_half) * inv_t);
        buf[u].z = __expf((buf[u].z - m_half) * inv_t);
        buf[u].w = __expf((buf[u].w - m_half) * inv_t);
        z += (buf[u].x + buf[u].y) + (buf[u].z + buf[u].w);
      }
    }
    for (int i = t0; i < t1; i += kThreads) z += __expf((__ldcg(row + i) - m_half) * inv_t);
    mine.s = block_sum(z, fred);
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // the partner has started
  if (tid == 0) {
    push_f32(&xc.st[half].m, mine.m);
    push_i32(&xc.st[half].i, mine.i);
    push_f32(&xc.st[half].s, mine.s);
  }
  cluster_sync_all();
  const Stat T = stat_merge(xc.st[0], xc.st[1], inv_t, typical);

  float H = 0.0f, tau = 0.0f;
  if (typical) {
    const float inv_s = 1.0f / T.s;
    float h = 0.0f;
    auto ent = [&](float p) { h += p * __logf(p + 1e-5f); };
    if (in_regs) {
      const float c = __expf((m_half - T.m) * inv_t) * inv_s;  // p = e c
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (tid + u * kThreads < V4) {
          ent(buf[u].x * c);
          ent(buf[u].y * c);
          ent(buf[u].z * c);
          ent(buf[u].w * c);
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
    for (int i = t0; i < t1; i += kThreads) ent(__expf((__ldcg(row + i) - T.m) * inv_t) * inv_s);
    h = block_sum(h, fred);
    if (tid == 0) push_f32(&xc.h[half], h);
    cluster_sync_all();
    H = -(xc.h[0] + xc.h[1]);
    tau = fminf(prm.eps, prm.delta * expf(-H));
  }
  // after the last exchange no CTA reads its partner's shared memory: the second CTA of the pair is done
  if (half) return;

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
  // the acceptance of this node's children (thread c decides child c): their candidate tokens against this
  // node's distribution
  if (my_child) {
    int ok = 0;
    float lp = 0.0f;
    if (my_tok < 0 || my_tok >= V) {
      mv_set_error(err, 3, MV_DEVERR_INDEX);
    } else if (typical) {
      lp = (z_tok - T.m) * inv_t - logf(T.s);  // log p(tok) under softmax(z / T)
      ok = lp > logf(tau);
    } else {
      ok = my_tok == T.i;
    }
    ws_child_ok[tid] = ok;
    ws_child_lp[tid] = lp;
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
  int acc = -1;  // threads without a path lose every comparison
  float like = 0.0f;
  bool bad = false;
  if (tid < n_paths) {
    int okv[MV_MAX_DEPTH + 1];
    float lpv[MV_MAX_DEPTH + 1];
#pragma unroll
    for (int j = 1; j <= MV_MAX_DEPTH; ++j) {  // the flags and log probabilities, all loads in flight at once
      const bool in = nd[j] >= 0 && nd[j] < n_nodes;
      bad |= nd[j] >= n_nodes;
      okv[j] = in ? __ldcg(ws_child_ok + nd[j]) : 0;
      lpv[j] = in ? __ldcg(ws_child_lp + nd[j]) : 0.0f;
    }
    acc = 0;
    bool alive = true;
#pragma unroll
    for (int j = 1; j <= MV_MAX_DEPTH; ++j) {
      alive = alive && j < width && nd[j] >= 0 && okv[j];
      if (alive) {
        ++acc;
        like += lpv[j];
      }
    }
  }
  if (__syncthreads_or(bad) && tid == 0) mv_set_error(err, 3, MV_DEVERR_INDEX);
  // best path: warp argmax, then warp 0 over the warps' winners
  __shared__ int s_acc[kThreads / 32], s_idx[kThreads / 32];
  __shared__ float s_like[kThreads / 32];
  __shared__ int s_best;
  {
    const int lane = tid & 31, warp = tid >> 5;
    int ba = acc, bi = tid;
    float bl = like;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const int oa = __shfl_xor_sync(0xffffffffu, ba, o), oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (path_better(oa, ol, oi, ba, bl, bi, typical)) {
        ba = oa;
        bi = oi;
        bl = ol;
      }
    }
    if (lane == 0) {
      s_acc[warp] = ba;
      s_idx[warp] = bi;
      s_like[warp] = bl;
    }
    __syncthreads();
    if (warp == 0) {
      ba = lane < kThreads / 32 ? s_acc[lane] : -1;
      bi = lane < kThreads / 32 ? s_idx[lane] : 0x7fffffff;
      bl = lane < kThreads / 32 ? s_like[lane] : 0.0f;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const int oa = __shfl_xor_sync(0xffffffffu, ba, o), oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
        if (path_better(oa, ol, oi, ba, bl, bi, typical)) {
          ba = oa;
          bi = oi;
          bl = ol;
        }
      }
      if (lane == 0) {
        s_best = ba > 0 ? bi : 0;  // nothing accepted: path 0 (its root only)
        *ticket = 0u;              // leave the counter zeroed for the next call
      }
    }
    __syncthreads();
  }
  // the result, written by the best path's own thread (its node list is in registers)
  if (tid == s_best) {
    const int n_acc = acc > 0 ? acc : 0;
    int nn = nd[0];
    int tk[MV_MAX_DEPTH + 1];
#pragma unroll
    for (int j = 0; j <= MV_MAX_DEPTH; ++j) {
      if (j == n_acc) nn = nd[j];
      tk[j] = j <= n_acc && nd[j] >= 0 ? tree_tokens[nd[j]] : -1;
    }
    const int next_root = __ldcg(ws_argmax + nn);
#pragma unroll
    for (int j = 0; j <= MV_MAX_DEPTH; ++j) {
      out->nodes[j] = j <= n_acc ? nd[j] : -1;
      out->tokens[j] = tk[j];
    }
    out->best = tid;
    out->acc = n_acc;
    out->n_tokens = n_acc + 1;
    out->next_node = nn;
    out->next_root = next_root;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * t->n_nodes);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;  // one pair of CTAs per node row
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = mv_pdl_enabled() ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, posterior_kernel, logits, V, ld, d_tree_tokens, t->d_retrieve, t->d_parent,
                         t->n_nodes, t->n_paths, t->depth + 1, prm, d_out, d_stats, d_argmax, ws_stats, ws_arg, ws_ok,
                         ws_lp, ticket, mv_error_word(), row_max, n_row_tiles, row_ld) != cudaSuccess)
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
