// Static token tree: choice list -> tree_indices, position ids, retrieve rows, parents, ancestor words.
//
// "大模型推理 memory bandwidth bound (5) - Medusa", 二.2 generate_medusa_buffers(): the tree is fixed before
// decoding and turned once into index buffers that stay resident on the device (also "OpenPangu7B-with-Medusa"
// README, 4: static tree tensors, fixed mask). Node order: root, then the rank tuples by (length, tuple).
// The attention mask is kept as MV_MASK_WORDS 64-bit words per node (bit j of the row = node j is an
// ancestor-or-self).
#include <algorithm>
#include <map>
#include <vector>

#include "common.cuh"

namespace {

using Path = std::vector<int32_t>;

bool path_less(const Path& a, const Path& b) {
  if (a.size() != b.size()) return a.size() < b.size();
  return a < b;
}

template <typename T>
mv_status upload(T** dst, const std::vector<T>& src) {
  *dst = nullptr;
  size_t bytes = std::max<size_t>(src.size(), 1) * sizeof(T);
  if (cudaMalloc(reinterpret_cast<void**>(dst), bytes) != cudaSuccess) return MV_ERR_CUDA;
  if (!src.empty() && cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
    return MV_ERR_CUDA;
  return MV_OK;
}

template <typename T>
T* host_copy(const std::vector<T>& v) {
  T* p = new T[std::max<size_t>(v.size(), 1)];
  std::copy(v.begin(), v.end(), p);
  return p;
}

}  // namespace

extern "C" mv_status mv_tree_create(const int32_t* ranks, const int32_t* lens, int32_t n_choices, int32_t topk,
                                    mv_tree** out) {
  if (!out || n_choices < 0 || topk < 1 || (n_choices > 0 && (!ranks || !lens))) return MV_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_choices + 1 > MV_MAX_NODES) return MV_ERR_TREE;

  std::vector<Path> paths;
  size_t off = 0;
  for (int32_t c = 0; c < n_choices; ++c) {
    if (lens[c] < 1 || lens[c] > MV_MAX_DEPTH) return MV_ERR_TREE;
    Path p(ranks + off, ranks + off + lens[c]);
    off += lens[c];
    for (int32_t r : p)
      if (r < 0 || r >= topk) return MV_ERR_TREE;
    paths.push_back(p);
  }
  std::sort(paths.begin(), paths.end(), path_less);
  if (std::adjacent_find(paths.begin(), paths.end()) != paths.end()) return MV_ERR_TREE;

  const int n = n_choices + 1;
  std::map<Path, int> node_of;
  node_of[Path()] = 0;
  for (int i = 0; i < n_choices; ++i) node_of[paths[i]] = i + 1;

  std::vector<int32_t> tree_indices(n), position_ids(n), parent(n);
  std::vector<uint64_t> anc((size_t)n * MV_MASK_WORDS, 0ull);
  tree_indices[0] = 0;
  position_ids[0] = 0;
  parent[0] = -1;
  anc[0] = 1ull;  // the root sees itself
  int depth = 0;
  for (int i = 1; i < n; ++i) {
    const Path& p = paths[i - 1];
    Path up(p.begin(), p.end() - 1);
    auto it = node_of.find(up);
    if (it == node_of.end()) return MV_ERR_TREE;  // not prefix-closed
    parent[i] = it->second;
    position_ids[i] = (int32_t)p.size();
    tree_indices[i] = 1 + topk * ((int32_t)p.size() - 1) + p.back();
    for (int w = 0; w < MV_MASK_WORDS; ++w)  // parents precede children in this order
      anc[(size_t)i * MV_MASK_WORDS + w] = anc[(size_t)parent[i] * MV_MASK_WORDS + w];
    anc[(size_t)i * MV_MASK_WORDS + (i >> 6)] |= 1ull << (i & 63);
    depth = std::max(depth, (int)p.size());
  }

  // leaves: nodes that are nobody's parent; one retrieve row each, in descending node order
  std::vector<char> has_child(n, 0);
  for (int i = 1; i < n; ++i) has_child[parent[i]] = 1;
  std::vector<int32_t> retrieve;
  int n_paths = 0;
  const int w = depth + 1;
  for (int i = n - 1; i >= 0; --i) {
    if (has_child[i]) continue;
    std::vector<int32_t> row(w, -1);
    for (int v = i; v >= 0; v = parent[v]) row[position_ids[v]] = v;
    retrieve.insert(retrieve.end(), row.begin(), row.end());
    ++n_paths;
  }

  mv_tree* t = new mv_tree();
  t->n_nodes = n;
  t->n_paths = n_paths;
  t->depth = depth;
  t->topk = topk;
  t->h_tree_indices = host_copy(tree_indices);
  t->h_position_ids = host_copy(position_ids);
  t->h_retrieve = host_copy(retrieve);
  t->h_parent = host_copy(parent);
  t->h_ancestors = host_copy(anc);
  // Without a CUDA device the handle keeps the host copies only (device pointers stay NULL); the kernel
  // entry points then refuse it with MV_ERR_CUDA. This keeps the host logic usable on GPU-less machines.
  int n_dev = 0;
  if (cudaGetDeviceCount(&n_dev) != cudaSuccess || n_dev == 0) {
    cudaGetLastError();
    t->device = -1;
    *out = t;
    return MV_OK;
  }
  cudaGetDevice(&t->device);
  mv_status s = MV_OK;
  if (s == MV_OK) s = upload(&t->d_tree_indices, tree_indices);
  if (s == MV_OK) s = upload(&t->d_position_ids, position_ids);
  if (s == MV_OK) s = upload(&t->d_retrieve, retrieve);
  if (s == MV_OK) s = upload(&t->d_parent, parent);
  if (s == MV_OK) s = upload(&t->d_ancestors, anc);
  if (s != MV_OK) {
    mv_tree_destroy(t);
    return s;
  }
  *out = t;
  return MV_OK;
}

extern "C" mv_status mv_tree_describe(const mv_tree* t, mv_tree_desc* d) {
  if (!t || !d) return MV_ERR_INVALID_ARG;
  d->n_nodes = t->n_nodes;
  d->n_paths = t->n_paths;
  d->depth = t->depth;
  d->topk = t->topk;
  d->tree_indices = t->h_tree_indices;
  d->position_ids = t->h_position_ids;
  d->retrieve = t->h_retrieve;
  d->parent = t->h_parent;
  d->ancestors = t->h_ancestors;
  d->d_tree_indices = t->d_tree_indices;
  d->d_position_ids = t->d_position_ids;
  d->d_retrieve = t->d_retrieve;
  d->d_parent = t->d_parent;
  d->d_ancestors = t->d_ancestors;
  return MV_OK;
}

extern "C" void mv_tree_destroy(mv_tree* t) {
  if (!t) return;
  delete[] t->h_tree_indices;
  delete[] t->h_position_ids;
  delete[] t->h_retrieve;
  delete[] t->h_parent;
  delete[] t->h_ancestors;
  cudaFree(t->d_tree_indices);
  cudaFree(t->d_position_ids);
  cudaFree(t->d_retrieve);
  cudaFree(t->d_parent);
  cudaFree(t->d_ancestors);
  delete t;
}
