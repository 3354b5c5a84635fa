// Parameters and host helpers of the tcgen05 projection kernel (gemm.cu).
#pragma once

#include "attn_core.cuh"
#include "common.cuh"

enum { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_QKV = 3 };
constexpr int kGemmMaxTiles = 1024;

struct GemmParams {
  int M;         // weight rows (output features); for SWIGLU the FFN width F (rows per gate/up matrix)
  int K;         // reduction length
  int n_tok;     // valid token columns (1..256; up to 64 per token group)
  int tok_ld;    // token stride of ssq, ssq_out and row_max (0: 64 x the launch's token groups)
  int paired;    // SWIGLU: tile = 64 rows of amap0 (gate) + the same 64 rows of amap1 (up)
  // Weight maps: 0 row-major (2-D maps); packed [row tile][k-block][rows][64] layout: 1 one k-block per load
  // (a0, and a1 for the up matrix of a paired phase); 2 a0 loads kKps consecutive k-blocks of a tile in one box,
  // a1 one; 3 (paired) gate and up of a layer in one allocation, a0 / a1 4-D maps whose box holds the gate and up
  // rows of kKps / one k-block in the order the MMA reads them.
  int packed_a;
  int act_box;   // token groups of map b2's box (0: none): a stage's activations, all its k-blocks and groups, in one box
  // derived (gemm_finish_params): k-blocks, tiles, CTAs per cluster (K slices per tile), clusters, CTAs
  int kbt, n_tiles, csize, n_clusters, grid;
  // RMSNorm scale of the input columns: s = 1/sqrt(sum(ssq[0..ssq_parts)) / norm_d + eps); null = 1
  const float* ssq;
  int ssq_parts, norm_d;
  float eps;
  // EPI_STORE
  float* out_f32;
  int ld_out;
  float2* row_max;  // optional [n_tiles][tok_ld]: per 128-row tile and token, (max, first argmax as int bits)
  // EPI_RESIDUAL (x, xb are [n][M]; ssq_out is [n_tiles][tok_ld])
  float* x;
  uint16_t* xb;
  float* ssq_out;
  // EPI_SWIGLU (act is [n][F])
  uint16_t* act;
  int F;
  // EPI_QKV: rows = [q heads | k heads | v heads] x D
  uint16_t* q_out;  // [n][H][D]
  uint16_t* kv;     // [L][2][H][S_max][D]
  int H, D, S_max, layer;
  const int32_t* cur_len;  // device prefix length (one per sequence when seq_rows > 0)
  const int32_t* pos_ids;  // [n] depth of each token (of each tree row when seq_rows > 0)
  // Several sequences in one pass (QKV): token j is row j % seq_rows of sequence j / seq_rows's tree; rows at or
  // past seq_n are padding (nothing is appended). The sequences' caches are kv_seq_stride elements apart.
  // seq_rows is 0 (one sequence) or 64 (one token group per sequence).
  int seq_rows, seq_n;
  size_t kv_seq_stride;
  float log2_theta;
  unsigned int* err;
};

// A chain of up to kGemmMaxPhases projections in one persistent launch: phase i+1's activations are phase i's
// output, so its activation loads wait for a device counter that every CTA bumps once it has finished phase i
// (its weight loads run ahead meanwhile). One cluster shape for all phases.
constexpr int kGemmMaxPhases = 4;
struct GemmPhase {
  int epi;
  CUtensorMap a0, a1, b;  // weights (a1: the up matrix of a paired phase), activations
  CUtensorMap b2;         // p.act_box: the activations as one box per pipeline stage (gemm_act_map_stage)
  GemmParams p;
};
// Counters of a chain: kGemmMaxPhases phase counters, the exit counter, the attention counter. Zero before the
// first launch; every launch leaves them zero again.
constexpr int kGemmAttnFlag = kGemmMaxPhases + 1;
constexpr int kGemmChainFlagWords = kGemmMaxPhases + 2;

// The tree attention of the chain's layer, run first inside the chain (its output is phase 0's activations):
// cluster q computes head q, its CTAs the head's key splits, on the epilogue warps, while the producer already
// streams phase 0's weights. D is 64 or 128; one sequence of at most 64 tree nodes.
struct GemmAttn {
  CUtensorMap kmap, vmap;  // the cache planes [H][S_max][D] (attn::Args plane_k / plane_v pick the layer's)
  attn::Args args;         // splits is set by the launch (= the chain's cluster size)
  int D;
};

bool gemm_weight_map(CUtensorMap* map, const void* w, int rows, int K, int box_rows);
bool gemm_weight_map_packed(CUtensorMap* map, const void* w, int rows, int K, int tile_rows);
// packed weights: a box of `depth` consecutive k-blocks of one row tile (one load per pipeline stage)
bool gemm_weight_map_packed_depth(CUtensorMap* map, const void* w, int rows, int K, int tile_rows, int depth);
// gate and up of a SwiGLU layer, both packed with 64-row tiles, up = gate + (packed bytes of gate): a box of
// `depth` k-blocks, each holding 64 gate rows then the same 64 up rows. False if the two are not laid out so.
bool gemm_weight_map_paired(CUtensorMap* map, const void* gate, const void* up, int F, int K, int depth);
// The k-blocks per pipeline stage of a launch over n_tok tokens (the box depth of packed_a 2 / 3 maps' a0).
int gemm_stage_kblocks(int n_tok);
bool gemm_act_map(CUtensorMap* map, const void* x, int rows, int K);
// rows x K bf16 activations (K % 64 == 0) as [k-block][row][64]: a box of 64 groups rows x the k-blocks of one
// pipeline stage of a launch over `groups` token groups (gemm_stage_kblocks), in the order the MMAs read them
bool gemm_act_map_stage(CUtensorMap* map, const void* x, int rows, int K, int groups);
// rows x K bf16 activations whose rows are ld elements apart (ld % 8 == 0)
bool gemm_act_map_strided(CUtensorMap* map, const void* x, int rows, int K, int ld);
void gemm_finish_params(GemmParams& p);
mv_status launch_gemm(int epi, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                      const GemmParams& p, cudaStream_t stream);
// ph[i].p must have its shape fields set (M, K, paired, F); the cluster plan is computed here. flags: see above
// (may be null when n == 1).
// independent: the phases read nothing another phase writes (no counters; flags may be null).
// attn: the layer's attention first (see GemmAttn); MV_ERR_UNSUPPORTED, with nothing launched, when this chain
// cannot run it (more than one token group, a cluster size above attn::kMaxSplits, fewer clusters than heads).
mv_status launch_gemm_chain(GemmPhase* ph, int n, unsigned int* flags, cudaStream_t stream,
                            bool independent = false, const GemmAttn* attn = nullptr);
