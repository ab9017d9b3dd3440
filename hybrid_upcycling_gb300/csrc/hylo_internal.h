// Internal launch interface between the C-ABI host code and the sm_103a kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace hylo {

// Tile sizes shared by host and device code.
constexpr int kBM = 128;      // token rows per tile (UMMA M, one TMEM lane per row)
constexpr int kBK = 64;       // k elements per pipeline stage (one 128-byte swizzle row)
constexpr int kGemmBN = 256;  // output columns per gradient-GEMM pair tile
constexpr int kFusedBN = 256; // vocabulary columns per fused pair tile (each CTA stages 128 W rows)
constexpr int kMaxSegments = 32;
constexpr int kStatFields = 6; // teacher max, teacher sum, student max, student sum, A, C

// Parameters of the fused dual-GEMM kernel (forward statistics or backward G tiles).
struct FusedParams {
  int N;            // token rows covered by the tensor maps of this launch
  int V;            // vocabulary size
  int kb_s, kb_t;   // 64-wide k-blocks of the student / teacher projections
  int token_tiles;  // ceil(N / 256): 256-token pair tiles
  int vtiles;       // ceil(V / kFusedBN)
  int nseg;         // vocabulary segments per pair tile
  int group;        // pair tiles per raster group (see unit_range)
  int units;        // token_tiles * nseg
  float c;          // log2(e) / tau
  float inv_tau;    // 1 / tau
  float* part;      // forward: partial statistics [kStatFields][nseg][N]
  const float* lse_s;  // backward: per-token log-sum-exps (natural log of sum exp(z/tau))
  const float* lse_t;
  const float* lse_gap;  // backward: precise lse_s - lse_t per token, or null (then lse_s - lse_t)
  float gscale;     // backward: grad_scale / (tau * N_total)
  int split;        // backward: also store G - bf16(G), rounded to bf16, through the second G map
  unsigned long long* progress;  // pacing counters [kMaxClusters] + off switch, zero at launch; null: no pacing
  WaitCtl ctl;
};

// One GEMM problem C[M, Nc] (=|+=) sum_k A[m, k] B[n, k] of the paired gradient kernel, tiled
// in 256 x 256 pair tiles (each CTA of a pair owns 128 rows of the tile).
struct GemmProblem {
  int M, Nc;
  int kblocks;               // ceil(K / 64)
  int m_tiles, n_tiles, tiles;
  int a_mn;                  // A operand MN-major (1) or K-major (0); B is MN-major
  int accumulate;            // 0: overwrite C, 1: add into C (TMA reduce-add)
};

constexpr int kMaxClusters = 128;

// Both gradient problems of one token chunk. Problem-0 (dh_s, K = V) tiles are dealt
// round-robin over the clusters. Clusters c >= p0_rem (p0_rem = tiles0 % nclusters, when
// nonzero) get one problem-0 tile fewer; they first share the problem-1 (dW_s) tiles
// [0, p1_split) round-robin among themselves, then all clusters share [p1_split, tiles1)
// round-robin, so concurrently running tiles are neighbours (their G and h_s blocks stay in L2)
// and every cluster finishes within about one problem-1 tile of the others.
struct GemmParams {
  GemmProblem prob[2];
  int nclusters;
  int p1_split;
  WaitCtl ctl;
};

// Fused dual-GEMM kernel on CTA pairs; bn = vocabulary columns per pair tile (kFusedBN).
// fused_prepare reports how many 2-CTA clusters fit on the device at once; a launch runs
// `clusters` clusters, each working through units (256-token tile, vocabulary segment).
cudaError_t fused_prepare(int bn, int* max_clusters);
cudaError_t launch_fused(int bn, bool backward, const CUtensorMap& hs, const CUtensorMap& Ws, const CUtensorMap& ht,
                         const CUtensorMap& Wt, const CUtensorMap& G, const CUtensorMap& G2, const FusedParams& p,
                         int clusters, cudaStream_t stream);
cudaError_t launch_combine(const float* part, int N, int nseg, float inv_tau, float* kl, float* lse_s,
                           float* lse_t, float* lse_gap, cudaStream_t stream);
cudaError_t launch_mean(const float* kl, int N, float* loss, cudaStream_t stream);

// "Fused KL" on precomputed bf16 logits [N, ld]: one row per cluster at a time (clusters of
// kSplit CTAs). kl_logits_prepare reports how many clusters fit on the device at once.
cudaError_t kl_logits_prepare(int* max_clusters);
cudaError_t launch_kl_logits(const uint16_t* zs, const uint16_t* zt, uint16_t* dz, int64_t ld, int N, int V, float tau,
                             float gscale, float* kl, float* lse_s, float* lse_t, const WaitCtl& ctl, int clusters,
                             cudaStream_t stream);

// Stage-I Enhanced-ILD loss on stacked [P, N, d] bf16 tensors (one warp per row).
cudaError_t launch_ild(const uint16_t* S, const uint16_t* T, int64_t P, int64_t N, int d, float grad_scale, float* norms,
                       float* loss, uint16_t* dS, int sms, cudaStream_t stream);

// Paired (cta_group::2) gradient GEMM: sets the shared-memory limit and reports how many
// 2-CTA clusters fit on the device at once; the launch runs p.nclusters clusters.
int gemm_smem_bytes();
cudaError_t gemm_prepare(int* max_clusters);
cudaError_t launch_gemm_pair(const CUtensorMap& A0, const CUtensorMap& B0, const CUtensorMap& C0, const CUtensorMap& A1,
                             const CUtensorMap& B1, const CUtensorMap& C1, const GemmParams& p, cudaStream_t stream);

}  // namespace hylo
