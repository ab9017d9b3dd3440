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
constexpr int kGemmBN = 256;  // d_s columns per gradient tile of the backward
constexpr int kFusedBN = 256; // vocabulary columns per fused pair tile (each CTA stages 128 W rows)
constexpr int kMaxSegments = 32;
constexpr int kStatFields = 6; // teacher max, teacher sum, student max, student sum, A, C

// Parameters of the fused forward kernel (teacher and student logit tiles folded into
// per-token softmax/KL statistics).
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
  float* part;      // partial statistics [kStatFields][nseg][N]
  unsigned long long* progress;  // pacing counters [kMaxClusters] + off switch; null: no pacing
  unsigned epoch;   // 1..65535, different from the previous paced launch on the same counters
  WaitCtl ctl;
};

constexpr int kMaxClusters = 128;

// Fused forward kernel on CTA pairs; bn = vocabulary columns per pair tile (kFusedBN).
// fused_prepare reports how many 2-CTA clusters fit on the device at once; a launch runs
// `clusters` clusters, each working through units (256-token tile, vocabulary segment).
cudaError_t fused_prepare(int bn, int* max_clusters);
cudaError_t launch_fused(int bn, const CUtensorMap& hs, const CUtensorMap& Ws, const CUtensorMap& ht,
                         const CUtensorMap& Wt, const FusedParams& p, int clusters, cudaStream_t stream);
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

// The backward as one persistent launch (kl_bwd_pipe.cu). The tokens are cut into TB blocks of
// R rows (R a multiple of 256, or one block of all N) and the vocabulary into VB blocks of bw
// words (a multiple of 256); block b = (b / VB, b % VB). Per block, "F" work items recompute
// the block's 256 x 256 logit tile pairs and write G = dL/dz_s (bf16) into ring slot b % kGRing
// of the workspace, and "M" work items add the block's contributions to dW_s (G^T h_s) and dh_s
// (G W_s). Items run in the queue order F(0), F(1), M(0), F(2), M(1), F(3), ..., M(B-1), dealt
// to clusters by an atomic counter; completion counters order M(b) after F(b) and after M(b-1)
// (same output tiles), and F(b) after M(b - kGRing) (same ring slot).
constexpr int kGRing = 3;
// Bytes of the G ring (one bf16 term) at most, whatever N, V and token_chunk. 128 MiB holds three
// blocks of 4096 tokens x 5376 words: fewer, wider vocabulary blocks than a 64 MiB ring, so dh_s
// is reduce-added half as often (24 instead of 51 times at V = 128256).
constexpr int64_t kGBlockBytes = int64_t(128) << 20;
struct BwdPipeParams {
  int N, V, d_s;
  int kb_s, kb_t;   // 64-wide k-blocks of the student / teacher projections
  int ntd;          // 256-column tiles of d_s
  int R, bw;        // token block rows, vocabulary block width
  int TB, VB, B;    // token blocks, vocabulary blocks, TB * VB
  float c;          // log2(e) / tau
  float gscale;     // grad_scale / (tau * N)
  const float* lse_s;
  const float* lse_t;
  const float* lse_gap;  // precise lse_s - lse_t, or null
  int split;        // also store G - bf16(G) (ring slots kGRing..2 kGRing-1) and add its products
  unsigned* ctrl;   // [0] work queue, [1] M-item completions, [2 + s] F-item completions of slot s; zero at launch
  WaitCtl ctl;
};
constexpr int kPipeCtrlWords = 2 + kGRing;

// Sets the shared-memory limit and reports how many 2-CTA clusters of the pipelined backward
// fit on the device at once.
cudaError_t bwd_pipe_prepare(int* max_clusters);
// Maps: hs, ht, Ws, Wt K-major (box 64 x 128); WsB, hsB MN-major (box 64 x 64); dh, dW fp32
// (box 32 x 32); G, GA, GT over the ring [slots][R][bw] bf16 (boxes 32 x 32 with 64-byte
// swizzle, 64 x 128, 64 x 64).
cudaError_t launch_bwd_pipe(const CUtensorMap* maps, const BwdPipeParams& p, int clusters, cudaStream_t stream);
constexpr int kPipeMaps = 11;

}  // namespace hylo
