// "Fused KL" on precomputed logits: the memory-bound sibling of the fused hidden-state KL.
// For every token row it reads the student and teacher logits (bf16, [N, V]), computes
// KL(softmax(z_t/tau) || softmax(z_s/tau)) and both log-sum-exps without storing
// probabilities, and optionally writes the gradient of grad_scale * mean(KL) with respect to
// the student logits, dz_s = grad_scale * (p_s - p_t) / (tau N), in bf16.
//
// The pages list "Fused KL" beside the "Fused Hidden-State KL" in the memory stack that makes
// 8B-teacher, 64K-token Stage-II distillation fit (Long-Context Aware Upcycling digest, section
// Key Ideas; section Method for the softmax+KL fusion); the loss is the KL between the two
// next-token distributions (HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage II).
//
// One CTA of 512 threads per SM walks rows persistently. Pass 1: each thread folds 32-column
// chunks of the row into running statistics (shared with the hidden-state kernel), the CTA
// merges them and one thread forms KL and the lse's in fp64. Pass 2 (gradient requested):
// the row is read again -- 152 rows in flight x 2 x 256 KB stay in the 129 MB L2 -- and dz_s
// is streamed out. HBM traffic per element: 4 B read (+ 2 B written with the gradient).
#include "hylo_internal.h"
#include "kl_stats.cuh"

namespace hylo {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint4 ldg_v4(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* z) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(w[i] << 16);
    z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// 32 consecutive logits of a row starting at column col0 (a multiple of 32); columns >= V read
// as 0 (they are masked by the caller).
__device__ __forceinline__ void load32(const uint16_t* row, int col0, int V, float (&z)[32]) {
  if (col0 + 32 <= V) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ldg_v4(row + col0 + 8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack_bf16x8(v[i], z + 8 * i);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) z[j] = (col0 + j < V) ? bf16_to_f32(row[col0 + j]) : 0.f;
  }
}

// Merge that also accepts an empty `r` (a thread or warp that saw no column).
__device__ __forceinline__ void merge_any(RowStats& r, const RowStats& o, float c) {
  if (o.mt == -INFINITY) return;
  if (r.mt == -INFINITY) {
    r = o;
    return;
  }
  merge_stats(r, o, c);
}

__device__ __forceinline__ RowStats shfl_stats(const RowStats& r, int off) {
  RowStats o;
  o.mt = __shfl_xor_sync(0xffffffffu, r.mt, off);
  o.st = __shfl_xor_sync(0xffffffffu, r.st, off);
  o.ms = __shfl_xor_sync(0xffffffffu, r.ms, off);
  o.ss = __shfl_xor_sync(0xffffffffu, r.ss, off);
  o.a = __shfl_xor_sync(0xffffffffu, r.a, off);
  o.cc = __shfl_xor_sync(0xffffffffu, r.cc, off);
  o.far = __shfl_xor_sync(0xffffffffu, static_cast<int>(r.far), off) != 0;
  return o;
}

struct LogitsParams {
  const uint16_t* zs;
  const uint16_t* zt;
  uint16_t* dz;   // gradient [N, ld] bf16, or null
  int64_t ld;     // row stride in elements
  int N, V;
  float c;        // log2(e) / tau
  float inv_tau;
  float gscale;   // grad_scale / (tau N)
  float* kl;
  float* lse_s;
  float* lse_t;
};

__global__ void __launch_bounds__(kThreads, 1) kl_logits_kernel(const LogitsParams p) {
  __shared__ RowStats warp_stats[kWarps];
  __shared__ float row_lse[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nchunks = (p.V + 31) / 32;
  for (int n = blockIdx.x; n < p.N; n += gridDim.x) {
    const uint16_t* zs_row = p.zs + static_cast<size_t>(n) * p.ld;
    const uint16_t* zt_row = p.zt + static_cast<size_t>(n) * p.ld;
    // ---- pass 1: statistics
    RowStats rs{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
    for (int ch = tid; ch < nchunks; ch += kThreads) {
      const int col0 = ch * 32;
      float zt[32], zs[32];
      load32(zt_row, col0, p.V, zt);
      load32(zs_row, col0, p.V, zs);
      const int valid = min(32, p.V - col0);
      if (valid == 32)
        fold_chunk<false>(rs, zt, zs, 32, p.c, p.inv_tau);
      else
        fold_chunk<true>(rs, zt, zs, valid, p.c, p.inv_tau);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) merge_any(rs, shfl_stats(rs, off), p.c);
    if (lane == 0) warp_stats[warp] = rs;
    __syncthreads();
    if (warp == 0) {
      rs = lane < kWarps ? warp_stats[lane] : RowStats{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) merge_any(rs, shfl_stats(rs, off), p.c);
      if (lane == 0) {
        double lt, ls;
        const double k = kl_from_stats(rs.mt, rs.st, rs.ms, rs.ss, rs.a, rs.cc, rs.far, p.inv_tau, lt, ls);
        p.kl[n] = static_cast<float>(k);
        p.lse_s[n] = static_cast<float>(ls);
        p.lse_t[n] = static_cast<float>(lt);
        row_lse[0] = static_cast<float>(lt);
        row_lse[1] = static_cast<float>(ls);
      }
    }
    __syncthreads();
    // ---- pass 2: dz_s = gscale (p_s - p_t), p_x = exp(z_x / tau - lse_x)
    if (p.dz != nullptr) {
      const float bt = row_lse[0] * kLog2e, bs = row_lse[1] * kLog2e;
      const float2 c2 = make_float2(p.c, p.c), gs2 = make_float2(p.gscale, p.gscale);
      const float2 nbt = make_float2(-bt, -bt), nbs = make_float2(-bs, -bs), m1 = make_float2(-1.f, -1.f);
      uint16_t* dz_row = p.dz + static_cast<size_t>(n) * p.ld;
      for (int ch = tid; ch < nchunks; ch += kThreads) {
        const int col0 = ch * 32;
        float zt[32], zs[32];
        load32(zt_row, col0, p.V, zt);
        load32(zs_row, col0, p.V, zs);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 pt = ex2_approx2(__ffma2_rn(make_float2(zt[2 * j], zt[2 * j + 1]), c2, nbt));
          const float2 ps = ex2_approx2(__ffma2_rn(make_float2(zs[2 * j], zs[2 * j + 1]), c2, nbs));
          const float2 g = __fmul2_rn(__ffma2_rn(pt, m1, ps), gs2);
          pk[j] = pack_bf16x2(g.x, g.y);
        }
        if (col0 + 32 <= p.V) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcs(reinterpret_cast<uint4*>(dz_row + col0 + 8 * i), make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < p.V) dz_row[col0 + j] = static_cast<uint16_t>((pk[j >> 1] >> (16 * (j & 1))) & 0xffffu);
        }
      }
    }
    __syncthreads();  // warp_stats and row_lse are reused by the next row
  }
}

}  // namespace

cudaError_t launch_kl_logits(const uint16_t* zs, const uint16_t* zt, uint16_t* dz, int64_t ld, int N, int V, float tau,
                             float gscale, float* kl, float* lse_s, float* lse_t, int grid, cudaStream_t stream) {
  LogitsParams p;
  p.zs = zs;
  p.zt = zt;
  p.dz = dz;
  p.ld = ld;
  p.N = N;
  p.V = V;
  p.c = kLog2e / tau;
  p.inv_tau = 1.0f / tau;
  p.gscale = gscale;
  p.kl = kl;
  p.lse_s = lse_s;
  p.lse_t = lse_t;
  kl_logits_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hylo
