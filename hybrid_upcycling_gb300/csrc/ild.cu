// Stage-I Enhanced-ILD alignment loss on GB300: for every (entry, token) row of the stacked
// student and teacher tensors S, T [P, N, d] (P = one entry per layer and per kind: layer
// outputs h and token-mixer outputs a), the Euclidean norm of the difference, their sum over
// entries averaged over tokens, and the gradient grad_scale * (S - T) / (N ||S - T||) in bf16.
// (Long-Context Aware Upcycling digest, section Method: L_ILD = sum_l ||h_s - h_t||_2 +
// ||a_s - a_t||_2; section Key Ideas: Stage I aligns hidden states and token-mixer outputs;
// HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage I: layer-wise alignment at 2K context.)
//
// HBM-bound. Rows of up to 16384 elements are held in registers: a group of 1, 2, 4 or 8 warps
// owns a row, each lane issues all of its 16-byte loads of both tensors at once (up to 8 + 8),
// the squared differences are reduced in fp32 (warp shuffles, then the group's warps through
// shared memory in a fixed order), and the bf16 gradient is formed from the same registers, so
// each input byte crosses HBM once. Longer rows take a one-warp-per-row kernel that reads the
// row a second time for the gradient. The grid is the number of blocks that fit on the device
// at once (a persistent grid-stride loop), so no block waits for a second wave.
#include "hylo_internal.h"

namespace hylo {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(uint4 v, float* z) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(w[i] << 16);
    z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float2 diff2(uint32_t a, uint32_t b) {
  return __fadd2_rn(make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u)),
                    make_float2(-__uint_as_float(b << 16), -__uint_as_float(b & 0xffff0000u)));
}

// One row per group of `wpr` warps (wpr in {1, 2, 4, 8}); each warp owns VPL * 32 consecutive
// 16-byte vectors of the row.
template <int VPL>
__global__ void __launch_bounds__(kThreads) ild_reg_kernel(const uint16_t* __restrict__ S,
                                                           const uint16_t* __restrict__ T, int64_t rows, int d,
                                                           int wpr, float gscale, float* __restrict__ norms,
                                                           uint16_t* __restrict__ dS) {
  __shared__ float red[2][kThreads / 32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int grp = wib / wpr, part = wib - grp * wpr;
  const int gpb = (kThreads / 32) / wpr;  // row groups per block
  const int nvec = d / 8;
  const int64_t ngroups = static_cast<int64_t>(gridDim.x) * gpb;
  int it = 0;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * gpb + grp; r < rows; r += ngroups, ++it) {
    const uint4* s = reinterpret_cast<const uint4*>(S + r * d);
    const uint4* t = reinterpret_cast<const uint4*>(T + r * d);
    const int v0 = part * 32 * VPL + lane;
    uint4 a[VPL], b[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = v0 + i * 32;
      a[i] = v < nvec ? __ldcs(s + v) : make_uint4(0u, 0u, 0u, 0u);
      b[i] = v < nvec ? __ldcs(t + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float2 dd = diff2(a[i].x, b[i].x);
      acc = __ffma2_rn(dd, dd, acc);
      dd = diff2(a[i].y, b[i].y);
      acc = __ffma2_rn(dd, dd, acc);
      dd = diff2(a[i].z, b[i].z);
      acc = __ffma2_rn(dd, dd, acc);
      dd = diff2(a[i].w, b[i].w);
      acc = __ffma2_rn(dd, dd, acc);
    }
    float ss = acc.x + acc.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (wpr > 1) {
      // Slots alternate by iteration: a warp reaches the next write of a slot only after the
      // group's barrier of the following iteration, i.e. after every warp read this one.
      if (lane == 0) red[it & 1][wib] = ss;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(wpr * 32) : "memory");
      ss = 0.f;
      for (int k = 0; k < wpr; ++k) ss += red[it & 1][grp * wpr + k];
    }
    const float nrm = sqrtf(ss);
    if (part == 0 && lane == 0) norms[r] = nrm;
    if (dS != nullptr) {
      const float sc = nrm > 0.f ? gscale / nrm : 0.f;
      const float2 sc2 = make_float2(sc, sc);
      uint4* g = reinterpret_cast<uint4*>(dS + r * d);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int v = v0 + i * 32;
        if (v < nvec) {
          float2 g0 = __fmul2_rn(diff2(a[i].x, b[i].x), sc2), g1 = __fmul2_rn(diff2(a[i].y, b[i].y), sc2);
          float2 g2 = __fmul2_rn(diff2(a[i].z, b[i].z), sc2), g3 = __fmul2_rn(diff2(a[i].w, b[i].w), sc2);
          __stcs(g + v, make_uint4(pack_bf16x2(g0.x, g0.y), pack_bf16x2(g1.x, g1.y), pack_bf16x2(g2.x, g2.y),
                                   pack_bf16x2(g3.x, g3.y)));
        }
      }
    }
  }
}

// Rows longer than 16384 elements: one warp per row, the gradient pass reads the row again.
__global__ void __launch_bounds__(kThreads) ild_kernel(const uint16_t* __restrict__ S, const uint16_t* __restrict__ T,
                                                       int64_t rows, int d, float gscale, float* __restrict__ norms,
                                                       uint16_t* __restrict__ dS) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int nvec = d / 8;  // d is a multiple of 8
  for (int64_t r = warp; r < rows; r += nwarps) {
    const uint4* s = reinterpret_cast<const uint4*>(S + r * d);
    const uint4* t = reinterpret_cast<const uint4*>(T + r * d);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      float a[8], b[8];
      unpack8(__ldg(s + v), a);
      unpack8(__ldg(t + v), b);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 dd = __fadd2_rn(make_float2(a[2 * j], a[2 * j + 1]), make_float2(-b[2 * j], -b[2 * j + 1]));
        acc = __ffma2_rn(dd, dd, acc);
      }
    }
    float ss = acc.x + acc.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float nrm = sqrtf(ss);
    if (lane == 0) norms[r] = nrm;
    if (dS != nullptr) {
      const float sc = nrm > 0.f ? gscale / nrm : 0.f;
      const float2 sc2 = make_float2(sc, sc);
      uint4* g = reinterpret_cast<uint4*>(dS + r * d);
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float a[8], b[8];
        unpack8(__ldg(s + v), a);
        unpack8(__ldg(t + v), b);
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 dd = __fadd2_rn(make_float2(a[2 * j], a[2 * j + 1]), make_float2(-b[2 * j], -b[2 * j + 1]));
          const float2 gg = __fmul2_rn(dd, sc2);
          pk[j] = pack_bf16x2(gg.x, gg.y);
        }
        __stcs(g + v, make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
    }
  }
}

// loss[0] = sum(norms[0..rows)) / N in a fixed order (one block): each thread sums its strided
// share in fp32 with Kahan compensation (error ~2 ulp whatever the count; GB300's fp64 rate is
// too low for hundreds of thousands of fp64 adds on one SM), then the 1024 partials are added
// in fp64 by a fixed tree.
__global__ void __launch_bounds__(1024) ild_sum_kernel(const float* __restrict__ norms, int64_t rows, int64_t N,
                                                       float* loss) {
  __shared__ double red[1024];
  float s = 0.f, comp = 0.f;
  for (int64_t i = threadIdx.x; i < rows; i += 1024) {
    const float y = norms[i] - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
  }
  red[threadIdx.x] = static_cast<double>(s) - static_cast<double>(comp);
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[0] = static_cast<float>(red[0] / static_cast<double>(N));
}

}  // namespace

cudaError_t launch_ild(const uint16_t* S, const uint16_t* T, int64_t P, int64_t N, int d, float grad_scale, float* norms,
                       float* loss, uint16_t* dS, int sms, cudaStream_t stream) {
  const int64_t rows = P * N;
  const float gscale = static_cast<float>(static_cast<double>(grad_scale) / static_cast<double>(N));
  const int nvec = d / 8;
  cudaError_t e;
  if (nvec <= 8 * 32 * 8) {
    int wpr = 1;
    while (wpr * 256 < nvec) wpr *= 2;  // warps per row, each owning up to 256 vectors
    const int per_warp = (nvec + wpr - 1) / wpr;
    const int vpl = per_warp <= 32 ? 1 : per_warp <= 64 ? 2 : per_warp <= 128 ? 4 : 8;
    const void* fn = vpl == 1 ? reinterpret_cast<const void*>(ild_reg_kernel<1>)
                     : vpl == 2 ? reinterpret_cast<const void*>(ild_reg_kernel<2>)
                     : vpl == 4 ? reinterpret_cast<const void*>(ild_reg_kernel<4>)
                                : reinterpret_cast<const void*>(ild_reg_kernel<8>);
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0)) != cudaSuccess) return e;
    const int64_t gpb = (kThreads / 32) / wpr;
    const int64_t want = (rows + gpb - 1) / gpb;
    const int64_t cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = static_cast<int>(want < cap ? want : cap);
    switch (vpl) {
      case 1: ild_reg_kernel<1><<<grid, kThreads, 0, stream>>>(S, T, rows, d, wpr, gscale, norms, dS); break;
      case 2: ild_reg_kernel<2><<<grid, kThreads, 0, stream>>>(S, T, rows, d, wpr, gscale, norms, dS); break;
      case 4: ild_reg_kernel<4><<<grid, kThreads, 0, stream>>>(S, T, rows, d, wpr, gscale, norms, dS); break;
      default: ild_reg_kernel<8><<<grid, kThreads, 0, stream>>>(S, T, rows, d, wpr, gscale, norms, dS); break;
    }
  } else {
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ild_kernel, kThreads, 0)) != cudaSuccess) return e;
    const int64_t want = (rows * 32 + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = static_cast<int>(want < cap ? want : cap);
    ild_kernel<<<grid, kThreads, 0, stream>>>(S, T, rows, d, gscale, norms, dS);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ild_sum_kernel<<<1, 1024, 0, stream>>>(norms, rows, N, loss);
  return cudaGetLastError();
}

}  // namespace hylo
