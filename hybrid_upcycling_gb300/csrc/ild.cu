// Stage-I Enhanced-ILD alignment loss on GB300: for every (entry, token) row of the stacked
// student and teacher tensors S, T [P, N, d] (P = one entry per layer and per kind: layer
// outputs h and token-mixer outputs a), the Euclidean norm of the difference, their sum over
// entries averaged over tokens, and the gradient grad_scale * (S - T) / (N ||S - T||) in bf16.
// (Long-Context Aware Upcycling digest, section Method: L_ILD = sum_l ||h_s - h_t||_2 +
// ||a_s - a_t||_2; section Key Ideas: Stage I aligns hidden states and token-mixer outputs;
// HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage I: layer-wise alignment at 2K context.)
//
// HBM-bound: one warp per row, 16-byte vector loads of both tensors once from DRAM, a warp
// reduction of the squared differences in fp32, and (gradient requested) a second read of the
// row -- served by L1/L2, the warp has just read it -- for the bf16 gradient store.
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

// loss[0] = sum(norms[0..rows)) / N, fixed-order fp64 reduction (one block).
__global__ void __launch_bounds__(1024) ild_sum_kernel(const float* __restrict__ norms, int64_t rows, int64_t N,
                                                       float* loss) {
  __shared__ double red[1024];
  double s = 0;
  for (int64_t i = threadIdx.x; i < rows; i += 1024) s += static_cast<double>(norms[i]);
  red[threadIdx.x] = s;
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
  const int64_t want = (rows * 32 + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8);
  const float gscale = static_cast<float>(static_cast<double>(grad_scale) / static_cast<double>(N));
  ild_kernel<<<grid, kThreads, 0, stream>>>(S, T, rows, d, gscale, norms, dS);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ild_sum_kernel<<<1, 1024, 0, stream>>>(norms, rows, N, loss);
  return cudaGetLastError();
}

}  // namespace hylo
