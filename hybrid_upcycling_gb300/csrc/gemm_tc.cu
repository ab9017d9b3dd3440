// Dense bf16 x bf16 -> fp32 GEMM on sm_103a tensor cores for the two student-gradient
// contractions of the fused hidden-state KL backward:
//     dh_s[chunk]  = G W_s      (A = G, K-major over the vocabulary; B = W_s, MN-major)
//     dW_s        += G^T h_s    (A = G^T, MN-major; B = h_s[chunk], MN-major)
// G = dL/dz_s is the bf16 gradient of one token chunk's student logits. The loss is the
// Stage-II KL distillation loss of the HyLo pages (Long-Context Aware Upcycling digest,
// section Method; HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage II); the pages do not
// describe the backward, these are the two contractions of the chain rule through z_s = h_s W_s^T.
//
// Persistent, warp-specialised: warp 0 issues TMA loads into a 4-stage ring, warp 1 issues
// tcgen05 UMMAs (M=128, N=256, K=16) into one of two 256-column TMEM accumulators, warps 2..5
// drain the other accumulator through 128-byte-swizzled staging into TMA stores (overwrite)
// or TMA reduce-adds (accumulate across token chunks).
#include "hylo_internal.h"

namespace hylo {
namespace {

constexpr int kThreads = 192;
constexpr int BN = kGemmBN;
constexpr int A_BYTES = kBM * kBK * 2;   // 16 KB
constexpr int B_BYTES = BN * kBK * 2;    // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 4;
constexpr int NACC = 2;                  // TMEM accumulators (2 x 256 columns)
constexpr int STAGING_BYTES = 4 * 2 * 32 * 128;  // per epilogue warp: 2 x (32 rows x 32 fp32)
constexpr int BAR_OFF = STAGES * STAGE_BYTES + STAGING_BYTES;
constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;
constexpr int SMEM = 1024 + BAR_OFF + NBARS * 8 + 16;
static_assert(SMEM <= 232448, "shared memory budget");

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Loads the A tile (128 rows of M x 64 of K) of k-block kb.
//   K-major: one box {64 k, 128 m}, rows of 128 B.
//   MN-major: two boxes {64 m, 64 k} (k rows of 64 m-elements), the second at +8 KB.
template <bool MN>
__device__ __forceinline__ void load_a(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int m0, int kb) {
  if (!MN) {
    tma_load_2d(dst, m, bar, kb * kBK, m0);
  } else {
    tma_load_2d(dst, m, bar, m0, kb * kBK);
    tma_load_2d(dst + 8192, m, bar, m0 + 64, kb * kBK);
  }
}

// Loads the B tile (256 rows of N x 64 of K): one box {64 k, 256 n}, or four {64 n, 64 k}.
template <bool MN>
__device__ __forceinline__ void load_b(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int n0, int kb) {
  if (!MN) {
    tma_load_2d(dst, m, bar, kb * kBK, n0);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) tma_load_2d(dst + i * 8192, m, bar, n0 + 64 * i, kb * kBK);
  }
}

// Descriptor of the k-th 16-deep slice of a staged tile.
//   K-major: advance 32 B inside the 128 B swizzle row; groups of 8 rows are 1024 B apart.
//   MN-major: advance 16 k-rows = 2048 B; 64-element M/N blocks are 8192 B apart (LBO),
//   groups of 8 k-rows 1024 B apart (SBO).
template <bool MN>
__device__ __forceinline__ uint64_t slice_desc(uint32_t base, int k) {
  return MN ? smem_desc_sw128(base + k * 2048, 8192, 1024) : smem_desc_sw128(base + k * 32, 0, 1024);
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_f32_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* afull = empty + STAGES;
  uint64_t* aempty = afull + NACC;
  uint64_t* drain = aempty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(afull + b, 1);
      mbar_init(aempty + b, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_c);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        const int mb = t / p.n_tiles, nb = t - mb * p.n_tiles;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 11)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
          armed |= 1u << stage;
          load_a<A_MN>(sa, &tm_a, full + stage, mb * kBM, kb);
          load_b<B_MN>(sa + A_BYTES, &tm_b, full + stage, nb * BN, kb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) drain_wait(full + s, s < stage ? phase : (phase ^ 1u), 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x, ++lt) {
        const int b = lt & 1;
        const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
        if (!wait_bounded(aempty + b, aph ^ 1u, abort_flag, p.ctl, 12)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 13)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma_bf16(d, slice_desc<A_MN>(sa, k), slice_desc<B_MN>(sb, k), kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty + stage);
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(afull + b);
      }
      if (!ok && issued) {
        umma_commit(drain);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    const int q = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* staging = smem + STAGES * STAGE_BYTES + (warp - 2) * 2 * 4096;
    int sbuf = 0, lt = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++lt) {
      const int mb = t / p.n_tiles, nb = t - mb * p.n_tiles;
      const int b = lt & 1;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      const bool w = wait_bounded(afull + b, aph, abort_flag, p.ctl, 14);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      const uint32_t acc = lane_base + static_cast<uint32_t>(b * BN);
      const int n_valid = p.Nc - nb * BN;  // columns of this tile inside C
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        if (ch * 32 >= n_valid) break;  // warp-uniform: nothing of this chunk lies inside C
        float v[32];
        tmem_ld32(acc + ch * 32, v);
        tmem_ld_wait();
        uint8_t* buf = staging + sbuf * 4096;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t rowaddr = smem_u32(buf) + lane * 128;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const uint32_t chunk = static_cast<uint32_t>(c4 ^ (lane & 7));
          st_shared_v4(rowaddr + chunk * 16, __float_as_uint(v[4 * c4]), __float_as_uint(v[4 * c4 + 1]),
                       __float_as_uint(v[4 * c4 + 2]), __float_as_uint(v[4 * c4 + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int c0 = nb * BN + ch * 32, r0 = mb * kBM + q * 32;
          if (p.accumulate)
            tma_reduce_add_2d(&tm_c, buf, c0, r0);
          else
            tma_store_2d(&tm_c, buf, c0, r0);
          bulk_commit_group();
        }
        sbuf ^= 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty + b);
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <bool A_MN, bool B_MN>
cudaError_t launch_impl(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& C, const GemmParams& p,
                        int grid, cudaStream_t stream) {
  gemm_bf16_f32_kernel<A_MN, B_MN><<<grid, kThreads, SMEM, stream>>>(A, B, C, p);
  return cudaGetLastError();
}

template <bool A_MN, bool B_MN>
cudaError_t prepare_impl() {
  return cudaFuncSetAttribute(gemm_bf16_f32_kernel<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
}

}  // namespace

int gemm_smem_bytes() { return SMEM; }

cudaError_t gemm_prepare(bool a_mn, bool b_mn) {
  if (!a_mn && b_mn) return prepare_impl<false, true>();
  if (a_mn && b_mn) return prepare_impl<true, true>();
  if (!a_mn && !b_mn) return prepare_impl<false, false>();
  return prepare_impl<true, false>();
}

cudaError_t launch_gemm(bool a_mn, bool b_mn, const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& C,
                        const GemmParams& p, int grid, cudaStream_t stream) {
  if (!a_mn && b_mn) return launch_impl<false, true>(A, B, C, p, grid, stream);
  if (a_mn && b_mn) return launch_impl<true, true>(A, B, C, p, grid, stream);
  if (!a_mn && !b_mn) return launch_impl<false, false>(A, B, C, p, grid, stream);
  return launch_impl<true, false>(A, B, C, p, grid, stream);
}

}  // namespace hylo
