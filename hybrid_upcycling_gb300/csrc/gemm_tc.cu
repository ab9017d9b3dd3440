// Dense bf16 x bf16 -> fp32 GEMM on sm_103a tensor cores for the two student-gradient
// contractions of the fused hidden-state KL backward, both in one launch per token chunk:
//     problem 0: dh_s[chunk]  = G W_s      (A = G, K-major over the vocabulary; B = W_s, MN-major)
//     problem 1: dW_s        += G^T h_s    (A = G^T, MN-major; B = h_s[chunk], MN-major)
// G = dL/dz_s is the bf16 gradient of one token chunk's student logits. The loss is the
// Stage-II KL distillation loss of the HyLo pages (Long-Context Aware Upcycling digest,
// section Method; HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage II); the pages do not
// describe the backward, these are the two contractions of the chain rule through z_s = h_s W_s^T.
//
// CTA pairs (clusters of 2 on an SM pair) share one 256 x 256 tile per UMMA
// (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16): each CTA stages 128 rows of A and 128
// rows of B, so each SM streams half the B operand it would alone. Warp 0 of each CTA issues
// its TMA loads (completion counted on the even CTA's barrier), warp 1 of the even CTA issues
// the UMMAs into one of two 256-column TMEM accumulators per CTA, warps 2..5 of both CTAs drain
// the other accumulator through 128-byte-swizzled staging into TMA stores (overwrite) or TMA
// reduce-adds (accumulate across token chunks).
//
// Schedule: persistent, one cluster per SM pair. The few long problem-0 tiles (K = V) are dealt
// round-robin first; the short problem-1 tiles follow round-robin in two phases (see
// GemmParams) so that all clusters finish together and concurrent tiles share L2.
#include "hylo_internal.h"

namespace hylo {
namespace {

constexpr int kThreads = 192;
constexpr int BN = kGemmBN;                      // 256 output columns per pair tile
constexpr int HB = BN / 2;                       // B rows staged per CTA
constexpr int A_BYTES = kBM * kBK * 2;           // 16 KB: this CTA's 128 rows of A
constexpr int B_BYTES = HB * kBK * 2;            // 16 KB: this CTA's 128 rows of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 6;
constexpr int NACC = 2;                          // TMEM accumulators (2 x 256 columns)
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

// The idx-th tile of cluster `cid` under the schedule described at GemmParams.
__device__ __forceinline__ bool tile_at(const GemmParams& p, int cid, int idx, int& prob, int& t) {
  const int ncl = p.nclusters;
  const int t0 = p.prob[0].tiles, t1 = p.prob[1].tiles;
  const int n0 = t0 > cid ? (t0 - 1 - cid) / ncl + 1 : 0;
  if (idx < n0) {
    prob = 0;
    t = cid + idx * ncl;
    return true;
  }
  int j = idx - n0;
  prob = 1;
  const int rem = t0 % ncl;
  if (rem != 0 && cid >= rem && p.p1_split > 0) {  // phase A: the clusters with one tile fewer
    const int e = ncl - rem, k = cid - rem;
    const int na = k < p.p1_split ? (p.p1_split - 1 - k) / e + 1 : 0;
    if (j < na) {
      t = k + j * e;
      return true;
    }
    j -= na;
  }
  t = p.p1_split + cid + j * ncl;  // phase B: all clusters
  return t < t1;
}

// Descriptor of the k-th 16-deep slice of a staged 128-row tile.
//   K-major: advance 32 B inside the 128 B swizzle row; groups of 8 rows are 1024 B apart.
//   MN-major: advance 16 k-rows = 2048 B; the two 64-element M/N blocks are 8192 B apart (LBO),
//   groups of 8 k-rows 1024 B apart (SBO).
__device__ __forceinline__ uint64_t slice_desc(bool mn, uint32_t base, int k) {
  return mn ? smem_desc_sw128(base + k * 2048, 8192, 1024) : smem_desc_sw128(base + k * 32, 0, 1024);
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_b0,
                 const __grid_constant__ CUtensorMap tm_c0, const __grid_constant__ CUtensorMap tm_a1,
                 const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_c1,
                 const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // used in the even CTA
  uint64_t* empty = full + STAGES;                                // both CTAs
  uint64_t* afull = empty + STAGES;                               // both CTAs
  uint64_t* aempty = afull + NACC;                                // used in the even CTA
  uint64_t* drain = aempty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the UMMAs
  const int cid = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(afull + b, 1);
      mbar_init(aempty + b, 2 * 4);  // four epilogue warps in each CTA of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_a0);
    prefetch_tmap(&tm_b0);
    prefetch_tmap(&tm_c0);
    prefetch_tmap(&tm_a1);
    prefetch_tmap(&tm_b1);
    prefetch_tmap(&tm_c1);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0;
      bool ok = true;
      int prob, t;
      for (int idx = 0; ok && tile_at(p, cid, idx, prob, t); ++idx) {
        const GemmProblem& P = p.prob[prob];
        const CUtensorMap* ma = prob ? &tm_a1 : &tm_a0;
        const CUtensorMap* mb = prob ? &tm_b1 : &tm_b0;
        const int mrow = (t / P.n_tiles) * 2 * kBM + static_cast<int>(rank) * kBM;  // this CTA's rows of A
        const int ncol = (t % P.n_tiles) * BN + static_cast<int>(rank) * HB;         // this CTA's rows of B
        for (int kb = 0; kb < P.kblocks; ++kb) {
          if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 11)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          const uint32_t fbar = mapa_shared(smem_u32(full + stage), 0);
          if (rank == 0) {
            mbar_arrive_expect_tx(full + stage, 2 * STAGE_BYTES);  // both CTAs' bytes
            armed |= 1u << stage;
          }
          if (!P.a_mn) {
            tma_load_2d_pair(sa, ma, fbar, kb * kBK, mrow);
          } else {
            tma_load_2d_pair(sa, ma, fbar, mrow, kb * kBK);
            tma_load_2d_pair(sa + 8192, ma, fbar, mrow + 64, kb * kBK);
          }
          tma_load_2d_pair(sb, mb, fbar, ncol, kb * kBK);
          tma_load_2d_pair(sb + 8192, mb, fbar, ncol + 64, kb * kBK);
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
    // ------------------------------------------------------------------ UMMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdescK = idesc_bf16_f32(2 * kBM, BN, false, true);
      constexpr uint32_t kIdescMN = idesc_bf16_f32(2 * kBM, BN, true, true);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true, issued = false;
      int prob, t;
      for (int idx = 0; ok && tile_at(p, cid, idx, prob, t); ++idx, ++lt) {
        const GemmProblem& P = p.prob[prob];
        const bool amn = P.a_mn != 0;
        const uint32_t idesc = amn ? kIdescMN : kIdescK;
        const int b = lt & 1;
        const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
        if (!wait_bounded(aempty + b, aph ^ 1u, abort_flag, p.ctl, 12)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < P.kblocks; ++kb) {
          if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 13)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma_bf16_pair(d, slice_desc(amn, sa, k), slice_desc(true, sb, k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit_pair(empty + stage, 0x3);
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(afull + b, 0x3);
      }
      if (!ok && issued) {
        umma_commit_pair(drain, 0x1);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* staging = smem + STAGES * STAGE_BYTES + (warp - 2) * 2 * 4096;
    const uint32_t aempty_leader0 = mapa_shared(smem_u32(aempty), 0);
    const uint32_t aempty_leader1 = mapa_shared(smem_u32(aempty + 1), 0);
    int sbuf = 0, lt = 0;
    int prob, t;
    for (int idx = 0; tile_at(p, cid, idx, prob, t); ++idx, ++lt) {
      const GemmProblem& P = p.prob[prob];
      const CUtensorMap* mc = prob ? &tm_c1 : &tm_c0;
      const int b = lt & 1;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      const bool w = wait_bounded(afull + b, aph, abort_flag, p.ctl, 14);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      const uint32_t acc = lane_base + static_cast<uint32_t>(b * BN);
      const int nb = t % P.n_tiles;
      const int r0 = (t / P.n_tiles) * 2 * kBM + static_cast<int>(rank) * kBM + q * 32;
      const int n_valid = P.Nc - nb * BN;  // columns of this tile inside C
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
        if (lane == 0 && r0 < P.M) {
          const int c0 = nb * BN + ch * 32;
          if (P.accumulate)
            tma_reduce_add_2d(mc, buf, c0, r0);
          else
            tma_store_2d(mc, buf, c0, r0);
          bulk_commit_group();
        }
        sbuf ^= 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(b ? aempty_leader1 : aempty_leader0);
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no cross-CTA signal may target a CTA that has exited
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace

int gemm_smem_bytes() { return SMEM; }

cudaError_t gemm_prepare(int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel, &cfg);
}

cudaError_t launch_gemm_pair(const CUtensorMap& A0, const CUtensorMap& B0, const CUtensorMap& C0, const CUtensorMap& A1,
                             const CUtensorMap& B1, const CUtensorMap& C1, const GemmParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * p.nclusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, A0, B0, C0, A1, B1, C1, p);
}

}  // namespace hylo
