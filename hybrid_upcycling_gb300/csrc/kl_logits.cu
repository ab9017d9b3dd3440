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
// One persistent CTA per SM walks its rows. A producer warp streams 8192-column chunks with
// 1-D bulk TMA copies into a 3-stage shared-memory ring; 8 consumer warps each take 32 columns
// of a chunk per thread (four 16-byte vectors, interleaved so every shared load of a warp is
// one contiguous 512-byte run). Pass 1 of a row folds its chunks into running statistics
// (shared with the hidden-state kernel); the CTA merges them through bounded mbarrier
// handoffs and one thread forms KL and the lse's in fp64. Pass 2 (gradient requested) streams
// the row again -- from L2 -- and stores dz_s. The two passes are software-pipelined across
// rows: stage k carries chunk c of row k (pass 1, from HBM) together with chunk c of row k-1
// (pass 2, from L2), so the HBM-bound and the exponential-bound halves of the work overlap.
// HBM traffic per element: 4 B read (+ 2 B written with the gradient) if pass 2 hits L2. It
// mostly does not: between a row's two passes the other SMs stream ~78 MB of logits plus their
// gradients, so pass 2 re-fetches from DRAM (ncu: L2 hit rate 0.4%, DRAM at 78% of peak,
// ~10 B moved per element). Keeping rows in shared memory across a cluster of 8 CTAs removed
// the re-fetch but serialised a per-row cross-CTA handoff and ran 3x slower; L2 eviction
// hints on the copies changed nothing measurable.
#include "hylo_internal.h"
#include "kl_stats.cuh"

namespace hylo {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one producer warp
constexpr int kChunk = 8192;                          // columns per stage
constexpr int kChunkBytes = kChunk * 2;               // per tensor
constexpr int kStages = 3;
constexpr int kStageBytes = 4 * kChunkBytes;  // pass-1 (z_t, z_s) and pass-2 (z_t, z_s) chunks
constexpr int kVecPerThread = 4;                      // 4 x 8 columns = 32 per thread per chunk
static_assert(kConsumerWarps * 32 * kVecPerThread * 8 == kChunk, "chunk split");
constexpr int kSmem = 1024 + kStages * kStageBytes + 1024;

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
  WaitCtl ctl;
};

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* z) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(w[i] << 16);
    z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
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

// Row of job-row k for this CTA (k = 0, 1, ...): blockIdx.x + k * gridDim.x.
__global__ void __launch_bounds__(kThreads, 1) kl_logits_kernel(const LogitsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* red_full = empty + kStages;  // consumer warps -> warp 0: per-warp statistics written
  uint64_t* red_done = red_full + 1;     // warp 0 -> consumers: row lse ready
  RowStats* warp_stats = reinterpret_cast<RowStats*>(red_done + 1);
  float* row_lse = reinterpret_cast<float*>(warp_stats + kConsumerWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(row_lse + 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    mbar_init(red_full, kConsumerWarps);
    mbar_init(red_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int nchunks = (p.V + kChunk - 1) / kChunk;
  const bool grad = p.dz != nullptr;
  const int my_rows = p.N > static_cast<int>(blockIdx.x) ? (p.N - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int job_rows = my_rows + (grad ? 1 : 0);  // the last job-row only finishes pass 2

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0;
      bool ok = true;
      for (int k = 0; ok && k < job_rows; ++k) {
        const bool p1 = k < my_rows, p2 = grad && k >= 1;
        const size_t n1 = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(k) * gridDim.x;
        const size_t n2 = n1 - gridDim.x;
        for (int ch = 0; ch < nchunks; ++ch) {
          if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 21)) {
            ok = false;
            break;
          }
          const int col0 = ch * kChunk;
          const int cols = min(kChunk, p.V - col0);
          const uint32_t bytes = static_cast<uint32_t>((cols + 7) & ~7) * 2u;  // within the row stride
          uint8_t* st = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(full + stage, (p1 ? 2 * bytes : 0u) + (p2 ? 2 * bytes : 0u));
          armed |= 1u << stage;
          if (p1) {
            bulk_load_1d(st, p.zt + n1 * p.ld + col0, bytes, full + stage);
            bulk_load_1d(st + kChunkBytes, p.zs + n1 * p.ld + col0, bytes, full + stage);
          }
          if (p2) {
            bulk_load_1d(st + 2 * kChunkBytes, p.zt + n2 * p.ld + col0, bytes, full + stage);
            bulk_load_1d(st + 3 * kChunkBytes, p.zs + n2 * p.ld + col0, bytes, full + stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < kStages; ++s) {
          if (!(armed & (1u << s))) continue;
          const uint32_t par = s < stage ? phase : (phase ^ 1u);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(full + s), par) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------------- consumers
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    float bt = 0.f, bs = 0.f;  // log2(e) * lse of the row whose gradient this job-row writes
    int vec[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) vec[i] = warp * 32 * kVecPerThread + lane + 32 * i;
    for (int k = 0; ok && k < job_rows; ++k) {
      const bool p1 = k < my_rows, p2 = grad && k >= 1;
      const int n1 = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
      const int n2 = n1 - static_cast<int>(gridDim.x);
      RowStats rs{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
      uint16_t* dz_row = p2 ? p.dz + static_cast<size_t>(n2) * p.ld : nullptr;
      for (int ch = 0; ch < nchunks; ++ch) {
        const bool w = wait_bounded(full + stage, phase, abort_flag, p.ctl, 22);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + stage * kStageBytes;
        const int col0 = ch * kChunk;
        const int cols = min(kChunk, p.V - col0);
        uint32_t valid = 0xffffffffu;
        if (cols < kChunk) {
          valid = 0;
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            const int left = cols - vec[i] * 8;  // valid columns in this vector
            const uint32_t m = left >= 8 ? 0xffu : (left > 0 ? ((1u << left) - 1u) : 0u);
            valid |= m << (8 * i);
          }
        }
        if (p1) {  // pass 1 of row n1: fold
          float zt[32], zs[32];
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            unpack_bf16x8(reinterpret_cast<const uint4*>(st)[vec[i]], zt + 8 * i);
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + kChunkBytes)[vec[i]], zs + 8 * i);
          }
          if (valid == 0xffffffffu)
            fold_chunk<false>(rs, zt, zs, valid, p.c, p.inv_tau);
          else if (valid != 0)
            fold_chunk<true>(rs, zt, zs, valid, p.c, p.inv_tau);
        }
        if (p2) {  // pass 2 of row n2: dz_s = gscale (p_s - p_t), p_x = 2^(z_x log2(e)/tau - lse_x log2(e))
          float zt[32], zs[32];
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + 2 * kChunkBytes)[vec[i]], zt + 8 * i);
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + 3 * kChunkBytes)[vec[i]], zs + 8 * i);
          }
          const float2 c2 = make_float2(p.c, p.c), gs2 = make_float2(p.gscale, p.gscale);
          const float2 nbt = make_float2(-bt, -bt), nbs = make_float2(-bs, -bs), m1 = make_float2(-1.f, -1.f);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 pt = ex2_approx2(__ffma2_rn(make_float2(zt[2 * j], zt[2 * j + 1]), c2, nbt));
            const float2 ps = ex2_approx2(__ffma2_rn(make_float2(zs[2 * j], zs[2 * j + 1]), c2, nbs));
            const float2 g = __fmul2_rn(__ffma2_rn(pt, m1, ps), gs2);
            pk[j] = pack_bf16x2(g.x, g.y);
          }
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            const uint32_t m = (valid >> (8 * i)) & 0xffu;
            uint16_t* dst = dz_row + col0 + vec[i] * 8;
            if (m == 0xffu) {
              __stcs(reinterpret_cast<uint4*>(dst), make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]));
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if ((m >> j) & 1u) dst[j] = static_cast<uint16_t>((pk[4 * i + (j >> 1)] >> (16 * (j & 1))) & 0xffffu);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok || !p1) break;
      // merge row n1's statistics: warps -> shared memory -> warp 0 -> kl, lse (and bt, bs for
      // the pass 2 of row n1 in the next job-row)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) merge_any(rs, shfl_stats(rs, off), p.c);
      const uint32_t par = static_cast<uint32_t>(k & 1);
      if (lane == 0) {
        warp_stats[warp] = rs;
        mbar_arrive(red_full);
      }
      if (warp == 0) {
        const bool w = wait_bounded(red_full, par, abort_flag, p.ctl, 23);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        RowStats r = lane < kConsumerWarps ? warp_stats[lane]
                                           : RowStats{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) merge_any(r, shfl_stats(r, off), p.c);
        if (lane == 0) {
          double lt, ls;
          const double kk = kl_from_stats(r.mt, r.st, r.ms, r.ss, r.a, r.cc, r.far, p.inv_tau, lt, ls);
          p.kl[n1] = static_cast<float>(kk);
          p.lse_s[n1] = static_cast<float>(ls);
          p.lse_t[n1] = static_cast<float>(lt);
          row_lse[0] = static_cast<float>(lt);
          row_lse[1] = static_cast<float>(ls);
          mbar_arrive(red_done);
        }
      }
      const bool w = wait_bounded(red_done, par, abort_flag, p.ctl, 24);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      bt = row_lse[0] * kLog2e;
      bs = row_lse[1] * kLog2e;
    }
  }
}

}  // namespace

cudaError_t kl_logits_prepare() {
  return cudaFuncSetAttribute(kl_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_kl_logits(const uint16_t* zs, const uint16_t* zt, uint16_t* dz, int64_t ld, int N, int V, float tau,
                             float gscale, float* kl, float* lse_s, float* lse_t, const WaitCtl& ctl, int grid,
                             cudaStream_t stream) {
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
  p.ctl = ctl;
  kl_logits_kernel<<<grid, kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hylo
