// Fused hidden-state KL on sm_103a: one persistent, warp-specialised kernel that computes
// the teacher and student logit tiles z_t = h_t W_t^T and z_s = h_s W_s^T on the tensor cores
// (tcgen05 UMMA, TMA-fed 128-byte-swizzled operands, fp32 accumulators in TMEM) and consumes
// them in the epilogue without writing logits to memory.
//
//   forward : folds each tile into running per-token softmax/KL statistics (online softmax
//             rescaled by the running max) and writes one set of partial statistics per
//             (token, vocabulary segment); a small combine kernel merges the segments.
//   backward: recomputes the tiles, forms G = grad_scale (p_s - p_t) / (tau N) from the saved
//             log-sum-exps and writes G in bf16 for the gradient GEMMs.
//
// The operation is the Stage-II distillation loss of the HyLo pages: the "Fused Hidden-State
// KL" that skips the teacher LM head and fuses softmax+KL (Long-Context Aware Upcycling
// digest, ftxj.github.io, section Method), with the KL between the student's and the teacher's
// next-token distributions, kl_weight 1.0, no cross-entropy (HyLo-Llama-8MLA8GDN-8K-SFT reading
// notes, kwkr.cn, section "two-stage training recipe", Stage II).
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues the UMMAs, warps
// 2..5 are the epilogue; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31, so each epilogue
// thread owns one token row of the 128-row tile and needs no cross-thread reduction.
#include <cfloat>
#include <cmath>

#include "hylo_internal.h"

namespace hylo {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

template <bool BWD>
struct FusedCfg {
  static constexpr int BN = kFusedBN;
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 4;
  // backward: per epilogue warp two staging buffers of 32 rows x 64 bf16 (128 B rows)
  static constexpr int STAGING_BYTES = BWD ? 4 * 2 * 32 * 128 : 0;
  static constexpr int NBUF = 512 / (2 * BN);  // TMEM buffers holding a (teacher, student) tile pair
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES + STAGING_BYTES;
  static constexpr int NBARS = 2 * STAGES + 2 * NBUF + 1;
  static constexpr int SMEM = 1024 + BAR_OFF + NBARS * 8 + 16;
  static_assert(NBUF >= 1, "TMEM holds at least one tile pair");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Waits used only while draining after an abort: time-limited, ignore the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ void unit_range(const FusedParams& p, int u, int& row0, int& vt0, int& vt1, int& seg) {
  const int ti = u / p.nseg;
  seg = u - ti * p.nseg;
  row0 = ti * kBM;
  vt0 = static_cast<int>((static_cast<long long>(seg) * p.vtiles) / p.nseg);
  vt1 = static_cast<int>((static_cast<long long>(seg + 1) * p.vtiles) / p.nseg);
}

// Running statistics of one token row over the vocabulary columns seen so far. Maxima are in
// raw logit units; sums are relative to exp(max / tau).
struct RowStats {
  float mt, st;  // teacher running max, sum_v exp((z_t - mt)/tau)
  float ms, ss;  // student running max, sum_v exp((z_s - ms)/tau)
  float a;       // sum_v exp((z_t - mt)/tau) * d_v, with d_v = (z_t - z_s)/tau
  float cc;      // sum_v exp((z_t - mt)/tau) * (exp(-d_v) - 1 + d_v)   (each term >= 0)
};

// g(d) = exp(-d) - 1 + d for |d| < 1/4 by its Taylor series through d^7 (truncation < 1e-8
// relative there); used so that near-identical distributions lose no digits to cancellation.
__device__ __forceinline__ float g_series(float d) {
  float t = fmaf(d, -1.0f / 5040.0f, 1.0f / 720.0f);
  t = fmaf(d, t, -1.0f / 120.0f);
  t = fmaf(d, t, 1.0f / 24.0f);
  t = fmaf(d, t, -1.0f / 6.0f);
  t = fmaf(d, t, 0.5f);
  return d * d * t;
}

// Folds 32 columns of one row into the running statistics. `valid` = number of columns of
// this chunk that lie inside the vocabulary (32 except in the last tile; MASKED only there).
template <bool MASKED>
__device__ __forceinline__ void fold_chunk(RowStats& r, const float (&zt)[32], const float (&zs)[32], int valid,
                                           float c, float inv_tau) {
  float cmt = -INFINITY, cms = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (!MASKED || j < valid) {
      cmt = fmaxf(cmt, zt[j]);
      cms = fmaxf(cms, zs[j]);
    }
  }
  const float nmt = fmaxf(r.mt, cmt);
  const float nms = fmaxf(r.ms, cms);
  const float at = ex2_approx((r.mt - nmt) * c);  // 0 on the first chunk (r.mt = -inf)
  const float as = ex2_approx((r.ms - nms) * c);
  r.st *= at;
  r.a *= at;
  r.cc *= at;
  r.ss *= as;
  r.mt = nmt;
  r.ms = nms;
  const float mtc = nmt * c, msc = nms * c;
  // K = exp((m_s - m_t)/tau) relates student exponentials to the teacher max:
  // es * K = exp((z_s - m_t)/tau) = et * exp(-d). Clamped so it stays finite; when the clamp
  // matters the combine step uses the direct formula instead of the cancellation-free one.
  const float K = ex2_approx(fminf((nms - nmt) * c, 126.0f));
  float st = 0.f, ss = 0.f, a = 0.f, cc = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const bool ok = !MASKED || j < valid;
    const float et = ok ? ex2_approx(fmaf(zt[j], c, -mtc)) : 0.f;
    const float es = ok ? ex2_approx(fmaf(zs[j], c, -msc)) : 0.f;
    const float d = ok ? (zt[j] - zs[j]) * inv_tau : 0.f;
    st += et;
    ss += es;
    a = fmaf(et, d, a);
    const float big = fmaf(es, K, fmaf(et, d, -et));
    cc += (fabsf(d) < 0.25f) ? et * g_series(d) : big;
  }
  r.st += st;
  r.ss += ss;
  r.a += a;
  r.cc += cc;
}

template <bool BWD>
__global__ void __launch_bounds__(kThreads, 1)
fused_kl_kernel(const __grid_constant__ CUtensorMap tm_hs, const __grid_constant__ CUtensorMap tm_Ws,
                const __grid_constant__ CUtensorMap tm_ht, const __grid_constant__ CUtensorMap tm_Wt,
                const __grid_constant__ CUtensorMap tm_G, const FusedParams p) {
  using C = FusedCfg<BWD>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::NBUF;
  uint64_t* drain = tempty + C::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_hs);
    prefetch_tmap(&tm_Ws);
    prefetch_tmap(&tm_ht);
    prefetch_tmap(&tm_Wt);
    if (BWD) prefetch_tmap(&tm_G);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kbt = p.kb_t, kbtot = p.kb_t + p.kb_s;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has been armed at least once
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int row0, vt0, vt1, seg;
        unit_range(p, u, row0, vt0, vt1, seg);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int col0 = vt * BN;
          for (int kb = 0; kb < kbtot; ++kb) {
            if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 1)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * C::STAGE_BYTES;
            uint8_t* sb = sa + C::A_BYTES;
            mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
            armed |= 1u << stage;
            if (kb < kbt) {
              tma_load_2d(sa, &tm_ht, full + stage, kb * kBK, row0);
              tma_load_2d(sb, &tm_Wt, full + stage, kb * kBK, col0);
            } else {
              const int k = kb - kbt;
              tma_load_2d(sa, &tm_hs, full + stage, k * kBK, row0);
              tma_load_2d(sb, &tm_Ws, full + stage, k * kBK, col0);
            }
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let every armed load land before the CTA can exit: the latest armed phase of stage s
        // has parity `phase` for stages below the current one and `phase ^ 1` otherwise.
        for (int s = 0; s < C::STAGES; ++s) {
          if (armed & (1u << s)) drain_wait(full + s, s < stage ? phase : (phase ^ 1u), 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int row0, vt0, vt1, seg;
        unit_range(p, u, row0, vt0, vt1, seg);
        for (int vt = vt0; ok && vt < vt1; ++vt, ++lt) {
          const int b = lt % C::NBUF;
          const uint32_t tph = static_cast<uint32_t>(lt / C::NBUF) & 1u;
          if (!wait_bounded(tempty + b, tph ^ 1u, abort_flag, p.ctl, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dT = tmem_base + static_cast<uint32_t>(b * 2 * BN);
          const uint32_t dS = dT + BN;
          for (int kb = 0; kb < kbtot; ++kb) {
            if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
            const bool teacher = kb < kbt;
            const uint32_t d = teacher ? dT : dS;
            const int kk = teacher ? kb : kb - kbt;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              umma_bf16(d, smem_desc_sw128(sa + k * 32, 0, 1024), smem_desc_sw128(sb + k * 32, 0, 1024), kIdesc,
                        (kk > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(empty + stage);
            issued = true;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(tfull + b);
        }
      }
      if (!ok && issued) {
        umma_commit(drain);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int lt = 0;
    bool ok = true;
    int sbuf = 0;
    uint8_t* staging = smem + C::STAGES * C::STAGE_BYTES + (warp - 2) * 2 * 4096;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      int row0, vt0, vt1, seg;
      unit_range(p, u, row0, vt0, vt1, seg);
      const int token = row0 + row;
      RowStats rs{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f};
      float bt = 0.f, bs = 0.f;
      if (BWD && token < p.N) {
        bt = p.lse_t[token] * kLog2e;
        bs = p.lse_s[token] * kLog2e;
      }
      for (int vt = vt0; vt < vt1; ++vt, ++lt) {
        const int b = lt % C::NBUF;
        const uint32_t tph = static_cast<uint32_t>(lt / C::NBUF) & 1u;
        bool w = wait_bounded(tfull + b, tph, abort_flag, p.ctl, 4);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tT = lane_base + static_cast<uint32_t>(b * 2 * BN);
        const uint32_t tS = tT + BN;
        if (!BWD) {
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            float zt[32], zs[32];
            tmem_ld32(tT + ch * 32, zt);
            tmem_ld32(tS + ch * 32, zs);
            tmem_ld_wait();
            const int col = vt * BN + ch * 32;
            const int valid = min(32, p.V - col);
            if (valid >= 32) {
              fold_chunk<false>(rs, zt, zs, 32, p.c, p.inv_tau);
            } else if (valid > 0) {
              fold_chunk<true>(rs, zt, zs, valid, p.c, p.inv_tau);
            }
          }
        } else {
#pragma unroll 1
          for (int ch2 = 0; ch2 < BN / 64; ++ch2) {
            uint8_t* buf = staging + sbuf * 4096;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            const uint32_t rowaddr = smem_u32(buf) + lane * 128;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float zt[32], zs[32];
              tmem_ld32(tT + ch2 * 64 + half * 32, zt);
              tmem_ld32(tS + ch2 * 64 + half * 32, zs);
              tmem_ld_wait();
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float pt0 = ex2_approx(fmaf(zt[2 * j], p.c, -bt));
                const float ps0 = ex2_approx(fmaf(zs[2 * j], p.c, -bs));
                const float pt1 = ex2_approx(fmaf(zt[2 * j + 1], p.c, -bt));
                const float ps1 = ex2_approx(fmaf(zs[2 * j + 1], p.c, -bs));
                pk[j] = pack_bf16x2((ps0 - pt0) * p.gscale, (ps1 - pt1) * p.gscale);
              }
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const uint32_t chunk = static_cast<uint32_t>((half * 4 + c4) ^ (lane & 7));
                st_shared_v4(rowaddr + chunk * 16, pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_G, buf, vt * BN + ch2 * 64, row0 + q * 32);
              bulk_commit_group();
            }
            sbuf ^= 1;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty + b);
      }
      if (!ok) break;
      if (!BWD && token < p.N) {
        const size_t NS = static_cast<size_t>(p.N);
        float* base = p.part + static_cast<size_t>(seg) * NS + token;
        const size_t fs = static_cast<size_t>(p.nseg) * NS;  // stride between fields
        base[0 * fs] = rs.mt;
        base[1 * fs] = rs.st;
        base[2 * fs] = rs.ms;
        base[3 * fs] = rs.ss;
        base[4 * fs] = rs.a;
        base[5 * fs] = rs.cc;
      }
    }
    if (BWD && lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Merges the per-segment statistics of each token (fp64) and writes kl, lse_s, lse_t.
// KL = A/S_t - lse_t + lse_s in general; when the two distributions are close the algebraically
// equal form KL = C' + log1p(C' - mu) - (C' - mu), with mu = A/S_t = E_pt[d] and
// C' = C/S_t = E_pt[exp(-d) - 1 + d] >= 0, avoids the cancellation of two ~log V terms.
__global__ void kl_combine_kernel(const float* __restrict__ part, int N, int nseg, float inv_tau,
                                  float* __restrict__ kl, float* __restrict__ lse_s, float* __restrict__ lse_t) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const size_t NS = static_cast<size_t>(N);
  const size_t fs = static_cast<size_t>(nseg) * NS;
  const float* b = part + n;
  double Mt = -INFINITY, Ms = -INFINITY;
  for (int s = 0; s < nseg; ++s) {
    Mt = fmax(Mt, static_cast<double>(b[s * NS]));
    Ms = fmax(Ms, static_cast<double>(b[2 * fs + s * NS]));
  }
  double St = 0, Ss = 0, A = 0, Cc = 0;
  const double it = inv_tau;
  for (int s = 0; s < nseg; ++s) {
    const double mt = b[s * NS], ms = b[2 * fs + s * NS];
    const double wt = (mt == -INFINITY) ? 0.0 : exp((mt - Mt) * it);
    const double ws = (ms == -INFINITY) ? 0.0 : exp((ms - Ms) * it);
    St += wt * b[fs + s * NS];
    A += wt * b[4 * fs + s * NS];
    Cc += wt * b[5 * fs + s * NS];
    Ss += ws * b[3 * fs + s * NS];
  }
  const double lt = Mt * it + log(St);
  const double ls = Ms * it + log(Ss);
  const double mu = A / St;
  const double cn = Cc / St;
  const double u = cn - mu;
  double k;
  if (isfinite(u) && fabs(u) < 0.5) {
    k = cn + (log1p(u) - u);
  } else {
    k = mu - lt + ls;
  }
  kl[n] = static_cast<float>(k);
  lse_s[n] = static_cast<float>(ls);
  lse_t[n] = static_cast<float>(lt);
}

// loss[0] = mean(kl[0..N)) with a fixed-order fp64 reduction (one block).
__global__ void __launch_bounds__(1024) kl_mean_kernel(const float* __restrict__ kl, int N, float* loss) {
  __shared__ double red[1024];
  double s = 0;
  for (int i = threadIdx.x; i < N; i += 1024) s += static_cast<double>(kl[i]);
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[0] = static_cast<float>(red[0] / static_cast<double>(N));
}

}  // namespace

int fused_smem_bytes(bool backward) { return backward ? FusedCfg<true>::SMEM : FusedCfg<false>::SMEM; }

cudaError_t fused_prepare(bool backward) {
  if (backward)
    return cudaFuncSetAttribute(fused_kl_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FusedCfg<true>::SMEM);
  return cudaFuncSetAttribute(fused_kl_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FusedCfg<false>::SMEM);
}

cudaError_t launch_fused(bool backward, const CUtensorMap& hs, const CUtensorMap& Ws, const CUtensorMap& ht,
                         const CUtensorMap& Wt, const CUtensorMap& G, const FusedParams& p, int grid,
                         cudaStream_t stream) {
  if (backward) {
    fused_kl_kernel<true><<<grid, kThreads, FusedCfg<true>::SMEM, stream>>>(hs, Ws, ht, Wt, G, p);
  } else {
    fused_kl_kernel<false><<<grid, kThreads, FusedCfg<false>::SMEM, stream>>>(hs, Ws, ht, Wt, G, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* part, int N, int nseg, float inv_tau, float* kl, float* lse_s,
                           float* lse_t, cudaStream_t stream) {
  const int threads = 256;
  kl_combine_kernel<<<(N + threads - 1) / threads, threads, 0, stream>>>(part, N, nseg, inv_tau, kl, lse_s, lse_t);
  return cudaGetLastError();
}

cudaError_t launch_mean(const float* kl, int N, float* loss, cudaStream_t stream) {
  kl_mean_kernel<<<1, 1024, 0, stream>>>(kl, N, loss);
  return cudaGetLastError();
}

}  // namespace hylo
