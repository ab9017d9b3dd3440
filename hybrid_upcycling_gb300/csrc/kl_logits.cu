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
// A cluster of kSplit CTAs works on one row at a time, each CTA on a contiguous column slice,
// and the clusters walk the rows. In each CTA a producer warp streams 6144-column chunks of
// its slice with 1-D bulk TMA copies into a 4-stage shared-memory ring; 12 consumer warps
// (three per scheduler) each take 16 columns of a chunk per thread (two 16-byte vectors,
// interleaved so every shared load of a warp is one contiguous 512-byte run). (With 8 warps of
// 32 columns and 8192-column chunks: 12.94 against 12.62 ms for 65536 x 128256.) Pass 1 folds the slice into running
// statistics (shared with the hidden-state kernel); pass 2 (gradient requested) streams the
// slice again and stores dz_s. Each stage carries pass 1 of row k together with pass 2 of
// row k - kLag, so the HBM-bound and the exponential-bound halves of the work overlap.
//
// No warp waits for a row's statistics: at the end of its pass 1 every warp deposits its
// partial and moves on; one warp, rotating with the row (k mod 12), merges the partials,
// exchanges the slice result with the other CTAs of the cluster through DSMEM (stores into
// every CTA's shared memory, release-arrive on its barrier; each CTA merges the kSplit
// partials in rank order, so all hold the same bits), forms lse, KL and the gap in fp32 and
// publishes what pass 2 needs. Pass 2 of row k starts kLag = 2 job-rows later, by which time
// that is long done. (A single warp merging every row while the others waited for it
// serialised ~6 us per row; fp64 on that one thread made it worse.) Every reused slot
// (partials, cluster exchange, row values) has its own full/empty barrier pair; all waits are
// time-bounded.
//
// HBM: pass 2 re-reads the row from DRAM, not L2 (ncu on 8192 x 128256: L2 hit rate ~0%,
// DRAM at 80% of its peak, ~10 B moved per element against 6 algorithmic): between a row's two
// passes every SM streams more than a whole row, >100 MB across the GPU. The consumers are
// about as slow: with pass 2 served from L2 by construction (a timing probe) the launch is only
// 2-4% faster, so the two limits coincide. Splitting rows over a
// cluster shortens that distance but measured slower on GB300 (8192 x 128256, one launch:
// kSplit 1: 1.66 ms, 2: 1.74, 4: 2.18, 8: 3.96): 4- and 8-CTA clusters leave 8 and 32 SMs
// idle (36 and 15 clusters resident), the per-row exchange adds latency that the 3-stage ring
// cannot hide, and even at kSplit 4 only 21% of pass 2 hit L2. L2 eviction-priority hints
// (keep pass-1 lines, drop pass-2 lines and the gradient) changed nothing. So kSplit = 1.
#include "hylo_internal.h"
#include "kl_stats.cuh"

namespace hylo {
namespace {

constexpr int kConsumerWarps = 12;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one producer warp
constexpr int kChunk = 6144;                          // columns per stage
constexpr int kChunkBytes = kChunk * 2;               // per tensor
constexpr int kStages = 4;
constexpr int kStageBytes = 4 * kChunkBytes;  // pass-1 (z_t, z_s) and pass-2 (z_t, z_s) chunks
constexpr int kVecPerThread = 2;              // 2 x 8 columns = 16 per thread per chunk
constexpr int kCols = 8 * kVecPerThread;
static_assert(kConsumerWarps * 32 * kVecPerThread * 8 == kChunk, "chunk split");
constexpr int kTail = 2048;                   // barriers and exchange slots
constexpr int kSmem = 1024 + kStages * kStageBytes + kTail;
constexpr int kSplit = 1;  // CTAs per cluster, one column slice of each row per CTA
constexpr int kLag = 2;    // pass 2 of a row runs this many job-rows after its pass 1

// Partial statistics of one slice as exchanged between the CTAs of a cluster.
struct XStats {
  float v[6];     // mt, st, ms, ss, a, cc
  uint32_t far;
};

// What pass 2 of a row needs: log2(e) lse_t, log2(e) lse_s and -log2(e) (lse_s - lse_t).
struct RowVals {
  float bt, bs, ngl;
};

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

__device__ __forceinline__ RowStats bcast_stats(const RowStats& r) {
  RowStats o;
  o.mt = __shfl_sync(0xffffffffu, r.mt, 0);
  o.st = __shfl_sync(0xffffffffu, r.st, 0);
  o.ms = __shfl_sync(0xffffffffu, r.ms, 0);
  o.ss = __shfl_sync(0xffffffffu, r.ss, 0);
  o.a = __shfl_sync(0xffffffffu, r.a, 0);
  o.cc = __shfl_sync(0xffffffffu, r.cc, 0);
  o.far = __shfl_sync(0xffffffffu, static_cast<int>(r.far), 0) != 0;
  return o;
}

// log1p(u) - u in fp32: by its Taylor series -u^2/2 + u^3/3 - ... through u^11 for |u| < 1/4
// (truncation < 2e-7 relative there), otherwise directly (|result| > 0.026, no cancellation).
__device__ __forceinline__ float log1p_minus_id(float u) {
  if (fabsf(u) < 0.25f) {
    float t = 1.0f / 11.0f;
    t = fmaf(u, t, -1.0f / 10.0f);
    t = fmaf(u, t, 1.0f / 9.0f);
    t = fmaf(u, t, -1.0f / 8.0f);
    t = fmaf(u, t, 1.0f / 7.0f);
    t = fmaf(u, t, -1.0f / 6.0f);
    t = fmaf(u, t, 1.0f / 5.0f);
    t = fmaf(u, t, -1.0f / 4.0f);
    t = fmaf(u, t, 1.0f / 3.0f);
    t = fmaf(u, t, -0.5f);
    return u * u * t;
  }
  return log1pf(u) - u;
}

// Final per-row values from merged statistics, in fp32 (the same forms as kl_from_stats):
// lse_x = m_x/tau + log S_x; with u = C' - mu, KL = C' + (log1p(u) - u) and the gap
// lse_s - lse_t = log1p(u) when the distributions are close, else KL = mu - lse_t + lse_s.
__device__ __forceinline__ float row_final(const RowStats& r, float inv_tau, float& lse_t, float& lse_s,
                                           float& gap) {
  lse_t = r.mt * inv_tau + logf(r.st);
  lse_s = r.ms * inv_tau + logf(r.ss);
  const float mu = r.a / r.st, cn = r.cc / r.st, u = cn - mu;
  if (!r.far && isfinite(u) && fabsf(u) < 0.5f) {
    gap = log1pf(u);
    return cn + log1p_minus_id(u);
  }
  gap = lse_s - lse_t;
  return mu - lse_t + lse_s;
}

// Cluster c (of gridDim.x / kSplit) takes rows c, c + nclusters, ...; CTA rank q of the
// cluster takes columns [q w, (q + 1) w) of each, w = ceil(V / kSplit) rounded up to 8.
// Job-row k of a CTA carries pass 1 of its k-th row and pass 2 of its (k - kLag)-th row.
__global__ void __launch_bounds__(kThreads, 1) kl_logits_kernel(const LogitsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* red_full = empty + kStages;  // [2] all warps' partials of a row deposited
  uint64_t* red_empty = red_full + 2;    // [2] the merging warp has read them
  uint64_t* vals_full = red_empty + 2;   // [2] a row's RowVals published
  uint64_t* xfull = vals_full + 2;       // [2] every CTA's slice partial of a row has arrived here
  uint64_t* xempty = xfull + 2;          // [2] every CTA has read this CTA's partial of a row
  RowStats* warp_stats = reinterpret_cast<RowStats*>(xempty + 2);                  // [2][warps]
  XStats* xstats = reinterpret_cast<XStats*>(warp_stats + 2 * kConsumerWarps);     // [2][kSplit]
  RowVals* rowvals = reinterpret_cast<RowVals*>(xstats + 2 * kSplit);              // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(rowvals + 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(red_full + b, kConsumerWarps);
      mbar_init(red_empty + b, 1);
      mbar_init(vals_full + b, 1);
      mbar_init(xfull + b, kSplit);
      mbar_init(xempty + b, kSplit);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync_all();  // peers arrive on xfull / xempty only after they are initialised

  const uint32_t q = cluster_ctarank();
  const int cl = static_cast<int>(blockIdx.x) / kSplit, ncl = static_cast<int>(gridDim.x) / kSplit;
  const int wslice = ((p.V + kSplit - 1) / kSplit + 7) & ~7;
  const int lo = min(p.V, static_cast<int>(q) * wslice), hi = min(p.V, lo + wslice);
  const int nchunks = (hi - lo + kChunk - 1) / kChunk;
  const bool grad = p.dz != nullptr;
  const int my_rows = p.N > cl ? (p.N - 1 - cl) / ncl + 1 : 0;
  const int job_rows = my_rows + (grad && my_rows > 0 ? kLag : 0);  // the last kLag only finish pass 2

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0;
      bool ok = true;
      for (int k = 0; ok && k < job_rows; ++k) {
        const bool p1 = k < my_rows, p2 = grad && k >= kLag;
        const size_t n1 = static_cast<size_t>(cl) + static_cast<size_t>(k) * ncl;
        const size_t n2 = n1 - static_cast<size_t>(kLag) * ncl;
        for (int ch = 0; ch < nchunks; ++ch) {
          if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 21)) {
            ok = false;
            break;
          }
          const int col0 = lo + ch * kChunk;
          const int cols = min(kChunk, hi - col0);
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
    int vec[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) vec[i] = warp * 32 * kVecPerThread + lane + 32 * i;
    for (int k = 0; ok && k < job_rows; ++k) {
      const bool p1 = k < my_rows, p2 = grad && k >= kLag;
      const int n1 = cl + k * ncl;
      const int n2 = n1 - kLag * ncl;
      float bt = 0.f, bs = 0.f, ngl = 0.f;
      if (p2) {  // the values of row k - kLag, published by its merging warp
        const int b2 = (k - kLag) & 1;
        const bool w = wait_bounded(vals_full + b2, static_cast<uint32_t>((k - kLag) >> 1) & 1u, abort_flag,
                                    p.ctl, 26);
        if (!__all_sync(0xffffffffu, w)) break;
        bt = rowvals[b2].bt;
        bs = rowvals[b2].bs;
        ngl = rowvals[b2].ngl;
      }
      RowStats rs{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
      uint16_t* dz_row = p2 ? p.dz + static_cast<size_t>(n2) * p.ld : nullptr;
      for (int ch = 0; ch < nchunks; ++ch) {
        const bool w = wait_bounded(full + stage, phase, abort_flag, p.ctl, 22);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + stage * kStageBytes;
        const int col0 = lo + ch * kChunk;
        const int cols = min(kChunk, hi - col0);
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
          float zt[kCols], zs[kCols];
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            unpack_bf16x8(reinterpret_cast<const uint4*>(st)[vec[i]], zt + 8 * i);
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + kChunkBytes)[vec[i]], zs + 8 * i);
          }
          if (valid == 0xffffffffu)
            fold_chunk<false, kCols>(rs, zt, zs, valid, p.c, p.inv_tau);
          else if (valid != 0)
            fold_chunk<true, kCols>(rs, zt, zs, valid, p.c, p.inv_tau);
        }
        if (p2) {  // pass 2 of row n2: dz_s = gscale (p_s - p_t)
          float zt[kCols], zs[kCols];
#pragma unroll
          for (int i = 0; i < kVecPerThread; ++i) {
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + 2 * kChunkBytes)[vec[i]], zt + 8 * i);
            unpack_bf16x8(reinterpret_cast<const uint4*>(st + 3 * kChunkBytes)[vec[i]], zs + 8 * i);
          }
          const float2 c2 = make_float2(p.c, p.c), gs2 = make_float2(p.gscale, p.gscale);
          const float2 nbt = make_float2(-bt, -bt), nbs = make_float2(-bs, -bs), ngl2 = make_float2(ngl, ngl);
          uint32_t pk[kCols / 2];
#pragma unroll
          for (int j = 0; j < kCols / 2; ++j) {
            const float2 g = __fmul2_rn(prob_diff2(make_float2(zt[2 * j], zt[2 * j + 1]),
                                                   make_float2(zs[2 * j], zs[2 * j + 1]), c2, nbt, nbs, ngl2),
                                        gs2);
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
      if (!ok) break;
      if (!p1) continue;  // a job-row that only finishes pass 2 of an earlier row
      // ---- row n1: deposit this warp's partial; the row's merging warp takes it from there
      const int b = k & 1;
      const uint32_t use = static_cast<uint32_t>(k >> 1) & 1u;  // phase parity of slot b's current use
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) merge_any(rs, shfl_stats(rs, off), p.c);
      {
        const bool w = wait_bounded(red_empty + b, use ^ 1u, abort_flag, p.ctl, 23);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      if (lane == 0) {
        warp_stats[b * kConsumerWarps + warp] = rs;
        mbar_arrive(red_full + b);
      }
      if (warp != k % kConsumerWarps) continue;
      // ---- merging warp of row n1
      {
        const bool w = wait_bounded(red_full + b, use, abort_flag, p.ctl, 24);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      RowStats r = lane < kConsumerWarps ? warp_stats[b * kConsumerWarps + lane]
                                         : RowStats{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty + b);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) merge_any(r, shfl_stats(r, off), p.c);
      r = bcast_stats(r);  // lane 0's merge order, the same bits in every lane
      // this CTA's slot b in every peer must have been read (row k - 2) before it is rewritten
      {
        const bool w = wait_bounded<true>(xempty + b, use ^ 1u, abort_flag, p.ctl, 25);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      if (lane < kSplit) {  // lane j hands this slice's statistics to CTA j of the cluster
        const uint32_t dst = mapa_shared(smem_u32(&xstats[b * kSplit + static_cast<int>(q)]), lane);
        const float v[6] = {r.mt, r.st, r.ms, r.ss, r.a, r.cc};
#pragma unroll
        for (int i = 0; i < 6; ++i) st_cluster_u32(dst + 4 * i, __float_as_uint(v[i]));
        st_cluster_u32(dst + 24, r.far ? 1u : 0u);
        mbar_arrive_remote(mapa_shared(smem_u32(xfull + b), lane));
      }
      {
        const bool w = wait_bounded<true>(xfull + b, use, abort_flag, p.ctl, 27);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      RowStats m{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
      if (lane == 0) {
        for (int j = 0; j < kSplit; ++j) {  // rank order: every CTA forms the same bits
          const XStats& x = xstats[b * kSplit + j];
          merge_any(m, RowStats{x.v[0], x.v[1], x.v[2], x.v[3], x.v[4], x.v[5], x.far != 0u}, p.c);
        }
      }
      __syncwarp();
      if (lane < kSplit) mbar_arrive_remote(mapa_shared(smem_u32(xempty + b), lane));  // slots read
      if (lane == 0) {
        float lt, ls, gp;
        const float kk = row_final(m, p.inv_tau, lt, ls, gp);
        rowvals[b] = RowVals{lt * kLog2e, ls * kLog2e, -gp * kLog2e};
        mbar_arrive(vals_full + b);
        if (q == 0) {
          p.kl[n1] = kk;
          p.lse_s[n1] = ls;
          p.lse_t[n1] = lt;
        }
      }
    }
  }
  // No CTA may leave while a peer can still store into its shared memory.
  __syncwarp();
  cluster_sync_all();
}

}  // namespace

static cudaLaunchConfig_t logits_config(cudaLaunchAttribute* attr, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kSplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t kl_logits_prepare(int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(kl_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = logits_config(attr, 1, nullptr);
  return cudaOccupancyMaxActiveClusters(max_clusters, kl_logits_kernel, &cfg);
}

cudaError_t launch_kl_logits(const uint16_t* zs, const uint16_t* zt, uint16_t* dz, int64_t ld, int N, int V, float tau,
                             float gscale, float* kl, float* lse_s, float* lse_t, const WaitCtl& ctl, int clusters,
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
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = logits_config(attr, clusters, stream);
  return cudaLaunchKernelEx(&cfg, kl_logits_kernel, p);
}

}  // namespace hylo
