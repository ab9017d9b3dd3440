// Fused hidden-state KL forward on sm_103a: one persistent, warp-specialised kernel that
// computes the teacher and student logit tiles z_t = h_t W_t^T and z_s = h_s W_s^T on the tensor
// cores (tcgen05 UMMA, TMA-fed 128-byte-swizzled operands, fp32 accumulators in TMEM) and folds
// them in the epilogue into running per-token softmax/KL statistics (online softmax rescaled by
// the running max), without writing logits to memory. It writes one set of partial statistics
// per (token, vocabulary segment); a small combine kernel merges the segments. (The backward,
// which recomputes the same tiles, is kl_bwd_pipe.cu.)
//
// The operation is the Stage-II distillation loss of the HyLo pages: the "Fused Hidden-State
// KL" that skips the teacher LM head and fuses softmax+KL (Long-Context Aware Upcycling
// digest, ftxj.github.io, section Method), with the KL between the student's and the teacher's
// next-token distributions, kl_weight 1.0, no cross-entropy (HyLo-Llama-8MLA8GDN-8K-SFT reading
// notes, kwkr.cn, section "two-stage training recipe", Stage II).
//
// Roles (384 threads per CTA): warp 0 issues the TMA loads, warp 1 of the even CTA owns TMEM
// and issues the UMMAs for the pair, warp 2 of the even CTA paces the pair against the other
// clusters on its vocabulary segment, warps 4..11 are the epilogue (warpgroup 0 gives registers
// to the two epilogue warpgroups: setmaxnreg 56 / 224). Warp w may read only TMEM lanes
// 32*(w%4) .. 32*(w%4)+31, so each epilogue thread owns one token row of its CTA's 128-row
// tile: warps 4..7 take columns 0..127 of the 256-column tile, warps 8..11 columns 128..255.
// TMEM: the teacher tile in columns 0..255 (half 0), the student tile in 256..511 (half 1).
// The UMMA warp signals half 0 as soon as the teacher UMMAs are done; the epilogue copies its
// row's 128 teacher logits into registers and frees half 0, so the next tile's teacher UMMAs
// (two thirds of its work at d_t = 2 d_s) run while the epilogue folds the student tile, and
// half 1 is free again long before the next student UMMAs.
#include <cfloat>
#include <cmath>

#include "hylo_internal.h"
#include "kl_stats.cuh"

namespace hylo {
namespace {

constexpr int kEpiWarps = 8;                   // two per TMEM lane quarter, one per column half
constexpr int kEpiWarp0 = 4;                   // first epilogue warp (warpgroups 1 and 2)
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kRegsControl = 56;               // per thread, warpgroup 0 (TMA, UMMA)
constexpr int kRegsEpilogue = 224;             // per thread, warpgroups 1 and 2
static_assert(128 * kRegsControl + 256 * kRegsEpilogue <= kThreads * 168, "register split");

// A CTA pair (cluster of 2 on an SM pair) computes a 256-token x BN-word tile with one
// tcgen05.mma.cta_group::2 per 16-deep slice (M = 256): each CTA stages its 128 token rows of
// h and BN/2 rows of W, and each CTA's TMEM holds its 128 rows of the teacher and student
// tiles. kFusedBN = 256: one (teacher, student) pair fills the 512 TMEM columns. (BN = 128
// would fit two pairs, but N = 128 UMMAs measured 22% slower end to end on GB300, on one CTA
// or on a pair.)
template <int BN_>
struct FusedCfg {
  static constexpr int BN = BN_;         // vocabulary columns per pair tile
  static constexpr int HB = BN / 2;      // W rows staged per CTA
  static constexpr int HALF = BN / 2;    // columns per epilogue warp
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = HB * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // as many stages as fit beside the alignment pad and the barriers (7 at BN = 256)
  static constexpr int STAGES = (232448 - 1024 - 256) / STAGE_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  // full[S], empty[S], tfull[2], tempty[2] (teacher half, student half), merge_full, merge_empty, drain
  static constexpr int NBARS = 2 * STAGES + 4 + 3;
  // then the TMEM address, the abort flag and the pacing permit
  static constexpr int SMEM = 1024 + BAR_OFF + NBARS * 8 + 32;
  static_assert(2 * BN == 512 && HALF % 64 == 0 && HB % 8 == 0, "tile shape");
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

// Pacing of clusters that share a vocabulary segment. The units a cluster runs at the same
// index k as its peers read the same LM-head tiles in the same order; left alone, clusters
// drift apart by more tiles than L2 holds and each re-reads the tiles from DRAM (measured on
// the 64K forward: ~190 GB of DRAM reads per launch). Before loading a vocabulary tile, the
// even CTA's producer publishes its position (k, tile) and starts the tile only once every
// peer has reached at least tile - kPaceLead of the same unit index (or finished all its
// units). The peers' words are polled by a warp of its own (pace_peers), which publishes in
// shared memory how far the producer may go, so the producer's loads never wait on those
// global-memory round trips. The wait is a hint: a producer that waits longer than kPaceWaitNs
// (a peer not resident, e.g. SMs held by another kernel) sets the switch in slot kMaxClusters
// and from then on no producer of the launch paces, so a late peer costs at most one such
// wait, never correctness.
// (Measured: DRAM reads of the 64K forward ~250 -> ~70 GB, 3-7% less time per kernel.)
// Every word carries the launch's 16-bit epoch in its top bits, so the counters need no
// clearing between launches: a word from an earlier launch reads as "not started yet", and the
// switch is on only while it holds this launch's epoch. Low 48 bits: (k << 24) | tile.
constexpr unsigned long long kPaceLead = 2;
constexpr unsigned long long kPaceWaitNs = 200000ull;
constexpr unsigned long long kPaceLow = (1ull << 48) - 1;  // low-bits value meaning "no more units"

// Work unit u = (256-token pair tile, vocabulary segment); row0 = the pair tile's first token.
__device__ __forceinline__ void unit_range(const FusedParams& p, int u, int& row0, int& vt0, int& vt1, int& seg) {
  // Grouped raster: units run group by group (p.group pair tiles x every segment), segment-major
  // inside a group. The clusters active at any time then share few segments, each swept in the
  // same order by many clusters (its LM-head tiles come from DRAM about once and from L2 for the
  // others), while the group's hidden-state tiles, re-read for every vocabulary tile, stay
  // within an L2-sized working set.
  const int per_group = p.group * p.nseg;
  const int g = u / per_group;
  const int t0 = g * p.group;
  const int gt = min(p.group, p.token_tiles - t0);  // pair tiles in this group (the last may be short)
  const int r = u - g * per_group;
  seg = r / gt;
  const int ti = t0 + (r - seg * gt);
  row0 = ti * 2 * kBM;
  vt0 = static_cast<int>((static_cast<long long>(seg) * p.vtiles) / p.nseg);
  vt1 = static_cast<int>((static_cast<long long>(seg + 1) * p.vtiles) / p.nseg);
}

// The pacing warp of the even CTA. For each of the cluster's units in turn it polls the words of
// the peers on the same segment (independent loads, eight at a time) and stores in `permit` one
// more than the furthest position ((unit index << 24) | tile) the producer may start: kPaceLead
// tiles past the slowest peer, 0 while a peer has not started the unit index, and past the
// unit's last tile once no peer can hold it back any more. `permit` only grows; it becomes
// unlimited once pacing is switched off. The warp ends after the last unit, on an abort, or
// after kPaceGiveUpNs without any peer moving (then it switches pacing off itself).
constexpr unsigned long long kPaceGiveUpNs = 8 * kPaceWaitNs;

__device__ void pace_peers(const FusedParams& p, int cid, int ncl, volatile unsigned long long* permit,
                           volatile int* abort_flag) {
  volatile unsigned long long* prog = p.progress;
  const unsigned long long ep = static_cast<unsigned long long>(p.epoch) << 48;
  unsigned long long given = 0;  // the value last stored in permit
  for (int u = cid, kunit = 0; u < p.units; u += ncl, ++kunit) {
    int row0, vt0, vt1, seg;
    unit_range(p, u, row0, vt0, vt1, seg);
    uint32_t pend[kMaxClusters / 32] = {};  // bit j: cluster j's unit at this index is on this segment
    for (int j = 0; j < ncl; ++j) {
      const int uj = j + kunit * ncl;
      if (j == cid || uj >= p.units) continue;
      int r_, a_, b_, sj;
      unit_range(p, uj, r_, a_, b_, sj);
      if (sj == seg) pend[j >> 5] |= 1u << (j & 31);
    }
    const unsigned long long last = (static_cast<unsigned long long>(kunit) << 24) |
                                    static_cast<unsigned long long>(vt1 - vt0 - 1);
    uint64_t t_move = globaltimer_ns();
    unsigned long long seen = 0;  // sum of the pending peers' positions at the last poll
    while (true) {
      if (*abort_flag) return;
      if (prog[kMaxClusters] == ep) {  // pacing was switched off for this launch
        *permit = ~0ull;
        return;
      }
      unsigned long long allow = last + 1, sum = 0;
      bool pending = false;
#pragma unroll 1
      for (int w = 0; w < kMaxClusters / 32; ++w) {
        uint32_t bits = pend[w];
        while (bits != 0u) {
          int js[8];
          unsigned long long vs[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            js[i] = bits != 0u ? 32 * w + __ffs(static_cast<int>(bits)) - 1 : -1;
            bits &= bits - 1u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) vs[i] = js[i] >= 0 ? prog[js[i]] : 0ull;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (js[i] < 0) continue;
            const unsigned long long v = vs[i];
            const unsigned long long lo = v & kPaceLow;
            if ((v & ~kPaceLow) != ep) {  // not started in this launch: holds everything back
              allow = 0;
              pending = true;
            } else if (lo == kPaceLow || lo + kPaceLead >= last) {  // can no longer hold this unit back
              pend[w] &= ~(1u << (js[i] & 31));
            } else {
              allow = min(allow, lo + kPaceLead + 1);
              sum += lo + 1;
              pending = true;
            }
          }
        }
      }
      if (allow > given) {
        given = allow;
        *permit = allow;
      }
      if (!pending) break;
      const uint64_t now = globaltimer_ns();
      if (sum != seen) {
        seen = sum;
        t_move = now;
      } else if (now - t_move > kPaceGiveUpNs) {  // no peer moved: give up pacing for the launch
        prog[kMaxClusters] = ep;
        *permit = ~0ull;
        return;
      }
      __nanosleep(200);
    }
  }
}

template <int BN_>
__global__ void __launch_bounds__(kThreads, 1)
fused_kl_kernel(const __grid_constant__ CUtensorMap tm_hs, const __grid_constant__ CUtensorMap tm_Ws,
                const __grid_constant__ CUtensorMap tm_ht, const __grid_constant__ CUtensorMap tm_Wt,
                const FusedParams p) {
  using C = FusedCfg<BN_>;
  constexpr int BN = C::BN;
  constexpr int HB = C::HB;
  constexpr int HALF = C::HALF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);  // used in the even CTA
  uint64_t* empty = full + C::STAGES;       // both CTAs: stage free (UMMAs done reading it)
  uint64_t* tfull = empty + C::STAGES;      // both CTAs: TMEM half h (0 teacher, 1 student) complete
  uint64_t* tempty = tfull + 2;             // even CTA: half h read by both CTAs' epilogues
  uint64_t* merge_full = tempty + 2;        // column half 1 -> half 0 statistics handoff
  uint64_t* merge_empty = merge_full + 1;
  uint64_t* drain = merge_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile unsigned long long* permit = reinterpret_cast<volatile unsigned long long*>(drain + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the UMMAs
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 2 * kEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(merge_full, kEpiWarps / 2);
    mbar_init(merge_empty, kEpiWarps / 2);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *permit = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tm_hs);
    prefetch_tmap(&tm_Ws);
    prefetch_tmap(&tm_ht);
    prefetch_tmap(&tm_Wt);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after();
  // Everything above touched only this CTA's own resources; from here on global memory (the
  // pacing counters, the statistics) may be shared with the previous kernel in the stream.
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem_base = *tmem_slot;
  const int kbt = p.kb_t, kbtot = p.kb_t + p.kb_s;
  const int my_rows = static_cast<int>(rank) * kBM;  // this CTA's token rows inside a pair tile

  if (warp < kEpiWarp0) setmaxnreg_dec<kRegsControl>();  // each warpgroup changes its registers at once
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has been armed at least once (even CTA)
      bool ok = true;
      bool pace = p.progress != nullptr && rank == 0;
      const unsigned long long ep = static_cast<unsigned long long>(p.epoch) << 48;
      for (int u = cid, kunit = 0; ok && u < p.units; u += ncl, ++kunit) {
        int row0, vt0, vt1, seg;
        unit_range(p, u, row0, vt0, vt1, seg);
        const int arow = row0 + my_rows;
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int brow = vt * BN + static_cast<int>(rank) * HB;
          if (pace) {
            const unsigned long long mine =
                (static_cast<unsigned long long>(kunit) << 24) | static_cast<unsigned long long>(vt - vt0);
            reinterpret_cast<volatile unsigned long long*>(p.progress)[cid] = ep | mine;
            if (*permit <= mine) {
              const uint64_t t0 = globaltimer_ns();
              while (*permit <= mine) {
                if (*abort_flag) break;
                if (globaltimer_ns() - t0 > kPaceWaitNs) {  // give up pacing for the whole launch
                  reinterpret_cast<volatile unsigned long long*>(p.progress)[kMaxClusters] = ep;
                  pace = false;
                  break;
                }
              }
            }
          }
          for (int kb = 0; kb < kbtot; ++kb) {
            if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 1)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * C::STAGE_BYTES;
            uint8_t* sb = sa + C::A_BYTES;
            const uint32_t fbar = mapa_shared(smem_u32(full + stage), 0);
            if (rank == 0) {
              mbar_arrive_expect_tx(full + stage, 2 * C::STAGE_BYTES);  // both CTAs' bytes
              armed |= 1u << stage;
            }
            if (kb < kbt) {
              tma_load_2d_pair(sa, &tm_ht, fbar, kb * kBK, arow);
              tma_load_2d_pair(sb, &tm_Wt, fbar, kb * kBK, brow);
            } else {
              const int k = kb - kbt;
              tma_load_2d_pair(sa, &tm_hs, fbar, k * kBK, arow);
              tma_load_2d_pair(sb, &tm_Ws, fbar, k * kBK, brow);
            }
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (p.progress != nullptr && rank == 0)  // no more units
        *reinterpret_cast<volatile unsigned long long*>(p.progress + cid) =
            (static_cast<unsigned long long>(p.epoch) << 48) | kPaceLow;
      if (!ok) {
        // Let every armed load land before the CTA can exit: the latest armed phase of stage s
        // has parity `phase` for stages below the current one and `phase ^ 1` otherwise.
        for (int s = 0; s < C::STAGES; ++s) {
          if (armed & (1u << s)) drain_wait(full + s, s < stage ? phase : (phase ^ 1u), 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ UMMA issuer (even CTA)
    // Teacher tile (K = d_t) into half 0, then student tile (K = d_s) into half 1 of both CTAs;
    // each half is awaited just before its own UMMAs and signalled as soon as they are done.
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true, issued = false;
      for (int u = cid; ok && u < p.units; u += ncl) {
        int row0, vt0, vt1, seg;
        unit_range(p, u, row0, vt0, vt1, seg);
        for (int vt = vt0; ok && vt < vt1; ++vt, ++lt) {
          const uint32_t tph = static_cast<uint32_t>(lt) & 1u;
          for (int kb = 0; kb < kbtot; ++kb) {
            if (kb == 0 || kb == kbt) {
              if (kb == kbt) umma_commit_pair(tfull + 0, 0x3);
              if (!wait_bounded(tempty + (kb == 0 ? 0 : 1), tph ^ 1u, abort_flag, p.ctl, 2)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
            const bool teacher = kb < kbt;
            const uint32_t d = tmem_base + (teacher ? 0u : static_cast<uint32_t>(BN));
            const int kk = teacher ? kb : kb - kbt;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              umma_bf16_pair(d, smem_desc_sw128(sa + k * 32, 0, 1024), smem_desc_sw128(sb + k * 32, 0, 1024), kIdesc,
                             (kk > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit_pair(empty + stage, 0x3);
            issued = true;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair(tfull + 1, 0x3);
        }
      }
      if (!ok && issued) {
        umma_commit_pair(drain, 0x1);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ pacing (even CTA)
    if (lane == 0 && rank == 0 && p.progress != nullptr) pace_peers(p, cid, ncl, permit, abort_flag);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    setmaxnreg_inc<kRegsEpilogue>();
    const int e = warp - kEpiWarp0;  // 0..7
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int h = e >> 2;           // column half of the tile: [h*HALF, h*HALF + HALF)
    const int row = q * 32 + lane;  // token row inside this CTA's 128 rows
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * HALF);
    int lt = 0, lu = 0;
    bool ok = true;
    for (int u = cid; ok && u < p.units; u += ncl, ++lu) {
      int row0, vt0, vt1, seg;
      unit_range(p, u, row0, vt0, vt1, seg);
      const int token = row0 + my_rows + row;
      RowStats rs{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
      for (int vt = vt0; vt < vt1; ++vt, ++lt) {
        const uint32_t tph = static_cast<uint32_t>(lt) & 1u;
        // the teacher tile: this row's 128 logits of the column half into registers, then half 0
        // goes back to the UMMAs
        bool w = wait_bounded(tfull + 0, tph, abort_flag, p.ctl, 4);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float zt[HALF];
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) tmem_ld32_at(lane_base + static_cast<uint32_t>(c * 32), zt + 32 * c);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(tempty + 0), 0));
        w = wait_bounded(tfull + 1, tph, abort_flag, p.ctl, 4);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int col_base = vt * BN + h * HALF;
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) {
          float zs[32];
          tmem_ld32(lane_base + static_cast<uint32_t>(BN + c * 32), zs);
          tmem_ld_wait();
          const int valid = min(32, p.V - (col_base + c * 32));
          if (valid >= 32) {
            fold_chunk<false>(rs, zt + 32 * c, zs, 0xffffffffu, p.c, p.inv_tau);
          } else if (valid > 0) {
            fold_chunk<true>(rs, zt + 32 * c, zs, (1u << valid) - 1u, p.c, p.inv_tau);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(tempty + 1), 0));
      }
      if (!ok) break;
      // Column half 1 hands its statistics to half 0, which merges them and writes the result.
      // The hand-off goes through the unit's own slot of the partial statistics (each unit, a
      // (pair tile, segment), owns its slots), read back by the same CTA: no shared memory, which
      // leaves room for a seventh operand stage.
      const uint32_t par = static_cast<uint32_t>(lu & 1);
      const size_t NS = static_cast<size_t>(p.N);
      const size_t fs = static_cast<size_t>(p.nseg) * NS;  // stride between fields
      float* base = p.part + static_cast<size_t>(seg) * NS + token;
      if (h == 1) {
        bool w = wait_bounded(merge_empty, par ^ 1u, abort_flag, p.ctl, 5);
        if (!__all_sync(0xffffffffu, w)) break;
        if (token < p.N) {
          base[0 * fs] = rs.mt;
          base[1 * fs] = rs.st;
          base[2 * fs] = rs.ms;
          base[3 * fs] = rs.ss;
          base[4 * fs] = rs.a;
          base[5 * fs] = rs.far ? -1.f : rs.cc;  // cc >= 0 otherwise, so -1 marks "far"
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_full);
      } else {
        bool w = wait_bounded(merge_full, par, abort_flag, p.ctl, 6);
        if (!__all_sync(0xffffffffu, w)) break;
        RowStats o{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, false};
        if (token < p.N) {
          const float occ = base[5 * fs];
          o = RowStats{base[0 * fs], base[1 * fs], base[2 * fs], base[3 * fs], base[4 * fs],
                       occ < 0.f ? 0.f : occ, occ < 0.f};
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_empty);
        if (token < p.N) {
          merge_stats(rs, o, p.c);
          base[0 * fs] = rs.mt;
          base[1 * fs] = rs.st;
          base[2 * fs] = rs.ms;
          base[3 * fs] = rs.ss;
          base[4 * fs] = rs.a;
          base[5 * fs] = rs.far ? -1.f : rs.cc;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no cross-CTA signal may target a CTA that has exited
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// Merges the per-segment statistics of each token (fp64) and writes kl, lse_s, lse_t and,
// when `gap` is not null, the precise lse_s - lse_t.
// KL = A/S_t - lse_t + lse_s in general; when C is valid (marked by C >= 0) and the two
// distributions are close, the algebraically equal form
// KL = C' + log1p(C' - mu) - (C' - mu), with mu = A/S_t = E_pt[d] and
// C' = C/S_t = E_pt[exp(-d) - 1 + d] >= 0, avoids the cancellation of two ~log V terms.
__global__ void kl_combine_kernel(const float* __restrict__ part, int N, int nseg, float inv_tau,
                                  float* __restrict__ kl, float* __restrict__ lse_s, float* __restrict__ lse_t,
                                  float* __restrict__ gap) {
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
  bool far = false;
  const double it = inv_tau;
  for (int s = 0; s < nseg; ++s) {
    const double mt = b[s * NS], ms = b[2 * fs + s * NS];
    const double wt = (mt == -INFINITY) ? 0.0 : exp((mt - Mt) * it);
    const double ws = (ms == -INFINITY) ? 0.0 : exp((ms - Ms) * it);
    const double cs = b[5 * fs + s * NS];
    St += wt * b[fs + s * NS];
    A += wt * b[4 * fs + s * NS];
    far = far || cs < 0.0;
    Cc += wt * cs;
    Ss += ws * b[3 * fs + s * NS];
  }
  double lt, ls, gp;
  const double k = kl_from_stats(Mt, St, Ms, Ss, A, Cc, far, it, lt, ls, gp);
  kl[n] = static_cast<float>(k);
  lse_s[n] = static_cast<float>(ls);
  lse_t[n] = static_cast<float>(lt);
  if (gap != nullptr) gap[n] = static_cast<float>(gp);
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

// attr must hold two entries: the cluster shape and programmatic stream serialization (the
// kernel may start while its predecessor finishes; see grid_dep_wait()).
template <int BN>
cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, int clusters, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = FusedCfg<BN>::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int BN>
cudaError_t prepare_one(int* max_clusters) {
  cudaError_t e =
      cudaFuncSetAttribute(fused_kl_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, FusedCfg<BN>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<BN>(attr, 1, nullptr);
  cfg.numAttrs = 1;  // occupancy: the cluster shape only
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, fused_kl_kernel<BN>, &cfg)) != cudaSuccess) return e;
  if (n < *max_clusters) *max_clusters = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t fused_prepare(int bn, int* max_clusters) {
  if (bn != kFusedBN) return cudaErrorInvalidValue;
  *max_clusters = 1 << 30;
  return prepare_one<kFusedBN>(max_clusters);
}

cudaError_t launch_fused(int bn, const CUtensorMap& hs, const CUtensorMap& Ws, const CUtensorMap& ht,
                         const CUtensorMap& Wt, const FusedParams& p, int clusters, cudaStream_t stream) {
  if (bn != kFusedBN) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<kFusedBN>(attr, clusters, stream);
  return cudaLaunchKernelEx(&cfg, fused_kl_kernel<kFusedBN>, hs, Ws, ht, Wt, p);
}

cudaError_t launch_combine(const float* part, int N, int nseg, float inv_tau, float* kl, float* lse_s,
                           float* lse_t, float* gap, cudaStream_t stream) {
  const int threads = 256;
  kl_combine_kernel<<<(N + threads - 1) / threads, threads, 0, stream>>>(part, N, nseg, inv_tau, kl, lse_s, lse_t,
                                                                         gap);
  return cudaGetLastError();
}

cudaError_t launch_mean(const float* kl, int N, float* loss, cudaStream_t stream) {
  kl_mean_kernel<<<1, 1024, 0, stream>>>(kl, N, loss);
  return cudaGetLastError();
}

}  // namespace hylo
