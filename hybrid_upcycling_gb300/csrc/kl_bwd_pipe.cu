// Backward of the fused hidden-state KL on sm_103a as ONE persistent launch.
//
// The loss is the Stage-II distillation loss of the HyLo pages: KL between the teacher's and
// the student's next-token distributions, kl_weight 1.0, no cross-entropy, computed from the
// final hidden states with the LM-head projections inside the loss (Long-Context Aware
// Upcycling digest, ftxj.github.io, section Method; HyLo-Llama-8MLA8GDN-8K-SFT reading notes,
// kwkr.cn, Stage II). The pages do not describe the backward; with z_s = h_s W_s^T and
// G = dL/dz_s = grad_scale (p_s - p_t) / (tau N), the student's gradients are the two
// contractions dh_s = G W_s and dW_s = G^T h_s.
//
// Work. The tokens are cut into blocks of R rows and the vocabulary into blocks of bw words
// (see BwdPipeParams). Per block b, "F" items each recompute one 256-token x 256-word pair tile
// of teacher and student logits (tcgen05 UMMA, TMEM accumulators), form G from the saved
// log-sum-exps and store it in bf16 into ring slot b % 3 of the workspace; "M" items each
// compute one 256 x 256 tile of the block's contribution to dW_s (K = the block's tokens) or
// dh_s (K = the block's words) from that slot and store or reduce-add it. G never needs more
// than three blocks of memory, and the gradient products of block b overlap the recompute of
// blocks b+1 and b+2 on other SMs, so one launch runs the whole backward without the tails
// of separate kernels.
//
// Order and dependencies. Items are taken from a global atomic counter in the order F(0),
// F(1), M(0), F(2), M(1), F(3), ..., M(B-1). Each CTA counts the items it completes (after its
// stores are complete) with a release-add on a counter in the workspace; an item that reads
// what others write first waits, with acquire loads, until the counters reach the totals that
// precede it in the order: M(b) needs F(b) (its G) and M(b-1) (the same dh_s / dW_s tiles,
// so the additions happen in a fixed order and results are deterministic); F(b) needs
// M(b-3) (the ring slot it overwrites). Every dependency points to an earlier item, taken by a
// running CTA, so the launch cannot deadlock whatever the residency; in this order the waits
// almost never block.
//
// Roles (384 threads per CTA of a cluster pair): warp 2 of the even CTA takes items from the
// queue, waits for their dependencies and publishes them to both CTAs through a shared-memory
// item ring, up to kItemDepth items ahead of the loads, so that the global-memory round trips of
// the queue and the counters stay off the path between two items' TMA loads; warp 0 of each CTA
// issues the TMA loads; warp 1 of the even CTA issues the UMMAs; warps 4..11 of both CTAs are
// the epilogue (lane quarter w & 3, column half
// (w - 4) >> 2 of each 256-column accumulator). Warpgroup 0 gives registers to the two epilogue
// warpgroups (setmaxnreg: 56 and 224 per thread).
//
// TMEM holds two 256-column halves. An M item takes one; an F item takes one for the teacher
// tile and the other for the student tile. The UMMA warp signals the teacher half as soon as its
// tiles are done, and the epilogue copies all 128 teacher logits of its row into registers and
// frees that half before the student tile is even complete; it frees the student half after
// forming G. Halves are handed out so that the next item's UMMAs always start in the half
// freed first (after an F item, its teacher half; after an M item, the other half), so the
// epilogue's work overlaps the UMMAs of the next item instead of stalling them.
#include <cmath>

#include "hylo_internal.h"
#include "kl_stats.cuh"

namespace hylo {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;                      // first epilogue warp (warpgroups 1 and 2)
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kRegsControl = 56;                  // per thread, warpgroup 0 (scheduler, TMA, UMMA)
constexpr int kRegsEpilogue = 224;                // per thread, warpgroups 1 and 2
static_assert(128 * kRegsControl + 256 * kRegsEpilogue <= kThreads * 168, "register split");
constexpr int BN = 256;                           // columns of every pair tile
constexpr int HB = BN / 2;                        // B rows staged per CTA
constexpr int A_BYTES = kBM * kBK * 2;            // 16 KB: this CTA's 128 rows of A
constexpr int B_BYTES = HB * kBK * 2;             // 16 KB: this CTA's 128 rows of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 6;
// per epilogue warp: 32 rows x 128 B (M items: 32 fp32 columns, 128-byte swizzle; F items: two
// tiles of 32 rows x 32 bf16 columns, 64-byte swizzle)
constexpr int STAGING_BYTES = kEpiWarps * 4096;
constexpr int kItemDepth = 3;
constexpr int ITEM_OFF = STAGES * STAGE_BYTES + STAGING_BYTES;
constexpr int BAR_OFF = ITEM_OFF + kItemDepth * 32;
// full[S], empty[S], tfull[2], tempty[2], ifull[D], iempty[D], drain
constexpr int NBARS = 2 * STAGES + 4 + 2 * kItemDepth + 1;
// after the barriers: TMEM address, abort flag, items completed per epilogue warp
constexpr int SMEM = 1024 + BAR_OFF + NBARS * 8 + 8 + 4 * kEpiWarps;
static_assert(SMEM <= 232448, "shared memory budget");

// Threads that release an item-ring slot: in each CTA the producer and the epilogue warps, and
// the even CTA's UMMA thread.
constexpr int kItemConsumers = 2 * (1 + kEpiWarps) + 1;

enum : int { kItemF = 0, kItemDW = 1, kItemDH = 2, kItemEnd = 3 };
// kMapG: G tile stores, box 32 x 32 words with 64-byte swizzle
enum : int { kMapHs = 0, kMapHt, kMapWs, kMapWt, kMapWsB, kMapHsB, kMapDh, kMapDW, kMapG, kMapGA, kMapGT };

struct PipeMaps {
  CUtensorMap m[kPipeMaps];
};

// A work item as published to both CTAs. Before loading, wait until ctrl[ctr0] >= tgt0 and
// ctrl[ctr1] >= tgt1 (a target of 0 needs no wait).
struct Item {
  int kind, b, idx, pad;
  unsigned ctr0, tgt0, ctr1, tgt1;
};
static_assert(sizeof(Item) == 32, "item size");

struct Geo {
  int tb, vb;   // token block, vocabulary block
  int r0, v0;   // first token, first word
  int R, Vb;    // tokens, words in the block
  int tt, vt;   // 256-token tiles, 256-word tiles
  int slot;     // G ring slot
};

__device__ __forceinline__ Geo geo(const BwdPipeParams& p, int b) {
  Geo g;
  g.tb = b / p.VB;
  g.vb = b - g.tb * p.VB;
  g.r0 = g.tb * p.R;
  g.v0 = g.vb * p.bw;
  g.R = min(p.R, p.N - g.r0);
  g.Vb = min(p.bw, p.V - g.v0);
  g.tt = (g.R + BN - 1) / BN;
  g.vt = (g.Vb + BN - 1) / BN;
  g.slot = b % kGRing;
  return g;
}

__device__ __forceinline__ int items_f(const BwdPipeParams& p, int b) {
  const Geo g = geo(p, b);
  return g.tt * g.vt;
}

__device__ __forceinline__ int items_m(const BwdPipeParams& p, int b) {
  const Geo g = geo(p, b);
  return (g.vt + g.tt) * p.ntd;
}

// Walks the queue order part by part: segment j holds M(j-2) (part 0) if 0 <= j-2 < B and F(j)
// (part 1) if j < B. It keeps, per counter, the completion total of the parts already passed
// (each CTA of a pair adds 1 per item, so totals count 2 per item).
struct Cursor {
  int j, part, base, size;
  unsigned cum_m;          // M items of the parts passed
  unsigned cum_f[kGRing];  // F items of the parts passed, per ring slot
  bool end;
};

__device__ __forceinline__ void cursor_init(Cursor& c, const BwdPipeParams& p) {
  c.j = 0;
  c.part = 1;
  c.base = 0;
  c.size = items_f(p, 0);
  c.cum_m = 0;
  for (int s = 0; s < kGRing; ++s) c.cum_f[s] = 0;
  c.end = false;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const BwdPipeParams& p) {
  const int b = c.part == 0 ? c.j - 2 : c.j;
  if (c.part == 0)
    c.cum_m += 2u * static_cast<unsigned>(c.size);
  else
    c.cum_f[b % kGRing] += 2u * static_cast<unsigned>(c.size);
  c.base += c.size;
  if (c.part == 0 && c.j < p.B) {
    c.part = 1;
  } else {
    while (true) {
      ++c.j;
      if (c.j - 2 >= p.B) {
        c.end = true;
        c.size = 0;
        return;
      }
      if (c.j >= 2) {
        c.part = 0;
        break;
      }
      if (c.j < p.B) {
        c.part = 1;
        break;
      }
    }
  }
  const int nb = c.part == 0 ? c.j - 2 : c.j;
  c.size = c.part == 0 ? items_m(p, nb) : items_f(p, nb);
}

// The item with queue index i (the cursor only moves forward; i never decreases per caller).
__device__ __forceinline__ Item cursor_item(Cursor& c, const BwdPipeParams& p, int i) {
  while (!c.end && i >= c.base + c.size) cursor_next(c, p);
  Item it{};
  if (c.end) {
    it.kind = kItemEnd;
    return it;
  }
  const int b = c.part == 0 ? c.j - 2 : c.j;
  const int local = i - c.base;
  it.b = b;
  if (c.part == 1) {
    it.kind = kItemF;
    it.idx = local;
    if (b >= kGRing) {  // every M item of blocks <= b - 3 (the parts passed, minus M(b-2))
      it.ctr0 = 1;
      it.tgt0 = c.cum_m - 2u * static_cast<unsigned>(items_m(p, b - 2));
    }
  } else {
    const Geo g = geo(p, b);
    const int ndw = g.vt * p.ntd;
    it.kind = local < ndw ? kItemDW : kItemDH;
    it.idx = local < ndw ? local : local - ndw;
    it.ctr0 = 2 + g.slot;  // every F item of block b
    it.tgt0 = c.cum_f[g.slot];
    it.ctr1 = 1;           // every M item of blocks < b
    it.tgt1 = c.cum_m;
  }
  return it;
}

// Waits for ctrl[ctr] >= target (acquire); false on abort or time-out (then it raises the
// CTA's abort flag and records the site).
__device__ __forceinline__ bool wait_count(const unsigned* ctrl, unsigned ctr, unsigned target, volatile int* abort_flag,
                                           const WaitCtl& ctl, int site) {
  if (target == 0u) return true;
  const unsigned* a = ctrl + ctr;
  if (ld_acquire_gpu(a) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(128);
    if (ld_acquire_gpu(a) >= target) return true;
    if ((it & 7u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > ctl.limit_ns) {
        *abort_flag = 1;
        atomicCAS(ctl.status, 0, kDevTimeoutBase + site);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Descriptor of the k-th 16-deep slice of a staged 128-row tile (128-byte swizzle).
//   K-major: advance 32 B inside the swizzle row; groups of 8 rows 1024 B apart.
//   MN-major: advance 16 k-rows = 2048 B; the two 64-element M/N blocks are 8192 B apart (LBO),
//   groups of 8 k-rows 1024 B apart (SBO).
__device__ __forceinline__ uint64_t slice_desc(bool mn, uint32_t base, int k) {
  return mn ? smem_desc_sw128(base + k * 2048, 8192, 1024) : smem_desc_sw128(base + k * 32, 0, 1024);
}

// 64-deep k-blocks of an M item (both passes when split).
template <bool SPLIT>
__device__ __forceinline__ int m_kblocks(const Geo& g, int kind) {
  const int k = kind == kItemDW ? (g.R + kBK - 1) / kBK : (g.Vb + kBK - 1) / kBK;
  return SPLIT ? 2 * k : k;
}

template <bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_pipe_kernel(const __grid_constant__ PipeMaps maps, const BwdPipeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* staging_all = smem + STAGES * STAGE_BYTES;
  Item* items = reinterpret_cast<Item*>(smem + ITEM_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // used in the even CTA
  uint64_t* empty = full + STAGES;                                // both CTAs
  uint64_t* tfull = empty + STAGES;                               // both CTAs: TMEM half h written
  uint64_t* tempty = tfull + 2;                                   // even CTA: half h drained (both CTAs)
  uint64_t* ifull = tempty + 2;                                   // both CTAs: item slot published
  uint64_t* iempty = ifull + kItemDepth;                          // even CTA: item slot released
  uint64_t* drain = iempty + kItemDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* epi_done = tmem_slot + 2;  // [kEpiWarps]: items whose stores each epilogue warp has completed

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: schedules and issues the UMMAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(tfull + h, 1);
      mbar_init(tempty + h, 2 * kEpiWarps);
    }
    for (int k = 0; k < kItemDepth; ++k) {
      mbar_init(ifull + k, 1);
      mbar_init(iempty + k, kItemConsumers);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    for (int w = 0; w < kEpiWarps; ++w) epi_done[w] = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    for (int m = 0; m < kPipeMaps; ++m) prefetch_tmap(&maps.m[m]);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after();
  grid_dep_wait();  // the workspace and outputs may be shared with the previous kernel in the stream
  grid_dep_launch();
  const uint32_t tmem_base = *tmem_slot;
  const int kbt = p.kb_t, kbf = p.kb_t + p.kb_s;

  if (warp < kEpiWarp0) setmaxnreg_dec<kRegsControl>();  // each warpgroup changes its registers at once
  if (warp == 2) {
    // ------------------------------------------------------------------ scheduler (even CTA)
    if (lane == 0 && rank == 0) {
      Cursor cur;
      cursor_init(cur, p);
      const uint32_t peer_items = mapa_shared(smem_u32(items), 1);
      const uint32_t peer_ifull = mapa_shared(smem_u32(ifull), 1);
      int next_i = static_cast<int>(atomicAdd(p.ctrl, 1u));
      for (int k = 0;; ++k) {
        const int slot = k % kItemDepth;
        const uint32_t par = static_cast<uint32_t>(k / kItemDepth) & 1u;
        if (!wait_bounded<true>(iempty + slot, par ^ 1u, abort_flag, p.ctl, 21)) break;
        const Item it = cursor_item(cur, p, next_i);
        if (it.kind != kItemEnd) {
          next_i = static_cast<int>(atomicAdd(p.ctrl, 1u));  // the next item, fetched ahead
          // the item is published only once what it reads is complete
          if (!wait_count(p.ctrl, it.ctr0, it.tgt0, abort_flag, p.ctl, 23) ||
              !wait_count(p.ctrl, it.ctr1, it.tgt1, abort_flag, p.ctl, 24))
            break;
        }
        items[slot] = it;
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&it);
        for (int q = 0; q < 8; ++q) st_cluster_u32(peer_items + slot * 32 + q * 4, w[q]);
        mbar_arrive(ifull + slot);
        mbar_arrive_remote(peer_ifull + slot * 8);
        if (it.kind == kItemEnd) break;
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0;
      bool ok = true;
      const uint32_t lead_iempty = mapa_shared(smem_u32(iempty), 0);
      const uint32_t full_lead = mapa_shared(smem_u32(full), 0);  // full[0] of the even CTA
      for (int k = 0; ok; ++k) {
        const int slot = k % kItemDepth;
        const uint32_t par = static_cast<uint32_t>(k / kItemDepth) & 1u;
        if (!wait_bounded<true>(ifull + slot, par, abort_flag, p.ctl, 22)) break;
        const Item it = items[slot];
        if (rank == 0)
          mbar_arrive(iempty + slot);
        else
          mbar_arrive_remote(lead_iempty + slot * 8);
        if (it.kind == kItemEnd) break;
        // the G tiles this item reads were stored by TMA in other CTAs, whose completion the
        // scheduler observed (acquire) before publishing the item
        fence_proxy_async_global();
        // Every coordinate is set up once per item: a stage then costs only its wait, its arming
        // and its TMA instructions (the producer, not the tensor cores, limited the M items while
        // it also did this arithmetic per stage).
        const Geo g = geo(p, it.b);
        const int r_a = static_cast<int>(rank) * kBM;  // this CTA's rows of the A tile
        const int r_b = static_cast<int>(rank) * HB;   // this CTA's rows of the B tile
        bool fine = true;
        auto next = [&](uint8_t*& sa, uint32_t& fb) -> bool {  // wait for a free stage and arm it
          if (!wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.ctl, 25)) return false;
          sa = smem + stage * STAGE_BYTES;
          fb = full_lead + static_cast<uint32_t>(stage) * 8u;
          if (rank == 0) {
            mbar_arrive_expect_tx(full + stage, 2 * STAGE_BYTES);  // both CTAs' bytes
            armed |= 1u << stage;
          }
          return true;
        };
        auto advance = [&]() {
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        };
        if (it.kind == kItemF) {  // teacher tile over d_t, then student tile over d_s
          const int ti = it.idx % g.tt, vi = it.idx / g.tt;
          const int arow = g.r0 + ti * BN + r_a, brow = g.v0 + vi * BN + r_b;
          for (int kb = 0; fine && kb < kbt; ++kb) {
            uint8_t* sa;
            uint32_t fb;
            if (!(fine = next(sa, fb))) break;
            tma_load_2d_pair(sa, &maps.m[kMapHt], fb, kb * kBK, arow);
            tma_load_2d_pair(sa + A_BYTES, &maps.m[kMapWt], fb, kb * kBK, brow);
            advance();
          }
          for (int kb = 0; fine && kb < p.kb_s; ++kb) {
            uint8_t* sa;
            uint32_t fb;
            if (!(fine = next(sa, fb))) break;
            tma_load_2d_pair(sa, &maps.m[kMapHs], fb, kb * kBK, arow);
            tma_load_2d_pair(sa + A_BYTES, &maps.m[kMapWs], fb, kb * kBK, brow);
            advance();
          }
        } else {
          const int mi = it.idx / p.ntd, nj = it.idx - mi * p.ntd;
          const int mrow = mi * BN + r_a;   // A rows: words (dW_s) or tokens (dh_s) of the block
          const int ncol = nj * BN + r_b;   // B rows: this CTA's d_s columns
          if (it.kind == kItemDW) {  // A = G^T (word-major), B = h_s of the block's tokens; K = tokens
            const int nk = (g.R + kBK - 1) / kBK;
            for (int term = 0; fine && term < (SPLIT ? 2 : 1); ++term) {
              const int z = g.slot + term * kGRing;
              for (int kk = 0; kk < nk; ++kk) {
                uint8_t* sa;
                uint32_t fb;
                if (!(fine = next(sa, fb))) break;
                const int k0 = kk * kBK;
                tma_load_3d_pair(sa, &maps.m[kMapGT], fb, mrow, k0, z);
                tma_load_3d_pair(sa + 8192, &maps.m[kMapGT], fb, mrow + 64, k0, z);
                tma_load_2d_pair(sa + A_BYTES, &maps.m[kMapHsB], fb, ncol, g.r0 + k0);
                tma_load_2d_pair(sa + A_BYTES + 8192, &maps.m[kMapHsB], fb, ncol + 64, g.r0 + k0);
                advance();
              }
            }
          } else {  // A = G (token rows, K-major), B = W_s of the block's words; K = words
            const int nk = (g.Vb + kBK - 1) / kBK;
            for (int term = 0; fine && term < (SPLIT ? 2 : 1); ++term) {
              const int z = g.slot + term * kGRing;
              for (int kk = 0; kk < nk; ++kk) {
                uint8_t* sa;
                uint32_t fb;
                if (!(fine = next(sa, fb))) break;
                const int k0 = kk * kBK;
                tma_load_3d_pair(sa, &maps.m[kMapGA], fb, k0, mrow, z);
                tma_load_2d_pair(sa + A_BYTES, &maps.m[kMapWsB], fb, ncol, g.v0 + k0);
                tma_load_2d_pair(sa + A_BYTES + 8192, &maps.m[kMapWsB], fb, ncol + 64, g.v0 + k0);
                advance();
              }
            }
          }
        }
        if (!fine) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        // Let every armed load land before the CTA can exit: the latest armed phase of stage s
        // has parity `phase` for stages below the current one and `phase ^ 1` otherwise.
        for (int s = 0; s < STAGES; ++s) {
          if (armed & (1u << s)) drain_wait(full + s, s < stage ? phase : (phase ^ 1u), 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ UMMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdescF = idesc_bf16_f32(2 * kBM, BN, false, false);
      constexpr uint32_t kIdescDH = idesc_bf16_f32(2 * kBM, BN, false, true);
      constexpr uint32_t kIdescDW = idesc_bf16_f32(2 * kBM, BN, true, true);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses[2] = {0u, 0u};
      int hp = 0;
      bool ok = true, issued = false;
      for (int k = 0; ok; ++k) {
        const int slot = k % kItemDepth;
        const uint32_t par = static_cast<uint32_t>(k / kItemDepth) & 1u;
        if (!wait_bounded(ifull + slot, par, abort_flag, p.ctl, 26)) {
          ok = false;
          break;
        }
        const Item it = items[slot];
        mbar_arrive(iempty + slot);
        if (it.kind == kItemEnd) break;
        const Geo g = geo(p, it.b);
        if (it.kind == kItemF) {
          // teacher tile (K = d_t) into half t = hp, student tile (K = d_s) into the other; each
          // half is awaited just before its own UMMAs, and the teacher half is signalled as soon
          // as its UMMAs are done
          const int t = hp, sh = hp ^ 1;
          for (int kb = 0; kb < kbf; ++kb) {
            if (kb == 0 || kb == kbt) {
              const int h = kb == 0 ? t : sh;
              if (kb == kbt) umma_commit_pair(tfull + t, 0x3);
              if (!wait_bounded(tempty + h, (uses[h] & 1u) ^ 1u, abort_flag, p.ctl, 27)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 28)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t sb = sa + A_BYTES;
            const bool teacher = kb < kbt;
            const uint32_t d = tmem_base + static_cast<uint32_t>((teacher ? t : sh) * BN);
            const int kk = teacher ? kb : kb - kbt;
#pragma unroll
            for (int q = 0; q < kBK / 16; ++q) {
              umma_bf16_pair(d, smem_desc_sw128(sa + q * 32, 0, 1024), smem_desc_sw128(sb + q * 32, 0, 1024), kIdescF,
                             (kk > 0 || q > 0) ? 1u : 0u);
            }
            umma_commit_pair(empty + stage, 0x3);
            issued = true;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair(tfull + sh, 0x3);
          ++uses[0];
          ++uses[1];
        } else {
          const int h = hp;
          hp ^= 1;
          if (!wait_bounded(tempty + h, (uses[h] & 1u) ^ 1u, abort_flag, p.ctl, 29)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool amn = it.kind == kItemDW;
          const uint32_t idesc = amn ? kIdescDW : kIdescDH;
          const uint32_t d = tmem_base + static_cast<uint32_t>(h * BN);
          const int nkb = m_kblocks<SPLIT>(g, it.kind);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(full + stage, phase, abort_flag, p.ctl, 30)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t sb = sa + A_BYTES;
#pragma unroll
            for (int q = 0; q < kBK / 16; ++q) {
              umma_bf16_pair(d, slice_desc(amn, sa, q), slice_desc(true, sb, q), idesc, (kb > 0 || q > 0) ? 1u : 0u);
            }
            umma_commit_pair(empty + stage, 0x3);
            issued = true;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair(tfull + h, 0x3);
          ++uses[h];
        }
      }
      if (!ok && issued) {
        umma_commit_pair(drain, 0x1);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    setmaxnreg_inc<kRegsEpilogue>();
    const int e = warp - kEpiWarp0;  // 0..7
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int hc = e >> 2;           // column half of a 256-column accumulator
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(hc * HB);
    uint8_t* staging = staging_all + e * 4096;
    const uint32_t rowaddr = smem_u32(staging) + lane * 128;  // M items: this lane's 128-byte row
    const uint32_t row64 = smem_u32(staging) + lane * 64;     // F items: this lane's 64-byte row
    const uint32_t swz64 = static_cast<uint32_t>((lane >> 1) & 3);
    const uint32_t lead_iempty = mapa_shared(smem_u32(iempty), 0);
    const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);
    uint32_t uses[2] = {0u, 0u};
    int hp = 0;
    for (int k = 0;; ++k) {
      const int slot = k % kItemDepth;
      const uint32_t par = static_cast<uint32_t>(k / kItemDepth) & 1u;
      const bool got = rank == 0 ? wait_bounded(ifull + slot, par, abort_flag, p.ctl, 31)
                                 : wait_bounded<true>(ifull + slot, par, abort_flag, p.ctl, 31);
      if (!__all_sync(0xffffffffu, got)) break;
      const Item it = items[slot];
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(iempty + slot);
        else
          mbar_arrive_remote(lead_iempty + slot * 8);
      }
      if (it.kind == kItemEnd) break;
      const Geo g = geo(p, it.b);
      unsigned ctr;
      if (it.kind == kItemF) {
        ctr = 2u + static_cast<unsigned>(g.slot);
        const int ti = it.idx % g.tt, vi = it.idx / g.tt;
        const int row_local = ti * BN + static_cast<int>(rank) * kBM + q * 32;  // first slot row of this warp
        const int token = g.r0 + row_local + lane;
        float bt = 0.f, bs = 0.f, ngl = 0.f;
        if (token < p.N) {
          const float lt_ = p.lse_t[token], ls_ = p.lse_s[token];
          bt = lt_ * kLog2e;
          bs = ls_ * kLog2e;
          ngl = -(p.lse_gap != nullptr ? p.lse_gap[token] : ls_ - lt_) * kLog2e;
        }
        const int t = hp, sh = hp ^ 1;
        // the teacher tile: all 128 logits of this row and column half into registers, then the
        // half goes back to the UMMAs
        const bool wt = wait_bounded(tfull + t, uses[t] & 1u, abort_flag, p.ctl, 32);
        if (!__all_sync(0xffffffffu, wt)) break;
        tc_fence_after();
        float zt[HB];
#pragma unroll
        for (int c = 0; c < HB / 32; ++c) tmem_ld32_at(lane_base + static_cast<uint32_t>(t * BN + c * 32), zt + 32 * c);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(lead_tempty + t * 8);
        const bool ws = wait_bounded(tfull + sh, uses[sh] & 1u, abort_flag, p.ctl, 32);
        if (!__all_sync(0xffffffffu, ws)) break;
        tc_fence_after();
        ++uses[0];
        ++uses[1];
        const int col_local = vi * BN + hc * HB;  // first block column of this warp
        const float2 c2v = make_float2(p.c, p.c), gs2 = make_float2(p.gscale, p.gscale);
        const float2 nbt = make_float2(-bt, -bt), nbs = make_float2(-bs, -bs), ngl2 = make_float2(ngl, ngl);
#pragma unroll
        for (int c = 0; c < HB / 32; ++c) {
          float zs[32];
          tmem_ld32(lane_base + static_cast<uint32_t>(sh * BN + c * 32), zs);
          tmem_ld_wait();
          const int vcols = g.Vb - (col_local + c * 32);  // columns of this chunk inside the vocabulary
          uint32_t pk[16], pl[16];  // G in bf16 and (split) its bf16 rounding remainder
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float2 gv = __fmul2_rn(prob_diff2(make_float2(zt[32 * c + 2 * j], zt[32 * c + 2 * j + 1]),
                                              make_float2(zs[2 * j], zs[2 * j + 1]), c2v, nbt, nbs, ngl2),
                                   gs2);
            if (vcols < 32) {  // the vocabulary ends inside this chunk: G = 0 past it
              if (2 * j >= vcols) gv.x = 0.f;
              if (2 * j + 1 >= vcols) gv.y = 0.f;
            }
            const uint32_t hi = pack_bf16x2(gv.x, gv.y);
            pk[j] = hi;
            if (SPLIT)
              pl[j] = pack_bf16x2(gv.x - __uint_as_float(hi << 16), gv.y - __uint_as_float(hi & 0xffff0000u));
          }
          // 32 x 32 tiles of 64-byte rows, 64-byte swizzle (16-byte chunk i of row r at i ^ ((r >> 1) & 3));
          // plain G alternates the two 2 KB tiles, split G puts bf16(G) in the first, the remainder in the second
          const uint32_t buf = SPLIT ? 0u : static_cast<uint32_t>((c & 1) * 2048);
          if (lane == 0) {
            if (SPLIT)
              bulk_wait_group_read<0>();
            else
              bulk_wait_group_read<1>();
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t a = row64 + buf + ((static_cast<uint32_t>(i) ^ swz64) << 4);
            st_shared_v4(a, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            if (SPLIT) st_shared_v4(a + 2048, pl[4 * i], pl[4 * i + 1], pl[4 * i + 2], pl[4 * i + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row_local < p.R) {
            tma_store_3d(&maps.m[kMapG], staging + buf, col_local + c * 32, row_local, g.slot);
            if (SPLIT) tma_store_3d(&maps.m[kMapG], staging + 2048, col_local + c * 32, row_local, g.slot + kGRing);
            bulk_commit_group();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(lead_tempty + sh * 8);
      } else {
        ctr = 1u;
        const int h = hp;
        hp ^= 1;
        const bool w = wait_bounded(tfull + h, uses[h] & 1u, abort_flag, p.ctl, 33);
        if (!__all_sync(0xffffffffu, w)) break;
        tc_fence_after();
        const int mi = it.idx / p.ntd, nj = it.idx - (it.idx / p.ntd) * p.ntd;
        const bool dw = it.kind == kItemDW;
        const CUtensorMap* mc = dw ? &maps.m[kMapDW] : &maps.m[kMapDh];
        const int row = (dw ? g.v0 : g.r0) + mi * BN + static_cast<int>(rank) * kBM + q * 32;
        const int rows_total = dw ? p.V : p.N;
        const bool accumulate = dw ? g.tb > 0 : g.vb > 0;
        const int col0 = nj * BN + hc * HB;
        const int n_valid = p.d_s - col0;
        const uint32_t acc = lane_base + static_cast<uint32_t>(h * BN);
#pragma unroll 1
        for (int ch = 0; ch < HB / 32; ++ch) {
          if (ch * 32 >= n_valid) break;  // warp-uniform: nothing of this chunk lies inside the output
          float v[32];
          tmem_ld32(acc + ch * 32, v);
          tmem_ld_wait();
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const uint32_t chunk = static_cast<uint32_t>(c4 ^ (lane & 7));
            st_shared_v4(rowaddr + chunk * 16, __float_as_uint(v[4 * c4]), __float_as_uint(v[4 * c4 + 1]),
                         __float_as_uint(v[4 * c4 + 2]), __float_as_uint(v[4 * c4 + 3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row < rows_total) {
            if (accumulate)
              tma_reduce_add_2d(mc, staging, col0 + ch * 32, row);
            else
              tma_store_2d(mc, staging, col0 + ch * 32, row);
            bulk_commit_group();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(lead_tempty + h * 8);
        ++uses[h];
      }
      // The item is complete in this CTA once every epilogue warp's stores have landed: each
      // warp publishes its count of completed items, and warp 0 counts the item in the
      // workspace for the items that wait on it once all eight have reached it.
      const uint32_t ndone = static_cast<uint32_t>(k) + 1u;
      if (lane == 0) {
        bulk_wait_group<0>();
        fence_proxy_async_global();
        st_release_cta_shared(epi_done + e, ndone);
      }
      bool counted = true;
      if (e == 0 && lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        for (int w = 1; counted && w < kEpiWarps; ++w) {
          while (ld_acquire_cta_shared(epi_done + w) < ndone) {
            if (*abort_flag) {
              counted = false;
              break;
            }
            if (globaltimer_ns() - t0 > p.ctl.limit_ns) {
              *abort_flag = 1;
              atomicCAS(p.ctl.status, 0, kDevTimeoutBase + 34);
              counted = false;
              break;
            }
          }
        }
        if (counted) red_release_gpu_add(p.ctrl + ctr, 1u);
      }
      if (!__shfl_sync(0xffffffffu, counted ? 1 : 0, 0)) break;
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

cudaLaunchConfig_t pipe_config(cudaLaunchAttribute* attr, int clusters, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

}  // namespace

cudaError_t bwd_pipe_prepare(int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(bwd_pipe_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_pipe_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pipe_config(attr, 1, nullptr);
  cfg.numAttrs = 1;  // occupancy: the cluster shape only
  return cudaOccupancyMaxActiveClusters(max_clusters, bwd_pipe_kernel<false>, &cfg);
}

cudaError_t launch_bwd_pipe(const CUtensorMap* maps, const BwdPipeParams& p, int clusters, cudaStream_t stream) {
  PipeMaps pm;
  for (int m = 0; m < kPipeMaps; ++m) pm.m[m] = maps[m];
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pipe_config(attr, clusters, stream);
  return p.split ? cudaLaunchKernelEx(&cfg, bwd_pipe_kernel<true>, pm, p)
                 : cudaLaunchKernelEx(&cfg, bwd_pipe_kernel<false>, pm, p);
}

}  // namespace hylo
