// Per-row softmax/KL statistics shared by the fused hidden-state kernel and the
// logits-input kernel: an online (running-max, rescaled-sum) fold of teacher and student
// logits, the merge of two partial sets, and the final KL.
//
// The loss is KL(p_t || p_s) between the teacher's and the student's next-token distributions
// (HyLo-Llama-8MLA8GDN-8K-SFT reading notes, section "two-stage training recipe", Stage II;
// the softmax+KL fusion of the Long-Context Aware Upcycling digest, section Method).
#pragma once

#include <cmath>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace hylo {

constexpr float kLog2e = 1.4426950408889634f;

// Running statistics of one token row over the vocabulary columns seen so far. Maxima are in
// raw logit units; sums are relative to exp(max / tau).
struct RowStats {
  float mt, st;  // teacher running max, sum_v exp((z_t - mt)/tau)
  float ms, ss;  // student running max, sum_v exp((z_s - ms)/tau)
  float a;       // sum_v exp((z_t - mt)/tau) * d_v, with d_v = (z_t - z_s)/tau
  float cc;      // sum_v exp((z_t - mt)/tau) * (exp(-d_v) - 1 + d_v)   (each term >= 0)
  bool far;      // exp((m_s - m_t)/tau) overflowed: cc is not valid, the direct KL form is used
};

// g(d) = exp(-d) - 1 + d by its Taylor series through d^7, for |d| < 1/4 (truncation < 2e-8
// relative there); used so that near-identical distributions lose no digits to cancellation.
__device__ __forceinline__ float2 g_series2(float2 d) {
  float2 t = __ffma2_rn(d, make_float2(-1.0f / 5040.0f, -1.0f / 5040.0f), make_float2(1.0f / 720.0f, 1.0f / 720.0f));
  t = __ffma2_rn(d, t, make_float2(-1.0f / 120.0f, -1.0f / 120.0f));
  t = __ffma2_rn(d, t, make_float2(1.0f / 24.0f, 1.0f / 24.0f));
  t = __ffma2_rn(d, t, make_float2(-1.0f / 6.0f, -1.0f / 6.0f));
  t = __ffma2_rn(d, t, make_float2(0.5f, 0.5f));
  return __fmul2_rn(__fmul2_rn(d, d), t);
}

__device__ __forceinline__ float2 ex2_approx2(float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); }

// Folds 32 columns of one row into the running statistics (column pairs in packed fp32x2
// arithmetic). Column j takes part iff bit j of `valid` is set (all bits except at the end of
// the vocabulary; MASKED only there: masked columns enter as z_t = z_s = max - 2^10 tau, whose
// exponentials flush to zero and whose d is 0). At least one column must be valid.
// Each column adds e_t g(d) to C: the Taylor series for |d| < 1/4, otherwise
// e_t (exp(-d) - 1 + d) = e_s K - e_t + e_t d with K = exp((m_s - m_t)/tau), which uses no
// extra exponential. K is clamped to stay finite; if the clamp engages the row is marked far.
// zt_in, zs_in: 32 consecutive values each (register arrays indexed with compile-time offsets).
template <bool MASKED, int W = 32>
__device__ __forceinline__ void fold_chunk(RowStats& r, const float* zt_in, const float* zs_in, uint32_t valid,
                                           float c, float inv_tau) {
  float cmt = -INFINITY, cms = -INFINITY;
#pragma unroll
  for (int j = 0; j < W; ++j) {
    if (!MASKED || ((valid >> j) & 1u)) {
      cmt = fmaxf(cmt, zt_in[j]);
      cms = fmaxf(cms, zs_in[j]);
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
  const float kexp = (nms - nmt) * c;
  r.far = r.far || !(kexp < 126.f);
  const float K = ex2_approx(fminf(kexp, 126.f));
  const float2 c2 = make_float2(c, c), it2 = make_float2(inv_tau, inv_tau), m1 = make_float2(-1.f, -1.f);
  const float2 K2 = make_float2(K, K);
  const float2 nmtc = make_float2(-nmt * c, -nmt * c), nmsc = make_float2(-nms * c, -nms * c);
  const float fill = fminf(nmt, nms) - 1024.f / c;  // value of a masked column
  float2 st = make_float2(0.f, 0.f), ss = st, a = st, cc = st;
#pragma unroll
  for (int j = 0; j < W / 2; ++j) {
    float2 zt = make_float2(zt_in[2 * j], zt_in[2 * j + 1]);
    float2 zs = make_float2(zs_in[2 * j], zs_in[2 * j + 1]);
    if (MASKED) {
      if (!((valid >> (2 * j)) & 1u)) zt.x = zs.x = fill;
      if (!((valid >> (2 * j + 1)) & 1u)) zt.y = zs.y = fill;
    }
    const float2 et = ex2_approx2(__ffma2_rn(zt, c2, nmtc));
    const float2 es = ex2_approx2(__ffma2_rn(zs, c2, nmsc));
    const float2 d = __fmul2_rn(__ffma2_rn(zs, m1, zt), it2);  // (z_t - z_s) / tau
    st = __fadd2_rn(st, et);
    ss = __fadd2_rn(ss, es);
    const float2 etd = __fmul2_rn(et, d);
    a = __fadd2_rn(a, etd);
    const float2 small = __fmul2_rn(et, g_series2(d));
    const float2 big = __ffma2_rn(es, K2, __ffma2_rn(et, m1, etd));
    cc = __fadd2_rn(cc, make_float2(fabsf(d.x) < 0.25f ? small.x : big.x, fabsf(d.y) < 0.25f ? small.y : big.y));
  }
  r.st += st.x + st.y;
  r.ss += ss.x + ss.y;
  r.a += a.x + a.y;
  r.cc += cc.x + cc.y;
}

// Merges the statistics of another set of columns of the same row into `r`. `r` must have
// seen at least one column; `o` may be empty (maxima -inf, sums 0).
__device__ __forceinline__ void merge_stats(RowStats& r, const RowStats& o, float c) {
  const float mt = fmaxf(r.mt, o.mt), ms = fmaxf(r.ms, o.ms);
  const float wr = ex2_approx((r.mt - mt) * c), wo = ex2_approx((o.mt - mt) * c);
  const float vr = ex2_approx((r.ms - ms) * c), vo = ex2_approx((o.ms - ms) * c);
  r.st = r.st * wr + o.st * wo;
  r.a = r.a * wr + o.a * wo;
  r.cc = r.cc * wr + o.cc * wo;
  r.ss = r.ss * vr + o.ss * vo;
  r.mt = mt;
  r.ms = ms;
  r.far = r.far || o.far;
}

// Final per-token values from merged statistics (maxima in raw logit units, sums relative to
// exp(max/tau)): lse_x = m_x/tau + log S_x and KL = A/S_t - lse_t + lse_s; when C is valid
// (not `far`) and the two distributions are close (|C' - mu| < 1/2, mu = A/S_t, C' = C/S_t),
// the algebraically equal KL = C' + log1p(C' - mu) - (C' - mu) avoids subtracting two ~log V
// numbers. The same quantity gives the gap lse_s - lse_t = log1p(C' - mu) (C' - mu =
// sum_v e_t (exp(-d_v) - 1) / S_t = S_s exp((m_s - m_t)/tau) / S_t - 1), exact to a few fp32
// ulps of the gap itself rather than of lse.
__device__ __forceinline__ double kl_from_stats(double mt, double st, double ms, double ss, double a, double cc,
                                                bool far, double inv_tau, double& lse_t, double& lse_s,
                                                double& gap) {
  lse_t = mt * inv_tau + log(st);
  lse_s = ms * inv_tau + log(ss);
  const double mu = a / st;
  const double cn = cc / st;
  const double u = cn - mu;
  if (!far && isfinite(u) && fabs(u) < 0.5) {
    gap = log1p(u);
    return cn + (log1p(u) - u);
  }
  gap = lse_s - lse_t;
  return mu - lse_t + lse_s;
}

// (p_s - p_t) for two columns, p_x = 2^(z_x c - b_x) with c = log2(e)/tau, b_x = lse_x log2(e).
// Where the two probabilities are close, |D| < 1/64 with D = (z_s - z_t) c - (lse_s - lse_t)
// log2(e) = log2(p_s / p_t), the difference is formed as p_t (2^D - 1), 2^D - 1 = e^x - 1 by
// its Taylor series x + x^2/2 + x^3/6 in x = D ln 2 (truncation < 6e-8 relative there), so
// that near-identical distributions lose no digits to cancellation; elsewhere |p_s - p_t| is
// at least 1% of p_t and the direct p_s - p_t keeps ~1e-4 relative accuracy, far below the
// bf16 rounding of the result. `ngl` is -(lse_s - lse_t) log2(e) from the precise gap.
__device__ __forceinline__ float2 prob_diff2(float2 zt, float2 zs, float2 c2, float2 nbt, float2 nbs, float2 ngl) {
  const float2 pt = ex2_approx2(__ffma2_rn(zt, c2, nbt));
  const float2 ps = ex2_approx2(__ffma2_rn(zs, c2, nbs));
  const float2 D = __ffma2_rn(__fadd2_rn(zs, make_float2(-zt.x, -zt.y)), c2, ngl);
  const float2 x = __fmul2_rn(D, make_float2(0.6931471805599453f, 0.6931471805599453f));
  float2 t = __ffma2_rn(x, make_float2(1.0f / 6.0f, 1.0f / 6.0f), make_float2(0.5f, 0.5f));
  t = __ffma2_rn(x, t, make_float2(1.0f, 1.0f));
  const float2 small = __fmul2_rn(pt, __fmul2_rn(x, t));
  const float2 big = __fadd2_rn(ps, make_float2(-pt.x, -pt.y));
  return make_float2(fabsf(D.x) < 0.015625f ? small.x : big.x, fabsf(D.y) < 0.015625f ? small.y : big.y);
}

}  // namespace hylo
