// Host side of the C ABI declared in include/hylo_kl.h: argument checks, the sm_103 guard,
// TMA tensor-map construction, the vocabulary-segment heuristic, the backward token-chunk
// loop, and the per-device status word that kernels use to report a timed-out wait.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/hylo_kl.h"
#include "hylo_internal.h"

namespace hylo {
namespace {

__device__ int g_device_status;  // 0, or the first device-side error code since the last read

thread_local std::string g_last_error;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  bool sm103 = false;
  int sms = 0;
  int fused_clusters = 0;  // 2-CTA clusters of the fused kernels resident at once
  int logits_clusters = 0; // clusters of the logits kernel resident at once
  int pipe_clusters = 0;   // 2-CTA clusters of the pipelined backward resident at once
  unsigned pace_epoch = 0;  // epoch of the last paced fused launch on this device
  int* status = nullptr;
  std::string why;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

hylo_status fail(hylo_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

hylo_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HYLO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Vocabulary columns per fused pair tile.
constexpr int fused_bn() { return kFusedBN; }

unsigned long long wait_limit_ns() {
  static const unsigned long long v = [] {
    const char* s = std::getenv("HYLO_KL_WAIT_LIMIT_MS");
    long long ms = s ? std::atoll(s) : 5000;
    if (ms <= 0) ms = 5000;
    return static_cast<unsigned long long>(ms) * 1000000ull;
  }();
  return v;
}

// Looks up (once per device) the architecture, SM count, status-word address and kernel
// attributes of the current device.
hylo_status current_device(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(HYLO_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.sm103 = (major == 10 && minor == 3);
    if (!d.sm103) {
      char b[128];
      snprintf(b, sizeof(b), "device %d is sm_%d%d; this library runs only on sm_103 (GB300)", dev, major, minor);
      d.why = b;
    } else {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
      d.status = static_cast<int*>(p);
      if ((e = fused_prepare(fused_bn(), &d.fused_clusters)) != cudaSuccess ||
          (e = bwd_pipe_prepare(&d.pipe_clusters)) != cudaSuccess ||
          (e = kl_logits_prepare(&d.logits_clusters)) != cudaSuccess)
        return cuda_fail(e, "kernel set-up");
      if (d.pipe_clusters < 1 || d.fused_clusters < 1 || d.logits_clusters < 1)
        return fail(HYLO_ERR_CUDA, "no thread-block cluster of the kernels fits on the device");
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
          return fail(HYLO_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    d.init = true;
  }
  if (!d.sm103) return fail(HYLO_ERR_ARCH, "%s", d.why.c_str());
  *out = &d;
  return HYLO_OK;
}

// 2-D tensor map, 128-byte swizzle, zero fill outside the tensor.
hylo_status make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HYLO_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult %d", static_cast<int>(r));
  return HYLO_OK;
}

// A fresh epoch (1..65535) for a paced fused launch: the pacing counters are never cleared,
// their words carry the epoch of the launch that wrote them.
unsigned next_epoch(DeviceState* d) {
  std::lock_guard<std::mutex> lock(g_mu);
  d->pace_epoch = d->pace_epoch % 65534u + 2u;  // 2..65535; tag 1 is reserved for captured launches
  return d->pace_epoch;
}


// 3-D tensor map [outer2][outer1][inner] (contiguous), zero fill outside; 128-byte swizzle
// unless `swizzle` says otherwise.
hylo_status make_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer1,
                        uint64_t outer2, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer1,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[3] = {inner, outer1, outer2};
  cuuint64_t strides[2] = {row_bytes, row_bytes * outer1};
  cuuint32_t box[3] = {box_inner, box_outer1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HYLO_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed with CUresult %d", static_cast<int>(r));
  return HYLO_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The backward stages G = dL/dz_s (bf16) in a ring of kGRing blocks of R tokens x bw words:
// at most kGBlockBytes in all, whatever N, V or token_chunk. R = token_chunk rounded up to a
// multiple of 256 (at most kMaxBlockTokens, at most N rounded up), so bw is at least
// kGBlockBytes / (2 kGRing kMaxBlockTokens) = 682 -> 512 words.
constexpr int64_t kMaxBlockTokens = 32768;

int64_t pipe_rows(int64_t N, int64_t token_chunk) {
  int64_t c = token_chunk <= 0 ? 4096 : token_chunk;
  if (c > kMaxBlockTokens) c = kMaxBlockTokens;
  c = cdiv(c, 256) * 256;
  const int64_t n = cdiv(N, 256) * 256;
  return c < n ? c : n;
}

int64_t pipe_width(int64_t R, int64_t V) {
  const int64_t w = kGBlockBytes / (kGRing * R * 2) / 256 * 256;
  const int64_t vmax = cdiv(V, 256) * 256;
  return w < vmax ? w : vmax;
}

bool sizes_ok(int64_t N, int64_t d_s, int64_t d_t, int64_t V) {
  return N >= 1 && V >= 1 && N <= 0x7fffffffLL && V <= 0x7fffffffLL && d_s >= 8 && d_t >= 8 && d_s <= 65536 &&
         d_t <= 65536 && d_s % 8 == 0 && d_t % 8 == 0;
}

size_t fwd_bytes(int64_t N) { return static_cast<size_t>(kStatFields) * kMaxSegments * N * sizeof(float); }

// Bytes of the backward's G ring (one bf16 term): at most kGBlockBytes.
size_t bwd_bytes(int64_t N, int64_t V, int64_t token_chunk) {
  const int64_t R = pipe_rows(N, token_chunk);
  return static_cast<size_t>(kGRing) * R * pipe_width(R, V) * 2;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The fused kernels' pacing counters (one per cluster, then the switch that turns pacing off)
// follow the statistics or G region.
constexpr size_t kProgressBytes = ((kMaxClusters + 1) * sizeof(unsigned long long) + 255) & ~size_t(255);

// The pacing words' tag for a forward launch. An eager launch takes the next rolling tag and
// needs no clearing (words of earlier launches carry other tags). A launch captured into a CUDA
// graph would replay its captured tag, so during capture the words are cleared on the stream
// first (the memset is captured with the launch) and the fixed tag 1 is used: every replay
// starts from cleared words and paces its clusters like an eager launch.
hylo_status pace_tag(DeviceState* dev, unsigned long long* progress, cudaStream_t stream, unsigned* tag) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs == cudaStreamCaptureStatusActive) {
    if ((e = cudaMemsetAsync(progress, 0, kProgressBytes, stream)) != cudaSuccess)
      return cuda_fail(e, "clear the pacing words");
    *tag = 1u;
    return HYLO_OK;
  }
  *tag = next_epoch(dev);
  return HYLO_OK;
}

// Pacing matters only when clusters run several units each (units > grid); the counters' words
// hold the unit index in 24 bits.
bool pace_launch(int64_t units, int64_t grid) { return units > grid && units / grid < (int64_t(1) << 23); }

// Number of vocabulary segments per pair tile: the work units (256-token tile, segment) are
// dealt round-robin to the persistent CTA pairs, so pick the split that minimises
// waves x (vocab tiles per segment), with a small cost per extra segment.
double segment_cost(int64_t token_tiles, int64_t vtiles, int workers, int s) {
  const int64_t units = token_tiles * s;
  const int64_t waves = cdiv(units, workers);
  const int64_t per = cdiv(vtiles, s);
  return static_cast<double>(waves * per) * (1.0 + 0.002 * s);
}

int choose_segments(int64_t token_tiles, int64_t vtiles, int workers) {
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= kMaxSegments && s <= vtiles; ++s) {
    const double cost = segment_cost(token_tiles, vtiles, workers, s);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

hylo_status check_common(const void* h_s, const void* W_s, const void* h_t, const void* W_t, int64_t N, int64_t d_s,
                         int64_t d_t, int64_t V, float tau, void* workspace, size_t workspace_bytes,
                         size_t need) {
  if (!h_s || !W_s || !h_t || !W_t || !workspace) return fail(HYLO_ERR_NULL, "a required pointer is NULL");
  if (!sizes_ok(N, d_s, d_t, V))
    return fail(HYLO_ERR_DIM, "invalid sizes N=%lld d_s=%lld d_t=%lld V=%lld (d must be a multiple of 8, 8..65536)",
                static_cast<long long>(N), static_cast<long long>(d_s), static_cast<long long>(d_t),
                static_cast<long long>(V));
  if (!aligned(h_s, 16) || !aligned(W_s, 16) || !aligned(h_t, 16) || !aligned(W_t, 16))
    return fail(HYLO_ERR_ALIGN, "input pointers must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(HYLO_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (!(std::isfinite(tau) && tau > 0.f)) return fail(HYLO_ERR_TAU, "tau must be finite and > 0");
  if (workspace_bytes < need)
    return fail(HYLO_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes, need);
  return HYLO_OK;
}

}  // namespace
}  // namespace hylo

using namespace hylo;

extern "C" {

size_t hylo_kl_workspace_bytes(int64_t N, int64_t d_s, int64_t d_t, int64_t V, int64_t token_chunk) {
  g_last_error.clear();
  if (!sizes_ok(N, d_s, d_t, V)) return 0;
  const size_t f = round256(fwd_bytes(N)), b = round256(bwd_bytes(N, V, token_chunk));
  return (f > b ? f : b) + kProgressBytes;
}

size_t hylo_kl_workspace_bytes_split(int64_t N, int64_t d_s, int64_t d_t, int64_t V, int64_t token_chunk) {
  g_last_error.clear();
  if (!sizes_ok(N, d_s, d_t, V)) return 0;
  const size_t f = round256(fwd_bytes(N)), b = 2 * round256(bwd_bytes(N, V, token_chunk));
  return (f > b ? f : b) + kProgressBytes;
}

hylo_status hylo_kl_forward(const uint16_t* h_s, const uint16_t* W_s, const uint16_t* h_t, const uint16_t* W_t,
                            int64_t N, int64_t d_s, int64_t d_t, int64_t V, float tau, int64_t token_chunk,
                            float* kl, float* lse_s, float* lse_t, float* lse_gap, float* loss, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
  g_last_error.clear();
  (void)token_chunk;  // the forward needs O(N) scratch whatever the chunk
  if (!kl || !lse_s || !lse_t || !loss) return fail(HYLO_ERR_NULL, "an output pointer is NULL");
  const size_t stats_bytes = sizes_ok(N, d_s, d_t, V) ? round256(fwd_bytes(N)) : 0;
  hylo_status st = check_common(h_s, W_s, h_t, W_t, N, d_s, d_t, V, tau, workspace, workspace_bytes,
                                stats_bytes + kProgressBytes);
  if (st != HYLO_OK) return st;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != HYLO_OK) return st;

  CUtensorMap m_hs, m_Ws, m_ht, m_Wt;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((st = make_map(&m_hs, h_s, bf, d_s, N, d_s * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&m_ht, h_t, bf, d_t, N, d_t * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&m_Ws, W_s, bf, d_s, V, d_s * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;
  if ((st = make_map(&m_Wt, W_t, bf, d_t, V, d_t * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;

  FusedParams p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.kb_s = static_cast<int>(cdiv(d_s, kBK));
  p.kb_t = static_cast<int>(cdiv(d_t, kBK));
  p.token_tiles = static_cast<int>(cdiv(N, 2 * kBM));
  p.vtiles = static_cast<int>(cdiv(V, fused_bn()));
  p.nseg = choose_segments(p.token_tiles, p.vtiles, dev->fused_clusters);
  p.units = p.token_tiles * p.nseg;
  p.group = 1;  // tile-major: least DRAM traffic (measured at 64K: 229 GB per launch against 291-417 GB
                // for raster groups of 4-32 pair tiles, 58.7 against up to 66.7 ms)
  p.c = 1.4426950408889634f / tau;
  p.inv_tau = 1.0f / tau;
  p.part = static_cast<float*>(workspace);
  p.ctl = WaitCtl{dev->status, wait_limit_ns()};
  const int grid = p.units < dev->fused_clusters ? p.units : dev->fused_clusters;

  if (pace_launch(p.units, grid)) {
    p.progress = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + stats_bytes);
    unsigned tag = 0;
    if ((st = pace_tag(dev, p.progress, stream, &tag)) != HYLO_OK) return st;
    p.epoch = tag;
  }
  cudaError_t e = launch_fused(fused_bn(), m_hs, m_Ws, m_ht, m_Wt, p, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch fused forward");
  e = launch_combine(p.part, p.N, p.nseg, p.inv_tau, kl, lse_s, lse_t, lse_gap, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch combine");
  e = launch_mean(kl, p.N, loss, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch mean");
  return HYLO_OK;
}

}  // extern "C"

namespace {

// Both backward entry points: one launch of the pipelined backward (kl_bwd_pipe.cu) over
// token blocks of pipe_rows() tokens and vocabulary blocks of pipe_width() words, with the G
// ring in the workspace. split: G is also kept as bf16(G - bf16(G)) in a second ring, and each
// gradient tile accumulates the products of both terms.
hylo_status backward_impl(const uint16_t* h_s, const uint16_t* W_s, const uint16_t* h_t, const uint16_t* W_t,
                          int64_t N, int64_t d_s, int64_t d_t, int64_t V, float tau, int64_t token_chunk,
                          const float* lse_s, const float* lse_t, const float* lse_gap, float grad_scale,
                          float* dh_s, float* dW_s, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                          bool split) {
  g_last_error.clear();
  if (!lse_s || !lse_t || !dh_s || !dW_s) return fail(HYLO_ERR_NULL, "an lse or gradient pointer is NULL");
  const size_t g_bytes = sizes_ok(N, d_s, d_t, V) ? round256(bwd_bytes(N, V, token_chunk)) : 0;
  const size_t g_total = split ? 2 * g_bytes : g_bytes;
  hylo_status st = check_common(h_s, W_s, h_t, W_t, N, d_s, d_t, V, tau, workspace, workspace_bytes,
                                g_total + kProgressBytes);
  if (st != HYLO_OK) return st;
  if (!std::isfinite(grad_scale)) return fail(HYLO_ERR_TAU, "grad_scale must be finite");
  if (!aligned(dh_s, 16) || !aligned(dW_s, 16)) return fail(HYLO_ERR_ALIGN, "gradient pointers must be 16-byte aligned");
  const int64_t R = pipe_rows(N, token_chunk), bw = pipe_width(R, V);
  const int64_t TB = cdiv(N, R), VB = cdiv(V, bw), ntd = cdiv(d_s, kGemmBN);
  // work items: per block, its 256 x 256 G tiles and its dW_s and dh_s tiles (< 2^30 so that
  // the queue index and the completion counts fit their 32-bit counters)
  const int64_t items = cdiv(N, 256) * cdiv(V, 256) + (TB * cdiv(V, 256) + VB * cdiv(N, 256)) * ntd;
  if (items >= (int64_t(1) << 30))
    return fail(HYLO_ERR_DIM, "N=%lld x V=%lld needs %lld backward work items, more than 2^30",
                static_cast<long long>(N), static_cast<long long>(V), static_cast<long long>(items));
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != HYLO_OK) return st;

  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUtensorMap maps[kPipeMaps];
  uint16_t* G = static_cast<uint16_t*>(workspace);
  const uint64_t slots = static_cast<uint64_t>(split ? 2 * kGRing : kGRing);
  if ((st = make_map(&maps[0], h_s, bf, d_s, N, d_s * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&maps[1], h_t, bf, d_t, N, d_t * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&maps[2], W_s, bf, d_s, V, d_s * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;
  if ((st = make_map(&maps[3], W_t, bf, d_t, V, d_t * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;
  if ((st = make_map(&maps[4], W_s, bf, d_s, V, d_s * 2, 64, kBK)) != HYLO_OK) return st;  // MN-major B of dh
  if ((st = make_map(&maps[5], h_s, bf, d_s, N, d_s * 2, 64, kBK)) != HYLO_OK) return st;  // MN-major B of dW
  if ((st = make_map(&maps[6], dh_s, f32, d_s, N, d_s * 4, 32, 32)) != HYLO_OK) return st;
  if ((st = make_map(&maps[7], dW_s, f32, d_s, V, d_s * 4, 32, 32)) != HYLO_OK) return st;
  if ((st = make_map_3d(&maps[8], G, bf, bw, R, slots, bw * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != HYLO_OK)
    return st;  // G tile stores (32 x 32)
  if ((st = make_map_3d(&maps[9], G, bf, bw, R, slots, bw * 2, kBK, kBM)) != HYLO_OK) return st;  // K-major A of dh
  if ((st = make_map_3d(&maps[10], G, bf, bw, R, slots, bw * 2, 64, kBK)) != HYLO_OK) return st;  // MN-major A of dW

  BwdPipeParams p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.d_s = static_cast<int>(d_s);
  p.kb_s = static_cast<int>(cdiv(d_s, kBK));
  p.kb_t = static_cast<int>(cdiv(d_t, kBK));
  p.ntd = static_cast<int>(ntd);
  p.R = static_cast<int>(R);
  p.bw = static_cast<int>(bw);
  p.TB = static_cast<int>(TB);
  p.VB = static_cast<int>(VB);
  p.B = static_cast<int>(TB * VB);
  p.c = 1.4426950408889634f / tau;
  p.gscale = static_cast<float>(static_cast<double>(grad_scale) / (static_cast<double>(tau) * N));
  p.lse_s = lse_s;
  p.lse_t = lse_t;
  p.lse_gap = lse_gap;
  p.split = split ? 1 : 0;
  p.ctrl = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + g_total);
  p.ctl = WaitCtl{dev->status, wait_limit_ns()};
  cudaError_t e = cudaMemsetAsync(p.ctrl, 0, kPipeCtrlWords * sizeof(unsigned), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clear the backward's work counters");
  const int clusters = static_cast<int>(items < dev->pipe_clusters ? items : dev->pipe_clusters);
  e = launch_bwd_pipe(maps, p, clusters, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch pipelined backward");
  return HYLO_OK;
}

}  // namespace

extern "C" {

hylo_status hylo_kl_backward(const uint16_t* h_s, const uint16_t* W_s, const uint16_t* h_t, const uint16_t* W_t,
                             int64_t N, int64_t d_s, int64_t d_t, int64_t V, float tau, int64_t token_chunk,
                             const float* lse_s, const float* lse_t, const float* lse_gap, float grad_scale,
                             float* dh_s, float* dW_s, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return backward_impl(h_s, W_s, h_t, W_t, N, d_s, d_t, V, tau, token_chunk, lse_s, lse_t, lse_gap, grad_scale, dh_s,
                       dW_s, workspace, workspace_bytes, stream, false);
}

hylo_status hylo_kl_backward_split(const uint16_t* h_s, const uint16_t* W_s, const uint16_t* h_t,
                                   const uint16_t* W_t, int64_t N, int64_t d_s, int64_t d_t, int64_t V, float tau,
                                   int64_t token_chunk, const float* lse_s, const float* lse_t, const float* lse_gap,
                                   float grad_scale, float* dh_s, float* dW_s, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  return backward_impl(h_s, W_s, h_t, W_t, N, d_s, d_t, V, tau, token_chunk, lse_s, lse_t, lse_gap, grad_scale, dh_s,
                       dW_s, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace hylo {
namespace {

// Waits on an mbarrier that nothing ever arrives on, through the same time-limited wait the
// pipelined kernels use: the wait gives up after the limit and records a timeout in the
// device status word, then the kernel returns normally.
__global__ void wait_timeout_kernel(WaitCtl ctl) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(&bar, 0, &abort_flag, ctl, 99);
}

}  // namespace
}  // namespace hylo

extern "C" {

hylo_status hylo_kl_selftest_wait_timeout(int limit_ms, cudaStream_t stream) {
  g_last_error.clear();
  if (limit_ms < 1 || limit_ms > 1000) return fail(HYLO_ERR_DIM, "limit_ms must be in [1, 1000]");
  DeviceState* dev = nullptr;
  hylo_status st = current_device(&dev);
  if (st != HYLO_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(WaitCtl{dev->status, static_cast<unsigned long long>(limit_ms) * 1000000ull});
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch wait-timeout self-test");
  return HYLO_OK;
}

hylo_status hylo_fused_kl_logits(const uint16_t* z_s, const uint16_t* z_t, int64_t N, int64_t V, int64_t ld,
                                 float tau, float grad_scale, float* kl, float* lse_s, float* lse_t, float* loss,
                                 uint16_t* dz_s, cudaStream_t stream) {
  g_last_error.clear();
  if (!z_s || !z_t || !kl || !lse_s || !lse_t || !loss) return fail(HYLO_ERR_NULL, "a required pointer is NULL");
  if (N < 1 || V < 1 || N > 0x7fffffffLL || V > 0x7fffffffLL || ld < V || ld % 8 != 0)
    return fail(HYLO_ERR_DIM, "invalid sizes N=%lld V=%lld ld=%lld (need ld >= V, ld a multiple of 8)",
                static_cast<long long>(N), static_cast<long long>(V), static_cast<long long>(ld));
  if (!aligned(z_s, 16) || !aligned(z_t, 16) || (dz_s && !aligned(dz_s, 16)))
    return fail(HYLO_ERR_ALIGN, "logit pointers must be 16-byte aligned");
  if (!(std::isfinite(tau) && tau > 0.f)) return fail(HYLO_ERR_TAU, "tau must be finite and > 0");
  if (!std::isfinite(grad_scale)) return fail(HYLO_ERR_TAU, "grad_scale must be finite");
  DeviceState* dev = nullptr;
  hylo_status st = current_device(&dev);
  if (st != HYLO_OK) return st;
  const float gscale = static_cast<float>(static_cast<double>(grad_scale) / (static_cast<double>(tau) * N));
  const int clusters = N < dev->logits_clusters ? static_cast<int>(N) : dev->logits_clusters;
  cudaError_t e = launch_kl_logits(z_s, z_t, dz_s, ld, static_cast<int>(N), static_cast<int>(V), tau, gscale, kl, lse_s,
                                   lse_t, WaitCtl{dev->status, wait_limit_ns()}, clusters, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch logits KL");
  e = launch_mean(kl, static_cast<int>(N), loss, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch mean");
  return HYLO_OK;
}

hylo_status hylo_ild_loss(const uint16_t* S, const uint16_t* T, int64_t P, int64_t N, int64_t d, float grad_scale,
                          float* norms, float* loss, uint16_t* dS, cudaStream_t stream) {
  g_last_error.clear();
  if (!S || !T || !norms || !loss) return fail(HYLO_ERR_NULL, "a required pointer is NULL");
  if (P < 1 || N < 1 || d < 8 || d % 8 != 0 || d > 65536 || N > (int64_t(1) << 40) / P)
    return fail(HYLO_ERR_DIM, "invalid sizes P=%lld N=%lld d=%lld (d a multiple of 8, 8..65536)",
                static_cast<long long>(P), static_cast<long long>(N), static_cast<long long>(d));
  if (!aligned(S, 16) || !aligned(T, 16) || (dS && !aligned(dS, 16)))
    return fail(HYLO_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(grad_scale)) return fail(HYLO_ERR_TAU, "grad_scale must be finite");
  DeviceState* dev = nullptr;
  hylo_status st = current_device(&dev);
  if (st != HYLO_OK) return st;
  cudaError_t e = launch_ild(S, T, P, N, static_cast<int>(d), grad_scale, norms, loss, dS, dev->sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch ILD loss");
  return HYLO_OK;
}

hylo_status hylo_kl_sync_status(cudaStream_t stream) {
  g_last_error.clear();
  DeviceState* dev = nullptr;
  hylo_status st = current_device(&dev);
  if (st != HYLO_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int code = 0;
  if ((e = cudaMemcpyFromSymbol(&code, g_device_status, sizeof(int))) != cudaSuccess)
    return cuda_fail(e, "read device status");
  if (code != 0) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int))) != cudaSuccess)
      return cuda_fail(e, "clear device status");
    return fail(HYLO_ERR_TIMEOUT, "a device-side pipeline wait timed out (site %d)", code - kDevTimeoutBase);
  }
  return HYLO_OK;
}

const char* hylo_kl_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Forward without caller-provided workspace, for callers that cannot allocate device memory.
// The per-token partial statistics live in a fixed file-scope device array instead.
namespace hylo {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr size_t kNoAllocFloats = kNoAllocScratchBytes / sizeof(float);
// The last kProgressBytes hold the pacing counters; the statistics get the rest.
constexpr size_t kNoAllocStatFloats = (kNoAllocScratchBytes - kProgressBytes) / sizeof(float);
// Largest N whose statistics fit with one vocabulary segment: (16 MiB - 1280 B) / (6 fields * 4 B).
constexpr int64_t kNoAllocMaxTokens = static_cast<int64_t>(kNoAllocStatFloats / kStatFields);

// Every device that loads this library holds this array until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

float* g_noalloc_ptr[kMaxDevices] = {};

// Looks up, once per device and with that device current, the device address of the array.
// Host code must not pass g_noalloc_scratch itself to a kernel: on the host that name is only a
// stand-in for the device symbol.
hylo_status noalloc_scratch(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(HYLO_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return HYLO_OK;
}

}  // namespace
}  // namespace hylo

extern "C" hylo_status hylo_kl_forward_noalloc(const uint16_t* h_s, const uint16_t* W_s, const uint16_t* h_t,
                                               const uint16_t* W_t, int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                               float tau, int64_t token_chunk, float* kl, float* lse_s,
                                               float* lse_t, float* lse_gap, float* loss, cudaStream_t stream) {
  g_last_error.clear();
  (void)token_chunk;
  if (!h_s || !W_s || !h_t || !W_t || !kl || !lse_s || !lse_t || !loss)
    return fail(HYLO_ERR_NULL, "a required pointer is NULL");
  if (!sizes_ok(N, d_s, d_t, V))
    return fail(HYLO_ERR_DIM, "invalid sizes N=%lld d_s=%lld d_t=%lld V=%lld (d must be a multiple of 8, 8..65536)",
                static_cast<long long>(N), static_cast<long long>(d_s), static_cast<long long>(d_t),
                static_cast<long long>(V));
  if (N > kNoAllocMaxTokens)
    return fail(HYLO_ERR_DIM, "N=%lld exceeds the %lld tokens whose statistics fit the %zu-byte built-in scratch",
                static_cast<long long>(N), static_cast<long long>(kNoAllocMaxTokens), kNoAllocScratchBytes);
  if (!aligned(h_s, 16) || !aligned(W_s, 16) || !aligned(h_t, 16) || !aligned(W_t, 16))
    return fail(HYLO_ERR_ALIGN, "input pointers must be 16-byte aligned");
  if (!(std::isfinite(tau) && tau > 0.f)) return fail(HYLO_ERR_TAU, "tau must be finite and > 0");
  DeviceState* dev = nullptr;
  hylo_status st = current_device(&dev);
  if (st != HYLO_OK) return st;
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != HYLO_OK) return st;

  CUtensorMap m_hs, m_Ws, m_ht, m_Wt;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((st = make_map(&m_hs, h_s, bf, d_s, N, d_s * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&m_ht, h_t, bf, d_t, N, d_t * 2, kBK, kBM)) != HYLO_OK) return st;
  if ((st = make_map(&m_Ws, W_s, bf, d_s, V, d_s * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;
  if ((st = make_map(&m_Wt, W_t, bf, d_t, V, d_t * 2, kBK, fused_bn() / 2)) != HYLO_OK) return st;

  FusedParams p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.kb_s = static_cast<int>(cdiv(d_s, kBK));
  p.kb_t = static_cast<int>(cdiv(d_t, kBK));
  p.token_tiles = static_cast<int>(cdiv(N, 2 * kBM));
  p.vtiles = static_cast<int>(cdiv(V, fused_bn()));
  // as many vocabulary segments as the heuristic wants, but no more than the scratch holds
  const int64_t fit = static_cast<int64_t>(kNoAllocStatFloats) / (static_cast<int64_t>(kStatFields) * N);
  const int want = choose_segments(p.token_tiles, p.vtiles, dev->fused_clusters);
  p.nseg = static_cast<int>(want < fit ? want : fit);
  p.units = p.token_tiles * p.nseg;
  p.group = 1;  // tile-major, as in hylo_kl_forward
  p.c = 1.4426950408889634f / tau;
  p.inv_tau = 1.0f / tau;
  p.part = scratch;  // every (segment, token) slot read by the combine step is written first
  p.ctl = WaitCtl{dev->status, wait_limit_ns()};
  const int grid = p.units < dev->fused_clusters ? p.units : dev->fused_clusters;
  if (pace_launch(p.units, grid)) {  // counters at the scratch's tail; epoch-tagged (cleared only under capture)
    p.progress = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(scratch) + kNoAllocScratchBytes -
                                                       kProgressBytes);
    unsigned tag = 0;
    if ((st = pace_tag(dev, p.progress, stream, &tag)) != HYLO_OK) return st;
    p.epoch = tag;
  }

  cudaError_t e = launch_fused(fused_bn(), m_hs, m_Ws, m_ht, m_Wt, p, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch fused forward");
  e = launch_combine(p.part, p.N, p.nseg, p.inv_tau, kl, lse_s, lse_t, lse_gap, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch combine");
  e = launch_mean(kl, p.N, loss, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launch mean");
  return HYLO_OK;
}
