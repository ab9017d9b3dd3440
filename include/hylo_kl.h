/*
 * hylo_kl.h — C ABI of the fused hidden-state KL distillation loss (GB300, sm_103a).
 *
 * The operation. Stage II of HyLo trains the upcycled hybrid student end to end against a
 * Llama-3.1-8B teacher with a KL loss between the two next-token distributions, weight 1.0
 * and no cross-entropy term (HyLo-Llama-8MLA8GDN-8K-SFT reading notes, kwkr.cn, section
 * "two-stage training recipe", Stage II). To fit an 8B teacher at 64K tokens the loss takes
 * the FINAL HIDDEN STATES of both models (the teacher's LM head is skipped), applies both
 * LM-head projections itself, fuses the softmax with the KL, and walks the tokens in chunks
 * of 4096 (Long-Context Aware Upcycling digest, ftxj.github.io, section Method; section Key
 * Ideas). The pages print no formula; this library computes, for every token n:
 *
 *     z_s = h_s[n] W_s^T,  z_t = h_t[n] W_t^T                 (over the full vocabulary V)
 *     p_x = softmax(z_x / tau),  lse_x[n] = logsumexp(z_x / tau)
 *     kl[n] = KL(p_t || p_s) = sum_v p_t,v (log p_t,v - log p_s,v)
 *     loss  = (1/N) sum_n kl[n]
 * and the gradients of grad_scale * loss with respect to the student's h_s and W_s:
 *     G[n, v] = grad_scale * (p_s,v - p_t,v) / (tau N),  dh_s = G W_s,  dW_s = G^T h_s.
 * The N x V logit tensor is never stored. No teacher gradients (the teacher is frozen).
 *
 * Conventions shared by every call:
 *   - All pointers except `stream` and `workspace` sizes are DEVICE pointers on the current
 *     CUDA device, owned by the caller; the library never allocates or frees memory.
 *   - h_s [N, d_s], h_t [N, d_t], W_s [V, d_s], W_t [V, d_t]: bfloat16 bit patterns
 *     (uint16), row-major and contiguous (W like nn.Linear.weight: [vocab, hidden]).
 *   - d_s and d_t must be multiples of 8 (16-byte rows); every pointer must be 16-byte
 *     aligned. 1 <= N, V <= 2^31 - 1; 8 <= d_s, d_t <= 65536; tau finite and > 0.
 *   - float outputs are fp32. Every call is asynchronous on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and returns after enqueueing its kernels.
 *   - The returned status covers argument checks, the architecture check and launch errors.
 *     Device-side failures (a pipeline wait that exceeded its time limit) are recorded in a
 *     per-device status word; read it with hylo_kl_sync_status().
 *   - `workspace` is device scratch of at least hylo_kl_workspace_bytes(...) bytes, 256-byte
 *     aligned, not shared with a call still running on another stream.
 *   - Calls require an sm_103 device (GB300); otherwise HYLO_ERR_ARCH. There is no fallback.
 *   - Calls may be captured into a CUDA graph once one call has run eagerly on the device (it
 *     sets the kernels up). Replays give the same results and pace like eager calls: a forward
 *     captured with pacing also captures a memset of its 1280 pacing bytes.
 *
 * Accuracy (against an fp64 evaluation of the formulas above, bf16 inputs taken as exact):
 *   - kl[n] within 1e-3 (1 + kl[n]); loss within 1e-4 relative; lse_s, lse_t, lse_gap within
 *     2e-5 (1 + |lse|). The tensor cores accumulate each logit in fp32 over d/16 steps, which
 *     can drift by up to (d/16) 2^-23 of the logits' scale in one direction: above
 *     d = 13421 that bound exceeds 1e-4, and at the largest accepted d = 65536 the mean loss
 *     is held to 4.9e-4 relative instead (measured 1.3e-4).
 *   - hylo_kl_backward rounds G to bf16 once before the gradient products: about 1e-3
 *     relative (Frobenius) on spread distributions, but up to 2^-8 per token where one or two
 *     words dominate a token's gradient (near one-hot distributions, a student differing from
 *     its teacher on few words), which can exceed 2e-3. hylo_kl_backward_split keeps G to ~16
 *     bits (~1e-5) and meets 2e-3 on every input tested, at about +40% backward time.
 */
#ifndef HYLO_KL_H
#define HYLO_KL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HYLO_OK = 0,
  HYLO_ERR_NULL = -1,      /* a required pointer is NULL */
  HYLO_ERR_DIM = -2,       /* a size is out of range or not a multiple of 8 where required */
  HYLO_ERR_ALIGN = -3,     /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  HYLO_ERR_TAU = -4,       /* tau is not finite and > 0, or grad_scale is not finite */
  HYLO_ERR_WORKSPACE = -5, /* workspace_bytes is smaller than hylo_kl_workspace_bytes() */
  HYLO_ERR_CUDA = -6,      /* a CUDA runtime or driver call failed (see hylo_kl_last_error) */
  HYLO_ERR_TIMEOUT = -7,   /* a device-side pipeline wait exceeded its limit (device status) */
  HYLO_ERR_ARCH = -8       /* the current device is not sm_103 */
} hylo_status;

/* Bytes of device workspace that hylo_kl_forward and hylo_kl_backward need for these sizes:
 * the larger of the forward's per-token partial softmax statistics (6 x 32 x N fp32, O(N)) and
 * the backward's ring of three blocks of G = dL/dz_s (bf16; R tokens x bw words each, with
 * R = token_chunk rounded up to a multiple of 256, at most 32768, and bw = 128 MiB / (6 R)
 * rounded down to 256 words: at most 128 MiB in all, whatever N, V and token_chunk), plus 1280
 * bytes of counters (the forward's pacing words; the backward's work queue and completion
 * counts). So the extra memory is O(N) + 128 MiB, never O(N * V) or O(token_chunk * V).
 * Returns 0 for invalid sizes. token_chunk <= 0 means 4096. */
size_t hylo_kl_workspace_bytes(int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                               int64_t token_chunk);

/* Forward: kl[N], lse_s[N], lse_t[N] (natural-log units of z/tau) and loss[0] = mean(kl).
 * One fused pass: each CTA pair computes student and teacher logit tiles on the tensor cores
 * and folds them into running softmax/KL statistics; nothing of size N x V is written.
 * lse_gap[N] is optional (NULL: not written): lse_s - lse_t computed from the statistics as
 * log1p of a sum of per-word differences, so it keeps the digits that the difference of the
 * two fp32 lse values (each rounded at ~1e-6 of log V) loses when the distributions are
 * close; hand it to hylo_kl_backward.
 * token_chunk (<= 0 means 4096) does not change the results; the forward uses O(N) scratch
 * whatever its value. kl, lse_s, lse_t, lse_gap and loss may not alias the inputs. */
hylo_status hylo_kl_forward(const uint16_t* h_s, const uint16_t* W_s,
                            const uint16_t* h_t, const uint16_t* W_t,
                            int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                            float tau, int64_t token_chunk,
                            float* kl, float* lse_s, float* lse_t, float* lse_gap, float* loss,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward: dh_s [N, d_s] and dW_s [V, d_s] (fp32, OVERWRITTEN, not accumulated) for
 * grad_scale * loss, from the lse_s / lse_t (and lse_gap, if not NULL) that hylo_kl_forward
 * wrote for the same inputs. One persistent launch walks the tokens in blocks of R rows and
 * the vocabulary in blocks of bw words (see hylo_kl_workspace_bytes); per block it recomputes
 * both logit tiles, forms G into the workspace's ring, and adds G W_s into dh_s and G^T h_s
 * into dW_s on the tensor cores, in a fixed order (results are deterministic). At most
 * 2^30 work items (about N x V / 65536 + gradient tiles) per call, else HYLO_ERR_DIM. Where
 * p_s and p_t of a word agree to within a factor 2^(1/4), G takes the form
 * p_t (2^D - 1), D = log2(p_s / p_t) from the logit difference and lse_gap, which has no
 * cancellation; with lse_gap NULL the gap is lse_s - lse_t, whose rounding bounds the
 * relative accuracy of G at ~1e-6 / |p_s / p_t - 1|. Results match for any token_chunk up
 * to fp32 summation order. */
hylo_status hylo_kl_backward(const uint16_t* h_s, const uint16_t* W_s,
                             const uint16_t* h_t, const uint16_t* W_t,
                             int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                             float tau, int64_t token_chunk,
                             const float* lse_s, const float* lse_t, const float* lse_gap,
                             float grad_scale, float* dh_s, float* dW_s,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward with G kept to ~16 significant bits: G is stored as the sum of two bf16 terms,
 * bf16(G) and bf16(G - bf16(G)), and every dh_s / dW_s tile accumulates the products of both
 * terms (twice the k-blocks of the plain backward). Same arguments and results as
 * hylo_kl_backward, with a gradient error of ~1e-5 relative instead of the ~1e-3 that one
 * bf16 rounding of G leaves -- which matters where a token's gradient is dominated by one or
 * two words (near one-hot distributions, or a student that differs from its teacher on few
 * words), where one rounding alone can exceed 2e-3. The G ring is doubled (2 x 128 MiB at
 * most): pass at least hylo_kl_workspace_bytes_split(...) bytes. (The pages describe no such
 * variant; it is a precision option of this library.) */
size_t hylo_kl_workspace_bytes_split(int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                     int64_t token_chunk);
hylo_status hylo_kl_backward_split(const uint16_t* h_s, const uint16_t* W_s,
                                   const uint16_t* h_t, const uint16_t* W_t,
                                   int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                   float tau, int64_t token_chunk,
                                   const float* lse_s, const float* lse_t, const float* lse_gap,
                                   float grad_scale, float* dh_s, float* dW_s,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Forward that allocates nothing and takes no workspace. (The pages describe no such call;
 * it has no counterpart there.) It is for callers that cannot allocate device memory: a
 * plugin that may only use the buffers its host framework hands it, or a loop that must not
 * call cudaMalloc (which can synchronise the device) between steps. Instead of a workspace,
 * the per-token partial statistics go to a 16 MiB array built into the library, which every
 * GPU that loads the library holds until the process exits.
 *   - Same arguments, outputs and results as hylo_kl_forward, minus the workspace pair.
 *   - N may be at most 698997 ((16 MiB - 1280 bytes of pacing counters) / 24 bytes of
 *     statistics per token); larger N returns HYLO_ERR_DIM with a message. Larger N may use
 *     fewer vocabulary segments than hylo_kl_forward would, which changes results only by fp32
 *     summation order. Launches of several waves pace their clusters like hylo_kl_forward, with
 *     the counters at the end of the built-in array.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls share the one array per device and it keeps the last call's contents (each call
 *     writes every statistics slot it reads, and the pacing counters carry the launch's tag,
 *     so nothing needs clearing, except under stream capture, where they are cleared). Calls that overlap on the GPU
 *     (different streams, or threads without ordering) race on it: serialise them. */
hylo_status hylo_kl_forward_noalloc(const uint16_t* h_s, const uint16_t* W_s,
                                    const uint16_t* h_t, const uint16_t* W_t,
                                    int64_t N, int64_t d_s, int64_t d_t, int64_t V,
                                    float tau, int64_t token_chunk,
                                    float* kl, float* lse_s, float* lse_t, float* lse_gap,
                                    float* loss, cudaStream_t stream);

/* "Fused KL" on precomputed logits (Long-Context Aware Upcycling digest, section Key Ideas:
 * the memory stack lists Fused KL beside the Fused Hidden-State KL). z_s and z_t are the
 * student's and teacher's logits, [N, V] bf16 bit patterns with row stride ld elements
 * (ld >= V, a multiple of 8; pointers 16-byte aligned). Writes kl[N], lse_s[N], lse_t[N] and
 * loss[0] = mean(kl) exactly as hylo_kl_forward would for logits z = h W^T, and, if dz_s is
 * not NULL, the gradient of grad_scale * loss with respect to z_s,
 * dz_s[n, v] = grad_scale * (p_s - p_t) / (tau N), as bf16 in an [N, ld] buffer (columns
 * v >= V untouched). One kernel; reads each logit once for the statistics and, with a
 * gradient, once more for dz_s (from DRAM: between a row's two passes the GPU streams more
 * than L2 holds). Needs no workspace. */
hylo_status hylo_fused_kl_logits(const uint16_t* z_s, const uint16_t* z_t,
                                 int64_t N, int64_t V, int64_t ld,
                                 float tau, float grad_scale,
                                 float* kl, float* lse_s, float* lse_t, float* loss,
                                 uint16_t* dz_s, cudaStream_t stream);

/* Stage-I Enhanced-ILD alignment loss (Long-Context Aware Upcycling digest, section Method:
 * L_ILD = sum over layers of ||h_s - h_t||_2 + ||a_s - a_t||_2, layer outputs h and token-mixer
 * outputs a; HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage I). S (student) and T (teacher)
 * stack the aligned tensors as [P, N, d] bf16 bit patterns, row-major and contiguous (P = one
 * entry per layer and per kind, N tokens, d a multiple of 8; pointers 16-byte aligned).
 * Writes norms[p*N + n] = ||S[p,n,:] - T[p,n,:]||_2 (fp32), loss[0] = sum(norms) / N, and, if
 * dS is not NULL, the gradient of grad_scale * loss with respect to S,
 * grad_scale * (S - T) / (N ||S - T||) per row (0 where the row difference is 0), as bf16
 * [P, N, d]. The teacher gets no gradient. Needs no workspace. */
hylo_status hylo_ild_loss(const uint16_t* S, const uint16_t* T, int64_t P, int64_t N, int64_t d,
                          float grad_scale, float* norms, float* loss, uint16_t* dS,
                          cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the current device's status word:
 * HYLO_OK, or HYLO_ERR_TIMEOUT if a kernel gave up on a pipeline wait since the last read
 * (its outputs are then invalid), or HYLO_ERR_CUDA if the synchronisation failed. */
hylo_status hylo_kl_sync_status(cudaStream_t stream);

/* Diagnostic (the pages have no counterpart): enqueues on `stream` a one-warp kernel that
 * waits on a pipeline barrier nothing ever signals, through the same time-limited wait the
 * loss kernels use. After limit_ms (1..1000) the wait gives up, records a timeout in the device
 * status word and the kernel returns, so the next hylo_kl_sync_status() returns
 * HYLO_ERR_TIMEOUT and the device stays usable. Returns HYLO_ERR_DIM for other limits. */
hylo_status hylo_kl_selftest_wait_timeout(int limit_ms, cudaStream_t stream);

/* Thread-local text describing the last non-OK status returned on this thread ("" if none).
 * The pointer stays valid until the next library call on the same thread. */
const char* hylo_kl_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* HYLO_KL_H */
