/*
 * fa2.h -- C ABI of libfa2.so, the FlashAttention-2 forward pass (and its
 * backward pass) for GB300 (sm_103a).
 *
 * The operation (per batch b, head h and query row i):
 *
 *     s_ij   = scale * sum_c Q[b,h,i,c] * K[b,h,j,c]
 *     O[b,h,i,:] = sum_{j in J_i} softmax_{j in J_i}(s_ij) * V[b,h,j,:]
 *     LSE[b,h,i] = log sum_{j in J_i} exp(s_ij)           (natural log)
 *
 * with J_i = {0 .. Nk-1}, or {j : j <= i} when causal (top-left aligned:
 * query i sees keys 0..i, so no row is ever empty).  This is exact
 * scaled-dot-product attention computed the FlashAttention-2 way: Q blocks in
 * the outer loop (one thread block each), K/V blocks streamed in the inner
 * loop with an online softmax (running max m and sum l, correction by
 * exp(m_old - m_new)), normalisation once after the loop, and the per-row
 * logsumexp L = m + log l as a second output.  Sources: "FlashAttention 怎么做?
 * online softmax 怎么更新?" (sections 推导/关键公式 and the FlashAttention-2
 * question), "FlashAttention-2 算法架构升级" (sections 一 and 二),
 * "Flash Attention 全解析(上)" (sections 1.2 and 3.2), and the host wrapper of
 * "Triton内核实战" (separate query and key lengths, an fp32 [B,H,Lq] side
 * buffer for the row statistic).
 *
 * Memory and ownership.  All tensor arguments are DEVICE pointers owned by
 * the caller; the library never allocates, frees or keeps them.  Layouts are
 * dense row-major BHSD:
 *     Q   bf16  [B, H, Nq, d]      K, V  bf16  [B, H, Nk, d]
 *     O   fp32  [B, H, Nq, d]      LSE   fp32  [B, H, Nq]
 * Q, K, V and O must be 16-byte aligned, LSE 4-byte aligned.  O and LSE are
 * fully overwritten; no other memory is written.  The library keeps no state
 * between calls apart from a per-device status word (fa2_device_status).
 *
 * Errors.  Calls are asynchronous on `stream`.  The return value reports
 * argument errors (found on the host before anything is launched; nothing is
 * written then) and launch errors.  A kernel that gives up waiting on one of
 * its internal barriers (about 2 s) returns early, leaves its outputs
 * incomplete and sets the device status word, which fa2_device_status reads.
 *
 * Kernel variants.  Two environment variables, read at every call, choose
 * between kernels that compute the same results (up to the rounding order
 * of their sums) for head dimension 128: FA2_FORWARD_KERNEL = "pair" runs
 * the forward passes on CTA pairs (two-SM tensor-core MMAs), "single" on
 * one-CTA kernels; FA2_BACKWARD_KERNEL = "two_tile" runs the backward pass
 * with two 64-query tiles in flight, "one_tile" with one 128-query tile.
 * Unset (or any other value) selects the default, the measured faster
 * choice: "single" and "one_tile".
 */
#ifndef FA2_H
#define FA2_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *fa2_stream_t;

typedef enum {
  FA2_OK = 0,
  FA2_ERR_NULL = 1,     /* a required pointer is NULL */
  FA2_ERR_ALIGN = 2,    /* Q/K/V/O not 16-byte aligned, or LSE not 4-byte aligned */
  FA2_ERR_SHAPE = 3,    /* negative size, Nk < 1 with rows to compute, or a size past the limits */
  FA2_ERR_HEADDIM = 4,  /* d not supported (forward 64, 128 or 256; SIMT and backward 64 or 128) */
  FA2_ERR_LAUNCH = 5,   /* the CUDA launch or a CUDA call failed */
  FA2_ERR_TIMEOUT = 6,  /* a kernel gave up waiting on an internal barrier */
  FA2_ERR_SCALE = 7,    /* scale not finite and > 0 */
  FA2_ERR_MEMORY = 8,   /* a pointer is not device memory, or its buffer is too small */
  FA2_ERR_DEVICE = 9,   /* no usable sm_103 device is current */
  FA2_ERR_SCRATCH = 10, /* split-KV scratch needed exceeds the library's static buffer */
  FA2_ERR_DTYPE = 11    /* unsupported element type combination */
} fa2_status;

/* Element types for fa2_forward_typed. */
typedef enum { FA2_DTYPE_BF16 = 0, FA2_DTYPE_FP16 = 1, FA2_DTYPE_FP32 = 2 } fa2_dtype;

/*
 * FlashAttention-2 forward on the tensor cores (tcgen05 MMAs accumulating in
 * tensor memory, TMA-fed K/V pipeline).
 *   Q, K, V   device bf16 inputs (layouts above)
 *   O, LSE    device fp32 outputs
 *   B, H      batch and head counts (B*H <= 2^31-1)
 *   Nq, Nk    query and key lengths (may differ; Nk >= 1 when B*H*Nq > 0)
 *   d         head dimension, 64, 128 or 256 (256: one 128-row query tile per
 *             CTA and one CTA per SM, the K/V tiles being 64 KB each)
 *   causal    nonzero: mask keys j > i
 *   scale     score scale, finite and > 0 (usually 1/sqrt(d))
 *   stream    CUDA stream (NULL = legacy default stream)
 * B*H*Nq == 0 is a valid empty problem: nothing is launched, FA2_OK.
 */
int fa2_forward(const void *Q, const void *K, const void *V, float *O, float *LSE, int B, int H,
                int Nq, int Nk, int d, int causal, float scale, fa2_stream_t stream);

/*
 * fa2_forward with a choice of element types: Q, K, V are bf16 or fp16
 * (qkv_dtype = FA2_DTYPE_BF16 / FA2_DTYPE_FP16, the same for all three); O is
 * fp32 (o_dtype = FA2_DTYPE_FP32) or the Q/K/V type (o_dtype = qkv_dtype: O
 * in the input dtype, as the "Triton内核实战" wrapper returns it).  LSE is
 * always fp32.  With fp16 inputs P is rounded to fp16 for the P V product.
 * Other combinations return FA2_ERR_DTYPE.  Layouts, sizes, limits and other
 * errors as fa2_forward; a 16-bit O must be 16-byte aligned and hold
 * B*H*Nq*d elements.
 */
int fa2_forward_typed(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                      int H, int Nq, int Nk, int d, int causal, float scale, int qkv_dtype,
                      int o_dtype, fa2_stream_t stream);

/*
 * The same operation on the CUDA cores, fp32 arithmetic, one thread per query
 * row.  A plain second implementation used to cross-check fa2_forward on the
 * device; slow.  Same arguments, limits and errors, plus B*H <= 65535 and
 * d = 64 or 128 (256 returns FA2_ERR_HEADDIM).
 */
int fa2_forward_simt(const void *Q, const void *K, const void *V, float *O, float *LSE, int B,
                     int H, int Nq, int Nk, int d, int causal, float scale, fa2_stream_t stream);

/*
 * Bytes of device workspace fa2_forward_splitkv needs for `num_splits` key
 * ranges: num_splits * B*H*Nq * (d + 1) * 4 bytes, rounded up.  0 for
 * invalid arguments.  Pure host arithmetic (no CUDA call).
 */
size_t fa2_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * Split-KV forward ("Flash Decoding", "Flash Attention 全解析(上)" section 4):
 * the keys are cut into up to `num_splits` ranges of whole 128-key tiles
 * (ceil(tiles / num_splits) tiles each) and every (b, h, Q block, range) is
 * a separate thread block, so short-query / long-key problems fill the GPU.
 * Each range's normalised output and logsumexp go to `workspace`; a second
 * kernel merges them into O and LSE (the merge of fa2_merge).  Same
 * arguments, results (up to rounding) and errors as fa2_forward, plus:
 *   num_splits      1..64 (1, or a problem with a single key tile, runs
 *                   fa2_forward and does not touch the workspace)
 *   workspace       device memory, 256-byte aligned, caller-owned, at least
 *                   fa2_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
 *                   bytes (FA2_ERR_NULL / FA2_ERR_ALIGN / FA2_ERR_MEMORY);
 *                   its contents on return are unspecified
 *   workspace_size  size of that buffer in bytes
 */
int fa2_forward_splitkv(const void *Q, const void *K, const void *V, float *O, float *LSE, int B,
                        int H, int Nq, int Nk, int d, int causal, float scale, int num_splits,
                        void *workspace, size_t workspace_size, fa2_stream_t stream);

/*
 * Split count for fa2_forward_splitkv: the number of key ranges that fills
 * the GPU best when the (b, h, query block) grid alone would leave SMs idle
 * ("Flash Attention 全解析(上)" section 4: Flash Decoding splits the keys
 * when batch x heads x query blocks cannot occupy every SM).  When the
 * grid of 128-row query blocks is smaller than one wave (two such CTAs per
 * SM), it estimates the run time of each count from 1 to
 * min(64, ceil(Nk / 128)) as waves of CTAs times (key tiles per CTA + 4,
 * a CTA's fixed start and end cost), plus 5 tiles for the merge when the
 * keys are split, and returns the smallest count with the least estimate;
 * 1 when the grid already fills the GPU or the problem is empty.
 *   B, H, Nq, Nk  the problem's sizes (negative sizes give 1)
 *   sm_count      SMs of the target GPU; <= 0 queries the current device
 *                 (1 is returned if that query fails)
 * Host arithmetic only apart from that query; launches nothing.
 */
int fa2_splitkv_recommended_splits(int B, int H, int Nq, int Nk, int sm_count);

/*
 * Merge of attention results computed over disjoint key subsets: the
 * ring-attention merge of "FlashAttention 怎么做?online softmax 怎么更新?"
 * (two parts) and the reduction step of Flash Decoding (many parts).  Part p
 * holds, per row r, the normalised output O_parts[p][r][:] and the
 * logsumexp LSE_parts[p][r] (natural log) over its keys; the result is
 *     LSE[r] = log sum_p exp(LSE_parts[p][r])
 *     O[r]   = sum_p exp(LSE_parts[p][r] - LSE[r]) O_parts[p][r]
 * A part with LSE = -inf contributes nothing; if every part has -inf the row
 * gets O = 0 and LSE = -inf.
 *   O_parts    device fp32 [num_parts, rows, d], 16-byte aligned
 *   LSE_parts  device fp32 [num_parts, rows], 4-byte aligned
 *   num_parts  1..64;  rows >= 0 (0: nothing launched);  d: 64, 128 or 256
 *   O, LSE     device fp32 [rows, d] and [rows] outputs (must not overlap the parts)
 */
int fa2_merge(const float *O_parts, const float *LSE_parts, int num_parts, long long rows, int d,
              float *O, float *LSE, fa2_stream_t stream);

/*
 * Split-KV forward that allocates nothing and needs no workspace from the
 * caller.  The pages have no counterpart; it exists for callers that cannot
 * allocate device memory where they call attention -- for example a plugin
 * or custom operator inside a framework that owns all device memory and
 * hands it no allocator, or a server that reserves its memory at start-up
 * and forbids allocation while serving -- and so cannot supply the
 * workspace fa2_forward_splitkv needs.
 *
 * Same arguments, results and errors as fa2_forward_splitkv without the
 * workspace.  The partial results live in one 32 MiB device array inside
 * the library (33554432 bytes, held on every device that loads the library
 * until the process exits); a problem that needs more, i.e. whose
 * fa2_splitkv_workspace_bytes(B, H, Nq, d, num_splits) for the ranges
 * actually used exceeds 32 MiB, is rejected with FA2_ERR_SCRATCH and nothing
 * is launched.  The first call on a device looks up the array's device
 * address (with that device current); make that first call before any
 * stream capture.  If the lookup fails the call returns FA2_ERR_LAUNCH and
 * the next call tries again.  All calls share the array: calls whose kernels may
 * overlap on the GPU (other streams, other host threads) race on it and
 * must be serialised by the caller.  The array keeps the last call's
 * contents; no call depends on them.  The function never calls cudaMalloc,
 * cudaFree or any other allocating routine.
 */
int fa2_forward_splitkv_static(const void *Q, const void *K, const void *V, float *O, float *LSE,
                               int B, int H, int Nq, int Nk, int d, int causal, float scale,
                               int num_splits, fa2_stream_t stream);

/*
 * fa2_forward with the inputs and outputs in host memory.  Q, K and V are
 * copied into caller-owned device buffers, the forward pass runs, and O and
 * LSE are copied back, in `chunks` groups of consecutive (b, h) heads: the
 * copies in of one group, the computation of another and the copies out of
 * a third run at the same time on three streams of the library's own
 * (created by the first call on a device and kept until the process exits,
 * together with their events).  Group c holds about B*H * w_c / sum(w)
 * heads, w_c = min(c + 1, chunks - c), and at least one: the first and last
 * groups are small, so little copying precedes the first computation and
 * little work follows the last copy in.  The result is that of
 * fa2_forward; the heads are independent, so no group needs another's
 * data.
 *   Qh, Kh, Vh       host (or any CUDA-addressable) bf16 inputs, layouts as
 *                    above; page-locked memory lets the copies overlap the
 *                    computation, pageable memory gives the same results
 *   Oh, LSEh         host fp32 outputs, fully overwritten
 *   Qd, Kd, Vd, Od, LSEd  device buffers of the full sizes, caller-owned,
 *                    checked as fa2_forward checks its pointers; on return
 *                    they hold the inputs and outputs
 *   chunks           1..16 groups of heads (more than B*H acts as B*H)
 *   stream           the whole call is asynchronous and ordered on `stream`:
 *                    the copies in start after the work queued on `stream`
 *                    before the call, and work queued on `stream` after it
 *                    starts once every copy out has completed; synchronise
 *                    `stream` before reading Oh and LSEh
 * Errors as fa2_forward, plus FA2_ERR_SHAPE for `chunks` out of range and
 * FA2_ERR_NULL for a null host pointer.  Calls on one device are enqueued
 * one at a time (a lock), but the library's streams are shared: concurrent
 * calls run one after another on the GPU.
 */
int fa2_forward_host(const void *Qh, const void *Kh, const void *Vh, float *Oh, float *LSEh,
                     void *Qd, void *Kd, void *Vd, float *Od, float *LSEd, int B, int H, int Nq,
                     int Nk, int d, int causal, float scale, int chunks, fa2_stream_t stream);

/*
 * Bytes of device workspace fa2_backward needs: 2 * (B*H * ceil(Nq/128)*128 *
 * 4 bytes), each half rounded up to 256 bytes.  0 for negative sizes.
 */
size_t fa2_backward_workspace_bytes(int B, int H, int Nq);

/*
 * Backward pass: the gradients of the attention above with respect to Q, K
 * and V for an upstream gradient dO.  The pages name this pass -- it reuses
 * the forward pass's per-row logsumexp and recomputes the scores block by
 * block ("FlashAttention 怎么做?", FlashAttention-2 question; "Triton内核实战",
 * closing section) -- but print no formulas; it computes the chain rule of
 * the definition:
 *     p_ij  = exp(s_ij - LSE_i)            (j in J_i)
 *     dV_j  = sum_i p_ij dO_i              dp_ij = dO_i . v_j
 *     D_i   = dO_i . O_i                   ds_ij = p_ij (dp_ij - D_i)
 *     dQ_i  = scale sum_j ds_ij k_j        dK_j  = scale sum_i ds_ij q_i
 *   Q, K, V   device bf16 inputs of the forward pass (layouts above)
 *   O, LSE    device fp32 outputs of fa2_forward for these inputs
 *   dO        device bf16 [B, H, Nq, d], the upstream gradient
 *   dQ        device fp32 [B, H, Nq, d]  } outputs, fully overwritten
 *   dK, dV    device fp32 [B, H, Nk, d]  }
 *   workspace device scratch of fa2_backward_workspace_bytes(B, H, Nq) bytes
 *             or more, 256-byte aligned, owned by the caller; its contents
 *             on entry do not matter
 *   B, H, Nq, Nk, d, causal, scale, stream   as in fa2_forward, but d = 64
 *             or 128 (256 returns FA2_ERR_HEADDIM)
 * Q, K, V, O, dO, dQ, dK and dV must be 16-byte aligned, LSE 4-byte aligned.
 * B*H == 0 is a valid empty problem.  Nq == 0 with Nk > 0 writes zeros to dK
 * and dV (no query sees any key); Q, K, V, O, dO, LSE, dQ and workspace may
 * then be NULL.  Nk == 0 with Nq > 0 is FA2_ERR_SHAPE.  Keys that no query
 * sees under the causal mask (j >= Nq) get zero gradients.  Errors as for
 * fa2_forward; the other outputs are undefined after an error found on the
 * device.
 */
int fa2_backward(const void *Q, const void *K, const void *V, const float *O, const void *dO,
                 const float *LSE, float *dQ, float *dK, float *dV, int B, int H, int Nq, int Nk,
                 int d, int causal, float scale, void *workspace, size_t workspace_size,
                 fa2_stream_t stream);

/*
 * fa2_backward with fp16 inputs: Q, K, V and dO are all bf16
 * (qkv_dtype = FA2_DTYPE_BF16, the same as fa2_backward) or all fp16
 * (FA2_DTYPE_FP16); P and dS are then rounded to that type for their MMAs.
 * O, LSE, dQ, dK and dV stay fp32.  Other values return FA2_ERR_DTYPE.
 * Arguments, limits and errors otherwise as fa2_backward.
 */
int fa2_backward_typed(const void *Q, const void *K, const void *V, const float *O, const void *dO,
                       const float *LSE, float *dQ, float *dK, float *dV, int B, int H, int Nq,
                       int Nk, int d, int causal, float scale, int qkv_dtype, void *workspace,
                       size_t workspace_size, fa2_stream_t stream);

/* Static description of a status code (never NULL). */
const char *fa2_status_string(int status);

/*
 * Synchronises `stream`, then reports whether any kernel of this library on
 * the current device has set its device status word since the last reset:
 * FA2_OK, FA2_ERR_TIMEOUT, or FA2_ERR_LAUNCH if the synchronisation itself
 * failed.  reset != 0 clears the word afterwards.
 */
int fa2_device_status(fa2_stream_t stream, int reset);

/*
 * Check of the failure path every pipeline wait has: launches one CTA whose
 * thread waits, with the same bounded wait the kernels use, on an internal
 * barrier that nothing completes.  The wait gives up after timeout_ns of
 * wall time (1e3 <= timeout_ns <= 1e10, else FA2_ERR_SHAPE) and the kernel
 * sets the device status word and returns, so that fa2_device_status then
 * reports FA2_ERR_TIMEOUT and the context stays usable.  Asynchronous on
 * `stream`; returns FA2_OK once launched.
 */
int fa2_check_wait_timeout(unsigned long long timeout_ns, fa2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA2_H */
