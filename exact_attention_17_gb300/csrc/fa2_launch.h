// Internal: launch entry points of the kernel translation units.  Each .cu
// file instantiates one family of kernels so that they compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa2_bwd2_sm103.cuh"
#include "fa2_bwd_sm103.cuh"
#include "fa2_fwd_simt.cuh"
#include "fa2_fwd_pair_sm103.cuh"
#include "fa2_fwd_sm103.cuh"

namespace fa2host {

// Raise the dynamic shared-memory limit of every kernel in the unit (current device).
cudaError_t prepare_tc_d64_bf16();
cudaError_t prepare_tc_d128_bf16();
cudaError_t prepare_tc_d64_f16();
cudaError_t prepare_tc_d128_f16();
cudaError_t prepare_tc_d256_bf16();
cudaError_t prepare_tc_d256_f16();
cudaError_t prepare_simt();

// subs: query sub-tiles of 128 rows per CTA (1 or 2; head dimension 256: 1).  mo: the map the epilogue stores O (or
// the split-KV partial O) through.
#define FA2_DECLARE_TC_LAUNCH(name)                                                          \
  cudaError_t name(int subs, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,      \
                   const CUtensorMap& mv, const CUtensorMap& mo, const fa2dev::FwdParams& p, \
                   unsigned grid, cudaStream_t s);
FA2_DECLARE_TC_LAUNCH(launch_tc_d64_bf16)
FA2_DECLARE_TC_LAUNCH(launch_tc_d128_bf16)
FA2_DECLARE_TC_LAUNCH(launch_tc_d64_f16)
FA2_DECLARE_TC_LAUNCH(launch_tc_d128_f16)
FA2_DECLARE_TC_LAUNCH(launch_tc_d256_bf16)
FA2_DECLARE_TC_LAUNCH(launch_tc_d256_f16)
#undef FA2_DECLARE_TC_LAUNCH
cudaError_t launch_simt(int d, bool causal, const fa2dev::SimtParams& p, dim3 grid, cudaStream_t s);

// Two-SM forward (clusters of two CTAs), head dimension 128.  mk_half: K with
// 64-row boxes; mq, mv: 128-row boxes.  grid: an even number of CTAs.
cudaError_t prepare_tc_pair_d128();
cudaError_t launch_tc_pair_d128(bool causal, bool f16, const CUtensorMap& mq, const CUtensorMap& mk_half,
                                const CUtensorMap& mv, const CUtensorMap& mo, const fa2dev::FwdParams& p,
                                unsigned grid, cudaStream_t s);

// Merge of S partial results (normalised O [S, R, d], LSE [S, R]) into O [R, d], LSE [R].
cudaError_t launch_combine(int d, const float* O_part, const float* LSE_part, int S, long long R,
                           float* O, float* LSE, cudaStream_t s);

// Backward pass (fa2_bwd.cu).
cudaError_t prepare_bwd();
// mdq: fp32 [BH][Nq][d] map of dQ, 32-column boxes, 128-byte swizzle (TMA reductions).
// f16: Q, K, V and dO are fp16 (else bf16).
cudaError_t launch_bwd(int d, bool causal, bool f16, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                       const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s);
// D_i = dO_i . O_i and LSE_i log2(e) into [BH][Nq_pad] arrays; dQ rows zeroed.
cudaError_t launch_bwd_pre(int d, bool f16, const float* O, const void* dO, const float* LSE, float* dQ,
                           float* L2, float* Dr, long long rows, int Nq, int Nq_pad, cudaStream_t s);
cudaError_t launch_zero(float* p, long long n, cudaStream_t s);

// Two-tile backward kernel (fa2_bwd2.cu), head dimension 128.  mq64, mdo64:
// 64-row boxes; mk, mv: 128-row boxes; mdq32: fp32 dQ with 32 x 32 boxes.
cudaError_t prepare_bwd2();
cudaError_t launch_bwd2(bool causal, bool f16, const CUtensorMap& mq64, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdo64, const CUtensorMap& mdq32,
                        const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s);

}  // namespace fa2host
