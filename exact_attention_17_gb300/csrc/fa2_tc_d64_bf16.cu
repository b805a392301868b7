// Tensor-core forward kernels: head dimension 64, bf16 inputs (causal and non-causal).
#include "fa2_launch.h"

namespace fa2host {

cudaError_t prepare_tc_d64_bf16() {
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<64, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fa2dev::FwdConfig<64>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<64, true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa2dev::FwdConfig<64>::kSmemBytes);
}

cudaError_t launch_tc_d64_bf16(bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const fa2dev::FwdParams& p, unsigned grid,
                              cudaStream_t s) {
  constexpr uint32_t smem = fa2dev::FwdConfig<64>::kSmemBytes;
  if (causal)
    fa2dev::fa2_fwd_tc_kernel<64, true, false><<<grid, fa2dev::kThreads, smem, s>>>(mq, mk, mv, p);
  else
    fa2dev::fa2_fwd_tc_kernel<64, false, false><<<grid, fa2dev::kThreads, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace fa2host
