// Tensor-core forward kernels: head dimension 128, fp16 inputs (causal and non-causal).
#include "fa2_launch.h"

namespace fa2host {

cudaError_t prepare_tc_d128_f16() {
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<128, false, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fa2dev::FwdConfig<128>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<128, true, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa2dev::FwdConfig<128>::kSmemBytes);
}

cudaError_t launch_tc_d128_f16(bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const fa2dev::FwdParams& p, unsigned grid,
                              cudaStream_t s) {
  constexpr uint32_t smem = fa2dev::FwdConfig<128>::kSmemBytes;
  if (causal)
    fa2dev::fa2_fwd_tc_kernel<128, true, true><<<grid, fa2dev::kThreads, smem, s>>>(mq, mk, mv, p);
  else
    fa2dev::fa2_fwd_tc_kernel<128, false, true><<<grid, fa2dev::kThreads, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace fa2host
