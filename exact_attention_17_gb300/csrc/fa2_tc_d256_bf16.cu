// Tensor-core forward kernels: head dimension 256, bf16 inputs (causal and
// non-causal; one query sub-tile per CTA, one CTA per SM).
#include "fa2_launch.h"

namespace fa2host {

namespace {
constexpr uint32_t kSmem = fa2dev::FwdConfig<256, 1>::kSmemBytes;
constexpr int kThreads = fa2dev::FwdShape<1>::kThreads;
}  // namespace

cudaError_t prepare_tc_d256_bf16() {
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<256, false, false, 1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<256, true, false, 1>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_tc_d256_bf16(int subs, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& mo, const fa2dev::FwdParams& p, unsigned grid,
                              cudaStream_t s) {
  if (subs != 1) return cudaErrorInvalidValue;
  if (causal)
    fa2dev::fa2_fwd_tc_kernel<256, true, false, 1><<<grid, kThreads, kSmem, s>>>(mq, mk, mv, mo, p);
  else
    fa2dev::fa2_fwd_tc_kernel<256, false, false, 1><<<grid, kThreads, kSmem, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace fa2host
