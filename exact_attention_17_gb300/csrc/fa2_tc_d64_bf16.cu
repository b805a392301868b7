// Tensor-core forward kernels: head dimension 64, bf16 inputs (causal and
// non-causal; one or two query sub-tiles per CTA).
#include "fa2_launch.h"

namespace fa2host {

namespace {
template <int SUBS>
cudaError_t set_limits() {
  constexpr uint32_t smem = fa2dev::FwdConfig<64, SUBS>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<64, false, false, SUBS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_tc_kernel<64, true, false, SUBS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int SUBS>
cudaError_t run(bool causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const CUtensorMap& mo, const fa2dev::FwdParams& p, unsigned grid, cudaStream_t s) {
  constexpr uint32_t smem = fa2dev::FwdConfig<64, SUBS>::kSmemBytes;
  constexpr int threads = fa2dev::FwdShape<SUBS>::kThreads;
  if (causal)
    fa2dev::fa2_fwd_tc_kernel<64, true, false, SUBS><<<grid, threads, smem, s>>>(mq, mk, mv, mo, p);
  else
    fa2dev::fa2_fwd_tc_kernel<64, false, false, SUBS><<<grid, threads, smem, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t prepare_tc_d64_bf16() {
  const cudaError_t e = set_limits<1>();
  return e != cudaSuccess ? e : set_limits<2>();
}

cudaError_t launch_tc_d64_bf16(int subs, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& mo, const fa2dev::FwdParams& p, unsigned grid,
                              cudaStream_t s) {
  return subs == 1 ? run<1>(causal, mq, mk, mv, mo, p, grid, s) : run<2>(causal, mq, mk, mv, mo, p, grid, s);
}

}  // namespace fa2host
