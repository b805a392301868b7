// Two-SM (CTA pair) forward kernels, head dimension 128: bf16 and fp16
// inputs, causal and non-causal.  Launched as clusters of two CTAs.
#include "fa2_launch.h"

namespace fa2host {

namespace {
template <bool CAUSAL, bool F16>
cudaError_t set_limit() {
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_pair_kernel<CAUSAL, F16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fa2dev::PairConfig::kSmemBytes);
}

template <bool CAUSAL, bool F16>
cudaError_t run(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                const fa2dev::FwdParams& p, unsigned grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(fa2dev::PairConfig::kThreads, 1, 1);
  cfg.dynamicSmemBytes = fa2dev::PairConfig::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa2dev::fa2_fwd_pair_kernel<CAUSAL, F16>, mq, mk, mv, mo, p);
}
}  // namespace

cudaError_t prepare_tc_pair_d128() {
  cudaError_t e = set_limit<false, false>();
  if (e == cudaSuccess) e = set_limit<true, false>();
  if (e == cudaSuccess) e = set_limit<false, true>();
  if (e == cudaSuccess) e = set_limit<true, true>();
  return e;
}

cudaError_t launch_tc_pair_d128(bool causal, bool f16, const CUtensorMap& mq, const CUtensorMap& mk_half,
                                const CUtensorMap& mv, const CUtensorMap& mo, const fa2dev::FwdParams& p,
                                unsigned grid, cudaStream_t s) {
  if (grid % 2 != 0) return cudaErrorInvalidValue;
  if (f16)
    return causal ? run<true, true>(mq, mk_half, mv, mo, p, grid, s) : run<false, true>(mq, mk_half, mv, mo, p, grid, s);
  return causal ? run<true, false>(mq, mk_half, mv, mo, p, grid, s) : run<false, false>(mq, mk_half, mv, mo, p, grid, s);
}

}  // namespace fa2host
