// Two-tile backward kernel, head dimension 128 (bf16 or fp16 inputs, causal
// and not).
#include "fa2_launch.h"

namespace fa2host {

namespace {
template <bool CAUSAL, bool F16>
cudaError_t set_limit_bwd2() {
  return cudaFuncSetAttribute(fa2dev::fa2_bwd2_tc_kernel<CAUSAL, F16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fa2dev::Bwd2Config::kSmemBytes);
}

template <bool CAUSAL, bool F16>
void run_bwd2(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
              const CUtensorMap& mdq, const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s) {
  fa2dev::fa2_bwd2_tc_kernel<CAUSAL, F16>
      <<<grid, fa2dev::kBwdThreads, fa2dev::Bwd2Config::kSmemBytes, s>>>(mq, mk, mv, mdo, mdq, p);
}
}  // namespace

cudaError_t prepare_bwd2() {
  cudaError_t e = set_limit_bwd2<false, false>();
  if (e == cudaSuccess) e = set_limit_bwd2<true, false>();
  if (e == cudaSuccess) e = set_limit_bwd2<false, true>();
  if (e == cudaSuccess) e = set_limit_bwd2<true, true>();
  return e;
}

cudaError_t launch_bwd2(bool causal, bool f16, const CUtensorMap& mq64, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdo64, const CUtensorMap& mdq32,
                        const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s) {
  if (f16)
    causal ? run_bwd2<true, true>(mq64, mk, mv, mdo64, mdq32, p, grid, s)
           : run_bwd2<false, true>(mq64, mk, mv, mdo64, mdq32, p, grid, s);
  else
    causal ? run_bwd2<true, false>(mq64, mk, mv, mdo64, mdq32, p, grid, s)
           : run_bwd2<false, false>(mq64, mk, mv, mdo64, mdq32, p, grid, s);
  return cudaGetLastError();
}

}  // namespace fa2host
