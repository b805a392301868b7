// CUDA-core cross-check kernels (head dimensions 64 and 128, causal and not).
#include "fa2_launch.h"

namespace fa2host {

namespace {
template <int D, bool C>
cudaError_t set_limit() {
  return cudaFuncSetAttribute(fa2dev::fa2_fwd_simt_kernel<D, C>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa2dev::simt_smem_bytes<D>());
}
template <int D, bool C>
cudaError_t run(const fa2dev::SimtParams& p, dim3 grid, cudaStream_t s) {
  fa2dev::fa2_fwd_simt_kernel<D, C><<<grid, fa2dev::kSimtRows, fa2dev::simt_smem_bytes<D>(), s>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t prepare_simt() {
  cudaError_t e;
  if ((e = set_limit<64, false>()) != cudaSuccess) return e;
  if ((e = set_limit<64, true>()) != cudaSuccess) return e;
  if ((e = set_limit<128, false>()) != cudaSuccess) return e;
  return set_limit<128, true>();
}

cudaError_t launch_simt(int d, bool causal, const fa2dev::SimtParams& p, dim3 grid, cudaStream_t s) {
  if (d == 64) return causal ? run<64, true>(p, grid, s) : run<64, false>(p, grid, s);
  return causal ? run<128, true>(p, grid, s) : run<128, false>(p, grid, s);
}

}  // namespace fa2host
