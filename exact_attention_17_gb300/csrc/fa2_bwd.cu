// Backward-pass kernels: the pre-pass, the zero fill and the tensor-core
// kernel for head dimensions 64 and 128 (bf16 inputs, causal and not).
#include "fa2_launch.h"

namespace fa2dev {

// Zero `n` floats (gradients of keys that no query sees).
__global__ void fa2_zero_kernel(float* __restrict__ p, long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    p[i] = 0.f;
}

}  // namespace fa2dev

namespace fa2host {

namespace {
template <int D>
cudaError_t set_limits_bwd() {
  constexpr uint32_t smem = fa2dev::BwdConfig<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_bwd_tc_kernel<D, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_bwd_tc_kernel<D, true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int D>
void run_bwd(bool causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
             const CUtensorMap& mdo, const CUtensorMap& mdq, const fa2dev::BwdParams& p, unsigned grid,
             cudaStream_t s) {
  constexpr uint32_t smem = fa2dev::BwdConfig<D>::kSmemBytes;
  if (causal)
    fa2dev::fa2_bwd_tc_kernel<D, true, false><<<grid, fa2dev::kBwdThreads, smem, s>>>(mq, mk, mv, mdo, mdq, p);
  else
    fa2dev::fa2_bwd_tc_kernel<D, false, false><<<grid, fa2dev::kBwdThreads, smem, s>>>(mq, mk, mv, mdo, mdq, p);
}
}  // namespace

cudaError_t prepare_bwd() {
  const cudaError_t e = set_limits_bwd<64>();
  return e != cudaSuccess ? e : set_limits_bwd<128>();
}

cudaError_t launch_bwd(int d, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                       const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s) {
  if (d == 64)
    run_bwd<64>(causal, mq, mk, mv, mdo, mdq, p, grid, s);
  else
    run_bwd<128>(causal, mq, mk, mv, mdo, mdq, p, grid, s);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(int d, const float* O, const void* dO, const float* LSE, float* dQ,
                           float* L2, float* Dr, long long rows, int Nq, int Nq_pad, cudaStream_t s) {
  const long long blocks = (rows * 32 + 255) / 256;
  const uint16_t* g = static_cast<const uint16_t*>(dO);
  if (d == 64)
    fa2dev::fa2_bwd_pre_kernel<64, false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad);
  else
    fa2dev::fa2_bwd_pre_kernel<128, false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad);
  return cudaGetLastError();
}

cudaError_t launch_zero(float* p, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fa2dev::fa2_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p, n);
  return cudaGetLastError();
}

}  // namespace fa2host
