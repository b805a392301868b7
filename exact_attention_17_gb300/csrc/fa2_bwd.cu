// Backward-pass kernels: the pre-pass, the zero fill and the tensor-core
// kernel for head dimensions 64 and 128 (bf16 or fp16 inputs, causal and not).
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
template <int D, bool F16>
cudaError_t set_limits_bwd() {
  constexpr uint32_t smem = fa2dev::BwdConfig<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fa2dev::fa2_bwd_tc_kernel<D, false, F16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa2dev::fa2_bwd_tc_kernel<D, true, F16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int D, bool F16>
void run_bwd(bool causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
             const CUtensorMap& mdo, const CUtensorMap& mdq, const fa2dev::BwdParams& p, unsigned grid,
             cudaStream_t s) {
  constexpr uint32_t smem = fa2dev::BwdConfig<D>::kSmemBytes;
  if (causal)
    fa2dev::fa2_bwd_tc_kernel<D, true, F16><<<grid, fa2dev::kBwdThreads, smem, s>>>(mq, mk, mv, mdo, mdq, p);
  else
    fa2dev::fa2_bwd_tc_kernel<D, false, F16><<<grid, fa2dev::kBwdThreads, smem, s>>>(mq, mk, mv, mdo, mdq, p);
}

template <int D, bool F16>
void run_bwd_pre(const float* O, const uint16_t* g, const float* LSE, float* dQ, float* L2, float* Dr,
                 long long rows, int Nq, int Nq_pad, cudaStream_t s) {
  const long long blocks = (rows * 32 + 255) / 256;
  fa2dev::fa2_bwd_pre_kernel<D, F16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(O, g, LSE, dQ, L2, Dr, rows,
                                                                                 Nq, Nq_pad);
}
}  // namespace

cudaError_t prepare_bwd() {
  cudaError_t e = set_limits_bwd<64, false>();
  if (e == cudaSuccess) e = set_limits_bwd<128, false>();
  if (e == cudaSuccess) e = set_limits_bwd<64, true>();
  if (e == cudaSuccess) e = set_limits_bwd<128, true>();
  return e;
}

cudaError_t launch_bwd(int d, bool causal, bool f16, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                       const fa2dev::BwdParams& p, unsigned grid, cudaStream_t s) {
  if (d == 64)
    f16 ? run_bwd<64, true>(causal, mq, mk, mv, mdo, mdq, p, grid, s)
        : run_bwd<64, false>(causal, mq, mk, mv, mdo, mdq, p, grid, s);
  else
    f16 ? run_bwd<128, true>(causal, mq, mk, mv, mdo, mdq, p, grid, s)
        : run_bwd<128, false>(causal, mq, mk, mv, mdo, mdq, p, grid, s);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(int d, bool f16, const float* O, const void* dO, const float* LSE, float* dQ,
                           float* L2, float* Dr, long long rows, int Nq, int Nq_pad, cudaStream_t s) {
  const uint16_t* g = static_cast<const uint16_t*>(dO);
  if (d == 64)
    f16 ? run_bwd_pre<64, true>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad, s)
        : run_bwd_pre<64, false>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad, s);
  else
    f16 ? run_bwd_pre<128, true>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad, s)
        : run_bwd_pre<128, false>(O, g, LSE, dQ, L2, Dr, rows, Nq, Nq_pad, s);
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
