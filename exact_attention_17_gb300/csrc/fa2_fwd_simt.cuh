// FlashAttention-2 forward on the CUDA cores (fp32 throughout).
//
// A second, deliberately plain GPU implementation of the same operation,
// used to cross-check the tensor-core path on the device; it is not tuned.
// One thread owns one query row; K/V blocks of 32 keys are staged in shared
// memory as fp32.  Per block it follows the online-softmax update of
// "FlashAttention 怎么做?online softmax 怎么更新?" (推导/关键公式) with the
// FlashAttention-2 lazy normalisation (divide by l once at the end) and the
// per-row logsumexp of the same page.  P stays in fp32 (no bf16 rounding).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa2dev {

struct SimtParams {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  float* O;
  float* LSE;
  int Nq;
  int Nk;
  float scale_log2;
};

constexpr int kSimtRows = 64;
constexpr int kSimtKeys = 32;

template <int D>
constexpr uint32_t simt_smem_bytes() {
  return (kSimtRows * (D + 1) + 2 * kSimtKeys * D) * 4;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kSimtRows) fa2_fwd_simt_kernel(const SimtParams p) {
  extern __shared__ float fsm[];
  float* sq = fsm;                                 // [rows][D+1]
  float* sk = fsm + kSimtRows * (D + 1);           // [keys][D]
  float* sv = sk + kSimtKeys * D;                  // [keys][D]
  const int bh = blockIdx.y;
  const int row0 = blockIdx.x * kSimtRows;
  const int t = threadIdx.x;
  const int qi = row0 + t;
  const size_t qbase = static_cast<size_t>(bh) * p.Nq * D;
  const size_t kbase = static_cast<size_t>(bh) * p.Nk * D;

  for (int x = t; x < kSimtRows * D; x += kSimtRows) {
    const int r = x / D, c = x - r * D;
    sq[r * (D + 1) + c] = row0 + r < p.Nq ? __bfloat162float(p.Q[qbase + static_cast<size_t>(row0 + r) * D + c]) : 0.f;
  }

  float o[D];
#pragma unroll
  for (int c = 0; c < D; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  // keys this CTA needs: all, or up to its last row under the causal mask
  const int kend = CAUSAL ? min(p.Nk, min(row0 + kSimtRows, p.Nq)) : p.Nk;
  const int lim = CAUSAL ? min(p.Nk, qi + 1) : p.Nk;

  for (int k0 = 0; k0 < kend; k0 += kSimtKeys) {
    __syncthreads();
    for (int x = t; x < kSimtKeys * D; x += kSimtRows) {
      const int r = x / D, c = x - r * D;
      const bool in = k0 + r < p.Nk;
      sk[x] = in ? __bfloat162float(p.K[kbase + static_cast<size_t>(k0 + r) * D + c]) : 0.f;
      sv[x] = in ? __bfloat162float(p.V[kbase + static_cast<size_t>(k0 + r) * D + c]) : 0.f;
    }
    __syncthreads();
    float s[kSimtKeys];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSimtKeys; ++j) {
      float acc = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) acc = fmaf(sq[t * (D + 1) + c], sk[j * D + c], acc);
      s[j] = k0 + j < lim ? acc * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[j]);
    }
    const float m_new = fmaxf(m, mx);
    const float off = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = m == -INFINITY ? 0.f : exp2f(m - m_new);
    float rs = 0.f;
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] *= alpha;
#pragma unroll
    for (int j = 0; j < kSimtKeys; ++j) {
      const float pj = exp2f(s[j] - off);
      rs += pj;
#pragma unroll
      for (int c = 0; c < D; ++c) o[c] = fmaf(pj, sv[j * D + c], o[c]);
    }
    l = l * alpha + rs;
    m = m_new;
  }
  if (qi < p.Nq) {
    const float inv = 1.f / l;
    float* orow = p.O + qbase + static_cast<size_t>(qi) * D;
#pragma unroll
    for (int c = 0; c < D; c += 4)
      *reinterpret_cast<float4*>(orow + c) = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
    p.LSE[static_cast<size_t>(bh) * p.Nq + qi] = (m + log2f(l)) * 0.69314718055994531f;
  }
}

}  // namespace fa2dev
