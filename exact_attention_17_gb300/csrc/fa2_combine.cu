// Merge of attention results computed over disjoint key subsets.
//
// Part s holds, per row r, the normalised output O_s[r] and the logsumexp
// L_s[r] of the row's scores over the keys of part s.  Over the union of the
// keys, L = log sum_s exp(L_s) and O = sum_s exp(L_s - L) O_s: the merge of
// "FlashAttention 怎么做?online softmax 怎么更新?" (ring attention question,
// two parts) and the global reduction of "Flash Attention 全解析(上)"
// section 4.3 (Flash Decoding, many parts).  A part with L_s = -inf (no
// kept key) contributes nothing.  Computed as m = max_s L_s,
// w_s = exp(L_s - m), L = m + log sum_s w_s, O = sum_s (w_s / sum) O_s.
#include "fa2_launch.h"

namespace fa2dev {

constexpr int kCombineWarps = 8;

// One warp per row; lane t owns D/32 consecutive output columns.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    fa2_combine_kernel(const float* __restrict__ O_part, const float* __restrict__ LSE_part,
                       int S, long long R, float* __restrict__ O, float* __restrict__ LSE) {
  constexpr int V = D / 32;
  const long long r = static_cast<long long>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R) return;

  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, LSE_part[s * R + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < S; s += 32) sum += expf(LSE_part[s * R + r] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  if (sum > 0.f) {
    const float inv = 1.f / sum;
    for (int s = 0; s < S; ++s) {
      const float ls = LSE_part[s * R + r];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - mx) * inv;
      const float* src = O_part + (s * R + r) * D + lane * V;
      if constexpr (V % 4 == 0) {
#pragma unroll
        for (int q = 0; q < V; q += 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + q);
          acc[q] = fmaf(w, x.x, acc[q]); acc[q + 1] = fmaf(w, x.y, acc[q + 1]);
          acc[q + 2] = fmaf(w, x.z, acc[q + 2]); acc[q + 3] = fmaf(w, x.w, acc[q + 3]);
        }
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, x.x, acc[0]); acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  float* dst = O + r * D + lane * V;
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int q = 0; q < V; q += 4)
      *reinterpret_cast<float4*>(dst + q) = make_float4(acc[q], acc[q + 1], acc[q + 2], acc[q + 3]);
  } else
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
  if (lane == 0) LSE[r] = sum > 0.f ? mx + logf(sum) : -INFINITY;
}

}  // namespace fa2dev

namespace fa2host {

cudaError_t launch_combine(int d, const float* O_part, const float* LSE_part, int S, long long R,
                           float* O, float* LSE, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const long long blocks = (R + fa2dev::kCombineWarps - 1) / fa2dev::kCombineWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (d == 64)
    fa2dev::fa2_combine_kernel<64><<<grid, fa2dev::kCombineWarps * 32, 0, s>>>(O_part, LSE_part, S, R, O, LSE);
  else if (d == 128)
    fa2dev::fa2_combine_kernel<128><<<grid, fa2dev::kCombineWarps * 32, 0, s>>>(O_part, LSE_part, S, R, O, LSE);
  else
    fa2dev::fa2_combine_kernel<256><<<grid, fa2dev::kCombineWarps * 32, 0, s>>>(O_part, LSE_part, S, R, O, LSE);
  return cudaGetLastError();
}

}  // namespace fa2host
