// The logit q_i . k_j / h of the LLA kernel weight w_ij = exp(q_i . k_j / h) ("Parallax" blog,
// s.2 Canonical Formulation), evaluated from the shifted key k_j - c as
// (q_i . (k_j - c) + q_i . c) / h. Every CUDA-core stage calls these two functions, with one
// fixed operation order, so the moments and readout passes see bit-identical weights.
#pragma once

namespace lla {

template <int D>
__device__ __forceinline__ float dot_c(const float* __restrict__ x, const float* __restrict__ c) {
  float s = 0.f;
#pragma unroll 16
  for (int a = 0; a < D; ++a) s = fmaf(x[a], c[a], s);
  return s;
}

template <int D>
__device__ __forceinline__ float logit(const float* __restrict__ qrow,
                                       const float* __restrict__ krow_shifted, float qc,
                                       float inv_h) {
  float s = 0.f;
#pragma unroll 16
  for (int a = 0; a < D; ++a) s = fmaf(qrow[a], krow_shifted[a], s);
  return (s + qc) * inv_h;
}

}  // namespace lla
