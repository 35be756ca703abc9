// Debug entry: raw max-shifted kernel-weighted moments of selected queries.
//
// For query i of head bh: m = max_{j<=i} q_i.k_j/h, w_j = exp(q_i.k_j/h - m), and the sums
// omega = sum w, sk = sum w k, sv = sum w v, Skk = sum w k k^T, Svk = sum w v k^T over the causal
// prefix -- the quantities from which the pages' omega_i, mu_i and Sigma_i ("Parallax" blog s.2
// Canonical Formulation) follow by centring at q_i. One CTA per selected query, fp64
// accumulation; a checking tool, not a fast path.
#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int kDbgThreads = 256;
constexpr int kDbgChunk = 64;
constexpr int kMaxEntriesPerThread = (1 + 64 + 64 + 64 * 64 + 64 * 64 + kDbgThreads - 1) / kDbgThreads;

template <typename TIn>
__global__ void __launch_bounds__(kDbgThreads)
debug_moments_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                     const int64_t* __restrict__ idx, long long total, int T, int D, int DV,
                     double inv_h, float* m_o, float* om_o, float* sk_o, float* sv_o,
                     float* skk_o, float* svk_o, int* status) {
  __shared__ double qd[64];
  __shared__ double wj[kDbgChunk];
  __shared__ double red[kDbgThreads];
  __shared__ float kc[kDbgChunk][64];
  __shared__ float vc[kDbgChunk][64];
  const int n = blockIdx.x, tid = threadIdx.x;
  const long long r = idx[n];
  if (r < 0 || r >= total) {
    if (tid == 0) atomicOr(status, kStatusBadIndex);
    return;
  }
  const long long bh = r / T;
  const int i = (int)(r % T);
  const long long base = bh * T;
  for (int a = tid; a < D; a += kDbgThreads) qd[a] = (double)ldf(q, r * D + a);
  __syncthreads();

  double mx = -INFINITY;
  for (int j = tid; j <= i; j += kDbgThreads) {
    double s = 0.0;
    for (int a = 0; a < D; ++a) s += qd[a] * (double)ldf(k, (base + j) * D + a);
    mx = fmax(mx, s * inv_h);
  }
  red[tid] = mx;
  __syncthreads();
  for (int st = kDbgThreads / 2; st > 0; st >>= 1) {
    if (tid < st) red[tid] = fmax(red[tid], red[tid + st]);
    __syncthreads();
  }
  const double m = red[0];

  // entry e: 0 omega | 1..D sk | D+1..D+DV sv | then Skk (D*D) | then Svk (DV*D)
  const int nent = 1 + D + DV + D * D + DV * D;
  double acc[kMaxEntriesPerThread];
  for (int t = 0; t < kMaxEntriesPerThread; ++t) acc[t] = 0.0;

  for (int j0 = 0; j0 <= i; j0 += kDbgChunk) {
    const int jn = min(kDbgChunk, i + 1 - j0);
    __syncthreads();
    for (int e = tid; e < jn * D; e += kDbgThreads) kc[e / D][e % D] = ldf(k, (base + j0 + e / D) * D + e % D);
    for (int e = tid; e < jn * DV; e += kDbgThreads) vc[e / DV][e % DV] = ldf(v, (base + j0 + e / DV) * DV + e % DV);
    __syncthreads();
    for (int j = tid; j < jn; j += kDbgThreads) {
      double s = 0.0;
      for (int a = 0; a < D; ++a) s += qd[a] * (double)kc[j][a];
      wj[j] = exp(s * inv_h - m);
    }
    __syncthreads();
    for (int t = 0; t < kMaxEntriesPerThread; ++t) {
      const int e = tid + t * kDbgThreads;
      if (e >= nent) break;
      double s = 0.0;
      for (int j = 0; j < jn; ++j) {
        double f;
        if (e == 0) f = 1.0;
        else if (e <= D) f = kc[j][e - 1];
        else if (e <= D + DV) f = vc[j][e - 1 - D];
        else if (e < 1 + D + DV + D * D) { const int x = e - 1 - D - DV; f = (double)kc[j][x / D] * kc[j][x % D]; }
        else { const int x = e - 1 - D - DV - D * D; f = (double)vc[j][x / D] * kc[j][x % D]; }
        s += wj[j] * f;
      }
      acc[t] += s;
    }
  }
  for (int t = 0; t < kMaxEntriesPerThread; ++t) {
    const int e = tid + t * kDbgThreads;
    if (e >= nent) break;
    const float val = (float)acc[t];
    if (e == 0) { if (om_o) om_o[n] = val; }
    else if (e <= D) { if (sk_o) sk_o[(long long)n * D + e - 1] = val; }
    else if (e <= D + DV) { if (sv_o) sv_o[(long long)n * DV + e - 1 - D] = val; }
    else if (e < 1 + D + DV + D * D) { if (skk_o) skk_o[(long long)n * D * D + e - 1 - D - DV] = val; }
    else { if (svk_o) svk_o[(long long)n * DV * D + e - 1 - D - DV - D * D] = val; }
  }
  if (tid == 0 && m_o) m_o[n] = (float)m;
}

}  // namespace

cudaError_t launch_debug_moments(const Args& a, const int64_t* idx, int n, float* m, float* omega,
                                 float* sk, float* sv, float* Skk, float* Svk, int* status,
                                 cudaStream_t s) {
  const double inv_h = 1.0 / (double)a.h;
  if (a.dtype == LLA_F32)
    debug_moments_kernel<float><<<n, kDbgThreads, 0, s>>>(
        static_cast<const float*>(a.q), static_cast<const float*>(a.k),
        static_cast<const float*>(a.v), idx, a.rows(), a.T, a.d, a.dv, inv_h, m, omega, sk, sv,
        Skk, Svk, status);
  else
    debug_moments_kernel<__nv_bfloat16><<<n, kDbgThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), idx, a.rows(), a.T, a.d, a.dv, inv_h, m, omega,
        sk, sv, Skk, Svk, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
