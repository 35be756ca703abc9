// Per-query ridge solve of the causal LLA forward, plus the per-head key reference point.
//
// From the augmented Gram moments of one query (omega, s = sum p (k - c), S = sum p (k-c)(k-c)^T)
// the solve forms the centred key moment C_kk = S - s s^T / omega, adds the ridge
// lambda' = lambda * exp(-m_i) (the moments are scaled by exp(-m_i), so the absolute ridge of the
// pages' objective scales with them), factors C_kk + lambda' I = L L^T (Cholesky) and returns
//   y = (C_kk + lambda' I)^-1 (q_i - kbar_i),   kbar_i = c + s / omega,
// together with kbar_i - c. With these the output is
//   o_i = vbar_i + C_vk y   ("Parallax" blog s.2 Canonical Formulation, centred closed form),
// which the readout stage evaluates in one more pass over the prefix.
// One warp solves one query; the d x d factor lives in that warp's shared memory.
#include <cfloat>
#include <type_traits>

#include "lla_internal.cuh"

namespace lla {
namespace {

// ----------------------------------------------------------------------------- means
// Per-head reference points: c = mean of the head's finite keys (blockIdx.y == 0) and
// c_v = mean of its finite values (blockIdx.y == 1). Any fixed c and c_v leave the result
// unchanged in exact arithmetic (shifting keys does not change their centred moments; shifting
// values shifts the intercept by the same amount); central ones keep the fp32 sums small. A
// non-finite element is skipped so that it cannot poison the rows that never see it.
template <typename TIn>
__global__ void __launch_bounds__(256)
mean_kernel(const TIn* __restrict__ k, const TIn* __restrict__ v, int T, int D, int DV,
            float* __restrict__ kmean, float* __restrict__ vmean, int zero_keys) {
  extern __shared__ float red[];  // [256]
  const bool val = blockIdx.y == 1;
  const int W = val ? DV : D;
  const long long bh = blockIdx.x;
  const TIn* x = (val ? v : k) + bh * T * W;
  float* mean = (val ? vmean : kmean) + bh * W;
  const int tid = threadIdx.x;
  const int rows_per = 256 / W;  // W divides 256
  const int a = tid % W, r0 = tid / W;
  float s = 0.f;
  for (int j = r0; j < T; j += rows_per) {
    const float e = ldf(x, (long long)j * W + a);
    if (isfinite(e)) s += e;
  }
  red[tid] = s;
  __syncthreads();
  if (tid < W) {
    float t = 0.f;
    for (int r = 0; r < rows_per; ++r) t += red[r * W + tid];
    mean[tid] = (zero_keys && !val) ? 0.f : t / (float)T;
  }
}

// ----------------------------------------------------------------------------- solve
constexpr int kWarpsPerBlock = 4;

template <int D>
struct SolveCfg {
  static constexpr int LS = D + 1;                  // row stride of the factor (conflict-free)
  static constexpr int WARP_FLOATS = D * LS + 2 * D; // factor + right-hand side + shift vector
};

template <int D, bool PRECISE>
__device__ __forceinline__ int gidx(int a, int b) {  // a <= b
  return gram_block_index(D, a >> 2, b >> 2) * 16 + (a & 3) * 4 + (b & 3);
}

// Moment layouts: FMT 0 = augmented-Gram 4x4 blocks (CUDA-core stage, gram_floats(D) per row);
// FMT 1 = tensor-core stage ([sk (D) | upper triangle of S row by row], TC_ROW floats per row,
// omega in its own array).
constexpr int TC_ROW = 2208;

template <int D, int FMT>
__device__ __forceinline__ int moff(int a, int b) {  // a <= b; b == D means the constant 1
  if (FMT == 0) return gram_block_index(D, a >> 2, b >> 2) * 16 + (a & 3) * 4 + (b & 3);
  if (b == D) return a;
  return D + a * D - a * (a - 1) / 2 + (b - a);
}

template <typename TIn, int D, bool PRECISE, int FMT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
solve_kernel(const TIn* __restrict__ q, const float* __restrict__ kmean,
             const float* __restrict__ mom, const float* __restrict__ mom_lo,
             const float* __restrict__ omega, const float* __restrict__ mrow, int T,
             long long rows, float lam, float* __restrict__ y_out, float* __restrict__ kbar_out,
             int* __restrict__ status) {
  using C = SolveCfg<D>;
  constexpr int G = FMT == 0 ? gram_floats(D) : TC_ROW;
  constexpr int LS = C::LS;
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* Lw = smem + warp * C::WARP_FLOATS;  // [D][LS]
  float* rv = Lw + D * LS;                   // [D]
  float* kb = rv + D;                        // [D] kbar - c
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= rows) return;  // whole warp leaves together
  const long long bh = row / T;
  const float* g = mom + row * G;
  const float* gl = PRECISE ? mom_lo + row * G : nullptr;

  // omega, kbar - c and the right-hand side q - kbar = (q - c) - (kbar - c). The centring runs
  // in double for fp32 inputs (the compensated moments carry more than fp32 precision) and in
  // float otherwise.
  using R = typename std::conditional<PRECISE, double, float>::type;
  R om = FMT == 0 ? g[gidx<D, PRECISE>(D, D)] : omega[row];
  if (PRECISE && FMT == 0) om += gl[gidx<D, PRECISE>(D, D)];
  const R inv_om = R(1) / om;
  for (int a = lane; a < D; a += 32) {
    const int ix = moff<D, FMT>(a, D);
    R s = g[ix];
    if (PRECISE) s += gl[ix];
    const R kbar = s * inv_om;
    kb[a] = (float)kbar;
    const R qa = (R)ldf(q, row * D + a) - (R)kmean[bh * D + a];
    rv[a] = (float)(qa - kbar);
  }
  // ridge scaled by exp(-m), kept inside the normal fp32 range
  double lp = (double)lam * exp(-(double)mrow[row]);
  lp = fmin(fmax(lp, (double)FLT_MIN), (double)FLT_MAX);
  __syncwarp();

  // C_kk + lambda' I, lower triangle, C[i][j] = S[j][i] - s_i s_j / omega.
  for (int e = lane; e < D * D; e += 32) {
    const int i = e / D, j = e % D;
    if (j > i) continue;
    const int ix = moff<D, FMT>(j, i);
    R sij = g[ix];
    if (PRECISE) sij += gl[ix];
    const int si = moff<D, FMT>(i, D), sj = moff<D, FMT>(j, D);
    R s_i = g[si], s_j = g[sj];
    if (PRECISE) { s_i += gl[si]; s_j += gl[sj]; }
    R c = sij - s_i * (s_j * inv_om);
    if (i == j) c += (R)lp;
    Lw[i * LS + j] = (float)c;
  }
  __syncwarp();

  // Cholesky, right-looking, column by column.
  bool ok = true;
  for (int kk = 0; kk < D; ++kk) {
    const float dkk = Lw[kk * LS + kk];
    if (!(dkk > 0.f)) { ok = false; break; }  // uniform across the warp
    const float lkk = sqrtf(dkk);
    const float inv = 1.f / lkk;
    __syncwarp();
    for (int i = kk + 1 + lane; i < D; i += 32) Lw[i * LS + kk] *= inv;
    if (lane == 0) Lw[kk * LS + kk] = lkk;
    __syncwarp();
    for (int i = kk + 1 + lane; i < D; i += 32) {
      const float lik = Lw[i * LS + kk];
      for (int j = kk + 1; j <= i; ++j) Lw[i * LS + j] = fmaf(-lik, Lw[j * LS + kk], Lw[i * LS + j]);
    }
    __syncwarp();
  }
  if (!ok) {
    if (lane == 0) atomicOr(status, kStatusNumerical);
    for (int a = lane; a < D; a += 32) {
      y_out[row * D + a] = __int_as_float(0x7fc00000);
      kbar_out[row * D + a] = __int_as_float(0x7fc00000);
    }
    return;
  }
  // L z = r
  for (int j = 0; j < D; ++j) {
    const float zj = rv[j] / Lw[j * LS + j];
    __syncwarp();
    for (int i = j + 1 + lane; i < D; i += 32) rv[i] = fmaf(-Lw[i * LS + j], zj, rv[i]);
    if (lane == 0) rv[j] = zj;
    __syncwarp();
  }
  // L^T y = z
  for (int j = D - 1; j >= 0; --j) {
    const float yj = rv[j] / Lw[j * LS + j];
    __syncwarp();
    for (int i = lane; i < j; i += 32) rv[i] = fmaf(-Lw[j * LS + i], yj, rv[i]);
    if (lane == 0) rv[j] = yj;
    __syncwarp();
  }
  for (int a = lane; a < D; a += 32) {
    y_out[row * D + a] = rv[a];
    kbar_out[row * D + a] = kb[a];
  }
}

template <typename TIn, int D, bool PRECISE, int FMT = 0>
cudaError_t launch_solve_t(const Args& a, const Workspace& ws, cudaStream_t s) {
  const size_t smem = sizeof(float) * kWarpsPerBlock * SolveCfg<D>::WARP_FLOATS;
  auto kern = solve_kernel<TIn, D, PRECISE, FMT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long rows = a.rows();
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  kern<<<(unsigned)blocks, kWarpsPerBlock * 32, smem, s>>>(
      static_cast<const TIn*>(a.q), ws.kmean, ws.mom, ws.mom_lo, ws.omega, ws.m, a.T, rows, a.lam,
      ws.y, ws.kbar, ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const Args& a, const Workspace& ws, cudaStream_t s) {
  const dim3 grid((unsigned)a.BH(), 2);
  if (a.dtype == LLA_F32)
    mean_kernel<float><<<grid, 256, 256 * sizeof(float), s>>>(
        static_cast<const float*>(a.k), static_cast<const float*>(a.v), a.T, a.d, a.dv, ws.kmean,
        ws.vmean, ws.path == kPathTensorCore);
  else
    mean_kernel<__nv_bfloat16><<<grid, 256, 256 * sizeof(float), s>>>(
        static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.v), a.T, a.d,
        a.dv, ws.kmean, ws.vmean, ws.path == kPathTensorCore);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_solve(const Args& a, const Workspace& ws, cudaStream_t s) {
  if (ws.path == kPathTensorCore) return launch_solve_t<__nv_bfloat16, 64, false, 1>(a, ws, s);
  const bool f32 = a.dtype == LLA_F32;
  switch (a.d) {
    case 16: return f32 ? launch_solve_t<float, 16, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 16, false>(a, ws, s);
    case 32: return f32 ? launch_solve_t<float, 32, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 32, false>(a, ws, s);
    case 64: return f32 ? launch_solve_t<float, 64, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 64, false>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lla
