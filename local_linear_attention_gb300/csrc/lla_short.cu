// Exact outputs of early rows with short causal prefixes (the forward, both paths).
//
// With n <= d keys the centred key covariance C_kk has rank below d (and with a few more it is
// nearly singular), and the primal ridge solution y = (C_kk + lambda' I)^-1 (q - kbar) carries a
// component outside the keys' span of size about |q - kbar| / lambda' (lambda' = lambda e^-m, the
// ridge of the max-shifted weights),
// which the readout's k . y - kbar . y must cancel: fp32 cannot once lambda' is small against
// |q - kbar| |k| (a large common key offset seen by an aligned query makes m large), and the fp32
// factorisation of the nearly singular system may fail outright. The same intercept of the
// weighted ridge regression ("Parallax" blog, s.2 Canonical Formulation) in its dual form over
// the n keys (n <= 64 here) never forms that component:
//   o = vbar + Vc^T W^(1/2) (K' + lambda' I)^-1 W^(1/2) Xc (q - kbar),
//   K' = W^(1/2) Xc Xc^T W^(1/2)  (n x n),
// with Xc, Vc the keys and values centred at the weighted means and W = diag(w). The solves list
// such rows (lla_solve.cu says which) and mark them for the readout, which leaves their output
// alone; this pass computes each listed row's output in float64 from the call's own q, k, v, h
// and lambda -- logits, row max, weights and ridge included -- and writes it. It runs on a side
// stream, concurrently with the readout (lla_api.cu forks it after the solve and joins it before
// the call's last step). One CTA per listed row, the CTAs striding over the list; nothing runs
// when it is empty.
//
// K' is singular by construction: the centring makes sum_j w_j Xc_j = 0, so W^(1/2) 1 is a null
// vector, and more than d keys, or keys that are linearly dependent, add more. The right-hand
// side W^(1/2) Xc (q - kbar) lies in the range of K', and the ridge solution -- for lambda' -> 0
// the minimum-norm one -- has no component along any null vector; but the output
// Vc^T W^(1/2) z does depend on such components, and with lambda' below the rounding of |K'| the
// rounding of the right-hand side along them would be divided by lambda'. So the known null
// vector is deflated (tr(K') s s^T added, s = W^(1/2) 1 / |.|, an eigenvector whose right-hand
// side component is zero) and the ridge is floored at kFloor times the largest diagonal entry:
// the remaining null directions then carry rounding / floor, and a direction of the keys whose
// variance is a fraction f of the largest is biased by about kFloor / f. kFloor = 1e-12 balances
// the two (float64 rounding of K' is ~n eps ~ 1e-14 of its largest entry; n = d random keys leave
// f ~ 1e-5): against the oracle, 1e-10 gave 2.5e-3 on such a prefix, 1e-14 7e-3 from rounding,
// 1e-12 at most 9e-5 over offset, i.i.d., repeated-key and n > d prefixes. A non-finite K' or
// right-hand side (non-finite inputs) gives NaN and LLA_ERR_NUMERICAL.
#include <cuda_bf16.h>

#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int NT = 256;
constexpr int NMAX = kShortMaxKeys;  // keys of a listed row's prefix, at most
constexpr int LD = 65;               // row stride (doubles) of the centred keys, values and K'
constexpr int kGrid = 152;
constexpr double kFloor = 1e-12;     // ridge floor, relative to the largest diagonal entry of K'

// xc, vc, kk [NMAX][LD]; sw, z, lg, dinv [NMAX]; g, kb, vb [64]; red [NT / 32]
constexpr size_t kSmem = sizeof(double) * (3 * NMAX * LD + 4 * NMAX + 3 * 64 + NT / 32);

__device__ __forceinline__ double in64(const float* p, long long i) { return (double)p[i]; }
__device__ __forceinline__ double in64(const __nv_bfloat16* p, long long i) {
  return (double)__bfloat162float(p[i]);
}
__device__ __forceinline__ void out_store(float* p, long long i, double x) { p[i] = (float)x; }
__device__ __forceinline__ void out_store(__nv_bfloat16* p, long long i, double x) {
  p[i] = __float2bfloat16_rn((float)x);
}

__device__ __forceinline__ double block_sum(double x, double* red) {
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  double t = 0.0;
  for (int k = 0; k < NT / 32; ++k) t += red[k];
  return t;
}

__device__ __forceinline__ double block_max(double x, double* red) {
  for (int o = 16; o > 0; o >>= 1) x = fmax(x, __shfl_xor_sync(0xffffffffu, x, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  double t = red[0];
  for (int k = 1; k < NT / 32; ++k) t = fmax(t, red[k]);
  return t;
}

template <typename TIn, int D>
__global__ void __launch_bounds__(NT)
short_prefix_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                    const TIn* __restrict__ v, const int* __restrict__ list,
                    const int* __restrict__ count, int T, double inv_h, double log_lam, int dv,
                    TIn* __restrict__ out, int* __restrict__ status) {
  static_assert(D <= 64 && NT == 4 * NMAX, "four threads per key in the logits");
  extern __shared__ double sm[];
  double* xc = sm;               // [NMAX][LD] centred keys (D used)
  double* vc = xc + NMAX * LD;   // [NMAX][LD] centred values (dv used)
  double* kk = vc + NMAX * LD;   // [NMAX][LD] K' + lambda' I, then its Cholesky factor
  double* sw = kk + NMAX * LD;   // [NMAX] square roots of the weights
  double* z = sw + NMAX;         // [NMAX] right-hand side, then the solution
  double* lg = z + NMAX;         // [NMAX] logits
  double* dinv = lg + NMAX;      // [NMAX] reciprocal pivots (0 where skipped)
  double* g = dinv + NMAX;       // [64] q - kbar
  double* kb = g + 64;           // [64] kbar
  double* vb = kb + 64;          // [64] vbar
  double* red = vb + 64;         // [NT / 32] reduction scratch
  const int tid = threadIdx.x, lane = tid & 31;
  const int nrows = *count;
  for (int e = blockIdx.x; e < nrows; e += gridDim.x) {
    const int row = list[e];
    const int bh = row / T, pos = row - bh * T, n = pos + 1;  // n <= NMAX (the solves' rule)
    const long long base = (long long)bh * T;
    // logits q . k_j / h (four threads per key), their max m, the weights exp(s - m), the ridge
    {
      const int j = tid >> 2, part = tid & 3;
      double s = 0.0;
      if (j < n)
        for (int a = part * (D / 4); a < (part + 1) * (D / 4); ++a)
          s += in64(q, (long long)row * D + a) * in64(k, (base + j) * D + a);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (j < n && part == 0) lg[j] = s * inv_h;
    }
    __syncthreads();
    const double m = block_max(tid < n ? lg[tid] : -INFINITY, red);
    const double wj = tid < n ? exp(lg[tid] - m) : 0.0;
    if (tid < NMAX) sw[tid] = sqrt(wj);
    const double om = block_sum(wj, red);
    const double lp = exp(log_lam - m);
    // weighted means of the keys (threads 0 .. D-1) and of the values (threads 64 .. 64+dv-1)
    if (tid < D) {
      double sk = 0.0;
      for (int j = 0; j < n; ++j) sk += sw[j] * sw[j] * in64(k, (base + j) * D + tid);
      kb[tid] = sk / om;
      g[tid] = in64(q, (long long)row * D + tid) - kb[tid];
    } else if (tid >= 64 && tid < 64 + dv) {
      const int c = tid - 64;
      double sv = 0.0;
      for (int j = 0; j < n; ++j) sv += sw[j] * sw[j] * in64(v, (base + j) * dv + c);
      vb[c] = sv / om;
    }
    __syncthreads();
    for (int t = tid; t < n * D; t += NT) {
      const int j = t / D, a = t % D;
      xc[j * LD + a] = in64(k, (base + j) * D + a) - kb[a];
    }
    for (int t = tid; t < n * dv; t += NT) {
      const int j = t / dv, c = t % dv;
      vc[j * LD + c] = in64(v, (base + j) * dv + c) - vb[c];
    }
    __syncthreads();
    // K' + lambda' I (lower triangle) and the right-hand side W^(1/2) Xc (q - kbar)
    for (int t = tid; t < n * n; t += NT) {
      const int j = t / n, l = t % n;
      if (l > j) continue;
      double s = 0.0;
      for (int a = 0; a < D; ++a) s += xc[j * LD + a] * xc[l * LD + a];
      kk[j * LD + l] = sw[j] * sw[l] * s + (j == l ? lp : 0.0);
    }
    if (tid < n) {
      double s = 0.0;
      for (int a = 0; a < D; ++a) s += xc[tid * LD + a] * g[a];
      z[tid] = sw[tid] * s;
    }
    __syncthreads();
    // deflate the null vector W^(1/2) 1 of K' (its squared norm is omega)
    const double tr = block_sum(tid < n ? kk[tid * LD + tid] - lp : 0.0, red);
    const double defl = tr / om;
    for (int t = tid; t < n * n; t += NT) {
      const int j = t / n, l = t % n;
      if (l <= j) kk[j * LD + l] += defl * sw[j] * sw[l];
    }
    __syncthreads();
    // the ridge floor, then Cholesky (lower, in place), the whole CTA on each trailing update
    const double fin = block_sum(tid < n ? kk[tid * LD + tid] + fabs(z[tid]) : 0.0, red);
    const bool ok = isfinite(fin) && isfinite(om);
    const double dmax = block_max(tid < n ? kk[tid * LD + tid] : 0.0, red);
    const double lift = fmax(kFloor * dmax - lp, 0.0);
    if (tid < n) kk[tid * LD + tid] += lift;
    __syncthreads();
    const int nf = ok ? n : 0;
    for (int c = 0; c < nf; ++c) {
      const double piv = kk[c * LD + c];
      // a pivot lost to rounding (not expected above the floor): a zero coordinate in both solves
      const bool skip = !(piv > 0.0);
      const double lcc = skip ? 0.0 : sqrt(piv);
      const double inv = skip ? 0.0 : 1.0 / lcc;
      __syncthreads();  // every thread has read the pivot
      for (int r = c + 1 + tid; r < n; r += NT) kk[r * LD + c] *= inv;
      if (tid == 0) {
        kk[c * LD + c] = lcc;
        dinv[c] = inv;
      }
      __syncthreads();
      const int w = n - c - 1;
      for (int t = tid; t < w * w; t += NT) {
        const int rr = t / w, cc = t % w;
        if (cc <= rr)
          kk[(c + 1 + rr) * LD + c + 1 + cc] -= kk[(c + 1 + rr) * LD + c] * kk[(c + 1 + cc) * LD + c];
      }
      __syncthreads();
    }
    if (!ok && tid == 0) atomicOr(status, kStatusNumerical);
    // L u = rhs, then L^T z = u: one warp, lane l holding rows l and l + 32
    if (tid < 32) {
      double z0 = lane < nf ? z[lane] : 0.0, z1 = lane + 32 < nf ? z[lane + 32] : 0.0;
      for (int c = 0; c < nf; ++c) {
        const double zc = __shfl_sync(0xffffffffu, c < 32 ? z0 : z1, c & 31) * dinv[c];
        if (lane == (c & 31)) (c < 32 ? z0 : z1) = zc;
        if (lane > c && lane < nf) z0 -= kk[lane * LD + c] * zc;
        if (lane + 32 > c && lane + 32 < nf) z1 -= kk[(lane + 32) * LD + c] * zc;
      }
      for (int c = nf - 1; c >= 0; --c) {
        const double zc = __shfl_sync(0xffffffffu, c < 32 ? z0 : z1, c & 31) * dinv[c];
        if (lane == (c & 31)) (c < 32 ? z0 : z1) = zc;
        if (lane < c) z0 -= kk[c * LD + lane] * zc;
        if (lane + 32 < c) z1 -= kk[c * LD + lane + 32] * zc;
      }
      __syncwarp();
      if (lane < n) z[lane] = z0;
      if (lane + 32 < n) z[lane + 32] = z1;
    }
    __syncthreads();
    if (tid < dv) {
      double o = vb[tid];
      for (int j = 0; j < n; ++j) o += sw[j] * z[j] * vc[j * LD + tid];
      if (!ok) o = __longlong_as_double(0x7FF8000000000000ll);  // NaN: non-finite input
      out_store(out, (long long)row * dv + tid, o);
    }
    __syncthreads();
  }
}

template <typename TIn, int D>
cudaError_t launch_t(const Args& a, const Workspace& ws, cudaStream_t s) {
  auto kern = short_prefix_kernel<TIn, D>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (err != cudaSuccess) return err;
  kern<<<kGrid, NT, kSmem, s>>>(static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k),
                                static_cast<const TIn*>(a.v), ws.short_rows, ws.short_count, a.T,
                                1.0 / (double)a.h, log((double)a.lam), a.dv,
                                static_cast<TIn*>(a.out), ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_short_prefix(const Args& a, const Workspace& ws, cudaStream_t s) {
  const bool f32 = a.dtype == LLA_F32;
  switch (a.d) {
    case 16: return f32 ? launch_t<float, 16>(a, ws, s) : launch_t<__nv_bfloat16, 16>(a, ws, s);
    case 32: return f32 ? launch_t<float, 32>(a, ws, s) : launch_t<__nv_bfloat16, 32>(a, ws, s);
    case 64: return f32 ? launch_t<float, 64>(a, ws, s) : launch_t<__nv_bfloat16, 64>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lla
