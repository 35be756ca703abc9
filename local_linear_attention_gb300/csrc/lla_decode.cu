// Decode: one query per head against a key/value cache of L positions, for LLA and for Parallax.
//
// The query attends to every cached position (it is the newest token; its own key and value are
// already appended), so the definitions are those of the prefill forward for its last row:
//  * LLA ("Parallax" blog, s.2 Canonical Formulation): the intercept of the weighted ridge fit,
//    o = vbar + C_vk (C_kk + lambda I)^-1 (q - kbar), w_j = exp(q . k_j / h);
//  * Parallax (s.2 "Parallax", Appendix B with eta = 0): o = vbar - Sigma_KV r, computed as the
//    blog's streaming combination (1 + d2/d1) O1/d1 - O2/d1 (Appendix C), with O1 = sum p_j v_j,
//    O2 = sum p_j (r . k_j) v_j, d1 = sum p_j, d2 = sum p_j (r . k_j).
//
// With one query per head, the per-head work is a reduction over the cache; decode batches have
// few heads and long caches, so the cache of each head is split over S CTAs ("split-KV", as the
// blog's decode kernel does, Appendix C): each CTA reduces its chunk of keys to partial sums
// shifted by the chunk's own maximum logit, writes them to a workspace, and the last CTA of the
// head to finish (an atomic arrival counter after a memory fence) merges them, rescaling each by
// exp((m_s - M) / h) with M the largest chunk shift, in a fixed order (so the result does not
// depend on which CTA arrives last), and writes the output. For LLA the merged moments are
// centred and the d x d ridge system is solved by Cholesky, in double precision (one small system
// per head).
//
// CUDA-core kernels (Parallax, and LLA for every shape but bf16 d = dv = 64): each CTA streams its
// chunk through a ring of raw key/value tiles in shared memory (cp.async, two tiles ahead of the
// one being reduced) with a running maximum, four threads per key form the logits, one thread per
// key the weight, and the LLA second moments accumulate in 4 x 4 register tiles (two shared loads
// per 16 FMAs). For bf16 d = dv = 64 the LLA second moments of a chunk are two tensor-core
// contractions over its keys (lla_decode_tc_kernel, below).
#include <cfloat>
#include <cstdint>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

using tc::cp_async16;
using tc::cp_async_commit;
using tc::cp_async_wait;

constexpr int NT = 256;   // threads per CTA
constexpr int TK = 64;    // keys per shared-memory tile

template <typename TIn>
__device__ __forceinline__ float ld(const TIn* p, long long i) { return ldf(p, i); }

// Arrival of one CTA of head bh after its partial sums are written; true for the last one, which
// then sees every CTA's partials.
__device__ __forceinline__ bool last_arrival(int* counter, int S, int* flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *flag = atomicAdd(counter, 1) == S - 1;
  __syncthreads();
  if (*flag) __threadfence();
  return *flag;
}

__global__ void zero_counters(int* c, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) c[i] = 0;
}

// The running maximum of one tile: threads 0..TK-1 hold the logits of the tile's keys (-inf
// past its end); returns max(m_run, tile max) to every thread (two block barriers inside).
__device__ __forceinline__ float tile_max(float sj, float m_run, float* red) {
  float x = threadIdx.x < TK ? sj : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  if ((threadIdx.x & 31) == 0 && threadIdx.x < TK) red[threadIdx.x >> 5] = x;
  __syncthreads();
  float r = m_run;
  for (int i = 0; i < TK / 32; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float tof(float x) { return x; }
__device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }

// Two adjacent elements as fp32 (one 4- or 8-byte shared load).
__device__ __forceinline__ void load_pair(const float* p, float (&x)[2]) {
  const float2 u = *reinterpret_cast<const float2*>(p);
  x[0] = u.x; x[1] = u.y;
}
__device__ __forceinline__ void load_pair(const __nv_bfloat16* p, float (&x)[2]) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  x[0] = __uint_as_float(w << 16); x[1] = __uint_as_float(w & 0xFFFF0000u);
}

// n contiguous elements at p (16-byte aligned when n * sizeof(TIn) is a multiple of 16, else
// 8-byte aligned) as fp32, with 16- or 8-byte shared loads.
template <typename TIn, int N>
__device__ __forceinline__ void load_row(const TIn* p, float (&x)[N]) {
  constexpr int BYTES = N * (int)sizeof(TIn);
  if constexpr (BYTES % 16 == 0) {
#pragma unroll
    for (int c = 0; c < BYTES / 16; ++c) {
      const uint4 u = reinterpret_cast<const uint4*>(p)[c];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(TIn) == 2) {
          x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
          x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
          x[4 * c + i] = __uint_as_float(w[i]);
        }
      }
    }
  } else {
    static_assert(BYTES == 8, "row segment of 8 bytes");
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    if constexpr (sizeof(TIn) == 2) {
      x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
      x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
      x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    }
  }
}

// Logits q . k_j and r . k_j of a tile kept in the input type (the Parallax decode's cp.async
// ring) into sS / sT (-inf past n): four threads per key, each with a contiguous quarter of the
// row, completed by two shuffles within the four.
template <typename TIn, int D, bool PROBE>
__device__ __forceinline__ void tile_logits_raw(const TIn* kt, const float* qs, const float* rs,
                                                int n, float* sS, float* sT) {
  static_assert(TK * 4 == NT, "four threads per key");
  constexpr int SEG = D / 4;
  const int key = threadIdx.x >> 2, part = threadIdx.x & 3;
  float a = 0.f, b = 0.f;
  if (key < n) {
    float kv[SEG];
    load_row<TIn, SEG>(kt + key * D + part * SEG, kv);
#pragma unroll
    for (int u = 0; u < SEG; ++u) {
      a = fmaf(qs[part * SEG + u], kv[u], a);
      if (PROBE) b = fmaf(rs[part * SEG + u], kv[u], b);
    }
  }
  a += __shfl_xor_sync(0xffffffffu, a, 1);
  a += __shfl_xor_sync(0xffffffffu, a, 2);
  if (PROBE) {
    b += __shfl_xor_sync(0xffffffffu, b, 1);
    b += __shfl_xor_sync(0xffffffffu, b, 2);
  }
  if (part == 0) {
    sS[key] = key < n ? a : -INFINITY;
    if (PROBE) sT[key] = b;
  }
}

// exp((m_old - m_new) / h): the factor that moves sums shifted by m_old to the shift m_new.
__device__ __forceinline__ float rescale(float m_old, float m_new, float inv_h) {
  return m_old == -INFINITY ? 0.f : __expf((m_old - m_new) * inv_h);
}

// ------------------------------------------------------------------------------------ Parallax
// Partial of a chunk: [m, d1, d2, O1[DV], O2[DV]].
template <int D, int DV>
constexpr int px_part() { return 3 + 2 * DV; }

// The Parallax decode streams its chunk through a ring of PX_ST raw (input-type) K/V tiles
// filled with cp.async, PX_ST - 1 tiles ahead of the one being reduced: the reduction per key is
// small, so the kernel is bound by how many cache bytes each SM keeps in flight.
constexpr int PX_ST = 3;
template <typename TIn, int D, int DV>
constexpr size_t px_smem() { return (size_t)PX_ST * TK * (D + DV) * sizeof(TIn); }

// Tile `it` of the chunk [j0, j1) of a head's cache (kb: [L, D], vb: [L, DV]) into slot
// it % PX_ST of the raw rings (16-byte cp.async copies; rows past the chunk are zero-filled
// without being read). One commit group per call, empty past the last tile, so that a thread's
// cp.async.wait_group<PX_ST - 1> after prefetching tile it + PX_ST - 1 covers tile it.
template <typename TIn, int D, int DV>
__device__ __forceinline__ void prefetch_tile(TIn* kring, TIn* vring, const TIn* kb,
                                              const TIn* vb, int j0, int j1, int it, int ntl) {
  if (it < ntl) {
    const int t0 = j0 + it * TK, n = min(TK, j1 - t0), slot = it % PX_ST;
    constexpr int KR = D * (int)sizeof(TIn) / 16, VR = DV * (int)sizeof(TIn) / 16;
    const char* ks = reinterpret_cast<const char*>(kb + (long long)t0 * D);
    const char* vs = reinterpret_cast<const char*>(vb + (long long)t0 * DV);
    char* kd = reinterpret_cast<char*>(kring + slot * TK * D);
    char* vd = reinterpret_cast<char*>(vring + slot * TK * DV);
    for (int e = threadIdx.x; e < TK * KR; e += NT) {
      const bool in = e / KR < n;
      cp_async16(kd + 16 * e, ks + (in ? 16 * e : 0), in ? 16u : 0u);
    }
    for (int e = threadIdx.x; e < TK * VR; e += NT) {
      const bool in = e / VR < n;
      cp_async16(vd + 16 * e, vs + (in ? 16 * e : 0), in ? 16u : 0u);
    }
  }
  cp_async_commit();
}

template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NT)
parallax_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                       const TIn* __restrict__ v, const TIn* __restrict__ r, int L, int S,
                       float inv_h, float* __restrict__ part, int* __restrict__ counter,
                       TIn* __restrict__ out) {
  // Accumulation: thread t takes value columns 2 cp, 2 cp + 1 (cp = t % (DV/2)) of both branches
  // for the keys of group t / (DV/2) (NG groups, keys jj = group + NG i).
  constexpr int NG = NT / (DV / 2);
  __shared__ float qs[D], rs[D], red[NT / 32];
  extern __shared__ __align__(16) uint8_t px_ring[];
  TIn* kring = reinterpret_cast<TIn*>(px_ring);  // [PX_ST][TK * D]
  TIn* vring = kring + PX_ST * TK * D;           // [PX_ST][TK * DV]
  __shared__ float pt[TK], tt[TK], sS[TK], sT[TK];
  __shared__ float og_s[NG][2 * DV], dsum[2][2], tot[2 * DV + 2];
  __shared__ double alpha[512];
  __shared__ int is_last;
  const long long bh = blockIdx.x / S;
  const int s = blockIdx.x % S, tid = threadIdx.x;
  const int chunk = (L + S - 1) / S;
  const int j0 = s * chunk, j1 = min(L, j0 + chunk);
  for (int a = tid; a < D; a += NT) {
    qs[a] = ld(q, bh * D + a);
    rs[a] = ld(r, bh * D + a);
  }
  const TIn* kb = k + bh * (long long)L * D;
  const TIn* vb = v + bh * (long long)L * DV;
  // One pass with a running maximum m: every sum is kept shifted by the current m and rescaled
  // when a tile raises it.
  float m = -INFINITY, d1 = 0.f, d2 = 0.f;
  float o1a = 0.f, o1b = 0.f, o2a = 0.f, o2b = 0.f;
  const int cp = tid % (DV / 2), og = tid / (DV / 2);
  const int ntl = j1 > j0 ? (j1 - j0 + TK - 1) / TK : 0;
  for (int it = 0; it < PX_ST - 1; ++it) prefetch_tile<TIn, D, DV>(kring, vring, kb, vb, j0, j1, it, ntl);
  for (int it = 0; it < ntl; ++it) {
    const int t0 = j0 + it * TK, n = min(TK, j1 - t0), slot = it % PX_ST;
    prefetch_tile<TIn, D, DV>(kring, vring, kb, vb, j0, j1, it + PX_ST - 1, ntl);
    cp_async_wait<PX_ST - 1>();  // this thread's copies of tile `it` have landed
    __syncthreads();             // ... and everyone else's
    const TIn* kt = kring + slot * TK * D;
    const TIn* vt = vring + slot * TK * DV;
    tile_logits_raw<TIn, D, true>(kt, qs, rs, n, sS, sT);
    __syncthreads();
    const float sj = tid < TK ? sS[tid] : -INFINITY, tj = tid < TK ? sT[tid] : 0.f;
    const float mn = tile_max(sj, m, red);
    const float sc = rescale(m, mn, inv_h);
    m = mn;
    o1a *= sc; o1b *= sc; o2a *= sc; o2b *= sc;
    d1 *= sc;
    d2 *= sc;
    if (tid < TK) {
      const float p = tid < n ? __expf((sj - m) * inv_h) : 0.f;
      pt[tid] = p;
      tt[tid] = p * tj;
      d1 += p;
      d2 += p * tj;
    }
    __syncthreads();
    for (int jj = og; jj < n; jj += NG) {
      float vv[2];
      load_pair(vt + jj * DV + 2 * cp, vv);
      const float p = pt[jj], pr = tt[jj];
      o1a = fmaf(p, vv[0], o1a); o1b = fmaf(p, vv[1], o1b);
      o2a = fmaf(pr, vv[0], o2a); o2b = fmaf(pr, vv[1], o2b);
    }
    __syncthreads();  // slot `it` is refilled by the prefetch PX_ST - 1 iterations on
    (void)t0;
  }
  cp_async_wait<0>();
  // Reductions in a fixed order (no atomics), so that the result is reproducible.
  og_s[og][2 * cp] = o1a;
  og_s[og][2 * cp + 1] = o1b;
  og_s[og][DV + 2 * cp] = o2a;
  og_s[og][DV + 2 * cp + 1] = o2b;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
  }
  static_assert(TK == 64, "d1 and d2 are summed over the two warps of key threads");
  if ((tid & 31) == 0 && tid < TK) { dsum[tid >> 5][0] = d1; dsum[tid >> 5][1] = d2; }
  __syncthreads();
  float* pp = part + blockIdx.x * (long long)px_part<D, DV>();
  if (tid == 0) { pp[0] = m; pp[1] = dsum[0][0] + dsum[1][0]; pp[2] = dsum[0][1] + dsum[1][1]; }
  for (int c = tid; c < 2 * DV; c += NT) {
    float t = 0.f;
    for (int g = 0; g < NG; ++g) t += og_s[g][c];
    pp[3 + c] = t;
  }
  if (!last_arrival(counter + bh, S, &is_last)) return;
  // merge (the last CTA of the head): every partial moved to the largest chunk maximum M
  const float* hp = part + bh * S * (long long)px_part<D, DV>();
  float M = -INFINITY;
  for (int t = 0; t < S; ++t) M = fmaxf(M, __ldcg(hp + t * px_part<D, DV>()));
  for (int t = tid; t < S; t += NT) {
    const float mt = __ldcg(hp + t * px_part<D, DV>());
    alpha[t] = mt == -INFINITY ? 0.0 : exp((double)(mt - M) * inv_h);
  }
  __syncthreads();
  for (int c = tid; c < 2 * DV + 2; c += NT) {
    double acc = 0.0;
    for (int t = 0; t < S; ++t)
      acc += alpha[t] * (double)__ldcg(hp + t * px_part<D, DV>() + 1 + c);
    tot[c] = (float)acc;
  }
  __syncthreads();
  const float D1 = tot[0], D2 = tot[1];
  for (int c = tid; c < DV; c += NT)
    stf(out, bh * DV + c, (1.f + D2 / D1) * tot[2 + c] / D1 - tot[2 + DV + c] / D1);
}

// ------------------------------------------------------------------------------------ LLA
// Partial of a chunk: [m, omega, sk[D], sv[DV], Skk[D][D] (upper 4 x 4 blocks), Svk[DV][D]].
template <int D, int DV>
constexpr int lla_part() { return 2 + D + DV + D * D + DV * D; }

// The last CTA of head bh to arrive: merges the S partials of the head in a fixed order
// (log-sum-exp weights computed once per split), centres the moments, solves the d x d ridge
// system by Cholesky and writes o = vbar + C_vk y, all in double precision. qs: the query (fp32,
// shared memory); dsm: dynamic shared memory of at least sizeof(double) * (P + D + S) bytes.
template <typename TIn, int D, int DV>
__device__ void lla_merge_solve(const float* qs, const float* __restrict__ part, long long bh,
                                int S, float inv_h, float lam, float* dsm, int* fail_flag,
                                TIn* __restrict__ out, int* __restrict__ status) {
  constexpr int P = lla_part<D, DV>();
  const int tid = threadIdx.x, nt = blockDim.x;
  int& fail_s = *fail_flag;

  // ---- merge (fp32: the partials are fp32 sums, the weights <= 1), then centre and solve in
  // double precision
  double* mom = reinterpret_cast<double*>(dsm);  // [P - 1]: omega, sk, sv, Skk, Svk (merged)
  double* z = mom + P;                           // [D]: q - kbar, then y
  float* alpha = reinterpret_cast<float*>(z + D);  // [S]
  const float* hp = part + bh * S * (long long)P;
  float M = -INFINITY;
  for (int t = 0; t < S; ++t) M = fmaxf(M, __ldcg(hp + t * (long long)P));
  for (int t = tid; t < S; t += nt) {
    const float mt = __ldcg(hp + t * (long long)P);
    alpha[t] = mt == -INFINITY ? 0.f : expf((mt - M) * inv_h);
  }
  __syncthreads();
  constexpr int SKK0 = 1 + D + DV;  // offset of Skk in mom (mom[e] is partial entry 1 + e)
  for (int e = tid; e < P - 1; e += nt) {
    const bool lower = e >= SKK0 && e < SKK0 + D * D && (e - SKK0) / D > (e - SKK0) % D;
    float acc = 0.f;
    if (!lower) {
      // eight independent loads in flight per step, summed in split order
      int t = 0;
      for (; t + 8 <= S; t += 8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __ldcg(hp + (t + u) * (long long)P + 1 + e);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc = fmaf(alpha[t + u], x[u], acc);
      }
      for (; t < S; ++t) acc = fmaf(alpha[t], __ldcg(hp + t * (long long)P + 1 + e), acc);
    }
    mom[e] = (double)acc;
  }
  __syncthreads();
  const double omega = mom[0];
  const double* msk = mom + 1;
  const double* msv = msk + D;
  double* A = mom + SKK0;                // Skk (upper) -> C_kk + lambda' I -> its Cholesky factor
  const double* Svk = A + D * D;
  const double lp = (double)lam * exp(-(double)M * inv_h);  // ridge scaled by exp(-M/h)
  for (int e = tid; e < D * D; e += nt) {
    const int a = e / D, b = e % D;
    if (a <= b) {
      const double c = A[e] - msk[a] * msk[b] / omega + (a == b ? lp : 0.0);
      A[e] = c;
      A[b * D + a] = c;
    }
  }
  for (int a = tid; a < D; a += nt) z[a] = (double)qs[a] - msk[a] / omega;
  if (tid == 0) fail_s = 0;
  __syncthreads();
  // Cholesky A = L L^T (lower triangle in place), column by column
  for (int c = 0; c < D; ++c) {
    if (tid == 0) {
      const double piv = A[c * D + c];
      if (!(piv > 0.0)) fail_s = 1;
      A[c * D + c] = sqrt(piv > 0.0 ? piv : 1.0);
    }
    __syncthreads();
    for (int i = c + 1 + tid; i < D; i += nt) A[i * D + c] /= A[c * D + c];
    __syncthreads();
    for (int e = tid; e < D * D; e += nt) {
      const int i = e / D, j = e % D;
      if (j > c && i >= j) A[i * D + j] -= A[i * D + c] * A[j * D + c];
    }
    __syncthreads();
  }
  // L w = z, then L^T y = w, by warp 0 (dot products across its lanes)
  if (tid < 32) {
    for (int i = 0; i < D; ++i) {
      double t = 0.0;
      for (int j = tid; j < i; j += 32) t += A[i * D + j] * z[j];
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (tid == 0) z[i] = (z[i] - t) / A[i * D + i];
      __syncwarp();
    }
    for (int i = D - 1; i >= 0; --i) {
      double t = 0.0;
      for (int j = i + 1 + tid; j < D; j += 32) t += A[j * D + i] * z[j];
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (tid == 0) z[i] = (z[i] - t) / A[i * D + i];
      __syncwarp();
    }
  }
  __syncthreads();
  // o = vbar + C_vk y,  C_vk = Svk - sv sk^T / omega
  const bool bad = fail_s != 0;
  for (int c = tid; c < DV; c += nt) {
    double o = msv[c] / omega;
    for (int b = 0; b < D; ++b) o += (Svk[c * D + b] - msv[c] * msk[b] / omega) * z[b];
    stf(out, bh * DV + c, bad ? __int_as_float(0x7fc00000) : (float)o);
  }
  if (tid == 0 && (bad || !(omega > 0.0))) atomicOr(status, kStatusNumerical);
}

template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NT)
lla_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                  int L, int S, float inv_h, float lam, float* __restrict__ part,
                  int* __restrict__ counter, TIn* __restrict__ out, int* __restrict__ status) {
  constexpr int P = lla_part<D, DV>();
  constexpr int NBK = (D / 4) * (D / 4 + 1) / 2;   // upper-triangle 4 x 4 blocks of Skk
  constexpr int NB = NBK + (DV / 4) * (D / 4);      // then the blocks of Svk
  constexpr int TPB = (NB + NT - 1) / NT;           // blocks per thread
  extern __shared__ __align__(16) float dsm[];
  __shared__ float qs[D], red[NT / 32], sS[TK];
  __shared__ int is_last, fail_s;
  float* kt = dsm;               // [TK][D]
  float* pk = kt + TK * D;       // [TK][D]: p_j k_j
  float* pv = pk + TK * D;       // [TK][DV]: p_j v_j
  float* pw = pv + TK * DV;      // [TK]: p_j
  TIn* kring = reinterpret_cast<TIn*>(pw + TK);  // [PX_ST][TK * D] raw key tiles
  TIn* vring = kring + PX_ST * TK * D;           // [PX_ST][TK * DV] raw value tiles
  const long long bh = blockIdx.x / S;
  const int s = blockIdx.x % S, tid = threadIdx.x;
  const int chunk = (L + S - 1) / S;
  const int j0 = s * chunk, j1 = min(L, j0 + chunk);
  for (int a = tid; a < D; a += NT) qs[a] = ld(q, bh * D + a);
  const TIn* kb = k + bh * (long long)L * D;
  const TIn* vb = v + bh * (long long)L * DV;
  // This thread's blocks: row block ar and column block cr (Skk: ar <= cr; Svk: rows of V).
  int ar[TPB], cr[TPB];
#pragma unroll
  for (int u = 0; u < TPB; ++u) {
    int b = tid + u * NT;
    ar[u] = -1;
    cr[u] = 0;
    if (b < NBK) {
      int row = 0;
      while (b >= D / 4 - row) { b -= D / 4 - row; ++row; }
      ar[u] = row;
      cr[u] = row + b;
    } else if (b < NB) {
      b -= NBK;
      ar[u] = D / 4 + b / (D / 4);  // >= D/4 marks a Svk block (its V row block is ar - D/4)
      cr[u] = b % (D / 4);
    }
  }
  float2 acc[TPB][8];  // 4 rows x 2 column pairs per block
#pragma unroll
  for (int u = 0; u < TPB; ++u)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[u][e] = make_float2(0.f, 0.f);
  float m = -INFINITY, sk = 0.f, sv = 0.f, om = 0.f;  // thread a < D: sk[a]; then sv, omega
  // The chunk streams through the raw rings (cp.async, PX_ST - 1 tiles ahead), as in the
  // Parallax decode; each tile is converted to fp32 (k, p k, p v) once its weights are known.
  const int ntl = j1 > j0 ? (j1 - j0 + TK - 1) / TK : 0;
  for (int it = 0; it < PX_ST - 1; ++it) prefetch_tile<TIn, D, DV>(kring, vring, kb, vb, j0, j1, it, ntl);
  for (int it = 0; it < ntl; ++it) {
    const int t0 = j0 + it * TK, n = min(TK, j1 - t0), slot = it % PX_ST;
    prefetch_tile<TIn, D, DV>(kring, vring, kb, vb, j0, j1, it + PX_ST - 1, ntl);
    cp_async_wait<PX_ST - 1>();
    __syncthreads();  // tile `it` has landed; the previous tile's products are all read
    const TIn* kr = kring + slot * TK * D;
    const TIn* vr = vring + slot * TK * DV;
    tile_logits_raw<TIn, D, false>(kr, qs, nullptr, n, sS, nullptr);
    __syncthreads();
    const float sj = tid < TK ? sS[tid] : -INFINITY;
    const float mn = tile_max(sj, m, red);
    const float sc = rescale(m, mn, inv_h);
    m = mn;
    sk *= sc;
    sv *= sc;
    om *= sc;
    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
    for (int u = 0; u < TPB; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[u][e] = __fmul2_rn(acc[u][e], sc2);
    if (tid < TK) pw[tid] = tid < n ? __expf((sj - m) * inv_h) : 0.f;
    __syncthreads();
    for (int e = tid; e < TK * D; e += NT) {
      const float kv = tof(kr[e]);
      kt[e] = kv;
      pk[e] = pw[e / D] * kv;
    }
    for (int e = tid; e < TK * DV; e += NT) pv[e] = pw[e / DV] * tof(vr[e]);
    __syncthreads();
    if (tid < D) for (int jj = 0; jj < n; ++jj) sk += pk[jj * D + tid];
    else if (tid < D + DV) for (int jj = 0; jj < n; ++jj) sv += pv[jj * DV + tid - D];
    else if (tid == D + DV) for (int jj = 0; jj < n; ++jj) om += pw[jj];
#pragma unroll
    for (int u = 0; u < TPB; ++u) {
      if (ar[u] >= 0) {
        const bool kk = ar[u] < D / 4;
        const float* x = kk ? pk + ar[u] * 4 : pv + (ar[u] - D / 4) * 4;
        const int xs = kk ? D : DV;
        const float* kc = kt + cr[u] * 4;
        for (int jj = 0; jj < n; ++jj) {
          const float4 xa = *reinterpret_cast<const float4*>(x + jj * xs);
          const float4 kv4 = *reinterpret_cast<const float4*>(kc + jj * D);
          const float2 k01 = make_float2(kv4.x, kv4.y), k23 = make_float2(kv4.z, kv4.w);
          const float xr[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 xi = make_float2(xr[i], xr[i]);
            acc[u][2 * i] = __ffma2_rn(xi, k01, acc[u][2 * i]);
            acc[u][2 * i + 1] = __ffma2_rn(xi, k23, acc[u][2 * i + 1]);
          }
        }
      }
    }
    (void)t0;
  }
  cp_async_wait<0>();
  float* pp = part + blockIdx.x * (long long)P;
  if (tid == 0) pp[0] = m;
  if (tid < D) pp[2 + tid] = sk;
  else if (tid < D + DV) pp[2 + D + tid - D] = sv;
  else if (tid == D + DV) pp[1] = om;
#pragma unroll
  for (int u = 0; u < TPB; ++u) {
    if (ar[u] >= 0) {
      const bool kk = ar[u] < D / 4;
      float* dst = pp + 2 + D + DV + (kk ? ar[u] * 4 * D : D * D + (ar[u] - D / 4) * 4 * D) + cr[u] * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dst[i * D] = acc[u][2 * i].x;
        dst[i * D + 1] = acc[u][2 * i].y;
        dst[i * D + 2] = acc[u][2 * i + 1].x;
        dst[i * D + 3] = acc[u][2 * i + 1].y;
      }
    }
  }
  if (!last_arrival(counter + bh, S, &is_last)) return;
  lla_merge_solve<TIn, D, DV>(qs, part, bh, S, inv_h, lam, dsm, &fail_s, out, status);
}

// ------------------------------------------------------------------------------- LLA, tensor cores
// bf16, d = dv = 64. The moment sums of a chunk are two contractions over its keys,
//   Skk = sum_j (p_j k_j) k_j^T,   Svk = sum_j (p_j v_j) k_j^T,
// which run on the tensor cores (tcgen05, one CTA, M = 128, N = 64, fp32 accumulators in tensor
// memory): A = [hi(p_j x_j); lo(p_j x_j)] (128 rows, x = k or v: each product split exactly into
// two bf16 values), B = the key tile. The weights are rounded to bf16 first, as in the forward's
// moments stage, so that every product p_j x_ja k_jb is exact and only the fp32 sums round;
// sum p k, sum p v and omega are summed on the CUDA cores from the same products. The shift of
// the sums moves only when a tile's maximum logit exceeds it by more than 8 ln 2 h (the weights
// stay <= 256 in between), so the accumulators in tensor memory are rescaled rarely. The partial
// of a chunk has the layout of lla_decode_kernel's, and the merge is the same.
namespace dtc {
constexpr int D = 64;
constexpr int TKT = 64;                    // keys per tile
constexpr int ST = 4;                      // key / value ring stages
constexpr int NCW = 8;                     // compute warps; warp NCW loads
constexpr int NTC = (NCW + 1) * 32;
constexpr int A_BYTES = 128 * TKT * 2;     // one A operand: 128 rows x 64 keys, bf16
constexpr int KT_BYTES = TKT * D * 2;      // one key or value tile
constexpr int SM_A = 0;                    // A_k, A_v
constexpr int SM_K = SM_A + 2 * A_BYTES;   // ST key tiles (core-matrix layout: the B operand)
constexpr int SM_V = SM_K + ST * KT_BYTES; // ST value tiles (the same layout)
constexpr int SMEM = SM_V + ST * KT_BYTES; // 96 KiB
constexpr int XLD = 65;                    // row stride (floats) of the accumulator copy
static_assert(2 * 128 * XLD * 4 <= SMEM, "accumulator copy fits the tiles' space");
constexpr uint32_t T_KK = 0, T_VK = 64, TMEM_COLS = 128;
constexpr float kShiftSlack = 5.545177444479562f;  // 8 ln 2
// 16-byte chunk c (elements 8c .. 8c + 7) of key row j of a key tile: core matrix (j / 8, c) of
// 128 bytes, 8-key groups 1024 bytes apart (read by the MMA as an MN-major B operand: K = keys).
__device__ __forceinline__ int kofs(int j, int c) { return (j >> 3) * 1024 + c * 128 + (j & 7) * 16; }
// 16-byte chunk f (rows 8f .. 8f + 7) of key column j of an A operand: core matrix (j / 8, f),
// 8-key groups 2048 bytes apart (an MN-major A operand: M = 128 rows, K = keys).
__device__ __forceinline__ int aofs(int j, int f) { return (j >> 3) * 2048 + f * 128 + (j & 7) * 16; }
__device__ __forceinline__ uint32_t bmul2(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t bfma2(uint32_t x, uint32_t y, uint32_t z) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  return r;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
// Barrier among the compute warps only (named barrier 1; the loader warp does not take part).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ float ex2f_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// The exact products p * x[0..7] (x: 8 bf16 in a 16-byte word) as hi and lo bf16 words, and their
// fp32 values added to acc[0..7].
__device__ __forceinline__ void split_products(uint32_t pp, const uint4& x, uint4& hi, uint4& lo,
                                               float (&acc)[8]) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    h[t] = bmul2(pp, xw[t]);
    l[t] = bfma2(pp, xw[t], h[t] ^ 0x80008000u);
    acc[2 * t] += lo16(h[t]) + lo16(l[t]);
    acc[2 * t + 1] += hi16(h[t]) + hi16(l[t]);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
}  // namespace dtc

__global__ void __launch_bounds__(dtc::NTC)
lla_decode_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, int L, int S, float inv_h, float lam,
                     float* __restrict__ part, int* __restrict__ counter,
                     __nv_bfloat16* __restrict__ out, int* __restrict__ status) {
  using namespace dtc;
  using namespace tc;
  constexpr int P = lla_part<D, D>();
  static_assert(NCW * 32 == 256 && TKT * 4 == 256, "four threads per key; eight per chunk");
  extern __shared__ __align__(1024) float dtc_smem[];
  float* const dsm = dtc_smem;
  uint8_t* const sm = reinterpret_cast<uint8_t*>(dsm);
  __shared__ float qs[D], red[NCW], sS[TKT], xo[NCW];
  __shared__ float xs[NCW][2][D];
  __shared__ uint64_t mbar;            // the MMAs of a tile completed (one phase per tile)
  __shared__ uint64_t full[ST], empty[ST];  // ring slot landed / released by its tile's MMAs
  __shared__ uint32_t tmem_base_s;
  __shared__ int is_last, fail_s, abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long bh = blockIdx.x / S;
  const int s = blockIdx.x % S;
  const int chunk = (L + S - 1) / S;
  const int j0 = s * chunk, j1 = min(L, j0 + chunk);
  const int ntl = j1 > j0 ? (j1 - j0 + TKT - 1) / TKT : 0;
  const __nv_bfloat16* kb = k + bh * (long long)L * D;
  const __nv_bfloat16* vb = v + bh * (long long)L * D;
  for (int a = tid; a < D; a += dtc::NTC) qs[a] = __bfloat162float(q[bh * D + a]);
  if (tid == 0) {
    mbar_init(&mbar, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 32);  // one cp.async completion arrival per loader lane
      mbar_init(&empty[i], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  volatile int* abort_p = &abort_flag;

  float m = -INFINITY;  // the shift of this CTA's sums (raw logit units)
  float acc_k[8], acc_v[8], om = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) { acc_k[e] = 0.f; acc_v[e] = 0.f; }
  if (warp == NCW) {
    // ---- loader: tile it into ring slot it % ST once the MMAs of tile it - ST released it; each
    // lane's copies complete on the slot's barrier (rows past the chunk zero-filled unread)
    for (int it = 0; it < ntl; ++it) {
      const int slot = it % ST;
      if (it >= ST && !mbar_wait(&empty[slot], ((it / ST) - 1) & 1, status, kStatusTimeout, abort_p)) break;
      const int t0 = j0 + it * TKT, n = min(TKT, j1 - t0);
      uint8_t* kd = sm + SM_K + slot * KT_BYTES;
      uint8_t* vd = sm + SM_V + slot * KT_BYTES;
#pragma unroll 4
      for (int e = lane; e < TKT * 8; e += 32) {
        // each group of eight lanes: eight consecutive keys, one chunk (distinct banks)
        const int j = (e & 7) + 8 * (e >> 6), c = (e >> 3) & 7;
        const bool in = j < n;
        const long long row = in ? (long long)(t0 + j) : 0;
        cp_async16(kd + kofs(j, c), kb + row * D + c * 8, in ? 16u : 0u);
        cp_async16(vd + kofs(j, c), vb + row * D + c * 8, in ? 16u : 0u);
      }
      cp_async_mbar_arrive(&full[slot]);
    }
    cp_async_commit();
    cp_async_wait<0>();  // nothing of this warp is in flight past here
  } else {
    // ---- compute warps 0 .. NCW - 1 (named barrier 1 among them)
    // A operands: elements 8 c8 .. 8 c8 + 7 of keys jr and jr + 32; each group of eight lanes
    // takes eight consecutive keys of one chunk (16-byte loads and stores in distinct banks).
    const int c8 = (tid >> 3) & 7, jr = (tid & 7) + 8 * (tid >> 6);
    const float c2 = inv_h * 1.4426950408889634f;
    for (int it = 0; it < ntl; ++it) {
      const int n = min(TKT, j1 - (j0 + it * TKT)), slot = it % ST;
      if (!mbar_wait(&full[slot], (it / ST) & 1, status, kStatusTimeout, abort_p)) *abort_p = 1;
      const uint8_t* kt = sm + SM_K + slot * KT_BYTES;
      const uint8_t* vt = sm + SM_V + slot * KT_BYTES;
      {  // logits: four threads per key, a quarter of the row each; each warp's maximum
        const int key = tid >> 2, q4 = tid & 3;
        float a = 0.f;
        if (key < n) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint4 w = *reinterpret_cast<const uint4*>(kt + kofs(key, 2 * q4 + h2));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int f = 16 * q4 + 8 * h2 + 2 * t;
              a = fmaf(qs[f], lo16(ww[t]), a);
              a = fmaf(qs[f + 1], hi16(ww[t]), a);
            }
          }
        }
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        const float sa = key < n ? a : -INFINITY;
        if (q4 == 0) sS[key] = sa;
        float wm = sa;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        if (lane == 0) red[warp] = wm;
      }
      // The MMAs of tile it - 1 read the A operands rebuilt below (and a rescale needs their sums
      // final): their issuer waits for them before the barrier.
      if (tid == 0 && it >= 1 && !mbar_wait(&mbar, (it - 1) & 1, status, kStatusTimeout, abort_p))
        *abort_p = 1;
      compute_sync();
      float tm = red[0];
#pragma unroll
      for (int w = 1; w < NCW; ++w) tm = fmaxf(tm, red[w]);
      if (m == -INFINITY || (tm - m) * inv_h > kShiftSlack) {
        if (m != -INFINITY) {  // move the accumulated sums to the new shift
          const float sc = __expf((m - tm) * inv_h);
          tc_fence_after();
          const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16) + (warp >> 2) * 64;
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t x[16];
            tmem_ld16(tl + c0, x);
            tmem_ld_wait();
            uint32_t y0[8], y1[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              y0[t] = __float_as_uint(__uint_as_float(x[t]) * sc);
              y1[t] = __float_as_uint(__uint_as_float(x[8 + t]) * sc);
            }
            tmem_st8(tl + c0, y0);
            tmem_st8(tl + c0 + 8, y1);
          }
          tmem_st_wait();
          tc_fence_before();
#pragma unroll
          for (int e = 0; e < 8; ++e) { acc_k[e] *= sc; acc_v[e] *= sc; }
          om *= sc;
        }
        m = tm;
      }
      uint8_t* ak = sm + SM_A;
      uint8_t* av = ak + A_BYTES;
      const float mc = m * c2;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = jr + 32 * u;
        // the weight (bf16), formed by each of the eight threads that use it
        const float p = j < n ? lo16(pack2(ex2f_approx(fmaf(sS[j], c2, -mc)), 0.f)) : 0.f;
        if (c8 == 0) om += p;
        const uint32_t pp = pack2(p, p);  // exact: p is a bf16 value
        const uint4 kw = *reinterpret_cast<const uint4*>(kt + kofs(j, c8));
        const uint4 vw = *reinterpret_cast<const uint4*>(vt + kofs(j, c8));
        uint4 h, l;
        split_products(pp, kw, h, l, acc_k);
        *reinterpret_cast<uint4*>(ak + aofs(j, c8)) = h;
        *reinterpret_cast<uint4*>(ak + aofs(j, 8 + c8)) = l;
        split_products(pp, vw, h, l, acc_v);
        *reinterpret_cast<uint4*>(av + aofs(j, c8)) = h;
        *reinterpret_cast<uint4*>(av + aofs(j, 8 + c8)) = l;
      }
      fence_proxy_async_smem();  // the A operands (generic-proxy writes) before the MMAs read them
      compute_sync();
      if (tid == 0) {
        tc_fence_after();
        fence_proxy_async_smem();  // the key tile's cp.async writes
        const uint64_t adk = smem_desc(smem_u32(ak), 2048, 128);
        const uint64_t adv = smem_desc(smem_u32(av), 2048, 128);
        const uint64_t bd = smem_desc(smem_u32(kt), 1024, 128);
        constexpr uint32_t id = idesc_bf16(128, D, true, true);
#pragma unroll
        for (int s4 = 0; s4 < TKT / 16; ++s4) {
          const uint32_t acc = (it > 0 || s4 > 0) ? 1u : 0u;
          mma_ss(tbase + T_KK, adk + (uint64_t)(s4 * (4096 >> 4)), bd + (uint64_t)(s4 * (2048 >> 4)), id, acc);
          mma_ss(tbase + T_VK, adv + (uint64_t)(s4 * (4096 >> 4)), bd + (uint64_t)(s4 * (2048 >> 4)), id, acc);
        }
        mma_commit(&mbar);
        mma_commit(&empty[slot]);  // the slot's key and value tiles are no longer read
      }
    }
    if (tid == 0) {
      // every MMA has completed before the accumulators are read and tensor memory is released
      // (a bounded wait, whatever the abort flag says)
      volatile int never = 0;
      if (ntl >= 1) mbar_wait(&mbar, (ntl - 1) & 1, status, kStatusTimeout, &never);
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp < NCW) {
    // sums of the CUDA-core partials: over the eight keys of each lane group (lanes 1, 2, 4
    // apart), then in the final sums over the four key groups (warps 2 kg + c8 / 4) in a fixed
    // order
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        acc_k[e] += __shfl_xor_sync(0xffffffffu, acc_k[e], o);
        acc_v[e] += __shfl_xor_sync(0xffffffffu, acc_v[e], o);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) om += __shfl_xor_sync(0xffffffffu, om, o);
    if ((lane & 7) == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xs[warp][0][8 * (lane >> 3) + e] = acc_k[e];
        xs[warp][1][8 * (lane >> 3) + e] = acc_v[e];
      }
    }
    if (lane == 0) xo[warp] = om;
    // the accumulators (128 rows: hi rows 0..63, lo rows 64..127) into shared memory
    float* xm = dsm;  // [2][128][XLD]
    const int quarter = warp & 3, mat = warp >> 2, row = quarter * 32 + lane;
    const uint32_t tl = tbase + ((uint32_t)(quarter * 32) << 16) + mat * 64;
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t x[16];
      tmem_ld16(tl + c0, x);
      tmem_ld_wait();
      // an empty chunk (the last splits of a long cache can get none) has no sums in tensor
      // memory: its partial is zero, weighted 0 by the merge
#pragma unroll
      for (int t = 0; t < 16; ++t)
        xm[(mat * 128 + row) * XLD + c0 + t] = ntl > 0 ? __uint_as_float(x[t]) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
  const float* xm = dsm;
  float* pp = part + blockIdx.x * (long long)P;
  if (tid == 0) {
    float o = 0.f;
    for (int w = 0; w < NCW; ++w) o += xo[w];
    pp[0] = m;
    pp[1] = o;
  }
  if (tid < 2 * D) {
    const int which = tid / D, a = tid % D, c = a >> 3;  // element a: chunk c, lane group c & 3
    float sum = 0.f;
    for (int kg = 0; kg < 4; ++kg) sum += xs[2 * kg + (c >> 2)][which][8 * (c & 3) + (a & 7)];
    pp[2 + tid] = sum;  // sk[a] (which 0), then sv[a]
  }
  for (int e = tid; e < 2 * D * D; e += dtc::NTC) {
    const int mat = e / (D * D), a = (e / D) % D, b = e % D;
    pp[2 + 2 * D + e] = xm[(mat * 128 + a) * XLD + b] + xm[(mat * 128 + 64 + a) * XLD + b];
  }
  if (!last_arrival(counter + bh, S, &is_last)) return;
  lla_merge_solve<__nv_bfloat16, D, D>(qs, part, bh, S, inv_h, lam, dsm, &fail_s, out, status);
}

bool decode_on_tc(const DecodeArgs& a) {
  return !a.r && a.dtype == LLA_BF16 && a.d == 64 && a.dv == 64 && a.path != kPathCudaCore;
}

int choose_splits(long long BH, int L, int per_sm = 2) {
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long s = ((long long)per_sm * sms + BH - 1) / BH;  // about per_sm CTAs per SM
  const long long smax = (L + TK - 1) / TK;  // at least a tile of keys per CTA
  if (s > smax) s = smax;
  if (s > 512) s = 512;
  return s < 1 ? 1 : (int)s;
}

template <typename TIn, int D, int DV>
cudaError_t launch_px(const DecodeArgs& a, void* ws, cudaStream_t st) {
  const int S = choose_splits(a.BH(), a.L);
  float* part = static_cast<float*>(ws);
  int* cnt = reinterpret_cast<int*>(part + a.BH() * S * px_part<D, DV>());
  zero_counters<<<(unsigned)((a.BH() + 255) / 256), 256, 0, st>>>(cnt, (int)a.BH());
  count_launch();
  auto kern = parallax_decode_kernel<TIn, D, DV>;
  constexpr size_t smem = px_smem<TIn, D, DV>();
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)(a.BH() * S), NT, smem, st>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
      static_cast<const TIn*>(a.r), a.L, S, 1.f / a.h, part, cnt, static_cast<TIn*>(a.out));
  count_launch();
  return cudaGetLastError();
}

template <typename TIn, int D, int DV>
cudaError_t launch_ll(const DecodeArgs& a, void* ws, int* status, cudaStream_t st) {
  const int S = choose_splits(a.BH(), a.L);
  float* part = static_cast<float*>(ws);
  int* cnt = reinterpret_cast<int*>(part + a.BH() * S * lla_part<D, DV>());
  constexpr int P = lla_part<D, DV>();
  const size_t tiles = sizeof(float) * (TK * D * 2 + TK * DV + TK) + px_smem<TIn, D, DV>();
  const size_t solve = sizeof(double) * (P + D + S);
  const size_t smem = tiles > solve ? tiles : solve;
  auto kern = lla_decode_kernel<TIn, D, DV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  zero_counters<<<(unsigned)((a.BH() + 255) / 256), 256, 0, st>>>(cnt, (int)a.BH());
  count_launch();
  kern<<<(unsigned)(a.BH() * S), NT, smem, st>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
      a.L, S, 1.f / a.h, a.lam, part, cnt, static_cast<TIn*>(a.out), status);
  count_launch();
  return cudaGetLastError();
}

// The tensor-core split kernel takes about four CTAs' worth of chunks per SM (two resident).
int decode_splits(const DecodeArgs& a) {
  return decode_on_tc(a) ? choose_splits(a.BH(), a.L, 4) : choose_splits(a.BH(), a.L);
}

cudaError_t launch_ll_tc(const DecodeArgs& a, void* ws, int* status, cudaStream_t st) {
  constexpr int D = dtc::D;
  constexpr int P = lla_part<D, D>();
  const int S = decode_splits(a);
  float* part = static_cast<float*>(ws);
  int* cnt = reinterpret_cast<int*>(part + a.BH() * S * P);
  const size_t solve = sizeof(double) * (P + D + S);
  const size_t smem = solve > (size_t)dtc::SMEM ? solve : (size_t)dtc::SMEM;
  cudaError_t err = cudaFuncSetAttribute(lla_decode_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  zero_counters<<<(unsigned)((a.BH() + 255) / 256), 256, 0, st>>>(cnt, (int)a.BH());
  count_launch();
  lla_decode_tc_kernel<<<(unsigned)(a.BH() * S), dtc::NTC, smem, st>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.L, S, 1.f / a.h, a.lam, part, cnt,
      static_cast<__nv_bfloat16*>(a.out), status);
  count_launch();
  return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch(const DecodeArgs& a, void* ws, int* status, cudaStream_t st) {
  if (decode_on_tc(a)) return launch_ll_tc(a, ws, status, st);
#define LLA_DEC(DD, VV)                                                                  \
  if (a.d == DD && a.dv == VV)                                                           \
    return a.r ? launch_px<TIn, DD, VV>(a, ws, st) : launch_ll<TIn, DD, VV>(a, ws, status, st);
  LLA_DEC(16, 16) LLA_DEC(16, 32) LLA_DEC(16, 64)
  LLA_DEC(32, 16) LLA_DEC(32, 32) LLA_DEC(32, 64)
  LLA_DEC(64, 16) LLA_DEC(64, 32) LLA_DEC(64, 64)
#undef LLA_DEC
  return cudaErrorInvalidValue;
}

}  // namespace

size_t decode_workspace_bytes(const DecodeArgs& a) {
  const int S = decode_splits(a);
  const size_t per = a.r ? (size_t)(3 + 2 * a.dv) : (size_t)(2 + a.d + a.dv + a.d * a.d + a.dv * a.d);
  return sizeof(float) * per * (size_t)a.BH() * S + sizeof(int) * (size_t)a.BH() + 256;
}

cudaError_t launch_decode(const DecodeArgs& a, void* ws, int* status, cudaStream_t st) {
  return a.dtype == LLA_F32 ? dispatch<float>(a, ws, status, st)
                            : dispatch<__nv_bfloat16>(a, ws, status, st);
}

}  // namespace lla
