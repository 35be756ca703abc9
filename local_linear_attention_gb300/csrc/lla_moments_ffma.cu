// CUDA-core moments stage of the causal LLA forward.
//
// For every query i of a tile and its causal prefix j <= i this kernel accumulates the
// kernel-weighted moments that the closed form of LLA needs ("Parallax" blog, s.2 Canonical
// Formulation: omega_i = sum_j w_ij and the weighted first and second key moments):
//   omega = sum p_j,  s = sum p_j (k_j - c),  S = sum p_j (k_j - c)(k_j - c)^T,
// with p_j = exp(q_i.k_j/h - m_i) (m_i the exact row max, found in a first pass over the prefix)
// and c a per-head key reference point (the key mean). Shifting the keys by a constant leaves the
// centred moments, and hence LLA, unchanged but removes most of the cancellation when the key
// cloud sits far from the origin. All of omega, s and S come out of one Gram matrix of the
// augmented keys kt = [k - c, 1], accumulated as upper-triangular 4x4 blocks.
//
// Precision: for bf16 inputs the fp32 products k_a*k_b are exact and plain fp32 accumulation is
// used. For fp32 inputs every term is added as an exact fp32 product pair into a TwoSum-
// compensated (hi, lo) accumulator, so the moments carry roughly twice fp32's precision: the
// ridge solve downstream needs it when lambda is small and the keys are nearly low-rank.
#include "lla_internal.cuh"
#include "lla_logit.cuh"

namespace lla {
namespace {

template <int D, bool PRECISE>
struct MomCfg {
  static constexpr int NBLK = gram_nblk(D);
  static constexpr int DP = NBLK * 4;        // padded augmented key length
  static constexpr int NB = gram_nblocks(D); // 4x4 blocks per query
  static constexpr int RQ = PRECISE ? 4 : 8; // queries per thread
  static constexpr int QG = NB >= 192 ? 1 : 192 / NB;  // query groups per CTA
  static constexpr int TQ = QG * RQ;         // queries per CTA
  static constexpr int NT_USED = QG * NB;
  static constexpr int NT = (NT_USED + 31) / 32 * 32;
  static constexpr int BC = 32;              // keys per shared-memory tile
  static constexpr int KS = DP + 4;          // key row stride (floats), keeps rows 16B aligned
  static constexpr int SMEM_FLOATS = TQ * D + 2 * TQ + BC * KS + BC * TQ + D + BC;
};

template <typename TIn, int D, bool PRECISE>
__global__ void __launch_bounds__(MomCfg<D, PRECISE>::NT)
moments_ffma_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                    const float* __restrict__ kmean, int T, int BH, float inv_h,
                    float* __restrict__ m_out, float* __restrict__ mom,
                    float* __restrict__ mom_lo) {
  using C = MomCfg<D, PRECISE>;
  constexpr int TQ = C::TQ, BC = C::BC, DP = C::DP, KS = C::KS, NT = C::NT, RQ = C::RQ;
  constexpr int G = gram_floats(D);
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [TQ][D]
  float* qc = Qs + TQ * D;                       // [TQ] q . c
  float* mrow = qc + TQ;                         // [TQ] running row max
  float* Ks = mrow + TQ;                         // [BC][KS] augmented shifted keys
  float* Ps = Ks + BC * KS;                      // pass 1: logits [TQ][BC]; pass 2: p [BC][TQ]
  float* cs = Ps + BC * TQ;                      // [D]
  int* bad = reinterpret_cast<int*>(cs + D);     // [BC] key has a non-finite element

  const int ntiles = (T + TQ - 1) / TQ;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);  // longest causal prefixes first
  const long long bh = blockIdx.x % BH;
  const int i0 = tile * TQ;
  const int nq = min(TQ, T - i0);
  const int jend = i0 + nq;  // keys [0, jend) are visible to some query of the tile
  const TIn* qb = q + bh * T * D;
  const TIn* kb = k + bh * T * D;
  const int tid = threadIdx.x;

  for (int a = tid; a < D; a += NT) cs[a] = kmean[bh * D + a];
  for (int e = tid; e < TQ * D; e += NT) {
    const int r = e / D;
    Qs[e] = r < nq ? ldf(qb, (long long)(i0 + r) * D + (e % D)) : 0.f;
  }
  __syncthreads();
  for (int r = tid; r < TQ; r += NT) {
    qc[r] = dot_c<D>(Qs + r * D, cs);
    mrow[r] = -INFINITY;
  }

  // Stages keys [j0, j0 + BC) as augmented shifted rows. A non-finite element is replaced by
  // the reference point and the key flagged; its logit is then NaN, so only the rows whose
  // prefix contains it become NaN (a masked weight of 0 times a NaN key would poison the tile).
  // Ends with a barrier.
  auto load_keys = [&](int j0) {
    for (int j = tid; j < BC; j += NT) bad[j] = 0;
    __syncthreads();
    for (int e = tid; e < BC * DP; e += NT) {
      const int j = e / DP, a = e % DP;
      float x;
      if (a < D) {
        x = 0.f;
        if (j0 + j < jend) {
          x = ldf(kb, (long long)(j0 + j) * D + a);
          if (!isfinite(x)) { x = cs[a]; bad[j] = 1; }
          x -= cs[a];
        }
      } else {
        x = (a == D) ? 1.f : 0.f;
      }
      Ks[j * KS + a] = x;
    }
    __syncthreads();
  };
  const float qnan = __int_as_float(0x7fc00000);

  // Pass 1: exact row max of the logits over the causal prefix.
  for (int j0 = 0; j0 < jend; j0 += BC) {
    __syncthreads();
    load_keys(j0);
    for (int e = tid; e < TQ * BC; e += NT) {
      const int r = e / BC, j = e % BC;
      float s = -INFINITY;
      if (r < nq && j0 + j <= i0 + r)
        s = bad[j] ? qnan : logit<D>(Qs + r * D, Ks + j * KS, qc[r], inv_h);
      Ps[e] = s;
    }
    __syncthreads();
    for (int r = tid; r < TQ; r += NT) {
      float mx = mrow[r];
      for (int j = 0; j < BC; ++j) mx = fmaxf(mx, Ps[r * BC + j]);
      mrow[r] = mx;
    }
  }

  // Thread roles for the Gram accumulation: query group qg, 4x4 block (ba, bb), ba <= bb.
  const bool active = tid < C::NT_USED;
  const int qg = tid / C::NB, bi = tid % C::NB;
  int ba = 0, bb = 0;
  {
    int rem = bi;
    for (ba = 0; ba < C::NBLK; ++ba) {
      const int len = C::NBLK - ba;
      if (rem < len) { bb = ba + rem; break; }
      rem -= len;
    }
  }
  const int a0 = ba * 4, b0 = bb * 4, q0 = qg * RQ;

  float acc[RQ][4][4];
  float accl[PRECISE ? RQ : 1][4][4];
#pragma unroll
  for (int r = 0; r < RQ; ++r)
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        acc[r][u][w] = 0.f;
        if (PRECISE) accl[PRECISE ? r : 0][u][w] = 0.f;
      }

  // Pass 2: weights and moments.
  for (int j0 = 0; j0 < jend; j0 += BC) {
    __syncthreads();
    load_keys(j0);
    for (int e = tid; e < TQ * BC; e += NT) {
      const int r = e / BC, j = e % BC;
      float p = 0.f;
      if (r < nq && j0 + j <= i0 + r)
        p = bad[j] ? qnan : expf(logit<D>(Qs + r * D, Ks + j * KS, qc[r], inv_h) - mrow[r]);
      Ps[j * TQ + r] = p;
    }
    __syncthreads();
    if (active) {
      const int jn = min(BC, jend - j0);
      for (int j = 0; j < jn; ++j) {
        float pv[RQ];
#pragma unroll
        for (int r = 0; r < RQ; r += 4) {
          const float4 t = *reinterpret_cast<const float4*>(Ps + j * TQ + q0 + r);
          pv[r] = t.x; pv[r + 1] = t.y; pv[r + 2] = t.z; pv[r + 3] = t.w;
        }
        const float4 ta = *reinterpret_cast<const float4*>(Ks + j * KS + a0);
        const float4 tb = *reinterpret_cast<const float4*>(Ks + j * KS + b0);
        const float ka[4] = {ta.x, ta.y, ta.z, ta.w};
        const float kv[4] = {tb.x, tb.y, tb.z, tb.w};
        if (!PRECISE) {
          float f[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 4; ++w) f[u][w] = ka[u] * kv[w];
#pragma unroll
          for (int r = 0; r < RQ; ++r)
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int w = 0; w < 4; ++w) acc[r][u][w] = fmaf(pv[r], f[u][w], acc[r][u][w]);
        } else {
#pragma unroll
          for (int r = 0; r < RQ; ++r)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float t = pv[r] * ka[u];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float p, e;
                two_prod(t, kv[w], p, e);
                two_sum_acc(acc[r][u][w], accl[PRECISE ? r : 0][u][w], p);
                accl[PRECISE ? r : 0][u][w] += e;
              }
            }
        }
      }
    }
  }

  if (active) {
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      if (q0 + r < nq) {
        const long long row = bh * T + i0 + q0 + r;
        float4* dst = reinterpret_cast<float4*>(mom + row * G + bi * 16);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dst[u] = make_float4(acc[r][u][0], acc[r][u][1], acc[r][u][2], acc[r][u][3]);
        if (PRECISE) {
          float4* dl = reinterpret_cast<float4*>(mom_lo + row * G + bi * 16);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int rr = PRECISE ? r : 0;
            dl[u] = make_float4(accl[rr][u][0], accl[rr][u][1], accl[rr][u][2], accl[rr][u][3]);
          }
        }
      }
    }
  }
  for (int r = tid; r < nq; r += NT) m_out[bh * T + i0 + r] = mrow[r];
}

template <typename TIn, int D, bool PRECISE>
cudaError_t launch_t(const Args& a, const Workspace& ws, cudaStream_t s) {
  using C = MomCfg<D, PRECISE>;
  const size_t smem = sizeof(float) * C::SMEM_FLOATS;
  auto kern = moments_ffma_kernel<TIn, D, PRECISE>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long ntiles = (a.T + C::TQ - 1) / C::TQ;
  const long long blocks = ntiles * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, C::NT, smem, s>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), ws.kmean, a.T, (int)a.BH(),
      1.0f / a.h, ws.m, ws.mom, ws.mom_lo);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_moments_ffma(const Args& a, const Workspace& ws, cudaStream_t s) {
  const bool f32 = a.dtype == LLA_F32;
  switch (a.d) {
    case 16: return f32 ? launch_t<float, 16, true>(a, ws, s) : launch_t<__nv_bfloat16, 16, false>(a, ws, s);
    case 32: return f32 ? launch_t<float, 32, true>(a, ws, s) : launch_t<__nv_bfloat16, 32, false>(a, ws, s);
    case 64: return f32 ? launch_t<float, 64, true>(a, ws, s) : launch_t<__nv_bfloat16, 64, false>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lla
