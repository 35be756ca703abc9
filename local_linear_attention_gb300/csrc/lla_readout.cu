// Readout stage of the causal LLA forward (CUDA cores).
//
// Given the ridge-solve result y_i and the weighted key mean kbar_i of every query, one streaming
// pass over the causal prefix evaluates
//   o_i = c_v + sum_j p_ij (v_j - c_v) / omega_i  +  sum_j p_ij (v_j - c_v) t_ij,
//   t_ij = (k_j - kbar_i) . y_i,
// i.e. vbar_i + C_vk y_i, the centred closed form of the LLA intercept ("Parallax" blog, s.2
// Canonical Formulation). Since sum_j p_ij t_ij = 0, the second sum needs no separate vbar term.
// The pass has the two-branch shape of the blog's streaming algorithm (s.3 "One extra branch,
// no extra I/O"): a softmax branch (omega, sum p v) and a covariance branch (sum p t v with t
// the probe score), sharing the weights and the K/V tiles.
//
// Rounding: t is formed from k_j - kbar_i element by element rather than as k.y - kbar.y, which
// would cancel catastrophically when y is large (small ridge, query far from the keys); values
// are shifted by the per-head value mean c_v so that the covariance-branch sum does not carry a
// large constant that cancels. A non-finite key or value is zeroed in shared memory and flagged,
// so that exactly the rows whose prefix contains it come out NaN.
#include "lla_internal.cuh"
#include "lla_logit.cuh"

namespace lla {
namespace {

constexpr int kReadoutThreads = 256;

template <int D, int DV>
struct RoCfg {
  static constexpr int NEC = DV / 4;                        // 4-wide output chunks per query
  static constexpr int NRG = kReadoutThreads / NEC;         // query groups
  static constexpr int TQ = NRG > 32 ? NRG : 32;            // queries per CTA
  static constexpr int RPT = TQ / NRG;                      // queries per thread
  static constexpr int BC = 32;                             // keys per tile
  static constexpr int KS = D + 1;                          // key row stride (conflict-free)
  static constexpr int PS = TQ + 1;                         // weight row stride
  static constexpr int SMEM_FLOATS =
      3 * TQ * D + 2 * TQ + BC * KS + BC * DV + 2 * BC * PS + D + DV + BC;
};

template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(kReadoutThreads)
readout_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
               const float* __restrict__ kmean, const float* __restrict__ vmean,
               const float* __restrict__ mrow_g, const float* __restrict__ y,
               const float* __restrict__ kbar, int T, int BH, float inv_h,
               TIn* __restrict__ out) {
  using C = RoCfg<D, DV>;
  constexpr int TQ = C::TQ, BC = C::BC, KS = C::KS, PS = C::PS, RPT = C::RPT, NEC = C::NEC;
  constexpr int NT = kReadoutThreads;
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [TQ][D]
  float* Ys = Qs + TQ * D;                       // [TQ][D]
  float* KBs = Ys + TQ * D;                      // [TQ][D] kbar - c
  float* qc = KBs + TQ * D;                      // [TQ]
  float* mr = qc + TQ;                           // [TQ]
  float* Vs = mr + TQ;                           // [BC][DV] v - c_v (16B aligned: offsets are /4)
  float* Ks = Vs + BC * DV;                      // [BC][KS] k - c
  float* Pw = Ks + BC * KS;                      // [BC][PS] p
  float* Pt = Pw + BC * PS;                      // [BC][PS] p * t
  float* cs = Pt + BC * PS;                      // [D]
  float* cvs = cs + D;                           // [DV]
  int* bad = reinterpret_cast<int*>(cvs + DV);   // [BC] non-finite key or value

  const int ntiles = (T + TQ - 1) / TQ;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);
  const long long bh = blockIdx.x % BH;
  const int i0 = tile * TQ;
  const int nq = min(TQ, T - i0);
  const int jend = i0 + nq;
  const long long base = bh * T;
  const int tid = threadIdx.x;

  for (int a = tid; a < D; a += NT) cs[a] = kmean[bh * D + a];
  for (int a = tid; a < DV; a += NT) cvs[a] = vmean[bh * DV + a];
  for (int e = tid; e < TQ * D; e += NT) {
    const int r = e / D;
    const bool in = r < nq;
    const long long g = (base + i0 + r) * D + (e % D);
    Qs[e] = in ? ldf(q, g) : 0.f;
    Ys[e] = in ? y[g] : 0.f;
    KBs[e] = in ? kbar[g] : 0.f;
  }
  for (int r = tid; r < TQ; r += NT) mr[r] = r < nq ? mrow_g[base + i0 + r] : 0.f;
  __syncthreads();
  for (int r = tid; r < TQ; r += NT) qc[r] = dot_c<D>(Qs + r * D, cs);

  const int ec = tid % NEC, rg = tid / NEC;
  float sv[RPT][4], o2[RPT][4], om[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    om[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) sv[r][c] = o2[r][c] = 0.f;
  }

  for (int j0 = 0; j0 < jend; j0 += BC) {
    __syncthreads();
    for (int j = tid; j < BC; j += NT) bad[j] = 0;
    __syncthreads();
    for (int e = tid; e < BC * D; e += NT) {
      const int j = e / D, a = e % D;
      float x = 0.f;
      if (j0 + j < jend) {
        x = ldf(k, (base + j0 + j) * D + a);
        if (!isfinite(x)) { x = cs[a]; bad[j] = 1; }
        x -= cs[a];
      }
      Ks[j * KS + a] = x;
    }
    for (int e = tid; e < BC * DV; e += NT) {
      const int j = e / DV, a = e % DV;
      float x = 0.f;
      if (j0 + j < jend) {
        x = ldf(v, (base + j0 + j) * DV + a);
        if (!isfinite(x)) { x = cvs[a]; bad[j] = 1; }
        x -= cvs[a];
      }
      Vs[e] = x;
    }
    __syncthreads();
    for (int e = tid; e < TQ * BC; e += NT) {
      const int r = e / BC, j = e % BC;
      float p = 0.f, pt = 0.f;
      if (r < nq && j0 + j <= i0 + r) {
        p = bad[j] ? __int_as_float(0x7fc00000)
                   : expf(logit<D>(Qs + r * D, Ks + j * KS, qc[r], inv_h) - mr[r]);
        float t = 0.f;
#pragma unroll 16
        for (int a = 0; a < D; ++a) t = fmaf(Ys[r * D + a], Ks[j * KS + a] - KBs[r * D + a], t);
        pt = p * t;
      }
      Pw[j * PS + r] = p;
      Pt[j * PS + r] = pt;
    }
    __syncthreads();
    const int jn = min(BC, jend - j0);
    for (int j = 0; j < jn; ++j) {
      const float4 vv = *reinterpret_cast<const float4*>(Vs + j * DV + ec * 4);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const int rr = rg + r * C::NRG;
        const float p = Pw[j * PS + rr], pt = Pt[j * PS + rr];
        om[r] += p;
        sv[r][0] = fmaf(p, vv.x, sv[r][0]);
        sv[r][1] = fmaf(p, vv.y, sv[r][1]);
        sv[r][2] = fmaf(p, vv.z, sv[r][2]);
        sv[r][3] = fmaf(p, vv.w, sv[r][3]);
        o2[r][0] = fmaf(pt, vv.x, o2[r][0]);
        o2[r][1] = fmaf(pt, vv.y, o2[r][1]);
        o2[r][2] = fmaf(pt, vv.z, o2[r][2]);
        o2[r][3] = fmaf(pt, vv.w, o2[r][3]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int rr = rg + r * C::NRG;
    // a row listed for the exact pass (kbar[row][0] == kListedBits) is written by that pass
    if (rr < nq && __float_as_uint(KBs[rr * D]) != kListedBits) {
      const long long o = (base + i0 + rr) * DV + ec * 4;
      const float inv = 1.f / om[r];
#pragma unroll
      for (int c = 0; c < 4; ++c) stf(out, o + c, cvs[ec * 4 + c] + fmaf(sv[r][c], inv, o2[r][c]));
    }
  }
}

template <typename TIn, int D, int DV>
cudaError_t launch_ro_t(const Args& a, const Workspace& ws, cudaStream_t s) {
  using C = RoCfg<D, DV>;
  const size_t smem = sizeof(float) * C::SMEM_FLOATS;
  auto kern = readout_kernel<TIn, D, DV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)((a.T + C::TQ - 1) / C::TQ) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, kReadoutThreads, smem, s>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
      ws.kmean, ws.vmean, ws.m, ws.y, ws.kbar, a.T, (int)a.BH(), 1.0f / a.h,
      static_cast<TIn*>(a.out));
  count_launch();
  return cudaGetLastError();
}

template <typename TIn, int D>
cudaError_t launch_ro_dv(const Args& a, const Workspace& ws, cudaStream_t s) {
  switch (a.dv) {
    case 16: return launch_ro_t<TIn, D, 16>(a, ws, s);
    case 32: return launch_ro_t<TIn, D, 32>(a, ws, s);
    case 64: return launch_ro_t<TIn, D, 64>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t launch_ro_d(const Args& a, const Workspace& ws, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_ro_dv<TIn, 16>(a, ws, s);
    case 32: return launch_ro_dv<TIn, 32>(a, ws, s);
    case 64: return launch_ro_dv<TIn, 64>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_readout(const Args& a, const Workspace& ws, cudaStream_t s) {
  return a.dtype == LLA_F32 ? launch_ro_d<float>(a, ws, s) : launch_ro_d<__nv_bfloat16>(a, ws, s);
}

}  // namespace lla
