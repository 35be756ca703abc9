// Causal Parallax backward with a given probe R ("Parallax" blog, Appendix F "Parallax backward
// (closed form)": row scalars cached by a forward-like pass, then a row-tile pass for dQ, dR and
// a column-tile pass for dK, dV). The appendix's formulas did not survive, so the gradient is
// taken from the forward itself (s.2 "Parallax", Appendix B with eta = 0). For query i with
// p_ij = softmax_j(q_i . k_j / h) over j <= i, t_ij = r_i . k_j and tbar_i = sum_j p_ij t_ij:
//   o_i = sum_j a_ij v_j,  a_ij = p_ij (1 + tbar_i - t_ij)     (= vbar_i - Sigma_KV^(i) r_i).
// With the upstream gradient dO_i, g_ij = dO_i . v_j and the row scalars
//   G_i = dO_i . vbar_i = sum_j p_ij g_ij,   D_i = dO_i . o_i + G_i tbar_i,
// every pair (i, j <= i) contributes
//   dt_ij = p_ij (G_i - g_ij),   ds_ij = p_ij ((1 + tbar_i - t_ij) g_ij + G_i t_ij - D_i),
//   dq_i += ds_ij k_j / h,  dr_i += dt_ij k_j,  dk_j += ds_ij q_i / h + dt_ij r_i,
//   dv_j += a_ij dO_i.
//
// bf16 inputs with d = dv = 64 take the tensor-core passes (lla_parallax_bwd_tc.cu). Every other
// shape and dtype (and bf16 d = dv = 64 when the CUDA-core path is requested) takes three launches
// on CUDA cores (fp32 arithmetic):
//  * stats: the forward's online pass (running max with rescale), ending with the row scalars
//    m_i (max logit), 1 / omega_i, tbar_i, G_i, D_i -- 5 floats per row in a float[8] record;
//  * rows: one block per 64-query tile streams the key/value tiles of its causal prefix and
//    accumulates dq, dr;
//  * columns: one block per 64-key tile streams the query tiles from its first key on (with their
//    row scalars) and accumulates dk, dv.
// Four threads per query (or key) each own a quarter of the coordinates, as in the CUDA-core
// forward; each partial dot product is completed by two shuffles within the four.
#include <cstdint>

#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int BT = 64;  // queries (rows pass, stats) or keys (columns pass) per block
constexpr int BS = 32;  // keys (rows pass) or queries (columns pass) per shared-memory tile
constexpr int NTHREADS = BT * 4;
constexpr int STAT = 8;  // floats per row record: m, 1/omega, tbar, G, D, (pad)

__device__ __forceinline__ float sum4(float x, unsigned gmask) {
  x += __shfl_xor_sync(gmask, x, 1);
  x += __shfl_xor_sync(gmask, x, 2);
  return x;
}

// ----------------------------------------------------------------------------- stats
template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NTHREADS)
pbw_stats_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                 const TIn* __restrict__ rp, const TIn* __restrict__ dout, int T, int BH,
                 float inv_h, float* __restrict__ stats) {
  constexpr int DQ = D / 4, DVQ = DV / 4;
  __shared__ float ks[BS][D + 1];
  __shared__ float vs[BS][DV + 1];
  const int tid = threadIdx.x;
  const int part = tid & 3, rl = tid >> 2;
  const int ntiles = (T + BT - 1) / BT;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);  // longest prefixes first
  const long long bh = blockIdx.x % BH;
  const long long base = bh * T;
  const int i0 = tile * BT;
  const int i = i0 + rl;
  const bool valid = i < T;
  const int jend = min(T, i0 + BT);
  const unsigned gmask = 0xFu << ((threadIdx.x & 31) & ~3);

  float qv[DQ], rv[DQ], o1[DVQ], o2[DVQ];
#pragma unroll
  for (int u = 0; u < DQ; ++u) {
    qv[u] = valid ? ldf(q, (base + i) * D + part + 4 * u) * inv_h : 0.f;
    rv[u] = valid ? ldf(rp, (base + i) * D + part + 4 * u) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < DVQ; ++u) o1[u] = o2[u] = 0.f;
  float m = -INFINITY, d1 = 0.f, d2 = 0.f;
  for (int j0 = 0; j0 < jend; j0 += BS) {
    __syncthreads();
    for (int e = tid; e < BS * D; e += NTHREADS) {
      const int jj = e / D, a = e % D;
      ks[jj][a] = j0 + jj < jend ? ldf(k, (base + j0 + jj) * D + a) : 0.f;
    }
    for (int e = tid; e < BS * DV; e += NTHREADS) {
      const int jj = e / DV, c = e % DV;
      vs[jj][c] = j0 + jj < jend ? ldf(v, (base + j0 + jj) * DV + c) : 0.f;
    }
    __syncthreads();
    const int nj = min(BS, (valid ? i + 1 : 0) - j0);
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f, t = 0.f;
#pragma unroll
      for (int u = 0; u < DQ; ++u) {
        s = fmaf(qv[u], ks[jj][part + 4 * u], s);
        t = fmaf(rv[u], ks[jj][part + 4 * u], t);
      }
      s = sum4(s, gmask);
      t = sum4(t, gmask);
      if (s > m) {
        const float sc = expf(m - s);
        d1 *= sc;
        d2 *= sc;
#pragma unroll
        for (int u = 0; u < DVQ; ++u) { o1[u] *= sc; o2[u] *= sc; }
        m = s;
      }
      const float p = expf(s - m), pt = p * t;
      d1 += p;
      d2 += pt;
#pragma unroll
      for (int u = 0; u < DVQ; ++u) {
        const float vv = vs[jj][part + 4 * u];
        o1[u] = fmaf(p, vv, o1[u]);
        o2[u] = fmaf(pt, vv, o2[u]);
      }
    }
  }
  // Row scalars: vbar = O1 / d1, tbar = d2 / d1, o = (1 + tbar) vbar - O2 / d1.
  const float inv = valid ? 1.f / d1 : 0.f;
  const float tbar = d2 * inv;
  float g = 0.f, od = 0.f;
#pragma unroll
  for (int u = 0; u < DVQ; ++u) {
    const float dy = valid ? ldf(dout, (base + i) * DV + part + 4 * u) : 0.f;
    const float vb = o1[u] * inv;
    g = fmaf(dy, vb, g);
    od = fmaf(dy, fmaf(1.f + tbar, vb, -o2[u] * inv), od);
  }
  g = sum4(g, gmask);
  od = sum4(od, gmask);
  if (valid && part == 0) {
    float* st = stats + (base + i) * STAT;
    st[0] = m;
    st[1] = inv;
    st[2] = tbar;
    st[3] = g;
    st[4] = fmaf(g, tbar, od);
  }
}

// ----------------------------------------------------------------------------- rows: dq, dr
template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NTHREADS)
pbw_rows_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                const TIn* __restrict__ rp, const TIn* __restrict__ dout,
                const float* __restrict__ stats, int T, int BH, float inv_h,
                TIn* __restrict__ dq, TIn* __restrict__ dr) {
  constexpr int DQ = D / 4, DVQ = DV / 4;
  __shared__ float ks[BS][D + 1];
  __shared__ float vs[BS][DV + 1];
  const int tid = threadIdx.x;
  const int part = tid & 3, rl = tid >> 2;
  const int ntiles = (T + BT - 1) / BT;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);
  const long long bh = blockIdx.x % BH;
  const long long base = bh * T;
  const int i0 = tile * BT;
  const int i = i0 + rl;
  const bool valid = i < T;
  const int jend = min(T, i0 + BT);
  const unsigned gmask = 0xFu << ((threadIdx.x & 31) & ~3);

  float qv[DQ], rv[DQ], dyv[DVQ], aq[DQ], ar[DQ];
#pragma unroll
  for (int u = 0; u < DQ; ++u) {
    qv[u] = valid ? ldf(q, (base + i) * D + part + 4 * u) * inv_h : 0.f;
    rv[u] = valid ? ldf(rp, (base + i) * D + part + 4 * u) : 0.f;
    aq[u] = ar[u] = 0.f;
  }
#pragma unroll
  for (int u = 0; u < DVQ; ++u) dyv[u] = valid ? ldf(dout, (base + i) * DV + part + 4 * u) : 0.f;
  float m = 0.f, inv_om = 0.f, tbar = 0.f, G = 0.f, Dr = 0.f;
  if (valid) {
    const float* st = stats + (base + i) * STAT;
    m = st[0]; inv_om = st[1]; tbar = st[2]; G = st[3]; Dr = st[4];
  }
  for (int j0 = 0; j0 < jend; j0 += BS) {
    __syncthreads();
    for (int e = tid; e < BS * D; e += NTHREADS) {
      const int jj = e / D, a = e % D;
      ks[jj][a] = j0 + jj < jend ? ldf(k, (base + j0 + jj) * D + a) : 0.f;
    }
    for (int e = tid; e < BS * DV; e += NTHREADS) {
      const int jj = e / DV, c = e % DV;
      vs[jj][c] = j0 + jj < jend ? ldf(v, (base + j0 + jj) * DV + c) : 0.f;
    }
    __syncthreads();
    const int nj = min(BS, (valid ? i + 1 : 0) - j0);
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f, t = 0.f, g = 0.f;
#pragma unroll
      for (int u = 0; u < DQ; ++u) {
        s = fmaf(qv[u], ks[jj][part + 4 * u], s);
        t = fmaf(rv[u], ks[jj][part + 4 * u], t);
      }
#pragma unroll
      for (int u = 0; u < DVQ; ++u) g = fmaf(dyv[u], vs[jj][part + 4 * u], g);
      s = sum4(s, gmask);
      t = sum4(t, gmask);
      g = sum4(g, gmask);
      const float p = expf(s - m) * inv_om;
      const float ds = p * (fmaf(1.f + tbar - t, g, G * t) - Dr);
      const float dt = p * (G - g);
#pragma unroll
      for (int u = 0; u < DQ; ++u) {
        const float kk = ks[jj][part + 4 * u];
        aq[u] = fmaf(ds, kk, aq[u]);
        ar[u] = fmaf(dt, kk, ar[u]);
      }
    }
  }
  if (valid) {
#pragma unroll
    for (int u = 0; u < DQ; ++u) {
      stf(dq, (base + i) * D + part + 4 * u, aq[u] * inv_h);
      stf(dr, (base + i) * D + part + 4 * u, ar[u]);
    }
  }
}

// ----------------------------------------------------------------------------- columns: dk, dv
template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NTHREADS)
pbw_cols_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                const TIn* __restrict__ rp, const TIn* __restrict__ dout,
                const float* __restrict__ stats, int T, int BH, float inv_h,
                TIn* __restrict__ dk, TIn* __restrict__ dv) {
  constexpr int DQ = D / 4, DVQ = DV / 4;
  __shared__ float qs[BS][D + 1];   // q / h
  __shared__ float rs[BS][D + 1];
  __shared__ float ys[BS][DV + 1];  // dO
  __shared__ float ss[BS][STAT];
  const int tid = threadIdx.x;
  const int part = tid & 3, cl = tid >> 2;
  const long long bh = blockIdx.x % BH;
  const int tile = (int)(blockIdx.x / BH);  // most queries (earliest keys) first
  const long long base = bh * T;
  const int j0 = tile * BT;
  const int j = j0 + cl;
  const bool valid = j < T;
  const unsigned gmask = 0xFu << ((threadIdx.x & 31) & ~3);

  float kv[DQ], vv[DVQ], ak[DQ], av[DVQ];
#pragma unroll
  for (int u = 0; u < DQ; ++u) {
    kv[u] = valid ? ldf(k, (base + j) * D + part + 4 * u) : 0.f;
    ak[u] = 0.f;
  }
#pragma unroll
  for (int u = 0; u < DVQ; ++u) {
    vv[u] = valid ? ldf(v, (base + j) * DV + part + 4 * u) : 0.f;
    av[u] = 0.f;
  }
  for (int i0 = j0; i0 < T; i0 += BS) {
    __syncthreads();
    for (int e = tid; e < BS * D; e += NTHREADS) {
      const int ii = e / D, a = e % D;
      const bool in = i0 + ii < T;
      qs[ii][a] = in ? ldf(q, (base + i0 + ii) * D + a) * inv_h : 0.f;
      rs[ii][a] = in ? ldf(rp, (base + i0 + ii) * D + a) : 0.f;
    }
    for (int e = tid; e < BS * DV; e += NTHREADS) {
      const int ii = e / DV, c = e % DV;
      ys[ii][c] = i0 + ii < T ? ldf(dout, (base + i0 + ii) * DV + c) : 0.f;
    }
    for (int e = tid; e < BS * STAT; e += NTHREADS) {
      const int ii = e / STAT, c = e % STAT;
      ss[ii][c] = i0 + ii < T ? stats[(base + i0 + ii) * STAT + c] : 0.f;
    }
    __syncthreads();
    // queries i of this tile with j <= i < T (the same for the four threads of a key)
    const int ib = valid ? max(0, j - i0) : BS;
    const int ie = min(BS, T - i0);
    for (int ii = ib; ii < ie; ++ii) {
      float s = 0.f, t = 0.f, g = 0.f;
#pragma unroll
      for (int u = 0; u < DQ; ++u) {
        s = fmaf(qs[ii][part + 4 * u], kv[u], s);
        t = fmaf(rs[ii][part + 4 * u], kv[u], t);
      }
#pragma unroll
      for (int u = 0; u < DVQ; ++u) g = fmaf(ys[ii][part + 4 * u], vv[u], g);
      s = sum4(s, gmask);
      t = sum4(t, gmask);
      g = sum4(g, gmask);
      const float m = ss[ii][0], inv_om = ss[ii][1], tbar = ss[ii][2], G = ss[ii][3];
      const float Dr = ss[ii][4];
      const float p = expf(s - m) * inv_om;
      const float ds = p * (fmaf(1.f + tbar - t, g, G * t) - Dr);
      const float dt = p * (G - g);
      const float a = p * (1.f + tbar - t);
#pragma unroll
      for (int u = 0; u < DQ; ++u)
        ak[u] = fmaf(ds, qs[ii][part + 4 * u], fmaf(dt, rs[ii][part + 4 * u], ak[u]));
#pragma unroll
      for (int u = 0; u < DVQ; ++u) av[u] = fmaf(a, ys[ii][part + 4 * u], av[u]);
    }
  }
  if (valid) {
#pragma unroll
    for (int u = 0; u < DQ; ++u) stf(dk, (base + j) * D + part + 4 * u, ak[u]);
#pragma unroll
    for (int u = 0; u < DVQ; ++u) stf(dv, (base + j) * DV + part + 4 * u, av[u]);
  }
}

template <typename TIn, int D, int DV>
cudaError_t launch_all(const ParallaxBwdArgs& a, float* stats, cudaStream_t s) {
  const long long blocks = (long long)((a.T + BT - 1) / BT) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const TIn* q = static_cast<const TIn*>(a.q);
  const TIn* k = static_cast<const TIn*>(a.k);
  const TIn* v = static_cast<const TIn*>(a.v);
  const TIn* r = static_cast<const TIn*>(a.r);
  const TIn* dy = static_cast<const TIn*>(a.dout);
  const float inv_h = 1.0f / a.h;
  const int BH = (int)a.BH();
  pbw_stats_kernel<TIn, D, DV><<<(unsigned)blocks, NTHREADS, 0, s>>>(q, k, v, r, dy, a.T, BH,
                                                                      inv_h, stats);
  count_launch();
  pbw_rows_kernel<TIn, D, DV><<<(unsigned)blocks, NTHREADS, 0, s>>>(
      q, k, v, r, dy, stats, a.T, BH, inv_h, static_cast<TIn*>(a.dq), static_cast<TIn*>(a.dr));
  count_launch();
  pbw_cols_kernel<TIn, D, DV><<<(unsigned)blocks, NTHREADS, 0, s>>>(
      q, k, v, r, dy, stats, a.T, BH, inv_h, static_cast<TIn*>(a.dk), static_cast<TIn*>(a.dv));
  count_launch();
  return cudaGetLastError();
}

template <typename TIn, int D>
cudaError_t dispatch_dv(const ParallaxBwdArgs& a, float* stats, cudaStream_t s) {
  switch (a.dv_) {
    case 16: return launch_all<TIn, D, 16>(a, stats, s);
    case 32: return launch_all<TIn, D, 32>(a, stats, s);
    default: return launch_all<TIn, D, 64>(a, stats, s);
  }
}

template <typename TIn>
cudaError_t dispatch_d(const ParallaxBwdArgs& a, float* stats, cudaStream_t s) {
  switch (a.d) {
    case 16: return dispatch_dv<TIn, 16>(a, stats, s);
    case 32: return dispatch_dv<TIn, 32>(a, stats, s);
    default: return dispatch_dv<TIn, 64>(a, stats, s);
  }
}

}  // namespace

size_t parallax_bwd_workspace_bytes(const ParallaxBwdArgs& a) {
  return (size_t)a.BH() * (size_t)a.T * STAT * sizeof(float);
}

cudaError_t launch_parallax_bwd(const ParallaxBwdArgs& a, void* ws, int path, int* status,
                                cudaStream_t s) {
  float* stats = static_cast<float*>(ws);
  if (path != kPathCudaCore && a.dtype == LLA_BF16 && a.d == 64 && a.dv_ == 64)
    return launch_parallax_bwd_tc(a, stats, status, s);
  return a.dtype == LLA_F32 ? dispatch_d<float>(a, stats, s)
                            : dispatch_d<__nv_bfloat16>(a, stats, s);
}

}  // namespace lla
