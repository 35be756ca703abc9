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
#include "lla_tc_ptx.cuh"

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
            float* __restrict__ kmean, float* __restrict__ vmean, int zero_keys,
            int* __restrict__ short_count) {
  extern __shared__ float red[];  // [256]
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *short_count = 0;  // this call's list
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

// ----------------------------------------------------------------------------- key frame
// The tensor-core path accumulates exact products of bf16 keys in fp32. When a head's keys sit
// far from the origin, the raw second moment sum p k k^T is much larger than its centred part
// C_kk = S - s s^T / omega, and fp32 rounding of S can exceed the smallest eigenvalues of
// C_kk + lambda' I (queries beyond the keys, small ridge): the factorisation then fails. So the
// path works in a per-head frame: a reference key c (feature a shifted by the key mean rounded to
// bf16 when that mean exceeds a quarter of the feature's spread, else 0) is subtracted once, and
// the moments, the solve and the readout all use kt = bf16(k - c). Shifting leaves the centred
// moments, and hence LLA, unchanged; rounding the shifted keys to bf16 (exact when c = 0 or when
// k - c is representable) perturbs the keys, consistently for every stage. Non-finite keys stay
// non-finite in the frame.

// Partial sums of k and k^2 per feature over chunk blockIdx.y of head blockIdx.x (finite keys).
__global__ void __launch_bounds__(256)
key_stats_kernel(const __nv_bfloat16* __restrict__ k, int T, float* __restrict__ part,
                 int* __restrict__ rep_count, int* __restrict__ short_count) {
  constexpr int D = 64;
  __shared__ float red[2][256];
  const int tid = threadIdx.x, a = tid & (D - 1), r0 = tid >> 6;
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {  // this call's repair and short lists
    rep_count[0] = 0;
    *short_count = 0;
  }
  const long long bh = blockIdx.x;
  const int ch = blockIdx.y;
  const int t0 = (int)((long long)T * ch / kKeyStatChunks);
  const int t1 = (int)((long long)T * (ch + 1) / kKeyStatChunks);
  float s = 0.f, s2 = 0.f;
  for (int j = t0 + r0; j < t1; j += 256 / D) {
    const float x = __bfloat162float(k[(bh * T + j) * D + a]);
    if (isfinite(x)) {
      s += x;
      s2 = fmaf(x, x, s2);
    }
  }
  red[0][tid] = s;
  red[1][tid] = s2;
  __syncthreads();
  if (tid < 2 * D) {
    const int w = tid / D;  // 0: sum, 1: sum of squares
    float t = 0.f;
    for (int r = 0; r < 256 / D; ++r) t += red[w][r * D + a];
    part[((bh * kKeyStatChunks + ch) * 2 + w) * D + a] = t;
  }
}

// The head's reference key c from the partial sums (every CTA of the head derives it in the same
// order, so all agree), then its chunk of the shifted keys kt = bf16(k - c), eight at a time.
constexpr int kShiftChunks = 8;
__global__ void __launch_bounds__(256)
shift_keys_kernel(const __nv_bfloat16* __restrict__ k, int T, const float* __restrict__ part,
                  float* __restrict__ kref, __nv_bfloat16* __restrict__ ksh) {
  constexpr int D = 64;
  __shared__ float cs[D];
  const int tid = threadIdx.x;
  const long long bh = blockIdx.x;
  if (tid < D) {
    double s = 0.0, s2 = 0.0;
    for (int ch = 0; ch < kKeyStatChunks; ++ch) {
      s += part[((bh * kKeyStatChunks + ch) * 2) * D + tid];
      s2 += part[((bh * kKeyStatChunks + ch) * 2 + 1) * D + tid];
    }
    const double mean = s / T, var = fmax(s2 / T - mean * mean, 0.0);
    const float c = 16.0 * mean * mean > var ? __bfloat162float(__float2bfloat16_rn((float)mean)) : 0.f;
    cs[tid] = c;
    if (blockIdx.y == 0) kref[bh * D + tid] = c;
  }
  __syncthreads();
  const long long n8 = (long long)T * D / 8;  // groups of eight keys' features of this head
  const long long g0 = n8 * blockIdx.y / kShiftChunks, g1 = n8 * (blockIdx.y + 1) / kShiftChunks;
  const uint4* src = reinterpret_cast<const uint4*>(k + bh * T * D);
  uint4* dst = reinterpret_cast<uint4*>(ksh + bh * T * D);
  for (long long g = g0 + tid; g < g1; g += 256) {
    const uint4 x = src[g];
    const int a0 = (int)((g * 8) & (D - 1));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float lo = __uint_as_float(w[t] << 16) - cs[a0 + 2 * t];
      const float hi = __uint_as_float(w[t] & 0xFFFF0000u) - cs[a0 + 2 * t + 1];
      const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
      o[t] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    dst[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ----------------------------------------------------------------------------- solve
constexpr int kWarpsPerBlock = 4;

// Moment layouts: FMT 0 = augmented-Gram 4x4 blocks (CUDA-core stage, gram_floats(D) per row, plus
// as many compensation terms for fp32 inputs); FMT 1 = tensor-core stage (d = 64, TC_ROW floats
// per row in the order tc_slot() decodes, omega in its own array).
constexpr int TC_ROW = 2208;

// Slot of feature (a, b), a <= b <= 64, in a tensor-core moment row (the tensor-core moments
// stage documents the order: row pairs (a, b), (a, b+1) for even b, then odd diagonal pairs).
__device__ __forceinline__ int tc_slot(int a, int b) {
  if (a == b && (a & 1)) return 2 * (1088 + ((a - 1) >> 2)) + (((a - 1) >> 1) & 1);
  const int t = a >> 1;
  int rs = 65 * t - t * (t - 1);
  if (a & 1) rs += 33 - t;
  const int b0 = a + (a & 1);
  return 2 * (rs + ((b - b0) >> 1)) + ((b - b0) & 1);
}

template <int D, int FMT>
__device__ __forceinline__ int moff(int a, int b) {  // a <= b; b == D means the constant 1
  if (FMT == 0) return gram_block_index(D, a >> 2, b >> 2) * 16 + (a & 3) * 4 + (b & 3);
  return tc_slot(a, b);
}

template <int D, bool PRECISE, int FMT>
struct SolveCfg {
  static constexpr int ROW = FMT == 0 ? gram_floats(D) : TC_ROW;   // floats of one moment row
  static constexpr int STAGE = (PRECISE ? 2 : 1) * ROW;             // staged per warp (hi [+ lo])
  static constexpr int LS = 68;                                     // row stride of L in smem
  static constexpr int BUF = STAGE > D * LS ? STAGE : D * LS;       // then reused for L's rows
  static constexpr int WARP_FLOATS = BUF + 2 * 64;                  // + two column buffers
  static constexpr int NSLOT = D == 64 ? 2 : 1;                     // rows per lane
};

// State of one lane during the factorisation: its rows (slot 0: row rr0 = lane, entries
// 0..W0-1; slot 1 (d = 64 only): row rr1 = 63 - lane, entries 0..63), right-hand sides and the
// reciprocals of the factor's diagonal for those rows. Entries beyond a row's diagonal are
// padding: they are updated along with the rest (that is cheaper than masking them) and never read.
template <int D>
struct CholLane {
  static constexpr int NS = D == 64 ? 2 : 1;
  static constexpr int W0 = D < 32 ? D : 32;
  static constexpr int W1 = NS == 2 ? D : 1;
  float a0[W0], a1[W1];
  float z[NS];
  float invd[NS];
  int rr0, rr1;
  bool live0;
  bool ok;
};

// Column K of the right-looking factorisation, with the forward substitution as an extra column
// (template recursion keeps every register index static).
template <int D, int K>
__device__ __forceinline__ void chol_column(CholLane<D>& L, float* colbuf) {
  constexpr int NS = CholLane<D>::NS, W0 = CholLane<D>::W0;
  constexpr bool second = NS == 2 && K >= 32;  // slot of row K in its owner lane
  constexpr int owner = second ? D - 1 - K : K;
  const float mine = second ? L.a1[NS == 2 ? K : 0] : L.a0[K < W0 ? K : 0];
  float piv = __shfl_sync(0xffffffffu, mine, owner);
  if (!(piv > 0.f)) { L.ok = false; piv = 1.f; }  // rows of a failed factorisation become NaN
  const float inv = rsqrtf(piv), lkk = piv * inv;
  const float zk = __shfl_sync(0xffffffffu, second ? L.z[NS - 1] : L.z[0], owner) * inv;
  float* cb = colbuf + (K & 1) * 64;
  if constexpr (K < W0) {
    L.a0[K] *= inv;  // L[rr0][K] below the diagonal (padding above it)
    if (L.rr0 == K) { L.a0[K] = lkk; L.invd[0] = inv; L.z[0] = zk; }
    if (L.live0) cb[L.rr0] = L.a0[K];
  }
  if constexpr (NS == 2) {
    L.a1[K] *= inv;
    if (L.rr1 == K) { L.a1[K] = lkk; L.invd[NS - 1] = inv; L.z[NS - 1] = zk; }
    cb[L.rr1] = L.a1[K];
  }
  __syncwarp();
  // trailing update (rows at or above K only touch their padding), column read 4 at a time
  if constexpr (K + 1 < W0) {
    const float lik = L.a0[K];
#pragma unroll
    for (int jb = (K + 1) / 4; jb < W0 / 4; ++jb) {
      const float4 c4 = reinterpret_cast<const float4*>(cb)[jb];
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (4 * jb + u > K) L.a0[4 * jb + u] = fmaf(-lik, cv[u], L.a0[4 * jb + u]);
    }
    if (L.rr0 > K) L.z[0] = fmaf(-lik, zk, L.z[0]);
  }
  if constexpr (NS == 2) {
    const float lik = L.a1[K];
#pragma unroll
    for (int jb = (K + 1) / 4; jb < D / 4; ++jb) {
      const float4 c4 = reinterpret_cast<const float4*>(cb)[jb];
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (4 * jb + u > K) L.a1[4 * jb + u] = fmaf(-lik, cv[u], L.a1[4 * jb + u]);
    }
    if (L.rr1 > K) L.z[NS - 1] = fmaf(-lik, zk, L.z[NS - 1]);
  }
  if constexpr (K + 1 < D) chol_column<D, K + 1>(L, colbuf);
}

// Backward substitution L^T y = z', column by column from the last row: y_k = w_k / L[k][k],
// then w_m -= L[k][m] y_k for m < k. Rows of L are read from shared memory (Lrows[k * 68 + m]).
template <int D, int K>
__device__ __forceinline__ void back_column(const CholLane<D>& L, const float* Lrows, float& w0,
                                            float& w1, float& y0, float& y1) {
  constexpr int NS = CholLane<D>::NS;
  constexpr bool second = NS == 2 && K >= 32;
  constexpr int owner = second ? D - 1 - K : K;
  const float l0 = Lrows[K * 68 + L.rr0];
  const float l1 = NS == 2 ? Lrows[K * 68 + L.rr1] : 0.f;
  const float own = second ? w1 * L.invd[NS - 1] : w0 * L.invd[0];
  const float yk = __shfl_sync(0xffffffffu, own, owner);
  if (L.rr0 == K) y0 = yk;
  if (NS == 2 && L.rr1 == K) y1 = yk;
  if (L.rr0 < K) w0 = fmaf(-l0, yk, w0);
  if (NS == 2 && L.rr1 < K) w1 = fmaf(-l1, yk, w1);
  if constexpr (K > 0) back_column<D, K - 1>(L, Lrows, w0, w1, y0, y1);
}

// One warp solves (C_kk + lambda' I) y = q - kbar for one query, C_kk = S - s s^T / omega from that
// query's moments, by a Cholesky factorisation held in registers: lane l owns row l and, for
// d = 64, also row 63 - l (so that every lane holds 65 entries of the lower triangle). Column k of
// the factor is broadcast through shared memory; the forward substitution rides along as an extra
// column of the factorisation; the backward substitution reduces across the warp.
template <typename TIn, int D, bool PRECISE, int FMT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 3)
solve_kernel(const TIn* __restrict__ q, const float* __restrict__ kmean,
             const float* __restrict__ mom, const float* __restrict__ mom_lo,
             const float* __restrict__ omega, const float* __restrict__ mrow, int T,
             long long rows, float lam, float* __restrict__ y_out, float* __restrict__ kbar_out,
             int* __restrict__ short_count, int* __restrict__ short_rows,
             int* __restrict__ status) {
  using C = SolveCfg<D, PRECISE, FMT>;
  constexpr int NS = CholLane<D>::NS;
  constexpr int W0 = CholLane<D>::W0;
  using R = typename std::conditional<PRECISE, double, float>::type;
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* g = smem + warp * C::WARP_FLOATS;  // staged moment row (hi, then lo); later L's rows
  float* colbuf = g + C::BUF;               // [2][64]
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= rows) return;  // whole warp leaves together
  const long long bh = row / T;

  // Stage the moment row with 16-byte asynchronous copies, all in flight at once before the one
  // wait (rows are 16-byte aligned: ROW % 4 == 0).
  {
    const float4* src = reinterpret_cast<const float4*>(mom + row * C::ROW);
    float4* dst = reinterpret_cast<float4*>(g);
    constexpr int NV = C::ROW / 4;
#pragma unroll 1
    for (int t = lane; t < NV; t += 32) tc::cp_async16(dst + t, src + t, 16u);
    if (PRECISE) {
      const float4* srl = reinterpret_cast<const float4*>(mom_lo + row * C::ROW);
#pragma unroll 1
      for (int t = lane; t < NV; t += 32) tc::cp_async16(dst + NV + t, srl + t, 16u);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<0>();
  }
  __syncwarp();
  auto M = [&](int a, int b) -> R {  // moment entry, hi + lo
    const int ix = moff<D, FMT>(a, b);
    R v = g[ix];
    if (PRECISE) v += (R)g[C::ROW + ix];
    return v;
  };

  const R om = FMT == 0 ? M(D, D) : (R)omega[row];
  const R inv_om = R(1) / om;
  double lpd = (double)lam * exp(-(double)mrow[row]);  // ridge scaled by exp(-m)
  lpd = fmin(fmax(lpd, (double)FLT_MIN), (double)FLT_MAX);
  const R lp = (R)lpd;

  // This lane's rows, their right-hand sides q - kbar and their lower-triangle entries.
  CholLane<D> L;
  L.rr0 = lane;
  L.rr1 = D - 1 - lane;
  L.live0 = lane < D;
  L.ok = true;
  const bool live0 = L.live0;
  int rr[NS];
  rr[0] = L.rr0;
  if (NS == 2) rr[NS - 1] = L.rr1;
  float kb[NS];
  float kb1 = 0.f, ctr = 0.f;  // this lane's share of |kbar|_1 and tr(C_kk) (short-prefix rule)
#pragma unroll
  for (int t = 0; t < NS; ++t) {
    L.invd[t] = 1.f;
    const int r = rr[t];
    if (t == 0 && !live0) { L.z[0] = 0.f; kb[0] = 0.f; continue; }
    const R sr = M(r, D);
    const R kbar = sr * inv_om;
    kb[t] = (float)kbar;
    kb1 += fabsf((float)kbar);
    ctr += (float)(M(r, r) - sr * kbar);
    L.z[t] = (float)((R)ldf(q, row * D + r) - (R)kmean[bh * D + r] - kbar);
  }
#pragma unroll
  for (int j = 0; j < W0; ++j) {
    float c = 0.f;
    if (live0 && j <= rr[0]) {
      R v = M(j, rr[0]) - M(j, D) * (M(rr[0], D) * inv_om);
      if (j == rr[0]) v += lp;
      c = (float)v;
    }
    L.a0[j] = c;
  }
  if constexpr (NS == 2) {
#pragma unroll
    for (int j = 0; j < D; ++j) {
      float c = 0.f;
      if (j <= rr[NS - 1]) {
        R v = M(j, rr[NS - 1]) - M(j, D) * (M(rr[NS - 1], D) * inv_om);
        if (j == rr[NS - 1]) v += lp;
        c = (float)v;
      }
      L.a1[j] = c;
    }
  }

  // Factorisation, with the forward substitution (L z' = z) as an extra column.
  __syncwarp();  // every lane is done with the staged moments; the buffer now holds L's rows
  chol_column<D, 0>(L, colbuf);
  // A prefix of at most d keys (rank-deficient centred covariance) goes to the exact pass
  // (lla_short.cu), which writes its output: every such row of fp32 inputs; so does any prefix
  // of at most kShortMaxKeys keys whose factorisation failed or whose |k . y| the readout could
  // not cancel against kbar . y (kShortY, kShortY32). Its y is zero and kbar[row][0]
  // kListedBits, which the readout skips.
  constexpr bool kF32 = std::is_same<TIn, float>::value;
  const int n_keys = (int)(row - bh * T) + 1;
  const bool short_prefix = n_keys <= kShortMaxKeys;
  auto list_short = [&]() {
    if (lane == 0) short_rows[atomicAdd(short_count, 1)] = (int)row;
    for (int a = lane; a < D; a += 32) {
      y_out[row * D + a] = 0.f;
      kbar_out[row * D + a] = a == 0 ? __uint_as_float(kListedBits) : 0.f;
    }
  };
  if ((kF32 && n_keys <= D) || (short_prefix && !L.ok)) {
    list_short();
    return;
  }
  if (!L.ok) {
    if (lane == 0) atomicOr(status, kStatusNumerical);
    const float qn = __int_as_float(0x7fc00000);
    for (int a = lane; a < D; a += 32) { y_out[row * D + a] = qn; kbar_out[row * D + a] = qn; }
    return;
  }
  // This lane's rows of L to shared memory (row-major, stride LS = 68 floats: conflict-free
  // 16-byte stores across the lanes of a phase).
  float* Lrows = g;
  if (live0) {
#pragma unroll
    for (int j = 0; j < W0; j += 4)
      *reinterpret_cast<float4*>(Lrows + rr[0] * C::LS + j) =
          make_float4(L.a0[j], L.a0[j + 1], L.a0[j + 2], L.a0[j + 3]);
  }
  if constexpr (NS == 2) {
#pragma unroll
    for (int j = 0; j < D; j += 4)
      *reinterpret_cast<float4*>(Lrows + rr[NS - 1] * C::LS + j) =
          make_float4(L.a1[j], L.a1[j + 1], L.a1[j + 2], L.a1[j + 3]);
  }
  __syncwarp();
  // Backward substitution L^T y = z'.
  float w0 = L.z[0], w1 = L.z[NS - 1], y0 = 0.f, y1 = 0.f;
  back_column<D, D - 1>(L, Lrows, w0, w1, y0, y1);
  if (short_prefix) {
    float ymax = fmaxf(live0 ? fabsf(y0) : 0.f, NS == 2 ? fabsf(y1) : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, o));
      kb1 += __shfl_xor_sync(0xffffffffu, kb1, o);
      ctr += __shfl_xor_sync(0xffffffffu, ctr, o);
    }
    // |kbar|_1 + sqrt(d tr(C_kk) / omega): the scale of the frame keys
    const float kscale = kb1 + sqrtf(fmaxf((float)D * ctr * (float)inv_om, 0.f));
    if (!(ymax * kscale <= (kF32 ? kShortY32 : kShortY))) {
      list_short();
      return;
    }
  }
  if (live0) {
    y_out[row * D + rr[0]] = y0;
    kbar_out[row * D + rr[0]] = kb[0];
  }
  if (NS == 2) {
    y_out[row * D + rr[NS - 1]] = y1;
    kbar_out[row * D + rr[NS - 1]] = kb[NS - 1];
  }
}

// ----------------------------------------------------------------------------- solve, tensor-core rows
// d = 64 with the tensor-core stage's moment rows (2208 floats in the order tc_slot() decodes;
// omega and the row max in their own arrays). A right-looking Cholesky per query, the right-hand
// side riding along as the forward substitution, two queries per warp: half-warp h solves query
// 2w + h, lane l of a half owning rows l, 31 - l, 32 + l and 63 - l of its matrix (four rows, a
// balanced share of the triangle). Shared memory bounds this factorisation -- every column is
// broadcast to the lanes that update the trailing rows -- so it is arranged for that:
//  * a column broadcast is one shared-memory load for both queries of a warp (each half reads its
//    own query's column); with one query per warp the broadcasts saturated the L1/shared data pipe
//    at half the rate per query;
//  * the moment row goes from global memory straight into the registers that hold the matrix (for
//    a fixed triangle row j the slots of (j, r), r > j, are consecutive). The loads and the
//    assembly are unpredicated: a lane's entries past its row's diagonal are padding, computed and
//    never read, and the odd diagonal entries (which sit outside the rows' runs) enter as a
//    correction added to the pivot;
//  * column k of the factor goes to shared memory once (column-major, packed: column c holds rows
//    4 floor(c / 4) .. 63), where the trailing update reads it and the backward substitution reads
//    four entries of a row per vector load;
//  * the trailing updates run as packed fp32 pairs (fma.rn.f32x2: the same single-rounded FMA on
//    two lanes of a 64-bit register pair), which halves their instruction count;
//  * the pivots' reciprocal square roots and the forward-substituted right-hand side are kept per
//    column in shared memory, the solution per row likewise, so that no lane has to pick out the
//    values of its own rows with compare-and-select; and the next pivot is formed from its owner's
//    registers, so the chain from pivot to pivot does not wait for the column's broadcast.
namespace stc {
constexpr int D = 64;

// Slot of (a, b) in a tensor-core moment row for b >= a + (a & 1) (the run of row a):
// run_base(a) + b. For every a and 0 <= b < 64, run_base(a) + b stays inside the row.
__host__ __device__ constexpr int run_base(int a) {
  const int t = a >> 1;
  const int rs = 65 * t - t * (t - 1) + ((a & 1) ? 33 - t : 0);
  return 2 * rs - (a + (a & 1));
}
static_assert(run_base(D - 1) + D - 1 < TC_ROW, "unpredicated loads stay inside the row");

// x -= s * c on a packed pair (x0, x1) with c = (c0, c1); ns = -s. One packed fp32 FMA (the same
// single-rounded FMA on both lanes of a 64-bit register pair).
__device__ __forceinline__ void fma2(float& x0, float& x1, float ns, float c0, float c1) {
  const float2 r = __ffma2_rn(make_float2(ns, ns), make_float2(c0, c1), make_float2(x0, x1));
  x0 = r.x;
  x1 = r.y;
}

// a[j] -= lik * cb[j] for K < j < N (ns = -lik); cb is 16-byte aligned.
template <int N, int K>
__device__ __forceinline__ void trail(float (&a)[N], float ns, const float* cb) {
  constexpr int j0 = K + 1;
  if constexpr (j0 < N) {
    if constexpr (j0 & 1) a[j0] = fmaf(ns, cb[j0], a[j0]);
    constexpr int je = (j0 + 1) & ~1;  // first even index >= j0
    constexpr int jq = (je + 3) & ~3;  // first multiple of 4 >= je
    if constexpr (je < jq && je < N) {
      const float2 c = *reinterpret_cast<const float2*>(cb + je);
      fma2(a[je], a[je + 1], ns, c.x, c.y);
    }
#pragma unroll
    for (int j = jq; j < N; j += 4) {
      const float4 c = *reinterpret_cast<const float4*>(cb + j);
      fma2(a[j], a[j + 1], ns, c.x, c.y);
      fma2(a[j + 2], a[j + 3], ns, c.z, c.w);
    }
  }
}

}  // namespace stc

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

namespace stc4 {
constexpr int D = 64;
constexpr int WARPS = 2;                   // warps per block, two queries each
constexpr int QPB = 2 * WARPS;             // queries per block
constexpr int LC = 2176;                   // packed factor
// factor; (z', 1/L_kk) per column; y; 4 floats of padding, so that the two queries of a warp
// start 16 bytes apart in the banks and their halves' column broadcasts do not conflict (the
// first of them holds the query's key scale for the short-prefix rule)
constexpr int Q_FLOATS = LC + 2 * D + D + 4;
constexpr size_t SMEM_BYTES = sizeof(float) * QPB * Q_FLOATS;

__host__ __device__ constexpr int col_start(int c) { return 4 * (c / 4); }
// first float of column c: the sum of the lengths 64 - col_start(k) of the columns k < c
__host__ __device__ constexpr int col_base(int c) {
  return 256 * (c / 4) - 8 * (c / 4) * (c / 4 - 1) + (c % 4) * (D - 4 * (c / 4));
}
static_assert(col_base(D) == LC, "packed factor size");
// the rows of lane group g (array g) span [16 g, 16 g + 15]; array g holds entries 0 .. 16 g + 15
__host__ __device__ constexpr int group_of(int r) { return r >> 4; }

using stc::fma2;
using stc::run_base;
using stc::trail;

struct Lane {
  float a0[16], a1[32], a2[48], a3[64];  // rows l, 31 - l, 32 + l, 63 - l (entries past the
                                         // diagonal are padding, computed and never read)
  float dg[4];  // diagonal corrections (the odd diagonals and lambda'), added to the pivot
  float z[4];   // right-hand sides, updated by the forward substitution until used
  int l;        // lane within the half-warp
  int hb;       // first lane of the half-warp
  bool ok;
};

template <int G, int J>
__device__ __forceinline__ float& at(Lane& L) {
  if constexpr (G == 0) return L.a0[J < 16 ? J : 0];
  else if constexpr (G == 1) return L.a1[J < 32 ? J : 0];
  else if constexpr (G == 2) return L.a2[J < 48 ? J : 0];
  else return L.a3[J];
}
// row of array G for lane l
__device__ __forceinline__ int row_of(int G, int l) {
  return G == 0 ? l : G == 1 ? 31 - l : G == 2 ? 32 + l : 63 - l;
}
template <int K>
__host__ __device__ constexpr int owner_of() {
  constexpr int g = group_of(K);
  return g == 0 ? K : g == 1 ? 31 - K : g == 2 ? K - 32 : 63 - K;
}

// Column K's entry of array G's row: scale it and store it into the packed column (rows at or
// past the column's first stored row; a row of array G can lie before it only when K is in the
// same 16-row group).
template <int G, int K>
__device__ __forceinline__ void scale_store(Lane& L, float inv, float* cb) {
  if constexpr (K < 16 * G + 16) {
    float& x = at<G, K>(L);
    x *= inv;
    constexpr int cs = col_start(K);
    if constexpr (16 * G >= cs) {
      cb[row_of(G, L.l)] = x;
    } else {
      const int r = row_of(G, L.l);
      if (r >= cs) cb[r] = x;
    }
  }
}
template <int G, int K>
__device__ __forceinline__ void update(Lane& L, const float* cb, float zk) {
  if constexpr (K < 16 * G + 15) {
    if constexpr (G == 0) trail<16, K>(L.a0, -L.a0[K], cb);
    else if constexpr (G == 1) trail<32, K>(L.a1, -L.a1[K], cb);
    else if constexpr (G == 2) trail<48, K>(L.a2, -L.a2[K], cb);
    else trail<64, K>(L.a3, -L.a3[K], cb);
  }
  if constexpr (K < 16 * G + 16) L.z[G] = fmaf(-at<G, K>(L), zk, L.z[G]);
}

template <int K>
__device__ __forceinline__ void column(Lane& L, float* Lc, float2* zi, float mine) {
  constexpr int g = group_of(K);
  const float piv = __shfl_sync(0xffffffffu, mine, L.hb + owner_of<K>());
  L.ok = L.ok && piv > 0.f;  // false for NaN too; a failed query is solved again by the repair pass
  const float inv = rsqrtf(piv);
  const float zk = __shfl_sync(0xffffffffu, L.z[g], L.hb + owner_of<K>()) * inv;
  if (L.l == 0) zi[K] = make_float2(zk, inv);
  float* cb = Lc + col_base(K) - col_start(K);  // cb[r] = entry (r, K)
  scale_store<0, K>(L, inv, cb);
  scale_store<1, K>(L, inv, cb);
  scale_store<2, K>(L, inv, cb);
  scale_store<3, K>(L, inv, cb);
  float next = 0.f;  // the next pivot from its owner's registers (row K + 1's entries K, K + 1)
  if constexpr (K + 1 < D) {
    constexpr int ng = group_of(K + 1);
    next = fmaf(-at<ng, K>(L), at<ng, K>(L), at<ng, K + 1>(L)) + L.dg[ng];
  }
  __syncwarp();
  update<0, K>(L, cb, zk);
  update<1, K>(L, cb, zk);
  update<2, K>(L, cb, zk);
  update<3, K>(L, cb, zk);
  if constexpr (K + 1 < D) column<K + 1>(L, Lc, zi, next);
}
}  // namespace stc4

// Output for the tensor-core readout: y as three exact bf16 parts (y = y1 + y2 + y3; 24
// significant bits, so that the readout's Y K^T keeps y's precision on the tensor cores), each
// part a row of 64 bf16 stored as 32 packed pairs, and cy = kbar . y. For the CUDA-core readout
// (value width other than 64) also y and kbar in fp32 (y_out, kbar_out; else null).
//
// PAGE: the page form of the same solve ("Parallax" blog, s.2 Canonical Formulation, with the
// query-centred z_j = k_j - q_i): rho* = Sigma^-1 mu with Sigma = sum p z z^T + lambda' I and
// mu = sum p z = s - omega q. In the moments at hand Sigma = S - s s^T / omega + mu mu^T / omega
// + lambda' I: the centred matrix plus one rank-one term. The output is then rho* in place of y
// and cy = q . rho*, so that the readout's t_ij = k_j . rho* - cy is the page's z_ij . rho*.
template <bool PAGE>
__global__ void __launch_bounds__(stc4::WARPS * 32, 4)
solve_tc_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ kref,
                 const float* __restrict__ mom, const float* __restrict__ omega,
                 const float* __restrict__ mrow, long long rows, int T, float lam,
                 uint32_t* __restrict__ ytc, float* __restrict__ cy_out,
                 float* __restrict__ y_out, float* __restrict__ kbar_out, int* __restrict__ rep,
                 int* __restrict__ short_count, int* __restrict__ short_rows,
                 int* __restrict__ status) {
  using namespace stc4;
  extern __shared__ float4 smem4[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4;
  const long long row_req = (long long)blockIdx.x * QPB + 2 * warp + half;
  const bool live = row_req < rows;
  const long long row = live ? row_req : rows - 1;  // a half past the end mirrors the last row
  if (__all_sync(0xffffffffu, !live)) return;        // whole warp past the end
  float* Lc = reinterpret_cast<float*>(smem4) + (2 * warp + half) * Q_FLOATS;
  float2* zi = reinterpret_cast<float2*>(Lc + LC);
  float* ys = Lc + LC + 2 * D;
  float* sv = reinterpret_cast<float*>(zi);  // before the factorisation: s, then (page) mu
  float* muv = sv + D;
  const float* g = mom + row * TC_ROW;

  Lane L;
  L.l = lane & 15;
  L.hb = lane & 16;
  L.ok = true;
  const int r[4] = {L.l, 31 - L.l, 32 + L.l, 63 - L.l};
#pragma unroll
  for (int j = 0; j < 16; ++j) L.a0[j] = __ldcs(g + run_base(j) + r[0]);
#pragma unroll
  for (int j = 0; j < 32; ++j) L.a1[j] = __ldcs(g + run_base(j) + r[1]);
#pragma unroll
  for (int j = 0; j < 48; ++j) L.a2[j] = __ldcs(g + run_base(j) + r[2]);
#pragma unroll
  for (int j = 0; j < 64; ++j) L.a3[j] = __ldcs(g + run_base(j) + r[3]);
  const float om = omega[row];
  const float lp = fminf(fmaxf(expf(logf(lam) - mrow[row]), FLT_MIN), FLT_MAX);
  const int bh = (int)row / T;  // rows < 2^31
  float kb[4], qa[4], mu[4];
  const float inv_om = 1.f / om;
  float kb1 = 0.f, ctr = 0.f;  // |kbar|_1 and tr(C_kk), for the key scale of the short-prefix rule
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float d = __ldcs(g + tc_slot(r[i], r[i])), x = __ldcs(g + run_base(r[i]) + r[i]);
    const float s = __ldcs(g + run_base(r[i]) + D);
    kb1 += fabsf(s * inv_om);
    ctr += fmaf(-s, s * inv_om, d);
    L.dg[i] = (d - x) + lp;  // x is d for even rows, the zero slot before the run for odd rows
    qa[i] = ldf(q, row * D + r[i]) - kref[bh * D + r[i]];
    mu[i] = fmaf(-om, qa[i], s);  // page form: mu = s - omega q
    kb[i] = s * inv_om;
    sv[r[i]] = s;
    if (PAGE) muv[r[i]] = mu[i];
    L.z[i] = PAGE ? mu[i] : qa[i] - kb[i];
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    kb1 += __shfl_xor_sync(0xffffffffu, kb1, o);
    ctr += __shfl_xor_sync(0xffffffffu, ctr, o);
  }
  // |kbar|_1 + sqrt(d tr(C_kk) / omega), at least |kbar|_1 + sum_a sqrt(C_aa / omega) (equal for
  // isotropic keys); parked in the query's padding until the end
  if (L.l == 0) Lc[LC + 3 * D] = kb1 + sqrtf(fmaxf(D * ctr * inv_om, 0.f));
  __syncwarp();
  // C_kk = S - s s^T / omega (page form: + mu mu^T / omega) on every array entry
#pragma unroll
  for (int j = 0; j < D; j += 4) {
    const float4 s4 = *reinterpret_cast<const float4*>(sv + j);
    const float sj[4] = {s4.x, s4.y, s4.z, s4.w};
    float mj[4] = {0.f, 0.f, 0.f, 0.f};
    if (PAGE) {
      const float4 m4 = *reinterpret_cast<const float4*>(muv + j);
      mj[0] = m4.x; mj[1] = m4.y; mj[2] = m4.z; mj[3] = m4.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = j + u;
      auto upd = [&](float& a, int i) {
        float v = fmaf(-sj[u], kb[i], a);
        if (PAGE) v = fmaf(mj[u], mu[i] * inv_om, v);
        a = v;
      };
      if (jj < 16) upd(L.a0[jj & 15], 0);
      if (jj < 32) upd(L.a1[jj & 31], 1);
      if (jj < 48) upd(L.a2[jj < 48 ? jj : 0], 2);
      upd(L.a3[jj], 3);
    }
  }
  __syncwarp();  // s and mu are read; the area now takes (z', 1/L_kk)
  stc4::column<0>(L, Lc, zi, L.a0[0] + L.dg[0]);
  const unsigned fails = __ballot_sync(0xffffffffu, !L.ok);
  const bool my_fail = ((fails >> L.hb) & 0xFFFFu) != 0;
  __syncwarp();
  // Backward substitution L^T y = z', four rows at a time from the bottom; each lane reads the
  // factor entries L[KB..KB+3][r] of its rows r (column r of the packed factor).
  float w[4], iv[4];
  const float* lcr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = zi[r[i]];
    w[i] = t.x;
    iv[i] = t.y;
    lcr[i] = Lc + col_base(r[i]) - col_start(r[i]);
  }
#pragma unroll
  for (int KB = D - 4; KB >= 0; KB -= 4) {
    float e[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 c = *reinterpret_cast<const float4*>(lcr[i] + KB);
      e[i][0] = c.x; e[i][1] = c.y; e[i][2] = c.z; e[i][3] = c.w;
    }
#pragma unroll
    for (int t = 3; t >= 0; --t) {
      const int K = KB + t;
      const int gk = K >> 4;
      const int owner = gk == 0 ? K : gk == 1 ? 31 - K : gk == 2 ? K - 32 : 63 - K;
      const float yk = __shfl_sync(0xffffffffu, w[gk] * iv[gk], L.hb + owner);
      if (L.l == 0) ys[K] = yk;
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = fmaf(-e[i][t], yk, w[i]);
    }
  }
  __syncwarp();
  uint32_t* yrow = ytc + row * 3 * (D / 2);
  // A prefix of at most d keys whose factorisation failed, or whose |k . y| the readout could
  // not cancel against kbar . y (kShortY), goes to the exact pass (lla_short.cu), which writes
  // its output; its y is zero and its cy (kbar[row][0] for a CUDA-core readout) kListedBits.
  bool short_row = false;
  if ((int)(row - (long long)bh * T) + 1 <= D) {
    const float4 t4 = *reinterpret_cast<const float4*>(ys + 4 * L.l);  // y[4l .. 4l + 3]
    float ymax = fmaxf(fmaxf(fabsf(t4.x), fabsf(t4.y)), fmaxf(fabsf(t4.z), fabsf(t4.w)));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, o));
    short_row = my_fail || !(ymax * Lc[LC + 3 * D] <= kShortY);
  }
  if (short_row) {
    if (!live) return;
    if (L.l == 0) {
      short_rows[atomicAdd(short_count, 1)] = (int)row;
      cy_out[row] = __uint_as_float(kListedBits);
    }
    reinterpret_cast<uint2*>(yrow)[L.l] = make_uint2(0u, 0u);
    reinterpret_cast<uint2*>(yrow + D / 2)[L.l] = make_uint2(0u, 0u);
    reinterpret_cast<uint2*>(yrow + D)[L.l] = make_uint2(0u, 0u);
    if (y_out)
      for (int i = 0; i < 4; ++i) {
        y_out[row * D + r[i]] = 0.f;
        kbar_out[row * D + r[i]] = r[i] == 0 ? __uint_as_float(kListedBits) : 0.f;
      }
    return;
  }
  if (my_fail) {
    // A non-positive pivot: the query goes to the precise repair pass (repair_kernel), which
    // overwrites its y; if the repair list is full, the query is NaN.
    if (live && L.l == 0) {
      const int slot = atomicAdd(rep, 1);
      if (slot < kMaxRepairRows) {
        rep[1 + slot] = (int)row;
      } else {
        atomicOr(status, kStatusNumerical);
        cy_out[row] = __int_as_float(0x7fc00000);
        for (int p = 0; p < 3 * (D / 2); ++p) yrow[p] = 0x7FC07FC0u;  // bf16 NaN pairs
        if (y_out)
          for (int a = 0; a < D; ++a)
            y_out[row * D + a] = kbar_out[row * D + a] = __int_as_float(0x7fc00000);
      }
    }
    return;
  }
  // Lane l of a half writes elements 4l .. 4l + 3 of each part (two packed pairs).
  const float4 y4 = *reinterpret_cast<const float4*>(ys + 4 * L.l);
  const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
  uint32_t p1[2], p2[2], p3[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float ya = yv[2 * h], yb = yv[2 * h + 1];
    p1[h] = pack_bf16(ya, yb);
    const float ra = ya - __uint_as_float(p1[h] << 16), rb = yb - __uint_as_float(p1[h] & 0xFFFF0000u);
    p2[h] = pack_bf16(ra, rb);
    p3[h] = pack_bf16(ra - __uint_as_float(p2[h] << 16), rb - __uint_as_float(p2[h] & 0xFFFF0000u));
  }
  float c = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) c = fmaf(PAGE ? qa[i] : kb[i], ys[r[i]], c);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (!live) return;
  reinterpret_cast<uint2*>(yrow)[L.l] = make_uint2(p1[0], p1[1]);
  reinterpret_cast<uint2*>(yrow + D / 2)[L.l] = make_uint2(p2[0], p2[1]);
  reinterpret_cast<uint2*>(yrow + D)[L.l] = make_uint2(p3[0], p3[1]);
  if (L.l == 0) cy_out[row] = c;
  if (y_out) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y_out[row * D + r[i]] = ys[r[i]];
      kbar_out[row * D + r[i]] = kb[i];
    }
  }
}

// ----------------------------------------------------------------------------- precise repair
// Rows whose tensor-core factorisation met a non-positive pivot are solved again here, exactly
// enough for any conditioning the fp64 factorisation can handle: the same weighted problem (the
// bf16 weights of the weight images, the same bf16 keys in the head's frame, so that the readout
// stays consistent with it) with the sums formed without rounding error worth the name. Each
// term p_j x_a x_b is a product of three bf16 values, 24 significant bits, hence exact in fp32; the
// terms are summed in compensated fp32 pairs (TwoSum), centred and factored in fp64. One CTA per
// row (the CTAs stride over the list); nothing runs when the list is empty.
namespace rep {
constexpr int D = 64;
constexpr int NE = 1 + D + D * (D + 1) / 2;  // omega, s, upper triangle of S
constexpr int NT = 256;
constexpr int EPT = (NE + NT - 1) / NT;      // entries per thread
constexpr int KC = 64;                       // keys per staged chunk
}  // namespace rep
constexpr int kRepairGrid = 152;

template <bool PAGE>
__global__ void __launch_bounds__(rep::NT)
repair_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ ksh,
              const float* __restrict__ kref, const uint8_t* __restrict__ pimg,
              const float* __restrict__ mrow, const int* __restrict__ rep, int T, float lam,
              uint32_t* __restrict__ ytc, float* __restrict__ cy_out, float* __restrict__ y_out,
              float* __restrict__ kbar_out, int* __restrict__ status) {
  using namespace rep;
  // the staged key chunk during the sums, then the fp64 system (the two are never live together)
  __shared__ __align__(16) double buf[D * (D + 1)];
  __shared__ float ps[KC];
  __shared__ double vs[D], zs[D];
  __shared__ int fail;
  float (*ks)[D + 1] = reinterpret_cast<float (*)[D + 1]>(buf);
  double (*C)[D + 1] = reinterpret_cast<double (*)[D + 1]>(buf);
  static_assert(sizeof(float) * KC * (D + 1) <= sizeof(double) * D * (D + 1), "buffer reuse");
  const int tid = threadIdx.x;
  const int count = min(rep[0], kMaxRepairRows);

  // this thread's entries: e = 0 omega, 1..D the s_a, then S_ab (a <= b) row by row
  int ea[EPT], eb[EPT];
#pragma unroll
  for (int m = 0; m < EPT; ++m) {
    int e = tid + m * NT, a = -1, b = -1;
    if (e >= NE) { a = -2; }
    else if (e >= 1 && e <= D) { a = e - 1; }
    else if (e > D) {
      int t = e - 1 - D;
      a = 0;
      while (t >= D - a) { t -= D - a; ++a; }
      b = a + t;
    }
    ea[m] = a;
    eb[m] = b;
  }

  for (int slot = blockIdx.x; slot < count; slot += gridDim.x) {
    const long long row = rep[1 + slot];
    const long long bh = row / T;
    const int i = (int)(row % T);
    const int ptile = i / 256, rank = (i % 256) / 128, r = i % 128;
    const uint8_t* img0 = pimg + pscr::first_block(bh, T, ptile, rank) * pscr::kBlockBytes;
    float hi[EPT], lo[EPT];
#pragma unroll
    for (int m = 0; m < EPT; ++m) hi[m] = lo[m] = 0.f;
    for (int j0 = 0; j0 <= i; j0 += KC) {
      __syncthreads();
      for (int e = tid; e < KC * D; e += NT) {
        const int jj = e / D, a = e % D, j = j0 + jj;
        ks[jj][a] = j <= i ? __bfloat162float(ksh[(bh * T + j) * D + a]) : 0.f;
      }
      for (int jj = tid; jj < KC; jj += NT) {
        const int j = j0 + jj;
        float p = 0.f;
        if (j <= i) {
          const int b = j / pscr::kKeys, c = j % pscr::kKeys;
          const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(
              img0 + (size_t)b * pscr::kBlockBytes + (c / 8) * 2048 + r * 16) + (c % 8);
          p = __bfloat162float(*w);
        }
        ps[jj] = p;
      }
      __syncthreads();
      const int jn = min(KC, i + 1 - j0);
      for (int jj = 0; jj < jn; ++jj) {
        const float p = ps[jj];
#pragma unroll
        for (int m = 0; m < EPT; ++m) {
          if (ea[m] < -1) continue;
          float x = p;                                  // exact: three bf16 factors at most
          if (ea[m] >= 0) x *= ks[jj][ea[m]];
          if (eb[m] >= 0) x *= ks[jj][eb[m]];
          const float t = hi[m] + x, z = t - hi[m];     // TwoSum into (hi, lo)
          lo[m] += (hi[m] - (t - z)) + (x - z);
          hi[m] = t;
        }
      }
    }
    __syncthreads();
    // the sums into the fp64 system: C[a][b] = S_ab (a <= b), C[a][D] = s_a, C[0][0..] etc.
    double om_local = 0.0;
#pragma unroll
    for (int m = 0; m < EPT; ++m) {
      const double v = (double)hi[m] + (double)lo[m];
      if (ea[m] == -1) vs[0] = v;  // omega kept apart in vs[0] until zs is formed
      else if (ea[m] >= 0 && eb[m] < 0) C[ea[m]][D] = v;
      else if (ea[m] >= 0) C[ea[m]][eb[m]] = v;
      (void)om_local;
    }
    __syncthreads();
    const double om = vs[0];
    __syncthreads();
    const double lp = fmin(fmax((double)lam * exp(-(double)mrow[row]), (double)FLT_MIN), (double)FLT_MAX);
    if (tid < D) {
      const double qa = (double)__bfloat162float(q[row * D + tid]) - (double)kref[bh * D + tid];
      const double sa = C[tid][D];
      vs[tid] = sa / om;                               // kbar (head frame)
      zs[tid] = PAGE ? sa - om * qa : qa - sa / om;    // page: mu = s - omega q; centred: q - kbar
    }
    __syncthreads();
    // centred system (page form: plus mu mu^T / omega), lower triangle, ridge on the diagonal
    for (int e = tid; e < D * D; e += NT) {
      const int a = e / D, b = e % D;
      if (b > a) continue;
      double v = C[b][a] - C[a][D] * C[b][D] / om;  // S stored at [min][max]
      if (PAGE) v += zs[a] * zs[b] / om;
      if (a == b) v += lp;
      C[a][b] = v;
    }
    if (tid == 0) fail = 0;
    __syncthreads();
    // Cholesky C = L L^T in place (lower triangle), column by column
    for (int kk = 0; kk < D; ++kk) {
      if (tid == 0) {
        const double d = C[kk][kk];
        if (!(d > 0.0)) fail = 1;
        C[kk][kk] = d > 0.0 ? sqrt(d) : 1.0;
      }
      __syncthreads();
      const double lkk = C[kk][kk];
      for (int a = kk + 1 + tid; a < D; a += NT) C[a][kk] /= lkk;
      __syncthreads();
      for (int e = tid; e < D * D; e += NT) {
        const int a = e / D, b = e % D;
        if (a > kk && b > kk && b <= a) C[a][b] -= C[a][kk] * C[b][kk];
      }
      __syncthreads();
    }
    if (tid < 32) {
      // forward and backward substitution (one warp; lane t owns rows t and t + 32)
      double w0 = zs[tid], w1 = zs[tid + 32];
      for (int kk = 0; kk < D; ++kk) {
        const double own = kk < 32 ? w0 : w1;
        const double xk = __shfl_sync(0xffffffffu, own, kk & 31) / C[kk][kk];
        if (tid == (kk & 31)) { if (kk < 32) w0 = xk; else w1 = xk; }
        if (tid > kk) w0 -= C[tid][kk] * xk;
        if (tid + 32 > kk) w1 -= C[tid + 32][kk] * xk;
      }
      for (int kk = D - 1; kk >= 0; --kk) {
        const double own = kk < 32 ? w0 : w1;
        const double yk = __shfl_sync(0xffffffffu, own, kk & 31) / C[kk][kk];
        if (tid == (kk & 31)) { if (kk < 32) w0 = yk; else w1 = yk; }
        if (tid < kk) w0 -= C[kk][tid] * yk;
        if (tid + 32 < kk) w1 -= C[kk][tid + 32] * yk;
      }
      zs[tid] = w0;       // y
      zs[tid + 32] = w1;
    }
    __syncthreads();
    uint32_t* yrow = ytc + row * 3 * (D / 2);
    if (fail) {
      if (tid == 0) {
        atomicOr(status, kStatusNumerical);
        cy_out[row] = __int_as_float(0x7fc00000);
      }
      if (tid < 3 * (D / 2)) yrow[tid] = 0x7FC07FC0u;  // bf16 NaN pairs
      if (y_out && tid < D) {
        y_out[row * D + tid] = __int_as_float(0x7fc00000);
        kbar_out[row * D + tid] = __int_as_float(0x7fc00000);
      }
      continue;
    }
    if (tid < 32) {
      // y as three bf16 parts, lane l writing elements 2l and 2l + 1 of each; cy = kbar . y
      // (page form: q . rho*, q in the head's frame)
      const float ya = (float)zs[2 * tid], yb = (float)zs[2 * tid + 1];
      const uint32_t p1 = pack_bf16(ya, yb);
      const float ra = ya - __uint_as_float(p1 << 16), rb = yb - __uint_as_float(p1 & 0xFFFF0000u);
      const uint32_t p2 = pack_bf16(ra, rb);
      const uint32_t p3 =
          pack_bf16(ra - __uint_as_float(p2 << 16), rb - __uint_as_float(p2 & 0xFFFF0000u));
      yrow[tid] = p1;
      yrow[D / 2 + tid] = p2;
      yrow[D + tid] = p3;
      double c = 0.0;
      for (int a = tid; a < D; a += 32) {
        const double qa = (double)__bfloat162float(q[row * D + a]) - (double)kref[bh * D + a];
        c += (PAGE ? qa : vs[a]) * zs[a];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (tid == 0) cy_out[row] = (float)c;
    }
    if (y_out && tid < D) {
      y_out[row * D + tid] = (float)zs[tid];
      kbar_out[row * D + tid] = (float)vs[tid];
    }
  }
}

cudaError_t launch_solve_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  const long long rows = a.rows();
  const long long blocks = (rows + stc4::QPB - 1) / stc4::QPB;
  auto kern = ws.form == kFormPage ? solve_tc_kernel<true> : solve_tc_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)stc4::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)blocks, stc4::WARPS * 32, stc4::SMEM_BYTES, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), ws.kref, ws.mom, ws.omega, ws.m, rows, a.T, a.lam,
      ws.ytc, ws.cy,
      a.dv == 64 ? nullptr : ws.y, a.dv == 64 ? nullptr : ws.kbar, ws.rep, ws.short_count,
      ws.short_rows, ws.status);
  count_launch();
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  auto rk = ws.form == kFormPage ? repair_kernel<true> : repair_kernel<false>;
  rk<<<kRepairGrid, rep::NT, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), ws.ksh, ws.kref, static_cast<const uint8_t*>(ws.pscr),
      ws.m, ws.rep, a.T, a.lam, ws.ytc, ws.cy, a.dv == 64 ? nullptr : ws.y,
      a.dv == 64 ? nullptr : ws.kbar, ws.status);
  count_launch();
  return cudaGetLastError();
}

template <typename TIn, int D, bool PRECISE, int FMT = 0>
cudaError_t launch_solve_t(const Args& a, const Workspace& ws, cudaStream_t s) {
  const size_t smem = sizeof(float) * kWarpsPerBlock * SolveCfg<D, PRECISE, FMT>::WARP_FLOATS;
  auto kern = solve_kernel<TIn, D, PRECISE, FMT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long rows = a.rows();
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  kern<<<(unsigned)blocks, kWarpsPerBlock * 32, smem, s>>>(
      static_cast<const TIn*>(a.q), ws.kmean, ws.mom, ws.mom_lo, ws.omega, ws.m, a.T, rows, a.lam,
      ws.y, ws.kbar, ws.short_count, ws.short_rows, ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const Args& a, const Workspace& ws, cudaStream_t s) {
  if (ws.path == kPathTensorCore) {  // the keys in the head's frame (see key_stats_kernel)
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
    key_stats_kernel<<<dim3((unsigned)a.BH(), kKeyStatChunks), 256, 0, s>>>(k, a.T, ws.kstat,
                                                                          ws.rep, ws.short_count);
    count_launch();
    shift_keys_kernel<<<dim3((unsigned)a.BH(), kShiftChunks), 256, 0, s>>>(k, a.T, ws.kstat,
                                                                           ws.kref, ws.ksh);
    count_launch();
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  // The tensor-core readout (dv = 64) forms every value term from centred weights and needs no
  // value reference point; the CG strategy keeps its keys unshifted.
  if (ws.path != kPathCudaCore && a.dv == 64) return cudaSuccess;
  const dim3 grid((unsigned)a.BH(), 2);
  if (a.dtype == LLA_F32)
    mean_kernel<float><<<grid, 256, 256 * sizeof(float), s>>>(
        static_cast<const float*>(a.k), static_cast<const float*>(a.v), a.T, a.d, a.dv, ws.kmean,
        ws.vmean, ws.path == kPathTensorCore, ws.short_count);
  else
    mean_kernel<__nv_bfloat16><<<grid, 256, 256 * sizeof(float), s>>>(
        static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.v), a.T, a.d,
        a.dv, ws.kmean, ws.vmean, ws.path == kPathTensorCore, ws.short_count);
  count_launch();
  cudaError_t err = cudaGetLastError();
  // The CUDA-core readout after the tensor-core solve (dv != 64) works in the solve's key frame.
  if (err == cudaSuccess && ws.path == kPathTensorCore)
    err = cudaMemcpyAsync(ws.kmean, ws.kref, a.BH() * a.d * sizeof(float),
                          cudaMemcpyDeviceToDevice, s);
  return err;
}

cudaError_t launch_solve(const Args& a, const Workspace& ws, cudaStream_t s) {
  if (ws.path == kPathTensorCore) return launch_solve_tc(a, ws, s);
  const bool f32 = a.dtype == LLA_F32;
  switch (a.d) {
    case 16: return f32 ? launch_solve_t<float, 16, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 16, false>(a, ws, s);
    case 32: return f32 ? launch_solve_t<float, 32, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 32, false>(a, ws, s);
    case 64: return f32 ? launch_solve_t<float, 64, true>(a, ws, s) : launch_solve_t<__nv_bfloat16, 64, false>(a, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lla
