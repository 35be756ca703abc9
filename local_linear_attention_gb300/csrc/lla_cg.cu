// Matrix-free conjugate-gradient strategy for the ridge systems of the causal LLA forward
// (bf16 inputs, d = dv = 64; selected per call with lla_options.path = LLA_PATH_CG).
//
// The closed form o_i = vbar_i + C_vk y_i needs y_i = (C_kk + lambda' I)^-1 (q_i - kbar_i) per
// query. The dense strategy accumulates C_kk (d x d per query) on the tensor cores and factors it.
// This one solves the same system by conjugate gradients, as the "Parallax" blog (s.2
// "Difficulties in Scaling LLA") describes exact LLA being computed: every product C_kk p_i is one
// streaming pass over the causal prefix, C_kk p = sum_j w_ij ((k_j - kbar_i) . p_i) k_j, which is
// the readout kernel with V := K, y := p and only its covariance branch kept (matvec mode). Each
// query row iterates until its residual falls below rel_tol times the initial one (or the
// iteration cap), and a query tile whose rows have all converged is skipped by later passes, so a
// tile costs as many passes as its slowest row needs.
//
// Kernels here: the per-row CG start (r = p = q - kbar, x = 0) and update (alpha, x, r, beta, p)
// and the hand-over of x to the readout (three exact bf16 parts and kbar . x), one CTA per query
// tile (one warp per query row, lane l holding dimensions 2l and 2l + 1). The state (r, p, A p,
// r.r) lives in the moments region of the workspace, which this strategy does not otherwise use.
#include <cfloat>

#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int D = 64;
constexpr int TILE = 128;    // query rows per tile (the readout's tile)
constexpr int NWARP = 32;    // warps per CTA: a tile is handled in TILE / NWARP row rounds
constexpr int kCheckEvery = 8;  // iterations between the host's tests for convergence

struct CgState {
  float* r;          // [R, 64] residual
  float* p;          // [R, 64] search direction
  float* ap;         // [R, 64] C_kk p from the matvec pass
  float* rr;         // [R] r . r
  float* rr0;        // [R] initial r . r
  int* row_active;   // [R] row not yet converged
  int* tile_active;  // [BH * ntiles] some row of the tile not yet converged
  int* counts;       // [max_iters + 1] active tiles after each iteration
};

CgState carve_cg(const Args& a, const Workspace& ws) {
  const size_t R = (size_t)a.rows();
  const int ntiles = (a.T + TILE - 1) / TILE;
  CgState st;
  float* f = ws.mom;
  st.r = f;
  st.p = f + R * D;
  st.ap = f + 2 * R * D;
  st.rr = f + 3 * R * D;
  st.rr0 = st.rr + R;
  int* n = reinterpret_cast<int*>(st.rr0 + R);
  st.row_active = n;
  st.tile_active = n + R;
  st.counts = st.tile_active + (size_t)a.BH() * ntiles;
  return st;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Writes (a, b) = elements 2l, 2l + 1 of a vector as three exact bf16 parts of row `row`.
__device__ __forceinline__ void put_parts(uint32_t* ytc, long long row, int lane, float a, float b) {
  const uint32_t p1 = pack_bf16(a, b);
  const float ra = a - __uint_as_float(p1 << 16), rb = b - __uint_as_float(p1 & 0xFFFF0000u);
  const uint32_t p2 = pack_bf16(ra, rb);
  const uint32_t p3 =
      pack_bf16(ra - __uint_as_float(p2 << 16), rb - __uint_as_float(p2 & 0xFFFF0000u));
  uint32_t* y = ytc + row * 3 * (D / 2);
  y[lane] = p1;
  y[D / 2 + lane] = p2;
  y[D + lane] = p3;
}

// y := 0 for the kbar pass: zero parts and cy = 0.
__global__ void cg_zero_kernel(uint32_t* __restrict__ ytc, float* __restrict__ cy, long long rows) {
  const long long n = rows * 3 * (D / 2);
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x) {
    ytc[t] = 0u;
    if (t < rows) cy[t] = 0.f;
  }
}

// Start: x = 0, r = p = q - kbar, rr = rr0 = r . r; the readout's y := p.
__global__ void __launch_bounds__(NWARP * 32)
cg_init_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ kbar, int T, int BH,
               int max_iters, float* __restrict__ x, CgState st, uint32_t* __restrict__ ytc,
               float* __restrict__ cy) {
  __shared__ int any;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (T + TILE - 1) / TILE;
  const long long bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  if (threadIdx.x == 0) any = 0;
  if (blockIdx.x == 0)
    for (int t = threadIdx.x; t <= max_iters; t += blockDim.x) st.counts[t] = 0;
  __syncthreads();
  for (int rr = warp; rr < TILE; rr += NWARP) {
    const int i = tile * TILE + rr;
    if (i >= T) break;
    const long long row = bh * T + i;
    const uint32_t qw = reinterpret_cast<const uint32_t*>(q + row * D)[lane];
    const float2 kb = reinterpret_cast<const float2*>(kbar + row * D)[lane];
    const float r0 = __uint_as_float(qw << 16) - kb.x, r1 = __uint_as_float(qw & 0xFFFF0000u) - kb.y;
    const float rrv = warp_sum(r0 * r0 + r1 * r1);
    // A non-finite start (a non-finite query or key in the prefix) makes x NaN at once: the row
    // comes out NaN and the hand-over reports it. rr = 0 means y = 0 is exact.
    const bool bad = !(rrv == rrv) || rrv == INFINITY;
    const bool act = rrv > 0.f && !bad;
    const float xs = bad ? __int_as_float(0x7fc00000) : 0.f;
    const float s0 = act ? r0 : 0.f, s1 = act ? r1 : 0.f;
    reinterpret_cast<float2*>(x + row * D)[lane] = make_float2(xs, xs);
    reinterpret_cast<float2*>(st.r + row * D)[lane] = make_float2(r0, r1);
    reinterpret_cast<float2*>(st.p + row * D)[lane] = make_float2(s0, s1);
    const float c = warp_sum(kb.x * s0 + kb.y * s1);
    put_parts(ytc, row, lane, s0, s1);
    if (lane == 0) {
      st.rr[row] = rrv;
      st.rr0[row] = rrv;
      st.row_active[row] = act ? 1 : 0;
      cy[row] = c;
      if (act) any = 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) st.tile_active[bh * ntiles + tile] = any;
}

// One CG step per active row from ap = C_kk p (the matvec pass): with A = C_kk + lambda' I,
// alpha = rr / p.Ap, x += alpha p, r -= alpha Ap, then either the row has converged
// (r.r <= tol2 * rr0: p := 0, so later passes leave it alone) or beta = r.r / rr, p = r + beta p.
__global__ void __launch_bounds__(NWARP * 32)
cg_update_kernel(const float* __restrict__ kbar, const float* __restrict__ mrow, int T, int BH,
                 float lam, float tol2, int it, float* __restrict__ x, CgState st,
                 uint32_t* __restrict__ ytc, float* __restrict__ cy) {
  __shared__ int any;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (T + TILE - 1) / TILE;
  const long long bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  if (!st.tile_active[bh * ntiles + tile]) return;  // the whole CTA: nothing left to do
  if (threadIdx.x == 0) any = 0;
  __syncthreads();
  for (int rr = warp; rr < TILE; rr += NWARP) {
    const int i = tile * TILE + rr;
    if (i >= T) break;
    const long long row = bh * T + i;
    if (!st.row_active[row]) continue;
    double lpd = (double)lam * exp(-(double)mrow[row]);  // ridge scaled by exp(-m)
    lpd = fmin(fmax(lpd, (double)FLT_MIN), (double)FLT_MAX);
    const float lp = (float)lpd;
    const float2 p = reinterpret_cast<const float2*>(st.p + row * D)[lane];
    const float2 a = reinterpret_cast<const float2*>(st.ap + row * D)[lane];
    const float ap0 = fmaf(lp, p.x, a.x), ap1 = fmaf(lp, p.y, a.y);
    const float pap = warp_sum(p.x * ap0 + p.y * ap1);
    const float rrv = st.rr[row];
    float2 xv = reinterpret_cast<const float2*>(x + row * D)[lane];
    float2 rv = reinterpret_cast<const float2*>(st.r + row * D)[lane];
    float rrn = rrv;
    bool done;
    if (pap > 0.f) {
      const float alpha = rrv / pap;
      xv.x = fmaf(alpha, p.x, xv.x);
      xv.y = fmaf(alpha, p.y, xv.y);
      rv.x = fmaf(-alpha, ap0, rv.x);
      rv.y = fmaf(-alpha, ap1, rv.y);
      rrn = warp_sum(rv.x * rv.x + rv.y * rv.y);
      done = rrn <= tol2 * st.rr0[row] || !(rrn == rrn);
      if (!(rrn == rrn)) xv.x = xv.y = __int_as_float(0x7fc00000);
    } else {
      // Breakdown: p.Ap not positive (A is positive definite, so only once p has lost all
      // precision) or not finite (then x is made NaN, and the hand-over reports it).
      done = true;
      if (!(pap == pap)) xv.x = xv.y = __int_as_float(0x7fc00000);
    }
    reinterpret_cast<float2*>(x + row * D)[lane] = xv;
    reinterpret_cast<float2*>(st.r + row * D)[lane] = rv;
    float n0 = 0.f, n1 = 0.f;
    if (!done) {
      const float beta = rrn / rrv;
      n0 = fmaf(beta, p.x, rv.x);
      n1 = fmaf(beta, p.y, rv.y);
    }
    reinterpret_cast<float2*>(st.p + row * D)[lane] = make_float2(n0, n1);
    const float2 kb = reinterpret_cast<const float2*>(kbar + row * D)[lane];
    const float c = warp_sum(kb.x * n0 + kb.y * n1);
    put_parts(ytc, row, lane, n0, n1);
    if (lane == 0) {
      st.rr[row] = rrn;
      st.row_active[row] = done ? 0 : 1;
      cy[row] = c;
      if (!done) any = 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    st.tile_active[bh * ntiles + tile] = any;
    if (any) atomicAdd(&st.counts[it], 1);
  }
}

// Hand-over: y := x for the readout (three exact bf16 parts, cy = kbar . x); a non-finite x is
// reported as LLA_ERR_NUMERICAL (its row comes out non-finite).
__global__ void __launch_bounds__(NWARP * 32)
cg_final_kernel(const float* __restrict__ kbar, int T, const float* __restrict__ x,
                uint32_t* __restrict__ ytc, float* __restrict__ cy, int* __restrict__ status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (T + TILE - 1) / TILE;
  const long long bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  for (int rr = warp; rr < TILE; rr += NWARP) {
    const int i = tile * TILE + rr;
    if (i >= T) break;
    const long long row = bh * T + i;
    const float2 xv = reinterpret_cast<const float2*>(x + row * D)[lane];
    const float2 kb = reinterpret_cast<const float2*>(kbar + row * D)[lane];
    const float c = warp_sum(kb.x * xv.x + kb.y * xv.y);
    put_parts(ytc, row, lane, xv.x, xv.y);
    const bool bad = __any_sync(0xffffffffu, !isfinite(xv.x) || !isfinite(xv.y));
    if (lane == 0) {
      cy[row] = c;
      if (bad) atomicOr(status, kStatusNumerical);
    }
  }
}

}  // namespace

size_t cg_state_bytes(const Args& a) {
  const size_t R = (size_t)a.rows();
  const int ntiles = (a.T + TILE - 1) / TILE;
  return sizeof(float) * (3 * R * D + 2 * R) + sizeof(int) * (R + (size_t)a.BH() * ntiles + 1025);
}

// The "solve" stage of the CG strategy: kbar (one readout pass with y = 0 and V := K), then CG
// iterations (matvec pass + update) until no tile is active or max_iters passes have run, then the
// hand-over of x. Synchronises the stream every kCheckEvery iterations to read how many tiles are
// still active (so this stage cannot be captured in a CUDA graph).
cudaError_t launch_cg_solve(const Args& a, const Workspace& ws, cudaStream_t s, int max_iters,
                            float rel_tol) {
  const CgState st = carve_cg(a, ws);
  const int ntiles = (a.T + TILE - 1) / TILE;
  const long long blocks = (long long)ntiles * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = (unsigned)blocks;
  cudaError_t err;
  // kbar = sum_j w_ij k_j / omega_i: the readout with y = 0 (zero parts, cy = 0) and V := K.
  cg_zero_kernel<<<1216, 256, 0, s>>>(ws.ytc, ws.cy, a.rows());
  count_launch();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if ((err = launch_readout_tc_f32(a, ws, s, a.k, ws.ytc, ws.cy, ws.kbar, nullptr, false)) != cudaSuccess)
    return err;
  cg_init_kernel<<<g, NWARP * 32, 0, s>>>(static_cast<const __nv_bfloat16*>(a.q), ws.kbar, a.T,
                                          (int)a.BH(), max_iters, ws.y, st, ws.ytc, ws.cy);
  count_launch();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const float tol2 = rel_tol * rel_tol;
  for (int it = 0; it < max_iters; ++it) {
    if ((err = launch_readout_tc_f32(a, ws, s, a.k, ws.ytc, ws.cy, st.ap, st.tile_active, true)) !=
        cudaSuccess)
      return err;
    cg_update_kernel<<<g, NWARP * 32, 0, s>>>(ws.kbar, ws.m, a.T, (int)a.BH(), a.lam, tol2, it,
                                              ws.y, st, ws.ytc, ws.cy);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((it + 1) % kCheckEvery == 0 && it + 1 < max_iters) {
      int active = 0;
      if ((err = cudaMemcpyAsync(&active, st.counts + it, sizeof(int), cudaMemcpyDeviceToHost, s)) !=
          cudaSuccess)
        return err;
      if ((err = cudaStreamSynchronize(s)) != cudaSuccess) return err;
      if (active == 0) break;
    }
  }
  cg_final_kernel<<<g, NWARP * 32, 0, s>>>(ws.kbar, a.T, ws.y, ws.ytc, ws.cy, ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
