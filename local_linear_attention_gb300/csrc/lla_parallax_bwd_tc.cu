// Tensor-core passes of the causal Parallax backward (bf16, d = dv = 64; tcgen05 + TMEM).
//
// The gradient (see lla_parallax_bwd.cu for its derivation from the forward of the "Parallax"
// blog, s.2 and Appendix B with eta = 0): with p_ij = exp((q_i.k_j - m_i)/h) / omega_i over
// j <= i, t_ij = r_i . k_j, g_ij = dO_i . v_j and the row record {m_i, 1/omega_i, tbar_i, G_i,
// D_i} of the statistics pass,
//   ds_ij = p_ij ((1 + tbar_i - t_ij) g_ij + G_i t_ij - D_i),  dt_ij = p_ij (G_i - g_ij),
//   a_ij = p_ij (1 + tbar_i - t_ij),
//   dQ = dS K / h,  dR = dT K,  dK = dS^T Q / h + dT^T R,  dV = A^T dO.
// The blog's Appendix F splits the backward the same way: a row-tile pass (dQ, dR) and a
// column-tile pass (dK, dV), because the two reductions run in opposite directions.
//
// Rows pass: one CTA per 128-query tile; per 64-key block of its causal prefix, S = Q K^T,
// T = R K^T and G = dO V^T (tcgen05.mma, operands from shared memory, fp32 in tensor memory);
// eight warps (two per tensor-memory lane quarter, one thread per query row, each taking 32 of
// the block's 64 keys) turn them into dS and dT (bf16, written to tensor memory), and
// dQ += dS K, dR += dT K (A from tensor memory, B = the key block read as an MN-major operand)
// accumulate in tensor memory.
// Columns pass: one CTA per 128-key tile; per 64-query block from the tile's first key on,
// S^T = K Q^T, T^T = K R^T, G^T = V dO^T; the eight warps (one thread per key row, 32 of the
// block's queries each) take the block's row records from shared memory and form dS^T / h,
// dT^T and A^T; dK += dS^T Q + dT^T R and dV += A^T dO.
// The elementwise step is a chain of exponentials and shared-memory reads per element; two
// warps per lane quarter give each scheduler a second warp to hide it behind.
// Warp roles (10 warps): 0 issues every MMA (one thread) and owns the tensor-memory allocation;
// 1 stages the streamed blocks with cp.async (several in flight); 2-9 the elementwise step and
// the output (warps 2-5 the first half of each block and dQ / dK, warps 6-9 the second half and
// dR / dV). All mbarrier waits are bounded.
#include <cstdint>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int BM = 128;  // rows of the resident tile (queries or keys)
constexpr int BB = 64;   // rows of a streamed block (keys or queries): N = 64 score MMAs
constexpr int KS = 6;
constexpr int NWARPS = 10;  // MMA issuer, loader, 8 elementwise warps (two per lane quarter)
constexpr int NTHREADS = NWARPS * 32;
constexpr int TILE = BM * D * 2;     // 16 KiB
constexpr int STAGE = BB * D * 2;    // 8 KiB
constexpr int STAT = 8;              // floats per row record
constexpr uint32_t TMEM_COLS = 512;

__device__ __forceinline__ int kmaj_off(int r, int c) { return (r >> 3) * 1024 + c * 128 + (r & 7) * 16; }
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, kStatusTimeout, abort));
}

// A [BM x 64] bf16 tile of `src` rows r0 .. r0 + n - 1 (zero past n) into the K-major layout.
__device__ __forceinline__ void load_tile(uint8_t* dst, const __nv_bfloat16* src, long long r0,
                                          int n, int tid) {
  for (int e = tid; e < BM * (D / 8); e += NTHREADS) {
    const int r = e >> 3, c = e & 7;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < n) val = *reinterpret_cast<const uint4*>(src + (r0 + r) * D + c * 8);
    *reinterpret_cast<uint4*>(dst + kmaj_off(r, c)) = val;
  }
}

// BB rows (row < nrows, else zeros) of a [., 64] bf16 tensor into a K-major stage, by one warp:
// lane -> (row, chunk) as in the other stages (each 8-lane phase writes 8 distinct bank groups).
__device__ __forceinline__ void stage_block(uint8_t* dst, const __nv_bfloat16* src, long long r0,
                                            int nrows, int lane) {
  static_assert(BB == 64, "lane mapping for 64-row blocks");
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int r = (lane & 7) + 8 * (t & 7), c = (lane >> 3) + 4 * (t >> 3);
    const bool in = r < nrows;
    cp_async16(dst + kmaj_off(r, c), src + (in ? r0 + r : 0) * D + c * 8, in ? 16u : 0u);
  }
}

// ============================================================================ rows: dQ, dR
namespace rows {
constexpr uint32_t T_S = 0, T_T = 64, T_G = 128;  // 64 fp32 each (one buffer)
constexpr uint32_t T_DS = 192, T_DT = 256;        // 2 x 32 (packed bf16) each
constexpr uint32_t T_DQ = 320, T_DR = 384;        // 64 fp32 each
constexpr int SM_Q = 0, SM_R = SM_Q + TILE, SM_Y = SM_R + TILE;
constexpr int SM_K = SM_Y + TILE, SM_V = SM_K + KS * STAGE;
constexpr int SM_BAR = SM_V + KS * STAGE;
constexpr int SMEM_BYTES = SM_BAR + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

struct Barriers {
  uint64_t kvfull[KS], kvempty[KS];
  uint64_t sfull[2], sfree[2], pfull[2], pfree[2];
  uint64_t accfull, done;
};
static_assert(sizeof(Barriers) <= 256, "barrier region");

__global__ void __launch_bounds__(NTHREADS, 1)
pbw_rows_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ rp,
                   const __nv_bfloat16* __restrict__ dout, const float* __restrict__ stats, int T,
                   int BH, float inv_h, __nv_bfloat16* __restrict__ dq,
                   __nv_bfloat16* __restrict__ dr, int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + SM_BAR);
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = (T + BM - 1) / BM;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);  // longest causal prefixes first
  const long long bh = blockIdx.x % BH;
  const int i0 = tile * BM;
  const int nq = min(BM, T - i0);
  const int jend = i0 + nq;
  const int nb = (jend + BB - 1) / BB;
  const long long base = bh * T;

  load_tile(smem + SM_Q, q, base + i0, nq, tid);
  load_tile(smem + SM_R, rp, base + i0, nq, tid);
  load_tile(smem + SM_Y, dout, base + i0, nq, tid);
  if (tid == 0) {
    for (int s = 0; s < KS; ++s) { mbar_init(&bar.kvfull[s], 32); mbar_init(&bar.kvempty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 8);
      mbar_init(&bar.pfull[s], 8);
      mbar_init(&bar.pfree[s], 1);
    }
    mbar_init(&bar.accfull, 1);
    mbar_init(&bar.done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  volatile int* abort_p = &abort_flag;
  const int TO = kStatusTimeout;

  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t qd = smem_desc(smem_u32(smem + SM_Q), 128, 1024);
      const uint64_t rd = smem_desc(smem_u32(smem + SM_R), 128, 1024);
      const uint64_t yd = smem_desc(smem_u32(smem + SM_Y), 128, 1024);
      const uint64_t kd = smem_desc(smem_u32(smem + SM_K), 128, 1024);
      const uint64_t vd = smem_desc(smem_u32(smem + SM_V), 128, 1024);
      // The key block as the MN-major B operand of dS K: K = keys (8-key groups 1024 B apart),
      // N = features (8-feature groups 128 B apart).
      const uint64_t kmn = smem_desc(smem_u32(smem + SM_K), 1024, 128);
      constexpr uint32_t id_s = idesc_bf16(BM, BB, false, false);
      constexpr uint32_t id_o = idesc_bf16(BM, D, false, true);
      constexpr uint32_t stage16 = STAGE >> 4;
      bool ok = true;
      int st = 0;
      uint32_t kpar = 0;
      for (int g = 0; g <= nb && ok; ++g) {
        if (g < nb) {
          // one S / T / G buffer: free once the previous block's scores were read
          ok = g >= 1 ? mbar_wait2(&bar.kvfull[st], kpar, &bar.sfree[0], (g - 1) & 1, status, TO,
                                   abort_p)
                      : mbar_wait(&bar.kvfull[st], kpar, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          fence_proxy_async_smem();  // the stage's cp.async writes, before the async-proxy reads
          const uint64_t kst = kd + (uint64_t)(st * stage16), vst = vd + (uint64_t)(st * stage16);
#pragma unroll
          for (int s = 0; s < D / 16; ++s) {
            mma_ss(tbase + T_S, qd + 16 * s, kst + 16 * s, id_s, s > 0);
            mma_ss(tbase + T_T, rd + 16 * s, kst + 16 * s, id_s, s > 0);
            mma_ss(tbase + T_G, yd + 16 * s, vst + 16 * s, id_s, s > 0);
          }
          mma_commit(&bar.sfull[0]);
          if (++st == KS) { st = 0; kpar ^= 1; }
        }
        if (g >= 1) {
          const int h = g - 1, pb = h & 1, sth = h % KS;
          ok = mbar_wait(&bar.pfull[pb], (h >> 1) & 1, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kms = kmn + (uint64_t)(sth * stage16);
#pragma unroll
          for (int s = 0; s < BB / 16; ++s) {
            const uint64_t b = kms + (uint64_t)(s * (2048 >> 4));
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            mma_ts(tbase + T_DQ, tbase + T_DS + pb * 32 + s * 8, b, id_o, acc);
            mma_ts(tbase + T_DR, tbase + T_DT + pb * 32 + s * 8, b, id_o, acc);
          }
          mma_commit(&bar.pfree[pb]);
          mma_commit(&bar.kvempty[sth]);
          if (h == nb - 1) mma_commit(&bar.accfull);
        }
      }
      if (!ok) *abort_p = 1;
      mma_commit(&bar.done);
      volatile int never = 0;
      mbar_wait(&bar.done, 0, status, TO, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ K / V loader
    for (int g = 0; g < nb; ++g) {
      {
        const int st = g % KS;
        if (g >= KS && !warp_wait(&bar.kvempty[st], ((g / KS) - 1) & 1, status, abort_p)) break;
        const int nrows = min(BB, jend - g * BB);
        stage_block(smem + SM_K + st * STAGE, k, base + g * BB, nrows, lane);
        stage_block(smem + SM_V + st * STAGE, v, base + g * BB, nrows, lane);
        cp_async_mbar_arrive(&bar.kvfull[st]);  // this lane's copies of the block, on completion
      }
    }
    cp_async_commit();
    cp_async_wait<0>();  // nothing of this warp is in flight at teardown
  } else {
    // ------------------------------------------------------------------ dS, dT and the output
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;  // this warp's half of each block (32 columns)
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float c2 = inv_h * 1.4426950408889634f;  // log2(e) / h
    float m = 0.f, inv_om = 0.f, tbar = 0.f, G = 0.f, Dr = 0.f;
    if (valid) {
      const float4 s4 = *reinterpret_cast<const float4*>(stats + (base + i) * STAT);
      m = s4.x; inv_om = s4.y; tbar = s4.z; G = s4.w;
      Dr = stats[(base + i) * STAT + 4];
    }
    const float mc = m * c2;
    bool ok = true;
    for (int h = 0; h < nb && ok; ++h) {
      if (!warp_wait(&bar.sfull[0], h & 1, status, abort_p)) { ok = false; break; }
      tc_fence_after();
      const int pb = h & 1;
      {  // this warp's 32 columns of the block
        uint32_t sv[32], tv[32], gv[32];
        tmem_ld16(lane_base + T_S + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
        tmem_ld16(lane_base + T_S + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
        tmem_ld16(lane_base + T_T + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&tv[0]));
        tmem_ld16(lane_base + T_T + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&tv[16]));
        tmem_ld16(lane_base + T_G + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&gv[0]));
        tmem_ld16(lane_base + T_G + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&gv[16]));
        tmem_ld_wait();
        {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.sfree[0]);
        }
        const int j0 = h * BB + 32 * hf;
        uint32_t dsw[16], dtw[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float ds[2], dt[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float p = (valid && j0 + c + u <= i)
                                ? ex2(fmaf(__uint_as_float(sv[c + u]), c2, -mc)) * inv_om
                                : 0.f;
            const float t = __uint_as_float(tv[c + u]), gg = __uint_as_float(gv[c + u]);
            ds[u] = p * (fmaf(1.f + tbar - t, gg, G * t) - Dr);
            dt[u] = p * (G - gg);
          }
          dsw[c / 2] = pack_bf16(ds[0], ds[1]);
          dtw[c / 2] = pack_bf16(dt[0], dt[1]);
        }
        {
          if (h >= 2 && !warp_wait(&bar.pfree[pb], ((h >> 1) - 1) & 1, status, abort_p)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st8(lane_base + T_DS + pb * 32 + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&dsw[0]));
        tmem_st8(lane_base + T_DS + pb * 32 + 16 * hf + 8,
                 *reinterpret_cast<uint32_t(*)[8]>(&dsw[8]));
        tmem_st8(lane_base + T_DT + pb * 32 + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&dtw[0]));
        tmem_st8(lane_base + T_DT + pb * 32 + 16 * hf + 8,
                 *reinterpret_cast<uint32_t(*)[8]>(&dtw[8]));
      }
      if (!ok) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.pfull[pb]);
    }
    if (ok && warp_wait(&bar.accfull, 0, status, abort_p)) {
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        // half 0 writes dQ (the accumulated ds k, times 1/h), half 1 dR
        uint32_t a[16];
        tmem_ld16(lane_base + (hf ? T_DR : T_DQ) + c0, a);
        tmem_ld_wait();
        if (valid) {
          const float sc = hf ? 1.f : inv_h;
          uint32_t pa[8];
#pragma unroll
          for (int t = 0; t < 16; t += 2)
            pa[t / 2] = pack_bf16(__uint_as_float(a[t]) * sc, __uint_as_float(a[t + 1]) * sc);
          uint4* o = reinterpret_cast<uint4*>((hf ? dr : dq) + (base + i) * D + c0);
          o[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
          o[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}
}  // namespace rows

// ============================================================================ columns: dK, dV
namespace cols {
constexpr uint32_t T_S = 0, T_T = 64, T_G = 128;     // 64 fp32 each (one buffer)
constexpr uint32_t T_DS = 192, T_DT = 256, T_A = 320;  // 2 x 32 (packed bf16) each
constexpr uint32_t T_DK = 384, T_DV = 448;           // 64 fp32 each
constexpr int SM_K = 0, SM_V = SM_K + TILE;
constexpr int SM_QS = SM_V + TILE, SM_RS = SM_QS + KS * STAGE, SM_YS = SM_RS + KS * STAGE;
constexpr int SM_SS = SM_YS + KS * STAGE;  // KS x 64 row records
constexpr int SS_STAGE = BB * STAT * 4;    // 2 KiB
constexpr int SM_BAR = SM_SS + KS * SS_STAGE;
constexpr int SMEM_BYTES = SM_BAR + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

struct Barriers {
  uint64_t qfull[KS], qempty[KS];
  uint64_t sfull[2], sfree[2], pfull[2], pfree[2];
  uint64_t accfull, done;
};
static_assert(sizeof(Barriers) <= 256, "barrier region");

__global__ void __launch_bounds__(NTHREADS, 1)
pbw_cols_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ rp,
                   const __nv_bfloat16* __restrict__ dout, const float* __restrict__ stats, int T,
                   int BH, float inv_h, __nv_bfloat16* __restrict__ dk,
                   __nv_bfloat16* __restrict__ dv, int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + SM_BAR);
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = (int)(blockIdx.x / BH);  // most queries (earliest keys) first
  const long long bh = blockIdx.x % BH;
  const int j0 = tile * BM;
  const int nk = min(BM, T - j0);
  const int qb0 = j0 / BB;                     // first query block that sees this tile
  const int nblk = (T + BB - 1) / BB - qb0;    // query blocks streamed
  const long long base = bh * T;

  load_tile(smem + SM_K, k, base + j0, nk, tid);
  load_tile(smem + SM_V, v, base + j0, nk, tid);
  if (tid == 0) {
    for (int s = 0; s < KS; ++s) { mbar_init(&bar.qfull[s], 32); mbar_init(&bar.qempty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 8);
      mbar_init(&bar.pfull[s], 8);
      mbar_init(&bar.pfree[s], 1);
    }
    mbar_init(&bar.accfull, 1);
    mbar_init(&bar.done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  volatile int* abort_p = &abort_flag;
  const int TO = kStatusTimeout;

  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t kd = smem_desc(smem_u32(smem + SM_K), 128, 1024);
      const uint64_t vd = smem_desc(smem_u32(smem + SM_V), 128, 1024);
      const uint64_t qd = smem_desc(smem_u32(smem + SM_QS), 128, 1024);
      const uint64_t rd = smem_desc(smem_u32(smem + SM_RS), 128, 1024);
      const uint64_t yd = smem_desc(smem_u32(smem + SM_YS), 128, 1024);
      // Query blocks as MN-major B operands of the dK / dV products: K = queries (8-query
      // groups 1024 B apart), N = features (8-feature groups 128 B apart).
      const uint64_t qmn = smem_desc(smem_u32(smem + SM_QS), 1024, 128);
      const uint64_t rmn = smem_desc(smem_u32(smem + SM_RS), 1024, 128);
      const uint64_t ymn = smem_desc(smem_u32(smem + SM_YS), 1024, 128);
      constexpr uint32_t id_s = idesc_bf16(BM, BB, false, false);
      constexpr uint32_t id_o = idesc_bf16(BM, D, false, true);
      constexpr uint32_t stage16 = STAGE >> 4;
      bool ok = true;
      int st = 0;
      uint32_t qpar = 0;
      for (int g = 0; g <= nblk && ok; ++g) {
        if (g < nblk) {
          // one S / T / G buffer: free once the previous block's scores were read
          ok = g >= 1 ? mbar_wait2(&bar.qfull[st], qpar, &bar.sfree[0], (g - 1) & 1, status, TO,
                                   abort_p)
                      : mbar_wait(&bar.qfull[st], qpar, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          fence_proxy_async_smem();  // the stage's cp.async writes, before the async-proxy reads
          const uint64_t o = (uint64_t)(st * stage16);
#pragma unroll
          for (int s = 0; s < D / 16; ++s) {
            mma_ss(tbase + T_S, kd + 16 * s, qd + o + 16 * s, id_s, s > 0);
            mma_ss(tbase + T_T, kd + 16 * s, rd + o + 16 * s, id_s, s > 0);
            mma_ss(tbase + T_G, vd + 16 * s, yd + o + 16 * s, id_s, s > 0);
          }
          mma_commit(&bar.sfull[0]);
          if (++st == KS) { st = 0; qpar ^= 1; }
        }
        if (g >= 1) {
          const int h = g - 1, pb = h & 1, sth = h % KS;
          ok = mbar_wait(&bar.pfull[pb], (h >> 1) & 1, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          const uint64_t o = (uint64_t)(sth * stage16);
#pragma unroll
          for (int s = 0; s < BB / 16; ++s) {
            const uint64_t so = o + (uint64_t)(s * (2048 >> 4));
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            mma_ts(tbase + T_DK, tbase + T_DS + pb * 32 + s * 8, qmn + so, id_o, acc);
            mma_ts(tbase + T_DK, tbase + T_DT + pb * 32 + s * 8, rmn + so, id_o, 1u);
            mma_ts(tbase + T_DV, tbase + T_A + pb * 32 + s * 8, ymn + so, id_o, acc);
          }
          mma_commit(&bar.pfree[pb]);
          mma_commit(&bar.qempty[sth]);
          if (h == nblk - 1) mma_commit(&bar.accfull);
        }
      }
      if (!ok) *abort_p = 1;
      mma_commit(&bar.done);
      volatile int never = 0;
      mbar_wait(&bar.done, 0, status, TO, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ Q / R / dO / record loader
    for (int g = 0; g < nblk; ++g) {
      {
        const int st = g % KS;
        if (g >= KS && !warp_wait(&bar.qempty[st], ((g / KS) - 1) & 1, status, abort_p)) break;
        const int r0 = (qb0 + g) * BB;
        const int nrows = min(BB, T - r0);
        stage_block(smem + SM_QS + st * STAGE, q, base + r0, nrows, lane);
        stage_block(smem + SM_RS + st * STAGE, rp, base + r0, nrows, lane);
        stage_block(smem + SM_YS + st * STAGE, dout, base + r0, nrows, lane);
        // 64 records of 32 bytes: four 16-byte copies per lane
        float* sdst = reinterpret_cast<float*>(smem + SM_SS + st * SS_STAGE);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int e = lane + 32 * t, rr = e >> 1, half4 = e & 1;
          const bool in = rr < nrows;
          cp_async16(sdst + rr * STAT + 4 * half4,
                     stats + (base + (in ? r0 + rr : 0)) * STAT + 4 * half4, in ? 16u : 0u);
        }
        cp_async_mbar_arrive(&bar.qfull[st]);  // this lane's copies of the block, on completion
      }
    }
    cp_async_commit();
    cp_async_wait<0>();  // nothing of this warp is in flight at teardown
  } else {
    // ------------------------------------------------------------------ dS^T, dT^T, A^T, output
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;  // this warp's half of each block (32 columns)
    const int r = quarter * 32 + lane;
    const int j = j0 + r;
    const bool valid = r < nk;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float c2 = inv_h * 1.4426950408889634f;
    bool ok = true;
    for (int h = 0; h < nblk && ok; ++h) {
      const int sth = h % KS, pb = h & 1;
      // the block's records: read after the loader's own completion signal for the stage
      if (!warp_wait(&bar.qfull[sth], (h / KS) & 1, status, abort_p) ||
          !warp_wait(&bar.sfull[0], h & 1, status, abort_p)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* rec = reinterpret_cast<const float*>(smem + SM_SS + sth * SS_STAGE);
      {  // this warp's 32 queries of the block
        uint32_t sv[32], tv[32], gv[32];
        tmem_ld16(lane_base + T_S + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
        tmem_ld16(lane_base + T_S + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
        tmem_ld16(lane_base + T_T + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&tv[0]));
        tmem_ld16(lane_base + T_T + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&tv[16]));
        tmem_ld16(lane_base + T_G + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&gv[0]));
        tmem_ld16(lane_base + T_G + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&gv[16]));
        tmem_ld_wait();
        {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.sfree[0]);
        }
        const int iq0 = (qb0 + h) * BB + 32 * hf;
        const float* rh = rec + 32 * hf * STAT;
        uint32_t dsw[16], dtw[16], aw[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float ds[2], dt[2], a[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = iq0 + c + u;
            const float4 s4 = *reinterpret_cast<const float4*>(rh + (c + u) * STAT);
            const float Dr = rh[(c + u) * STAT + 4];
            const float p = (valid && j <= i && i < T)
                                ? ex2((__uint_as_float(sv[c + u]) - s4.x) * c2) * s4.y
                                : 0.f;
            const float t = __uint_as_float(tv[c + u]), gg = __uint_as_float(gv[c + u]);
            const float w = 1.f + s4.z - t;
            ds[u] = p * (fmaf(w, gg, s4.w * t) - Dr) * inv_h;
            dt[u] = p * (s4.w - gg);
            a[u] = p * w;
          }
          dsw[c / 2] = pack_bf16(ds[0], ds[1]);
          dtw[c / 2] = pack_bf16(dt[0], dt[1]);
          aw[c / 2] = pack_bf16(a[0], a[1]);
        }
        {
          if (h >= 2 && !warp_wait(&bar.pfree[pb], ((h >> 1) - 1) & 1, status, abort_p)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t co = pb * 32 + 16 * hf;
        tmem_st8(lane_base + T_DS + co, *reinterpret_cast<uint32_t(*)[8]>(&dsw[0]));
        tmem_st8(lane_base + T_DS + co + 8, *reinterpret_cast<uint32_t(*)[8]>(&dsw[8]));
        tmem_st8(lane_base + T_DT + co, *reinterpret_cast<uint32_t(*)[8]>(&dtw[0]));
        tmem_st8(lane_base + T_DT + co + 8, *reinterpret_cast<uint32_t(*)[8]>(&dtw[8]));
        tmem_st8(lane_base + T_A + co, *reinterpret_cast<uint32_t(*)[8]>(&aw[0]));
        tmem_st8(lane_base + T_A + co + 8, *reinterpret_cast<uint32_t(*)[8]>(&aw[8]));
      }
      if (!ok) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.pfull[pb]);
    }
    if (ok && warp_wait(&bar.accfull, 0, status, abort_p)) {
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        // half 0 writes dK, half 1 dV
        uint32_t a[16];
        tmem_ld16(lane_base + (hf ? T_DV : T_DK) + c0, a);
        tmem_ld_wait();
        if (valid) {
          uint32_t pk[8];
#pragma unroll
          for (int t = 0; t < 16; t += 2)
            pk[t / 2] = pack_bf16(__uint_as_float(a[t]), __uint_as_float(a[t + 1]));
          uint4* o = reinterpret_cast<uint4*>((hf ? dv : dk) + (base + j) * D + c0);
          o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}
}  // namespace cols

}  // namespace

cudaError_t launch_parallax_bwd_tc(const ParallaxBwdArgs& a, float* stats, int* status,
                                   cudaStream_t s) {
  cudaError_t err = launch_parallax_stats_tc(a, stats, status, s);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)((a.T + BM - 1) / BM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const auto* q = static_cast<const __nv_bfloat16*>(a.q);
  const auto* k = static_cast<const __nv_bfloat16*>(a.k);
  const auto* v = static_cast<const __nv_bfloat16*>(a.v);
  const auto* r = static_cast<const __nv_bfloat16*>(a.r);
  const auto* dy = static_cast<const __nv_bfloat16*>(a.dout);
  const float inv_h = 1.0f / a.h;
  const int BH = (int)a.BH();
  err = cudaFuncSetAttribute(rows::pbw_rows_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             rows::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  rows::pbw_rows_tc_kernel<<<(unsigned)blocks, NTHREADS, rows::SMEM_BYTES, s>>>(
      q, k, v, r, dy, stats, a.T, BH, inv_h, static_cast<__nv_bfloat16*>(a.dq),
      static_cast<__nv_bfloat16*>(a.dr), status);
  count_launch();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  err = cudaFuncSetAttribute(cols::pbw_cols_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             cols::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  cols::pbw_cols_tc_kernel<<<(unsigned)blocks, NTHREADS, cols::SMEM_BYTES, s>>>(
      q, k, v, r, dy, stats, a.T, BH, inv_h, static_cast<__nv_bfloat16*>(a.dk),
      static_cast<__nv_bfloat16*>(a.dv), status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
