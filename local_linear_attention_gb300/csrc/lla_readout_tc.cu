// Tensor-core readout stage of the causal LLA forward (bf16 inputs, d = 64; tcgen05 + TMEM).
//
// With y_i = (C_kk + lambda' I)^-1 (q_i - kbar_i) from the ridge solve, one streaming pass over
// the causal prefix evaluates the centred closed form of the LLA intercept ("Parallax" blog, s.2
// Canonical Formulation)
//   o_i = vbar_i + C_vk y_i = O1_i / omega_i + O2_i,
//   O1 = P V,  O2 = (P .* t) V,  t_ij = k_j . y_i - kbar_i . y_i,
// where P holds the kernel weights exactly as the tensor-core moments stage rounded them (same
// S = Q K^T contraction, same exponent, same bf16 rounding), so the fitted moments and this pass
// describe one weighted problem (and sum_j p_ij t_ij = 0 up to rounding). The pass has the
// two-branch shape of the blog's streaming algorithm (s.3 "One extra branch, no extra I/O"): a
// softmax branch (O1, omega) and a covariance branch (O2) over the same K/V tiles.
//
// Precision: y can be large (small ridge, rank-deficient early prefixes), and its component
// outside the span of the keys must cancel between k_j . y and kbar . y; y therefore enters the
// Y K^T contraction as three exact bf16 parts (y = y1 + y2 + y3, 24 significant bits), and the
// covariance-branch weights p * t enter P2 V as an exact-to-16-bits hi/lo pair.
//
// Warp roles (6 warps): 0 issues every tcgen05.mma and owns the TMEM allocation; 1 stages key and
// value blocks; 2-5 (one thread per query = TMEM lane) turn S and T into P and P2 and write the
// output. All waits are bounded.
#include <cstdint>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int DV = 64;
constexpr int BM = 128;
constexpr int KB = 32;
constexpr int KS = 6;
constexpr int KLAG = KS - 2;
constexpr int NWARPS = 6;
constexpr int NTHREADS = NWARPS * 32;

// tensor-memory columns
constexpr uint32_t T_O1 = 0;            // 64 fp32: P V
constexpr uint32_t T_O2 = 64;           // 64 fp32: P2 V
constexpr uint32_t T_S = 128;           // 2 x 32 fp32: Q K^T
constexpr uint32_t T_T = 192;           // 2 x 32 fp32: Y K^T
constexpr uint32_t T_P = 256;           // 2 x 16: bf16 P
constexpr uint32_t T_P2H = 288;         // 2 x 16: bf16 hi part of P .* t
constexpr uint32_t T_P2L = 320;         // 2 x 16: bf16 lo part
constexpr uint32_t TMEM_COLS = 512;

// shared memory (bytes)
constexpr int TILE = BM * D * 2;                    // 128 x 64 bf16 = 16 KiB
constexpr int SM_Q = 0;
constexpr int SM_Y = SM_Q + TILE;                   // 3 tiles: y1, y2, y3
constexpr int SM_K = SM_Y + 3 * TILE;
constexpr int KV_STAGE = KB * D * 2;                // 4 KiB
constexpr int SM_V = SM_K + KS * KV_STAGE;
constexpr int SM_BAR = SM_V + KS * KV_STAGE;
constexpr int SMEM_BYTES = SM_BAR + 256;

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
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, kStatusTimeout, abort));
}

struct Barriers {
  uint64_t kvfull[KS], kvempty[KS];
  uint64_t sfull[2], sfree[2];
  uint64_t pfull[2], pfree[2];
  uint64_t accfull, done;
};

template <typename TOut>
__global__ void __launch_bounds__(NTHREADS, 1)
readout_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const float* __restrict__ mraw,
                  const float* __restrict__ y, const float* __restrict__ kbar, int T, int BH,
                  float inv_h, TOut* __restrict__ out, int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + SM_BAR);
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = (T + BM - 1) / BM;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);
  const long long bh = blockIdx.x % BH;
  const int i0 = tile * BM;
  const int nq = min(BM, T - i0);
  const int jend = i0 + nq;
  const int nb = (jend + KB - 1) / KB;
  const long long base = bh * T;

  // Q tile (bf16, as the moments stage had it).
  for (int e = tid; e < BM * (D / 8); e += NTHREADS) {
    const int r = e >> 3, c = e & 7;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < nq) val = *reinterpret_cast<const uint4*>(q + (base + i0 + r) * D + c * 8);
    *reinterpret_cast<uint4*>(smem + SM_Q + kmaj_off(r, c)) = val;
  }
  // y split into three exact bf16 parts; one row (query) per thread of warps 2..5.
  if (warp >= 2) {
    const int r = (warp & 3) * 32 + lane;
    const bool valid = r < nq;
    const float* yr = y + (base + i0 + r) * D;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w1[4], w2[4], w3[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float a = 0.f, b = 0.f;
        if (valid) { a = yr[c * 8 + 2 * t]; b = yr[c * 8 + 2 * t + 1]; }
        w1[t] = pack_bf16(a, b);
        const float a2 = a - bf16_lo(w1[t]), b2 = b - bf16_hi(w1[t]);
        w2[t] = pack_bf16(a2, b2);
        w3[t] = pack_bf16(a2 - bf16_lo(w2[t]), b2 - bf16_hi(w2[t]));
      }
      *reinterpret_cast<uint4*>(smem + SM_Y + kmaj_off(r, c)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
      *reinterpret_cast<uint4*>(smem + SM_Y + TILE + kmaj_off(r, c)) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
      *reinterpret_cast<uint4*>(smem + SM_Y + 2 * TILE + kmaj_off(r, c)) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < KS; ++s) { mbar_init(&bar.kvfull[s], 1); mbar_init(&bar.kvempty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 4);
      mbar_init(&bar.pfull[s], 4);
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

  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Base descriptors plus start-address offsets in 16-byte units (see the moments stage).
      const uint64_t qd = smem_desc(smem_u32(smem + SM_Q), 128, 1024);
      const uint64_t yd = smem_desc(smem_u32(smem + SM_Y), 128, 1024);
      const uint64_t kd = smem_desc(smem_u32(smem + SM_K), 128, 1024);
      // V block as the MN-major B operand: K = keys (8-key groups 1024 B apart), N = value
      // features (8-feature groups 128 B apart).
      const uint64_t vd = smem_desc(smem_u32(smem + SM_V), 1024, 128);
      constexpr uint32_t id_s = idesc_bf16(BM, KB, false, false);
      constexpr uint32_t id_o = idesc_bf16(BM, DV, false, true);
      constexpr uint32_t tile16 = TILE >> 4, stage16 = KV_STAGE >> 4;
      const uint32_t t_s = tbase + T_S, t_t = tbase + T_T;
      bool ok = true;
      for (int g = 0; g <= nb && ok; ++g) {
        if (g < nb) {
          const int st = g % KS, sb = g & 1;
          ok = mbar_wait(&bar.kvfull[st], (g / KS) & 1, status, kStatusTimeout, abort_p);
          if (ok && g >= 2)
            ok = mbar_wait(&bar.sfree[sb], ((g >> 1) - 1) & 1, status, kStatusTimeout, abort_p);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kst = kd + (uint64_t)(st * stage16);
          const uint32_t ts = t_s + sb * KB, tt = t_t + sb * KB;
#pragma unroll
          for (int s = 0; s < D / 16; ++s) mma_ss(ts, qd + 16 * s, kst + 16 * s, id_s, s > 0);
#pragma unroll
          for (int part = 0; part < 3; ++part)
#pragma unroll
            for (int s = 0; s < D / 16; ++s)
              mma_ss(tt, yd + part * tile16 + 16 * s, kst + 16 * s, id_s,
                     (part > 0 || s > 0) ? 1u : 0u);
          mma_commit(&bar.sfull[sb]);
        }
        if (g >= 1) {
          const int h = g - 1, pb = h & 1, st = h % KS;
          ok = mbar_wait(&bar.pfull[pb], (h >> 1) & 1, status, kStatusTimeout, abort_p);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vst = vd + (uint64_t)(st * stage16);
#pragma unroll
          for (int s = 0; s < KB / 16; ++s) {
            const uint64_t vds = vst + (uint64_t)(s * (2048 >> 4));
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            mma_ts(tbase + T_O1, tbase + T_P + pb * 16 + s * 8, vds, id_o, acc);
            mma_ts(tbase + T_O2, tbase + T_P2H + pb * 16 + s * 8, vds, id_o, acc);
            mma_ts(tbase + T_O2, tbase + T_P2L + pb * 16 + s * 8, vds, id_o, 1u);
          }
          mma_commit(&bar.pfree[pb]);
          mma_commit(&bar.kvempty[st]);
          if (h == nb - 1) mma_commit(&bar.accfull);
        }
      }
      if (!ok) *abort_p = 1;
      mma_commit(&bar.done);
      volatile int never = 0;
      mbar_wait(&bar.done, 0, status, kStatusTimeout, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ K/V loader
    // cp.async copies with several blocks in flight; same conflict-free lane mapping and
    // completion -> proxy fence -> arrive protocol as the moments stage's loader.
    const __nv_bfloat16* kbp = k + base * D;
    const __nv_bfloat16* vbp = v + base * DV;
    bool ok = true;
    for (int g = 0; g < nb + KLAG; ++g) {
      if (g < nb) {
        const int st = g % KS;
        if (g >= KS && !warp_wait(&bar.kvempty[st], ((g / KS) - 1) & 1, status, abort_p)) {
          ok = false;
          break;
        }
        uint8_t* kd = smem + SM_K + st * KV_STAGE;
        uint8_t* vd = smem + SM_V + st * KV_STAGE;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int r = (lane & 7) + 8 * (t & 3), c = (lane >> 3) + 4 * (t >> 2);
          const int j = g * KB + r;
          const bool in = j < jend;
          const long long jj = in ? j : 0;
          cp_async16(kd + kmaj_off(r, c), kbp + jj * D + c * 8, in ? 16u : 0u);
          cp_async16(vd + kmaj_off(r, c), vbp + jj * DV + c * 8, in ? 16u : 0u);
        }
      }
      cp_async_commit();
      if (g >= KLAG) {
        cp_async_wait<KLAG>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.kvfull[(g - KLAG) % KS]);
      }
    }
    if (!ok) cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------------ weights + output
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float c2 = inv_h * 1.4426950408889634f;
    const float mc = valid ? mraw[base + i] * c2 : 0.f;
    float cy = 0.f;  // kbar . y
    if (valid) {
      const float* yr = y + (base + i) * D;
      const float* kr = kbar + (base + i) * D;
#pragma unroll 8
      for (int a = 0; a < D; ++a) cy = fmaf(kr[a], yr[a], cy);
    }
    float om = 0.f;
    for (int g = 0; g < nb; ++g) {
      const int sb = g & 1;
      if (!warp_wait(&bar.sfull[sb], (g >> 1) & 1, status, abort_p)) break;
      tc_fence_after();
      uint32_t sv[KB], tv[KB];
      tmem_ld16(lane_base + T_S + sb * KB, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
      tmem_ld16(lane_base + T_S + sb * KB + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
      tmem_ld16(lane_base + T_T + sb * KB, *reinterpret_cast<uint32_t(*)[16]>(&tv[0]));
      tmem_ld16(lane_base + T_T + sb * KB + 16, *reinterpret_cast<uint32_t(*)[16]>(&tv[16]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.sfree[sb]);
      const int j0 = g * KB;
      uint32_t pw[KB / 2], hw[KB / 2], lw[KB / 2];
#pragma unroll
      for (int c = 0; c < KB; c += 2) {
        const float p0 = (valid && j0 + c <= i) ? ex2(fmaf(__uint_as_float(sv[c]), c2, -mc)) : 0.f;
        const float p1 =
            (valid && j0 + c + 1 <= i) ? ex2(fmaf(__uint_as_float(sv[c + 1]), c2, -mc)) : 0.f;
        const uint32_t w = pack_bf16(p0, p1);
        pw[c / 2] = w;
        const float r0 = bf16_lo(w), r1 = bf16_hi(w);
        om += r0 + r1;
        const float q0 = r0 * (__uint_as_float(tv[c]) - cy);
        const float q1 = r1 * (__uint_as_float(tv[c + 1]) - cy);
        const uint32_t hh = pack_bf16(q0, q1);
        hw[c / 2] = hh;
        lw[c / 2] = pack_bf16(q0 - bf16_lo(hh), q1 - bf16_hi(hh));
      }
      const int pb = g & 1;
      if (g >= 2 && !warp_wait(&bar.pfree[pb], ((g >> 1) - 1) & 1, status, abort_p)) break;
      tc_fence_after();
      tmem_st8(lane_base + T_P + pb * 16, *reinterpret_cast<uint32_t(*)[8]>(&pw[0]));
      tmem_st8(lane_base + T_P + pb * 16 + 8, *reinterpret_cast<uint32_t(*)[8]>(&pw[8]));
      tmem_st8(lane_base + T_P2H + pb * 16, *reinterpret_cast<uint32_t(*)[8]>(&hw[0]));
      tmem_st8(lane_base + T_P2H + pb * 16 + 8, *reinterpret_cast<uint32_t(*)[8]>(&hw[8]));
      tmem_st8(lane_base + T_P2L + pb * 16, *reinterpret_cast<uint32_t(*)[8]>(&lw[0]));
      tmem_st8(lane_base + T_P2L + pb * 16 + 8, *reinterpret_cast<uint32_t(*)[8]>(&lw[8]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.pfull[pb]);
      if (g == nb - 1) {
        if (!warp_wait(&bar.accfull, 0, status, abort_p)) break;
        tc_fence_after();
        const float inv = 1.f / om;
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 16) {
          uint32_t o1[16], o2[16];
          tmem_ld16(lane_base + T_O1 + c0, o1);
          tmem_ld16(lane_base + T_O2 + c0, o2);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int t = 0; t < 16; ++t)
              stf(out, (base + i) * DV + c0 + t,
                  fmaf(__uint_as_float(o1[t]), inv, __uint_as_float(o2[t])));
          }
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

}  // namespace

cudaError_t launch_readout_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  auto kern = readout_tc_kernel<__nv_bfloat16>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)((a.T + BM - 1) / BM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, NTHREADS, SMEM_BYTES, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), ws.mraw, ws.y, ws.kbar, a.T, (int)a.BH(),
      1.0f / a.h, static_cast<__nv_bfloat16*>(a.out), ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
