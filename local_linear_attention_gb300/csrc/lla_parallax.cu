// Causal Parallax forward with a given probe R ("Parallax" blog s.2 "Parallax" and Appendix B with
// eta = 0; the streaming form of s.3 "One extra branch, no extra I/O"):
//   o_i = o_SA_i - Sigma_KV^(i) r_i = (1 + d2/d1) O1/d1 - O2/d1,
//   P1 = exp(Q K^T / h) (causal), S2 = R K^T, P2 = P1 .* S2,
//   O1 = P1 V, d1 = rowsum P1, O2 = P2 V, d2 = rowsum P2
// (the combination printed in the blog's Appendix C). Both branches stream the same K/V blocks.
//
// Two implementations:
//  * tensor cores (bf16, d = dv = 64): one CTA per 128-query tile, keys in blocks of 64 (so that
//    Q K^T and R K^T are N = 64 MMAs: a tcgen05.mma costs about as long at N = 32). A first
//    sweep over the causal
//    prefix takes the exact row max of Q K^T (so no running rescale of the accumulators is
//    needed); the second sweep computes S1 = Q K^T and S2 = R K^T with tcgen05.mma (Q, R and K
//    from shared memory), turns them into P1 (bf16) and P2 = P1 .* S2 (an exact-to-16-bits bf16
//    hi/lo pair, so that the covariance term, a difference of two sums, keeps its precision), and
//    accumulates O1 = P1 V and O2 = P2 V in tensor memory. d1 and d2 are summed in fp32 from the
//    same rounded weights. Eight softmax warps, two per tensor-memory lane quarter, each take
//    one 32-key half of every block (one warp per scheduler left the exponential chain exposed).
//  * CUDA cores (every other shape and dtype): online softmax with running rescale, four threads
//    per query (each owns a quarter of the q, r, O1 and O2 coordinates), fp32 accumulation.
// All mbarrier waits are bounded.
#include <cstdint>
#include <type_traits>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"
#include "lla_tmap.cuh"

namespace lla {
namespace {

using namespace tc;

// ============================================================================ tensor cores
namespace ptc {

constexpr int D = 64;
constexpr int DV = 64;
constexpr int BM = 128;
constexpr int KB = 64;  // keys per block: N = 64 for Q K^T and R K^T
constexpr int KS = 6;
constexpr int NWARPS = 10;  // MMA issuer, loader, 8 softmax warps (two per lane quarter)
constexpr int NTHREADS = NWARPS * 32;

// tensor-memory columns
constexpr uint32_t T_O1 = 0;     // 64 fp32: P1 V
constexpr uint32_t T_O2 = 64;    // 64 fp32: P2 V
constexpr uint32_t T_S = 128;    // 2 x 64 fp32: Q K^T
constexpr uint32_t T_T = 256;    // 2 x 64 fp32: R K^T
constexpr uint32_t T_P = 384;    // 32: bf16 P1 (one buffer: the next block's is written once the
constexpr uint32_t T_P2H = 416;  // 32: bf16 hi part of P2    previous block's P V MMAs completed)
constexpr uint32_t T_P2L = 448;  // 32: bf16 lo part of P2
constexpr uint32_t TMEM_COLS = 512;

// shared memory (bytes)
constexpr int TILE = BM * D * 2;  // 128 x 64 bf16 = 16 KiB
constexpr int SM_Q = 0;
constexpr int SM_R = SM_Q + TILE;
constexpr int SM_K = SM_R + TILE;
constexpr int KV_STAGE = KB * D * 2;  // 8 KiB
constexpr int SM_V = SM_K + KS * KV_STAGE;
constexpr int SM_BAR = SM_V + KS * KV_STAGE;
constexpr int SM_X = SM_BAR + 256;  // [2 halves][5 values][BM] per-row partials of the two halves
constexpr int NXV = 5;              // m, d1, d2, and (STATS) dout . vbar, dout . o
constexpr int SMEM_BYTES = SM_X + 2 * NXV * BM * 4;
constexpr int SMEM_LAUNCH = SMEM_BYTES + 1024;  // slack for aligning the base to 1024 bytes
static_assert(SM_K % 1024 == 0 && SM_V % 1024 == 0 && KV_STAGE % 1024 == 0,
              "128-byte swizzled key and value stages on 1024-byte boundaries");

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
  uint64_t pfull, pfree;
  uint64_t accfull, done;
  uint64_t rowx;  // the two halves of each row exchanged m (phase 0), d1 and d2 (1), STATS sums (2)
};
static_assert(sizeof(Barriers) <= SM_X - SM_BAR, "barrier region");

// Steps g = 0 .. nb-1 are the max sweep (Q K^T only), g = nb .. 2nb-1 the main sweep over the
// same key blocks b = g - nb.
//
// STATS (the backward's row scalars, given the upstream gradient dout): instead of o, each row
// writes the record {m, 1/omega, tbar, G, D} to stats[row * 8 ..]: m the max of the raw logits
// q.k (before 1/h), omega = d1 the sum of its weights exp((q.k - m)/h), tbar = d2/d1,
// G = dout . vbar with vbar = O1/d1, and D = dout . o + G tbar with o = (1 + tbar) vbar - O2/d1.
template <bool STATS>
__global__ void __launch_bounds__(NTHREADS, 1)
parallax_tc_kernel(const __nv_bfloat16* __restrict__ q, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __nv_bfloat16* __restrict__ rp,
                   int T, int BH, float inv_h, __nv_bfloat16* __restrict__ out,
                   const __nv_bfloat16* __restrict__ dout, float* __restrict__ stats,
                   int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
  const int nb = (jend + KB - 1) / KB;
  const long long base = bh * T;

  // Q and R tiles (zero rows past the end of the sequence).
  for (int e = tid; e < 2 * BM * (D / 8); e += NTHREADS) {
    const int which = e / (BM * (D / 8)), ee = e % (BM * (D / 8));
    const int r = ee >> 3, c = ee & 7;
    const __nv_bfloat16* src = which ? rp : q;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < nq) val = *reinterpret_cast<const uint4*>(src + (base + i0 + r) * D + c * 8);
    *reinterpret_cast<uint4*>(smem + (which ? SM_R : SM_Q) + kmaj_off(r, c)) = val;
  }
  if (tid == 0) {
    for (int s = 0; s < KS; ++s) { mbar_init(&bar.kvfull[s], 1); mbar_init(&bar.kvempty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 8);

    }
    mbar_init(&bar.pfull, 8);
    mbar_init(&bar.rowx, 8);
    mbar_init(&bar.pfree, 1);
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
      // Base descriptors plus start-address offsets in 16-byte units.
      const uint64_t qd = smem_desc(smem_u32(smem + SM_Q), 128, 1024);
      const uint64_t rd = smem_desc(smem_u32(smem + SM_R), 128, 1024);
      // key and value blocks 128-byte swizzled (the TMA copies' layout): K-major keys, the V
      // block as the MN-major B operand (a key's 64 values one 128-byte row, 8-key atoms 1024 B
      // apart)
      const uint64_t kd = smem_desc_sw128(smem_u32(smem + SM_K), 1024);
      const uint64_t vd = smem_desc_sw128(smem_u32(smem + SM_V), 1024);
      constexpr uint32_t id_s = idesc_bf16(BM, KB, false, false);
      constexpr uint32_t id_o = idesc_bf16(BM, DV, false, true);
      constexpr uint32_t stage16 = KV_STAGE >> 4;
      bool ok = true;
      int st = 0;
      uint32_t kpar = 0;
      for (int g = 0; g <= 2 * nb && ok; ++g) {
        if (g < 2 * nb) {
          const int sb = g & 1;
          ok = g >= 2 ? mbar_wait2(&bar.kvfull[st], kpar, &bar.sfree[sb], ((g >> 1) - 1) & 1,
                                   status, TO, abort_p)
                      : mbar_wait(&bar.kvfull[st], kpar, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          fence_proxy_async_smem();  // the stage's cp.async writes, before the async-proxy reads
          const uint64_t kst = kd + (uint64_t)(st * stage16);
          const uint32_t ts = tbase + T_S + sb * KB, tt = tbase + T_T + sb * KB;
#pragma unroll
          for (int s = 0; s < D / 16; ++s) mma_ss(ts, qd + 16 * s, kst + 2 * s, id_s, s > 0);
          if (g >= nb) {
#pragma unroll
            for (int s = 0; s < D / 16; ++s) mma_ss(tt, rd + 16 * s, kst + 2 * s, id_s, s > 0);
          }
          mma_commit(&bar.sfull[sb]);
          if (g < nb) mma_commit(&bar.kvempty[st]);  // max sweep: only Q K^T reads the stage
          if (++st == KS) { st = 0; kpar ^= 1; }
        }
        if (g >= nb + 1) {
          const int h = g - 1 - nb, sth = (h + nb) % KS;
          ok = mbar_wait(&bar.pfull, h & 1, status, TO, abort_p);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vst = vd + (uint64_t)(sth * stage16);
#pragma unroll
          for (int s = 0; s < KB / 16; ++s) {
            const uint64_t vds = vst + (uint64_t)(s * (2048 >> 4));
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            mma_ts(tbase + T_O1, tbase + T_P + s * 8, vds, id_o, acc);
            mma_ts(tbase + T_O2, tbase + T_P2H + s * 8, vds, id_o, acc);
            mma_ts(tbase + T_O2, tbase + T_P2L + s * 8, vds, id_o, 1u);
          }
          mma_commit(&bar.pfree);
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
    // ------------------------------------------------------------------ K/V loader
    // One thread: per block a TMA tensor copy of the 64 keys (and in the main sweep one of the 64
    // values), completing on the stage's barrier kvfull (rows past the head read as zeros; keys
    // past the tile's causal end are masked by the softmax warps).
    if (lane == 0) {
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      int issued = 0;
      for (int g = 0; g < 2 * nb; ++g) {
        const int st = g % KS, b = g < nb ? g : g - nb;
        if (g >= KS && !mbar_wait(&bar.kvempty[st], ((g / KS) - 1) & 1, status, TO, abort_p))
          break;
        const bool withv = g >= nb;
        mbar_arrive_expect_tx(&bar.kvfull[st], withv ? 2 * KV_STAGE : KV_STAGE);
        tma_load_3d(smem + SM_K + st * KV_STAGE, &kmap, 0, b * KB, (int)bh, &bar.kvfull[st]);
        if (withv)
          tma_load_3d(smem + SM_V + st * KV_STAGE, &vmap, 0, b * KB, (int)bh, &bar.kvfull[st]);
        issued = g + 1;
      }
      // Nothing may land in this CTA's shared memory after it exits: wait (bounded) for the
      // copies of the last stages filled; a normal run finds them complete.
      volatile int never = 0;
      for (int g = issued > KS ? issued - KS : 0; g < issued; ++g)
        mbar_wait(&bar.kvfull[g % KS], (g / KS) & 1, status, TO, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ weights + output
    // Two warps per tensor-memory lane quarter (one thread per query row each): `hf` takes
    // columns 32 hf .. 32 hf + 31 of every key block (and of the output); the halves' row max,
    // sums and (STATS) dot products are combined through shared memory on barrier rowx.
    const int quarter = warp & 3, hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float c2 = inv_h * 1.4426950408889634f;  // log2(e) / h
    float* const xp = reinterpret_cast<float*>(smem + SM_X);  // [hf][value][BM]
    auto xput = [&](int v, float x) { xp[(hf * NXV + v) * BM + r] = x; };
    auto xsum = [&](int v) { return xp[v * BM + r] + xp[(NXV + v) * BM + r]; };
    float m = -INFINITY, d1 = 0.f, d2 = 0.f;
    for (int g = 0; g < 2 * nb; ++g) {
      const int sb = g & 1;
      if (!warp_wait(&bar.sfull[sb], (g >> 1) & 1, status, abort_p)) break;
      tc_fence_after();
      const bool main_sweep = g >= nb;
      const int h = g - nb;
      const float mc = m * c2;
      uint32_t sv[32], tv[32];
      tmem_ld16(lane_base + T_S + sb * KB + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
      tmem_ld16(lane_base + T_S + sb * KB + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
      if (main_sweep) {
        tmem_ld16(lane_base + T_T + sb * KB + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&tv[0]));
        tmem_ld16(lane_base + T_T + sb * KB + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&tv[16]));
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.sfree[sb]);
      const int jb = (main_sweep ? h : g) * KB + 32 * hf;
      // keys jb .. jb + 31 all at or before this row: no causal mask (rows past the tile's end
      // have zero queries and finite logits, and nothing of theirs is stored)
      const bool full = jb + 31 <= i;
      if (!main_sweep) {  // max sweep
        if (full) {
#pragma unroll
          for (int c = 0; c < 32; ++c) m = fmaxf(m, __uint_as_float(sv[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (valid && jb + c <= i) m = fmaxf(m, __uint_as_float(sv[c]));
        }
        if (g == nb - 1) {  // the two halves' maxima
          xput(0, m);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.rowx);
          if (!warp_wait(&bar.rowx, 0, status, abort_p)) break;
          m = fmaxf(xp[r], xp[NXV * BM + r]);
        }
        continue;
      }
      uint32_t pw[16], hw[16], lw[16];
      auto weights = [&](auto masked) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float p0, p1;
          if constexpr (decltype(masked)::value) {
            p0 = (valid && jb + c <= i) ? ex2(fmaf(__uint_as_float(sv[c]), c2, -mc)) : 0.f;
            p1 = (valid && jb + c + 1 <= i) ? ex2(fmaf(__uint_as_float(sv[c + 1]), c2, -mc)) : 0.f;
          } else {
            p0 = ex2(fmaf(__uint_as_float(sv[c]), c2, -mc));
            p1 = ex2(fmaf(__uint_as_float(sv[c + 1]), c2, -mc));
          }
          const uint32_t w = pack_bf16(p0, p1);
          pw[c / 2] = w;
          const float r0 = bf16_lo(w), r1 = bf16_hi(w);
          d1 += r0 + r1;
          const float q0 = r0 * __uint_as_float(tv[c]);
          const float q1 = r1 * __uint_as_float(tv[c + 1]);
          d2 += q0 + q1;
          const uint32_t hh = pack_bf16(q0, q1);
          hw[c / 2] = hh;
          lw[c / 2] = pack_bf16(q0 - bf16_lo(hh), q1 - bf16_hi(hh));
        }
      };
      if (full) weights(std::false_type{});
      else weights(std::true_type{});
      // one P buffer: the previous block's P V MMAs must have completed
      if (h >= 1 && !warp_wait(&bar.pfree, (h - 1) & 1, status, abort_p)) break;
      tc_fence_after();
      tmem_st8(lane_base + T_P + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&pw[0]));
      tmem_st8(lane_base + T_P + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&pw[8]));
      tmem_st8(lane_base + T_P2H + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&hw[0]));
      tmem_st8(lane_base + T_P2H + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&hw[8]));
      tmem_st8(lane_base + T_P2L + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&lw[0]));
      tmem_st8(lane_base + T_P2L + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&lw[8]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.pfull);
      if (h == nb - 1) {
        // the halves' d1 and d2 (summed in a fixed order), then this half's output columns
        xput(1, d1);
        xput(2, d2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.rowx);
        if (!warp_wait(&bar.rowx, 1, status, abort_p)) break;
        const float D1 = xsum(1), D2 = xsum(2);
        if (!warp_wait(&bar.accfull, 0, status, abort_p)) break;
        tc_fence_after();
        const float inv = 1.f / D1;
        const float f1 = (1.f + D2 * inv) * inv;
        float gs = 0.f, od = 0.f;  // STATS: dout . vbar, dout . o over this half's columns
#pragma unroll
        for (int c1 = 0; c1 < DV / 2; c1 += 16) {
          const int c0 = (DV / 2) * hf + c1;
          uint32_t o1[16], o2[16];
          tmem_ld16(lane_base + T_O1 + c0, o1);
          tmem_ld16(lane_base + T_O2 + c0, o2);
          tmem_ld_wait();
          if (STATS) {
            if (valid) {
              const uint4* dy = reinterpret_cast<const uint4*>(dout + (base + i) * DV + c0);
#pragma unroll
              for (int hv = 0; hv < 2; ++hv) {
                const uint4 w4 = dy[hv];
                const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                  const int cc = 8 * hv + t;
                  const float dyv = (t & 1) ? bf16_hi(ws[t / 2]) : bf16_lo(ws[t / 2]);
                  const float o1v = __uint_as_float(o1[cc]), o2v = __uint_as_float(o2[cc]);
                  gs = fmaf(dyv, o1v * inv, gs);
                  od = fmaf(dyv, fmaf(o1v, f1, -o2v * inv), od);
                }
              }
            }
          } else if (valid) {
            uint32_t packed[8];
#pragma unroll
            for (int t = 0; t < 16; t += 2)
              packed[t / 2] =
                  pack_bf16(fmaf(__uint_as_float(o1[t]), f1, -__uint_as_float(o2[t]) * inv),
                            fmaf(__uint_as_float(o1[t + 1]), f1, -__uint_as_float(o2[t + 1]) * inv));
            uint4* dst = reinterpret_cast<uint4*>(out + (base + i) * DV + c0);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
        if (STATS) {
          xput(3, gs);
          xput(4, od);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.rowx);
          if (!warp_wait(&bar.rowx, 0, status, abort_p)) break;  // phase 2
          if (hf == 0 && valid) {
            const float G = xsum(3), Od = xsum(4);
            const float tbar = D2 * inv;
            *reinterpret_cast<float4*>(stats + (base + i) * 8) = make_float4(m, inv, tbar, G);
            stats[(base + i) * 8 + 4] = fmaf(G, tbar, Od);
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

}  // namespace ptc

// ============================================================================ CUDA cores
namespace pcc {

constexpr int BQ = 64;   // queries per block
constexpr int BK = 32;   // keys per shared-memory tile
constexpr int NTHREADS = BQ * 4;

template <typename TIn, int D, int DV>
__global__ void __launch_bounds__(NTHREADS)
parallax_cc_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                   const TIn* __restrict__ rp, int T, int BH, float inv_h, TIn* __restrict__ out) {
  constexpr int DQ = D / 4, DVQ = DV / 4;
  __shared__ float ks[BK][D + 1];
  __shared__ float vs[BK][DV + 1];
  const int tid = threadIdx.x;
  const int part = tid & 3, rl = tid >> 2;
  const int ntiles = (T + BQ - 1) / BQ;
  const int tile = ntiles - 1 - (int)(blockIdx.x / BH);
  const long long bh = blockIdx.x % BH;
  const long long base = bh * T;
  const int i0 = tile * BQ;
  const int i = i0 + rl;
  const bool valid = i < T;
  const int jend = min(T, i0 + BQ);
  const unsigned gmask = 0xFu << ((threadIdx.x & 31) & ~3);  // the four threads of this query

  // This thread's coordinates a = part + 4u of q and r, and c = part + 4u of the outputs.
  float qv[DQ], rv[DQ], o1[DVQ], o2[DVQ];
#pragma unroll
  for (int u = 0; u < DQ; ++u) {
    qv[u] = valid ? ldf(q, (base + i) * D + part + 4 * u) * inv_h : 0.f;
    rv[u] = valid ? ldf(rp, (base + i) * D + part + 4 * u) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < DVQ; ++u) o1[u] = o2[u] = 0.f;
  float m = -INFINITY, d1 = 0.f, d2 = 0.f;

  for (int j0 = 0; j0 < jend; j0 += BK) {
    __syncthreads();
    for (int e = tid; e < BK * D; e += NTHREADS) {
      const int jj = e / D, a = e % D;
      ks[jj][a] = j0 + jj < jend ? ldf(k, (base + j0 + jj) * D + a) : 0.f;
    }
    for (int e = tid; e < BK * DV; e += NTHREADS) {
      const int jj = e / DV, c = e % DV;
      vs[jj][c] = j0 + jj < jend ? ldf(v, (base + j0 + jj) * DV + c) : 0.f;
    }
    __syncthreads();
    const int nj = min(BK, (valid ? i + 1 : 0) - j0);  // keys of this tile in the causal prefix
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f, t = 0.f;
#pragma unroll
      for (int u = 0; u < DQ; ++u) {
        s = fmaf(qv[u], ks[jj][part + 4 * u], s);
        t = fmaf(rv[u], ks[jj][part + 4 * u], t);
      }
      s += __shfl_xor_sync(gmask, s, 1);
      t += __shfl_xor_sync(gmask, t, 1);
      s += __shfl_xor_sync(gmask, s, 2);
      t += __shfl_xor_sync(gmask, t, 2);
      if (s > m) {  // running max: rescale what was accumulated against the old one
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
  if (valid) {
    const float inv = 1.f / d1;
    const float f1 = (1.f + d2 * inv) * inv;
#pragma unroll
    for (int u = 0; u < DVQ; ++u)
      stf(out, (base + i) * DV + part + 4 * u, fmaf(o1[u], f1, -o2[u] * inv));
  }
}

template <typename TIn, int D, int DV>
cudaError_t launch_cc(const Args& a, const void* r, cudaStream_t s) {
  const long long blocks = (long long)((a.T + BQ - 1) / BQ) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  parallax_cc_kernel<TIn, D, DV><<<(unsigned)blocks, NTHREADS, 0, s>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
      static_cast<const TIn*>(r), a.T, (int)a.BH(), 1.0f / a.h, static_cast<TIn*>(a.out));
  count_launch();
  return cudaGetLastError();
}

template <typename TIn, int D>
cudaError_t dispatch_dv(const Args& a, const void* r, cudaStream_t s) {
  switch (a.dv) {
    case 16: return launch_cc<TIn, D, 16>(a, r, s);
    case 32: return launch_cc<TIn, D, 32>(a, r, s);
    default: return launch_cc<TIn, D, 64>(a, r, s);
  }
}

template <typename TIn>
cudaError_t dispatch_d(const Args& a, const void* r, cudaStream_t s) {
  switch (a.d) {
    case 16: return dispatch_dv<TIn, 16>(a, r, s);
    case 32: return dispatch_dv<TIn, 32>(a, r, s);
    default: return dispatch_dv<TIn, 64>(a, r, s);
  }
}

}  // namespace pcc

// Tensor maps of the keys and values ([BH][T][64] bf16, boxes of 64 rows x 64 features, 128-byte
// swizzled) for the tensor-core kernel.
cudaError_t parallax_kv_maps(const void* k, const void* v, int T, long long BH, CUtensorMap* kmap,
                             CUtensorMap* vmap) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint32_t ones[3] = {1, 1, 1};
  const cuuint64_t dims[3] = {(cuuint64_t)ptc::D, (cuuint64_t)T, (cuuint64_t)BH};
  const cuuint64_t str[2] = {(cuuint64_t)ptc::D * 2, (cuuint64_t)T * ptc::D * 2};
  const cuuint32_t box[3] = {(cuuint32_t)ptc::D, (cuuint32_t)ptc::KB, 1};
  static_assert(ptc::D == ptc::DV, "one tensor-map shape for keys and values");
  for (int t = 0; t < 2; ++t)
    if (encode(t ? vmap : kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(t ? v : k),
               dims, str, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace

// The backward's row scalars (bf16, d = dv = 64): the tensor-core forward with the STATS epilogue.
cudaError_t launch_parallax_stats_tc(const ParallaxBwdArgs& a, float* stats, int* status,
                                     cudaStream_t s) {
  CUtensorMap kmap, vmap;
  cudaError_t err = parallax_kv_maps(a.k, a.v, a.T, a.BH(), &kmap, &vmap);
  if (err != cudaSuccess) return err;
  auto kern = ptc::parallax_tc_kernel<true>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ptc::SMEM_LAUNCH);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)((a.T + ptc::BM - 1) / ptc::BM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, ptc::NTHREADS, ptc::SMEM_LAUNCH, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), kmap, vmap,
      static_cast<const __nv_bfloat16*>(a.r), a.T,
      (int)a.BH(), 1.0f / a.h, nullptr, static_cast<const __nv_bfloat16*>(a.dout), stats, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_parallax(const Args& a, const void* r, int path, int* status, cudaStream_t s) {
  if (path == kPathTensorCore && a.dtype == LLA_BF16 && a.d == 64 && a.dv == 64) {
    CUtensorMap kmap, vmap;
    cudaError_t err = parallax_kv_maps(a.k, a.v, a.T, a.BH(), &kmap, &vmap);
    if (err != cudaSuccess) return err;
    auto kern = ptc::parallax_tc_kernel<false>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ptc::SMEM_LAUNCH);
    if (err != cudaSuccess) return err;
    const long long blocks = (long long)((a.T + ptc::BM - 1) / ptc::BM) * a.BH();
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)blocks, ptc::NTHREADS, ptc::SMEM_LAUNCH, s>>>(
        static_cast<const __nv_bfloat16*>(a.q), kmap, vmap, static_cast<const __nv_bfloat16*>(r),
        a.T,
        (int)a.BH(), 1.0f / a.h, static_cast<__nv_bfloat16*>(a.out), nullptr, nullptr, status);
    count_launch();
    return cudaGetLastError();
  }
  return a.dtype == LLA_F32 ? pcc::dispatch_d<float>(a, r, s)
                            : pcc::dispatch_d<__nv_bfloat16>(a, r, s);
}

}  // namespace lla
