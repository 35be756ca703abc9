// Tensor-core readout stage of the causal LLA forward (bf16 inputs, d = dv = 64; tcgen05 + TMEM).
//
// With y_i = (C_kk + lambda' I)^-1 (q_i - kbar_i) from the ridge solve, one streaming pass over
// the causal prefix evaluates the centred closed form of the LLA intercept ("Parallax" blog, s.2
// Canonical Formulation)
//   o_i = vbar_i + C_vk y_i = O1_i / omega_i + O2_i,
//   O1 = P V,  O2 = (P .* t) V,  t_ij = k_j . y_i - kbar_i . y_i,
// and, since omega_i (the sum of the rounded weights) is known before this pass, as one product
//   o_i = (P .* A) V,  a_ij = 1 / omega_i + t_ij  (kFused: the centred form's bf16 output),
// where P holds the kernel weights exactly as the moments stage rounded them: the pass reads them
// back from the moments stage's weight scratch (bf16 images already in the layout of a tcgen05
// operand), so the fitted moments and this pass describe one weighted problem (and
// sum_j p_ij t_ij = 0 up to rounding), and neither Q K^T nor an exponential is recomputed. The
// pass has the two-branch shape of the blog's streaming algorithm (s.3 "One extra branch, no extra
// I/O"): a softmax branch (O1, omega) and a covariance branch (O2) over the same K/V tiles.
//
// Precision: y can be large (small ridge, rank-deficient early prefixes), and its component
// outside the span of the keys must cancel between k_j . y and kbar . y; y therefore enters the
// Y K^T contraction as three exact bf16 parts (y = y1 + y2 + y3, 24 significant bits; the solve
// writes them, with cy = kbar . y), and the covariance-branch weights p * t enter P2 V as an
// exact-to-16-bits hi/lo pair (kFused: the fused weights p * (1/omega + t) as that pair, which
// rounds the softmax part p / omega to 2^-17 of |p (1/omega + t)|, ~1e-5 of the output).
//
// With the page form of the solve (y := rho* = Sigma^-1 mu, cy := q . rho*; kPage), t_ij is the
// page's z_ij . rho* with z = k - q, and the same two branches give the page's exact-LLA epilogue
// ("Parallax" blog, s.2 Canonical Formulation and Appendix B):
//   o_i = sum p (1 - t) v / sum p (1 - t) = (O1_i - O2_i) / (omega_i - d2_i),  d2 = sum_j p_ij t_ij.
//
// The same pass, with V := K and y := a conjugate-gradient direction p and only the covariance
// branch kept (kMatvec), returns C_kk p: the matrix-free product that the CG strategy for the
// ridge system needs (C_kk p = sum_j p_ij ((k_j - kbar) . p) k_j). Tiles whose flag in
// `tile_active` is 0 are skipped.
//
// One CTA per 128-query tile; keys in chunks of 64 (two weight images). Warp roles (7 warps):
// 0 issues T = Y K^T (12 MMAs per chunk, N = 64) and owns the TMEM allocation; 6 issues
// O1 += P V (P straight from shared memory) and O2 += P2 V (P2 from tensor memory), 12 MMAs per
// chunk; 1 stages the key and value chunks by TMA tensor copies (128-byte swizzled, read by the
// MMAs through swizzled descriptors) and the weight images by a bulk copy; 2-5 (one thread per
// query = TMEM lane) turn
// T and P into P2 and write the output. Two issuing threads, because each tcgen05.mma costs its
// issuing thread about as long as the tensor core takes to run one of these. All waits are
// bounded.
#include <cstdint>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"
#include "lla_tmap.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int DV = 64;
constexpr int BM = 128;                 // query rows per CTA = TMEM lanes
constexpr int CK = 64;                  // keys per chunk
constexpr int KS = 5;                   // chunk pipeline stages
constexpr int NWARPS = 7;
constexpr int NTHREADS = NWARPS * 32;
static_assert(BM == pscr::kRows && CK == 2 * pscr::kKeys, "a chunk is two weight images");

// tensor-memory columns
constexpr uint32_t T_O1 = 0;            // 64 fp32: P V
constexpr uint32_t T_O2 = 64;           // 64 fp32: P2 V
constexpr uint32_t T_T = 128;           // 2 x 64 fp32: Y K^T
constexpr uint32_t T_P2H = 256;         // 2 x 32: bf16 hi part of P .* t (64 keys)
constexpr uint32_t T_P2L = 320;         // 2 x 32: bf16 lo part
constexpr uint32_t TMEM_COLS = 512;
static_assert(T_P2L + 2 * (CK / 2) <= TMEM_COLS, "tensor memory budget");

// shared memory (bytes)
constexpr int TILE = BM * D * 2;                    // 128 x 64 bf16 = 16 KiB
constexpr int SM_Y = 0;                             // 3 tiles: y1, y2, y3
constexpr int KV_BYTES = CK * D * 2;                // 8 KiB: one key or value chunk
constexpr int P_BYTES = 2 * pscr::kBlockBytes;      // 16 KiB: the chunk's two weight images
constexpr int STAGE = 2 * KV_BYTES + P_BYTES;       // K, V, P of one chunk
constexpr int SM_ST = SM_Y + 3 * TILE;
constexpr int SM_BAR = SM_ST + KS * STAGE;
constexpr int SMEM_BYTES = SM_BAR + 256;
constexpr int SMEM_LAUNCH = SMEM_BYTES + 1024;  // slack for aligning the base to 1024 bytes
static_assert(SMEM_LAUNCH <= 227 * 1024, "shared memory budget");
static_assert(SM_ST % 1024 == 0 && STAGE % 1024 == 0 && KV_BYTES % 1024 == 0,
              "128-byte swizzled stages on 1024-byte boundaries");

// Byte offset of 16-byte chunk c (elements 8c..8c+7) of row r in a K-major tile whose rows hold
// 64 elements: core matrix (r / 8, c) of 128 bytes, row groups 1024 bytes apart.
__device__ __forceinline__ int kmaj_off(int r, int c) { return (r >> 3) * 1024 + c * 128 + (r & 7) * 16; }

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
  uint64_t pfull[KS];    // the chunk's weight images have landed (bulk copy, transaction count)
  uint64_t tfull[2], tfree[2];
  uint64_t p2full[2], p2free[2];
  uint64_t accfull, done_t, done_o;
};
static_assert(sizeof(Barriers) <= 256, "barrier region");

template <typename TOut, bool kMatvec, bool kPage, bool kFused>
__global__ void __launch_bounds__(NTHREADS, 1)
readout_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const uint4* __restrict__ pimg, const uint32_t* __restrict__ ytc,
                  const float* __restrict__ cy_in, const float* __restrict__ omega_in, int T,
                  int BH, TOut* __restrict__ out, const int* __restrict__ tile_active,
                  int* __restrict__ status) {
  static_assert(!kFused || (!kMatvec && !kPage), "the fused product is the centred form's");
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
  const int nck = (jend + CK - 1) / CK;
  const long long base = bh * T;
  if (tile_active && !tile_active[bh * ntiles + tile]) return;  // the whole CTA, before any setup
  // This tile's weight images: tile = 2 ptile + rank in the moments stage's pairing.
  const int ptile = tile >> 1, rank = tile & 1;
  const uint4* const pt = pimg + pscr::first_block(bh, T, ptile, rank) * (pscr::kBlockBytes / 16);
  const int nimg = pscr::pair_blocks(T, ptile);

  // The three parts of the tile's Y (rows of 64 bf16) into the core-matrix layout, by all
  // threads (rows past the tile's end are zero-filled).
  for (int e = tid; e < 3 * BM * 8; e += NTHREADS) {
    const int part = e / (BM * 8), rem = e % (BM * 8), r = rem >> 3, c = rem & 7;
    const bool in = r < nq;
    const uint32_t* src = ytc + ((base + i0 + (in ? r : 0)) * 3 + part) * (D / 2) + c * 4;
    cp_async16(smem + SM_Y + part * TILE + kmaj_off(r, c), src, in ? 16u : 0u);
  }
  cp_async_commit();
  cp_async_wait<0>();
  if (tid == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar.kvfull[s], 1);  // the loader's arrival with the key and value bytes
      mbar_init(&bar.kvempty[s], 1);
      mbar_init(&bar.pfull[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.tfull[s], 1);
      mbar_init(&bar.tfree[s], 4);
      mbar_init(&bar.p2full[s], 4);
      mbar_init(&bar.p2free[s], 1);
    }
    mbar_init(&bar.accfull, 1);
    mbar_init(&bar.done_t, 1);
    mbar_init(&bar.done_o, 1);
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
  constexpr uint32_t stage16 = STAGE >> 4;

  if (warp == 0) {
    // ------------------------------------------------------------------ T = Y K^T issuer
    if (lane == 0) {
      // Base descriptors plus start-address offsets in 16-byte units (see the moments stage).
      const uint64_t yd = smem_desc(smem_u32(smem + SM_Y), 128, 1024);
      const uint64_t kd = smem_desc_sw128(smem_u32(smem + SM_ST), 1024);
      constexpr uint32_t id_t = idesc_bf16(BM, CK, false, false);
      constexpr uint32_t tile16 = TILE >> 4;
      bool ok = true;
      for (int c = 0; c < nck && ok; ++c) {
        const int st = c % KS, tb = c & 1;
        ok = mbar_wait(&bar.kvfull[st], (c / KS) & 1, status, kStatusTimeout, abort_p);
        if (ok && c >= 2)
          ok = mbar_wait(&bar.tfree[tb], ((c >> 1) - 1) & 1, status, kStatusTimeout, abort_p);
        if (!ok) break;
        tc_fence_after();
        fence_proxy_async_smem();  // the stage's cp.async writes, before the async-proxy reads
        const uint64_t kst = kd + (uint64_t)(st * stage16);
        const uint32_t tt = tbase + T_T + tb * CK;
#pragma unroll
        for (int part = 0; part < 3; ++part)
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            mma_ss(tt, yd + part * tile16 + 16 * s, kst + 2 * s, id_t,  // K-steps: 32 B in a row
                   (part > 0 || s > 0) ? 1u : 0u);
        mma_commit(&bar.tfull[tb]);
      }
      if (!ok) *abort_p = 1;
      mma_commit(&bar.done_t);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------------ O1, O2 issuer
    if (lane == 0) {
      // P images as the K-major A operand (K-adjacent core matrices 2048 B apart, M-adjacent
      // 128 B); the V chunk as the MN-major B operand, 128-byte swizzled: a key's 64 values are
      // one 128-byte row, 8-key atoms 1024 B apart.
      const uint64_t pd = smem_desc(smem_u32(smem + SM_ST + 2 * KV_BYTES), 2048, 128);
      const uint64_t vd = smem_desc_sw128(smem_u32(smem + SM_ST + KV_BYTES), 1024);
      constexpr uint32_t id_o = idesc_bf16(BM, DV, false, true);
      bool ok = true;
      for (int c = 0; c < nck && ok; ++c) {
        const int st = c % KS, pb = c & 1;
        ok = mbar_wait2(&bar.kvfull[st], (c / KS) & 1, &bar.p2full[pb], (c >> 1) & 1, status,
                        kStatusTimeout, abort_p) &&
             mbar_wait(&bar.pfull[st], (c / KS) & 1, status, kStatusTimeout, abort_p);
        if (!ok) break;
        tc_fence_after();
        fence_proxy_async_smem();
        const uint64_t vst = vd + (uint64_t)(st * stage16);
        const uint64_t pst = pd + (uint64_t)(st * stage16);
#pragma unroll
        for (int s = 0; s < CK / 16; ++s) {
          const uint64_t vds = vst + (uint64_t)(s * (2048 >> 4));  // keys 16s.. : 2 x 1024 B
          // keys 16s..16s+15: image s / 2, K-adjacent core matrices 2 (s % 2), 2 (s % 2) + 1
          const uint64_t pds = pst + (uint64_t)((s >> 1) * (pscr::kBlockBytes >> 4) + (s & 1) * (4096 >> 4));
          const uint32_t acc = (c > 0 || s > 0) ? 1u : 0u;
          if (!kMatvec && !kFused) mma_ss(tbase + T_O1, pds, vds, id_o, acc);
          mma_ts(tbase + T_O2, tbase + T_P2H + pb * (CK / 2) + s * 8, vds, id_o, acc);
          mma_ts(tbase + T_O2, tbase + T_P2L + pb * (CK / 2) + s * 8, vds, id_o, 1u);
        }
        mma_commit(&bar.p2free[pb]);
        mma_commit(&bar.kvempty[st]);  // T's reads of this stage completed before p2full
        if (c == nck - 1) mma_commit(&bar.accfull);
      }
      if (!ok) *abort_p = 1;
      mma_commit(&bar.done_o);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ K/V/P loader
    // One thread: per chunk a TMA tensor copy of the 64 keys and one of the 64 values (rows past
    // the head read as zeros; keys past the tile's causal end have zero weights), completing on
    // the stage's barrier kvfull, and one bulk copy of the chunk's two weight images as they are
    // (pfull). A tile's images cover its chunks: pair_blocks counts blocks up to the pair's last
    // key, in pairs.
    if (lane == 0) {
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      int issued = 0;
      for (int c = 0; c < nck; ++c) {
        const int st = c % KS;
        if (c >= KS && !mbar_wait(&bar.kvempty[st], ((c / KS) - 1) & 1, status, kStatusTimeout,
                                  abort_p))
          break;
        uint8_t* kdst = smem + SM_ST + st * STAGE;
        mbar_arrive_expect_tx(&bar.kvfull[st], 2 * KV_BYTES);
        tma_load_3d(kdst, &kmap, 0, c * CK, (int)bh, &bar.kvfull[st]);
        tma_load_3d(kdst + KV_BYTES, &vmap, 0, c * CK, (int)bh, &bar.kvfull[st]);
        mbar_arrive_expect_tx(&bar.pfull[st], P_BYTES);
        bulk_g2s(kdst + 2 * KV_BYTES, pt + (long long)2 * c * (pscr::kBlockBytes / 16), P_BYTES,
                 &bar.pfull[st]);
        issued = c + 1;
      }
      // Nothing may land in this CTA's shared memory after it exits: wait (bounded) for the
      // copies of the last stages filled; a normal run finds them complete.
      volatile int never = 0;
      for (int c = issued > KS ? issued - KS : 0; c < issued; ++c) {
        mbar_wait(&bar.kvfull[c % KS], (c / KS) & 1, status, kStatusTimeout, &never);
        mbar_wait(&bar.pfull[c % KS], (c / KS) & 1, status, kStatusTimeout, &never);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ weights + output
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float cy = valid ? cy_in[base + i] : 0.f;  // kbar . y (page form: q . rho*)
    const bool store = valid && __float_as_uint(cy) != kListedBits;  // else the exact pass writes
    const float inv_om = kFused && valid ? 1.f / omega_in[base + i] : 0.f;
    float om = 0.f, d2 = 0.f;
    bool ok = true;
    for (int c = 0; c < nck; ++c) {
      const int st = c % KS, tb = c & 1;
      if (!warp_wait(&bar.pfull[st], (c / KS) & 1, status, abort_p) ||
          !warp_wait(&bar.tfull[tb], (c >> 1) & 1, status, abort_p)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t tv[CK];
#pragma unroll
      for (int q4 = 0; q4 < CK / 16; ++q4)
        tmem_ld16(lane_base + T_T + tb * CK + 16 * q4, *reinterpret_cast<uint32_t(*)[16]>(&tv[16 * q4]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.tfree[tb]);
      // This row's 64 weights: 16-byte chunk kc of image m at m * 8192 + kc * 2048 + r * 16.
      const uint8_t* prow = smem + SM_ST + st * STAGE + 2 * KV_BYTES + r * 16;
      uint32_t hw[CK / 2], lw[CK / 2];
#pragma unroll
      for (int kc = 0; kc < CK / 8; ++kc) {
        const uint4 pv = *reinterpret_cast<const uint4*>(prow + (kc >> 2) * pscr::kBlockBytes + (kc & 3) * 2048);
        const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = 8 * kc + 2 * u;
          const float r0 = bf16_lo(pw[u]), r1 = bf16_hi(pw[u]);
          if (!kFused) om += r0 + r1;
          const float q0 = r0 * ((__uint_as_float(tv[j]) - cy) + inv_om);
          const float q1 = r1 * ((__uint_as_float(tv[j + 1]) - cy) + inv_om);
          if (kPage) d2 += q0 + q1;
          const uint32_t hh = pack_bf16(q0, q1);
          hw[j / 2] = hh;
          lw[j / 2] = pack_bf16(q0 - bf16_lo(hh), q1 - bf16_hi(hh));
        }
      }
      const int pb = c & 1;
      if (c >= 2 && !warp_wait(&bar.p2free[pb], ((c >> 1) - 1) & 1, status, abort_p)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int q4 = 0; q4 < CK / 16; ++q4) {
        tmem_st8(lane_base + T_P2H + pb * (CK / 2) + 8 * q4, *reinterpret_cast<uint32_t(*)[8]>(&hw[8 * q4]));
        tmem_st8(lane_base + T_P2L + pb * (CK / 2) + 8 * q4, *reinterpret_cast<uint32_t(*)[8]>(&lw[8 * q4]));
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p2full[pb]);
    }
    if (ok && warp_wait(&bar.accfull, 0, status, abort_p)) {
      tc_fence_after();
      const float inv = kPage ? 1.f / (om - d2) : 1.f / om;
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 16) {
        uint32_t o1[16], o2[16];
        if (!kMatvec && !kFused) tmem_ld16(lane_base + T_O1 + c0, o1);
        tmem_ld16(lane_base + T_O2 + c0, o2);
        tmem_ld_wait();
        if (store) {
#pragma unroll
          for (int t = 0; t < 16; ++t)
            stf(out, (base + i) * DV + c0 + t,
                (kMatvec || kFused) ? __uint_as_float(o2[t])
                : kPage ? (__uint_as_float(o1[t]) - __uint_as_float(o2[t])) * inv
                        : fmaf(__uint_as_float(o1[t]), inv, __uint_as_float(o2[t])));
        }
      }
    }
  }

  // Teardown: tensor memory is released only after every MMA of both issuers has completed
  // (bounded waits, whatever the abort flag says).
  if (warp == 0 && lane == 0) {
    volatile int never = 0;
    mbar_wait(&bar.done_t, 0, status, kStatusTimeout, &never);
    mbar_wait(&bar.done_o, 0, status, kStatusTimeout, &never);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

template <typename TOut, bool kMatvec, bool kPage = false, bool kFused = false>
cudaError_t launch_ro(const Args& a, const Workspace& ws, cudaStream_t s, const void* keys,
                      const void* v, const uint32_t* ytc, const float* cy, TOut* out,
                      const int* tile_active) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  // keys and values: [BH][T][64] bf16, boxes of 64 rows x 64 features, 128-byte swizzled
  CUtensorMap kmap, vmap;
  const cuuint32_t ones[3] = {1, 1, 1};
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.T, (cuuint64_t)a.BH()};
  const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.T * D * 2};
  const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)CK, 1};
  static_assert(D == DV, "one tensor-map shape for keys and values");
  for (int t = 0; t < 2; ++t)
    if (encode(t ? &vmap : &kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void*>(t ? v : keys), dims, str, box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  auto kern = readout_tc_kernel<TOut, kMatvec, kPage, kFused>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
  if (err != cudaSuccess) return err;
  const long long blocks = (long long)((a.T + BM - 1) / BM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, NTHREADS, SMEM_LAUNCH, s>>>(
      kmap, vmap, static_cast<const uint4*>(ws.pscr), ytc, cy, ws.omega, a.T, (int)a.BH(), out,
      tile_active, ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_readout_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  // the keys in the frame the moments and the solve used (unshifted for the CG strategy)
  const void* keys = ws.path == kPathTensorCore ? static_cast<const void*>(ws.ksh) : a.k;
  return ws.form == kFormPage
             ? launch_ro<__nv_bfloat16, false, true>(a, ws, s, keys, a.v, ws.ytc, ws.cy, out,
                                                     nullptr)
             : launch_ro<__nv_bfloat16, false, false, true>(a, ws, s, keys, a.v, ws.ytc, ws.cy, out,
                                                            nullptr);
}

cudaError_t launch_readout_tc_f32(const Args& a, const Workspace& ws, cudaStream_t s,
                                  const void* v, const uint32_t* ytc, const float* cy, float* out,
                                  const int* tile_active, bool matvec) {
  return matvec ? launch_ro<float, true>(a, ws, s, a.k, v, ytc, cy, out, tile_active)
                : launch_ro<float, false>(a, ws, s, a.k, v, ytc, cy, out, tile_active);
}

}  // namespace lla
