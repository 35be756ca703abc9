// Weight sweeps of the tensor-core moments stage of the causal LLA forward (bf16 inputs, d = 64;
// tcgen05 + TMEM).
//
// For every query i and its causal prefix j <= i this kernel computes the kernel weights of the
// closed form of LLA ("Parallax" blog, s.2 Canonical Formulation), max-shifted:
//     p_ij = exp((q_i . k_j - m_i) / h),  m_i = max_{j <= i} q_i . k_j,
// rounded to bf16 and stored as tcgen05 operand images (the weight scratch, pscr:: in the internal
// header), which the moment contraction and the readout read back; and per row m_i / h and
// omega_i = sum_j p_ij (the sum of the rounded weights, so that every later stage describes one
// weighted problem). Keys are the original bf16 keys: the weights do not depend on the key frame.
//
// Two sweeps over the key prefix: the first finds the exact row max, the second forms the weights.
// Q K^T runs on chunks of four 32-key blocks (N = 128; a tcgen05.mma costs about as long at N = 32
// as at N = 128) on CTA pairs (cluster of two, cta_group::2, M = 256): each CTA holds 128 query rows
// (its tensor-memory lanes) and stages half of every key block (16 keys), and the even CTA (the
// leader) issues the MMAs. The logits of a chunk land in one of three tensor-memory buffers, so
// Q K^T runs ahead of the softmax warps.
//
// Warp roles per CTA (18 warps): 0 issues Q K^T (leader; one thread) and owns the tensor-memory
// allocation, and in the peer relays its landed key blocks to the leader; 1 stages key blocks by
// TMA tensor copies (one thread; 128-byte swizzled, the layout the Q K^T B operand reads);
// 2-17 are the softmax warps: four per tensor-memory lane quarter, each taking 8 keys of every
// block (one thread per query row), so that a block's chain of tensor-memory load, exponentials,
// packing and stores is short. Every mbarrier wait is bounded.
#include <cstdint>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"
#include "lla_tmap.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int BM = 128;                     // query rows per CTA = TMEM lanes
constexpr int PM = 2 * BM;                  // query rows per CTA pair = MMA M
constexpr int KB = 32;                      // keys per block
constexpr int SCH = 4;                      // key blocks per sweep chunk (one Q K^T of N = 128)
constexpr int KS = 32;                      // key-tile pipeline stages (eight sweep chunks)
constexpr int KC = KS / 4;                  // chunk slots: the stages of a chunk fill and free together
constexpr int NSM = 16;                     // softmax warps: four per TMEM lane quarter
constexpr int NPART = NSM / 4;              // parts of a block's keys (8 keys each)
constexpr int NWARPS = 2 + NSM;             // + Q K^T issuer, key loader
constexpr int NTHREADS = NWARPS * 32;
constexpr int NSC = 3;                      // S buffers (SCH blocks each)
static_assert(BM == pscr::kRows && KB == pscr::kKeys && PM == 2 * BM, "weight scratch layout");
static_assert(KB == 8 * NPART, "a part is one 16-byte chunk of a block's image row");

// tensor-memory columns (the same in both CTAs of a pair)
constexpr uint32_t T_S = 0;                       // NSC x 128 columns of fp32 logits
constexpr uint32_t T_Q = NSC * SCH * KB;          // 32 columns: the Q tile, A operand of Q K^T
constexpr uint32_t TMEM_COLS = 512;
static_assert(T_Q + D / 2 <= TMEM_COLS, "tensor memory budget");

// shared-memory layout (bytes; the same offsets in both CTAs of a pair)
constexpr int SM_K = 0;                              // KS x (16 x 64 bf16)
constexpr int K_STAGE = KB / 2 * D * 2;              // the 16 keys of a block this CTA contributes
constexpr int K_SLOT = SCH * K_STAGE;                // a chunk slot: 64 keys, 8 KiB
constexpr int SM_BAR = SM_K + KS * K_STAGE;
constexpr int SMEM_BYTES = SM_BAR + 8192;
// More than half of an SM's shared memory, so that at most one CTA (and one TMEM allocation of
// all 512 columns) is resident per SM.
constexpr int SMEM_LAUNCH = SMEM_BYTES + 1024 > 120 * 1024 ? SMEM_BYTES + 1024 : 120 * 1024;
constexpr int P_BLOCK = BM * KB * 2;  // one 8 KiB image

// A key stage holds the 16 keys of a block that this CTA contributes to Q K^T: 16 rows of 128
// bytes in the 128-byte swizzled layout of the TMA copy (two 1024-byte atoms of 8 rows). The
// stages form chunk slots of SCH = 4 consecutive stages (8 KiB), so that a slot is one K-major
// N = 128 operand for the pair (64 keys from each CTA, atoms 1024 bytes apart).
static_assert(KS % SCH == 0 && SCH == 4 && K_STAGE == 2048 && K_SLOT == SCH * K_STAGE,
              "key stage layout");

// Barriers marked (L) are used in the leader CTA only and collect arrivals from both CTAs; those
// marked (M) are arrived on by multicast commits from the leader's Q K^T issuer in both CTAs.
struct Barriers {
  uint64_t kfull[KC];       // the chunk's four key blocks staged by this CTA's loader
  uint64_t kfull_peer[KC];  // (L) the same in the peer
  uint64_t kempty[KC];      // (M) the chunk's stages consumed by Q K^T
  uint64_t sfull[NSC];      // (M) S = Q K^T of a sweep chunk in tensor memory
  uint64_t sfree[NSC];      // (L) S read by both CTAs' softmax warps
  uint64_t qready;          // (L) both CTAs' Q tiles in tensor memory
  uint64_t done_qk;         // (M) every MMA of the Q K^T issuer completed
  uint64_t rowx;            // this CTA's softmax parts exchanged row max / omega
  uint32_t tmem_base;
  int abort_flag;
  float part_m[NPART][BM];  // per-row partial maxima of the parts
  float part_o[NPART][BM];  // per-row partial weight sums of the parts (a separate array: a fast
                            // warp may finish the weight sweep before a slow one has read the maxima)
};
static_assert(sizeof(Barriers) <= 8192, "barrier region");

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
weights_tc_kernel(const __nv_bfloat16* __restrict__ q, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap kmap5, bool chunk_copies, int T, int BH, float inv_h, float* __restrict__ m_out,
                  float* __restrict__ omega_out, uint4* __restrict__ pimg, int fault,
                  int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzled key stages need 1024-byte alignment
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + SM_BAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;
  const int npairs = (T + PM - 1) / PM;
  const int pair_lin = (int)(blockIdx.x >> 1);
  const int ptile = npairs - 1 - pair_lin / BH;  // longest causal prefixes first
  const long long bh = pair_lin % BH;
  const int i0p = ptile * PM;
  const int i0 = i0p + rank * BM;                // this CTA's first query row
  const int nq = max(0, min(BM, T - i0));
  const int jend = min(T, i0p + PM);             // both CTAs stream the pair's key prefix
  const int nb = pscr::pair_blocks(T, ptile);    // even: a last block past jend has zero weights
  const int nb4 = (nb + SCH - 1) / SCH * SCH;    // each sweep padded with zero blocks to chunks
  const int G = 2 * nb4;                         // key blocks streamed: max sweep, weight sweep
  const long long base = bh * T;
  uint4* const ptile_p = pimg + pscr::first_block(bh, T, ptile, rank) * (P_BLOCK / 16);
  // Rows of this CTA's key stage: the Q K^T operand takes rows 0..15 of each CTA's stage as its
  // N/2 keys, so CTA 1 keeps keys 16..31 of a block in rows 0..15 (row = key ^ 16 * rank).
  const int krot = 16 * rank;

  if (tid == 0) {
    for (int s = 0; s < KC; ++s) {
      mbar_init(&bar.kfull[s], 1);  // the loader's arrival with the chunk's transaction bytes
      mbar_init(&bar.kfull_peer[s], 1);
      mbar_init(&bar.kempty[s], 1);
    }
    for (int s = 0; s < NSC; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 2 * NSM);
    }
    mbar_init(&bar.qready, 2 * 4);
    mbar_init(&bar.done_qk, 1);
    mbar_init(&bar.rowx, NSM);
    bar.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(&bar.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tbase = bar.tmem_base;
  volatile int* abort_p = &bar.abort_flag;
  const int TO = kStatusTimeout;

  if (warp == 0) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------------- Q K^T issuer (leader)
      const uint64_t kd = smem_desc_sw128(smem_u32(smem + SM_K), 1024);
      constexpr uint32_t id_qk = idesc_bf16(PM, SCH * KB, false, false);
      const uint32_t t_s = tbase + T_S, t_q = tbase + T_Q;
      bool ok = mbar_wait(&bar.qready, 0, status, TO, abort_p);
      const int nchunks = G / SCH;
      for (int u = 0; u < nchunks && ok; ++u) {
        // chunk u: key blocks g = SCH u .. SCH u + 3 in chunk slot cs (stages 4 cs .. 4 cs + 3)
        const int sb = u % NSC, cs = u % KC, st0 = SCH * cs;
        const uint32_t kpar = (uint32_t)((u / KC) & 1);
        ok = mbar_wait2(&bar.kfull[cs], kpar, &bar.kfull_peer[cs], kpar, status, TO, abort_p);
        if (ok && u >= NSC)
          ok = mbar_wait(&bar.sfree[sb], ((u / NSC) - 1) & 1, status, TO, abort_p);
        if (!ok) break;
        tc_fence_after();
        fence_proxy_async_smem();  // the stages' cp.async writes, before the async-proxy reads
        // Every descriptor is a base descriptor plus a start-address offset (16-byte units, which
        // cannot carry out of the 14-bit field since shared memory is below 256 KiB).
        const uint64_t kst = kd + (uint64_t)((st0 / SCH) * (K_SLOT >> 4));
        const uint32_t ts = t_s + sb * (SCH * KB);
        mma2_ts(ts, t_q, kst, id_qk, 0u);  // K-steps of 16 features: 32 bytes within the rows
        mma2_ts(ts, t_q + 8, kst + 2, id_qk, 1u);
        mma2_ts(ts, t_q + 16, kst + 4, id_qk, 1u);
        mma2_ts(ts, t_q + 24, kst + 6, id_qk, 1u);
        mma2_commit_both(&bar.sfull[sb]);
        mma2_commit_both(&bar.kempty[cs]);
      }
      if (!ok) *abort_p = 1;
      mma2_commit_both(&bar.done_qk);
    } else if (!leader && lane == 0) {
      // Relay (the peer CTA): the leader's Q K^T reads this CTA's half of every block, so each
      // landed chunk is fenced for the async proxy and reported to the leader. A chunk slot is
      // refilled only after the Q K^T that needs this report, so no phase is skipped.
      for (int u = 0; u < G / SCH; ++u) {
        const int cs = u % KC;
        if (!mbar_wait(&bar.kfull[cs], (u / KC) & 1, status, TO, abort_p)) break;
        fence_proxy_async_smem();
        mbar_arrive_cluster_relaxed(&bar.kfull_peer[cs], 0);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ key-tile loader
    // One thread: per chunk one arrival with the chunk's transaction bytes, then the chunk's keys
    // that this CTA contributes (16 of every block) by TMA: one copy of the whole chunk when T is
    // a multiple of 32 (kmap5 views a head's keys as blocks x halves x 16 rows), else one copy per
    // block. Rows past the head's end read as zeros; keys past the pair's causal end are real
    // keys whose logits the softmax masks. The loader shares its scheduler with busy softmax
    // warps and gets few issue slots, so its loop runs once per chunk with few instructions.
    // With the test-only fault LLA_FAULT_WITHHOLD_KEYS the first key block (the first chunk, with
    // chunk copies) is never copied: every wait that needs it runs out after the wait limit, so
    // the timeout path can be tested.
    if (lane == 0) {
      tma_prefetch_map(chunk_copies ? &kmap5 : &kmap);
      int issued = 0;  // chunks whose copies were started
      for (int u = 0; u < G / SCH; ++u) {
        const int cs = u % KC;
        if (u >= KC && !mbar_wait(&bar.kempty[cs], ((u / KC) - 1) & 1, status, TO, abort_p)) break;
        mbar_arrive_expect_tx(&bar.kfull[cs], K_SLOT);
        issued = u + 1;
        const int b0 = (SCH * u) % nb4;  // sweep blocks >= nb: never read
        uint8_t* dst = smem + SM_K + cs * K_SLOT;
        const bool withhold = u == 0 && fault == LLA_FAULT_WITHHOLD_KEYS;
        if (chunk_copies) {  // blocks b0 .. b0 + 3, half `rank`
          if (!withhold) tma_load_5d(dst, &kmap5, 0, 0, rank, b0, (int)bh, &bar.kfull[cs]);
        } else {
#pragma unroll
          for (int t = 0; t < SCH; ++t)
            if (!(withhold && t == 0))
              tma_load_3d(dst + t * K_STAGE, &kmap, 0, (b0 + t) * KB + krot, (int)bh,
                          &bar.kfull[cs]);
        }
      }
      // Nothing may land in this CTA's shared memory after it exits: wait (bounded) for the
      // copies of the last chunks started; a normal run finds them complete.
      volatile int never = 0;
      for (int u = issued > KC ? issued - KC : 0; u < issued; ++u)
        mbar_wait(&bar.kfull[u % KC], (u / KC) & 1, status, TO, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    // Four warps per TMEM lane quarter: part p takes keys 8p .. 8p + 7 of each block (one 16-byte
    // chunk of the block's image row). Row max and omega are combined across the parts through
    // shared memory (barrier rowx: phase 0 after the max sweep, phase 1 at the end).
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const float c2 = inv_h * 1.4426950408889634f;  // log2(e) / h
    if (part == 0) {  // this row of Q into tensor memory (packed bf16 pairs, 32 columns)
      const uint4* qr = reinterpret_cast<const uint4*>(q + (base + (valid ? i : 0)) * D);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
        if (valid) { v0 = qr[2 * c]; v1 = qr[2 * c + 1]; }
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        tmem_st8(lane_base + T_Q + 8 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&bar.qready, leader);
    }
    float m = -INFINITY;
    float2 om2 = make_float2(0.f, 0.f);  // omega as two partial sums (packed fp32 adds)
    bool ok = true;
    // Sweep chunk u covers key blocks b0 .. b0 + SCH - 1. Column n of its S buffer holds key
    // 16 (n / 64) + n % 16 of block (n % 64) / 16 (the pair's B operand: 64 rows from each CTA),
    // so this thread's 8 logits of block b0 + t are columns 64 (part / 2) + 16 t + 8 (part % 2).
    const int col_part = 64 * (part >> 1) + 8 * (part & 1);
    constexpr int kChunk = 2048 / 16;  // chunk stride of an image, in 16-byte units
    for (int u = 0; u < G / SCH && ok; ++u) {
      const int sb = u % NSC;
      if (!warp_wait(&bar.sfull[sb], (u / NSC) & 1, status, TO, abort_p)) { ok = false; break; }
      tc_fence_after();
      const bool max_sweep = SCH * u < nb4;
      const int b0 = (SCH * u) % nb4;
      // the chunk's logits of this thread, all four loads in flight before one wait; the buffer
      // is free as soon as they have completed
      uint32_t sv[SCH][8];
#pragma unroll
      for (int t = 0; t < SCH; ++t)
        tmem_ld8(lane_base + T_S + sb * (SCH * KB) + col_part + t * 16, sv[t]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&bar.sfree[sb], leader);
#pragma unroll
      for (int t = 0; t < SCH; ++t) {
        const int b = b0 + t;
        if (b >= nb) break;  // padding blocks of the chunk
        const int j0 = b * KB + 8 * part;
        // keys j0 .. j0 + 7 all at or before this row: no causal mask (rows past the tile's end
        // have zero queries and finite logits, and nothing of theirs is stored)
        const bool full = j0 + 7 <= i;
        if (max_sweep) {
          if (full) {
#pragma unroll
            for (int c = 0; c < 8; ++c) m = fmaxf(m, __uint_as_float(sv[t][c]));
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              if (valid && j0 + c <= i) m = fmaxf(m, __uint_as_float(sv[t][c]));
          }
          if (b == nb - 1) {  // combine the parts' row maxima
            bar.part_m[part][r] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.rowx);
            if (!warp_wait(&bar.rowx, 0, status, TO, abort_p)) { ok = false; break; }
#pragma unroll
            for (int p2 = 0; p2 < NPART; ++p2) m = fmaxf(m, bar.part_m[p2][r]);
          }
          continue;
        }
        // exponents (s - m) c2 of a key pair in one packed fp32 FMA, the rounded weights' sum in
        // packed fp32 adds (the softmax warps are issue-bound)
        const float2 c22 = make_float2(c2, c2), nmc2 = make_float2(-m * c2, -m * c2);
        uint32_t pw[4];
        if (full) {
#pragma unroll
          for (int c = 0; c < 8; c += 2) {
            const float2 e = __ffma2_rn(
                make_float2(__uint_as_float(sv[t][c]), __uint_as_float(sv[t][c + 1])), c22, nmc2);
            pw[c / 2] = pack_bf16(ex2(e.x), ex2(e.y));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; c += 2) {
            const float2 e = __ffma2_rn(
                make_float2(__uint_as_float(sv[t][c]), __uint_as_float(sv[t][c + 1])), c22, nmc2);
            const float p0 = (valid && j0 + c <= i) ? ex2(e.x) : 0.f;
            const float p1 = (valid && j0 + c + 1 <= i) ? ex2(e.y) : 0.f;
            pw[c / 2] = pack_bf16(p0, p1);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          om2 = __fadd2_rn(om2, make_float2(__uint_as_float(pw[c] << 16),
                                            __uint_as_float(pw[c] & 0xFFFF0000u)));
        // This row's 8 weights as chunk `part` of the block's image.
        ptile_p[(long long)b * (P_BLOCK / 16) + part * kChunk + r] =
            make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
    }
    if (ok) {  // combine the parts' omega
      bar.part_o[part][r] = om2.x + om2.y;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.rowx);
      if (warp_wait(&bar.rowx, 1, status, TO, abort_p) && part == 0 && valid) {
        float s = 0.f;
#pragma unroll
        for (int p2 = 0; p2 < NPART; ++p2) s += bar.part_o[p2][r];
        m_out[base + i] = m * inv_h;
        omega_out[base + i] = s;
      }
    }
  }

  // Teardown: tensor memory is released only after every MMA of the pair has completed (bounded
  // wait, whatever the abort flag says), and neither CTA exits before the other has made its last
  // arrival on it.
  if (warp == 0 && lane == 0) {
    volatile int never = 0;
    mbar_wait(&bar.done_qk, 0, status, TO, &never);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}

}  // namespace

size_t moments_tc_pscratch_bytes(long long BH, int T) {
  return (size_t)BH * (size_t)pscr::blocks_per_head(T) * P_BLOCK;
}

cudaError_t launch_weights_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  // the original keys: [BH][T][64] bf16, boxes of 16 keys x 64 features, 128-byte swizzled
  CUtensorMap kmap;
  const cuuint32_t ones[3] = {1, 1, 1};
  const cuuint64_t kdims[3] = {(cuuint64_t)D, (cuuint64_t)a.T, (cuuint64_t)a.BH()};
  const cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.T * D * 2};
  const cuuint32_t kbox[3] = {(cuuint32_t)D, (cuuint32_t)(KB / 2), 1};
  if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k), kdims, kstr, kbox,
             ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // When T is a multiple of 32: a head's keys as [T / 32 blocks][2 halves][16 rows][64], so that
  // one box {64, 16, 1, 4, 1} is a sweep chunk's 16-key halves of four blocks.
  CUtensorMap kmap5 = kmap;
  const bool chunk_copies = a.T % KB == 0;
  if (chunk_copies) {
    const cuuint32_t ones5[5] = {1, 1, 1, 1, 1};
    const cuuint64_t dims5[5] = {(cuuint64_t)D, (cuuint64_t)(KB / 2), 2, (cuuint64_t)(a.T / KB),
                                 (cuuint64_t)a.BH()};
    const cuuint64_t str5[4] = {(cuuint64_t)D * 2, (cuuint64_t)(KB / 2) * D * 2,
                                (cuuint64_t)KB * D * 2, (cuuint64_t)a.T * D * 2};
    const cuuint32_t box5[5] = {(cuuint32_t)D, (cuuint32_t)(KB / 2), 1, (cuuint32_t)SCH, 1};
    if (encode(&kmap5, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a.k), dims5, str5,
               box5, ones5, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = weights_tc_kernel;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
  if (err != cudaSuccess) return err;
  const long long blocks = 2ll * ((a.T + PM - 1) / PM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, NTHREADS, SMEM_LAUNCH, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), kmap, kmap5, chunk_copies, a.T, (int)a.BH(),
      1.0f / a.h, ws.m, ws.omega, static_cast<uint4*>(ws.pscr), a.fault, ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
