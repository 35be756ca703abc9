// Tensor-core moment contraction of the causal LLA forward (bf16 inputs, d = 64; tcgen05 + TMEM,
// operands fed by TMA).
//
// For every query i and its causal prefix j <= i this kernel accumulates the kernel-weighted
// moments of the closed form of LLA ("Parallax" blog, s.2 Canonical Formulation): omega = sum p_j,
// sum p_j k_j and the upper triangle of sum p_j k_j k_j^T (keys in the head's frame,
// kt = bf16(k - c), written by the prep stage), as one contraction
//     mom[i, f] = sum_j P[i, j] F[j, f]
// of the weights P (bf16, exp((q_i.k_j - m_i)/h), already computed and stored as tcgen05 operand
// images by the weight sweeps of the moments kernel) with the exact key-product features F
// (lla_features.cuh: hi and lo bf16 parts of every k_a k_b, a <= b, plus k_a and 1).
//
// Layout of the work:
//  * A CTA pair (cluster of two, tcgen05 cta_group::2, M = 256) covers 256 consecutive queries of
//    one head: each CTA holds 128 query rows (its tensor-memory lanes) and one half of every
//    feature tile (the B operand is split N/2 + N/2 between the pair's shared memories), so each
//    SM generates half of the features.
//  * The 2208 feature slots are swept in 5 passes of 448 accumulator columns (N = 256 + 192): the
//    weights come from shared memory (A operand), so all of tensor memory holds accumulators.
//    Each pass streams the key prefix again in rounds of 64 keys (two weight images; the image
//    count of a tile is even).
//  * Per round and CTA: the 64 keys (8 KB, TMA with 128-byte swizzling, rows past the sequence
//    zero-filled) land in a ring of 4 key slots, up to two rounds ahead of the rest; the CTA's two
//    weight images (16 KB, TMA, prefetched into L2 four rounds ahead: they come from DRAM) land in
//    one of 2 round slots; 14 generator warps in two groups (one per 32-key half of the round)
//    turn the keys into the CTA's half of the hi/lo feature tiles (2 x 28 KB) of the round slot;
//    one thread issues the round's 16 MMAs (2 halves x 2 K-steps of 16 keys x 2 N chunks x hi, lo)
//    after one combined wait, then one commit. Each MMA costs its issuing thread about half the
//    time the tensor core takes to run it and every barrier test or commit as much as a few MMAs,
//    so one thread keeps the pipe busy only with this much tensor work per synchronisation.
//  * After each pass eight drain warps move the accumulators out of tensor memory: 32 x 32
//    blocks through a 128-byte-swizzled shared buffer (conflict-free row stores), written to the
//    moment rows by TMA tensor stores (rows past the head and columns past 2208 are clipped).
//
// Synchronisation (every wait bounded; all barriers at the same offsets in both CTAs). Every ring
// is used in round order by the same waiters, so each parity wait is on the current or the next
// phase of its barrier, never two ahead:
//  kfull[k]  this CTA's keys of key slot k landed (TMA transaction bytes)
//  kempty[k] both generator groups of this CTA have read them
//  pfull[u]  this CTA's weight images of round slot u landed (TMA transaction bytes)
//  full[u]   (leader) the features of round slot u are written in both CTAs, and the peer's
//            images have landed (reported by the peer's warp 0)
//  empty[u]  the round's MMAs completed (multicast commit): round slot u may be refilled
//  accfull   the accumulators of a pass are final (multicast commit)
//  accfree   (leader) both CTAs have read them out
//  done      every MMA of the pair completed (multicast commit), before tensor memory is freed
// The TMA thread and the drain warps wait for their own last copies before the CTA exits.
//
// Output per query row: mom[row][slot] (fp32, slots in the feature order of lla_features.cuh; the
// row stride is 2208 floats).
#include <cstdint>

#include "lla_features.cuh"
#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"
#include "lla_tmap.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int BM = 128;                    // query rows per CTA = tensor-memory lanes
constexpr int PM = 2 * BM;                 // query rows per CTA pair = MMA M
constexpr int KB = 32;                     // keys per weight image (a half-round)
constexpr int RK = 2 * KB;                 // keys per round
constexpr int NA = 256, NBB = 192;         // the two MMAs of a K-step (N chunks)
constexpr int NCH = NA + NBB;              // accumulator columns (features) per pass
constexpr int NFS = feat::kFeatureSlots;   // 2208: row stride of the moment rows
constexpr int NPASS = (NFS + NCH - 1) / NCH;  // 5
constexpr int GA = NA / 16, GB = NBB / 16;    // 8-feature groups each CTA holds per chunk
constexpr int GLOC = GA + GB;                 // 28 per CTA per pass
constexpr int NRS = 2;                     // round slots (weights + features)
constexpr int NKS = 4;                     // key slots (rounds)
constexpr int PFR = 4;                     // weight images prefetched into L2 this many rounds ahead
constexpr int NGW = 7;                     // generator warps per group (4 feature groups each)
constexpr int NDR = 8;                     // drain warps (two per tensor-memory lane quarter)
constexpr int W_MMA = 0, W_TMA = 1, W_GEN0 = 2, W_DR0 = W_GEN0 + 2 * NGW;
constexpr int NWARPS = W_DR0 + NDR;        // 24
constexpr int NTHREADS = NWARPS * 32;
static_assert(GLOC == 4 * NGW, "four feature groups per generator warp");
static_assert(W_DR0 % 4 == 0, "drain warp w reads tensor-memory lane quarter w % 4");
static_assert(BM == pscr::kRows && KB == pscr::kKeys, "weight image layout");

// shared memory (offsets from a 1024-byte aligned base; the same in both CTAs of a pair)
constexpr int K_BYTES = RK * D * 2;        // 8192: 64 keys x 128 B, 128-byte swizzled
constexpr int P_BYTES = BM * KB * 2;       // 8192: one weight image
constexpr int F_HALF = GLOC * 512;         // 14336: hi (or lo) features of the CTA's groups
constexpr int F_STEP = 2 * F_HALF;         // hi and lo of one half-round
constexpr int SLOT = 2 * P_BYTES + 2 * F_STEP;  // a round slot: two images, then two feature sets
constexpr int SM_K = 0;
constexpr int SM_R = SM_K + NKS * K_BYTES;
constexpr int STG_BYTES = 32 * 32 * 4;     // drain staging: 32 rows x 32 fp32, 128-byte swizzled
constexpr int SM_STG = SM_R + NRS * SLOT;
constexpr int SM_BAR = SM_STG + NDR * STG_BYTES;
constexpr int SMEM_USED = SM_BAR + 1024;
constexpr int SMEM_LAUNCH = SMEM_USED + 1024;  // slack for aligning the base
static_assert(K_BYTES % 1024 == 0 && SLOT % 1024 == 0 && SM_STG % 1024 == 0 &&
              STG_BYTES % 1024 == 0, "1024-byte alignment of the swizzled regions and slots");
static_assert(SMEM_LAUNCH <= 227 * 1024, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
static_assert(NCH <= (int)TMEM_COLS, "accumulators fit tensor memory");

struct Bars {
  uint64_t kfull[NKS];
  uint64_t kempty[NKS];
  uint64_t pfull[NRS];
  uint64_t full[NRS];
  uint64_t empty[NRS];
  uint64_t accfull, accfree, done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 1024, "barrier region");

// Global 8-feature group of a pass held by CTA `rank` as local group lg: chunk A (N = 256) has
// global groups 0..31 (CTA 0 holds 0..15, CTA 1 16..31), chunk B (N = 192) groups 32..55
// (CTA 0 holds 32..43, CTA 1 44..55).
__host__ __device__ constexpr int global_group(int rank, int lg) {
  return lg < GA ? rank * GA + lg : 2 * GA + rank * GB + (lg - GA);
}

template <int PASS, int RANK, int LG0, int LG1>
__device__ __forceinline__ void gen_groups(const uint32_t (&kw)[33], uint8_t* fhi, uint8_t* flo,
                                           int row_off) {
  if constexpr (LG0 < LG1) {
    constexpr int slot0 = PASS * NCH + global_group(RANK, LG0) * 8;
    feat::feature_group<slot0 / 2>(kw, fhi + LG0 * 512 + row_off, flo + LG0 * 512 + row_off);
    gen_groups<PASS, RANK, LG0 + 1, LG1>(kw, fhi, flo, row_off);
  }
}

template <int PASS, int RANK>
__device__ __forceinline__ void gen_pr(int fw, const uint32_t (&kw)[33], uint8_t* fhi,
                                       uint8_t* flo, int row_off) {
  switch (fw) {
    case 0: gen_groups<PASS, RANK, 0, 4>(kw, fhi, flo, row_off); break;
    case 1: gen_groups<PASS, RANK, 4, 8>(kw, fhi, flo, row_off); break;
    case 2: gen_groups<PASS, RANK, 8, 12>(kw, fhi, flo, row_off); break;
    case 3: gen_groups<PASS, RANK, 12, 16>(kw, fhi, flo, row_off); break;
    case 4: gen_groups<PASS, RANK, 16, 20>(kw, fhi, flo, row_off); break;
    case 5: gen_groups<PASS, RANK, 20, 24>(kw, fhi, flo, row_off); break;
    default: gen_groups<PASS, RANK, 24, 28>(kw, fhi, flo, row_off); break;
  }
}

template <int PASS>
__device__ __forceinline__ void gen_pass(int rank, int fw, const uint32_t (&kw)[33], uint8_t* fhi,
                                         uint8_t* flo, int row_off) {
  if (rank == 0) gen_pr<PASS, 0>(fw, kw, fhi, flo, row_off);
  else gen_pr<PASS, 1>(fw, kw, fhi, flo, row_off);
}

__device__ __forceinline__ void generate(int pass, int rank, int fw, const uint32_t (&kw)[33],
                                         uint8_t* fhi, uint8_t* flo, int row_off) {
  switch (pass) {
    case 0: gen_pass<0>(rank, fw, kw, fhi, flo, row_off); break;
    case 1: gen_pass<1>(rank, fw, kw, fhi, flo, row_off); break;
    case 2: gen_pass<2>(rank, fw, kw, fhi, flo, row_off); break;
    case 3: gen_pass<3>(rank, fw, kw, fhi, flo, row_off); break;
    default: gen_pass<4>(rank, fw, kw, fhi, flo, row_off); break;
  }
}
static_assert(NPASS == 5, "generate() dispatches five passes");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
moments_pass_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap pmap,
                       const __grid_constant__ CUtensorMap mmap, int T, int BH,
                       int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars& bar = *reinterpret_cast<Bars*>(smem + SM_BAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;
  const int npairs = (T + PM - 1) / PM;
  const int pair_lin = (int)(blockIdx.x >> 1);
  const int ptile = npairs - 1 - pair_lin / BH;  // longest causal prefixes first
  const int bh = pair_lin % BH;
  const int i0 = ptile * PM + rank * BM;         // this CTA's first query row
  const int nb = pscr::pair_blocks(T, ptile);    // key blocks of 32 (even)
  const int nr = nb / 2;                         // rounds per pass
  const int R = NPASS * nr;                      // rounds: pass r / nr, key blocks 2 (r % nr) + 0, 1
  const int pblk0 = (int)pscr::first_block(bh, T, ptile, rank);

  if (tid == 0) {
    for (int k = 0; k < NKS; ++k) {
      mbar_init(&bar.kfull[k], 1);
      mbar_init(&bar.kempty[k], 2 * NGW);  // both generator groups of this CTA
    }
    for (int u = 0; u < NRS; ++u) {
      mbar_init(&bar.pfull[u], 1);
      mbar_init(&bar.full[u], 4 * NGW + 1);  // both groups of both CTAs, the peer's report
      mbar_init(&bar.empty[u], 1);
    }
    mbar_init(&bar.accfull, 1);
    mbar_init(&bar.accfree, 2 * NDR);
    mbar_init(&bar.done, 1);
    bar.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    tmem_alloc_pair(&bar.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == W_TMA && lane == 0) {
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&pmap);
    tma_prefetch_map(&mmap);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tbase = bar.tmem_base;
  volatile int* abort_p = &bar.abort_flag;
  const int TO = kStatusTimeout;

  if (warp == W_MMA) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer (leader)
      const uint64_t pdesc = smem_desc(smem_u32(smem + SM_R), 2048, 128);  // A: K-major images
      const uint64_t fdesc = smem_desc(smem_u32(smem + SM_R + 2 * P_BYTES), 128, 512);  // B
      constexpr uint32_t id_a = idesc_bf16(PM, NA, false, true);
      constexpr uint32_t id_b = idesc_bf16(PM, NBB, false, true);
      constexpr uint64_t kB = (uint64_t)(GA * 512 >> 4);   // chunk B's local groups
      constexpr uint64_t kLo = (uint64_t)(F_HALF >> 4);     // lo tile after the hi tile
      bool ok = true;
      int rb = 0, pass = 0;  // round within the pass
      for (int r = 0; r < R && ok; ++r) {
        const int u = r % NRS;
        const uint32_t par = (uint32_t)((r / NRS) & 1);
        ok = mbar_wait2(&bar.full[u], par, &bar.pfull[u], par, status, TO, abort_p);
        if (ok && rb == 0 && pass > 0) ok = mbar_wait(&bar.accfree, (pass - 1) & 1, status, TO, abort_p);
        if (!ok) break;
        tc_fence_after();
        // Descriptors: a base descriptor plus a start-address offset in 16-byte units (shared
        // memory is below 256 KiB, so the 14-bit field never carries).
        const uint64_t so = (uint64_t)(u * (SLOT >> 4));
#pragma unroll
        for (int j = 0; j < 2; ++j) {      // half-rounds: keys 32 j .. 32 j + 31
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {  // K-steps of 16 keys
            const uint64_t a = pdesc + so + (uint64_t)((j * P_BYTES + ks * 4096) >> 4);
            const uint64_t fh = fdesc + so + (uint64_t)((j * F_STEP + ks * 256) >> 4);
            const uint32_t acc = (rb > 0 || j > 0 || ks > 0) ? 1u : 0u;
            mma2_ss(tbase, a, fh, id_a, acc);
            mma2_ss(tbase, a, fh + kLo, id_a, 1u);
            mma2_ss(tbase + NA, a, fh + kB, id_b, acc);
            mma2_ss(tbase + NA, a, fh + kB + kLo, id_b, 1u);
          }
        }
        mma2_commit_both(&bar.empty[u]);
        if (rb == nr - 1) mma2_commit_both(&bar.accfull);
        if (++rb == nr) { rb = 0; ++pass; }
      }
      if (!ok) *abort_p = 1;
      mma2_commit_both(&bar.done);
    } else if (!leader && lane == 0) {
      // ---------------------------------------------------------------- relay (peer)
      // The leader's MMAs read this CTA's weight images of every round: each landed pair is
      // reported on the leader's full barrier of its slot. A slot is refilled only after the
      // MMAs that need this report, so no phase is skipped.
      for (int r = 0; r < R; ++r) {
        const int u = r % NRS;
        if (!mbar_wait(&bar.pfull[u], (r / NRS) & 1, status, TO, abort_p)) break;
        mbar_arrive_cluster_relaxed(&bar.full[u], 0);
      }
    }
    __syncwarp();
  } else if (warp == W_TMA) {
    // ------------------------------------------------------------------ TMA producer
    // Keys run up to NKS - NRS rounds ahead of the weight images (the generators need them first);
    // the images of round r + PFR are prefetched into L2 when round r's are loaded.
    if (lane == 0) {
      constexpr int KA = NKS - NRS;
      int kiss = 0, piss = 0;  // rounds whose keys / images have been issued
      for (int r = 0; r < PFR && r < R; ++r) tma_prefetch_3d(&pmap, 0, 0, pblk0 + 2 * (r % nr));
      for (int t = 0; t < R + KA; ++t) {
        if (t < R) {  // keys of round t
          const int k = t % NKS;
          if (t >= NKS && !mbar_wait(&bar.kempty[k], ((t / NKS) - 1) & 1, status, TO, abort_p)) break;
          mbar_arrive_expect_tx(&bar.kfull[k], K_BYTES);
          tma_load_3d(smem + SM_K + k * K_BYTES, &kmap, 0, RK * (t % nr), bh, &bar.kfull[k]);
          kiss = t + 1;
        }
        const int r = t - KA;  // images of round r
        if (r >= 0) {
          const int u = r % NRS;
          if (r >= NRS && !mbar_wait(&bar.empty[u], ((r / NRS) - 1) & 1, status, TO, abort_p)) break;
          if (r + PFR < R) tma_prefetch_3d(&pmap, 0, 0, pblk0 + 2 * ((r + PFR) % nr));
          mbar_arrive_expect_tx(&bar.pfull[u], 2 * P_BYTES);
          tma_load_3d(smem + SM_R + u * SLOT, &pmap, 0, 0, pblk0 + 2 * (r % nr), &bar.pfull[u]);
          piss = r + 1;
        }
      }
      // Nothing may land in this CTA's shared memory after it exits: wait for the copies of the
      // last slots filled (a normal run finds them complete).
      volatile int never = 0;
      for (int t = kiss - NKS > 0 ? kiss - NKS : 0; t < kiss; ++t)
        mbar_wait(&bar.kfull[t % NKS], (t / NKS) & 1, status, TO, &never);
      for (int r = piss - NRS > 0 ? piss - NRS : 0; r < piss; ++r)
        mbar_wait(&bar.pfull[r % NRS], (r / NRS) & 1, status, TO, &never);
    }
    __syncwarp();
  } else if (warp < W_DR0) {
    // ------------------------------------------------------------------ feature generators
    // Group g generates the features of keys 32 g .. 32 g + 31 of every round (lane = key); warp
    // fw of the group generates local feature groups 4 fw .. 4 fw + 3.
    const int gw = warp - W_GEN0, g = gw / NGW, fw = gw % NGW;
    const int row_off = (lane >> 3) * 128 + (lane & 7) * 16;  // key `lane` in a feature tile
    const int key = g * KB + lane;                             // row of the round's key box
    const int swz = key & 7;                                   // its 128-byte swizzle
    for (int r = 0; r < R; ++r) {
      const int k = r % NKS, u = r % NRS;
      if (!warp_wait(&bar.kfull[k], (r / NKS) & 1, status, TO, abort_p)) break;
      const uint8_t* kst = smem + SM_K + k * K_BYTES + key * 128;
      uint32_t kw[33];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(kst + ((c ^ swz) << 4));
        kw[4 * c] = v.x; kw[4 * c + 1] = v.y; kw[4 * c + 2] = v.z; kw[4 * c + 3] = v.w;
      }
      kw[32] = 0x00003F80u;  // bf16 one (constant feature) and zero (padding)
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.kempty[k]);
      // the round slot's previous features (round r - NRS) have been consumed
      if (r >= NRS && !warp_wait(&bar.empty[u], ((r / NRS) - 1) & 1, status, TO, abort_p)) break;
      uint8_t* fhi = smem + SM_R + u * SLOT + 2 * P_BYTES + g * F_STEP;
      generate(r / nr, rank, fw, kw, fhi, fhi + F_HALF, row_off);
      fence_proxy_async_smem();  // the generic-proxy stores, before the MMA's async-proxy reads
      __syncwarp();
      if (lane == 0) arrive_leader(&bar.full[u], leader);
    }
  } else {
    // ------------------------------------------------------------------ drain
    // Warp (quarter, half) reads 32 rows x 224 columns per pass in blocks of 32 columns; each
    // block goes through this warp's staging buffer (row `lane` at lane * 128, its 16-byte chunk c
    // at chunk c ^ (lane & 7): the 128-byte swizzle of the tensor map) to one TMA store.
    const int dw = warp - W_DR0, quarter = warp & 3, half = dw >> 2;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    uint8_t* stg = smem + SM_STG + dw * STG_BYTES;
    uint8_t* my_row = stg + lane * 128;
    const int swz = lane & 7;
    constexpr int C0 = NCH / 2;  // columns per half
    for (int pass = 0; pass < NPASS; ++pass) {
      if (!warp_wait(&bar.accfull, pass & 1, status, TO, abort_p)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = half * C0; c < half * C0 + C0; c += 32) {
        uint32_t v0[16], v1[16];
        tmem_ld16(lane_base + c, v0);
        tmem_ld16(lane_base + c + 16, v1);
        if (lane == 0) bulk_wait_read0();  // the previous block's store has read the buffer
        tmem_ld_wait();
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(my_row + ((q ^ swz) << 4)) =
              make_uint4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]);
          *reinterpret_cast<uint4*>(my_row + (((q + 4) ^ swz) << 4)) =
              make_uint4(v1[4 * q], v1[4 * q + 1], v1[4 * q + 2], v1[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&mmap, pass * NCH + c, i0 + quarter * 32, bh, stg);
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&bar.accfree, leader);
    }
    if (lane == 0) bulk_wait0();  // every store of this warp complete
    __syncwarp();
  }

  // Teardown: tensor memory is released only after every MMA of the pair has completed (bounded
  // wait, whatever the abort flag says), and neither CTA exits before the other has made its last
  // arrival on it.
  if (warp == W_MMA && lane == 0) {
    volatile int never = 0;
    mbar_wait(&bar.done, 0, status, TO, &never);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}
static_assert(NCH % 64 == 0, "drain blocks of 32 columns per half");

}  // namespace

cudaError_t launch_moments_pass_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint32_t ones[3] = {1, 1, 1};
  // keys in the head's frame (the prep stage's bf16(k - c)): [BH][T][64] bf16, boxes of 32 keys
  // x 64 features, 128-byte swizzled
  CUtensorMap kmap, pmap;
  const cuuint64_t kdims[3] = {(cuuint64_t)D, (cuuint64_t)a.T, (cuuint64_t)a.BH()};
  const cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.T * D * 2};
  const cuuint32_t kbox[3] = {(cuuint32_t)D, (cuuint32_t)RK, 1};
  if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws.ksh, kdims, kstr, kbox,
             ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // weight images: [blocks][64 rows][128 B], one 8 KB box per image, copied as laid out
  const long long nblocks = a.BH() * pscr::blocks_per_head(a.T);
  if (nblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const cuuint64_t pdims[3] = {64, 64, (cuuint64_t)nblocks};
  const cuuint64_t pstr[2] = {128, (cuuint64_t)P_BYTES};
  const cuuint32_t pbox[3] = {64, 64, 2};  // a round's two images
  if (encode(&pmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws.pscr, pdims, pstr, pbox, ones,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // moment rows: [BH][T][2208] fp32, stored in 32 x 32 boxes, 128-byte swizzled in shared memory
  CUtensorMap mmap;
  const cuuint64_t mdims[3] = {(cuuint64_t)NFS, (cuuint64_t)a.T, (cuuint64_t)a.BH()};
  const cuuint64_t mstr[2] = {(cuuint64_t)NFS * 4, (cuuint64_t)a.T * NFS * 4};
  const cuuint32_t mbox[3] = {32, 32, 1};
  if (encode(&mmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws.mom, mdims, mstr, mbox, ones,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto kern = moments_pass_tc_kernel;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
  if (err != cudaSuccess) return err;
  const long long blocks = 2ll * ((a.T + PM - 1) / PM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, NTHREADS, SMEM_LAUNCH, s>>>(kmap, pmap, mmap, a.T, (int)a.BH(),
                                                       ws.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
