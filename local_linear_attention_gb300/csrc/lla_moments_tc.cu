// Tensor-core moments stage of the causal LLA forward (bf16 inputs, d = 64; tcgen05 + TMEM).
//
// Computes, for every query i and its causal prefix j <= i, the kernel-weighted moments that the
// closed form of LLA needs ("Parallax" blog, s.2 Canonical Formulation): omega = sum p_j,
// sk = sum p_j k_j and the upper triangle of S = sum p_j k_j k_j^T, with
// p_j = exp((q_i.k_j - m_i)/h) and m_i the exact row max of q_i.k_j over the prefix.
//
// As a GEMM: [queries x keys] (P) times [keys x 2144 features] (F, the products k_a * 1 and
// k_a * k_b, a <= b) into fp32 accumulators in tensor memory. Three facts shape it:
//  * The products must be exact: rounding k_a k_b to bf16 breaks the Gram structure of S and
//    makes the ridge system indefinite, whereas rounding the weights p to bf16 only perturbs the
//    weights (all moments still describe one weighted problem). Each product of two bf16 values
//    (16 significant bits) is split exactly into hi = bf16(k_a k_b) and lo = k_a k_b - hi, both
//    exact bf16, with one packed multiply and one packed fused multiply-add; every feature column
//    is then contracted twice (hi and lo) into the same accumulator.
//  * 2144 fp32 accumulator columns do not fit the 512 columns of tensor memory, so the features
//    are swept in 6 passes of 368 columns; each pass streams the key prefix again. A first sweep
//    computes the exact row max m_i (Q K^T and a max); a second sweep computes P (bf16) and
//    stores it to a scratch, from which every feature pass takes it again. Q K^T and the
//    exponentials thus never wait behind a feature contraction in the tensor pipe. The sweeps
//    run Q K^T on chunks of four key blocks (N = 128): a tcgen05.mma costs about as long at
//    N = 32 as at N = 128.
//  * Feature tiles are generated per key block into shared memory and read back by the MMA, a
//    per-block cost on every SM. Two CTAs on two SMs (a cluster pair) therefore
//    share every MMA (tcgen05 cta_group::2, M = 256): each CTA holds 128 query rows (its tensor
//    memory lanes) and generates and holds half of every feature tile (the B operand is split
//    N/2 + N/2 between the pair's shared memories), halving the feature work per SM.
//
// A pair covers 256 consecutive queries of one head; both CTAs stream the same key blocks (up to
// the pair's last query; the causal mask zeroes the keys past a row). The even CTA (the leader)
// issues all MMAs; its barriers that gate an MMA collect arrivals from both CTAs (mapa + remote
// arrive), and MMA completion is signalled to both CTAs (multicast commit).
//
// Warp roles per CTA (24 warps): 0 issues Q K^T (leader; one thread) and owns the TMEM
// allocation; 22 and 23 issue the feature contraction (leader; one thread each, alternate key
// blocks); in the peer CTA warp 0 relays its landed sweep blocks to the leader; 1 stages key
// blocks (32 keys x 64) into shared memory (cp.async, completion counted on each stage's barrier,
// every stage in flight); 2-9 turn S into P (one thread per query = TMEM lane, two warps
// per lane quarter splitting the keys of a block), put P into tensor memory for each feature step
// and drain the accumulators after each pass; 10-21 generate this CTA's half of the exact hi/lo
// feature tiles (one lane per key; two groups of six warps take alternate key blocks). P has
// seven buffers in tensor memory (the A operand of the feature contraction), the feature tiles
// five in shared memory.
// All operands in shared memory use the no-swizzle core-matrix layout. Every mbarrier wait is
// bounded.
//
// Feature order (2208 slots = 1104 pairs, the layout of each output row): the upper triangle of
// kt kt^T for the augmented key kt = [k_0..k_63, 1, 0], row by row: for row a, the pairs
// (a, b), (a, b+1) for even b from a (even a) or a+1 (odd a) up to 64 -- so one operand of each
// packed product is a key word exactly as loaded -- then the 16 pairs of odd diagonal entries
// (4u+1, 4u+1), (4u+3, 4u+3). Slot (a, 64) holds sum p k_a, slots (a, 65) are zero padding.
// Output per query row (fp32): mom_tc[row][slot], omega[row], m[row] = m_i / h; and the bf16
// weight images in the weight scratch.
#include <cstdint>
#include <type_traits>

#include "lla_internal.cuh"
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

using namespace tc;

constexpr int D = 64;
constexpr int BM = 128;                     // query rows per CTA = TMEM lanes
constexpr int PM = 2 * BM;                  // query rows per CTA pair = MMA M
constexpr int KB = 32;                      // keys per block
constexpr int NCH = 368;                    // features (accumulator columns) per pass
constexpr int NPASS = 6;
constexpr int NFP = NPASS * NCH;            // 2208, padded feature count (row stride of mom_tc)
constexpr int NA = 192, NB_ = NCH - NA;     // split of a pass into two MMAs (N <= 256)
constexpr int GA = NA / 16, GB = NB_ / 16;  // 8-feature groups each CTA holds for either MMA
constexpr int GLOC = GA + GB;               // 23 groups per CTA per pass
constexpr int SCH = 4;                      // key blocks per sweep chunk (one Q K^T of N = 128)
constexpr int KS = 12;                      // key-tile pipeline stages (three sweep chunks)
constexpr int NSM = 8;                      // softmax warps: two per TMEM lane quarter
constexpr int NFG = 12;                     // feature-generation warps: two groups of NFGW that
constexpr int NFGW = NFG / 2;               //   take alternate key blocks
constexpr int NWARPS = 4 + NSM + NFG;       // + Q K^T issuer, key loader, two feature issuers
constexpr int NTHREADS = NWARPS * 32;
constexpr int NBUF = 7;                     // P buffers (tensor memory, feature passes only)
constexpr int NFB = 5;                      // F buffers (shared memory)
constexpr int NSC = 3;                      // S buffers of the sweeps (SCH blocks each)
static_assert(BM == pscr::kRows && KB == pscr::kKeys && PM == 2 * BM, "weight scratch layout");

// tensor-memory columns (the same in both CTAs of a pair)
constexpr uint32_t T_ACC = 0;
// The two sweeps and the feature passes use tensor memory at different times: the logits S of the
// sweeps take the accumulator and weight columns (idle until the first feature pass, which starts
// only after the softmax warps have read the last S), so that Q K^T can run NSC chunks ahead of
// the softmax warps; the weights P of the feature passes take NBUF buffers after the
// accumulators, so that a step's weights can be in place several steps ahead of its MMAs.
constexpr uint32_t T_S = T_ACC;             // NSC x 128 columns of fp32 logits (sweeps)
constexpr uint32_t T_P = NCH;               // NBUF x 16 columns of packed bf16 weights (passes)
constexpr uint32_t T_Q = T_P + NBUF * (KB / 2);  // 32 columns: the Q tile, A operand of Q K^T
constexpr uint32_t TMEM_COLS = 512;
static_assert(T_S + NSC * SCH * KB <= T_Q, "sweep S buffers below the Q tile");
static_assert(T_Q + D / 2 <= TMEM_COLS, "tensor memory budget");

// shared-memory layout (bytes; the same offsets in both CTAs of a pair)
constexpr int SM_K = 0;                              // KS x (32 x 64 bf16)
constexpr int K_STAGE = KB * D * 2;
constexpr int SM_F = SM_K + KS * K_STAGE;            // [NFB][hi, lo][23 groups x 512 B]
constexpr int F_HALF = GLOC * 512;
constexpr int F_BUF = 2 * F_HALF;
// One key block of P (128 rows x 32 keys, bf16) in the global P scratch: 16-byte chunk kc (keys
// 8kc..8kc+7) of row r at kc * 2048 + r * 16, so that each warp's stores of one chunk are 512
// contiguous bytes.
constexpr int P_BLOCK = BM * KB * 2;
constexpr int EPI_LD = 36;                           // row stride (floats) of the drain buffer
constexpr int SM_EPI = SM_F + NFB * F_BUF;           // NSM x (32 rows x 36 floats)
// Feature passes take each thread's weights back from the global scratch PD key blocks ahead of
// use (a per-thread ring in shared memory filled with cp.async): the scratch does
// not fit L2, and one block of look-ahead (~740 cycles of tensor work) is shorter than a DRAM miss.
constexpr int PD = 3;
constexpr int SM_PR = SM_EPI + NSM * 32 * EPI_LD * 4;  // NSM x PD x 32 lanes x 32 bytes
constexpr int SM_BAR = SM_PR + NSM * PD * 32 * 32;
constexpr int SMEM_BYTES = SM_BAR + 2048;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
// More than half of an SM's shared memory, so that at most one CTA (and one TMEM allocation of
// all 512 columns) is resident per SM.
constexpr int SMEM_LAUNCH = SMEM_BYTES > 120 * 1024 ? SMEM_BYTES : 120 * 1024;

// Pair p of the feature order (see the file comment): row a and even column b, or, for the odd
// diagonal pairs, u = a.
struct PairSpec { int a, b; bool diag; };
constexpr int kRowPairs = 1088;
__host__ __device__ constexpr PairSpec pair_spec(int p) {
  if (p >= kRowPairs) return PairSpec{p - kRowPairs, 0, true};
  int a = 0;
  while (true) {
    const int cnt = (a % 2 == 0) ? 33 - a / 2 : 32 - (a - 1) / 2;
    if (p < cnt) return PairSpec{a, (a % 2 == 0 ? a : a + 1) + 2 * p, false};
    p -= cnt;
    ++a;
  }
}
static_assert(2 * (kRowPairs + 16) == NFP, "feature order fills the padded row");

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t x, uint32_t y, uint32_t z) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  return r;
}
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

// One group of 8 feature slots (pairs P0..P0+3) for this lane's key: 4 hi words and 4 lo words,
// stored as one 16-byte row of the group's core matrix. kw[t] = k[2t] | k[2t+1] << 16 for t < 32,
// kw[32] = bf16(1) | 0 << 16 (the constant feature and the zero pad).
template <int P0>
__device__ __forceinline__ void feature_group(const uint32_t (&kw)[33], uint8_t* hi_row,
                                              uint8_t* lo_row) {
  uint32_t h[4], l[4];
  auto one = [&](auto tpair) {
    constexpr int T = decltype(tpair)::value;
    constexpr PairSpec ps = pair_spec(P0 + T);
    uint32_t x, y;
    if constexpr (ps.diag) {  // (k[4u+1], k[4u+3]) squared
      x = __byte_perm(kw[2 * ps.a], kw[2 * ps.a + 1], 0x7632);
      y = x;
    } else {                  // (k[a], k[a]) times (k[b], k[b+1])
      x = __byte_perm(kw[ps.a >> 1], 0u, (ps.a & 1) ? 0x3232 : 0x1010);
      y = kw[ps.b >> 1];
    }
    const uint32_t hv = bf16x2_mul(x, y);
    h[T] = hv;
    l[T] = bf16x2_fma(x, y, hv ^ 0x80008000u);
  };
  one(std::integral_constant<int, 0>{});
  one(std::integral_constant<int, 1>{});
  one(std::integral_constant<int, 2>{});
  one(std::integral_constant<int, 3>{});
  *reinterpret_cast<uint4*>(hi_row) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_row) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Global 8-feature group of a pass held by CTA `RANK` as its local group LG: the first GA local
// groups belong to the N = 192 MMA (CTA 0 holds its groups 0..11, CTA 1 its groups 12..23), the
// other GB to the N = 176 MMA (groups 24..34 and 35..45).
__host__ __device__ constexpr int global_group(int rank, int lg) {
  return lg < GA ? rank * GA + lg : 2 * GA + rank * GB + (lg - GA);
}

// Local groups [LG0, LG1) of pass PASS for one key (lane), written into the F buffer halves at
// row offset `row_off` (= (key / 8) * 128 + (key % 8) * 16).
template <int PASS, int RANK, int LG0, int LG1>
__device__ __forceinline__ void feature_groups(const uint32_t (&kw)[33], uint8_t* fhi, uint8_t* flo,
                                               int row_off) {
  if constexpr (LG0 < LG1) {
    feature_group<(PASS * NCH + global_group(RANK, LG0) * 8) / 2>(kw, fhi + LG0 * 512 + row_off,
                                                                  flo + LG0 * 512 + row_off);
    feature_groups<PASS, RANK, LG0 + 1, LG1>(kw, fhi, flo, row_off);
  }
}

// Split of the 23 local groups among the NFGW warps of a feature group: 5 x 4, then 3.
__host__ __device__ constexpr int fw_begin(int fw) { return 4 * fw < GLOC ? 4 * fw : GLOC; }
static_assert(NFGW == 6 && fw_begin(NFGW) == GLOC && fw_begin(NFGW - 1) < GLOC, "groups split");

template <int PASS, int RANK>
__device__ __forceinline__ void generate_pr(int fw, const uint32_t (&kw)[33], uint8_t* fhi,
                                            uint8_t* flo, int row_off) {
  switch (fw) {
    case 0: feature_groups<PASS, RANK, fw_begin(0), fw_begin(1)>(kw, fhi, flo, row_off); break;
    case 1: feature_groups<PASS, RANK, fw_begin(1), fw_begin(2)>(kw, fhi, flo, row_off); break;
    case 2: feature_groups<PASS, RANK, fw_begin(2), fw_begin(3)>(kw, fhi, flo, row_off); break;
    case 3: feature_groups<PASS, RANK, fw_begin(3), fw_begin(4)>(kw, fhi, flo, row_off); break;
    case 4: feature_groups<PASS, RANK, fw_begin(4), fw_begin(5)>(kw, fhi, flo, row_off); break;
    default: feature_groups<PASS, RANK, fw_begin(5), GLOC>(kw, fhi, flo, row_off); break;
  }
}

template <int PASS>
__device__ __forceinline__ void generate_pass(int rank, int fw, const uint32_t (&kw)[33],
                                              uint8_t* fhi, uint8_t* flo, int row_off) {
  if (rank == 0) generate_pr<PASS, 0>(fw, kw, fhi, flo, row_off);
  else generate_pr<PASS, 1>(fw, kw, fhi, flo, row_off);
}

__device__ __forceinline__ void generate(int pass, int rank, int fw, const uint32_t (&kw)[33],
                                         uint8_t* fhi, uint8_t* flo, int row_off) {
  switch (pass) {
    case 0: generate_pass<0>(rank, fw, kw, fhi, flo, row_off); break;
    case 1: generate_pass<1>(rank, fw, kw, fhi, flo, row_off); break;
    case 2: generate_pass<2>(rank, fw, kw, fhi, flo, row_off); break;
    case 3: generate_pass<3>(rank, fw, kw, fhi, flo, row_off); break;
    case 4: generate_pass<4>(rank, fw, kw, fhi, flo, row_off); break;
    default: generate_pass<5>(rank, fw, kw, fhi, flo, row_off); break;
  }
}

// Byte offset, from the first key stage, of 16-byte chunk c (elements 8c..8c+7) of row r of key
// stage st. Each stage is a K-major tile of 32 rows x 64 elements in 8-row groups of eight
// 128-byte core matrices (chunks 128 bytes apart). The stages form chunks of SCH = 4 consecutive
// stages (16 KiB), and within a chunk the row groups are ordered (rows 0..15 of stages 0..3, then
// rows 16..31 of stages 0..3): the 16 rows that a CTA contributes to Q K^T from each of the 4
// stages are then 8 row groups 1024 bytes apart, one N = 128 operand for the pair.
__device__ __forceinline__ int kst_off(int st, int r, int c) {
  return (st >> 2) * (SCH * K_STAGE) + (r >> 4) * (SCH * K_STAGE / 2) +
         (2 * (st & 3) + ((r >> 3) & 1)) * 1024 + c * 128 + (r & 7) * 16;
}
static_assert(KS % SCH == 0 && SCH == 4 && K_STAGE == 4096, "key stage layout");

// Wait executed by all 32 lanes of a warp; the outcome is made warp-uniform so that an abort seen
// by one lane takes the whole warp out of its loop together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, kStatusTimeout, abort));
}

// Barriers marked (L) are used in the leader CTA only and collect arrivals from both CTAs; those
// marked (M) are arrived on by multicast commits from the leader's MMA issuers in both CTAs.
struct Barriers {
  uint64_t kfull[KS];           // key block staged by this CTA's loader
  uint64_t kfull_peer[KS];      // (L) key block staged by the peer's loader (for Q K^T only)
  uint64_t kempty[KS];          // key stage consumed: (M) Q K^T commit or 1 extra arrival, + NFGW
  uint64_t sfull[NSC];          // (M) S = Q K^T of a sweep chunk in tensor memory
  uint64_t sfree[NSC];          // (L) S read by both CTAs' softmax warps
  uint64_t pfull[NBUF];         // (L) P written to tensor memory in both CTAs
  uint64_t ffull[NFB];          // (L) F halves written in both CTAs
  uint64_t pfree[NBUF];         // (M) the feature MMAs of a step completed (P buffer free)
  uint64_t ffree[NFB];          // (M) the same, for the F buffer
  uint64_t accfull;             // (M) the accumulators of a pass are final
  uint64_t accfree;             // (L) both CTAs drained them
  uint64_t qready;              // (L) both CTAs' Q tiles in tensor memory
  uint64_t hand[2];             // (L) feature issuer t has issued its latest step
  uint64_t done_qk, done_f[2];  // (M) every MMA of the Q K^T issuer / feature issuer t completed
  uint64_t rowx;                // this CTA's softmax halves exchanged row max / omega
  float part[2][BM];            // per-row partial results of the two softmax halves
};

static_assert(sizeof(Barriers) <= 2048, "barrier region");

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(n)
      : "memory");
}

// Arrival of one of this CTA's producers on a leader barrier (L). Every producer has completed
// what the leader consumes before it arrives (see mbar_arrive_cluster_relaxed), so the peer's
// arrival needs no cluster-wide release, and the leader's issuers test these barriers with the
// ordinary (CTA-scope) wait; the leader's own producers arrive locally.
__device__ __forceinline__ void arrive_leader(uint64_t* bar, bool leader) {
  if (leader) mbar_arrive(bar);
  else mbar_arrive_cluster_relaxed(bar, 0);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
moments_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int T,
                  int BH, float inv_h, float* __restrict__ m_out,
                  float* __restrict__ omega_out, float* __restrict__ mom, uint4* __restrict__ pimg,
                  int npass, int fault, int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + SM_BAR);
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

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
  const int nb = pscr::pair_blocks(T, ptile);     // even: a last block past jend has zero weights
  // key blocks streamed: max sweep, weight sweep (each padded with zero blocks to nb4, whole
  // chunks of SCH), npass feature passes (NPASS for the moments, 0 when only the weights, m and
  // omega are wanted)
  const int nb4 = (nb + SCH - 1) / SCH * SCH;
  const int G = 2 * nb4 + npass * nb;
  const long long base = bh * T;
  // This CTA's P blocks in the scratch (layout: pscr:: in the internal header).
  uint4* const ptile_p = pimg + pscr::first_block(bh, T, ptile, rank) * (P_BLOCK / 16);
  // Rows of this CTA's key stage: the Q K^T operand takes rows 0..15 of each CTA's stage as its
  // N/2 keys, so CTA 1 keeps keys 16..31 of a block in rows 0..15 (row = key ^ 16 * rank).
  const int krot = 16 * rank;

  if (tid == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar.kfull[s], 32);  // one cp.async completion arrival per loader lane
      mbar_init(&bar.kfull_peer[s], 1);
      mbar_init(&bar.kempty[s], 1 + NFGW);
    }
    for (int s = 0; s < NSC; ++s) {
      mbar_init(&bar.sfull[s], 1);
      mbar_init(&bar.sfree[s], 2 * NSM);
    }
    for (int s = 0; s < NBUF; ++s) {
      mbar_init(&bar.pfull[s], 2 * NSM);
      mbar_init(&bar.pfree[s], 1);
    }
    for (int s = 0; s < NFB; ++s) {
      mbar_init(&bar.ffull[s], 2 * NFGW);
      mbar_init(&bar.ffree[s], 1);
    }
    mbar_init(&bar.accfull, nb >= 2 ? 2 : 1);  // one commit per feature issuer with steps in a pass
    mbar_init(&bar.accfree, 2 * NSM);
    mbar_init(&bar.qready, 2 * 4);
    mbar_init(&bar.done_qk, 1);
    mbar_init(&bar.done_f[0], 1);
    mbar_init(&bar.done_f[1], 1);
    mbar_init(&bar.hand[0], 1);
    mbar_init(&bar.hand[1], 1);
    mbar_init(&bar.rowx, NSM);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(&tmem_base_s, TMEM_COLS);
    tmem_relinquish_pair();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  volatile int* abort_p = &abort_flag;
  const int TO = kStatusTimeout;

  if (warp == 0) {
    // ------------------------------------------------------------------ Q K^T issuer (leader)
    // Two threads issue the tensor-core work (this one and the feature issuer): a single thread's
    // serial issue cost -- mbarrier tests, descriptor arithmetic and the MMA/commit instructions
    // -- exceeds the tensor work of a key block. tcgen05.commit tracks the issuing thread's own
    // MMAs, so each thread signals and drains its own. Q K^T runs only in the max and weight
    // sweeps, one chunk of SCH key blocks (N = 128) per MMA group: an MMA costs its issuer about
    // as long at N = 32 as at N = 128.
    if (leader && lane == 0) {
      const uint64_t kd = smem_desc(smem_u32(smem + SM_K), 128, 1024);
      constexpr uint32_t id_qk = idesc_bf16(PM, SCH * KB, false, false);
      const uint32_t t_s = tbase + T_S, t_q = tbase + T_Q;
      bool ok = mbar_wait(&bar.qready, 0, status, TO, abort_p);
      const int nchunks = 2 * nb4 / SCH;
      for (int u = 0; u < nchunks && ok; ++u) {
        // chunk u: key blocks g = SCH u .. SCH u + 3 in stages st0 .. st0 + 3 (fill g / KS)
        const int sb = u % NSC, st0 = (SCH * u) % KS;
        const uint32_t kpar = (uint32_t)((SCH * u / KS) & 1);
        for (int t = 0; t < SCH && ok; ++t)
          ok = mbar_wait2(&bar.kfull[st0 + t], kpar, &bar.kfull_peer[st0 + t], kpar, status, TO,
                          abort_p);
        if (ok && u >= NSC)
          ok = mbar_wait(&bar.sfree[sb], ((u / NSC) - 1) & 1, status, TO, abort_p);
        if (!ok) break;
        tc_fence_after();
        fence_proxy_async_smem();  // the stages' cp.async writes, before the async-proxy reads
        // Every descriptor is a base descriptor plus a start-address offset (16-byte units, which
        // cannot carry out of the 14-bit field since shared memory is below 256 KiB).
        const uint64_t kst = kd + (uint64_t)((st0 / SCH) * (SCH * K_STAGE >> 4));
        const uint32_t ts = t_s + sb * (SCH * KB);
        mma2_ts(ts, t_q, kst, id_qk, 0u);
        mma2_ts(ts, t_q + 8, kst + 16, id_qk, 1u);
        mma2_ts(ts, t_q + 16, kst + 32, id_qk, 1u);
        mma2_ts(ts, t_q + 24, kst + 48, id_qk, 1u);
        mma2_commit_both(&bar.sfull[sb]);
        for (int t = 0; t < SCH; ++t) mma2_commit_both(&bar.kempty[st0 + t]);
      }
      if (!ok) *abort_p = 1;
      mma2_commit_both(&bar.done_qk);
    } else if (!leader && lane == 0) {
      // Relay (the peer CTA): the leader's Q K^T reads this CTA's half of every sweep block, so
      // each landed block is fenced for the async proxy and reported to the leader. A stage is
      // refilled only after the Q K^T that needs this report, so no phase is skipped.
      for (int g = 0; g < 2 * nb4; ++g) {
        const int st = g % KS;
        if (!mbar_wait(&bar.kfull[st], (g / KS) & 1, status, TO, abort_p)) break;
        fence_proxy_async_smem();
        mbar_arrive_cluster_relaxed(&bar.kfull_peer[st], 0);
      }
    }
    __syncwarp();
  } else if (warp >= NWARPS - 2) {
    // ------------------------------------------------------------------ feature issuers (leader)
    // Issuing a step's 8 MMAs takes about as long as the tensor core takes to run them (the MMA
    // queue is shallow), and one thread's barrier tests between steps left the pipe idle. Two
    // threads therefore take alternate steps: while one issues step h, the other tests the
    // barriers of step h + 1, then waits only for the hand-off (hand[]) that says step h is
    // issued, so the issue order -- and the accumulation order -- stays fixed. The hand-off is
    // bracketed by tcgen05 fences, which order one thread's MMAs after the other's. Each thread
    // commits its own MMAs; both commit to accfull at the end of a pass.
    if (leader && lane == 0) {
      const int t = warp - (NWARPS - 2);
      const uint64_t fd = smem_desc(smem_u32(smem + SM_F), 128, 512);
      constexpr uint32_t id_a = idesc_bf16(PM, NA, false, true);
      constexpr uint32_t id_b = idesc_bf16(PM, NB_, false, true);
      constexpr uint32_t nb_off = GA * 512 / 16;  // local group GA: the N = 176 MMA's half
      const uint32_t t_acc = tbase + T_ACC, t_p = tbase + T_P;
      const int H = nb * npass;
      bool ok = true;
      int b = t % nb, pass = t / nb;  // block and pass of step h
      for (int h = t; h < H && ok; h += 2) {
        const int pb = h % NBUF, fb = h % NFB;
        ok = mbar_wait2(&bar.pfull[pb], (h / NBUF) & 1, &bar.ffull[fb], (h / NFB) & 1, status, TO,
                        abort_p);
        if (ok && b == 0 && pass >= 1)
          ok = mbar_wait(&bar.accfree, (pass - 1) & 1, status, TO, abort_p);
        if (ok && h >= 1) ok = mbar_wait(&bar.hand[t ^ 1], ((h - 1) >> 1) & 1, status, TO, abort_p);
        if (!ok) break;
        tc_fence_after();
        const uint64_t fh = fd + (uint64_t)(fb * (F_BUF >> 4));
        const uint64_t fl = fh + (F_HALF >> 4);
        const uint32_t a0 = t_p + pb * (KB / 2);
        const uint32_t acc0 = b > 0 ? 1u : 0u;
        // K-step 0 (keys 0..15), then K-step 1 (keys 16..31; +256 B in the F tiles); the hi and lo
        // tiles of each feature column go into the same accumulator.
        mma2_ts(t_acc, a0, fh, id_a, acc0);
        mma2_ts(t_acc, a0, fl, id_a, 1u);
        mma2_ts(t_acc + NA, a0, fh + nb_off, id_b, acc0);
        mma2_ts(t_acc + NA, a0, fl + nb_off, id_b, 1u);
        mma2_ts(t_acc, a0 + 8, fh + 16, id_a, 1u);
        mma2_ts(t_acc, a0 + 8, fl + 16, id_a, 1u);
        mma2_ts(t_acc + NA, a0 + 8, fh + nb_off + 16, id_b, 1u);
        mma2_ts(t_acc + NA, a0 + 8, fl + nb_off + 16, id_b, 1u);
        tc_fence_before();
        mbar_arrive(&bar.hand[t]);
        mma2_commit_both(&bar.pfree[pb]);
        mma2_commit_both(&bar.ffree[fb]);
        if (b >= nb - 2) mma2_commit_both(&bar.accfull);  // this thread's last step of the pass
        b += 2;
        while (b >= nb) { b -= nb; ++pass; }
      }
      if (!ok) *abort_p = 1;
      mma2_commit_both(&bar.done_f[t]);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ key-tile loader
    // cp.async 16-byte copies, every stage in flight. Lane -> (row, chunk) mapping:
    // rows (lane & 7) + 8 * (t & 3), chunks (lane >> 3) + 4 * (t >> 2): each 8-lane phase writes
    // 8 distinct bank groups, and each warp request reads whole 32-byte sectors. Each lane's
    // copies of a block complete on the stage's barrier (cp.async.mbarrier.arrive), so the loader
    // never waits for its own copies; the consumers that read through the async proxy (Q K^T)
    // fence after their wait (cp.async writes belong to the generic proxy).
    // With the test-only fault LLA_FAULT_WITHHOLD_KEYS the first key block is never staged: every
    // wait that needs it runs out after the wait limit, so the timeout path can be tested.
    const __nv_bfloat16* kb = k + base * D;
    for (int g = 0; g < G; ++g) {
      const int st = g % KS;
      const int b = g < 2 * nb4 ? g % nb4 : (g - 2 * nb4) % nb;  // sweep blocks >= nb: zeros
      if (g >= KS && !warp_wait(&bar.kempty[st], ((g / KS) - 1) & 1, status, abort_p)) break;
      if (g == 0 && fault == LLA_FAULT_WITHHOLD_KEYS) continue;
      uint8_t* dst = smem + SM_K;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int r = (lane & 7) + 8 * (t & 3), c = (lane >> 3) + 4 * (t >> 2);
        const int j = b * KB + (r ^ krot);
        const bool in = j < jend;
        cp_async16(dst + kst_off(st, r, c), kb + (long long)(in ? j : 0) * D + c * 8, in ? 16u : 0u);
      }
      cp_async_mbar_arrive(&bar.kfull[st]);
    }
    cp_async_commit();
    cp_async_wait<0>();  // nothing of this warp is in flight at teardown
  } else if (warp < 2 + NSM) {
    // ------------------------------------------------------------------ softmax + epilogue
    // Two warps per TMEM lane quarter: `half` 0 takes key columns 0..15 of each block and
    // accumulator columns [0, NA); half 1 takes keys 16..31 and columns [NA, NCH). Row max and
    // omega are combined across the halves through shared memory (barrier rowx: phase 0 after the
    // max sweep, phase 1 at the end). In the weight sweep each thread stores its 16 weights of
    // each block to the scratch; in the feature passes it reads its own stores back and writes
    // them to tensor memory, so Q K^T and the exponentials run only twice.
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;
    const bool valid = r < nq;
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const int c_lo = half * (KB / 2);
    const float c2 = inv_h * 1.4426950408889634f;  // log2(e) / h
    if (half == 0) {  // this row of Q into tensor memory (packed bf16 pairs, 32 columns)
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
    float* epi = reinterpret_cast<float*>(smem + SM_EPI) + (warp - 2) * 32 * EPI_LD;
    // Drains this half's accumulator columns of feature pass `pass` into its slots of mom.
    // Through a per-warp shared buffer, so that each store instruction writes whole 128-byte
    // lines of 4 rows instead of 16 bytes of 32 rows.
    auto drain = [&](int pass) -> bool {
      if (!warp_wait(&bar.accfull, pass & 1, status, abort_p)) return false;
      tc_fence_after();
      const int e0 = half ? NA : 0, e1 = half ? NCH : NA;
      const long long row0 = base + i0 + quarter * 32;
#pragma unroll 1
      for (int c0 = e0; c0 < e1; c0 += 32) {
        const int w = min(32, e1 - c0);
        uint32_t v[16];
        tmem_ld16(lane_base + T_ACC + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 4; ++t)
          *reinterpret_cast<uint4*>(epi + lane * EPI_LD + 4 * t) =
              make_uint4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
        if (w > 16) {
          tmem_ld16(lane_base + T_ACC + c0 + 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 4; ++t)
            *reinterpret_cast<uint4*>(epi + lane * EPI_LD + 16 + 4 * t) =
                make_uint4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
        }
        __syncwarp();
        const int chunk = lane & 7;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int rr = 4 * it + (lane >> 3);
          if (quarter * 32 + rr < nq && 4 * chunk < w)
            *reinterpret_cast<float4*>(mom + (row0 + rr) * NFP + pass * NCH + c0 + 4 * chunk) =
                *reinterpret_cast<const float4*>(epi + rr * EPI_LD + 4 * chunk);
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&bar.accfree, leader);
      return true;
    };
    float m = -INFINITY, om = 0.f;
    bool ok = true;
    // Sweep chunk u covers key blocks b0 .. b0 + SCH - 1. Column n of its S buffer holds key
    // 16 (n / 64) + n % 16 of block (n % 64) / 16 (the pair's B operand: 64 rows from each CTA),
    // so this thread's 16 logits of block b0 + t are columns 64 half + 16 t .. + 15.
    for (int u = 0; u < 2 * nb4 / SCH && ok; ++u) {
      const int sb = u % NSC;
      if (!warp_wait(&bar.sfull[sb], (u / NSC) & 1, status, abort_p)) { ok = false; break; }
      tc_fence_after();
      const bool max_sweep = SCH * u < nb4;
      const int b0 = (SCH * u) % nb4;
      for (int t = 0; t < SCH && ok; ++t) {
        uint32_t sv[KB / 2];
        tmem_ld16(lane_base + T_S + sb * (SCH * KB) + half * (SCH * KB / 2) + t * (KB / 2), sv);
        tmem_ld_wait();
        if (t == SCH - 1) {  // the chunk's S is read: the buffer is free
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&bar.sfree[sb], leader);
        }
        const int b = b0 + t;
        if (b >= nb) continue;  // padding block of the chunk
        const int j0 = b * KB + c_lo;
        if (max_sweep) {
#pragma unroll
          for (int c = 0; c < KB / 2; ++c)
            if (valid && j0 + c <= i) m = fmaxf(m, __uint_as_float(sv[c]));
          if (b == nb - 1) {  // combine the two halves' row maxima
            bar.part[half][r] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.rowx);
            if (!warp_wait(&bar.rowx, 0, status, abort_p)) { ok = false; break; }
            m = fmaxf(m, bar.part[half ^ 1][r]);
          }
          continue;
        }
        const float mc = m * c2;
        uint32_t pw[KB / 4];
#pragma unroll
        for (int c = 0; c < KB / 2; c += 2) {
          const float p0 =
              (valid && j0 + c <= i) ? ex2(fmaf(__uint_as_float(sv[c]), c2, -mc)) : 0.f;
          const float p1 =
              (valid && j0 + c + 1 <= i) ? ex2(fmaf(__uint_as_float(sv[c + 1]), c2, -mc)) : 0.f;
          pw[c / 2] = pack_bf16(p0, p1);
          om += __uint_as_float(pw[c / 2] << 16) + __uint_as_float(pw[c / 2] & 0xFFFF0000u);
        }
        // This row's 16 weights as chunks 2*half and 2*half + 1 of the block's image.
        constexpr int kChunk = 2048 / 16;  // chunk stride of the image, in 16-byte units
        uint4* pdst = ptile_p + (long long)b * (P_BLOCK / 16) + (2 * half) * kChunk + r;
        pdst[0] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        pdst[kChunk] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      }
    }
    {
      // This thread's weights of feature step h (block h % nb; the weight sweep stored them:
      // same row, same 16 keys), copied PD steps ahead into slot h % PD of this thread's ring.
      constexpr int kChunk = 2048 / 16;
      // slot s, chunk c of this lane at ring + s * 64 + c * 32 (a warp's accesses are contiguous)
      uint4* ring = reinterpret_cast<uint4*>(smem + SM_PR) + (warp - 2) * PD * 64 + lane;
      const int hend = nb * npass;
      auto fetch = [&](int hh) {
        if (hh < hend) {
          const uint4* src =
              ptile_p + (long long)(hh % nb) * (P_BLOCK / 16) + (2 * half) * kChunk + r;
          uint4* dst = ring + (hh % PD) * 64;
          cp_async16(dst, src, 16u);
          cp_async16(dst + 32, src + kChunk, 16u);
        }
        cp_async_commit();  // an empty group past the end keeps the wait count uniform
      };
      if (ok)
        for (int t = 0; t < PD; ++t) fetch(t);
      int h = 0;  // feature step index
      for (int pass = 0; pass < npass && ok; ++pass) {
        for (int b = 0; b < nb; ++b, ++h) {
          cp_async_wait<PD - 1>();
          const uint4* slot = ring + (h % PD) * 64;
          const uint4 c0 = slot[0], c1 = slot[32];
          const int pb = h % NBUF;
          if (h >= NBUF &&
              !warp_wait(&bar.pfree[pb], ((h / NBUF) - 1) & 1, status, abort_p)) { ok = false; break; }
          tc_fence_after();
          const uint32_t pw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          tmem_st8(lane_base + T_P + pb * (KB / 2) + half * (KB / 4), pw);
          tmem_st_wait();
          fetch(h + PD);  // the slot's values are consumed (stored to tensor memory)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&bar.pfull[pb], leader);
        }
        if (ok) ok = drain(pass);
      }
      cp_async_wait<0>();
    }
    if (ok) {  // combine the halves' omega
      bar.part[half][r] = om;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.rowx);
      if (warp_wait(&bar.rowx, 1, status, abort_p) && half == 0 && valid) {
        m_out[base + i] = m * inv_h;
        omega_out[base + i] = om + bar.part[1][r];
      }
    }
  } else {
    // ------------------------------------------------------------------ feature generation (warps 10-21)
    // Group `grp` (warps 10-15 or 16-21) takes the key blocks of steps g with g % 2 == grp, so
    // each warp has two steps' time for its serial chain (barrier tests, key-word loads, the
    // products, the proxy fence).
    const int fwi = warp - 2 - NSM, grp = fwi / NFGW, fw = fwi % NFGW;
    const int row_off = (lane >> 3) * 128 + (lane & 7) * 16;  // key `lane` in the F tiles
    int st = grp, h = grp - 2 * nb4, pass = -1, bcnt = 0;
    uint32_t kpar = 0;
    for (int g = grp; g < G; g += 2) {
      if (!warp_wait(&bar.kfull[st], kpar, status, abort_p)) break;
      if (g < 2 * nb4) {  // max and weight sweeps: nothing to generate
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.kempty[st]);
      } else {
        if (pass < 0) { pass = h / nb; bcnt = h % nb; }  // this group's first feature step
        const int fb = h % NFB;
        uint32_t kw[33];
        const uint8_t* kst = smem + SM_K;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(kst + kst_off(st, lane ^ krot, c));
          kw[4 * c] = v.x; kw[4 * c + 1] = v.y; kw[4 * c + 2] = v.z; kw[4 * c + 3] = v.w;
        }
        kw[32] = 0x00003F80u;  // bf16 one (constant feature) and zero (padding)
        __syncwarp();
        // Feature passes run no Q K^T, whose completion is the stage's other release: warp 0 of
        // the group arrives for it.
        if (lane == 0) mbar_arrive_cnt(&bar.kempty[st], fw == 0 ? 2u : 1u);
        if (h >= NFB && !warp_wait(&bar.ffree[fb], ((h / NFB) - 1) & 1, status, abort_p)) break;
        uint8_t* fhi = smem + SM_F + fb * F_BUF;
        generate(pass, rank, fw, kw, fhi, fhi + F_HALF, row_off);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) arrive_leader(&bar.ffull[fb], leader);
      }
      // next step of this group: g + 2
      h += 2;
      if (pass >= 0) {
        bcnt += 2;
        while (bcnt >= nb) { bcnt -= nb; ++pass; }
      }
      st += 2;
      if (st >= KS) { st -= KS; kpar ^= 1; }
    }
  }

  // Teardown: tensor memory is released only after every MMA of the pair has completed (bounded
  // waits, whatever the abort flag says), and neither CTA exits before the other has made its
  // last arrival on it.
  if (warp == 0 && lane == 0) {
    volatile int never = 0;
    mbar_wait(&bar.done_qk, 0, status, TO, &never);
    mbar_wait(&bar.done_f[0], 0, status, TO, &never);
    mbar_wait(&bar.done_f[1], 0, status, TO, &never);
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

size_t moments_tc_row_floats() { return NFP; }

size_t moments_tc_pscratch_bytes(long long BH, int T) {
  return (size_t)BH * (size_t)pscr::blocks_per_head(T) * P_BLOCK;
}

namespace {
cudaError_t launch_tc(const Args& a, const Workspace& ws, cudaStream_t s, int npass) {
  auto kern = moments_tc_kernel;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
  if (err != cudaSuccess) return err;
  const long long blocks = 2ll * ((a.T + PM - 1) / PM) * a.BH();
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, NTHREADS, SMEM_LAUNCH, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k), a.T,
      (int)a.BH(), 1.0f / a.h, ws.m, ws.omega, ws.mom, static_cast<uint4*>(ws.pscr), npass,
      a.fault, ws.status);
  count_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_moments_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  return launch_tc(a, ws, s, NPASS);
}

cudaError_t launch_weights_tc(const Args& a, const Workspace& ws, cudaStream_t s) {
  return launch_tc(a, ws, s, 0);
}

}  // namespace lla
