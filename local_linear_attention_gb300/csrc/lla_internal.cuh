// Internal declarations shared by the liblla translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lla.h"

namespace lla {

// Bits of the per-device status word (see lla_stream_status()).
enum : int {
  kStatusNumerical = 1 << 0,
  kStatusTimeout = 1 << 1,
  kStatusBadIndex = 1 << 2,
};

// Problem description after host-side validation.
struct Args {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int B, H, T, d, dv;
  float h, lam;
  int dtype;  // lla_dtype
  // Per-call options (lla_options), validated by the API layer.
  int path_req = 0;      // lla_path requested (0 = automatic)
  int form = 0;          // kFormCentred or kFormPage
  int cg_iters = 1024;   // conjugate-gradient strategy: iteration cap
  float cg_tol = 1e-3f;  //   and relative residual tolerance
  int fault = 0;         // test-only fault of the tensor-core moments stage (lla_test_fault)
  long long BH() const { return (long long)B * H; }
  long long rows() const { return (long long)B * H * T; }
};

// Augmented-key Gram layout used by the CUDA-core moments path.
// The augmented key is kt = [k - c, 1, 0...] of padded length DP = 4*NBLK; the moments of a
// query are the upper-triangular 4x4 blocks of sum_j p_j kt_j kt_j^T, block (ba, bb) with
// ba <= bb stored as 16 consecutive floats (row-major inside the block), blocks enumerated
// row by row. G(D, D) = omega, G(a, D) = sum p (k - c)_a, G(a, b) = sum p (k - c)_a (k - c)_b.
__host__ __device__ constexpr int gram_nblk(int D) { return (D + 1 + 3) / 4; }
__host__ __device__ constexpr int gram_nblocks(int D) { return gram_nblk(D) * (gram_nblk(D) + 1) / 2; }
__host__ __device__ constexpr int gram_floats(int D) { return gram_nblocks(D) * 16; }
__host__ __device__ constexpr int gram_block_index(int D, int ba, int bb) {
  return ba * gram_nblk(D) - ba * (ba - 1) / 2 + (bb - ba);
}

// Device scratch carved out of one workspace allocation.
struct Workspace {
  float* kmean;   // [BH, d]        per-head key reference point c
  float* vmean;   // [BH, dv]       per-head value reference point c_v
  float* m;       // [BH*T]         row max of the logits q.k/h over the causal prefix
  float* mom;     // [BH*T, G]      augmented Gram moments (hi part)
  float* mom_lo;  // [BH*T, G]      compensation terms (fp32 inputs only, else nullptr)
  float* y;       // [BH*T, d]      ridge-solve result y = (C_kk + lambda' I)^-1 (q - kbar)
  float* kbar;    // [BH*T, d]      kbar - c, the weighted key mean in the shifted frame
  float* omega;   // [BH*T]         sum of the weights (tensor-core moments path)
  uint32_t* ytc;  // [BH*T, 3, d/2]  tensor-core path: y as three exact bf16 parts (y = y1 + y2 + y3),
                  //                each part a row of d bf16 (packed pairs), for the readout
  float* cy;      // [BH*T]         tensor-core path: kbar . y
  void* pscr;     // tensor-core path: the kernel weights P of feature pass 0, bf16, one 8 KiB
                  // image per (head, query tile, key block), reused by the later passes
  __nv_bfloat16* ksh;  // [BH*T, d]  tensor-core path: the keys in the head's frame, bf16(k - c)
  float* kref;         // [BH, d]    tensor-core path: the head's reference key c (bf16 values)
  float* kstat;        // [BH, kKeyStatChunks, 2, d]  partial sums of k and k^2 for choosing c
  int* rep;            // tensor-core path: [1 + kMaxRepairRows] count, then rows whose
                       // factorisation the precise repair pass redoes; one more int after them
  int* short_count;    // rows listed for the exact pass (lla_short.cu) ...
  int* short_rows;     // ... and their flat indices, at most BH * min(T, 64) (tensor-core path:
                       // the int after rep's rows, and kstat, free once the key frame is chosen;
                       // CUDA-core path: a region of its own)
  int* status;    // device status word of the current device
  int path;       // kPathCudaCore or kPathTensorCore: which moments stage (and layout) is used
  int form;       // kFormCentred or kFormPage: which closed form the solve and readout evaluate
};

// Moments implementations. The tensor-core stage handles bf16 inputs with d = 64 and leaves the
// keys unshifted (c = 0: shifted bf16 keys would no longer multiply exactly); everything else
// uses the CUDA-core stage.
enum : int { kPathCudaCore = 1, kPathTensorCore = 2, kPathCG = 3 };
// Closed forms of the intercept (both exact): the centred one, o = vbar + C_vk y, and the page's,
// o = sum p (1 - z . rho*) v / sum p (1 - z . rho*) with z = k - q. The page form runs on the
// tensor-core dense strategy with d = dv = 64 only.
enum : int { kFormCentred = 0, kFormPage = 1 };
int choose_path(const Args& a);

size_t workspace_bytes(const Args& a);
void carve_workspace(const Args& a, void* base, Workspace* ws);

// bf16 inputs with d < 64 run on the d = dv = 64 tensor-core path with zero-padded copies of q,
// k and v (lla_pad.cu; the padded features change nothing). Copies a's q, k, v ([rows][d] and
// [rows][dv] bf16) to [rows][64] with zeros after, and the first dv columns of o64 back to a.out.
inline bool pad_eligible(const Args& a) {
  return a.dtype == LLA_BF16 && a.d < 64 && a.path_req != kPathCudaCore;
}
cudaError_t launch_pad_inputs(const Args& a, void* q64, void* k64, void* v64, cudaStream_t s);
cudaError_t launch_unpad_output(const Args& a, const void* o64, cudaStream_t s);

// Kernel launchers (one per stage). Each returns the launch error, if any.
cudaError_t launch_prep(const Args& a, const Workspace& ws, cudaStream_t s);
cudaError_t launch_moments_ffma(const Args& a, const Workspace& ws, cudaStream_t s);
// The moment contraction of the tensor-core path (lla_moments_pass_tc.cu): reads the weight
// images that launch_weights_tc wrote and fills the moment rows.
cudaError_t launch_moments_pass_tc(const Args& a, const Workspace& ws, cudaStream_t s);
size_t moments_tc_pscratch_bytes(long long BH, int T);

// Layout of the tensor-core path's weight scratch: the bf16 kernel weights P of every (head,
// query tile, key block), written by the moments stage's weight sweeps and read back by the moment
// contraction, the readout and the precise repair pass. Query tiles of 128 rows go in pairs
// (ptile: 256 queries); a pair streams key blocks 0..nb-1 of 32 keys, nb = 2 ceil(min(T,
// 256 (ptile + 1)) / 64) (an even count: the contraction takes key blocks two at a time; a block
// past the pair's last key holds zero weights). A pair's rank-0 tile's nb blocks come first, then
// its rank-1 tile's; the pairs of a head follow one another (a full pair p holds 2 x 8 (p + 1)
// blocks). A block is an 8 KiB image in which 16-byte chunk kc (keys 8kc..8kc+7) of row r sits at
// kc * 2048 + r * 16: the no-swizzle K-major core-matrix layout of a 128 x 32 bf16 tcgen05
// operand (K-adjacent core matrices 2048 B apart, M-adjacent 128 B).
namespace pscr {
constexpr int kRows = 128;
constexpr int kKeys = 32;
constexpr int kBlockBytes = kRows * kKeys * 2;
__host__ __device__ inline int pair_blocks(int T, int ptile) {
  const int jend = T < 256 * (ptile + 1) ? T : 256 * (ptile + 1);
  return 2 * ((jend + 2 * kKeys - 1) / (2 * kKeys));
}
__host__ __device__ inline long long blocks_per_head(int T) {
  const long long np = (T + 255) / 256;
  return np > 0 ? 8 * (np - 1) * np + 2ll * pair_blocks(T, (int)np - 1) : 0;
}
// Index (in blocks) of block 0 of tile (ptile, rank) of head bh.
__host__ __device__ inline long long first_block(long long bh, int T, int ptile, int rank) {
  return bh * blocks_per_head(T) + 8ll * ptile * (ptile + 1) + (long long)rank * pair_blocks(T, ptile);
}
}  // namespace pscr
// Chunks of a head's keys whose partial statistics choose the tensor-core path's key reference.
constexpr int kKeyStatChunks = 16;
// Rows per call whose tensor-core ridge factorisation may be redone by the precise repair pass
// (more failing rows than this are reported as LLA_ERR_NUMERICAL and left NaN).
constexpr int kMaxRepairRows = 4096;
// Rows whose causal prefix holds at most kShortMaxKeys keys may be recomputed exactly
// (lla_short.cu); the solve lists them: with at most d keys (the centred key covariance then has
// rank below d), every row of an fp32 call and the rows of a bf16 call whose factorisation failed;
// besides, any such row whose |y|_inf (|kbar - c|_1 + sqrt(d tr(C_kk) / omega)) -- the size of
// k . y against which the readout's k . y - kbar . y must cancel -- exceeds kShortY (bf16) or
// kShortY32 (fp32). Measured on bf16 inputs, rows below kShortY stay within about 1e-2 of the
// exact output (about 1e-7 of the statistic at worst); rows above it (a tiny effective ridge with
// the query far from kbar, as with a large common key offset) reached 0.11.
constexpr int kShortMaxKeys = 64;
constexpr float kShortY = 1e6f;
constexpr float kShortY32 = 1e3f;
// The solves mark a listed row for the readouts with this quiet-NaN pattern (in cy on the
// tensor-core readout's input, in kbar[row][0] on the CUDA-core readout's): the readout then
// leaves the row's output to the exact pass, which runs concurrently. A row whose solve failed
// outright (repair list full) carries the plain NaN 0x7fc00000 instead and is stored as NaN.
constexpr uint32_t kListedBits = 0x7fc0beefu;
// The tensor-core stage may run for these sizes (whatever path is requested at call time).
inline bool tc_eligible(const Args& a) { return a.dtype == LLA_BF16 && a.d == 64; }
cudaError_t launch_solve(const Args& a, const Workspace& ws, cudaStream_t s);
cudaError_t launch_readout(const Args& a, const Workspace& ws, cudaStream_t s);
cudaError_t launch_readout_tc(const Args& a, const Workspace& ws, cudaStream_t s);
// The exact pass over the rows the solve listed (after the readout; overwrites their output).
cudaError_t launch_short_prefix(const Args& a, const Workspace& ws, cudaStream_t s);
// Entries of the CUDA-core path's short-row region: the count, then at most
// BH * min(T, kShortMaxKeys) rows.
inline size_t short_list_ints(const Args& a) {
  return 1 + (size_t)a.BH() * (size_t)(a.T < kShortMaxKeys ? a.T : kShortMaxKeys);
}
// The tensor-core readout pass with fp32 output, values `v` (bf16, [B,H,T,64]), y given as
// three bf16 parts and kbar . y, tiles with tile_active[tile] == 0 skipped (null: none); matvec:
// only the covariance branch (out = C_vk y, which is C_kk y for v = k).
cudaError_t launch_readout_tc_f32(const Args& a, const Workspace& ws, cudaStream_t s,
                                  const void* v, const uint32_t* ytc, const float* cy, float* out,
                                  const int* tile_active, bool matvec);
// The weight sweeps of the tensor-core path (lla_weights_tc.cu): m, omega and the weight images.
cudaError_t launch_weights_tc(const Args& a, const Workspace& ws, cudaStream_t s);
// Conjugate-gradient strategy for the ridge systems (bf16, d = dv = 64): fills ytc and cy like
// the tensor-core solve, with its state in the moments region of the workspace.
cudaError_t launch_cg_solve(const Args& a, const Workspace& ws, cudaStream_t s, int max_iters,
                            float rel_tol);
size_t cg_state_bytes(const Args& a);
// Causal Parallax forward with probe r (same layout as q); tensor cores when path ==
// kPathTensorCore and the shape is bf16 with d = dv = 64, CUDA cores otherwise.
cudaError_t launch_parallax(const Args& a, const void* r, int path, int* status, cudaStream_t s);
cudaError_t launch_debug_moments(const Args& a, const int64_t* idx, int n, float* m,
                                 float* omega, float* sk, float* sv, float* Skk, float* Svk,
                                 int* status, cudaStream_t s);

// Decode: one query per head against a cache of L keys/values (q, r: [B,H,d]; k: [B,H,L,d];
// v: [B,H,L,dv]; out: [B,H,dv]). r == nullptr: LLA; otherwise Parallax with probe r.
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* r;
  void* out;
  int B, H, L, d, dv;
  float h, lam;
  int dtype;
  int path = 0;  // LLA, bf16, d = dv = 64: tensor cores unless kPathCudaCore
  long long BH() const { return (long long)B * H; }
};
// Causal Parallax backward (the gradients of lla_parallax_forward with respect to q, k, v, r).
struct ParallaxBwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* r;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  void* dr;
  int B, H, T, d, dv_;
  float h;
  int dtype;
  long long BH() const { return (long long)B * H; }
};
size_t parallax_bwd_workspace_bytes(const ParallaxBwdArgs& a);
// All three passes; bf16 with d = dv = 64 on tensor cores unless path == kPathCudaCore.
cudaError_t launch_parallax_bwd(const ParallaxBwdArgs& a, void* ws, int path, int* status,
                                cudaStream_t s);
// Tensor-core pieces (bf16, d = dv = 64): the row records from the tensor-core forward, then
// the rows and columns passes.
cudaError_t launch_parallax_stats_tc(const ParallaxBwdArgs& a, float* stats, int* status,
                                     cudaStream_t s);
cudaError_t launch_parallax_bwd_tc(const ParallaxBwdArgs& a, float* stats, int* status,
                                   cudaStream_t s);

size_t decode_workspace_bytes(const DecodeArgs& a);
cudaError_t launch_decode(const DecodeArgs& a, void* ws, int* status, cudaStream_t s);

void count_launch();

// ---------------------------------------------------------------------------------------------
// Device helpers.
__device__ __forceinline__ float ldf(const float* p, long long i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stf(float* p, long long i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, long long i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// Error-free transforms on fp32 pairs (Knuth's TwoSum; the FMA-based exact product).
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x) {
  float t = hi + x;
  float z = t - hi;
  lo += (hi - (t - z)) + (x - z);
  hi = t;
}
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = a * b;
  e = fmaf(a, b, -p);
}

}  // namespace lla
