// Zero padding of bf16 inputs with d (and dv) below 64 to the d = dv = 64 tensor-core path.
//
// Extra key features that are zero for every key and query leave the LLA intercept unchanged:
// their logit terms q_a k_a vanish, so the weights are the same; their moments (sum p k_a, sum p
// k_a k_b) are exactly zero, so the ridge system is block-diagonal with lambda' I on the padded
// block, whose right-hand side (q - kbar on those features) is zero as well, so y is zero there
// and the readout's k_j . y gains nothing. Extra value features that are zero give zero output
// columns, which are dropped. The padded copies are row-major [BH*T][64] bf16.
#include "lla_internal.cuh"

namespace lla {
namespace {

// dst[row][0:8) (16-byte chunks of 8 bf16) = src[row][0:nsrc) followed by zeros; blockIdx.y
// selects the tensor (q, k, v).
__global__ void pad_rows_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                const uint4* __restrict__ v, int qk_chunks, int v_chunks,
                                uint4* __restrict__ q64, uint4* __restrict__ k64,
                                uint4* __restrict__ v64, long long rows) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * 8) return;
  const long long r = idx >> 3;
  const int c = (int)(idx & 7);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (blockIdx.y == 0) q64[idx] = c < qk_chunks ? q[r * qk_chunks + c] : zero;
  else if (blockIdx.y == 1) k64[idx] = c < qk_chunks ? k[r * qk_chunks + c] : zero;
  else v64[idx] = c < v_chunks ? v[r * v_chunks + c] : zero;
}

// out[row][0:nout) = o64[row][0:nout) (16-byte chunks).
__global__ void unpad_rows_kernel(const uint4* __restrict__ o64, int out_chunks,
                                  uint4* __restrict__ out, long long rows) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * out_chunks) return;
  const long long r = idx / out_chunks;
  const int c = (int)(idx - r * out_chunks);
  out[idx] = o64[r * 8 + c];
}

constexpr int kPadThreads = 256;

}  // namespace

cudaError_t launch_pad_inputs(const Args& a, void* q64, void* k64, void* v64, cudaStream_t s) {
  const long long rows = a.rows();
  const long long blocks = (rows * 8 + kPadThreads - 1) / kPadThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  pad_rows_kernel<<<dim3((unsigned)blocks, 3), kPadThreads, 0, s>>>(
      static_cast<const uint4*>(a.q), static_cast<const uint4*>(a.k),
      static_cast<const uint4*>(a.v), a.d / 8, a.dv / 8, static_cast<uint4*>(q64),
      static_cast<uint4*>(k64), static_cast<uint4*>(v64), rows);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_unpad_output(const Args& a, const void* o64, cudaStream_t s) {
  const long long rows = a.rows();
  const int out_chunks = a.dv / 8;
  const long long blocks = (rows * out_chunks + kPadThreads - 1) / kPadThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  unpad_rows_kernel<<<(unsigned)blocks, kPadThreads, 0, s>>>(
      static_cast<const uint4*>(o64), out_chunks, static_cast<uint4*>(a.out), rows);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lla
