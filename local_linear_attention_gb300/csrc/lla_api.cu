// C ABI of liblla: argument validation, scratch management, stage dispatch, device status word,
// launch counting and stage timing. Kernels live in the other translation units.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "lla_internal.cuh"

namespace lla {

// Per-device status word; kernels receive its address (see device_status()).
__device__ int g_status;

namespace {

std::atomic<unsigned long long> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_status_ptr[kMaxDevices] = {};
bool g_pool_ready[kMaxDevices] = {};

// The exact pass over short rank-deficient prefixes (lla_short.cu) runs on a side stream of the
// current device, concurrently with the readout: `fork` orders it after the solve on the call's
// stream, `join` orders the rest of the call after it. One side stream and event pair per device,
// created on first use, the stream at the device's highest priority: both grids become ready when
// the solve ends, and the pass's CTAs (which cannot share an SM with a readout CTA) must be
// dispatched before the readout's waves fill the GPU, not after them. The device's `mu` is held
// from the fork to the join's wait so that concurrent calls cannot wait on each other's records.
// The stream and events live until the process exits.
struct SideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;  // guards creation
SideStream g_side[kMaxDevices];

// The current device's side stream, created on first use (all three objects, or none).
cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream& sd = g_side[dev];
  std::lock_guard<std::mutex> lk(g_side_mu);
  if (!sd.s) {
    int least = 0, greatest = 0;
    cudaStream_t st = nullptr;
    cudaEvent_t ef = nullptr, ej = nullptr;
    err = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (err == cudaSuccess) err = cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ef, cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ej, cudaEventDisableTiming);
    if (err != cudaSuccess) {
      if (ej) cudaEventDestroy(ej);
      if (ef) cudaEventDestroy(ef);
      if (st) cudaStreamDestroy(st);
      return err;
    }
    sd.fork = ef;
    sd.join = ej;
    sd.s = st;
  }
  *out = &sd;
  return cudaSuccess;
}

// Address of the status word on the current device (resolved once per device).
cudaError_t device_status(int** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_status);
    if (err != cudaSuccess) return err;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// Once per device, for the entry points that take their scratch from the stream-ordered
// allocator: memory freed with cudaFreeAsync stays in the device's default pool instead of going
// back to the driver at every synchronisation, so repeated calls reuse their scratch. (Entry
// points that allocate nothing leave the pool's settings alone.)
cudaError_t ensure_pool() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_pool_ready[dev]) {
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      unsigned long long thr = ~0ULL;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
    g_pool_ready[dev] = true;
  }
  return cudaSuccess;
}

// Validates per-call options into `a` (forward: every field; other operations: path only).
int apply_options(const lla_options* o, bool forward, Args* a) {
  if (!o) return LLA_OK;
  for (int r : o->reserved)
    if (r != 0) return LLA_ERR_INVALID_ARG;
  if (o->path < LLA_PATH_AUTO || o->path > LLA_PATH_CG) return LLA_ERR_INVALID_ARG;
  if (!forward) {
    if (o->path == LLA_PATH_CG || o->form != 0 || o->cg_max_iters != 0 || o->cg_rel_tol != 0.f ||
        o->test_fault != 0)
      return LLA_ERR_INVALID_ARG;
    a->path_req = o->path;
    return LLA_OK;
  }
  if (o->form != LLA_FORM_CENTRED && o->form != LLA_FORM_PAGE) return LLA_ERR_INVALID_ARG;
  if (o->cg_max_iters < 0 || o->cg_max_iters > 1024) return LLA_ERR_INVALID_ARG;
  if (!(o->cg_rel_tol >= 0.f && o->cg_rel_tol < 1.f)) return LLA_ERR_INVALID_ARG;
  if (o->test_fault != LLA_FAULT_NONE && o->test_fault != LLA_FAULT_WITHHOLD_KEYS)
    return LLA_ERR_INVALID_ARG;
  a->path_req = o->path;
  a->form = o->form;
  a->cg_iters = o->cg_max_iters > 0 ? o->cg_max_iters : 1024;
  a->cg_tol = o->cg_rel_tol > 0.f ? o->cg_rel_tol : 1e-3f;
  a->fault = o->test_fault;
  return LLA_OK;
}

// ------------------------------------------------------------------------- stage timing
struct ProfRec {
  cudaEvent_t ev[LLA_NUM_STAGES + 1];
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_finite_pos(float x) { return std::isfinite(x) && x > 0.f; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point. Returns LLA_OK or an error status.
int check_shape(int B, int H, int T, int d, int dv, int dtype) {
  if (B < 0 || H < 0 || T < 0) return LLA_ERR_INVALID_ARG;
  if (dtype != LLA_F32 && dtype != LLA_BF16) return LLA_ERR_INVALID_ARG;
  if (!(d == 16 || d == 32 || d == 64) || !(dv == 16 || dv == 32 || dv == 64))
    return LLA_ERR_UNSUPPORTED;
  if ((long long)B * H * T >= (1LL << 31)) return LLA_ERR_UNSUPPORTED;
  return LLA_OK;
}

int check_forward(const Args& a) {
  int st = check_shape(a.B, a.H, a.T, a.d, a.dv, a.dtype);
  if (st != LLA_OK) return st;
  if (!is_finite_pos(a.h) || !is_finite_pos(a.lam)) return LLA_ERR_INVALID_ARG;
  if (a.rows() == 0) return LLA_OK;
  if (!a.q || !a.k || !a.v || !a.out) return LLA_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.out))
    return LLA_ERR_INVALID_ARG;
  return LLA_OK;
}

Args make_args(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int d,
               int dv, float h, float lam, int dtype) {
  Args a;
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.B = B; a.H = H; a.T = T; a.d = d; a.dv = dv;
  a.h = h; a.lam = lam; a.dtype = dtype;
  return a;
}

size_t elem_bytes(int dtype) { return dtype == LLA_F32 ? 4 : 2; }

// Runs every stage on `s` with scratch `base`. `user` (non-null) is the caller's call when `a` is
// its zero-padded d = dv = 64 form: the padding runs with the first stage, the copy of the
// output's columns back with the last.
int run_stages(const Args& a, void* base, cudaStream_t s, const Args* user) {
  Workspace ws;
  carve_workspace(a, base, &ws);
  if (ws.form == kFormPage && !(ws.path == kPathTensorCore && a.dv == 64)) return LLA_ERR_UNSUPPORTED;
  if (a.fault != 0 && ws.path != kPathTensorCore) return LLA_ERR_UNSUPPORTED;
  if (device_status(&ws.status) != cudaSuccess) return LLA_ERR_CUDA;
  ProfRec rec;
  bool prof = false;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof = g_prof_on;
  }
  if (prof) {
    for (auto& e : rec.ev)
      if (cudaEventCreate(&e) != cudaSuccess) return LLA_ERR_CUDA;
    cudaEventRecord(rec.ev[0], s);
  }
  auto none = [](const Args&, const Workspace&, cudaStream_t) { return cudaSuccess; };
  const bool tc = ws.path == kPathTensorCore;
  cudaError_t (*stages[LLA_NUM_STAGES])(const Args&, const Workspace&, cudaStream_t) = {
      launch_prep,
      tc ? launch_weights_tc : +none,
      tc ? launch_moments_pass_tc : launch_moments_ffma,
      launch_solve,
      (tc && a.dv == 64) ? launch_readout_tc : launch_readout};
  if (ws.path == kPathCG) {  // matrix-free CG for the ridge systems (bf16, d = dv = 64)
    stages[1] = launch_weights_tc;
    stages[2] = none;
    stages[3] = [](const Args& a2, const Workspace& w2, cudaStream_t s2) {
      return launch_cg_solve(a2, w2, s2, a2.cg_iters, a2.cg_tol);
    };
    stages[4] = launch_readout_tc;
  }
  // `main` on the call's stream with `side` beside it on the side stream: both ordered after
  // what the call's stream has enqueued so far, and the rest of the call after both.
  auto beside = [&](cudaError_t (*main)(const Args&, const Workspace&, cudaStream_t),
                    cudaError_t (*side)(const Args&, const Workspace&, cudaStream_t)) {
    SideStream* sd = nullptr;
    if (side_stream(&sd) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(sd->mu);
    return cudaEventRecord(sd->fork, s) == cudaSuccess &&
           cudaStreamWaitEvent(sd->s, sd->fork, 0) == cudaSuccess &&
           side(a, ws, sd->s) == cudaSuccess && cudaEventRecord(sd->join, sd->s) == cudaSuccess &&
           main(a, ws, s) == cudaSuccess && cudaStreamWaitEvent(s, sd->join, 0) == cudaSuccess;
  };
  for (int i = 0; i < LLA_NUM_STAGES; ++i) {
    if (i == 0 && user && launch_pad_inputs(*user, const_cast<void*>(a.q), const_cast<void*>(a.k),
                                            const_cast<void*>(a.v), s) != cudaSuccess)
      return LLA_ERR_CUDA;
    bool ok = true;
    if (tc && i == 0) {
      // the key frame runs beside the weight sweeps, which read the original keys (stage 1)
    } else if (tc && i == 1) {
      ok = beside(stages[1], stages[0]);
    } else if (i == LLA_NUM_STAGES - 1 && ws.path != kPathCG) {
      // the readout, with the exact pass over the rows the solve listed beside it
      ok = beside(stages[i], launch_short_prefix);
    } else {
      ok = stages[i](a, ws, s) == cudaSuccess;
    }
    if (!ok) return LLA_ERR_CUDA;
    if (i == LLA_NUM_STAGES - 1 && user && launch_unpad_output(*user, a.out, s) != cudaSuccess)
      return LLA_ERR_CUDA;
    if (prof) cudaEventRecord(rec.ev[i + 1], s);
  }
  if (prof) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back(rec);
  }
  return LLA_OK;
}

// The padded form of a call: d = dv = 64, q, k, v and out in the first four regions of `base`.
Args padded_args(const Args& a, void* base, void** rest) {
  const size_t row = align_up((size_t)a.rows() * 64 * 2);
  char* p = static_cast<char*>(base);
  Args a64 = a;
  a64.d = a64.dv = 64;
  a64.q = p;
  a64.k = p + row;
  a64.v = p + 2 * row;
  a64.out = p + 3 * row;
  *rest = p + 4 * row;
  return a64;
}

int run_forward(const Args& a, void* base, cudaStream_t s) {
  if (!pad_eligible(a)) return run_stages(a, base, s, nullptr);
  void* rest = nullptr;
  const Args a64 = padded_args(a, base, &rest);
  return run_stages(a64, rest, s, &a);
}

}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int choose_path(const Args& a) {
  const bool tc_ok = tc_eligible(a);
  const int req = a.path_req;
  if (req == kPathCudaCore || !tc_ok) return kPathCudaCore;
  if (req == kPathCG && a.dv == 64) return kPathCG;
  return kPathTensorCore;
}

size_t workspace_bytes(const Args& a) {
  if (pad_eligible(a)) {  // four padded [rows][64] bf16 tensors, then the d = 64 scratch
    Args a64 = a;
    a64.d = a64.dv = 64;
    return 4 * align_up((size_t)a.rows() * 64 * 2) + workspace_bytes(a64);
  }
  const size_t BH = (size_t)a.BH(), R = (size_t)a.rows();
  const size_t G = (size_t)gram_floats(a.d);
  size_t n = 0;
  n += align_up(BH * a.d * sizeof(float));               // kmean
  n += align_up(BH * a.dv * sizeof(float));              // vmean
  n += align_up(R * sizeof(float));                      // m
  n += align_up(R * G * sizeof(float));                  // mom
  if (a.dtype == LLA_F32) n += align_up(R * G * sizeof(float));  // mom_lo
  n += align_up(R * a.d * sizeof(float));                // y
  n += align_up(R * a.d * sizeof(float));                // kbar
  n += align_up(R * sizeof(float));                      // omega
  if (tc_eligible(a)) {
    n += align_up(R * 3 * a.d * 2);                      // ytc
    n += align_up(R * sizeof(float));                    // cy
    n += align_up(moments_tc_pscratch_bytes(a.BH(), a.T));  // pscr
    n += align_up(R * a.d * 2);                          // ksh
    n += align_up(BH * a.d * sizeof(float));             // kref
    n += align_up(BH * kKeyStatChunks * 2 * a.d * sizeof(float));  // kstat
    n += align_up((2 + kMaxRepairRows) * sizeof(int));   // rep, then the short-row count
  } else {
    n += align_up(short_list_ints(a) * sizeof(int));     // short-row count and list
  }
  return n;
}

void carve_workspace(const Args& a, void* base, Workspace* ws) {
  const size_t BH = (size_t)a.BH(), R = (size_t)a.rows();
  const size_t G = (size_t)gram_floats(a.d);
  char* p = static_cast<char*>(base);
  auto take = [&](size_t bytes) { char* r = p; p += align_up(bytes); return reinterpret_cast<float*>(r); };
  ws->kmean = take(BH * a.d * sizeof(float));
  ws->vmean = take(BH * a.dv * sizeof(float));
  ws->m = take(R * sizeof(float));
  ws->mom = take(R * G * sizeof(float));
  ws->mom_lo = a.dtype == LLA_F32 ? take(R * G * sizeof(float)) : nullptr;
  ws->y = take(R * a.d * sizeof(float));
  ws->kbar = take(R * a.d * sizeof(float));
  ws->omega = take(R * sizeof(float));
  const bool tc = tc_eligible(a);
  ws->ytc = tc ? reinterpret_cast<uint32_t*>(take(R * 3 * a.d * 2)) : nullptr;
  ws->cy = tc ? take(R * sizeof(float)) : nullptr;
  ws->pscr = tc ? take(moments_tc_pscratch_bytes(a.BH(), a.T)) : nullptr;
  ws->ksh = tc ? reinterpret_cast<__nv_bfloat16*>(take(R * a.d * 2)) : nullptr;
  ws->kref = tc ? take(BH * a.d * sizeof(float)) : nullptr;
  ws->kstat = tc ? take(BH * kKeyStatChunks * 2 * a.d * sizeof(float)) : nullptr;
  ws->rep = tc ? reinterpret_cast<int*>(take((2 + kMaxRepairRows) * sizeof(int))) : nullptr;
  if (tc) {
    ws->short_count = ws->rep + 1 + kMaxRepairRows;
    ws->short_rows = reinterpret_cast<int*>(ws->kstat);
  } else {
    ws->short_count = reinterpret_cast<int*>(take(short_list_ints(a) * sizeof(int)));
    ws->short_rows = ws->short_count + 1;
  }
  ws->status = nullptr;
  ws->path = choose_path(a);
  ws->form = a.form;
}

}  // namespace lla

using namespace lla;

extern "C" {

size_t lla_workspace_size(int B, int H, int T, int d, int dv, int dtype) {
  if (check_shape(B, H, T, d, dv, dtype) != LLA_OK) return 0;
  Args a = make_args(nullptr, nullptr, nullptr, nullptr, B, H, T, d, dv, 1.f, 1.f, dtype);
  return a.rows() == 0 ? 0 : workspace_bytes(a);
}

int lla_forward_ex(const void* q, const void* k, const void* v, void* out, int B, int H, int T,
                   int d, int dv, float h, float lambda, int dtype, const lla_options* opts,
                   void* workspace, size_t workspace_bytes_, void* stream) {
  Args a = make_args(q, k, v, out, B, H, T, d, dv, h, lambda, dtype);
  int st = apply_options(opts, true, &a);
  if (st != LLA_OK) return st;
  st = check_forward(a);
  if (st != LLA_OK || a.rows() == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) % 256) != 0 ||
        workspace_bytes_ < workspace_bytes(a))
      return LLA_ERR_INVALID_ARG;
    return run_forward(a, workspace, s);
  }
  if (ensure_pool() != cudaSuccess) return LLA_ERR_CUDA;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, workspace_bytes(a), s) != cudaSuccess) return LLA_ERR_CUDA;
  st = run_forward(a, ws, s);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == LLA_OK) st = LLA_ERR_CUDA;
  return st;
}

int lla_forward_ws(const void* q, const void* k, const void* v, void* out, int B, int H, int T,
                   int d, int dv, float h, float lambda, int dtype, void* workspace,
                   size_t workspace_bytes_, void* stream) {
  if (!workspace) {  // lla_forward_ex would allocate; this entry point never does
    const Args a = make_args(q, k, v, out, B, H, T, d, dv, h, lambda, dtype);
    const int st = check_forward(a);
    return (st != LLA_OK || a.rows() == 0) ? st : LLA_ERR_INVALID_ARG;
  }
  return lla_forward_ex(q, k, v, out, B, H, T, d, dv, h, lambda, dtype, nullptr, workspace,
                        workspace_bytes_, stream);
}

int lla_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int d,
                int dv, float h, float lambda, int dtype, void* stream) {
  return lla_forward_ex(q, k, v, out, B, H, T, d, dv, h, lambda, dtype, nullptr, nullptr, 0,
                        stream);
}

int lla_forward_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                     int B, int H, int T, int d, int dv, float h, float lambda, int dtype,
                     void* stream) {
  Args a = make_args(q_host, k_host, v_host, out_host, B, H, T, d, dv, h, lambda, dtype);
  int st = check_shape(B, H, T, d, dv, dtype);
  if (st != LLA_OK) return st;
  if (!is_finite_pos(h) || !is_finite_pos(lambda)) return LLA_ERR_INVALID_ARG;
  if (a.rows() == 0) return LLA_OK;
  if (!q_host || !k_host || !v_host || !out_host) return LLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = nullptr;
  if (device_status(&status) != cudaSuccess || ensure_pool() != cudaSuccess) return LLA_ERR_CUDA;
  const size_t eb = elem_bytes(dtype);
  const size_t nqk = (size_t)a.rows() * d * eb, nv = (size_t)a.rows() * dv * eb;
  const size_t off_k = align_up(nqk), off_v = off_k + align_up(nqk), off_o = off_v + align_up(nv);
  const size_t off_ws = off_o + align_up(nv);
  char* dev = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&dev), off_ws + workspace_bytes(a), s) != cudaSuccess)
    return LLA_ERR_CUDA;
  bool ok = cudaMemcpyAsync(dev, q_host, nqk, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(dev + off_k, k_host, nqk, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(dev + off_v, v_host, nv, cudaMemcpyHostToDevice, s) == cudaSuccess;
  if (ok) {
    Args ad = make_args(dev, dev + off_k, dev + off_v, dev + off_o, B, H, T, d, dv, h, lambda, dtype);
    st = run_forward(ad, dev + off_ws, s);
    ok = st == LLA_OK &&
         cudaMemcpyAsync(out_host, dev + off_o, nv, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  }
  cudaFreeAsync(dev, s);
  if (cudaStreamSynchronize(s) != cudaSuccess) return LLA_ERR_CUDA;
  if (!ok) return st != LLA_OK ? st : LLA_ERR_CUDA;
  return lla_stream_status(stream);
}

int lla_moments(const void* q, const void* k, const void* v, const int64_t* idx, int n, float* m,
                float* omega, float* sk, float* sv, float* Skk, float* Svk, int B, int H, int T,
                int d, int dv, float h, int dtype, void* stream) {
  int st = check_shape(B, H, T, d, dv, dtype);
  if (st != LLA_OK) return st;
  if (!is_finite_pos(h) || n < 0) return LLA_ERR_INVALID_ARG;
  if (n == 0) return LLA_OK;
  if (!q || !k || !v || !idx) return LLA_ERR_INVALID_ARG;
  int* status = nullptr;
  if (device_status(&status) != cudaSuccess) return LLA_ERR_CUDA;
  const Args a = make_args(q, k, v, nullptr, B, H, T, d, dv, h, 1.f, dtype);
  return launch_debug_moments(a, idx, n, m, omega, sk, sv, Skk, Svk, status,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LLA_OK
             : LLA_ERR_CUDA;
}

int lla_parallax_forward_ex(const void* q, const void* k, const void* v, const void* r, void* out,
                            int B, int H, int T, int d, int dv, float h, int dtype,
                            const lla_options* opts, void* stream) {
  Args a = make_args(q, k, v, out, B, H, T, d, dv, h, 1.f, dtype);
  int st = apply_options(opts, false, &a);
  if (st != LLA_OK) return st;
  st = check_forward(a);
  if (st != LLA_OK || a.rows() == 0) return st;
  if (!r || !aligned16(r)) return LLA_ERR_INVALID_ARG;
  int* status = nullptr;
  if (device_status(&status) != cudaSuccess) return LLA_ERR_CUDA;
  const int path = a.path_req == kPathCudaCore ? kPathCudaCore : kPathTensorCore;
  return launch_parallax(a, r, path, status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LLA_OK
             : LLA_ERR_CUDA;
}

int lla_parallax_forward(const void* q, const void* k, const void* v, const void* r, void* out,
                         int B, int H, int T, int d, int dv, float h, int dtype, void* stream) {
  return lla_parallax_forward_ex(q, k, v, r, out, B, H, T, d, dv, h, dtype, nullptr, stream);
}

namespace {
int run_decode(const DecodeArgs& a, const lla_options* opts, void* stream) {
  Args oa;
  const int ost = apply_options(opts, false, &oa);
  if (ost != LLA_OK) return ost;
  if (a.B < 0 || a.H < 0 || a.L < 0) return LLA_ERR_INVALID_ARG;
  if (a.dtype != LLA_F32 && a.dtype != LLA_BF16) return LLA_ERR_INVALID_ARG;
  if (!(a.d == 16 || a.d == 32 || a.d == 64) || !(a.dv == 16 || a.dv == 32 || a.dv == 64))
    return LLA_ERR_UNSUPPORTED;
  if (a.BH() * (long long)a.L >= (1LL << 31)) return LLA_ERR_UNSUPPORTED;
  if (!is_finite_pos(a.h) || (!a.r && !is_finite_pos(a.lam))) return LLA_ERR_INVALID_ARG;
  if (a.BH() == 0) return LLA_OK;
  if (a.L == 0) return LLA_ERR_INVALID_ARG;  // nothing to attend to
  if (!a.q || !a.k || !a.v || !a.out || !aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) ||
      !aligned16(a.out))
    return LLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = nullptr;
  if (device_status(&status) != cudaSuccess || ensure_pool() != cudaSuccess) return LLA_ERR_CUDA;
  DecodeArgs b = a;
  b.path = oa.path_req == kPathCudaCore ? kPathCudaCore : kPathTensorCore;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, decode_workspace_bytes(b), s) != cudaSuccess) return LLA_ERR_CUDA;
  int st = launch_decode(b, ws, status, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == LLA_OK) st = LLA_ERR_CUDA;
  return st;
}
}  // namespace

int lla_decode_ex(const void* q, const void* k, const void* v, void* out, int B, int H, int L,
                  int d, int dv, float h, float lambda, int dtype, const lla_options* opts,
                  void* stream) {
  DecodeArgs a{q, k, v, nullptr, out, B, H, L, d, dv, h, lambda, dtype};
  return run_decode(a, opts, stream);
}

int lla_decode(const void* q, const void* k, const void* v, void* out, int B, int H, int L, int d,
               int dv, float h, float lambda, int dtype, void* stream) {
  return lla_decode_ex(q, k, v, out, B, H, L, d, dv, h, lambda, dtype, nullptr, stream);
}

int lla_parallax_decode_ex(const void* q, const void* k, const void* v, const void* r, void* out,
                           int B, int H, int L, int d, int dv, float h, int dtype,
                           const lla_options* opts, void* stream) {
  if (B > 0 && H > 0 && (!r || !aligned16(r))) return LLA_ERR_INVALID_ARG;
  DecodeArgs a{q, k, v, r, out, B, H, L, d, dv, h, 1.f, dtype};
  if (!r) return LLA_ERR_INVALID_ARG;
  return run_decode(a, opts, stream);
}

int lla_parallax_decode(const void* q, const void* k, const void* v, const void* r, void* out,
                        int B, int H, int L, int d, int dv, float h, int dtype, void* stream) {
  return lla_parallax_decode_ex(q, k, v, r, out, B, H, L, d, dv, h, dtype, nullptr, stream);
}

int lla_parallax_backward_ex(const void* q, const void* k, const void* v, const void* r,
                             const void* dout, void* dq, void* dk, void* dv, void* dr, int B,
                             int H, int T, int d, int dv_, float h, int dtype,
                             const lla_options* opts, void* stream) {
  Args oa;
  int st = apply_options(opts, false, &oa);
  if (st != LLA_OK) return st;
  st = check_shape(B, H, T, d, dv_, dtype);
  if (st != LLA_OK) return st;
  if (!is_finite_pos(h)) return LLA_ERR_INVALID_ARG;
  if ((long long)B * H * T == 0) return LLA_OK;
  const void* ptrs[9] = {q, k, v, r, dout, dq, dk, dv, dr};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = nullptr;
  if (device_status(&status) != cudaSuccess || ensure_pool() != cudaSuccess) return LLA_ERR_CUDA;
  const ParallaxBwdArgs a{q, k, v, r, dout, dq, dk, dv, dr, B, H, T, d, dv_, h, dtype};
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, parallax_bwd_workspace_bytes(a), s) != cudaSuccess) return LLA_ERR_CUDA;
  const int path = oa.path_req == kPathCudaCore ? kPathCudaCore : kPathTensorCore;
  st = launch_parallax_bwd(a, ws, path, status, s) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == LLA_OK) st = LLA_ERR_CUDA;
  return st;
}

int lla_parallax_backward(const void* q, const void* k, const void* v, const void* r,
                          const void* dout, void* dq, void* dk, void* dv, void* dr, int B, int H,
                          int T, int d, int dv_, float h, int dtype, void* stream) {
  return lla_parallax_backward_ex(q, k, v, r, dout, dq, dk, dv, dr, B, H, T, d, dv_, h, dtype,
                                  nullptr, stream);
}

int lla_stream_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LLA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return LLA_ERR_CUDA;
  int* dummy;
  if (device_status(&dummy) != cudaSuccess) return LLA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status, sizeof(int)) != cudaSuccess) return LLA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return LLA_ERR_CUDA;
  if (word & kStatusBadIndex) return LLA_ERR_INVALID_ARG;
  if (word & kStatusTimeout) return LLA_ERR_TIMEOUT;
  if (word & kStatusNumerical) return LLA_ERR_NUMERICAL;
  return LLA_OK;
}

const char* lla_status_string(int status) {
  switch (status) {
    case LLA_OK: return "LLA_OK: success";
    case LLA_ERR_INVALID_ARG: return "LLA_ERR_INVALID_ARG: invalid argument";
    case LLA_ERR_UNSUPPORTED: return "LLA_ERR_UNSUPPORTED: unsupported size (d, dv in {16,32,64}; B*H*T < 2^31)";
    case LLA_ERR_CUDA: return "LLA_ERR_CUDA: a CUDA call or kernel launch failed";
    case LLA_ERR_NUMERICAL: return "LLA_ERR_NUMERICAL: non-positive pivot in a ridge solve";
    case LLA_ERR_TIMEOUT: return "LLA_ERR_TIMEOUT: a bounded device wait gave up";
  }
  return "unknown lla status";
}

int lla_version(void) {
  return LLA_VERSION_MAJOR * 10000 + LLA_VERSION_MINOR * 100 + LLA_VERSION_PATCH;
}

unsigned long long lla_launch_count(void) { return g_launches.load(); }

int lla_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return LLA_OK;
}

int lla_profile_collect(float* stage_ms, int max_stages, int* n_calls) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  float sum[LLA_NUM_STAGES] = {0.f};
  int st = LLA_OK;
  for (auto& r : recs) {
    if (cudaEventSynchronize(r.ev[LLA_NUM_STAGES]) != cudaSuccess) st = LLA_ERR_CUDA;
    for (int i = 0; i < LLA_NUM_STAGES && st == LLA_OK; ++i) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.ev[i], r.ev[i + 1]) != cudaSuccess) st = LLA_ERR_CUDA;
      sum[i] += ms;
    }
    for (auto& e : r.ev) cudaEventDestroy(e);
  }
  if (stage_ms)
    for (int i = 0; i < max_stages && i < LLA_NUM_STAGES; ++i) stage_ms[i] = sum[i];
  if (n_calls) *n_calls = (int)recs.size();
  return st;
}

}  // extern "C"
