// host.cu -- the C ABI of libringattn.so (declared in include/ringattn.h):
// argument validation, TMA tensor-map encoding, the device status word, and
// dispatch to the kernels.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <string>
#include <vector>

#include "../../include/ringattn.h"
#include "common.cuh"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- device state
__device__ unsigned int g_device_status;  // first bounded-wait time-out code, 0 if none
__device__ ra::CheckRec g_check_rec;      // bounds checks and event counts (checked build)
// SM clock records of timed kernels: block 0's clock64 and %globaltimer at its
// start and at its end (a ring of slots handed out by kt_begin).
constexpr int kClkSlots = 256;
__device__ unsigned long long g_clk_rec[kClkSlots][4];

constexpr int kMaxDevices = 64;
struct DevState {
  bool ready = false;
  int num_sms = 0;
  unsigned int* status = nullptr;  // device address of g_device_status
  ra::CheckRec* chk = nullptr;     // device address of g_check_rec
  unsigned long long* clk = nullptr;   // device address of g_clk_rec
};
DevState g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(RA_ERR_UNSUPPORTED, "libringattn is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<unsigned int*>(p);
    e = cudaGetSymbolAddress(&p, g_check_rec);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(check record)");
    d.chk = static_cast<ra::CheckRec*>(p);
    e = cudaGetSymbolAddress(&p, g_clk_rec);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(clock records)");
    d.clk = static_cast<unsigned long long*>(p);
    d.ready = true;
  }
  *out = &d;
  return RA_OK;
}

std::atomic<int> g_wait_test{0};   // one-shot: next bf16 forward withholds its first Q tile
std::atomic<int> g_fwd_kernel{RA_FWD_SINGLE};   // which bf16 forward kernel (ra_set_fwd_kernel)
std::atomic<uint64_t*> g_timing_buf{nullptr};
std::atomic<size_t> g_timing_n{0};

// ------------------------------------------------------- kernel timing (opt-in)
// While enabled, each ra_fwd / ra_bwd call records CUDA events on its stream
// around its kernels; ra_kernel_times() reads and releases them.
constexpr int kMaxTimedKernels = 16;
struct TimedCall {
  int call;           // ra_call_kind
  int nk;             // kernels timed (events = nk + 1)
  int dev;
  cudaEvent_t ev[kMaxTimedKernels + 1];
  int k0;             // kernel index of the first timed kernel
  int slot[kMaxTimedKernels];   // clock record slot of each kernel, or -1
};
std::atomic<bool> g_kt_on{false};
std::mutex g_kt_mu;
std::deque<TimedCall> g_kt_calls;
std::map<int, std::vector<cudaEvent_t>> g_kt_pool;   // idle events per device
int g_clk_next = 0, g_clk_used = 0;                  // clock slots (guarded by g_kt_mu)

// Events (and clock record slots for the kernels in `clock_mask`) for one call
// of `nk` kernels on the current device, or null when timing is off (or an
// event cannot be created: the call then runs untimed).
TimedCall* kt_begin(int call, int nk, int k0 = 0, unsigned clock_mask = 0) {
  if (!g_kt_on.load() || nk > kMaxTimedKernels) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_kt_mu);
  TimedCall tc{call, nk, dev, {}, k0, {}};
  for (int k = 0; k < nk; ++k) {
    tc.slot[k] = -1;
    if ((clock_mask >> k) & 1u && g_clk_used < kClkSlots) {
      tc.slot[k] = g_clk_next;
      g_clk_next = (g_clk_next + 1) % kClkSlots;
      ++g_clk_used;
    }
  }
  auto& pool = g_kt_pool[dev];
  for (int k = 0; k <= nk; ++k) {
    if (pool.empty()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) {
        for (int m = 0; m < k; ++m) pool.push_back(tc.ev[m]);
        return nullptr;
      }
      pool.push_back(e);
    }
    tc.ev[k] = pool.back();
    pool.pop_back();
  }
  g_kt_calls.push_back(tc);
  return &g_kt_calls.back();
}
cudaEvent_t* kt_events(TimedCall* tc) { return tc ? tc->ev : nullptr; }
// The clock record of kernel k of a timed call, or null.
unsigned long long* kt_clock(const DevState* d, const TimedCall* tc, int k) {
  return (tc && tc->slot[k] >= 0) ? d->clk + 4 * static_cast<size_t>(tc->slot[k]) : nullptr;
}

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 [BH, S, D] viewed as a 3-D tensor (D innermost); box = 64 cols x
// `box_rows` rows x 1 head, 128-byte swizzle (one box row = 128 bytes).
int make_map_bf16(CUtensorMap* m, const void* base, int64_t BH, int64_t S, int64_t D, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(S * D * 2)};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return RA_OK;
}

// ---------------------------------------------------------------- validation
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_sizes(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N) {
  if (B < 1 || H < 1 || S < 1 || D < 1 || N < 1)
    return fail(RA_ERR_ARG, "sizes must be >= 1 (B=%lld H=%lld S=%lld D=%lld N=%lld)", (long long)B,
                (long long)H, (long long)S, (long long)D, (long long)N);
  if (S % N != 0) return fail(RA_ERR_ARG, "S=%lld is not a multiple of N=%lld", (long long)S, (long long)N);
  if (B > INT_MAX / H) return fail(RA_ERR_ARG, "B*H exceeds 2^31-1");
  if (S > INT_MAX || D > INT_MAX) return fail(RA_ERR_ARG, "S or D exceeds 2^31-1");
  const int64_t bh = B * H;
  if (bh > INT64_MAX / S || bh * S > INT64_MAX / D / 4) return fail(RA_ERR_ARG, "B*H*S*D overflows");
  return RA_OK;
}
int check_enums(int causal, int layout, int dtype) {
  if (causal != 0 && causal != 1) return fail(RA_ERR_ARG, "causal must be 0 or 1 (got %d)", causal);
  if (layout != RA_CONTIGUOUS && layout != RA_STRIPED) return fail(RA_ERR_ARG, "bad layout %d", layout);
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_ARG, "bad dtype %d", dtype);
  return RA_OK;
}

// Validates and launches one forward over tensors of S rows cut into N blocks.
// `strict` and `use_timing` serve ra_fwd_step (one block pair as a 1-block call).
int fwd_impl(const void* Q, const void* K, const void* V, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
             int causal, int layout, int dtype, void* O, float* LSE, void* stream, int strict, bool use_timing,
             float* O_acc = nullptr, float* LSE_acc = nullptr) {
  const bool fold = O_acc != nullptr;
  if (!Q || !K || !V || (fold ? !LSE_acc : (!O || !LSE))) return fail(RA_ERR_ARG, "ra_fwd: null pointer");
  if (fold && (!aligned(O_acc, 16) || !aligned(LSE_acc, 4)))
    return fail(RA_ERR_ARG, "ra_fwd_step_fold: O_acc must be 16-byte and LSE_acc 4-byte aligned");
  int rc = check_sizes(B, H, S, D, N);
  if (rc != RA_OK) return rc;
  if ((rc = check_enums(causal, layout, dtype)) != RA_OK) return rc;
  if (!fold && !aligned(LSE, 4)) return fail(RA_ERR_ARG, "ra_fwd: LSE must be 4-byte aligned");
  if (fold && dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ra_fwd_step_fold: only the bf16 path folds");
  if (dtype == RA_BF16) {
    if (D != 128) return fail(RA_ERR_UNSUPPORTED, "ra_fwd: bf16 path needs D == 128 (got %lld)", (long long)D);
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || (!fold && !aligned(O, 16)))
      return fail(RA_ERR_ARG, "ra_fwd: bf16 tensors must be 16-byte aligned");
  } else {
    if (D % 4 != 0 || D > 128)
      return fail(RA_ERR_UNSUPPORTED, "ra_fwd: f32 path needs D %% 4 == 0 and D <= 128 (got %lld)", (long long)D);
    if (!aligned(Q, 4) || !aligned(K, 4) || !aligned(V, 4) || !aligned(O, 4))
      return fail(RA_ERR_ARG, "ra_fwd: f32 tensors must be 4-byte aligned");
  }
  uint64_t* timing = use_timing ? g_timing_buf.load() : nullptr;
  if (timing && g_timing_n.load() < static_cast<size_t>(N * N))
    return fail(RA_ERR_ARG, "timing buffer holds %zu entries, N*N = %lld needed", g_timing_n.load(),
                (long long)(N * N));
  DevState* d = nullptr;
  if ((rc = device_state(&d)) != RA_OK) return rc;

  ra::FwdArgs a;
  a.Q = Q; a.K = K; a.V = V; a.O = O; a.LSE = LSE;
  a.B = B; a.H = H; a.S = S; a.D = D; a.N = N;
  a.causal = causal;
  a.striped = layout == RA_STRIPED;
  a.strict = strict;
  a.withhold_first_q = dtype == RA_BF16 ? g_wait_test.exchange(0) : 0;
  a.status = d->status;
  a.timing = reinterpret_cast<unsigned long long*>(timing);
  a.stream = static_cast<cudaStream_t>(stream);
  a.num_sms = d->num_sms;
  // bf16: the SM-pair kernel (2-CTA clusters) when selected, else one CTA per SM.
  const bool pair = dtype == RA_BF16 && g_fwd_kernel.load() == RA_FWD_PAIR;
  if (pair) {
    const int slots = ra::fwd_pair_clusters();
    if (slots < 0) return fail(RA_ERR_CUDA, "ra_fwd: cluster occupancy query failed");
    if (slots == 0) return fail(RA_ERR_UNSUPPORTED, "ra_fwd: no 2-CTA cluster of the pair kernel fits on this device");
  }
  TimedCall* tc = kt_begin(RA_CALL_FWD, 1, pair ? 1 : 0, dtype == RA_BF16 ? 1u : 0u);
  a.ev = kt_events(tc);
  a.clk = kt_clock(d, tc, 0);
  a.chk = d->chk;
  a.O_acc = O_acc;
  a.LSE_acc = LSE_acc;
  cudaError_t e;
  if (dtype == RA_BF16) {
    CUtensorMap mq, mk, mv;
    if ((rc = make_map_bf16(&mq, Q, B * H, S, D, 128)) != RA_OK) return rc;
    if ((rc = make_map_bf16(&mk, K, B * H, S, D, pair ? 64 : 128)) != RA_OK) return rc;
    if ((rc = make_map_bf16(&mv, V, B * H, S, D, 128)) != RA_OK) return rc;
    e = pair ? ra::launch_fwd_bf16_pair(a, &mq, &mk, &mv) : ra::launch_fwd_bf16(a, &mq, &mk, &mv);
  } else {
    e = ra::launch_fwd_f32(a);
  }
  if (e != cudaSuccess) return cuda_fail(e, "ra_fwd launch");
  return RA_OK;
}

}  // namespace

namespace ra {
// Lets other translation units of the library report through ra_last_error().
void set_last_error(const std::string& msg) { g_last_error = msg; }

cudaError_t raise_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;   // (device, kernel) pairs already raised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({dev, func})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, func});
  return e;
}
}  // namespace ra

extern "C" {

const char* ra_last_error(void) { return g_last_error.c_str(); }
const char* ra_version(void) { return RA_CHECKS ? "ringattn 0.2 sm_103a checked" : "ringattn 0.2 sm_103a"; }

int ra_read_checks(ra_check_report* out, void* stream) {
  static_assert(sizeof(ra_check_report) == sizeof(ra::CheckRec), "report layout mirrors the device record");
  if (!out) return fail(RA_ERR_ARG, "ra_read_checks: null pointer");
  if (!RA_CHECKS) return fail(RA_ERR_UNSUPPORTED, "ra_read_checks: this is not the checked build");
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != RA_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  ra::CheckRec r;
  e = cudaMemcpyFromSymbol(&r, g_check_rec, sizeof(r));
  if (e != cudaSuccess) return cuda_fail(e, "read check record");
  const ra::CheckRec zero = {};
  e = cudaMemcpyToSymbol(g_check_rec, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear check record");
  memcpy(out, &r, sizeof(r));
  return RA_OK;
}

int ra_set_timing_buffer(uint64_t* dev_buf, size_t n) {
  if (dev_buf != nullptr && n < 1) return fail(RA_ERR_ARG, "timing buffer of size 0");
  g_timing_n.store(dev_buf ? n : 0);
  g_timing_buf.store(dev_buf);
  return RA_OK;
}

int ra_set_wait_test(int enable) {
  if (enable != 0 && enable != 1) return fail(RA_ERR_ARG, "ra_set_wait_test: enable must be 0 or 1");
  g_wait_test.store(enable);
  return RA_OK;
}

int ra_set_fwd_kernel(int kind) {
  if (kind != RA_FWD_SINGLE && kind != RA_FWD_PAIR)
    return fail(RA_ERR_ARG, "ra_set_fwd_kernel: kind must be RA_FWD_SINGLE or RA_FWD_PAIR (got %d)", kind);
  g_fwd_kernel.store(kind);
  return RA_OK;
}

int ra_set_kernel_timing(int enable) {
  if (enable != 0 && enable != 1) return fail(RA_ERR_ARG, "ra_set_kernel_timing: enable must be 0 or 1");
  std::lock_guard<std::mutex> lk(g_kt_mu);
  g_kt_on.store(enable == 1);
  if (!enable) {   // pending records are dropped; their events go back to the pool
    for (auto& c : g_kt_calls)
      for (int k = 0; k <= c.nk; ++k) g_kt_pool[c.dev].push_back(c.ev[k]);
    g_kt_calls.clear();
    g_clk_used = 0;
  }
  return RA_OK;
}

int ra_kernel_times(ra_kernel_time* out, int capacity, int* count) {
  if (!count || (capacity > 0 && !out) || capacity < 0) return fail(RA_ERR_ARG, "ra_kernel_times: bad arguments");
  std::lock_guard<std::mutex> lk(g_kt_mu);
  int n = 0, rc = RA_OK;
  for (auto& c : g_kt_calls) {
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != c.dev) cudaSetDevice(c.dev);
    cudaError_t e = cudaEventSynchronize(c.ev[c.nk]);
    for (int k = 0; k < c.nk; ++k) {
      float ms = -1.f, mhz = -1.f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, c.ev[k], c.ev[k + 1]);
      if (e == cudaSuccess && c.slot[k] >= 0) {
        unsigned long long r[4] = {0, 0, 0, 0};
        e = cudaMemcpyFromSymbol(r, g_clk_rec, sizeof(r), sizeof(r) * static_cast<size_t>(c.slot[k]));
        if (e == cudaSuccess && r[3] > r[1] && r[2] > r[0])
          mhz = static_cast<float>(static_cast<double>(r[2] - r[0]) / static_cast<double>(r[3] - r[1]) * 1e3);
      }
      if (n < capacity) out[n] = ra_kernel_time{c.call, c.k0 + k, ms, mhz};
      ++n;
    }
    if (prev != c.dev) cudaSetDevice(prev);
    if (e != cudaSuccess && rc == RA_OK) rc = cuda_fail(e, "ra_kernel_times");
    for (int k = 0; k <= c.nk; ++k) g_kt_pool[c.dev].push_back(c.ev[k]);
  }
  g_kt_calls.clear();
  g_clk_used = 0;
  *count = n;
  if (rc == RA_OK && n > capacity)
    rc = fail(RA_ERR_ARG, "ra_kernel_times: %d records, room for %d (the rest were dropped)", n, capacity);
  return rc;
}

int ra_check_device_status(void* stream) {
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
    return fail(RA_ERR_TIMEOUT, "a device-side wait timed out (code 0x%x); outputs are unspecified", v);
  }
  return RA_OK;
}


int ra_fwd(const void* Q, const void* K, const void* V, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
           int causal, int layout, int dtype, void* O, float* LSE, void* stream) {
  return fwd_impl(Q, K, V, B, H, S, D, N, causal, layout, dtype, O, LSE, stream, 0, true);
}

int ra_fwd_step(const void* Q_i, const void* K_j, const void* V_j, int64_t B, int64_t H, int64_t c, int64_t D,
                int64_t N, int64_t i, int64_t j, int causal, int layout, int dtype, void* O, float* LSE,
                void* stream) {
  if (N < 1 || i < 0 || i >= N || j < 0 || j >= N)
    return fail(RA_ERR_ARG, "ra_fwd_step: need 0 <= i, j < N (i=%lld j=%lld N=%lld)", (long long)i, (long long)j,
                (long long)N);
  int rc = check_enums(causal, layout, dtype);
  if (rc != RA_OK) return rc;
  const bool striped = layout == RA_STRIPED;
  if (causal && !striped && j > i) {
    // Every key of block j comes after every query of block i: the partial is
    // empty (O = 0, LSE = -inf), which ra_merge treats as "no keys".
    if (!Q_i || !K_j || !V_j || !O || !LSE) return fail(RA_ERR_ARG, "ra_fwd_step: null pointer");
    if ((rc = check_sizes(B, H, c, D, 1)) != RA_OK) return rc;
    if (!aligned(LSE, 4)) return fail(RA_ERR_ARG, "ra_fwd_step: LSE must be 4-byte aligned");
    DevState* d = nullptr;
    if ((rc = device_state(&d)) != RA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t esz = dtype == RA_BF16 ? 2 : 4;
    cudaError_t e = cudaMemsetAsync(O, 0, static_cast<size_t>(B * H * c * D) * esz, st);
    if (e == cudaSuccess) e = ra::launch_fill(LSE, B * H * c, -INFINITY, st, d->num_sms);
    if (e != cudaSuccess) return cuda_fail(e, "ra_fwd_step fill");
    return RA_OK;
  }
  // One block pair as a 1-block problem: a per-element mask only on
  // diagonal-type pairs; a striped pair with j > i also hides the key at the
  // query's own row (that key is a later token).
  const int pair_causal = (causal && (striped || j == i)) ? 1 : 0;
  const int strict = (causal && striped && j > i) ? 1 : 0;
  return fwd_impl(Q_i, K_j, V_j, B, H, c, D, 1, pair_causal, layout, dtype, O, LSE, stream, strict, false);
}

int ra_fwd_step_fold(const void* Q_i, const void* K_j, const void* V_j, int64_t B, int64_t H, int64_t c,
                     int64_t D, int64_t N, int64_t i, int64_t j, int causal, int layout, int dtype, float* O_acc,
                     float* LSE_acc, void* stream) {
  if (N < 1 || i < 0 || i >= N || j < 0 || j >= N)
    return fail(RA_ERR_ARG, "ra_fwd_step_fold: need 0 <= i, j < N (i=%lld j=%lld N=%lld)", (long long)i,
                (long long)j, (long long)N);
  int rc = check_enums(causal, layout, dtype);
  if (rc != RA_OK) return rc;
  if (!Q_i || !K_j || !V_j || !O_acc || !LSE_acc) return fail(RA_ERR_ARG, "ra_fwd_step_fold: null pointer");
  const bool striped = layout == RA_STRIPED;
  if (causal && !striped && j > i) {
    // Every key of block j comes after every query of block i: nothing to fold.
    if ((rc = check_sizes(B, H, c, D, 1)) != RA_OK) return rc;
    if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ra_fwd_step_fold: only the bf16 path folds");
    return RA_OK;
  }
  const int pair_causal = (causal && (striped || j == i)) ? 1 : 0;
  const int strict = (causal && striped && j > i) ? 1 : 0;
  return fwd_impl(Q_i, K_j, V_j, B, H, c, D, 1, pair_causal, layout, dtype, nullptr, nullptr, stream, strict, false,
                  O_acc, LSE_acc);
}

int ra_merge(void* O_a, float* lse_a, const void* O_b, const float* lse_b, int64_t rows, int64_t D, int dtype,
             void* stream) {
  if (rows < 0) return fail(RA_ERR_ARG, "ra_merge: rows < 0");
  if (D < 1 || D > 1024) return fail(RA_ERR_ARG, "ra_merge: D must be in 1..1024 (got %lld)", (long long)D);
  if (dtype != RA_F32 && dtype != RA_BF16 && dtype != RA_F32_BF16)
    return fail(RA_ERR_ARG, "ra_merge: bad dtype %d", dtype);
  if (rows == 0) return RA_OK;
  if (!O_a || !lse_a || !O_b || !lse_b) return fail(RA_ERR_ARG, "ra_merge: null pointer");
  const uintptr_t aal = dtype == RA_BF16 ? 2 : 4, bal = dtype == RA_F32 ? 4 : 2;
  if (!aligned(O_a, aal) || !aligned(O_b, bal) || !aligned(lse_a, 4) || !aligned(lse_b, 4))
    return fail(RA_ERR_ARG, "ra_merge: misaligned pointer");
  if (rows > INT64_MAX / D) return fail(RA_ERR_ARG, "ra_merge: rows*D overflows");
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != RA_OK) return rc;
  const int kind = dtype == RA_BF16 ? ra::MERGE_BF16 : dtype == RA_F32_BF16 ? ra::MERGE_F32_BF16 : ra::MERGE_F32;
  cudaError_t e = ra::launch_merge(O_a, lse_a, O_b, lse_b, rows, D, kind, static_cast<cudaStream_t>(stream),
                                   d->num_sms, d->chk);
  if (e != cudaSuccess) return cuda_fail(e, "ra_merge launch");
  return RA_OK;
}

}  // extern "C"

namespace {
// Workspace parts: lse2 and D_vec per padded query row.
struct WsLayout {
  uint64_t vec_bytes, total;
};
bool ws_layout(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N, WsLayout* w) {
  if (B < 1 || H < 1 || S < 1 || D < 1 || N < 1 || S % N != 0) return false;
  if (B > INT_MAX / H) return false;
  const int64_t bh = B * H;
  if (bh > INT64_MAX / S || bh * S > INT64_MAX / D / 8) return false;
  const int64_t c = S / N;
  const int64_t padded = N * ((c + 127) / 128) * 128;   // per head
  if (bh > INT64_MAX / padded / 8) return false;
  auto up = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
  w->vec_bytes = up(static_cast<uint64_t>(bh * padded) * 4);
  w->total = 2 * w->vec_bytes;
  return true;
}
}  // namespace

extern "C" {

size_t ra_bwd_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N) {
  WsLayout w;
  return ws_layout(B, H, S, D, N, &w) ? static_cast<size_t>(w.total) : 0;
}

}  // extern "C"

namespace {
// Validates and launches one backward over tensors of S rows cut into N
// blocks.  `strict` and `accumulate` serve ra_bwd_step.
int bwd_impl(const char* who, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             const void* dO, void* dQ, void* dK, void* dV, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
             int causal, int layout, int dtype, void* workspace, size_t ws_bytes, void* stream, int strict,
             int accumulate) {
  if (!Q || !K || !V || !O || !LSE || !dO || !dQ || !dK || !dV || !workspace)
    return fail(RA_ERR_ARG, "%s: null pointer", who);
  int rc = check_sizes(B, H, S, D, N);
  if (rc != RA_OK) return rc;
  if ((rc = check_enums(causal, layout, dtype)) != RA_OK) return rc;
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "%s: only the bf16 path is implemented", who);
  if (D != 128) return fail(RA_ERR_UNSUPPORTED, "%s: bf16 path needs D == 128 (got %lld)", who, (long long)D);
  const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return fail(RA_ERR_ARG, "%s: tensors must be 16-byte aligned", who);
  if (!aligned(LSE, 4)) return fail(RA_ERR_ARG, "%s: LSE must be 4-byte aligned", who);
  if (!aligned(workspace, 256)) return fail(RA_ERR_ARG, "%s: workspace must be 256-byte aligned", who);
  WsLayout wl;
  if (!ws_layout(B, H, S, D, N, &wl)) return fail(RA_ERR_ARG, "%s: workspace size overflows", who);
  if (ws_bytes < wl.total)
    return fail(RA_ERR_ARG, "%s: workspace of %zu bytes, %llu needed", who, ws_bytes,
                (unsigned long long)wl.total);
  DevState* d = nullptr;
  if ((rc = device_state(&d)) != RA_OK) return rc;

  ra::BwdArgs a;
  a.Q = Q; a.K = K; a.V = V; a.O = O; a.LSE = LSE; a.dO = dO;
  a.dQ = dQ; a.dK = dK; a.dV = dV;
  a.nlse2 = static_cast<float*>(workspace);
  a.ndvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + wl.vec_bytes);
  a.B = B; a.H = H; a.S = S; a.D = D; a.N = N;
  a.causal = causal;
  a.striped = layout == RA_STRIPED;
  a.strict = strict;
  a.accumulate = accumulate;
  a.status = d->status;
  a.stream = static_cast<cudaStream_t>(stream);
  a.num_sms = d->num_sms;
  a.chk = d->chk;
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = make_map_bf16(&mq, Q, B * H, S, D, 128)) != RA_OK) return rc;
  if ((rc = make_map_bf16(&mk, K, B * H, S, D, 128)) != RA_OK) return rc;
  if ((rc = make_map_bf16(&mv, V, B * H, S, D, 128)) != RA_OK) return rc;
  if ((rc = make_map_bf16(&mdo, dO, B * H, S, D, 128)) != RA_OK) return rc;
  TimedCall* tc = accumulate ? nullptr : kt_begin(RA_CALL_BWD, 3, 0, 0x6u);
  a.ev = kt_events(tc);
  a.clk_dkv = kt_clock(d, tc, 1);
  a.clk_dq = kt_clock(d, tc, 2);
  cudaError_t e = ra::launch_bwd_bf16(a, &mq, &mk, &mv, &mdo);
  if (e == cudaErrorNotSupported) return fail(RA_ERR_UNSUPPORTED, "%s: kernel not built", who);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return RA_OK;
}
}  // namespace

extern "C" {

int ra_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO, void* dQ,
           void* dK, void* dV, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N, int causal, int layout,
           int dtype, void* workspace, size_t ws_bytes, void* stream) {
  return bwd_impl("ra_bwd", Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, S, D, N, causal, layout, dtype, workspace,
                  ws_bytes, stream, 0, 0);
}

int ra_bwd_step(const void* Q_i, const void* K_j, const void* V_j, const void* O_i, const float* LSE_i,
                const void* dO_i, float* dQ_i, float* dK_j, float* dV_j, int64_t B, int64_t H, int64_t c, int64_t D,
                int64_t N, int64_t i, int64_t j, int causal, int layout, int dtype, void* workspace,
                size_t ws_bytes, void* stream) {
  if (N < 1 || i < 0 || i >= N || j < 0 || j >= N)
    return fail(RA_ERR_ARG, "ra_bwd_step: need 0 <= i, j < N (i=%lld j=%lld N=%lld)", (long long)i, (long long)j,
                (long long)N);
  int rc = check_enums(causal, layout, dtype);
  if (rc != RA_OK) return rc;
  const bool striped = layout == RA_STRIPED;
  if (causal && !striped && j > i) {
    // No query of block i sees a key of block j: nothing to add.
    if (!Q_i || !K_j || !V_j || !O_i || !LSE_i || !dO_i || !dQ_i || !dK_j || !dV_j || !workspace)
      return fail(RA_ERR_ARG, "ra_bwd_step: null pointer");
    return check_sizes(B, H, c, D, 1);
  }
  // The pair as a 1-block problem, masked as in ra_fwd_step.
  const int pair_causal = (causal && (striped || j == i)) ? 1 : 0;
  const int strict = (causal && striped && j > i) ? 1 : 0;
  return bwd_impl("ra_bwd_step", Q_i, K_j, V_j, O_i, LSE_i, dO_i, dQ_i, dK_j, dV_j, B, H, c, D, 1, pair_causal,
                  layout, dtype, workspace, ws_bytes, stream, strict, 1);
}

}  // extern "C"

namespace {
// Decode workspace: per-chunk partial outputs [items, D] and LSEs [items].
struct DecWs {
  ra::DecodePlan plan;
  uint64_t o_bytes, total;
};
bool dec_ws(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N, DecWs* w) {
  if (B < 1 || H < 1 || S < 1 || D < 1 || N < 1 || D > 4096) return false;
  if (B > INT_MAX / H) return false;
  const int64_t bh = B * H;
  if (bh > INT64_MAX / S || bh * S > INT64_MAX / D / 4) return false;
  if (!ra::decode_plan(bh, S, N, &w->plan)) return false;
  if (w->plan.items > INT64_MAX / D / 8) return false;
  auto up = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
  w->o_bytes = up(static_cast<uint64_t>(w->plan.items * D) * 4);
  w->total = w->o_bytes + up(static_cast<uint64_t>(w->plan.items) * 4);
  return true;
}
}  // namespace

extern "C" {

size_t ra_decode_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N) {
  DecWs w;
  return dec_ws(B, H, S, D, N, &w) ? static_cast<size_t>(w.total) : 0;
}

int ra_decode(const void* q, const void* K, const void* V, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
              int dtype, void* O, float* LSE, void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !K || !V || !O || !LSE || !workspace) return fail(RA_ERR_ARG, "ra_decode: null pointer");
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_ARG, "bad dtype %d", dtype);
  DecWs w;
  if (!dec_ws(B, H, S, D, N, &w))
    return fail(RA_ERR_ARG, "ra_decode: invalid sizes (B=%lld H=%lld S=%lld D=%lld N=%lld)", (long long)B,
                (long long)H, (long long)S, (long long)D, (long long)N);
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ra_decode: only the bf16 path is implemented");
  if (D != 128) return fail(RA_ERR_UNSUPPORTED, "ra_decode: bf16 path needs D == 128 (got %lld)", (long long)D);
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16))
    return fail(RA_ERR_ARG, "ra_decode: q, K and V must be 16-byte aligned");
  if (!aligned(O, 2) || !aligned(LSE, 4)) return fail(RA_ERR_ARG, "ra_decode: misaligned O or LSE");
  if (!aligned(workspace, 256)) return fail(RA_ERR_ARG, "ra_decode: workspace must be 256-byte aligned");
  if (ws_bytes < w.total)
    return fail(RA_ERR_ARG, "ra_decode: workspace of %zu bytes, %llu needed", ws_bytes,
                (unsigned long long)w.total);
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != RA_OK) return rc;
  ra::DecodeArgs a;
  a.q = q; a.K = K; a.V = V; a.O = O; a.LSE = LSE;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.o_bytes);
  a.B = B; a.H = H; a.S = S; a.N = N;
  a.plan = w.plan;
  a.status = d->status;
  a.stream = static_cast<cudaStream_t>(stream);
  a.num_sms = d->num_sms;
  a.ev = kt_events(kt_begin(RA_CALL_DECODE, 2));
  a.chk = d->chk;
  cudaError_t e = ra::launch_decode_bf16(a);
  if (e != cudaSuccess) return cuda_fail(e, "ra_decode launch");
  return RA_OK;
}

}  // extern "C"

namespace {
int64_t ffn_block_rows(int64_t T, int64_t block_rows) { return block_rows < T ? block_rows : T; }
bool ffn_sizes_ok(int64_t T, int64_t h, int64_t f, int64_t block_rows) {
  if (T < 1 || h < 256 || f < 128 || block_rows < 1) return false;
  if (h % 256 != 0 || f % 128 != 0) return false;
  if (h > INT_MAX || f > INT_MAX || T > INT_MAX) return false;
  return T <= INT64_MAX / h / 2 && ffn_block_rows(T, block_rows) <= INT64_MAX / f / 2;
}
}  // namespace

extern "C" {

// Workspace: the block's intermediate H (block_rows x f bf16), then one tile
// counter (int) per launch of the call (two per block).
size_t ra_ffn_workspace_bytes(int64_t T, int64_t h, int64_t f, int64_t block_rows) {
  if (!ffn_sizes_ok(T, h, f, block_rows)) return 0;
  const int64_t c = ffn_block_rows(T, block_rows), nblocks = (T + c - 1) / c;
  return static_cast<size_t>((c * f * 2 + 255) / 256 * 256 + (2 * nblocks * 4 + 255) / 256 * 256);
}

int ra_ffn(const void* X, const void* W1, const void* W3, const void* W2, void* Y, int64_t T, int64_t h, int64_t f,
           int64_t block_rows, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (!X || !W1 || !W3 || !W2 || !Y || !workspace) return fail(RA_ERR_ARG, "ra_ffn: null pointer");
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_ARG, "bad dtype %d", dtype);
  if (!ffn_sizes_ok(T, h, f, block_rows))
    return fail(RA_ERR_ARG, "ra_ffn: need T, block_rows >= 1, h a multiple of 256, f a multiple of 128 "
                "(T=%lld h=%lld f=%lld block_rows=%lld)", (long long)T, (long long)h, (long long)f,
                (long long)block_rows);
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "ra_ffn: only the bf16 path is implemented");
  const void* ptrs[] = {X, W1, W3, W2, Y, workspace};
  for (const void* q : ptrs)
    if (!aligned(q, 16)) return fail(RA_ERR_ARG, "ra_ffn: tensors and workspace must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(RA_ERR_ARG, "ra_ffn: workspace must be 256-byte aligned");
  const int64_t c = ffn_block_rows(T, block_rows);
  const size_t need = ra_ffn_workspace_bytes(T, h, f, block_rows);
  if (ws_bytes < need) return fail(RA_ERR_ARG, "ra_ffn: workspace of %zu bytes, %zu needed", ws_bytes, need);
  int* counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + (c * f * 2 + 255) / 256 * 256);
  DevState* d = nullptr;
  int rc = device_state(&d);
  if (rc != RA_OK) return rc;
  CUtensorMap m1, m3, m2, mh;
  if ((rc = make_map_bf16(&m1, W1, 1, f, h, 128)) != RA_OK) return rc;
  if ((rc = make_map_bf16(&m3, W3, 1, f, h, 128)) != RA_OK) return rc;
  if ((rc = make_map_bf16(&m2, W2, 1, h, f, 128)) != RA_OK) return rc;
  const int64_t nblocks = (T + c - 1) / c;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t me = cudaMemsetAsync(counters, 0, static_cast<size_t>(2 * nblocks) * sizeof(int), st);
  if (me != cudaSuccess) return cuda_fail(me, "ra_ffn: clearing the tile counters");
  cudaEvent_t* ev = kt_events(kt_begin(RA_CALL_FFN, static_cast<int>(2 * nblocks)));
  for (int64_t b = 0; b < nblocks; ++b) {
    const int64_t r0 = b * c, rows = (T - r0 < c) ? T - r0 : c;
    const char* xb = static_cast<const char*>(X) + r0 * h * 2;
    char* yb = static_cast<char*>(Y) + r0 * h * 2;
    CUtensorMap mx;
    if ((rc = make_map_bf16(&mx, xb, 1, rows, h, 128)) != RA_OK) return rc;
    if ((rc = make_map_bf16(&mh, workspace, 1, rows, f, 128)) != RA_OK) return rc;
    // The first launch keeps full stream order (X may come from the caller's
    // previous kernel); later ones overlap the previous launch's last wave.
    ra::FfnGemmArgs up{rows, f, h, 1, workspace, f, d->status, st, d->num_sms, b > 0 ? 1 : 0, counters + 2 * b, d->chk};
    ra::FfnGemmArgs down{rows, h, f, 0, yb, h, d->status, st, d->num_sms, 1, counters + 2 * b + 1, d->chk};
    if (ev) cudaEventRecord(ev[2 * b], st);
    cudaError_t e = ra::launch_ffn_gemm(up, &mx, &m1, &m3);
    if (e != cudaSuccess) return cuda_fail(e, "ra_ffn launch (up)");
    if (ev) cudaEventRecord(ev[2 * b + 1], st);
    e = ra::launch_ffn_gemm(down, &mh, &m2, &m2);
    if (e != cudaSuccess) return cuda_fail(e, "ra_ffn launch (down)");
  }
  if (ev) cudaEventRecord(ev[2 * nblocks], st);
  return RA_OK;
}

}  // extern "C"
