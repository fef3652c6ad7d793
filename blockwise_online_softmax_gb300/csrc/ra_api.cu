// Host side of the C ABI declared in include/ra.h: argument checks, TMA
// tensor-map encoding, the ring schedule, stream-ordered scratch, tracing
// and device status.  Host code only; the kernels live in the other units.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ra.h"
#include "ra_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Default wait bound for the kernels' mbarrier waits: 2^31 SM cycles,
// about one second at the maximum SM clock.
constexpr long long kWaitLimit = 1LL << 31;

// ----------------------------------------------------------------- tracing
struct TraceRec {
  int kind;
  cudaEvent_t start;
  cudaEvent_t stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;       // recorded since the last reset
std::vector<cudaEvent_t> g_ev_pool;  // spare events

cudaEvent_t take_event() {
  if (!g_ev_pool.empty()) {
    cudaEvent_t e = g_ev_pool.back();
    g_ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one kernel launch with an event pair on its stream while
// tracing is on.
struct TraceScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  bool on = false;
  TraceScope(int k, cudaStream_t s) : kind(k), st(s) {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (!g_trace_on) return;
    a = take_event();
    b = take_event();
    if (a && b && cudaEventRecord(a, st) == cudaSuccess) on = true;
  }
  void done(bool launched) {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (!on) {
      if (a) g_ev_pool.push_back(a);
      if (b) g_ev_pool.push_back(b);
      return;
    }
    if (launched && cudaEventRecord(b, st) == cudaSuccess) {
      g_trace.push_back({kind, a, b});
    } else {
      g_ev_pool.push_back(a);
      g_ev_pool.push_back(b);
    }
  }
};

// ----------------------------------------------------------------- scratch
// Scratch and staging buffers come from a memory pool the library owns on
// each device.  Its release threshold is unlimited, so memory freed at the
// end of a call stays mapped for the next one: a fresh multi-GB mapping
// costs milliseconds per call, which the default pool (threshold 0) would
// pay every time.  ra_release_cached_memory() trims the pools.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t scratch_pool(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_pool_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return e;
    }
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

// Stream-ordered allocation from the current device's pool; the buffer is
// returned with cudaFreeAsync like any other.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t st) {
  cudaMemPool_t pool = nullptr;
  cudaError_t e = scratch_pool(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(p, bytes, pool, st);
}

// ----------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return RA_OK;
}

// 3-D map over a token-major bf16 tensor [rows, heads, d]: dims (d, heads,
// rows).  The box is 64 elements (128 B, one swizzle span) x 1 head x
// box_rows rows, with 128-byte swizzle.  Rows past the end read as zero.
int encode_map(CUtensorMap* map, const void* base, long long rows, int heads, int d,
               int box_rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return RA_OK;
}

// 3-D map over an fp32 output [rows, heads, d] for tile stores: dims (d,
// heads, rows), box 32 elements (128 B, one swizzle span) x 1 head x 128
// rows, 128-byte swizzle.  Returns false, and leaves the error state alone,
// when the driver cannot map the tensor (the kernel then stores row by
// row).
bool encode_out_map(CUtensorMap* map, float* base, long long rows, int heads, int d) {
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(heads) * d * 4};
  const cuuint32_t box[3] = {32, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the decode queries [n_q, heads, d] whose box is tq tokens
// of g consecutive heads (one row tile of a KV head's query rows), 64
// columns wide: the box lands in shared memory as g * tq rows of 128 bytes,
// row qi * g + hl, with 128-byte swizzle.
int encode_q_group_map(CUtensorMap* map, const void* base, long long n_q, int heads, int g,
                       long long tq, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(tq)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled (query group) failed (CUresult %d)", (int)r);
  return RA_OK;
}

// ----------------------------------------------------------------- checks
int check_common(int d, int heads, int dtype) {
  if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID, "dtype %d is not RA_F32 or RA_BF16", dtype);
  if (d != 64 && d != 128) return fail(RA_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  if (heads < 1 || heads > 65535) return fail(RA_ERR_INVALID, "heads=%d out of range [1, 65535]", heads);
  return RA_OK;
}

int check_heads(int heads, int kv_heads) {
  if (kv_heads < 1) return fail(RA_ERR_INVALID, "kv_heads=%d must be >= 1", kv_heads);
  if (heads % kv_heads != 0) return fail(RA_ERR_INVALID, "heads=%d is not a multiple of kv_heads=%d", heads, kv_heads);
  return RA_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  int i = 0;
  for (const void* p : ps) {
    if (!p) return fail(RA_ERR_INVALID, "pointer argument %d is NULL", i);
    if (!aligned16(p)) return fail(RA_ERR_INVALID, "pointer argument %d is not 16-byte aligned", i);
    ++i;
  }
  return RA_OK;
}

// Run one block-update launch (mode 0 or 1), picking the kernel by dtype.
int run_update(ra::FwdArgs& a, int d, int dtype, cudaStream_t st) {
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  a.wait_limit = kWaitLimit;
  if (a.nwork == 0 || a.cq == 0 || a.ck == 0) return RA_OK;
  cudaError_t e;
  if (dtype == RA_BF16) {
    int rc = get_encoder();
    if (rc != RA_OK) return rc;
    CUtensorMap tq, tk, tv;
    if ((rc = encode_map(&tq, a.q, a.q_rows, a.heads, d)) != RA_OK) return rc;
    if ((rc = encode_map(&tk, a.k, a.kv_rows, a.kv_heads, d)) != RA_OK) return rc;
    if ((rc = encode_map(&tv, a.v, a.kv_rows, a.kv_heads, d)) != RA_OK) return rc;
    CUtensorMap to;
    std::memset(&to, 0, sizeof(to));
    a.o_tma = encode_out_map(&to, a.o, a.q_rows, a.heads, d) ? 1 : 0;
    TraceScope ts(RA_KERNEL_BLOCK_UPDATE_BF16, st);
    e = ra::launch_umma_update(a, d, tq, tk, tv, to, st);
    ts.done(e == cudaSuccess);
  } else {
    TraceScope ts(RA_KERNEL_BLOCK_UPDATE_F32, st);
    e = ra::launch_simt_update(a, d, st);
    ts.done(e == cudaSuccess);
  }
  if (e != cudaSuccess) return cuda_fail(e, "block-update launch");
  return RA_OK;
}

// ----------------------------------------------------------------- masks
// "All positions valid": larger than any sequence, small enough that
// position arithmetic on it cannot overflow.
constexpr long long kAllValid = 1LL << 60;

// Host copy of the mask arguments, checked.
struct MaskSpec {
  int layout = RA_LAYOUT_CONTIGUOUS;
  int causal = 0;
  long long window = 0;
  long long n_valid = kAllValid;
  const int* cu_seqlens = nullptr;
  int ndocs = 0;
};

int check_mask(int layout, int causal, long long window, long long n_valid,
               const int* cu_seqlens, int ndocs, MaskSpec* out) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED)
    return fail(RA_ERR_INVALID, "layout=%d is not a ra_layout value", layout);
  if (causal != 0 && causal != 1) return fail(RA_ERR_INVALID, "causal=%d is not 0 or 1", causal);
  if (window < 0) return fail(RA_ERR_INVALID, "window=%lld is negative", window);
  if (ndocs < 0) return fail(RA_ERR_INVALID, "ndocs=%d is negative", ndocs);
  if (ndocs > 0 && !cu_seqlens) return fail(RA_ERR_INVALID, "ndocs=%d with a NULL cu_seqlens", ndocs);
  if (ndocs > 0 && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(RA_ERR_INVALID, "cu_seqlens is not 4-byte aligned");
  out->layout = layout;
  out->causal = causal;
  out->window = window > kAllValid ? kAllValid : window;  // wider than any sequence
  out->n_valid = (n_valid < 0 || n_valid > kAllValid) ? kAllValid : n_valid;
  out->cu_seqlens = ndocs > 0 ? cu_seqlens : nullptr;
  out->ndocs = ndocs;
  return RA_OK;
}

void put_mask(ra::FwdArgs& a, const MaskSpec& mk) {
  a.layout = mk.layout;
  a.mask.causal = mk.causal;
  a.mask.window = mk.window;
  a.mask.n_valid = mk.n_valid;
  a.mask.cu_seqlens = mk.cu_seqlens;
  a.mask.ndocs = mk.ndocs;
}

// Positions of a block's rows below n_valid, as arithmetic progressions
// (start, count, step): one for contiguous and striped blocks, two for a
// zigzag block.
struct Prog {
  long long start, count, step;
};

int block_progs(const MaskSpec& mk, int P, long long c, long long blk, Prog out[2]) {
  int n = 0;
  if (mk.layout == RA_LAYOUT_ZIGZAG) {
    const long long h = c / 2;
    out[n++] = {blk * h, h, 1};
    out[n++] = {(2LL * P - 1 - blk) * h, h, 1};
  } else if (mk.layout == RA_LAYOUT_STRIPED) {
    out[n++] = {blk, c, P};
  } else {
    out[n++] = {blk * c, c, 1};
  }
  for (int i = 0; i < n; ++i) {
    Prog& g = out[i];
    if (g.start >= mk.n_valid) {
      g.count = 0;
    } else {
      const long long fit = (mk.n_valid - g.start + g.step - 1) / g.step;
      g.count = fit < g.count ? fit : g.count;
    }
  }
  return n;
}

long long floor_div(long long a, long long b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
long long ceil_div(long long a, long long b) { return -floor_div(-a, b); }

// Whether ring pair (i, j) may hold an allowed (query, key) pair under the
// causal and window rules and the valid length.  Documents are ignored, so
// the answer is exact or a safe "yes".
bool pair_may_see(const MaskSpec& mk, int P, long long c, int i, int j) {
  const long long big = 1LL << 61;
  // Allowed values of q - k.
  const long long A = mk.causal ? 0 : (mk.window > 0 ? -(mk.window - 1) : -big);
  const long long B = mk.window > 0 ? mk.window - 1 : big;
  Prog qp[2], kp[2];
  const int nq = block_progs(mk, P, c, i, qp), nk = block_progs(mk, P, c, j, kp);
  for (int x = 0; x < nq; ++x)
    for (int y = 0; y < nk; ++y) {
      const Prog& u = qp[x];
      const Prog& w = kp[y];
      if (u.count == 0 || w.count == 0) continue;
      // q - k = delta + step * m with m = a - b in [-(w.count-1), u.count-1].
      const long long delta = u.start - w.start;
      long long mlo = ceil_div(A - delta, u.step), mhi = floor_div(B - delta, u.step);
      if (mlo < -(w.count - 1)) mlo = -(w.count - 1);
      if (mhi > u.count - 1) mhi = u.count - 1;
      if (mlo <= mhi) return true;
    }
  return false;
}

// Ranks i that take part in ring step s.  The launch covers one range of
// ranks: the span of those whose pair may see a key; the CTAs of a rank in
// that span with nothing to do exit at once.
constexpr int kMaxScannedRanks = 4096;

void set_step_ranks(ra::FwdArgs& a, const MaskSpec& mk, int P, long long c, int s) {
  a.i0 = 0;
  a.nwork = P;
  if (P > kMaxScannedRanks) return;
  int first = -1, last = -1;
  for (int i = 0; i < P; ++i) {
    if (!pair_may_see(mk, P, c, i, ((i - s) % P + P) % P)) continue;
    if (first < 0) first = i;
    last = i;
  }
  a.i0 = first < 0 ? 0 : first;
  a.nwork = first < 0 ? 0 : last - first + 1;
}

int ring_args_check(long long N, int P, int s, int d, int heads, int kv_heads, int dtype,
                    int layout) {
  int rc;
  if ((rc = check_common(d, heads, dtype)) != RA_OK) return rc;
  if ((rc = check_heads(heads, kv_heads)) != RA_OK) return rc;
  if (N < 0) return fail(RA_ERR_INVALID, "N=%lld is negative", N);
  if (P < 1 || P > 65535) return fail(RA_ERR_INVALID, "P=%d out of range [1, 65535]", P);
  if (N % P != 0) return fail(RA_ERR_INVALID, "N=%lld is not a multiple of P=%d", N, P);
  if (layout == RA_LAYOUT_ZIGZAG && (N / P) % 2 != 0)
    return fail(RA_ERR_INVALID, "zigzag layout: the block length N/P=%lld is odd", N / P);
  if (s < 0 || s >= P) return fail(RA_ERR_INVALID, "ring step s=%d out of range [0, P)", s);
  if (N > (1LL << 31) - 256) return fail(RA_ERR_UNSUPPORTED, "N=%lld exceeds the 32-bit TMA row coordinate", N);
  return RA_OK;
}

int ring_step_impl(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                   long long N, int P, int s, const MaskSpec& mk, int d, int heads, int kv_heads,
                   int dtype, cudaStream_t st) {
  ra::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.m = m; a.l = l; a.o = o;
  a.cq = N / P;
  a.ck = N / P;
  a.q_rows = N;
  a.kv_rows = N;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.mode = 1;
  a.P = P;
  a.s = s;
  put_mask(a, mk);
  set_step_ranks(a, mk, P, N / P, s);
  return run_update(a, d, dtype, st);
}

// The bf16 ring in one launch: every rank's state stays on chip for all P
// steps, and the kernel writes out and lse itself (no scratch, no init or
// finalize launch).
constexpr int kFusedMaxSteps = 256;
constexpr int kHostGroups = 8;  // KV-head groups of the pipelined host-buffer ring (8 measured best)

// Query heads h0 .. h0 + nh - 1 only (nh = 0: all of them).
int ring_fused_impl(const void* q, const void* k, const void* v, float* out, float* lse,
                    long long N, int P, const MaskSpec& mk, int d, int heads, int kv_heads,
                    cudaStream_t st, int h0 = 0, int nh = 0) {
  ra::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = out; a.m = lse; a.l = nullptr;
  a.cq = N / P;
  a.ck = N / P;
  a.q_rows = N;
  a.kv_rows = N;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.mode = 1;
  a.P = P;
  a.s = 0;
  a.i0 = 0;
  a.nwork = P;
  a.h0 = h0;
  a.nh = nh;
  put_mask(a, mk);
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  a.wait_limit = kWaitLimit;
  if (a.cq == 0) return RA_OK;
  int rc = get_encoder();
  if (rc != RA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = encode_map(&tq, q, N, heads, d)) != RA_OK) return rc;
  if ((rc = encode_map(&tk, k, N, kv_heads, d)) != RA_OK) return rc;
  if ((rc = encode_map(&tv, v, N, kv_heads, d)) != RA_OK) return rc;
  CUtensorMap to;
  std::memset(&to, 0, sizeof(to));
  a.o_tma = encode_out_map(&to, out, N, heads, d) ? 1 : 0;
  TraceScope ts(RA_KERNEL_RING_FUSED_BF16, st);
  cudaError_t e = ra::launch_umma_ring(a, d, tq, tk, tv, to, st);
  ts.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "fused ring launch");
  return RA_OK;
}

// The fp32 ring in one launch (FFMA kernel, state on chip, finalized at
// the end).
int ring_fused_f32_impl(const void* q, const void* k, const void* v, float* out, float* lse,
                        long long N, int P, const MaskSpec& mk, int d, int heads, int kv_heads,
                        cudaStream_t st) {
  ra::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = out; a.m = lse; a.l = nullptr;
  a.cq = N / P;
  a.ck = N / P;
  a.q_rows = N;
  a.kv_rows = N;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.mode = 1;
  a.P = P;
  a.nwork = P;
  put_mask(a, mk);
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  a.wait_limit = kWaitLimit;
  if (a.cq == 0) return RA_OK;
  TraceScope ts(RA_KERNEL_RING_FUSED_F32, st);
  cudaError_t e = ra::launch_simt_ring(a, d, st);
  ts.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "fused fp32 ring launch");
  return RA_OK;
}

// Whether a ring forward runs as one fused launch (no state in HBM, no
// scratch): bf16 with P <= kFusedMaxSteps, and fp32.
bool ring_is_fused(int dtype, int P) {
  return dtype == RA_F32 || (dtype == RA_BF16 && P <= kFusedMaxSteps);
}

int ring_forward_impl(const void* q, const void* k, const void* v, float* out, float* lse,
                      long long N, int P, const MaskSpec& mk, int d, int heads, int kv_heads,
                      int dtype, cudaStream_t st, float* l_scratch) {
  if (dtype == RA_BF16 && P <= kFusedMaxSteps)
    return ring_fused_impl(q, k, v, out, lse, N, P, mk, d, heads, kv_heads, st);
  if (dtype == RA_F32) return ring_fused_f32_impl(q, k, v, out, lse, N, P, mk, d, heads, kv_heads, st);
  const long long rows = N;
  TraceScope t0(RA_KERNEL_STATE_INIT, st);
  cudaError_t e = ra::launch_state_init(lse, l_scratch, out, rows, heads, d, st);
  t0.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "state-init launch");
  for (int s = 0; s < P; ++s) {
    int rc = ring_step_impl(q, k, v, lse, l_scratch, out, N, P, s, mk, d, heads, kv_heads,
                            dtype, st);
    if (rc != RA_OK) return rc;
  }
  TraceScope t1(RA_KERNEL_FINALIZE, st);
  e = ra::launch_finalize(lse, l_scratch, out, out, lse, rows, heads, d, st);
  t1.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  return RA_OK;
}

MaskSpec plain_mask(int causal) {
  MaskSpec mk;
  mk.causal = causal ? 1 : 0;
  return mk;
}

// ra_ring_forward and ra_ring_forward_masked: one fused launch (bf16 with
// P <= 256, and fp32), else the step loop with the l scratch from the
// stream's pool allocator.
int ring_forward_alloc(const void* q, const void* k, const void* v, float* out, float* lse,
                       long long N, int P, const MaskSpec& mk, int d, int heads, int kv_heads,
                       int dtype, void* stream) {
  int rc;
  if ((rc = check_ptrs({q, k, v, out, lse})) != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ring_is_fused(dtype, P))
    return ring_forward_impl(q, k, v, out, lse, N, P, mk, d, heads, kv_heads, dtype, st, nullptr);
  float* l_scratch = nullptr;
  const size_t l_bytes = static_cast<size_t>(N) * heads * sizeof(float);
  cudaError_t e = scratch_alloc(reinterpret_cast<void**>(&l_scratch), l_bytes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_ALLOC, "pool allocation of %zu bytes for the l state failed: %s", l_bytes,
                cudaGetErrorString(e));
  }
  rc = ring_forward_impl(q, k, v, out, lse, N, P, mk, d, heads, kv_heads, dtype, st, l_scratch);
  e = cudaFreeAsync(l_scratch, st);
  if (rc == RA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  return rc;
}

// ----------------------------------------------------------------- fixed scratch
// Scratch for ra_ring_forward_noalloc: the l state ([N, heads] fp32) of the
// ring lives in this statically sized device array instead of memory taken
// from an allocator.  The array is part of the library's device image, so
// every GPU that loads libra.so holds its 16 MiB until the process exits.
constexpr long long kNoAllocMaxRowsHeads = 1LL << 22;  // N * heads <= 4,194,304
static __device__ __align__(256) float g_noalloc_l[kNoAllocMaxRowsHeads];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_l on the current device.  Host code only sees
// a host-side stand-in for the symbol, so the address must be looked up;
// this happens once per device, with that device current.
int noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_l);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress of the fixed scratch");
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return RA_OK;
}

// ----------------------------------------------------------------- backward
int ring_backward_impl(const void* q, const void* k, const void* v, const float* out,
                       const float* lse, const void* dout, float* dq, float* dk, float* dv,
                       long long N, int P, const MaskSpec& mk, int d, int heads, int kv_heads,
                       cudaStream_t st) {
  float* dvec = nullptr;
  cudaError_t e = scratch_alloc(reinterpret_cast<void**>(&dvec),
                                  static_cast<size_t>(N) * heads * sizeof(float), st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_ALLOC, "pool allocation of the D vector failed: %s", cudaGetErrorString(e));
  }
  int rc = RA_OK;
  {
    TraceScope t0(RA_KERNEL_BWD_PRE, st);
    e = ra::launch_bwd_pre(out, dout, dvec, N, heads, d, st);
    t0.done(e == cudaSuccess);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(dq, 0, static_cast<size_t>(N) * heads * d * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dk, 0, static_cast<size_t>(N) * kv_heads * d * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, static_cast<size_t>(N) * kv_heads * d * 4, st);
  if (e != cudaSuccess) rc = cuda_fail(e, "backward set-up");
  CUtensorMap tq, tk, tv, to;
  if (rc == RA_OK) rc = get_encoder();
  if (rc == RA_OK) rc = encode_map(&tq, q, N, heads, d);
  if (rc == RA_OK) rc = encode_map(&tk, k, N, kv_heads, d);
  if (rc == RA_OK) rc = encode_map(&tv, v, N, kv_heads, d);
  if (rc == RA_OK) rc = encode_map(&to, dout, N, heads, d);
  for (int s = 0; rc == RA_OK && s < P; ++s) {
    ra::BwdArgs b{};
    ra::FwdArgs& a = b.f;
    a.q = q; a.k = k; a.v = v;
    a.cq = N / P;
    a.ck = N / P;
    a.q_rows = N;
    a.kv_rows = N;
    a.heads = heads;
    a.kv_heads = kv_heads;
    a.mode = 1;
    a.P = P;
    a.s = s;
    a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    a.wait_limit = kWaitLimit;
    put_mask(a, mk);
    set_step_ranks(a, mk, P, N / P, s);
    if (a.nwork == 0 || a.cq == 0) continue;
    b.lse = lse;
    b.dvec = dvec;
    b.dq = dq;
    b.dk = dk;
    b.dv = dv;
    {
      TraceScope t1(RA_KERNEL_BWD_DQ, st);
      e = ra::launch_bwd_dq(b, d, tq, tk, tv, to, st);
      t1.done(e == cudaSuccess);
    }
    if (e == cudaSuccess) {
      TraceScope t2(RA_KERNEL_BWD_DKDV, st);
      e = ra::launch_bwd_dkdv(b, d, tq, tk, tv, to, st);
      t2.done(e == cudaSuccess);
    }
    if (e != cudaSuccess) rc = cuda_fail(e, "backward launch");
  }
  e = cudaFreeAsync(dvec, st);
  if (rc == RA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  return rc;
}

// ----------------------------------------------------------------- decode
// A decode row tile holds 128 query rows: floor(128 / g) tokens of the g
// heads that share a KV head.
constexpr int kDecodeMaxRows = 128;

int decode_args_check(const void* q, const void* k, const void* v, long long n_q, long long n_kv,
                      int d, int heads, int kv_heads, long long window, int dtype) {
  int rc;
  if ((rc = check_common(d, heads, dtype)) != RA_OK) return rc;
  if ((rc = check_heads(heads, kv_heads)) != RA_OK) return rc;
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "the decode path takes bf16 q, k, v");
  if (n_q < 0 || n_kv < 0) return fail(RA_ERR_INVALID, "n_q=%lld or n_kv=%lld is negative", n_q, n_kv);
  if (n_kv > (1LL << 31) - 256) return fail(RA_ERR_UNSUPPORTED, "n_kv=%lld exceeds the 32-bit TMA row coordinate", n_kv);
  if (window < 0) return fail(RA_ERR_INVALID, "window=%lld is negative", window);
  if (heads / kv_heads > kDecodeMaxRows)
    return fail(RA_ERR_UNSUPPORTED,
                "heads / kv_heads = %d query heads per KV head exceeds %d (one token's rows "
                "must fit a %d-row tile)",
                heads / kv_heads, kDecodeMaxRows, kDecodeMaxRows);
  if (n_q > (1LL << 24))
    return fail(RA_ERR_UNSUPPORTED, "n_q=%lld query tokens exceeds 2^24; use the ring forward",
                n_q);
  // One reduction CTA per (query row, head): the count must fit a grid.
  if (n_q * heads > 0x7FFFFFFFLL)
    return fail(RA_ERR_UNSUPPORTED, "n_q * heads = %lld rows exceeds 2^31 - 1", n_q * heads);
  (void)q; (void)k; (void)v;
  return RA_OK;
}

// The split-K chunk kernel over nshard shards of shard_len keys, then
// either the fold of each shard's chunk states into that shard's state
// (m, l, o: [nshard][rows]) or, with out and lse given, the reduction over
// every shard and the finalize straight into out and lse.
int decode_run(const void* q, const void* k, const void* v, float* m, float* l, float* o,
               long long n_q, long long n_kv, long long shard_len, int nshard, long long q_off,
               long long kv_off, int causal, long long window, int d, int heads, int kv_heads,
               cudaStream_t st, float* out = nullptr, float* lse = nullptr) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Row tiles: tq tokens of the g heads of a KV head, g * tq <= 128 rows.
  const int g = heads / kv_heads;
  long long tq = kDecodeMaxRows / g;
  if (tq > n_q) tq = n_q;
  const long long ntile = (n_q + tq - 1) / tq;
  // One CTA per SM at a time; about six waves; chunks of whole 128-key
  // tiles, at least one.  Each CTA pays a pipeline fill, so fewer, longer
  // chunks win up to the point where the last partial wave leaves SMs
  // idle: on 1M keys in 64 shards x 8 KV heads (512 units on 152 SMs), six
  // waves (two chunks per shard) measured 10% faster than three (one chunk,
  // 3.4 waves) and than ten or seventeen.
  const long long waves = 6, gran = 128;
  const long long units = static_cast<long long>(kv_heads) * nshard * ntile;
  long long want = (waves * sms + units - 1) / units;
  if (want < 1) want = 1;
  long long chunk = (shard_len + want - 1) / want;
  chunk = ((chunk + gran - 1) / gran) * gran;
  if (chunk < 128) chunk = 128;
  const long long nsplit = (shard_len + chunk - 1) / chunk;
  const long long rows = n_q * heads;  // state rows of one shard
  const size_t n_part = static_cast<size_t>(nshard) * nsplit * rows;
  float* part = nullptr;
  cudaError_t e = scratch_alloc(reinterpret_cast<void**>(&part),
                                  n_part * (2 + static_cast<size_t>(d)) * sizeof(float), st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_ALLOC, "pool allocation of the decode partial states failed: %s",
                cudaGetErrorString(e));
  }
  int rc = get_encoder();
  CUtensorMap tk, tv, tmq;
  if (rc == RA_OK) rc = encode_map(&tk, k, n_kv, kv_heads, d);
  if (rc == RA_OK) rc = encode_map(&tv, v, n_kv, kv_heads, d);
  if (rc == RA_OK) rc = encode_q_group_map(&tmq, q, n_q, heads, g, tq, d);
  if (rc == RA_OK) {
    ra::DecArgs a{};
    a.q = q;
    a.po = part;
    a.pm = part + n_part * d;
    a.pl = a.pm + n_part;
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.shard_len = shard_len;
    a.chunk = chunk;
    a.q_off = q_off;
    a.kv_off = kv_off;
    a.heads = heads;
    a.kv_heads = kv_heads;
    a.nsplit = static_cast<int>(nsplit);
    a.tq = tq;
    a.ntile = static_cast<int>(ntile);
    a.nshard = nshard;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    a.wait_limit = kWaitLimit;
    a.mask.causal = causal ? 1 : 0;
    a.mask.window = window > kAllValid ? kAllValid : window;
    a.mask.n_valid = kAllValid;
    TraceScope t0(RA_KERNEL_DECODE_SPLIT, st);
    e = ra::launch_decode_tc(a, d, tmq, tk, tv, st);
    t0.done(e == cudaSuccess);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "decode split launch");
    } else if (out) {
      TraceScope t1(RA_KERNEL_DECODE_COMBINE, st);
      e = ra::launch_decode_reduce(out, lse, a.pm, a.pl, a.po, rows, nshard * a.nsplit, d, st);
      t1.done(e == cudaSuccess);
      if (e != cudaSuccess) rc = cuda_fail(e, "decode reduce launch");
    } else {
      TraceScope t1(RA_KERNEL_DECODE_COMBINE, st);
      e = ra::launch_decode_combine(m, l, o, a.pm, a.pl, a.po, rows, a.nsplit, nshard, d, st);
      t1.done(e == cudaSuccess);
      if (e != cudaSuccess) rc = cuda_fail(e, "decode combine launch");
    }
  }
  e = cudaFreeAsync(part, st);
  if (rc == RA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  return rc;
}

}  // namespace

extern "C" {

int ra_abi_version(void) { return 3; }

const char* ra_status_string(int status) {
  switch (status) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID: return "RA_ERR_INVALID";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    case RA_ERR_ALLOC: return "RA_ERR_ALLOC";
    default: return "RA_ERR_UNKNOWN";
  }
}

const char* ra_last_error(void) { return g_last_error.c_str(); }

int ra_state_init(float* m, float* l, float* o, long long c, int d, int heads, void* stream) {
  int rc;
  if ((rc = check_common(d, heads, RA_F32)) != RA_OK) return rc;
  if (c < 0) return fail(RA_ERR_INVALID, "c=%lld is negative", c);
  if (c == 0) return RA_OK;
  if ((rc = check_ptrs({m, l, o})) != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TraceScope ts(RA_KERNEL_STATE_INIT, st);
  cudaError_t e = ra::launch_state_init(m, l, o, c, heads, d, st);
  ts.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "state-init launch");
  return RA_OK;
}

int ra_block_update_masked(const void* q, const void* k, const void* v, float* m, float* l,
                           float* o, long long c_q, long long c_kv, int d, int heads,
                           int kv_heads, int layout, int P, int q_block, int kv_block,
                           long long q_off, long long kv_off, int causal, long long window,
                           long long n_valid, const int* cu_seqlens, int ndocs, int dtype,
                           void* stream) {
  int rc;
  if ((rc = check_common(d, heads, dtype)) != RA_OK) return rc;
  if ((rc = check_heads(heads, kv_heads)) != RA_OK) return rc;
  MaskSpec mk;
  if ((rc = check_mask(layout, causal, window, n_valid, cu_seqlens, ndocs, &mk)) != RA_OK) return rc;
  if (c_q < 0 || c_kv < 0) return fail(RA_ERR_INVALID, "c_q=%lld or c_kv=%lld is negative", c_q, c_kv);
  if (c_q > (1LL << 31) - 256 || c_kv > (1LL << 31) - 256)
    return fail(RA_ERR_UNSUPPORTED, "a block length exceeds the 32-bit TMA row coordinate");
  if (layout != RA_LAYOUT_CONTIGUOUS) {
    if (P < 1 || P > 65535) return fail(RA_ERR_INVALID, "P=%d out of range [1, 65535]", P);
    if (q_block < 0 || q_block >= P || kv_block < 0 || kv_block >= P)
      return fail(RA_ERR_INVALID, "q_block=%d / kv_block=%d out of range [0, P)", q_block, kv_block);
  }
  if (layout == RA_LAYOUT_ZIGZAG && (c_q != c_kv || c_q % 2 != 0))
    return fail(RA_ERR_INVALID, "zigzag layout needs c_q == c_kv and an even block length");
  if (c_q == 0 || c_kv == 0) return RA_OK;
  if ((rc = check_ptrs({q, k, v, m, l, o})) != RA_OK) return rc;
  ra::FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.m = m; a.l = l; a.o = o;
  a.cq = c_q;
  a.ck = c_kv;
  a.q_rows = c_q;
  a.kv_rows = c_kv;
  a.q_off = q_off;
  a.kv_off = kv_off;
  a.q_blk = layout == RA_LAYOUT_CONTIGUOUS ? 0 : q_block;
  a.kv_blk = layout == RA_LAYOUT_CONTIGUOUS ? 0 : kv_block;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.mode = 0;
  a.P = layout == RA_LAYOUT_CONTIGUOUS ? 1 : P;
  a.s = 0;
  a.nwork = 1;
  put_mask(a, mk);
  return run_update(a, d, dtype, static_cast<cudaStream_t>(stream));
}

int ra_block_update(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                    long long c, int d, int heads, int kv_heads, long long q_off,
                    long long kv_off, int causal, int dtype, void* stream) {
  return ra_block_update_masked(q, k, v, m, l, o, c, c, d, heads, kv_heads, RA_LAYOUT_CONTIGUOUS,
                                1, 0, 0, q_off, kv_off, causal ? 1 : 0, 0, -1, nullptr, 0, dtype,
                                stream);
}

int ra_merge(float* m_a, float* l_a, float* o_a, const float* m_b, const float* l_b,
             const float* o_b, long long c, int d, int heads, void* stream) {
  int rc;
  if ((rc = check_common(d, heads, RA_F32)) != RA_OK) return rc;
  if (c < 0) return fail(RA_ERR_INVALID, "c=%lld is negative", c);
  if (c == 0) return RA_OK;
  if ((rc = check_ptrs({m_a, l_a, o_a, m_b, l_b, o_b})) != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TraceScope ts(RA_KERNEL_MERGE, st);
  cudaError_t e = ra::launch_merge(m_a, l_a, o_a, m_b, l_b, o_b, c, heads, d, st);
  ts.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return RA_OK;
}

int ra_finalize(const float* m, const float* l, const float* o, float* out, float* lse,
                long long c, int d, int heads, void* stream) {
  int rc;
  if ((rc = check_common(d, heads, RA_F32)) != RA_OK) return rc;
  if (c < 0) return fail(RA_ERR_INVALID, "c=%lld is negative", c);
  if (c == 0) return RA_OK;
  if ((rc = check_ptrs({m, l, o, out, lse})) != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TraceScope ts(RA_KERNEL_FINALIZE, st);
  cudaError_t e = ra::launch_finalize(m, l, o, out, lse, c, heads, d, st);
  ts.done(e == cudaSuccess);
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  return RA_OK;
}

int ra_ring_step_masked(const void* q, const void* k, const void* v, float* m, float* l,
                        float* o, long long N, int P, int s, int layout, int causal,
                        long long window, long long n_valid, const int* cu_seqlens, int ndocs,
                        int d, int heads, int kv_heads, int dtype, void* stream) {
  int rc = ring_args_check(N, P, s, d, heads, kv_heads, dtype, layout);
  if (rc != RA_OK) return rc;
  MaskSpec mk;
  if ((rc = check_mask(layout, causal, window, n_valid, cu_seqlens, ndocs, &mk)) != RA_OK) return rc;
  if (N == 0) return RA_OK;
  if ((rc = check_ptrs({q, k, v, m, l, o})) != RA_OK) return rc;
  return ring_step_impl(q, k, v, m, l, o, N, P, s, mk, d, heads, kv_heads, dtype,
                        static_cast<cudaStream_t>(stream));
}

int ra_ring_step(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                 long long N, int P, int s, int causal, int d, int heads, int kv_heads,
                 int dtype, void* stream) {
  return ra_ring_step_masked(q, k, v, m, l, o, N, P, s, RA_LAYOUT_CONTIGUOUS, causal ? 1 : 0, 0,
                             -1, nullptr, 0, d, heads, kv_heads, dtype, stream);
}

int ra_ring_forward_masked(const void* q, const void* k, const void* v, float* out, float* lse,
                           long long N, int P, int layout, int causal, long long window,
                           long long n_valid, const int* cu_seqlens, int ndocs, int d,
                           int heads, int kv_heads, int dtype, void* stream) {
  int rc = ring_args_check(N, P, 0, d, heads, kv_heads, dtype, layout);
  if (rc != RA_OK) return rc;
  MaskSpec mk;
  if ((rc = check_mask(layout, causal, window, n_valid, cu_seqlens, ndocs, &mk)) != RA_OK) return rc;
  if (N == 0) return RA_OK;
  return ring_forward_alloc(q, k, v, out, lse, N, P, mk, d, heads, kv_heads, dtype, stream);
}

int ra_ring_forward(const void* q, const void* k, const void* v, float* out, float* lse,
                    long long N, int P, int causal, int d, int heads, int kv_heads, int dtype,
                    void* stream) {
  int rc = ring_args_check(N, P, 0, d, heads, kv_heads, dtype, RA_LAYOUT_CONTIGUOUS);
  if (rc != RA_OK) return rc;
  if (N == 0) return RA_OK;
  return ring_forward_alloc(q, k, v, out, lse, N, P, plain_mask(causal), d, heads, kv_heads,
                            dtype, stream);
}

// The bf16 host-buffer ring in pipelined groups of KV heads (heads never
// interact): the inputs of group G + 1 copy in and the outputs of group
// G - 1 copy out while group G runs.  Copies are pitched (a group is a
// column range of every token row) on two helper streams; the kernels run
// on the caller's stream and a third helper stream in turn; events order
// them all.  Device buffers are allocated on the caller's stream and freed
// there once every copy and kernel is done.
static int ring_forward_host_pipelined(const void* q_host, const void* k_host,
                                       const void* v_host, float* out_host, float* lse_host,
                                       long long N, int P, int causal, int d, int heads,
                                       int kv_heads, cudaStream_t st) {
  const int g = heads / kv_heads;
  int ng = kv_heads < kHostGroups ? kv_heads : kHostGroups;
  while (kv_heads % ng) --ng;
  const int gkv = kv_heads / ng, gq = gkv * g;
  const size_t q_bytes = static_cast<size_t>(N) * heads * d * 2;
  const size_t kv_bytes = static_cast<size_t>(N) * kv_heads * d * 2;
  const size_t out_bytes = static_cast<size_t>(N) * heads * d * sizeof(float);
  const size_t rh_bytes = static_cast<size_t>(N) * heads * sizeof(float);
  void *dq = nullptr, *dk = nullptr, *dv = nullptr;
  float *dout = nullptr, *dlse = nullptr;
  cudaStream_t s_in = nullptr, s_out = nullptr, s_c1 = nullptr;
  cudaEvent_t ev_alloc = nullptr, ev_end = nullptr, ev_inall = nullptr, ev_c1 = nullptr;
  cudaEvent_t ev_in[kHostGroups] = {}, ev_run[kHostGroups] = {};
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
    return e == cudaSuccess;
  };
  auto alloc = [&](void** p, size_t n) { ok(scratch_alloc(p, n, st)); };
  alloc(&dq, q_bytes);
  alloc(&dk, kv_bytes);
  alloc(&dv, kv_bytes);
  alloc(reinterpret_cast<void**>(&dout), out_bytes);
  alloc(reinterpret_cast<void**>(&dlse), rh_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    int rc = fail(RA_ERR_ALLOC, "pool allocation of device staging failed: %s",
                  cudaGetErrorString(e));
    void* bufs[5] = {dq, dk, dv, dout, dlse};
    for (void* p : bufs)
      if (p) cudaFreeAsync(p, st);
    return rc;
  }
  ok(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking));
  ok(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking));
  ok(cudaStreamCreateWithFlags(&s_c1, cudaStreamNonBlocking));
  ok(cudaEventCreateWithFlags(&ev_alloc, cudaEventDisableTiming));
  ok(cudaEventCreateWithFlags(&ev_c1, cudaEventDisableTiming));
  ok(cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming));
  ok(cudaEventCreateWithFlags(&ev_inall, cudaEventDisableTiming));
  for (int G = 0; G < ng; ++G) {
    ok(cudaEventCreateWithFlags(&ev_in[G], cudaEventDisableTiming));
    ok(cudaEventCreateWithFlags(&ev_run[G], cudaEventDisableTiming));
  }
  int rc = RA_OK;
  if (e == cudaSuccess) {
    ok(cudaEventRecord(ev_alloc, st));
    ok(cudaStreamWaitEvent(s_in, ev_alloc, 0));
    ok(cudaStreamWaitEvent(s_c1, ev_alloc, 0));
    const size_t qrow = static_cast<size_t>(heads) * d * 2, kvrow = static_cast<size_t>(kv_heads) * d * 2;
    for (int G = 0; G < ng && e == cudaSuccess; ++G) {
      const size_t qo = static_cast<size_t>(G) * gq * d * 2, ko = static_cast<size_t>(G) * gkv * d * 2;
      const size_t qw = static_cast<size_t>(gq) * d * 2, kw = static_cast<size_t>(gkv) * d * 2;
      ok(cudaMemcpy2DAsync(static_cast<char*>(dq) + qo, qrow, static_cast<const char*>(q_host) + qo,
                           qrow, qw, N, cudaMemcpyHostToDevice, s_in));
      ok(cudaMemcpy2DAsync(static_cast<char*>(dk) + ko, kvrow, static_cast<const char*>(k_host) + ko,
                           kvrow, kw, N, cudaMemcpyHostToDevice, s_in));
      ok(cudaMemcpy2DAsync(static_cast<char*>(dv) + ko, kvrow, static_cast<const char*>(v_host) + ko,
                           kvrow, kw, N, cudaMemcpyHostToDevice, s_in));
      ok(cudaEventRecord(ev_in[G], s_in));
    }
    cudaEventRecord(ev_inall, s_in);  // after every copy that was enqueued
    // Groups alternate between two compute streams, so the CTAs of group
    // G+1 fill the SMs that group G's last wave leaves idle.
    cudaStream_t cs[2] = {st, s_c1};
    for (int G = 0; G < ng && e == cudaSuccess && rc == RA_OK; ++G) {
      cudaStream_t c = cs[G & 1];
      ok(cudaStreamWaitEvent(c, ev_in[G], 0));
      if (e != cudaSuccess) break;
      rc = ring_fused_impl(dq, dk, dv, dout, dlse, N, P, plain_mask(causal), d, heads, kv_heads,
                           c, G * gq, gq);
      ok(cudaEventRecord(ev_run[G], c));
      ok(cudaStreamWaitEvent(s_out, ev_run[G], 0));
      const size_t orow = static_cast<size_t>(heads) * d * 4, oo = static_cast<size_t>(G) * gq * d * 4;
      ok(cudaMemcpy2DAsync(reinterpret_cast<char*>(out_host) + oo, orow,
                           reinterpret_cast<const char*>(dout) + oo, orow,
                           static_cast<size_t>(gq) * d * 4, N, cudaMemcpyDeviceToHost, s_out));
    }
    // LSE is small: one contiguous copy after the last group.
    if (e == cudaSuccess && rc == RA_OK)
      ok(cudaMemcpyAsync(lse_host, dlse, rh_bytes, cudaMemcpyDeviceToHost, s_out));
    // The caller's stream, which frees the buffers, waits for every copy.
    cudaEventRecord(ev_end, s_out);
    cudaEventRecord(ev_c1, s_c1);
    cudaStreamWaitEvent(st, ev_end, 0);
    cudaStreamWaitEvent(st, ev_inall, 0);
    cudaStreamWaitEvent(st, ev_c1, 0);
  }
  void* bufs[5] = {dq, dk, dv, dout, dlse};
  for (void* p : bufs)
    if (p) cudaFreeAsync(p, st);
  if (s_in) cudaStreamDestroy(s_in);
  if (s_out) cudaStreamDestroy(s_out);
  if (s_c1) cudaStreamDestroy(s_c1);
  if (ev_alloc) cudaEventDestroy(ev_alloc);
  if (ev_c1) cudaEventDestroy(ev_c1);
  if (ev_end) cudaEventDestroy(ev_end);
  if (ev_inall) cudaEventDestroy(ev_inall);
  for (int G = 0; G < ng; ++G) {
    if (ev_in[G]) cudaEventDestroy(ev_in[G]);
    if (ev_run[G]) cudaEventDestroy(ev_run[G]);
  }
  if (rc != RA_OK) return rc;
  if (e != cudaSuccess) return cuda_fail(e, "pipelined host-buffer ring");
  return RA_OK;
}

int ra_ring_forward_host(const void* q_host, const void* k_host, const void* v_host,
                         float* out_host, float* lse_host, long long N, int P, int causal, int d,
                         int heads, int kv_heads, int dtype, void* stream) {
  int rc = ring_args_check(N, P, 0, d, heads, kv_heads, dtype, RA_LAYOUT_CONTIGUOUS);
  if (rc != RA_OK) return rc;
  if (N == 0) return RA_OK;
  if (!q_host || !k_host || !v_host || !out_host || !lse_host)
    return fail(RA_ERR_INVALID, "a host pointer is NULL");
  if (dtype == RA_BF16 && P <= kFusedMaxSteps) {
    rc = ring_forward_host_pipelined(q_host, k_host, v_host, out_host, lse_host, N, P, causal, d,
                                     heads, kv_heads, static_cast<cudaStream_t>(stream));
    const int st_rc = ra_device_status(stream);
    if (rc != RA_OK) return rc;
    return st_rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t esz = dtype == RA_BF16 ? 2 : 4;
  const size_t q_bytes = static_cast<size_t>(N) * heads * d * esz;
  const size_t kv_bytes = static_cast<size_t>(N) * kv_heads * d * esz;
  const size_t out_bytes = static_cast<size_t>(N) * heads * d * sizeof(float);
  const size_t rh_bytes = static_cast<size_t>(N) * heads * sizeof(float);
  void *dq = nullptr, *dk = nullptr, *dv = nullptr;
  float *dout = nullptr, *dlse = nullptr, *dl = nullptr;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void** p, size_t n) {
    if (e == cudaSuccess) e = scratch_alloc(p, n, st);
  };
  alloc(&dq, q_bytes);
  alloc(&dk, kv_bytes);
  alloc(&dv, kv_bytes);
  alloc(reinterpret_cast<void**>(&dout), out_bytes);
  alloc(reinterpret_cast<void**>(&dlse), rh_bytes);
  alloc(reinterpret_cast<void**>(&dl), rh_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    rc = fail(RA_ERR_ALLOC, "pool allocation of device staging failed: %s", cudaGetErrorString(e));
  } else {
    e = cudaMemcpyAsync(dq, q_host, q_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k_host, kv_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v_host, kv_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "host-to-device copy");
    } else {
      rc = ring_forward_impl(dq, dk, dv, dout, dlse, N, P, plain_mask(causal), d, heads, kv_heads,
                             dtype, st, dl);
      if (rc == RA_OK) {
        e = cudaMemcpyAsync(out_host, dout, out_bytes, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(lse_host, dlse, rh_bytes, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) rc = cuda_fail(e, "device-to-host copy");
      }
    }
  }
  void* bufs[6] = {dq, dk, dv, dout, dlse, dl};
  for (void* p : bufs)
    if (p) cudaFreeAsync(p, st);
  const int st_rc = ra_device_status(stream);
  if (rc != RA_OK) return rc;
  return st_rc;
}

int ra_ring_forward_noalloc(const void* q, const void* k, const void* v, float* out, float* lse,
                            long long N, int P, int causal, int d, int heads, int kv_heads,
                            int dtype, void* stream) {
  int rc = ring_args_check(N, P, 0, d, heads, kv_heads, dtype, RA_LAYOUT_CONTIGUOUS);
  if (rc != RA_OK) return rc;
  // The documented limit holds for every dtype, although the bf16 ring (one
  // fused launch) needs no scratch.  It is checked before the pointers and
  // before any launch, so an over-the-limit call never touches its buffers.
  if (N * heads > kNoAllocMaxRowsHeads)
    return fail(RA_ERR_UNSUPPORTED,
                "N * heads = %lld exceeds the fixed scratch of ra_ring_forward_noalloc (%lld "
                "rows x heads); use ra_ring_forward",
                N * heads, kNoAllocMaxRowsHeads);
  if (N == 0) return RA_OK;
  if ((rc = check_ptrs({q, k, v, out, lse})) != RA_OK) return rc;
  if (ring_is_fused(dtype, P))
    return ring_forward_impl(q, k, v, out, lse, N, P, plain_mask(causal), d, heads, kv_heads,
                             dtype, static_cast<cudaStream_t>(stream), nullptr);
  float* l_scratch = nullptr;
  if ((rc = noalloc_scratch(&l_scratch)) != RA_OK) return rc;
  // The state-init kernel zeroes the l rows this call uses, so whatever a
  // previous call left in the array does not matter.
  return ring_forward_impl(q, k, v, out, lse, N, P, plain_mask(causal), d, heads, kv_heads, dtype,
                           static_cast<cudaStream_t>(stream), l_scratch);
}

int ra_ring_backward_masked(const void* q, const void* k, const void* v, const float* out,
                            const float* lse, const void* dout, float* dq, float* dk, float* dv,
                            long long N, int P, int layout, int causal, long long window,
                            long long n_valid, const int* cu_seqlens, int ndocs, int d, int heads,
                            int kv_heads, int dtype, void* stream) {
  int rc = ring_args_check(N, P, 0, d, heads, kv_heads, dtype, layout);
  if (rc != RA_OK) return rc;
  if (dtype != RA_BF16) return fail(RA_ERR_UNSUPPORTED, "the backward ring takes bf16 q, k, v, dout");
  MaskSpec mk;
  if ((rc = check_mask(layout, causal, window, n_valid, cu_seqlens, ndocs, &mk)) != RA_OK) return rc;
  if (N == 0) return RA_OK;
  if ((rc = check_ptrs({q, k, v, out, lse, dout, dq, dk, dv})) != RA_OK) return rc;
  return ring_backward_impl(q, k, v, out, lse, dout, dq, dk, dv, N, P, mk, d, heads, kv_heads,
                            static_cast<cudaStream_t>(stream));
}

int ra_ring_backward(const void* q, const void* k, const void* v, const float* out,
                     const float* lse, const void* dout, float* dq, float* dk, float* dv,
                     long long N, int P, int causal, int d, int heads, int kv_heads, int dtype,
                     void* stream) {
  return ra_ring_backward_masked(q, k, v, out, lse, dout, dq, dk, dv, N, P, RA_LAYOUT_CONTIGUOUS,
                                 causal ? 1 : 0, 0, -1, nullptr, 0, d, heads, kv_heads, dtype,
                                 stream);
}

int ra_decode_partial(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                      long long n_q, long long n_kv, int d, int heads, int kv_heads,
                      long long q_off, long long kv_off, int causal, long long window,
                      int dtype, void* stream) {
  int rc = decode_args_check(q, k, v, n_q, n_kv, d, heads, kv_heads, window, dtype);
  if (rc != RA_OK) return rc;
  if (n_q == 0 || n_kv == 0) return RA_OK;
  if ((rc = check_ptrs({q, k, v, m, l, o})) != RA_OK) return rc;
  return decode_run(q, k, v, m, l, o, n_q, n_kv, n_kv, 1, q_off, kv_off, causal, window, d, heads,
                    kv_heads, static_cast<cudaStream_t>(stream));
}

int ra_decode_forward(const void* q, const void* k, const void* v, float* out, float* lse,
                      long long n_q, long long n_kv, int P, long long q_off, int causal,
                      long long window, int d, int heads, int kv_heads, int dtype,
                      void* stream) {
  int rc = decode_args_check(q, k, v, n_q, n_kv, d, heads, kv_heads, window, dtype);
  if (rc != RA_OK) return rc;
  if (P < 1 || P > 65535) return fail(RA_ERR_INVALID, "P=%d out of range [1, 65535]", P);
  if (n_q == 0) return RA_OK;
  if ((rc = check_ptrs({q, out, lse})) != RA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = n_q * heads;
  if (n_kv == 0) {  // no key: every row is empty (out = 0, lse = -inf)
    float* l0 = nullptr;
    cudaError_t e = scratch_alloc(reinterpret_cast<void**>(&l0), rows * sizeof(float), st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(RA_ERR_ALLOC, "pool allocation of %lld floats failed", rows);
    }
    e = ra::launch_state_init(lse, l0, out, n_q, heads, d, st);
    if (e == cudaSuccess) e = ra::launch_finalize(lse, l0, out, out, lse, n_q, heads, d, st);
    const cudaError_t ef = cudaFreeAsync(l0, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode empty-key launch");
    return ef == cudaSuccess ? RA_OK : cuda_fail(ef, "cudaFreeAsync");
  }
  if ((rc = check_ptrs({k, v})) != RA_OK) return rc;
  const long long shard_len = (n_kv + P - 1) / P;
  const int nshard = static_cast<int>((n_kv + shard_len - 1) / shard_len);
  // Each shard's chunks give partial states; one launch then folds them all
  // (the global reduction of the merge operator) and finalizes.
  return decode_run(q, k, v, nullptr, nullptr, nullptr, n_q, n_kv, shard_len, nshard, q_off, 0,
                    causal, window, d, heads, kv_heads, st, out, lse);
}

int ra_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int a = 0, b = 0, c = 0, w = 0;
  if ((e = ra::take_umma_status(&a)) != cudaSuccess) return cuda_fail(e, "reading the tcgen05 kernel status");
  if ((e = ra::take_simt_status(&b)) != cudaSuccess) return cuda_fail(e, "reading the fp32 kernel status");
  if ((e = ra::take_decode_status(&c)) != cudaSuccess) return cuda_fail(e, "reading the decode kernel status");
  if ((e = ra::take_bwd_status(&w)) != cudaSuccess) return cuda_fail(e, "reading the backward kernel status");
  if (a != 0 || b != 0 || c != 0 || w != 0)
    return fail(RA_ERR_TIMEOUT, "a kernel gave up a bounded wait (codes 0x%x, 0x%x, 0x%x, 0x%x)",
                a, b, c, w);
  return RA_OK;
}

int ra_selftest_wait_timeout(long long limit_cycles, void* stream) {
  if (limit_cycles < 0) return fail(RA_ERR_INVALID, "limit_cycles must be >= 0");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = ra::launch_wait_selftest(limit_cycles, st);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ra_device_status(stream);
}

int ra_trace_enable(int on) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  g_trace_on = on != 0;
  return RA_OK;
}

int ra_cached_memory(long long* bytes) {
  if (!bytes) return fail(RA_ERR_INVALID, "bytes is NULL");
  *bytes = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return RA_OK;
  std::lock_guard<std::mutex> g(g_pool_mu);
  if (!g_pool[dev]) return RA_OK;
  uint64_t held = 0;
  e = cudaMemPoolGetAttribute(g_pool[dev], cudaMemPoolAttrReservedMemCurrent, &held);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolGetAttribute");
  *bytes = static_cast<long long>(held);
  return RA_OK;
}

int ra_release_cached_memory(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return RA_OK;
  std::lock_guard<std::mutex> g(g_pool_mu);
  if (!g_pool[dev]) return RA_OK;
  e = cudaMemPoolTrimTo(g_pool[dev], 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolTrimTo");
  return RA_OK;
}

int ra_trace_reset(void) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  for (auto& r : g_trace) {
    g_ev_pool.push_back(r.start);
    g_ev_pool.push_back(r.stop);
  }
  g_trace.clear();
  return RA_OK;
}

int ra_trace_query(int kind, long long* launches, double* total_ms) {
  if (kind < 0 || kind >= RA_KERNEL_KINDS) return fail(RA_ERR_INVALID, "unknown kernel kind %d", kind);
  if (!launches || !total_ms) return fail(RA_ERR_INVALID, "NULL output pointer");
  std::lock_guard<std::mutex> g(g_trace_mu);
  long long n = 0;
  double ms = 0.0;
  for (auto& r : g_trace) {
    if (r.kind != kind) continue;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float x = 0.f;
    e = cudaEventElapsedTime(&x, r.start, r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    ms += x;
    ++n;
  }
  *launches = n;
  *total_ms = ms;
  return RA_OK;
}

}  // extern "C"
