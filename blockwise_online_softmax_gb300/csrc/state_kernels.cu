// State kernels: identity init, log-sum-exp merge, finalize.  All three are
// HBM-bound streams over [rows, heads] scalars and [rows, heads, d] fp32
// vectors, moved as coalesced float4 accesses by grid-stride loops over
// grids sized to fill every SM.
#include <cmath>
#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreads = 256;

__global__ void state_init_kernel(float* __restrict__ m, float* __restrict__ l,
                                  float4* __restrict__ o4, long long n_rh, long long n_o4) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (long long i = t0; i < n_rh; i += stride) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = t0; i < n_o4; i += stride) o4[i] = z;
}

// Scale factors of a (+) b for one (row, head).  Both sides relative to
// m = max(m_a, m_b).  When both are -inf (two empty states) the result is
// the empty state: the factors are 1 and the sums stay 0.
__device__ __forceinline__ void merge_factors(float ma, float mb, float& m, float& ea, float& eb) {
  m = fmaxf(ma, mb);
  const float mref = (m == -INFINITY) ? 0.f : m;
  ea = (ma == -INFINITY) ? (m == -INFINITY ? 1.f : 0.f) : expf(ma - mref);
  eb = (mb == -INFINITY) ? (m == -INFINITY ? 1.f : 0.f) : expf(mb - mref);
}

// The merge streams O~ as float4s in warp-sized chunks: a warp takes
// kRows * 32 consecutive float4s per iteration, whole (row, head) entries
// of D / 4 float4s each (kRows entries at D = 128, 2 kRows at D = 64), so
// its addresses are one base plus constant offsets and each lane issues
// 2 kRows independent loads of O~ before any arithmetic.  Lane e loads
// the scalars (m, l) of both states for the chunk's entry e, computes that
// entry's factors and writes its new scalars; the factors reach the lanes
// holding the entry's O~ by shuffles.  Each lane reads and writes only its
// own float4s and its own entry's scalars, so merging into a in place is
// safe.  The grid-strided form of the finalize below, in which every lane
// loads its entry's scalars as a warp broadcast, reached 0.86 of the HBM
// copy bandwidth on the merge: its four scalar loads per float4 pair, not
// DRAM, set the pace.
constexpr int kRows = 16;

template <int D>
struct Chunk {
  static constexpr int V = D / 4;             // float4s per (row, head)
  static constexpr int RPU = 32 / V;          // entries per 32 float4s
  static constexpr int ENTRIES = kRows * RPU; // entries per warp iteration
  static_assert(ENTRIES <= 32, "one lane per entry");
};

__device__ __forceinline__ long long warp_id_global() {
  return static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
}

template <int D>
__global__ void __launch_bounds__(kThreads) merge_kernel(
    float* __restrict__ m_a, float* __restrict__ l_a, float4* __restrict__ o_a,
    const float* __restrict__ m_b, const float* __restrict__ l_b,
    const float4* __restrict__ o_b, long long n_rh) {
  using C = Chunk<D>;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  const int lane = threadIdx.x & 31;
  for (long long rh0 = warp_id_global() * C::ENTRIES; rh0 < n_rh; rh0 += nwarps * C::ENTRIES) {
    const bool full = rh0 + C::ENTRIES <= n_rh;
    const long long r0 = rh0 + lane / C::V;  // the entry of this lane's float4 at u = 0
    const bool own = lane < C::ENTRIES && rh0 + lane < n_rh;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    if (own) {
      ma = m_a[rh0 + lane];
      la = l_a[rh0 + lane];
      mb = __ldg(m_b + rh0 + lane);
      lb = __ldg(l_b + rh0 + lane);
    }
    float4* pa = o_a + rh0 * C::V + lane;
    const float4* pb = o_b + rh0 * C::V + lane;
    float4 x[kRows], y[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if (full || r0 + u * C::RPU < n_rh) {
        x[u] = pa[u * 32];
        y[u] = __ldg(pb + u * 32);
      }
    }
    float m, ea, eb;
    merge_factors(ma, mb, m, ea, eb);
    if (own) {
      l_a[rh0 + lane] = ea * la + eb * lb;
      m_a[rh0 + lane] = m;
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int src = u * C::RPU + lane / C::V;
      const float fa = __shfl_sync(0xffffffffu, ea, src);
      const float fb = __shfl_sync(0xffffffffu, eb, src);
      if (full || r0 + u * C::RPU < n_rh)
        pa[u * 32] = make_float4(fa * x[u].x + fb * y[u].x, fa * x[u].y + fb * y[u].y,
                                 fa * x[u].z + fb * y[u].z, fa * x[u].w + fb * y[u].w);
    }
  }
}

// The finalize streams its one input and one output grid-strided: a
// thread takes kUnroll float4s a grid stride apart (float4 e of the
// [rows * heads, D] array belongs to (row, head) rh = e / (D / 4)) and
// issues all their loads, and those of the m and l of their (row, head)
// as warp broadcasts, before any arithmetic.  The lane that holds the
// first float4 of a (row, head) writes its LSE.  A (row, head) lies within
// one warp, and its scalars are read by the warp's loads, which a
// __syncwarp puts before that lane's store, so the in-place form (out = o,
// lse = m) is safe.  The loop runs over warp-aligned bases, so every lane
// of a warp takes the same number of iterations and reaches each
// __syncwarp.  With one read per write this form runs at the copy
// bandwidth; the chunked form of the merge measured 1% slower here.
constexpr int kUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kThreads) finalize_kernel(
    const float* m, const float* l, const float4* o, float4* out, float* lse, long long n4) {
  constexpr int V = D / 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (long long w0 = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       w0 < n4; w0 += kUnroll * stride) {
    float4 x[kUnroll];
    float mm[kUnroll], ll[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long e = w0 + u * stride + lane;
      if (e < n4) {
        const long long rh = e / V;
        x[u] = o[e];
        mm[u] = m[rh];
        ll[u] = l[rh];
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long e = w0 + u * stride + lane;
      if (e < n4) {
        const bool seen = ll[u] > 0.f;
        const float inv = seen ? 1.f / ll[u] : 0.f;
        out[e] = make_float4(x[u].x * inv, x[u].y * inv, x[u].z * inv, x[u].w * inv);
        if (e % V == 0) lse[e / V] = seen ? mm[u] + logf(ll[u]) : -INFINITY;
      }
    }
  }
}

// Grid of the streaming kernels: every SM holds as many CTAs of `kernel`
// as fit, and no more CTAs than the work needs (`n4` threads' worth).
template <typename K>
int stream_grid(K kernel, long long n4) {
  int dev = 0, sms = 148, per_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long want = (n4 + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(sms) * per_sm;
  return static_cast<int>(want < cap ? want : cap);
}

// Threads the merge needs: one per kRows float4s.
long long chunk_threads(long long n_rh, int d) {
  return (n_rh * (d / 4) + kRows - 1) / kRows;
}

}  // namespace

cudaError_t launch_state_init(float* m, float* l, float* o, long long rows, int heads, int d,
                              cudaStream_t st) {
  const long long n_rh = rows * heads;
  const long long n_o4 = n_rh * d / 4;
  if (n_rh == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n_o4 + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  state_init_kernel<<<static_cast<int>(blocks), kThreads, 0, st>>>(
      m, l, reinterpret_cast<float4*>(o), n_rh, n_o4);
  return cudaGetLastError();
}

cudaError_t launch_merge(float* m_a, float* l_a, float* o_a, const float* m_b, const float* l_b,
                         const float* o_b, long long rows, int heads, int d, cudaStream_t st) {
  const long long n_rh = rows * heads;
  if (n_rh == 0) return cudaSuccess;
  const long long threads = chunk_threads(n_rh, d);
  float4* oa = reinterpret_cast<float4*>(o_a);
  const float4* ob = reinterpret_cast<const float4*>(o_b);
  if (d == 128)
    merge_kernel<128><<<stream_grid(merge_kernel<128>, threads), kThreads, 0, st>>>(
        m_a, l_a, oa, m_b, l_b, ob, n_rh);
  else
    merge_kernel<64><<<stream_grid(merge_kernel<64>, threads), kThreads, 0, st>>>(
        m_a, l_a, oa, m_b, l_b, ob, n_rh);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* m, const float* l, const float* o, float* out,
                            float* lse, long long rows, int heads, int d, cudaStream_t st) {
  const long long n4 = rows * heads * d / 4;
  if (n4 == 0) return cudaSuccess;
  const float4* o4 = reinterpret_cast<const float4*>(o);
  float4* out4 = reinterpret_cast<float4*>(out);
  if (d == 128)
    finalize_kernel<128><<<stream_grid(finalize_kernel<128>, n4), kThreads, 0, st>>>(
        m, l, o4, out4, lse, n4);
  else
    finalize_kernel<64><<<stream_grid(finalize_kernel<64>, n4), kThreads, 0, st>>>(
        m, l, o4, out4, lse, n4);
  return cudaGetLastError();
}

}  // namespace ra
