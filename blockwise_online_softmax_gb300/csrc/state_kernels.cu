// State kernels: identity init, log-sum-exp merge, finalize.  All three are
// HBM-bound streams over [rows, heads] scalars and [rows, heads, d] fp32
// vectors, moved as coalesced float4 accesses by grid-stride loops sized to
// fill every SM.
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

// Merge and finalize stream O~ as float4s: float4 e of the [rows * heads,
// D] array belongs to (row, head) rh = e / (D / 4).  A thread takes kUnroll
// float4s a grid stride apart and issues every load of all of them (O~, and
// m and l of their (row, head), which the lanes sharing a (row, head) read
// as one broadcast) before any arithmetic, so each thread keeps several
// independent requests in flight.  The lane that holds the first float4 of
// a (row, head) writes its scalars.  A (row, head) lies within one warp
// (D / 4 = 32 or 16 consecutive float4s), and its scalars are read by the
// warp's loads, which a __syncwarp puts before that lane's store, so the
// in-place forms (merge into a; finalize with out = o, lse = m) are safe.
// The loop runs over warp-aligned bases, so every lane of a warp takes the
// same number of iterations and reaches each __syncwarp.
constexpr int kUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kThreads) merge_kernel(
    float* __restrict__ m_a, float* __restrict__ l_a, float4* __restrict__ o_a,
    const float* __restrict__ m_b, const float* __restrict__ l_b,
    const float4* __restrict__ o_b, long long n4) {
  constexpr int V = D / 4;  // float4s per (row, head)
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (long long w0 = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       w0 < n4; w0 += kUnroll * stride) {
    float4 x[kUnroll], y[kUnroll];
    float ma[kUnroll], mb[kUnroll], la[kUnroll], lb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long e = w0 + u * stride + lane;
      if (e < n4) {
        const long long rh = e / V;
        x[u] = o_a[e];
        y[u] = __ldg(&o_b[e]);
        ma[u] = m_a[rh];
        la[u] = l_a[rh];
        mb[u] = __ldg(&m_b[rh]);
        lb[u] = __ldg(&l_b[rh]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long e = w0 + u * stride + lane;
      if (e < n4) {
        float m, ea, eb;
        merge_factors(ma[u], mb[u], m, ea, eb);
        o_a[e] = make_float4(ea * x[u].x + eb * y[u].x, ea * x[u].y + eb * y[u].y,
                             ea * x[u].z + eb * y[u].z, ea * x[u].w + eb * y[u].w);
        if (e % V == 0) {
          const long long rh = e / V;
          l_a[rh] = ea * la[u] + eb * lb[u];
          m_a[rh] = m;
        }
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) finalize_kernel(
    const float* m, const float* l, const float4* o, float4* out, float* lse, long long n4) {
  // `out` may alias `o` and `lse` may alias `m` (see above).
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
// as fit, and no more CTAs than the work needs.
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
  const long long n4 = rows * heads * d / 4;
  if (n4 == 0) return cudaSuccess;
  float4* oa = reinterpret_cast<float4*>(o_a);
  const float4* ob = reinterpret_cast<const float4*>(o_b);
  if (d == 128)
    merge_kernel<128><<<stream_grid(merge_kernel<128>, n4), kThreads, 0, st>>>(m_a, l_a, oa, m_b,
                                                                                l_b, ob, n4);
  else
    merge_kernel<64><<<stream_grid(merge_kernel<64>, n4), kThreads, 0, st>>>(m_a, l_a, oa, m_b,
                                                                              l_b, ob, n4);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* m, const float* l, const float* o, float* out,
                            float* lse, long long rows, int heads, int d, cudaStream_t st) {
  const long long n4 = rows * heads * d / 4;
  if (n4 == 0) return cudaSuccess;
  const float4* o4 = reinterpret_cast<const float4*>(o);
  float4* out4 = reinterpret_cast<float4*>(out);
  if (d == 128)
    finalize_kernel<128><<<stream_grid(finalize_kernel<128>, n4), kThreads, 0, st>>>(m, l, o4,
                                                                                      out4, lse, n4);
  else
    finalize_kernel<64><<<stream_grid(finalize_kernel<64>, n4), kThreads, 0, st>>>(m, l, o4, out4,
                                                                                    lse, n4);
  return cudaGetLastError();
}

}  // namespace ra
