// State kernels: identity init, log-sum-exp merge, finalize.  All three are
// HBM-bound streams over [rows, heads] scalars and [rows, heads, d] fp32
// vectors.  Merge and finalize give one warp to one (row, head): lane 0
// reads the two scalars, and the per-row factors reach the other lanes by
// warp shuffle.  The d-vector then moves as coalesced float4 (d = 128) or
// float2 (d = 64) accesses, one 512- or 256-byte run per warp.
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

template <int D>
__global__ void merge_kernel(float* __restrict__ m_a, float* __restrict__ l_a,
                             float* __restrict__ o_a, const float* __restrict__ m_b,
                             const float* __restrict__ l_b, const float* __restrict__ o_b,
                             long long n_rh) {
  const int lane = threadIdx.x & 31;
  const long long rh = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (rh >= n_rh) return;  // warp-uniform
  float m = 0.f, ea = 0.f, eb = 0.f;
  if (lane == 0) {
    const float ma = m_a[rh], mb = m_b[rh];
    merge_factors(ma, mb, m, ea, eb);
    l_a[rh] = ea * l_a[rh] + eb * l_b[rh];
    m_a[rh] = m;
  }
  ea = __shfl_sync(0xffffffffu, ea, 0);
  eb = __shfl_sync(0xffffffffu, eb, 0);
  if constexpr (D == 128) {
    float4* pa = reinterpret_cast<float4*>(o_a + rh * D) + lane;
    const float4 x = *pa;
    const float4 y = reinterpret_cast<const float4*>(o_b + rh * D)[lane];
    *pa = make_float4(ea * x.x + eb * y.x, ea * x.y + eb * y.y, ea * x.z + eb * y.z,
                      ea * x.w + eb * y.w);
  } else {
    float2* pa = reinterpret_cast<float2*>(o_a + rh * D) + lane;
    const float2 x = *pa;
    const float2 y = reinterpret_cast<const float2*>(o_b + rh * D)[lane];
    *pa = make_float2(ea * x.x + eb * y.x, ea * x.y + eb * y.y);
  }
}

template <int D>
__global__ void finalize_kernel(const float* m, const float* l, const float* o, float* out,
                                float* lse, long long n_rh) {
  // `out` may alias `o` and `lse` may alias `m`: every element is read
  // before it is written, by the same thread.
  const int lane = threadIdx.x & 31;
  const long long rh = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (rh >= n_rh) return;
  float inv = 0.f;
  if (lane == 0) {
    const float mm = m[rh], ll = l[rh];
    float val;
    if (ll > 0.f) {
      inv = 1.f / ll;
      val = mm + logf(ll);
    } else {
      val = -INFINITY;
    }
    lse[rh] = val;
  }
  inv = __shfl_sync(0xffffffffu, inv, 0);
  if constexpr (D == 128) {
    const float4 x = reinterpret_cast<const float4*>(o + rh * D)[lane];
    reinterpret_cast<float4*>(out + rh * D)[lane] =
        make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
  } else {
    const float2 x = reinterpret_cast<const float2*>(o + rh * D)[lane];
    reinterpret_cast<float2*>(out + rh * D)[lane] = make_float2(x.x * inv, x.y * inv);
  }
}

int grid_for_warps(long long n_warps) {
  const long long warps_per_block = kThreads / 32;
  return static_cast<int>((n_warps + warps_per_block - 1) / warps_per_block);
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
  const int grid = grid_for_warps(n_rh);
  if (d == 128)
    merge_kernel<128><<<grid, kThreads, 0, st>>>(m_a, l_a, o_a, m_b, l_b, o_b, n_rh);
  else
    merge_kernel<64><<<grid, kThreads, 0, st>>>(m_a, l_a, o_a, m_b, l_b, o_b, n_rh);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* m, const float* l, const float* o, float* out,
                            float* lse, long long rows, int heads, int d, cudaStream_t st) {
  const long long n_rh = rows * heads;
  if (n_rh == 0) return cudaSuccess;
  const int grid = grid_for_warps(n_rh);
  if (d == 128)
    finalize_kernel<128><<<grid, kThreads, 0, st>>>(m, l, o, out, lse, n_rh);
  else
    finalize_kernel<64><<<grid, kThreads, 0, st>>>(m, l, o, out, lse, n_rh);
  return cudaGetLastError();
}

}  // namespace ra
