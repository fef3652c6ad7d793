// fp32 block update and fused ring on the FFMA pipes.  fp32 inputs are held to 1e-5,
// which tf32 tensor cores cannot meet.  It follows the same recurrence as
// the tcgen05 kernel, in natural-log units.
//
// A CTA owns 64 query rows of one head.  It stages 64-key K/V tiles in
// shared memory and loops over the tiles of the K/V block:
//   S = Q K^T * scale   (4x4 register tile per thread),
//   mask,               (each row's interval of allowed keys)
//   row max / sum       (one warp per 8 rows, warp shuffles),
//   O = alpha O + P V   (O in registers, 4 rows x d/16 columns per thread).
// Only key tiles that some row of the CTA may see are visited.
#include <cmath>
#include <cstdint>

#include "ra_internal.h"

namespace ra {

__device__ int g_simt_status = 0;

namespace {

constexpr int BQ = 64;
constexpr int BK = 64;
constexpr int NT = 256;

template <int D>
struct SimtSmem {
  float q[BQ][D + 1];
  float k[BK][D + 1];
  float v[BK][D + 1];
  float s[BQ][BK + 1];
  float m[BQ];
  float l[BQ];
  float alpha[BQ];
  int lo[BQ];  // allowed keys of row r: lo[r] <= key index < hi[r]
  int hi[BQ];
};

// Per-row key intervals of this query tile for one K/V block (lo, hi) into
// shared memory.  The caller synchronizes before they are read.
template <int D>
__device__ __forceinline__ void row_intervals(const FwdArgs& a, const Work& wk, long long q_tile0,
                                              long long vb, SimtSmem<D>& sm) {
  const int tid = threadIdx.x;
  if (tid < BQ) {
    long long lo = 0, hi = 0;
    if (q_tile0 + tid < a.cq) row_keys(a, wk, q_tile0 + tid, vb, &lo, &hi);
    sm.lo[tid] = static_cast<int>(lo);
    sm.hi[tid] = static_cast<int>(hi);
  }
}

// This CTA's Q tile (64 rows of head h) into shared memory.
template <int D>
__device__ __forceinline__ void load_q_tile(const FwdArgs& a, const Work& wk, long long q_tile0,
                                            int h, SimtSmem<D>& sm) {
  const float* __restrict__ Q = static_cast<const float*>(a.q);
  for (int i = threadIdx.x; i < BQ * D / 4; i += NT) {
    const int r = i / (D / 4), c4 = i % (D / 4);
    const long long gr = q_tile0 + r;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gr < a.cq)
      x = reinterpret_cast<const float4*>(Q + ((wk.q_base + gr) * a.heads + h) * D)[c4];
    sm.q[r][4 * c4 + 0] = x.x;
    sm.q[r][4 * c4 + 1] = x.y;
    sm.q[r][4 * c4 + 2] = x.z;
    sm.q[r][4 * c4 + 3] = x.w;
  }
}

// Fold the key tiles [t_first, t_end) of one K/V block into the running
// state: m, l in shared memory, O~ in registers (rows ty + 16 i, columns
// tx + 16 j).  The Q tile and the row intervals are in shared memory and
// synchronized.
template <int D>
__device__ __forceinline__ void fold_block(const FwdArgs& a, const Work& wk, int kh, int t_first,
                                           int t_end, SimtSmem<D>& sm,
                                           float (&acc)[4][D / 16]) {
  constexpr int OC = D / 16;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int lane = tid & 31, warp = tid >> 5;
  const float* __restrict__ K = static_cast<const float*>(a.k);
  const float* __restrict__ V = static_cast<const float*>(a.v);
  for (long long t = t_first; t < t_end; ++t) {
    const long long k0 = t * BK;
    for (int i = tid; i < BK * D / 4; i += NT) {
      const int r = i / (D / 4), c4 = i % (D / 4);
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
      if (k0 + r < a.ck) {
        const long long off = ((wk.kv_base + k0 + r) * a.kv_heads + kh) * D;
        x = reinterpret_cast<const float4*>(K + off)[c4];
        y = reinterpret_cast<const float4*>(V + off)[c4];
      }
      sm.k[r][4 * c4 + 0] = x.x; sm.k[r][4 * c4 + 1] = x.y;
      sm.k[r][4 * c4 + 2] = x.z; sm.k[r][4 * c4 + 3] = x.w;
      sm.v[r][4 * c4 + 0] = y.x; sm.v[r][4 * c4 + 1] = y.y;
      sm.v[r][4 * c4 + 2] = y.z; sm.v[r][4 * c4 + 3] = y.w;
    }
    __syncthreads();

    // S = Q K^T * scale, masked.
    float sacc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sacc[i][j] = 0.f;
#pragma unroll 8
    for (int x = 0; x < D; ++x) {
      float qa[4], kb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qa[i] = sm.q[ty + 16 * i][x];
#pragma unroll
      for (int j = 0; j < 4; ++j) kb[j] = sm.k[tx + 16 * j][x];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sacc[i][j] = fmaf(qa[i], kb[j], sacc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty + 16 * i;
      const long long lo = sm.lo[r], hi = sm.hi[r];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int cidx = tx + 16 * j;
        const long long kl = k0 + cidx;
        const bool ok = kl >= lo && kl < hi;
        sm.s[r][cidx] = ok ? sacc[i][j] * a.scale : -INFINITY;
      }
    }
    __syncthreads();

    // Row statistics: warp w takes rows 8w .. 8w+7, two columns per lane.
#pragma unroll
    for (int rr = 0; rr < BQ / 8; ++rr) {
      const int r = warp * (BQ / 8) + rr;
      const float s0 = sm.s[r][lane], s1 = sm.s[r][lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = sm.m[r];
      const float m_new = fmaxf(m_old, mx);
      const float mref = (m_new == -INFINITY) ? 0.f : m_new;
      const float p0 = expf(s0 - mref), p1 = expf(s1 - mref);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      // alpha = exp(m_old - m_new); a still-empty row keeps its state.
      const float alpha = (m_new == -INFINITY) ? 1.f : expf(m_old - mref);
      sm.s[r][lane] = p0;
      sm.s[r][lane + 32] = p1;
      __syncwarp();
      if (lane == 0) {
        sm.alpha[r] = alpha;
        sm.l[r] = alpha * sm.l[r] + sum;
        sm.m[r] = m_new;
      }
    }
    __syncthreads();

    // O = alpha O + P V.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float al = sm.alpha[ty + 16 * i];
#pragma unroll
      for (int j = 0; j < OC; ++j) acc[i][j] *= al;
    }
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      float p[4], vv[OC];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = sm.s[ty + 16 * i][kk];
#pragma unroll
      for (int j = 0; j < OC; ++j) vv[j] = sm.v[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < OC; ++j) acc[i][j] = fmaf(p[i], vv[j], acc[i][j]);
    }
    __syncthreads();
  }
}

template <int D>
__global__ void __launch_bounds__(NT) simt_update_kernel(const FwdArgs a) {
  extern __shared__ float4 smem_f4[];
  SimtSmem<D>& sm = *reinterpret_cast<SimtSmem<D>*>(smem_f4);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int h = blockIdx.y;
  const int kh = h / (a.heads / a.kv_heads);
  const Work wk = decode_work(a, blockIdx.z);
  const long long q_tile0 = static_cast<long long>(blockIdx.x) * BQ;
  if (q_tile0 >= a.cq) return;

  // Key tiles [t_first, t_end) hold every key some row of this tile may see.
  const long long vb = valid_bound(a.mask);
  int t_first, t_end;
  tile_range(a, wk, q_tile0, q_tile0 + BQ, vb, BK, &t_first, &t_end);
  if (t_end <= t_first) return;  // state unchanged
  row_intervals(a, wk, q_tile0, vb, sm);
  load_q_tile(a, wk, q_tile0, h, sm);
  if (tid < BQ) {
    const long long gr = q_tile0 + tid;
    float mm = -INFINITY, ll = 0.f;
    if (gr < a.cq) {
      const long long si = (wk.state_base + gr) * a.heads + h;
      mm = a.m[si];
      ll = a.l[si];
    }
    sm.m[tid] = mm;
    sm.l[tid] = ll;
  }
  constexpr int OC = D / 16;  // output columns per thread: tx + 16 * j
  float acc[4][OC];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long gr = q_tile0 + ty + 16 * i;
    const float* src = a.o + ((wk.state_base + gr) * a.heads + h) * D;
#pragma unroll
    for (int j = 0; j < OC; ++j) acc[i][j] = (gr < a.cq) ? src[tx + 16 * j] : 0.f;
  }
  __syncthreads();
  fold_block<D>(a, wk, kh, t_first, t_end, sm, acc);

  // State out.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long gr = q_tile0 + ty + 16 * i;
    if (gr < a.cq) {
      float* dst = a.o + ((wk.state_base + gr) * a.heads + h) * D;
#pragma unroll
      for (int j = 0; j < OC; ++j) dst[tx + 16 * j] = acc[i][j];
    }
  }
  if (tid < BQ) {
    const long long gr = q_tile0 + tid;
    if (gr < a.cq) {
      const long long si = (wk.state_base + gr) * a.heads + h;
      a.m[si] = sm.m[tid];
      a.l[si] = sm.l[tid];
    }
  }
}

// The whole fp32 ring in one launch: CTA (query tile, head, rank i) keeps
// its 64 query rows and their state (m, l in shared memory, O~ in
// registers) for every ring step s = 0 .. P-1, folding K/V block
// j = (i - s) mod P, and finalizes at the end: out = O~ / l and
// lse = m + ln l (0 and -inf for a row that saw no key).  The same folds in
// the same order as one launch per step, without the state's round trips
// through HBM.  out [rows, heads, d] and lse [rows, heads] are a.o and a.m.
template <int D>
__global__ void __launch_bounds__(NT) simt_ring_kernel(const FwdArgs a) {
  extern __shared__ float4 smem_f4[];
  SimtSmem<D>& sm = *reinterpret_cast<SimtSmem<D>*>(smem_f4);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int h = blockIdx.y;
  const int kh = h / (a.heads / a.kv_heads);
  const int i = static_cast<int>(blockIdx.z);
  const long long q_tile0 = static_cast<long long>(blockIdx.x) * BQ;
  if (q_tile0 >= a.cq) return;
  const long long vb = valid_bound(a.mask);
  constexpr int OC = D / 16;
  float acc[4][OC];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < OC; ++j) acc[r][j] = 0.f;
  if (tid < BQ) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  bool q_loaded = false;
  for (int s = 0; s < a.P; ++s) {
    Work wk;
    const int j = (i - s + a.P) % a.P;
    wk.q_base = static_cast<long long>(i) * a.cq;
    wk.kv_base = static_cast<long long>(j) * a.ck;
    wk.state_base = wk.q_base;
    wk.qmap = PosMap{a.layout, a.P, a.cq, i, wk.q_base};
    wk.kmap = PosMap{a.layout, a.P, a.ck, j, wk.kv_base};
    int t_first, t_end;
    tile_range(a, wk, q_tile0, q_tile0 + BQ, vb, BK, &t_first, &t_end);
    if (t_end <= t_first) continue;  // uniform across the CTA
    __syncthreads();  // the previous step's readers of lo/hi are done
    row_intervals(a, wk, q_tile0, vb, sm);
    if (!q_loaded) {
      load_q_tile(a, wk, q_tile0, h, sm);
      q_loaded = true;
    }
    __syncthreads();
    fold_block<D>(a, wk, kh, t_first, t_end, sm, acc);
  }
  __syncthreads();
  // Finalize.
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = ty + 16 * r;
    const long long gr = q_tile0 + row;
    if (gr < a.cq) {
      const float ll = sm.l[row];
      const float inv = ll > 0.f ? 1.f / ll : 0.f;
      float* dst = a.o + ((static_cast<long long>(i) * a.cq + gr) * a.heads + h) * D;
#pragma unroll
      for (int j = 0; j < OC; ++j) dst[tx + 16 * j] = acc[r][j] * inv;
    }
  }
  if (tid < BQ) {
    const long long gr = q_tile0 + tid;
    if (gr < a.cq) {
      const float ll = sm.l[tid];
      a.m[(static_cast<long long>(i) * a.cq + gr) * a.heads + h] =
          ll > 0.f ? sm.m[tid] + logf(ll) : -INFINITY;
    }
  }
}

template <int D>
cudaError_t launch_ring_d(const FwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(SimtSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(simt_ring_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.cq + BQ - 1) / BQ), a.heads, a.P);
  simt_ring_kernel<D><<<grid, NT, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(SimtSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(simt_update_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.cq + BQ - 1) / BQ), a.heads, a.nwork);
  simt_update_kernel<D><<<grid, NT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_update(const FwdArgs& a, int d, cudaStream_t st) {
  return d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

cudaError_t launch_simt_ring(const FwdArgs& a, int d, cudaStream_t st) {
  return d == 128 ? launch_ring_d<128>(a, st) : launch_ring_d<64>(a, st);
}

cudaError_t take_simt_status(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_simt_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_simt_status, &zero, sizeof(int));
}

}  // namespace ra
