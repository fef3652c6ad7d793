// Decode / short-query attention: a few query tokens against a long K/V
// history, the regime of "Ring Attention：把超长序列沿设备环流动", section
// "训练与推理的适用方式不同".  There a decode step has one new query per
// sequence but must read the whole cached K/V; instead of rotating K/V
// blocks, the query goes to every K/V shard, each shard computes a local
// attention state, and a global online-softmax reduction combines them.
//
// The work is HBM-bound: each K/V byte is read once and meets only
// g * n_q query rows (g = heads / kv_heads), a few FLOPs per byte.  So this
// path runs on the CUDA cores, not the tensor pipe, and is built to keep
// HBM busy:
//   * a CTA takes one KV head and one chunk of one shard's keys (split-K);
//     the grid covers splits x KV heads x shards, a few waves of the SMs;
//   * its four warps each stream their own 32-key K/V tiles through a
//     private ring of shared-memory stages, filled by TMA with 128-byte
//     swizzle, so no warp waits on another inside the loop;
//   * lane t owns key t of a tile for Q K^T (the query rows, pre-scaled by
//     log2(e)/sqrt(d), are broadcast from shared memory) and a slice of the
//     d output columns for P V;
//   * each warp keeps its own online-softmax state; the four are merged in
//     shared memory, and the CTA writes one partial state (m, l, O~).
// decode_combine_kernel then folds a shard's partial states into that
// shard's running state, one warp per (query row, head).  Across shards the
// host reduces with the merge kernel of ra_merge, in a tree.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {

__device__ int g_decode_status = 0;

namespace {

constexpr int DW = 4;         // warps per CTA, each an independent stream
constexpr int KT = 32;        // keys per warp tile: one per lane
constexpr int CHUNK = KT * 128;  // one 64-column swizzled chunk of a 32-row tile

template <int D>
struct DecCfg {
  static constexpr int NCH = D / 64;                 // 64-column chunks per row
  static constexpr int TILE = NCH * CHUNK;           // bytes of one K (or V) tile
  static constexpr int NST = D == 128 ? 3 : 4;       // stages per warp
  static constexpr int STAGE = 2 * TILE;             // K tile, then V tile
  static constexpr int WARP_BYTES = NST * STAGE;
  static constexpr int COLS = D / 32;                // output columns per lane
};

template <int D, int RM>
struct DecSmem {
  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_Q = OFF_STAGES + DW * DecCfg<D>::WARP_BYTES;  // fp32 [RM][D]
  static constexpr int OFF_P = OFF_Q + RM * D * 4;                       // fp32 [DW][RM][KT]
  static constexpr int OFF_LIM = OFF_P + DW * RM * KT * 4;               // int [RM][2]
  static constexpr int OFF_BAR = OFF_LIM + RM * 8;                       // [DW][NST] mbarriers
  static constexpr int OFF_FLAG = OFF_BAR + DW * DecCfg<D>::NST * 8;
  static constexpr int BYTES = OFF_FLAG + 16 + 1024;                     // + alignment slack
  static_assert(BYTES <= 232448, "shared memory budget");
  // The warps' merge area reuses their stage buffers after the loop.
  static_assert(RM * (D + 2) * 4 <= DecCfg<D>::WARP_BYTES, "merge area fits a warp's stages");
};

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
// bf16 pair -> two fp32 (exact: a bf16 is the high half of an fp32).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, int RM>
__global__ void __launch_bounds__(DW * 32, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const DecArgs a) {
  using C = DecCfg<D>;
  using S = DecSmem<D, RM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  float* q_s = reinterpret_cast<float*>(smem + S::OFF_Q);
  int* lim = reinterpret_cast<int*>(smem + S::OFF_LIM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::OFF_FLAG);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, kh = blockIdx.y, shard = blockIdx.z;
  const int g = a.heads / a.kv_heads;
  const int R = g * static_cast<int>(a.n_q);  // rows r = qi * g + hl, head kh * g + hl

  // Keys of this CTA: [c0, c1) of shard `shard`.
  const long long sh0 = static_cast<long long>(shard) * a.shard_len;
  const long long sh1 = sh0 + a.shard_len < a.n_kv ? sh0 + a.shard_len : a.n_kv;
  const long long c0 = sh0 + static_cast<long long>(split) * a.chunk;
  const long long c1 = c0 + a.chunk < sh1 ? c0 + a.chunk : sh1;

  // Allowed keys of each row, clipped to [c0, c1).
  const long long vb = valid_bound(a.mask);
  if (tid < RM) {
    long long lo = 0, hi = 0;
    if (tid < R) {
      const long long qp = a.q_off + tid / g;
      long long plo, phi;
      if (qp < vb && allowed_positions(a.mask, qp, &plo, &phi)) {
        const PosMap km{kContiguous, 1, a.n_kv, 0, a.kv_off};
        lo = count_below(km, plo);
        hi = count_below(km, phi);
      }
    }
    lo = lo > c0 ? lo : c0;
    hi = hi < c1 ? hi : c1;
    if (hi < lo) hi = lo;
    lim[2 * tid] = static_cast<int>(lo);
    lim[2 * tid + 1] = static_cast<int>(hi);
  }
  // Query rows -> fp32, scaled into log2 units.
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  for (int i = tid; i < RM * D; i += DW * 32) {
    const int r = i / D, x = i % D;
    float val = 0.f;
    if (r < R) {
      const long long qi = r / g;
      const int h = kh * g + r % g;
      val = __bfloat162float(q[(qi * a.heads + h) * D + x]) * a.scale_log2;
    }
    q_s[i] = val;
  }
  if (tid == 0) {
    for (int i = 0; i < DW * C::NST; ++i) mbar_init(sb + S::OFF_BAR + 8 * i, 1);
    *abort_flag = *reinterpret_cast<volatile int*>(&g_decode_status) != 0 ? 1 : 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Key range some row may see; tiles of 32 keys aligned on the global key
  // index, dealt round-robin to the warps.
  int klo = static_cast<int>(c1), khi = static_cast<int>(c0);
  for (int r = 0; r < R && r < RM; ++r) {
    if (lim[2 * r + 1] > lim[2 * r]) {
      klo = lim[2 * r] < klo ? lim[2 * r] : klo;
      khi = lim[2 * r + 1] > khi ? lim[2 * r + 1] : khi;
    }
  }
  const int t_begin = klo / KT;
  const int t_end = khi > klo ? (khi + KT - 1) / KT : t_begin;
  const int n_tiles = t_end - t_begin;
  const int nw = n_tiles > warp ? (n_tiles - warp + DW - 1) / DW : 0;  // this warp's tiles

  const uint32_t wbase = sb + S::OFF_STAGES + warp * C::WARP_BYTES;
  const uint32_t wbar = sb + S::OFF_BAR + 8 * warp * C::NST;
  const long long lim_cycles = a.wait_limit;
  auto issue = [&](int it) {  // lane 0: tile `it` of this warp into its stage
    const int st = it % C::NST;
    const int key0 = (t_begin + warp + it * DW) * KT;
    const uint32_t dst = wbase + st * C::STAGE;
    mbar_arrive_expect_tx(wbar + 8 * st, C::STAGE);
#pragma unroll
    for (int ch = 0; ch < C::NCH; ++ch) {
      tma_load_3d(dst + ch * CHUNK, &tmK, wbar + 8 * st, ch * 64, kh, key0);
      tma_load_3d(dst + C::TILE + ch * CHUNK, &tmV, wbar + 8 * st, ch * 64, kh, key0);
    }
  };
  int issued = 0;  // lane 0: tiles whose copies were started
  if (lane == 0 && !*abort_flag) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (; issued < nw && issued < C::NST; ++issued) issue(issued);
  }
  __syncwarp();

  // Warp state per row: m (log2 units), this lane's share of l, and this
  // lane's output columns as fp32 pairs (one FFMA2 updates two).
  constexpr int CP = C::COLS / 2;
  float m_r[RM], l_r[RM];
  uint64_t o2[RM][CP];
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    m_r[r] = -INFINITY;
    l_r[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CP; ++c) o2[r][c] = f2pack(0.f, 0.f);
  }
  const uint32_t p_w = sb + S::OFF_P + warp * RM * KT * 4;
  const uint32_t q_sa = sb + S::OFF_Q;
  bool ok = !*abort_flag;
  int done = 0;  // tiles consumed
  for (int it = 0; it < nw && ok; ++it) {
    const int st = it % C::NST;
    ok = wait_bar(wbar + 8 * st, static_cast<uint32_t>(it / C::NST) & 1u, abort_flag,
                  &g_decode_status, 0x41, lim_cycles);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const uint32_t sK = wbase + st * C::STAGE;
    const uint32_t sV = sK + C::TILE;
    const int key = (t_begin + warp + it * DW) * KT + lane;

    // S = q . k for this lane's key, every row (log2 units): even and odd
    // columns summed in the two halves of an FFMA2 accumulator.
    uint64_t s2[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) s2[r] = f2pack(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < C::NCH; ++ch) {
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint4 kw = lds128(sK + ch * CHUNK + lane * 128 + ((p ^ (lane & 7)) << 4));
        const uint64_t k01 = f2pack(bf_lo(kw.x), bf_hi(kw.x));
        const uint64_t k23 = f2pack(bf_lo(kw.y), bf_hi(kw.y));
        const uint64_t k45 = f2pack(bf_lo(kw.z), bf_hi(kw.z));
        const uint64_t k67 = f2pack(bf_lo(kw.w), bf_hi(kw.w));
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          const uint32_t qa = q_sa + (r * D + ch * 64 + p * 8) * 4;
          const uint4 x = lds128(qa), y = lds128(qa + 16);
          uint64_t acc = s2[r];
          acc = ffma2(f2pack(__uint_as_float(x.x), __uint_as_float(x.y)), k01, acc);
          acc = ffma2(f2pack(__uint_as_float(x.z), __uint_as_float(x.w)), k23, acc);
          acc = ffma2(f2pack(__uint_as_float(y.x), __uint_as_float(y.y)), k45, acc);
          acc = ffma2(f2pack(__uint_as_float(y.z), __uint_as_float(y.w)), k67, acc);
          s2[r] = acc;
        }
      }
    }
    float s[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      float a0, a1;
      f2unpack(s2[r], a0, a1);
      s[r] = a0 + a1;
    }
    // Mask, then the online-softmax update of each row's warp state.
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      const bool allowed = key >= lim[2 * r] && key < lim[2 * r + 1];
      const float sv = allowed ? s[r] : -INFINITY;
      float mt = sv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m_r[r], mt);
      const float mref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m_r[r] - mref);  // m_r = -inf gives 0 (the sums are 0 then)
      const float pv = ex2(sv - mref);         // masked keys give 0
      m_r[r] = m_new;
      l_r[r] = l_r[r] * alpha + pv;
      const uint64_t al2 = f2pack(alpha, alpha);
#pragma unroll
      for (int c = 0; c < CP; ++c) o2[r][c] = fmul2(o2[r][c], al2);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(p_w + (r * KT + lane) * 4), "f"(pv) : "memory");
    }
    __syncwarp();
    // O += P V: lane owns columns [COLS*lane, COLS*lane + COLS).
    const int x0 = C::COLS * lane;
    const int ch = x0 / 64, piece = (x0 % 64) / 8;
    const uint32_t vcol = sV + ch * CHUNK + (x0 % 8) * 2;
#pragma unroll 4
    for (int t4 = 0; t4 < KT; t4 += 4) {
      float pr[RM][4];
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        const uint4 w4 = lds128(p_w + (r * KT + t4) * 4);
        pr[r][0] = __uint_as_float(w4.x);
        pr[r][1] = __uint_as_float(w4.y);
        pr[r][2] = __uint_as_float(w4.z);
        pr[r][3] = __uint_as_float(w4.w);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t4 + u;
        const uint32_t va = vcol + t * 128 + ((piece ^ (t & 7)) << 4);
        uint64_t v2[CP];
        if constexpr (CP == 2) {
          const uint2 w2 = lds64(va);
          v2[0] = f2pack(bf_lo(w2.x), bf_hi(w2.x));
          v2[1] = f2pack(bf_lo(w2.y), bf_hi(w2.y));
        } else {
          const uint32_t w1 = lds32(va);
          v2[0] = f2pack(bf_lo(w1), bf_hi(w1));
        }
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          const uint64_t pp = f2pack(pr[r][u], pr[r][u]);
#pragma unroll
          for (int c = 0; c < CP; ++c) o2[r][c] = ffma2(pp, v2[c], o2[r][c]);
        }
      }
    }
    __syncwarp();
    done = it + 1;
    // Stage st is free again: refill it with tile it + NST.
    if (lane == 0 && it + C::NST < nw) {
      fence_proxy_async_smem();
      issue(it + C::NST);
      issued = it + C::NST + 1;
    }
    __syncwarp();
  }
  if (!ok && lane == 0) {
    // Drain (bounded) the copies still in flight before the CTA exits.
    volatile int no_abort = 0;
    for (int it = done; it < issued; ++it)
      wait_bar(wbar + 8 * (it % C::NST), static_cast<uint32_t>(it / C::NST) & 1u, &no_abort,
               nullptr, 0, lim_cycles);
  }
  __syncwarp();

  // Warp state -> shared memory (over this warp's own stages, all consumed).
  float* mw = reinterpret_cast<float*>(smem + S::OFF_STAGES + warp * C::WARP_BYTES);
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    float ls = l_r[r];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    if (lane == 0) {
      mw[r * (D + 2)] = m_r[r];
      mw[r * (D + 2) + 1] = ls;
    }
#pragma unroll
    for (int c = 0; c < CP; ++c) {
      float y0, y1;
      f2unpack(o2[r][c], y0, y1);
      mw[r * (D + 2) + 2 + C::COLS * lane + 2 * c] = y0;
      mw[r * (D + 2) + 2 + C::COLS * lane + 2 * c + 1] = y1;
    }
  }
  __syncthreads();
  if (*abort_flag) return;

  // Merge the DW warp states; write this CTA's partial state in natural-log
  // units: partial index ((shard * nsplit + split) * n_q + qi) * heads + h.
  for (int i = tid; i < R * D; i += DW * 32) {
    const int r = i / D, x = i % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < DW; ++w) {
      const float* mr = reinterpret_cast<float*>(smem + S::OFF_STAGES + w * C::WARP_BYTES);
      mx = fmaxf(mx, mr[r * (D + 2)]);
    }
    const float mref = mx == -INFINITY ? 0.f : mx;
    float ov = 0.f, lv = 0.f;
#pragma unroll
    for (int w = 0; w < DW; ++w) {
      const float* mr = reinterpret_cast<float*>(smem + S::OFF_STAGES + w * C::WARP_BYTES);
      const float e = ex2(mr[r * (D + 2)] - mref);
      ov = fmaf(e, mr[r * (D + 2) + 2 + x], ov);
      lv = fmaf(e, mr[r * (D + 2) + 1], lv);
    }
    const long long qi = r / g;
    const int h = kh * g + r % g;
    const long long pidx =
        ((static_cast<long long>(shard) * a.nsplit + split) * a.n_q + qi) * a.heads + h;
    a.po[pidx * D + x] = ov;
    if (x == 0) {
      a.pm[pidx] = mx == -INFINITY ? -INFINITY : mx * kLn2;
      a.pl[pidx] = lv;
    }
  }
}

// Folds the nsplit partial states of each shard into that shard's running
// state (in place), one warp per (shard, query row, head).  The running
// state takes part as one more term, so a call adds to what was there.
template <int D>
__global__ void decode_combine_kernel(float* __restrict__ m, float* __restrict__ l,
                                      float* __restrict__ o, const float* __restrict__ pm,
                                      const float* __restrict__ pl, const float* __restrict__ po,
                                      long long rows_per_shard, int nsplit, long long n_rh) {
  const int lane = threadIdx.x & 31;
  const long long rh = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (rh >= n_rh) return;  // warp-uniform
  const long long shard = rh / rows_per_shard, row = rh % rows_per_shard;
  auto pidx = [&](int s) -> long long {
    return (shard * nsplit + s) * rows_per_shard + row;
  };
  // Max over the running state and every split, lanes striding the splits.
  const float m0 = m[rh];
  float mx = m0;
  for (int s = lane; s < nsplit; s += 32) mx = fmaxf(mx, pm[pidx(s)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (mx == -INFINITY) return;  // nothing allowed anywhere: the state stays as it is
  float lsum = 0.f;
  for (int s = lane; s < nsplit; s += 32) lsum += expf(pm[pidx(s)] - mx) * pl[pidx(s)];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
  const float e0 = expf(m0 - mx);  // m0 = -inf gives 0
  constexpr int CPL = D / 32;      // columns per lane
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = e0 * o[rh * D + CPL * lane + c];
  for (int s = 0; s < nsplit; ++s) {
    const float ms = pm[pidx(s)];
    if (ms == -INFINITY) continue;  // warp-uniform
    const float e = expf(ms - mx);
    const float* src = po + pidx(s) * D + CPL * lane;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = fmaf(e, src[c], acc[c]);
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) o[rh * D + CPL * lane + c] = acc[c];
  if (lane == 0) {
    l[rh] = e0 * l[rh] + lsum;
    m[rh] = mx;
  }
}

template <int D, int RM>
cudaError_t launch_split(const DecArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t st) {
  using S = DecSmem<D, RM>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, RM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.nsplit), static_cast<unsigned>(a.kv_heads),
            static_cast<unsigned>(a.nshard));
  decode_split_kernel<D, RM><<<grid, DW * 32, S::BYTES, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_split_d(const DecArgs& a, int rows, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st) {
  if (rows <= 4) return launch_split<D, 4>(a, tk, tv, st);
  if (rows <= 8) return launch_split<D, 8>(a, tk, tv, st);
  return launch_split<D, 16>(a, tk, tv, st);
}

}  // namespace

cudaError_t launch_decode_split(const DecArgs& a, int d, const CUtensorMap& tk,
                                const CUtensorMap& tv, cudaStream_t st) {
  const int rows = (a.heads / a.kv_heads) * static_cast<int>(a.n_q);
  return d == 128 ? launch_split_d<128>(a, rows, tk, tv, st) : launch_split_d<64>(a, rows, tk, tv, st);
}

cudaError_t launch_decode_combine(float* m, float* l, float* o, const float* pm, const float* pl,
                                  const float* po, long long rows_per_shard, int nsplit,
                                  int nshard, int d, cudaStream_t st) {
  const long long n_rh = rows_per_shard * nshard;
  if (n_rh == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (n_rh * 32 + threads - 1) / threads;
  if (d == 128)
    decode_combine_kernel<128><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        m, l, o, pm, pl, po, rows_per_shard, nsplit, n_rh);
  else
    decode_combine_kernel<64><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        m, l, o, pm, pl, po, rows_per_shard, nsplit, n_rh);
  return cudaGetLastError();
}

cudaError_t take_decode_status(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_decode_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(int));
}

}  // namespace ra
