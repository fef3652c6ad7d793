// Decode / short-query attention: a few query tokens against a long K/V
// history, the regime of "Ring Attention：把超长序列沿设备环流动", section
// "训练与推理的适用方式不同".  There a decode step has one new query per
// sequence but must read the whole cached K/V; instead of rotating K/V
// blocks, the query goes to every K/V shard, each shard computes a local
// attention state, and a global online-softmax reduction combines them.
//
// The work is HBM-bound: each K/V byte is read once and meets only the
// g * n_q query rows of its KV head (g = heads / kv_heads).  The layout is
// built around that read:
//   * decode_tc_kernel: a CTA takes one KV head and one chunk of one
//     shard's keys (split-K; the grid covers chunks x row tiles x KV heads
//     x shards, a few waves of the SMs).  The KV head's query rows sit in
//     128-row tiles (one for up to 128 rows, the usual case), so tcgen05
//     products give S = Q K^T and O += P V for a whole
//     128-key tile at a time; the unused rows of the tile cost tensor time,
//     which the pipe has to spare, not bytes.  It writes one partial state
//     (m, l, O~) per chunk.
//   * decode_combine_kernel folds a shard's chunk states into that shard's
//     running state, one warp per (shard, query row, head) (one shard's
//     partial state, ra_decode_partial).
//   * decode_reduce_kernel folds the chunk states of every shard and
//     finalizes, one CTA per (query row, head) (the whole decode,
//     ra_decode_forward): the global reduction of the merge operator and
//     the normalization in one launch.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {

__device__ int g_decode_status = 0;

namespace {

// ------------------------------------------------------------------ chunk kernel
// The KV head's g * n_q query rows are gathered into 128-row query tiles of
// tq = floor(128 / g) tokens each (a 3-D TMA box of g heads x tq tokens,
// row qi * g + hl; the rest of the tile is zero); a CTA takes one row tile
// and walks its key chunk in 128-key tiles with
// S = Q K^T and O += P V in TMEM and the online softmax of the forward
// kernel on one thread per row.  S is double-buffered in
// TMEM: the product S(k+2) runs while the softmax works on S(k), and the
// softmax waits for P V(k-1) before it touches O.  Roles (256 threads):
// warps 0-3 softmax, warp 4 TMA, warp 5 MMA issuer and TMEM owner.  Every
// wait is bounded.
namespace tc {

constexpr int BT = 128;
constexpr uint32_t CHB = 128 * 128;  // one 64-column swizzled chunk of a 128-row tile

template <int D>
struct TCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  // K/V stages (K and V of one tile each): QK runs two tiles ahead of P V.
  static constexpr int NST = D == 128 ? 3 : 4;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_ST = OFF_Q + TILE;   // stage s: K at OFF_ST + 2*s*TILE, V after
  static constexpr uint32_t OFF_BAR = OFF_ST + NST * 2 * TILE;
  static constexpr int B_Q = 0, B_F = 1, B_E = B_F + NST, B_S = B_E + NST,  // B_S: 2 buffers
                       B_P = B_S + 2, B_PV = B_P + 1, B_O = B_PV + 1, B_DRAIN = B_O + 1,
                       NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr uint32_t C_S = 0, C_O = 2 * BT;  // TMEM: S buffers 0, 1 (then P), O
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(C_O + D <= TMEM_COLS, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(256, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const DecArgs a) {
  using C = TCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = static_cast<int>(blockIdx.x) % a.nsplit;
  const int rt = static_cast<int>(blockIdx.x) / a.nsplit;  // row tile: tokens qa .. qa + qn - 1
  const int kh = blockIdx.y, shard = blockIdx.z;
  const int g = a.heads / a.kv_heads;
  const long long qa = static_cast<long long>(rt) * a.tq;
  const long long qn = a.tq < a.n_q - qa ? a.tq : a.n_q - qa;
  const int R = g * static_cast<int>(qn);
  const long long sh0 = static_cast<long long>(shard) * a.shard_len;
  const long long sh1 = sh0 + a.shard_len < a.n_kv ? sh0 + a.shard_len : a.n_kv;
  const long long c0 = sh0 + static_cast<long long>(split) * a.chunk;
  const long long c1 = c0 + a.chunk < sh1 ? c0 + a.chunk : sh1;
  const long long vb = valid_bound(a.mask);
  const PosMap km{kContiguous, 1, a.n_kv, 0, a.kv_off};
  // Allowed keys of query token qi, clipped to this CTA's chunk.
  auto keys_of = [&](long long qi, long long* lo, long long* hi) {
    *lo = c0;
    *hi = c0;
    const long long qp = a.q_off + qi;
    long long plo, phi;
    if (qp < vb && allowed_positions(a.mask, qp, &plo, &phi)) {
      const long long l = count_below(km, plo), h = count_below(km, phi);
      *lo = l > c0 ? l : c0;
      *hi = h < c1 ? h : c1;
      if (*hi < *lo) *hi = *lo;
    }
  };
  // Rows grow in position with r (r = qi * g + hl), so the first and last
  // query tokens bound the key range of the tile.
  long long lo0, hi0, lo1, hi1;
  keys_of(qa, &lo0, &hi0);
  keys_of(qa + qn - 1, &lo1, &hi1);
  const long long klo = lo0 < lo1 ? lo0 : lo1, khi = hi0 > hi1 ? hi0 : hi1;
  const long long kb = (klo / BT) * BT;
  const int n = khi > klo ? static_cast<int>((khi - kb + BT - 1) / BT) : 0;
  const long long lim = a.wait_limit;
  const long long pbase = (static_cast<long long>(shard) * a.nsplit + split) * a.n_q;
  if (n == 0) {
    // No key of this chunk is allowed: an empty partial state.
    for (int i = tid; i < R * D; i += 256) {
      const long long qi = qa + (i / D) / g;
      const int h = kh * g + (i / D) % g;
      const long long pidx = (pbase + qi) * a.heads + h;
      a.po[pidx * D + i % D] = 0.f;
      if (i % D == 0) {
        a.pm[pidx] = -INFINITY;
        a.pl[pidx] = 0.f;
      }
    }
    return;
  }
  // Zero the query tile: rows R..127 stay zero, rows 0..R-1 come by TMA.
  for (int i = tid; i < static_cast<int>(C::TILE / 16); i += 256)
    reinterpret_cast<uint4*>(smem + C::OFF_Q)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bar(i), i == C::B_P ? 128u : 1u);
    *abort_flag = *reinterpret_cast<volatile int*>(&g_decode_status) != 0 ? 1 : 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (*abort_flag) return;
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      // The box is g heads x tq tokens; tokens past n_q (a last partial
      // tile) are filled with zeros and counted like the rest.
      mbar_arrive_expect_tx(bar(C::B_Q),
                            static_cast<uint32_t>(g * a.tq) * 128u * C::NCH);
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_load_3d(sb + C::OFF_Q + ch * CHB, &tmQ, bar(C::B_Q), ch * 64, kh * g,
                    static_cast<int>(qa));
      int issued = 0;
      bool ok = true;
      for (int k = 0; k < n; ++k) {
        const int st = k % C::NST;
        if (k >= C::NST)
          ok = wait_bar(bar(C::B_E + st), (static_cast<uint32_t>(k / C::NST) & 1u) ^ 1u,
                        abort_flag, &g_decode_status, 0x71, lim);
        if (!ok) break;
        const uint32_t dst = sb + C::OFF_ST + st * 2 * C::TILE;
        const int krow = static_cast<int>(kb + static_cast<long long>(k) * BT);
        mbar_arrive_expect_tx(bar(C::B_F + st), 2 * C::TILE);
        for (int ch = 0; ch < C::NCH; ++ch) {
          tma_load_3d(dst + ch * CHB, &tmK, bar(C::B_F + st), ch * 64, kh, krow);
          tma_load_3d(dst + C::TILE + ch * CHB, &tmV, bar(C::B_F + st), ch * 64, kh, krow);
        }
        issued = k + 1;
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int k = issued > C::NST ? issued - C::NST : 0; k < issued; ++k)
          wait_bar(bar(C::B_F + k % C::NST), static_cast<uint32_t>(k / C::NST) & 1u, &no_abort,
                   nullptr, 0, lim);
        wait_bar(bar(C::B_Q), 0, &no_abort, nullptr, 0, lim);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t lead = lane == 0 ? 1u : 0u;
    constexpr uint32_t idesc_qk = idesc_bf16(BT, BT, 0);
    constexpr uint32_t idesc_pv = idesc_bf16(BT, D, 1);
    const uint64_t qdesc = sdesc_sw128(sb + C::OFF_Q, 16, 1024);
    // S(k) = Q K(k)^T into S buffer k % 2.
    auto qk = [&](int k) {
      const int st = k % C::NST;
      const uint32_t sbuf = tmem + C::C_S + static_cast<uint32_t>(k & 1) * BT;
      const uint64_t kd = sdesc_sw128(sb + C::OFF_ST + st * 2 * C::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = ((kk >> 2) * CHB + (kk & 3) * 32) >> 4;
        mma_ss_lead(lead, sbuf, qdesc + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
      }
      tc_commit_lead(lead, bar(C::B_S + (k & 1)));
    };
    auto wait_full = [&](int k) -> bool {
      return wait_bar(bar(C::B_F + k % C::NST), static_cast<uint32_t>(k / C::NST) & 1u,
                      abort_flag, &g_decode_status, 0x73, lim);
    };
    bool ok = wait_bar(bar(C::B_Q), 0, abort_flag, &g_decode_status, 0x72, lim);
    if (ok) ok = wait_full(0);
    if (ok) {
      tc_fence_after();
      qk(0);
      if (n > 1) {
        ok = wait_full(1);
        if (ok) {
          tc_fence_after();
          qk(1);
        }
      }
    }
    for (int k = 0; k < n && ok; ++k) {
      const int st = k % C::NST;
      ok = wait_bar(bar(C::B_P), static_cast<uint32_t>(k) & 1u, abort_flag, &g_decode_status,
                    0x74, lim);
      if (!ok) break;
      tc_fence_after();
      const uint64_t vd = sdesc_sw128(sb + C::OFF_ST + st * 2 * C::TILE + C::TILE, CHB, 1024);
      const uint32_t pbuf = tmem + C::C_S + static_cast<uint32_t>(k & 1) * BT;
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ts_lead(lead, tmem + C::C_O, pbuf + kk * 8,
                    vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, 1u);
      tc_commit_lead(lead, bar(C::B_E + st));
      tc_commit_lead(lead, bar(C::B_PV));
      if (k + 1 == n) tc_commit_lead(lead, bar(C::B_O));
      if (k + 2 < n) {
        ok = wait_full(k + 2);
        if (!ok) break;
        tc_fence_after();
        qk(k + 2);  // into buffer k % 2, in issue order after P V(k), which reads P(k) there
      }
    }
    volatile int no_abort = 0;
    tc_commit_lead(lead, bar(C::B_DRAIN));
    wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool valid = r < R;
    long long rlo = 0, rhi = 0;
    if (valid) keys_of(qa + r / g, &rlo, &rhi);
    const int row_lo = static_cast<int>(rlo - kb), row_hi = static_cast<int>(rhi - kb);
    {
      uint32_t z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_st32(tl + C::C_O + cc * 32, z);
      tmem_wait_st();
    }
    // Each thread's first arrival on B_P comes after its zeroed O row is in
    // TMEM, so the first P V accumulates onto zeros.
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    float m_used = -INFINITY, m_true = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int k = 0; k < n; ++k) {
      const uint32_t s_col = C::C_S + static_cast<uint32_t>(k & 1) * BT;
      ok = wait_bar(bar(C::B_S + (k & 1)), static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                    &g_decode_status, 0x75, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tl + s_col + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      const int lo_j = row_lo - k * BT, hi_j = row_hi - k * BT;
      if (lo_j > 0 || hi_j < BT) {
#pragma unroll
        for (int j = 0; j < BT; ++j)
          if (j < lo_j || j >= hi_j) sr[j >> 5][j & 31] = 0xff800000u;  // -inf
      }
#define RA_S(j) __uint_as_float(sr[(j) >> 5][(j) & 31])
      float mx0 = fmaxf(RA_S(0), RA_S(4)), mx1 = fmaxf(RA_S(1), RA_S(5));
      float mx2 = fmaxf(RA_S(2), RA_S(6)), mx3 = fmaxf(RA_S(3), RA_S(7));
#pragma unroll
      for (int j = 8; j < BT; j += 8) {
        mx0 = fmax3(mx0, RA_S(j + 0), RA_S(j + 4));
        mx1 = fmax3(mx1, RA_S(j + 1), RA_S(j + 5));
        mx2 = fmax3(mx2, RA_S(j + 2), RA_S(j + 6));
        mx3 = fmax3(mx3, RA_S(j + 3), RA_S(j + 7));
      }
      const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
      float alpha = 1.f;
      if (m_tile > m_true) {
        m_true = m_tile;
        alpha = ex2(m_used - m_true);  // m_used = -inf gives 0
        m_used = m_true;
      }
      // O is stable once P V(k-1) is done.  Wait for it on every tile (not
      // only when rescaling), so each phase of the barrier is waited in
      // order and a parity can never match a stale phase.
      if (k > 0) {
        ok = wait_bar(bar(C::B_PV), static_cast<uint32_t>(k - 1) & 1u, abort_flag,
                      &g_decode_status, 0x77, lim);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        const uint64_t al2 = f2pack(alpha, alpha);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tl + C::C_O + cc * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float y0, y1;
            f2unpack(fmul2(f2pack(__uint_as_float(o[j]), __uint_as_float(o[j + 1])), al2), y0, y1);
            o[j] = __float_as_uint(y0);
            o[j + 1] = __float_as_uint(y1);
          }
          tmem_st32(tl + C::C_O + cc * 32, o);
        }
      }
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      const uint64_t nm2 = f2pack(-mref, -mref);
      uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
      for (int j = 0; j < BT; j += 4) {
        float x0, x1, x2, x3;
        f2unpack(ffma2(f2pack(RA_S(j), RA_S(j + 1)), sl2x2, nm2), x0, x1);
        f2unpack(ffma2(f2pack(RA_S(j + 2), RA_S(j + 3)), sl2x2, nm2), x2, x3);
        const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
        acc0 = fadd2(acc0, f2pack(p0, p1));
        acc1 = fadd2(acc1, f2pack(p2, p3));
        sr[(j / 2) >> 5][(j / 2) & 31] = bf16x2_rn(p0, p1);
        sr[(j / 2 + 1) >> 5][(j / 2 + 1) & 31] = bf16x2_rn(p2, p3);
      }
#undef RA_S
      tmem_st32(tl + s_col, sr[0]);
      tmem_st32(tl + s_col + 32, sr[1]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_P));
      float sa, sbb;
      f2unpack(fadd2(acc0, acc1), sa, sbb);
      l_run = l_run * alpha + (sa + sbb);
    }
    if (ok) {
      ok = wait_bar(bar(C::B_O), 0u, abort_flag, &g_decode_status, 0x76, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      uint32_t o[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tl + C::C_O + cc * 32, o[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) reg_fence32(o[cc]);
      if (valid) {
        const long long pidx = (pbase + qa + r / g) * a.heads + kh * g + r % g;
        float4* dst = reinterpret_cast<float4*>(a.po + pidx * D);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[cc * 8 + j] = make_float4(__uint_as_float(o[cc][4 * j]), __uint_as_float(o[cc][4 * j + 1]),
                                          __uint_as_float(o[cc][4 * j + 2]),
                                          __uint_as_float(o[cc][4 * j + 3]));
        a.pm[pidx] = m_true == -INFINITY ? -INFINITY : m_true * kLn2;
        a.pl[pidx] = l_run;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace tc

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

// The global reduction and the finalize in one launch: for each (query row,
// head), the chunk partial states of every shard are folded with the
// online-softmax merge (one max, then the rescaled sums) and the result is
// normalized, out = O / l and lse = m + ln l (out = 0 and lse = -inf where
// no key is allowed).  One CTA per (row, head): its warps take every
// RW-th partial, lanes hold D / 32 columns each, and the warps' sums meet
// in shared memory.
constexpr int RW = 8;  // warps per CTA of the reduction
template <int D>
__global__ void __launch_bounds__(RW * 32)
decode_reduce_kernel(float* __restrict__ out, float* __restrict__ lse,
                     const float* __restrict__ pm, const float* __restrict__ pl,
                     const float* __restrict__ po, long long rows, int np) {
  constexpr int CPL = D / 32;  // columns per lane
  __shared__ float s_max[RW], s_l[RW];
  __shared__ __align__(16) float s_o[RW][D];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long rh = blockIdx.x;
  float mx = -INFINITY;
  for (int p = tid; p < np; p += RW * 32) mx = fmaxf(mx, pm[p * rows + rh]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_max[warp] = mx;
  __syncthreads();
  mx = s_max[0];
#pragma unroll
  for (int w = 1; w < RW; ++w) mx = fmaxf(mx, s_max[w]);
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  float lsum = 0.f;
  if (mx > -INFINITY) {
    for (int p = warp; p < np; p += RW) {
      const float ms = pm[p * rows + rh];
      if (ms == -INFINITY) continue;  // warp-uniform: an empty partial adds nothing
      const float e = expf(ms - mx);
      lsum = fmaf(e, pl[p * rows + rh], lsum);
      const float* src = po + (p * rows + rh) * D + CPL * lane;
      if constexpr (CPL == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(e, x.x, acc[0]);
        acc[1] = fmaf(e, x.y, acc[1]);
        acc[2] = fmaf(e, x.z, acc[2]);
        acc[3] = fmaf(e, x.w, acc[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(e, x.x, acc[0]);
        acc[1] = fmaf(e, x.y, acc[1]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) s_o[warp][CPL * lane + c] = acc[c];
  if (lane == 0) s_l[warp] = lsum;
  __syncthreads();
  float l = 0.f;
#pragma unroll
  for (int w = 0; w < RW; ++w) l += s_l[w];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int x = tid; x < D; x += RW * 32) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < RW; ++w) o += s_o[w][x];
    out[rh * D + x] = o * inv;
  }
  if (tid == 0) lse[rh] = l > 0.f ? mx + logf(l) : -INFINITY;
}

template <int D>
cudaError_t launch_tc_d(const DecArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, cudaStream_t st) {
  using C = tc::TCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.nsplit) * static_cast<unsigned>(a.ntile),
            static_cast<unsigned>(a.kv_heads), static_cast<unsigned>(a.nshard));
  tc::decode_tc_kernel<D><<<grid, 256, C::SMEM, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecArgs& a, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t st) {
  return d == 128 ? launch_tc_d<128>(a, tq, tk, tv, st) : launch_tc_d<64>(a, tq, tk, tv, st);
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

cudaError_t launch_decode_reduce(float* out, float* lse, const float* pm, const float* pl,
                                 const float* po, long long rows, int np, int d, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (d == 128)
    decode_reduce_kernel<128><<<static_cast<unsigned>(rows), RW * 32, 0, st>>>(out, lse, pm, pl,
                                                                               po, rows, np);
  else
    decode_reduce_kernel<64><<<static_cast<unsigned>(rows), RW * 32, 0, st>>>(out, lse, pm, pl,
                                                                             po, rows, np);
  return cudaGetLastError();
}

cudaError_t take_decode_status(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_decode_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(int));
}

}  // namespace ra
