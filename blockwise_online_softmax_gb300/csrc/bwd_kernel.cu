// Backward of the ring: gradients of O = softmax(S) V, S = Q K^T / sqrt(d),
// for one ring step of every virtual rank.  "Ring Attention：把超长序列沿
// 设备环流动", section "Backward 需要让梯度也沿环传播": every (Q block, K/V
// block) pair adds to dQ of the query block and to dK, dV of the K/V block
// (which travel with the block and arrive home fully summed), and the
// softmax is recomputed from the log-sum-exp saved by the forward, as the
// FlashAttention backward does.  Per pair, with P = exp(S - LSE),
// D = rowsum(dO * O):
//   dP = dO V^T,   dS = P * (dP - D) / sqrt(d),
//   dQ += dS K,    dK += dS^T Q,    dV += P^T dO.
//
// Two tcgen05 kernels and a pre-pass:
//   bwd_pre_kernel      D = rowsum(dO * O), one warp per (row, head).
//   bwd_dq_kernel<D>    Q-stationary: a CTA owns 128 query rows of one head
//                       and walks the K/V tiles they may see.  S and dP go
//                       to TMEM; the softmax warpgroup turns them into dS
//                       (bf16, written over S); dQ += dS K reads dS from
//                       TMEM.  S is double-buffered, so the softmax of one
//                       tile overlaps dQ of the previous tile and S of the
//                       next.  dQ stays in TMEM for the whole block.
//   bwd_dkdv_kernel<D>  K/V-stationary: a CTA owns 128 keys of one KV head
//                       and walks the query tiles, of every query head of
//                       its group, that may see them.  S^T - lse sqrt(d)
//                       and dP^T - D go to TMEM (the per-query terms enter
//                       as one extra K-step of each product); the softmax
//                       warpgroup writes P^T over S^T and dS^T over dP^T,
//                       32 queries at a time, and dV += P^T dO and
//                       dK += dS^T Q read each chunk from TMEM as soon as
//                       it is written.  No atomics: in one launch each K/V
//                       block belongs to one rank, each key tile to one CTA.
// The accumulators (dQ, dK, dV, fp32) live in HBM between ring steps, like
// the forward's (m, l, O~) state.  Masks and layouts are the forward's: a
// per-row interval of allowed key rows.
//
// Roles (256 threads): warps 0-3 the softmax warpgroup (one thread per
// TMEM lane), warp 4 the TMA producer (K ring in the dQ kernel), warp 5 the
// MMA issuer (it also owns the TMEM allocation), warp 6 the V producer of
// the dQ kernel.  Every wait is bounded.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {

__device__ int g_bwd_status = 0;

namespace {

constexpr int BT = 128;              // rows of every tile (TMEM lanes, keys or queries)
constexpr int NTH = 256;
constexpr uint32_t CHB = 128 * 128;  // one 64-column swizzled chunk of a 128-row tile
constexpr uint32_t TMEM_COLS = 512;

template <int D>
struct BCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr int NST = 2;  // stages of the streamed operand pair
  // Augmentation tiles: 128 rows x 16 bf16 (one K-step), K-major without
  // swizzle: element (r, k) at (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16
  // + (k % 8) * 2, i.e. 8x16-byte core matrices, LBO 128 (along K), SBO 256
  // (along rows).
  static constexpr uint32_t AUG = BT * 32;
  // shared memory: K and V resident, NST stages of (Q, dO), the ones tile,
  // NST stages of (lse, D) augmentation tiles, per-query key intervals
  static constexpr uint32_t OFF_R0 = 0;
  static constexpr uint32_t OFF_R1 = OFF_R0 + TILE;
  static constexpr uint32_t OFF_ST = OFF_R1 + TILE;  // stage s: tiles at OFF_ST + s*2*TILE
  static constexpr uint32_t OFF_ONES = OFF_ST + NST * 2 * TILE;
  static constexpr uint32_t OFF_AUG = OFF_ONES + AUG;      // stage s: lse at +s*2*AUG, D at +AUG
  // int2 [3][BT]: three buffers, since the tile after next is staged while
  // a lagging warp may still read the previous tile's intervals.
  static constexpr uint32_t OFF_LM = OFF_AUG + NST * 2 * AUG;
  static constexpr uint32_t OFF_BAR = OFF_LM + 3 * BT * 8;
  static constexpr int B_R = 0;             // resident tiles loaded
  static constexpr int B_F = 1;             // NST: stage full
  static constexpr int B_E = B_F + NST;     // NST: stage free
  // 2: augmentation tiles of tile it written (128 arrivals), alternating by
  // the parity of it: the softmax warps stage one tile ahead, so one
  // barrier could complete two phases before the MMA thread waits for the
  // first of them.
  static constexpr int B_A = B_E + NST;
  static constexpr int B_S = B_A + 2;       // S^T and dP^T done
  static constexpr int NPC = BT / 32;       // softmax chunks of 32 queries
  static constexpr int B_P = B_S + 1;       // NPC: chunk c of P^T, dS^T in TMEM (128 arrivals)
  static constexpr int B_O = B_P + NPC;     // last accumulating MMA done
  static constexpr int B_DRAIN = B_O + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr uint32_t C_S = 0;       // S^T (then P^T, bf16 pairs)
  static constexpr uint32_t C_DP = BT;     // dP^T (then dS^T, bf16 pairs)
  static constexpr uint32_t C_A0 = 2 * BT; // dV
  static constexpr uint32_t C_A1 = 2 * BT + D;  // dK
  static_assert(C_A1 + D <= TMEM_COLS, "TMEM budget");
};

// Descriptor of a K-major tile without swizzle (see BCfg::AUG).
__device__ __forceinline__ uint64_t sdesc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version; swizzle field (61..63) = 0: none
  return d;
}

// v as the sum of three bf16 (a + b + c within ~2^-24 |v|), packed for
// row elements k = 0, 1 (first word) and 2 (second word).
__device__ __forceinline__ uint2 bf16_split3(float v) {
  const __nv_bfloat16 a = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(a);
  const __nv_bfloat16 b = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b);
  const __nv_bfloat16 c = __float2bfloat16_rn(r2);
  return make_uint2(static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16),
                    static_cast<uint32_t>(__bfloat16_as_ushort(c)));
}

// ------------------------------------------------------------------ shared pieces
// S-like tile product: D[tmem] = A B^T over d, both operands K-major in
// shared memory (128 rows x d, 128-byte swizzle).
template <int D>
__device__ __forceinline__ void mma_rows(uint32_t lead, uint32_t d_tmem, uint64_t adesc,
                                         uint64_t bdesc) {
  constexpr uint32_t idesc = idesc_bf16(BT, BT, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = ((kk >> 2) * CHB + (kk & 3) * 32) >> 4;
    mma_ss_lead(lead, d_tmem, adesc + off, bdesc + off, idesc, kk > 0 ? 1u : 0u);
  }
}
// Accumulating product: D[tmem] += A[tmem, bf16 pairs, 128 x 128] B, with B
// a 128-row tile used MN-major (its d columns are the N extent).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t lead, uint32_t d_tmem, uint32_t a_tmem,
                                        uint64_t bdesc_mn) {
  constexpr uint32_t idesc = idesc_bf16(BT, D, 1);
#pragma unroll
  for (int kk = 0; kk < BT / 16; ++kk)
    mma_ts_lead(lead, d_tmem, a_tmem + kk * 8, bdesc_mn + static_cast<uint64_t>((kk * 2048) >> 4),
                idesc, 1u);
}

// The same, over the 32 rows of B (two K-steps) starting at step kk0.
template <int D>
__device__ __forceinline__ void mma_acc_part(uint32_t lead, uint32_t d_tmem, uint32_t a_tmem,
                                             uint64_t bdesc_mn, int kk0) {
  constexpr uint32_t idesc = idesc_bf16(BT, D, 1);
#pragma unroll
  for (int kk = kk0; kk < kk0 + 2; ++kk)
    mma_ts_lead(lead, d_tmem, a_tmem + kk * 8, bdesc_mn + static_cast<uint64_t>((kk * 2048) >> 4),
                idesc, 1u);
}

__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int nch,
                                          int head, int row) {
  for (int ch = 0; ch < nch; ++ch) tma_load_3d(dst + ch * CHB, tm, bar, ch * 64, head, row);
}

// fp32 accumulator rows HBM <-> TMEM (one row per thread, d columns).
template <int D>
__device__ __forceinline__ void acc_to_tmem(uint32_t taddr, const float* src, bool valid) {
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t r[32];
    if (valid) {
      const float4* s4 = reinterpret_cast<const float4*>(src + cc * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = s4[j];
        r[4 * j] = __float_as_uint(x.x);
        r[4 * j + 1] = __float_as_uint(x.y);
        r[4 * j + 2] = __float_as_uint(x.z);
        r[4 * j + 3] = __float_as_uint(x.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    }
    tmem_st32(taddr + cc * 32, r);
  }
}
template <int D>
__device__ __forceinline__ void tmem_to_acc(uint32_t taddr, float* dst, bool valid) {
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t r[32];
    tmem_ld32(taddr + cc * 32, r);
    tmem_wait_ld();
    reg_fence32(r);
    if (valid) {
      float4* d4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        d4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    }
  }
}

// Rows r of the query block (valid prefix [0, nvr)) whose key interval
// meets key rows [k0, k1): both interval ends grow with r, so that is one
// range [*ra, *rb), found by two binary searches.
__device__ __forceinline__ void query_range(const FwdArgs& a, const Work& wk, long long k0,
                                            long long k1, long long vb, long long* ra,
                                            long long* rb) {
  const long long nvr = count_below(wk.qmap, vb) < wk.qmap.c ? count_below(wk.qmap, vb) : wk.qmap.c;
  long long lo = 0, hi = nvr;  // first r with hi_r > k0
  while (lo < hi) {
    const long long mid = (lo + hi) >> 1;
    long long l, h;
    row_keys(a, wk, mid, vb, &l, &h);
    if (h > k0) hi = mid; else lo = mid + 1;
  }
  *ra = lo;
  lo = *ra;
  hi = nvr;  // first r with lo_r >= k1
  while (lo < hi) {
    const long long mid = (lo + hi) >> 1;
    long long l, h;
    row_keys(a, wk, mid, vb, &l, &h);
    if (l >= k1) hi = mid; else lo = mid + 1;
  }
  *rb = lo;
}

__global__ void bwd_pre_kernel(const float* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                               float* __restrict__ dvec, long long n_rh, int d) {
  const int lane = threadIdx.x & 31;
  const long long rh = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (rh >= n_rh) return;
  float acc = 0.f;
  for (int x = lane; x < d; x += 32)
    acc = fmaf(out[rh * d + x], __bfloat162float(dout[rh * d + x]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dvec[rh] = acc;
}

// ------------------------------------------------------------------ dQ kernel
// Shared memory and TMEM of the dQ kernel.  S is double-buffered in TMEM so
// that the softmax warps work on tile k while the tensor pipe runs
// dQ += dS(k-1) K(k-1) and S(k+1) = Q K(k+1)^T.  K and V stream through
// separate rings: K(k) is read by S(k) and by dQ(k), V(k) only by dP(k).
template <int D>
struct QCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr int NSK = (D == 64) ? 4 : 3;
  static constexpr int NSV = 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_O = OFF_Q + TILE;
  static constexpr uint32_t OFF_K = OFF_O + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE;
  static constexpr int B_R = 0;            // Q and dO loaded
  static constexpr int B_KF = 1;           // NSK: K stage full
  static constexpr int B_KE = B_KF + NSK;  // NSK: K stage free
  static constexpr int B_VF = B_KE + NSK;  // NSV: V stage full
  static constexpr int B_VE = B_VF + NSV;  // NSV: V stage free
  static constexpr int B_S = B_VE + NSV;   // S(k) and dP(k) done
  static constexpr int B_P = B_S + 1;      // dS(k) in TMEM (128 arrivals)
  static constexpr int B_O = B_P + 1;      // last dQ product done
  static constexpr int B_DRAIN = B_O + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns: S buffers (dS written over them as bf16 pairs), dP, dQ.
  static constexpr uint32_t C_S0 = 0;
  static constexpr uint32_t C_DP = BT;
  static constexpr uint32_t C_A = 2 * BT;
  static constexpr uint32_t C_S1 = 2 * BT + D;
  static_assert(C_S1 + BT <= TMEM_COLS, "TMEM budget");
};

// Streams tiles 0..n-1 of a K or V ring (rows kv_base + (t0 + k) * BT) into
// NS shared-memory stages.  Returns false on an abort, after draining
// (bounded) the copies still in flight.
template <int NS>
__device__ __forceinline__ bool produce_ring(const CUtensorMap* tm, uint32_t base, uint32_t tile,
                                             int nch, uint32_t b_full, uint32_t b_empty,
                                             int head, long long row0, int n,
                                             volatile int* abort_flag, int code, long long lim) {
  int issued = 0;
  bool ok = true;
  for (int k = 0; k < n; ++k) {
    const int st = k % NS;
    if (k >= NS)
      ok = wait_bar(b_empty + 8u * st, (static_cast<uint32_t>(k / NS) & 1u) ^ 1u, abort_flag,
                    &g_bwd_status, code, lim);
    if (!ok) break;
    mbar_arrive_expect_tx(b_full + 8u * st, tile);
    load_tile(base + st * tile, tm, b_full + 8u * st, nch, head,
              static_cast<int>(row0 + static_cast<long long>(k) * BT));
    issued = k + 1;
  }
  if (!ok) {
    volatile int no_abort = 0;
    for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
      wait_bar(b_full + 8u * (k % NS), static_cast<uint32_t>(k / NS) & 1u, &no_abort, nullptr, 0,
               lim);
  }
  return ok;
}

template <int D>
__global__ void __launch_bounds__(NTH, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const BwdArgs b) {
  using C = QCfg<D>;
  const FwdArgs& a = b.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, kh = h / (a.heads / a.kv_heads);
  const Work wk = decode_work(a, blockIdx.z);
  const long long row0 = static_cast<long long>(blockIdx.x) * BT;
  const long long vb = valid_bound(a.mask);
  int t0, t1;
  tile_range(a, wk, row0, row0 + BT, vb, BT, &t0, &t1);
  const int n = t1 - t0;
  if (n <= 0) return;  // these rows see no key of the block: dQ unchanged
  const long long lim = a.wait_limit;

  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bar(i), i == C::B_P ? 128u : 1u);
    *abort_flag = *reinterpret_cast<volatile int*>(&g_bwd_status) != 0 ? 1 : 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (*abort_flag) return;
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ = sb + C::OFF_Q, sO = sb + C::OFF_O;
  const long long krow0 = wk.kv_base + static_cast<long long>(t0) * BT;

  if (warp == 4) {
    // ---------------------------------------------------------------- K producer (and Q, dO)
    if (lane == 0) {
      const int qrow = static_cast<int>(wk.q_base + row0);
      mbar_arrive_expect_tx(bar(C::B_R), 2 * C::TILE);
      load_tile(sQ, &tmQ, bar(C::B_R), C::NCH, h, qrow);
      load_tile(sO, &tmO, bar(C::B_R), C::NCH, h, qrow);
      if (!produce_ring<C::NSK>(&tmK, sb + C::OFF_K, C::TILE, C::NCH, bar(C::B_KF), bar(C::B_KE),
                                kh, krow0, n, abort_flag, 0x51, lim)) {
        volatile int no_abort = 0;
        wait_bar(bar(C::B_R), 0, &no_abort, nullptr, 0, lim);
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ---------------------------------------------------------------- V producer
    if (lane == 0)
      produce_ring<C::NSV>(&tmV, sb + C::OFF_V, C::TILE, C::NCH, bar(C::B_VF), bar(C::B_VE), kh,
                           krow0, n, abort_flag, 0x57, lim);
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    // Order: S(0), dP(0); S(1); then per tile k, once dS(k) is in TMEM:
    // dP(k+1), dQ += dS(k) K(k), S(k+2).  The softmax of tile k+1 needs only
    // dP(k+1) after dS(k): it overlaps dQ(k) and S(k+2).  S(k+2) overwrites
    // the buffer dQ(k) reads; the tensor pipe runs them in issue order.
    const uint32_t lead = lane == 0 ? 1u : 0u;
    const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
    const uint64_t odesc = sdesc_sw128(sO, 16, 1024);
    auto k_st = [&](int k) { return sb + C::OFF_K + static_cast<uint32_t>(k % C::NSK) * C::TILE; };
    auto v_st = [&](int k) { return sb + C::OFF_V + static_cast<uint32_t>(k % C::NSV) * C::TILE; };
    auto s_col = [&](int k) { return (k & 1) ? C::C_S1 : C::C_S0; };
    auto wait_k = [&](int k) {
      return wait_bar(bar(C::B_KF + k % C::NSK), static_cast<uint32_t>(k / C::NSK) & 1u,
                      abort_flag, &g_bwd_status, 0x53, lim);
    };
    auto wait_v = [&](int k) {
      return wait_bar(bar(C::B_VF + k % C::NSV), static_cast<uint32_t>(k / C::NSV) & 1u,
                      abort_flag, &g_bwd_status, 0x58, lim);
    };
    bool ok = wait_bar(bar(C::B_R), 0, abort_flag, &g_bwd_status, 0x52, lim);
    if (ok) ok = wait_k(0);
    if (ok) ok = wait_v(0);
    if (ok) {
      tc_fence_after();
      mma_rows<D>(lead, tmem + C::C_S0, qdesc, sdesc_sw128(k_st(0), 16, 1024));  // S = Q K^T
      mma_rows<D>(lead, tmem + C::C_DP, odesc, sdesc_sw128(v_st(0), 16, 1024));  // dP = dO V^T
      tc_commit_lead(lead, bar(C::B_S));
      tc_commit_lead(lead, bar(C::B_VE));
    }
    if (ok && n > 1) {
      ok = wait_k(1);
      if (ok) mma_rows<D>(lead, tmem + C::C_S1, qdesc, sdesc_sw128(k_st(1), 16, 1024));
    }
    for (int k = 0; k < n && ok; ++k) {
      ok = wait_bar(bar(C::B_P), static_cast<uint32_t>(k) & 1u, abort_flag, &g_bwd_status, 0x54,
                    lim);
      if (!ok) break;
      tc_fence_after();
      if (k + 1 < n) {
        ok = wait_v(k + 1);
        if (!ok) break;
        mma_rows<D>(lead, tmem + C::C_DP, odesc, sdesc_sw128(v_st(k + 1), 16, 1024));
        tc_commit_lead(lead, bar(C::B_S));  // covers S(k+1), issued earlier
        tc_commit_lead(lead, bar(C::B_VE + (k + 1) % C::NSV));
      }
      mma_acc<D>(lead, tmem + C::C_A, tmem + s_col(k), sdesc_sw128(k_st(k), CHB, 1024));  // dQ += dS K
      tc_commit_lead(lead, bar(C::B_KE + k % C::NSK));
      if (k + 1 == n) tc_commit_lead(lead, bar(C::B_O));
      if (k + 2 < n) {
        ok = wait_k(k + 2);
        if (!ok) break;
        mma_rows<D>(lead, tmem + s_col(k), qdesc, sdesc_sw128(k_st(k + 2), 16, 1024));
      }
    }
    volatile int no_abort = 0;
    tc_commit_lead(lead, bar(C::B_DRAIN));
    wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int row = warp * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const long long grow = row0 + row;
    const bool valid = grow < a.cq;
    const long long sidx = (wk.state_base + grow) * a.heads + h;
    float lse2 = -INFINITY, dr = 0.f;
    int row_lo = 0, row_hi = 0;
    if (valid) {
      lse2 = b.lse[sidx] * kLog2e;
      dr = b.dvec[sidx];
      long long lo, hi;
      row_keys(a, wk, grow, vb, &lo, &hi);
      row_lo = static_cast<int>(lo);
      row_hi = static_cast<int>(hi);
    }
    acc_to_tmem<D>(tl + C::C_A, b.dq + sidx * D, valid);
    tmem_wait_st();
    // Key tiles full_0 .. full_0 + n_full - 1 lie wholly inside the row's
    // interval and need no mask (one unsigned compare decides).
    const int full_0 = (row_lo + BT - 1) / BT;
    const int n_full = row_hi / BT - full_0 > 0 ? row_hi / BT - full_0 : 0;
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    // dS = P * (dP * scale - D * scale): one FFMA2 and one FMUL2 per pair.
    const uint64_t nlse2 = f2pack(-lse2, -lse2), ndr2 = f2pack(-dr * a.scale, -dr * a.scale);
    const uint64_t scx2 = f2pack(a.scale, a.scale);
    bool ok = true;
    for (int k = 0; k < n; ++k) {
      ok = wait_bar(bar(C::B_S), static_cast<uint32_t>(k) & 1u, abort_flag, &g_bwd_status, 0x55,
                    lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int t = t0 + k;
      const bool masked = static_cast<unsigned>(t - full_0) >= static_cast<unsigned>(n_full);
      const int lo_j = row_lo - t * BT, hi_j = row_hi - t * BT;
      const uint32_t cs = tl + ((k & 1) ? C::C_S1 : C::C_S0);
#pragma unroll
      for (int c = 0; c < BT / 32; ++c) {
        uint32_t s[32], dp[32], w[16];
        tmem_ld32(cs + c * 32, s);
        tmem_ld32(tl + C::C_DP + c * 32, dp);
        tmem_wait_ld();
        reg_fence32(s);
        reg_fence32(dp);
        // Three branch-free passes (exponentials, mask, dS), so the 16
        // column pairs of a pass are independent chains in one block.
        float p[32];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float x0, x1;
          f2unpack(ffma2(f2pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), sl2x2, nlse2),
                   x0, x1);
          p[j] = ex2(x0);
          p[j + 1] = ex2(x1);
        }
        if (masked) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (!(c * 32 + j >= lo_j && c * 32 + j < hi_j)) p[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint64_t t2 =
              ffma2(f2pack(__uint_as_float(dp[j]), __uint_as_float(dp[j + 1])), scx2, ndr2);
          float d0, d1;
          f2unpack(fmul2(f2pack(p[j], p[j + 1]), t2), d0, d1);
          w[j / 2] = bf16x2_rn(d0, d1);
        }
        // dS pairs over columns [16c, 16c + 16) of the S buffer: already read.
        tmem_st16(cs + c * 16, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_P));
    }
    if (ok) {
      ok = wait_bar(bar(C::B_O), 0u, abort_flag, &g_bwd_status, 0x56, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      tmem_to_acc<D>(tl + C::C_A, b.dq + sidx * D, valid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dK/dV kernel
// The per-query terms enter the products: S^T and dP^T each get one more
// K-step, a ones column block of the keys against three bf16 terms of
// -lse * sqrt(d) (resp. -D) per query, so TMEM holds S^T - lse * sqrt(d)
// and dP^T - D.  The softmax warps then need no per-query data for full
// tiles: P = 2^(x * log2(e) / sqrt(d)) and dS = P * (y / sqrt(d)).
template <int D>
__global__ void __launch_bounds__(NTH, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                const BwdArgs b) {
  using C = BCfg<D>;
  const FwdArgs& a = b.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kh = blockIdx.y, g = a.heads / a.kv_heads;
  const Work wk = decode_work(a, blockIdx.z);
  const long long k0 = static_cast<long long>(blockIdx.x) * BT;
  const long long k1 = k0 + BT < a.ck ? k0 + BT : a.ck;
  const long long vb = valid_bound(a.mask);
  long long ra, rb;
  query_range(a, wk, k0, k1, vb, &ra, &rb);
  const int qt0 = static_cast<int>(ra / BT);
  const int nq = rb > ra ? static_cast<int>((rb + BT - 1) / BT) - qt0 : 0;
  const int n = nq * g;  // iterations: query heads of the group x query tiles
  if (n <= 0) return;    // no query sees these keys: dK, dV unchanged
  const long long lim = a.wait_limit;

  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i)
      mbar_init(bar(i), ((i >= C::B_P && i < C::B_P + C::NPC) || i == C::B_A || i == C::B_A + 1)
                            ? 128u
                            : 1u);
    *abort_flag = *reinterpret_cast<volatile int*>(&g_bwd_status) != 0 ? 1 : 0;
    fence_mbar_init();
  }
  // Augmentation tiles: zero everywhere; the ones tile has 1 at k = 0, 1, 2
  // of every row (k < 8 lies in the first core matrix of each row).
  for (uint32_t off = static_cast<uint32_t>(tid) * 16; off < (1 + 2 * C::NST) * C::AUG;
       off += NTH * 16)
    *reinterpret_cast<uint4*>(smem + C::OFF_ONES + off) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (tid < BT)
    *reinterpret_cast<uint2*>(smem + C::OFF_ONES + (tid >> 3) * 256 + (tid & 7) * 16) =
        make_uint2(0x3F803F80u, 0x00003F80u);
  fence_proxy_async_smem();
  __syncthreads();
  if (*abort_flag) return;
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sK = sb + C::OFF_R0, sV = sb + C::OFF_R1;
  auto it_head = [&](int it) { return kh * g + it / nq; };
  auto it_row = [&](int it) { return static_cast<long long>(qt0 + it % nq) * BT; };

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const int krow = static_cast<int>(wk.kv_base + k0);
      mbar_arrive_expect_tx(bar(C::B_R), 2 * C::TILE);
      load_tile(sK, &tmK, bar(C::B_R), C::NCH, kh, krow);
      load_tile(sV, &tmV, bar(C::B_R), C::NCH, kh, krow);
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n; ++it) {
        const int st = it % C::NST;
        if (it >= C::NST)
          ok = wait_bar(bar(C::B_E + st), (static_cast<uint32_t>(it / C::NST) & 1u) ^ 1u,
                        abort_flag, &g_bwd_status, 0x61, lim);
        if (!ok) break;
        const uint32_t dst = sb + C::OFF_ST + st * 2 * C::TILE;
        const int qrow = static_cast<int>(wk.q_base + it_row(it));
        mbar_arrive_expect_tx(bar(C::B_F + st), 2 * C::TILE);
        load_tile(dst, &tmQ, bar(C::B_F + st), C::NCH, it_head(it), qrow);
        load_tile(dst + C::TILE, &tmO, bar(C::B_F + st), C::NCH, it_head(it), qrow);
        issued = it + 1;
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int it = issued > C::NST ? issued - C::NST : 0; it < issued; ++it)
          wait_bar(bar(C::B_F + it % C::NST), static_cast<uint32_t>(it / C::NST) & 1u, &no_abort,
                   nullptr, 0, lim);
        wait_bar(bar(C::B_R), 0, &no_abort, nullptr, 0, lim);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t lead = lane == 0 ? 1u : 0u;
    constexpr uint32_t idesc_s = idesc_bf16(BT, BT, 0);
    const uint64_t kdesc = sdesc_sw128(sK, 16, 1024);
    const uint64_t vdesc = sdesc_sw128(sV, 16, 1024);
    const uint64_t ones = sdesc_noswz(sb + C::OFF_ONES, 128, 256);
    bool ok = wait_bar(bar(C::B_R), 0, abort_flag, &g_bwd_status, 0x62, lim);
    for (int it = 0; it < n && ok; ++it) {
      const int st = it % C::NST;
      ok = wait_bar(bar(C::B_F + st), static_cast<uint32_t>(it / C::NST) & 1u, abort_flag,
                    &g_bwd_status, 0x63, lim);
      if (ok)
        ok = wait_bar(bar(C::B_A + (it & 1)), static_cast<uint32_t>(it >> 1) & 1u, abort_flag,
                      &g_bwd_status, 0x67, lim);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sQ = sb + C::OFF_ST + st * 2 * C::TILE;
      const uint32_t sO = sQ + C::TILE;
      const uint32_t sA = sb + C::OFF_AUG + st * 2 * C::AUG;
      mma_rows<D>(lead, tmem + C::C_S, kdesc, sdesc_sw128(sQ, 16, 1024));   // S^T = K Q^T
      mma_ss_lead(lead, tmem + C::C_S, ones, sdesc_noswz(sA, 128, 256), idesc_s, 1u);  // - lse sqrt(d)
      mma_rows<D>(lead, tmem + C::C_DP, vdesc, sdesc_sw128(sO, 16, 1024));  // dP^T = V dO^T
      mma_ss_lead(lead, tmem + C::C_DP, ones, sdesc_noswz(sA + C::AUG, 128, 256), idesc_s, 1u);  // - D
      tc_commit_lead(lead, bar(C::B_S));
      // dV += P^T dO and dK += dS^T Q, one 32-query chunk at a time as the
      // softmax warps publish it, so these products overlap their later
      // chunks.
      const uint64_t odesc_mn = sdesc_sw128(sO, CHB, 1024);
      const uint64_t qdesc_mn = sdesc_sw128(sQ, CHB, 1024);
#pragma unroll
      for (int c = 0; c < C::NPC; ++c) {
        ok = wait_bar(bar(C::B_P + c), static_cast<uint32_t>(it) & 1u, abort_flag, &g_bwd_status,
                      0x64, lim);
        if (!ok) break;
        tc_fence_after();
        mma_acc_part<D>(lead, tmem + C::C_A0, tmem + C::C_S, odesc_mn, 2 * c);   // dV
        mma_acc_part<D>(lead, tmem + C::C_A1, tmem + C::C_DP, qdesc_mn, 2 * c);  // dK
      }
      if (!ok) break;
      tc_commit_lead(lead, bar(C::B_E + st));
      if (it + 1 == n) tc_commit_lead(lead, bar(C::B_O));
    }
    volatile int no_abort = 0;
    tc_commit_lead(lead, bar(C::B_DRAIN));
    wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int t = warp * 32 + lane;  // key row of the tile = TMEM lane; query t when staging
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const long long kidx = k0 + t;
    const bool kvalid = kidx < a.ck;
    const long long kst = (wk.kv_base + kidx) * a.kv_heads + kh;
    acc_to_tmem<D>(tl + C::C_A0, b.dv + kst * D, kvalid);
    acc_to_tmem<D>(tl + C::C_A1, b.dk + kst * D, kvalid);
    tmem_wait_st();
    int2* lmt = reinterpret_cast<int2*>(smem + C::OFF_LM);
    // Stages query t of tile `it`: its -lse * sqrt(d) and -D as three bf16
    // terms into the augmentation tiles of stage it % NST, and its allowed
    // key rows [lo, hi) for the mask.  Returns whether the query sees every
    // key of this key tile.  Queries with no allowed key (or past the
    // block) get zero terms; the mask covers them.
    auto stage = [&](int it) -> bool {
      const long long r = it_row(it) + t;
      float vl = 0.f, vd = 0.f;
      int lo = 0, hi = 0;
      if (r < a.cq) {
        const long long qi = (wk.state_base + r) * a.heads + it_head(it);
        const float lse = b.lse[qi];
        if (lse > -INFINITY) vl = -lse / a.scale;
        vd = -b.dvec[qi];
        long long l, h;
        row_keys(a, wk, r, vb, &l, &h);
        lo = static_cast<int>(l);
        hi = static_cast<int>(h);
      }
      uint8_t* aug = smem + C::OFF_AUG + (it % C::NST) * 2 * C::AUG + (t >> 3) * 256 + (t & 7) * 16;
      *reinterpret_cast<uint2*>(aug) = bf16_split3(vl);
      *reinterpret_cast<uint2*>(aug + C::AUG) = bf16_split3(vd);
      lmt[(it % 3) * BT + t] = make_int2(lo, hi);
      return r < a.cq && lo <= k0 && hi >= k0 + BT && k0 + BT <= a.ck;
    };
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2), scx2 = f2pack(a.scale, a.scale);
    // Tile 0 is staged here; tile it + 1 while the products of tile it run.
    // The augmentation stage of tile it + 1 was last read by the products
    // of tile it - 1, which finished before this group read their results.
    // Every softmax thread passes named barrier 2 once per tile, aborted or
    // not, so the warps are at most one tile apart.
    bool full = named_bar_and(2, 128, stage(0));
    fence_proxy_async_smem();
    mbar_arrive(bar(C::B_A));  // tile 0: barrier B_A + 0, phase 0
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      bool full_next = false;
      if (it + 1 < n) {
        full_next = named_bar_and(2, 128, stage(it + 1));
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_A + ((it + 1) & 1)));
      }
      if (ok) {
        ok = wait_bar(bar(C::B_S), static_cast<uint32_t>(it) & 1u, abort_flag, &g_bwd_status,
                      0x65, lim);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        const int2* lb = lmt + (it % 3) * BT;
        // Rolled: the chunk loop body is large, and one copy keeps the
        // softmax warps' code in the instruction cache.
#pragma unroll 1
        for (int c = 0; c < BT / 32; ++c) {
          uint32_t s[32], dp[32], wp[16], wd[16];
          tmem_ld32(tl + C::C_S + c * 32, s);
          tmem_ld32(tl + C::C_DP + c * 32, dp);
          tmem_wait_ld();
          reg_fence32(s);
          reg_fence32(dp);
          // Three branch-free passes (exponentials, mask, dS), so the 16
          // column pairs of a pass are independent chains in one block.
          float p[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float x0, x1;
            f2unpack(fmul2(f2pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), sl2x2), x0,
                     x1);
            p[j] = ex2(x0);
            p[j + 1] = ex2(x1);
          }
          if (!full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int2 m = lb[c * 32 + j];
              if (!(kvalid && kidx >= m.x && kidx < m.y)) p[j] = 0.f;
            }
          }
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const uint64_t t2 =
                fmul2(f2pack(__uint_as_float(dp[j]), __uint_as_float(dp[j + 1])), scx2);
            float d0, d1;
            f2unpack(fmul2(f2pack(p[j], p[j + 1]), t2), d0, d1);
            wp[j / 2] = bf16x2_rn(p[j], p[j + 1]);
            wd[j / 2] = bf16x2_rn(d0, d1);
          }
          tmem_st16(tl + C::C_S + c * 16, wp);   // P^T pairs over read S^T columns
          tmem_st16(tl + C::C_DP + c * 16, wd);  // dS^T pairs over read dP^T columns
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_P + c));
        }
      }
      full = full_next;
    }
    if (ok) {
      ok = wait_bar(bar(C::B_O), 0u, abort_flag, &g_bwd_status, 0x66, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      tmem_to_acc<D>(tl + C::C_A0, b.dv + kst * D, kvalid);
      tmem_to_acc<D>(tl + C::C_A1, b.dk + kst * D, kvalid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_dq_d(const BwdArgs& b, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  using C = QCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((b.f.cq + BT - 1) / BT), b.f.heads, b.f.nwork);
  bwd_dq_kernel<D><<<grid, NTH, C::SMEM, st>>>(tq, tk, tv, to, b);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& b, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  using C = BCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((b.f.ck + BT - 1) / BT), b.f.kv_heads, b.f.nwork);
  bwd_dkdv_kernel<D><<<grid, NTH, C::SMEM, st>>>(tq, tk, tv, to, b);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const float* out, const void* dout, float* dvec, long long rows,
                           int heads, int d, cudaStream_t st) {
  const long long n_rh = rows * heads;
  if (n_rh == 0) return cudaSuccess;
  const long long blocks = (n_rh * 32 + 255) / 256;
  bwd_pre_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      out, static_cast<const __nv_bfloat16*>(dout), dvec, n_rh, d);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdArgs& b, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  return d == 128 ? launch_dq_d<128>(b, tq, tk, tv, to, st) : launch_dq_d<64>(b, tq, tk, tv, to, st);
}

cudaError_t launch_bwd_dkdv(const BwdArgs& b, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  return d == 128 ? launch_dkdv_d<128>(b, tq, tk, tv, to, st)
                  : launch_dkdv_d<64>(b, tq, tk, tv, to, st);
}

cudaError_t take_bwd_status(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_bwd_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
}

}  // namespace ra
