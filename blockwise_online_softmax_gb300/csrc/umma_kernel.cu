// bf16 block update on the 5th-generation tensor cores (tcgen05 / TMEM / TMA).
//
// One CTA folds one K/V block into the running state of 256 query rows of
// one head, held as two 128-row query tiles Q0 and Q1.  This is the
// "FlashAttention_Update(Q_i, K_j, V_j, m_i, l_i, O_i)" of "Ring Attention
// Paper Breakdown", section 2.  Inside the block, K/V tiles of 128 keys
// stream through shared memory.  This is the inner level of the two-level
// blocking in "Ring Attention：把超长序列沿设备环流动", section
// "两层分块如何嵌套".  Both query tiles share each K/V tile, which halves
// the L2-to-SM traffic per FLOP.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0..3  softmax group 0: one thread per row of Q0 (TMEM lane
//               32*warp+lane).
//   warps 4..7  softmax group 1: the same for Q1.
//   warp 8      TMA producer for Q0, Q1 (once) and the K tiles.
//   warp 9      Allocates TMEM.  Lane 0 issues every tcgen05.mma.
//   warp 10     TMA producer for the V tiles.
//   warp 11     idle.
// K and V stream through two rings of shared-memory stages (2 deep at
// d = 128, 4 at d = 64).  Slot c of the rings holds K(c) and V(c-1) of the
// visit: the MMA thread needs exactly that pair in iteration c-1 (PV with
// V(c-1), QK with K(c)), so one full barrier (both producers' bytes) and one
// empty barrier (one commit) per slot cover both rings.
// A softmax thread reads its S row from TMEM, takes the row max,
// exponentiates, writes P back as bf16 over its S row, rescales its O~ row
// in TMEM when the max grows, and loads and stores the state.
//
// Registers: the CTA launches with 168 per thread (three warps share each
// SM sub-partition's 16K registers).  The producer/MMA warpgroup then gives
// some back and the softmax warpgroups take them (setmaxnreg): 208/88 at
// d = 128 and 224/56 at d = 64, with 2*128*softmax + 128*control = 384*168.
//
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P_g overwrites the first 64 columns of S_g, two bf16 per 32-bit column,
// and is the A operand of O_g += P_g V read from TMEM.
//
// MMA issue order per K/V tile t (prologue: QK0(0), QK1(0)):
//   PV0(t), QK0(t+1), PV1(t), QK1(t+1).
// While softmax group 0 works on S0(t+1), the tensor pipe runs PV1(t) and
// QK1(t+1).  While group 1 works on S1(t+1), it runs PV0(t+1) and
// QK0(t+2).  Every tcgen05.mma of the CTA comes from one thread, and they
// run in issue order.  That order lets QK_g(t+1) overwrite the columns
// from which PV_g(t) reads P_g(t).
//
// Rescale rule: each row's max in use follows the exact running max, so the
// largest weight of a row is exactly 1 and is exact in bf16.  A lazy rule
// (move the max only when it grows by 2^k) saves O~ read-scale-writes.  But
// it makes the dominant weight 2^delta, which bf16 rounds by up to 2^-8
// relative, and on rows where one key dominates that error reaches
// |v| * 2^-8.  The code keeps the max in use and the true max apart, so
// the threshold is a single constant.  The stored state is canonical: it
// is relative to the exact running max.
//
// Every wait is bounded.  A time-out records a code in g_umma_status.  All
// roles of the CTA then leave their loops, in-flight TMA and MMA work is
// drained (bounded), and TMEM is freed.  CTAs that start later in the
// launch do no work.
#include <cmath>
#include <cstdint>

#include "fwd_tile.cuh"
#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {

__device__ int g_umma_status = 0;

namespace {

using namespace fwd;

constexpr int NTHREADS = (NQ + 1) * 128;
constexpr uint32_t REGS_LAUNCH = 168;

template <int D>
struct Cfg {
  static constexpr int NCH = D / 64;                  // 128-byte chunks per row
  static constexpr uint32_t TILE_BYTES = BM * D * 2;  // one Q, K or V tile
  // K and V stage counts, equal since a slot takes one stage of each ring
  // (192 KB of shared memory in all at d = 128).  A third V stage fits in
  // 227 KB but measured slower: the L1 share of the unified SRAM drops too
  // far for the state loads and stores.
  static constexpr int NSK = (D == 64) ? 4 : 2;
  static constexpr int NSV = NSK;
  static constexpr uint32_t S_COL = 0;                // S_g at S_COL + g * BN
  static constexpr uint32_t O_COL = 2 * BN;           // O_g at O_COL + g * D
  // barriers
  static constexpr int B_Q = 0;
  // Slot c of the K/V rings carries K(c) and V(c-1) (visit order), both
  // in stage c % NSK: one full barrier (2 arrivals + bytes) and one empty
  // barrier per stage.
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + NSK;
  static constexpr int B_SF = B_KE + NSK;     // NQ: QK_g done
  static constexpr int B_PF = B_SF + NQ;  // NQ: P_g written (128 arrivals)
  static constexpr int B_OD = B_PF + NQ;  // NQ: last PV_g done
  static constexpr int B_DRAIN = B_OD + NQ;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQ * TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(O_COL + NQ * D <= TMEM_COLS, "TMEM budget");
  // setmaxnreg split of the launch allocation.  The MMA issuer must not
  // spill: a local-memory access in its loop stalls the tensor pipe.  At
  // d = 128 it needs more than 72 registers, so the softmax warps give up
  // 8 (their few spills sit outside the tile loop).
  static constexpr uint32_t REGS_SOFTMAX = (D == 64) ? 224 : 208;
  static constexpr uint32_t REGS_CONTROL = (D == 64) ? 56 : 88;
  static_assert(NQ * 128 * REGS_SOFTMAX + 128 * REGS_CONTROL == NTHREADS * REGS_LAUNCH,
                "setmaxnreg split must add up to the launch allocation");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
};

// Slot-ring producer: slot c = 0..n takes tile c of the visit (K, v_lag = 0)
// or tile c - 1 (V, v_lag = 1) into stage c % NS; a slot without a tile is
// a plain arrival.  The two producers share the slot barriers: a full
// barrier completes on both arrivals and all bytes, an empty barrier on the
// MMA thread's one commit per slot.  Returns false on an abort, after draining (bounded) the
// copies still in flight.
template <int D, int NS>
__device__ __forceinline__ bool produce_slots(const Work& wk, const TileSeq& seq, int kh,
                                              uint32_t sbase, uint32_t b_full, uint32_t b_empty,
                                              const CUtensorMap* tm, int v_lag,
                                              volatile int* abort_flag, int code, long long lim) {
  using C = Cfg<D>;
  tma_prefetch_desc(tm);
  int issued = 0;
  bool ok = true;
  for (int c = 0; c <= seq.n; ++c) {
    const int st = c % NS;
    const uint32_t ph = static_cast<uint32_t>(c / NS) & 1u;
    if (c >= NS) ok = wait_bar(b_empty + 8u * st, ph ^ 1u, abort_flag, &g_umma_status, code, lim);
    if (!ok) break;
    const int t = c - v_lag;
    if (t >= 0 && t < seq.n) {
      const int kv_row = static_cast<int>(wk.kv_base + static_cast<long long>(seq.at(t)) * BN);
      mbar_arrive_expect_tx(b_full + 8u * st, C::TILE_BYTES);
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_load_3d(sbase + st * C::TILE_BYTES + ch * CHUNK_BYTES, tm, b_full + 8u * st, ch * 64,
                    kh, kv_row);
    } else {
      mbar_arrive(b_full + 8u * st);
    }
    issued = c + 1;
  }
  if (!ok) {
    volatile int no_abort = 0;
    for (int c = (issued > NS ? issued - NS : 0); c < issued; ++c)
      wait_bar(b_full + 8u * (c % NS), static_cast<uint32_t>(c / NS) & 1u, &no_abort, nullptr, 0,
               lim);
  }
  return ok;
}

// Producers (warps 8 and 10) and MMA issuer (warp 9); warp 11 falls through.
template <int D>
__device__ __forceinline__ void control_roles(const FwdArgs& a, const Work& wk, long long row0,
                                              const int (&ta)[NQ], const int (&tb)[NQ],
                                              const TileSeq& seq, uint32_t tmem,
                                              uint32_t sQ, uint32_t sK, uint32_t sV,
                                              uint32_t bar0, volatile int* abort_flag,
                                              const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int kh = h / (a.heads / a.kv_heads);
  const long long lim = a.wait_limit;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    // Warp 8 loads Q0, Q1 and the K tiles; warp 10 loads the V tiles.  Each
    // waits only on its own stages, so a V stage still held by the PV
    // products never delays a K load.
    if (lane == 0 && seq.n > 0) {
      if (warp == 8) {
        tma_prefetch_desc(tmQ);
        mbar_arrive_expect_tx(bar(C::B_Q), NQ * C::TILE_BYTES);
#pragma unroll
        for (int g = 0; g < NQ; ++g) {
          const int q_row = static_cast<int>(wk.q_base + row0 + g * BM);
#pragma unroll
          for (int ch = 0; ch < C::NCH; ++ch)
            tma_load_3d(sQ + g * C::TILE_BYTES + ch * CHUNK_BYTES, tmQ, bar(C::B_Q), ch * 64, h,
                        q_row);
        }
        if (!produce_slots<D, C::NSK>(wk, seq, kh, sK, bar(C::B_KF), bar(C::B_KE), tmK, 0,
                                      abort_flag, 0x11, lim)) {
          volatile int no_abort = 0;
          wait_bar(bar(C::B_Q), 0, &no_abort, nullptr, 0, lim);
        }
      } else {
        produce_slots<D, C::NSK>(wk, seq, kh, sV, bar(C::B_KF), bar(C::B_KE), tmV, 1, abort_flag,
                                 0x12, lim);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 runs the whole loop alone; the other lanes wait at the end.
    // Measured against the whole warp running it with every MMA and commit
    // predicated on lane 0: +1.5% on a fused ring (the per-product issue
    // cost is lower from one lane).
    if (lane == 0 && seq.n > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 1);
      // All shared-memory descriptors are built once.  Moving a descriptor's
      // start address by `off` bytes adds off >> 4 to it (the field cannot
      // carry out, since shared addresses are below 256 KB).
      const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
      const uint64_t kdesc = sdesc_sw128(sK, 16, 1024);
      const uint64_t vdesc = sdesc_sw128(sV, CHUNK_BYTES, 1024);
      constexpr uint64_t TILE16 = C::TILE_BYTES >> 4;  // one tile, in descriptor units
      auto qk = [&](int g, int sk) {
        const uint32_t d_tmem = tmem + C::S_COL + static_cast<uint32_t>(g) * BN;
        const uint64_t a0 = qdesc + static_cast<uint64_t>(g) * TILE16;
        const uint64_t b0 = kdesc + static_cast<uint64_t>(sk) * TILE16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major, 128-byte swizzle: 16 elements = 32 bytes along a row;
          // every 4 steps move to the next 64-wide column chunk.
          const uint64_t off = ((kk >> 2) * CHUNK_BYTES + (kk & 3) * 32) >> 4;
          mma_ss(d_tmem, a0 + off, b0 + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF + g));
      };
      // O_g += P_g V over the 128 keys of the tile.
      auto pv = [&](int g, int sv) {
        const uint32_t p_tmem = tmem + C::S_COL + static_cast<uint32_t>(g) * BN;
        const uint32_t o_tmem = tmem + C::O_COL + static_cast<uint32_t>(g) * D;
        const uint64_t b0 = vdesc + static_cast<uint64_t>(sv) * TILE16;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // P: two bf16 per 32-bit TMEM column, 8 columns per 16 keys.
          // V (MN-major, 128-byte swizzle): 16 keys = two 8-row groups of
          // 1024 B (SBO); the 64-wide column chunks sit CHUNK_BYTES apart (LBO).
          mma_ts(o_tmem, p_tmem + kk * 8, b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv,
                 1u);
        }
      };
      bool ok = wait_bar(bar(C::B_Q), 0, abort_flag, &g_umma_status, 0x21, lim);
      if (ok) ok = wait_bar(bar(C::B_KF), 0, abort_flag, &g_umma_status, 0x22, lim);
      // The loop runs over the visit index k (tile seq.at(k)); it needs no
      // tile index, only where each group's run of tiles starts in the
      // visit (ks) and how long it is (ne).  A group's tiles are contiguous
      // in the visit.  Every instruction here delays the tensor pipe, so
      // the per-group test is one subtract and one unsigned compare.
      int ks[NQ], ne[NQ];
#pragma unroll
      for (int g = 0; g < NQ; ++g) {
        ne[g] = tb[g] > ta[g] ? tb[g] - ta[g] : 0;
        ks[g] = ta[g] < seq.a0 + seq.na ? ta[g] - seq.a0 : seq.na + (ta[g] - seq.b0);
      }
      if (ok) {
        tc_fence_after();
        if (ks[0] == 0 && ne[0] > 0) qk(0, 0);
        if (ks[1] == 0 && ne[1] > 0) qk(1, 0);
        tc_commit(bar(C::B_KE));
      }
      for (int k = 0; k < seq.n && ok; ++k) {
        // Slot k + 1: V(k) and K(k + 1), both in stage (k + 1) % NSK.
        const int sv = (k + 1) % C::NSK;
        const int sk1 = sv;
        // Both operand tiles of this iteration first (one wait), so the PV
        // and QK products of a group issue back to back.
        ok = wait_bar(bar(C::B_KF + sv), static_cast<uint32_t>((k + 1) / C::NSK) & 1u, abort_flag,
                      &g_umma_status, 0x24, lim);
        if (!ok) break;
#pragma unroll
        for (int g = 0; g < NQ; ++g) {
          const int kg = k - ks[g];  // tile kg of group g's run
          if (static_cast<unsigned>(kg) < static_cast<unsigned>(ne[g])) {
            ok = wait_bar(bar(C::B_PF + g), static_cast<uint32_t>(kg) & 1u, abort_flag,
                          &g_umma_status, 0x23, lim);
            if (!ok) break;
            tc_fence_after();
            pv(g, sv);
          }
          if (static_cast<unsigned>(kg + 1) < static_cast<unsigned>(ne[g])) qk(g, sk1);
        }
        if (!ok) break;
        tc_commit(bar(C::B_KE + sv));
      }
      if (ok) {
        // Only the epilogues wait for the P.V products (each tile's softmax
        // knows PV_g(t-1) is done from S_g(t)).  Both groups' epilogues wait
        // for every product of the CTA: they stage the state in the K/V
        // stages, which the other group's last products may still read.
        tc_commit(bar(C::B_OD));
        tc_commit(bar(C::B_OD + 1));
      }
      // Drain every MMA issued so far before TMEM can be freed.
      volatile int no_abort = 0;
      tc_commit(bar(C::B_DRAIN));
      wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    }
    __syncwarp();
  }
}

template <int D>
__device__ __forceinline__ void softmax_role(const FwdArgs& a, const Work& wk, long long row0,
                                             const int (&ta)[NQ], const int (&tb)[NQ],
                                             long long vb, uint32_t tmem, uint32_t bar0,
                                             uint32_t sK, uint32_t sV, const CUtensorMap* tmO,
                                             volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const long long lim = a.wait_limit;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  {
    // ------------------------------------------------------------ softmax
    const int g = warp >> 2;       // query tile of this group
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = C::S_COL + static_cast<uint32_t>(g) * BN;
    const uint32_t o_col = C::O_COL + static_cast<uint32_t>(g) * D;
    const long long grow = row0 + g * BM + row;  // row within the block
    const bool valid = grow < a.cq;
    const long long sidx = (wk.state_base + grow) * a.heads + h;
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    // Select, not index: g is not a compile-time constant here.
    const int t_first = g ? ta[1] : ta[0], t_end = g ? tb[1] : tb[0];

    if (t_end > t_first) {
      // Keys row_lo .. row_hi-1 of the K/V block are allowed for this row.
      // Tiles full_0 .. full_0 + n_full - 1 lie wholly inside that range and
      // need no mask.
      int row_lo = 0, row_hi = 0;
      if (valid) {
        long long lo, hi;
        row_keys(a, wk, grow, vb, &lo, &hi);
        row_lo = static_cast<int>(lo);
        row_hi = static_cast<int>(hi);
      }
      const int full_0 = (row_lo + BN - 1) / BN;
      const int n_full = row_hi / BN - full_0 > 0 ? row_hi / BN - full_0 : 0;
      float m_ld = -INFINITY, l_run = 0.f;
      if (valid) {
        m_ld = a.m[sidx];
        l_run = a.l[sidx];
      }
      // O~ state: HBM -> TMEM.
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        if (valid) {
          const float4* src = reinterpret_cast<const float4*>(a.o + sidx * D + cc * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x = src[j];
            r[4 * j + 0] = __float_as_uint(x.x);
            r[4 * j + 1] = __float_as_uint(x.y);
            r[4 * j + 2] = __float_as_uint(x.z);
            r[4 * j + 3] = __float_as_uint(x.w);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        tmem_st32(tl + o_col + cc * 32, r);
      }
      tmem_wait_st();

      float m_used = m_ld * kLog2e;  // log2 units; -inf stays -inf
      float m_true = m_used;
      bool m_moved = false;
      bool ok = true;

      for (int t = t_first; t < t_end; ++t) {
        ok = softmax_tile<D>(tl, s_col, o_col, t, row_lo, row_hi, full_0, n_full, sl2,
                                    sl2x2, bar(C::B_SF + g), bar(C::B_PF + g),
                                    static_cast<uint32_t>(t - t_first) & 1u, abort_flag,
                                    &g_umma_status, lim, m_used, m_true, m_moved, l_run);
        if (!ok) break;
      }

      if (ok) {
        // The one commit on B_OD + g follows the CTA's last product.
        ok = wait_bar(bar(C::B_OD + g), 0u, abort_flag, &g_umma_status, 0x33, lim);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok && a.o_tma && row0 + (g + 1) * BM <= a.cq) {
        // Every row of the tile lies in the block: O~ goes back to HBM
        // through shared memory and TMA tensor stores, as in the fused
        // ring's epilogue (group 0 stages in the K stages, group 1 in the V
        // stages, 128-byte swizzle; the group's P barrier, with all its
        // phases done, gathers the 128 rows for one more phase).
        static_assert(BM * D * 4 <= C::NSK * C::TILE_BYTES, "state tile staging fits");
        tc_fence_after();
        const float fin = (m_used == m_true) ? 1.f : ex2(m_used - m_true);
        const uint32_t stage = g == 0 ? sK : sV;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tl + o_col + cc * 32, r);
          tmem_wait_ld();
          reg_fence32(r);
          const uint32_t rb = stage + static_cast<uint32_t>(cc * BM * 128 + row * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(rb + (static_cast<uint32_t>(j ^ (row & 7)) << 4),
                         __float_as_uint(__uint_as_float(r[4 * j + 0]) * fin),
                         __float_as_uint(__uint_as_float(r[4 * j + 1]) * fin),
                         __float_as_uint(__uint_as_float(r[4 * j + 2]) * fin),
                         __float_as_uint(__uint_as_float(r[4 * j + 3]) * fin));
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_PF + g));
        if (row == 0 &&
            wait_bar(bar(C::B_PF + g), static_cast<uint32_t>(t_end - t_first) & 1u, abort_flag,
                     &g_umma_status, 0x34, lim)) {
          const int s_row = static_cast<int>(wk.state_base + row0 + g * BM);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
            tma_store_3d(tmO, stage + static_cast<uint32_t>(cc * BM * 128), cc * 32, h, s_row);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        if (valid) {
          a.l[sidx] = l_run * fin;
          a.m[sidx] = m_moved ? m_true * kLn2 : m_ld;
        }
      } else if (ok) {
        tc_fence_after();
        // Canonical state: rescale once from m_used to the exact running max.
        const float fin = (m_used == m_true) ? 1.f : ex2(m_used - m_true);
        uint32_t r[D / 32][32];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tl + o_col + cc * 32, r[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          reg_fence32(r[cc]);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(a.o + sidx * D + cc * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(r[cc][4 * j + 0]) * fin,
                                   __uint_as_float(r[cc][4 * j + 1]) * fin,
                                   __uint_as_float(r[cc][4 * j + 2]) * fin,
                                   __uint_as_float(r[cc][4 * j + 3]) * fin);
          }
        }
        if (valid) {
          a.l[sidx] = l_run * fin;
          a.m[sidx] = m_moved ? m_true * kLn2 : m_ld;
        }
      }
    }
  }

}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
umma_update_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const FwdArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::OFF_Q;
  const uint32_t sK = s_base + C::OFF_K;
  const uint32_t sV = s_base + C::OFF_V;
  const uint32_t bar0 = s_base + C::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const Work wk = decode_work(a, blockIdx.z);
  // Under causal masking the later query rows carry more work, so they are
  // launched first.
  const int pair = a.mask.causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                                 : static_cast<int>(blockIdx.x);
  const long long row0 = static_cast<long long>(pair) * (NQ * BM);
  const long long vb = valid_bound(a.mask);
  int ta[NQ], tb[NQ];
#pragma unroll
  for (int g = 0; g < NQ; ++g)
    tile_range(a, wk, row0 + g * BM, row0 + (g + 1) * BM, vb, BN, &ta[g], &tb[g]);
  const TileSeq seq = make_seq(ta, tb);
  // A CTA whose rows see no key of this block leaves their state as it is.
  if (seq.n == 0) return;

  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      const bool pf = i >= C::B_PF && i < C::B_PF + NQ;
      const bool kvf = i >= C::B_KF && i < C::B_KF + C::NSK;
      mbar_init(bar(i), pf ? 128u : (kvf ? 2u : 1u));
    }
    // A CTA that starts after another one of this launch gave up a wait
    // does no work.
    *abort_flag = *reinterpret_cast<volatile int*>(&g_umma_status) != 0 ? 1 : 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (*abort_flag) return;  // uniform across the CTA: read after the barrier
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The role branches never merge again: each ends at named barrier 1 (all
  // threads), after which the MMA warp frees TMEM.  Register budgets differ
  // per branch.
  if (warp >= 8) {
    regs_dec<C::REGS_CONTROL>();
    control_roles<D>(a, wk, row0, ta, tb, seq, tmem, sQ, sK, sV, bar0, abort_flag, &tmQ, &tmK, &tmV);
    tc_fence_before();
    named_bar_sync(1, NTHREADS);
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    softmax_role<D>(a, wk, row0, ta, tb, vb, tmem, bar0, sK, sV, &tmO, abort_flag);
    tc_fence_before();
    named_bar_sync(1, NTHREADS);
  }
}

// ====================================================================== fused ring
// One launch runs the whole ring ("Ring Attention Paper Breakdown", section
// 2: Q_i stays while the K/V blocks j = (i - s) mod P, s = 0 .. P-1, come
// by).  A CTA owns 256 query rows of one head of block i and keeps them,
// and their running state (m, l, O~), on chip for every step: the state
// lives in registers and TMEM from the first K/V tile to the last, and the
// CTA finalizes at the end (O = O~ / l, LSE).  The ring hop is the producer
// moving on to the next block's rows: its first tiles load into the same
// stage ring while the tensor pipe works on the previous block's last ones.
// Every role walks the same visit: the steps in ring order, within a step
// the union of the two query tiles' key-tile ranges (as in the one-step
// kernel), skipping steps whose pair has no allowed key.

// The work item of a fused-ring CTA: rank i, query head h and query-tile
// pair.  The query heads of a launch are taken in chunks of 2^a.ring_lc
// consecutive heads (4 when the head count allows: one KV head's query heads
// under GQA 4:1).  The grid is (query-tile pairs, 2^ring_lc x P, chunks):
// the launch order (x fastest, then y, then z) runs one chunk after the
// other, so the CTAs that run at the same time read the K/V blocks of a few
// heads, which stay in L2 for all of them; within a chunk it is rank-major,
// and under causal masking with the contiguous layout the ranks with the
// most blocks, and within a rank the later query tiles, come first, so
// that a launch of one or two waves still starts all its heaviest CTAs
// first.  Shifts and masks of the block index only: cheap enough for the
// compiler to recompute rather than keep live across the register split.
struct RingItem {
  int i, h, pair;
};
__device__ __forceinline__ RingItem ring_item(const FwdArgs& a) {
  // The block index is read with volatile moves so that every call
  // recomputes the item where it is used instead of the compiler keeping
  // one copy live through the roles.
  uint32_t bx, by, bz;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(bx));
  asm volatile("mov.u32 %0, %%ctaid.y;" : "=r"(by));
  asm volatile("mov.u32 %0, %%ctaid.z;" : "=r"(bz));
  const bool heavy_first = a.mask.causal && a.layout == kContiguous;
  const int y = static_cast<int>(by);
  const int r = y >> a.ring_lc;
  RingItem it;
  it.h = a.h0 + (static_cast<int>(bz) << a.ring_lc) + (y & ((1 << a.ring_lc) - 1));
  it.i = heavy_first ? a.P - 1 - r : r;
  it.pair = a.mask.causal ? static_cast<int>(gridDim.x - 1 - bx) : static_cast<int>(bx);
  return it;
}

// Slot-ring producer over the whole visit: slot c takes visit tile c (K,
// v_lag = 0) or c - 1 (V, v_lag = 1); a slot without a tile is a plain
// arrival (slot 0 for V, the slot after the last tile for K).  Returns false
// on an abort, after draining (bounded) the copies still in flight.
template <int D, int NS>
__device__ __forceinline__ bool produce_ring(const FwdArgs& a, const StepVisit* rec, int kh,
                                             uint32_t sbase, uint32_t b_full,
                                             uint32_t b_empty, const CUtensorMap* tm, int v_lag,
                                             volatile int* abort_flag, int code, long long lim) {
  using C = Cfg<D>;
  tma_prefetch_desc(tm);
  int c = 0;
  auto fill = [&](long long kv_row, bool tile) -> bool {
    const int st = c % NS;
    if (c >= NS &&
        !wait_bar(b_empty + 8u * st, (static_cast<uint32_t>(c / NS) & 1u) ^ 1u, abort_flag,
                  &g_umma_status, code, lim))
      return false;
    if (tile) {
      mbar_arrive_expect_tx(b_full + 8u * st, C::TILE_BYTES);
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_load_3d(sbase + st * C::TILE_BYTES + ch * CHUNK_BYTES, tm, b_full + 8u * st, ch * 64,
                    kh, static_cast<int>(kv_row));
    } else {
      mbar_arrive(b_full + 8u * st);
    }
    ++c;
    return true;
  };
  bool ok = true;
  if (v_lag) ok = fill(0, false);
  for (int s = next_step(rec, a.P, 0); s < a.P && ok; s = next_step(rec, a.P, s + 1)) {
    const TileSeq seq = rec[s].seq;
    const long long kv_base = rec[s].kv_base;
    for (int k = 0; k < seq.n && ok; ++k)
      ok = fill(kv_base + static_cast<long long>(seq.at(k)) * BN, true);
  }
  if (ok && !v_lag) ok = fill(0, false);
  if (!ok) {
    volatile int no_abort = 0;
    for (int x = (c > NS ? c - NS : 0); x < c; ++x)
      wait_bar(b_full + 8u * (x % NS), static_cast<uint32_t>(x / NS) & 1u, &no_abort, nullptr, 0,
               lim);
  }
  return ok;
}

// Producers (warps 8 and 10) and MMA issuer (warp 9) of the fused ring; the
// visit is not empty (the kernel returns early otherwise).
template <int D>
__device__ __forceinline__ void ring_control_roles(const FwdArgs& a, const StepVisit* rec,
                                                   long long row0, uint32_t tmem, uint32_t sQ,
                                                   uint32_t sK, uint32_t sV, uint32_t bar0,
                                                   volatile int* abort_flag,
                                                   const CUtensorMap* tmK,
                                                   const CUtensorMap* tmV) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = ring_item(a).h;
  const int kh = h / (a.heads / a.kv_heads);
  const long long lim = a.wait_limit;
  auto bar = [&](int x) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(x); };
  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      if (warp == 8) {
        // The Q tiles were requested in the kernel prologue.
        if (!produce_ring<D, C::NSK>(a, rec, kh, sK, bar(C::B_KF), bar(C::B_KE), tmK, 0,
                                     abort_flag, 0x11, lim)) {
          volatile int no_abort = 0;
          wait_bar(bar(C::B_Q), 0, &no_abort, nullptr, 0, lim);
        }
      } else {
        produce_ring<D, C::NSK>(a, rec, kh, sV, bar(C::B_KF), bar(C::B_KE), tmV, 1, abort_flag,
                                0x12, lim);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // As in the one-step kernel (lane 0 alone), with the visit index K
    // running over every step: slot K + 1 holds V(K) and K(K + 1).  At the
    // last tile of a step the look-ahead QK is the next step's first tile,
    // whose groups are known from the next step's visit, computed when the
    // step begins.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 1);
      const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
      const uint64_t kdesc = sdesc_sw128(sK, 16, 1024);
      const uint64_t vdesc = sdesc_sw128(sV, CHUNK_BYTES, 1024);
      constexpr uint64_t TILE16 = C::TILE_BYTES >> 4;
      auto qk = [&](int g, int sk) {
        const uint32_t d_tmem = tmem + C::S_COL + static_cast<uint32_t>(g) * BN;
        const uint64_t a0 = qdesc + static_cast<uint64_t>(g) * TILE16;
        const uint64_t b0 = kdesc + static_cast<uint64_t>(sk) * TILE16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * CHUNK_BYTES + (kk & 3) * 32) >> 4;
          mma_ss(d_tmem, a0 + off, b0 + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF + g));
      };
      auto pv = [&](int g, int sv) {
        const uint32_t p_tmem = tmem + C::S_COL + static_cast<uint32_t>(g) * BN;
        const uint32_t o_tmem = tmem + C::O_COL + static_cast<uint32_t>(g) * D;
        const uint64_t b0 = vdesc + static_cast<uint64_t>(sv) * TILE16;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(o_tmem, p_tmem + kk * 8, b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv,
                 1u);
      };
      // The current step's visit in registers; of the next non-empty step
      // only which groups its first tile has.
      int s_cur = next_step(rec, a.P, 0);
      int s_nxt = next_step(rec, a.P, s_cur + 1);
      TileSeq seq = rec[s_cur].seq;
      int ks[NQ], ne[NQ];
#pragma unroll
      for (int g = 0; g < NQ; ++g) {
        ks[g] = rec[s_cur].ks[g];
        ne[g] = rec[s_cur].ne[g];
      }
      bool ok = wait_bar(bar(C::B_Q), 0, abort_flag, &g_umma_status, 0x21, lim);
      if (ok) ok = wait_bar(bar(C::B_KF), 0, abort_flag, &g_umma_status, 0x22, lim);
      if (ok) {
        tc_fence_after();
        if (ks[0] == 0 && ne[0] > 0) qk(0, 0);
        if (ks[1] == 0 && ne[1] > 0) qk(1, 0);
        tc_commit(bar(C::B_KE));
      }
      int K = 0;            // visit index over all steps
      int cnt[NQ] = {0, 0};  // tiles of each group so far (its P barrier's phase)
      while (ok) {
        bool nx[NQ];
#pragma unroll
        for (int g = 0; g < NQ; ++g)
          nx[g] = s_nxt < a.P && rec[s_nxt].ks[g] == 0 && rec[s_nxt].ne[g] > 0;
        for (int k = 0; k < seq.n && ok; ++k, ++K) {
          const int sv = (K + 1) % C::NSK;  // slot K + 1: V(K) and K(K + 1)
          ok = wait_bar(bar(C::B_KF + sv), static_cast<uint32_t>((K + 1) / C::NSK) & 1u, abort_flag,
                        &g_umma_status, 0x24, lim);
          if (!ok) break;
          const bool last = k + 1 == seq.n;
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            const int kg = k - ks[g];
            if (static_cast<unsigned>(kg) < static_cast<unsigned>(ne[g])) {
              ok = wait_bar(bar(C::B_PF + g), static_cast<uint32_t>(cnt[g]) & 1u, abort_flag,
                            &g_umma_status, 0x23, lim);
              if (!ok) break;
              ++cnt[g];
              tc_fence_after();
              pv(g, sv);
            }
            const bool qn =
                last ? nx[g] : static_cast<unsigned>(kg + 1) < static_cast<unsigned>(ne[g]);
            if (qn) qk(g, sv);
          }
          if (!ok) break;
          tc_commit(bar(C::B_KE + sv));
        }
        if (!ok || s_nxt >= a.P) break;
        s_cur = s_nxt;
        s_nxt = next_step(rec, a.P, s_cur + 1);
        seq = rec[s_cur].seq;
#pragma unroll
        for (int g = 0; g < NQ; ++g) {
          ks[g] = rec[s_cur].ks[g];
          ne[g] = rec[s_cur].ne[g];
        }
      }
      if (ok) {
        // Both groups' epilogues wait for the last products of the visit.
        tc_commit(bar(C::B_OD));
        tc_commit(bar(C::B_OD + 1));
      }
      volatile int no_abort = 0;
      tc_commit(bar(C::B_DRAIN));
      wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    }
    __syncwarp();
  }
}

// Softmax groups of the fused ring.  The state starts empty (m = -inf,
// l = 0, O~ = 0 in TMEM) and never leaves the CTA; at the end each valid
// row writes O = O~ / l and LSE = ln 2 * (m + log2 l) (m in log2 units; O~
// and l are relative to the same m), or 0 and -inf for a row that saw no
// key.  out is [rows, heads, d] and lse [rows, heads], like the state.
template <int D>
__device__ __forceinline__ void ring_softmax_role(const FwdArgs& a, const StepVisit* rec,
                                                  long long row0, long long vb, uint32_t tmem,
                                                  uint32_t bar0, uint32_t sK, uint32_t sV,
                                                  const CUtensorMap* tmO,
                                                  volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long lim = a.wait_limit;
  auto bar = [&](int x) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(x); };
  const int g = warp >> 2;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const uint32_t s_col = C::S_COL + static_cast<uint32_t>(g) * BN;
  const uint32_t o_col = C::O_COL + static_cast<uint32_t>(g) * D;
  const long long grow = row0 + g * BM + row;  // row within this CTA's query block
  const bool valid = grow < a.cq;
  const float sl2 = a.scale_log2;
  const uint64_t sl2x2 = f2pack(sl2, sl2);
  {
    uint32_t z[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) tmem_st32(tl + o_col + cc * 32, z);
    tmem_wait_st();
  }
  float m_used = -INFINITY, m_true = -INFINITY, l_run = 0.f;
  bool m_moved = false;
  bool ok = true;
  int cnt = 0;  // tiles so far: the phase of this group's S barrier
  for (int s = 0; s < a.P && ok; ++s) {
    // Select, not index: g is not a compile-time constant here.
    const int t0 = g ? rec[s].ta[1] : rec[s].ta[0], t1 = g ? rec[s].tb[1] : rec[s].tb[0];
    if (t1 <= t0) continue;
    const Work wk = ring_work(a, ring_item(a).i, s);
    int row_lo = 0, row_hi = 0;
    if (valid) {
      long long lo, hi;
      row_keys(a, wk, grow, vb, &lo, &hi);
      row_lo = static_cast<int>(lo);
      row_hi = static_cast<int>(hi);
    }
    const int full_0 = (row_lo + BN - 1) / BN;
    const int n_full = row_hi / BN - full_0 > 0 ? row_hi / BN - full_0 : 0;
    for (int t = t0; t < t1; ++t) {
      ok = softmax_tile<D>(tl, s_col, o_col, t, row_lo, row_hi, full_0, n_full, sl2, sl2x2,
                                  bar(C::B_SF + g), bar(C::B_PF + g),
                                  static_cast<uint32_t>(cnt) & 1u, abort_flag, &g_umma_status,
                                  lim, m_used, m_true, m_moved, l_run);
      ++cnt;
      if (!ok) break;
    }
  }
  if (ok && cnt > 0) {
    ok = wait_bar(bar(C::B_OD + g), 0u, abort_flag, &g_umma_status, 0x33, lim);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  const bool seen = l_run > 0.f;
  const float inv = seen ? 1.f / l_run : 0.f;
  const RingItem it = ring_item(a);
  const long long oidx = (static_cast<long long>(it.i) * a.cq + grow) * a.heads + it.h;
  float* dst = a.o + oidx * D;
  if (cnt > 0 && a.o_tma && row0 + (g + 1) * BM <= a.cq) {
    // Every row of the tile lies in this block: stage O in shared memory
    // and store the tile with the tensor map.  The K/V stages are free once
    // the last products are done (every MMA has completed when B_OD
    // fires): group 0 stages in the K stages, group 1 in the V stages.
    // The layout is the map's box, D / 32 boxes of 128 rows x 128 bytes,
    // with the 16-byte chunks of row r XOR-permuted by r % 8 (the 128-byte
    // swizzle), so that the eight lanes of a store phase hit distinct banks.
    // Row by row from registers, each thread would write its own 512-byte
    // row, every store instruction of a warp touching 32 rows.
    static_assert(BM * D * 4 <= C::NSK * C::TILE_BYTES, "O tile staging fits in the K/V stages");
    const uint32_t stage = g == 0 ? sK : sV;
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t r[32];
      tmem_ld32(tl + o_col + cc * 32, r);
      tmem_wait_ld();
      reg_fence32(r);
      const uint32_t rb = stage + static_cast<uint32_t>(cc * BM * 128 + row * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(rb + (static_cast<uint32_t>(j ^ (row & 7)) << 4),
                     __float_as_uint(__uint_as_float(r[4 * j + 0]) * inv),
                     __float_as_uint(__uint_as_float(r[4 * j + 1]) * inv),
                     __float_as_uint(__uint_as_float(r[4 * j + 2]) * inv),
                     __float_as_uint(__uint_as_float(r[4 * j + 3]) * inv));
    }
    // The group's P barrier, whose cnt phases are all done (the MMA warp
    // waited for the last one before the last P.V), gathers the 128 rows:
    // one more phase, waited for (bounded) by the thread that issues the
    // stores.  A wait that gives up skips the stores; the status word has
    // the error.
    fence_proxy_async_smem();
    mbar_arrive(bar(C::B_PF + g));
    if (row == 0 && wait_bar(bar(C::B_PF + g), static_cast<uint32_t>(cnt) & 1u, abort_flag,
                             &g_umma_status, 0x34, lim)) {
      const int q_row = static_cast<int>(static_cast<long long>(it.i) * a.cq + row0 + g * BM);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc)
        tma_store_3d(tmO, stage + static_cast<uint32_t>(cc * BM * 128), cc * 32, it.h, q_row);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  } else if (cnt > 0) {
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t r[32];
      tmem_ld32(tl + o_col + cc * 32, r);
      tmem_wait_ld();
      reg_fence32(r);
      if (valid) {
        float4* d4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d4[j] = make_float4(__uint_as_float(r[4 * j + 0]) * inv,
                              __uint_as_float(r[4 * j + 1]) * inv,
                              __uint_as_float(r[4 * j + 2]) * inv,
                              __uint_as_float(r[4 * j + 3]) * inv);
      }
    }
  } else if (valid) {
#pragma unroll
    for (int j = 0; j < D / 4; ++j)
      reinterpret_cast<float4*>(dst)[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (valid) a.m[oidx] = seen ? (m_used + log2f(l_run)) * kLn2 : -INFINITY;
}

// Grid (query-tile pairs, 2^ring_lc x P, head chunks); see ring_item for
// the order.
template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
umma_ring_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 const FwdArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::OFF_Q;
  const uint32_t sK = s_base + C::OFF_K;
  const uint32_t sV = s_base + C::OFF_V;
  const uint32_t bar0 = s_base + C::OFF_BAR;
  auto bar = [&](int x) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // The launch's status word, read first so that its latency passes under
  // the set-up below.
  int launch_status = 0;
  if (tid == 0) launch_status = *reinterpret_cast<volatile int*>(&g_umma_status);
  const RingItem it = ring_item(a);
  const int i = it.i;
  const int h = it.h;
  const int pair = it.pair;
  const long long row0 = static_cast<long long>(pair) * (NQ * BM);
  const long long vb = valid_bound(a.mask);
  // Barriers, the Q request and the tensor-memory allocation come first:
  // they need only the work item, so the Q load and the allocation run
  // under the visit computation below (about 3,000 cycles per CTA).
  if (tid == 8 * 32) {
    for (int x = 0; x < C::NBAR; ++x) {
      const bool pf = x >= C::B_PF && x < C::B_PF + NQ;
      const bool kvf = x >= C::B_KF && x < C::B_KF + C::NSK;
      mbar_init(bar(x), pf ? 128u : (kvf ? 2u : 1u));
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    // From here on every path waits for B_Q before the CTA exits (the MMA
    // warp, the K producer when it gives up, or this thread on the early
    // exits below).
    mbar_arrive_expect_tx(bar(C::B_Q), NQ * C::TILE_BYTES);
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
      const int q_row = static_cast<int>(static_cast<long long>(i) * a.cq + row0 + g * BM);
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_load_3d(sQ + g * C::TILE_BYTES + ch * CHUNK_BYTES, &tmQ, bar(C::B_Q), ch * 64, h,
                    q_row);
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  // The visit table: every step's tile ranges, computed once by all threads
  // before the roles split the registers.
  StepVisit* rec = reinterpret_cast<StepVisit*>(smem + C::OFF_MISC + 16);
  for (int s = tid; s < a.P; s += NTHREADS) rec[s] = step_visit(a, i, s, row0, vb);
  if (tid == 0) *abort_flag = launch_status != 0 ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool no_keys = next_step(rec, a.P, 0) == a.P;
  if (no_keys || *abort_flag) {  // uniform across the CTA: read after the barrier
    // Rows that see no key anywhere: O = 0 and LSE = -inf, and no pipeline.
    if (no_keys && tid < NQ * BM) {
      const long long grow = row0 + tid;
      if (grow < a.cq) {
        const long long oidx = (static_cast<long long>(i) * a.cq + grow) * a.heads + h;
#pragma unroll
        for (int j = 0; j < D / 4; ++j)
          reinterpret_cast<float4*>(a.o + oidx * D)[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        a.m[oidx] = -INFINITY;
      }
    }
    // The Q tiles land in shared memory before the CTA may exit.
    if (tid == 8 * 32) {
      volatile int no_abort = 0;
      wait_bar(bar(C::B_Q), 0, &no_abort, nullptr, 0, a.wait_limit);
    }
    if (warp == 9) tmem_dealloc(tmem, TMEM_COLS);
    return;
  }
  if (warp >= 8) {
    regs_dec<C::REGS_CONTROL>();
    ring_control_roles<D>(a, rec, row0, tmem, sQ, sK, sV, bar0, abort_flag, &tmK, &tmV);
    tc_fence_before();
    named_bar_sync(1, NTHREADS);
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    ring_softmax_role<D>(a, rec, row0, vb, tmem, bar0, sK, sV, &tmO, abort_flag);
    tc_fence_before();
    named_bar_sync(1, NTHREADS);
  }
}

template <int D>
cudaError_t launch_ring_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  using C = Cfg<D>;
  constexpr uint32_t smem = C::SMEM_BYTES + kRingMaxSteps * sizeof(StepVisit);
  static_assert(smem <= 232448, "shared memory budget of the fused ring");
  if (a.P > kRingMaxSteps) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(umma_ring_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int nh = a.nh > 0 ? a.nh : a.heads;
  FwdArgs b = a;
  b.ring_lc = nh % 4 == 0 ? 2 : (nh % 2 == 0 ? 1 : 0);
  dim3 grid(static_cast<unsigned>((a.cq + NQ * BM - 1) / (NQ * BM)),
            static_cast<unsigned>(a.P << b.ring_lc), static_cast<unsigned>(nh >> b.ring_lc));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  umma_ring_kernel<D><<<grid, NTHREADS, smem, st>>>(tq, tk, tv, to, b);
  return cudaGetLastError();
}

// One CTA waits on an mbarrier nothing will arrive on.  Used to test that a
// bounded wait gives up and reports instead of hanging.
__global__ void wait_selftest_kernel(long long limit) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&b), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_bar(smem_u32(&b), 0, reinterpret_cast<volatile int*>(&abort_flag), &g_umma_status, 0x7F,
             limit);
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(umma_update_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.cq + NQ * BM - 1) / (NQ * BM)), a.heads, a.nwork);
  umma_update_kernel<D><<<grid, NTHREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_umma_update(const FwdArgs& a, int d, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& to, cudaStream_t st) {
  return d == 128 ? launch_d<128>(a, tq, tk, tv, to, st) : launch_d<64>(a, tq, tk, tv, to, st);
}

cudaError_t launch_umma_ring(const FwdArgs& a, int d, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, cudaStream_t st) {
  return d == 128 ? launch_ring_d<128>(a, tq, tk, tv, to, st)
                  : launch_ring_d<64>(a, tq, tk, tv, to, st);
}

cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(limit_cycles);
  return cudaGetLastError();
}

cudaError_t take_umma_status(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_umma_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_umma_status, &zero, sizeof(int));
}

}  // namespace ra
