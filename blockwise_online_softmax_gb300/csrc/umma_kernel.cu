// bf16 block update on the 5th-generation tensor cores (tcgen05 / TMEM / TMA).
//
// One CTA folds one K/V block into the running state of a 128-row query
// tile of one head.  This is the "FlashAttention_Update(Q_i, K_j, V_j, m_i,
// l_i, O_i)" of "Ring Attention Paper Breakdown", section 2.  Inside the
// block, the K/V tiles of 128 keys stream through shared memory.  This is
// the inner level of the two-level blocking in "Ring Attention：
// 把超长序列沿设备环流动", section "两层分块如何嵌套".
//
// Warp roles (192 threads):
//   warp 0      TMA producer.  It loads the Q tile once, then the K and V
//               tiles into an NST-deep ring of shared-memory stages.
//   warp 1      Allocates TMEM.  Lane 0 issues every tcgen05.mma: S = Q K^T
//               into one of two TMEM S buffers, then O += P V with P read
//               from TMEM (P overwrites its S buffer).
//   warps 2..5  Softmax / correction / epilogue, one thread per query row.
//               A thread owns TMEM lane (row) 32*(warp%4)+lane.  It reads
//               its S row, takes the row max, exponentiates, writes P back
//               as bf16, rescales its O row when the max grows, and stores
//               the state at the end.
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D).  512 are
// allocated.
//
// Pipelining: QK^T of tile t+1 is issued before PV of tile t, so the
// tensor pipe runs S(t+1) while the softmax warps work on S(t).  All
// tcgen05.mma of the CTA come from one thread and run in issue order.
// That order is what lets QK^T(t+2) overwrite the TMEM that PV(t) reads.
//
// Rescale rule: the row max in use (m_used) follows the true running max
// exactly (RESCALE_THRESHOLD = 0).  The largest weight of a row is then
// exactly 1 and is exact in bf16.  A lazy rule, moving m_used only when the
// max grows by 2^k, would save read-scale-writes of O in TMEM.  But the
// dominant weight would become 2^delta, and bf16 rounds that by up to
// 2^-8 relative.  On rows where one key dominates (large logits, planted
// keys) that error reaches |v| * 2^-8 in O.  The code keeps m_used and
// m_true apart, so the threshold stays a single constant.  At the end
// the state is rescaled to the exact running max, so the stored
// (m, l, O~) is the unique canonical state.
//
// Every wait is bounded.  A time-out records a code in g_umma_status.  All
// roles then leave their loops, in-flight TMA and MMA work is drained
// (bounded), and TMEM is freed before exit.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {

__device__ int g_umma_status = 0;

namespace {

constexpr int BM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int NTHREADS = 192;
constexpr uint32_t CHUNK_BYTES = 128 * 128;  // 128 rows x 128 B (one swizzle span)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 0;
constexpr uint32_t O_COL = 256;
constexpr float RESCALE_THRESHOLD = 0.0f;  // log2 units; see the rescale rule above

template <int D>
struct Cfg {
  static constexpr int NCH = D / 64;                       // 128-byte chunks per row
  static constexpr uint32_t TILE_BYTES = BM * D * 2;       // one Q/K/V tile
  static constexpr int NST = (D == 64) ? 4 : 2;            // K/V stages
  // barriers
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + NST;
  static constexpr int B_VF = B_KE + NST;
  static constexpr int B_VE = B_VF + NST;
  static constexpr int B_SF = B_VE + NST;  // 2
  static constexpr int B_PF = B_SF + 2;    // 2
  static constexpr int B_OD = B_PF + 2;
  static constexpr int B_DRAIN = B_OD + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + NST * TILE_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
umma_update_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
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
  const int lane = tid & 31;
  const int h = blockIdx.y;
  const int kh = h / (a.heads / a.kv_heads);
  const Work wk = decode_work(a, blockIdx.z);
  const long long q_tile0 = static_cast<long long>(blockIdx.x) * BM;

  // Key tiles to visit: all of them, or, under causal masking, up to the
  // one holding the last key some row of this tile may see.
  const long long kv_tiles = (a.c + BN - 1) / BN;
  long long nt_ll = kv_tiles;
  if (a.causal) {
    const long long last_row = (q_tile0 + BM - 1 < a.c - 1) ? q_tile0 + BM - 1 : a.c - 1;
    const long long last_key = wk.q_pos0 + last_row - wk.kv_pos0;
    nt_ll = (last_key < 0) ? 0 : (last_key / BN + 1 < kv_tiles ? last_key / BN + 1 : kv_tiles);
  }
  const int nt = static_cast<int>(nt_ll);

  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_PF || i == C::B_PF + 1) cnt = 128;  // every softmax thread arrives
      mbar_init(bar(i), cnt);
    }
    // A CTA that starts after another one of this launch gave up a wait
    // does no work.
    *abort_flag = *reinterpret_cast<volatile int*>(&g_umma_status) != 0 ? 1 : 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (*abort_flag) return;  // uniform across the CTA: read after the barrier
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = a.wait_limit;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int q_row = static_cast<int>(wk.q_base + q_tile0);
      mbar_arrive_expect_tx(bar(C::B_Q), C::TILE_BYTES);
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_load_3d(sQ + ch * CHUNK_BYTES, &tmQ, bar(C::B_Q), ch * 64, h, q_row);
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int st = t % C::NST;
        const uint32_t ph = static_cast<uint32_t>(t / C::NST) & 1u;
        const int kv_row = static_cast<int>(wk.kv_base + static_cast<long long>(t) * BN);
        if (t >= C::NST)
          ok = wait_bar(bar(C::B_KE + st), ph ^ 1u, abort_flag, &g_umma_status, 0x11, lim);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_KF + st), C::TILE_BYTES);
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch)
          tma_load_3d(sK + st * C::TILE_BYTES + ch * CHUNK_BYTES, &tmK, bar(C::B_KF + st),
                      ch * 64, kh, kv_row);
        if (t >= C::NST)
          ok = wait_bar(bar(C::B_VE + st), ph ^ 1u, abort_flag, &g_umma_status, 0x12, lim);
        if (!ok) {
          issued = t + 1;  // K of tile t is in flight
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VF + st), C::TILE_BYTES);
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch)
          tma_load_3d(sV + st * C::TILE_BYTES + ch * CHUNK_BYTES, &tmV, bar(C::B_VF + st),
                      ch * 64, kh, kv_row);
        issued = t + 1;
      }
      if (!ok) {
        // Drain: wait (bounded) for the copies still in flight before the
        // CTA's shared memory is given up.
        volatile int no_abort = 0;
        wait_bar(bar(C::B_Q), 0, &no_abort, nullptr, 0, lim);
        for (int t = (issued > C::NST ? issued - C::NST : 0); t < issued; ++t) {
          const int st = t % C::NST;
          const uint32_t ph = static_cast<uint32_t>(t / C::NST) & 1u;
          wait_bar(bar(C::B_KF + st), ph, &no_abort, nullptr, 0, lim);
          wait_bar(bar(C::B_VF + st), ph, &no_abort, nullptr, 0, lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 1);
      bool ok = wait_bar(bar(C::B_Q), 0, abort_flag, &g_umma_status, 0x21, lim);
      tc_fence_after();
      auto issue_qk = [&](int t) -> bool {
        const int st = t % C::NST;
        const uint32_t ph = static_cast<uint32_t>(t / C::NST) & 1u;
        if (!wait_bar(bar(C::B_KF + st), ph, abort_flag, &g_umma_status, 0x22, lim)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + S_COL0 + static_cast<uint32_t>(t & 1) * BN;
        const uint32_t kbase = sK + st * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
          mma_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                 idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF + (t & 1)));
        tc_commit(bar(C::B_KE + st));
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int t = 0; t < nt && ok; ++t) {
        if (t + 1 < nt) {
          ok = issue_qk(t + 1);
          if (!ok) break;
        }
        const int b = t & 1;
        ok = wait_bar(bar(C::B_PF + b), static_cast<uint32_t>(t >> 1) & 1u, abort_flag,
                      &g_umma_status, 0x23, lim);
        if (!ok) break;
        const int st = t % C::NST;
        ok = wait_bar(bar(C::B_VF + st), static_cast<uint32_t>(t / C::NST) & 1u, abort_flag,
                      &g_umma_status, 0x24, lim);
        if (!ok) break;
        tc_fence_after();
        const uint32_t p_tmem = tmem + S_COL0 + static_cast<uint32_t>(b) * BN;
        const uint32_t vbase = sV + st * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // P columns: two bf16 per 32-bit column, 8 columns per 16 keys.
          // V (MN-major): 16 keys = two 8-row groups of 1024 B; the 64-wide
          // column chunks of V sit CHUNK_BYTES apart.
          mma_ts(tmem + O_COL, p_tmem + kk * 8,
                 sdesc_sw128(vbase + kk * 2048, CHUNK_BYTES, 1024), idesc_pv, 1u);
        }
        tc_commit(bar(C::B_OD));
        tc_commit(bar(C::B_VE + st));
      }
      // Drain every MMA issued so far before TMEM can be freed.
      volatile int no_abort = 0;
      tc_commit(bar(C::B_DRAIN));
      wait_bar(bar(C::B_DRAIN), 0, &no_abort, nullptr, 0, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const long long grow = q_tile0 + row;
    const bool valid = grow < a.c;
    const long long sidx = (wk.state_base + grow) * a.heads + h;
    const long long qpos = wk.q_pos0 + grow;
    const float sl2 = a.scale_log2;

    if (nt > 0) {
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
        tmem_st32(tl + O_COL + cc * 32, r);
      }
      tmem_wait_st();

      float m_used = m_ld * kLog2e;  // log2 units; -inf stays -inf
      float m_true = m_used;
      bool m_moved = false;
      bool ok = true;

      for (int t = 0; t < nt; ++t) {
        const int b = t & 1;
        ok = wait_bar(bar(C::B_SF + b), static_cast<uint32_t>(t >> 1) & 1u, abort_flag,
                      &g_umma_status, 0x31, lim);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float s[BN];
        {
          uint32_t r[32];
#pragma unroll
          for (int cc = 0; cc < BN / 32; ++cc) {
            tmem_ld32(tl + S_COL0 + b * BN + cc * 32, r);
            tmem_wait_ld();
            reg_fence32(r);
#pragma unroll
            for (int j = 0; j < 32; ++j) s[cc * 32 + j] = __uint_as_float(r[j]);
          }
        }
        // Mask: key j of this tile is allowed iff j < lim_j.  The tail
        // (kv local index < c) and the causal rule (key position <= query
        // position) are both upper bounds on j.
        long long lim_j = a.c - static_cast<long long>(t) * BN;
        if (a.causal) {
          const long long cl = qpos - wk.kv_pos0 - static_cast<long long>(t) * BN + 1;
          lim_j = cl < lim_j ? cl : lim_j;
        }
        if (lim_j < BN) {
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j >= lim_j) s[j] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int j = 4; j < BN; j += 4) {
          mx0 = fmaxf(mx0, s[j + 0]);
          mx1 = fmaxf(mx1, s[j + 1]);
          mx2 = fmaxf(mx2, s[j + 2]);
          mx3 = fmaxf(mx3, s[j + 3]);
        }
        const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        if (m_tile > m_true) {
          m_true = m_tile;
          m_moved = true;
        }
        const bool need = m_true > m_used + RESCALE_THRESHOLD;
        float alpha = 1.f;
        if (need) {
          alpha = ex2(m_used - m_true);  // m_used = -inf gives 0
          m_used = m_true;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        float sum0 = 0.f, sum1 = 0.f;
        uint32_t pk[BN / 2];
#pragma unroll
        for (int j = 0; j < BN; j += 2) {
          const float p0 = ex2(fmaf(s[j], sl2, -mref));
          const float p1 = ex2(fmaf(s[j + 1], sl2, -mref));
          sum0 += p0;
          sum1 += p1;
          __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);  // p0 in the low half
          pk[j / 2] = *reinterpret_cast<uint32_t*>(&v2);
        }
        l_run = l_run * alpha + (sum0 + sum1);
        {
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = pk[j];
          tmem_st32(tl + S_COL0 + b * BN, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = pk[32 + j];
          tmem_st32(tl + S_COL0 + b * BN + 32, r);
        }
        // PV(t-1) must have landed before O~ is touched and before PV(t)
        // is released.  Waiting on every tile keeps this thread's count of
        // the PV barrier's phases exact: at this point PV(t) is not issued
        // yet, so at most PV(t-1) is outstanding and the parity test cannot
        // alias.  PV(t-1) was issued when softmax(t) started, so the wait
        // rarely blocks.
        if (t > 0) {
          ok = wait_bar(bar(C::B_OD), static_cast<uint32_t>(t - 1) & 1u, abort_flag,
                        &g_umma_status, 0x32, lim);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, need)) {
          // Rescale O~ in TMEM by alpha (1 for rows whose max did not move).
          uint32_t r[D / 32][32];
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tl + O_COL + cc * 32, r[cc]);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            reg_fence32(r[cc]);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              r[cc][j] = __float_as_uint(__uint_as_float(r[cc][j]) * alpha);
            tmem_st32(tl + O_COL + cc * 32, r[cc]);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::B_PF + b));
      }

      if (ok) {
        // PV(nt-1) is the only one that can still be outstanding.
        ok = wait_bar(bar(C::B_OD), static_cast<uint32_t>(nt - 1) & 1u, abort_flag,
                      &g_umma_status, 0x33, lim);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        // Canonical state: rescale once from m_used to the exact running max.
        const float fin = (m_used == m_true) ? 1.f : ex2(m_used - m_true);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tl + O_COL + cc * 32, r);
          tmem_wait_ld();
          reg_fence32(r);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(a.o + sidx * D + cc * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(r[4 * j + 0]) * fin,
                                   __uint_as_float(r[4 * j + 1]) * fin,
                                   __uint_as_float(r[4 * j + 2]) * fin,
                                   __uint_as_float(r[4 * j + 3]) * fin);
          }
        }
        if (valid) {
          a.l[sidx] = l_run * fin;
          a.m[sidx] = m_moved ? m_true * kLn2 : m_ld;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
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
                     const CUtensorMap& tv, cudaStream_t st) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(umma_update_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.c + BM - 1) / BM), a.heads, a.nwork);
  umma_update_kernel<D><<<grid, NTHREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_umma_update(const FwdArgs& a, int d, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  return d == 128 ? launch_d<128>(a, tq, tk, tv, st) : launch_d<64>(a, tq, tk, tv, st);
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
