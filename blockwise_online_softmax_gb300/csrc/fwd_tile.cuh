// Tile machinery shared by the tcgen05 forward kernels (the one-step block
// update and the fused ring): the visit of a
// CTA's query tiles over a K/V block, the per-tile softmax of one row, and
// the per-step visit table of the fused ring.  Device code only, included
// by the kernel translation units.
#pragma once
#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "ra_internal.h"

namespace ra {
namespace fwd {

constexpr int BM = 128;  // rows per query tile (= TMEM lanes)
constexpr int NQ = 2;    // query tiles per CTA
constexpr int BN = 128;  // keys per K/V tile
constexpr uint32_t CHUNK_BYTES = 128 * 128;  // 128 rows x 128 B (one swizzle span)
constexpr uint32_t TMEM_COLS = 512;
// Rescale rule: each row's max in use follows the exact running max (the
// threshold is 0, in log2 units), so the largest weight of a row is exactly
// 1 and exact in bf16.
constexpr float RESCALE_THRESHOLD = 0.0f;

// The K/V tiles a CTA visits: the union of its two query tiles' ranges
// [ta[g], tb[g]), in increasing order.  Ranges that overlap or touch merge;
// otherwise the visit is two runs with the gap skipped.
struct TileSeq {
  int a0;  // first tile of the first run
  int na;  // length of the first run
  int b0;  // first tile of the second run
  int n;   // total tiles
  __device__ __forceinline__ int at(int k) const { return k < na ? a0 + k : b0 + (k - na); }
};

__device__ __forceinline__ TileSeq make_seq(const int (&ta)[NQ], const int (&tb)[NQ]) {
  // Written with selects only: a runtime index into ta/tb would put them
  // in local memory.
  const int a0 = ta[0], b0 = tb[0], a1 = ta[1], b1 = tb[1];
  const int n0 = b0 - a0, n1 = b1 - a1;
  TileSeq q{0, 0, 0, 0};
  if (n0 <= 0 && n1 <= 0) return q;
  if (n0 <= 0 || n1 <= 0) {
    q.a0 = n0 > 0 ? a0 : a1;
    q.na = n0 > 0 ? n0 : n1;
  } else if (a1 <= b0 && a0 <= b1) {
    q.a0 = a0 < a1 ? a0 : a1;
    q.na = (b0 > b1 ? b0 : b1) - q.a0;
  } else {
    const bool f0 = a0 < a1;
    q.a0 = f0 ? a0 : a1;
    q.na = f0 ? n0 : n1;
    q.b0 = f0 ? a1 : a0;
    q.n = f0 ? n1 : n0;
  }
  q.n += q.na;
  return q;
}

// One K/V tile of one softmax row (TMEM lane): wait for S (barrier b_s,
// phase parity `parity`), mask the keys outside [row_lo, row_hi) on tiles
// that cut that interval (tiles full_0 .. full_0 + n_full - 1 need no mask),
// move the row max, rescale O~ in TMEM when it moved, write P over S and
// arrive on b_p.  The running state is m_used / m_true (log2 units) and
// l_run.  Returns false after an abort.  `status` is the launch's device
// status word.
template <int D>
__device__ __forceinline__ bool softmax_tile(uint32_t tl, uint32_t s_col, uint32_t o_col, int t,
                                             int row_lo, int row_hi, int full_0, int n_full,
                                             float sl2, uint64_t sl2x2, uint32_t b_s,
                                             uint32_t b_p, uint32_t parity,
                                             volatile int* abort_flag, int* status, long long lim,
                                             float& m_used, float& m_true, bool& m_moved,
                                             float& l_run) {
  bool ok = wait_bar(b_s, parity, abort_flag, status, 0x31, lim);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  tc_fence_after();
  // S row: 128 fp32 scores, loaded once into registers.
  uint32_t sr[BN / 32][32];
#pragma unroll
  for (int cc = 0; cc < BN / 32; ++cc) tmem_ld32(tl + s_col + cc * 32, sr[cc]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < BN / 32; ++cc) reg_fence32(sr[cc]);
#define RA_S(j) __uint_as_float(sr[(j) >> 5][(j) & 31])
  // Mask: key j of this tile is allowed iff lo_j <= j < hi_j.
  if (static_cast<unsigned>(t - full_0) >= static_cast<unsigned>(n_full)) {
    const int lo_j = row_lo - t * BN, hi_j = row_hi - t * BN;
#pragma unroll
    for (int j = 0; j < BN; ++j)
      if (j < lo_j || j >= hi_j) sr[j >> 5][j & 31] = 0xff800000u;  // -inf
  }
  // Row max: four independent chains over columns 0..127, two new
  // values per three-input max.
  float mx0 = fmaxf(RA_S(0), RA_S(4)), mx1 = fmaxf(RA_S(1), RA_S(5));
  float mx2 = fmaxf(RA_S(2), RA_S(6)), mx3 = fmaxf(RA_S(3), RA_S(7));
#pragma unroll
  for (int j = 8; j < BN; j += 8) {
    mx0 = fmax3(mx0, RA_S(j + 0), RA_S(j + 4));
    mx1 = fmax3(mx1, RA_S(j + 1), RA_S(j + 5));
    mx2 = fmax3(mx2, RA_S(j + 2), RA_S(j + 6));
    mx3 = fmax3(mx3, RA_S(j + 3), RA_S(j + 7));
  }
  static_assert(BN % 8 == 0, "the max loop covers columns in groups of 8");
  const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
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
  // O~_g is stable here: S_g(t) comes from QK_g(t), which the MMA thread
  // issued after PV_g(t-1), and the commit that signalled S_g(t)
  // covers every earlier MMA.  Rescale it before any of P_g(t) is
  // published, since PV_g(t) accumulates on top.
  if (__any_sync(0xffffffffu, need)) {
    // 32 columns at a time: the S row still occupies 128 registers.
    const uint64_t al2 = f2pack(alpha, alpha);
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t r[32];
      tmem_ld32(tl + o_col + cc * 32, r);
      tmem_wait_ld();
      reg_fence32(r);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float y0, y1;
        f2unpack(fmul2(f2pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), al2), y0,
                 y1);
        r[j] = __float_as_uint(y0);
        r[j + 1] = __float_as_uint(y1);
      }
      tmem_st32(tl + o_col + cc * 32, r);
    }
  }
  const float mref = (m_used == -INFINITY) ? 0.f : m_used;
  const uint64_t nmref2 = f2pack(-mref, -mref);
  // P = 2^(s * log2(e)/sqrt(d) - m), two lanes per FFMA2; row sum in
  // two FADD2 accumulators; P rounded to bf16 in pairs, written over
  // the first half of the same registers.
  uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int j = 0; j < BN; j += 4) {
    float x0, x1, x2, x3;
    f2unpack(ffma2(f2pack(RA_S(j), RA_S(j + 1)), sl2x2, nmref2), x0, x1);
    f2unpack(ffma2(f2pack(RA_S(j + 2), RA_S(j + 3)), sl2x2, nmref2), x2, x3);
    const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
    acc0 = fadd2(acc0, f2pack(p0, p1));
    acc1 = fadd2(acc1, f2pack(p2, p3));
    // pair k = j/2 goes to word k; k < j, so the scores it overwrites
    // have already been read.
    sr[(j / 2) >> 5][(j / 2) & 31] = bf16x2_rn(p0, p1);
    sr[(j / 2 + 1) >> 5][(j / 2 + 1) & 31] = bf16x2_rn(p2, p3);
  }
  tmem_st32(tl + s_col, sr[0]);
  tmem_st32(tl + s_col + 32, sr[1]);
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(b_p);
#undef RA_S
  float sa, sb;
  f2unpack(fadd2(acc0, acc1), sa, sb);
  l_run = l_run * alpha + (sa + sb);
  return true;
}


// Rank i at ring step s: the same work item as the one-step launch.
__device__ __forceinline__ Work ring_work(const FwdArgs& a, int i, int s) {
  Work wk;
  const int j = (i - s + a.P) % a.P;
  wk.q_base = static_cast<long long>(i) * a.cq;
  wk.kv_base = static_cast<long long>(j) * a.ck;
  wk.state_base = wk.q_base;
  wk.qmap = PosMap{a.layout, a.P, a.cq, i, wk.q_base};
  wk.kmap = PosMap{a.layout, a.P, a.ck, j, wk.kv_base};
  return wk;
}

// The visit of one step: the union of the groups' tile ranges, where each
// group's run starts in it (ks) and its length (ne), and the K/V block's
// first row.
struct StepVisit {
  long long kv_base;
  TileSeq seq;
  int ta[NQ], tb[NQ];  // the groups' tile ranges within the K/V block
  int ks[NQ], ne[NQ];
};

// Steps of one fused launch at most (the visit table is in shared memory).
constexpr int kRingMaxSteps = 256;

__device__ __forceinline__ StepVisit step_visit(const FwdArgs& a, int i, int s, long long row0,
                                                long long vb) {
  const Work wk = ring_work(a, i, s);
  int ta[NQ], tb[NQ];
#pragma unroll
  for (int g = 0; g < NQ; ++g)
    tile_range(a, wk, row0 + g * BM, row0 + (g + 1) * BM, vb, BN, &ta[g], &tb[g]);
  StepVisit v;
  v.seq = make_seq(ta, tb);
#pragma unroll
  for (int g = 0; g < NQ; ++g) {
    v.ta[g] = ta[g];
    v.tb[g] = tb[g];
    v.ne[g] = tb[g] > ta[g] ? tb[g] - ta[g] : 0;
    v.ks[g] = ta[g] < v.seq.a0 + v.seq.na ? ta[g] - v.seq.a0 : v.seq.na + (ta[g] - v.seq.b0);
  }
  v.kv_base = wk.kv_base;
  return v;
}

// The first step at or after s whose visit (in the table) is not empty, or
// P if none.
__device__ __forceinline__ int next_step(const StepVisit* rec, int P, int s) {
  while (s < P && rec[s].seq.n == 0) ++s;
  return s;
}

}  // namespace fwd
}  // namespace ra
