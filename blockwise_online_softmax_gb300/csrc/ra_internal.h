// Internal interface between the C-ABI host code (ra_api.cu) and the
// kernel translation units.  Not installed and not part of the ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace ra {

// Token layouts: how the rows of a block map to global sequence positions.
// Positions grow with the row index inside a block under all three, so
// the keys of a block that a query may see always form one interval of
// row indices.
enum Layout : int {
  kContiguous = 0,  // block b holds positions [b*c, (b+1)*c)
  kZigzag = 1,      // block b holds chunks b and 2P-1-b of length c/2
  kStriped = 2,     // block b holds positions b, b+P, b+2P, ...
};

// Position map of one block: layout, rank count, block length, block index
// and (contiguous only) the position of row 0.
struct PosMap {
  int layout;
  int P;
  long long c;
  long long blk;
  long long off;
};

__host__ __device__ inline long long pos_of(const PosMap& m, long long r) {
  if (m.layout == kZigzag) {
    const long long h = m.c >> 1;
    return r < h ? m.blk * h + r : (2LL * m.P - 1 - m.blk) * h + (r - h);
  }
  if (m.layout == kStriped) return r * m.P + m.blk;
  return m.off + r;
}

__host__ __device__ inline long long clamp_ll(long long x, long long lo, long long hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

// Number of rows r in [0, c) of the block whose position is below x.
__host__ __device__ inline long long count_below(const PosMap& m, long long x) {
  if (m.layout == kZigzag) {
    const long long h = m.c >> 1;
    return clamp_ll(x - m.blk * h, 0, h) + clamp_ll(x - (2LL * m.P - 1 - m.blk) * h, 0, h);
  }
  if (m.layout == kStriped) {
    const long long y = x - m.blk;  // rows r with r*P < y
    return y <= 0 ? 0 : clamp_ll((y + m.P - 1) / m.P, 0, m.c);
  }
  return clamp_ll(x - m.off, 0, m.c);
}

// The mask: key position kp is allowed for query position qp when both are
// below n_valid, lie in the same document, and (causal) kp <= qp and
// (window > 0) |qp - kp| < window.  Documents are the position intervals
// [cu[d], cu[d+1]) of cu_seqlens; positions before cu[0] or at or past
// cu[ndocs] belong to none.  Positions may be negative (block offsets are
// free in a single block update).
struct MaskArgs {
  int causal;
  int ndocs;               // 0: one document holding every position
  long long window;        // 0: no window
  long long n_valid;       // positions >= n_valid are padding
  const int* cu_seqlens;   // device array of ndocs + 1 positions, or null
};

// Positions below this bound may hold a query or a key.
__device__ __forceinline__ long long valid_bound(const MaskArgs& k) {
  long long x = k.n_valid;
  if (k.ndocs > 0) {
    const long long e = k.cu_seqlens[k.ndocs];
    x = e < x ? e : x;
  }
  return x;
}

// Allowed key positions [*plo, *phi) for a query position qp below
// valid_bound; false if qp lies before the first document.
__device__ __forceinline__ bool allowed_positions(const MaskArgs& k, long long qp, long long* plo,
                                                  long long* phi) {
  long long lo = -(1LL << 60), hi = k.n_valid;
  if (k.ndocs > 0) {
    if (qp < k.cu_seqlens[0]) return false;
    // Document of qp: the last d with cu[d] <= qp (cu nondecreasing).
    int a = 0, b = k.ndocs;
    while (b - a > 1) {
      const int mid = (a + b) >> 1;
      if (k.cu_seqlens[mid] <= qp) a = mid; else b = mid;
    }
    lo = k.cu_seqlens[a];
    const long long e = k.cu_seqlens[a + 1];
    hi = e < hi ? e : hi;
  }
  if (k.causal) hi = qp + 1 < hi ? qp + 1 : hi;
  if (k.window > 0) {
    const long long w0 = qp - k.window + 1;
    lo = w0 > lo ? w0 : lo;
    if (!k.causal) hi = qp + k.window < hi ? qp + k.window : hi;
  }
  *plo = lo;
  *phi = hi;
  return true;
}

// One launch of a block-update kernel.  It either folds a single (Q
// block, K/V block) pair (mode 0) or runs one ring step for the virtual
// ranks i0 .. i0 + nwork - 1 (mode 1).
struct FwdArgs {
  const void* q;  // tensor base pointers (token-major)
  const void* k;
  const void* v;
  float* m;       // state base pointers
  float* l;
  float* o;
  long long cq;       // query rows per block
  long long ck;       // key rows per block
  long long q_rows;   // rows in the q tensor
  long long kv_rows;  // rows in the k/v tensors
  long long q_off;    // mode 0, contiguous layout: position of q row 0
  long long kv_off;   // mode 0, contiguous layout: position of k/v row 0
  int q_blk;          // mode 0: block index of the q block in the layout
  int kv_blk;         // mode 0: block index of the k/v block
  int layout;
  int heads;
  int kv_heads;
  int mode;  // 0 = one block pair, 1 = ring step s
  int P;
  int s;
  int nwork;         // grid.z: number of (i, j) pairs in the launch
  int i0;            // mode 1: grid.z index w runs rank i0 + w
  float scale;       // 1/sqrt(d)
  float scale_log2;  // log2(e)/sqrt(d)
  long long wait_limit;  // SM cycles before a bounded wait gives up
  MaskArgs mask;
  int h0;  // fused ring: first query head of the launch (grid.y runs h0 .. h0 + nh - 1)
  int nh;  // fused ring: query heads in the launch (0: all `heads`)
  int ring_lc;  // fused ring: log2 of the heads per chunk of the launch order (set by its launcher)
  int o_tma;    // 1 when the launch has a tensor map over o for its tile stores (bf16 kernels)
};

// Decoded work item of grid.z index w.
struct Work {
  long long q_base;      // first Q row of the block, in the q tensor
  long long kv_base;     // first K/V row of the block, in the k/v tensors
  long long state_base;  // first state row
  PosMap qmap;           // positions of the query rows
  PosMap kmap;           // positions of the key rows
};

__host__ __device__ inline Work decode_work(const FwdArgs& a, int w) {
  Work wk;
  if (a.mode == 0) {
    wk.q_base = 0;
    wk.kv_base = 0;
    wk.state_base = 0;
    wk.qmap = PosMap{a.layout, a.P, a.cq, a.q_blk, a.q_off};
    wk.kmap = PosMap{a.layout, a.P, a.ck, a.kv_blk, a.kv_off};
  } else {
    const int i = a.i0 + w;
    const int j = (i - a.s + a.P) % a.P;  // K/V block held at step s
    wk.q_base = static_cast<long long>(i) * a.cq;
    wk.kv_base = static_cast<long long>(j) * a.ck;
    wk.state_base = wk.q_base;
    wk.qmap = PosMap{a.layout, a.P, a.cq, i, wk.q_base};
    wk.kmap = PosMap{a.layout, a.P, a.ck, j, wk.kv_base};
  }
  return wk;
}

// Key-row interval [*lo, *hi) of the K/V block that query row r of the
// block may see; empty (lo >= hi) for a padding row.
__device__ __forceinline__ void row_keys(const FwdArgs& a, const Work& wk, long long r,
                                         long long vb, long long* lo, long long* hi) {
  const long long qp = pos_of(wk.qmap, r);
  long long plo, phi;
  if (qp >= vb || !allowed_positions(a.mask, qp, &plo, &phi)) {
    *lo = 0;
    *hi = 0;
    return;
  }
  *lo = count_below(wk.kmap, plo);
  *hi = count_below(wk.kmap, phi);
}

// Key tiles [*t0, *t1) (tiles of bn rows) that some valid row of query rows
// [r0, r1) may see.  Query positions and both interval ends grow with the
// row, so the first and the last valid row bound the range.  (Rows before
// the first document come first; they give the empty interval [0, 0),
// which only widens the range.)
__device__ __forceinline__ void tile_range(const FwdArgs& a, const Work& wk, long long r0,
                                           long long r1, long long vb, int bn, int* t0, int* t1) {
  *t0 = 0;
  *t1 = 0;
  const long long nvr = count_below(wk.qmap, vb);  // valid rows are a prefix
  if (r1 > wk.qmap.c) r1 = wk.qmap.c;
  if (r1 > nvr) r1 = nvr;
  if (r0 >= r1) return;
  long long lo0, hi0, lo1, hi1;
  row_keys(a, wk, r0, vb, &lo0, &hi0);
  row_keys(a, wk, r1 - 1, vb, &lo1, &hi1);
  if (hi1 <= lo0) return;
  *t0 = static_cast<int>(lo0 / bn);
  *t1 = static_cast<int>((hi1 + bn - 1) / bn);
}

// One launch of the decode chunk kernel: n_q query tokens against n_kv
// keys cut into nshard shards of shard_len keys, each shard into nsplit
// chunks of `chunk` keys (a multiple of 128).  CTA (split, kv head, shard)
// writes the partial state of its KV head's g * n_q rows to
// pm/pl [nshard][nsplit][n_q][heads] and po [..][d].
struct DecArgs {
  const void* q;  // [n_q, heads, d] bf16
  float* pm;
  float* pl;
  float* po;
  long long n_q;
  long long n_kv;
  long long shard_len;
  long long chunk;
  long long q_off;   // position of query row 0
  long long kv_off;  // position of key 0
  int heads;
  int kv_heads;
  int nsplit;
  int nshard;
  long long tq;      // query tokens per row tile (g * tq <= 128 rows)
  int ntile;         // row tiles: ceil(n_q / tq); grid.x = nsplit * ntile
  float scale_log2;  // log2(e)/sqrt(d)
  long long wait_limit;
  MaskArgs mask;
};

// One launch of a backward kernel: the forward's launch description (q, k,
// v, blocks, ranks, mask; m, l, o unused) plus the gradient tensors.
struct BwdArgs {
  FwdArgs f;
  const float* lse;   // [q_rows, heads], natural log
  const float* dvec;  // [q_rows, heads]: rowsum(dO * O)
  float* dq;          // [q_rows, heads, d], accumulated
  float* dk;          // [kv_rows, kv_heads, d], accumulated
  float* dv;
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Kernel launchers.  Each returns cudaSuccess or the launch error.
cudaError_t launch_state_init(float* m, float* l, float* o, long long rows, int heads, int d,
                              cudaStream_t st);
cudaError_t launch_merge(float* m_a, float* l_a, float* o_a, const float* m_b, const float* l_b,
                         const float* o_b, long long rows, int heads, int d, cudaStream_t st);
cudaError_t launch_finalize(const float* m, const float* l, const float* o, float* out,
                            float* lse, long long rows, int heads, int d, cudaStream_t st);
cudaError_t launch_simt_update(const FwdArgs& a, int d, cudaStream_t st);
// The whole fp32 ring forward in one launch: a.o is the output [rows,
// heads, d] and a.m the LSE [rows, heads] (natural log); a.l is unused.
cudaError_t launch_simt_ring(const FwdArgs& a, int d, cudaStream_t st);
// One block-update launch (bf16).  With a.o_tma set, `to` maps the state
// a.o like launch_umma_ring's output map (rows: a.q_rows) and the kernel
// stores whole state tiles with it.
cudaError_t launch_umma_update(const FwdArgs& a, int d, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& to, cudaStream_t st);
// The whole ring forward of every rank in one launch (bf16): a.o is the
// output [rows, heads, d] and a.m the LSE [rows, heads]; a.l is unused.
// With a.o_tma set, `to` maps a.o (fp32, dims (d, heads, rows), box 32 x 1
// x 128, 128-byte swizzle) and the kernel stores whole output tiles with it.
cudaError_t launch_umma_ring(const FwdArgs& a, int d, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, cudaStream_t st);
cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st);
cudaError_t launch_decode_tc(const DecArgs& a, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_decode_combine(float* m, float* l, float* o, const float* pm, const float* pl,
                                  const float* po, long long rows_per_shard, int nsplit,
                                  int nshard, int d, cudaStream_t st);
// Folds the np partial states of every (row, head) (partial p of row rh at
// p * rows + rh) and finalizes into out [rows, d] and lse [rows].
cudaError_t launch_decode_reduce(float* out, float* lse, const float* pm, const float* pl,
                                 const float* po, long long rows, int np, int d, cudaStream_t st);

// Device status words (one per kernel translation unit): read and clear.
cudaError_t take_umma_status(int* code);
cudaError_t take_simt_status(int* code);
cudaError_t take_decode_status(int* code);
cudaError_t launch_bwd_pre(const float* out, const void* dout, float* dvec, long long rows,
                           int heads, int d, cudaStream_t st);
cudaError_t launch_bwd_dq(const BwdArgs& b, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const BwdArgs& b, int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t st);
cudaError_t take_bwd_status(int* code);

}  // namespace ra
