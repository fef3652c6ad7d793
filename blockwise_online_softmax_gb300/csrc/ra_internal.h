// Internal interface between the C-ABI host code (ra_api.cu) and the
// kernel translation units.  Not installed and not part of the ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace ra {

// One launch of the block-update kernel.  It either folds a single (Q
// block, K/V block) pair (mode 0) or runs one ring step for every virtual
// rank (mode 1).
struct FwdArgs {
  const void* q;  // tensor base pointers (token-major)
  const void* k;
  const void* v;
  float* m;       // state base pointers
  float* l;
  float* o;
  long long c;        // block length: rows per Q block and per K/V block
  long long q_rows;   // rows in the q tensor
  long long kv_rows;  // rows in the k/v tensors
  long long q_off;    // mode 0: global position of q row 0
  long long kv_off;   // mode 0: global position of k/v row 0
  int heads;
  int kv_heads;
  int causal;
  int mode;  // 0 = one block pair, 1 = ring step s over all ranks
  int P;
  int s;
  int nwork;         // grid.z: number of (i, j) pairs in the launch
  float scale;       // 1/sqrt(d)
  float scale_log2;  // log2(e)/sqrt(d)
  long long wait_limit;  // SM cycles before a bounded wait gives up
};

// Decoded work item of grid.z index w.
struct Work {
  long long q_base;      // first Q row of the block, in the q tensor
  long long kv_base;     // first K/V row of the block, in the k/v tensors
  long long state_base;  // first state row
  long long q_pos0;      // global position of the block's first query
  long long kv_pos0;     // global position of the block's first key
};

__host__ __device__ inline Work decode_work(const FwdArgs& a, int w) {
  Work wk;
  if (a.mode == 0) {
    wk.q_base = 0;
    wk.kv_base = 0;
    wk.state_base = 0;
    wk.q_pos0 = a.q_off;
    wk.kv_pos0 = a.kv_off;
  } else {
    const int i = a.causal ? a.s + w : w;      // causal: ranks i < s hold a future block
    const int j = (i - a.s + a.P) % a.P;       // K/V block held at step s
    wk.q_base = static_cast<long long>(i) * a.c;
    wk.kv_base = static_cast<long long>(j) * a.c;
    wk.state_base = wk.q_base;
    wk.q_pos0 = wk.q_base;
    wk.kv_pos0 = wk.kv_base;
  }
  return wk;
}

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
cudaError_t launch_umma_update(const FwdArgs& a, int d, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st);

// Device status words (one per kernel translation unit): read and clear.
cudaError_t take_umma_status(int* code);
cudaError_t take_simt_status(int* code);

}  // namespace ra
