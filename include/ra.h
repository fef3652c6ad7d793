/*
 * ra.h -- C ABI of the GB300 blockwise online-softmax library (libra.so).
 *
 * The library computes the per-device hot path of Ring Attention on one
 * GPU.  Virtual rank i keeps its query block Q_i.  At ring step s it folds
 * in the K/V block j = (i - s) mod P by the online-softmax rescale.  The
 * running state (m, l, O~) stays in HBM between steps.  Then comes a merge
 * or a finalize.
 *
 * Sources, by page title and section:
 *  [MATH]  "Ring Attention Math Deep -- Belgavi.AI Lab": "The online-softmax
 *          identity that makes streaming legal", "The ring schedule:
 *          passing K/V around", "Accumulation math, step by step", "A worked
 *          numeric example".
 *  [PB]    "Ring Attention Paper Breakdown: Blockwise Distributed
 *          Transformers for Near-Infinite Context": "2. Ring Topology &
 *          Asynchronous Double-Buffered KV Circulation", "3. Cross-Device
 *          Online Softmax Accumulator Math", "4. Zero-Overhead Overlapping
 *          Condition & Roofline Analysis".
 *  [XF]    xf_ring_attention (aicassindra.com): "The architecture: every
 *          piece explained", "End-to-end flow".
 *  [SP]    "Ring Attention：把超长序列沿设备环流动": "环是怎样工作的",
 *          "局部 Softmax 为什么不能直接相加", "Causal Attention
 *          让环不再完全对称", "位置编码必须使用全局位置".
 *  [GUIDE] "RingAttention: Scaling LLM Context to 10M Tokens": "1.
 *          Incremental Online Softmax Accumulation", "Causal Masking:
 *          Striped and Zig-Zag RingAttention".
 *  [TEST]  "Ring Attention：把超长序列沿设备环流动": "正确性测试应覆盖哪些边界"
 *          (its lists "分片边界" and "Mask 与位置").
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout.  All tensors are token-major and dense, with batch 1:
 *   Q:  [rows, heads, d]       (bf16 or fp32, as `dtype` says)
 *   K, V: [rows, kv_heads, d]
 *   m, l: [rows, heads] fp32   (running max, running sum of exp)
 *   o (O~): [rows, heads, d] fp32 (unnormalized running output)
 * Query head h reads KV head h / (heads / kv_heads), so consecutive groups
 * of query heads share one KV head (GQA; heads % kv_heads must be 0).
 *
 * Scores.  s = (q . k) / sqrt(d), with 1/sqrt(d) rounded to fp32 [MATH],
 * [PB] step 1.  The state is in natural-log units: m = max s, l = sum
 * exp(s - m), o = sum exp(s - m) v.
 *
 * Causal mask.  Key t is allowed for query r when kv_off + t <= q_off + r,
 * on global token positions [SP] "位置编码必须使用全局位置".
 *
 * Types.  dtype RA_BF16 runs the tcgen05 tensor-core path: bf16 operands,
 * fp32 accumulation, and P rounded to bf16 before the P V product.  dtype
 * RA_F32 runs an fp32 FFMA path.  d must be 64 or 128.
 *
 * Pointers.  All pointers are device pointers, except for the *_host
 * call.  Each pointer must be 16-byte aligned.  The caller owns every
 * buffer.  No call keeps a pointer after it returns.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).
 * Compute calls only enqueue work and return.  A call returns RA_OK once
 * its launches are enqueued.  A launch failure returns RA_ERR_CUDA.
 * Device-side wait timeouts are reported by ra_device_status().
 *
 * Errors.  Every call returns an ra_status.  Arguments are checked before
 * any launch, and a bad argument returns RA_ERR_INVALID without touching
 * memory.  ra_last_error() returns a message for the calling thread's last
 * failure.  Zero-size work (c == 0 or N == 0) is RA_OK and launches
 * nothing.
 */
#ifndef RA_H
#define RA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID = -1,     /* bad argument: null/misaligned pointer, shape, dtype */
  RA_ERR_UNSUPPORTED = -2, /* well-formed but outside what the kernels handle */
  RA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  RA_ERR_TIMEOUT = -4,     /* a kernel gave up a bounded wait (see ra_device_status) */
  RA_ERR_ALLOC = -5        /* stream-ordered allocation of scratch failed */
} ra_status;

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

/*
 * Token layouts: which global sequence positions the c rows of block b
 * (rows [b*c, (b+1)*c) of a ring tensor) hold.  [PB] section 5 and [GUIDE]
 * "Causal Masking: Striped and Zig-Zag RingAttention" give the two
 * balanced assignments; [MATH] "Causal masking, load balance, and other
 * wrinkles" names them.
 *   RA_LAYOUT_CONTIGUOUS: row r holds position b*c + r.
 *   RA_LAYOUT_ZIGZAG:     the sequence is cut into 2P chunks of c/2; block
 *                         b holds chunk b, then chunk 2P-1-b.
 *   RA_LAYOUT_STRIPED:    row r holds position r*P + b (token t lives on
 *                         rank t mod P).
 * The caller lays the tensors out that way; the library only maps rows to
 * positions for the mask.  Under every layout positions grow with the row
 * index inside a block.
 */
typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0,
  RA_LAYOUT_ZIGZAG = 1,
  RA_LAYOUT_STRIPED = 2
} ra_layout;

/* Kernel kinds for the tracing calls. */
typedef enum {
  RA_KERNEL_STATE_INIT = 0,
  RA_KERNEL_BLOCK_UPDATE_BF16 = 1, /* tcgen05 / TMEM / TMA kernel */
  RA_KERNEL_BLOCK_UPDATE_F32 = 2,  /* fp32 FFMA kernel */
  RA_KERNEL_MERGE = 3,
  RA_KERNEL_FINALIZE = 4,
  RA_KERNEL_DECODE_SPLIT = 5,   /* decode split-K chunk kernel (tcgen05, TMA) */
  RA_KERNEL_DECODE_COMBINE = 6, /* folds split partial states: into a shard's state
                                   (ra_decode_partial) or over every shard with the
                                   finalize (ra_decode_forward) */
  RA_KERNEL_BWD_PRE = 7,        /* backward: D = rowsum(dO * O) */
  RA_KERNEL_BWD_DQ = 8,         /* backward: dQ (tcgen05, Q-stationary) */
  RA_KERNEL_BWD_DKDV = 9,       /* backward: dK, dV (tcgen05, K/V-stationary) */
  RA_KERNEL_RING_FUSED_BF16 = 10, /* the whole bf16 ring forward in one launch (tcgen05) */
  RA_KERNEL_RING_FUSED_F32 = 11,  /* the whole fp32 ring forward in one launch (FFMA) */
  RA_KERNEL_KINDS = 12
} ra_kernel_kind;

/*
 * ra_state_init -- set c rows of state to the merge identity (m, l, O~) =
 * (-inf, 0, 0) [XF] "End-to-end flow", [MATH] "Accumulation math, step by
 * step".
 *   m, l: [c, heads] fp32 ; o: [c, heads, d] fp32 (written).
 */
int ra_state_init(float* m, float* l, float* o, long long c, int d, int heads, void* stream);

/*
 * ra_block_update -- fold one K/V block into the running state of one query
 * block.  This is [PB] section 3, steps 1-7, also [MATH] "Accumulation math,
 * step by step" and [GUIDE] section 1, in the unnormalized-O~ form:
 *   S = Q K^T / sqrt(d);  m' = max(m, rowmax S);  alpha = exp(m - m');
 *   P = exp(S - m');  l' = alpha l + rowsum P;  O~' = alpha O~ + P V.
 *   q: [c, heads, d], the first row of Q_i (global position q_off).
 *   k, v: [c, kv_heads, d], the first row of K_j, V_j (global position kv_off).
 *   m, l, o: the state of Q_i's c rows, updated in place.  On return, m is
 *           the exact running max of the allowed scores (-inf for a row
 *           with none yet).  l and o are taken relative to that m.
 *   causal: nonzero applies the causal mask on global positions.  The
 *           kernel skips key tiles that lie wholly in the future and masks
 *           elementwise only the tiles that cross the diagonal [SP] "Causal
 *           Attention 让环不再完全对称".  A row with no allowed key keeps
 *           its state.
 *   dtype: RA_BF16 (q, k, v are bf16) or RA_F32 (q, k, v are fp32).
 */
int ra_block_update(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                    long long c, int d, int heads, int kv_heads, long long q_off,
                    long long kv_off, int causal, int dtype, void* stream);

/*
 * ra_merge -- a <- a (+) b on c rows of two partial states: m = max(m_a,
 * m_b), then each side is rescaled by exp(m_side - m) and the two are added
 * [XF] "The architecture: every piece explained" (online softmax
 * accumulator), [SP] "局部 Softmax 为什么不能直接相加".  The identity
 * state is neutral.  m_a/l_a/o_a are updated in place.  b is read only and
 * must not overlap a.
 */
int ra_merge(float* m_a, float* l_a, float* o_a, const float* m_b, const float* l_b,
             const float* o_b, long long c, int d, int heads, void* stream);

/*
 * ra_finalize -- out = O~ / l and lse = m + ln l ([MATH] "After the final
 * block: out = o / l").  The log-sum-exp is kept for backward recompute
 * ([SP] "Backward 需要让梯度也沿环传播").  A row with l = 0 gets out = 0
 * and lse = -inf.
 *   out: [c, heads, d] fp32 and lse: [c, heads] fp32 (written).  `out` may
 *   be the same buffer as `o`, and `lse` may be the same buffer as `m`
 *   (in place).  Any other overlap is not allowed.
 */
int ra_finalize(const float* m, const float* l, const float* o, float* out, float* lse,
                long long c, int d, int heads, void* stream);

/*
 * ra_ring_step -- one step s of the ring schedule for all P virtual ranks
 * at once ([MATH] "The ring schedule: passing K/V around", [PB] section 2).
 * Virtual rank i folds block j = (i - s) mod P of K/V into its state.
 * Under `causal`, ranks whose block j lies in the future (j > i) are
 * skipped at launch granularity.  Each rank's diagonal block (s = 0) is
 * masked elementwise.  The "hop" is the block index advancing on the
 * device.  No bytes move.
 *   q: [N, heads, d]; k, v: [N, kv_heads, d]; m, l: [N, heads]; o: [N, heads, d].
 *   N = P * c, 0 <= s < P.  Block i holds tokens [i*c, (i+1)*c).
 */
int ra_ring_step(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                 long long N, int P, int s, int causal, int d, int heads, int kv_heads,
                 int dtype, void* stream);

/*
 * ra_ring_forward -- the whole per-device forward loop of [MATH]
 * "Accumulation math, step by step" for all P virtual ranks: every rank i
 * folds the K/V blocks j = (i - s) mod P, s = 0 .. P-1, into the state of
 * its queries, then finalizes ([PB] §2).
 *   out: [N, heads, d] fp32: O = O~ / l (0 for a row that sees no key).
 *   lse: [N, heads] fp32: LSE = m + ln l (-inf for such a row).
 * bf16 with P <= 256 (tcgen05), and fp32 (FFMA): one fused launch.  Each
 * rank's state stays on chip across all P steps and the kernel writes out
 * and lse once; no scratch.  bf16 with P > 256: the state init, P
 * ring-step launches with the O~ state in `out` and m in `lse`, then the
 * finalize.  The l state ([N, heads] fp32) is then the only scratch,
 * allocated stream-ordered on `stream` from the library's scratch pool
 * (see ra_cached_memory) and freed the same way; a failed allocation
 * returns RA_ERR_ALLOC.  Both give the results of init + ra_ring_step for
 * s = 0..P-1 + ra_finalize, the fused launches up to the last roundings of
 * the finalize.
 */
int ra_ring_forward(const void* q, const void* k, const void* v, float* out, float* lse,
                    long long N, int P, int causal, int d, int heads, int kv_heads, int dtype,
                    void* stream);

/*
 * ra_ring_forward_host -- ra_ring_forward on HOST buffers.  It copies q, k
 * and v to device buffers (stream-ordered, from the scratch pool), runs the
 * ring, copies out and lse back, frees the buffers, and synchronizes
 * `stream` before it returns.  Pinned host memory makes the copies
 * asynchronous DMA.  In bf16 the work is split into up to 8 groups of KV
 * heads (heads never interact): group G runs while group G + 1 copies in
 * and group G - 1 copies out; the copies go on two streams the call
 * creates and destroys, the groups' launches alternate between `stream`
 * and a third such stream, and events order them all.  The results are
 * those of ra_ring_forward, bit for bit.  Device wait timeouts are checked
 * before return and give RA_ERR_TIMEOUT.  The pages have no counterpart:
 * this is the host-to-host form of the call, for callers whose tensors
 * live in host memory.
 */
int ra_ring_forward_host(const void* q_host, const void* k_host, const void* v_host,
                         float* out_host, float* lse_host, long long N, int P, int causal, int d,
                         int heads, int kv_heads, int dtype, void* stream);

/*
 * ra_ring_forward_noalloc -- ra_ring_forward for callers that cannot let the
 * library allocate device memory.  Examples: an application that reserves
 * the whole GPU for its own memory pool, where a cudaMalloc from inside the
 * library would fail or break the pool's accounting; or one that must fix
 * its peak device footprint before it starts.  The pages have no
 * counterpart to this call; it is a deployment convenience.
 *   Arguments, layouts and results are those of ra_ring_forward.  The l
 *   state lives in a fixed 16 MiB device array that is part of the library
 *   (N * heads <= 4,194,304 fp32 entries), instead of memory from the
 *   scratch pool.  Every GPU that loads the library holds that array until
 *   the process exits.  The call calls no cudaMalloc, cudaFree or other
 *   allocating routine.
 *   Larger problems return RA_ERR_UNSUPPORTED; use ra_ring_forward for them.
 *   The first call on a device looks up the array's device address once,
 *   with that device current.  Make that first call before any stream
 *   capture starts.
 *   Only the calls that run the ring step by step use the array: bf16
 *   inputs with P > 256.  fp32 calls, and bf16 calls with P <= 256, run one
 *   fused launch, which keeps its state on chip and never touches the
 *   array.  Calls that use it share the one array.  Each clears the
 *   rows it uses first, so what an earlier call left there does not
 *   matter.  But two such calls that overlap on the GPU (different
 *   streams, not ordered) race on the array and both results are
 *   undefined.  The size limit is checked first, before the pointers and
 *   before any launch, for every dtype.
 */
int ra_ring_forward_noalloc(const void* q, const void* k, const void* v, float* out, float* lse,
                            long long N, int P, int causal, int d, int heads, int kv_heads,
                            int dtype, void* stream);

/*
 * Masked variants.  The mask arguments below are the same in the three
 * calls; [TEST] lists these cases (padding of the last rank with a valid
 * length, packed documents that must not see each other, sliding-window
 * and segment masks, non-causal and causal).  Key position kp is allowed
 * for query position qp when all of these hold:
 *   - qp < n_valid and kp < n_valid (n_valid < 0: no padding).  A query
 *     row at or past n_valid sees nothing; after a whole ring its output
 *     is 0 and its lse -inf.
 *   - documents (ndocs > 0): cu_seqlens is a DEVICE array of ndocs + 1
 *     nondecreasing int32 positions with cu_seqlens[0] = 0; document d is
 *     [cu_seqlens[d], cu_seqlens[d+1]).  qp and kp lie in the same
 *     document; positions at or past cu_seqlens[ndocs] belong to none and
 *     are treated as padding.  The array is read by the kernels, not
 *     checked; a malformed one gives undefined results (reads stay inside
 *     its ndocs + 1 entries).
 *   - causal: kp <= qp.
 *   - window > 0: |qp - kp| < window.  With causal that is the `window`
 *     most recent positions, qp itself included.
 * A query with no allowed key keeps its state.  Key tiles that no row of a
 * query tile may see are not visited, and only tiles that cut a row's
 * interval are masked elementwise.
 *
 * ra_block_update_masked -- ra_block_update with the full mask, a layout,
 * and query and key blocks of different lengths.
 *   q: [c_q, heads, d]; k, v: [c_kv, kv_heads, d]; m, l, o: [c_q, heads(, d)].
 *   layout RA_LAYOUT_CONTIGUOUS: positions are q_off + r and kv_off + t;
 *     P, q_block and kv_block are ignored.
 *   layout RA_LAYOUT_ZIGZAG / RA_LAYOUT_STRIPED: the blocks are blocks
 *     q_block and kv_block (0 <= both < P) of that layout with block length
 *     c_q (zigzag: c_q == c_kv, even); q_off and kv_off are ignored.
 */
int ra_block_update_masked(const void* q, const void* k, const void* v, float* m, float* l,
                           float* o, long long c_q, long long c_kv, int d, int heads,
                           int kv_heads, int layout, int P, int q_block, int kv_block,
                           long long q_off, long long kv_off, int causal, long long window,
                           long long n_valid, const int* cu_seqlens, int ndocs, int dtype,
                           void* stream);

/*
 * ra_ring_step_masked -- ra_ring_step with a layout and the full mask.
 * Block i of every tensor holds the positions `layout` gives it (N = P*c;
 * zigzag needs c even).  Ranks whose pair (i, j) holds no allowed
 * (query, key) pair under the causal, window and valid-length rules are
 * not launched; with a zigzag or striped layout under causal every rank
 * has work at every step [PB] section 5.
 */
int ra_ring_step_masked(const void* q, const void* k, const void* v, float* m, float* l,
                        float* o, long long N, int P, int s, int layout, int causal,
                        long long window, long long n_valid, const int* cu_seqlens, int ndocs,
                        int d, int heads, int kv_heads, int dtype, void* stream);

/*
 * ra_ring_forward_masked -- ra_ring_forward with a layout and the full
 * mask: state init, ra_ring_step_masked for s = 0 .. P-1, finalize.  The
 * outputs are in the tensors' row order (the layout's order), like q.
 * Scratch as in ra_ring_forward.
 */
int ra_ring_forward_masked(const void* q, const void* k, const void* v, float* out, float* lse,
                           long long N, int P, int layout, int causal, long long window,
                           long long n_valid, const int* cu_seqlens, int ndocs, int d,
                           int heads, int kv_heads, int dtype, void* stream);

/*
 * ra_ring_backward -- gradients of the ring forward for all P virtual ranks
 * ("Ring Attention：把超长序列沿设备环流动", section "Backward 需要让梯度也
 * 沿环传播"; [XF] "End-to-end flow": the backward ring carries the K/V
 * blocks and their gradient accumulators, which arrive home fully summed
 * after P steps).  For the loss L with dL/dO = dout:
 *   P = exp(S - LSE) is recomputed from the saved lse, D = rowsum(dout * out),
 *   dP = dout V^T, dS = P (dP - D) / sqrt(d),
 *   dq = dS K, dk = dS^T Q (summed over each KV head's query heads),
 *   dv = P^T dout (likewise).
 *   q, k, v: the forward's inputs (bf16).  out [N, heads, d] and lse
 *   [N, heads]: the forward's outputs (fp32).  dout: [N, heads, d] bf16.
 *   dq: [N, heads, d]; dk, dv: [N, kv_heads, d]: fp32, written (zeroed
 *   first, then accumulated over the ring steps).
 * Step s runs, for every rank i with block j = (i - s) mod P, a
 * Q-stationary tcgen05 kernel adding to dq of block i and a
 * K/V-stationary one adding to dk, dv of block j; within a launch every
 * block has one writer, so nothing is atomic.  P and dS are rounded to bf16
 * for their products, as in the forward.  Scratch: D ([N, heads] fp32),
 * stream-ordered on `stream` from the scratch pool.  dtype must be RA_BF16.
 */
int ra_ring_backward(const void* q, const void* k, const void* v, const float* out,
                     const float* lse, const void* dout, float* dq, float* dk, float* dv,
                     long long N, int P, int causal, int d, int heads, int kv_heads, int dtype,
                     void* stream);

/* ra_ring_backward with a layout and the full mask (as ra_ring_forward_masked). */
int ra_ring_backward_masked(const void* q, const void* k, const void* v, const float* out,
                            const float* lse, const void* dout, float* dq, float* dk, float* dv,
                            long long N, int P, int layout, int causal, long long window,
                            long long n_valid, const int* cu_seqlens, int ndocs, int d, int heads,
                            int kv_heads, int dtype, void* stream);

/*
 * Decode and short query blocks ("Ring Attention：把超长序列沿设备环流动",
 * section "训练与推理的适用方式不同").  A decode step has a few new query
 * tokens per sequence and a long K/V history.  Rotating K/V blocks around a
 * ring does not pay there; the query goes to every K/V shard, each shard
 * computes a partial (m, l, O~) state of the query rows, and the shards'
 * states are combined by the online-softmax merge.
 *
 * ra_decode_partial -- fold one K/V shard into the running state of n_q
 * query rows (in place, like ra_block_update), for deployments where each
 * device holds one shard and merges states with ra_merge afterwards.
 *   q: [n_q, heads, d] bf16, token positions q_off .. q_off + n_q - 1.
 *   k, v: [n_kv, kv_heads, d] bf16, positions kv_off .. kv_off + n_kv - 1.
 *   m, l: [n_q, heads] fp32; o: [n_q, heads, d] fp32 (updated in place).
 *   causal and window: as in the masked calls (kp <= qp; |qp - kp| < window).
 *   heads / kv_heads must be <= 128, n_q <= 2^24 and n_q * heads <= 2^31 - 1
 *   (RA_ERR_UNSUPPORTED otherwise).  A KV head's query
 *   rows (token qi of its g heads is row qi * g + hl) go in 128-row tiles of
 *   floor(128 / g) tokens; with (heads / kv_heads) * n_q <= 128, the decode
 *   case, they are one tile and each K/V byte is read once.  Each further
 *   tile reads the keys again: long query blocks belong to
 *   ra_block_update_masked.  dtype must be RA_BF16.
 * The work is HBM-bound: the keys of each KV head are streamed in chunks
 * spread over the SMs (split-K), each chunk giving one partial state, and a
 * second kernel folds them into m, l, o.  A chunk runs on the tensor cores
 * with one row tile of the KV head's query rows.  The partial states
 * (chunks x n_q x heads x (d + 2) fp32) are allocated stream-ordered on
 * `stream` from the scratch pool.
 */
int ra_decode_partial(const void* q, const void* k, const void* v, float* m, float* l, float* o,
                      long long n_q, long long n_kv, int d, int heads, int kv_heads,
                      long long q_off, long long kv_off, int causal, long long window,
                      int dtype, void* stream);

/*
 * ra_decode_forward -- the whole decode attention of n_q query tokens
 * against a K/V history of n_kv tokens (positions 0 .. n_kv - 1) split into
 * P shards of ceil(n_kv / P) keys: the partial states of every shard (one
 * launch over all shards, each shard in a few key chunks), then one launch
 * that folds all of them with the merge operator of ra_merge (the global
 * reduction; [SP] "训练与推理的适用方式不同": the query goes to every shard,
 * each shard gives a local state, a global online-softmax reduction
 * combines them) and finalizes.
 *   out: [n_q, heads, d] fp32; lse: [n_q, heads] fp32 (written).
 * Query positions are q_off .. q_off + n_q - 1 (for decode after a history
 * of n_kv tokens that includes the new ones: q_off = n_kv - n_q).  With
 * n_kv = 0 every row gets out = 0 and lse = -inf.  Scratch as above.
 */
int ra_decode_forward(const void* q, const void* k, const void* v, float* out, float* lse,
                      long long n_q, long long n_kv, int P, long long q_off, int causal,
                      long long window, int d, int heads, int kv_heads, int dtype,
                      void* stream);

/*
 * ra_device_status -- synchronize `stream`, then read and clear the
 * library's device-side error words.  Every mbarrier wait in the kernels is
 * bounded.  A wait that runs out records a code and makes its CTA leave
 * cleanly.  The call returns RA_ERR_TIMEOUT if any code was recorded since
 * the last call, RA_ERR_CUDA if the synchronize failed, else RA_OK.  While
 * a code is recorded, block-update CTAs that start do no work (so one
 * failed wait cannot turn into a long cascade).  Results of launches made
 * since the failure are therefore invalid until this call clears the code.
 * The pages have no counterpart to this call or the next: they are the
 * library's failure detection.
 */
int ra_device_status(void* stream);

/*
 * ra_selftest_wait_timeout -- failure-detection self test.  It launches one
 * CTA that waits, with a bound of `limit_cycles` SM cycles, on an mbarrier
 * that nothing arrives on.  It then returns what ra_device_status returns
 * (RA_ERR_TIMEOUT when the bounded wait works).  Nothing faults and nothing
 * hangs.
 */
int ra_selftest_wait_timeout(long long limit_cycles, void* stream);

/*
 * Cached scratch memory.  Every buffer the library allocates for itself
 * (the l state of ra_ring_forward on the step path, the device staging of
 * ra_ring_forward_host, the D vector of the backward, the partial states of
 * decode) comes, stream-ordered, from a memory pool that the library
 * creates on each device at first use.  The pool keeps what is freed into
 * it mapped, so the next call of the same size maps nothing: a call that
 * needs a few GB of staging does not pay milliseconds for a fresh mapping.
 * Ownership stays with the library, and what the pool holds is bounded by
 * the largest set of buffers one call (or concurrent calls) held.
 *
 * ra_cached_memory -- write to *bytes the memory the current device's pool
 *   holds (in use or cached); 0 before any allocation.  RA_ERR_INVALID if
 *   `bytes` is NULL.
 * ra_release_cached_memory -- return to the driver what the current
 *   device's pool holds and no call is using.  Memory that an enqueued call
 *   will still free stays until the work before that free has completed:
 *   synchronize the streams first to release everything.
 * The pages have no counterpart to these two calls: they are the library's
 * memory management, not part of the method.
 */
int ra_cached_memory(long long* bytes);
int ra_release_cached_memory(void);

/* Tracing.  When enabled, the library records a CUDA event pair on the
 * launching stream around every kernel it launches.  ra_trace_query then
 * synchronizes those events.  It returns the number of launches of `kind`
 * and their summed device time in milliseconds since the last reset.
 * These and the status helpers below have no counterpart on the pages. */
int ra_trace_enable(int on);
int ra_trace_reset(void);
int ra_trace_query(int kind, long long* launches, double* total_ms);

const char* ra_status_string(int status);
const char* ra_last_error(void);
int ra_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H */
