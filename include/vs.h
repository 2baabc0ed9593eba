/*
 * vs.h -- C ABI of the GB300 (sm_103a) Vertical-Slash sparse attention library
 * (libvs.so).
 *
 * The library implements the hot path of MTraining's dynamic sparse
 * attention ("MTraining: Distributed Dynamic Sparse Attention for Efficient
 * Ultra-Long Context Training"): the online Vertical-Slash estimator of
 * Algorithm 1, the sparse index (Algorithm 1 `sparseformat`, Algorithm 2
 * `convert_index`), causal GQA attention forward and backward restricted to
 * the selected columns and diagonals (Eq. 1, Eq. 2), and the 64-token
 * block-level striping of Balanced Sparse Ring Attention (section 4.2).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors live in device memory and are token-major "BSHD": element
 *    (b, n, h, c) of x is at x + b*s[0] + n*s[1] + h*s[2] + c, in elements,
 *    with the channel dimension contiguous.  Q, K, V, O, dO, dQ, dK, dV are
 *    bf16; LSE is fp32 [B][Hq][Nq] (contiguous); scores are fp32 [B][Hq][N].
 *    Strides must be multiples of 8 elements (16 bytes) and base pointers
 *    16-byte aligned (TMA requirement).
 *  - The KV head of query head h is h / (Hq / Hkv) (GQA grouping).
 *  - The caller owns every buffer.  The library never allocates, frees or
 *    synchronises, except the status, count and trace readers
 *    (vs_check_status, vs_estimate_noalloc_status, vs_index_counts,
 *    vs_trace_report), which synchronise and say so.
 *  - Every compute call is asynchronous on `stream`.
 *  - Argument and shape errors are returned synchronously and nothing is
 *    launched.  Errors found on the device (bad index lists, a bounded wait
 *    that ran out) are recorded in the first 32-bit word of the workspace or
 *    index arena that the call received; kernels never trap.  Read them with
 *    vs_check_status.  A status word that already holds a failure when a
 *    call starts makes that call's kernels skip their work.
 *  - Same inputs give the same output bits: no floating-point atomics touch
 *    any output or score.
 *  - Supported: head_dim d in {64, 128}; N a multiple of 64; Hq a multiple of
 *    Hkv; 1 <= kv, ks <= N; last_q == 64.
 */
#ifndef VS_H_
#define VS_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VS_OK = 0,
  VS_ERR_ARG = 1,       /* null pointer or bad scalar argument */
  VS_ERR_SHAPE = 2,     /* unsupported shape, stride or alignment */
  VS_ERR_WORKSPACE = 3, /* workspace or index arena too small */
  VS_ERR_INDEX = 4,     /* (device) index list out of range, unsorted or duplicated */
  VS_ERR_TIMEOUT = 5,   /* (device) a bounded wait ran out */
  VS_ERR_CUDA = 6,      /* CUDA runtime error while encoding or launching */
  VS_ERR_SCORE = 7      /* (device) a score is negative, not finite, or the list's total is >= 2^13 */
} vs_status;

/* Problem shape.  Nq / Nk are the local query / key lengths (equal unless a
 * striped shard pairs one worker's queries with another worker's keys).
 * Strides are in elements: [0] batch, [1] token, [2] head.
 *   sq: Q, dQ      sk: K, dK      sv: V, dV      so: O, dO               */
typedef struct {
  int B, Nq, Nk, Hq, Hkv, d;
  int64_t sq[3], sk[3], sv[3], so[3];
} vs_shape;

/* Where the local tokens sit on the global sequence of N_global tokens: local
 * 64-token block j of the query tensor is global block world * j + q_rank,
 * that of the key tensor world * j + kv_rank.  Two uses:
 *   - a striped shard pair (Balanced Sparse Ring Attention, section 4.2 (ii)
 *     and Algorithm 2): global block j lives on worker j mod world at local
 *     block j / world; the queries belong to worker q_rank, the keys to worker
 *     kv_rank (ranks below world), N_global = world * Nq;
 *   - a pair of contiguous windows (world 1, rank = the window's first
 *     global block), e.g. one chunk of a ZigZag worker's queries against one
 *     chunk of another worker's keys (section 2, Figure 1).
 * Every local block must lie inside the global sequence.  Pass NULL for an
 * unstriped problem (identity positions). */
typedef struct {
  int world, stripe, q_rank, kv_rank;
  int64_t N_global;
} vs_stripe;

/* ---------------------------------------------------------------------------
 * vs_estimate -- online Vertical-Slash estimation (Algorithm 1, first four
 * lines; section 4.1 (i)).
 *
 * For every (b, h): the observation window is the last `last_q` query rows
 * n_i = N - last_q + i.  A_hat = softmax(scale * Q[n_i] K^T) over causal keys
 * m <= n_i.  Vertical score v[m] = sum_i A_hat[i, m]; slash score
 * s[o] = sum_i A_hat[i, n_i - o].  Then v_idx = argtopk(v, kv) and
 * s_idx = argtopk(s, ks) under the total order (score descending, index
 * ascending), each list written sorted ascending.
 *
 *   shape     Nq == Nk == N (global, unstriped tensors)
 *   q, k      bf16 BSHD
 *   last_q    must be 64
 *   kv, ks    budgets, 1..N
 *   v_idx     int32 [B][Hq][kv]      (out)
 *   s_idx     int32 [B][Hq][ks]      (out)
 *   v_score   fp32 [B][Hq][N] or NULL (out; kept in the workspace if NULL)
 *   s_score   fp32 [B][Hq][N] or NULL
 *   ws        device workspace of at least vs_estimate_workspace() bytes
 * ------------------------------------------------------------------------- */
size_t vs_estimate_workspace(const vs_shape* shape, int last_q);
vs_status vs_estimate(const vs_shape* shape, const void* q, const void* k, int last_q, int kv, int ks, float scale,
                      int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws, size_t ws_bytes,
                      cudaStream_t stream);

/* vs_estimate_group -- vs_estimate with one selection per KV group (a
 * variant of the per-head selection: the Hq / Hkv query heads that share a
 * KV head share one index).  The group's scores are the sums of its heads'
 * scores (fp32, added in head order); every head of the group gets
 * argtopk of those sums, so v_idx / s_idx rows of one group are equal.
 * Arguments, workspace and outputs as for vs_estimate (v_score / s_score
 * still receive the per-head scores). */
vs_status vs_estimate_group(const vs_shape* shape, const void* q, const void* k, int last_q, int kv, int ks,
                            float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_estimate_topp / vs_select_topp -- top-p budgets (Algorithm 1, the
 * `topp` and `Pool` lines; section 4.1 (i) online budget approximation and
 * (ii) kernel-aware granularity).
 *
 * Instead of fixed kv / ks, each (b, h) gets the smallest budgets that
 * recall a fraction of its observed attention mass:
 *   kv = min(topp(v, pv), kv_max)
 *   ks = min(64 * topp(Pool(s, 64), ps), ks_max, N)
 * where topp(x, p) is the smallest k whose k largest entries of x sum to at
 * least p * sum(x), and Pool sums 64 consecutive slash offsets (the slash
 * tiles are 64 x 64 blocks).  Then v_idx = argtopk(v, kv) and s_idx =
 * argtopk(s, ks) as in vs_estimate.  The decision is exact and reproducible:
 * a score x counts floor(x * 2^40) integer mass units, the target is
 * ceil(p * T) for the unit total T (one double product), and the budget is
 * the smallest k whose k largest unit counts reach it.
 *
 *   pv, ps        fractions in [0, 1]
 *   kv_max/ks_max list capacities, 1..N
 *   v_idx         int32 [B][Hq][kv_max] (out): the kv selected columns,
 *                 ascending, then -1
 *   s_idx         int32 [B][Hq][ks_max] (out): the ks selected offsets,
 *                 ascending, then -1
 *   kv, ks        int32 [B][Hq] device (out): the budgets
 * vs_estimate_topp takes the remaining arguments of vs_estimate (same
 * workspace).  vs_select_topp runs the budget and selection step alone on
 * given scores (fp32 [B][H][N], device): ws is a device buffer of at least
 * 256 bytes whose first word is the status word.
 * Limits: N <= 1,572,864.  Device errors: VS_ERR_SCORE (that head's lists
 * are then empty and its budgets 0).
 * ------------------------------------------------------------------------- */
vs_status vs_estimate_topp(const vs_shape* shape, const void* q, const void* k, int last_q, double pv, double ps,
                           int kv_max, int ks_max, float scale, int32_t* v_idx, int32_t* s_idx, int32_t* kv,
                           int32_t* ks, float* v_score, float* s_score, void* ws, size_t ws_bytes,
                           cudaStream_t stream);
vs_status vs_select_topp(int B, int H, int N, const float* v_score, const float* s_score, double pv, double ps,
                         int kv_max, int ks_max, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks, void* ws,
                         size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_estimate_noalloc -- vs_estimate without a caller workspace.  (The paper
 * has no counterpart: this is a deployment convenience of this library.)
 *
 * Some callers cannot hand the library a workspace of their own: operator or
 * plugin code run inside an engine that owns all device memory and forbids
 * allocation while it executes, or latency-critical loops where cudaMalloc's
 * implicit device-wide synchronisation would stall every other stream.  This
 * entry point computes exactly what vs_estimate computes, with the same
 * kernels, but keeps its scratch (row statistics, row LSEs and slash
 * partials) in a
 * fixed 32 MiB array of the library's static device memory, which every GPU
 * that loads the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments as for vs_estimate, except that v_score and s_score are
 *   required (the scores live in the caller's buffers, not in the scratch).
 *   Scratch needed: 256 + B*Hq*32 KiB + B*Hq*256 + B*Hq*ceil(N/128)*768
 *   bytes (each term rounded up to 256); larger problems are rejected with
 *   VS_ERR_WORKSPACE before any launch (for example B*Hq = 16 fits N up to
 *   343936).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current), which may load the
 * library's module onto the device; make that first call before any stream
 * capture.  A first call made while `stream` is capturing is refused with
 * VS_ERR_ARG before any CUDA work.  Every call on a device shares the one
 * array: calls that overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  The array keeps the last
 * call's contents; each call clears the status header at its start and
 * writes every other scratch element it reads.
 *
 * Device errors (VS_ERR_TIMEOUT from a bounded wait) go to the status word
 * at the start of the array instead of a caller workspace; the kernels after
 * the failing one then skip their work, leaving the outputs unspecified.
 * Read the word with vs_estimate_noalloc_status after the call and before
 * the next call on the device, which clears it.
 * ------------------------------------------------------------------------- */
vs_status vs_estimate_noalloc(const vs_shape* shape, const void* q, const void* k, int last_q, int kv, int ks,
                              float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score,
                              cudaStream_t stream);

/* Status of the last vs_estimate_noalloc call on the current device: reads
 * the scratch's status word, resets it to VS_OK and returns the code it held
 * (VS_OK if no call has run on the device).  Synchronises `stream`, which
 * should be the stream of that call. */
vs_status vs_estimate_noalloc_status(cudaStream_t stream);

/* Self-test of the status path above (no counterpart in the paper): writes
 * `code` into the scratch's status word of the current device, as a failing
 * kernel would, and synchronises `stream`.  vs_estimate_noalloc_status then
 * returns `code`. */
vs_status vs_estimate_noalloc_selftest_plant(int code, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_build_block_index -- the sparse index (Algorithm 1 `sparseformat`,
 * Algorithm 2 `convert_index`).
 *
 * Turns the selected columns (v_idx, global, sorted) and diagonals (s_idx,
 * global offsets n - m, sorted) into the arena the attention kernels read.
 * A list may end in entries equal to -1 (a top-p budget below the list's
 * capacity); they select nothing, and a list of only -1 is empty.
 * The mask it encodes is exact at token level:
 *     M[n, m] = (m <= n) and (m in v_idx or n - m in s_idx)
 * on global positions.  It is covered by
 *   - slash tiles: 128 query rows x 64 keys, holding the entries with a
 *     selected offset whose key is not a selected column, and
 *   - vertical bars: the selected columns gathered into chunks (64 keys for
 *     the query-major passes, 128 for the key-major pass), holding every
 *     causal entry of those columns,
 * so each entry of M is computed exactly once.  With `stripe` set, the arena
 * describes one ring step: worker q_rank's queries against worker kv_rank's
 * keys.  The arena begins with a 256-byte header whose first int32 is the
 * device status word.
 *
 *   v_idx  int32 [B][Hq][kv]; s_idx int32 [B][Hq][ks] (device)
 *   arena  device buffer of at least vs_block_index_bytes() bytes; fully
 *          rewritten by this call
 * Device errors: VS_ERR_INDEX when a list is out of range, unsorted, has
 * duplicates, or has an entry after a -1 (the arena then describes an empty
 * mask).
 * ------------------------------------------------------------------------- */
size_t vs_block_index_bytes(const vs_shape* shape, int kv, int ks, const vs_stripe* stripe);
vs_status vs_build_block_index(const vs_shape* shape, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                               const vs_stripe* stripe, void* arena, size_t arena_bytes, cudaStream_t stream);

/* vs_build_block_index with flags.  VS_INDEX_BLOCK_COVER selects the
 * block-cover reading of the slashes (section 4.1 (ii): the slashes taken at
 * the granularity of the kernel's 64 x 64 tiles): the mask becomes
 *     M[n, m] = (m <= n) and (m in v_idx or block diagonal
 *               floor(n/64) - floor(m/64) is active),
 * on global positions, where block diagonal D is active iff some selected
 * offset o has |o - 64 D| <= 63 (the slash passes through its blocks).
 * VS_INDEX_PACK_GQA packs the query heads of a KV group into the query-major
 * tiles (a variant for one selection per KV group, as vs_estimate_group
 * makes): a tile holds 128 / g tokens of all g = Hq / Hkv heads, so every
 * K / V block it loads feeds g heads and a slash costs one 64-key unit per
 * 128 / g tokens instead of two per 128 rows of one head.  It needs the
 * lists of a group's heads to be equal (else VS_ERR_INDEX on the device),
 * an unstriped problem without VS_INDEX_BLOCK_COVER (else VS_ERR_ARG) and
 * g dividing 128, g >= 2 (else VS_ERR_SHAPE).  The mask is unchanged; the
 * query-major work counts of a group are reported at its first head.  The
 * attention calls read the flags from the arena.  Other flag bits:
 * VS_ERR_ARG. */
enum { VS_INDEX_BLOCK_COVER = 1, VS_INDEX_PACK_GQA = 2 };
vs_status vs_build_block_index_ex(const vs_shape* shape, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                                  const vs_stripe* stripe, int flags, void* arena, size_t arena_bytes,
                                  cudaStream_t stream);

/* Work counts of an arena, for FLOP accounting (copies 4 x int64 per (b, h)
 * to host memory; synchronises the stream):
 *   [0] query-major slash tiles (128 x 64)    [1] query-major bar chunks (128 x 64)
 *   [2] key-major slash units (128 x 64)      [3] key-major bar units (128 x 64)
 * out: int64 [B][Hq][4] in host memory. */
vs_status vs_index_counts(const void* arena, int64_t* out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_attn_fwd -- dynamic sparse FlashAttention forward, y = sparse(softmax(
 * Q K^T * scale) V, ivs) (Algorithm 1, last line; `block_bar_sparse_attention
 * _forward` of Algorithm 2).
 *
 * For every query row n with a non-empty mask row: O_n = sum_{m in M(n)}
 * softmax(S)_nm v_m and LSE_n = log sum_{m in M(n)} exp(S_nm), S = scale Q K^T.
 * Rows with an empty mask get O = 0 and LSE = -inf.
 *
 *   q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] bf16; o [B,Nq,Hq,d] bf16 (out)
 *   lse    fp32 [B][Hq][Nq] (out; in accumulate mode also in)
 *   o_acc  NULL, or fp32 [B][Nq][Hq][d] contiguous: accumulate mode
 *          (`merge_out_and_lse` of Algorithm 2).  The call merges its partial
 *          result into (o_acc, lse): LSE' = log(e^LSE + e^LSE_step),
 *          O' = (e^LSE O_acc + e^LSE_step O_step) / e^LSE', and writes o =
 *          bf16(O').  Start a ring with o_acc = 0 and lse = -inf.
 *   arena  from vs_build_block_index for the same shape (and stripe)
 *   ws     at least vs_attn_fwd_workspace() bytes
 * ------------------------------------------------------------------------- */
size_t vs_attn_fwd_workspace(const vs_shape* shape);
vs_status vs_attn_fwd(const vs_shape* shape, const void* q, const void* k, const void* v, const void* arena,
                      float scale, void* o, float* lse, float* o_acc, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_attn_bwd -- sparse backward on the same mask (section 3.2: the backward
 * inherits the forward's sparsity; Eq. 1, Eq. 2).
 *
 *   D_n   = rowsum(dO_n * O_n)                 (= rowsum(dA * A))
 *   P     = exp(S - LSE), dA = dO V^T
 *   dS    = P * (dA - D)                       (Eq. 1)
 *   dV    = P^T dO, dQ = scale dS K, dK = scale dS^T Q   (Eq. 2)
 * dK and dV of a KV head are summed over its query heads.  All products are
 * restricted to M.
 *
 *   o, lse     the forward's outputs (in a ring: the merged ones)
 *   dO         bf16 [B,Nq,Hq,d] (strides so)
 *   dq         bf16 out; dk, dv bf16 out [B,Nk,Hkv,d]
 *   dq_acc     NULL, or fp32 [B][Nq][Hq][d] contiguous: accumulate mode for a
 *              ring step (dq_acc += dQ_step; dq = bf16(dq_acc))
 *   ws         at least vs_attn_bwd_workspace() bytes
 * ------------------------------------------------------------------------- */
size_t vs_attn_bwd_workspace(const vs_shape* shape, int kv);
vs_status vs_attn_bwd(const vs_shape* shape, const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk, void* dv,
                      float* dq_acc, void* ws, size_t ws_bytes, cudaStream_t stream);

/* vs_attn_bwd with an accumulate mode for dK and dV as well (a key window
 * that receives the gradients of several query windows, as the two chunks of
 * a ZigZag worker do at one ring step):
 *   dkv_acc  NULL, or fp32 [2][B][Nk][Hkv][d] contiguous (dK, then dV):
 *            dkv_acc += this call's dK / dV; dk = bf16(dK sum), dv likewise.
 * Other arguments as for vs_attn_bwd. */
vs_status vs_attn_bwd_ex(const vs_shape* shape, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk,
                         void* dv, float* dq_acc, float* dkv_acc, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * striped_permute -- block-level striping (section 4.2 (ii), 64-token
 * stripes): global block j of x [B, N, H, d] goes to shard j mod world at
 * local block j / world of y [world, B, N/world, H, d] (both contiguous bf16).
 * inverse = 1 maps shards back.  only_rank >= 0 writes just that shard
 * (y then holds one shard [B, N/world, H, d]); -1 writes all.
 * ------------------------------------------------------------------------- */
vs_status striped_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int stripe, int inverse,
                          int only_rank, cudaStream_t stream);

/* vs_ring_permute -- striped_permute for either ring layout (layout as for
 * vs_ring_work below): VS_LAYOUT_STRIPED (64-token stripes, N a multiple of
 * 64 world) or VS_LAYOUT_ZIGZAG (section 2, Figure 1: 2 world chunks of
 * N / (2 world) tokens, worker r holds chunks r and 2 world - 1 - r in that
 * order; N a multiple of 128 world).  Shard layout, inverse and only_rank as
 * for striped_permute. */
vs_status vs_ring_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int layout, int inverse,
                          int only_rank, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * vs_ring_work -- work of a context-parallel ring under the VS mask (section
 * 3.3, worker- and step-level imbalance; section 4.2, Balanced Sparse Ring
 * Attention; section 2, Striped vs ZigZag Ring Attention).
 *
 * out[r][q] = number of entries of the mask on the global sequence,
 *     M[n, m] = (m <= n) and (m in v_idx or n - m in s_idx),
 * whose query n lives on worker r and key m on worker q, summed over (b, h).
 * At ring step s worker r attends to the keys of worker (r - s) mod world, so
 * its effective work at that step is out[r][(r - s) mod world].
 *   layout  VS_LAYOUT_STRIPED: 64-token block j on worker j mod world
 *           (N a multiple of 64 world); VS_LAYOUT_ZIGZAG: 2 world chunks of
 *           N / (2 world) tokens, worker r holds chunks r and 2 world - 1 - r
 *           (N a multiple of 2 world)
 *   v_idx   int32 [B][H][kv], s_idx int32 [B][H][ks]: global lists as for
 *           vs_build_block_index (ascending, optionally ending in -1)
 *   out     int64 [world][world] device (out; overwritten)
 *   ws      device buffer of at least 256 bytes; its first word is the status
 *           word (VS_ERR_INDEX for a bad list)
 * Limits: 1 <= world <= 64, N < 2^31 and about N <= 1.2M at world 64 (the
 * column bitmap and its prefix counts live in shared memory).
 * ------------------------------------------------------------------------- */
enum { VS_LAYOUT_STRIPED = 0, VS_LAYOUT_ZIGZAG = 1 };
vs_status vs_ring_work(int B, int H, int64_t N, const int32_t* v_idx, int kv, const int32_t* s_idx, int ks,
                       int world, int layout, int64_t* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Reads the device status word at the start of a workspace or index arena,
 * resets it to VS_OK, and returns the code it held.  Synchronises `stream`. */
vs_status vs_check_status(void* ws_or_arena, cudaStream_t stream);

/* Failure-detection self-test (no counterpart in the pages: it checks the
 * bounded waits every kernel above relies on).  Launches one CTA whose two
 * warps wait on mbarriers that nothing arrives on.  The first wait runs out
 * after the kernels' wait budget (about two seconds), records VS_ERR_TIMEOUT
 * in the device status word at the start of `ws` (ws_bytes >= 256) and
 * raises the CTA's abort flag, on which the other warp gives up; both warps
 * then return, and each adds 1 to the int at byte offset 4 of `ws` (100 if a
 * wait had completed).  Returns VS_OK once launched; vs_check_status(ws)
 * then reports VS_ERR_TIMEOUT.  The CUDA context stays usable. */
vs_status vs_selftest_wait_timeout(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* vs_status_string(vs_status status);

/* Number of kernels the library launched since load (for launch counting). */
int64_t vs_launch_count(void);

/* ---------------------------------------------------------------------------
 * Kernel tracing (profiling aid; not part of the method).  While enabled,
 * every kernel the library launches is bracketed by a pair of CUDA events
 * recorded on the launching stream.  vs_trace_report synchronises the device,
 * then returns, per kernel name in first-launch order, the launch count and
 * the summed event time in milliseconds; it writes at most `max_kernels`
 * entries, names as NUL-separated strings into `names` (capacity names_len),
 * and returns the number of distinct kernels (or -1 on a CUDA error).
 * vs_trace_enable(0) stops recording; vs_trace_reset drops the records.
 * Not thread-safe; not for use during CUDA graph capture.
 * ------------------------------------------------------------------------- */
void vs_trace_enable(int on);
void vs_trace_reset(void);
int vs_trace_report(char* names, int names_len, int64_t* counts, double* ms, int max_kernels);

#ifdef __cplusplus
}
#endif
#endif /* VS_H_ */
