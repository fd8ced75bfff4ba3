/*
 * libscout: the GPU side of GPU-CPU collaborative block-sparse decode attention
 * (ScoutAttention, arXiv 2603.27138), for NVIDIA GB300 (sm_103a).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers are DEVICE memory owned by the caller unless the comment says host.
 *   The library never allocates or frees device memory and never synchronises
 *   the device; scratch space is a caller-provided workspace.
 * - Every call is asynchronous on the given stream and returns SCOUT_OK once
 *   the work is enqueued.  Arguments are checked on the host before any launch;
 *   a rejected call launches nothing.  A launch failure reported by the CUDA
 *   runtime returns SCOUT_ERR_CUDA.
 * - The host-side entry points (scout_plan_recall, scout_plan_recall_pages,
 *   scout_recall_intervals, scout_cpu_attend(_scalar), scout_cpu_pool_*,
 *   scout_cpu_attend_async) are the exception: host pointers only, no GPU
 *   involved, synchronous except scout_cpu_attend_async.  scout_cpu_attend runs on
 *   worker threads it starts and joins within the call; the pool calls run on the
 *   caller's pool.
 * - bf16 tensors are IEEE bfloat16 (2 bytes); fp32 are IEEE binary32.
 * - Shapes: B sequences, Hq query heads, Hkv KV heads (G = Hq / Hkv query heads
 *   per KV head, 1 <= G <= 8), D = 128 head dims, P tokens per KV block
 *   (16, 32 or 64), nblk_cap blocks per (sequence, KV head) in the tables.
 *   A "unit" is one (sequence b, KV head h): u = b * Hkv + h.
 * - Device-side bounds problems (a page-table slot outside the pool, a block
 *   index outside the table) never fault: the offending block is skipped and,
 *   when dev_status is not NULL, bit SCOUT_DEV_BAD_INDEX is OR-ed into
 *   *dev_status.  Bounded waits that expire set SCOUT_DEV_TIMEOUT.
 * - No C++ exception crosses this interface and the library keeps no mutable
 *   global state: calls on different streams with different buffers are
 *   independent.  The one exception is scout_score_topk_noalloc, whose scratch
 *   is a device array inside the library shared by all its calls: overlapping
 *   calls of it must be serialised (see its comment).
 */
#ifndef SCOUT_H_
#define SCOUT_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif
#ifdef __cplusplus
extern "C" {
#endif

typedef enum scout_status {
  SCOUT_OK = 0,
  SCOUT_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size */
  SCOUT_ERR_UNSUPPORTED = 2,  /* D != 128, P not in {16,32,64}, G > 8, misaligned pointer */
  SCOUT_ERR_WORKSPACE = 3,    /* workspace missing or smaller than *_workspace_bytes() */
  SCOUT_ERR_CUDA = 4,         /* the CUDA runtime rejected a launch or copy */
  SCOUT_ERR_TIMEOUT = 5       /* a bounded host-side wait expired */
} scout_status;

/* bits OR-ed into the optional device status word */
#define SCOUT_DEV_BAD_INDEX 1
#define SCOUT_DEV_TIMEOUT 2

typedef enum scout_digest_kind {
  SCOUT_DIGEST_MINMAX = 0, /* Quest: channel-wise min and max of K over a block */
  SCOUT_DIGEST_MEAN = 1    /* MoBA: channel-wise mean of K over a block */
} scout_digest_kind;

/* OR-ed into scout_score_topk's kind: pool a GQA group's scores by their sum instead of
 * their maximum (a variant; the pages do not say how a group's heads share a selection). */
#define SCOUT_POOL_SUM 0x10

/* Launch options (pass NULL for the defaults).  max_ctas bounds the CTAs a
 * persistent kernel launches (at most one per SM each): kernels of independent
 * work, e.g. the next layer's selection and this layer's attention (Algorithm 1),
 * can then share the SMs from separate streams.  0 means one CTA per SM; a
 * negative value is SCOUT_ERR_INVALID_ARG.  scout_score_topk deals whole units to
 * its CTAs as they start, so it also takes the SMs other kernels free up while it
 * runs; its default (0) is the fewest CTAs that take ceil(units / SMs) units each
 * (a last round of units then keeps as many SMs streaming as the others).  For
 * scout_predict_q it bounds the split-K factor S so that
 * (N / 128) * S <= max_ctas; the grid keeps at least one CTA per 128-row tile of W.
 *
 * Early starts (programmatic dependent launch), for scout_predict_q,
 * scout_score_topk and scout_sparse_attn(_merge).  Each of these kernels may start
 * before the kernel it depends on has finished, do the part of its work that does
 * not read that kernel's output, and wait for that kernel (its completion and the
 * visibility of its writes) just before the first read that may:
 *   scout_predict_q    streams W, then waits before it reads X;
 *   scout_score_topk   streams digests, then waits before it reads q;
 *   scout_sparse_attn  sets up its barriers, then waits before its first global read.
 * Each writes its outputs only after that wait.  Everything else it reads must be
 * complete before the kernel it depends on started.  Two ways to start early:
 *   pdl = 1          the dependency is the previous kernel on the same stream;
 *   early_event      set on the launch of the kernel depended on (the primary): the
 *                    event (created with cudaEventDisableTiming) is recorded
 *                    programmatically and fires before the primary completes, once
 *                    every CTA of it has passed its trigger: scout_predict_q at its
 *                    start, scout_score_topk once its last unit has been handed out,
 *                    scout_sparse_attn once its attention warps are done.  One of the
 *                    three kernels launched on a stream that waits for the event then
 *                    starts early as above.  Anything else that waits for the event
 *                    (a copy, a host wait, another library's kernel) is NOT ordered
 *                    after the primary's writes: record a plain event after the call
 *                    for those.  NULL: no programmatic event. */
typedef struct scout_launch {
  int max_ctas;
  int pdl;
  cudaEvent_t early_event;
  int inject; /* fault injection for tests; 0 (SCOUT_INJECT_NONE) in normal use */
} scout_launch;

/* Values of scout_launch.inject.  They make a failure happen without faulting or hanging
 * the GPU, so that tests can check how it is reported and that it does no lasting harm.
 *   SCOUT_INJECT_ABANDON  scout_score_topk only: every CTA behaves as if a bounded wait of
 *     its copy-issuing warp had expired after its first unit: it reports SCOUT_DEV_TIMEOUT,
 *     hands out no further work, lets every copy it started land, and leaves the scoring
 *     warps to wait for a stage that never comes, under a short poll limit (a real bounded
 *     wait that expires).  The units it skipped keep stale lists.  The call still leaves
 *     its workspace counter at zero, so the next call on the same workspace is correct.
 *   SCOUT_INJECT_COPY_FAIL  scout_recall_async and scout_recall_gather_async only: the
 *     call returns SCOUT_ERR_CUDA as if the CUDA runtime had refused a copy or the launch
 *     (scout_recall_async: its second run of copies, after the first was enqueued;
 *     scout_recall_gather_async: the gather launch, so nothing is enqueued). */
#define SCOUT_INJECT_NONE 0
#define SCOUT_INJECT_ABANDON 1
#define SCOUT_INJECT_COPY_FAIL 2

/* Human-readable name of a status code (static string, never NULL). */
const char* scout_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int scout_version(void);

/* ------------------------------------------------------------------------ *
 * Layer-ahead query prediction.
 * ScoutAttention (arXiv HTML), section 3.3 and Algorithm 1: the next layer's
 * query is predicted from the current layer's input, Q_pred^{i+1} = W_Q^{i+1} X^i.
 *
 * X  bf16 [M][K] row-major (one row per sequence), W bf16 [N][K] row-major
 * (linear-layer layout, N = Hq * D), Q bf16 [M][N] row-major; Q = X W^T with
 * fp32 accumulation, rounded to nearest bf16.  Requires 1 <= M <= 256,
 * N % 128 == 0, K % 64 == 0, and 16-byte-aligned X, W, Q.
 * Runs on the tensor cores (tcgen05, TMA-fed), with K split over the CTAs of a
 * thread-block cluster and reduced through distributed shared memory.  No
 * workspace.  dev_status (may be NULL) receives SCOUT_DEV_TIMEOUT if a bounded
 * pipeline wait expires.
 * ------------------------------------------------------------------------ */
int scout_predict_q(const void* X, const void* W, void* Q, int M, int N, int K, int32_t* dev_status,
                    const scout_launch* launch, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Block digests.
 * ScoutAttention (arXiv HTML), section 2.2: each fixed-size KV block is
 * summarised by a digest; Quest uses channel-wise min/max pooling of K, MoBA
 * mean pooling.  The digest of block j covers its valid tokens
 * t in [jP, min((j+1)P, seq_len[b])).
 *
 * K_pool     bf16 [n_slots][P][D]: block j of unit u lives in slot page_table[u][j]
 * page_table int32 [B][Hkv][nblk_cap]
 * seq_len    int32 [B]
 * block_list int32 [n_list][2] of (u, j) pairs to (re)build, or NULL for every
 *            valid block of every unit (prefill).  Blocks without valid tokens
 *            are left untouched.
 * digest     MINMAX: bf16 [B][Hkv][nblk_cap][2][D] (min row, then max row)
 *            MEAN:   fp32 [B][Hkv][nblk_cap][D]
 * Min/max are exact.  The mean is a compensated fp32 sum divided by the count.
 * ------------------------------------------------------------------------ */
int scout_build_digest(int kind, const void* K_pool, int64_t n_slots, const int32_t* page_table,
                       const int32_t* seq_len, int B, int Hkv, int D, int P, int nblk_cap,
                       const int32_t* block_list, int n_list, void* digest, int32_t* dev_status,
                       cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Digest scoring, top-k selection and residency split.
 * ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1: the GPU takes the
 * top-k blocks by query-digest dot product (B_pred), compares them with the
 * blocks resident in GPU memory (B_gpu) and marks the rest for the CPU
 * (B_cpu = B_pred \ B_gpu).
 *
 * Score of block j for query head h:  MINMAX  sum_c max(q_hc min_jc, q_hc max_jc)
 *                                     MEAN    sum_c q_hc mean_jc
 * One selection per unit: the block score is the maximum over the G query
 * heads of the unit (with kind | SCOUT_POOL_SUM: their sum, added in the order
 * ((h0 + h1) + (h2 + h3)) + ((h4 + h5) + (h6 + h7)) in fp32).  Valid blocks are
 * j < ceil(seq_len[b] / P).
 * Top-k: k_eff = min(k, valid blocks) blocks by (score desc, index asc).
 *
 * q            bf16 [B][Hq][D]   (query head hq belongs to KV head hq / G)
 * digest       as written by scout_build_digest for the same kind
 * resident_bits uint32 [B][Hkv][ceil(nblk_cap/32)]: bit j%32 of word j/32 set
 *              when block j is in GPU memory
 * prev_cpu_list int32 [B][Hkv][k] / prev_cpu_count int32 [B][Hkv]: the previous
 *              step's CPU list, or both NULL (then delta = cpu list).  They may
 *              alias cpu_list / cpu_count.
 * Outputs (all [B][Hkv][k] int32 lists in ascending block order, entries past
 * the count set to -1; counts int32 [B][Hkv]):
 *   scores     fp32 [B][Hkv][nblk_cap] pooled scores (-inf past the valid
 *              blocks), or NULL
 *   topk_idx/topk_count  B_pred;  res_list/res_count  B_pred with bit set;
 *   cpu_list/cpu_count   B_pred with bit clear;  delta_list/delta_count
 *   cpu list minus the previous cpu list.
 * workspace    scout_score_topk_workspace_bytes() bytes (4 * B * Hkv rounded
 *              up to 256; the kernel uses its first word, a unit ticket
 *              counter); it must be zero before the first use and every call,
 *              including one whose bounded waits expired, leaves it zero.
 * dev_status   int32 (may be NULL): SCOUT_DEV_TIMEOUT is OR-ed in when a bounded
 *              wait expired; the lists of the units left unfinished are then
 *              stale.  The call still returns SCOUT_OK (the failure is found on
 *              the device, after the launch).
 * Requires k >= 1, nblk_cap <= 8192, G <= 8.
 * ------------------------------------------------------------------------ */
size_t scout_score_topk_workspace_bytes(int B, int Hkv, int nblk_cap);
int scout_score_topk(int kind, const void* q, const void* digest, const int32_t* seq_len,
                     const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                     const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                     int k, float* scores, int32_t* topk_idx, int32_t* topk_count, int32_t* res_list,
                     int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count, int32_t* delta_list,
                     int32_t* delta_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     const scout_launch* launch, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * scout_score_topk without a caller workspace (no counterpart in the paper).
 *
 * For callers that cannot allocate device memory when they select blocks: an
 * engine that reserves all GPU memory in one pool at start-up and forbids later
 * cudaMalloc calls, or a host that loads this library as a plugin without giving
 * it an allocator.  Same arguments and results as scout_score_topk, minus the
 * workspace and the launch options.  The scratch is one fixed device array of
 * scout_score_topk_noalloc_max_bytes() bytes (4 MiB) inside the library, held by
 * every GPU that loads it until the process exits.  The kernel uses one counter
 * word of it, but the array is sized like the caller workspace, so it accepts
 * B * Hkv <= 1,048,576 units; a call whose scout_score_topk_workspace_bytes(B, Hkv,
 * nblk_cap) exceeds the array returns SCOUT_ERR_WORKSPACE.  Every argument is
 * checked before anything is enqueued: a rejected call leaves the array alone.
 * It never calls cudaMalloc or cudaFree.  The array's device address is looked up
 * (cudaGetSymbolAddress, with the caller's device current) on every call made
 * outside a stream capture, so it stays right after cudaDeviceReset; a call
 * inside a capture uses the address the last call outside one found on that
 * device, so make one call on each device before capturing.  Each call zeroes
 * the array's counter on `stream` before its kernel.  All calls share the one
 * array, so calls whose kernels overlap on the GPU (different streams, or
 * different host threads) race: serialise them.
 * ------------------------------------------------------------------------ */
size_t scout_score_topk_noalloc_max_bytes(void);
int scout_score_topk_noalloc(int kind, const void* q, const void* digest, const int32_t* seq_len,
                             const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                             const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                             int k, float* scores, int32_t* topk_idx, int32_t* topk_count, int32_t* res_list,
                             int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count, int32_t* delta_list,
                             int32_t* delta_count, int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * List of every resident block (a variant of which blocks the GPU attends).
 * ScoutAttention (arXiv HTML), Algorithm 1 writes the GPU's share as
 * GPUATTN(Q, B_gpu), which can be read as all the blocks in GPU memory rather than
 * the selected ones among them (section 3.2).  This builds that list, so that
 * scout_sparse_attn(_merge) can attend it: per unit, the valid blocks
 * j < ceil(seq_len[b] / P) whose residency bit is set, ascending.
 *
 * resident_bits uint32 [B][Hkv][ceil(nblk_cap/32)], seq_len int32 [B];
 * list int32 [B][Hkv][cap] (entries past the count set to -1), count int32
 * [B][Hkv].  A unit with more than cap such blocks gets its first cap of them and
 * SCOUT_DEV_OVERFLOW in dev_status (may be NULL).  One warp per unit.
 * ------------------------------------------------------------------------ */
#define SCOUT_DEV_OVERFLOW 4
int scout_resident_list(const uint32_t* resident_bits, const int32_t* seq_len, int B, int Hkv, int P, int nblk_cap,
                        int cap, int32_t* list, int32_t* count, int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * GPU partial attention over the resident selected blocks.
 * ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1 (A_gpu): the GPU
 * attends the top-k blocks that reside in its memory.
 *
 * For query head hq of sequence b (unit u = b * Hkv + hq / G): the tokens of
 * blocks res_list[u][0 .. res_count[u]) with t < seq_len[b];
 * s_t = scale * q . k_t;  O_part = sum_t softmax(s)_t v_t (normalised, fp32
 * [B][Hq][D]);  lse_part = ln sum_t exp(s_t) (fp32 [B][Hq]).  An empty set
 * gives O = 0 and lse = -inf.  The work is balanced over the SMs by splitting
 * the total block count evenly, split units being combined by LSE; when the
 * grid covers every unit and every unit is small, each CTA takes one whole unit.
 * workspace: scout_sparse_attn_workspace_bytes() bytes; its first 4 * B * Hkv
 * bytes must be zero before the first use and are left zero by every call.
 * K_pool / V_pool must be 16-byte aligned.  Requires G <= 8, res_count <= k,
 * B * Hkv <= 4096 and B * Hkv * k <= 2^28 (else SCOUT_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------ */
size_t scout_sparse_attn_workspace_bytes(int B, int Hq, int Hkv, int D, int P);
int scout_sparse_attn(const void* q, const void* K_pool, const void* V_pool, int64_t n_slots,
                      const int32_t* page_table, const int32_t* seq_len, const int32_t* res_list,
                      const int32_t* res_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k,
                      float scale, float* O_part, float* lse_part, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, const scout_launch* launch, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * GPU partial attention fused with the merge of the CPU partial.
 * ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1 (A_gpu, then
 * MERGE(A_gpu, A_cpu)): scout_sparse_attn followed by scout_merge in one launch;
 * the GPU partial never goes through memory.
 * Arguments as scout_sparse_attn, then O_cpu fp32 [B][Hq][D] and lse_cpu fp32
 * [B][Hq] (the CPU partial, lse = -inf when empty), O_out bf16 [B][Hq][D] and
 * lse_out fp32 [B][Hq] (may be NULL).  O_cpu must be 16-byte and O_out 8-byte
 * aligned.  The merge is the formula of scout_merge, evaluated in fp32.
 * ------------------------------------------------------------------------ */
int scout_sparse_attn_merge(const void* q, const void* K_pool, const void* V_pool, int64_t n_slots,
                            const int32_t* page_table, const int32_t* seq_len, const int32_t* res_list,
                            const int32_t* res_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k,
                            float scale, const float* O_cpu, const float* lse_cpu, void* O_out, float* lse_out,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            const scout_launch* launch, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Merge of the GPU and CPU partial results.
 * ScoutAttention (arXiv HTML), section 3.2 (FlashAttention / online-softmax
 * combination of the two devices' intermediate results) and Algorithm 1 (MERGE).
 *
 * For each of rows = B * Hq query heads:  m = max(lse_a, lse_b),
 * O = (e^{lse_a - m} O_a + e^{lse_b - m} O_b) / (e^{lse_a - m} + e^{lse_b - m}),
 * lse = m + ln(e^{lse_a - m} + e^{lse_b - m}); two empty partials give O = 0,
 * lse = -inf.  O_a, O_b fp32 [rows][D]; lse_a, lse_b fp32 [rows];
 * O_out bf16 [rows][D]; lse_out fp32 [rows] (may be NULL).
 * ------------------------------------------------------------------------ */
int scout_merge(const float* O_a, const float* lse_a, const float* O_b, const float* lse_b, int rows, int D,
                void* O_out, float* lse_out, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Asynchronous periodic recall (host side).
 * ScoutAttention (arXiv HTML), section 3.4: important blocks are periodically
 * copied from host memory back into GPU memory, off the critical path; the
 * copy is started after a layer's attention and only needed one step later.
 *
 * One op moves block `block` of unit `unit` from the host copy of the cache
 * into pool slot `slot`; `evict_block` (or -1) is the block that held the slot
 * before.  host_K / host_V: host memory (pinned for asynchronous copies),
 * layout bf16 [B][Hkv][nblk_cap][P][D].  ops is a HOST array.
 *
 * scout_recall_async: on side_stream, waits for wait_event (may be NULL), copies
 * K and V of every op (adjacent ops with consecutive blocks and slots become one
 * cudaMemcpyAsync), then records done_event (may be NULL).  host_K / host_V may be
 * any pinned host memory.  If a copy is refused (SCOUT_ERR_CUDA), the copies before
 * it stay enqueued and done_event is not recorded: the slots the ops name then hold
 * undefined bytes while the tables still give them to the evicted blocks, so the
 * caller must commit the evictions alone (the same ops with block = -1) before the
 * pool is read again.
 * scout_recall_gather_async: the same move as ONE kernel on side_stream, which reads
 * the pages straight from host memory (a warp per K or V page, 16-byte loads) and
 * writes them into their slots; scattered pages cost no copy call each.  d_ops is a
 * DEVICE array of the ops; host_K / host_V must be pinned host memory mapped into the
 * device's address space (cudaHostAlloc / cudaMallocHost, or cudaHostRegister-ed, on
 * a system with unified addressing; 16-byte aligned), else SCOUT_ERR_UNSUPPORTED.  An
 * op outside the tables or the pool is skipped and SCOUT_DEV_BAD_INDEX set in
 * dev_status (may be NULL).  A refused launch enqueues nothing and records no
 * done_event, so the pool and the tables are as before.
 * scout_commit_residency: on stream, waits for wait_event (normally the recall's
 * done_event), then for every op clears evict_block's page-table entry (-1) and
 * residency bit, and afterwards sets block's entry to slot and its bit (an op with
 * block = -1 only evicts).
 * d_ops is a DEVICE copy of the same ops.  Until the commit runs, the tables
 * still describe the old residency, so a failed or unfinished copy never makes a
 * block look resident.
 * ------------------------------------------------------------------------ */
typedef struct scout_recall_op {
  int32_t unit;
  int32_t block;
  int32_t slot;
  int32_t evict_block;
} scout_recall_op;

int scout_recall_async(const scout_recall_op* ops, int n_ops, const void* host_K, const void* host_V,
                       void* K_pool, void* V_pool, int64_t n_slots, int B, int Hkv, int D, int P,
                       int nblk_cap, const scout_launch* launch, cudaEvent_t wait_event, cudaStream_t side_stream,
                       cudaEvent_t done_event);
int scout_recall_gather_async(const scout_recall_op* d_ops, int n_ops, const void* host_K, const void* host_V,
                              void* K_pool, void* V_pool, int64_t n_slots, int B, int Hkv, int D, int P,
                              int nblk_cap, int32_t* dev_status, const scout_launch* launch, cudaEvent_t wait_event,
                              cudaStream_t side_stream, cudaEvent_t done_event);
int scout_commit_residency(const scout_recall_op* d_ops, int n_ops, int32_t* page_table, uint32_t* resident_bits,
                           int64_t n_slots, int B, int Hkv, int nblk_cap, cudaEvent_t wait_event,
                           cudaStream_t stream);

/* Plan of one recall step (host code, HOST memory in and out).
 * ScoutAttention (arXiv HTML), section 3.4 says only that important blocks are
 * recalled periodically; the policy here is a reading: per unit u, the selected
 * blocks that are not resident come in, the most important first (score
 * descending, lower block first), each into the slot of a resident block that is
 * not selected, the least important first (score ascending, lower block first);
 * the unit's resident set keeps its size and the recall stops when either side
 * runs out.
 * scores fp32 [units][nblk_cap] (the pooled scores scout_score_topk writes, -inf
 * past the valid blocks), topk_idx int32 [units][k] and topk_count [units],
 * resident_bits uint32 [units][ceil(nblk_cap / 32)], page_table int32
 * [units][nblk_cap].  Writes up to max_ops ops (per unit in ascending block
 * order) and their number to *n_ops.  SCOUT_ERR_WORKSPACE if more are needed;
 * SCOUT_ERR_INVALID_ARG for a list entry out of range or a resident block
 * without a slot. */
int scout_plan_recall(const float* scores, const int32_t* topk_idx, const int32_t* topk_count,
                      const uint32_t* resident_bits, const int32_t* page_table, int units, int nblk_cap, int k,
                      scout_recall_op* ops, int max_ops, int* n_ops);

/* ------------------------------------------------------------------------ *
 * Recall plan with residency per page (host code): a page is one block of one
 * sequence for all its KV heads (32 tokens x 8 heads x K and V = 128 KB in the
 * Qwen3 layout), the transfer unit whose PCIe rate the pages compare with
 * per-token transfers (arXiv HTML, the background on recall-based offloading,
 * Figure 3).  Selection stays per (sequence,
 * KV head) and the residency bits of a sequence's heads are identical.
 * Reading (section 3.4 leaves it open): per sequence, the pages some head selects
 * that are not resident come in, the most important first (importance = the
 * largest of its heads' scores; ties to the lower block); each takes the slots of
 * a resident page that no head selects, the least important first; the plan
 * stops when either side runs out.  Each pair becomes one op per KV head, (unit,
 * incoming block, that unit's slot of the evicted block, evicted block), grouped
 * by unit and, within a unit, in ascending incoming block order.
 * Arguments as for scout_plan_recall with units = B * Hkv.  Errors: as for
 * scout_plan_recall, plus SCOUT_ERR_INVALID_ARG when the residency bits of one
 * sequence's heads differ or an evicted page lacks a slot in some head. */
int scout_plan_recall_pages(const float* scores, const int32_t* topk_idx, const int32_t* topk_count,
                            const uint32_t* resident_bits, const int32_t* page_table, int B, int Hkv, int nblk_cap,
                            int k, scout_recall_op* ops, int max_ops, int* n_ops);

/* ------------------------------------------------------------------------ *
 * Per-layer recall intervals from an offline profile (host code).
 * ScoutAttention (arXiv HTML), section 3.4: the recall interval of each layer is
 * the largest number of decoding steps that keeps the measured CPU compute ratio
 * (tokens computed on the CPU over the sparse budget) below a threshold beta
 * (12% by default in the pages), read from a profiling run without recalls.
 *
 * ratio     fp32 [layers][steps] host: layer l's CPU compute ratio at the (s+1)-th
 *           decoding step after its resident set was refreshed (prefill or recall)
 * interval  int32 [layers] host out: the largest n in [1, steps] with
 *           ratio[l][s] < beta for every s < n; 1 when even the first step is not
 *           below beta (recall every step); steps when no profiled step reaches beta
 *           (the profile's horizon bounds the interval).  A NaN ratio counts as not
 *           below beta.
 * Errors (nothing written): SCOUT_ERR_INVALID_ARG for a NULL pointer, layers or
 * steps <= 0, or beta not a positive finite number. */
int scout_recall_intervals(const float* ratio, int layers, int steps, float beta, int32_t* interval);

/* ------------------------------------------------------------------------ *
 * CPU-side attention over the offloaded blocks (host code; no GPU involved).
 * ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1 (CPUAttn of B_cpu,
 * spawned one layer ahead): the selected blocks that are not resident on the GPU
 * are attended on the CPU, next to the host copy of the KV cache, with the
 * predicted query; the GPU merges the result with its own partial
 * (scout_merge, scout_sparse_attn_merge).
 *
 * q         bf16 [B][Hq][D] host: the query of the CPU side (Q_pred, one layer ahead)
 * K, V      bf16 [B][Hkv][nblk_cap][P][D] host: every block of the layer in logical
 *           order (block j of unit u = b * Hkv + kvh at K + ((u * nblk_cap + j) * P) * D)
 * seq_len   int32 [B] host; tokens t >= seq_len[b] are masked
 * cpu_list  int32 [B][Hkv][k] host, cpu_count int32 [B][Hkv] host: the CPU work list
 *           as scout_score_topk writes it (the first cpu_count[u] entries are used)
 * O_cpu     fp32 [B][Hq][D] host out: per query head the normalised output over the
 *           tokens of the unit's listed blocks (query head h reads KV head h / (Hq / Hkv))
 * lse_cpu   fp32 [B][Hq] host out: natural-log LSE of scale * q.k over those tokens;
 *           a unit with no token gives O = 0, LSE = -inf
 * n_threads worker threads, the calling thread included (0: one per hardware thread);
 *           never more than one per unit.  Units are dealt to the threads one at a time.
 * Synchronous: returns when every unit is done.  fp32 arithmetic, online softmax block
 * by block; each block's K and V are read once for all Hq / Hkv query heads of its KV
 * head, in register tiles of 4-wide fp32 vectors (the compiler's generic vectors: NEON on
 * AArch64).  No allocation visible to the caller; the threads live for the call.
 * Errors (nothing written): SCOUT_ERR_INVALID_ARG for a NULL pointer, a non-positive
 * size, Hq not a multiple of Hkv (or more than 8 query heads per KV head), scale <= 0,
 * a count outside [0, k] or a listed block outside [0, nblk_cap);
 * SCOUT_ERR_UNSUPPORTED for D != 128 or P not in {16, 32, 64}. */
int scout_cpu_attend(const void* q, const void* K, const void* V, const int32_t* seq_len, const int32_t* cpu_list,
                     const int32_t* cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k,
                     float scale, float* O_cpu, float* lse_cpu, int n_threads);

/* scout_cpu_attend_scalar: the same call, arguments, checks and outputs, computed with plain
 * scalar loops (16 partial sums per dot product, no register tiles): the portable form the
 * tiled one is checked against.  The two agree to fp32 rounding (they sum in different
 * orders), not bit for bit. */
int scout_cpu_attend_scalar(const void* q, const void* K, const void* V, const int32_t* seq_len,
                            const int32_t* cpu_list, const int32_t* cpu_count, int B, int Hq, int Hkv, int D, int P,
                            int nblk_cap, int k, float scale, float* O_cpu, float* lse_cpu, int n_threads);

/* ------------------------------------------------------------------------ *
 * The CPU side on a caller-owned pool of worker threads (host code).
 * ScoutAttention (arXiv HTML), section 3.3 and Algorithm 1: the CPU attention of
 * layer i+1 is spawned one layer ahead and runs while the GPU computes layer i; its
 * partial must be back before layer i+1 merges it.  A pipeline calling this every
 * layer keeps one pool (no thread start per call) and waits for each layer's
 * partial with a bound, so a late CPU side is reported instead of stalling it.
 *
 * scout_cpu_pool_create(n_threads): n_threads workers (0: one per hardware thread);
 *   NULL if no thread could be started.  scout_cpu_pool_threads: their number.
 * scout_cpu_attend_async(pool, ...): the arguments and checks of scout_cpu_attend
 *   (same errors, nothing written on error); starts the job on the pool's workers and
 *   returns at once.  One job at a time: SCOUT_ERR_INVALID_ARG while the previous
 *   one runs.  The buffers must stay valid until the job is done.  Results are bit
 *   for bit those of scout_cpu_attend (a unit is one worker's, whatever the count).
 * scout_cpu_pool_wait(pool, timeout_us): SCOUT_OK once the job is done (or when no
 *   job was started), SCOUT_ERR_TIMEOUT if it is still running after timeout_us
 *   microseconds (it keeps running: wait again, or destroy the pool, which waits).
 * scout_cpu_pool_destroy(pool): waits for a running job, joins the workers, frees
 *   the pool (NULL is a no-op).  No thread of the pool outlives it.
 * ------------------------------------------------------------------------ */
typedef struct scout_cpu_pool scout_cpu_pool;
scout_cpu_pool* scout_cpu_pool_create(int n_threads);
int scout_cpu_pool_threads(const scout_cpu_pool* pool);
void scout_cpu_pool_destroy(scout_cpu_pool* pool);
int scout_cpu_attend_async(scout_cpu_pool* pool, const void* q, const void* K, const void* V, const int32_t* seq_len,
                           const int32_t* cpu_list, const int32_t* cpu_count, int B, int Hq, int Hkv, int D, int P,
                           int nblk_cap, int k, float scale, float* O_cpu, float* lse_cpu);
int scout_cpu_pool_wait(scout_cpu_pool* pool, int64_t timeout_us);

#ifdef __cplusplus
}
#endif
#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#endif /* SCOUT_H_ */
