/*
 * rsa.h -- C ABI of librsa: blockwise ring self-attention (forward) on one
 * NVIDIA GB300 (sm_103a).
 *
 * Pages cited:
 *   [P1] "Sequence parallelism -- splitting the token dimension across GPUs"
 *        (llmdaily, day 58)
 *   [P3] "Sequence Parallelism" (glossary entry, zhongzhoutan-coder terms)
 *
 * The sequence of length T is cut into N contiguous chunks of T/N tokens
 * ([P1] "Split tokens across four GPUs").  Query chunks stay put while the
 * key/value chunks are visited in ring order ([P1] "A better mental model:
 * move blocks past the queries"); each (query chunk, KV chunk) pair gives a
 * partial output and a row log-sum-exp, folded into the running result with
 * the online-softmax rescale e^{m - m_new} ([P1] "But softmax seems to
 * require all attention scores at once").  All N chunks live on one GPU; a
 * ring step is a change of base address, not a copy.
 *
 * Conventions for every call:
 *   - Tensors are dense row-major.  q, k, v and out are [B, H, T, d]
 *     (d = d_k, the head dimension); lse is [B, H, T].  "Row" means one
 *     (b, h, t) query row.
 *   - Pointers named q, k, v, out, lse, o_*, lse_* and workspace are DEVICE
 *     pointers on the current CUDA device, 16-byte aligned (the *_host
 *     arguments of rsa_ring_attn_fwd_host are host pointers).  The caller
 *     owns every buffer it passes.  The library allocates no device memory
 *     at call time; its state is a device-side error word, the 64 MiB
 *     scratch array of rsa_ring_attn_fwd_noalloc (reserved when its device
 *     code loads), the host blocks handed out by rsa_host_alloc, and two
 *     copy streams with a pool of events per device for
 *     rsa_ring_attn_fwd_host.
 *   - Scores are scaled by 1/sqrt(d) ([P1] "Attention wants keys and values
 *     from other tokens", the attention equation); the scale is not a
 *     parameter.  lse is the natural-log log-sum-exp of the scaled scores.
 *   - Causal means query position t sees keys 0..t inclusive ([P1] "Causal
 *     attention gives us another optimization"; the page's token 30,000
 *     attends to 1..30,000).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and is
 *     asynchronous: results are valid once the stream has passed the call.
 *     No call synchronises, except rsa_check_device_error.
 *   - Arguments are validated before anything is launched, so a call that
 *     returns RSA_ERR_INVALID_ARG or RSA_ERR_UNSUPPORTED has no side effect.
 *     A failed launch returns RSA_ERR_CUDA.  A device-side wait that ran past
 *     its time limit sets the device error word; rsa_check_device_error then
 *     returns RSA_ERR_TIMEOUT.  Nothing aborts, exits or traps.
 *   - rsa_last_error_string() describes the last failure on this thread.
 *
 * Supported shapes: fp32 inputs with d in {64, 128} (SIMT kernel), bf16
 * inputs with d in {64, 128} (tcgen05 tensor-core kernel).
 */
#ifndef RSA_H
#define RSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *rsa_stream_t; /* the same handle as cudaStream_t */
typedef struct CUevent_st *rsa_event_t;   /* the same handle as cudaEvent_t */

typedef enum {
    RSA_OK = 0,
    RSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, N does not divide T ... */
    RSA_ERR_UNSUPPORTED = 2, /* valid request this build does not serve (dtype, d, device) */
    RSA_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
    RSA_ERR_TIMEOUT = 4      /* a device wait exceeded its limit (see rsa_set_wait_limit_ns) */
} rsa_status;

typedef enum { RSA_F32 = 0, RSA_BF16 = 1 } rsa_dtype;

/*
 * One (query chunk, KV chunk) pair -- the block step of [P1] "A better mental
 * model: move blocks past the queries": the queries q[:, :, q_off : q_off+q_len]
 * attend to the keys/values k, v[:, :, kv_off : kv_off+kv_len]:
 *   o_blk   = softmax(Q_i K_j^T / sqrt(d)) V_j       [B, H, q_len, d], dtype dt
 *   lse_blk = log sum_j e^{s_j}                      [B, H, q_len], fp32
 * q, k, v are the FULL [B, H, T, d] tensors; the offsets are global token
 * positions, so the causal mask compares kv_off + c with q_off + r.  Rows with
 * no allowed key get o_blk = 0 and lse_blk = -inf.
 * Requires 0 <= q_off, q_off + q_len <= T, 0 <= kv_off, kv_off + kv_len <= T,
 * q_len, kv_len >= 1.
 */
rsa_status rsa_block_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt,
                              int B, int H, int64_t T, int d,
                              int64_t q_off, int64_t q_len, int64_t kv_off, int64_t kv_len,
                              int causal, void *o_blk, float *lse_blk, rsa_stream_t stream);

/*
 * One (query block, KV block) pair on buffers that hold only part of the
 * sequence, folded into a running fp32 accumulator -- the per-round step of
 * a rank in a multi-GPU ring ([P1] "A better mental model: move blocks past
 * the queries": a rank keeps its queries and receives other ranks' K/V
 * blocks into a local buffer; [P1] "But softmax seems to require all
 * attention scores at once": each block is folded into running statistics).
 *   q        [B, H, q_rows, d]  this rank's queries (dtype dt)
 *   k, v     [B, H, kv_rows, d] a K/V block (own or received), dtype dt
 *   acc      [B, H, q_rows, d]  fp32 accumulator (normalised o)
 *   lse      [B, H, q_rows]     fp32 running log-sum-exp (and the final lse)
 *   out      [B, H, q_rows, d]  the result, dtype dt
 * The pair is query rows [q_row0, q_row0 + q_len) -- at global sequence
 * positions q_pos, q_pos + 1, ... -- against key rows [kv_row0, kv_row0 +
 * kv_len) at global positions kv_pos, ...; the positions drive the causal
 * mask (key position <= query position), the rows the memory accesses.
 * fold says what happens to the pair's (o, lse) for those query rows:
 *   RSA_FOLD_FIRST  written to acc and lse (the rows' first pair)
 *   RSA_FOLD_MERGE  merged into acc and lse in place (the rule of rsa_merge)
 *   RSA_FOLD_LAST   merged with acc and lse and written to out and lse
 *                   (acc is only read)
 *   RSA_FOLD_ONLY   the rows' only pair: written to out and lse (acc unused)
 * A row whose running lse is -inf is empty and its acc values are not read.
 * Requires the row ranges inside their tensors and non-negative positions;
 * acc must be given unless fold is RSA_FOLD_ONLY, out for RSA_FOLD_LAST and
 * RSA_FOLD_ONLY.
 */
enum { RSA_FOLD_FIRST = 0, RSA_FOLD_MERGE = 1, RSA_FOLD_LAST = 2, RSA_FOLD_ONLY = 3 };
rsa_status rsa_block_attn_fold(const void *q, int64_t q_rows, const void *k, const void *v, int64_t kv_rows,
                               rsa_dtype dt, int B, int H, int d,
                               int64_t q_row0, int64_t q_pos, int64_t q_len,
                               int64_t kv_row0, int64_t kv_pos, int64_t kv_len,
                               int causal, int fold, float *acc, float *lse, void *out,
                               rsa_stream_t stream);

/*
 * The pair list of one rank in a ring of N ranks over a sequence of T
 * tokens ([P1] "A better mental model: move blocks past the queries": in
 * round r rank i holds the K/V block of rank (i - r) mod N; [P1] "Causal
 * attention gives us another optimization": pairs whose keys all lie after
 * their queries are skipped).  Which tokens a rank owns:
 *   RSA_LAYOUT_CONTIGUOUS  rank i owns tokens [i T/N, (i+1) T/N)
 *   RSA_LAYOUT_ZIGZAG      with S = T/(2N): rank i owns the two pieces
 *                          [i S, (i+1) S) and [(2N-1-i) S, (2N-i) S), in
 *                          that order in its buffers, so that under the
 *                          causal mask every rank does the same work in
 *                          every round after the first
 * Each step is 9 int64 values, in execution order (rounds ascending):
 *   round, src_rank (= (rank - round) mod N, whose K/V block the step reads),
 *   q_row0, q_pos, q_len, kv_row0, kv_pos, kv_len, fold
 * ready for rsa_block_attn_fold (kv_row0 indexes src_rank's buffer).  Writes
 * up to `cap` steps and their count to *n_steps.  Needs N | T (2N | T for
 * zigzag).  Host only.
 */
enum { RSA_LAYOUT_CONTIGUOUS = 0, RSA_LAYOUT_ZIGZAG = 1 };
rsa_status rsa_rank_ring_plan(int N, int rank, int64_t T, int causal, int layout, int64_t *steps, int cap,
                              int *n_steps);

/*
 * Online-softmax merge, in place, of [P1] "But softmax seems to require all
 * attention scores at once" written for normalised partials:
 *   a = lse_acc, b = lse_blk, M = max(a, b), L = M + ln(e^{a-M} + e^{b-M})
 *   o_acc <- o_acc e^{a-L} + o_blk e^{b-L},   lse_acc <- L
 * over `rows` contiguous rows of d values.  o_acc is fp32; o_blk has dtype
 * blk_dt.  A row whose lse is -inf is empty: its o values are not used (they
 * may hold anything, NaN included), so merging with it is the identity, and
 * two empty rows give o = 0, lse = -inf.
 */
rsa_status rsa_merge(float *o_acc, float *lse_acc, const void *o_blk, rsa_dtype blk_dt,
                     const float *lse_blk, int64_t rows, int d, rsa_stream_t stream);

/*
 * The same merge as rsa_merge, but the result is written to `out` (dtype
 * out_dt, rounded to nearest even for bf16) and `lse_out` instead of back
 * into the accumulator: the last merge of a ring.  o_acc/lse_acc are read
 * only.  lse_out may alias lse_acc.
 */
rsa_status rsa_merge_finalize(const float *o_acc, const float *lse_acc, const void *o_blk,
                              rsa_dtype blk_dt, const float *lse_blk, int64_t rows, int d,
                              void *out, rsa_dtype out_dt, float *lse_out, rsa_stream_t stream);

/*
 * Bytes of device workspace rsa_ring_attn_fwd needs for this shape (written
 * to *bytes): an fp32 accumulator [B, H, T, d] (none when N = 1).  (The
 * RSA_RING_SEPARATE_MERGE variant needs more; see
 * rsa_ring_attn_workspace_size_ex.)
 */
rsa_status rsa_ring_attn_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N,
                                        int causal, size_t *bytes);

/*
 * Whole ring on one GPU ([P1] "A better mental model: move blocks past the
 * queries", with [P1] "Causal attention gives us another optimization"):
 * round r pairs query chunk i with KV chunk (i - r) mod N; when causal, pairs
 * whose KV chunk lies after the query chunk are skipped, leaving N(N+1)/2
 * pairs.  Round 0 (the diagonal) writes straight into the accumulator (or into
 * out/lse for a chunk visited once); in every later round each pair's block
 * epilogue folds its (o, lse) into the fp32 accumulator with the merge rule of
 * rsa_merge, and a chunk's last pair writes out (dtype dt) and lse.  (Pairs of
 * one round never share a query chunk, so the in-place fold is race-free.)
 * Requires N >= 1 and N dividing T.  `workspace` must hold
 * rsa_ring_attn_workspace_size() bytes.  The call only enqueues kernels on
 * `stream` (no synchronisation, no allocation), so a stream capture records
 * the whole ring as one CUDA graph that can be replayed.
 */
rsa_status rsa_ring_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt,
                             int B, int H, int64_t T, int d, int N, int causal,
                             void *out, float *lse, void *workspace, size_t ws_bytes,
                             rsa_stream_t stream);

/*
 * rsa_ring_attn_fwd for callers that cannot allocate device memory (the pages
 * have no counterpart; this is a library convenience).  Some callers cannot
 * provide a workspace: their device memory belongs to another allocator that
 * must not be bypassed, or a cudaMalloc (with the synchronisation it may
 * imply) is not allowed where they run.  This call uses a fixed 64 MiB
 * scratch array built into the library instead and allocates nothing.
 * Arguments and results are those of rsa_ring_attn_fwd; a shape whose
 * workspace (rsa_ring_attn_workspace_size) exceeds 64 MiB is rejected with
 * RSA_ERR_INVALID_ARG.  The 64 MiB are reserved on a device when the
 * library's device code is loaded into that device's context -- no later
 * than this call's first use there, and, under eager module loading
 * (CUDA_MODULE_LOADING=EAGER), on every device the process initialises even
 * if this call is never made -- and stay reserved until the process exits.
 * The first call in each CUDA context looks up the scratch address (and
 * again in a new context, e.g. after cudaDeviceReset); make it before any
 * stream capture.  All calls share the one scratch array, so calls that may
 * overlap on the GPU (different streams or unsynchronised host threads) race
 * and must be serialised by the caller.
 */
rsa_status rsa_ring_attn_fwd_noalloc(const void *q, const void *k, const void *v, rsa_dtype dt,
                                     int B, int H, int64_t T, int d, int N, int causal,
                                     void *out, float *lse, rsa_stream_t stream);

/*
 * rsa_ring_attn_fwd with profiling: before and after each kernel launch it
 * records ev_start[i] / ev_stop[i] on `stream` and sets kind[i] to 0 for a
 * block-attention launch or 1 for a merge launch.  `cap` is the length of the
 * three arrays (host memory; the events are created by the caller); the number
 * of launches is written to *n_launches (the call fails with
 * RSA_ERR_INVALID_ARG, before launching anything, if cap is too small).
 */
rsa_status rsa_ring_attn_fwd_timed(const void *q, const void *k, const void *v, rsa_dtype dt,
                                   int B, int H, int64_t T, int d, int N, int causal,
                                   void *out, float *lse, void *workspace, size_t ws_bytes,
                                   rsa_stream_t stream, rsa_event_t *ev_start,
                                   rsa_event_t *ev_stop, int *kind, int cap, int *n_launches);

/*
 * Ring variant flags for rsa_ring_attn_fwd_ex / rsa_ring_attn_workspace_size_ex.
 *
 * RSA_RING_FUSED_MERGE (the default of rsa_ring_attn_fwd; 0 means the same):
 * rounds after the first do not write partials; each pair's block epilogue
 * folds its (o, lse) straight into the fp32 accumulator with the same merge
 * rule as rsa_merge (and the chunk's last pair writes out/lse).  No merge
 * launches and no partial buffers: the workspace is the accumulator alone.
 *
 * RSA_RING_SEPARATE_MERGE: every round after the first writes its pairs'
 * fp32 partials (o, lse) to the workspace and one merge-kernel launch folds
 * them into the accumulator (the chunk's last merge writes out/lse).  The
 * workspace adds one round's partials.  Same results within rounding.
 *
 * The two exclude each other.
 */
#define RSA_RING_FUSED_MERGE 1u
#define RSA_RING_SEPARATE_MERGE 2u

/* Workspace bytes for rsa_ring_attn_fwd_ex with these flags. */
rsa_status rsa_ring_attn_workspace_size_ex(rsa_dtype dt, int B, int H, int64_t T, int d, int N,
                                           int causal, unsigned flags, size_t *bytes);

/*
 * rsa_ring_attn_fwd with variant `flags` and optional profiling: when
 * ev_start, ev_stop and kind are all non-NULL it records events around each
 * launch as rsa_ring_attn_fwd_timed does (kind 0 block attention, 1 merge);
 * when all three are NULL nothing is recorded.  *n_launches (if non-NULL)
 * receives the number of kernel launches.  flags = 0 (or
 * RSA_RING_FUSED_MERGE) is rsa_ring_attn_fwd.
 */
rsa_status rsa_ring_attn_fwd_ex(const void *q, const void *k, const void *v, rsa_dtype dt,
                                int B, int H, int64_t T, int d, int N, int causal, unsigned flags,
                                void *out, float *lse, void *workspace, size_t ws_bytes,
                                rsa_stream_t stream, rsa_event_t *ev_start, rsa_event_t *ev_stop,
                                int *kind, int cap, int *n_launches);

/*
 * Page-locked host memory for streaming copies (the one call of this library
 * that allocates; it allocates host memory only).  The block is `bytes`
 * rounded up to the transparent-huge-page size, aligned to it, advised for
 * huge pages, zeroed (so every page exists) and registered with the CUDA
 * driver.  Rationale: copy-engine transfers from page-locked memory on base
 * pages were measured to lose most of their bandwidth once the memory had sat
 * idle for some seconds (from 211 GB/s towards 10-20 GB/s on GB300 hosts with
 * 64 KiB pages), while huge-page-backed memory kept its speed.  Registering
 * pins the pages, which may make the kernel migrate them and split huge
 * pages; the huge-page share is therefore measured after registering, and a
 * block below 90% is given back and allocated again (up to four attempts,
 * the best one kept).  If no attempt reaches 90% the block comes from
 * cudaHostAlloc instead.  *ptr receives the block (NULL on failure).
 * Release it with rsa_host_free.  Host only; needs the CUDA driver.
 */
enum { RSA_HOST_HUGE = 1, RSA_HOST_PINNED = 2 };
rsa_status rsa_host_alloc(size_t bytes, void **ptr);
rsa_status rsa_host_free(void *ptr);
/*
 * What rsa_host_alloc handed out at `ptr`: its usable bytes, the bytes the
 * kernel currently backs with huge pages (0 for RSA_HOST_PINNED), and its
 * kind (RSA_HOST_HUGE: huge-page memory registered with the driver;
 * RSA_HOST_PINNED: cudaHostAlloc).  Any output pointer may be NULL.
 */
rsa_status rsa_host_info(const void *ptr, size_t *bytes, size_t *huge_bytes, int *kind);

/*
 * How rsa_ring_attn_fwd_host moves each host tensor (process wide; set
 * before the calls it should affect):
 *   RSA_HOST_COPY_AUTO     (default) per copy: the copy engines
 *                          (cudaMemcpyAsync) for pageable memory and for a
 *                          copy whose range of a block from rsa_host_alloc
 *                          is still at least 90% on huge pages; a copy
 *                          kernel otherwise, i.e. for page-locked memory on
 *                          base pages (cudaHostAlloc, cudaHostRegister) and
 *                          for the parts of a library block that the kernel
 *                          has split.  Each call reads each such tensor's
 *                          huge-page regions from the kernel's page tables
 *                          once (Linux 6.7 on); older kernels give no
 *                          regions, and then the whole tensor goes one way,
 *                          by its block's AnonHugePages in /proc/self/smaps
 *   RSA_HOST_COPY_ENGINES  always the copy engines
 *   RSA_HOST_COPY_SM       the copy kernel for all page-locked memory
 * The copy kernel (256-thread CTAs on half as many CTAs as the GPU has SMs,
 * beside the ring's CTAs)
 * reads and writes the page-locked memory through its mapped address.
 * Measured on GB300 hosts: copy-engine transfers of page-locked memory on
 * 64 KiB pages fell from 211 GB/s towards 10 GB/s within seconds of idling,
 * and huge-page blocks copied at 5-120 GB/s once the kernel had split some
 * of their pages, while the copy kernel moved the same memory at 193-211
 * GB/s alone and about 127 GB/s beside the ring, which it slowed by about a
 * tenth; copy engines beside the ring slowed it by 2%.
 * Returns RSA_ERR_INVALID_ARG for another mode.
 */
enum { RSA_HOST_COPY_AUTO = 0, RSA_HOST_COPY_ENGINES = 1, RSA_HOST_COPY_SM = 2 };
rsa_status rsa_set_host_copy_mode(int mode);

/*
 * The path rsa_ring_attn_fwd_host would take now for one copy of the host
 * buffer [ptr, ptr + bytes): RSA_HOST_PATH_ENGINES or RSA_HOST_PATH_KERNEL.
 * The call itself copies a tensor slab by slab and decides each copy on its
 * own range, so a tensor whose block is split in places moves partly each way.
 */
enum { RSA_HOST_PATH_ENGINES = 1, RSA_HOST_PATH_KERNEL = 2 };
rsa_status rsa_host_copy_path(const void *ptr, size_t bytes, int *path);

/*
 * The slab plan of rsa_ring_attn_fwd_host: how many heads each slab holds, in
 * streaming order, for BH = B*H heads cut into about `groups` slabs of at most
 * ceil(BH/groups) heads.  With ramp, the plan starts at an eighth of the
 * largest slab and grows about 1.6x per slab, keeps equal slabs in the middle
 * and shrinks back to an eighth at the end, so each slab's copy hides under
 * the ring of the slab before it and only a small first copy in and last copy
 * out are exposed.  Without ramp: equal slabs.  Writes up to `cap` entries
 * and their count to *n_slabs.  Host only.
 */
rsa_status rsa_host_slab_plan(int BH, int groups, int ramp, int *slabs, int cap, int *n_slabs);

/*
 * Device workspace for rsa_ring_attn_fwd_host: two slots of the largest
 * slab's q, k, v, out and lse, plus the ring workspace of one slab.
 */
rsa_status rsa_ring_attn_host_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N,
                                             int causal, size_t *bytes);

/*
 * rsa_ring_attn_fwd from host memory to host memory, the copies overlapped
 * with the ring ([P1] "A better mental model: move blocks past the queries":
 * blocks stream past queries that stay put).  q_host, k_host, v_host
 * [B, H, T, d] (dtype dt) and out_host [B, H, T, d], lse_host [B, H, T] fp32
 * are HOST pointers.  The B*H heads are independent problems, so they are cut
 * into slabs (rsa_host_slab_plan(B*H, 8, 1)): while the ring of slab g runs on
 * `stream`, slab g+1 is copied in and slab g-1 copied out on two copy streams
 * the library creates for the current device on its first call there (with
 * their events; all are kept until the process exits).  Each slab of each
 * tensor moves by the copy engines or by a copy kernel, decided per copy
 * (rsa_set_host_copy_mode).  Device slabs are
 * double-buffered in `workspace` (a DEVICE pointer, 256-byte aligned, at
 * least rsa_ring_attn_host_workspace_size() bytes).  The results equal
 * rsa_ring_attn_fwd's bit for bit.
 *   - The host buffers should be page-locked (rsa_host_alloc, cudaHostAlloc or
 *     cudaHostRegister); pageable memory works but the CUDA runtime then
 *     stages each copy and the overlap is lost.
 *   - The call returns once everything is enqueued; out_host and lse_host
 *     hold the results once `stream` has passed the call.  The inputs must
 *     not change, and the outputs must not be read, before then.
 *   - Calls from several host threads on one device are serialised while
 *     they enqueue.
 *   - Argument errors are found before anything is enqueued.  A CUDA error
 *     during enqueueing returns RSA_ERR_CUDA and may leave earlier slabs'
 *     copies and rings enqueued.
 */
rsa_status rsa_ring_attn_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                                  rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal,
                                  void *out_host, float *lse_host, void *workspace, size_t ws_bytes,
                                  rsa_stream_t stream);

/*
 * Decode against a distributed KV cache ([P1] "Training and inference stress
 * this dimension differently": the history of keys and values is split
 * across devices, a new query is evaluated against every block and the
 * partial results are combined).  The cache k, v [B, H, T, d] is cut into N
 * contiguous shards of T/N keys (here all on this GPU); each shard is cut
 * further into splits for parallelism.  Every split yields an fp32 partial
 * (o, lse) for each query row, and the partials are folded with the rule of
 * rsa_merge.
 *   q    [B, H, q_len, d]: the q_len newest tokens, at global positions
 *        T - q_len .. T - 1 (their keys and values are already in the cache)
 *   out  [B, H, q_len, d] (dtype dt), lse [B, H, q_len] fp32
 * causal: row r sees keys 0 .. T - q_len + r; otherwise every key.
 * Requires 1 <= q_len <= T and N dividing T.  `workspace` must hold
 * rsa_decode_workspace_size() bytes.
 */
rsa_status rsa_decode_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int q_len, int N,
                                     size_t *bytes);
rsa_status rsa_decode_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt,
                               int B, int H, int64_t T, int d, int q_len, int N, int causal,
                               void *out, float *lse, void *workspace, size_t ws_bytes,
                               rsa_stream_t stream);

/*
 * Two-pass Ring Self-Attention ([P3] "How It Works", steps 1-2), the form that
 * keeps whole score rows: for each query chunk n in turn, the score pass
 * visits the key chunks in ring order (n - r) mod N and fills the full score
 * rows S^n = Q_n K^T / sqrt(d) (future keys -inf when causal); softmax is
 * taken over each full row (lse = log-sum-exp of the row); the output pass
 * visits the value chunks in the same ring order and accumulates
 * O^n = sum_j P^n_j V_j in fp32.  Same inputs and outputs as
 * rsa_ring_attn_fwd; the workspace holds one chunk's fp32 scores and bf16
 * probabilities, B*H*(T/N)*T*6 bytes -- the O(L/N * L) memory the online
 * merge avoids -- plus per-row statistics of each 64 keys of the row,
 * B*H*(T/N)*(T/64)*8 bytes (each part rounded up to 256 bytes).  Built for
 * bf16 with d = 128 and T/N a multiple of 128 (RSA_ERR_UNSUPPORTED
 * otherwise).
 */
rsa_status rsa_two_pass_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N,
                                       size_t *bytes);
rsa_status rsa_two_pass_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt,
                                 int B, int H, int64_t T, int d, int N, int causal,
                                 void *out, float *lse, void *workspace, size_t ws_bytes,
                                 rsa_stream_t stream);

/*
 * Host-only view of the ring schedule used by rsa_ring_attn_fwd: the pairs of
 * round r (0-based) as (q_chunk[p], kv_chunk[p]) in host arrays of length
 * `cap`; their count goes to *n_pairs.  No GPU needed.
 */
rsa_status rsa_ring_schedule(int N, int causal, int round, int *q_chunk, int *kv_chunk, int cap,
                             int *n_pairs);

/* Set the limit (nanoseconds, >= 1 ms) of every device-side wait; default 2 s. */
rsa_status rsa_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Which bf16 tensor-core kernel computes the blocks of later calls (process
 * wide).  Both give the result of rsa_block_attn_fwd; they differ in how the
 * work is laid out on the GPU:
 *   RSA_BLOCK_KERNEL_ONE_SM  one CTA per 256 query rows of a (pair, head);
 *   RSA_BLOCK_KERNEL_TWO_SM  one pair of CTAs (a two-CTA cluster) per 512
 *                            rows, sharing each K/V tile through the paired
 *                            (cta_group::2) MMA; used for d = 128 when a
 *                            pair has at least 512 query rows and its key
 *                            range is not split (not the decode path);
 *   RSA_BLOCK_KERNEL_AUTO    (default) the one-SM kernel, measured the
 *                            faster of the two on every workload this
 *                            library is benchmarked on.
 * Returns RSA_ERR_INVALID_ARG for any other value.  Host only.
 */
enum { RSA_BLOCK_KERNEL_AUTO = 0, RSA_BLOCK_KERNEL_ONE_SM = 1, RSA_BLOCK_KERNEL_TWO_SM = 2 };
rsa_status rsa_set_block_kernel(int which);

/*
 * Failure injection for testing callers' error handling (process wide, off
 * by default).  With countdown = n >= 0, the library's next n kernel
 * launches proceed and the one after that is not made: the call making it
 * returns RSA_ERR_CUDA with "injected launch failure" in
 * rsa_last_error_string(), exactly as if the launch had failed, and the
 * injection switches itself off.  Launches of the same call before it have
 * been enqueued; nothing after it is.  countdown < 0 switches it off.  Host
 * only; no GPU fault is involved.
 */
rsa_status rsa_debug_inject_launch_failure(int countdown);

/*
 * 1 if this library was built with RSA_DEBUG: its kernels then check the
 * indices of their computed global-memory accesses (output, accumulator and
 * lse rows, fp32 K/V rows, merge rows, the two-pass statistics, lse and
 * output rows); an access that fails its check is skipped, and the first
 * failure's site code and index are recorded for rsa_check_device_error,
 * which reports RSA_ERR_CUDA.  No trap.  0 for the normal build, whose
 * kernels carry no such checks.
 */
int rsa_debug_checks(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device: RSA_OK, RSA_ERR_TIMEOUT if a kernel gave up on a wait, or
 * RSA_ERR_CUDA if a bounds check of an RSA_DEBUG build failed (the text gives
 * the site code and the first bad index).
 */
rsa_status rsa_check_device_error(rsa_stream_t stream);

/*
 * Self-test of the wait limit: launches one block that waits, with the
 * current limit, on a shared-memory barrier nothing ever arrives at; the wait
 * gives up and sets the device error word, which rsa_check_device_error
 * reports as RSA_ERR_TIMEOUT.  The block then exits normally.
 */
rsa_status rsa_selftest_wait_timeout(rsa_stream_t stream);

const char *rsa_status_string(rsa_status status);
const char *rsa_last_error_string(void);
int rsa_version(void); /* major * 10000 + minor * 100 + patch */

#ifdef __cplusplus
}
#endif

#endif /* RSA_H */
