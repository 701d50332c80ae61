/*
 * msa.h -- C ABI of the GB300 (sm_103a) MSA block-sparse top-k attention backward.
 *
 * The operation is the backward pass of MiniMax-M3 MSA attention as stated on
 * the NVIDIA NeMo AutoModel API pages for minimax_m3_vl: every query chunk of
 * C = 8 tokens and each index head attends only to its selected top-k key
 * blocks of B = 64 keys, causally within the packed documents of cu_seqlens,
 * with G = 16 query heads sharing one index/KV head; the pass returns dQ, dK
 * and dV in bf16 ("msa_backward_sm100" page, module docstring and
 * run_backward; "msa_schedule" page, MSABackwardSchedule).
 *
 * Conventions shared by every call:
 *  - Every pointer named "device" is CUDA device memory owned by the caller.
 *    The library allocates nothing, never synchronises and keeps no state
 *    between calls except memoised device queries (SM count, capability).
 *  - Calls are asynchronous and ordered on the given stream (a cudaStream_t
 *    passed as void*; NULL is the legacy default stream).
 *  - Tensors are row-major THD: [tokens, heads, head_dim] with head_dim
 *    contiguous, the view the pages' _head_major helper describes.  bf16
 *    tensors are passed as uint16_t bit patterns.  Every pointer must be
 *    16-byte aligned (the pages' _operand helper).
 *  - The return value reports errors detectable on the host.  Errors found on
 *    the device (capacity, invalid selection, timeout) are written to the
 *    caller's device word *d_status with the first error winning; the caller
 *    sets it to 0 before a sequence of calls and reads it after a sync.  Each
 *    kernel returns without touching its outputs if *d_status is already
 *    non-zero, so tables from a failed build are never consumed.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  The pages raise TypeError/ValueError on a malformed schedule
 * ("msa_schedule" page, MSABackwardSchedule, Raises) and NotImplementedError
 * on a device that is not the one the kernels are built for ("kernels" page,
 * require_sm100); here both become integer codes. */
enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARGUMENT = 1,   /* null / misaligned pointer, bad size or count        */
  MSA_ERR_UNSUPPORTED_DEVICE = 2, /* compute capability is not 10.3 (sm_103a build)     */
  MSA_ERR_UNSUPPORTED_SHAPE = 3,  /* a shape the kernels are not built for               */
  MSA_ERR_CAPACITY = 4,           /* edge_cap or task_cap too small (device-detected)    */
  MSA_ERR_INVALID_SELECTION = 5,  /* sel entry out of range, non-causal or repeated      */
  MSA_ERR_TIMEOUT = 6,            /* a bounded device wait expired                       */
  MSA_ERR_CUDA = 7,               /* a CUDA launch or runtime call failed                */
  MSA_ERR_INVALID_DOCUMENTS = 8,  /* cu_seqlens / kv_doc_starts inconsistent (device)    */
  MSA_ERR_SCRATCH_TOO_SMALL = 9   /* problem exceeds the no-allocation scratch array     */
};

/* Problem description.  Mirrors run_backward's tensor contract
 * ("msa_backward_sm100" page, run_backward parameters) and the schedule's
 * cu_seqlens / document_workspace_starts ("msa_schedule" page).
 *
 * num_docs        N >= 1 documents packed along the token axis.
 * total_tokens    T = cu_seqlens[N].
 * cu_seqlens      device int32 [N+1]; cu[0] = 0, strictly increasing.
 * kv_doc_starts   device int32 [N]; K/V row of each document's first key.
 *                 Equal to cu_seqlens[0..N) for compact K/V; a multiple of
 *                 128 per document for the pages' aligned workspace.  Ranges
 *                 [kv_doc_starts[d], kv_doc_starts[d] + len_d) must increase
 *                 with d and not overlap.  K/V rows outside every document
 *                 must hold finite values; their gradients are written as 0.
 * kv_rows         W, rows of the K/V workspace (W = T for compact K/V).
 * num_q_heads     Hq; num_index_heads = num_kv_heads = Hq / 16.
 * head_dim        128.   block_size 64.   query_chunk 8.
 * topk            K, 1 <= K <= 32, slots per (index head, query chunk).
 * num_blocks      NB = sum_d ceil(len_d / block_size) (host copy, for sizing).
 * num_chunks      NC = sum_d ceil(len_d / query_chunk).
 * softmax_scale   scale applied to q.k (the pages use head_dim ** -0.5).
 */
typedef struct {
  int32_t num_docs;
  int32_t total_tokens;
  const int32_t* cu_seqlens;
  const int32_t* kv_doc_starts;
  int32_t kv_rows;
  int32_t num_q_heads;
  int32_t num_index_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t query_chunk;
  int32_t topk;
  int32_t num_blocks;
  int32_t num_chunks;
  float softmax_scale;
} msa_problem;

/* Columns of a task_meta row: the pages' scheduler_metadata column order
 * (index_head, row_linear, q_begin, q_count, document_ordinal,
 * document_local_kblock) ("msa_schedule" page, MSABackwardSchedule).
 * q_begin is the CSR offset of the task's first query entry. */
enum { MSA_TASK_META_COLS = 6 };

/* Layout of the int32 walk descriptor written by msa_build_tasks: the CTA
 * walk rule of the "msa_schedule" page (rows_per_cta, chunk_map).
 * walk[MSA_WALK_ROWS] rows (tasks); [MSA_WALK_ROWS_PER_CTA] R (4 below 2400
 * rows, else 64); [MSA_WALK_FULL] full units of R rows; [MSA_WALK_TAIL] tail
 * rows; [MSA_WALK_GRID] units = full + min(tail, num_sms); [MSA_WALK_SMS]. */
enum {
  MSA_WALK_ROWS = 0, MSA_WALK_ROWS_PER_CTA = 1, MSA_WALK_FULL = 2, MSA_WALK_TAIL = 3,
  MSA_WALK_GRID = 4, MSA_WALK_SMS = 5, MSA_WALK_LEN = 8
};

/* Bytes of device workspace one sequence msa_build_k2q -> msa_build_tasks ->
 * msa_bwd needs (the calls may share one buffer, used in stream order).
 * Returns 0 if the problem is invalid. */
size_t msa_workspace_bytes(const msa_problem* p, int64_t edge_cap, int64_t task_cap,
                           int32_t task_tile_chunks);
/* msa_workspace_bytes for a backward run with options (MSA_BWD_DQ_FP32 adds
 * an fp32 dQ accumulator of T * Hq * 128 * 4 bytes).  Returns 0 for an
 * invalid problem or an unknown option bit. */
size_t msa_workspace_bytes_opts(const msa_problem* p, int64_t edge_cap, int64_t task_cap,
                                int32_t task_tile_chunks, uint32_t options);

/* Key-block -> query CSR ("msa_bindings" page, build_k2q_csr;
 * "msa_schedule" page, row_ptr and q_indices).
 *
 * sel        device int32 [Hi, NC, K]: for index head hi and global query
 *            chunk g (document-major numbering), the document-local key
 *            blocks the chunk attends; -1 marks an empty slot (any slot).
 *            Valid entries are distinct and causal: b * block_size <= the
 *            chunk's first query position; otherwise *d_status =
 *            MSA_ERR_INVALID_SELECTION.
 * row_ptr    device int32 [Hi, NB+1] out: row r = blk_off[d] + b of head hi
 *            holds q_indices[hi][row_ptr[hi][r] .. row_ptr[hi][r+1]).
 * q_indices  device int32 [Hi, edge_cap] out: document-local query positions
 *            of each row, ascending.  Entries past a head's last row are
 *            left untouched.
 * edge_cap   capacity per head; too small -> *d_status = MSA_ERR_CAPACITY.
 * The result is deterministic (bit-identical on every run).
 */
int msa_build_k2q(const msa_problem* p, const int32_t* sel, int32_t* row_ptr, int32_t* q_indices,
                  int64_t edge_cap, int32_t* d_status, void* ws, size_t ws_bytes, void* stream);

/* msa_build_k2q for callers that cannot allocate device memory.  The pages
 * have no counterpart: this entry point exists for library users, not for the
 * method.  Some callers may not call cudaMalloc at all: a host framework whose
 * caching allocator or fixed memory pool owns all device memory, or a latency-
 * sensitive path that cannot afford cudaMalloc's implicit synchronisation.
 * They still pass sel, row_ptr, q_indices and d_status, exactly as for
 * msa_build_k2q; the build's scratch (document offsets, per-group counts and
 * row totals) lives in one array of MSA_NOALLOC_SCRATCH_BYTES that the library
 * holds on every GPU that loads it, until the process exits.
 *  - The scratch a problem needs is about 8 (N+1) + 4 Hi NB (G+1) bytes, with
 *    G = ceil(NC / S) scatter groups of S = max(64, ceil(NC / 128)) query
 *    chunks (so G <= 128); a problem needing more is rejected with
 *    MSA_ERR_SCRATCH_TOO_SMALL before anything is launched.  One document of
 *    131,072 tokens with 8 index heads needs about 8.5 MB.
 *  - The first call on a device looks up the array's device address (a
 *    runtime query made once per device, with that device current); make that
 *    first call before any stream capture begins.  The address is kept with
 *    the ID of the CUDA context it belongs to: after cudaDeviceReset (a new
 *    context, where the array may sit elsewhere) the next call looks it up
 *    again, and that call too should come before any capture.
 *  - Every call uses the same array and it keeps what the last call left
 *    there; the build overwrites all of it before reading, so nothing in it
 *    needs to start at zero.  Calls whose kernels overlap on the GPU (other
 *    streams, other host threads) race on the array and must be serialised by
 *    the caller.
 * It allocates nothing and returns the same codes as msa_build_k2q. */
#define MSA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int msa_build_k2q_noalloc(const msa_problem* p, const int32_t* sel, int32_t* row_ptr,
                          int32_t* q_indices, int64_t edge_cap, int32_t* d_status, void* stream);

/* Task rows and CTA walk of the KV-parallel backward ("msa_backward_sm100"
 * page, module docstring: task rows of 8 queries x 16 heads bucketed by
 * (batch, index_head, key_block); "msa_schedule" page, chunk_map,
 * rows_per_cta, grid_launch_bound).
 *
 * Each CSR row is cut into consecutive groups of query_chunk entries; a group
 * is one task (one query chunk against one key block).  Tasks are ordered by
 * index head, then query tile (global chunk / task_tile_chunks; 0 = a single
 * tile), then key-block row, then CSR offset.
 * task_meta   device int32 [task_cap, 6] out (MSA_TASK_META_COLS).
 * task_q_rows device int32 [task_cap, query_chunk] out: compact token row of
 *             each query slot, -1 past q_count.  Slots of one task are
 *             consecutive tokens of one chunk.
 * task_q_pos  device int32 [task_cap, query_chunk] out: document-local
 *             position of each slot, -1 past q_count.
 * walk        device int32 [MSA_WALK_LEN] out.
 * num_sms     SMs the walk is sized for; 0 = the current device's count.
 * Too many tasks for task_cap -> *d_status = MSA_ERR_CAPACITY.
 */
int msa_build_tasks(const msa_problem* p, const int32_t* row_ptr, const int32_t* q_indices,
                    int64_t edge_cap, int32_t task_tile_chunks, int32_t* task_meta,
                    int32_t* task_q_rows, int32_t* task_q_pos, int32_t* walk, int64_t task_cap,
                    int32_t num_sms, int32_t* d_status, void* ws, size_t ws_bytes, void* stream);

/* The backward pass ("msa_backward_sm100" page, run_backward): preprocess
 * D = rowsum(dO * O), the KV-parallel tcgen05 kernel over the task rows, and
 * the postprocess cast of the fp32 accumulators to bf16.
 *
 * q, o, dout  device bf16 [T, Hq, 128]; lse device fp32 [T, Hq] natural-log
 *             log-sum-exp of the forward.
 * k, v        device bf16 [W, Hkv, 128].
 * task_*      tables written by msa_build_tasks for this problem.
 * dq          device bf16 [T, Hq, 128] out.
 * dk, dv      device bf16 [W, Hkv, 128] out; rows outside every document 0.
 * ws          workspace of at least msa_workspace_bytes() bytes.
 */
int msa_bwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
            const uint16_t* o, const uint16_t* dout, const float* lse, const int32_t* task_meta,
            const int32_t* task_q_rows, const int32_t* task_q_pos, const int32_t* walk,
            int64_t task_cap, uint16_t* dq, uint16_t* dk, uint16_t* dv, int32_t* d_status,
            void* ws, size_t ws_bytes, void* stream);

/* msa_bwd split at its kernel boundaries, for callers that interleave their
 * own work or time the stages: stages is a mask of MSA_STAGE_* run in order
 * preprocess -> main -> postprocess on the stream.  msa_bwd is
 * stages = MSA_STAGE_ALL.  The stages communicate through ws, so a later
 * stage must see the same ws, tables and inputs as the earlier ones. */
enum { MSA_STAGE_PREPROCESS = 1, MSA_STAGE_MAIN = 2, MSA_STAGE_POSTPROCESS = 4, MSA_STAGE_ALL = 7 };
/* Option bit of the same mask: accumulate dQ in fp32.  By default each
 * task's fp32 dQ (over its 64 keys) is rounded to bf16 and reduce-added into
 * the bf16 dQ output, as the pages' bf16 dQ pool is ("msa_schedule" page,
 * the bf16x2 dQ pool; "msa_backward_sm100" page, dQ atomics), so a row of dQ
 * takes one bf16 rounding per task that feeds it.  With MSA_BWD_DQ_FP32 the
 * tasks reduce-add fp32 tiles into an fp32 buffer in ws (twice the reduce
 * traffic), which the postprocess rounds once to bf16.  ws must then hold
 * msa_workspace_bytes_opts(..., MSA_BWD_DQ_FP32) bytes, and every stage of
 * one backward must be called with the same option. */
enum { MSA_BWD_DQ_FP32 = 8 };
/* Self-test bit of the same mask (no counterpart in the pages; outputs are
 * not to be used): the main stage runs with its reduce warps idle, so the
 * hand-offs that wait for them (the task-info ring, the dQ buffers) run out
 * their 2 s bound, every role of the kernel aborts, in-flight copies are
 * waited for, and *d_status reads MSA_ERR_TIMEOUT.  The context stays usable.
 * Not combinable with MSA_BWD_DQ_FP32 (MSA_ERR_INVALID_ARGUMENT). */
enum { MSA_BWD_SELFTEST_HOLD_REDUCE = 16 };
int msa_bwd_staged(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const uint16_t* o, const uint16_t* dout, const float* lse, const int32_t* task_meta,
                   const int32_t* task_q_rows, const int32_t* task_q_pos, const int32_t* walk,
                   int64_t task_cap, uint16_t* dq, uint16_t* dk, uint16_t* dv, int32_t* d_status,
                   void* ws, size_t ws_bytes, void* stream, uint32_t stages);

/* The forward pass that produces O and LSE from the same selection
 * ("msa_bindings" page, sparse_atten_func, the flat forward): for each query
 * row, softmax(scale * q k^T) over the keys of its chunk's selected blocks
 * that precede or equal it, times V.  One pass with an online softmax; P is
 * rounded to bf16 for the P V product, everything else accumulates in fp32.
 * q     device bf16 [T, Hq, 128];  k, v device bf16 [W, Hkv, 128].
 * sel   device int32 [Hi, NC, K], as for msa_build_k2q (validated there,
 *       not here: call the forward with a selection the CSR build accepted).
 * o     device bf16 [T, Hq, 128] out;  lse device fp32 [T, Hq] out (natural
 *       log; -inf for a query that attends no key, whose O is 0).
 * ws    device workspace of at least 8 * (num_docs + 1) bytes rounded up to
 *       256 (msa_workspace_bytes() is always enough); caller-owned.
 * Returns MSA_ERR_INVALID_ARGUMENT for a null or misaligned pointer or a short
 * ws, MSA_ERR_CUDA if a launch fails; a device wait that exceeds its bound
 * writes MSA_ERR_TIMEOUT to *d_status.  Asynchronous on stream.
 */
int msa_fwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
            const int32_t* sel, uint16_t* o, float* lse, int32_t* d_status, void* ws,
            size_t ws_bytes, void* stream);

/* Block scorer and top-k selection: writes the sel array that msa_build_k2q
 * and msa_fwd consume ("msa_bindings" page, MSAKernels.fmha_sm100, the scorer
 * launcher; "msa_schedule" page, INDEX_DIM = 128 index dims per index head).
 * The pages name the scorer but not its score; this call computes:
 *  - per index head, the pooled index query of every query chunk and the
 *    pooled index key of every key block: the mean of the tokens' index
 *    vectors inside the document (fp32 sum in token order, divided by the
 *    token count, rounded to bf16);
 *  - score(chunk, block) = the fp32 dot product of the two pooled vectors,
 *    summed in ascending index-dim order;
 *  - sel[hi][g] = the chunk's diagonal block (the one holding its first
 *    query), then the topk - 1 blocks before it with the highest scores (a tie
 *    goes to the lower block) by descending score, then -1; every entry is a
 *    document-local block id and causal, so the result is a valid selection.
 * q_index, k_index  device bf16 [T, Hi, 128]: index query / key of each token
 *                   (compact token rows, the cu_seqlens order).
 * sel               device int32 [Hi, NC, topk] out.
 * ws                device workspace of at least msa_workspace_bytes() bytes
 *                   (it holds the pooled vectors).
 * Deterministic: the same inputs give the same sel on every run.  Returns
 * MSA_ERR_INVALID_ARGUMENT for a null or misaligned pointer or a short ws;
 * device-detected document errors go to *d_status.  Asynchronous on stream. */
int msa_select_topk(const msa_problem* p, const uint16_t* q_index, const uint16_t* k_index, int32_t* sel,
                    int32_t* d_status, void* ws, size_t ws_bytes, void* stream);

/* Forward work plan ("msa_bindings" page, MSAKernels.fmha_sm100_plan, the
 * planner launcher; "msa_schedule" page, MSABackwardSchedule's
 * scheduler_metadata and work_count): the forward's work items, built on the
 * device with no host synchronisation.
 * One item per (index head, query chunk), written as a scheduler_metadata row
 * in the pages' column order (MSA_TASK_META_COLS): index_head, row_linear =
 * the global query chunk, q_begin = its first token row, q_count = its token
 * count, document_ordinal, document_local_kblock = the key block holding its
 * first query.  Rows are ordered longest first: descending number of selected
 * blocks, ties in (index head, chunk) order, items selecting no block last, so
 * a persistent walk over them meets the long items first.
 * sel                 device int32 [Hi, NC, K], as for msa_fwd.
 * scheduler_metadata  device int32 [Hi * NC, 6] out: every item, once.
 * work_count          device int32 [1] out: items that select at least one
 *                     block (the rows before the empty ones).
 * ws                  workspace of at least msa_workspace_bytes() bytes.
 * Deterministic.  Asynchronous on stream; argument errors are return codes,
 * document errors go to *d_status. */
int msa_plan_forward(const msa_problem* p, const int32_t* sel, int32_t* scheduler_metadata,
                     int32_t* work_count, int32_t* d_status, void* ws, size_t ws_bytes, void* stream);

/* msa_fwd walking the items in the order of a plan written by
 * msa_plan_forward for the same problem and selection (the w-th item the
 * persistent CTAs take is row w of scheduler_metadata).  O and LSE are the
 * same, bit for bit, as msa_fwd's: every item is computed the same way
 * whichever CTA takes it. */
int msa_fwd_planned(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* sel, const int32_t* scheduler_metadata, uint16_t* o, float* lse,
                    int32_t* d_status, void* ws, size_t ws_bytes, void* stream);

/* Self-test of the bounded device waits (no counterpart in the pages).
 * Launches one small kernel that waits, with the same bounded mbarrier wait
 * every kernel of this library uses, for an mbarrier phase that nothing
 * completes.  After the wait limit (2 s) the kernel writes MSA_ERR_TIMEOUT to
 * *d_status (first error wins) and returns normally: no fault, no hang, and
 * the CUDA context stays usable.  d_status: device int32, caller-owned.
 * Returns MSA_ERR_INVALID_ARGUMENT for a null or misaligned d_status,
 * MSA_ERR_CUDA if the launch fails.  Asynchronous on stream. */
int msa_selftest_wait_timeout(int32_t* d_status, void* stream);

/* Host-side walk rule ("msa_schedule" page): rows_per_cta, chunk_map and
 * grid_launch_bound.  chunk_map writes (full, tail, grid) to out3. */
int32_t msa_rows_per_cta(int64_t num_rows);
void msa_chunk_map(int64_t num_rows, int32_t rows_per_cta, int32_t num_sms, int64_t* out3);
int64_t msa_grid_launch_bound(int64_t capacity, int32_t num_sms);

/* Memoised device queries ("kernels" page, sm_capability and sm_count: a
 * device's capability cannot change, so it is looked up once per device). */
int msa_device_capability(int32_t device, int32_t* major, int32_t* minor);
int msa_device_sm_count(int32_t device, int32_t* sm_count);

/* Static text for a status code. */
const char* msa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
