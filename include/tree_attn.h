/*
 * tree_attn.h -- C ABI of the GB300 (sm_103a) batched tree-attention library
 * (libtreeattn.so).
 *
 * The operation is the one the page "tree_attn.py"
 * (python/tvm/relax/frontend/nn/llm/tree_attn.py) generates as
 * ``batch_tree_attn`` (``tree_attn`` for GPUs, ``tree_attn_cpu`` for CPUs):
 * ragged, multi-sequence grouped-query attention in which q row r of
 * sequence b attends kv column c iff c lies in the sequence's causal prefix
 * or c's tree node is an ancestor-or-self of r's tree node, decided from the
 * DFS [enter, exit) intervals of ``_check_tree_order`` on that page.  RoPE
 * (``_rope`` on the page "_kernel_common.py",
 * python/tvm/relax/frontend/nn/llm/_kernel_common.py) is optionally applied
 * to q and k as they are loaded.  The outputs are the attention output and
 * the base-2 log-sum-exp (``m + log2(d)``, the ``lse_store`` epilogue).
 *
 * Conventions shared by every entry point:
 *   - Pointers named "device" are CUDA device pointers owned by the caller;
 *     the library never frees them and keeps no reference after returning.
 *   - ``stream`` is a ``cudaStream_t`` passed as ``void*`` (NULL = the
 *     legacy default stream).  Launching entry points are asynchronous on it
 *     and never synchronise the host.
 *   - Errors detectable from the arguments alone are returned synchronously
 *     before anything is launched.  The contents of device index arrays are
 *     not read on the host in the launching calls (see
 *     ``tree_attn_check_inputs``).
 *   - Only the current CUDA device is used.
 */
#ifndef TREE_ATTN_H_
#define TREE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TA_OK = 0,
  TA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, bad scalar         */
  TA_ERR_UNSUPPORTED = 2,      /* valid but not built: head_dim, group size  */
  TA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed          */
  TA_ERR_DEVICE_TIMEOUT = 4    /* a bounded device-side wait expired         */
} ta_status;

typedef enum { TA_FP16 = 0, TA_BF16 = 1 } ta_dtype;

/* Problem sizes.  The page's PrimFunc takes these from buffer shapes and
 * generator constants (h_kv, h_q, d, dtype); a C ABI passes them explicitly.
 *   batch_size  B, number of sequences (>= 1)
 *   total_q     rows of q / out / lse           (q_indptr[B])
 *   total_kv    rows of k / v                   (kv_indptr[B])
 *   total_tree  rows of tree_order              (mn_indptr[B])
 *   h_q, h_kv   heads; h_q % h_kv == 0, group size g = h_q / h_kv <= 128
 *   head_dim    64 or 128
 *   dtype       element type of q, k, v and out
 *   rotary_mode 0 or 1: whether the calls this workspace serves apply RoPE
 *               (it sizes the workspace; it must match their rotary_mode) */
typedef struct {
  int32_t batch_size;
  int32_t total_q;
  int32_t total_kv;
  int32_t total_tree;
  int32_t h_q;
  int32_t h_kv;
  int32_t head_dim;
  ta_dtype dtype;
  int32_t rotary_mode;
} ta_dims;

/* Bytes of device workspace ``tree_attn`` needs for these sizes (a multiple
 * of 256; 0 on invalid dims).  The workspace holds the per-launch work plan
 * (tile classes, the cost-ordered work queue), a device status word and,
 * with RoPE, the cos/sin table of the kv tokens and the rotated k
 * (total_kv * h_kv * head_dim elements, rotated once per call instead of
 * once per q tile that reads it), and when tree_attn splits the kv range
 * (tree_attn_auto_split_chunks > 1) the split-KV partial states, as
 * tree_attn_split_workspace_size(dims, that cap).  It depends on the dims and
 * the current device's SM count only, so one allocation serves every call
 * with the same dims on that kind of GPU. */
size_t tree_attn_workspace_size(const ta_dims* dims);

/* The split-KV chunk cap tree_attn uses for these dims on the current device
 * (0 on invalid dims).  1: no split.  tree_attn splits when the work units
 * (a unit is 2 q tiles of 128 / g rows of one sequence and kv head) number
 * fewer than the SMs even at their lower bound ceil(total_q / (256 / g)) x
 * h_kv, while the sequences average at least 2048 kv rows; the cap is then
 * ceil(4 x SMs / ((ceil(total_q / (256 / g)) + batch_size) x h_kv)) clamped
 * to 2..16 (about four work records per SM), and the plan picks the chunk
 * length (chunk_tiles 0 of tree_attn_split).  A split result equals the
 * unsplit one up to float32 rounding order (merge of base-2 LSE states). */
int32_t tree_attn_auto_split_chunks(const ta_dims* dims);

/* Batched tree attention.  Layouts (all row-major, contiguous, device):
 *   q               [total_q, h_q, head_dim]   dtype
 *   q_indptr        [B+1] int32, q rows of sequence b are
 *                   q_indptr[b] .. q_indptr[b+1]-1
 *   k, v            [total_kv, h_kv, head_dim] dtype
 *   kv_indptr       [B+1] int32, kv rows of sequence b
 *   q_rope_position [total_kv] int32, the RoPE position of every kv token;
 *                   q row r of sequence b takes the position of its own tree
 *                   node's kv slot.  May be NULL iff rotary_mode == 0.
 *   mn_indptr       [B+1] int32, tree nodes of sequence b are tree_order
 *                   rows mn_indptr[b] .. mn_indptr[b+1]-1
 *   tree_order      [total_tree][2] int32, (enter, exit) DFS interval of each
 *                   node, exit exclusive
 *   out             [total_q, h_q, head_dim] dtype   (written)
 *   lse             [total_q, h_q] float32, base-2 log-sum-exp (written);
 *                   natural-log LSE = lse * ln 2
 * For sequence b let qo = q rows, kv = kv rows, T = tree nodes; the last T kv
 * rows are the tree nodes in node order, the first kv - T the prefix, and the
 * q rows are the last qo tree nodes (0 <= qo <= T <= kv).  A q row none of
 * whose columns is visible gets out = 0 and lse = -inf.
 *   rotary_mode     0: no RoPE; 1: rotate-half RoPE on q and k at load time
 *                   (any other value, or one that differs from
 *                   dims->rotary_mode, is TA_ERR_INVALID_ARGUMENT)
 *   rope_scale      position multiplier (finite)
 *   rope_theta      RoPE base (finite, > 0)
 *   sm_scale        score scale (finite), typically 1/sqrt(head_dim)
 *   workspace       device buffer of >= tree_attn_workspace_size(dims) bytes,
 *                   256-byte aligned, zero-filled once before its first use
 *                   (e.g. cudaMemset); every call leaves it ready for the
 *                   next one.  Calls that may overlap on the GPU must use
 *                   distinct workspaces.
 * q, k, v and out must be 16-byte aligned.  Returns TA_OK once the work is
 * enqueued; device-side failures are reported by tree_attn_device_status.
 * When tree_attn_auto_split_chunks(dims) > 1 the call is tree_attn_split with
 * that cap and chunk_tiles 0 (plan, attention and merge kernels). */
ta_status tree_attn(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                    const int32_t* kv_indptr, const int32_t* q_rope_position,
                    const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                    float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                    float sm_scale, const ta_dims* dims, void* workspace,
                    size_t workspace_bytes, void* stream);

/* The two launches of unsplit tree_attn (these never split the kv range), for
 * callers that reuse one tree layout across calls (every layer of a model
 * verifies the same draft tree):
 *   tree_attn_plan  enumerates the (sequence, q tile) work items, classifies
 *                   every (q tile, kv tile) pair as empty / partial / full
 *                   from the DFS intervals and orders the items
 *                   longest-first; it reads only the index arrays (the RoPE
 *                   arguments are validated, not used).
 *   tree_attn_run   with rotary_mode == 1 the RoPE of every kv token (its
 *                   cos/sin from q_rope_position, rope_scale and rope_theta,
 *                   and its rotated keys), then the attention kernel proper,
 *                   consuming the plan that the last tree_attn_plan (or
 *                   tree_attn) left in ``workspace``.
 * tree_attn_run must follow a plan made on the same workspace with the same
 * dims, index-array contents, positions, rotary_mode, rope_scale and
 * rope_theta; q, k, v, out, lse and sm_scale may change between runs.
 * Arguments mean what they mean for tree_attn; both are asynchronous. */
ta_status tree_attn_plan(const int32_t* q_indptr, const int32_t* kv_indptr,
                         const int32_t* q_rope_position, const int32_t* mn_indptr,
                         const int32_t* tree_order, int32_t rotary_mode, float rope_scale,
                         float rope_theta, const ta_dims* dims, void* workspace,
                         size_t workspace_bytes, void* stream);

ta_status tree_attn_run(const void* q, const void* k, const void* v, const int32_t* q_indptr,
                        const int32_t* kv_indptr, const int32_t* q_rope_position,
                        const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                        float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                        float sm_scale, const ta_dims* dims, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Allocation-free variant of tree_attn (the pages have no counterpart: it is
 * a deployment convenience of this library).  Some callers cannot allocate
 * device memory: a serving engine that has handed all free HBM to its own
 * pool (typically the KV cache) and forbids further cudaMalloc, or a host
 * framework whose plugins may not call allocation routines because they
 * synchronise the device or escape the framework's memory accounting.  This
 * entry point takes the same arguments as tree_attn minus the workspace and
 * uses a static device array of 32 MiB (held by every GPU that loads the
 * library until the process exits) as its workspace; it calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - It never splits the kv range (tree_attn_split with max_chunks 1).
 *   - Problems whose unsplit workspace (tree_attn_split_workspace_size(dims,
 *     1)) exceeds 32 MiB are rejected
 *     with TA_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call clears the array's work counters (two cudaMemsetAsync on
 *     ``stream``) and then runs tree_attn on it.  All calls share the one
 *     array, so calls that may overlap on the GPU (different streams without
 *     ordering between them) race and must not be issued. */
ta_status tree_attn_noalloc(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                            const int32_t* kv_indptr, const int32_t* q_rope_position,
                            const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                            float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                            float sm_scale, const ta_dims* dims, void* stream);

/* Synchronises ``stream`` and reads and clears the device status word that
 * earlier tree_attn_noalloc calls on the current device left in the static
 * scratch array (the caller never sees that array's address): TA_OK,
 * TA_ERR_DEVICE_TIMEOUT if a bounded wait expired, TA_ERR_INVALID_ARGUMENT if
 * the index arrays broke the layout rules (nothing was computed), TA_ERR_CUDA
 * on a CUDA error.  Like tree_attn_device_status, but for the array. */
ta_status tree_attn_noalloc_device_status(void* stream);

/* ---- Paged KV cache ------------------------------------------------------
 * The same tree attention with K and V held in a paged cache, as the page
 * "tree_attn.py" generates it in ``tree_attn_with_paged_kv_cache`` (GPU) and
 * ``tree_attn_with_paged_kv_cache_cpu``; kv lengths follow
 * ``_get_kv_chunk_len`` of the page "_kernel_common.py" without a sliding
 * window (the pages disable it for tree attention).
 *   batch_size, total_q, total_tree, h_q, h_kv, head_dim, dtype
 *               as in ta_dims
 *   num_pages   pages in the pool (>= 1): the pages buffer is
 *               [num_pages, 2, h_kv, 16, head_dim]
 *   nnz_pages   entries of page_values (= page_indptr[B]) */
typedef struct {
  int32_t batch_size;
  int32_t total_q;
  int32_t total_tree;
  int32_t h_q;
  int32_t h_kv;
  int32_t head_dim;
  ta_dtype dtype;
  int32_t num_pages;
  int32_t nnz_pages;
} ta_paged_dims;

/* Bytes of device workspace tree_attn_paged needs (0 on invalid dims); the
 * same rules as tree_attn_workspace_size. */
size_t tree_attn_paged_workspace_size(const ta_paged_dims* dims);

/* Tree attention over a paged KV cache (one call: plan and run).  Layouts
 * (device, contiguous):
 *   q, out, lse, q_indptr, mn_indptr, tree_order   as for tree_attn
 *   pages        [num_pages, 2, h_kv, 16, head_dim] dtype: plane 0 holds K,
 *                plane 1 holds V, 16 kv slots per page
 *   page_indptr  [B+1] int32: sequence b owns page_values[page_indptr[b] ..
 *                page_indptr[b+1]-1], in kv order
 *   page_values  [nnz_pages] int32 physical page indices (an index outside
 *                [0, num_pages) reads zeros)
 *   length_info  [B] int32, the number of slots used in each sequence's last
 *                page (1..16 when the sequence owns a page); sequence b has
 *                kv = (pages - 1) * 16 + length_info[b] rows, 0 without pages
 * kv row r of sequence b is slot r % 16 of page page_values[page_indptr[b] +
 * r / 16]; the tree mask, the q rows and the outputs are those of tree_attn
 * with that kv length.  Slots past a sequence's kv length are never used (their
 * contents may be anything, NaN included).  The pages assert that this kernel
 * has no RoPE: rotary_mode must be 0 (else TA_ERR_UNSUPPORTED), and the pages'
 * position arguments (k_rope_pos_offset, q_rope_position) are therefore not
 * taken.  Inconsistent page tables (indptr not ending at nnz_pages, a
 * length_info outside 1..16) are reported by tree_attn_device_status and
 * nothing is computed.  q, pages and out must be 16-byte aligned; the
 * workspace follows tree_attn's rules.  Asynchronous on stream. */
ta_status tree_attn_paged(const void* q, const int32_t* q_indptr, const void* pages,
                          const int32_t* page_indptr, const int32_t* page_values,
                          const int32_t* length_info, const int32_t* mn_indptr,
                          const int32_t* tree_order, void* out, float* lse, int32_t rotary_mode,
                          float sm_scale, const ta_paged_dims* dims, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ---- Split-KV ------------------------------------------------------------
 * The same tree attention with the kv tiles of long (sequence, q tile) pairs
 * cut into chunks that run as separate work items, so that a batch of few
 * but long sequences (a long shared prefix before a small draft tree) still
 * covers every SM.  The pages have no split-KV; it rests on the base-2 LSE
 * their ``lse_store`` epilogue emits (page "tree_attn.py"), which is what
 * merges attention over disjoint kv sets: each chunk writes its float32
 * partial output O_i / l_i and lse_i to the workspace, and a merge kernel
 * forms lse = log2(sum_i 2^lse_i) and out = sum_i 2^(lse_i - lse) O_i / l_i.
 * Results equal tree_attn's up to float32 rounding order (not bit for bit).
 *
 * Bytes of device workspace tree_attn_split needs for these dims and chunk
 * cap: tree_attn_workspace_size's plus, per possible work record
 * (((total_q + R - 1) / R + batch_size) * max_chunks of them, R the q rows per
 * tile), an h_kv x 128 x head_dim float32 partial output and its lse.
 * 0 on invalid dims or max_chunks outside 1..16. */
size_t tree_attn_split_workspace_size(const ta_dims* dims, int32_t max_chunks);

/* tree_attn with split-KV (one call: plan, attention, merge).  Arguments as
 * for tree_attn, plus:
 *   max_chunks   1..16, the most chunks one (sequence, q tile) pair is cut
 *                into (1: no split, the result is then tree_attn's exactly)
 *   chunk_tiles  target chunk length in kv tiles of 128 columns (>= 0); a
 *                pair whose kv tiles up to its last row's own slot number c
 *                gets min(max_chunks, ceil(c / chunk_tiles)) chunks.  0 lets
 *                the plan choose it from the batch's total work: a quarter of
 *                one SM's share of it, at least 8.
 * The chunks of a pair split the range of its kv tiles up to its last
 * non-empty tile into equal lengths.  workspace must hold at least
 * tree_attn_split_workspace_size(dims, max_chunks) bytes, with tree_attn's
 * other rules.  Asynchronous on stream. */
ta_status tree_attn_split(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                          const int32_t* kv_indptr, const int32_t* q_rope_position,
                          const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                          float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                          float sm_scale, int32_t max_chunks, int32_t chunk_tiles,
                          const ta_dims* dims, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Merges n_parts attention states over disjoint kv sets of the same rows
 * into the state over their union, with the base-2 LSE rule above (parts of
 * lse = -inf contribute nothing; a row whose parts are all -inf gets out = 0
 * and lse = -inf).  Layouts (device, contiguous):
 *   parts  [n_parts, rows, head_dim] dtype, each part normalised (as
 *          tree_attn's out); rows = total_q * h_q for tree_attn outputs
 *   lses   [n_parts, rows] float32, base-2
 *   out    [rows, head_dim] dtype (written);  lse [rows] float32 (written)
 * head_dim 64 or 128 (else TA_ERR_UNSUPPORTED); parts and out 16-byte
 * aligned.  Asynchronous on stream. */
ta_status tree_attn_merge_states(const void* parts, const float* lses, int32_t n_parts,
                                 int64_t rows, int32_t head_dim, ta_dtype dtype, void* out,
                                 float* lse, void* stream);

/* Synchronises ``stream``, reads and clears the device status word that the
 * kernels of earlier calls left in ``workspace`` (TA_ERR_DEVICE_TIMEOUT if a
 * bounded wait expired, TA_ERR_CUDA on a CUDA error, else TA_OK). */
ta_status tree_attn_device_status(void* workspace, void* stream);

/* Test hooks for the failure detection of this library (the pages have no
 * counterpart; their only checks are compile-time asserts such as
 * ``check_thread_limits`` on the page "_kernel_common.py").  Every hand-off
 * between the warps of the attention kernel is an mbarrier wait bounded by a
 * wall-clock limit (2 s); when one runs out the kernel records
 * TA_ERR_DEVICE_TIMEOUT in the workspace status word, lets its in-flight
 * copies and tensor-core operations land, frees its tensor memory and
 * returns, and tree_attn_device_status reports it.  These hooks let a test
 * take that path on purpose, for the attention kernels launched by later
 * calls made on the calling host thread:
 *   wait_limit_ns  the limit of every bounded wait (0: the default 2 s)
 *   stall          1: the MMA thread of every pipeline first waits on a
 *                  barrier that nothing arrives on, so that this wait runs
 *                  out after wait_limit_ns and every other warp then gives up
 *                  its own waits; 0: normal operation
 * Returns TA_ERR_INVALID_ARGUMENT for stall outside {0, 1}.  Not for
 * production use: a stalled call computes nothing. */
ta_status tree_attn_set_wait_hooks(uint64_t wait_limit_ns, int32_t stall);

/* Work scheduling of the attention kernels launched by later calls on the
 * calling host thread (page "tile_scheduler.py", the persistent schedulers and
 * ``ClusterLaunchControlScheduler``):
 *   mode 0  one CTA per SM; CTA b takes the b-th work unit of the
 *           longest-first list, then units from an atomic counter in the
 *           workspace, one fetched ahead of use;
 *   mode 1  (default) one CTA per possible work unit; CTA b takes unit b, and when it
 *           starts a unit it asks the hardware (clusterlaunchcontrol.try_cancel)
 *           to cancel the launch of a CTA that has not started yet and then
 *           takes that CTA's unit; CTAs past the last unit are cancelled the
 *           same way so that they do not launch empty.
 * Both give the same results bit for bit; mode 1 measured equal or faster on
 * every benchmarked workload (spec-decode 31.6 -> 30.4 us).  Returns
 * TA_ERR_INVALID_ARGUMENT for any other mode. */
ta_status tree_attn_set_scheduler(int32_t mode);

/* The CUDA runtime's description of the error behind the calling thread's
 * most recent TA_ERR_CUDA ("no error" if there was none; static storage).
 * A failure that has no CUDA error of its own (no device, a tensor map the
 * driver rejects) reads as an invalid-value error. */
const char* tree_attn_last_cuda_error(void);

/* Human-readable name of a status code (static storage). */
const char* tree_attn_status_string(ta_status s);

/* Test helper: dense visibility of every (q row, kv column) pair, evaluated
 * by the same device mask code the attention kernel uses.  Writes
 * vis[total_q][max_kv] bytes (1 = visible) where column c of q row
 * q_indptr[b] + r is kv column c of sequence b; columns >= kv_len are 0.
 * Index arrays and vis are device pointers.  max_kv must be >= every
 * sequence's kv length.  Asynchronous on stream. */
ta_status tree_attn_mask_dense(const int32_t* q_indptr, const int32_t* kv_indptr,
                               const int32_t* mn_indptr, const int32_t* tree_order,
                               int32_t batch_size, int32_t total_q, int32_t max_kv,
                               uint8_t* vis, void* stream);

/* Host-side validation of HOST copies of the index arrays, for callers and
 * tests: indptr arrays start at 0, are non-decreasing and end at the dims'
 * totals; per sequence 0 <= qo <= T <= kv; every interval has
 * 0 <= enter < exit <= T and the intervals of a sequence nest (any two are
 * disjoint or one contains the other).  ``q_rope_position`` is accepted for
 * symmetry with tree_attn and not inspected (every int32 position is valid).
 * Returns TA_OK or TA_ERR_INVALID_ARGUMENT. */
ta_status tree_attn_check_inputs(const int32_t* q_indptr, const int32_t* kv_indptr,
                                 const int32_t* mn_indptr, const int32_t* tree_order,
                                 const int32_t* q_rope_position, const ta_dims* dims);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H_ */
