// ta_api.cu -- host side of the C ABI declared in include/tree_attn.h:
// argument validation, workspace layout, TMA tensor-map encoding and the two
// launches (plan kernel, persistent attention kernel) of one tree_attn call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/tree_attn.h"
#include "ta_launch.h"

using ta::WsHeader;
using ta::WsLayout;

namespace {

constexpr unsigned long long kDeviceWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// The CUDA error behind this thread's last TA_ERR_CUDA (cudaSuccess if none).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Test hooks of the calling thread (tree_attn_set_wait_hooks): the bounded
// wait limit of the attention kernels it launches (0: kDeviceWaitLimitNs) and
// whether their MMA threads first wait on a barrier that nothing arrives on.
thread_local unsigned long long g_wait_limit_ns = 0;
thread_local int g_stall = 0;

unsigned long long wait_limit_ns() { return g_wait_limit_ns ? g_wait_limit_ns : kDeviceWaitLimitNs; }

// Work scheduling of the attention kernels the calling thread launches
// (tree_attn_set_scheduler): 0 the atomic work queue over one CTA per SM,
// 1 (default) cluster launch control over one CTA per work unit.
thread_local int g_sched = 1;

// Attention grid: one CTA per SM (atomic queue), or one per possible work
// unit (cluster launch control: the CTAs that run take the units of those
// that have not started yet).
int attn_grid(int64_t max_items, int nsm) {
  if (g_sched == 1) return (int)max_items;
  return (int)(max_items < nsm ? max_items : nsm);
}

// TA_ERR_CUDA for a failed CUDA call, remembering its error; TA_OK otherwise.
ta_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TA_OK;
  g_last_cuda_error = e;
  return TA_ERR_CUDA;
}

// TA_ERR_CUDA for a failed step with no CUDA error of its own (a tensor map
// the driver rejects, no device), recorded as an invalid value.
ta_status cuda_failure() { return cuda_status(cudaErrorInvalidValue); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool dims_valid(const ta_dims* d) {
  if (!d) return false;
  if (d->batch_size < 1 || d->total_q < 0 || d->total_kv < 0 || d->total_tree < 0) return false;
  if (d->h_q < 1 || d->h_kv < 1 || d->h_q % d->h_kv != 0) return false;
  if (d->dtype != TA_FP16 && d->dtype != TA_BF16) return false;
  if (d->head_dim < 1) return false;
  if (d->rotary_mode != 0 && d->rotary_mode != 1) return false;
  return true;
}

ta_status dims_supported(const ta_dims* d) {
  if (d->head_dim != 64 && d->head_dim != 128) return TA_ERR_UNSUPPORTED;
  if (d->h_q / d->h_kv > ta::kMaxGroup) return TA_ERR_UNSUPPORTED;
  return TA_OK;
}

WsLayout layout_of(const ta_dims* d, int max_chunks = 1) {
  return ta::make_ws_layout(d->batch_size, d->total_q, d->total_kv, d->h_q / d->h_kv, d->h_kv,
                            d->head_dim, d->rotary_mode != 0, max_chunks);
}

// Workspace bytes for dims and a split-KV chunk cap (1: unsplit); 0 when the
// dims are invalid or unsupported or a table index would overflow int32.
size_t ws_size(const ta_dims* d, int max_chunks) {
  if (!dims_valid(d) || dims_supported(d) != TA_OK) return 0;
  if (max_chunks < 1 || max_chunks > ta::kMaxChunks) return 0;
  const WsLayout L = layout_of(d, max_chunks);
  if (L.class_bytes >= (int64_t)INT32_MAX || L.max_records * d->h_kv >= (int64_t)INT32_MAX)
    return 0;
  return L.total;
}

// Split-KV chunk cap of the one-call entry point for dims on a GPU of nsm
// SMs.  1 (no split) unless the (sequence, unit) pairs times the kv heads
// leave SMs without work while the sequences are long on average (at least
// two chunks of the least automatic length each); then enough chunks for
// about four work records per SM, 2 .. kMaxChunks.  The pair count is taken
// from its lower bound ceil(total_q / U) and the workspace from its upper
// bound (one more pair per sequence), so the choice depends on dims alone.
int auto_max_chunks(const ta_dims* d, int nsm) {
  if (!dims_valid(d) || nsm <= 0 || d->total_q == 0) return 1;
  const int64_t U = ta::rows_per_unit(d->h_q / d->h_kv);
  const int64_t pairs_lo = ta::ceil_div(d->total_q, U);
  if (pairs_lo * d->h_kv >= nsm) return 1;
  const int64_t long_kv = (int64_t)d->batch_size * 2 * ta::kMinChunkTiles * ta::kBlockN;
  if ((int64_t)d->total_kv < long_kv) return 1;
  const int64_t pairs_hi = pairs_lo + d->batch_size;
  const int64_t c = ta::ceil_div(4LL * nsm, pairs_hi * d->h_kv);
  return (int)std::min<int64_t>(ta::kMaxChunks, std::max<int64_t>(2, c));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D tensor map over [rows, heads, d] (d fastest) with a {64, box_heads,
// box_rows} box and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, ta_dtype dt, int rows, int heads, int d,
              int box_heads, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t gstride[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUtensorMapDataType t =
      dt == TA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(m, t, 3, const_cast<void*>(base), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D tensor map over the paged cache [pages, 2, h_kv, 16, d] (d fastest)
// with a {64, 16, 1, 1, 1} box (one page's 16 slots of one column block) and
// 128-byte swizzle; an out-of-range page index reads zeros.
bool make_pages_map(CUtensorMap* m, const void* base, ta_dtype dt, int num_pages, int h_kv,
                    int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[5] = {(cuuint64_t)d, (cuuint64_t)ta::kPageSize, (cuuint64_t)h_kv, 2,
                              (cuuint64_t)num_pages};
  const cuuint64_t row = (cuuint64_t)d * 2;
  const cuuint64_t gstride[4] = {row, row * ta::kPageSize, row * ta::kPageSize * h_kv,
                                 row * ta::kPageSize * h_kv * 2};
  const cuuint32_t box[5] = {64u, (cuuint32_t)ta::kPageSize, 1u, 1u, 1u};
  const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
  const CUtensorMapDataType t =
      dt == TA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(m, t, 5, const_cast<void*>(base), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

size_t tree_attn_workspace_size(const ta_dims* dims) {
  return ws_size(dims, auto_max_chunks(dims, sm_count()));
}

int32_t tree_attn_auto_split_chunks(const ta_dims* dims) {
  if (!dims_valid(dims)) return 0;
  return auto_max_chunks(dims, sm_count());
}

size_t tree_attn_split_workspace_size(const ta_dims* dims, int32_t max_chunks) {
  return ws_size(dims, max_chunks);
}

}  // extern "C"

namespace {

// Checks shared by the plan and run halves.
ta_status check_common(const int32_t* q_indptr, const int32_t* kv_indptr,
                       const int32_t* mn_indptr, const int32_t* tree_order, int32_t rotary_mode,
                       const ta_dims* dims, const void* workspace, size_t workspace_bytes,
                       int max_chunks = 1) {
  if (!dims_valid(dims)) return TA_ERR_INVALID_ARGUMENT;
  if (max_chunks < 1 || max_chunks > ta::kMaxChunks) return TA_ERR_INVALID_ARGUMENT;
  const ta_status sup = dims_supported(dims);
  if (sup != TA_OK) return sup;
  if (!q_indptr || !kv_indptr || !mn_indptr || !workspace) return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_tree > 0 && !tree_order) return TA_ERR_INVALID_ARGUMENT;
  if (rotary_mode != 0 && rotary_mode != 1) return TA_ERR_INVALID_ARGUMENT;
  if (rotary_mode != dims->rotary_mode) return TA_ERR_INVALID_ARGUMENT;
  if (!aligned(workspace, 256)) return TA_ERR_INVALID_ARGUMENT;
  const size_t need = ws_size(dims, max_chunks);
  if (need == 0) return TA_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_q > 0 && dims->total_kv == 0) return TA_ERR_INVALID_ARGUMENT;  // qo <= T <= kv
  return TA_OK;
}

ta_status check_plan_args(const int32_t* q_rope_position, int32_t rotary_mode, float rope_scale,
                          float rope_theta, const ta_dims* dims) {
  if (rotary_mode == 1 && !q_rope_position && dims->total_kv > 0) return TA_ERR_INVALID_ARGUMENT;
  if (rotary_mode == 1 && (!std::isfinite(rope_scale) || !std::isfinite(rope_theta) ||
                           !(rope_theta > 0.f)))
    return TA_ERR_INVALID_ARGUMENT;
  return TA_OK;
}

ta_status check_run_args(const void* q, const void* k, const void* v, const void* out,
                         const float* lse, float sm_scale, const ta_dims* dims) {
  if (dims->total_q > 0 && (!q || !out || !lse)) return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_kv > 0 && (!k || !v)) return TA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return TA_ERR_INVALID_ARGUMENT;
  if ((q && !aligned(q, 16)) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
      (out && !aligned(out, 16)))
    return TA_ERR_INVALID_ARGUMENT;
  return TA_OK;
}

struct WsPtrs {
  WsHeader* hdr;
  ta::ItemRec* sorted;
  uint8_t* classes;
  float2* rope_cs;
  int4* merge;        // split-KV only
  float* part_o;
  float* part_lse;
};

WsPtrs ws_ptrs(void* workspace, const WsLayout& L) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool split = L.max_records > L.max_pairs;
  return WsPtrs{reinterpret_cast<WsHeader*>(ws),
                reinterpret_cast<ta::ItemRec*>(ws + L.off_sorted),
                ws + L.off_classes,
                reinterpret_cast<float2*>(ws + L.off_rope),
                split ? reinterpret_cast<int4*>(ws + L.off_merge) : nullptr,
                split ? reinterpret_cast<float*>(ws + L.off_part_o) : nullptr,
                split ? reinterpret_cast<float*>(ws + L.off_part_lse) : nullptr};
}

// fl32(theta^(2i/d)) for i < d/2, the RoPE frequency denominators of
// ``_rope`` (page "_kernel_common.py"), rounded once from float64; 1 past d/2
void rope_denominators(float rope_theta, int head_dim, float* den) {
  for (int i = 0; i < 64; ++i) den[i] = 1.f;
  const double l2 = std::log2((double)rope_theta);
  for (int i = 0; i < head_dim / 2; ++i)
    den[i] = (float)std::exp2(l2 * ((2.0 * i) / (double)head_dim));
}

// The key rotation of a call with RoPE: K, positions and RoPE constants.
struct RopeArgs {
  const void* k;
  const int32_t* pos;
  float scale, theta;
};

ta::KrotParams krot_params(const ta_dims* dims, const RopeArgs& ra) {
  ta::KrotParams kp{};
  rope_denominators(ra.theta, dims->head_dim, kp.rope_den);
  kp.rope_scale = ra.scale;
  kp.total_kv = dims->total_kv;
  kp.h_kv = dims->h_kv;
  return kp;
}

// Whether a one-call entry point folds the key rotation into the plan
// kernel: when the rotation is a short latency tail (at most 64 kv tokens
// per SM, about two per rotating warp) that the plan's idle warps absorb;
// a larger rotation runs as its own kernel, which measured faster.
bool fold_rotation(const ta_dims* dims, int nsm) {
  return dims->rotary_mode == 1 && (int64_t)dims->total_kv <= 64LL * nsm;
}

// The plan kernel (work records, tile classes, longest-first order).  With
// ``rope`` it also does the run's key rotation on its idle warps, over a
// grid of at least 2 CTAs per SM (measured against 1 and 4 on spec-decode).
ta_status launch_plan_checked(const int32_t* q_indptr, const int32_t* kv_indptr,
                              const int32_t* mn_indptr, const int32_t* tree_order,
                              const ta_dims* dims, void* workspace, cudaStream_t st,
                              int max_chunks = 1, int chunk_tiles = 0,
                              const RopeArgs* rope = nullptr) {
  const int g = dims->h_q / dims->h_kv;
  const WsLayout L = layout_of(dims, max_chunks);
  const WsPtrs w = ws_ptrs(workspace, L);
  const int nsm = sm_count();
  if (nsm <= 0) return cuda_failure();
  ta::PlanParams pp{};
  pp.q_indptr = q_indptr;
  pp.kv_indptr = kv_indptr;
  pp.mn_indptr = mn_indptr;
  pp.tree_order = tree_order;
  pp.batch = dims->batch_size;
  pp.g = g;
  pp.R = ta::rows_per_item(g);
  pp.h_kv = dims->h_kv;
  pp.head_dim = dims->head_dim;
  pp.total_q = dims->total_q;
  pp.total_kv = dims->total_kv;
  pp.total_tree = dims->total_tree;
  pp.max_pairs = L.max_pairs;
  pp.max_chunks = max_chunks;
  pp.chunk_tiles = chunk_tiles;
  pp.pipes = nsm;   // one attention pipeline per SM
  pp.merge = w.merge;
  pp.hdr = w.hdr;
  pp.sorted = w.sorted;
  pp.classes = w.classes;
  int grid = (int)L.max_pairs;
  if (rope != nullptr && dims->total_kv > 0) {
    pp.rot = 1 + 2 * (dims->head_dim == 128) + (dims->dtype == TA_BF16);
    pp.rot_k = static_cast<const uint32_t*>(rope->k);
    pp.rot_out = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + L.off_krot);
    pp.rot_pos = rope->pos;
    pp.rot_cs = reinterpret_cast<float4*>(w.rope_cs);
    pp.kp = krot_params(dims, *rope);
    if (grid < 2 * nsm) grid = 2 * nsm;
  }
  return cuda_status(ta::launch_plan(pp, grid, st));
}

ta_status launch_run_checked(const void* q, const void* k, const void* v, const int32_t* q_indptr,
                             const int32_t* kv_indptr, const int32_t* q_rope_position,
                             const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                             float* lse, int32_t rotary_mode, float rope_scale,
                             float rope_theta, float sm_scale, const ta_dims* dims,
                             void* workspace, cudaStream_t st, int max_chunks = 1,
                             bool keys_rotated = false) {
  // the index arrays reach the kernels through the plan's records
  (void)q_indptr;
  (void)kv_indptr;
  (void)mn_indptr;
  const int g = dims->h_q / dims->h_kv;
  const int R = ta::rows_per_item(g);
  const int D = dims->head_dim;
  const WsLayout L = layout_of(dims, max_chunks);
  const WsPtrs w = ws_ptrs(workspace, L);
  const int nsm = sm_count();
  if (nsm <= 0) return cuda_failure();
  // with RoPE the keys are rotated once per call (every q tile of a sequence
  // reads them) -- by the plan kernel of a one-call entry point, else here --
  // and the attention kernel loads the rotated copy
  const void* k_attn = k;
  if (rotary_mode == 1) {
    void* krot = static_cast<uint8_t*>(workspace) + L.off_krot;
    if (!keys_rotated) {
      const ta::KrotParams kp =
          krot_params(dims, RopeArgs{k, q_rope_position, rope_scale, rope_theta});
      // one resident wave at most (8 warps per CTA, one token per warp at a time)
      const int64_t want = ((int64_t)dims->total_kv + 7) / 8;
      const int kgrid = (int)(want < 4 * nsm ? want : 4 * nsm);
      const cudaError_t ke = ta::launch_krot(k, krot, q_rope_position, w.rope_cs, kp, D,
                                             dims->dtype == TA_BF16, kgrid, st);
      if (ke != cudaSuccess) return cuda_status(ke);
    }
    k_attn = krot;
  }
  CUtensorMap tm_q, tm_k, tm_v;
  if (!make_map(&tm_q, q, dims->dtype, dims->total_q, dims->h_q, D, g, R) ||
      !make_map(&tm_k, k_attn, dims->dtype, dims->total_kv, dims->h_kv, D, 1, ta::kKvBoxRows) ||
      !make_map(&tm_v, v, dims->dtype, dims->total_kv, dims->h_kv, D, 1, ta::kKvBoxRows))
    return cuda_failure();
  ta::AttnParams ap{};
  ap.tree_order = tree_order;
  ap.out = out;
  ap.lse = lse;
  ap.sorted = w.sorted;
  ap.classes = w.classes;
  ap.rope_cs = w.rope_cs;
  ap.hdr = w.hdr;
  ap.h_q = dims->h_q;
  ap.h_kv = dims->h_kv;
  ap.g = g;
  ap.R = R;
  ap.rotary = rotary_mode;
  ap.max_records = L.max_records;
  ap.scale_log2 = sm_scale * 1.4426950408889634f;
  ap.timeout_ns = wait_limit_ns();
  ap.debug_stall = g_stall;
  ap.sched_clc = g_sched;
  ap.part_o = w.part_o;
  ap.part_lse = w.part_lse;
  const int64_t max_items = L.max_records * dims->h_kv;
  const int grid = attn_grid(max_items, nsm);
  cudaError_t e;
  const bool bf16 = dims->dtype == TA_BF16;
  if (D == 64)
    e = bf16 ? ta::launch_attn<64, true, false>(tm_q, tm_k, tm_v, ap, grid, st)
             : ta::launch_attn<64, false, false>(tm_q, tm_k, tm_v, ap, grid, st);
  else
    e = bf16 ? ta::launch_attn<128, true, false>(tm_q, tm_k, tm_v, ap, grid, st)
             : ta::launch_attn<128, false, false>(tm_q, tm_k, tm_v, ap, grid, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (max_chunks > 1) {
    // split-KV: the chunks' partial states of every split pair into out / lse
    ta::MergeParams mp{};
    mp.merge = w.merge;
    mp.part_o = w.part_o;
    mp.part_lse = w.part_lse;
    mp.out = out;
    mp.lse = lse;
    mp.hdr = w.hdr;
    mp.max_pairs = L.max_pairs;
    mp.max_records = L.max_records;
    mp.h_q = dims->h_q;
    mp.h_kv = dims->h_kv;
    mp.g = g;
    const int64_t units =
        L.max_pairs * dims->h_kv * (ta::kTilesPerUnit * ta::kBlockM / 8);   // 8 rows each
    const int mgrid = (int)(units < 16 * nsm ? units : 16 * nsm);
    const cudaError_t me = ta::launch_merge(mp, D, bf16, mgrid, st);
    if (me != cudaSuccess) return cuda_status(me);
  }
  return TA_OK;
}

}  // namespace

extern "C" {

ta_status tree_attn_plan(const int32_t* q_indptr, const int32_t* kv_indptr,
                         const int32_t* q_rope_position, const int32_t* mn_indptr,
                         const int32_t* tree_order, int32_t rotary_mode, float rope_scale,
                         float rope_theta, const ta_dims* dims, void* workspace,
                         size_t workspace_bytes, void* stream) {
  ta_status s = check_common(q_indptr, kv_indptr, mn_indptr, tree_order, rotary_mode, dims,
                             workspace, workspace_bytes);
  if (s != TA_OK) return s;
  s = check_plan_args(q_rope_position, rotary_mode, rope_scale, rope_theta, dims);
  if (s != TA_OK) return s;
  if (dims->total_q == 0) return TA_OK;
  return launch_plan_checked(q_indptr, kv_indptr, mn_indptr, tree_order, dims, workspace,
                             static_cast<cudaStream_t>(stream));
}

ta_status tree_attn_run(const void* q, const void* k, const void* v, const int32_t* q_indptr,
                        const int32_t* kv_indptr, const int32_t* q_rope_position,
                        const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                        float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                        float sm_scale, const ta_dims* dims, void* workspace,
                        size_t workspace_bytes, void* stream) {
  ta_status s = check_common(q_indptr, kv_indptr, mn_indptr, tree_order, rotary_mode, dims,
                             workspace, workspace_bytes);
  if (s != TA_OK) return s;
  s = check_plan_args(q_rope_position, rotary_mode, rope_scale, rope_theta, dims);
  if (s != TA_OK) return s;
  s = check_run_args(q, k, v, out, lse, sm_scale, dims);
  if (s != TA_OK) return s;
  if (dims->total_q == 0) return TA_OK;
  return launch_run_checked(q, k, v, q_indptr, kv_indptr, q_rope_position, mn_indptr, tree_order,
                            out, lse, rotary_mode, rope_scale, rope_theta, sm_scale, dims,
                            workspace, static_cast<cudaStream_t>(stream));
}

ta_status tree_attn(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                    const int32_t* kv_indptr, const int32_t* q_rope_position,
                    const int32_t* mn_indptr, const int32_t* tree_order, void* out, float* lse,
                    int32_t rotary_mode, float rope_scale, float rope_theta, float sm_scale,
                    const ta_dims* dims, void* workspace, size_t workspace_bytes, void* stream) {
  // few, long sequences go through split-KV (the plan picks the chunk length)
  const int max_chunks = dims_valid(dims) ? auto_max_chunks(dims, sm_count()) : 1;
  return tree_attn_split(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order,
                         out, lse, rotary_mode, rope_scale, rope_theta, sm_scale, max_chunks, 0,
                         dims, workspace, workspace_bytes, stream);
}

ta_status tree_attn_split(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                          const int32_t* kv_indptr, const int32_t* q_rope_position,
                          const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                          float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                          float sm_scale, int32_t max_chunks, int32_t chunk_tiles,
                          const ta_dims* dims, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (chunk_tiles < 0) return TA_ERR_INVALID_ARGUMENT;
  ta_status s = check_common(q_indptr, kv_indptr, mn_indptr, tree_order, rotary_mode, dims,
                             workspace, workspace_bytes, max_chunks);
  if (s != TA_OK) return s;
  s = check_plan_args(q_rope_position, rotary_mode, rope_scale, rope_theta, dims);
  if (s != TA_OK) return s;
  s = check_run_args(q, k, v, out, lse, sm_scale, dims);
  if (s != TA_OK) return s;
  if (dims->total_q == 0) return TA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RopeArgs ra{k, q_rope_position, rope_scale, rope_theta};
  const bool rot = fold_rotation(dims, sm_count());
  s = launch_plan_checked(q_indptr, kv_indptr, mn_indptr, tree_order, dims, workspace, st,
                          max_chunks, chunk_tiles, rot ? &ra : nullptr);
  if (s != TA_OK) return s;
  return launch_run_checked(q, k, v, q_indptr, kv_indptr, q_rope_position, mn_indptr,
                            tree_order, out, lse, rotary_mode, rope_scale, rope_theta,
                            sm_scale, dims, workspace, st, max_chunks, rot);
}

ta_status tree_attn_merge_states(const void* parts, const float* lses, int32_t n_parts,
                                 int64_t rows, int32_t head_dim, ta_dtype dtype, void* out,
                                 float* lse, void* stream) {
  if (n_parts < 1 || rows < 0) return TA_ERR_INVALID_ARGUMENT;
  if (dtype != TA_FP16 && dtype != TA_BF16) return TA_ERR_INVALID_ARGUMENT;
  if (head_dim < 1) return TA_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return TA_ERR_UNSUPPORTED;
  if (rows == 0) return TA_OK;
  if (!parts || !lses || !out || !lse) return TA_ERR_INVALID_ARGUMENT;
  if (!aligned(parts, 16) || !aligned(out, 16)) return TA_ERR_INVALID_ARGUMENT;
  const int nsm = sm_count();
  if (nsm <= 0) return cuda_failure();
  const int64_t ctas = (rows + 7) / 8;   // 8 rows (warps) per CTA
  const int grid = (int)(ctas < 8 * nsm ? ctas : 8 * nsm);
  const cudaError_t e =
      ta::launch_merge_states(parts, lses, n_parts, (long long)rows, head_dim, dtype == TA_BF16,
                              out, lse, grid, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

ta_status tree_attn_device_status(void* workspace, void* stream) {
  if (!workspace) return TA_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  unsigned int err = 0;
  e = cudaMemcpy(&err, &hdr->error, sizeof(err), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (err != 0) {
    e = cudaMemset(&hdr->error, 0, sizeof(err));
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (err & ta::DEVERR_TIMEOUT) return TA_ERR_DEVICE_TIMEOUT;
  if (err & ta::DEVERR_BAD_INDPTR) return TA_ERR_INVALID_ARGUMENT;
  return TA_OK;
}

const char* tree_attn_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

ta_status tree_attn_set_wait_hooks(uint64_t wait_limit_ns, int32_t stall) {
  if (stall != 0 && stall != 1) return TA_ERR_INVALID_ARGUMENT;
  g_wait_limit_ns = wait_limit_ns;
  g_stall = stall;
  return TA_OK;
}

ta_status tree_attn_set_scheduler(int32_t mode) {
  if (mode != 0 && mode != 1) return TA_ERR_INVALID_ARGUMENT;
  g_sched = mode;
  return TA_OK;
}

const char* tree_attn_status_string(ta_status s) {
  switch (s) {
    case TA_OK: return "TA_OK";
    case TA_ERR_INVALID_ARGUMENT: return "TA_ERR_INVALID_ARGUMENT";
    case TA_ERR_UNSUPPORTED: return "TA_ERR_UNSUPPORTED";
    case TA_ERR_CUDA: return "TA_ERR_CUDA";
    case TA_ERR_DEVICE_TIMEOUT: return "TA_ERR_DEVICE_TIMEOUT";
  }
  return "TA_ERR_UNKNOWN";
}

ta_status tree_attn_mask_dense(const int32_t* q_indptr, const int32_t* kv_indptr,
                               const int32_t* mn_indptr, const int32_t* tree_order,
                               int32_t batch_size, int32_t total_q, int32_t max_kv, uint8_t* vis,
                               void* stream) {
  if (!q_indptr || !kv_indptr || !mn_indptr || !tree_order || !vis) return TA_ERR_INVALID_ARGUMENT;
  if (batch_size < 1 || total_q < 0 || max_kv < 0) return TA_ERR_INVALID_ARGUMENT;
  if (total_q == 0 || max_kv == 0) return TA_OK;
  const cudaError_t e = ta::launch_mask_dense(q_indptr, kv_indptr, mn_indptr, tree_order,
                                              batch_size, total_q, max_kv, vis,
                                              static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

ta_status tree_attn_check_inputs(const int32_t* q_indptr, const int32_t* kv_indptr,
                                 const int32_t* mn_indptr, const int32_t* tree_order,
                                 const int32_t* q_rope_position, const ta_dims* dims) {
  (void)q_rope_position;
  if (!dims_valid(dims) || !q_indptr || !kv_indptr || !mn_indptr) return TA_ERR_INVALID_ARGUMENT;
  const int B = dims->batch_size;
  if (q_indptr[0] != 0 || kv_indptr[0] != 0 || mn_indptr[0] != 0) return TA_ERR_INVALID_ARGUMENT;
  if (q_indptr[B] != dims->total_q || kv_indptr[B] != dims->total_kv ||
      mn_indptr[B] != dims->total_tree)
    return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_tree > 0 && !tree_order) return TA_ERR_INVALID_ARGUMENT;
  std::vector<int> stack;
  for (int b = 0; b < B; ++b) {
    const int qo = q_indptr[b + 1] - q_indptr[b];
    const int kv = kv_indptr[b + 1] - kv_indptr[b];
    const int T = mn_indptr[b + 1] - mn_indptr[b];
    if (qo < 0 || T < qo || kv < T) return TA_ERR_INVALID_ARGUMENT;
    // intervals: 0 <= enter < exit <= T and laminar (sort by enter, check nesting)
    std::vector<std::pair<int, int>> iv(T);
    for (int i = 0; i < T; ++i) {
      const int e = tree_order[2 * (mn_indptr[b] + i)], x = tree_order[2 * (mn_indptr[b] + i) + 1];
      if (e < 0 || x <= e || x > T) return TA_ERR_INVALID_ARGUMENT;
      iv[i] = {e, -x};
    }
    std::sort(iv.begin(), iv.end());
    stack.clear();
    for (const auto& pr : iv) {
      const int e = pr.first, x = -pr.second;
      while (!stack.empty() && stack.back() <= e) stack.pop_back();
      if (!stack.empty() && x > stack.back()) return TA_ERR_INVALID_ARGUMENT;  // overlaps
      stack.push_back(x);
    }
  }
  return TA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point: tree_attn with its workspace in a static
// device array instead of caller memory.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB on every device

// Zero-initialised with the module; each GPU that loads the library holds one
// copy until the process exits.  In host code this name is only a stand-in
// for the symbol: the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this set-up).  The cached
// address belongs to the device's primary context: it does not survive a
// cudaDeviceReset of that device.
void* noalloc_scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

ta_status tree_attn_noalloc(const void* q, const int32_t* q_indptr, const void* k, const void* v,
                            const int32_t* kv_indptr, const int32_t* q_rope_position,
                            const int32_t* mn_indptr, const int32_t* tree_order, void* out,
                            float* lse, int32_t rotary_mode, float rope_scale, float rope_theta,
                            float sm_scale, const ta_dims* dims, void* stream) {
  if (!dims_valid(dims)) return TA_ERR_INVALID_ARGUMENT;
  const size_t need = ws_size(dims, 1);   // never split: the scratch stays small
  if (need == 0) return dims_supported(dims) != TA_OK ? TA_ERR_UNSUPPORTED : TA_ERR_INVALID_ARGUMENT;
  if (need > kNoAllocScratchBytes) return TA_ERR_UNSUPPORTED;  // problem too large for the scratch
  void* ws = noalloc_scratch_address();
  if (ws == nullptr) return cuda_failure();
  // the work-queue and plan counters must start at zero (the status word at
  // offset 8 is left as it is)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* hdr = static_cast<uint8_t*>(ws);
  cudaError_t e = cudaMemsetAsync(hdr, 0, 8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(hdr + 12, 0, sizeof(WsHeader) - 12, st);
  if (e != cudaSuccess) return cuda_status(e);
  return tree_attn_split(q, q_indptr, k, v, kv_indptr, q_rope_position, mn_indptr, tree_order,
                         out, lse, rotary_mode, rope_scale, rope_theta, sm_scale, 1, 0, dims, ws,
                         kNoAllocScratchBytes, stream);
}

ta_status tree_attn_noalloc_device_status(void* stream) {
  void* ws = noalloc_scratch_address();
  if (ws == nullptr) return cuda_failure();
  return tree_attn_device_status(ws, stream);
}

}  // extern "C"


// ---------------------------------------------------------------------------
// paged KV cache
// ---------------------------------------------------------------------------
namespace {

bool paged_dims_valid(const ta_paged_dims* d) {
  if (!d) return false;
  if (d->batch_size < 1 || d->total_q < 0 || d->total_tree < 0) return false;
  if (d->h_q < 1 || d->h_kv < 1 || d->h_q % d->h_kv != 0) return false;
  if (d->dtype != TA_FP16 && d->dtype != TA_BF16) return false;
  if (d->head_dim < 1 || d->num_pages < 1 || d->nnz_pages < 0) return false;
  if ((int64_t)d->nnz_pages * ta::kPageSize > INT32_MAX) return false;
  return true;
}

// The contiguous-layout dims whose workspace serves a paged call: the kv
// rows of the batch are at most nnz_pages * 16.
ta_dims as_dims(const ta_paged_dims* d) {
  ta_dims x{};
  x.batch_size = d->batch_size;
  x.total_q = d->total_q;
  x.total_kv = d->nnz_pages * ta::kPageSize;
  x.total_tree = d->total_tree;
  x.h_q = d->h_q;
  x.h_kv = d->h_kv;
  x.head_dim = d->head_dim;
  x.dtype = d->dtype;
  x.rotary_mode = 0;
  return x;
}

}  // namespace

extern "C" {

size_t tree_attn_paged_workspace_size(const ta_paged_dims* dims) {
  if (!paged_dims_valid(dims)) return 0;
  const ta_dims d = as_dims(dims);
  return ws_size(&d, 1);   // the paged kernel does not split
}

ta_status tree_attn_paged(const void* q, const int32_t* q_indptr, const void* pages,
                          const int32_t* page_indptr, const int32_t* page_values,
                          const int32_t* length_info, const int32_t* mn_indptr,
                          const int32_t* tree_order, void* out, float* lse, int32_t rotary_mode,
                          float sm_scale, const ta_paged_dims* dims, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!paged_dims_valid(dims)) return TA_ERR_INVALID_ARGUMENT;
  if (rotary_mode != 0) return TA_ERR_UNSUPPORTED;   // as the pages assert for this kernel
  const ta_dims d = as_dims(dims);
  const ta_status sup = dims_supported(&d);
  if (sup != TA_OK) return sup;
  if (!q_indptr || !page_indptr || !length_info || !mn_indptr || !workspace || !pages)
    return TA_ERR_INVALID_ARGUMENT;
  if (dims->nnz_pages > 0 && !page_values) return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_tree > 0 && !tree_order) return TA_ERR_INVALID_ARGUMENT;
  if (!aligned(workspace, 256) || !aligned(pages, 16)) return TA_ERR_INVALID_ARGUMENT;
  const size_t need = ws_size(&d, 1);
  if (need == 0) return TA_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return TA_ERR_INVALID_ARGUMENT;
  if (dims->total_q > 0 && dims->nnz_pages == 0) return TA_ERR_INVALID_ARGUMENT;
  ta_status s = check_run_args(q, pages, pages, out, lse, sm_scale, &d);
  if (s != TA_OK) return s;
  if (dims->total_q == 0) return TA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int g = d.h_q / d.h_kv;
  const int R = ta::rows_per_item(g);
  const WsLayout L = layout_of(&d);
  const WsPtrs w = ws_ptrs(workspace, L);
  const int nsm = sm_count();
  if (nsm <= 0) return cuda_failure();
  // plan: kv lengths from the page table
  ta::PlanParams pp{};
  pp.q_indptr = q_indptr;
  pp.kv_indptr = nullptr;
  pp.mn_indptr = mn_indptr;
  pp.tree_order = tree_order;
  pp.paged = 1;
  pp.page_indptr = page_indptr;
  pp.length_info = length_info;
  pp.nnz_pages = dims->nnz_pages;
  pp.batch = d.batch_size;
  pp.g = g;
  pp.R = R;
  pp.h_kv = d.h_kv;
  pp.head_dim = d.head_dim;
  pp.total_q = d.total_q;
  pp.total_kv = d.total_kv;
  pp.total_tree = d.total_tree;
  pp.max_pairs = L.max_pairs;
  pp.max_chunks = 1;
  pp.chunk_tiles = 0;
  pp.pipes = nsm;   // one attention pipeline per SM
  pp.merge = nullptr;
  pp.hdr = w.hdr;
  pp.sorted = w.sorted;
  pp.classes = w.classes;
  const cudaError_t pe = ta::launch_plan(pp, (int)L.max_pairs, st);
  if (pe != cudaSuccess) return cuda_status(pe);
  // run: K and V tiles gathered page by page from the pool
  CUtensorMap tm_q, tm_pages;
  if (!make_map(&tm_q, q, d.dtype, d.total_q, d.h_q, d.head_dim, g, R) ||
      !make_pages_map(&tm_pages, pages, d.dtype, dims->num_pages, d.h_kv, d.head_dim))
    return cuda_failure();
  ta::AttnParams ap{};
  ap.tree_order = tree_order;
  ap.out = out;
  ap.lse = lse;
  ap.sorted = w.sorted;
  ap.classes = w.classes;
  ap.rope_cs = w.rope_cs;
  ap.hdr = w.hdr;
  ap.page_values = page_values;
  ap.num_pages = dims->num_pages;
  ap.h_q = d.h_q;
  ap.h_kv = d.h_kv;
  ap.g = g;
  ap.R = R;
  ap.rotary = 0;
  ap.max_records = L.max_records;
  ap.scale_log2 = sm_scale * 1.4426950408889634f;
  ap.timeout_ns = wait_limit_ns();
  ap.debug_stall = g_stall;
  ap.sched_clc = g_sched;
  ap.part_o = nullptr;
  ap.part_lse = nullptr;
  const int64_t max_items = L.max_records * d.h_kv;
  const int grid = attn_grid(max_items, nsm);
  const bool bf16 = d.dtype == TA_BF16;
  cudaError_t e;
  if (d.head_dim == 64)
    e = bf16 ? ta::launch_attn<64, true, true>(tm_q, tm_pages, tm_pages, ap, grid, st)
             : ta::launch_attn<64, false, true>(tm_q, tm_pages, tm_pages, ap, grid, st);
  else
    e = bf16 ? ta::launch_attn<128, true, true>(tm_q, tm_pages, tm_pages, ap, grid, st)
             : ta::launch_attn<128, false, true>(tm_q, tm_pages, tm_pages, ap, grid, st);
  return cuda_status(e);
}

}  // extern "C"
