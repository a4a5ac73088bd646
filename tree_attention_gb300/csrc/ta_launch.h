// ta_launch.h -- internal interface between the C-ABI host code (ta_api.cu)
// and the kernel translation units (ta_plan.cu, ta_attn.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "ta_layout.h"

namespace ta {

// Launches a kernel of this library with programmatic dependent launch: its
// CTAs may be scheduled while the previous kernel on the stream is still
// running, and every kernel here executes pdl_wait() (griddepcontrol.wait)
// before it reads or writes anything that kernel may touch, so stream order
// is kept while launch latency and prologues overlap.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Key rotation: the RoPE frequency denominators fl32(theta^(2i/d)) for
// i < d/2 (``_rope``, page "_kernel_common.py"; rounded once from float64 on
// the host), the position scale and the sizes.
struct KrotParams {
  float rope_den[64];
  float rope_scale;
  int total_kv, h_kv;
};

struct PlanParams {
  const int32_t* q_indptr;
  const int32_t* kv_indptr;
  const int32_t* mn_indptr;
  const int32_t* tree_order;
  // paged KV cache (paged != 0): kv rows come from 16-slot pages; kv_indptr
  // is unused, the kv length of sequence b is (pages - 1) * 16 + length_info[b]
  int paged;
  const int32_t* page_indptr;
  const int32_t* length_info;
  int nnz_pages;
  int batch, g, R, h_kv, head_dim, total_q, total_kv, total_tree;
  int64_t max_pairs;
  // split-KV: a pair's kv tiles are cut into up to max_chunks records of
  // about chunk_tiles tiles (0: chosen from the batch's total work so that
  // the items cover the ``pipes`` pipelines of the attention grid -- one
  // per SM -- a few times); max_chunks == 1 disables it
  int max_chunks, chunk_tiles, pipes;
  int4* merge;       // per pair (split-KV): q_row0, q rows, chunks, first record
  // one-call entry points: the plan kernel also does the key rotation of the
  // run (krot_kernel's work) on the warps the plan leaves idle.  rot: 0 none,
  // else 1 + 2 * (head_dim == 128) + (dtype == bf16)
  int rot;
  const uint32_t* rot_k;
  uint32_t* rot_out;
  const int32_t* rot_pos;
  float4* rot_cs;
  KrotParams kp;
  WsHeader* hdr;
  ItemRec* sorted;   // one record per (sequence, q tile) or chunk of one, longest first
  uint8_t* classes;
};

struct AttnParams {
  const int32_t* tree_order;
  void* out;
  float* lse;
  const ItemRec* sorted;
  const uint8_t* classes;
  const float2* rope_cs;   // [total_kv][head_dim / 2] cos/sin per kv token (RoPE)
  WsHeader* hdr;
  const int32_t* page_values;   // paged KV cache: physical page of each (sequence, page)
  int num_pages;                // pages in the pool (an out-of-range page reads zeros)
  int h_q, h_kv, g, R, rotary;
  int64_t max_records;  // capacity of the record table in the workspace
  float scale_log2;     // sm_scale * log2(e)
  unsigned long long timeout_ns;
  // test hook: the MMA threads first wait on a barrier that nothing arrives
  // on, so that the bounded wait runs out and the abort path runs
  int debug_stall;
  // 0: one CTA per SM takes its first unit by CTA index and the rest from the
  // atomic work queue; 1: one CTA per possible unit, and a CTA that finishes
  // takes the unit of a CTA not yet started by cancelling its launch
  // (cluster launch control)
  int sched_clc;
  // split-KV partial states of the records with part >= 0: O / l in float32
  // [record][h_kv][128 packed rows][d] and the base-2 lse [record][h_kv][128]
  float* part_o;
  float* part_lse;
};

struct MergeParams {
  const int4* merge;           // per pair: q_row0, q rows, chunks, first record
  const float* part_o;
  const float* part_lse;
  void* out;
  float* lse;
  const WsHeader* hdr;         // num_pairs
  int64_t max_pairs, max_records;
  int h_q, h_kv, g;
};

// Plan kernel: sequence/tile enumeration, tile classification and LPT
// ordering.  ``grid`` >= max_pairs.
cudaError_t launch_plan(const PlanParams& p, int grid, cudaStream_t stream);


// RoPE of every kv token: the cos/sin table row of token t at position
// rope_pos[t] (rope_cs[t][i] = (cos, sin) of frequency i) and the rotated
// keys krot[t, h, :] = rope(k[t, h, :]).
cudaError_t launch_krot(const void* k, void* krot, const int32_t* rope_pos, float2* rope_cs,
                        const KrotParams& kp, int head_dim, bool bf16, int grid,
                        cudaStream_t stream);

// Dense mask export (test helper).
cudaError_t launch_mask_dense(const int32_t* q_indptr, const int32_t* kv_indptr,
                              const int32_t* mn_indptr, const int32_t* tree_order, int batch,
                              int total_q, int max_kv, uint8_t* vis, cudaStream_t stream);

// Split-KV: combines the partial states of every split pair into out / lse
// (the base-2 log-sum-exp merge of attention states over disjoint kv sets).
cudaError_t launch_merge(const MergeParams& p, int head_dim, bool bf16, int grid,
                         cudaStream_t stream);

// Stand-alone merge of n_parts attention states per row: parts [n][rows][d]
// and lses [n][rows] -> out [rows][d], lse [rows].
cudaError_t launch_merge_states(const void* parts, const float* lses, int n_parts,
                                long long rows, int head_dim, bool bf16, void* out, float* lse,
                                int grid, cudaStream_t stream);

// Persistent tree-attention kernel.
template <int D, bool BF16, bool PAGED>
cudaError_t launch_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const AttnParams& p, int grid, cudaStream_t stream);

}  // namespace ta
