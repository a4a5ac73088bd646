// ta_plan.cu -- the plan kernel of batched tree attention and the dense
// mask export used by tests.
//
// One launch of the plan kernel:
//   1. enumerates the (sequence, q tile) pairs of the ragged batch (the
//      ``advance_tile_batch`` walk of the page "_kernel_common.py", done once
//      up front instead of per CTA), validating the index arrays on the way;
//   2. classifies every (q tile, kv tile) as EMPTY / PARTIAL / FULL from the
//      DFS intervals of ``_check_tree_order`` (page "tree_attn.py"), exactly:
//      the q tile's enter indices are sorted and, for each kv column, the
//      number of them inside the column's [enter, exit) interval is counted;
//   3. orders the pairs longest-first (LPT) for the attention kernel's
//      work queue (the last CTA to finish does a counting sort);
//   4. fills the RoPE cos/sin table, one entry per (kv token, frequency), in
//      the float32 steps of ``_rope`` (page "_kernel_common.py"): angle =
//      fl32(fl32(pos * scale) / fl32(theta^(2i/d))), cos and sin of it
//      rounded correctly to float32 (cr_sincosf).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ta_device.cuh"
#include "ta_sincos.cuh"
#include "ta_launch.h"

namespace ta {
namespace {

constexpr int kPlanThreads = 256;

// Exclusive block-wide scan of two int64 values (256 threads).
__device__ void block_exclusive_scan2(long long& a, long long& b, long long& total_a,
                                      long long& total_b, long long* s_a, long long* s_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long ta = __shfl_up_sync(0xffffffffu, ia, o);
    const long long tb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
    }
  }
  if (lane == 31) {
    s_a[warp] = ia;
    s_b[warp] = ib;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long ra = 0, rb = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      const long long xa = s_a[w], xb = s_b[w];
      s_a[w] = ra;
      s_b[w] = rb;
      ra += xa;
      rb += xb;
    }
    s_a[kPlanThreads / 32] = ra;
    s_b[kPlanThreads / 32] = rb;
  }
  __syncthreads();
  a = s_a[warp] + ia - a;
  b = s_b[warp] + ib - b;
  total_a = s_a[kPlanThreads / 32];
  total_b = s_b[kPlanThreads / 32];
  __syncthreads();
}

// First index in sorted keys[0, n) whose value is >= x.
__device__ __forceinline__ int lower_bound(const int* keys, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (keys[mid] < x)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
  __shared__ long long s_scan_a[kPlanThreads / 32 + 1], s_scan_b[kPlanThreads / 32 + 1];
  __shared__ int s_keys[kBlockM];
  __shared__ int s_pair_b, s_pair_t;
  __shared__ long long s_pair_off;
  __shared__ int s_any[kPlanThreads / 32], s_all[kPlanThreads / 32];
  __shared__ int s_count[2];
  __shared__ float s_den[64];
  __shared__ int s_last;
  __shared__ int s_hist[kCostBuckets];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.batch, R = p.R;

  // ---- 1. enumerate (sequence, q tile) pairs and validate the index arrays
  const int per = (B + kPlanThreads - 1) / kPlanThreads;
  const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
  long long my_tiles = 0, my_seg = 0;
  int bad = 0;
  for (int b = b_lo; b < b_hi; ++b) {
    const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
    const int kv = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int tl = p.mn_indptr[b + 1] - p.mn_indptr[b];
    if (qo < 0 || tl < qo || kv < tl) {
      bad = 1;
      continue;
    }
    const long long tiles = (qo + R - 1) / R;
    const long long kvt = (kv + kBlockN - 1) / kBlockN;
    my_tiles += tiles;
    my_seg += tiles * ((kvt + 15) / 16 * 16);
  }
  if (tid == 0) {
    if (p.q_indptr[0] != 0 || p.kv_indptr[0] != 0 || p.mn_indptr[0] != 0 ||
        p.q_indptr[B] != p.total_q || p.kv_indptr[B] != p.total_kv ||
        p.mn_indptr[B] != p.total_tree)
      bad = 1;
  }
  bad = __syncthreads_or(bad);
  long long excl_tiles = my_tiles, excl_seg = my_seg, total_tiles, total_seg;
  block_exclusive_scan2(excl_tiles, excl_seg, total_tiles, total_seg, s_scan_a, s_scan_b);
  if (total_tiles > p.max_pairs) bad = 1;

  const long long pair = blockIdx.x;
  if (!bad && pair >= excl_tiles && pair < excl_tiles + my_tiles) {
    long long tcum = excl_tiles, scum = excl_seg;
    for (int b = b_lo; b < b_hi; ++b) {
      const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
      const int kv = p.kv_indptr[b + 1] - p.kv_indptr[b];
      const long long tiles = (qo + R - 1) / R;
      const long long seg = ((kv + kBlockN - 1) / kBlockN + 15) / 16 * 16;
      if (pair < tcum + tiles) {
        s_pair_b = b;
        s_pair_t = (int)(pair - tcum);
        s_pair_off = scum + (pair - tcum) * seg;
        break;
      }
      tcum += tiles;
      scum += tiles * seg;
    }
  }
  if (tid < 2) s_count[tid] = 0;
  __syncthreads();

  // ---- 2. classify the kv tiles of this pair
  if (!bad && pair < total_tiles) {
    const int b = s_pair_b, t = s_pair_t;
    const long long off = s_pair_off;
    const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
    const int kv = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int tree_base = p.mn_indptr[b];
    const int tl = p.mn_indptr[b + 1] - tree_base;
    const int ts = kv - tl;
    const int r0 = t * R;
    const int nrows = min(R, qo - r0);
    if (tid < kBlockM)
      s_keys[tid] = tid < nrows ? p.tree_order[2 * (tree_base + r0 + tid + tl - qo)] : INT_MAX;
    __syncthreads();
    // bitonic sort of the q rows' enter indices
    for (int k = 2; k <= kBlockM; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        if (tid < kBlockM) {
          const int ixj = tid ^ j;
          if (ixj > tid) {
            const int a = s_keys[tid], c = s_keys[ixj];
            const bool up = (tid & k) == 0;
            if ((a > c) == up) {
              s_keys[tid] = c;
              s_keys[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    const int kvt = (kv + kBlockN - 1) / kBlockN;
    for (int j0 = 0; j0 < kvt; j0 += 2) {
      const int half = tid >> 7;  // two kv tiles per pass
      const int j = j0 + half;
      const int c = j * kBlockN + (tid & (kBlockN - 1));
      const bool in = j < kvt && c < kv;
      int cnt = 0;
      if (in) {
        if (c < ts) {
          cnt = nrows;
        } else {
          const int2 iv = reinterpret_cast<const int2*>(p.tree_order)[tree_base + c - ts];
          cnt = max(0, lower_bound(s_keys, nrows, iv.y) - lower_bound(s_keys, nrows, iv.x));
        }
      }
      const unsigned any = __ballot_sync(0xffffffffu, in && cnt > 0);
      const unsigned notall = __ballot_sync(0xffffffffu, in && cnt != nrows);
      if (lane == 0) {
        s_any[warp] = any != 0u;
        s_all[warp] = notall == 0u;
      }
      __syncthreads();
      if ((tid & (kBlockN - 1)) == 0 && j < kvt) {
        const int w0 = half * 4;
        const int a = s_any[w0] | s_any[w0 + 1] | s_any[w0 + 2] | s_any[w0 + 3];
        const int al = s_all[w0] & s_all[w0 + 1] & s_all[w0 + 2] & s_all[w0 + 3];
        const bool ragged = (j + 1) * kBlockN > kv;
        const uint8_t cls = !a ? kTileEmpty : ((al && !ragged) ? kTileFull : kTilePartial);
        p.classes[off + j] = cls;
        if (cls != kTileEmpty) s_count[half] += 1;
      }
      __syncthreads();
    }
    if (tid == 0) {
      PairInfo pi;
      pi.b = b;
      pi.t = t;
      pi.class_off = (int32_t)off;
      pi.n_tiles = s_count[0] + s_count[1];
      p.pairs[pair] = pi;
    }
  }

  // ---- 4. RoPE cos/sin table: angle = fl32(fl32(pos * scale) / fl32(theta^(2i/d)))
  if (p.rotary) {
    const int half = p.head_dim / 2;
    if (tid < half)
      s_den[tid] = (float)pow((double)p.rope_theta, (2.0 * tid) / (double)p.head_dim);
    __syncthreads();
    const long long tpc = ((long long)p.total_kv + gridDim.x - 1) / gridDim.x;
    const long long tok0 = (long long)blockIdx.x * tpc;
    const long long tok1 = min((long long)p.total_kv, tok0 + tpc);
    if (tok1 > tok0) {
      const long long n = (tok1 - tok0) * half;
      for (long long idx = tid; idx < n; idx += kPlanThreads) {
        const long long tok = tok0 + idx / half;
        const int i = (int)(idx % half);
        const float s = __fmul_rn((float)p.rope_pos[tok], p.rope_scale);
        const float ang = __fdiv_rn(s, s_den[i]);
        float sn, cs;
        cr_sincosf(ang, &sn, &cs);
        p.rope_cs[tok * half + i] = make_float2(cs, sn);
      }
    }
  }

  // ---- 3. the last CTA orders the pairs longest-first
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.hdr->plan_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const long long np = bad ? 0 : total_tiles;
  for (int i = tid; i < kCostBuckets; i += kPlanThreads) s_hist[i] = 0;
  __syncthreads();
  for (long long i = tid; i < np; i += kPlanThreads) {
    const int c = min(__ldcg(&p.pairs[i].n_tiles), kCostBuckets - 1);
    atomicAdd(&s_hist[kCostBuckets - 1 - c], 1);
  }
  __syncthreads();
  {
    constexpr int per_t = kCostBuckets / kPlanThreads;
    long long sum = 0;
    for (int i = 0; i < per_t; ++i) sum += s_hist[tid * per_t + i];
    long long excl = sum, dummy = 0, tot, tot2;
    block_exclusive_scan2(excl, dummy, tot, tot2, s_scan_a, s_scan_b);
    long long run = excl;
    for (int i = 0; i < per_t; ++i) {
      const int v = s_hist[tid * per_t + i];
      s_hist[tid * per_t + i] = (int)run;
      run += v;
    }
  }
  __syncthreads();
  for (long long i = tid; i < np; i += kPlanThreads) {
    const int c = min(__ldcg(&p.pairs[i].n_tiles), kCostBuckets - 1);
    const int pos = atomicAdd(&s_hist[kCostBuckets - 1 - c], 1);
    p.sorted[pos] = (int32_t)i;
  }
  if (tid == 0) {
    p.hdr->num_pairs = (unsigned int)np;
    p.hdr->num_items = (unsigned int)(np * p.h_kv);
    p.hdr->queue_head = 0;
    p.hdr->queue_done = 0;
    p.hdr->plan_done = 0;
    if (bad) atomicOr(&p.hdr->error, DEVERR_BAD_INDPTR);
    __threadfence();
  }
}

__global__ void mask_dense_kernel(const int32_t* __restrict__ q_indptr,
                                  const int32_t* __restrict__ kv_indptr,
                                  const int32_t* __restrict__ mn_indptr,
                                  const int32_t* __restrict__ tree_order, int batch, int max_kv,
                                  uint8_t* __restrict__ vis) {
  const int row = blockIdx.x;
  int lo = 0, hi = batch;  // largest b with q_indptr[b] <= row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (q_indptr[mid] <= row)
      lo = mid;
    else
      hi = mid;
  }
  const int b = lo;
  const int qo = q_indptr[b + 1] - q_indptr[b];
  const int kv = kv_indptr[b + 1] - kv_indptr[b];
  const int tree_base = mn_indptr[b];
  const int tl = mn_indptr[b + 1] - tree_base;
  const int ts = kv - tl;
  const int r = row - q_indptr[b];
  const int e_row = tree_order[2 * (tree_base + r + tl - qo)];
  for (int c = threadIdx.x; c < max_kv; c += blockDim.x) {
    const int2 iv = column_interval(tree_order, tree_base, c, kv, ts);
    vis[(size_t)row * max_kv + c] = (iv.x <= e_row && e_row < iv.y) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, int grid, cudaStream_t stream) {
  plan_kernel<<<grid, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_mask_dense(const int32_t* q_indptr, const int32_t* kv_indptr,
                              const int32_t* mn_indptr, const int32_t* tree_order, int batch,
                              int total_q, int max_kv, uint8_t* vis, cudaStream_t stream) {
  if (total_q <= 0) return cudaSuccess;
  mask_dense_kernel<<<total_q, 128, 0, stream>>>(q_indptr, kv_indptr, mn_indptr, tree_order,
                                                 batch, max_kv, vis);
  return cudaGetLastError();
}

}  // namespace ta
