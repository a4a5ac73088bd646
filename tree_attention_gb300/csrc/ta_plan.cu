// ta_plan.cu -- the plan kernel of batched tree attention and the dense
// mask export used by tests.
//
// One launch of the plan kernel does, per CTA, two independent jobs in two
// warp groups (synchronised with named barriers, so neither waits for the
// other):
//   group A (warps 0-3)
//     1. enumerates the (sequence, q tile) pairs of the ragged batch (the
//        ``advance_tile_batch`` walk of the page "_kernel_common.py", done
//        once up front instead of per CTA), validating the index arrays;
//     2. classifies every (q tile, kv tile) of its pair as EMPTY / PARTIAL /
//        FULL from the DFS intervals of ``_check_tree_order`` (page
//        "tree_attn.py"), exactly: the q rows' enter indices are sorted and,
//        for each kv column, two binary searches count the rows inside the
//        column's [enter, exit) interval; then writes the pair's item record;
//   group B (warps 4-7)
//     4. fills a slice of the RoPE cos/sin table, one entry per (kv token,
//        frequency), in the float32 steps of ``_rope`` (page
//        "_kernel_common.py"): angle = fl32(fl32(pos * scale) /
//        fl32(theta^(2i/d))), cos and sin of it rounded correctly to float32
//        (cr_sincosf).
// Finally (3.) the last CTA to finish orders the item records longest-first
// (LPT) for the attention kernel's work queue with a counting sort.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ta_device.cuh"
#include "ta_launch.h"
#include "ta_sincos.cuh"

namespace ta {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kGroup = 128;  // threads per warp group
constexpr int kBarA = 1, kBarB = 2;
constexpr int kPassTiles = 256;  // kv tiles classified per pass

__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGroup) : "memory");
}

// Exclusive scan of two int64 values over ``nthreads`` threads (a multiple
// of 32) starting at thread ``first``; ``sync`` synchronises those threads.
template <typename Sync>
__device__ void exclusive_scan2(long long& a, long long& b, long long& total_a,
                                long long& total_b, long long* s_a, long long* s_b, int first,
                                int nthreads, Sync sync) {
  const int t = threadIdx.x - first;
  const int lane = t & 31, warp = t >> 5, nwarps = nthreads >> 5;
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
  sync();
  if (t == 0) {
    long long ra = 0, rb = 0;
    for (int w = 0; w < nwarps; ++w) {
      const long long xa = s_a[w], xb = s_b[w];
      s_a[w] = ra;
      s_b[w] = rb;
      ra += xa;
      rb += xb;
    }
    s_a[nwarps] = ra;
    s_b[nwarps] = rb;
  }
  sync();
  a = s_a[warp] + ia - a;
  b = s_b[warp] + ib - b;
  total_a = s_a[nwarps];
  total_b = s_b[nwarps];
  sync();
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

__device__ __forceinline__ long long seg_bytes(int kv) {
  return ((kv + kBlockN - 1) / kBlockN + 15) / 16 * 16;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
  __shared__ long long s_scan_a[9], s_scan_b[9];
  __shared__ int s_keys[kBlockM];
  __shared__ int s_pair_b, s_pair_t;
  __shared__ long long s_pair_off, s_total;
  __shared__ int s_bad;
  __shared__ int s_any[kPassTiles], s_notall[kPassTiles];
  __shared__ uint32_t s_cls2[3];
  __shared__ int s_count;
  __shared__ double s_log2_theta;
  __shared__ float s_den[64];
  __shared__ float4 s_sct[27];
  __shared__ int s_last;
  __shared__ int s_hist[kCostBuckets];

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if (tid < kGroup) {
    // ======================= group A: enumerate and classify ================
    const int B = p.batch, R = p.R;
    if (tid == 0) {
      s_bad = (p.q_indptr[0] != 0 || p.kv_indptr[0] != 0 || p.mn_indptr[0] != 0 ||
               p.q_indptr[B] != p.total_q || p.kv_indptr[B] != p.total_kv ||
               p.mn_indptr[B] != p.total_tree);
      s_count = 0;
    }
    const int per = (B + kGroup - 1) / kGroup;
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
      my_tiles += tiles;
      my_seg += tiles * seg_bytes(kv);
    }
    long long ex_tiles = my_tiles, ex_seg = my_seg, total_tiles, total_seg;
    exclusive_scan2(ex_tiles, ex_seg, total_tiles, total_seg, s_scan_a, s_scan_b, 0, kGroup,
                    [] { group_sync(kBarA); });
    if (bad) atomicOr(&s_bad, 1);
    const long long pair = blockIdx.x;
    if (pair >= ex_tiles && pair < ex_tiles + my_tiles) {
      long long tcum = ex_tiles, scum = ex_seg;
      for (int b = b_lo; b < b_hi; ++b) {
        const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
        const int kv = p.kv_indptr[b + 1] - p.kv_indptr[b];
        const long long tiles = (qo + R - 1) / R;
        if (pair < tcum + tiles) {
          s_pair_b = b;
          s_pair_t = (int)(pair - tcum);
          s_pair_off = scum + (pair - tcum) * seg_bytes(kv);
          break;
        }
        tcum += tiles;
        scum += tiles * seg_bytes(kv);
      }
    }
    group_sync(kBarA);
    const bool ok = !s_bad && total_tiles <= p.max_pairs;
    if (tid == 0) {
      s_total = total_tiles;
      if (!ok) s_bad = 1;
    }
    if (ok && pair < total_tiles) {
      const int b = s_pair_b, t = s_pair_t;
      const long long off = s_pair_off;
      const int q0 = p.q_indptr[b];
      const int qo = p.q_indptr[b + 1] - q0;
      const int kv_base = p.kv_indptr[b];
      const int kv = p.kv_indptr[b + 1] - kv_base;
      const int tree_base = p.mn_indptr[b];
      const int tl = p.mn_indptr[b + 1] - tree_base;
      const int ts = kv - tl;
      const int r0 = t * R;
      const int nrows = min(R, qo - r0);
      s_keys[tid] =
          tid < nrows ? p.tree_order[2 * (tree_base + r0 + tid + tl - qo)] : INT_MAX;
      group_sync(kBarA);
      // bitonic sort of the q rows' enter indices (128 keys, one per thread)
      for (int k = 2; k <= kBlockM; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
          const int ixj = tid ^ j;
          if (ixj > tid) {
            const int a = s_keys[tid], c = s_keys[ixj];
            const bool up = (tid & k) == 0;
            if ((a > c) == up) {
              s_keys[tid] = c;
              s_keys[ixj] = a;
            }
          }
          group_sync(kBarA);
        }
      }
      const int kvt = (kv + kBlockN - 1) / kBlockN;
      if (tid < 3) s_cls2[tid] = 0;
      // up to kPassTiles kv tiles per pass; every thread takes every 128th
      // column of the pass and folds its verdict into per-tile flags
      for (int j0 = 0; j0 < kvt; j0 += kPassTiles) {
        const int nt = min(kPassTiles, kvt - j0);
        for (int i = tid; i < nt; i += kGroup) {
          s_any[i] = 0;
          s_notall[i] = 0;
        }
        group_sync(kBarA);
        const int c_end = min(kv, (j0 + nt) * kBlockN);
        for (int c = j0 * kBlockN + tid; c < c_end; c += kGroup) {
          int cnt;
          if (c < ts) {
            cnt = nrows;
          } else {
            const int2 iv = reinterpret_cast<const int2*>(p.tree_order)[tree_base + c - ts];
            cnt = max(0, lower_bound(s_keys, nrows, iv.y) - lower_bound(s_keys, nrows, iv.x));
          }
          const int jt = c / kBlockN - j0;
          if (cnt > 0 && !s_any[jt]) s_any[jt] = 1;
          if (cnt != nrows && !s_notall[jt]) s_notall[jt] = 1;
        }
        group_sync(kBarA);
        for (int i = tid; i < nt; i += kGroup) {
          const int j = j0 + i;
          const bool ragged = (j + 1) * kBlockN > kv;
          const uint8_t cls =
              !s_any[i] ? kTileEmpty : ((!s_notall[i] && !ragged) ? kTileFull : kTilePartial);
          p.classes[off + j] = cls;
          if (cls != kTileEmpty) atomicAdd(&s_count, 1);
          if (kvt <= kInlineTiles) atomicOr(&s_cls2[j >> 4], (uint32_t)cls << (2 * (j & 15)));
        }
        group_sync(kBarA);
      }
      if (tid == 0) {
        ItemRec r;
        r.b = b;
        r.t = t;
        r.q_row0 = q0 + r0;
        r.nq = nrows;
        r.qo = qo;
        r.kv = kv;
        r.tl = tl;
        r.ts = ts;
        r.kv_base = kv_base;
        r.tree_base = tree_base;
        r.n_tiles = s_count;
        r.class_off = (int32_t)off;
        r.kvt = kvt;
        r.cls2[0] = s_cls2[0];
        r.cls2[1] = s_cls2[1];
        r.cls2[2] = s_cls2[2];
        p.recs[pair] = r;
      }
    }
  } else if (p.rotary) {
    // ======================= group B: RoPE ==================================
    const int tb = tid - kGroup;
    const int wb = tb >> 5, lane = tb & 31;
    const int D = p.head_dim, half = D / 2;
    if (tb == 0) s_log2_theta = log2((double)p.rope_theta);
    if (tb < 27)
      s_sct[tb] = make_float4(kSinCosTable[tb][0], kSinCosTable[tb][1], kSinCosTable[tb][2],
                              kSinCosTable[tb][3]);
    group_sync(kBarB);
    // fl32(theta^(2i/d)), through float64 so that the float32 rounding is right
    if (tb < half) s_den[tb] = (float)exp2(s_log2_theta * ((2.0 * tb) / (double)D));
    group_sync(kBarB);
    // every warp owns a contiguous run of kv tokens
    const long long nwarps = (long long)gridDim.x * (kGroup / 32);
    const long long per = ((long long)p.total_kv + nwarps - 1) / nwarps;
    const long long t0 = ((long long)blockIdx.x * (kGroup / 32) + wb) * per;
    const long long t1 = min((long long)p.total_kv, t0 + per);
    if (t0 < t1) {
      // lane l computes frequencies (2l, 2l+1) (d = 128) or, for d = 64, lanes
      // 0..15 compute them and lanes 16..31 repeat the work of lanes 0..15
      const int pl = (D == 128) ? lane : (lane & 15);
      const int i0 = 2 * pl, i1 = 2 * pl + 1;
      for (long long base = t0; base < t1; base += 32) {
        const long long my_tok = base + lane;
        const int my_pos = my_tok < t1 ? p.rope_pos[my_tok] : 0;
        const int ntok = (int)min(32LL, t1 - base);
        const float den0 = s_den[i0], den1 = s_den[i1];
        // two tokens per step: four independent sin/cos evaluations in flight
        for (int u = 0; u < ntok; u += 2) {
          const bool two = u + 1 < ntok;
          const int pos_a = __shfl_sync(0xffffffffu, my_pos, u);
          const int pos_b = __shfl_sync(0xffffffffu, my_pos, two ? u + 1 : u);
          const float sa = __fmul_rn((float)pos_a, p.rope_scale);
          const float sb = __fmul_rn((float)pos_b, p.rope_scale);
          float s0a, c0a, s1a, c1a, s0b, c0b, s1b, c1b;
          cr_sincosf(__fdiv_rn(sa, den0), &s0a, &c0a, s_sct);
          cr_sincosf(__fdiv_rn(sa, den1), &s1a, &c1a, s_sct);
          cr_sincosf(__fdiv_rn(sb, den0), &s0b, &c0b, s_sct);
          cr_sincosf(__fdiv_rn(sb, den1), &s1b, &c1b, s_sct);
          if (D == 128 || lane < 16) {
            float4* row = reinterpret_cast<float4*>(p.rope_cs + (base + u) * half);
            row[pl] = make_float4(c0a, s0a, c1a, s1a);
            if (two) row[half / 2 + pl] = make_float4(c0b, s0b, c1b, s1b);
          }
        }
      }
    }
  }

  // ======================= 3. the last CTA orders the records ===============
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.hdr->plan_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const long long np = s_bad ? 0 : s_total;
  for (int i = tid; i < kCostBuckets; i += kPlanThreads) s_hist[i] = 0;
  __syncthreads();
  for (long long i = tid; i < np; i += kPlanThreads) {
    const int c = min(__ldcg(&p.recs[i].n_tiles), kCostBuckets - 1);
    atomicAdd(&s_hist[kCostBuckets - 1 - c], 1);
  }
  __syncthreads();
  {
    constexpr int per_t = kCostBuckets / kPlanThreads;
    long long sum = 0;
    for (int i = 0; i < per_t; ++i) sum += s_hist[tid * per_t + i];
    long long excl = sum, dummy = 0, tot, tot2;
    exclusive_scan2(excl, dummy, tot, tot2, s_scan_a, s_scan_b, 0, kPlanThreads,
                    [] { __syncthreads(); });
    long long run = excl;
    for (int i = 0; i < per_t; ++i) {
      const int v = s_hist[tid * per_t + i];
      s_hist[tid * per_t + i] = (int)run;
      run += v;
    }
  }
  __syncthreads();
  for (long long i = tid; i < np; i += kPlanThreads) {
    const int4* src = reinterpret_cast<const int4*>(&p.recs[i]);
    int4 r[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) r[w] = __ldcg(src + w);
    const int c = min(r[2].z, kCostBuckets - 1);  // n_tiles is the 11th field
    const int pos = atomicAdd(&s_hist[kCostBuckets - 1 - c], 1);
    int4* dst = reinterpret_cast<int4*>(&p.sorted[pos]);
#pragma unroll
    for (int w = 0; w < 4; ++w) dst[w] = r[w];
  }
  if (tid == 0) {
    p.hdr->num_pairs = (unsigned int)np;
    p.hdr->num_items = (unsigned int)(np * p.h_kv);
    p.hdr->queue_head = 0;
    p.hdr->queue_done = 0;
    p.hdr->plan_done = 0;
    if (s_bad) atomicOr(&p.hdr->error, DEVERR_BAD_INDPTR);
    __threadfence();
  }
}

// One warp per kv token at a time: lane l holds the cos/sin of frequencies
// (2l', 2l'+1) (one float4 of the table row) and rotates those element pairs
// of every kv head -- words l' of the first half and d/4 + l' of the second
// half of the head's row -- with the float32 steps of ``_rope``.  For d = 64
// lanes 16..31 take the odd heads.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) krot_kernel(const uint32_t* __restrict__ k,
                                                   uint32_t* __restrict__ krot,
                                                   const float4* __restrict__ cs, int total_kv,
                                                   int h_kv) {
  constexpr int kWords = D / 2;  // 32-bit words per head row
  const int lane = threadIdx.x & 31;
  const int pl = (D == 128) ? lane : (lane & 15);
  const int h0 = (D == 128) ? 0 : (lane >> 4);
  constexpr int hstep = (D == 128) ? 1 : 2;
  pdl_wait();
  pdl_trigger();
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long tok = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
       tok < total_kv; tok += warps) {
    const float4 c = __ldg(cs + tok * (D / 4) + pl);  // (cos, sin) of 2 frequencies
    for (int hb = h0; hb < h_kv; hb += 8 * hstep) {
      uint32_t w0[8], w1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int h = hb + u * hstep;
        if (h < h_kv) {
          const long long e = (tok * h_kv + h) * kWords;
          w0[u] = __ldg(k + e + pl);
          w1[u] = __ldg(k + e + kWords / 2 + pl);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int h = hb + u * hstep;
        if (h < h_kv) {
          const float2 x0 = unpack2<BF16>(w0[u]);
          const float2 x1 = unpack2<BF16>(w1[u]);
          // first half: cos*x[j] + sin*(-x[j+d/2]); second half: cos*x[j] + sin*x[j-d/2]
          const float y0a = __fadd_rn(__fmul_rn(c.x, x0.x), __fmul_rn(c.y, -x1.x));
          const float y0b = __fadd_rn(__fmul_rn(c.z, x0.y), __fmul_rn(c.w, -x1.y));
          const float y1a = __fadd_rn(__fmul_rn(c.x, x1.x), __fmul_rn(c.y, x0.x));
          const float y1b = __fadd_rn(__fmul_rn(c.z, x1.y), __fmul_rn(c.w, x0.y));
          const long long e = (tok * h_kv + h) * kWords;
          krot[e + pl] = pack2<BF16>(y0a, y0b);
          krot[e + kWords / 2 + pl] = pack2<BF16>(y1a, y1b);
        }
      }
    }
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
  return launch_pdl(plan_kernel, dim3(grid), dim3(kPlanThreads), 0, stream, p);
}

cudaError_t launch_krot(const void* k, void* krot, const float2* rope_cs, int total_kv, int h_kv,
                        int head_dim, bool bf16, int grid, cudaStream_t stream) {
  if (total_kv <= 0) return cudaSuccess;
  const uint32_t* kin = static_cast<const uint32_t*>(k);
  uint32_t* kout = static_cast<uint32_t*>(krot);
  const float4* cs = reinterpret_cast<const float4*>(rope_cs);
  cudaError_t e;
  if (head_dim == 128) {
    if (bf16)
      e = launch_pdl(krot_kernel<true, 128>, dim3(grid), dim3(256), 0, stream, kin, kout,
                     cs, total_kv, h_kv);
    else
      e = launch_pdl(krot_kernel<false, 128>, dim3(grid), dim3(256), 0, stream, kin, kout,
                     cs, total_kv, h_kv);
  } else {
    if (bf16)
      e = launch_pdl(krot_kernel<true, 64>, dim3(grid), dim3(256), 0, stream, kin, kout,
                     cs, total_kv, h_kv);
    else
      e = launch_pdl(krot_kernel<false, 64>, dim3(grid), dim3(256), 0, stream, kin, kout,
                     cs, total_kv, h_kv);
  }
  return e;
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
