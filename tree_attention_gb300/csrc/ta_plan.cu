// ta_plan.cu -- the plan kernel of batched tree attention and the dense
// mask export used by tests.
//
// One launch of the plan kernel, every CTA:
//   1. walks the (sequence, unit) pairs of the ragged batch -- a unit is two
//      consecutive Q tiles of 128 packed rows each (the
//      ``advance_tile_batch`` walk of the page "_kernel_common.py", done once
//      up front), validating the index arrays, and places its own pair in the
//      longest-first (LPT) order of the attention kernel's work queue by an
//      estimated cost -- no global barrier, no serial tail;
//   2. (all warps) classifies every kv tile of its pair as EMPTY / PARTIAL /
//      FULL for each of its two Q tiles, exactly, from the DFS intervals of
//      ``_check_tree_order`` (page "tree_attn.py") and writes the pair's item
//      record -- with split-KV, one record per chunk of the pair's kv tiles
//      plus the pair's merge record;
//   3. for the one-call entry points, (the CTAs without a pair first) the
//      run's key rotation: every kv token's RoPE cos/sin and rotated keys.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ta_device.cuh"
#include "ta_launch.h"
#include "ta_sincos.cuh"

namespace ta {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kGroup = 128;  // threads per warp group (one group per Q tile of a unit)
constexpr int kBarA = 1;     // named barriers kBarA (tile A's group), kBarA + 1 (tile B's)
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

// kv rows and kv base of sequence b: contiguous (kv_indptr) or paged (the
// ``_get_kv_chunk_len`` of the page "_kernel_common.py" without a sliding
// window: (pages - 1) * 16 + last_page_len, 0 without pages; the base is then
// the sequence's first page-table entry)
__device__ __forceinline__ int seq_kv_len(const PlanParams& p, int b) {
  if (!p.paged) return p.kv_indptr[b + 1] - p.kv_indptr[b];
  const int np = p.page_indptr[b + 1] - p.page_indptr[b];
  return np > 0 ? (np - 1) * kPageSize + p.length_info[b] : 0;
}
__device__ __forceinline__ int seq_kv_base(const PlanParams& p, int b) {
  return p.paged ? p.page_indptr[b] : p.kv_indptr[b];
}
// a paged sequence's own table entries must be consistent
__device__ __forceinline__ bool seq_pages_bad(const PlanParams& p, int b) {
  if (!p.paged) return false;
  const int np = p.page_indptr[b + 1] - p.page_indptr[b];
  return np < 0 || (np > 0 && (p.length_info[b] < 1 || p.length_info[b] > kPageSize));
}

__device__ __forceinline__ long long seg_bytes(int kv) {
  return ((kv + kBlockN - 1) / kBlockN + 15) / 16 * 16;
}

// Estimated cost of unit t of a sequence (units of U q rows), in kv tiles,
// for the longest-first order: the kv tiles up to the unit's last row's own
// slot (exact for trees whose nodes come after their parents, as in a causal
// prefix; only the order and the split of the work depend on it).
__device__ __forceinline__ int pair_tiles(int qo, int kv, int U, int t) {
  const long long end = (long long)kv - max(0LL, (long long)qo - (long long)(t + 1) * U);
  return (int)((end + kBlockN - 1) / kBlockN);
}

// Split-KV: chunks of a pair of estimated cost ``tiles`` (1 when not split).
__device__ __forceinline__ int pair_chunks(int tiles, int chunk_tiles, int max_chunks) {
  if (max_chunks <= 1) return 1;
  return max(1, min(max_chunks, (tiles + chunk_tiles - 1) / chunk_tiles));
}

// Cost bucket of each of a pair's records: its chunks' estimated cost.
__device__ __forceinline__ int record_bucket(int tiles, int chunks) {
  return min(kCostBuckets - 1, (tiles + chunks - 1) / chunks);
}

// Split-KV chunk size when the caller leaves it to the plan: about a quarter
// of the per-pipeline share of the batch's work, at least kMinChunkTiles.
__device__ __forceinline__ int auto_chunk_tiles(long long total_tiles, int h_kv, int pipes) {
  const long long per = (total_tiles * h_kv + 4LL * pipes - 1) / (4LL * pipes);
  return (int)max((long long)kMinChunkTiles, min(per, (long long)INT_MAX));
}

// RoPE (``_rope`` on the page "_kernel_common.py") of one kv token, by one
// warp: lane l evaluates the cos/sin of frequencies (2l', 2l'+1) in the
// pages' float32 steps -- angle = fl32(fl32(pos * scale) / fl32(theta^(2i/d))),
// cos and sin of it rounded correctly to float32 (cr_sincosf) -- writes them
// to the token's row of the cos/sin table (read by the attention kernel for
// its q rows) and rotates those element pairs of every kv head: words l' of
// the first half and d/4 + l' of the second half of the head's row.  For
// d = 64 lanes 16..31 take the odd heads.  The first heads' keys are loaded
// before the sin/cos evaluation, so the loads are in flight while it runs.
template <bool BF16, int D>
__device__ __forceinline__ void rope_token(const uint32_t* __restrict__ k,
                                           uint32_t* __restrict__ krot, float4* __restrict__ cs,
                                           long long tok, int ps, const KrotParams& kp,
                                           const float4* sct, int lane) {
  constexpr int kWords = D / 2;  // 32-bit words per head row
  const int pl = (D == 128) ? lane : (lane & 15);
  const int h0 = (D == 128) ? 0 : (lane >> 4);
  constexpr int hstep = (D == 128) ? 1 : 2;
  const int h_kv = kp.h_kv;
  uint32_t w0[8], w1[8];
  auto load = [&](int hb) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int h = hb + u * hstep;
      if (h < h_kv) {
        const long long e = (tok * h_kv + h) * kWords;
        w0[u] = __ldg(k + e + pl);
        w1[u] = __ldg(k + e + kWords / 2 + pl);
      }
    }
  };
  load(h0);
  float c0, s0, c1, s1;
  {
    const float sc = __fmul_rn((float)ps, kp.rope_scale);
    cr_sincosf(__fdiv_rn(sc, kp.rope_den[2 * pl]), &s0, &c0, sct);
    cr_sincosf(__fdiv_rn(sc, kp.rope_den[2 * pl + 1]), &s1, &c1, sct);
  }
  if (D == 128 || lane < 16) cs[tok * (D / 4) + pl] = make_float4(c0, s0, c1, s1);
  for (int hb = h0; hb < h_kv; hb += 8 * hstep) {
    if (hb != h0) load(hb);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int h = hb + u * hstep;
      if (h < h_kv) {
        const float2 x0 = unpack2<BF16>(w0[u]);
        const float2 x1 = unpack2<BF16>(w1[u]);
        // first half: cos*x[j] + sin*(-x[j+d/2]); second half: cos*x[j] + sin*x[j-d/2]
        const float y0a = __fadd_rn(__fmul_rn(c0, x0.x), __fmul_rn(s0, -x1.x));
        const float y0b = __fadd_rn(__fmul_rn(c1, x0.y), __fmul_rn(s1, -x1.y));
        const float y1a = __fadd_rn(__fmul_rn(c0, x1.x), __fmul_rn(s0, x0.x));
        const float y1b = __fadd_rn(__fmul_rn(c1, x1.y), __fmul_rn(s1, x0.y));
        const long long e = (tok * h_kv + h) * kWords;
        krot[e + pl] = pack2<BF16>(y0a, y0b);
        krot[e + kWords / 2 + pl] = pack2<BF16>(y1a, y1b);
      }
    }
  }
}

// Warp ``rank`` of ``nwarps`` takes kv tokens rank, rank + nwarps, ...  (not
// inlined: the plan kernel calls one of four instances, which would
// otherwise bloat its code)
template <bool BF16, int D>
__device__ __noinline__ void rope_tokens(const uint32_t* k, uint32_t* krot, const int32_t* pos, float4* cs,
                            const KrotParams& kp, const float4* sct, long long rank,
                            long long nwarps, int lane) {
  for (long long tok = rank; tok < kp.total_kv; tok += nwarps)
    rope_token<BF16, D>(k, krot, cs, tok, __ldg(pos + tok), kp, sct, lane);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
  __shared__ long long s_scan_a[9], s_scan_b[9];
  __shared__ int s_keys[kTilesPerUnit * kBlockM];   // sorted enter keys: tile A, tile B
  __shared__ int s_pair_b, s_pair_t, s_pair_cost, s_pair_chunks;
  __shared__ long long s_total_cost;
  __shared__ int s_last;
  __shared__ int s_ccount[kMaxChunks], s_ccount_a[kMaxChunks], s_ccount_b[kMaxChunks];
  __shared__ long long s_pair_off;
  __shared__ int s_bad, s_rank;
  __shared__ int s_any[kTilesPerUnit][kPassTiles], s_notall[kTilesPerUnit][kPassTiles];
  __shared__ uint32_t s_cls;
  __shared__ int s_count, s_count_a, s_count_b;
  __shared__ int s_hist[kCostBuckets];
  __shared__ float4 s_sct[27];

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.batch, R = p.R, U = kTilesPerUnit * p.R;   // q rows per Q tile / unit
  // ---- 0. constants and counters of this CTA
  for (int i = tid; i < kCostBuckets; i += kPlanThreads) s_hist[i] = 0;
  if (p.rot && tid < 27)
    s_sct[tid] = make_float4(kSinCosTable[tid][0], kSinCosTable[tid][1], kSinCosTable[tid][2],
                             kSinCosTable[tid][3]);
  if (tid == 0) {
    s_bad = 0;
    s_count = 0;
    s_count_a = 0;
    s_count_b = 0;
    s_rank = 0;
    s_total_cost = 0;
    s_last = 0;
  }
  if (tid < kMaxChunks) {
    s_ccount[tid] = 0;
    s_ccount_a[tid] = 0;
    s_ccount_b[tid] = 0;
  }
  __syncthreads();
  // the ends of the index arrays, read by the last thread alongside the
  // sequences' entries below (one round trip for both)
  if (tid == kPlanThreads - 1) {
    const bool kv_bad = p.paged ? (p.page_indptr[0] != 0 || p.page_indptr[B] != p.nnz_pages)
                                : (p.kv_indptr[0] != 0 || p.kv_indptr[B] != p.total_kv);
    if (p.q_indptr[0] != 0 || p.mn_indptr[0] != 0 || kv_bad || p.q_indptr[B] != p.total_q ||
        p.mn_indptr[B] != p.total_tree)
      atomicOr(&s_bad, 1);
  }

  // ---- 1. the (sequence, q tile) pairs: every CTA walks the whole batch
  // (the ``advance_tile_batch`` walk of the page "_kernel_common.py", done up
  // front), validating the index arrays and counting pairs per cost
  const int per = (B + kPlanThreads - 1) / kPlanThreads;
  const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
  const bool split = p.max_chunks > 1;
  long long my_tiles = 0, my_seg = 0, my_cost = 0;
  int bad = 0;
  for (int b = b_lo; b < b_hi; ++b) {
    const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
    const int kv = seq_kv_len(p, b);
    const int tl = p.mn_indptr[b + 1] - p.mn_indptr[b];
    if (qo < 0 || tl < qo || kv < tl || seq_pages_bad(p, b)) {
      bad = 1;
      continue;
    }
    const int tiles = (qo + U - 1) / U;
    my_tiles += tiles;
    my_seg += (long long)tiles * seg_bytes(kv);
    for (int t = 0; t < tiles; ++t) {
      const int c = pair_tiles(qo, kv, U, t);
      if (split)
        my_cost += c;
      else
        atomicAdd(&s_hist[min(kCostBuckets - 1, c)], 1);
    }
  }
  if (bad) atomicOr(&s_bad, 1);
  if (split && my_cost) atomicAdd((unsigned long long*)&s_total_cost, (unsigned long long)my_cost);
  long long ex_tiles = my_tiles, ex_seg = my_seg, total_tiles, total_seg;
  exclusive_scan2(ex_tiles, ex_seg, total_tiles, total_seg, s_scan_a, s_scan_b, 0, kPlanThreads,
                  [] { __syncthreads(); });
  const bool ok = !s_bad && total_tiles <= p.max_pairs;
  const long long n_pairs = ok ? total_tiles : 0;
  // split-KV: every CTA derives the same chunking from the same totals, and
  // each pair adds its chunk count to the bucket of its chunks' cost
  const int chunk_tiles =
      !split ? 1 : (p.chunk_tiles > 0 ? p.chunk_tiles
                                      : auto_chunk_tiles(s_total_cost, p.h_kv, p.pipes));
  if (split) {
    for (int b = b_lo; b < b_hi; ++b) {
      const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
      const int kv = seq_kv_len(p, b);
      const int tl = p.mn_indptr[b + 1] - p.mn_indptr[b];
      if (qo < 0 || tl < qo || kv < tl || seq_pages_bad(p, b)) continue;
      const int tiles = (qo + U - 1) / U;
      for (int t = 0; t < tiles; ++t) {
        const int c = pair_tiles(qo, kv, U, t);
        const int nch = pair_chunks(c, chunk_tiles, p.max_chunks);
        atomicAdd(&s_hist[record_bucket(c, nch)], nch);
      }
    }
    __syncthreads();
  }

  // ---- 2. where each cost bucket starts in the longest-first order: the
  // pairs of higher cost come first
  {
    constexpr int per_t = kCostBuckets / kPlanThreads;
    long long sum = 0;
    for (int i = 0; i < per_t; ++i) sum += s_hist[kCostBuckets - 1 - (tid * per_t + i)];
    long long start = sum, dummy = 0, tot, tot2;
    exclusive_scan2(start, dummy, tot, tot2, s_scan_a, s_scan_b, 0, kPlanThreads,
                    [] { __syncthreads(); });
    for (int i = 0; i < per_t; ++i) {
      const int c = kCostBuckets - 1 - (tid * per_t + i);
      const int v = s_hist[c];
      s_hist[c] = (int)start;
      start += v;
    }
    // tot: the work records (one per pair, or one per chunk when split)
    if (blockIdx.x == 0 && tid == 0) {
      p.hdr->num_pairs = (unsigned int)n_pairs;
      p.hdr->num_items = ok ? (unsigned int)(tot * p.h_kv) : 0u;
      p.hdr->queue_head = 0;
      p.hdr->queue_done = 0;
      if (!ok) atomicOr(&p.hdr->error, DEVERR_BAD_INDPTR);
    }
  }

  // ---- 3. this CTA's pair and its place: the bucket's start plus the pairs
  // of the same cost earlier in (sequence, q tile) order
  const long long pair = blockIdx.x;
  if (ok && pair >= ex_tiles && pair < ex_tiles + my_tiles) {
    long long tcum = ex_tiles, scum = ex_seg;
    for (int b = b_lo; b < b_hi; ++b) {
      const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
      const int kv = seq_kv_len(p, b);
      const long long tiles = (qo + U - 1) / U;
      if (pair < tcum + tiles) {
        const int t = (int)(pair - tcum);
        s_pair_b = b;
        s_pair_t = t;
        s_pair_off = scum + (long long)t * seg_bytes(kv);
        const int c = pair_tiles(qo, kv, U, t);
        const int nch = pair_chunks(c, chunk_tiles, p.max_chunks);
        s_pair_chunks = nch;
        s_pair_cost = record_bucket(c, nch);
        break;
      }
      tcum += tiles;
      scum += tiles * seg_bytes(kv);
    }
  }
  __syncthreads();
  const bool has_pair = ok && pair < total_tiles;
  // the pair's q rows' enter indices, loaded now so that the round trip
  // overlaps the ranking below: threads 0-127 take tile A's rows, threads
  // 128-255 tile B's
  int key = INT_MAX, nrows = 0, n_a = 0, n_b = 0;
  // a pair whose only kv tile holds its own tree (no causal prefix) needs no
  // look-up: each of its Q tiles with rows sees at least its rows' own nodes
  // there, so the tile is PARTIAL for it (the softmax's per-column test
  // decides the rest; a FULL tile taken as PARTIAL gives the same result)
  bool one_tile = false;
  if (has_pair) {
    const int b = s_pair_b;
    const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
    const int tree_base = p.mn_indptr[b];
    const int tl = p.mn_indptr[b + 1] - tree_base;
    const int kv = seq_kv_len(p, b);
    one_tile = kv <= kBlockN && kv == tl && s_pair_chunks == 1;
    const int r0 = s_pair_t * U;
    nrows = min(U, qo - r0);
    n_a = min(R, nrows);
    n_b = nrows - n_a;
    const int grp = tid / kGroup, lt = tid % kGroup;
    if (!one_tile && lt < (grp ? n_b : n_a))
      key = p.tree_order[2 * (tree_base + r0 + grp * R + lt + tl - qo)];
  }
  if (has_pair) {
    // records of the same bucket that come earlier in (sequence, q tile) order
    const int pb = s_pair_b, pt = s_pair_t, pc = s_pair_cost;
    int cnt = 0;
    for (int b = b_lo; b < min(b_hi, pb + 1); ++b) {
      const int qo = p.q_indptr[b + 1] - p.q_indptr[b];
      const int kv = seq_kv_len(p, b);
      const int tiles = (qo + U - 1) / U;
      const int t_end = b < pb ? tiles : pt;
      for (int t = 0; t < t_end; ++t) {
        const int c = pair_tiles(qo, kv, U, t);
        const int nch = pair_chunks(c, chunk_tiles, p.max_chunks);
        cnt += record_bucket(c, nch) == pc ? nch : 0;
      }
    }
    if (cnt) atomicAdd(&s_rank, cnt);
  }
  __syncthreads();

  // ---- 4. classify the pair's kv tiles for both Q tiles (warps 0-3 sort
  // tile A's keys, warps 4-7 tile B's, then all warps take the columns) and
  // write its record
  if (has_pair) {
    const int b = s_pair_b, t = s_pair_t;
    const long long off = s_pair_off;
    const long long pos = (long long)s_hist[s_pair_cost] + s_rank;
    const int q0 = p.q_indptr[b];
    const int qo = p.q_indptr[b + 1] - q0;
    const int kv_base = seq_kv_base(p, b);
    const int kv = seq_kv_len(p, b);
    const int tree_base = p.mn_indptr[b];
    const int tl = p.mn_indptr[b + 1] - tree_base;
    const int ts = kv - tl;
    const int r0 = t * U;
    if (one_tile) {
      const uint8_t cls = (uint8_t)(kTilePartial | ((n_b > 0 ? kTilePartial : kTileEmpty) << 2));
      if (tid == 0) {
        p.classes[off] = cls;
        ItemRec r;
        r.part = -1;
        r.r0 = r0;
        r.q_row0 = q0 + r0;
        r.nq = nrows;
        r.qo = qo;
        r.kv = kv;
        r.tl = tl;
        r.tile_lo = 0;
        r.kv_base = kv_base;
        r.tree_base = tree_base;
        r.n_tiles = 1;
        r.class_off = (int32_t)off;
        r.kvt = 1;
        r.n_a = 1;
        r.n_b = n_b > 0 ? 1 : 0;
        r.cls = cls;
        p.sorted[pos] = r;
        if (p.merge) p.merge[pair] = make_int4(q0 + r0, nrows, 1, (int)pos);
      }
    } else {
    // exact classification from the DFS intervals of ``_check_tree_order``
    // (page "tree_attn.py"), for each Q tile of the unit: its rows' enter
    // indices are sorted (warps 0-3 tile A's, warps 4-7 tile B's: bitonic,
    // one key per thread); a kv column is seen by some row of a tile iff the
    // first key not below its enter index is below its exit index, and by
    // every row iff its interval holds the smallest and the largest key
    {
      const int grp = tid / kGroup, lt = tid % kGroup;
      const int ng = grp ? n_b : n_a;
      int* keys = s_keys + grp * kBlockM;
      if (ng <= 32) {
        // one warp, shuffles only
        if (lt < 32) {
          int x = key;
          for (int k = 2; k <= 32; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
              const int y = __shfl_xor_sync(0xffffffffu, x, j);
              const bool keep_min = ((lt & j) == 0) == ((lt & k) == 0);
              x = keep_min ? min(x, y) : max(x, y);
            }
          }
          keys[lt] = x;
        }
        group_sync(kBarA + grp);
      } else {
        keys[lt] = key;
        group_sync(kBarA + grp);
        for (int k = 2; k <= kBlockM; k <<= 1) {
          for (int j = k >> 1; j > 0; j >>= 1) {
            const int ixj = lt ^ j;
            if (ixj > lt) {
              const int a = keys[lt], c = keys[ixj];
              const bool up = (lt & k) == 0;
              if ((a > c) == up) {
                keys[lt] = c;
                keys[ixj] = a;
              }
            }
            group_sync(kBarA + grp);
          }
        }
      }
    }
    if (tid == 0) s_cls = 0;
    __syncthreads();
    const int* keys_a = s_keys;
    const int* keys_b = s_keys + kBlockM;
    const int kmin_a = keys_a[0], kmax_a = keys_a[n_a - 1];
    const int kmin_b = n_b > 0 ? keys_b[0] : 0, kmax_b = n_b > 0 ? keys_b[n_b - 1] : 0;
    const int kvt = (kv + kBlockN - 1) / kBlockN;
    // tiles wholly inside the causal prefix are FULL for every row (a pair
    // has at least one row, and such a tile ends at or before the tree
    // start, so it is not ragged): their columns need no look-up
    const int prefix_tiles = ts / kBlockN;
    // up to kPassTiles kv tiles per pass; every thread takes every 256th
    // column of the pass and folds its verdict into per-tile flags
    for (int j0 = 0; j0 < kvt; j0 += kPassTiles) {
      const int nt = min(kPassTiles, kvt - j0);
      for (int i = tid; i < nt; i += kPlanThreads) {
        s_any[0][i] = 0;
        s_notall[0][i] = 0;
        s_any[1][i] = 0;
        s_notall[1][i] = 0;
      }
      __syncthreads();
      const int c_end = min(kv, (j0 + nt) * kBlockN);
      // kColBatch columns per thread per step, their intervals loaded before
      // any is used, so that the loads' round trips overlap
      constexpr int kColBatch = 8;
      const int2* order2 = reinterpret_cast<const int2*>(p.tree_order) + tree_base;
      for (int c0 = max(j0, prefix_tiles) * kBlockN + tid; c0 < c_end;
           c0 += kPlanThreads * kColBatch) {
        int2 iv[kColBatch];
#pragma unroll
        for (int u = 0; u < kColBatch; ++u) {
          const int c = c0 + u * kPlanThreads;
          iv[u] = (c < c_end && c >= ts) ? order2[c - ts] : make_int2(0, 0);
        }
#pragma unroll
        for (int u = 0; u < kColBatch; ++u) {
          const int c = c0 + u * kPlanThreads;
          if (c >= c_end) break;
          // prefix columns (of the tile that holds the tree start) are seen by every row
          bool any_a = true, all_a = true, any_b = n_b > 0, all_b = true;
          if (c >= ts) {
            const int lo = lower_bound(keys_a, n_a, iv[u].x);
            any_a = lo < n_a && keys_a[lo] < iv[u].y;
            all_a = iv[u].x <= kmin_a && kmax_a < iv[u].y;
            if (n_b > 0) {
              const int lb = lower_bound(keys_b, n_b, iv[u].x);
              any_b = lb < n_b && keys_b[lb] < iv[u].y;
              all_b = iv[u].x <= kmin_b && kmax_b < iv[u].y;
            }
          }
          const int jt = c / kBlockN - j0;
          if (any_a && !s_any[0][jt]) s_any[0][jt] = 1;
          if (!all_a && !s_notall[0][jt]) s_notall[0][jt] = 1;
          if (any_b && !s_any[1][jt]) s_any[1][jt] = 1;
          if (!all_b && !s_notall[1][jt]) s_notall[1][jt] = 1;
        }
      }
      __syncthreads();
      for (int i = tid; i < nt; i += kPlanThreads) {
        const int j = j0 + i;
        const bool ragged = (j + 1) * kBlockN > kv;
        auto tile_cls = [&](int x) -> uint8_t {
          if (x == 1 && n_b == 0) return kTileEmpty;
          if (j < prefix_tiles) return kTileFull;
          if (!s_any[x][i]) return kTileEmpty;
          return (!s_notall[x][i] && !ragged) ? kTileFull : kTilePartial;
        };
        const uint8_t cls_a = tile_cls(0), cls_b = tile_cls(1);
        const uint8_t cls = (uint8_t)(cls_a | (cls_b << 2));
        p.classes[off + j] = cls;
        if (cls != kTileEmpty) {
          atomicAdd(&s_count, 1);
          if (split) atomicMax(&s_last, j + 1);
        }
        if (cls_a != kTileEmpty) atomicAdd(&s_count_a, 1);
        if (cls_b != kTileEmpty) atomicAdd(&s_count_b, 1);
        if (kvt <= kInlineTiles) atomicOr(&s_cls, (uint32_t)cls << (4 * j));
      }
      __syncthreads();
    }
    // split-KV: the tiles up to the last non-empty one are cut into nch
    // ranges of (nearly) equal length; each range's non-empty tiles are
    // counted from the classes just written (this CTA's own stores)
    const int nch = s_pair_chunks;
    const int last = s_last;
    if (nch > 1) {
      for (int j = tid; j < last; j += kPlanThreads) {
        const int cls = p.classes[off + j];
        if (cls == kTileEmpty) continue;
        int c = 0;
        while (c + 1 < nch && j >= (int)((long long)last * (c + 1) / nch)) ++c;
        atomicAdd(&s_ccount[c], 1);
        if (cls & 3) atomicAdd(&s_ccount_a[c], 1);
        if (cls >> 2) atomicAdd(&s_ccount_b[c], 1);
      }
      __syncthreads();
    }
    if (tid < nch) {
      ItemRec r;
      r.part = nch > 1 ? (int32_t)(pos + tid) : -1;
      r.r0 = r0;
      r.q_row0 = q0 + r0;
      r.nq = nrows;
      r.qo = qo;
      r.kv = kv;
      r.tl = tl;
      r.tile_lo = nch > 1 ? (int32_t)((long long)last * tid / nch) : 0;
      r.kv_base = kv_base;
      r.tree_base = tree_base;
      r.n_tiles = nch > 1 ? s_ccount[tid] : s_count;
      r.class_off = (int32_t)off;
      r.kvt = kvt;
      r.n_a = nch > 1 ? s_ccount_a[tid] : s_count_a;
      r.n_b = nch > 1 ? s_ccount_b[tid] : s_count_b;
      r.cls = s_cls;
      p.sorted[pos + tid] = r;
    }
    if (tid == 0 && p.merge)
      p.merge[pair] = make_int4(q0 + r0, nrows, nch, (int)pos);
    }
  }

  // ---- 5. (one-call entry points) the run's key rotation: every kv token's
  // cos/sin and rotated keys (rope_token), dealt out over the warps of the
  // grid, those of the CTAs without a pair first: the folded rotation is
  // small (fewer tokens than those warps, typically), so the classifying
  // CTAs take part only when it is not
  if (p.rot) {
    const long long grid = gridDim.x;
    const long long n_busy = ok ? min(total_tiles, grid) : 0;   // CTAs with a pair: 0..n_busy-1
    const long long idle_warps = (grid - n_busy) * 8;
    const long long rank = !has_pair ? ((long long)blockIdx.x - n_busy) * 8 + warp
                                     : idle_warps + (long long)blockIdx.x * 8 + warp;
    const long long nw = grid * 8;
    switch (p.rot) {
      case 1:
        rope_tokens<false, 64>(p.rot_k, p.rot_out, p.rot_pos, p.rot_cs, p.kp, s_sct, rank, nw, lane);
        break;
      case 2:
        rope_tokens<true, 64>(p.rot_k, p.rot_out, p.rot_pos, p.rot_cs, p.kp, s_sct, rank, nw, lane);
        break;
      case 3:
        rope_tokens<false, 128>(p.rot_k, p.rot_out, p.rot_pos, p.rot_cs, p.kp, s_sct, rank, nw,
                                lane);
        break;
      default:
        rope_tokens<true, 128>(p.rot_k, p.rot_out, p.rot_pos, p.rot_cs, p.kp, s_sct, rank, nw,
                               lane);
        break;
    }
  }
}

// The key-rotation kernel of the two-launch run (tree_attn_run): one warp per
// kv token at a time.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) krot_kernel(const uint32_t* __restrict__ k,
                                                   uint32_t* __restrict__ krot,
                                                   const int32_t* __restrict__ pos,
                                                   float4* __restrict__ cs,
                                                   const KrotParams kp) {
  __shared__ float4 s_sct[27];
  if (threadIdx.x < 27)
    s_sct[threadIdx.x] = make_float4(kSinCosTable[threadIdx.x][0], kSinCosTable[threadIdx.x][1],
                                     kSinCosTable[threadIdx.x][2], kSinCosTable[threadIdx.x][3]);
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  const long long rank = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  rope_tokens<BF16, D>(k, krot, pos, cs, kp, s_sct, rank, nwarps, threadIdx.x & 31);
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

cudaError_t launch_krot(const void* k, void* krot, const int32_t* rope_pos, float2* rope_cs,
                        const KrotParams& kp, int head_dim, bool bf16, int grid,
                        cudaStream_t stream) {
  if (kp.total_kv <= 0) return cudaSuccess;
  const uint32_t* kin = static_cast<const uint32_t*>(k);
  uint32_t* kout = static_cast<uint32_t*>(krot);
  float4* cs = reinterpret_cast<float4*>(rope_cs);
  if (head_dim == 128)
    return bf16 ? launch_pdl(krot_kernel<true, 128>, dim3(grid), dim3(256), 0, stream, kin, kout,
                             rope_pos, cs, kp)
                : launch_pdl(krot_kernel<false, 128>, dim3(grid), dim3(256), 0, stream, kin,
                             kout, rope_pos, cs, kp);
  return bf16 ? launch_pdl(krot_kernel<true, 64>, dim3(grid), dim3(256), 0, stream, kin, kout,
                           rope_pos, cs, kp)
              : launch_pdl(krot_kernel<false, 64>, dim3(grid), dim3(256), 0, stream, kin, kout,
                           rope_pos, cs, kp);
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
