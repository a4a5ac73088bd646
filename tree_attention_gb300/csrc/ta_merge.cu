// ta_merge.cu -- merging attention states over disjoint kv sets.
//
// The base-2 log-sum-exp that the ``lse_store`` epilogue of the page
// "tree_attn.py" emits (lse = m + log2(d)) is what makes attention over a kv
// set decomposable: for states (o_i, lse_i) over disjoint column sets,
//   lse = log2(sum_i 2^lse_i),   o = sum_i 2^(lse_i - lse) * o_i,
// with parts of lse = -inf (nothing visible) contributing nothing.  Two
// kernels apply it: the split-KV merge, which combines the float32 partial
// states the attention kernel left for the chunks of each split (sequence,
// q tile) pair, and a stand-alone merge of caller-provided states.
#include <cuda_runtime.h>

#include <cstdint>

#include "ta_device.cuh"
#include "ta_launch.h"

namespace ta {
namespace {

constexpr int kMergeThreads = 256;   // 8 warps, one row per warp at a time

template <int D>
struct RowVec;   // the D / 32 columns one lane holds
template <>
struct RowVec<128> {
  float v[4];
};
template <>
struct RowVec<64> {
  float v[2];
};

template <int D>
__device__ __forceinline__ RowVec<D> load_f32(const float* row, int lane) {
  RowVec<D> r;
  if constexpr (D == 128) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(row) + lane);
    r.v[0] = x.x;
    r.v[1] = x.y;
    r.v[2] = x.z;
    r.v[3] = x.w;
  } else {
    const float2 x = __ldg(reinterpret_cast<const float2*>(row) + lane);
    r.v[0] = x.x;
    r.v[1] = x.y;
  }
  return r;
}

template <int D, bool BF16>
__device__ __forceinline__ RowVec<D> load_half(const uint16_t* row, int lane) {
  RowVec<D> r;
  if constexpr (D == 128) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(row) + lane);
    const float2 a = unpack2<BF16>(x.x), b = unpack2<BF16>(x.y);
    r.v[0] = a.x;
    r.v[1] = a.y;
    r.v[2] = b.x;
    r.v[3] = b.y;
  } else {
    const float2 a = unpack2<BF16>(__ldg(reinterpret_cast<const uint32_t*>(row) + lane));
    r.v[0] = a.x;
    r.v[1] = a.y;
  }
  return r;
}

template <int D, bool BF16>
__device__ __forceinline__ void store_half(uint16_t* row, const float* v, int lane) {
  if constexpr (D == 128)
    reinterpret_cast<uint2*>(row)[lane] = make_uint2(pack2<BF16>(v[0], v[1]), pack2<BF16>(v[2], v[3]));
  else
    reinterpret_cast<uint32_t*>(row)[lane] = pack2<BF16>(v[0], v[1]);
}

// One row (one warp): ``lse_of(c)`` and ``o_of(c)`` give part c's lse and
// this lane's D / 32 columns of its output.  The lanes fetch 32 parts' lse
// at once and the parts' rows are loaded unconditionally (a part of lse
// -inf is then dropped by a select, so whatever its row holds never enters
// the sum).  Writes the merged row in the storage dtype and, from lane 0,
// its lse.
template <int D, bool BF16, typename LseOf, typename OOf>
__device__ __forceinline__ void merge_row(int n, LseOf lse_of, OOf o_of, uint16_t* out_row,
                                          float* lse_out, int lane) {
  constexpr int V = D / 32;
  float m = -INFINITY;
  for (int c0 = 0; c0 < n; c0 += 32)
    if (c0 + lane < n) m = fmaxf(m, lse_of(c0 + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float z = 0.f;
  if (m != -INFINITY) {
    for (int c0 = 0; c0 < n; c0 += 32) {
      const float lc = c0 + lane < n ? lse_of(c0 + lane) : -INFINITY;
      const float wl = lc == -INFINITY ? 0.f : exp2f(lc - m);
      z += wl;
      const int nb = min(32, n - c0);
#pragma unroll 4
      for (int j = 0; j < nb; ++j) {
        const float w = __shfl_sync(0xffffffffu, wl, j);
        const RowVec<D> o = o_of(c0 + j);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += w != 0.f ? w * o.v[i] : 0.f;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] *= inv;
  store_half<D, BF16>(out_row, acc, lane);
  if (lane == 0) *lse_out = z > 0.f ? m + log2f(z) : -INFINITY;
}

// merge_row for n <= kMax parts with every load of the row in flight at once:
// the lanes fetch the lses while all parts' rows are loaded into registers.
template <int D, bool BF16, int kMax, typename LseOf, typename OOf>
__device__ __forceinline__ void merge_row_few(int n, LseOf lse_of, OOf o_of, uint16_t* out_row,
                                              float* lse_out, int lane) {
  constexpr int V = D / 32;
  const float lc = lane < n ? lse_of(lane) : -INFINITY;
  RowVec<D> o[kMax];
#pragma unroll
  for (int c = 0; c < kMax; ++c)
    if (c < n) o[c] = o_of(c);
  float m = lc;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  const float wl = (m == -INFINITY || lc == -INFINITY) ? 0.f : exp2f(lc - m);
  float z = wl;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) z += __shfl_xor_sync(0xffffffffu, z, s);
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
  for (int c = 0; c < kMax; ++c) {
    if (c < n) {
      const float w = __shfl_sync(0xffffffffu, wl, c);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += w != 0.f ? w * o[c].v[i] : 0.f;
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] *= inv;
  store_half<D, BF16>(out_row, acc, lane);
  if (lane == 0) *lse_out = z > 0.f ? m + log2f(z) : -INFINITY;
}

// Split-KV merge: a unit is 8 packed rows of one (pair, kv head), one row per
// warp.  A pair's partial states hold its two Q tiles' 128 packed rows each
// (packed row = q row in the tile * g + head in the group, the row order of
// the attention kernel's tiles), tile A's first.
constexpr int kMergeRowsPerUnit = kMergeThreads / 32;
constexpr int kMergeRowsPerItem = kTilesPerUnit * kBlockM;
constexpr int kMergeUnitsPerItem = kMergeRowsPerItem / kMergeRowsPerUnit;
static_assert(kMaxChunks <= 32, "one lane per chunk's lse");

template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned int np = *(volatile const unsigned int*)&p.hdr->num_pairs;
  const long long n_pairs = (long long)np < p.max_pairs ? (long long)np : p.max_pairs;
  const long long units = n_pairs * p.h_kv * kMergeUnitsPerItem;
  const int g = p.g, R = kBlockM / p.g;
  uint16_t* outp = static_cast<uint16_t*>(p.out);
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int part8 = (int)(u % kMergeUnitsPerItem);
    const long long ph = u / kMergeUnitsPerItem;
    const int pair = (int)(ph / p.h_kv), kvh = (int)(ph % p.h_kv);
    const int4 mr = p.merge[pair];   // q_row0, q rows, chunks, first record
    if (mr.z <= 1 || mr.z > kMaxChunks || mr.w < 0 || (long long)mr.w + mr.z > p.max_records)
      continue;
    const int pr = part8 * kMergeRowsPerUnit + warp;
    const int tile = pr / kBlockM, local = pr % kBlockM;
    if (local >= R * g) continue;
    const int qr = tile * R + local / g, hh = local % g;
    if (qr >= mr.y) continue;
    const size_t orow = (size_t)(mr.x + qr) * p.h_q + (size_t)kvh * g + hh;
    auto slot = [&](int c) {
      return (((size_t)(mr.w + c)) * p.h_kv + kvh) * kMergeRowsPerItem + pr;
    };
    merge_row_few<D, BF16, kMaxChunks>(
        mr.z, [&](int c) { return __ldg(p.part_lse + slot(c)); },
        [&](int c) { return load_f32<D>(p.part_o + slot(c) * D, lane); }, outp + orow * D,
        p.lse + orow, lane);
  }
}

// Stand-alone merge: parts [n][rows][D] in the storage dtype, lses [n][rows].
template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeThreads)
    merge_states_kernel(const uint16_t* __restrict__ parts, const float* __restrict__ lses,
                        int n, long long rows, uint16_t* __restrict__ out,
                        float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  for (long long row = (long long)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    auto lse_of = [&](int c) { return __ldg(lses + (size_t)c * rows + row); };
    auto o_of = [&](int c) { return load_half<D, BF16>(parts + ((size_t)c * rows + row) * D, lane); };
    if (n <= 8)
      merge_row_few<D, BF16, 8>(n, lse_of, o_of, out + row * D, lse + row, lane);
    else
      merge_row<D, BF16>(n, lse_of, o_of, out + row * D, lse + row, lane);
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int head_dim, bool bf16, int grid,
                         cudaStream_t stream) {
  const dim3 g(grid), b(kMergeThreads);
  if (head_dim == 128)
    return bf16 ? launch_pdl(merge_kernel<128, true>, g, b, 0, stream, p)
                : launch_pdl(merge_kernel<128, false>, g, b, 0, stream, p);
  return bf16 ? launch_pdl(merge_kernel<64, true>, g, b, 0, stream, p)
              : launch_pdl(merge_kernel<64, false>, g, b, 0, stream, p);
}

cudaError_t launch_merge_states(const void* parts, const float* lses, int n_parts,
                                long long rows, int head_dim, bool bf16, void* out, float* lse,
                                int grid, cudaStream_t stream) {
  const uint16_t* in = static_cast<const uint16_t*>(parts);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (head_dim == 128) {
    if (bf16)
      merge_states_kernel<128, true><<<grid, kMergeThreads, 0, stream>>>(in, lses, n_parts, rows, o, lse);
    else
      merge_states_kernel<128, false><<<grid, kMergeThreads, 0, stream>>>(in, lses, n_parts, rows, o, lse);
  } else {
    if (bf16)
      merge_states_kernel<64, true><<<grid, kMergeThreads, 0, stream>>>(in, lses, n_parts, rows, o, lse);
    else
      merge_states_kernel<64, false><<<grid, kMergeThreads, 0, stream>>>(in, lses, n_parts, rows, o, lse);
  }
  return cudaGetLastError();
}

}  // namespace ta
