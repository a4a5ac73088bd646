// ta_attn.cu -- persistent batched tree-attention kernel for sm_103a.
//
// Computes what ``batch_tree_attn`` of the page "tree_attn.py" computes
// (per q row and head: masked online softmax of sm_scale * q.k in log2
// units, output O / d and lse = m + log2(d)), re-designed for one GB300 SM.
//
// Each CTA runs two independent pipelines side by side (so that one hides
// the other's latencies); both pop (sequence, q tile, kv head) work items
// from one longest-first queue.  A pipeline is six warps:
//   producer   stages the item's work, TMA-loads the packed Q tile and the
//              item's non-empty K/V tiles (64 kv rows each) into a 2-stage
//              ring, with each partial tile's column intervals beside it
//   MMA        one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//              score buffers, then O += P V with P read from TMEM
//   softmax    four warps, one TMEM lane (= packed row) per thread: inline
//              RoPE of the Q tile, tree mask, online softmax with a lazily
//              moved reference max, P (fp16/bf16) written over its own score
//              buffer in TMEM, O rescale, final O / l and lse stores
// Keys arrive rotated (the run rotates them once per call).  Every cross-warp
// hand-off is an mbarrier with a bounded wait.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ta_device.cuh"
#include "ta_launch.h"

namespace ta {
namespace {

constexpr int kPipes = 2;
constexpr int kWarpsPerPipe = 6;
constexpr int kThreads = kPipes * kWarpsPerPipe * 32;
constexpr int kStages = 2;   // K/V ring depth per pipeline
constexpr int kSlots = 2;    // work-item slots per pipeline

enum Bar : int {
  B_ITEM_FULL = 0,                       // [kSlots]
  B_ITEM_EMPTY = B_ITEM_FULL + kSlots,   // [kSlots]
  B_Q_FULL = B_ITEM_EMPTY + kSlots,
  B_Q_READY,
  B_Q_EMPTY,
  B_K_FULL,                              // [kStages]
  B_V_FULL = B_K_FULL + kStages,         // [kStages]
  B_EX_FULL = B_V_FULL + kStages,        // [kStages]
  // a K (V) stage is free again when the QK (PV) of the tile in it has
  // completed: with two stages and two score buffers, tile c uses stage and
  // buffer c & 1, so the producer waits on S_FULL (PV_DONE) of that index
  // and the MMA thread commits nothing extra per tile
  B_S_FULL = B_EX_FULL + kStages,        // [2] score buffer written (K stage read)
  B_P_FULL = B_S_FULL + 2,               // [2] P written over the score buffer
  B_PV_DONE = B_P_FULL + 2,              // [2] PV reading that P is complete (V stage read)
  B_O_FREE = B_PV_DONE + 2,
  B_DRAIN,
  B_STALL,                               // test hook: nothing ever arrives on it
  B_COUNT
};

struct Item {
  ItemRec r;
  int valid, kvh, pad[14];
};
static_assert(sizeof(Item) == 128, "item slot size");

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;               // 128-byte column blocks per row
  static constexpr int kQAtomBytes = kBlockM * 128;    // 128 rows x 128 bytes
  static constexpr int kKVAtomBytes = kBlockN * 128;   // 64 rows x 128 bytes
  static constexpr int kQBytes = kAtoms * kQAtomBytes;
  static constexpr int kKVBytes = kAtoms * kKVAtomBytes;
  static constexpr int kOstBytes = 32 * 64;            // per softmax warp: 32 rows x 64 bytes
  // one pipeline's shared memory
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffEX = kOffV + kStages * kKVBytes;    // [kStages][kBlockN] int2
  static constexpr int kOffOst = kOffEX + kStages * kBlockN * 8;
  static constexpr int kOffItems = kOffOst + 4 * kOstBytes;
  static constexpr int kOffBar = kOffItems + kSlots * (int)sizeof(Item);
  static constexpr int kPipeUsed = kOffBar + 32 * 8;
  static constexpr int kPipeBytes = (kPipeUsed + 1023) / 1024 * 1024;
  // CTA-wide: TMEM address and abort flag after both pipelines
  static constexpr int kOffCta = kPipes * kPipeBytes;
  static constexpr int kSmemAlloc = kOffCta + 128 + 1024;   // room to align the base to 1024
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemPipe = 256;   // columns per pipeline
  static constexpr uint32_t kTmemO = 0;        // accumulator
  static constexpr uint32_t kTmemS = 128;      // score buffer sb at 128 + 64 * sb (P over it)
};

struct CtaShared {
  uint32_t tmem_base;
  int abort;
};

struct Pipe {
  uint8_t* smem;     // this pipeline's shared memory
  uint64_t* bar;
  Item* items;
  volatile int* abort;
  unsigned int* dev_error;
  unsigned long long limit_ns;
  uint32_t tmem;     // this pipeline's first TMEM column (lane 0)
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait(&bar[b], parity, abort, dev_error, limit_ns);
  }
  // every lane of the warp waits; the warp proceeds only if all lanes saw it
  __device__ bool warp_wait(int b, uint32_t parity) const {
    const bool ok = mbar_wait(&bar[b], parity, abort, dev_error, limit_ns);
    return __all_sync(0xffffffffu, ok);
  }
  // wait used while draining after an abort: ignores the abort flag
  __device__ bool drain_wait(int b, uint32_t parity) const {
    int no_abort = 0;
    return mbar_wait(&bar[b], parity, &no_abort, dev_error, 200000000ull);
  }
};

// Iterates the non-empty kv tiles of a work item from its first tile
// (tile_lo, past 0 for a split-KV chunk): from the record's inline 2-bit
// classes for short sequences, else from the plan's class bytes.
struct TileIter {
  const uint8_t* cls;
  int kvt, j;
  bool inl;
  uint32_t w0, w1, w2, w3;   // inline classes, or the current 16 class bytes
  __device__ TileIter(const ItemRec& r, const uint8_t* classes)
      : cls(classes + r.class_off), kvt(r.kvt), j(r.tile_lo - 1), inl(r.kvt <= kInlineTiles) {
    w0 = r.cls2[0];
    w1 = r.cls2[1];
    w2 = r.cls2[2];
    w3 = 0;
    if (!inl && (r.tile_lo & 15)) {
      // a range that starts inside a 16-tile group: load that group now
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(cls + (r.tile_lo & ~15)));
      w0 = v.x;
      w1 = v.y;
      w2 = v.z;
      w3 = v.w;
    }
  }
  // advances to the next non-empty tile; returns its class (0 when done)
  __device__ int next() {
    while (true) {
      ++j;
      if (j >= kvt) return 0;
      int c;
      if (inl) {
        const uint32_t w = j < 16 ? w0 : (j < 32 ? w1 : w2);
        c = (w >> (2 * (j & 15))) & 3;
      } else {
        if ((j & 15) == 0) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(cls + j));
          w0 = v.x;
          w1 = v.y;
          w2 = v.z;
          w3 = v.w;
        }
        const int q = (j & 15) >> 2;
        const uint32_t w = q == 0 ? w0 : (q == 1 ? w1 : (q == 2 ? w2 : w3));
        c = (w >> (8 * (j & 3))) & 0xff;
      }
      if (c != kTileEmpty) return c;
    }
  }
};

// ---------------------------------------------------------------------------
// producer warp (lane 0 issues; all lanes stage mask intervals)
// ---------------------------------------------------------------------------
template <int D, bool PAGED>
__device__ void run_producer(const Pipe& pp, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const AttnParams& p, int pipe, int lane) {
  using C = Cfg<D>;
  uint8_t* sQ = pp.smem + C::kOffQ;
  uint8_t* sK = pp.smem + C::kOffK;
  uint8_t* sV = pp.smem + C::kOffV;
  int2* sEX = reinterpret_cast<int2*>(pp.smem + C::kOffEX);
  // the plan kernel wrote the item count; never trust it beyond the table size
  const unsigned long long cap = (unsigned long long)p.max_records * (unsigned long long)p.h_kv;
  const unsigned long long n_items = *(volatile unsigned int*)&p.hdr->num_items;
  const unsigned int num_items = (unsigned int)(n_items < cap ? n_items : cap);
  const int g = p.g, R = p.R;
  uint32_t it = 0, kv_it = 0, q_it = 0;
  uint32_t issued_k = 0, issued_v = 0;   // loads issued (stage = count % kStages)
  bool aborted = false;
  // the first item of every pipeline is fixed (pipeline p of CTA b takes
  // item 2b + p, the items being in longest-first order already), the rest
  // come from the queue, which starts after those 2 x grid items
  const unsigned int n_static = (unsigned int)(kPipes * gridDim.x);
  unsigned int idx = (unsigned int)(kPipes * blockIdx.x + pipe);
  // lanes 0-3 hold the next record (16 bytes each), fetched one item ahead
  int4 rec_next = make_int4(0, 0, 0, 0);
  if (idx < num_items && lane < 4)
    rec_next = __ldg(reinterpret_cast<const int4*>(p.sorted + idx / p.h_kv) + lane);
  for (;;) {
    const int slot = it % kSlots;
    if (!pp.warp_wait(B_ITEM_EMPTY + slot, ((it / kSlots) & 1) ^ 1)) { aborted = true; break; }
    Item& s = pp.items[slot];
    if (idx >= num_items) {
      if (lane == 0) {
        s.valid = 0;
        mbar_arrive(&pp.bar[B_ITEM_FULL + slot]);
      }
      break;
    }
    if (lane < 4) reinterpret_cast<int4*>(&s.r)[lane] = rec_next;
    const int kvh = idx % p.h_kv;
    // pop the next index now; its round trip overlaps this item's issue
    unsigned int nidx = 0;
    if (lane == 0) {
      nidx = n_static + atomicAdd(&p.hdr->queue_head, 1u);
      s.valid = 1;
      s.kvh = kvh;
    }
    __syncwarp();
    const ItemRec r = s.r;
    if (lane == 0) mbar_arrive(&pp.bar[B_ITEM_FULL + slot]);
    if (r.n_tiles > 0) {
      if (!pp.warp_wait(B_Q_EMPTY, (q_it & 1) ^ 1)) { aborted = true; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&pp.bar[B_Q_FULL], (uint32_t)(C::kAtoms * 128 * g * R));
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d(sQ + a * C::kQAtomBytes, tm_q, &pp.bar[B_Q_FULL], a * 64, kvh * g,
                      r.q_row0);
      }
      ++q_it;
      TileIter ti(r, p.classes);
      for (int n = 0; n < r.n_tiles; ++n) {
        const int cls = ti.next();
        const int j = ti.j;
        const int row0 = r.kv_base + j * kBlockN;
        const int stage = kv_it % kStages;
        const uint32_t empty_par = ((kv_it / kStages) & 1) ^ 1;
        const uint32_t bytes = (uint32_t)C::kKVBytes;
        // paged cache: kv tile j is logical pages 4j .. 4j+3 of the sequence;
        // lanes 0-3 look up their physical pages, a missing page (past the
        // sequence's last) takes an out-of-range page index, read as zeros
        int ph0 = 0, ph1 = 0, ph2 = 0, ph3 = 0;
        if constexpr (PAGED) {
          const int np = (r.kv + kPageSize - 1) / kPageSize;
          const int lp = j * (kBlockN / kPageSize) + lane;
          int phys = p.num_pages;
          if (lane < kBlockN / kPageSize && lp < np) phys = __ldg(p.page_values + r.kv_base + lp);
          ph0 = __shfl_sync(0xffffffffu, phys, 0);
          ph1 = __shfl_sync(0xffffffffu, phys, 1);
          ph2 = __shfl_sync(0xffffffffu, phys, 2);
          ph3 = __shfl_sync(0xffffffffu, phys, 3);
        }
        // one K or V tile into ``dst`` (kv plane 0 = K, 1 = V of the paged cache)
        auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int plane) {
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a) {
            if constexpr (PAGED) {
              const int phs[4] = {ph0, ph1, ph2, ph3};
#pragma unroll
              for (int q = 0; q < kBlockN / kPageSize; ++q)
                tma_load_5d(dst + a * C::kKVAtomBytes + q * kPageSize * 128, map, bar, a * 64, 0,
                            kvh, plane, phs[q]);
            } else {
              tma_load_3d(dst + a * C::kKVAtomBytes, map, bar, a * 64, kvh, row0);
            }
          }
        };
        if (!pp.warp_wait(B_S_FULL + stage, empty_par)) { aborted = true; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&pp.bar[B_K_FULL + stage], bytes);
          load_tile(sK + stage * C::kKVBytes, tm_k, &pp.bar[B_K_FULL + stage], 0);
        }
        ++issued_k;
        if (!pp.warp_wait(B_PV_DONE + stage, empty_par)) { aborted = true; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&pp.bar[B_V_FULL + stage], bytes);
          load_tile(sV + stage * C::kKVBytes, tm_v, &pp.bar[B_V_FULL + stage], 1);
        }
        ++issued_v;
        // column intervals of a partial tile for the mask (FULL tiles need none)
        if (cls == kTilePartial) {
          int2* ex = sEX + stage * kBlockN;
#pragma unroll
          for (int q = 0; q < kBlockN / 32; ++q)
            ex[q * 32 + lane] =
                column_interval(p.tree_order, r.tree_base, j * kBlockN + q * 32 + lane, r.kv,
                                r.kv - r.tl);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pp.bar[B_EX_FULL + stage]);
        ++kv_it;
      }
      if (aborted) break;
    }
    idx = __shfl_sync(0xffffffffu, nidx, 0);
    if (idx < num_items && lane < 4)
      rec_next = __ldg(reinterpret_cast<const int4*>(p.sorted + idx / p.h_kv) + lane);
    ++it;
  }
  if (aborted && lane == 0) {
    // let every copy already in flight land before the CTA's memory goes away
    if (q_it > 0) pp.drain_wait(B_Q_FULL, (q_it - 1) & 1);
    // the last load issued into each stage: load i went to stage i % kStages
    // and completes that stage's phase i / kStages
    for (uint32_t i = issued_k > kStages ? issued_k - kStages : 0; i < issued_k; ++i)
      pp.drain_wait(B_K_FULL + i % kStages, (i / kStages) & 1);
    for (uint32_t i = issued_v > kStages ? issued_v - kStages : 0; i < issued_v; ++i)
      pp.drain_wait(B_V_FULL + i % kStages, (i / kStages) & 1);
  }
}

// ---------------------------------------------------------------------------
// MMA warp (one thread)
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__device__ void run_mma(const Pipe& pp, const AttnParams& p) {
  using C = Cfg<D>;
  // descriptors of k-step 0; a k-step or stage offset is added to the
  // descriptor's 14-bit start-address field (addresses stay below 256 KB)
  static_assert(kStages == 2, "descriptor selection below assumes two stages");
  const uint64_t dq0 = sw128_desc(smem_u32(pp.smem + C::kOffQ), 0);
  const uint64_t dk_s0 = sw128_desc(smem_u32(pp.smem + C::kOffK), 0);
  const uint64_t dk_s1 = dk_s0 + (uint64_t)(C::kKVBytes >> 4);
  const uint64_t dv_s0 = sw128_desc(smem_u32(pp.smem + C::kOffV), C::kKVAtomBytes);
  const uint64_t dv_s1 = dv_s0 + (uint64_t)(C::kKVBytes >> 4);
  constexpr uint32_t idesc_pv = umma_idesc_f16(BF16, 128, D, /*b_mn_major=*/true);
  const int q_bar = p.rotary ? B_Q_READY : B_Q_FULL;
  uint32_t it = 0, kv_it = 0, q_it = 0, o_it = 0;
  bool issued_any = false;
  // test hook: a wait that runs out before any MMA is issued (the other warps
  // then find the abort flag in their own waits)
  if (p.debug_stall) pp.wait(B_STALL, 0);
  for (; !p.debug_stall;) {
    const int slot = it % kSlots;
    if (!pp.wait(B_ITEM_FULL + slot, (it / kSlots) & 1)) break;
    const Item& s = pp.items[slot];
    if (!s.valid) break;
    const ItemRec r = s.r;
    if (r.n_tiles > 0) {
      if (!pp.wait(q_bar, q_it & 1)) break;
      ++q_it;
      tc_fence_after();
      TileIter ti(r, p.classes);
      bool ok = true;
      // S(c) = Q K(c)^T into score buffer c & 1, once the PV that read the P
      // of tile c - 2 out of that buffer has completed
      auto issue_qk = [&](int m, int nvalid) -> bool {
        const uint32_t c = kv_it + m;
        const int stage = c % kStages;
        if (c >= 2 && !pp.wait(B_PV_DONE + (c & 1), ((c - 2) >> 1) & 1)) return false;
        if (!pp.wait(B_K_FULL + stage, (c / kStages) & 1)) return false;
        tc_fence_after();
        const int sb = c & 1;
        const int n_eff = (nvalid + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(BF16, 128, n_eff, false);
        const uint64_t dk = stage ? dk_s1 : dk_s0;
        const uint32_t d_s = pp.tmem + C::kTmemS + 64 * sb;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qo = (uint32_t)(((k >> 2) * C::kQAtomBytes + (k & 3) * 32) >> 4);
          const uint32_t ko = (uint32_t)(((k >> 2) * C::kKVAtomBytes + (k & 3) * 32) >> 4);
          umma_f16(d_s, dq0 + qo, dk + ko, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&pp.bar[B_S_FULL + sb]);
        issued_any = true;
        if (m == r.n_tiles - 1) umma_commit(&pp.bar[B_Q_EMPTY]);
        return true;
      };
      ti.next();
      int nv_cur = min(kBlockN, r.kv - ti.j * kBlockN);
      int nv_next = 0;
      if (!issue_qk(0, nv_cur)) break;
      for (int n = 0; n < r.n_tiles; ++n) {
        if (n + 1 < r.n_tiles) {
          ti.next();
          nv_next = min(kBlockN, r.kv - ti.j * kBlockN);
          if (!issue_qk(n + 1, nv_next)) { ok = false; break; }
        }
        const uint32_t c = kv_it + n;
        const int stage = c % kStages;
        const int pb = c & 1;
        if (!pp.wait(B_P_FULL + pb, (c >> 1) & 1)) { ok = false; break; }
        if (!pp.wait(B_V_FULL + stage, (c / kStages) & 1)) { ok = false; break; }
        if (n == 0) {
          if (!pp.wait(B_O_FREE, (o_it & 1) ^ 1)) { ok = false; break; }
          ++o_it;
        }
        tc_fence_after();
        const int nk = (nv_cur + 15) >> 4;   // 16-row k-steps holding valid kv rows
        const uint64_t dv = stage ? dv_s1 : dv_s0;
        const uint32_t pcol = pp.tmem + C::kTmemS + 64 * pb;   // P: two elements per column
#pragma unroll
        for (int k = 0; k < kBlockN / 16; ++k) {
          if (k < nk)
            umma_f16_tmem_a(pp.tmem + C::kTmemO, pcol + k * 8, dv + (uint64_t)(k * 16 * 128 >> 4),
                            idesc_pv, (n > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&pp.bar[B_PV_DONE + pb]);
        nv_cur = nv_next;
      }
      if (!ok) break;
      kv_it += r.n_tiles;
    }
    mbar_arrive(&pp.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
  if (*pp.abort && issued_any) {
    umma_commit(&pp.bar[B_DRAIN]);
    pp.drain_wait(B_DRAIN, 0);
  }
}

// ---------------------------------------------------------------------------
// softmax warps: RoPE on Q, softmax, O correction, epilogue
// ---------------------------------------------------------------------------
// Inline RoPE of this warp's 32 packed rows of the Q tile.  Task = (q row,
// 16-byte block c of the first half of the head dimension): one load of the
// row's cos/sin for that block, applied to the block and its partner block in
// the second half, for each of the q row's heads that lie in these 32 rows.
// Tasks are taken 64 at a time (two per lane); rope_load issues the loads of
// one batch so that the first batch can be fetched before the Q tile lands.
struct RopeRange {
  int row_lo, row_hi, qr_lo, ntask;
};

template <int D>
__device__ __forceinline__ RopeRange rope_range(int nq, int g, int wq) {
  constexpr int kHalfChunks = D / 16;  // 16-byte blocks in half a row
  RopeRange rr;
  rr.row_lo = wq * 32;
  rr.row_hi = rr.row_lo + 32;
  rr.qr_lo = rr.row_lo / g;
  const int qr_hi = min(nq, (rr.row_hi + g - 1) / g);   // q rows touching this quadrant
  rr.ntask = max(0, qr_hi - rr.qr_lo) * kHalfChunks;
  return rr;
}

template <int D>
__device__ __forceinline__ void rope_load(float4 (&cv)[2][4], const float2* __restrict__ cs,
                                          long long tok0, const RopeRange& rr, int t0, int lane) {
  constexpr int kHalfChunks = D / 16;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int task = t0 + u * 32 + lane;
    if (task < rr.ntask) {
      const int qr = rr.qr_lo + task / kHalfChunks, c = task % kHalfChunks;
      const float4* csp = reinterpret_cast<const float4*>(cs + (tok0 + qr) * (D / 2) + c * 8);
#pragma unroll
      for (int i = 0; i < 4; ++i) cv[u][i] = __ldg(csp + i);
    }
  }
}

// Applies the rotation with the first batch already in ``cv``.
template <int D, bool BF16>
__device__ void rope_q_rows(uint8_t* tile, const float2* __restrict__ cs, long long tok0,
                            const RopeRange& rr, int g, int lane, float4 (&cv)[2][4]) {
  constexpr int kHalfChunks = D / 16;
  for (int t0 = 0; t0 < rr.ntask; t0 += 64) {
    if (t0 > 0) rope_load<D>(cv, cs, tok0, rr, t0, lane);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int task = t0 + u * 32 + lane;
      if (task >= rr.ntask) continue;
      const int qr = rr.qr_lo + task / kHalfChunks, c = task % kHalfChunks;
      const int h_lo = max(0, rr.row_lo - qr * g), h_hi = min(g, rr.row_hi - qr * g);
      for (int h = h_lo; h < h_hi; ++h) {
        const int row = qr * g + h;
        uint8_t* lo;
        uint8_t* hi;
        if constexpr (D == 128) {
          lo = tile + row * 128 + ((c ^ (row & 7)) * 16);
          hi = tile + kBlockM * 128 + row * 128 + ((c ^ (row & 7)) * 16);
        } else {
          lo = tile + row * 128 + ((c ^ (row & 7)) * 16);
          hi = tile + row * 128 + (((c + 4) ^ (row & 7)) * 16);
        }
        const uint4 a = *reinterpret_cast<const uint4*>(lo);
        const uint4 b = *reinterpret_cast<const uint4*>(hi);
        const uint32_t au[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bu[4] = {b.x, b.y, b.z, b.w};
        uint32_t ao[4], bo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 x0 = unpack2<BF16>(au[i]);
          const float2 x1 = unpack2<BF16>(bu[i]);
          const float c0 = cv[u][i].x, s0 = cv[u][i].y, c1 = cv[u][i].z, s1 = cv[u][i].w;
          // first half: cos*x[j] + sin*(-x[j+d/2]); second half: cos*x[j] + sin*x[j-d/2]
          const float y0a = __fadd_rn(__fmul_rn(c0, x0.x), __fmul_rn(s0, -x1.x));
          const float y0b = __fadd_rn(__fmul_rn(c1, x0.y), __fmul_rn(s1, -x1.y));
          const float y1a = __fadd_rn(__fmul_rn(c0, x1.x), __fmul_rn(s0, x0.x));
          const float y1b = __fadd_rn(__fmul_rn(c1, x1.y), __fmul_rn(s1, x0.y));
          ao[i] = pack2<BF16>(y0a, y0b);
          bo[i] = pack2<BF16>(y1a, y1b);
        }
        *reinterpret_cast<uint4*>(lo) = make_uint4(ao[0], ao[1], ao[2], ao[3]);
        *reinterpret_cast<uint4*>(hi) = make_uint4(bo[0], bo[1], bo[2], bo[3]);
      }
    }
  }
}

template <int D, bool BF16, bool PAGED>
__device__ void softmax_loop(const Pipe& pp, const AttnParams& p, int sw, int lane);

// The softmax warps' loop; on every way out (the work is done, or a bounded
// wait gave up) the warp waits for its own TMEM loads and stores to finish
// before the CTA frees the TMEM.
template <int D, bool BF16, bool PAGED>
__device__ void run_softmax(const Pipe& pp, const AttnParams& p, int sw, int lane) {
  softmax_loop<D, BF16, PAGED>(pp, p, sw, lane);
  tmem_wait_ld();
  tmem_wait_st();
}

template <int D, bool BF16, bool PAGED>
__device__ void softmax_loop(const Pipe& pp, const AttnParams& p, int sw, int lane) {
  using C = Cfg<D>;
  const int wq = sw;                          // TMEM lane quadrant (warp index mod 4)
  const int row = wq * 32 + lane;             // packed row = TMEM lane
  const uint32_t t_row = pp.tmem + ((uint32_t)(wq * 32) << 16);
  const int2* sEX = reinterpret_cast<const int2*>(pp.smem + C::kOffEX);
  uint8_t* ost = pp.smem + C::kOffOst + wq * C::kOstBytes;
  const float c2 = p.scale_log2;
  const int g = p.g, R = p.R;
  const bool in_pack = row < g * R;
  const int qr = in_pack ? row / g : 0;
  const int hh = in_pack ? row - qr * g : 0;
  uint32_t it = 0, gi = 0, q_it = 0;  // gi: kv tiles processed by this pipeline
  for (;;) {
    const int slot = it % kSlots;
    if (!pp.warp_wait(B_ITEM_FULL + slot, (it / kSlots) & 1)) return;
    const Item& s = pp.items[slot];
    if (!s.valid) return;
    const ItemRec r = s.r;
    const int kvh = s.kvh;
    const bool valid = in_pack && qr < r.nq;
    const int head = kvh * g + hh;
    const size_t orow = (size_t)(r.q_row0 + qr) * p.h_q + head;
    int e_row = INT_MIN;
    if (valid) e_row = __ldg(&p.tree_order[2 * (r.tree_base + r.t * R + qr + r.tl - r.qo)]);
    float m_ref = -INFINITY, l = 0.f;
    if (r.n_tiles > 0) {
      if (p.rotary) {
        // q row r of the tile takes the position of its own tree node's kv
        // slot (the first cos/sin batch is fetched while the Q tile lands)
        const long long qtok0 = (long long)r.kv_base + (r.kv - r.qo) + (long long)r.t * R;
        const RopeRange rr = rope_range<D>(r.nq, g, wq);
        float4 cv[2][4];
        rope_load<D>(cv, p.rope_cs, qtok0, rr, 0, lane);
        if (!pp.warp_wait(B_Q_FULL, q_it & 1)) return;
        rope_q_rows<D, BF16>(pp.smem + C::kOffQ, p.rope_cs, qtok0, rr, g, lane, cv);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pp.bar[B_Q_READY]);
      }
      ++q_it;
      TileIter ti(r, p.classes);
      for (int n = 0; n < r.n_tiles; ++n, ++gi) {
        const int cls = ti.next();
        const int nvalid = min(kBlockN, r.kv - ti.j * kBlockN);
        const int stage = gi % kStages;
        const int sb = gi & 1;
        // visibility bits of this row for the tile's 64 columns
        uint32_t mw0, mw1;
        if (cls == kTilePartial) {
          if (!pp.warp_wait(B_EX_FULL + stage, (gi / kStages) & 1)) return;
          const int4* e4 = reinterpret_cast<const int4*>(sEX + stage * kBlockN);
          mw0 = 0;
          mw1 = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int4 a = e4[i], b = e4[16 + i];
            mw0 |= (uint32_t)(a.x <= e_row && e_row < a.y) << (2 * i);
            mw0 |= (uint32_t)(a.z <= e_row && e_row < a.w) << (2 * i + 1);
            mw1 |= (uint32_t)(b.x <= e_row && e_row < b.y) << (2 * i);
            mw1 |= (uint32_t)(b.z <= e_row && e_row < b.w) << (2 * i + 1);
          }
        } else {
          mw0 = mw1 = 0xffffffffu;  // FULL tiles are never ragged
        }
        if (!pp.warp_wait(B_S_FULL + sb, (gi >> 1) & 1)) return;
        tc_fence_after();
        const uint32_t t_s = t_row + C::kTmemS + 64 * sb;
        // the whole 64-column score row in registers: one TMEM round trip
        float v[64];
        {
          float a[32], b[32];
          tmem_ld32(t_s, a);
          if (nvalid > 32) tmem_ld32(t_s + 32, b);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = a[i];
            v[32 + i] = nvalid > 32 ? b[i] : 0.f;
          }
        }
        // masked row max in log2 units (eight independent chains)
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
        if (cls == kTileFull) {
#pragma unroll
          for (int i = 0; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], v[i] * c2);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const uint32_t bit = i < 32 ? (mw0 >> i) & 1u : (mw1 >> (i - 32)) & 1u;
            if (bit) mx8[i & 7] = fmaxf(mx8[i & 7], v[i] * c2);
          }
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // move the reference max only when it grew by more than 2^8; the
        // final O / l and lse = m + log2(l) do not depend on the reference
        const float m_new = fmaxf(m_ref, mx);
        float ref = m_ref;
        if (m_new > m_ref + 8.f) ref = m_new;
        const float alpha = (ref == m_ref) ? 1.f : ex2_approx(m_ref - ref);
        m_ref = ref;
        const float m_use = (ref == -INFINITY) ? 0.f : ref;
        // P = exp2(s * c2 - m) on visible columns, packed two per 32-bit word
        float l8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) l8[k] = 0.f;
        float pk[32];
        if (cls == kTileFull) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = ex2_approx(fmaf(v[2 * i], c2, -m_use));
            const float p1 = ex2_approx(fmaf(v[2 * i + 1], c2, -m_use));
            l8[i & 7] += p0 + p1;
            pk[i] = __uint_as_float(pack2<BF16>(p0, p1));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int i0 = 2 * i, i1 = 2 * i + 1;
            const uint32_t b0 = i0 < 32 ? (mw0 >> i0) & 1u : (mw1 >> (i0 - 32)) & 1u;
            const uint32_t b1 = i1 < 32 ? (mw0 >> i1) & 1u : (mw1 >> (i1 - 32)) & 1u;
            const float p0 = b0 ? ex2_approx(fmaf(v[i0], c2, -m_use)) : 0.f;
            const float p1 = b1 ? ex2_approx(fmaf(v[i1], c2, -m_use)) : 0.f;
            l8[i & 7] += p0 + p1;
            pk[i] = __uint_as_float(pack2<BF16>(p0, p1));
          }
        }
        l = l * alpha + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
        // P over the first 32 columns of its own score buffer
        tmem_st32(t_s, pk);
        // rescale the running O when the reference moved (after the PV of
        // tile gi - 1, the last one that wrote O)
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t pv = gi - 1;
          if (!pp.warp_wait(B_PV_DONE + (pv & 1), (pv >> 1) & 1)) return;
          tc_fence_after();
#pragma unroll
          for (int oc = 0; oc < D / 32; ++oc) {
            float o[32];
            tmem_ld32(t_row + C::kTmemO + oc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(t_row + C::kTmemO + oc * 32, o);
          }
        }
        if constexpr (PAGED) {
          // the last page of a sequence may be partly filled: its remaining
          // slots hold whatever the cache holds (not necessarily finite), so
          // the V rows from the sequence's end to the next 16-row step of the
          // PV are zeroed before the PV reads them (P is 0 there)
          if (nvalid < kBlockN && (nvalid & 15)) {
            if (!pp.warp_wait(B_V_FULL + stage, (gi / kStages) & 1)) return;
            const int r0 = nvalid, nr = ((nvalid + 15) & ~15) - nvalid;
            uint8_t* vt = pp.smem + C::kOffV + stage * C::kKVBytes;
            for (int i = wq * 32 + lane; i < nr * 8 * C::kAtoms; i += 128) {
              const int a = i / (nr * 8), rem = i % (nr * 8);
              *reinterpret_cast<uint4*>(vt + a * C::kKVAtomBytes + (r0 + rem / 8) * 128 +
                                        (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pp.bar[B_P_FULL + sb]);
      }
      // epilogue: wait for the last PV (tile gi - 1), then O / l and lse
      const uint32_t pv = gi - 1;
      if (!pp.warp_wait(B_PV_DONE + (pv & 1), (pv >> 1) & 1)) return;
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? m_ref + log2f(l) : -INFINITY;
    if (r.part >= 0) {
      // split-KV chunk: O / l and lse in float32 into the record's partial
      // state (packed row = TMEM lane), merged with the pair's other chunks
      // by the merge kernel
      const size_t prow = ((size_t)r.part * p.h_kv + kvh) * kBlockM + row;
      if (valid) p.part_lse[prow] = lse_v;
      float4* po = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll
      for (int oc = 0; oc < D / 32; ++oc) {
        float o[32];
        if (r.n_tiles > 0) {
          tmem_ld32(t_row + C::kTmemO + oc * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (oc == D / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && r.n_tiles > 0) mbar_arrive(&pp.bar[B_O_FREE]);
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[oc * 8 + i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                         o[4 * i + 3] * inv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pp.bar[B_ITEM_EMPTY + slot]);
      ++it;
      continue;
    }
    if (valid) p.lse[orow] = lse_v;
    // O / l in the storage dtype: 64 columns per TMEM round trip, written 32
    // columns (64 bytes per row) at a time through the warp's staging buffer,
    // then as whole-warp 16-byte stores of 8 rows x 64 bytes
    uint16_t* outp = reinterpret_cast<uint16_t*>(p.out);
    long long ro[4];
    int ok[4];
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const int src = st * 8 + (lane >> 2);   // row within the quadrant
      ro[st] = __shfl_sync(0xffffffffu, (long long)orow, src);
      ok[st] = __shfl_sync(0xffffffffu, valid ? 1 : 0, src);
    }
#pragma unroll
    for (int oc2 = 0; oc2 < D / 64; ++oc2) {
      float oa[32], ob[32];
      if (r.n_tiles > 0) {
        tmem_ld32(t_row + C::kTmemO + oc2 * 64, oa);
        tmem_ld32(t_row + C::kTmemO + oc2 * 64 + 32, ob);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) oa[i] = ob[i] = 0.f;
      }
      if (oc2 == D / 64 - 1) {
        // O is out of TMEM: the next item's first PV may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && r.n_tiles > 0) mbar_arrive(&pp.bar[B_O_FREE]);
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int oc = oc2 * 2 + hf;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = hf ? ob[2 * i] : oa[2 * i];
          const float x1 = hf ? ob[2 * i + 1] : oa[2 * i + 1];
          pk[i] = pack2<BF16>(x0 * inv, x1 * inv);
        }
        __syncwarp();   // the previous chunk's readers are done with the buffer
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          *reinterpret_cast<uint4*>(ost + lane * 64 + ((cc ^ ((lane >> 1) & 3)) * 16)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        __syncwarp();
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const int src = st * 8 + (lane >> 2);
          const int cc = lane & 3;
          const uint4 val =
              *reinterpret_cast<const uint4*>(ost + src * 64 + ((cc ^ ((src >> 1) & 3)) * 16));
          if (ok[st]) *reinterpret_cast<uint4*>(outp + ro[st] * D + oc * 32 + cc * 8) = val;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pp.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
}

// ---------------------------------------------------------------------------
template <int D, bool BF16, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  CtaShared* cta = reinterpret_cast<CtaShared*>(smem + C::kOffCta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pipe = warp / kWarpsPerPipe, pw = warp % kWarpsPerPipe;
  Pipe pp;
  pp.smem = smem + pipe * C::kPipeBytes;
  pp.bar = reinterpret_cast<uint64_t*>(pp.smem + C::kOffBar);
  pp.items = reinterpret_cast<Item*>(pp.smem + C::kOffItems);
  pp.abort = &cta->abort;
  pp.dev_error = &p.hdr->error;
  pp.limit_ns = p.timeout_ns;

  if (pw == 0 && lane == 0) {
    uint64_t* bar = pp.bar;
    const uint32_t consumers = 1u + 4u;   // MMA thread + softmax warps
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bar[B_ITEM_FULL + i], 1);
      mbar_init(&bar[B_ITEM_EMPTY + i], consumers);
    }
    mbar_init(&bar[B_Q_FULL], 1);
    mbar_init(&bar[B_Q_READY], 4);
    mbar_init(&bar[B_Q_EMPTY], 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar[B_K_FULL + i], 1);
      mbar_init(&bar[B_V_FULL + i], 1);
      mbar_init(&bar[B_EX_FULL + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[B_S_FULL + i], 1);
      mbar_init(&bar[B_P_FULL + i], 4);
      mbar_init(&bar[B_PV_DONE + i], 1);
    }
    mbar_init(&bar[B_O_FREE], 4);
    mbar_init(&bar[B_DRAIN], 1);
    mbar_init(&bar[B_STALL], 1);
    if (pipe == 0) cta->abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // rows of the Q tile that no TMA box covers (g * R < 128) must read as zero
  if (p.g * p.R < kBlockM) {
    uint4* q4 = reinterpret_cast<uint4*>(pp.smem + C::kOffQ);
    for (int i = pw * 32 + lane; i < C::kQBytes / 16; i += kWarpsPerPipe * 32)
      q4[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(&cta->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pp.tmem = cta->tmem_base + pipe * C::kTmemPipe;
  // everything above is private to the CTA; the plan, the rotated keys and
  // the work queue belong to the kernels before this one on the stream
  pdl_wait();

  if (pw == 0) {
    run_producer<D, PAGED>(pp, &tm_q, &tm_k, &tm_v, p, pipe, lane);
  } else if (pw == 1) {
    if (lane == 0) run_mma<D, BF16>(pp, p);
  } else {
    // softmax warp pw - 2 of this pipeline; its TMEM lane quadrant is warp % 4
    run_softmax<D, BF16, PAGED>(pp, p, warp & 3, lane);
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(cta->tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    // the last CTA re-arms the work queue so the plan can be reused
    __threadfence();
    const unsigned int done = atomicAdd(&p.hdr->queue_done, 1u);
    if (done == gridDim.x - 1) {
      p.hdr->queue_head = 0;
      p.hdr->queue_done = 0;
      __threadfence();
    }
  }
}

}  // namespace

template <int D, bool BF16, bool PAGED>
cudaError_t launch_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const AttnParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  static_assert(C::kSmemAlloc <= 227 * 1024, "shared memory budget");
  static_assert(B_COUNT <= 32, "barrier area");
  auto kern = attn_kernel<D, BF16, PAGED>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmemAlloc, stream, tm_q, tm_k, tm_v, p);
}

#define TA_INSTANTIATE(D, BF, PG)                                                       \
  template cudaError_t launch_attn<D, BF, PG>(const CUtensorMap&, const CUtensorMap&, \
                                              const CUtensorMap&, const AttnParams&, int, \
                                              cudaStream_t);
TA_INSTANTIATE(64, false, false)
TA_INSTANTIATE(64, true, false)
TA_INSTANTIATE(128, false, false)
TA_INSTANTIATE(128, true, false)
TA_INSTANTIATE(64, false, true)
TA_INSTANTIATE(64, true, true)
TA_INSTANTIATE(128, false, true)
TA_INSTANTIATE(128, true, true)
#undef TA_INSTANTIATE

}  // namespace ta
