// ta_attn.cu -- persistent batched tree-attention kernel for sm_103a.
//
// Computes what ``batch_tree_attn`` of the page "tree_attn.py" computes
// (per q row and head: masked online softmax of sm_scale * q.k in log2
// units, output O / d and lse = m + log2(d)), re-designed for one GB300 SM.
//
// One CTA per SM pops work units from a longest-first queue.  A unit is two
// consecutive Q tiles (A and B, 128 packed rows each) of one (sequence, kv
// head); both stream the same kv tiles of 128 columns, so every K/V tile
// loaded into shared memory serves two Q tiles.  Tensor memory holds one
// score buffer and one output accumulator per Q tile (S_A, S_B, O_A, O_B:
// 128 columns each).  Warp roles:
//   warp 0      producer: stages each unit's record (and, on the contiguous
//               path, its q rows' DFS enter indices), TMA-loads its Q tiles
//               (one buffer each) and its K tiles (two stages)
//   warp 1      MMA issuer (one thread): for kv tile t, PV_A(t-1) then
//               QK_A(t), PV_B(t-1) then QK_B(t) (tcgen05.mma, M = 128,
//               N = 128; P read from tensor memory), so that each tile's
//               softmax overlaps the other tile's tensor-core work
//   warp 2      V producer: TMA-loads the V tiles (two stages) and stages each
//               partial tile's column intervals beside them
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B (one TMEM
//               lane = packed row per thread): tree mask, online softmax
//               against a lazily moved reference, P (fp16/bf16) written over
//               the first half of the tile's score buffer, the rare rescale
//               of O, and the tile's epilogue once its last PV is done (O / l
//               and lse from tensor memory to global memory)
//   warps 12-15 correction: RoPE of each unit's Q tiles (before their first
//               QK^T)
// A kv tile that is empty for one Q tile (the plan classifies each tile for
// A and B) is skipped by that tile's QK^T, softmax and PV.  Keys arrive
// rotated (the run rotates them once per call).  Every cross-warp hand-off
// is an mbarrier with a bounded wait.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "ta_device.cuh"
#include "ta_launch.h"

namespace ta {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 2;   // K/V ring depth
constexpr int kSlots = 4;    // work-unit slots (producer, MMA, softmax, correction)
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpProducerV = 2;
constexpr int kWarpSoftmax = 4;      // warps 4..7 tile A, 8..11 tile B
constexpr int kWarpCorrection = 12;  // warps 12..15

// Register split (setmaxnreg) of the 512 threads' launch allocation of 128
// each (65,536 in all): the producer / MMA warpgroup gives registers up, the
// softmax warpgroups take them, the correction warps (RoPE only) keep theirs.
constexpr uint32_t kRegsLaunch = 128;
constexpr uint32_t kRegsIssue = 112;       // warps 0-3
constexpr uint32_t kRegsSoftmax = 136;     // warps 4-11
constexpr uint32_t kRegsCorrection = 128;  // warps 12-15
static_assert(128 * (kRegsIssue + 2 * kRegsSoftmax + kRegsCorrection) <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
static_assert(kRegsIssue <= kRegsLaunch && kRegsSoftmax >= kRegsLaunch &&
                  kRegsCorrection >= kRegsLaunch,
              "the first warpgroup gives registers up, the others take them");

enum Bar : int {
  B_ITEM_FULL = 0,                     // [kSlots] record staged
  B_ITEM_EMPTY = B_ITEM_FULL + kSlots, // [kSlots] MMA, V producer, softmax and correction warps done
  B_Q_FULL = B_ITEM_EMPTY + kSlots,    // [2] Q buffer of tile A / B landed
  B_Q_READY = B_Q_FULL + 2,            // [2] ... rotated (RoPE)
  B_Q_EMPTY = B_Q_READY + 2,           // [2] ... read by the unit's last QK^T
  B_K_FULL = B_Q_EMPTY + 2,            // [kStages]
  B_V_FULL = B_K_FULL + kStages,       // [kStages]
  B_EX_FULL = B_V_FULL + kStages,      // [kStages] column intervals of a partial tile
  // one commit per kv tile t on KV_DONE[t & 1], after its QK^Ts: it reports
  // tile t's QK^Ts (its K stage free) and tile t - 1's PVs (its V stage free)
  B_KV_DONE = B_EX_FULL + kStages,     // [kStages]
  B_S_FULL = B_KV_DONE + kStages,      // [2] score buffer of tile A / B written
  B_P_FULL = B_S_FULL + 2,             // [2] P written over it
  B_O_FULL = B_P_FULL + 2,             // [2] the unit's last PV into O_A / O_B done
  B_O_FREE = B_O_FULL + 2,             // [2] the tile's epilogue read O_A / O_B
  B_DRAIN = B_O_FREE + 2,
  B_STALL,                             // test hook: nothing ever arrives on it
  B_CLC,                               // launch-cancel response landed
  B_COUNT
};
constexpr int kBarSlots = 48;

struct Item {
  ItemRec r;
  int valid, kvh, pad[14];
};
static_assert(sizeof(Item) == 128, "item slot size");

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;               // 128-byte column blocks per row
  static constexpr int kQAtomBytes = kBlockM * 128;    // 128 rows x 128 bytes
  static constexpr int kKVAtomBytes = kBlockN * 128;   // 128 rows x 128 bytes
  static constexpr int kQBytes = kAtoms * kQAtomBytes;
  static constexpr int kKVBytes = kAtoms * kKVAtomBytes;
  static constexpr int kOstBytes = 32 * 64;            // per softmax warp: 32 rows x 64 bytes
  static constexpr int kOffQ = 0;                                   // [2] tile A, tile B
  static constexpr int kOffK = kOffQ + 2 * kQBytes;                 // [kStages]
  static constexpr int kOffV = kOffK + kStages * kKVBytes;          // [kStages]
  static constexpr int kOffEX = kOffV + kStages * kKVBytes;         // int2 [kStages][kBlockN]
  static constexpr int kOffOst = kOffEX + kStages * kBlockN * 8;    // [2 tiles][4 warps]
  static constexpr int kOffEq = kOffOst + 8 * kOstBytes;           // int [kSlots][2][kBlockM]
  static constexpr int kOffItems = kOffEq + kSlots * 2 * kBlockM * 4;
  static constexpr int kOffBar = kOffItems + kSlots * (int)sizeof(Item);
  static constexpr int kOffCta = kOffBar + kBarSlots * 8;
  static constexpr int kOffClc = kOffCta + 64;    // 16-byte launch-cancel response
  static constexpr int kUsed = kOffClc + 16;
  static constexpr int kSmemAlloc = kUsed + 1024;   // room to align the base to 1024
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 0;      // S of tile x at 128 * x (P over its first half)
  static constexpr uint32_t kTmemO = 256;    // O of tile x at 256 + 128 * x
};

struct CtaShared {
  uint32_t tmem_base;
  int abort;
};

struct Ctx {
  uint8_t* smem;
  void* clc_resp;
  uint64_t* bar;
  Item* items;
  volatile int* abort;
  unsigned int* dev_error;
  unsigned long long limit_ns;
  uint32_t tmem;     // first TMEM column (lane 0)
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait(&bar[b], parity, abort, dev_error, limit_ns);
  }
  // every lane of the warp waits; the warp proceeds only if all lanes saw it
  __device__ bool warp_wait(int b, uint32_t parity) const {
    const bool ok = mbar_wait(&bar[b], parity, abort, dev_error, limit_ns);
    return __all_sync(0xffffffffu, ok);
  }
  // waits whose bounded retry loop is one out-of-line function per register
  // budget instead of a copy at every wait site, which keeps the roles' loops
  // small: warp_wait_sm for the softmax warpgroups, warp_wait_cr for the
  // correction warps, wait_is / warp_wait_is for the producer, V producer and
  // MMA warps.  (A function called from regions of different setmaxnreg
  // budgets cannot be register-allocated.)
  __device__ bool warp_wait_sm(int b, uint32_t parity) const;
  __device__ bool warp_wait_cr(int b, uint32_t parity) const;
  __device__ bool wait_is(int b, uint32_t parity) const;
  __device__ bool warp_wait_is(int b, uint32_t parity) const;
  // wait used while draining after an abort: ignores the abort flag
  __device__ bool drain_wait(int b, uint32_t parity) const {
    int no_abort = 0;
    return mbar_wait(&bar[b], parity, &no_abort, dev_error, 200000000ull);
  }
};

__device__ __noinline__ bool softmax_wait_slow(uint64_t* bar, uint32_t parity,
                                               volatile int* abort, unsigned int* dev_error,
                                               uint64_t limit_ns) {
  return mbar_wait(bar, parity, abort, dev_error, limit_ns);
}
__device__ __noinline__ bool correction_wait_slow(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, unsigned int* dev_error,
                                                  uint64_t limit_ns) {
  return mbar_wait(bar, parity, abort, dev_error, limit_ns);
}
__device__ bool Ctx::warp_wait_cr(int b, uint32_t parity) const {
  const bool ok = mbar_try_wait(&bar[b], parity) ||
                  correction_wait_slow(&bar[b], parity, abort, dev_error, limit_ns);
  return __all_sync(0xffffffffu, ok);
}
__device__ bool Ctx::warp_wait_sm(int b, uint32_t parity) const {
  const bool ok = mbar_try_wait(&bar[b], parity) ||
                  softmax_wait_slow(&bar[b], parity, abort, dev_error, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

__device__ __noinline__ bool issue_wait_slow(uint64_t* bar, uint32_t parity,
                                             volatile int* abort, unsigned int* dev_error,
                                             uint64_t limit_ns) {
  return mbar_wait(bar, parity, abort, dev_error, limit_ns);
}
__device__ bool Ctx::wait_is(int b, uint32_t parity) const {
  return mbar_try_wait(&bar[b], parity) ||
         issue_wait_slow(&bar[b], parity, abort, dev_error, limit_ns);
}
__device__ bool Ctx::warp_wait_is(int b, uint32_t parity) const {
  const bool ok = mbar_try_wait(&bar[b], parity) ||
                  issue_wait_slow(&bar[b], parity, abort, dev_error, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Iterates the kv tiles of a work unit that are non-empty for tile A or B
// from its first tile (tile_lo, past 0 for a split-KV chunk): from the
// record's inline 4-bit classes for short sequences, else from the plan's
// class bytes.  next() returns the tile's class byte (A's class in bits 0-1,
// B's in 2-3; 0 when done).
struct TileIter {
  const uint8_t* cls;
  int kvt, j;
  bool inl;
  uint32_t w0, w1, w2, w3;   // inline classes, or the current 16 class bytes
  __device__ TileIter() : cls(nullptr), kvt(0), j(0), inl(true), w0(0), w1(0), w2(0), w3(0) {}
  __device__ TileIter(const ItemRec& r, const uint8_t* classes)
      : cls(classes + r.class_off), kvt(r.kvt), j(r.tile_lo - 1), inl(r.kvt <= kInlineTiles) {
    w0 = r.cls;
    w1 = w2 = w3 = 0;
    if (!inl && (r.tile_lo & 15)) {
      // a range that starts inside a 16-tile group: load that group now
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(cls + (r.tile_lo & ~15)));
      w0 = v.x;
      w1 = v.y;
      w2 = v.z;
      w3 = v.w;
    }
  }
  __device__ int next() {
    while (true) {
      ++j;
      if (j >= kvt) return 0;
      int c;
      if (inl) {
        c = (w0 >> (4 * j)) & 15;
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

// q rows of tile x (0: A, 1: B) of a unit record
__device__ __forceinline__ int tile_rows(const ItemRec& r, int x, int R) {
  return max(0, min(R, r.nq - x * R));
}
__device__ __forceinline__ int tile_count(const ItemRec& r, int x) { return x ? r.n_b : r.n_a; }
static_assert(offsetof(ItemRec, q_row0) == 8 && offsetof(ItemRec, n_a) == 52 &&
                  offsetof(ItemRec, n_b) == 56,
              "record words read by the producer's Q prefetch");

// ---------------------------------------------------------------------------
// producer warps (lane 0 issues): warp 0 stages the units and loads their Q
// tiles and K, warp 2 loads V and stages the mask intervals, so that neither
// kind of load waits behind the other's stage release
// ---------------------------------------------------------------------------
// The physical pages of kv tile j of a paged sequence (logical pages 8j ..
// 8j + 7), looked up by lanes 0-7 and shared with the warp; a page past the
// sequence's last takes an out-of-range index, read as zeros.
constexpr int kPagesPerTile = kBlockN / kPageSize;
__device__ __forceinline__ void tile_pages(const AttnParams& p, const ItemRec& r, int j, int lane,
                                           int (&ph)[kPagesPerTile]) {
  const int np = (r.kv + kPageSize - 1) / kPageSize;
  const int lp = j * kPagesPerTile + lane;
  int phys = p.num_pages;
  if (lane < kPagesPerTile && lp < np) phys = __ldg(p.page_values + r.kv_base + lp);
#pragma unroll
  for (int q = 0; q < kPagesPerTile; ++q) ph[q] = __shfl_sync(0xffffffffu, phys, q);
}

// One K or V tile (kv plane 0 = K, 1 = V of the paged cache) into ``dst``.
template <int D, bool PAGED>
__device__ __forceinline__ void load_kv_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                             int plane, int kvh, int row0,
                                             const int (&ph)[kPagesPerTile]) {
  using C = Cfg<D>;
#pragma unroll
  for (int a = 0; a < C::kAtoms; ++a) {
    if constexpr (PAGED) {
#pragma unroll
      for (int q = 0; q < kPagesPerTile; ++q)
        tma_load_5d(dst + a * C::kKVAtomBytes + q * kPageSize * 128, map, bar, a * 64, 0, kvh,
                    plane, ph[q]);
    } else {
      tma_load_3d(dst + a * C::kKVAtomBytes, map, bar, a * 64, kvh, row0);
    }
  }
}

template <int D, bool PAGED>
__device__ void run_producer(const Ctx& cx, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const AttnParams& p, int lane) {
  using C = Cfg<D>;
  uint8_t* sQ = cx.smem + C::kOffQ;
  uint8_t* sK = cx.smem + C::kOffK;
  // the plan kernel wrote the item count; never trust it beyond the table size
  const unsigned long long cap = (unsigned long long)p.max_records * (unsigned long long)p.h_kv;
  const unsigned long long n_items = *(volatile unsigned int*)&p.hdr->num_items;
  const unsigned int num_items = (unsigned int)(n_items < cap ? n_items : cap);
  const int g = p.g, R = p.R;
  uint32_t it = 0, kv_it = 0, q_it[2] = {0, 0};
  uint32_t issued_k = 0;   // loads issued (stage = count % kStages)
  // cluster launch control: requests stop at the first that finds no launch
  // left; at most one is in flight (lane 0's copies count)
  bool clc_live = p.sched_clc != 0, clc_pending = false;
  uint32_t clc_phase = 0;
  bool aborted = false;
  // the first unit of every CTA is fixed (CTA b takes item b, the items being
  // in longest-first order already); the rest come from the queue, which
  // starts after those grid items, or with cluster launch control from the
  // CTAs whose launches this one cancels
  const unsigned int n_static = gridDim.x;
  unsigned int idx = blockIdx.x;
  // lanes 0-3 hold the next record (16 bytes each), fetched one item ahead
  int4 rec_next = make_int4(0, 0, 0, 0);
  if (idx < num_items && lane < 4)
    rec_next = __ldg(reinterpret_cast<const int4*>(p.sorted + idx / p.h_kv) + lane);
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait(B_ITEM_EMPTY + slot, ((it / kSlots) & 1) ^ 1)) { aborted = true; break; }
    Item& s = cx.items[slot];
    if (idx >= num_items) {
      if (lane == 0) {
        s.valid = 0;
        mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
      }
      break;
    }
    if (lane < 4) reinterpret_cast<int4*>(&s.r)[lane] = rec_next;
    const int kvh = idx % p.h_kv;
    // pop the next index now; its round trip overlaps this unit's issue
    unsigned int nidx = 0;
    if (lane == 0) {
      if (!p.sched_clc) {
        nidx = n_static + atomicAdd(&p.hdr->queue_head, 1u);
      } else if (clc_live) {
        // ask for the unit of a CTA that has not started (read after this
        // unit's loads are issued)
        mbar_arrive_expect_tx(&cx.bar[B_CLC], 16);
        clc_try_cancel(cx.clc_resp, &cx.bar[B_CLC]);
        clc_pending = true;
      }
      s.valid = 1;
      s.kvh = kvh;
    }
    __syncwarp();
    const ItemRec r = s.r;
    if constexpr (!PAGED) {
      // the DFS enter index of each q row of the unit's two tiles (INT_MIN
      // past a tile's rows or for a tile that attends nothing), read by the
      // softmax warps' interval tests from the slot (the paged producer,
      // busy with page look-ups, leaves them to the softmax warps)
      int* eq = reinterpret_cast<int*>(cx.smem + C::kOffEq) + slot * 2 * kBlockM;
      int v[2 * kBlockM / 32];
#pragma unroll
      for (int k = 0; k < 2 * kBlockM / 32; ++k) {
        const int x = k / (kBlockM / 32), i = (k % (kBlockM / 32)) * 32 + lane;
        v[k] = INT_MIN;
        if (tile_count(r, x) > 0 && i < tile_rows(r, x, R))
          v[k] = __ldg(&p.tree_order[2 * (r.tree_base + r.r0 + x * R + i + r.tl - r.qo)]);
      }
#pragma unroll
      for (int k = 0; k < 2 * kBlockM / 32; ++k) eq[k * 32 + lane] = v[k];
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
    if (r.n_tiles > 0) {
      // the Q tiles that attend anything (each into its own buffer)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (tile_count(r, x) == 0) continue;
        if (!cx.warp_wait(B_Q_EMPTY + x, (q_it[x] & 1) ^ 1)) { aborted = true; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&cx.bar[B_Q_FULL + x], (uint32_t)(C::kAtoms * 128 * g * R));
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sQ + x * C::kQBytes + a * C::kQAtomBytes, tm_q, &cx.bar[B_Q_FULL + x],
                        a * 64, kvh * g, r.q_row0 + x * R);
        }
        ++q_it[x];
      }
      if (aborted) break;
      TileIter ti(r, p.classes);
      for (int n = 0; n < r.n_tiles; ++n) {
        ti.next();
        const int j = ti.j;
        const int row0 = r.kv_base + j * kBlockN;
        const int stage = kv_it % kStages;
        int ph[kPagesPerTile];
        if constexpr (PAGED) tile_pages(p, r, j, lane, ph);
        // the K stage is free once the QK^Ts of the tile two back are done
        if (!cx.warp_wait(B_KV_DONE + stage, ((kv_it / kStages) & 1) ^ 1)) { aborted = true; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&cx.bar[B_K_FULL + stage], (uint32_t)C::kKVBytes);
          load_kv_tile<D, PAGED>(sK + stage * C::kKVBytes, tm_k, &cx.bar[B_K_FULL + stage], 0, kvh,
                                 row0, ph);
        }
        ++issued_k;
        ++kv_it;
      }
      if (aborted) break;
    }
    if (p.sched_clc) {
      // the cancelled CTA's index is this CTA's next unit; a CTA past the
      // last unit is cancelled as well (and the next one asked for), so that
      // none of them launches only to find no work
      int stop = 0;
      nidx = num_items;
      if (lane == 0 && clc_live) {
        for (;;) {
          if (!cx.wait(B_CLC, clc_phase)) {
            stop = 1;
            break;
          }
          clc_pending = false;
          clc_phase ^= 1u;
          uint32_t x = 0;
          if (!clc_query(cx.clc_resp, &x)) {
            clc_live = false;   // every launch has started: no further requests
            break;
          }
          if (x < num_items) {
            nidx = x;
            break;
          }
          mbar_arrive_expect_tx(&cx.bar[B_CLC], 16);
          clc_try_cancel(cx.clc_resp, &cx.bar[B_CLC]);
          clc_pending = true;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) {
        aborted = true;
        break;
      }
    }
    idx = __shfl_sync(0xffffffffu, nidx, 0);
    if (idx < num_items) {
      if (lane < 4) rec_next = __ldg(reinterpret_cast<const int4*>(p.sorted + idx / p.h_kv) + lane);
      // warm L2 with the next unit's Q tiles while this unit's last kv tiles
      // run: their loads wait for this unit's last QK^Ts, then hit L2.
      // Record words: q_row0 = 2 (lane 0, .z), n_a / n_b = 13 / 14 (lane 3, .y / .z).
      const int nq_row0 = __shfl_sync(0xffffffffu, rec_next.z, 0);
      const int nn_a = __shfl_sync(0xffffffffu, rec_next.y, 3);
      const int nn_b = __shfl_sync(0xffffffffu, rec_next.z, 3);
      if (lane == 0) {
        const int nkvh = (int)(idx % (unsigned)p.h_kv);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if ((x ? nn_b : nn_a) > 0)
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a)
              tma_prefetch_l2_3d(tm_q, a * 64, nkvh * g, nq_row0 + x * R);
      }
    }
    ++it;
  }
  if (aborted && lane == 0) {
    // a launch-cancel request still in flight writes shared memory too
    if (clc_pending) cx.drain_wait(B_CLC, clc_phase);
    // let every copy already in flight land before the CTA's memory goes away:
    // the last load issued into each Q buffer and each K stage (load i of a
    // stage went to stage i % 2 and completes that stage's phase i / 2)
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (q_it[x] > 0) cx.drain_wait(B_Q_FULL + x, (q_it[x] - 1) & 1);
    for (uint32_t i = issued_k > kStages ? issued_k - kStages : 0; i < issued_k; ++i)
      cx.drain_wait(B_K_FULL + i % kStages, (i / kStages) & 1);
  }
}

template <int D, bool PAGED>
__device__ void run_producer_v(const Ctx& cx, const CUtensorMap* tm_v, const AttnParams& p,
                               int lane) {
  using C = Cfg<D>;
  uint8_t* sV = cx.smem + C::kOffV;
  int2* sEX = reinterpret_cast<int2*>(cx.smem + C::kOffEX);
  uint32_t it = 0, kv_it = 0, issued_v = 0;
  bool aborted = false;
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait_is(B_ITEM_FULL + slot, (it / kSlots) & 1)) { aborted = true; break; }
    const Item& s = cx.items[slot];
    const int valid = s.valid;
    const ItemRec r = s.r;
    const int kvh = s.kvh;
    __syncwarp();
    // the record is in registers: the slot is no longer needed here
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
    if (!valid) break;
    TileIter ti(r, p.classes);
    for (int n = 0; n < r.n_tiles; ++n) {
      const int cls = ti.next();
      const int j = ti.j;
      const int row0 = r.kv_base + j * kBlockN;
      const int stage = kv_it % kStages;
      int ph[kPagesPerTile];
      if constexpr (PAGED) tile_pages(p, r, j, lane, ph);
      // the V stage is free once the PVs of the tile two back are done: the
      // commit of the tile after it reports them
      if (kv_it >= kStages &&
          !cx.warp_wait_is(B_KV_DONE + ((kv_it - 1) & 1), ((kv_it - 1) >> 1) & 1)) {
        aborted = true;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&cx.bar[B_V_FULL + stage], (uint32_t)C::kKVBytes);
        load_kv_tile<D, PAGED>(sV + stage * C::kKVBytes, tm_v, &cx.bar[B_V_FULL + stage], 1, kvh,
                               row0, ph);
      }
      ++issued_v;
      // column intervals of a tile partial for tile A or B (FULL tiles need
      // none), as start and length: a row sees the column iff its enter
      // index minus start is below length, compared unsigned.  Written after
      // the PVs of the tile two back -- behind both softmaxes' reads of this
      // stage's intervals -- have completed.
      if ((cls & 3) == kTilePartial || (cls >> 2) == kTilePartial) {
        int2* ex = sEX + stage * kBlockN;
#pragma unroll
        for (int q = 0; q < kBlockN / 32; ++q) {
          const int2 iv = column_interval(p.tree_order, r.tree_base, j * kBlockN + q * 32 + lane,
                                          r.kv, r.kv - r.tl);
          // an empty interval (a column past the sequence's end) gets
          // length 0, which no row passes
          ex[q * 32 + lane] =
              make_int2(iv.x, iv.y > iv.x ? (int)((uint32_t)iv.y - (uint32_t)iv.x) : 0);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cx.bar[B_EX_FULL + stage]);
      ++kv_it;
    }
    if (aborted) break;
  }
  if (aborted && lane == 0) {
    // the last V load issued into each stage must land before the CTA exits
    for (uint32_t i = issued_v > kStages ? issued_v - kStages : 0; i < issued_v; ++i)
      cx.drain_wait(B_V_FULL + i % kStages, (i / kStages) & 1);
  }
}

// ---------------------------------------------------------------------------
// MMA warp (one thread)
// ---------------------------------------------------------------------------
// For kv tile t of a unit: PV_A(t-1), QK_A(t), PV_B(t-1), QK_B(t) -- a Q tile
// for which kv tile t is empty skips that QK^T and, one tile later, that PV.
// A QK^T overwrites the score buffer whose P the same Q tile's previous PV
// reads; tcgen05.mma operations issued by one thread execute in issue order,
// so it follows that PV without waiting for it.
template <int D, bool BF16>
__device__ void run_mma(const Ctx& cx, const AttnParams& p) {
  using C = Cfg<D>;
  // descriptors of k-step 0; a k-step or buffer offset is added to the
  // descriptor's 14-bit start-address field (addresses stay below 256 KB)
  static_assert(kStages == 2, "descriptor selection below assumes two stages");
  const uint64_t dq0 = sw128_desc(smem_u32(cx.smem + C::kOffQ), 0);
  const uint64_t dq1 = dq0 + (uint64_t)(C::kQBytes >> 4);
  const uint64_t dk0 = sw128_desc(smem_u32(cx.smem + C::kOffK), 0);
  const uint64_t dk1 = dk0 + (uint64_t)(C::kKVBytes >> 4);
  const uint64_t dv0 = sw128_desc(smem_u32(cx.smem + C::kOffV), C::kKVAtomBytes);
  const uint64_t dv1 = dv0 + (uint64_t)(C::kKVBytes >> 4);
  constexpr uint32_t idesc_pv = umma_idesc_f16(BF16, 128, D, /*b_mn_major=*/true);
  const int q_bar = p.rotary ? B_Q_READY : B_Q_FULL;
  uint32_t it = 0, kc = 0;   // unit slots consumed, kv tiles (K / V stage phases)
  // per Q tile x (bit x): parity of its PVs issued (P_FULL phase), of its
  // units entered (Q phase), of its units whose PVs started (O_FREE phase)
  uint32_t kp = 0, qx = 0, ox = 0;
  bool ok = true, issued_any = false;
  // test hook: a wait that runs out before any MMA is issued (the other warps
  // then find the abort flag in their own waits)
  if (p.debug_stall) {
    cx.wait_is(B_STALL, 0);
    ok = false;
  }
  using X0 = std::integral_constant<int, 0>;
  using X1 = std::integral_constant<int, 1>;
  while (ok) {
    const int slot = it % kSlots;
    if (!cx.wait_is(B_ITEM_FULL + slot, (it / kSlots) & 1)) break;
    const Item& s = cx.items[slot];
    const int valid = s.valid;
    const ItemRec r = s.r;
    // the record is in registers: the slot is no longer needed here
    mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
    if (!valid) break;
    if (r.n_tiles == 0) continue;
    // QK^Ts still to issue per Q tile in this unit (its Q buffer is released
    // after the last); a tile's Q is waited for at its first QK^T
    int left0 = r.n_a, left1 = r.n_b;
    bool q_ok0 = false, q_ok1 = false;
    uint32_t v_kc = 0xFFFFFFFFu;   // the kv tile whose V stage was last waited for
    // the PV each Q tile owes for its previous kv tile: valid kv columns
    // (bits 0-7; 0: none), K/V stage (bit 8), that stage's phase (bit 9)
    uint32_t pend0 = 0, pend1 = 0;
    bool started0 = false, started1 = false;
    auto issue_pv = [&](auto xc) -> bool {
      constexpr int x = decltype(xc)::value;
      uint32_t& pend = x ? pend1 : pend0;
      bool& started = x ? started1 : started0;
      const int nv = (int)(pend & 0xFFu), stage = (int)((pend >> 8) & 1u);
      if (!cx.wait_is(B_P_FULL + x, (kp >> x) & 1)) return false;
      const uint32_t tile_kc = kc - 1;   // a pending PV belongs to the previous kv tile
      if (v_kc != tile_kc) {
        if (!cx.wait_is(B_V_FULL + stage, (pend >> 9) & 1)) return false;
        v_kc = tile_kc;
      }
      // O is free once the epilogue of the Q tile's previous unit read it
      if (!started && !cx.wait_is(B_O_FREE + x, ((ox >> x) & 1) ^ 1)) return false;
      tc_fence_after();
      const int nk = (nv + 15) >> 4;   // 16-row k-steps holding valid kv rows
      const uint64_t dv = stage ? dv1 : dv0;
      const uint32_t pcol = cx.tmem + C::kTmemS + 128 * x;   // P: two elements per column
      const uint32_t d_o = cx.tmem + C::kTmemO + 128 * x;
#pragma unroll
      for (int k = 0; k < kBlockN / 16; ++k) {
        if (k < nk)
          umma_f16_tmem_a(d_o, pcol + k * 8, dv + (uint64_t)(k * 16 * 128 >> 4), idesc_pv,
                          (started || k > 0) ? 1u : 0u);
      }
      if (!started) {
        started = true;
        ox ^= 1u << x;
      }
      kp ^= 1u << x;
      pend = 0;
      return true;
    };
    // one Q tile's part of kv tile n: its owed PV, then its QK^T if the tile
    // is non-empty for it
    auto bracket = [&](auto xc, int cls, int nvalid, int stage, bool& k_ready) -> bool {
      constexpr int x = decltype(xc)::value;
      uint32_t& pend = x ? pend1 : pend0;
      if (pend && !issue_pv(xc)) return false;
      if ((cls >> (2 * x)) & 3) {
        bool& q_ok = x ? q_ok1 : q_ok0;
        if (!q_ok) {
          if (!cx.wait_is(q_bar + x, (qx >> x) & 1)) return false;
          qx ^= 1u << x;
          q_ok = true;
        }
        if (!k_ready) {
          if (!cx.wait_is(B_K_FULL + stage, (kc >> 1) & 1)) return false;
          // the tile's column intervals too: a softmax warpgroup whose Q tile
          // skips kv tiles could otherwise reach this tile while the V
          // producer is two tiles behind, and its own wait on the two-stage
          // EX_FULL barrier would then match the older phase of the same
          // parity.  Waiting here keeps every phase in order.
          if (!cx.wait_is(B_EX_FULL + stage, (kc >> 1) & 1)) return false;
          k_ready = true;
        }
        // S = Q K^T of this Q tile (K from TMA, Q from TMA or the correction
        // warps' proxy-fenced stores: no tcgen05 fence needed)
        const uint32_t idesc = umma_idesc_f16(BF16, 128, (nvalid + 15) & ~15, false);
        const uint64_t dq = x ? dq1 : dq0;
        const uint64_t dk = stage ? dk1 : dk0;
        const uint32_t d_s = cx.tmem + C::kTmemS + 128 * x;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qo = (uint32_t)(((k >> 2) * C::kQAtomBytes + (k & 3) * 32) >> 4);
          const uint32_t ko = (uint32_t)(((k >> 2) * C::kKVAtomBytes + (k & 3) * 32) >> 4);
          umma_f16(d_s, dq + qo, dk + ko, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&cx.bar[B_S_FULL + x]);
        issued_any = true;
        pend = (uint32_t)nvalid | ((uint32_t)stage << 8) | (((kc >> 1) & 1u) << 9);
        int& left = x ? left1 : left0;
        if (--left == 0) umma_commit(&cx.bar[B_Q_EMPTY + x]);   // the unit's last QK^T of this tile
      }
      return true;
    };
    TileIter ti(r, p.classes);
    for (int n = 0; n < r.n_tiles; ++n) {
      const int cls = ti.next();
      const int nvalid = min(kBlockN, r.kv - ti.j * kBlockN);
      const int stage = kc & 1;
      bool k_ready = false;
      if (!bracket(X0{}, cls, nvalid, stage, k_ready) || !bracket(X1{}, cls, nvalid, stage, k_ready)) {
        ok = false;
        break;
      }
      umma_commit(&cx.bar[B_KV_DONE + stage]);   // this tile's QK^Ts, the previous tile's PVs
      ++kc;
    }
    if (!ok) break;
    // the unit's last PVs; each tile's output is complete after its own
    // (tile A's epilogue does not wait for tile B's last P)
    if (pend0 && !issue_pv(X0{})) break;
    if (started0) umma_commit(&cx.bar[B_O_FULL + 0]);
    if (pend1 && !issue_pv(X1{})) break;
    if (started1) umma_commit(&cx.bar[B_O_FULL + 1]);
  }
  if (*cx.abort && issued_any) {
    umma_commit(&cx.bar[B_DRAIN]);
    cx.drain_wait(B_DRAIN, 0);
  }
}

// ---------------------------------------------------------------------------
// RoPE of the Q tiles (correction warps)
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

// ---------------------------------------------------------------------------
// softmax warps (warpgroup x: rows of Q tile x, their scores and epilogue)
// ---------------------------------------------------------------------------
// Writes Q tile x's rows of a unit: O / l in the storage dtype and
// lse = m + log2(l) (or, for a split-KV chunk, float32 O / l and lse into its
// partial state).  With ``has_o`` the tile's O is read from TMEM once the
// unit's last PV is done (O_FULL phase ``o_par``; lse, 1 / l and the row
// addresses are prepared before that wait) and the buffer released; without,
// the tile attended nothing: out = 0, lse = -inf.  False if the wait gave up.
template <int D, bool BF16, bool SPLIT>
__device__ bool store_tile(const Ctx& cx, const AttnParams& p, const ItemRec& r, int x, int kvh,
                           int wq, int lane, bool has_o, uint32_t o_par, float m_ref, float l) {
  using C = Cfg<D>;
  const int row = wq * 32 + lane;
  const uint32_t t_o = cx.tmem + ((uint32_t)(wq * 32) << 16) + C::kTmemO + 128 * x;
  uint8_t* ost = cx.smem + C::kOffOst + (x * 4 + wq) * C::kOstBytes;
  const int g = p.g, R = p.R;
  const bool in_pack = row < g * R;
  const int qr = in_pack ? row / g : 0;
  const int hh = in_pack ? row - qr * g : 0;
  const bool valid = in_pack && qr < tile_rows(r, x, R);
  const int head = kvh * g + hh;
  const size_t orow = (size_t)(r.q_row0 + x * R + qr) * p.h_q + head;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse_v = l > 0.f ? m_ref + log2f(l) : -INFINITY;
  if (SPLIT && r.part >= 0) {
    // split-KV chunk: O / l and lse in float32 into the record's partial
    // state (tile x's 128 packed rows, packed row = TMEM lane), merged with
    // the pair's other chunks by the merge kernel
    const size_t prow = (((size_t)r.part * p.h_kv + kvh) * kTilesPerUnit + x) * kBlockM + row;
    if (valid) p.part_lse[prow] = lse_v;
    if (has_o) {
      if (!cx.warp_wait_sm(B_O_FULL + x, o_par)) return false;
      tc_fence_after();
    }
    float4* po = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll
    for (int oc = 0; oc < D / 32; ++oc) {
      float o[32];
      if (has_o) {
        tmem_ld32(t_o + oc * 32, o);
        tmem_wait_ld(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (oc == D / 32 - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && has_o) mbar_arrive(&cx.bar[B_O_FREE + x]);
      }
      if (valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          po[oc * 8 + i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                       o[4 * i + 3] * inv);
      }
    }
    return true;
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
  if (has_o) {
    if (!cx.warp_wait_sm(B_O_FULL + x, o_par)) return false;
    tc_fence_after();
  }
#pragma unroll
  for (int oc2 = 0; oc2 < D / 64; ++oc2) {
    float oa[32], ob2[32];
    if (has_o) {
      tmem_ld32(t_o + oc2 * 64, oa);
      tmem_ld32(t_o + oc2 * 64 + 32, ob2);
      tmem_wait_ld(oa);
      tmem_wait_ld(ob2);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) oa[i] = ob2[i] = 0.f;
    }
    if (oc2 == D / 64 - 1) {
      // O is out of TMEM: the Q tile's next unit may accumulate into it
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && has_o) mbar_arrive(&cx.bar[B_O_FREE + x]);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int oc = oc2 * 2 + hf;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = hf ? ob2[2 * i] : oa[2 * i];
        const float x1 = hf ? ob2[2 * i + 1] : oa[2 * i + 1];
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
  return true;
}

// The rare reference move of one 32-column chunk (some row's P sum above
// 256), kept out of the softmax's chunk loop so that its code is fetched
// only when it runs.  The chunk's scores are read again from tensor memory
// (its P is not yet written over them) and formed exactly as the loop formed
// them (the loop's m_use; the mask from its visibility word ``w`` or the
// column intervals; a row that took its reference m_ref in this chunk
// subtracts it); then, as in the loop, the chunk's max moves the reference of
// the rows whose max outgrew it by more than 2^8 (rescaling this tile's P
// chunks already written) and the chunk's P is written.  Returns the row's
// (m_ref, alpha_t, lsum, chunk sum).
// The rare rescale of a Q tile's running O (D columns of this warp's rows
// in tensor memory) by the product of the tile's reference moves, out of the
// tile loop.
template <int D>
__device__ __noinline__ void rescale_o(uint32_t t_o, float alpha_t) {
#pragma unroll 1
  for (int oc = 0; oc < D / 32; ++oc) {
    float o[32];
    tmem_ld32(t_o + oc * 32, o);
    tmem_wait_ld(o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= alpha_t;
    tmem_st32(t_o + oc * 32, o);
  }
}

template <bool BF16, int GL>
__device__ __noinline__ float4 chunk_ref_move(uint32_t t_s, int q, float c2, float m_use, bool fr,
                                              float m_ref, float alpha_t, float lsum,
                                              bool partial, uint32_t w, const int2* ivs,
                                              int e_row) {
  float x[32];
  tmem_ld32(t_s + 32 * q, x);
  tmem_wait_ld(x);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 t = ffma2(make_float2(x[2 * i], x[2 * i + 1]), make_float2(c2, c2),
                           make_float2(-m_use, -m_use));
    x[2 * i] = t.x;
    x[2 * i + 1] = t.y;
  }
  if (partial) {
    if constexpr (GL > 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!((w >> i) & 1u)) x[i] = -INFINITY;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int4 e = reinterpret_cast<const int4*>(ivs + 32 * q)[i];
        if (!((uint32_t)(e_row - e.x) < (uint32_t)e.y)) x[2 * i] = -INFINITY;
        if (!((uint32_t)(e_row - e.z) < (uint32_t)e.w)) x[2 * i + 1] = -INFINITY;
      }
    }
  }
  if (fr) {
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] -= m_ref;
  }
  float m4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) m4[k] = x[k];
#pragma unroll
  for (int i = 4; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
  const float tmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
  const bool mv = tmax > 8.f;
  uint32_t pk[16];
  float csum;
  if (__any_sync(0xffffffffu, mv)) {
    const float a = mv ? ex2_approx(-tmax) : 1.f;
    const float sh = mv ? tmax : 0.f;
    if (mv) m_ref += tmax;
    alpha_t *= a;
    lsum *= a;
    csum = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p0 = ex2_approx(x[2 * i] - sh), p1 = ex2_approx(x[2 * i + 1] - sh);
      csum += p0 + p1;
      pk[i] = pack2<BF16>(p0, p1);
    }
    if (q > 0) {
      // this tile's P chunks already written: rescale them in TMEM
      tmem_wait_st();
      for (int j = 0; j < q; ++j) {
        uint32_t v[16];
        tmem_ld16(t_s + 16 * j, v);
        tmem_wait_ld(v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 f = unpack2<BF16>(v[i]);
          v[i] = pack2<BF16>(f.x * a, f.y * a);
        }
        tmem_st16(t_s + 16 * j, v);
      }
    }
  } else {
    // no row moved: the chunk's P and sum as the loop formed them
    float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p0 = ex2_approx(x[2 * i]), p1 = ex2_approx(x[2 * i + 1]);
      if (i & 1)
        lb = fadd2(lb, make_float2(p0, p1));
      else
        la = fadd2(la, make_float2(p0, p1));
      pk[i] = pack2<BF16>(p0, p1);
    }
    csum = (la.x + la.y) + (lb.x + lb.y);
  }
  tmem_st16(t_s + 16 * q, pk);
  return make_float4(m_ref, alpha_t, lsum, csum);
}

template <int D, bool BF16, bool PAGED, int GL, bool SPLIT>
__device__ void softmax_loop(const Ctx& cx, const AttnParams& p, int x, int wq, int lane) {
  using C = Cfg<D>;
  const int row = wq * 32 + lane;             // packed row = TMEM lane
  const uint32_t t_row = cx.tmem + ((uint32_t)(wq * 32) << 16);
  const int2* sEX = reinterpret_cast<const int2*>(cx.smem + C::kOffEX);
  const float c2 = p.scale_log2;
  const int g = p.g, R = p.R;
  const bool in_pack = row < g * R;
  const int qr = in_pack ? row / g : 0;
  // slots, kv tiles of the units, tiles of this Q tile, units in which it attends
  uint32_t it = 0, c = 0, kx = 0, sx = 0;
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait_sm(B_ITEM_FULL + slot, (it / kSlots) & 1)) return;
    const Item& s = cx.items[slot];
    if (!s.valid) return;
    const ItemRec r = s.r;
    const int kvh = s.kvh;
    const bool valid = in_pack && qr < tile_rows(r, x, R);
    // the row's DFS enter index (staged with the record by the producer on
    // the contiguous path)
    int e_row = INT_MIN;
    if constexpr (PAGED) {
      if (valid && tile_count(r, x) > 0)
        e_row = __ldg(&p.tree_order[2 * (r.tree_base + r.r0 + x * R + qr + r.tl - r.qo)]);
    } else {
      if (valid) e_row = reinterpret_cast<const int*>(cx.smem + C::kOffEq)[(slot * 2 + x) * kBlockM + qr];
    }
    float m_ref = -INFINITY, l = 0.f;
    bool first = true;
    TileIter ti(r, p.classes);
    for (int n = 0; n < r.n_tiles; ++n, ++c) {
      const int cls = (ti.next() >> (2 * x)) & 3;
      if (cls == kTileEmpty) continue;
      const int nvalid = min(kBlockN, r.kv - ti.j * kBlockN);
      const int sb = c & 1;   // the kv tile's K / V stage (its column intervals)
      const bool partial = cls == kTilePartial;
      if (partial && !cx.warp_wait_sm(B_EX_FULL + sb, (c >> 1) & 1)) return;
      if (!cx.warp_wait_sm(B_S_FULL + x, kx & 1)) return;
      tc_fence_after();
      const uint32_t t_s = t_row + C::kTmemS + 128 * x;
      // One pass over the tile's 32-column chunks (a rolled loop: the code
      // stays small enough for the instruction cache).  Scores are taken
      // relative to the row's running reference, t = s * c2 - m, and P = 2^t
      // is formed at once; only when a chunk's P sum exceeds 256 (so that
      // some t may exceed 8), or the row has no reference yet, is the chunk's
      // max taken and the reference moved -- this tile's P columns already
      // written, l and (before this tile's PV) O rescaled -- and P formed
      // again.  P = 2^t <= 256 throughout.
      const int nch = (nvalid + 31) >> 5;
      const int2* ivs = sEX + sb * kBlockN;
      float alpha_t = 1.f;   // product of this tile's reference moves
      float lsum = 0.f;
      // some row of the warp has no reference yet (usually only in the
      // unit's first tile)
      bool need_ref = __any_sync(0xffffffffu, m_ref == -INFINITY);
#pragma unroll 1
      for (int q = 0; q < nch; ++q) {
        float x[32];
        tmem_ld32(t_s + 32 * q, x);
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t wv = 0xffffffffu;   // the chunk's visibility word (GL > 0, PARTIAL)
        bool fr = false;             // the row took its reference from this chunk
        tmem_wait_ld(x);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 t = ffma2(make_float2(x[2 * i], x[2 * i + 1]), make_float2(c2, c2),
                                 make_float2(-m_use, -m_use));
          x[2 * i] = t.x;
          x[2 * i + 1] = t.y;
        }
        if (partial) {
          // column c is visible iff e_row lies in its interval, stored by
          // the V producer as (start, length): (e_row - start) < length unsigned
          if constexpr (GL > 0) {
            // g a multiple of GL (4 or 8): lanes GL*k .. GL*k + GL - 1 hold
            // heads of one q row.  Lane s of those tests columns s, s + GL,
            // s + 2 GL, ... of the chunk, and 32 / GL ballots give the row's
            // 32 visibility bits (bit i: column i)
            const int base = lane & ~(GL - 1), sl = lane & (GL - 1);
            uint32_t& w = wv;
            w = 0;
#pragma unroll
            for (int k = 0; k < 32 / GL; ++k) {
              const int2 e = ivs[32 * q + GL * k + sl];
              const uint32_t b =
                  __ballot_sync(0xffffffffu, (uint32_t)(e_row - e.x) < (uint32_t)e.y);
              w |= ((b >> base) & ((1u << GL) - 1u)) << (GL * k);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!((w >> i) & 1u)) x[i] = -INFINITY;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int4 e = reinterpret_cast<const int4*>(ivs + 32 * q)[i];
              if (!((uint32_t)(e_row - e.x) < (uint32_t)e.y)) x[2 * i] = -INFINITY;
              if (!((uint32_t)(e_row - e.z) < (uint32_t)e.w)) x[2 * i + 1] = -INFINITY;
            }
          }
        }
        // a row without a reference yet (its first visible columns, usually
        // the unit's first tile) takes it from this chunk's max before any
        // exponential: nothing before carries weight (l, O and this tile's P
        // are 0), so the factor is 0
        if (need_ref && __any_sync(0xffffffffu, m_ref == -INFINITY)) {
          float m4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = x[k];
#pragma unroll
          for (int i = 4; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
          const float tmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          if (m_ref == -INFINITY && tmax > -INFINITY) {
            m_ref = tmax;   // m_use was 0
            fr = true;
            alpha_t = 0.f;
            lsum = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] -= tmax;
          }
        }
        // P, two per 32-bit word, for columns 16q .. 16q + 15 of the score
        // buffer (read by the PV's k-steps 2q and 2q + 1)
        uint32_t pk[16];
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(x[2 * i]), p1 = ex2_approx(x[2 * i + 1]);
          if (i & 1)
            lb = fadd2(lb, make_float2(p0, p1));
          else
            la = fadd2(la, make_float2(p0, p1));
          pk[i] = pack2<BF16>(p0, p1);
        }
        float csum = (la.x + la.y) + (lb.x + lb.y);
        if (__any_sync(0xffffffffu, !(csum <= 256.f))) {
          // some t may exceed 8: the reference-move path, out of line; it
          // writes the chunk's P itself
          const float4 mr = chunk_ref_move<BF16, GL>(t_s, q, c2, m_use, fr, m_ref, alpha_t, lsum,
                                                     partial, wv, ivs, e_row);
          m_ref = mr.x;
          alpha_t = mr.y;
          lsum = mr.z + mr.w;
        } else {
          lsum += csum;
          tmem_st16(t_s + 16 * q, pk);
        }
      }
      l = l * alpha_t + lsum;
      // rescale the running O when the reference moved: the PV of this Q
      // tile's previous kv tile, the last one that wrote O, was issued
      // before the QK^T whose completion S_FULL reported, so it is done
      if (!first && __any_sync(0xffffffffu, alpha_t != 1.f))
        rescale_o<D>(t_row + C::kTmemO + 128 * x, alpha_t);
      if constexpr (PAGED) {
        // the last page of a sequence may be partly filled: its remaining
        // slots hold whatever the cache holds (not necessarily finite), so
        // the V rows from the sequence's end to the next 16-row step of the
        // PV are zeroed before the PV reads them (P is 0 there); both Q
        // tiles' softmax warps may write the same zeros
        if (nvalid < kBlockN && (nvalid & 15)) {
          if (!cx.warp_wait_sm(B_V_FULL + sb, (c >> 1) & 1)) return;
          const int r0 = nvalid, nr = ((nvalid + 15) & ~15) - nvalid;
          uint8_t* vt = cx.smem + C::kOffV + sb * C::kKVBytes;
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
      if (lane == 0) mbar_arrive(&cx.bar[B_P_FULL + x]);
      ++kx;
      first = false;
    }
    // the tile's epilogue, as soon as its last PV is done (while the next
    // unit's Q tiles land and rotate); a tile that attended nothing is
    // written as out = 0, lse = -inf
    const bool has_o = tile_count(r, x) > 0;
    if (!store_tile<D, BF16, SPLIT>(cx, p, r, x, kvh, wq, lane, has_o, sx & 1, m_ref, l)) return;
    if (has_o) ++sx;
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
}

// The softmax warps' loop; on every way out (the work is done, or a bounded
// wait gave up) the warp waits for its own TMEM loads and stores to finish
// before the CTA frees the TMEM.
template <int D, bool BF16, bool PAGED, int GL, bool SPLIT>
__device__ void run_softmax(const Ctx& cx, const AttnParams& p, int x, int wq, int lane) {
  softmax_loop<D, BF16, PAGED, GL, SPLIT>(cx, p, x, wq, lane);
  tmem_wait_ld();
  tmem_wait_st();
}

// ---------------------------------------------------------------------------
// correction warps: RoPE of Q
// ---------------------------------------------------------------------------
// The correction warps rotate each unit's Q tiles under RoPE (a tile's first
// QK^T waits for its rotation); the softmax warpgroups write the epilogues.
template <int D, bool BF16>
__device__ void correction_loop(const Ctx& cx, const AttnParams& p, int wq, int lane) {
  using C = Cfg<D>;
  const int g = p.g, R = p.R;
  // slots; per Q tile x (bit x): parity of its units with tiles
  uint32_t it = 0, qi = 0;
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait_cr(B_ITEM_FULL + slot, (it / kSlots) & 1)) return;
    const Item& s = cx.items[slot];
    if (!s.valid) break;
    const ItemRec r = s.r;
    if (p.rotary && r.n_tiles > 0) {
#pragma unroll 1
      for (int x = 0; x < 2; ++x) {
        if (tile_count(r, x) == 0) continue;
        // q row r of the tile takes the position of its own tree node's kv
        // slot (the first cos/sin batch is fetched while the Q tile lands)
        const long long qtok0 =
            (long long)r.kv_base + (r.kv - r.qo) + (long long)r.r0 + (long long)x * R;
        const RopeRange rr = rope_range<D>(tile_rows(r, x, R), g, wq);
        float4 cv[2][4];
        rope_load<D>(cv, p.rope_cs, qtok0, rr, 0, lane);
        if (!cx.warp_wait_cr(B_Q_FULL + x, (qi >> x) & 1)) return;
        rope_q_rows<D, BF16>(cx.smem + C::kOffQ + x * C::kQBytes, p.rope_cs, qtok0, rr, g, lane,
                             cv);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_Q_READY + x]);
        qi ^= 1u << x;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
}

template <int D, bool BF16>
__device__ void run_correction(const Ctx& cx, const AttnParams& p, int wq, int lane) {
  correction_loop<D, BF16>(cx, p, wq, lane);
  tmem_wait_ld();
  tmem_wait_st();
}

// ---------------------------------------------------------------------------
// GL: the softmax's mask test shared by groups of GL lanes of one q row (g a
// multiple of GL), or per lane (GL = 0)
template <int D, bool BF16, bool PAGED, int GL, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  CtaShared* cta = reinterpret_cast<CtaShared*>(smem + C::kOffCta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.smem = smem;
  cx.clc_resp = smem + C::kOffClc;
  cx.bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  cx.items = reinterpret_cast<Item*>(smem + C::kOffItems);
  cx.abort = &cta->abort;
  cx.dev_error = &p.hdr->error;
  cx.limit_ns = p.timeout_ns;

  if (warp == 0 && lane == 0) {
    uint64_t* bar = cx.bar;
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bar[B_ITEM_FULL + i], 1);
      // MMA thread, V producer, two softmax warpgroups and the correction warps
      mbar_init(&bar[B_ITEM_EMPTY + i], 1 + 1 + 8 + 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[B_Q_FULL + i], 1);
      mbar_init(&bar[B_Q_READY + i], 4);
      mbar_init(&bar[B_Q_EMPTY + i], 1);
      mbar_init(&bar[B_S_FULL + i], 1);
      mbar_init(&bar[B_P_FULL + i], 4);
      mbar_init(&bar[B_O_FULL + i], 1);
      mbar_init(&bar[B_O_FREE + i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar[B_K_FULL + i], 1);
      mbar_init(&bar[B_V_FULL + i], 1);
      mbar_init(&bar[B_EX_FULL + i], 1);
      mbar_init(&bar[B_KV_DONE + i], 1);
    }
    mbar_init(&bar[B_DRAIN], 1);
    mbar_init(&bar[B_STALL], 1);
    mbar_init(&bar[B_CLC], 1);
    cta->abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // rows of the Q buffers that no TMA box covers (g * R < 128) must read as zero
  if (p.g * p.R < kBlockM) {
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::kOffQ);
    for (int i = threadIdx.x; i < 2 * C::kQBytes / 16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) tmem_alloc(&cta->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = cta->tmem_base;
  // everything above is private to the CTA; the plan, the rotated keys and
  // the work queue belong to the kernels before this one on the stream
  pdl_wait();

  if (warp < kWarpSoftmax) {
    regs_dec<kRegsIssue>();
    if (warp == kWarpProducer) {
      run_producer<D, PAGED>(cx, &tm_q, &tm_k, p, lane);
    } else if (warp == kWarpMma) {
      if (lane == 0) run_mma<D, BF16>(cx, p);
    } else if (warp == kWarpProducerV) {
      run_producer_v<D, PAGED>(cx, &tm_v, p, lane);
    }
  } else if (warp < kWarpCorrection) {
    regs_inc<kRegsSoftmax>();
    run_softmax<D, BF16, PAGED, GL, SPLIT>(cx, p, (warp - kWarpSoftmax) >> 2, warp & 3, lane);
  } else {
    regs_inc<kRegsCorrection>();
    run_correction<D, BF16>(cx, p, warp & 3, lane);
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(cta->tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0 && !p.sched_clc) {
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
  static_assert(B_COUNT <= kBarSlots, "barrier area");
  // groups of 8 lanes pay (ragged-large, g = 8: -3.6 %); groups of 4 measured
  // slower than the per-lane test on prefix+tree (g = 4), so g = 4 stays per lane
  // calls whose records may be split-KV chunks (a workspace with partial
  // states) take the kernel with the float32 partial-state epilogue; the
  // others leave that code out
  auto kern = (p.g % 8 == 0) ? attn_kernel<D, BF16, PAGED, 8, false>
                             : attn_kernel<D, BF16, PAGED, 0, false>;
  if constexpr (!PAGED) {
    if (p.part_o != nullptr)
      kern = (p.g % 8 == 0) ? attn_kernel<D, BF16, PAGED, 8, true>
                            : attn_kernel<D, BF16, PAGED, 0, true>;
  }
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
