// ta_attn.cu -- persistent batched tree-attention kernel for sm_103a.
//
// Computes what ``batch_tree_attn`` of the page "tree_attn.py" computes
// (per q row and head: masked online softmax of sm_scale * q.k in log2
// units, output O / d and lse = m + log2(d)), re-designed for one GB300 SM:
//
//   warp 0      work queue + producer: pops (sequence, q tile, kv head) items
//               in longest-first order, stages the item's per-row DFS enter
//               indices, TMA-loads the packed Q tile into one of two Q
//               buffers and the item's non-empty K/V tiles (64 kv rows each)
//               into a 3-stage ring, with each partial tile's column
//               intervals beside it; it runs up to a whole item ahead
//   warp 1      TMEM owner and tcgen05 issuer: S = Q K^T into one of two TMEM
//               score buffers, then O += P V into the TMEM accumulator
//   warps 2-5   softmax / correction / epilogue, one TMEM lane (= packed row)
//               per thread: tree mask, online softmax with a lazily moved
//               reference max, P (fp16/bf16) into one of two shared buffers,
//               O rescale, final O / l and lse stores
//   warps 6-9   inline RoPE on the staged Q tile (keys arrive rotated: the
//               run rotates them once per call), rotate-half with float32
//               products, rounded to the storage dtype
//
// Every cross-warp hand-off is an mbarrier with a bounded wait.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ta_device.cuh"
#include "ta_launch.h"

namespace ta {
namespace {

constexpr int kThreads = 320;
constexpr int kStages = 3;    // K/V ring depth
constexpr int kQStages = 2;   // Q buffers
constexpr int kSlots = 4;     // work-item slots

enum Bar : int {
  B_ITEM_FULL = 0,                       // [kSlots]
  B_ITEM_EMPTY = B_ITEM_FULL + kSlots,   // [kSlots]
  B_Q_FULL = B_ITEM_EMPTY + kSlots,      // [kQStages]
  B_Q_READY = B_Q_FULL + kQStages,       // [kQStages]
  B_Q_EMPTY = B_Q_READY + kQStages,      // [kQStages]
  B_K_FULL = B_Q_EMPTY + kQStages,       // [kStages]
  B_V_FULL = B_K_FULL + kStages,         // [kStages]
  B_EX_FULL = B_V_FULL + kStages,        // [kStages]
  B_KV_EMPTY = B_EX_FULL + kStages,      // [kStages]
  B_S_FULL = B_KV_EMPTY + kStages,       // [2]
  B_S_FREE = B_S_FULL + 2,               // [2]
  B_P_FREE = B_S_FREE + 2,               // [2]
  B_P_FULL = B_P_FREE + 2,               // [2] one per P buffer: a warp may run a tile ahead
  B_O_FREE = B_P_FULL + 2,
  B_DRAIN,
  B_COUNT
};

struct Item {
  ItemRec r;
  int valid, kvh, pad[14];
  int e_row[kBlockM];  // DFS enter index of every packed row's node (INT_MIN: none)
};
static_assert(sizeof(Item) == 128 + 4 * kBlockM, "item slot size");

struct Misc {
  uint32_t tmem_base;
  int abort;
  int pad[30];
  Item items[kSlots];
};

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;               // 128-byte column blocks per row
  static constexpr int kQAtomBytes = kBlockM * 128;    // 128 rows x 128 bytes
  static constexpr int kKVAtomBytes = kBlockN * 128;   // 64 rows x 128 bytes
  static constexpr int kQBytes = kAtoms * kQAtomBytes;
  static constexpr int kKVBytes = kAtoms * kKVAtomBytes;
  static constexpr int kPBytes = kBlockM * 128;        // 128 x 64 elements = one atom
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQStages * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffP = kOffV + kStages * kKVBytes;
  static constexpr int kOffEX = kOffP + 2 * kPBytes;          // [kStages][kBlockN] int2
  static constexpr int kOffBar = kOffEX + kStages * kBlockN * 8;
  static constexpr int kOffMisc = kOffBar + 64 * 8;
  static constexpr int kSmemUsed = kOffMisc + (int)sizeof(Misc);
  static constexpr int kSmemAlloc = kSmemUsed + 1024;   // room to align the base to 1024
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemS = 128;  // score buffer sb at column 128 + 64 * sb
};

struct Ctx {
  uint8_t* smem;
  uint64_t* bar;
  Misc* misc;
  unsigned int* dev_error;
  unsigned long long limit_ns;
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait(&bar[b], parity, &misc->abort, dev_error, limit_ns);
  }
  // every lane of the warp waits; the warp proceeds only if all lanes saw it
  __device__ bool warp_wait(int b, uint32_t parity) const {
    const bool ok = mbar_wait(&bar[b], parity, &misc->abort, dev_error, limit_ns);
    return __all_sync(0xffffffffu, ok);
  }
  // wait used while draining after an abort: ignores the abort flag
  __device__ bool drain_wait(int b, uint32_t parity) const {
    int no_abort = 0;
    return mbar_wait(&bar[b], parity, &no_abort, dev_error, 200000000ull);
  }
};

// Iterates the non-empty kv tiles of a work item: from the record's inline
// 2-bit classes for short sequences, else from the plan's class bytes.
struct TileIter {
  const uint8_t* cls;
  int kvt, j;
  bool inl;
  uint32_t w[4];
  __device__ TileIter(const ItemRec& r, const uint8_t* classes)
      : cls(classes + r.class_off), kvt(r.kvt), j(-1), inl(r.kvt <= kInlineTiles) {
    if (inl) {
      w[0] = r.cls2[0];
      w[1] = r.cls2[1];
      w[2] = r.cls2[2];
      w[3] = 0;
    }
  }
  // advances to the next non-empty tile; returns its class (0 when done)
  __device__ int next() {
    while (true) {
      ++j;
      if (j >= kvt) return 0;
      int c;
      if (inl) {
        c = (w[j >> 4] >> (2 * (j & 15))) & 3;
      } else {
        if ((j & 15) == 0) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(cls + j));
          w[0] = v.x;
          w[1] = v.y;
          w[2] = v.z;
          w[3] = v.w;
        }
        c = (w[(j & 15) >> 2] >> (8 * (j & 3))) & 0xff;
      }
      if (c != kTileEmpty) return c;
    }
  }
};

// ---------------------------------------------------------------------------
// warp 0: work queue + producer (lane 0 issues; all lanes stage intervals)
// ---------------------------------------------------------------------------
template <int D>
__device__ void run_producer(const Ctx& cx, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const AttnParams& p, int lane) {
  using C = Cfg<D>;
  uint8_t* sQ = cx.smem + C::kOffQ;
  uint8_t* sK = cx.smem + C::kOffK;
  uint8_t* sV = cx.smem + C::kOffV;
  int2* sEX = reinterpret_cast<int2*>(cx.smem + C::kOffEX);
  // the plan kernel wrote the item count; never trust it beyond the table size
  const unsigned long long cap = (unsigned long long)p.max_pairs * (unsigned long long)p.h_kv;
  const unsigned long long n_items = *(volatile unsigned int*)&p.hdr->num_items;
  const unsigned int num_items = (unsigned int)(n_items < cap ? n_items : cap);
  const int g = p.g, R = p.R;
  uint32_t it = 0, kv_it = 0, q_it = 0;
  uint32_t issued[kStages] = {0, 0, 0};
  bool aborted = false;
  unsigned int idx = 0;
  if (lane == 0) idx = atomicAdd(&p.hdr->queue_head, 1u);
  idx = __shfl_sync(0xffffffffu, idx, 0);
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait(B_ITEM_EMPTY + slot, ((it / kSlots) & 1) ^ 1)) { aborted = true; break; }
    Item& s = cx.misc->items[slot];
    if (idx >= num_items) {
      if (lane == 0) {
        s.valid = 0;
        mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
      }
      break;
    }
    if (lane < 4)
      reinterpret_cast<int4*>(&s.r)[lane] =
          __ldg(reinterpret_cast<const int4*>(p.sorted + idx / p.h_kv) + lane);
    const int kvh = idx % p.h_kv;
    // pop the next index now; its round trip overlaps this item's issue
    unsigned int nidx = 0;
    if (lane == 0) nidx = atomicAdd(&p.hdr->queue_head, 1u);
    __syncwarp();
    const ItemRec r = s.r;
    if (r.n_tiles > 0) {
      // the Q tile first: its load overlaps the staging below
      const int qs = q_it % kQStages;
      if (!cx.warp_wait(B_Q_EMPTY + qs, ((q_it / kQStages) & 1) ^ 1)) { aborted = true; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&cx.bar[B_Q_FULL + qs], (uint32_t)(C::kAtoms * 128 * g * R));
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d(sQ + qs * C::kQBytes + a * C::kQAtomBytes, tm_q, &cx.bar[B_Q_FULL + qs],
                      a * 64, kvh * g, r.q_row0);
      }
      ++q_it;
    }
    // DFS enter index of each packed row's tree node
#pragma unroll
    for (int k4 = 0; k4 < kBlockM / 32; ++k4) {
      const int row = k4 * 32 + lane;
      const int qr = row / g;
      int e = INT_MIN;
      if (row < g * R && qr < r.nq)
        e = __ldg(&p.tree_order[2 * (r.tree_base + r.t * R + qr + r.tl - r.qo)]);
      s.e_row[row] = e;
    }
    if (lane == 0) {
      s.valid = 1;
      s.kvh = kvh;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
    idx = __shfl_sync(0xffffffffu, nidx, 0);
    if (r.n_tiles > 0) {
      TileIter ti(r, p.classes);
      for (int n = 0; n < r.n_tiles; ++n) {
        const int cls = ti.next();
        const int j = ti.j;
        const int row0 = r.kv_base + j * kBlockN;
        const int stage = kv_it % kStages;
        if (!cx.warp_wait(B_KV_EMPTY + stage, ((kv_it / kStages) & 1) ^ 1)) { aborted = true; break; }
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)C::kKVBytes;
          mbar_arrive_expect_tx(&cx.bar[B_K_FULL + stage], bytes);
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sK + stage * C::kKVBytes + a * C::kKVAtomBytes, tm_k,
                        &cx.bar[B_K_FULL + stage], a * 64, kvh, row0);
          mbar_arrive_expect_tx(&cx.bar[B_V_FULL + stage], bytes);
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sV + stage * C::kKVBytes + a * C::kKVAtomBytes, tm_v,
                        &cx.bar[B_V_FULL + stage], a * 64, kvh, row0);
        }
        // column intervals of a partial tile for the mask (FULL tiles need none)
        if (cls == kTilePartial) {
          int2* ex = sEX + stage * kBlockN;
#pragma unroll
          for (int q = 0; q < kBlockN / 32; ++q)
            ex[q * 32 + lane] =
                column_interval(p.tree_order, r.tree_base, j * kBlockN + q * 32 + lane, r.kv, r.ts);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_EX_FULL + stage]);
        ++issued[stage];
        ++kv_it;
      }
      if (aborted) break;
    }
    ++it;
  }
  if (aborted && lane == 0) {
    // let every copy already in flight land before the CTA's memory goes away
    for (int qs = 0; qs < kQStages; ++qs) {
      const uint32_t n = q_it / kQStages + (qs < (int)(q_it % kQStages) ? 1 : 0);
      if (n > 0) cx.drain_wait(B_Q_FULL + qs, (n - 1) & 1);
    }
    for (int st = 0; st < kStages; ++st) {
      if (issued[st] > 0) {
        cx.drain_wait(B_K_FULL + st, (issued[st] - 1) & 1);
        cx.drain_wait(B_V_FULL + st, (issued[st] - 1) & 1);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// warp 1: tcgen05 issuer (one thread)
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__device__ void run_mma(const Ctx& cx, uint32_t tmem, const AttnParams& p) {
  using C = Cfg<D>;
  const uint32_t sQ = smem_u32(cx.smem + C::kOffQ);
  const uint32_t sK = smem_u32(cx.smem + C::kOffK);
  const uint32_t sV = smem_u32(cx.smem + C::kOffV);
  const uint32_t sP = smem_u32(cx.smem + C::kOffP);
  constexpr uint32_t idesc_pv = umma_idesc_f16(BF16, 128, D, /*b_mn_major=*/true);
  const int q_bar = p.rotary ? B_Q_READY : B_Q_FULL;
  uint32_t it = 0, kv_it = 0, q_it = 0, o_it = 0;
  bool issued_any = false;
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.wait(B_ITEM_FULL + slot, (it / kSlots) & 1)) break;
    const Item& s = cx.misc->items[slot];
    if (!s.valid) break;
    const ItemRec r = s.r;
    if (r.n_tiles > 0) {
      const int qs = q_it % kQStages;
      if (!cx.wait(q_bar + qs, (q_it / kQStages) & 1)) break;
      ++q_it;
      tc_fence_after();
      const uint32_t qst = sQ + qs * C::kQBytes;
      TileIter ti(r, p.classes);
      bool ok = true;
      // S(m) = Q K(m)^T into score buffer (kv_it + m) & 1
      auto issue_qk = [&](int m, int nvalid) -> bool {
        const uint32_t c = kv_it + m;
        const int stage = c % kStages;
        if (!cx.wait(B_K_FULL + stage, (c / kStages) & 1)) return false;
        const int sb = c & 1;
        if (!cx.wait(B_S_FREE + sb, ((c >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const int n_eff = (nvalid + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(BF16, 128, n_eff, false);
        const uint32_t kst = sK + stage * C::kKVBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          umma_f16(tmem + C::kTmemS + 64 * sb,
                   sw128_desc(qst + (k >> 2) * C::kQAtomBytes + (k & 3) * 32, 0),
                   sw128_desc(kst + (k >> 2) * C::kKVAtomBytes + (k & 3) * 32, 0), idesc,
                   k > 0 ? 1u : 0u);
        }
        umma_commit(&cx.bar[B_S_FULL + sb]);
        issued_any = true;
        if (m == r.n_tiles - 1) umma_commit(&cx.bar[B_Q_EMPTY + qs]);
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
        if (!cx.wait(B_P_FULL + pb, (c >> 1) & 1)) { ok = false; break; }
        if (!cx.wait(B_V_FULL + stage, (c / kStages) & 1)) { ok = false; break; }
        if (n == 0) {
          if (!cx.wait(B_O_FREE, (o_it & 1) ^ 1)) { ok = false; break; }
          ++o_it;
        }
        tc_fence_after();
        const int n_eff = (nv_cur + 15) & ~15;
        const uint32_t vst = sV + stage * C::kKVBytes;
        const uint32_t pst = sP + pb * C::kPBytes;
        for (int k = 0; k < n_eff / 16; ++k) {
          umma_f16(tmem + C::kTmemO, sw128_desc(pst + k * 32, 0),
                   sw128_desc(vst + k * 16 * 128, C::kKVAtomBytes), idesc_pv,
                   (n > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&cx.bar[B_P_FREE + pb]);
        umma_commit(&cx.bar[B_KV_EMPTY + stage]);
        nv_cur = nv_next;
      }
      if (!ok) break;
      kv_it += r.n_tiles;
    }
    mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
  if (cx.misc->abort && issued_any) {
    umma_commit(&cx.bar[B_DRAIN]);
    cx.drain_wait(B_DRAIN, 0);
  }
}

// ---------------------------------------------------------------------------
// warps 2-5: softmax, O correction and epilogue (one packed row per thread)
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__device__ void run_softmax(const Ctx& cx, uint32_t tmem, const AttnParams& p, int warp,
                            int lane) {
  using C = Cfg<D>;
  const int wq = warp & 3;                     // TMEM lane quadrant of this warp
  const int row = wq * 32 + lane;              // packed row = TMEM lane
  const uint32_t t_row = tmem + ((uint32_t)(wq * 32) << 16);
  const int2* sEX = reinterpret_cast<const int2*>(cx.smem + C::kOffEX);
  uint8_t* sP = cx.smem + C::kOffP + row * 128;
  const float c2 = p.scale_log2;
  const int g = p.g, R = p.R;
  const bool in_pack = row < g * R;
  const int qr = in_pack ? row / g : 0;
  const int hh = in_pack ? row - qr * g : 0;
  uint32_t it = 0, gi = 0;  // gi: kv tiles processed by this CTA (S, P and stage index)
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait(B_ITEM_FULL + slot, (it / kSlots) & 1)) return;
    const Item& s = cx.misc->items[slot];
    if (!s.valid) return;
    const ItemRec r = s.r;
    const int kvh = s.kvh;
    const int e_row = s.e_row[row];
    const bool valid = in_pack && qr < r.nq;
    const int head = kvh * g + hh;
    const size_t orow = (size_t)(r.q_row0 + qr) * p.h_q + head;
    float m_ref = -INFINITY, l = 0.f;
    if (r.n_tiles > 0) {
      TileIter ti(r, p.classes);
      for (int n = 0; n < r.n_tiles; ++n, ++gi) {
        const int cls = ti.next();
        const int nvalid = min(kBlockN, r.kv - ti.j * kBlockN);
        const int stage = gi % kStages;
        const int sb = gi & 1;
        // visibility bits of this row for the tile's 64 columns
        uint32_t mw0, mw1;
        if (cls == kTilePartial) {
          if (!cx.warp_wait(B_EX_FULL + stage, (gi / kStages) & 1)) return;
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
        if (!cx.warp_wait(B_S_FULL + sb, (gi >> 1) & 1)) return;
        tc_fence_after();
        // the whole 64-column score row in registers: one TMEM round trip
        float v[64];
        {
          float a[32], b[32];
          const uint32_t t_s = t_row + C::kTmemS + 64 * sb;
          tmem_ld32(t_s, a);
          if (nvalid > 32) tmem_ld32(t_s + 32, b);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = a[i];
            v[32 + i] = nvalid > 32 ? b[i] : 0.f;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_S_FREE + sb]);
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
        // P = exp2(s * c2 - m) on visible columns, in registers
        float l8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) l8[k] = 0.f;
        uint32_t pk[32];
        if (cls == kTileFull) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = ex2_approx(fmaf(v[2 * i], c2, -m_use));
            const float p1 = ex2_approx(fmaf(v[2 * i + 1], c2, -m_use));
            l8[i & 7] += p0 + p1;
            pk[i] = pack2<BF16>(p0, p1);
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
            pk[i] = pack2<BF16>(p0, p1);
          }
        }
        l = l * alpha + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
        // P buffer gi & 1 is free once the PV of tile gi - 2 has completed
        if (!cx.warp_wait(B_P_FREE + (gi & 1), ((gi >> 1) & 1) ^ 1)) return;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const int chunk = cc ^ (row & 7);
          *reinterpret_cast<uint4*>(sP + (gi & 1) * C::kPBytes + chunk * 16) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        // rescale the running O when the reference moved (after the PV of
        // tile gi - 1, which is the last one that wrote O)
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t pv = gi - 1;
          if (!cx.warp_wait(B_P_FREE + (pv & 1), (pv >> 1) & 1)) return;
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
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_P_FULL + (gi & 1)]);
      }
      // epilogue: wait for the last PV (tile gi - 1), then O / l and lse
      const uint32_t pv = gi - 1;
      if (!cx.warp_wait(B_P_FREE + (pv & 1), (pv >> 1) & 1)) return;
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? m_ref + log2f(l) : -INFINITY;
    // O / l in the storage dtype goes to the P buffers first (both are free:
    // the item's last PV has completed), as 128-byte swizzled rows; d in
    // [64a, 64a + 64) lands in buffer a
    uint8_t* ostage = cx.smem + C::kOffP;
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
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(o[2 * i] * inv, o[2 * i + 1] * inv);
      uint8_t* rowp = ostage + (oc >> 1) * C::kPBytes + row * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(rowp + ((((oc & 1) * 4 + cc) ^ (row & 7)) * 16)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
    }
    if (valid) p.lse[orow] = lse_v;
    tc_fence_before();
    __syncwarp();
    if (lane == 0 && r.n_tiles > 0) mbar_arrive(&cx.bar[B_O_FREE]);  // O is out of TMEM
    // each warp writes its own 32 rows with whole-warp coalesced 16-byte stores
    {
      constexpr int kChunks = D / 8;              // 16-byte chunks per row
      constexpr int kRowsPerStep = 32 / kChunks;
      const int ch = lane % kChunks;
      uint16_t* outp = reinterpret_cast<uint16_t*>(p.out);
#pragma unroll 4
      for (int st = 0; st < 32 / kRowsPerStep; ++st) {
        const int src = st * kRowsPerStep + lane / kChunks;  // row within the quadrant
        const long long ro = __shfl_sync(0xffffffffu, (long long)orow, src);
        const int ok = __shfl_sync(0xffffffffu, valid ? 1 : 0, src);
        const int rr = wq * 32 + src;
        const uint4 val = *reinterpret_cast<const uint4*>(
            ostage + (ch >> 3) * C::kPBytes + rr * 128 + (((ch & 7) ^ (rr & 7)) * 16));
        if (ok) *reinterpret_cast<uint4*>(outp + ro * D + ch * 8) = val;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
}

// ---------------------------------------------------------------------------
// warps 6-9: inline RoPE on the staged Q tile
// ---------------------------------------------------------------------------
// Task = (q row of the tile, 16-byte block c of the first half of the head
// dimension): one load of the row's cos/sin for that block, applied to the
// block and its partner block in the second half, for each of the row's g
// heads (packed rows qr * g .. qr * g + g - 1).
template <int D, bool BF16>
__device__ void rope_q_tile(uint8_t* tile, const float2* __restrict__ cs, long long tok0, int nq,
                            int g, int t) {
  constexpr int kHalfChunks = D / 16;  // 16-byte blocks in half a row
  constexpr int kBatch = 2;            // tasks whose loads are in flight together
  const int ntask = nq * kHalfChunks;
  for (int t0 = t; t0 < ntask; t0 += 128 * kBatch) {
    float4 cv[kBatch][4];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int task = t0 + u * 128;
      if (task < ntask) {
        const int qr = task / kHalfChunks, c = task % kHalfChunks;
        const float4* csp = reinterpret_cast<const float4*>(cs + (tok0 + qr) * (D / 2) + c * 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) cv[u][i] = __ldg(csp + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int task = t0 + u * 128;
      if (task >= ntask) continue;
      const int qr = task / kHalfChunks, c = task % kHalfChunks;
      for (int h = 0; h < g; ++h) {
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

template <int D, bool BF16>
__device__ void run_rope(const Ctx& cx, const AttnParams& p, int warp, int lane) {
  using C = Cfg<D>;
  const int t = (warp - 6) * 32 + lane;
  uint8_t* sQ = cx.smem + C::kOffQ;
  const int g = p.g, R = p.R;
  uint32_t it = 0, q_it = 0;
  for (;;) {
    const int slot = it % kSlots;
    if (!cx.warp_wait(B_ITEM_FULL + slot, (it / kSlots) & 1)) return;
    const Item& s = cx.misc->items[slot];
    if (!s.valid) return;
    const ItemRec r = s.r;
    if (r.n_tiles > 0) {
      const int qs = q_it % kQStages;
      if (!cx.warp_wait(B_Q_FULL + qs, (q_it / kQStages) & 1)) return;
      ++q_it;
      // q row r of the tile takes the position of its own tree node's kv slot
      const long long qtok0 = (long long)r.kv_base + r.ts + (r.tl - r.qo) + (long long)r.t * R;
      rope_q_tile<D, BF16>(sQ + qs * C::kQBytes, p.rope_cs, qtok0, r.nq, g, t);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cx.bar[B_Q_READY + qs]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    ++it;
  }
}

// ---------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctx cx;
  cx.smem = smem;
  cx.bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  cx.misc = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  cx.dev_error = &p.hdr->error;
  cx.limit_ns = p.timeout_ns;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    const uint32_t consumers = 5u + (p.rotary ? 4u : 0u);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&cx.bar[B_ITEM_FULL + i], 1);
      mbar_init(&cx.bar[B_ITEM_EMPTY + i], consumers);
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&cx.bar[B_Q_FULL + i], 1);
      mbar_init(&cx.bar[B_Q_READY + i], 4);
      mbar_init(&cx.bar[B_Q_EMPTY + i], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&cx.bar[B_K_FULL + i], 1);
      mbar_init(&cx.bar[B_V_FULL + i], 1);
      mbar_init(&cx.bar[B_EX_FULL + i], 1);
      mbar_init(&cx.bar[B_KV_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cx.bar[B_S_FULL + i], 1);
      mbar_init(&cx.bar[B_S_FREE + i], 4);
      mbar_init(&cx.bar[B_P_FREE + i], 1);
      mbar_init(&cx.bar[B_P_FULL + i], 4);
    }
    mbar_init(&cx.bar[B_O_FREE], 4);
    mbar_init(&cx.bar[B_DRAIN], 1);
    cx.misc->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // rows of the Q buffers that no TMA box covers (g * R < 128) must read as zero
  if (p.g * p.R < kBlockM) {
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::kOffQ);
    for (int i = threadIdx.x; i < kQStages * C::kQBytes / 16; i += kThreads)
      q4[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(&cx.misc->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cx.misc->tmem_base;

  if (warp == 0) {
    run_producer<D>(cx, &tm_q, &tm_k, &tm_v, p, lane);
  } else if (warp == 1) {
    if (lane == 0) run_mma<D, BF16>(cx, tmem, p);
  } else if (warp < 6) {
    run_softmax<D, BF16>(cx, tmem, p, warp, lane);
  } else if (p.rotary) {
    run_rope<D, BF16>(cx, p, warp, lane);
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
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

template <int D, bool BF16>
cudaError_t launch_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const AttnParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  static_assert(C::kSmemAlloc <= 227 * 1024, "shared memory budget");
  static_assert(B_COUNT <= 64, "barrier area");
  auto kern = attn_kernel<D, BF16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::kSmemAlloc, stream>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

template cudaError_t launch_attn<64, false>(const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const AttnParams&, int,
                                            cudaStream_t);
template cudaError_t launch_attn<64, true>(const CUtensorMap&, const CUtensorMap&,
                                           const CUtensorMap&, const AttnParams&, int,
                                           cudaStream_t);
template cudaError_t launch_attn<128, false>(const CUtensorMap&, const CUtensorMap&,
                                             const CUtensorMap&, const AttnParams&, int,
                                             cudaStream_t);
template cudaError_t launch_attn<128, true>(const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const AttnParams&, int,
                                            cudaStream_t);

}  // namespace ta
