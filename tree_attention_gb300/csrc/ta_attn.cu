// ta_attn.cu -- persistent batched tree-attention kernel for sm_103a.
//
// Computes what ``batch_tree_attn`` of the page "tree_attn.py" computes
// (per q row and head: masked online softmax of sm_scale * q.k in log2
// units, output O / d and lse = m + log2(d)), re-designed for one GB300 SM:
//
//   warp 0      work queue + TMA producer: pops (sequence, q tile, kv head)
//               items in longest-first order, loads the packed Q tile once
//               and the non-empty K/V tiles of the item into a 2-stage ring
//   warp 1      TMEM owner and tcgen05 issuer: S = Q K^T into one of two TMEM
//               score buffers, then O += P V into the TMEM accumulator
//   warps 2-5   softmax / correction / epilogue, one TMEM lane (= packed row)
//               per thread: tree mask, online softmax with a lazily moved
//               reference max, P (fp16/bf16) to shared memory, O rescale,
//               final O / l and lse stores
//   warps 6-9   inline RoPE: rotate the staged Q and K tiles in shared memory
//               (rotate-half, float32 products, rounded to the storage dtype)
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
constexpr int kStages = 2;

enum Bar : int {
  B_ITEM_FULL = 0,    // [2]
  B_ITEM_EMPTY = 2,   // [2]
  B_Q_FULL = 4,
  B_Q_READY = 5,
  B_Q_EMPTY = 6,
  B_K_FULL = 7,       // [2]
  B_V_FULL = 9,       // [2]
  B_K_READY = 11,     // [2]
  B_KV_EMPTY = 13,    // [2]
  B_S_FULL = 15,      // [2]
  B_S_FREE = 17,      // [2]
  B_P_FULL = 19,
  B_P_FREE = 20,
  B_O_FREE = 21,
  B_DRAIN = 22,
  B_COUNT = 23
};

struct Item {
  int valid, b, t, kvh, n_tiles, class_off, q_row0, qo, kv, tl, ts, kv_base, tree_base, nq;
  int pad[2];
};

struct Misc {
  uint32_t tmem_base;
  int abort;
  int pad[14];
  Item items[2];
};

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;           // 128-byte column blocks per row
  static constexpr int kAtomBytes = 128 * 128;    // 128 rows x 128 bytes
  static constexpr int kTileBytes = kAtoms * kAtomBytes;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffEX = kOffP + 2 * kAtomBytes;   // P is 128 x 128 elements
  static constexpr int kOffBar = kOffEX + 4 * kBlockN * 8;
  static constexpr int kOffMisc = kOffBar + 32 * 8;
  static constexpr int kSmemUsed = kOffMisc + (int)sizeof(Misc);
  // request more than half of an SM's shared memory so that exactly one CTA
  // (and one 512-column TMEM allocation) lives on each SM
  static constexpr int kSmemAlloc =
      (kSmemUsed + 1024) > 120 * 1024 ? (kSmemUsed + 1024) : 120 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemS = 128;  // S buffer sb at column 128 + 128 * sb
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

// Iterates the non-empty kv tiles of a work item from the plan's class bytes.
struct TileIter {
  const uint8_t* cls;
  int kvt, j;
  uint32_t w[4];
  __device__ TileIter(const uint8_t* c, int n) : cls(c), kvt(n), j(-1) {}
  // advances to the next non-empty tile; returns its class (0 when done)
  __device__ int next() {
    while (true) {
      ++j;
      if (j >= kvt) return 0;
      if ((j & 15) == 0) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(cls + j));
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
      }
      const int c = (w[(j & 15) >> 2] >> (8 * (j & 3))) & 0xff;
      if (c != kTileEmpty) return c;
    }
  }
};

__device__ __forceinline__ int kv_tiles(int kv) { return (kv + kBlockN - 1) / kBlockN; }

// ---------------------------------------------------------------------------
// warp 0: work queue + TMA producer (one thread)
// ---------------------------------------------------------------------------
template <int D>
__device__ void run_producer(const Ctx& cx, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const AttnParams& p) {
  using C = Cfg<D>;
  uint8_t* sQ = cx.smem + C::kOffQ;
  uint8_t* sK = cx.smem + C::kOffK;
  uint8_t* sV = cx.smem + C::kOffV;
  // the plan kernel wrote the item count; never trust it beyond the table size
  const unsigned long long cap = (unsigned long long)p.max_pairs * (unsigned long long)p.h_kv;
  unsigned long long n_items = *(volatile unsigned int*)&p.hdr->num_items;
  const unsigned int num_items = (unsigned int)(n_items < cap ? n_items : cap);
  uint32_t it = 0, kv_it = 0, q_it = 0;
  uint32_t issued[kStages] = {0, 0};
  bool aborted = false;
  for (;;) {
    const int slot = it & 1;
    if (!cx.wait(B_ITEM_EMPTY + slot, ((it >> 1) & 1) ^ 1)) { aborted = true; break; }
    Item& s = cx.misc->items[slot];
    const unsigned int idx = atomicAdd(&p.hdr->queue_head, 1u);
    if (idx >= num_items) {
      s.valid = 0;
      mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
      break;
    }
    const int pair = __ldg(&p.sorted[idx / p.h_kv]);
    const int kvh = idx % p.h_kv;
    if (pair < 0 || pair >= p.max_pairs) {   // a workspace that was never zero-filled
      atomicOr(&p.hdr->error, DEVERR_BAD_INDPTR);
      s.valid = 0;
      mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
      break;
    }
    const PairInfo pi = reinterpret_cast<const PairInfo*>(p.pairs)[pair];
    const int b = pi.b;
    const int q0 = __ldg(&p.q_indptr[b]), q1 = __ldg(&p.q_indptr[b + 1]);
    const int k0 = __ldg(&p.kv_indptr[b]), k1 = __ldg(&p.kv_indptr[b + 1]);
    const int m0 = __ldg(&p.mn_indptr[b]), m1 = __ldg(&p.mn_indptr[b + 1]);
    s.valid = 1;
    s.b = b;
    s.t = pi.t;
    s.kvh = kvh;
    s.n_tiles = pi.n_tiles;
    s.class_off = pi.class_off;
    s.q_row0 = q0 + pi.t * p.R;
    s.qo = q1 - q0;
    s.kv = k1 - k0;
    s.tl = m1 - m0;
    s.ts = s.kv - s.tl;
    s.kv_base = k0;
    s.tree_base = m0;
    s.nq = min(p.R, s.qo - pi.t * p.R);
    mbar_arrive(&cx.bar[B_ITEM_FULL + slot]);
    if (pi.n_tiles > 0) {
      if (!cx.wait(B_Q_EMPTY, (q_it & 1) ^ 1)) { aborted = true; break; }
      mbar_arrive_expect_tx(&cx.bar[B_Q_FULL], (uint32_t)(C::kAtoms * 128 * p.g * p.R));
#pragma unroll
      for (int a = 0; a < C::kAtoms; ++a)
        tma_load_3d(sQ + a * C::kAtomBytes, tm_q, &cx.bar[B_Q_FULL], a * 64, kvh * p.g,
                    s.q_row0);
      ++q_it;
      TileIter ti(p.classes + pi.class_off, kv_tiles(s.kv));
      const int kv = s.kv;
      for (int n = 0; n < pi.n_tiles; ++n) {
        ti.next();
        const int j = ti.j;
        const int stage = kv_it & 1;
        if (!cx.wait(B_KV_EMPTY + stage, ((kv_it >> 1) & 1) ^ 1)) { aborted = true; break; }
        const int nvalid = min(kBlockN, kv - j * kBlockN);
        const int nbox = nvalid > kKvBoxRows ? 2 : 1;
        const uint32_t bytes = (uint32_t)(C::kAtoms * nbox * kKvBoxRows * 128);
        const int row0 = k0 + j * kBlockN;
        mbar_arrive_expect_tx(&cx.bar[B_K_FULL + stage], bytes);
        for (int a = 0; a < C::kAtoms; ++a)
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_3d(sK + stage * C::kTileBytes + a * C::kAtomBytes + bx * kKvBoxRows * 128,
                        tm_k, &cx.bar[B_K_FULL + stage], a * 64, kvh, row0 + bx * kKvBoxRows);
        mbar_arrive_expect_tx(&cx.bar[B_V_FULL + stage], bytes);
        for (int a = 0; a < C::kAtoms; ++a)
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_3d(sV + stage * C::kTileBytes + a * C::kAtomBytes + bx * kKvBoxRows * 128,
                        tm_v, &cx.bar[B_V_FULL + stage], a * 64, kvh, row0 + bx * kKvBoxRows);
        ++issued[stage];
        ++kv_it;
      }
      if (aborted) break;
    }
    ++it;
  }
  if (aborted) {
    // let every copy already in flight land before the CTA's memory goes away
    if (q_it > 0) cx.drain_wait(B_Q_FULL, (q_it - 1) & 1);
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
  const int k_bar = p.rotary ? B_K_READY : B_K_FULL;
  uint32_t it = 0, kv_it = 0, s_it = 0, q_it = 0, o_it = 0, pf_it = 0;
  bool issued_any = false;
  for (;;) {
    const int slot = it & 1;
    if (!cx.wait(B_ITEM_FULL + slot, (it >> 1) & 1)) break;
    const Item s = cx.misc->items[slot];
    if (!s.valid) break;
    if (s.n_tiles > 0) {
      if (!cx.wait(q_bar, q_it & 1)) break;
      ++q_it;
      tc_fence_after();
      TileIter ti(p.classes + s.class_off, kv_tiles(s.kv));
      int nv_next = 0;
      bool ok = true;
      // S(m) = Q K(m)^T into score buffer s_it & 1
      auto issue_qk = [&](int m, int nvalid) -> bool {
        const uint32_t c = kv_it + m;
        const int stage = c & 1;
        if (!cx.wait(k_bar + stage, (c >> 1) & 1)) return false;
        const int sb = s_it & 1;
        if (!cx.wait(B_S_FREE + sb, ((s_it >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const int n_eff = (nvalid + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(BF16, 128, n_eff, false);
        const uint32_t kst = sK + stage * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = (k >> 2) * C::kAtomBytes + (k & 3) * 32;
          umma_f16(tmem + C::kTmemS + 128 * sb, sw128_desc(sQ + koff, 0),
                   sw128_desc(kst + koff, 0), idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&cx.bar[B_S_FULL + sb]);
        issued_any = true;
        ++s_it;
        if (m == s.n_tiles - 1) umma_commit(&cx.bar[B_Q_EMPTY]);
        return true;
      };
      ti.next();
      int nv_cur = min(kBlockN, s.kv - ti.j * kBlockN);
      if (!issue_qk(0, nv_cur)) break;
      for (int n = 0; n < s.n_tiles; ++n) {
        if (n + 1 < s.n_tiles) {
          ti.next();
          nv_next = min(kBlockN, s.kv - ti.j * kBlockN);
          if (!issue_qk(n + 1, nv_next)) { ok = false; break; }
        }
        const uint32_t c = kv_it + n;
        const int stage = c & 1;
        if (!cx.wait(B_P_FULL, pf_it & 1)) { ok = false; break; }
        ++pf_it;
        if (!cx.wait(B_V_FULL + stage, (c >> 1) & 1)) { ok = false; break; }
        if (n == 0) {
          if (!cx.wait(B_O_FREE, (o_it & 1) ^ 1)) { ok = false; break; }
          ++o_it;
        }
        tc_fence_after();
        const int n_eff = (nv_cur + 15) & ~15;
        const uint32_t vst = sV + stage * C::kTileBytes;
        for (int k = 0; k < n_eff / 16; ++k) {
          const uint32_t aoff = (k >> 2) * C::kAtomBytes + (k & 3) * 32;
          umma_f16(tmem + C::kTmemO, sw128_desc(sP + aoff, 0),
                   sw128_desc(vst + k * 16 * 128, C::kAtomBytes), idesc_pv,
                   (n > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&cx.bar[B_P_FREE]);
        umma_commit(&cx.bar[B_KV_EMPTY + stage]);
        nv_cur = nv_next;
      }
      if (!ok) break;
      kv_it += s.n_tiles;
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
  int2* ex = reinterpret_cast<int2*>(cx.smem + C::kOffEX) + (warp - 2) * kBlockN;
  uint8_t* sP = cx.smem + C::kOffP;
  const float c2 = p.scale_log2;
  const int g = p.g, R = p.R;
  const bool in_pack = row < g * R;
  const int qr = in_pack ? row / g : 0;
  const int hh = in_pack ? row - qr * g : 0;
  uint32_t it = 0, s_it = 0, pf_it = 0;
  for (;;) {
    const int slot = it & 1;
    if (!cx.warp_wait(B_ITEM_FULL + slot, (it >> 1) & 1)) return;
    const Item s = cx.misc->items[slot];
    if (!s.valid) return;
    const bool valid = in_pack && qr < s.nq;
    const int head = s.kvh * g + hh;
    const size_t orow = (size_t)(s.q_row0 + qr) * p.h_q + head;
    int e_row = INT_MIN;
    if (valid) e_row = __ldg(&p.tree_order[2 * (s.tree_base + s.t * R + qr + s.tl - s.qo)]);
    float m_ref = -INFINITY, l = 0.f;
    if (s.n_tiles > 0) {
      TileIter ti(p.classes + s.class_off, kv_tiles(s.kv));
      for (int n = 0; n < s.n_tiles; ++n) {
        const int cls = ti.next();
        const int j = ti.j;
        const int nvalid = min(kBlockN, s.kv - j * kBlockN);
        const int nchunk = (nvalid + 31) >> 5;
        const int sb = s_it & 1;
        // visibility bits of this row for the tile's columns
        uint32_t mw[4];
        if (cls == kTilePartial) {
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ex[q * 32 + lane] =
                column_interval(p.tree_order, s.tree_base, j * kBlockN + q * 32 + lane, s.kv, s.ts);
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t bits = 0;
            const int4* e4 = reinterpret_cast<const int4*>(ex + q * 32);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int4 v = e4[i];
              bits |= (uint32_t)(v.x <= e_row && e_row < v.y) << (2 * i);
              bits |= (uint32_t)(v.z <= e_row && e_row < v.w) << (2 * i + 1);
            }
            mw[q] = bits;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int rem = nvalid - q * 32;
            mw[q] = rem >= 32 ? 0xffffffffu : (rem > 0 ? ((1u << rem) - 1u) : 0u);
          }
        }
        if (!cx.warp_wait(B_S_FULL + sb, (s_it >> 1) & 1)) return;
        tc_fence_after();
        const uint32_t t_s = t_row + C::kTmemS + 128 * sb;
        // pass 1: masked row max in log2 units
        float mx = -INFINITY;
        for (int q = 0; q < nchunk; ++q) {
          float v[32];
          tmem_ld32(t_s + q * 32, v);
          tmem_wait_ld();
          const uint32_t bits = mw[q];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if ((bits >> i) & 1u) mx = fmaxf(mx, v[i] * c2);
        }
        // move the reference max only when it grew by more than 2^8; the
        // final O / l and lse = m + log2(l) do not depend on the reference
        const float m_new = fmaxf(m_ref, mx);
        float ref = m_ref;
        if (m_new > m_ref + 8.f) ref = m_new;
        const float alpha = (ref == m_ref) ? 1.f : ex2_approx(m_ref - ref);
        l *= alpha;
        m_ref = ref;
        const float m_use = (ref == -INFINITY) ? 0.f : ref;
        if (n > 0) {
          if (!cx.warp_wait(B_P_FREE, pf_it & 1)) return;
          ++pf_it;
          tc_fence_after();
        }
        // pass 2: P = exp2(s * c2 - m) on visible columns, row sum, P -> smem
        for (int q = 0; q < nchunk; ++q) {
          float v[32];
          tmem_ld32(t_s + q * 32, v);
          tmem_wait_ld();
          const uint32_t bits = mw[q];
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ((bits >> (2 * i)) & 1u) ? ex2_approx(fmaf(v[2 * i], c2, -m_use)) : 0.f;
            const float p1 =
                ((bits >> (2 * i + 1)) & 1u) ? ex2_approx(fmaf(v[2 * i + 1], c2, -m_use)) : 0.f;
            l += p0 + p1;
            pk[i] = pack2<BF16>(p0, p1);
          }
          // columns q*32 .. q*32+31 = 128-byte atom q/2, 16-byte chunks (q&1)*4 .. +3
          uint8_t* prow = sP + (q >> 1) * C::kAtomBytes + row * 128;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int chunk = ((q & 1) * 4 + cc) ^ (row & 7);
            *reinterpret_cast<uint4*>(prow + chunk * 16) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_S_FREE + sb]);
        ++s_it;
        // rescale the running O when the reference moved (PV of the previous
        // tile is complete: P_FREE was awaited above)
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int oc = 0; oc < D / 32; ++oc) {
            float v[32];
            tmem_ld32(t_row + C::kTmemO + oc * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_row + C::kTmemO + oc * 32, v);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_P_FULL]);
      }
      // epilogue: wait for the last PV, then O / l and the base-2 lse
      if (!cx.warp_wait(B_P_FREE, pf_it & 1)) return;
      ++pf_it;
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? m_ref + log2f(l) : -INFINITY;
    using T = uint16_t;
    T* orow_ptr = reinterpret_cast<T*>(p.out) + orow * D;
#pragma unroll
    for (int oc = 0; oc < D / 32; ++oc) {
      float v[32];
      if (s.n_tiles > 0) {
        tmem_ld32(t_row + C::kTmemO + oc * 32, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      if (valid) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(v[2 * i] * inv, v[2 * i + 1] * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow_ptr + oc * 32);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          dst[cc] = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      }
    }
    if (valid) p.lse[orow] = lse_v;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (s.n_tiles > 0) mbar_arrive(&cx.bar[B_O_FREE]);
      mbar_arrive(&cx.bar[B_ITEM_EMPTY + slot]);
    }
    ++it;
  }
}

// ---------------------------------------------------------------------------
// warps 6-9: inline RoPE on the staged Q and K tiles
// ---------------------------------------------------------------------------
// Rotate rows [0, nrows) of a 128-row tile in shared memory.  ``token_of``
// maps a tile row to its kv-token index (or -1 to leave the row as is).
template <int D, bool BF16, typename TokenOf>
__device__ void rope_tile(uint8_t* tile, const float2* __restrict__ cs, int rw, int lane,
                          TokenOf token_of) {
  constexpr int kHalfChunks = D / 16;          // 16-byte chunks in half a row
  constexpr int kRowsPerPass = 32 / kHalfChunks;
  const int sub = lane / kHalfChunks;
  const int c = lane % kHalfChunks;
  for (int r0 = rw * 32; r0 < rw * 32 + 32; r0 += kRowsPerPass) {
    const int row = r0 + sub;
    const long long tok = token_of(row);
    if (tok < 0) continue;
    // element block [8c, 8c+8) of the first half and its partner block in the second
    uint8_t *lo, *hi;
    if constexpr (D == 128) {
      lo = tile + row * 128 + ((c ^ (row & 7)) * 16);
      hi = tile + 128 * 128 + row * 128 + ((c ^ (row & 7)) * 16);
    } else {
      lo = tile + row * 128 + ((c ^ (row & 7)) * 16);
      hi = tile + row * 128 + (((c + 4) ^ (row & 7)) * 16);
    }
    const uint4 a = *reinterpret_cast<const uint4*>(lo);
    const uint4 b = *reinterpret_cast<const uint4*>(hi);
    const float4* csp = reinterpret_cast<const float4*>(cs + tok * (D / 2) + c * 8);
    float cosv[8], sinv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = __ldg(csp + i);
      cosv[2 * i] = t.x;
      sinv[2 * i] = t.y;
      cosv[2 * i + 1] = t.z;
      sinv[2 * i + 1] = t.w;
    }
    const uint32_t au[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bu[4] = {b.x, b.y, b.z, b.w};
    uint32_t ao[4], bo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x0 = unpack2<BF16>(au[i]);
      const float2 x1 = unpack2<BF16>(bu[i]);
      const float c0 = cosv[2 * i], s0 = sinv[2 * i], c1 = cosv[2 * i + 1], s1 = sinv[2 * i + 1];
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

template <int D, bool BF16>
__device__ void run_rope(const Ctx& cx, const AttnParams& p, int warp, int lane) {
  using C = Cfg<D>;
  const int rw = warp - 6;
  uint8_t* sQ = cx.smem + C::kOffQ;
  uint8_t* sK = cx.smem + C::kOffK;
  const int g = p.g, R = p.R;
  uint32_t it = 0, kv_it = 0, q_it = 0;
  for (;;) {
    const int slot = it & 1;
    if (!cx.warp_wait(B_ITEM_FULL + slot, (it >> 1) & 1)) return;
    const Item s = cx.misc->items[slot];
    if (!s.valid) return;
    if (s.n_tiles > 0) {
      if (!cx.warp_wait(B_Q_FULL, q_it & 1)) return;
      ++q_it;
      // q row r of the tile takes the position of its own tree node's kv slot
      const long long qtok0 = (long long)s.kv_base + s.ts + (s.tl - s.qo) + (long long)s.t * R;
      rope_tile<D, BF16>(sQ, p.rope_cs, rw, lane, [&](int row) -> long long {
        if (row >= g * R) return -1;
        const int qr = row / g;
        return qr < s.nq ? qtok0 + qr : -1;
      });
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cx.bar[B_Q_READY]);
      TileIter ti(p.classes + s.class_off, kv_tiles(s.kv));
      for (int n = 0; n < s.n_tiles; ++n) {
        ti.next();
        const int j = ti.j;
        const int nvalid = min(kBlockN, s.kv - j * kBlockN);
        const uint32_t c = kv_it + n;
        const int stage = c & 1;
        if (!cx.warp_wait(B_K_FULL + stage, (c >> 1) & 1)) return;
        const long long ktok0 = (long long)s.kv_base + (long long)j * kBlockN;
        rope_tile<D, BF16>(sK + stage * C::kTileBytes, p.rope_cs, rw, lane,
                           [&](int row) -> long long { return row < nvalid ? ktok0 + row : -1; });
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cx.bar[B_K_READY + stage]);
      }
      kv_it += s.n_tiles;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cx.bar[B_ITEM_FULL + i], 1);
      mbar_init(&cx.bar[B_ITEM_EMPTY + i], consumers);
      mbar_init(&cx.bar[B_K_FULL + i], 1);
      mbar_init(&cx.bar[B_V_FULL + i], 1);
      mbar_init(&cx.bar[B_K_READY + i], 4);
      mbar_init(&cx.bar[B_KV_EMPTY + i], 1);
      mbar_init(&cx.bar[B_S_FULL + i], 1);
      mbar_init(&cx.bar[B_S_FREE + i], 4);
    }
    mbar_init(&cx.bar[B_Q_FULL], 1);
    mbar_init(&cx.bar[B_Q_READY], 4);
    mbar_init(&cx.bar[B_Q_EMPTY], 1);
    mbar_init(&cx.bar[B_P_FULL], 4);
    mbar_init(&cx.bar[B_P_FREE], 1);
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
  // rows of the Q tile that no TMA box covers (g * R < 128) must read as zero
  if (p.g * p.R < kBlockM) {
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::kOffQ);
    for (int i = threadIdx.x; i < C::kTileBytes / 16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(&cx.misc->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cx.misc->tmem_base;

  if (warp == 0) {
    if (lane == 0) run_producer<D>(cx, &tm_q, &tm_k, &tm_v, p);
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
