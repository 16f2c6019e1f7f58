// Split-KV paged decode: persistent warps, each with its own TMA ring.
//
// Same partition and partial states as the rest of the library (vllm-rlt PR
// #128, "Purpose", decode bullets: each row's keys cut into NSPLIT
// contiguous, tile-aligned parts chosen from the row's own length, an fp32
// partial softmax state per part, merged by a second kernel).  What changes
// is how the bytes move, because decode is bound by HBM bandwidth:
//
//  * A work item is (row, KV head, split, 16-row block of GQA-packed query
//    rows).  Each warp takes one item at a time from a counter in the
//    workspace and streams the item's keys in 16-token page slots: one TMA
//    box per slot for K and one for V (16 keys x the whole d of one head,
//    as 128-byte pieces), straight from the block table into the warp's
//    private ring of NS slots.  The warp keeps
//    NS-1 slots in flight and prefetches across item boundaries, so HBM
//    never waits for a warp to start its next item.  Eight warps per CTA
//    (four for 16 KB slots) give each SM sub-partition two independent
//    chains of dependent work to interleave.
//  * The math per slot is warp-level MMA (m16n8k16) on the transposed
//    products, keys on the M side: S^T = K Q^T, then O^T += V^T P^T.  Q is
//    the B operand of S^T and lives in registers for the whole item; K and
//    V are read once each with ldmatrix (V transposed by ldmatrix itself);
//    P^T is S^T's accumulator moved across lanes with movmatrix.  The
//    online softmax reduces over the 8 lanes that share a query row, and a
//    row's exponent reference moves only when its maximum passes it by more
//    than a factor of 256, so O^T is rarely rescaled.  At the end of an item
//    the warp writes (acc[d], m, l) of its rows for that split.
//  * fp8 E5M2 caches (1Cat-vLLM PR #616, original description: an fp8_e5m2
//    KV cache dequantized in the kernel): an E5M2 code in the high byte of a
//    16-bit word is the same binary16 value.  K words of four codes widen
//    into two binary16 pairs (Q's reduction index is permuted to match);
//    V is loaded by ldmatrix.trans as code pairs of two keys, and one byte
//    permute per operand register places the codes.  The per-tensor k_scale
//    is folded into the logit scale, v_scale into the merge.
//  * No block-wide barrier anywhere: warps only wait on their own mbarriers.
//    All waits are clock-bounded.
//
// The result of an item depends only on its row's data and length, never on
// which warp ran it or when, so the outputs stay bitwise batch-invariant.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_sm100.cuh"

namespace pa {
bool encode_kv_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                   int64_t tokens);

// The cache as (128-byte piece, token, piece index, head) with boxes of one
// 16-token page slot of one head, every piece: [piece][16 keys][128 B].
bool encode_slot_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                     int64_t tokens);

namespace {

using namespace sm100;

template <int D, bool KV8>
struct DecCfg {
  static constexpr int ELT = KV8 ? 1 : 2;
  static constexpr int NCH = D * ELT / 128;                // 128-byte boxes per key row
  static constexpr int SEGS = D * ELT / 16;                // 16-byte segments per key row
  static constexpr uint32_t HALF = 16 * D * ELT;           // K (or V) of one 16-key slot
  static constexpr uint32_t SLOT = 2 * HALF;
  static constexpr int W = SLOT >= 16384 ? 4 : 8;          // warps per CTA, one ring each
  static constexpr int NS_FIT = (224 * 1024) / (W * SLOT);
  static constexpr int G = NS_FIT >= 6 ? 2 : 1;            // slots consumed per iteration
  static constexpr int NS = (NS_FIT < 16 ? NS_FIT : 16) / G * G;  // ring slots per warp
  static constexpr uint32_t OFF_BAR = W * NS * SLOT;       // all rings first (1 KB aligned)
  static constexpr uint32_t OFF_META = OFF_BAR + W * NS * 8;
  static constexpr uint32_t SMEM = OFF_META + W * NS * 8 + 1024;
  static_assert(SLOT % 1024 == 0, "slot alignment");
  static_assert(NS >= 2 * G && NS % G == 0 && NS <= 32, "ring depth");
  static_assert(SMEM <= 232448, "shared memory budget");
};

constexpr int META_BAD = 1 << 30;  // block-table entry out of range: no copy
constexpr int META_PAD = 1 << 29;  // padding slot of an item: no copy

// Waits for the phase with the given parity; every lane polls, lane 0 alone
// decides to give up (after WAIT_LIMIT_CYCLES), so the warp leaves together.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, int lane,
                                               uint32_t* err) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((it & WAIT_CHECK_MASK) == WAIT_CHECK_MASK) {
      const int late = __shfl_sync(0xffffffffu, (int)(clock64() - t0 > WAIT_LIMIT_CYCLES), 0);
      if (late) {
        if (lane == 0) atomicOr(err, PA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Byte offset of 16-byte segment `seg` of key row `key` (0..15) in a slot
// half: [segs / 8][16 rows][128 B] with the 128-byte swizzle the TMA boxes
// produce (16-byte unit index XOR row % 8).  Eight consecutive rows at one
// segment fall in eight different bank groups.
__device__ __forceinline__ uint32_t seg_off(int key, int seg) {
  return (uint32_t)((seg >> 3) * 2048 + key * 128 + (((seg & 7) ^ (key & 7)) << 4));
}

// 8x8 transpose of 16-bit elements across the warp: lane (g, t) gives
// M[g][2t..2t+1] and receives M[2t][g], M[2t+1][g].
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// A binary16 pair (as produced from E5M2 codes) in the compute type.
template <typename T>
__device__ __forceinline__ uint32_t h2_to(uint32_t h);
template <>
__device__ __forceinline__ uint32_t h2_to<__half>(uint32_t h) {
  return h;
}
template <>
__device__ __forceinline__ uint32_t h2_to<__nv_bfloat16>(uint32_t h) {
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  return pack2<__nv_bfloat16>(f.x, f.y);
}

struct Item {
  int b, kh, split, mblk;
  int qs, qb, L, M, r0, k0, k1, nchunks, slot_base;
};

// Decodes item id -> its row, head, split and key range.  Returns false for
// items with nothing to do (empty split, block past the row's query rows,
// a row routed elsewhere).
__device__ __forceinline__ bool item_info(const AttnArgs& a, int id, int n_mblk, Item& f) {
  const Problem& p = a.p;
  f.mblk = id % n_mblk;
  int rest = id / n_mblk;
  f.split = rest % a.split_cap;
  rest /= a.split_cap;
  f.kh = rest % p.hkv;
  if (a.tokenwise) {
    // one-token rows: unit = decode slot; token i of row b is a row of its
    // own with q = 1 and L = L_b - q_b + 1 + i
    const int slot = rest / p.hkv;
    if (a.n_slots && slot >= (int)*a.n_slots) return false;
    if (slot >= a.max_slots) return false;
    const int t = a.slot_tok ? __ldg(a.slot_tok + slot) : slot;
    if (t < 0 || t >= p.total_q || p.num_rows <= 0) return false;
    int lo = 0, hi = p.num_rows - 1;  // row of token t: largest b with cu_q[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int qs = __ldg(p.cu_q + lo), qb = __ldg(p.cu_q + lo + 1) - qs;
    if (t < qs || t >= qs + qb) return false;
    f.b = lo;
    f.qs = t;
    f.qb = 1;
    f.slot_base = slot;
    f.L = __ldg(p.seq_lens + lo) - qb + 1 + (t - qs);
  } else {
    f.b = rest / p.hkv;
    if (a.row_order) f.b = __ldg(a.row_order + f.b);
    f.qs = __ldg(p.cu_q + f.b);
    f.qb = __ldg(p.cu_q + f.b + 1) - f.qs;
    if (f.qb <= 0 || f.qs < 0 || f.qs + f.qb > p.total_q) return false;
    f.slot_base = f.qs;
    if (a.dec_base) {
      f.slot_base = __ldg(a.dec_base + f.b);
      if (f.slot_base < 0) return false;
    }
    if ((int64_t)f.slot_base + f.qb > a.max_slots) return false;
    if (f.qb > a.max_decode_q) {
      // a row too long for the decode path (only the device can see it
      // without host mirrors): skipped and flagged
      atomicOr(p.err, PA_DEVERR_DECODE_Q);
      return false;
    }
    f.L = __ldg(p.seq_lens + f.b);
    if (a.long_tc && dec_is_long(f.L, 1)) return false;  // on the tile kernel
  }
  f.M = f.qb * p.g;
  f.r0 = f.mblk * 16;
  if (f.r0 >= f.M) return false;
  const int tps = dec_split_tiles(f.L, a.by_len);
  f.k0 = f.split * tps * DEC_KT;
  if (f.k0 >= f.L) return false;
  f.k1 = min(f.k0 + tps * DEC_KT, f.L);
  f.nchunks = (f.k1 - f.k0 + 15) / 16;
  return true;
}

// Same-launch merge (FUSED; vllm-rlt PR #128, Test Result: a follow-up
// merges inside the decode launch, bitwise equal to the two-kernel path).
// Once its items are done, every warp arrives at a grid-wide barrier (a
// counter in the workspace, waited on with the same clock bound as every
// other wait); then the warps take the (decode token, query head) pairs in
// turn and merge each with the merge kernel's arithmetic (merge16), lane =
// D / 32 consecutive head-dim columns.  Used for decode calls whose grid is
// smaller than the GPU, where the second launch costs more than the merge.
template <typename T, int D>
__device__ __forceinline__ void merge_pair(const AttnArgs& a, int slot, int h, int lane) {
  constexpr int NC = D / 32;
  const Problem& p = a.p;
  const float2* ml = a.part_ml + ((int64_t)slot * p.hq + h) * a.split_stride;
  const float* acc = a.part_acc + ((int64_t)slot * p.hq + h) * a.split_stride * D + lane * NC;
  float2 mlv[NSPLIT];
  float av[NC][NSPLIT];
#pragma unroll
  for (int k = 0; k < NSPLIT; ++k) {
    // L2 loads: the states were written by other SMs in this launch
    mlv[k] = __ldcg(ml + k);
#pragma unroll
    for (int c = 0; c < NC; c += 2) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(acc + (int64_t)k * D + c));
      av[c][k] = v.x;
      av[c + 1][k] = v.y;
    }
  }
  const int t = a.slot_tok ? __ldg(a.slot_tok + slot) : slot;
  float res[NC];
  merge16<NC>(mlv, av, merge_splits(a, t), p.v_scale, res);
  T* out = static_cast<T*>(a.out) + ((int64_t)t * p.hq + h) * D + lane * NC;
#pragma unroll
  for (int c = 0; c < NC; c += 2)
    *reinterpret_cast<uint32_t*>(out + c) = pack2<T>(res[c], res[c + 1]);
}

template <typename T, bool KV8, int D, bool FUSED>
__global__ void __launch_bounds__(DecCfg<D, KV8>::W * 32, 1)
    decode_tma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, int total_items, int n_mblk,
                      uint32_t* counters, int merge_slots) {
  using C = DecCfg<D, KV8>;
  constexpr int NS = C::NS;
  constexpr int KSTEPS = D / 16;  // 16-wide reduction steps of S over the head dim
  constexpr int MT = D / 16;      // 16-row tiles of O^T over the head dim
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const uint32_t wring = base + warp * NS * C::SLOT;  // this warp's slots
  const uint32_t bar0 = base + C::OFF_BAR + warp * NS * 8;
  int2* meta = reinterpret_cast<int2*>(smem + C::OFF_META) + warp * NS;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncwarp();

  // ---- producer (warp-uniform state; lane 0 issues the copies) -------------
  // The cursor walks the item's 16-key slots, padded to a multiple of G.  The
  // block-table entries come from two 32-entry windows held one per lane
  // (the next window is loaded while the current one is in use), so a slot's
  // page costs one shuffle instead of a dependent global load.
  int cur_id = -1, cur_chunk = 0, cur_n = 0;
  int pcol = 0, poff = 0, wbase = 0, win = -1, win_next = -1;
  Item cur{};
  auto bt_entry = [&](int col) {
    return col < p.max_pages ? __ldg(p.bt + (int64_t)cur.b * p.max_pages + col) : -1;
  };
  auto fetch = [&]() {
    // next non-empty item, or cur_id = -1
    for (;;) {
      int id = 0;
      if (lane == 0) id = (int)atomicAdd(counters, 1u);
      id = __shfl_sync(0xffffffffu, id, 0);
      if (id >= total_items) {
        cur_id = -1;
        return;
      }
      if (item_info(a, id, n_mblk, cur)) {
        cur_id = id;
        cur_chunk = 0;
        cur_n = (cur.nchunks + C::G - 1) / C::G * C::G;
        pcol = cur.k0 / p.page_size;
        poff = cur.k0 % p.page_size;
        wbase = pcol & ~31;
        win = bt_entry(wbase + lane);
        win_next = bt_entry(wbase + 32 + lane);
        return;
      }
    }
  };
  auto issue = [&](int s) {
    // the cursor's next slot into ring slot s (or mark the end)
    const uint32_t bar = bar0 + 8 * s;
    if (cur_id < 0) {
      if (lane == 0) meta[s] = make_int2(-1, 0);
      return;
    }
    if (cur_chunk >= cur.nchunks) {
      if (lane == 0) {
        meta[s] = make_int2(cur_id, cur_chunk | META_PAD);
        mbar_arrive(bar);
      }
    } else {
      if (pcol >= wbase + 32) {  // pages advance at most one column per slot
        wbase += 32;
        win = win_next;
        win_next = bt_entry(wbase + 32 + lane);
      }
      const int page = __shfl_sync(0xffffffffu, win, pcol - wbase);
      if (lane == 0) {
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.err, PA_DEVERR_BAD_PAGE);
          meta[s] = make_int2(cur_id, cur_chunk | META_BAD);
          mbar_arrive(bar);
        } else {
          const int tok0 = page * p.page_size + poff;
          meta[s] = make_int2(cur_id, cur_chunk);
          mbar_arrive_expect_tx(bar, C::SLOT);
          const uint32_t dK = wring + s * C::SLOT, dV = dK + C::HALF;
          // one box per half: all NCH 128-byte chunks of the slot's 16 keys
          tma_load_4d(dK, &tmK, 0, tok0, 0, cur.kh, bar);
          tma_load_4d(dV, &tmV, 0, tok0, 0, cur.kh, bar);
        }
      }
      poff += 16;
      if (poff >= p.page_size) {
        poff -= p.page_size;
        ++pcol;
      }
    }
    if (++cur_chunk >= cur_n) fetch();
  };
  fetch();
  for (int s = 0; s < NS - C::G; ++s) issue(s);
  __syncwarp();

  // ---- consumer -------------------------------------------------------------
  // The warp computes the transposed products, keys on the MMA's M side:
  //   S^T[16 keys x 16 rows]  = K[16 x d] . Q^T[d x 16]
  //   O^T[d x 16 rows]       += V^T[d x 16 keys] . P^T[16 keys x 16 rows]
  // so Q (the B operand of S^T) stays in registers for the whole item, K
  // and V are read once per slot with ldmatrix (V transposed by ldmatrix
  // itself), and P^T is S^T's accumulator moved across lanes by movmatrix.
  // Rows are the item's 16 GQA-packed query rows, two n-tiles of 8; an item
  // with at most 8 rows runs the first n-tile only.  Each iteration takes G
  // consecutive ring slots of one item (items are padded to a multiple of
  // G), which gives the dependent MMA chains G-fold independence and shares
  // the softmax reductions.
  //
  // Lane (gid, tig) holds, per n-tile j, rows 8j+2tig and 8j+2tig+1; of
  // S^T, keys gid and gid+8 of each slot; of O^T, two head-dim columns per
  // 16-column tile:  16-bit caches 16mt+gid and 16mt+8+gid, E5M2 caches
  // 16mt+2gid and 16mt+2gid+1.
  //
  // For E5M2 K, one 32-bit word of a key row holds four codes; widened they
  // are two binary16 pairs, so within each 16-wide reduction step the lane's
  // operand slots (2tig, 2tig+1 | 2tig+8, 2tig+9) hold head-dim columns
  // 4tig .. 4tig+3, and Q's fragments are loaded with the same order.
  constexpr int G = C::G;
  uint32_t phase = 0;                   // bit s: parity of ring slot s
  bool aborted = false;
  int it_id = -1;
  Item f{};
  bool two = false;                  // the item has a second n-tile of rows
  uint32_t qf[KSTEPS][2][2];         // Q^T fragments, per step and n-tile
  float o[2][MT][4];                 // O^T accumulators
  float m_use[2][2], l_run[2][2];    // per row: exponent reference, partial sum
  int last[2][2];                    // per row: last visible key, -1 for padding
  const float sl2 = p.sl2;
  const int key_lane = lane & 15, seg_lane = lane >> 4;
  for (int s = 0;; s = (s + G == NS ? 0 : s + G)) {
    // refill the group consumed by the previous iteration (at the start: the
    // one group the prologue left empty), NS-G slots ahead of this group
    {
      const int r = s == 0 ? NS - G : s - G;
#pragma unroll
      for (int u = 0; u < G; ++u) issue(r + u);
    }
    __syncwarp();
    const int2 mt0 = meta[s];
    if (mt0.x < 0) break;
    bool ok = true;
#pragma unroll
    for (int u = 0; u < G; ++u)
      ok = ok && mbar_wait_warp(bar0 + 8 * (s + u), (phase >> (s + u)) & 1u, lane, p.err);
    if (!ok) {
      aborted = true;
      break;
    }
#pragma unroll
    for (int u = 0; u < G; ++u) phase ^= 1u << (s + u);
    if (mt0.x != it_id) {
      // a new item: its rows' Q fragments, fresh state
      it_id = mt0.x;
      item_info(a, it_id, n_mblk, f);
      two = f.M - f.r0 > 8;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int R = f.r0 + 8 * j + gid;
        const T* qrow = static_cast<const T*>(a.q) +
                        ((int64_t)(f.qs + R / p.g) * p.hq + f.kh * p.g + R % p.g) * D;
        const bool qok = R < f.M;
#pragma unroll
        for (int kd = 0; kd < KSTEPS; ++kd) {
          if constexpr (KV8) {
            const uint2 v = qok ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * kd + 4 * tig))
                                : make_uint2(0u, 0u);
            qf[kd][j][0] = v.x;
            qf[kd][j][1] = v.y;
          } else {
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + 16 * kd + 2 * tig);
            qf[kd][j][0] = qok ? __ldg(q32) : 0u;
            qf[kd][j][1] = qok ? __ldg(q32 + 4) : 0u;
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int Rr = f.r0 + 8 * j + 2 * tig + e;
          last[j][e] = Rr < f.M ? f.L - f.qb + Rr / p.g : -1;
          m_use[j][e] = -INFINITY;
          l_run[j][e] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) o[j][m][0] = o[j][m][1] = o[j][m][2] = o[j][m][3] = 0.f;
      }
    }
    const int chunk0 = mt0.y & 0xFFFF;
    int kb[G], nvalid[G];
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int my = meta[s + u].y;
      kb[u] = f.k0 + 16 * (chunk0 + u);
      nvalid[u] = (my & (META_BAD | META_PAD)) ? 0 : min(16, f.L - kb[u]);
      if (nvalid[u] < 16) {
        // keys past the row's end, padding slots and slots behind a bad
        // table entry: zero their V rows so stale or poisoned bytes never
        // reach P V (their logits are masked, whatever K holds)
        const uint32_t sV = wring + (s + u) * C::SLOT + C::HALF;
        for (int e = lane; e < (16 - nvalid[u]) * C::SEGS; e += 32)
          st_shared_v4(sV + seg_off(nvalid[u] + e / C::SEGS, e % C::SEGS),
                       make_uint4(0u, 0u, 0u, 0u));
        __syncwarp();
      }
    }

    // The slot math, compiled once per count of 8-row n-tiles so that the
    // unrolled MMA sequences carry no branches.
    auto math = [&](auto nt_const) {
      constexpr int NT = decltype(nt_const)::value;
      // accumulator sets per slot for S^T: two shorten the dependent MMA
      // chain where registers allow (one n-tile, or d <= 128)
      constexpr int NACC = G == 1 && (NT == 1 || D <= 128) ? 2 : 1;
      // S^T = K Q^T.  ldmatrix x4 at segments (sb, sb+1): lanes 0-15 address
      // key rows 0-15 of segment sb, lanes 16-31 of segment sb+1.
      float sa[G][NACC][NT][4];
#pragma unroll
      for (int u = 0; u < G; ++u)
#pragma unroll
        for (int c = 0; c < NACC; ++c)
#pragma unroll
          for (int j = 0; j < NT; ++j)
            sa[u][c][j][0] = sa[u][c][j][1] = sa[u][c][j][2] = sa[u][c][j][3] = 0.f;
#pragma unroll
      for (int sb = 0; sb < C::SEGS; sb += 2) {
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const uint32_t sK = wring + (s + u) * C::SLOT;
          uint32_t r0, r1, r2, r3;
          ldsm_x4(sK + seg_off(key_lane, sb + seg_lane), r0, r1, r2, r3);
          if constexpr (KV8) {
            // r0/r1: keys gid/gid+8 of segment sb, r2/r3 of sb+1: two steps
            uint32_t a0[4], a1[4];
            e5m2x4_to<T>(r0, a0[0], a0[2]);
            e5m2x4_to<T>(r1, a0[1], a0[3]);
            e5m2x4_to<T>(r2, a1[0], a1[2]);
            e5m2x4_to<T>(r3, a1[1], a1[3]);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              mma16816<T>(sa[u][0][j], a0, qf[sb][j][0], qf[sb][j][1]);
              mma16816<T>(sa[u][NACC - 1][j], a1, qf[sb + 1][j][0], qf[sb + 1][j][1]);
            }
          } else {
            // one step: head-dim columns 8*sb .. 8*sb+15
            const uint32_t af[4] = {r0, r1, r2, r3};
            const int kd = sb >> 1, c = NACC == 1 ? 0 : (kd & 1);
#pragma unroll
            for (int j = 0; j < NT; ++j) mma16816<T>(sa[u][c][j], af, qf[kd][j][0], qf[kd][j][1]);
          }
        }
      }
      // sc[u][j][e + 2h] = logit of row 8j+2tig+e, key kb[u]+gid+8h (log2
      // units, masked), kept in sa[u][0]
      bool need = false;
      float mx[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float m = -INFINITY;
#pragma unroll
          for (int u = 0; u < G; ++u) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = e + 2 * h;
              float x = sa[u][0][j][c];
              if (NACC == 2) x += sa[u][NACC - 1][j][c];
              x = gid + 8 * h < nvalid[u] && kb[u] + gid + 8 * h <= last[j][e] ? x * sl2
                                                                                : -INFINITY;
              sa[u][0][j][c] = x;
              m = fmaxf(m, x);
            }
          }
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
          mx[j][e] = m;
          need |= m > m_use[j][e] + 8.f;
        }
      }
      // lazy rescale: the exponent reference of a row moves only when the
      // row's maximum passes it by more than 8 (a factor of 256), so
      // p = 2^(x - ref) <= 256 and O^T is rescaled rarely.  The decision
      // depends on the row's own logits only.
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float alpha = 1.f;
            if (mx[j][e] > m_use[j][e] + 8.f) {
              alpha = exp2f(m_use[j][e] - mx[j][e]);
              m_use[j][e] = mx[j][e];
            }
            l_run[j][e] *= alpha;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              o[j][m][e] *= alpha;
              o[j][m][e + 2] *= alpha;
            }
          }
        }
      }
      // P^T fragments: pack S^T's (row pair, key) values, transpose with movmatrix
      uint32_t pb[G][NT][2];
#pragma unroll
      for (int u = 0; u < G; ++u) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float pv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float ref = m_use[j][c & 1] == -INFINITY ? 0.f : m_use[j][c & 1];
            pv[c] = exp2f(sa[u][0][j][c] - ref);
            l_run[j][c & 1] += pv[c];
          }
          pb[u][j][0] = movm_t(pack2<T>(pv[0], pv[1]));  // keys 2tig, 2tig+1 of row gid
          pb[u][j][1] = movm_t(pack2<T>(pv[2], pv[3]));  // keys 8+2tig, 9+2tig
        }
      }

      // O^T += V^T P^T
      if constexpr (KV8) {
        // ldmatrix.trans on the codes as 16-bit pairs: lane (gid, tig) gets
        // keys 2tig, 2tig+1 of head-dim columns 2gid, 2gid+1 of a segment;
        // one byte permute per operand register places each code in the
        // high byte of a binary16 (the exact E5M2 -> binary16 widening).
#pragma unroll
        for (int sb = 0; sb < C::SEGS; sb += 2) {
#pragma unroll
          for (int u = 0; u < G; ++u) {
            const uint32_t sV = wring + (s + u) * C::SLOT + C::HALF;
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(sV + seg_off(key_lane, sb + seg_lane), r0, r1, r2, r3);
            const uint32_t aa[4] = {h2_to<T>(__byte_perm(r0, 0u, 0x2404)),
                                    h2_to<T>(__byte_perm(r0, 0u, 0x3414)),
                                    h2_to<T>(__byte_perm(r1, 0u, 0x2404)),
                                    h2_to<T>(__byte_perm(r1, 0u, 0x3414))};
            const uint32_t ab[4] = {h2_to<T>(__byte_perm(r2, 0u, 0x2404)),
                                    h2_to<T>(__byte_perm(r2, 0u, 0x3414)),
                                    h2_to<T>(__byte_perm(r3, 0u, 0x2404)),
                                    h2_to<T>(__byte_perm(r3, 0u, 0x3414))};
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              mma16816<T>(o[j][sb], aa, pb[u][j][0], pb[u][j][1]);
              mma16816<T>(o[j][sb + 1], ab, pb[u][j][0], pb[u][j][1]);
            }
          }
        }
      } else {
        // x4.trans: keys 0-7 / 8-15 (lane bit 4) of segments 2mt / 2mt+1 (lane bit 3)
        const int vkey = (lane & 7) + ((lane >> 4) << 3), vseg = (lane >> 3) & 1;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
          for (int u = 0; u < G; ++u) {
            const uint32_t sV = wring + (s + u) * C::SLOT + C::HALF;
            uint32_t af[4];
            ldsm_x4_t(sV + seg_off(vkey, 2 * m + vseg), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int j = 0; j < NT; ++j) mma16816<T>(o[j][m], af, pb[u][j][0], pb[u][j][1]);
          }
        }
      }
    };
    if (two)
      math(std::integral_constant<int, 2>{});
    else
      math(std::integral_constant<int, 1>{});

    if (chunk0 + G >= f.nchunks) {
      // item done: this split's partial state of the block's rows
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float lt = l_run[j][e];
          lt += __shfl_xor_sync(0xffffffffu, lt, 4);
          lt += __shfl_xor_sync(0xffffffffu, lt, 8);
          lt += __shfl_xor_sync(0xffffffffu, lt, 16);
          const int R = f.r0 + 8 * j + 2 * tig + e;
          if (R >= f.M) continue;
          const int64_t slot = f.slot_base + R / p.g;
          const int64_t ps = (slot * p.hq + f.kh * p.g + R % p.g) * a.split_stride + f.split;
          float* acc = a.part_acc + ps * D;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if constexpr (KV8) {
              *reinterpret_cast<float2*>(acc + 16 * m + 2 * gid) =
                  make_float2(o[j][m][e], o[j][m][e + 2]);
            } else {
              acc[16 * m + gid] = o[j][m][e];
              acc[16 * m + 8 + gid] = o[j][m][e + 2];
            }
          }
          if (gid == 0) a.part_ml[ps] = make_float2(m_use[j][e], lt);
        }
      }
    }
    // the group is consumed; the next iteration refills it with TMA (async
    // writes after this warp's generic reads and zero-fills)
    fence_proxy_async_smem();
    __syncwarp();
  }

  // a timed-out warp may still have copies landing: let them finish (slots
  // waited on successfully in the failed group still hold their old parity,
  // so their drain returns at once)
  if (aborted && lane == 0) {
    for (int s = 0; s < NS; ++s)
      if (meta[s].x >= 0) mbar_drain(bar0 + 8 * s, (phase >> s) & 1u, p.err);
  }
  __syncwarp();
  const uint32_t n_warps = gridDim.x * C::W;
  if constexpr (FUSED) {
    // grid-wide barrier: every warp's partial states are written.  One
    // arrival per CTA, once all of its warps are done with their items.
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
      int ok = 1;
      // cumulative: releases the writes of the whole CTA (ordered before it
      // by the block barrier) to the CTAs that see the arrival
      __threadfence();
      atomicAdd(counters + 2, 1u);
      const long long t0 = clock64();
      while (*reinterpret_cast<volatile uint32_t*>(counters + 2) < gridDim.x) {
        if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
          atomicOr(p.err, PA_DEVERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
      __threadfence();
      s_ok = ok;
    }
    __syncthreads();
    if (s_ok) {
      const int n_pairs = merge_slots * p.hq;
      for (int u = blockIdx.x * C::W + warp; u < n_pairs; u += (int)n_warps)
        merge_pair<T, D>(a, u / p.hq, u % p.hq, lane);
    }
    __syncwarp();
  }
  // the last warp of the grid resets the counters for the next call
  if (lane == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(counters + 1, 1u);
    if (done == n_warps - 1) {
      counters[0] = 0u;
      counters[1] = 0u;
      counters[2] = 0u;
      __threadfence();
    }
  }
}

template <int D, bool KV8>
int dec_grid(int total_items, int sms) {
  using C = DecCfg<D, KV8>;
  int grid = sms > 0 ? sms : 148;  // persistent: one CTA per SM
  if (total_items < grid * C::W) grid = (total_items + C::W - 1) / C::W;
  return grid < 1 ? 1 : grid;
}

template <typename T, bool KV8, int D>
cudaError_t launch_dec(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       int total_items, int n_mblk, uint32_t* counters, int merge_slots,
                       int sms, cudaStream_t st) {
  using C = DecCfg<D, KV8>;
  auto k = merge_slots > 0 ? decode_tma_kernel<T, KV8, D, true>
                           : decode_tma_kernel<T, KV8, D, false>;
  static DeviceFlags attr, attr_f;
  cudaError_t e = (merge_slots > 0 ? attr_f : attr).once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  const int grid = dec_grid<D, KV8>(total_items, sms);
  k<<<grid, C::W * 32, C::SMEM, st>>>(a, tk, tv, total_items, n_mblk, counters, merge_slots);
  return cudaGetLastError();
}

template <typename T, bool KV8>
cudaError_t launch_dec_d(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                         int items, int n_mblk, uint32_t* cnt, int merge_slots, int sms,
                         cudaStream_t st) {
  switch (a.p.d) {
    case 64:
      if constexpr (!KV8)
        return launch_dec<T, KV8, 64>(a, tk, tv, items, n_mblk, cnt, merge_slots, sms, st);
      break;
    case 128: return launch_dec<T, KV8, 128>(a, tk, tv, items, n_mblk, cnt, merge_slots, sms, st);
    case 256: return launch_dec<T, KV8, 256>(a, tk, tv, items, n_mblk, cnt, merge_slots, sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_tma_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16) || cache_tokens >= (int64_t(1) << 31)) return false;
  if (kv_dtype == q_dtype) return d == 64 || d == 128 || d == 256;
  return kv_dtype == PA_E5M2 && (d == 128 || d == 256);
}

int decode_tma_grid(int d, bool kv8, int64_t items, int sms) {
  const int n = items >= (int64_t(1) << 31) ? INT32_MAX : (int)items;
  if (kv8) return d == 128 ? dec_grid<128, true>(n, sms) : dec_grid<256, true>(n, sms);
  return d == 64 ? dec_grid<64, false>(n, sms)
                 : d == 128 ? dec_grid<128, false>(n, sms) : dec_grid<256, false>(n, sms);
}

cudaError_t launch_decode_tma(const AttnArgs& a, int q_dtype, int kv_dtype, int n_mblk,
                              int n_units, int merge_slots, int sms, cudaStream_t st) {
  if (a.p.num_rows == 0 || n_mblk == 0 || n_units <= 0) return cudaSuccess;
  const int64_t items = (int64_t)n_units * a.p.hkv * a.split_cap * n_mblk;
  if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv;
  if (!encode_slot_map(&tk, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_slot_map(&tv, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens))
    return cudaErrorInvalidValue;
  uint32_t* counters = reinterpret_cast<WsHeader*>(a.p.err)->pad;
  const bool kv8 = kv_dtype == PA_E5M2;
  const int it = (int)items, ms = merge_slots;
  if (q_dtype == PA_BF16)
    return kv8 ? launch_dec_d<__nv_bfloat16, true>(a, tk, tv, it, n_mblk, counters, ms, sms, st)
               : launch_dec_d<__nv_bfloat16, false>(a, tk, tv, it, n_mblk, counters, ms, sms, st);
  return kv8 ? launch_dec_d<__half, true>(a, tk, tv, it, n_mblk, counters, ms, sms, st)
             : launch_dec_d<__half, false>(a, tk, tv, it, n_mblk, counters, ms, sms, st);
}

}  // namespace pa
