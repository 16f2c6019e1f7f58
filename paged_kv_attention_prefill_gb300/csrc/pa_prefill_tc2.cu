// Varlen causal paged prefill on the tcgen05 tensor cores, two query tiles
// per CTA (head dims 64 and 128).
//
// The same attention as every other path of the library (packed varlen
// batch, one block table per row, bottom-right causal alignment, GQA, online
// softmax over key tiles: vllm-rlt PR #128, "Purpose", prefill bullets).
// The layout keeps the tensor core busy while the softmax of a tile runs:
//
//  * A CTA owns 256 GQA-packed query rows of one (row, KV head) as two
//    128-row query tiles A and B (the heads that share the KV head stacked
//    along M: 1Cat-vLLM PR #1279, commit 1).  Every K/V tile brought in by
//    TMA serves both query tiles.
//  * Warp 0 streams K tiles and warp 2 V tiles, one 16-token page slot per
//    TMA box (1Cat-vLLM PR #616, original description: any page size that is
//    a multiple of 16), into two shared-memory rings.  The slot that holds a
//    row's last key is copied by hand with the keys past the end zero-filled.
//    With pages of at least 128 tokens (the kernel's WIDE instance), a tile
//    whose slots are one run of one page takes one box per 128-byte chunk.
//  * Warp 1, one thread, issues tcgen05.mma for both query tiles in turn:
//    S_t = Q_t K^T into tile t's S columns of TMEM, O_t += P_t V with P_t
//    read from TMEM.  While one softmax warpgroup works on its S, the tensor
//    core computes the other tile's products.
//  * Warpgroup 1 runs the softmax of tile A, warpgroup 2 that of tile B; each
//    thread owns one query row (one TMEM lane) over all 128 key columns, so
//    the row maximum needs no exchange between threads.  P (16-bit) is
//    written over S in TMEM.  O is rescaled only when a row's maximum grows
//    by more than 2^8; the final O / l is the same.
//  * setmaxnreg moves registers from the producer / MMA warpgroup to the two
//    softmax warpgroups.
//
// Every wait is bounded (about two seconds); on a timeout the CTA raises the
// workspace flag, drains the copies and MMAs it started, frees TMEM and
// exits.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_sm100.cuh"

namespace pa {
bool encode_kv_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                   int64_t tokens);
bool encode_kv_map_rows(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                        int64_t tokens, int rows);

namespace {

using namespace sm100;

// Registers per thread at launch (384 threads, one CTA per SM) and after the
// split, which must fit in what the CTA was launched with:
// 128 * reg_low + 256 * reg_high <= 384 * REG_LAUNCH.  With an fp8 cache the
// producer / widening warpgroup needs more.
constexpr int REG_LAUNCH = 168;
constexpr int reg_low(bool kv8) { return kv8 ? 88 : 72; }
constexpr int reg_high(bool kv8) { return kv8 ? 200 : 216; }
static_assert(128 * reg_low(false) + 256 * reg_high(false) <= 384 * REG_LAUNCH &&
                  128 * reg_low(true) + 256 * reg_high(true) <= 384 * REG_LAUNCH,
              "register split");

template <int D, bool KV8>
struct Tc2Cfg {
  static constexpr int BM = 128;                    // rows per query tile = TMEM lanes
  static constexpr int BN = 128;                    // keys per tile
  // 16-bit K / V stages the MMAs read.  With an fp8 cache the tiles arrive as
  // codes in their own rings (S8 stages each) and are widened into these, so
  // fewer 16-bit stages are needed (K is read by both S products back to
  // back; V's stage must cover the widening of the next tile).
  static constexpr int KS = KV8 ? 1 : (D == 64 ? 4 : 2);
  static constexpr int VS = KV8 ? 2 : (D == 64 ? 4 : 3);
  static constexpr int S8 = KV8 ? 2 : 1;             // (one unused stage index without fp8)
  static constexpr int NCH = D / 64;                // 128-byte column chunks of d
  static constexpr int SLOTS = BN / 16;             // 16-token page slots per key tile
  static constexpr uint32_t Q_BYTES = BM * D * 2;   // one query tile
  static constexpr uint32_t KV_BYTES = BN * D * 2;  // K (or V) of one key tile, 16-bit
  static constexpr uint32_t KV8_BYTES = BN * D;     // K (or V) of one key tile, fp8 codes
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KS * KV_BYTES;
  static constexpr uint32_t OFF_K8 = OFF_V + VS * KV_BYTES;
  static constexpr uint32_t OFF_V8 = OFF_K8 + (KV8 ? S8 * KV8_BYTES : 0);
  static constexpr uint32_t OFF_BAR = OFF_V8 + (KV8 ? S8 * KV8_BYTES : 0);
  static constexpr uint32_t BAR_AREA = 320;        // mbarriers, then TMEM address and flags
  static constexpr uint32_t SMEM = OFF_BAR + BAR_AREA + 16 + 1024;  // alignment slack
  // TMEM: tile t owns columns [t * TILE_COLS, +BN) for S (P over it) and
  // [t * TILE_COLS + BN, +D) for O.
  static constexpr uint32_t TILE_COLS = BN + D;
  static constexpr uint32_t TMEM_COLS = 512;
  // barrier indices
  static constexpr int B_KF = 0, B_KE = KS, B_VF = 2 * KS, B_VE = 2 * KS + VS,
                       B_SF = 2 * KS + 2 * VS,  // [2] S_t written
      B_PF = B_SF + 2,                          // [2] P_t of keys 0-63 written (4 warps)
      B_PF2 = B_PF + 2,                         // [2] P_t of keys 64-127 written (4 warps)
      B_OF = B_PF2 + 2,                         // [2] O_t += P_t V done
      B_Q = B_OF + 2,                           // [2] Q_t staged (128 arrivals)
      B_DRAIN = B_Q + 2,                        // every MMA done
      B_K8F = B_DRAIN + 1, B_K8E = B_K8F + S8,  // fp8 code rings: full / empty
      B_V8F = B_K8E + S8, B_V8E = B_V8F + S8, NBAR = B_V8E + S8;
  static_assert(2 * TILE_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NBAR * 8 <= BAR_AREA, "barrier area");
  static_assert(!KV8 || D == 128, "fp8 caches: one 128-byte TMA box per key row");
};

template <typename T, int D, bool KV8, bool WIDE>
__global__ void __launch_bounds__(384, 1)
    prefill_tc2_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmKw,
                       const __grid_constant__ CUtensorMap tmVw) {
  using C = Tc2Cfg<D, KV8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t sK8 = base + C::OFF_K8, sV8 = base + C::OFF_V8;
  const uint32_t bar0 = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::BAR_AREA);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::BAR_AREA + 4);
  // the item's part index when its key range is cut, else -1 (read back by
  // the epilogue, so the softmax warps need not keep it in registers)
  volatile int* part_slot = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::BAR_AREA + 8);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item (uniform over the CTA) -----------------------------------
  // 1-D grid, KV head fastest: the work list is longest-first, so the CTAs
  // dispatched last are the shortest of all heads
  const int item = blockIdx.x / p.hkv, kh = blockIdx.x % p.hkv;
  if (item >= (int)*a.n_tiles) return;
  const int2 wi = a.tiles[item];
  const int b = wi.x, mb = wi.y & 0xFFFFFF, part = wi.y >> 24;
  const int qs = __ldg(p.cu_q + b);
  const int qb = __ldg(p.cu_q + b + 1) - qs;
  const int L = __ldg(p.seq_lens + b);
  if (qb <= 0) return;
  if (qs < 0 || qs + qb > p.total_q) {
    if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return;
  }
  const int g = p.g, M = qb * g, R0 = mb * 2 * C::BM;
  if (R0 >= M) return;
  // keys any row of a query tile (of the item) sees
  auto k_end_of = [&](int r0, int rows) {
    const int r_last = min(r0 + rows, M) - 1;
    return min(L, L - qb + r_last / g + 1);
  };
  // The item's key range [k0, k1): the whole range, or one part of it
  int per_u;
  const int k_item = k_end_of(R0, 2 * C::BM);
  const bool cut = pf_part_count(k_item, a.pf_parts, a.pf_min_units, &per_u) > 1;
  const int k0 = cut ? part * per_u * PF_UNIT : 0;
  const int k1 = cut ? min(k_item, (part + 1) * per_u * PF_UNIT) : k_item;
  // key tiles of each query tile in the range (0 for an empty tile B)
  auto tiles_of = [&](int r0) {
    if (r0 >= M) return 0;
    const int hi = min(k_end_of(r0, C::BM), k1);
    return hi > k0 ? (hi - k0 + C::BN - 1) / C::BN : 0;
  };
  const int nA = tiles_of(R0), nB = tiles_of(R0 + C::BM);
  const int n_kv = max(nA, nB);

  // ---- barriers and TMEM ----------------------------------------------------
  if (threadIdx.x == 0) {
    // fp8 caches: the 16-bit stages are filled by the two widening warps
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_KF + s), KV8 ? 2 : 1);
      mbar_init(bar(C::B_KE + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_VF + s), KV8 ? 2 : 1);
      mbar_init(bar(C::B_VE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SF + t), 1);
      mbar_init(bar(C::B_PF + t), 4);
      mbar_init(bar(C::B_PF2 + t), 4);
      mbar_init(bar(C::B_OF + t), 1);
      mbar_init(bar(C::B_Q + t), 128);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    for (int s = 0; s < C::S8; ++s) {
      mbar_init(bar(C::B_K8F + s), 1);
      mbar_init(bar(C::B_K8E + s), 2);
      mbar_init(bar(C::B_V8F + s), 1);
      mbar_init(bar(C::B_V8E + s), 2);
    }
    *abort_flag = 0;
    *part_slot = cut ? part : -1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    setmaxnreg_dec<reg_low(KV8)>();
    if (KV8 && warp == 0) {
      // ===== fp8 cache: warp 0 streams the K and V codes of each key tile ======
      // into the code rings, one TMA box (16 keys x 128 codes) per page slot
      // (with pages of 128 tokens or more, one per tile in one page); the
      // slot holding the row's last key is copied by hand, zero-filled.
      const uint8_t* kc8 = static_cast<const uint8_t*>(a.kc);
      const uint8_t* vc8 = static_cast<const uint8_t*>(a.vc);
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (WIDE) {
          tma_prefetch_desc(&tmKw);
          tma_prefetch_desc(&tmVw);
        }
      }
      const int P = p.page_size;
      const int64_t bt_row = (int64_t)b * p.max_pages;
      int j = 0;
      int started[2] = {0, 0};  // K / V code units whose copies were started
      bool ok = true;
      for (; j < n_kv; ++j) {
        const int st = j % C::S8;
        const int kbase = k0 + j * C::BN;
        int kind = 0, tok0 = 0;
        if (lane < C::SLOTS) {
          const int s0 = kbase + 16 * lane;
          if (s0 >= L) {
            kind = 3;
          } else {
            const int col = s0 / P;
            const int page = col < p.max_pages ? __ldg(p.bt + bt_row + col) : -1;
            if (page < 0 || page >= p.num_pages) {
              atomicOr(p.err, PA_DEVERR_BAD_PAGE);
              kind = 3;
            } else {
              tok0 = page * P + (s0 % P);
              kind = (s0 + 16 <= L) ? 1 : 2;
            }
          }
        }
        const uint32_t manual_all = __ballot_sync(0xffffffffu, kind >= 2);
        const int n_tma = __popc(__ballot_sync(0xffffffffu, kind == 1));
        // every slot whole and in one run of one page: one box per tile
        const int tok_first = __shfl_sync(0xffffffffu, tok0, 0);
        const bool whole = WIDE && __all_sync(0xffffffffu, lane >= C::SLOTS ||
                                                                     (kind == 1 && tok0 == tok_first + 16 * lane));
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          if (j >= C::S8)
            ok = mbar_wait(bar((kv ? C::B_V8E : C::B_K8E) + st), ((j / C::S8) - 1) & 1, abort_flag,
                           p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const uint32_t dst = (kv ? sV8 : sK8) + st * C::KV8_BYTES;
          const uint8_t* cache = kv ? vc8 : kc8;
          if (whole) {
            const uint32_t fb = bar((kv ? C::B_V8F : C::B_K8F) + st);
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, (uint32_t)C::BN * 128u);
              tma_load_3d(dst, kv ? (const void*)&tmVw : (const void*)&tmKw, 0, kh, tok_first, fb);
            }
            __syncwarp();
            ++started[kv];
            continue;
          }
          uint32_t manual = manual_all;
          while (manual) {
            const int s = __ffs(manual) - 1;
            manual &= manual - 1;
            const int ks = __shfl_sync(0xffffffffu, kind, s);
            const int t0 = __shfl_sync(0xffffffffu, tok0, s);
            const int nvalid = ks == 2 ? L - (kbase + 16 * s) : 0;
            for (int it = lane; it < 16 * 8; it += 32) {
              const int unit = it & 7, rr = it >> 3;
              uint4 v = make_uint4(0u, 0u, 0u, 0u);
              if (rr < nvalid)
                v = __ldg(reinterpret_cast<const uint4*>(
                    cache + ((int64_t)(t0 + rr) * p.hkv + kh) * D + unit * 16));
              const int row = 16 * s + rr;
              st_shared_v4(dst + row * 128 + ((unit ^ (row & 7)) << 4), v);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          const uint32_t fb = bar((kv ? C::B_V8F : C::B_K8F) + st);
          if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_tma * 16u * 128u);
          __syncwarp();
          if (kind == 1) tma_load_3d(dst + lane * 16 * 128, kv ? (const void*)&tmV : (const void*)&tmK, 0, kh, tok0, fb);
          ++started[kv];
        }
        if (!ok) break;
      }
      if (!ok) {
        // copies this warp started may still be landing: wait for them (the
        // last S8 units of each ring; earlier ones were consumed already)
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
          for (int jj = max(0, started[kv] - C::S8); jj < started[kv]; ++jj)
            mbar_drain(bar((kv ? C::B_V8F : C::B_K8F) + jj % C::S8), (jj / C::S8) & 1, p.err);
      }
    } else if (KV8 && (warp == 2 || warp == 3)) {
      // ===== fp8 cache: warps 2 and 3 widen every K and V tile =================
      // (keys [64 (warp - 2), +64) each) into the 16-bit swizzled tiles the
      // MMAs read.  An E5M2 code in the high byte of a binary16 is the same
      // value (exact); for bf16 Q it is widened through fp32, also exactly.
      // Lane = 16 codes of one key per step.
      const int key0 = 64 * (warp - 2);
      const int u = lane & 7, c = u >> 2, va = 2 * (u & 3);
      auto widen = [&](uint32_t src, uint32_t dst) {
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
          const int key = key0 + 4 * it + (lane >> 3);
          const uint4 w = ld_shared_v4(src + key * 128 + ((u ^ (key & 7)) << 4));
          uint4 lo, hi;
          e5m2x4_to<T>(w.x, lo.x, lo.y);
          e5m2x4_to<T>(w.y, lo.z, lo.w);
          e5m2x4_to<T>(w.z, hi.x, hi.y);
          e5m2x4_to<T>(w.w, hi.z, hi.w);
          const uint32_t row = dst + c * (C::BN * 128) + key * 128;
          st_shared_v4(row + ((va ^ (key & 7)) << 4), lo);
          st_shared_v4(row + (((va + 1) ^ (key & 7)) << 4), hi);
        }
        // the MMAs read the tile through the async proxy; TMA overwrites the
        // codes next
        fence_proxy_async_smem();
        __syncwarp();
      };
      bool ok = true;
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st8 = j % C::S8;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int NS = kv ? C::VS : C::KS, st = j % NS;
          ok = ok && mbar_wait(bar((kv ? C::B_V8F : C::B_K8F) + st8), (j / C::S8) & 1, abort_flag,
                               p.err);
          if (ok && j >= NS)
            ok = mbar_wait(bar((kv ? C::B_VE : C::B_KE) + st), ((j / NS) - 1) & 1, abort_flag,
                           p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          widen((kv ? sV8 : sK8) + st8 * C::KV8_BYTES, (kv ? sV : sK) + st * C::KV_BYTES);
          if (lane == 0) {
            mbar_arrive(bar((kv ? C::B_VF : C::B_KF) + st));
            mbar_arrive(bar((kv ? C::B_V8E : C::B_K8E) + st8));
          }
        }
      }
    } else if (!KV8 && (warp == 0 || warp == 2)) {
      // ============ producers: warp 0 streams K tiles, warp 2 V tiles ========
      const bool isK = warp == 0;
      const int NS = isK ? C::KS : C::VS;
      const int B_FULL = isK ? C::B_KF : C::B_VF, B_EMPTY = isK ? C::B_KE : C::B_VE;
      const uint32_t ring = isK ? sK : sV;
      const void* tmap = isK ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmV);
      // the same view with one box per key tile, for tiles whose keys lie in
      // one page
      const void* tmapw = isK ? static_cast<const void*>(&tmKw) : static_cast<const void*>(&tmVw);
      const T* cache = static_cast<const T*>(isK ? a.kc : a.vc);
      if (lane == 0) {
        tma_prefetch_desc(tmap);
        if (WIDE) tma_prefetch_desc(tmapw);
      }
      const int P = p.page_size;
      const int64_t bt_row = (int64_t)b * p.max_pages;
      int j = 0;
      bool ok = true;
      for (; j < n_kv; ++j) {
        const int st = j % NS;
        if (j >= NS) ok = mbar_wait(bar(B_EMPTY + st), ((j / NS) - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const int kbase = k0 + j * C::BN;
        const uint32_t dst = ring + st * C::KV_BYTES;
        // slot `lane`: 1 = whole slot by TMA, 2 = partial (copied by hand), 3 = zero-fill
        int kind = 0, tok0 = 0;
        if (lane < C::SLOTS) {
          const int s0 = kbase + 16 * lane;
          if (s0 >= L) {
            kind = 3;
          } else {
            const int col = s0 / P;
            const int page = col < p.max_pages ? __ldg(p.bt + bt_row + col) : -1;
            if (page < 0 || page >= p.num_pages) {
              atomicOr(p.err, PA_DEVERR_BAD_PAGE);
              kind = 3;
            } else {
              tok0 = page * P + (s0 % P);
              kind = (s0 + 16 <= L) ? 1 : 2;
            }
          }
        }
        const int tok_first = __shfl_sync(0xffffffffu, tok0, 0);
        if (WIDE && __all_sync(0xffffffffu, lane >= C::SLOTS ||
                                                      (kind == 1 && tok0 == tok_first + 16 * lane))) {
          // every slot whole and in one run of one page: one box per chunk
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_FULL + st), (uint32_t)C::BN * D * 2u);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(dst + c * (C::BN * 128), tmapw, c * 64, kh, tok_first, bar(B_FULL + st));
          }
          __syncwarp();
          continue;
        }
        uint32_t manual = __ballot_sync(0xffffffffu, kind >= 2);
        while (manual) {
          const int s = __ffs(manual) - 1;
          manual &= manual - 1;
          const int ks = __shfl_sync(0xffffffffu, kind, s);
          const int t0 = __shfl_sync(0xffffffffu, tok0, s);
          const int nvalid = ks == 2 ? L - (kbase + 16 * s) : 0;
          for (int it = lane; it < 16 * C::NCH * 8; it += 32) {
            const int piece = it & 7, rest = it >> 3;
            const int c = rest % C::NCH, rr = rest / C::NCH;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < nvalid) {
              const T* src = cache + ((int64_t)(t0 + rr) * p.hkv + kh) * D + c * 64 + piece * 8;
              v = __ldg(reinterpret_cast<const uint4*>(src));
            }
            const int row = 16 * s + rr;
            st_shared_v4(dst + c * (C::BN * 128) + row * 128 + ((piece ^ (row & 7)) << 4), v);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int n_tma = __popc(__ballot_sync(0xffffffffu, kind == 1));
        if (lane == 0) mbar_arrive_expect_tx(bar(B_FULL + st), (uint32_t)n_tma * 16u * D * 2u);
        __syncwarp();
        if (kind == 1) {
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(dst + c * (C::BN * 128) + lane * 16 * 128, tmap, c * 64, kh, tok0,
                        bar(B_FULL + st));
        }
      }
      if (!ok) {
        // copies this warp started may still be landing: wait for them
        for (int jj = max(0, j - NS); jj < j; ++jj)
          mbar_drain(bar(B_FULL + jj % NS), (jj / NS) & 1, p.err);
      }
    } else if (warp == 1) {
      // ===================== MMA issuer (one thread) ===========================
      // In-order, with blocking waits: per key tile j and query tile t,
      //   O_t += P_t(j) V   once P_t(j) is written, then
      //   S_t(j+1)          once that product is done (S_t(j+1) overwrites
      //                     the columns P_t(j) is read from),
      // tile A first.  The commit of S_t(j+1) covers the P V product before
      // it, so when the softmax sees S_t(j+1), O_t is stable.  A K (V) stage
      // is released once both tiles have issued their products with it.
      if (lane == 0) {
        constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
        constexpr uint32_t idS = idesc_f16(fmt, 128, C::BN, false);
        constexpr uint32_t idO = idesc_f16(fmt, 128, D, true);
        const int ntl[2] = {nA, nB};
        auto issue_S = [&](int t, int j) {
          const int st = j % C::KS;
          if (!mbar_wait(bar(C::B_KF + st), (j / C::KS) & 1, abort_flag, p.err)) return false;
          tc_fence_after();
          // descriptors of the first step; later steps add their byte offset
          // (>> 4) to the start-address field, which never carries out of it.
          // The issue cost is on the critical path: one MMA is 64 cycles of
          // tensor work.
          const uint64_t a0 = sdesc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
          const uint64_t b0 = sdesc_sw128(sK + st * C::KV_BYTES, 16, 1024);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t ad = a0 + (uint64_t)(((k >> 2) * (C::BM * 128) + (k & 3) * 32) >> 4);
            const uint64_t bd = b0 + (uint64_t)(((k >> 2) * (C::BN * 128) + (k & 3) * 32) >> 4);
            tc_mma_f16(tmem + t * C::TILE_COLS, ad, bd, idS, k > 0 ? 1u : 0u);
          }
          tc_commit(bar(C::B_SF + t));
          return true;
        };
        auto issue_PV = [&](int t, int j) {
          // in two halves of 64 keys: the first half's products start while
          // the softmax still computes the second half's P
          const int sv = j % C::VS;
          if (!mbar_wait(bar(C::B_VF + sv), (j / C::VS) & 1, abort_flag, p.err)) return false;
          const uint32_t tb = tmem + t * C::TILE_COLS;
          const uint64_t b0 = sdesc_sw128(sV + sv * C::KV_BYTES, C::BN * 128, 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait(bar((h ? C::B_PF2 : C::B_PF) + t), j & 1, abort_flag, p.err))
              return false;
            tc_fence_after();
#pragma unroll
            for (int k = h * C::BN / 32; k < (h + 1) * C::BN / 32; ++k) {
              // A = P from TMEM: 16 keys = 8 columns of 16-bit pairs
              const uint64_t bd = b0 + (uint64_t)((k * 16 * 128) >> 4);
              tc_mma_f16_ts(tb + C::BN, tb + 8 * k, bd, idO, (j > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit(bar(C::B_OF + t));
          return true;
        };
        bool ok = true;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (ok && ntl[t] > 0) ok = mbar_wait(bar(C::B_Q + t), 0, abort_flag, p.err);
        if (ok) tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (ok && ntl[t] > 0) ok = issue_S(t, 0);
        if (ok && n_kv > 0) tc_commit(bar(C::B_KE + 0));
        for (int j = 0; ok && j < n_kv; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (ok && j < ntl[t]) {
              ok = issue_PV(t, j);
              if (ok && j + 1 < ntl[t]) {
                ok = mbar_wait(bar(C::B_OF + t), j & 1, abort_flag, p.err);
                if (ok) {
                  tc_fence_after();
                  ok = issue_S(t, j + 1);
                }
              }
            }
          }
          if (!ok) break;
          tc_commit(bar(C::B_VE + j % C::VS));
          if (j + 1 < n_kv) tc_commit(bar(C::B_KE + (j + 1) % C::KS));
        }
        // nothing this thread issued may still run once TMEM is freed
        tc_commit(bar(C::B_DRAIN));
        mbar_drain(bar(C::B_DRAIN), 0, p.err);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<reg_high(KV8)>();
    // ============ softmax and epilogue of query tile t ========================
    // Thread = one query row = one TMEM lane of the tile.  The loop never
    // leaves early: after a timed-out wait it runs on (flag raised, waits
    // return at once), so the CTA always reaches its final barrier.
    const int t = (warp >> 2) - 1;
    const int q4 = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;     // row of the tile == TMEM lane
    const int R = R0 + t * C::BM + r;
    const bool valid = R < M;
    const int i = valid ? R / g : 0, hg = valid ? R % g : 0;
    // last visible key of this row, counted from the start of the key range
    const int last = valid ? L - qb + i - k0 : NO_MASK;
    const int64_t qoff = ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
    const int n = t ? nB : nA;
    const uint32_t q_t = sQ + t * C::Q_BYTES;
    if (n > 0) {
      const T* qrow = static_cast<const T*>(a.q) + qoff;
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const uint4 v = valid ? __ldg(reinterpret_cast<const uint4*>(qrow + c * 64 + pc * 8))
                                : make_uint4(0u, 0u, 0u, 0u);
          st_shared_v4(q_t + c * (C::BM * 128) + r * 128 + ((pc ^ (r & 7)) << 4), v);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_Q + t));
    }
    const uint32_t trow = tmem + t * C::TILE_COLS + ((uint32_t)(q4 * 32) << 16);
    const float sl2 = p.sl2;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j) {
      mbar_wait(bar(C::B_SF + t), j & 1, abort_flag, p.err);
      tc_fence_after();
      // S_t(j) was issued after O_t += P_t(j-1) V completed, and its commit
      // covers every earlier MMA: O_t is stable here.
      // the row's logits as pairs (keys 2k, 2k + 1): the exponent argument
      // and the row sum run on the paired fp32 instructions, each lane of
      // which rounds as its scalar form does
      float2 x[C::BN / 2];
      float mt;  // max raw logit of the row in this tile (masked keys -> -inf)
      {
        uint32_t u[C::BN];
        mt = tmem_ld_red_max_x128(trow, u);  // the load also returns the row's max
#pragma unroll
        for (int k = 0; k < C::BN / 2; ++k)
          x[k] = make_float2(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1]));
      }
      const int kb = j * C::BN;
      if (kb + C::BN - 1 > last) {
        // a tile on the row's diagonal: mask, and take the max of what is left
#pragma unroll
        for (int k = 0; k < C::BN / 2; ++k) {
          if (kb + 2 * k > last) x[k].x = -INFINITY;
          if (kb + 2 * k + 1 > last) x[k].y = -INFINITY;
        }
        float pm[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          pm[2 * u] = x[u].x;
          pm[2 * u + 1] = x[u].y;
        }
#pragma unroll
        for (int k = 4; k < C::BN / 2; ++k) {
          pm[2 * (k & 3)] = fmaxf(pm[2 * (k & 3)], x[k].x);
          pm[2 * (k & 3) + 1] = fmaxf(pm[2 * (k & 3) + 1], x[k].y);
        }
        mt = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      }
      const float m_new = fmaxf(m_used, mt * sl2);  // sl2 > 0: max commutes with the scale
      float factor = 1.f;
      bool need = false;
      if (j == 0) {
        m_used = m_new;
      } else if (m_new > m_used + 8.f) {
        need = true;
        factor = ex2(m_used - m_new);
        m_used = m_new;
      }
      const float nmu = m_used == -INFINITY ? 0.f : -m_used;
      // O is rescaled before any of this tile's P is published (the P V
      // product of the previous tile is done: S_t(j) was issued after it)
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::BN + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st_x32(trow + C::BN + c * 32, o);
        }
      }
      // P (16-bit pairs) over the first BN / 2 columns of S, in two halves of
      // 64 keys, each published as soon as it is in TMEM
      // partial row sums, fixed order: key k adds into sum k mod 8
      float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      const float2 sl2v = make_float2(sl2, sl2), nmv = make_float2(nmu, nmu);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int k = 32 * h; k < 32 * h + 32; ++k) {
          float2 y = __ffma2_rn(x[k], sl2v, nmv);
          y.x = ex2(y.x);
          y.y = ex2(y.y);
          x[k] = y;
          ps[k & 3] = __fadd2_rn(ps[k & 3], y);
        }
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack2<T>(x[32 * h + k].x, x[32 * h + k].y);
        tmem_st_x32_nowait(trow + 32 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        // every lane's stores are done: one arrival per warp
        __syncwarp();
        if (lane == 0) mbar_arrive(bar((h ? C::B_PF2 : C::B_PF) + t));
      }
      const float rs = ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) +
                       ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
      l = l * factor + rs;
    }
    // ---- epilogue: out = O / l * v_scale, or this part's (O, m, l) ----
    T* orow = static_cast<T*>(a.out) + qoff;
    const int part_e = *part_slot;
    if (part_e >= 0) {
      // unnormalised O, the maximum it is relative to and the row sum, for
      // the merge (a row that saw no key of the part: l = 0, skipped there)
      const int64_t slot = ((int64_t)(qs + i) * p.hq + kh * g + hg) * a.pf_parts + part_e;
      if (n > 0) {
        mbar_wait(bar(C::B_OF + t), (n - 1) & 1, abort_flag, p.err);
        tc_fence_after();
      }
      if (valid) a.pf_ml[slot] = make_float2(n > 0 ? m_used : -INFINITY, n > 0 ? l : 0.f);
      float* prow = a.pf_acc + slot * D;
      if (n > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::BN + c * 32, o);
          if (valid) {
#pragma unroll
            for (int w = 0; w < 8; ++w)
              *reinterpret_cast<uint4*>(prow + c * 32 + 4 * w) =
                  make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
          }
        }
      }
    } else if (n > 0) {
      mbar_wait(bar(C::B_OF + t), (n - 1) & 1, abort_flag, p.err);
      tc_fence_after();
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(trow + C::BN + c * 32, o);
        if (valid) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 v;
            v.x = pack2<T>(__uint_as_float(o[8 * w + 0]) * inv, __uint_as_float(o[8 * w + 1]) * inv);
            v.y = pack2<T>(__uint_as_float(o[8 * w + 2]) * inv, __uint_as_float(o[8 * w + 3]) * inv);
            v.z = pack2<T>(__uint_as_float(o[8 * w + 4]) * inv, __uint_as_float(o[8 * w + 5]) * inv);
            v.w = pack2<T>(__uint_as_float(o[8 * w + 6]) * inv, __uint_as_float(o[8 * w + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * w) = v;
          }
        }
      }
    } else if (valid) {
      // no key visible to any row of the tile
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        *reinterpret_cast<uint4*>(orow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <typename T, int D, bool KV8>
cudaError_t launch_tc2(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tkw, const CUtensorMap& tvw, int grid_x, cudaStream_t st) {
  using C = Tc2Cfg<D, KV8>;
  // pages that can hold a whole key tile: the kernel that may copy a tile in
  // one box per chunk
  const bool wide = a.p.page_size >= C::BN;
  auto k = wide ? prefill_tc2_kernel<T, D, KV8, true> : prefill_tc2_kernel<T, D, KV8, false>;
  static DeviceFlags attr, attr_w;
  cudaError_t e = (wide ? attr_w : attr).once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  k<<<dim3((unsigned)grid_x * a.p.hkv), 384, C::SMEM, st>>>(a, tk, tv, tkw, tvw);
  return cudaGetLastError();
}

template <typename T, int D, bool KV8>
bool regs_ok() {
  // the register split is only safe when the kernel launches with exactly
  // REG_LAUNCH registers per thread
  static int ok = -1;
  if (ok < 0) {
    cudaFuncAttributes fa{};
    cudaFuncAttributes fw{};
    ok = cudaFuncGetAttributes(&fa, prefill_tc2_kernel<T, D, KV8, false>) == cudaSuccess &&
         cudaFuncGetAttributes(&fw, prefill_tc2_kernel<T, D, KV8, true>) == cudaSuccess &&
         fa.numRegs == REG_LAUNCH && fw.numRegs == REG_LAUNCH;
  }
  return ok == 1;
}

}  // namespace

bool prefill_tc2_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16) || cache_tokens >= (int64_t(1) << 31))
    return false;
  const bool bf = q_dtype == PA_BF16;
  if (kv_dtype == PA_E5M2 && d == 128)
    return bf ? regs_ok<__nv_bfloat16, 128, true>() : regs_ok<__half, 128, true>();
  if (kv_dtype != q_dtype || !(d == 64 || d == 128)) return false;
  if (d == 64) return bf ? regs_ok<__nv_bfloat16, 64, false>() : regs_ok<__half, 64, false>();
  return bf ? regs_ok<__nv_bfloat16, 128, false>() : regs_ok<__half, 128, false>();
}

cudaError_t launch_prefill_tc2(const AttnArgs& a, int q_dtype, int kv_dtype, int grid_x,
                               cudaStream_t st) {
  if (grid_x == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  // boxes of one 16-token page slot, and of one 128-key tile (BN)
  static_assert(Tc2Cfg<64, false>::BN == 128 && Tc2Cfg<128, false>::BN == 128 &&
                    Tc2Cfg<128, true>::BN == 128,
                "tile box");
  CUtensorMap tk, tv, tkw, tvw;
  if (!encode_kv_map(&tk, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map_rows(&tkw, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens, 128) ||
      !encode_kv_map_rows(&tvw, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens, 128))
    return cudaErrorInvalidValue;
  const bool bf = q_dtype == PA_BF16;
  if (kv_dtype == PA_E5M2) {
    if (a.p.d != 128) return cudaErrorInvalidValue;
    return bf ? launch_tc2<__nv_bfloat16, 128, true>(a, tk, tv, tkw, tvw, grid_x, st)
              : launch_tc2<__half, 128, true>(a, tk, tv, tkw, tvw, grid_x, st);
  }
  switch (a.p.d) {
    case 64: return bf ? launch_tc2<__nv_bfloat16, 64, false>(a, tk, tv, tkw, tvw, grid_x, st)
                       : launch_tc2<__half, 64, false>(a, tk, tv, tkw, tvw, grid_x, st);
    case 128: return bf ? launch_tc2<__nv_bfloat16, 128, false>(a, tk, tv, tkw, tvw, grid_x, st)
                        : launch_tc2<__half, 128, false>(a, tk, tv, tkw, tvw, grid_x, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
