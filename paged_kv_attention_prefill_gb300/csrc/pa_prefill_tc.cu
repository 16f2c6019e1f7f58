// Varlen causal paged prefill on the tcgen05 tensor cores (sm_103a), head
// dim 256: `prefill_tc_kernel` for 16-bit caches, `prefill_tc8_kernel` (at
// the end of the file) for fp8 E5M2 caches widened in shared memory.
//
// Computes the same attention as every other path of the library (the
// packed-varlen interface with one block table per row and bottom-right
// causal alignment, GQA, online softmax over key tiles: vllm-rlt PR #128,
// "Purpose", prefill bullets), laid out for d = 256, where TMEM holds one
// query tile's O (256 columns) next to little else:
//
//  * A CTA owns 128 GQA-packed query rows of one (row, KV head) -- the query
//    heads that share the KV head stacked into the MMA's M dimension
//    (1Cat-vLLM PR #1279, commit 1).
//  * Q lives in TMEM (128 columns of 16-bit pairs) as the A operand of
//    S = Q K^T, so the S product reads only K from shared memory (an MMA
//    with both operands there, M = N = 128, asks for the whole shared-memory
//    bandwidth) and S tiles have 128 keys (an N = 64 MMA runs at about two
//    thirds of the rate).  TMEM: S 128 columns, O 256, Q 128.
//  * P goes to shared memory (the A operand of P V), so S's columns are free
//    as soon as the softmax holds S in registers: S(j + 1) is computed while
//    the softmax of tile j runs.
//  * Warp 0 streams K tiles (128 keys, two stages) and warp 2 V half tiles
//    (64 keys, two stages) with TMA, one box per 16-token page slot
//    straight from the block table (1Cat-vLLM PR #616, original description:
//    any page size that is a multiple of 16); the slot holding the row's last
//    key is copied by hand with the keys past the row's end zero-filled.
//    With pages of at least 128 tokens (a kernel instance of its own), a
//    unit whose slots are one run of one page takes one box per 128-byte
//    chunk instead: the issue of one TMA request per slot and chunk, not the
//    copies' flight time, was what held these kernels back (the mixed
//    workload's chunk row, pages of 784 tokens: 6.83 -> 5.31 ms).
//  * Warp 1, one thread, issues S(0), then per key tile j: S(j + 1) once the
//    softmax has read S(j), and O += P(j) V in two 64-key halves, each once
//    that half of P(j) is in shared memory.
//  * Warps 4-11, two warpgroups sharing each query row (TMEM lane) by key
//    columns, read S, mask, swap their partial row maxima through shared
//    memory, run the online softmax and write their half of P, once the
//    previous tile's product has read it.  O is rescaled in TMEM only when a
//    row's maximum grows by more than 2^8, after that product is done.
//    Finally they normalise O and store their halves of the rows.
//
// Every wait is bounded (about two seconds); a CTA that runs out sets a
// workspace flag, drains its own copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "pa_sm100.cuh"

namespace pa {
namespace {

using namespace sm100;

struct TcCfg {
  static constexpr int D = 256;
  static constexpr int BM = 128;                      // query rows per CTA = TMEM lanes
  static constexpr int BN = 128;                      // keys per S tile
  static constexpr int HB = 64;                       // keys per V stage (half a tile)
  // Shared memory: K 2 x 64 KB + V 2 x 32 KB + P 32 KB + 1 KB; the K/V
  // rings are what is left for hiding the copies' latency
  static constexpr int KS = 2, VS = 2;                // K tile stages, V half stages
  static constexpr int NCH = D / 64;                  // 128-byte column chunks of d
  static constexpr uint32_t K_BYTES = BN * D * 2;     // K of one tile: [chunk][128 keys][128 B]
  static constexpr uint32_t V_BYTES = HB * D * 2;     // V of a half tile: [chunk][64 keys][128 B]
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KS * K_BYTES;
  static constexpr uint32_t P_BYTES = BM * BN * 2;    // P: [64-key half][128 rows][128 B]
  static constexpr uint32_t OFF_P = OFF_V + VS * V_BYTES;
  static constexpr uint32_t OFF_X = OFF_P + P_BYTES;  // [2][128] floats: partial maxima / sums
  static constexpr uint32_t OFF_BAR = OFF_X + 2 * BM * 4;
  static constexpr uint32_t BAR_AREA = 192;           // mbarriers, then TMEM address and flags
  static constexpr uint32_t SMEM = OFF_BAR + BAR_AREA + 16 + 1024;  // alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = BN;               // S in [0, BN)
  static constexpr uint32_t Q_COL = O_COL + D;
  // barrier indices
  static constexpr int B_KF = 0, B_KE = KS, B_VF = 2 * KS, B_VE = 2 * KS + VS,
                       B_SF = 2 * KS + 2 * VS,        // S(j) written
      B_SC = B_SF + 1,                                // S(j) read by the softmax (8 warps)
      B_PF = B_SC + 1,                                // [2] P(j) half h in shared memory (4 warps)
      B_PV = B_PF + 2,                                // [2] O += P(j) V, half h, done
      B_Q = B_PV + 2,                                 // Q in TMEM (8 warps)
      B_DRAIN = B_Q + 1, NBAR = B_DRAIN + 1;
  static_assert(Q_COL + D / 2 == TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NBAR * 8 <= BAR_AREA, "barrier area");
};

template <typename T, bool DEC, bool WIDE>
__global__ void __launch_bounds__(384, 1)
    prefill_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmKw,
                      const __grid_constant__ CUtensorMap tmVw) {
  using C = TcCfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sP = base + C::OFF_P;
  volatile float* xch = reinterpret_cast<volatile float*>(smem + C::OFF_X);
  const uint32_t bar0 = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::BAR_AREA);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::BAR_AREA + 4);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- barriers and TMEM ----------------------------------------------------
  auto init_barriers = [&]() {
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_KF + s), 1);
      mbar_init(bar(C::B_KE + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_VF + s), 1);
      mbar_init(bar(C::B_VE + s), 1);
    }
    mbar_init(bar(C::B_SF), 1);
    mbar_init(bar(C::B_SC), 8);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::B_PF + h), 4);
      mbar_init(bar(C::B_PV + h), 1);
    }
    mbar_init(bar(C::B_Q), 8);
    mbar_init(bar(C::B_DRAIN), 1);
    fence_mbar_init();
  };
  if (threadIdx.x == 0) {
    init_barriers();
    *abort_flag = 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- work items ------------------------------------------------------------
  // Prefill: one item per CTA, a 1-D grid with the KV head slowest (CTAs that
  // run together read the same heads' K/V: L2 reuse; within a head the work
  // list is longest-first).
  // DEC (long-row decode, PA_SPLITS_BY_LENGTH): the CTAs take the (item, KV
  // head) units of the long-row list in turn; an item is one split of a
  // decode row's length-only partition for one block of its GQA-packed query
  // rows, and its result is that split's fp32 partial state (acc, m, l),
  // written where the decode kernel writes it.  The barriers are made afresh
  // for every unit after the first; TMEM is held for all of them.
  const int n_work = DEC ? (int)*a.n_long * p.hkv : 1;
  int done_units = 0;
  for (int unit = DEC ? (int)blockIdx.x : 0; unit < n_work;
       unit += DEC ? (int)gridDim.x : n_work) {
  int b, mb, part = 0, kh, split = 0;
  int64_t slot_base = 0;
  if constexpr (DEC) {
    const int2 wi = a.long_items[unit / p.hkv];
    kh = unit % p.hkv;
    b = wi.x & 0xFFFFFF;
    mb = wi.x >> 24;
    split = wi.y;
  } else {
    const int n_items = (int)(gridDim.x / p.hkv);
    const int item = blockIdx.x % n_items;
    kh = blockIdx.x / n_items;
    if (item >= (int)*a.n_tiles) continue;
    const int2 wi = a.tiles[item];
    b = wi.x;
    mb = wi.y & 0xFFFFFF;
    part = wi.y >> 24;
  }
  const int qs = __ldg(p.cu_q + b);
  const int qb = __ldg(p.cu_q + b + 1) - qs;
  const int L = __ldg(p.seq_lens + b);
  if (qb <= 0) continue;
  if (qs < 0 || qs + qb > p.total_q) {
    if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    continue;
  }
  const int g = p.g, M = qb * g, R0 = mb * C::BM;
  if (R0 >= M) continue;
  int k0, k1;
  bool cut;
  if constexpr (DEC) {
    slot_base = a.dec_base ? (int64_t)__ldg(a.dec_base + b) : (int64_t)qs;
    if (slot_base < 0 || slot_base + qb > a.max_slots) continue;
    const int tps = dec_split_tiles(L, 1);
    k0 = split * tps * DEC_KT;
    if (k0 >= L) continue;
    k1 = min(k0 + tps * DEC_KT, L);
    cut = true;
  } else {
    const int r_last = min(R0 + C::BM, M) - 1;
    const int k_end = min(L, L - qb + r_last / g + 1);  // keys any row of the tile can see
    // the item's key range [k0, k1): the whole range, or one part of it
    int per_u;
    cut = pf_part_count(k_end, a.pf_parts, a.pf_min_units, &per_u) > 1;
    k0 = cut ? part * per_u * PF_UNIT : 0;
    k1 = cut ? min(k_end, (part + 1) * per_u * PF_UNIT) : k_end;
  }
  const int n_tiles = k1 > k0 ? (k1 - k0 + C::BN - 1) / C::BN : 0;
  if (DEC && done_units > 0) {
    // every role is past the previous unit's last barrier operation (the
    // block-wide barrier at its end): make the barriers afresh
    if (threadIdx.x == 0) {
      for (int i = 0; i < C::NBAR; ++i) mbar_inval(bar(i));
      init_barriers();
    }
    __syncthreads();
  }
  ++done_units;

  if (warp == 0 || warp == 2) {
    // ============== producers: warp 0 streams K tiles, warp 2 V halves =======
    // Unit u of a producer: a K tile of BN keys (warp 0) or a V half tile of
    // HB keys (warp 2), each a run of 16-token page slots.
    const bool isK = warp == 0;
    const int NS = isK ? C::KS : C::VS;
    const int UK = isK ? C::BN : C::HB;                 // keys per unit
    const uint32_t UB = isK ? C::K_BYTES : C::V_BYTES;  // bytes per unit
    const int B_FULL = isK ? C::B_KF : C::B_VF, B_EMPTY = isK ? C::B_KE : C::B_VE;
    const uint32_t ring = isK ? sK : sV;
    const void* tmap = isK ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmV);
    // the same view with one box per unit (UK rows), for units whose keys
    // lie in one page
    const void* tmapw = isK ? static_cast<const void*>(&tmKw) : static_cast<const void*>(&tmVw);
    const T* cache = static_cast<const T*>(isK ? a.kc : a.vc);
    if (lane == 0) {
      tma_prefetch_desc(tmap);
      if (WIDE) tma_prefetch_desc(tmapw);
    }
    const int P = p.page_size;
    const int64_t bt_row = (int64_t)b * p.max_pages;
    const int n_units = isK ? n_tiles : 2 * n_tiles;
    int u = 0;
    bool ok = true;
    for (; u < n_units; ++u) {
      const int st = u % NS;
      if (u >= NS) ok = mbar_wait(bar(B_EMPTY + st), ((u / NS) - 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int kbase = k0 + u * UK;
      const uint32_t dst = ring + st * UB;
      const int slots = UK / 16;
      // slot `lane`: 1 = whole slot by TMA, 2 = partial (copied by hand), 3 = zero-fill
      int kind = 0, tok0 = 0;
      if (lane < slots) {
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
      if (WIDE &&
          __all_sync(0xffffffffu, lane >= slots || (kind == 1 && tok0 == tok_first + 16 * lane))) {
        // every slot whole and in one run of one page: one box per chunk
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_FULL + st), (uint32_t)UK * D * 2u);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(dst + c * (UK * 128), tmapw, c * 64, kh, tok_first, bar(B_FULL + st));
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
          st_shared_v4(dst + c * (UK * 128) + row * 128 + ((piece ^ (row & 7)) << 4), v);
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
          tma_load_3d(dst + c * (UK * 128) + lane * 16 * 128, tmap, c * 64, kh, tok0,
                      bar(B_FULL + st));
      }
    }
    if (!ok) {
      // copies this warp started may still be landing: wait for them
      for (int uu = max(0, u - NS); uu < u; ++uu)
        mbar_drain(bar(B_FULL + uu % NS), (uu / NS) & 1, p.err);
    } else if (DEC) {
      // the barriers are made afresh for the next unit: first let the
      // products release the last stages (their commits arrive here)
      for (int uu = max(0, n_units - NS); uu < n_units; ++uu)
        mbar_wait(bar(B_EMPTY + uu % NS), (uu / NS) & 1, abort_flag, p.err);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (one thread) =======================
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
      constexpr uint32_t idS = idesc_f16(fmt, 128, C::BN, false);
      constexpr uint32_t idO = idesc_f16(fmt, 128, D, true);
      // S(j) = Q K(j)^T: A = Q from TMEM (16 head-dim columns = 8 columns
      // of 16-bit pairs per step)
      auto issue_S = [&](int j) {
        const int st = j % C::KS;
        if (!mbar_wait(bar(C::B_KF + st), (j / C::KS) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint64_t b0 = sdesc_sw128(sK + st * C::K_BYTES, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t bd = b0 + (uint64_t)(((k >> 2) * (C::BN * 128) + (k & 3) * 32) >> 4);
          tc_mma_f16_ts(tmem, tmem + C::Q_COL + 8 * k, bd, idS, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF));
        tc_commit(bar(C::B_KE + st));
        return true;
      };
      bool ok = n_tiles == 0 || mbar_wait(bar(C::B_Q), 0, abort_flag, p.err);
      if (ok) tc_fence_after();
      if (ok && n_tiles > 0) ok = issue_S(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        // S(j + 1) as soon as the softmax holds S(j) in registers (P goes to
        // shared memory, so nothing else lives in S's columns)
        if (j + 1 < n_tiles) {
          ok = mbar_wait(bar(C::B_SC), j & 1, abort_flag, p.err);
          if (ok) {
            tc_fence_after();
            ok = issue_S(j + 1);
          }
          if (!ok) break;
        }
        // O += P(j) V(j) in two halves of HB keys, each once its half of
        // P(j) is in shared memory: A = P (K-major), B = V (N-major)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = 2 * j + h, sv = q % C::VS;
          ok = mbar_wait(bar(C::B_PF + h), j & 1, abort_flag, p.err);
          if (ok) ok = mbar_wait(bar(C::B_VF + sv), (q / C::VS) & 1, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint64_t a0 = sdesc_sw128(sP + h * (C::BM * 128), 16, 1024);
          const uint64_t v0 = sdesc_sw128(sV + sv * C::V_BYTES, C::HB * 128, 1024);
#pragma unroll
          for (int k = 0; k < C::HB / 16; ++k) {
            const uint64_t ad = a0 + (uint64_t)((k * 32) >> 4);
            const uint64_t bd = v0 + (uint64_t)((k * 16 * 128) >> 4);
            tc_mma_f16(tmem + C::O_COL, ad, bd, idO, (j > 0 || h > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(C::B_VE + sv));
          tc_commit(bar(C::B_PV + h));
        }
      }
      // nothing this thread issued may still run once TMEM is freed
      tc_commit(bar(C::B_DRAIN));
      mbar_drain(bar(C::B_DRAIN), 0, p.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============ Q, softmax, epilogue =========================================
    // Warpgroup hf (warps 4-7: hf = 0, warps 8-11: hf = 1) owns key columns
    // [hf BN/2, (hf+1) BN/2) of each S tile and head-dim columns [hf d/2,
    // (hf+1) d/2) of Q and of O.  The loop never leaves early: after a
    // timed-out wait it runs on (flag raised, waits return at once), so both
    // warpgroups always meet the same barriers.
    constexpr int HN = C::BN / 2, HD = D / 2;
    const int hf = warp >= 8 ? 1 : 0;
    const int q4 = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;     // tile row == TMEM lane
    const int R = R0 + r;
    const bool valid = R < M;
    const int i = valid ? R / g : 0, hg = valid ? R % g : 0;
    // last visible key, from k0 (a decode split also ends at k1)
    const int last = valid ? min(L - qb + i, k1 - 1) - k0 : NO_MASK;
    const int64_t qoff = ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    {
      // this warpgroup's half of the row's Q into TMEM (16-bit pairs)
      const T* qrow = static_cast<const T*>(a.q) + qoff + hf * HD;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(qrow + c * 64 + w * 8))
                                : make_uint4(0u, 0u, 0u, 0u);
          v[4 * w] = u.x;
          v[4 * w + 1] = u.y;
          v[4 * w + 2] = u.z;
          v[4 * w + 3] = u.w;
        }
        tmem_st_x32(trow + C::Q_COL + hf * (HD / 2) + c * 32, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_Q));
    }
    const float sl2 = p.sl2;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      mbar_wait(bar(C::B_SF), j & 1, abort_flag, p.err);
      tc_fence_after();
      // S(j) may run while the previous P V product still does: O and P's
      // buffer are touched only after waiting for that product
      // the logits as pairs (keys 2k, 2k + 1) for the paired fp32
      // instructions below, each lane of which rounds as its scalar form does
      float2 x[HN / 2];
      float mt;  // max raw logit of this half tile (masked keys -> -inf)
      {
        uint32_t u[HN];
        mt = tmem_ld_red_max_x64(trow + hf * HN, u);  // the load also returns the max
#pragma unroll
        for (int k = 0; k < HN / 2; ++k)
          x[k] = make_float2(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1]));
      }
      const int kb = j * C::BN + hf * HN;
      if (kb + HN - 1 > last) {
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) {
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
        for (int k = 4; k < HN / 2; ++k) {
          pm[2 * (k & 3)] = fmaxf(pm[2 * (k & 3)], x[k].x);
          pm[2 * (k & 3) + 1] = fmaxf(pm[2 * (k & 3) + 1], x[k].y);
        }
        mt = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      }
      {
        // swap partial maxima through shared memory; then S(j) is consumed
        // and the next S may overwrite it.  (The next tile's write here comes
        // after S(j + 1), which waits for every warp's arrival below, so the
        // other warpgroup has read this value by then.)
        xch[hf * C::BM + r] = mt;
        named_bar_sync(1, 256);
        mt = fmaxf(mt, xch[(hf ^ 1) * C::BM + r]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_SC));
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
      if (__any_sync(0xffffffffu, need)) {
        // the previous P V product (its commit covers every earlier MMA)
        mbar_wait(bar(C::B_PV + 1), (j - 1) & 1, abort_flag, p.err);
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st_x32(trow + C::O_COL + hf * HD + c * 32, o);
        }
      }
      // partial row sums, fixed order: key k adds into sum k mod 8
      float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      {
        const float2 sl2v = make_float2(sl2, sl2), nmv = make_float2(nmu, nmu);
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) {
          float2 y = __ffma2_rn(x[k], sl2v, nmv);
          y.x = ex2(y.x);
          y.y = ex2(y.y);
          x[k] = y;
          ps[k & 3] = __fadd2_rn(ps[k & 3], y);
        }
      }
      {
        // P (16-bit) of this warpgroup's keys into half hf of P's buffer
        // (the A operand of P V: 128-byte rows, 128-byte swizzle), once the
        // previous tile's product has read that half; one arrival per warp
        uint32_t pk[HN / 2];
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) pk[k] = pack2<T>(x[k].x, x[k].y);
        if (j > 0) mbar_wait(bar(C::B_PV + hf), (j - 1) & 1, abort_flag, p.err);
        const uint32_t prow = sP + hf * (C::BM * 128) + r * 128;
#pragma unroll
        for (int pc = 0; pc < 8; ++pc)
          st_shared_v4(prow + ((pc ^ (r & 7)) << 4),
                       make_uint4(pk[4 * pc], pk[4 * pc + 1], pk[4 * pc + 2], pk[4 * pc + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PF + hf));
      }
      const float rs = ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) +
                       ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
      l = l * factor + rs;
    }
    // ---- epilogue: out = O / (l_0 + l_1) * v_scale, or this part's state ----
    if (n_tiles > 0) {
      mbar_wait(bar(C::B_PV + 1), (n_tiles - 1) & 1, abort_flag, p.err);
      tc_fence_after();
    }
    // the partial row sums, swapped through shared memory once every read
    // of the maxima is done, added in warpgroup order
    named_bar_sync(1, 256);
    xch[hf * C::BM + r] = l;
    named_bar_sync(1, 256);
    const float lo = xch[(hf ^ 1) * C::BM + r];
    const float lt = hf == 0 ? l + lo : lo + l;
    T* orow = static_cast<T*>(a.out) + qoff + hf * HD;
    if (cut) {
      // this part's unnormalised O (each warpgroup its d / 2 columns), the
      // maximum it is relative to and the row sum, for the merge: a prefill
      // key-range part, or a decode split (in the decode kernel's layout)
      const int64_t slot =
          DEC ? ((slot_base + i) * p.hq + kh * g + hg) * a.split_stride + split
              : ((int64_t)(qs + i) * p.hq + kh * g + hg) * a.pf_parts + part;
      float2* mlp = DEC ? a.part_ml : a.pf_ml;
      if (valid && hf == 0)
        mlp[slot] = make_float2(n_tiles > 0 ? m_used : -INFINITY, n_tiles > 0 ? lt : 0.f);
      float* prow = (DEC ? a.part_acc : a.pf_acc) + slot * D + hf * HD;
      if (n_tiles > 0) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
          if (valid) {
#pragma unroll
            for (int w = 0; w < 8; ++w)
              *reinterpret_cast<uint4*>(prow + c * 32 + 4 * w) =
                  make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
          }
        }
      }
    } else if (n_tiles > 0) {
      const float inv = lt > 0.f ? p.v_scale / lt : 0.f;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
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
      for (int c = 0; c < HD / 8; ++c)
        *reinterpret_cast<uint4*>(orow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  }  // work items

  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// fp8 E5M2 caches at d = 256: Q in TMEM and 128-key S tiles as above, but P
// stays over S in TMEM (its 32 KB of shared memory go to the code rings), so
// S(j) waits for the previous P V product.  The codes are streamed by TMA
// into their own rings (warp 0 the K codes, warp 2 the V codes, each ring
// requested as soon as its stage is free; warp 3 idle) and widened by a
// fourth warpgroup (warps 12-15) into the 16-bit tiles the MMAs read: an E5M2 code is
// the high byte of the binary16 of the same value, and for bf16 Q it is
// widened through fp32, also exactly.  Shared memory: 16-bit K 64 KB (one
// tile), 16-bit V 2 x 32 KB (the two halves of a tile), K codes 2 x 32 KB,
// V codes 2 x 16 KB, and the 1 KB through which the two softmax warpgroups
// swap partial row maxima and sums.
struct Tc8Cfg {
  static constexpr int D = 256;
  static constexpr int BM = 128;                      // query rows per CTA = TMEM lanes
  static constexpr int BN = 128;                      // keys per S tile
  static constexpr int HB = 64;                       // keys per V half
  static constexpr int NC8 = D / 128;                 // 128-byte chunks of a code row
  static constexpr uint32_t K_BYTES = BN * D * 2;     // 16-bit K: [chunk][128 keys][128 B]
  static constexpr uint32_t V_BYTES = HB * D * 2;     // 16-bit V half: [chunk][64 keys][128 B]
  static constexpr uint32_t K8_BYTES = BN * D;        // K codes: [chunk][128 keys][128 B]
  static constexpr uint32_t V8_BYTES = HB * D;        // V codes: [chunk][64 keys][128 B]
  static constexpr int S8 = 2;                        // code stages (K and V each)
  static constexpr int NW = 4;                        // widening warps (12-15)
  static constexpr int THREADS = 512;                 // four warpgroups
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + K_BYTES;
  static constexpr uint32_t OFF_K8 = OFF_V + 2 * V_BYTES;
  static constexpr uint32_t OFF_V8 = OFF_K8 + S8 * K8_BYTES;
  static constexpr uint32_t OFF_X = OFF_V8 + S8 * V8_BYTES;  // [2][128] floats: partial maxima / sums
  static constexpr uint32_t OFF_BAR = OFF_X + 2 * BM * 4;
  static constexpr uint32_t BAR_AREA = 192;           // mbarriers, then TMEM address and flags
  static constexpr uint32_t SMEM = OFF_BAR + BAR_AREA + 16 + 1024;  // alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = BN;               // S in [0, BN), P over its first BN / 2
  static constexpr uint32_t Q_COL = O_COL + D;
  // barrier indices
  static constexpr int B_KF = 0,                      // 16-bit K tile widened (NW warps)
      B_KE = B_KF + 1,                                // S(j) done with it
      B_VF = B_KE + 1,                                // [2] 16-bit V half h widened (NW warps)
      B_VE = B_VF + 2,                                // [2] P V half h done with it
      B_SF = B_VE + 2,                                // S(j) written
      B_PF = B_SF + 1,                                // P(j) written (8 warps)
      B_PV = B_PF + 1,                                // O += P(j) V done
      B_Q = B_PV + 1,                                 // Q in TMEM (8 warps)
      B_DRAIN = B_Q + 1,
      B_K8F = B_DRAIN + 1, B_K8E = B_K8F + S8,        // code rings: full (TMA) / empty (NW warps)
      B_V8F = B_K8E + S8, B_V8E = B_V8F + S8, NBAR = B_V8E + S8;
  static_assert(Q_COL + D / 2 == TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NBAR * 8 <= BAR_AREA, "barrier area");
};

template <typename T, bool WIDE>
__global__ void __launch_bounds__(Tc8Cfg::THREADS, 1)
    prefill_tc8_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmKw,
                       const __grid_constant__ CUtensorMap tmVw) {
  using C = Tc8Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t sK8 = base + C::OFF_K8, sV8 = base + C::OFF_V8;
  volatile float* xch = reinterpret_cast<volatile float*>(smem + C::OFF_X);
  const uint32_t bar0 = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::BAR_AREA);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::BAR_AREA + 4);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item (uniform over the CTA) -----------------------------------
  // 1-D grid, KV head slowest: CTAs that run together read the same heads'
  // K/V (L2 reuse); within a head the work list is longest-first
  const int n_items = (int)(gridDim.x / p.hkv);
  const int item = blockIdx.x % n_items, kh = blockIdx.x / n_items;
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
  const int g = p.g, M = qb * g, R0 = mb * C::BM;
  if (R0 >= M) return;
  const int r_last = min(R0 + C::BM, M) - 1;
  const int k_end = min(L, L - qb + r_last / g + 1);  // keys any row of the tile can see
  // the item's key range [k0, k1): the whole range, or one part of it
  int per_u;
  const bool cut = pf_part_count(k_end, a.pf_parts, a.pf_min_units, &per_u) > 1;
  const int k0 = cut ? part * per_u * PF_UNIT : 0;
  const int k1 = cut ? min(k_end, (part + 1) * per_u * PF_UNIT) : k_end;
  const int n_tiles = k1 > k0 ? (k1 - k0 + C::BN - 1) / C::BN : 0;

  // ---- barriers and TMEM ----------------------------------------------------
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KF), C::NW);
    mbar_init(bar(C::B_KE), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_VF + s), C::NW);
      mbar_init(bar(C::B_VE + s), 1);
    }
    mbar_init(bar(C::B_SF), 1);
    mbar_init(bar(C::B_PF), 8);
    mbar_init(bar(C::B_PV), 1);
    mbar_init(bar(C::B_Q), 8);
    mbar_init(bar(C::B_DRAIN), 1);
    for (int s = 0; s < C::S8; ++s) {
      mbar_init(bar(C::B_K8F + s), 1);
      mbar_init(bar(C::B_K8E + s), C::NW);
      mbar_init(bar(C::B_V8F + s), 1);
      mbar_init(bar(C::B_V8E + s), C::NW);
    }
    *abort_flag = 0;
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

  if (warp == 0 || warp == 2) {
    // ===== warp 0 streams the K codes of each key tile (128 keys), warp 2 ==
    // the V codes in 64-key halves, into the code rings: one TMA box (16
    // keys x 128 codes) per page slot and 128-code chunk of the row (with
    // pages of 128 tokens or more, one per chunk of a unit in one page); the slot
    // holding the row's last key is copied by hand, zero-filled past the
    // row's end.  Two warps, so that a ring waiting for its stage to be
    // widened never holds back the other ring's requests (the codes take
    // thousands of cycles to arrive).
    const bool isK = warp == 0;
    const uint8_t* cache8 = static_cast<const uint8_t*>(isK ? a.kc : a.vc);
    const void* tmap = isK ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmV);
    // the same view with one box per unit, for units whose keys lie in one page
    const void* tmapw = isK ? static_cast<const void*>(&tmKw) : static_cast<const void*>(&tmVw);
    if (lane == 0) {
      tma_prefetch_desc(tmap);
      if (WIDE) tma_prefetch_desc(tmapw);
    }
    const int P = p.page_size;
    const int64_t bt_row = (int64_t)b * p.max_pages;
    // `rows` keys from kbase into the [chunk][rows][128 B] code tile dst
    auto unit = [&](const void* tmap, const void* tmapw, const uint8_t* cache, int kbase, int rows,
                    uint32_t dst, uint32_t fb) {
      // slot `lane`: 1 = whole slot by TMA, 2 = partial (by hand), 3 = zero-fill
      int kind = 0, tok0 = 0;
      if (lane < rows / 16) {
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
      if (WIDE && __all_sync(0xffffffffu,
                             lane >= rows / 16 || (kind == 1 && tok0 == tok_first + 16 * lane))) {
        // every slot whole and in one run of one page: one box per chunk
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, (uint32_t)rows * (uint32_t)D);
#pragma unroll
          for (int c8 = 0; c8 < C::NC8; ++c8)
            tma_load_3d(dst + c8 * (rows * 128), tmapw, c8 * 128, kh, tok_first, fb);
        }
        __syncwarp();
        return;
      }
      uint32_t manual = __ballot_sync(0xffffffffu, kind >= 2);
      while (manual) {
        const int s = __ffs(manual) - 1;
        manual &= manual - 1;
        const int ks = __shfl_sync(0xffffffffu, kind, s);
        const int t0 = __shfl_sync(0xffffffffu, tok0, s);
        const int nvalid = ks == 2 ? L - (kbase + 16 * s) : 0;
        for (int it = lane; it < 16 * (D / 16); it += 32) {
          const int u16 = it % (D / 16), rr = it / (D / 16);  // 16-code unit of key row rr
          const int c8 = u16 >> 3, pu = u16 & 7;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (rr < nvalid)
            v = __ldg(reinterpret_cast<const uint4*>(cache + ((int64_t)(t0 + rr) * p.hkv + kh) * D +
                                                     u16 * 16));
          const int row = 16 * s + rr;
          st_shared_v4(dst + c8 * (rows * 128) + row * 128 + ((pu ^ (row & 7)) << 4), v);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int n_tma = __popc(__ballot_sync(0xffffffffu, kind == 1));
      if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_tma * 16u * (uint32_t)D);
      __syncwarp();
      if (kind == 1) {
#pragma unroll
        for (int c8 = 0; c8 < C::NC8; ++c8)
          tma_load_3d(dst + c8 * (rows * 128) + lane * 16 * 128, tmap, c8 * 128, kh, tok0, fb);
      }
    };
    // units: K tiles of BN keys (warp 0) or V halves of HB keys (warp 2)
    const int n_units = isK ? n_tiles : 2 * n_tiles;
    const int UK = isK ? C::BN : C::HB;
    const uint32_t ring = isK ? sK8 : sV8, UB = isK ? C::K8_BYTES : C::V8_BYTES;
    const int B_FULL = isK ? C::B_K8F : C::B_V8F, B_EMPTY = isK ? C::B_K8E : C::B_V8E;
    bool ok = true;
    int u = 0;  // units started
    for (; u < n_units; ++u) {
      if (u >= C::S8) ok = mbar_wait(bar(B_EMPTY + (u & 1)), ((u >> 1) - 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      unit(tmap, tmapw, cache8, k0 + u * UK, UK, ring + (u & 1) * UB, bar(B_FULL + (u & 1)));
    }
    if (!ok) {
      // copies this warp started may still be landing: wait for them
      for (int uu = max(0, u - C::S8); uu < u; ++uu)
        mbar_drain(bar(B_FULL + (uu & 1)), (uu >> 1) & 1, p.err);
    }
  } else if (warp >= 12) {
    // ===== warps 12-15 widen every K tile (32 keys each) and V half (16 =====
    // keys each) into the 16-bit tiles; lane = 16 codes of one key per step
    const int ww = warp - 12;
    const int u8 = lane & 7, c = u8 >> 2, va = 2 * (u8 & 3);
    auto widen = [&](uint32_t src, uint32_t dst, int rows, int key0, int nkeys) {
#pragma unroll
      for (int c8 = 0; c8 < C::NC8; ++c8) {
#pragma unroll 4
        for (int it = 0; it < nkeys / 4; ++it) {
          const int key = key0 + 4 * it + (lane >> 3);
          const uint4 w = ld_shared_v4(src + c8 * (rows * 128) + key * 128 + ((u8 ^ (key & 7)) << 4));
          uint4 lo, hi;
          e5m2x4_to<T>(w.x, lo.x, lo.y);
          e5m2x4_to<T>(w.y, lo.z, lo.w);
          e5m2x4_to<T>(w.z, hi.x, hi.y);
          e5m2x4_to<T>(w.w, hi.z, hi.w);
          const uint32_t row = dst + (2 * c8 + c) * (rows * 128) + key * 128;
          st_shared_v4(row + ((va ^ (key & 7)) << 4), lo);
          st_shared_v4(row + (((va + 1) ^ (key & 7)) << 4), hi);
        }
      }
      // the MMAs read the tile through the async proxy; TMA overwrites the
      // codes next
      fence_proxy_async_smem();
      __syncwarp();
    };
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      ok = mbar_wait(bar(C::B_K8F + (j & 1)), (j >> 1) & 1, abort_flag, p.err);
      if (ok && j >= 1) ok = mbar_wait(bar(C::B_KE), (j - 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      widen(sK8 + (j & 1) * C::K8_BYTES, sK, C::BN, (C::BN / C::NW) * ww, C::BN / C::NW);
      if (lane == 0) {
        mbar_arrive(bar(C::B_KF));
        mbar_arrive(bar(C::B_K8E + (j & 1)));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = 2 * j + h;
        ok = mbar_wait(bar(C::B_V8F + (q & 1)), (q >> 1) & 1, abort_flag, p.err);
        if (ok && j >= 1) ok = mbar_wait(bar(C::B_VE + h), (j - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        widen(sV8 + (q & 1) * C::V8_BYTES, sV + h * C::V_BYTES, C::HB, (C::HB / C::NW) * ww,
              C::HB / C::NW);
        if (lane == 0) {
          mbar_arrive(bar(C::B_VF + h));
          mbar_arrive(bar(C::B_V8E + (q & 1)));
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (one thread) =======================
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
      constexpr uint32_t idS = idesc_f16(fmt, 128, C::BN, false);
      constexpr uint32_t idO = idesc_f16(fmt, 128, D, true);
      bool ok = n_tiles == 0 || mbar_wait(bar(C::B_Q), 0, abort_flag, p.err);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < n_tiles; ++j) {
        // S(j) = Q K(j)^T: A = Q from TMEM; it overwrites P(j-1), so the
        // previous P V product must be done
        ok = mbar_wait(bar(C::B_KF), j & 1, abort_flag, p.err);
        if (ok && j >= 1) ok = mbar_wait(bar(C::B_PV), (j - 1) & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint64_t b0 = sdesc_sw128(sK, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t bd = b0 + (uint64_t)(((k >> 2) * (C::BN * 128) + (k & 3) * 32) >> 4);
          tc_mma_f16_ts(tmem, tmem + C::Q_COL + 8 * k, bd, idS, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF));
        tc_commit(bar(C::B_KE));
        // O += P(j) V(j), V in two halves of HB keys
        ok = mbar_wait(bar(C::B_PF), j & 1, abort_flag, p.err);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (ok) ok = mbar_wait(bar(C::B_VF + h), j & 1, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint64_t v0 = sdesc_sw128(sV + h * C::V_BYTES, C::HB * 128, 1024);
#pragma unroll
          for (int k = 0; k < C::HB / 16; ++k) {
            // A = P from TMEM: 16 keys = 8 columns of 16-bit pairs
            const uint64_t bd = v0 + (uint64_t)((k * 16 * 128) >> 4);
            tc_mma_f16_ts(tmem + C::O_COL, tmem + (h * (C::HB / 16) + k) * 8, bd, idO,
                          (j > 0 || h > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(C::B_VE + h));
        }
        if (!ok) break;
        tc_commit(bar(C::B_PV));
      }
      // nothing this thread issued may still run once TMEM is freed
      tc_commit(bar(C::B_DRAIN));
      mbar_drain(bar(C::B_DRAIN), 0, p.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============ Q, softmax, epilogue (warps 4-11) ============================
    // Warpgroup hf (warps 4-7: hf = 0, warps 8-11: hf = 1) owns key columns
    // [hf BN/2, (hf+1) BN/2) of each S tile and head-dim columns [hf d/2,
    // (hf+1) d/2) of Q and of O.  The loop never leaves early: after a
    // timed-out wait it runs on (flag raised, waits return at once), so both
    // warpgroups always meet the same barriers.
    constexpr int HN = C::BN / 2, HD = D / 2;
    const int hf = warp >= 8 ? 1 : 0;
    const int q4 = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;     // tile row == TMEM lane
    const int R = R0 + r;
    const bool valid = R < M;
    const int i = valid ? R / g : 0, hg = valid ? R % g : 0;
    const int last = valid ? L - qb + i - k0 : NO_MASK;  // last visible key, from k0
    const int64_t qoff = ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    {
      // this warpgroup's half of the row's Q into TMEM (16-bit pairs)
      const T* qrow = static_cast<const T*>(a.q) + qoff + hf * HD;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(qrow + c * 64 + w * 8))
                                : make_uint4(0u, 0u, 0u, 0u);
          v[4 * w] = u.x;
          v[4 * w + 1] = u.y;
          v[4 * w + 2] = u.z;
          v[4 * w + 3] = u.w;
        }
        tmem_st_x32(trow + C::Q_COL + hf * (HD / 2) + c * 32, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_Q));
    }
    const float sl2 = p.sl2;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      mbar_wait(bar(C::B_SF), j & 1, abort_flag, p.err);
      tc_fence_after();
      // S(j) was issued after the previous P V product completed: O is stable
      // the logits as pairs (keys 2k, 2k + 1) for the paired fp32
      // instructions below, each lane of which rounds as its scalar form does
      float2 x[HN / 2];
      float mt;  // max raw logit of this half tile (masked keys -> -inf)
      {
        uint32_t u[HN];
        mt = tmem_ld_red_max_x64(trow + hf * HN, u);  // the load also returns the max
#pragma unroll
        for (int k = 0; k < HN / 2; ++k)
          x[k] = make_float2(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1]));
      }
      const int kb = j * C::BN + hf * HN;
      if (kb + HN - 1 > last) {
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) {
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
        for (int k = 4; k < HN / 2; ++k) {
          pm[2 * (k & 3)] = fmaxf(pm[2 * (k & 3)], x[k].x);
          pm[2 * (k & 3) + 1] = fmaxf(pm[2 * (k & 3) + 1], x[k].y);
        }
        mt = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      }
      {
        // swap partial maxima through shared memory (the next tile's write
        // comes after S(j + 1), which waits for this tile's P V product,
        // which waits for both warpgroups' P, published after these reads)
        xch[hf * C::BM + r] = mt;
        named_bar_sync(1, 256);
        mt = fmaxf(mt, xch[(hf ^ 1) * C::BM + r]);
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
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st_x32(trow + C::O_COL + hf * HD + c * 32, o);
        }
      }
      // partial row sums, fixed order: key k adds into sum k mod 8
      float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      {
        const float2 sl2v = make_float2(sl2, sl2), nmv = make_float2(nmu, nmu);
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) {
          float2 y = __ffma2_rn(x[k], sl2v, nmv);
          y.x = ex2(y.x);
          y.y = ex2(y.y);
          x[k] = y;
          ps[k & 3] = __fadd2_rn(ps[k & 3], y);
        }
      }
      {
        // P (16-bit pairs) over this warpgroup's keys: HN / 2 columns at the
        // start of S, then one arrival per warp
        uint32_t pk[HN / 2];
#pragma unroll
        for (int k = 0; k < HN / 2; ++k) pk[k] = pack2<T>(x[k].x, x[k].y);
        tmem_st_x32(trow + hf * (HN / 2), pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PF));
      }
      const float rs = ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) +
                       ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
      l = l * factor + rs;
    }
    // ---- epilogue: out = O / (l_0 + l_1) * v_scale, or this part's state ----
    if (n_tiles > 0) {
      mbar_wait(bar(C::B_PV), (n_tiles - 1) & 1, abort_flag, p.err);
      tc_fence_after();
    }
    // the partial row sums, swapped through shared memory once every read
    // of the maxima is done, added in warpgroup order
    named_bar_sync(1, 256);
    xch[hf * C::BM + r] = l;
    named_bar_sync(1, 256);
    const float lo = xch[(hf ^ 1) * C::BM + r];
    const float lt = hf == 0 ? l + lo : lo + l;
    T* orow = static_cast<T*>(a.out) + qoff + hf * HD;
    if (cut) {
      // this part's unnormalised O (each warpgroup its d / 2 columns), the
      // maximum it is relative to and the row sum, for the merge
      const int64_t slot = ((int64_t)(qs + i) * p.hq + kh * g + hg) * a.pf_parts + part;
      if (valid && hf == 0)
        a.pf_ml[slot] = make_float2(n_tiles > 0 ? m_used : -INFINITY, n_tiles > 0 ? lt : 0.f);
      float* prow = a.pf_acc + slot * D + hf * HD;
      if (n_tiles > 0) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
          if (valid) {
#pragma unroll
            for (int w = 0; w < 8; ++w)
              *reinterpret_cast<uint4*>(prow + c * 32 + 4 * w) =
                  make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
          }
        }
      }
    } else if (n_tiles > 0) {
      const float inv = lt > 0.f ? p.v_scale / lt : 0.f;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(trow + C::O_COL + hf * HD + c * 32, o);
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
      for (int c = 0; c < HD / 8; ++c)
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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

// [tokens, Hkv, d] view of a cache, boxes of `rows` tokens x 1 head x 128
// bytes (64 16-bit elements or 128 fp8 codes), 128-byte swizzle: 16 rows for
// one page slot, a whole key tile or V half for the large-page kernels.
bool encode_kv_map_rows(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                        int64_t tokens, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int elt = kv_dtype == PA_E5M2 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * elt, (cuuint64_t)hkv * d * elt};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elt), 1, (cuuint32_t)rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = kv_dtype == PA_E5M2   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(tm, dt, 3, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                   int64_t tokens) {
  return encode_kv_map_rows(tm, cache, kv_dtype, d, hkv, tokens, 16);
}

// [tokens, Hkv, d] cache viewed as (128-byte piece, token, piece index, head)
// with boxes of (128 bytes, 16 tokens, all d / 128 pieces, 1 head): one copy
// lands a 16-token page slot of one head as [piece][16 keys][128 B], 128-byte
// swizzle -- the layout of a decode ring slot half.
bool encode_slot_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                     int64_t tokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int elt = kv_dtype == PA_E5M2 ? 1 : 2;
  const int per = 128 / elt, pieces = d * elt / 128;
  cuuint64_t dims[4] = {(cuuint64_t)per, (cuuint64_t)tokens, (cuuint64_t)pieces, (cuuint64_t)hkv};
  cuuint64_t strides[3] = {(cuuint64_t)hkv * d * elt, 128, (cuuint64_t)d * elt};
  cuuint32_t box[4] = {(cuuint32_t)per, 16, (cuuint32_t)pieces, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = kv_dtype == PA_E5M2   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(tm, dt, 4, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <typename T>
cudaError_t launch_tc(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap* tkw, const CUtensorMap* tvw, int grid_x, bool kv8,
                      cudaStream_t st) {
  // pages that can hold a whole key tile: the kernels that may copy a unit in
  // one box per chunk
  const bool wide = a.p.page_size >= TcCfg::BN;
  if (kv8) {
    auto k = wide ? prefill_tc8_kernel<T, true> : prefill_tc8_kernel<T, false>;
    static DeviceFlags attr8, attr8w;
    cudaError_t e = (wide ? attr8w : attr8).once([&] {
      return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Tc8Cfg::SMEM);
    });
    if (e != cudaSuccess) return e;
    k<<<dim3((unsigned)grid_x * a.p.hkv), Tc8Cfg::THREADS, Tc8Cfg::SMEM, st>>>(a, tk, tv, *tkw,
                                                                              *tvw);
    return cudaGetLastError();
  }
  auto k = wide ? prefill_tc_kernel<T, false, true> : prefill_tc_kernel<T, false, false>;
  static DeviceFlags attr16, attr16w;
  cudaError_t e = (wide ? attr16w : attr16).once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM);
  });
  if (e != cudaSuccess) return e;
  k<<<dim3((unsigned)grid_x * a.p.hkv), 384, TcCfg::SMEM, st>>>(a, tk, tv, *tkw, *tvw);
  return cudaGetLastError();
}

}  // namespace

namespace {

// The long-row decode splits on the same kernel (one CTA per SM at most; the
// CTAs take the list's (item, KV head) units in turn).
template <typename T>
cudaError_t launch_tc_long(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tkw, const CUtensorMap& tvw, int grid,
                           cudaStream_t st) {
  const bool wide = a.p.page_size >= TcCfg::BN;
  auto k = wide ? prefill_tc_kernel<T, true, true> : prefill_tc_kernel<T, true, false>;
  static DeviceFlags attr, attrw;
  cudaError_t e = (wide ? attrw : attr).once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM);
  });
  if (e != cudaSuccess) return e;
  k<<<dim3((unsigned)grid), 384, TcCfg::SMEM, st>>>(a, tk, tv, tkw, tvw);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_long(const AttnArgs& a, int q_dtype, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  if (a.p.d != 256) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv, tkw, tvw;
  if (!encode_kv_map(&tk, a.kc, q_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, q_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map_rows(&tkw, a.kc, q_dtype, a.p.d, a.p.hkv, tokens, TcCfg::BN) ||
      !encode_kv_map_rows(&tvw, a.vc, q_dtype, a.p.d, a.p.hkv, tokens, TcCfg::HB))
    return cudaErrorInvalidValue;
  return q_dtype == PA_BF16 ? launch_tc_long<__nv_bfloat16>(a, tk, tv, tkw, tvw, grid, st)
                            : launch_tc_long<__half>(a, tk, tv, tkw, tvw, grid, st);
}

bool prefill_tc_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  return (q_dtype == PA_BF16 || q_dtype == PA_F16) && (kv_dtype == q_dtype || kv_dtype == PA_E5M2) &&
         d == 256 && cache_tokens < (int64_t(1) << 31) && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, int q_dtype, int kv_dtype, int grid_x,
                              cudaStream_t st) {
  if (grid_x == 0) return cudaSuccess;
  if (a.p.d != 256) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv, tkw, tvw;
  if (!encode_kv_map(&tk, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens))
    return cudaErrorInvalidValue;
  const bool kv8 = kv_dtype == PA_E5M2;
  // one box per K tile (BN keys) or V half (HB keys): the same in both kernels
  static_assert(TcCfg::BN == Tc8Cfg::BN && TcCfg::HB == Tc8Cfg::HB, "unit sizes");
  if (!encode_kv_map_rows(&tkw, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens, TcCfg::BN) ||
      !encode_kv_map_rows(&tvw, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens, TcCfg::HB))
    return cudaErrorInvalidValue;
  return q_dtype == PA_BF16 ? launch_tc<__nv_bfloat16>(a, tk, tv, &tkw, &tvw, grid_x, kv8, st)
                            : launch_tc<__half>(a, tk, tv, &tkw, &tvw, grid_x, kv8, st);
}

}  // namespace pa
