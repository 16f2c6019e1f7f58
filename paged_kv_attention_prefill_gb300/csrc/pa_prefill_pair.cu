// Varlen causal paged prefill on CTA pairs (head dim 128, 16-bit caches).
//
// The same attention as every other path of the library (packed varlen
// batch, one block table per row, bottom-right causal alignment, GQA, online
// softmax over key tiles: vllm-rlt PR #128, "Purpose", prefill bullets),
// laid out for two SMs working on one 256-row block:
//
//  * A cluster of two CTAs owns 256 GQA-packed query rows of one (row, KV
//    head) -- the query heads that share the KV head stacked along M
//    (1Cat-vLLM PR #1279, commit 1) -- each CTA 128 of them, one per TMEM
//    lane.  The products are tcgen05 MMAs of M = 256 issued by one thread of
//    rank 0 for both SMs: S = Q K^T with Q in TMEM (A split by rows between
//    the CTAs) and each CTA holding half of the K tile's keys (B split along
//    N), then O += P V with P in TMEM and each CTA holding half of the V
//    tile's head-dim columns.  So each SM keeps only half of every K/V tile
//    in shared memory: six stages of each ring fit, three times what one SM
//    holding whole tiles for 256 rows can keep in flight.
//  * TMEM per CTA: two S buffers of 128 key columns (P written over the
//    first half of its buffer), O (128 columns) and Q (64 columns of 16-bit
//    pairs).  S(j + 2) goes into tile j's buffer once O += P(j) V is done,
//    so the S product of the next tile runs during the softmax of this one.
//  * Warp 0 streams this CTA's half of each K tile and warp 2 its half of
//    each V tile, one TMA box per 16-token page slot straight from the block
//    table (1Cat-vLLM PR #616, original description: any page size that is a
//    multiple of 16); the slot with the row's last key is copied by hand with
//    the keys past the end zero-filled.  In rank 1, warp 1 relays each
//    stage's arrival to rank 0's barrier, where the MMA thread waits for
//    both halves.
//  * Warpgroups 1 and 2 take alternate key tiles (each thread one query row
//    over all 128 keys).  The row's exponent reference is handed from one
//    warpgroup to the other through shared memory as soon as a tile's
//    maximum is known, so the exponentials of tile j run while the other
//    warpgroup starts on tile j + 1; the reference moves only when a row's
//    maximum passes it by more than 2^8 (then O is rescaled in TMEM after
//    the previous product).  Each warpgroup keeps the row sum of its own
//    tiles; the two are added at the end.
//
// Every wait is bounded; a CTA whose wait runs out raises the workspace
// flag and the other CTA's abort flag, drains what it started, and both
// reach the final cluster barrier before TMEM is freed.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_sm100.cuh"

namespace pa {
bool encode_kv_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                   int64_t tokens);

namespace {

using namespace sm100;

// Registers per thread at launch (384 threads, one CTA per SM) and after the
// split between the producer / MMA warpgroup and the two softmax warpgroups.
constexpr int PR_REG_LAUNCH = 168;
constexpr int PR_REG_LOW = 72, PR_REG_HIGH = 216;
static_assert(128 * PR_REG_LOW + 256 * PR_REG_HIGH <= 384 * PR_REG_LAUNCH, "register split");

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int BM = 128;                   // rows per CTA = TMEM lanes (256 per pair)
  static constexpr int BN = 128;                   // keys per tile
  static constexpr int HK = BN / 2;                // keys of a K tile held by each CTA
  static constexpr int HD = D / 2;                 // head-dim columns of a V tile per CTA
  static constexpr int KS = 6, VS = 6;             // ring stages
  static constexpr uint32_t K_BYTES = HK * D * 2;  // [2 chunks of 64 d][64 keys][128 B]
  static constexpr uint32_t V_BYTES = BN * HD * 2; // [128 keys][128 B] (64 d columns)
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KS * K_BYTES;
  static constexpr uint32_t OFF_M = OFF_V + VS * V_BYTES;  // [2][128] floats: row references
  static constexpr uint32_t OFF_L = OFF_M + 2 * BM * 4;    // [2][128] floats: final row sums
  static constexpr uint32_t OFF_BAR = OFF_L + 2 * BM * 4;
  static constexpr uint32_t BAR_AREA = 320;        // mbarriers, then TMEM address and flags
  static constexpr uint32_t SMEM = OFF_BAR + BAR_AREA + 16 + 1024;  // alignment slack
  static constexpr uint32_t S_COL = 0;             // S buffers [0, BN) and [BN, 2 BN)
  static constexpr uint32_t O_COL = 2 * BN;
  static constexpr uint32_t Q_COL = O_COL + D;
  static constexpr uint32_t TMEM_COLS = 512;
  // barrier indices
  static constexpr int B_KF = 0, B_KE = KS, B_VF = 2 * KS, B_VE = 2 * KS + VS,
                       B_SF = 2 * KS + 2 * VS,     // [2] S in buffer b written (commit)
      B_PF = B_SF + 2,                             // [2][2] P(j) half h published, j % 2 (rank 0: 8 warps)
      B_OD = B_PF + 4,                             // [2] O += P(j) V done, j % 2 (commit)
      B_Q = B_OD + 2,                              // Q in TMEM (rank 0: 8 warps)
      B_MH = B_Q + 1,                              // [2] row reference after tile j, j % 2
      B_DRAIN = B_MH + 2, NBAR = B_DRAIN + 1;
  static_assert(Q_COL + D / 2 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NBAR * 8 <= BAR_AREA, "barrier area");
};

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    prefill_pair_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  using C = PairCfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V;
  volatile float* mref = reinterpret_cast<volatile float*>(smem + C::OFF_M);
  volatile float* lsum = reinterpret_cast<volatile float*>(smem + C::OFF_L);
  const uint32_t bar0 = base + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::BAR_AREA);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::BAR_AREA + 4);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  // the other CTA's abort flag, and rank 0's barriers, as cluster addresses
  const uint32_t peer_abort = mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u);
  auto lead_bar = [&](int i) { return mapa_shared(bar(i), 0); };

  // ---- work item (uniform over the pair) --------------------------------------
  // 1-D grid of pairs, KV head fastest: the work list is longest-first
  const int pair_id = blockIdx.x >> 1;
  const int item = pair_id / p.hkv, kh = pair_id % p.hkv;
  if (item >= (int)*a.n_tiles) return;
  const int2 wi = a.tiles[item];
  const int b = wi.x, mb = wi.y & 0xFFFFFF, part = wi.y >> 24;
  const int qs = __ldg(p.cu_q + b);
  const int qb = __ldg(p.cu_q + b + 1) - qs;
  const int L = __ldg(p.seq_lens + b);
  if (qb <= 0) return;
  if (qs < 0 || qs + qb > p.total_q) {
    if (threadIdx.x == 0 && leader) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return;
  }
  const int g = p.g, M = qb * g, R0 = mb * 2 * C::BM;
  if (R0 >= M) return;
  // keys any row of the 256-row block sees, and the item's part of them
  const int k_item = min(L, L - qb + (min(R0 + 2 * C::BM, M) - 1) / g + 1);
  int per_u;
  const bool cut = pf_part_count(k_item, a.pf_parts, a.pf_min_units, &per_u) > 1;
  const int k0 = cut ? part * per_u * PF_UNIT : 0;
  const int k1 = cut ? min(k_item, (part + 1) * per_u * PF_UNIT) : k_item;
  const int n = k1 > k0 ? (k1 - k0 + C::BN - 1) / C::BN : 0;

  // ---- barriers and TMEM ----------------------------------------------------
  if (threadIdx.x == 0) {
    // rank 0's full barriers also take the relayed arrival of rank 1's half
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_KF + s), leader ? 2 : 1);
      mbar_init(bar(C::B_KE + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_VF + s), leader ? 2 : 1);
      mbar_init(bar(C::B_VE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SF + t), 1);
      mbar_init(bar(C::B_PF + t), 8);
      mbar_init(bar(C::B_PF + 2 + t), 8);
      mbar_init(bar(C::B_OD + t), 1);
      mbar_init(bar(C::B_MH + t), 4);
    }
    mbar_init(bar(C::B_Q), 8);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers exist before any arrival crosses the pair
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    setmaxnreg_dec<PR_REG_LOW>();
    if (warp == 0 || warp == 2) {
      // ======= producers: warp 0 this CTA's half of each K tile (keys
      // [64 rank, +64) of it), warp 2 its half of each V tile (head-dim
      // columns [64 rank, +64)) =============================================
      const bool isK = warp == 0;
      const int NS = isK ? C::KS : C::VS;
      const uint32_t UB = isK ? C::K_BYTES : C::V_BYTES;
      const int B_FULL = isK ? C::B_KF : C::B_VF, B_EMPTY = isK ? C::B_KE : C::B_VE;
      const uint32_t ring = isK ? sK : sV;
      const void* tmap = isK ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmV);
      const T* cache = static_cast<const T*>(isK ? a.kc : a.vc);
      const int nslot = isK ? C::HK / 16 : C::BN / 16;  // page slots per unit
      const int NCH = isK ? 2 : 1;                      // 64-element chunks per key row
      const int col0 = isK ? 0 : C::HD * (int)rank;     // first head-dim column copied
      if (lane == 0) tma_prefetch_desc(tmap);
      const int P = p.page_size;
      const int64_t bt_row = (int64_t)b * p.max_pages;
      int u = 0;
      bool ok = true;
      for (; u < n; ++u) {
        const int st = u % NS;
        if (u >= NS)
          ok = mbar_wait_cl(bar(B_EMPTY + st), ((u / NS) - 1) & 1, abort_flag, peer_abort, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const int kbase = k0 + u * C::BN + (isK ? C::HK * (int)rank : 0);
        const uint32_t dst = ring + st * UB;
        // slot `lane`: 1 = whole slot by TMA, 2 = partial (copied by hand), 3 = zero-fill
        int kind = 0, tok0 = 0;
        if (lane < nslot) {
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
        uint32_t manual = __ballot_sync(0xffffffffu, kind >= 2);
        while (manual) {
          const int s = __ffs(manual) - 1;
          manual &= manual - 1;
          const int ks = __shfl_sync(0xffffffffu, kind, s);
          const int t0 = __shfl_sync(0xffffffffu, tok0, s);
          const int nvalid = ks == 2 ? L - (kbase + 16 * s) : 0;
          for (int it = lane; it < 16 * NCH * 8; it += 32) {
            const int piece = it & 7, rest = it >> 3;
            const int c = rest % NCH, rr = rest / NCH;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < nvalid) {
              const T* src =
                  cache + ((int64_t)(t0 + rr) * p.hkv + kh) * D + col0 + c * 64 + piece * 8;
              v = __ldg(reinterpret_cast<const uint4*>(src));
            }
            const int row = 16 * s + rr;
            const uint32_t rows = isK ? C::HK : C::BN;
            st_shared_v4(dst + c * (rows * 128) + row * 128 + ((piece ^ (row & 7)) << 4), v);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int n_tma = __popc(__ballot_sync(0xffffffffu, kind == 1));
        if (lane == 0)
          mbar_arrive_expect_tx(bar(B_FULL + st), (uint32_t)(n_tma * 16 * NCH * 128));
        __syncwarp();
        if (kind == 1) {
          const uint32_t rows = isK ? C::HK : C::BN;
          for (int c = 0; c < NCH; ++c)
            tma_load_3d(dst + c * (rows * 128) + lane * 16 * 128, tmap, col0 + c * 64, kh, tok0,
                        bar(B_FULL + st));
        }
      }
      if (!ok) {
        // copies this warp started may still be landing: wait for them
        for (int uu = max(0, u - NS); uu < u; ++uu)
          mbar_drain(bar(B_FULL + uu % NS), (uu / NS) & 1, p.err);
      } else {
        // the releases of the last stages (rank 0's commits arrive in both
        // CTAs): every arrival has landed before the CTA can leave
        for (int uu = max(0, n - NS); uu < n; ++uu)
          mbar_wait_cl(bar(B_EMPTY + uu % NS), (uu / NS) & 1, abort_flag, peer_abort, p.err);
      }
    } else if (warp == 1 && !leader) {
      // ============== rank 1: relay each stage's arrival to rank 0 ============
      if (lane == 0) {
        for (int u = 0; u < n; ++u) {
          if (!mbar_wait_cl(bar(C::B_KF + u % C::KS), (u / C::KS) & 1, abort_flag, peer_abort,
                            p.err))
            break;
          mbar_arrive_cluster(lead_bar(C::B_KF + u % C::KS));
          if (!mbar_wait_cl(bar(C::B_VF + u % C::VS), (u / C::VS) & 1, abort_flag, peer_abort,
                            p.err))
            break;
          mbar_arrive_cluster(lead_bar(C::B_VF + u % C::VS));
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ===================== rank 0: MMA issuer (one thread) ====================
      //   S(0), S(1), then per key tile j: O += P(j) V in two 64-key halves
      //   (each once that half of P(j) is published by both CTAs), then
      //   S(j + 2) into tile j's buffer once that product is done.
      if (lane == 0) {
        constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
        constexpr uint32_t idS = idesc_f16(fmt, 256, C::BN, false);
        constexpr uint32_t idO = idesc_f16(fmt, 256, D, true);
        auto issue_S = [&](int j) {
          const int st = j % C::KS;
          if (!mbar_wait_cl(bar(C::B_KF + st), (j / C::KS) & 1, abort_flag, peer_abort, p.err))
            return false;
          tc_fence_after();
          const uint64_t b0 = sdesc_sw128(sK + st * C::K_BYTES, 16, 1024);
          const uint32_t sd = tmem + C::S_COL + (uint32_t)(j & 1) * C::BN;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t bd = b0 + (uint64_t)(((k >> 2) * (C::HK * 128) + (k & 3) * 32) >> 4);
            tc_mma_pair_ts(sd, tmem + C::Q_COL + 8 * k, bd, idS, k > 0 ? 1u : 0u);
          }
          tc_commit_pair(bar(C::B_SF + (j & 1)));
          tc_commit_pair(bar(C::B_KE + st));
          return true;
        };
        auto issue_PV = [&](int j) {
          const int sv = j % C::VS;
          if (!mbar_wait_cl(bar(C::B_VF + sv), (j / C::VS) & 1, abort_flag, peer_abort, p.err))
            return false;
          const uint64_t b0 = sdesc_sw128(sV + sv * C::V_BYTES, C::BN * 128, 1024);
          const uint32_t pa = tmem + C::S_COL + (uint32_t)(j & 1) * C::BN;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait_cl(bar(C::B_PF + 2 * (j & 1) + h), (j >> 1) & 1, abort_flag, peer_abort,
                              p.err))
              return false;
            tc_fence_after();
#pragma unroll
            for (int k = 4 * h; k < 4 * h + 4; ++k) {
              // A = P from TMEM: 16 keys = 8 columns of 16-bit pairs
              const uint64_t bd = b0 + (uint64_t)((k * 16 * 128) >> 4);
              tc_mma_pair_ts(tmem + C::O_COL, pa + 8 * k, bd, idO, (j > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit_pair(bar(C::B_VE + sv));
          tc_commit_pair(bar(C::B_OD + (j & 1)));
          return true;
        };
        bool ok = n == 0 || mbar_wait_cl(bar(C::B_Q), 0, abort_flag, peer_abort, p.err);
        if (ok) tc_fence_after();
        if (ok && n > 0) ok = issue_S(0);
        if (ok && n > 1) ok = issue_S(1);
        for (int j = 0; ok && j < n; ++j) {
          ok = issue_PV(j);
          if (ok && j + 2 < n) {
            // tile j's S buffer holds P(j) until this product is done
            ok = mbar_wait_cl(bar(C::B_OD + (j & 1)), (j >> 1) & 1, abort_flag, peer_abort, p.err);
            if (ok) {
              tc_fence_after();
              ok = issue_S(j + 2);
            }
          }
        }
        // nothing this thread issued may still run once TMEM is freed
        tc_commit_pair_self(bar(C::B_DRAIN));
        mbar_drain(bar(C::B_DRAIN), 0, p.err);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<PR_REG_HIGH>();
    // ============ softmax of alternate key tiles, epilogue ====================
    // Warpgroup w (warps 4-7: w = 0, warps 8-11: w = 1) takes tiles j = w,
    // w + 2, ...; thread = one query row = one TMEM lane.  The loop never
    // leaves early: after a timed-out wait it runs on (waits return at once),
    // so every warp reaches the final barriers.
    const int w = (warp >> 2) - 1;
    const int q4 = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;     // row of the CTA's tile == TMEM lane
    const int R = R0 + (int)rank * C::BM + r;
    const bool valid = R < M;
    const int i = valid ? R / g : 0, hg = valid ? R % g : 0;
    // last visible key of this row, counted from the start of the key range
    const int last = valid ? min(L - qb + i, k1 - 1) - k0 : -1 - k0;
    const int64_t qoff = ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t pf_bar0 = leader ? bar(C::B_PF) : lead_bar(C::B_PF);
    if (w == 0 && n > 0) {
      // this row's Q into TMEM (16-bit pairs), then published to rank 0
      const T* qrow = static_cast<const T*>(a.q) + qoff;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8) {
          const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(qrow + c * 64 + u8 * 8))
                                : make_uint4(0u, 0u, 0u, 0u);
          v[4 * u8] = u.x;
          v[4 * u8 + 1] = u.y;
          v[4 * u8 + 2] = u.z;
          v[4 * u8 + 3] = u.w;
        }
        tmem_st_x32(trow + C::Q_COL + c * 32, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar(C::B_Q));
        else
          mbar_arrive_cluster(lead_bar(C::B_Q));
      }
    }
    const float sl2 = p.sl2;
    float m_w = -INFINITY, l_w = 0.f;  // this warpgroup's reference and row sum
    for (int j = w; j < n; j += 2) {
      const uint32_t buf = (uint32_t)(j & 1) * C::BN;
      mbar_wait_cl(bar(C::B_SF + (j & 1)), (j >> 1) & 1, abort_flag, peer_abort, p.err);
      tc_fence_after();
      float x[C::BN];
      float mt;  // max raw logit of the row in this tile (masked keys -> -inf)
      {
        uint32_t u[C::BN];
        mt = tmem_ld_red_max_x128(trow + C::S_COL + buf, u);
#pragma unroll
        for (int k = 0; k < C::BN; ++k) x[k] = __uint_as_float(u[k]);
      }
      const int kb = j * C::BN;
      if (kb + C::BN - 1 > last) {
#pragma unroll
        for (int k = 0; k < C::BN; ++k)
          if (kb + k > last) x[k] = -INFINITY;
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = x[u];
#pragma unroll
        for (int k = 8; k < C::BN; ++k) pm[k & 7] = fmaxf(pm[k & 7], x[k]);
        mt = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      }
      // the row's reference after tile j - 1 (from the other warpgroup)
      float m_in = -INFINITY;
      if (j > 0) {
        mbar_wait(bar(C::B_MH + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, p.err);
        m_in = mref[((j - 1) & 1) * C::BM + r];
      }
      // this warpgroup's row sum follows the reference
      if (m_in != m_w) {
        l_w = m_w == -INFINITY ? 0.f : l_w * ex2(m_w - m_in);
        m_w = m_in;
      }
      const float m_new = fmaxf(m_in, mt * sl2);  // sl2 > 0: max commutes with the scale
      float factor = 1.f;
      bool need = false;
      float ref = m_in;
      if (j == 0) {
        ref = m_new;
      } else if (m_new > m_in + 8.f) {
        need = true;
        factor = ex2(m_in - m_new);
        ref = m_new;
      }
      // hand the reference on to the other warpgroup before the exponentials
      mref[(j & 1) * C::BM + r] = ref;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_MH + (j & 1)));
      l_w *= factor;
      m_w = ref;
      const float nmu = ref == -INFINITY ? 0.f : -ref;
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // partial row sums, fixed order
#pragma unroll
      for (int k = 0; k < C::BN; ++k) {
        x[k] = ex2(fmaf(x[k], sl2, nmu));
        ps[k & 7] += x[k];
      }
      // O += P(j - 1) V must be done before O is rescaled
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        mbar_wait_cl(bar(C::B_OD + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, peer_abort,
                     p.err);
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st_x32(trow + C::O_COL + c * 32, o);
        }
      }
      // P (16-bit pairs) over the first BN / 2 columns of the tile's S
      // buffer, in two halves of 64 keys, each published to rank 0
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack2<T>(x[64 * h + 2 * k], x[64 * h + 2 * k + 1]);
        tmem_st_x32_nowait(trow + C::S_COL + buf + 32 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(pf_bar0 + 8u * (2 * (j & 1) + h));
          else
            mbar_arrive_cluster(pf_bar0 + 8u * (2 * (j & 1) + h));
        }
      }
      l_w += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
    }
    // ---- epilogue: out = O / l * v_scale, or this part's (O, m, l) ----
    // the final reference, both warpgroups' row sums brought to it and added
    // in warpgroup order
    float m_fin = -INFINITY;
    if (n > 0) {
      mbar_wait(bar(C::B_MH + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag, p.err);
      m_fin = mref[((n - 1) & 1) * C::BM + r];
    }
    if (m_w != m_fin) l_w = m_w == -INFINITY ? 0.f : l_w * ex2(m_w - m_fin);
    lsum[w * C::BM + r] = l_w;
    named_bar_sync(1, 256);
    const float lt = lsum[r] + lsum[C::BM + r];
    if (n > 0) {
      mbar_wait_cl(bar(C::B_OD + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag, peer_abort,
                   p.err);
      tc_fence_after();
    }
    // this warpgroup's half of the head-dim columns
    const int c0 = w * (D / 2);
    T* orow = static_cast<T*>(a.out) + qoff + c0;
    if (cut) {
      const int64_t slot = ((int64_t)(qs + i) * p.hq + kh * g + hg) * a.pf_parts + part;
      if (valid && w == 0)
        a.pf_ml[slot] = make_float2(n > 0 ? m_fin : -INFINITY, n > 0 ? lt : 0.f);
      float* prow = a.pf_acc + slot * D + c0;
      if (n > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          tmem_ld_x32(trow + C::O_COL + c0 + c * 32, o);
          if (valid) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *reinterpret_cast<uint4*>(prow + c * 32 + 4 * e) =
                  make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
      }
    } else if (n > 0) {
      const float inv = lt > 0.f ? p.v_scale / lt : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld_x32(trow + C::O_COL + c0 + c * 32, o);
        if (valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack2<T>(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            v.y = pack2<T>(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            v.z = pack2<T>(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            v.w = pack2<T>(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * e) = v;
          }
        }
      }
    } else if (valid) {
      // no key visible to any row of the block
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        *reinterpret_cast<uint4*>(orow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA frees TMEM or leaves while the pair's MMAs or arrivals may
  // still touch the other
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <typename T>
cudaError_t launch_pair(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        int grid_x, cudaStream_t st) {
  auto k = prefill_pair_kernel<T>;
  static DeviceFlags attr;
  cudaError_t e = attr.once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM);
  });
  if (e != cudaSuccess) return e;
  k<<<dim3(2u * (unsigned)grid_x * a.p.hkv), 384, PairCfg::SMEM, st>>>(a, tk, tv);
  return cudaGetLastError();
}

template <typename T>
bool pair_regs_ok() {
  // the register split is only safe when the kernel launches with exactly
  // PR_REG_LAUNCH registers per thread
  static int ok = -1;
  if (ok < 0) {
    cudaFuncAttributes fa{};
    ok = cudaFuncGetAttributes(&fa, prefill_pair_kernel<T>) == cudaSuccess &&
         fa.numRegs == PR_REG_LAUNCH;
  }
  return ok == 1;
}

}  // namespace

bool prefill_pair_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16) || kv_dtype != q_dtype || d != 128 ||
      cache_tokens >= (int64_t(1) << 31))
    return false;
  return q_dtype == PA_BF16 ? pair_regs_ok<__nv_bfloat16>() : pair_regs_ok<__half>();
}

cudaError_t launch_prefill_pair(const AttnArgs& a, int q_dtype, int grid_x, cudaStream_t st) {
  if (grid_x == 0) return cudaSuccess;
  if (a.p.d != 128) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, a.kc, q_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, q_dtype, a.p.d, a.p.hkv, tokens))
    return cudaErrorInvalidValue;
  return q_dtype == PA_BF16 ? launch_pair<__nv_bfloat16>(a, tk, tv, grid_x, st)
                            : launch_pair<__half>(a, tk, tv, grid_x, st);
}

}  // namespace pa
