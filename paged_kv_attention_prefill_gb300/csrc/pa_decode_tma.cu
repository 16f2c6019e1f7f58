// Split-KV paged decode for 16-bit KV caches: persistent warps, each with its
// own TMA ring.
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
//    box per 64 columns of K and of V, straight from the block table into
//    the warp's private ring of NS slots.  The warp keeps NS-1 slots in
//    flight and prefetches across item boundaries, so HBM never waits for a
//    warp to start its next item.
//  * The math per slot is warp-level MMA (m16n8k16): S = Q K^T for the 16
//    rows x 16 keys, the online softmax in registers, O += P V.  At the end
//    of an item the warp writes (acc[d], m, l) of its rows for that split.
//  * No block-wide barrier anywhere: warps only wait on their own mbarriers.
//    All waits are clock-bounded.
//
// The result of an item depends only on its row's data and length, never on
// which warp ran it or when, so the outputs stay bitwise batch-invariant.
#include <cudaTypedefs.h>

#include "pa_sm100.cuh"

namespace pa {
bool encode_kv_map(CUtensorMap* tm, const void* cache, int q_dtype, int d, int hkv,
                   int64_t tokens);

namespace {

using namespace sm100;

constexpr int DEC_WARPS = 4;

template <int D>
struct DecCfg {
  static constexpr int NCH = D / 64;                      // 128-byte column chunks
  static constexpr uint32_t HALF = 16 * D * 2;             // K (or V) of one 16-key slot
  static constexpr uint32_t SLOT = 2 * HALF;
  static constexpr uint32_t QB = 16 * D * 2;               // the item's 16 query rows
  static constexpr int NS = D == 256 ? 3 : (D == 128 ? 6 : 8);  // ring slots per warp
  static constexpr uint32_t WARP_BYTES = NS * SLOT + QB;   // multiple of 1024
  static constexpr uint32_t OFF_BAR = DEC_WARPS * WARP_BYTES;
  static constexpr uint32_t OFF_META = OFF_BAR + DEC_WARPS * NS * 8;
  static constexpr uint32_t SMEM = OFF_META + DEC_WARPS * NS * 8 + 1024;
  static_assert(WARP_BYTES % 1024 == 0, "slot alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t swz_chunked(int row, int col_elem) {
  // 16-bit element column -> byte offset in a [NCH][16 rows][128 B] tile with
  // the 128-byte swizzle (the layout the TMA boxes produce)
  const int chunk = col_elem >> 6, piece = (col_elem & 63) >> 3;
  return (uint32_t)(chunk * 2048 + row * 128 + ((piece ^ (row & 7)) << 4));
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
  f.split = rest % NSPLIT;
  rest /= NSPLIT;
  f.kh = rest % p.hkv;
  f.b = rest / p.hkv;
  f.qs = __ldg(p.cu_q + f.b);
  f.qb = __ldg(p.cu_q + f.b + 1) - f.qs;
  if (f.qb <= 0 || f.qs < 0 || f.qs + f.qb > p.total_q) return false;
  f.slot_base = f.qs;
  if (a.dec_base) {
    f.slot_base = __ldg(a.dec_base + f.b);
    if (f.slot_base < 0) return false;
  }
  if ((int64_t)f.slot_base + f.qb > a.max_slots) return false;
  f.L = __ldg(p.seq_lens + f.b);
  f.M = f.qb * p.g;
  f.r0 = f.mblk * 16;
  if (f.r0 >= f.M) return false;
  const int n_tiles = (f.L + DEC_KT - 1) / DEC_KT;
  const int tps = (n_tiles + NSPLIT - 1) / NSPLIT;
  f.k0 = f.split * tps * DEC_KT;
  if (f.k0 >= f.L) return false;
  f.k1 = min(f.k0 + tps * DEC_KT, f.L);
  f.nchunks = (f.k1 - f.k0 + 15) / 16;
  return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1)
    decode_tma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, int total_items, int n_mblk,
                      uint32_t* counters) {
  using C = DecCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const uint32_t wbase = base + warp * C::WARP_BYTES;   // this warp's slots, then its Q
  const uint32_t sQ = wbase + NS * C::SLOT;
  const uint32_t bar0 = base + C::OFF_BAR + warp * NS * 8;
  int2* meta = reinterpret_cast<int2*>(smem + C::OFF_META) + warp * NS;
  volatile int abort_local = 0;  // per-warp: a timed-out wait ends this warp's work

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncwarp();

  // ---- producer cursor (lane 0 only) --------------------------------------
  int cur_id = -1, cur_chunk = 0;
  Item cur{};
  auto fetch = [&]() {
    // lane 0: next non-empty item, or -1
    for (;;) {
      const int id = (int)atomicAdd(counters, 1u);
      if (id >= total_items) return -1;
      if (item_info(a, id, n_mblk, cur)) return id;
    }
  };
  auto issue = [&](int s) {
    // lane 0: put the cursor's next 16-key slot into ring slot s (or mark end)
    if (cur_id < 0) {
      meta[s] = make_int2(-1, 0);
      return;
    }
    const int s0 = cur.k0 + 16 * cur_chunk;
    const int col = s0 / p.page_size;
    const int page = col < p.max_pages ? __ldg(p.bt + (int64_t)cur.b * p.max_pages + col) : -1;
    const uint32_t bar = bar0 + 8 * s;
    if (page < 0 || page >= p.num_pages) {
      atomicOr(p.err, PA_DEVERR_BAD_PAGE);
      meta[s] = make_int2(cur_id, cur_chunk | (1 << 30));  // consumer zero-fills
      mbar_arrive(bar);
    } else {
      const int tok0 = page * p.page_size + (s0 % p.page_size);
      meta[s] = make_int2(cur_id, cur_chunk);
      mbar_arrive_expect_tx(bar, C::SLOT);
      const uint32_t dK = wbase + s * C::SLOT, dV = dK + C::HALF;
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(dK + c * 2048, &tmK, c * 64, cur.kh, tok0, bar);
        tma_load_3d(dV + c * 2048, &tmV, c * 64, cur.kh, tok0, bar);
      }
    }
    if (++cur_chunk >= cur.nchunks) {
      cur_chunk = 0;
      cur_id = fetch();
    }
  };
  if (lane == 0) {
    cur_id = fetch();
    for (int s = 0; s < NS - 1; ++s) issue(s);
  }
  __syncwarp();

  // ---- consumer ---------------------------------------------------------------
  uint32_t phase = 0;  // bit s: parity of ring slot s
  int it_id = -1;
  Item f{};
  int last[2] = {-1, -1};
  float o[D / 8][4];
  float m_run[2], l_run[2];
  const float sl2 = p.sl2;
  for (int s = 0;; s = (s + 1 == NS ? 0 : s + 1)) {
    // refill the slot consumed by the previous iteration (at the start: the
    // one slot the prologue left empty), NS-1 slots ahead of this one
    if (lane == 0) issue(s == 0 ? NS - 1 : s - 1);
    __syncwarp();
    const int2 mt = meta[s];
    if (mt.x < 0) break;
    if (!mbar_wait(bar0 + 8 * s, (phase >> s) & 1u, &abort_local, p.err)) break;
    phase ^= 1u << s;
    const int chunk = mt.y & 0xFFFF;
    const bool bad = (mt.y >> 30) & 1;
    if (mt.x != it_id) {
      // a new item: its rows' queries into the swizzled Q tile, fresh state
      it_id = mt.x;
      item_info(a, it_id, n_mblk, f);
      for (int e = lane; e < 16 * (D / 8); e += 32) {
        const int r = e / (D / 8), c8 = e % (D / 8);
        const int R = f.r0 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (R < f.M) {
          const T* src = static_cast<const T*>(a.q) +
                         ((int64_t)(f.qs + R / p.g) * p.hq + f.kh * p.g + R % p.g) * D + c8 * 8;
          v = __ldg(reinterpret_cast<const uint4*>(src));
        }
        *reinterpret_cast<uint4*>(smem + (sQ - base) + swz_chunked(r, c8 * 8)) = v;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int R = f.r0 + gid + 8 * h;
        last[h] = R < f.M ? f.L - f.qb + R / p.g : -1;
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    }
    const uint32_t sK = wbase + s * C::SLOT, sV = sK + C::HALF;
    const int kb = f.k0 + 16 * chunk;
    const int nvalid = bad ? 0 : min(16, f.L - kb);
    if (nvalid < 16) {
      // keys past the row's end (or behind a bad table entry): zero their
      // K and V rows so stale or poisoned bytes never reach the products
      for (int e = lane; e < (16 - nvalid) * 2 * (D / 8); e += 32) {
        const int kv = e & 1, rest = e >> 1;
        const int r = nvalid + rest / (D / 8), c8 = rest % (D / 8);
        *reinterpret_cast<uint4*>(smem + ((kv ? sV : sK) - base) + swz_chunked(r, c8 * 8)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncwarp();

    // S = Q K^T: 16 rows x 16 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kd = 0; kd < D / 16; ++kd) {
      uint32_t af[4], b0, b1, b2, b3;
      ldsm_x4(sQ + swz_chunked(lane & 15, kd * 16 + (lane >> 4) * 8), af[0], af[1], af[2],
              af[3]);
      ldsm_x4(sK + swz_chunked((lane & 7) + ((lane >> 4) << 3), kd * 16 + ((lane >> 3) & 1) * 8),
              b0, b1, b2, b3);
      mma16816<T>(sc[0], af, b0, b1);
      mma16816<T>(sc[1], af, b2, b3);
    }
    // mask, online softmax (log2 units)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const int j = kb + n * 8 + 2 * tig + (e & 1);
        const float x = j <= last[h] ? sc[n][e] * sl2 : -INFINITY;
        sc[n][e] = x;
        mx[h] = fmaxf(mx[h], x);
      }
    }
    float alpha[2], m_use[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float m_new = fmaxf(m_run[h], mx[h]);
      m_use[h] = m_new == -INFINITY ? 0.f : m_new;
      alpha[h] = exp2f(m_run[h] - m_use[h]);
      m_run[h] = m_new;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = exp2f(sc[n][e] - m_use[e >> 1]);
        sc[n][e] = pv;
        rs[e >> 1] += pv;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += P V
    uint32_t pf[4];
    pf[0] = pack2<T>(sc[0][0], sc[0][1]);
    pf[1] = pack2<T>(sc[0][2], sc[0][3]);
    pf[2] = pack2<T>(sc[1][0], sc[1][1]);
    pf[3] = pack2<T>(sc[1][2], sc[1][3]);
#pragma unroll
    for (int nd = 0; nd < D / 16; ++nd) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sV + swz_chunked((lane & 7) + (((lane >> 3) & 1) << 3), nd * 16 + (lane >> 4) * 8),
                b0, b1, b2, b3);
      mma16816<T>(o[2 * nd], pf, b0, b1);
      mma16816<T>(o[2 * nd + 1], pf, b2, b3);
    }

    if (chunk == f.nchunks - 1) {
      // item done: this split's partial state of the block's rows
      float lt[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        lt[h] = l_run[h] + __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], 2);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int R = f.r0 + gid + 8 * h;
        if (R >= f.M) continue;
        const int64_t slot = f.slot_base + R / p.g;
        const int64_t ps = (slot * p.hq + f.kh * p.g + R % p.g) * NSPLIT + f.split;
        float* acc = a.part_acc + ps * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2*>(acc + n * 8 + 2 * tig) = make_float2(o[n][2 * h], o[n][2 * h + 1]);
        if (tig == 0) a.part_ml[ps] = make_float2(m_run[h], lt[h]);
      }
    }
    // the slot is consumed; the next iteration refills it with TMA (async
    // writes after this warp's generic reads and zero-fills)
    fence_proxy_async_smem();
    __syncwarp();
  }

  // a timed-out warp still has copies landing: let them finish before exit
  if (abort_local) {
    for (int s = 0; s < NS; ++s)
      if (meta[s].x >= 0) mbar_drain(bar0 + 8 * s, (phase >> s) & 1u, p.err);
  }
  __syncwarp();
  // the last warp of the grid resets the item counter for the next call
  if (lane == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(counters + 1, 1u);
    if (done == gridDim.x * DEC_WARPS - 1) {
      counters[0] = 0u;
      counters[1] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

bool decode_tma_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  return (q_dtype == PA_BF16 || q_dtype == PA_F16) && kv_dtype == q_dtype &&
         (d == 64 || d == 128 || d == 256) && cache_tokens < (int64_t(1) << 31);
}

template <typename T, int D>
static cudaError_t launch_dec(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                              int total_items, int n_mblk, uint32_t* counters, cudaStream_t st) {
  using C = DecCfg<D>;
  auto k = decode_tma_kernel<T, D>;
  static DeviceFlags attr;
  cudaError_t e = attr.once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int grid = sms > 0 ? sms : 148;  // persistent: one CTA per SM
  if (total_items < grid * DEC_WARPS) grid = (total_items + DEC_WARPS - 1) / DEC_WARPS;
  if (grid < 1) grid = 1;
  k<<<grid, DEC_WARPS * 32, C::SMEM, st>>>(a, tk, tv, total_items, n_mblk, counters);
  return cudaGetLastError();
}

cudaError_t launch_decode_tma(const AttnArgs& a, int q_dtype, int n_mblk, cudaStream_t st) {
  if (a.p.num_rows == 0 || n_mblk == 0) return cudaSuccess;
  const int64_t items = (int64_t)a.p.num_rows * a.p.hkv * NSPLIT * n_mblk;
  if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, a.kc, q_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, q_dtype, a.p.d, a.p.hkv, tokens))
    return cudaErrorInvalidValue;
  uint32_t* counters = reinterpret_cast<WsHeader*>(a.p.err)->pad;
  const bool bf = q_dtype == PA_BF16;
  switch (a.p.d) {
    case 64: return bf ? launch_dec<__nv_bfloat16, 64>(a, tk, tv, (int)items, n_mblk, counters, st)
                       : launch_dec<__half, 64>(a, tk, tv, (int)items, n_mblk, counters, st);
    case 128: return bf ? launch_dec<__nv_bfloat16, 128>(a, tk, tv, (int)items, n_mblk, counters, st)
                        : launch_dec<__half, 128>(a, tk, tv, (int)items, n_mblk, counters, st);
    case 256: return bf ? launch_dec<__nv_bfloat16, 256>(a, tk, tv, (int)items, n_mblk, counters, st)
                        : launch_dec<__half, 256>(a, tk, tv, (int)items, n_mblk, counters, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
