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
//    box per 128 bytes of a key row, for K and for V, straight from the
//    block table into the warp's private ring of NS slots.  The warp keeps
//    NS-1 slots in flight and prefetches across item boundaries, so HBM
//    never waits for a warp to start its next item.
//  * The math per slot is warp-level MMA (m16n8k16): S = Q K^T for the 16
//    rows x 16 keys, the online softmax in registers, O += P V.  At the end
//    of an item the warp writes (acc[d], m, l) of its rows for that split.
//  * fp8 E5M2 caches (1Cat-vLLM PR #616, original description: an fp8_e5m2
//    KV cache dequantized in the kernel): an E5M2 code in the high byte of a
//    16-bit word is the same binary16 value, so K is widened straight from
//    the raw slot into MMA operands -- four consecutive codes of one key
//    become two fp16 pairs, and Q's reduction index is permuted the same way
//    so the dot product is unchanged -- while V is widened once per slot
//    into a 16-bit staging tile for the transposed fragment loads.  The
//    per-tensor k_scale is folded into the logit scale, v_scale into the
//    merge.
//  * No block-wide barrier anywhere: warps only wait on their own mbarriers.
//    All waits are clock-bounded.
//
// The result of an item depends only on its row's data and length, never on
// which warp ran it or when, so the outputs stay bitwise batch-invariant.
#include <cudaTypedefs.h>

#include "pa_sm100.cuh"

namespace pa {
bool encode_kv_map(CUtensorMap* tm, const void* cache, int kv_dtype, int d, int hkv,
                   int64_t tokens);

namespace {

using namespace sm100;

constexpr int DEC_WARPS = 4;

template <int D, bool KV8>
struct DecCfg {
  static constexpr int ELT = KV8 ? 1 : 2;
  static constexpr int NCH = D * ELT / 128;                // 128-byte boxes per key row
  static constexpr uint32_t HALF = 16 * D * ELT;           // K (or V) of one 16-key slot
  static constexpr uint32_t SLOT = 2 * HALF;
  static constexpr int NS = KV8 ? (D == 256 ? 5 : 8) : (D == 256 ? 3 : (D == 128 ? 6 : 8));
  static constexpr uint32_t STG = KV8 ? 16 * D * 2 : 0;    // widened V of one slot
  static constexpr uint32_t QB = 16 * D * 2;
  static constexpr uint32_t AUX = STG + QB;
  static constexpr uint32_t OFF_AUX = DEC_WARPS * NS * SLOT;  // all rings first (1 KB aligned)
  static constexpr uint32_t OFF_BAR = OFF_AUX + DEC_WARPS * AUX;
  static constexpr uint32_t OFF_META = OFF_BAR + DEC_WARPS * NS * 8;
  static constexpr uint32_t SMEM = OFF_META + DEC_WARPS * NS * 8 + 1024;
  static_assert(SLOT % 1024 == 0, "slot alignment");
  static_assert(AUX % 16 == 0, "aux alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// 16-bit element (row, col) -> byte offset in a [D/64][16 rows][128 B] tile
// with the 128-byte swizzle (the layout the TMA boxes produce).
__device__ __forceinline__ uint32_t swz16(int row, int col) {
  const int chunk = col >> 6, piece = (col & 63) >> 3;
  return (uint32_t)(chunk * 2048 + row * 128 + ((piece ^ (row & 7)) << 4));
}
// Q tile of the fp8 path: rows of D 16-bit values, 8-byte units XOR-swizzled
// by row so the permuted 64-bit operand loads of 16 lanes hit 32 banks.
template <int D>
__device__ __forceinline__ uint32_t qswz8(int row, int col) {
  const int unit = (col >> 2) ^ ((row & 7) << 2);
  return (uint32_t)(row * D * 2 + unit * 8 + (col & 3) * 2);
}
// fp8 byte (row, col) -> byte offset in a [D/128][16 rows][128 B] tile, same swizzle.
__device__ __forceinline__ uint32_t swz8(int row, int col) {
  const int chunk = col >> 7, piece = (col & 127) >> 4;
  return (uint32_t)(chunk * 2048 + row * 128 + ((piece ^ (row & 7)) << 4) + (col & 15));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
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

template <typename T, bool KV8, int D>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1)
    decode_tma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, int total_items, int n_mblk,
                      uint32_t* counters) {
  using C = DecCfg<D, KV8>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const Problem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const uint32_t wring = base + warp * NS * C::SLOT;       // this warp's slots
  const uint32_t sStg = base + C::OFF_AUX + warp * C::AUX; // fp8: widened V
  const uint32_t sQ = sStg + C::STG;                       // the item's 16 query rows
  const uint32_t bar0 = base + C::OFF_BAR + warp * NS * 8;
  int2* meta = reinterpret_cast<int2*>(smem + C::OFF_META) + warp * NS;
  volatile int abort_local = 0;  // a timed-out wait ends this warp's work

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
    // next non-empty item, or -1
    for (;;) {
      const int id = (int)atomicAdd(counters, 1u);
      if (id >= total_items) return -1;
      if (item_info(a, id, n_mblk, cur)) return id;
    }
  };
  auto issue = [&](int s) {
    // the cursor's next 16-key slot into ring slot s (or mark the end)
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
      meta[s] = make_int2(cur_id, cur_chunk | (1 << 30));  // the consumer zero-fills
      mbar_arrive(bar);
    } else {
      const int tok0 = page * p.page_size + (s0 % p.page_size);
      meta[s] = make_int2(cur_id, cur_chunk);
      mbar_arrive_expect_tx(bar, C::SLOT);
      const uint32_t dK = wring + s * C::SLOT, dV = dK + C::HALF;
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(dK + c * 2048, &tmK, c * (128 / C::ELT), cur.kh, tok0, bar);
        tma_load_3d(dV + c * 2048, &tmV, c * (128 / C::ELT), cur.kh, tok0, bar);
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

  // ---- consumer -------------------------------------------------------------
  uint32_t phase = 0;  // bit s: parity of ring slot s
  int it_id = -1;
  Item f{};
  int last[2] = {-1, -1};
  float o[D / 8][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
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
      // a new item: its rows' queries into the Q tile, fresh state
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
        st_shared_v4(sQ + (KV8 ? qswz8<D>(r, c8 * 8) : swz16(r, c8 * 8)), v);
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
    const uint32_t sK = wring + s * C::SLOT, sV = sK + C::HALF;
    const int kb = f.k0 + 16 * chunk;
    const int nvalid = bad ? 0 : min(16, f.L - kb);
    if (nvalid < 16) {
      // keys past the row's end (or behind a bad table entry): zero their
      // K and V rows so stale or poisoned bytes never reach the products
      constexpr int PIECES = D * C::ELT / 16;  // 16-byte pieces per key row
      for (int e = lane; e < (16 - nvalid) * 2 * PIECES; e += 32) {
        const int kv = e & 1, rest = e >> 1;
        const int r = nvalid + rest / PIECES, pc = rest % PIECES;
        const uint32_t off = KV8 ? swz8(r, pc * 16) : swz16(r, pc * 8);
        st_shared_v4((kv ? sV : sK) + off, make_uint4(0u, 0u, 0u, 0u));
      }
    }
    __syncwarp();
    uint32_t sVf = sV;  // 16-bit V tile the PV fragments come from
    if (KV8) {
      // widen this slot's V codes into the 16-bit staging tile
      for (int e = lane; e < 16 * (D / 16); e += 32) {
        const int r = e & 15, pc = e >> 4;  // 8 lanes of a quarter-warp: 8 rows, one piece
        const uint4 w = ld_shared_v4(sV + swz8(r, pc * 16));
        uint4 lo, hi;
        e5m2x4_to<T>(w.x, lo.x, lo.y);
        e5m2x4_to<T>(w.y, lo.z, lo.w);
        e5m2x4_to<T>(w.z, hi.x, hi.y);
        e5m2x4_to<T>(w.w, hi.z, hi.w);
        st_shared_v4(sStg + swz16(r, pc * 16), lo);
        st_shared_v4(sStg + swz16(r, pc * 16 + 8), hi);
      }
      __syncwarp();
      sVf = sStg;
    }

    // S = Q K^T: 16 rows x 16 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kd = 0; kd < D / 16; ++kd) {
      uint32_t af[4], b0, b1, b2, b3;
      if (KV8) {
        // reduction index permuted within each 16-wide step: operand slots
        // (2t, 2t+1 | 2t+8, 2t+9) hold head-dim columns 4t .. 4t+3
        const uint2 q0 = ld_shared_v2(sQ + qswz8<D>(gid, kd * 16 + 4 * tig));
        const uint2 q1 = ld_shared_v2(sQ + qswz8<D>(gid + 8, kd * 16 + 4 * tig));
        af[0] = q0.x;
        af[1] = q1.x;
        af[2] = q0.y;
        af[3] = q1.y;
        e5m2x4_to<T>(ld_shared_u32(sK + swz8(gid, kd * 16 + 4 * tig)), b0, b1);
        e5m2x4_to<T>(ld_shared_u32(sK + swz8(gid + 8, kd * 16 + 4 * tig)), b2, b3);
      } else {
        ldsm_x4(sQ + swz16(lane & 15, kd * 16 + (lane >> 4) * 8), af[0], af[1], af[2], af[3]);
        ldsm_x4(sK + swz16((lane & 7) + ((lane >> 4) << 3), kd * 16 + ((lane >> 3) & 1) * 8), b0,
                b1, b2, b3);
      }
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
      ldsm_x4_t(sVf + swz16((lane & 7) + (((lane >> 3) & 1) << 3), nd * 16 + (lane >> 4) * 8), b0,
                b1, b2, b3);
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

  // a timed-out warp may still have copies landing: let them finish
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

template <typename T, bool KV8, int D>
cudaError_t launch_dec(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       int total_items, int n_mblk, uint32_t* counters, cudaStream_t st) {
  using C = DecCfg<D, KV8>;
  auto k = decode_tma_kernel<T, KV8, D>;
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

template <typename T, bool KV8>
cudaError_t launch_dec_d(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                         int items, int n_mblk, uint32_t* cnt, cudaStream_t st) {
  switch (a.p.d) {
    case 64:
      if constexpr (!KV8) return launch_dec<T, KV8, 64>(a, tk, tv, items, n_mblk, cnt, st);
      break;
    case 128: return launch_dec<T, KV8, 128>(a, tk, tv, items, n_mblk, cnt, st);
    case 256: return launch_dec<T, KV8, 256>(a, tk, tv, items, n_mblk, cnt, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_tma_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens) {
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16) || cache_tokens >= (int64_t(1) << 31)) return false;
  if (kv_dtype == q_dtype) return d == 64 || d == 128 || d == 256;
  return kv_dtype == PA_E5M2 && (d == 128 || d == 256);
}

cudaError_t launch_decode_tma(const AttnArgs& a, int q_dtype, int kv_dtype, int n_mblk,
                              cudaStream_t st) {
  if (a.p.num_rows == 0 || n_mblk == 0) return cudaSuccess;
  const int64_t items = (int64_t)a.p.num_rows * a.p.hkv * NSPLIT * n_mblk;
  if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)a.p.num_pages * a.p.page_size;
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, a.kc, kv_dtype, a.p.d, a.p.hkv, tokens) ||
      !encode_kv_map(&tv, a.vc, kv_dtype, a.p.d, a.p.hkv, tokens))
    return cudaErrorInvalidValue;
  uint32_t* counters = reinterpret_cast<WsHeader*>(a.p.err)->pad;
  const bool kv8 = kv_dtype == PA_E5M2;
  if (q_dtype == PA_BF16)
    return kv8 ? launch_dec_d<__nv_bfloat16, true>(a, tk, tv, (int)items, n_mblk, counters, st)
               : launch_dec_d<__nv_bfloat16, false>(a, tk, tv, (int)items, n_mblk, counters, st);
  return kv8 ? launch_dec_d<__half, true>(a, tk, tv, (int)items, n_mblk, counters, st)
             : launch_dec_d<__half, false>(a, tk, tv, (int)items, n_mblk, counters, st);
}

}  // namespace pa
