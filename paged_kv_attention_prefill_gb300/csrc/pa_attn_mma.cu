// Paged attention tiles on warp-level MMA (m16n8k16, fp32 accumulate) for
// 16-bit queries and a 16-bit or fp8 E5M2 KV cache.
//
// One template, two modes:
//
//  * MODE_DECODE -- split-KV decode (vllm-rlt PR #128, "Purpose", decode
//    bullets): a CTA owns one (row, 16-row block of GQA-packed query rows,
//    KV head, split).  The row's keys are cut into NSPLIT contiguous parts of
//    whole DEC_KT-key tiles, chosen from the row's own length only; the CTA
//    streams its part through a cp.async ring, the four warps take 16 keys of
//    each 64-key tile apiece, each keeps its own online-softmax state, and at
//    the end the warps are combined in fixed order into one fp32 partial
//    state (acc[d], m, l) for the merge kernel.
//
//  * MODE_PREFILL -- varlen causal paged prefill (same page, prefill
//    bullets): a CTA owns one (row, 64-row block of GQA-packed query rows, KV
//    head), the four warps take 16 query rows apiece, and the CTA walks every
//    key tile up to the causal bound of its last row with online softmax,
//    writing the normalized output.
//
// GQA packing (1Cat-vLLM PR #1279, commit 1: query rows of the heads that
// share a KV head stacked into one tile): packed row R of a row with q_b new
// tokens is (token R / g, head-in-group R % g), 0 <= R < q_b * g.
//
// Every CTA's arithmetic depends only on its own row's lengths and data, and
// the page size only changes addresses, so results are bitwise independent of
// the rest of the batch, the page size and the physical page order.
#include "pa_internal.cuh"

namespace pa {

constexpr int MODE_DECODE = 0;
constexpr int MODE_PREFILL = 1;
constexpr int KT = 64;  // keys per tile

// cp.async ring depth (tiles in flight + 1) per head dim / cache type / mode,
// chosen so one CTA fits the 227 KB of shared memory.
constexpr int ring_depth(int d, bool kv8, int mode) {
  return kv8 ? 4 : (d == 256 ? (mode == MODE_DECODE ? 3 : 2) : (mode == MODE_DECODE ? 4 : 3));
}

template <typename T, bool KV8, int D, int MODE, int STAGES>
struct MmaCfg {
  static constexpr int ROWS = MODE == MODE_DECODE ? DEC_ROWS : PF_BM;
  static constexpr int ROWB = D * 2;               // bytes of a 16-bit row
  static constexpr int RAWB = KV8 ? D : D * 2;     // bytes of a cached key row
  static constexpr int CHR = RAWB / 16;            // 16-byte chunks of a cached row
  static constexpr int NKW = MODE == MODE_DECODE ? 16 : KT;  // keys per warp per tile
  static constexpr int Q_BYTES = ROWS * ROWB;
  static constexpr int STAGE_BYTES = 2 * KT * RAWB;         // K and V
  static constexpr int STAGING_BYTES = KV8 ? 2 * KT * ROWB : 0;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int MERGE_BYTES = MODE == MODE_DECODE ? 4 * 16 * D * 4 + 2048 : 0;
  static constexpr int SMEM = Q_BYTES + (RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES) +
                              STAGING_BYTES;
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
  static_assert(SMEM <= 232448, "one CTA must fit in 227 KB of shared memory");
};

// Byte offset of 16-byte chunk c of row r in a swizzled 16-bit tile: the
// chunk index is XORed with r % 8 so that the eight rows an ldmatrix reads
// hit eight different bank groups.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * ROWB + ((c ^ (r & 7)) << 4));
}

template <typename T, bool KV8, int D, int MODE, int STAGES>
__global__ void __launch_bounds__(128, 1) attn_mma_kernel(const AttnArgs a) {
  using C = MmaCfg<T, KV8, D, MODE, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* ring = smem + C::Q_BYTES;
  uint8_t* staging = ring + (C::RING_BYTES > C::MERGE_BYTES ? C::RING_BYTES : C::MERGE_BYTES);

  const Problem& p = a.p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;

  // ---- work item ---------------------------------------------------------
  int b, mblk, kh, split = 0;
  if (MODE == MODE_DECODE) {
    // grid (rows x m-blocks, Hkv x NSPLIT): the m-blocks of a row are adjacent
    // so CTAs reading the same keys run together and share L2
    const int n_mblk = a.dec_mblk;
    b = blockIdx.x / n_mblk;
    mblk = blockIdx.x % n_mblk;
    kh = blockIdx.y / NSPLIT;
    split = blockIdx.y % NSPLIT;
  } else {
    if (blockIdx.x >= *a.n_tiles) return;
    const int2 t = a.tiles[blockIdx.x];
    b = t.x;
    mblk = t.y;
    kh = blockIdx.y;
  }
  const int qs = __ldg(p.cu_q + b);
  const int qb = __ldg(p.cu_q + b + 1) - qs;
  const int L = __ldg(p.seq_lens + b);
  if (qb <= 0) return;
  if (qs < 0 || qs + qb > p.total_q) {  // malformed cu_seqlens_q: never index q/out with it
    if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return;
  }
  int slot_base = qs;
  if (MODE == MODE_DECODE) {
    if (a.dec_base) {
      slot_base = __ldg(a.dec_base + b);
      if (slot_base < 0) return;  // not a decode row
    }
    if (qb > a.max_decode_q && mblk == 0 && blockIdx.y == 0 && tid == 0)
      atomicOr(p.err, PA_DEVERR_DECODE_Q);
    if ((int64_t)slot_base + qb > a.max_slots) return;  // flagged above; never written
  }
  const int g = p.g;
  const int M = qb * g;
  const int r0 = mblk * C::ROWS;
  if (r0 >= M) return;

  // key range of this CTA
  int k0, k1;
  if (MODE == MODE_DECODE) {
    const int n_tiles = (L + KT - 1) / KT;
    const int tps = (n_tiles + NSPLIT - 1) / NSPLIT;
    k0 = split * tps * KT;
    if (k0 >= L) return;  // empty split: the merge kernel knows from L alone
    k1 = min(k0 + tps * KT, L);
  } else {
    const int r_last = min(r0 + C::ROWS, M) - 1;
    k0 = 0;
    k1 = min(L, L - qb + r_last / g + 1);  // <= 0 when no row sees a key: zeros out
  }
  const int n_st = k1 > k0 ? (k1 - k0 + KT - 1) / KT : 0;

  // ---- Q tile -------------------------------------------------------------
  {
    const uint8_t* qbase = static_cast<const uint8_t*>(a.q);
    constexpr int CHQ = D / 8;
    for (int e = tid; e < C::ROWS * CHQ; e += 128) {
      const int r = e / CHQ, c = e % CHQ;
      const int R = r0 + r;
      const uint8_t* src = qbase;
      int bytes = 0;
      if (R < M) {
        const int i = R / g, hg = R % g;
        src = qbase + ((int64_t)(qs + i) * p.hq + kh * g + hg) * C::ROWB + c * 16;
        bytes = 16;
      }
      cp_async16(smem_u32(Qs + swz<C::ROWB>(r, c)), src, bytes);
    }
    cp_async_commit();
  }

  // ---- KV ring ------------------------------------------------------------
  const uint8_t* kc = static_cast<const uint8_t*>(a.kc);
  const uint8_t* vc = static_cast<const uint8_t*>(a.vc);
  constexpr int ELT = KV8 ? 1 : 2;
  const int my_key = tid >> 1;            // each key row is loaded by two threads
  const int my_c0 = (tid & 1) * (C::CHR / 2);

  auto load_stage = [&](int st) {
    const int j = k0 + st * KT + my_key;
    uint8_t* Kd = ring + (st % STAGES) * C::STAGE_BYTES;
    uint8_t* Vd = Kd + KT * C::RAWB;
    int64_t off = -1;
    if (j < k1) off = kv_offset(p, b, j, kh);
    const uint8_t* ks = kc;
    const uint8_t* vs = vc;
    int bytes = 0;
    if (off >= 0) {
      ks = kc + off * ELT;
      vs = vc + off * ELT;
      bytes = 16;
    }
#pragma unroll
    for (int cc = 0; cc < C::CHR / 2; ++cc) {
      const int c = my_c0 + cc;
      const uint32_t o = KV8 ? (uint32_t)(my_key * C::RAWB + c * 16) : swz<C::ROWB>(my_key, c);
      cp_async16(smem_u32(Kd + o), ks + (bytes ? c * 16 : 0), bytes);
      cp_async16(smem_u32(Vd + o), vs + (bytes ? c * 16 : 0), bytes);
    }
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < n_st) load_stage(s);
    cp_async_commit();
  }

  // ---- per-warp state -----------------------------------------------------
  constexpr int NT = C::NKW / 8;       // n8 tiles of logits per warp
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  const int wrow0 = MODE == MODE_DECODE ? 0 : warp * 16;  // warp's first tile row
  const int wkey0 = MODE == MODE_DECODE ? warp * 16 : 0;  // warp's first key in a tile
  // causal bound (last visible key) of this thread's two rows
  int last[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int R = r0 + wrow0 + gid + 8 * h;
    last[h] = R < M ? L - qb + R / g : -1;
  }
  const float sl2 = p.sl2;

  for (int st = 0; st < n_st; ++st) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const uint8_t* Kt;
    const uint8_t* Vt;
    if (KV8) {
      // dequantize the chunks this thread loaded into the 16-bit staging tile
      const uint8_t* Kr = ring + (st % STAGES) * C::STAGE_BYTES;
      const uint8_t* Vr = Kr + KT * C::RAWB;
#pragma unroll
      for (int cc = 0; cc < C::CHR / 2; ++cc) {
        const int c = my_c0 + cc;
        const uint32_t ro = my_key * C::RAWB + c * 16;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const uint4 w = *reinterpret_cast<const uint4*>((kv ? Vr : Kr) + ro);
          uint4 lo, hi;
          e5m2x4_to<T>(w.x, lo.x, lo.y);
          e5m2x4_to<T>(w.y, lo.z, lo.w);
          e5m2x4_to<T>(w.z, hi.x, hi.y);
          e5m2x4_to<T>(w.w, hi.z, hi.w);
          uint8_t* dst = staging + kv * KT * C::ROWB;
          *reinterpret_cast<uint4*>(dst + swz<C::ROWB>(my_key, 2 * c)) = lo;
          *reinterpret_cast<uint4*>(dst + swz<C::ROWB>(my_key, 2 * c + 1)) = hi;
        }
      }
      __syncthreads();
      Kt = staging;
      Vt = staging + KT * C::ROWB;
    } else {
      Kt = ring + (st % STAGES) * C::STAGE_BYTES;
      Vt = Kt + KT * C::RAWB;
    }
    // prefetch the tile STAGES-1 ahead into the slot freed last iteration
    if (st + STAGES - 1 < n_st) load_stage(st + STAGES - 1);
    cp_async_commit();

    // ---- S = Q K^T for this warp's rows and keys ----
    float s[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const uint32_t qa = smem_u32(Qs), ka = smem_u32(Kt), va = smem_u32(Vt);
#pragma unroll
    for (int kd = 0; kd < D / 16; ++kd) {
      uint32_t af[4];
      ldsm_x4(qa + swz<C::ROWB>(wrow0 + (lane & 15), kd * 2 + (lane >> 4)), af[0], af[1], af[2],
              af[3]);
#pragma unroll
      for (int kg = 0; kg < NT / 2; ++kg) {
        uint32_t b0, b1, b2, b3;
        const int key = wkey0 + kg * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(ka + swz<C::ROWB>(key, kd * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma16816<T>(s[2 * kg], af, b0, b1);
        mma16816<T>(s[2 * kg + 1], af, b2, b3);
      }
    }

    // ---- mask, online softmax ----
    const int kbase = k0 + st * KT + wkey0;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const int j = kbase + n * 8 + 2 * tig + (e & 1);
        const float x = j <= last[h] ? s[n][e] * sl2 : -INFINITY;
        s[n][e] = x;
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
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = exp2f(s[n][e] - m_use[e >> 1]);
        s[n][e] = pv;
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

    // ---- O += P V ----
#pragma unroll
    for (int kg = 0; kg < NT / 2; ++kg) {
      uint32_t pf[4];
      pf[0] = pack2<T>(s[2 * kg][0], s[2 * kg][1]);
      pf[1] = pack2<T>(s[2 * kg][2], s[2 * kg][3]);
      pf[2] = pack2<T>(s[2 * kg + 1][0], s[2 * kg + 1][1]);
      pf[3] = pack2<T>(s[2 * kg + 1][2], s[2 * kg + 1][3]);
      const int key = wkey0 + kg * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(va + swz<C::ROWB>(key, nd * 2 + (lane >> 4)), b0, b1, b2, b3);
        mma16816<T>(o[2 * nd], pf, b0, b1);
        mma16816<T>(o[2 * nd + 1], pf, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // full row sums of this warp
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }

  if (MODE == MODE_PREFILL) {
    T* out = static_cast<T*>(a.out);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = r0 + wrow0 + gid + 8 * h;
      if (R >= M) continue;
      const int i = R / g, hg = R % g;
      const float inv = l_run[h] > 0.f ? p.v_scale / l_run[h] : 0.f;
      T* dst = out + ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const uint32_t v = pack2<T>(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
        *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * tig) = v;
      }
    }
    return;
  }

  // ---- decode: combine the four warps in fixed order, write the partial ----
  __syncthreads();  // every warp is done with the ring; reuse it
  float* red = reinterpret_cast<float*>(ring);          // [4][16][D]
  float* ms = red + 4 * 16 * D;                         // [4][16]
  float* ls = ms + 4 * 16;                              // [4][16]
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = gid + 8 * (e >> 1);
      red[(warp * 16 + row) * D + n * 8 + 2 * tig + (e & 1)] = o[n][e];
    }
  }
  if (tig == 0) {
    ms[warp * 16 + gid] = m_run[0];
    ms[warp * 16 + gid + 8] = m_run[1];
    ls[warp * 16 + gid] = l_run[0];
    ls[warp * 16 + gid + 8] = l_run[1];
  }
  __syncthreads();
  float* wts = ls + 4 * 16;                             // [4][16] weights, then [16] M*, [16] l*
  if (tid < 16) {
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mstar = fmaxf(mstar, ms[w * 16 + tid]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = (mstar == -INFINITY) ? 0.f : exp2f(ms[w * 16 + tid] - mstar);
      wts[w * 16 + tid] = f;
      lsum += ls[w * 16 + tid] * f;
    }
    wts[64 + tid] = mstar;
    wts[80 + tid] = lsum;
  }
  __syncthreads();
  const int Hq = p.hq;
  for (int e = tid; e < 16 * D; e += 128) {
    const int row = e / D, col = e % D;
    const int R = r0 + row;
    if (R >= M) continue;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc += red[(w * 16 + row) * D + col] * wts[w * 16 + row];
    const int i = R / g, hg = R % g;
    const int64_t slot = slot_base + i;
    a.part_acc[((slot * Hq + kh * g + hg) * a.split_stride + split) * D + col] = acc;
  }
  if (tid < 16) {
    const int R = r0 + tid;
    if (R < M) {
      const int i = R / g, hg = R % g;
      const int64_t slot = slot_base + i;
      a.part_ml[(slot * Hq + kh * g + hg) * a.split_stride + split] = make_float2(wts[64 + tid], wts[80 + tid]);
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch
// ---------------------------------------------------------------------------
template <typename T, bool KV8, int D, int MODE, int STAGES>
static cudaError_t launch_one(const AttnArgs& a, dim3 grid, cudaStream_t st) {
  using C = MmaCfg<T, KV8, D, MODE, STAGES>;
  auto k = attn_mma_kernel<T, KV8, D, MODE, STAGES>;
  static DeviceFlags attr_set;
  cudaError_t e = attr_set.once([&] {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (e != cudaSuccess) return e;
  k<<<grid, 128, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t dispatch(const AttnArgs& a, int q_dtype, int kv_dtype, dim3 grid,
                            cudaStream_t st) {
  const bool kv8 = kv_dtype == PA_E5M2;
  const int d = a.p.d;
#define PA_CASE(TT, DD)                                                       \
  if (d == DD) {                                                              \
    if (kv8) return launch_one<TT, true, DD, MODE, ring_depth(DD, true, MODE)>(a, grid, st); \
    return launch_one<TT, false, DD, MODE, ring_depth(DD, false, MODE)>(a, grid, st);       \
  }
  if (q_dtype == PA_BF16) {
    PA_CASE(__nv_bfloat16, 64)
    PA_CASE(__nv_bfloat16, 128)
    PA_CASE(__nv_bfloat16, 256)
  } else if (q_dtype == PA_F16) {
    PA_CASE(__half, 64)
    PA_CASE(__half, 128)
    PA_CASE(__half, 256)
  }
#undef PA_CASE
  return cudaErrorInvalidValue;
}

bool decode_mma_supported(int q_dtype, int kv_dtype, int d) {
  return (q_dtype == PA_BF16 || q_dtype == PA_F16) && (kv_dtype == q_dtype || kv_dtype == PA_E5M2) &&
         (d == 64 || d == 128 || d == 256);
}
bool prefill_mma_supported(int q_dtype, int kv_dtype, int d) {
  return decode_mma_supported(q_dtype, kv_dtype, d);
}

cudaError_t launch_decode_mma(const AttnArgs& a, int q_dtype, int kv_dtype, int n_mblk,
                              cudaStream_t st) {
  if (a.p.num_rows == 0 || n_mblk == 0) return cudaSuccess;
  dim3 grid((unsigned)a.p.num_rows * n_mblk, a.p.hkv * NSPLIT);
  return dispatch<MODE_DECODE>(a, q_dtype, kv_dtype, grid, st);
}

cudaError_t launch_prefill_mma(const AttnArgs& a, int q_dtype, int kv_dtype, int max_tiles,
                               cudaStream_t st) {
  if (max_tiles == 0) return cudaSuccess;
  dim3 grid(max_tiles, a.p.hkv);
  return dispatch<MODE_PREFILL>(a, q_dtype, kv_dtype, grid, st);
}

}  // namespace pa
