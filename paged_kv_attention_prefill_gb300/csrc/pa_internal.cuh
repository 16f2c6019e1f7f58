// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "paged_attn.h"

namespace pa {

// Per-device "done once" flags (for function attributes, which are set per
// device).  Racing threads may both run the action; it is idempotent.
struct DeviceFlags {
  std::atomic<uint64_t> mask{0};
  template <typename F>
  cudaError_t once(F&& f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = f();
    if (e == cudaSuccess) mask.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// ---------------------------------------------------------------------------
// Workspace layout (offsets in bytes from the workspace start).
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t err;          // sticky PA_DEVERR_* flags
  uint32_t n_tiles;      // prefill work items written by the plan kernel
  uint32_t n_slots;      // decode token slots written by the plan kernel
  uint32_t n_long;       // long-row decode work items (PA_SPLITS_BY_LENGTH)
  uint32_t pad[60];      // [0, 2): the TMA decode kernel's work counter
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct WsLayout {
  size_t dec_base;   // int32 [num_rows]   partial-slot base of each decode row, -1 otherwise
  size_t row_order;  // int32 [num_rows]   decode rows, longest split first
  size_t slot_tok;   // int32 [max_slots]  global token of each decode slot
  size_t tiles;      // int2  [max_tiles]  (row, m-block) prefill work items
  size_t part_acc;   // float [max_slots, Hq, split_stride, d]
  size_t part_ml;    // float2[max_slots, Hq, split_stride]  (m in log2 units, l)
  size_t long_items; // int2  [max_long]  long-row decode items (row | m-block << 24, split)
  size_t pf_ml;      // float2[total_q, Hq, pf_parts]  prefill key-range parts (0 bytes when off)
  size_t pf_acc;     // float [total_q, Hq, pf_parts, d]
  size_t total;
  int64_t max_slots;
  int64_t max_tiles;
  int64_t max_long;
  int split_stride;  // partial states per (decode token, query head)
};

constexpr int NSPLIT = 16;      // split-KV parts per decode row
constexpr int DEC_KT = 64;      // keys per decode tile; the split partition unit

// Length-only split count for long rows (num_splits = PA_SPLITS_BY_LENGTH).
// Rows of at most LONG_MIN_TILES decode tiles (32768 keys) keep the 16-part
// partition; longer rows get parts of LONG_TPS tiles (2048 keys), at most
// NSPLIT_MAX of them (longer parts past 262144 keys).  The count depends on
// the row's length alone (vllm-rlt PR #128, "Purpose", decode bullets: a
// length-only partition keeps a row's bits independent of the batch).
constexpr int NSPLIT_MAX = 128;
constexpr int LONG_MIN_TILES = 512;
constexpr int LONG_TPS = 32;
constexpr int LONG_BM = 128;    // GQA-packed query rows per long-row work item

// Decode tiles per split of a row with L keys.
__host__ __device__ inline int dec_split_tiles(int L, int by_len) {
  const int n_tiles = L > 0 ? (L + DEC_KT - 1) / DEC_KT : 0;
  if (!by_len || n_tiles <= LONG_MIN_TILES) return (n_tiles + NSPLIT - 1) / NSPLIT;
  // an even count, so a long row's parts are whole 128-key tensor-core tiles
  const int t = ((n_tiles + NSPLIT_MAX - 1) / NSPLIT_MAX + 1) & ~1;
  return t > LONG_TPS ? t : LONG_TPS;
}
// Non-empty splits of a row with L keys.
__host__ __device__ inline int dec_num_splits(int L, int by_len) {
  const int tps = dec_split_tiles(L, by_len);
  return tps ? ((L + DEC_KT - 1) / DEC_KT + tps - 1) / tps : 0;
}
// A row whose splits run on the long-row (tcgen05) decode kernel.
__host__ __device__ inline bool dec_is_long(int L, int by_len) {
  return by_len && L > LONG_MIN_TILES * DEC_KT;
}
// "Last visible key" of a padding row of a query tile (past the row's
// queries): no key is masked, so its warps never take the diagonal path on
// every tile.  Its logits are finite (its Q is zero and the keys past a row's
// end are zero-filled) and its outputs are never stored.
constexpr int NO_MASK = 1 << 30;
constexpr int DEC_ROWS = 16;    // GQA-packed query rows per decode CTA
constexpr int PF_BM = 64;       // GQA-packed query rows per prefill CTA (mma.sync path)

// Prefill key-range parts (1Cat-vLLM PR #1279, commit 5: a CTA's key range
// cut into whole-tile ranges merged by log-sum-exp).  A work item's keys
// [0, k_end) are counted in units of PF_UNIT keys (a multiple of every
// prefill key tile) and cut into at most `max_parts` parts of equal whole
// units (the last takes the rest), each of at least `min_units` units.  With
// a fixed part count the cut depends on k_end alone, so a row's result never
// depends on the rest of the batch, the page size or the physical pages.
constexpr int PF_UNIT = 128;
constexpr int PF_PART_UNITS = 128;   // 16384 keys: least part for a part count the caller fixes
constexpr int PF_AUTO_UNITS = 8;     // 1024 keys: least part for a count chosen per call
constexpr int PF_AUTO_MAX = 4;       // the most parts a count chosen per call takes
constexpr int PF_MAX_PARTS = 16;

WsLayout workspace_layout(int num_rows, int total_q, int hq, int d, int max_decode_q, int g,
                          int pf_parts, int by_len);

// Parts of a work item whose rows see keys [0, k_end): sets the units per
// part and returns the part count (0 for k_end <= 0, 1 when not cut).
__host__ __device__ inline int pf_part_count(int k_end, int max_parts, int min_units,
                                             int* per_units) {
  if (k_end <= 0) {
    *per_units = 0;
    return 0;
  }
  const int n_u = (k_end + PF_UNIT - 1) / PF_UNIT;
  int parts = max_parts > 1 ? (n_u + min_units - 1) / min_units : 1;
  if (parts > max_parts) parts = max_parts;
  if (parts < 1) parts = 1;
  const int per = (n_u + parts - 1) / parts;
  *per_units = per;
  return (n_u + per - 1) / per;
}

// ---------------------------------------------------------------------------
// Device-side problem description, passed by value to every kernel.
// ---------------------------------------------------------------------------
struct Problem {
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* bt;
  int num_rows;
  int total_q;     // rows of q / out: a row whose tokens fall outside is skipped
  int max_pages;
  int num_pages;
  int page_size;
  int hq, hkv, g, d;
  float sl2;       // softmax_scale * k_scale * log2(e): logits in log2 units
  float v_scale;
  uint32_t* err;
};

struct AttnArgs {
  Problem p;
  const void* q;
  const void* kc;
  const void* vc;
  void* out;
  float* part_acc;
  float2* part_ml;
  const int32_t* dec_base;   // mixed: slot base per row (-1: not a decode row); null: slot = token
  const int32_t* slot_tok;   // mixed: global token per slot; null: slot = token
  const int32_t* row_order;  // decode work order of the rows; null: row order
  const int2* tiles;         // prefill work list: (row, m-block | part << 24)
  const uint32_t* n_tiles;   // its length (device)
  int pf_parts;              // prefill key-range parts per work item at most (<= 1: not cut)
  int pf_min_units;          // least PF_UNIT units per part
  float* pf_acc;             // partial states of cut work items
  float2* pf_ml;
  int max_decode_q;
  int64_t max_slots;         // decode slots the workspace holds
  int dec_mblk;              // decode grid: 16-row query blocks per row (per token if tokenwise)
  int tokenwise;             // decode rows with q_b > 1 expanded into one-token rows
  const uint32_t* n_slots;   // mixed: decode slots in use (device); null: every token is a slot
  int split_stride;          // partial states per (decode token, query head): 16 or NSPLIT_MAX
  int by_len;                // length-only split count for long rows (PA_SPLITS_BY_LENGTH)
  int long_tc;               // ... whose parts run on the tile kernel (the decode kernel skips them)
  int split_cap;             // split indices per (row or slot, KV head) on the decode kernel
  const int2* long_items;    // long-row decode items (row | m-block << 24, split)
  const uint32_t* n_long;    // their count (device)
  int64_t max_long;          // entries the list holds
};

// Launchers (one per translation unit family).  Return cudaError_t.
cudaError_t launch_plan(const AttnArgs& a, int mode_mixed, int max_decode_q, int bm,
                        int max_tiles, cudaStream_t st);
cudaError_t launch_decode_mma(const AttnArgs& a, int q_dtype, int kv_dtype, int n_mblk,
                              cudaStream_t st);
cudaError_t launch_prefill_mma(const AttnArgs& a, int q_dtype, int kv_dtype, int max_tiles,
                               cudaStream_t st);
cudaError_t launch_merge(const AttnArgs& a, int q_dtype, int n_slots, cudaStream_t st);
// Merges the key-range parts of the prefill work items that were cut (bm:
// query rows per work item); tokens of uncut items are left as written.
cudaError_t launch_pf_merge(const AttnArgs& a, int q_dtype, int bm, int mixed, cudaStream_t st);
// Rows with more work per decode split first (rows off the decode path
// last); written to `order` for 2 <= num_rows <= MAX_ORDER_ROWS.
constexpr int MAX_ORDER_ROWS = 4096;
cudaError_t launch_row_order(const AttnArgs& a, int32_t* order, cudaStream_t st);
cudaError_t launch_f32(const AttnArgs& a, int decode_mode, int grid_x, int n_mblk,
                       cudaStream_t st);
bool prefill_mma_supported(int q_dtype, int kv_dtype, int d);
// tcgen05 prefill at d = 256 (16-bit q with a same-type or fp8 E5M2 cache,
// cache < 2^31 tokens)
constexpr int PF_BM_TC = 128;
bool prefill_tc_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens);
cudaError_t launch_prefill_tc(const AttnArgs& a, int q_dtype, int kv_dtype, int grid_x,
                              cudaStream_t st);
// tcgen05 prefill with two query tiles per CTA (16-bit Q; same-type cache at
// d = 64 or 128, or an fp8 E5M2 cache at d = 128)
constexpr int PF_BM_TC2 = 256;
bool prefill_tc2_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens);
cudaError_t launch_prefill_tc2(const AttnArgs& a, int q_dtype, int kv_dtype, int grid_x,
                               cudaStream_t st);
// persistent TMA-fed split-KV decode (16-bit q; same-type or fp8 E5M2 cache)
bool decode_tma_supported(int q_dtype, int kv_dtype, int d, int64_t cache_tokens);
// n_units: rows (packed) or decode slots (tokenwise) the work items range over;
// merge_slots > 0: the kernel also merges the partial states of that many
// decode slots itself (no merge kernel); sms: the device's SM count
cudaError_t launch_decode_tma(const AttnArgs& a, int q_dtype, int kv_dtype, int n_mblk,
                              int n_units, int merge_slots, int sms, cudaStream_t st);
// CTAs of that launch (one per SM at most)
int decode_tma_grid(int d, bool kv8, int64_t items, int sms);
bool decode_mma_supported(int q_dtype, int kv_dtype, int d);
// Long-row decode (PA_SPLITS_BY_LENGTH): the list of work items of the rows
// longer than LONG_MIN_TILES decode tiles, then their splits on the tcgen05
// tile kernel (d = 256, 16-bit q with a same-type cache), which writes the
// same fp32 partial states as the decode kernel.  `max_items` bounds the list.
cudaError_t launch_long_items(const AttnArgs& a, int2* items, int64_t max_items,
                              cudaStream_t st);
cudaError_t launch_decode_long(const AttnArgs& a, int q_dtype, int grid, cudaStream_t st);

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills the chunk
// (the source address is then not read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D, m16n8k16, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* c, const uint32_t* a, uint32_t b0,
                                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float* c, const uint32_t* a, uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed pair of 16-bit values (round to nearest even).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_float<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ float from_float<float>(float x) {
  return x;
}

// fp8 E5M2 has the sign, exponent and top two fraction bits of binary16, so
// placing a code in the high byte of a 16-bit word gives the same value as a
// binary16, exactly.  For a bf16 target the binary16 is widened to fp32 and
// narrowed to bf16, also exactly (every E5M2 value is a bf16 value).
template <typename T>
__device__ __forceinline__ void e5m2x4_to(uint32_t w, uint32_t& lo, uint32_t& hi);
template <>
__device__ __forceinline__ void e5m2x4_to<__half>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, 0u, 0x1404);
  hi = __byte_perm(w, 0u, 0x3424);
}
template <>
__device__ __forceinline__ void e5m2x4_to<__nv_bfloat16>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t h0 = __byte_perm(w, 0u, 0x1404), h1 = __byte_perm(w, 0u, 0x3424);
  __half2 a = *reinterpret_cast<__half2*>(&h0), b = *reinterpret_cast<__half2*>(&h1);
  float2 fa = __half22float2(a), fb = __half22float2(b);
  lo = pack2<__nv_bfloat16>(fa.x, fa.y);
  hi = pack2<__nv_bfloat16>(fb.x, fb.y);
}

// Row of global query token t: the largest b with cu_q[b] <= t.
__device__ __forceinline__ int row_of_token(const Problem& p, int t) {
  int lo = 0, hi = p.num_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Splits of the partition a decode token's partial states come from: those
// of its row's length (of the token's own prefix for one-token verify rows).
__device__ __forceinline__ int merge_splits(const AttnArgs& a, int t) {
  const Problem& p = a.p;
  const int b = row_of_token(p, t);
  int L = __ldg(p.seq_lens + b);
  if (a.tokenwise) {
    const int qs = __ldg(p.cu_q + b), qb = __ldg(p.cu_q + b + 1) - qs;
    L = L - qb + 1 + (t - qs);
  }
  return dec_num_splits(L, a.by_len);
}

// The split-KV merge of one (token, head) for NC columns (vllm-rlt PR #128,
// "Purpose", decode: the partial softmax states combined by log-sum-exp):
// M = max_k m_k over the splits k < nsp with l_k > 0, w_k = 2^(m_k - M),
// res = (sum_k w_k acc_k) / (sum_k w_k l_k) * v_scale, summed in the fixed
// order k = 0..15, so a row's result never depends on the batch; 0 when no
// split saw a key.  Both the merge kernel and the decode kernel's
// same-launch merge use it, so their results are the same bits.
template <int NC>
__device__ __forceinline__ void merge16(const float2 (&ml)[NSPLIT], const float (&acc)[NC][NSPLIT],
                                        int nsp, float v_scale, float (&res)[NC]) {
  float mstar = -INFINITY;
#pragma unroll
  for (int k = 0; k < NSPLIT; ++k)
    if (k < nsp && ml[k].y > 0.f) mstar = fmaxf(mstar, ml[k].x);
  float w[NSPLIT];
  float lsum = 0.f;
#pragma unroll
  for (int k = 0; k < NSPLIT; ++k) {
    w[k] = 0.f;
    if (k < nsp && ml[k].y > 0.f) {
      w[k] = exp2f(ml[k].x - mstar);
      lsum += w[k] * ml[k].y;
    }
  }
  const float inv = lsum > 0.f ? v_scale / lsum : 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NSPLIT; ++k)
      if (w[k] != 0.f) s += w[k] * acc[c][k];
    res[c] = s * inv;
  }
}

// Physical element offset of key j of row b, KV head kh, or -1 if the block
// table entry is out of range (then the error flag is raised).
__device__ __forceinline__ int64_t kv_offset(const Problem& p, int b, int j, int kh) {
  const int P = p.page_size;
  const int col = j / P;
  if (col >= p.max_pages) {
    atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return -1;
  }
  const int page = __ldg(p.bt + (int64_t)b * p.max_pages + col);
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return -1;
  }
  return (((int64_t)page * P + (j % P)) * p.hkv + kh) * (int64_t)p.d;
}

#endif  // __CUDACC__

}  // namespace pa
