// Row plan (the mixed call's router), the split-KV merge, and the fp32 path.
#include "pa_internal.cuh"

namespace pa {

// In-place descending bitonic sort of npow (a power of two) keys in shared
// memory by one 1024-thread CTA.
__device__ void bitonic_sort_desc(unsigned long long* keys, int npow) {
  const int tid = threadIdx.x;
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npow; i += 1024) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = keys[i], y = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            keys[i] = y;
            keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------
// Plan: classify rows and lay out the work of one call (one CTA).
//
// Mixed mode (1Cat-vLLM PR #616, original description, "Purpose": short
// decode and speculative-verify rows are routed to a single paged-decode
// launch and left out of the prefill work): a row with 1 <= q_b <= max_decode_q gets
// q_b consecutive decode slots (its partial states); every other row with
// q_b > 0 gets ceil(q_b * g / bm) prefill work items.  Prefill-only mode
// sends every row with q_b > 0 to the prefill list.  Work items of a row are
// listed last block first (the blocks with the most visible keys first).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(const AttnArgs a, int mixed, int max_dq,
                                                    int bm, WsHeader* hdr, int32_t* dec_base,
                                                    int32_t* slot_tok, int2* tiles, int max_tiles,
                                                    int64_t max_slots) {
  __shared__ int s_tiles[1024], s_slots[1024];
  __shared__ int s_tot_tiles, s_tot_slots;
  const Problem& p = a.p;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_tot_tiles = 0;
    s_tot_slots = 0;
  }
  __syncthreads();
  for (int c0 = 0; c0 < p.num_rows; c0 += 1024) {
    const int b = c0 + tid;
    int qb = 0, qs = 0;
    if (b < p.num_rows) {
      qs = p.cu_q[b];
      qb = p.cu_q[b + 1] - qs;
    }
    if (qs < 0 || qs + qb > p.total_q) qb = 0;  // malformed row: the kernels skip it too
    const bool dec = mixed && qb >= 1 && qb <= max_dq;
    const int nmb = (!dec && qb > 0) ? (qb * p.g + bm - 1) / bm : 0;
    // work items of the row: one per m-block, or one per key-range part
    int nt = nmb;
    if (a.pf_parts > 1 && nmb > 0) {
      const int L = p.seq_lens[b];
      nt = 0;
      for (int m = 0; m < nmb; ++m) {
        int per;
        const int r_last = min((m + 1) * bm, qb * p.g) - 1;
        const int k_end = min(L, L - qb + r_last / p.g + 1);
        nt += max(1, pf_part_count(k_end, a.pf_parts, a.pf_min_units, &per));
      }
    }
    const int ns = dec ? qb : 0;
    s_tiles[tid] = nt;
    s_slots[tid] = ns;
    __syncthreads();
    // inclusive Hillis-Steele scan over the chunk
    for (int off = 1; off < 1024; off <<= 1) {
      const int vt = tid >= off ? s_tiles[tid - off] : 0;
      const int vs = tid >= off ? s_slots[tid - off] : 0;
      __syncthreads();
      s_tiles[tid] += vt;
      s_slots[tid] += vs;
      __syncthreads();
    }
    const int t_off = s_tot_tiles + s_tiles[tid] - nt;
    const int s_off = s_tot_slots + s_slots[tid] - ns;
    if (b < p.num_rows) {
      if (mixed) dec_base[b] = dec ? s_off : -1;
      for (int k = 0; k < ns; ++k)
        if (s_off + k < max_slots) slot_tok[s_off + k] = qs + k;
      if (nt == nmb) {
        for (int m = 0; m < nt; ++m)
          if (t_off + m < max_tiles) tiles[t_off + m] = make_int2(b, nt - 1 - m);
      } else {
        const int L = p.seq_lens[b];
        int k = t_off;
        for (int m = nmb - 1; m >= 0; --m) {
          int per;
          const int r_last = min((m + 1) * bm, qb * p.g) - 1;
          const int k_end = min(L, L - qb + r_last / p.g + 1);
          const int parts = max(1, pf_part_count(k_end, a.pf_parts, a.pf_min_units, &per));
          for (int c = 0; c < parts; ++c, ++k)
            if (k < max_tiles) tiles[k] = make_int2(b, m | (c << 24));
        }
      }
    }
    __syncthreads();
    if (tid == 1023) {
      s_tot_tiles += s_tiles[1023];
      s_tot_slots += s_slots[1023];
    }
    __syncthreads();
  }
  if (tid == 0) {
    hdr->n_tiles = (uint32_t)min(s_tot_tiles, max_tiles);
    hdr->n_slots = (uint32_t)min((int64_t)s_tot_slots, max_slots);
  }

  // Longest-first order of the prefill work items (by the keys the item's
  // rows can see, in its part), so the CTAs dispatched last are the short
  // ones; equal items keep the parts of one key range together.  Items are
  // independent, so the order changes no result.  Lists longer than 4096
  // items keep row order.
  __syncthreads();
  const int n = min(s_tot_tiles, max_tiles);
  if (n < 2 || n > 4096) return;
  __shared__ unsigned long long keys[4096];
  __shared__ int s_bad;
  int npow = 2;
  while (npow < n) npow <<= 1;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int i = tid; i < npow; i += 1024) {
    unsigned long long key = 0ull;
    if (i < n) {
      const int2 t = tiles[i];
      const int mb = t.y & 0xFFFFFF, c = t.y >> 24;
      const int qs = p.cu_q[t.x], qb = p.cu_q[t.x + 1] - qs, L = p.seq_lens[t.x];
      const int r_last = min((mb + 1) * bm, qb * p.g) - 1;
      int work = max(0, min(L, L - qb + r_last / p.g + 1));
      if (a.pf_parts > 1) {
        int per;
        if (pf_part_count(work, a.pf_parts, a.pf_min_units, &per) > 1)
          work = min(work - c * per * PF_UNIT, per * PF_UNIT);
      }
      if (t.x >= (1 << 20) || mb >= (1 << 14) || c >= 16) s_bad = 1;
      // 26 bits of work (64-key units), row, part, m-block
      const unsigned long long w64 = (unsigned long long)((unsigned)work + 63u) >> 6;
      key = (w64 << 38) | ((unsigned long long)t.x << 18) | ((unsigned)c << 14) | (unsigned)mb;
    }
    keys[i] = key;
  }
  __syncthreads();
  if (s_bad) return;
  bitonic_sort_desc(keys, npow);
  for (int i = tid; i < n; i += 1024) {
    const unsigned long long key = keys[i];
    const int c = (int)((key >> 14) & 0xFu), mb = (int)(key & 0x3FFFu);
    tiles[i] = make_int2((int)((key >> 18) & 0xFFFFFu), mb | (c << 24));
  }
}

cudaError_t launch_plan(const AttnArgs& a, int mode_mixed, int max_decode_q, int bm,
                        int max_tiles, cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.p.err);
  plan_kernel<<<1, 1024, 0, st>>>(a, mode_mixed, max_decode_q, bm, hdr,
                                  const_cast<int32_t*>(a.dec_base),
                                  const_cast<int32_t*>(a.slot_tok), const_cast<int2*>(a.tiles),
                                  max_tiles, a.max_slots);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Long-row decode items (PA_SPLITS_BY_LENGTH, one CTA).  Every decode row
// longer than LONG_MIN_TILES decode tiles contributes one item per split of
// its length-only partition and per block of LONG_BM GQA-packed query rows:
// (row | block << 24, split), listed row by row.  The long-row kernel runs
// each item once per KV head.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) long_items_kernel(const AttnArgs a, int2* items,
                                                          int64_t max_items) {
  __shared__ int s_cnt[1024];
  __shared__ int s_tot;
  const Problem& p = a.p;
  const int tid = threadIdx.x;
  if (tid == 0) s_tot = 0;
  __syncthreads();
  for (int c0 = 0; c0 < p.num_rows; c0 += 1024) {
    const int b = c0 + tid;
    int cnt = 0, nsp = 0, nmb = 0;
    if (b < p.num_rows) {
      const int qs = p.cu_q[b], qb = p.cu_q[b + 1] - qs, L = p.seq_lens[b];
      const bool dec = qb >= 1 && qb <= a.max_decode_q && qs >= 0 && qs + qb <= p.total_q &&
                       (a.dec_base == nullptr || a.dec_base[b] >= 0);
      if (dec && dec_is_long(L, 1)) {
        nsp = dec_num_splits(L, 1);
        nmb = (qb * p.g + LONG_BM - 1) / LONG_BM;
        cnt = nsp * nmb;
      }
    }
    s_cnt[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int v = tid >= off ? s_cnt[tid - off] : 0;
      __syncthreads();
      s_cnt[tid] += v;
      __syncthreads();
    }
    const int64_t o = (int64_t)s_tot + s_cnt[tid] - cnt;
    for (int k = 0; k < cnt; ++k)
      if (o + k < max_items) items[o + k] = make_int2(b | ((k % nmb) << 24), k / nmb);
    __syncthreads();
    if (tid == 1023) s_tot += s_cnt[1023];
    __syncthreads();
  }
  if (tid == 0)
    reinterpret_cast<WsHeader*>(p.err)->n_long = (uint32_t)min((int64_t)s_tot, max_items);
}

cudaError_t launch_long_items(const AttnArgs& a, int2* items, int64_t max_items,
                              cudaStream_t st) {
  if (a.p.num_rows >= (1 << 24)) return cudaErrorInvalidValue;
  long_items_kernel<<<1, 1024, 0, st>>>(a, items, max_items);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Decode work order.  The persistent decode kernel hands out its items
// (row, KV head, split, row block) in row order; listing the rows whose
// splits hold the most keys first (longest processing time first) keeps the
// items taken last short, so fewer warps idle at the end of the call.  Items
// are independent, so the order changes no result.  Rows off the decode
// path (mixed calls) go last; ties keep row order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) row_order_kernel(const AttnArgs a, int32_t* order) {
  __shared__ unsigned long long keys[MAX_ORDER_ROWS];
  const Problem& p = a.p;
  const int n = p.num_rows;  // 2 .. MAX_ORDER_ROWS, checked by the host
  int npow = 2;
  while (npow < n) npow <<= 1;
  for (int i = threadIdx.x; i < npow; i += 1024) {
    unsigned long long key = 0ull;  // padding sorts below every row
    if (i < n) {
      const int qs = p.cu_q[i], qb = p.cu_q[i + 1] - qs;
      const bool dec = qb >= 1 && qs >= 0 && qs + qb <= p.total_q &&
                       (a.dec_base == nullptr || a.dec_base[i] >= 0);
      unsigned work = 0;
      if (dec) {
        const int L = max(p.seq_lens[i], 0);
        // rows on the long-row kernel take no decode-kernel items: last
        work = a.long_tc && dec_is_long(L, 1) ? 0u : (unsigned)dec_split_tiles(L, a.by_len) + 1u;
      }
      key = ((unsigned long long)work << 32) | (unsigned)(n - i);
    }
    keys[i] = key;
  }
  __syncthreads();
  bitonic_sort_desc(keys, npow);
  for (int i = threadIdx.x; i < n; i += 1024) order[i] = n - (int)(keys[i] & 0xFFFFFFFFull);
}

cudaError_t launch_row_order(const AttnArgs& a, int32_t* order, cudaStream_t st) {
  if (a.p.num_rows < 2 || a.p.num_rows > MAX_ORDER_ROWS) return cudaErrorInvalidValue;
  row_order_kernel<<<1, 1024, 0, st>>>(a, order);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Merge (vllm-rlt PR #128, "Purpose", decode: the second kernel combining the
// fp32 partial states of a (row, head)).  For one decode token and query
// head: M = max_k m_k over the splits with l_k > 0, w_k = 2^(m_k - M),
// out = (sum_k w_k acc_k) / (sum_k w_k l_k) * v_scale, summed in the fixed
// order k = 0, 1, ... so a row's result never depends on the batch.  A token
// with no visible key gets 0.  The split count comes from the row's length
// exactly as the decode kernels cut it: 16, or for a long row under
// PA_SPLITS_BY_LENGTH up to NSPLIT_MAX.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(64) merge_kernel(const AttnArgs a, const uint32_t* n_slots_dev,
                                                   int n_slots) {
  const Problem& p = a.p;
  const int slot = blockIdx.x;
  const int h = blockIdx.y;
  if (n_slots_dev && slot >= (int)*n_slots_dev) return;
  if (slot >= n_slots) return;
  // The first 16 partial states and this thread's accumulator columns are
  // loaded before the row lookup, so their latency overlaps it: splits past
  // the row's last (never written: stale bytes) get weight 0 and are not
  // read further.
  constexpr int CPT = D / 64;  // accumulator columns per thread
  const float2* ml = a.part_ml + ((int64_t)slot * p.hq + h) * a.split_stride;
  const float* acc = a.part_acc + ((int64_t)slot * p.hq + h) * a.split_stride * D;
  float2 mlv[NSPLIT];
  float av[CPT][NSPLIT];
#pragma unroll
  for (int k = 0; k < NSPLIT; ++k) {
    mlv[k] = ml[k];
#pragma unroll
    for (int c = 0; c < CPT; ++c) av[c][k] = acc[k * D + threadIdx.x + 64 * c];
  }
  const int t = a.slot_tok ? a.slot_tok[slot] : slot;
  const int nsp = merge_splits(a, t);
  T* out = static_cast<T*>(a.out) + ((int64_t)t * p.hq + h) * D;

  if (nsp > NSPLIT) {
    // a long row: the same arithmetic over all of its splits, in order
    float mstar = -INFINITY;
    for (int k = 0; k < nsp; ++k) {
      const float2 v = ml[k];
      if (v.y > 0.f) mstar = fmaxf(mstar, v.x);
    }
    float lsum = 0.f, s[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) s[c] = 0.f;
    for (int k0 = 0; k0 < nsp; k0 += 8) {
      float2 v[8];
      float x[CPT][8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u < nsp ? k0 + u : nsp - 1;
        v[u] = ml[k];
#pragma unroll
        for (int c = 0; c < CPT; ++c) x[c][u] = acc[(int64_t)k * D + threadIdx.x + 64 * c];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (k0 + u < nsp && v[u].y > 0.f) {
          const float w = exp2f(v[u].x - mstar);
          lsum += w * v[u].y;
#pragma unroll
          for (int c = 0; c < CPT; ++c) s[c] += w * x[c][u];
        }
      }
    }
    const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c) out[threadIdx.x + 64 * c] = from_float<T>(s[c] * inv);
    return;
  }

  float res[CPT];
  merge16<CPT>(mlv, av, nsp, p.v_scale, res);
#pragma unroll
  for (int c = 0; c < CPT; ++c) out[threadIdx.x + 64 * c] = from_float<T>(res[c]);
}

cudaError_t launch_merge(const AttnArgs& a, int q_dtype, int n_slots, cudaStream_t st) {
  if (n_slots <= 0 || a.p.num_rows == 0) return cudaSuccess;
  const uint32_t* nsd =
      a.slot_tok ? &reinterpret_cast<const WsHeader*>(a.p.err)->n_slots : nullptr;
  dim3 grid(n_slots, a.p.hq);
#define PA_M(TT, DD)                                                     \
  if (a.p.d == DD) {                                                     \
    merge_kernel<TT, DD><<<grid, 64, 0, st>>>(a, nsd, n_slots);          \
    return cudaGetLastError();                                           \
  }
  if (q_dtype == PA_BF16) {
    PA_M(__nv_bfloat16, 64) PA_M(__nv_bfloat16, 128) PA_M(__nv_bfloat16, 256)
  } else if (q_dtype == PA_F16) {
    PA_M(__half, 64) PA_M(__half, 128) PA_M(__half, 256)
  } else if (q_dtype == PA_F32) {
    PA_M(float, 64) PA_M(float, 128) PA_M(float, 256)
  }
#undef PA_M
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Merge of prefill key-range parts (1Cat-vLLM PR #1279, commit 5: the parts
// of a CTA's key range combined by log-sum-exp).  For one prefill token and
// query head whose work item was cut: M = max_c m_c over the parts with
// l_c > 0, w_c = 2^(m_c - M), out = (sum_c w_c acc_c) / (sum_c w_c l_c) *
// v_scale in the fixed order c = 0, 1, ...  The part count is recomputed
// from the work item's key count exactly as the plan kernel cut it.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(64) pf_merge_kernel(const AttnArgs a, int bm, int mixed) {
  const Problem& p = a.p;
  const int t = blockIdx.x, h = blockIdx.y;
  int lo = 0, hi = p.num_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int qs = __ldg(p.cu_q + b), qb = __ldg(p.cu_q + b + 1) - qs;
  if (t < qs || t >= qs + qb || qs + qb > p.total_q) return;
  if (mixed && qb <= a.max_decode_q) return;  // a decode row
  const int L = __ldg(p.seq_lens + b);
  const int M = qb * p.g;
  const int R = (t - qs) * p.g + h % p.g;  // GQA-packed row within the row's query rows
  const int mb = R / bm;
  const int r_last = min((mb + 1) * bm, M) - 1;
  int per;
  const int k_end = min(L, L - qb + r_last / p.g + 1);
  const int parts = pf_part_count(k_end, a.pf_parts, a.pf_min_units, &per);
  if (parts <= 1) return;  // written by the prefill kernel itself

  const float2* ml = a.pf_ml + ((int64_t)t * p.hq + h) * a.pf_parts;
  float mstar = -INFINITY;
  for (int c = 0; c < parts; ++c) {
    const float2 v = ml[c];
    if (v.y > 0.f) mstar = fmaxf(mstar, v.x);
  }
  float w[PF_MAX_PARTS];
  float lsum = 0.f;
#pragma unroll
  for (int c = 0; c < PF_MAX_PARTS; ++c) {
    w[c] = 0.f;
    if (c < parts) {
      const float2 v = ml[c];
      if (v.y > 0.f) {
        w[c] = exp2f(v.x - mstar);
        lsum += w[c] * v.y;
      }
    }
  }
  const float inv = lsum > 0.f ? p.v_scale / lsum : 0.f;
  const float* acc = a.pf_acc + ((int64_t)t * p.hq + h) * a.pf_parts * D;
  T* out = static_cast<T*>(a.out) + ((int64_t)t * p.hq + h) * D;
  for (int col = threadIdx.x; col < D; col += 64) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < PF_MAX_PARTS; ++c)
      if (w[c] != 0.f) s += w[c] * acc[c * D + col];
    out[col] = from_float<T>(s * inv);
  }
}

cudaError_t launch_pf_merge(const AttnArgs& a, int q_dtype, int bm, int mixed, cudaStream_t st) {
  if (a.pf_parts <= 1 || a.p.total_q == 0 || a.p.num_rows == 0) return cudaSuccess;
  dim3 grid(a.p.total_q, a.p.hq);
#define PA_M(TT, DD)                                                   \
  if (a.p.d == DD) {                                                   \
    pf_merge_kernel<TT, DD><<<grid, 64, 0, st>>>(a, bm, mixed);        \
    return cudaGetLastError();                                         \
  }
  if (q_dtype == PA_BF16) {
    PA_M(__nv_bfloat16, 64) PA_M(__nv_bfloat16, 128) PA_M(__nv_bfloat16, 256)
  } else if (q_dtype == PA_F16) {
    PA_M(__half, 64) PA_M(__half, 128) PA_M(__half, 256)
  }
#undef PA_M
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// fp32 path: full-precision fp32 products on the FMA pipes (vllm-rlt PR #128,
// "Purpose", prefill bullets: fp32 inputs keep IEEE fp32 multiplies, with no
// reduced-precision tensor-core arithmetic).  A CTA owns 16 GQA-packed query rows of
// one (row, KV head) and either one decode split (partial state out, the same
// partition and merge as the 16-bit path) or the row's whole causal range
// (normalized output).  Warp w holds rows 4w..4w+3; each lane holds d/32
// consecutive columns; keys are taken one at a time.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) f32_kernel(const AttnArgs a, int decode_mode) {
  constexpr int E = D / 32;
  const Problem& p = a.p;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int b, mblk, kh, split = 0;
  if (decode_mode) {
    b = blockIdx.x / a.dec_mblk;
    mblk = blockIdx.x % a.dec_mblk;
    kh = blockIdx.y / NSPLIT;
    split = blockIdx.y % NSPLIT;
  } else {
    if (blockIdx.x >= *a.n_tiles) return;
    const int2 t = a.tiles[blockIdx.x];
    b = t.x;
    mblk = t.y;
    kh = blockIdx.y;
  }
  const int qs = p.cu_q[b];
  const int qb = p.cu_q[b + 1] - qs;
  const int L = p.seq_lens[b];
  if (qb <= 0) return;
  if (qs < 0 || qs + qb > p.total_q) {
    if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
    return;
  }
  int slot_base = qs;
  if (decode_mode && a.dec_base) {
    slot_base = a.dec_base[b];
    if (slot_base < 0) return;
  }
  if (decode_mode && qb > a.max_decode_q && mblk == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    atomicOr(p.err, PA_DEVERR_DECODE_Q);
  if (decode_mode && (int64_t)slot_base + qb > a.max_slots) return;
  const int g = p.g, M = qb * g;
  const int r0 = mblk * 16;
  if (r0 >= M) return;
  int k0, k1;
  if (decode_mode) {
    const int n_tiles = (L + DEC_KT - 1) / DEC_KT;
    const int tps = (n_tiles + NSPLIT - 1) / NSPLIT;
    k0 = split * tps * DEC_KT;
    if (k0 >= L) return;
    k1 = min(k0 + tps * DEC_KT, L);
  } else {
    k0 = 0;
    k1 = min(L, L - qb + (min(r0 + 16, M) - 1) / g + 1);
  }

  const float* qp = static_cast<const float*>(a.q);
  const float* kc = static_cast<const float*>(a.kc);
  const float* vc = static_cast<const float*>(a.vc);
  float qv[4][E], o[4][E], m[4], l[4];
  int last[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int R = r0 + warp * 4 + r;
    last[r] = R < M ? L - qb + R / g : -1;
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      o[r][e] = 0.f;
      qv[r][e] = R < M ? qp[((int64_t)(qs + R / g) * p.hq + kh * g + R % g) * D + lane * E + e] : 0.f;
    }
  }
  int kmax = k1 - 1;
  kmax = min(kmax, max(max(last[0], last[1]), max(last[2], last[3])));
  for (int j = k0; j <= kmax; ++j) {
    const int64_t off = kv_offset(p, b, j, kh);
    float kv[E], vv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kv[e] = off >= 0 ? kc[off + lane * E + e] : 0.f;
      vv[e] = off >= 0 ? vc[off + lane * E + e] : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(qv[r][e], kv[e], s);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o2);
      if (j > last[r]) continue;
      const float x = s * p.sl2;
      const float mn = fmaxf(m[r], x);
      const float al = exp2f(m[r] - mn);
      const float pj = exp2f(x - mn);
      l[r] = l[r] * al + pj;
#pragma unroll
      for (int e = 0; e < E; ++e) o[r][e] = fmaf(pj, vv[e], o[r][e] * al);
      m[r] = mn;
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int R = r0 + warp * 4 + r;
    if (R >= M) continue;
    const int i = R / g, hg = R % g;
    if (decode_mode) {
      const int64_t slot = slot_base + i;
      const int64_t base = (slot * p.hq + kh * g + hg) * a.split_stride + split;
#pragma unroll
      for (int e = 0; e < E; ++e) a.part_acc[base * D + lane * E + e] = o[r][e];
      if (lane == 0) a.part_ml[base] = make_float2(m[r], l[r]);
    } else {
      const float inv = l[r] > 0.f ? p.v_scale / l[r] : 0.f;
      float* out = static_cast<float*>(a.out) + ((int64_t)(qs + i) * p.hq + kh * g + hg) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) out[lane * E + e] = o[r][e] * inv;
    }
  }
}

cudaError_t launch_f32(const AttnArgs& a, int decode_mode, int grid_x, int n_mblk,
                       cudaStream_t st) {
  dim3 grid;
  if (decode_mode) {
    if (a.p.num_rows == 0 || n_mblk == 0) return cudaSuccess;
    grid = dim3((unsigned)a.p.num_rows * n_mblk, a.p.hkv * NSPLIT);
  } else {
    if (grid_x == 0) return cudaSuccess;
    grid = dim3(grid_x, a.p.hkv);
  }
  switch (a.p.d) {
    case 64: f32_kernel<64><<<grid, 128, 0, st>>>(a, decode_mode); break;
    case 128: f32_kernel<128><<<grid, 128, 0, st>>>(a, decode_mode); break;
    case 256: f32_kernel<256><<<grid, 128, 0, st>>>(a, decode_mode); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa
