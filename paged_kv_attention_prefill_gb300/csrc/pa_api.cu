// C ABI of the paged attention library: argument checks, workspace layout,
// routing and launches.  No allocation, no stream synchronization.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <functional>
#include <queue>
#include <vector>

#include "pa_internal.cuh"

namespace pa {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int64_t max_tiles_for(int num_rows, int total_q, int g, int bm, int pf_parts) {
  return (((int64_t)total_q * g + bm - 1) / bm + num_rows) * std::max(1, pf_parts);
}

WsLayout workspace_layout(int num_rows, int total_q, int hq, int d, int max_decode_q, int g,
                          int pf_parts, int by_len) {
  WsLayout w{};
  w.max_slots = std::min<int64_t>(total_q, (int64_t)num_rows * max_decode_q);
  w.split_stride = by_len ? NSPLIT_MAX : NSPLIT;
  // long-row items: every row long, every split, every 128-row block
  w.max_long = by_len ? (int64_t)num_rows * NSPLIT_MAX *
                            (((int64_t)max_decode_q * g + LONG_BM - 1) / LONG_BM)
                      : 0;
  // the smallest tile height in use
  w.max_tiles = max_tiles_for(num_rows, total_q, g, 16, pf_parts);
  size_t off = sizeof(WsHeader);
  w.dec_base = off;
  off += align_up((size_t)num_rows * 4, 256);
  w.row_order = off;
  off += align_up((size_t)num_rows * 4, 256);
  w.slot_tok = off;
  off += align_up((size_t)w.max_slots * 4, 256);
  w.tiles = off;
  off += align_up((size_t)w.max_tiles * 8, 256);
  w.part_ml = off;
  off += align_up((size_t)w.max_slots * hq * w.split_stride * 8, 256);
  w.part_acc = off;
  off += align_up((size_t)w.max_slots * hq * w.split_stride * d * 4, 256);
  w.long_items = off;
  off += align_up((size_t)w.max_long * 8, 256);
  const size_t pf = pf_parts > 1 ? (size_t)total_q * hq * pf_parts : 0;
  w.pf_ml = off;
  off += align_up(pf * 8, 256);
  w.pf_acc = off;
  off += pf * d * 4;
  w.total = align_up(off, 256);
  return w;
}

namespace {

// The device address of the array paged_attn_decode_static uses (end of file).
pa_status static_scratch_address(void** out);

struct Resolved {
  int hq, hkv, g, d, P;
  int qd, kvd;
  float scale, k_scale, v_scale;
  int max_dq;
  int tokenwise;      // decode rows with q_b > 1 as one-token rows
  bool host;          // host mirrors present
  int host_max_q_dec; // mixed/decode: largest q_b among decode rows (host mirrors)
  int host_tiles;     // prefill work items (host mirrors), for the tile height in use
  int host_slots;     // decode slots (host mirrors)
  bool tc;            // prefill on the tcgen05 kernel
  bool tc2;           // prefill on the two-tile tcgen05 kernel
  int pf_bm;          // query rows per prefill work item
  int pf_parts;       // prefill parts the workspace holds (prefill_kv_parts, 4 for auto)
  bool pf_auto;       // part count chosen per call
  int pf_cut;         // key-range parts in use (the tcgen05 kernels cut; others do not)
  int pf_min_units;   // least 128-key units per part
  int by_len;         // length-only split count for long decode rows
  bool long_tc;       // long decode rows on the tcgen05 kernel
  int split_cap;      // split indices per (row, KV head) on the decode kernel
  int host_long;      // long-row decode work items (host mirrors)
  int host_short;     // decode rows on the decode kernel (host mirrors)
  int merge_mode;     // PA_MERGE_*
};

// 0 = not checked, 1 = sm_103, 2 = other
std::atomic<uint8_t> g_dev_ok[64];

pa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_NO_DEVICE;
  const int slot = dev & 63;
  uint8_t s = g_dev_ok[slot].load(std::memory_order_acquire);
  if (s == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return PA_ERR_NO_DEVICE;
    s = (maj == 10 && min == 3) ? 1 : 2;
    g_dev_ok[slot].store(s, std::memory_order_release);
  }
  return s == 1 ? PA_OK : PA_ERR_NO_DEVICE;
}

pa_status resolve_params(const pa_params* prm, Resolved* r) {
  if (!prm) return PA_ERR_INVALID_ARG;
  if (prm->num_q_heads <= 0 || prm->num_kv_heads <= 0 ||
      prm->num_q_heads % prm->num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (prm->page_size <= 0 || prm->page_size % 16 != 0) return PA_ERR_INVALID_ARG;
  if (prm->head_dim <= 0) return PA_ERR_INVALID_ARG;
  if (prm->head_dim != 64 && prm->head_dim != 128 && prm->head_dim != 256)
    return PA_ERR_UNSUPPORTED;
  const int qd = prm->q_dtype, kvd = prm->kv_dtype;
  if (qd != PA_BF16 && qd != PA_F16 && qd != PA_F32) return PA_ERR_UNSUPPORTED;
  if (!(kvd == qd || (kvd == PA_E5M2 && qd != PA_F32))) return PA_ERR_UNSUPPORTED;
  if (prm->num_splits != 0 && prm->num_splits != NSPLIT &&
      prm->num_splits != PA_SPLITS_BY_LENGTH)
    return PA_ERR_UNSUPPORTED;
  r->by_len = prm->num_splits == PA_SPLITS_BY_LENGTH;
  if (prm->merge_mode != PA_MERGE_AUTO && prm->merge_mode != PA_MERGE_SEPARATE &&
      prm->merge_mode != PA_MERGE_SAME_LAUNCH)
    return PA_ERR_INVALID_ARG;
  r->merge_mode = prm->merge_mode;
  if (prm->max_decode_q < 0) return PA_ERR_INVALID_ARG;
  if (!(std::isfinite(prm->softmax_scale) && std::isfinite(prm->k_scale) &&
        std::isfinite(prm->v_scale)))
    return PA_ERR_INVALID_ARG;
  r->hq = prm->num_q_heads;
  r->hkv = prm->num_kv_heads;
  r->g = r->hq / r->hkv;
  r->d = prm->head_dim;
  r->P = prm->page_size;
  r->qd = qd;
  r->kvd = kvd;
  r->scale = prm->softmax_scale != 0.f ? prm->softmax_scale : 1.f / std::sqrt((float)r->d);
  r->k_scale = prm->k_scale != 0.f ? prm->k_scale : 1.f;
  r->v_scale = prm->v_scale != 0.f ? prm->v_scale : 1.f;
  r->max_dq = prm->max_decode_q ? prm->max_decode_q : 16;
  if (prm->verify_mode != PA_VERIFY_PACKED && prm->verify_mode != PA_VERIFY_TOKENWISE)
    return PA_ERR_INVALID_ARG;
  r->tokenwise = prm->verify_mode == PA_VERIFY_TOKENWISE;
  r->pf_auto = prm->prefill_kv_parts == PA_PREFILL_PARTS_AUTO;
  if (!r->pf_auto && (prm->prefill_kv_parts < 0 || prm->prefill_kv_parts > PF_MAX_PARTS))
    return PA_ERR_INVALID_ARG;
  r->pf_parts = r->pf_auto ? PF_AUTO_MAX : prm->prefill_kv_parts;
  r->pf_cut = 0;
  r->pf_min_units = PF_PART_UNITS;
  return PA_OK;
}

enum Entry { E_PREFILL, E_DECODE, E_MIXED };

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Part count for prefill_kv_parts = PA_PREFILL_PARTS_AUTO (1Cat-vLLM PR #1279,
// commit 5: the launcher picks the split count, up to 4, that finishes in the
// fewest full-CTA times on the device).  The work items' key counts are known
// from the host mirrors; for K = 1..4 the items are cut (equal runs of whole
// 128-key units, at least PF_AUTO_UNITS each) and the CTAs (one per item,
// part and KV head, one per SM) are handed out longest first to the earliest
// free SM, the way the work list is ordered and the hardware dispatches it;
// a CTA costs its 128-key units plus a fixed start-up.  The K with the
// earliest finish wins; a cut must beat K = 1 by 3 % (its merge costs too).
// Launches with four or more waves of CTAs, or with short items, are not cut.
int choose_parts(const std::vector<int>& k_ends, int hkv, int sms) {
  constexpr double START_UNITS = 2.0;
  const int64_t n1 = (int64_t)k_ends.size() * hkv;
  if (sms <= 0 || n1 == 0 || n1 >= 4LL * sms) return 1;
  int longest = 0;
  for (int k : k_ends) longest = std::max(longest, k);
  if (longest < 64 * PF_UNIT) return 1;
  double base = 0.0, best = 0.0;
  int best_k = 1;
  std::vector<double> cost;
  for (int K = 1; K <= PF_AUTO_MAX; ++K) {
    cost.clear();
    for (int k : k_ends) {
      int per = 0;
      const int parts = std::max(1, pf_part_count(k, K, PF_AUTO_UNITS, &per));
      const int n_u = (std::max(k, 0) + PF_UNIT - 1) / PF_UNIT;
      for (int c = 0; c < parts; ++c) {
        const int units = parts == 1 ? n_u : std::min(per, n_u - c * per);
        for (int h = 0; h < hkv; ++h) cost.push_back(units + START_UNITS);
      }
    }
    std::sort(cost.begin(), cost.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int s = 0; s < sms; ++s) free_at.push(0.0);
    double finish = 0.0;
    for (double c : cost) {
      const double t = free_at.top() + c;
      free_at.pop();
      free_at.push(t);
      finish = std::max(finish, t);
    }
    if (K == 1) {
      base = best = finish;
    } else if (finish < 0.97 * base && finish < best) {
      best = finish;
      best_k = K;
    }
  }
  return best_k;
}

pa_status validate(Entry entry, const pa_params* prm, const pa_batch* bat, const void* q,
                   const void* kc, const void* vc, void* out, void* ws, size_t ws_bytes,
                   Resolved* r) {
  pa_status s = resolve_params(prm, r);
  if (s != PA_OK) return s;
  if (entry == E_DECODE) r->pf_parts = 0;  // no prefill work: no part states
  if (!bat || bat->num_rows < 0 || bat->total_q < 0 || bat->num_pages < 0 ||
      bat->max_pages_per_row < 0)
    return PA_ERR_INVALID_ARG;
  if (!ws) return PA_ERR_INVALID_ARG;
  if (bat->num_rows > 0) {
    if (!bat->cu_seqlens_q || !bat->seq_lens || !bat->block_table) return PA_ERR_INVALID_ARG;
    if (bat->max_pages_per_row <= 0 || bat->num_pages <= 0) return PA_ERR_INVALID_ARG;
  }
  if (bat->total_q > 0 && (!q || !out)) return PA_ERR_INVALID_ARG;
  if (bat->num_rows > 0 && (!kc || !vc)) return PA_ERR_INVALID_ARG;
  if ((int64_t)bat->total_q * r->g > INT32_MAX / 2) return PA_ERR_INVALID_ARG;
  const WsLayout w =
      workspace_layout(bat->num_rows, bat->total_q, r->hq, r->d, r->max_dq, r->g, r->pf_parts,
                       r->by_len);
  if (ws_bytes < w.total) return PA_ERR_WORKSPACE_TOO_SMALL;

  const int64_t cache_tokens = (int64_t)bat->num_pages * r->P;
  r->tc2 = prefill_tc2_supported(r->qd, r->kvd, r->d, cache_tokens);
  r->tc = !r->tc2 && prefill_tc_supported(r->qd, r->kvd, r->d, cache_tokens);
  // one-token verify rows run on the TMA decode kernel only
  if (r->tokenwise && entry != E_PREFILL && !decode_tma_supported(r->qd, r->kvd, r->d, cache_tokens))
    return PA_ERR_UNSUPPORTED;
  // length-only split counts for long rows: the TMA decode kernel runs any
  // count; the long rows' parts go to the tcgen05 tile kernel where it is
  // built (d = 256, 16-bit q with a same-type cache)
  r->long_tc = false;
  r->split_cap = NSPLIT;
  if (r->by_len && entry != E_PREFILL) {
    if (r->tokenwise || !decode_tma_supported(r->qd, r->kvd, r->d, cache_tokens))
      return PA_ERR_UNSUPPORTED;
    r->long_tc = r->d == 256 && r->kvd == r->qd &&
                 prefill_tc_supported(r->qd, r->kvd, r->d, cache_tokens);
    // without host mirrors the decode kernel's split indices cover the most
    // parts a row can have (a tighter bound comes from the mirrors below)
    if (!r->long_tc) r->split_cap = NSPLIT_MAX;
  }
  r->pf_bm = r->tc2 ? PF_BM_TC2 : r->tc ? PF_BM_TC : (r->qd == PA_F32 ? 16 : PF_BM);
  // an explicit part count applies as given; a count chosen per call needs
  // the host mirrors (below)
  r->pf_cut = (r->tc2 || r->tc) && !r->pf_auto && r->pf_parts > 1 ? r->pf_parts : 0;
  r->host = bat->cu_seqlens_q_host && bat->seq_lens_host;
  r->host_max_q_dec = 0;
  r->host_tiles = 0;
  r->host_slots = 0;
  r->host_long = 0;
  r->host_short = 0;
  int host_cap = 1;  // most parts of a row on the decode kernel
  if (r->host) {
    const int32_t* cu = bat->cu_seqlens_q_host;
    const int32_t* lens = bat->seq_lens_host;
    if (bat->num_rows > 0 && cu[0] != 0) return PA_ERR_INVALID_ARG;
    if (cu[bat->num_rows] != bat->total_q) return PA_ERR_INVALID_ARG;
    const int bm = r->pf_bm;
    std::vector<int> k_ends;  // key count of every prefill work item
    for (int b = 0; b < bat->num_rows; ++b) {
      const int qb = cu[b + 1] - cu[b];
      const int L = lens[b];
      if (qb < 0 || L < 0) return PA_ERR_INVALID_ARG;
      if ((int64_t)L > (int64_t)bat->max_pages_per_row * r->P) return PA_ERR_INVALID_ARG;
      const bool dec = entry == E_DECODE || (entry == E_MIXED && qb >= 1 && qb <= r->max_dq);
      if (entry == E_DECODE && qb > r->max_dq) return PA_ERR_INVALID_ARG;
      if (dec) {
        r->host_max_q_dec = std::max(r->host_max_q_dec, qb);
        r->host_slots += qb;
        if (r->long_tc && qb >= 1 && dec_is_long(L, 1)) {
          r->host_long += dec_num_splits(L, 1) * ((qb * r->g + LONG_BM - 1) / LONG_BM);
        } else if (qb >= 1) {
          ++r->host_short;
          host_cap = std::max(host_cap, dec_num_splits(L, r->by_len));
        }
      } else if (qb > 0) {
        const int nmb = (qb * r->g + bm - 1) / bm;
        for (int m = 0; m < nmb; ++m) {
          const int r_last = std::min((m + 1) * bm, qb * r->g) - 1;
          k_ends.push_back(std::min(L, L - qb + r_last / r->g + 1));
        }
      }
    }
    if (r->by_len && !r->long_tc) r->split_cap = host_cap;
    // a part count chosen per call: only without decode rows, which run
    // beside the prefill on the same SMs and take a share the count cannot
    // see -- unless those rows' long splits run as short tile-kernel items
    // (PA_SPLITS_BY_LENGTH), where the decode rows take a small share
    if (r->pf_auto && (r->tc2 || r->tc) && entry != E_DECODE &&
        (r->host_slots == 0 || r->long_tc)) {
      const int K = choose_parts(k_ends, r->hkv, sm_count());
      r->pf_cut = K > 1 ? K : 0;
      r->pf_min_units = PF_AUTO_UNITS;
    }
    for (int k : k_ends) {
      int per;
      r->host_tiles +=
          r->pf_cut > 1 ? std::max(1, pf_part_count(k, r->pf_cut, r->pf_min_units, &per)) : 1;
    }
  }
  return check_device();
}

AttnArgs make_args(const Resolved& r, const pa_batch* bat, const void* q, const void* kc,
                   const void* vc, void* out, void* ws) {
  const WsLayout w =
      workspace_layout(bat->num_rows, bat->total_q, r.hq, r.d, r.max_dq, r.g, r.pf_parts, r.by_len);
  uint8_t* base = static_cast<uint8_t*>(ws);
  AttnArgs a{};
  a.p.cu_q = bat->cu_seqlens_q;
  a.p.seq_lens = bat->seq_lens;
  a.p.bt = bat->block_table;
  a.p.num_rows = bat->num_rows;
  a.p.total_q = bat->total_q;
  a.p.max_pages = bat->max_pages_per_row;
  a.p.num_pages = bat->num_pages;
  a.p.page_size = r.P;
  a.p.hq = r.hq;
  a.p.hkv = r.hkv;
  a.p.g = r.g;
  a.p.d = r.d;
  a.p.sl2 = r.scale * r.k_scale * 1.4426950408889634f;
  a.p.v_scale = r.v_scale;
  a.p.err = reinterpret_cast<uint32_t*>(base);
  a.q = q;
  a.kc = kc;
  a.vc = vc;
  a.out = out;
  a.part_acc = reinterpret_cast<float*>(base + w.part_acc);
  a.part_ml = reinterpret_cast<float2*>(base + w.part_ml);
  a.dec_base = nullptr;
  a.slot_tok = nullptr;
  a.row_order = nullptr;
  a.tiles = reinterpret_cast<const int2*>(base + w.tiles);
  a.n_tiles = &reinterpret_cast<const WsHeader*>(base)->n_tiles;
  a.max_decode_q = r.max_dq;
  a.max_slots = w.max_slots;
  a.tokenwise = r.tokenwise;
  a.n_slots = nullptr;
  a.pf_parts = r.pf_cut;
  a.pf_min_units = r.pf_min_units;
  a.pf_ml = reinterpret_cast<float2*>(base + w.pf_ml);
  a.pf_acc = reinterpret_cast<float*>(base + w.pf_acc);
  a.split_stride = w.split_stride;
  a.by_len = r.by_len;
  a.long_tc = r.long_tc ? 1 : 0;
  a.split_cap = r.split_cap;
  a.long_items = reinterpret_cast<const int2*>(base + w.long_items);
  a.n_long = &reinterpret_cast<const WsHeader*>(base)->n_long;
  a.max_long = w.max_long;
  return a;
}

int32_t* row_order_of(void* ws, const pa_batch* bat, const Resolved& r) {
  const WsLayout w =
      workspace_layout(bat->num_rows, bat->total_q, r.hq, r.d, r.max_dq, r.g, r.pf_parts, r.by_len);
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + w.row_order);
}

inline pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// A second stream (and two events) per host thread and device, made on first
// use and kept for the life of the thread: a mixed call runs its decode rows
// there, next to the prefill on the caller's stream.  Per thread, so that
// calls from different host threads never wait on each other's work; the
// objects are never destroyed (the driver reclaims them with the context).
struct AuxStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
};
AuxStream* aux_stream() {
  thread_local AuxStream aux[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  AuxStream& x = aux[dev];
  if (x.failed) return nullptr;
  if (!x.st) {
    if (cudaStreamCreateWithFlags(&x.st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) {
      x.failed = true;
      cudaGetLastError();
      return nullptr;
    }
  }
  return &x;
}

int decode_mblocks(const Resolved& r, int max_q) {
  // tokenwise verify rows: one token's g query rows per work item
  return ((r.tokenwise ? 1 : max_q) * r.g + DEC_ROWS - 1) / DEC_ROWS;
}

// Launches the decode CTAs and the merge for the rows routed to decode.
// The persistent decode kernel takes its items in row order; listing the rows
// with the longest splits first keeps the last items short, so fewer warps
// idle at the end.  Small batches skip the extra launch.
constexpr int ORDER_MIN_ROWS = 16;

cudaError_t run_decode(const AttnArgs& a0, const Resolved& r, int n_mblk, int n_slots,
                       int32_t* order, bool same_launch_ok, cudaStream_t st) {
  AttnArgs a = a0;
  a.dec_mblk = n_mblk;
  cudaError_t e = cudaSuccess;
  if (r.long_tc && (!r.host || r.host_long > 0)) {
    // rows longer than 32768 keys: the list of their (row, 128-row block,
    // split) items, then those splits on the tcgen05 tile kernel
    e = launch_long_items(a, const_cast<int2*>(a.long_items), a.max_long, st);
    if (e != cudaSuccess) return e;
    const int grid = r.host ? r.host_long * r.hkv : sm_count();
    e = launch_decode_long(a, r.qd, grid, st);
    if (e != cudaSuccess) return e;
  }
  if (r.long_tc && r.host && r.host_short == 0) {
    // every decode row was long: nothing for the decode kernel
  } else if (r.qd == PA_F32)
    e = launch_f32(a, 1, 0, n_mblk, st);
  else if (decode_tma_supported(r.qd, r.kvd, r.d, (int64_t)a.p.num_pages * a.p.page_size)) {
    if (!r.tokenwise && order && a.p.num_rows >= ORDER_MIN_ROWS &&
        a.p.num_rows <= MAX_ORDER_ROWS) {
      e = launch_row_order(a, order, st);
      if (e != cudaSuccess) return e;
      a.row_order = order;
    }
    // packed: work items range over rows; tokenwise: over decode slots
    const int units = r.tokenwise ? (int)std::min<int64_t>(a.p.total_q, a.max_slots)
                                  : a.p.num_rows;
    // the merge in the same launch: asked for, or (by default) when the
    // decode grid leaves SMs idle, so the second launch would cost more
    const int sms = sm_count();
    int merge_slots = 0;
    if (same_launch_ok && !r.by_len && r.merge_mode != PA_MERGE_SEPARATE) {
      const int64_t items = (int64_t)units * r.hkv * a.split_cap * n_mblk;
      if (r.merge_mode == PA_MERGE_SAME_LAUNCH ||
          decode_tma_grid(r.d, r.kvd == PA_E5M2, items, sms) < sms)
        merge_slots = n_slots;
    }
    e = launch_decode_tma(a, r.qd, r.kvd, n_mblk, units, merge_slots, sms, st);
    if (e == cudaSuccess && merge_slots > 0) return e;
  } else
    e = launch_decode_mma(a, r.qd, r.kvd, n_mblk, st);
  if (e != cudaSuccess) return e;
  return launch_merge(a, r.qd, n_slots, st);
}

// The prefill kernel over the work list, then (when work items were cut into
// key-range parts) the merge of the parts.
cudaError_t run_prefill(const AttnArgs& a, const Resolved& r, int grid_tiles, int mixed,
                        cudaStream_t st) {
  if (r.qd == PA_F32) return launch_f32(a, 0, grid_tiles, 0, st);
  cudaError_t e;
  if (r.tc2)
    e = launch_prefill_tc2(a, r.qd, r.kvd, grid_tiles, st);
  else if (r.tc)
    e = launch_prefill_tc(a, r.qd, r.kvd, grid_tiles, st);
  else
    return launch_prefill_mma(a, r.qd, r.kvd, grid_tiles, st);
  if (e != cudaSuccess || grid_tiles == 0) return e;
  return launch_pf_merge(a, r.qd, r.pf_bm, mixed, st);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

size_t paged_attn_workspace_size(const pa_params* params, int32_t num_rows, int32_t total_q) {
  Resolved r;
  if (resolve_params(params, &r) != PA_OK || num_rows < 0 || total_q < 0) return 0;
  return workspace_layout(num_rows, total_q, r.hq, r.d, r.max_dq, r.g, r.pf_parts, r.by_len).total;
}

pa_status paged_attn_prefill(const pa_params* params, const pa_batch* batch, const void* q,
                             const void* k_cache, const void* v_cache, void* out,
                             void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  Resolved r;
  pa_status s = validate(E_PREFILL, params, batch, q, k_cache, v_cache, out, workspace,
                         workspace_bytes, &r);
  if (s != PA_OK) return s;
  if (batch->num_rows == 0 || batch->total_q == 0) return PA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = make_args(r, batch, q, k_cache, v_cache, out, workspace);
  const int bm = r.pf_bm;
  const int max_tiles =
      (int)max_tiles_for(batch->num_rows, batch->total_q, r.g, bm, r.pf_cut);
  cudaError_t e = launch_plan(a, 0, 0, bm, max_tiles, st);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  const int grid = r.host ? r.host_tiles : max_tiles;
  return cuda_status(run_prefill(a, r, grid, 0, st));
}

pa_status paged_attn_decode(const pa_params* params, const pa_batch* batch, const void* q,
                            const void* k_cache, const void* v_cache, void* out,
                            void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  Resolved r;
  pa_status s = validate(E_DECODE, params, batch, q, k_cache, v_cache, out, workspace,
                         workspace_bytes, &r);
  if (s != PA_OK) return s;
  if (batch->num_rows == 0 || batch->total_q == 0) return PA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = make_args(r, batch, q, k_cache, v_cache, out, workspace);
  const int max_q = r.host ? r.host_max_q_dec : r.max_dq;
  const int n_slots = (int)std::min<int64_t>(batch->total_q, a.max_slots);
  return cuda_status(run_decode(a, r, decode_mblocks(r, max_q), n_slots,
                                row_order_of(workspace, batch, r), true, st));
}

pa_status paged_attn_mixed(const pa_params* params, const pa_batch* batch, const void* q,
                           const void* k_cache, const void* v_cache, void* out,
                           void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  Resolved r;
  pa_status s = validate(E_MIXED, params, batch, q, k_cache, v_cache, out, workspace,
                         workspace_bytes, &r);
  if (s != PA_OK) return s;
  if (batch->num_rows == 0 || batch->total_q == 0) return PA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = make_args(r, batch, q, k_cache, v_cache, out, workspace);
  const WsLayout w = workspace_layout(batch->num_rows, batch->total_q, r.hq, r.d, r.max_dq, r.g,
                                     r.pf_parts, r.by_len);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  a.dec_base = reinterpret_cast<const int32_t*>(base + w.dec_base);
  a.slot_tok = reinterpret_cast<const int32_t*>(base + w.slot_tok);
  a.n_slots = &reinterpret_cast<const WsHeader*>(base)->n_slots;
  const int bm = r.pf_bm;
  const int max_tiles =
      (int)max_tiles_for(batch->num_rows, batch->total_q, r.g, bm, r.pf_cut);
  cudaError_t e = launch_plan(a, 1, r.max_dq, bm, max_tiles, st);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  // decode rows: the grid covers every row; rows routed to prefill exit at once
  const int max_q = r.host ? r.host_max_q_dec : r.max_dq;
  const int n_slots = r.host ? r.host_slots : (int)a.max_slots;
  const int grid = r.host ? r.host_tiles : max_tiles;
  // With both kinds of rows, the decode rows run on a second stream next to
  // the prefill (they touch disjoint output rows and workspace regions): the
  // decode kernel takes as many SMs as it has work for, the prefill CTAs the
  // rest.  Fork after the plan, join before the call returns.
  AuxStream* aux = (max_q > 0 && grid > 0) ? aux_stream() : nullptr;
  cudaStream_t dst = st;
  if (aux) {
    if (cudaEventRecord(aux->fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(aux->st, aux->fork, 0) != cudaSuccess)
      return PA_ERR_CUDA;
    dst = aux->st;
  }
  // the prefill grid is submitted first, so its CTAs take the SMs and the
  // decode rows' CTAs fill the SMs its last wave leaves idle
  e = run_prefill(a, r, grid, 1, st);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (max_q > 0) {
    e = run_decode(a, r, decode_mblocks(r, max_q), n_slots, row_order_of(workspace, batch, r),
                   false, dst);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  if (aux && cudaEventRecord(aux->join, aux->st) != cudaSuccess) return PA_ERR_CUDA;
  if (aux && cudaStreamWaitEvent(st, aux->join, 0) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status paged_attn_read_errors(void* workspace, pa_stream_t stream, uint32_t* flags) {
  if (!flags) return PA_ERR_INVALID_ARG;
  if (!workspace) {
    // the error word of the array paged_attn_decode_static uses
    pa_status s = static_scratch_address(&workspace);
    if (s != PA_OK) return s;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, 4, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  *flags = v;
  return PA_OK;
}

const char* paged_attn_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported head_dim or dtype combination";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_NO_DEVICE: return "no sm_103 device is current";
  }
  return "unknown status";
}

int32_t paged_attn_version(void) { return 200; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Split-KV decode for callers that cannot allocate device memory.
//
// The decode path needs scratch memory (the partial softmax states and a
// small header).  Callers that cannot hand the library a workspace -- a
// plugin running inside a program that has already reserved all device
// memory for its own pool, or a plain C host that must keep its device
// memory use fixed after start-up and has no allocator to own a buffer's
// lifetime -- use paged_attn_decode_static instead.  Its scratch is this
// file-scope device array: every GPU that loads the library holds it until
// the process exits, and no call allocates or frees anything.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// The current CUDA context's unique id (0 if none is current).  Looked up
// through the driver entry points the runtime hands out, so the library links
// no driver library.  Neither call allocates or touches a stream.
unsigned long long current_context_id() {
  using GetCur = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCur get_cur = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault,
                                            &q) == cudaSuccess && q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetCur>(f) : nullptr;
  }();
  static GetId get_id = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                       cudaSuccess && q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<GetId>(f) : nullptr;
  }();
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

std::mutex g_static_mu;
struct StaticAddr {
  unsigned long long ctx = 0;  // context the address belongs to
  void* addr = nullptr;
};
StaticAddr g_static_addr[64];  // per device

// The array's device address in the current context (with that device
// current).  In host code the array's name is only a host-side stand-in, so
// the kernels must be given this address.  It is looked up once per context:
// a context torn down and made again (cudaDeviceReset) gets a new id, and the
// address is looked up afresh, since the module may then sit elsewhere.
pa_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_NO_DEVICE;
  if (dev < 0 || dev >= 64) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticAddr& e = g_static_addr[dev];
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || ctx != e.ctx || !e.addr) {
    void* p = nullptr;
    // makes the device's primary context current if no context is yet
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    const unsigned long long now = current_context_id();
    if (now == 0) return PA_ERR_CUDA;
    e.ctx = now;
    e.addr = p;
  }
  *out = e.addr;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status paged_attn_decode_static(const pa_params* params, const pa_batch* batch,
                                              const void* q, const void* k_cache,
                                              const void* v_cache, void* out,
                                              pa_stream_t stream) {
  using namespace pa;
  Resolved r;
  // size check against the fixed array (any non-null stand-in for the
  // workspace pointer: the address is only looked up below)
  pa_status s = validate(E_DECODE, params, batch, q, k_cache, v_cache, out,
                         reinterpret_cast<void*>(uintptr_t(1)), PA_STATIC_SCRATCH_BYTES, &r);
  if (s != PA_OK) return s;
  if (batch->num_rows == 0 || batch->total_q == 0) return PA_OK;
  void* ws = nullptr;
  s = static_scratch_address(&ws);
  if (s != PA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents; the header's work counts
  // and the decode kernel's work counter must start at zero.  The error word
  // (the first 4 bytes) is left as it is: it is sticky, like a workspace's,
  // and paged_attn_read_errors(NULL, ...) reads and clears it.
  if (cudaMemsetAsync(static_cast<uint8_t*>(ws) + 4, 0, sizeof(WsHeader) - 4, st) != cudaSuccess)
    return PA_ERR_CUDA;
  AttnArgs a = make_args(r, batch, q, k_cache, v_cache, out, ws);
  const int max_q = r.host ? r.host_max_q_dec : r.max_dq;
  const int n_slots = (int)std::min<int64_t>(batch->total_q, a.max_slots);
  return cuda_status(
      run_decode(a, r, decode_mblocks(r, max_q), n_slots, row_order_of(ws, batch, r), true, st));
}
