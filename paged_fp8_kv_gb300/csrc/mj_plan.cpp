// Host plan: occupancy-pinned split-KV work list.
//
// Source: the "mjolnir/t5_decode.py" page, `plan_split_kv` and `SplitPlan`
// (host helpers section).  The plan is pure integer code; it makes no CUDA
// call, so it can run on any host thread while the GPU works.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <queue>
#include <cstring>
#include <vector>

#include "mj_internal.h"

namespace mj {

bool verbose() {
  static const bool on = [] {
    const char* v = std::getenv("MJ_VERBOSE");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

mj_status check_params(const mj_decode_params* p) {
  if (!p) return MJ_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || p->q_len < 1 || p->h_k < 1 || p->h_r < 1) return MJ_ERR_INVALID_ARG;
  if (p->max_blocks < 1 || p->num_pages < 1) return MJ_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return MJ_ERR_INVALID_ARG;
  if (p->max_splits < 1 || p->max_splits > kMaxSplits) return MJ_ERR_INVALID_ARG;
  if (p->head_dim != kHeadDim) return MJ_ERR_UNSUPPORTED;
  if (p->page_size != 16 && p->page_size != 32 && p->page_size != 64 && p->page_size != 128)
    return MJ_ERR_UNSUPPORTED;
  if (p->q_dtype != MJ_BF16 && p->q_dtype != MJ_E4M3) return MJ_ERR_UNSUPPORTED;
  if (p->kernel < MJ_KERNEL_AUTO || p->kernel > MJ_KERNEL_TENSOR_CORE_QROWS) return MJ_ERR_INVALID_ARG;
  if (p->l2_prefetch < -1 || p->l2_prefetch > 8) return MJ_ERR_INVALID_ARG;
  if (p->kv_evict_first < -1 || p->kv_evict_first > 1) return MJ_ERR_INVALID_ARG;
  if (p->kv_format < MJ_KV_E4M3 || p->kv_format > MJ_KV_NVFP4) return MJ_ERR_INVALID_ARG;
  // nvfp4: converted to e4m3 in the swap-AB kernel, for e4m3 Q (the page's
  // fp8-Q path) and up to 32 packed rows
  if (p->kv_format == MJ_KV_NVFP4 &&
      (p->q_dtype != MJ_E4M3 || static_cast<int64_t>(p->q_len) * p->h_r > 32 ||
       (p->kernel != MJ_KERNEL_AUTO && p->kernel != MJ_KERNEL_TENSOR_CORE)))
    return MJ_ERR_UNSUPPORTED;
  // narrow pools: the tensor-core kernels only (the MMA reads the codes)
  if (p->kv_format != MJ_KV_E4M3 && p->kernel != MJ_KERNEL_AUTO && p->kernel != MJ_KERNEL_TENSOR_CORE &&
      p->kernel != MJ_KERNEL_TENSOR_CORE_QROWS)
    return MJ_ERR_UNSUPPORTED;
  // int32 index ranges used by the kernels
  const int64_t n_q = static_cast<int64_t>(p->q_len) * p->h_r;
  if (n_q > 4096 || static_cast<int64_t>(p->num_seqs) * p->h_k * n_q > (int64_t{1} << 30))
    return MJ_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->max_blocks) * p->page_size > (int64_t{1} << 30)) return MJ_ERR_UNSUPPORTED;
  if (p->kernel == MJ_KERNEL_TENSOR_CORE_GROUPED) {
    int g, rh;
    if (!tcg_supported(p->h_k, static_cast<int>(n_q), &g, &rh)) return MJ_ERR_UNSUPPORTED;
  }
  return MJ_OK;
}

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Plan model constants (GB300, measured): K+V bytes of one 128-row tile of
// one kv head; sustained KV bandwidth of the per-head kernels; time per tile
// of one CTA while the SM's other slots stream too (one SM streams a tile
// in about 0.65 us, shared by its co-resident CTAs; the query-rows kernel
// owns its SM and takes 0.9 us a tile); the per-CTA start cost in tiles; the
// merge kernel's share of a step (launched as a programmatic dependent);
// the margin a finer plan must win by.
constexpr double kTilePairBytes = 128.0 * 256.0;
constexpr double kPlanBandwidth = 5.45e6;  // bytes per microsecond
constexpr double kPlanSmTileUs = 0.65;
constexpr double kPlanQRowsTileUs = 0.9;
constexpr int64_t kPlanCtaOverheadTiles = 1;
constexpr double kPlanMergeUs = 2.5;
constexpr double kPlanMargin = 0.95;
// Finer plans tried: the co-resident CTAs times these thirds (3, 5, 8 and
// 12 slots per SM for three co-resident CTAs).
constexpr int kPlanThirds[] = {3, 5, 8, 12};
constexpr int64_t kPlanModelMaxUnits = 1 << 16;

struct Item {
  int32_t seq, begin, end, slot;
};

// Longest-first greedy schedule of `units` copies of every cost (sorted
// descending, plus `overhead` each) on n_slots slots, each copy to a least
// loaded slot; returns the largest slot load.  The least load never
// decreases along such a schedule (a least loaded slot only grows), so a
// histogram of slot loads with a moving minimum gives the same loads as a
// heap in time linear in the copies and the loads.
int64_t greedy_makespan(const std::vector<int64_t>& costs, int64_t units, int64_t n_slots, int64_t overhead) {
  if (costs.empty() || n_slots < 1) return 0;
  int64_t total = 0;
  for (int64_t c : costs) total += (c + overhead) * units;
  const int64_t bound = total / n_slots + costs.front() + overhead + 1;  // > every slot load
  int64_t makespan = 0;
  if (bound <= (int64_t{1} << 22)) {
    std::vector<int64_t> count(static_cast<size_t>(bound) + 1, 0);  // slots per load
    count[0] = n_slots;
    int64_t lo = 0;  // the least load
    for (int64_t c : costs)
      for (int64_t u = 0; u < units; ++u) {
        while (count[lo] == 0) ++lo;
        const int64_t t = lo + c + overhead;
        --count[lo];
        ++count[t];
        makespan = std::max(makespan, t);
      }
    return makespan;
  }
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> load;
  for (int64_t i = 0; i < n_slots; ++i) load.push(0);
  for (int64_t c : costs)
    for (int64_t u = 0; u < units; ++u) {
      const int64_t t = load.top() + c + overhead;
      load.pop();
      load.push(t);
      makespan = std::max(makespan, t);
    }
  return makespan;
}

}  // namespace

}  // namespace mj

extern "C" mj_status mj_decode_plan(const mj_decode_params* params, mj_plan_opts* opts,
                                    const int32_t* seq_lens_host, int32_t* work_out,
                                    int32_t work_cap, int32_t* num_work, int32_t* n_splits_out,
                                    int32_t* chunk_tiles) {
  using namespace mj;
  mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!opts || !seq_lens_host || !work_out || !num_work || !n_splits_out || work_cap < 1)
    return MJ_ERR_INVALID_ARG;
  if (opts->sm_count < 0 || opts->ctas_per_sm < 0 || opts->n_q_tiles < 0 || opts->force_splits < 0 ||
      opts->min_chunk_tiles < 0 || opts->pad_to < 0)
    return MJ_ERR_INVALID_ARG;

  const KernelChoice kc = choose_kernel(*params);
  const bool default_cps = opts->ctas_per_sm == 0;
  if (opts->sm_count == 0) opts->sm_count = kDefaultSmCount;
  if (opts->ctas_per_sm == 0) opts->ctas_per_sm = kc.ctas_per_sm;
  if (opts->n_q_tiles == 0) opts->n_q_tiles = kc.n_q_tiles;
  if (opts->min_chunk_tiles == 0) opts->min_chunk_tiles = 1;

  const int b = params->num_seqs;
  const int64_t max_len = static_cast<int64_t>(params->max_blocks) * params->page_size;
  std::vector<int64_t> tiles(b);
  int64_t longest = 0;
  for (int i = 0; i < b; ++i) {
    const int64_t L = seq_lens_host[i];
    if (L < 0 || L > max_len) return MJ_ERR_INVALID_ARG;
    tiles[i] = std::max<int64_t>(1, ceil_div(L, kTileRows));
    longest = std::max(longest, tiles[i]);
  }

  const int64_t floor_chunk =
      std::max<int64_t>(opts->min_chunk_tiles, ceil_div(longest, params->max_splits));

  auto total_chunks = [&](int64_t chunk) {
    int64_t s = 0;
    for (int64_t t : tiles) s += ceil_div(t, chunk);
    return s;
  };

  // The occupancy-pinned chunk for `ctas_per_sm` (co-resident (CTA, kv
  // head) pairs per SM): the smallest chunk whose chunks fill one wave.
  auto chunk_for = [&](int64_t ctas_per_sm) -> int64_t {
    const int64_t per_wave = static_cast<int64_t>(opts->sm_count) * ctas_per_sm;
    const int64_t slots =
        std::max<int64_t>(1, per_wave / (static_cast<int64_t>(params->h_k) * opts->n_q_tiles));
    if (opts->force_splits > 0) return std::max(floor_chunk, ceil_div(longest, opts->force_splits));
    if (b >= slots || params->max_splits == 1) return longest;
    // total_chunks() is non-increasing in chunk
    int64_t lo = floor_chunk, hi = std::max(floor_chunk, longest);
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (total_chunks(mid) <= slots)
        hi = mid;
      else
        lo = mid + 1;
    }
    return lo;
  };

  // Library default for the per-head kernels: the plan for 1, 5/3, 8/3 or
  // 4 times the co-resident CTAs, whichever a simple model says ends first.
  // One wave of the occupancy-pinned plan leaves SMs idle behind the
  // longest chunk when a few long sequences dominate; a finer plan balances
  // (the hardware hands the next CTA to the first free slot) but may add a
  // merge.  Model: time = max(bytes / bandwidth, longest slot of a greedy
  // longest-first assignment x time per tile of a CTA) + the merge.
  // (Measured on the GQA decode workload, 64 sequences of 512-8192 keys,
  // 8 kv heads, with a two-stage instance at three CTAs per SM: 3, 4, 5, 6,
  // 8, 12 slots per SM gave 124.9, 122.9, 116.7, 124.9, 120.8, 120.8 us per
  // step and the model picked 5.)
  if (default_cps && opts->force_splits == 0 && params->max_splits > 1 &&
      kc.kind != KernelKind::kTensorCoreGrouped) {
    const int64_t units_per_item = static_cast<int64_t>(params->h_k) * opts->n_q_tiles;
    const int64_t n_slots = static_cast<int64_t>(opts->sm_count) * kc.ctas_per_sm;
    int64_t sum_tiles = 0;
    for (int64_t t : tiles) sum_tiles += t;
    const double stream_us = static_cast<double>(sum_tiles) * units_per_item * kTilePairBytes / kPlanBandwidth;
    // (a CTA of paired q tiles does twice the work per tile)
    const double tile_us = kc.kind == KernelKind::kTensorCoreQRows
                               ? kPlanQRowsTileUs * (kc.rows_per_cta > 128 ? 2 : 1)
                               : kPlanSmTileUs * kc.ctas_per_sm;
    double best = 0;
    int64_t best_cps = kc.ctas_per_sm, prev_cps = 0;
    for (int thirds : kPlanThirds) {
      const int64_t cps = (static_cast<int64_t>(kc.ctas_per_sm) * thirds + 2) / 3;
      if (cps == prev_cps) continue;
      prev_cps = cps;
      const int64_t chunk = chunk_for(cps);
      std::vector<int64_t> costs;
      for (int64_t t : tiles)
        for (int64_t beg = 0; beg < t; beg += chunk) costs.push_back(std::min(chunk, t - beg));
      if (static_cast<int64_t>(costs.size()) * units_per_item > kPlanModelMaxUnits) break;  // keep the plan cheap
      std::stable_sort(costs.begin(), costs.end(), [](int64_t x, int64_t y) { return x > y; });
      const int64_t makespan = greedy_makespan(costs, units_per_item, n_slots, kPlanCtaOverheadTiles);
      const bool splits = static_cast<int64_t>(costs.size()) > b;
      const double est = std::max(stream_us, makespan * tile_us) + (splits ? kPlanMergeUs : 0.0);
      if (thirds == 3 || est < best * kPlanMargin) {
        best = est;
        best_cps = cps;
      }
    }
    opts->ctas_per_sm = static_cast<int32_t>(best_cps);
  }

  const int64_t chunk = chunk_for(opts->ctas_per_sm);
  std::vector<Item> items;
  items.reserve(static_cast<size_t>(total_chunks(chunk)));
  for (int i = 0; i < b; ++i) {
    const int64_t k = ceil_div(tiles[i], chunk);
    if (k > params->max_splits) return MJ_ERR_INVALID_ARG;  // force_splits beyond max_splits
    n_splits_out[i] = static_cast<int32_t>(k);
    for (int64_t s = 0; s < k; ++s) {
      const int64_t beg = s * chunk;
      const int64_t end = std::min(tiles[i], beg + chunk);
      items.push_back({i, static_cast<int32_t>(beg), static_cast<int32_t>(end), static_cast<int32_t>(s)});
    }
  }
  std::stable_sort(items.begin(), items.end(), [](const Item& x, const Item& y) {
    return (x.end - x.begin) > (y.end - y.begin);
  });
  const int64_t n_items = static_cast<int64_t>(items.size());
  if (opts->pad_to > 0 && opts->pad_to < n_items) return MJ_ERR_INVALID_ARG;
  const int64_t n_out = opts->pad_to > 0 ? opts->pad_to : n_items;
  if (n_out > work_cap) return MJ_ERR_CAPACITY;
  for (int64_t i = 0; i < n_out; ++i) {
    const Item it = i < n_items ? items[i] : Item{0, 0, 0, 0};
    work_out[4 * i + 0] = it.seq;
    work_out[4 * i + 1] = it.begin;
    work_out[4 * i + 2] = it.end;
    work_out[4 * i + 3] = it.slot;
  }
  *num_work = static_cast<int32_t>(n_out);
  if (chunk_tiles) *chunk_tiles = static_cast<int32_t>(chunk);
  if (verbose()) {
    // a summary in the spirit of the page's SplitPlan repr: the options the
    // rule ran with, the chunk it chose and how the sequences were cut
    int64_t split_seqs = 0, max_k = 0, sum_tiles = 0;
    for (int i = 0; i < b; ++i) {
      split_seqs += n_splits_out[i] > 1;
      max_k = std::max<int64_t>(max_k, n_splits_out[i]);
      sum_tiles += tiles[i];
    }
    const int64_t slots = std::max<int64_t>(
        1, static_cast<int64_t>(opts->sm_count) * opts->ctas_per_sm / (static_cast<int64_t>(params->h_k) * opts->n_q_tiles));
    std::fprintf(stderr,
                 "mj_decode_plan: SplitPlan(kernel=%s, num_seqs=%d, h_k=%d, n_q=%d, sm_count=%d, ctas_per_sm=%d%s, "
                 "n_q_tiles=%d, slots=%lld, max_splits=%d, force_splits=%d, chunk_tiles=%lld, tiles=%lld "
                 "(longest %lld), work_items=%lld, padding=%lld, split_seqs=%lld, max_n_splits=%lld)\n",
                 kc.name, b, params->h_k, params->q_len * params->h_r, opts->sm_count, opts->ctas_per_sm,
                 default_cps ? " (library choice)" : "", opts->n_q_tiles, static_cast<long long>(slots),
                 params->max_splits, opts->force_splits, static_cast<long long>(chunk),
                 static_cast<long long>(sum_tiles), static_cast<long long>(longest), static_cast<long long>(n_items),
                 static_cast<long long>(n_out - n_items), static_cast<long long>(split_seqs),
                 static_cast<long long>(max_k));
  }
  return MJ_OK;
}

extern "C" mj_status mj_check_preconditions(const mj_decode_params* params, const int32_t* block_table_host,
                                            const int32_t* seq_lens_host, const float* q_descale,
                                            const float* k_descale, const float* v_descale, int64_t qd_seq,
                                            int64_t qd_head, int64_t kd_seq, int64_t kd_head, int64_t vd_seq,
                                            int64_t vd_head, int32_t* bad_seq) {
  using namespace mj;
  if (bad_seq) *bad_seq = -1;
  const mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!block_table_host || !seq_lens_host || !q_descale || !k_descale || !v_descale) return MJ_ERR_INVALID_ARG;
  const int64_t strides[6] = {qd_seq, qd_head, kd_seq, kd_head, vd_seq, vd_head};
  for (int64_t s : strides)
    if (s < 0) return MJ_ERR_INVALID_ARG;
  const mj_decode_params& p = *params;
  const int64_t max_len = static_cast<int64_t>(p.max_blocks) * p.page_size;
  for (int b = 0; b < p.num_seqs; ++b) {
    bool ok = true;
    const int64_t L = seq_lens_host[b];
    if (L < 0 || L > max_len) ok = false;
    // pages below ceil(L / page_size) are read; later entries may hold anything
    const int64_t pages = ok ? (L + p.page_size - 1) / p.page_size : 0;
    for (int64_t j = 0; ok && j < pages; ++j) {
      const int32_t pg = block_table_host[static_cast<int64_t>(b) * p.max_blocks + j];
      if (pg < 0 || pg >= p.num_pages) ok = false;
    }
    // the kernels take the raw-score maximum and then scale: every descale
    // must be finite and positive
    for (int g = 0; ok && g < p.h_k; ++g) {
      const float d[3] = {q_descale[b * qd_seq + g * qd_head], k_descale[b * kd_seq + g * kd_head],
                          v_descale[b * vd_seq + g * vd_head]};
      for (float x : d)
        if (!std::isfinite(x) || !(x > 0.f)) ok = false;
    }
    if (!ok) {
      if (bad_seq) *bad_seq = b;
      return MJ_ERR_INVALID_ARG;
    }
  }
  return MJ_OK;
}
