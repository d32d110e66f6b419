// Split planner: turns sequence lengths into the work list of the partial
// kernel.  Host only, integer arithmetic only, deterministic.
//
// The KV range of each sequence is cut into page ranges, one CTA each
// ("vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower", section
// "What SplitKV is trying to do"), and every launched CTA owns real work --
// the invariant whose loss that page dissects in "The actual bug is one
// missing constructor argument".  How many splits to use trades parallelism
// against the merge: "Shipped: 484.5 tok/s on one GB300 ...", section "Why 8
// splits lost", saw the extra combine work eat a faster split kernel, so the
// automatic choice below charges every split a merge cost.
#include <algorithm>
#include <functional>
#include <queue>

#include "internal.h"

namespace splitkv {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Splits per sequence for one chunk size (pages per split), n_b / chunk
// rounded up or down, clamped to [1, min(n_b, kMaxSplits)].
std::vector<int32_t> splits_for_chunk(const std::vector<int32_t>& n_pages, int64_t chunk,
                                      bool round_up) {
  std::vector<int32_t> S(n_pages.size());
  for (size_t b = 0; b < n_pages.size(); ++b) {
    const int64_t n = n_pages[b];
    if (n <= 0) {
      S[b] = 1;
      continue;
    }
    int64_t s = round_up ? ceil_div(n, chunk) : n / chunk;
    s = std::min<int64_t>(s, std::min<int64_t>(n, kMaxSplits));
    S[b] = static_cast<int32_t>(std::max<int64_t>(s, 1));
  }
  return S;
}

// Largest machine load when `costs` are list-scheduled largest first onto
// `machines` identical machines (each item goes to the least-loaded one).
int64_t lpt_makespan(std::vector<int64_t> costs, int machines) {
  std::sort(costs.begin(), costs.end(), std::greater<int64_t>());
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> loads;
  for (int i = 0; i < machines; ++i) loads.push(0);
  int64_t worst = 0;
  for (int64_t c : costs) {
    int64_t l = loads.top() + c;
    loads.pop();
    loads.push(l);
    worst = std::max(worst, l);
  }
  return worst;
}

// Page range of split s out of S over n pages: [floor(s*n/S), floor((s+1)*n/S)).
inline int32_t split_edge(int64_t s, int64_t n, int64_t S) {
  return static_cast<int32_t>((s * n) / S);
}

// Automatic choice: one chunk size for the whole batch, scored by the
// makespan of its items on the machine's work-item slots plus a per-split
// merge charge.  `slots` = items that run at once; a split is `units` items
// of `hpi` KV heads each.
std::vector<int32_t> choose_splits(const std::vector<int32_t>& n_pages, int units, int hpi,
                                   int slots) {
  int64_t total = 0, nmax = 1;
  for (int32_t n : n_pages) {
    total += n;
    nmax = std::max<int64_t>(nmax, n);
  }
  total *= units;
  std::vector<std::pair<int64_t, bool>> cands;
  for (int k = 1; k <= kMaxWaves; ++k) {
    const int64_t c = std::max<int64_t>(1, ceil_div(total, int64_t(k) * slots));
    cands.push_back({c, true});
    cands.push_back({c, false});
  }
  cands.push_back({nmax, true});

  std::vector<int32_t> best_S;
  int64_t best = -1;
  for (const auto& cand : cands) {
    std::vector<int32_t> S = splits_for_chunk(n_pages, cand.first, cand.second);
    std::vector<int64_t> costs;
    int32_t smax = 1;
    for (size_t b = 0; b < n_pages.size(); ++b) {
      const int64_t n = n_pages[b];
      smax = std::max(smax, S[b]);
      if (n <= 0) {
        for (int u = 0; u < units; ++u) costs.push_back(kItemOverhead);
        continue;
      }
      for (int32_t s = 0; s < S[b]; ++s) {
        const int64_t pages = split_edge(s + 1, n, S[b]) - split_edge(s, n, S[b]);
        for (int u = 0; u < units; ++u) costs.push_back(16 * pages * hpi + kItemOverhead);
      }
    }
    const int64_t score = lpt_makespan(costs, slots) + int64_t(kCombineCost) * smax;
    if (best < 0 || score < best) {
      best = score;
      best_S = S;
    }
  }
  return best_S;
}

// Workspace layout of a plan, and the host image of its uploaded part.
void layout_workspace(splitkv_plan_s* p) {
  const splitkv_desc_t& d = p->desc;
  const int B = d.batch;
  p->rows = rows_per_item(d);
  p->n_ctas = p->n_items * ctas_per_item(d);
  // Everything before off_log is uploaded from the host.
  size_t off = 0;
  p->off_status = off;
  off = align_up(off + sizeof(int32_t));
  p->off_items = off;
  off = align_up(off + p->items.size() * sizeof(int32_t));
  p->off_groups = off;
  off = align_up(off + p->groups.size() * sizeof(int32_t));
  p->off_seqlens = off;
  off = align_up(off + size_t(B) * sizeof(int32_t));
  p->off_tickets = off;  // group tickets, then one bundle ticket per slot
  off = align_up(off + size_t(p->n_groups + p->n_slots) * sizeof(int32_t));
  p->upload_bytes = off;
  p->off_log = off;
  off = align_up(off + size_t(p->n_ctas) * kLogFields * sizeof(int32_t));
  p->off_lse = off;
  off = align_up(off + size_t(p->n_slots) * p->rows * sizeof(float));
  p->off_o = off;
  off = align_up(off + size_t(p->n_slots) * p->rows * d.v_dim * sizeof(float));
  p->total = off;

  p->upload.assign(p->upload_bytes, 0);
  auto put = [&](size_t at, const std::vector<int32_t>& v) {
    if (!v.empty()) std::copy(reinterpret_cast<const unsigned char*>(v.data()),
                              reinterpret_cast<const unsigned char*>(v.data() + v.size()),
                              p->upload.begin() + at);
  };
  put(p->off_items, p->items);
  put(p->off_groups, p->groups);
  put(p->off_seqlens, p->seq_lens);
}

}  // namespace

void build_plan(splitkv_plan_s* p) {
  const splitkv_desc_t& d = p->desc;
  const int B = d.batch, hkv = d.num_kv_heads, P = d.page_size;
  const int hpi = heads_per_item(d);  // an item covers KV heads [h0, h0 + hpi)
  std::vector<int32_t> n_pages(B);
  for (int b = 0; b < B; ++b) n_pages[b] = static_cast<int32_t>(ceil_div(p->seq_lens[b], P));

  std::vector<int32_t> S(B);
  if (p->num_splits > 0) {
    for (int b = 0; b < B; ++b) S[b] = n_pages[b] > 0 ? std::min(p->num_splits, n_pages[b]) : 1;
  } else {
    // An item that launches several CTAs takes that many of the resident slots.
    const int slots = std::max(1, p->num_sms * ctas_per_sm(d) / ctas_per_item(d));
    S = choose_splits(n_pages, hkv / hpi, hpi, slots);
  }

  // Combine groups and partial slots, in (b, h_kv) order.
  p->groups.clear();
  std::vector<int32_t> group_of(size_t(B) * hkv, -1), slot_of(size_t(B) * hkv, -1);
  int32_t slots = 0;
  for (int b = 0; b < B; ++b) {
    if (n_pages[b] <= 0 || S[b] <= 1) continue;
    for (int h = 0; h < hkv; h += hpi) {
      group_of[size_t(b) * hkv + h] = static_cast<int32_t>(p->groups.size() / kGroupFields);
      slot_of[size_t(b) * hkv + h] = slots;
      p->groups.insert(p->groups.end(), {b, h, S[b], slots});
      slots += S[b];
    }
  }
  p->n_groups = static_cast<int32_t>(p->groups.size() / kGroupFields);
  p->n_slots = slots;
  p->max_group_splits = 0;
  for (int32_t g = 0; g < p->n_groups; ++g)
    p->max_group_splits = std::max(p->max_group_splits, p->groups[size_t(g) * kGroupFields + 2]);

  struct Item {
    int32_t f[SPLITKV_ITEM_FIELDS];
  };
  std::vector<Item> items;
  for (int b = 0; b < B; ++b) {
    const int64_t n = n_pages[b];
    for (int h = 0; h < hkv; h += hpi) {
      const int32_t g = group_of[size_t(b) * hkv + h];
      const int32_t slot0 = slot_of[size_t(b) * hkv + h];
      if (n <= 0) {
        items.push_back({{b, h, 0, 1, 0, 0, -1, -1}});
        continue;
      }
      for (int32_t s = 0; s < S[b]; ++s) {
        items.push_back({{b, h, s, S[b], split_edge(s, n, S[b]), split_edge(s + 1, n, S[b]),
                          g >= 0 ? slot0 + s : -1, g}});
      }
    }
  }
  std::stable_sort(items.begin(), items.end(), [](const Item& x, const Item& y) {
    const int32_t lx = x.f[SPLITKV_ITEM_PAGE1] - x.f[SPLITKV_ITEM_PAGE0];
    const int32_t ly = y.f[SPLITKV_ITEM_PAGE1] - y.f[SPLITKV_ITEM_PAGE0];
    if (lx != ly) return lx > ly;
    for (int k : {SPLITKV_ITEM_B, SPLITKV_ITEM_HKV, SPLITKV_ITEM_SPLIT})
      if (x.f[k] != y.f[k]) return x.f[k] < y.f[k];
    return false;
  });
  p->n_items = static_cast<int32_t>(items.size());
  p->items.resize(items.size() * SPLITKV_ITEM_FIELDS);
  for (size_t i = 0; i < items.size(); ++i)
    std::copy(items[i].f, items[i].f + SPLITKV_ITEM_FIELDS, p->items.begin() + i * SPLITKV_ITEM_FIELDS);

  layout_workspace(p);
}

void build_fixed_plan(splitkv_plan_s* p) {
  const splitkv_desc_t& d = p->desc;
  const int B = d.batch, hpi = heads_per_item(d), U = d.num_kv_heads / hpi, S = p->num_splits;
  p->seq_lens.assign(B, 0);
  p->n_items = B * U * S;
  p->items.assign(size_t(p->n_items) * SPLITKV_ITEM_FIELDS, 0);
  p->groups.clear();
  for (int b = 0; b < B; ++b)
    for (int u = 0; u < U; ++u) {
      const int g = b * U + u;
      for (int s = 0; s < S; ++s) {
        int32_t* it = p->items.data() + size_t(g * S + s) * SPLITKV_ITEM_FIELDS;
        const int32_t f[SPLITKV_ITEM_FIELDS] = {b, u * hpi, s, 0, 0, 0, -1, -1};
        std::copy(f, f + SPLITKV_ITEM_FIELDS, it);
      }
      if (S > 1) p->groups.insert(p->groups.end(), {b, u * hpi, 0, g * S});
    }
  p->n_groups = static_cast<int32_t>(p->groups.size() / kGroupFields);
  p->n_slots = S > 1 ? p->n_items : 0;
  p->max_group_splits = S > 1 ? S : 0;  // the refresh kernel writes S_b <= S
  layout_workspace(p);
}

}  // namespace splitkv
