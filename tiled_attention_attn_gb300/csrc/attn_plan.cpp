// Host-side schedule for the persistent forward kernel; see attn_plan.h.
#include "attn_plan.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <limits>
#include <queue>
#include <utility>

#include "attn_params.h"

namespace attn {
namespace {

struct Pair {
  int bh, mb, kv_end, kl0, kl1;
  long cost;   // tile pairs (sub-tile x key tile) the block computes
};

struct Cand {
  int pair;      // index into pairs
  int a, e;      // key-tile range
  int split, n_split;
  double cost;
};

long piece_cost(const Pair& p, int a, int e) {
  const long c0 = std::max(0, std::min(e, p.kl0 + 1) - a);
  const long c1 = std::max(0, std::min(e, p.kl1 + 1) - a);
  return c0 + c1;
}

// Fixed per-unit cost in tile pairs (Q load, pipeline fill and drain,
// epilogue), the extra store of a split piece, the combine pass, and the
// lone tail of a causal block's last piece: its last key tile has only the
// second sub-tile active, so that tile's softmax -> P.V chain runs with no
// other sub-tile's MMAs beside it (per-CTA phase traces of the L = 8192,
// d = 128 causal forward: pieces ending on the diagonal take 1.4-2.9 us more
// than their tile count predicts, ~2.5 tile pairs).
struct CostModel {
  double unit, split_extra, combine, tail;
};

CostModel cost_model(int d) {
  if (d == 128) return {2.0, 1.0, 3.0, 2.5};
  return {4.0, 2.0, 6.0, 0.0};
}

double assign(std::vector<Cand>& units, int num_sms, std::vector<int>& cta_of, int& n_ctas) {
  std::stable_sort(units.begin(), units.end(), [](const Cand& x, const Cand& y) { return x.cost > y.cost; });
  n_ctas = std::max(1, std::min<int>(num_sms, static_cast<int>(units.size())));
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < n_ctas; ++c) heap.push({0.0, c});
  cta_of.assign(units.size(), 0);
  double makespan = 0.0;
  for (size_t i = 0; i < units.size(); ++i) {
    Slot s = heap.top();
    heap.pop();
    cta_of[i] = s.second;
    s.first += units[i].cost;
    makespan = std::max(makespan, s.first);
    heap.push(s);
  }
  return makespan;
}

void build_units(const std::vector<Pair>& pairs, double target, const CostModel& cm,
                 std::vector<Cand>& units, bool& any_split) {
  units.clear();
  any_split = false;
  for (size_t i = 0; i < pairs.size(); ++i) {
    const Pair& p = pairs[i];
    int n = 1;
    if (p.kv_end > 1 && static_cast<double>(p.cost) > target) {
      n = static_cast<int>(std::ceil(static_cast<double>(p.cost) / target));
      n = std::min(n, std::min(p.kv_end, kMaxSplits));
    }
    if (n > 1) any_split = true;
    const double tail = (p.kl0 != p.kl1) ? cm.tail : 0.0;
    // the last piece ends on the block's last key tile and carries the lone
    // tail: it starts where its cost comes closest to an equal share, and the
    // tiles before it are cut into n - 1 equal pieces
    int a_last = static_cast<int>(static_cast<long>(n - 1) * p.kv_end / n);
    if (n > 1 && tail > 0.0) {
      const double share = (static_cast<double>(piece_cost(p, 0, p.kv_end)) + tail) / n;
      double best_gap = std::numeric_limits<double>::infinity();
      for (int a = n - 1; a < p.kv_end; ++a) {
        const double gap = std::fabs(static_cast<double>(piece_cost(p, a, p.kv_end)) + tail - share);
        if (gap < best_gap) {
          best_gap = gap;
          a_last = a;
        }
      }
    }
    for (int s = 0; s < n; ++s) {
      const int a = (s == n - 1) ? a_last : static_cast<int>(static_cast<long>(s) * a_last / (n - 1));
      const int e = (s == n - 1) ? p.kv_end : static_cast<int>(static_cast<long>(s + 1) * a_last / (n - 1));
      const double c = static_cast<double>(piece_cost(p, a, e)) + cm.unit + (n > 1 ? cm.split_extra : 0.0) +
                       (e == p.kv_end ? tail : 0.0);
      units.push_back({static_cast<int>(i), a, e, s, n, c});
    }
  }
}

}  // namespace

bool make_plan(int B, int Hq, int Hkv, int Lq, int Lk, int d, bool causal, int num_sms, Plan& out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq <= 0 || Lk < 0 || num_sms <= 0) return false;
  if (d != 64 && d != 128) return false;
  const int group = Hq / Hkv;
  const int n_mb = (Lq + kBlockRows - 1) / kBlockRows;
  const long long n_pairs = static_cast<long long>(B) * Hq * n_mb;
  if (n_pairs > (1LL << 26) || static_cast<long long>(B) * Hq > std::numeric_limits<int>::max()) return false;

  // query blocks in (batch, KV head, block, query head in group) order, so the
  // query heads that share a KV head sit next to each other
  std::vector<Pair> pairs;
  pairs.reserve(static_cast<size_t>(n_pairs));
  long total = 0, max_cost = 0;
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < Hkv; ++g)
      for (int mb = 0; mb < n_mb; ++mb)
        for (int hh = 0; hh < group; ++hh) {
          const int h = g * group + hh;
          Pair p;
          p.bh = b * Hq + h;
          p.mb = mb;
          p.kl0 = kv_last_tile(mb * kBlockRows, 0, Lq, Lk, causal);
          p.kl1 = kv_last_tile(mb * kBlockRows, 1, Lq, Lk, causal);
          p.kv_end = std::max(p.kl0, p.kl1) + 1;
          p.cost = piece_cost(p, 0, p.kv_end);
          total += p.cost;
          max_cost = std::max(max_cost, p.cost);
          pairs.push_back(p);
        }

  const CostModel cm = cost_model(d);
  const double avg = (static_cast<double>(total) + cm.unit * static_cast<double>(pairs.size())) / num_sms;
  std::vector<double> targets = {std::numeric_limits<double>::infinity()};
  if (static_cast<double>(max_cost) > 0.75 * avg) {
    // piece sizes are whole key tiles, so the best target can sit anywhere:
    // a fine grid of fractions of the average CTA load
    for (double f = 0.25; f <= 3.0 + 1e-9; f += 0.03125)
      if (f * avg >= 1.0) targets.push_back(f * avg);
  }

  double best = std::numeric_limits<double>::infinity();
  std::vector<Cand> best_units;
  std::vector<int> best_cta;
  int best_ctas = 0;
  for (double tgt : targets) {
    std::vector<Cand> units;
    bool any_split = false;
    build_units(pairs, tgt, cm, units, any_split);
    std::vector<int> cta_of;
    int n_ctas = 0;
    double ms = assign(units, num_sms, cta_of, n_ctas);
    if (any_split) ms += cm.combine;
    if (ms < best - 1e-9 || (std::fabs(ms - best) <= 1e-9 && units.size() < best_units.size())) {
      best = ms;
      best_units = std::move(units);
      best_cta = std::move(cta_of);
      best_ctas = n_ctas;
    }
  }

  // workspace slots for split groups, in pair order
  std::vector<int> slot_base(pairs.size(), -1);
  out = Plan();
  int n_slots = 0;
  {
    std::vector<int> nsplit(pairs.size(), 1);
    for (const Cand& c : best_units) nsplit[c.pair] = c.n_split;
    for (size_t i = 0; i < pairs.size(); ++i)
      if (nsplit[i] > 1) {
        slot_base[i] = n_slots;
        out.groups.push_back({pairs[i].bh, pairs[i].mb, n_slots, nsplit[i]});
        n_slots += nsplit[i];
      }
  }

  // per-CTA lists, each in assignment order (longest first)
  out.n_ctas = best_ctas;
  out.n_partials = n_slots;
  out.makespan = best;
  std::vector<std::vector<int>> per_cta(best_ctas);
  for (size_t i = 0; i < best_units.size(); ++i) per_cta[best_cta[i]].push_back(static_cast<int>(i));
  out.cta_off.assign(best_ctas + 1, 0);
  out.units.reserve(best_units.size());
  for (int c = 0; c < best_ctas; ++c) {
    out.cta_off[c] = static_cast<int>(out.units.size());
    for (int i : per_cta[c]) {
      const Cand& u = best_units[i];
      const Pair& p = pairs[u.pair];
      const int slot = (u.n_split > 1) ? slot_base[u.pair] + u.split : -1;
      out.units.push_back({p.bh, p.mb, u.a, u.e, u.split, u.n_split, slot, c});
    }
  }
  out.cta_off[best_ctas] = static_cast<int>(out.units.size());
  return true;
}

// ---------------------------------------------------------------------------
// CTA-pair schedule: a unit is a 256-row query block (128 rows per CTA of the
// pair) against a range of 256-key tiles; both CTAs run the same tiles, so a
// unit's cost is its tile count plus a fixed cost per unit (query load,
// pipeline fill, epilogue) and, for split pieces, the partial write and the
// share of the merge.
// ---------------------------------------------------------------------------
namespace {

struct PairBlock {
  int bh, mb, n_tiles;
};

void build_pair_units(const std::vector<PairBlock>& blocks, double target, double c_unit, double c_split,
                      std::vector<Cand>& units, bool& any_split) {
  units.clear();
  any_split = false;
  for (size_t i = 0; i < blocks.size(); ++i) {
    const PairBlock& b = blocks[i];
    int n = 1;
    if (b.n_tiles > 1 && static_cast<double>(b.n_tiles) > target) {
      n = static_cast<int>(std::ceil(static_cast<double>(b.n_tiles) / target));
      n = std::min(n, std::min(b.n_tiles, kMaxSplits));
    }
    if (n > 1) any_split = true;
    for (int s = 0; s < n; ++s) {
      const int a = static_cast<int>(static_cast<long>(s) * b.n_tiles / n);
      const int e = static_cast<int>(static_cast<long>(s + 1) * b.n_tiles / n);
      units.push_back({static_cast<int>(i), a, e, s, n, (e - a) + c_unit + (n > 1 ? c_split : 0.0)});
    }
  }
}

}  // namespace

bool make_plan_pair(int B, int Hq, int Hkv, int Lq, int Lk, bool causal, int num_pairs, Plan& out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq <= 0 || Lk < 0 || num_pairs <= 0) return false;
  const int group = Hq / Hkv;
  const int n_mb = (Lq + kPairBlock - 1) / kPairBlock;
  const long long n_blocks = static_cast<long long>(B) * Hq * n_mb;
  if (n_blocks > (1LL << 26) || static_cast<long long>(B) * Hq > std::numeric_limits<int>::max()) return false;
  const int n_kt = (Lk + kPairBN - 1) / kPairBN;
  std::vector<PairBlock> blocks;
  blocks.reserve(static_cast<size_t>(n_blocks));
  long total = 0;
  int max_tiles = 0;
  // (batch, KV head, block, query head in group): query heads sharing a KV
  // head sit side by side
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < Hkv; ++g)
      for (int mb = 0; mb < n_mb; ++mb)
        for (int hh = 0; hh < group; ++hh) {
          int nt = n_kt;
          if (causal) {
            const int last_row = std::min(mb * kPairBlock + kPairBlock - 1, Lq - 1);
            const long max_key = static_cast<long>(last_row) + (Lk - Lq);
            nt = (max_key < 0) ? 0 : std::min<int>(n_kt, static_cast<int>(max_key / kPairBN) + 1);
          }
          blocks.push_back({b * Hq + g * group + hh, mb, nt});
          total += nt;
          max_tiles = std::max(max_tiles, nt);
        }
  const double c_unit = 0.5, c_split = 0.25;
  const double avg = (static_cast<double>(total) + c_unit * static_cast<double>(blocks.size())) / num_pairs;
  std::vector<double> targets = {std::numeric_limits<double>::infinity()};
  if (static_cast<double>(max_tiles) > 0.75 * avg) {
    for (double f = 0.25; f <= 3.0 + 1e-9; f += 0.03125)
      if (f * avg >= 1.0) targets.push_back(f * avg);
  }
  double best = std::numeric_limits<double>::infinity();
  std::vector<Cand> best_units;
  std::vector<int> best_cta;
  int best_n = 0;
  for (double tgt : targets) {
    std::vector<Cand> units;
    bool any_split = false;
    build_pair_units(blocks, tgt, c_unit, c_split, units, any_split);
    std::vector<int> cta_of;
    int n_workers = 0;
    const double ms = assign(units, num_pairs, cta_of, n_workers);
    // the pieces of a split block wait for each other before merging: a
    // pair runs at most one split piece, as its first unit, so every piece
    // is running when another waits for it
    if (any_split) {
      std::vector<int> n_split_pieces(n_workers, 0);
      bool ok = true;
      for (size_t i = 0; i < units.size() && ok; ++i)
        if (units[i].n_split > 1 && ++n_split_pieces[cta_of[i]] > 1) ok = false;
      if (!ok) continue;
    }
    if (ms < best - 1e-9 || (std::fabs(ms - best) <= 1e-9 && units.size() < best_units.size())) {
      best = ms;
      best_units = std::move(units);
      best_cta = std::move(cta_of);
      best_n = n_workers;
    }
  }
  out = Plan();
  std::vector<int> slot_base(blocks.size(), -1);
  int n_slots = 0;
  {
    std::vector<int> nsplit(blocks.size(), 1);
    for (const Cand& c : best_units) nsplit[c.pair] = c.n_split;
    for (size_t i = 0; i < blocks.size(); ++i)
      if (nsplit[i] > 1) {
        slot_base[i] = n_slots;
        out.groups.push_back({blocks[i].bh, blocks[i].mb, n_slots, nsplit[i]});
        n_slots += nsplit[i];
      }
  }
  out.n_ctas = best_n;   // pairs
  out.n_partials = n_slots;
  out.makespan = best;
  std::vector<std::vector<int>> per(best_n);
  for (size_t i = 0; i < best_units.size(); ++i) per[best_cta[i]].push_back(static_cast<int>(i));
  out.cta_off.assign(best_n + 1, 0);
  out.units.reserve(best_units.size());
  for (int c = 0; c < best_n; ++c) {
    out.cta_off[c] = static_cast<int>(out.units.size());
    // the split piece (at most one) first
    std::stable_partition(per[c].begin(), per[c].end(), [&](int i) { return best_units[i].n_split > 1; });
    for (int i : per[c]) {
      const Cand& u = best_units[i];
      const PairBlock& b = blocks[u.pair];
      const int slot = (u.n_split > 1) ? slot_base[u.pair] + u.split : -1;
      out.units.push_back({b.bh, b.mb, u.a, u.e, u.split, u.n_split, slot, c});
    }
  }
  out.cta_off[best_n] = static_cast<int>(out.units.size());
  return true;
}

bool make_plan_cluster(int B, int Hq, int Hkv, int Lq, int Lk, bool causal, int cs, Plan& out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq <= 0 || Lk < 0) return false;
  if (cs != 2 && cs != 4 && cs != 8) return false;
  const int group = Hq / Hkv;
  const int n_mb = (Lq + kBlockRows - 1) / kBlockRows;
  const long long n_ctas = static_cast<long long>(B) * Hq * n_mb * cs;
  if (n_ctas > (1LL << 24)) return false;
  out = Plan();
  out.units.reserve(static_cast<size_t>(n_ctas));
  int c = 0;
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < Hkv; ++g)
      for (int mb = 0; mb < n_mb; ++mb)
        for (int hh = 0; hh < group; ++hh) {
          const int kl0 = kv_last_tile(mb * kBlockRows, 0, Lq, Lk, causal);
          const int kl1 = kv_last_tile(mb * kBlockRows, 1, Lq, Lk, causal);
          const int T = std::max(kl0, kl1) + 1;
          for (int s = 0; s < cs; ++s, ++c) {
            const int a = static_cast<int>(static_cast<long>(s) * T / cs);
            const int e = static_cast<int>(static_cast<long>(s + 1) * T / cs);
            out.units.push_back({b * Hq + g * group + hh, mb, a, e, s, cs, -1, c});
            out.cta_off.push_back(c);
            out.makespan = std::max(out.makespan, static_cast<double>(e - a));
          }
        }
  out.cta_off.push_back(c);
  out.n_ctas = c;
  out.n_partials = 0;
  return true;
}

}  // namespace attn
