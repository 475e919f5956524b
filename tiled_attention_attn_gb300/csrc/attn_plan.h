// Host-side schedule for the persistent forward kernel (dense inputs).
//
// The work of one (batch, query head) is cut into 256-row query blocks; a
// block reads the 128-key tiles its rows may see (all of them, or those up to
// the diagonal when causal; fully masked tiles are never scheduled).  Blocks
// whose tile count would dominate the makespan are split along the key range
// into pieces whose partial (u, m, l) a combine pass merges with the same
// r = exp(m_s - M) rescaling the online softmax applies across tiles.  Units
// are then placed longest first on the least-loaded CTA (the "persistent
// kernel" of page S23-J17 §5.4: resident CTAs fetch their next block of work
// instead of relaunching).
#pragma once
#include <vector>

namespace attn {

struct PlanUnit {
  int bh, m_block, kv_begin, kv_end, split, n_split, slot, cta;
};

struct PlanGroup {
  int bh, m_block, slot_base, n_split;
};

struct Plan {
  std::vector<PlanUnit> units;   // ordered by CTA, then by execution order
  std::vector<int> cta_off;      // n_ctas + 1
  std::vector<PlanGroup> groups; // split-KV groups (combine pass)
  int n_ctas = 0;
  int n_partials = 0;
  double makespan = 0;           // in cost units (one 128x128 query-key tile pair)
};

// Builds the schedule; returns false on arguments it cannot plan.
bool make_plan(int B, int Hq, int Hkv, int Lq, int Lk, int d, bool causal, int num_sms, Plan& out);

// The schedule of the CTA-pair forward: units are 256-row query blocks (128
// rows per CTA) against ranges of 256-key tiles [kv_begin, kv_end), placed on
// `num_pairs` SM pairs (Plan::n_ctas counts pairs, PlanUnit::cta is the
// pair).  Split pieces of one block share a group; the kernel merges them.
bool make_plan_pair(int B, int Hq, int Hkv, int Lq, int Lk, bool causal, int num_pairs, Plan& out);

// The schedule of the in-cluster merge: every 256-row query block split
// into `cs` key-range pieces of equal tile counts (a block with fewer tiles
// than cs has empty pieces), piece s of block g on CTA g * cs + s, one unit
// per CTA; no workspace slots and no combine groups.
bool make_plan_cluster(int B, int Hq, int Hkv, int Lq, int Lk, bool causal, int cs, Plan& out);

}  // namespace attn
