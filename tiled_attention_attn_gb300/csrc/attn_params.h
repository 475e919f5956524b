// Parameters shared by the host launcher and the sm_103a kernels.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "attn.h"

#define ATTN_DEVERR_WAIT_TIMEOUT_SITE(site) (ATTN_DEVERR_WAIT_TIMEOUT | (site))

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__
#else
#define ATTN_HD
#endif

namespace attn {

constexpr int kBM = 128;        // query rows per sub-tile (one TMEM lane per row)
constexpr int kBN = 128;        // keys per KV tile
constexpr int kNSub = 2;        // query sub-tiles per work unit (256 query rows)
constexpr int kBlockRows = kBM * kNSub;
constexpr int kThreads = 320;   // 8 softmax warps + 1 TMA warp + 1 MMA warp
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr int kVarlenMaxB = 4096;   // sequences per varlen call (prefix table in smem)
constexpr int kVarlenSortMax = 32;  // the sorting varlen variant ranks at most this many sequences
constexpr int kUnitInts = 8;        // ints per scheduled work unit
constexpr int kGroupInts = 4;       // ints per split-KV group
constexpr int kMaxSplits = 64;      // split pieces per group
constexpr int kInlineUnits = 200;   // schedules up to this size travel in the kernel parameters
constexpr int kInlineCtas = 160;

// Phase trace streams and tags (attn_trace_enable).  An event is two 64-bit
// words: (tag << 56 | sub-tile << 48 | unit << 24 | key tile) and the SM clock.
enum TraceStream : int { kTrProducer = 0, kTrMMA = 1, kTrSoftmax0 = 2, kTrSoftmax1 = 3, kTrStreams = 4 };
enum TraceTag : int {
  kTagStart = 1, kTagQIssue = 2, kTagKIssue = 3, kTagVIssue = 4,
  kTagQFull = 10, kTagSIssue = 11, kTagPFull = 12, kTagPVIssue = 13, kTagKFull = 14, kTagVFull = 15,
  kTagUnitEnd = 16, kTagVWait = 17, kTagPWait = 18,
  kTagSFull = 20, kTagPArrive = 21, kTagODone = 23, kTagEpiDone = 24, kTagUnitBegin = 25,
  kTagMaxDone = 26, kTagPvWait = 27, kTagPvDone = 28, kTagSFreeWait = 29,
  kTagPartDone = 30, kTagSlice = 31, kTagMergeDone = 32, kTagEpiStore = 33,
  kTagGEnter = 40, kTagGExit = 41,   // the second word holds %globaltimer (ns) instead of the SM clock
};

// Wait-site codes (low byte of ATTN_DEVERR_WAIT_TIMEOUT).
enum WaitSite : int {
  kSiteQEmpty = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSiteVFull,
  kSiteSFull, kSitePFull, kSiteODone, kSiteDrain, kSiteSelftest, kSiteDsFull,
  kSiteSFree, kSitePvDone, kSiteMerge, kSiteXchg
};

struct FwdParams {
  CUtensorMap tm_q;            // (d, Hq, L, B) or packed (d, Hq, total, 1); box 64 x 1 x 128 x 1
                               // (64 x group x 128/group x 1 when pack_log2 > 0)
  CUtensorMap tm_k;            // (d, Hkv, L, B) or packed
  CUtensorMap tm_v;
  void* o;                     // like q
  float* lse;                  // (B, Hq, Lq) or (Hq, total)
  const int* cu_seqlens;       // varlen only: query row offsets (B+1)
  const int* cu_seqlens_k;     // varlen only: key row offsets (B+1); the same array for self-attention
  const int* units;            // dense schedule, kUnitInts per unit, grouped by CTA
  const int* cta_off;          // dense: first unit of every CTA, n_ctas + 1 entries
  void* part_o;                // split-KV partial outputs O_s = u_s / l_s, fp32 [slot][2][D/4][128][4]
  float* part_ml;              // split-KV partial (m, l) [slot][2][128][2]
  // In-cluster merge (dense): a cluster of cluster_merge CTAs holds the
  // cluster_merge pieces of one query block, piece s on cluster rank s, one
  // unit per CTA; the pieces' partials stay in shared memory and are merged
  // over distributed shared memory (no workspace, no combine pass).  0: off.
  int cluster_merge;
  int* err;                    // device error word
  unsigned long long* trace;   // optional phase trace (traced build, attn_trace_enable), else null
  int trace_cap;               // events per stream per CTA
  unsigned long long timeout_ns;
  int B, Hq, Hkv, Lq, Lk, group;
  // varlen only: log2 of the query heads of one key/value group that share a
  // tile (0: a tile holds 128 rows of one head).  With 2^pack_log2 = group a
  // tile holds 128 / group tokens x group heads, row r = token r >> pack_log2,
  // head r & (group - 1), and tm_q's box is 64 x group x (128 / group) x 1.
  int pack_log2;
  // Decode mode (varlen only): one query per sequence, sequence b's query at
  // row b of q (cu_seqlens unused, may be null).  vl_split > 0 cuts the keys
  // of every (sequence, head group) into pieces of at most vl_split tiles,
  // each its own unit writing a partial (slot = unit index) that the decode
  // combine merges; CTA 0 writes the per-sequence unit prefix (B + 1 ints)
  // and a malformed-offsets flag to vl_pref_out for that pass.
  int vl_decode;
  int vl_split;
  int* vl_pref_out;
  // Rotary embedding of Q inside the kernel (the ROPE instantiations, dense
  // only): rope_cs[pos * rot / 2 + i] = (cos, sin) of pos * base^(-2 i / rot);
  // query row i of a sequence has position i + rope_qoff; GPT-J pairs
  // (2i, 2i+1) when rope_gptj, else GPT-NeoX pairs (i, i + rot/2).
  const float* rope_cs;   // float2 pairs
  int rope_rot;
  int rope_gptj;
  int rope_qoff;
  float scale_log2;            // scale * log2(e)
  float scale;
  // A small schedule is copied here so that a CTA learns its first unit from
  // the launch itself instead of a global-memory read (n_inline = 0: use
  // units / cta_off).
  int n_inline;
  int cta_off_inline[kInlineCtas + 1];
  int units_inline[kInlineUnits * kUnitInts];
};

// Merge of the decode mode's split pieces: one block per (sequence, head
// group) and 16-column slice; rows are the group's query heads.
struct DecodeCombineParams {
  const void* part_o;          // fp32 partials, the forward's [slot][2][D/4][128][4] layout
  const float* part_ml;        // (m, l) per slot, sub-tile and row
  const int* pref;             // units before each sequence (B + 1), then the malformed flag
  const int* cu_seqlens_k;
  void* o;                     // (B, Hq, D)
  float* lse;                  // (Hq, B)
  int B, Hq, pack_log2, split;
};

// Tiles of `split` keys each covering a sequence of k_len keys; a sequence
// without keys is one (empty) piece.
ATTN_HD inline int decode_pieces(int k_len, int split) {
  const int tiles = (k_len + kBN - 1) / kBN;
  if (split <= 0 || tiles <= split) return 1;
  return (tiles + split - 1) / split;
}

// ---------------------------------------------------------------------------
// The CTA-pair forward (tcgen05 .cta_group::2): a work unit is a 256-row
// query block (128 rows in each CTA of the pair) against a range of 256-key
// tiles; each CTA holds its own query rows, half of every key tile (128 keys)
// and half of the columns of every value tile (d/2 of 256 keys).
// ---------------------------------------------------------------------------
constexpr int kPairThreads = 384;          // 8 softmax warps, TMA warp, two MMA warps, 1 spare warp
// Registers: launched at 168 per thread (384 x 168 = 64,512); the softmax
// warpgroups raise theirs to 216 and the third warpgroup lowers its to 72:
// 256 x 216 + 128 x 72 = 64,512, exactly the launch allocation.
constexpr int kPairRegsSoftmax = 216;
constexpr int kPairRegsOther = 72;
static_assert(256 * kPairRegsSoftmax + 128 * kPairRegsOther <= kPairThreads * 168, "register split");
constexpr int kPairRows = 128;             // query rows per CTA
constexpr int kPairBlock = 2 * kPairRows;  // query rows per unit (both CTAs)
constexpr int kPairBN = 256;               // keys per key tile (128 in each CTA)
constexpr int kInlinePairs = 80;           // pair schedules up to this many pairs travel inline
constexpr int kPairInlineUnits = 160;

struct PairParams {
  CUtensorMap tm_q;            // (d, Hq, Lq, B), box 64 x 1 x 128 x 1
  CUtensorMap tm_k;            // (d, Hkv, Lk, B), box 64 x 1 x 128 x 1
  CUtensorMap tm_v;            // (d, Hkv, Lk, B), box d/2 x 1 x 256 x 1
  CUtensorMap tm_o;            // (d, Hq, Lq, B), box 64 x 1 x 128 x 1 (the epilogue's stores)
  void* o;                     // (B, Lq, Hq, d)
  float* lse;                  // (B, Hq, Lq)
  const int* units;            // kUnitInts per unit, grouped by pair
  const int* pair_off;         // first unit of every pair, n_pairs + 1 entries
  float* part_u;               // split pieces: unnormalised u, fp32 [slot][2][d/4][128][4]
  float* part_ml;              // split pieces: (m, l) [slot][2][128] float2
  unsigned long long* counters;   // split pieces: one word per (slot, CTA of the pair)
  unsigned int epoch;          // this call's tag in the counter words
  int* err;
  unsigned long long* trace;   // optional phase trace (traced build, attn_trace_enable), else null
  int trace_cap;               // events per stream per CTA
  unsigned long long timeout_ns;
  int B, Hq, Hkv, Lq, Lk, group;
  float scale_log2;            // scale * log2(e)
  int n_inline;                // 1: the schedule is in the arrays below
  int pair_off_inline[kInlinePairs + 1];
  int units_inline[kPairInlineUnits * kUnitInts];
};

struct CombineParams {
  const int* groups;           // kGroupInts per group: bh, m_block, slot_base, n_split
  const void* part_o;
  const float* part_ml;
  void* o;
  float* lse;
  int Hq, Lq;
};

// Last 128-key tile (inclusive) that holds an allowed key for query sub-tile
// `t` of the block starting at query `q_row0`, each sub-tile covering `span`
// queries (128, or 128 / group when a group's heads share the tile), or -1 if
// the sub-tile has no valid query or no allowed key.  Causal keeps key j for
// query i iff j <= i + (k_len - q_len).
ATTN_HD inline int kv_last_tile(int q_row0, int t, int q_len, int k_len, bool causal, int span = kBM) {
  const int first = q_row0 + t * span;
  if (first >= q_len || k_len <= 0) return -1;
  int last_row = first + span - 1;
  if (last_row > q_len - 1) last_row = q_len - 1;
  int last = (k_len + kBN - 1) / kBN - 1;
  if (causal) {
    const int max_key = last_row + (k_len - q_len);
    if (max_key < 0) return -1;
    const int lt = max_key / kBN;
    if (lt < last) last = lt;
  }
  return last;
}

}  // namespace attn
