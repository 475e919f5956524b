// One decoding step on tensor cores with the keys on the MMA's M dimension.
//
// A decoding step gives each sequence one query: the G = Hq / Hkv query
// heads of a key/value head are G rows of attention against the sequence's
// cache (page S23-J17, clxhxhhr.top/posts/5544, §3.1: the running max m, the
// exp-sum l and the accumulator u, rescaled by r = 2^(m_old - m_new) when m
// grows).  The forward kernel's tile would hold G valid query rows of 128,
// and its softmax, one thread per query row and 128 keys per thread, would
// set the pace.  Here both products are transposed:
//   S^T = K Q^T   (M = 128 keys of the tile, N = 16 or 32 head columns, K = d)
//   u^T += V^T P^T (M = d = 128, N = the head columns, K = 128 keys)
// so the tile's keys sit on the 128 TMEM lanes and each softmax thread owns
// one key: G exponentials per tile instead of 128.  The tile's max over keys
// is a reduction across threads (redux.sync within a warp, then the four
// warps through shared memory); the exp-sum is kept per thread and reduced
// once per unit.  V is
// the A operand in its natural (keys x d) layout, read MN-major; P^T is
// written by the softmax threads into shared memory as the K-major B operand.
//
// Head dimension DA = 128 or 64.  A ring stage holds two 64-column chunks of
// K and of V (128-byte rows, 128-byte swizzle): with DA = 128 the two column
// halves of one 128-key tile, with DA = 64 two consecutive 128-key tiles, so
// that one softmax step (one max exchange across the four warps, the step's
// fixed cost) covers 256 keys.  At DA = 64 each tile has its own S^T
// columns, and one P.V serves both tiles: V read MN-major with M = 128 spans
// the stage's two chunks (rows 0-63 = d of tile a, rows 64-127 = d of tile
// b), and P^T has 2 x 16 rows (tile a's heads, then tile b's), so the
// product's diagonal blocks are u_a (lanes 0-63, columns 0-15) and u_b
// (lanes 64-127, columns 16-31); the off-diagonal blocks are never read.
// u = u_a + u_b is summed through shared memory at the unit's end.
//
// Work units are (sequence, key/value head, piece of the cache), the same
// schedule as the packed forward's decode mode, run round-robin over the
// CTAs; a cut cache's pieces leave fp32 partials that the decode combine
// merges.  CTA layout (192 threads, one CTA per SM):
//   warp 0     TMA producer (Q of the unit's heads, K and V tiles through a ring)
//   warp 1     TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2-5  softmax (thread = key of the tile for S^T, = d for u^T)
// Every wait is bounded (time limit, abort flag), as in the forward kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "attn_launch.h"
#include "attn_params.h"
#include "ptx.cuh"

namespace attn {
namespace dtc {

constexpr int kThreads = 192;
constexpr int kWarpTMA = 0;
constexpr int kWarpMMA = 1;
constexpr int kKeys = 128;   // keys per tile
constexpr int kD = 128;      // head dimension of the shared-memory tiles (the largest DA)

template <int NQ, int DA>
struct Cfg {
  static constexpr int kTPS = kD / DA;                 // 128-key tiles per softmax step
  static constexpr int kStages = (NQ == 16) ? 3 : 2;   // key/value ring (shared memory bounds it)
  static constexpr int kTile = kKeys * kD * 2;       // one stage of K or of V (two 64-column chunks), bytes
  static constexpr int kQChunk = NQ * 128;           // one 64-column chunk of the Q tile (NQ rows x 128 B)
  static constexpr int kQ = (DA / 64) * kQChunk;     // the Q tile (NQ rows x DA columns)
  static constexpr int kRows = kTPS * NQ;            // P^T rows of a step (the P.V's N)
  static constexpr int kPChunk = kRows * 128;        // one 64-key chunk of P^T
  static constexpr int kP = 2 * kPChunk;             // P^T of a step (kRows rows x 128 keys)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffQ = kOffV + kStages * kTile;   // two Q slots
  static constexpr int kOffP = kOffQ + 2 * kQ;            // two P^T buffers
  static constexpr int kOffRed = kOffP + 2 * kP;          // [parity][warp][NQ] floats
  // barriers: kv_full[S], kv_empty[S], q_full[2], q_empty[2], s_full[2],
  // p_full[2], p_free[2], o_free, red, drain, xch
  static constexpr int kOffBar = kOffRed + 2 * 4 * NQ * 4;
  static constexpr int kNBars = 2 * kStages + 14;
  static constexpr int kOffMisc = kOffBar + kNBars * 8;   // tmem slot, abort flag, bad flag
  static constexpr int kOffPref = kOffMisc + 64;          // units before each sequence (B + 1 ints)
  // sequences per call: the prefix table takes what shared memory leaves,
  // less 1 KB so that the merge pass's blocks (a programmatic dependent
  // launch) fit beside the CTA and wait there
  static constexpr int kMaxB = (227 * 1024 - 2048 - kOffPref) / 4 - 1 < kVarlenMaxB
                                   ? (227 * 1024 - 2048 - kOffPref) / 4 - 1
                                   : kVarlenMaxB;
  static constexpr int kSmem = kOffPref + 4 * (kMaxB + 1) + 1024;
  static_assert(kSmem <= 227 * 1024 && kMaxB >= 1024, "shared memory");
  // S^T: two buffers of kTPS tiles, then u^T (kRows columns)
  static constexpr int kUsedCols = 3 * kTPS * NQ;
  static constexpr uint32_t kTmemCols = kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128 : 256;
};

struct Params {
  CUtensorMap tm_q;    // q (B, Hq, d) as (d, Hq, B, 1), box 64 x G x 1 x 1
  CUtensorMap tm_k;    // k (total_k, Hkv, d) as (d, Hkv, total_k, 1), box 64 x 1 x 128 x 1
  CUtensorMap tm_v;
  void* o;             // (B, Hq, d)
  float* lse;          // (Hq, B)
  const int* cu_seqlens_k;
  int* pref_out;       // the unit prefix (B + 1) and the malformed flag, for the merge
  void* part_o;        // fp32 partials [slot][2][d/4][128][4] (sub-tile 0 used)
  float* part_ml;      // (m, l) [slot][2][128]
  int* err;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, total_k, G, split;
  float scale_log2;
};

struct Unit {
  int b, g;            // sequence, key/value head (= head group)
  int k_len, row_k;    // keys of the sequence, their first row in k / v
  int t0, t1;          // key tiles of this piece
  int n_split, slot;
};

__device__ __forceinline__ void decode_unit(const Params& p, const int* pref, int u, Unit& U) {
  int lo = 0, hi = p.B;   // largest b with pref[b] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= u) lo = mid; else hi = mid;
  }
  U.b = lo;
  U.row_k = __ldg(p.cu_seqlens_k + lo);
  U.k_len = __ldg(p.cu_seqlens_k + lo + 1) - U.row_k;
  const int pcs = decode_pieces(U.k_len, p.split);
  // units of a sequence: (piece, key/value head) with the head fastest, so
  // that CTAs running side by side read the same keys of neighbouring heads
  const int local = u - pref[lo];
  const int piece = local / p.Hkv;
  U.g = local - piece * p.Hkv;
  const int tiles = (U.k_len + kKeys - 1) / kKeys;
  U.n_split = pcs;
  U.slot = (pcs > 1) ? u : -1;
  U.t0 = (pcs > 1) ? piece * p.split : 0;
  U.t1 = (pcs > 1) ? min(tiles, U.t0 + p.split) : tiles;
}

// Shared-memory byte offset of element (row, col) in a K-major tile of
// 128-byte rows under the 128-byte swizzle (16-byte granule index XOR the
// row within its 8-row atom); col counts 16-bit elements within a 64-column
// chunk.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

template <int NQ>
__device__ __forceinline__ void tld(uint32_t taddr, float (&x)[NQ]) {
  if constexpr (NQ == 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
    tmem_wait_ld(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(r[i]);
  } else {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr, r);
    tmem_wait_ld(r);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
  }
}
template <int NQ>
__device__ __forceinline__ void tst(uint32_t taddr, const float (&x)[NQ]) {
  if constexpr (NQ == 16) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(x[i]);
    tmem_st_32x32b_x16(taddr, r);
  } else {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(x[i]);
    tmem_st_32x32b_x32(taddr, r);
  }
}

// Instruction descriptor (kind::f16, fp32 accumulator) with A read MN-major.
__host__ __device__ constexpr uint32_t idesc_a_mn(int M, int N, bool bf16) {
  return idesc_f16_f32acc(M, N, bf16, false) | (1u << 15);
}

template <int NQ, int GT, bool BF16, int DA>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ Params p) {
  static_assert(GT >= 1 && GT <= NQ, "query heads per key/value head");
  using C = Cfg<NQ, DA>;
  static_assert(DA == 128 || DA == 64, "head dimension");
  constexpr int kTPS = C::kTPS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ, sP = sbase + C::kOffP;
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto b_kv_full = [&](int s) { return bar0 + 8 * s; };
  auto b_kv_empty = [&](int s) { return bar0 + 8 * (C::kStages + s); };
  const uint32_t bar1 = bar0 + 8 * 2 * C::kStages;
  auto b_q_full = [&](int s) { return bar1 + 8 * s; };
  auto b_q_empty = [&](int s) { return bar1 + 8 * (2 + s); };
  auto b_s_full = [&](int s) { return bar1 + 8 * (4 + s); };
  auto b_p_full = [&](int s) { return bar1 + 8 * (6 + s); };
  // p_free(b): the P.V that read P^T buffer b has completed (one phase per use)
  auto b_p_free = [&](int s) { return bar1 + 8 * (8 + s); };
  const uint32_t b_o_free = bar1 + 8 * 10;
  const uint32_t b_red = bar1 + 8 * 11;
  const uint32_t b_drain = bar1 + 8 * 12;
  const uint32_t b_xch = bar1 + 8 * 13;   // u_b handed over (head_dim 64)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  int* pref = reinterpret_cast<int*>(smem + C::kOffPref);
  WaitCtl wc{p.err, abort_flag, p.timeout_ns};

  if (tid == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(b_kv_full(s), 1);
      mbar_init(b_kv_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_q_full(s), 1);
      mbar_init(b_q_empty(s), 1);
      mbar_init(b_s_full(s), 1);
      mbar_init(b_p_full(s), 4);   // the four softmax warps
      mbar_init(b_p_free(s), 1);
    }
    mbar_init(b_o_free, 4);
    mbar_init(b_red, 4);
    mbar_init(b_drain, 1);
    mbar_init(b_xch, 2);
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTMA && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == 2) {
    // validate cu_seqlens_k and build the unit prefix: sequence b has
    // Hkv x pieces(b) units
    int carry = 0;
    bool bad = lane == 0 && __ldg(p.cu_seqlens_k) != 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int cnt = 0;
      if (b < p.B) {
        const int ak = __ldg(p.cu_seqlens_k + b), ek = __ldg(p.cu_seqlens_k + b + 1);
        if (ek < ak || ek > p.total_k) bad = true;
        cnt = p.Hkv * decode_pieces(max(ek - ak, 0), p.split);
      }
      int x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (b < p.B) pref[b + 1] = carry + x;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) pref[0] = 0;
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      *bad_flag = 1;
      atomicCAS(p.err, 0, ATTN_DEVERR_BAD_SEQLENS);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_launch_dependents();
  const int n_units = (*bad_flag) ? 0 : pref[p.B];
  if (blockIdx.x == 0) {
    for (int i = tid; i <= p.B; i += kThreads) p.pref_out[i] = pref[i];
    if (tid == 0) p.pref_out[p.B + 1] = *bad_flag;
  }
  if (*bad_flag) {
    // malformed offsets: every row O = 0, lse = -inf
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    T* out = reinterpret_cast<T*>(p.o);
    for (long long r = static_cast<long long>(blockIdx.x) * kThreads + tid; r < static_cast<long long>(p.B) * p.Hq;
         r += static_cast<long long>(gridDim.x) * kThreads) {
      uint4* d4 = reinterpret_cast<uint4*>(out + r * DA);
#pragma unroll
      for (int i = 0; i < DA / 8; ++i) d4[i] = make_uint4(0, 0, 0, 0);
      const long long b = r / p.Hq, h = r - b * p.Hq;
      p.lse[h * p.B + b] = -INFINITY;
    }
  }

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t q_cnt = 0, kv_cnt = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        Unit U;
        decode_unit(p, pref, u, U);
        if (U.t1 <= U.t0) continue;
        const int qs = q_cnt & 1;
        if (!mbar_wait(b_q_empty(qs), ((q_cnt >> 1) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQEmpty))) break;
        mbar_arrive_expect_tx(b_q_full(qs), (DA / 64) * p.G * 128);
        for (int c = 0; c < DA / 64; ++c)
          tma_load_4d(sQ + qs * C::kQ + c * C::kQChunk, &p.tm_q, b_q_full(qs), c * 64, U.g * p.G, U.b, 0);
        ++q_cnt;
        for (int t = U.t0; t < U.t1; t += kTPS) {
          const int st = kv_cnt % C::kStages;
          if (!mbar_wait(b_kv_empty(st), ((kv_cnt / C::kStages) & 1) ^ 1, wc,
                         ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKEmpty))) { ok = false; break; }
          // chunk c: columns 64c.. of tile t (DA = 128) or tile t + c (DA = 64).
          // A segment's odd last tile at DA = 64 loads no K chunk 1 (its S^T is
          // not computed) and a V chunk 1 of zeros, from rows past total_k
          // (the fill value): the step's P.V multiplies that chunk by P = 0
          const int nc = (kTPS == 1) ? 2 : min(2, U.t1 - t);
          mbar_arrive_expect_tx(b_kv_full(st), (2 * nc + (nc < 2 ? 1 : 0)) * 16384);
          for (int c = 0; c < nc; ++c) {
            const int col = (kTPS == 1) ? c * 64 : 0, row = U.row_k + (kTPS == 1 ? t : t + c) * kKeys;
            tma_load_4d(sK + st * C::kTile + c * 16384, &p.tm_k, b_kv_full(st), col, U.g, row, 0);
            tma_load_4d(sV + st * C::kTile + c * 16384, &p.tm_v, b_kv_full(st), col, U.g, row, 0);
          }
          if (nc < 2) tma_load_4d(sV + st * C::kTile + 16384, &p.tm_v, b_kv_full(st), 0, U.g, p.total_k, 0);
          ++kv_cnt;
        }
      }
      if (*abort_flag) {
        // let the loads already issued land before the CTA exits
        for (int s = 0; s < C::kStages; ++s) {
          const uint32_t n = (kv_cnt + C::kStages - 1 - s) / C::kStages;
          if (n > 0) mbar_wait(b_kv_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
        for (int s = 0; s < 2; ++s) {
          const uint32_t n = (q_cnt + 1 - s) / 2;
          if (n > 0) mbar_wait(b_q_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
      }
    }
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(kKeys, NQ, BF16, false);   // A = K, B = Q: both K-major
      constexpr uint32_t kIdescO = idesc_a_mn(kD, C::kRows, BF16);            // A = V read MN-major, B = P^T
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV, 16384, 1024);
      const uint64_t dp0 = sdesc_sw128(sP, 16, 1024);
      const uint32_t t_u = tmem + 2 * kTPS * NQ;   // u^T columns
      uint32_t q_cnt = 0, kv_cnt = 0, s_cnt = 0, p_cnt = 0, units_done = 0;
      bool ok = true;
      auto issue_pv = [&](int st, int pb, bool first) {   // stage st, P^T buffer pb
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t a = dv0 + ((st * C::kTile + kk * 2048) >> 4);
          const uint64_t b = dp0 + ((pb * C::kP + (kk >> 2) * C::kPChunk + (kk & 3) * 32) >> 4);
          umma_ss(t_u, a, b, kIdescO, (first && kk == 0) ? 0u : 1u);
        }
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        Unit U;
        decode_unit(p, pref, u, U);
        if (U.t1 <= U.t0) continue;
        const int qs = q_cnt & 1;
        if (!mbar_wait(b_q_full(qs), (q_cnt >> 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull))) break;
        ++q_cnt;
        tc_fence_after();
        // before the unit's first P.V (which overwrites u^T), the previous
        // unit's epilogue must have read u^T
        auto wait_o_free = [&]() -> bool {
          if (units_done == 0) return true;
          if (!mbar_wait(b_o_free, (units_done - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone))) return false;
          tc_fence_after();
          return true;
        };
        int prev_pb = -1;
        bool first_pv = true;
        // u^T += V^T P^T of the tile in stage vst, P^T buffer pb; the stage
        // (K and V) is released after it
        auto do_pv = [&](int vst, int pb, bool first) -> bool {
          if (!mbar_wait(b_p_full(pb), (p_cnt >> 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePFull))) return false;
          ++p_cnt;
          if (first && !wait_o_free()) return false;
          tc_fence_after();
          issue_pv(vst, pb, first);
          umma_commit(b_kv_empty(vst));
          umma_commit(b_p_free(pb));
          return true;
        };
        int prev_st = -1;
        for (int t = U.t0; t < U.t1; t += kTPS) {
          const int st = kv_cnt % C::kStages;
          const int nt = min(kTPS, U.t1 - t);
          if (!mbar_wait(b_kv_full(st), (kv_cnt / C::kStages) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) {
            ok = false;
            break;
          }
          ++kv_cnt;
          tc_fence_after();
          // S^T of the step's tiles into buffer s_cnt & 1: its previous
          // contents (two steps back) were consumed, since this thread has
          // waited for that step's P
          const int sb = s_cnt & 1;
          for (int x = 0; x < nt; ++x) {
#pragma unroll
            for (int kk = 0; kk < DA / 16; ++kk) {
              const uint32_t off = ((x + (kk >> 2)) * 16384 + (kk & 3) * 32) >> 4;
              const uint32_t offq = ((qs * C::kQ + (kk >> 2) * C::kQChunk + (kk & 3) * 32) >> 4);
              umma_ss(tmem + (sb * kTPS + x) * NQ, dk0 + ((st * C::kTile) >> 4) + off, dq0 + offq, kIdescS,
                      kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(b_s_full(sb));
          ++s_cnt;
          if (prev_pb >= 0) {
            if (!do_pv(prev_st, prev_pb, first_pv)) {
              ok = false;
              break;
            }
            first_pv = false;
          }
          prev_st = st;
          prev_pb = sb;
        }
        if (!ok) break;
        // the unit's last step
        if (!do_pv(prev_st, prev_pb, first_pv)) break;
        umma_commit(b_q_empty(qs));
        ++units_done;
      }
      umma_commit(b_drain);
      mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const int sw = warp - 2;                       // softmax warp 0..3
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may address
    const int lrow = quarter * 32 + lane;          // TMEM lane: key of the tile (S^T), d (u^T)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // u^T columns this thread's lane holds: at DA = 64 lanes 64-127 keep u_b
    const uint32_t t_u = tmem + lane_off + 2 * kTPS * NQ + ((kTPS == 2 && lrow >= 64) ? NQ : 0);
    const float c = p.scale_log2;
    constexpr int G = GT;
    uint32_t s_cnt = 0, red_cnt = 0, xch_cnt = 0;
    uint32_t free_seen[2] = {0, 0};   // phases of p_free(b) observed
    uint32_t tiles_total = 0;   // steps (P^T buffer uses) so far for this CTA (all units)
    bool ok = true;
    // reduces v over the 128 softmax threads (max or sum), all get the result:
    // within a warp by redux.sync (max) or shuffles (sum), then across the
    // four warps through shared memory
    auto reduce = [&](float (&v)[NQ], bool is_max) -> bool {
#pragma unroll
      for (int h = 0; h < NQ; ++h) {
        if (h >= G) break;
        float x = v[h];
        if (is_max) {
          asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(x) : "f"(v[h]));
        } else {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        }
        v[h] = x;
      }
      const int par = red_cnt & 1;
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < NQ; ++h)
          if (h < G) red[(par * 4 + sw) * NQ + h] = v[h];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b_red);
      if (!mbar_wait_warp(b_red, red_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteXchg))) return false;
      ++red_cnt;
#pragma unroll
      for (int h = 0; h < NQ; ++h) {
        if (h >= G) break;
        const float a = red[(par * 4 + 0) * NQ + h], b = red[(par * 4 + 1) * NQ + h];
        const float e = red[(par * 4 + 2) * NQ + h], f = red[(par * 4 + 3) * NQ + h];
        v[h] = is_max ? fmaxf(fmaxf(a, b), fmaxf(e, f)) : (a + b) + (e + f);
      }
      return true;
    };
    // waits until the P.V of this CTA's tile g (counted over all its units)
    // has completed, and with it every earlier one.  Tile g's product read
    // P^T buffer g & 1 and completes phase g >> 1 of p_free(g & 1); phases of
    // one buffer are observed in order and never fall two behind (tile g + 2
    // writes that buffer only after this wait), so the parity test is exact.
    auto pv_wait = [&](uint32_t g) -> bool {
      const int b = g & 1;
      while (free_seen[b] <= (g >> 1)) {
        if (!mbar_wait_warp(b_p_free(b), free_seen[b] & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePvDone)))
          return false;
        ++free_seen[b];
      }
      tc_fence_after();
      return true;
    };
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      Unit U;
      decode_unit(p, pref, u, U);
      const size_t orow0 = static_cast<size_t>(U.b) * p.Hq + U.g * G;   // first output row (b, head)
      if (U.t1 <= U.t0) {
        // a sequence without keys: O = 0, lse = -inf
        T* dst = reinterpret_cast<T*>(p.o);
        if (lrow < DA)
          for (int h = 0; h < G; ++h) dst[(orow0 + h) * DA + lrow] = T(0.0f);
        if (sw == 0 && lane < G) p.lse[static_cast<size_t>(U.g * G + lane) * p.B + U.b] = -INFINITY;
        continue;
      }
      float m[NQ], l[NQ];
#pragma unroll
      for (int h = 0; h < NQ; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
      }
      const uint32_t tile0 = tiles_total;
      for (int t = U.t0; t < U.t1; t += kTPS) {
        const uint32_t i = tiles_total - tile0;   // step within the unit
        const int sb = s_cnt & 1;
        if (!mbar_wait_warp(b_s_full(sb), (s_cnt >> 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFull))) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        // this thread's key in each tile of the step
        float s[kTPS][NQ];
        bool valid[kTPS];
#pragma unroll
        for (int y = 0; y < kTPS; ++y) {
          tld<NQ>(tmem + lane_off + (sb * kTPS + y) * NQ, s[y]);
          valid[y] = t + y < U.t1 && (t + y) * kKeys + lrow < U.k_len;
        }
        float x[NQ];
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          x[h] = valid[0] ? s[0][h] : -INFINITY;
#pragma unroll
          for (int y = 1; y < kTPS; ++y) x[h] = fmaxf(x[h], valid[y] ? s[y][h] : -INFINITY);
        }
        if (!reduce(x, true)) { ok = false; break; }
        // running max (scaled units) with the stale-max rule of the forward
        // kernel: rescale only when the max grows by more than 2^8
        float r[NQ];
        bool any_resc = false;
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          r[h] = 1.0f;
          if (h >= G) continue;
          const float mt = (x[h] == -INFINITY) ? -INFINITY : x[h] * c;
          if (mt > m[h] && (i == 0 || m[h] == -INFINITY || mt - m[h] > 8.0f)) {
            r[h] = (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - mt);
            m[h] = mt;
            any_resc = true;
          }
        }
        // P^T of these keys into buffer sb, once the P.V that read it two
        // steps back (this CTA's step tiles_total - 2) has completed
        if (tiles_total >= 2 && !pv_wait(tiles_total - 2)) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          if (h >= G) break;
          const float mh = (m[h] == -INFINITY) ? 0.0f : m[h];
          float e_sum = 0.0f;
#pragma unroll
          for (int y = 0; y < kTPS; ++y) {
            const float e = valid[y] ? ex2_approx(s[y][h] * c - mh) : 0.0f;
            e_sum += e;
            uint8_t* pbuf = smem + C::kOffP + sb * C::kP + (lrow >> 6) * C::kPChunk;
            *reinterpret_cast<T*>(pbuf + sw128(y * NQ + h, lrow & 63)) = T(e);
          }
          l[h] = l[h] * r[h] + e_sum;
        }
        // u^T rescale (rare): needs the previous step's P.V complete.  m is
        // the same in every thread, so the decision is too; the vote keeps the
        // warp-collective TMEM accesses below uniform regardless.
        any_resc = __any_sync(0xffffffffu, any_resc);
        if (i > 0 && any_resc) {
          if (!pv_wait(tiles_total - 1)) { ok = false; break; }
          float o[NQ];
          tld<NQ>(t_u, o);
#pragma unroll
          for (int h = 0; h < NQ; ++h) o[h] *= r[h];
          tst<NQ>(t_u, o);
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p_full(sb));
        ++tiles_total;
      }
      if (!ok) break;
      // the unit's exp-sums over all keys, then u^T / l
      if (!reduce(l, false)) break;
      if (!pv_wait(tiles_total - 1)) break;
      float o[NQ];
      tld<NQ>(t_u, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_o_free);   // u^T may be overwritten by the next unit
      if constexpr (kTPS == 2) {
        // u = u_a + u_b: lanes 64-127 hand u_b over through the first P^T
        // buffer, idle now that every P.V so far has completed; the next
        // P^T write follows the next max exchange, which all four warps
        // reach only after this
        float* xch = reinterpret_cast<float*>(smem + C::kOffP);
        if (lrow >= 64) {
#pragma unroll
          for (int h = 0; h < NQ; ++h)
            if (h < G) xch[h * 64 + (lrow - 64)] = o[h];
          __syncwarp();
          if (lane == 0) mbar_arrive(b_xch);
        } else {
          if (!mbar_wait_warp(b_xch, xch_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteXchg))) break;
#pragma unroll
          for (int h = 0; h < NQ; ++h)
            if (h < G) o[h] += xch[h * 64 + lrow];
        }
        ++xch_cnt;
      }
      if (U.n_split <= 1) {
        T* dst = reinterpret_cast<T*>(p.o);
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          if (h >= G || lrow >= DA) break;
          dst[(orow0 + h) * DA + lrow] = T((l[h] > 0.0f) ? o[h] / l[h] : 0.0f);
        }
        if (sw == 0 && lane < G) {
          float lv = 0.0f, mv = 0.0f;
#pragma unroll
          for (int h = 0; h < NQ; ++h)
            if (h == lane) {
              lv = l[h];
              mv = m[h];
            }
          p.lse[static_cast<size_t>(U.g * G + lane) * p.B + U.b] =
              (lv > 0.0f) ? mv * 0.69314718055994531f + __logf(lv) : -INFINITY;
        }
      } else {
        // a piece: O_s = u^T / l in fp32 and (m, l), rows = heads of the group
        float* po = reinterpret_cast<float*>(p.part_o);
        const size_t pbase = static_cast<size_t>(U.slot) * kNSub * (DA / 4);
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          if (h >= G || lrow >= DA) break;
          po[((pbase + (lrow >> 2)) * kBM + h) * 4 + (lrow & 3)] = (l[h] > 0.0f) ? o[h] / l[h] : 0.0f;
        }
        if (sw == 0 && lane < G) {
          float lv = 0.0f, mv = -INFINITY;
#pragma unroll
          for (int h = 0; h < NQ; ++h)
            if (h == lane) {
              lv = l[h];
              mv = m[h];
            }
          reinterpret_cast<float2*>(p.part_ml)[static_cast<size_t>(U.slot) * kNSub * kBM + lane] =
              make_float2(lv > 0.0f ? mv : -INFINITY, lv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NQ, int GT, bool BF16, int DA>
cudaError_t launch(const Params& p, int grid, cudaStream_t stream) {
  constexpr int smem = Cfg<NQ, DA>::kSmem;
  static bool attr_done[64] = {};   // per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(decode_tc_kernel<NQ, GT, BF16, DA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  decode_tc_kernel<NQ, GT, BF16, DA><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dtc

int decode_tc_max_b(int d) { return d == 64 ? dtc::Cfg<16, 64>::kMaxB : dtc::Cfg<16, 128>::kMaxB; }

cudaError_t launch_decode_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, void* o,
                             float* lse, const int* cu_k, int* pref_out, void* part_o, float* part_ml, int* err,
                             unsigned long long timeout_ns, int B, int Hq, int Hkv, int total_k, int split,
                             float scale_log2, bool bf16, int d, int grid, cudaStream_t stream) {
  dtc::Params p;
  p.tm_q = tm_q;
  p.tm_k = tm_k;
  p.tm_v = tm_v;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens_k = cu_k;
  p.pref_out = pref_out;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.err = err;
  p.timeout_ns = timeout_ns;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.total_k = total_k;
  p.G = Hq / Hkv;
  p.split = split;
  p.scale_log2 = scale_log2;
  // the query heads per key/value head that attn_decode accepts: 1, 2, 4, 8
  if (d == 64) {
    switch (p.G) {
      case 1: return bf16 ? dtc::launch<16, 1, true, 64>(p, grid, stream) : dtc::launch<16, 1, false, 64>(p, grid, stream);
      case 2: return bf16 ? dtc::launch<16, 2, true, 64>(p, grid, stream) : dtc::launch<16, 2, false, 64>(p, grid, stream);
      case 4: return bf16 ? dtc::launch<16, 4, true, 64>(p, grid, stream) : dtc::launch<16, 4, false, 64>(p, grid, stream);
      case 8: return bf16 ? dtc::launch<16, 8, true, 64>(p, grid, stream) : dtc::launch<16, 8, false, 64>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (d != 128) return cudaErrorInvalidValue;
  switch (p.G) {
    case 1: return bf16 ? dtc::launch<16, 1, true, 128>(p, grid, stream) : dtc::launch<16, 1, false, 128>(p, grid, stream);
    case 2: return bf16 ? dtc::launch<16, 2, true, 128>(p, grid, stream) : dtc::launch<16, 2, false, 128>(p, grid, stream);
    case 4: return bf16 ? dtc::launch<16, 4, true, 128>(p, grid, stream) : dtc::launch<16, 4, false, 128>(p, grid, stream);
    case 8: return bf16 ? dtc::launch<16, 8, true, 128>(p, grid, stream) : dtc::launch<16, 8, false, 128>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
