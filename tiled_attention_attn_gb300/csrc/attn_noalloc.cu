// attn_fwd_noalloc: the bf16 forward for callers that cannot allocate device
// memory (their memory belongs to a pool or caching allocator that has
// already reserved it, or they cannot afford cudaFree's device-wide
// synchronisation).  Same kernels as attn_fwd; the schedule and the split-KV
// partials live in one file-scope device array instead of library
// allocations.  No cudaMalloc, cudaFree or allocating library routine is
// called here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <tuple>
#include <vector>

#include "attn.h"
#include "attn_internal.h"
#include "attn_launch.h"
#include "attn_params.h"
#include "attn_plan.h"

namespace attn {
namespace {

constexpr size_t kSchedBytes = 4u << 20;     // schedule: units, CTA offsets, split groups
constexpr size_t kPartBytes = 20u << 20;     // split-KV partial accumulators and (m, l)
constexpr size_t kScratchBytes = kSchedBytes + kPartBytes;
static_assert(kScratchBytes == ATTN_NOALLOC_SCRATCH_BYTES, "scratch size and header disagree");

// The scratch.  In host code this name is only a stand-in for the symbol:
// its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

using ShapeKey = std::tuple<int, int, int, int, int, int, int>;   // B, Hq, Hkv, Lq, Lk, d, causal

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  DeviceInfo info;
  // host copy of the last shape's schedule (rebuilt when the shape changes)
  bool have_plan = false;
  ShapeKey key{};
  Plan plan;
  std::vector<int> units, groups;
  size_t off_cta = 0, off_groups = 0, off_ml = 0;
};

std::mutex g_na_mu;
NoAllocDevice g_na[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: the device address of the array.
int setup(int dev, NoAllocDevice& st) {
  if (st.ready) return ATTN_OK;
  int rc = device_info(dev, st.info);
  if (rc) return rc;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ELAUNCH;
  st.scratch = static_cast<unsigned char*>(ptr);
  st.ready = true;
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace attn

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int Lq, int Lk, int d, int causal, float scale, const int* cu,
                                cudaStream_t stream) {
  using namespace attn;
  // the same host-side checks as attn_fwd
  if (!q || !k || !v || !o || !lse) return ATTN_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4)) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0) return ATTN_EINVAL;
  if (Hq % Hkv != 0) return ATTN_EINVAL;
  if (causal != 0 && causal != 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_EINVAL;
  if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
  const bool varlen = cu != nullptr;
  if (varlen && (Lq != Lk || B > kVarlenMaxB)) return ATTN_EINVAL;
  const long long rows_q = varlen ? static_cast<long long>(Lq) : static_cast<long long>(B) * Lq;
  const long long rows_k = varlen ? static_cast<long long>(Lk) : static_cast<long long>(B) * Lk;
  if (rows_q * Hq > (1LL << 31) - 1 || rows_k * Hkv > (1LL << 31) - 1) return ATTN_EINVAL;
  if (static_cast<long long>(Lq) + kBlockRows > (1LL << 30) || static_cast<long long>(Lk) + kBN > (1LL << 30))
    return ATTN_EINVAL;
  if (Lq == 0) return ATTN_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_na_mu);
  NoAllocDevice& st = g_na[dev];
  int rc = setup(dev, st);
  if (rc) return rc;
  if (!st.info.supported) return ATTN_EUNSUPPORTED;

  static thread_local FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int Lk_map = Lk > 0 ? Lk : 1;
  const int Bm = varlen ? 1 : B;
  if ((rc = encode_map(q, true, d, Hq, Lq, Bm, p.tm_q))) return rc;
  if ((rc = encode_map(k, true, d, Hkv, Lk_map, Bm, p.tm_k))) return rc;
  if ((rc = encode_map(v, true, d, Hkv, Lk_map, Bm, p.tm_v))) return rc;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu;
  p.cu_seqlens_k = cu;   // self-attention: queries and keys share the offsets
  p.err = st.info.err_word;
  p.timeout_ns = wait_timeout_ns();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.group = Hq / Hkv;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;

  int grid = 0;
  bool combine = false;
  if (!varlen) {
    const ShapeKey key{B, Hq, Hkv, Lq, Lk, d, causal};
    if (!st.have_plan || st.key != key) {
      st.have_plan = false;
      if (!make_plan(B, Hq, Hkv, Lq, Lk, d, causal != 0, st.info.sm_count, st.plan)) return ATTN_EINVAL;
      const Plan& pl = st.plan;
      st.units.assign(pl.units.size() * kUnitInts, 0);
      for (size_t i = 0; i < pl.units.size(); ++i) {
        const PlanUnit& u = pl.units[i];
        const int e[kUnitInts] = {u.bh, u.m_block, u.kv_begin, u.kv_end, u.split, u.n_split, u.slot, u.cta};
        std::memcpy(&st.units[i * kUnitInts], e, sizeof(e));
      }
      st.groups.assign(pl.groups.size() * kGroupInts, 0);
      for (size_t i = 0; i < pl.groups.size(); ++i) {
        const PlanGroup& g = pl.groups[i];
        const int e[kGroupInts] = {g.bh, g.m_block, g.slot_base, g.n_split};
        std::memcpy(&st.groups[i * kGroupInts], e, sizeof(e));
      }
      st.off_cta = align256(st.units.size() * sizeof(int));
      st.off_groups = st.off_cta + align256(pl.cta_off.size() * sizeof(int));
      const size_t sched = st.off_groups + align256(st.groups.size() * sizeof(int));
      st.off_ml = align256(static_cast<size_t>(pl.n_partials) * kNSub * kBM * d * 4);   // fp32 partials
      const size_t part = st.off_ml + static_cast<size_t>(pl.n_partials) * kNSub * kBM * 2 * sizeof(float);
      if (sched > kSchedBytes || part > kPartBytes) return ATTN_ETOOLARGE;
      st.key = key;
      st.have_plan = true;
    }
    // The schedule the kernels read: small ones travel in the launch
    // parameters; larger ones are written into the array on every call, in
    // stream order just before the kernels (another call with another shape
    // in between cannot leave a stale schedule behind).
    const Plan& pl = st.plan;
    const bool inline_ok = pl.groups.empty() && static_cast<int>(pl.units.size()) <= kInlineUnits &&
                           pl.n_ctas <= kInlineCtas;
    if (inline_ok) {
      p.n_inline = 1;
      std::memcpy(p.units_inline, st.units.data(), st.units.size() * sizeof(int));
      std::memcpy(p.cta_off_inline, pl.cta_off.data(), pl.cta_off.size() * sizeof(int));
    } else {
      int* s = reinterpret_cast<int*>(st.scratch);
      if (upload_ints(s, st.units.data(), st.units.size(), stream) ||
          upload_ints(reinterpret_cast<int*>(st.scratch + st.off_cta), pl.cta_off.data(), pl.cta_off.size(), stream) ||
          (!st.groups.empty() &&
           upload_ints(reinterpret_cast<int*>(st.scratch + st.off_groups), st.groups.data(), st.groups.size(), stream)))
        return ATTN_ELAUNCH;
      p.units = reinterpret_cast<const int*>(st.scratch);
      p.cta_off = reinterpret_cast<const int*>(st.scratch + st.off_cta);
    }
    p.part_o = st.scratch + kSchedBytes;
    p.part_ml = reinterpret_cast<float*>(st.scratch + kSchedBytes + st.off_ml);
    grid = st.plan.n_ctas;
    combine = !st.plan.groups.empty();
  } else {
    const long long bound = static_cast<long long>(Hq) * (B + (Lq + kBlockRows - 1) / kBlockRows);
    grid = static_cast<int>(bound < st.info.sm_count ? bound : st.info.sm_count);
  }
  if (grid <= 0) return ATTN_OK;
  FwdLauncher launch = (d == 64) ? fwd_launcher_d64(true, causal != 0, varlen) : fwd_launcher_d128(true, causal != 0, varlen);
  if (launch(p, grid, stream) != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  if (combine) {
    CombineParams cp;
    cp.groups = reinterpret_cast<const int*>(st.scratch + st.off_groups);
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.o = o;
    cp.lse = lse;
    cp.Hq = Hq;
    cp.Lq = Lq;
    CombineLauncher cl = (d == 64) ? combine_launcher_d64(true) : combine_launcher_d128(true);
    if (cl(cp, static_cast<int>(st.plan.groups.size()), stream) != cudaSuccess) return ATTN_ELAUNCH;
    count_launch();
  }
  return ATTN_OK;
}
