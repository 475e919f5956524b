// C ABI of the attention forward library: argument checks, TMA descriptor and
// schedule caches, workspace, launches and the device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <vector>

#include "attn.h"
#include "attn_cache.h"
#include "attn_internal.h"
#include "attn_launch.h"
#include "attn_pair_launch.h"
#include "attn_params.h"
#include "attn_plan.h"
#include "ptx.cuh"

namespace attn {

// First device-side error since the last attn_get_error() (0 = none).
__device__ int g_attn_err;

namespace {

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_pair_forward{0};   // attn_set_pair_forward
std::atomic<int> g_cluster_merge{0};  // attn_set_cluster_merge: 0, 2, 4 or 8
std::atomic<int> g_decode_tc{1};      // attn_set_decode_path
unsigned long long* g_trace = nullptr;   // attn_trace_enable (traced build only)
int g_trace_cap = 0;

// per-call timing events (attn_profile_*)
struct ProfileRec {
  cudaEvent_t start = nullptr, mid = nullptr, end = nullptr;
  int device = 0;
};
std::vector<ProfileRec> g_prof;
int g_prof_next = 0;
int g_prof_cap = 0;

void profile_free() {
  for (ProfileRec& r : g_prof) {
    if (r.start) cudaEventDestroy(r.start);
    if (r.mid) cudaEventDestroy(r.mid);
    if (r.end) cudaEventDestroy(r.end);
  }
  g_prof.clear();
  g_prof_next = 0;
  g_prof_cap = 0;
}

// Returns the record for this call, or nullptr when profiling is off or full.
ProfileRec* profile_slot(int dev) {
  if (g_prof_next >= g_prof_cap) return nullptr;
  ProfileRec& r = g_prof[g_prof_next];
  if (!r.start) {
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.mid) != cudaSuccess ||
        cudaEventCreate(&r.end) != cudaSuccess)
      return nullptr;
    r.device = dev;
  }
  ++g_prof_next;
  return &r;
}
std::atomic<int> g_last_dev_err{0};
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

using MapKey = std::tuple<uintptr_t, int, int, int, int, int, int, int>;   // ptr, dtype, d, H, L, B, box heads, box rows
using PlanKey = std::tuple<int, int, int, int, int, int, int>;   // B, Hq, Hkv, Lq, Lk, d, causal

constexpr size_t kMaxPlans = 256;   // schedules cached per device and kernel

// A schedule and its device copy.  The copy is written in stream order by an
// upload kernel (the values travel in its parameters), so the first call of a
// shape neither synchronises nor copies from pageable memory.
struct DevPlan {
  Plan host;
  std::vector<int> flat;   // units (kUnitInts each) | CTA or pair offsets | split groups (kGroupInts each)
  size_t off_cta = 0, off_groups = 0;
  int* dbuf = nullptr;
  bool async_alloc = false;   // dbuf from cudaMallocAsync (else cudaMalloc, during a capture)
  bool pinned = false;        // a captured graph reads dbuf: kept until the process exits
  bool uploaded = false;      // an upload outside any capture has been enqueued
  cudaStream_t up_stream = nullptr;
  cudaEvent_t ready = nullptr;                                // after that upload
  std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;     // last launch on each stream
  uint64_t lru = 0;
  const int* units() const { return dbuf; }
  const int* cta_off() const { return dbuf + off_cta; }
  const int* groups() const { return dbuf + off_groups; }
};

// A library-owned device buffer grown on demand.  Growth never frees a buffer
// mid-stream: the old one is released with cudaFreeAsync on the calling
// stream (ordered after the calls that used it, which the header requires to
// be ordered before this one), or kept for the life of the process if a
// captured graph may still use it.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  bool async_alloc = false;
  bool pinned = false;
  std::vector<void*> kept;
};

struct DevState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  int* err_word = nullptr;
  std::map<MapKey, CUtensorMap> maps;
  LruCache<PlanKey, DevPlan> plans{kMaxPlans};        // single-CTA kernel schedules
  LruCache<PlanKey, DevPlan> pair_plans{kMaxPlans};   // CTA-pair kernel schedules
  LruCache<PlanKey, DevPlan> cluster_plans{kMaxPlans};   // in-cluster merge schedules (causal + 2 * cluster size)
  Workspace part;        // single-CTA split pieces: O_s then (m, l)
  Workspace pair_part;   // CTA-pair split pieces: u then (m, l)
  Workspace pair_cnt;    // CTA-pair merge counters (epoch-tagged words, zeroed when allocated)
  unsigned int epoch = 0;
  Workspace rope_tab;    // attn_fwd_rope: the (cos, sin) table ...
  int rope_rot = 0, rope_npos = 0;   // ... for this rotary dimension and positions 0 .. rope_npos - 1
  float rope_base = 0.0f;
  Workspace rope_k;      // attn_fwd_rope: the rotated keys
};

std::map<int, DevState> g_dev;

int init_device(int dev, DevState& st) {
  if (st.ready) return ATTN_OK;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_ELAUNCH;
  st.sm_count = prop.multiProcessorCount;
  st.supported = (prop.major == 10 && prop.minor == 3);
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word), g_attn_err) != cudaSuccess) return ATTN_ELAUNCH;
  if (!get_encode()) return ATTN_ELAUNCH;
  st.ready = true;
  return ATTN_OK;
}

// 4-D map over (d, H, L, B) for a contiguous (B, L, H, d) 16-bit tensor,
// box box_inner x box_h x (box_rows / box_h) x 1, 128-byte swizzle: rows
// ordered (position, head) with the head fastest.
int get_map(DevState& st, const void* ptr, bool bf16, int d, int H, int L, int B, CUtensorMap& out, int box_h = 1,
            int box_rows = kBM, int box_inner = 64) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), bf16 ? 1 : 0, d, H, L, B, box_h, box_rows * 1024 + box_inner};
  auto it = st.maps.find(key);
  if (it != st.maps.end()) {
    out = it->second;
    return ATTN_OK;
  }
  CUtensorMap m;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(L) * H * d * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_h),
                             static_cast<cuuint32_t>(box_rows / box_h), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(&m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return ATTN_EINVAL;
  if (st.maps.size() > 4096) st.maps.clear();   // host memory only
  st.maps.emplace(key, m);
  out = m;
  return ATTN_OK;
}

// cudaMalloc inside a stream capture: the calling thread's capture mode is
// relaxed for the call (allocation is otherwise refused under the global
// mode), then restored.
cudaError_t malloc_in_capture(void** p, size_t bytes) {
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  const cudaError_t e = cudaMalloc(p, bytes);
  cudaThreadExchangeStreamCaptureMode(&mode);
  return e;
}

// True while `stream` is being captured into a graph (or when that cannot be
// told, which is treated the same way: nothing is freed or evicted).
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// ---- stream-ordered upload of int arrays: the values ride in the kernel's
// parameters (up to 28 KB per launch), so no host buffer has to outlive the
// call and the copy is captured like any kernel.
constexpr int kUploadInts = 7168;
struct UploadParams {
  int* dst;
  int n;
  int data[kUploadInts];
};
__global__ void __launch_bounds__(256) upload_kernel(const __grid_constant__ UploadParams p) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += gridDim.x * blockDim.x) p.dst[i] = p.data[i];
}

}  // namespace

int upload_ints(int* dst, const int* src, size_t n, cudaStream_t stream) {
  static thread_local UploadParams p;
  for (size_t off = 0; off < n; off += kUploadInts) {
    const int cnt = static_cast<int>(std::min<size_t>(kUploadInts, n - off));
    p.dst = dst + off;
    p.n = cnt;
    std::memcpy(p.data, src + off, static_cast<size_t>(cnt) * sizeof(int));
    upload_kernel<<<(cnt + 255) / 256, 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
    g_launches.fetch_add(1);
  }
  return ATTN_OK;
}

namespace {

void release_plan(DevPlan& pl, cudaStream_t stream) {
  // the free is ordered after the upload and after every launch that read it
  if (pl.ready) {
    cudaStreamWaitEvent(stream, pl.ready, 0);
    cudaEventDestroy(pl.ready);
  }
  for (auto& u : pl.uses) {
    cudaStreamWaitEvent(stream, u.second, 0);
    cudaEventDestroy(u.second);
  }
  if (pl.dbuf && pl.async_alloc) cudaFreeAsync(pl.dbuf, stream);
  pl.dbuf = nullptr;
}

// The device copy of `key`'s schedule, current on `stream` when the call's
// kernels run.  `make` builds the host plan.
// A schedule that `inline_ok` accepts travels in the kernel parameters and
// gets no device copy.
template <class MakeFn, class InlineFn>
int get_plan(LruCache<PlanKey, DevPlan>& cache, const PlanKey& key, cudaStream_t stream, MakeFn make,
             InlineFn inline_ok, DevPlan*& out) {
  const bool cap = capturing(stream);
  DevPlan* pl = cache.find(key);
  if (!pl) {
    auto dp = std::make_unique<DevPlan>();
    if (!make(dp->host)) return ATTN_EINVAL;
    const Plan& h = dp->host;
    std::vector<int>& f = dp->flat;
    f.reserve(h.units.size() * kUnitInts + h.cta_off.size() + h.groups.size() * kGroupInts);
    for (const PlanUnit& u : h.units) {
      const int e[kUnitInts] = {u.bh, u.m_block, u.kv_begin, u.kv_end, u.split, u.n_split, u.slot, u.cta};
      f.insert(f.end(), e, e + kUnitInts);
    }
    dp->off_cta = f.size();
    f.insert(f.end(), h.cta_off.begin(), h.cta_off.end());
    dp->off_groups = f.size();
    for (const PlanGroup& g : h.groups) {
      const int e[kGroupInts] = {g.bh, g.m_block, g.slot_base, g.n_split};
      f.insert(f.end(), e, e + kGroupInts);
    }
    const size_t bytes = f.size() * sizeof(int);
    if (inline_ok(dp->host)) {
      // no device copy
    } else if (cap) {
      if (malloc_in_capture(reinterpret_cast<void**>(&dp->dbuf), bytes) != cudaSuccess) return ATTN_ENOMEM;
    } else {
      if (cudaMallocAsync(reinterpret_cast<void**>(&dp->dbuf), bytes, stream) != cudaSuccess) return ATTN_ENOMEM;
      dp->async_alloc = true;
    }
    pl = cache.insert(key, std::move(dp), !cap, [&](DevPlan& v) { release_plan(v, stream); });
  }
  if (!pl->dbuf) {
    // inline schedule
  } else if (cap) {
    // the graph carries its own upload, re-run at every replay
    pl->pinned = true;
    if (int rc = upload_ints(pl->dbuf, pl->flat.data(), pl->flat.size(), stream)) return rc;
  } else if (!pl->uploaded) {
    if (int rc = upload_ints(pl->dbuf, pl->flat.data(), pl->flat.size(), stream)) return rc;
    if (!pl->ready && cudaEventCreateWithFlags(&pl->ready, cudaEventDisableTiming) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaEventRecord(pl->ready, stream) != cudaSuccess) return ATTN_ELAUNCH;
    pl->uploaded = true;
    pl->up_stream = stream;
  } else if (pl->up_stream != stream) {
    if (cudaStreamWaitEvent(stream, pl->ready, 0) != cudaSuccess) return ATTN_ELAUNCH;
  }
  out = pl;
  return ATTN_OK;
}

// Records, outside captures, that the kernels just enqueued on `stream` read
// `pl` (its memory is freed only after them).
void note_use(DevPlan* pl, cudaStream_t stream) {
  if (!pl || !pl->dbuf || pl->pinned || capturing(stream)) return;
  for (auto& u : pl->uses)
    if (u.first == stream) {
      cudaEventRecord(u.second, stream);
      return;
    }
  cudaEvent_t e;
  if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return;
  cudaEventRecord(e, stream);
  pl->uses.emplace_back(stream, e);
}

int ws_ensure(Workspace& w, size_t need, cudaStream_t stream, bool zero) {
  const bool cap = capturing(stream);
  if (need <= w.bytes) {
    if (cap) w.pinned = true;
    return ATTN_OK;
  }
  const size_t nb = std::max(need, 2 * w.bytes);
  void* np = nullptr;
  if (cap) {
    if (malloc_in_capture(&np, nb) != cudaSuccess) return ATTN_ENOMEM;
  } else {
    if (cudaMallocAsync(&np, nb, stream) != cudaSuccess) return ATTN_ENOMEM;
  }
  if (zero && cudaMemsetAsync(np, 0, nb, stream) != cudaSuccess) return ATTN_ELAUNCH;
  if (w.ptr) {
    if (w.pinned || !w.async_alloc || cap)
      w.kept.push_back(w.ptr);
    else
      cudaFreeAsync(w.ptr, stream);
  }
  w.ptr = np;
  w.bytes = nb;
  w.async_alloc = !cap;
  w.pinned = cap;
  return ATTN_OK;
}

// The dense forward on CTA pairs (head_dim 128): split pieces are merged
// inside the kernel, so one launch per call.
int fwd_pair(DevState& st, int dev, bool bf16, const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int Lq, int Lk, int d, bool causal, float scale, cudaStream_t stream) {
  const PlanKey key{B, Hq, Hkv, Lq, Lk, d, causal ? 1 : 0};
  auto fits = [](const Plan& h) {
    return static_cast<int>(h.units.size()) <= kPairInlineUnits && h.n_ctas <= kInlinePairs;
  };
  DevPlan* pl = nullptr;
  int rc = get_plan(
      st.pair_plans, key, stream,
      [&](Plan& h) { return make_plan_pair(B, Hq, Hkv, Lq, Lk, causal, st.sm_count / 2, h); }, fits, pl);
  if (rc) return rc;
  static thread_local PairParams p;
  std::memset(&p, 0, sizeof(p));
  const int Lk_map = Lk > 0 ? Lk : 1;
  if ((rc = get_map(st, q, bf16, d, Hq, Lq, B, p.tm_q))) return rc;
  if ((rc = get_map(st, k, bf16, d, Hkv, Lk_map, B, p.tm_k))) return rc;
  if ((rc = get_map(st, v, bf16, d, Hkv, Lk_map, B, p.tm_v, 1, kPairBN, d / 2))) return rc;
  if ((rc = get_map(st, o, bf16, d, Hq, Lq, B, p.tm_o))) return rc;
  p.o = o;
  p.lse = lse;
  const Plan& h = pl->host;
  if (h.n_partials > 0) {
    const size_t n = static_cast<size_t>(h.n_partials);
    const size_t u_bytes = n * 2 * kPairRows * d * 4;
    const size_t ml_bytes = n * 2 * kPairRows * 2 * sizeof(float);
    if ((rc = ws_ensure(st.pair_part, u_bytes + ml_bytes, stream, false))) return rc;
    if ((rc = ws_ensure(st.pair_cnt, n * 2 * sizeof(unsigned long long), stream, true))) return rc;
    p.part_u = static_cast<float*>(st.pair_part.ptr);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(st.pair_part.ptr) + u_bytes);
    p.counters = static_cast<unsigned long long*>(st.pair_cnt.ptr);
  }
  if (++st.epoch == 0) st.epoch = 1;
  p.epoch = st.epoch;
  p.err = st.err_word;
  p.trace = g_trace;
  p.trace_cap = g_trace_cap;
  p.timeout_ns = g_timeout_ns.load();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.group = Hq / Hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (fits(h)) {
    p.n_inline = 1;
    std::memcpy(p.units_inline, pl->flat.data(), h.units.size() * kUnitInts * sizeof(int));
    std::memcpy(p.pair_off_inline, h.cta_off.data(), h.cta_off.size() * sizeof(int));
  } else {
    p.units = pl->units();
    p.pair_off = pl->cta_off();
  }
  if (h.n_ctas <= 0) return ATTN_OK;
  ProfileRec* prof = profile_slot(dev);
  if (prof && cudaEventRecord(prof->start, stream) != cudaSuccess) return ATTN_ELAUNCH;
  if (pair_launcher_d128(bf16, causal)(p, h.n_ctas, h.n_partials > 0, stream) != cudaSuccess) return ATTN_ELAUNCH;
  g_launches.fetch_add(1);
  note_use(pl, stream);
  if (prof && (cudaEventRecord(prof->mid, stream) != cudaSuccess || cudaEventRecord(prof->end, stream) != cudaSuccess))
    return ATTN_ELAUNCH;
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The rotary embedding of Q applied inside the forward kernel (attn_fwd_rope).
struct RopeArgs {
  const float2* cs;   // the (cos, sin) table
  int rot, gptj, q_offset;
};

int fwd(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
        int Lq, int Lk, int d, int causal, float scale, const int* cu, const int* cu_k, cudaStream_t stream,
        const RopeArgs* rope = nullptr) {
  // ---- host-side argument checks (nothing is enqueued on failure)
  if (!q || !k || !v || !o || !lse) return ATTN_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4)) return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0) return ATTN_EINVAL;
  if (Hq % Hkv != 0) return ATTN_EINVAL;
  if (causal != 0 && causal != 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_EINVAL;
  if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
  const bool varlen = cu != nullptr;
  if (!varlen && cu_k != nullptr) return ATTN_EINVAL;
  // queries with their own key offsets (cross-attention, a key/value cache):
  // key counts may differ widely between sequences
  const bool own_keys = varlen && cu_k != nullptr && cu_k != cu;
  if (varlen) {
    // one offsets array serves queries and keys (self-attention) unless the
    // keys have their own (cross-attention, a key/value cache)
    if ((cu_k == nullptr && Lq != Lk) || B > kVarlenMaxB) return ATTN_EINVAL;
    if (cu_k == nullptr) cu_k = cu;
  }
  // sizes: TMA coordinates and the kernel's row arithmetic are 32-bit
  const long long rows_q = varlen ? static_cast<long long>(Lq) : static_cast<long long>(B) * Lq;
  const long long rows_k = varlen ? static_cast<long long>(Lk) : static_cast<long long>(B) * Lk;
  if (rows_q * Hq > (1LL << 31) - 1 || rows_k * Hkv > (1LL << 31) - 1) return ATTN_EINVAL;
  if (static_cast<long long>(Lq) + kBlockRows > (1LL << 30) || static_cast<long long>(Lk) + kBN > (1LL << 30))
    return ATTN_EINVAL;
  if (Lq == 0) return ATTN_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  int rc = init_device(dev, st);
  if (rc) return rc;
  if (!st.supported) return ATTN_EUNSUPPORTED;
  if (!varlen && !rope && d == 128 && g_pair_forward.load() != 0 && st.sm_count >= 2)
    return fwd_pair(st, dev, bf16, q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal != 0, scale, stream);

  static thread_local FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int Lk_map = Lk > 0 ? Lk : 1;
  const int Bm = varlen ? 1 : B;
  // Packed sequences with grouped heads: the group's query heads share each
  // tile (128 / group positions x group heads), so a key/value tile is read
  // once per group instead of once per head, and a short query (one decode
  // token) fills group rows of the tile instead of one.  Never more units
  // than one head per tile; a group of 2 to 32 heads, a power of two.
  const int group = Hq / Hkv;
  int pack_log2 = 0;
  if (varlen && group >= 2 && group <= 32 && (group & (group - 1)) == 0)
    while ((1 << pack_log2) < group) ++pack_log2;
  if ((rc = get_map(st, q, bf16, d, Hq, Lq, Bm, p.tm_q, 1 << pack_log2))) return rc;
  if ((rc = get_map(st, k, bf16, d, Hkv, Lk_map, Bm, p.tm_k))) return rc;
  if ((rc = get_map(st, v, bf16, d, Hkv, Lk_map, Bm, p.tm_v))) return rc;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu;
  p.cu_seqlens_k = cu_k;
  p.err = st.err_word;
  p.trace = g_trace;
  p.trace_cap = g_trace_cap;
  p.timeout_ns = g_timeout_ns.load();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.group = group;
  p.pack_log2 = pack_log2;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;

  FwdLauncher launch = (d == 64) ? fwd_launcher_d64(bf16, causal != 0, varlen)
                                 : fwd_launcher_d128(bf16, causal != 0, varlen);
  if (own_keys && B <= kVarlenSortMax)
    launch = (d == 64) ? fwd_sorted_launcher_d64(bf16, causal != 0) : fwd_sorted_launcher_d128(bf16, causal != 0);
  if (rope) {
    p.rope_cs = reinterpret_cast<const float*>(rope->cs);
    p.rope_rot = rope->rot;
    p.rope_gptj = rope->gptj;
    p.rope_qoff = rope->q_offset;
    launch = (d == 64) ? fwd_rope_launcher_d64(bf16, causal != 0) : fwd_rope_launcher_d128(bf16, causal != 0);
  }
  int grid = 0;
  DevPlan* plan = nullptr;
  const int cs = (!varlen && !rope) ? g_cluster_merge.load() : 0;
  if (cs > 0) {
    // in-cluster merge: equal pieces, one per CTA of a cluster of cs
    const PlanKey key{B, Hq, Hkv, Lq, Lk, d, causal + 2 * cs};
    auto fits = [](const Plan& h) {
      return static_cast<int>(h.units.size()) <= kInlineUnits && h.n_ctas <= kInlineCtas;
    };
    rc = get_plan(
        st.cluster_plans, key, stream,
        [&](Plan& h) { return make_plan_cluster(B, Hq, Hkv, Lq, Lk, causal != 0, cs, h); }, fits, plan);
    if (rc) return rc;
    if (fits(plan->host)) {
      p.n_inline = 1;
      std::memcpy(p.units_inline, plan->flat.data(), plan->host.units.size() * kUnitInts * sizeof(int));
      std::memcpy(p.cta_off_inline, plan->host.cta_off.data(), plan->host.cta_off.size() * sizeof(int));
    } else {
      p.units = plan->units();
      p.cta_off = plan->cta_off();
    }
    p.cluster_merge = cs;
    grid = plan->host.n_ctas;
  } else if (!varlen) {
    const PlanKey key{B, Hq, Hkv, Lq, Lk, d, causal};
    // the combine pass reads the split groups from the device copy
    auto fits = [](const Plan& h) {
      return h.groups.empty() && static_cast<int>(h.units.size()) <= kInlineUnits && h.n_ctas <= kInlineCtas;
    };
    rc = get_plan(
        st.plans, key, stream,
        [&](Plan& h) { return make_plan(B, Hq, Hkv, Lq, Lk, d, causal != 0, st.sm_count, h); }, fits, plan);
    if (rc) return rc;
    if (plan->host.n_partials > 0) {
      const size_t n = static_cast<size_t>(plan->host.n_partials);
      const size_t o_bytes = n * kNSub * kBM * d * 4;   // fp32
      const size_t ml_bytes = n * kNSub * kBM * 2 * sizeof(float);
      if ((rc = ws_ensure(st.part, o_bytes + ml_bytes, stream, false))) return rc;
      p.part_o = st.part.ptr;
      p.part_ml = reinterpret_cast<float*>(static_cast<char*>(st.part.ptr) + o_bytes);
    }
    if (static_cast<int>(plan->host.units.size()) <= kInlineUnits && plan->host.n_ctas <= kInlineCtas) {
      p.n_inline = 1;
      std::memcpy(p.units_inline, plan->flat.data(), plan->host.units.size() * kUnitInts * sizeof(int));
      std::memcpy(p.cta_off_inline, plan->host.cta_off.data(), plan->host.cta_off.size() * sizeof(int));
    } else {
      p.units = plan->units();
      p.cta_off = plan->cta_off();
    }
    grid = plan->host.n_ctas;
  } else {
    // units = sum over sequences of Hq * ceil(len / 256) <= Hq * (B + ceil(total / 256));
    // packed heads give (Hq / g) * ceil(len * g / 256), never more
    const long long bound = static_cast<long long>(Hq) * (B + (Lq + kBlockRows - 1) / kBlockRows);
    grid = static_cast<int>(std::min<long long>(st.sm_count, bound));
  }
  if (grid <= 0) return ATTN_OK;
  ProfileRec* prof = profile_slot(dev);
  if (prof && cudaEventRecord(prof->start, stream) != cudaSuccess) return ATTN_ELAUNCH;
  if (launch(p, grid, stream) != cudaSuccess) return ATTN_ELAUNCH;
  g_launches.fetch_add(1);
  if (prof && cudaEventRecord(prof->mid, stream) != cudaSuccess) return ATTN_ELAUNCH;
  if (plan && !plan->host.groups.empty()) {
    CombineParams cp;
    cp.groups = plan->groups();
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.o = o;
    cp.lse = lse;
    cp.Hq = Hq;
    cp.Lq = Lq;
    CombineLauncher cl = (d == 64) ? combine_launcher_d64(bf16) : combine_launcher_d128(bf16);
    if (cl(cp, static_cast<int>(plan->host.groups.size()), stream) != cudaSuccess) return ATTN_ELAUNCH;
    g_launches.fetch_add(1);
  }
  note_use(plan, stream);
  if (prof && cudaEventRecord(prof->end, stream) != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

// One decoding step through the packed forward's tensor-core tiles: decode
// mode of the varlen kernel (query b at row b, the group's query heads in
// one tile) with every cache cut into pieces when the (sequence, head group)
// units alone would leave SMs idle; the pieces' partials are merged by the
// decode combine.  Arguments are checked by attn_decode.
int fwd_decode(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
               int total_k, int d, float scale, const int* cu_k, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  int rc = init_device(dev, st);
  if (rc) return rc;
  if (!st.supported) return ATTN_EUNSUPPORTED;
  const int group = Hq / Hkv;
  int lp = 0;
  while ((1 << lp) < group) ++lp;
  const int n_hg = Hq >> lp;
  // head_dim 64 and 128 run the transposed decode kernel (keys on the MMA's
  // M dimension); other head dims, or more sequences than its prefix table
  // holds, the packed forward in decode mode.  The transposed kernel's
  // softmax step covers 256 keys at head_dim 64, 128 otherwise.
  const bool transposed = (d == 64 || d == 128) && B <= decode_tc_max_b(d);
  const long long step_keys = (transposed && d == 64) ? 2 * kBN : kBN;
  // Pieces per cache: the units (B x n_hg x pieces) run in rounds of one per
  // CTA, so with caches of equal length (the host cannot read cu_seqlens_k;
  // the mean length stands in) the call costs rounds x (steps per piece +
  // kDecodeUnitCost), a unit's fixed cost (Q load, pipeline fill, epilogue)
  // in step-times.  The piece count that minimises it wins, fewer pieces on
  // ties; split = 0 leaves every cache whole, else it counts key tiles (whole
  // steps).  `tiles` bounds the sum over sequences of their key tiles (a
  // partial tile per sequence at most).
  const long long units0 = static_cast<long long>(B) * n_hg;
  const long long tiles = (static_cast<long long>(total_k) + kBN - 1) / kBN + B;
  const long long t_seq =
      std::max<long long>(1, ((static_cast<long long>(total_k) + B - 1) / B + step_keys - 1) / step_keys);
  const long long grid_max = st.sm_count;
  constexpr double kDecodeUnitCost = 1.5;
  long long best_pcs = 1;
  double best = 1e300;
  for (long long pcs = 1; pcs <= std::min<long long>(t_seq, 4096); ++pcs) {
    const long long rounds = (units0 * pcs + grid_max - 1) / grid_max;
    const double cost = static_cast<double>(rounds) * (static_cast<double>((t_seq + pcs - 1) / pcs) + kDecodeUnitCost);
    if (cost < best * (1.0 - 1e-9)) {
      best = cost;
      best_pcs = pcs;
    }
  }
  const int split = best_pcs > 1 ? static_cast<int>((t_seq + best_pcs - 1) / best_pcs * (step_keys / kBN)) : 0;
  const long long max_units = split > 0 ? static_cast<long long>(n_hg) * (tiles / split + 1 + B) : units0;
  if (max_units > (1LL << 30)) return ATTN_EINVAL;

  static thread_local FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (transposed) {
    if ((rc = get_map(st, q, bf16, d, Hq, B, 1, p.tm_q, group, group))) return rc;
  } else {
    if ((rc = get_map(st, q, bf16, d, Hq, B, 1, p.tm_q, 1 << lp))) return rc;
  }
  if ((rc = get_map(st, k, bf16, d, Hkv, total_k, 1, p.tm_k))) return rc;
  if ((rc = get_map(st, v, bf16, d, Hkv, total_k, 1, p.tm_v))) return rc;
  // workspace: the unit prefix and malformed flag (B + 2 ints), then the
  // pieces' (m, l) and fp32 partial outputs in the forward's slot layout
  const size_t pref_bytes = (static_cast<size_t>(B + 2) * sizeof(int) + 255) & ~size_t(255);
  const size_t ml_bytes = split > 0 ? static_cast<size_t>(max_units) * kNSub * kBM * 2 * sizeof(float) : 0;
  const size_t o_bytes = split > 0 ? static_cast<size_t>(max_units) * kNSub * kBM * d * sizeof(float) : 0;
  if ((rc = ws_ensure(st.part, pref_bytes + ml_bytes + o_bytes, stream, false))) return rc;
  char* ws = static_cast<char*>(st.part.ptr);
  p.vl_pref_out = reinterpret_cast<int*>(ws);
  p.part_ml = reinterpret_cast<float*>(ws + pref_bytes);
  p.part_o = ws + pref_bytes + ml_bytes;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = nullptr;
  p.cu_seqlens_k = cu_k;
  p.err = st.err_word;
  p.trace = g_trace;
  p.trace_cap = g_trace_cap;
  p.timeout_ns = g_timeout_ns.load();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = B;
  p.Lk = total_k;
  p.group = group;
  p.pack_log2 = lp;
  p.vl_decode = 1;
  p.vl_split = split;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  FwdLauncher launch = (d == 64) ? fwd_launcher_d64(bf16, false, true) : fwd_launcher_d128(bf16, false, true);
  // The units run in rounds of one per CTA.  With units of equal cost (the
  // mean cache length), a last round shorter than the grid leaves SMs idle
  // while the others run their extra unit at the per-SM rate, below what HBM
  // gives when every SM streams.  The smallest grid that keeps the same
  // number of rounds gives every CTA the same number of units; it is taken
  // when it keeps at least 80 % of the SMs (fewer SMs stream below the HBM
  // rate: 256 units on 128 CTAs ran 2-4 % faster than on 152, 192 units on
  // 96 CTAs 2-3 % slower).
  const long long units_est = units0 * best_pcs;
  const long long rounds_est = (units_est + st.sm_count - 1) / st.sm_count;
  const long long grid_even = (units_est + rounds_est - 1) / rounds_est;
  const int grid = static_cast<int>(std::min<long long>(
      std::min<long long>(st.sm_count, max_units), 5 * grid_even >= 4LL * st.sm_count ? grid_even : st.sm_count));
  ProfileRec* prof = profile_slot(dev);
  if (prof && cudaEventRecord(prof->start, stream) != cudaSuccess) return ATTN_ELAUNCH;
  const cudaError_t le = transposed
                             ? launch_decode_tc(p.tm_q, p.tm_k, p.tm_v, o, lse, cu_k, p.vl_pref_out, p.part_o,
                                                p.part_ml, p.err, p.timeout_ns, B, Hq, Hkv, total_k, split,
                                                p.scale_log2, bf16, d, grid, stream)
                             : launch(p, grid, stream);
  if (le != cudaSuccess) return ATTN_ELAUNCH;
  g_launches.fetch_add(1);
  if (prof && cudaEventRecord(prof->mid, stream) != cudaSuccess) return ATTN_ELAUNCH;
  if (split > 0) {
    DecodeCombineParams cp;
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.pref = p.vl_pref_out;
    cp.cu_seqlens_k = cu_k;
    cp.o = o;
    cp.lse = lse;
    cp.B = B;
    cp.Hq = Hq;
    cp.pack_log2 = lp;
    cp.split = split;
    DecodeCombineLauncher cl = (d == 64) ? decode_combine_launcher_d64(bf16) : decode_combine_launcher_d128(bf16);
    if (cl(cp, B * n_hg, stream) != cudaSuccess) return ATTN_ELAUNCH;
    g_launches.fetch_add(1);
  }
  if (prof && cudaEventRecord(prof->end, stream) != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

bool decode_tensor_cores() { return g_decode_tc.load() != 0; }

// attention(rope(q, q_offset + i), rope(k, j), v): K through the rotary pass
// into a library workspace, Q rotated by the forward kernel in shared memory
// at the start of every unit, from a cached (cos, sin) table.
int fwd_rope(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
             int Lq, int Lk, int d, int causal, float scale, int rot, float base, int gptj, int q_offset,
             cudaStream_t stream) {
  if (!q || !k || !v) return ATTN_EINVAL;
  if (rot <= 0 || rot > d || rot % 16 != 0 || !(base > 1.0f) || !std::isfinite(base)) return ATTN_EINVAL;
  if ((gptj != 0 && gptj != 1) || q_offset < 0 || B <= 0 || Hkv <= 0 || Lk < 0 || Lq < 0) return ATTN_EINVAL;
  if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
  if (static_cast<long long>(Lq) + q_offset > (1LL << 30)) return ATTN_EINVAL;
  if (Lq == 0) return ATTN_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  const int n_pos = std::max(1, std::max(Lk, Lq + q_offset));
  const size_t k_bytes = static_cast<size_t>(B) * Lk * Hkv * d * 2;
  const float2* cs = nullptr;
  void* k_rot = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevState& st = g_dev[dev];
    int rc = init_device(dev, st);
    if (rc) return rc;
    if (!st.supported) return ATTN_EUNSUPPORTED;
    // the table, recomputed only when the rotation or the positions it covers change
    if (st.rope_rot != rot || st.rope_base != base || st.rope_npos < n_pos) {
      const int np = std::max(n_pos, st.rope_rot == rot && st.rope_base == base ? 2 * st.rope_npos : n_pos);
      if ((rc = ws_ensure(st.rope_tab, static_cast<size_t>(np) * (rot / 2) * sizeof(float2), stream, false))) return rc;
      if ((rc = rope_table(static_cast<float2*>(st.rope_tab.ptr), np, rot, base, stream))) return rc;
      st.rope_rot = rot;
      st.rope_base = base;
      st.rope_npos = np;
    } else if (capturing(stream)) {
      st.rope_tab.pinned = true;
    }
    cs = static_cast<const float2*>(st.rope_tab.ptr);
    if (k_bytes > 0) {
      if ((rc = ws_ensure(st.rope_k, k_bytes, stream, false))) return rc;
      k_rot = st.rope_k.ptr;
    }
  }
  if (k_bytes > 0) {
    const int rc = attn_rotary(k, k_rot, B, Lk, Hkv, d, rot, base, gptj, nullptr, 0, nullptr, bf16 ? 0 : 1, stream);
    if (rc) return rc;
  }
  const RopeArgs ra{cs, rot, gptj, q_offset};
  return fwd(bf16, q, k_bytes > 0 ? k_rot : k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal, scale, nullptr, nullptr,
             stream, &ra);
}

__global__ void selftest_wait_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl wc{err, &abort_flag, timeout_ns};
  // nothing arrives on `bar`: the wait must run out and report
  mbar_wait(smem_u32(&bar), 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSelftest));
}

}  // namespace

int device_info(int dev, DeviceInfo& out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  const int rc = init_device(dev, st);
  if (rc) return rc;
  out.sm_count = st.sm_count;
  out.supported = st.supported;
  out.err_word = st.err_word;
  return ATTN_OK;
}

int encode_map(const void* ptr, bool bf16, int d, int H, int L, int B, CUtensorMap& out) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!get_encode()) return ATTN_ELAUNCH;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(L) * H * d * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(&out, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_EINVAL;
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }
unsigned long long* trace_buffer(int* events_per_stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  *events_per_stream = g_trace_cap;
  return g_trace;
}
void count_launch() { g_launches.fetch_add(1); }

int decode_on_tensor_cores(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                           int Hkv, int total_k, int d, float scale, const int* cu_k, cudaStream_t stream) {
  return fwd_decode(bf16, q, k, v, o, lse, B, Hq, Hkv, total_k, d, scale, cu_k, stream);
}
bool decode_tensor_cores_enabled() { return decode_tensor_cores(); }

cudaError_t launch_selftest_wait(int* err_word, unsigned long long timeout_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err_word, timeout_ns);
  return cudaGetLastError();
}

}  // namespace attn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Lq,
             int Lk, int d, int causal, float scale, const int* cu_seqlens_or_null, cudaStream_t stream) {
  return attn::fwd(true, q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal, scale, cu_seqlens_or_null, nullptr, stream);
}

int attn_fwd_fp16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                  int Lq, int Lk, int d, int causal, float scale, const int* cu_seqlens_or_null,
                  cudaStream_t stream) {
  return attn::fwd(false, q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal, scale, cu_seqlens_or_null, nullptr,
                   stream);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                    int total_q, int total_k, int d, int causal, float scale, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int fp16, cudaStream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k || (fp16 != 0 && fp16 != 1)) return ATTN_EINVAL;
  return attn::fwd(fp16 == 0, q, k, v, o, lse, B, Hq, Hkv, total_q, total_k, d, causal, scale, cu_seqlens_q,
                   cu_seqlens_k, stream);
}

int attn_get_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ELAUNCH;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, attn::g_attn_err, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
  attn::g_last_dev_err.store(h);
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(attn::g_attn_err, &zero, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    return ATTN_EDEVICE;
  }
  return ATTN_OK;
}

int attn_last_device_error(void) { return attn::g_last_dev_err.load(); }

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported head_dim or device (needs head_dim 64/128 on sm_103)";
    case ATTN_ELAUNCH: return "CUDA launch or runtime failure";
    case ATTN_ENOMEM: return "workspace allocation failed";
    case ATTN_EDEVICE: return "a kernel reported a device-side error (see attn_last_device_error)";
    case ATTN_ETOOLARGE:
      return "problem needs more scratch than the static buffer of attn_fwd_noalloc holds; use attn_fwd";
    default: return "unknown error";
  }
}

void attn_set_wait_timeout_ns(unsigned long long ns) { attn::g_timeout_ns.store(ns < 1000 ? 1000 : ns); }

int attn_selftest_wait_timeout(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  std::lock_guard<std::mutex> lock(attn::g_mu);
  attn::DevState& st = attn::g_dev[dev];
  int rc = attn::init_device(dev, st);
  if (rc) return rc;
  return attn::launch_selftest_wait(st.err_word, attn::g_timeout_ns.load(), stream) == cudaSuccess ? ATTN_OK
                                                                                                   : ATTN_ELAUNCH;
}

unsigned long long attn_launch_count(void) { return attn::g_launches.load(); }

int attn_trace_enable(void* dev_buf, int events_per_stream) {
#if !defined(ATTN_TRACE) || !ATTN_TRACE
  (void)dev_buf;
  (void)events_per_stream;
  return ATTN_EUNSUPPORTED;   // trace points exist only in the traced build
#else
  std::lock_guard<std::mutex> lock(attn::g_mu);
  if (dev_buf == nullptr || events_per_stream <= 0) {
    attn::g_trace = nullptr;
    attn::g_trace_cap = 0;
    return ATTN_OK;
  }
  if (reinterpret_cast<uintptr_t>(dev_buf) % 16 != 0) return ATTN_EINVAL;
  attn::g_trace = static_cast<unsigned long long*>(dev_buf);
  attn::g_trace_cap = events_per_stream;
  return ATTN_OK;
#endif
}

int attn_profile_enable(int n) {
  std::lock_guard<std::mutex> lock(attn::g_mu);
  if (n < 0) return ATTN_EINVAL;
  if (static_cast<int>(attn::g_prof.size()) < n) {
    attn::g_prof.resize(static_cast<size_t>(n));
  }
  attn::g_prof_next = 0;
  attn::g_prof_cap = n;
  return ATTN_OK;
}

void attn_profile_disable(void) {
  std::lock_guard<std::mutex> lock(attn::g_mu);
  attn::profile_free();
}

int attn_profile_read(float* main_ms, float* call_ms, int max, int* n) {
  std::lock_guard<std::mutex> lock(attn::g_mu);
  if (!n || (max > 0 && (!main_ms || !call_ms))) return ATTN_EINVAL;
  const int cnt = attn::g_prof_next;
  *n = cnt;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return ATTN_ELAUNCH;
  for (int i = 0; i < cnt && i < max; ++i) {
    attn::ProfileRec& r = attn::g_prof[i];
    if (cudaSetDevice(r.device) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaEventSynchronize(r.end) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaEventElapsedTime(&main_ms[i], r.start, r.mid) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaEventElapsedTime(&call_ms[i], r.start, r.end) != cudaSuccess) return ATTN_ELAUNCH;
  }
  cudaSetDevice(prev);
  return ATTN_OK;
}

void attn_set_pair_forward(int enable) { attn::g_pair_forward.store(enable ? 1 : 0); }

void attn_set_cluster_merge(int cluster_size) {
  if (cluster_size == 0 || cluster_size == 2 || cluster_size == 4 || cluster_size == 8)
    attn::g_cluster_merge.store(cluster_size);
}
int attn_cluster_merge(void) { return attn::g_cluster_merge.load(); }

int attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Lq,
                  int Lk, int d, int causal, float scale, int rot_dim, float base, int interleaved, int q_offset,
                  int fp16, cudaStream_t stream) {
  if (fp16 != 0 && fp16 != 1) return ATTN_EINVAL;
  return attn::fwd_rope(fp16 == 0, q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal, scale, rot_dim, base, interleaved,
                        q_offset, stream);
}

void attn_set_decode_path(int tensor_cores) { attn::g_decode_tc.store(tensor_cores ? 1 : 0); }
int attn_decode_path(void) { return attn::g_decode_tc.load(); }

int attn_pair_forward_used(int d, int varlen) {
  return (attn::g_pair_forward.load() != 0 && d == 128 && varlen == 0) ? 1 : 0;
}

int attn_plan_pair(int B, int Hq, int Hkv, int Lq, int Lk, int causal, int num_pairs, int* units, int max_units,
                   int* n_units, int* n_pairs, int* n_partials) {
  if (!n_units || !n_pairs || !n_partials || (max_units > 0 && !units)) return ATTN_EINVAL;
  if (causal != 0 && causal != 1) return ATTN_EINVAL;
  attn::Plan pl;
  if (!attn::make_plan_pair(B, Hq, Hkv, Lq, Lk, causal != 0, num_pairs, pl)) return ATTN_EINVAL;
  *n_units = static_cast<int>(pl.units.size());
  *n_pairs = pl.n_ctas;
  *n_partials = pl.n_partials;
  if (static_cast<int>(pl.units.size()) > max_units) return ATTN_ENOMEM;
  for (size_t i = 0; i < pl.units.size(); ++i) {
    const attn::PlanUnit& u = pl.units[i];
    const int e[attn::kUnitInts] = {u.bh, u.m_block, u.kv_begin, u.kv_end, u.split, u.n_split, u.slot, u.cta};
    std::memcpy(units + i * attn::kUnitInts, e, sizeof(e));
  }
  return ATTN_OK;
}

int attn_cache_stats(int* plans, int* pinned) {
  if (!plans || !pinned) return ATTN_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  std::lock_guard<std::mutex> lock(attn::g_mu);
  attn::DevState& st = attn::g_dev[dev];
  int n = 0, pn = 0;
  auto count = [&](attn::DevPlan& e) {
    ++n;
    if (e.pinned) ++pn;
  };
  st.plans.for_each(count);
  st.pair_plans.for_each(count);
  *plans = n;
  *pinned = pn;
  return ATTN_OK;
}

int attn_selftest_plan_cache(int n_keys, int capacity, int pin_every, int* max_live, int* released) {
  // the cache policy alone, with host-side entries: no device memory
  if (!max_live || !released || n_keys < 0 || capacity <= 0) return ATTN_EINVAL;
  struct Fake {
    bool pinned = false;
    uint64_t lru = 0;
  };
  attn::LruCache<int, Fake> c(static_cast<size_t>(capacity));
  int rel = 0, mx = 0;
  auto release = [&](Fake&) { ++rel; };
  for (int i = 0; i < n_keys; ++i) {
    Fake* f = c.find(i % (2 * capacity + 7));
    if (!f) {
      auto e = std::make_unique<Fake>();
      e->pinned = pin_every > 0 && (i % pin_every) == 0;
      c.insert(i % (2 * capacity + 7), std::move(e), true, release);
    }
    mx = std::max(mx, static_cast<int>(c.size()));
  }
  *max_live = mx;
  *released = rel;
  return ATTN_OK;
}

int attn_plan(int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, int num_sms, int* units, int max_units,
              int* n_units, int* n_ctas, int* n_partials) {
  if (!n_units || !n_ctas || !n_partials || (max_units > 0 && !units)) return ATTN_EINVAL;
  if (causal != 0 && causal != 1) return ATTN_EINVAL;
  attn::Plan pl;
  if (!attn::make_plan(B, Hq, Hkv, Lq, Lk, d, causal != 0, num_sms, pl)) return ATTN_EINVAL;
  *n_units = static_cast<int>(pl.units.size());
  *n_ctas = pl.n_ctas;
  *n_partials = pl.n_partials;
  if (static_cast<int>(pl.units.size()) > max_units) return ATTN_ENOMEM;
  for (size_t i = 0; i < pl.units.size(); ++i) {
    const attn::PlanUnit& u = pl.units[i];
    const int e[attn::kUnitInts] = {u.bh, u.m_block, u.kv_begin, u.kv_end, u.split, u.n_split, u.slot, u.cta};
    std::memcpy(units + i * attn::kUnitInts, e, sizeof(e));
  }
  return ATTN_OK;
}

}  // extern "C"
