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
#include "attn_internal.h"
#include "attn_launch.h"
#include "attn_params.h"
#include "attn_plan.h"
#include "ptx.cuh"

namespace attn {

// First device-side error since the last attn_get_error() (0 = none).
__device__ int g_attn_err;

namespace {

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<unsigned long long> g_launches{0};
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

using MapKey = std::tuple<uintptr_t, int, int, int, int, int, int>;   // ptr, dtype, d, H, L, B, box heads
using PlanKey = std::tuple<int, int, int, int, int, int, int>;   // B, Hq, Hkv, Lq, Lk, d, causal

struct DevPlan {
  Plan host;
  std::vector<int> flat_units;   // kUnitInts per unit, the layout the kernel reads
  int* d_units = nullptr;
  int* d_cta_off = nullptr;
  int* d_groups = nullptr;
};

struct DevState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  int* err_word = nullptr;
  std::map<MapKey, CUtensorMap> maps;
  std::map<PlanKey, std::unique_ptr<DevPlan>> plans;
  void* part_o = nullptr;
  float* part_ml = nullptr;
  size_t part_o_bytes = 0, part_ml_bytes = 0;
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
// box 64 x box_h x (128 / box_h) x 1: one 128-byte swizzle atom wide and 128
// shared-memory rows high, rows ordered (position, head) with the head fastest.
int get_map(DevState& st, const void* ptr, bool bf16, int d, int H, int L, int B, CUtensorMap& out, int box_h = 1) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), bf16 ? 1 : 0, d, H, L, B, box_h};
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
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(kBM / box_h), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(&m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return ATTN_EINVAL;
  if (st.maps.size() > 4096) st.maps.clear();
  st.maps.emplace(key, m);
  out = m;
  return ATTN_OK;
}

int get_plan(DevState& st, int B, int Hq, int Hkv, int Lq, int Lk, int d, bool causal, cudaStream_t stream,
             DevPlan*& out) {
  const PlanKey key{B, Hq, Hkv, Lq, Lk, d, causal ? 1 : 0};
  auto it = st.plans.find(key);
  if (it != st.plans.end()) {
    out = it->second.get();
    return ATTN_OK;
  }
  auto dp = std::make_unique<DevPlan>();
  if (!make_plan(B, Hq, Hkv, Lq, Lk, d, causal, st.sm_count, dp->host)) return ATTN_EINVAL;
  const Plan& pl = dp->host;
  std::vector<int> units(pl.units.size() * kUnitInts);
  for (size_t i = 0; i < pl.units.size(); ++i) {
    const PlanUnit& u = pl.units[i];
    const int e[kUnitInts] = {u.bh, u.m_block, u.kv_begin, u.kv_end, u.split, u.n_split, u.slot, u.cta};
    std::memcpy(&units[i * kUnitInts], e, sizeof(e));
  }
  dp->flat_units = units;
  std::vector<int> groups(pl.groups.size() * kGroupInts);
  for (size_t i = 0; i < pl.groups.size(); ++i) {
    const PlanGroup& g = pl.groups[i];
    const int e[kGroupInts] = {g.bh, g.m_block, g.slot_base, g.n_split};
    std::memcpy(&groups[i * kGroupInts], e, sizeof(e));
  }
  auto upload = [&](const std::vector<int>& v, int*& dst) -> bool {
    if (v.empty()) return true;
    if (cudaMalloc(&dst, v.size() * sizeof(int)) != cudaSuccess) return false;
    return cudaMemcpy(dst, v.data(), v.size() * sizeof(int), cudaMemcpyHostToDevice) == cudaSuccess;
  };
  (void)stream;
  if (!upload(units, dp->d_units) || !upload(pl.cta_off, dp->d_cta_off) || !upload(groups, dp->d_groups)) {
    cudaFree(dp->d_units);
    cudaFree(dp->d_cta_off);
    cudaFree(dp->d_groups);
    return ATTN_ENOMEM;
  }
  if (st.plans.size() > 256) st.plans.clear();   // bounded cache (device buffers of dropped plans leak)
  out = dp.get();
  st.plans.emplace(key, std::move(dp));
  return ATTN_OK;
}

int ensure_workspace(DevState& st, int n_partials, int d) {
  const size_t need_o = static_cast<size_t>(n_partials) * kNSub * kBM * d * 2;   // fp16
  const size_t need_ml = static_cast<size_t>(n_partials) * kNSub * kBM * 2 * sizeof(float);
  if (need_o > st.part_o_bytes) {
    if (st.part_o) cudaFree(st.part_o);
    st.part_o = nullptr;
    st.part_o_bytes = 0;
    if (cudaMalloc(&st.part_o, need_o) != cudaSuccess) return ATTN_ENOMEM;
    st.part_o_bytes = need_o;
  }
  if (need_ml > st.part_ml_bytes) {
    if (st.part_ml) cudaFree(st.part_ml);
    st.part_ml = nullptr;
    st.part_ml_bytes = 0;
    if (cudaMalloc(&st.part_ml, need_ml) != cudaSuccess) return ATTN_ENOMEM;
    st.part_ml_bytes = need_ml;
  }
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int fwd(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
        int Lq, int Lk, int d, int causal, float scale, const int* cu, const int* cu_k, cudaStream_t stream) {
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

  FwdParams p;
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
  int grid = 0;
  DevPlan* plan = nullptr;
  if (!varlen) {
    if ((rc = get_plan(st, B, Hq, Hkv, Lq, Lk, d, causal != 0, stream, plan))) return rc;
    if (plan->host.n_partials > 0) {
      if ((rc = ensure_workspace(st, plan->host.n_partials, d))) return rc;
      p.part_o = st.part_o;
      p.part_ml = st.part_ml;
    }
    p.units = plan->d_units;
    p.cta_off = plan->d_cta_off;
    if (static_cast<int>(plan->host.units.size()) <= kInlineUnits && plan->host.n_ctas <= kInlineCtas) {
      p.n_inline = 1;
      std::memcpy(p.units_inline, plan->flat_units.data(), plan->flat_units.size() * sizeof(int));
      std::memcpy(p.cta_off_inline, plan->host.cta_off.data(), plan->host.cta_off.size() * sizeof(int));
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
    cp.groups = plan->d_groups;
    cp.part_o = st.part_o;
    cp.part_ml = st.part_ml;
    cp.o = o;
    cp.lse = lse;
    cp.Hq = Hq;
    cp.Lq = Lq;
    CombineLauncher cl = (d == 64) ? combine_launcher_d64(bf16) : combine_launcher_d128(bf16);
    if (cl(cp, static_cast<int>(plan->host.groups.size()), stream) != cudaSuccess) return ATTN_ELAUNCH;
    g_launches.fetch_add(1);
  }
  if (prof && cudaEventRecord(prof->end, stream) != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
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
