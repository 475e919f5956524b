// C ABI of the attention backward: argument checks, the tensor maps, the
// per-device workspace of the first pass and the three launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "attn.h"
#include "attn_bwd_launch.h"
#include "attn_internal.h"

namespace attn {
namespace {

// lse2 and D of the last call's shape, grown on demand and kept per device
struct BwdWorkspace {
  float* buf = nullptr;
  size_t floats = 0;
};
std::map<int, BwdWorkspace> g_bwd_ws;
std::mutex g_bwd_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Dense (cu_q null): q (B, Lq, Hq, d), k (B, Lk, Hkv, d).  Varlen: Lq and Lk
// are the packed row counts, q (Lq, Hq, d), k (Lk, Hkv, d), offsets cu_q and
// cu_k (B+1 each, on the device; never read here).
int bwd(bool bf16, const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
        void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
        const int* cu_q, const int* cu_k, cudaStream_t stream) {
  const bool varlen = cu_q != nullptr;
  if (varlen != (cu_k != nullptr)) return ATTN_EINVAL;
  // a tensor with no elements may be passed as a null pointer
  if (Lq != 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_EINVAL;
  if (Lk != 0 && (!k || !v || !dk || !dv)) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0 || Hq % Hkv != 0) return ATTN_EINVAL;
  if (causal != 0 && causal != 1) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_EINVAL;
  if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
  const long long rows_q = varlen ? Lq : static_cast<long long>(B) * Lq;
  const long long rows_k = varlen ? Lk : static_cast<long long>(B) * Lk;
  if (rows_q * Hq > (1LL << 31) - 1 || rows_k * Hkv > (1LL << 31) - 1) return ATTN_EINVAL;
  if (static_cast<long long>(Lq) + kBM > (1LL << 30) || static_cast<long long>(Lk) + kBN > (1LL << 30))
    return ATTN_EINVAL;
  const size_t row_bytes = static_cast<size_t>(d) * 2;
  if (Lq == 0 || Lk == 0) {
    // no (query, key) pair: every gradient is zero
    if (Lq != 0 && cudaMemsetAsync(dq, 0, static_cast<size_t>(rows_q) * Hq * row_bytes, stream) != cudaSuccess)
      return ATTN_ELAUNCH;
    if (Lk != 0 && (cudaMemsetAsync(dk, 0, static_cast<size_t>(rows_k) * Hkv * row_bytes, stream) != cudaSuccess ||
                    cudaMemsetAsync(dv, 0, static_cast<size_t>(rows_k) * Hkv * row_bytes, stream) != cudaSuccess))
      return ATTN_ELAUNCH;
    return ATTN_OK;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  DeviceInfo info;
  int rc = device_info(dev, info);
  if (rc) return rc;
  if (!info.supported) return ATTN_EUNSUPPORTED;

  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int Bm = varlen ? 1 : B;   // packed tensors are one (total, H, d) batch for TMA
  if ((rc = encode_map(q, bf16, d, Hq, Lq, Bm, p.tm_q))) return rc;
  if ((rc = encode_map(dout, bf16, d, Hq, Lq, Bm, p.tm_do))) return rc;
  if ((rc = encode_map(k, bf16, d, Hkv, Lk, Bm, p.tm_k))) return rc;
  if ((rc = encode_map(v, bf16, d, Hkv, Lk, Bm, p.tm_v))) return rc;
  p.n_qt = (Lq + kBM - 1) / kBM;
  p.n_kt = (Lk + kBN - 1) / kBN;
  p.Lq_pad = p.n_qt * kBM;
  if (!varlen && (p.n_qt > 65535 || p.n_kt > 65535)) return ATTN_EINVAL;   // grid.y
  // varlen: at most B + total / 128 tiles (each sequence's last tile may be partial)
  const long long qt_max = static_cast<long long>(B) + p.n_qt, kt_max = static_cast<long long>(B) + p.n_kt;
  if (varlen && (qt_max * Hq > (1LL << 31) - 1 || kt_max * Hkv > (1LL << 31) - 1)) return ATTN_EINVAL;
  const size_t vec_floats = varlen ? static_cast<size_t>(Hq) * qt_max * kBM : static_cast<size_t>(B) * Hq * p.Lq_pad;
  const size_t need = 2 * vec_floats + (varlen ? 2 * static_cast<size_t>(B + 1) : 0);   // + tile tables (ints)

  std::lock_guard<std::mutex> lock(g_bwd_mu);
  BwdWorkspace& ws = g_bwd_ws[dev];
  if (need > ws.floats) {
    if (ws.buf) cudaFree(ws.buf);
    ws.buf = nullptr;
    ws.floats = 0;
    if (cudaMalloc(&ws.buf, need * sizeof(float)) != cudaSuccess) return ATTN_ENOMEM;
    ws.floats = need;
  }
  p.lse2 = ws.buf;
  p.dvec = ws.buf + vec_floats;
  int* pref = varlen ? reinterpret_cast<int*>(ws.buf + 2 * vec_floats) : nullptr;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.tile_pref = pref;
  p.q = q;
  p.dout = dout;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.err = info.err_word;
  p.timeout_ns = wait_timeout_ns();
  p.trace = trace_buffer(&p.trace_cap);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.group = Hq / Hkv;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;

  BwdPrep pr;
  pr.o = o;
  pr.dout = dout;
  pr.lse = lse;
  pr.pref = pref;
  const long long threads = static_cast<long long>(vec_floats) * 8;
  const long long blocks = (threads + 255) / 256;
  const long long cap = static_cast<long long>(info.sm_count > 0 ? info.sm_count : 1) * 8;
  pr.grid = static_cast<int>(blocks < cap ? blocks : cap);
  pr.grid_kv = varlen ? static_cast<int>(kt_max * Hkv) : 0;
  pr.grid_q = varlen ? static_cast<int>(qt_max * Hq) : 0;

  BwdLauncher launch = (d == 64) ? bwd_launcher_d64(bf16, causal != 0, varlen)
                                 : bwd_launcher_d128(bf16, causal != 0, varlen);
  if (launch(p, pr, stream) != cudaSuccess) return ATTN_ELAUNCH;
  for (int i = 0; i < (varlen ? 4 : 3); ++i) count_launch();
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale, int fp16,
             cudaStream_t stream) {
  if (fp16 != 0 && fp16 != 1) return ATTN_EINVAL;
  return attn::bwd(fp16 == 0, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Lq, Lk, d, causal, scale, nullptr,
                   nullptr, stream);
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int total_q, int total_k, int d, int causal,
                    float scale, const int* cu_seqlens_q, const int* cu_seqlens_k, int fp16, cudaStream_t stream) {
  if (fp16 != 0 && fp16 != 1) return ATTN_EINVAL;
  if (!cu_seqlens_q || !cu_seqlens_k) return ATTN_EINVAL;
  return attn::bwd(fp16 == 0, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, total_q, total_k, d, causal, scale,
                   cu_seqlens_q, cu_seqlens_k, stream);
}

}  // extern "C"
