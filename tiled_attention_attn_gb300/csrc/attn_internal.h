// Internal helpers shared by the library's entry-point translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct DeviceInfo {
  int sm_count = 0;
  bool supported = false;   // sm_103
  int* err_word = nullptr;  // device address of the error word
};

// Queries (once per device, cached) the SM count, whether the device is an
// sm_103 part, and the device address of the error word.  Allocates nothing.
int device_info(int dev, DeviceInfo& out);

// Encodes the 4-D TMA map over (d, H, L, B) of a contiguous (B, L, H, d)
// 16-bit tensor, box 64 x 1 x 128 x 1, without caching.  Allocates nothing.
int encode_map(const void* ptr, bool bf16, int d, int H, int L, int B, CUtensorMap& out);

// Writes n ints from host memory to device memory `dst` in stream order: a
// small kernel carries the values in its parameters (no pinned buffer, no
// synchronisation, nothing allocated).  Counts its launches.
int upload_ints(int* dst, const int* src, size_t n, cudaStream_t stream);

// Current barrier-wait time limit and the launch counter of attn_launch_count().
unsigned long long wait_timeout_ns();
// The phase-trace buffer set by attn_trace_enable (traced build), or null.
unsigned long long* trace_buffer(int* events_per_stream);
void count_launch();

// attn_decode on the packed forward's tensor-core tiles (decode mode of the
// varlen kernel, caches cut into pieces merged by the decode combine), and
// whether attn_decode takes that route (attn_set_decode_path, default on).
// The caller has checked the arguments; needs total_k > 0, B <= kVarlenMaxB.
int decode_on_tensor_cores(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                           int Hkv, int total_k, int d, float scale, const int* cu_k, cudaStream_t stream);
bool decode_tensor_cores_enabled();

// Writes cs[pos * rot / 2 + i] = (cos, sin) of pos * base^(-2 i / rot) for
// pos < n_pos with the arithmetic of the rotary pass (one launch on stream).
int rope_table(float2* cs, int n_pos, int rot, float base, cudaStream_t stream);

}  // namespace attn
