// The packed varlen forward kernels that may place their units in order of
// the sequences' key counts (the sorting variant, for queries with their own
// key offsets: cross-attention, a key/value cache), both head dimensions, in
// a translation unit of their own so that the build compiles them beside the
// others.
#include "attn_kernels.inc"

namespace attn {
FwdLauncher fwd_sorted_launcher_d64(bool bf16, bool causal) {
  if (bf16) return causal ? launch_fwd<64, true, true, true, false, true> : launch_fwd<64, true, false, true, false, true>;
  return causal ? launch_fwd<64, false, true, true, false, true> : launch_fwd<64, false, false, true, false, true>;
}
FwdLauncher fwd_sorted_launcher_d128(bool bf16, bool causal) {
  if (bf16)
    return causal ? launch_fwd<128, true, true, true, false, true> : launch_fwd<128, true, false, true, false, true>;
  return causal ? launch_fwd<128, false, true, true, false, true> : launch_fwd<128, false, false, true, false, true>;
}
}  // namespace attn
