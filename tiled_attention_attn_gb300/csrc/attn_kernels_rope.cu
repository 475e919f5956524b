// The dense forward kernels with the rotary embedding of Q applied in the
// kernel, for both head dimensions (a translation unit of their own so that
// the build compiles them beside the others).
#include "attn_kernels.inc"

namespace attn {
FwdLauncher fwd_rope_launcher_d64(bool bf16, bool causal) {
  if (bf16) return causal ? launch_fwd<64, true, true, false, true> : launch_fwd<64, true, false, false, true>;
  return causal ? launch_fwd<64, false, true, false, true> : launch_fwd<64, false, false, false, true>;
}
FwdLauncher fwd_rope_launcher_d128(bool bf16, bool causal) {
  if (bf16) return causal ? launch_fwd<128, true, true, false, true> : launch_fwd<128, true, false, false, true>;
  return causal ? launch_fwd<128, false, true, false, true> : launch_fwd<128, false, false, false, true>;
}
}  // namespace attn
