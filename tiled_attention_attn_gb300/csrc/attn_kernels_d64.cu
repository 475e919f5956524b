// Forward and combine kernels for head_dim 64.
#include "attn_kernels.inc"

namespace attn {
FwdLauncher fwd_launcher_d64(bool bf16, bool causal, bool varlen) { return pick_fwd<64>(bf16, causal, varlen); }
CombineLauncher combine_launcher_d64(bool bf16) {
  return bf16 ? launch_combine<64, true> : launch_combine<64, false>;
}
DecodeCombineLauncher decode_combine_launcher_d64(bool bf16) {
  return bf16 ? launch_combine_decode<64, true> : launch_combine_decode<64, false>;
}
}  // namespace attn
