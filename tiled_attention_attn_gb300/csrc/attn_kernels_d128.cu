// Forward and combine kernels for head_dim 128.
#include "attn_kernels.inc"

namespace attn {
FwdLauncher fwd_launcher_d128(bool bf16, bool causal, bool varlen) { return pick_fwd<128>(bf16, causal, varlen); }
CombineLauncher combine_launcher_d128(bool bf16) {
  return bf16 ? launch_combine<128, true> : launch_combine<128, false>;
}
DecodeCombineLauncher decode_combine_launcher_d128(bool bf16) {
  return bf16 ? launch_combine_decode<128, true> : launch_combine_decode<128, false>;
}
}  // namespace attn
