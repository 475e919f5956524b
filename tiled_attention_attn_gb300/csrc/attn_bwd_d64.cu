// Backward kernels for head_dim 64.
#include "attn_bwd_kernels.inc"

namespace attn {
BwdLauncher bwd_launcher_d64(bool bf16, bool causal, bool varlen) { return pick_bwd<64>(bf16, causal, varlen); }
}  // namespace attn
