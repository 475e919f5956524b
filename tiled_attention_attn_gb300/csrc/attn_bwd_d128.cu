// Backward kernels for head_dim 128.
#include "attn_bwd_kernels.inc"

namespace attn {
BwdLauncher bwd_launcher_d128(bool bf16, bool causal, bool varlen) { return pick_bwd<128>(bf16, causal, varlen); }
}  // namespace attn
