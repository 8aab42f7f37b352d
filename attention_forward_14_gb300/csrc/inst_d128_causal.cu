// head_dim 128 instances of the fused forward, causal mask.
#include "launch.h"
namespace attn {
ATTN_DEFINE_INSTANCE(128, __half, true)
ATTN_DEFINE_INSTANCE(128, __nv_bfloat16, true)
}  // namespace attn
