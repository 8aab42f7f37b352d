// head_dim 128 instances of the fused forward, no mask.
#include "launch.h"
namespace attn {
ATTN_DEFINE_INSTANCE(128, __half, false)
ATTN_DEFINE_INSTANCE(128, __nv_bfloat16, false)
}  // namespace attn
