// head_dim 64 instances of the fused forward.
#include "launch.h"
namespace attn {
ATTN_DEFINE_INSTANCE(64, __half, false)
ATTN_DEFINE_INSTANCE(64, __half, true)
ATTN_DEFINE_INSTANCE(64, __nv_bfloat16, false)
ATTN_DEFINE_INSTANCE(64, __nv_bfloat16, true)
}  // namespace attn
