// head_dim 128 instances of the fused forward with e4m3 inputs.
#include "launch.h"
namespace attn {
ATTN_DEFINE_INSTANCE(128, __nv_fp8_e4m3, false)
ATTN_DEFINE_INSTANCE(128, __nv_fp8_e4m3, true)
}  // namespace attn
