// Instances of the fused forward with e4m3 inputs (head_dim 128 and 64).
#include "launch.h"
namespace attn {
ATTN_DEFINE_INSTANCE(128, __nv_fp8_e4m3, false)
ATTN_DEFINE_INSTANCE(128, __nv_fp8_e4m3, true)
ATTN_DEFINE_INSTANCE(64, __nv_fp8_e4m3, false)
ATTN_DEFINE_INSTANCE(64, __nv_fp8_e4m3, true)
}  // namespace attn
