// Launch wrappers of the attention backward kernels (instances in
// attn_bwd_inst.cu), called by the C ABI in attn_fwd_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"

namespace attn {
namespace bwd {

struct BwdLaunchArgs {
    CUtensorMap q, k, v, dout;
    CUtensorMap dq_acc;  // fp32 [bh][sq][128], box 128 x 64 rows, no swizzle (reduce-add target)
    BwdParams p;
    int grid;       // main kernel CTAs (persistent)
    int sm_count;
    cudaStream_t stream;
};

// prep -> main -> dQ convert, all on a.stream.  T: __half or __nv_bfloat16.
template <typename T, bool CAUSAL>
cudaError_t launch_bwd(const BwdLaunchArgs &a);

extern template cudaError_t launch_bwd<__half, false>(const BwdLaunchArgs &);
extern template cudaError_t launch_bwd<__half, true>(const BwdLaunchArgs &);
extern template cudaError_t launch_bwd<__nv_bfloat16, false>(const BwdLaunchArgs &);
extern template cudaError_t launch_bwd<__nv_bfloat16, true>(const BwdLaunchArgs &);

}  // namespace bwd
}  // namespace attn
