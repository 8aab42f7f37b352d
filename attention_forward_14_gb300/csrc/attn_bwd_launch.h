// Launch wrappers of the attention backward kernels (instances in
// attn_bwd_inst.cu), called by the C ABI in attn_fwd_api.cu.
#pragma once

#include <atomic>
#include <type_traits>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"

namespace attn {
namespace bwd {

struct BwdLaunchArgs {
    CUtensorMap q, k, v, dout;
    CUtensorMap dq_acc;  // fp32 [bh][sq][D] reduce-add target (box and swizzle per Cfg<D>)
    BwdParams p;
    int grid;       // main kernel CTAs (persistent)
    int sm_count;
    cudaStream_t stream;
    // The calling library's flag, for the current device, of whether each
    // instance's shared-memory opt-in is set (indexed by bwd_instance_id; see
    // LaunchArgs::attr_ready for why it is not a static of the launcher).
    std::atomic<int> *attr_ready;
};

constexpr int kBwdInstances = 16;  // {fp16, bf16} x {causal, not} x head dim {64, 128} x {dense, packed}

template <typename T, bool CAUSAL, int D, bool VARLEN>
constexpr int bwd_instance_id()
{
    return (((std::is_same<T, __nv_bfloat16>::value ? 1 : 0) * 2 + (CAUSAL ? 1 : 0)) * 2 + (D == 64 ? 0 : 1)) * 2 +
           (VARLEN ? 1 : 0);
}

// prep -> main -> dQ convert, all on a.stream.  T: __half or __nv_bfloat16;
// D: head dim 64 or 128; VARLEN: packed sequences (a.p.cu_q set).
template <typename T, bool CAUSAL, int D, bool VARLEN>
cudaError_t launch_bwd(const BwdLaunchArgs &a);

#define ATTN_BWD_EXTERN(T, C, D, V) extern template cudaError_t launch_bwd<T, C, D, V>(const BwdLaunchArgs &);
#define ATTN_BWD_EXTERN_V(V)                      \
    ATTN_BWD_EXTERN(__half, false, 64, V)         \
    ATTN_BWD_EXTERN(__half, true, 64, V)          \
    ATTN_BWD_EXTERN(__nv_bfloat16, false, 64, V)  \
    ATTN_BWD_EXTERN(__nv_bfloat16, true, 64, V)   \
    ATTN_BWD_EXTERN(__half, false, 128, V)        \
    ATTN_BWD_EXTERN(__half, true, 128, V)         \
    ATTN_BWD_EXTERN(__nv_bfloat16, false, 128, V) \
    ATTN_BWD_EXTERN(__nv_bfloat16, true, 128, V)
ATTN_BWD_EXTERN_V(false)
ATTN_BWD_EXTERN_V(true)
#undef ATTN_BWD_EXTERN_V
#undef ATTN_BWD_EXTERN

}  // namespace bwd
}  // namespace attn
