// Instances of the attention backward: {fp16, bf16} x {causal, not} x head
// dim {64, 128} for the dense layout (ATTN_BWD_INST_VARLEN unset) or the
// packed one (attn_bwd_inst_varlen.cu sets it), and the launch sequence
// prep -> main -> dQ convert.
#include <atomic>

#include "attn_bwd_launch.h"

namespace attn {
namespace bwd {

template <typename T, bool CAUSAL, int D, bool VARLEN>
cudaError_t launch_bwd(const BwdLaunchArgs &a)
{
    // The shared-memory opt-in is a per-device property of the function:
    // set it once per device (the flag belongs to the calling library).
    cudaError_t e;
    std::atomic<int> &ready = a.attr_ready[bwd_instance_id<T, CAUSAL, D, VARLEN>()];
    if (ready.load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(attn_bwd_kernel<T, CAUSAL, D, VARLEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<D>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        ready.store(1, std::memory_order_release);
    }
    const int64_t prep_rows = static_cast<int64_t>(a.p.bh) * a.p.sq_pad;
    int prep_blocks = static_cast<int>((prep_rows * (D / 8) + 255) / 256);
    if (prep_blocks > 8 * a.sm_count) prep_blocks = 8 * a.sm_count;
    attn_bwd_prep_kernel<T, D, VARLEN><<<prep_blocks, 256, 0, a.stream>>>(a.p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_bwd_kernel<T, CAUSAL, D, VARLEN><<<a.grid, Cfg<D>::THREADS, Cfg<D>::SMEM_BYTES, a.stream>>>(a.q, a.k, a.v, a.dout,
                                                                                              a.dq_acc, a.p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dQ rows: [bh, sq] dense, [total_q, heads] packed
    const int64_t dq_rows = a.p.cu_q ? static_cast<int64_t>(a.p.total_q) * a.p.heads : static_cast<int64_t>(a.p.bh) * a.p.sq;
    const int64_t n8 = dq_rows * D / 8;
    int cv_blocks = static_cast<int>((n8 + 255) / 256);
    if (cv_blocks > 8 * a.sm_count) cv_blocks = 8 * a.sm_count;
    if (cv_blocks < 1) cv_blocks = 1;
    attn_bwd_dq_convert_kernel<T><<<cv_blocks, 256, 0, a.stream>>>(a.p.dq_acc, reinterpret_cast<T *>(a.p.dq), n8);
    return cudaGetLastError();
}


#ifndef ATTN_BWD_INST_VARLEN
#define ATTN_BWD_INST_VARLEN false
#endif
#define ATTN_BWD_INST(T, C, D) template cudaError_t launch_bwd<T, C, D, ATTN_BWD_INST_VARLEN>(const BwdLaunchArgs &);
ATTN_BWD_INST(__half, false, 64)
ATTN_BWD_INST(__half, true, 64)
ATTN_BWD_INST(__nv_bfloat16, false, 64)
ATTN_BWD_INST(__nv_bfloat16, true, 64)
ATTN_BWD_INST(__half, false, 128)
ATTN_BWD_INST(__half, true, 128)
ATTN_BWD_INST(__nv_bfloat16, false, 128)
ATTN_BWD_INST(__nv_bfloat16, true, 128)
#undef ATTN_BWD_INST

}  // namespace bwd
}  // namespace attn
