// Instances of the attention backward: {fp16, bf16} x {causal, not} x head
// dim {64, 128}, and the launch sequence prep -> main -> dQ convert.
#include <atomic>

#include "attn_bwd_launch.h"

namespace attn {
namespace bwd {

template <typename T, bool CAUSAL, int D>
cudaError_t launch_bwd(const BwdLaunchArgs &a)
{
    // The shared-memory opt-in is a per-device property of the function:
    // set it once per device.
    static std::atomic<unsigned long long> attr_set{0ull};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(attn_bwd_kernel<T, CAUSAL, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<D>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    const int64_t prep_rows = static_cast<int64_t>(a.p.bh) * a.p.sq_pad;
    int prep_blocks = static_cast<int>((prep_rows * (D / 8) + 255) / 256);
    if (prep_blocks > 8 * a.sm_count) prep_blocks = 8 * a.sm_count;
    attn_bwd_prep_kernel<T, D><<<prep_blocks, 256, 0, a.stream>>>(a.p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_bwd_kernel<T, CAUSAL, D><<<a.grid, Cfg<D>::THREADS, Cfg<D>::SMEM_BYTES, a.stream>>>(a.q, a.k, a.v, a.dout,
                                                                                              a.dq_acc, a.p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n8 = static_cast<int64_t>(a.p.bh) * a.p.sq * D / 8;
    int cv_blocks = static_cast<int>((n8 + 255) / 256);
    if (cv_blocks > 8 * a.sm_count) cv_blocks = 8 * a.sm_count;
    if (cv_blocks < 1) cv_blocks = 1;
    attn_bwd_dq_convert_kernel<T><<<cv_blocks, 256, 0, a.stream>>>(a.p.dq_acc, reinterpret_cast<T *>(a.p.dq), n8);
    return cudaGetLastError();
}

template cudaError_t launch_bwd<__half, false, 64>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__half, true, 64>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__nv_bfloat16, false, 64>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__nv_bfloat16, true, 64>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__half, false, 128>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__half, true, 128>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__nv_bfloat16, false, 128>(const BwdLaunchArgs &);
template cudaError_t launch_bwd<__nv_bfloat16, true, 128>(const BwdLaunchArgs &);

}  // namespace bwd
}  // namespace attn
