// Internal launch interface between the C-ABI layer and the kernel
// instantiations (one translation unit per group of instances so that the
// build compiles them in parallel).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

struct LaunchArgs {
    CUtensorMap q, k, v, o;
    FwdParams p;
    int grid;
    cudaStream_t stream;
    // The calling library's flags, for the current device, of whether each
    // instance's dynamic shared-memory opt-in is set (indexed by
    // fwd_instance_id).  They belong to the library that launches: a
    // function-local static here would be one object for the whole process
    // (a unique symbol), shared with any other library built from these
    // sources (the checked build), whose kernels are other functions.
    std::atomic<int> *attr_ready;
};

constexpr int kFwdInstances = 12;  // head dim {64, 128} x {fp16, bf16, e4m3} x {causal, not}

template <int D, typename T, bool CAUSAL>
constexpr int fwd_instance_id()
{
    return ((D == 64 ? 0 : 1) * 3 + (Elem<T>::FP8 ? 2 : (Elem<T>::BF16 ? 1 : 0))) * 2 + (CAUSAL ? 1 : 0);
}

// The dynamic shared-memory opt-in is a per-device attribute of each
// instance: set it the first time an instance runs on a device.
template <int D, typename T, bool CAUSAL>
cudaError_t launch_fwd(const LaunchArgs &a)
{
    constexpr int smem = Cfg<D, Elem<T>::BYTES>::SMEM_BYTES;
    auto kern = attn_fwd_kernel<D, T, CAUSAL>;
    std::atomic<int> &ready = a.attr_ready[fwd_instance_id<D, T, CAUSAL>()];
    if (ready.load(std::memory_order_acquire) == 0) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        ready.store(1, std::memory_order_release);
    }
    kern<<<a.grid, Cfg<D, Elem<T>::BYTES>::THREADS, smem, a.stream>>>(a.q, a.k, a.v, a.o, a.p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fill_empty(void *o, float *lse, int64_t rows, int d, cudaStream_t stream)
{
    int64_t n = rows * d;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    attn_fill_empty_kernel<T><<<blocks, 256, 0, stream>>>(static_cast<T *>(o), lse, rows, d);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_kvcache_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                  const int32_t *seqlens, int64_t bh, int64_t h, int64_t s_new, int64_t s_cache, int d,
                                  int sm_count, cudaStream_t stream)
{
    const int64_t n = bh * s_new * (d * static_cast<int64_t>(sizeof(T)) / 16);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    attn_kvcache_append_kernel<T><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const T *>(k_new), static_cast<const T *>(v_new), static_cast<T *>(k_cache),
        static_cast<T *>(v_cache), seqlens, bh, h, s_new, s_cache, d);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_kvcache_append_paged(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                                        const int32_t *seqlens, const int32_t *block_table, int64_t bh, int64_t h,
                                        int64_t s_new, int64_t pages_per_seq, int64_t page_size, int64_t num_pages,
                                        int d, int sm_count, cudaStream_t stream)
{
    const int64_t n = bh * s_new * (d * static_cast<int64_t>(sizeof(T)) / 16);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    attn_kvcache_append_paged_kernel<T><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const T *>(k_new), static_cast<const T *>(v_new), static_cast<T *>(k_pool),
        static_cast<T *>(v_pool), seqlens, block_table, bh, h, s_new, pages_per_seq, page_size, num_pages, d);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_splitkv_combine(const float *o_part, const float *lse_part, void *o, float *lse, int64_t rows,
                                   int num_splits, int sm_count, cudaStream_t stream)
{
    int64_t blocks = (rows + 7) / 8;  // one warp per row, 8 warps per block
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    attn_splitkv_combine_kernel<T, D><<<static_cast<int>(blocks), 256, 0, stream>>>(
        o_part, lse_part, static_cast<T *>(o), lse, rows, num_splits);
    return cudaGetLastError();
}

#define ATTN_DECLARE_INSTANCE(D, T, C) extern template cudaError_t launch_fwd<D, T, C>(const LaunchArgs &);
#define ATTN_DEFINE_INSTANCE(D, T, C) template cudaError_t launch_fwd<D, T, C>(const LaunchArgs &);

ATTN_DECLARE_INSTANCE(64, __half, false)
ATTN_DECLARE_INSTANCE(64, __half, true)
ATTN_DECLARE_INSTANCE(64, __nv_bfloat16, false)
ATTN_DECLARE_INSTANCE(64, __nv_bfloat16, true)
ATTN_DECLARE_INSTANCE(128, __half, false)
ATTN_DECLARE_INSTANCE(128, __half, true)
ATTN_DECLARE_INSTANCE(128, __nv_bfloat16, false)
ATTN_DECLARE_INSTANCE(128, __nv_bfloat16, true)
ATTN_DECLARE_INSTANCE(128, __nv_fp8_e4m3, false)
ATTN_DECLARE_INSTANCE(128, __nv_fp8_e4m3, true)
ATTN_DECLARE_INSTANCE(64, __nv_fp8_e4m3, false)
ATTN_DECLARE_INSTANCE(64, __nv_fp8_e4m3, true)

}  // namespace attn
