// C ABI of the fused attention forward and backward (declared in
// include/attn_fwd.h): argument validation, TMA tensor maps, persistent grid
// sizing, dispatch to the <head_dim, dtype, causal> instances, device
// watchdog status.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn_bwd_launch.h"
#include "attn_fwd.h"
#include "launch.h"
#include "sched_ticket.h"

namespace {

using namespace attn;

thread_local std::string g_err;

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#ifdef ATTN_TRACE_ENABLE
unsigned long long *g_trace_buf = nullptr;  // timeline builds only: where launches record
#endif

// Watchdog status word, one per device that loads this library.
__device__ uint32_t g_watchdog[4];

// Counter slots of the forward's dynamic schedule.  Each launch that uses
// one takes the next slot in turn, tagged with its own generation number
// (sched_ticket.h); the kernel leaves the slot at zero when it finishes, so a
// slot is ready again once its previous launch has ended.  A launch that
// finds its slot still held by another generation (more than kSchedSlots
// such launches in flight) reports STATUS_SCHED_COLLISION instead of sharing
// the counters.
__device__ int32_t g_fwd_sched[kSchedWords * kSchedSlots];

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;
    int32_t *sched = nullptr;
    std::atomic<uint64_t> sched_next{0};
    std::atomic<int> sched_pinned{-1};  // testing hook: every launch on this slot
    std::atomic<int> fwd_attr[kFwdInstances] = {};  // shared-memory opt-in set, per kernel instance
    std::atomic<int> bwd_attr[bwd::kBwdInstances] = {};
};
DeviceInfo g_dev[kMaxDevices];

// Queried once per device, with that device current.
int device_info(DeviceInfo **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceInfo &di = g_dev[dev];
    std::call_once(di.once, [&] {
        cudaError_t r = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (r == cudaSuccess && di.cc_major == 10 && di.cc_minor == 3)
            r = cudaGetSymbolAddress(reinterpret_cast<void **>(&di.status), g_watchdog);
        if (r == cudaSuccess && di.cc_major == 10 && di.cc_minor == 3)
            r = cudaGetSymbolAddress(reinterpret_cast<void **>(&di.sched), g_fwd_sched);
        di.err = r;
    });
    if (di.err != cudaSuccess) return cuda_fail(di.err, "device query");
    if (di.cc_major != 10 || di.cc_minor != 3)
        return fail(ATTN_ERR_ARCH, "device %d is compute capability %d.%d; this library is built for sm_103a only", dev,
                    di.cc_major, di.cc_minor);
    *out = &di;
    return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encode(PFN_cuTensorMapEncodeTiled_v12000 *fn)
{
    std::call_once(g_encode_once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!g_encode) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    *fn = g_encode;
    return ATTN_OK;
}

// cuTensorMapEncodeTiled (rank 3, no interleave, unit element strides, 256-B
// L2 promotion, no OOB fill) through a small per-thread cache keyed by every
// other argument.  A map is a pure function of those arguments (the address
// and the shape), so a cached map is exactly the one the encoder would
// produce again; calls that reuse their buffers skip the encode.
struct MapKey {
    const void *ptr;
    int dt, swizzle;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kMapCache = 16;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

int encode_map(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, const cuuint64_t (&dims)[3],
               const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3], CUtensorMapSwizzle swizzle, const char *what)
{
    MapKey key;
    memset(&key, 0, sizeof(key));  // padding too: keys are compared bytewise
    key.ptr = ptr;
    key.dt = static_cast<int>(dt);
    key.swizzle = static_cast<int>(swizzle);
    memcpy(key.dims, dims, sizeof(key.dims));
    memcpy(key.strides, strides, sizeof(key.strides));
    memcpy(key.box, box, sizeof(key.box));
    for (const MapEntry &e : t_maps)
        if (e.used && memcmp(&e.key, &key, sizeof(key)) == 0) {
            *map = e.map;
            return ATTN_OK;
        }
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    const int rc = get_encode(&enc);
    if (rc != ATTN_OK) return rc;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (%s) failed (CUresult %d)", what, static_cast<int>(r));
    MapEntry &slot = t_maps[t_map_next];
    t_map_next = (t_map_next + 1) % kMapCache;
    slot.key = key;
    slot.map = *map;
    slot.used = true;
    return ATTN_OK;
}

// 3-D view [bh, s, d] of a contiguous [b, h, s, d] tensor; box = 128 rows x
// one 128-byte swizzle panel (64 16-bit or 128 8-bit elements), so rows past
// s of each head are zero-filled by the copy engine rather than read from the
// next head.  Rows shorter than 128 bytes (8-bit, d = 64) are one 64-byte
// panel with the 64-byte swizzle.
int make_map(CUtensorMap *map, const void *ptr, int dtype, int64_t bh, int64_t s, int64_t d, int elem_bytes = 2,
             int box_rows = 128)
{
    const int64_t row_bytes = d * elem_bytes < 128 ? d * elem_bytes : 128;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(s), static_cast<cuuint64_t>(bh)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * elem_bytes), static_cast<cuuint64_t>(s * d * elem_bytes)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(row_bytes / elem_bytes), static_cast<cuuint32_t>(box_rows), 1};
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return encode_map(map, dt, ptr, dims, strides, box,
                      row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, "dense");
}

// Packed [tokens, h, d] tensor seen as 3-D [tokens][h][d]: box = 64
// elements x 1 head x 128 tokens, the same 128-row x 128-byte shared-memory
// image as the dense map.  Rows past the last token are zero-filled.
int make_map_packed(CUtensorMap *map, const void *ptr, int dtype, int64_t tokens, int64_t h, int64_t d,
                    int box_rows = 128)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(h * d * 2)};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    return encode_map(map, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ptr,
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "packed");
}

// The backward's fp32 dQ accumulator [bh, sq, d] as 3-D [bh][sq][d] for the
// tile reduce-adds: d = 128, RED_ROWS rows x 128 columns, row-major in
// shared memory (no swizzle); d = 64, 128 rows x 32 columns with the
// 128-byte swizzle.  Rows past sq are clipped by the copy engine.
int make_map_f32_rows(CUtensorMap *map, void *ptr, int64_t bh, int64_t s, int64_t d)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(s), static_cast<cuuint64_t>(bh)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 4), static_cast<cuuint64_t>(s * d * 4)};
    const bool wide = d == 128;
    const cuuint32_t box[3] = {wide ? 128u : 32u, wide ? static_cast<cuuint32_t>(bwd::Cfg<128>::RED_ROWS) : 128u, 1};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, dims, strides, box,
                      wide ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, "fp32 rows");
}

// The same for a packed [tokens, h, d] accumulator (varlen backward), as
// 3-D [tokens][h][d] with boxes of one head.
int make_map_f32_packed(CUtensorMap *map, void *ptr, int64_t tokens, int64_t h, int64_t d)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 4), static_cast<cuuint64_t>(h * d * 4)};
    const bool wide = d == 128;
    const cuuint32_t box[3] = {wide ? 128u : 32u, 1, wide ? static_cast<cuuint32_t>(bwd::Cfg<128>::RED_ROWS) : 128u};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, dims, strides, box,
                      wide ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, "fp32 packed");
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxSeq = int64_t(1) << 30;

// The size, head-dim, dtype and scale checks of every forward entry point
// (no pointer is looked at).
int validate_sizes(int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d, float scale, int dtype)
{
    if (b < 0 || h < 0 || sq < 0 || sk < 0)
        return fail(ATTN_ERR_SHAPE, "negative size: b=%lld h=%lld sq=%lld sk=%lld", (long long)b, (long long)h,
                    (long long)sq, (long long)sk);
    if (sq > kMaxSeq || sk > kMaxSeq)
        return fail(ATTN_ERR_SHAPE, "sequence length above 2^30: sq=%lld sk=%lld", (long long)sq, (long long)sk);
    if (b > 0 && h >= (int64_t(1) << 31) / b)
        return fail(ATTN_ERR_SHAPE, "b*h not below 2^31: b=%lld h=%lld", (long long)b, (long long)h);
    if (d != 64 && d != 128) return fail(ATTN_ERR_HEADDIM, "head dim %lld not supported (64 or 128)", (long long)d);
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_DTYPE, "dtype %d is not fp16 (0) or bf16 (1)", dtype);
    if (!std::isfinite(scale)) return fail(ATTN_ERR_SCALE, "scale is not finite");
    return ATTN_OK;
}

int validate(const void *q, const void *k, const void *v, const void *o, const float *lse, int64_t b, int64_t h,
             int64_t sq, int64_t sk, int64_t d, float scale, int dtype, bool *nothing)
{
    const int rc = validate_sizes(b, h, sq, sk, d, scale, dtype);
    if (rc != ATTN_OK) return rc;
    *nothing = (b * h * sq == 0);
    if (*nothing) return ATTN_OK;
    if (!o) return fail(ATTN_ERR_NULL, "o is NULL");
    if (sk > 0 && (!q || !k || !v)) return fail(ATTN_ERR_NULL, "q, k or v is NULL");
    if (!aligned(o, 16) || (sk > 0 && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))))
        return fail(ATTN_ERR_ALIGN, "q, k, v and o must be 16-byte aligned");
    if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_ALIGN, "lse must be 4-byte aligned");
    return ATTN_OK;
}

template <int D, typename T>
cudaError_t dispatch_causal(const LaunchArgs &a, bool causal)
{
    return causal ? launch_fwd<D, T, true>(a) : launch_fwd<D, T, false>(a);
}

struct SplitArgs {
    int num_splits = 1;
    float *o_part = nullptr;
    float *lse_part = nullptr;
};

// KV cache: per batch element, the number of valid keys is
// clamp(seqlens[b], 0, sk) + add, at most sk (sk is the cache capacity).
// Units of unequal work (per-element lengths) are handed out dynamically.
struct CacheArgs {
    const int32_t *seqlens = nullptr;
    int32_t add = 0;
    // paged: K and V are pools [num_pages][page_size][h][d]; the capacity
    // (the sk of run) is pages_per_seq * page_size
    const int32_t *block_table = nullptr;
    int64_t pages_per_seq = 0, page_size = 0, num_pages = 0;
};

// Head planes per group of the causal unit order: as many as keep the K and
// V of the group's heads (sk keys of d elements) within 48 MB of L2.
int32_t l2_group(int64_t bh, int64_t sk, int64_t d, int64_t elem_bytes)
{
    const int64_t per_head = 2 * sk * d * elem_bytes;
    int64_t g = per_head > 0 ? (int64_t(48) << 20) / per_head : bh;
    if (g < 1) g = 1;
    if (g > bh) g = bh;
    return static_cast<int32_t>(g);
}

// The next counter slot of the dynamic schedule on this device, and the
// generation that tags this launch in it.
int32_t *sched_slot(DeviceInfo *di, uint32_t *gen)
{
    const SchedTicket t = sched_ticket(di->sched_next.fetch_add(1, std::memory_order_relaxed),
                                       di->sched_pinned.load(std::memory_order_relaxed));
    *gen = t.gen;
    return di->sched + kSchedWords * t.slot;
}

int64_t kv_tiles(int64_t sk) { return (sk + 127) / 128; }

int64_t splitkv_bytes(int64_t bh, int64_t sq, int64_t d, int64_t splits)
{
    return splits * bh * sq * (d + 2) * 4;
}

int run(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h, int64_t sq, int64_t sk,
        int64_t d, int causal, float scale, int dtype, cudaStream_t stream, int withheld_load, uint64_t timeout_ns,
        const SplitArgs &split = SplitArgs(), const CacheArgs &cache = CacheArgs(), int extra_units = 0)
{
    bool nothing = false;
    int rc = validate(q, k, v, o, lse, b, h, sq, sk, d, scale, dtype, &nothing);
    if (rc != ATTN_OK || nothing) return rc;
    DeviceInfo *di = nullptr;
    rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    const int64_t bh = b * h;
    cudaError_t e;
    if (sk == 0) {
        e = (dtype == ATTN_BF16) ? launch_fill_empty<__nv_bfloat16>(o, lse, bh * sq, static_cast<int>(d), stream)
                                 : launch_fill_empty<__half>(o, lse, bh * sq, static_cast<int>(d), stream);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "launch (empty keys)");
    }
    LaunchArgs a;
    if ((rc = make_map(&a.q, q, dtype, bh, sq, d)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.o, o, dtype, bh, sq, d, 2, 32)) != ATTN_OK) return rc;  // stores of 32 rows
    if (cache.block_table != nullptr) {
        const int64_t pool = cache.num_pages * cache.page_size;
        if ((rc = make_map_packed(&a.k, k, dtype, pool, h, d)) != ATTN_OK) return rc;
        if ((rc = make_map_packed(&a.v, v, dtype, pool, h, d)) != ATTN_OK) return rc;
    } else {
        if ((rc = make_map(&a.k, k, dtype, bh, sk, d)) != ATTN_OK) return rc;
        if ((rc = make_map(&a.v, v, dtype, bh, sk, d)) != ATTN_OK) return rc;
    }
    FwdParams &p = a.p;
    p.o = o;
    p.lse = lse;
    p.status = di->status;
    p.bh = static_cast<int32_t>(bh);
    p.sq = static_cast<int32_t>(sq);
    p.sk = static_cast<int32_t>(sk);
    p.num_mblk = static_cast<int32_t>((sq + 255) / 256);
    p.num_splits = split.num_splits;
    p.o_part = split.o_part;
    p.lse_part = split.lse_part;
    p.cu_q = p.cu_k = nullptr;
    p.heads = static_cast<int32_t>(h);
    p.total_q = static_cast<int32_t>(sq);
    p.total_k = static_cast<int32_t>(sk);
    p.seqlens_k = cache.seqlens;
    p.seqlens_add = cache.add;
    p.block_table = cache.block_table;
    p.pages_per_seq = static_cast<int32_t>(cache.pages_per_seq);
    p.page_size = static_cast<int32_t>(cache.page_size);
    p.num_pages = static_cast<int32_t>(cache.num_pages);
    p.sched = cache.seqlens != nullptr ? sched_slot(di, &p.sched_gen) : nullptr;
    const int64_t units = bh * p.num_mblk * split.num_splits;
    if (units > INT32_MAX) return fail(ATTN_ERR_SHAPE, "too many work units (%lld)", (long long)units);
    p.num_units = static_cast<int32_t>(units + extra_units);  // extra units: the bounds self-test only
    p.sl2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.o_scale = 1.f;
    p.timeout_ns = timeout_ns;
    p.withheld_load = withheld_load;
#ifdef ATTN_TRACE_ENABLE
    p.trace = g_trace_buf;
#endif
    a.grid = static_cast<int>(p.num_units < di->sm_count ? p.num_units : di->sm_count);
    a.stream = stream;
    a.attr_ready = di->fwd_attr;
    const bool c = causal != 0;
    if (d == 64)
        e = (dtype == ATTN_BF16) ? dispatch_causal<64, __nv_bfloat16>(a, c) : dispatch_causal<64, __half>(a, c);
    else
        e = (dtype == ATTN_BF16) ? dispatch_causal<128, __nv_bfloat16>(a, c) : dispatch_causal<128, __half>(a, c);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    if (split.num_splits > 1) {
        const int64_t rows = bh * sq;
        if (d == 64)
            e = (dtype == ATTN_BF16) ? launch_splitkv_combine<__nv_bfloat16, 64>(split.o_part, split.lse_part, o, lse,
                                                                               rows, split.num_splits, di->sm_count, stream)
                                     : launch_splitkv_combine<__half, 64>(split.o_part, split.lse_part, o, lse, rows,
                                                                         split.num_splits, di->sm_count, stream);
        else
            e = (dtype == ATTN_BF16) ? launch_splitkv_combine<__nv_bfloat16, 128>(split.o_part, split.lse_part, o, lse,
                                                                                rows, split.num_splits, di->sm_count, stream)
                                     : launch_splitkv_combine<__half, 128>(split.o_part, split.lse_part, o, lse, rows,
                                                                          split.num_splits, di->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return ATTN_OK;
}

constexpr uint64_t kDefaultTimeoutNs = 2000ull * 1000ull * 1000ull;  // 2 s per wait

// ---------------------------------------------------------------- host-buffer pipeline
//
// attn_fwd_host splits a large problem into chunks of whole heads and
// overlaps the host->device copy of chunk c+1 and the device->host copy of
// chunk c-1 with the forward of chunk c: copies in on one internal stream,
// the forwards on the caller's stream, copies out on a second internal
// stream, ordered by events.  The streams and events are created once per
// device; a mutex keeps one call's record/wait sequence together.

constexpr int kPipeChunks = 8;
constexpr int64_t kPipeMinBytes = int64_t(64) << 20;  // smaller problems: one chunk

struct HostPipe {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kPipeChunks] = {}, out[kPipeChunks] = {};
    std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
    HostPipe &hp = g_pipe[dev];
    std::call_once(hp.once, [&] {
        cudaError_t r = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
        if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
        if (r == cudaSuccess) r = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
        if (r == cudaSuccess) r = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
        for (int c = 0; c < kPipeChunks && r == cudaSuccess; ++c) {
            r = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming);
            if (r == cudaSuccess) r = cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming);
        }
        hp.err = r;
    });
    if (hp.err != cudaSuccess) return cuda_fail(hp.err, "host pipeline streams");
    *out = &hp;
    return ATTN_OK;
}

// ---------------------------------------------------------------- backward

int64_t bwd_sq_pad(int64_t sq) { return (sq + 127) / 128 * 128; }

// fp32 dQ accumulator [bh, sq, d], LSE2 and D [bh, sq_pad] each, and 256
// bytes for the scheduler's unit counter.
int64_t bwd_workspace_bytes(int64_t bh, int64_t sq, int64_t d)
{
    return bh * sq * d * 4 + 2 * bh * bwd_sq_pad(sq) * 4 + 256;
}

// Heads per scheduling group of the backward: the group's fp32 dQ
// accumulator, Q and dO (8 * sq * d bytes per head) fit in 64 MB, half of
// L2, while its units run.
int32_t bwd_group(int64_t bh, int64_t sq, int64_t d)
{
    const int64_t per_head = 8 * sq * d;
    int64_t g = per_head > 0 ? (int64_t(64) << 20) / per_head : bh;
    if (g < 1) g = 1;
    if (g > bh) g = bh;
    return static_cast<int32_t>(g);
}

template <bool VARLEN>
cudaError_t launch_bwd_any(const bwd::BwdLaunchArgs &a, int64_t d, int dtype, int causal)
{
    if (d == 128) {
        if (dtype == ATTN_BF16)
            return causal ? bwd::launch_bwd<__nv_bfloat16, true, 128, VARLEN>(a)
                          : bwd::launch_bwd<__nv_bfloat16, false, 128, VARLEN>(a);
        return causal ? bwd::launch_bwd<__half, true, 128, VARLEN>(a) : bwd::launch_bwd<__half, false, 128, VARLEN>(a);
    }
    if (dtype == ATTN_BF16)
        return causal ? bwd::launch_bwd<__nv_bfloat16, true, 64, VARLEN>(a)
                      : bwd::launch_bwd<__nv_bfloat16, false, 64, VARLEN>(a);
    return causal ? bwd::launch_bwd<__half, true, 64, VARLEN>(a) : bwd::launch_bwd<__half, false, 64, VARLEN>(a);
}

// Self-test knobs: extra_units > 0 hands out that many units past the end
// of the problem (bounds self-test); withheld_load >= 0 never issues that
// CTA-local Q load, and timeout_ns bounds every wait (watchdog self-test).
int run_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse, void *dq,
            void *dk, void *dv, int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d, int causal, float scale,
            int dtype, void *workspace, int64_t workspace_bytes, cudaStream_t stream, int extra_units = 0,
            int withheld_load = -1, uint64_t timeout_ns = kDefaultTimeoutNs)
{
    if (b < 0 || h < 0 || sq < 0 || sk < 0)
        return fail(ATTN_ERR_SHAPE, "negative size: b=%lld h=%lld sq=%lld sk=%lld", (long long)b, (long long)h,
                    (long long)sq, (long long)sk);
    if (sq > kMaxSeq || sk > kMaxSeq)
        return fail(ATTN_ERR_SHAPE, "sequence length above 2^30: sq=%lld sk=%lld", (long long)sq, (long long)sk);
    if (b > 0 && h >= (int64_t(1) << 31) / b)
        return fail(ATTN_ERR_SHAPE, "b*h not below 2^31: b=%lld h=%lld", (long long)b, (long long)h);
    if (d != 64 && d != 128) return fail(ATTN_ERR_HEADDIM, "backward: head dim %lld not supported (64 or 128)", (long long)d);
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_DTYPE, "dtype %d is not fp16 (0) or bf16 (1)", dtype);
    if (!std::isfinite(scale)) return fail(ATTN_ERR_SCALE, "scale is not finite");
    const int64_t bh = b * h;
    if (bh == 0) return ATTN_OK;
    if (bh * ((sq + 127) / 128) * ((sk + 127) / 128) > INT32_MAX)
        return fail(ATTN_ERR_SHAPE, "too many work units");
    const bool rows = sq > 0, keys = sk > 0;
    if ((rows && !dq) || (keys && (!dk || !dv))) return fail(ATTN_ERR_NULL, "dq, dk or dv is NULL");
    if ((rows && !aligned(dq, 16)) || (keys && (!aligned(dk, 16) || !aligned(dv, 16))))
        return fail(ATTN_ERR_ALIGN, "dq, dk and dv must be 16-byte aligned");
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    const size_t qbytes = static_cast<size_t>(bh * sq * d) * 2, kbytes = static_cast<size_t>(bh * sk * d) * 2;
    cudaError_t e;
    if (!rows || !keys) {  // no queries: dK = dV = 0; no keys: dQ = 0
        if (rows && (e = cudaMemsetAsync(dq, 0, qbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dq");
        if (keys && (e = cudaMemsetAsync(dk, 0, kbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dk");
        if (keys && (e = cudaMemsetAsync(dv, 0, kbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dv");
        return ATTN_OK;
    }
    if (!q || !k || !v || !o || !dout || !lse) return fail(ATTN_ERR_NULL, "q, k, v, o, dout or lse is NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16))
        return fail(ATTN_ERR_ALIGN, "q, k, v, o and dout must be 16-byte aligned");
    if (!aligned(lse, 4)) return fail(ATTN_ERR_ALIGN, "lse must be 4-byte aligned");
    const int64_t need = bwd_workspace_bytes(bh, sq, d);
    if (!workspace) return fail(ATTN_ERR_NULL, "workspace is NULL");
    if (!aligned(workspace, 16)) return fail(ATTN_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (workspace_bytes < need)
        return fail(ATTN_ERR_SHAPE, "workspace too small: %lld bytes, need %lld", (long long)workspace_bytes,
                    (long long)need);
    bwd::BwdLaunchArgs a;
    if ((rc = make_map(&a.q, q, dtype, bh, sq, d)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.dout, dout, dtype, bh, sq, d)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.k, k, dtype, bh, sk, d)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.v, v, dtype, bh, sk, d)) != ATTN_OK) return rc;
    if ((rc = make_map_f32_rows(&a.dq_acc, workspace, bh, sq, d)) != ATTN_OK) return rc;
    bwd::BwdParams &p = a.p;
    const int64_t sq_pad = bwd_sq_pad(sq);
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq_acc = static_cast<float *>(workspace);
    p.lse2 = p.dq_acc + bh * sq * d;
    p.dsum = p.lse2 + bh * sq_pad;
    p.counter = reinterpret_cast<int32_t *>(p.dsum + bh * sq_pad);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = di->status;
    p.bh = static_cast<int32_t>(bh);
    p.sq = static_cast<int32_t>(sq);
    p.sk = static_cast<int32_t>(sk);
    p.sq_pad = static_cast<int32_t>(sq_pad);
    p.num_kblk = static_cast<int32_t>((sk + 127) / 128);
    p.num_units = static_cast<int32_t>(bh * p.num_kblk) + extra_units;
    p.group = bwd_group(bh, sq, d);
#ifdef ATTN_TRACE_ENABLE
    p.trace = g_trace_buf;
#endif
    p.sl2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.scale = scale;
    p.timeout_ns = timeout_ns;
#if ATTN_CHECKED
    p.withheld_load = withheld_load;
#else
    (void)withheld_load;
#endif
    p.cu_q = p.cu_k = nullptr;
    p.heads = static_cast<int32_t>(h);
    p.total_q = static_cast<int32_t>(sq);
    p.total_k = static_cast<int32_t>(sk);
    a.grid = p.num_units < di->sm_count ? p.num_units : di->sm_count;
    a.sm_count = di->sm_count;
    a.stream = stream;
    a.attr_ready = di->bwd_attr;
    e = launch_bwd_any<false>(a, d, dtype, causal);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "backward launch");
}

// fp32 dQ accumulator [total_q, h, d], LSE2 and D [batch * h, sq_pad], the
// scheduler's counter.
int64_t bwd_varlen_workspace_bytes(int64_t batch, int64_t h, int64_t total_q, int64_t max_seqlen_q, int64_t d)
{
    return total_q * h * d * 4 + 2 * batch * h * bwd_sq_pad(max_seqlen_q) * 4 + 256;
}

int run_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                   void *dq, void *dk, void *dv, const int32_t *cu_q, const int32_t *cu_k, int64_t batch, int64_t h,
                   int64_t total_q, int64_t total_k, int64_t max_q, int64_t max_k, int64_t d, int causal, float scale,
                   int dtype, void *workspace, int64_t workspace_bytes, cudaStream_t stream)
{
    if (batch < 0 || h < 0 || total_q < 0 || total_k < 0 || max_q < 0 || max_k < 0)
        return fail(ATTN_ERR_SHAPE, "negative varlen size");
    if (total_q > INT32_MAX || total_k > INT32_MAX || max_q > total_q || max_k > total_k)
        return fail(ATTN_ERR_SHAPE, "varlen totals above 2^31-1 or max lengths above the totals");
    if (h > 0 && batch >= (int64_t(1) << 31) / h) return fail(ATTN_ERR_SHAPE, "batch*h not below 2^31");
    if (d != 64 && d != 128) return fail(ATTN_ERR_HEADDIM, "backward: head dim %lld not supported (64 or 128)", (long long)d);
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_DTYPE, "dtype %d is not fp16 (0) or bf16 (1)", dtype);
    if (!std::isfinite(scale)) return fail(ATTN_ERR_SCALE, "scale is not finite");
    if (batch == 0 || h == 0) return ATTN_OK;
    const bool rows = total_q > 0, keys = total_k > 0;
    if ((rows && !dq) || (keys && (!dk || !dv))) return fail(ATTN_ERR_NULL, "dq, dk or dv is NULL");
    if ((rows && !aligned(dq, 16)) || (keys && (!aligned(dk, 16) || !aligned(dv, 16))))
        return fail(ATTN_ERR_ALIGN, "dq, dk and dv must be 16-byte aligned");
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    const size_t qbytes = static_cast<size_t>(total_q * h * d) * 2, kbytes = static_cast<size_t>(total_k * h * d) * 2;
    cudaError_t e;
    if (!rows || !keys || max_q == 0 || max_k == 0) {  // no query or no key anywhere: the gradients that exist are 0
        if (rows && (e = cudaMemsetAsync(dq, 0, qbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dq");
        if (keys && (e = cudaMemsetAsync(dk, 0, kbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dk");
        if (keys && (e = cudaMemsetAsync(dv, 0, kbytes, stream)) != cudaSuccess) return cuda_fail(e, "zero dv");
        return ATTN_OK;
    }
    if (!q || !k || !v || !o || !dout || !lse) return fail(ATTN_ERR_NULL, "q, k, v, o, dout or lse is NULL");
    if (!cu_q || !cu_k) return fail(ATTN_ERR_NULL, "cu_seqlens_q / cu_seqlens_k is NULL");
    if (!aligned(cu_q, 4) || !aligned(cu_k, 4)) return fail(ATTN_ERR_ALIGN, "cu_seqlens must be 4-byte aligned");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16))
        return fail(ATTN_ERR_ALIGN, "q, k, v, o and dout must be 16-byte aligned");
    if (!aligned(lse, 4)) return fail(ATTN_ERR_ALIGN, "lse must be 4-byte aligned");
    const int64_t bh = batch * h;
    const int64_t num_kblk = (max_k + 127) / 128;
    if (bh * num_kblk > INT32_MAX) return fail(ATTN_ERR_SHAPE, "too many work units");
    const int64_t need = bwd_varlen_workspace_bytes(batch, h, total_q, max_q, d);
    if (!workspace) return fail(ATTN_ERR_NULL, "workspace is NULL");
    if (!aligned(workspace, 16)) return fail(ATTN_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (workspace_bytes < need)
        return fail(ATTN_ERR_SHAPE, "workspace too small: %lld bytes, need %lld", (long long)workspace_bytes,
                    (long long)need);
    bwd::BwdLaunchArgs a;
    if ((rc = make_map_packed(&a.q, q, dtype, total_q, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.dout, dout, dtype, total_q, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.k, k, dtype, total_k, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.v, v, dtype, total_k, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_f32_packed(&a.dq_acc, workspace, total_q, h, d)) != ATTN_OK) return rc;
    bwd::BwdParams &p = a.p;
    const int64_t sq_pad = bwd_sq_pad(max_q);
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq_acc = static_cast<float *>(workspace);
    p.lse2 = p.dq_acc + total_q * h * d;
    p.dsum = p.lse2 + bh * sq_pad;
    p.counter = reinterpret_cast<int32_t *>(p.dsum + bh * sq_pad);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = di->status;
    p.bh = static_cast<int32_t>(bh);
    p.sq = static_cast<int32_t>(max_q);
    p.sk = static_cast<int32_t>(max_k);
    p.sq_pad = static_cast<int32_t>(sq_pad);
    p.num_kblk = static_cast<int32_t>(num_kblk);
    p.num_units = static_cast<int32_t>(bh * num_kblk);
    p.group = bwd_group(bh, max_q, d);
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.heads = static_cast<int32_t>(h);
    p.total_q = static_cast<int32_t>(total_q);
    p.total_k = static_cast<int32_t>(total_k);
#ifdef ATTN_TRACE_ENABLE
    p.trace = g_trace_buf;
#endif
    p.sl2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.scale = scale;
    p.timeout_ns = kDefaultTimeoutNs;
    a.grid = p.num_units < di->sm_count ? p.num_units : di->sm_count;
    a.sm_count = di->sm_count;
    a.stream = stream;
    a.attr_ready = di->bwd_attr;
    e = launch_bwd_any<true>(a, d, dtype, causal);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "backward launch");
}

// Scratch of attn_fwd_splitkv_noalloc: a fixed device array that every GPU
// loading this library holds until the process exits.  In host code the name
// only stands for the symbol; its device address comes from
// cudaGetSymbolAddress, fetched once per device with that device current.
static __device__ __align__(256) float g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

struct NoallocSlot {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *ptr = nullptr;
};
NoallocSlot g_noalloc[kMaxDevices];

}  // namespace

extern "C" {

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h, int64_t sq,
             int64_t sk, int64_t d, int causal, float scale, int dtype, void *stream)
{
    g_err.clear();
    return run(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, static_cast<cudaStream_t>(stream), -1,
               kDefaultTimeoutNs);
}

int attn_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host, float *lse_host,
                  void *q_dev, void *k_dev, void *v_dev, void *o_dev, float *lse_dev, int64_t b, int64_t h, int64_t sq,
                  int64_t sk, int64_t d, int causal, float scale, int dtype, void *stream)
{
    g_err.clear();
    bool nothing = false;
    int rc = validate(q_dev, k_dev, v_dev, o_dev, lse_dev, b, h, sq, sk, d, scale, dtype, &nothing);
    if (rc != ATTN_OK || nothing) return rc;
    if (!o_host || (sk > 0 && (!q_host || !k_host || !v_host)))
        return fail(ATTN_ERR_NULL, "a host buffer is NULL");
    DeviceInfo *di = nullptr;
    if ((rc = device_info(&di)) != ATTN_OK) return rc;
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(&hp)) != ATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t bh = b * h;
    const int64_t qrow = sq * d * 2, krow = sk * d * 2;  // bytes per head
    const bool lse_out = lse_host && lse_dev;
    const int64_t total = bh * (2 * qrow + 2 * krow);
    const int chunks = (total < kPipeMinBytes || bh < 2) ? 1 : static_cast<int>(bh < kPipeChunks ? bh : kPipeChunks);
    const int64_t per = (bh + chunks - 1) / chunks;
    auto bytes_at = [](const void *p, int64_t off) { return static_cast<const char *>(p) + off; };
    auto mbytes_at = [](void *p, int64_t off) { return static_cast<char *>(p) + off; };

    std::lock_guard<std::mutex> lock(hp->mu);
    cudaError_t e;
    if ((e = cudaEventRecord(hp->start, st)) != cudaSuccess) return cuda_fail(e, "record start");
    if ((e = cudaStreamWaitEvent(hp->h2d, hp->start, 0)) != cudaSuccess) return cuda_fail(e, "order copies in");
    if ((e = cudaStreamWaitEvent(hp->d2h, hp->start, 0)) != cudaSuccess) return cuda_fail(e, "order copies out");
    for (int c = 0; c < chunks; ++c) {
        const int64_t h0 = c * per;
        const int64_t nh = (h0 + per <= bh) ? per : bh - h0;
        if (nh <= 0) break;
        if (sk > 0) {
            if ((e = cudaMemcpyAsync(mbytes_at(q_dev, h0 * qrow), bytes_at(q_host, h0 * qrow), nh * qrow,
                                     cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess)
                return cuda_fail(e, "copy q to device");
            if ((e = cudaMemcpyAsync(mbytes_at(k_dev, h0 * krow), bytes_at(k_host, h0 * krow), nh * krow,
                                     cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess)
                return cuda_fail(e, "copy k to device");
            if ((e = cudaMemcpyAsync(mbytes_at(v_dev, h0 * krow), bytes_at(v_host, h0 * krow), nh * krow,
                                     cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess)
                return cuda_fail(e, "copy v to device");
        }
        if ((e = cudaEventRecord(hp->in[c], hp->h2d)) != cudaSuccess) return cuda_fail(e, "record copy-in");
        if ((e = cudaStreamWaitEvent(st, hp->in[c], 0)) != cudaSuccess) return cuda_fail(e, "wait copy-in");
        // the chunk's heads seen as one batch of nh heads ([b, h] flatten to b*h)
        rc = run(bytes_at(q_dev, h0 * qrow), bytes_at(k_dev, h0 * krow), bytes_at(v_dev, h0 * krow),
                 mbytes_at(o_dev, h0 * qrow), lse_dev ? lse_dev + h0 * sq : nullptr, 1, nh, sq, sk, d, causal, scale,
                 dtype, st, -1, kDefaultTimeoutNs);
        if (rc != ATTN_OK) return rc;
        if ((e = cudaEventRecord(hp->out[c], st)) != cudaSuccess) return cuda_fail(e, "record forward");
        if ((e = cudaStreamWaitEvent(hp->d2h, hp->out[c], 0)) != cudaSuccess) return cuda_fail(e, "wait forward");
        if ((e = cudaMemcpyAsync(mbytes_at(o_host, h0 * qrow), bytes_at(o_dev, h0 * qrow), nh * qrow,
                                 cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess)
            return cuda_fail(e, "copy o to host");
        if (lse_out && (e = cudaMemcpyAsync(lse_host + h0 * sq, lse_dev + h0 * sq, nh * sq * 4, cudaMemcpyDeviceToHost,
                                            hp->d2h)) != cudaSuccess)
            return cuda_fail(e, "copy lse to host");
    }
    if ((e = cudaEventRecord(hp->done, hp->d2h)) != cudaSuccess) return cuda_fail(e, "record done");
    if ((e = cudaStreamWaitEvent(st, hp->done, 0)) != cudaSuccess) return cuda_fail(e, "wait done");
    return ATTN_OK;
}

int64_t attn_fwd_splitkv_workspace_bytes(int64_t b, int64_t h, int64_t sq, int64_t d, int num_splits)
{
    g_err.clear();
    if (b < 0 || h < 0 || sq < 0 || (d != 64 && d != 128) || num_splits < 1 || num_splits > 1024)
        return fail(ATTN_ERR_SHAPE, "invalid split-KV workspace query");
    return num_splits == 1 ? 0 : splitkv_bytes(b * h, sq, d, num_splits);
}

int attn_fwd_splitkv_default_splits(int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d, int causal)
{
    g_err.clear();
    (void)causal;
    if (b < 0 || h < 0 || sq < 0 || sk < 0 || (d != 64 && d != 128))
        return fail(ATTN_ERR_SHAPE, "invalid split-KV size query");
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    const int64_t units = b * h * ((sq + 255) / 256);
    const int64_t tiles = kv_tiles(sk);
    const int64_t sms = di->sm_count;
    // Many query rows that already fill the GPU: splitting only adds the
    // fp32 partials' traffic (a few hundred KB per unit).
    if (units <= 0 || tiles <= 1 || (units >= sms && sq > 64)) return 1;
    // Otherwise the split count whose units fill the persistent CTAs' waves
    // best, less 1% per wave (each unit has a fixed start-up cost), with at
    // least two key tiles per split.
    int64_t cap = tiles / 2 > 1 ? tiles / 2 : 1;
    if (cap > 1024) cap = 1024;
    int64_t best = 1;
    double best_score = -1.0;
    for (int64_t s = 1; s <= cap; ++s) {
        const int64_t u = units * s;
        const int64_t waves = (u + sms - 1) / sms;
        const double score = static_cast<double>(u) / static_cast<double>(waves * sms) - 0.01 * static_cast<double>(waves);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = s;
        }
    }
    return static_cast<int>(best);
}

int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h,
                     int64_t sq, int64_t sk, int64_t d, int causal, float scale, int dtype, int num_splits,
                     void *workspace, int64_t workspace_bytes, void *stream)
{
    g_err.clear();
    bool nothing = false;
    int rc = validate(q, k, v, o, lse, b, h, sq, sk, d, scale, dtype, &nothing);
    if (rc != ATTN_OK || nothing) return rc;
    if (num_splits < 1 || num_splits > 1024) return fail(ATTN_ERR_SHAPE, "num_splits %d not in 1..1024", num_splits);
    if (sk == 0 || num_splits == 1)
        return run(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, static_cast<cudaStream_t>(stream), -1,
                   kDefaultTimeoutNs);
    if (num_splits > kv_tiles(sk))
        return fail(ATTN_ERR_SHAPE, "num_splits %d exceeds the %lld key tiles of 128", num_splits,
                    (long long)kv_tiles(sk));
    const int64_t need = splitkv_bytes(b * h, sq, d, num_splits);
    if (!workspace) return fail(ATTN_ERR_NULL, "split-KV workspace is NULL (%lld bytes needed)", (long long)need);
    if (!aligned(workspace, 16)) return fail(ATTN_ERR_ALIGN, "split-KV workspace must be 16-byte aligned");
    if (workspace_bytes < need)
        return fail(ATTN_ERR_SHAPE, "split-KV workspace of %lld bytes is smaller than the %lld needed",
                    (long long)workspace_bytes, (long long)need);
    SplitArgs sa;
    sa.num_splits = num_splits;
    sa.o_part = static_cast<float *>(workspace);
    sa.lse_part = sa.o_part + static_cast<int64_t>(num_splits) * b * h * sq * d;
    return run(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, static_cast<cudaStream_t>(stream), -1,
               kDefaultTimeoutNs, sa);
}

// Split-KV forward for callers that cannot allocate device memory (see the
// header): the partial results go to the fixed scratch array above instead
// of a caller workspace.  Allocates nothing.
int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h,
                             int64_t sq, int64_t sk, int64_t d, int causal, float scale, int dtype, int num_splits,
                             void *stream)
{
    g_err.clear();
    // The checks of attn_fwd_splitkv that need no pointer come first (the
    // same codes for the same mistakes: a bad head dim is ATTN_ERR_HEADDIM);
    // they bound b*h below 2^31 and sq by 2^30, so the scratch size is
    // computed without overflow (in double, then compared).
    int rc = validate_sizes(b, h, sq, sk, d, scale, dtype);
    if (rc != ATTN_OK) return rc;
    if (num_splits < 1 || num_splits > 1024) return fail(ATTN_ERR_SHAPE, "num_splits %d not in 1..1024", num_splits);
    const double need = (num_splits == 1 || sk == 0)
                            ? 0.0
                            : static_cast<double>(num_splits) * static_cast<double>(b * h) * static_cast<double>(sq) *
                                  static_cast<double>(d + 2) * 4.0;
    if (need > static_cast<double>(ATTN_NOALLOC_SCRATCH_BYTES))
        return fail(ATTN_ERR_SHAPE,
                    "attn_fwd_splitkv_noalloc: %d splits of b=%lld h=%lld sq=%lld d=%lld need %.0f bytes of scratch, "
                    "more than its fixed %lld; use fewer splits, or attn_fwd_splitkv with a workspace",
                    num_splits, (long long)b, (long long)h, (long long)sq, (long long)d, need,
                    (long long)ATTN_NOALLOC_SCRATCH_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
    NoallocSlot &slot = g_noalloc[dev];
    std::call_once(slot.once, [&] { slot.err = cudaGetSymbolAddress(&slot.ptr, g_noalloc_scratch); });
    if (slot.err != cudaSuccess) return cuda_fail(slot.err, "cudaGetSymbolAddress of the no-alloc scratch");
    if (slot.ptr == nullptr) return fail(ATTN_ERR_CUDA, "no-alloc scratch has no device address");
    // Every element the merge reads is written earlier by the same call, so
    // nothing in the scratch has to start at zero.
    return attn_fwd_splitkv(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, num_splits, slot.ptr,
                            static_cast<int64_t>(ATTN_NOALLOC_SCRATCH_BYTES), stream);
}

// Attention against a KV cache with a length per batch element, after
// (optionally) writing the new tokens' keys and values into the cache at
// each element's current length.  Split-KV as in attn_fwd_splitkv.  With
// `paged`, the caches are page pools addressed through a block table.
struct PagedArgs {
    const int32_t *block_table;
    int64_t num_pages, page_size, pages_per_seq;
};

static int kvcache_impl(const void *q, void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                        const int32_t *cache_seqlens, void *o, float *lse, int64_t b, int64_t h, int64_t sq,
                        int64_t s_cache, int64_t s_new, int64_t d, int causal, float scale, int dtype, int num_splits,
                        void *workspace, int64_t workspace_bytes, void *stream, const PagedArgs *paged)
{
    bool nothing = false;
    int rc = validate(q, k_cache, v_cache, o, lse, b, h, sq, s_cache, d, scale, dtype, &nothing);
    if (rc != ATTN_OK) return rc;
    if (s_new < 0 || s_new > kMaxSeq) return fail(ATTN_ERR_SHAPE, "s_new %lld not in 0..2^30", (long long)s_new);
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(ATTN_ERR_NULL, "k_new and v_new must both be given or both be NULL");
    if (s_new > 0 && k_new == nullptr) return fail(ATTN_ERR_NULL, "s_new is %lld but k_new / v_new are NULL", (long long)s_new);
    if (num_splits < 1 || num_splits > 1024) return fail(ATTN_ERR_SHAPE, "num_splits %d not in 1..1024", num_splits);
    const int64_t bh = b * h;
    const bool append = bh * s_new > 0 && s_cache > 0;
    if (bh == 0 || (nothing && !append)) return ATTN_OK;
    if (cache_seqlens == nullptr) return fail(ATTN_ERR_NULL, "cache_seqlens is NULL");
    if (!aligned(cache_seqlens, 4)) return fail(ATTN_ERR_ALIGN, "cache_seqlens must be 4-byte aligned");
    if (paged) {
        if (paged->block_table == nullptr) return fail(ATTN_ERR_NULL, "block_table is NULL");
        if (!aligned(paged->block_table, 4)) return fail(ATTN_ERR_ALIGN, "block_table must be 4-byte aligned");
    }
    const int64_t esz = 2;  // fp16 / bf16 (validate checked the dtype)
    if (append) {
        if (!k_cache || !v_cache) return fail(ATTN_ERR_NULL, "k_cache or v_cache is NULL");
        if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
            return fail(ATTN_ERR_ALIGN, "k_new, v_new, k_cache and v_cache must be 16-byte aligned");
        // the copy reads the new rows while it writes the cache: no overlap
        const uintptr_t nb = static_cast<uintptr_t>(bh * s_new * d * esz);
        const uintptr_t cb = static_cast<uintptr_t>(paged ? paged->num_pages * paged->page_size * h * d * esz
                                                          : bh * s_cache * d * esz);
        const void *news[2] = {k_new, v_new};
        const void *caches[2] = {k_cache, v_cache};
        for (const void *nw : news)
            for (const void *ca : caches) {
                const uintptr_t a0 = reinterpret_cast<uintptr_t>(nw), c0 = reinterpret_cast<uintptr_t>(ca);
                if (a0 < c0 + cb && c0 < a0 + nb)
                    return fail(ATTN_ERR_SHAPE, "k_new / v_new overlap k_cache / v_cache");
            }
    }
    if (!nothing && s_cache > 0 && num_splits > kv_tiles(s_cache))
        return fail(ATTN_ERR_SHAPE, "num_splits %d exceeds the %lld key tiles of 128", num_splits,
                    (long long)kv_tiles(s_cache));
    SplitArgs sa;
    if (!nothing && s_cache > 0 && num_splits > 1) {
        const int64_t need = splitkv_bytes(bh, sq, d, num_splits);
        if (!workspace) return fail(ATTN_ERR_NULL, "split-KV workspace is NULL (%lld bytes needed)", (long long)need);
        if (!aligned(workspace, 16)) return fail(ATTN_ERR_ALIGN, "split-KV workspace must be 16-byte aligned");
        if (workspace_bytes < need)
            return fail(ATTN_ERR_SHAPE, "split-KV workspace of %lld bytes is smaller than the %lld needed",
                        (long long)workspace_bytes, (long long)need);
        sa.num_splits = num_splits;
        sa.o_part = static_cast<float *>(workspace);
        sa.lse_part = sa.o_part + static_cast<int64_t>(num_splits) * bh * sq * d;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (append) {
        DeviceInfo *di = nullptr;
        rc = device_info(&di);
        if (rc != ATTN_OK) return rc;
        const int dd = static_cast<int>(d);
        cudaError_t e;
        if (paged)
            e = (dtype == ATTN_BF16)
                    ? launch_kvcache_append_paged<__nv_bfloat16>(k_new, v_new, k_cache, v_cache, cache_seqlens,
                                                                 paged->block_table, bh, h, s_new, paged->pages_per_seq,
                                                                 paged->page_size, paged->num_pages, dd, di->sm_count, st)
                    : launch_kvcache_append_paged<__half>(k_new, v_new, k_cache, v_cache, cache_seqlens,
                                                          paged->block_table, bh, h, s_new, paged->pages_per_seq,
                                                          paged->page_size, paged->num_pages, dd, di->sm_count, st);
        else
            e = (dtype == ATTN_BF16) ? launch_kvcache_append<__nv_bfloat16>(k_new, v_new, k_cache, v_cache, cache_seqlens,
                                                                             bh, h, s_new, s_cache, dd, di->sm_count, st)
                                     : launch_kvcache_append<__half>(k_new, v_new, k_cache, v_cache, cache_seqlens, bh, h,
                                                                     s_new, s_cache, dd, di->sm_count, st);
        if (e != cudaSuccess) return cuda_fail(e, "launch (cache append)");
    }
    if (nothing) return ATTN_OK;
    CacheArgs ca;
    ca.seqlens = cache_seqlens;
    ca.add = static_cast<int32_t>(s_new);
    if (paged) {
        ca.block_table = paged->block_table;
        ca.pages_per_seq = paged->pages_per_seq;
        ca.page_size = paged->page_size;
        ca.num_pages = paged->num_pages;
    }
    return run(q, k_cache, v_cache, o, lse, b, h, sq, s_cache, d, causal, scale, dtype, st, -1, kDefaultTimeoutNs, sa,
               ca);
}

int attn_fwd_kvcache(const void *q, void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                     const int32_t *cache_seqlens, void *o, float *lse, int64_t b, int64_t h, int64_t sq,
                     int64_t s_cache, int64_t s_new, int64_t d, int causal, float scale, int dtype, int num_splits,
                     void *workspace, int64_t workspace_bytes, void *stream)
{
    g_err.clear();
    return kvcache_impl(q, k_cache, v_cache, k_new, v_new, cache_seqlens, o, lse, b, h, sq, s_cache, s_new, d, causal,
                        scale, dtype, num_splits, workspace, workspace_bytes, stream, nullptr);
}

// The KV-cache forward over a paged cache (see the header).
int attn_fwd_kvcache_paged(const void *q, void *k_pool, void *v_pool, const void *k_new, const void *v_new,
                           const int32_t *cache_seqlens, const int32_t *block_table, void *o, float *lse, int64_t b,
                           int64_t h, int64_t sq, int64_t num_pages, int64_t page_size, int64_t pages_per_seq,
                           int64_t s_new, int64_t d, int causal, float scale, int dtype, int num_splits,
                           void *workspace, int64_t workspace_bytes, void *stream)
{
    g_err.clear();
    if (page_size < 128 || page_size % 128 != 0)
        return fail(ATTN_ERR_SHAPE, "page_size %lld is not a positive multiple of 128", (long long)page_size);
    if (num_pages < 1 || pages_per_seq < 1)
        return fail(ATTN_ERR_SHAPE, "num_pages and pages_per_seq must be at least 1");
    if (num_pages > INT32_MAX / page_size)
        return fail(ATTN_ERR_SHAPE, "the pool holds more than 2^31-1 tokens");
    if (pages_per_seq > kMaxSeq / page_size)
        return fail(ATTN_ERR_SHAPE, "pages_per_seq * page_size above 2^30");
    const PagedArgs pg{block_table, num_pages, page_size, pages_per_seq};
    return kvcache_impl(q, k_pool, v_pool, k_new, v_new, cache_seqlens, o, lse, b, h, sq, pages_per_seq * page_size,
                        s_new, d, causal, scale, dtype, num_splits, workspace, workspace_bytes, stream, &pg);
}

int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_k, int64_t batch, int64_t h, int64_t total_q, int64_t total_k,
                    int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d, int causal, float scale, int dtype,
                    void *stream)
{
    g_err.clear();
    if (batch < 0 || h < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
        return fail(ATTN_ERR_SHAPE, "negative varlen size");
    if (total_q > INT32_MAX || total_k > INT32_MAX || max_seqlen_q > total_q || max_seqlen_k > total_k)
        return fail(ATTN_ERR_SHAPE, "varlen totals above 2^31-1 or max lengths above the totals");
    bool nothing = false;
    // validate pointers/d/dtype/scale as a dense problem of total_q rows
    int rc = validate(q, k, v, o, lse, 1, h, total_q, total_k, d, scale, dtype, &nothing);
    if (rc != ATTN_OK || nothing || batch == 0 || max_seqlen_q == 0) return rc;
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(ATTN_ERR_NULL, "cu_seqlens_q / cu_seqlens_k is NULL");
    if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return fail(ATTN_ERR_ALIGN, "cu_seqlens must be 4-byte aligned");
    DeviceInfo *di = nullptr;
    rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (total_k == 0) {  // no key anywhere: every row gets O = 0, LSE = -inf
        e = (dtype == ATTN_BF16) ? launch_fill_empty<__nv_bfloat16>(o, lse, total_q * h, static_cast<int>(d), st)
                                 : launch_fill_empty<__half>(o, lse, total_q * h, static_cast<int>(d), st);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "launch (empty keys)");
    }
    LaunchArgs a;
    if ((rc = make_map_packed(&a.q, q, dtype, total_q, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.k, k, dtype, total_k, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.v, v, dtype, total_k, h, d)) != ATTN_OK) return rc;
    if ((rc = make_map_packed(&a.o, o, dtype, total_q, h, d, 32)) != ATTN_OK) return rc;  // stores of 32 rows
    FwdParams &p = a.p;
    p.o = o;
    p.lse = lse;
    p.status = di->status;
    const int64_t bh = batch * h;
    if (bh > INT32_MAX) return fail(ATTN_ERR_SHAPE, "batch*h too large");
    p.bh = static_cast<int32_t>(bh);
    p.sq = static_cast<int32_t>(max_seqlen_q);
    p.sk = static_cast<int32_t>(max_seqlen_k);
    p.num_mblk = static_cast<int32_t>((max_seqlen_q + 255) / 256);
    p.num_splits = 1;
    p.o_part = nullptr;
    p.lse_part = nullptr;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.sched = sched_slot(di, &p.sched_gen);  // sequences differ in length: hand units out dynamically
    p.group = l2_group(bh, max_seqlen_k, d, 2);
    p.heads = static_cast<int32_t>(h);
    p.total_q = static_cast<int32_t>(total_q);
    p.total_k = static_cast<int32_t>(total_k);
    const int64_t units = bh * p.num_mblk;
    if (units > INT32_MAX) return fail(ATTN_ERR_SHAPE, "too many work units (%lld)", (long long)units);
    p.num_units = static_cast<int32_t>(units);
    p.sl2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.o_scale = 1.f;
    p.timeout_ns = kDefaultTimeoutNs;
    p.withheld_load = -1;
#ifdef ATTN_TRACE_ENABLE
    p.trace = g_trace_buf;
#endif
    a.grid = static_cast<int>(units < di->sm_count ? units : di->sm_count);
    a.stream = st;
    a.attr_ready = di->fwd_attr;
    const bool c = causal != 0;
    if (d == 64)
        e = (dtype == ATTN_BF16) ? dispatch_causal<64, __nv_bfloat16>(a, c) : dispatch_causal<64, __half>(a, c);
    else
        e = (dtype == ATTN_BF16) ? dispatch_causal<128, __nv_bfloat16>(a, c) : dispatch_causal<128, __half>(a, c);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch (varlen)");
    return ATTN_OK;
}

int attn_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h, int64_t sq,
                 int64_t sk, int64_t d, int causal, float scale, float descale_q, float descale_k, float descale_v,
                 void *stream)
{
    g_err.clear();
    if (d != 64 && d != 128)
        return fail(ATTN_ERR_HEADDIM, "the e4m3 forward supports head dims 64 and 128 (got %lld)", (long long)d);
    if (!std::isfinite(descale_q) || !std::isfinite(descale_k) || !std::isfinite(descale_v))
        return fail(ATTN_ERR_SCALE, "descale factors must be finite");
    const double sqk = static_cast<double>(scale) * descale_q * descale_k;
    if (!std::isfinite(sqk) || !std::isfinite(static_cast<float>(sqk)))
        return fail(ATTN_ERR_SCALE, "scale * descale_q * descale_k is not finite in fp32");
    bool nothing = false;
    // pointer, size and alignment checks as for a bf16 problem (O is bf16)
    int rc = validate(q, k, v, o, lse, b, h, sq, sk, d, scale, ATTN_BF16, &nothing);
    if (rc != ATTN_OK || nothing) return rc;
    DeviceInfo *di = nullptr;
    rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t bh = b * h;
    cudaError_t e;
    if (sk == 0) {
        e = launch_fill_empty<__nv_bfloat16>(o, lse, bh * sq, static_cast<int>(d), st);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "launch (empty keys)");
    }
    LaunchArgs a;
    if ((rc = make_map(&a.q, q, ATTN_BF16, bh, sq, d, 1)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.k, k, ATTN_BF16, bh, sk, d, 1)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.v, v, ATTN_BF16, bh, sk, d, 1)) != ATTN_OK) return rc;
    if ((rc = make_map(&a.o, o, ATTN_BF16, bh, sq, d, 2, 32)) != ATTN_OK) return rc;  // bf16 output, 32-row stores
    FwdParams &p = a.p;
    p.o = o;
    p.lse = lse;
    p.status = di->status;
    p.bh = static_cast<int32_t>(bh);
    p.sq = static_cast<int32_t>(sq);
    p.sk = static_cast<int32_t>(sk);
    p.num_mblk = static_cast<int32_t>((sq + 255) / 256);
    p.num_splits = 1;
    p.o_part = nullptr;
    p.lse_part = nullptr;
    p.cu_q = p.cu_k = nullptr;
    p.heads = static_cast<int32_t>(h);
    p.total_q = static_cast<int32_t>(sq);
    p.total_k = static_cast<int32_t>(sk);
    const int64_t units = bh * p.num_mblk;
    if (units > INT32_MAX) return fail(ATTN_ERR_SHAPE, "too many work units (%lld)", (long long)units);
    p.num_units = static_cast<int32_t>(units);
    p.sl2e = static_cast<float>(sqk * 1.4426950408889634074);
    p.o_scale = descale_v;
    p.timeout_ns = kDefaultTimeoutNs;
    p.withheld_load = -1;
#ifdef ATTN_TRACE_ENABLE
    p.trace = g_trace_buf;
#endif
    a.grid = static_cast<int>(units < di->sm_count ? units : di->sm_count);
    a.stream = st;
    a.attr_ready = di->fwd_attr;
    if (d == 64)
        e = causal ? launch_fwd<64, __nv_fp8_e4m3, true>(a) : launch_fwd<64, __nv_fp8_e4m3, false>(a);
    else
        e = causal ? launch_fwd<128, __nv_fp8_e4m3, true>(a) : launch_fwd<128, __nv_fp8_e4m3, false>(a);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch (e4m3)");
    return ATTN_OK;
}

const char *attn_last_error(void) { return g_err.c_str(); }

int attn_fwd_status(uint32_t *out)
{
    g_err.clear();
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    uint32_t w[4];
    e = cudaMemcpy(w, di->status, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read watchdog status");
    if (out) memcpy(out, w, sizeof(w));
    return static_cast<int>(w[0]);
}

int attn_fwd_status_clear(void)
{
    g_err.clear();
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    // after the device is idle, so that no launch holds a schedule slot
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(di->status, 0, 4 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(di->sched, 0, sizeof(int32_t) * kSchedWords * kSchedSlots);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "clear watchdog status");
}

int attn_fwd_debug_status(void) { return attn_fwd_status(nullptr); }

int attn_fwd_sched_pin_slot(int slot)
{
    g_err.clear();
    if (slot < -1 || slot >= kSchedSlots) return fail(ATTN_ERR_SHAPE, "slot %d not in -1..%d", slot, kSchedSlots - 1);
    DeviceInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != ATTN_OK) return rc;
    di->sched_pinned.store(slot, std::memory_order_relaxed);
    return ATTN_OK;
}

int attn_fwd_watchdog_selftest(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h,
                               int64_t sq, int64_t sk, int64_t d, int causal, float scale, int dtype, int withheld_load,
                               int timeout_ms, void *stream)
{
    g_err.clear();
    if (timeout_ms <= 0 || timeout_ms > 10000) return fail(ATTN_ERR_SHAPE, "timeout_ms must be in 1..10000");
    if (withheld_load < 0) return fail(ATTN_ERR_SHAPE, "withheld_load must be >= 0");
    if (b < 0 || h < 0 || sq < 0 || b * h * sq > 4096 || sk > 1024)
        return fail(ATTN_ERR_SHAPE, "self-test wants a tiny problem");
    int rc = attn_fwd_status_clear();
    if (rc != ATTN_OK) return rc;
    rc = run(q, k, v, o, lse, b, h, sq, sk, d, causal, scale, dtype, static_cast<cudaStream_t>(stream), withheld_load,
             static_cast<uint64_t>(timeout_ms) * 1000000ull);
    if (rc != ATTN_OK) return rc;
    return attn_fwd_status(nullptr);
}

int attn_fwd_bounds_selftest(const void *q, const void *k, const void *v, void *o, float *lse, int64_t b, int64_t h,
                             int64_t sq, int64_t sk, int64_t d, float scale, int dtype, void *stream)
{
    g_err.clear();
#if ATTN_CHECKED
    if (b < 0 || h < 0 || sq < 1 || sk < 1 || b * h * sq > 4096 || sk > 1024)
        return fail(ATTN_ERR_SHAPE, "self-test wants a tiny problem with rows and keys");
    int rc = attn_fwd_status_clear();
    if (rc != ATTN_OK) return rc;
    // one unit past the end of a dense, unsplit problem: the decoded head
    // plane is out of range, which the checks catch before any access
    rc = run(q, k, v, o, lse, b, h, sq, sk, d, 0, scale, dtype, static_cast<cudaStream_t>(stream), -1,
             kDefaultTimeoutNs, SplitArgs(), CacheArgs(), 1);
    if (rc != ATTN_OK) return rc;
    return attn_fwd_status(nullptr);
#else
    (void)q, (void)k, (void)v, (void)o, (void)lse, (void)b, (void)h, (void)sq, (void)sk, (void)d, (void)scale;
    (void)dtype, (void)stream;
    return fail(ATTN_ERR_BUILD, "attn_fwd_bounds_selftest needs the checked build (libattn_fwd_checked.so)");
#endif
}

int attn_bwd_watchdog_selftest(const void *q, const void *k, const void *v, const void *o, const void *dout,
                               const float *lse, void *dq, void *dk, void *dv, int64_t b, int64_t h, int64_t sq,
                               int64_t sk, int64_t d, int causal, float scale, int dtype, void *workspace,
                               int64_t workspace_bytes, int withheld_load, int timeout_ms, void *stream)
{
    g_err.clear();
#if ATTN_CHECKED
    if (timeout_ms <= 0 || timeout_ms > 10000) return fail(ATTN_ERR_SHAPE, "timeout_ms must be in 1..10000");
    if (withheld_load < 0) return fail(ATTN_ERR_SHAPE, "withheld_load must be >= 0");
    if (b < 1 || h < 1 || sq < 1 || sk < 1 || b * h * sq > 4096 || sk > 1024)
        return fail(ATTN_ERR_SHAPE, "self-test wants a tiny problem with rows and keys");
    int rc = attn_fwd_status_clear();
    if (rc != ATTN_OK) return rc;
    rc = run_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, sq, sk, d, causal, scale, dtype, workspace, workspace_bytes,
                 static_cast<cudaStream_t>(stream), 0, withheld_load, static_cast<uint64_t>(timeout_ms) * 1000000ull);
    if (rc != ATTN_OK) return rc;
    return attn_fwd_status(nullptr);
#else
    (void)q, (void)k, (void)v, (void)o, (void)dout, (void)lse, (void)dq, (void)dk, (void)dv, (void)b, (void)h;
    (void)sq, (void)sk, (void)d, (void)causal, (void)scale, (void)dtype, (void)workspace, (void)workspace_bytes;
    (void)withheld_load, (void)timeout_ms, (void)stream;
    return fail(ATTN_ERR_BUILD, "attn_bwd_watchdog_selftest needs the checked build (libattn_fwd_checked.so)");
#endif
}

int attn_bwd_bounds_selftest(const void *q, const void *k, const void *v, const void *o, const void *dout,
                             const float *lse, void *dq, void *dk, void *dv, int64_t b, int64_t h, int64_t sq,
                             int64_t sk, int64_t d, float scale, int dtype, void *workspace, int64_t workspace_bytes,
                             void *stream)
{
    g_err.clear();
#if ATTN_CHECKED
    if (b < 1 || h < 1 || sq < 1 || sk < 1 || b * h * sq > 4096 || sk > 1024)
        return fail(ATTN_ERR_SHAPE, "self-test wants a tiny problem with rows and keys");
    int rc = attn_fwd_status_clear();
    if (rc != ATTN_OK) return rc;
    // one unit past the end of a dense, unmasked problem: its index is out of
    // range, which every warp role finds before decoding it
    rc = run_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, sq, sk, d, 0, scale, dtype, workspace, workspace_bytes,
                 static_cast<cudaStream_t>(stream), 1);
    if (rc != ATTN_OK) return rc;
    return attn_fwd_status(nullptr);
#else
    (void)q, (void)k, (void)v, (void)o, (void)dout, (void)lse, (void)dq, (void)dk, (void)dv, (void)b, (void)h;
    (void)sq, (void)sk, (void)d, (void)scale, (void)dtype, (void)workspace, (void)workspace_bytes, (void)stream;
    return fail(ATTN_ERR_BUILD, "attn_bwd_bounds_selftest needs the checked build (libattn_fwd_checked.so)");
#endif
}

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse, void *dq,
             void *dk, void *dv, int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d, int causal, float scale,
             int dtype, void *workspace, int64_t workspace_bytes, void *stream)
{
    g_err.clear();
    return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, sq, sk, d, causal, scale, dtype, workspace,
                   workspace_bytes, static_cast<cudaStream_t>(stream));
}

int attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                    void *dq, void *dk, void *dv, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                    int64_t batch, int64_t h, int64_t total_q, int64_t total_k, int64_t max_seqlen_q,
                    int64_t max_seqlen_k, int64_t d, int causal, float scale, int dtype, void *workspace,
                    int64_t workspace_bytes, void *stream)
{
    g_err.clear();
    return run_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, h, total_q, total_k,
                          max_seqlen_q, max_seqlen_k, d, causal, scale, dtype, workspace, workspace_bytes,
                          static_cast<cudaStream_t>(stream));
}

int64_t attn_bwd_varlen_workspace_bytes(int64_t batch, int64_t h, int64_t total_q, int64_t max_seqlen_q, int64_t d)
{
    g_err.clear();
    if (batch < 0 || h < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_q > total_q || total_q > INT32_MAX)
        return fail(ATTN_ERR_SHAPE, "invalid varlen backward workspace query");
    if (d != 64 && d != 128) return fail(ATTN_ERR_HEADDIM, "backward: head dim %lld not supported (64 or 128)", (long long)d);
    return bwd_varlen_workspace_bytes(batch, h, total_q, max_seqlen_q, d);
}

int64_t attn_bwd_workspace_bytes(int64_t b, int64_t h, int64_t sq, int64_t d)
{
    g_err.clear();
    if (b < 0 || h < 0 || sq < 0 || sq > kMaxSeq || (b > 0 && h >= (int64_t(1) << 31) / b))
        return fail(ATTN_ERR_SHAPE, "invalid backward workspace query");
    if (d != 64 && d != 128) return fail(ATTN_ERR_HEADDIM, "backward: head dim %lld not supported (64 or 128)", (long long)d);
    return bwd_workspace_bytes(b * h, sq, d);
}

const char *attn_version(void) { return "attn_fwd sm_103a 0.1"; }

#ifdef ATTN_TRACE_ENABLE
// Timeline builds only: device buffer that later launches record into.
void attn_trace_set(unsigned long long *device_buffer) { g_trace_buf = device_buffer; }
#endif

}  // extern "C"
