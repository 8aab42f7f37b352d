// Attention backward for sm_103a (GB300): gradients dQ, dK, dV of
// O = softmax(scale * Q K^T [+ causal]) V for a given dO, from the forward's
// O and natural log-sum-exp LSE.
//
// What is computed (the chain rule through the forward's definition; the
// pages name the backward -- the bwd / varlen_bwd entry points of
// "05 · kernel 工程与四代演化" 6.1 -- without stating it):
//   P = exp(scale * Q K^T - LSE)   (recomputed; masked keys give 0)
//   dV = P^T dO,   dP = dO V^T,   D = rowsum(dO * O)  ( = rowsum(P * dP) )
//   dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q
//
// Three launches on the caller's stream:
//   attn_bwd_prep_kernel    D per query row, LSE * log2(e) per row (+inf for
//                           padding and rows that see no key), and a zeroed
//                           fp32 dQ accumulator;
//   attn_bwd_kernel         one persistent CTA per SM; a work unit is one
//                           block of 128 keys of one head.  K and V stay in
//                           shared memory while the unit streams 128-query
//                           tiles of Q, dO (and their LSE, D) through a
//                           two-stage TMA ring.  Per tile, on the tensor
//                           cores (tcgen05.mma, accumulators in TMEM):
//                             S^T  = K Q^T           [keys x queries]
//                             dP^T = V dO^T
//                             dV  += P^T dO          (P^T read from TMEM)
//                             dK  += dS^T Q          (dS^T read from TMEM)
//                             dQ^T = K^T dS^T        (both from shared)
//                           dV and dK accumulate in TMEM over the tiles of
//                           the unit; each tile's dQ is staged in shared
//                           memory and added into the fp32 accumulator by
//                           the copy engine (a TMA reduce-add);
//   attn_bwd_dq_convert_kernel  dQ = accumulator cast to the input type.
//
// CTA of 16 warps:
//   warps 0-3 / 4-7   softmax groups: each thread owns one key row (a TMEM
//                     lane) and 64 of the tile's 128 query columns; it
//                     turns S^T into P^T (kept in fp32 registers, stored to
//                     TMEM as 16-bit for the dV product) and dP^T into dS^T
//                     (stored to TMEM for dK and to shared memory for dQ)
//   warps 8-11        dQ drain (TMEM -> shared -> TMA reduce-add) and the dK / dV
//                     epilogue of each unit
//   warp 12           MMA issuer, tensor-memory owner
//   warp 13           TMA producer
//   warps 14-15       no work (they complete warpgroup 3)
// Tensor memory (512 columns): dV [0,128), dK [128,256), S^T/P^T [256,384),
// dP^T/dS^T then dQ^T [384,512).
//
// Every wait is bounded, as in the forward: a wait that runs out records
// where in the status word, raises the CTA's abort flag, and the CTA winds
// down (copies and MMAs drained, tensor memory freed) and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <type_traits>

#include "ptx.cuh"

// Checked build: with ATTN_CHECKED=1 every computed copy coordinate, global
// output offset, decoded unit, tensor-memory base and shared-memory window
// of the backward is compared with its bounds (see in_bounds).  Off by
// default.
#ifndef ATTN_CHECKED
#define ATTN_CHECKED 0
#endif

namespace attn {
namespace bwd {

struct BwdParams {
    const void *o;         // forward output [bh, sq, D] of T   (prep)
    const void *dout;      // dO [bh, sq, D] of T                (prep)
    const float *lse;      // forward LSE [bh, sq] (natural log)  (prep)
    float *lse2;           // [bh, sq_pad]: LSE * log2(e); +inf for padding / no key
    float *dsum;           // [bh, sq_pad]: D = rowsum(dO * O); 0 for padding
    float *dq_acc;         // [bh, sq, D] fp32 accumulator of dQ
    void *dq;              // [bh, sq, D] of T                   (convert)
    void *dk, *dv;         // [bh, sk, D] of T
    uint32_t *status;      // watchdog status word (4 x u32)
    int32_t bh, sq, sk, sq_pad;
    int32_t num_kblk;      // ceil(sk / 128)
    int32_t num_units;     // bh * num_kblk
    int32_t group;         // heads per scheduling group (see decode_unit)
    int32_t *counter;      // next unit to hand out (zeroed by the prep kernel)
    // Varlen (packed sequences): cu_q / cu_k are the batch+1 cumulative
    // offsets (device int32).  Q, O, dO, dQ and the dQ accumulator are
    // [total_q, heads, D]; K, V, dK, dV [total_k, heads, D]; LSE [heads,
    // total_q].  bh is then batch * heads (sequence-major), sq / sk the
    // maximum lengths, and lse2 / dsum are [bh, sq_pad] per sequence.
    // nullptr: the dense [b, h, s, D] layout.
    const int32_t *cu_q;
    const int32_t *cu_k;
    int32_t heads;
    int32_t total_q, total_k;
    float sl2e;            // scale * log2(e)
    float scale;           // folded into dS
    uint64_t timeout_ns;
#if ATTN_CHECKED
    int32_t withheld_load = -1;  // watchdog self-test: this CTA-local Q load is never issued
#endif
#ifdef ATTN_TRACE_ENABLE
    unsigned long long *trace;  // per-warp event records (timeline builds only)
#endif
};

// Pipeline timeline hooks, compiled out unless ATTN_TRACE_ENABLE is defined
// (a separate diagnostic build recording {clock, event, arg} per warp).
#ifdef ATTN_TRACE_ENABLE
#define BWD_TRACE_DECL uint32_t bwd_trace_n = 0;
#define BWD_TRACE(ev, arg) bwd_trace_record(p, bwd_trace_n, (ev), (arg))
__device__ __forceinline__ void bwd_trace_record(const BwdParams &p, uint32_t &n, uint32_t ev, uint32_t arg)
{
    constexpr uint32_t kCtas = 4, kWarps = 16, kEvents = 16384;
    if (p.trace == nullptr || blockIdx.x >= kCtas || (threadIdx.x & 31) != 0 || n >= kEvents) return;
    const uint32_t w = threadIdx.x >> 5;
    unsigned long long *rec = p.trace + 2ull * ((blockIdx.x * kWarps + w) * kEvents + n);
    rec[0] = clock64();
    rec[1] = (static_cast<unsigned long long>(ev) << 32) | arg;
    ++n;
}
#else
#define BWD_TRACE_DECL
#define BWD_TRACE(ev, arg) ((void)0)
#endif

enum : uint32_t {
    BEV_MMA_WAIT_P = 1, BEV_MMA_GOT_P, BEV_MMA_WAIT_DS, BEV_MMA_GOT_DS, BEV_MMA_WAIT_DQE, BEV_MMA_GOT_DQE,
    BEV_MMA_WAIT_Q, BEV_MMA_GOT_Q, BEV_MMA_ISSUED_DV, BEV_MMA_ISSUED_S, BEV_MMA_ISSUED_DKDQ, BEV_MMA_ISSUED_DP,
    BEV_SM_WAIT_S = 20, BEV_SM_GOT_S, BEV_SM_P_DONE, BEV_SM_WAIT_DP, BEV_SM_GOT_DP, BEV_SM_DS_DONE,
    BEV_DR_WAIT = 40, BEV_DR_GOT, BEV_DR_RELEASED, BEV_DR_DONE, BEV_DR_DKV_WAIT, BEV_DR_DKV_GOT, BEV_DR_DKV_DONE,
    BEV_LD_WAIT = 60, BEV_LD_GOT,
};

enum : uint32_t {
    SITE_BWD_LOAD_KV_EMPTY = 21,
    SITE_BWD_LOAD_Q_EMPTY = 22,
    SITE_BWD_MMA_KV_FULL = 23,
    SITE_BWD_MMA_Q_FULL = 24,
    SITE_BWD_MMA_P_FULL = 25,
    SITE_BWD_MMA_DS_FULL = 26,
    SITE_BWD_MMA_DQ_EMPTY = 27,
    SITE_BWD_MMA_DKV_EMPTY = 28,
    SITE_BWD_SM_S_FULL = 29,
    SITE_BWD_SM_DP_FULL = 30,
    SITE_BWD_DRAIN_DQ_FULL = 31,
    SITE_BWD_DRAIN_DKV_FULL = 32,
    SITE_BWD_SMEM_ALIGN = 33,
    SITE_BWD_UNIT_FULL = 34,
    SITE_BWD_UNIT_EMPTY = 35,
    SITE_BWD_LOAD_DO_EMPTY = 36,
    SITE_BWD_MMA_DO_FULL = 37,
    SITE_BWD_DRAIN_SYNC = 38,
    // checked builds: the index that failed its bounds
    SITE_BWD_CHK_SMEM = 40,     // dynamic shared memory window too small for the layout
    SITE_BWD_CHK_TMEM = 41,     // tensor-memory allocation not the expected 512 columns at lane 0
    SITE_BWD_CHK_UNIT = 42,     // claimed or decoded unit outside the problem
    SITE_BWD_CHK_KV_LOAD = 43,  // K/V copy coordinates
    SITE_BWD_CHK_Q_LOAD = 44,   // Q / dO copy coordinates, LSE / D vector rows
    SITE_BWD_CHK_DQ_RED = 45,   // dQ reduce-add coordinates
    SITE_BWD_CHK_DKV_ROW = 46,  // dK / dV row written by a thread
    SITE_BWD_CHK_PREP = 47,     // prep kernel: O / dO / accumulator / LSE offsets
};

// Status codes (the forward's): a wait that ran out, and an index or layout
// outside its bounds.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBounds = 3u;

// Sizes for head dim D (64 or 128).  Tiles are always 128 rows (keys or
// queries) of 128-byte swizzle panels of 64 elements.
template <int D_>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int BN = 128;                  // keys per unit = TMEM lanes
    static constexpr int BM = 128;                  // queries per tile
    static constexpr int PANEL_BYTES = 128 * 128;   // 128 rows x 128 B (64 elements)
    static constexpr int NPANEL = D / 64;
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;  // a Q, K, V or dO tile [128 rows][D]
    static constexpr int DS_BYTES = 2 * PANEL_BYTES;          // dS^T [128 keys][128 queries]
    // D = 128: dQ^T = K^T dS^T (lanes = head dim), staged in the tile's dO
    // slot.  D = 64: dQ = dS K (lanes = queries: an M = 64 product would
    // have another accumulator layout), staged in a buffer of its own.
    static constexpr bool DQ_T = (D == 128);
    static constexpr int STAGE_BYTES = DQ_T ? 0 : BM * D * 4;
    // stages of the Q / dO ring (a third at D = 64, where it fits, was slower)
    static constexpr int NSTAGE = 2;
    // rows of dQ per reduce-add when D = 128 (the staged half-tile of 64
    // rows is sent as 64 / RED_ROWS bulk reduces)
#ifndef ATTN_BWD_RED_ROWS
#define ATTN_BWD_RED_ROWS 64
#endif
    static constexpr int RED_ROWS = ATTN_BWD_RED_ROWS;
    static_assert(64 % RED_ROWS == 0, "reduce rows");
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int CTL_OFF = 0;               // barriers, TMEM address, abort flag
    static constexpr int LD_OFF = 1024;             // per stage: lse2[128], dsum[128]
    static constexpr int LD_STAGE_BYTES = 1024;
    static constexpr int K_OFF = LD_OFF + NSTAGE * LD_STAGE_BYTES;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int Q_OFF = V_OFF + TILE_BYTES;  // stage s: Q at Q_OFF + s*2*TILE, dO after it
    static constexpr int DS_OFF = Q_OFF + NSTAGE * 2 * TILE_BYTES;
    static constexpr int ST_OFF = DS_OFF + DS_BYTES;  // dQ staging (D = 64)
    static constexpr int SMEM_BYTES = ST_OFF + STAGE_BYTES;
    // tensor memory columns.  D = 128 fills all 512, and dQ^T reuses the
    // dP^T / dS^T columns; D = 64 gives dQ 64 columns of its own, so that
    // the next tile's dP^T need not wait for dQ to leave tensor memory.
    static constexpr int TM_DV = 0, TM_DK = D, TM_S = 2 * D, TM_DP = 2 * D + 128;
    static constexpr int TM_DQ = DQ_T ? TM_DP : TM_DP + 128;
    static constexpr int TMEM_COLS = 512;
    static constexpr int THREADS = 512;
    // setmaxnreg budgets: 2 x 128 softmax threads, 128 drain threads (a
    // dQ row of the tile in registers: 128 values for D = 128, 64 for
    // D = 64), 128 others; both splits add up to 512 * 128 registers, the
    // launch's 128 per thread: (144 + 144 + 136 + 88) and (152 + 152 + 120 + 88).
    static constexpr int REGS_SOFTMAX = D == 128 ? 144 : 152;
    static constexpr int REGS_DRAIN = D == 128 ? 136 : 120;
    static constexpr int REGS_OTHER = 88;
    static_assert(LD_OFF + NSTAGE * LD_STAGE_BYTES <= K_OFF, "control / LSE area");
    static_assert(K_OFF % 1024 == 0 && V_OFF % 1024 == 0 && Q_OFF % 1024 == 0 && DS_OFF % 1024 == 0 &&
                      ST_OFF % 1024 == 0, "swizzle atoms need 1 KiB alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(NSTAGE == 2, "stage barriers in Ctl");
    static_assert(TM_DP + 128 <= TMEM_COLS && TM_DQ + (DQ_T ? BM : D) <= TMEM_COLS, "tensor memory budget");
    static_assert(REGS_SOFTMAX * 2 + REGS_DRAIN + REGS_OTHER == 4 * 128, "register split");
};

struct Ctl {
    uint64_t kv_full, kv_empty;
    uint64_t q_full[2], q_empty[2];    // Q and the LSE / D vectors of a stage
    uint64_t do_full[2], do_empty[2];  // dO of a stage (its slot also stages dQ when D = 128)
    uint64_t s_full, dp_full, p_full, ds_full;
    uint64_t dq_full, dq_empty;
    uint64_t dkv_full, dkv_empty;
    uint64_t mma_done;
    uint64_t dr_sync;                      // the four drain warps meet here
    uint64_t unit_full[4], unit_empty[4];  // ring of claimed unit indices
    int32_t unit_idx[4];
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Ctl) <= 1024, "control block");
constexpr int kUnitRing = 4;
constexpr int kUnitReaders = 13;  // MMA warp + 8 softmax warps + 4 drain warps

// ---------------------------------------------------------------- PTX used only here

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Tile reduce-add shared -> global through the copy engine (the adds are
// done at L2), tracked as a bulk group of this thread.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ... and have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 16 columns of 32-bit from this thread's lane.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 64 columns of 32-bit from this thread's lane (two loads, one wait).
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&r)[64])
{
#define BWD_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : BWD_R8(0), BWD_R8(8), BWD_R8(16), BWD_R8(24), BWD_R8(32), BWD_R8(40), BWD_R8(48), BWD_R8(56)
        : "r"(taddr), "r"(taddr + 32)
        : "memory");
#undef BWD_R8
}

// Instruction descriptor, kind::f16, fp32 accumulate, with the major-ness
// of both operands (bit 15: A MN-major, bit 16: B MN-major).
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool bf16, bool a_mn, bool b_mn)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Zero rows [valid, 128) of a shared-memory tile of NPANEL panels of 128
// rows x 128 bytes (a row is 128 contiguous bytes of a panel whatever the
// swizzle).  Packed sequences: a tile that runs past a sequence's end holds
// the next sequence's tokens, which every product must see as zeros (their
// probabilities are zero, but 0 * x with x non-finite would not be).  Called
// by a whole warp; the proxy fence makes the stores visible to the tensor
// cores, which the elected lane drives after the closing __syncwarp.
template <int NPANEL>
__device__ __forceinline__ void zero_rows_from(uint32_t tile, int valid)
{
    if (valid >= 128) return;
    const int lane = threadIdx.x & 31;
    const int first = valid > 0 ? valid : 0;
    const int chunks = (128 - first) * 8;  // 16-byte chunks per panel
    for (int pn = 0; pn < NPANEL; ++pn)
        for (int c = lane; c < chunks; c += 32)
            st_shared_v4(tile + pn * 16384 + first * 128 + c * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    __syncwarp();
}

// ---------------------------------------------------------------- waits

// Forced inline: the callers run under different setmaxnreg budgets.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, Ctl *ctl, const BwdParams &p, uint32_t site)
{
    volatile uint32_t *abort_flag = &ctl->abort;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1u;
            if (atomicCAS(&p.status[0], 0u, kStatusTimeout) == 0u) {
                p.status[1] = blockIdx.x;
                p.status[2] = threadIdx.x >> 5;
                p.status[3] = site;
                __threadfence();
            }
            return false;
        }
    }
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, Ctl *ctl, const BwdParams &p, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, ctl, p, site);
}

// bar_wait by every lane of a warp, with a warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl *ctl, const BwdParams &p, uint32_t site)
{
    const bool w = bar_wait(bar, parity, ctl, p, site);
    return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ void record_bounds(const BwdParams &p, uint32_t site)
{
    if (atomicCAS(&p.status[0], 0u, kStatusBounds) == 0u) {
        p.status[1] = blockIdx.x;
        p.status[2] = threadIdx.x >> 5;
        p.status[3] = site;
        __threadfence();
    }
}

// Checked builds: `ok` false records kStatusBounds at `site` and raises the
// CTA's abort flag, so that the other warps wind down as after a wait that
// ran out; the caller skips the access.  Normal builds: always true (the
// condition is not evaluated).
#if ATTN_CHECKED
#define BWD_IN_BOUNDS(cond, site) in_bounds((cond), ctl, p, (site))
__device__ __forceinline__ bool in_bounds(bool ok, Ctl *ctl, const BwdParams &p, uint32_t site)
{
    if (!ok) {
        *reinterpret_cast<volatile uint32_t *>(&ctl->abort) = 1u;
        record_bounds(p, site);
    }
    return ok;
}
#else
#define BWD_IN_BOUNDS(cond, site) true
#endif

// Bounded wait that ignores the abort flag (lets this thread's own copies
// and MMAs land before the CTA frees its resources).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > timeout_ns) break;
}

// ---------------------------------------------------------------- schedule

struct Unit {
    int bh;      // (sequence, head) index: rows of lse2 / dsum; dense: the head plane
    int head;    // varlen: head index (a TMA coordinate of the packed maps)
    int kb;      // key block (keys 128*kb ..)
    int sq, sk;  // query / key length of the unit's sequence
    int q_tok0;  // varlen: token of query 0 / key 0 of the sequence (else 0)
    int k_tok0;
    int t0;      // first query tile that sees a key of the block
    int n;       // number of query tiles (0: no work for the MMAs)
    bool zero;   // the block has keys but the sequence has no query: dK = dV = 0
};

// Units are handed out in order from a global counter (dynamic
// scheduling).  The order is by groups of `group` heads; within a group, by
// key block (block 0 sees every query tile when causal: the heaviest
// first), then head.  A group's fp32 dQ accumulator, Q and dO are sized on
// the host to stay in L2 while its units run, and the light blocks of the
// last group fill the tail.  Key j sees query i iff j <= i + (sk - sq)
// (bottom-right alignment, as in the forward).
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Unit decode_unit(int u, const BwdParams &p)
{
    Unit un;
    const int per_group = p.group * p.num_kblk;
    const int g = u / per_group;
    const int r = u - g * per_group;
    const int h0 = g * p.group;
    const int gsz = min(p.group, p.bh - h0);
    un.kb = r / gsz;
    un.bh = h0 + (r - un.kb * gsz);
    if constexpr (VARLEN) {
        const int seq = un.bh / p.heads;
        un.head = un.bh - seq * p.heads;
        un.q_tok0 = p.cu_q[seq];
        un.sq = p.cu_q[seq + 1] - un.q_tok0;
        un.k_tok0 = p.cu_k[seq];
        un.sk = p.cu_k[seq + 1] - un.k_tok0;
        // offsets outside the packed tensors: treat as an empty sequence
        if (un.q_tok0 < 0 || un.sq < 0 || un.q_tok0 + un.sq > p.total_q || un.k_tok0 < 0 || un.sk < 0 ||
            un.k_tok0 + un.sk > p.total_k)
            un.sq = un.sk = 0;
    } else {
        un.head = 0;
        un.q_tok0 = un.k_tok0 = 0;
        un.sq = p.sq;
        un.sk = p.sk;
    }
    constexpr int BM = 128, BN = 128;  // query tile, key block (both sizes)
    const bool has_keys = un.kb * BN < un.sk;
    const int n_tiles = has_keys ? (un.sq + BM - 1) / BM : 0;
    int t0 = 0;
    if (CAUSAL) {
        const int first_q = un.kb * BN - (un.sk - un.sq);  // smallest query that sees key 128*kb
        t0 = first_q > 0 ? first_q / BM : 0;
    }
    un.t0 = min(t0, n_tiles);
    un.n = n_tiles - un.t0;
    un.zero = has_keys && un.n == 0;
    return un;
}

// Checked builds: the decoded unit lies within the problem (its key block,
// head plane, query tiles and, packed, its sequence's token ranges).
template <bool VARLEN>
__device__ __forceinline__ bool unit_ok(const Unit &un, const BwdParams &p)
{
    bool in = un.bh >= 0 && un.bh < p.bh && un.kb >= 0 && un.kb < p.num_kblk && un.t0 >= 0 && un.n >= 0 &&
              (un.t0 + un.n) * 128 < un.sq + 128;
    if constexpr (VARLEN)
        in = in && un.head >= 0 && un.head < p.heads && un.q_tok0 >= 0 && un.q_tok0 + un.sq <= p.total_q &&
             un.k_tok0 >= 0 && un.k_tok0 + un.sk <= p.total_k;
    else
        in = in && un.sq == p.sq && un.sk == p.sk;
    return in;
}

// The k-th unit index of this CTA from the ring (-1: no more work), read by
// a whole warp; lane 0 then releases the slot.
__device__ __forceinline__ bool next_unit(uint32_t k, int &u, Ctl *ctl, const BwdParams &p)
{
    const uint32_t slot = k % kUnitRing;
    const uint32_t full = smem_addr(&ctl->unit_full[slot]);
    if (!warp_wait(full, (k / kUnitRing) & 1u, ctl, p, SITE_BWD_UNIT_FULL)) return false;
    u = *reinterpret_cast<volatile int32_t *>(&ctl->unit_idx[slot]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&ctl->unit_empty[slot]));
    return true;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t u);

template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t u)
{
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u));
}

template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t u)
{
    return __half22float2(*reinterpret_cast<__half2 *>(&u));
}

// ---------------------------------------------------------------- prep

// One query row per D/8 threads: D = sum_c dO[c] O[c] (fp32), the row's
// LSE in base 2, and a zeroed accumulator row.  Rows past the sequence's
// query count (up to sq_pad) get the padding values (LSE2 = +inf, so that
// P = 0 there, and D = 0).
template <typename T, int D, bool VARLEN>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p)
{
    constexpr int TPR = D / 8;  // threads per row, 8 elements each
    // rows is a multiple of 128 (sq_pad is) and the rows of a warp are
    // consecutive, so all of a warp's rows run the same iterations and the
    // TPR-wide shuffles below always have their whole warp.
    const int64_t rows = static_cast<int64_t>(p.bh) * p.sq_pad;
    const int sub = threadIdx.x % TPR;
    const int shift = (TPR == 16) ? 4 : 3;
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.counter = 0;
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> shift; r < rows;
         r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> shift) {
        const int64_t bh = r / p.sq_pad;  // (sequence, head) when packed; the head plane when dense
        const int i = static_cast<int>(r - bh * p.sq_pad);
        // where query row i of this (sequence, head) lives
        int sq = p.sq;
        int64_t elem, lse_at;  // element offset of the row in O / dO / dQ, and its LSE index
        if constexpr (VARLEN) {
            const int seq = static_cast<int>(bh / p.heads);
            const int head = static_cast<int>(bh - static_cast<int64_t>(seq) * p.heads);
            const int tok0 = p.cu_q[seq];
            sq = p.cu_q[seq + 1] - tok0;
            if (tok0 < 0 || sq < 0 || tok0 + sq > p.total_q) sq = 0;  // as the main kernel: an empty sequence
            elem = (static_cast<int64_t>(tok0 + i) * p.heads + head) * D;
            lse_at = static_cast<int64_t>(head) * p.total_q + tok0 + i;
        } else {
            elem = (bh * p.sq + i) * D;
            lse_at = bh * p.sq + i;
        }
        bool valid = i < sq;
#if ATTN_CHECKED
        {
            // the row of O / dO / the accumulator and its LSE entry are inside their tensors
            const int64_t o_rows = VARLEN ? static_cast<int64_t>(p.total_q) * p.heads : static_cast<int64_t>(p.bh) * p.sq;
            const int64_t lses = VARLEN ? static_cast<int64_t>(p.heads) * p.total_q : static_cast<int64_t>(p.bh) * p.sq;
            if (valid && !(elem >= 0 && elem / D < o_rows && lse_at >= 0 && lse_at < lses)) {
                record_bounds(p, SITE_BWD_CHK_PREP);
                valid = false;
            }
        }
#endif
        float acc = 0.f;
        if (valid) {
            const int64_t off = elem + sub * 8;
            const uint4 a = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.o) + off);
            const uint4 b = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.dout) + off);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 x = unpack2<T>(av[c]), y = unpack2<T>(bv[c]);
                acc = fmaf(x.x, y.x, acc);
                acc = fmaf(x.y, y.y, acc);
            }
            float4 *z = reinterpret_cast<float4 *>(p.dq_acc + off);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
        if (sub == 0) {
            float l2 = INFINITY;
            if (valid) {
                const float l = p.lse[lse_at];
                l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
            }
            p.lse2[r] = l2;
            p.dsum[r] = valid ? acc : 0.f;
        }
    }
}

// dQ = accumulator (fp32, scale already applied) rounded to T, 8 elements
// per thread and step.
template <typename T>
__global__ void __launch_bounds__(256) attn_bwd_dq_convert_kernel(const float *acc, T *dq, int64_t n8)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
        reinterpret_cast<uint4 *>(dq)[i] =
            make_uint4(pack2<T>(a.x, a.y), pack2<T>(a.z, a.w), pack2<T>(b.x, b.y), pack2<T>(b.z, b.w));
    }
}

// ---------------------------------------------------------------- main kernel

template <typename T, bool CAUSAL, int D, bool VARLEN>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdQacc, const BwdParams p)
{
    using C = Cfg<D>;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = idesc(128, C::BM, BF16, false, false);   // S^T, dP^T: [keys x queries]
    constexpr uint32_t IDESC_ACC = idesc(128, C::D, BF16, false, true);   // dV, dK: A from TMEM, B MN-major
    // dQ^T = K^T dS^T [D x queries] (D = 128) or dQ = dS K [queries x D] (D = 64); both operands MN-major
    constexpr uint32_t IDESC_DQ = C::DQ_T ? idesc(C::D, C::BM, BF16, true, true) : idesc(C::BM, C::D, BF16, true, true);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base_addr = smem_addr(smem_raw);
    // The whole budget is used, with no room to realign: the dynamic shared
    // window starts 1 KiB aligned.  Should it not, report and do nothing.
    if ((base_addr & 1023u) != 0u) {
        if (threadIdx.x == 0 && atomicCAS(&p.status[0], 0u, kStatusBounds) == 0u) {
            p.status[1] = blockIdx.x;
            p.status[2] = 0u;
            p.status[3] = SITE_BWD_SMEM_ALIGN;
        }
        return;
    }
    Ctl *ctl = reinterpret_cast<Ctl *>(smem_raw + C::CTL_OFF);
    const uint32_t sLD = base_addr + C::LD_OFF;
    const uint32_t sK = base_addr + C::K_OFF;
    const uint32_t sV = base_addr + C::V_OFF;
    const uint32_t sQ = base_addr + C::Q_OFF;  // stage s: Q at sQ + s*2*TILE, dO at + TILE
    const uint32_t sDS = base_addr + C::DS_OFF;
    const uint32_t sST = base_addr + C::ST_OFF;  // dQ staging (D = 64)
    const float *ld_smem = reinterpret_cast<const float *>(smem_raw + C::LD_OFF);

    auto B = [&](const uint64_t &bar) { return smem_addr(&bar); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    BWD_TRACE_DECL

    if (threadIdx.x == 0) {
        mbar_init(B(ctl->kv_full), 1);
        mbar_init(B(ctl->kv_empty), 1);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(B(ctl->q_full[s]), 1);
            mbar_init(B(ctl->q_empty[s]), 1);
            mbar_init(B(ctl->do_full[s]), 1);
            mbar_init(B(ctl->do_empty[s]), 1);
        }
        mbar_init(B(ctl->s_full), 1);
        mbar_init(B(ctl->dp_full), 1);
        mbar_init(B(ctl->p_full), 8);   // one arrive per softmax warp
        mbar_init(B(ctl->ds_full), 8);
        mbar_init(B(ctl->dq_full), 1);
        mbar_init(B(ctl->dq_empty), 4);  // one arrive per drain warp
        mbar_init(B(ctl->dkv_full), 1);
        mbar_init(B(ctl->dkv_empty), 4);
        mbar_init(B(ctl->mma_done), 1);
        mbar_init(B(ctl->dr_sync), 4);
        for (int s = 0; s < kUnitRing; ++s) {
            mbar_init(B(ctl->unit_full[s]), 1);
            mbar_init(B(ctl->unit_empty[s]), kUnitReaders);
        }
        ctl->abort = 0u;
        fence_barrier_init();
    }
    if (warp == 12) {
        tmem_alloc(smem_addr(&ctl->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 13 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmdQacc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
#if ATTN_CHECKED
    {
        uint32_t dsmem;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dsmem));
        const bool window = static_cast<uint32_t>(C::SMEM_BYTES) <= dsmem;
        const bool tcols = (tmem >> 16) == 0u && (tmem & 0xFFFFu) + C::TMEM_COLS <= 512u;
        const bool setup_ok = (threadIdx.x != 0) || (BWD_IN_BOUNDS(window, SITE_BWD_CHK_SMEM) &&
                                                     BWD_IN_BOUNDS(tcols, SITE_BWD_CHK_TMEM));
        // every thread takes the same decision: no role starts on a bad layout
        if (!__syncthreads_and(setup_ok ? 1 : 0)) goto wind_down;
    }
#endif

    if (warp >= 12) {
        regs_dec<C::REGS_OTHER>();
        if (warp == 13) {
            // ------------------------------------------------------------ producer
            const uint64_t pol = l2_evict_normal();
            uint32_t un_it = 0, q_it = 0;
            bool ok = true;
            for (uint32_t kq = 0; ok; ++kq) {
                // claim the next unit and publish it to the other warps
                const uint32_t slot = kq % kUnitRing;
                ok = warp_wait(B(ctl->unit_empty[slot]), ((kq / kUnitRing) & 1u) ^ 1u, ctl, p, SITE_BWD_UNIT_EMPTY);
                if (!ok) break;
                int u = -1;
                if (lane == 0) {
                    u = atomicAdd(p.counter, 1);
                    if (u >= p.num_units) u = -1;
                    ctl->unit_idx[slot] = u;
                    mbar_arrive(B(ctl->unit_full[slot]));
                }
                u = __shfl_sync(0xffffffffu, u, 0);
                if (u < 0) break;
                if (!BWD_IN_BOUNDS(static_cast<int64_t>(u) < static_cast<int64_t>(p.bh) * p.num_kblk,
                                   SITE_BWD_CHK_UNIT)) {  // before decode reads any offset
                    ok = false;
                    break;
                }
                const Unit un = decode_unit<CAUSAL, VARLEN>(u, p);
                if (!BWD_IN_BOUNDS(unit_ok<VARLEN>(un, p), SITE_BWD_CHK_UNIT)) {
                    ok = false;
                    break;
                }
                if (un.n == 0) continue;
                // TMA coordinates after the 64-column panel: dense maps are
                // [bh][s][D] (row, plane = bh); packed maps are [token][head][D]
                // (row = head, plane = token).
                constexpr bool vl = VARLEN;
                auto qrow = [&](int r) { return vl ? un.head : r; };
                auto qplane = [&](int r) { return vl ? un.q_tok0 + r : un.bh; };
                auto krow = [&](int r) { return vl ? un.head : r; };
                auto kplane = [&](int r) { return vl ? un.k_tok0 + r : un.bh; };
                ok = warp_wait(B(ctl->kv_empty), (un_it & 1u) ^ 1u, ctl, p, SITE_BWD_LOAD_KV_EMPTY);
                if (!ok) break;
                if (!BWD_IN_BOUNDS(un.kb * C::BN < un.sk &&
                                       (vl ? un.k_tok0 + un.kb * C::BN < p.total_k && un.head < p.heads : un.bh < p.bh),
                                   SITE_BWD_CHK_KV_LOAD)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(B(ctl->kv_full), 2 * C::TILE_BYTES);
                    for (int pn = 0; pn < C::NPANEL; ++pn) {
                        tma_load_3d(sK + pn * C::PANEL_BYTES, &tmK, B(ctl->kv_full), pn * 64, krow(un.kb * C::BN),
                                    kplane(un.kb * C::BN), pol);
                        tma_load_3d(sV + pn * C::PANEL_BYTES, &tmV, B(ctl->kv_full), pn * 64, krow(un.kb * C::BN),
                                    kplane(un.kb * C::BN), pol);
                    }
                }
                __syncwarp();
                ++un_it;
                for (int t = 0; t < un.n && ok; ++t) {
                    const uint32_t st = q_it % C::NSTAGE;
                    BWD_TRACE(BEV_LD_WAIT, q_it);
                    ok = warp_wait(B(ctl->q_empty[st]), ((q_it / C::NSTAGE) & 1u) ^ 1u, ctl, p, SITE_BWD_LOAD_Q_EMPTY);
                    BWD_TRACE(BEV_LD_GOT, q_it);
                    if (!ok) break;
                    const int q0 = (un.t0 + t) * C::BM;
                    const uint32_t q_tile = sQ + st * 2 * C::TILE_BYTES;
                    // the tile's Q / dO rows and its LSE / D vector rows (checked once: dO uses the same)
                    if (!BWD_IN_BOUNDS(q0 >= 0 && q0 < un.sq &&
                                           (vl ? un.q_tok0 + q0 < p.total_q && un.head < p.heads : un.bh < p.bh) &&
                                           static_cast<int64_t>(un.bh) * p.sq_pad + q0 + C::BM <=
                                               static_cast<int64_t>(p.bh) * p.sq_pad,
                                       SITE_BWD_CHK_Q_LOAD)) {
                        ok = false;
                        break;
                    }
#if ATTN_CHECKED
                    const bool issue_q = static_cast<int32_t>(q_it) != p.withheld_load;
#else
                    constexpr bool issue_q = true;  // (a compare here costs the d = 64 kernel 1.5%)
#endif
                    if (issue_q && elect_one()) {
                        const uint32_t bar = B(ctl->q_full[st]);
                        mbar_arrive_expect_tx(bar, C::TILE_BYTES + 2 * C::BM * 4);
                        for (int pn = 0; pn < C::NPANEL; ++pn)
                            tma_load_3d(q_tile + pn * C::PANEL_BYTES, &tmQ, bar, pn * 64, qrow(q0), qplane(q0), pol);
                        const size_t row = static_cast<size_t>(un.bh) * p.sq_pad + q0;
                        bulk_load(sLD + st * C::LD_STAGE_BYTES, p.lse2 + row, C::BM * 4, bar);
                        bulk_load(sLD + st * C::LD_STAGE_BYTES + C::BM * 4, p.dsum + row, C::BM * 4, bar);
                    }
                    __syncwarp();
                    // D = 128: dO's slot is also where the previous user of the
                    // stage staged its dQ: wait for that to be read out
                    ok = warp_wait(B(ctl->do_empty[st]), ((q_it / C::NSTAGE) & 1u) ^ 1u, ctl, p, SITE_BWD_LOAD_DO_EMPTY);
                    if (!ok) break;
                    if (elect_one()) {
                        const uint32_t bar = B(ctl->do_full[st]);
                        mbar_arrive_expect_tx(bar, C::TILE_BYTES);
                        for (int pn = 0; pn < C::NPANEL; ++pn)
                            tma_load_3d(q_tile + C::TILE_BYTES + pn * C::PANEL_BYTES, &tmdO, bar, pn * 64, qrow(q0),
                                        qplane(q0), pol);
                    }
                    __syncwarp();
                    ++q_it;
                }
            }
            // Wind-down: let the last copies land before the CTA exits.
            if (un_it > 0) drain_wait(B(ctl->kv_full), (un_it - 1) & 1u, p.timeout_ns);
            for (uint32_t k = (q_it > C::NSTAGE ? q_it - C::NSTAGE : 0u); k < q_it; ++k) {
#if ATTN_CHECKED
                if (static_cast<int32_t>(k) != p.withheld_load)
#endif
                    drain_wait(B(ctl->q_full[k % C::NSTAGE]), (k / C::NSTAGE) & 1u, p.timeout_ns);
                drain_wait(B(ctl->do_full[k % C::NSTAGE]), (k / C::NSTAGE) & 1u, p.timeout_ns);
            }
            __syncwarp();
        } else if (warp == 12) {
            // ------------------------------------------------------------ MMA issuer
            uint32_t un_it = 0, q_it = 0, tile_it = 0;  // tile_it: tiles issued so far (all units)
            bool ok = true;
            const uint32_t dK0 = desc_lo(sK, 16);              // K, K-major (A of S^T)
            const uint32_t dV0 = desc_lo(sV, 16);              // V, K-major (A of dP^T)
            const uint32_t dKt0 = desc_lo(sK, C::PANEL_BYTES); // K MN-major: A of dQ^T (D = 128), B of dQ (D = 64)
            const uint32_t dDS0 = desc_lo(sDS, C::PANEL_BYTES);// dS^T MN-major: B of dQ^T, A of dQ
            auto kmajor_step = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32) >> 4); };
            // [keys x queries] = A(K or V) . B(Q or dO)^T over the head dim
            auto issue_kq = [&](uint32_t a0, uint32_t b0, uint32_t d) {
#pragma unroll
                for (int kk = 0; kk < C::D / 16; ++kk)
                    mma_ss(d, a0 + kmajor_step(kk), b0 + kmajor_step(kk), IDESC_S, kk > 0 ? 1u : 0u);
            };
            // acc += A(TMEM, [keys x queries] 16-bit) . B([queries x D], MN-major) over the tile's queries
            auto issue_acc = [&](uint32_t d, uint32_t a_tm, uint32_t b0, bool accumulate) {
#pragma unroll
                for (int s = 0; s < C::BM / 16; ++s)
                    mma_ts(d, a_tm + 64 * (s >> 2) + 8 * (s & 3), b0 + ((s * 16 * 128) >> 4), IDESC_ACC,
                           (accumulate || s > 0) ? 1u : 0u);
            };
            // dQ^T [D x queries] = K^T . dS^T, or dQ [queries x D] = dS . K, over the unit's keys
            auto issue_dq = [&](uint32_t d) {
#pragma unroll
                for (int s = 0; s < C::BN / 16; ++s) {
                    const uint32_t kt = dKt0 + ((s * 16 * 128) >> 4), ds = dDS0 + ((s * 16 * 128) >> 4);
                    if constexpr (C::DQ_T)
                        mma_ss(d, kt, ds, IDESC_DQ, s > 0 ? 1u : 0u);
                    else
                        mma_ss(d, ds, kt, IDESC_DQ, s > 0 ? 1u : 0u);
                }
            };
            auto q_desc = [&](uint32_t st, bool dout, uint32_t lbo) {
                return desc_lo(sQ + st * 2 * C::TILE_BYTES + (dout ? C::TILE_BYTES : 0), lbo);
            };
            uint32_t dq_pending = 0u;  // 1 when a dQ^T in TMEM has not been drained yet
            for (uint32_t kq = 0; ok; ++kq) {
                int u;
                if (!(ok = next_unit(kq, u, ctl, p))) break;
                if (u < 0) break;
                if (!BWD_IN_BOUNDS(static_cast<int64_t>(u) < static_cast<int64_t>(p.bh) * p.num_kblk,
                                   SITE_BWD_CHK_UNIT)) {  // before decode reads any offset
                    ok = false;
                    break;
                }
                const Unit un = decode_unit<CAUSAL, VARLEN>(u, p);
                if (!BWD_IN_BOUNDS(unit_ok<VARLEN>(un, p), SITE_BWD_CHK_UNIT)) {
                    ok = false;
                    break;
                }
                if (un.n == 0) continue;
                if (!(ok = warp_wait(B(ctl->kv_full), un_it & 1u, ctl, p, SITE_BWD_MMA_KV_FULL))) break;
                if constexpr (VARLEN) {  // keys past the sequence's end
                    zero_rows_from<C::NPANEL>(sK, un.sk - un.kb * C::BN);
                    zero_rows_from<C::NPANEL>(sV, un.sk - un.kb * C::BN);
                }
                if (!(ok = warp_wait(B(ctl->q_full[q_it % C::NSTAGE]), (q_it / C::NSTAGE) & 1u, ctl, p, SITE_BWD_MMA_Q_FULL))) break;
                if constexpr (VARLEN)  // queries past the sequence's end
                    zero_rows_from<C::NPANEL>(sQ + (q_it % C::NSTAGE) * 2 * C::TILE_BYTES, un.sq - un.t0 * C::BM);
                tc_fence_after();
                if (elect_one()) {
                    issue_kq(dK0, q_desc(q_it % C::NSTAGE, false, 16), tmem + C::TM_S);
                    tc_commit(B(ctl->s_full));
                }
                __syncwarp();
                if (C::DQ_T && dq_pending) {  // the previous unit's last dQ^T still occupies the dP^T columns
                    if (!(ok = warp_wait(B(ctl->dq_empty), (tile_it - 1) & 1u, ctl, p, SITE_BWD_MMA_DQ_EMPTY))) break;
                    dq_pending = 0u;
                }
                if (!(ok = warp_wait(B(ctl->do_full[q_it % C::NSTAGE]), (q_it / C::NSTAGE) & 1u, ctl, p, SITE_BWD_MMA_DO_FULL))) break;
                if constexpr (VARLEN)
                    zero_rows_from<C::NPANEL>(sQ + (q_it % C::NSTAGE) * 2 * C::TILE_BYTES + C::TILE_BYTES, un.sq - un.t0 * C::BM);
                tc_fence_after();
                if (elect_one()) {
                    issue_kq(dV0, q_desc(q_it % C::NSTAGE, true, 16), tmem + C::TM_DP);
                    tc_commit(B(ctl->dp_full));
                }
                __syncwarp();
                for (int t = 0; t < un.n && ok; ++t) {
                    const uint32_t st = q_it % C::NSTAGE;
                    // dV += P^T dO
                    BWD_TRACE(BEV_MMA_WAIT_P, tile_it);
                    if (!(ok = warp_wait(B(ctl->p_full), tile_it & 1u, ctl, p, SITE_BWD_MMA_P_FULL))) break;
                    BWD_TRACE(BEV_MMA_GOT_P, tile_it);
                    if (t == 0 && un_it > 0 &&
                        !(ok = warp_wait(B(ctl->dkv_empty), (un_it - 1) & 1u, ctl, p, SITE_BWD_MMA_DKV_EMPTY)))
                        break;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_acc(tmem + C::TM_DV, tmem + C::TM_S, q_desc(st, true, C::PANEL_BYTES), t > 0);
                        // D = 64: dV is the last reader of the tile's dO (its dQ is
                        // staged elsewhere), so the slot goes back from here
                        if constexpr (!C::DQ_T) tc_commit(B(ctl->do_empty[st]));
                    }
                    __syncwarp();
                    BWD_TRACE(BEV_MMA_ISSUED_DV, tile_it);
                    // S^T of the next tile (its P^T columns were just consumed, in order)
                    const bool more = t + 1 < un.n;
                    if (more) {
                        BWD_TRACE(BEV_MMA_WAIT_Q, tile_it);
                        if (!(ok = warp_wait(B(ctl->q_full[(q_it + 1) % C::NSTAGE]), ((q_it + 1) / C::NSTAGE) & 1u, ctl, p,
                                             SITE_BWD_MMA_Q_FULL)))
                            break;
                        BWD_TRACE(BEV_MMA_GOT_Q, tile_it);
                        if constexpr (VARLEN)
                            zero_rows_from<C::NPANEL>(sQ + ((q_it + 1) % C::NSTAGE) * 2 * C::TILE_BYTES,
                                                      un.sq - (un.t0 + t + 1) * C::BM);
                        tc_fence_after();
                        if (elect_one()) {
                            issue_kq(dK0, q_desc((q_it + 1) % C::NSTAGE, false, 16), tmem + C::TM_S);
                            tc_commit(B(ctl->s_full));
                        }
                        __syncwarp();
                    }
                    // dK += dS^T Q, then dQ^T = K^T dS^T into the dP^T columns
                    BWD_TRACE(BEV_MMA_WAIT_DS, tile_it);
                    if (!(ok = warp_wait(B(ctl->ds_full), tile_it & 1u, ctl, p, SITE_BWD_MMA_DS_FULL))) break;
                    BWD_TRACE(BEV_MMA_GOT_DS, tile_it);
                    if (!C::DQ_T && dq_pending) {  // D = 64: the previous dQ has left its columns
                        if (!(ok = warp_wait(B(ctl->dq_empty), (tile_it - 1) & 1u, ctl, p, SITE_BWD_MMA_DQ_EMPTY)))
                            break;
                        dq_pending = 0u;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        issue_acc(tmem + C::TM_DK, tmem + C::TM_DP, q_desc(st, false, C::PANEL_BYTES), t > 0);
                        issue_dq(tmem + C::TM_DQ);
                        tc_commit(B(ctl->dq_full));
                        tc_commit(B(ctl->q_empty[st]));
                        if (!more) {
                            tc_commit(B(ctl->kv_empty));
                            tc_commit(B(ctl->dkv_full));
                        }
                    }
                    __syncwarp();
                    BWD_TRACE(BEV_MMA_ISSUED_DKDQ, tile_it);
                    dq_pending = 1u;
                    ++tile_it;
                    ++q_it;
                    // dP^T of the next tile (D = 128: once dQ^T has been drained)
                    if (more) {
                        if constexpr (C::DQ_T) {
                            BWD_TRACE(BEV_MMA_WAIT_DQE, tile_it);
                            if (!(ok = warp_wait(B(ctl->dq_empty), (tile_it - 1) & 1u, ctl, p, SITE_BWD_MMA_DQ_EMPTY)))
                                break;
                            BWD_TRACE(BEV_MMA_GOT_DQE, tile_it);
                            dq_pending = 0u;
                        }
                        if (!(ok = warp_wait(B(ctl->do_full[q_it % C::NSTAGE]), (q_it / C::NSTAGE) & 1u, ctl, p,
                                             SITE_BWD_MMA_DO_FULL)))
                            break;
                        if constexpr (VARLEN)
                            zero_rows_from<C::NPANEL>(sQ + (q_it % C::NSTAGE) * 2 * C::TILE_BYTES + C::TILE_BYTES,
                                                      un.sq - (un.t0 + t + 1) * C::BM);
                        tc_fence_after();
                        if (elect_one()) {
                            issue_kq(dV0, q_desc(q_it % C::NSTAGE, true, 16), tmem + C::TM_DP);
                            tc_commit(B(ctl->dp_full));
                        }
                        __syncwarp();
                    }
                }
                ++un_it;
            }
            // Every MMA issued must complete before tensor memory is freed.
            if (elect_one()) tc_commit(B(ctl->mma_done));
            __syncwarp();
            drain_wait(B(ctl->mma_done), 0u, p.timeout_ns);
            __syncwarp();
        }
    } else if (warp >= 8) {
        if constexpr (C::REGS_DRAIN > 128)
            regs_inc<C::REGS_DRAIN>();
        else
            regs_dec<C::REGS_DRAIN>();
        // ---------------------------------------------------------------- dQ drain + dK/dV epilogue
        // Per tile the dQ product comes out of tensor memory, which is
        // released at once, is staged as fp32 rows in shared memory and is
        // added into the accumulator by the copy engine (TMA reduce-add).
        //   D = 128: dQ^T, this thread holds head-dim column dcol for the 128
        //            queries; staged as [64 queries][128] in the tile's dO
        //            slot (free: dP^T and dV have read it), two halves.
        //   D = 64:  dQ, this thread holds query row dcol's 64 columns;
        //            staged in a buffer of its own as two [128][32] boxes
        //            with the 128-byte swizzle (conflict-free row writes).
        // D = 128: the dO slot goes back to the producer once the reduces
        // have read the staging (D = 64: the MMA warp returns it after dV).
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const int dcol = quad * 32 + lane;
        const bool issuer = (warp == 8 && lane == 0);
        uint32_t tile_it = 0, un_it = 0, q_it = 0, sync_ph = 0;
        bool ok = true;
        // the four drain warps meet (bounded, like every other wait)
        auto drain_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(B(ctl->dr_sync));
            const bool r = warp_wait(B(ctl->dr_sync), sync_ph, ctl, p, SITE_BWD_DRAIN_SYNC);
            sync_ph ^= 1u;
            return r;
        };
        for (uint32_t kq = 0; ok; ++kq) {
            int u;
            if (!(ok = next_unit(kq, u, ctl, p))) break;
            if (u < 0) break;
            if (!BWD_IN_BOUNDS(static_cast<int64_t>(u) < static_cast<int64_t>(p.bh) * p.num_kblk,
                               SITE_BWD_CHK_UNIT)) {  // before decode reads any offset
                ok = false;
                break;
            }
            const Unit un = decode_unit<CAUSAL, VARLEN>(u, p);
            if (!BWD_IN_BOUNDS(unit_ok<VARLEN>(un, p), SITE_BWD_CHK_UNIT)) {
                ok = false;
                break;
            }
            constexpr bool vl = VARLEN;
            auto key_offset = [&](int key) {  // element offset of key row `key` of the unit's sequence in dK / dV
                return vl ? (static_cast<size_t>(un.k_tok0 + key) * p.heads + un.head) * C::D
                          : (static_cast<size_t>(un.bh) * p.sk + key) * C::D;
            };
            // checked builds: the row is one of dK's / dV's rows
            auto dkv_row_ok = [&](int key) {
                const size_t rows = vl ? static_cast<size_t>(p.total_k) * p.heads : static_cast<size_t>(p.bh) * p.sk;
                return key >= 0 && key_offset(key) / C::D < rows;
            };
            if (un.n == 0) {
                if (un.zero) {  // a sequence with keys but no query: its dK and dV are 0
                    const int key = un.kb * C::BN + quad * 32 + lane;
#if ATTN_CHECKED
                    if (!__all_sync(0xffffffffu, BWD_IN_BOUNDS(key >= un.sk || dkv_row_ok(key), SITE_BWD_CHK_DKV_ROW))) {
                        ok = false;
                        break;
                    }
#endif
                    if (key < un.sk)
#pragma unroll
                        for (int which = 0; which < 2; ++which) {
                            uint4 *out = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(which ? p.dk : p.dv) + key_offset(key));
                            for (int c = 0; c < C::D / 8; ++c) out[c] = make_uint4(0u, 0u, 0u, 0u);
                        }
                }
                continue;
            }
            // reduce-add coordinates (dense [bh][sq][D]; packed [token][head][D])
            auto rrow = [&](int r) { return vl ? un.head : r; };
            auto rplane = [&](int r) { return vl ? un.q_tok0 + r : un.bh; };
            for (int t = 0; t < un.n && ok; ++t) {
                BWD_TRACE(BEV_DR_WAIT, tile_it);
                if (!(ok = warp_wait(B(ctl->dq_full), tile_it & 1u, ctl, p, SITE_BWD_DRAIN_DQ_FULL))) break;
                BWD_TRACE(BEV_DR_GOT, tile_it);
                ++tile_it;
                tc_fence_after();
                const uint32_t st = q_it % C::NSTAGE;
                const int q0 = (un.t0 + t) * C::BM;
                // the reduce-adds start at a row of the tile's sequence (rows past the
                // tensor are dropped by the copy engine)
                if (!BWD_IN_BOUNDS(q0 >= 0 && q0 < un.sq &&
                                       (vl ? un.q_tok0 + q0 < p.total_q && un.head < p.heads : un.bh < p.bh),
                                   SITE_BWD_CHK_DQ_RED)) {
                    ok = false;
                    break;
                }
                if constexpr (C::DQ_T) {
                    uint32_t v[128];
                    tmem_ld128_wait(tmem + lane_off + C::TM_DP, v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B(ctl->dq_empty));
                    BWD_TRACE(BEV_DR_RELEASED, tile_it);
                    const uint32_t stage_buf = sQ + st * 2 * C::TILE_BYTES + C::TILE_BYTES;  // the dO slot
#pragma unroll
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (h == 1 && !(ok = drain_sync())) break;  // the first reduce has read the slot
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            st_shared_f32(stage_buf + (c * C::D + dcol) * 4, __uint_as_float(v[64 * h + c]));
                        fence_proxy_async_smem();
                        if (!(ok = drain_sync())) break;
                        if (issuer) {
#pragma unroll
                            for (int r0 = 0; r0 < 64; r0 += C::RED_ROWS)
                                tma_reduce_add_3d(&tmdQacc, stage_buf + r0 * C::D * 4, 0, rrow(q0 + 64 * h + r0),
                                                  rplane(q0 + 64 * h + r0));
                            bulk_commit_group();
                            bulk_wait_read_all();
                        }
                    }
                } else {
                    uint32_t v[64];
                    tmem_ld64_wait(tmem + lane_off + C::TM_DQ, v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B(ctl->dq_empty));
                    BWD_TRACE(BEV_DR_RELEASED, tile_it);
                    // the previous tile's reduces have read the staging
                    if (!(ok = drain_sync())) break;
#pragma unroll
                    for (int box = 0; box < 2; ++box)
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t chunk = static_cast<uint32_t>(c ^ (dcol & 7));
                            st_shared_v4(sST + box * (C::BM * 128) + dcol * 128 + chunk * 16, v[32 * box + 4 * c],
                                         v[32 * box + 4 * c + 1], v[32 * box + 4 * c + 2], v[32 * box + 4 * c + 3]);
                        }
                    fence_proxy_async_smem();
                    if (!(ok = drain_sync())) break;
                    if (issuer) {
                        tma_reduce_add_3d(&tmdQacc, sST, 0, rrow(q0), rplane(q0));
                        tma_reduce_add_3d(&tmdQacc, sST + C::BM * 128, 32, rrow(q0), rplane(q0));
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                }
                if (!ok) break;
                if (C::DQ_T && issuer) mbar_arrive(B(ctl->do_empty[st]));  // the staging in the dO slot is read
                ++q_it;
                BWD_TRACE(BEV_DR_DONE, tile_it);
            }
            if (!ok) break;
            // dK, dV of the unit: this thread's key row, D columns each
            BWD_TRACE(BEV_DR_DKV_WAIT, un_it);
            if (!(ok = warp_wait(B(ctl->dkv_full), un_it & 1u, ctl, p, SITE_BWD_DRAIN_DKV_FULL))) break;
            BWD_TRACE(BEV_DR_DKV_GOT, un_it);
            ++un_it;
            tc_fence_after();
            const int key = un.kb * C::BN + quad * 32 + lane;
            const bool valid = key < un.sk;
#if ATTN_CHECKED
            if (!__all_sync(0xffffffffu, BWD_IN_BOUNDS(!valid || dkv_row_ok(key), SITE_BWD_CHK_DKV_ROW))) {
                ok = false;
                break;
            }
#endif
            const size_t roff = key_offset(valid ? key : 0);
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                uint4 *out = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(which ? p.dk : p.dv) + roff);
                const uint32_t src = tmem + lane_off + (which ? C::TM_DK : C::TM_DV);
#pragma unroll
                for (int ch = 0; ch < C::D / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32_wait(src + 32 * ch, v);
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = pack2<T>(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
                    if (valid) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            out[ch * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B(ctl->dkv_empty));
            BWD_TRACE(BEV_DR_DKV_DONE, un_it);
        }
    } else {
        regs_inc<C::REGS_SOFTMAX>();
        // ---------------------------------------------------------------- softmax groups
        const int g = warp >> 2;     // query half of the tile: columns 64g .. 64g+63
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // key row within the unit's block
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::TM_S + 64 * g;
        const uint32_t tDP = tmem + lane_off + C::TM_DP + 64 * g;
        const float sl2e = p.sl2e, scale = p.scale;
        uint32_t tile_it = 0, q_it = 0;
        bool ok = true;
        for (uint32_t kq = 0; ok; ++kq) {
            int u;
            if (!(ok = next_unit(kq, u, ctl, p))) break;
            if (u < 0) break;
            if (!BWD_IN_BOUNDS(static_cast<int64_t>(u) < static_cast<int64_t>(p.bh) * p.num_kblk,
                               SITE_BWD_CHK_UNIT)) {  // before decode reads any offset
                ok = false;
                break;
            }
            const Unit un = decode_unit<CAUSAL, VARLEN>(u, p);
            if (!BWD_IN_BOUNDS(unit_ok<VARLEN>(un, p), SITE_BWD_CHK_UNIT)) {
                ok = false;
                break;
            }
            if (un.n == 0) continue;
            const int key = un.kb * C::BN + r;
            const int sk_ = VARLEN ? un.sk : p.sk, sq_ = VARLEN ? un.sq : p.sq;
            const bool row_ok = key < sk_;
            const int diag = key - (sk_ - sq_);  // the first query this key row sees
            for (int t = 0; t < un.n && ok; ++t) {
                const uint32_t st = q_it % C::NSTAGE;
                // the tile's LSE / D vectors arrive with Q and dO
                if (!(ok = warp_wait(B(ctl->q_full[st]), (q_it / C::NSTAGE) & 1u, ctl, p, SITE_BWD_SM_S_FULL))) break;
                BWD_TRACE(BEV_SM_WAIT_S, tile_it);
                if (!(ok = warp_wait(B(ctl->s_full), tile_it & 1u, ctl, p, SITE_BWD_SM_S_FULL))) break;
                BWD_TRACE(BEV_SM_GOT_S, tile_it);
                tc_fence_after();
                const int q0 = (un.t0 + t) * C::BM + 64 * g;  // first query of this thread's columns
                // columns c < lim are masked for this key row (key j sees query i iff i >= j - (sk - sq))
                int lim = CAUSAL ? diag - q0 : 0;
                if (!row_ok) lim = 64;
                const bool masked = __any_sync(0xffffffffu, lim > 0);
                const float *l2 = ld_smem + st * (C::LD_STAGE_BYTES / 4) + 64 * g;
                const float *dsv = l2 + C::BM;
                // P^T of this thread's 64 columns, rounded to T, two per word: the
                // dV product and dS both use these values.
                uint32_t pk[32];
                {
                    uint32_t sr[64];
                    tmem_ld64_wait(tS, sr);
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float4 lv = *reinterpret_cast<const float4 *>(l2 + c);
                        const float lvv[4] = {lv.x, lv.y, lv.z, lv.w};
                        float x[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x[e] = ex2_approx(fmaf(__uint_as_float(sr[c + e]), sl2e, -lvv[e]));
                            if (masked && (c + e) < lim) x[e] = 0.f;
                        }
                        pk[c / 2] = pack2<T>(x[0], x[1]);
                        pk[c / 2 + 1] = pack2<T>(x[2], x[3]);
                    }
                }
                tmem_st16(tS, *reinterpret_cast<const uint32_t(*)[16]>(pk));
                tmem_st16(tS + 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(ctl->p_full));
                BWD_TRACE(BEV_SM_P_DONE, tile_it);
                // dS^T = scale * P^T (dP^T - D)
                BWD_TRACE(BEV_SM_WAIT_DP, tile_it);
                if (!(ok = warp_wait(B(ctl->dp_full), tile_it & 1u, ctl, p, SITE_BWD_SM_DP_FULL))) break;
                BWD_TRACE(BEV_SM_GOT_DP, tile_it);
                tc_fence_after();
                {
                    uint32_t dr[64];
                    tmem_ld64_wait(tDP, dr);
                    // HALVES stores each half of 32 queries as soon as it is packed
                    // (fewer live registers: the varlen instances need that)
                    constexpr int HALVES = VARLEN ? 2 : 1;
                    constexpr int W = 32 / HALVES;  // packed words per pass
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh) {
                        uint32_t dk[W];
#pragma unroll
                        for (int c = 0; c < 2 * W; c += 4) {
                            const int cc = 2 * W * hh + c;
                            const float4 dv4 = *reinterpret_cast<const float4 *>(dsv + cc);
                            const float2 p01 = unpack2<T>(pk[cc / 2]), p23 = unpack2<T>(pk[cc / 2 + 1]);
                            const float pv[4] = {p01.x, p01.y, p23.x, p23.y};
                            const float dvv[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
                            float ds[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) ds[e] = scale * pv[e] * (__uint_as_float(dr[cc + e]) - dvv[e]);
                            dk[c / 2] = pack2<T>(ds[0], ds[1]);
                            dk[c / 2 + 1] = pack2<T>(ds[2], ds[3]);
                        }
#pragma unroll
                        for (int q16 = 0; q16 < W / 16; ++q16)
                            tmem_st16(tDP + W * hh + 16 * q16, *reinterpret_cast<const uint32_t(*)[16]>(dk + 16 * q16));
                        // shared copy for dQ: MN-major operand, panel g (queries 64g..),
                        // row r, 16-byte chunks of the row, 128-byte swizzle
#pragma unroll
                        for (int k8 = 0; k8 < W / 4; ++k8) {
                            const uint32_t chunk = static_cast<uint32_t>((W / 4 * hh + k8) ^ (r & 7));
                            st_shared_v4(sDS + g * C::PANEL_BYTES + r * 128 + chunk * 16, dk[4 * k8], dk[4 * k8 + 1],
                                         dk[4 * k8 + 2], dk[4 * k8 + 3]);
                        }
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(ctl->ds_full));
                BWD_TRACE(BEV_SM_DS_DONE, tile_it);
                ++tile_it;
                ++q_it;
            }
        }
    }

#if ATTN_CHECKED
wind_down:
#endif
    if (warp == 8 && lane == 0) bulk_wait_all();  // the dQ reduces have landed
    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace bwd
}  // namespace attn
