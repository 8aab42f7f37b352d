// Fused attention forward for sm_103a (GB300): TMA + mbarrier ring +
// tcgen05.mma into tensor memory, online exp2 softmax with lazy rescaling.
//
// What is computed: O = softmax(scale * Q K^T [+ causal mask]) V and the
// natural log-sum-exp per row ("flash-attn 实现 prefill 阶段", 问题分析:
// attention formula over [b, h, s, d]; flash-attention-minimal
// forward_kernel: scale after the dot product, online recurrence with a
// running row max m and row sum l, O rescaled when m changes).
//
// How (one persistent CTA per SM, 12 warps):
//   warps 0-3   softmax group 0  -- Q tile 0 (rows 0..127 of the unit)
//   warps 4-7   softmax group 1  -- Q tile 1 (rows 128..255 of the unit)
//   warp  8     MMA issuer (one thread) + tensor-memory owner
//   warp  9     TMA producer (one thread)
//   warps 10-11 no work (they complete warpgroup 2, whose registers are
//               handed to the softmax groups: 216 per softmax thread, 72
//               for the others; 256*216 + 128*72 = 384*168 at launch,
//               and 216 + 216 + 72 = 3*168 on each SM sub-partition)
// Epilogue: each softmax warp writes its 32 finished rows (O / row sum,
// rounded) into its own 4 KiB shared-memory slice, 64 columns at a time,
// and its lane 0 has the copy engine store the slice to global memory
// (whole 128-byte rows instead of one 16-byte piece of 32 rows per store).
// A work unit is (batch*head, 256-row block).  Per unit the producer loads
// the two Q tiles once and streams K_j, V_j tiles (128 keys each) through an
// NSLOT-deep shared-memory ring.  The MMA thread computes S_t = Q_t K_j^T
// into tensor memory (128 lanes x 128 fp32 columns per tile), waits for the
// softmax group to overwrite S_t in place with P_t (rounded to the input
// type, two per 32-bit column), then issues O_t += P_t V_j with P read from
// tensor memory.  The two Q tiles alternate so that one group's softmax runs
// while the tensor core works on the other tile.  Each softmax thread owns
// one row (one tensor-memory lane): no cross-thread reductions.
//
// Softmax (per row, log2 domain): x = s * scale * log2(e); m_new =
// max(m, rowmax x).  O and the row sums are rescaled by 2^(m - m_new) only
// when m_new - m > 8 for some row of the warp (lazy rescale; the stale max
// cancels exactly between O and the sums, and p = 2^(x - m) stays <= 256).
// Two row sums are kept: l of the fp32 p (LSE = (m + log2 l) * ln 2) and lr
// of p as rounded to the input type for the P.V product; O is divided by lr
// so that the weights applied to V sum to one (the rounding of a dominant p
// then cancels instead of showing up in O).
//
// Every wait is bounded: when a wait runs out the kernel records where in a
// status word, tells the other warps, waits for its own copies and MMAs,
// frees tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <type_traits>

#include "ptx.cuh"

namespace attn {

// Checked build: with ATTN_CHECKED=1 every computed load/store coordinate,
// global output offset, decoded unit, tensor-memory base and shared-memory
// window is compared with its bounds (see in_bounds).  Off by default.
#ifndef ATTN_CHECKED
#define ATTN_CHECKED 0
#endif

// Build options of the producer (see the producer warp).
#ifndef ATTN_KV_PREFETCH
#define ATTN_KV_PREFETCH 0
#endif
#ifndef ATTN_Q_EVICT_FIRST
#define ATTN_Q_EVICT_FIRST 0
#endif

struct FwdParams {
    void *o;               // [bh, sq, D] of T
    float *lse;            // [bh, sq] or nullptr
    uint32_t *status;      // 4 words: code, block, warp, site
    int32_t bh;            // b * h
    int32_t sq, sk;
    int32_t num_mblk;      // ceil(sq / 256)
    int32_t num_units;     // bh * num_mblk
    float sl2e;            // scale * log2(e) (e4m3: times the Q and K descales)
    float o_scale;         // multiplier of O (e4m3: the V descale; else 1)
    uint64_t timeout_ns;   // bound of every wait
    int32_t withheld_load; // K/V load index never issued (watchdog self-test), -1 = none
    // Split-KV: the K/V tiles each (bh, row block) sees are cut into
    // num_splits near-equal ranges.  With num_splits > 1 the kernel writes, per
    // split, O normalised by its own rounded-P sum (fp32, o_part
    // [split][bh][sq][D]) and two natural log-sum-exps (lse_part
    // [split][bh][sq][2]: of the fp32 p, and of p as rounded); a combine
    // kernel merges the splits.  num_splits == 1: o / lse written directly.
    int32_t num_splits;
    float *o_part;
    float *lse_part;
    // Varlen (packed sequences): cu_q / cu_k are the batch+1 cumulative
    // sequence offsets (device int32); Q, O are [total_q, heads, D], K, V
    // [total_k, heads, D], LSE [heads, total_q].  bh is then batch * heads,
    // sq / sk the maximum lengths.  nullptr: the dense [b, h, s, D] layout.
    const int32_t *cu_q;
    const int32_t *cu_k;
    int32_t heads;
    int32_t total_q, total_k;
    // KV cache (dense layout): sk is the capacity of the cache and batch
    // element b has min(clamp(seqlens_k[b], 0, sk) + seqlens_add, sk) valid
    // keys (device int32 [b]; bh = b * heads).  nullptr: all sk keys.
    const int32_t *seqlens_k = nullptr;
    int32_t seqlens_add = 0;
    // Paged KV cache: K and V are a pool of pages [num_pages][page_size]
    // [heads][D] (read through packed maps, like varlen), and logical key r
    // of batch element b lives in page block_table[b * pages_per_seq +
    // r / page_size], row r % page_size.  page_size is a multiple of the
    // 128-key tile, so no tile straddles two pages.  nullptr: not paged.
    const int32_t *block_table = nullptr;
    int32_t pages_per_seq = 0;
    int32_t page_size = 0;
    int32_t num_pages = 0;
    // Dynamic schedule: one slot of kSchedWords words {next unit to hand
    // out, CTAs finished, owner generation, unused}, all zero when the slot is
    // free.  Each CTA first claims the slot for this launch's generation
    // `sched_gen` (owner 0 -> gen); a CTA that finds another generation there
    // records a collision in the status word and takes no unit.  The last
    // CTA to finish sets the slot back to zero.  nullptr: every CTA takes a
    // fixed share of the units (unit_at).
    int32_t *sched = nullptr;
    uint32_t sched_gen = 0;
    // Causal unit order: > 0 orders the units in groups of `group` head
    // planes, heaviest row block first within each group, so that the K/V
    // the units in flight stream stay in L2; 0 orders all heads heaviest
    // first.
    int32_t group = 0;
#ifdef ATTN_TRACE_ENABLE
    unsigned long long *trace;  // per-warp event records (timeline builds only)
#endif
};

// Timeline event codes (see the hooks below).
enum : uint32_t {
    EV_SM_WAIT_S = 1, EV_SM_GOT_S, EV_SM_LD, EV_SM_MAX, EV_SM_RESCALE, EV_SM_EXP, EV_SM_ARRIVE,
    EV_SM_EPI_WAIT, EV_SM_EPI_GOT, EV_SM_EPI_DONE,
    EV_MMA_WAIT_Q = 20, EV_MMA_GOT_Q, EV_MMA_WAIT_KV, EV_MMA_GOT_KV, EV_MMA_WAIT_P, EV_MMA_GOT_P, EV_MMA_ISSUED,
    EV_LD_WAIT = 40, EV_LD_GOT,
    EV_K_ENTRY = 60, EV_K_READY, EV_K_EXIT,
    EV_SM_EPI_WRITTEN = 81,
    EV_REGS = 90, EV_UNIT, EV_DECODED, EV_Q_ISSUED,
};

// Pipeline timeline hooks.  Compiled out unless ATTN_TRACE_ENABLE is defined
// (a separate diagnostic build that records {clock, event, arg} per warp).
#ifdef ATTN_TRACE_ENABLE
#define ATTN_TRACE_DECL uint32_t attn_trace_n = 0;
#define ATTN_TRACE(ev, arg) attn_trace_record(p, attn_trace_n, (ev), (arg))
__device__ __forceinline__ void attn_trace_record(const FwdParams &p, uint32_t &n, uint32_t ev, uint32_t arg)
{
    constexpr uint32_t kCtas = 4, kWarps = 12, kEvents = 16384;
#ifdef ATTN_TRACE_SPARSE
    // sparse timelines: only the events that bound a softmax tile, the MMA
    // warp's waits and the producer's slot waits, so that the hooks disturb
    // the pipeline less
    if (ev != EV_SM_GOT_S && ev != EV_SM_EXP && ev != EV_SM_ARRIVE && ev != EV_LD_WAIT && ev != EV_LD_GOT &&
        (ev < EV_MMA_WAIT_KV || ev > EV_MMA_GOT_P))
        return;
#endif
    if (p.trace == nullptr || blockIdx.x >= kCtas || (threadIdx.x & 31) != 0 || n >= kEvents) return;
    const uint32_t w = threadIdx.x >> 5;
    unsigned long long *rec = p.trace + 2ull * ((blockIdx.x * kWarps + w) * kEvents + n);
    rec[0] = clock64();
    rec[1] = (static_cast<unsigned long long>(ev) << 32) | arg;
    ++n;
}
#else
#define ATTN_TRACE_DECL
#define ATTN_TRACE(ev, arg) ((void)0)
#endif


// Watchdog sites (recorded in status[3]).
enum : uint32_t {
    SITE_LOAD_Q_EMPTY = 1,
    SITE_LOAD_KV_EMPTY = 2,
    SITE_MMA_Q_FULL = 3,
    SITE_MMA_KV_FULL = 4,
    SITE_MMA_P_FULL = 5,
    SITE_SOFTMAX_S_FULL = 6,
    SITE_SOFTMAX_O_FULL = 7,
    SITE_DRAIN = 8,
    SITE_UNIT_FULL = 9,
    SITE_UNIT_EMPTY = 10,
    SITE_SCHED_SLOT = 11,
};

// Status codes (status[0]): a wait that ran out, and a dynamic-schedule
// slot that another launch still held.
enum : uint32_t {
    STATUS_TIMEOUT = 1,
    STATUS_SCHED_COLLISION = 2,
    STATUS_BOUNDS = 3,  // checked builds: a computed index outside its bounds
};

// Bounds-check sites of the checked build (recorded in status[3]).
enum : uint32_t {
    SITE_CHK_SMEM = 20,     // dynamic shared memory window too small for the layout
    SITE_CHK_TMEM = 21,     // tensor-memory allocation not the expected 512 columns at lane 0
    SITE_CHK_UNIT = 22,     // decoded unit outside the problem
    SITE_CHK_Q_LOAD = 23,   // Q copy coordinates
    SITE_CHK_KV_LOAD = 24,  // K/V copy coordinates (page lookup included)
    SITE_CHK_O_TILE = 25,   // O copy-engine store coordinates
    SITE_CHK_O_ROW = 26,    // O / LSE row written by a thread
    SITE_CHK_O_PART = 27,   // split partial row
};

// Input element types: fp16, bf16 (16-bit, kind::f16 MMAs, P two per
// tensor-memory column) and e4m3 (8-bit, kind::f8f6f4 MMAs, P four per
// column, output in bf16).  SHIFT is the log2 offset of the exp reference
// and TAU the lazy-rescale threshold (both log2 units).  For e4m3 the
// reference sits 8 below the row max, so P spans [0, 256] and uses the
// 8-bit range instead of flushing small values ("05 · kernel 工程与四代演化"
// 4.4); TAU = 0.5 keeps P <= 2^8.5 < 448, the e4m3 maximum.
template <typename T>
struct Elem;
template <>
struct Elem<__half> {
    static constexpr int BYTES = 2;
    static constexpr bool FP8 = false;
    static constexpr bool BF16 = false;
    static constexpr float SHIFT = 0.f, TAU = 8.f;
    using Out = __half;
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int BYTES = 2;
    static constexpr bool FP8 = false;
    static constexpr bool BF16 = true;
    static constexpr float SHIFT = 0.f, TAU = 8.f;
    using Out = __nv_bfloat16;
};
template <>
struct Elem<__nv_fp8_e4m3> {
    static constexpr int BYTES = 1;
    static constexpr bool FP8 = true;
    static constexpr bool BF16 = false;  // format code 0 = e4m3 in kind::f8f6f4
    static constexpr float SHIFT = 8.f, TAU = 0.5f;
    using Out = __nv_bfloat16;
};

template <int D_, int EB = 2>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int BM = 128;                 // rows per Q tile = TMEM lanes
    static constexpr int QT = 2;                   // Q tiles per unit
    static constexpr int UNIT_ROWS = BM * QT;      // 256
    static constexpr int BN = 128;                 // keys per K/V tile
    // A panel is 128 rows of ROW_BYTES with the swizzle of that width: 128
    // bytes, or 64 bytes when a whole row is shorter (8-bit, head dim 64).
    static constexpr int ROW_BYTES = (D * EB < 128) ? D * EB : 128;
    static constexpr int PANEL_ELEMS = ROW_BYTES / EB;
    static constexpr int NPANEL = D * EB / ROW_BYTES;
    static constexpr int PANEL_BYTES = 128 * ROW_BYTES;
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;  // one Q, K or V tile
    static constexpr int NSLOT = (TILE_BYTES == 2 * PANEL_BYTES) ? 4 : 8;
    static constexpr uint32_t DESC_HI = ROW_BYTES == 128 ? kDescHi : kDescHi64;
    static constexpr int QK_STEPS = D * EB / 32;   // 32-byte k-steps of S = Q K^T
    static constexpr int KSTEPS_PER_ROW = ROW_BYTES / 32;
    static constexpr int PV_KEYS = 32 / EB;        // keys per k-step of O += P V
    static constexpr int PV_STEPS = BN / PV_KEYS;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int Q_OFF = CTL_BYTES;
    static constexpr int KV_OFF = Q_OFF + QT * TILE_BYTES;
    // O staging: a 32-row x 128-byte slice (64 columns of the 16-bit
    // output) per softmax warp, written by the warp and stored to global
    // memory by the copy engine, O_NPANEL times per tile.
    static constexpr int O_PANEL_COLS = 64;
    static constexpr int O_NPANEL = D / O_PANEL_COLS;
    static constexpr int OST_WARP_BYTES = 32 * 128;
    static constexpr int OST_BYTES = 4 * OST_WARP_BYTES;  // per softmax group
    static constexpr int OST_OFF = KV_OFF + NSLOT * TILE_BYTES;
    // Head dim 64, 16-bit: tensor memory has room for the row sums of P as
    // rounded, so the tensor core computes them and the softmax does not.
    // The P.V product is N = 64 + 16 wide: its B operand is V's 64 columns
    // followed by a block of ones (16 rows x 128 bytes of shared memory,
    // reached through the descriptor's leading byte offset), so columns
    // 64..79 of the accumulator hold the rounded row sums, rescaled with O.
    static constexpr bool LR_MMA = (D == 64 && EB == 2);
    static constexpr int PV_N = LR_MMA ? D + 16 : D;
    static constexpr int TMEM_O_STRIDE = LR_MMA ? 128 : D;  // O_t (and its row sums) at TMEM_O + t*stride
    static constexpr int ONES_OFF = OST_OFF + QT * OST_BYTES;
    static constexpr int ONES_BYTES = LR_MMA ? 2048 : 0;
    static constexpr int SMEM_BYTES = ONES_OFF + ONES_BYTES + 1024;  // +1 KiB for alignment
    static constexpr int TMEM_COLS = 512;
    static constexpr int TMEM_S = 0;               // S_t at column t*BN (P_t aliases it)
    static constexpr int TMEM_O = QT * BN;         // O_t at TMEM_O + t*TMEM_O_STRIDE
    static constexpr int THREADS = 384;
    static constexpr int REGS_SOFTMAX = 216;
    static constexpr int REGS_OTHER = 72;
    static_assert(TMEM_O + QT * TMEM_O_STRIDE <= TMEM_COLS && PV_N <= TMEM_O_STRIDE, "tensor memory budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Ctl {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_half[2], p_full[2], o_full[2];
    uint64_t mma_done;
    uint64_t unit_full[4], unit_empty[4];  // ring of claimed unit indices (dynamic schedule)
    int32_t unit_idx[4];
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t collided;  // the schedule slot belongs to another launch: take no unit
};
static_assert(sizeof(Ctl) <= 1024, "control block");
constexpr int kUnitRing = 4;
constexpr int kUnitReaders = 9;  // the MMA warp and the 8 softmax warps

struct Unit {
    int bh;      // dense: b*h index of the head plane; varlen: head index
    int row0;    // first query row of the unit within its sequence
    int sq, sk;  // query / key length of the unit's sequence
    int q_tok0;  // varlen: token of query row 0 of the sequence (else 0)
    int k_tok0;  // varlen: token of key 0 of the sequence (else 0)
    int jb;      // first K/V tile of the unit
    int n;       // number of K/V tiles (0: the rows see no key in this range)
    int split;   // split index (0 without split-KV)
};

template <int D, bool CAUSAL>
__device__ __forceinline__ Unit decode_unit(int u, const FwdParams &p)
{
    using C = Cfg<D>;
    Unit un;
    un.split = u % p.num_splits;
    const int v = u / p.num_splits;  // (bh, row block) index
    int mblk, bh;
    if (CAUSAL && p.group > 0) {  // head groups, heaviest row blocks first within each
        const int per = p.group * p.num_mblk;
        const int g = v / per;
        const int r = v - g * per;
        const int gsize = min(p.group, p.bh - g * p.group);
        mblk = p.num_mblk - 1 - r / gsize;
        bh = g * p.group + r % gsize;
    } else if (CAUSAL) {  // heaviest row blocks first
        mblk = p.num_mblk - 1 - v / p.bh;
        bh = v % p.bh;
    } else {       // consecutive units share a head (K/V reuse in L2)
        bh = v / p.num_mblk;
        mblk = v % p.num_mblk;
    }
    un.row0 = mblk * C::UNIT_ROWS;
    if (p.cu_q != nullptr) {
        const int seq = bh / p.heads;
        un.bh = bh % p.heads;
        un.q_tok0 = p.cu_q[seq];
        un.sq = p.cu_q[seq + 1] - un.q_tok0;
        un.k_tok0 = p.cu_k[seq];
        un.sk = p.cu_k[seq + 1] - un.k_tok0;
        // offsets outside the packed tensors: treat as an empty sequence
        if (un.q_tok0 < 0 || un.sq < 0 || un.q_tok0 + un.sq > p.total_q || un.k_tok0 < 0 || un.sk < 0 ||
            un.k_tok0 + un.sk > p.total_k)
            un.sq = un.sk = 0;
    } else {
        un.bh = bh;
        un.q_tok0 = un.k_tok0 = 0;
        un.sq = p.sq;
        un.sk = p.sk;
        if (p.seqlens_k != nullptr) {
            const int cached = min(max(p.seqlens_k[bh / p.heads], 0), p.sk);
            un.sk = static_cast<int>(min(static_cast<long long>(cached) + p.seqlens_add, static_cast<long long>(p.sk)));
        }
    }
    const int last = min(un.row0 + C::UNIT_ROWS - 1, un.sq - 1);
    const int kend = CAUSAL ? min(un.sk, last + 1 + (un.sk - un.sq)) : un.sk;
    const int n_all = (kend > 0 && un.row0 < un.sq) ? (kend + C::BN - 1) / C::BN : 0;
    // the unit's own tile range, cut into num_splits near-equal parts (the
    // splits of a row block share its work whatever its visible length)
    const int per = (n_all + p.num_splits - 1) / p.num_splits;
    un.jb = un.split * per;
    un.n = max(0, min(n_all, un.jb + per) - un.jb);
    return un;
}

// Element offset of query row `row` (within the unit's sequence) in O, and
// its index in LSE, for either layout.
__device__ __forceinline__ size_t o_row_offset(const FwdParams &p, const Unit &un, int row, int D)
{
    if (p.cu_q != nullptr)
        return (static_cast<size_t>(un.q_tok0 + row) * p.heads + un.bh) * D;
    return (static_cast<size_t>(un.bh) * p.sq + row) * D;
}

__device__ __forceinline__ size_t lse_index(const FwdParams &p, const Unit &un, int row)
{
    if (p.cu_q != nullptr) return static_cast<size_t>(un.bh) * p.total_q + un.q_tok0 + row;
    return static_cast<size_t>(un.bh) * p.sq + row;
}

// Rows of O (and entries of LSE) in either layout.
__device__ __forceinline__ size_t o_rows_total(const FwdParams &p)
{
    return p.cu_q != nullptr ? static_cast<size_t>(p.total_q) * p.heads : static_cast<size_t>(p.bh) * p.sq;
}

// A decoded unit lies inside the problem: its head plane (head, when
// packed), its rows and its key tiles lie within the tensors the maps and
// the output pointers describe.
__device__ __forceinline__ bool unit_in_bounds(int u, const Unit &un, const FwdParams &p, int unit_rows, int bn)
{
    if (u < 0 || u >= p.num_units || un.row0 < 0 || un.jb < 0 || un.n < 0 || un.split < 0 || un.split >= p.num_splits)
        return false;
    if (un.row0 >= p.num_mblk * unit_rows) return false;
    // (an empty split range may start past the last key tile: it reads nothing)
    const long long key_cap = (static_cast<long long>(p.sk) + bn - 1) / bn * bn;
    if (un.n > 0 && static_cast<long long>(un.jb + un.n) * bn > key_cap) return false;
    if (p.cu_q != nullptr) {
        if (un.bh >= p.heads || un.q_tok0 < 0 || un.k_tok0 < 0 || un.q_tok0 + un.sq > p.total_q ||
            un.k_tok0 + un.sk > p.total_k || un.sq > p.sq || un.sk > p.sk)
            return false;
        return un.n == 0 || (un.jb + un.n - 1) * bn < un.sk;
    }
    return un.bh < p.bh && un.sq == p.sq && un.sk >= 0 && un.sk <= p.sk;
}

// Zero rows [valid, BN) of the V tile at shared address `tile`, in every
// panel (a row is 128 contiguous bytes of a panel whatever the swizzle).
// Those are keys past the end of the unit's sequence that the tile copy
// still brought in, from the unused part of a KV cache or from the next
// packed sequence: their probabilities are zero, but a NaN or an infinity
// stored there would reach O through 0 * x in the P.V product.  Called by
// a whole warp; the proxy fence makes the stores visible to the MMA that
// the elected lane issues after the following __syncwarp.
template <int D, int EB>
__device__ __forceinline__ void zero_v_tail_rows(uint32_t tile, int valid)
{
    using C = Cfg<D, EB>;
    const int lane = threadIdx.x & 31;
    const int chunks = (C::BN - valid) * (C::ROW_BYTES / 16);  // 16-byte chunks per panel
    for (int pn = 0; pn < C::NPANEL; ++pn)
        for (int c = lane; c < chunks; c += 32)
            st_shared_v4(tile + pn * C::PANEL_BYTES + valid * C::ROW_BYTES + c * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    __syncwarp();
}

// The i-th work unit of this CTA.  Rounds of gridDim.x units are dealt out
// in alternating directions (boustrophedon): with the causal heaviest-first
// order this evens out the per-CTA work to within a fraction of a percent
// (a plain stride leaves the CTAs that draw the heaviest unit of every round
// several percent behind).  The last round may be partial: callers skip
// indices >= num_units and keep going until i * gridDim.x >= num_units.
__device__ __forceinline__ int unit_at(int i)
{
    const int g = static_cast<int>(gridDim.x);
    const int c = (i & 1) ? (g - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
    return i * g + c;
}

// The first failure of a launch (or of earlier launches, until the status is
// cleared) is kept: {code, block, warp, site}.
__device__ __forceinline__ void record_status(uint32_t *status, uint32_t code, uint32_t site)
{
    if (atomicCAS(&status[0], 0u, code) == 0u) {
        status[1] = blockIdx.x;
        status[2] = threadIdx.x >> 5;
        status[3] = site;
        __threadfence();
    }
}

// Checked builds: `ok` false records STATUS_BOUNDS at `site` and raises the
// CTA's abort flag, so that the other warps wind down as after a wait that
// ran out; the caller skips the access.  Normal builds: always true (the
// condition is not evaluated).
#if ATTN_CHECKED
#define ATTN_IN_BOUNDS(cond, site) in_bounds((cond), ctl, p, (site))
__device__ __forceinline__ bool in_bounds(bool ok, Ctl *ctl, const FwdParams &p, uint32_t site)
{
    if (!ok) {
        *reinterpret_cast<volatile uint32_t *>(&ctl->abort) = 1u;
        record_status(p.status, STATUS_BOUNDS, site);
    }
    return ok;
}
#else
#define ATTN_IN_BOUNDS(cond, site) true
#endif

static __device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, Ctl *ctl, const FwdParams &p,
                                              uint32_t site)
{
    volatile uint32_t *abort_flag = &ctl->abort;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1u;
            record_status(p.status, STATUS_TIMEOUT, site);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to let this thread's own
// copies and MMAs land before the CTA frees its resources).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > timeout_ns) break;
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, Ctl *ctl, const FwdParams &p,
                                         uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, ctl, p, site);
}

// bar_wait by every lane of a warp, with a warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl *ctl, const FwdParams &p, uint32_t site)
{
    const bool w = bar_wait(bar, parity, ctl, p, site);
    return __all_sync(0xffffffffu, w);
}

// The i-th unit of this CTA, for a warp that consumes the schedule (the MMA
// and softmax warps), called by the whole warp.  u = -1: no more units;
// u = -2: a hole in the last round of the fixed deal (skip it).  With the
// dynamic schedule the index comes from the ring the producer fills, and
// lane 0 releases the slot.  Returns false when a wait gave up.
__device__ __forceinline__ bool consumer_unit(uint32_t i, int &u, Ctl *ctl, const FwdParams &p)
{
    if (p.sched == nullptr) {
        if (static_cast<long long>(i) * gridDim.x >= p.num_units) {
            u = -1;
        } else {
            u = unit_at(static_cast<int>(i));
            if (u >= p.num_units) u = -2;
        }
        return true;
    }
    const uint32_t slot = i % kUnitRing;
    if (!warp_wait(smem_addr(&ctl->unit_full[slot]), (i / kUnitRing) & 1u, ctl, p, SITE_UNIT_FULL)) return false;
    u = *reinterpret_cast<volatile int32_t *>(&ctl->unit_idx[slot]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&ctl->unit_empty[slot]));
    return true;
}

// The same for the producer warp, which with the dynamic schedule claims
// the next unit from the global counter (in order: the unit order is the
// priority order) and publishes it in the ring.
__device__ __forceinline__ bool producer_unit(uint32_t i, int &u, Ctl *ctl, const FwdParams &p)
{
    if (p.sched == nullptr) return consumer_unit(i, u, ctl, p);
    const uint32_t slot = i % kUnitRing;
    if (!warp_wait(smem_addr(&ctl->unit_empty[slot]), ((i / kUnitRing) & 1u) ^ 1u, ctl, p, SITE_UNIT_EMPTY))
        return false;
    int v = -1;
    if ((threadIdx.x & 31) == 0) {
        v = ctl->collided ? -1 : atomicAdd(p.sched, 1);
        if (v >= p.num_units) v = -1;
        ctl->unit_idx[slot] = v;
        mbar_arrive(smem_addr(&ctl->unit_full[slot]));
    }
    u = __shfl_sync(0xffffffffu, v, 0);
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
__device__ __forceinline__ float add_halves(uint32_t u, float acc);

template <>
__device__ __forceinline__ float add_halves<__nv_bfloat16>(uint32_t u, float acc)
{
    return add_halves_bf16(u, acc);
}

template <>
__device__ __forceinline__ float add_halves<__half>(uint32_t u, float acc)
{
    return add_halves_f16(u, acc);
}

// Columns >= lim of this row get the identity of the row reduction (+inf
// for a min, -inf for a max), so they neither set the extreme nor, after
// exp_store_tile's own mask, contribute a probability.
__device__ __forceinline__ void mask_columns(uint32_t (&sr)[128], int lim, bool neg)
{
    const uint32_t ident = __float_as_uint(neg ? INFINITY : -INFINITY);
#pragma unroll
    for (int c = 0; c < 128; ++c) sr[c] = (c < lim) ? sr[c] : ident;
}

// Row maximum (minimum when NEG) of the 128 raw logits: eight independent
// chains (chain i takes columns i, i+8, ..., i+120) of 3-input max/min.
template <bool NEG>
__device__ __forceinline__ float row_extreme(const uint32_t (&sr)[128])
{
    auto f3 = [](float a, float b, float c) { return NEG ? min3f(a, b, c) : max3f(a, b, c); };
    auto f2 = [](float a, float b) { return NEG ? fminf(a, b) : fmaxf(a, b); };
    auto col = [&](int i, int k) { return __uint_as_float(sr[i + 8 * k]); };
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        r[i] = f3(col(i, 0), col(i, 1), col(i, 2));
#pragma unroll
        for (int k = 3; k < 15; k += 2) r[i] = f3(r[i], col(i, k), col(i, k + 1));
        r[i] = f2(r[i], col(i, 15));
    }
    const float a = f3(r[0], r[1], r[2]), b = f3(r[3], r[4], r[5]);
    return f3(a, b, f2(r[6], r[7]));
}

// O row *= alpha in tensor memory (D fp32 columns of this thread's lane).
template <int D>
__device__ __forceinline__ void rescale_rows(uint32_t tO, float alpha)
{
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t orr[32];
        tmem_ld32_wait(tO + ch * 32, orr);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(orr[2 * c]), __uint_as_float(orr[2 * c + 1])), a2);
            orr[2 * c] = __float_as_uint(v.x);
            orr[2 * c + 1] = __float_as_uint(v.y);
        }
        tmem_st32(tO + ch * 32, orr);
    }
}

// This warp's tensor-memory stores are complete: every lane waits for its
// own and orders them before the warp barrier, and one lane arrives on
// `bar` for the warp (the P hand-off barriers count warps, not threads: 32
// arrivals on one shared-memory word per warp cost more than the barrier).
__device__ __forceinline__ void warp_announce_tmem(uint32_t bar)
{
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// p = 2^(s*sl2e - m_use) for the 128 columns of this row; P (rounded to T,
// two per 32-bit column) is stored into the first 64 tensor-memory columns
// at tS.  The first half (keys 0..63) is stored and announced on `half_bar`
// as soon as it is ready, so the P.V product can start on it while the
// second half is computed.  Returns {sum of p, sum of p as rounded}; the
// second is 0 when LR is false (the tensor core sums the rounded P).  The
// caller waits for the second store (tmem_wait_st) and announces it.
template <typename T, bool MASKED, bool LR = true>
__device__ __forceinline__ float2 exp_store_tile(const uint32_t (&sr)[128], int lim, float sl2e, float m_use, uint32_t tS,
                                                 uint32_t half_bar)
{
    const float2 sc2 = make_float2(sl2e, sl2e);
    const float2 nm2 = make_float2(-m_use, -m_use);
    float2 l4[4];
    float lr4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        l4[i] = make_float2(0.f, 0.f);
        lr4[i] = 0.f;
    }
    if constexpr (!Elem<T>::FP8) {
        uint32_t pa[32], pb[32];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nm2);
            if (MASKED) {
                x.x = (2 * c < lim) ? x.x : -INFINITY;
                x.y = (2 * c + 1 < lim) ? x.y : -INFINITY;
            }
            const float p0 = ex2_approx(x.x);
            const float p1 = ex2_approx(x.y);
            l4[c & 3] = __fadd2_rn(l4[c & 3], make_float2(p0, p1));
            const uint32_t pk = pack2<T>(p0, p1);
            if constexpr (LR) lr4[c & 3] = add_halves<T>(pk, lr4[c & 3]);
            if (c < 32)
                pa[c] = pk;
            else
                pb[c - 32] = pk;
            if (c == 31) {
                tmem_st32(tS, pa);
                warp_announce_tmem(half_bar);
            }
        }
        tmem_st32(tS + 32, pb);
    } else {
        // e4m3: four per 32-bit column; 32 columns for the 128 keys
        uint32_t pa[16], pb[16];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1])), sc2, nm2);
            float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3])), sc2, nm2);
            if (MASKED) {
                x0.x = (4 * c < lim) ? x0.x : -INFINITY;
                x0.y = (4 * c + 1 < lim) ? x0.y : -INFINITY;
                x1.x = (4 * c + 2 < lim) ? x1.x : -INFINITY;
                x1.y = (4 * c + 3 < lim) ? x1.y : -INFINITY;
            }
            const float p0 = ex2_approx(x0.x), p1 = ex2_approx(x0.y);
            const float p2 = ex2_approx(x1.x), p3 = ex2_approx(x1.y);
            l4[c & 3] = __fadd2_rn(l4[c & 3], __fadd2_rn(make_float2(p0, p1), make_float2(p2, p3)));
            const uint32_t lo = pack_e4m3x2(p0, p1), hi = pack_e4m3x2(p2, p3);
            lr4[c & 3] = add_halves_f16(e4m3x2_to_f16x2(lo), lr4[c & 3]);
            lr4[c & 3] = add_halves_f16(e4m3x2_to_f16x2(hi), lr4[c & 3]);
            const uint32_t pk = lo | (hi << 16);
            if (c < 16)
                pa[c] = pk;
            else
                pb[c - 16] = pk;
            if (c == 15) {
                tmem_st16(tS, pa);
                warp_announce_tmem(half_bar);
            }
        }
        tmem_st16(tS + 16, pb);
    }
    const float2 a = __fadd2_rn(l4[0], l4[1]);
    const float2 b = __fadd2_rn(l4[2], l4[3]);
    return make_float2((a.x + a.y) + (b.x + b.y), (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]));
}

template <typename T>
__device__ __forceinline__ void store_row_zero(const FwdParams &p, const Unit &un, int row, int D)
{
    if (row >= un.sq) return;
    if (p.num_splits > 1) {  // an empty split range: weight 0 in the combine
        const size_t r = (static_cast<size_t>(un.split) * p.bh + un.bh) * p.sq + row;
        float4 *dst = reinterpret_cast<float4 *>(p.o_part + r * D);
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.lse_part[2 * r] = -INFINITY;
        p.lse_part[2 * r + 1] = -INFINITY;
        return;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<typename Elem<T>::Out *>(p.o) + o_row_offset(p, un, row, D));
    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse) p.lse[lse_index(p, un, row)] = -INFINITY;
}

// Whether the 32 rows of a warp starting at row r0 go through the warp's
// staging slice and the copy engine (rows past the end of a dense tensor are
// dropped by the copy engine).  Not for split partials (fp32, written row by
// row), not for rows that all lie past the sequence, and not for packed rows
// that run past their sequence, whose last rows belong to the next one.
template <typename C>
__device__ __forceinline__ bool o_staged(const FwdParams &p, const Unit &un, int r0)
{
    if (p.num_splits > 1 || r0 >= un.sq) return false;
    return p.cu_q == nullptr || r0 + 32 <= un.sq;
}

template <int D, typename T, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p)
{
    using E = Elem<T>;
    using C = Cfg<D, E::BYTES>;
    using TO = typename E::Out;
    // format code 1 = bf16 in kind::f16; 0 = f16, or e4m3 in kind::f8f6f4
    constexpr uint32_t IDESC_QK = idesc_f16(128, C::BN, E::BF16, false);
    constexpr uint32_t IDESC_PV = idesc_f16(128, C::PV_N, E::BF16, true);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_addr - raw_addr);
    Ctl *ctl = reinterpret_cast<Ctl *>(smem);
    const uint32_t sQ = base_addr + C::Q_OFF;    // Q tile t at sQ + t*TILE_BYTES
    const uint32_t sKV = base_addr + C::KV_OFF;  // slot s at sKV + s*TILE_BYTES
    const uint32_t sOst = base_addr + C::OST_OFF;  // O staging panel of group t at sOst + t*OST_BYTES

    auto B = [&](const uint64_t &bar) { return smem_addr(&bar); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    ATTN_TRACE_DECL
    ATTN_TRACE(EV_K_ENTRY, 0);

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(B(ctl->q_full[t]), 1);
            mbar_init(B(ctl->q_empty[t]), 1);
            mbar_init(B(ctl->s_full[t]), 1);
            mbar_init(B(ctl->p_half[t]), 4);  // one arrival per softmax warp
            mbar_init(B(ctl->p_full[t]), 4);
            mbar_init(B(ctl->o_full[t]), 1);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(B(ctl->kv_full[s]), 1);
            mbar_init(B(ctl->kv_empty[s]), 1);
        }
        mbar_init(B(ctl->mma_done), 1);
        for (int s = 0; s < kUnitRing; ++s) {
            mbar_init(B(ctl->unit_full[s]), 1);
            mbar_init(B(ctl->unit_empty[s]), kUnitReaders);
        }
        ctl->abort = 0u;
        ctl->collided = 0u;
        if (p.sched != nullptr) {
            // take the schedule slot for this launch, or find it held by
            // another one (more launches in flight than there are slots)
            const uint32_t prev = atomicCAS(reinterpret_cast<unsigned int *>(p.sched + 2), 0u, p.sched_gen);
            if (prev != 0u && prev != p.sched_gen) {
                ctl->collided = 1u;
                record_status(p.status, STATUS_SCHED_COLLISION, SITE_SCHED_SLOT);
            }
            __threadfence();
        }
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_addr(&ctl->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (C::LR_MMA) {
        if (threadIdx.x < C::ONES_BYTES / 16) {  // the block of ones (1.0 in T, two per word)
            const uint32_t one2 = E::BF16 ? 0x3F803F80u : 0x3C003C00u;
            st_shared_v4(base_addr + C::ONES_OFF + threadIdx.x * 16, one2, one2, one2, one2);
            fence_proxy_async_smem();
        }
    }
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    ATTN_TRACE(EV_K_READY, 0);
#if ATTN_CHECKED
    {
        uint32_t dsmem;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dsmem));
        const bool window = (base_addr - raw_addr) + C::SMEM_BYTES - 1024u <= dsmem;
        const bool tcols = (tmem >> 16) == 0u && (tmem & 0xFFFFu) + C::TMEM_COLS <= 512u;
        const bool setup_ok = (threadIdx.x != 0) || (ATTN_IN_BOUNDS(window, SITE_CHK_SMEM) &&
                                                     ATTN_IN_BOUNDS(tcols, SITE_CHK_TMEM));
        // every thread takes the same decision: no role starts on a bad layout
        if (!__syncthreads_and(setup_ok ? 1 : 0)) goto wind_down;
    }
#endif

    if (warp >= 8) {
      // Warpgroup 2: the setmaxnreg and all of this warpgroup's work sit in
      // one warpgroup-uniform branch, so the compiler knows the budget.
      regs_dec<C::REGS_OTHER>();
      ATTN_TRACE(EV_REGS, 0);
      if (warp == 9) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the schedule, so counters and addresses are
        // warp-uniform; one elected lane issues the copies.  Q is read by
        // one unit only (evict-first in L2).  Each K/V tile is requested
        // from L2 ATTN_KV_PREFETCH tiles ahead of its load, so that the load
        // (issued only when a ring slot frees up) finds it there.
        const uint64_t pol_q = ATTN_Q_EVICT_FIRST ? l2_evict_first() : l2_evict_normal();
        const uint64_t pol_kv = l2_evict_normal();
        uint32_t kv_it = 0, q_it = 0;
        bool ok = true;
        for (uint32_t i = 0; ok; ++i) {
            int u;
            if (!(ok = producer_unit(i, u, ctl, p))) break;
            if (u == -1) break;
            if (u < 0) continue;
            ATTN_TRACE(EV_UNIT, u);
            if (!ATTN_IN_BOUNDS(u < p.num_units, SITE_CHK_UNIT)) {  // before decode reads any offset
                ok = false;
                break;
            }
            const Unit un = decode_unit<D, CAUSAL>(u, p);
            ATTN_TRACE(EV_DECODED, u);
            if (!ATTN_IN_BOUNDS(unit_in_bounds(u, un, p, C::UNIT_ROWS, C::BN), SITE_CHK_UNIT)) {
                ok = false;
                break;
            }
            if (un.n == 0) continue;
            // TMA coordinates (after the 64-column panel): dense maps are
            // [bh][s][D] (row, plane = bh); varlen maps are [token][head][D]
            // (row = head, plane = token).
            const bool vl = p.cu_q != nullptr;
            const bool paged = p.block_table != nullptr;
            auto row_coord = [&](int r) { return vl ? un.bh : r; };
            auto plane_coord = [&](int r) { return vl ? un.q_tok0 + r : un.bh; };
            auto krow_coord = [&](int r) { return vl ? un.bh : (paged ? un.bh % p.heads : r); };
            auto kplane_coord = [&](int r) {
                if (vl) return un.k_tok0 + r;
                if (!paged) return un.bh;
                // the pool token of logical key r; a page index outside the
                // pool gives a coordinate past its end (the copy reads zeros)
                const long long pg = p.block_table[static_cast<long long>(un.bh / p.heads) * p.pages_per_seq +
                                                   r / p.page_size];
                if (pg < 0 || pg >= p.num_pages) return static_cast<int>(static_cast<long long>(p.num_pages) * p.page_size);
                return static_cast<int>(pg * p.page_size + r % p.page_size);
            };
            for (int t = 0; t < C::QT && ok; ++t) {
                ok = warp_wait(B(ctl->q_empty[t]), (q_it & 1u) ^ 1u, ctl, p, SITE_LOAD_Q_EMPTY);
                if (!ok) break;
                {
                    // the tile starts inside the unit's padded rows (a tile
                    // wholly past the end reads zeros, as the copy engine fills)
                    const int qr = un.row0 + t * C::BM;
                    if (!ATTN_IN_BOUNDS(qr < p.num_mblk * C::UNIT_ROWS && (vl ? un.q_tok0 + qr < p.total_q + C::UNIT_ROWS
                                                                             : un.bh < p.bh),
                                        SITE_CHK_Q_LOAD)) {
                        ok = false;
                        break;
                    }
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(B(ctl->q_full[t]), C::TILE_BYTES);
                    for (int pn = 0; pn < C::NPANEL; ++pn)
                        tma_load_3d(sQ + t * C::TILE_BYTES + pn * C::PANEL_BYTES, &tmQ, B(ctl->q_full[t]),
                                    pn * C::PANEL_ELEMS, row_coord(un.row0 + t * C::BM), plane_coord(un.row0 + t * C::BM),
                                    pol_q);
                }
                __syncwarp();
            }
            if (!ok) break;
            ++q_it;
            ATTN_TRACE(EV_Q_ISSUED, u);
            if (ATTN_KV_PREFETCH > 0 && elect_one()) {
                for (int jj = 0; jj < ATTN_KV_PREFETCH && jj < un.n; ++jj)
                    for (int pn = 0; pn < C::NPANEL; ++pn) {
                        tma_prefetch_3d(&tmK, pn * C::PANEL_ELEMS, krow_coord((un.jb + jj) * C::BN),
                                        kplane_coord((un.jb + jj) * C::BN));
                        tma_prefetch_3d(&tmV, pn * C::PANEL_ELEMS, krow_coord((un.jb + jj) * C::BN),
                                        kplane_coord((un.jb + jj) * C::BN));
                    }
            }
            __syncwarp();
            for (int j = 0; j < un.n && ok; ++j) {
                if (ATTN_KV_PREFETCH > 0 && j + ATTN_KV_PREFETCH < un.n && elect_one()) {
                    for (int pn = 0; pn < C::NPANEL; ++pn) {
                        tma_prefetch_3d(&tmK, pn * C::PANEL_ELEMS, krow_coord((un.jb + j + ATTN_KV_PREFETCH) * C::BN),
                                        kplane_coord((un.jb + j + ATTN_KV_PREFETCH) * C::BN));
                        tma_prefetch_3d(&tmV, pn * C::PANEL_ELEMS, krow_coord((un.jb + j + ATTN_KV_PREFETCH) * C::BN),
                                        kplane_coord((un.jb + j + ATTN_KV_PREFETCH) * C::BN));
                    }
                }
                __syncwarp();
                for (int which = 0; which < 2; ++which) {
                    const uint32_t slot = kv_it % C::NSLOT;
                    ATTN_TRACE(EV_LD_WAIT, kv_it);
                    ok = warp_wait(B(ctl->kv_empty[slot]), ((kv_it / C::NSLOT) & 1u) ^ 1u, ctl, p,
                                   SITE_LOAD_KV_EMPTY);
                    ATTN_TRACE(EV_LD_GOT, kv_it);
                    if (!ok) break;
#if ATTN_CHECKED
                    {
                        // the tile starts at a visible key of a plane (token, page) of the map
                        const int kr = (un.jb + j) * C::BN;
                        const int kp = kplane_coord(kr), kh = krow_coord(kr);
                        bool in = kr < (p.sk + C::BN - 1) / C::BN * C::BN && kr >= 0;
                        if (vl)
                            in = in && kp >= 0 && kp < p.total_k && kh < p.heads;
                        else if (paged)
                            in = in && kp >= 0 && static_cast<long long>(kp) <= static_cast<long long>(p.num_pages) * p.page_size &&
                                 kh < p.heads;
                        else
                            in = in && kp < p.bh;
                        if (!ATTN_IN_BOUNDS(in, SITE_CHK_KV_LOAD)) {
                            ok = false;
                            break;
                        }
                    }
#endif
                    if (static_cast<int32_t>(kv_it) != p.withheld_load && elect_one()) {
                        mbar_arrive_expect_tx(B(ctl->kv_full[slot]), C::TILE_BYTES);
                        const CUtensorMap *m = which ? &tmV : &tmK;
                        for (int pn = 0; pn < C::NPANEL; ++pn)
                            tma_load_3d(sKV + slot * C::TILE_BYTES + pn * C::PANEL_BYTES, m, B(ctl->kv_full[slot]),
                                        pn * C::PANEL_ELEMS, krow_coord((un.jb + j) * C::BN),
                                        kplane_coord((un.jb + j) * C::BN), pol_kv);
                    }
                    __syncwarp();
                    ++kv_it;
                }
            }
        }
        {
            // Wind-down: wait (bounded) for the last copies this warp issued,
            // so that no copy lands after the CTA exits even when a consumer
            // gave up (normally these have long completed).
            const uint32_t first = kv_it > C::NSLOT ? kv_it - C::NSLOT : 0u;
            for (uint32_t i = first; i < kv_it; ++i) {
                if (static_cast<int32_t>(i) == p.withheld_load) continue;
                drain_wait(B(ctl->kv_full[i % C::NSLOT]), (i / C::NSLOT) & 1u, p.timeout_ns);
            }
            if (q_it > 0)
                for (int t = 0; t < C::QT; ++t)
                    drain_wait(B(ctl->q_full[t]), (q_it - 1) & 1u, p.timeout_ns);
        }
        __syncwarp();
      } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule and waits; one elected lane (the
        // same one every time: all lanes are active) issues the MMAs and the
        // commits that track them.
        uint32_t kv_it = 0, q_it = 0;
        uint32_t p_ph0 = 0u, p_ph1 = 0u;
        bool ok = true;
        // keys past a unit's end are in bounds of the V copy (not zero-filled);
        // the 8-bit forward is dense only, where the copy engine zero-fills them
        const bool zero_tail = !E::FP8 && (p.cu_k != nullptr || p.seqlens_k != nullptr);
        auto kv_wait = [&](uint32_t &slot) -> bool {
            slot = kv_it % C::NSLOT;
            ATTN_TRACE(EV_MMA_WAIT_KV, kv_it);
            const bool r = warp_wait(B(ctl->kv_full[slot]), (kv_it / C::NSLOT) & 1u, ctl, p, SITE_MMA_KV_FULL);
            ATTN_TRACE(EV_MMA_GOT_KV, kv_it);
            ++kv_it;
            return r;
        };
        // Low descriptor words of the first k-step; later k-steps add their
        // byte offset >> 4 to the start-address field, which cannot carry
        // (shared addresses stay below 2^18).
        const uint32_t dq0 = desc_lo(sQ, 16);
        const uint32_t dk0 = desc_lo(sKV, 16);
        const uint32_t dv0 = desc_lo(sKV, C::PANEL_BYTES);
        const uint32_t ones_addr = base_addr + C::ONES_OFF;
        auto issue_qk = [&](int t, uint32_t kslot) {
            const uint32_t a0 = dq0 + ((t * C::TILE_BYTES) >> 4);
            const uint32_t b0 = dk0 + ((kslot * C::TILE_BYTES) >> 4);
            const uint32_t d = tmem + C::TMEM_S + t * C::BN;
#pragma unroll
            for (int kk = 0; kk < C::QK_STEPS; ++kk) {  // 32 bytes of the head dim per step
                const uint32_t off =
                    ((kk / C::KSTEPS_PER_ROW) * C::PANEL_BYTES + (kk % C::KSTEPS_PER_ROW) * 32) >> 4;
                if constexpr (E::FP8)
                    mma_ss_f8(d, a0 + off, b0 + off, IDESC_QK, kk > 0 ? 1u : 0u, C::DESC_HI);
                else
                    mma_ss(d, a0 + off, b0 + off, IDESC_QK, kk > 0 ? 1u : 0u);
            }
        };
        // O_t (+)= P_t V over keys [64*half, 64*half + 64) of the tile.
        auto issue_pv = [&](int t, uint32_t vslot, bool accumulate, int half) {
            const uint32_t b0 = dv0 + ((vslot * C::TILE_BYTES) >> 4);
            const uint32_t a = tmem + C::TMEM_S + t * C::BN;  // P_t, 32 bits of keys per column
            const uint32_t d = tmem + C::TMEM_O + t * C::TMEM_O_STRIDE;
#pragma unroll
            for (int k2 = 0; k2 < C::PV_STEPS / 2; ++k2) {
                const int kk = half * (C::PV_STEPS / 2) + k2;
                const uint32_t bo = (kk * C::PV_KEYS * C::ROW_BYTES) >> 4;  // PV_KEYS rows
                if constexpr (E::FP8)
                    mma_ts_f8(d, a + kk * 8, b0 + bo, IDESC_PV, (accumulate || kk > 0) ? 1u : 0u, C::DESC_HI);
                else if constexpr (C::LR_MMA) {
                    // [V | ones]: the ones block is the second 64-column atom along N
                    const uint32_t vaddr = sKV + vslot * C::TILE_BYTES + kk * C::PV_KEYS * C::ROW_BYTES;
                    mma_ts(d, a + kk * 8, desc_lo(vaddr, ones_addr - vaddr), IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
                } else
                    mma_ts(d, a + kk * 8, b0 + bo, IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
            }
        };
        for (uint32_t i = 0; ok; ++i) {
            int u;
            if (!(ok = consumer_unit(i, u, ctl, p))) break;
            if (u == -1) break;
            if (u < 0) continue;
            ATTN_TRACE(EV_UNIT, u);
            if (!ATTN_IN_BOUNDS(u < p.num_units, SITE_CHK_UNIT)) {  // before decode reads any offset
                ok = false;
                break;
            }
            const Unit un = decode_unit<D, CAUSAL>(u, p);
            ATTN_TRACE(EV_DECODED, u);
            if (!ATTN_IN_BOUNDS(unit_in_bounds(u, un, p, C::UNIT_ROWS, C::BN), SITE_CHK_UNIT)) {
                ok = false;
                break;
            }
            if (un.n == 0) continue;
            ATTN_TRACE(EV_MMA_WAIT_Q, u);
            for (int t = 0; t < C::QT && ok; ++t)
                ok = warp_wait(B(ctl->q_full[t]), q_it & 1u, ctl, p, SITE_MMA_Q_FULL);
            ATTN_TRACE(EV_MMA_GOT_Q, u);
            if (!ok) break;
            ++q_it;
            // Q tile 1 holds none of the unit's rows (short queries, as in
            // decoding): its products are skipped, and its softmax group
            // skips the unit too.  Its copy is still made (and released).
            const bool two = un.row0 + C::BM < un.sq;
            uint32_t kslot;
            if (!(ok = kv_wait(kslot))) break;
            tc_fence_after();
            if (elect_one()) {
                issue_qk(0, kslot);
                tc_commit(B(ctl->s_full[0]));
                if (two) {
                    issue_qk(1, kslot);
                    tc_commit(B(ctl->s_full[1]));
                }
                tc_commit(B(ctl->kv_empty[kslot]));
                if (un.n == 1) tc_commit(B(ctl->q_empty[0]));
                if (un.n == 1 || !two) tc_commit(B(ctl->q_empty[1]));
            }
            __syncwarp();
            for (int j = 0; j < un.n && ok; ++j) {
                const bool more = j + 1 < un.n;
                uint32_t vslot, nslot = 0;
                if (!(ok = kv_wait(vslot))) break;
                if (zero_tail) {
                    const int valid = un.sk - (un.jb + j) * C::BN;  // > 0: the tile holds a visible key
                    if (valid < C::BN) zero_v_tail_rows<D, E::BYTES>(sKV + vslot * C::TILE_BYTES, valid);
                }
                if (more && !(ok = kv_wait(nslot))) break;
                // tile 0
                ATTN_TRACE(EV_MMA_WAIT_P, 0);
                if (!(ok = warp_wait(B(ctl->p_half[0]), p_ph0, ctl, p, SITE_MMA_P_FULL))) break;
                tc_fence_after();
                if (elect_one()) issue_pv(0, vslot, j > 0, 0);
                __syncwarp();
                if (!(ok = warp_wait(B(ctl->p_full[0]), p_ph0, ctl, p, SITE_MMA_P_FULL))) break;
                ATTN_TRACE(EV_MMA_GOT_P, 0);
                p_ph0 ^= 1u;
                tc_fence_after();
                if (elect_one()) {
                    issue_pv(0, vslot, true, 1);
                    if (!two) tc_commit(B(ctl->kv_empty[vslot]));
                    if (!more) tc_commit(B(ctl->o_full[0]));
                    if (more) {
                        issue_qk(0, nslot);
                        tc_commit(B(ctl->s_full[0]));
                        if (!two) tc_commit(B(ctl->kv_empty[nslot]));
                        if (j + 2 == un.n) tc_commit(B(ctl->q_empty[0]));
                    }
                }
                __syncwarp();
                if (!two) continue;
                // tile 1
                ATTN_TRACE(EV_MMA_WAIT_P, 1);
                if (!(ok = warp_wait(B(ctl->p_half[1]), p_ph1, ctl, p, SITE_MMA_P_FULL))) break;
                tc_fence_after();
                if (elect_one()) issue_pv(1, vslot, j > 0, 0);
                __syncwarp();
                if (!(ok = warp_wait(B(ctl->p_full[1]), p_ph1, ctl, p, SITE_MMA_P_FULL))) break;
                ATTN_TRACE(EV_MMA_GOT_P, 1);
                p_ph1 ^= 1u;
                tc_fence_after();
                if (elect_one()) {
                    issue_pv(1, vslot, true, 1);
                    tc_commit(B(ctl->kv_empty[vslot]));
                    if (!more) tc_commit(B(ctl->o_full[1]));
                    if (more) {
                        issue_qk(1, nslot);
                        tc_commit(B(ctl->s_full[1]));
                        tc_commit(B(ctl->kv_empty[nslot]));
                        if (j + 2 == un.n) tc_commit(B(ctl->q_empty[1]));
                    }
                }
                __syncwarp();
            }
        }
        // Every MMA issued must complete before tensor memory is freed.
        if (elect_one()) tc_commit(B(ctl->mma_done));
        __syncwarp();
        drain_wait(B(ctl->mma_done), 0u, p.timeout_ns);
        __syncwarp();
      }
    } else {
        regs_inc<C::REGS_SOFTMAX>();
        ATTN_TRACE(EV_REGS, 0);
        // ------------------------------------------------------------ softmax groups
        const int t = warp >> 2;      // Q tile of this group
        const int quad = warp & 3;    // TMEM lane quadrant this warp may access
        const int r_in_tile = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::TMEM_S + t * C::BN;
        const uint32_t tO = tmem + lane_off + C::TMEM_O + t * C::TMEM_O_STRIDE;
        const float sl2e = p.sl2e;
        const bool neg = sl2e < 0.f;  // the row maximum of scale*s is scale*min(s)
        uint32_t s_ph = 0u, o_ph = 0u;
        uint32_t epi_n = 0u;  // O panels this group has staged so far
        bool ok = true;
        for (uint32_t i = 0; ok; ++i) {
            int u;
            if (!(ok = consumer_unit(i, u, ctl, p))) break;
            if (u == -1) break;
            if (u < 0) continue;
            ATTN_TRACE(EV_UNIT, u);
            if (!ATTN_IN_BOUNDS(u < p.num_units, SITE_CHK_UNIT)) {  // before decode reads any offset
                ok = false;
                break;
            }
            const Unit un = decode_unit<D, CAUSAL>(u, p);
            ATTN_TRACE(EV_DECODED, u);
            if (!ATTN_IN_BOUNDS(unit_in_bounds(u, un, p, C::UNIT_ROWS, C::BN), SITE_CHK_UNIT)) {
                ok = false;
                break;
            }
            const int row = un.row0 + t * C::BM + r_in_tile;
            if (un.n == 0) {
                const bool in = row >= un.sq || (p.num_splits > 1 ? un.split < p.num_splits
                                                                  : o_row_offset(p, un, row, D) / D < o_rows_total(p));
                if (__all_sync(0xffffffffu, ATTN_IN_BOUNDS(in, SITE_CHK_O_ROW)))
                    store_row_zero<T>(p, un, row, D);
                continue;
            }
            if (t == 1 && un.row0 + C::BM >= un.sq) continue;  // no row here: the tile is not computed
            // keys visible to this row: [0, kend)
            const int kend = CAUSAL ? min(un.sk, row + 1 + (un.sk - un.sq)) : un.sk;
            // l: sum of p in fp32 (gives LSE); lr: sum of p as rounded for
            // the P.V product (normalises O, so its weights sum to one).
            float m = -INFINITY, l = 0.f, lr = 0.f;
            for (int j = 0; j < un.n; ++j) {
                ATTN_TRACE(EV_SM_WAIT_S, j);
                bool w = bar_wait(B(ctl->s_full[t]), s_ph, ctl, p, SITE_SOFTMAX_S_FULL);
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                ATTN_TRACE(EV_SM_GOT_S, j);
                s_ph ^= 1u;
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld128_wait(tS, sr);
                ATTN_TRACE(EV_SM_LD, j);
                const int lim = kend - (un.jb + j) * C::BN;  // columns >= lim are masked
                // Only diagonal and last tiles need the mask; the warp takes
                // one path or the other as a whole, so full tiles carry no
                // per-element mask work.
                const bool masked = __any_sync(0xffffffffu, lim < C::BN);
                if (masked) mask_columns(sr, lim, neg);
                float mraw;
                if (neg)
                    mraw = row_extreme<true>(sr);
                else
                    mraw = row_extreme<false>(sr);
                // a row with no visible key in this tile contributes nothing
                const float mx = (mraw == (neg ? INFINITY : -INFINITY)) ? -INFINITY : mraw * sl2e;
                const float m_new = fmaxf(m, mx);
                if (j > 0) {
                    const bool need = (m_new - m) > E::TAU;
                    if (__any_sync(0xffffffffu, need)) {
                        const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
                        rescale_rows<D>(tO, alpha);
                        if constexpr (C::LR_MMA)  // the rounded row sum, column D of the accumulator
                            tmem_st1(tO + D, __float_as_uint(__uint_as_float(tmem_ld1_wait(tO + D)) * alpha));
                        l *= alpha;
                        lr *= alpha;
                        m = m_new;
                        ATTN_TRACE(EV_SM_RESCALE, j);
                    }
                } else {
                    m = m_new;
                }
                ATTN_TRACE(EV_SM_MAX, j);
                const float m_use = ((m == -INFINITY) ? 0.f : m) - E::SHIFT;  // exp reference
                float2 sums;  // {sum of p, sum of p as rounded}
                if (masked)
                    sums = exp_store_tile<T, true, !C::LR_MMA>(sr, lim, sl2e, m_use, tS, B(ctl->p_half[t]));
                else
                    sums = exp_store_tile<T, false, !C::LR_MMA>(sr, lim, sl2e, m_use, tS, B(ctl->p_half[t]));
                l += sums.x;
                lr += sums.y;
                ATTN_TRACE(EV_SM_EXP, j);
                warp_announce_tmem(B(ctl->p_full[t]));
                ATTN_TRACE(EV_SM_ARRIVE, j);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> T, LSE
            {
                ATTN_TRACE(EV_SM_EPI_WAIT, u);
                bool w = bar_wait(B(ctl->o_full[t]), o_ph, ctl, p, SITE_SOFTMAX_O_FULL);
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                ATTN_TRACE(EV_SM_EPI_GOT, u);
                o_ph ^= 1u;
                tc_fence_after();
                if constexpr (C::LR_MMA) lr = __uint_as_float(tmem_ld1_wait(tO + D));
                const float inv_l = (lr > 0.f) ? p.o_scale / lr : 0.f;
                const float m_ref = m - E::SHIFT;  // reference of l and lr
                const bool valid = row < un.sq;
                if (p.num_splits > 1) {
                    // split partial: O / lr in fp32, both log-sum-exps
                    const size_t r = (static_cast<size_t>(un.split) * p.bh + un.bh) * p.sq + (valid ? row : 0);
                    if (!__all_sync(0xffffffffu, ATTN_IN_BOUNDS(r < static_cast<size_t>(p.num_splits) * p.bh * p.sq,
                                                                 SITE_CHK_O_PART))) {
                        ok = false;
                        break;
                    }
                    float4 *dstf = reinterpret_cast<float4 *>(p.o_part + r * D);
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t orr[32];
                        tmem_ld32_wait(tO + ch * 32, orr);
                        if (valid) {
#pragma unroll
                            for (int v4 = 0; v4 < 8; ++v4)
                                dstf[ch * 8 + v4] = make_float4(__uint_as_float(orr[4 * v4]) * inv_l,
                                                                __uint_as_float(orr[4 * v4 + 1]) * inv_l,
                                                                __uint_as_float(orr[4 * v4 + 2]) * inv_l,
                                                                __uint_as_float(orr[4 * v4 + 3]) * inv_l);
                        }
                    }
                    if (valid) {
                        p.lse_part[2 * r] = (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
                        p.lse_part[2 * r + 1] = (lr > 0.f) ? (m_ref + log2f(lr)) * 0.69314718055994531f : -INFINITY;
                    }
                    ATTN_TRACE(EV_SM_EPI_DONE, u);
                    tc_fence_before();
                    continue;
                }
                const int tile_row0 = un.row0 + t * C::BM;
                // The copy engine stores whole 128-row panels and drops rows
                // past the end of the tensor; in the packed layout those rows
                // belong to the next sequence, so a packed tile that runs past
                // its sequence is stored row by row instead.
                if (o_staged<C>(p, un, tile_row0 + quad * 32)) {
                    // This warp's 32 rows go through its staging slice, 64
                    // columns at a time; lane 0 has the copy engine store the
                    // slice and, before the slice is written again, waits
                    // until the copy engine has read it.
                    const uint32_t slice = sOst + warp * C::OST_WARP_BYTES;
                    const uint32_t my_row = slice + static_cast<uint32_t>(lane) * 128u;
                    const uint32_t swz = static_cast<uint32_t>(lane & 7);
#pragma unroll
                    for (int pn = 0; pn < C::O_NPANEL; ++pn) {
                        if (lane == 0 && epi_n > 0) bulk_wait_read_all();
                        __syncwarp();
                        // this row's 64 columns, 16-bit, in the 128-byte swizzle
                        // of the output map: 16-byte chunk c at c ^ (row % 8)
                        uint32_t orr[64];
                        tmem_ld64_wait(tO + pn * 64, orr);
#pragma unroll
                        for (int chunk = 0; chunk < 8; ++chunk) {
                            uint32_t pk[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const int col = chunk * 8 + 2 * c;
                                const float2 v = __fmul2_rn(
                                    make_float2(__uint_as_float(orr[col]), __uint_as_float(orr[col + 1])),
                                    make_float2(inv_l, inv_l));
                                pk[c] = pack2<TO>(v.x, v.y);
                            }
                            st_shared_v4(my_row + ((static_cast<uint32_t>(chunk) ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int r0 = tile_row0 + quad * 32;
                            const bool vl = p.cu_q != nullptr;
                            if (ATTN_IN_BOUNDS(r0 >= 0 && r0 < un.sq && (vl ? un.q_tok0 + r0 + 32 <= p.total_q && un.bh < p.heads
                                                                          : un.bh < p.bh),
                                               SITE_CHK_O_TILE)) {
                                tma_store_3d(&tmO, slice, pn * C::O_PANEL_COLS, vl ? un.bh : r0,
                                             vl ? un.q_tok0 + r0 : un.bh);
                                bulk_commit_group();
                            }
                        }
                        ATTN_TRACE(EV_SM_EPI_WRITTEN, pn);
                        ++epi_n;
                    }
                } else {
                    if (!__all_sync(0xffffffffu,
                                    ATTN_IN_BOUNDS(!valid || o_row_offset(p, un, row, D) / D < o_rows_total(p),
                                                   SITE_CHK_O_ROW))) {
                        ok = false;
                        break;
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<TO *>(p.o) +
                                                           o_row_offset(p, un, valid ? row : 0, D));
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t orr[32];
                        tmem_ld32_wait(tO + ch * 32, orr);
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float2 v = __fmul2_rn(
                                make_float2(__uint_as_float(orr[2 * c]), __uint_as_float(orr[2 * c + 1])),
                                make_float2(inv_l, inv_l));
                            pk[c] = pack2<TO>(v.x, v.y);
                        }
                        if (valid) {
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                dst[ch * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                }
                if (valid && p.lse && ATTN_IN_BOUNDS(lse_index(p, un, row) < o_rows_total(p), SITE_CHK_O_ROW))
                    p.lse[lse_index(p, un, row)] =
                        (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
                ATTN_TRACE(EV_SM_EPI_DONE, u);
                tc_fence_before();
            }
        }
        // this warp's O stores complete before the CTA's shared memory goes
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

#if ATTN_CHECKED
wind_down:
#endif
    ATTN_TRACE(EV_K_EXIT, 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // Dynamic schedule: every claim of this CTA has returned; the last CTA
    // to get here leaves the slot free (zero) for the next launch, clearing
    // the owner last.  A CTA that found the slot held by another launch never
    // touched its counters and is not counted; the slot then stays held by
    // this launch until attn_fwd_status_clear (the collision was reported).
    if (p.sched != nullptr && threadIdx.x == 0 && !ctl->collided) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            p.sched[0] = 0;
            p.sched[1] = 0;
            __threadfence();
            atomicExch(reinterpret_cast<unsigned int *>(p.sched + 2), 0u);
        }
    }
}

// Split-KV combine: one warp per query row.  The splits of a row are
// partial softmaxes over disjoint key ranges; merging them is the same
// rescale-and-add step as the online recurrence over key tiles
// (flash-attention-minimal forward_kernel), done once over the splits:
//   LSE = ln sum_s exp(lse_s)                      (fp32 sums)
//   O   = sum_s w_s O_s,  w_s = exp(lser_s - ln sum_t exp(lser_t))
// where O_s is normalised by its own rounded-P sum and lser_s is the
// log of that sum, so the weights applied to V still sum to one.
template <typename T, int D>
__global__ void __launch_bounds__(256)
    attn_splitkv_combine_kernel(const float *o_part, const float *lse_part, T *o, float *lse, int64_t rows,
                                int num_splits)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    constexpr int PER_LANE = D / 32;  // 4 (D = 128) or 2 (D = 64)
    for (int64_t r = warp; r < rows; r += nwarps) {
        float mx = -INFINITY, mxr = -INFINITY;
        for (int sp = lane; sp < num_splits; sp += 32) {
            mx = fmaxf(mx, lse_part[2 * (sp * rows + r)]);
            mxr = fmaxf(mxr, lse_part[2 * (sp * rows + r) + 1]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            mxr = fmaxf(mxr, __shfl_xor_sync(0xffffffffu, mxr, off));
        }
        float acc[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
        float sum = 0.f, sumr = 0.f;
        if (mxr != -INFINITY) {
            for (int sp = 0; sp < num_splits; ++sp) {
                const float ls = lse_part[2 * (sp * rows + r)];
                const float lr = lse_part[2 * (sp * rows + r) + 1];
                sum += expf(ls - mx);
                const float w = expf(lr - mxr);
                sumr += w;
                if (w > 0.f) {
                    const float *src = o_part + (sp * rows + r) * D + lane * PER_LANE;
#pragma unroll
                    for (int i = 0; i < PER_LANE; ++i) acc[i] += w * src[i];
                }
            }
        }
        const float inv = (sumr > 0.f) ? 1.f / sumr : 0.f;
        T *dst = o + r * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) dst[i] = T(acc[i] * inv);
        if (lse && lane == 0) lse[r] = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    }
}

// KV-cache append: row t of k_new / v_new of head plane bh goes to position
// clamp(seqlens[bh / h], 0, s_cache) + t of the same plane of the cache;
// rows that would land at or past s_cache are not written.  One thread per
// 16-byte chunk of K and of V.
template <typename T>
__global__ void attn_kvcache_append_kernel(const T *k_new, const T *v_new, T *k_cache, T *v_cache,
                                           const int32_t *seqlens, int64_t bh, int64_t h, int64_t s_new,
                                           int64_t s_cache, int d)
{
    const int cpr = d * static_cast<int>(sizeof(T)) / 16;  // chunks per row
    const int64_t n = bh * s_new * cpr;
    const uint4 *kn = reinterpret_cast<const uint4 *>(k_new);
    const uint4 *vn = reinterpret_cast<const uint4 *>(v_new);
    uint4 *kc = reinterpret_cast<uint4 *>(k_cache);
    uint4 *vc = reinterpret_cast<uint4 *>(v_cache);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / cpr;
        const int c = static_cast<int>(i - row * cpr);
        const int64_t plane = row / s_new;
        const int64_t t = row - plane * s_new;
        const int64_t start = min(max(static_cast<int64_t>(seqlens[plane / h]), int64_t(0)), s_cache);
        const int64_t pos = start + t;
        if (pos >= s_cache) continue;
        const int64_t dst = (plane * s_cache + pos) * cpr + c;
        kc[dst] = kn[i];
        vc[dst] = vn[i];
    }
}

// The same for a paged cache: logical position pos of batch element e is
// row pos % page_size of page block_table[e * pages_per_seq + pos /
// page_size] of the pool [num_pages][page_size][h][d]; positions at or past
// pages_per_seq * page_size, and pages outside the pool, are not written.
template <typename T>
__global__ void attn_kvcache_append_paged_kernel(const T *k_new, const T *v_new, T *k_pool, T *v_pool,
                                                 const int32_t *seqlens, const int32_t *block_table, int64_t bh,
                                                 int64_t h, int64_t s_new, int64_t pages_per_seq, int64_t page_size,
                                                 int64_t num_pages, int d)
{
    const int cpr = d * static_cast<int>(sizeof(T)) / 16;  // chunks per row
    const int64_t n = bh * s_new * cpr;
    const int64_t cap = pages_per_seq * page_size;
    const uint4 *kn = reinterpret_cast<const uint4 *>(k_new);
    const uint4 *vn = reinterpret_cast<const uint4 *>(v_new);
    uint4 *kp = reinterpret_cast<uint4 *>(k_pool);
    uint4 *vp = reinterpret_cast<uint4 *>(v_pool);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / cpr;
        const int c = static_cast<int>(i - row * cpr);
        const int64_t plane = row / s_new;
        const int64_t t = row - plane * s_new;
        const int64_t e = plane / h, head = plane - e * h;
        const int64_t pos = min(max(static_cast<int64_t>(seqlens[e]), int64_t(0)), cap) + t;
        if (pos >= cap) continue;
        const int64_t page = block_table[e * pages_per_seq + pos / page_size];
        if (page < 0 || page >= num_pages) continue;
        const int64_t token = page * page_size + pos % page_size;
        const int64_t dst = (token * h + head) * cpr + c;
        kp[dst] = kn[i];
        vp[dst] = vn[i];
    }
}

// sk == 0: every row sees no key.  O = 0, LSE = -inf.
template <typename T>
__global__ void attn_fill_empty_kernel(T *o, float *lse, int64_t rows, int d)
{
    const int64_t n = rows * d;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        o[i] = T(0.f);
    if (lse)
        for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x)
            lse[i] = -INFINITY;
}

}  // namespace attn
