// FlashAttention-2 forward pass for GB300 (sm_103a): the 16-bit kernel.
//
// What is computed: exact attention O = softmax(scale * Q K^T) V plus the
// per-row logsumexp, tile by tile with an online softmax so the N x N scores
// never reach HBM ("A Case Study in CUDA Kernel Fusion: Implementing
// FlashAttention-2 on NVIDIA Hopper Architecture using the CUTLASS Library",
// abstract), for the slice under "Kernel Specification" in "FlashAttention-2
// from scratch on Ampere, Part 1": forward only, non-causal, equal lengths,
// lengths divisible by the block size, 16-bit I/O, fp32 softmax.
//
// How. A persistent grid (one CTA per SM) walks work items; an item is two
// 128-row query tiles of one KV head (query heads that share a KV head are
// packed into one contiguous block of rows). 512 threads in four warpgroups:
//   WG0, WG1  softmax for query tile 0 / 1: thread = query row = TMEM lane
//   WG2       correction: rescales O in TMEM when a row's max grows, and the
//             epilogue (O / l -> 16 bit, LSE) for both tiles
//   WG3       warp 12: TMA producer (Q tiles, then K_0, V_0, K_1, V_1, ...
//             through a ring of 128-byte-swizzled shared-memory stages);
//             warp 13: TMEM allocator and MMA issuer (the warp runs the loop
//             converged; elect.sync picks the lane that issues each
//             tcgen05.mma / tcgen05.commit); warps 14-15 idle
// Registers are moved between warpgroups with setmaxnreg (softmax 176,
// correction 104, producer/MMA 56 per thread).
// TMEM (512 columns x 128 lanes, fp32): S_0 | S_1 | O_0 | O_1. The softmax
// writes P (16-bit, two per column) over the first half of its S columns and
// the MMA thread consumes it from TMEM as the A operand of O += P V.
// Issue order per KV tile j: PV(0,j), QK(0,j+1), PV(1,j), QK(1,j+1), so the
// exponentials of one query tile overlap the tensor-core work of the other
// (the "overlapping copy and GEMM operations" of the Hopper case study and
// the interleaving of on-chip work with computation of the Ampere series,
// done here with warp specialisation). The running max is exact (FA2's
// online softmax): the largest weight of every row is exactly 1 in 16 bits;
// O and l are rescaled whenever a row's max grows.
//
// Device code only; fa2_fwd_sm103.cu holds the host side and the C ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa2.h"
#include "ptx_sm103.cuh"

namespace fa2 {

constexpr int kBM = 128;           // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;           // keys per K/V tile
constexpr int kNQ = 2;             // query tiles per work item
constexpr int kThreads = 512;
constexpr int kCorrWarp0 = 8;      // warps 8..11
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kRegSoftmax = 176;  // 2 x 176 + 104 + 56 = 512 = 65536 / 128
constexpr uint32_t kRegCorr = 104;
constexpr uint32_t kRegOther = 56;

// Where a watchdog gave up (bits 8..15 of the status word).
enum WaitSite : int {
    kSiteQFull = 1,
    kSiteKvEmpty = 2,
    kSiteKvFull = 3,
    kSiteSFull = 4,
    kSitePFull = 5,
    kSiteOFull = 6,
    kSiteDrain = 7,
    kSiteQEmpty = 8,
    kSiteAlpha = 9,
    kSiteStats = 10,
};

struct Params {
    void* o;             // [rows_q, D] 16-bit
    float* lse;          // [rows_q]
    long long wait_limit_ns;
    int n_kv_tiles;      // N / 128
    int q_tiles;         // (Hq / Hkv) * N / 128: packed query tiles per KV head
    int pairs;           // ceil(q_tiles / 2): work items per KV head
    int total_items;     // pairs * B * Hkv
    int kv_rows;         // N
    int debug_flags;
    float scale_log2;    // scale * log2(e)
    // General mode only (ragged / unequal lengths, causal); tiles per head.
    int nq, nk;          // query and key length per head
    int causal;          // key j allowed for query i iff j < min(nk, i + 1 + nk - nq)
    int heads_q;         // B * Hq
    int hq;              // Hq
    int group;           // Hq / Hkv
    int tq;              // ceil(nq / 128): query tiles per head
    int heads_kv;        // B * Hkv
    // Extents for the debug build's checks: rows of the [rows, D] views of
    // Q / O / LSE and of K / V (equal-length mode), or per head (nq, nk).
    long long rows_q, rows_kv;
    // FP8 kernel only: fp32 descales per (batch, KV head) group.
    const float* q_descale;
    const float* k_descale;
    const float* v_descale;
};

template <int D>
struct Layout {
    static constexpr int kBlkBytes = kBM * 128;        // 128 rows x 64 elements
    static constexpr int kTileBytes = kBM * D * 2;     // one Q, K or V tile
    static constexpr int kStages = D == 128 ? 4 : 8;   // K/V ring stages
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kNQ * kTileBytes;
    // Epilogue staging: 128 rows x 64 columns of 16-bit O (128 bytes a row),
    // one 32-row slice per correction warp, which reads it back transposed.
    static constexpr int kStageOff = kRingOff + kStages * kTileBytes;
    static constexpr int kStageBytes = kBM * 128;
    static constexpr int kBarOff = kStageOff + kStageBytes;
    // q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] alpha[2] stats[2]
    // p_full[2] o_full[2] mma_done stats_free[2]
    static constexpr int kNumBars = 2 * kStages + 17;
    static constexpr int kRowOff = kBarOff + kNumBars * 8;   // per-row floats
    // alpha[2][128], m[2][128], l[2][128]
    static constexpr int kMiscOff = kRowOff + 3 * kNQ * kBM * 4;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + 1024-byte alignment slack
    // TMEM columns: S_0 | S_1 | O_0 | O_1
    static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
    static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + D * t; }
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ int g_fa2_status;  // per device; 0 = OK

// Debug builds (compiled with FA2_DEBUG: libfa2_debug.so) check every tile
// start a TMA copy is given and every global row a thread stores or loads
// outside TMA against the extents the host planned with. A failed check
// records FA2_ERR_BOUNDS and its site in the status word and skips the
// access (it never traps). Release builds compile the checks away: the
// condition is not even evaluated.
enum DbgSite : int {
    kDbgQTile = 32,     // a query tile's first row
    kDbgKvTile = 33,    // a K/V tile's first row
    kDbgORow = 34,      // an O / LSE row stored by the epilogue
    kDbgBwdRow = 35,    // a row the backward reads (LSE, D) or stores (dQ, dK, dV)
};
#ifdef FA2_DEBUG
__device__ __forceinline__ bool dbg_in_bounds(bool ok, int site) {
    if (!ok) atomicCAS(&g_fa2_status, 0, FA2_ERR_BOUNDS | (site << 8));
    return ok;
}
#define FA2_DBG_OK(cond, site) (::fa2::dbg_in_bounds((cond), (site)))
#else
#define FA2_DBG_OK(cond, site) (true)
#endif

struct Waiter {
    volatile int* abort_flag;
    long long limit_ns;

    // Waits for the phase `parity` of `bar`. Returns false if the CTA is
    // aborting (another wait ran out) or this wait ran out, in which case it
    // records the site in the status word and raises the CTA's abort flag.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int site) const {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (true) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if (*abort_flag) return false;
            if (static_cast<long long>(ptx::globaltimer_ns() - t0) > limit_ns) {
                *abort_flag = 1;
                atomicCAS(&g_fa2_status, 0, FA2_ERR_TIMEOUT | (site << 8));
                return false;
            }
        }
    }

    // Waits for N phases at once, the N tests in flight together, instead of
    // N waits one after the other. In the MMA warps this shortens the time
    // from the last of the N barriers completing to the next MMA issue
    // (measured: +4.5% for the forward), although a single test of a
    // completed barrier takes only ~20 cycles, with or without MMAs running.
    template <int N>
    __device__ __forceinline__ bool wait_all(const uint32_t (&bar)[N], const uint32_t (&parity)[N], int site) const {
        bool d[N];
        bool all = true;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            d[i] = ptx::mbar_try_wait(bar[i], parity[i]);
            all = all && d[i];
        }
        if (all) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (true) {
            all = true;
#pragma unroll
            for (int i = 0; i < N; ++i) {
                if (!d[i]) d[i] = ptx::mbar_try_wait(bar[i], parity[i]);
                all = all && d[i];
            }
            if (all) return true;
            if (*abort_flag) return false;
            if (static_cast<long long>(ptx::globaltimer_ns() - t0) > limit_ns) {
                *abort_flag = 1;
                atomicCAS(&g_fa2_status, 0, FA2_ERR_TIMEOUT | (site << 8));
                return false;
            }
        }
    }

    // Waits for phase `parity` of `bar`; meanwhile tests phase `tparity` of
    // `tbar` too, without waiting for it, and sets `seen` once it is
    // complete (so a later wait for it can be skipped).
    __device__ __forceinline__ bool wait_and_test(uint32_t bar, uint32_t parity, int site, uint32_t tbar,
                                                  uint32_t tparity, bool& seen) const {
        bool done = ptx::mbar_try_wait(bar, parity);
        if (!seen) seen = ptx::mbar_test_wait(tbar, tparity);
        if (done) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (true) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if (!seen) seen = ptx::mbar_test_wait(tbar, tparity);
            if (*abort_flag) return false;
            if (static_cast<long long>(ptx::globaltimer_ns() - t0) > limit_ns) {
                *abort_flag = 1;
                atomicCAS(&g_fa2_status, 0, FA2_ERR_TIMEOUT | (site << 8));
                return false;
            }
        }
    }

    // Same, ignoring the abort flag: used to let in-flight copies land
    // before an aborting CTA exits.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (static_cast<long long>(ptx::globaltimer_ns() - t0) > limit_ns) {
                atomicCAS(&g_fa2_status, 0, FA2_ERR_TIMEOUT | (kSiteDrain << 8));
                return false;
            }
        }
        return true;
    }
};

template <int D>
struct Bars {
    uint32_t base;
    static constexpr int S = Layout<D>::kStages;
    __device__ uint32_t q_full(int t) const { return base + 8 * t; }
    __device__ uint32_t q_empty(int t) const { return base + 8 * (2 + t); }
    __device__ uint32_t kv_full(int s) const { return base + 8 * (4 + s); }
    __device__ uint32_t kv_empty(int s) const { return base + 8 * (4 + S + s); }
    __device__ uint32_t s_full(int t) const { return base + 8 * (4 + 2 * S + t); }
    __device__ uint32_t alpha_ready(int t) const { return base + 8 * (6 + 2 * S + t); }
    __device__ uint32_t stats_ready(int t) const { return base + 8 * (8 + 2 * S + t); }
    __device__ uint32_t p_full(int t) const { return base + 8 * (10 + 2 * S + t); }
    __device__ uint32_t o_full(int t) const { return base + 8 * (12 + 2 * S + t); }
    __device__ uint32_t mma_done() const { return base + 8 * (14 + 2 * S); }
    __device__ uint32_t stats_free(int t) const { return base + 8 * (15 + 2 * S + t); }
};

// One work item: two packed query tiles of one KV head.
struct Item {
    int n_tiles;   // 1 or 2
    int q_row0;    // first query row of tile 0 in the [rows_q, D] view
    int kv_row0;   // first K/V row of the KV head
};

__device__ __forceinline__ Item make_item(const Params& p, int item) {
    const int group = item / p.pairs;
    const int qt0 = kNQ * (item - group * p.pairs);
    return Item{min(kNQ, p.q_tiles - qt0), (group * p.q_tiles + qt0) * kBM, group * p.kv_rows};
}

// General mode: an item is tiles 2p, 2p+1 of one query head. Per tile, the
// KV tiles it needs (nkv) and the first KV tile that needs masking (jmask):
// row i may attend keys j < kend(i) = min(nk, i + 1 + nk - nq) when causal,
// j < nk otherwise; kend grows with i, so the tile's last valid row sets nkv
// and its first row sets jmask. Causal items run heaviest first.
struct ItemG {
    int n_tiles;
    int head;      // b * Hq + hq
    int kvhead;    // b * Hkv + hq / group
    int q0;        // first row of tile 0 within the head
    int nkv[2];
    int jmask[2];
};

__device__ __forceinline__ int kend_of(const Params& p, int i) {
    return p.causal ? min(p.nk, i + 1 + p.nk - p.nq) : p.nk;
}

__device__ __forceinline__ ItemG make_item_gen(const Params& p, int it) {
    ItemG g;
    int pidx;
    if (p.causal) {
        pidx = p.pairs - 1 - it / p.heads_q;
        g.head = it % p.heads_q;
    } else {
        pidx = it % p.pairs;
        g.head = it / p.pairs;
    }
    const int b = g.head / p.hq;
    g.kvhead = b * (p.hq / p.group) + (g.head - b * p.hq) / p.group;
    g.q0 = 2 * pidx * kBM;
    g.n_tiles = min(kNQ, p.tq - 2 * pidx);
    for (int t = 0; t < 2; ++t) {
        g.nkv[t] = 0;
        g.jmask[t] = 0;
        if (t < g.n_tiles) {
            const int r0 = g.q0 + t * kBM;
            const int hi = kend_of(p, min(r0 + kBM - 1, p.nq - 1));
            const int lo = kend_of(p, r0);
            g.nkv[t] = hi <= 0 ? 0 : (hi + kBN - 1) / kBN;
            g.jmask[t] = lo <= 0 ? 0 : lo / kBN;
        }
    }
    return g;
}

// Items of this CTA. Equal-length mode: it, it + grid, ... (every item has
// the same work). General mode: boustrophedon over the heaviest-first item
// order, so round k goes to CTAs 0..grid-1 for even k and grid-1..0 for odd
// k; the CTA that takes the heaviest item of one round takes the lightest of
// the next. For causal items (work ~ query-tile pair index) this evens the
// CTAs' totals: at B4 H16 N4096 the busiest CTA does 1.01x the mean work
// instead of 1.14x.
template <bool kSnake>
__device__ __forceinline__ int next_item(int it) {
    if constexpr (!kSnake) {
        return it + static_cast<int>(gridDim.x);
    } else {
        const int g = static_cast<int>(gridDim.x);
        const int k = it / g + 1;
        return k * g + ((k & 1) ? g - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
    }
}

// ---------------------------------------------------------------- producer

// BarsT: any barrier set with this layout's q_full, q_empty, kv_full and
// kv_empty (the d = 64 three-buffer kernel shares this producer).
template <int D, class BarsT>
__device__ __forceinline__ void producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                         const Params& p, uint32_t sbase, const BarsT& bars, const Waiter& w) {
    using L = Layout<D>;
    constexpr int S = L::kStages;
    const bool load_q = (p.debug_flags & 1) == 0;
    int ring = 0;           // K/V ring items issued
    int nq[2] = {0, 0};     // Q loads issued per tile slot
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x) {
        const Item item = make_item(p, it);
        // Ring entry k of this item: K_{k/2} (k even) or V_{k/2} (k odd).
        auto load_kv = [&](int k) {
            const int s = ring % S;
            if (!(ok = w.wait(bars.kv_empty(s), ((ring / S) & 1) ^ 1, kSiteKvEmpty))) return;
            const uint32_t dst = sbase + L::kRingOff + s * L::kTileBytes;
            const CUtensorMap* tm = (k & 1) ? tmV : tmK;
            const int row = item.kv_row0 + (k >> 1) * kBN;
            ptx::mbar_arrive_expect_tx(bars.kv_full(s), L::kTileBytes);
            if (FA2_DBG_OK(row + kBN <= p.rows_kv, kDbgKvTile))
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk)
                    ptx::tma_load_2d(dst + blk * L::kBlkBytes, tm, blk * 64, row, bars.kv_full(s));
            ++ring;
        };
        // K_0 and V_0 first: their stages free up a step or more before the
        // Q slots do (a Q slot is released by the item's last QK of that
        // tile), and a copy takes thousands of cycles under load, so the
        // next item's first QK would otherwise wait for K_0.
        constexpr int kPre = 2;
        for (int k = 0; k < kPre && ok; ++k) load_kv(k);
        for (int t = 0; t < item.n_tiles && ok; ++t) {
            if (!(ok = w.wait(bars.q_empty(t), (nq[t] & 1) ^ 1, kSiteQEmpty))) break;
            if (load_q) {
                const uint32_t dst = sbase + L::kQOff + t * L::kTileBytes;
                ptx::mbar_arrive_expect_tx(bars.q_full(t), L::kTileBytes);
                if (FA2_DBG_OK(item.q_row0 + t * kBM + kBM <= p.rows_q, kDbgQTile))
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk)
                        ptx::tma_load_2d(dst + blk * L::kBlkBytes, tmQ, blk * 64, item.q_row0 + t * kBM,
                                         bars.q_full(t));
            }
            ++nq[t];
        }
        // Warm L2 with the query tiles this CTA takes next.
        const int nxt = it + gridDim.x;
        if (ok && nxt < p.total_items) {
            const Item ni = make_item(p, nxt);
            for (int t = 0; t < ni.n_tiles; ++t)
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk)
                    ptx::tma_prefetch_l2_2d(tmQ, blk * 64, ni.q_row0 + t * kBM);
        }
        for (int k = kPre; k < 2 * p.n_kv_tiles && ok; ++k) load_kv(k);
    }
    if (!ok) {
        // Aborting: let every copy this CTA started land before it exits.
        const int first = ring > S ? ring - S : 0;
        for (int r = first; r < ring; ++r) w.drain(bars.kv_full(r % S), (r / S) & 1);
        if (load_q)
            for (int t = 0; t < 2; ++t)
                if (nq[t] > 0) w.drain(bars.q_full(t), (nq[t] - 1) & 1);
    }
}

// ---------------------------------------------------------------- MMA issuer

// S = Q K^T over d in steps of K = 16: both operands K-major, 128-byte
// swizzle; step kk reads 64-column block kk/4 at byte offset 32*(kk%4)
// (offsets below in 16-byte units).
template <int D>
__device__ __forceinline__ void qk_kloop(uint32_t dst, uint64_t qd, uint64_t kd, uint32_t idesc) {
    constexpr uint32_t kBlk = Layout<D>::kBlkBytes >> 4;
    if constexpr (D == 128)
        ptx::mma_ss_kloop<2, 4, 6, kBlk, kBlk + 2, kBlk + 4, kBlk + 6, 2, 4, 6, kBlk, kBlk + 2, kBlk + 4, kBlk + 6, 8>(
            dst, qd, kd, idesc, 0u);
    else
        ptx::mma_ss_kloop<2, 4, 6, 0, 0, 0, 0, 2, 4, 6, 0, 0, 0, 0, 4>(dst, qd, kd, idesc, 0u);
}

// O (+)= P V over the 128 keys of a tile in steps of K = 16: P from TMEM
// (8 columns of packed pairs per step), V MN-major (16 rows of 128 B).
__device__ __forceinline__ void pv_kloop(uint32_t dst, uint32_t pa, uint64_t vd, uint32_t idesc, uint32_t acc) {
    ptx::mma_ts_kloop8(dst, pa, vd, idesc, acc);
}

template <int D, bool kBf16>
__device__ __forceinline__ void mma_issuer(const Params& p, uint32_t sbase, uint32_t tmem, const Bars<D>& bars,
                                           const Waiter& w) {
    using L = Layout<D>;
    constexpr int S = L::kStages;
    constexpr uint32_t kAB = kBf16 ? 1u : 0u;
    constexpr uint32_t kIdS = ptx::idesc_f16(kAB, 0, 0, kBM, kBN);  // S = Q K^T, both K-major
    constexpr uint32_t kIdO = ptx::idesc_f16(kAB, 0, 1, kBM, D);    // O += P V, V MN-major

    auto stage_addr = [&](int r) { return sbase + L::kRingOff + (r % S) * L::kTileBytes; };
    // A descriptor's start-address field is addr >> 4 in its low 14 bits;
    // every tile lies below 256 KB, so base + (offset >> 4) never carries out.
    auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint64_t qd = ptx::desc_sw128(sbase + L::kQOff + t * L::kTileBytes, 16, 1024);
        const uint64_t kd = ptx::desc_sw128(kaddr, 16, 1024);
        qk_kloop<D>(tmem + L::col_s(t), qd, kd, kIdS);
    };
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint64_t vd = ptx::desc_sw128(vaddr, L::kBlkBytes, 1024);
        pv_kloop(tmem + L::col_o(t), tmem + L::col_s(t), vd, kIdO, acc ? 1u : 0u);
    };
    // Every lane of the warp waits; the result is made warp-uniform.
    auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
        return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
    };
    auto wait_ring = [&](int r) { return wait_u(bars.kv_full(r % S), (r / S) & 1, kSiteKvFull); };

    const int nkv = p.n_kv_tiles;
    int ring = 0;                 // K/V ring items consumed
    int nq[2] = {0, 0};           // items seen per tile slot (q_full phases)
    int np[2] = {0, 0};           // P tiles consumed per tile slot (p_full phases)
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x) {
        const int nt = make_item(p, it).n_tiles;
        for (int t = 0; t < nt && ok; ++t) ok = wait_u(bars.q_full(t), nq[t] & 1, kSiteQFull);
        if (!ok || !(ok = wait_ring(ring))) break;
        ptx::tc_fence_after();
        for (int t = 0; t < nt; ++t) {
            issue_qk(t, stage_addr(ring));
            ptx::tc_commit_elect(bars.s_full(t));
            if (nkv == 1) ptx::tc_commit_elect(bars.q_empty(t));
        }
        ptx::tc_commit_elect(bars.kv_empty(ring % S));
        int k_ring = ring;
        ++ring;
        for (int j = 0; j < nkv; ++j) {
            const bool more = j + 1 < nkv;
            const int v_ring = ring++;
            if (more) k_ring = ring++;
            // V_j, K_{j+1} and P(0, j) are waited for together, so nothing
            // but the MMAs sits between P becoming ready and the next QK.
            const int kr = more ? k_ring : v_ring;
            const uint32_t wb[3] = {bars.kv_full(v_ring % S), bars.kv_full(kr % S), bars.p_full(0)};
            const uint32_t wp[3] = {static_cast<uint32_t>((v_ring / S) & 1), static_cast<uint32_t>((kr / S) & 1),
                                    static_cast<uint32_t>(np[0] & 1)};
            if (!(ok = __shfl_sync(0xffffffffu, w.wait_all<3>(wb, wp, kSiteKvFull) ? 1 : 0, 0) != 0)) break;
            for (int t = 0; t < nt; ++t) {
                if (t > 0 && !(ok = wait_u(bars.p_full(t), np[t] & 1, kSitePFull))) break;
                ++np[t];
                ptx::tc_fence_after();
                issue_pv(t, stage_addr(v_ring), j > 0);
                if (t == nt - 1) ptx::tc_commit_elect(bars.kv_empty(v_ring % S));
                if (more) {
                    issue_qk(t, stage_addr(k_ring));
                    ptx::tc_commit_elect(bars.s_full(t));
                    if (j + 2 == nkv) ptx::tc_commit_elect(bars.q_empty(t));
                    if (t == nt - 1) ptx::tc_commit_elect(bars.kv_empty(k_ring % S));
                } else {
                    ptx::tc_commit_elect(bars.o_full(t));
                }
            }
            if (!ok) break;
        }
        for (int t = 0; t < nt; ++t) ++nq[t];
    }
    // Every MMA issued above must finish before the CTA frees its TMEM.
    ptx::tc_commit_elect(bars.mma_done());
    w.drain(bars.mma_done(), 0);
    __syncwarp();
}


// ---------------------------------------------------------------- general mode: producer and MMA

template <int D>
__device__ __forceinline__ void producer_gen(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                             const Params& p, uint32_t sbase, const Bars<D>& bars, const Waiter& w) {
    using L = Layout<D>;
    constexpr int S = L::kStages;
    const bool load_q = (p.debug_flags & 1) == 0;
    int ring = 0;
    int nq[2] = {0, 0};
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<true>(it)) {
        const ItemG g = make_item_gen(p, it);
        for (int t = 0; t < g.n_tiles && ok; ++t) {
            if (g.nkv[t] == 0) continue;
            if (!(ok = w.wait(bars.q_empty(t), (nq[t] & 1) ^ 1, kSiteQEmpty))) break;
            if (load_q) {
                const uint32_t dst = sbase + L::kQOff + t * L::kTileBytes;
                ptx::mbar_arrive_expect_tx(bars.q_full(t), L::kTileBytes);
                if (FA2_DBG_OK(g.head < p.heads_q && g.q0 + t * kBM < p.nq, kDbgQTile))
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk)
                        ptx::tma_load_3d(dst + blk * L::kBlkBytes, tmQ, blk * 64, g.q0 + t * kBM, g.head,
                                         bars.q_full(t));
            }
            ++nq[t];
        }
        const int nmax = max(g.nkv[0], g.nkv[1]);
        for (int k = 0; k < 2 * nmax && ok; ++k) {
            const int s = ring % S;
            if (!(ok = w.wait(bars.kv_empty(s), ((ring / S) & 1) ^ 1, kSiteKvEmpty))) break;
            const uint32_t dst = sbase + L::kRingOff + s * L::kTileBytes;
            const CUtensorMap* tm = (k & 1) ? tmV : tmK;
            ptx::mbar_arrive_expect_tx(bars.kv_full(s), L::kTileBytes);
            if (FA2_DBG_OK(g.kvhead < p.heads_kv && (k >> 1) * kBN < p.nk, kDbgKvTile))
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk)
                    ptx::tma_load_3d(dst + blk * L::kBlkBytes, tm, blk * 64, (k >> 1) * kBN, g.kvhead,
                                     bars.kv_full(s));
            ++ring;
        }
    }
    if (!ok) {
        const int first = ring > S ? ring - S : 0;
        for (int r = first; r < ring; ++r) w.drain(bars.kv_full(r % S), (r / S) & 1);
        if (load_q)
            for (int t = 0; t < 2; ++t)
                if (nq[t] > 0) w.drain(bars.q_full(t), (nq[t] - 1) & 1);
    }
}

// Same issue order as mma_issuer, with a KV tile count per query tile: at KV
// tile j only the tiles with j < nkv[t] take part, and each ring stage is
// released after its last user.
template <int D, bool kBf16>
__device__ __forceinline__ void mma_issuer_gen(const Params& p, uint32_t sbase, uint32_t tmem, const Bars<D>& bars,
                                               const Waiter& w) {
    using L = Layout<D>;
    constexpr int S = L::kStages;
    constexpr uint32_t kAB = kBf16 ? 1u : 0u;
    constexpr uint32_t kIdS = ptx::idesc_f16(kAB, 0, 0, kBM, kBN);
    constexpr uint32_t kIdO = ptx::idesc_f16(kAB, 0, 1, kBM, D);
    auto stage_addr = [&](int r) { return sbase + L::kRingOff + (r % S) * L::kTileBytes; };
    auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint64_t qd = ptx::desc_sw128(sbase + L::kQOff + t * L::kTileBytes, 16, 1024);
        const uint64_t kd = ptx::desc_sw128(kaddr, 16, 1024);
        qk_kloop<D>(tmem + L::col_s(t), qd, kd, kIdS);
    };
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint64_t vd = ptx::desc_sw128(vaddr, L::kBlkBytes, 1024);
        pv_kloop(tmem + L::col_o(t), tmem + L::col_s(t), vd, kIdO, acc ? 1u : 0u);
    };
    auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
        return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
    };
    auto wait_ring = [&](int r) { return wait_u(bars.kv_full(r % S), (r / S) & 1, kSiteKvFull); };

    int ring = 0;
    int nq[2] = {0, 0};
    int np[2] = {0, 0};
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<true>(it)) {
        const ItemG g = make_item_gen(p, it);
        const int nmax = max(g.nkv[0], g.nkv[1]);
        if (nmax == 0) continue;
        for (int t = 0; t < 2 && ok; ++t)
            if (g.nkv[t] > 0) ok = wait_u(bars.q_full(t), nq[t] & 1, kSiteQFull);
        if (!ok || !(ok = wait_ring(ring))) break;
        ptx::tc_fence_after();
        for (int t = 0; t < 2; ++t) {
            if (g.nkv[t] == 0) continue;
            issue_qk(t, stage_addr(ring));
            ptx::tc_commit_elect(bars.s_full(t));
            if (g.nkv[t] == 1) ptx::tc_commit_elect(bars.q_empty(t));
        }
        ptx::tc_commit_elect(bars.kv_empty(ring % S));
        int k_ring = ring;
        ++ring;
        for (int j = 0; j < nmax; ++j) {
            const bool more = j + 1 < nmax;
            const int v_ring = ring++;
            if (more) k_ring = ring++;
            // V_j, K_{j+1} and P of the first tile taking part, together.
            const int t0 = j < g.nkv[0] ? 0 : 1;
            const int kr = more ? k_ring : v_ring;
            const uint32_t wb[3] = {bars.kv_full(v_ring % S), bars.kv_full(kr % S), bars.p_full(t0)};
            const uint32_t wp[3] = {static_cast<uint32_t>((v_ring / S) & 1), static_cast<uint32_t>((kr / S) & 1),
                                    static_cast<uint32_t>(np[t0] & 1)};
            if (!(ok = __shfl_sync(0xffffffffu, w.wait_all<3>(wb, wp, kSiteKvFull) ? 1 : 0, 0) != 0)) break;
            const int last_v = j < g.nkv[1] ? 1 : 0;                 // last tile reading V_j
            const int last_k = (more && j + 1 < g.nkv[1]) ? 1 : 0;   // last tile reading K_{j+1}
            for (int t = 0; t < 2; ++t) {
                if (j >= g.nkv[t]) continue;
                if (t != t0 && !(ok = wait_u(bars.p_full(t), np[t] & 1, kSitePFull))) break;
                ++np[t];
                ptx::tc_fence_after();
                issue_pv(t, stage_addr(v_ring), j > 0);
                if (t == last_v) ptx::tc_commit_elect(bars.kv_empty(v_ring % S));
                if (j + 1 < g.nkv[t]) {
                    issue_qk(t, stage_addr(k_ring));
                    ptx::tc_commit_elect(bars.s_full(t));
                    if (j + 2 == g.nkv[t]) ptx::tc_commit_elect(bars.q_empty(t));
                    if (t == last_k) ptx::tc_commit_elect(bars.kv_empty(k_ring % S));
                } else {
                    ptx::tc_commit_elect(bars.o_full(t));
                }
            }
            if (!ok) break;
        }
        for (int t = 0; t < 2; ++t)
            if (g.nkv[t] > 0) ++nq[t];
    }
    ptx::tc_commit_elect(bars.mma_done());
    w.drain(bars.mma_done(), 0);
    __syncwarp();
}

// Hands one row's rescale factor to the correction warpgroup (store, then
// arrive) and returns it as read back from shared memory. The caller makes
// its exponentials depend on the read-back: the arrive feeds nothing else in
// this thread, so the compiler was free to schedule it after the whole
// exponential loop, and did -- the correction warpgroup then started only
// when this warpgroup had finished the step (measured with clock64 traces:
// the factor became visible ~1200 cycles after S instead of ~560, and a
// step took 11% longer). A volatile load is not moved above the arrive.
__device__ __forceinline__ float publish_alpha(float* slot, float alpha, uint32_t bar) {
    *slot = alpha;
    ptx::mbar_arrive(bar);
    return ptx::ld_volatile_shared_f32(ptx::smem_addr(slot));
}

// ---------------------------------------------------------------- softmax

// 32-column TMEM load/store into slice [off, off+32) of a register array;
// `off` is a compile-time constant after unrolling.
template <int N>
__device__ __forceinline__ void ld_slice(uint32_t taddr, uint32_t (&r)[N], int off) {
    if (off == 0) ptx::tmem_ld32_at<0>(taddr, r);
    if constexpr (N > 32) if (off == 32) ptx::tmem_ld32_at<32 % N>(taddr, r);
    if constexpr (N > 64) if (off == 64) ptx::tmem_ld32_at<64 % N>(taddr, r);
    if constexpr (N > 96) if (off == 96) ptx::tmem_ld32_at<96 % N>(taddr, r);
}

template <int N>
__device__ __forceinline__ void st_slice(uint32_t taddr, const uint32_t (&r)[N], int off) {
    if (off == 0) ptx::tmem_st32_at<0>(taddr, r);
    if constexpr (N > 32) if (off == 32) ptx::tmem_st32_at<32 % N>(taddr, r);
    if constexpr (N > 64) if (off == 64) ptx::tmem_st32_at<64 % N>(taddr, r);
    if constexpr (N > 96) if (off == 96) ptx::tmem_st32_at<96 % N>(taddr, r);
}

template <int D, bool kBf16, bool kGen>
__device__ __forceinline__ void softmax_role(const Params& p, uint32_t tmem, uint8_t* smem, const Bars<D>& bars,
                                             const Waiter& w, int t) {
    using L = Layout<D>;
    const int row = threadIdx.x & 127;          // row within the query tile = TMEM lane
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(row & ~31) << 16);
    const uint32_t colS = L::col_s(t);
    float* alpha_buf = reinterpret_cast<float*>(smem + L::kRowOff) + t * kBM;
    float* m_buf = alpha_buf + kNQ * kBM;
    float* l_buf = m_buf + kNQ * kBM;
    const float c = p.scale_log2;
    const uint64_t c2 = ptx::f2_pack(c, c);

    int n_s = 0;       // S tiles consumed (s_full / alpha / p_full phases); bit 30: item parity (general mode)
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<kGen>(it)) {
        int nkv, jmask = 0x7fffffff, kend_row = 0;
        if constexpr (kGen) {
            const ItemG g = make_item_gen(p, it);
            if (t >= g.n_tiles || g.nkv[t] == 0) continue;
            nkv = g.nkv[t];
            jmask = g.jmask[t];
            kend_row = kend_of(p, g.q0 + t * kBM + row);
        } else {
            if (t >= make_item(p, it).n_tiles) continue;
            nkv = p.n_kv_tiles;
        }
        // m and l of the previous item must have been read by the epilogue
        // before this item's last step overwrites them. With two or more
        // steps that is already so: S(t, 1) follows PV(t, 0), which waits
        // for the correction warpgroup's p_full arrival of step 0, which
        // follows its epilogue of the previous item. A one-step item
        // (general mode only: the host sends N = 128 there) waits for the
        // epilogue's stats_free arrival (at once for the first item: a fresh
        // barrier's preceding phase).
        if constexpr (kGen) {
            if (nkv == 1) {
                ok = w.wait(bars.stats_free(t), ((n_s >> 30) & 1) ^ 1, kSiteStats);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
        }
        float m = -INFINITY;  // running row max of the scaled scores, log2 units
        float l = 0.0f;       // running sum of exp2(s*c - m)
        for (int j = 0; j < nkv; ++j, ++n_s) {
            ok = w.wait(bars.s_full(t), n_s & 1, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t s[kBN];
            float m_tile;
            if constexpr (kGen) {
                ptx::tmem_ld32_at<0>(row_addr + colS + 0, s);
                ptx::tmem_ld32_at<32>(row_addr + colS + 32, s);
                ptx::tmem_ld32_at<64>(row_addr + colS + 64, s);
                ptx::tmem_ld32_at<96>(row_addr + colS + 96, s);
                ptx::tmem_wait_ld();
                // Keys at or past kend(row) (the causal diagonal, the end of
                // a ragged key sequence, TMA's zero fill) get -inf.
                if (j >= jmask) {
                    const int lim = kend_row - j * kBN;
#pragma unroll
                    for (int c = 0; c < kBN; ++c) s[c] = c < lim ? s[c] : 0xFF800000u;
                }
                // Row max: eight independent chains of 3-input max, then combine.
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float a = __uint_as_float(s[k]);
#pragma unroll
                    for (int i = 1; i < 15; i += 2)
                        a = ptx::max3(a, __uint_as_float(s[k + 8 * i]), __uint_as_float(s[k + 8 * (i + 1)]));
                    mx[k] = fmaxf(a, __uint_as_float(s[k + 120]));
                }
                m_tile = fmaxf(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], ptx::max3(mx[5], mx[6], mx[7]))) *
                         c;
            } else {
                // Row max from the loads themselves (no masking here).
                float mq[4];
                ptx::tmem_ld32_max_at<0>(row_addr + colS + 0, s, mq[0]);
                ptx::tmem_ld32_max_at<32>(row_addr + colS + 32, s, mq[1]);
                ptx::tmem_ld32_max_at<64>(row_addr + colS + 64, s, mq[2]);
                ptx::tmem_ld32_max_at<96>(row_addr + colS + 96, s, mq[3]);
                ptx::tmem_wait_ld();
                m_tile = fmaxf(ptx::max3(mq[0], mq[1], mq[2]), mq[3]) * c;
            }
            // Hand the correction warpgroup this row's rescale factor
            // (exactly 1 when the max does not move).
            const float m_new = fmaxf(m, m_tile);
            const float alpha = (j == 0 || m_new == m) ? 1.0f : ptx::ex2_approx(m - m_new);
            alpha_buf[row] = alpha;
            ptx::mbar_arrive(bars.alpha_ready(t));
            l *= alpha;
            m = m_new;
            // A row with no allowed key so far keeps m = -inf; exponentiate
            // against 0 then, so its weights are exp2(-inf) = 0.
            const float m_use = (kGen && m == -INFINITY) ? 0.0f : m;

            // P = exp2(S*c - m) on pairs: one packed FMA, two MUFU ex2 (or the
            // FMA-pipe polynomial), one packed add into four partial row sums,
            // one 16-bit pack.
            const uint64_t nm2 = ptx::f2_pack(-m_use, -m_use);
            uint64_t acc[4] = {0, 0, 0, 0};
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int i = 0; i < kBN / 2; ++i) {
                const uint64_t x =
                    ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, nm2);
                // One pair in eight is exponentiated on the FMA pipe, which
                // shortens the MUFU-bound stretch of this loop.
                float p0, p1;
                if (!kGen && (i & 7) == 7) {  // masked -inf keys need the MUFU's exact 0
                    ptx::f2_unpack(ptx::ex2_poly_f2(x), p0, p1);
                } else {
                    float x0, x1;
                    ptx::f2_unpack(x, x0, x1);
                    p0 = ptx::ex2_approx(x0);
                    p1 = ptx::ex2_approx(x1);
                }
                acc[i & 3] = ptx::f2_add(acc[i & 3], ptx::f2_pack(p0, p1));
                pk[i] = ptx::pack2<kBf16>(p0, p1);
            }
            float a0, a1;
            ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), a0, a1);
            l += a0 + a1;
            ptx::tmem_st32_at<0>(row_addr + colS, pk);
            ptx::tmem_st32_at<32>(row_addr + colS + 32, pk);
            if (j + 1 == nkv) {
                m_buf[row] = m;
                l_buf[row] = l;
                ptx::mbar_arrive(bars.stats_ready(t));
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bars.p_full(t));
        }
        if constexpr (kGen) n_s ^= 1 << 30;    // item parity (stats_free phase)
    }
}

// ---------------------------------------------------------------- correction + epilogue

// Stores 32 rows x 64 columns of 16-bit O (hv: the calling lane's row as 32
// packed pairs) through the warp's 4 KB staging slice: each lane writes its
// own row, then the warp reads back so that eight lanes cover one row's 128
// bytes and each store instruction writes four whole 128-byte lines. The 16-
// byte chunk c of row r sits at chunk c ^ (r mod 8) in the slice, so both
// the row-per-lane writes and the transposed reads hit every bank group
// equally. first_row: the output row of the warp's first row in the [rows,
// D] view; col0: the first column; rows_valid: how many of the 32 rows exist
// (a ragged end); rows_total bounds the debug check.
template <int D>
__device__ __forceinline__ void store_o_rows(const uint32_t (&hv)[32], uint32_t wslice, int lane, void* out,
                                             int first_row, int col0, int rows_valid, long long rows_total) {
    __syncwarp();   // the previous call's reads of the slice are done
#pragma unroll
    for (int c = 0; c < 8; ++c)
        ptx::st_shared_v4(wslice + static_cast<uint32_t>(lane) * 128u + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4),
                          hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
    __syncwarp();
    // lane: row 4i + lane / 8 of the 32 (step i), chunk lane % 8
    const int r0 = lane >> 3;
    const uint32_t rd = wslice + static_cast<uint32_t>(r0) * 128u + (static_cast<uint32_t>((lane & 7) ^ r0) << 4);
    uint4* gdst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + static_cast<size_t>(first_row + r0) * D +
                                           col0) + (lane & 7);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // row 4i + lane / 8: its chunk sits at (lane % 8) ^ (row % 8)
        // = (lane % 8) ^ (lane / 8) ^ (4 (i % 2)): odd steps flip bit 2
        const uint4 v = ptx::ld_shared_v4((rd ^ ((i & 1) << 6)) + static_cast<uint32_t>(i) * 512u);
        if (4 * i + r0 < rows_valid && FA2_DBG_OK(first_row + r0 + 4 * i < rows_total, kDbgORow))
            gdst[static_cast<size_t>(4 * i) * (D / 8)] = v;
    }
}

// Shared by the 16-bit and the FP8 kernel (L, BarsT: their shared-memory
// layout and barriers; kFp8: O is also multiplied by the item's V descale and
// the LSE loses the 2^8 the FP8 softmax scales its weights by).
template <class L, class BarsT, int D, bool kBf16, bool kGen, bool kFp8>
__device__ __forceinline__ void correction_role(const Params& p, uint32_t tmem, uint8_t* smem, uint32_t sbase,
                                                const BarsT& bars, const Waiter& w) {
    constexpr int kChunk = 32;        // O is rescaled 32 columns at a time
    constexpr int kHalves = D / 64;   // the epilogue stores 64 columns (128 bytes a row) at a time
    const int q = (threadIdx.x / 32) & 3;      // TMEM lane quarter
    const int lane = threadIdx.x & 31;
    const int row = 32 * q + lane;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const float* rowbuf = reinterpret_cast<const float*>(smem + L::kRowOff);  // alpha | m | l
    // This warp's 32-row slice of the staging buffer (128 bytes a row). The
    // 16-byte chunk c of row r sits at chunk c ^ (r mod 8), so that both the
    // row-per-lane writes and the transposed reads hit every bank group
    // equally (4 wavefronts per 512 bytes, the minimum).
    const uint32_t wslice = sbase + L::kStageOff + static_cast<uint32_t>(q) * (32u * 128u);

    int n_s[2] = {0, 0};
    int n_items[2] = {0, 0};
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<kGen>(it)) {
        // row0: first row of tile 0 in the output view; q0: the same row's
        // index within its head (general mode, for the ragged-end check).
        int n_tiles, nkv[2], row0, q0 = 0, head = 0, grp;
        if constexpr (kGen) {
            const ItemG g = make_item_gen(p, it);
            n_tiles = g.n_tiles;
            nkv[0] = g.nkv[0];
            nkv[1] = g.nkv[1];
            row0 = g.head * p.nq + g.q0;
            q0 = g.q0;
            head = g.head;
            grp = g.kvhead;
        } else {
            const Item item = make_item(p, it);
            n_tiles = item.n_tiles;
            nkv[0] = nkv[1] = p.n_kv_tiles;
            row0 = item.q_row0;
            grp = it / p.pairs;         // the item's (batch, KV head)
        }
        float out_scale = 1.0f;         // O = out_scale * O_acc / l
        if constexpr (kFp8) out_scale = __ldg(p.v_descale + grp);
        const int nmax = max(nkv[0], n_tiles > 1 ? nkv[1] : 0);
        for (int j = 0; j < nmax && ok; ++j) {
            for (int t = 0; t < n_tiles; ++t) {
                if (j >= nkv[t]) continue;
                ok = w.wait(bars.alpha_ready(t), n_s[t] & 1, kSiteAlpha);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ++n_s[t];
                const float alpha = rowbuf[t * kBM + row];
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                    // PV(t, j-1) has completed: the softmax saw S(t, j), whose
                    // commit follows it; PV(t, j) waits for this warpgroup's
                    // p_full arrival below.
                    ptx::tc_fence_after();
                    const uint32_t colO = L::col_o(t);
                    const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
                    for (int h = 0; h < D; h += kChunk) {
                        uint32_t o[kChunk];
                        ptx::tmem_ld32_at<0>(row_addr + colO + h, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < kChunk / 2; ++i) {
                            float o0, o1;
                            ptx::f2_unpack(
                                ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                            a2),
                                o0, o1);
                            o[2 * i] = __float_as_uint(o0);
                            o[2 * i + 1] = __float_as_uint(o1);
                        }
                        ptx::tmem_st32_at<0>(row_addr + colO + h, o);
                    }
                    ptx::tmem_wait_st();
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(bars.p_full(t));
            }
        }
        // Epilogue for each tile of the item: O / l -> 16 bit, stored in
        // whole 128-byte lines through the warp's staging slice; LSE direct.
        // The next item's first PV overwrites O only after this
        // warpgroup's next p_full arrival, which comes after these loads.
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int grow = row0 + t * kBM + row;
            // Rows past a ragged query end are computed but not stored.
            const bool valid = !kGen || q0 + t * kBM + row < p.nq;
            if (kGen && nkv[t] == 0) {
                // No row of this tile may attend any key: O = 0, LSE = -inf.
                if (valid && FA2_DBG_OK(grow < p.rows_q, kDbgORow)) {
                    uint4* z = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + static_cast<size_t>(grow) * D);
#pragma unroll
                    for (int v = 0; v < D / 8; ++v) z[v] = make_uint4(0, 0, 0, 0);
                    p.lse[grow] = -INFINITY;
                }
                continue;
            }
            ok = w.wait(bars.stats_ready(t), n_items[t] & 1, kSiteStats);
            if (ok) ok = w.wait(bars.o_full(t), n_items[t] & 1, kSiteOFull);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            ++n_items[t];
            ptx::tc_fence_after();
            const float m = rowbuf[(2 + t) * kBM + row];
            const float l = rowbuf[(4 + t) * kBM + row];
            if constexpr (kGen) ptx::mbar_arrive(bars.stats_free(t));   // m, l read: may be overwritten
            // l = 0 only for a row with no allowed key: O = 0, LSE = -inf.
            const float inv_l = (!kGen || l > 0.0f) ? out_scale * ptx::rcp_approx(l) : 0.0f;
            const uint32_t colO = L::col_o(t);
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
                // 64 columns -> 32 packed pairs. At d = 128 each 32-column
                // load is converted before the next (fewer live registers:
                // no spills); at d = 64 both loads share one wait.
                uint32_t hv[32];
                if constexpr (D == 128) {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        uint32_t o[32];
                        ptx::tmem_ld32_at<0>(row_addr + colO + 64 * h + 32 * part, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            hv[16 * part + i] = ptx::pack2<kBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                                                  __uint_as_float(o[2 * i + 1]) * inv_l);
                    }
                } else {
                    uint32_t o[64];
                    ptx::tmem_ld32_at<0>(row_addr + colO, o);
                    ptx::tmem_ld32_at<32>(row_addr + colO + 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        hv[i] = ptx::pack2<kBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                                  __uint_as_float(o[2 * i + 1]) * inv_l);
                }
                store_o_rows<D>(hv, wslice, lane, p.o, row0 + t * kBM + 32 * q, 64 * h,
                                kGen ? p.nq - (q0 + t * kBM + 32 * q) : 32, p.rows_q);
            }
            if (!ok) break;
            constexpr float kLog2Off = kFp8 ? 8.0f : 0.0f;
            if (valid && FA2_DBG_OK(grow < p.rows_q, kDbgORow))
                p.lse[grow] = (!kGen || l > 0.0f) ? (m + ptx::lg2_approx(l) - kLog2Off) * 0.69314718055994530942f
                                                  : -INFINITY;
        }
        ptx::tc_fence_before();
    }
}

// ---------------------------------------------------------------- kernel

template <int D, bool kBf16, bool kGen>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const Bars<D> bars{sbase + L::kBarOff};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars.q_full(t), 1);
            ptx::mbar_init(bars.q_empty(t), 1);
            ptx::mbar_init(bars.s_full(t), 1);
            ptx::mbar_init(bars.alpha_ready(t), kBM);
            ptx::mbar_init(bars.stats_ready(t), kBM);
            ptx::mbar_init(bars.stats_free(t), kBM);   // the epilogue's threads have read m, l
            ptx::mbar_init(bars.p_full(t), 2 * kBM);  // softmax + correction warpgroups
            ptx::mbar_init(bars.o_full(t), 1);
        }
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(bars.kv_full(s), 1);
            ptx::mbar_init(bars.kv_empty(s), 1);
        }
        ptx::mbar_init(bars.mma_done(), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kLoadWarp && lane == 0) {
        ptx::tma_prefetch_desc(&tmQ);
        ptx::tma_prefetch_desc(&tmK);
        ptx::tma_prefetch_desc(&tmV);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter w{abort_flag, p.wait_limit_ns};

    if (warp < kCorrWarp0) {
        ptx::setmaxnreg_inc<kRegSoftmax>();
        softmax_role<D, kBf16, kGen>(p, tmem, smem, bars, w, warp / 4);
    } else if (warp < kLoadWarp) {
        ptx::setmaxnreg_dec<kRegCorr>();
        correction_role<L, Bars<D>, D, kBf16, kGen, false>(p, tmem, smem, sbase, bars, w);
    } else {
        ptx::setmaxnreg_dec<kRegOther>();
        if (warp == kLoadWarp) {
            if (lane == 0) {
                if constexpr (kGen)
                    producer_gen<D>(&tmQ, &tmK, &tmV, p, sbase, bars, w);
                else
                    producer<D>(&tmQ, &tmK, &tmV, p, sbase, bars, w);
            }
            __syncwarp();
        } else if (warp == kMmaWarp) {
            if constexpr (kGen)
                mma_issuer_gen<D, kBf16>(p, sbase, tmem, bars, w);
            else
                mma_issuer<D, kBf16>(p, sbase, tmem, bars, w);  // whole warp, one lane issues
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
}


}  // namespace fa2
