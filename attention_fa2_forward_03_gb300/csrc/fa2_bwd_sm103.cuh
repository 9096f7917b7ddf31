// Backward pass of the attention forward (device code). It shares the
// forward's status word, watchdog and PTX wrappers (fa2_fwd_sm103.cuh);
// fa2_fwd_sm103.cu holds the host side.
//
// The forward pages exclude the backward pass ("FlashAttention-2 from
// scratch on Ampere, Part 1", Kernel Specification: forward pass only); the
// forward keeps the per-row logsumexp so the backward can recompute
// P = exp(S - LSE) tile by tile instead of storing it. With D = rowsum(dO o O):
//     dP = dO V^T, dS = P o (dP - D), dV = P^T dO, dK = scale dS^T Q,
//     dQ = scale dS K.
// Three kernels, all on one stream, none using atomics:
//   fa2_bwd_delta_kernel  D for every query row (memory bound)
//   fa2_bwd_dkdv_kernel   persistent, one 128-key tile at a time:
//                         S^T = K Q^T and dP^T = V dO^T (keys in TMEM
//                         lanes), P^T and dS^T
//                         formed by the elementwise warps and written back
//                         to TMEM as 16-bit, then dV += P^T dO and
//                         dK += dS^T Q as MMAs with A from TMEM; dK and dV
//                         accumulate over every query tile (and every query
//                         head of a KV head) in TMEM
//   fa2_bwd_dq_kernel     persistent, one 128-query tile at a time:
//                         S = Q K^T, dP = dO V^T, dS in TMEM, dQ += dS K
// Warps 0-7 elementwise (warp w: TMEM lanes 32 (w % 4) .. + 31, one row per
// thread, columns 64 (w / 4) .. + 63 of the tile, so two warps per scheduler
// hide each other's latency), warp 8 TMA producer, warp 9 TMEM allocator and
// MMA issuer. Each half's 16-bit results (P^T, dS^T, dS) are packed into the
// first 32 of its own 64 fp32 columns -- never into the other warp's, which
// may not have been read yet -- and the MMAs read A in those two halves.
// TMEM: S | dP | two d-column accumulators (dK/dV), S0 | S1 | dP | dQ (dQ).
//
// Overlap. The elementwise step of a tile runs in two phases with their own
// barriers: P as soon as S is in TMEM (while the tensor core computes dP),
// then dS once dP is (while the tensor core runs the first product that
// consumes P). dK/dV issues S, dP, dV (after P), dK (after dS) per query
// tile; dQ double-buffers S, so S of the next key tile is computed during
// the current tile's elementwise work whenever its K/V stage has arrived.
#pragma once

#include "fa2_fwd_sm103.cuh"

namespace fa2 {
namespace bwd {

constexpr int kEwThreads = 256;   // warps 0-7
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;

struct Params {
    const void* o;        // forward output [rows, D]
    const float* lse;     // forward logsumexp [rows]
    const void* dout;     // upstream gradient [rows, D]
    float* delta;         // D = rowsum(dO o O) [rows]
    void* dq;             // [B*Hq*N, D]
    void* dk;             // [B*Hkv*N, D]
    void* dv;             // [B*Hkv*N, D]
    long long wait_limit_ns;
    int debug_flags;      // watchdog test hook: bit 0 skips the dK/dV kernel's query-tile loads
    int n;                // N: rows per head (any positive length)
    int n_tiles;          // ceil(N / 128)
    int hq, group;        // Hq, Hq / Hkv
    int causal;
    float scale;          // softmax scale
    float scale_log2;     // scale * log2(e)
    // Extents for the debug build's checks.
    int heads_q, heads_kv;        // B * Hq, B * Hkv
    long long rows_q, rows_kv;    // B * Hq * N, B * Hkv * N
};

// ---------------------------------------------------------------- D = rowsum(dO o O)

// 16 lanes per row, each one 16-byte chunk of dO and O (d = 128) or one
// 8-byte... the row is split into 16 equal 16-bit runs.
template <int D, bool kBf16>
__global__ void __launch_bounds__(256) fa2_bwd_delta_kernel(const void* o, const void* dout, float* delta,
                                                            long long rows) {
    constexpr int kPer = D / 16;  // 16-bit values per lane
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 16;
    const int part = threadIdx.x & 15;
    float acc = 0.0f;
    if (row < rows) {
        const uint16_t* op = static_cast<const uint16_t*>(o) + row * D + part * kPer;
        const uint16_t* dp = static_cast<const uint16_t*>(dout) + row * D + part * kPer;
        uint32_t ov[kPer / 2], dv[kPer / 2];
        if constexpr (kPer == 8) {
            const uint4 a = *reinterpret_cast<const uint4*>(op);
            const uint4 b = *reinterpret_cast<const uint4*>(dp);
            ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
            dv[0] = b.x; dv[1] = b.y; dv[2] = b.z; dv[3] = b.w;
        } else {
            const uint2 a = *reinterpret_cast<const uint2*>(op);
            const uint2 b = *reinterpret_cast<const uint2*>(dp);
            ov[0] = a.x; ov[1] = a.y;
            dv[0] = b.x; dv[1] = b.y;
        }
#pragma unroll
        for (int i = 0; i < kPer / 2; ++i) {
            float o0, o1, d0, d1;
            ptx::unpack2<kBf16>(ov[i], o0, o1);
            ptx::unpack2<kBf16>(dv[i], d0, d1);
            acc = fmaf(o0, d0, acc);
            acc = fmaf(o1, d1, acc);
        }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) delta[row] = acc;
}

// ---------------------------------------------------------------- shared pieces

__device__ __forceinline__ void store_row_16(void* base, long long row, int d, int col0, const uint32_t (&h)[16]) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + row * d + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
}

// Write columns [c0, c1) of a d-column fp32 TMEM accumulator row (times
// `mul`) as 16-bit; `store` false skips the global stores (a row past a
// ragged end). The whole warp must call this together: the TMEM loads are
// warp-collective (.sync.aligned) and may not sit in a divergent branch.
template <int D, bool kBf16>
__device__ __forceinline__ void store_acc_row(uint32_t row_addr, uint32_t col, float mul, void* out,
                                              long long grow, long long rows, int c0, int c1, bool store) {
    if ((c1 - c0) % 64 == 0) {   // warp-uniform: 64 columns per TMEM wait (half the round trips)
#pragma unroll 1
        for (int cc = c0; cc < c1; cc += 64) {
            uint32_t a[64];
            ptx::tmem_ld32_at<0>(row_addr + col + cc, a);
            ptx::tmem_ld32_at<32>(row_addr + col + cc + 32, a);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h[i] = ptx::pack2<kBf16>(__uint_as_float(a[32 * half + 2 * i]) * mul,
                                             __uint_as_float(a[32 * half + 2 * i + 1]) * mul);
                if (store && FA2_DBG_OK(grow < rows, kDbgBwdRow)) store_row_16(out, grow, D, cc + 32 * half, h);
            }
        }
        return;
    }
#pragma unroll 1
    for (int cc = c0; cc < c1; cc += 32) {
        uint32_t a[32];
        ptx::tmem_ld32(row_addr + col + cc, a);
        ptx::tmem_wait_ld();
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            h[i] = ptx::pack2<kBf16>(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
        if (store && FA2_DBG_OK(grow < rows, kDbgBwdRow)) store_row_16(out, grow, D, cc, h);
    }
}

// ---------------------------------------------------------------- dK, dV


// dK/dV kernel layout: K and V of the current key tile, then separate rings
// for the query tiles (3 stages: Q(n) is read by S^T(n), issued as early as
// mid-step n-1, and by dK(n) at the end of step n) and the upstream-gradient
// tiles (2 stages: dO(n) is read by dP^T(n) and dV(n) only). LSE and D are
// read by the elementwise warps from global memory, one step ahead.
template <int D>
struct DkdvLayout {
    static constexpr int kBlkBytes = 128 * 128;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kQStages = 3, kDoStages = 2;
    static constexpr int kFixedOff = 0;                               // K | V
    static constexpr int kQOff = 2 * kTileBytes;
    static constexpr int kDoOff = kQOff + kQStages * kTileBytes;
    static constexpr int kBarOff = kDoOff + kDoStages * kTileBytes;
    // fixed_full, q_full[3], q_empty[3], do_full[2], do_empty[2], s_full, dp_full, p_full, ds_full, acc_full,
    // fixed_empty
    static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDoStages + 6;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
};

struct DkdvBars {
    uint32_t base;
    static constexpr int QS = 3, DS = 2;
    __device__ uint32_t fixed_full() const { return base; }
    __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
    __device__ uint32_t q_empty(int s) const { return base + 8 * (1 + QS + s); }
    __device__ uint32_t do_full(int s) const { return base + 8 * (1 + 2 * QS + s); }
    __device__ uint32_t do_empty(int s) const { return base + 8 * (1 + 2 * QS + DS + s); }
    __device__ uint32_t s_full() const { return base + 8 * (1 + 2 * QS + 2 * DS); }
    __device__ uint32_t dp_full() const { return base + 8 * (2 + 2 * QS + 2 * DS); }
    __device__ uint32_t p_full() const { return base + 8 * (3 + 2 * QS + 2 * DS); }
    __device__ uint32_t ds_full() const { return base + 8 * (4 + 2 * QS + 2 * DS); }
    __device__ uint32_t acc_full() const { return base + 8 * (5 + 2 * QS + 2 * DS); }
    __device__ uint32_t fixed_empty() const { return base + 8 * (6 + 2 * QS + 2 * DS); }
};

// The 128-row tiles of a persistent backward CTA (key tiles for dK/dV, query
// tiles for dQ), `heads` heads of n_tiles tiles each. Without the mask every
// tile costs the same (n_tiles steps per head of work), so CTA c takes tiles
// c, c + grid, c + 2 grid, ... in (head, tile) order: the CTAs running at one
// time share few heads, whose operands stay in L2. With the causal mask tile
// m costs n_tiles - m (dK/dV) or m + 1 (dQ) steps, so tiles are taken in pairs
// (m, n_tiles - 1 - m) of equal total cost n_tiles + 1, pair index u = c,
// c + grid, ...; the middle tile of an odd count is a pair alone. Returns 0
// past the last tile, 1 for a tile (tile, head), 2 for the empty second half
// of a lone middle tile (skipped by every role alike).
__device__ __forceinline__ int bwd_tile(int causal, int n_tiles, int heads, int slot, int& tile, int& head) {
    if (!causal) {
        const long long t = blockIdx.x + static_cast<long long>(slot) * gridDim.x;
        if (t >= static_cast<long long>(n_tiles) * heads) return 0;
        head = static_cast<int>(t / n_tiles);
        tile = static_cast<int>(t % n_tiles);
        return 1;
    }
    const int half = (n_tiles + 1) / 2;
    const long long u = blockIdx.x + static_cast<long long>(slot >> 1) * gridDim.x;
    if (u >= static_cast<long long>(half) * heads) return 0;
    head = static_cast<int>(u / half);
    const int m = static_cast<int>(u % half);
    tile = (slot & 1) ? n_tiles - 1 - m : m;
    return ((slot & 1) && tile == m) ? 2 : 1;
}

// Persistent: one CTA per SM walks its key tiles (bwd_tile). Per key tile
// the roles run as before; across tiles the K/V buffer is reloaded once the
// previous tile's last S^T and dP^T have read it (fixed_empty), the
// step-indexed barriers and the Q/dO rings keep counting, and the next tile's
// first products (S^T, dP^T) run on the tensor core while the elementwise
// warps store the previous tile's dK and dV. The first dV of a tile, which
// overwrites the accumulator, waits for that tile's first P^T, which the
// elementwise warps publish only after their accumulator loads.
template <int D, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        const Params p) {
    using L = DkdvLayout<D>;
    constexpr int QS = L::kQStages, DS = L::kDoStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const DkdvBars bars{sbase + L::kBarOff};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int heads_per_batch = p.hq / p.group;   // KV heads per batch

    if (threadIdx.x == 0) {
        ptx::mbar_init(bars.fixed_full(), 1);
        ptx::mbar_init(bars.fixed_empty(), 1);
        for (int s = 0; s < QS; ++s) {
            ptx::mbar_init(bars.q_full(s), 1);
            ptx::mbar_init(bars.q_empty(s), 1);
        }
        for (int s = 0; s < DS; ++s) {
            ptx::mbar_init(bars.do_full(s), 1);
            ptx::mbar_init(bars.do_empty(s), 1);
        }
        ptx::mbar_init(bars.s_full(), 1);
        ptx::mbar_init(bars.dp_full(), 1);
        ptx::mbar_init(bars.p_full(), kEwThreads);
        ptx::mbar_init(bars.ds_full(), kEwThreads);
        ptx::mbar_init(bars.acc_full(), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter w{abort_flag, p.wait_limit_ns};
    // Ring stage of global step n (steps count across this CTA's tiles).
    auto q_addr = [&](int n) { return sbase + L::kQOff + (n % QS) * L::kTileBytes; };
    auto do_addr = [&](int n) { return sbase + L::kDoOff + (n % DS) * L::kTileBytes; };
    // Per key tile: its query steps run over the group's query heads in
    // turn, query tiles first .. n_tiles - 1 of each (tensor maps are
    // [heads, N, d]: a tile never crosses heads, rows past N read as zero).
    auto first_of = [&](int kt) { return p.causal ? kt : 0; };
    auto steps_of = [&](int kt) { return p.group * (p.n_tiles - first_of(kt)); };
    auto q_head = [&](int kvh, int g) {
        const int b = kvh / heads_per_batch;
        return b * p.hq + (kvh - b * heads_per_batch) * p.group + g;
    };

    if (warp == kLoadWarp) {
        if (lane == 0) {
            int nq = 0, nd = 0, nf = 0;   // Q, dO and K/V tiles issued
            const bool load_q = (p.debug_flags & 1) == 0;
            bool ok = true;
            int kt, kvh;
            for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_kv, slot, kt, kvh)) != 0; ++slot) {
                if (r == 2) continue;
                // K and V of this tile, once the previous tile's last S^T and dP^T have read theirs
                if (!(ok = w.wait(bars.fixed_empty(), (nf & 1) ^ 1, kSiteKvEmpty))) break;
                ptx::mbar_arrive_expect_tx(bars.fixed_full(), 2 * L::kTileBytes);
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk) {
                    if (!FA2_DBG_OK(kvh < p.heads_kv && kt * 128 < p.n, kDbgKvTile)) break;
                    ptx::tma_load_3d(sbase + L::kFixedOff + blk * L::kBlkBytes, &tmK, blk * 64, kt * 128, kvh,
                                     bars.fixed_full());
                    ptx::tma_load_3d(sbase + L::kFixedOff + L::kTileBytes + blk * L::kBlkBytes, &tmV, blk * 64,
                                     kt * 128, kvh, bars.fixed_full());
                }
                ++nf;
                const int first = first_of(kt), steps = steps_of(kt);
                int g = 0, i = first;
                for (int n = 0; n < steps && ok; ++n) {
                    const int qh = q_head(kvh, g);
                    if (!(ok = w.wait(bars.q_empty(nq % QS), ((nq / QS) & 1) ^ 1, kSiteKvEmpty))) break;
                    ptx::mbar_arrive_expect_tx(bars.q_full(nq % QS), L::kTileBytes);
                    if (load_q && FA2_DBG_OK(qh < p.heads_q && i * 128 < p.n, kDbgQTile))
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            ptx::tma_load_3d(q_addr(nq) + blk * L::kBlkBytes, &tmQ, blk * 64, i * 128, qh,
                                             bars.q_full(nq % QS));
                    ++nq;
                    if (!(ok = w.wait(bars.do_empty(nd % DS), ((nd / DS) & 1) ^ 1, kSiteKvEmpty))) break;
                    ptx::mbar_arrive_expect_tx(bars.do_full(nd % DS), L::kTileBytes);
                    if (FA2_DBG_OK(qh < p.heads_q && i * 128 < p.n, kDbgQTile))
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            ptx::tma_load_3d(do_addr(nd) + blk * L::kBlkBytes, &tmDO, blk * 64, i * 128, qh,
                                             bars.do_full(nd % DS));
                    ++nd;
                    if (++i == p.n_tiles) {
                        i = first;
                        ++g;
                    }
                }
            }
            if (!ok) {
                // let every copy this CTA started land before it exits
                for (int r2 = nq > QS ? nq - QS : 0; r2 < nq; ++r2) w.drain(bars.q_full(r2 % QS), (r2 / QS) & 1);
                for (int r2 = nd > DS ? nd - DS : 0; r2 < nd; ++r2) w.drain(bars.do_full(r2 % DS), (r2 / DS) & 1);
            }
            if (nf > 0) w.drain(bars.fixed_full(), (nf - 1) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t kAB = kBf16 ? 1u : 0u;
        constexpr uint32_t kIdT = ptx::idesc_f16(kAB, 0, 0, 128, 128);  // S^T, dP^T: both K-major
        constexpr uint32_t kIdA = ptx::idesc_f16(kAB, 0, 1, 128, D);    // dV, dK: B MN-major
        auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
            return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
        };
        const uint64_t kdesc = ptx::desc_sw128(sbase + L::kFixedOff, 16, 1024);
        const uint64_t vdesc = ptx::desc_sw128(sbase + L::kFixedOff + L::kTileBytes, 16, 1024);
        auto issue_s = [&](int n) {   // S^T of global step n, once Q(n) has landed
            qk_kloop<D>(tmem + L::kColS, kdesc, ptx::desc_sw128(q_addr(n), 16, 1024), kIdT);
            ptx::tc_commit_elect(bars.s_full());
        };
        int nb = 0;     // global steps of the tiles before this one
        int nf = 0;     // tiles started
        bool ok = true;
        int kt, kvh;
        for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_kv, slot, kt, kvh)) != 0; ++slot) {
            if (r == 2) continue;
            const int steps = steps_of(kt);
            ok = wait_u(bars.fixed_full(), nf & 1, kSiteQFull);
            ++nf;
            if (ok) ok = wait_u(bars.q_full(nb % QS), (nb / QS) & 1, kSiteKvFull);
            if (ok) {
                ptx::tc_fence_after();
                issue_s(nb);
            }
            int s_issued = 1;       // steps of this tile whose S^T has been issued
            bool do_seen = false;   // dO(n) observed landed while waiting for dS^T(n-1)
            for (int n = 0; n < steps && ok; ++n) {
                const int ng = nb + n;
                // dP^T = V dO(n)^T
                if (!do_seen && !(ok = wait_u(bars.do_full(ng % DS), (ng / DS) & 1, kSiteKvFull))) break;
                ptx::tc_fence_after();
                qk_kloop<D>(tmem + L::kColDP, vdesc, ptx::desc_sw128(do_addr(ng), 16, 1024), kIdT);
                ptx::tc_commit_elect(bars.dp_full());
                // the tile's K and V are read for the last time by now-issued products
                if (n + 1 == steps) ptx::tc_commit_elect(bars.fixed_empty());
                // dV += P^T dO as soon as P^T is in TMEM (16-bit over the S
                // columns; dO as the MN-major B operand); dO(n) is then free
                if (!(ok = wait_u(bars.p_full(), ng & 1, kSitePFull))) break;
                ptx::tc_fence_after();
                ptx::mma_ts_kloop8_split(tmem + L::kColAcc0, tmem + L::kColS,
                                         ptx::desc_sw128(do_addr(ng), L::kBlkBytes, 1024), kIdA, n > 0 ? 1u : 0u);
                ptx::tc_commit_elect(bars.do_empty(ng % DS));
                // S^T of the next step if Q(n+1) is here (it overwrites P^T(n)
                // only after dV has read it: in order), so the elementwise warps
                // go from dS^T(n) straight to P^T(n+1)
                if (s_issued == n + 1 && n + 1 < steps) {
                    const uint32_t bar = bars.q_full((ng + 1) % QS);
                    const uint32_t par = ((ng + 1) / QS) & 1;
                    if (__shfl_sync(0xffffffffu, ptx::mbar_test_wait(bar, par) ? 1 : 0, 0)) {
                        ptx::tc_fence_after();
                        issue_s(ng + 1);
                        ++s_issued;
                    }
                }
                // dK += dS^T Q once dS^T is; Q(n) is then free. The wait also
                // tests whether dO(n+1) has landed, so that the next step's
                // dP^T needs no separate wait.
                do_seen = n + 1 >= steps;
                ok = __shfl_sync(0xffffffffu,
                                 w.wait_and_test(bars.ds_full(), ng & 1, kSitePFull, bars.do_full((ng + 1) % DS),
                                                 ((ng + 1) / DS) & 1, do_seen) ? 1 : 0, 0) != 0;
                do_seen = __all_sync(0xffffffffu, do_seen);
                if (!ok) break;
                ptx::tc_fence_after();
                ptx::mma_ts_kloop8_split(tmem + L::kColAcc1, tmem + L::kColDP,
                                         ptx::desc_sw128(q_addr(ng), L::kBlkBytes, 1024), kIdA, n > 0 ? 1u : 0u);
                ptx::tc_commit_elect(bars.q_empty(ng % QS));
                if (s_issued == n + 1 && n + 1 < steps) {
                    if (!(ok = wait_u(bars.q_full((ng + 1) % QS), ((ng + 1) / QS) & 1, kSiteKvFull))) break;
                    ptx::tc_fence_after();
                    issue_s(ng + 1);
                    ++s_issued;
                }
            }
            // dK and dV of this tile are complete once every product above is
            // (committed on an abort too: the drain below waits for it)
            ptx::tc_commit_elect(bars.acc_full());
            nb += steps;
        }
        // every product must finish before the CTA frees its TMEM
        if (nf > 0) w.drain(bars.acc_full(), (nf - 1) & 1);
        __syncwarp();
    } else {
        // elementwise: thread = key row of the tile = TMEM lane; columns
        // (query rows) [c0, c0 + 64)
        const int row = 32 * (warp & 3) + lane;
        const int c0 = 64 * (warp >> 2);
        const uint32_t row_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        const float c = p.scale_log2;
        constexpr float kLog2e = 1.4426950408889634f;
        // This warp's 64 query columns of a step: lane x holds -LSE log2 e
        // and D of columns c0 + x and c0 + 32 + x (from global memory, one
        // step ahead); the loops take them by shuffle. A query past N (a
        // ragged last tile) gets -LSE = -inf and D = 0: its P^T and dS^T
        // columns are exactly 0.
        float nl_nx[2] = {0.0f, 0.0f}, d_nx[2] = {0.0f, 0.0f};
        int nb = 0;   // global steps of the tiles before this one
        int nf = 0;   // tiles done
        bool ok = true;
        int kt, kvh;
        for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_kv, slot, kt, kvh)) != 0; ++slot) {
            if (r == 2) continue;
            const int first = first_of(kt), steps = steps_of(kt);
            auto fetch = [&](int gg, int ii) {
                const long long base = static_cast<long long>(q_head(kvh, gg)) * p.n;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int q = ii * 128 + c0 + 32 * h + lane;
                    const bool in = q < p.n && FA2_DBG_OK(base + q < p.rows_q, kDbgBwdRow);
                    nl_nx[h] = in ? -__ldg(p.lse + base + q) * kLog2e : -INFINITY;
                    d_nx[h] = in ? __ldg(p.delta + base + q) : 0.0f;
                }
            };
            int g = 0, qi = first;
            fetch(g, qi);
            for (int n = 0; n < steps; ++n) {
                const int ng = nb + n;
                const float l2v[2] = {nl_nx[0], nl_nx[1]};
                const float dv2[2] = {d_nx[0], d_nx[1]};
                const bool diag = p.causal && qi == kt;  // query q may see key k only if q >= k
                if (++qi == p.n_tiles) {
                    qi = first;
                    ++g;
                }
                if (n + 1 < steps) fetch(g, qi);
                ok = w.wait(bars.s_full(), ng & 1, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // P phase: P^T = exp2(S^T c - LSE log2 e) -> 16-bit over S^T
                float pf[64];
                {
                    uint32_t sv[64];
                    ptx::tmem_ld32_at<0>(row_addr + L::kColS + c0, sv);
                    ptx::tmem_ld32_at<32>(row_addr + L::kColS + c0 + 32, sv);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float nl = __shfl_sync(0xffffffffu, l2v[j / 32], j % 32);
                        pf[j] = ptx::ex2_approx(fmaf(__uint_as_float(sv[j]), c, nl));
                    }
                }
                if (diag) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) pf[j] = c0 + j < row ? 0.0f : pf[j];
                }
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) pk[x] = ptx::pack2<kBf16>(pf[cc + 2 * x], pf[cc + 2 * x + 1]);
                    ptx::tmem_st16(row_addr + L::kColS + c0 + cc / 2, pk);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bars.p_full());
                // dS phase: dS^T = P^T o (dP^T - D) -> 16-bit over dP^T
                ok = w.wait(bars.dp_full(), ng & 1, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                {
                    uint32_t dp[64];
                    ptx::tmem_ld32_at<0>(row_addr + L::kColDP + c0, dp);
                    ptx::tmem_ld32_at<32>(row_addr + L::kColDP + c0 + 32, dp);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 32) {
                        uint32_t dk[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int j = cc + 2 * x;
                            const float d0 = __shfl_sync(0xffffffffu, dv2[cc / 32], 2 * x);
                            const float d1 = __shfl_sync(0xffffffffu, dv2[cc / 32], 2 * x + 1);
                            dk[x] = ptx::pack2<kBf16>(pf[j] * (__uint_as_float(dp[j]) - d0),
                                                      pf[j + 1] * (__uint_as_float(dp[j + 1]) - d1));
                        }
                        ptx::tmem_st16(row_addr + L::kColDP + c0 + cc / 2, dk);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bars.ds_full());
            }
            if (!ok) break;
            ok = w.wait(bars.acc_full(), nf & 1, kSiteOFull);
            ++nf;
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // key rows past N (a ragged last tile) are not stored
            const long long grow = static_cast<long long>(kvh) * p.n + kt * 128 + row;
            const bool valid = kt * 128 + row < p.n;
            if (c0 == 0)   // warp-uniform: warps 0-3 write dV, warps 4-7 dK
                store_acc_row<D, kBf16>(row_addr, L::kColAcc0, 1.0f, p.dv, grow, p.rows_kv, 0, D, valid);
            else
                store_acc_row<D, kBf16>(row_addr, L::kColAcc1, p.scale, p.dk, grow, p.rows_kv, 0, D, valid);
            // the accumulator loads are complete (store_acc_row waits for
            // each); order them before the next tile's P^T arrival, which
            // lets the first dV of that tile overwrite the accumulator
            ptx::tc_fence_before();
            nb += steps;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dQ

// dQ kernel layout: Q and dO of the current query tile, then separate rings
// for the key tiles (3 stages: K(j) is read by S(j), issued as early as
// mid-step j-1, and by dQ(j)) and the value tiles (2 stages: V(j) is read by
// dP(j) only).
template <int D>
struct DqLayout {
    static constexpr int kBlkBytes = 128 * 128;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr int kFixedOff = 0;                               // Q | dO
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    // fixed_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], dp_full, ds_full, acc_full,
    // fixed_empty
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 6;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    // TMEM: S0 | S1 | dP | dQ
    static constexpr uint32_t kColS0 = 0, kColDP = 256, kColAcc = 384;
};

struct DqBars {
    uint32_t base;
    static constexpr int KS = 3, VS = 2;
    __device__ uint32_t fixed_full() const { return base; }
    __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
    __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + KS + s); }
    __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * KS + s); }
    __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 2 * KS + VS + s); }
    __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 2 * KS + 2 * VS + b); }
    __device__ uint32_t dp_full() const { return base + 8 * (3 + 2 * KS + 2 * VS); }
    __device__ uint32_t ds_full() const { return base + 8 * (4 + 2 * KS + 2 * VS); }
    __device__ uint32_t acc_full() const { return base + 8 * (5 + 2 * KS + 2 * VS); }
    __device__ uint32_t fixed_empty() const { return base + 8 * (6 + 2 * KS + 2 * VS); }
};

// Persistent like the dK/dV kernel: one CTA per SM walks its query tiles
// (bwd_tile over the B * H_q query heads). Q and dO of the next tile load
// once the current tile's last S and dP have read the buffer; the step
// barriers (S double-buffered by global step parity) and the K/V rings count
// across tiles; the next tile's first dQ, which overwrites the accumulator,
// waits for its first dS, published after the previous tile's dQ loads.
template <int D, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      const Params p) {
    using L = DqLayout<D>;
    constexpr int KS = L::kKStages, VS = L::kVStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const DqBars bars{sbase + L::kBarOff};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    // KV head of query head qh (b * Hq + query head)
    auto kvh_of = [&](int qh) {
        const int b = qh / p.hq;
        return b * (p.hq / p.group) + (qh - b * p.hq) / p.group;
    };
    auto steps_of = [&](int qt) { return p.causal ? qt + 1 : p.n_tiles; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bars.fixed_full(), 1);
        ptx::mbar_init(bars.fixed_empty(), 1);
        for (int s = 0; s < KS; ++s) {
            ptx::mbar_init(bars.k_full(s), 1);
            ptx::mbar_init(bars.k_empty(s), 1);
        }
        for (int s = 0; s < VS; ++s) {
            ptx::mbar_init(bars.v_full(s), 1);
            ptx::mbar_init(bars.v_empty(s), 1);
        }
        ptx::mbar_init(bars.s_full(0), 1);
        ptx::mbar_init(bars.s_full(1), 1);
        ptx::mbar_init(bars.dp_full(), 1);
        ptx::mbar_init(bars.ds_full(), kEwThreads);
        ptx::mbar_init(bars.acc_full(), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter w{abort_flag, p.wait_limit_ns};
    // Ring stage of global step n (steps count across this CTA's tiles).
    auto k_addr = [&](int n) { return sbase + L::kKOff + (n % KS) * L::kTileBytes; };
    auto v_addr = [&](int n) { return sbase + L::kVOff + (n % VS) * L::kTileBytes; };

    if (warp == kLoadWarp) {
        if (lane == 0) {
            int nk = 0, nv = 0, nf = 0;   // K, V and Q/dO tiles issued
            bool ok = true;
            int qt, qh;
            for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_q, slot, qt, qh)) != 0; ++slot) {
                if (r == 2) continue;
                // Q and dO of this tile, once the previous tile's last S and dP have read theirs
                if (!(ok = w.wait(bars.fixed_empty(), (nf & 1) ^ 1, kSiteKvEmpty))) break;
                ptx::mbar_arrive_expect_tx(bars.fixed_full(), 2 * L::kTileBytes);
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk) {
                    if (!FA2_DBG_OK(qh < p.heads_q && qt * 128 < p.n, kDbgQTile)) break;
                    ptx::tma_load_3d(sbase + L::kFixedOff + blk * L::kBlkBytes, &tmQ, blk * 64, qt * 128, qh,
                                     bars.fixed_full());
                    ptx::tma_load_3d(sbase + L::kFixedOff + L::kTileBytes + blk * L::kBlkBytes, &tmDO, blk * 64,
                                     qt * 128, qh, bars.fixed_full());
                }
                ++nf;
                const int kvh = kvh_of(qh), steps = steps_of(qt);
                for (int n = 0; n < steps && ok; ++n) {
                    if (!(ok = w.wait(bars.k_empty(nk % KS), ((nk / KS) & 1) ^ 1, kSiteKvEmpty))) break;
                    ptx::mbar_arrive_expect_tx(bars.k_full(nk % KS), L::kTileBytes);
                    if (FA2_DBG_OK(kvh < p.heads_kv && n * 128 < p.n, kDbgKvTile))
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            ptx::tma_load_3d(k_addr(nk) + blk * L::kBlkBytes, &tmK, blk * 64, n * 128, kvh,
                                             bars.k_full(nk % KS));
                    ++nk;
                    if (!(ok = w.wait(bars.v_empty(nv % VS), ((nv / VS) & 1) ^ 1, kSiteKvEmpty))) break;
                    ptx::mbar_arrive_expect_tx(bars.v_full(nv % VS), L::kTileBytes);
                    if (FA2_DBG_OK(kvh < p.heads_kv && n * 128 < p.n, kDbgKvTile))
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            ptx::tma_load_3d(v_addr(nv) + blk * L::kBlkBytes, &tmV, blk * 64, n * 128, kvh,
                                             bars.v_full(nv % VS));
                    ++nv;
                }
            }
            if (!ok) {
                for (int r2 = nk > KS ? nk - KS : 0; r2 < nk; ++r2) w.drain(bars.k_full(r2 % KS), (r2 / KS) & 1);
                for (int r2 = nv > VS ? nv - VS : 0; r2 < nv; ++r2) w.drain(bars.v_full(r2 % VS), (r2 / VS) & 1);
            }
            if (nf > 0) w.drain(bars.fixed_full(), (nf - 1) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t kAB = kBf16 ? 1u : 0u;
        constexpr uint32_t kIdS = ptx::idesc_f16(kAB, 0, 0, 128, 128);  // S, dP: both K-major
        constexpr uint32_t kIdQ = ptx::idesc_f16(kAB, 0, 1, 128, D);    // dQ += dS K: K MN-major
        auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
            return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
        };
        const uint64_t qdesc = ptx::desc_sw128(sbase + L::kFixedOff, 16, 1024);
        const uint64_t dodesc = ptx::desc_sw128(sbase + L::kFixedOff + L::kTileBytes, 16, 1024);
        // S of global step n into buffer n % 2, once K(n) has landed
        auto issue_s = [&](int n) {
            qk_kloop<D>(tmem + L::kColS0 + 128u * (n & 1), qdesc, ptx::desc_sw128(k_addr(n), 16, 1024), kIdS);
            ptx::tc_commit_elect(bars.s_full(n & 1));
        };
        int nb = 0;     // global steps of the tiles before this one
        int nf = 0;     // tiles started
        bool ok = true;
        int qt, qh;
        for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_q, slot, qt, qh)) != 0; ++slot) {
            if (r == 2) continue;
            const int steps = steps_of(qt);
            ok = wait_u(bars.fixed_full(), nf & 1, kSiteQFull);
            ++nf;
            if (ok) ok = wait_u(bars.k_full(nb % KS), (nb / KS) & 1, kSiteKvFull);
            if (ok) {
                ptx::tc_fence_after();
                issue_s(nb);
            }
            int s_issued = 1;      // steps of this tile whose S has been issued
            bool v_seen = false;   // V(n) observed landed while waiting for dS(n-1)
            for (int n = 0; n < steps && ok; ++n) {
                const int ng = nb + n;
                // dP = dO V(n)^T; V(n) is then free
                if (!v_seen && !(ok = wait_u(bars.v_full(ng % VS), (ng / VS) & 1, kSiteKvFull))) break;
                ptx::tc_fence_after();
                qk_kloop<D>(tmem + L::kColDP, dodesc, ptx::desc_sw128(v_addr(ng), 16, 1024), kIdS);
                ptx::tc_commit_elect(bars.dp_full());
                ptx::tc_commit_elect(bars.v_empty(ng % VS));
                // the tile's Q and dO are read for the last time by now-issued products
                if (n + 1 == steps) ptx::tc_commit_elect(bars.fixed_empty());
                // S of the next key tile now if K(n+1) is here, so it is ready
                // when the elementwise warps finish this tile
                if (s_issued == n + 1 && n + 1 < steps) {
                    const uint32_t bar = bars.k_full((ng + 1) % KS);
                    const uint32_t par = ((ng + 1) / KS) & 1;
                    if (__shfl_sync(0xffffffffu, ptx::mbar_test_wait(bar, par) ? 1 : 0, 0)) {
                        ptx::tc_fence_after();
                        issue_s(ng + 1);
                        ++s_issued;
                    }
                }
                // dQ += dS K once dS is in TMEM (16-bit over the dP columns; K as
                // the MN-major B operand); K(n) is then free. The wait also tests
                // whether V(n+1) has landed (see the dK/dV kernel).
                v_seen = n + 1 >= steps;
                ok = __shfl_sync(0xffffffffu,
                                 w.wait_and_test(bars.ds_full(), ng & 1, kSitePFull, bars.v_full((ng + 1) % VS),
                                                 ((ng + 1) / VS) & 1, v_seen) ? 1 : 0, 0) != 0;
                v_seen = __all_sync(0xffffffffu, v_seen);
                if (!ok) break;
                ptx::tc_fence_after();
                ptx::mma_ts_kloop8_split(tmem + L::kColAcc, tmem + L::kColDP,
                                         ptx::desc_sw128(k_addr(ng), L::kBlkBytes, 1024), kIdQ, n > 0 ? 1u : 0u);
                ptx::tc_commit_elect(bars.k_empty(ng % KS));
                if (s_issued == n + 1 && n + 1 < steps) {
                    if (!(ok = wait_u(bars.k_full((ng + 1) % KS), ((ng + 1) / KS) & 1, kSiteKvFull))) break;
                    ptx::tc_fence_after();
                    issue_s(ng + 1);
                    ++s_issued;
                }
            }
            // dQ of this tile is complete once every product above is
            // (committed on an abort too: the drain below waits for it)
            ptx::tc_commit_elect(bars.acc_full());
            nb += steps;
        }
        // every product must finish before the CTA frees its TMEM
        if (nf > 0) w.drain(bars.acc_full(), (nf - 1) & 1);
        __syncwarp();
    } else {
        // elementwise: thread = query row of the tile = TMEM lane; columns
        // (keys) [c0, c0 + 64)
        const int row = 32 * (warp & 3) + lane;
        const int c0 = 64 * (warp >> 2);
        const uint32_t row_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        const float c = p.scale_log2;
        const int key_end = p.n - (p.n_tiles - 1) * 128;   // keys of the last key tile (1..128)
        int nb = 0;   // global steps of the tiles before this one
        int nf = 0;   // tiles done
        bool ok = true;
        int qt, qh;
        for (int slot = 0, r; ok && (r = bwd_tile(p.causal, p.n_tiles, p.heads_q, slot, qt, qh)) != 0; ++slot) {
            if (r == 2) continue;
            const int steps = steps_of(qt);
            // A query row past N (a ragged last tile) gets LSE = +inf and D = 0:
            // its P and dS are exactly 0 and it is not stored.
            const bool row_valid = qt * 128 + row < p.n;
            const long long grow = static_cast<long long>(qh) * p.n + qt * 128 + row;
            const bool in = row_valid && FA2_DBG_OK(grow < p.rows_q, kDbgBwdRow);
            const float lse2 = in ? p.lse[grow] * 1.4426950408889634f : INFINITY;
            const float dl = in ? p.delta[grow] : 0.0f;
            for (int n = 0; n < steps; ++n) {
                const int ng = nb + n;
                ok = w.wait(bars.s_full(ng & 1), (ng >> 1) & 1, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const bool diag = p.causal && n == qt;  // key k visible to query q only if k <= q
                // P phase: P = exp2(S c - LSE log2 e), kept in registers
                const uint32_t colS = L::kColS0 + 128u * (ng & 1);
                float pf[64];
                {
                    uint32_t sv[64];
                    ptx::tmem_ld32_at<0>(row_addr + colS + c0, sv);
                    ptx::tmem_ld32_at<32>(row_addr + colS + c0 + 32, sv);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 64; ++j) pf[j] = ptx::ex2_approx(fmaf(__uint_as_float(sv[j]), c, -lse2));
                }
                if (diag) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) pf[j] = c0 + j > row ? 0.0f : pf[j];
                }
                if (n == p.n_tiles - 1 && key_end < 128) {   // keys past N (zero-filled K) get no weight
#pragma unroll
                    for (int j = 0; j < 64; ++j) pf[j] = c0 + j >= key_end ? 0.0f : pf[j];
                }
                // dS phase: dS = P o (dP - D) -> 16-bit over dP
                ok = w.wait(bars.dp_full(), ng & 1, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                {
                    uint32_t dp[64];
                    ptx::tmem_ld32_at<0>(row_addr + L::kColDP + c0, dp);
                    ptx::tmem_ld32_at<32>(row_addr + L::kColDP + c0 + 32, dp);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 32) {
                        uint32_t dk[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int j = cc + 2 * x;
                            dk[x] = ptx::pack2<kBf16>(pf[j] * (__uint_as_float(dp[j]) - dl),
                                                      pf[j + 1] * (__uint_as_float(dp[j + 1]) - dl));
                        }
                        ptx::tmem_st16(row_addr + L::kColDP + c0 + cc / 2, dk);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bars.ds_full());
            }
            if (!ok) break;
            ok = w.wait(bars.acc_full(), nf & 1, kSiteOFull);
            ++nf;
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            store_acc_row<D, kBf16>(row_addr, L::kColAcc, p.scale, p.dq, grow, p.rows_q, c0 * D / 128,
                                    (c0 + 64) * D / 128, row_valid);
            // the accumulator loads are complete; order them before the next
            // tile's first dS arrival, which lets its first dQ overwrite them
            ptx::tc_fence_before();
            nb += steps;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace bwd
}  // namespace fa2
