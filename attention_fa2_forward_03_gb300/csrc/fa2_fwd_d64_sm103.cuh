// FlashAttention-2 forward for GB300 (sm_103a), head dimension 64, equal
// lengths: P in TMEM columns of its own, so the next S is computed while the
// current softmax runs.
//
// What is computed is exactly the 16-bit kernel's (fa2_fwd_sm103.cuh): the
// forward of "A Case Study in CUDA Kernel Fusion: Implementing FlashAttention-2
// on NVIDIA Hopper Architecture using the CUTLASS Library" (abstract) on the
// slice under "Kernel Specification" in "FlashAttention-2 from scratch on
// Ampere, Part 1", with the same tiles (two 128-row query tiles of one KV
// head per item, 128-key steps), the same online softmax (exact running
// max, P rounded to the input type, l summed from the fp32 weights), roles
// and epilogue.
//
// What differs is where P lives. The 16-bit kernel writes P over the S it
// came from, so S of a tile's next step can only be computed after P V of
// this step has read P: per tile the softmax, the hand-off to the MMA warp
// and P V + Q K^T run one after the other, and at d = 64 (where the
// products are short and the softmax is not) the softmax warpgroups wait
// for their own MMAs about half the time. At d = 64 the two tiles' S and O
// take 384 of the 512 TMEM columns, which leaves room for each tile's P:
//     TMEM: S_0 | S_1 | O_0 | O_1 | P_0 | P_1  (128, 128, 64, 64, 64, 64)
// so a softmax warpgroup releases S as soon as it has loaded it (s_free),
// the tile's next S is computed during the rest of the softmax, and the
// softmax goes from one step to the next without waiting for the tensor
// core. P_t of step j is written only after P V of step j - 1 has read P_t
// (pv_done), which the tensor core finished long before. Two warps issue
// the MMAs, one every Q K^T and one every P V: the two streams touch
// disjoint TMEM, so neither waits behind the other's barriers.
//
// Hand-offs per tile t (every barrier is at most one phase ahead of each
// of its waiters; each line says why):
//   s_full(t)   QK warp -> softmax t  next S(t) is issued only after s_free
//   s_free(t)   softmax t -> QK warp  next load of S(t) waits for s_full
//   alpha(t, c & 1)  softmax t -> correction, c = the tile's step count: a
//               slot is rewritten two steps later, after the P store of the
//               step between, which waits for P V of this step, which waits
//               for the correction's p_full arrival of this step
//   p_full(t)   softmax t + correction -> PV warp
//   pv_done(t)  PV warp -> softmax t (before storing P) and correction
//               (before rescaling O, and before the epilogue reads it); the
//               next P V(t) needs both of their p_full arrivals
//   stats(t)    softmax t -> correction (m, l of the item's last step)
#pragma once

#include "fa2_fwd_sm103.cuh"

namespace fa2 {
namespace d64 {

constexpr int kD = 64;

// Shared memory: Q, the K/V ring and the staging slices exactly as the
// 16-bit kernel's d = 64 layout, then this kernel's barriers and row data.
struct Lay {
    using B = Layout<kD>;
    static constexpr int kQOff = B::kQOff;
    static constexpr int kRingOff = B::kRingOff;
    static constexpr int kStageOff = B::kStageOff;
    static constexpr int kTileBytes = B::kTileBytes;
    static constexpr int kBlkBytes = B::kBlkBytes;
    static constexpr int kStages = B::kStages;
    static constexpr int kBarOff = B::kBarOff;
    // q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] s_free[2]
    // alpha[2][2] p_full[2] pv_done[2] stats[2] mma_done[2]
    static constexpr int kNumBars = 2 * kStages + 20;
    static constexpr int kRowOff = kBarOff + kNumBars * 8;
    // alpha[2 tiles][2 slots][128], m[2][128], l[2][128]
    static constexpr int kMiscOff = (kRowOff + 8 * kBM * 4 + 15) & ~15;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + 1024-byte alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
    static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + 64u * t; }
    static __device__ __forceinline__ uint32_t col_p(int t) { return 384u + 64u * t; }
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct BarsD64 {
    uint32_t base;
    static constexpr int S = Lay::kStages;
    __device__ uint32_t q_full(int t) const { return base + 8 * t; }
    __device__ uint32_t q_empty(int t) const { return base + 8 * (2 + t); }
    __device__ uint32_t kv_full(int s) const { return base + 8 * (4 + s); }
    __device__ uint32_t kv_empty(int s) const { return base + 8 * (4 + S + s); }
    __device__ uint32_t s_full(int t) const { return base + 8 * (4 + 2 * S + t); }
    __device__ uint32_t s_free(int t) const { return base + 8 * (6 + 2 * S + t); }
    __device__ uint32_t alpha_ready(int t, int slot) const { return base + 8 * (8 + 2 * S + 2 * t + slot); }
    __device__ uint32_t p_full(int t) const { return base + 8 * (12 + 2 * S + t); }
    __device__ uint32_t pv_done(int t) const { return base + 8 * (14 + 2 * S + t); }
    __device__ uint32_t stats_ready(int t) const { return base + 8 * (16 + 2 * S + t); }
    __device__ uint32_t mma_done(int k) const { return base + 8 * (18 + 2 * S + k); }
};

// ---------------------------------------------------------------- MMA issuers

// Two warps issue the MMAs: warp 13 every S = Q K^T, warp 14 every P V.
// With P in its own columns the two streams touch disjoint TMEM (S_t
// against O_t and P_t), so neither has to wait for the other; each waits
// only for the barriers of its own products, and each S is issued the
// moment the softmax has released the tile's previous S.

// S(t) of every (item, step), tile by tile.
template <bool kBf16>
__device__ __forceinline__ void qk_issuer(const Params& p, uint32_t sbase, uint32_t tmem, const BarsD64& bars,
                                          const Waiter& w) {
    constexpr int S = Lay::kStages;
    constexpr uint32_t kIdS = ptx::idesc_f16(kBf16 ? 1u : 0u, 0, 0, kBM, kBN);  // both K-major
    auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
        return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
    };
    const int nkv = p.n_kv_tiles;
    uint32_t q_par = 0;    // bit t: parity of the next q_full(t) wait
    uint32_t sf_par = 0;   // bit t: parity of the next s_free(t) wait
    uint32_t s_prev = 0;   // bit t: an S(t) has been issued before (its s_free is due)
    int ring0 = 0;         // ring index of the item's K_0
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x, ring0 += 2 * nkv) {
        const int nt = make_item(p, it).n_tiles;
        for (int j = 0; j < nkv && ok; ++j) {
            const int kr = ring0 + 2 * j;
            for (int t = 0; t < nt; ++t) {
                const bool prev = (s_prev >> t) & 1u;
                if (prev && !(ok = wait_u(bars.s_free(t), (sf_par >> t) & 1u, kSiteSFull))) break;
                if (j == 0 && !(ok = wait_u(bars.q_full(t), (q_par >> t) & 1u, kSiteQFull))) break;
                if (t == 0 && !(ok = wait_u(bars.kv_full(kr % S), (kr / S) & 1, kSiteKvFull))) break;
                if (prev) sf_par ^= 1u << t;
                if (j == 0) q_par ^= 1u << t;
                s_prev |= 1u << t;
                ptx::tc_fence_after();
                const uint64_t qd = ptx::desc_sw128(sbase + Lay::kQOff + t * Lay::kTileBytes, 16, 1024);
                const uint64_t kd = ptx::desc_sw128(sbase + Lay::kRingOff + (kr % S) * Lay::kTileBytes, 16, 1024);
                ptx::mma_ss_kloop<2, 4, 6, 0, 0, 0, 0, 2, 4, 6, 0, 0, 0, 0, 4>(tmem + Lay::col_s(t), qd, kd, kIdS,
                                                                              0u);
                ptx::tc_commit_elect(bars.s_full(t));
                if (j == nkv - 1) ptx::tc_commit_elect(bars.q_empty(t));       // last read of Q_t
                if (t == nt - 1) ptx::tc_commit_elect(bars.kv_empty(kr % S));  // last read of K_j
            }
        }
    }
    // Every MMA this warp issued must finish before the CTA frees its TMEM.
    ptx::tc_commit_elect(bars.mma_done(0));
    w.drain(bars.mma_done(0), 0);
    __syncwarp();
}

// O_t (+)= P_t V_j of every (item, step), tile by tile.
template <bool kBf16>
__device__ __forceinline__ void pv_issuer(const Params& p, uint32_t sbase, uint32_t tmem, const BarsD64& bars,
                                          const Waiter& w) {
    constexpr int S = Lay::kStages;
    constexpr uint32_t kIdO = ptx::idesc_f16(kBf16 ? 1u : 0u, 0, 1, kBM, kD);   // V MN-major
    auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
        return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
    };
    const int nkv = p.n_kv_tiles;
    uint32_t pf_par = 0;   // bit t: parity of the next p_full(t) wait
    int ring0 = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x, ring0 += 2 * nkv) {
        const int nt = make_item(p, it).n_tiles;
        for (int j = 0; j < nkv && ok; ++j) {
            const int vr = ring0 + 2 * j + 1;
            for (int t = 0; t < nt; ++t) {
                if (t == 0 && !(ok = wait_u(bars.kv_full(vr % S), (vr / S) & 1, kSiteKvFull))) break;
                if (!(ok = wait_u(bars.p_full(t), (pf_par >> t) & 1u, kSitePFull))) break;
                pf_par ^= 1u << t;
                ptx::tc_fence_after();
                const uint64_t vd =
                    ptx::desc_sw128(sbase + Lay::kRingOff + (vr % S) * Lay::kTileBytes, Lay::kBlkBytes, 1024);
                ptx::mma_ts_kloop8(tmem + Lay::col_o(t), tmem + Lay::col_p(t), vd, kIdO, j > 0 ? 1u : 0u);
                ptx::tc_commit_elect(bars.pv_done(t));
                if (t == nt - 1) ptx::tc_commit_elect(bars.kv_empty(vr % S));  // last read of V_j
            }
        }
    }
    ptx::tc_commit_elect(bars.mma_done(1));
    w.drain(bars.mma_done(1), 0);
    __syncwarp();
}

// ---------------------------------------------------------------- softmax

// Warpgroup t runs tile t of every item: thread = query row = TMEM lane.
template <bool kBf16>
__device__ __forceinline__ void softmax_role(const Params& p, uint32_t tmem, uint8_t* smem, const BarsD64& bars,
                                             const Waiter& w, int t) {
    const int row = threadIdx.x & 127;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(row & ~31) << 16);
    const uint32_t colS = Lay::col_s(t), colP = Lay::col_p(t);
    float* alpha_buf = reinterpret_cast<float*>(smem + Lay::kRowOff) + 2 * t * kBM;   // [2 slots][128]
    float* m_buf = reinterpret_cast<float*>(smem + Lay::kRowOff) + 4 * kBM + t * kBM;
    float* l_buf = m_buf + 2 * kBM;
    const float c = p.scale_log2;
    const uint64_t c2 = ptx::f2_pack(c, c);
    const int nkv = p.n_kv_tiles;

    uint32_t sf_par = 0, pv_par = 0;
    int cnt = 0;   // S(t) tiles consumed by this warpgroup
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x) {
        if (t >= make_item(p, it).n_tiles) continue;
        float m = -INFINITY;  // running row max of the scaled scores, log2 units
        float l = 0.0f;       // running sum of exp2(s*c - m)
        for (int j = 0; j < nkv; ++j, ++cnt) {
            ok = w.wait(bars.s_full(t), sf_par, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            sf_par ^= 1u;
            ptx::tc_fence_after();
            uint32_t s[kBN];
            float mq[4];
            ptx::tmem_ld32_max_at<0>(row_addr + colS + 0, s, mq[0]);
            ptx::tmem_ld32_max_at<32>(row_addr + colS + 32, s, mq[1]);
            ptx::tmem_ld32_max_at<64>(row_addr + colS + 64, s, mq[2]);
            ptx::tmem_ld32_max_at<96>(row_addr + colS + 96, s, mq[3]);
            ptx::tmem_wait_ld();
            // S is in registers: the MMA warp may compute the next S(t).
            ptx::tc_fence_before();
            ptx::mbar_arrive(bars.s_free(t));
            const float m_tile = fmaxf(ptx::max3(mq[0], mq[1], mq[2]), mq[3]) * c;
            const float m_new = fmaxf(m, m_tile);
            const float alpha = (j == 0 || m_new == m) ? 1.0f : ptx::ex2_approx(m - m_new);
            // The read-back keeps both arrives ahead of the exponentials in
            // the compiled schedule (publish_alpha).
            const float alpha_r = publish_alpha(alpha_buf + (cnt & 1) * kBM + row, alpha, bars.alpha_ready(t, cnt & 1));
            l *= alpha_r;
            m = m_new + 0.0f * alpha_r;   // alpha_r is finite: m_new, after the read-back

            // P = exp2(S*c - m) on pairs, every exponential on the MUFU: here
            // the softmax is bound by issue slots, not by the MUFU, and the
            // FMA-pipe polynomial the 16-bit kernel runs for one pair in
            // eight measured 4.4% slower. Each half of the row's 64 packed
            // pairs goes to TMEM as soon as it is done (fewer live registers);
            // P_t is free once P V of the tile's previous step has read it.
            const uint64_t nm2 = ptx::f2_pack(-m, -m);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[kBN / 4];
#pragma unroll
                for (int k = 0; k < kBN / 4; ++k) {
                    const int i = half * (kBN / 4) + k;
                    const uint64_t x =
                        ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, nm2);
                    float x0, x1;
                    ptx::f2_unpack(x, x0, x1);
                    const float p0 = ptx::ex2_approx(x0);
                    const float p1 = ptx::ex2_approx(x1);
                    acc[i & 3] = ptx::f2_add(acc[i & 3], ptx::f2_pack(p0, p1));
                    pk[k] = ptx::pack2<kBf16>(p0, p1);
                }
                if (half == 0 && cnt > 0) {
                    ok = w.wait(bars.pv_done(t), pv_par, kSitePFull);
                    pv_par ^= 1u;
                }
                if (half == 0) ptx::tc_fence_after();
                ptx::tmem_st32_at<0>(row_addr + colP + 32 * half, pk);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            float a0, a1;
            ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), a0, a1);
            l += a0 + a1;
            if (j + 1 == nkv) {
                m_buf[row] = m;
                l_buf[row] = l;
                ptx::mbar_arrive(bars.stats_ready(t));
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bars.p_full(t));
        }
    }
}

// ---------------------------------------------------------------- correction + epilogue

template <bool kBf16>
__device__ __forceinline__ void correction_role(const Params& p, uint32_t tmem, uint8_t* smem, uint32_t sbase,
                                                const BarsD64& bars, const Waiter& w) {
    const int q = (threadIdx.x / 32) & 3;      // TMEM lane quarter
    const int lane = threadIdx.x & 31;
    const int row = 32 * q + lane;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const float* rows = reinterpret_cast<const float*>(smem + Lay::kRowOff);   // alpha[2][2][128] | m[2][128] | l[2][128]
    const uint32_t wslice = sbase + Lay::kStageOff + static_cast<uint32_t>(q) * (32u * 128u);
    const int nkv = p.n_kv_tiles;

    uint32_t a_par = 0;    // bit 2t + slot: parity of the next alpha_ready(t, slot) wait
    uint32_t pv_par = 0;   // bit t: parity of the next pv_done(t) wait
    uint32_t st_par = 0;   // bit t: parity of the next stats_ready(t) wait
    int cnt[2] = {0, 0};   // steps seen per tile
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x) {
        const Item item = make_item(p, it);
        const int nt = item.n_tiles;
        for (int j = 0; j < nkv && ok; ++j) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (t >= nt) break;
                const int slot = cnt[t] & 1;
                const int ab = 2 * t + slot;
                ok = w.wait(bars.alpha_ready(t, slot), (a_par >> ab) & 1u, kSiteAlpha);
                // From step 1 on, P V of the tile's previous step must have
                // completed before O is rescaled (waited for even when no
                // row needs it, to keep the phases in step).
                if (ok && j > 0) ok = w.wait(bars.pv_done(t), (pv_par >> t) & 1u, kSiteOFull);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                a_par ^= 1u << ab;
                if (j > 0) pv_par ^= 1u << t;
                ++cnt[t];
                const float alpha = rows[ab * kBM + row];
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                    ptx::tc_fence_after();
                    const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
                    for (int h = 0; h < kD; h += 32) {
                        uint32_t o[32];
                        ptx::tmem_ld32_at<0>(row_addr + Lay::col_o(t) + h, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float o0, o1;
                            ptx::f2_unpack(
                                ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                            a2),
                                o0, o1);
                            o[2 * i] = __float_as_uint(o0);
                            o[2 * i + 1] = __float_as_uint(o1);
                        }
                        ptx::tmem_st32_at<0>(row_addr + Lay::col_o(t) + h, o);
                    }
                    ptx::tmem_wait_st();
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(bars.p_full(t));
            }
        }
        // Epilogue: O / l -> 16 bit through the warp's staging slice, LSE.
        // The next item's first P V into O_t waits for this warpgroup's next
        // p_full arrival, which comes after these loads.
        for (int t = 0; t < nt && ok; ++t) {
            ok = w.wait(bars.stats_ready(t), (st_par >> t) & 1u, kSiteStats);
            if (ok) ok = w.wait(bars.pv_done(t), (pv_par >> t) & 1u, kSiteOFull);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            st_par ^= 1u << t;
            pv_par ^= 1u << t;
            ptx::tc_fence_after();
            const float m = rows[(4 + t) * kBM + row];
            const float l = rows[(6 + t) * kBM + row];
            const float inv_l = ptx::rcp_approx(l);
            uint32_t hv[32];
            {
                uint32_t o[64];
                ptx::tmem_ld32_at<0>(row_addr + Lay::col_o(t), o);
                ptx::tmem_ld32_at<32>(row_addr + Lay::col_o(t) + 32, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    hv[i] = ptx::pack2<kBf16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            }
            store_o_rows<kD>(hv, wslice, lane, p.o, item.q_row0 + t * kBM + 32 * q, 0, 32, p.rows_q);
            const int grow = item.q_row0 + t * kBM + row;
            if (FA2_DBG_OK(grow < p.rows_q, kDbgORow)) p.lse[grow] = (m + ptx::lg2_approx(l)) * 0.69314718055994530942f;
        }
        ptx::tc_fence_before();
    }
}

}  // namespace d64

// ---------------------------------------------------------------- kernel

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_d64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = d64::Lay;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const d64::BarsD64 bars{sbase + L::kBarOff};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars.q_full(t), 1);
            ptx::mbar_init(bars.q_empty(t), 1);
            ptx::mbar_init(bars.s_full(t), 1);
            ptx::mbar_init(bars.s_free(t), kBM);
            ptx::mbar_init(bars.alpha_ready(t, 0), kBM);
            ptx::mbar_init(bars.alpha_ready(t, 1), kBM);
            ptx::mbar_init(bars.p_full(t), 2 * kBM);   // softmax + correction warpgroups
            ptx::mbar_init(bars.pv_done(t), 1);
            ptx::mbar_init(bars.stats_ready(t), kBM);
        }
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(bars.kv_full(s), 1);
            ptx::mbar_init(bars.kv_empty(s), 1);
        }
        ptx::mbar_init(bars.mma_done(0), 1);
        ptx::mbar_init(bars.mma_done(1), 1);
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
        d64::softmax_role<kBf16>(p, tmem, smem, bars, w, warp / 4);
    } else if (warp < kLoadWarp) {
        ptx::setmaxnreg_dec<kRegCorr>();
        d64::correction_role<kBf16>(p, tmem, smem, sbase, bars, w);
    } else {
        ptx::setmaxnreg_dec<kRegOther>();
        if (warp == kLoadWarp) {
            if (lane == 0) producer<d64::kD>(&tmQ, &tmK, &tmV, p, sbase, bars, w);
            __syncwarp();
        } else if (warp == kMmaWarp) {
            d64::qk_issuer<kBf16>(p, sbase, tmem, bars, w);   // whole warp, one lane issues
        } else if (warp == kMmaWarp + 1) {
            d64::pv_issuer<kBf16>(p, sbase, tmem, bars, w);
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
