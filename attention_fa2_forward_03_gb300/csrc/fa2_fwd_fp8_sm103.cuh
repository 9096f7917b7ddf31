// FP8 (e4m3) attention forward for GB300 (sm_103a). Device code; it shares
// the 16-bit kernel's work items, parameters, watchdog and roles' constants
// (fa2_fwd_sm103.cuh). fa2_fwd_sm103.cu holds the host side.
//
// What is computed: attention on quantised inputs with the scales applied
// inside the kernel, the inference variant of "FlashAttention-3 for
// Inference: INT8 Quantization and Query Head Packing for MQA/GQA" (Colfax
// Research author page), which names in-kernel pre-processing of the inputs
// by specialised warps and query-head packing. Q, K, V are e4m3 codes with
// one fp32 descale per (batch, KV head) and tensor; O is bf16, LSE fp32:
//   S = (scale * dq * dk) * Q8 K8^T                      (tcgen05 kind::f8f6f4)
//   P' = exp2(S log2e - m + 8) in (0, 256], rounded to e4m3   (m: exact row max)
//   O = dv * (P'8 V8) / l',   l' = sum of the unrounded P'
//   LSE = (m + log2 l' - 8) * ln 2
// The 2^8 factor moves P's range (0, 1] up to where e4m3 has its precision;
// it cancels in O / l' and is taken out of the LSE.
//
// How: the 16-bit kernel's persistent, warp-specialised pipeline (two query
// tiles per item, softmax warpgroups 0-1, correction warpgroup 2, TMA
// producer warp 12, MMA warp 13) with both GEMMs on 8-bit operands and P
// packed four per TMEM column. The P V product reads V where TMA put it,
// dims contiguous, as an MN-major B operand: tcgen05 takes 8-bit operands in
// either major order, so V needs no transposition (the Hopper kernel of the
// FA3-for-inference page transposes V in shared memory because its 8-bit
// wgmma takes K-major operands only). Head dimension 128 (one 128-byte
// swizzle row per tile row, so the MN-major V tile is a single swizzle atom
// wide).
//
// Two modes, as in the 16-bit kernel: equal lengths N % 128 == 0 without a
// mask (kGen = false: query-head packing, 2-D tensor maps), and the general
// mode (kGen = true: unequal and ragged lengths, the bottom-right causal
// mask; one query head per item, 3-D maps whose rows past a head's end read
// as zero, masked keys set to -inf before the row max). Key tiles start at
// key 0 in both, so each tile's weights are rounded against the same running
// max as without the mask.
#pragma once

#include "fa2_fwd_sm103.cuh"

namespace fa2 {
namespace fp8 {

constexpr int kD = 128;              // head dimension = bytes per tile row
constexpr int kTile = kBM * kD;      // 16 KB: one Q, K, V or V^T tile
constexpr int kStages = 8;           // K/V ring (K_j, V_j, K_{j+1}, ...)

struct Lay {
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kNQ * kTile;
    // Epilogue staging: 128 rows x 64 bf16 columns (the 16-bit kernel's form)
    static constexpr int kStageOff = kRingOff + kStages * kTile;
    static constexpr int kStageBytes = kBM * 128;
    static constexpr int kBarOff = kStageOff + kStageBytes;
    // q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] alpha[2] stats[2]
    // p_full[2] o_full[2] mma_done stats_free[2]
    static constexpr int kNumBars = 2 * kStages + 17;
    static constexpr int kRowOff = kBarOff + kNumBars * 8;  // alpha[2][128], m[2][128], l[2][128]
    static constexpr int kMiscOff = kRowOff + 3 * kNQ * kBM * 4;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static constexpr uint32_t kTmemCols = 512;  // S_0 | S_1 | O_0 | O_1
    static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
    static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + kD * t; }
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct BarsF8 {
    uint32_t base;
    static constexpr int S = kStages;
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

// (batch, KV head) group of a work item: the index of its descales.
__device__ __forceinline__ int item_group(const Params& p, int item) { return item / p.pairs; }

// ---------------------------------------------------------------- producer

__device__ __forceinline__ void producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                         const Params& p, uint32_t sbase, const BarsF8& bars, const Waiter& w) {
    constexpr int S = kStages;
    int ring = 0;
    int nq[2] = {0, 0};
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it += gridDim.x) {
        const Item item = make_item(p, it);
        auto load_kv = [&](int k) {
            const int s = ring % S;
            if (!(ok = w.wait(bars.kv_empty(s), ((ring / S) & 1) ^ 1, kSiteKvEmpty))) return;
            ptx::mbar_arrive_expect_tx(bars.kv_full(s), kTile);
            if (FA2_DBG_OK(item.kv_row0 + (k >> 1) * kBN + kBN <= p.rows_kv, kDbgKvTile))
                ptx::tma_load_2d(sbase + Lay::kRingOff + s * kTile, (k & 1) ? tmV : tmK, 0,
                                 item.kv_row0 + (k >> 1) * kBN, bars.kv_full(s));
            ++ring;
        };
        // K_0, V_0 before the Q tiles (the 16-bit producer says why).
        constexpr int kPre = 2;
        for (int k = 0; k < kPre && ok; ++k) load_kv(k);
        for (int t = 0; t < item.n_tiles && ok; ++t) {
            if (!(ok = w.wait(bars.q_empty(t), (nq[t] & 1) ^ 1, kSiteQEmpty))) break;
            ptx::mbar_arrive_expect_tx(bars.q_full(t), kTile);
            if (FA2_DBG_OK(item.q_row0 + t * kBM + kBM <= p.rows_q, kDbgQTile))
                ptx::tma_load_2d(sbase + Lay::kQOff + t * kTile, tmQ, 0, item.q_row0 + t * kBM, bars.q_full(t));
            ++nq[t];
        }
        const int nxt = it + gridDim.x;
        if (ok && nxt < p.total_items) {
            const Item ni = make_item(p, nxt);
            for (int t = 0; t < ni.n_tiles; ++t) ptx::tma_prefetch_l2_2d(tmQ, 0, ni.q_row0 + t * kBM);
        }
        for (int k = kPre; k < 2 * p.n_kv_tiles && ok; ++k) load_kv(k);
    }
    if (!ok) {
        const int first = ring > S ? ring - S : 0;
        for (int r = first; r < ring; ++r) w.drain(bars.kv_full(r % S), (r / S) & 1);
        for (int t = 0; t < 2; ++t)
            if (nq[t] > 0) w.drain(bars.q_full(t), (nq[t] - 1) & 1);
    }
}

// General mode: one query head per item (make_item_gen), 3-D maps; only
// tiles with keys to attend load Q, and an item loads K_j, V_j for
// j < max(nkv[0], nkv[1]).
__device__ __forceinline__ void producer_gen(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                             const Params& p, uint32_t sbase, const BarsF8& bars, const Waiter& w) {
    constexpr int S = kStages;
    int ring = 0;
    int nq[2] = {0, 0};
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<true>(it)) {
        const ItemG g = make_item_gen(p, it);
        for (int t = 0; t < g.n_tiles && ok; ++t) {
            if (g.nkv[t] == 0) continue;
            if (!(ok = w.wait(bars.q_empty(t), (nq[t] & 1) ^ 1, kSiteQEmpty))) break;
            ptx::mbar_arrive_expect_tx(bars.q_full(t), kTile);
            if (FA2_DBG_OK(g.head < p.heads_q && g.q0 + t * kBM < p.nq, kDbgQTile))
                ptx::tma_load_3d(sbase + Lay::kQOff + t * kTile, tmQ, 0, g.q0 + t * kBM, g.head, bars.q_full(t));
            ++nq[t];
        }
        const int nmax = max(g.nkv[0], g.nkv[1]);
        for (int k = 0; k < 2 * nmax && ok; ++k) {
            const int s = ring % S;
            if (!(ok = w.wait(bars.kv_empty(s), ((ring / S) & 1) ^ 1, kSiteKvEmpty))) break;
            ptx::mbar_arrive_expect_tx(bars.kv_full(s), kTile);
            if (FA2_DBG_OK(g.kvhead < p.heads_kv && (k >> 1) * kBN < p.nk, kDbgKvTile))
                ptx::tma_load_3d(sbase + Lay::kRingOff + s * kTile, (k & 1) ? tmV : tmK, 0, (k >> 1) * kBN, g.kvhead,
                                 bars.kv_full(s));
            ++ring;
        }
    }
    if (!ok) {
        const int first = ring > S ? ring - S : 0;
        for (int r = first; r < ring; ++r) w.drain(bars.kv_full(r % S), (r / S) & 1);
        for (int t = 0; t < 2; ++t)
            if (nq[t] > 0) w.drain(bars.q_full(t), (nq[t] - 1) & 1);
    }
}

// ---------------------------------------------------------------- MMA issuer

__device__ __forceinline__ void mma_issuer(const Params& p, uint32_t sbase, uint32_t tmem, const BarsF8& bars,
                                           const Waiter& w) {
    constexpr int S = kStages;
    // e4m3 x e4m3 -> f32; Q and K K-major, V MN-major
    constexpr uint32_t kIdS = ptx::idesc_f16(0u, 0, 0, kBM, kBN);
    constexpr uint32_t kIdO = ptx::idesc_f16(0u, 0, 1, kBM, kD);
    auto stage_addr = [&](int r) { return sbase + Lay::kRingOff + (r % S) * kTile; };
    auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint64_t qd = ptx::desc_sw128(sbase + Lay::kQOff + t * kTile, 16, 1024);
        const uint64_t kd = ptx::desc_sw128(kaddr, 16, 1024);
        ptx::mma_ss_kloop4_f8(tmem + Lay::col_s(t), qd, kd, kIdS, 0u);
    };
    // V MN-major: one 128-byte swizzle atom across the 128 dims (the leading
    // offset is never stepped over), 1024 B between groups of 8 keys.
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint64_t vd = ptx::desc_sw128(vaddr, kTile, 1024);
        ptx::mma_ts_kloop4_f8_mn(tmem + Lay::col_o(t), tmem + Lay::col_s(t), vd, kIdO, acc ? 1u : 0u);
    };
    auto wait_u = [&](uint32_t bar, uint32_t parity, int site) {
        return __shfl_sync(0xffffffffu, w.wait(bar, parity, site) ? 1 : 0, 0) != 0;
    };
    auto wait_ring = [&](int r) { return wait_u(bars.kv_full(r % S), (r / S) & 1, kSiteKvFull); };

    const int nkv = p.n_kv_tiles;
    int ring = 0;
    int nq[2] = {0, 0};
    int np[2] = {0, 0};
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
            // V_j, K_{j+1} and P(0, j) are waited for together.
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
    ptx::tc_commit_elect(bars.mma_done());
    w.drain(bars.mma_done(), 0);
    __syncwarp();
}

// General mode: mma_issuer's order with a KV tile count per query tile (as
// the 16-bit kernel's general issuer): at KV tile j only tiles with
// j < nkv[t] take part; V_j's and K_{j+1}'s stages are released after their
// last user.
__device__ __forceinline__ void mma_issuer_gen(const Params& p, uint32_t sbase, uint32_t tmem, const BarsF8& bars,
                                               const Waiter& w) {
    constexpr int S = kStages;
    constexpr uint32_t kIdS = ptx::idesc_f16(0u, 0, 0, kBM, kBN);
    constexpr uint32_t kIdO = ptx::idesc_f16(0u, 0, 1, kBM, kD);
    auto stage_addr = [&](int r) { return sbase + Lay::kRingOff + (r % S) * kTile; };
    auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint64_t qd = ptx::desc_sw128(sbase + Lay::kQOff + t * kTile, 16, 1024);
        const uint64_t kd = ptx::desc_sw128(kaddr, 16, 1024);
        ptx::mma_ss_kloop4_f8(tmem + Lay::col_s(t), qd, kd, kIdS, 0u);
    };
    // V MN-major: one 128-byte swizzle atom across the 128 dims (the leading
    // offset is never stepped over), 1024 B between groups of 8 keys.
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint64_t vd = ptx::desc_sw128(vaddr, kTile, 1024);
        ptx::mma_ts_kloop4_f8_mn(tmem + Lay::col_o(t), tmem + Lay::col_s(t), vd, kIdO, acc ? 1u : 0u);
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

// ---------------------------------------------------------------- softmax

template <bool kGen>
__device__ __forceinline__ void softmax_role(const Params& p, uint32_t tmem, uint8_t* smem, const BarsF8& bars,
                                             const Waiter& w, int t) {
    const int row = threadIdx.x & 127;
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(row & ~31) << 16);
    const uint32_t colS = Lay::col_s(t);
    float* alpha_buf = reinterpret_cast<float*>(smem + Lay::kRowOff) + t * kBM;
    float* m_buf = alpha_buf + kNQ * kBM;
    float* l_buf = m_buf + kNQ * kBM;

    int n_s = 0;      // S tiles consumed; bit 30: item parity (general mode)
    bool ok = true;
    for (int it = blockIdx.x; it < p.total_items && ok; it = next_item<kGen>(it)) {
        int nkv, grp, jmask = 0x7fffffff, kend_row = 0;
        if constexpr (kGen) {
            const ItemG g = make_item_gen(p, it);
            if (t >= g.n_tiles || g.nkv[t] == 0) continue;
            nkv = g.nkv[t];
            jmask = g.jmask[t];
            kend_row = kend_of(p, g.q0 + t * kBM + row);
            grp = g.kvhead;
        } else {
            if (t >= make_item(p, it).n_tiles) continue;
            nkv = p.n_kv_tiles;
            grp = item_group(p, it);
        }
        // log2-domain factor of the raw code products: scale * log2(e) * dq * dk
        float c = p.scale_log2 * __ldg(p.q_descale + grp) * __ldg(p.k_descale + grp);
        // A zero descale makes every score 0; c = FLT_MIN gives the same
        // weights (exp2 of |s c| < 2^-90 is 1) and keeps masked keys at
        // -inf * c = -inf instead of NaN.
        if constexpr (kGen) c = fmaxf(c, 1.17549435e-38f);
        const uint64_t c2 = ptx::f2_pack(c, c);
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
        float m = -INFINITY;
        float l = 0.0f;       // sum of the unrounded 2^8-scaled weights
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
                    for (int e = 0; e < kBN; ++e) s[e] = e < lim ? s[e] : 0xFF800000u;
                }
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
                float mq[4];   // row max of each 32-column load
                ptx::tmem_ld32_max_at<0>(row_addr + colS + 0, s, mq[0]);
                ptx::tmem_ld32_max_at<32>(row_addr + colS + 32, s, mq[1]);
                ptx::tmem_ld32_max_at<64>(row_addr + colS + 64, s, mq[2]);
                ptx::tmem_ld32_max_at<96>(row_addr + colS + 96, s, mq[3]);
                ptx::tmem_wait_ld();
                m_tile = fmaxf(ptx::max3(mq[0], mq[1], mq[2]), mq[3]) * c;
            }
            // c > 0, so the max of c*s is c times the max of s
            const float m_new = fmaxf(m, m_tile);
            const float alpha = (j == 0 || m_new == m) ? 1.0f : ptx::ex2_approx(m - m_new);
            alpha_buf[row] = alpha;
            ptx::mbar_arrive(bars.alpha_ready(t));
            l *= alpha;
            m = m_new;
            // A row with no allowed key so far keeps m = -inf; exponentiate
            // against 0 then, so its weights are exp2(-inf) = 0.
            const float m_use = (kGen && m == -INFINITY) ? 0.0f : m;

            // P' = exp2(S c - m + 8), four at a time into one TMEM column.
            const uint64_t nm2 = ptx::f2_pack(8.0f - m_use, 8.0f - m_use);
            uint64_t acc[4] = {0, 0, 0, 0};
            uint32_t pk[kBN / 4];
#pragma unroll
            for (int i = 0; i < kBN / 4; ++i) {
                float pr[4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = 4 * i + 2 * h;
                    const uint64_t x =
                        ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), c2, nm2);
                    // every exponential on the MUFU: the softmax is bound by
                    // issue slots here, and the FMA-pipe polynomial the
                    // 16-bit kernel runs for one pair in eight measured 4.7%
                    // slower in this kernel
                    float x0, x1;
                    ptx::f2_unpack(x, x0, x1);
                    pr[2 * h] = ptx::ex2_approx(x0);
                    pr[2 * h + 1] = ptx::ex2_approx(x1);
                    acc[(2 * i + h) & 3] = ptx::f2_add(acc[(2 * i + h) & 3], ptx::f2_pack(pr[2 * h], pr[2 * h + 1]));
                }
                pk[i] = ptx::pack4_e4m3(pr[0], pr[1], pr[2], pr[3]);
            }
            float a0, a1;
            ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), a0, a1);
            l += a0 + a1;
            ptx::tmem_st32_at<0>(row_addr + colS, pk);
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

}  // namespace fp8

// ---------------------------------------------------------------- kernel

template <bool kGen>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = fp8::Lay;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const fp8::BarsF8 bars{sbase + L::kBarOff};
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
            ptx::mbar_init(bars.p_full(t), 2 * kBM);
            ptx::mbar_init(bars.o_full(t), 1);
        }
        for (int s = 0; s < fp8::kStages; ++s) {
            ptx::mbar_init(bars.kv_full(s), 1);
            ptx::mbar_init(bars.kv_empty(s), 1);   // the MMA warp's commit
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
        fp8::softmax_role<kGen>(p, tmem, smem, bars, w, warp / 4);
    } else if (warp < kLoadWarp) {
        ptx::setmaxnreg_dec<kRegCorr>();
        correction_role<L, fp8::BarsF8, fp8::kD, true, kGen, true>(p, tmem, smem, sbase, bars, w);
    } else {
        ptx::setmaxnreg_dec<kRegOther>();
        if (warp == kLoadWarp) {
            if (lane == 0) {
                if constexpr (kGen)
                    fp8::producer_gen(&tmQ, &tmK, &tmV, p, sbase, bars, w);
                else
                    fp8::producer(&tmQ, &tmK, &tmV, p, sbase, bars, w);
            }
            __syncwarp();
        } else if (warp == kMmaWarp) {
            if constexpr (kGen)
                fp8::mma_issuer_gen(p, sbase, tmem, bars, w);
            else
                fp8::mma_issuer(p, sbase, tmem, bars, w);
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
