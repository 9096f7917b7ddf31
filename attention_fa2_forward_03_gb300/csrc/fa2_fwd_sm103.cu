// FlashAttention-2 forward and backward for GB300 (sm_103a): host side and C ABI.
//
// The kernels: fa2_fwd_sm103.cuh (16-bit forward), fa2_fwd_fp8_sm103.cuh (FP8
// forward), fa2_bwd_sm103.cuh (backward). This file plans the launches
// (tensor maps, persistent grid, work items), checks arguments and device,
// and exports the functions declared in include/fa2.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "fa2.h"
#include "fa2_bwd_sm103.cuh"
#include "fa2_fwd_fp8_sm103.cuh"
#include "fa2_fwd_sm103.cuh"
#include "fa2_fwd_d64_sm103.cuh"

// ==================================================================== host

namespace {

using fa2::Layout;
using fa2::Params;

std::atomic<long long> g_wait_limit_ns{2000000000LL};
std::atomic<int> g_debug_flags{0};

// The planner's kernel table has one shape with a choice: d = 64 with equal
// lengths runs fa2_fwd_d64_kernel (P in TMEM columns of its own, two MMA
// warps; the default, measured faster) or, with this bit set, the 16-bit
// kernel's d = 64 path (P written over S, one MMA warp).
constexpr int kTileCfgD64Shared = 1;
constexpr int kTileCfgMask = kTileCfgD64Shared;
std::atomic<int> g_tile_cfg{-1};   // -1: FA2_TILE_CFG not read yet

int tile_cfg() {
    const int c = g_tile_cfg.load(std::memory_order_acquire);
    if (c >= 0) return c;
    int v = 0;
    if (const char* e = std::getenv("FA2_TILE_CFG"))
        if (std::strcmp(e, "d64=shared") == 0) v = kTileCfgD64Shared;
    int expected = -1;
    g_tile_cfg.compare_exchange_strong(expected, v, std::memory_order_acq_rel);
    return g_tile_cfg.load(std::memory_order_acquire);
}
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kMaxDevices = 64;
// Kernel slots: 16-bit forward 0-7, backward dK/dV 8-11, FP8 forward 12-13,
// backward dQ 14-17, d = 64 equal-length forward 18-19.
constexpr int kKernelSlots = 20;
// Per-device facts, read without a lock: every field is an atomic written
// with release and read with acquire, and two threads that probe the same
// device at once store the same values.
struct DeviceState {
    std::atomic<int> state;     // 0 = not probed, 1 = compute capability 10.3, 2 = other
    std::atomic<int> sm_count;
    std::atomic<bool> smem_set[kKernelSlots];  // dynamic shared-memory limit raised for kernel slot i
};
DeviceState g_dev[kMaxDevices];  // static storage: zero-initialised

// A CUDA call of this library failed: return FA2_ERR_CUDA and leave no
// (non-sticky) error of ours pending for the caller's next cudaGetLastError.
fa2_status cuda_fail() {
    (void)cudaGetLastError();
    return FA2_ERR_CUDA;
}

fa2_status get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return FA2_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail();
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FA2_OK;
}

fa2_status check_device(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
    DeviceState& st = g_dev[dev];
    int s = st.state.load(std::memory_order_acquire);
    if (s == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail();
        st.sm_count.store(sms, std::memory_order_relaxed);
        s = (major == 10 && minor == 3) ? 1 : 2;
        st.state.store(s, std::memory_order_release);
    }
    *dev_out = dev;
    return s == 1 ? FA2_OK : FA2_ERR_UNSUPPORTED;
}

int sm_count(int dev) { return g_dev[dev].sm_count.load(std::memory_order_relaxed); }

// Raises the dynamic shared-memory limit of `kern` on device `dev` once.
template <typename K>
fa2_status set_smem(int dev, int slot, K kern, int bytes) {
    std::atomic<bool>& done = g_dev[dev].smem_set[slot];
    if (done.load(std::memory_order_acquire)) return FA2_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return cuda_fail();
    done.store(true, std::memory_order_release);
    return FA2_OK;
}

// Queues one kernel and judges the launch by its own return code (not by
// cudaGetLastError, which would also report an error left pending earlier).
template <typename... Exp, typename... Act>
fa2_status launch_kernel(void (*kern)(Exp...), dim3 grid, int threads, int smem, cudaStream_t stream,
                         Act&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...) == cudaSuccess ? FA2_OK : cuda_fail();
}

// 2-D view [rows, d] of a 16-bit tensor, boxes of 128 rows x 64 elements
// (128 bytes, the widest box the 128-byte swizzle allows).
fa2_status encode_map(CUtensorMap* m, const void* ptr, uint64_t rows, int d) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ptr), dims, strides, box,
                          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

// 3-D view [mats, rows, d] of a 16-bit tensor (general mode): a box of 128
// rows never crosses into the next head, and rows past `rows` read as zero.
fa2_status encode_map_3d(CUtensorMap* m, const void* ptr, uint64_t mats, uint64_t rows, int d) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), rows, mats};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, rows * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(ptr), dims, strides, box,
                          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

template <int D, bool kBf16, bool kGen = false>
fa2_status launch(int dev, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                  const Params& p, dim3 grid, cudaStream_t stream) {
    constexpr int kSmem = Layout<D>::kSmemBytes;
    auto kern = fa2::fa2_fwd_kernel<D, kBf16, kGen>;
    const int slot = (D == 128 ? 0 : 2) + (kBf16 ? 0 : 1) + (kGen ? 4 : 0);
    const fa2_status st = set_smem(dev, slot, kern, kSmem);
    if (st != FA2_OK) return st;
    return launch_kernel(kern, grid, fa2::kThreads, kSmem, stream, mq, mk, mv, p);
}

// The d = 64 equal-length kernel (P in TMEM columns of its own).
template <bool kBf16>
fa2_status launch_d64(int dev, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const Params& p, dim3 grid, cudaStream_t stream) {
    constexpr int kSmem = fa2::d64::Lay::kSmemBytes;
    auto kern = fa2::fa2_fwd_d64_kernel<kBf16>;
    const fa2_status st = set_smem(dev, kBf16 ? 18 : 19, kern, kSmem);
    if (st != FA2_OK) return st;
    return launch_kernel(kern, grid, fa2::kThreads, kSmem, stream, mq, mk, mv, p);
}

// 2-D view [rows, 128] of an 8-bit tensor (FP8 kernel): boxes of 128 rows x
// 128 bytes, the full width of the 128-byte swizzle.
fa2_status encode_map_u8(CUtensorMap* m, const void* ptr, uint64_t rows) {
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

// 3-D view [mats, rows, 128] of an 8-bit tensor (FP8 general mode): a box
// never crosses into the next head, and rows past `rows` read as zero.
fa2_status encode_map_u8_3d(CUtensorMap* m, const void* ptr, uint64_t mats, uint64_t rows) {
    cuuint64_t dims[3] = {128, rows, mats};
    cuuint64_t strides[2] = {128, rows * 128};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

template <bool kGen>
fa2_status launch_fp8(int dev, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const Params& p, dim3 grid, cudaStream_t stream) {
    constexpr int kSmem = fa2::fp8::Lay::kSmemBytes;
    constexpr int kSlot = kGen ? 13 : 12;
    auto kern = fa2::fa2_fwd_fp8_kernel<kGen>;
    const fa2_status st = set_smem(dev, kSlot, kern, kSmem);
    if (st != FA2_OK) return st;
    return launch_kernel(kern, grid, fa2::kThreads, kSmem, stream, mq, mk, mv, p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// The general-mode kernel (any lengths, optional causal mask) on checked
// arguments. Also takes equal-length calls with N = 128, whose items have a
// single KV tile: the kernels' equal-length mode relies on every item
// having two or more.
fa2_status fwd_general(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q, int H_kv,
                       int N_q, int N_k, int d, float scale, int causal, fa2_dtype dtype, cudaStream_t stream) {
    const long long heads_q = static_cast<long long>(B) * H_q;
    const long long rows_q = heads_q * N_q;
    const long long rows_kv = static_cast<long long>(B) * H_kv * N_k;
    const long long tq = (N_q + fa2::kBM - 1) / fa2::kBM;
    const long long items = heads_q * ((tq + fa2::kNQ - 1) / fa2::kNQ);
    // Item indices stay below 2^31 - 4096 so that a CTA's next index (at most
    // two grids further) never overflows.
    if (rows_q > 0x7FFFFFFFLL || rows_kv > 0x7FFFFFFFLL || items > 0x7FFFFFFFLL - 4096) return FA2_ERR_UNSUPPORTED;

    int dev = 0;
    fa2_status st = check_device(&dev);
    if (st != FA2_OK) return st;
    if ((st = get_encoder()) != FA2_OK) return st;

    CUtensorMap mq, mk, mv;
    if (encode_map_3d(&mq, q, static_cast<uint64_t>(heads_q), static_cast<uint64_t>(N_q), d) != FA2_OK ||
        encode_map_3d(&mk, k, static_cast<uint64_t>(B) * H_kv, static_cast<uint64_t>(N_k), d) != FA2_OK ||
        encode_map_3d(&mv, v, static_cast<uint64_t>(B) * H_kv, static_cast<uint64_t>(N_k), d) != FA2_OK)
        return cuda_fail();

    Params p{};
    p.o = o;
    p.lse = lse;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.debug_flags = g_debug_flags.load();
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.nq = N_q;
    p.nk = N_k;
    p.causal = causal;
    p.heads_q = static_cast<int>(heads_q);
    p.hq = H_q;
    p.group = H_q / H_kv;
    p.tq = static_cast<int>(tq);
    p.pairs = static_cast<int>((tq + fa2::kNQ - 1) / fa2::kNQ);
    p.total_items = static_cast<int>(items);
    p.heads_kv = B * H_kv;
    p.rows_q = rows_q;
    p.rows_kv = rows_kv;
    const dim3 grid(static_cast<unsigned>(std::min<long long>(items, sm_count(dev))));

    const bool bf = dtype == FA2_BF16;
    if (d == 128)
        return bf ? launch<128, true, true>(dev, mq, mk, mv, p, grid, stream)
                  : launch<128, false, true>(dev, mq, mk, mv, p, grid, stream);
    return bf ? launch<64, true, true>(dev, mq, mk, mv, p, grid, stream)
              : launch<64, false, true>(dev, mq, mk, mv, p, grid, stream);
}

// FP8 counterpart of fwd_general (d = 128).
fa2_status fwd_fp8_general(const void* q, const void* k, const void* v, const float* q_descale,
                           const float* k_descale, const float* v_descale, void* o, float* lse, int B, int H_q,
                           int H_kv, int N_q, int N_k, float scale, int causal, cudaStream_t stream) {
    const long long heads_q = static_cast<long long>(B) * H_q;
    const long long rows_q = heads_q * N_q;
    const long long rows_kv = static_cast<long long>(B) * H_kv * N_k;
    const long long tq = (N_q + fa2::kBM - 1) / fa2::kBM;
    const long long items = heads_q * ((tq + fa2::kNQ - 1) / fa2::kNQ);
    // Item indices stay below 2^31 - 4096 so that a CTA's next index (at most
    // two grids further) never overflows.
    if (rows_q > 0x7FFFFFFFLL || rows_kv > 0x7FFFFFFFLL || items > 0x7FFFFFFFLL - 4096) return FA2_ERR_UNSUPPORTED;

    int dev = 0;
    fa2_status st = check_device(&dev);
    if (st != FA2_OK) return st;
    if ((st = get_encoder()) != FA2_OK) return st;

    CUtensorMap mq, mk, mv;
    const uint64_t hkv = static_cast<uint64_t>(B) * H_kv;
    if (encode_map_u8_3d(&mq, q, static_cast<uint64_t>(heads_q), static_cast<uint64_t>(N_q)) != FA2_OK ||
        encode_map_u8_3d(&mk, k, hkv, static_cast<uint64_t>(N_k)) != FA2_OK ||
        encode_map_u8_3d(&mv, v, hkv, static_cast<uint64_t>(N_k)) != FA2_OK)
        return cuda_fail();

    Params p{};
    p.o = o;
    p.lse = lse;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.debug_flags = g_debug_flags.load();
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.nq = N_q;
    p.nk = N_k;
    p.causal = causal;
    p.heads_q = static_cast<int>(heads_q);
    p.hq = H_q;
    p.group = H_q / H_kv;
    p.tq = static_cast<int>(tq);
    p.pairs = static_cast<int>((tq + fa2::kNQ - 1) / fa2::kNQ);
    p.total_items = static_cast<int>(items);
    p.heads_kv = B * H_kv;
    p.rows_q = rows_q;
    p.rows_kv = rows_kv;
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    const dim3 grid(static_cast<unsigned>(std::min<long long>(items, sm_count(dev))));
    return launch_fp8<true>(dev, mq, mk, mv, p, grid, stream);
}

}  // namespace

extern "C" {

fa2_status fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                       int H_kv, int N, int d, float scale, fa2_dtype dtype, cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return FA2_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA2_ERR_INVALID_ARG;
    if (dtype != FA2_BF16 && dtype != FA2_FP16) return FA2_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA2_ERR_UNSUPPORTED;
    if (N % fa2::kBM != 0) return FA2_ERR_UNSUPPORTED;
    if (N == fa2::kBN) return fwd_general(q, k, v, o, lse, B, H_q, H_kv, N, N, d, scale, 0, dtype, stream);
    // TMA coordinates and row indices are 32-bit.
    const long long rows_q = static_cast<long long>(B) * H_q * N;
    const long long groups = static_cast<long long>(B) * H_kv;
    if (rows_q > 0x7FFFFFFFLL) return FA2_ERR_UNSUPPORTED;

    int dev = 0;
    fa2_status st = check_device(&dev);
    if (st != FA2_OK) return st;
    if ((st = get_encoder()) != FA2_OK) return st;

    CUtensorMap mq, mk, mv;
    const uint64_t rows_kv = static_cast<uint64_t>(B) * H_kv * N;
    if (encode_map(&mq, q, static_cast<uint64_t>(rows_q), d) != FA2_OK ||
        encode_map(&mk, k, rows_kv, d) != FA2_OK || encode_map(&mv, v, rows_kv, d) != FA2_OK)
        return cuda_fail();

    Params p{};
    p.o = o;
    p.lse = lse;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.n_kv_tiles = N / fa2::kBN;
    p.q_tiles = (H_q / H_kv) * (N / fa2::kBM);
    p.pairs = (p.q_tiles + fa2::kNQ - 1) / fa2::kNQ;
    p.total_items = static_cast<int>(p.pairs * groups);
    p.kv_rows = N;
    p.heads_kv = B * H_kv;
    p.rows_q = rows_q;
    p.rows_kv = static_cast<long long>(rows_kv);
    p.debug_flags = g_debug_flags.load();
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    // Persistent grid: one CTA per SM (shared memory and TMEM admit one).
    const dim3 grid(static_cast<unsigned>(std::min<long long>(p.total_items, sm_count(dev))));

    const bool bf = dtype == FA2_BF16;
    if (d == 128)
        return bf ? launch<128, true>(dev, mq, mk, mv, p, grid, stream)
                  : launch<128, false>(dev, mq, mk, mv, p, grid, stream);
    if (tile_cfg() & kTileCfgD64Shared)
        return bf ? launch<64, true>(dev, mq, mk, mv, p, grid, stream)
                  : launch<64, false>(dev, mq, mk, mv, p, grid, stream);
    return bf ? launch_d64<true>(dev, mq, mk, mv, p, grid, stream) : launch_d64<false>(dev, mq, mk, mv, p, grid, stream);
}

fa2_status fa2_fwd_fp8(const void* q, const void* k, const void* v, const float* q_descale,
                       const float* k_descale, const float* v_descale, void* o, float* lse, int B, int H_q,
                       int H_kv, int N, int d, float scale, cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse || !q_descale || !k_descale || !v_descale) return FA2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA2_ERR_INVALID_ARG;
    if (!aligned4(q_descale) || !aligned4(k_descale) || !aligned4(v_descale)) return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return FA2_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA2_ERR_INVALID_ARG;
    if (d != fa2::fp8::kD) return FA2_ERR_UNSUPPORTED;
    if (N % fa2::kBM != 0) return FA2_ERR_UNSUPPORTED;
    if (N == fa2::kBN)
        return fwd_fp8_general(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N, N, scale, 0, stream);
    const long long rows_q = static_cast<long long>(B) * H_q * N;
    const long long groups = static_cast<long long>(B) * H_kv;
    if (rows_q > 0x7FFFFFFFLL) return FA2_ERR_UNSUPPORTED;

    int dev = 0;
    fa2_status st = check_device(&dev);
    if (st != FA2_OK) return st;
    if ((st = get_encoder()) != FA2_OK) return st;

    CUtensorMap mq, mk, mv;
    const uint64_t rows_kv = static_cast<uint64_t>(B) * H_kv * N;
    if (encode_map_u8(&mq, q, static_cast<uint64_t>(rows_q)) != FA2_OK || encode_map_u8(&mk, k, rows_kv) != FA2_OK ||
        encode_map_u8(&mv, v, rows_kv) != FA2_OK)
        return cuda_fail();

    Params p{};
    p.o = o;
    p.lse = lse;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.n_kv_tiles = N / fa2::kBN;
    p.q_tiles = (H_q / H_kv) * (N / fa2::kBM);
    p.pairs = (p.q_tiles + fa2::kNQ - 1) / fa2::kNQ;
    p.total_items = static_cast<int>(p.pairs * groups);
    p.kv_rows = N;
    p.heads_kv = B * H_kv;
    p.rows_q = rows_q;
    p.rows_kv = static_cast<long long>(rows_kv);
    p.debug_flags = g_debug_flags.load();
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    const dim3 grid(static_cast<unsigned>(std::min<long long>(p.total_items, sm_count(dev))));
    return launch_fp8<false>(dev, mq, mk, mv, p, grid, stream);
}

fa2_status fa2_fwd_fp8_ex(const void* q, const void* k, const void* v, const float* q_descale,
                          const float* k_descale, const float* v_descale, void* o, float* lse, int B, int H_q,
                          int H_kv, int N_q, int N_k, int d, float scale, int causal, cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse || !q_descale || !k_descale || !v_descale) return FA2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA2_ERR_INVALID_ARG;
    if (!aligned4(q_descale) || !aligned4(k_descale) || !aligned4(v_descale)) return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_q <= 0 || N_k <= 0 || d <= 0) return FA2_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA2_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
    if (d != fa2::fp8::kD) return FA2_ERR_UNSUPPORTED;
    // The plain case is the multiple-of-128 kernel.
    if (!causal && N_q == N_k && N_q % fa2::kBM == 0)
        return fa2_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N_q, d, scale, stream);
    return fwd_fp8_general(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N_q, N_k, scale, causal,
                           stream);
}

fa2_status fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                   int d, float scale, fa2_dtype dtype, cudaStream_t stream) {
    return fa2_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, dtype, stream);
}

fa2_status fa2_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                      int H_kv, int N_q, int N_k, int d, float scale, int causal, fa2_dtype dtype,
                      cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_q <= 0 || N_k <= 0 || d <= 0) return FA2_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA2_ERR_INVALID_ARG;
    if (dtype != FA2_BF16 && dtype != FA2_FP16) return FA2_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA2_ERR_UNSUPPORTED;
    // The plain case is the multiple-of-128 kernel.
    if (!causal && N_q == N_k && N_q % fa2::kBM == 0)
        return fa2_fwd_gqa(q, k, v, o, lse, B, H_q, H_kv, N_q, d, scale, dtype, stream);
    return fwd_general(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, scale, causal, dtype, stream);
}

}  // extern "C"

namespace {

// The argument and size checks that fa2_bwd and fa2_bwd_noalloc share (every
// pointer but fa2_bwd's `delta`), in the order the header documents:
// FA2_ERR_INVALID_ARG before FA2_ERR_UNSUPPORTED.
fa2_status bwd_check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N, int d,
                          float scale, int causal, fa2_dtype dtype) {
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (const void* x : ptrs)
        if (!x || !aligned16(x)) return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return FA2_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FA2_ERR_INVALID_ARG;
    if (dtype != FA2_BF16 && dtype != FA2_FP16) return FA2_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA2_ERR_UNSUPPORTED;
    const long long rows_q = static_cast<long long>(B) * H_q * N;
    if (rows_q > 0x7FFFFFFFLL || static_cast<long long>(B) * H_q > 65535) return FA2_ERR_UNSUPPORTED;
    return FA2_OK;
}

// The backward's three launches on checked arguments and a checked device.
fa2_status bwd_launch(int dev, const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H_q, int H_kv,
                      int N, int d, float scale, int causal, fa2_dtype dtype, cudaStream_t stream) {
    fa2_status st = get_encoder();
    if (st != FA2_OK) return st;
    const long long rows_q = static_cast<long long>(B) * H_q * N;
    // [heads, N, d] views: tiles never cross heads; rows past a ragged N read as 0
    CUtensorMap mq, mk, mv, mdo;
    const uint64_t hq = static_cast<uint64_t>(B) * H_q, hkv = static_cast<uint64_t>(B) * H_kv;
    const uint64_t n = static_cast<uint64_t>(N);
    if (encode_map_3d(&mq, q, hq, n, d) != FA2_OK || encode_map_3d(&mk, k, hkv, n, d) != FA2_OK ||
        encode_map_3d(&mv, v, hkv, n, d) != FA2_OK || encode_map_3d(&mdo, dout, hq, n, d) != FA2_OK)
        return FA2_ERR_CUDA;

    fa2::bwd::Params p{};
    p.o = o;
    p.lse = lse;
    p.dout = dout;
    p.delta = delta;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.debug_flags = g_debug_flags.load();
    p.n = N;
    p.n_tiles = (N + fa2::kBM - 1) / fa2::kBM;
    p.hq = H_q;
    p.group = H_q / H_kv;
    p.causal = causal;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.heads_q = B * H_q;
    p.heads_kv = B * H_kv;
    p.rows_q = rows_q;
    p.rows_kv = static_cast<long long>(B) * H_kv * N;
    const bool bf = dtype == FA2_BF16;
    const dim3 gdelta(static_cast<unsigned>((rows_q + 15) / 16));
    // dK/dV and dQ: persistent, one CTA per SM over the key (query) tiles,
    // in pairs of equal total cost under the causal mask
    const long long kv_units = static_cast<long long>(causal ? (p.n_tiles + 1) / 2 : p.n_tiles) * B * H_kv;
    const dim3 gkv(static_cast<unsigned>(std::min<long long>(kv_units, sm_count(dev))));
    const long long q_units = static_cast<long long>(causal ? (p.n_tiles + 1) / 2 : p.n_tiles) * B * H_q;
    const dim3 gq(static_cast<unsigned>(std::min<long long>(q_units, sm_count(dev))));

    auto run = [&](auto delta_k, auto dkdv_k, auto dq_k, int smem_kv, int smem_q, int slot) -> fa2_status {
        fa2_status s = set_smem(dev, slot, dkdv_k, smem_kv);
        if (s == FA2_OK) s = set_smem(dev, slot + 6, dq_k, smem_q);
        if (s == FA2_OK) s = launch_kernel(delta_k, gdelta, 256, 0, stream, o, dout, delta, rows_q);
        if (s == FA2_OK) s = launch_kernel(dkdv_k, gkv, fa2::bwd::kThreads, smem_kv, stream, mq, mk, mv, mdo, p);
        if (s == FA2_OK) s = launch_kernel(dq_k, gq, fa2::bwd::kThreads, smem_q, stream, mq, mk, mv, mdo, p);
        return s;
    };
    using namespace fa2::bwd;
    if (d == 128)
        return bf ? run(fa2_bwd_delta_kernel<128, true>, fa2_bwd_dkdv_kernel<128, true>, fa2_bwd_dq_kernel<128, true>,
                        DkdvLayout<128>::kSmemBytes, DqLayout<128>::kSmemBytes, 8)
                  : run(fa2_bwd_delta_kernel<128, false>, fa2_bwd_dkdv_kernel<128, false>,
                        fa2_bwd_dq_kernel<128, false>, DkdvLayout<128>::kSmemBytes, DqLayout<128>::kSmemBytes, 9);
    return bf ? run(fa2_bwd_delta_kernel<64, true>, fa2_bwd_dkdv_kernel<64, true>, fa2_bwd_dq_kernel<64, true>,
                    DkdvLayout<64>::kSmemBytes, DqLayout<64>::kSmemBytes, 10)
              : run(fa2_bwd_delta_kernel<64, false>, fa2_bwd_dkdv_kernel<64, false>, fa2_bwd_dq_kernel<64, false>,
                    DkdvLayout<64>::kSmemBytes, DqLayout<64>::kSmemBytes, 11);
}

}  // namespace

extern "C" {

fa2_status fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H_q, int H_kv,
                   int N, int d, float scale, int causal, fa2_dtype dtype, cudaStream_t stream) {
    if (!delta || !aligned16(delta)) return FA2_ERR_INVALID_ARG;
    fa2_status st = bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N, d, scale, causal, dtype);
    if (st != FA2_OK) return st;
    int dev = 0;
    if ((st = check_device(&dev)) != FA2_OK) return st;
    return bwd_launch(dev, q, k, v, o, lse, dout, dq, dk, dv, delta, B, H_q, H_kv, N, d, scale, causal, dtype,
                      stream);
}

}  // extern "C"

// ---------------------------------------------------------------- backward without allocation

// Scratch for fa2_bwd_noalloc: the per-row D = rowsum(dO o O) of the
// backward, for at most kNoAllocMaxRows query rows (4 MiB of fp32). Every GPU
// that loads this library keeps this array until the process exits. In host
// code the name stands for the array but is not its device address: that
// comes from cudaGetSymbolAddress, asked on every call with the caller's
// device current, so the address always belongs to the context the kernels
// run in (after cudaDeviceReset, or under another context, the array may
// live elsewhere).
static constexpr long long kNoAllocMaxRows = 1LL << 20;
static __device__ __align__(256) float fa2_noalloc_delta[kNoAllocMaxRows];

extern "C" {

fa2_status fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N,
                           int d, float scale, int causal, fa2_dtype dtype, cudaStream_t stream) {
    // fa2_bwd's checks first, so the same arguments give the same errors.
    fa2_status st = bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N, d, scale, causal, dtype);
    if (st != FA2_OK) return st;
    int dev = 0;
    if ((st = check_device(&dev)) != FA2_OK) return st;
    if (static_cast<long long>(B) * H_q * N > kNoAllocMaxRows) return FA2_ERR_UNSUPPORTED;
    // The array's address in the current context (a host-side lookup; the
    // first one on a device may load this library's device code there).
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, fa2_noalloc_delta) != cudaSuccess || !ptr) return cuda_fail();
    // D is written in full by the first kernel of the backward before it is
    // read, so nothing left from an earlier call needs clearing.
    return bwd_launch(dev, q, k, v, o, lse, dout, dq, dk, dv, static_cast<float*>(ptr), B, H_q, H_kv, N, d, scale,
                      causal, dtype, stream);
}

fa2_status fa2_check_status(cudaStream_t stream) {
    // The status word read is that of the stream's device; the current
    // device is switched to it for the read and then restored.
    int sdev = 0, cur = 0;
    if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return cuda_fail();
    if (cudaStreamSynchronize(stream) != cudaSuccess) return cuda_fail();
    if (cudaGetDevice(&cur) != cudaSuccess) return cuda_fail();
    if (sdev != cur && cudaSetDevice(sdev) != cudaSuccess) return cuda_fail();
    fa2_status result = FA2_OK;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fa2::g_fa2_status, sizeof(int)) != cudaSuccess) {
        result = cuda_fail();
    } else if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(fa2::g_fa2_status, &zero, sizeof(int)) != cudaSuccess)
            result = cuda_fail();
        else
            result = (v & 0xFF) == FA2_ERR_TIMEOUT || (v & 0xFF) == FA2_ERR_BOUNDS ? static_cast<fa2_status>(v & 0xFF)
                                                                                   : FA2_ERR_CUDA;
    }
    if (sdev != cur && cudaSetDevice(cur) != cudaSuccess) return cuda_fail();
    return result;
}

const char* fa2_status_string(fa2_status s) {
    switch (s) {
        case FA2_OK: return "FA2_OK";
        case FA2_ERR_INVALID_ARG: return "FA2_ERR_INVALID_ARG";
        case FA2_ERR_UNSUPPORTED: return "FA2_ERR_UNSUPPORTED";
        case FA2_ERR_CUDA: return "FA2_ERR_CUDA";
        case FA2_ERR_TIMEOUT: return "FA2_ERR_TIMEOUT";
        case FA2_ERR_BOUNDS: return "FA2_ERR_BOUNDS";
    }
    return "FA2_ERR_UNKNOWN";
}

int64_t fa2_set_wait_limit_ns(int64_t limit_ns) {
    if (limit_ns <= 0) limit_ns = 2000000000LL;
    return g_wait_limit_ns.exchange(limit_ns);
}

int fa2_set_debug_flags(int flags) { return g_debug_flags.exchange(flags); }

int fa2_set_tile_config(int config) {
    if (config < 0 || (config & ~kTileCfgMask) != 0) return -1;
    (void)tile_cfg();   // the environment's value first, so the previous value is the one in effect
    return g_tile_cfg.exchange(config, std::memory_order_acq_rel);
}

#ifdef FA2_DEBUG
const char* fa2_version(void) { return "fa2-sm103a 0.3.0 debug"; }
#else
const char* fa2_version(void) { return "fa2-sm103a 0.3.0"; }
#endif

}  // extern "C"
