// Thin inline-PTX wrappers for the sm_100-family asynchronous machinery used
// by the attention kernel: mbarriers, TMA tensor copies, tcgen05 MMAs and
// tensor memory (TMEM). Written from the PTX ISA's descriptions of these
// instructions; every wrapper is one instruction (or a fixed short sequence).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa2 {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float ld_volatile_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.volatile.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// true once the phase with the given parity has completed
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of phase `parity` of an mbarrier.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled copy global -> shared, completion counted in bytes on `bar`.
// x is the innermost (contiguous) coordinate in elements, y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 3-D tiled copy global -> shared: x innermost element, y row, z matrix.
// Rows past the tensor's extent are filled with zeros (and still counted in
// the transaction bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Prefetch a 2-D tile into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y)
                 : "memory");
}

// ------------------------------------------------------------------ registers

// Warpgroup-wide register reallocation: every warp of the warpgroup executes
// the same instruction. The grants of all warpgroups must add up to the
// per-thread budget the block was launched with.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ tcgen05 / TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// A whole K-loop of one GEMM (4 or 8 MMAs of K = 16) in one sequence: one
// elect.sync, the accumulate predicates set once, and each step's descriptor
// offsets (16-byte units, compile-time immediates) added to the low words of
// the base descriptors. The start-address field occupies the low 14 bits and
// every address stays below 256 KB, so the low-word add never carries.
// Step 0 accumulates iff `acc`; later steps always accumulate.
template <uint32_t A1, uint32_t A2, uint32_t A3, uint32_t A4, uint32_t A5, uint32_t A6, uint32_t A7,
          uint32_t B1, uint32_t B2, uint32_t B3, uint32_t B4, uint32_t B5, uint32_t B6, uint32_t B7, int NSTEP>
__device__ __forceinline__ void mma_ss_kloop(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t acc) {
    static_assert(NSTEP == 4 || NSTEP == 8, "4 or 8 steps");
    if constexpr (NSTEP == 8) {
        asm volatile(
            "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 alo, ahi, blo, bhi, t0, t1;\n\t.reg .b64 a, b;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\t"
            "setp.eq.b32 pt, %4, %4;\n\t"
            "mov.b64 {alo, ahi}, %1;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
            "add.u32 t0, alo, %5;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %12;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %6;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %13;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %7;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %14;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %8;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %15;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %9;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %16;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %10;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %17;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %11;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %18;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "}" ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc),
            "n"(A1), "n"(A2), "n"(A3), "n"(A4), "n"(A5), "n"(A6), "n"(A7),
            "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 alo, ahi, blo, bhi, t0, t1;\n\t.reg .b64 a, b;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\t"
            "setp.eq.b32 pt, %4, %4;\n\t"
            "mov.b64 {alo, ahi}, %1;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
            "add.u32 t0, alo, %5;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %8;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %6;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %9;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "add.u32 t0, alo, %7;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, %10;\n\tmov.b64 b, {t1, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
            "}" ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc),
            "n"(A1), "n"(A2), "n"(A3), "n"(B1), "n"(B2), "n"(B3)
            : "memory");
    }
}

// Same for O += P V with P (A) read from TMEM: 8 steps, A advances 8
// columns and B (V, MN-major) 2048 bytes per step.
__device__ __forceinline__ void mma_ts_kloop8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 blo, bhi, t0, t1;\n\t.reg .b64 b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.eq.b32 pt, %4, %4;\n\t"
        "mov.b64 {blo, bhi}, %2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
        "add.u32 t0, %1, 8;\n\tadd.u32 t1, blo, 128;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 16;\n\tadd.u32 t1, blo, 256;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 24;\n\tadd.u32 t1, blo, 384;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 32;\n\tadd.u32 t1, blo, 512;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 40;\n\tadd.u32 t1, blo, 640;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 48;\n\tadd.u32 t1, blo, 768;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 56;\n\tadd.u32 t1, blo, 896;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with A in two 32-column halves 64 columns apart: K-steps 0-3
// read A columns 0..31, steps 4-7 columns 64..95 (each half of a row's
// 16-bit values packed inside the fp32 columns it was computed from).
__device__ __forceinline__ void mma_ts_kloop8_split(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                    uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 blo, bhi, t0, t1;\n\t.reg .b64 b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.eq.b32 pt, %4, %4;\n\t"
        "mov.b64 {blo, bhi}, %2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
        "add.u32 t0, %1, 8;\n\tadd.u32 t1, blo, 128;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 16;\n\tadd.u32 t1, blo, 256;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 24;\n\tadd.u32 t1, blo, 384;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 64;\n\tadd.u32 t1, blo, 512;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 72;\n\tadd.u32 t1, blo, 640;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 80;\n\tadd.u32 t1, blo, 768;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 88;\n\tadd.u32 t1, blo, 896;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b, %3, pt;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed. Warp-collective: the converged warp executes it, elect.sync
// picks the lane that commits (the same lane that issues the MMAs, so the
// commit covers them), and the operands stay warp-uniform.
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM
// lane (lane = warp's lane quarter base + laneid).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}


// Offset forms of the 32-column load/store that read or write a slice of a
// larger register array; OFF must be a compile-time constant so the array
// stays in registers.
template <int OFF, int NREG>
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&r)[NREG]) {
    static_assert(OFF + 32 <= NREG, "slice out of range");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]),
          "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]),
          "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]),
          "=r"(r[OFF + 14]), "=r"(r[OFF + 15]), "=r"(r[OFF + 16]), "=r"(r[OFF + 17]),
          "=r"(r[OFF + 18]), "=r"(r[OFF + 19]), "=r"(r[OFF + 20]), "=r"(r[OFF + 21]),
          "=r"(r[OFF + 22]), "=r"(r[OFF + 23]), "=r"(r[OFF + 24]), "=r"(r[OFF + 25]),
          "=r"(r[OFF + 26]), "=r"(r[OFF + 27]), "=r"(r[OFF + 28]), "=r"(r[OFF + 29]),
          "=r"(r[OFF + 30]), "=r"(r[OFF + 31])
        : "r"(taddr));
}

template <int OFF, int NREG>
__device__ __forceinline__ void tmem_st32_at(uint32_t taddr, const uint32_t (&r)[NREG]) {
    static_assert(OFF + 32 <= NREG, "slice out of range");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[OFF + 0]), "r"(r[OFF + 1]), "r"(r[OFF + 2]), "r"(r[OFF + 3]), "r"(r[OFF + 4]),
        "r"(r[OFF + 5]), "r"(r[OFF + 6]), "r"(r[OFF + 7]), "r"(r[OFF + 8]), "r"(r[OFF + 9]),
        "r"(r[OFF + 10]), "r"(r[OFF + 11]), "r"(r[OFF + 12]), "r"(r[OFF + 13]), "r"(r[OFF + 14]),
        "r"(r[OFF + 15]), "r"(r[OFF + 16]), "r"(r[OFF + 17]), "r"(r[OFF + 18]), "r"(r[OFF + 19]),
        "r"(r[OFF + 20]), "r"(r[OFF + 21]), "r"(r[OFF + 22]), "r"(r[OFF + 23]), "r"(r[OFF + 24]),
        "r"(r[OFF + 25]), "r"(r[OFF + 26]), "r"(r[OFF + 27]), "r"(r[OFF + 28]), "r"(r[OFF + 29]),
        "r"(r[OFF + 30]), "r"(r[OFF + 31])
        : "memory");
}

// The same 32-column load that also returns, per thread, the maximum of the
// 32 fp32 values it loaded (tcgen05.ld.red, an sm_103a instruction): the
// row max of a score tile comes out of the TMEM loads instead of a tree of
// max instructions.
template <int OFF, int NREG>
__device__ __forceinline__ void tmem_ld32_max_at(uint32_t taddr, uint32_t (&r)[NREG], float& mx) {
    static_assert(OFF + 32 <= NREG, "slice out of range");
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
        : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]),
          "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]),
          "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]),
          "=r"(r[OFF + 14]), "=r"(r[OFF + 15]), "=r"(r[OFF + 16]), "=r"(r[OFF + 17]),
          "=r"(r[OFF + 18]), "=r"(r[OFF + 19]), "=r"(r[OFF + 20]), "=r"(r[OFF + 21]),
          "=r"(r[OFF + 22]), "=r"(r[OFF + 23]), "=r"(r[OFF + 24]), "=r"(r[OFF + 25]),
          "=r"(r[OFF + 26]), "=r"(r[OFF + 27]), "=r"(r[OFF + 28]), "=r"(r[OFF + 29]),
          "=r"(r[OFF + 30]), "=r"(r[OFF + 31]), "=f"(mx)
        : "r"(taddr));
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor for tcgen05.mma with the 128-byte swizzle:
// start address, leading- and stride-dimension byte offsets (all >> 4), the
// descriptor version bit (46) and the swizzle mode (61..63 = 2 for 128 B).
// The tile must sit on a 1024-byte boundary (the swizzle pattern's period).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for tcgen05.mma with fp32 accumulation.
// ab_type: with kind::f16 0 = fp16, 1 = bf16; with kind::f8f6f4 0 = e4m3. a_mn / b_mn: operand is MN-major (1) or
// K-major (0). M in {64, 128}, N a multiple of 16 up to 256.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_type, uint32_t a_mn, uint32_t b_mn,
                                                 uint32_t M, uint32_t N) {
    return (1u << 4)                 // D format: f32
           | (ab_type << 7)          // A format
           | (ab_type << 10)         // B format
           | (a_mn << 15)            // A major
           | (b_mn << 16)            // B major
           | ((N >> 3) << 17)        // N / 8
           | ((M >> 4) << 24);       // M / 16
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32 pairs (sm_100 family): a 64-bit register holds {lo, hi} and one
// instruction applies the operation to both halves with fp32 rounding.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}


// exp2 of a pair of x <= 0 on the FMA pipe instead of the MUFU, for a share
// of the softmax's exponentials. Cody-Waite range reduction (Cody and Waite,
// "Software Manual for the Elementary Functions", 1980): x = n + f with n the
// nearest integer (by adding and subtracting 1.5 * 2^23) and |f| <= 1/2; 2^f
// by a degree-3 polynomial with constant term exactly 1 whose other
// coefficients are a relative-error minimax fit on [-1/2, 1/2] computed for
// this kernel (max relative error 1.0e-4); 2^n is applied by adding n << 23 to
// the result's bit pattern. x is clamped to -125 first so the scaled result
// stays a normal number; exp2(0) is exactly 1.
__device__ __forceinline__ uint64_t ex2_poly_f2(uint64_t x2) {
    float x0, x1;
    f2_unpack(x2, x0, x1);
    x0 = fmaxf(x0, -125.0f);
    x1 = fmaxf(x1, -125.0f);
    const uint64_t xc = f2_pack(x0, x1);
    const uint64_t t = f2_add(xc, f2_pack(12582912.0f, 12582912.0f));
    const uint64_t r = f2_add(t, f2_pack(-12582912.0f, -12582912.0f));
    const uint64_t f = f2_fma(r, f2_pack(-1.0f, -1.0f), xc);
    uint64_t p = f2_fma(f2_pack(0.055009059607982635f, 0.055009059607982635f), f,
                        f2_pack(0.2422109693288803f, 0.2422109693288803f));
    p = f2_fma(p, f, f2_pack(0.6932829022407532f, 0.6932829022407532f));
    p = f2_fma(p, f, f2_pack(1.0f, 1.0f));
    float p0, p1, t0, t1;
    f2_unpack(p, p0, p1);
    f2_unpack(t, t0, t1);
    // bits(t) = bits(1.5 * 2^23) + n and bits(1.5 * 2^23) << 23 vanishes mod 2^32
    const uint32_t b0 = __float_as_uint(t0) * 8388608u + __float_as_uint(p0);
    const uint32_t b1 = __float_as_uint(t1) * 8388608u + __float_as_uint(p1);
    return f2_pack(__uint_as_float(b0), __uint_as_float(b1));
}

// Widen a 16-bit pair (lo in bits 0..15) to two fp32 values, exactly.
template <bool kBf16>
__device__ __forceinline__ void unpack2(uint32_t v, float& lo, float& hi) {
    if constexpr (kBf16) {
        lo = __uint_as_float(v << 16);
        hi = __uint_as_float(v & 0xFFFF0000u);
    } else {
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(v));
    }
}

// Pack two fp32 values into a 16-bit pair: `lo` in bits 0..15, `hi` in 16..31,
// each rounded to nearest-even. kBf16 selects bf16, otherwise fp16.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (kBf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------- 8-bit (kind::f8f6f4)

// S (+)= A B^T over one 128-byte K extent of e4m3 operands: 4 MMAs of K = 32,
// both operands K-major with the 128-byte swizzle; step kk starts 32*kk bytes
// into the rows (+2 per step in the descriptors' 16-byte units). Step 0
// accumulates iff `acc`. idesc carries the operand formats (e4m3 = 0).
__device__ __forceinline__ void mma_ss_kloop4_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 alo, ahi, blo, bhi, t0, t1;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.eq.b32 pt, %4, %4;\n\t"
        "mov.b64 {alo, ahi}, %1;\n\t"
        "mov.b64 {blo, bhi}, %2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p0;\n\t"
        "add.u32 t0, alo, 2;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, 2;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, pt;\n\t"
        "add.u32 t0, alo, 4;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, 4;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, pt;\n\t"
        "add.u32 t0, alo, 6;\n\tmov.b64 a, {t0, ahi};\n\tadd.u32 t1, blo, 6;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, pt;\n\t"
        "}" ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// O (+)= P V with P (e4m3, four per 32-bit column) read from TMEM and V
// MN-major in shared memory (rows of 128 one-byte values, 128-byte swizzle):
// 4 MMAs of K = 32; A advances 8 columns and B 32 rows (4096 B) per step.
__device__ __forceinline__ void mma_ts_kloop4_f8_mn(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                    uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 blo, bhi, t0, t1;\n\t.reg .b64 b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.eq.b32 pt, %4, %4;\n\t"
        "mov.b64 {blo, bhi}, %2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p0;\n\t"
        "add.u32 t0, %1, 8;\n\tadd.u32 t1, blo, 256;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 16;\n\tadd.u32 t1, blo, 512;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [t0], b, %3, pt;\n\t"
        "add.u32 t0, %1, 24;\n\tadd.u32 t1, blo, 768;\n\tmov.b64 b, {t1, bhi};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [t0], b, %3, pt;\n\t"
        "}" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Four fp32 values to four e4m3 bytes, x0 in bits 0..7: round to nearest
// even, saturating at +-448 (the conversion puts its first source in the
// upper byte of each 16-bit half).
__device__ __forceinline__ uint32_t pack4_e4m3(float x0, float x1, float x2, float x3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
    return r;
}

}  // namespace ptx
}  // namespace fa2
