// sv_device.cuh -- device helpers shared by the sv kernels (sm_103a).
//
// PTX wrappers for mbarriers, bulk / tensor (TMA) copies, ldmatrix and the
// bf16 mma; and the single-precision building blocks of the sampled
// acceptance whose arithmetic is fixed so that a host implementation can
// reproduce every decision bit for bit:
//   * sv_exp      Cody-Waite reduction (Cody & Waite, "Software Manual for the
//                 Elementary Functions", 1980) + degree-7 Taylor polynomial;
//   * philox4x32_10  Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
//                 3", SC'11;
//   * canonical pairwise summation: leaves are the vocab entries zero-padded
//                 to a power of two, each tree node is the float sum of its
//                 two contiguous halves.
// All float arithmetic that decides an integer uses the explicitly rounded
// intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn, __fmaf_rn) so the compiler
// cannot contract or reassociate it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sv.h"

namespace sv {

// --------------------------------------------------------------------------
// error word
// --------------------------------------------------------------------------

__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

// Self-checks compiled in with -DSV_DEBUG: a failed check sets bit 31 and
// the check's code (bits 8..23) in the error word -- above the public
// SV_DEVERR_* bits -- and the guarded access is skipped.  Without SV_DEBUG
// the checks vanish.
#ifdef SV_DEBUG
__device__ __forceinline__ bool sv_check(bool ok, unsigned int* err, unsigned int code) {
    if (!ok) raise_error(err, 0x80000000u | (1u << (8 + (code & 15))));
    return ok;
}
#define SV_CHECK(cond, err, code) ::sv::sv_check((cond), (err), (code))
#else
#define SV_CHECK(cond, err, code) true
#endif

// --------------------------------------------------------------------------
// addresses, timers
// --------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// --------------------------------------------------------------------------
// mbarrier + bulk copies
// --------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of an mbarrier phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~2 s of wall time (or a
// large iteration count), raises SV_DEVERR_TIMEOUT and returns false.  The
// copies these barriers track cannot fail short of a device fault, so the
// bound only guarantees that no kernel of this library can spin forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) break;
    }
    raise_error(err, SV_DEVERR_TIMEOUT);
    return false;
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all
// of this thread's outstanding copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled tensor copy (TMA) global -> shared, completing on `bar`.
// x (innermost coordinate) times the element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// max(a, b, c) in one instruction (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Three-input minimum that is NaN if any input is NaN (max.f32 and min.f32
// without .NaN return the other operand instead).
__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
    float r;
    asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Bulk prefetch of [p, p + bytes) into L2: a hint that moves no data into
// the CTA.  p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Split cluster barrier.  Every CTA of a cluster must have started before any
// CTA touches another's shared memory: arrive early, wait right before the
// first distributed-shared-memory access.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Full cluster barrier with release / acquire ordering of shared-memory
// writes (local and remote).  Warp-collective (.aligned): call it from
// converged warps only -- a warp whose other lanes are still busy (a lone
// producer lane) must __syncwarp() first.
__device__ __forceinline__ void cluster_sync_warp() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------------
// tensor-core fragments (mma.sync m16n8k16, bf16 in, fp32 accumulate)
// --------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x via the SFU (attention softmax only; not used where bits must match).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Address of 16-byte chunk `chunk` (0..7) of row `row` inside a TMA box of
// 128-byte rows written with CU_TENSOR_MAP_SWIZZLE_128B (box base 1024-aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t box_base, int row, int chunk) {
    return box_base + row * 128 + (((chunk ^ (row & 7)) & 7) << 4);
}

// --------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// --------------------------------------------------------------------------

// Allocates `ncols` TMEM columns (power of two >= 32); one full warp calls it
// and the base address is written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile
// (start address, leading and stride byte offsets; descriptor version 1).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // version
    d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// M x N tile; a_mn / b_mn select the MN-major (transposed) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                   // D: f32
           | (1u << 7)                                 // A: bf16
           | (1u << 10)                                // B: bf16
           | (static_cast<uint32_t>(a_mn) << 15)
           | (static_cast<uint32_t>(b_mn) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M rows = TMEM lanes, K-major, two bf16
// per 32-bit column) read from tensor memory, issued by one thread.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// tcgen05.ld of 16 columns and its wait in one statement, so the registers
// cannot be used before the load has landed.
__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane and the wait, as a
// single statement.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 64 columns (four x16 loads) and one wait, as a single statement.
__device__ __forceinline__ void tmem_ld64_sync(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr), "r"(taddr + 16), "r"(taddr + 32), "r"(taddr + 48)
        : "memory");
}

// Writes 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Half-lane shape 16x32bx2: a warp touches the first 16 lanes of its TMEM
// quadrant; threads 0..15 read lane (base + t) at columns c.., threads 16..31
// read lane (base + t - 16) at columns c + OFF.. (register k = column + k).
// Two threads per row, each with its own column range.
template <int OFF>
__device__ __forceinline__ void tmem_ld16_h_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "n"(OFF)
        : "memory");
}

// 32 columns per thread (two x16 half-lane loads at c and c + 16) and one wait.
template <int OFF>
__device__ __forceinline__ void tmem_ld32_h_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32], %34;\n\t"
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33], %34;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr), "r"(taddr + 16), "n"(OFF)
        : "memory");
}

template <int OFF>
__device__ __forceinline__ void tmem_st16_h(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %17, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "n"(OFF)
        : "memory");
}

template <int OFF>
__device__ __forceinline__ void tmem_st8_h(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x8.b32 [%0], %9, {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "n"(OFF)
                 : "memory");
}

// Barrier over a subset of the CTA's warps (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// --------------------------------------------------------------------------
// exponential with a fixed operation sequence
// --------------------------------------------------------------------------

__device__ __forceinline__ float sv_exp(float x) {
    if (x != x) return x;
    if (x < -104.0f) return 0.0f;                 // below half the least subnormal
    if (x > 88.0f) return __int_as_float(0x7f800000);
    const float kInvLn2 = 1.44269504088896340736f;
    const float kLn2Head = 0.693145751953125f;    // 12 significant bits: n * head exact
    const float kLn2Tail = 1.428606820309417232e-06f;
    // n = rint(x / ln 2): adding 1.5 * 2^23 rounds to an integer (ties to even)
    // and leaves it in the low mantissa bits, which gives k without a convert
    const float kRound = 12582912.0f;
    const float t = __fadd_rn(__fmul_rn(x, kInvLn2), kRound);
    const float n = __fsub_rn(t, kRound);
    float r = __fmaf_rn(-n, kLn2Head, x);
    r = __fmaf_rn(-n, kLn2Tail, r);
    float s = 1.0f / 5040.0f;                      // Taylor coefficients 1/k!
    s = __fmaf_rn(s, r, 1.0f / 720.0f);
    s = __fmaf_rn(s, r, 1.0f / 120.0f);
    s = __fmaf_rn(s, r, 1.0f / 24.0f);
    s = __fmaf_rn(s, r, 1.0f / 6.0f);
    s = __fmaf_rn(s, r, 0.5f);
    s = __fmaf_rn(s, r, 1.0f);
    s = __fmaf_rn(s, r, 1.0f);
    const int k = __float_as_int(t) - __float_as_int(kRound);
    if (k >= -126) return __fmul_rn(s, __int_as_float((k + 127) << 23));
    // 2^k subnormal: an exact scaling by 2^(k+64), then one rounding by 2^-64
    return __fmul_rn(__fmul_rn(s, __int_as_float((k + 64 + 127) << 23)), __int_as_float((127 - 64) << 23));
}

// sv_exp without branches, for the softmax terms exp(z - M) (argument <= 0):
// the same operations on max(x, -104), so several evaluations can interleave;
// below -104 the clamped evaluation is exp(-104) ~ 6.8e-46, which rounds to 0
// like sv_exp's underflow return.  The scaling by 2^k is always done as
// 2^(k+64) (exact: the product is normal) and then 2^-64, whose single rounding
// is the one sv_exp's subnormal branch performs, and which is exact whenever
// the result is normal.  Bit-identical to sv_exp for every x <= 0 that is not
// NaN (for x above ~44, 2^(k+64) would overflow).
__device__ __forceinline__ float sv_exp_nb(float x) {
    const float kInvLn2 = 1.44269504088896340736f;
    const float kLn2Head = 0.693145751953125f;
    const float kLn2Tail = 1.428606820309417232e-06f;
    const float kRound = 12582912.0f;   // as in sv_exp
    const float xc = fmaxf(x, -104.0f);
    const float t = __fadd_rn(__fmul_rn(xc, kInvLn2), kRound);
    const float n = __fsub_rn(t, kRound);
    float r = __fmaf_rn(-n, kLn2Head, xc);
    r = __fmaf_rn(-n, kLn2Tail, r);
    float s = 1.0f / 5040.0f;
    s = __fmaf_rn(s, r, 1.0f / 720.0f);
    s = __fmaf_rn(s, r, 1.0f / 120.0f);
    s = __fmaf_rn(s, r, 1.0f / 24.0f);
    s = __fmaf_rn(s, r, 1.0f / 6.0f);
    s = __fmaf_rn(s, r, 0.5f);
    s = __fmaf_rn(s, r, 1.0f);
    s = __fmaf_rn(s, r, 1.0f);
    const int k = __float_as_int(t) - __float_as_int(kRound);
    return __fmul_rn(__fmul_rn(s, __int_as_float((k + 64 + 127) << 23)), __int_as_float((127 - 64) << 23));
}

// sv_exp for -86.5 < x <= 0, where every result is a normal number: the same
// reduction and polynomial, then s * 2^k as an addition of k to the exponent
// field of s.  There, k >= -125 and s lies in [0.707, 1.415], so s * 2^k is
// normal and the multiplication by 2^k is exact: the field addition gives the
// same bits as sv_exp's rounded product, without the clamp and the two
// multiplies of sv_exp_nb.
__device__ __forceinline__ float sv_exp_nrm(float x) {
    const float kInvLn2 = 1.44269504088896340736f;
    const float kLn2Head = 0.693145751953125f;
    const float kLn2Tail = 1.428606820309417232e-06f;
    const float kRound = 12582912.0f;   // as in sv_exp
    const float t = __fadd_rn(__fmul_rn(x, kInvLn2), kRound);
    const float n = __fsub_rn(t, kRound);
    float r = __fmaf_rn(-n, kLn2Head, x);
    r = __fmaf_rn(-n, kLn2Tail, r);
    float s = 1.0f / 5040.0f;
    s = __fmaf_rn(s, r, 1.0f / 720.0f);
    s = __fmaf_rn(s, r, 1.0f / 120.0f);
    s = __fmaf_rn(s, r, 1.0f / 24.0f);
    s = __fmaf_rn(s, r, 1.0f / 6.0f);
    s = __fmaf_rn(s, r, 0.5f);
    s = __fmaf_rn(s, r, 1.0f);
    s = __fmaf_rn(s, r, 1.0f);
    const uint32_t k = __float_as_uint(t) - __float_as_uint(kRound);   // two's complement of k
    return __uint_as_float(__float_as_uint(s) + (k << 23));
}

// Lower bound of the arguments sv_exp_nrm takes.
constexpr float kExpNormalMin = -86.5f;

// a / b rounded to nearest even, given rb = 1/b rounded to nearest (e.g.
// __frcp_rn(b), formed once per divisor), by Markstein's correction step
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990): q = a rb is
// within about an ulp of a / b, the remainder a - b q is exact in one fused
// multiply-add, and q + (a - b q) rb rounds to a / b.  Taken where a and b
// lie in [2^-60, 2^60], so that every intermediate is a normal number (a probe
// over 4.8e9 quotients there -- every significand of a against 64 special
// divisors at three scales, and random pairs -- matched __fdiv_rn bit for
// bit); elsewhere the correctly rounded division itself.
__device__ __forceinline__ float div_rn_by(float a, float b, float rb) {
    if (a >= 0x1p-60f && a <= 0x1p60f && b >= 0x1p-60f && b <= 0x1p60f) {
        const float q = __fmul_rn(a, rb);
        const float r = __fmaf_rn(-q, b, a);
        return __fmaf_rn(r, rb, q);
    }
    return __fdiv_rn(a, b);
}

// Two-input minimum that is NaN if either input is NaN.
__device__ __forceinline__ float fmin_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// --------------------------------------------------------------------------
// Philox4x32-10
// --------------------------------------------------------------------------

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
    const uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    const uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi_a = __umulhi(kMulA, c.x), lo_a = kMulA * c.x;
        const uint32_t hi_b = __umulhi(kMulB, c.z), lo_b = kMulB * c.z;
        c = make_uint4(hi_b ^ c.y ^ k.x, lo_b, hi_a ^ c.w ^ k.y, lo_a);
        k.x += kWeylA;
        k.y += kWeylB;
    }
    return c;
}

__device__ __forceinline__ float uniform24(uint32_t w) {
    return __fmul_rn(static_cast<float>(w >> 8), 5.9604644775390625e-08f);   // * 2^-24, exact
}

// The acceptance (word 0) and sampling (word 1) uniforms of tree node u.
__device__ __forceinline__ float2 node_uniforms(uint64_t seed, uint64_t step, int b, int u, const float* uniforms,
                                                int R) {
    if (uniforms) {
        const float* p = uniforms + (static_cast<size_t>(b) * R + u) * 2;
        return make_float2(p[0], p[1]);
    }
    const uint4 w = philox4x32_10(
        make_uint4(static_cast<uint32_t>(b), static_cast<uint32_t>(u), static_cast<uint32_t>(step),
                   static_cast<uint32_t>(step >> 32)),
        make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
    return make_float2(uniform24(w.x), uniform24(w.y));
}

// --------------------------------------------------------------------------
// canonical pairwise summation pieces
// --------------------------------------------------------------------------

// Node over 4 contiguous leaves: (a+b) + (c+d).
__device__ __forceinline__ float quad_sum(float4 v) {
    return __fadd_rn(__fadd_rn(v.x, v.y), __fadd_rn(v.z, v.w));
}

// Lane i holds the node over leaves [i*s, (i+1)*s); returns (in every lane)
// the node over all 32*s leaves.  Step `off` pairs lanes i and i^off, which
// are adjacent siblings at that level, and float addition is commutative, so
// both partners hold the same parent value.
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// --------------------------------------------------------------------------
// draft trees
// --------------------------------------------------------------------------

// Children of node u in index order, for a chain (parent == nullptr: the only
// child of u is u+1) or a tree.
__device__ __forceinline__ int next_child(const int* par, int R, int u, int after) {
    if (par == nullptr) return (after < 0 && u + 1 < R) ? u + 1 : -1;
    for (int c = (after < 0 ? u + 1 : after + 1); c < R; ++c)
        if (par[c] == u) return c;
    return -1;
}

// Loads and validates the tree of sequence b into shared memory; returns
// false (and raises SV_DEVERR_TREE) if it is malformed.
__device__ inline bool load_tree(const int32_t* parent, int b, int R, int* par_s, unsigned int* err) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < R; j += blockDim.x) {
        const int p = parent[static_cast<size_t>(b) * R + j];
        par_s[j] = p;
        if ((j == 0 && p != -1) || (j > 0 && (p < 0 || p >= j))) bad = 1;
    }
    __syncthreads();
    const bool ok = bad == 0;
    if (!ok && threadIdx.x == 0) raise_error(err, SV_DEVERR_TREE);
    return ok;
}

// --------------------------------------------------------------------------
// greedy argmax as 64-bit keys
// --------------------------------------------------------------------------
// The greedy token of a row is its largest logit, NaN skipped, ties (and
// -0 == +0) going to the lowest column.  That order is the unsigned order of
//     key(x, col) = (okey(x) << 32) | ~col,
// where okey maps every float other than NaN to an unsigned word in the
// float order (+0 and -0 to the same word) and NaN to 0, below every other
// word; ~col makes the lower column the larger word on equal values.  A
// block of columns is then summarised by the largest key of its entries,
// and the row by the largest key of its blocks' keys.

__device__ __forceinline__ uint32_t argmax_okey(float x) {
    if (x != x) return 0u;
    const uint32_t b = __float_as_uint(__fadd_rn(x, 0.0f));   // -0 + 0 = +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t argmax_key(uint32_t okey, int col) {
    return (static_cast<uint64_t>(okey) << 32) | static_cast<uint32_t>(~col);
}

// Column of the largest key: the complement of its low word; a key whose
// high word is 0 summarises only NaN (or no column), and the row's token is
// then column 0.
__device__ __forceinline__ int argmax_col(uint64_t key) {
    return (key >> 32) == 0 ? 0 : static_cast<int>(~static_cast<uint32_t>(key));
}

// Largest key over the warp's lanes (every lane gets it): two redux steps,
// first the high words, then the low words of the lanes that hold the
// largest high word.
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
    const uint32_t hi = static_cast<uint32_t>(k >> 32), lo = static_cast<uint32_t>(k);
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    return (static_cast<uint64_t>(mhi) << 32) | mlo;
}

}  // namespace sv
