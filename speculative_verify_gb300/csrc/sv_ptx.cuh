// sv_ptx.cuh -- thin inline-PTX wrappers used by the sm_103a kernels:
// mbarriers, bulk and tensor (TMA) copies global -> shared, cp.async,
// L2 cache policies, the fp16 and bf16 tensor-core MMAs and the int4 ->
// fp16x2 / bf16x2 dequantisations.
#pragma once

#include <cstdint>

namespace sv {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of shared memory.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` nanoseconds.  Returns false on time-out; the caller records the
// error and carries on, so no thread ever waits without bound.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- L2 policies

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- bulk / tensor copies

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

// 2-D tiled tensor copy of one box at coordinates (c0 innermost, c1) into
// shared memory (128-byte aligned), completing on `bar`.  Out-of-range parts
// of the box are filled with zeros and still count towards the bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar),
                   "l"(policy)
                 : "memory");
}

// Four rows (r0..r3, any order, out-of-range rows read as zeros) of a 2-D
// tensor map whose box is one row high, columns c0 .. c0 + box width - 1,
// into shared memory as 4 consecutive box rows; completes on `bar`.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void *tmap, int c0, int r0, int r1, int r2, int r3,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
                   "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), L2 only.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// As cp_async_16, with an L2 eviction-policy hint.
__device__ __forceinline__ void cp_async_16_hint(uint32_t dst, const void *src, uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
// The arrival is one of the barrier's expected arrivals (.noinc).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- gpu-scope atomics

// atomicAdd with acquire-release semantics at GPU scope: orders this
// thread's earlier writes before the add and later reads after it.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Release add without a result: the thread does not wait for it.  Writes
// made before it by this thread, and by the threads of its warp ordered
// before it by __syncwarp(), are visible to an acquire load that sees it.
__device__ __forceinline__ void red_add_release_gpu(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Load with acquire semantics at GPU scope: later reads of this thread see
// every write released before the value it returns.
__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float4 ldcg_f4(const float *p)
{
    return __ldcg(reinterpret_cast<const float4 *>(p));
}

// ---------------------------------------------------------------- dependent launch

// Let the next kernel in the stream start launching its CTAs now.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous kernel in the stream has completed and its writes
// are visible (a no-op when this kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait_prior()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- named barriers

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- shared loads

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------- global loads

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h)
{
    return __uint_as_float(h << 16);
}

// ---------------------------------------------------------------- dequant

__device__ __forceinline__ uint32_t mulhi(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two nibbles -> two bf16 levels.  v holds nibble a in bits 0..3 and nibble
// b in bits 16..19 (other bits ignored).  OR-ing a nibble into the mantissa
// of bf16 128.0 (0x4300, where the bf16 spacing is exactly 1) gives 128 + n;
// one packed fma with 1.0 and -136.0 gives n - 8 exactly.  Result: low half
// = level(a), high half = level(b).
__device__ __forceinline__ uint32_t dequant2(uint32_t v)
{
    uint32_t q, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(q) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(0x3F803F80u), "r"(0xC308C308u));
    return r;
}

// fp16 levels.  fp16 1024.0 (0x6400) has spacing 1 and a 10-bit mantissa,
// so a nibble fits either at bits 0..3 (value 1024 + n) or at bits 4..7
// (value 1024 + 16 n) without touching the exponent; a word then needs one
// shift (by 8) for its four nibble pairs instead of three.
// Low position: v holds nibble a in bits 0..3 and b in bits 16..19;
// (1024 + n) * 1 - 1032 = n - 8.
__device__ __forceinline__ uint32_t dequant2_f16_lo(uint32_t v)
{
    uint32_t q, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(q) : "r"(v), "r"(0x000F000Fu), "r"(0x64006400u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(0x3C003C00u), "r"(0xE408E408u));
    return r;
}

// High position: nibble a in bits 4..7 and b in bits 20..23;
// (1024 + 16 n) / 16 - 72 = n - 8.
__device__ __forceinline__ uint32_t dequant2_f16_hi(uint32_t v)
{
    uint32_t q, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(q) : "r"(v), "r"(0x00F000F0u), "r"(0x64006400u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(0x2C002C00u), "r"(0xD480D480u));
    return r;
}

// c + a.lo * b.lo + a.hi * b.hi: two fp16 x fp16 products added to an fp32
// accumulator by the mixed-precision fma (products exact in fp32, each add
// rounded to fp32).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float c)
{
    float d;
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 t, al, bl, %3;\n\tfma.rn.f32.f16 %0, ah, bh, t;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------- tensor core

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (16x8 fp32) = A (16x16 fp16, row) * B (16x8 fp16, col), no accumulator input.
__device__ __forceinline__ void mma_f16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Exponent s for the fp16 copy of an activation row whose largest magnitude
// has bf16 bits mx (sign cleared): 2^s * max lies in [2^14, 2^15), below the
// fp16 maximum 65504.  Clamped to [-120, 120] so that 2^s and 2^-s are normal
// fp32 numbers; 0 for an all-zero row.
__device__ __forceinline__ int xres_shift(unsigned mx)
{
    if (mx == 0u) return 0;
    const int s = 141 - static_cast<int>(mx >> 7);
    return s < -120 ? -120 : (s > 120 ? 120 : s);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Two floats -> fp16x2 (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (16x8 fp32) = A (16x16 bf16, row) * B (16x8 bf16, col), no accumulator input.
__device__ __forceinline__ void mma_bf16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// ---------------------------------------------------------------- tcgen05 (5th-generation tensor cores)
//
// Tensor memory (TMEM) addresses: bits 31..16 lane, bits 15..0 column.  A
// warp reaches lanes 32 * (warp id % 4) .. + 31 only.

// Allocate `ncols` (a power of 2, 32..512) TMEM columns; the base address
// is written to shared memory at `dst`.  One whole warp executes it.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// This thread's 64 registers -> 64 consecutive TMEM columns of its lane.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, "
                 "%33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, "
                 "%49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};"
                 ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                 "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                 "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                 "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]),
                 "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]),
                 "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]),
                 "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]),
                 "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
                 : "memory");
}

// This thread's 32 registers -> 32 consecutive TMEM columns of its lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                 "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                 "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                 "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive TMEM columns of this thread's lane -> 32 registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                   "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                   "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                   "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                   "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] x B[smem]: kind::f16, one CTA, A and D in tensor
// memory, B described by a shared-memory matrix descriptor.  accumulate = 0
// overwrites D.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The mbarrier at `bar` gets one arrival once every tcgen05 operation this
// thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Whole-warp forms: every lane of the warp calls them with the same
// (warp-uniform) operands and one elected lane issues.  Issued this way an
// M128 x N32 x K16 MMA costs the warp about 20 cycles against about 47 when
// one lane issues inside a lane branch.
__device__ __forceinline__ void tc_mma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Eight MMAs of one 128-column group (K = 8 x 16) from one elected lane of
// the calling warp: A at a + 8k (tensor-memory columns), B at descriptor
// b + 64k (1024 bytes further along K each); the first adds to D only when
// `accumulate` is set, the others always add.
__device__ __forceinline__ void tc_mma8_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p, t;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 p, %18, 0;\n\t"
                 "setp.eq.b32 t, %18, %18;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, p;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, t;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(a_tmem + 8u), "r"(a_tmem + 16u), "r"(a_tmem + 24u),
                   "r"(a_tmem + 32u), "r"(a_tmem + 40u), "r"(a_tmem + 48u), "r"(a_tmem + 56u),
                   "l"(b_desc), "l"(b_desc + 64u), "l"(b_desc + 128u), "l"(b_desc + 192u),
                   "l"(b_desc + 256u), "l"(b_desc + 320u), "l"(b_desc + 384u), "l"(b_desc + 448u),
                   "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Two commits (and optionally a third when bar3 != 0) from one elected lane.
__device__ __forceinline__ void tc_commit23_warp(uint32_t bar1, uint32_t bar2, uint32_t bar3)
{
    asm volatile("{\n\t.reg .pred e, c;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.and.b32 c, %2, 0, e;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t"
                 "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%2];\n\t}"
                 ::"r"(bar1), "r"(bar2), "r"(bar3)
                 : "memory");
}

__device__ __forceinline__ void tc_commit_warp(uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 ::"r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------- argmax keys

// 64-bit key that orders (value, token id) by value, then by LOWER id:
// high word = order-preserving map of the fp32 bits (-0 folded onto +0, NaN
// below everything), low word = 0xFFFFFFFF - id.  Key 0 means "no candidate".
__device__ __forceinline__ unsigned long long make_key(float v, uint32_t id)
{
    uint32_t u = __float_as_uint(v);
    if (v == 0.0f) u = 0u;
    uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (v != v) o = 0u;
    return (static_cast<unsigned long long>(o) << 32) |
           static_cast<unsigned long long>(0xFFFFFFFFu - id);
}

// The largest key among the warp's 32 lanes (all lanes get it): the largest
// high word, then the largest low word among the lanes holding it -- the
// 64-bit maximum, in two single-instruction warp reductions.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k)
{
    const uint32_t hi = static_cast<uint32_t>(k >> 32), lo = static_cast<uint32_t>(k);
    const uint32_t bh = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t bl = __reduce_max_sync(0xFFFFFFFFu, hi == bh ? lo : 0u);
    return (static_cast<unsigned long long>(bh) << 32) | bl;
}

__device__ __forceinline__ float key_value(unsigned long long k)
{
    uint32_t o = static_cast<uint32_t>(k >> 32);
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ int32_t key_id(unsigned long long k)
{
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
}

__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src)
{
    uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    lo = __shfl_sync(0xFFFFFFFFu, lo, src);
    hi = __shfl_sync(0xFFFFFFFFu, hi, src);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m)
{
    uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    lo = __shfl_xor_sync(0xFFFFFFFFu, lo, m);
    hi = __shfl_xor_sync(0xFFFFFFFFu, hi, m);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}

}  // namespace sv
