// kda_tc.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a / sm_103a) tensor-core path:
// mbarriers, bulk async copies (TMA engine, non-tensor form), tensor memory (TMEM) allocation,
// tcgen05.mma of kind::tf32 and kind::f16, tcgen05.commit, tcgen05.ld / tcgen05.st and the
// tcgen05 fences.
//
// Operand images in shared memory use the canonical no-swizzle K-major layout: the tile is cut
// into "core matrices" of 8 rows x 16 bytes (4 tf32 or 8 fp16 elements per row, 128 bytes per
// core matrix); core (row group rg, k group kc) sits at byte rg * SBO + kc * LBO with LBO = 128
// (k groups adjacent) and SBO = 8 rows x the row's bytes (one 8-row slab holds all K).  One MMA
// step consumes 32 bytes of K (8 tf32 or 16 fp16), i.e. two core matrices: the descriptor start
// advances by 256 bytes per step.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- image layout ---------------------------------------------------------------------------
// Float index of element (row, k) in a K-major no-swizzle image with K columns.
__host__ __device__ __forceinline__ uint32_t img_index(uint32_t row, uint32_t k, uint32_t K)
{
    return (((row >> 3) * (K >> 2) + (k >> 2)) << 5) + ((row & 7u) << 2) + (k & 3u);
}

// Round an fp32 value to the nearest tf32 (10 explicit mantissa bits), ties away from zero.
__device__ __forceinline__ float round_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// ---- descriptors ------------------------------------------------------------------------------
// Shared-memory matrix descriptor (no swizzle, descriptor version 1).  In both major-nesses the
// leading byte offset (LBO) is the distance between core matrices adjacent along K and the stride
// byte offset (SBO) the distance between core matrices adjacent along M (or N).  A K-major core
// matrix is 8 rows of M/N x 16 bytes of K; an MN-major one is 8 rows of K x 16 bytes of M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    // base offset 0, absolute LBO mode 0, layout type 0 = no swizzle
    return d;
}

// Instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N)
{
    return (1u << 4)            // D format: f32
         | (2u << 7)            // A format: tf32
         | (2u << 10)           // B format: tf32
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

// Instruction descriptor of kind::f16 with fp16 A and B and an fp32 accumulator.  a_mn / b_mn select
// the MN-major ("transposed") shared-memory layout for A / B; K-major otherwise.  An A operand in
// TMEM is always K-major.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, bool a_mn = false, bool b_mn = false)
{
    return (1u << 4)                  // D format: f32
         | (a_mn ? (1u << 15) : 0u)   // A major-ness
         | (b_mn ? (1u << 16) : 0u)   // B major-ness
         | ((N >> 3) << 17)           // N / 8   (A and B format 0 = f16)
         | ((M >> 4) << 24);          // M / 16
}

// Two fp32 values rounded to fp16 (nearest even) and packed: lo in bits 0..15, hi in 16..31.
// This is the order a kind::f16 A operand in TMEM expects: column c holds k = 2c and 2c + 1.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- mbarriers ----------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
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

// Wait for the phase with the given parity to complete; gives up after max_iter polls and
// returns false (the caller records an error instead of hanging).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter)
{
    for (uint32_t i = 0; i < max_iter; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Prefetch of a global range into L2 (no destination, no completion): 16-byte aligned address,
// size a multiple of 16 bytes.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---- bulk async copy global -> shared (non-tensor TMA), completion via mbarrier tx bytes ---
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- tensor (tiled) bulk copy global -> shared through a tensor map ----------------------------------
// 2D box at element coordinates (x = innermost, y); x * element size must be a multiple of 16 bytes.
// Elements outside the tensor read as zero.  tmap is the address of a CUtensorMap kernel parameter
// (__grid_constant__).  Completion is signalled on the mbarrier as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// ---- bulk async copy shared -> global (bulk-group completion) -------------------------------------
// src and dst 16-byte aligned, bytes a multiple of 16.  The issuing thread tracks completion with
// bulk_commit / bulk_wait_read (the shared source may be reused) / bulk_wait (writes done).
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Named barrier over COUNT threads that also returns, to each of them, whether any passed a true
// flag: a loop exit decided after it is the same for every participant.
template <int ID, int COUNT>
__device__ __forceinline__ bool bar_any(bool flag)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag), "n"(ID), "n"(COUNT)
        : "memory");
    return r != 0;
}
template <int ID, int COUNT>
__device__ __forceinline__ void bar_sync() { asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory"); }

// ---- tensor memory ------------------------------------------------------------------------------
// Warp-wide: allocate ncols (power of two >= 32) TMEM columns; the base address goes to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- MMA ------------------------------------------------------------------------------------------
// D[tmem] (+)= A[tmem] * B[smem desc]^T
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T    (kind::f16: fp16 A in TMEM as packed pairs, fp16 B image)
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T    (kind::f16, both operands in shared memory)
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on *bar when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// ---- TMEM <-> registers, 32 lanes x 32 bits ---------------------------------------------------------
// Each thread of a warp reads (writes) its own TMEM lane, columns taddr.col .. +15.  The wait is in
// the same asm statement, so the registers cannot be consumed before the load has landed and the
// store has completed before the function returns.
#define KDA_R16(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
    "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7]), "=r"(r[i + 8]), "=r"(r[i + 9]), "=r"(r[i + 10]), \
    "=r"(r[i + 11]), "=r"(r[i + 12]), "=r"(r[i + 13]), "=r"(r[i + 14]), "=r"(r[i + 15])
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v)
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : KDA_R16(0)
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

#undef KDA_R16

// Store without waiting; follow a batch of these with tmem_wait_st() before the data is consumed.
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const float* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_st16u_nowait(uint32_t taddr, const uint32_t* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8u_nowait(uint32_t taddr, const uint32_t* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Eight fp32 values rounded to fp16 (nearest even) as one 16-byte vector, element i at bytes 2i.
__device__ __forceinline__ uint4 pack8_f16(const float* x)
{
    return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                      pack_f16x2(x[6], x[7]));
}
// The two fp16 halves of a packed pair as fp32 (lo = bits 0..15).
__device__ __forceinline__ void unpack_f16x2(uint32_t p, float& lo, float& hi)
{
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(p));
}

}  // namespace tc
}  // namespace kda
