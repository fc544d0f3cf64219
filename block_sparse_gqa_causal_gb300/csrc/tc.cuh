// tc.cuh -- Blackwell (sm_100-family, here sm_103a) building blocks written
// as inline PTX: mbarriers with bounded waits, TMA tile loads, TMEM
// allocation, tcgen05.mma (kind::f16, bf16 in / fp32 accumulate in TMEM),
// tcgen05.commit and tcgen05.ld.  Encodings follow the PTX ISA's
// descriptions of the shared-memory matrix descriptor and the instruction
// descriptor for .kind::f16.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace msa {
namespace tc {

// ------------------------------------------------------------------ mbarrier
MSA_DEV void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
MSA_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::); }
MSA_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::); }

MSA_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
MSA_DEV void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
MSA_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe (test_wait never suspends the thread): for loops that
// poll several barriers and act on whichever is ready first.
MSA_DEV bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after ~2^26 polls (seconds), records a timeout in
// the status word and returns false.  Callers then skip their remaining
// work so the kernel ends instead of hanging.
constexpr uint32_t kSpinLimit = 1u << 26;
MSA_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, DeviceStatus *st, int site, volatile int *abort_flag,
                       uint32_t limit = kSpinLimit)
{
    for (uint32_t it = 0; it < limit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 1023u) == 1023u && abort_flag && *abort_flag) return false;
    }
    report(st, kDevTimeout, site, (int)parity);
    if (abort_flag) *abort_flag = 1;
    return false;
}

// The bounded wait run by every lane of a warp, with the same outcome on all
// of them (warp-uniform code such as an elected MMA issuer follows).
MSA_DEV bool mbar_wait_warp(uint64_t *bar, uint32_t parity, DeviceStatus *st, int site, volatile int *abort_flag)
{
    const bool r = mbar_wait(bar, parity, st, site, abort_flag);
    return __all_sync(0xffffffffu, r);
}

// ------------------------------------------------------------------ TMA
MSA_DEV void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];\n" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
MSA_DEV void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z, int w)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
        "%6}], [%2];\n" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
MSA_DEV void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Bring a 4-D tile into L2 (no shared-memory destination, no completion to
// wait for): a later tile load of the same box then hits L2.
MSA_DEV void tma_prefetch_4d(const CUtensorMap *map, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
MSA_DEV void prefetch_l2(const void *gmem) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(gmem)); }

// ------------------------------------------------------------------ TMEM
// Allocation is warp-wide; the allocated column base is written to smem.
MSA_DEV void tmem_alloc(uint32_t *smem_slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols));
}
MSA_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::); }
MSA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
MSA_DEV void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::); }
MSA_DEV void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes (64 bf16 of K), 8-row core groups 1024 bytes
// apart (stride byte offset), leading byte offset unused for this layout
// (encoded as 1), version field = 1, swizzle mode 2 (128B).  The tile base
// must be 1024-byte aligned; advancing K by 16 elements inside the 128-byte
// row adds 32 bytes to the start address.
MSA_DEV uint64_t sdesc_k128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)1 << 16;                             // leading byte offset (unused)
    d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset
    d |= (uint64_t)1 << 46;                             // version
    d |= (uint64_t)2 << 61;                             // 128B swizzle
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both operands
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4)                       // D format f32
           | (1u << 7)                     // A format bf16
           | (1u << 10)                    // B format bf16
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
MSA_DEV void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, K-major) read from tensor
// memory -- row m in lane m, 16-bit elements packed two per 32-bit column in
// K order (lower K in the low half) -- B through its shared-memory descriptor.
MSA_DEV void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate));
}

// One lane of a converged warp (the lowest active one) gets true: the lane
// that issues a warp's tensor-core instructions, so that the code around
// them (waits, descriptors) runs warp-uniform.
MSA_DEV bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n .reg .pred p;\n .reg .b32 r;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(pred));
    return pred != 0;
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
MSA_DEV void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive fp32 columns, waited for inside the same asm
// statement so no instruction can read the registers before they land:
// thread t of warp w gets TMEM lane 32*(w%4) + t, columns col..col+31.
MSA_DEV void tmem_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}


// 32 lanes x 16 consecutive fp32 columns (same conventions as tmem_ld32).
MSA_DEV void tmem_ld16(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Shared-memory matrix descriptor with explicit byte offsets (128B swizzle).
// For a K-major operand (rows = M/N, 128-byte rows of K) the stride byte
// offset is the step between 8-row groups and the leading byte offset is
// unused.  For an MN-major operand (rows = K, 128-byte rows holding 64
// consecutive M/N elements) the leading byte offset is the step between
// 64-element atoms along M/N and the stride byte offset the step between
// 8-row groups along K.
MSA_DEV uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Advance a shared-memory descriptor by a byte offset (a multiple of 16).
// The start address sits in the low 14 bits in 16-byte units and no
// shared-memory address (< 256 KB) carries out of that field, so one 32-bit
// add on the low word does it: the MMA issuers precompute their base
// descriptors once and advance them with this single add per instruction,
// which keeps a lone issuing thread ahead of the tensor pipe.
MSA_DEV uint64_t desc_adv(uint64_t d, uint32_t bytes)
{
    const uint32_t lo = (uint32_t)d + (bytes >> 4), hi = (uint32_t)(d >> 32);
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

// instruction-descriptor bits selecting MN-major A / B
constexpr uint32_t kAMajorMN = 1u << 15;
constexpr uint32_t kBMajorMN = 1u << 16;

// Batched TMEM loads: issue several tcgen05.ld (no wait) and then one
// tmem_wait32 per destination array.  The wait takes the destination
// registers as read-write operands, so nothing that consumes them can be
// scheduled before it.
MSA_DEV void tmem_ld32_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
MSA_DEV void tmem_ld16_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers (thread t of warp
// w writes lane 32*(w%4) + t); complete once tmem_wait_st returns.
MSA_DEV void tmem_st16(uint32_t taddr, const uint32_t *r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
MSA_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

MSA_DEV void tmem_wait32(uint32_t *r)
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                   "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
                   "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
MSA_DEV void tmem_ld8_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
// Waits for every tcgen05.ld of this thread issued so far; r (8 registers)
// is tied so nothing that reads it moves above the wait.
MSA_DEV void tmem_wait8(uint32_t *r)
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}
MSA_DEV void tmem_wait16(uint32_t *r)
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Hardware base-2 exponential / logarithm approximations (MUFU), used
// where a few ulp of error is far below the tolerances of the outputs.
MSA_DEV float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
MSA_DEV float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte fp32 reduction into global memory (no return value).
MSA_DEV void red_add_v4(float *addr, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

}  // namespace tc
}  // namespace msa
