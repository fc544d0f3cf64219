// common.cuh -- device helpers shared by the MSA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MSA_DEV __device__ __forceinline__

namespace msa {

// ------------------------------------------------------------------ status
// The first 256 bytes of every workspace hold this word.  Kernels record the
// first device-side failure here instead of trapping, so the context stays
// usable and the host can report it.
struct DeviceStatus {
    int code;   // 0 ok, 5 wait ran out, 6 other device check
    int where;  // kernel-specific site id
    int info;   // e.g. the offending index
    int pad;
};
constexpr int kStatusBytes = 256;
constexpr int kDevTimeout = 5;
constexpr int kDevCheck = 6;

MSA_DEV void report(DeviceStatus *st, int code, int where, int info)
{
    if (st && atomicCAS(&st->code, 0, code) == 0) {
        st->where = where;
        st->info = info;
    }
}

// ------------------------------------------------------------------ packing
MSA_DEV uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

MSA_DEV float bf16_to_f(uint16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

MSA_DEV float2 unpack_bf16(uint32_t x)
{
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

MSA_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ------------------------------------------------------------------ warp sums
// Column sums across a warp.  Each lane holds v[0..N), one value per column;
// afterwards out[h] on lane l is the sum over all 32 lanes of column
// (l mod min(N, 32)) + 32 h.  Each exchange step halves the per-lane array:
// a lane keeps the columns whose next index bit equals its own lane bit and
// adds in its partner's copy of them (N - 1 shuffles for N <= 32, where the
// remaining lane bits are then summed by xor steps).  v is overwritten.
template <int N>
MSA_DEV void lane_colsum(float (&v)[N], int lane, float (&out)[(N + 31) / 32])
{
    static_assert(N >= 1 && (N & (N - 1)) == 0 && N <= 64, "N must be a power of two up to 64");
    constexpr int W = N < 32 ? N : 32;
#pragma unroll
    for (int o = 1; o < W; o <<= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < N / (2 * o); ++i) {
            const float a = v[2 * i], c = v[2 * i + 1];
            v[i] = (hi ? c : a) + __shfl_xor_sync(0xffffffffu, hi ? a : c, o);
        }
    }
#pragma unroll
    for (int h = 0; h < (N + 31) / 32; ++h) out[h] = v[h];
#pragma unroll
    for (int o = W; o < 32; o <<= 1) out[0] += __shfl_xor_sync(0xffffffffu, out[0], o);
}

// Streaming form of lane_colsum<32>: feed the values of columns c = 0..31 in
// order (c a constant after unrolling).  Pairs are combined as soon as both
// exist, so at most one pending value per level stays live (lv[0..4]); after
// column 31, lv[5] on lane l holds the sum over the warp of column l.
MSA_DEV void colsum32_push(float (&lv)[6], float x, int c, int lane)
{
    if ((c & 1) == 0) {
        lv[0] = x;
        return;
    }
    float cur = x;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int o = 1 << k;
        const bool hi = (lane & o) != 0;
        const float a = lv[k];
        cur = (hi ? cur : a) + __shfl_xor_sync(0xffffffffu, hi ? a : cur, o);
        if (k == 4) {
            lv[5] = cur;
            return;
        }
        if (((c >> (k + 1)) & 1) == 0) {
            lv[k + 1] = cur;
            return;
        }
    }
}

// ------------------------------------------------------------------ cp.async
MSA_DEV void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
// zero-fills the 16 smem bytes when !valid (src-size 0)
MSA_DEV void cp_async16_zfill(void *smem, const void *gmem, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(valid ? 16 : 0));
}
MSA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
MSA_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ------------------------------------------------------------------ ldmatrix
MSA_DEV void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
MSA_DEV void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
MSA_DEV void ldsm_x2(uint32_t &r0, uint32_t &r1, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(p)));
}
MSA_DEV void ldsm_x2_t(uint32_t &r0, uint32_t &r1, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(p)));
}

// ------------------------------------------------------------------ mma.sync
// D(16x8,f32) += A(16x16,bf16,row) * B(16x8,bf16,col)
MSA_DEV void mma16816(float *c, const uint32_t *a, const uint32_t *b)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ------------------------------------------------------------------ misc
MSA_DEV float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
MSA_DEV float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// fp32 atomic add without a return value (compiles to a reduction)
MSA_DEV void red_add(float *p, float v) { atomicAdd(p, v); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Order-preserving map of a finite fp32 to uint32 (larger float -> larger key).
// -0 is first turned into +0, so two equal scores always get equal keys and
// their order falls to the block index.
MSA_DEV uint32_t float_key(float f)
{
    uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Ranking key of a candidate block: score first, then the lower block index
// (one unsigned compare orders by (score desc, index asc)); 0 means "none".
MSA_DEV unsigned long long block_key(float s, int c)
{
    return ((unsigned long long)float_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)c);
}

MSA_DEV unsigned long long shfl64(unsigned long long v, int src)
{
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
    return ((unsigned long long)hi << 32) | lo;
}

MSA_DEV unsigned long long shfl64_xor(unsigned long long v, int m)
{
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}

// descending bitonic sort of one 64-bit key per lane
MSA_DEV unsigned long long sort_desc64(unsigned long long v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long o = shfl64_xor(v, stride);
            const bool desc = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    return v;
}

// a bitonic sequence across the lanes -> descending order
MSA_DEV unsigned long long merge_desc64(unsigned long long v, int lane)
{
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long o = shfl64_xor(v, stride);
        v = ((lane & stride) == 0) ? (v > o ? v : o) : (v < o ? v : o);
    }
    return v;
}

// Barrier `id` (1..15) over `nthreads` threads (a multiple of 32) of the CTA.
MSA_DEV void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace msa
