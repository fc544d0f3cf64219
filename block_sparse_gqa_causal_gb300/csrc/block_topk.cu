// block_topk.cu -- top-k block selection of MSA ("Sparse Attention · Part
// II", section 3.2): the query's local block c0 always takes one slot, the
// other k-1 go to the earlier blocks with the largest block scores.  Ties go
// to the lower block index.  No exponentials: scores are compared raw, since
// softmax is monotone (the "exp-free" selection of the MSA summary page).
//
// One warp per (b, i, r) row.  A candidate is the 64-bit key
//   (order-preserving bits of the fp32 score) << 32 | (0xFFFFFFFF - c)
// so one unsigned compare ranks by score, then by lower index.  The warp
// keeps its current best k-1 keys distributed over lanes (lane m holds the
// m-th best) and streams the row in 32-wide coalesced chunks; only keys
// above the current (k-1)-th best are inserted.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ unsigned long long make_key(float s, int c)
{
    return ((unsigned long long)float_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)c);
}

__device__ __forceinline__ unsigned long long shfl64(unsigned long long v, int src)
{
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long shfl64_up(unsigned long long v, int delta)
{
    const uint32_t lo = __shfl_up_sync(0xffffffffu, (uint32_t)v, delta);
    const uint32_t hi = __shfl_up_sync(0xffffffffu, (uint32_t)(v >> 32), delta);
    return ((unsigned long long)hi << 32) | lo;
}

// ascending bitonic sort of one int per lane across the warp
__device__ __forceinline__ int warp_sort_asc(int v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int other = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool up = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            v = (lower == up) ? min(v, other) : max(v, other);
        }
    }
    return v;
}

__global__ void __launch_bounds__(kWarps * 32)
block_topk_kernel(Problem p, const float *__restrict__ bs, int32_t *__restrict__ sel)
{
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long rows = (long long)p.B * p.Nq * p.Hkv;
    if (row >= rows) return;
    const int r = (int)(row % p.Hkv);
    const long long bi = row / p.Hkv;
    const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int c0 = (int)(pos / 128);
    const int k = p.topk;
    int32_t *out = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * k;

    if (c0 + 1 <= k) {               // every visible block is selected
        if (lane < k) out[lane] = lane <= c0 ? lane : -1;
        return;
    }
    const int K1 = k - 1;            // slots the indexer chooses, 0..31
    const float *src = bs + row * p.nb;
    unsigned long long best = 0ull;  // 0 is below every real key
    for (int base = 0; base < c0; base += 32) {
        const int c = base + lane;
        const unsigned long long key = c < c0 ? make_key(__ldg(src + c), c) : 0ull;
        unsigned long long thr = K1 > 0 ? shfl64(best, K1 - 1) : ~0ull;
        unsigned mask = __ballot_sync(0xffffffffu, key > thr);
        while (mask) {
            const int srcl = __ffs(mask) - 1;
            mask &= mask - 1;
            const unsigned long long ck = shfl64(key, srcl);
            if (!(ck > thr)) continue;
            const int at = __popc(__ballot_sync(0xffffffffu, lane < K1 && best > ck));
            const unsigned long long up = shfl64_up(best, 1);
            if (lane > at) best = up;
            else if (lane == at) best = ck;
            thr = shfl64(best, K1 - 1);
        }
    }
    int id = lane < K1 ? (int)(0xFFFFFFFFu - (uint32_t)best) : (lane == K1 ? c0 : 0x7fffffff);
    id = warp_sort_asc(id, lane);
    if (lane < k) out[lane] = id;
}

}  // namespace

cudaError_t launch_block_topk(const Problem &p, const float *bs, int32_t *sel, DeviceStatus *,
                              cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Nq * p.Hkv;
    const long long grid = (rows + kWarps - 1) / kWarps;
    block_topk_kernel<<<(unsigned)grid, kWarps * 32, 0, s>>>(p, bs, sel);
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
