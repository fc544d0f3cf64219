// block_mask.cu -- block-mask encoding of a selection and its traversal
// ("Sparse Attention · Part II", section 4.3, "Turn support into a block
// mask").
//
// A query tile is 128 consecutive query rows of one (batch, group).  Its
// mask has one bit per key block, set when some query of the tile selected
// that block; 32 flags share an unsigned word (block c: word c/32, bit
// c%32), so the mask is the OR-union of the tile's selections -- the set of
// K/V blocks a tile-wide consumer has to visit.  The traversal counts each
// word's set bits (popc), turns the counts into output offsets, and visits
// a word's bits by rank, writing the tile's active blocks in ascending order.
//
// One CTA per (tile, group, batch): the tile's selections (128 x topk ids)
// are OR-ed into shared-memory words with shared atomics, the words go out
// coalesced, warp 0 scans the word counts, and each thread walks its words.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
block_mask_kernel(Problem p, const int32_t *__restrict__ sel, uint32_t *__restrict__ mask,
                  int32_t *__restrict__ counts, int32_t *__restrict__ active)
{
    extern __shared__ uint32_t sw[];             // W words, then W + 1 prefix counts
    const int t = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const int W = (p.nb + 31) / 32;
    int *pre = reinterpret_cast<int *>(sw + W);
    for (int w = threadIdx.x; w < W; w += kThreads) sw[w] = 0u;
    __syncthreads();
    const int i0 = t * 128, nq = min(128, p.Nq - i0);
    const int32_t *src = sel + (((long long)b * p.Hkv + r) * p.Nq + i0) * p.topk;
    for (int e = threadIdx.x; e < nq * p.topk; e += kThreads) {
        const int c = __ldg(src + e);
        if (c >= 0 && c < p.nb) atomicOr(&sw[c >> 5], 1u << (c & 31));   // -1 padding and ids >= nb set nothing
    }
    __syncthreads();
    const long long tile = ((long long)b * p.Hkv + r) * gridDim.x + t;
    uint32_t *dst = mask + tile * W;
    for (int w = threadIdx.x; w < W; w += kThreads) dst[w] = sw[w];
    if (!counts && !active) return;
    if (threadIdx.x < 32) {
        // exclusive prefix of the words' set-bit counts, 32 words at a time
        const int lane = threadIdx.x;
        int carry = 0;
        for (int w0 = 0; w0 < W; w0 += 32) {
            const int w = w0 + lane;
            const int c = w < W ? __popc(sw[w]) : 0;
            int x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += o;
            }
            if (w < W) pre[w] = carry + x - c;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            pre[W] = carry;
            if (counts) counts[tile] = carry;
        }
    }
    if (!active) return;
    __syncthreads();
    int32_t *out = active + tile * p.nb;
    for (int w = threadIdx.x; w < W; w += kThreads) {
        // the rank-th set bit is the lowest one left after clearing the rank lower ones
        uint32_t word = sw[w];
        const int n = __popc(word);
        for (int rank = 0; rank < n; ++rank) {
            out[pre[w] + rank] = 32 * w + (__ffs(word) - 1);
            word &= word - 1u;
        }
    }
    for (int x = pre[W] + threadIdx.x; x < p.nb; x += kThreads) out[x] = -1;
}

}  // namespace

size_t block_mask_smem_bytes(const Problem &p) { return (size_t)(2 * ((p.nb + 31) / 32) + 1) * 4; }

cudaError_t launch_block_mask(const Problem &p, const int32_t *sel, uint32_t *mask, int32_t *counts, int32_t *active,
                              cudaStream_t s)
{
    const size_t smem = block_mask_smem_bytes(p);
    cudaError_t e = cudaFuncSetAttribute(block_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int T = (p.Nq + 127) / 128;
    {
        TimedLaunch timed_("block_mask_kernel", s);
        block_mask_kernel<<<dim3(T, p.Hkv, p.B), kThreads, smem, s>>>(p, sel, mask, counts, active);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
