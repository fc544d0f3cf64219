// block_topk.cu -- top-k block selection of MSA ("Sparse Attention · Part
// II", section 3.2): the query's local block c0 always takes one slot, the
// other k-1 go to the earlier blocks with the largest block scores.  Ties go
// to the lower block index.  No exponentials: scores are compared raw, since
// softmax is monotone (the "exp-free" selection of the MSA summary page).
//
// One warp per (b, i, r) row, streamed in segments of 32*R scores (R per
// lane, coalesced loads all in flight).  Per segment, a conservative cutoff
// (section 4.2 of the same page: the k-th largest of a subset of at least k
// elements never exceeds the global k-th largest) is the (k-1)-th largest of
// the 32 lane maxima (for k > 17: of each lane's two largest scores); only
// scores at or above it, and above the current
// (k-1)-th best, survive.  Survivors become 64-bit keys
//   (order-preserving bits of the fp32 score) << 32 | (0xFFFFFFFF - c),
// so one unsigned compare ranks by score then by lower index; they are
// sorted 32 at a time and merged into the running top-(k-1), which is kept
// sorted across the lanes.
//
// Rows of at most 1,024 earlier blocks (every prefill row up to 128K tokens)
// take a shorter road, warp_topk_regs: the row is held in registers, the
// (k-1)-th largest score T is found among the few scores that pass the same
// cutoff, and the chosen blocks are written in index order by ballots, with
// no 64-bit keys and no running list.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kWarps = 8;
constexpr int kR = 16;                 // scores per lane per segment
constexpr int kSeg = 32 * kR;

// descending bitonic sort of one float per lane
__device__ __forceinline__ float sort_desc_f(float v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            v = (lower == desc) ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return v;
}

// a bitonic sequence of floats across the lanes -> descending order
__device__ __forceinline__ float merge_desc_f(float v, int lane)
{
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, stride);
        v = ((lane & stride) == 0) ? fmaxf(v, o) : fminf(v, o);
    }
    return v;
}

// ascending bitonic sort of one int per lane
__device__ __forceinline__ int sort_asc_i(int v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool up = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            v = (lower == up) ? min(v, o) : max(v, o);
        }
    }
    return v;
}

__device__ __forceinline__ float key_value(unsigned long long key)
{
    const uint32_t u = (uint32_t)(key >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// One warp's running top-(k-1) over the segments base0, base0 + step, ... of
// a row's earlier blocks [0, c0); best (lane m: m-th best key, 0 = empty)
// is updated in place.  buf: this warp's kSeg-key scratch.
__device__ __forceinline__ void warp_topk(const float *__restrict__ src, int c0, int K1, int base0, int step,
                                          unsigned long long *buf, unsigned long long &best, int lane)
{
    for (int base = base0; K1 > 0 && base < c0; base += step) {
        float v[kR];
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            const int c = base + j * 32 + lane;
            v[j] = c < c0 ? __ldg(src + c) : -INFINITY;
        }
        // the lane's two largest scores (of 16 distinct positions)
        float lmax = v[0], l2 = -INFINITY;
#pragma unroll
        for (int j = 1; j < kR; ++j) {
            l2 = fmaxf(l2, fminf(lmax, v[j]));
            lmax = fmaxf(lmax, v[j]);
        }
        float tau;
        if (K1 <= 16) {
            tau = __shfl_sync(0xffffffffu, sort_desc_f(lmax, lane), K1 - 1);
        } else {
            // larger k: the (k-1)-th largest of the 64 values formed by each lane's two
            // largest (still a subset of the segment, so still a valid cutoff, but far
            // tighter than the (k-1)-th of the 32 lane maxima when k-1 nears 32)
            const float a = sort_desc_f(lmax, lane), c = sort_desc_f(l2, lane);
            const float top = merge_desc_f(fmaxf(a, __shfl_sync(0xffffffffu, c, 31 - lane)), lane);
            tau = __shfl_sync(0xffffffffu, top, K1 - 1);
        }
        const unsigned long long kth = shfl64(best, K1 - 1);
        const float t_run = kth ? key_value(kth) : -INFINITY;
        // survivors: >= the segment cutoff and strictly above the running
        // (k-1)-th value (an equal value here has a larger index and loses)
        int cnt = 0;
#pragma unroll
        for (int j = 0; j < kR; ++j) cnt += (v[j] >= tau && v[j] > t_run && v[j] != -INFINITY) ? 1 : 0;
        int off = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, off, d);
            if (lane >= d) off += o;
        }
        const int total = __shfl_sync(0xffffffffu, off, 31);
        off -= cnt;
        if (total == 0) continue;
#pragma unroll
        for (int j = 0; j < kR; ++j)
            if (v[j] >= tau && v[j] > t_run && v[j] != -INFINITY) buf[off++] = block_key(v[j], base + j * 32 + lane);
        __syncwarp();
        for (int c32 = 0; c32 < total; c32 += 32) {
            unsigned long long ck = (c32 + lane < total) ? buf[c32 + lane] : 0ull;
            ck = sort_desc64(ck, lane);
            // top 32 of two descending lists: pairwise max against the reversed list is bitonic
            const unsigned long long rev = shfl64(ck, 31 - lane);
            best = merge_desc64(best > rev ? best : rev, lane);
        }
        __syncwarp();
    }
}

// One warp's top-(k-1) of a row whose c0 earlier blocks fit in J registers
// per lane (c0 <= 32 J), written with the local block into out:
//   1. tau = the (k-1)-th largest of each lane's largest score (of its two
//      largest for k > 17): a subset of the row, so tau <= T, the row's
//      (k-1)-th largest score, and at least k-1 scores reach it (the
//      lanes' second-largest scores alone would give a looser cutoff: about
//      1.75 (k-1) survivors against 1.5 (k-1), too often over 64);
//   2. the scores >= tau, at most 64, are collected in block order by
//      ballots (survivor t of the row goes to lane t % 32, slot t / 32);
//      T, their (k-1)-th largest, is found by taking out the largest (or,
//      when T lies nearer the bottom, the smallest) values one at a time,
//      all copies of a value at once, with warp max / min reductions on
//      order-preserving keys;
//   3. every survivor > T is chosen, and of those equal to T the first in
//      block order, up to k-1 in all (ties to the lower index); a ballot
//      gives each its output slot, so the list comes out ascending, the
//      local block last.
// Returns false with nothing written when more than 64 scores pass the
// cutoff or the cutoff is not finite (-inf or NaN scores); warp_topk then
// takes the row.  sbuf: 64 floats and 64 ints of this warp's scratch.
template <int J>
__device__ __forceinline__ bool warp_topk_regs(const float *__restrict__ src, int c0, int K1, float *sbuf,
                                               int32_t *out, int lane)
{
    float v[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int c = j * 32 + lane;
        v[j] = c < c0 ? __ldg(src + c) : -INFINITY;
    }
    float m1 = -INFINITY, m2 = -INFINITY;          // the lane's two largest
#pragma unroll
    for (int j = 0; j < J; ++j) {
        m2 = fmaxf(m2, fminf(m1, v[j]));
        m1 = fmaxf(m1, v[j]);
    }
    float tau;
    if (K1 <= 16) {
        tau = __shfl_sync(0xffffffffu, sort_desc_f(m1, lane), K1 - 1);
    } else {
        const float a = sort_desc_f(m1, lane), b = sort_desc_f(m2, lane);
        tau = __shfl_sync(0xffffffffu, merge_desc_f(fmaxf(a, __shfl_sync(0xffffffffu, b, 31 - lane)), lane), K1 - 1);
    }
    if (!(tau > -INFINITY)) return false;
    int *sidx = reinterpret_cast<int *>(sbuf + 64);
    const unsigned lt = (1u << lane) - 1u;
    int m = 0;                                     // survivors so far (warp-uniform)
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (j * 32 >= c0) break;
        const bool sv = v[j] >= tau;
        const unsigned bal = __ballot_sync(0xffffffffu, sv);
        const int at = m + __popc(bal & lt);
        if (sv && at < 64) {
            sbuf[at] = v[j];
            sidx[at] = j * 32 + lane;
        }
        m += __popc(bal);
    }
    if (m > 64) return false;
    __syncwarp();
    const float a0 = lane < m ? sbuf[lane] : -INFINITY, b0 = lane + 32 < m ? sbuf[lane + 32] : -INFINITY;
    const int ia = sidx[lane], ib = sidx[lane + 32];
    __syncwarp();
    // survivors a0 (block order 0..31) then b0 (32..63) as keys; padding 0,
    // below every score's key
    const uint32_t ka = lane < m ? float_key(a0) : 0u, kb = lane + 32 < m ? float_key(b0) : 0u;
    const bool top = K1 <= m - K1 + 1;            // T is the K1-th from the top or the (m-K1+1)-th from the bottom
    int rank = top ? K1 : m - K1 + 1;
    const uint32_t gone = top ? 0u : 0xFFFFFFFFu;  // taken-out values and padding
    uint32_t xa = lane < m ? ka : gone, xb = lane + 32 < m ? kb : gone, tk;
    for (;;) {
        const uint32_t e = top ? __reduce_max_sync(0xffffffffu, max(xa, xb))
                               : __reduce_min_sync(0xffffffffu, min(xa, xb));
        const int copies = __popc(__ballot_sync(0xffffffffu, xa == e)) + __popc(__ballot_sync(0xffffffffu, xb == e));
        if (rank <= copies) {
            tk = e;
            break;
        }
        rank -= copies;
        if (xa == e) xa = gone;
        if (xb == e) xb = gone;
    }
    const unsigned ga = __ballot_sync(0xffffffffu, ka > tk), gb = __ballot_sync(0xffffffffu, kb > tk);
    const unsigned ea = __ballot_sync(0xffffffffu, ka == tk), eb = __ballot_sync(0xffffffffu, kb == tk);
    const int need_eq = K1 - __popc(ga) - __popc(gb);          // 1 .. number equal to T
    const bool sa = ((ga >> lane) & 1u) || (((ea >> lane) & 1u) && __popc(ea & lt) < need_eq);
    const bool sb = ((gb >> lane) & 1u) || (((eb >> lane) & 1u) && __popc(ea) + __popc(eb & lt) < need_eq);
    const unsigned ba = __ballot_sync(0xffffffffu, sa), bb = __ballot_sync(0xffffffffu, sb);
    if (sa) out[__popc(ba & lt)] = ia;
    if (sb) out[__popc(ba) + __popc(bb & lt)] = ib;
    if (lane == 0) out[K1] = c0;
    return true;
}

// the k-1 chosen blocks plus the local block, ascending, into out
__device__ __forceinline__ void write_selection(int32_t *out, unsigned long long best, int K1, int c0, int k, int lane)
{
    int id = lane < K1 ? (int)(0xFFFFFFFFu - (uint32_t)best) : (lane == K1 ? c0 : 0x7fffffff);
    id = sort_asc_i(id, lane);
    if (lane < k) out[lane] = id;
}

__global__ void __launch_bounds__(kWarps * 32)
block_topk_kernel(Problem p, const float *__restrict__ bs, int32_t *__restrict__ sel)
{
    __shared__ unsigned long long cand_buf[kWarps][kSeg];
    const int lane = threadIdx.x & 31;
    const int wi = threadIdx.x >> 5;
    const long long row = (long long)blockIdx.x * kWarps + wi;
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
    if (K1 > 0 && c0 <= 1024) {
        float *sbuf = reinterpret_cast<float *>(cand_buf[wi]);
        const bool done = c0 <= 256   ? warp_topk_regs<8>(src, c0, K1, sbuf, out, lane)
                          : c0 <= 512 ? warp_topk_regs<16>(src, c0, K1, sbuf, out, lane)
                                      : warp_topk_regs<32>(src, c0, K1, sbuf, out, lane);
        if (done) return;
        __syncwarp();
    }
    unsigned long long best = 0ull;  // lane m: m-th best key so far (0 = empty)
    warp_topk(src, c0, K1, 0, kSeg, cand_buf[wi], best, lane);
    write_selection(out, best, K1, c0, k, lane);
}

// Few rows with many blocks (decode): one CTA of kWarps warps per row, warp w
// taking segments w, w + kWarps, ...; warp 0 then merges the warps' lists
// (each sorted descending) with the same bitonic merge.
__global__ void __launch_bounds__(kWarps * 32)
block_topk_split_kernel(Problem p, const float *__restrict__ bs, int32_t *__restrict__ sel)
{
    __shared__ unsigned long long cand_buf[kWarps][kSeg];
    __shared__ unsigned long long lists[kWarps][32];
    const int lane = threadIdx.x & 31;
    const int wi = threadIdx.x >> 5;
    const long long row = blockIdx.x;
    const int r = (int)(row % p.Hkv);
    const long long bi = row / p.Hkv;
    const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int c0 = (int)(pos / 128);
    const int k = p.topk;
    int32_t *out = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * k;
    if (c0 + 1 <= k) {
        if (wi == 0 && lane < k) out[lane] = lane <= c0 ? lane : -1;
        return;
    }
    const int K1 = k - 1;
    unsigned long long best = 0ull;
    warp_topk(bs + row * p.nb, c0, K1, wi * kSeg, kWarps * kSeg, cand_buf[wi], best, lane);
    lists[wi][lane] = best;
    __syncthreads();
    if (wi == 0) {
#pragma unroll 1
        for (int w = 1; w < kWarps; ++w) {
            const unsigned long long rev = lists[w][31 - lane];
            best = merge_desc64(best > rev ? best : rev, lane);
        }
        write_selection(out, best, K1, c0, k, lane);
    }
}

// Decode with the fused selection: the score kernel's CTA for slice y of a
// row's blocks left that row's 16 best keys of the slice, in descending
// order, at cand[(row * slices + y) * 16 ..] (0 = no block).  The row's k-1
// best blocks are among them (each slice keeps at least k-1).  Only slices
// starting before the row's local block c0 are read: a slice whose blocks
// lie past every row of its tile was skipped by the score kernel and holds
// nothing of this call (its memory is stale).  One CTA per
// row: warp w takes the slice pairs w, w + 8, ... (all its loads issued
// before any merge); the two descending lists of a pair, the second
// reversed, form a bitonic sequence, sorted by one bitonic merge and merged
// into the warp's running top-32; warp 0 then merges the warps' lists.
constexpr int kMergeBatch = 4;   // slice pairs per warp per batch of loads

__global__ void __launch_bounds__(kWarps * 32)
block_topk_merge_kernel(Problem p, const unsigned long long *__restrict__ cand, int slices, int span,
                        int32_t *__restrict__ sel)
{
    __shared__ unsigned long long lists[kWarps][32];
    const int lane = threadIdx.x & 31;
    const int wi = threadIdx.x >> 5;
    const long long row = blockIdx.x;
    const int r = (int)(row % p.Hkv);
    const long long bi = row / p.Hkv;
    const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int c0 = (int)(pos / 128);
    const int k = p.topk;
    int32_t *out = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * k;
    if (c0 + 1 <= k) {
        if (wi == 0 && lane < k) out[lane] = lane <= c0 ? lane : -1;
        return;
    }
    const unsigned long long *src = cand + row * slices * 16;
    const int ys = min(slices, (c0 + span - 1) / span);   // slices holding blocks before c0
    const int pairs = (ys + 1) / 2;
    unsigned long long best = 0ull;
    for (int t0 = wi; t0 < pairs; t0 += kWarps * kMergeBatch) {
        unsigned long long ck[kMergeBatch];
#pragma unroll
        for (int t = 0; t < kMergeBatch; ++t) {
            const int y = 2 * (t0 + t * kWarps) + (lane >> 4);
            ck[t] = y < ys ? __ldg(src + (long long)y * 16 + (lane & 15)) : 0ull;
        }
#pragma unroll
        for (int t = 0; t < kMergeBatch; ++t) {
            const unsigned long long v = merge_desc64(shfl64(ck[t], lane < 16 ? lane : 47 - lane), lane);
            const unsigned long long rev = shfl64(v, 31 - lane);
            best = merge_desc64(best > rev ? best : rev, lane);
        }
    }
    lists[wi][lane] = best;
    __syncthreads();
    if (wi == 0) {
#pragma unroll 1
        for (int w = 1; w < kWarps; ++w) {
            const unsigned long long rev = lists[w][31 - lane];
            best = merge_desc64(best > rev ? best : rev, lane);
        }
        write_selection(out, best, k - 1, c0, k, lane);
    }
}

}  // namespace

cudaError_t launch_block_topk_merge(const Problem &p, const unsigned long long *cand, int slices, int span,
                                    int32_t *sel, cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Nq * p.Hkv;
    {
        TimedLaunch timed_("block_topk_merge_kernel", s);
        block_topk_merge_kernel<<<(unsigned)rows, kWarps * 32, 0, s>>>(p, cand, slices, span, sel);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_block_topk(const Problem &p, const float *bs, int32_t *sel, DeviceStatus *,
                              cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Nq * p.Hkv;
    if (rows * 4 < (long long)p.num_sms && p.nb > 4 * kSeg) {
        // few long rows: a CTA per row
        TimedLaunch timed_("block_topk_kernel", s);
        block_topk_split_kernel<<<(unsigned)rows, kWarps * 32, 0, s>>>(p, bs, sel);
    } else {
        const long long grid = (rows + kWarps - 1) / kWarps;
        TimedLaunch timed_("block_topk_kernel", s);
        block_topk_kernel<<<(unsigned)grid, kWarps * 32, 0, s>>>(p, bs, sel);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
