// inverse_index.cu -- for every (batch, group, key block) the list of query
// rows that selected that block (the key-major kernels walk these lists).
//
// Counting sort without global hot spots: CTA t of a (b, group) pair takes
// query rows [t*kRowsPerCta, (t+1)*kRowsPerCta) and histograms their selected
// blocks in shared memory; a scan kernel turns the per-CTA histograms into
// each CTA's write offset inside each bucket (and the bucket offsets), and
// the fill kernel replays the same rows with shared-memory cursors, in row
// order: every bucket lists its queries in ascending row order, the same on
// every run, so the key-major kernels accumulate dK, dV and dK_idx in a fixed
// order and the gradients are reproducible bit for bit.  Entries
// that are not a valid selection for their row (a block after the query's
// own, or beyond the keys) are reported through the status word and skipped.
// Each list entry packs the query row with the slot of the block in that
// row's selection (see pack_entry), so consumers need no search.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kRowsPerCta = 512;
constexpr int kThreads = 256;

__device__ __forceinline__ bool valid_sel(const Problem &p, int c, int i)
{
    return c >= 0 && c < p.nb && (long long)c * 128 <= (long long)p.q_offset + i;
}

// cta_hist[(br * nct + t) * nb + c] = entries of CTA t for bucket (br, c)
__global__ void __launch_bounds__(kThreads) index_count_kernel(Problem p, const int32_t *__restrict__ sel, int nct,
                                                               int32_t *__restrict__ cta_hist, DeviceStatus *st)
{
    extern __shared__ int32_t hist[];
    const int t = blockIdx.x, br = blockIdx.y;
    for (int c = threadIdx.x; c < p.nb; c += kThreads) hist[c] = 0;
    __syncthreads();
    const int i0 = t * kRowsPerCta, i1 = min(p.Nq, i0 + kRowsPerCta);
    const int32_t *base = sel + (long long)br * p.Nq * p.topk;
    for (long long x = (long long)i0 * p.topk + threadIdx.x; x < (long long)i1 * p.topk; x += kThreads) {
        const int c = base[x];
        if (c < 0) continue;
        const int i = (int)(x / p.topk);
        if (!valid_sel(p, c, i)) { report(st, kDevCheck, 51, c); continue; }
        atomicAdd(&hist[c], 1);
    }
    __syncthreads();
    int32_t *out = cta_hist + ((long long)br * nct + t) * p.nb;
    for (int c = threadIdx.x; c < p.nb; c += kThreads) out[c] = hist[c];
}

// One thread per bucket: exclusive scan over the CTAs of its (b, group);
// writes the bucket total and each CTA's offset inside the bucket.
__global__ void index_cta_scan_kernel(Problem p, int nct, const int32_t *__restrict__ cta_hist,
                                      int32_t *__restrict__ cta_base, int32_t *__restrict__ cnt)
{
    const long long bucket = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (bucket >= (long long)p.B * p.Hkv * p.nb) return;
    const long long br = bucket / p.nb;
    const int c = (int)(bucket % p.nb);
    int run = 0;
    for (int t = 0; t < nct; ++t) {
        const long long o = (br * nct + t) * p.nb + c;
        const int v = cta_hist[o];
        cta_base[o] = run;
        run += v;
    }
    cnt[bucket] = run;
}

// exclusive scan of cnt[0..n) into off[0..n], single CTA of 1024 threads
__global__ void __launch_bounds__(1024) index_bucket_scan_kernel(const int32_t *__restrict__ cnt,
                                                                 int32_t *__restrict__ off, int n)
{
    __shared__ int part[1024];
    const int per = (n + 1023) / 1024;
    const int lo = threadIdx.x * per, hi = min(n, lo + per);
    int s = 0;
    for (int x = lo; x < hi; ++x) s += cnt[x];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {
        const int v = threadIdx.x >= (unsigned)d ? part[threadIdx.x - d] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int x = lo; x < hi; ++x) {
        off[x] = run;
        run += cnt[x];
    }
    if (threadIdx.x == 1023) off[n] = part[1023];
}

// The CTA's (row, slot) entries are taken in rounds of kThreads consecutive
// entries.  Within a warp the lanes holding the same block are ranked by
// lane (__match_any_sync), and the warps of a round claim their cursor
// ranges one after another, so entries land in entry order -- row order,
// since a row selects a block at most once.
__global__ void __launch_bounds__(kThreads) index_fill_kernel(Problem p, const int32_t *__restrict__ sel, int nct,
                                                              const int32_t *__restrict__ cta_base,
                                                              const int32_t *__restrict__ off,
                                                              int32_t *__restrict__ list)
{
    extern __shared__ int32_t cursor[];
    const int t = blockIdx.x, br = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t *cb = cta_base + ((long long)br * nct + t) * p.nb;
    const int32_t *ob = off + (long long)br * p.nb;
    for (int c = threadIdx.x; c < p.nb; c += kThreads) cursor[c] = ob[c] + cb[c];
    __syncthreads();
    const int i0 = t * kRowsPerCta, i1 = min(p.Nq, i0 + kRowsPerCta);
    const int32_t *base = sel + (long long)br * p.Nq * p.topk;
    const long long x1 = (long long)i1 * p.topk;
    for (long long xb = (long long)i0 * p.topk; xb < x1; xb += kThreads) {
        const long long x = xb + threadIdx.x;
        int c = -1, i = 0;
        if (x < x1) {
            c = base[x];
            i = (int)(x / p.topk);
            if (!valid_sel(p, c, i)) c = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        const int leader = __ffs(peers) - 1;
        const int rank = __popc(peers & ((1u << lane) - 1u));
        for (int w = 0; w < kThreads / 32; ++w) {
            if (warp == w) {
                int start = 0;
                if (c >= 0 && lane == leader) {
                    start = cursor[c];
                    cursor[c] = start + __popc(peers);
                }
                start = __shfl_sync(0xffffffffu, start, leader);
                if (c >= 0) list[start + rank] = pack_entry(i, (int)(x % p.topk));
            }
            __syncthreads();
        }
    }
}

}  // namespace

size_t inverse_index_scratch_ints(const Problem &p)
{
    const long long nct = (p.Nq + kRowsPerCta - 1) / kRowsPerCta;
    return (size_t)(2 * p.B * p.Hkv * nct * p.nb);
}

cudaError_t launch_inverse_index(const Problem &p, const int32_t *sel, int32_t *cnt, int32_t *off, int32_t *scratch,
                                 int32_t *list, DeviceStatus *st, cudaStream_t s)
{
    const int nct = (p.Nq + kRowsPerCta - 1) / kRowsPerCta;
    const long long nbk = (long long)p.B * p.Hkv * p.nb;
    int32_t *cta_hist = scratch;
    int32_t *cta_base = scratch + (long long)p.B * p.Hkv * nct * p.nb;
    const size_t sm = (size_t)p.nb * sizeof(int32_t);
    if (sm > 200 * 1024) return cudaErrorInvalidValue;   // > 51200 key blocks: not supported
    cudaError_t e;
    if (sm > 48 * 1024) {
        if ((e = cudaFuncSetAttribute(index_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(index_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess) return e;
    }
    const dim3 grid(nct, p.B * p.Hkv);
    {
        TimedLaunch timed_("index_count_kernel", s);
        index_count_kernel<<<grid, kThreads, sm, s>>>(p, sel, nct, cta_hist, st);
    }
    note_launch();
    {
        TimedLaunch timed_("index_cta_scan_kernel", s);
        index_cta_scan_kernel<<<(unsigned)((nbk + 255) / 256), 256, 0, s>>>(p, nct, cta_hist, cta_base, cnt);
    }
    note_launch();
    {
        TimedLaunch timed_("index_bucket_scan_kernel", s);
        index_bucket_scan_kernel<<<1, 1024, 0, s>>>(cnt, off, (int)nbk);
    }
    note_launch();
    {
        TimedLaunch timed_("index_fill_kernel", s);
        index_fill_kernel<<<grid, kThreads, sm, s>>>(p, sel, nct, cta_base, off, list);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
