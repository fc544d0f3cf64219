// sparse_attn_fwd.cu -- main branch of MSA: exact block-sparse GQA attention.
//
// "Sparse Attention · Part II", section 3.2: every query head of a group
// attends, with its own logits, to the causally visible tokens of the
// blocks selected for (query, group) and normalises over that set only.
// Flash-style: scores, the running max/sum and the output accumulator stay
// on chip (section 4.1 of the same page); each K/V tile is staged once in
// shared memory and used by all G heads of the group (section 3.2 notes the
// selected blocks' KV loads can be shared across the group's heads).
//
// One CTA (4 warps) per (b, i, r), or, when those are too few to fill the
// GPU (decode), nsplit CTAs per (b, i, r) each taking a contiguous share of
// the row's chunks (split-KV, as in flash decoding): they write unnormalised
// partial states that sparse_attn_merge_kernel folds.  The selected blocks
// are cut into 64-token chunks (the local block stops at the query); chunks
// stream through a two-stage cp.async pipeline.  Warp w handles tokens
// [16w, 16w+16) of every chunk with its own online softmax; the four partial
// states are merged at the end.  MMA rows are the G heads (padded to 16).
#include <algorithm>
#include <type_traits>

#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 64;
constexpr int kMaxChunks = 64;   // 2 chunks per block, topk <= 32

template <int D>
struct FwdSmem {
    static constexpr int ROW = D * 2;                   // bytes per bf16 row
    static constexpr int Q_BYTES = 16 * ROW;
    static constexpr int KV_BYTES = kChunk * ROW;       // one K or V chunk
    static constexpr int STAGE = 2 * KV_BYTES;          // K + V
    static constexpr int OFF_STAGES = Q_BYTES;
    static constexpr int OFF_CHUNKS = OFF_STAGES + 2 * STAGE;
    static constexpr int SMEM = OFF_CHUNKS + kMaxChunks * 8;
};

template <int D>
__device__ __forceinline__ int swz(int row, int ch)
{
    return row * (D * 2) + ((ch ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads)
sparse_attn_fwd_kernel(Problem p, const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                       const bf16 *__restrict__ v, const int32_t *__restrict__ sel,
                       bf16 *__restrict__ o, float *__restrict__ lse, int nsplit, float *__restrict__ part_o,
                       float2 *__restrict__ part_ml, DeviceStatus *st)
{
    using S = FwdSmem<D>;
    constexpr int CH = D / 8;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sQ = smem;
    int2 *chunks = reinterpret_cast<int2 *>(smem + S::OFF_CHUNKS);
    __shared__ int n_chunks;

    const int i = blockIdx.x / nsplit, sp = blockIdx.x % nsplit, r = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * p.topk;

    if (warp == 0) {
        // the row's chunk list, in selection order: lane m takes selected block m
        // (topk <= 32), its chunks go after those of the lanes below it
        const int c = lane < p.topk ? srow[lane] : -1;
        long long start = 0, end = 0;
        if (c >= 0) {
            if ((long long)c * 128 > pos) report(st, kDevCheck, 31, c);
            else {
                start = (long long)c * 128;
                end = min(min(start + 128, pos + 1), (long long)p.Nk);
            }
        }
        const int nck = end > start ? (int)((end - start + kChunk - 1) / kChunk) : 0;
        int off = nck;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o2 = __shfl_up_sync(0xffffffffu, off, d);
            if (lane >= d) off += o2;
        }
        off -= nck;
        for (int x = 0; x < nck; ++x) {
            const long long s0 = start + (long long)x * kChunk;
            chunks[off + x] = make_int2((int)s0, (int)min((long long)kChunk, end - s0));
        }
        if (lane == 31) n_chunks = off + nck;
    }
    // Q rows of the group's heads (rows >= G are zero)
    const bf16 *qrow = q + (((long long)b * p.Nq + i) * p.Hq + (long long)r * G) * D;
    for (int idx = tid; idx < 16 * CH; idx += kThreads) {
        const int row = idx / CH, ch = idx % CH;
        cp_async16_zfill(sQ + swz<D>(row, ch), qrow + (row < G ? row : 0) * D + ch * 8, row < G);
    }
    cp_async_commit();
    __syncthreads();
    // this CTA's share of the row's chunks
    const int c_lo = (int)((long long)n_chunks * sp / nsplit), c_hi = (int)((long long)n_chunks * (sp + 1) / nsplit);
    const int nc = c_hi - c_lo;

    const bf16 *kb = k + ((long long)b * p.kv_rows * p.Hkv + r) * D;
    const bf16 *vb = v + ((long long)b * p.kv_rows * p.Hkv + r) * D;
    const long long jstride = (long long)p.Hkv * D;
    auto load_chunk = [&](int ci, int stage) {
        uint8_t *sk = smem + S::OFF_STAGES + stage * S::STAGE;
        uint8_t *sv = sk + S::KV_BYTES;
        const int2 cj = chunks[c_lo + ci];
        for (int idx = tid; idx < kChunk * CH; idx += kThreads) {
            const int row = idx / CH, ch = idx % CH;
            const bool ok = row < cj.y;
            const long long j = cj.x + (ok ? row : 0);
            cp_async16_zfill(sk + swz<D>(row, ch), kb + j * jstride + ch * 8, ok);
            cp_async16_zfill(sv + swz<D>(row, ch), vb + j * jstride + ch * 8, ok);
        }
    };
    if (nc > 0) load_chunk(0, 0);
    cp_async_commit();

    const int g = lane >> 2, t = lane & 3;
    const float sl2 = p.scale * kLog2e;
    uint32_t af[D / 16][4];
    float acc_o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc_o[n][0] = acc_o[n][1] = acc_o[n][2] = acc_o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // row g (rows g+8 are padding)

    for (int ci = 0; ci < nc; ++ci) {
        const int stage = ci & 1;
        if (ci + 1 < nc) load_chunk(ci + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (ci == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                ldsm_x4(af[ks][0], af[ks][1], af[ks][2], af[ks][3], sQ + swz<D>(lane & 15, ks * 2 + (lane >> 4)));
        }
        const uint8_t *sk = smem + S::OFF_STAGES + stage * S::STAGE;
        const uint8_t *sv = sk + S::KV_BYTES;
        const int len = chunks[c_lo + ci].y;
        const int kw = warp * 16;           // this warp's first token in the chunk
        if (kw < len) {
            float sc[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t b0[2], b1[2];
                ldsm_x4(b0[0], b0[1], b1[0], b1[1],
                        sk + swz<D>(kw + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)));
                mma16816(sc[0], af[ks], b0);
                mma16816(sc[1], af[ks], b1);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kk = kw + n * 8 + 2 * t + e;
                    sc[n][e] = kk < len ? sc[n][e] * sl2 : -INFINITY;
                    mx = fmaxf(mx, sc[n][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);          // finite: token kw is valid
            const float alpha = exp2f(m_run - m_new);       // 0 when m_run = -inf
            float ps = 0.f;
            uint32_t pa[4];
            float pv[2][2];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    pv[n][e] = exp2f(sc[n][e] - m_new);
                    ps += pv[n][e];
                }
            pa[0] = pack_bf16(pv[0][0], pv[0][1]);
            pa[1] = 0u;                                     // rows g+8: padding
            pa[2] = pack_bf16(pv[1][0], pv[1][1]);
            pa[3] = 0u;
            l_run = l_run * alpha + ps;
            m_run = m_new;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                acc_o[n][0] *= alpha;
                acc_o[n][1] *= alpha;
            }
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0[2], b1[2];
                ldsm_x4_t(b0[0], b0[1], b1[0], b1[1],
                          sv + swz<D>(kw + (lane & 7) + (((lane >> 3) & 1) << 3), np * 2 + (lane >> 4)));
                mma16816(acc_o[np * 2], pa, b0);
                mma16816(acc_o[np * 2 + 1], pa, b1);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the four warps' partial states (rows g < G only)
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    float *sO = reinterpret_cast<float *>(smem + S::OFF_STAGES);     // [4][8][D]
    float *sM = sO + 4 * 8 * D;                                       // [4][8]
    float *sL = sM + 4 * 8;
    if (g < G) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            sO[(warp * 8 + g) * D + n * 8 + 2 * t] = acc_o[n][0];
            sO[(warp * 8 + g) * D + n * 8 + 2 * t + 1] = acc_o[n][1];
        }
        if (t == 0) {
            sM[warp * 8 + g] = m_run;
            sL[warp * 8 + g] = l_run;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kThreads) {
        const int h = idx / D, col = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sM[w * 8 + h]);
        float L = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = M == -INFINITY ? 0.f : exp2f(sM[w * 8 + h] - M);
            L += f * sL[w * 8 + h];
            acc += f * sO[(w * 8 + h) * D + col];
        }
        const int hh = r * G + h;
        const long long orow = ((long long)b * p.Nq + i) * p.Hq + hh;
        if (nsplit == 1) {
            o[orow * D + col] = __float2bfloat16_rn(acc / L);
            if (col == 0) lse[((long long)b * p.Hq + hh) * p.Nq + i] = (M + log2f(L)) * kLn2;
        } else {
            // unnormalised partial state of this share (M = -inf, L = 0 when it holds no token)
            part_o[(orow * nsplit + sp) * D + col] = acc;
            if (col == 0) part_ml[orow * nsplit + sp] = make_float2(M, L);
        }
    }
}

// Folds the nsplit partial states of one (b, i, h) row: warp per row.
template <int D>
__global__ void __launch_bounds__(256) sparse_attn_merge_kernel(Problem p, int nsplit, const float *__restrict__ part_o,
                                                                const float2 *__restrict__ part_ml,
                                                                bf16 *__restrict__ o, float *__restrict__ lse)
{
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)p.B * p.Nq * p.Hq) return;
    constexpr int PER = D / 32;
    // the first eight shares' rows are requested together with the (max, sum) pairs
    float x[8][PER];
    auto load8 = [&](int s0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float *src = part_o + (row * nsplit + min(s0 + u, nsplit - 1)) * D;
#pragma unroll
            for (int e = 0; e < PER; ++e) x[u][e] = __ldg(src + lane + 32 * e);
        }
    };
    load8(0);
    const float2 ml = lane < nsplit ? part_ml[row * nsplit + lane] : make_float2(-INFINITY, 0.f);
    float M = ml.x;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
    float L = f * ml.y;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    // eight shares' rows in flight at a time
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
        if (s0 > 0) load8(s0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float w = s0 + u < nsplit ? __shfl_sync(0xffffffffu, f, (s0 + u) & 31) : 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = w != 0.f ? fmaf(w, x[u][e], acc[e]) : acc[e];
        }
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < PER; ++e) o[row * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
    if (lane == 0) {
        const int h = (int)(row % p.Hq);
        const long long bi = row / p.Hq;
        const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
        lse[((long long)b * p.Hq + h) * p.Nq + i] = (M + log2f(L)) * kLn2;
    }
}

}  // namespace

int sparse_attn_splits(const Problem &p)
{
    const long long ctas = (long long)p.Nq * p.Hkv * p.B;
    if (ctas >= p.num_sms) return 1;
    // about one CTA per SM (more shares only lengthen the merge: at 1M-token decode the
    // kernel takes the same time with 5 to 32 shares), at most 32 shares (the merge
    // holds one per lane) and at most one per 64-token chunk
    return (int)std::min<long long>(std::min<long long>(32, 2LL * p.topk), ((long long)p.num_sms + ctas - 1) / ctas);
}

cudaError_t launch_sparse_attn_fwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v,
                                   const int32_t *sel, bf16 *o, float *lse, float *split_ws, DeviceStatus *st,
                                   cudaStream_t s)
{
    const int nsplit = split_ws ? sparse_attn_splits(p) : 1;
    const long long rows = (long long)p.B * p.Nq * p.Hq;
    float *part_o = split_ws;
    float2 *part_ml = split_ws ? reinterpret_cast<float2 *>(split_ws + rows * nsplit * p.d) : nullptr;
    dim3 grid(p.Nq * nsplit, p.Hkv, p.B);
    auto run = [&](auto dtag) {
        constexpr int D = decltype(dtag)::value;
        const int sm = FwdSmem<D>::SMEM;
        cudaFuncSetAttribute(sparse_attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        {
            TimedLaunch timed_("sparse_attn_fwd_kernel", s);
            sparse_attn_fwd_kernel<D><<<grid, kThreads, sm, s>>>(p, q, k, v, sel, o, lse, nsplit, part_o, part_ml, st);
        }
        note_launch();
        if (nsplit > 1) {
            {
                TimedLaunch timed_("sparse_attn_merge_kernel", s);
                sparse_attn_merge_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, nsplit, part_o, part_ml, o, lse);
            }
            note_launch();
        }
    };
    if (p.d == 128) run(std::integral_constant<int, 128>{});
    else run(std::integral_constant<int, 64>{});
    return cudaGetLastError();
}

}  // namespace msa
