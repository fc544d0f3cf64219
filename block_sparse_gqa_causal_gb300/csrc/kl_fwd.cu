// kl_fwd.cu -- KL alignment loss of MSA ("Sparse Attention · Part II",
// section 3.2, the L_KL equation).
//
// For query i and group r over the selected token set T:
//   teacher  Pt_j = (1/G) sum_h exp(l_{h,j} - lse_h)   (main-branch weights,
//            each head normalised over T; lse_h comes from the forward)
//   student  s_j  = scale_idx <q_idx, k_idx_j>,  Ps = softmax_T(s)
//   KL(Pt || Ps) = sum_j Pt_j log Pt_j - sum_j Pt_j s_j + log sum_j exp(s_j)
// using sum_j Pt_j = 1.  All three sums are accumulated in one pass over T,
// so neither distribution is stored.  The scalar loss is
// kl_coef / (B Nq Hkv) * sum over rows, reduced in a fixed order.
//
// One CTA (4 warps) per (b, i, r), 64-token chunks of K and K_idx in a
// two-stage cp.async pipeline, warp w owns tokens [16w, 16w+16) of each
// chunk.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 64;
constexpr int kMaxChunks = 64;

template <int D, int DI>
struct KlSmem {
    static constexpr int Q_BYTES = 8 * D * 2;        // the group's heads, zero rows past G
    static constexpr int QI_BYTES = 8 * DI * 2;      // row 0: index query, rows 1..7 zero
    static constexpr int K_BYTES = kChunk * D * 2;
    static constexpr int KI_BYTES = kChunk * DI * 2;
    static constexpr int STAGE = K_BYTES + KI_BYTES;
    static constexpr int OFF_QI = Q_BYTES;
    static constexpr int OFF_STAGES = Q_BYTES + QI_BYTES;
    static constexpr int OFF_CHUNKS = OFF_STAGES + 2 * STAGE;
    static constexpr int SMEM = OFF_CHUNKS + kMaxChunks * 8;
};

template <int W>
__device__ __forceinline__ int swz(int row, int ch)
{
    return row * (W * 2) + ((ch ^ (row & 7)) << 4);
}

// Transposed tiles: MMA rows are 16 tokens, the 8 MMA columns are the
// group's heads (S^T = K Q^T) or the index query (s^T = K_idx q_idx^T, column
// 0).  Thread (g, t) of a warp then holds tokens g and g+8 for heads 2t, 2t+1;
// the teacher is a sum over heads, i.e. over the 4 lanes of a quad, and the
// per-token terms are spread over lanes t = 0 (token g) and t = 1 (token g+8).
template <int D, int DI>
__global__ void __launch_bounds__(kThreads)
kl_fwd_kernel(Problem p, const bf16 *__restrict__ q, const bf16 *__restrict__ k,
              const bf16 *__restrict__ q_idx, const bf16 *__restrict__ k_idx,
              const int32_t *__restrict__ sel, const float *__restrict__ lse,
              float *__restrict__ lse_idx, float *__restrict__ kl_rows, DeviceStatus *st)
{
    using S = KlSmem<D, DI>;
    extern __shared__ __align__(128) uint8_t smem[];
    int2 *chunks = reinterpret_cast<int2 *>(smem + S::OFF_CHUNKS);
    __shared__ int n_chunks;
    __shared__ float s_lse2[8];
    __shared__ float red[4][32][4];   // [warp][lane][A, B, m, l]

    const int i = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * p.topk;

    if (tid == 0) {
        int n = 0;
        for (int m = 0; m < p.topk; ++m) {
            const int c = srow[m];
            if (c < 0) continue;
            if ((long long)c * 128 > pos) { report(st, kDevCheck, 41, c); continue; }
            const long long start = (long long)c * 128;
            const long long end = min(min(start + 128, pos + 1), (long long)p.Nk);
            for (long long s0 = start; s0 < end && n < kMaxChunks; s0 += kChunk)
                chunks[n++] = make_int2((int)s0, (int)min((long long)kChunk, end - s0));
        }
        n_chunks = n;
    }
    if (tid < 8) s_lse2[tid] = tid < G ? lse[((long long)b * p.Hq + r * G + tid) * p.Nq + i] * kLog2e : 0.f;
    const bf16 *qrow = q + (((long long)b * p.Nq + i) * p.Hq + (long long)r * G) * D;
    for (int idx = tid; idx < 8 * (D / 8); idx += kThreads) {
        const int row = idx / (D / 8), ch = idx % (D / 8);
        cp_async16_zfill(smem + swz<D>(row, ch), qrow + (row < G ? row : 0) * D + ch * 8, row < G);
    }
    const bf16 *qirow = q_idx + (((long long)b * p.Nq + i) * p.Hkv + r) * DI;
    for (int idx = tid; idx < 8 * (DI / 8); idx += kThreads) {
        const int row = idx / (DI / 8), ch = idx % (DI / 8);
        cp_async16_zfill(smem + S::OFF_QI + swz<DI>(row, ch), qirow + ch * 8, row == 0);
    }
    cp_async_commit();
    __syncthreads();
    const int nc = n_chunks;

    const bf16 *kb = k + ((long long)b * p.kv_rows * p.Hkv + r) * D;
    const long long jstride = (long long)p.Hkv * D;
    const bf16 *kib = k_idx + (long long)b * p.kv_rows * DI;
    auto load_chunk = [&](int ci, int stage) {
        uint8_t *sk = smem + S::OFF_STAGES + stage * S::STAGE;
        uint8_t *ski = sk + S::K_BYTES;
        const int2 cj = chunks[ci];
        for (int idx = tid; idx < kChunk * (D / 8); idx += kThreads) {
            const int row = idx / (D / 8), ch = idx % (D / 8);
            const bool ok = row < cj.y;
            cp_async16_zfill(sk + swz<D>(row, ch), kb + (cj.x + (ok ? row : 0)) * jstride + ch * 8, ok);
        }
        for (int idx = tid; idx < kChunk * (DI / 8); idx += kThreads) {
            const int row = idx / (DI / 8), ch = idx % (DI / 8);
            const bool ok = row < cj.y;
            cp_async16_zfill(ski + swz<DI>(row, ch), kib + (long long)(cj.x + (ok ? row : 0)) * DI + ch * 8, ok);
        }
    };
    if (nc > 0) load_chunk(0, 0);
    cp_async_commit();

    const int g = lane >> 2, t = lane & 3;
    const float sl2 = p.scale * kLog2e;
    const float si2 = p.scale_idx * kLog2e;
    const float invG = 1.f / (float)G;
    const bool h0_ok = 2 * t < G, h1_ok = 2 * t + 1 < G;
    const float lse2_0 = s_lse2[(2 * t) & 7], lse2_1 = s_lse2[(2 * t + 1) & 7];
    // B fragments of the 8 head rows and of the index query, kept in registers
    uint32_t bq[D / 16][2], bi[DI / 16][2];
    // per-lane partial sums over the tokens it owns: sum Pt log2 Pt, sum Pt s2, online lse of s2
    float accA = 0.f, accB = 0.f, ms = -INFINITY, ls = 0.f;

    for (int ci = 0; ci < nc; ++ci) {
        const int stage = ci & 1;
        if (ci + 1 < nc) load_chunk(ci + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (ci == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                ldsm_x2(bq[ks][0], bq[ks][1], smem + swz<D>(lane & 7, ks * 2 + ((lane >> 3) & 1)));
#pragma unroll
            for (int ks = 0; ks < DI / 16; ++ks)
                ldsm_x2(bi[ks][0], bi[ks][1], smem + S::OFF_QI + swz<DI>(lane & 7, ks * 2 + ((lane >> 3) & 1)));
        }
        const uint8_t *sk = smem + S::OFF_STAGES + stage * S::STAGE;
        const uint8_t *ski = sk + S::K_BYTES;
        const int len = chunks[ci].y;
        const int kw = warp * 16;
        if (kw < len) {
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, si[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a[4];
                ldsm_x4(a[0], a[1], a[2], a[3], sk + swz<D>(kw + (lane & 15), ks * 2 + (lane >> 4)));
                mma16816(sc, a, bq[ks]);
            }
#pragma unroll
            for (int ks = 0; ks < DI / 16; ++ks) {
                uint32_t a[4];
                ldsm_x4(a[0], a[1], a[2], a[3], ski + swz<DI>(kw + (lane & 15), ks * 2 + (lane >> 4)));
                mma16816(si, a, bi[ks]);
            }
            const bool okA = kw + g < len, okB = kw + g + 8 < len;     // tokens g and g+8
            float pA = (okA && h0_ok ? exp2f(sc[0] * sl2 - lse2_0) : 0.f) + (okA && h1_ok ? exp2f(sc[1] * sl2 - lse2_1) : 0.f);
            float pB = (okB && h0_ok ? exp2f(sc[2] * sl2 - lse2_0) : 0.f) + (okB && h1_ok ? exp2f(sc[3] * sl2 - lse2_1) : 0.f);
            pA += __shfl_xor_sync(0xffffffffu, pA, 1);
            pA += __shfl_xor_sync(0xffffffffu, pA, 2);
            pB += __shfl_xor_sync(0xffffffffu, pB, 1);
            pB += __shfl_xor_sync(0xffffffffu, pB, 2);
            // index score of tokens g, g+8 sits in column 0 (lane t = 0 of the quad)
            const float sA = __shfl_sync(0xffffffffu, si[0], lane & ~3);
            const float sB = __shfl_sync(0xffffffffu, si[2], lane & ~3);
            if (t < 2 && (t == 0 ? okA : okB)) {
                const float pt = (t == 0 ? pA : pB) * invG;
                const float s2 = (t == 0 ? sA : sB) * si2;
                if (pt > 0.f) accA += pt * log2f(pt);
                accB += pt * s2;
                const float mn = fmaxf(ms, s2);
                ls = ls * exp2f(ms - mn) + exp2f(s2 - mn);
                ms = mn;
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    red[warp][lane][0] = accA;
    red[warp][lane][1] = accB;
    red[warp][lane][2] = ms;
    red[warp][lane][3] = ls;
    __syncthreads();
    if (warp == 0) {
        // lane u combines slot u of every warp, then a warp reduction
        float A = 0.f, Bs = 0.f, M = -INFINITY;
        for (int w = 0; w < 4; ++w) {
            A += red[w][lane][0];
            Bs += red[w][lane][1];
            M = fmaxf(M, red[w][lane][2]);
        }
        A = warp_sum(A);
        Bs = warp_sum(Bs);
        M = warp_max(M);
        float L = 0.f;
        for (int w = 0; w < 4; ++w)
            if (red[w][lane][3] > 0.f) L += red[w][lane][3] * exp2f(red[w][lane][2] - M);
        L = warp_sum(L);
        if (lane == 0) {
            const float lse2_idx = M + log2f(L);
            // KL in nats: (sum Pt log2 Pt - sum Pt s2 + lse2) * ln 2
            const long long oi = ((long long)b * p.Hkv + r) * p.Nq + i;
            lse_idx[oi] = lse2_idx * kLn2;
            kl_rows[oi] = (A - Bs + lse2_idx) * kLn2;
        }
    }
}

__global__ void __launch_bounds__(1024) kl_reduce_kernel(const float *__restrict__ kl_rows, long long n,
                                                          float scale, float *__restrict__ out)
{
    __shared__ double part[1024];
    // runs of 16 coalesced rows summed in fp32 (4 independent chains), each
    // run added into a double: few fp64 adds, a fixed order, fp64-level total
    double acc = 0.0;
    long long x = threadIdx.x;
    for (; x + 15 * 1024 < n; x += 16 * 1024) {
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 16; ++u) a[u & 3] += kl_rows[x + (long long)u * 1024];
        acc += (double)((a[0] + a[1]) + (a[2] + a[3]));
    }
    for (; x < n; x += 1024) acc += (double)kl_rows[x];
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = (float)(part[0] * (double)scale);
}

template <int D, int DI>
cudaError_t launch_kl_t(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                        const int32_t *sel, const float *lse, float *lse_idx, float *kl_rows,
                        DeviceStatus *st, cudaStream_t s)
{
    const int sm = KlSmem<D, DI>::SMEM;
    cudaFuncSetAttribute(kl_fwd_kernel<D, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    {
        TimedLaunch timed_("kl_fwd_kernel", s);
        kl_fwd_kernel<D, DI><<<dim3(p.Nq, p.Hkv, p.B), kThreads, sm, s>>>(p, q, k, q_idx, k_idx, sel, lse, lse_idx,
                                                                          kl_rows, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kl_fwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx,
                          const bf16 *k_idx, const int32_t *sel, const float *lse, float *lse_idx,
                          float *kl_rows, DeviceStatus *st, cudaStream_t s)
{
    if (p.d == 128 && p.d_idx == 128) return launch_kl_t<128, 128>(p, q, k, q_idx, k_idx, sel, lse, lse_idx, kl_rows, st, s);
    if (p.d == 128 && p.d_idx == 64) return launch_kl_t<128, 64>(p, q, k, q_idx, k_idx, sel, lse, lse_idx, kl_rows, st, s);
    if (p.d == 64 && p.d_idx == 128) return launch_kl_t<64, 128>(p, q, k, q_idx, k_idx, sel, lse, lse_idx, kl_rows, st, s);
    return launch_kl_t<64, 64>(p, q, k, q_idx, k_idx, sel, lse, lse_idx, kl_rows, st, s);
}

cudaError_t launch_kl_reduce(const Problem &p, const float *kl_rows, float kl_coef, float *kl_loss,
                             cudaStream_t s)
{
    const long long n = (long long)p.B * p.Hkv * p.Nq;
    const double scale = (double)kl_coef / (double)n;
    {
        TimedLaunch timed_("kl_reduce_kernel", s);
        kl_reduce_kernel<<<1, 1024, 0, s>>>(kl_rows, n, (float)scale, kl_loss);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
