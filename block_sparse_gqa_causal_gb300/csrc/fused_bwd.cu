// fused_bwd.cu -- fused main + index backward of MSA.
//
// "Sparse Attention · Part II", section 3.2: the loss is the task loss (here
// sum(dO . O)) plus the KL alignment loss; the teacher is detached and the
// selection carries no gradient, so the main branch's gradients come from dO
// alone and the index branch's from the KL alone.  The MSA kernel write-up
// on the first page fuses the two backward passes because the index
// gradient needs the main attention probabilities, and expands the KL so
// that neither distribution is materialised: with Pt the teacher and
// Ps = softmax(s) the student on the selected set,
//     dKL/ds_j = Ps_j - Pt_j       (sum_j Pt_j = 1)
// which needs only the forward's per-head lse (for Pt) and the KL pass's
// lse_idx (for Ps), both recomputed per tile from the logits.
//
// Layout: key-major.  An inverse index lists, per (b, group r, block c), the
// queries that selected c.  One CTA owns 64 keys (half a block) of one
// (b, r); it stages its K, V and K_idx rows once, then walks its query list
// in chunks of 64 (query, head) rows, recomputing S = QK^T, P, dP = dO V^T
// and dS on chip.  dK and dV of its keys accumulate in registers (one owner,
// no atomics); dK_idx (shared by all groups) accumulates in shared memory
// and is added to an fp32 buffer once; dQ and dQ_idx receive fp32
// reductions (one per selected block) and are rounded to bf16 at the end.
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 64;      // keys per CTA
constexpr int kQH = 64;        // (query, head) rows per chunk

template <int W>
__device__ __forceinline__ int swz(int row, int ch)
{
    return row * (W * 2) + ((ch ^ (row & 7)) << 4);
}

template <int D, int DI>
struct BwdSmem {
    static constexpr int QCP = 64;                       // max queries per chunk (G = 1)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + kKeys * D * 2;
    static constexpr int OFF_KI = OFF_V + kKeys * D * 2;
    static constexpr int OFF_Q = OFF_KI + kKeys * DI * 2;
    static constexpr int OFF_DO = OFF_Q + kQH * D * 2;
    static constexpr int OFF_QI = OFF_DO + kQH * D * 2;
    static constexpr int OFF_PT = OFF_QI + QCP * DI * 2;          // fp32 [64 keys][kQH + 4]
    static constexpr int PT_LD = kQH + 4;
    static constexpr int OFF_DS = OFF_PT + kKeys * PT_LD * 4;     // bf16 [64 keys][64 qh], swizzled
    static constexpr int OFF_SIG = OFF_DS + kKeys * kQH * 2;      // bf16 [64 keys][QCP]
    static constexpr int OFF_DKI = OFF_SIG + kKeys * QCP * 2;     // fp32 [64 keys][DI]
    static constexpr int OFF_ROWS = OFF_DKI + kKeys * DI * 4;
    // per-chunk row data: lse2[kQH], Dd[kQH], lsei2[QCP], qpos[QCP]
    static constexpr int SMEM = OFF_ROWS + (2 * kQH + 2 * QCP) * 4;
};

// ------------------------------------------------------------------ prep
// D[b, h, i] = sum_e dO * O over one (b, i, h) row.  A warp covers 8 rows;
// each lane loads 16 bytes of O and dO per row (all loads in flight), lanes
// sharing a row reduce with shuffles.  DD = d.
template <int DD>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(Problem p, const bf16 *__restrict__ o,
                                                         const bf16 *__restrict__ d_o, float *__restrict__ D)
{
    constexpr int LPR = DD / 8;                  // lanes per row
    constexpr int RPI = 32 / LPR;                // rows per load instruction
    constexpr int NT = 8 / RPI;
    const int lane = threadIdx.x & 31;
    const long long nrows = (long long)p.B * p.Nq * p.Hq;
    const long long row0 = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 8;
    uint4 a[NT], c[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const long long row = row0 + t * RPI + lane / LPR;
        const bool ok = row < nrows;
        a[t] = ok ? __ldg(reinterpret_cast<const uint4 *>(o + row * DD) + lane % LPR) : make_uint4(0, 0, 0, 0);
        c[t] = ok ? __ldg(reinterpret_cast<const uint4 *>(d_o + row * DD) + lane % LPR) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const uint32_t aw[4] = {a[t].x, a[t].y, a[t].z, a[t].w}, cw[4] = {c[t].x, c[t].y, c[t].z, c[t].w};
        float acc = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const float2 x = unpack_bf16(aw[q4]), y = unpack_bf16(cw[q4]);
            acc += x.x * y.x + x.y * y.y;
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long row = row0 + t * RPI + lane / LPR;
        if (lane % LPR == 0 && row < nrows) {
            const int h = (int)(row % p.Hq);
            const long long bi = row / p.Hq;
            const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
            D[((long long)b * p.Hq + h) * p.Nq + i] = acc;
        }
    }
}

__global__ void f32_to_bf16_kernel(const float *__restrict__ src, bf16 *__restrict__ dst, long long n)
{
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n / 2; x += (long long)gridDim.x * blockDim.x) {
        const float2 v = reinterpret_cast<const float2 *>(src)[x];
        reinterpret_cast<uint32_t *>(dst)[x] = pack_bf16(v.x, v.y);
    }
}

// Sums the per-slot partial rows of one output row (one warp per row):
// out[row] = sum over the valid slots s of part[row * topk + s].  Rows are
// (b, i, h) over H heads; head h belongs to group h / Gh, whose selection
// decides which slots hold a partial (same validity rule as the inverse
// index).  A row's partials are contiguous: each lane loads 16 bytes of
// several slots at once (DD/8 lanes per slot), and lanes holding the same
// features of different slots add up with shuffles.  DD = 128 or 64.
template <int DD>
__global__ void __launch_bounds__(256)
bwd_combine_kernel(Problem p, const int32_t *__restrict__ sel, const bf16 *__restrict__ part, bf16 *__restrict__ out,
                   int H, int Gh)
{
    constexpr int LPS = DD / 8;                 // lanes per slot row
    constexpr int SPI = 32 / LPS;               // slots per load instruction
    constexpr int GI = 16 / SPI;                // load instructions per group of 16 slots
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)p.B * p.Nq * H) return;
    const int h = (int)(row % H);
    const long long bi = row / H;
    const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + (((long long)b * p.Hkv + h / Gh) * p.Nq + i) * p.topk;
    const uint4 *src = reinterpret_cast<const uint4 *>(part + row * p.topk * DD);
    auto load_group = [&](uint4 (&u)[GI], int g0) {
#pragma unroll
        for (int t = 0; t < GI; ++t) {
            const int s = g0 + t * SPI + lane / LPS;
            u[t] = s < p.topk ? __ldg(src + s * LPS + lane % LPS) : make_uint4(0, 0, 0, 0);
        }
    };
    // the first 16 slots are requested before the selection arrives (invalid
    // slots are masked below, their bytes never written): one round trip
    uint4 u[GI];
    load_group(u, 0);
    const int cl = lane < p.topk ? __ldg(srow + lane) : -1;
    const unsigned mask = __ballot_sync(0xffffffffu, cl >= 0 && cl < p.nb && (long long)cl * 128 <= pos);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int g0 = 0; g0 < p.topk; g0 += 16) {
        if (g0 > 0) load_group(u, g0);
#pragma unroll
        for (int t = 0; t < GI; ++t) {
            if (!((mask >> ((g0 + t * SPI + lane / LPS) & 31)) & 1u)) continue;
            const uint32_t w[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float2 x = unpack_bf16(w[q4]);
                acc[2 * q4] += x.x;
                acc[2 * q4 + 1] += x.y;
            }
        }
    }
#pragma unroll
    for (int off = LPS; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    if (lane < LPS)
        reinterpret_cast<uint4 *>(out + row * DD)[lane] =
            make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                       pack_bf16(acc[6], acc[7]));
}

// ------------------------------------------------------------------ main
template <int D, int DI>
__global__ void __launch_bounds__(kThreads, 1)
fused_bwd_kernel(Problem p, const bf16 *__restrict__ q, const bf16 *__restrict__ k, const bf16 *__restrict__ v,
                 const bf16 *__restrict__ d_o, const float *__restrict__ lse, const bf16 *__restrict__ q_idx,
                 const bf16 *__restrict__ k_idx, const float *__restrict__ lse_idx, float kl_coef,
                 const float *__restrict__ Dg, const int32_t *__restrict__ bucket_off,
                 const int32_t *__restrict__ bucket_q, bf16 *__restrict__ dk, bf16 *__restrict__ dv,
                 float *__restrict__ dq_acc, float *__restrict__ dqi_acc, float *__restrict__ dki_acc)
{
    using S = BwdSmem<D, DI>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sK = smem + S::OFF_K;
    uint8_t *sV = smem + S::OFF_V;
    uint8_t *sKi = smem + S::OFF_KI;
    uint8_t *sQ = smem + S::OFF_Q;
    uint8_t *sdO = smem + S::OFF_DO;
    uint8_t *sQi = smem + S::OFF_QI;
    float *sPT = reinterpret_cast<float *>(smem + S::OFF_PT);
    uint8_t *sDS = smem + S::OFF_DS;
    bf16 *sSig = reinterpret_cast<bf16 *>(smem + S::OFF_SIG);
    float *sDKI = reinterpret_cast<float *>(smem + S::OFF_DKI);
    float *sLse2 = reinterpret_cast<float *>(smem + S::OFF_ROWS);
    float *sDd = sLse2 + kQH;
    float *sLsei2 = sDd + kQH;
    int *sPos = reinterpret_cast<int *>(sLsei2 + S::QCP);

    const int G = p.G;
    const int QC = kQH / G;                 // queries per chunk
    const int QCP = QC < 16 ? 16 : QC;      // padded to a k16 / m16 tile
    const int NQT = QCP / 8;                // n-tiles over queries
    const int c = blockIdx.x >> 1, half = blockIdx.x & 1;
    const int r = blockIdx.y, b = blockIdx.z;
    const long long j0 = (long long)c * 128 + half * kKeys;
    const int nkeys = (int)min((long long)kKeys, (long long)p.Nk - j0);
    if (nkeys <= 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kw = warp * 16;
    const float sl2 = p.scale * kLog2e, si2 = p.scale_idx * kLog2e;
    const float coef = kl_coef / ((float)p.B * (float)p.Nq * (float)p.Hkv);
    const long long jstride = (long long)p.Hkv * D;

    // stage this CTA's keys: K, V (head r) and K_idx; zero the dK_idx accumulator
    {
        const bf16 *kb = k + ((long long)b * p.kv_rows * p.Hkv + r) * D;
        const bf16 *vb = v + ((long long)b * p.kv_rows * p.Hkv + r) * D;
        const bf16 *kib = k_idx + (long long)b * p.kv_rows * DI;
        for (int idx = tid; idx < kKeys * (D / 8); idx += kThreads) {
            const int row = idx / (D / 8), ch = idx % (D / 8);
            const bool ok = row < nkeys;
            const long long j = j0 + (ok ? row : 0);
            cp_async16_zfill(sK + swz<D>(row, ch), kb + j * jstride + ch * 8, ok);
            cp_async16_zfill(sV + swz<D>(row, ch), vb + j * jstride + ch * 8, ok);
        }
        for (int idx = tid; idx < kKeys * (DI / 8); idx += kThreads) {
            const int row = idx / (DI / 8), ch = idx % (DI / 8);
            const bool ok = row < nkeys;
            cp_async16_zfill(sKi + swz<DI>(row, ch), kib + (j0 + (ok ? row : 0)) * DI + ch * 8, ok);
        }
        cp_async_commit();
        for (int idx = tid; idx < kKeys * DI; idx += kThreads) sDKI[idx] = 0.f;
    }

    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];

    float acc_dk[D / 8][4], acc_dv[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_dk[n][e] = acc_dv[n][e] = 0.f;

    for (int qc = qbeg; qc < qend; qc += QC) {
        const int nq = min(QC, qend - qc);
        // ---- load the chunk's rows
        for (int idx = tid; idx < kQH * (D / 8); idx += kThreads) {
            const int row = idx / (D / 8), ch = idx % (D / 8);
            const int qq = row / G, gg = row % G;
            const bool ok = qq < nq;
            const int i = ok ? entry_row(bucket_q[qc + qq]) : 0;
            const long long off = (((long long)b * p.Nq + i) * p.Hq + (long long)r * G + gg) * D + ch * 8;
            cp_async16_zfill(sQ + swz<D>(row, ch), q + off, ok);
            cp_async16_zfill(sdO + swz<D>(row, ch), d_o + off, ok);
        }
        for (int idx = tid; idx < QCP * (DI / 8); idx += kThreads) {
            const int row = idx / (DI / 8), ch = idx % (DI / 8);
            const bool ok = row < nq;
            const int i = ok ? entry_row(bucket_q[qc + row]) : 0;
            cp_async16_zfill(sQi + swz<DI>(row, ch), q_idx + (((long long)b * p.Nq + i) * p.Hkv + r) * DI + ch * 8, ok);
        }
        cp_async_commit();
        for (int row = tid; row < kQH; row += kThreads) {
            const int qq = row / G, gg = row % G;
            if (qq < nq) {
                const int i = entry_row(bucket_q[qc + qq]);
                const long long hi = ((long long)b * p.Hq + r * G + gg) * p.Nq + i;
                sLse2[row] = lse[hi] * kLog2e;
                sDd[row] = Dg[hi];
            } else {
                sLse2[row] = INFINITY;
                sDd[row] = 0.f;
            }
        }
        for (int row = tid; row < QCP; row += kThreads) {
            if (row < nq) {
                const int i = entry_row(bucket_q[qc + row]);
                sLsei2[row] = lse_idx[((long long)b * p.Hkv + r) * p.Nq + i] * kLog2e;
                sPos[row] = i;   // q_offset == 0
            } else {
                sLsei2[row] = INFINITY;
                sPos[row] = -1;
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // ---- main branch: per warp, keys kw..kw+15 against all 64 rows
#pragma unroll
        for (int sc = 0; sc < 2; ++sc) {
            float accS[4][4], accP[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) accS[n][e] = accP[n][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t ak[4], av[4];
                ldsm_x4(ak[0], ak[1], ak[2], ak[3], sK + swz<D>(kw + (lane & 15), ks * 2 + (lane >> 4)));
                ldsm_x4(av[0], av[1], av[2], av[3], sV + swz<D>(kw + (lane & 15), ks * 2 + (lane >> 4)));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    const int row = sc * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int ch = ks * 2 + ((lane >> 3) & 1);
                    uint32_t bq0[2], bq1[2], bd0[2], bd1[2];
                    ldsm_x4(bq0[0], bq0[1], bq1[0], bq1[1], sQ + swz<D>(row, ch));
                    ldsm_x4(bd0[0], bd0[1], bd1[0], bd1[1], sdO + swz<D>(row, ch));
                    mma16816(accS[np * 2], ak, bq0);
                    mma16816(accS[np * 2 + 1], ak, bq1);
                    mma16816(accP[np * 2], av, bd0);
                    mma16816(accP[np * 2 + 1], av, bd1);
                }
            }
            // P^T and dS^T on this warp's 16 keys x 32 rows
#pragma unroll
            for (int n = 0; n < 4; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = kw + g + (e >> 1) * 8;          // row of the C fragment
                    const int qh = sc * 32 + n * 8 + 2 * t + (e & 1);
                    const int pos = sPos[qh / G];
                    const bool ok = key < nkeys && (j0 + key) <= pos;
                    const float pr = ok ? exp2f(accS[n][e] * sl2 - sLse2[qh]) : 0.f;
                    accS[n][e] = pr;
                    accP[n][e] = pr * (accP[n][e] - sDd[qh]);
                    sPT[key * S::PT_LD + qh] = pr;
                }
                const int ch = (sc * 32 + n * 8) / 8;   // 16-byte chunk of the qh row
                // dS^T bf16 rows key g and g+8, columns 2t, 2t+1 of chunk ch
                *reinterpret_cast<uint32_t *>(sDS + swz<kQH>(kw + g, ch) + 4 * t) = pack_bf16(accP[n][0], accP[n][1]);
                *reinterpret_cast<uint32_t *>(sDS + swz<kQH>(kw + g + 8, ch) + 4 * t) = pack_bf16(accP[n][2], accP[n][3]);
            }
            // dV += P^T dO, dK += dS^T Q  (k = 32 rows of this sub-chunk)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t ap[4], as[4];
                ap[0] = pack_bf16(accS[2 * kk][0], accS[2 * kk][1]);
                ap[1] = pack_bf16(accS[2 * kk][2], accS[2 * kk][3]);
                ap[2] = pack_bf16(accS[2 * kk + 1][0], accS[2 * kk + 1][1]);
                ap[3] = pack_bf16(accS[2 * kk + 1][2], accS[2 * kk + 1][3]);
                as[0] = pack_bf16(accP[2 * kk][0], accP[2 * kk][1]);
                as[1] = pack_bf16(accP[2 * kk][2], accP[2 * kk][3]);
                as[2] = pack_bf16(accP[2 * kk + 1][0], accP[2 * kk + 1][1]);
                as[3] = pack_bf16(accP[2 * kk + 1][2], accP[2 * kk + 1][3]);
                const int rowb = sc * 32 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int np = 0; np < D / 16; ++np) {
                    const int ch = np * 2 + (lane >> 4);
                    uint32_t bd0[2], bd1[2], bq0[2], bq1[2];
                    ldsm_x4_t(bd0[0], bd0[1], bd1[0], bd1[1], sdO + swz<D>(rowb, ch));
                    ldsm_x4_t(bq0[0], bq0[1], bq1[0], bq1[1], sQ + swz<D>(rowb, ch));
                    mma16816(acc_dv[np * 2], ap, bd0);
                    mma16816(acc_dv[np * 2 + 1], ap, bd1);
                    mma16816(acc_dk[np * 2], as, bq0);
                    mma16816(acc_dk[np * 2 + 1], as, bq1);
                }
            }
        }
        __syncthreads();   // sPT and sDS complete

        // ---- dQ rows [16w, 16w+16) = dS (rows x 64 keys) K (64 keys x D), two column halves
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            float acc[D / 16][4];
#pragma unroll
            for (int n = 0; n < D / 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kKeys / 16; ++ks) {
                uint32_t a[4];
                ldsm_x4_t(a[0], a[1], a[2], a[3],
                          sDS + swz<kQH>(ks * 16 + (lane & 7) + ((lane >> 4) << 3), 2 * warp + ((lane >> 3) & 1)));
#pragma unroll
                for (int np = 0; np < D / 32; ++np) {
                    uint32_t b0[2], b1[2];
                    ldsm_x4_t(b0[0], b0[1], b1[0], b1[1],
                              sK + swz<D>(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                          hc * (D / 16) + np * 2 + (lane >> 4)));
                    mma16816(acc[np * 2], a, b0);
                    mma16816(acc[np * 2 + 1], a, b1);
                }
            }
#pragma unroll
            for (int half8 = 0; half8 < 2; ++half8) {
                const int qh = warp * 16 + g + half8 * 8;
                const int qq = qh / G, gg = qh % G;
                if (qq < nq) {
                    const int i = entry_row(bucket_q[qc + qq]);
                    float *dst = dq_acc + (((long long)b * p.Nq + i) * p.Hq + (long long)r * G + gg) * D + hc * (D / 2);
#pragma unroll
                    for (int n = 0; n < D / 16; ++n) {
                        red_add(dst + n * 8 + 2 * t, p.scale * acc[n][half8 * 2]);
                        red_add(dst + n * 8 + 2 * t + 1, p.scale * acc[n][half8 * 2 + 1]);
                    }
                }
            }
        }

        // ---- index branch: s^T = K_idx Q_idx^T on this warp's keys
        {
            float accI[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) accI[n][0] = accI[n][1] = accI[n][2] = accI[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < DI / 16; ++ks) {
                uint32_t a[4];
                ldsm_x4(a[0], a[1], a[2], a[3], sKi + swz<DI>(kw + (lane & 15), ks * 2 + (lane >> 4)));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np * 2 < NQT) {
                        uint32_t b0[2], b1[2];
                        ldsm_x4(b0[0], b0[1], b1[0], b1[1],
                                sQi + swz<DI>(np * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)));
                        mma16816(accI[np * 2], a, b0);
                        mma16816(accI[np * 2 + 1], a, b1);
                    }
                }
            }
            // dsigma^T = coef (Ps - Pt) -> registers (as A fragments) and smem (for dQ_idx)
            const float invG = 1.f / (float)G;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                if (n < NQT) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = kw + g + (e >> 1) * 8;
                        const int qq = n * 8 + 2 * t + (e & 1);
                        const int pos = sPos[qq];
                        const bool ok = key < nkeys && (j0 + key) <= pos;
                        float ds = 0.f;
                        if (ok) {
                            const float ps = exp2f(accI[n][e] * si2 - sLsei2[qq]);
                            float pt = 0.f;
                            for (int gg = 0; gg < G; ++gg) pt += sPT[key * S::PT_LD + qq * G + gg];
                            ds = coef * (ps - pt * invG);
                        }
                        accI[n][e] = ds;
                    }
                    reinterpret_cast<uint32_t *>(sSig + (kw + g) * S::QCP)[n * 4 + t] = pack_bf16(accI[n][0], accI[n][1]);
                    reinterpret_cast<uint32_t *>(sSig + (kw + g + 8) * S::QCP)[n * 4 + t] = pack_bf16(accI[n][2], accI[n][3]);
                }
            }
            // dK_idx (this warp's 16 keys x DI) += dsigma^T (16 x QCP) Q_idx (QCP x DI), in column quarters
#pragma unroll
            for (int qd = 0; qd < DI / 32; ++qd) {
                float acc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (kk * 2 < NQT) {
                        uint32_t a[4];
                        a[0] = pack_bf16(accI[2 * kk][0], accI[2 * kk][1]);
                        a[1] = pack_bf16(accI[2 * kk][2], accI[2 * kk][3]);
                        a[2] = pack_bf16(accI[2 * kk + 1][0], accI[2 * kk + 1][1]);
                        a[3] = pack_bf16(accI[2 * kk + 1][2], accI[2 * kk + 1][3]);
                        const int rowb = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                        for (int np = 0; np < 2; ++np) {
                            uint32_t b0[2], b1[2];
                            ldsm_x4_t(b0[0], b0[1], b1[0], b1[1], sQi + swz<DI>(rowb, qd * 4 + np * 2 + (lane >> 4)));
                            mma16816(acc[np * 2], a, b0);
                            mma16816(acc[np * 2 + 1], a, b1);
                        }
                    }
                }
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    float *d0 = sDKI + (kw + g) * DI + qd * 32 + n * 8 + 2 * t;
                    float *d1 = sDKI + (kw + g + 8) * DI + qd * 32 + n * 8 + 2 * t;
                    d0[0] += acc[n][0];
                    d0[1] += acc[n][1];
                    d1[0] += acc[n][2];
                    d1[1] += acc[n][3];
                }
            }
        }
        __syncthreads();   // sSig complete

        // ---- dQ_idx (QCP x DI) = dsigma (QCP x 64 keys) K_idx (64 x DI); warp w owns DI/4 columns
        {
            constexpr int NT = DI / 32;     // n-tiles per warp (4 or 2)
            for (int mt = 0; mt < QCP / 16; ++mt) {
                float acc[NT][4];
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks) {
                    uint32_t a[4];
                    // A = dsigma rows (queries) from the [key][q] buffer, transposed on load
                    const int krow = ks * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int qcol = mt * 16 + ((lane >> 3) & 1) * 8;
                    ldsm_x4_t(a[0], a[1], a[2], a[3], sSig + krow * S::QCP + qcol);
#pragma unroll
                    for (int np = 0; np < NT / 2; ++np) {
                        uint32_t b0[2], b1[2];
                        ldsm_x4_t(b0[0], b0[1], b1[0], b1[1],
                                  sKi + swz<DI>(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                                warp * (NT) + np * 2 + (lane >> 4)));
                        mma16816(acc[np * 2], a, b0);
                        mma16816(acc[np * 2 + 1], a, b1);
                    }
                }
#pragma unroll
                for (int half8 = 0; half8 < 2; ++half8) {
                    const int qq = mt * 16 + g + half8 * 8;
                    if (qq < nq) {
                        const int i = entry_row(bucket_q[qc + qq]);
                        float *dst = dqi_acc + (((long long)b * p.Nq + i) * p.Hkv + r) * DI + warp * (DI / 4);
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            red_add(dst + n * 8 + 2 * t, p.scale_idx * acc[n][half8 * 2]);
                            red_add(dst + n * 8 + 2 * t + 1, p.scale_idx * acc[n][half8 * 2 + 1]);
                        }
                    }
                }
            }
        }
        __syncthreads();   // before the next chunk overwrites the row buffers
    }

    // ---- write dK, dV of this CTA's keys; add dK_idx into the fp32 buffer
#pragma unroll
    for (int half8 = 0; half8 < 2; ++half8) {
        const int key = kw + g + half8 * 8;
        if (key < nkeys) {
            const long long j = j0 + key;
            bf16 *pk = dk + ((long long)b * p.kv_rows + j) * jstride + (long long)r * D;
            bf16 *pv = dv + ((long long)b * p.kv_rows + j) * jstride + (long long)r * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                *reinterpret_cast<uint32_t *>(pk + n * 8 + 2 * t) =
                    pack_bf16(p.scale * acc_dk[n][half8 * 2], p.scale * acc_dk[n][half8 * 2 + 1]);
                *reinterpret_cast<uint32_t *>(pv + n * 8 + 2 * t) =
                    pack_bf16(acc_dv[n][half8 * 2], acc_dv[n][half8 * 2 + 1]);
            }
        }
    }
    if (qend > qbeg) {
        for (int idx = tid; idx < nkeys * DI; idx += kThreads) {
            const int key = idx / DI, col = idx % DI;
            red_add(dki_acc + ((long long)b * p.kv_rows + j0 + key) * DI + col, p.scale_idx * sDKI[idx]);
        }
    }
}

template <int D, int DI>
cudaError_t launch_main(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *d_o,
                        const float *lse, const bf16 *q_idx, const bf16 *k_idx, const float *lse_idx, float kl_coef,
                        const BwdWork &w, bf16 *dk, bf16 *dv, cudaStream_t s)
{
    const int sm = BwdSmem<D, DI>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(fused_bwd_kernel<D, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (e != cudaSuccess) return e;
    {
        TimedLaunch timed_("fused_bwd_kernel", s);
        fused_bwd_kernel<D, DI><<<dim3(p.nb * 2, p.Hkv, p.B), kThreads, sm, s>>>(
            p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w.D, w.bucket_off, w.bucket_q, dk, dv, w.dq_acc,
            w.dqi_acc, w.dki_acc);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_combine(const Problem &p, const int32_t *sel, const bf16 *part, bf16 *out, int H, int Gh,
                               cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Nq * H;
    {
        TimedLaunch timed_("bwd_combine_kernel", s);
        bwd_combine_kernel<128><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, part, out, H, Gh);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_fused_bwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *o,
                             const bf16 *d_o, const float *lse, const bf16 *q_idx, const bf16 *k_idx,
                             const int32_t *sel, const float *lse_idx, float kl_coef, bf16 *dq, bf16 *dk, bf16 *dv,
                             bf16 *dq_idx, bf16 *dk_idx, const BwdWork &w, DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e;
    const long long n_dq = (long long)p.B * p.Nq * p.Hq * p.d;
    const long long n_dqi = (long long)p.B * p.Nq * p.Hkv * p.d_idx;
    const long long n_dki = (long long)p.B * p.Nk * p.d_idx;
    const bool tc = bwd_tc(p);
    if (!tc) {
        if ((e = cudaMemsetAsync(w.dq_acc, 0, n_dq * 4, s)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(w.dqi_acc, 0, n_dqi * 4, s)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(w.dki_acc, 0, n_dki * 4, s)) != cudaSuccess) return e;
    }

    const long long rows = (long long)p.B * p.Nq * p.Hq;
    if (!w.D_ready) {
        {
            TimedLaunch timed_("bwd_rowdot_kernel", s);
            if (p.d == 128) bwd_rowdot_kernel<128><<<(unsigned)((rows + 63) / 64), 256, 0, s>>>(p, o, d_o, w.D);
            else bwd_rowdot_kernel<64><<<(unsigned)((rows + 63) / 64), 256, 0, s>>>(p, o, d_o, w.D);
        }
        note_launch();
    }
    if (!w.index_ready &&
        (e = launch_inverse_index(p, sel, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, st, s)) != cudaSuccess)
        return e;

    if (tc) {
        // main branch: dK, dV and the dQ partial rows
        if ((e = launch_bwd_main_tc(p, q, k, v, d_o, lse, w, dk, dv, st, s)) != cudaSuccess) return e;
        // index branch: the teacher rebuilt from its own logit tiles next to the index
        // scores; dq_idx partial rows, each group's dK_idx share and the KL loss terms
        if ((e = launch_index_teacher_tc(p, q, k, q_idx, k_idx, lse, lse_idx, kl_coef, w.bucket_off, w.bucket_q, w.klt,
                                         w.dqi_part, w.dki_acc, st, s)) != cudaSuccess)
            return e;
        if (w.klt && (e = launch_kl_rows_combine(p, sel, lse_idx, w.klt, w.kl_rows, s)) != cudaSuccess) return e;
        {
            TimedLaunch timed_("bwd_combine_kernel", s);
            bwd_combine_kernel<128><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, w.dq_part, dq, p.Hq, p.G);
        }
        note_launch();
        const long long rows_i = (long long)p.B * p.Nq * p.Hkv;
        {
            TimedLaunch timed_("bwd_combine_kernel", s);
            bwd_combine_kernel<128><<<(unsigned)((rows_i + 7) / 8), 256, 0, s>>>(p, sel, w.dqi_part, dq_idx, p.Hkv, 1);
        }
        note_launch();
        if ((e = launch_dki_group_sum(p, w.dki_acc, dk_idx, s)) != cudaSuccess) return e;
        return cudaGetLastError();
    } else {
        if (p.d == 128) e = launch_main<128, 64>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, s);
        else if (p.d_idx == 128) e = launch_main<64, 128>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, s);
        else e = launch_main<64, 64>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, s);
        if (e != cudaSuccess) return e;
        {
            TimedLaunch timed_("f32_to_bf16_kernel", s);
            f32_to_bf16_kernel<<<4 * p.num_sms, 256, 0, s>>>(w.dq_acc, dq, n_dq);
        }
        note_launch();
        {
            TimedLaunch timed_("f32_to_bf16_kernel", s);
            f32_to_bf16_kernel<<<4 * p.num_sms, 256, 0, s>>>(w.dqi_acc, dq_idx, n_dqi);
        }
        note_launch();
    }
    {
        TimedLaunch timed_("f32_to_bf16_kernel", s);
        f32_to_bf16_kernel<<<4 * p.num_sms, 256, 0, s>>>(w.dki_acc, dk_idx, n_dki);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
