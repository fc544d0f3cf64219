// fused_bwd.cu -- fused main + index backward of MSA: the orchestration
// around the two tensor-core kernels, and the per-slot combines.
//
// "Sparse Attention · Part II", section 3.2: the loss is the task loss (here
// sum(dO . O)) plus the KL alignment loss; the teacher is detached and the
// selection carries no gradient, so the main branch's gradients come from dO
// alone and the index branch's from the KL alone.  With Pt the teacher and
// Ps = softmax(s) the student on the selected set the KL expands to
//     dKL/ds_j = Ps_j - Pt_j       (sum_j Pt_j = 1)
// which needs only the forward's per-head lse (for Pt) and the KL pass's
// lse_idx (for Ps), both recomputed per tile from the logits.
//
// Layout: key-major over the inverse index (per (b, group r, block c), the
// queries that selected c).  bwd_main_tc.cu gives dK, dV and the dQ partial
// rows; index_teacher_tc.cu the dq_idx partial rows, each group's dK_idx share
// and the KL loss terms; the combines below sum a row's partials (one per
// selected block) in a fixed order, so the gradients are reproducible.
#include "msa_internal.h"

namespace msa {
namespace {

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

}  // namespace

cudaError_t launch_bwd_combine(const Problem &p, const int32_t *sel, const bf16 *part, bf16 *out, int H, int Gh,
                               int width, cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Nq * H;
    {
        TimedLaunch timed_("bwd_combine_kernel", s);
        if (width == 128) bwd_combine_kernel<128><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, part, out, H, Gh);
        else bwd_combine_kernel<64><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, part, out, H, Gh);
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
    if (!bwd_tc(p)) return cudaErrorInvalidValue;
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
    // main branch: dK, dV and the dQ partial rows
    if ((e = launch_bwd_main_tc(p, q, k, v, d_o, lse, w, dk, dv, st, s)) != cudaSuccess) return e;
    // index branch: the teacher rebuilt from its own logit tiles next to the index
    // scores; dq_idx partial rows, each group's dK_idx share and the KL loss terms
    if ((e = launch_index_teacher_tc(p, q, k, q_idx, k_idx, lse, lse_idx, kl_coef, w.bucket_off, w.bucket_q, w.klt,
                                     w.dqi_part, w.dki_acc, st, s)) != cudaSuccess)
        return e;
    if (w.klt && (e = launch_kl_rows_combine(p, sel, lse_idx, w.klt, w.kl_rows, s)) != cudaSuccess) return e;
    if ((e = launch_bwd_combine(p, sel, w.dq_part, dq, p.Hq, p.G, p.d, s)) != cudaSuccess) return e;
    if ((e = launch_bwd_combine(p, sel, w.dqi_part, dq_idx, p.Hkv, 1, p.d_idx, s)) != cudaSuccess) return e;
    return launch_dki_group_sum(p, w.dki_acc, dk_idx, s);
}

}  // namespace msa
