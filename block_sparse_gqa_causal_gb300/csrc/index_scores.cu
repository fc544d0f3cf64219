// index_scores.cu -- index branch of MSA: token scores and block max-pool.
//
// "Sparse Attention · Part II", section 3.2: per query and GQA group, the
// group's index query is dotted with the index key head shared by all
// groups over every causally visible token, and each 128-token block is
// scored by its largest visible token score.  The N x N token scores never
// leave the SM: each CTA reduces a 128 x 128 score tile to 128 block scores.
//
// Rows of the GEMM are "flat" (query, group) rows rho = i*Hkv + r of one
// batch entry (q_idx [B, Nq, Hkv, d_idx] is exactly that matrix), so a tile
// mixes the groups of a few queries and all of them share the K_idx block
// in shared memory.  Columns are the 128 keys of one block.  A CTA owns 128
// rows and walks the key blocks its rows can see (optionally a slice of
// them, when few row tiles exist, e.g. in decode).
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kRows = 128;
constexpr int kThreads = 256;

template <int DI>
struct IdxTile {
    static constexpr int CH = DI / 8;               // 16-byte chunks per row
    static constexpr int BYTES = kRows * DI * 2;    // one [128][DI] bf16 tile
    static constexpr int SMEM = 3 * BYTES;          // Q tile + 2 K_idx stages
};

// XOR-swizzled byte offset of 16-byte chunk `ch` of row `row` (kills the
// 8-way bank conflicts of ldmatrix on 128/256-byte rows).
template <int DI>
__device__ __forceinline__ int swz(int row, int ch)
{
    return row * (DI * 2) + ((ch ^ (row & 7)) << 4);
}

template <int DI>
__global__ void __launch_bounds__(kThreads, 2)
index_scores_kernel(Problem p, const bf16 *__restrict__ q_idx, const bf16 *__restrict__ k_idx,
                    float *__restrict__ bs, int splits)
{
    using T = IdxTile<DI>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sK = smem + T::BYTES;

    const int b = blockIdx.z;
    const int rows_total = p.Nq * p.Hkv;
    const int tile = gridDim.x - 1 - blockIdx.x;   // long (late) tiles first
    const int rho0 = tile * kRows;
    const int rho_last = min(rho0 + kRows - 1, rows_total - 1);
    const long long pos_first = (long long)p.q_offset + rho0 / p.Hkv;
    const long long pos_last = (long long)p.q_offset + rho_last / p.Hkv;
    const int c_all = (int)(min(pos_last, (long long)p.Nk - 1) / 128) + 1;
    const int span = (c_all + splits - 1) / splits;
    const int c_begin = blockIdx.y * span;
    const int c_end = min(c_all, c_begin + span);
    if (c_begin >= c_end) return;

    const bf16 *qb = q_idx + (long long)b * rows_total * DI;
    const bf16 *kb = k_idx + (long long)b * p.kv_rows * DI;
    const int tid = threadIdx.x;

    for (int idx = tid; idx < kRows * T::CH; idx += kThreads) {
        const int row = idx / T::CH, ch = idx % T::CH;
        const int rho = rho0 + row;
        const bool ok = rho < rows_total;
        cp_async16_zfill(sQ + swz<DI>(row, ch), qb + (long long)(ok ? rho : 0) * DI + ch * 8, ok);
    }
    auto load_k = [&](int c, int stage) {
        uint8_t *dst = sK + stage * T::BYTES;
        for (int idx = tid; idx < kRows * T::CH; idx += kThreads) {
            const int row = idx / T::CH, ch = idx % T::CH;
            const long long j = (long long)c * 128 + row;
            const bool ok = j < p.Nk;
            cp_async16_zfill(dst + swz<DI>(row, ch), kb + (ok ? j : 0) * DI + ch * 8, ok);
        }
    };
    load_k(c_begin, 0);
    cp_async_commit();

    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rA = warp * 16 + g, rB = rA + 8;
    const int rhoA = rho0 + rA, rhoB = rho0 + rB;
    const long long posA = (long long)p.q_offset + rhoA / p.Hkv;
    const long long posB = (long long)p.q_offset + rhoB / p.Hkv;
    const bool validA = rhoA < rows_total, validB = rhoB < rows_total;
    float *outA = bs + ((long long)b * rows_total + rhoA) * p.nb;
    float *outB = bs + ((long long)b * rows_total + rhoB) * p.nb;

    uint32_t af[DI / 16][4];
    for (int c = c_begin; c < c_end; ++c) {
        const int stage = (c - c_begin) & 1;
        if (c + 1 < c_end) load_k(c + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (c == c_begin) {
#pragma unroll
            for (int ks = 0; ks < DI / 16; ++ks)
                ldsm_x4(af[ks][0], af[ks][1], af[ks][2], af[ks][3],
                        sQ + swz<DI>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)));
        }
        const uint8_t *sk = sK + stage * T::BYTES;
        const long long j0 = (long long)c * 128;
        const bool full = (j0 + 127 <= pos_first) && (j0 + 128 <= p.Nk);
        float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float acc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < DI / 16; ++ks) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int key = half * 64 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    uint32_t b0[2], b1[2];
                    ldsm_x4(b0[0], b0[1], b1[0], b1[1], sk + swz<DI>(key, ks * 2 + ((lane >> 3) & 1)));
                    mma16816(acc[np * 2], af[ks], b0);
                    mma16816(acc[np * 2 + 1], af[ks], b1);
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float vA = acc[n][e], vB = acc[n][2 + e];
                    if (!full) {
                        const long long j = j0 + half * 64 + n * 8 + 2 * t + e;
                        if (j > posA || j >= p.Nk) vA = -INFINITY;
                        if (j > posB || j >= p.Nk) vB = -INFINITY;
                    }
                    mA = fmaxf(mA, vA);
                    mB = fmaxf(mB, vB);
                }
            }
        }
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
        if (t == 0) {
            // scale after the max: a positive scale commutes with max
            if (validA && j0 <= posA) outA[c] = mA * p.scale_idx;
            if (validB && j0 <= posB) outB[c] = mB * p.scale_idx;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_index_scores(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs,
                                DeviceStatus *, cudaStream_t s)
{
    const int rows_total = p.Nq * p.Hkv;
    const int tiles = (rows_total + kRows - 1) / kRows;
    int splits = 1;
    const long long ctas = (long long)tiles * p.B;
    if (ctas < 2LL * p.num_sms) splits = (int)min((long long)p.nb, (2LL * p.num_sms + ctas - 1) / ctas);
    dim3 grid(tiles, splits, p.B);
    if (p.d_idx == 128) {
        const int sm = IdxTile<128>::SMEM;
        cudaFuncSetAttribute(index_scores_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        index_scores_kernel<128><<<grid, kThreads, sm, s>>>(p, q_idx, k_idx, bs, splits);
        note_launch();
    } else {
        const int sm = IdxTile<64>::SMEM;
        cudaFuncSetAttribute(index_scores_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        index_scores_kernel<64><<<grid, kThreads, sm, s>>>(p, q_idx, k_idx, bs, splits);
        note_launch();
    }
    return cudaGetLastError();
}

}  // namespace msa
