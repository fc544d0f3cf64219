// index_proj.cu -- the index projections of MSA and their weight gradient,
// on the tcgen05 tensor cores.
//
// "Sparse Attention · Part II", section 3.2, the detachment equation: the
// index queries and keys are linear maps of the DETACHED hidden states,
//   Q_idx = stopgrad(X) W_q^idx,   K_idx = stopgrad(X) W_k^idx,
// so the KL loss trains W_q^idx and W_k^idx and sends nothing into X:
//   dW_q^idx = X^T dQ_idx,   dW_k^idx = X^T dK_idx   (no dX).
// X [T, Dm] (T = B*N tokens), W_q^idx [Dm, Hkv*d_idx] (group r's index query
// in columns r*d_idx ..), W_k^idx [Dm, d_idx], row-major bf16.  The outputs
// q_idx [T, Hkv, d_idx] and k_idx [T, d_idx] are bf16 (the layouts the index
// branch reads); the weight gradients fp32.
//
// One GEMM kernel for both: a CTA computes a 128 x BN tile (BN = d_idx: one
// group's index-query columns, or the index-key columns), K in 64-wide
// blocks through a TMA ring, the accumulator in TMEM.  Forward: A = X
// (K-major), B = the weight (MN-major: its rows are K).  Weight gradient:
// A = X^T (X read MN-major: its rows are K = tokens), B = dQ_idx or dK_idx
// (MN-major); the token range is split over several CTAs when the tiles
// alone cannot fill the GPU, each writing an fp32 partial that a second
// kernel sums in split order (deterministic; no atomics).
//
// Roles: warp 0 issues the TMA loads, warp 1 owns TMEM and issues the MMAs,
// warps 2..5 drain the accumulator (one output row per thread).
#include <algorithm>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kSt = 3;
constexpr int kThreads = 192;
constexpr int SUB = BM * 128;                  // [128 rows][64 bf16] or two [64 rows][64 bf16] halves
constexpr int STAGE = 2 * SUB;                 // A (16 KB) + B (up to 16 KB)
constexpr int OFF_BAR = kSt * STAGE;
constexpr int ALLOC = OFF_BAR + 256 + 1024;

template <int BN, bool kGradW>
__global__ void __launch_bounds__(kThreads, 1)
index_proj_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_bq,
                  const __grid_constant__ CUtensorMap tmap_bk, int M, int Kdim, int ntq, int kb_per_split,
                  bf16 *__restrict__ outq, bf16 *__restrict__ outk, float *__restrict__ partial, long long nout,
                  DeviceStatus *st)
{
    // tile (m, n): n < ntq is group n's index-query columns, n == ntq the index-key columns
    const int mt = blockIdx.x, nt = blockIdx.y, split = blockIdx.z;
    const int m0 = mt * BM;
    const int nkb = (Kdim + BK - 1) / BK;
    const int kb0 = split * kb_per_split, kb1 = min(nkb, kb0 + kb_per_split);
    const bool is_k = nt == ntq;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + kSt, *acc_full = bars + 2 * kSt;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kSt + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < kSt; ++a) {
            tc::mbar_init(&full[a], 1);
            tc::mbar_init(&empty[a], 1);
        }
        tc::mbar_init(acc_full, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, BN);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    constexpr int A_BYTES = BM * BK * 2, B_BYTES = BK * BN * 2;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const CUtensorMap *tb = is_k ? &tmap_bk : &tmap_bq;
            const int bcol = is_k ? 0 : nt * BN;
            for (int kb = kb0; kb < kb1; ++kb) {
                const int it = kb - kb0, s = it % kSt;
                if (!tc::mbar_wait(&empty[s], ((uint32_t)(it / kSt) & 1u) ^ 1u, st, 161, abort_flag)) break;
                uint8_t *sa = sm + s * STAGE, *sb = sa + SUB;
                tc::mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
                if constexpr (!kGradW) {
                    // X rows m0.., K columns kb*64..: one [128 rows][64] box
                    tc::tma_load_3d(sa, &tmap_a, &full[s], kb * BK, m0, 0);
                } else {
                    // X rows (tokens) kb*64.., columns (Dm) m0.. and m0+64..: two [64][64] boxes
                    tc::tma_load_3d(sa, &tmap_a, &full[s], m0, kb * BK, 0);
                    tc::tma_load_3d(sa + SUB / 2, &tmap_a, &full[s], m0 + 64, kb * BK, 0);
                }
                // B rows (K) kb*64.., columns bcol..: BN/64 boxes of [64 rows][64]
#pragma unroll
                for (int h = 0; h < BN / 64; ++h) tc::tma_load_3d(sb + h * (SUB / 2), tb, &full[s], bcol + 64 * h, kb * BK, 0);
            }
        }
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer (warp-uniform; one
            // elect.sync lane issues)
            constexpr uint32_t I = tc::idesc_bf16(BM, BN) | tc::kBMajorMN | (kGradW ? tc::kAMajorMN : 0u);
            bool ok = true;
            for (int kb = kb0; ok && kb < kb1; ++kb) {
                const int it = kb - kb0, s = it % kSt;
                if (!tc::mbar_wait_warp(&full[s], (uint32_t)(it / kSt) & 1u, st, 162, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t sa = smem_u32(sm + s * STAGE), sb = sa + SUB;
                const uint64_t dA = kGradW ? tc::sdesc_sw128(sa, SUB / 2, 1024) : tc::sdesc_k128(sa);
                const uint64_t dB = tc::sdesc_sw128(sb, SUB / 2, 1024);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks)
                        tc::mma_bf16(tmem, tc::desc_adv(dA, kGradW ? ks * 2048 : ks * 32), tc::desc_adv(dB, ks * 2048),
                                     I, it > 0 || ks > 0);
                    tc::mma_commit(&empty[s]);
                }
                __syncwarp();
            }
            if (tc::elect_one()) tc::mma_commit(acc_full);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ epilogue: row m0 + 32*(warp%4) + lane
        const int qd = warp & 3;
        const int row = m0 + qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        bool ok = tc::mbar_wait(acc_full, 0, st, 163, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        if (ok) {
#pragma unroll
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                if (kb1 > kb0) {
                    tc::tmem_ld32_nowait(tmem + lane_base + c, v);
                    tc::tmem_wait32(v);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = 0u;
                }
                if (row < M) {
                    if constexpr (!kGradW) {
                        bf16 *dst = is_k ? outk + (long long)row * BN + c : outq + (long long)row * ntq * BN + nt * BN + c;
#pragma unroll
                        for (int x = 0; x < 32; x += 8)
                            *reinterpret_cast<uint4 *>(dst + x) = make_uint4(
                                pack_bf16(__uint_as_float(v[x]), __uint_as_float(v[x + 1])),
                                pack_bf16(__uint_as_float(v[x + 2]), __uint_as_float(v[x + 3])),
                                pack_bf16(__uint_as_float(v[x + 4]), __uint_as_float(v[x + 5])),
                                pack_bf16(__uint_as_float(v[x + 6]), __uint_as_float(v[x + 7])));
                    } else {
                        // fp32 partial [split][M][nout]: the query-weight columns, then the key-weight ones
                        float *dst = partial + ((long long)split * M + row) * nout + (long long)nt * BN + c;
#pragma unroll
                        for (int x = 0; x < 32; x += 4)
                            *reinterpret_cast<float4 *>(dst + x) =
                                make_float4(__uint_as_float(v[x]), __uint_as_float(v[x + 1]), __uint_as_float(v[x + 2]),
                                            __uint_as_float(v[x + 3]));
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, BN);
    }
}

// dWq / dWk from the splits' partials, summed in split order
__global__ void __launch_bounds__(256) proj_split_sum_kernel(const float *__restrict__ partial, int splits, int M,
                                                             long long nout, long long nq, float *__restrict__ dwq,
                                                             float *__restrict__ dwk)
{
    const long long n = (long long)M * nout;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x) {
        float a = 0.f;
        for (int sp = 0; sp < splits; ++sp) a += partial[(long long)sp * n + x];
        const long long row = x / nout, col = x % nout;
        if (col < nq) dwq[row * nq + col] = a;
        else dwk[row * (nout - nq) + (col - nq)] = a;
    }
}

// 2-D bf16 tensor map {cols, rows} with a {64, box_rows} box
cudaError_t tmap_2d(CUtensorMap *map, const void *base, long long cols, long long rows, unsigned box_rows)
{
    return make_tmap_bf16_3d(map, base, (unsigned long long)cols, (unsigned long long)rows, 1,
                             (unsigned long long)cols * 2, (unsigned long long)cols * rows * 2, 64, box_rows);
}

template <int BN, bool kGradW>
cudaError_t launch_t(const ProjProblem &pp, const bf16 *a, const bf16 *bq, const bf16 *bk, bf16 *outq, bf16 *outk,
                     float *partial, int splits, DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(index_proj_kernel<BN, kGradW>, cudaFuncAttributeMaxDynamicSharedMemorySize, ALLOC);
    if (e != cudaSuccess) return e;
    const long long nq = (long long)pp.Hkv * pp.d_idx;
    CUtensorMap ta, tbq, tbk;
    // A: X [T][Dm]; B: the weights [Dm][cols] (forward) or dQ_idx / dK_idx [T][cols] (weight gradient)
    if ((e = tmap_2d(&ta, a, pp.Dm, pp.T, kGradW ? 64 : BM)) != cudaSuccess) return e;
    const long long brows = kGradW ? pp.T : pp.Dm;
    if ((e = tmap_2d(&tbq, bq, nq, brows, 64)) != cudaSuccess) return e;
    if ((e = tmap_2d(&tbk, bk, pp.d_idx, brows, 64)) != cudaSuccess) return e;
    const int M = kGradW ? pp.Dm : pp.T;
    const int Kdim = kGradW ? pp.T : pp.Dm;
    const int nkb = (Kdim + BK - 1) / BK;
    const int kps = (nkb + splits - 1) / splits;
    const dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)(pp.Hkv + 1), (unsigned)splits);
    {
        TimedLaunch timed_(kGradW ? "index_proj_dw_kernel" : "index_proj_fwd_kernel", s);
        index_proj_kernel<BN, kGradW><<<grid, kThreads, ALLOC, s>>>(ta, tbq, tbk, M, Kdim, pp.Hkv, kps, outq, outk,
                                                                    partial, nq + pp.d_idx, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

int index_proj_splits(const ProjProblem &pp)
{
    // the weight gradient's tiles alone: ceil(Dm/128) x (Hkv + 1); split the token
    // range until about two CTAs per SM, keeping at least 8 K-blocks per split
    const int tiles = ((pp.Dm + BM - 1) / BM) * (pp.Hkv + 1);
    const int nkb = (pp.T + BK - 1) / BK;
    int splits = (2 * pp.num_sms + tiles - 1) / tiles;
    splits = std::min(splits, std::max(1, nkb / 8));
    return std::max(1, splits);
}

size_t index_proj_partial_floats(const ProjProblem &pp)
{
    return (size_t)index_proj_splits(pp) * pp.Dm * ((size_t)pp.Hkv * pp.d_idx + pp.d_idx);
}

cudaError_t launch_index_proj_fwd(const ProjProblem &pp, const bf16 *x, const bf16 *wq, const bf16 *wk, bf16 *q_idx,
                                  bf16 *k_idx, DeviceStatus *st, cudaStream_t s)
{
    return pp.d_idx == 128 ? launch_t<128, false>(pp, x, wq, wk, q_idx, k_idx, nullptr, 1, st, s)
                           : launch_t<64, false>(pp, x, wq, wk, q_idx, k_idx, nullptr, 1, st, s);
}

cudaError_t launch_index_proj_dw(const ProjProblem &pp, const bf16 *x, const bf16 *dq_idx, const bf16 *dk_idx,
                                 float *dwq, float *dwk, float *partial, DeviceStatus *st, cudaStream_t s)
{
    // the tiles write [split][Dm][Hkv*d_idx + d_idx] partials; the sum kernel adds
    // the splits in order and separates the query- and key-weight columns
    const int splits = index_proj_splits(pp);
    const long long nq = (long long)pp.Hkv * pp.d_idx, nout = nq + pp.d_idx;
    cudaError_t e = pp.d_idx == 128 ? launch_t<128, true>(pp, x, dq_idx, dk_idx, nullptr, nullptr, partial, splits, st, s)
                                    : launch_t<64, true>(pp, x, dq_idx, dk_idx, nullptr, nullptr, partial, splits, st, s);
    if (e != cudaSuccess) return e;
    {
        TimedLaunch timed_("proj_split_sum_kernel", s);
        proj_split_sum_kernel<<<4 * pp.num_sms, 256, 0, s>>>(partial, splits, pp.Dm, nout, nq, dwq, dwk);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
