// fused_bwd_tc.cu -- fused main + index backward of MSA on the tcgen05 tensor
// cores (d = d_idx = 128).
//
// Same mathematics and key-major layout as fused_bwd.cu ("Sparse Attention ·
// Part II", section 3.2: detached teacher, no gradient through selection; the
// KL expansion dKL/ds_j = Ps_j - Pt_j from the MSA kernel write-up): one CTA
// owns one 128-token key block of one (b, group) and walks the queries that
// selected it, 32 (query, head) rows per chunk.  All GEMMs run on tcgen05
// with fp32 accumulators in TMEM (512 columns):
//   S^T  = K Q^T,  dP^T = V dO^T,  s^T = K_idx q_idx^T         (per chunk)
//   dV  += P^T dO,  dK += dS^T Q,  dK_idx += dsig^T q_idx      (whole CTA)
//   dQ^T = K^T dS^T,  dQ_idx^T = K_idx^T dsig^T               (per chunk)
// Operands are bf16 in 128-byte-swizzled shared memory; the same Q / dO /
// q_idx / K tiles serve as K-major operands in one GEMM and MN-major in
// another, so nothing is transposed by hand.  The epilogue warps (one key
// row per thread) turn S^T, dP^T, s^T into P^T, dS^T and dsig^T (bf16, back
// to shared memory), and send dQ^T, dQ_idx^T to fp32 reductions.
//
// Roles: warp 0 gathers rows with cp.async (+ mbarrier arrivals), warp 1
// allocates TMEM and issues every MMA from one thread, warps 2..5 are the
// epilogue.  Every wait is bounded and reports through the status word.
#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int D = 128;
constexpr int DI = 128;
constexpr int kKeys = 128;
constexpr int kNQ = 32;          // (query, head) rows per chunk
constexpr int kNQI = 16;         // query slots per chunk
constexpr int kStages = 2;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (2 + kEpiWarps);

constexpr int SUB = kKeys * 128;                 // [128 rows][64 bf16] swizzled tile
constexpr int OFF_K = 0;                         // K, V, K_idx: two d-halves each
constexpr int OFF_V = OFF_K + 2 * SUB;
constexpr int OFF_KI = OFF_V + 2 * SUB;
constexpr int OFF_P = OFF_KI + 2 * SUB;          // P^T    [128 keys][64] (32 used)
constexpr int OFF_DS = OFF_P + SUB;              // dS^T
constexpr int OFF_SIG = OFF_DS + SUB;            // dsig^T [128 keys][64] (16 used)
constexpr int OFF_STG = OFF_SIG + SUB;
constexpr int STG_Q = 0;                         // Q:     2 x [32][64] (4 KB each)
constexpr int STG_DO = 8192;                     // dO:    2 x [32][64]
constexpr int STG_QI = 16384;                    // q_idx: 2 x [16][64] (2 KB each)
constexpr int STG_ROWS = 20480;
constexpr int STG_BYTES = 21504;
constexpr int OFF_RED = OFF_STG + kStages * STG_BYTES;   // fp32 staging [kNQ + kNQI][128] for the reductions
constexpr int OFF_BAR = OFF_RED + (kNQ + kNQI) * D * 4;
constexpr int SMEM_ALLOC = OFF_BAR + 512 + 1024;

// TMEM columns
constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_DKI = 256, TM_S = 384, TM_DP = 416, TM_SI = 448, TM_DQ = 464,
                   TM_DQI = 496;

struct StageRows {
    float lse2[kNQ];    // LSE * log2(e) of each (query, head) row; +inf when unused
    float dd[kNQ];      // rowsum(dO * O)
    float lsei2[kNQI];  // lse_idx * log2(e) of each query; +inf when unused
    int pos[kNQI];      // position of each query; -1 when unused
    int qi[kNQI];       // query index
    int nq;             // queries in this chunk
};

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// qis[qq] for a runtime qq without spilling the array to local memory
template <int N>
__device__ __forceinline__ int qsel(const int (&qis)[N], int qq)
{
    int v = qis[0];
#pragma unroll
    for (int u = 1; u < N; ++u)
        if (qq == u) v = qis[u];
    return v;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
fused_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_do,
                    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q,
                    const bf16 *__restrict__ d_o, const float *__restrict__ lse, const bf16 *__restrict__ q_idx,
                    const float *__restrict__ lse_idx, float kl_coef,
                    const float *__restrict__ Dg, const int32_t *__restrict__ bucket_off,
                    const int32_t *__restrict__ bucket_q, bf16 *__restrict__ dk, bf16 *__restrict__ dv,
                    float *__restrict__ dq_acc, float *__restrict__ dqi_acc, float *__restrict__ dki_acc,
                    DeviceStatus *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + kStages;
    uint64_t *kv_full = bars + 2 * kStages, *s_full = kv_full + 1, *tm_free = s_full + 1, *p_full = tm_free + 1;
    uint64_t *p_free = p_full + 1, *dq_full = p_free + 1, *dq_free = dq_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(dq_free + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // x = group, y = key block: the heavy early blocks of every group start first
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    constexpr int QC = (kNQ / G < kNQI) ? kNQ / G : kNQI;   // queries per chunk
    const long long j0 = (long long)c * kKeys;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    const int nch = (qend - qbeg + QC - 1) / QC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // 32 cp.async arrivals + 32 row-data arrivals (+ lane 0's expect_tx
            // arrival for the TMA-loaded Q and dO rows when G == 8)
            tc::mbar_init(&full[s], G == 8 ? 65 : 64);
            tc::mbar_init(&empty[s], 1 + kEpiWarps);        // grads MMAs done + epilogue has read the rows
        }
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(s_full, 1);
        tc::mbar_init(tm_free, kEpiWarps);
        tc::mbar_init(p_full, kEpiWarps);
        tc::mbar_init(p_free, 1);
        tc::mbar_init(dq_full, 1);
        tc::mbar_init(dq_free, kEpiWarps);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ producer
        // K, V and K_idx tiles of this (b, group, block) by TMA; rows past Nk read as zeros
        if (lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::prefetch_tmap(&tmap_do);
            tc::mbar_arrive_expect_tx(kv_full, 6 * SUB);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc::tma_load_4d(sm + OFF_K + h * SUB, &tmap_k, kv_full, h * 64, r, (int)j0, b);
                tc::tma_load_4d(sm + OFF_V + h * SUB, &tmap_v, kv_full, h * 64, r, (int)j0, b);
                tc::tma_load_3d(sm + OFF_KI + h * SUB, &tmap_ki, kv_full, h * 64, (int)j0, b);
            }
        }
        if constexpr (QC < kNQI) {
            // q_idx rows QC..kNQI-1 of both stages are never loaded: zero them once
            for (int x = lane; x < kStages * 2 * (kNQI - QC) * 8; x += 32) {
                const int st_ = x / (2 * (kNQI - QC) * 8), y = x % (2 * (kNQI - QC) * 8);
                const int h = y / ((kNQI - QC) * 8), row = QC + (y / 8) % (kNQI - QC), ch = y % 8;
                *reinterpret_cast<uint4 *>(sm + OFF_STG + st_ * STG_BYTES + STG_QI + h * (kNQI * 128) + swz(row, ch)) =
                    make_uint4(0, 0, 0, 0);
            }
        }
        // entries of chunk m are fetched during chunk m-1; the per-row values
        // that depend on them are loaded before waiting for a free stage
        int ent = lane < min(QC, qend - qbeg) ? __ldg(bucket_q + qbeg + lane) : 0;
        for (int m = 0; m < nch; ++m) {
            const int s = m & 1;
            const int q0 = qbeg + m * QC;
            const int nq = min(QC, qend - q0);
            const int ent_next = (m + 1 < nch && lane < min(QC, qend - q0 - QC)) ? __ldg(bucket_q + q0 + QC + lane) : 0;
            // row values: lane = (query, head) row for lse2 / dd, lane = query for lsei2
            const int my_q = lane < kNQI && lane < nq ? entry_row(ent) : 0;
            const int rq = lane / G, rg = lane % G;
            const bool rok = lane < QC * G && rq < nq;
            const int ri = __shfl_sync(0xffffffffu, entry_row(ent), rq < 32 ? rq : 0);
            const long long hi = ((long long)b * p.Hq + r * G + rg) * p.Nq + ri;
            const float v_lse2 = rok ? __ldg(lse + hi) * kLog2e : INFINITY;
            const float v_dd = rok ? __ldg(Dg + hi) : 0.f;
            const bool qok = lane < kNQI && lane < nq;
            const float v_lsei2 = qok ? __ldg(lse_idx + ((long long)b * p.Hkv + r) * p.Nq + my_q) * kLog2e : INFINITY;
            if (!tc::mbar_wait(&empty[s], ((uint32_t)(m >> 1) & 1u) ^ 1u, st, 21, abort_flag)) break;
            uint8_t *stg = sm + OFF_STG + s * STG_BYTES;
            StageRows *rows = reinterpret_cast<StageRows *>(stg + STG_ROWS);
            if (lane < kNQI) {
                rows->qi[lane] = my_q;
                rows->lsei2[lane] = v_lsei2;
                rows->pos[lane] = qok ? my_q : -1;        // training layout: q_offset == 0
            }
            rows->lse2[lane] = v_lse2;
            rows->dd[lane] = v_dd;
            if (lane == 0) rows->nq = nq;
            __syncwarp();
            if constexpr (G == 8) {
                // Q and dO: one TMA box {64 features, 8 heads} per query and half
                // (1024 bytes, on a swizzle-pattern boundary); padding slots read
                // rows past the end of the tensors (zero fill)
                if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * kNQ * D * 2);
                __syncwarp();
                if (lane < 2 * QC) {
                    const int qq = lane >> 1, h = lane & 1;
                    const int z = qq < nq ? b * p.Nq + rows->qi[qq] : p.B * p.Nq;
                    tc::tma_load_3d(stg + STG_Q + h * (kNQ * 128) + qq * 1024, &tmap_q, &full[s], h * 64, r * G, z);
                    tc::tma_load_3d(stg + STG_DO + h * (kNQ * 128) + qq * 1024, &tmap_do, &full[s], h * 64, r * G, z);
                }
            } else {
                // Q and dO rows (row rho = qq*G + g): 16 lanes per 256-byte row, 2 rows per step
#pragma unroll 4
                for (int it = 0; it < kNQ / 2; ++it) {
                    const int rho = it * 2 + (lane >> 4), ch = lane & 15;
                    const int qq = rho / G, g = rho % G;
                    const bool ok = rho < QC * G && qq < nq;
                    const int i = rows->qi[qq < kNQI ? qq : 0];
                    const long long off = (((long long)b * p.Nq + i) * p.Hq + (long long)r * G + g) * D + ch * 8;
                    const int o = (ch >> 3) * (kNQ * 128) + swz(rho, ch & 7);
                    cp_async16_zfill(stg + STG_Q + o, q + off, ok);
                    cp_async16_zfill(stg + STG_DO + o, d_o + off, ok);
                }
            }
            // q_idx rows of the chunk's queries (zero for padding slots)
#pragma unroll
            for (int it = 0; it < (QC * 16 + 31) / 32; ++it) {
                const int row = it * 2 + (lane >> 4), ch = lane & 15;
                if (row < QC) {
                    const bool ok = row < nq;
                    cp_async16_zfill(stg + STG_QI + (ch >> 3) * (kNQI * 128) + swz(row, ch & 7),
                                     q_idx + (((long long)b * p.Nq + rows->qi[row]) * p.Hkv + r) * DI + ch * 8, ok);
                }
            }
            cp_async_arrive_noinc(&full[s]);
            tc::mbar_arrive(&full[s]);
            ent = ent_next;
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t I_S = tc::idesc_bf16(128, kNQ);
            constexpr uint32_t I_SI = tc::idesc_bf16(128, kNQI);
            constexpr uint32_t I_DKV = tc::idesc_bf16(128, 128) | tc::kBMajorMN;
            constexpr uint32_t I_DQ = tc::idesc_bf16(128, kNQ) | tc::kAMajorMN | tc::kBMajorMN;
            constexpr uint32_t I_DQI = tc::idesc_bf16(128, kNQI) | tc::kAMajorMN | tc::kBMajorMN;
            const uint32_t aK = smem_u32(sm + OFF_K), aV = smem_u32(sm + OFF_V), aKI = smem_u32(sm + OFF_KI);
            const uint32_t aP = smem_u32(sm + OFF_P), aDS = smem_u32(sm + OFF_DS), aSIG = smem_u32(sm + OFF_SIG);
            auto issue_scores = [&](int n) {
                const uint32_t stg = smem_u32(sm + OFF_STG + (n & 1) * STG_BYTES);
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                    tc::mma_bf16(tmem + TM_S, tc::sdesc_k128(aK + h * SUB + ko),
                                 tc::sdesc_k128(stg + STG_Q + h * (kNQ * 128) + ko), I_S, ks > 0);
                    tc::mma_bf16(tmem + TM_DP, tc::sdesc_k128(aV + h * SUB + ko),
                                 tc::sdesc_k128(stg + STG_DO + h * (kNQ * 128) + ko), I_S, ks > 0);
                    tc::mma_bf16(tmem + TM_SI, tc::sdesc_k128(aKI + h * SUB + ko),
                                 tc::sdesc_k128(stg + STG_QI + h * (kNQI * 128) + ko), I_SI, ks > 0);
                }
                tc::mma_commit(s_full);
            };
            auto issue_grads = [&](int n) {
                const uint32_t stg = smem_u32(sm + OFF_STG + (n & 1) * STG_BYTES);
                const bool first = n == 0;
                // dV += P^T dO, dK += dS^T Q : K = 32 rows of the chunk (2 steps)
                for (int ks = 0; ks < kNQ / 16; ++ks) {
                    const uint64_t bdo = tc::sdesc_sw128(stg + STG_DO + ks * 2048, kNQ * 128, 1024);
                    const uint64_t bq = tc::sdesc_sw128(stg + STG_Q + ks * 2048, kNQ * 128, 1024);
                    tc::mma_bf16(tmem + TM_DV, tc::sdesc_k128(aP + ks * 32), bdo, I_DKV, !(first && ks == 0));
                    tc::mma_bf16(tmem + TM_DK, tc::sdesc_k128(aDS + ks * 32), bq, I_DKV, !(first && ks == 0));
                }
                // dK_idx += dsig^T q_idx : K = 16 query slots (1 step)
                tc::mma_bf16(tmem + TM_DKI, tc::sdesc_k128(aSIG), tc::sdesc_sw128(stg + STG_QI, kNQI * 128, 1024),
                             I_DKV, !first);
                // dQ^T = K^T dS^T, dQ_idx^T = K_idx^T dsig^T : K = 128 keys (8 steps)
                for (int ks = 0; ks < kKeys / 16; ++ks) {
                    tc::mma_bf16(tmem + TM_DQ, tc::sdesc_sw128(aK + ks * 2048, SUB, 1024),
                                 tc::sdesc_sw128(aDS + ks * 2048, SUB, 1024), I_DQ, ks > 0);
                    tc::mma_bf16(tmem + TM_DQI, tc::sdesc_sw128(aKI + ks * 2048, SUB, 1024),
                                 tc::sdesc_sw128(aSIG + ks * 2048, SUB, 1024), I_DQI, ks > 0);
                }
                tc::mma_commit(&empty[n & 1]);
                tc::mma_commit(dq_full);
                tc::mma_commit(p_free);
            };
            bool ok = tc::mbar_wait(kv_full, 0, st, 22, abort_flag);
            int issued = 0;
            if (ok && nch > 0) {
                ok = tc::mbar_wait(&full[0], 0, st, 23, abort_flag);
                if (ok) {
                    tc::fence_proxy_async();
                    tc::fence_after_sync();
                    issue_scores(0);
                }
            }
            for (int n = 0; ok && n < nch; ++n) {
                if (n + 1 < nch) {
                    if (!tc::mbar_wait(&full[(n + 1) & 1], (uint32_t)((n + 1) >> 1) & 1u, st, 24, abort_flag)) break;
                    if (!tc::mbar_wait(tm_free, (uint32_t)n & 1u, st, 25, abort_flag)) break;
                    tc::fence_proxy_async();
                    tc::fence_after_sync();
                    issue_scores(n + 1);
                }
                if (!tc::mbar_wait(p_full, (uint32_t)n & 1u, st, 26, abort_flag)) break;
                if (n > 0 && !tc::mbar_wait(dq_free, (uint32_t)(n - 1) & 1u, st, 27, abort_flag)) break;
                tc::fence_after_sync();
                issue_grads(n);
                issued = n + 1;
            }
            if (*abort_flag && issued > 0) tc::mbar_wait(dq_full, (uint32_t)(issued - 1) & 1u, nullptr, 0, nullptr);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;              // key row (S/dP/s phase) and d row (dQ phase)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const long long j = j0 + kr;
        const bool key_ok = j < p.Nk;
        const float sl2 = p.scale * kLog2e, si2 = p.scale_idx * kLog2e;
        const float coef = kl_coef / ((float)p.B * (float)p.Nq * (float)p.Hkv);
        const float invG = 1.f / (float)G;
        bool ok = true;
        for (int n = 0; ok && n < nch; ++n) {
            const uint8_t *stg = sm + OFF_STG + (n & 1) * STG_BYTES;
            const StageRows *rows = reinterpret_cast<const StageRows *>(stg + STG_ROWS);
            if (!tc::mbar_wait(&full[n & 1], (uint32_t)(n >> 1) & 1u, st, 31, abort_flag)) { ok = false; break; }
            if (!tc::mbar_wait(s_full, (uint32_t)n & 1u, st, 32, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t svr[kNQ], dpr[kNQ], sir[kNQI];
            tc::tmem_ld32_nowait(tmem + lane_base + TM_S, svr);
            tc::tmem_ld32_nowait(tmem + lane_base + TM_DP, dpr);
            tc::tmem_ld16_nowait(tmem + lane_base + TM_SI, sir);
            tc::tmem_wait32(svr);
            tc::tmem_wait32(dpr);
            tc::tmem_wait16(sir);
            const float *sv = reinterpret_cast<const float *>(svr);
            const float *dp = reinterpret_cast<const float *>(dpr);
            const float *si = reinterpret_cast<const float *>(sir);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tm_free);
            // P^T, dS^T rows (this key against the chunk's (query, head) rows)
            uint32_t pk[kNQ / 2], dk2[kNQ / 2];
            float pt[kNQI];
#pragma unroll
            for (int u = 0; u < kNQI; ++u) pt[u] = 0.f;
#pragma unroll
            for (int rho = 0; rho < kNQ; rho += 2) {
                float pr[2], dsv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int rr = rho + e;
                    const int qq = rr / G;
                    const bool vis = key_ok && qq < kNQI && j <= rows->pos[qq < kNQI ? qq : 0];
                    pr[e] = vis ? tc::ex2(sv[rr] * sl2 - rows->lse2[rr]) : 0.f;
                    dsv[e] = pr[e] * (dp[rr] - rows->dd[rr]);
                    if (qq < kNQI) pt[qq] += pr[e];
                }
                pk[rho / 2] = pack_bf16(pr[0], pr[1]);
                dk2[rho / 2] = pack_bf16(dsv[0], dsv[1]);
            }
            uint32_t sg[kNQI / 2];
#pragma unroll
            for (int u = 0; u < kNQI; u += 2) {
                float ds2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int qq = u + e;
                    const bool vis = key_ok && j <= rows->pos[qq];
                    const float ps = vis ? tc::ex2(si[qq] * si2 - rows->lsei2[qq]) : 0.f;
                    ds2[e] = vis ? coef * (ps - pt[qq] * invG) : 0.f;
                }
                sg[u / 2] = pack_bf16(ds2[0], ds2[1]);
            }
            if (n > 0 && !tc::mbar_wait(p_free, (uint32_t)(n - 1) & 1u, st, 33, abort_flag)) { ok = false; break; }
#pragma unroll
            for (int c16 = 0; c16 < kNQ / 8; ++c16) {
                *reinterpret_cast<uint4 *>(sm + OFF_P + swz(kr, c16)) =
                    make_uint4(pk[c16 * 4], pk[c16 * 4 + 1], pk[c16 * 4 + 2], pk[c16 * 4 + 3]);
                *reinterpret_cast<uint4 *>(sm + OFF_DS + swz(kr, c16)) =
                    make_uint4(dk2[c16 * 4], dk2[c16 * 4 + 1], dk2[c16 * 4 + 2], dk2[c16 * 4 + 3]);
            }
#pragma unroll
            for (int c16 = 0; c16 < kNQI / 8; ++c16)
                *reinterpret_cast<uint4 *>(sm + OFF_SIG + swz(kr, c16)) =
                    make_uint4(sg[c16 * 4], sg[c16 * 4 + 1], sg[c16 * 4 + 2], sg[c16 * 4 + 3]);
            // keep what the reduction phase needs; the stage can then be refilled
            const int nq = rows->nq;
            int qis[QC];
#pragma unroll
            for (int u = 0; u < QC; ++u) qis[u] = rows->qi[u];
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(p_full);
                tc::mbar_arrive(&empty[n & 1]);
            }
            // dQ^T, dQ_idx^T rows (this thread: feature kr)
            if (!tc::mbar_wait(dq_full, (uint32_t)n & 1u, st, 34, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t dqr[kNQ], dqir[kNQI];
            tc::tmem_ld32_nowait(tmem + lane_base + TM_DQ, dqr);
            tc::tmem_ld16_nowait(tmem + lane_base + TM_DQI, dqir);
            tc::tmem_wait32(dqr);
            tc::tmem_wait16(dqir);
            const float *dqv = reinterpret_cast<const float *>(dqr);
            const float *dqiv = reinterpret_cast<const float *>(dqir);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(dq_free);
            // transpose this warp's 32 feature rows through shared memory so each
            // reduction covers 16 contiguous bytes of one (query, head) row
            float *red = reinterpret_cast<float *>(sm + OFF_RED) + quarter * ((kNQ + kNQI) * 32);
            __syncwarp();
#pragma unroll
            for (int rr = 0; rr < kNQ; ++rr) red[rr * 32 + lane] = dqv[rr];
#pragma unroll
            for (int qq = 0; qq < kNQI; ++qq) red[(kNQ + qq) * 32 + lane] = dqiv[qq];
            __syncwarp();
            const int dbase = quarter * 32;
            for (int x = lane; x < (QC * G) * 8; x += 32) {
                const int rr = x >> 3, d4 = (x & 7) * 4;
                const int qq = rr / G, g = rr % G;
                if (qq < nq) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(red + rr * 32 + d4);
                    tc::red_add_v4(dq_acc + (((long long)b * p.Nq + qsel(qis, qq)) * p.Hq + (long long)r * G + g) * D +
                                       dbase + d4,
                                   p.scale * v4.x, p.scale * v4.y, p.scale * v4.z, p.scale * v4.w);
                }
            }
            for (int x = lane; x < nq * 8; x += 32) {
                const int qq = x >> 3, d4 = (x & 7) * 4;
                const float4 v4 = *reinterpret_cast<const float4 *>(red + (kNQ + qq) * 32 + d4);
                tc::red_add_v4(dqi_acc + (((long long)b * p.Nq + qsel(qis, qq)) * p.Hkv + r) * DI + dbase + d4,
                               p.scale_idx * v4.x, p.scale_idx * v4.y, p.scale_idx * v4.z, p.scale_idx * v4.w);
            }
            __syncwarp();
        }
        // ---- dK, dV (owned) and dK_idx (shared by the groups) of this key
        if (ok && key_ok) {
            bf16 *pk = dk + ((long long)b * p.kv_rows + j) * ((long long)p.Hkv * D) + (long long)r * D;
            bf16 *pv = dv + ((long long)b * p.kv_rows + j) * ((long long)p.Hkv * D) + (long long)r * D;
            float *pki = dki_acc + ((long long)b * p.kv_rows + j) * DI;
            if (nch == 0) {
                for (int cc = 0; cc < D; cc += 8) {
                    *reinterpret_cast<uint4 *>(pk + cc) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(pv + cc) = make_uint4(0, 0, 0, 0);
                }
            } else {
                tc::fence_after_sync();
                for (int c32 = 0; c32 < 4; ++c32) {
                    float a[32];
                    tc::tmem_ld32(tmem + lane_base + TM_DV + c32 * 32, a);
#pragma unroll
                    for (int x = 0; x < 32; x += 8)
                        *reinterpret_cast<uint4 *>(pv + c32 * 32 + x) =
                            make_uint4(pack_bf16(a[x], a[x + 1]), pack_bf16(a[x + 2], a[x + 3]),
                                       pack_bf16(a[x + 4], a[x + 5]), pack_bf16(a[x + 6], a[x + 7]));
                    tc::tmem_ld32(tmem + lane_base + TM_DK + c32 * 32, a);
#pragma unroll
                    for (int x = 0; x < 32; x += 8)
                        *reinterpret_cast<uint4 *>(pk + c32 * 32 + x) = make_uint4(
                            pack_bf16(p.scale * a[x], p.scale * a[x + 1]), pack_bf16(p.scale * a[x + 2], p.scale * a[x + 3]),
                            pack_bf16(p.scale * a[x + 4], p.scale * a[x + 5]), pack_bf16(p.scale * a[x + 6], p.scale * a[x + 7]));
                    tc::tmem_ld32(tmem + lane_base + TM_DKI + c32 * 32, a);
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        tc::red_add_v4(pki + c32 * 32 + x, p.scale_idx * a[x], p.scale_idx * a[x + 1],
                                       p.scale_idx * a[x + 2], p.scale_idx * a[x + 3]);
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

template <int G>
cudaError_t launch_g(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *d_o, const float *lse,
                     const bf16 *q_idx, const bf16 *k_idx, const float *lse_idx, float kl_coef, const BwdWork &w,
                     bf16 *dk, bf16 *dv, DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(fused_bwd_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tdo, tk, tv, tki;
    {
        const unsigned long long dq[3] = {(unsigned long long)D, (unsigned long long)p.Hq, (unsigned long long)p.B * p.Nq};
        const unsigned long long sq[2] = {D * 2ull, (unsigned long long)p.Hq * D * 2ull};
        const unsigned bq[3] = {64, (unsigned)G, 1};
        if ((e = make_tmap_bf16(&tq, q, 3, dq, sq, bq)) != cudaSuccess) return e;
        if ((e = make_tmap_bf16(&tdo, d_o, 3, dq, sq, bq)) != cudaSuccess) return e;
        // K/V as [B][Nk][Hkv][D], K_idx as [B][Nk][DI] (rows past Nk are out of bounds)
        const unsigned long long dk4[4] = {(unsigned long long)D, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                           (unsigned long long)p.B};
        const unsigned long long sk[3] = {D * 2ull, (unsigned long long)p.Hkv * D * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * D * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk4, sk, bk)) != cudaSuccess) return e;
        if ((e = make_tmap_bf16(&tv, v, 4, dk4, sk, bk)) != cudaSuccess) return e;
        const unsigned long long di[3] = {(unsigned long long)DI, (unsigned long long)p.Nk, (unsigned long long)p.B};
        const unsigned long long si[2] = {DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull};
        const unsigned bi[3] = {64, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    }
    fused_bwd_tc_kernel<G><<<dim3(p.Hkv, p.nb, p.B), kThreads, SMEM_ALLOC, s>>>(
        tq, tdo, tk, tv, tki, p, q, d_o, lse, q_idx, lse_idx, kl_coef, w.D, w.bucket_off, w.bucket_q, dk, dv,
        w.dq_acc, w.dqi_acc, w.dki_acc, st);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_bwd_tc_main(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *d_o,
                                     const float *lse, const bf16 *q_idx, const bf16 *k_idx, const float *lse_idx,
                                     float kl_coef, const BwdWork &w, bf16 *dk, bf16 *dv, DeviceStatus *st,
                                     cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_g<1>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, st, s);
    case 2: return launch_g<2>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, st, s);
    case 4: return launch_g<4>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, st, s);
    default: return launch_g<8>(p, q, k, v, d_o, lse, q_idx, k_idx, lse_idx, kl_coef, w, dk, dv, st, s);
    }
}

}  // namespace msa
