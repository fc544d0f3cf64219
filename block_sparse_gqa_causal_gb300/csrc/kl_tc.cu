// kl_tc.cu -- KL alignment loss of MSA, key-major on the tcgen05 tensor cores.
//
// "Sparse Attention · Part II", section 3.2 (the L_KL equation): for query i
// and group r over the selected token set T, with the detached teacher
// Pt_j = (1/G) sum_h exp(l_{h,j} - lse_h) and the student Ps = softmax_T(s),
//   KL = sum_j Pt_j log Pt_j - sum_j Pt_j s_j + log sum_j exp(s_j).
// Every term is a sum over T, so it splits over the selected blocks.  As in
// the key-major forward, one CTA keeps one 128-token block of K and K_idx of
// one group on chip and takes the queries that selected it 128 (query, head)
// rows at a time:
//   S^T = K Q^T   (M = 128 keys, N = 128 (query, head) columns)
//   s^T = K_idx q_idx^T   (M = 128 keys, N = the chunk's queries)
// With keys on TMEM lanes, the teacher's average over the G heads of a query
// is a sum of G adjacent columns inside one thread; each warp then reduces
// its 32 keys and writes, per (query, group, selected block, warp),
//   (sum Pt log2 Pt, sum Pt s2, max s2, sum 2^(s2 - max s2))   (s2 = s log2 e)
// and a combine kernel folds a row's partials in a fixed order, so the loss
// is reproducible and nothing is accumulated with atomics.
#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kRows = 128;          // (query, head) columns per chunk
constexpr int kKeys = 128;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int SUB = 128 * 128;

struct KlMeta {
    int i[kRows];
    int pos[kRows];
    int slot[kRows];
    float lse2[kRows];              // per (query, head) column: forward lse * log2(e)
    int nq;
};

template <int D, int DI, int G>
struct KlLayout {
    static constexpr int QPC = kRows / G;                   // queries per chunk
    static constexpr int NS = QPC < 16 ? 16 : QPC;          // index columns (MMA N >= 16)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_KI = OFF_K + (D / 64) * SUB;
    static constexpr int OFF_Q = OFF_KI + (DI / 64) * SUB;                  // 2 stages
    static constexpr int QI_ROWS_BYTES = NS * 128;                          // one [NS][64] sub-tile
    static constexpr int OFF_QI = OFF_Q + 2 * (D / 64) * SUB;               // 2 stages x DI/64 sub-tiles
    static constexpr int OFF_META = OFF_QI + 2 * (DI / 64) * ((QI_ROWS_BYTES + 1023) & ~1023);
    static constexpr int META_BYTES = (int)((sizeof(KlMeta) + 255) & ~size_t(255));
    static constexpr int SG = (32 / G) < 8 ? (32 / G) : 8;              // queries per reduction group
    static constexpr int OFF_RED = OFF_META + 2 * META_BYTES;             // per warp [3*SG][32] floats
    static constexpr int OFF_BAR = OFF_RED + kEpiWarps * 3 * SG * 32 * 4;
    static constexpr int ALLOC = OFF_BAR + 256 + 1024;
    static constexpr int QI_SUB = (QI_ROWS_BYTES + 1023) & ~1023;         // stride of q_idx sub-tiles
    static constexpr uint32_t TM_S = 0, TM_SI = 256;
};

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Bucket entries of one chunk: lane handles query slots lane, lane+32, ...
template <int EPL>
__device__ __forceinline__ void load_entries(int (&e)[EPL], const int32_t *__restrict__ bucket_q, int q0, int nq,
                                             int lane)
{
#pragma unroll
    for (int t = 0; t < EPL; ++t) {
        const int qq = lane + 32 * t;
        e[t] = qq < nq ? __ldg(bucket_q + q0 + qq) : 0;
    }
}

// Writes the chunk's metadata (query row, position, slot) from its entries.
template <int EPL>
__device__ __forceinline__ void store_meta(int *mi, int *mpos, int *mslot, const int (&e)[EPL], int qpc, int nq,
                                           const Problem &p, int lane)
{
#pragma unroll
    for (int t = 0; t < EPL; ++t) {
        const int qq = lane + 32 * t;
        if (qq < qpc) {
            const bool ok = qq < nq;
            const int i = ok ? entry_row(e[t]) : 0;
            mi[qq] = i;
            mpos[qq] = ok ? p.q_offset + i : -1;
            mslot[qq] = ok ? entry_slot(e[t]) : 0;
        }
    }
}

template <int D, int DI, int G>
__global__ void __launch_bounds__(kThreads, 1)
kl_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
             const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q,
             const bf16 *__restrict__ q_idx, const float *__restrict__ lse,
             const int32_t *__restrict__ bucket_off, const int32_t *__restrict__ bucket_q,
             float4 *__restrict__ part, DeviceStatus *st)
{
    using L = KlLayout<D, DI, G>;
    constexpr int QPC = L::QPC, NS = L::NS;
    // x = group, y = key block: the heavy early blocks of every group start first
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    if (qend <= qbeg) return;
    const int nch = (qend - qbeg + QPC - 1) / QPC;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint64_t *q_full = bars, *q_empty = bars + 2, *s_full = bars + 4, *s_free = bars + 6, *kv_full = bars + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 9);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long j0 = (long long)c * kKeys;

    if (threadIdx.x == 0) {
        for (int a = 0; a < 2; ++a) {
            // 32 cp.async arrivals + 32 metadata arrivals (+ lane 0's expect_tx
            // arrival for the TMA-loaded Q rows when G == 8)
            tc::mbar_init(&q_full[a], G == 8 ? 65 : 64);
            tc::mbar_init(&q_empty[a], 1 + kEpiWarps);
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kEpiWarps);
        }
        tc::mbar_init(kv_full, 1);
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
        // K and K_idx tiles of this (b, group, block) by TMA; rows past Nk read as zeros
        if (lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::mbar_arrive_expect_tx(kv_full, (D / 64 + DI / 64) * SUB);
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb)
                tc::tma_load_4d(sm + L::OFF_K + kb * SUB, &tmap_k, kv_full, kb * 64, r, (int)j0, b);
#pragma unroll
            for (int kb = 0; kb < DI / 64; ++kb)
                tc::tma_load_3d(sm + L::OFF_KI + kb * SUB, &tmap_ki, kv_full, kb * 64, (int)j0, b);
        }
        constexpr int EPL = (QPC + 31) / 32;
        constexpr int RPL = kRows / 32;                       // (query, head) rows per lane
        int ent[EPL], ent_next[EPL];
        load_entries(ent, bucket_q, qbeg, min(QPC, qend - qbeg), lane);
        for (int m = 0; m < nch; ++m) {
            const int a = m & 1;
            const int q0 = qbeg + m * QPC;
            const int nq = min(QPC, qend - q0);
            // this chunk's LSE values and the next chunk's entries are fetched
            // before waiting for a free stage
            float lv[RPL];
#pragma unroll
            for (int t = 0; t < RPL; ++t) {
                const int rho = lane + 32 * t, qq = rho / G, g = rho % G;
                int e = 0;
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    const int v = __shfl_sync(0xffffffffu, ent[u], qq & 31);
                    if ((qq >> 5) == u) e = v;
                }
                lv[t] = qq < nq ? __ldg(lse + ((long long)b * p.Hq + r * G + g) * p.Nq + entry_row(e)) : 0.f;
            }
            if (m + 1 < nch) load_entries(ent_next, bucket_q, q0 + QPC, min(QPC, qend - q0 - QPC), lane);
            if (!tc::mbar_wait(&q_empty[a], ((uint32_t)(m >> 1) & 1u) ^ 1u, st, 81, abort_flag)) break;
            KlMeta *meta = reinterpret_cast<KlMeta *>(sm + L::OFF_META + a * L::META_BYTES);
            store_meta(meta->i, meta->pos, meta->slot, ent, QPC, nq, p, lane);
            if (lane == 0) meta->nq = nq;
#pragma unroll
            for (int t = 0; t < RPL; ++t) {
                const int rho = lane + 32 * t;
                meta->lse2[rho] = rho / G < nq ? lv[t] * kLog2e : INFINITY;
            }
            __syncwarp();
            uint8_t *sq = sm + L::OFF_Q + a * ((D / 64) * SUB);
            if constexpr (G == 8) {
                // one TMA box {64 features, 8 heads} per query and 64-feature half:
                // 1024 bytes, so every box starts on a swizzle-pattern boundary.
                // Padding slots read rows past the end of q (zero fill).
                if (lane == 0) tc::mbar_arrive_expect_tx(&q_full[a], kRows * D * 2);
                __syncwarp();
#pragma unroll
                for (int t = 0; t < EPL; ++t) {
                    const int qq = lane + 32 * t;
                    if (qq < QPC) {
                        const int z = qq < nq ? b * p.Nq + entry_row(ent[t]) : p.B * p.Nq;
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb)
                            tc::tma_load_3d(sq + kb * SUB + qq * (G * 128), &tmap_q, &q_full[a], kb * 64, r * G, z);
                    }
                }
            } else {
                constexpr int CPR = D / 8, RPI = 32 / CPR;
#pragma unroll 8
                for (int it = 0; it < kRows / RPI; ++it) {
                    const int rho = it * RPI + lane / CPR, ch = lane % CPR;
                    const int qq = rho / G, g = rho % G;
                    cp_async16_zfill(sq + (ch >> 3) * SUB + swz(rho, ch & 7),
                                     q + (((long long)b * p.Nq + meta->i[qq]) * p.Hq + (long long)r * G + g) * D + ch * 8,
                                     qq < nq);
                }
            }
            uint8_t *sqi = sm + L::OFF_QI + a * ((DI / 64) * L::QI_SUB);
            {
                constexpr int CPR = DI / 8, RPI = 32 / CPR;
#pragma unroll 4
                for (int it = 0; it < NS / RPI; ++it) {
                    const int row = it * RPI + lane / CPR, ch = lane % CPR;
                    const bool ok = row < nq;
                    cp_async16_zfill(sqi + (ch >> 3) * L::QI_SUB + swz(row, ch & 7),
                                     q_idx + (((long long)b * p.Nq + (ok ? meta->i[row] : 0)) * p.Hkv + r) * DI + ch * 8,
                                     ok);
                }
            }
            cp_async_arrive_noinc(&q_full[a]);
            tc::mbar_arrive(&q_full[a]);
#pragma unroll
            for (int t = 0; t < EPL; ++t) ent[t] = ent_next[t];
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t I_S = tc::idesc_bf16(128, kRows);
            constexpr uint32_t I_SI = tc::idesc_bf16(128, NS);
            const uint32_t aK = smem_u32(sm + L::OFF_K), aKI = smem_u32(sm + L::OFF_KI);
            bool ok = tc::mbar_wait(kv_full, 0, st, 82, abort_flag);
            if (ok) tc::fence_proxy_async();
            int issued = 0;
            for (int n = 0; ok && n < nch; ++n) {
                const int a = n & 1;
                const uint32_t ph = (uint32_t)(n >> 1) & 1u;
                if (!tc::mbar_wait(&q_full[a], ph, st, 83, abort_flag)) break;
                if (!tc::mbar_wait(&s_free[a], ph ^ 1u, st, 84, abort_flag)) break;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint32_t aQ = smem_u32(sm + L::OFF_Q + a * ((D / 64) * SUB));
                const uint32_t aQI = smem_u32(sm + L::OFF_QI + a * ((DI / 64) * L::QI_SUB));
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * SUB + (ks & 3) * 32;
                    tc::mma_bf16(tmem + L::TM_S + a * 128, tc::sdesc_k128(aK + off), tc::sdesc_k128(aQ + off), I_S,
                                 ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < DI / 16; ++ks) {
                    tc::mma_bf16(tmem + L::TM_SI + a * 128, tc::sdesc_k128(aKI + (ks >> 2) * SUB + (ks & 3) * 32),
                                 tc::sdesc_k128(aQI + (ks >> 2) * L::QI_SUB + (ks & 3) * 32), I_SI, ks > 0);
                }
                tc::mma_commit(&s_full[a]);
                tc::mma_commit(&q_empty[a]);
                issued = n + 1;
            }
            if (*abort_flag && issued > 0) {
                const int m = issued - 1;
                tc::mbar_wait(&s_full[m & 1], (uint32_t)(m >> 1) & 1u, nullptr, 0, nullptr);
            }
        }
    } else {
        // ------------------------------------------------ epilogue: one key per thread
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;
        const long long j = j0 + kr;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale * kLog2e, si2 = p.scale_idx * kLog2e;
        const float invG = 1.f / (float)G;
        for (int n = 0; n < nch; ++n) {
            const int a = n & 1;
            const uint32_t ph = (uint32_t)(n >> 1) & 1u;
            const KlMeta *meta = reinterpret_cast<const KlMeta *>(sm + L::OFF_META + a * L::META_BYTES);
            if (!tc::mbar_wait(&q_full[a], ph, st, 91, abort_flag)) break;
            if (!tc::mbar_wait(&s_full[a], ph, st, 92, abort_flag)) break;
            tc::fence_after_sync();
            const int nq = meta->nq;
            // queries in groups of 32 / G per 32-column TMEM slice
            constexpr int QS = 32 / G;            // queries per 32-column slice
            constexpr int SG = L::SG;             // queries per reduction group
            float *red = reinterpret_cast<float *>(sm + L::OFF_RED) + quarter * (3 * SG * 32);
#pragma unroll
            for (int c32 = 0; c32 < kRows / 32; ++c32) {
                uint32_t sv[32], si[32];
                tc::tmem_ld32_nowait(tmem + lane_base + L::TM_S + a * 128 + c32 * 32, sv);
                tc::tmem_ld32_nowait(tmem + lane_base + L::TM_SI + a * 128 + ((c32 * QS) / 32) * 32, si);
                tc::tmem_wait32(sv);
                tc::tmem_wait32(si);
#pragma unroll
                for (int sg = 0; sg < QS / SG; ++sg) {
                    // per-key terms of SG queries -> shared memory, one row per (query, term)
                    float s2v[SG];
                    bool visv[SG];
#pragma unroll
                    for (int u = 0; u < SG; ++u) {
                        const int ql = sg * SG + u;                 // query within the slice
                        const int qq = c32 * QS + ql;               // query within the chunk
                        const bool vis = qq < nq && j <= meta->pos[qq] && j < p.Nk;
                        float pt = 0.f;
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            pt += vis ? tc::ex2(__uint_as_float(sv[ql * G + g]) * sl2 - meta->lse2[qq * G + g]) : 0.f;
                        pt *= invG;
                        const float s2 = vis ? __uint_as_float(si[qq & 31]) * si2 : -INFINITY;
                        red[(u * 3 + 0) * 32 + lane] = pt > 0.f ? pt * tc::lg2(pt) : 0.f;
                        red[(u * 3 + 1) * 32 + lane] = vis ? pt * s2 : 0.f;
                        red[(u * 3 + 2) * 32 + lane] = s2;
                        s2v[u] = s2;
                        visv[u] = vis;
                    }
                    __syncwarp();
                    // lane l < 3*SG reduces row l over the warp's 32 keys (sum, sum, max)
                    float res = 0.f;
                    if (lane < 3 * SG) {
                        const float *row = red + lane * 32;
                        if (lane % 3 == 2) {
                            float m = -INFINITY;
#pragma unroll
                            for (int k2 = 0; k2 < 32; ++k2) m = fmaxf(m, row[(k2 + lane) & 31]);
                            res = m;
                        } else {
#pragma unroll
                            for (int k2 = 0; k2 < 32; ++k2) res += row[(k2 + lane) & 31];
                        }
                    }
                    __syncwarp();
                    float Mv[SG];
#pragma unroll
                    for (int u = 0; u < SG; ++u) {
                        Mv[u] = __shfl_sync(0xffffffffu, res, u * 3 + 2);
                        red[u * 32 + lane] = (visv[u] && Mv[u] != -INFINITY) ? tc::ex2(s2v[u] - Mv[u]) : 0.f;
                    }
                    __syncwarp();
                    float Z = 0.f;
                    if (lane < SG) {
#pragma unroll
                        for (int k2 = 0; k2 < 32; ++k2) Z += red[lane * 32 + ((k2 + lane) & 31)];
                    }
                    const float Aq = __shfl_sync(0xffffffffu, res, (lane % SG) * 3);
                    const float Bq = __shfl_sync(0xffffffffu, res, (lane % SG) * 3 + 1);
                    const float Mq = __shfl_sync(0xffffffffu, res, (lane % SG) * 3 + 2);
                    const int qq = c32 * QS + sg * SG + lane;
                    if (lane < SG && qq < nq) {
                        const long long row = ((long long)b * p.Hkv + r) * p.Nq + meta->i[qq];
                        part[(row * p.topk + meta->slot[qq]) * kEpiWarps + quarter] = make_float4(Aq, Bq, Mq, Z);
                    }
                    __syncwarp();
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&s_free[a]);
                tc::mbar_arrive(&q_empty[a]);
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

// Thread per (b, r, i): fold the row's partials (slots in order, then warps).
__global__ void kl_combine_kernel(Problem p, const int32_t *__restrict__ sel, const float4 *__restrict__ part,
                                  float *__restrict__ lse_idx, float *__restrict__ kl_rows)
{
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= (long long)p.B * p.Hkv * p.Nq) return;
    const int i = (int)(row % p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + row * p.topk;
    float A = 0.f, Bv = 0.f, M = -INFINITY;
    for (int t = 0; t < p.topk; ++t) {
        const int cc = srow[t];
        if (cc < 0 || cc >= p.nb || (long long)cc * 128 > pos) continue;
        for (int w = 0; w < kEpiWarps; ++w) {
            const float4 v = part[(row * p.topk + t) * kEpiWarps + w];
            A += v.x;
            Bv += v.y;
            M = fmaxf(M, v.z);
        }
    }
    float Z = 0.f;
    for (int t = 0; t < p.topk; ++t) {
        const int cc = srow[t];
        if (cc < 0 || cc >= p.nb || (long long)cc * 128 > pos) continue;
        for (int w = 0; w < kEpiWarps; ++w) {
            const float4 v = part[(row * p.topk + t) * kEpiWarps + w];
            if (v.w > 0.f) Z += v.w * exp2f(v.z - M);
        }
    }
    const float lse2 = M + log2f(Z);
    lse_idx[row] = lse2 * kLn2;
    kl_rows[row] = (A - Bv + lse2) * kLn2;
}

template <int D, int DI, int G>
cudaError_t launch_ddg(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                       const int32_t *sel, const float *lse, const KlWork &w, DeviceStatus *st, cudaStream_t s)
{
    using L = KlLayout<D, DI, G>;
    cudaError_t e = cudaFuncSetAttribute(kl_tc_kernel<D, DI, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tki;
    {
        const unsigned long long dq[3] = {(unsigned long long)D, (unsigned long long)p.Hq, (unsigned long long)p.B * p.Nq};
        const unsigned long long sq[2] = {D * 2ull, (unsigned long long)p.Hq * D * 2ull};
        const unsigned bq[3] = {64, (unsigned)G, 1};
        if ((e = make_tmap_bf16(&tq, q, 3, dq, sq, bq)) != cudaSuccess) return e;
        // K as [B][Nk][Hkv][D], K_idx as [B][Nk][DI] (rows past Nk are out of bounds)
        const unsigned long long dk[4] = {(unsigned long long)D, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                          (unsigned long long)p.B};
        const unsigned long long sk[3] = {D * 2ull, (unsigned long long)p.Hkv * D * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * D * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk, sk, bk)) != cudaSuccess) return e;
        const unsigned long long di[3] = {(unsigned long long)DI, (unsigned long long)p.Nk, (unsigned long long)p.B};
        const unsigned long long si[2] = {DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull};
        const unsigned bi[3] = {64, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    }
    {
        TimedLaunch timed_("kl_tc_kernel", s);
        kl_tc_kernel<D, DI, G><<<dim3(p.Hkv, p.nb, p.B), kThreads, L::ALLOC, s>>>(tq, tk, tki, p, q, q_idx, lse,
                                                                                 w.bucket_off, w.bucket_q, w.part, st);
    }
    note_launch();
    return cudaGetLastError();
}

template <int D, int DI>
cudaError_t launch_dd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                      const int32_t *sel, const float *lse, const KlWork &w, DeviceStatus *st, cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_ddg<D, DI, 1>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    case 2: return launch_ddg<D, DI, 2>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    case 4: return launch_ddg<D, DI, 4>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    default: return launch_ddg<D, DI, 8>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    }
}

}  // namespace

cudaError_t launch_kl_keymajor(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                               const int32_t *sel, const float *lse, float *lse_idx, float *kl_rows, const KlWork &w,
                               DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e = launch_inverse_index(p, sel, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, st, s);
    if (e != cudaSuccess) return e;
    if (p.d == 128 && p.d_idx == 128) e = launch_dd<128, 128>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    else if (p.d == 128) e = launch_dd<128, 64>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    else if (p.d_idx == 128) e = launch_dd<64, 128>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    else e = launch_dd<64, 64>(p, q, k, q_idx, k_idx, sel, lse, w, st, s);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Hkv * p.Nq;
    {
        TimedLaunch timed_("kl_combine_kernel", s);
        kl_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p, sel, w.part, lse_idx, kl_rows);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
