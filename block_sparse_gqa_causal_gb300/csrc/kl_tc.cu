// kl_tc.cu -- KL alignment loss of MSA, key-major on the tcgen05 tensor cores.
//
// "Sparse Attention · Part II", section 3.2 (the L_KL equation): for query i
// and group r over the selected token set T, with the detached teacher
// Pt_j = (1/G) sum_h exp(l_{h,j} - lse_h) and the student Ps = softmax_T(s),
//   KL = sum_j Pt_j log Pt_j - sum_j Pt_j s_j + log sum_j exp(s_j).
// Every term is a sum over T, so it splits over the selected blocks.  Two
// passes over the buckets of the inverse index (the queries that selected
// each (b, group, block)), each CTA keeping one 128-token block on chip:
//
//  1. teacher: S^T = K Q^T (M = 128 keys, N = 128 (query, head) rows).  With
//     keys on the TMEM lanes the mean over a query's G heads is a sum of G
//     adjacent columns inside one thread; Pt is written as fp16 per (bucket
//     entry, key).
//  2. index: s = q_idx K_idx^T (M = 128 queries, N = 128 keys).  With queries
//     on the TMEM lanes every sum over the block's keys stays in one thread:
//       (sum Pt log2 Pt, sum Pt s2, max s2, sum 2^(s2 - max s2))   (s2 = s log2 e)
//     per (query, group, selected block, half of the keys).
// A combine kernel folds a row's partials in a fixed order, so the loss is
// reproducible and nothing is accumulated with atomics.
//
// Training runs only the index pass without the teacher (max and sum of
// 2^s2, i.e. lse_idx, which the backward needs first): the fused backward
// recomputes the teacher anyway and folds the two teacher sums of the loss
// into its own tiles, and bwd_kl_combine_kernel below assembles the rows.
#include <cuda_fp16.h>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kKeys = 128;
constexpr int kRows = 128;                 // teacher pass: (query, head) rows per chunk
constexpr int kQ = 128;                    // index pass: queries per chunk
constexpr int kEpiWarps = 8;
constexpr int kProd2 = 2 + kEpiWarps;      // second producer warp: the two take alternate chunks
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr int kStages = 3;
constexpr int kParts = 2;                  // partials per (query, group, slot): the two key halves
constexpr int SUB = 128 * 128;             // [128 rows][64 bf16] swizzled sub-tile

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait with the same outcome on every lane (warp-collective TMEM
// loads follow).
__device__ __forceinline__ bool wwait(uint64_t *bar, uint32_t parity, DeviceStatus *st, int site,
                                      volatile int *abort_flag)
{
    const bool r = tc::mbar_wait(bar, parity, st, site, abort_flag);
    return __all_sync(0xffffffffu, r);
}

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

// ============================================================== pass 1: teacher
// A [128 rows][D] tile is stored as 8-row groups of D/64 feature halves
// (1024-byte swizzle atoms): row rho, half h at (rho/8)*(D/64)*1024 + h*1024
// + (rho%8)*128.  With groups of 8 heads one query's rows form one group,
// which a single TMA box fills.
template <int D>
struct TeacherLayout {
    static constexpr int H = D / 64;
    static constexpr int TILE = kRows * D * 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + H * SUB;          // kStages tiles
    static constexpr int OFF_META = OFF_Q + kStages * TILE;
    struct Meta {
        float lse2[kRows];     // lse * log2(e) per (query, head) row
        int pos[kRows];        // position per query slot (-1: padding)
        int qi[kRows];         // query index per slot
        int e0, nq;
    };
    static constexpr int META_BYTES = (int)((sizeof(Meta) + 127) & ~size_t(127));
    static constexpr int OFF_BAR = OFF_META + kStages * META_BYTES;
    static constexpr int ALLOC = OFF_BAR + 256 + 1024;
};

template <int D>
__device__ __forceinline__ int roff(int rho, int half, int ch)
{
    return (rho >> 3) * (D / 64) * 1024 + half * 1024 + (rho & 7) * 128 + (((ch ^ rho) & 7) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
kl_teacher_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     Problem p, const bf16 *__restrict__ q, const float *__restrict__ lse,
                     const int32_t *__restrict__ bucket_off, const int32_t *__restrict__ bucket_q,
                     __half *__restrict__ pt_out, DeviceStatus *st)
{
    using L = TeacherLayout<D>;
    using Meta = typename L::Meta;
    constexpr int QPC = kRows / G;
    constexpr int EPL = (QPC + 31) / 32;
    // x = group, y = key block: the heavy early blocks of every group start first
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    if (qend <= qbeg) return;
    const int nch = (qend - qbeg + QPC - 1) / QPC;
    const long long j0 = (long long)c * kKeys;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint64_t *full = bars, *empty = bars + kStages, *s_full = bars + 2 * kStages, *s_free = s_full + 2;
    uint64_t *kv_full = s_free + 2, *done = kv_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < kStages; ++a) {
            // G == 8: lane 0's expect_tx arrival + 32 row-data arrivals;
            // otherwise 32 cp.async arrivals + 32 row-data arrivals
            tc::mbar_init(&full[a], G == 8 ? 33 : 64);
            tc::mbar_init(&empty[a], 1 + kEpiWarps);       // S MMA done + epilogue has read the row data
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kEpiWarps);
        }
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == kProd2) {
        // ------------------------------------------------ producers (warp 0: even chunks, kProd2: odd)
        const int pw = warp == 0 ? 0 : 1;
        if (pw == 0 && lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::mbar_arrive_expect_tx(kv_full, L::H * SUB);
#pragma unroll
            for (int h = 0; h < L::H; ++h)
                tc::tma_load_4d(sm + L::OFF_K + h * SUB, &tmap_k, kv_full, h * 64, r, (int)j0, b);
        }
        // Entries run two chunks ahead and the rows' LSE one chunk ahead, so
        // no load is waited for on the way to the next stage.
        auto load_lse = [&](float (&vl)[4], const int (&e_)[EPL], int nqx) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int rho = lane + 32 * t, qq = rho / G, g = rho % G;
                int e = 0;
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    const int x = __shfl_sync(0xffffffffu, e_[u], qq & 31);
                    if ((qq >> 5) == u) e = x;
                }
                vl[t] = qq < nqx ? __ldg(lse + ((long long)b * p.Hq + r * G + g) * p.Nq + entry_row(e)) : INFINITY;
            }
        };
        int ent[EPL], ent1[EPL], ent2[EPL];
        const int qb0 = qbeg + pw * QPC;           // this producer's first chunk
        load_entries(ent, bucket_q, qb0, min(QPC, qend - qb0), lane);
        load_entries(ent1, bucket_q, qb0 + 2 * QPC, min(QPC, qend - qb0 - 2 * QPC), lane);
        float vl[4], vl_next[4];
        load_lse(vl, ent, min(QPC, qend - qb0));
        for (int m = pw; m < nch; m += 2) {
            const int s = m % kStages;
            const int q0 = qbeg + m * QPC;
            const int nq = min(QPC, qend - q0);
            load_entries(ent2, bucket_q, q0 + 4 * QPC, min(QPC, qend - q0 - 4 * QPC), lane);
            if (m + 2 < nch) load_lse(vl_next, ent1, min(QPC, qend - q0 - 2 * QPC));
            if (!tc::mbar_wait(&empty[s], ((uint32_t)(m / kStages) & 1u) ^ 1u, st, 81, abort_flag)) break;
            Meta *meta = reinterpret_cast<Meta *>(sm + L::OFF_META + s * L::META_BYTES);
#pragma unroll
            for (int t = 0; t < 4; ++t) meta->lse2[lane + 32 * t] = vl[t] * kLog2e;
#pragma unroll
            for (int t = 0; t < EPL; ++t) {
                const int qq = lane + 32 * t;
                if (qq < QPC) {
                    const bool ok = qq < nq;
                    const int i = ok ? entry_row(ent[t]) : 0;
                    meta->qi[qq] = i;
                    meta->pos[qq] = ok ? p.q_offset + i : -1;
                }
            }
            if (lane == 0) {
                meta->e0 = q0;
                meta->nq = nq;
            }
            __syncwarp();
            uint8_t *sq = sm + L::OFF_Q + s * L::TILE;
            if constexpr (G == 8) {
                // one TMA box {64 features, 8 heads, D/64 halves} per query fills
                // its row group; padding slots read past the end (zero fill)
                if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], L::TILE);
                __syncwarp();
                if (lane < QPC) {
                    const int z = lane < nq ? b * p.Nq + entry_row(ent[0]) : p.B * p.Nq;
                    tc::tma_load_4d(sq + lane * (L::H * 1024), &tmap_q, &full[s], 0, r * G, 0, z);
                }
            } else {
                constexpr int CPR = D / 8, RPI = 32 / CPR;
#pragma unroll 4
                for (int it = 0; it < kRows / RPI; ++it) {
                    const int rho = it * RPI + lane / CPR, ch = lane % CPR;
                    const int qq = rho / G, g = rho % G;
                    cp_async16_zfill(sq + roff<D>(rho, ch >> 3, ch & 7),
                                     q + (((long long)b * p.Nq + meta->qi[qq]) * p.Hq + (long long)r * G + g) * D + ch * 8,
                                     qq < nq);
                }
                cp_async_arrive_noinc(&full[s]);
            }
            tc::mbar_arrive(&full[s]);
#pragma unroll
            for (int t = 0; t < EPL; ++t) {
                ent[t] = ent1[t];
                ent1[t] = ent2[t];
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) vl[t] = vl_next[t];
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t I_S = tc::idesc_bf16(128, kRows);
            const uint64_t dK = tc::sdesc_k128(smem_u32(sm + L::OFF_K));
            bool ok = tc::mbar_wait(kv_full, 0, st, 82, abort_flag);
            for (int n = 0; ok && n < nch; ++n) {
                if (!tc::mbar_wait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, st, 83, abort_flag)) break;
                if (n >= 2 && !tc::mbar_wait(&s_free[n & 1], ((uint32_t)(n >> 1) & 1u) ^ 1u, st, 84, abort_flag)) break;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint64_t dQ = tc::sdesc_sw128(smem_u32(sm + L::OFF_Q + (n % kStages) * L::TILE), 16, L::H * 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                    // B = Q rows, K-major, 8-row groups (D/64) KB apart
                    tc::mma_bf16(tmem + (n & 1) * kRows, tc::desc_adv(dK, h * SUB + ko), tc::desc_adv(dQ, h * 1024 + ko),
                                 I_S, ks > 0);
                }
                tc::mma_commit(&s_full[n & 1]);
                tc::mma_commit(&empty[n % kStages]);
            }
            tc::mma_commit(done);
            tc::mbar_wait(done, 0, nullptr, 0, nullptr);
        }
    } else if (warp < kProd2) {
        // ------------------------------------------------ epilogue: one key per thread
        const int qd = warp & 3, hf = (warp - 2) >> 2;
        const int kr = qd * 32 + lane;
        const long long j = j0 + kr;
        const bool key_ok = j < p.Nk;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const float sl2 = p.scale * kLog2e, invG = 1.f / (float)G;
        constexpr int QH = 64 / G;                  // queries among this warp's 64 columns
        for (int n = 0; n < nch; ++n) {
            const Meta *meta = reinterpret_cast<const Meta *>(sm + L::OFF_META + (n % kStages) * L::META_BYTES);
            if (!wwait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, st, 91, abort_flag)) break;
            if (!wwait(&s_full[n & 1], (uint32_t)(n >> 1) & 1u, st, 92, abort_flag)) break;
            tc::fence_after_sync();
            uint32_t sv[2][32];
            tc::tmem_ld32_nowait(tmem + lane_base + (n & 1) * kRows + hf * 64, sv[0]);
            tc::tmem_ld32_nowait(tmem + lane_base + (n & 1) * kRows + hf * 64 + 32, sv[1]);
            // row data into registers while the loads land
            float l2[64];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const float4 l4 = reinterpret_cast<const float4 *>(meta->lse2 + hf * 64)[x];
                l2[4 * x] = l4.x; l2[4 * x + 1] = l4.y; l2[4 * x + 2] = l4.z; l2[4 * x + 3] = l4.w;
            }
            unsigned long long vmask = 0;           // bit u: this key is visible to query u of the half
#pragma unroll
            for (int u = 0; u < QH; ++u)
                vmask |= (key_ok && j <= (long long)meta->pos[hf * QH + u]) ? (1ull << u) : 0ull;
            const int nq = meta->nq, e0 = meta->e0;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[n % kStages]);   // row data now in registers
            tc::tmem_wait32(sv[0]);
            tc::tmem_wait32(sv[1]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s_free[n & 1]);
            float e[64];
#pragma unroll
            for (int col = 0; col < 64; ++col)
                e[col] = tc::ex2(__uint_as_float(sv[col >> 5][col & 31]) * sl2 - l2[col]);
#pragma unroll
            for (int u = 0; u < QH; ++u) {
                // pairwise sum over the query's G heads (adjacent columns)
                float t[G];
#pragma unroll
                for (int g = 0; g < G; ++g) t[g] = e[u * G + g];
#pragma unroll
                for (int w = G / 2; w > 0; w >>= 1)
#pragma unroll
                    for (int g = 0; g < w; ++g) t[g] += t[g + w];
                const int qq = hf * QH + u;
                const bool vis = (vmask >> u) & 1ull;
                if (qq < nq) pt_out[(long long)(e0 + qq) * kKeys + kr] = __float2half_rn(vis ? t[0] * invG : 0.f);
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

// ============================================================== pass 2: index
template <int DI>
struct IndexLayout {
    static constexpr int H = DI / 64;
    static constexpr int OFF_KI = 0;
    static constexpr int OFF_Q = OFF_KI + H * SUB;          // kStages x q_idx [128 queries][DI]
    static constexpr int OFF_META = OFF_Q + kStages * H * SUB;
    struct Meta {
        int pos[kQ];           // position (-1: padding)
        int qi[kQ];
        int slot[kQ];
        int e0, nq;
    };
    static constexpr int META_BYTES = (int)((sizeof(Meta) + 127) & ~size_t(127));
    static constexpr int OFF_BAR = OFF_META + kStages * META_BYTES;
    static constexpr int ALLOC = OFF_BAR + 256 + 1024;
};

template <int DI, bool kTeacher>
__global__ void __launch_bounds__(kThreads, 1)
kl_index_tc_kernel(const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q_idx,
                   const int32_t *__restrict__ bucket_off, const int32_t *__restrict__ bucket_q,
                   const __half *__restrict__ pt, float4 *__restrict__ part, DeviceStatus *st)
{
    using L = IndexLayout<DI>;
    using Meta = typename L::Meta;
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    if (qend <= qbeg) return;
    const int nch = (qend - qbeg + kQ - 1) / kQ;
    const long long j0 = (long long)c * kKeys;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint64_t *full = bars, *empty = bars + kStages, *s_full = bars + 2 * kStages, *s_free = s_full + 2;
    uint64_t *kv_full = s_free + 2, *done = kv_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < kStages; ++a) {
            tc::mbar_init(&full[a], 64);                   // 32 cp.async arrivals + 32 row-data arrivals
            tc::mbar_init(&empty[a], 1 + kEpiWarps);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kEpiWarps);
        }
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == kProd2) {
        // ------------------------------------------------ producers (warp 0: even chunks, kProd2: odd)
        const int pw = warp == 0 ? 0 : 1;
        if (pw == 0 && lane == 0) {
            tc::mbar_arrive_expect_tx(kv_full, L::H * SUB);
#pragma unroll
            for (int h = 0; h < L::H; ++h) tc::tma_load_3d(sm + L::OFF_KI + h * SUB, &tmap_ki, kv_full, h * 64, (int)j0, b);
        }
        int ent[4], ent_next[4];
        load_entries(ent, bucket_q, qbeg + pw * kQ, min(kQ, qend - qbeg - pw * kQ), lane);
        for (int m = pw; m < nch; m += 2) {
            const int s = m % kStages;
            const int q0 = qbeg + m * kQ;
            const int nq = min(kQ, qend - q0);
            if (m + 2 < nch) load_entries(ent_next, bucket_q, q0 + 2 * kQ, min(kQ, qend - q0 - 2 * kQ), lane);
            if (!tc::mbar_wait(&empty[s], ((uint32_t)(m / kStages) & 1u) ^ 1u, st, 85, abort_flag)) break;
            Meta *meta = reinterpret_cast<Meta *>(sm + L::OFF_META + s * L::META_BYTES);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int qq = lane + 32 * t;
                const bool ok = qq < nq;
                const int i = ok ? entry_row(ent[t]) : 0;
                meta->qi[qq] = i;
                meta->pos[qq] = ok ? p.q_offset + i : -1;
                meta->slot[qq] = ok ? entry_slot(ent[t]) : 0;
            }
            if (lane == 0) {
                meta->e0 = q0;
                meta->nq = nq;
            }
            // q_idx rows: lane l gathers whole rows l, l+32, l+64, l+96 (its own entries)
            uint8_t *sq = sm + L::OFF_Q + s * (L::H * SUB);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int row = lane + 32 * t;
                const bf16 *src = q_idx + (((long long)b * p.Nq + entry_row(ent[t])) * p.Hkv + r) * DI;
#pragma unroll
                for (int ch = 0; ch < DI / 8; ++ch)
                    cp_async16_zfill(sq + (ch >> 3) * SUB + swz(row, ch & 7), src + ch * 8, row < nq);
            }
            cp_async_arrive_noinc(&full[s]);
            tc::mbar_arrive(&full[s]);
#pragma unroll
            for (int t = 0; t < 4; ++t) ent[t] = ent_next[t];
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer: s = q_idx K_idx^T
            constexpr uint32_t I_S = tc::idesc_bf16(128, kKeys);
            const uint64_t dKI = tc::sdesc_k128(smem_u32(sm + L::OFF_KI));
            bool ok = tc::mbar_wait(kv_full, 0, st, 86, abort_flag);
            for (int n = 0; ok && n < nch; ++n) {
                if (!tc::mbar_wait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, st, 87, abort_flag)) break;
                if (n >= 2 && !tc::mbar_wait(&s_free[n & 1], ((uint32_t)(n >> 1) & 1u) ^ 1u, st, 88, abort_flag)) break;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint64_t dQ = tc::sdesc_k128(smem_u32(sm + L::OFF_Q + (n % kStages) * (L::H * SUB)));
#pragma unroll
                for (int ks = 0; ks < DI / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * SUB + (ks & 3) * 32;
                    tc::mma_bf16(tmem + (n & 1) * kKeys, tc::desc_adv(dQ, off), tc::desc_adv(dKI, off), I_S, ks > 0);
                }
                tc::mma_commit(&s_full[n & 1]);
                tc::mma_commit(&empty[n % kStages]);
            }
            tc::mma_commit(done);
            tc::mbar_wait(done, 0, nullptr, 0, nullptr);
        }
    } else if (warp < kProd2) {
        // ------------------------------------------------ epilogue: one query per thread, 64 keys
        const int qd = warp & 3, hf = (warp - 2) >> 2;
        const int u = qd * 32 + lane;               // query slot in the chunk (TMEM lane)
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const float si2 = p.scale_idx * kLog2e;
        const long long jb = j0 + hf * 64;          // first key of this warp's half
        for (int n = 0; n < nch; ++n) {
            const Meta *meta = reinterpret_cast<const Meta *>(sm + L::OFF_META + (n % kStages) * L::META_BYTES);
            if (!wwait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, st, 93, abort_flag)) break;
            const int nq = meta->nq, e0 = meta->e0;
            const bool valid = u < nq;
            const long long pos = valid ? (long long)meta->pos[u] : -1;
            const int qi = meta->qi[u], slot = meta->slot[u];
            // the teacher's 64 values for this query and key half
            uint4 tv[8];
            if constexpr (kTeacher) {
                const uint4 *src = reinterpret_cast<const uint4 *>(pt + (long long)(e0 + (valid ? u : 0)) * kKeys + hf * 64);
#pragma unroll
                for (int x = 0; x < 8; ++x) tv[x] = valid ? __ldg(src + x) : make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[n % kStages]);   // row data read
            if (!wwait(&s_full[n & 1], (uint32_t)(n >> 1) & 1u, st, 94, abort_flag)) break;
            tc::fence_after_sync();
            uint32_t sv[2][32];
            tc::tmem_ld32_nowait(tmem + lane_base + (n & 1) * kKeys + hf * 64, sv[0]);
            tc::tmem_ld32_nowait(tmem + lane_base + (n & 1) * kKeys + hf * 64 + 32, sv[1]);
            tc::tmem_wait32(sv[0]);
            tc::tmem_wait32(sv[1]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s_free[n & 1]);
            // visible keys of this half: jb .. jb + nvis - 1
            const int nvis = (int)max(0LL, min(min(pos, (long long)p.Nk - 1) - jb + 1, 64LL));
            float M = -INFINITY;
#pragma unroll
            for (int x = 0; x < 64; ++x)
                if (x < nvis) M = fmaxf(M, __uint_as_float(sv[x >> 5][x & 31]) * si2);
            float A = 0.f, Bv = 0.f, Z = 0.f;
#pragma unroll
            for (int x = 0; x < 64; x += 8) {
                uint32_t w4[4] = {0u, 0u, 0u, 0u};
                if constexpr (kTeacher) {
                    w4[0] = tv[x / 8].x;
                    w4[1] = tv[x / 8].y;
                    w4[2] = tv[x / 8].z;
                    w4[3] = tv[x / 8].w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int col = x + e;
                    const float s2 = __uint_as_float(sv[col >> 5][col & 31]) * si2;
                    const __half2 h2 = *reinterpret_cast<const __half2 *>(&w4[e >> 1]);
                    const float ptv = (e & 1) ? __high2float(h2) : __low2float(h2);
                    if (col < nvis) {
                        Z += tc::ex2(s2 - M);
                        if constexpr (kTeacher) {
                            Bv += ptv * s2;
                            A += ptv > 0.f ? ptv * tc::lg2(ptv) : 0.f;
                        }
                    }
                }
            }
            if (valid) {
                const long long row = ((long long)b * p.Hkv + r) * p.Nq + qi;
                part[(row * p.topk + slot) * kParts + hf] = make_float4(A, Bv, M, Z);
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

// Folds a (query, group) row's partials over its valid slots in a fixed
// order: lse_idx = (M + log2 Z) ln 2 and KL = (A - B + M + log2 Z) ln 2.
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
        for (int w = 0; w < kParts; ++w) {
            const float4 v = part[(row * p.topk + t) * kParts + w];
            A += v.x;
            Bv += v.y;
            M = fmaxf(M, v.z);
        }
    }
    float Z = 0.f;
    for (int t = 0; t < p.topk; ++t) {
        const int cc = srow[t];
        if (cc < 0 || cc >= p.nb || (long long)cc * 128 > pos) continue;
        for (int w = 0; w < kParts; ++w) {
            const float4 v = part[(row * p.topk + t) * kParts + w];
            if (v.w > 0.f) Z += v.w * exp2f(v.z - M);
        }
    }
    const float lse2 = M + log2f(Z);
    lse_idx[row] = lse2 * kLn2;
    if (kl_rows) kl_rows[row] = (A - Bv + lse2) * kLn2;
}

// KL of each (query, group) row from the fused backward's partials: per valid
// slot the sum of Pt log2 Pt (kla) and four key-quarter sums of Pt s log2 e
// (klb); KL = (A - B) ln 2 + lse_idx.  Fixed order, no atomics.
__global__ void bwd_kl_combine_kernel(Problem p, const int32_t *__restrict__ sel, const float *__restrict__ lse_idx,
                                      const float *__restrict__ kla, const float4 *__restrict__ klb,
                                      float *__restrict__ kl_rows)
{
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= (long long)p.B * p.Hkv * p.Nq) return;
    const long long pos = (long long)p.q_offset + (row % p.Nq);
    const int32_t *srow = sel + row * p.topk;
    float A = 0.f, Bv = 0.f;
    for (int t = 0; t < p.topk; ++t) {
        const int cc = srow[t];
        if (cc < 0 || cc >= p.nb || (long long)cc * 128 > pos) continue;
        const float4 b = klb[row * p.topk + t];
        A += kla[row * p.topk + t];
        Bv += (b.x + b.y) + (b.z + b.w);
    }
    kl_rows[row] = (A - Bv) * kLn2 + lse_idx[row];
}

template <int D, int G>
cudaError_t launch_teacher(const Problem &p, const bf16 *q, const bf16 *k, const float *lse, const KlWork &w,
                           DeviceStatus *st, cudaStream_t s)
{
    using L = TeacherLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(kl_teacher_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk;
    {
        // Q as {d within a half, head, half, query row}: one box {64, G, D/64, 1}
        // is a query's G head rows in every feature half
        const unsigned long long dq4[4] = {64, (unsigned long long)p.Hq, (unsigned long long)(D / 64),
                                           (unsigned long long)p.B * p.Nq};
        const unsigned long long sq4[3] = {D * 2ull, 128ull, (unsigned long long)p.Hq * D * 2ull};
        const unsigned bq4[4] = {64, (unsigned)G, (unsigned)(D / 64), 1};
        if ((e = make_tmap_bf16(&tq, q, 4, dq4, sq4, bq4)) != cudaSuccess) return e;
        // K as [B][Nk][Hkv][D] (rows past Nk are out of bounds)
        const unsigned long long dk[4] = {(unsigned long long)D, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                          (unsigned long long)p.B};
        const unsigned long long sk[3] = {D * 2ull, (unsigned long long)p.Hkv * D * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * D * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk, sk, bk)) != cudaSuccess) return e;
    }
    {
        TimedLaunch timed_("kl_teacher_tc_kernel", s);
        kl_teacher_tc_kernel<D, G><<<dim3(p.Hkv, p.nb, p.B), kThreads, L::ALLOC, s>>>(tq, tk, p, q, lse, w.bucket_off,
                                                                                    w.bucket_q, w.pt, st);
    }
    note_launch();
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_teacher_d(const Problem &p, const bf16 *q, const bf16 *k, const float *lse, const KlWork &w,
                             DeviceStatus *st, cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_teacher<D, 1>(p, q, k, lse, w, st, s);
    case 2: return launch_teacher<D, 2>(p, q, k, lse, w, st, s);
    case 4: return launch_teacher<D, 4>(p, q, k, lse, w, st, s);
    default: return launch_teacher<D, 8>(p, q, k, lse, w, st, s);
    }
}

template <int DI, bool kTeacher>
cudaError_t launch_index(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, const KlWork &w, DeviceStatus *st,
                         cudaStream_t s)
{
    using L = IndexLayout<DI>;
    cudaError_t e =
        cudaFuncSetAttribute(kl_index_tc_kernel<DI, kTeacher>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tki;
    const unsigned long long di[3] = {(unsigned long long)DI, (unsigned long long)p.Nk, (unsigned long long)p.B};
    const unsigned long long si[2] = {DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull};
    const unsigned bi[3] = {64, (unsigned)kKeys, 1};
    if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    {
        TimedLaunch timed_("kl_index_tc_kernel", s);
        kl_index_tc_kernel<DI, kTeacher><<<dim3(p.Hkv, p.nb, p.B), kThreads, L::ALLOC, s>>>(
            tki, p, q_idx, w.bucket_off, w.bucket_q, w.pt, w.part, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

size_t kl_part_count(const Problem &p) { return (size_t)p.B * p.Hkv * p.Nq * p.topk * kParts; }

cudaError_t launch_kl_keymajor(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                               const int32_t *sel, const float *lse, float *lse_idx, float *kl_rows, const KlWork &w,
                               DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e = w.index_ready ? cudaSuccess
                                  : launch_inverse_index(p, sel, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, st, s);
    if (e != cudaSuccess) return e;
    if (w.pt) {
        e = p.d == 128 ? launch_teacher_d<128>(p, q, k, lse, w, st, s) : launch_teacher_d<64>(p, q, k, lse, w, st, s);
        if (e != cudaSuccess) return e;
        e = p.d_idx == 128 ? launch_index<128, true>(p, q_idx, k_idx, w, st, s)
                           : launch_index<64, true>(p, q_idx, k_idx, w, st, s);
    } else {
        // lse_idx only (kl_rows must be nullptr)
        e = p.d_idx == 128 ? launch_index<128, false>(p, q_idx, k_idx, w, st, s)
                           : launch_index<64, false>(p, q_idx, k_idx, w, st, s);
    }
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Hkv * p.Nq;
    {
        TimedLaunch timed_("kl_combine_kernel", s);
        kl_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p, sel, w.part, lse_idx, kl_rows);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_bwd_kl_combine(const Problem &p, const int32_t *sel, const float *lse_idx, const float *kla,
                                  const float *klb, float *kl_rows, cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Hkv * p.Nq;
    {
        TimedLaunch timed_("bwd_kl_combine_kernel", s);
        bwd_kl_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(
            p, sel, lse_idx, kla, reinterpret_cast<const float4 *>(klb), kl_rows);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
