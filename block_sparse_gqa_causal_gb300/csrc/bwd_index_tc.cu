// bwd_index_tc.cu -- index-branch backward of MSA on the tcgen05 tensor cores
// (d_idx = 128), key-major.
//
// "Sparse Attention · Part II", section 3.2: the index branch learns only
// from the KL alignment loss, with the teacher detached.  Expanding the KL,
// its gradient with respect to the index logit s_j of a selected key is
//     dKL/ds_j = Ps_j - Pt_j,
// Ps the index softmax over the selected set (normalised by lse_idx) and Pt
// the teacher, which the main-branch backward kernel leaves per (bucket
// entry, key).  One CTA owns one 128-key block of K_idx for one (b, group)
// and walks the bucket's queries in chunks of 128, keys as the MMA's M:
//   s^T = K_idx q_idx^T                              (M = 128 keys, N = 128 queries)
//   dsig = coef (exp2(s*scale_idx*log2e - lse_idx*log2e) - Pt) on visible keys
//   dq_idx^T = K_idx^T dsig^T                        (M = 128 features, N = 128 queries)
//   dK_idx += dsig^T q_idx                           (M = 128 keys, N = 128 features)
// dq_idx leaves as bf16 partial rows per (query, group, slot), summed by the
// combine kernel; dK_idx (shared by all groups) is added to an fp32 buffer
// once per CTA.  coef = scale_idx * kl_coef / (B * Nq * Hkv): the mean over
// (query, group) rows of the per-row KL, times the factor scale_idx that
// both gradients take from s = scale_idx q_idx . k_idx.  The kKL instantiation also gives the loss
// term sum_j Pt_j s_j log2(e) of each (query, group, selected block), one
// partial per lane quarter of keys (a transposing warp sum); with the
// teacher's sum of Pt log2 Pt and lse_idx it makes the KL of each row.
//
// Roles: warps 0 and 18 gather q_idx rows (cp.async) and row data for
// alternate chunks, warp 1 owns TMEM and issues the MMAs, warps 2..17 are
// the epilogue (TMEM lanes 32*(w%4).., query columns 32*((w-2)/4) .. +31).
// s^T and dsig^T are double-buffered.
#include <cuda_fp16.h>

#include <type_traits>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int DI = 128;
constexpr int kKeys = 128;
constexpr int kQ = 128;                        // queries per chunk
constexpr int kEpiWarps = 16;
constexpr int kCols = 128 / (kEpiWarps / 4);    // query columns per epilogue warp
constexpr int kHalves = kCols / 32;
constexpr int kProd2 = 2 + kEpiWarps;          // second producer warp: the two take alternate chunks
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr int SUB = 128 * 128;                 // [128 rows][64 bf16] swizzled sub-tile
constexpr int OFF_KI = 0;                      // K_idx: 2 feature halves
constexpr int kStages = 3;                     // q_idx stages
constexpr int OFF_STG = OFF_KI + 2 * SUB;      // kStages x q_idx [128 queries][128 features]
constexpr int OFF_SIG = OFF_STG + kStages * 2 * SUB;   // dsig^T [128 keys][128 queries]
constexpr int OFF_META = OFF_SIG + 2 * SUB;

struct Meta {
    float lsei2[kQ];        // lse_idx * log2(e) (+inf for padding)
    int pos[kQ];            // position (-1 for padding)
    int qi[kQ];
    int slot[kQ];
    int e0;                 // bucket-list index of the chunk's first entry
    int nq;
};
constexpr int META_BYTES = (int)((sizeof(Meta) + 127) & ~size_t(127));
constexpr int OFF_STAGE = OFF_META + kStages * META_BYTES;   // per epilogue warp: dq_idx [64 rows][32 features] bf16
constexpr int STAGE_BYTES = kCols * 64;
constexpr int OFF_BAR = OFF_STAGE + kEpiWarps * STAGE_BYTES;
constexpr int ALLOC = OFF_BAR + 256 + 1024;

constexpr uint32_t TM_S = 0, TM_DKI = 256, TM_DQI = 384;   // TM_S: 2 x 128

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool wwait(uint64_t *bar, uint32_t parity, DeviceStatus *st, int site,
                                      volatile int *abort_flag)
{
    const bool r = tc::mbar_wait(bar, parity, st, site, abort_flag);
    return __all_sync(0xffffffffu, r);
}

template <bool kKL>
__global__ void __launch_bounds__(kThreads, 1)
bwd_index_tc_kernel(const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q_idx,
                    const float *__restrict__ lse_idx, float coef, const int32_t *__restrict__ bucket_off,
                    const int32_t *__restrict__ bucket_q, const __half *__restrict__ pt,
                    const int32_t *__restrict__ pt_off,
                    bf16 *__restrict__ dqi_part, float *__restrict__ dki_acc, float *__restrict__ klb,
                    DeviceStatus *st)
{
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    if (qend <= qbeg) return;                          // no query selected this block: nothing to add
    const int nch = (qend - qbeg + kQ - 1) / kQ;
    const long long j0 = (long long)c * kKeys;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + 3, *s_full = bars + 6, *s_free = bars + 8;
    uint64_t *g_full = bars + 10, *g_free = bars + 11;
    uint64_t *dq_full = bars + 12, *dq_free = bars + 13, *kv_full = bars + 14, *done = bars + 15;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < kStages; ++a) {
            tc::mbar_init(&full[a], 64);               // 32 cp.async arrivals + 32 row-data arrivals
            tc::mbar_init(&empty[a], 1 + kEpiWarps);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kEpiWarps);
        }
        tc::mbar_init(g_full, kEpiWarps);
        tc::mbar_init(g_free, 1);
        tc::mbar_init(dq_full, 1);
        tc::mbar_init(dq_free, kEpiWarps);
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(done, 1);
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

    if (warp == 0 || warp == kProd2) {
        // ------------------------------------------------ producers (warp 0: even chunks, kProd2: odd)
        const int pw = warp == 0 ? 0 : 1;
        if (pw == 0 && lane == 0) {
            tc::mbar_arrive_expect_tx(kv_full, 2 * SUB);
#pragma unroll
            for (int h = 0; h < 2; ++h) tc::tma_load_3d(sm + OFF_KI + h * SUB, &tmap_ki, kv_full, h * 64, (int)j0, b);
        }
        // entries two chunks ahead, lse_idx one chunk ahead; lane l gathers whole
        // q_idx rows l, l+32, l+64, l+96 of a chunk (its own entries)
        auto load_ent = [&](int (&e)[4], int q0, int nqx) {
#pragma unroll
            for (int t = 0; t < 4; ++t) e[t] = lane + 32 * t < nqx ? __ldg(bucket_q + q0 + lane + 32 * t) : 0;
        };
        auto load_lse = [&](float (&vl)[4], const int (&e)[4], int nqx) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                vl[t] = lane + 32 * t < nqx ? __ldg(lse_idx + ((long long)b * p.Hkv + r) * p.Nq + entry_row(e[t])) : INFINITY;
        };
        int ent[4], ent1[4], ent2[4];
        float vl[4], vl_next[4];
        const int qb0 = qbeg + pw * kQ;             // this producer's first chunk
        load_ent(ent, qb0, qend - qb0);
        load_ent(ent1, qb0 + 2 * kQ, qend - qb0 - 2 * kQ);
        load_lse(vl, ent, qend - qb0);
        for (int m = pw; m < nch; m += 2) {
            const int s = m % kStages;
            const int q0 = qbeg + m * kQ;
            const int nq = min(kQ, qend - q0);
            load_ent(ent2, q0 + 4 * kQ, qend - q0 - 4 * kQ);
            if (m + 2 < nch) load_lse(vl_next, ent1, qend - q0 - 2 * kQ);
            if (!tc::mbar_wait(&empty[s], ((uint32_t)(m / kStages) & 1u) ^ 1u, st, 121, abort_flag)) break;
            Meta *meta = reinterpret_cast<Meta *>(sm + OFF_META + s * META_BYTES);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int qq = lane + 32 * t;
                const bool ok = qq < nq;
                const int i = ok ? entry_row(ent[t]) : 0;
                meta->lsei2[qq] = vl[t] * kLog2e;
                meta->qi[qq] = i;
                meta->pos[qq] = ok ? p.q_offset + i : -1;
                meta->slot[qq] = ok ? entry_slot(ent[t]) : 0;
            }
            if (lane == 0) {
                meta->e0 = q0;
                meta->nq = nq;
            }
            uint8_t *sq = sm + OFF_STG + s * (2 * SUB);
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
            for (int t = 0; t < 4; ++t) {
                ent[t] = ent1[t];
                ent1[t] = ent2[t];
                vl[t] = vl_next[t];
            }
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t I_S = tc::idesc_bf16(128, kQ);
            constexpr uint32_t I_DKI = tc::idesc_bf16(128, DI) | tc::kBMajorMN;
            constexpr uint32_t I_DQI = tc::idesc_bf16(128, kQ) | tc::kAMajorMN | tc::kBMajorMN;
            const uint32_t aKI = smem_u32(sm + OFF_KI), sg = smem_u32(sm + OFF_SIG);
            const uint64_t dKI = tc::sdesc_k128(aKI), dKIT = tc::sdesc_sw128(aKI, SUB, 1024);
            const uint64_t dSGT = tc::sdesc_sw128(sg, SUB, 1024), dSG = tc::sdesc_k128(sg);
            auto issue_s = [&](int n) {
                const uint64_t dQ = tc::sdesc_k128(smem_u32(sm + OFF_STG + (n % kStages) * (2 * SUB)));
#pragma unroll
                for (int ks = 0; ks < DI / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * SUB + (ks & 3) * 32;
                    tc::mma_bf16(tmem + TM_S + (n & 1) * kQ, tc::desc_adv(dKI, off), tc::desc_adv(dQ, off), I_S, ks > 0);
                }
                tc::mma_commit(&s_full[n & 1]);
            };
            auto issue_g = [&](int n) {
                const uint64_t dQm = tc::sdesc_sw128(smem_u32(sm + OFF_STG + (n % kStages) * (2 * SUB)), SUB, 1024);
                // dq_idx^T = K_idx^T dsig^T: both operands read MN-major; K = 128 keys
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    tc::mma_bf16(tmem + TM_DQI, tc::desc_adv(dKIT, ks * 2048), tc::desc_adv(dSGT, ks * 2048), I_DQI,
                                 ks > 0);
                tc::mma_commit(dq_full);
                // dK_idx += dsig^T q_idx: A K-major over queries, B = q_idx read MN-major; K = 128 queries
#pragma unroll
                for (int ks = 0; ks < kQ / 16; ++ks)
                    tc::mma_bf16(tmem + TM_DKI, tc::desc_adv(dSG, (ks >> 2) * SUB + (ks & 3) * 32),
                                 tc::desc_adv(dQm, ks * 2048), I_DKI, n > 0 || ks > 0);
                tc::mma_commit(&empty[n % kStages]);
                tc::mma_commit(g_free);
            };
            bool ok = tc::mbar_wait(kv_full, 0, st, 122, abort_flag);
            if (ok) {
                ok = tc::mbar_wait(&full[0], 0, st, 123, abort_flag);
                if (ok) {
                    tc::fence_proxy_async();
                    tc::fence_after_sync();
                    issue_s(0);
                }
            }
            for (int n = 0; ok && n < nch; ++n) {
                if (n + 1 < nch) {
                    const int m = n + 1;
                    if (!tc::mbar_wait(&full[m % kStages], (uint32_t)(m / kStages) & 1u, st, 124, abort_flag)) break;
                    if (m >= 2 && !tc::mbar_wait(&s_free[m & 1], ((uint32_t)(m >> 1) & 1u) ^ 1u, st, 125, abort_flag))
                        break;
                    tc::fence_proxy_async();
                    tc::fence_after_sync();
                    issue_s(m);
                }
                if (!tc::mbar_wait(g_full, (uint32_t)n & 1u, st, 126, abort_flag)) break;
                if (n >= 1 && !tc::mbar_wait(dq_free, (uint32_t)(n - 1) & 1u, st, 127, abort_flag)) break;
                tc::fence_after_sync();
                issue_g(n);
            }
            tc::mma_commit(done);
            tc::mbar_wait(done, 0, nullptr, 0, nullptr);
        }
    } else if (warp < kProd2) {
        // ------------------------------------------------ epilogue
        const int qd = warp & 3, hf = (warp - 2) >> 2;
        const int kr = qd * 32 + lane;              // key (s^T phase) or feature (dq_idx^T phase)
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const long long j = j0 + kr;
        const bool key_ok = j < p.Nk;
        const float si2 = p.scale_idx * kLog2e;
        const int cb = hf * kCols;                  // first query column of this warp
        long long rp_prev[kHalves];                 // partial rows of columns cb + 32 t + lane
#pragma unroll
        for (int t = 0; t < kHalves; ++t) rp_prev[t] = -1;
        bool ok = true;
        auto drain = [&](int m) -> bool {
            if (!wwait(dq_full, (uint32_t)m & 1u, st, 131, abort_flag)) return false;
            tc::fence_after_sync();
            uint32_t v[kHalves][32];
#pragma unroll
            for (int t = 0; t < kHalves; ++t) tc::tmem_ld32_nowait(tmem + lane_base + TM_DQI + cb + 32 * t, v[t]);
#pragma unroll
            for (int t = 0; t < kHalves; ++t) tc::tmem_wait32(v[t]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(dq_free);
            // transpose the warp's [32 features][kCols queries] block through shared
            // memory, then write 64 contiguous bytes per row with 16-byte stores
            uint8_t *stage = sm + OFF_STAGE + (warp - 2) * STAGE_BYTES;
#pragma unroll
            for (int t = 0; t < kHalves; ++t)
#pragma unroll
                for (int cc = 0; cc < 32; ++cc)
                    *reinterpret_cast<bf16 *>(stage + (32 * t + cc) * 64 + lane * 2) =
                        __float2bfloat16_rn(__uint_as_float(v[t][cc]));
            __syncwarp();
#pragma unroll
            for (int it = 0; it < kCols / 8; ++it) {
                const int row = it * 8 + (lane >> 2), q4 = lane & 3;
                const long long rix = __shfl_sync(0xffffffffu, rp_prev[it >> 2], row & 31);
                const uint4 x = *reinterpret_cast<const uint4 *>(stage + row * 64 + q4 * 16);
                if (rix >= 0) *reinterpret_cast<uint4 *>(dqi_part + rix * DI + qd * 32 + q4 * 8) = x;
            }
            __syncwarp();
            return true;
        };
        for (int n = 0; ok && n < nch; ++n) {
            const int s = n % kStages, sb = n & 1;
            const Meta *meta = reinterpret_cast<const Meta *>(sm + OFF_META + s * META_BYTES);
            if (!wwait(&full[s], (uint32_t)(n / kStages) & 1u, st, 132, abort_flag)) { ok = false; break; }
            const int nq = meta->nq;
            // the teacher of this key for entries 128n + cb .. + kCols-1: 8-entry
            // groups, 16 bytes each (padding entries beyond nq are masked below)
            uint4 tv[kCols / 8];
            {
                const __half *src = pt + ((long long)pt_off[bucket] + (long long)n * 128 + cb) * kKeys + kr * 8;
#pragma unroll
                for (int x = 0; x < kCols / 8; ++x)
                    tv[x] = __ldg(reinterpret_cast<const uint4 *>(src + (long long)x * 8 * kKeys));
            }
            if (!wwait(&s_full[sb], (uint32_t)(n >> 1) & 1u, st, 133, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t sv_[kHalves][32];
#pragma unroll
            for (int t = 0; t < kHalves; ++t) tc::tmem_ld32_nowait(tmem + lane_base + TM_S + sb * kQ + cb + 32 * t, sv_[t]);
            long long rp_cur[kHalves], kl_cur[kHalves];
#pragma unroll
            for (int t = 0; t < kHalves; ++t) {
                const int u = cb + 32 * t + lane;
                rp_cur[t] = u < nq ? (((long long)b * p.Nq + meta->qi[u]) * p.Hkv + r) * p.topk + meta->slot[u] : -1;
                kl_cur[t] = u < nq ? (((long long)b * p.Hkv + r) * p.Nq + meta->qi[u]) * p.topk + meta->slot[u] : -1;
            }
#pragma unroll
            for (int t = 0; t < kHalves; ++t) tc::tmem_wait32(sv_[t]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s_free[sb]);
            uint32_t sg[kCols / 2];
            // no per-element mask where every query of the warp's columns sees the whole block
            int pmin = meta->pos[cb + lane];
#pragma unroll
            for (int t = 1; t < kHalves; ++t) pmin = min(pmin, meta->pos[cb + 32 * t + lane]);
            pmin = __reduce_min_sync(0xffffffffu, pmin);
            const bool all_vis = (long long)pmin >= j0 + kKeys - 1 && j0 + kKeys <= p.Nk;
            const int ji = (int)min(j, (long long)INT_MAX);
            auto dsig_tile = [&](auto all_tag) {
                constexpr bool kAll = decltype(all_tag)::value;
#pragma unroll
                for (int t = 0; t < kHalves; ++t) {
                    [[maybe_unused]] float lv[6];   // streaming warp sum of Pt s log2(e) (KL partial)
#pragma unroll
                    for (int cc = 32 * t; cc < 32 * t + 32; cc += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(meta->lsei2 + cb + cc);
                        int ps[4] = {0, 0, 0, 0};
                        if constexpr (!kAll) {
                            const int4 p4 = *reinterpret_cast<const int4 *>(meta->pos + cb + cc);
                            ps[0] = p4.x;
                            ps[1] = p4.y;
                            ps[2] = p4.z;
                            ps[3] = p4.w;
                        }
                        const float l2[4] = {l4.x, l4.y, l4.z, l4.w};
                        float g2[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = cc + e;
                            const float sv = __uint_as_float(sv_[col >> 5][col & 31]);
                            const __half2 h2 = *reinterpret_cast<const __half2 *>(
                                reinterpret_cast<const uint32_t *>(&tv[col >> 3]) + ((col & 7) >> 1));
                            const float ptv = (col & 1) ? __high2float(h2) : __low2float(h2);
                            const float gv = coef * (tc::ex2(sv * si2 - l2[e]) - ptv);
                            [[maybe_unused]] const float bv = kKL ? ptv * (sv * si2) : 0.f;
                            if constexpr (kAll) {
                                g2[e] = gv;
                                if constexpr (kKL) colsum32_push(lv, bv, col & 31, lane);
                            } else {
                                const bool vis = key_ok && ji <= ps[e];
                                g2[e] = vis ? gv : 0.f;
                                if constexpr (kKL) colsum32_push(lv, vis ? bv : 0.f, col & 31, lane);
                            }
                        }
                        sg[cc / 2] = pack_bf16(g2[0], g2[1]);
                        sg[cc / 2 + 1] = pack_bf16(g2[2], g2[3]);
                    }
                    if constexpr (kKL) {
                        if (kl_cur[t] >= 0) klb[kl_cur[t] * 4 + qd] = lv[5];   // lane l: column cb + 32 t + l
                    }
                }
            };
            if (all_vis) dsig_tile(std::true_type{});
            else dsig_tile(std::false_type{});
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[s]);   // the stage's row data is no longer read
            if (n >= 1 && !wwait(g_free, (uint32_t)(n - 1) & 1u, st, 134, abort_flag)) { ok = false; break; }
            uint8_t *dst = sm + OFF_SIG + (cb >> 6) * SUB;           // 64-query sub-tile of column cb
            const int ch0 = (cb & 63) >> 3;                           // its first 16-byte chunk
#pragma unroll
            for (int ch = 0; ch < kCols / 8; ++ch)
                *reinterpret_cast<uint4 *>(dst + swz(kr, ch0 + ch)) =
                    make_uint4(sg[ch * 4], sg[ch * 4 + 1], sg[ch * 4 + 2], sg[ch * 4 + 3]);
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(g_full);
            if (n >= 1 && !drain(n - 1)) { ok = false; break; }
#pragma unroll
            for (int t = 0; t < kHalves; ++t) rp_prev[t] = rp_cur[t];
        }
        if (ok) ok = drain(nch - 1);
        if (ok) {
            const int m = nch - 1;
            ok = wwait(g_free, (uint32_t)m & 1u, st, 135, abort_flag);
            tc::fence_after_sync();
        }
        if (ok) {
            // dK_idx of this key, features cb .. cb+kCols-1 (the warp's column range doubles as its feature range)
#pragma unroll
            for (int h2 = 0; h2 < kHalves; ++h2) {
                uint32_t a[32];
                tc::tmem_ld32_nowait(tmem + lane_base + TM_DKI + cb + h2 * 32, a);
                tc::tmem_wait32(a);
                if (key_ok) {
                    float *dst = dki_acc + ((long long)b * p.Nk + j) * DI + cb + h2 * 32;
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        tc::red_add_v4(dst + x, __uint_as_float(a[x]), __uint_as_float(a[x + 1]),
                                       __uint_as_float(a[x + 2]), __uint_as_float(a[x + 3]));
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

}  // namespace

cudaError_t launch_bwd_index_tc(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, const float *lse_idx,
                                float kl_coef, const BwdWork &w, DeviceStatus *st, cudaStream_t s)
{
    auto kern = w.klb ? bwd_index_tc_kernel<true> : bwd_index_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tki;
    const unsigned long long di[3] = {(unsigned long long)DI, (unsigned long long)p.Nk, (unsigned long long)p.B};
    const unsigned long long si[2] = {DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull};
    const unsigned bi[3] = {64, (unsigned)kKeys, 1};
    if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    const float coef = p.scale_idx * kl_coef / ((float)p.B * (float)p.Nq * (float)p.Hkv);
    {
        TimedLaunch timed_("bwd_index_tc_kernel", s);
        kern<<<dim3(p.Hkv, p.nb, p.B), kThreads, ALLOC, s>>>(tki, p, q_idx, lse_idx, coef, w.bucket_off,
                                                                           w.bucket_q, w.pt, w.pt_off, w.dqi_part, w.dki_acc,
                                                                           w.klb, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
