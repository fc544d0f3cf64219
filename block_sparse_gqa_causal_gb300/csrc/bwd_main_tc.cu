// bwd_main_tc.cu -- main-branch backward of MSA on the tcgen05 tensor cores,
// key-major.  The tiles hold 128 features; at d = 64 the upper 64 are zeros
// (TMA fills the boxes past the tensor's width, gathers zero-fill them), which
// add nothing to any product, and are never written back.
//
// "Sparse Attention · Part II", section 3.2: the main branch's gradients come
// from dO alone (the selection is not differentiated).  One CTA owns one
// 128-key block c of one (b, group r) and walks the queries that selected c
// (the inverse index) in chunks of 64 (query, head) rows.  With the keys as
// the MMA's M dimension, per chunk:
//   S^T = K Q^T,  dP^T = V dO^T                   (M = 128 keys, N = 64 rows)
//   P = exp2(S*scale*log2e - lse*log2e) on the keys each row may see,
//   dS = scale * P (dP - D),  D = rowsum(dO * O)   (the softmax scale folded in)
//   dQ^T = K^T dS^T                                (M = 128 features, N = 64 rows)
//   dV += P^T dO,  dK += dS^T Q                    (M = 128 keys, N = 128 features)
// dV and dK stay in TMEM for the whole bucket and are written once (one
// owner, no atomics).  A chunk's dQ leaves as one bf16 partial row per
// (query, head, slot); a combine kernel sums a row's slots (the split-KV
// pattern of the forward).  The KL's teacher and the index branch's backward
// are computed elsewhere (index_teacher_tc.cu) from their own logit tiles, so
// no probability distribution leaves this kernel.
//
// Roles: warps 0 and 11 load (TMA; alternate chunks), warp 1 owns TMEM and
// issues the score MMAs, warp 10 the gradient MMAs, warps 2..9 are the
// epilogue: warp w serves TMEM lanes 32*(w%4).. (keys) and column half
// (w-2)/4 of the chunk's 64 rows.  Warps 12..15 drain dQ^T (lanes are
// features) into the partial rows, off the epilogue's critical loop; the
// epilogue hands them each chunk's partial-row indices through a small ring.
// TMEM holds dV, dK and two 128-column slots; chunk n uses slot n%2 for S^T
// and dP^T.  The epilogue writes P^T and dS^T (bf16) back over the S^T half,
// where the dV and dK MMAs read them as their A operand; dQ^T then
// overwrites that half (issued after dV, dK by the same thread, so in
// order).  dS^T also goes to shared memory (double-buffered), the B operand
// of dQ^T.  The slot is free again once the drain has read dQ^T, so the
// scores of chunk n+1 run while the epilogue works on chunk n.
#include <cuda_fp16.h>

#include <type_traits>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int D = 128;
constexpr int kKeys = 128;
constexpr int kRows = 64;                       // (query, head) rows per chunk
constexpr int kEpiWarps = 8;
constexpr int kGradWarp = 2 + kEpiWarps;         // the second MMA issuer (gradients)
constexpr int kProd2 = 3 + kEpiWarps;            // second producer warp: the two take alternate chunks
constexpr int kDrainWarps = 4;                   // dQ^T drain: warps 4+kEpiWarps .. (one per TMEM lane quarter)
constexpr int kThreads = 32 * (4 + kEpiWarps + kDrainWarps);
constexpr int kRx = 4;                           // ring of chunk partial-row index lists
constexpr int SUBK = kKeys * 128;               // [128 keys][64 bf16] swizzled sub-tile
// A [64 rows][128 d] tile is stored as 8-row groups of {d 0..63, d 64..127}
// (1024-byte swizzle atoms): row rho, half h at (rho/8)*2048 + h*1024 + (rho%8)*128.
// With groups of 8 heads one query's rows form one group, which one TMA box fills.
constexpr int TILE_R = kRows * D * 2;
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + 2 * SUBK;
constexpr int kStages = 3;                      // Q/dO stages
constexpr int kDsBuf = 2;                       // dS^T tile buffers (shared memory)
constexpr int OFF_STG = OFF_V + 2 * SUBK;       // kStages x {Q, dO}
constexpr int STG_BYTES = 2 * TILE_R;
constexpr int OFF_DS = OFF_STG + kStages * STG_BYTES;  // dS^T [128 keys][64 rows] per buffer
constexpr int OFF_META = OFF_DS + kDsBuf * SUBK;

struct Meta {                 // per stage
    float lse2[kRows];        // lse * log2(e) of each row (+inf for padding)
    float dd[kRows];          // scale * rowsum(dO * O)
    int pos[kRows];           // position of each query slot (-1 for padding)
    int qi[kRows];            // query index
    int slot[kRows];          // slot of this block in the query's selection
    int e0;                   // bucket-list index of the chunk's first entry
    int nq;                   // queries in the chunk
};
constexpr int META_BYTES = (int)((sizeof(Meta) + 127) & ~size_t(127));
constexpr int OFF_RIDX = OFF_META + kStages * META_BYTES;    // kRx x [64 rows] partial-row index (-1: padding)
constexpr int OFF_BAR = OFF_RIDX + kRx * kRows * 8;
constexpr int ALLOC = OFF_BAR + 256 + 1024;

// slot a: S^T at TM_SLOT + 128a (then P^T, dS^T: warp half hf writes its 32
// rows' P^T at columns 32hf..32hf+15 and dS^T at 32hf+16.., packed bf16;
// then dQ^T), dP^T 64 columns above it
constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_SLOT = 256, TM_DP_OFF = 64;

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }
__device__ __forceinline__ int roff(int rho, int half, int ch)
{
    return (rho >> 3) * 2048 + half * 1024 + (rho & 7) * 128 + (((ch ^ rho) & 7) << 4);
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait whose outcome is the same on every lane of the warp, so the
// warp-collective TMEM loads that follow are never split.
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

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_do,
                   const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v, Problem p,
                   const bf16 *__restrict__ q, const bf16 *__restrict__ d_o, const float *__restrict__ lse,
                   const float *__restrict__ Dg, const int32_t *__restrict__ bucket_off,
                   const int32_t *__restrict__ bucket_q, bf16 *__restrict__ dk, bf16 *__restrict__ dv,
                   bf16 *__restrict__ dq_part, DeviceStatus *st)
{
    constexpr int QC = kRows / G;                 // queries per chunk
    constexpr int EPL = (QC + 31) / 32;           // bucket entries per producer lane
    // the (group, block) bucket of this CTA (visiting order: bucket_of)
    int r, c;
    bucket_of((int)blockIdx.x, p.Hkv, p.nb, p.num_sms, r, c);
    const int b = blockIdx.y;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    const int nch = (qend - qbeg + QC - 1) / QC;
    const long long j0 = (long long)c * kKeys;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + 3, *p_full = bars + 6, *ds_free = bars + 8;   // p_full, ds_free: 2 each
    uint64_t *dq_full = bars + 10, *slot_free = bars + 12;
    uint64_t *kv_full = bars + 14, *s_full = bars + 15, *done = bars + 17;   // s_full: 2 (one per slot)
    uint64_t *rx_full = bars + 18, *rx_free = bars + 18 + kRx;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 18 + 2 * kRx);
    long long *ridx_ring = reinterpret_cast<long long *>(sm + OFF_RIDX);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < kStages; ++a) {
            // G == 8: lane 0's expect_tx arrival + 32 row-data arrivals;
            // otherwise 32 cp.async arrivals + 32 row-data arrivals
            tc::mbar_init(&full[a], G == 8 ? 33 : 64);
            tc::mbar_init(&empty[a], 1 + kEpiWarps);   // grads MMAs done + epilogue has read the row data
        }
        for (int a = 0; a < kDsBuf; ++a) {
            tc::mbar_init(&p_full[a], kEpiWarps);
            tc::mbar_init(&ds_free[a], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&dq_full[a], 1);
            tc::mbar_init(&slot_free[a], kDrainWarps);
        }
        for (int a = 0; a < kRx; ++a) {
            tc::mbar_init(&rx_full[a], 2);              // the two epilogue warps of lane quarter 0
            tc::mbar_init(&rx_free[a], kDrainWarps);
        }
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(done, 2);                        // both MMA issuers
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
        // K and V tiles by TMA; rows past Nk read as zeros
        const int pw = warp == 0 ? 0 : 1;
        if (pw == 0 && lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::prefetch_tmap(&tmap_do);
            tc::mbar_arrive_expect_tx(kv_full, 4 * SUBK);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc::tma_load_4d(sm + OFF_K + h * SUBK, &tmap_k, kv_full, h * 64, r, (int)j0, b);
                tc::tma_load_4d(sm + OFF_V + h * SUBK, &tmap_v, kv_full, h * 64, r, (int)j0, b);
            }
        }
        // Entries run two chunks ahead and the rows' LSE and D one chunk ahead,
        // so no load is waited for on the way to the next stage.
        auto load_rows = [&](float (&vl)[2], float (&vd)[2], const int (&e_)[EPL], int nqx) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int rho = lane + 32 * t, qq = rho / G, g = rho % G;
                int e = 0;
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    const int x = __shfl_sync(0xffffffffu, e_[u], qq & 31);
                    if ((qq >> 5) == u) e = x;
                }
                const bool ok = qq < nqx;
                const long long hi = ((long long)b * p.Hq + r * G + g) * p.Nq + entry_row(e);
                vl[t] = ok ? __ldg(lse + hi) : INFINITY;
                vd[t] = ok ? __ldg(Dg + hi) : 0.f;
            }
        };
        int ent[EPL], ent1[EPL], ent2[EPL];
        const int qb0 = qbeg + pw * QC;              // this producer's first chunk
        load_entries(ent, bucket_q, qb0, min(QC, qend - qb0), lane);
        load_entries(ent1, bucket_q, qb0 + 2 * QC, min(QC, qend - qb0 - 2 * QC), lane);
        float vl[2], vd[2], vl_next[2], vd_next[2];
        load_rows(vl, vd, ent, min(QC, qend - qb0));
        for (int m = pw; m < nch; m += 2) {
            const int s = m % kStages;
            const int q0 = qbeg + m * QC;
            const int nq = min(QC, qend - q0);
            load_entries(ent2, bucket_q, q0 + 4 * QC, min(QC, qend - q0 - 4 * QC), lane);
            if (m + 2 < nch) load_rows(vl_next, vd_next, ent1, min(QC, qend - q0 - 2 * QC));
            if constexpr (G == 8) {
                // the Q and dO rows of this producer's next chunk (m + 2) into L2 while
                // this one waits for its stage, so its gathers do not wait on HBM
                if (lane < min(QC, qend - q0 - 2 * QC)) {
                    const int z2 = b * p.Nq + entry_row(ent1[0]);
                    tc::tma_prefetch_4d(&tmap_q, 0, r * G, 0, z2);
                    tc::tma_prefetch_4d(&tmap_do, 0, r * G, 0, z2);
                }
            }
            if (!tc::mbar_wait(&empty[s], ((uint32_t)(m / kStages) & 1u) ^ 1u, st, 101, abort_flag)) break;
            Meta *meta = reinterpret_cast<Meta *>(sm + OFF_META + s * META_BYTES);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                meta->lse2[lane + 32 * t] = vl[t] * kLog2e;
                meta->dd[lane + 32 * t] = vd[t] * p.scale;
            }
#pragma unroll
            for (int t = 0; t < EPL; ++t) {
                const int qq = lane + 32 * t;
                if (qq < QC) {
                    const bool ok = qq < nq;
                    const int i = ok ? entry_row(ent[t]) : 0;
                    meta->qi[qq] = i;
                    meta->pos[qq] = ok ? p.q_offset + i : -1;
                    meta->slot[qq] = ok ? entry_slot(ent[t]) : 0;
                }
            }
            if (lane == 0) {
                meta->e0 = q0;
                meta->nq = nq;
            }
            __syncwarp();
            uint8_t *sq = sm + OFF_STG + s * STG_BYTES, *sdo = sq + TILE_R;
            if constexpr (G == 8) {
                // one TMA box {64 features, 8 heads, 2 halves} per query and
                // tensor fills one 2048-byte row group; padding slots read
                // rows past the end (zero fill)
                if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * TILE_R);
                __syncwarp();
                if (lane < QC) {
                    const int z = lane < nq ? b * p.Nq + entry_row(ent[0]) : p.B * p.Nq;
                    tc::tma_load_4d(sq + lane * 2048, &tmap_q, &full[s], 0, r * G, 0, z);
                    tc::tma_load_4d(sdo + lane * 2048, &tmap_do, &full[s], 0, r * G, 0, z);
                }
            } else {
                // 64 rows x 16 chunks per tensor: lane covers chunk lane%16 of rows 2*it + lane/16
#pragma unroll 4
                for (int it = 0; it < kRows / 2; ++it) {
                    const int rho = it * 2 + (lane >> 4), ch = lane & 15;
                    const int qq = rho / G, g = rho % G;
                    const bool ok = qq < nq && ch * 8 < p.d;
                    const long long off =
                        (((long long)b * p.Nq + meta->qi[qq]) * p.Hq + (long long)r * G + g) * p.d + (ok ? ch * 8 : 0);
                    const int o = roff(rho, ch >> 3, ch & 7);
                    cp_async16_zfill(sq + o, q + off, ok);
                    cp_async16_zfill(sdo + o, d_o + off, ok);
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
            for (int t = 0; t < 2; ++t) {
                vl[t] = vl_next[t];
                vd[t] = vd_next[t];
            }
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer (the whole warp
            // runs the loop; one lane chosen by elect.sync issues)
            constexpr uint32_t I_S = tc::idesc_bf16(128, kRows);
            const uint64_t dK = tc::sdesc_k128(smem_u32(sm + OFF_K)), dV = tc::sdesc_k128(smem_u32(sm + OFF_V));
            auto issue_scores = [&](int n) {
                // B = Q / dO rows (K-major, 8-row groups 2048 bytes apart)
                const uint32_t sq = smem_u32(sm + OFF_STG + (n % kStages) * STG_BYTES);
                const uint64_t dQ = tc::sdesc_sw128(sq, 16, 2048), dDO = tc::sdesc_sw128(sq + TILE_R, 16, 2048);
                const uint32_t ts = tmem + TM_SLOT + (n & 1) * 128;
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                        tc::mma_bf16(ts, tc::desc_adv(dK, h * SUBK + ko), tc::desc_adv(dQ, h * 1024 + ko), I_S, ks > 0);
                        tc::mma_bf16(ts + TM_DP_OFF, tc::desc_adv(dV, h * SUBK + ko), tc::desc_adv(dDO, h * 1024 + ko),
                                     I_S, ks > 0);
                    }
                    tc::mma_commit(&s_full[n & 1]);
                }
                __syncwarp();
            };
            // Scores here, gradients on warp kGradWarp: the two streams touch
            // disjoint TMEM and shared memory, are ordered only through the
            // mbarriers, and issuing them from two threads overlaps their issue.
            bool ok = wwait(kv_full, 0, st, 102, abort_flag);
            if (ok) tc::fence_proxy_async();
            for (int ns = 0; ok && ns < nch; ++ns) {
                if (!wwait(&full[ns % kStages], (uint32_t)(ns / kStages) & 1u, st, 103, abort_flag)) break;
                // the slot's previous chunk (ns-2) has had its dQ^T drained
                if (ns >= 2 && !wwait(&slot_free[ns & 1], (uint32_t)((ns >> 1) - 1) & 1u, st, 104, abort_flag))
                    break;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                issue_scores(ns);
            }
            // every MMA this warp issued has completed once `done` fires (it also
            // waits for the gradient issuer's commit)
            if (tc::elect_one()) tc::mma_commit(done);
            __syncwarp();
            tc::mbar_wait(done, 0, nullptr, 0, nullptr);
        }
    } else if (warp == kGradWarp) {
        {
            // ------------------------------------------------ MMA issuer: gradients (warp-uniform,
            // one elected lane issues)
            constexpr uint32_t I_DKV = tc::idesc_bf16(128, 128) | tc::kBMajorMN;
            constexpr uint32_t I_DQ = tc::idesc_bf16(128, kRows) | tc::kAMajorMN | tc::kBMajorMN;
            const uint64_t dKT = tc::sdesc_sw128(smem_u32(sm + OFF_K), SUBK, 1024);
            const uint64_t dDST0 = tc::sdesc_sw128(smem_u32(sm + OFF_DS), SUBK, 1024);
            auto issue_grads = [&](int n) {
                const int db = n % kDsBuf;
                const uint32_t ts = tmem + TM_SLOT + (n & 1) * 128;
                const uint32_t sq = smem_u32(sm + OFF_STG + (n % kStages) * STG_BYTES);
                const uint64_t dQm = tc::sdesc_sw128(sq, 1024, 2048), dDOm = tc::sdesc_sw128(sq + TILE_R, 1024, 2048);
                // dV += P^T dO, dK += dS^T Q: A = P^T / dS^T from the slot (rows 16ks..
                // of the K dimension: warp half ks/2, 8 packed columns per step), B =
                // dO / Q read MN-major (feature halves 1024 bytes apart, 8-row groups
                // 2048 apart); K = 64 rows
                // dQ^T = K^T dS^T over the slot's S^T half (in order after the MMAs
                // below have read it): A = K read MN-major (64-feature atoms SUBK
                // apart), B = dS^T [keys][rows] MN-major; K = 128 keys
                const uint64_t dDST = tc::desc_adv(dDST0, db * SUBK);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < kRows / 16; ++ks) {
                        const bool acc = n > 0 || ks > 0;
                        const uint32_t col = (ks >> 1) * 32 + (ks & 1) * 8;
                        tc::mma_bf16_ts(tmem + TM_DV, ts + col, tc::desc_adv(dDOm, ks * 4096), I_DKV, acc);
                        tc::mma_bf16_ts(tmem + TM_DK, ts + col + 16, tc::desc_adv(dQm, ks * 4096), I_DKV, acc);
                    }
                    tc::mma_commit(&empty[n % kStages]);
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks)
                        tc::mma_bf16(ts, tc::desc_adv(dKT, ks * 2048), tc::desc_adv(dDST, ks * 2048), I_DQ, ks > 0);
                    tc::mma_commit(&dq_full[n & 1]);
                    tc::mma_commit(&ds_free[db]);
                }
                __syncwarp();
            };
            bool ok = wwait(kv_full, 0, st, 105, abort_flag);
            for (int ng = 0; ok && ng < nch; ++ng) {
                if (!wwait(&p_full[ng % kDsBuf], (uint32_t)(ng / kDsBuf) & 1u, st, 106, abort_flag)) break;
                tc::fence_after_sync();
                issue_grads(ng);
            }
            if (tc::elect_one()) tc::mma_commit(done);
            __syncwarp();
        }
    } else if (warp >= 4 + kEpiWarps) {
        // ------------------------------------------------ dQ^T drain: features 32*qd.. of all 64 rows
        const int qd = warp & 3;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        // lanes 2m, 2m+1 trade values so that each lane holds features (2m, 2m+1)
        // of one row of a row pair: lane 2m row 2t, lane 2m+1 row 2t+1; one
        // 4-byte store per lane writes two rows' 64 contiguous bytes each
        const int fpair = qd * 32 + (lane & ~1);          // this lane's first feature
        const int odd = lane & 1;
        auto store_rows = [&](auto dw_tag, const long long *rx, const uint32_t (&v)[32], int r0) {
            constexpr int DW = decltype(dw_tag)::value;
            const bool feat_ok = fpair < DW;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                // rows r0 + 2t (even lanes) and r0 + 2t + 1 (odd lanes)
                // even lane: keeps row 2t of its feature, gives row 2t+1; odd lane: keeps
                // row 2t+1, gives row 2t
                const float ev = __uint_as_float(v[2 * t]), od = __uint_as_float(v[2 * t + 1]);
                const float mine = odd ? od : ev, give = odd ? ev : od;
                const float other = __shfl_xor_sync(0xffffffffu, give, 1);
                const float lo = odd ? other : mine, hi = odd ? mine : other;
                const long long row = rx[r0 + 2 * t + odd];
                if (feat_ok && row >= 0)
                    *reinterpret_cast<uint32_t *>(dq_part + row * DW + fpair) = pack_bf16(lo, hi);
            }
        };
        for (int m = 0; m < nch; ++m) {
            const int pb = m & 1, x = m % kRx;
            if (!wwait(&rx_full[x], (uint32_t)(m / kRx) & 1u, st, 117, abort_flag)) break;
            if (!wwait(&dq_full[pb], (uint32_t)(m >> 1) & 1u, st, 111, abort_flag)) break;
            tc::fence_after_sync();
            uint32_t v0[32], v1[32];
            tc::tmem_ld32_nowait(tmem + lane_base + TM_SLOT + pb * 128, v0);
            tc::tmem_ld32_nowait(tmem + lane_base + TM_SLOT + pb * 128 + 32, v1);
            tc::tmem_wait32(v0);
            tc::tmem_wait32(v1);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&slot_free[pb]);
            const long long *rx = ridx_ring + x * kRows;
            if (p.d == 128) {
                store_rows(std::integral_constant<int, 128>{}, rx, v0, 0);
                store_rows(std::integral_constant<int, 128>{}, rx, v1, 32);
            } else {
                store_rows(std::integral_constant<int, 64>{}, rx, v0, 0);
                store_rows(std::integral_constant<int, 64>{}, rx, v1, 32);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&rx_free[x]);
        }
    } else if (warp < kGradWarp) {
        // ------------------------------------------------ epilogue
        const int qd = warp & 3, hf = (warp - 2) >> 2;
        const int kr = qd * 32 + lane;             // key (S/dP/P/dS phase) or feature (dQ phase)
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const long long j = j0 + kr;
        const bool key_ok = j < p.Nk;
        const float sl2 = p.scale * kLog2e;
        constexpr int NQH = 32 / G;                // query slots among this warp's 32 columns
        const int cb = hf * 32;                    // first column (row of the chunk) of this warp
        bool ok = true;
        for (int n = 0; ok && n < nch; ++n) {
            const int s = n % kStages, db = n % kDsBuf;
            const Meta *meta = reinterpret_cast<const Meta *>(sm + OFF_META + s * META_BYTES);
            if (!wwait(&full[s], (uint32_t)(n / kStages) & 1u, st, 112, abort_flag)) { ok = false; break; }
            if (!wwait(&s_full[n & 1], (uint32_t)(n >> 1) & 1u, st, 113, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t sv[32], dp[32];
            const uint32_t ts = tmem + lane_base + TM_SLOT + (n & 1) * 128 + cb;
            tc::tmem_ld32_nowait(ts, sv);
            tc::tmem_ld32_nowait(ts + TM_DP_OFF, dp);
            // row data while the loads land (LSE and D are read in the loop below)
            int pos[NQH];
#pragma unroll
            for (int u = 0; u < NQH; ++u) pos[u] = meta->pos[cb / G + u];
            const int nq = meta->nq;
            long long ridx_cur;
            {
                const int rho = cb + lane, qq = rho / G, g = rho % G;
                ridx_cur = qq < nq ? ((((long long)b * p.Nq + meta->qi[qq]) * p.Hq + (long long)r * G + g) * p.topk +
                                      meta->slot[qq])
                                   : -1;
            }
            tc::tmem_wait32(sv);
            tc::tmem_wait32(dp);
            // P^T, dS^T of this key against the warp's 32 rows.  The mask is
            // needed only where some row of the warp does not see the whole block
            // (a bucket's local-block queries, its padded tail, the last block)
            uint32_t pk[16], dk2[16];
            int lim[NQH];                              // last visible key offset per query (-1: none)
            int minpos = pos[0];
#pragma unroll
            for (int u = 0; u < NQH; ++u) {
                minpos = min(minpos, pos[u]);
                lim[u] = (int)max(-1LL, min(min((long long)pos[u], (long long)p.Nk - 1) - j0, (long long)kKeys - 1));
            }
            const bool all_vis = (long long)minpos >= j0 + kKeys - 1 && j0 + kKeys <= p.Nk;
            auto softmax_grad = [&](auto all_tag) {
                constexpr bool kAll = decltype(all_tag)::value;
#pragma unroll
                for (int cc = 0; cc < 32; cc += 2) {
                    float pr[2], ds[2];
                    const float2 l2 = *reinterpret_cast<const float2 *>(meta->lse2 + cb + cc);
                    const float2 dd = *reinterpret_cast<const float2 *>(meta->dd + cb + cc);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = cc + e, u = col / G;
                        const float x = tc::ex2(__uint_as_float(sv[col]) * sl2 - (e ? l2.y : l2.x));
                        if constexpr (kAll) pr[e] = x;
                        else pr[e] = kr <= lim[u] ? x : 0.f;
                        // dS carries the softmax scale, so dQ and dK need no rescaling
                        ds[e] = pr[e] * fmaf(__uint_as_float(dp[col]), p.scale, -(e ? dd.y : dd.x));
                    }
                    pk[cc / 2] = pack_bf16(pr[0], pr[1]);
                    dk2[cc / 2] = pack_bf16(ds[0], ds[1]);
                }
            };
            if (all_vis) softmax_grad(std::true_type{});
            else softmax_grad(std::false_type{});
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[s]);   // done with the stage's row data
            // P^T and dS^T over this warp's own S^T columns (read above) for the dV / dK MMAs
            tc::tmem_st16(ts, pk);
            tc::tmem_st16(ts + 16, dk2);
            if (n >= kDsBuf && !wwait(&ds_free[db], (uint32_t)((n - kDsBuf) / kDsBuf) & 1u, st, 114, abort_flag)) {
                ok = false;
                break;
            }
            if (qd == 0) {
                // this chunk's partial-row indices for the dQ drain
                if (n >= kRx && !wwait(&rx_free[n % kRx], (uint32_t)((n / kRx) - 1) & 1u, st, 116, abort_flag)) {
                    ok = false;
                    break;
                }
                ridx_ring[(n % kRx) * kRows + cb + lane] = ridx_cur;
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&rx_full[n % kRx]);
            }
            uint8_t *sd = sm + OFF_DS + db * SUBK;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int ch = hf * 4 + c4;
                *reinterpret_cast<uint4 *>(sd + swz(kr, ch)) =
                    make_uint4(dk2[c4 * 4], dk2[c4 * 4 + 1], dk2[c4 * 4 + 2], dk2[c4 * 4 + 3]);
            }
            tc::fence_proxy_async();
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&p_full[db]);
        }
        // ---- dK, dV of this key (this warp: features hf*64 .. hf*64+63)
        if (ok && nch > 0) {
            // the last chunk's buffer release follows every MMA of the bucket
            const int m = nch - 1;
            ok = wwait(&ds_free[m % kDsBuf], (uint32_t)(m / kDsBuf) & 1u, st, 115, abort_flag);
            tc::fence_after_sync();
        }
        if (ok && hf * 64 < p.d) {
            bf16 *pk_ = dk + (((long long)b * p.kv_rows + j) * p.Hkv + r) * p.d + hf * 64;
            bf16 *pv_ = dv + (((long long)b * p.kv_rows + j) * p.Hkv + r) * p.d + hf * 64;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t a[32], g2[32];
                if (nch > 0) {
                    tc::tmem_ld32_nowait(tmem + lane_base + TM_DV + hf * 64 + h2 * 32, a);
                    tc::tmem_ld32_nowait(tmem + lane_base + TM_DK + hf * 64 + h2 * 32, g2);
                    tc::tmem_wait32(a);
                    tc::tmem_wait32(g2);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) a[x] = g2[x] = 0u;
                }
                if (key_ok) {
#pragma unroll
                    for (int x = 0; x < 32; x += 8) {
                        *reinterpret_cast<uint4 *>(pv_ + h2 * 32 + x) = make_uint4(
                            pack_bf16(__uint_as_float(a[x]), __uint_as_float(a[x + 1])),
                            pack_bf16(__uint_as_float(a[x + 2]), __uint_as_float(a[x + 3])),
                            pack_bf16(__uint_as_float(a[x + 4]), __uint_as_float(a[x + 5])),
                            pack_bf16(__uint_as_float(a[x + 6]), __uint_as_float(a[x + 7])));
                        *reinterpret_cast<uint4 *>(pk_ + h2 * 32 + x) = make_uint4(
                            pack_bf16(__uint_as_float(g2[x]), __uint_as_float(g2[x + 1])),
                            pack_bf16(__uint_as_float(g2[x + 2]), __uint_as_float(g2[x + 3])),
                            pack_bf16(__uint_as_float(g2[x + 4]), __uint_as_float(g2[x + 5])),
                            pack_bf16(__uint_as_float(g2[x + 6]), __uint_as_float(g2[x + 7])));
                    }
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
                     const BwdWork &w, bf16 *dk, bf16 *dv, DeviceStatus *st, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(bwd_main_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tdo, tk, tv;
    {
        // Q / dO as {d within a half, head, half, query row}: one box {64, G, 2, 1}
        // is a query's G head rows in both feature halves (at d = 64 the second
        // half lies past the tensor and reads as zeros)
        const unsigned long long dq4[4] = {64, (unsigned long long)p.Hq, (unsigned long long)p.d / 64,
                                           (unsigned long long)p.B * p.Nq};
        const unsigned long long sq4[3] = {p.d * 2ull, 128ull, (unsigned long long)p.Hq * p.d * 2ull};
        const unsigned bq4[4] = {64, (unsigned)G, 2, 1};
        if ((e = make_tmap_bf16(&tq, q, 4, dq4, sq4, bq4)) != cudaSuccess) return e;
        if ((e = make_tmap_bf16(&tdo, d_o, 4, dq4, sq4, bq4)) != cudaSuccess) return e;
        // K/V as [B][Nk][Hkv][d] (rows past Nk, and features past d, are out of bounds)
        const unsigned long long dk4[4] = {(unsigned long long)p.d, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                           (unsigned long long)p.B};
        const unsigned long long sk[3] = {p.d * 2ull, (unsigned long long)p.Hkv * p.d * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * p.d * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk4, sk, bk)) != cudaSuccess) return e;
        if ((e = make_tmap_bf16(&tv, v, 4, dk4, sk, bk)) != cudaSuccess) return e;
    }
    {
        TimedLaunch timed_("bwd_main_tc_kernel", s);
        bwd_main_tc_kernel<G><<<dim3(p.Hkv * p.nb, p.B), kThreads, ALLOC, s>>>(
            tq, tdo, tk, tv, p, q, d_o, lse, w.D, w.bucket_off, w.bucket_q, dk, dv, w.dq_part, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_tc(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *d_o,
                               const float *lse, const BwdWork &w, bf16 *dk, bf16 *dv, DeviceStatus *st,
                               cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_g<1>(p, q, k, v, d_o, lse, w, dk, dv, st, s);
    case 2: return launch_g<2>(p, q, k, v, d_o, lse, w, dk, dv, st, s);
    case 4: return launch_g<4>(p, q, k, v, d_o, lse, w, dk, dv, st, s);
    default: return launch_g<8>(p, q, k, v, d_o, lse, w, dk, dv, st, s);
    }
}

}  // namespace msa
