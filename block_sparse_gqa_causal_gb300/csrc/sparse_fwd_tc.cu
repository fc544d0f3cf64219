// sparse_fwd_tc.cu -- main branch of MSA, key-major on the tcgen05 tensor cores.
//
// "Sparse Attention · Part II", section 3.2: each query head of a group
// attends, with its own logits, to the visible tokens of the blocks selected
// for (query, group), normalised over that set only.  Selection is per query,
// so neighbouring queries pick mostly different blocks; gathering K/V per
// query would move K+V of 16 blocks for every (query, group).  Instead the
// work is grouped by key block (the varlen view of block-sparse attention
// the MSA training-kernel write-up borrows from MoBA): one CTA keeps one
// 128-token K/V block of one group on chip and runs full 128 x 128 tiles over
// the (query, head) rows of every query that selected it:
//   S = Q K^T (M = 128 rows, N = 128 keys),  P = exp2(S - m) (row max m),
//   O_c = P V (unnormalised),  z = rowsum(P)
// and writes O_c (bf16) with (m, z) for that (query, head, slot).  A combine
// kernel then merges a row's slots exactly like a split-KV flash decode:
//   M = max m_c,  O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) z_c,
//   lse = (M + log2 sum_c 2^(m_c - M) z_c) ln 2.
//
// Roles: warps 0 and 10 load (alternate chunks), warp 1 owns TMEM and issues
// the MMAs, warps 2..9 (two warpgroups on alternate chunks, one row per
// thread) do the softmax and write the partials.  S and O accumulators are
// double-buffered in TMEM; P (bf16) is written back over its own S columns
// and read from there as the A operand of the O MMA, so P never touches
// shared memory (an S MMA into that buffer is issued only after the O MMA
// that reads it, and MMAs of one thread run in order).
#include <type_traits>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kRows = 128;                  // (query, head) rows per chunk
constexpr int kKeys = 128;
constexpr int kEpiWarps = 8;                // two warpgroups, taking alternate chunks
constexpr int kWgWarps = 4;
constexpr int kProd2 = 2 + kEpiWarps;        // second producer warp: the two take alternate chunks
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr int SUB = 128 * 128;              // [128 rows][64 bf16] swizzled sub-tile

template <int D>
struct FwdLayout {
    static constexpr int KB = D / 64;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KB * SUB;
    // Q stage: [128 rows][D] as 8-row groups of KB feature halves (1024-byte
    // swizzle atoms): row rho, half h at (rho/8)*KB*1024 + h*1024 + (rho%8)*128
    static constexpr int OFF_Q = OFF_V + KB * SUB;          // 2 stages x KB sub-tiles
    static constexpr int OFF_P = OFF_Q + 2 * KB * SUB;      // 2 x output staging [128 rows][D] bf16
    static constexpr int OFF_META = OFF_P + 2 * 2 * SUB;    // 2 stages x QueryMeta
    static constexpr int OFF_BAR = OFF_META + 2 * 2048;
    static constexpr int ALLOC = OFF_BAR + 256 + 1024;
    static constexpr uint32_t TM_S = 0;                     // 2 x 128 columns
    static constexpr uint32_t TM_O = 256;                   // 2 x D columns
};

struct QueryMeta {         // per chunk, per query slot of the chunk (<= 128 queries)
    int i[kRows];          // query index
    int pos[kRows];        // absolute position
    int slot[kRows];       // position of this block in the query's selection
    int nq;
};

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

// Bounded wait with the same outcome on every lane (warp-collective TMEM
// loads follow).
__device__ __forceinline__ bool wwait(uint64_t *bar, uint32_t parity, DeviceStatus *st, int site,
                                      volatile int *abort_flag)
{
    const bool r = tc::mbar_wait(bar, parity, st, site, abort_flag);
    return __all_sync(0xffffffffu, r);
}

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

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
sparse_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, Problem p, const bf16 *__restrict__ q,
                     const int32_t *__restrict__ bucket_off,
                     const int32_t *__restrict__ bucket_q, bf16 *__restrict__ part, float2 *__restrict__ stats,
                     DeviceStatus *st)
{
    using L = FwdLayout<D>;
    constexpr int QPC = kRows / G;                          // queries per chunk
    // the (group, block) bucket of this CTA (visiting order: bucket_of)
    int r, c;
    bucket_of((int)blockIdx.x, p.Hkv, p.nb, p.num_sms, r, c);
    const int b = blockIdx.y;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    if (qend <= qbeg) return;                               // nobody selected this block
    const int nch = (qend - qbeg + QPC - 1) / QPC;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint64_t *q_full = bars, *q_empty = bars + 2, *s_full = bars + 4, *s_free = bars + 6;
    uint64_t *p_full = bars + 8, *o_full = bars + 12, *o_free = bars + 14;
    uint64_t *kv_full = bars + 16, *done = bars + 17;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 18);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long j0 = (long long)c * kKeys;

    if (threadIdx.x == 0) {
        for (int a = 0; a < 2; ++a) {
            // G == 8: lane 0's expect_tx arrival + 32 metadata arrivals (TMA bytes);
            // otherwise 32 cp.async arrivals + 32 metadata arrivals
            tc::mbar_init(&q_full[a], G == 8 ? 33 : 64);
            // buffer a belongs to epilogue warpgroup a (chunks n with n % 2 == a)
            tc::mbar_init(&q_empty[a], 1 + kWgWarps);   // S MMAs done + epilogue has read the metadata
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kWgWarps);
            tc::mbar_init(&p_full[a], kWgWarps);
            tc::mbar_init(&o_full[a], 1);
            tc::mbar_init(&o_free[a], kWgWarps);
        }
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
        // K and V tiles of this (b, group, block) by TMA; rows past Nk read as zeros
        const int pw = warp == 0 ? 0 : 1;
        if (pw == 0 && lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::mbar_arrive_expect_tx(kv_full, 2 * L::KB * SUB);
#pragma unroll
            for (int kb = 0; kb < L::KB; ++kb) {
                tc::tma_load_4d(sm + L::OFF_K + kb * SUB, &tmap_k, kv_full, kb * 64, r, (int)j0, b);
                tc::tma_load_4d(sm + L::OFF_V + kb * SUB, &tmap_v, kv_full, kb * 64, r, (int)j0, b);
            }
        }
        constexpr int EPL = (QPC + 31) / 32;
        int ent[EPL], ent_next[EPL];
        load_entries(ent, bucket_q, qbeg + pw * QPC, min(QPC, qend - qbeg - pw * QPC), lane);
        for (int m = pw; m < nch; m += 2) {
            const int a = m & 1;
            const int q0 = qbeg + m * QPC;
            const int nq = min(QPC, qend - q0);
            // the next chunk's entries are fetched before waiting for a free stage
            if (m + 2 < nch) load_entries(ent_next, bucket_q, q0 + 2 * QPC, min(QPC, qend - q0 - 2 * QPC), lane);
            if (!tc::mbar_wait(&q_empty[a], ((uint32_t)(m >> 1) & 1u) ^ 1u, st, 61, abort_flag)) break;
            QueryMeta *meta = reinterpret_cast<QueryMeta *>(sm + L::OFF_META + a * 2048);
            store_meta(meta->i, meta->pos, meta->slot, ent, QPC, nq, p, lane);
            if (lane == 0) meta->nq = nq;
            __syncwarp();
            uint8_t *sq = sm + L::OFF_Q + a * (L::KB * SUB);
            if constexpr (G == 8) {
                // one TMA box {64 features, 8 heads, KB halves} per query fills its
                // row group (1024-byte aligned).  Padding slots read rows past the
                // end of q (zero fill).
                if (lane == 0) tc::mbar_arrive_expect_tx(&q_full[a], kRows * D * 2);
                __syncwarp();
                if (lane < QPC) {
                    const int z = lane < nq ? b * p.Nq + entry_row(ent[0]) : p.B * p.Nq;
                    tc::tma_load_4d(sq + lane * (L::KB * 1024), &tmap_q, &q_full[a], 0, r * G, 0, z);
                }
                tc::mbar_arrive(&q_full[a]);
                // the rows of this producer's next chunk (m + 2) into L2 now, so its
                // gathers do not wait on HBM
                if (m + 2 < nch && lane < min(QPC, qend - q0 - 2 * QPC))
                    tc::tma_prefetch_4d(&tmap_q, 0, r * G, 0, b * p.Nq + entry_row(ent_next[0]));
            } else {
                // Q rows: lanes cover whole 16-byte chunks of consecutive rows; the
                // query index comes from the metadata just written (shared memory)
                constexpr int CPR = D / 8;                     // 16-byte chunks per row
                constexpr int RPI = 32 / CPR;                  // rows per iteration
#pragma unroll 8
                for (int it = 0; it < kRows / RPI; ++it) {
                    const int rho = it * RPI + lane / CPR, ch = lane % CPR;
                    const int qq = rho / G, g = rho % G;
                    const bool ok = qq < nq;
                    const int i = meta->i[qq];
                    cp_async16_zfill(sq + (rho >> 3) * (L::KB * 1024) + (ch >> 3) * 1024 + swz(rho & 7, ch & 7),
                                     q + (((long long)b * p.Nq + i) * p.Hq + (long long)r * G + g) * D + ch * 8, ok);
                }
                cp_async_arrive_noinc(&q_full[a]);
                tc::mbar_arrive(&q_full[a]);
            }
#pragma unroll
            for (int t = 0; t < EPL; ++t) ent[t] = ent_next[t];
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer (the whole warp runs
            // the loop; one lane chosen by elect.sync issues)
            constexpr uint32_t I_S = tc::idesc_bf16(128, kKeys);
            constexpr uint32_t I_O = tc::idesc_bf16(128, D) | tc::kBMajorMN;
            const uint64_t dK = tc::sdesc_k128(smem_u32(sm + L::OFF_K));
            const uint64_t dV = tc::sdesc_sw128(smem_u32(sm + L::OFF_V), SUB, 1024);
            const uint64_t dQ0 = tc::sdesc_sw128(smem_u32(sm + L::OFF_Q), 16, L::KB * 1024);
            bool ok = wwait(kv_full, 0, st, 62, abort_flag);
            if (ok) tc::fence_proxy_async();
            auto issue_s = [&](int n) {
                const int a = n & 1;
                const uint64_t dQ = tc::desc_adv(dQ0, a * (L::KB * SUB));
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                        // A = Q rows (K-major, 8-row groups KB KB apart), B = K
                        tc::mma_bf16(tmem + L::TM_S + a * 128, tc::desc_adv(dQ, h * 1024 + ko),
                                     tc::desc_adv(dK, h * SUB + ko), I_S, ks > 0);
                    }
                    tc::mma_commit(&s_full[a]);
                    tc::mma_commit(&q_empty[a]);
                }
                __syncwarp();
            };
            auto issue_o = [&](int m) {
                const int a = m & 1;
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks) {
                        // A = P [rows][keys] from TMEM (16 keys = 8 packed columns per
                        // step); B = V [keys][d] read MN-major (atoms of 64 d, 8-key groups)
                        tc::mma_bf16_ts(tmem + L::TM_O + a * D, tmem + L::TM_S + a * 128 + ks * 8,
                                        tc::desc_adv(dV, ks * 2048), I_O, ks > 0);
                    }
                    tc::mma_commit(&o_full[a]);
                }
                __syncwarp();
            };
            // The two epilogue warpgroups run chunks n and n+1 at once, so S of
            // one chunk and O of another are issued in whichever order their
            // inputs become ready.
            int ns = 0, no = 0;
            uint32_t idle = 0;
            while (ok && no < nch) {
                bool did = false;
                // S(ns) overwrites the TMEM buffer holding P(ns-2): only after O(ns-2) is issued.
                // Each decision is lane 0's, so the warp never splits.
                bool go_s = ns < nch && (ns < 2 || no >= ns - 1) && tc::mbar_test(&q_full[ns & 1], (uint32_t)(ns >> 1) & 1u) &&
                            (ns < 2 || tc::mbar_test(&s_free[ns & 1], ((uint32_t)(ns >> 1) & 1u) ^ 1u));
                if (__shfl_sync(0xffffffffu, go_s, 0)) {
                    tc::fence_proxy_async();
                    tc::fence_after_sync();
                    issue_s(ns);
                    ++ns;
                    did = true;
                }
                bool go_o = no < ns && tc::mbar_test(&p_full[no & 1], (uint32_t)(no >> 1) & 1u) &&
                            (no < 2 || tc::mbar_test(&o_free[no & 1], ((uint32_t)(no >> 1) & 1u) ^ 1u));
                if (__shfl_sync(0xffffffffu, go_o, 0)) {
                    tc::fence_after_sync();
                    issue_o(no);
                    ++no;
                    did = true;
                }
                if (did) {
                    idle = 0;
                } else if (++idle >= tc::kSpinLimit) {
                    if (lane == 0) {
                        report(st, kDevTimeout, 63, ns * 65536 + no);
                        *abort_flag = 1;
                    }
                    ok = false;
                } else if ((idle & 1023u) == 1023u && __shfl_sync(0xffffffffu, *abort_flag, 0)) {
                    ok = false;
                }
            }
            // every MMA issued above has completed once `done` fires
            if (tc::elect_one()) tc::mma_commit(done);
            __syncwarp();
            tc::mbar_wait(done, 0, nullptr, 0, nullptr);
        }
    } else if (warp < kProd2) {
        // ------------------------------------------------ epilogue: one (query, head) row per thread
        // warpgroup wg takes chunks wg, wg + 2, ... (TMEM and smem buffers wg)
        const int quarter = warp & 3, wg = (warp - 2) >> 2;
        const int rho = quarter * 32 + lane;
        const int qq = rho / G, g = rho % G;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale * kLog2e;
        float pm = 0.f, pz = 0.f;            // (m, z) of the chunk whose output is pending
        int pi = 0, pslot = 0;
        bool pvalid = false;
        bool ok = true;
        // writes the partial output of chunk m (row data held in pm, pz, pi, pslot,
        // pvalid).  The rows go through this warpgroup's staging tile so that each
        // store covers whole 256-byte partial rows.
        auto emit = [&](int m) -> bool {
            const int am = m & 1;
            if (!wwait(&o_full[am], (uint32_t)(m >> 1) & 1u, st, 74, abort_flag)) return false;
            tc::fence_after_sync();
            const long long prow =
                pvalid ? (((long long)b * p.Nq + pi) * p.Hq + (long long)r * G + g) * p.topk + pslot : -1;
            uint8_t *stg = sm + L::OFF_P + am * (2 * SUB);
#pragma unroll
            for (int c64 = 0; c64 < D / 64; ++c64) {
                uint32_t o0[32], o1[32];
                tc::tmem_ld32_nowait(tmem + lane_base + L::TM_O + am * D + c64 * 64, o0);
                tc::tmem_ld32_nowait(tmem + lane_base + L::TM_O + am * D + c64 * 64 + 32, o1);
                tc::tmem_wait32(o0);
                tc::tmem_wait32(o1);
#pragma unroll
                for (int x = 0; x < 32; x += 8) {
                    const int c0 = c64 * 8 + x / 8, c1 = c0 + 4;      // 16-byte chunks of the row
                    *reinterpret_cast<uint4 *>(stg + (c0 >> 3) * SUB + swz(rho, c0 & 7)) = make_uint4(
                        pack_bf16(__uint_as_float(o0[x]), __uint_as_float(o0[x + 1])),
                        pack_bf16(__uint_as_float(o0[x + 2]), __uint_as_float(o0[x + 3])),
                        pack_bf16(__uint_as_float(o0[x + 4]), __uint_as_float(o0[x + 5])),
                        pack_bf16(__uint_as_float(o0[x + 6]), __uint_as_float(o0[x + 7])));
                    *reinterpret_cast<uint4 *>(stg + (c1 >> 3) * SUB + swz(rho, c1 & 7)) = make_uint4(
                        pack_bf16(__uint_as_float(o1[x]), __uint_as_float(o1[x + 1])),
                        pack_bf16(__uint_as_float(o1[x + 2]), __uint_as_float(o1[x + 3])),
                        pack_bf16(__uint_as_float(o1[x + 4]), __uint_as_float(o1[x + 5])),
                        pack_bf16(__uint_as_float(o1[x + 6]), __uint_as_float(o1[x + 7])));
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&o_free[am]);
            constexpr int CPR = D / 8, RPI = 32 / CPR;              // chunks per row, rows per store
#pragma unroll
            for (int it = 0; it < 32 / RPI; ++it) {
                const int rr = it * RPI + lane / CPR, ch = lane % CPR, rho2 = quarter * 32 + rr;
                const long long rix = __shfl_sync(0xffffffffu, prow, rr);
                const uint4 x = *reinterpret_cast<const uint4 *>(stg + (ch >> 3) * SUB + swz(rho2, ch & 7));
                if (rix >= 0) *reinterpret_cast<uint4 *>(part + rix * D + ch * 8) = x;
            }
            __syncwarp();
            if (pvalid) stats[prow] = make_float2(pm, pz);
            return true;
        };
        for (int n = wg; ok && n < nch; n += 2) {
            const int a = n & 1;
            const uint32_t ph = (uint32_t)(n >> 1) & 1u;
            const QueryMeta *meta = reinterpret_cast<const QueryMeta *>(sm + L::OFF_META + a * 2048);
            if (!wwait(&q_full[a], ph, st, 71, abort_flag)) { ok = false; break; }
            if (!wwait(&s_full[a], ph, st, 72, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            const bool valid = qq < meta->nq;
            const long long pos = valid ? meta->pos[qq] : -1;
            const int ci = valid ? meta->i[qq] : 0, cslot = valid ? meta->slot[qq] : 0;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&q_empty[a]);     // this chunk's metadata now lives in registers
            // last visible key of this block for this row, as an offset into the block
            const int lim = (int)max(-1LL, min(min(pos, (long long)p.Nk - 1) - j0, (long long)kKeys - 1));
            const uint32_t sbase = tmem + lane_base + L::TM_S + a * 128;
            // pass 1: row max over the visible keys
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent max chains
#pragma unroll
            for (int c64 = 0; c64 < 2; ++c64) {
                uint32_t s0[32], s1[32];
                tc::tmem_ld32_nowait(sbase + c64 * 64, s0);
                tc::tmem_ld32_nowait(sbase + c64 * 64 + 32, s1);
                tc::tmem_wait32(s0);
                tc::tmem_wait32(s1);
                if (lim >= c64 * 64 + 63) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        mq[jj & 3] = fmaxf(mq[jj & 3], fmaxf(__uint_as_float(s0[jj]), __uint_as_float(s1[jj])));
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if (c64 * 64 + jj <= lim) mq[jj & 3] = fmaxf(mq[jj & 3], __uint_as_float(s0[jj]));
                        if (c64 * 64 + 32 + jj <= lim) mq[jj & 3] = fmaxf(mq[jj & 3], __uint_as_float(s1[jj]));
                    }
                }
            }
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            const float msafe = mx == -INFINITY ? 0.f : mx * sl2;
            // pass 2: P = exp2(s*scale*log2e - m) as bf16 over the row's own S
            // columns (keys 32c..32c+31 -> packed columns 16c..16c+15), z = row sum
            // (no mask where every row of the warp sees the whole block; four
            // partial sums keep the row-sum chain short)
            float zp[4] = {0.f, 0.f, 0.f, 0.f};
            auto pass2 = [&](auto all_tag) {
                constexpr bool kAll = decltype(all_tag)::value;
#pragma unroll
                for (int c64 = 0; c64 < 2; ++c64) {
                    uint32_t sr[2][32];
                    tc::tmem_ld32_nowait(sbase + c64 * 64, sr[0]);
                    tc::tmem_ld32_nowait(sbase + c64 * 64 + 32, sr[1]);
                    tc::tmem_wait32(sr[0]);
                    tc::tmem_wait32(sr[1]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c32 = c64 * 2 + h;
                        uint32_t pk[16];
#pragma unroll
                        for (int jj = 0; jj < 32; jj += 2) {
                            const int jo = c32 * 32 + jj;
                            float e0 = tc::ex2(__uint_as_float(sr[h][jj]) * sl2 - msafe);
                            float e1 = tc::ex2(__uint_as_float(sr[h][jj + 1]) * sl2 - msafe);
                            if constexpr (!kAll) {
                                e0 = jo <= lim ? e0 : 0.f;
                                e1 = jo + 1 <= lim ? e1 : 0.f;
                            }
                            zp[(jj >> 1) & 3] += e0 + e1;
                            pk[jj / 2] = pack_bf16(e0, e1);
                        }
                        tc::tmem_st16(sbase + c32 * 16, pk);
                    }
                }
            };
            if (__all_sync(0xffffffffu, lim >= kKeys - 1)) pass2(std::true_type{});
            else pass2(std::false_type{});
            const float cm = msafe, cz = (zp[0] + zp[1]) + (zp[2] + zp[3]);
            const bool cvalid = valid && mx != -INFINITY;
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&s_free[a]);
                tc::mbar_arrive(&p_full[a]);
            }
            // this warpgroup's previous chunk leaves now, while the O MMA of this one runs
            if (n >= 2 && !emit(n - 2)) { ok = false; break; }
            pm = cm;
            pz = cz;
            pvalid = cvalid;
            pi = ci;
            pslot = cslot;
        }
        const int last = nch - 1 - ((nch - 1 - wg) & 1);      // this warpgroup's last chunk
        if (ok && last >= 0) emit(last);
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// One warp per (b, i, h) row: merge the row's slots.  The row's partials are
// contiguous; every lane loads 16 bytes of several slots at once (D/8 lanes
// per slot, all loads in flight while the slot weights are reduced), and
// lanes holding the same features of different slots add up with shuffles.
// With d_o given (the training step) it also writes the backward's
// Drow[b, h, i] = sum_e dO * O over the row, O taken as written (bf16).
template <int D>
__global__ void __launch_bounds__(256)
sparse_fwd_combine_kernel(Problem p, const int32_t *__restrict__ sel, const bf16 *__restrict__ part,
                          const float2 *__restrict__ stats, bf16 *__restrict__ o, float *__restrict__ lse,
                          const bf16 *__restrict__ d_o, float *__restrict__ Drow)
{
    constexpr int LPS = D / 8;                  // lanes per slot row
    constexpr int SPI = 32 / LPS;               // slots per load instruction
    constexpr int GI = 16 / SPI;                // load instructions per group of 16 slots
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)p.B * p.Nq * p.Hq) return;
    const int h = (int)(row % p.Hq);
    const long long bi = row / p.Hq;
    const int i = (int)(bi % p.Nq), b = (int)(bi / p.Nq);
    const int r = h / p.G;
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * p.topk;
    const uint4 *src = reinterpret_cast<const uint4 *>(part + row * p.topk * D);
    auto load_group = [&](uint4 (&u)[GI], int g0) {
#pragma unroll
        for (int t = 0; t < GI; ++t) {
            const int s = g0 + t * SPI + lane / LPS;
            u[t] = s < p.topk ? __ldg(src + s * LPS + lane % LPS) : make_uint4(0, 0, 0, 0);
        }
    };
    // the first 16 slots' partial rows are requested before the selection and
    // the slot statistics arrive (invalid slots are masked below, their bytes
    // never written), so a row costs one memory round trip
    uint4 u[GI];
    load_group(u, 0);
    const uint4 dov = d_o && lane < LPS ? __ldg(reinterpret_cast<const uint4 *>(d_o + row * D) + lane)
                                        : make_uint4(0u, 0u, 0u, 0u);
    const float2 mz_raw = lane < p.topk ? __ldg(stats + row * p.topk + lane) : make_float2(-INFINITY, 0.f);
    // slot validity (same rule as the inverse index)
    const int cl = lane < p.topk ? __ldg(srow + lane) : -1;
    const bool sv = cl >= 0 && cl < p.nb && (long long)cl * 128 <= pos;
    const unsigned mask = __ballot_sync(0xffffffffu, sv);
    const float2 mz = sv ? mz_raw : make_float2(-INFINITY, 0.f);
    const float M = warp_max(mz.x);
    const float w = sv ? exp2f(mz.x - M) : 0.f;
    const float Z = warp_sum(w * mz.y);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int g0 = 0; g0 < p.topk; g0 += 16) {
        if (g0 > 0) load_group(u, g0);
#pragma unroll
        for (int t = 0; t < GI; ++t) {
            const int s = (g0 + t * SPI + lane / LPS) & 31;
            const float ws = __shfl_sync(0xffffffffu, w, s);
            if (!((mask >> s) & 1u)) continue;
            const uint32_t wd[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float2 x = unpack_bf16(wd[q4]);
                acc[2 * q4] += ws * x.x;
                acc[2 * q4 + 1] += ws * x.y;
            }
        }
    }
#pragma unroll
    for (int off = LPS; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    const float inv = 1.f / Z;
    const uint4 ov = make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                                pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
    if (lane < LPS) reinterpret_cast<uint4 *>(o + row * D)[lane] = ov;
    if (lane == 0) lse[((long long)b * p.Hq + h) * p.Nq + i] = (M + log2f(Z)) * kLn2;
    if (d_o) {
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {dov.x, dov.y, dov.z, dov.w};
        float dd = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const float2 x = unpack_bf16(ow[q4]), y = unpack_bf16(gw[q4]);
            dd += x.x * y.x + x.y * y.y;
        }
        if (lane >= LPS) dd = 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
        if (lane == 0) Drow[((long long)b * p.Hq + h) * p.Nq + i] = dd;
    }
}

template <int D, int G>
cudaError_t launch_dg(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const int32_t *sel,
                      const FwdWork &w, DeviceStatus *st, cudaStream_t s)
{
    using L = FwdLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(sparse_fwd_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tv;
    {
        // Q as {d within a half, head, half, query row}: one box {64, G, D/64, 1}
        // is a query's G head rows in every feature half
        const unsigned long long dq4[4] = {64, (unsigned long long)p.Hq, (unsigned long long)(D / 64),
                                           (unsigned long long)p.B * p.Nq};
        const unsigned long long sq4[3] = {D * 2ull, 128ull, (unsigned long long)p.Hq * D * 2ull};
        const unsigned bq4[4] = {64, (unsigned)G, (unsigned)(D / 64), 1};
        if ((e = make_tmap_bf16(&tq, q, 4, dq4, sq4, bq4)) != cudaSuccess) return e;
        // K/V as [B][Nk][Hkv][D] (rows past Nk, even inside kv_rows, are out of bounds)
        const unsigned long long dk[4] = {(unsigned long long)D, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                          (unsigned long long)p.B};
        const unsigned long long sk[3] = {D * 2ull, (unsigned long long)p.Hkv * D * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * D * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk, sk, bk)) != cudaSuccess) return e;
        if ((e = make_tmap_bf16(&tv, v, 4, dk, sk, bk)) != cudaSuccess) return e;
    }
    {
        TimedLaunch timed_("sparse_fwd_tc_kernel", s);
        sparse_fwd_tc_kernel<D, G><<<dim3(p.Hkv * p.nb, p.B), kThreads, L::ALLOC, s>>>(
            tq, tk, tv, p, q, w.bucket_off, w.bucket_q, w.part, w.stats, st);
    }
    note_launch();
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const int32_t *sel,
                     const FwdWork &w, DeviceStatus *st, cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_dg<D, 1>(p, q, k, v, sel, w, st, s);
    case 2: return launch_dg<D, 2>(p, q, k, v, sel, w, st, s);
    case 4: return launch_dg<D, 4>(p, q, k, v, sel, w, st, s);
    default: return launch_dg<D, 8>(p, q, k, v, sel, w, st, s);
    }
}

}  // namespace

cudaError_t launch_sparse_fwd_keymajor(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v,
                                       const int32_t *sel, bf16 *o, float *lse, const FwdWork &w, DeviceStatus *st,
                                       cudaStream_t s)
{
    cudaError_t e = w.index_ready ? cudaSuccess
                                  : launch_inverse_index(p, sel, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, st, s);
    if (e != cudaSuccess) return e;
    e = p.d == 128 ? launch_d<128>(p, q, k, v, sel, w, st, s) : launch_d<64>(p, q, k, v, sel, w, st, s);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Nq * p.Hq;
    if (w.d_o && w.d_o_ready && (e = cudaStreamWaitEvent(s, w.d_o_ready, 0)) != cudaSuccess) return e;
    if (p.d == 128)
        {
            TimedLaunch timed_("sparse_fwd_combine_kernel", s);
            sparse_fwd_combine_kernel<128><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, w.part, w.stats, o, lse,
                                                                                     w.d_o, w.D);
        }
    else
        {
            TimedLaunch timed_("sparse_fwd_combine_kernel", s);
            sparse_fwd_combine_kernel<64><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, sel, w.part, w.stats, o, lse,
                                                                                    w.d_o, w.D);
        }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
