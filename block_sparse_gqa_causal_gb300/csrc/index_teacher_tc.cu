// index_teacher_tc.cu -- the KL alignment loss's teacher terms and the index
// branch's backward of MSA, key-major on the tcgen05 tensor cores, with the
// teacher recomputed on chip: neither probability distribution is written to
// memory.  The tiles hold 128 features; at d or d_idx = 64 the upper 64 are
// zeros (TMA fills boxes past the tensor's width, gathers zero-fill them),
// which add nothing to any product, and are never written back.
//
// "Sparse Attention · Part II", section 3.2: for query i and group r over the
// selected token set T, the teacher is Pt_j = (1/G) sum_h exp(l_{h,j} - lse_h)
// (each head normalised over T by the forward's lse; detached) and the
// student Ps = softmax_T(s), s_j = scale_idx <q_idx, k_idx_j>.  Expanding the
// KL with sum_j Pt_j = 1,
//   KL = sum_j Pt_j (log Pt_j - s_j) + lse_idx,    dKL/ds_j = Ps_j - Pt_j.
// Every term is a sum over the selected blocks, so one CTA per 128-key block
// of one (b, group) -- the queries that selected it come from the inverse
// index -- evaluates them in chunks of 64 queries, keys as the MMA's M:
//   S^T = K Q^T        (M = 128 keys, N = 128 (query, head) rows per
//                       sub-chunk, 128/G queries x G heads; 64 for G = 1)
//   s^T = K_idx q_idx^T (M = 128 keys, N = 64 queries)
// With keys on the TMEM lanes a query's G head rows are adjacent columns of
// one thread, so the teacher is a register sum, and it meets the index score
// of the same (key, query) in the same thread.  The chunk's q_idx rows are
// gathered in the order that puts each query's s^T column in the thread that
// holds its teacher.  Per (query, group, selected block) the kernel leaves
//   sum_j Pt_j (log2 Pt_j - s_j log2 e)            (one partial per lane quarter)
// and in the backward (kGrad)
//   dsig = coef (2^(s log2 e - lse_idx log2 e) - Pt)   on visible keys, bf16
//   dq_idx^T = K_idx^T dsig^T   (M = 128 features, N = 64 queries)
//   dK_idx  += dsig q_idx       (M = 128 keys, N = 128 features)
// dq_idx leaves as bf16 partial rows per (query, group, slot), summed by the
// combine kernel; dK_idx as this group's fp32 share of the block's keys,
// summed over the groups in a fixed order afterwards (no atomics).
// coef = scale_idx * kl_coef / (B Nq Hkv): the mean over (query, group) rows
// and the factor scale_idx that both gradients take from s.
//
// The main-branch backward computes the same logits; keeping this work in its
// tiles would need a third 128-column accumulator (dK_idx) next to dK and dV
// plus two score slots, more than TMEM's 512 columns.  Recomputing costs the
// G logit MMAs and the Q rows per slot, and no memory traffic for the teacher.
//
// Roles: warp 0 loads K and K_idx (TMA) and the Q sub-chunk tiles (one TMA
// box per query when G = 8, cp.async otherwise); warp 1 owns TMEM and issues
// the S^T MMAs; warps 2..17 are the epilogue (TMEM lanes 32*(w%4).., column
// quarter (w-2)/4: a quarter of each S^T sub-chunk and 16 of the 64 s^T
// columns); warp 18 gathers the chunk's q_idx rows and row data; warp 19
// issues the index-score and gradient MMAs.
#include <limits.h>

#include <type_traits>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int D = 128;                     // tile features (d, d_idx of 64 are zero-padded)
constexpr int kKeys = 128;
constexpr int kQ = 64;                     // queries per chunk (s^T columns)
constexpr int kEpiWarps = 16;              // 4 per TMEM lane quarter
constexpr int kWC = 16;                    // s^T / S^T columns per epilogue warp
constexpr int kProdI = 2 + kEpiWarps;      // q_idx rows and row data
constexpr int kIssI = 3 + kEpiWarps;       // issues the index-score and gradient MMAs
constexpr int kThreads = 32 * (4 + kEpiWarps);
constexpr int SUBK = kKeys * 128;          // [128 rows][64 bf16] swizzled sub-tile
constexpr int SUBI = kQ * 128;             // [64 rows][64 bf16] swizzled sub-tile
constexpr int TILE_I = 2 * SUBI;           // a chunk's q_idx rows, two feature halves
constexpr int kQBytes = 96 * 1024;         // the Q sub-chunk ring
constexpr int kISt = 2;                    // q_idx + row-data stages
constexpr int OFF_K = 0;
constexpr int OFF_KI = OFF_K + 2 * SUBK;
constexpr int OFF_Q = OFF_KI + 2 * SUBK;
constexpr int OFF_I = OFF_Q + kQBytes;

// A chunk's 64 queries x G heads of S^T are formed in sub-chunks of NS
// (query, head) columns, NS = 128 where G >= 2 (one MMA of N = 128 runs at
// the full tensor rate and halves the instructions the issuing thread waits
// through), 64 for G = 1.  Epilogue warp column quarter cq reads W = NS/4
// columns of each sub-chunk: QW = W/G queries, all heads of each.
template <int G>
struct Cfg {
    static constexpr int NS = G == 1 ? 64 : 128;
    static constexpr int NSUB = kQ * G / NS;        // sub-chunks per chunk
    static constexpr int QS = NS / G;               // queries per sub-chunk
    static constexpr int TILE_Q = NS * D * 2;       // NS (query, head) rows in 8-row groups of 2048 bytes
    static constexpr int QST = kQBytes / TILE_Q;    // Q stages
    static constexpr int SSLOTS = 256 / NS;         // S^T slots in TMEM (256 columns)
    static constexpr int W = NS / 4;                // columns of a sub-chunk per epilogue warp
    static constexpr int PPS = W / 8;               // 8-column pieces per sub-chunk
    static constexpr int QW = W / G;                // queries of a sub-chunk per epilogue warp
    static_assert(QST * TILE_Q == kQBytes && QST >= 3, "Q ring");
    static_assert(NSUB * QW == 16, "each epilogue warp holds 16 queries of a chunk");
};
constexpr int OFF_SG = OFF_I + kISt * TILE_I;        // dsig^T [128 keys][64 queries]
constexpr int OFF_META = OFF_SG + SUBK;

template <int G>
struct Meta {                 // per chunk, indexed by s^T column
    float lse2[kQ * G];       // lse * log2(e) of the column's query, head g at [c*G + g] (+inf: padding)
    float lsei2[kQ];          // lse_idx * log2(e) (+inf: padding)
    int pos[kQ];              // position (-1: padding)
    // (the row counts below are < 2^29: B Nq Hq < 2^24 and topk <= 32 on validated shapes)
    int ridx[kQ];             // dq_idx partial row ((b*Nq + i)*Hkv + r)*topk + slot (-1: padding)
    int kidx[kQ];             // KL partial ((b*Hkv + r)*Nq + i)*topk + slot (-1: padding)
    int pmin;                 // smallest position among the valid columns
};
template <int G>
constexpr int meta_bytes() { return (int)((sizeof(Meta<G>) + 127) & ~size_t(127)); }
template <int G>
constexpr int off_bar() { return OFF_META + kISt * meta_bytes<G>(); }
template <int G>
constexpr int alloc_bytes() { return off_bar<G>() + 512 + 1024; }
static_assert(alloc_bytes<8>() <= 227 * 1024, "shared memory");

// mbarriers (Q, row-data, S^T and s^T rings, the dsig pair, dq_idx^T,
// kv_full, one done per issuing thread) and the TMEM address + abort flag,
// in 512 bytes
template <int G>
constexpr int n_bars() { return 2 * Cfg<G>::QST + 2 * kISt + 2 * Cfg<G>::SSLOTS + 2 * 2 + 2 + 2 + 3; }
static_assert(n_bars<1>() * 8 + 8 <= 512 && n_bars<8>() * 8 + 8 <= 512, "barrier region");

// TMEM: dK_idx; 256 columns of S^T slots; two 64-column slots for s^T,
// where the chunk's dq_idx^T lands once the epilogue has read s^T
constexpr uint32_t TM_DKI = 0, TM_S = 128, TM_SI = TM_S + 256;
static_assert(TM_SI + 128 <= 512, "TMEM columns");

__device__ __forceinline__ int swz(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }
// row rho, feature half h of a [64 rows][128] tile in 8-row groups of 2048 bytes
__device__ __forceinline__ int roff(int rho, int half, int ch)
{
    return (rho >> 3) * 2048 + half * 1024 + (rho & 7) * 128 + (((ch ^ rho) & 7) << 4);
}

// s^T column c holds chunk query m QS + cq QW + t, for c = 16 cq + m QW + t:
// the query whose teacher the warps of column quarter cq sum from sub-chunk m
template <int G>
__device__ __forceinline__ int col_query(int c)
{
    constexpr int QW = Cfg<G>::QW;
    const int cq = c / kWC, k = c % kWC;
    return (k / QW) * Cfg<G>::QS + cq * QW + k % QW;
}

// Streaming transposing sum over the warp of 16 columns pushed in order
// (c = 0..15): pairs are combined as soon as both exist; after column 15,
// lane l holds the sum over all 32 lanes of column l % 16.
__device__ __forceinline__ void colsum16_push(float (&lv)[5], float x, int c, int lane)
{
    if ((c & 1) == 0) {
        lv[0] = x;
        return;
    }
    float cur = x;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int o = 1 << k;
        const bool hi = (lane & o) != 0;
        const float a = lv[k];
        cur = (hi ? cur : a) + __shfl_xor_sync(0xffffffffu, hi ? a : cur, o);
        if (k == 3) {
            lv[4] = cur + __shfl_xor_sync(0xffffffffu, cur, 16);
            return;
        }
        if (((c >> (k + 1)) & 1) == 0) {
            lv[k + 1] = cur;
            return;
        }
    }
}

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

template <int G, bool kGrad>
__global__ void __launch_bounds__(kThreads, 1)
index_teacher_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q,
                        const bf16 *__restrict__ q_idx, const float *__restrict__ lse,
                        const float *__restrict__ lse_idx, float coef, const int32_t *__restrict__ bucket_off,
                        const int32_t *__restrict__ bucket_q, float *__restrict__ klt, bf16 *__restrict__ dqi_part,
                        float *__restrict__ dki_g, DeviceStatus *st)
{
    using C = Cfg<G>;
    constexpr int QS = C::QS, NSUB = C::NSUB, QST = C::QST, SSLOTS = C::SSLOTS;
    using MetaT = Meta<G>;
    // the (group, block) bucket of this CTA (visiting order: bucket_of)
    int r, c;
    bucket_of((int)blockIdx.x, p.Hkv, p.nb, p.num_sms, r, c);
    const int b = blockIdx.y;
    const long long bucket = ((long long)b * p.Hkv + r) * p.nb + c;
    const int qbeg = bucket_off[bucket], qend = bucket_off[bucket + 1];
    const long long j0 = (long long)c * kKeys;
    if (qend <= qbeg) {
        if constexpr (kGrad) {
            // no query selected this block: the group's dK_idx share is zero
            float4 *dst = reinterpret_cast<float4 *>(dki_g + (((long long)b * p.Hkv + r) * p.Nk + j0) * p.d_idx);
            const int n4 = (int)(min((long long)kKeys, (long long)p.Nk - j0) * (p.d_idx / 4));
            for (int x = threadIdx.x; x < n4; x += kThreads) dst[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int nch = (qend - qbeg + kQ - 1) / kQ;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `sm`
    // stays a shared-memory access (no generic addressing)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + off_bar<G>());
    uint64_t *q_full = bars, *q_empty = q_full + QST, *i_full = q_empty + QST, *i_empty = i_full + kISt;
    uint64_t *s_full = i_empty + kISt, *s_free = s_full + SSLOTS, *si_full = s_free + SSLOTS;
    uint64_t *si_free = si_full + 2, *g_full = si_free + 2, *g_free = g_full + 1, *dq_full = g_free + 1;
    uint64_t *kv_full = dq_full + 2, *done = kv_full + 1;      // done[0]: S issuer, done[1]: index issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int a = 0; a < QST; ++a) {
            // G == 8: lane 0's expect_tx arrival; otherwise 32 cp.async + 32 lane arrivals
            tc::mbar_init(&q_full[a], G == 8 ? 1 : 64);
            tc::mbar_init(&q_empty[a], 1);
        }
        for (int a = 0; a < kISt; ++a) {
            tc::mbar_init(&i_full[a], 64);                 // 32 cp.async + 32 row-data arrivals
            tc::mbar_init(&i_empty[a], 1 + kEpiWarps);     // last MMA reading q_idx + row data read
        }
        for (int a = 0; a < SSLOTS; ++a) {
            tc::mbar_init(&s_full[a], 1);
            tc::mbar_init(&s_free[a], kEpiWarps);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&si_full[a], 1);
            // the slot is free once the epilogue has read what lands there last:
            // s^T (KL only) or the dq_idx^T that follows it (backward)
            tc::mbar_init(&si_free[a], kEpiWarps);
            tc::mbar_init(&dq_full[a], 1);
        }
        tc::mbar_init(g_full, kEpiWarps);                   // dsig tile written
        tc::mbar_init(g_free, 1);                           // its gradient MMAs done
        tc::mbar_init(kv_full, 1);
        tc::mbar_init(&done[0], 1);
        tc::mbar_init(&done[1], 1);
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
        // ------------------------------------------------ producer: K, K_idx, Q sub-chunks
        if (lane == 0) {
            if constexpr (G == 8) tc::prefetch_tmap(&tmap_q);
            tc::mbar_arrive_expect_tx(kv_full, 4 * SUBK);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc::tma_load_4d(sm + OFF_K + h * SUBK, &tmap_k, kv_full, h * 64, r, (int)j0, b);
                tc::tma_load_3d(sm + OFF_KI + h * SUBK, &tmap_ki, kv_full, h * 64, (int)j0, b);
            }
        }
        // a chunk's 64 bucket entries, lane l holding queries l and l + 32 (-1:
        // padding), loaded two chunks ahead.  The next chunk's Q rows are not
        // prefetched into L2: at G = 8 one TMA-unit prefetch per query cost this
        // warp as much issue time as the loads themselves and made it late at
        // every chunk boundary (9.25 -> 8.38 ms without it at 128K); at G = 4 the
        // per-line prefetches cost 3% of the kernel.  The three stages cover the
        // loads' latency.
        auto load_ent = [&](int (&e)[2], int n) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int x = qbeg + n * kQ + lane + 32 * t;
                e[t] = n < nch && x < qend ? __ldg(bucket_q + x) : -1;
            }
        };
        auto ent_of = [&](const int (&e)[2], int qq) {      // entry of chunk query qq (all lanes call)
            const int x0 = __shfl_sync(0xffffffffu, e[0], qq & 31), x1 = __shfl_sync(0xffffffffu, e[1], qq & 31);
            return qq < 32 ? x0 : x1;
        };
        int ent[2], ent1[2], ent2[2];
        load_ent(ent, 0);
        load_ent(ent1, 1);
        for (int n = 0; n < nch; ++n) {
            load_ent(ent2, n + 2);
            bool ok = true;
            for (int m = 0; m < NSUB; ++m) {
                const int u = n * NSUB + m, s = u % QST;
                if (!tc::mbar_wait(&q_empty[s], ((uint32_t)(u / QST) & 1u) ^ 1u, st, 141, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *sq = sm + OFF_Q + s * C::TILE_Q;
                if constexpr (G == 8) {
                    // one box {64 features, 8 heads, 2 halves} per query fills a 2048-byte
                    // row group; padding queries read rows past the end (zero fill)
                    static_assert(QS <= 32 && (QS & (QS - 1)) == 0, "one lane per query");
                    const int e = ent_of(ent, m * QS + (lane & (QS - 1)));
                    if (lane == 0) tc::mbar_arrive_expect_tx(&q_full[s], C::TILE_Q);
                    __syncwarp();
                    if (lane < QS) {
                        const int z = e >= 0 ? b * p.Nq + entry_row(e) : p.B * p.Nq;
                        tc::tma_load_4d(sq + lane * 2048, &tmap_q, &q_full[s], 0, r * G, 0, z);
                    }
                } else {
                    // NS rows x 16 chunks: lane covers chunk lane%16 of rows 2*it + lane/16
#pragma unroll 4
                    for (int it = 0; it < C::NS / 2; ++it) {
                        const int rho = it * 2 + (lane >> 4), ch = lane & 15;
                        const int g = rho % G;
                        const int e = ent_of(ent, m * QS + rho / G);
                        const int i = e >= 0 ? entry_row(e) : 0;
                        const bool ok = e >= 0 && ch * 8 < p.d;
                        const long long off =
                            (((long long)b * p.Nq + i) * p.Hq + (long long)r * G + g) * p.d + (ok ? ch * 8 : 0);
                        cp_async16_zfill(sq + roff(rho, ch >> 3, ch & 7), q + off, ok);
                    }
                    cp_async_arrive_noinc(&q_full[s]);
                    tc::mbar_arrive(&q_full[s]);
                }
            }
            if (!ok) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                ent[t] = ent1[t];
                ent1[t] = ent2[t];
            }
        }
        cp_async_wait<0>();
    } else if (warp == kProdI) {
        // ------------------------------------------------ producer: q_idx rows and row data per chunk
        // Entries two chunks ahead and their lse values one chunk ahead, in
        // registers, so a stage is filled as soon as it is free.  Lane l serves
        // s^T columns l and l + 32.
        struct Rows {
            int e[2];
            float l2[2][G];
            float li[2];
        };
        auto load_ent = [&](int (&e)[2], int n) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int x = qbeg + n * kQ + col_query<G>(lane + 32 * t);
                e[t] = n < nch && x < qend ? __ldg(bucket_q + x) : -1;
            }
        };
        auto load_vals = [&](Rows &v, const int (&e)[2]) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                v.e[t] = e[t];
                const bool ok = e[t] >= 0;
                const int i = ok ? entry_row(e[t]) : 0;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    v.l2[t][g] =
                        ok ? __ldg(lse + ((long long)b * p.Hq + (long long)r * G + g) * p.Nq + i) * kLog2e : INFINITY;
                v.li[t] = kGrad && ok ? __ldg(lse_idx + ((long long)b * p.Hkv + r) * p.Nq + i) * kLog2e : INFINITY;
            }
        };
        int e1[2], e2[2];
        Rows cur, nxt;
        {
            int e0[2];
            load_ent(e0, 0);
            load_ent(e1, 1);
            load_vals(cur, e0);
        }
        for (int n = 0; n < nch; ++n) {
            const int s = n % kISt;
            load_ent(e2, n + 2);
            if (n + 1 < nch) load_vals(nxt, e1);
            if (!tc::mbar_wait(&i_empty[s], ((uint32_t)(n / kISt) & 1u) ^ 1u, st, 142, abort_flag)) break;
            MetaT *mt = reinterpret_cast<MetaT *>(sm + OFF_META + s * meta_bytes<G>());
            uint8_t *si = sm + OFF_I + s * TILE_I;
            int pm = INT_MAX;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int col = lane + 32 * t;
                const bool ok = cur.e[t] >= 0;
                const int i = ok ? entry_row(cur.e[t]) : 0, slot = entry_slot(cur.e[t]);
                mt->pos[col] = ok ? p.q_offset + i : -1;
                if (ok) pm = min(pm, p.q_offset + i);
                mt->ridx[col] = ok ? (int)((((long long)b * p.Nq + i) * p.Hkv + r) * p.topk + slot) : -1;
                mt->kidx[col] = ok ? (int)((((long long)b * p.Hkv + r) * p.Nq + i) * p.topk + slot) : -1;
                mt->lsei2[col] = cur.li[t];
#pragma unroll
                for (int g = 0; g < G; ++g) mt->lse2[col * G + g] = cur.l2[t][g];
                const bf16 *src = q_idx + (((long long)b * p.Nq + i) * p.Hkv + r) * p.d_idx;
#pragma unroll
                for (int ch = 0; ch < D / 8; ++ch) {
                    const bool okc = ok && ch * 8 < p.d_idx;
                    cp_async16_zfill(si + (ch >> 3) * SUBI + swz(col, ch & 7), src + (okc ? ch * 8 : 0), okc);
                }
            }
            pm = __reduce_min_sync(0xffffffffu, pm);
            if (lane == 0) mt->pmin = pm;
            cp_async_arrive_noinc(&i_full[s]);
            tc::mbar_arrive(&i_full[s]);
#pragma unroll
            for (int t = 0; t < 2; ++t) e1[t] = e2[t];
            cur = nxt;
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer: S^T sub-chunks
            // (the whole warp runs the loop; one elected lane issues)
            constexpr uint32_t I_S = tc::idesc_bf16(128, C::NS);
            const uint64_t dK = tc::sdesc_k128(smem_u32(sm + OFF_K));
            // S^T of sub-chunk u: A = K (K-major), B = the Q rows (K-major, 8-row groups 2048 bytes apart)
            auto issue_S = [&](int u) -> bool {
                const int s = u % QST, slot = u % SSLOTS;
                if (!wwait(&q_full[s], (uint32_t)(u / QST) & 1u, st, 143, abort_flag)) return false;
                if (u >= SSLOTS && !wwait(&s_free[slot], (uint32_t)(u / SSLOTS - 1) & 1u, st, 144, abort_flag))
                    return false;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint64_t dQ = tc::sdesc_sw128(smem_u32(sm + OFF_Q + s * C::TILE_Q), 16, 2048);
                const uint32_t ts = tmem + TM_S + slot * C::NS;
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                        tc::mma_bf16(ts, tc::desc_adv(dK, h * SUBK + ko), tc::desc_adv(dQ, h * 1024 + ko), I_S, ks > 0);
                    }
                    tc::mma_commit(&s_full[slot]);
                    tc::mma_commit(&q_empty[s]);
                }
                __syncwarp();
                return true;
            };
            bool ok = wwait(kv_full, 0, st, 149, abort_flag);
            for (int u = 0; ok && u < nch * NSUB; ++u) ok = issue_S(u);
            if (tc::elect_one()) tc::mma_commit(&done[0]);
            __syncwarp();
            tc::mbar_wait(&done[0], 0, nullptr, 0, nullptr);
        }
    } else if (warp == kIssI) {
        {
            // ------------------------------------------------ MMA issuer: index scores and gradients.
            // A thread of its own on another scheduler than the S^T issuer: every
            // wait and issue of a single thread queues behind the epilogue's
            // exponentials, so two issuers keep the tensor pipe fed.
            constexpr uint32_t I_SI = tc::idesc_bf16(128, 64);
            constexpr uint32_t I_DQ = tc::idesc_bf16(128, 64) | tc::kAMajorMN | tc::kBMajorMN;
            constexpr uint32_t I_DKI = tc::idesc_bf16(128, D) | tc::kBMajorMN;
            const uint32_t aKI = smem_u32(sm + OFF_KI);
            const uint64_t dKI = tc::sdesc_k128(aKI), dKIT = tc::sdesc_sw128(aKI, SUBK, 1024);
            const uint32_t sg = smem_u32(sm + OFF_SG);
            const uint64_t dSGT = tc::sdesc_sw128(sg, SUBK, 1024), dSG = tc::sdesc_k128(sg);
            // s^T of chunk n: A = K_idx (K-major), B = the chunk's q_idx rows (K-major)
            auto issue_SI = [&](int n) -> bool {
                const int s = n % kISt;
                if (!wwait(&i_full[s], (uint32_t)(n / kISt) & 1u, st, 145, abort_flag)) return false;
                if (n >= 2 && !wwait(&si_free[n & 1], (uint32_t)((n >> 1) - 1) & 1u, st, 146, abort_flag))
                    return false;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint64_t dI = tc::sdesc_k128(smem_u32(sm + OFF_I + s * TILE_I));
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t h = ks >> 2, ko = (ks & 3) * 32;
                        tc::mma_bf16(tmem + TM_SI + (n & 1) * 64, tc::desc_adv(dKI, h * SUBK + ko),
                                     tc::desc_adv(dI, h * SUBI + ko), I_SI, ks > 0);
                    }
                    tc::mma_commit(&si_full[n & 1]);
                    if constexpr (!kGrad) tc::mma_commit(&i_empty[s]);
                }
                __syncwarp();
                return true;
            };
            // gradients of chunk n from the dsig tile; dq_idx^T goes over chunk n's s^T
            // (the epilogue has read it before writing dsig)
            auto issue_G = [&](int n) -> bool {
                if (!wwait(g_full, (uint32_t)n & 1u, st, 147, abort_flag)) return false;
                tc::fence_after_sync();
                const uint64_t dIm = tc::sdesc_sw128(smem_u32(sm + OFF_I + (n % kISt) * TILE_I), SUBI, 1024);
                if (tc::elect_one()) {
                    // dq_idx^T = K_idx^T dsig^T: both operands MN-major; K = 128 keys
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks)
                        tc::mma_bf16(tmem + TM_SI + (n & 1) * 64, tc::desc_adv(dKIT, ks * 2048),
                                     tc::desc_adv(dSGT, ks * 2048), I_DQ, ks > 0);
                    tc::mma_commit(&dq_full[n & 1]);
                    // dK_idx += dsig q_idx: A K-major over queries, B = q_idx MN-major; K = 64 queries
#pragma unroll
                    for (int ks = 0; ks < kQ / 16; ++ks)
                        tc::mma_bf16(tmem + TM_DKI, tc::desc_adv(dSG, ks * 32), tc::desc_adv(dIm, ks * 2048), I_DKI,
                                     n > 0 || ks > 0);
                    tc::mma_commit(&i_empty[n % kISt]);
                    tc::mma_commit(g_free);
                }
                __syncwarp();
                return true;
            };
            // the scores of chunk n+1 are issued before the gradients of chunk n, so the
            // tensor pipe works on them while the epilogue forms chunk n's dsig
            bool ok = wwait(kv_full, 0, st, 149, abort_flag);
            for (int n = 0; ok && n < nch; ++n) {
                ok = issue_SI(n);
                if constexpr (kGrad) {
                    if (ok && n >= 1) ok = issue_G(n - 1);
                }
            }
            if constexpr (kGrad) {
                if (ok) ok = issue_G(nch - 1);
            }
            if (tc::elect_one()) tc::mma_commit(&done[1]);
            __syncwarp();
            tc::mbar_wait(&done[1], 0, nullptr, 0, nullptr);
        }
    } else {
        // ------------------------------------------------ epilogue
        constexpr int QW = C::QW, PPS = C::PPS;    // queries, 8-column pieces of a sub-chunk per warp
        const int qd = warp & 3, cq = (warp - 2) >> 2;
        const int c0 = cq * kWC;                   // the warp's first s^T column
        const int cw = cq * C::W;                  // the warp's first column of an S^T sub-chunk
        const int kr = qd * 32 + lane;             // key (score phases) or feature (dq_idx^T drain)
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const long long j = j0 + kr;
        const bool key_ok = j < p.Nk;
        const int ji = (int)min(j, (long long)INT_MAX);
        const float sl2 = p.scale * kLog2e, si2 = p.scale_idx * kLog2e;
        const float invG = 1.f / (float)G;
        int rp_prev = -1;                          // dq_idx partial row of column c0 + lane%16, previous chunk
        bool ok = true;
        // dq_idx^T of chunk m (lanes are features 32 qd .., columns the queries
        // c0 ..): one partial row per step, the warp's 32 lanes writing its 64
        // contiguous bytes
        auto drain = [&](int m) -> bool {
            if (!wwait(&dq_full[m & 1], (uint32_t)(m >> 1) & 1u, st, 156, abort_flag)) return false;
            tc::fence_after_sync();
            uint32_t v[kWC];
            tc::tmem_ld16_nowait(tmem + lane_base + TM_SI + (m & 1) * 64 + c0, v);
            tc::tmem_wait16(v);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&si_free[m & 1]);
            // partial rows are DW = d_idx features apart; features past d_idx are
            // padding.  Lanes 2m, 2m+1 trade values so that each lane holds
            // features (2m, 2m+1) of one column of a column pair (lane 2m column
            // 2t, lane 2m+1 column 2t+1): one 4-byte store per lane
            const int fpair = qd * 32 + (lane & ~1), odd = lane & 1;
            auto store_rows = [&](auto dw_tag) {
                constexpr int DW = decltype(dw_tag)::value;
                const bool feat_ok = fpair < DW;
#pragma unroll
                for (int t = 0; t < kWC / 2; ++t) {
                    const float ev = __uint_as_float(v[2 * t]), od = __uint_as_float(v[2 * t + 1]);
                    const float mine = odd ? od : ev, give = odd ? ev : od;
                    const float other = __shfl_xor_sync(0xffffffffu, give, 1);
                    const int rix = __shfl_sync(0xffffffffu, rp_prev, 2 * t + odd);
                    if (feat_ok && rix >= 0)
                        *reinterpret_cast<uint32_t *>(dqi_part + (long long)rix * DW + fpair) =
                            pack_bf16(odd ? other : mine, odd ? mine : other);
                }
            };
            if (p.d_idx == 128) store_rows(std::integral_constant<int, 128>{});
            else store_rows(std::integral_constant<int, 64>{});
            return true;
        };
        for (int n = 0; ok && n < nch; ++n) {
            const int s = n % kISt;
            const MetaT *mt = reinterpret_cast<const MetaT *>(sm + OFF_META + s * meta_bytes<G>());
            if (!wwait(&i_full[s], (uint32_t)(n / kISt) & 1u, st, 151, abort_flag)) {
                ok = false;
                break;
            }
            // no per-element mask where every valid query of the chunk sees the whole
            // block (padding columns carry lse = +inf and zero rows: they add nothing)
            const bool all_vis = (long long)mt->pmin >= j0 + kKeys - 1 && j0 + kKeys <= p.Nk;
            // ---- teacher of this key for the warp's 16 queries, from the NSUB sub-chunks.
            // The warp's W columns of a sub-chunk are read as 8-column pieces in a
            // two-deep pipeline: piece i+1's TMEM load is in flight while piece i is
            // summed (a wait covers every load issued before it, so one at a time).
            constexpr int kPieces = NSUB * PPS;
            float pt[kWC];
#pragma unroll
            for (int k = 0; k < kWC; ++k) pt[k] = 0.f;
            auto teacher = [&](auto all_tag) {
                constexpr bool kAll = decltype(all_tag)::value;
                uint32_t buf[2][8];
                auto issue = [&](int i) -> bool {       // piece i: sub-chunk i/PPS, columns cw + 8*(i%PPS)
                    const int u = n * NSUB + i / PPS;
                    if (i % PPS == 0) {
                        if (!wwait(&s_full[u % SSLOTS], (uint32_t)(u / SSLOTS) & 1u, st, 152, abort_flag)) return false;
                        tc::fence_after_sync();
                    }
                    tc::tmem_ld8_nowait(tmem + lane_base + TM_S + (u % SSLOTS) * C::NS + cw + 8 * (i % PPS),
                                        buf[i & 1]);
                    return true;
                };
                if (!(ok = issue(0))) return;
                tc::tmem_wait8(buf[0]);
#pragma unroll
                for (int i = 0; i < kPieces; ++i) {
                    // At a sub-chunk's last piece the slot is released first (every
                    // piece is in registers) and the next sub-chunk is waited for only
                    // after this piece's sums, so neither wait holds up the other slot.
                    const bool last = i % PPS == PPS - 1;
                    if (last) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&s_free[(n * NSUB + i / PPS) % SSLOTS]);
                    } else if (i + 1 < kPieces) {
                        if (!(ok = issue(i + 1))) return;
                    }
                    const int m = i / PPS, part = i % PPS;
                    const float4 *l2 = reinterpret_cast<const float4 *>(mt->lse2 + (c0 + m * QW) * G + 8 * part);
#pragma unroll
                    for (int r4 = 0; r4 < 2; ++r4) {
                        const float4 l = l2[r4];
                        const float lv4[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int rho = 8 * part + 4 * r4 + e, k = m * QW + rho / G;
                            const float x = tc::ex2(__uint_as_float(buf[i & 1][4 * r4 + e]) * sl2 - lv4[e]);
                            if constexpr (kAll) pt[k] += x;
                            else pt[k] += (key_ok && ji <= mt->pos[c0 + k]) ? x : 0.f;
                        }
                    }
                    if (last && i + 1 < kPieces) {
                        if (!(ok = issue(i + 1))) return;
                    }
                    if (i + 1 < kPieces) tc::tmem_wait8(buf[(i + 1) & 1]);
                }
            };
            if (all_vis) teacher(std::true_type{});
            else teacher(std::false_type{});
            if (!ok) break;
#pragma unroll
            for (int k = 0; k < kWC; ++k) pt[k] *= invG;
            // ---- index scores of the same 16 queries: loss terms and dsig
            if (!wwait(&si_full[n & 1], (uint32_t)(n >> 1) & 1u, st, 153, abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            uint32_t sv[kWC];
            tc::tmem_ld16_nowait(tmem + lane_base + TM_SI + (n & 1) * 64 + c0, sv);
            tc::tmem_wait16(sv);
            tc::fence_before_sync();
            __syncwarp();
            if constexpr (!kGrad) {
                if (lane == 0) tc::mbar_arrive(&si_free[n & 1]);
            }
            float lv[5];                               // streaming warp sums of the loss terms
            [[maybe_unused]] uint32_t sg[kWC / 2];
            auto index_terms = [&](auto all_tag) {
                [[maybe_unused]] constexpr bool kAll = decltype(all_tag)::value;
                [[maybe_unused]] float li[kWC];
                if constexpr (kGrad) {
#pragma unroll
                    for (int r4 = 0; r4 < kWC / 4; ++r4) {
                        const float4 l = reinterpret_cast<const float4 *>(mt->lsei2 + c0)[r4];
                        li[4 * r4] = l.x;
                        li[4 * r4 + 1] = l.y;
                        li[4 * r4 + 2] = l.z;
                        li[4 * r4 + 3] = l.w;
                    }
                }
#pragma unroll
                for (int k = 0; k < kWC; k += 2) {
                    [[maybe_unused]] float gv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        // explicit roundings: the same bits whether or not the loss terms
                        // are formed (no contraction into an fma in one form only)
                        const float s2 = __fmul_rn(__uint_as_float(sv[k + e]), si2);
                        const float ptk = pt[k + e];      // zero on invisible keys and padding
                        if (klt) colsum16_push(lv, ptk > 0.f ? ptk * (tc::lg2(ptk) - s2) : 0.f, k + e, lane);
                        if constexpr (kGrad) {
                            const float g = coef * (tc::ex2(__fsub_rn(s2, li[k + e])) - ptk);
                            if constexpr (kAll) gv[e] = g;
                            else gv[e] = key_ok && ji <= mt->pos[c0 + k + e] ? g : 0.f;
                        }
                    }
                    if constexpr (kGrad) sg[k / 2] = pack_bf16(gv[0], gv[1]);
                }
            };
            if (all_vis) index_terms(std::true_type{});
            else index_terms(std::false_type{});
            if (klt && lane < kWC) {
                const int kx = mt->kidx[c0 + lane];            // lane l: column c0 + l
                if (kx >= 0) klt[(long long)kx * 4 + qd] = lv[4];
            }
            [[maybe_unused]] int rp_cur = -1;
            if constexpr (kGrad) rp_cur = mt->ridx[c0 + (lane & (kWC - 1))];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&i_empty[s]);     // the chunk's row data is no longer read
            if constexpr (kGrad) {
                // the tile is free once the previous chunk's gradient MMAs have read it
                if (n >= 1 && !wwait(g_free, (uint32_t)(n - 1) & 1u, st, 154, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *dst = sm + OFF_SG;                    // [128 keys][64 queries]: this warp's 32 bytes
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
                    *reinterpret_cast<uint4 *>(dst + swz(kr, 2 * cq + c2)) =
                        make_uint4(sg[4 * c2], sg[4 * c2 + 1], sg[4 * c2 + 2], sg[4 * c2 + 3]);
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(g_full);
                if (n >= 1 && !drain(n - 1)) {
                    ok = false;
                    break;
                }
                rp_prev = rp_cur;
            }
        }
        if constexpr (kGrad) {
            if (ok) ok = drain(nch - 1);
            if (ok) {
                // the last chunk's dK_idx MMAs have completed once its dsig tile is free
                ok = wwait(g_free, (uint32_t)(nch - 1) & 1u, st, 155, abort_flag);
                tc::fence_after_sync();
            }
            if (ok) {
                // this group's dK_idx share of this key, features 32 cq .. 32 cq + 31
                uint32_t a[32];
                tc::tmem_ld32_nowait(tmem + lane_base + TM_DKI + cq * 32, a);
                tc::tmem_wait32(a);
                if (key_ok && cq * 32 < p.d_idx) {
                    float *dst = dki_g + (((long long)b * p.Hkv + r) * p.Nk + j) * p.d_idx + cq * 32;
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4 *>(dst + x) =
                            make_float4(__uint_as_float(a[x]), __uint_as_float(a[x + 1]), __uint_as_float(a[x + 2]),
                                        __uint_as_float(a[x + 3]));
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

// dk_idx[b, j, :] = bf16( sum over groups r, in order, of dki_g[b, r, j, :] )
__global__ void __launch_bounds__(256) dki_group_sum_kernel(Problem p, const float4 *__restrict__ dki_g,
                                                            bf16 *__restrict__ dk_idx)
{
    const long long n4 = (long long)p.B * p.Nk * (p.d_idx / 4);
    const long long per_b = (long long)p.Nk * (p.d_idx / 4);
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (long long)gridDim.x * blockDim.x) {
        const long long bb = x / per_b, rest = x % per_b;
        float4 a = __ldg(dki_g + (bb * p.Hkv) * per_b + rest);
        for (int r = 1; r < p.Hkv; ++r) {
            const float4 v = __ldg(dki_g + (bb * p.Hkv + r) * per_b + rest);
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        }
        *reinterpret_cast<uint2 *>(dk_idx + x * 4) = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
    }
}

// KL of each (query, group) row from the per-slot, per-lane-quarter sums of
// Pt (log2 Pt - s log2 e): KL = ln 2 * (their sum over the valid slots) +
// lse_idx.  Fixed order, no atomics.
__global__ void kl_rows_combine_kernel(Problem p, const int32_t *__restrict__ sel, const float *__restrict__ lse_idx,
                                       const float4 *__restrict__ klt, float *__restrict__ kl_rows)
{
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= (long long)p.B * p.Hkv * p.Nq) return;
    const long long pos = (long long)p.q_offset + (row % p.Nq);
    const int32_t *srow = sel + row * p.topk;
    float T = 0.f;
    for (int t = 0; t < p.topk; ++t) {
        const int cc = srow[t];
        if (cc < 0 || cc >= p.nb || (long long)cc * 128 > pos) continue;
        const float4 v = klt[row * p.topk + t];
        T += (v.x + v.y) + (v.z + v.w);
    }
    kl_rows[row] = T * kLn2 + lse_idx[row];
}

template <int G, bool kGrad>
cudaError_t launch_g(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                     const float *lse, const float *lse_idx, float coef, const int32_t *bucket_off,
                     const int32_t *bucket_q, float *klt, bf16 *dqi_part, float *dki_g, DeviceStatus *st,
                     cudaStream_t s)
{
    constexpr int ALLOC = alloc_bytes<G>();
    cudaError_t e = cudaFuncSetAttribute(index_teacher_tc_kernel<G, kGrad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tki;
    {
        // Q as {d within a half, head, half, query row}: one box {64, G, 2, 1} is a
        // query's G head rows in both feature halves (at d = 64 the second half
        // lies past the tensor and reads as zeros)
        const unsigned long long dq4[4] = {64, (unsigned long long)p.Hq, (unsigned long long)p.d / 64,
                                           (unsigned long long)p.B * p.Nq};
        const unsigned long long sq4[3] = {p.d * 2ull, 128ull, (unsigned long long)p.Hq * p.d * 2ull};
        const unsigned bq4[4] = {64, (unsigned)G, 2, 1};
        if ((e = make_tmap_bf16(&tq, q, 4, dq4, sq4, bq4)) != cudaSuccess) return e;
        // K as [B][Nk][Hkv][d] (rows past Nk, features past d read as zeros)
        const unsigned long long dk4[4] = {(unsigned long long)p.d, (unsigned long long)p.Hkv, (unsigned long long)p.Nk,
                                           (unsigned long long)p.B};
        const unsigned long long sk[3] = {p.d * 2ull, (unsigned long long)p.Hkv * p.d * 2ull,
                                          (unsigned long long)p.kv_rows * p.Hkv * p.d * 2ull};
        const unsigned bk[4] = {64, 1, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tk, k, 4, dk4, sk, bk)) != cudaSuccess) return e;
        // K_idx as [B][Nk][d_idx]
        const unsigned long long di[3] = {(unsigned long long)p.d_idx, (unsigned long long)p.Nk,
                                          (unsigned long long)p.B};
        const unsigned long long si[2] = {p.d_idx * 2ull, (unsigned long long)p.kv_rows * p.d_idx * 2ull};
        const unsigned bi[3] = {64, (unsigned)kKeys, 1};
        if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    }
    {
        TimedLaunch timed_(kGrad ? "index_teacher_bwd_tc_kernel" : "index_teacher_kl_tc_kernel", s);
        index_teacher_tc_kernel<G, kGrad><<<dim3(p.Hkv * p.nb, p.B), kThreads, ALLOC, s>>>(
            tq, tk, tki, p, q, q_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g, st);
    }
    note_launch();
    return cudaGetLastError();
}

template <bool kGrad>
cudaError_t launch_grad(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                        const float *lse, const float *lse_idx, float coef, const int32_t *bucket_off,
                        const int32_t *bucket_q, float *klt, bf16 *dqi_part, float *dki_g, DeviceStatus *st,
                        cudaStream_t s)
{
    switch (p.G) {
    case 1: return launch_g<1, kGrad>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g, st, s);
    case 2: return launch_g<2, kGrad>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g, st, s);
    case 4: return launch_g<4, kGrad>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g, st, s);
    default: return launch_g<8, kGrad>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g, st, s);
    }
}

}  // namespace

cudaError_t launch_index_teacher_tc(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx,
                                    const bf16 *k_idx, const float *lse, const float *lse_idx, float kl_coef,
                                    const int32_t *bucket_off, const int32_t *bucket_q, float *klt, bf16 *dqi_part,
                                    float *dki_g, DeviceStatus *st, cudaStream_t s)
{
    if ((p.d != 64 && p.d != D) || (p.d_idx != 64 && p.d_idx != D)) return cudaErrorInvalidValue;
    const float coef = p.scale_idx * kl_coef / ((float)p.B * (float)p.Nq * (float)p.Hkv);
    if (dqi_part)
        return launch_grad<true>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, dqi_part, dki_g,
                                 st, s);
    return launch_grad<false>(p, q, k, q_idx, k_idx, lse, lse_idx, coef, bucket_off, bucket_q, klt, nullptr, nullptr,
                              st, s);
}

cudaError_t launch_dki_group_sum(const Problem &p, const float *dki_g, bf16 *dk_idx, cudaStream_t s)
{
    {
        TimedLaunch timed_("dki_group_sum_kernel", s);
        dki_group_sum_kernel<<<4 * p.num_sms, 256, 0, s>>>(p, reinterpret_cast<const float4 *>(dki_g), dk_idx);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_kl_rows_combine(const Problem &p, const int32_t *sel, const float *lse_idx, const float *klt,
                                   float *kl_rows, cudaStream_t s)
{
    const long long rows = (long long)p.B * p.Hkv * p.Nq;
    {
        TimedLaunch timed_("kl_rows_combine_kernel", s);
        kl_rows_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(
            p, sel, lse_idx, reinterpret_cast<const float4 *>(klt), kl_rows);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
