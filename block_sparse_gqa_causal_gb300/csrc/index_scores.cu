// index_scores.cu -- index branch of MSA: token scores and block max-pool,
// on the 5th-generation tensor cores (tcgen05 + TMEM, operands by TMA).
//
// "Sparse Attention · Part II", section 3.2: per query and GQA group, the
// group's index query is dotted with the index key head shared by all
// groups over every causally visible token, and each 128-token block is
// scored by its largest visible token score.  This is the only quadratic
// stage of the layer.  The N x N token scores never leave the SM: each
// 128 x 128 score tile lands in TMEM and is reduced there to 128 block
// scores by the epilogue warps.
//
// GEMM rows are the "flat" (query, group) rows rho = i*Hkv + r of one batch
// entry (q_idx [B, Nq, Hkv, d_idx] is exactly that row-major matrix), so all
// rows share the K_idx tile.  A CTA owns 256 rows (two M=128 tiles) and
// walks the key blocks those rows can see (or a slice of them when there
// are few row tiles, as in decode).  Roles:
//   warp 0      TMA producer: Q tiles once, then K_idx blocks into a 4-deep ring
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2..9  epilogue: TMEM -> registers, causal mask, row max, store
// Two TMEM accumulator sets (2 tiles x 128 fp32 columns each) alternate so
// the epilogue of block c overlaps the MMAs of block c+1.
//
// When a CTA sees every block of its rows and k <= 16 the selection happens
// here too: each epilogue thread owns one row and keeps the 16 best earlier
// blocks in registers (sorted by score, then lower index: a later block
// enters only with a strictly larger score), so the block scores need not
// round-trip through memory; the k-1 best plus the local block are written
// in ascending order, as the separate top-k kernel does.  When a row's
// blocks are split across CTAs (decode: few rows, long rows) the block
// scores of the CTA's slice stay in shared memory; after the last block
// each epilogue warp takes a row and leaves the slice's 16 best as ranking
// keys (warp bitonic sorts), and a small kernel merges the slices' lists.
#include <algorithm>

#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kTileRows = 256;     // two M=128 tiles
constexpr int kStages = 4;         // K_idx ring depth
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kSub = 128 * 128;    // one [128 rows][64 bf16] swizzled sub-tile, bytes
constexpr uint32_t kIdesc = tc::idesc_bf16(128, 128);
constexpr int kSelFloats = 7168;   // split selection: block scores of the CTA's rows x slice

template <int DI>
struct Smem {
    static constexpr int KB = DI / 64;                       // 128-byte K sub-tiles per row
    static constexpr int Q_BYTES = 2 * KB * kSub;
    static constexpr int K_BYTES = KB * kSub;
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_BAR = OFF_K + kStages * K_BYTES;
    static constexpr int OFF_SBS = OFF_BAR + 256;
    static constexpr int BYTES = OFF_SBS + kSelFloats * 4;
    // request at least ~120 KB so one CTA (which takes all 512 TMEM columns) runs per SM
    static constexpr int ALLOC = (BYTES + 1024 > 120 * 1024 ? BYTES + 1024 : 120 * 1024);
};

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
index_scores_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       Problem p, float *__restrict__ bs, int32_t *__restrict__ sel,
                       unsigned long long *__restrict__ cand, int span, DeviceStatus *st)
{
    using S = Smem<DI>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset from the __shared__ array itself, so every access through `smem`
    // stays a shared-memory access (no generic addressing)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;
    uint8_t *sK = smem + S::OFF_K;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    float *sbs = reinterpret_cast<float *>(smem + S::OFF_SBS);
    uint64_t *full = bars, *empty = bars + kStages, *q_full = bars + 2 * kStages;
    uint64_t *acc_full = q_full + 1, *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int b = blockIdx.z;
    const int rows_total = p.Nq * p.Hkv;
    const int tile = gridDim.x - 1 - blockIdx.x;     // heavy (late) tiles first
    const int row0 = tile * kTileRows;
    const int rows_here = min(kTileRows, rows_total - row0);
    const int mt = rows_here > 128 ? 2 : 1;
    const long long pos_first = (long long)p.q_offset + row0 / p.Hkv;
    const long long pos_last = (long long)p.q_offset + (row0 + rows_here - 1) / p.Hkv;
    const int c_all = (int)(min(pos_last, (long long)p.Nk - 1) / 128) + 1;
    const int c_begin = blockIdx.y * span;
    const int c_end = min(c_all, c_begin + span);
    if (c_begin >= c_end) return;
    const int nblk = c_end - c_begin;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(q_full, 1);
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&acc_full[a], 1);
            tc::mbar_init(&acc_empty[a], kEpiWarps);
        }
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
        {
            // ---------------- TMA producer (warp-uniform; one elect.sync lane issues)
            if (tc::elect_one()) {
                tc::prefetch_tmap(&tmap_q);
                tc::prefetch_tmap(&tmap_k);
                tc::mbar_arrive_expect_tx(q_full, mt * S::KB * kSub);
                for (int m = 0; m < mt; ++m)
                    for (int kb = 0; kb < S::KB; ++kb)
                        tc::tma_load_3d(sQ + (m * S::KB + kb) * kSub, &tmap_q, q_full, kb * 64, row0 + m * 128, b);
            }
            __syncwarp();
            int issued = 0;
            for (int n = 0; n < nblk; ++n) {
                const int s = n % kStages;
                const uint32_t ph = (uint32_t)(n / kStages) & 1u;
                if (!tc::mbar_wait_warp(&empty[s], ph ^ 1u, st, 11, abort_flag)) break;
                if (tc::elect_one()) {
                    tc::mbar_arrive_expect_tx(&full[s], S::KB * kSub);
                    for (int kb = 0; kb < S::KB; ++kb)
                        tc::tma_load_3d(sK + s * S::K_BYTES + kb * kSub, &tmap_k, &full[s], kb * 64,
                                        (c_begin + n) * 128, b);
                }
                __syncwarp();
                issued = n + 1;
            }
            if (*abort_flag) {
                // let this CTA's own copies land before it exits (bounded waits)
                tc::mbar_wait(q_full, 0, nullptr, 0, nullptr);
                for (int n = max(0, issued - kStages); n < issued; ++n)
                    tc::mbar_wait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, nullptr, 0, nullptr);
            }
        }
    } else if (warp == 1) {
        {
            // ---------------- MMA issuer (warp-uniform; one elect.sync lane issues)
            bool ok = tc::mbar_wait_warp(q_full, 0, st, 12, abort_flag);
            const uint64_t dq = tc::sdesc_k128(smem_u32(sQ));
            int issued = 0;
            for (int n = 0; ok && n < nblk; ++n) {
                const int s = n % kStages;
                const uint32_t ph = (uint32_t)(n / kStages) & 1u;
                const int a = n & 1;
                const uint32_t aph = (uint32_t)(n >> 1) & 1u;
                if (!tc::mbar_wait_warp(&acc_empty[a], aph ^ 1u, st, 13, abort_flag)) break;
                if (!tc::mbar_wait_warp(&full[s], ph, st, 14, abort_flag)) break;
                tc::fence_after_sync();
                const uint64_t dk = tc::sdesc_k128(smem_u32(sK + s * S::K_BYTES));
                if (tc::elect_one()) {
                    for (int m = 0; m < mt; ++m) {
                        const uint32_t d = tmem + (uint32_t)((a * 2 + m) * 128);
#pragma unroll
                        for (int ks = 0; ks < DI / 16; ++ks) {
                            const uint32_t off = (ks >> 2) * kSub + (ks & 3) * 32;
                            tc::mma_bf16(d, tc::desc_adv(dq, m * S::KB * kSub + off), tc::desc_adv(dk, off), kIdesc,
                                         ks > 0);
                        }
                    }
                    tc::mma_commit(&empty[s]);
                    tc::mma_commit(&acc_full[a]);
                }
                __syncwarp();
                issued = n + 1;
            }
            if (*abort_flag && issued > 0) {
                // MMAs complete in order: waiting for the last batch drains them all
                const int n = issued - 1;
                tc::mbar_wait(&acc_full[n & 1], (uint32_t)(n >> 1) & 1u, nullptr, 0, nullptr);
            }
        }
    } else {
        // ---------------- epilogue: warp -> (tile m, lane quarter q)
        const int e = warp - 2;
        const int m = e >> 2;
        const int q = warp & 3;
        const int row = m * 128 + q * 32 + lane;
        const int rho = row0 + row;
        const bool valid = rho < rows_total && m < mt;
        const long long pos = (long long)p.q_offset + (valid ? rho / p.Hkv : 0);
        const int c_last = valid ? (int)min((long long)c_end - 1, pos / 128) : -1;   // last block this row sees
        const int c0 = (int)(pos / 128);           // the row's local block
        float *out = bs ? bs + ((long long)b * rows_total + (valid ? rho : 0)) * p.nb : nullptr;
        // fused selection: the 16 best earlier blocks, descending by score
        float tv[16];
        int ti[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            tv[x] = -INFINITY;
            ti[x] = 0;
        }
        const bool vec_ok = (p.nb & 7) == 0;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        float grp[8];
        for (int n0 = 0; n0 < nblk; n0 += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int n = n0 + u;
                grp[u] = 0.f;
                if (n >= nblk) break;
                const int a = n & 1;
                const uint32_t aph = (uint32_t)(n >> 1) & 1u;
                if (!tc::mbar_wait(&acc_full[a], aph, st, 15, abort_flag)) { n0 = nblk; break; }
                tc::fence_after_sync();
                const int c = c_begin + n;
                const long long j0 = (long long)c * 128;
                float mx = -INFINITY;
                if (m < mt) {
                    const bool full_vis = (j0 + 127 <= pos_first) && (j0 + 128 <= p.Nk);
                    // last visible key offset of the block for this row (masked blocks only)
                    const int lim = (int)max(-1LL, min(min(pos, (long long)p.Nk - 1) - j0, 127LL));
                    const uint32_t base = tmem + lane_base + (uint32_t)((a * 2 + m) * 128);
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent max chains
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t v0[32], v1[32];
                        tc::tmem_ld32_nowait(base + h * 64, v0);
                        tc::tmem_ld32_nowait(base + h * 64 + 32, v1);
                        tc::tmem_wait32(v0);
                        tc::tmem_wait32(v1);
                        if (h == 1) {
                            // the accumulator is in registers: hand it back to the MMA
                            tc::fence_before_sync();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
                        }
                        if (full_vis) {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj)
                                m4[jj & 3] = fmaxf(m4[jj & 3], fmaxf(__uint_as_float(v0[jj]), __uint_as_float(v1[jj])));
                        } else {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) {
                                const int jo = h * 64 + jj;
                                const float a0 = jo <= lim ? __uint_as_float(v0[jj]) : -INFINITY;
                                const float a1 = jo + 32 <= lim ? __uint_as_float(v1[jj]) : -INFINITY;
                                m4[jj & 3] = fmaxf(m4[jj & 3], fmaxf(a0, a1));
                            }
                        }
                    }
                    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                } else {
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
                }
                grp[u] = mx * p.scale_idx;   // a positive scale commutes with max
                if (sel) {
                    const int c = c_begin + n;
                    const float sc = (valid && c < c0) ? grp[u] : -INFINITY;
                    if (__any_sync(0xffffffffu, sc > tv[15])) {
                        if (sc > tv[15]) {
                            tv[15] = sc;
                            ti[15] = c;
                        }
#pragma unroll
                        for (int x = 15; x > 0; --x) {
                            if (tv[x] > tv[x - 1]) {
                                const float t0 = tv[x];
                                tv[x] = tv[x - 1];
                                tv[x - 1] = t0;
                                const int t1 = ti[x];
                                ti[x] = ti[x - 1];
                                ti[x - 1] = t1;
                            }
                        }
                    }
                }
            }
            // store this row's scores for blocks c_begin+n0 .. (at most 8)
            const int c_lo = c_begin + n0;
            const int c_hi = min(c_lo + 7, c_last);
            if (cand && valid) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (n0 + u < nblk) sbs[row * span + n0 + u] = grp[u];
            }
            if (out && valid && c_hi >= c_lo) {
                if (vec_ok && c_hi == c_lo + 7) {
                    float4 *o4 = reinterpret_cast<float4 *>(out + c_lo);
                    o4[0] = make_float4(grp[0], grp[1], grp[2], grp[3]);
                    o4[1] = make_float4(grp[4], grp[5], grp[6], grp[7]);
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c_lo + u <= c_hi) out[c_lo + u] = grp[u];
                }
            }
        }
        if (cand) {
            // the slice's 16 best earlier blocks of each row, descending, as
            // ranking keys: warp e takes rows e, e + 8, ..., 32 scores at a time
            // sorted and merged into a running top-32
            named_bar_sync(1, kEpiWarps * 32);
            for (int rl = e; rl < rows_here; rl += kEpiWarps) {
                const int rr = row0 + rl;
                const long long pr = (long long)p.q_offset + rr / p.Hkv;
                const int ce = (int)min((long long)c_end, pr / 128) - c_begin;   // slice blocks before c0
                unsigned long long best = 0ull;
                for (int nn = 0; nn < ce; nn += 32) {
                    const int n = nn + lane;
                    unsigned long long key = n < ce ? block_key(sbs[rl * span + n], c_begin + n) : 0ull;
                    key = sort_desc64(key, lane);
                    const unsigned long long rev = shfl64(key, 31 - lane);
                    best = merge_desc64(best > rev ? best : rev, lane);
                }
                if (lane < 16) cand[(((long long)b * rows_total + rr) * gridDim.y + blockIdx.y) * 16 + lane] = best;
            }
        }
        if (sel && valid) {
            const int k = p.topk, i = rho / p.Hkv, r = rho % p.Hkv;
            int32_t *o = sel + (((long long)b * p.Hkv + r) * p.Nq + i) * k;
            int id[16];
#pragma unroll
            for (int x = 0; x < 16; ++x)
                id[x] = c0 + 1 <= k ? (x <= c0 ? x : 0x7fffffff) : (x < k - 1 ? ti[x] : (x == k - 1 ? c0 : 0x7fffffff));
            // ascending bitonic network over the 16 registers
#pragma unroll
            for (int size = 2; size <= 16; size <<= 1)
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int y = x ^ stride;
                        if (y > x) {
                            const bool up = (x & size) == 0;
                            if ((id[x] > id[y]) == up) {
                                const int t = id[x];
                                id[x] = id[y];
                                id[y] = t;
                            }
                        }
                    }
#pragma unroll
            for (int x = 0; x < 16; ++x)
                if (x < k) o[x] = id[x] == 0x7fffffff ? -1 : id[x];
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Row tiles and the block range each CTA covers: a tile's range is split
// when there are too few tiles to fill the GPU (slices start on 8-block
// boundaries).
void plan_grid(const Problem &p, int &tiles, int &splits, int &span)
{
    const long long rows_total = (long long)p.Nq * p.Hkv;
    tiles = (int)((rows_total + kTileRows - 1) / kTileRows);
    splits = 1;
    const long long ctas = (long long)tiles * p.B;
    if (ctas < (long long)p.num_sms) splits = (int)min((long long)(p.nb + 7) / 8, (p.num_sms + ctas - 1) / ctas);
    span = (p.nb + splits - 1) / splits;
    span = (span + 7) & ~7;
    splits = (p.nb + span - 1) / span;
}

// bs: scores out (nullptr: not stored); sel: selection out (fused form; the
// caller has checked that it applies); cand: per-slice candidate keys out
// (split form)
template <int DI>
cudaError_t launch_t(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs, int32_t *sel,
                     unsigned long long *cand, DeviceStatus *st, cudaStream_t s)
{
    using S = Smem<DI>;
    const long long rows_total = (long long)p.Nq * p.Hkv;
    CUtensorMap tq, tk;
    cudaError_t e = make_tmap_bf16_3d(&tq, q_idx, DI, rows_total, p.B, DI * 2ull, rows_total * DI * 2ull, 64, 128);
    if (e != cudaSuccess) return e;
    e = make_tmap_bf16_3d(&tk, k_idx, DI, p.kv_rows, p.B, DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull, 64,
                          128);
    if (e != cudaSuccess) return e;
    int tiles, splits, span;
    plan_grid(p, tiles, splits, span);
    e = cudaFuncSetAttribute(index_scores_tc_kernel<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e != cudaSuccess) return e;
    {
        TimedLaunch timed_("index_scores_tc_kernel", s);
        index_scores_tc_kernel<DI><<<dim3(tiles, splits, p.B), kThreads, S::ALLOC, s>>>(tq, tk, p, bs, sel, cand, span, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_scores(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs,
                                DeviceStatus *st, cudaStream_t s)
{
    return p.d_idx == 128 ? launch_t<128>(p, q_idx, k_idx, bs, nullptr, nullptr, st, s)
                          : launch_t<64>(p, q_idx, k_idx, bs, nullptr, nullptr, st, s);
}

// Split selection: rows split across CTAs, k <= 16, and each CTA's rows x
// slice of block scores fit the shared-memory buffer.
bool index_select_split(const Problem &p)
{
    int tiles, splits, span;
    plan_grid(p, tiles, splits, span);
    const long long rows = std::min((long long)kTileRows, (long long)p.Nq * p.Hkv);
    return splits > 1 && p.topk <= 16 && rows * span <= kSelFloats;
}

size_t index_select_scratch_floats(const Problem &p)
{
    // what the path launch_index_select takes (no scores asked for) reads and
    // writes: nothing when the selection is fused into the score kernel, the
    // per-slice candidate keys when rows are split across CTAs, else the
    // block scores between the score kernel and the top-k kernel
    if (index_select_fused(p)) return 0;
    const size_t rows = (size_t)p.B * p.Nq * p.Hkv;
    if (index_select_split(p)) {
        int tiles, splits, span;
        plan_grid(p, tiles, splits, span);
        return rows * (size_t)splits * 16 * 2;             // 16 8-byte keys per (row, slice)
    }
    return rows * (size_t)p.nb;                            // block scores
}

bool index_select_fused(const Problem &p)
{
    int tiles, splits, span;
    plan_grid(p, tiles, splits, span);
    return splits == 1 && p.topk <= 16;   // every CTA sees all blocks of its rows
}

cudaError_t launch_index_select(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs_out,
                                float *bs_scratch, int32_t *sel, DeviceStatus *st, cudaStream_t s)
{
    if (index_select_fused(p))   // every CTA sees all blocks of its rows: fused selection
        return p.d_idx == 128 ? launch_t<128>(p, q_idx, k_idx, bs_out, sel, nullptr, st, s)
                              : launch_t<64>(p, q_idx, k_idx, bs_out, sel, nullptr, st, s);
    if (!bs_out && bs_scratch && index_select_split(p)) {
        // rows split across CTAs, scores not wanted: each CTA leaves its slice's
        // 16 best blocks per row (the scratch holds index_select_scratch_floats),
        // then a second kernel merges the slices' lists
        int tiles, splits, span;
        plan_grid(p, tiles, splits, span);
        unsigned long long *cand = reinterpret_cast<unsigned long long *>(bs_scratch);
        cudaError_t e = p.d_idx == 128 ? launch_t<128>(p, q_idx, k_idx, nullptr, nullptr, cand, st, s)
                                       : launch_t<64>(p, q_idx, k_idx, nullptr, nullptr, cand, st, s);
        if (e != cudaSuccess) return e;
        return launch_block_topk_merge(p, cand, splits, span, sel, s);
    }
    float *bs = bs_out ? bs_out : bs_scratch;
    cudaError_t e = launch_index_scores(p, q_idx, k_idx, bs, st, s);
    if (e != cudaSuccess) return e;
    return launch_block_topk(p, bs, sel, st, s);
}

}  // namespace msa
