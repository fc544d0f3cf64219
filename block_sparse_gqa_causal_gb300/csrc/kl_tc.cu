// kl_tc.cu -- KL alignment loss of MSA, key-major on the tcgen05 tensor cores.
//
// "Sparse Attention · Part II", section 3.2 (the L_KL equation): for query i
// and group r over the selected token set T, with the detached teacher
// Pt_j = (1/G) sum_h exp(l_{h,j} - lse_h) and the student Ps = softmax_T(s),
//   KL = sum_j Pt_j log Pt_j - sum_j Pt_j s_j + log sum_j exp(s_j).
// Every term is a sum over T, so it splits over the selected blocks.  This
// file holds the index pass over the buckets of the inverse index (the
// queries that selected each (b, group, block)), each CTA keeping one
// 128-token block of K_idx on chip:
//   s = q_idx K_idx^T (M = 128 queries, N = 128 keys).  With queries on the
//   TMEM lanes every sum over the block's keys stays in one thread:
//     (max s2, sum 2^(s2 - max s2))   (s2 = s log2 e)
//   per (query, group, selected block, half of the keys),
// and the combine that folds a row's partials in a fixed order into lse_idx
// (reproducible; no atomics).  The teacher terms sum_j Pt_j (log2 Pt_j - s2)
// come from index_teacher_tc.cu, which rebuilds the teacher from its own
// logit tiles next to the index scores, so no distribution is stored.
// Training runs the index pass alone (lse_idx, which the backward needs
// first); the fused backward returns the loss.
#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kKeys = 128;
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

// ============================================================== index pass
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

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
kl_index_tc_kernel(const __grid_constant__ CUtensorMap tmap_ki, Problem p, const bf16 *__restrict__ q_idx,
                   const int32_t *__restrict__ bucket_off, const int32_t *__restrict__ bucket_q,
                   float2 *__restrict__ part, DeviceStatus *st)
{
    using L = IndexLayout<DI>;
    using Meta = typename L::Meta;
    // the (group, block) bucket of this CTA (visiting order: bucket_of)
    int r, c;
    bucket_of((int)blockIdx.x, p.Hkv, p.nb, p.num_sms, r, c);
    const int b = blockIdx.y;
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
        {
            // ------------------------------------------------ MMA issuer: s = q_idx K_idx^T
            // (warp-uniform; one elect.sync lane issues)
            constexpr uint32_t I_S = tc::idesc_bf16(128, kKeys);
            const uint64_t dKI = tc::sdesc_k128(smem_u32(sm + L::OFF_KI));
            bool ok = wwait(kv_full, 0, st, 86, abort_flag);
            for (int n = 0; ok && n < nch; ++n) {
                if (!wwait(&full[n % kStages], (uint32_t)(n / kStages) & 1u, st, 87, abort_flag)) break;
                if (n >= 2 && !wwait(&s_free[n & 1], ((uint32_t)(n >> 1) & 1u) ^ 1u, st, 88, abort_flag)) break;
                tc::fence_proxy_async();
                tc::fence_after_sync();
                const uint64_t dQ = tc::sdesc_k128(smem_u32(sm + L::OFF_Q + (n % kStages) * (L::H * SUB)));
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < DI / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * SUB + (ks & 3) * 32;
                        tc::mma_bf16(tmem + (n & 1) * kKeys, tc::desc_adv(dQ, off), tc::desc_adv(dKI, off), I_S, ks > 0);
                    }
                    tc::mma_commit(&s_full[n & 1]);
                    tc::mma_commit(&empty[n % kStages]);
                }
                __syncwarp();
            }
            if (tc::elect_one()) tc::mma_commit(done);
            __syncwarp();
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
            const int nq = meta->nq;
            const bool valid = u < nq;
            const long long pos = valid ? (long long)meta->pos[u] : -1;
            const int qi = meta->qi[u], slot = meta->slot[u];
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
            float Z = 0.f;
#pragma unroll
            for (int x = 0; x < 64; ++x)
                if (x < nvis) Z += tc::ex2(__uint_as_float(sv[x >> 5][x & 31]) * si2 - M);
            if (valid) {
                const long long row = ((long long)b * p.Hkv + r) * p.Nq + qi;
                part[(row * p.topk + slot) * kParts + hf] = make_float2(M, Z);
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
// order: lse_idx = (M + log2 Z) ln 2.
template <int MAXK>   // an upper bound of topk: the row's partials stay in registers
__global__ void kl_combine_kernel(Problem p, const int32_t *__restrict__ sel, const float2 *__restrict__ part,
                                  float *__restrict__ lse_idx)
{
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= (long long)p.B * p.Hkv * p.Nq) return;
    const int i = (int)(row % p.Nq);
    const long long pos = (long long)p.q_offset + i;
    const int32_t *srow = sel + row * p.topk;
    // the row's partials, both key halves of a slot in one 16-byte load, read once
    static_assert(kParts == 2, "one float4 per slot");
    const float4 *prow = reinterpret_cast<const float4 *>(part + row * p.topk * kParts);
    float4 v[MAXK];
    bool ok[MAXK];
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < MAXK; ++t) {
        ok[t] = false;
        if (t < p.topk) {
            const int cc = srow[t];
            ok[t] = cc >= 0 && cc < p.nb && (long long)cc * 128 <= pos;
            if (ok[t]) {
                v[t] = __ldg(prow + t);
                M = fmaxf(fmaxf(M, v[t].x), v[t].z);
            }
        }
    }
    float Z = 0.f;
#pragma unroll
    for (int t = 0; t < MAXK; ++t) {
        if (ok[t]) {
            if (v[t].y > 0.f) Z += v[t].y * exp2f(v[t].x - M);
            if (v[t].w > 0.f) Z += v[t].w * exp2f(v[t].z - M);
        }
    }
    lse_idx[row] = (M + log2f(Z)) * kLn2;
}

template <int DI>
cudaError_t launch_index(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, const KlWork &w, DeviceStatus *st,
                         cudaStream_t s)
{
    using L = IndexLayout<DI>;
    cudaError_t e = cudaFuncSetAttribute(kl_index_tc_kernel<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    CUtensorMap tki;
    const unsigned long long di[3] = {(unsigned long long)DI, (unsigned long long)p.Nk, (unsigned long long)p.B};
    const unsigned long long si[2] = {DI * 2ull, (unsigned long long)p.kv_rows * DI * 2ull};
    const unsigned bi[3] = {64, (unsigned)kKeys, 1};
    if ((e = make_tmap_bf16(&tki, k_idx, 3, di, si, bi)) != cudaSuccess) return e;
    {
        TimedLaunch timed_("kl_index_tc_kernel", s);
        kl_index_tc_kernel<DI><<<dim3(p.Hkv * p.nb, p.B), kThreads, L::ALLOC, s>>>(tki, p, q_idx, w.bucket_off,
                                                                                  w.bucket_q, w.part, st);
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
    if (kl_rows && (!w.klt || !bwd_tc(p))) return cudaErrorInvalidValue;
    cudaError_t e = w.index_ready ? cudaSuccess
                                  : launch_inverse_index(p, sel, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, st, s);
    if (e != cudaSuccess) return e;
    e = p.d_idx == 128 ? launch_index<128>(p, q_idx, k_idx, w, st, s) : launch_index<64>(p, q_idx, k_idx, w, st, s);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Hkv * p.Nq;
    {
        TimedLaunch timed_("kl_combine_kernel", s);
        if (p.topk <= 16) kl_combine_kernel<16><<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p, sel, w.part, lse_idx);
        else kl_combine_kernel<32><<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p, sel, w.part, lse_idx);
    }
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess || !kl_rows) return e;
    // the teacher terms per (query, group, slot), then the rows
    e = launch_index_teacher_tc(p, q, k, q_idx, k_idx, lse, nullptr, 0.f, w.bucket_off, w.bucket_q, w.klt, nullptr,
                                nullptr, st, s);
    if (e != cudaSuccess) return e;
    return launch_kl_rows_combine(p, sel, lse_idx, w.klt, kl_rows, s);
}

}  // namespace msa
