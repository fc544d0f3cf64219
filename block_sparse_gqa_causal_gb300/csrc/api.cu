// api.cu -- the C-ABI of libmsa.so (declared in include/msa.h): argument
// validation, workspace carve-up and kernel launches on the caller's stream.
#include <algorithm>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "msa.h"
#include "msa_internal.h"

using namespace msa;

namespace {

thread_local std::string g_err;
std::atomic<unsigned long long> g_launches{0};

msa_status fail(msa_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

msa_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void *ptr) { return ((uintptr_t)ptr & 15u) == 0; }

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

// Validates the shape and fills the internal problem description.
msa_status make_problem(const msa_shape *s, Problem &p)
{
    if (!s) return fail(MSA_ERR_INVALID_ARGUMENT, "shape is NULL");
    if (s->B < 1 || s->Nq < 1 || s->Nk < 1 || s->Hq < 1 || s->Hkv < 1 || s->d < 1 || s->d_idx < 1 ||
        s->block < 1 || s->topk < 1 || s->q_offset < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "shape has a non-positive size (B=%d Nq=%d Nk=%d Hq=%d Hkv=%d d=%d "
                    "d_idx=%d block=%d topk=%d q_offset=%d)", s->B, s->Nq, s->Nk, s->Hq, s->Hkv, s->d, s->d_idx,
                    s->block, s->topk, s->q_offset);
    if ((long long)s->q_offset + s->Nq > s->Nk)
        return fail(MSA_ERR_INVALID_ARGUMENT, "q_offset + Nq (%lld) exceeds Nk (%d): a visible key is missing",
                    (long long)s->q_offset + s->Nq, s->Nk);
    if (s->Hq % s->Hkv != 0) return fail(MSA_ERR_INVALID_ARGUMENT, "Hq (%d) is not a multiple of Hkv (%d)", s->Hq, s->Hkv);
    const long long kv_rows = s->kv_rows ? s->kv_rows : s->Nk;
    if (kv_rows < s->Nk) return fail(MSA_ERR_INVALID_ARGUMENT, "kv_rows (%lld) < Nk (%d)", kv_rows, s->Nk);
    if (s->block != 128) return fail(MSA_ERR_UNSUPPORTED, "block must be 128 (got %d)", s->block);
    if (s->d != 64 && s->d != 128) return fail(MSA_ERR_UNSUPPORTED, "d must be 64 or 128 (got %d)", s->d);
    if (s->d_idx != 64 && s->d_idx != 128) return fail(MSA_ERR_UNSUPPORTED, "d_idx must be 64 or 128 (got %d)", s->d_idx);
    if (s->topk > 32) return fail(MSA_ERR_UNSUPPORTED, "topk must be <= 32 (got %d)", s->topk);
    const int G = s->Hq / s->Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return fail(MSA_ERR_UNSUPPORTED, "Hq/Hkv must be 1, 2, 4 or 8 (got %d)", G);
    if (!(s->scale >= 0.f) || !(s->scale_idx >= 0.f) || isinf(s->scale) || isinf(s->scale_idx))
        return fail(MSA_ERR_INVALID_ARGUMENT, "scales must be finite and >= 0 (0 selects the default)");
    if ((long long)s->B * s->Nq * s->Hq >= (1LL << 31) / 128 || kv_rows * s->B >= (1LL << 31))
        return fail(MSA_ERR_UNSUPPORTED, "problem too large for 32-bit row indices");
    p.B = s->B; p.Nq = s->Nq; p.Nk = s->Nk; p.q_offset = s->q_offset; p.Hq = s->Hq; p.Hkv = s->Hkv;
    p.G = G; p.d = s->d; p.d_idx = s->d_idx; p.block = s->block; p.topk = s->topk;
    p.nb = (s->Nk + s->block - 1) / s->block;
    p.kv_rows = kv_rows;
    p.scale = s->scale > 0.f ? s->scale : 1.0f / sqrtf((float)s->d);
    p.scale_idx = s->scale_idx > 0.f ? s->scale_idx : 1.0f / sqrtf((float)s->d_idx);
    p.num_sms = sm_count();
    return MSA_OK;
}

struct Carve {
    char *base;
    size_t off = kStatusBytes;
    template <class T>
    T *take(size_t count)
    {
        T *ptr = reinterpret_cast<T *>(base + off);
        off = align256(off + count * sizeof(T));
        return ptr;
    }
};

// The forward and the KL group work by key block when the average selected
// block is shared by enough queries to fill 128-row tiles (prefill); with few
// queries per block (decode) they stream each query's blocks instead.
bool fwd_keymajor(const Problem &p) { return (long long)p.Nq * p.topk >= 8LL * p.nb; }

// selection scratch: block scores, or the split selection's candidate keys
size_t bs_bytes(const Problem &p) { return align256(index_select_scratch_floats(p) * sizeof(float)); }

// inverse index: counts, offsets, per-CTA scratch, query lists
size_t index_bytes(const Problem &p)
{
    const size_t nbk = (size_t)p.B * p.Hkv * p.nb;
    return 2 * align256((nbk + 1) * 4) + align256(inverse_index_scratch_ints(p) * 4) +
           align256((size_t)p.B * p.Hkv * p.Nq * p.topk * 4);
}

template <class W>
void carve_index(Carve &cv, const Problem &p, W &w)
{
    const size_t nbk = (size_t)p.B * p.Hkv * p.nb;
    w.bucket_cnt = cv.take<int32_t>(nbk + 1);
    w.bucket_off = cv.take<int32_t>(nbk + 1);
    w.bucket_scratch = cv.take<int32_t>(inverse_index_scratch_ints(p));
    w.bucket_q = cv.take<int32_t>((size_t)p.B * p.Hkv * p.Nq * p.topk);
}

size_t fwd_bytes(const Problem &p)
{
    if (!fwd_keymajor(p)) {
        // split-KV partial states (decode: too few rows to fill the GPU)
        const int ns = sparse_attn_splits(p);
        if (ns == 1) return 0;
        const size_t rows = (size_t)p.B * p.Nq * p.Hq * ns;
        return align256(rows * p.d * 4 + rows * 8);
    }
    const size_t rows = (size_t)p.B * p.Nq * p.Hq * p.topk;
    return align256(rows * p.d * 2) + align256(rows * 8) + index_bytes(p);
}
size_t klrows_bytes(const Problem &p) { return align256((size_t)p.B * p.Hkv * p.Nq * sizeof(float)); }
// KL teacher terms: four floats per (query, group, slot)
size_t klt_bytes(const Problem &p) { return align256((size_t)p.B * p.Hkv * p.Nq * p.topk * 16); }

// The KL forward runs key-major (the teacher rebuilt on the tensor cores next
// to the index scores) where the forward does; the rest (decode shapes)
// streams query by query.
bool kl_teacher_keymajor(const Problem &p) { return fwd_keymajor(p) && bwd_tc(p); }
size_t kl_bytes(const Problem &p, bool lse_only)
{
    if (!fwd_keymajor(p) || (!lse_only && !kl_teacher_keymajor(p))) return 0;
    return align256(kl_part_count(p) * sizeof(float2)) + (lse_only ? 0 : klt_bytes(p)) + index_bytes(p);
}

// backward: D, each group's fp32 dK_idx share, the inverse index and the
// per-slot dQ / dq_idx partial rows
size_t bwd_bytes(const Problem &p)
{
    const size_t dki = (size_t)p.B * p.Nk * p.d_idx * 4 * (size_t)p.Hkv;
    const size_t slots = (size_t)p.B * p.Nq * p.topk;
    return align256((size_t)p.B * p.Hq * p.Nq * 4) + align256(dki) + index_bytes(p) +
           align256(slots * p.Hq * p.d * 2) + align256(slots * p.Hkv * p.d_idx * 2);
}

// KL of the fused backward: rows (when the caller gives none) and the per-slot
// teacher terms
size_t bwdkl_bytes(const Problem &p) { return klrows_bytes(p) + klt_bytes(p); }

// one training step: the shared inverse index and D (the forward's combine
// leaves it for the backward) for the whole step, then one region that each
// phase's own buffers overlay in turn -- the selection's score scratch
// (unfused selection only), the forward's partial rows, the KL index pass's
// partials, the backward's dK_idx shares, partial rows and KL terms: each
// phase's partials are combined before the next phase writes (stream
// order).  Shapes outside the shared-index path run the four phases one
// after another in the same workspace, so the largest suffices.
bool train_shared_index(const Problem &p) { return fwd_keymajor(p) && bwd_tc(p); }
size_t train_phase_bytes(const Problem &p)
{
    const size_t rows = (size_t)p.B * p.Nq * p.Hq * p.topk, slots = (size_t)p.B * p.Nq * p.topk;
    const size_t fwd = align256(rows * p.d * 2) + align256(rows * 8);
    const size_t kl = align256(kl_part_count(p) * sizeof(float2));
    const size_t bwd = align256((size_t)p.B * p.Hkv * p.Nk * p.d_idx * 4) + align256(slots * p.Hq * p.d * 2) +
                       align256(slots * p.Hkv * p.d_idx * 2) + bwdkl_bytes(p);
    return std::max(std::max(bs_bytes(p), fwd), std::max(kl, bwd));
}
size_t train_bytes(const Problem &p)
{
    if (!train_shared_index(p)) {
        size_t n = bs_bytes(p);
        n = std::max(n, fwd_bytes(p));
        n = std::max(n, klrows_bytes(p) + kl_bytes(p, true));
        return std::max(n, bwd_bytes(p) + bwdkl_bytes(p));
    }
    return index_bytes(p) + align256((size_t)p.B * p.Hq * p.Nq * 4) + train_phase_bytes(p);
}

// The dense indexer warm-up runs the block-sparse kernels on the selection of
// every visible block: topk = nb (at most 32 blocks: 4,096 tokens), the
// tensor-core teacher and backward, a training sequence.
bool warmup_shape_ok(const Problem &p)
{
    return p.q_offset == 0 && p.Nq == p.Nk && p.kv_rows == p.Nk && bwd_tc(p) && p.nb <= 32;
}
Problem warmup_problem(const Problem &p)
{
    Problem w = p;
    w.topk = p.nb;
    return w;
}
size_t warmup_bytes(const Problem &p0)
{
    const Problem p = warmup_problem(p0);
    const size_t slots = (size_t)p.B * p.Nq * p.topk;               // per (b, query), all groups below
    const size_t rows = slots * p.Hq;
    return align256(slots * p.Hkv * 4) + index_bytes(p)              // selection, inverse index
           + align256((size_t)p.B * p.Nq * p.Hq * p.d * 2)           // the forward's output (not returned)
           + align256(rows * p.d * 2) + align256(rows * 8)          // forward partials
           + align256(kl_part_count(p) * sizeof(float2)) + klt_bytes(p) + klrows_bytes(p)
           + align256(slots * p.Hkv * p.d_idx * 2)                   // dq_idx partial rows
           + align256((size_t)p.B * p.Hkv * p.Nk * p.d_idx * 4);     // dK_idx shares per group
}

#define REQUIRE_PTR(ptr, name)                                                                         \
    do {                                                                                               \
        if (!(ptr)) return fail(MSA_ERR_INVALID_ARGUMENT, "%s is NULL", name);                         \
        if (!aligned16(ptr)) return fail(MSA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", name); \
    } while (0)

msa_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws) return fail(MSA_ERR_INVALID_ARGUMENT, "workspace is NULL");
    if (((uintptr_t)ws & 255u) != 0) return fail(MSA_ERR_INVALID_ARGUMENT, "workspace is not 256-byte aligned");
    if (ws_bytes < need) return fail(MSA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    return MSA_OK;
}

}  // namespace

namespace msa {
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {
struct TimingRec {
    std::string name;
    cudaEvent_t a = nullptr, b = nullptr;
};
std::mutex g_tmu;
bool g_timing = false;
std::vector<TimingRec> g_trecs;   // events are created once and reused
size_t g_tused = 0;
}  // namespace

TimedLaunch::TimedLaunch(const char *name, cudaStream_t s) : slot(-1), stream(s)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    if (!g_timing) return;
    if (g_tused == g_trecs.size()) {
        TimingRec r;
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
        g_trecs.push_back(r);
    }
    TimingRec &r = g_trecs[g_tused];
    r.name = name;
    if (cudaEventRecord(r.a, s) != cudaSuccess) return;
    slot = (long)g_tused++;
}

TimedLaunch::~TimedLaunch()
{
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_tmu);
    cudaEventRecord(g_trecs[(size_t)slot].b, stream);
}
msa_status problem_from_shape(const msa_shape *shape, Problem &p) { return make_problem(shape, p); }
msa_status set_error(msa_status st, const char *msg) { return fail(st, "%s", msg); }
}  // namespace msa

extern "C" {

const char *msa_version(void) { return "msa-gb300 0.1 (sm_103a)"; }

const char *msa_last_error(void) { return g_err.c_str(); }

unsigned long long msa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int msa_kernel_timing(int enable)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    const int prev = g_timing ? 1 : 0;
    g_timing = enable != 0;
    g_tused = 0;
    return prev;
}

size_t msa_kernel_timing_report(char *buf, size_t len)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    std::vector<std::pair<std::string, std::pair<long, double>>> agg;
    for (size_t x = 0; x < g_tused; ++x) {
        TimingRec &r = g_trecs[x];
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) ms = -1.f;
        size_t k = 0;
        while (k < agg.size() && agg[k].first != r.name) ++k;
        if (k == agg.size()) agg.push_back({r.name, {0, 0.0}});
        agg[k].second.first += 1;
        agg[k].second.second += ms < 0.f ? 0.0 : (double)ms;
    }
    std::string out;
    char line[256];
    for (auto &e : agg) {
        snprintf(line, sizeof line, "%s %ld %.6f\n", e.first.c_str(), e.second.first, e.second.second);
        out += line;
    }
    if (buf && len) {
        const size_t n = out.size() < len - 1 ? out.size() : len - 1;
        memcpy(buf, out.data(), n);
        buf[n] = 0;
    }
    return out.size() + 1;
}

size_t msa_workspace_size(const msa_shape *shape, int op)
{
    Problem p;
    if (make_problem(shape, p) != MSA_OK) return 0;
    switch (op) {
    case MSA_OP_INDEX_SELECT: return kStatusBytes + bs_bytes(p);
    case MSA_OP_SPARSE_ATTN_FWD: return kStatusBytes + fwd_bytes(p);
    case MSA_OP_KL_FWD: return kStatusBytes + klrows_bytes(p) + std::max(kl_bytes(p, false), kl_bytes(p, true));
    case MSA_OP_FUSED_BWD: return kStatusBytes + bwd_bytes(p);
    case MSA_OP_FUSED_BWD_KL: return kStatusBytes + bwd_bytes(p) + bwdkl_bytes(p);
    case MSA_OP_TRAIN_STEP: return kStatusBytes + train_bytes(p);
    case MSA_OP_WARMUP_KL: {
        if (!warmup_shape_ok(p)) {
            fail(MSA_ERR_UNSUPPORTED, "warmup_kl needs q_offset == 0, Nq == Nk == kv_rows and at "
                 "most 32 blocks (Nk <= 4096); got Nk=%d d=%d d_idx=%d", p.Nk, p.d, p.d_idx);
            return 0;
        }
        return kStatusBytes + warmup_bytes(p);
    }
    default: fail(MSA_ERR_INVALID_ARGUMENT, "unknown op %d", op); return 0;
    }
}

msa_status msa_index_select(const msa_shape *shape, const void *q_idx, const void *k_idx, int32_t *sel_idx,
                            float *block_scores, void *workspace, size_t workspace_bytes, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    if (!sel_idx) return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx is NULL");
    if (block_scores && !aligned16(block_scores)) return fail(MSA_ERR_INVALID_ARGUMENT, "block_scores is not 16-byte aligned");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + (block_scores ? 0 : bs_bytes(p)));
    if (st != MSA_OK) return st;
    Carve cv{static_cast<char *>(workspace)};
    float *scratch = block_scores ? nullptr : cv.take<float>(index_select_scratch_floats(p));
    DeviceStatus *ds = static_cast<DeviceStatus *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_index_select(p, static_cast<const bf16 *>(q_idx), static_cast<const bf16 *>(k_idx),
                                        block_scores, scratch, sel_idx, ds, s);
    if (e != cudaSuccess) return cuda_fail(e, "index_select launch");
    return MSA_OK;
}

msa_status msa_sparse_attn_fwd(const msa_shape *shape, const void *q, const void *k, const void *v,
                               const int32_t *sel_idx, void *o, float *lse, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(o, "o");
    if (!sel_idx) return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx is NULL");
    if (!lse) return fail(MSA_ERR_INVALID_ARGUMENT, "lse is NULL");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + fwd_bytes(p));
    if (st != MSA_OK) return st;
    DeviceStatus *ds = static_cast<DeviceStatus *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fwd_keymajor(p)) {
        Carve cv{static_cast<char *>(workspace)};
        const size_t rows = (size_t)p.B * p.Nq * p.Hq * p.topk;
        FwdWork w;
        w.part = cv.take<bf16>(rows * p.d);
        w.stats = cv.take<float2>(rows);
        carve_index(cv, p, w);
        e = launch_sparse_fwd_keymajor(p, static_cast<const bf16 *>(q), static_cast<const bf16 *>(k),
                                       static_cast<const bf16 *>(v), sel_idx, static_cast<bf16 *>(o), lse, w, ds, s);
    } else {
        float *split_ws = nullptr;
        if (sparse_attn_splits(p) > 1) {
            Carve cv{static_cast<char *>(workspace)};
            split_ws = cv.take<float>(fwd_bytes(p) / 4);
        }
        e = launch_sparse_attn_fwd(p, static_cast<const bf16 *>(q), static_cast<const bf16 *>(k),
                                   static_cast<const bf16 *>(v), sel_idx, static_cast<bf16 *>(o), lse, split_ws, ds, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "sparse_attn_fwd launch");
    return MSA_OK;
}

}  // extern "C"

namespace {
// KL forward on carved workspace.  rows == nullptr: lse_idx only (no teacher
// pass, key-major path; the fallback path computes rows into `scratch_rows`).
// kl_loss == nullptr: no reduction.
cudaError_t kl_forward(const Problem &p, const void *q, const void *k, const void *q_idx, const void *k_idx,
                       const int32_t *sel_idx, const float *lse, float kl_coef, float *lse_idx, float *rows,
                       float *scratch_rows, float *kl_loss, Carve &cv, DeviceStatus *ds, cudaStream_t s)
{
    cudaError_t e;
    if (rows ? kl_teacher_keymajor(p) : fwd_keymajor(p)) {
        KlWork w;
        w.part = cv.take<float2>(kl_part_count(p));
        w.klt = rows ? cv.take<float>((size_t)p.B * p.Hkv * p.Nq * p.topk * 4) : nullptr;
        carve_index(cv, p, w);
        e = launch_kl_keymajor(p, static_cast<const bf16 *>(q), static_cast<const bf16 *>(k),
                               static_cast<const bf16 *>(q_idx), static_cast<const bf16 *>(k_idx), sel_idx, lse,
                               lse_idx, rows, w, ds, s);
    } else {
        if (!rows) rows = scratch_rows;
        e = launch_kl_fwd(p, static_cast<const bf16 *>(q), static_cast<const bf16 *>(k),
                          static_cast<const bf16 *>(q_idx), static_cast<const bf16 *>(k_idx), sel_idx, lse, lse_idx,
                          rows, ds, s);
    }
    if (e != cudaSuccess || !kl_loss) return e;
    return launch_kl_reduce(p, rows, kl_coef, kl_loss, s);
}
}  // namespace

extern "C" {

msa_status msa_block_mask(const msa_shape *shape, const int32_t *sel_idx, uint32_t *mask, int32_t *tile_counts,
                          int32_t *tile_blocks, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    if (!sel_idx || !mask) return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx and mask must be non-NULL");
    if (((uintptr_t)sel_idx | (uintptr_t)mask | (uintptr_t)tile_counts | (uintptr_t)tile_blocks) & 3u)
        return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx, mask, tile_counts and tile_blocks must be 4-byte aligned");
    if (block_mask_smem_bytes(p) > 160 * 1024)
        return fail(MSA_ERR_UNSUPPORTED, "block_mask: %d key blocks, more than the supported 655,328", p.nb);
    cudaError_t e = launch_block_mask(p, sel_idx, mask, tile_counts, tile_blocks, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block_mask launch");
    return MSA_OK;
}

msa_status msa_kv_append(const msa_shape *shape, const void *k_new, const void *v_new, const void *k_idx_new,
                         void *k, void *v, void *k_idx, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);   // q_offset + Nq <= Nk <= kv_rows
    if (st != MSA_OK) return st;
    if (!k_new != !k || !v_new != !v || !k_idx_new != !k_idx)
        return fail(MSA_ERR_INVALID_ARGUMENT, "kv_append: give both or neither of each (new rows, cache) pair");
    if (!k && !v && !k_idx) return fail(MSA_ERR_INVALID_ARGUMENT, "kv_append: nothing to append");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_idx_new) || !aligned16(k) || !aligned16(v) ||
        !aligned16(k_idx))
        return fail(MSA_ERR_INVALID_ARGUMENT, "kv_append: pointers must be 16-byte aligned");
    cudaError_t e = launch_kv_append(p, static_cast<const bf16 *>(k_new), static_cast<const bf16 *>(v_new),
                                     static_cast<const bf16 *>(k_idx_new), static_cast<bf16 *>(k),
                                     static_cast<bf16 *>(v), static_cast<bf16 *>(k_idx),
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return MSA_OK;
}

msa_status msa_kl_fwd(const msa_shape *shape, const void *q, const void *k, const void *q_idx, const void *k_idx,
                      const int32_t *sel_idx, const float *lse, float kl_coef, float *lse_idx, float *kl_rows,
                      float *kl_loss, void *workspace, size_t workspace_bytes, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    if (!sel_idx || !lse || !lse_idx) return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx, lse and lse_idx must be non-NULL");
    const bool lse_only = !kl_rows && !kl_loss;
    if (!lse_only && !kl_loss)
        return fail(MSA_ERR_INVALID_ARGUMENT, "kl_loss is NULL (pass kl_rows and kl_loss both NULL for lse_idx only)");
    if (!isfinite(kl_coef)) return fail(MSA_ERR_INVALID_ARGUMENT, "kl_coef must be finite");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + (kl_rows ? 0 : klrows_bytes(p)) + kl_bytes(p, lse_only));
    if (st != MSA_OK) return st;
    Carve cv{static_cast<char *>(workspace)};
    float *scratch = kl_rows ? nullptr : cv.take<float>((size_t)p.B * p.Hkv * p.Nq);
    float *rows = kl_rows ? kl_rows : (lse_only ? nullptr : scratch);
    cudaError_t e = kl_forward(p, q, k, q_idx, k_idx, sel_idx, lse, kl_coef, lse_idx, rows, scratch, kl_loss, cv,
                               static_cast<DeviceStatus *>(workspace), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kl_fwd launch");
    return MSA_OK;
}

}  // extern "C"

namespace {
msa_status fused_bwd_impl(const msa_shape *shape, const void *q, const void *k, const void *v, const void *o,
                          const void *d_o, const float *lse, const void *q_idx, const void *k_idx,
                          const int32_t *sel_idx, const float *lse_idx, float kl_coef, void *dq, void *dk, void *dv,
                          void *dq_idx, void *dk_idx, bool with_kl, float *kl_rows, float *kl_loss, void *workspace,
                          size_t workspace_bytes, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    if (p.q_offset != 0 || p.Nq != p.Nk || p.kv_rows != p.Nk)
        return fail(MSA_ERR_UNSUPPORTED, "fused_bwd needs q_offset == 0, Nq == Nk and kv_rows == Nk");
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(o, "o");
    REQUIRE_PTR(d_o, "d_o");
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    REQUIRE_PTR(dq, "dq");
    REQUIRE_PTR(dk, "dk");
    REQUIRE_PTR(dv, "dv");
    REQUIRE_PTR(dq_idx, "dq_idx");
    REQUIRE_PTR(dk_idx, "dk_idx");
    if (!sel_idx || !lse || !lse_idx) return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx, lse and lse_idx must be non-NULL");
    if (with_kl && !kl_loss) return fail(MSA_ERR_INVALID_ARGUMENT, "kl_loss is NULL");
    if (!isfinite(kl_coef)) return fail(MSA_ERR_INVALID_ARGUMENT, "kl_coef must be finite");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + bwd_bytes(p) + (with_kl ? bwdkl_bytes(p) : 0));
    if (st != MSA_OK) return st;
    Carve cv{static_cast<char *>(workspace)};
    DeviceStatus *ds = static_cast<DeviceStatus *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    BwdWork w{};
    w.D = cv.take<float>((size_t)p.B * p.Hq * p.Nq);
    w.dki_acc = cv.take<float>((size_t)p.B * p.Nk * p.d_idx * (size_t)p.Hkv);
    carve_index(cv, p, w);
    const size_t slots = (size_t)p.B * p.Nq * p.topk;
    w.dq_part = cv.take<bf16>(slots * p.Hq * p.d);
    w.dqi_part = cv.take<bf16>(slots * p.Hkv * p.d_idx);
    float *rows = nullptr;
    cudaError_t e;
    if (with_kl) {
        rows = kl_rows ? kl_rows : cv.take<float>((size_t)p.B * p.Hkv * p.Nq);
        w.klt = cv.take<float>(slots * p.Hkv * 4);
        w.kl_rows = rows;
    }
    e = launch_fused_bwd(p, static_cast<const bf16 *>(q), static_cast<const bf16 *>(k), static_cast<const bf16 *>(v),
                         static_cast<const bf16 *>(o), static_cast<const bf16 *>(d_o), lse,
                         static_cast<const bf16 *>(q_idx), static_cast<const bf16 *>(k_idx), sel_idx, lse_idx, kl_coef,
                         static_cast<bf16 *>(dq), static_cast<bf16 *>(dk), static_cast<bf16 *>(dv),
                         static_cast<bf16 *>(dq_idx), static_cast<bf16 *>(dk_idx), w, ds, s);
    if (e != cudaSuccess) return cuda_fail(e, "fused_bwd launch");
    if (with_kl && (e = launch_kl_reduce(p, rows, kl_coef, kl_loss, s)) != cudaSuccess)
        return cuda_fail(e, "kl_reduce launch");
    return MSA_OK;
}
}  // namespace

extern "C" {

msa_status msa_fused_bwd(const msa_shape *shape, const void *q, const void *k, const void *v, const void *o,
                         const void *d_o, const float *lse, const void *q_idx, const void *k_idx,
                         const int32_t *sel_idx, const float *lse_idx, float kl_coef, void *dq, void *dk, void *dv,
                         void *dq_idx, void *dk_idx, void *workspace, size_t workspace_bytes, void *stream)
{
    return fused_bwd_impl(shape, q, k, v, o, d_o, lse, q_idx, k_idx, sel_idx, lse_idx, kl_coef, dq, dk, dv, dq_idx,
                          dk_idx, false, nullptr, nullptr, workspace, workspace_bytes, stream);
}

msa_status msa_fused_bwd_kl(const msa_shape *shape, const void *q, const void *k, const void *v, const void *o,
                            const void *d_o, const float *lse, const void *q_idx, const void *k_idx,
                            const int32_t *sel_idx, const float *lse_idx, float kl_coef, void *dq, void *dk, void *dv,
                            void *dq_idx, void *dk_idx, float *kl_rows, float *kl_loss, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    return fused_bwd_impl(shape, q, k, v, o, d_o, lse, q_idx, k_idx, sel_idx, lse_idx, kl_coef, dq, dk, dv, dq_idx,
                          dk_idx, true, kl_rows, kl_loss, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {
// The training step; ev_idx / ev_qkv / ev_do (nullable) are events the stream
// waits on just before the first work that reads q_idx and k_idx / q, k and v
// / d_o, so inputs still being copied in can overlap the earlier phases.
msa_status train_step_impl(const msa_shape *shape, const void *q, const void *k, const void *v, const void *q_idx,
                           const void *k_idx, const void *d_o, float kl_coef, int32_t *sel_idx, void *o, float *lse,
                           float *lse_idx, float *kl_rows, float *kl_loss, void *dq, void *dk, void *dv, void *dq_idx,
                           void *dk_idx, cudaEvent_t ev_idx, cudaEvent_t ev_qkv, cudaEvent_t ev_do, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    Problem p;
    msa_status st = make_problem(shape, p);
    if (st != MSA_OK) return st;
    if (p.q_offset != 0 || p.Nq != p.Nk || p.kv_rows != p.Nk)
        return fail(MSA_ERR_UNSUPPORTED, "train_step needs q_offset == 0, Nq == Nk and kv_rows == Nk");
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    REQUIRE_PTR(d_o, "d_o");
    REQUIRE_PTR(o, "o");
    REQUIRE_PTR(dq, "dq");
    REQUIRE_PTR(dk, "dk");
    REQUIRE_PTR(dv, "dv");
    REQUIRE_PTR(dq_idx, "dq_idx");
    REQUIRE_PTR(dk_idx, "dk_idx");
    if (!sel_idx || !lse || !lse_idx || !kl_loss)
        return fail(MSA_ERR_INVALID_ARGUMENT, "sel_idx, lse, lse_idx and kl_loss must be non-NULL");
    if (!isfinite(kl_coef)) return fail(MSA_ERR_INVALID_ARGUMENT, "kl_coef must be finite");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + train_bytes(p));
    if (st != MSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto wait = [&](cudaEvent_t ev) { return ev ? cudaStreamWaitEvent(s, ev, 0) : cudaSuccess; };
    cudaError_t e;
    if (!train_shared_index(p)) {
        // the four phases in turn, each carving the same workspace
        if ((e = wait(ev_idx)) != cudaSuccess) return cuda_fail(e, "train_step: waiting for q_idx, k_idx");
        if ((st = msa_index_select(shape, q_idx, k_idx, sel_idx, nullptr, workspace, workspace_bytes, stream)) != MSA_OK)
            return st;
        if ((e = wait(ev_qkv)) != cudaSuccess) return cuda_fail(e, "train_step: waiting for q, k, v");
        if ((st = msa_sparse_attn_fwd(shape, q, k, v, sel_idx, o, lse, workspace, workspace_bytes, stream)) != MSA_OK)
            return st;
        if ((st = msa_kl_fwd(shape, q, k, q_idx, k_idx, sel_idx, lse, kl_coef, lse_idx, nullptr, nullptr, workspace,
                             workspace_bytes, stream)) != MSA_OK)
            return st;
        if ((e = wait(ev_do)) != cudaSuccess) return cuda_fail(e, "train_step: waiting for d_o");
        return msa_fused_bwd_kl(shape, q, k, v, o, d_o, lse, q_idx, k_idx, sel_idx, lse_idx, kl_coef, dq, dk, dv, dq_idx,
                                dk_idx, kl_rows, kl_loss, workspace, workspace_bytes, stream);
    }
    DeviceStatus *ds = static_cast<DeviceStatus *>(workspace);
    Carve cv{static_cast<char *>(workspace)};
    BwdWork w{};
    carve_index(cv, p, w);
    w.D = cv.take<float>((size_t)p.B * p.Hq * p.Nq);
    // the phases' own buffers overlay one region (see train_bytes)
    const size_t region = cv.off;
    float *bs_scratch = index_select_fused(p) ? nullptr : cv.take<float>(index_select_scratch_floats(p));
    cv.off = region;
    const size_t rows = (size_t)p.B * p.Nq * p.Hq * p.topk;
    FwdWork fw;
    fw.part = cv.take<bf16>(rows * p.d);
    fw.stats = cv.take<float2>(rows);
    cv.off = region;
    KlWork kw;
    kw.part = cv.take<float2>(kl_part_count(p));
    kw.klt = nullptr;                                  // lse_idx only: the loss comes from the backward
    cv.off = region;
    w.dki_acc = cv.take<float>((size_t)p.B * p.Hkv * p.Nk * p.d_idx);
    const size_t slots = (size_t)p.B * p.Nq * p.topk;
    w.dq_part = cv.take<bf16>(slots * p.Hq * p.d);
    w.dqi_part = cv.take<bf16>(slots * p.Hkv * p.d_idx);
    float *rows_kl = kl_rows ? kl_rows : cv.take<float>((size_t)p.B * p.Hkv * p.Nq);
    w.klt = cv.take<float>(slots * p.Hkv * 4);
    w.kl_rows = rows_kl;
    // one inverse index of the selection serves the forward, the KL pass and the backward
    fw.bucket_cnt = kw.bucket_cnt = w.bucket_cnt;
    fw.bucket_off = kw.bucket_off = w.bucket_off;
    fw.bucket_scratch = kw.bucket_scratch = w.bucket_scratch;
    fw.bucket_q = kw.bucket_q = w.bucket_q;
    fw.index_ready = kw.index_ready = w.index_ready = true;
    fw.d_o = static_cast<const bf16 *>(d_o);           // the forward combine leaves D for the backward
    fw.D = w.D;
    fw.d_o_ready = ev_do;
    w.D_ready = true;
    const bf16 *bq = static_cast<const bf16 *>(q), *bk = static_cast<const bf16 *>(k), *bv = static_cast<const bf16 *>(v);
    const bf16 *bqi = static_cast<const bf16 *>(q_idx), *bki = static_cast<const bf16 *>(k_idx);
    if ((e = wait(ev_idx)) != cudaSuccess) return cuda_fail(e, "train_step: waiting for q_idx, k_idx");
    e = launch_index_select(p, bqi, bki, nullptr, bs_scratch, sel_idx, ds, s);
    if (e != cudaSuccess) return cuda_fail(e, "train_step: selection");
    if ((e = launch_inverse_index(p, sel_idx, w.bucket_cnt, w.bucket_off, w.bucket_scratch, w.bucket_q, ds, s)) != cudaSuccess)
        return cuda_fail(e, "train_step: inverse index");
    if ((e = wait(ev_qkv)) != cudaSuccess) return cuda_fail(e, "train_step: waiting for q, k, v");
    if ((e = launch_sparse_fwd_keymajor(p, bq, bk, bv, sel_idx, static_cast<bf16 *>(o), lse, fw, ds, s)) != cudaSuccess)
        return cuda_fail(e, "train_step: forward");
    if ((e = launch_kl_keymajor(p, bq, bk, bqi, bki, sel_idx, lse, lse_idx, nullptr, kw, ds, s)) != cudaSuccess)
        return cuda_fail(e, "train_step: lse_idx");
    if ((e = launch_fused_bwd(p, bq, bk, bv, static_cast<const bf16 *>(o), static_cast<const bf16 *>(d_o), lse, bqi, bki,
                              sel_idx, lse_idx, kl_coef, static_cast<bf16 *>(dq), static_cast<bf16 *>(dk),
                              static_cast<bf16 *>(dv), static_cast<bf16 *>(dq_idx), static_cast<bf16 *>(dk_idx), w, ds,
                              s)) != cudaSuccess)
        return cuda_fail(e, "train_step: backward");
    if ((e = launch_kl_reduce(p, rows_kl, kl_coef, kl_loss, s)) != cudaSuccess) return cuda_fail(e, "train_step: loss");
    return MSA_OK;
}
}  // namespace

extern "C" {

msa_status msa_train_step(const msa_shape *shape, const void *q, const void *k, const void *v, const void *q_idx,
                          const void *k_idx, const void *d_o, float kl_coef, int32_t *sel_idx, void *o, float *lse,
                          float *lse_idx, float *kl_rows, float *kl_loss, void *dq, void *dk, void *dv, void *dq_idx,
                          void *dk_idx, void *workspace, size_t workspace_bytes, void *stream)
{
    return train_step_impl(shape, q, k, v, q_idx, k_idx, d_o, kl_coef, sel_idx, o, lse, lse_idx, kl_rows, kl_loss, dq,
                           dk, dv, dq_idx, dk_idx, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream);
}

msa_status msa_train_step_staged(const msa_shape *shape, const void *q, const void *k, const void *v,
                                 const void *q_idx, const void *k_idx, const void *d_o, float kl_coef, int32_t *sel_idx,
                                 void *o, float *lse, float *lse_idx, float *kl_rows, float *kl_loss, void *dq,
                                 void *dk, void *dv, void *dq_idx, void *dk_idx, void *idx_ready, void *qkv_ready,
                                 void *do_ready, void *workspace, size_t workspace_bytes, void *stream)
{
    return train_step_impl(shape, q, k, v, q_idx, k_idx, d_o, kl_coef, sel_idx, o, lse, lse_idx, kl_rows, kl_loss, dq,
                           dk, dv, dq_idx, dk_idx, static_cast<cudaEvent_t>(idx_ready),
                           static_cast<cudaEvent_t>(qkv_ready), static_cast<cudaEvent_t>(do_ready), workspace,
                           workspace_bytes, stream);
}

msa_status msa_warmup_kl(const msa_shape *shape, const void *q, const void *k, const void *v, const void *q_idx,
                         const void *k_idx, float kl_coef, float *lse, float *lse_idx, float *kl_rows, float *kl_loss,
                         void *dq_idx, void *dk_idx, void *workspace, size_t workspace_bytes, void *stream)
{
    Problem p0;
    msa_status st = make_problem(shape, p0);
    if (st != MSA_OK) return st;
    if (!warmup_shape_ok(p0))
        return fail(MSA_ERR_UNSUPPORTED, "warmup_kl needs q_offset == 0, Nq == Nk == kv_rows and at "
                    "most 32 blocks (Nk <= 4096); got Nk=%d d=%d d_idx=%d", p0.Nk, p0.d, p0.d_idx);
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    REQUIRE_PTR(dq_idx, "dq_idx");
    REQUIRE_PTR(dk_idx, "dk_idx");
    if (!lse || !lse_idx || !kl_loss) return fail(MSA_ERR_INVALID_ARGUMENT, "lse, lse_idx and kl_loss must be non-NULL");
    if (!isfinite(kl_coef)) return fail(MSA_ERR_INVALID_ARGUMENT, "kl_coef must be finite");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + warmup_bytes(p0));
    if (st != MSA_OK) return st;
    const Problem p = warmup_problem(p0);
    DeviceStatus *ds = static_cast<DeviceStatus *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Carve cv{static_cast<char *>(workspace)};
    const size_t slots = (size_t)p.B * p.Nq * p.topk, rows = slots * p.Hq;
    int32_t *sel = cv.take<int32_t>(slots * p.Hkv);
    FwdWork fw;
    carve_index(cv, p, fw);
    bf16 *o = cv.take<bf16>((size_t)p.B * p.Nq * p.Hq * p.d);
    fw.part = cv.take<bf16>(rows * p.d);
    fw.stats = cv.take<float2>(rows);
    fw.index_ready = true;
    KlWork kw;
    kw.part = cv.take<float2>(kl_part_count(p));
    kw.klt = nullptr;
    kw.bucket_cnt = fw.bucket_cnt;
    kw.bucket_off = fw.bucket_off;
    kw.bucket_scratch = fw.bucket_scratch;
    kw.bucket_q = fw.bucket_q;
    kw.index_ready = true;
    float *klt = cv.take<float>(slots * p.Hkv * 4);
    float *rows_kl = cv.take<float>((size_t)p.B * p.Hkv * p.Nq);
    if (kl_rows) rows_kl = kl_rows;
    bf16 *dqi_part = cv.take<bf16>(slots * p.Hkv * p.d_idx);
    float *dki_g = cv.take<float>((size_t)p.B * p.Hkv * p.Nk * p.d_idx);
    const bf16 *bq = static_cast<const bf16 *>(q), *bk = static_cast<const bf16 *>(k);
    const bf16 *bqi = static_cast<const bf16 *>(q_idx), *bki = static_cast<const bf16 *>(k_idx);
    cudaError_t e;
    // every visible block selected: the dense teacher and student over the whole prefix
    if ((e = launch_dense_selection(p, sel, s)) != cudaSuccess) return cuda_fail(e, "warmup_kl: selection");
    if ((e = launch_inverse_index(p, sel, fw.bucket_cnt, fw.bucket_off, fw.bucket_scratch, fw.bucket_q, ds, s)) !=
        cudaSuccess)
        return cuda_fail(e, "warmup_kl: inverse index");
    // the dense main attention: its lse normalises each head's teacher probabilities
    if ((e = launch_sparse_fwd_keymajor(p, bq, bk, static_cast<const bf16 *>(v), sel, o, lse, fw, ds, s)) != cudaSuccess)
        return cuda_fail(e, "warmup_kl: main attention");
    if ((e = launch_kl_keymajor(p, bq, bk, bqi, bki, sel, lse, lse_idx, nullptr, kw, ds, s)) != cudaSuccess)
        return cuda_fail(e, "warmup_kl: lse_idx");
    if ((e = launch_index_teacher_tc(p, bq, bk, bqi, bki, lse, lse_idx, kl_coef, fw.bucket_off, fw.bucket_q, klt,
                                     dqi_part, dki_g, ds, s)) != cudaSuccess)
        return cuda_fail(e, "warmup_kl: teacher and index gradients");
    if ((e = launch_kl_rows_combine(p, sel, lse_idx, klt, rows_kl, s)) != cudaSuccess) return cuda_fail(e, "warmup_kl: rows");
    if ((e = launch_kl_reduce(p, rows_kl, kl_coef, kl_loss, s)) != cudaSuccess) return cuda_fail(e, "warmup_kl: loss");
    if ((e = launch_bwd_combine(p, sel, dqi_part, static_cast<bf16 *>(dq_idx), p.Hkv, 1, p.d_idx, s)) != cudaSuccess)
        return cuda_fail(e, "warmup_kl: dq_idx");
    if ((e = launch_dki_group_sum(p, dki_g, static_cast<bf16 *>(dk_idx), s)) != cudaSuccess)
        return cuda_fail(e, "warmup_kl: dk_idx");
    return MSA_OK;
}

}  // extern "C"

namespace {
msa_status make_proj(const msa_proj_shape *s, ProjProblem &pp)
{
    if (!s) return fail(MSA_ERR_INVALID_ARGUMENT, "shape is NULL");
    if (s->T < 1 || s->Dm < 1 || s->Hkv < 1 || s->d_idx < 1)
        return fail(MSA_ERR_INVALID_ARGUMENT, "projection shape has a non-positive size (T=%d Dm=%d Hkv=%d d_idx=%d)",
                    s->T, s->Dm, s->Hkv, s->d_idx);
    if (s->d_idx != 64 && s->d_idx != 128) return fail(MSA_ERR_UNSUPPORTED, "d_idx must be 64 or 128 (got %d)", s->d_idx);
    if (s->Dm % 8 != 0) return fail(MSA_ERR_UNSUPPORTED, "Dm must be a multiple of 8 (got %d)", s->Dm);
    if ((long long)s->T * s->Hkv * s->d_idx >= (1LL << 31) || (long long)s->T * s->Dm >= (1LL << 40))
        return fail(MSA_ERR_UNSUPPORTED, "projection too large");
    pp.T = s->T;
    pp.Dm = s->Dm;
    pp.Hkv = s->Hkv;
    pp.d_idx = s->d_idx;
    pp.num_sms = sm_count();
    return MSA_OK;
}
}  // namespace

extern "C" {

size_t msa_index_proj_workspace_size(const msa_proj_shape *shape)
{
    ProjProblem pp;
    if (make_proj(shape, pp) != MSA_OK) return 0;
    return kStatusBytes + align256(index_proj_partial_floats(pp) * sizeof(float));
}

msa_status msa_index_proj_fwd(const msa_proj_shape *shape, const void *x, const void *wq_idx, const void *wk_idx,
                              void *q_idx, void *k_idx, void *workspace, size_t workspace_bytes, void *stream)
{
    ProjProblem pp;
    msa_status st = make_proj(shape, pp);
    if (st != MSA_OK) return st;
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(wq_idx, "wq_idx");
    REQUIRE_PTR(wk_idx, "wk_idx");
    REQUIRE_PTR(q_idx, "q_idx");
    REQUIRE_PTR(k_idx, "k_idx");
    st = check_ws(workspace, workspace_bytes, kStatusBytes);
    if (st != MSA_OK) return st;
    cudaError_t e = launch_index_proj_fwd(pp, static_cast<const bf16 *>(x), static_cast<const bf16 *>(wq_idx),
                                          static_cast<const bf16 *>(wk_idx), static_cast<bf16 *>(q_idx),
                                          static_cast<bf16 *>(k_idx), static_cast<DeviceStatus *>(workspace),
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "index_proj_fwd launch");
    return MSA_OK;
}

msa_status msa_index_proj_bwd(const msa_proj_shape *shape, const void *x, const void *dq_idx, const void *dk_idx,
                              float *dwq_idx, float *dwk_idx, void *workspace, size_t workspace_bytes, void *stream)
{
    ProjProblem pp;
    msa_status st = make_proj(shape, pp);
    if (st != MSA_OK) return st;
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(dq_idx, "dq_idx");
    REQUIRE_PTR(dk_idx, "dk_idx");
    REQUIRE_PTR(dwq_idx, "dwq_idx");
    REQUIRE_PTR(dwk_idx, "dwk_idx");
    st = check_ws(workspace, workspace_bytes, kStatusBytes + align256(index_proj_partial_floats(pp) * sizeof(float)));
    if (st != MSA_OK) return st;
    float *partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + kStatusBytes);
    cudaError_t e = launch_index_proj_dw(pp, static_cast<const bf16 *>(x), static_cast<const bf16 *>(dq_idx),
                                         static_cast<const bf16 *>(dk_idx), dwq_idx, dwk_idx, partial,
                                         static_cast<DeviceStatus *>(workspace), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "index_proj_bwd launch");
    return MSA_OK;
}

msa_status msa_check_device_status(void *workspace, void *stream)
{
    if (!workspace) return fail(MSA_ERR_INVALID_ARGUMENT, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceStatus h{};
    cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (h.code == 0) return MSA_OK;
    e = cudaMemsetAsync(workspace, 0, sizeof h, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    if (h.code == kDevTimeout)
        return fail(MSA_ERR_TIMEOUT, "a device-side wait ran out (site %d, info %d)", h.where, h.info);
    return fail(MSA_ERR_DEVICE, "device-side check failed (code %d, site %d, info %d)", h.code, h.where, h.info);
}

}  // extern "C"
