// msa_internal.h -- problem description and kernel launchers shared by the
// C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace msa {

struct Problem {
    int B, Nq, Nk, q_offset, Hq, Hkv, G, d, d_idx, block, topk, nb;
    long long kv_rows;     // rows per batch entry of k, v, k_idx (>= Nk)
    float scale, scale_idx;
    int num_sms;
};

using bf16 = __nv_bfloat16;

// Counts kernel launches made by the library (read by msa_launch_count()).
void note_launch(int n = 1);

// Kernel timing hook (off unless msa_kernel_timing(1) is in effect): while
// alive, brackets the launch issued in its scope with CUDA events recorded on
// the launch's stream, filed under the kernel's name.
struct TimedLaunch {
    TimedLaunch(const char *name, cudaStream_t s);
    ~TimedLaunch();
    TimedLaunch(const TimedLaunch &) = delete;
    TimedLaunch &operator=(const TimedLaunch &) = delete;
    long slot;
    cudaStream_t stream;
};

// 3-D bf16 TMA tensor map (dims innermost first, strides of dims 1 and 2
// in bytes), box {box0, box1, 1}, 128-byte swizzle, zero fill out of bounds.
cudaError_t make_tmap_bf16_3d(CUtensorMap *map, const void *base, unsigned long long d0, unsigned long long d1,
                              unsigned long long d2, unsigned long long stride1_bytes,
                              unsigned long long stride2_bytes, unsigned box0, unsigned box1);
// Same for rank 1..5: dims innermost first, rank-1 strides in bytes, box per dim.
cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const unsigned long long *dims,
                           const unsigned long long *strides_bytes, const unsigned *box);

// Index branch: token scores + block max-pool.  bs: [B, Nq, Hkv, nb] fp32.
cudaError_t launch_index_scores(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs,
                                DeviceStatus *st, cudaStream_t s);
// Top-k block selection from block scores.  sel: [B, Hkv, Nq, topk].
cudaError_t launch_block_topk(const Problem &p, const float *bs, int32_t *sel, DeviceStatus *st,
                              cudaStream_t s);
// kv_append.cu: the new tokens' K, V and K_idx rows into the caches
cudaError_t launch_kv_append(const Problem &p, const bf16 *k_new, const bf16 *v_new, const bf16 *ki_new, bf16 *k,
                             bf16 *v, bf16 *ki, cudaStream_t s);
// Block mask of a selection (uint32 words per 128-query tile, one bit per
// key block), optionally each tile's active-block count and ascending list.
size_t block_mask_smem_bytes(const Problem &p);
cudaError_t launch_block_mask(const Problem &p, const int32_t *sel, uint32_t *mask, int32_t *counts, int32_t *active,
                              cudaStream_t s);
// Merge of per-slice candidate lists (16 descending block keys per (row,
// slice), slices of `span` blocks) into the selection: the second half of
// the fused decode selection.
cudaError_t launch_block_topk_merge(const Problem &p, const unsigned long long *cand, int slices, int span,
                                    int32_t *sel, cudaStream_t s);
// Index scores + selection: fused into the score kernel when every CTA sees
// all blocks of its rows and topk <= 16 (scores stored only if bs_out is set),
// else scores to bs_out (or bs_scratch) and the separate top-k kernel.
cudaError_t launch_index_select(const Problem &p, const bf16 *q_idx, const bf16 *k_idx, float *bs_out,
                                float *bs_scratch, int32_t *sel, DeviceStatus *st, cudaStream_t s);
// true when launch_index_select runs the fused form (no score scratch needed)
bool index_select_fused(const Problem &p);
// true when launch_index_select, with no scores wanted, selects in the
// split form (rows split across CTAs; per-slice candidates, then a merge)
bool index_select_split(const Problem &p);
// fp32 words of bs_scratch launch_index_select uses when bs_out is null, for
// the path it takes: none in the fused form, the per-slice candidate keys in
// the split form, else the block scores
size_t index_select_scratch_floats(const Problem &p);
// Key-major main branch forward (many queries per selected block).
struct FwdWork {
    bf16 *part;          // [B, Nq, Hq, topk, d] unnormalised partial outputs per selected block
    float2 *stats;       // [B, Nq, Hq, topk] (row max in log2 units, row sum)
    int32_t *bucket_cnt, *bucket_off, *bucket_scratch, *bucket_q;
    bool index_ready = false;   // the inverse index of sel is already in bucket_* (built once per step)
    // training step: with dO at hand the combine also leaves the backward's
    // D[b, h, i] = sum_e dO * O (O as written, bf16) -- one pass over O fewer
    const bf16 *d_o = nullptr;
    float *D = nullptr;
    cudaEvent_t d_o_ready = nullptr;   // the combine waits on it before reading d_o (nullable)
};
cudaError_t launch_sparse_fwd_keymajor(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v,
                                       const int32_t *sel, bf16 *o, float *lse, const FwdWork &w, DeviceStatus *st,
                                       cudaStream_t s);
// Main branch forward (query-major; few queries per selected block, e.g. decode).
// split_ws: [B*Nq*Hq*nsplit*d] fp32 partial outputs + [B*Nq*Hq*nsplit] float2 (m, l),
// nsplit = sparse_attn_splits(p); nullptr runs one CTA per (b, i, r)
int sparse_attn_splits(const Problem &p);
cudaError_t launch_sparse_attn_fwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v,
                                   const int32_t *sel, bf16 *o, float *lse, float *split_ws, DeviceStatus *st,
                                   cudaStream_t s);
// KL forward: per-row KL and lse_idx, then the deterministic scalar mean.
cudaError_t launch_kl_fwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx,
                          const bf16 *k_idx, const int32_t *sel, const float *lse, float *lse_idx,
                          float *kl_rows, DeviceStatus *st, cudaStream_t s);
// Key-major KL forward (many queries per selected block).
struct KlWork {
    float2 *part;        // [B, Hkv, Nq, topk, 2] (max s log2 e, sum 2^(s log2 e - max)) per key half
    float *klt;          // [B*Hkv*Nq*topk, 4] sums of Pt (log2 Pt - s log2 e) per lane quarter of the
                         // block's keys (teacher terms); nullptr: lse_idx only
    int32_t *bucket_cnt, *bucket_off, *bucket_scratch, *bucket_q;
    bool index_ready = false;
};
// float2 partials the key-major KL's index pass writes (two per (query, group, slot))
size_t kl_part_count(const Problem &p);
// lse_idx (index pass + combine) and, with w.klt and kl_rows set, the KL rows
// from the teacher terms of launch_index_teacher_tc
cudaError_t launch_kl_keymajor(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx, const bf16 *k_idx,
                               const int32_t *sel, const float *lse, float *lse_idx, float *kl_rows, const KlWork &w,
                               DeviceStatus *st, cudaStream_t s);
cudaError_t launch_kl_reduce(const Problem &p, const float *kl_rows, float kl_coef, float *kl_loss,
                             cudaStream_t s);
// The KL's teacher terms and (dqi_part set) the index-branch backward,
// key-major on the tcgen05 tensor cores (d, d_idx of 64 zero-padded to 128), the teacher
// recomputed from its own logit tiles: per (query, group, slot) klt (4 floats,
// nullable) and, for the backward, dq_idx partial rows in dqi_part and each
// group's fp32 dK_idx share in dki_g [B, Hkv, Nk, d_idx].
cudaError_t launch_index_teacher_tc(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *q_idx,
                                    const bf16 *k_idx, const float *lse, const float *lse_idx, float kl_coef,
                                    const int32_t *bucket_off, const int32_t *bucket_q, float *klt, bf16 *dqi_part,
                                    float *dki_g, DeviceStatus *st, cudaStream_t s);
// KL rows = ln 2 * (sum of a row's klt over its valid slots) + lse_idx
cudaError_t launch_kl_rows_combine(const Problem &p, const int32_t *sel, const float *lse_idx, const float *klt,
                                   float *kl_rows, cudaStream_t s);
// dk_idx = bf16 of the sum over groups, in order, of dki_g
cudaError_t launch_dki_group_sum(const Problem &p, const float *dki_g, bf16 *dk_idx, cudaStream_t s);

// Backward pieces.  Workspace carve-up is done by the caller (api.cu).
struct BwdWork {
    float *D;            // [B, Hq, Nq]    rowsum(dO * O)
    // dK_idx: each group's share [B, Hkv, Nk, d_idx], summed over the groups in order
    float *dki_acc;
    bf16 *dq_part;       // [B, Nq, Hq, topk, d]      dQ per selected block
    bf16 *dqi_part;      // [B, Nq, Hkv, topk, d_idx] dq_idx per selected block
    // KL loss terms per ((b, r, query), slot), four floats (nullptr when the loss
    // is not asked for): sums of Pt (log2 Pt - s log2 e) per lane quarter of
    // the block's keys
    float *klt;
    float *kl_rows;      // [B, Hkv, Nq] KL rows assembled from klt (when klt is set)
    int32_t *bucket_cnt; // [B*Hkv*nb]
    int32_t *bucket_off; // [B*Hkv*nb + 1]
    int32_t *bucket_scratch; // inverse_index_scratch_ints(p)
    int32_t *bucket_q;   // [B*Hkv*Nq*topk]  query rows per (b, r, block)
    bool index_ready;    // bucket_* already hold the inverse index of sel
    bool D_ready;        // D already holds rowsum(dO * O) (the training step's forward combine)
};
cudaError_t launch_fused_bwd(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v,
                             const bf16 *o, const bf16 *d_o, const float *lse, const bf16 *q_idx,
                             const bf16 *k_idx, const int32_t *sel, const float *lse_idx,
                             float kl_coef, bf16 *dq, bf16 *dk, bf16 *dv, bf16 *dq_idx,
                             bf16 *dk_idx, const BwdWork &w, DeviceStatus *st, cudaStream_t s);

// Inverse index: for every (b, group, block) the query rows that selected
// it.  cnt [nbk], off [nbk + 1], list [B*Hkv*Nq*topk]; scratch holds
// inverse_index_scratch_ints(p) ints (per-CTA histograms and offsets).
size_t inverse_index_scratch_ints(const Problem &p);
// list entry: query row i (< 2^26) and the slot (< 32) of the block in i's selection
__host__ __device__ __forceinline__ int32_t pack_entry(int i, int slot) { return (int32_t)(((uint32_t)slot << 26) | (uint32_t)i); }
__host__ __device__ __forceinline__ int entry_row(int32_t e) { return (int)((uint32_t)e & 0x3FFFFFFu); }
__host__ __device__ __forceinline__ int entry_slot(int32_t e) { return (int)((uint32_t)e >> 26); }
cudaError_t launch_inverse_index(const Problem &p, const int32_t *sel, int32_t *cnt, int32_t *off, int32_t *scratch,
                                 int32_t *list, DeviceStatus *st, cudaStream_t s);

// Order in which the key-major kernels visit the (group, key block) buckets
// of a batch: CTA x of a grid of Hkv * nb, early (larger) blocks first.
// When a group's blocks span several waves of the GPU (long sequences), the
// buckets go group by group, so the CTAs resident at one time share a
// group's query rows in L2 (each query's rows are gathered by every block it
// selected; at 131,072 tokens this saves 2 ms of a training step).  With
// fewer blocks the groups are interleaved instead (block c of every group,
// then c + 1): there the longest CTAs must start together or they make a
// tail, which costs more than L2 reuse gains (measured at 8,192 and 32,768).
__host__ __device__ __forceinline__ void bucket_of(int x, int Hkv, int nb, int num_sms, int &r, int &c)
{
    if (nb >= 4 * num_sms) {
        r = x / nb;
        c = x % nb;
    } else {
        r = x % Hkv;
        c = x / Hkv;
    }
}

// The backward runs on the tcgen05 kernels for d and d_idx of 64 or 128 (the
// tiles hold 128 features; 64 are zero-padded), i.e. for every valid shape.
inline bool bwd_tc(const Problem &p) { return (p.d == 64 || p.d == 128) && (p.d_idx == 64 || p.d_idx == 128); }
// tcgen05 main-branch backward: dK, dV and the dQ partials.
cudaError_t launch_bwd_main_tc(const Problem &p, const bf16 *q, const bf16 *k, const bf16 *v, const bf16 *d_o,
                               const float *lse, const BwdWork &w, bf16 *dk, bf16 *dv, DeviceStatus *st,
                               cudaStream_t s);

// Index projections of the detached hidden states (X [T, Dm], W_q^idx
// [Dm, Hkv*d_idx], W_k^idx [Dm, d_idx]) and their weight gradient.
struct ProjProblem {
    int T, Dm, Hkv, d_idx, num_sms;
};
// token-range splits of the weight gradient, and the fp32 partial floats it needs
int index_proj_splits(const ProjProblem &pp);
size_t index_proj_partial_floats(const ProjProblem &pp);
cudaError_t launch_index_proj_fwd(const ProjProblem &pp, const bf16 *x, const bf16 *wq, const bf16 *wk, bf16 *q_idx,
                                  bf16 *k_idx, DeviceStatus *st, cudaStream_t s);
cudaError_t launch_index_proj_dw(const ProjProblem &pp, const bf16 *x, const bf16 *dq_idx, const bf16 *dk_idx,
                                 float *dwq, float *dwk, float *partial, DeviceStatus *st, cudaStream_t s);
// Sum of a row's per-slot bf16 partial rows (width 64 or 128 features) over
// its valid slots: H rows per (b, query), head h in group h / Gh.
cudaError_t launch_bwd_combine(const Problem &p, const int32_t *sel, const bf16 *part, bf16 *out, int H, int Gh, int width,
                               cudaStream_t s);
// The selection that keeps every visible block (topk = nb): sel[b, r, i, t] =
// t for t <= c0(i), else -1 -- the dense warm-up's token set.
cudaError_t launch_dense_selection(const Problem &p, int32_t *sel, cudaStream_t s);

}  // namespace msa
