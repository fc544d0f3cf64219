/*
 * msa.h -- C-ABI of libmsa.so, the GB300 (sm_103a) implementation of the
 * MiniMax Sparse Attention (MSA) layer's data-parallel hot path.
 *
 * The operator is the one defined in "Sparse Attention · Part II"
 * (mtreviso.github.io/blog/sparse-attention-2.html), section 3.2 "MiniMax's
 * MSA": an index branch scores every causally visible token with one index
 * query per GQA group against a single index key head shared by all groups,
 * max-pools the token scores into 128-token block scores and keeps, per
 * query and group, the query's own (local) block plus the k-1 best earlier
 * blocks; the main branch runs exact GQA softmax attention over the visible
 * tokens of those blocks only; training adds the detached KL alignment loss
 * of that section and the backward pass.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous in the layouts below.  bf16 tensors are passed as
 *     `void*` to keep CUDA headers out of this file.
 *   - The library never allocates, frees or synchronises.  Every call only
 *     enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns.
 *   - Scratch memory ("workspace") comes from the caller: at least
 *     msa_workspace_size(shape, op) bytes, 256-byte aligned.  Its first 256
 *     bytes hold a device status word that the kernels set on a device-side
 *     error (a wait that ran out, an index out of range);
 *     msa_check_device_status() reads it.  Those 256 bytes must be zero
 *     before the first call on a workspace (msa_check_device_status() zeroes
 *     them again after reporting); the rest need not be initialised.  Calls
 *     that share one workspace must be ordered on one stream.
 *   - Errors: arguments are validated on the host before any launch; on
 *     failure nothing is launched and the call returns a non-zero
 *     msa_status; msa_last_error() then gives a message (per host thread).
 *
 * Shapes and layouts (B batch, Nq queries, Nk keys, Hq query heads, Hkv KV
 * heads = GQA groups, G = Hq/Hkv, head h belongs to group h / G):
 *   q, o, d_o, dq         [B, Nq, Hq, d]        bf16
 *   k, v, dk, dv          [B, kv_rows, Hkv, d]  bf16 (rows >= Nk unused)
 *   q_idx, dq_idx         [B, Nq, Hkv, d_idx]   bf16
 *   k_idx, dk_idx         [B, kv_rows, d_idx]   bf16
 *   sel_idx               [B, Hkv, Nq, topk]    int32, ascending block ids,
 *                                               then -1 padding
 *   block_scores          [B, Nq, Hkv, nb]      fp32, nb = ceil(Nk/block);
 *                                               entry c of row i is defined
 *                                               for c <= c0(i) only
 *   lse                   [B, Hq, Nq]           fp32, natural log
 *   lse_idx, kl_rows      [B, Hkv, Nq]          fp32
 * Query row i sits at absolute position pos(i) = q_offset + i and sees key j
 * iff j <= pos(i); its local block is c0(i) = pos(i) / block.  Requires
 * Nk >= q_offset + Nq (every visible key exists).
 *
 * Supported (else MSA_ERR_UNSUPPORTED): block == 128; d, d_idx in {64, 128};
 * 1 <= topk <= 32; Hq % Hkv == 0 with G in {1, 2, 4, 8}.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned pointer */
    MSA_ERR_UNSUPPORTED = 2,      /* valid shape outside what this build supports */
    MSA_ERR_WORKSPACE = 3,        /* workspace too small */
    MSA_ERR_CUDA = 4,             /* a kernel launch or CUDA query failed */
    MSA_ERR_TIMEOUT = 5,          /* a device-side wait ran out (from msa_check_device_status) */
    MSA_ERR_DEVICE = 6            /* another device-side check failed (msa_check_device_status) */
} msa_status;

typedef struct {
    int B, Nq, Nk, q_offset, Hq, Hkv, d, d_idx, block, topk;
    long long kv_rows;   /* rows per batch entry of k, v, k_idx and their grads; 0 -> Nk */
    float scale;         /* main logit scale; 0 -> 1/sqrt(d) */
    float scale_idx;     /* index score scale; 0 -> 1/sqrt(d_idx) */
} msa_shape;

enum {
    MSA_OP_INDEX_SELECT = 0,
    MSA_OP_SPARSE_ATTN_FWD = 1,
    MSA_OP_KL_FWD = 2,
    MSA_OP_FUSED_BWD = 3,
    MSA_OP_FUSED_BWD_KL = 4,
    MSA_OP_TRAIN_STEP = 5,
    MSA_OP_WARMUP_KL = 6
};

/* Bytes of workspace `op` needs for `shape` (0 on an invalid shape). */
size_t msa_workspace_size(const msa_shape *shape, int op);

/*
 * Index branch and selection (section 3.2: token scoring against the shared
 * index key head, block max-pool, top-k with the local block reserved).
 * For each batch b, query i and group r:
 *   s_j   = scale_idx * <q_idx[b,i,r,:], k_idx[b,j,:]>   for j <= pos(i)
 *   bs_c  = max over visible j in block c of s_j           (fp32)
 *   sel   = {c0(i)} + the topk-1 blocks c < c0(i) of largest bs_c, ties to
 *           the lower c; every visible block when c0(i)+1 <= topk.
 * Writes sel_idx; also block_scores when it is not NULL.  Otherwise the
 * scores never reach memory when topk <= 16: the score kernel ranks them in
 * its epilogue (when a row's blocks are split across CTAs, as in decode, each
 * CTA leaves its slice's 16 best in the workspace and a merge kernel picks
 * the row's selection); with topk > 16 they live in the workspace.  The
 * result is the same either way.  No exp is taken: ranking uses raw scores.
 */
msa_status msa_index_select(const msa_shape *shape, const void *q_idx, const void *k_idx,
                            int32_t *sel_idx, float *block_scores,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Main branch (section 3.2): exact block-sparse GQA attention.  For head h
 * of group r, over the token set T = {j <= pos(i) : j / block in sel_idx}:
 *   l_j = scale * <q[b,i,h,:], k[b,j,r,:]>,  P = softmax_T(l),
 *   o[b,i,h,:] = sum_j P_j v[b,j,r,:],       lse[b,h,i] = log sum_T exp(l_j).
 * Each selected K/V block is staged once for all G heads of the group.
 */
msa_status msa_sparse_attn_fwd(const msa_shape *shape, const void *q, const void *k, const void *v,
                               const int32_t *sel_idx, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * KL alignment loss (section 3.2, the L_KL equation).  Teacher
 * Pt_j = (1/G) sum_{h in r} exp(l_{h,j} - lse[b,h,i]) (from the forward's
 * lse; detached), student Ps = softmax_T(s) with s_j = scale_idx <q_idx, k_idx_j>:
 *   lse_idx[b,r,i] = log sum_T exp(s_j)
 *   kl_rows[b,r,i] = sum_T Pt_j (log Pt_j - s_j) + lse_idx    ( = KL(Pt||Ps) )
 *   *kl_loss       = kl_coef / (B Nq Hkv) * sum of kl_rows   (device scalar)
 * kl_rows may be NULL (then it lives in the workspace).  The sum is taken in
 * a fixed order, so kl_loss is reproducible run to run.
 * With kl_rows and kl_loss both NULL only lse_idx is computed (no teacher
 * pass): the training step's form, where msa_fused_bwd_kl returns the loss.
 */
msa_status msa_kl_fwd(const msa_shape *shape, const void *q, const void *k, const void *q_idx,
                      const void *k_idx, const int32_t *sel_idx, const float *lse, float kl_coef,
                      float *lse_idx, float *kl_rows, float *kl_loss,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Fused backward of  sum(d_o . o) + L_KL.  Main gradients (dq, dk, dv) are
 * the softmax-attention backward over each query's selected token set; the
 * index gradients use the expansion of the KL in the student logits,
 * dL/ds_j = kl_coef/(B Nq Hkv) * (Ps_j - Pt_j), so neither distribution is
 * stored.  The teacher and the selection carry no gradient; the index
 * branch gets none from d_o (section 3.2 on the two detachments).  Uses the
 * forward's o and lse and the KL forward's lse_idx.  Requires q_offset == 0
 * and Nq == Nk (training layout).  dk, dv, dk_idx are fully written (zero
 * for keys no query selected).  Every sum is taken in a fixed order: the
 * same inputs give the same bits on every call.
 */
msa_status msa_fused_bwd(const msa_shape *shape, const void *q, const void *k, const void *v,
                         const void *o, const void *d_o, const float *lse, const void *q_idx,
                         const void *k_idx, const int32_t *sel_idx, const float *lse_idx, float kl_coef,
                         void *dq, void *dk, void *dv, void *dq_idx, void *dk_idx,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * msa_fused_bwd plus the KL loss of the same step (section 3.2): the values
 * msa_kl_fwd would give for kl_rows and *kl_loss (same definitions, same
 * lse_idx), computed from the backward's own recomputation of the teacher,
 * so a training step runs msa_kl_fwd in its lse_idx-only form (kl_rows and
 * kl_loss NULL) and gets the loss here without a separate teacher pass.
 * kl_loss (device scalar) must be non-NULL; kl_rows may be NULL (then it
 * lives in the workspace).  Workspace: msa_workspace_size(MSA_OP_FUSED_BWD_KL).
 */
msa_status msa_fused_bwd_kl(const msa_shape *shape, const void *q, const void *k, const void *v,
                            const void *o, const void *d_o, const float *lse, const void *q_idx,
                            const void *k_idx, const int32_t *sel_idx, const float *lse_idx, float kl_coef,
                            void *dq, void *dk, void *dv, void *dq_idx, void *dk_idx,
                            float *kl_rows, float *kl_loss,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * One training step of the layer (section 3.2): msa_index_select, then
 * msa_sparse_attn_fwd, msa_kl_fwd in its lse_idx-only form and
 * msa_fused_bwd_kl, with their definitions, layouts and outputs (sel_idx,
 * o, lse, lse_idx, kl_rows (may be NULL), *kl_loss, and the five gradients
 * from d_o).  On the key-major path (>= 8 queries per selected block on
 * average, which every training shape with Nq == Nk meets) the per-block
 * query lists of the selection are built once for all phases; elsewhere the
 * phases run one after another.  Training layout only (q_offset == 0, Nq == Nk,
 * kv_rows == Nk).  Workspace: msa_workspace_size(MSA_OP_TRAIN_STEP).
 */
msa_status msa_train_step(const msa_shape *shape, const void *q, const void *k, const void *v,
                          const void *q_idx, const void *k_idx, const void *d_o, float kl_coef,
                          int32_t *sel_idx, void *o, float *lse, float *lse_idx, float *kl_rows,
                          float *kl_loss, void *dq, void *dk, void *dv, void *dq_idx, void *dk_idx,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * msa_train_step with its inputs still arriving: idx_ready, qkv_ready and
 * do_ready are CUDA events (cudaEvent_t, each may be NULL) recorded after the
 * writes of q_idx and k_idx, of q, k and v, and of d_o (for instance the
 * host-to-device copies of this step's inputs on another stream).  The call
 * makes its stream wait on each just before the first work that reads those
 * tensors -- the selection, the forward, and the forward's combine (which
 * reads d_o on the key-major path) or the backward -- so a copy of the later
 * inputs overlaps the earlier phases.  Results are those of msa_train_step.
 * The events must stay valid until the stream has passed those points.
 */
msa_status msa_train_step_staged(const msa_shape *shape, const void *q, const void *k, const void *v,
                                 const void *q_idx, const void *k_idx, const void *d_o, float kl_coef,
                                 int32_t *sel_idx, void *o, float *lse, float *lse_idx, float *kl_rows,
                                 float *kl_loss, void *dq, void *dk, void *dv, void *dq_idx, void *dk_idx,
                                 void *idx_ready, void *qkv_ready, void *do_ready,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Dense indexer warm-up (section 3.1, the warm-up loss L^I_warm, in MSA's
 * per-group form of section 3.2, which follows the warm-up with the same KL
 * restricted to the selected blocks).  Full attention is kept: for each
 * query i and group r over EVERY visible key j <= i,
 *   teacher  Pt_j = (1/G) sum_{h in r} softmax_j(l_{h,j})   (detached)
 *   student  Ps_j = softmax_j(s_j),  s_j = scale_idx <q_idx, k_idx_j>
 *   kl_rows[b,r,i] = KL(Pt || Ps),   *kl_loss = kl_coef / (B Nq Hkv) * sum of kl_rows
 * and the loss's gradient in the index inputs, dL/ds_j = coef (Ps_j - Pt_j),
 * chained into dq_idx [B, Nq, Hkv, d_idx] and dk_idx [B, Nk, d_idx] (bf16,
 * fully written); q, k, v get none (the teacher is detached).  Also returns
 * the dense main attention's lse [B, Hq, Nq] (the teacher's normaliser) and
 * lse_idx; kl_rows may be NULL.  It is MSA's own block-sparse path run on
 * the selection of every visible block, so shape->topk is ignored (any valid
 * value): training layout (q_offset == 0, Nq == Nk, kv_rows == Nk) and at
 * most 32 blocks (Nk <= 4096), else MSA_ERR_UNSUPPORTED.
 * Workspace: msa_workspace_size(shape, MSA_OP_WARMUP_KL).  Deterministic.
 */
msa_status msa_warmup_kl(const msa_shape *shape, const void *q, const void *k, const void *v, const void *q_idx,
                         const void *k_idx, float kl_coef, float *lse, float *lse_idx, float *kl_rows, float *kl_loss,
                         void *dq_idx, void *dk_idx, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Index projections (section 3.2, the detachment equation): the index
 * queries and keys are linear maps of the DETACHED hidden states,
 *   q_idx = stopgrad(X) W_q^idx,   k_idx = stopgrad(X) W_k^idx.
 * x [T, Dm] (T = B * N tokens), wq_idx [Dm, Hkv * d_idx] (group r's index
 * query in columns r*d_idx ..), wk_idx [Dm, d_idx], all bf16 row-major;
 * q_idx [T, Hkv, d_idx] and k_idx [T, d_idx] bf16 (the layouts the index
 * branch takes).  msa_index_proj_bwd gives the KL's gradient in the weights,
 *   dwq_idx = X^T dq_idx   [Dm, Hkv * d_idx],   dwk_idx = X^T dk_idx   [Dm, d_idx]
 * (fp32, fully written), and nothing for X: the loss does not reach the
 * backbone through the indexer.  Tensor-core GEMMs; the weight gradient
 * splits the token sum over several CTAs and adds the parts in a fixed
 * order (deterministic).  Supported: d_idx in {64, 128}, Dm a multiple of 8,
 * Hkv >= 1, T * Hkv * d_idx < 2^31.  Pointers 16-byte aligned.  The
 * workspace (msa_index_proj_workspace_size bytes, 256-byte aligned, first
 * 256 bytes zero as for the other calls) serves both calls.
 */
typedef struct {
    int T, Dm, Hkv, d_idx;
} msa_proj_shape;
size_t msa_index_proj_workspace_size(const msa_proj_shape *shape);
msa_status msa_index_proj_fwd(const msa_proj_shape *shape, const void *x, const void *wq_idx, const void *wk_idx,
                              void *q_idx, void *k_idx, void *workspace, size_t workspace_bytes, void *stream);
msa_status msa_index_proj_bwd(const msa_proj_shape *shape, const void *x, const void *dq_idx, const void *dk_idx,
                              float *dwq_idx, float *dwk_idx, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Index selection without any allocation, for callers that cannot allocate
 * device memory (a serving process whose memory pool is frozen after
 * warm-up, or a plugin given only raw device pointers).  There is no
 * counterpart of this call in the method's description: it computes exactly
 * what msa_index_select computes (same kernels, same sel_idx), but its
 * selection scratch (block scores, or the per-slice candidate lists of a
 * split row) is a static device array inside the library instead of a
 * caller workspace.  The caller still passes q_idx, k_idx and sel_idx
 * (layouts as above); block scores are not returned.
 *   - Limit: the scratch the shape's selection path needs, which is
 *     msa_workspace_size(shape, MSA_OP_INDEX_SELECT) - 256, must be <= 64 MiB,
 *     else MSA_ERR_WORKSPACE before any launch.  That is none for prefill
 *     shapes with topk <= 16 (the top-k runs inside the score kernel), 128
 *     bytes per (row, slice) when a row's blocks are split across CTAs
 *     (decode), and B * Nq * Hkv * ceil(Nk/block) * 4 bytes of block scores
 *     otherwise (topk > 16).  Every device that loads the library holds that
 *     array (64 MiB plus 256 bytes) until the process exits.
 *   - All calls share the array and it keeps the last call's contents;
 *     calls that overlap on the GPU race with each other.
 *   - The first call on each device looks up the array's address with that
 *     device current and keeps it; make it before any stream capture.  After
 *     a cudaDeviceReset the kept address is stale: do not call this entry
 *     point again in that process.
 *   - Device-side status is kept inside the array, cleared at every call,
 *     and not reported by this entry point.
 */
msa_status msa_index_select_noalloc(const msa_shape *shape, const void *q_idx, const void *k_idx,
                                    int32_t *sel_idx, void *stream);

/*
 * Block mask of a selection (section 4.3, "Turn support into a block mask").
 * A query tile is 128 consecutive query rows i of one (batch b, group r),
 * T = ceil(Nq/128) tiles per (b, r); its mask has one bit per key block c,
 * set when some query of the tile selected c (the OR-union of the tile's
 * selections), packed 32 to a word: block c is bit c%32 of word c/32.
 *   sel_idx      [B, Hkv, Nq, topk] int32 (as msa_index_select writes it);
 *                -1 entries are padding; ids >= nb are ignored.
 *   mask         [B, Hkv, T, W] uint32, W = ceil(nb/32), nb = ceil(Nk/block);
 *                the bits of blocks >= nb in the last word are zero.
 *   tile_counts  [B, Hkv, T] int32, the number of set bits (active blocks)
 *                per tile; may be NULL.
 *   tile_blocks  [B, Hkv, T, nb] int32, each tile's active blocks in
 *                ascending order (the traversal: per word, count the set
 *                bits, visit them by rank), then -1; may be NULL.
 * Caller-owned device memory, 4-byte aligned; no workspace; asynchronous on
 * stream.  nb above 655,328 -> MSA_ERR_UNSUPPORTED.
 */
msa_status msa_block_mask(const msa_shape *shape, const int32_t *sel_idx, uint32_t *mask, int32_t *tile_counts,
                          int32_t *tile_blocks, void *stream);

/* KV-cache append of a decode (or chunked prefill) step.  "Sparse
 * Attention · Part II", section 3.2: every token carries its own K and V
 * rows per KV head and one index key k_idx shared by the groups; section 4.1
 * notes that in decoding, reading the KV cache dominates.  A decode step
 * first adds the new token's rows to that cache, since its own query attends
 * to them.  Writes the Nq new tokens at positions q_offset .. q_offset+Nq-1
 * of the caches, in one launch:
 *   k_new, v_new   [B, Nq, Hkv, d] bf16     -> k, v   [B, kv_rows, Hkv, d]
 *   k_idx_new      [B, Nq, d_idx] bf16      -> k_idx  [B, kv_rows, d_idx]
 * Shape fields used: B, Nq, Hkv, d, d_idx, q_offset, kv_rows (the other
 * fields must form a valid shape, as for msa_index_select).  Each pair
 * (k_new, k), (v_new, v), (k_idx_new, k_idx) is copied when both are
 * non-NULL and skipped when both are NULL; at least one pair is given.
 * Caller-owned device memory, 16-byte aligned; sources and destinations
 * must not overlap.  q_offset + Nq > kv_rows, a half-given pair, or a
 * misaligned pointer -> MSA_ERR_INVALID_ARGUMENT before any launch.  No
 * workspace; asynchronous on stream. */
msa_status msa_kv_append(const msa_shape *shape, const void *k_new, const void *v_new, const void *k_idx_new,
                         void *k, void *v, void *k_idx, void *stream);

/* Message of the last failed call on this host thread ("" if none). */
const char *msa_last_error(void);

/* Synchronises `stream`, reads the device status word of `workspace`,
 * returns MSA_OK, MSA_ERR_TIMEOUT or MSA_ERR_DEVICE, and clears the word. */
msa_status msa_check_device_status(void *workspace, void *stream);

/* Self-test of the bounded device-side wait, with no counterpart in the
 * method.  Every kernel of the library waits on its pipeline barriers with a
 * poll limit; when a wait runs out it records code 5 in the workspace's
 * status word and the kernel returns instead of hanging, so the context stays
 * usable and msa_check_device_status() reports MSA_ERR_TIMEOUT.  This call
 * launches one thread that waits, with spin_limit polls (1 .. 2^24), on a
 * barrier in its own shared memory that nothing arrives on -- no copies or
 * tensor-core work in flight -- and then writes 1 to the int at byte 128 of
 * the workspace (2 if the wait had completed).  workspace: 256 bytes,
 * 256-byte aligned, status word zero.  Asynchronous on stream. */
msa_status msa_selftest_wait_timeout(void *workspace, unsigned int spin_limit, void *stream);

/* Library version string. *//* Library version string. */
const char *msa_version(void);

/* Number of kernels this process has launched through the library so far
 * (monotonic; for accounting launches in a timed region). */
unsigned long long msa_launch_count(void);

/* Kernel timing, a measurement aid with no counterpart in the method.
 * msa_kernel_timing(1) makes every later call bracket each kernel it launches
 * with a pair of CUDA events recorded on the call's stream (the events are
 * created on first use and reused); msa_kernel_timing(0) stops it.  Either
 * call forgets what was recorded before; the return value is the previous
 * setting.  Off by default: then no event is created or recorded. */
int msa_kernel_timing(int enable);

/* Waits for the recorded events and writes one line per kernel name,
 * "<kernel> <launches> <total milliseconds>\n", into buf (at most len bytes,
 * NUL-terminated).  Returns the size the whole report needs, NUL included. */
size_t msa_kernel_timing_report(char *buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
