// kv_append.cu -- the KV-cache update of a decode (or chunked prefill) step.
//
// "Sparse Attention · Part II", section 3.2: each token brings its K and V
// rows (one per KV head) and one index key k_idx shared by the groups;
// section 4.1 notes that in decoding, reading the KV cache dominates.  A
// decode step first adds the new token's rows to that cache, since its own
// query attends to them.  The Nq new tokens of every batch entry go to cache rows
// q_offset .. q_offset+Nq-1.  All three tensors move in one launch, 16 bytes
// per thread: a token's K row group (Hkv*d bf16), its V row group and its
// K_idx row are contiguous in both the source and the cache.
#include <algorithm>

#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 256;

// units (16-byte words) per token: K, V, then K_idx
__global__ void __launch_bounds__(kThreads)
kv_append_kernel(Problem p, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                 const uint4 *__restrict__ ki_new, uint4 *__restrict__ k, uint4 *__restrict__ v,
                 uint4 *__restrict__ ki)
{
    const int uk = k_new ? p.Hkv * p.d / 8 : 0;        // words of one token's K (and V) rows
    const int uv = v_new ? p.Hkv * p.d / 8 : 0;
    const int ui = ki_new ? p.d_idx / 8 : 0;
    const int per_tok = uk + uv + ui;
    const long long total = (long long)p.B * p.Nq * per_tok;
    for (long long x = (long long)blockIdx.x * kThreads + threadIdx.x; x < total;
         x += (long long)gridDim.x * kThreads) {
        const long long tok = x / per_tok;            // b * Nq + i
        int w = (int)(x - tok * per_tok);
        const long long b = tok / p.Nq, i = tok - b * p.Nq;
        const long long row = b * p.kv_rows + p.q_offset + i;   // cache row
        if (w < uk) {
            k[row * uk + w] = __ldg(k_new + tok * uk + w);
            continue;
        }
        w -= uk;
        if (w < uv) {
            v[row * uv + w] = __ldg(v_new + tok * uv + w);
            continue;
        }
        w -= uv;
        ki[row * ui + w] = __ldg(ki_new + tok * ui + w);
    }
}

}  // namespace

cudaError_t launch_kv_append(const Problem &p, const bf16 *k_new, const bf16 *v_new, const bf16 *ki_new, bf16 *k,
                             bf16 *v, bf16 *ki, cudaStream_t s)
{
    const long long per_tok = (k_new ? p.Hkv * p.d / 8 : 0) + (v_new ? p.Hkv * p.d / 8 : 0) +
                              (ki_new ? p.d_idx / 8 : 0);
    const long long total = (long long)p.B * p.Nq * per_tok;
    if (total == 0) return cudaSuccess;
    const long long want = (total + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)std::min<long long>(want, 8LL * p.num_sms);
    {
        TimedLaunch timed_("kv_append_kernel", s);
        kv_append_kernel<<<grid, kThreads, 0, s>>>(
            p, reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
            reinterpret_cast<const uint4 *>(ki_new), reinterpret_cast<uint4 *>(k), reinterpret_cast<uint4 *>(v),
            reinterpret_cast<uint4 *>(ki));
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
