// warmup.cu -- the selection that keeps every visible block, used by the
// dense indexer warm-up.
//
// "Sparse Attention · Part II", section 3.1: before sparse training the
// indexer is fitted to the main attention with full attention kept: the
// teacher is the main branch's probabilities over the whole visible prefix
// and the student the index scores' softmax over the same prefix.  Section
// 3.2 then restricts MSA's KL to the tokens of the selected blocks; with
// every visible block selected the two are the same loss, so the warm-up
// runs MSA's own block-sparse kernels on this selection.
#include "msa_internal.h"

namespace msa {
namespace {

__global__ void __launch_bounds__(256) dense_selection_kernel(Problem p, int32_t *__restrict__ sel)
{
    const long long n = (long long)p.B * p.Hkv * p.Nq * p.topk;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(x % p.topk);
        const int i = (int)((x / p.topk) % p.Nq);
        const int c0 = (p.q_offset + i) / p.block;
        sel[x] = t <= c0 ? t : -1;
    }
}

}  // namespace

cudaError_t launch_dense_selection(const Problem &p, int32_t *sel, cudaStream_t s)
{
    {
        TimedLaunch timed_("dense_selection_kernel", s);
        dense_selection_kernel<<<4 * p.num_sms, 256, 0, s>>>(p, sel);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace msa
