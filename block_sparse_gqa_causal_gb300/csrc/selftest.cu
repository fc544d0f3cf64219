// selftest.cu -- a check of the library's bounded device-side wait, with no
// counterpart in the method.
//
// Every kernel here waits on mbarriers through tc::mbar_wait, which gives up
// after a poll limit, records MSA_ERR_TIMEOUT's code in the caller's status
// word and lets the kernel end instead of hanging.  This kernel makes such a
// wait run out on purpose, safely: one thread initialises an mbarrier in its
// own shared memory that nothing ever arrives on (no copies, no MMAs, no
// other threads involved) and waits on it with a short limit.
#include "msa.h"
#include "msa_internal.h"
#include "tc.cuh"

namespace msa {
namespace {

__global__ void wait_timeout_probe_kernel(DeviceStatus *st, uint32_t limit, int *returned)
{
    __shared__ uint64_t bar;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    const bool done = tc::mbar_wait(&bar, 0, st, 901, nullptr, limit);
    *returned = done ? 2 : 1;          // 1: the wait gave up and the kernel went on
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_selftest_wait_timeout(void *workspace, unsigned int spin_limit, void *stream)
{
    if (!workspace || ((uintptr_t)workspace & 255u)) return MSA_ERR_INVALID_ARGUMENT;
    if (spin_limit == 0 || spin_limit > (1u << 24)) return MSA_ERR_INVALID_ARGUMENT;
    DeviceStatus *st = static_cast<DeviceStatus *>(workspace);
    // the kernel's own flag goes right after the status word (inside the 256 bytes)
    int *returned = reinterpret_cast<int *>(static_cast<char *>(workspace) + 128);
    wait_timeout_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(st, spin_limit, returned);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
