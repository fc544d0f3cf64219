// noalloc.cu -- index selection for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run MSA: code executing under an allocator that must not grow (a
// serving process that froze its memory pool after warm-up), or code that
// owns no allocator at all (a plugin handed only raw device pointers by its
// host framework).  msa_index_select needs scratch memory for the block
// scores between the scoring kernel and the top-k kernel, which normally
// comes from the caller's workspace.  msa_index_select_noalloc runs the same
// two kernels but takes that scratch from the file-scope device array below,
// which the CUDA runtime reserves when the library's module is loaded on a
// device; no call allocates anything.
//
// Limits and sharing:
//   * the array holds a 256-byte status word plus kScratchScoreBytes of
//     selection scratch; what the selection path taken for the shape needs
//     must fit: nothing when the top-k runs inside the score kernel (topk <=
//     16, every CTA sees all blocks of its rows: prefill), 128 bytes of
//     candidate keys per (row, slice) when a row's blocks are split across
//     CTAs (decode), else the block scores (B * Nq * Hkv * nb * 4 bytes);
//     larger needs are rejected with MSA_ERR_WORKSPACE before any launch;
//   * every device that loads the library holds the array until the process
//     exits;
//   * all calls share the one array: calls whose work overlaps on the GPU
//     (different streams without ordering, or several host threads) race;
//     the array keeps the last call's contents;
//   * on each device, the first call looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture.  A cudaDeviceReset destroys
//     the context that address belongs to: after one, the cached address is
//     stale and the entry point must not be called again in that process.
#include <stdio.h>

#include <mutex>

#include "msa.h"
#include "msa_internal.h"

namespace msa {
msa_status problem_from_shape(const msa_shape *shape, Problem &p);
msa_status set_error(msa_status st, const char *msg);
}  // namespace msa

using namespace msa;

namespace {

constexpr size_t kScratchScoreBytes = 64ull << 20;     // 64 MiB of selection scratch
constexpr size_t kScratchBytes = kStatusBytes + kScratchScoreBytes;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
cudaError_t scratch_on_current_device(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_select_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" msa_status msa_index_select_noalloc(const msa_shape *shape, const void *q_idx, const void *k_idx,
                                               int32_t *sel_idx, void *stream)
{
    Problem p;
    msa_status st = problem_from_shape(shape, p);
    if (st != MSA_OK) return st;
    const size_t need = index_select_scratch_floats(p) * sizeof(float);
    if (need > kScratchScoreBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "msa_index_select_noalloc: this shape's selection path needs %zu bytes of scratch, the static "
                 "array holds %zu (64 MiB)", need, kScratchScoreBytes);
        return set_error(MSA_ERR_WORKSPACE, msg);
    }
    if (!q_idx || !k_idx || !sel_idx) return set_error(MSA_ERR_INVALID_ARGUMENT, "q_idx, k_idx and sel_idx must be non-NULL");
    if (((uintptr_t)q_idx & 15u) || ((uintptr_t)k_idx & 15u))
        return set_error(MSA_ERR_INVALID_ARGUMENT, "q_idx and k_idx must be 16-byte aligned");
    void *scratch = nullptr;
    cudaError_t e = scratch_on_current_device(&scratch);
    if (e != cudaSuccess) return set_error(MSA_ERR_CUDA, cudaGetErrorString(e));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word must start at zero; the scratch a path reads is scratch it
    // wrote in the same call
    e = cudaMemsetAsync(scratch, 0, kStatusBytes, s);
    if (e != cudaSuccess) return set_error(MSA_ERR_CUDA, cudaGetErrorString(e));
    DeviceStatus *ds = static_cast<DeviceStatus *>(scratch);
    float *bs = reinterpret_cast<float *>(static_cast<char *>(scratch) + kStatusBytes);
    e = launch_index_select(p, static_cast<const bf16 *>(q_idx), static_cast<const bf16 *>(k_idx), nullptr, bs,
                            sel_idx, ds, s);
    if (e != cudaSuccess) return set_error(MSA_ERR_CUDA, cudaGetErrorString(e));
    return MSA_OK;
}
