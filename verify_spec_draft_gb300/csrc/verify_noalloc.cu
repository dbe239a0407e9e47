// verify_noalloc.cu - spec_verify for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: a plugin loaded into a host
// program that owns the GPU's memory through its own allocator and hands none of it
// out, or a serving process that has given nearly all device memory to a caching
// pool, where one more cudaMalloc would fail, and would synchronise the device on a
// latency-critical path even when it succeeds.  spec_verify_noalloc serves them: the
// verify kernels run unchanged, with their workspace placed in the fixed-size static
// device array below instead of caller memory.
//
// The array is a module global: every GPU that loads the library holds its
// kSpecNoallocScratchBytes until the process exits, and every call on a device shares
// it.  Its contents outlive a call, so each call clears the bytes it uses before the
// kernels start; two calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "spec.h"
#include "internal.h"
#include "spec_device.cuh"

namespace spec {

static_assert(SPEC_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size is a multiple of 256 bytes");

// Device-resident scratch.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_verify_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;

// Device address of g_verify_scratch on the current device, looked up on the first
// call made with that device current.
static cudaError_t scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[kNoallocMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_verify_scratch);
        if (e != cudaSuccess) return e;
        if (!ptr) return cudaErrorInvalidSymbol;
        addr[dev] = ptr;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace spec

using namespace spec;

extern "C" spec_status spec_verify_noalloc(const void* target_logits, spec_dtype target_dtype,
                                           const void* draft_logits, spec_dtype draft_dtype,
                                           const int32_t* draft_tokens, int B, int gamma, int V, int temperature,
                                           const uint64_t* seeds, int32_t* n_accepted_out, int32_t* committed_out,
                                           int32_t* bonus_out, int32_t* near_tie_out, spec_stream_t stream) {
    // the argument checks of spec_verify, made here so that nothing is enqueued for a
    // call that spec_verify would reject
    const bool t1 = temperature == 1;
    if ((target_dtype != SPEC_F32 && target_dtype != SPEC_BF16) ||
        (t1 && draft_dtype != SPEC_F32 && draft_dtype != SPEC_BF16))
        return SPEC_ERR_DTYPE;
    if (B < 1 || B > 65535 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
    if (temperature != 0 && !t1) return SPEC_ERR_INVALID_ARG;
    if (!target_logits || !draft_tokens || !n_accepted_out || !committed_out || !bonus_out) return SPEC_ERR_INVALID_ARG;
    if (t1 && (!draft_logits || !seeds)) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(target_logits) & 15u) || (t1 && (reinterpret_cast<uintptr_t>(draft_logits) & 15u)))
        return SPEC_ERR_ALIGN;
    const size_t need = verify_workspace_bytes(B, gamma, V);
    if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_SHAPE;   // larger than the static array
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return record_cuda_error(e);
    // the kernels expect zeroed scratch; the array still holds the previous call's bytes
    e = cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream);
    if (e != cudaSuccess) return record_cuda_error(e);
    return spec_verify(target_logits, target_dtype, draft_logits, draft_dtype, draft_tokens, B, gamma, V, temperature,
                       seeds, n_accepted_out, committed_out, bonus_out, near_tie_out, scratch, need, stream);
}
