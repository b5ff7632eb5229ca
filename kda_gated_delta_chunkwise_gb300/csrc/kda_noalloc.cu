// kda_varlen_prefill_noalloc: the packed-batch prefill for callers that may
// not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run KDA: code
// that runs under a memory pool or arena it does not own (a serving engine
// that pre-plans all device memory at start-up and forbids allocations on
// its request path), plug-ins whose host framework hands them only the
// tensors of the call, and callers on a path where an allocation would
// synchronise the device. kda_varlen_prefill needs a small scratch buffer
// (the longest-first sequence order, a work counter and a status word);
// this entry point takes that scratch from a fixed array compiled into the
// library instead, so the caller passes only inputs and outputs.
//
// The array lives in device memory of every GPU that loads the library, for
// as long as the process runs; it holds KDA_NOALLOC_MAX_SEQS sequences.
#include <atomic>

#include "kda_internal.cuh"

#define KDA_STR2(x) #x
#define KDA_STR(x) KDA_STR2(x)

namespace {

constexpr size_t kScratchBytes = ((size_t)KDA_NOALLOC_MAX_SEQS * sizeof(int32_t) + 255) / 256 * 256 + 256;

// Shared by every call on a device. Host code must not use this name as a
// device address: on the host it is only a stand-in symbol. Its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does it) and kept for the life of
// the process. cudaDeviceReset destroys the context that address belongs to,
// so this entry point must not be used on a device after it was reset.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_varlen_prefill_noalloc(const void *q, const void *k, const void *v,
                                                   kda_dtype_t qkv_dtype, const float *alpha,
                                                   const float *beta, const float *initial_state,
                                                   void *o, float *final_state,
                                                   const int32_t *cu_seqlens, int N, int T_total,
                                                   int H, int d_k, int d_v, int32_t *device_status,
                                                   kda_stream_t stream) {
    if (N > KDA_NOALLOC_MAX_SEQS)
        return kda::set_error(KDA_ERR_UNSUPPORTED,
                              "kda_varlen_prefill_noalloc takes at most " KDA_STR(KDA_NOALLOC_MAX_SEQS)
                              " sequences; use kda_varlen_prefill with a workspace for more");
    void *scratch = nullptr;
    if (N > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess)
            return kda::set_error(KDA_ERR_CUDA, "looking up the device address of the no-alloc scratch failed");
    }
    // The prep kernel of the packed path rewrites the whole scratch it uses on
    // every call (order, counter zeroed, status), so no clearing is needed.
    return kda_varlen_prefill(q, k, v, qkv_dtype, alpha, beta, initial_state, o, final_state, cu_seqlens, N,
                              T_total, H, d_k, d_v, scratch, scratch ? kScratchBytes : 0, device_status,
                              stream);
}
