// Internal declarations shared by the host layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Element loads/stores for the two input dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Gate of key channel c at token-head index th (= token * H + head): the
// channel's own gate, the token-head's scalar gate for every channel, or 1.
__device__ __forceinline__ float gate_at(const float *alpha, int gate, int64_t th, int c, int dk) {
    return gate == KDA_GATE_CHANNEL ? alpha[th * dk + c] : gate == KDA_GATE_SCALAR ? alpha[th] : 1.f;
}

// State slot of sequence n: slots[n] >= 0 is a slot whose state is read and
// written back, -1 - s is slot s starting from zeros (fresh = true). Without
// a slot map the state of sequence n is entry n.
__device__ __forceinline__ int64_t slot_of(const int32_t *slots, int n, bool &fresh) {
    if (!slots) {
        fresh = false;
        return n;
    }
    const int32_t s = slots[n];
    fresh = s < 0;
    return fresh ? -1 - (int64_t)s : (int64_t)s;
}

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_decode(const void *q, const void *k, const void *v, kda_dtype_t dt,
                          const float *alpha, int gate, const float *beta, float *state,
                          const int32_t *slots, int pool_size, int32_t *status, void *o,
                          int N, int H, int dk, int dv, cudaStream_t s);

// Prefill over sequences given by cu_seqlens (device) or, when cu_seqlens is
// null, B equal sequences of T tokens. `order` (device, nullable) lists the
// (sequence, head) work items to run, longest first; `counter` (device,
// nullable) is a zeroed work counter for persistent scheduling.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *alpha, *beta, *s0;
    void *o;
    float *sT;
    int gate;                   // kda_gate_t: the layout of alpha
    const int32_t *slots;       // nullable: state slot map (see slot_of); s0 and sT are then the pool
    bool fp8;                   // q, k, v are E4M3 codes with E8M0 scales qs, ks, vs (o is bf16)
    const uint8_t *qs, *ks, *vs;
    const int32_t *cu_seqlens;  // null: equal lengths
    int N, T, H, dk, dv;        // T: tokens per sequence (equal) or T_total (packed)
    kda_dtype_t dt;
    const int32_t *order;       // nullable: sequence order (longest first)
    int32_t *counter;           // nullable: persistent work counter
    const int32_t *dev_status;  // nullable: skip all work when *dev_status != 0
    int stall1;                 // self-test of the tensor-core kernel's bounded waits: 1 + the
                                // chunk at which its state chain stops (0, the default: never)
};

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
bool prefill_tc_supported(const PrefillArgs &a);
// Reads (and optionally clears) the tensor-core kernel's error word.
cudaError_t read_device_error(int *out, bool reset);

// Backward of the prefill (equal-length batches, per-channel gate). Every
// gradient is float32; d_o has the dtype of q, k, v.
struct BackwardArgs {
    const void *q, *k, *v, *d_o;
    kda_dtype_t dt;
    const float *alpha, *beta, *s0, *dsT;  // s0, dsT nullable (zeros)
    float *dq, *dk, *dvv, *dalpha, *dbeta;
    float *ds0;                            // nullable
    void *workspace;                       // backward_workspace_bytes, 16-byte aligned
    int gate;                              // kda_gate_t (layout of alpha and dalpha)
    int N, T, H, d_k, d_v;                 // packed: T is T_total
    const int32_t *cu_seqlens;             // nullable: packed sequences
    int32_t *dev_status;                   // packed, nullable: the device status word
};
size_t backward_workspace_bytes(int N, int T, int H, int dk, int dv, bool packed);
cudaError_t launch_backward(const BackwardArgs &b, cudaStream_t s);

// Varlen preparation: validates cu_seqlens, writes the status word, sorts the
// sequences by length (longest first) into `order` and zeroes `counter`.
// With a slot map it also checks that every slot lies in [0, pool_size).
cudaError_t launch_varlen_prep(const int32_t *cu_seqlens, int N, int T_total, int32_t *order,
                               int32_t *counter, int32_t *status, const int32_t *slots, int pool_size,
                               cudaStream_t s);

// kda_varlen_prefill with a gate kind (kda_gate_t) and no slot map.
kda_status_t varlen_prefill_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                 const float *alpha, int gate, const float *beta, const float *initial_state,
                                 void *o, float *final_state, const int32_t *cu_seqlens, int N, int T_total, int H,
                                 int d_k, int d_v, void *workspace, size_t workspace_bytes, int32_t *device_status,
                                 cudaStream_t s);

// Records `msg` as this thread's last error and returns `st`.
kda_status_t set_error(kda_status_t st, const char *msg);

}  // namespace kda
