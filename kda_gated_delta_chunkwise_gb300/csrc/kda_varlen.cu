// Packed-batch preparation for kda_varlen_prefill, entirely on the device
// (the host never reads cu_seqlens, so no synchronisation is needed).
//
// One CTA:
//   1. checks cu_seqlens (cu[0] == 0, never decreasing, cu[N] == T_total) and,
//      with a slot map, that every state slot lies in [0, pool_size); writes
//      KDA_DEV_OK, KDA_DEV_BAD_CU_SEQLENS or KDA_DEV_BAD_SLOT to the status
//      word; the prefill kernels that follow on the stream read it and skip
//      all work on a bad batch, so nothing is written out of bounds;
//   2. lists the sequences longest first (stable: equal lengths keep their
//      index order), so the longest recurrences start in the first wave and
//      the tail of the launch is made of short ones;
//   3. zeroes the work counter used by persistent kernels.
// Sorting uses ranks (rank_i = #{j : L_j > L_i, or L_j == L_i and j < i}),
// which is exact and deterministic; above kMaxSorted sequences the order is
// the identity (many sequences are short on average and the tail effect is
// small).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 1024;
constexpr int kMaxSorted = 4096;

__global__ void __launch_bounds__(kPrepThreads)
kda_varlen_prep_kernel(const int32_t *__restrict__ cu, int N, int T_total, int32_t *__restrict__ order,
                       int32_t *__restrict__ counter, int32_t *__restrict__ status,
                       const int32_t *__restrict__ slots, int pool_size) {
    __shared__ int bad, bad_slot;
    __shared__ int32_t len_s[kMaxSorted];
    const int tid = threadIdx.x;
    if (tid == 0) {
        bad = (cu[0] != 0 || cu[N] != T_total) ? 1 : 0;
        bad_slot = 0;
    }
    __syncthreads();
    for (int i = tid; i < N; i += kPrepThreads) {
        const int32_t lo = cu[i], hi = cu[i + 1];
        if (hi < lo) atomicOr(&bad, 1);
        if (N <= kMaxSorted) len_s[i] = hi - lo;
        if (slots) {
            bool fresh;
            const int64_t sl = slot_of(slots, i, fresh);
            if (sl >= pool_size) atomicOr(&bad_slot, 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        *status = bad ? KDA_DEV_BAD_CU_SEQLENS : bad_slot ? KDA_DEV_BAD_SLOT : KDA_DEV_OK;
        if (counter) *counter = 0;
    }
    if (bad_slot) return;
    if (bad) return;
    if (N <= kMaxSorted) {
        for (int i = tid; i < N; i += kPrepThreads) {
            const int32_t li = len_s[i];
            int rank = 0;
            for (int j = 0; j < N; ++j) {
                const int32_t lj = len_s[j];
                rank += (lj > li) || (lj == li && j < i);
            }
            order[rank] = i;
        }
    } else {
        for (int i = tid; i < N; i += kPrepThreads) order[i] = i;
    }
}

}  // namespace

cudaError_t launch_varlen_prep(const int32_t *cu_seqlens, int N, int T_total, int32_t *order,
                               int32_t *counter, int32_t *status, const int32_t *slots, int pool_size,
                               cudaStream_t s) {
    kda_varlen_prep_kernel<<<1, kPrepThreads, 0, s>>>(cu_seqlens, N, T_total, order, counter, status, slots,
                                                     pool_size);
    return cudaGetLastError();
}

}  // namespace kda
