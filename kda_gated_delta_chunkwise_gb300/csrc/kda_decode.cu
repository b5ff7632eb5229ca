// KDA decode step: one token per (sequence, head), state updated in place.
//
// Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
// (pwwt.cn), §四 (KDA update) and §二.1 (read-out), for a single token:
//     S' = Diag(alpha) S;  v_hat = S'^T k;  e = beta (v - v_hat)
//     S  <- S' + k e^T;    o = S^T q = S'^T q + (q . k) e
// The essay's §一 and §二 note that decode is bandwidth-bound and that KDA's
// state has a fixed size: this kernel streams each head's d_k x d_v fp32
// state through registers exactly once (one read, one in-place write).
//
// Layout of the work: one CTA of 256 threads per head. A thread owns 4
// consecutive value columns (one 16-byte vector) of DK / ROWS_PER_PASS rows,
// so a warp reads whole 512-byte row segments (fully coalesced 128-bit
// loads). All of a thread's loads are issued before any arithmetic. The two
// column reductions over key rows (S'^T k and S'^T q) go through shared
// memory; the rank-1 write then needs only the reduced error vector.
//
// Gate kinds: the per-channel gate, one scalar gate per head (Gated DeltaNet)
// or none (the delta rule). With a slot map the state of sequence n is the
// pool entry slots[n] (zeros for a fresh slot); an out-of-range slot skips
// its heads and reports KDA_DEV_BAD_SLOT.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

__device__ __forceinline__ float4 ld_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 v) {
    __stcs(reinterpret_cast<float4 *>(p), v);
}

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kDecodeThreads, 2)
kda_decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                  const float *__restrict__ alpha, int gate, const float *__restrict__ beta,
                  float *__restrict__ state, const int32_t *__restrict__ slots, int pool_size,
                  int32_t *__restrict__ status, int H, TIn *__restrict__ o) {
    constexpr int TPR = DV / 4;                     // threads per state row
    constexpr int RPP = kDecodeThreads / TPR;       // rows per pass
    constexpr int PASSES = DK / RPP;                // rows per thread
    static_assert(DK % RPP == 0 && DK % 32 == 0, "row split");

    __shared__ float s_a[DK], s_ak[DK], s_aq[DK], s_k[DK];
    __shared__ float s_qkp[DK / 32];
    __shared__ __align__(16) float s_red_v[RPP][DV];
    __shared__ __align__(16) float s_red_o[RPP][DV];
    __shared__ __align__(16) float s_e[DV];

    const int64_t head = blockIdx.x;
    const int tid = threadIdx.x;
    const int col = (tid % TPR) * 4;
    const int row0 = tid / TPR;
    bool fresh;
    const int64_t slot = slot_of(slots, (int)(head / H), fresh);
    if (slots && slot >= pool_size) {  // uniform over the CTA
        if (tid == 0 && status) atomicOr(status, KDA_DEV_BAD_SLOT);
        return;
    }
    float *S = state + (slot * H + head % H) * (int64_t)DK * DV;

    // Issue the whole state tile first: PASSES independent 16-byte loads.
    float4 s[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
        s[p] = fresh ? make_float4(0.f, 0.f, 0.f, 0.f) : ld_stream(S + (int64_t)(row0 + p * RPP) * DV + col);

    // Gate, gated key / query and the partial sums of q.k.
    if (tid < DK) {
        const float a = gate_at(alpha, gate, head, tid, DK);
        const float kk = to_f32(k[head * DK + tid]);
        const float qq = to_f32(q[head * DK + tid]);
        s_a[tid] = a;
        s_k[tid] = kk;
        s_ak[tid] = a * kk;
        s_aq[tid] = a * qq;
        float qk = qq * kk;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
        if ((tid & 31) == 0) s_qkp[tid >> 5] = qk;
    }
    __syncthreads();

    // Partial column sums of S'^T k and S'^T q over this thread's rows;
    // S' = Diag(alpha) S stays in registers for the write.
    float4 pv = make_float4(0.f, 0.f, 0.f, 0.f), po = pv;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = row0 + p * RPP;
        const float ak = s_ak[i], aq = s_aq[i], a = s_a[i];
        pv.x += ak * s[p].x; pv.y += ak * s[p].y; pv.z += ak * s[p].z; pv.w += ak * s[p].w;
        po.x += aq * s[p].x; po.y += aq * s[p].y; po.z += aq * s[p].z; po.w += aq * s[p].w;
        s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
    }
    *reinterpret_cast<float4 *>(&s_red_v[row0][col]) = pv;
    *reinterpret_cast<float4 *>(&s_red_o[row0][col]) = po;
    __syncthreads();

    if (tid < DV) {
        float vh = 0.f, op = 0.f;
#pragma unroll 8
        for (int r = 0; r < RPP; ++r) {
            vh += s_red_v[r][tid];
            op += s_red_o[r][tid];
        }
        float qk = 0.f;
#pragma unroll
        for (int w = 0; w < DK / 32; ++w) qk += s_qkp[w];
        const float e = beta[head] * (to_f32(v[head * DV + tid]) - vh);
        s_e[tid] = e;
        o[head * DV + tid] = from_f32<TIn>(op + qk * e);
    }
    __syncthreads();

    const float4 e4 = *reinterpret_cast<const float4 *>(&s_e[col]);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = row0 + p * RPP;
        const float kk = s_k[i];
        float4 r = s[p];
        r.x += kk * e4.x; r.y += kk * e4.y; r.z += kk * e4.z; r.w += kk * e4.w;
        st_stream(S + (int64_t)i * DV + col, r);
    }
}

template <int DK, int DV, typename TIn>
cudaError_t launch_decode_t(const void *q, const void *k, const void *v, const float *alpha, int gate,
                            const float *beta, float *state, const int32_t *slots, int pool_size,
                            int32_t *status, void *o, int N, int H, cudaStream_t s) {
    const int64_t heads = (int64_t)N * H;
    if (heads == 0) return cudaSuccess;
    kda_decode_kernel<DK, DV, TIn><<<(unsigned)heads, kDecodeThreads, 0, s>>>(
        (const TIn *)q, (const TIn *)k, (const TIn *)v, alpha, gate, beta, state, slots, pool_size, status, H,
        (TIn *)o);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, kda_dtype_t dt,
                          const float *alpha, int gate, const float *beta, float *state,
                          const int32_t *slots, int pool_size, int32_t *status, void *o,
                          int N, int H, int dk, int dv, cudaStream_t s) {
#define KDA_DECODE_CASE(DK_, DV_)                                                                     \
    if (dk == DK_ && dv == DV_) {                                                                     \
        return dt == KDA_BF16 ? launch_decode_t<DK_, DV_, __nv_bfloat16>(q, k, v, alpha, gate, beta, state, \
                                                                        slots, pool_size, status, o, N, H, s) \
                              : launch_decode_t<DK_, DV_, float>(q, k, v, alpha, gate, beta, state, slots,  \
                                                                pool_size, status, o, N, H, s);            \
    }
    KDA_DECODE_CASE(128, 128)
    KDA_DECODE_CASE(64, 64)
    KDA_DECODE_CASE(128, 64)
    KDA_DECODE_CASE(64, 128)
#undef KDA_DECODE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
