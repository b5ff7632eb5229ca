// Per-chunk tables of the chunkwise KDA algebra on CUDA cores (fp32), shared
// by the fp32 prefill kernel and the backward kernels.
//
// Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
// (pwwt.cn), the K3 essay: §四 (KDA update), §六.1 (chunks) and §六.2 (the
// WY form: the chunk's rank-1 updates gathered into a few dense products).
//
// For a chunk of C = 64 tokens (rows r, j; key channels c; gates in linear
// space):
//   p_r   = prod_{s<=r} alpha_s (per channel), gamma = p_{C-1}, mu = sqrt(gamma)
//   Kr    = k (.) p / mu,   Qr = q (.) p / mu,   Kc = k (.) (prod_{s>j} alpha_s) / mu
//   A     = strictly-lower( beta_r Kr Kc^T ),  P = lower-incl-diag( Qr Kc^T )
//   T     = (I + A)^{-1}                          (forward substitution)
// Every factor lies in [mu, 1/mu]. A chunk where some channel decays by more
// than e^-80 is flagged `slow`: its callers run it token by token instead.
// Rows past the end of the sequence read as k = q = 0, alpha = 1, beta = 0.
#pragma once

#include <cstddef>

#include "kda_internal.cuh"

namespace kda {
namespace simt {

constexpr int C = 64;          // chunk length
constexpr int VS = 64;         // value columns per CTA
constexpr int NT = 256;        // threads per CTA
constexpr float kMinGamma = 1.8e-35f;  // ~exp(-80): chunk decay limit of the WY form

// 16-byte aligned (and so sized in multiples of 16 bytes): the kernels read
// these tables, and the shared-memory arrays placed after them, as float4.
template <int DK> struct alignas(16) Tables {
    static constexpr int LDK = DK + 4;  // padded row of a [C][DK] table
    static constexpr int LDC = C + 4;   // padded row of a [C][C] table
    float Kr[C * LDK];
    float Qr[C * LDK];
    float Kc[C * LDK];
    float T[C * LDC];
    float P[C * LDC];
    float A[C * LDC];   // strictly lower A (only during the substitution; free afterwards)
    float mu[DK];
    float beta[C];
    float part[4 * DK];
    int slow;
};

static_assert(sizeof(Tables<64>) % 16 == 0 && sizeof(Tables<128>) % 16 == 0, "float4 alignment");
static_assert(offsetof(Tables<128>, Qr) % 16 == 0 && offsetof(Tables<128>, Kc) % 16 == 0 &&
                  offsetof(Tables<128>, T) % 16 == 0 && offsetof(Tables<128>, P) % 16 == 0 &&
                  offsetof(Tables<128>, A) % 16 == 0 && offsetof(Tables<64>, T) % 16 == 0,
              "float4 alignment");

template <typename TIn>
__device__ __forceinline__ float ld_in(const TIn *p, int64_t i) { return to_f32(p[i]); }

// Gate products, mu, the slow flag and the gated tables Kr, Qr, Kc of the
// chunk whose first token is tok0 (L valid rows), plus beta. One thread per
// channel and token segment. Ends with a barrier.
template <int DK, typename TIn>
__device__ void gate_tables(Tables<DK> &tb, const float *alpha, int gate, const TIn *q, const TIn *k,
                            const float *beta, int64_t tok0, int L, int H, int h) {
    constexpr int LDK = Tables<DK>::LDK;
    constexpr int SEG = NT / DK;       // token segments per channel
    constexpr int TPS = C / SEG;       // tokens per segment
    const int tid = threadIdx.x;
    const int c = tid % DK, seg = tid / DK;
    float al[TPS];
    float prod = 1.f;
#pragma unroll
    for (int i = 0; i < TPS; ++i) {
        const int r = seg * TPS + i;
        al[i] = r < L ? gate_at(alpha, gate, (tok0 + r) * H + h, c, DK) : 1.f;
        prod *= al[i];
    }
    tb.part[seg * DK + c] = prod;
    if (tid == 0) tb.slow = 0;
    __syncthreads();
    float before = 1.f, after = 1.f, gamma = 1.f;
#pragma unroll
    for (int s2 = 0; s2 < SEG; ++s2) {
        const float pt = tb.part[s2 * DK + c];
        if (s2 < seg) before *= pt;
        if (s2 > seg) after *= pt;
        gamma *= pt;
    }
    if (gamma < kMinGamma) tb.slow = 1;
    const float mu = sqrtf(gamma);
    const float inv_mu = 1.f / mu;
    if (seg == 0) tb.mu[c] = mu;
    // prefix (inclusive) and suffix (exclusive) products in this segment
    float pre = before;
    float suf[TPS];
    float s_acc = after;
#pragma unroll
    for (int i = TPS - 1; i >= 0; --i) {
        suf[i] = s_acc;
        s_acc *= al[i];
    }
#pragma unroll
    for (int i = 0; i < TPS; ++i) {
        const int r = seg * TPS + i;
        pre *= al[i];
        float kk = 0.f, qq = 0.f;
        if (r < L) {
            kk = ld_in(k, ((tok0 + r) * H + h) * DK + c);
            qq = ld_in(q, ((tok0 + r) * H + h) * DK + c);
        }
        const float e2 = pre * inv_mu, e3 = suf[i] * inv_mu;
        tb.Kr[r * LDK + c] = kk * e2;
        tb.Qr[r * LDK + c] = qq * e2;
        tb.Kc[r * LDK + c] = kk * e3;
    }
    if (tid < C) tb.beta[tid] = tid < L ? beta[(tok0 + tid) * H + h] : 0.f;
    __syncthreads();
}

// The gate factor p / mu of every row and channel of the chunk (the factor
// that made Kr and Qr) into E2 ([C][ld] floats), with the same arithmetic as
// gate_tables, so the same bits. Needs tb.mu of the chunk; uses tb.part as
// scratch. Ends with a barrier.
template <int DK>
__device__ void gate_factor_table(Tables<DK> &tb, float *E2, int ld, const float *alpha, int gate, int64_t tok0, int L,
                                  int H, int h) {
    constexpr int SEG = NT / DK;
    constexpr int TPS = C / SEG;
    const int tid = threadIdx.x;
    const int c = tid % DK, seg = tid / DK;
    float al[TPS];
    float prod = 1.f;
#pragma unroll
    for (int i = 0; i < TPS; ++i) {
        const int r = seg * TPS + i;
        al[i] = r < L ? gate_at(alpha, gate, (tok0 + r) * H + h, c, DK) : 1.f;
        prod *= al[i];
    }
    __syncthreads();  // earlier readers of tb.part are done
    tb.part[seg * DK + c] = prod;
    __syncthreads();
    float before = 1.f;
#pragma unroll
    for (int s2 = 0; s2 < SEG; ++s2)
        if (s2 < seg) before *= tb.part[s2 * DK + c];
    const float inv_mu = 1.f / tb.mu[c];
    float pre = before;
#pragma unroll
    for (int i = 0; i < TPS; ++i) {
        pre *= al[i];
        E2[(seg * TPS + i) * ld + c] = pre * inv_mu;
    }
    __syncthreads();
}

// A = beta (Kr Kc^T) strictly lower, P = Qr Kc^T lower incl. diagonal, then
// T = (I + A)^{-1} one row at a time (forward substitution). Ends with a
// barrier.
template <int DK> __device__ void wy_tables(Tables<DK> &tb) {
    constexpr int LDK = Tables<DK>::LDK, LDC = Tables<DK>::LDC;
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    {
        float accA[4][4], accP[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) accA[i][jj] = accP[i][jj] = 0.f;
        for (int c = 0; c < DK; c += 4) {
            float4 kr[4], qr[4], kc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                kr[i] = *reinterpret_cast<const float4 *>(&tb.Kr[(ty + 16 * i) * LDK + c]);
                qr[i] = *reinterpret_cast<const float4 *>(&tb.Qr[(ty + 16 * i) * LDK + c]);
                kc[i] = *reinterpret_cast<const float4 *>(&tb.Kc[(tx + 16 * i) * LDK + c]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    accA[i][jj] += kr[i].x * kc[jj].x + kr[i].y * kc[jj].y + kr[i].z * kc[jj].z + kr[i].w * kc[jj].w;
                    accP[i][jj] += qr[i].x * kc[jj].x + qr[i].y * kc[jj].y + qr[i].z * kc[jj].z + qr[i].w * kc[jj].w;
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int r = ty + 16 * i, j = tx + 16 * jj;
                tb.A[r * LDC + j] = j < r ? tb.beta[r] * accA[i][jj] : 0.f;
                tb.P[r * LDC + j] = j <= r ? accP[i][jj] : 0.f;
            }
    }
    __syncthreads();
    {
        const int j = tid / 4, part = tid % 4;  // column j, 4-way split of the sum
        for (int r = 0; r < C; ++r) {
            float s = 0.f;
            if (j < r)
                for (int sidx = j + part; sidx < r; sidx += 4) s += tb.A[r * LDC + sidx] * tb.T[sidx * LDC + j];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (part == 0) tb.T[r * LDC + j] = j < r ? -s : (j == r ? 1.f : 0.f);
            __syncthreads();
        }
    }
}

}  // namespace simt
}  // namespace kda
