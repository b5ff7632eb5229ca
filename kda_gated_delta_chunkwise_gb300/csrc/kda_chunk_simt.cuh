// Per-chunk tables of the chunkwise KDA algebra on CUDA cores (fp32) for the
// CUDA-core prefill; the backward shares the constants, the table layout and
// the inverse.
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
    float al[TPS], kk[TPS], qq[TPS];  // every load of the thread in flight at once
#pragma unroll
    for (int i = 0; i < TPS; ++i) {
        const int r = seg * TPS + i;
        const int64_t th = (tok0 + r) * H + h;
        const bool in = r < L;
        al[i] = in ? gate_at(alpha, gate, th, c, DK) : 1.f;
        kk[i] = in ? ld_in(k, th * DK + c) : 0.f;
        qq[i] = in ? ld_in(q, th * DK + c) : 0.f;
    }
    float prod = 1.f;
#pragma unroll
    for (int i = 0; i < TPS; ++i) prod *= al[i];
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
        const float e2 = pre * inv_mu, e3 = suf[i] * inv_mu;
        tb.Kr[r * LDK + c] = kk[i] * e2;
        tb.Qr[r * LDK + c] = qq[i] * e2;
        tb.Kc[r * LDK + c] = kk[i] * e3;
    }
    if (tid < C) tb.beta[tid] = tid < L ? beta[(tok0 + tid) * H + h] : 0.f;
    __syncthreads();
}

// A = beta (Kr Kc^T) strictly lower and P = Qr Kc^T lower incl. diagonal, in
// fp32 on CUDA cores. Ends with a barrier.
template <int DK> __device__ void wy_products(Tables<DK> &tb) {
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
}

// T = (I + A)^{-1} for a strictly lower A ([C][C + 4] tiles in shared
// memory; forward substitution on 16 x 16 blocks, then block products).
// Leaves A's upper triangle overwritten. Ends with a barrier.
struct TPair {
    float *A, *T;
};
__device__ inline void invert_unit_lower(TPair tb) {
    constexpr int LDC = C + 4;
    const int tid = threadIdx.x;
    // T = (I + A)^{-1} by blocks of 16 (A strictly lower, so T is unit lower):
    //   the four diagonal blocks by forward substitution, one thread per column;
    //   then T_{b+1,b} = -T_{b+1,b+1} A_{b+1,b} T_{b,b} for the pairs (0,1), (2,3);
    //   then T[32:64, 0:32] = -T[32:64, 32:64] (A[32:64, 0:32] T[0:32, 0:32]).
    // The products in between sit in A's upper triangle, which is zero and
    // unread: A[0:16, 16:32] and A[32:48, 48:64] for the pairs, A[0:32, 32:64]
    // for the 32 x 32 block.
    for (int e = tid; e < C * C; e += NT) tb.T[(e / C) * LDC + e % C] = 0.f;
    __syncthreads();
    if (tid < C) {
        const int bk = tid >> 4, col = tid & 15, o = 16 * bk;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = i == col ? 1.f : 0.f;
#pragma unroll
        for (int sidx = 0; sidx < 15; ++sidx)
#pragma unroll
            for (int r = sidx + 1; r < 16; ++r) x[r] -= tb.A[(o + r) * LDC + o + sidx] * x[sidx];
#pragma unroll
        for (int r = 0; r < 16; ++r) tb.T[(o + r) * LDC + o + col] = x[r];
    }
    __syncthreads();
    {
        // M = A_{b+1,b} T_{b,b} for both pairs: 2 x 256 entries, two per thread
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = tid + NT * u, pr = e >> 8, r = (e >> 4) & 15, c = e & 15, o = 32 * pr;
            float m = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) m += tb.A[(o + 16 + r) * LDC + o + kk] * tb.T[(o + kk) * LDC + o + c];
            tb.A[(o + r) * LDC + o + 16 + c] = m;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = tid + NT * u, pr = e >> 8, r = (e >> 4) & 15, c = e & 15, o = 32 * pr;
            float m = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) m += tb.T[(o + 16 + r) * LDC + o + 16 + kk] * tb.A[(o + kk) * LDC + o + 16 + c];
            tb.T[(o + 16 + r) * LDC + o + c] = -m;
        }
        __syncthreads();
        // M2 = A[32:64, 0:32] T[0:32, 0:32]: 1024 entries, four per thread
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = tid + NT * u, r = e >> 5, c = e & 31;
            float m = 0.f;
#pragma unroll 8
            for (int kk = 0; kk < 32; ++kk) m += tb.A[(32 + r) * LDC + kk] * tb.T[kk * LDC + c];
            tb.A[r * LDC + 32 + c] = m;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = tid + NT * u, r = e >> 5, c = e & 31;
            float m = 0.f;
#pragma unroll 8
            for (int kk = 0; kk < 32; ++kk) m += tb.T[(32 + r) * LDC + 32 + kk] * tb.A[kk * LDC + 32 + c];
            tb.T[(32 + r) * LDC + c] = -m;
        }
        __syncthreads();
    }
}

// The WY tables of a chunk whose gated tables are in tb: A, P, then T.
template <int DK> __device__ void wy_tables(Tables<DK> &tb) {
    wy_products<DK>(tb);
    invert_unit_lower(TPair{tb.A, tb.T});
}

}  // namespace simt
}  // namespace kda
