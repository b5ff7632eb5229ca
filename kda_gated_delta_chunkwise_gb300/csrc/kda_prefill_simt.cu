// KDA chunkwise prefill on CUDA cores, fp32 arithmetic throughout.
//
// Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
// (pwwt.cn), called the K3 essay: §四 (KDA update), §五 (transition
// products A_t ... A_{j+1}), §六.1 (chunks: recursion between chunks,
// parallel work inside) and §六.2 (WY form: a run of rank-1 updates becomes
// D - K W^T, handled as a few dense products per chunk).
//
// This is the fp32 path (fp32 inputs, 1e-4 accuracy) and the CUDA-core
// counterpart of the tensor-core kernel: it evaluates the same chunk algebra.
// For a chunk of C = 64 tokens with start state S0 (token rows r, j; key
// channels c; gates in linear space):
//
//   p_r    = prod_{s<=r} alpha_s        (cumulative gate product, per channel)
//   gamma  = p_{C-1},  mu = sqrt(gamma) (the chunk's mid-point in log space)
//   E2_r   = p_r / mu,  E3_j = (prod_{s>j} alpha_s) / mu
//   Kr = k (.) E2,  Qr = q (.) E2,  Kc = k (.) E3        (so Kr_r . Kc_j has
//                                      the factor exp(g_r - g_j) <= 1)
//   A  = strictly-lower( beta_r Kr Kc^T ),   P = lower-incl-diag( Qr Kc^T )
//   T  = (I + A)^{-1}                         (forward substitution)
//   St = Diag(mu) S0
//   X  = Kr St = (k (.) p) S0,   Y = Qr St = (q (.) p) S0
//   R  = Diag(beta) (V - X),     U = T R       (the pseudo-values)
//   O  = Y + P U                               (o_r = S_r^T q_r)
//   S1 = Diag(mu) (St + Kc^T U) = Diag(gamma) S0 + (k (.) prod_{s>j} alpha)^T U
//
// The essay's D - K W^T is the chunk transition Diag(gamma) - Khat^T T Diag(beta)
// (K (.) Gamma) implied here. Every factor stays within [mu, 1/mu]; chunks in
// which some channel decays by more than e^-80 (mu < e^-40) are instead run
// token by token (the plain §四 update), which is exact for any alpha in
// [0, 1], including 0.
//
// Work split: one CTA of 256 threads per (sequence, head, 64-column slice of
// d_v). The state slice lives in shared memory for the whole sequence.
#include "kda_chunk_simt.cuh"

namespace kda {
namespace {

using simt::C;
using simt::NT;
using simt::VS;
using simt::ld_in;

template <int DK> struct SimtSmem {
    float S[DK * VS];
    simt::Tables<DK> tb;
    float R[C * VS];
    float U[C * VS];
};

static_assert(offsetof(SimtSmem<64>, R) % 16 == 0 && offsetof(SimtSmem<128>, R) % 16 == 0 &&
                  offsetof(SimtSmem<64>, U) % 16 == 0 && offsetof(SimtSmem<128>, U) % 16 == 0 &&
                  offsetof(SimtSmem<128>, tb) % 16 == 0,
              "float4 accesses need 16-byte offsets");

template <int DK, typename TIn>
__global__ void __launch_bounds__(NT, 1) kda_prefill_simt_kernel(PrefillArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<DK> &sm = *reinterpret_cast<SimtSmem<DK> *>(smem_raw);
    simt::Tables<DK> &tb = sm.tb;
    constexpr int LDK = simt::Tables<DK>::LDK;
    constexpr int LDC = simt::Tables<DK>::LDC;

    if (a.dev_status && *a.dev_status != 0) return;

    const int tid = threadIdx.x;
    const int nslices = a.dv / VS;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % a.H;
    const int item = blockIdx.x / (nslices * a.H);
    const int n = a.order ? a.order[item] : item;
    int64_t t_begin, T;
    if (a.cu_seqlens) {
        t_begin = a.cu_seqlens[n];
        T = (int64_t)a.cu_seqlens[n + 1] - t_begin;
    } else {
        t_begin = (int64_t)n * a.T;
        T = a.T;
    }
    const int H = a.H, DV = a.dv;
    const int v0 = slice * VS;
    const TIn *q = (const TIn *)a.q;
    const TIn *k = (const TIn *)a.k;
    const TIn *v = (const TIn *)a.v;
    TIn *o = (TIn *)a.o;
    bool fresh;
    const int64_t state_off = (slot_of(a.slots, n, fresh) * H + h) * DK * DV;

    // ---- initial state slice ----
    for (int e = tid; e < DK * VS; e += NT) {
        const int c = e / VS, j = e % VS;
        sm.S[e] = (a.s0 && !fresh) ? a.s0[state_off + (int64_t)c * DV + v0 + j] : 0.f;
    }
    __syncthreads();

    // thread tiles for the 64-row products: rows ty + 16 i, 4 consecutive cols
    const int tx = tid % 16, ty = tid / 16;

    for (int64_t t0 = 0; t0 < T; t0 += C) {
        const int L = (int)((T - t0) < C ? (T - t0) : (int64_t)C);
        const int64_t tok0 = t_begin + t0;

        // ---- gate products, factors and the gated tables ----
        simt::gate_tables<DK, TIn>(tb, a.alpha, a.gate, q, k, a.beta, tok0, L, H, h);

        if (tb.slow) {
            // ---- exact token-by-token fallback for strongly decaying chunks ----
            for (int r = 0; r < L; ++r) {
                const int64_t tk = (tok0 + r) * H + h;
                const int j = tid % VS, part = tid / VS;  // 4 parts of the key rows
                float vh = 0.f;
                for (int c = part; c < DK; c += NT / VS)
                    vh += gate_at(a.alpha, a.gate, tk, c, DK) * ld_in(k, tk * DK + c) * sm.S[c * VS + j];
                sm.R[part * VS + j] = vh;
                __syncthreads();
                if (tid < VS) {
                    float s = 0.f;
                    for (int p2 = 0; p2 < NT / VS; ++p2) s += sm.R[p2 * VS + tid];
                    sm.U[tid] = a.beta[tk] * (ld_in(v, tk * DV + v0 + tid) - s);
                }
                __syncthreads();
                float op = 0.f;
                for (int c = part; c < DK; c += NT / VS) {
                    const float sn = gate_at(a.alpha, a.gate, tk, c, DK) * sm.S[c * VS + j] +
                                     ld_in(k, tk * DK + c) * sm.U[j];
                    sm.S[c * VS + j] = sn;
                    op += ld_in(q, tk * DK + c) * sn;
                }
                sm.R[part * VS + j] = op;
                __syncthreads();
                if (tid < VS) {
                    float s = 0.f;
                    for (int p2 = 0; p2 < NT / VS; ++p2) s += sm.R[p2 * VS + tid];
                    o[tk * DV + v0 + tid] = from_f32<TIn>(s);
                }
                __syncthreads();
            }
            continue;
        }

        // ---- A = beta (Kr Kc^T) strictly lower, P = Qr Kc^T, T = (I + A)^{-1} ----
        simt::wy_tables<DK>(tb);

        // ---- X = Kr St, Y = Qr St (St = Diag(mu) S0), R = beta (V - X) ----
        float y[4][4];
        {
            float x[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) x[i][jj] = y[i][jj] = 0.f;
            for (int c = 0; c < DK; c += 4) {
                float4 kr[4], qr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kr[i] = *reinterpret_cast<const float4 *>(&tb.Kr[(ty + 16 * i) * LDK + c]);
                    qr[i] = *reinterpret_cast<const float4 *>(&tb.Qr[(ty + 16 * i) * LDK + c]);
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const float m = tb.mu[c + cc];
                    float4 s4 = *reinterpret_cast<const float4 *>(&sm.S[(c + cc) * VS + 4 * tx]);
                    s4.x *= m; s4.y *= m; s4.z *= m; s4.w *= m;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float kv = cc == 0 ? kr[i].x : cc == 1 ? kr[i].y : cc == 2 ? kr[i].z : kr[i].w;
                        const float qv = cc == 0 ? qr[i].x : cc == 1 ? qr[i].y : cc == 2 ? qr[i].z : qr[i].w;
                        x[i][0] += kv * s4.x; x[i][1] += kv * s4.y; x[i][2] += kv * s4.z; x[i][3] += kv * s4.w;
                        y[i][0] += qv * s4.x; y[i][1] += qv * s4.y; y[i][2] += qv * s4.z; y[i][3] += qv * s4.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = ty + 16 * i;
                const float b = tb.beta[r];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float vv = r < L ? ld_in(v, ((tok0 + r) * H + h) * DV + v0 + 4 * tx + jj) : 0.f;
                    sm.R[r * VS + 4 * tx + jj] = b * (vv - x[i][jj]);
                }
            }
        }
        __syncthreads();

        // ---- U = T R ----
        {
            float u[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) u[i][jj] = 0.f;
            for (int j = 0; j < C; j += 4) {
                float4 t4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    t4[i] = *reinterpret_cast<const float4 *>(&tb.T[(ty + 16 * i) * LDC + j]);
#pragma unroll
                for (int jj2 = 0; jj2 < 4; ++jj2) {
                    const float4 r4 = *reinterpret_cast<const float4 *>(&sm.R[(j + jj2) * VS + 4 * tx]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float tv = jj2 == 0 ? t4[i].x : jj2 == 1 ? t4[i].y : jj2 == 2 ? t4[i].z : t4[i].w;
                        u[i][0] += tv * r4.x; u[i][1] += tv * r4.y; u[i][2] += tv * r4.z; u[i][3] += tv * r4.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(&sm.U[(ty + 16 * i) * VS + 4 * tx]) =
                    make_float4(u[i][0], u[i][1], u[i][2], u[i][3]);
        }
        __syncthreads();

        // ---- O = Y + P U (rows < L written) ----
        {
            for (int j = 0; j < C; j += 4) {
                float4 p4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    p4[i] = *reinterpret_cast<const float4 *>(&tb.P[(ty + 16 * i) * LDC + j]);
#pragma unroll
                for (int jj2 = 0; jj2 < 4; ++jj2) {
                    const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[(j + jj2) * VS + 4 * tx]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float pv = jj2 == 0 ? p4[i].x : jj2 == 1 ? p4[i].y : jj2 == 2 ? p4[i].z : p4[i].w;
                        y[i][0] += pv * u4.x; y[i][1] += pv * u4.y; y[i][2] += pv * u4.z; y[i][3] += pv * u4.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = ty + 16 * i;
                if (r < L) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        o[((tok0 + r) * H + h) * DV + v0 + 4 * tx + jj] = from_f32<TIn>(y[i][jj]);
                }
            }
        }

        // ---- S1 = Diag(mu) (Diag(mu) S0 + Kc^T U) ----
        {
            // tile: key rows 4 * ty2 .. +3 (+ 64 for DK = 128), 4 columns
            constexpr int RB = DK / 64;  // row blocks of 64
            float acc[RB][4][4];
#pragma unroll
            for (int b2 = 0; b2 < RB; ++b2)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) acc[b2][i][jj] = 0.f;
            for (int j = 0; j < C; ++j) {
                const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[j * VS + 4 * tx]);
#pragma unroll
                for (int b2 = 0; b2 < RB; ++b2) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&tb.Kc[j * LDK + 64 * b2 + 4 * ty]);
                    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[b2][i][0] += kv[i] * u4.x; acc[b2][i][1] += kv[i] * u4.y;
                        acc[b2][i][2] += kv[i] * u4.z; acc[b2][i][3] += kv[i] * u4.w;
                    }
                }
            }
            __syncthreads();  // every thread has read S (for X, Y) long before; U done
#pragma unroll
            for (int b2 = 0; b2 < RB; ++b2)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 64 * b2 + 4 * ty + i;
                    const float m = tb.mu[c];
                    float4 s4 = *reinterpret_cast<float4 *>(&sm.S[c * VS + 4 * tx]);
                    s4.x = m * (m * s4.x + acc[b2][i][0]);
                    s4.y = m * (m * s4.y + acc[b2][i][1]);
                    s4.z = m * (m * s4.z + acc[b2][i][2]);
                    s4.w = m * (m * s4.w + acc[b2][i][3]);
                    *reinterpret_cast<float4 *>(&sm.S[c * VS + 4 * tx]) = s4;
                }
        }
        __syncthreads();
    }

    // ---- final state slice ----
    if (a.sT) {
        for (int e = tid; e < DK * VS; e += NT) {
            const int c = e / VS, j = e % VS;
            a.sT[state_off + (int64_t)c * DV + v0 + j] = sm.S[e];
        }
    }
}

template <int DK, typename TIn>
cudaError_t launch_simt_t(const PrefillArgs &a, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.N * a.H * (a.dv / VS);
    if (blocks == 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(SimtSmem<DK>);
    auto kern = kda_prefill_simt_kernel<DK, TIn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s) {
    if (a.dv % VS != 0) return cudaErrorInvalidValue;
    if (a.dk == 128)
        return a.dt == KDA_BF16 ? launch_simt_t<128, __nv_bfloat16>(a, s) : launch_simt_t<128, float>(a, s);
    if (a.dk == 64)
        return a.dt == KDA_BF16 ? launch_simt_t<64, __nv_bfloat16>(a, s) : launch_simt_t<64, float>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace kda
