// KDA chunkwise prefill on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), bf16 q/k/v, fp32 gates, fp32 state, d_k = d_v = 128.
//
// Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
// (pwwt.cn), the K3 essay: §四 (KDA update S_t = (I - b k k^T) Diag(a) S + b k v^T),
// §五 (transition products), §六.1 (chunks: recursion between chunks, parallel
// work inside) and §六.2 (WY form: the chunk's rank-1 updates as a few dense
// products, transition D - K W^T).
//
// Chunk algebra (C = 64 tokens r, j; key channels c; value columns v), with
// p_r the cumulative gate product inside the chunk, gamma = p_{C-1} and
// mu = sqrt(gamma) the chunk's mid-point in log space:
//   Kr = k (.) p / mu,  Qr = q (.) p / mu,  Kc = k (.) (prod_{s>j} alpha) / mu
//   [A; P] = [Kr; Qr] Kc^T          A strictly lower x beta_r, P lower incl. diag
//   T = (I + A)^{-1}                forward substitution (CUDA cores + mma.sync)
//   St = Diag(mu) S                 (bf16 operand copy of the fp32 state)
//   [X; Y] = [Kr; Qr] St            X = (k (.) p) S, Y = (q (.) p) S
//   R = Diag(beta)(V - X);  U = T R;  O = Y + P U
//   S <- Diag(mu) (St + Kc^T U)     (fp32, accumulated in TMEM)
// Every gated factor lies in [mu, 1/mu]; a chunk in which some channel decays
// by more than e^-80 is run token by token instead (exact for alpha = 0).
//
// One CTA per (sequence, head, 64-wide slice of d_v); 448 threads:
//   warps 0-3   epilogue warpgroup: the state chain (R, U, O, S) - one TMEM lane each
//   warps 4-11  prep: gate products, gated tables, A/P read-out, T, the [T; P] tile
//   warp 12     TMA producer (q, k, alpha, v tiles; 2-deep rings)
//   warp 13     MMA issuer (one thread) and TMEM owner
// The prep of chunk n+1 overlaps the state chain of chunk n. All waits are
// bounded; on a timeout the CTA records an error and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int VS = 64;
constexpr int NSLICE = DV / VS;
constexpr int NTHREADS = 448;
constexpr int EPI_THREADS = 128;
constexpr int PREP_THREADS = 256;
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr float kMinGamma = 1.8e-35f;  // ~exp(-80)
constexpr int LDA = 68;                // fp32 row stride of the A / T scratch

// TMEM columns (fp32 accumulators, 128 lanes each)
constexpr uint32_t TM_AP0 = 0, TM_AP1 = 64, TM_XY = 128, TM_UO = 192, TM_D = 256, TM_COLS = 512;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_A0 = 0;          // 2 x 32 KB: raw k|q (TMA, 128B swizzle) -> [Kr; Qr]
constexpr uint32_t SM_B0 = 65536;      // 2 x 16 KB: Kc (K-major, 64 rows)
constexpr uint32_t SM_AL = 98304;      // 2 x 32 KB: alpha (fp32 [64][128]); then scratch
constexpr uint32_t SM_V = 163840;      // 2 x 8 KB: v slice (128B swizzle)
constexpr uint32_t SM_TP = 180224;     // 16 KB: [T; P] (K-major, 128 rows x 64)
constexpr uint32_t SM_ST = 196608;     // 16 KB: St (MN-major, 128 rows x 64)
constexpr uint32_t SM_RU = 212992;     // 8 KB: R then U (MN-major, 64 rows x 64)
constexpr uint32_t SM_MU = 221184;     // float[2][128]
constexpr uint32_t SM_BETA = 222208;   // float[2][64]
constexpr uint32_t SM_INFO = 222720;   // int[2][2]: valid rows, slow flag
constexpr uint32_t SM_FLAGS = 222736;  // int[4]: prep slow vote, abort
constexpr uint32_t SM_TMEM = 222752;   // uint32 TMEM base
constexpr uint32_t SM_BAR = 222784;    // mbarriers
constexpr uint32_t SM_RED = 223104;    // float[4][64] + float[64]: slow-path reductions
constexpr uint32_t SM_MSCR = 224384;   // float[3][16*16]: mma.sync staging
constexpr uint32_t SM_TOTAL = 227456;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;

enum Bar {
    B_QK_FULL = 0, B_QK_EMPTY = 2, B_AL_FULL = 4, B_AL_EMPTY = 6, B_V_FULL = 8, B_V_EMPTY = 10,
    B_TAB_FULL = 12, B_AP_FULL = 14, B_B0_EMPTY = 16, B_TP_FULL = 18, B_TP_EMPTY = 19,
    B_S_FULL = 20, B_XY_FULL = 21, B_R_FULL = 22, B_U_FULL = 23, B_UU_FULL = 24, B_D_FULL = 25,
    B_DRAIN = 26, B_COUNT = 27
};

struct TcParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *alpha, *beta, *s0;
    __nv_bfloat16 *o;
    float *sT;
    const int32_t *cu_seqlens;
    const int32_t *order;
    const int32_t *dev_status;
    int32_t *err;
    int N, T, H;
};

__device__ int g_tc_error = 0;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Offset of 16-byte chunk cc (elements 8cc..8cc+7) of row `row` in a
// 128B-swizzled tile whose rows are 128 bytes (MN-major operands, v tiles).
__device__ __forceinline__ uint32_t row128_chunk(uint32_t row, uint32_t cc) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((cc ^ (row & 7u)) << 4);
}

struct Smem {
    unsigned char *base;
    __device__ __forceinline__ uint64_t *bar(int i) const {
        return reinterpret_cast<uint64_t *>(base + SM_BAR) + i;
    }
    __device__ __forceinline__ volatile int *flags() const {
        return reinterpret_cast<volatile int *>(base + SM_FLAGS);
    }
    __device__ __forceinline__ int *info(int b) const { return reinterpret_cast<int *>(base + SM_INFO) + 2 * b; }
    __device__ __forceinline__ float *mu(int b) const { return reinterpret_cast<float *>(base + SM_MU) + 128 * b; }
    __device__ __forceinline__ float *beta(int b) const { return reinterpret_cast<float *>(base + SM_BETA) + 64 * b; }
};

__device__ __forceinline__ void report(const Smem &s, const TcParams &p, int code) {
    s.flags()[1] = 1;  // abort
    atomicOr(p.err ? p.err : &g_tc_error, code);
}
// Wait with the CTA-wide abort check; returns false when the CTA must stop.
__device__ __forceinline__ bool wait_bar(const Smem &s, const TcParams &p, int i, uint32_t parity) {
    if (s.flags()[1]) return false;
    if (mbar_wait(s.bar(i), parity)) return true;
    report(s, p, 2);
    return false;
}

// --------------------------------------------------------------------------
__global__ void __launch_bounds__(NTHREADS, 1)
kda_prefill_tc_kernel(TcParams p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ unsigned char smem_raw[];
    Smem s{reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))};
    if (p.dev_status && *p.dev_status != 0) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x % NSLICE;
    const int h = (blockIdx.x / NSLICE) % p.H;
    const int item = blockIdx.x / (NSLICE * p.H);
    const int seq = p.order ? p.order[item] : item;
    int64_t t_begin, T;
    if (p.cu_seqlens) {
        t_begin = p.cu_seqlens[seq];
        T = (int64_t)p.cu_seqlens[seq + 1] - t_begin;
    } else {
        t_begin = (int64_t)seq * p.T;
        T = p.T;
    }
    const int H = p.H;
    const int v0 = slice * VS;
    const int64_t state_off = ((int64_t)seq * H + h) * DK * DV;
    const int NC = (int)((T + C - 1) / C);

    if (NC == 0) {  // empty sequence: the final state is the initial one
        if (p.sT)
            for (int e = tid; e < DK * VS; e += NTHREADS) {
                const int c = e / VS, j = e % VS;
                p.sT[state_off + (int64_t)c * DV + v0 + j] = p.s0 ? p.s0[state_off + (int64_t)c * DV + v0 + j] : 0.f;
            }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(s.bar(B_QK_FULL + i), 1);
            mbar_init(s.bar(B_QK_EMPTY + i), 1);
            mbar_init(s.bar(B_AL_FULL + i), 1);
            mbar_init(s.bar(B_AL_EMPTY + i), 1);
            mbar_init(s.bar(B_V_FULL + i), 1);
            mbar_init(s.bar(B_V_EMPTY + i), EPI_THREADS);
            mbar_init(s.bar(B_TAB_FULL + i), PREP_THREADS);
            mbar_init(s.bar(B_AP_FULL + i), 1);
            mbar_init(s.bar(B_B0_EMPTY + i), 1);
        }
        mbar_init(s.bar(B_TP_FULL), PREP_THREADS);
        mbar_init(s.bar(B_TP_EMPTY), 1);
        mbar_init(s.bar(B_S_FULL), EPI_THREADS);
        mbar_init(s.bar(B_XY_FULL), 1);
        mbar_init(s.bar(B_R_FULL), EPI_THREADS);
        mbar_init(s.bar(B_U_FULL), 1);
        mbar_init(s.bar(B_UU_FULL), EPI_THREADS);
        mbar_init(s.bar(B_D_FULL), 1);
        mbar_init(s.bar(B_DRAIN), 1);
        s.flags()[0] = 0;
        s.flags()[1] = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(reinterpret_cast<uint32_t *>(s.base + SM_TMEM), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s.base + SM_TMEM);

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int n = 0; n < NC; ++n) {
                const int b = n & 1, kk = n >> 1;
                const int z = (int)(t_begin + (int64_t)n * C);
                if (n >= 2 && !wait_bar(s, p, B_QK_EMPTY + b, (kk - 1) & 1)) break;
                unsigned char *a0 = s.base + SM_A0 + b * 32768;
                mbar_arrive_expect_tx(s.bar(B_QK_FULL + b), 32768);
                tma_load_3d(a0 + 0, &tm_k, s.bar(B_QK_FULL + b), 0, h, z);
                tma_load_3d(a0 + 8192, &tm_q, s.bar(B_QK_FULL + b), 0, h, z);
                tma_load_3d(a0 + 16384, &tm_k, s.bar(B_QK_FULL + b), 64, h, z);
                tma_load_3d(a0 + 24576, &tm_q, s.bar(B_QK_FULL + b), 64, h, z);
                if (n >= 2 && !wait_bar(s, p, B_AL_EMPTY + b, (kk - 1) & 1)) break;
                mbar_arrive_expect_tx(s.bar(B_AL_FULL + b), 32768);
                tma_load_3d(s.base + SM_AL + b * 32768, &tm_a, s.bar(B_AL_FULL + b), 0, h, z);
                if (n >= 2 && !wait_bar(s, p, B_V_EMPTY + b, (kk - 1) & 1)) break;
                mbar_arrive_expect_tx(s.bar(B_V_FULL + b), 8192);
                tma_load_3d(s.base + SM_V + b * 8192, &tm_v, s.bar(B_V_FULL + b), v0, h, z);
                issued = n + 1;
            }
            // never leave copies in flight: wait (bounded) for the last ones
            for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n) {
                const int b = n & 1, kk = n >> 1;
                mbar_wait(s.bar(B_QK_FULL + b), kk & 1);
                mbar_wait(s.bar(B_AL_FULL + b), kk & 1);
                mbar_wait(s.bar(B_V_FULL + b), kk & 1);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t I_AP = idesc_bf16(128, 64, false, false);
            constexpr uint32_t I_KM_MN = idesc_bf16(128, 64, false, true);
            constexpr uint32_t I_MN_MN = idesc_bf16(128, 64, true, true);
            const uint32_t a0_base = smem_u32(s.base + SM_A0), b0_base = smem_u32(s.base + SM_B0);
            const uint32_t tp = smem_u32(s.base + SM_TP), st = smem_u32(s.base + SM_ST),
                           ru = smem_u32(s.base + SM_RU);
            auto mma0 = [&](int n) {
                const int b = n & 1;
                const uint32_t a0 = a0_base + b * 32768, b0 = b0_base + b * 16384;
                const uint32_t d = tmem + (b ? TM_AP1 : TM_AP0);
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(d, sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                              sdesc_sw128(b0 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), I_AP, ks > 0);
            };
            bool ok = wait_bar(s, p, B_TAB_FULL, 0);
            if (ok) {
                tc_fence_after();
                if (!s.info(0)[1]) mma0(0);
                umma_commit(s.bar(B_AP_FULL));
            }
            for (int n = 0; ok && n < NC; ++n) {
                const int b = n & 1;
                const bool fast = !s.info(b)[1];
                // MMA1: [X; Y] = [Kr; Qr] St
                if (!(ok = wait_bar(s, p, B_S_FULL, n & 1))) break;
                tc_fence_after();
                if (fast) {
                    const uint32_t a0 = a0_base + b * 32768;
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(tmem + TM_XY, sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                  sdesc_sw128(st + ks * 2048, 16384, 1024), I_KM_MN, ks > 0);
                }
                umma_commit(s.bar(B_XY_FULL));
                umma_commit(s.bar(B_QK_EMPTY + b));
                // MMA0 of the next chunk while the epilogue forms R
                if (n + 1 < NC) {
                    const int b1 = (n + 1) & 1;
                    if (!(ok = wait_bar(s, p, B_TAB_FULL + b1, ((n + 1) >> 1) & 1))) break;
                    tc_fence_after();
                    if (!s.info(b1)[1]) mma0(n + 1);
                    umma_commit(s.bar(B_AP_FULL + b1));
                }
                // MMA2: U = T R (rows 0-63 of [T; P] R)
                if (!(ok = wait_bar(s, p, B_R_FULL, n & 1))) break;
                if (!(ok = wait_bar(s, p, B_TP_FULL, n & 1))) break;
                tc_fence_after();
                if (fast)
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16(tmem + TM_UO, sdesc_sw128(tp + ks * 32, 16, 1024),
                                  sdesc_sw128(ru + ks * 2048, 8192, 1024), I_KM_MN, ks > 0);
                umma_commit(s.bar(B_U_FULL));
                // MMA3: D += Kc^T U (state update); MMA4: O2 = P U (rows 64-127)
                if (!(ok = wait_bar(s, p, B_UU_FULL, n & 1))) break;
                tc_fence_after();
                if (fast) {
                    const uint32_t b0 = b0_base + b * 16384;
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16(tmem + TM_D, sdesc_sw128(b0 + ks * 2048, 8192, 1024),
                                  sdesc_sw128(ru + ks * 2048, 8192, 1024), I_MN_MN, 1);
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16(tmem + TM_UO, sdesc_sw128(tp + ks * 32, 16, 1024),
                                  sdesc_sw128(ru + ks * 2048, 8192, 1024), I_KM_MN, ks > 0);
                }
                umma_commit(s.bar(B_D_FULL));
                umma_commit(s.bar(B_B0_EMPTY + b));
                umma_commit(s.bar(B_TP_EMPTY));
            }
            // drain: every MMA issued has completed before TMEM is released
            umma_commit(s.bar(B_DRAIN));
            mbar_wait(s.bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        // Group discipline (here and in the prep): a failed wait never leaves
        // the loop; the thread keeps passing the same named barriers with its
        // work switched off, and the next waits return at once (abort flag).
        const int l = tid;  // TMEM lane: key channel (state) or token row
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float mu_cur = 1.f;
        uint32_t r32[32];
        float sreg[64];
        bool ok = wait_bar(s, p, B_TAB_FULL, 0);
        {
            if (ok) mu_cur = s.mu(0)[l];
            const float *src = (ok && p.s0) ? p.s0 + state_off + (int64_t)l * DV + v0 : nullptr;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                float4 x = src ? *reinterpret_cast<const float4 *>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                sreg[j] = x.x; sreg[j + 1] = x.y; sreg[j + 2] = x.z; sreg[j + 3] = x.w;
            }
        }
        // St = Diag(m) S -> TMEM (fp32 accumulator base) and the bf16 MN-major operand
        auto write_st = [&](float m) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r32[j] = __float_as_uint(m * sreg[32 * hf + j]);
                tmem_st32(tmem + lane_off + TM_D + 32 * hf, r32);
            }
            unsigned char *st = s.base + SM_ST;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint4 w;
                w.x = pack_bf16(m * sreg[8 * cc + 0], m * sreg[8 * cc + 1]);
                w.y = pack_bf16(m * sreg[8 * cc + 2], m * sreg[8 * cc + 3]);
                w.z = pack_bf16(m * sreg[8 * cc + 4], m * sreg[8 * cc + 5]);
                w.w = pack_bf16(m * sreg[8 * cc + 6], m * sreg[8 * cc + 7]);
                *reinterpret_cast<uint4 *>(st + row128_chunk(l, cc)) = w;
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(s.bar(B_S_FULL));
        };
        write_st(mu_cur);

        for (int n = 0; n < NC; ++n) {
            const int b = n & 1, kk = n >> 1;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            const int64_t tok0 = t_begin + (int64_t)n * C;
            // E1: R = beta (V - X) for token rows 0-63
            ok = wait_bar(s, p, B_XY_FULL, n & 1) && ok;
            ok = wait_bar(s, p, B_V_FULL + b, kk & 1) && ok;
            tc_fence_after();
            // TMEM loads are warp-collective: every condition around them is warp-uniform
            const bool act = __all_sync(0xffffffffu, ok && s.info(b)[1] == 0);
            if (act && l < 64) {
                const float bt = s.beta(b)[l];
                const unsigned char *vt = s.base + SM_V + b * 8192;
                unsigned char *ru = s.base + SM_RU;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_XY + 32 * hf, r32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int cc = 4 * hf + c4;
                        const uint4 vv = *reinterpret_cast<const uint4 *>(vt + row128_chunk(l, cc));
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                        uint32_t ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 vf = unpack_bf16(vw[e]);
                            const float x0 = __uint_as_float(r32[8 * c4 + 2 * e]);
                            const float x1 = __uint_as_float(r32[8 * c4 + 2 * e + 1]);
                            ow[e] = pack_bf16(bt * (vf.x - x0), bt * (vf.y - x1));
                        }
                        *reinterpret_cast<uint4 *>(ru + row128_chunk(l, cc)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
                fence_proxy_async();
            }
            tc_fence_before();
            mbar_arrive(s.bar(B_R_FULL));
            mbar_arrive(s.bar(B_V_EMPTY + b));
            // E2: U -> bf16 operand (replaces R, which MMA2 has consumed)
            ok = wait_bar(s, p, B_U_FULL, n & 1) && ok;
            tc_fence_after();
            if (__all_sync(0xffffffffu, act && ok) && l < 64) {
                unsigned char *ru = s.base + SM_RU;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_UO + 32 * hf, r32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(r32[8 * c4 + 0]), __uint_as_float(r32[8 * c4 + 1]));
                        w.y = pack_bf16(__uint_as_float(r32[8 * c4 + 2]), __uint_as_float(r32[8 * c4 + 3]));
                        w.z = pack_bf16(__uint_as_float(r32[8 * c4 + 4]), __uint_as_float(r32[8 * c4 + 5]));
                        w.w = pack_bf16(__uint_as_float(r32[8 * c4 + 6]), __uint_as_float(r32[8 * c4 + 7]));
                        *reinterpret_cast<uint4 *>(ru + row128_chunk(l, 4 * hf + c4)) = w;
                    }
                }
                fence_proxy_async();
            }
            tc_fence_before();
            mbar_arrive(s.bar(B_UU_FULL));
            // E3: outputs and the state
            ok = wait_bar(s, p, B_D_FULL, n & 1) && ok;
            tc_fence_after();
            named_bar(2, EPI_THREADS);  // makes the slow-path decision group-uniform
            const bool go = s.flags()[1] == 0;
            const bool slow_g = go && s.info(b)[1] != 0;
            if (go && !slow_g) {
                if (l >= 64) {  // warps 2, 3: token rows of O
                    const int r = l - 64;
                    __nv_bfloat16 *dst = p.o + ((tok0 + r) * H + h) * DV + v0;
                    uint32_t y32[32];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        tmem_ld32(tmem + lane_off + TM_XY + 32 * hf, y32);
                        tmem_ld32(tmem + lane_off + TM_UO + 32 * hf, r32);
                        tmem_wait_ld();
                        if (r < L)
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = 8 * c4 + 2 * e;
                                w[e] = pack_bf16(__uint_as_float(y32[j]) + __uint_as_float(r32[j]),
                                                 __uint_as_float(y32[j + 1]) + __uint_as_float(r32[j + 1]));
                            }
                            *reinterpret_cast<uint4 *>(dst + 32 * hf + 8 * c4) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_D + 32 * hf, r32);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) sreg[32 * hf + j] = mu_cur * __uint_as_float(r32[j]);
                }
            } else if (slow_g) {
                // exact token-by-token update of this chunk (K3 essay §四), fp32;
                // mu = 1 for a slow chunk, so TMEM holds S itself
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_D + 32 * hf, r32);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) sreg[32 * hf + j] = __uint_as_float(r32[j]);
                }
                float *red = reinterpret_cast<float *>(s.base + SM_RED);
                for (int r = 0; r < L; ++r) {
                    const int64_t tk = (tok0 + r) * H + h;
                    const float a = p.alpha[tk * DK + l];
                    const float kf = __bfloat162float(p.k[tk * DK + l]);
                    const float qf = __bfloat162float(p.q[tk * DK + l]);
                    float part[64];
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        sreg[j] *= a;
                        part[j] = kf * sreg[j];
                    }
                    // butterfly reduce-scatter over the warp (64 -> 2 values per
                    // lane): lane ends with the sums of columns 2*lane, 2*lane+1
#pragma unroll
                    for (int nv = 64; nv >= 4; nv >>= 1) {
                        const int half = nv / 2, off = nv / 4;
                        const bool up = (lane & off) != 0;
#pragma unroll
                        for (int j = 0; j < half; ++j) {
                            const float send = up ? part[j] : part[j + half];
                            const float keep = up ? part[j + half] : part[j];
                            part[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                        }
                    }
                    red[warp * 64 + 2 * lane] = part[0];
                    red[warp * 64 + 2 * lane + 1] = part[1];
                    named_bar(2, EPI_THREADS);
                    if (l < 64) {
                        const float vh = red[l] + red[64 + l] + red[128 + l] + red[192 + l];
                        const float vv = __bfloat162float(p.v[tk * DV + v0 + l]);
                        red[256 + l] = p.beta[tk] * (vv - vh);
                    }
                    named_bar(2, EPI_THREADS);
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        sreg[j] += kf * red[256 + j];
                        part[j] = qf * sreg[j];
                    }
                    named_bar(2, EPI_THREADS);  // the error vector is read by all
#pragma unroll
                    for (int nv = 64; nv >= 4; nv >>= 1) {
                        const int half = nv / 2, off = nv / 4;
                        const bool up = (lane & off) != 0;
#pragma unroll
                        for (int j = 0; j < half; ++j) {
                            const float send = up ? part[j] : part[j + half];
                            const float keep = up ? part[j + half] : part[j];
                            part[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                        }
                    }
                    red[warp * 64 + 2 * lane] = part[0];
                    red[warp * 64 + 2 * lane + 1] = part[1];
                    named_bar(2, EPI_THREADS);
                    if (l < 64)
                        p.o[tk * DV + v0 + l] =
                            __float2bfloat16_rn(red[l] + red[64 + l] + red[128 + l] + red[192 + l]);
                    named_bar(2, EPI_THREADS);
                }
            }
            if (n == NC - 1) {
                if (go && p.sT) {
                    float *dst = p.sT + state_off + (int64_t)l * DV + v0;
#pragma unroll
                    for (int j = 0; j < 64; j += 4)
                        *reinterpret_cast<float4 *>(dst + j) = make_float4(sreg[j], sreg[j + 1], sreg[j + 2], sreg[j + 3]);
                }
            } else {
                ok = wait_bar(s, p, B_TAB_FULL + ((n + 1) & 1), ((n + 1) >> 1) & 1) && ok;
                if (ok) mu_cur = s.mu((n + 1) & 1)[l];
                write_st(mu_cur);
            }
        }
    } else {
        // ------------------------------------------------------------ prep (warps 4-11)
        const int pt = tid - 128;
        const int pw = warp - 4;  // 0..7
        const int co = pt & 15, tg = pt >> 4;

        auto prep_a = [&](int n) {
            const int b = n & 1, kk = n >> 1;
            const int64_t tok0 = t_begin + (int64_t)n * C;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            bool ok = wait_bar(s, p, B_QK_FULL + b, kk & 1);
            ok = wait_bar(s, p, B_AL_FULL + b, kk & 1) && ok;
            if (n >= 2) ok = wait_bar(s, p, B_B0_EMPTY + b, (kk - 1) & 1) && ok;
            if (pt == 0) s.flags()[0] = 0;
            float *al = reinterpret_cast<float *>(s.base + SM_AL + b * 32768);
            float a[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * tg + i;
                float4 x0 = make_float4(1.f, 1.f, 1.f, 1.f), x1 = x0;
                if (ok && r < L) {
                    x0 = *reinterpret_cast<const float4 *>(al + r * 128 + 8 * co);
                    x1 = *reinterpret_cast<const float4 *>(al + r * 128 + 8 * co + 4);
                }
                a[i][0] = x0.x; a[i][1] = x0.y; a[i][2] = x0.z; a[i][3] = x0.w;
                a[i][4] = x1.x; a[i][5] = x1.y; a[i][6] = x1.z; a[i][7] = x1.w;
            }
            float g[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) g[c] = a[0][c] * a[1][c] * a[2][c] * a[3][c];
            named_bar(1, PREP_THREADS);  // alpha read; its buffer becomes scan scratch
            *reinterpret_cast<float4 *>(al + tg * 128 + 8 * co) = make_float4(g[0], g[1], g[2], g[3]);
            *reinterpret_cast<float4 *>(al + tg * 128 + 8 * co + 4) = make_float4(g[4], g[5], g[6], g[7]);
            named_bar(1, PREP_THREADS);
            float before[8], after[8], gam[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) before[c] = after[c] = 1.f;
            for (int gi = 0; gi < 16; ++gi) {
                const float4 x0 = *reinterpret_cast<const float4 *>(al + gi * 128 + 8 * co);
                const float4 x1 = *reinterpret_cast<const float4 *>(al + gi * 128 + 8 * co + 4);
                const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (gi < tg) before[c] *= xs[c];
                    if (gi > tg) after[c] *= xs[c];
                }
            }
            bool bad = false;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                gam[c] = before[c] * g[c] * after[c];
                bad |= !(gam[c] >= kMinGamma);
            }
            if (bad) s.flags()[0] = 1;
            named_bar(1, PREP_THREADS);
            const bool slow = s.flags()[0] != 0;
            if (tg == 0)
#pragma unroll
                for (int c = 0; c < 8; ++c) s.mu(b)[8 * co + c] = slow ? 1.f : sqrtf(gam[c]);
            if (ok && !slow) {
                float inv[8], sfx[4][8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    inv[c] = 1.f / sqrtf(gam[c]);
                    sfx[3][c] = after[c];
                    sfx[2][c] = after[c] * a[3][c];
                    sfx[1][c] = sfx[2][c] * a[2][c];
                    sfx[0][c] = sfx[1][c] * a[1][c];
                }
                unsigned char *a0 = s.base + SM_A0 + b * 32768;
                unsigned char *b0 = s.base + SM_B0 + b * 16384;
                float pre[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) pre[c] = before[c];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * tg + i;
                    const uint32_t offk = kmajor_chunk(r, co, 128), offq = kmajor_chunk(64 + r, co, 128);
                    const uint4 kw = *reinterpret_cast<const uint4 *>(a0 + offk);
                    const uint4 qw = *reinterpret_cast<const uint4 *>(a0 + offq);
                    const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, qa[4] = {qw.x, qw.y, qw.z, qw.w};
                    uint32_t kr[4], qr[4], kc[4];
                    const bool v = r < L;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c0 = 2 * e, c1 = 2 * e + 1;
                        pre[c0] *= a[i][c0];
                        pre[c1] *= a[i][c1];
                        const float e2a = pre[c0] * inv[c0], e2b = pre[c1] * inv[c1];
                        const float e3a = sfx[i][c0] * inv[c0], e3b = sfx[i][c1] * inv[c1];
                        const float2 kf = unpack_bf16(ka[e]), qf = unpack_bf16(qa[e]);
                        kr[e] = v ? pack_bf16(kf.x * e2a, kf.y * e2b) : 0u;
                        qr[e] = v ? pack_bf16(qf.x * e2a, qf.y * e2b) : 0u;
                        kc[e] = v ? pack_bf16(kf.x * e3a, kf.y * e3b) : 0u;
                    }
                    *reinterpret_cast<uint4 *>(a0 + offk) = make_uint4(kr[0], kr[1], kr[2], kr[3]);
                    *reinterpret_cast<uint4 *>(a0 + offq) = make_uint4(qr[0], qr[1], qr[2], qr[3]);
                    *reinterpret_cast<uint4 *>(b0 + kmajor_chunk(r, co, 64)) = make_uint4(kc[0], kc[1], kc[2], kc[3]);
                }
            }
            if (pt < 64) s.beta(b)[pt] = pt < L ? p.beta[(tok0 + pt) * H + h] : 0.f;
            if (pt == 0) {
                s.info(b)[0] = L;
                s.info(b)[1] = slow ? 1 : 0;
            }
            fence_proxy_async();
            mbar_arrive(s.bar(B_TAB_FULL + b));
        };

        auto prep_b = [&](int n) {
            const int b = n & 1, kk = n >> 1;
            bool ok = wait_bar(s, p, B_AP_FULL + b, kk & 1);
            tc_fence_after();
            named_bar(1, PREP_THREADS);
            const bool go = s.flags()[1] == 0;
            const bool slow = s.info(b)[1] != 0;
            const bool work = go && !slow;  // group-uniform
            const int L = s.info(b)[0];
            float *asc = reinterpret_cast<float *>(s.base + SM_AL + b * 32768);        // A, stride LDA
            float *tsc = reinterpret_cast<float *>(s.base + SM_AL + (b ^ 1) * 32768);  // T, stride LDA
            uint32_t pbuf[16];
            const int q4 = warp & 3, half = pw >> 2;
            const int R = 32 * q4 + lane;  // TMEM lane = row of [A; P]
            if (work) {
                uint32_t r32[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + (b ? TM_AP1 : TM_AP0) + 32 * half, r32);
                tmem_wait_ld();
                if (R < 64) {
                    const float bt = s.beta(b)[R];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 32 * half + 4 * j4 + e;
                            w[e] = j < R ? bt * __uint_as_float(r32[4 * j4 + e]) : 0.f;
                        }
                        *reinterpret_cast<float4 *>(asc + R * LDA + 32 * half + 4 * j4) = make_float4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    const int r = R - 64;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = 32 * half + 2 * e;
                        const float x0 = (j <= r && r < L) ? __uint_as_float(r32[2 * e]) : 0.f;
                        const float x1 = (j + 1 <= r && r < L) ? __uint_as_float(r32[2 * e + 1]) : 0.f;
                        pbuf[e] = pack_bf16(x0, x1);
                    }
                }
                tc_fence_before();
            }
            named_bar(1, PREP_THREADS);
            if (work) {
                // T step 1: the four 16x16 diagonal blocks, column by column
                // (x_r -= A[r][s] x_s for s < r), 4 threads per column.
                const int blk = pt >> 6, col = (pt >> 2) & 15, part = pt & 3;
                const float *ab = asc + (16 * blk) * LDA + 16 * blk;
                float xr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) xr[i] = (part + 4 * i == col) ? 1.f : 0.f;
#pragma unroll
                for (int sidx = 0; sidx < 15; ++sidx) {
                    const float xs = __shfl_sync(0xffffffffu, xr[sidx >> 2], (lane & ~3) | (sidx & 3));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rl = part + 4 * i;
                        if (rl > sidx) xr[i] -= ab[rl * LDA + sidx] * xs;
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) tsc[(16 * blk + part + 4 * i) * LDA + 16 * blk + col] = xr[i];
            }
            named_bar(1, PREP_THREADS);
            // T step 2: off-diagonal blocks by distance, on mma.sync (tf32):
            // T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ
            const int g8 = lane >> 2, t4 = lane & 3;
            for (int d = 1; d <= 3; ++d) {
                if (work && pw < 4 - d) {
                    const int J = pw, I = pw + d;
                    float m[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) m[nt][e] = 0.f;
                    for (int K = J; K < I; ++K) {
#pragma unroll
                        for (int k8 = 0; k8 < 16; k8 += 8) {
                            const float *ar = asc + (16 * I) * LDA + 16 * K + k8;
                            const uint32_t af[4] = {to_tf32(ar[g8 * LDA + t4]), to_tf32(ar[(g8 + 8) * LDA + t4]),
                                                    to_tf32(ar[g8 * LDA + t4 + 4]), to_tf32(ar[(g8 + 8) * LDA + t4 + 4])};
                            const float *br = tsc + (16 * K + k8) * LDA + 16 * J;
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt)
                                mma_tf32(m[nt], af, to_tf32(br[t4 * LDA + 8 * nt + g8]),
                                         to_tf32(br[(t4 + 4) * LDA + 8 * nt + g8]));
                        }
                    }
                    float *ms = reinterpret_cast<float *>(s.base + SM_MSCR) + pw * 256;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        ms[g8 * 16 + 8 * nt + 2 * t4] = m[nt][0];
                        ms[g8 * 16 + 8 * nt + 2 * t4 + 1] = m[nt][1];
                        ms[(g8 + 8) * 16 + 8 * nt + 2 * t4] = m[nt][2];
                        ms[(g8 + 8) * 16 + 8 * nt + 2 * t4 + 1] = m[nt][3];
                    }
                    __syncwarp();
                    float t[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) t[nt][e] = 0.f;
#pragma unroll
                    for (int k8 = 0; k8 < 16; k8 += 8) {
                        const float *ar = tsc + (16 * I) * LDA + 16 * I + k8;
                        const uint32_t af[4] = {to_tf32(ar[g8 * LDA + t4]), to_tf32(ar[(g8 + 8) * LDA + t4]),
                                                to_tf32(ar[g8 * LDA + t4 + 4]), to_tf32(ar[(g8 + 8) * LDA + t4 + 4])};
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
                            mma_tf32(t[nt], af, to_tf32(ms[(k8 + t4) * 16 + 8 * nt + g8]),
                                     to_tf32(ms[(k8 + t4 + 4) * 16 + 8 * nt + g8]));
                    }
                    float *tb = tsc + (16 * I) * LDA + 16 * J;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        tb[g8 * LDA + 8 * nt + 2 * t4] = -t[nt][0];
                        tb[g8 * LDA + 8 * nt + 2 * t4 + 1] = -t[nt][1];
                        tb[(g8 + 8) * LDA + 8 * nt + 2 * t4] = -t[nt][2];
                        tb[(g8 + 8) * LDA + 8 * nt + 2 * t4 + 1] = -t[nt][3];
                    }
                    __syncwarp();
                }
                named_bar(1, PREP_THREADS);
            }
            // [T; P] -> the bf16 operand tile, once MMA4 of the previous chunk is done
            if (n >= 1) ok = wait_bar(s, p, B_TP_EMPTY, (n - 1) & 1) && ok;
            if (ok && work) {
                unsigned char *tpt = s.base + SM_TP;
                {
                    const int r = pt >> 2, cq = pt & 3;  // T row r, columns 16cq .. 16cq+15
                    const float *tr = tsc + r * LDA + 16 * cq;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 16 * cq + 8 * hh + 2 * e;
                            const float x0 = j < r ? tr[8 * hh + 2 * e] : (j == r ? 1.f : 0.f);
                            const float x1 = j + 1 < r ? tr[8 * hh + 2 * e + 1] : (j + 1 == r ? 1.f : 0.f);
                            w[e] = pack_bf16(x0, x1);
                        }
                        *reinterpret_cast<uint4 *>(tpt + kmajor_chunk(r, 2 * cq + hh, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                if (R >= 64) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(tpt + kmajor_chunk(R, 4 * half + c4, 128)) =
                            make_uint4(pbuf[4 * c4], pbuf[4 * c4 + 1], pbuf[4 * c4 + 2], pbuf[4 * c4 + 3]);
                }
                fence_proxy_async();
            }
            mbar_arrive(s.bar(B_TP_FULL));
            named_bar(1, PREP_THREADS);  // scratch reads done before the alpha buffer is refilled
            if (pt == 0) mbar_arrive(s.bar(B_AL_EMPTY + b));
        };

        prep_a(0);
        for (int n = 0; n < NC; ++n) {
            if (n + 1 < NC) prep_a(n + 1);
            prep_b(n);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

bool make_map(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *ptr, int inner, int H,
              int64_t tokens, int box_inner, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)inner * esize * H};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) {
    return a.dt == KDA_BF16 && a.dk == DK && a.dv == DV;
}

cudaError_t read_device_error(int *out, bool reset) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *out = v;
    if (reset && v) {
        const int z = 0;
        e = cudaMemcpyToSymbol(g_tc_error, &z, sizeof(int));
    }
    return e;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    if (!prefill_tc_supported(a)) return cudaErrorInvalidValue;
    const int64_t tokens = a.cu_seqlens ? (int64_t)a.T : (int64_t)a.N * a.T;
    const int64_t blocks = (int64_t)a.N * a.H * NSLICE;
    if (blocks == 0) return cudaSuccess;
    CUtensorMap mk, mq, ma, mv;
    // A map needs a non-empty extent; an empty token range never issues a copy.
    const int64_t ext = tokens > 0 ? tokens : 1;
    if (!make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, DK, a.H, ext, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, DK, a.H, ext, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.alpha, DK, a.H, ext, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, DV, a.H, ext, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    TcParams p;
    p.q = (const __nv_bfloat16 *)a.q;
    p.k = (const __nv_bfloat16 *)a.k;
    p.v = (const __nv_bfloat16 *)a.v;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.s0 = a.s0;
    p.o = (__nv_bfloat16 *)a.o;
    p.sT = a.sT;
    p.cu_seqlens = a.cu_seqlens;
    p.order = a.order;
    p.dev_status = a.dev_status;
    p.err = nullptr;
    p.N = a.N;
    p.T = a.T;
    p.H = a.H;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_prefill_tc_kernel<<<(unsigned)blocks, NTHREADS, SMEM_BYTES, stream>>>(p, mk, mq, ma, mv);
    return cudaGetLastError();
}

}  // namespace kda
