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
// One CTA per (sequence, head, 64-wide slice of d_v); 512 threads, four
// warpgroups with their own register budgets (setmaxnreg):
//   warps 0-3   epilogue: the state chain (R, U, O, S) - one TMEM lane each  144 regs
//   warps 4-7   gate: gate products, mu, the gated tables Kr, Qr, Kc        160 regs
//   warps 8-11  solve: A/P read-out, T = (I + A)^-1, the [T; P] tile        128 regs
//   warp 12     TMA producer (q, k, v tiles 2-deep; alpha 1-deep, freed early)
//   warp 13     MMA issuer of the state chain (one thread), TMEM owner
//   warp 14     MMA issuer of the intra-chunk [A; P] products (one thread);
//               tcgen05 commits track the issuing thread, so the two issuers
//               never wait for each other; warp 15 idle                      80 regs
// The three groups work on consecutive chunks at once: tables of chunk n+2,
// inverse of chunk n+1, state chain of chunk n. All waits are bounded; on a
// timeout the CTA records an error and winds down.
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
constexpr int NTHREADS = 512;
// Register shares per warpgroup. Each SM sub-partition holds one warp of
// every warpgroup, so the shares sum to 4 x 128 = the launch's allocation
// (a larger sum would make setmaxnreg.inc wait forever).
constexpr uint32_t REGS_EPI = 144, REGS_GATE = 160, REGS_SOLVE = 128, REGS_CTRL = 80;
static_assert(REGS_EPI + REGS_GATE + REGS_SOLVE + REGS_CTRL == 4 * 128, "register split");
constexpr int EPI_THREADS = 128;
constexpr int GATE_THREADS = 128;
constexpr int SOLVE_THREADS = 128;
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr int WARP_MMA0 = 14;
constexpr float kMinGamma = 1.8e-35f;  // ~exp(-80)

// TMEM columns (fp32 accumulators, 128 lanes each)
constexpr uint32_t TM_AP0 = 0, TM_AP1 = 64, TM_XY = 128, TM_UO = 192, TM_D = 256, TM_COLS = 512;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_A0 = 0;          // 2 x 32 KB: raw k|q (TMA, 128B swizzle) -> [Kr; Qr]
constexpr uint32_t SM_B0 = 65536;      // 2 x 16 KB: Kc (K-major, 64 rows)
constexpr uint32_t SM_AL = 98304;      // 32 KB: alpha (fp32 [64][128])
constexpr uint32_t SM_SOLVE = 131072;  // 32 KB: A and T (fp32 64x64 each, XOR-swizzled)
constexpr uint32_t SM_V = 163840;      // 2 x 8 KB: v slice (128B swizzle)
constexpr uint32_t SM_TP = 180224;     // 16 KB: [T; P] (K-major, 128 rows x 64)
constexpr uint32_t SM_ST = 196608;     // 16 KB: St (MN-major, 128 rows x 64)
constexpr uint32_t SM_RU = 212992;     // 8 KB: R then U (MN-major, 64 rows x 64)
constexpr uint32_t SM_MU = 221184;     // float[2][128]
constexpr uint32_t SM_BETA = 222208;   // float[2][64]
constexpr uint32_t SM_INFO = 222720;   // int[2][2]: valid rows, slow flag
constexpr uint32_t SM_FLAGS = 222736;  // int[8]: [1] abort, [4 + b] slow vote of chunk parity b
constexpr uint32_t SM_TMEM = 222768;   // uint32 TMEM base
constexpr uint32_t SM_BAR = 222784;    // mbarriers
constexpr uint32_t SM_RED = 223104;    // float[4][64] + float[64]: slow-path reductions
constexpr uint32_t SM_MSCR = 224384;   // float[3][16*16]: mma.sync staging
constexpr uint32_t SM_SCAN = 227456;   // float[4][128]: per-group gate products
constexpr uint32_t SM_TOTAL = 229504;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;

enum Bar {
    B_QK_FULL = 0, B_QK_EMPTY = 2, B_AL_FULL = 4, B_AL_EMPTY = 6, B_V_FULL = 8, B_V_EMPTY = 10,
    B_TAB_FULL = 12, B_AP_FULL = 14, B_B0_EMPTY = 16, B_TP_FULL = 18, B_TP_EMPTY = 19,
    B_S_FULL = 20, B_XY_FULL = 21, B_R_FULL = 22, B_U_FULL = 23, B_UU_FULL = 24, B_D_FULL = 25,
    B_DRAIN = 26, B_COUNT = 28  // B_DRAIN + 1: drain of the MMA0 issuer
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
// Two fp32 values packed in 64 bits, multiplied pairwise by one instruction.
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f2_hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }
// bf16 pair (low element in the low half) -> fp32 pair, and back (round to nearest even)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t u) {
    return (uint64_t)(u << 16) | ((uint64_t)(u & 0xffff0000u) << 32);
}
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t x) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "r"((uint32_t)(x >> 32)), "r"((uint32_t)x));
    return d;
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
// Index of element (r, c) of a 64x64 fp32 scratch matrix: rows of 64 floats,
// column bits 2-4 XOR-ed with the row's low bits, so that the mma.sync
// fragment loads (8 rows x 4 columns) and row-wise float4 accesses hit 32
// different banks without padding.
__device__ __forceinline__ int swz(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }
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

// Exact token-by-token update of one chunk (the K3 essay's §四 recurrence in
// fp32), used for chunks whose gates decay past the factorised range. The
// epilogue warpgroup holds the state slice in TMEM (lane = key channel,
// 64 value columns); this reads it, runs the chunk's tokens and writes the
// new state back. Rare; inlined (an out-of-line call costs the fast path
// register spills around the call site).
__device__ __forceinline__ void slow_chunk(const float *__restrict__ alpha, const __nv_bfloat16 *__restrict__ kin,
                                        const __nv_bfloat16 *__restrict__ qin, const __nv_bfloat16 *__restrict__ vin,
                                        const float *__restrict__ beta, __nv_bfloat16 *__restrict__ o, float *red,
                                        uint32_t tm_d, int l, int warp, int lane, int64_t tok0, int L, int H, int h,
                                        int v0) {
    float sreg[64];
    uint32_t r32[32];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        tmem_ld32(tm_d + 32 * hf, r32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) sreg[32 * hf + j] = __uint_as_float(r32[j]);
    }
    for (int r = 0; r < L; ++r) {
        const int64_t tk = (tok0 + r) * H + h;
        const float a = alpha[tk * DK + l];
        const float kf = __bfloat162float(kin[tk * DK + l]);
        const float qf = __bfloat162float(qin[tk * DK + l]);
        float part[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            sreg[j] *= a;
            part[j] = kf * sreg[j];
        }
        // butterfly reduce-scatter over the warp (64 -> 2 values per lane):
        // the lane ends with the sums of columns 2*lane and 2*lane+1
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
            const float vv = __bfloat162float(vin[tk * DV + v0 + l]);
            red[256 + l] = beta[tk] * (vv - vh);
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
        if (l < 64) o[tk * DV + v0 + l] = __float2bfloat16_rn(red[l] + red[64 + l] + red[128 + l] + red[192 + l]);
        named_bar(2, EPI_THREADS);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r32[j] = __float_as_uint(sreg[32 * hf + j]);
        tmem_st32(tm_d + 32 * hf, r32);
    }
    tmem_wait_st();
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
            mbar_init(s.bar(B_QK_EMPTY + i), 2);  // both MMA issuers read the q/k tile
            mbar_init(s.bar(B_AL_FULL + i), 1);
            mbar_init(s.bar(B_AL_EMPTY + i), 1);
            mbar_init(s.bar(B_V_FULL + i), 1);
            mbar_init(s.bar(B_V_EMPTY + i), EPI_THREADS);
            mbar_init(s.bar(B_TAB_FULL + i), GATE_THREADS);
            mbar_init(s.bar(B_AP_FULL + i), 1);
            mbar_init(s.bar(B_B0_EMPTY + i), 1);
        }
        mbar_init(s.bar(B_TP_FULL), SOLVE_THREADS);
        mbar_init(s.bar(B_TP_EMPTY), 1);
        mbar_init(s.bar(B_S_FULL), EPI_THREADS);
        mbar_init(s.bar(B_XY_FULL), 1);
        mbar_init(s.bar(B_R_FULL), EPI_THREADS);
        mbar_init(s.bar(B_U_FULL), 1);
        mbar_init(s.bar(B_UU_FULL), EPI_THREADS);
        mbar_init(s.bar(B_D_FULL), 1);
        mbar_init(s.bar(B_DRAIN), 1);
        mbar_init(s.bar(B_DRAIN + 1), 1);
        for (int i = 0; i < 8; ++i) s.flags()[i] = 0;
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

    if (warp >= 12) {
        regs_dec<REGS_CTRL>();
    }
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
                // alpha: one buffer, released by the gate group as soon as it
                // holds the chunk's gates in registers
                if (n >= 1 && !wait_bar(s, p, B_AL_EMPTY, (n - 1) & 1)) break;
                mbar_arrive_expect_tx(s.bar(B_AL_FULL), 32768);
                tma_load_3d(s.base + SM_AL, &tm_a, s.bar(B_AL_FULL), 0, h, z);
                if (n >= 2 && !wait_bar(s, p, B_V_EMPTY + b, (kk - 1) & 1)) break;
                mbar_arrive_expect_tx(s.bar(B_V_FULL + b), 8192);
                tma_load_3d(s.base + SM_V + b * 8192, &tm_v, s.bar(B_V_FULL + b), v0, h, z);
                issued = n + 1;
            }
            // never leave copies in flight: wait (bounded) for the last ones
            for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n) {
                const int b = n & 1, kk = n >> 1;
                mbar_wait(s.bar(B_QK_FULL + b), kk & 1);
                mbar_wait(s.bar(B_V_FULL + b), kk & 1);
            }
            if (issued > 0) mbar_wait(s.bar(B_AL_FULL), (issued - 1) & 1);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t I_KM_MN = idesc_bf16(128, 64, false, true);
            constexpr uint32_t I_MN_MN = idesc_bf16(128, 64, true, true);
            const uint32_t a0_base = smem_u32(s.base + SM_A0), b0_base = smem_u32(s.base + SM_B0);
            const uint32_t tp = smem_u32(s.base + SM_TP), st = smem_u32(s.base + SM_ST),
                           ru = smem_u32(s.base + SM_RU);
            bool ok = true;
            for (int n = 0; ok && n < NC; ++n) {
                const int b = n & 1;
                if (!(ok = wait_bar(s, p, B_TAB_FULL + b, (n >> 1) & 1))) break;
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
                umma_commit(s.bar(B_QK_EMPTY + b));  // with the MMA0 issuer's: 2 arrivals
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
    } else if (warp == WARP_MMA0) {
        // ------------------------------------------------------------ MMA0 issuer
        if (lane == 0) {
            constexpr uint32_t I_AP = idesc_bf16(128, 64, false, false);
            const uint32_t a0_base = smem_u32(s.base + SM_A0), b0_base = smem_u32(s.base + SM_B0);
            for (int n = 0; n < NC; ++n) {
                const int b = n & 1;
                if (!wait_bar(s, p, B_TAB_FULL + b, (n >> 1) & 1)) break;
                tc_fence_after();
                if (!s.info(b)[1]) {
                    const uint32_t a0 = a0_base + b * 32768, b0 = b0_base + b * 16384;
                    const uint32_t d = tmem + (b ? TM_AP1 : TM_AP0);
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(d, sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                  sdesc_sw128(b0 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), I_AP, ks > 0);
                }
                umma_commit(s.bar(B_AP_FULL + b));
                umma_commit(s.bar(B_QK_EMPTY + b));
            }
            umma_commit(s.bar(B_DRAIN + 1));
            mbar_wait(s.bar(B_DRAIN + 1), 0);
        }
        __syncwarp();
    } else if (warp >= 12) {
        // idle warps of the control warpgroup
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        regs_inc<REGS_EPI>();
        // Group discipline (here and in the gate / solve groups): a failed
        // wait never leaves the loop; the thread keeps passing the same named
        // barriers with its work switched off, and the next waits return at
        // once (abort flag). TMEM loads and stores are warp-collective, so the
        // conditions around them are warp-uniform.
        const int l = tid;  // TMEM lane: key channel (state) or token row
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tm_d = tmem + lane_off + TM_D;
        uint32_t r32[32];
        bool ok = wait_bar(s, p, B_TAB_FULL, 0);
        float mu_cur = ok ? s.mu(0)[l] : 1.f;
        // St_0 = Diag(mu_0) S0 -> TMEM (fp32 accumulator base) and the bf16 operand
        {
            const float *src = (ok && p.s0) ? p.s0 + state_off + (int64_t)l * DV + v0 : nullptr;
            unsigned char *st = s.base + SM_ST;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 f = src ? *reinterpret_cast<const float4 *>(src + 32 * hf + j)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[j] = mu_cur * f.x; x[j + 1] = mu_cur * f.y; x[j + 2] = mu_cur * f.z; x[j + 3] = mu_cur * f.w;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) r32[j] = __float_as_uint(x[j]);
                tmem_st32(tm_d + 32 * hf, r32);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    *reinterpret_cast<uint4 *>(st + row128_chunk(l, 4 * hf + c4)) =
                        make_uint4(pack_bf16(x[8 * c4], x[8 * c4 + 1]), pack_bf16(x[8 * c4 + 2], x[8 * c4 + 3]),
                                   pack_bf16(x[8 * c4 + 4], x[8 * c4 + 5]), pack_bf16(x[8 * c4 + 6], x[8 * c4 + 7]));
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(s.bar(B_S_FULL));
        }

        for (int n = 0; n < NC; ++n) {
            const int b = n & 1, kk = n >> 1;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            const int64_t tok0 = t_begin + (int64_t)n * C;
            // E1: R = beta (V - X) for token rows 0-63
            ok = wait_bar(s, p, B_XY_FULL, n & 1) && ok;
            ok = wait_bar(s, p, B_V_FULL + b, kk & 1) && ok;
            tc_fence_after();
            const bool act = __all_sync(0xffffffffu, ok && s.info(b)[1] == 0);
            if (act && l < 64) {
                const float bt = s.beta(b)[l];
                const unsigned char *vt = s.base + SM_V + b * 8192;
                unsigned char *ru = s.base + SM_RU;
                uint4 vrow[8];  // the whole v row first: no load waits behind an R store
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) vrow[cc] = *reinterpret_cast<const uint4 *>(vt + row128_chunk(l, cc));
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_XY + 32 * hf, r32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int cc = 4 * hf + c4;
                        const uint4 vv = vrow[cc];
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
            // E3: outputs, then the state S_{n+1} = mu_n D -> St_{n+1} = mu_{n+1} S_{n+1}
            ok = wait_bar(s, p, B_D_FULL, n & 1) && ok;
            tc_fence_after();
            named_bar(2, EPI_THREADS);  // makes the slow-path decision group-uniform
            const bool go = s.flags()[1] == 0;
            const bool slow_g = go && s.info(b)[1] != 0;
            if (!slow_g && l >= 64) {  // warps 2, 3: token rows of O = Y + P U
                const int r = l - 64;
                __nv_bfloat16 *dst = p.o + ((tok0 + r) * H + h) * DV + v0;
                uint32_t y32[32];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tmem_ld32(tmem + lane_off + TM_XY + 32 * hf, y32);
                    tmem_ld32(tmem + lane_off + TM_UO + 32 * hf, r32);
                    tmem_wait_ld();
                    if (go && r < L) {
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
            }
            if (slow_g)  // TMEM holds S_n (mu_n = 1); leaves S_{n+1} there
                slow_chunk(p.alpha, p.k, p.q, p.v, p.beta, p.o, reinterpret_cast<float *>(s.base + SM_RED), tm_d, l,
                           warp, lane, tok0, L, H, h, v0);
            const bool last = n == NC - 1;
            float mu_next = 1.f;
            if (!last) {
                ok = wait_bar(s, p, B_TAB_FULL + ((n + 1) & 1), ((n + 1) >> 1) & 1) && ok;
                if (ok) mu_next = s.mu((n + 1) & 1)[l];
            }
            unsigned char *st = s.base + SM_ST;
            float *fin = p.sT ? p.sT + state_off + (int64_t)l * DV + v0 : nullptr;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                tmem_ld32(tm_d + 32 * hf, r32);
                tmem_wait_ld();
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = mu_cur * __uint_as_float(r32[j]);
                if (last) {
                    if (go && fin)
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(fin + 32 * hf + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        x[j] *= mu_next;
                        r32[j] = __float_as_uint(x[j]);
                    }
                    tmem_st32(tm_d + 32 * hf, r32);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(st + row128_chunk(l, 4 * hf + c4)) =
                            make_uint4(pack_bf16(x[8 * c4], x[8 * c4 + 1]), pack_bf16(x[8 * c4 + 2], x[8 * c4 + 3]),
                                       pack_bf16(x[8 * c4 + 4], x[8 * c4 + 5]), pack_bf16(x[8 * c4 + 6], x[8 * c4 + 7]));
                }
            }
            if (!last) {
                tmem_wait_st();
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(s.bar(B_S_FULL));
            }
            mu_cur = mu_next;
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ gate group (warps 4-7)
        // Thread: value channels 4cq .. 4cq+3, token rows 16tg .. 16tg+15.
        regs_inc<REGS_GATE>();
        const int pt = tid - 128;
        const int cq = pt & 31, tg = pt >> 5;
        float *scan = reinterpret_cast<float *>(s.base + SM_SCAN);
        const float *al = reinterpret_cast<const float *>(s.base + SM_AL);
        for (int n = 0; n < NC; ++n) {
            const int b = n & 1, kk = n >> 1;
            const int64_t tok0 = t_begin + (int64_t)n * C;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            // beta of this chunk, loaded before the waits so its latency is hidden
            const float beta_r = pt < L ? p.beta[(tok0 + pt) * H + h] : 0.f;
            bool ok = wait_bar(s, p, B_QK_FULL + b, kk & 1);
            ok = wait_bar(s, p, B_AL_FULL, n & 1) && ok;
            if (pt == 0) s.flags()[4 + b] = 0;  // vote slot of this parity (last read two chunks ago)
            float4 a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * tg + i;
                a[i] = (ok && r < L) ? *reinterpret_cast<const float4 *>(al + r * 128 + 4 * cq)
                                     : make_float4(1.f, 1.f, 1.f, 1.f);
            }
            named_bar(1, GATE_THREADS);  // every gate is in registers: the buffer may refill
            if (pt == 0) mbar_arrive(s.bar(B_AL_EMPTY));
            float4 g = a[0];
#pragma unroll
            for (int i = 1; i < 16; ++i) {
                g.x *= a[i].x; g.y *= a[i].y; g.z *= a[i].z; g.w *= a[i].w;
            }
            *reinterpret_cast<float4 *>(scan + tg * 128 + 4 * cq) = g;
            named_bar(1, GATE_THREADS);
            float4 before = make_float4(1.f, 1.f, 1.f, 1.f), after = before;
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) {
                const float4 x = *reinterpret_cast<const float4 *>(scan + gi * 128 + 4 * cq);
                if (gi < tg) { before.x *= x.x; before.y *= x.y; before.z *= x.z; before.w *= x.w; }
                if (gi > tg) { after.x *= x.x; after.y *= x.y; after.z *= x.z; after.w *= x.w; }
            }
            const float gam[4] = {before.x * g.x * after.x, before.y * g.y * after.y, before.z * g.z * after.z,
                                  before.w * g.w * after.w};
            bool bad = false;
#pragma unroll
            for (int c = 0; c < 4; ++c) bad |= !(gam[c] >= kMinGamma);
            if (bad) s.flags()[4 + b] = 1;
            named_bar(1, GATE_THREADS);
            const bool slow = s.flags()[4 + b] != 0;
            float inv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) inv[c] = slow ? 1.f : rsqrtf(gam[c]);
            if (tg == 0)
                *reinterpret_cast<float4 *>(s.mu(b) + 4 * cq) =
                    slow ? make_float4(1.f, 1.f, 1.f, 1.f)
                         : make_float4(gam[0] * inv[0], gam[1] * inv[1], gam[2] * inv[2], gam[3] * inv[3]);
            if (ok && !slow) {
                unsigned char *a0 = s.base + SM_A0 + b * 32768;
                unsigned char *b0 = s.base + SM_B0 + b * 16384;
                // This thread's rows r = 16 tg + i live at
                //   row(i) = kp[i & 7] + (i >> 3) * 1024 + (i & 7) * 128      (k; q at +8192)
                // in the 128B-swizzled tile: the swizzle term depends only on i & 7.
                const uint32_t c8 = (uint32_t)cq >> 1;
                const uint32_t abase = (c8 >> 3) * 16384u + 2u * (uint32_t)tg * 1024u + 8u * (cq & 1);
                unsigned char *kp[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) kp[j] = a0 + abase + (((c8 & 7u) ^ (uint32_t)j) << 4);
                // same position in the 64-row Kc tile
                const ptrdiff_t kc_delta = (b0 - a0) - (ptrdiff_t)((c8 >> 3) * 8192u);
                if (L < C) {  // ragged tail: zero the raw k, q rows past the sequence once
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (16 * tg + i >= L) {
                            unsigned char *row = kp[i & 7] + (i >> 3) * 1024 + (i & 7) * 128;
                            *reinterpret_cast<uint2 *>(row) = make_uint2(0u, 0u);
                            *reinterpret_cast<uint2 *>(row + 8192) = make_uint2(0u, 0u);
                        }
                }
                const uint64_t inv01 = f2_make(inv[0], inv[1]), inv23 = f2_make(inv[2], inv[3]);
                const float mu[4] = {gam[0] * inv[0], gam[1] * inv[1], gam[2] * inv[2], gam[3] * inv[3]};
                // One pass over the rows with the running product p_r:
                //   Kr = k p / mu, Qr = q p / mu (in place), Kc = k (gamma / p) / mu = k mu / p
                uint64_t pr01 = f2_make(before.x, before.y), pr23 = f2_make(before.z, before.w);
                uint2 kcv[16];  // Kc rows, stored once MMA3 of chunk n-2 has released the buffer
                // Batches of 8 rows: a batch's loads are issued before its in-place stores.
#pragma unroll
                for (int i0 = 0; i0 < 16; i0 += 8) {
                    uint2 kw[8], qw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int i = i0 + j;
                        const unsigned char *row = kp[i & 7] + (i >> 3) * 1024 + (i & 7) * 128;
                        kw[j] = *reinterpret_cast<const uint2 *>(row);
                        qw[j] = *reinterpret_cast<const uint2 *>(row + 8192);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int i = i0 + j;
                        pr01 = f2_mul(pr01, f2_make(a[i].x, a[i].y));
                        pr23 = f2_mul(pr23, f2_make(a[i].z, a[i].w));
                        const uint64_t e2a = f2_mul(pr01, inv01), e2b = f2_mul(pr23, inv23);
                        const uint64_t e3a = f2_make(__fdividef(mu[0], f2_lo(pr01)), __fdividef(mu[1], f2_hi(pr01)));
                        const uint64_t e3b = f2_make(__fdividef(mu[2], f2_lo(pr23)), __fdividef(mu[3], f2_hi(pr23)));
                        const uint64_t k01 = bf2_to_f2(kw[j].x), k23 = bf2_to_f2(kw[j].y);
                        const uint64_t q01 = bf2_to_f2(qw[j].x), q23 = bf2_to_f2(qw[j].y);
                        unsigned char *row = kp[i & 7] + (i >> 3) * 1024 + (i & 7) * 128;
                        *reinterpret_cast<uint2 *>(row) = make_uint2(f2_to_bf2(f2_mul(k01, e2a)), f2_to_bf2(f2_mul(k23, e2b)));
                        *reinterpret_cast<uint2 *>(row + 8192) =
                            make_uint2(f2_to_bf2(f2_mul(q01, e2a)), f2_to_bf2(f2_mul(q23, e2b)));
                        kcv[i] = make_uint2(f2_to_bf2(f2_mul(k01, e3a)), f2_to_bf2(f2_mul(k23, e3b)));
                    }
                }
                if (n >= 2) ok = wait_bar(s, p, B_B0_EMPTY + b, (kk - 1) & 1) && ok;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    *reinterpret_cast<uint2 *>(kp[i & 7] + (i >> 3) * 1024 + (i & 7) * 128 + kc_delta) = kcv[i];
            } else if (n >= 2) {
                ok = wait_bar(s, p, B_B0_EMPTY + b, (kk - 1) & 1) && ok;  // keeps the phase order
            }
            if (pt < 64) s.beta(b)[pt] = beta_r;
            if (pt == 0) {
                s.info(b)[0] = L;
                s.info(b)[1] = slow ? 1 : 0;
            }
            fence_proxy_async();
            mbar_arrive(s.bar(B_TAB_FULL + b));
        }
    } else {
        // ------------------------------------------------------------ solve group (warps 8-11)
        regs_inc<REGS_SOLVE>();
        const int qt = tid - 256;
        const int q4 = warp & 3;       // TMEM lane quarter = warp index in the group
        const int R = 32 * q4 + lane;  // row of [A; P]
        float *asc = reinterpret_cast<float *>(s.base + SM_SOLVE);  // A (strictly lower, beta-scaled)
        float *tsc = asc + 64 * 64;                                  // T
        const int g8 = lane >> 2, t4 = lane & 3;
        for (int n = 0; n < NC; ++n) {
            const int b = n & 1, kk = n >> 1;
            bool ok = wait_bar(s, p, B_AP_FULL + b, kk & 1);
            ok = wait_bar(s, p, B_TAB_FULL + b, kk & 1) && ok;  // the gate group's beta / info
            tc_fence_after();
            named_bar(3, SOLVE_THREADS);
            const bool go = s.flags()[1] == 0;
            const bool work = go && s.info(b)[1] == 0;  // group-uniform
            const int L = s.info(b)[0];
            uint32_t pbuf[32];
            if (work) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t r32[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + (b ? TM_AP1 : TM_AP0) + 32 * hf, r32);
                    tmem_wait_ld();
                    if (R < 64) {
                        const float bt = s.beta(b)[R];
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            float w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = 32 * hf + 4 * j4 + e;
                                w[e] = j < R ? bt * __uint_as_float(r32[4 * j4 + e]) : 0.f;
                            }
                            *reinterpret_cast<float4 *>(asc + swz(R, 32 * hf + 4 * j4)) = make_float4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        const int r = R - 64;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = 32 * hf + 2 * e;
                            const float x0 = (j <= r && r < L) ? __uint_as_float(r32[2 * e]) : 0.f;
                            const float x1 = (j + 1 <= r && r < L) ? __uint_as_float(r32[2 * e + 1]) : 0.f;
                            pbuf[16 * hf + e] = pack_bf16(x0, x1);
                        }
                    }
                }
                tc_fence_before();
            }
            named_bar(3, SOLVE_THREADS);
            if (work && q4 < 2) {
                // T step 1: the four 16x16 diagonal blocks, one thread per column
                // (x_r -= A[r][s] x_s for s < r); rows are compile-time so the A
                // loads take immediate offsets from two base pointers (the
                // swizzle flips bit 4 of the column for rows with r & 7 >= 4).
                const int blk = 2 * q4 + (lane >> 4), col = lane & 15;
                const float *rowp = asc + (16 * blk) * 64;
                const float *b0p = rowp + 16 * blk, *b1p = rowp + ((16 * blk) ^ 16);
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = i == col ? 1.f : 0.f;
#pragma unroll
                for (int sidx = 0; sidx < 15; ++sidx) {
                    const float xs = x[sidx];
#pragma unroll
                    for (int rl = sidx + 1; rl < 16; ++rl) {
                        const int kc = sidx ^ ((rl & 7) << 2);  // swizzled column within the block pair
                        const float av = kc < 16 ? b0p[rl * 64 + kc] : b1p[rl * 64 + kc - 16];
                        x[rl] -= av * xs;
                    }
                }
#pragma unroll
                for (int rl = 0; rl < 16; ++rl) tsc[swz(16 * blk + rl, 16 * blk + col)] = x[rl];
            }
            named_bar(3, SOLVE_THREADS);
            if (work && q4 < 3) {
                // T step 2 for block column J = q4, one warp, on mma.sync (tf32):
                // T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ for I = J+1 .. 3
                const int J = q4;
                float *ms = reinterpret_cast<float *>(s.base + SM_MSCR) + J * 256;
                for (int I = J + 1; I < 4; ++I) {
                    float m[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) m[nt][e] = 0.f;
                    for (int K = J; K < I; ++K) {
#pragma unroll
                        for (int k8 = 0; k8 < 16; k8 += 8) {
                            const int r0 = 16 * I + g8, c0 = 16 * K + k8 + t4;
                            const uint32_t af[4] = {to_tf32(asc[swz(r0, c0)]), to_tf32(asc[swz(r0 + 8, c0)]),
                                                    to_tf32(asc[swz(r0, c0 + 4)]), to_tf32(asc[swz(r0 + 8, c0 + 4)])};
                            const int br = 16 * K + k8 + t4;
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                const int bc = 16 * J + 8 * nt + g8;
                                mma_tf32(m[nt], af, to_tf32(tsc[swz(br, bc)]), to_tf32(tsc[swz(br + 4, bc)]));
                            }
                        }
                    }
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
                        const int r0 = 16 * I + g8, c0 = 16 * I + k8 + t4;
                        const uint32_t af[4] = {to_tf32(tsc[swz(r0, c0)]), to_tf32(tsc[swz(r0 + 8, c0)]),
                                                to_tf32(tsc[swz(r0, c0 + 4)]), to_tf32(tsc[swz(r0 + 8, c0 + 4)])};
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
                            mma_tf32(t[nt], af, to_tf32(ms[(k8 + t4) * 16 + 8 * nt + g8]),
                                     to_tf32(ms[(k8 + t4 + 4) * 16 + 8 * nt + g8]));
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int c = 16 * J + 8 * nt + 2 * t4;
                        tsc[swz(16 * I + g8, c)] = -t[nt][0];
                        tsc[swz(16 * I + g8, c + 1)] = -t[nt][1];
                        tsc[swz(16 * I + g8 + 8, c)] = -t[nt][2];
                        tsc[swz(16 * I + g8 + 8, c + 1)] = -t[nt][3];
                    }
                    __syncwarp();
                }
            }
            named_bar(3, SOLVE_THREADS);
            // [T; P] -> the bf16 operand tile, once MMA4 of the previous chunk is done
            if (n >= 1) ok = wait_bar(s, p, B_TP_EMPTY, (n - 1) & 1) && ok;
            if (ok && work) {
                unsigned char *tpt = s.base + SM_TP;
                const int r = qt >> 1, hc = qt & 1;  // T row r, columns 32hc .. 32hc+31
                float4 tv[8];  // loads before the tile stores
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    tv[2 * c4] = *reinterpret_cast<const float4 *>(tsc + swz(r, 8 * (4 * hc + c4)));
                    tv[2 * c4 + 1] = *reinterpret_cast<const float4 *>(tsc + swz(r, 8 * (4 * hc + c4) + 4));
                }
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 4 * hc + c4;
                    const float4 x0 = tv[2 * c4], x1 = tv[2 * c4 + 1];
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * c8 + e;
                        y[e] = j < r ? xv[e] : (j == r ? 1.f : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(tpt + kmajor_chunk(r, c8, 128)) =
                        make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
                }
                if (R >= 64) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8)
                        *reinterpret_cast<uint4 *>(tpt + kmajor_chunk(R, c8, 128)) =
                            make_uint4(pbuf[4 * c8], pbuf[4 * c8 + 1], pbuf[4 * c8 + 2], pbuf[4 * c8 + 3]);
                }
                fence_proxy_async();
            }
            mbar_arrive(s.bar(B_TP_FULL));
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
