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
// One cluster of two CTAs per (sequence, head). CTA `rank` owns value columns
// 64 rank .. 64 rank + 63 of the state (its state chain) and, for the work
// both halves share, key channels 64 rank .. 64 rank + 63 of the gated tables
// and every other chunk's inverse (chunks n with n % 2 == rank). Each CTA
// pushes what it computed into its peer's shared memory with bulk copies
// (cp.async.bulk shared::cta -> shared::cluster) that complete on the peer's
// mbarriers; the tensor-core issuers signal buffer releases to both CTAs with
// multicast tcgen05.commit.
//
// 512 threads per CTA. Roles are placed by SM sub-partition (warp id mod 4),
// so that each sub-partition runs the code of only two busy roles (the
// instruction caches thrash with more):
//   warps 0-3        epilogue: the state chain (R, U, state), the outputs O
//   warps 6,7,10,11  gate (sub-partitions 2, 3): products, mu, Kr / Qr / Kc
//                    for this CTA's key channels; for chunks of this CTA's
//                    parity also the P rows of [A; P] (TMEM lanes 64-127)
//   warps 4,5,8,9    solve (sub-partitions 0, 1), chunks of this CTA's parity:
//                    the A rows (TMEM lanes 0-63), T = (I + A)^{-1}, T tile
//   warp 12          TMA producer of this CTA's q, k halves (the epilogue
//                    refills v itself; the gate reads alpha into registers)
//   warp 13          MMA issuer of the state chain (one thread), TMEM owner
//   warp 14          MMA issuer of [A; P] on this CTA's parity
//   warp 15          FP8 inputs only: k and q codes -> bf16 tiles (idle otherwise)
// FP8 inputs (E4M3 codes, one power-of-two scale per 32 channels): the TMA
// warp loads the codes into the Qr half of the slot, warp 15 turns them into
// the bf16 k and q tiles in place, so the gate runs the bf16 code; E1
// dequantises v; everything after that is the bf16 path.
// Register budgets per warpgroup (setmaxnreg): epilogue 152, warps 4-11 128,
// control 104. The groups work on consecutive chunks at once. All waits are
// bounded; a CTA whose wait times out records an error and winds down.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int VS = 64;      // value columns per CTA
constexpr int KH = 64;      // key channels per CTA in the gate
constexpr int NSLICE = DV / VS;
static_assert(NSLICE == 2, "one cluster of two CTAs per (sequence, head)");
constexpr int NTHREADS = 512;
// Register shares per warpgroup. Each SM sub-partition holds one warp of
// every warpgroup, so the shares sum to 4 x 128 = the launch's allocation
// (a larger sum would make setmaxnreg.inc wait forever).
constexpr uint32_t REGS_EPI = 152, REGS_PREP = 128, REGS_CTRL = 104;
static_assert(REGS_EPI + 2 * REGS_PREP + REGS_CTRL == 4 * 128, "register split");
// setmaxnreg.inc may only raise and .dec only lower a warp's count (from the
// launch's 128); the wrong one is an illegal instruction.
static_assert(REGS_EPI >= 128 && REGS_PREP == 128 && REGS_CTRL <= 128, "inc / dec (warpgroups 1, 2 keep 128)");
constexpr int EPI_THREADS = 128;
constexpr int GATE_THREADS = 128;
constexpr int SOLVE_THREADS = 128;
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr int WARP_AUX = 14;
constexpr int WARP_DQ = 15;
constexpr float kMinGamma = 1.8e-35f;  // ~exp(-80)

// TMEM columns (fp32 accumulators, 128 lanes each); AP, XY and UO are
// double-buffered by chunk parity.
constexpr uint32_t TM_AP = 0, TM_XY = 128, TM_UO = 256, TM_D = 384, TM_COLS = 512;

// shared memory map (offsets from a 1024-byte aligned base)
// Buffers by lifetime: A0 ([Kr; Qr]) is read by the first products of its
// chunk, Kc, mu, beta and the votes until the state update of their chunk;
// both cycle through 3 slots (slot n % 3), so the q, k copies, the gate and
// the inverse of chunk n + 3 may start as soon as the state chain has begun
// chunk n.
constexpr int NSLOT = 3;
constexpr uint32_t SM_A0 = 0;          // 3 x 32 KB: [Kr; Qr], two 16 KB key-channel halves (128B swizzle)
constexpr uint32_t SM_B0 = 98304;      // 3 x 16 KB: Kc (K-major, 64 rows), two 8 KB halves
constexpr uint32_t SM_SOLVE = 147456;  // 16 KB: A, overwritten in place by T (fp32 64x64, XOR-swizzled)
constexpr uint32_t SM_V = 163840;      // 8 KB: v slice (128B swizzle)
// T and the two P slots are 8 KB K-major tiles (64 rows x 64) laid out
// back to back, so [T; P0] and [P_{b-1}; P_b] are 128-row operands: the
// products U = T R and P_b U use rows 0-63 and rows 64-127 of them.
constexpr uint32_t SM_TP = 172032;     // 24 KB: T | P0 | P1
constexpr uint32_t SM_ST = 196608;     // 16 KB: St (MN-major, 128 rows x 64)
constexpr uint32_t SM_RU = 212992;     // 8 KB: R then U (MN-major, 64 rows x 64)
constexpr uint32_t SM_MU = 221184;     // float[3][128]
constexpr uint32_t SM_BETA = 222720;   // float[3][64]
constexpr uint32_t SM_VOTE = 223488;   // int[3][8]: slow vote of key half 0 at [0], half 1 at [4]
constexpr uint32_t SM_FLAGS = 223584;  // int[8]: [1] abort, [2] the peer's abort flag at exit
constexpr uint32_t SM_TMEM = 223616;   // uint32 TMEM base
constexpr uint32_t SM_BAR = 223632;    // mbarriers (up to 40)
constexpr uint32_t SM_RED = 223952;    // float[4][64] + float[64]: slow-path reductions
constexpr uint32_t SM_MSCR = 225232;   // float[4][16*8]: mma.sync staging (3 KB reserved)
constexpr uint32_t SM_SCAN = 228304;   // float4[8][16]: per-group gate products
constexpr uint32_t SM_TOTAL = 230352;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;

// Bytes one CTA pushes into its peer per chunk: its [Kr; Qr] half, its Kc
// half, its half of mu and its slow vote.
constexpr uint32_t PUSH_TAB = 16384 + 8192 + 256 + 16;
constexpr uint32_t PUSH_TILE = 8192;  // T or P
constexpr uint16_t BOTH = 3;  // CTA mask of the cluster

// A waiter of a parity wait must never fall two phases behind, nor run a
// phase ahead, of the barrier it waits on. Every waiter below sees every
// phase of its barriers: the tables of chunk n complete TAB_FULL[n % 6] (the
// [A; P] issuer and the solve group, which take every other chunk, then see
// every phase of the barriers of their parity), [A; P] of a CTA's i-th chunk
// completes AP_FULL[i % 2], and MMA2 of chunk n completes T_EMPTY[n % 2].
constexpr int NTAB = 2 * NSLOT;
enum Bar {
    B_QK_FULL = 0, B_QK_EMPTY = 3, B_V_FULL = 6, B_TAB_FULL = 7, B_B0_EMPTY = 13, B_O_READ = 16,
    B_AP_FULL = 18, B_T_FULL = 20, B_T_EMPTY = 21, B_P_FULL = 23, B_P_EMPTY = 25, B_S_FULL = 27, B_XY_FULL = 28,
    B_R_FULL = 29, B_U_FULL = 30, B_UU_FULL = 31, B_D_FULL = 32, B_DRAIN = 33, B_DRAIN_AUX = 34, B_DQ_FULL = 35,
    B_STALL = 38,  // self-test only: nothing ever arrives on it
    B_COUNT = 39
};
static_assert(B_COUNT <= 40, "mbarrier area");

struct TcParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *alpha, *beta, *s0;
    __nv_bfloat16 *o;
    float *sT;
    const int32_t *cu_seqlens;
    const int32_t *order;
    const int32_t *dev_status;
    int32_t *err;
    const int32_t *slots;  // nullable: state slot map (s0 and sT are then the pool)
    int gate;              // kda_gate_t
    const uint8_t *qs, *ks, *vs;  // FP8 inputs: E8M0 scales, one per 32 channels (q, k, v are E4M3)
    int N, T, H;
    int stall1;  // self-test of the bounded waits: 1 + the chunk at which the state-chain
                 // issuer waits on B_STALL (0: never)
};

// FP8 inputs (the MX block format): E4M3 codes, a power-of-two scale 2^(t-127)
// per 32 channels. Four codes -> four floats, scaled (exact: the scale is a
// power of two and the dequantised value fits fp32).
__device__ __forceinline__ float e8m0(uint8_t t) { return __uint_as_float((uint32_t)t << 23); }
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float sc, float (&f)[4]) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((unsigned short)(w & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((unsigned short)(w >> 16)));
    const __half2 a = *reinterpret_cast<const __half2 *>(&h01), c = *reinterpret_cast<const __half2 *>(&h23);
    f[0] = __low2float(a) * sc;
    f[1] = __high2float(a) * sc;
    f[2] = __low2float(c) * sc;
    f[3] = __high2float(c) * sc;
}
// One FP8 input element (token-head th, channel c of a d-channel row).
__device__ __forceinline__ float fp8_at(const uint8_t *x, const uint8_t *sc, int64_t th, int c, int d) {
    const uint32_t w = x[th * d + c];
    float f[4];
    e4m3x4_to_f32(w, e8m0(sc[th * (d / 32) + c / 32]), f);
    return f[0];
}

__device__ int g_tc_error = 0;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Two fp32 values packed in 64 bits, multiplied pairwise by one instruction.
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
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
// Hardware reciprocal (PTX rcp.approx): relative error far below the bf16
// rounding its results go through.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
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
    uint32_t peer;  // cluster rank of the other CTA
    __device__ __forceinline__ uint64_t *bar(int i) const {
        return reinterpret_cast<uint64_t *>(base + SM_BAR) + i;
    }
    __device__ __forceinline__ volatile int *flags() const {
        return reinterpret_cast<volatile int *>(base + SM_FLAGS);
    }
    // slot b3 = chunk % 3
    __device__ __forceinline__ float *mu(int b3) const { return reinterpret_cast<float *>(base + SM_MU) + 128 * b3; }
    __device__ __forceinline__ float *beta(int b3) const { return reinterpret_cast<float *>(base + SM_BETA) + 64 * b3; }
    __device__ __forceinline__ int *vote(int b3) const { return reinterpret_cast<int *>(base + SM_VOTE) + 8 * b3; }
    // A chunk runs token by token when either key half voted so.
    __device__ __forceinline__ bool slow(int b3) const {
        const volatile int *v = vote(b3);
        return (v[0] | v[4]) != 0;
    }
    // Cluster address of this CTA's shared-memory location p in the peer.
    __device__ __forceinline__ uint32_t remote(const void *p) const { return mapa(smem_u32(p), peer); }
};

// Bounded wait. try_wait suspends the thread for at most about a microsecond
// (kSuspendNs) while the phase is open, so the loop bound (kMaxWaitTries
// rounds) gives up after about a second, or after tens of milliseconds should
// try_wait return at once; both lie far beyond any wait of a working kernel. A timeout sets
// the abort flag (bit 1: this CTA timed out; the error is reported once at
// exit). After a failed wait the callers skip their remaining waits
// (ok = ok && wait_bar(...)), so a CTA that gives up winds down after at most
// one timeout per warp group.
constexpr uint32_t kMaxWaitTries = 1u << 20;
__device__ __forceinline__ bool wait_bar(const Smem &s, const TcParams &, int i, uint32_t parity) {
    uint32_t it = 0;
#pragma unroll 1
    while (!mbar_try_wait(s.bar(i), parity)) {
        if (++it > kMaxWaitTries) {
            s.flags()[1] = 3;
            return false;
        }
    }
    return true;
}

// Sum over the warp of eight per-lane values (one per column), reduced and
// scattered in 9 shuffles: the result is the column ((lane >> 2) & 7) sum,
// with column bits taken from lane bits 4, 3, 2 (high to low).
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane) {
    const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float send = u16 ? v[e] : v[e + 4];
        v[e] = (u16 ? v[e + 4] : v[e]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float send = u8 ? v[e] : v[e + 2];
        v[e] = (u8 ? v[e + 2] : v[e]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float x = (u4 ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, u4 ? v[0] : v[1], 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

// Exact token-by-token update of one chunk (the K3 essay's §四 recurrence in
// fp32), used for chunks whose gates decay past the factorised range. The
// epilogue warpgroup holds the state slice in TMEM (lane = key channel,
// 64 value columns) and updates it there, eight columns at a time; sums over
// the key channels go through warp shuffles and four per-warp partials in
// shared memory. Rare, so it is written for size rather than speed, and out
// of line: the hot loop of the epilogue stays contiguous in the instruction
// caches.
__device__ __noinline__ void slow_chunk(const float *__restrict__ alpha, int gate, const void *__restrict__ kin,
                                        const void *__restrict__ qin, const void *__restrict__ vin,
                                        const uint8_t *__restrict__ ks, const uint8_t *__restrict__ qs,
                                        const uint8_t *__restrict__ vs,
                                        const float *__restrict__ beta, __nv_bfloat16 *__restrict__ o, float *red,
                                        uint32_t tm_d, int l, int warp, int lane, int64_t tok0, int L, int H, int h,
                                        int v0) {
    const int col = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
    const bool writer = (lane & 3) == 0;
#pragma unroll 1
    for (int r = 0; r < L; ++r) {
        const int64_t tk = (tok0 + r) * H + h;
        const float a = gate_at(alpha, gate, tk, l, DK);
        // (FP8 inputs when scales are given, else bf16)
        const float kf = ks ? fp8_at((const uint8_t *)kin, ks, tk, l, DK)
                            : __bfloat162float(((const __nv_bfloat16 *)kin)[tk * DK + l]);
        const float qf = qs ? fp8_at((const uint8_t *)qin, qs, tk, l, DK)
                            : __bfloat162float(((const __nv_bfloat16 *)qin)[tk * DK + l]);
        // S' = Diag(alpha) S, and this warp's part of S'^T k
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t u[8];
            float part[8];
            tmem_ld8(tm_d + 8 * g, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float x = a * __uint_as_float(u[e]);
                u[e] = __float_as_uint(x);
                part[e] = kf * x;
            }
            tmem_st8(tm_d + 8 * g, u);
            const float sum = warp_sum8(part, lane);
            if (writer) red[warp * 64 + 8 * g + col] = sum;
        }
        tmem_wait_st();
        named_bar(2, EPI_THREADS);
        if (l < 64) {
            const float vh = red[l] + red[64 + l] + red[128 + l] + red[192 + l];
            const float vf = vs ? fp8_at((const uint8_t *)vin, vs, tk, v0 + l, DV)
                                : __bfloat162float(((const __nv_bfloat16 *)vin)[tk * DV + v0 + l]);
            red[256 + l] = beta[tk] * (vf - vh);
        }
        named_bar(2, EPI_THREADS);
        // S = S' + k e^T, and this warp's part of S^T q
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t u[8];
            float part[8];
            tmem_ld8(tm_d + 8 * g, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float x = __uint_as_float(u[e]) + kf * red[256 + 8 * g + e];
                u[e] = __float_as_uint(x);
                part[e] = qf * x;
            }
            tmem_st8(tm_d + 8 * g, u);
            const float sum = warp_sum8(part, lane);
            if (writer) red[warp * 64 + 8 * g + col] = sum;
        }
        tmem_wait_st();
        named_bar(2, EPI_THREADS);
        if (l < 64) o[tk * DV + v0 + l] = __float2bfloat16_rn(red[l] + red[64 + l] + red[128 + l] + red[192 + l]);
        named_bar(2, EPI_THREADS);
    }
}

// --------------------------------------------------------------------------
// GATE (a kda_gate_t) is a template parameter so that each gate kind keeps
// the per-chunk code of the gate group as small as the per-channel one; FP8
// selects E4M3 q, k, v with block scales (TMA brings the codes, the gate and
// E1 dequantise them).
template <int GATE, bool FP8>
__global__ void __cluster_dims__(NSLICE, 1, 1) __launch_bounds__(NTHREADS, 1)
kda_prefill_tc_kernel(TcParams p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t rank = cluster_rank();  // value half and key half of this CTA (blockIdx.x % 2)
    // The 1024-byte alignment is an offset into smem_raw (not an integer
    // round trip of its address), so the compiler keeps every access through
    // s.base in the shared state space instead of falling back to generic
    // loads and stores.
    Smem s{smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u), rank ^ 1u};
    // Both CTAs of a cluster read the same status word and sequence: they
    // leave here together or not at all.
    if (p.dev_status && *p.dev_status != 0) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    const int v0 = (int)rank * VS;   // first value column of this CTA's state slice
    const int c0 = (int)rank * KH;   // first key channel of this CTA's gate half
    bool fresh;  // a fresh slot starts from the zero state
    const int64_t state_off = (slot_of(p.slots, seq, fresh) * H + h) * DK * DV;
    const float *s0 = fresh ? nullptr : p.s0;
    const int NC = (int)((T + C - 1) / C);

    if (NC == 0) {  // empty sequence: the final state is the initial one
        if (p.sT)
            for (int e = tid; e < DK * VS; e += NTHREADS) {
                const int c = e / VS, j = e % VS;
                p.sT[state_off + (int64_t)c * DV + v0 + j] = s0 ? s0[state_off + (int64_t)c * DV + v0 + j] : 0.f;
            }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(s.bar(B_QK_FULL + i), 1);
            // MMA1 of both CTAs and MMA0 of the solving CTA (multicast commits),
            // and the solving CTA's solve group once it holds the chunk's
            // barrier phases (so no waiter of TAB_FULL / AP_FULL can fall two
            // phases behind)
            mbar_init(s.bar(B_QK_EMPTY + i), 4);
            mbar_init(s.bar(B_B0_EMPTY + i), 2);  // MMA3 of both CTAs
            mbar_init(s.bar(B_DQ_FULL + i), 1);   // FP8: the bf16 k, q tiles of the slot (warp 15)
        }
        // own gate (expecting the peer's bytes) + the peer's copies
        for (int i = 0; i < NTAB; ++i) mbar_init(s.bar(B_TAB_FULL + i), 1);
        for (int i = 0; i < 2; ++i) mbar_init(s.bar(B_O_READ + i), 64);
        mbar_init(s.bar(B_V_FULL), 1);   // v: loaded by the epilogue for its next chunk
        for (int i = 0; i < 2; ++i) mbar_init(s.bar(B_AP_FULL + i), 1);
        // T and P of a chunk: the solving CTA arrives locally, the other CTA
        // gets a remote arrive and the copy; released by MMA2 (T) / MMA4 (P)
        // of both CTAs
        mbar_init(s.bar(B_T_FULL), 1);
        for (int i = 0; i < 2; ++i) mbar_init(s.bar(B_T_EMPTY + i), 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(s.bar(B_P_FULL + i), 1);
            mbar_init(s.bar(B_P_EMPTY + i), 2);
        }
        mbar_init(s.bar(B_S_FULL), EPI_THREADS);
        mbar_init(s.bar(B_XY_FULL), 1);
        mbar_init(s.bar(B_R_FULL), 64);
        mbar_init(s.bar(B_U_FULL), 1);
        mbar_init(s.bar(B_UU_FULL), 64);
        mbar_init(s.bar(B_D_FULL), 1);
        mbar_init(s.bar(B_DRAIN), 1);
        mbar_init(s.bar(B_DRAIN_AUX), 1);
        mbar_init(s.bar(B_STALL), 1);
        for (int i = 0; i < 8; ++i) s.flags()[i] = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(reinterpret_cast<uint32_t *>(s.base + SM_TMEM), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive, copy or commit
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
            int nqk = 0;  // chunks whose q, k halves were issued
            for (int n = 0; n < NC; ++n) {
                const int b = n % NSLOT, kk = n / NSLOT;
                const int z = (int)(t_begin + (int64_t)n * C);
                // this CTA's key half of k and q (raw; the gate transforms them in place)
                if (n >= NSLOT && !wait_bar(s, p, B_QK_EMPTY + b, (kk - 1) & 1)) break;
                unsigned char *a0 = s.base + SM_A0 + b * 32768 + rank * 16384;
                if constexpr (FP8) {  // codes into the Qr half (64-byte rows); warp 15 makes the bf16 tiles
                    mbar_arrive_expect_tx(s.bar(B_QK_FULL + b), 8192);
                    tma_load_3d(a0 + 8192, &tm_k, s.bar(B_QK_FULL + b), c0, h, z);
                    tma_load_3d(a0 + 12288, &tm_q, s.bar(B_QK_FULL + b), c0, h, z);
                } else {
                    mbar_arrive_expect_tx(s.bar(B_QK_FULL + b), 16384);
                    tma_load_3d(a0, &tm_k, s.bar(B_QK_FULL + b), c0, h, z);
                    tma_load_3d(a0 + 8192, &tm_q, s.bar(B_QK_FULL + b), c0, h, z);
                }
                nqk = n + 1;
            }
            // never leave copies in flight: wait (bounded) for the last ones
            for (int n = nqk - NSLOT < 0 ? 0 : nqk - NSLOT; n < nqk; ++n)
                mbar_wait(s.bar(B_QK_FULL + n % NSLOT), (n / NSLOT) & 1);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA (state chain)
        if (lane == 0) {
            constexpr uint32_t I_KM_MN = idesc_bf16(128, 64, false, true);
            constexpr uint32_t I_MN_MN = idesc_bf16(128, 64, true, true);
            const uint32_t a0_base = smem_u32(s.base + SM_A0), b0_base = smem_u32(s.base + SM_B0);
            const uint32_t tp = smem_u32(s.base + SM_TP), st = smem_u32(s.base + SM_ST),
                           ru = smem_u32(s.base + SM_RU);
            bool ok = true;
            for (int n = 0; ok && n < NC; ++n) {
                const int b = n & 1, kk = n >> 1, b3 = n % NSLOT;
                if (n + 1 == p.stall1 && !(ok = wait_bar(s, p, B_STALL, 0))) break;
                if (!(ok = wait_bar(s, p, B_TAB_FULL + n % NTAB, (n / NTAB) & 1))) break;
                const bool fast = !s.slow(b3);
                const uint32_t xy = tmem + TM_XY + 64 * b, uo = tmem + TM_UO + 64 * b;
                // MMA1: [X; Y] = [Kr; Qr] St, once the outputs of chunk n-2 left XY[b]
                if (n >= 2 && !(ok = wait_bar(s, p, B_O_READ + b, (kk - 1) & 1))) break;
                if (!(ok = wait_bar(s, p, B_S_FULL, n & 1))) break;
                tc_fence_after();
                if (fast) {
                    const uint32_t a0 = a0_base + b3 * 32768;
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(xy, sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                  sdesc_sw128(st + ks * 2048, 16384, 1024), I_KM_MN, ks > 0);
                }
                umma_commit(s.bar(B_XY_FULL));
                umma_commit_mc(s.bar(B_QK_EMPTY + b3), BOTH);  // A0[b3] read
                // MMA2: U = T R (rows 0-63 of [T; P0] R)
                if (!(ok = wait_bar(s, p, B_R_FULL, n & 1))) break;
                if (!(ok = wait_bar(s, p, B_T_FULL, n & 1))) break;
                tc_fence_after();
                if (fast) {
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16(uo, sdesc_sw128(tp + ks * 32, 16, 1024), sdesc_sw128(ru + ks * 2048, 8192, 1024),
                                  I_KM_MN, ks > 0);
                }
                umma_commit(s.bar(B_U_FULL));
                umma_commit_mc(s.bar(B_T_EMPTY + b), BOTH);
                // MMA3: D += Kc^T U (state update); MMA4: O2 = P U (rows 64-127 of [P_{b-1}; P_b] U)
                if (!(ok = wait_bar(s, p, B_UU_FULL, n & 1))) break;
                if (!(ok = wait_bar(s, p, B_P_FULL + b, kk & 1))) break;
                tc_fence_after();
                if (fast) {
                    const uint32_t b0 = b0_base + b3 * 16384, pa = tp + 8192 * b;
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks) {
                        umma_bf16(tmem + TM_D, sdesc_sw128(b0 + ks * 2048, 8192, 1024),
                                  sdesc_sw128(ru + ks * 2048, 8192, 1024), I_MN_MN, 1);
                        umma_bf16(uo, sdesc_sw128(pa + ks * 32, 16, 1024), sdesc_sw128(ru + ks * 2048, 8192, 1024),
                                  I_KM_MN, ks > 0);
                    }
                }
                umma_commit(s.bar(B_D_FULL));
                umma_commit_mc(s.bar(B_B0_EMPTY + b3), BOTH);
                umma_commit_mc(s.bar(B_P_EMPTY + b), BOTH);
            }
            // drain: every MMA issued has completed before TMEM is released
            umma_commit(s.bar(B_DRAIN));
            mbar_wait(s.bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else if (warp == WARP_AUX) {
        // ------------------------------------------------------------ [A; P] issuer (this CTA's parity)
        if (lane == 0) {
            constexpr uint32_t I_AP = idesc_bf16(128, 64, false, false);
            for (int n = (int)rank, i = 0; n < NC; n += 2, ++i) {
                const int b3 = n % NSLOT;
                if (!wait_bar(s, p, B_TAB_FULL + n % NTAB, (n / NTAB) & 1)) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(s.base + SM_A0) + b3 * 32768;
                const uint32_t b0 = smem_u32(s.base + SM_B0) + b3 * 16384;
                if (!s.slow(b3)) {
                    const uint32_t d = tmem + TM_AP + 64 * (i & 1);
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(d, sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                  sdesc_sw128(b0 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), I_AP, ks > 0);
                }
                umma_commit(s.bar(B_AP_FULL + (i & 1)));
                umma_commit_mc(s.bar(B_QK_EMPTY + b3), BOTH);  // A0[b3] read
            }
            umma_commit(s.bar(B_DRAIN_AUX));
            mbar_wait(s.bar(B_DRAIN_AUX), 0);
        }
        __syncwarp();
    } else if (warp == WARP_DQ) {
        // ------------------------------------------------------------ FP8: k, q codes -> bf16 tiles
        // Lane: token rows lane and lane + 32 of this CTA's key half. The codes
        // (64-byte rows: k at +8192, q at +12288 of the half) become the tiles
        // the TMA writes for bf16 inputs (128-byte rows, 16-byte chunks swizzled
        // by the row's low three bits): k over the Kr half, q over the Qr half.
        // Four passes (k rows 0-31, 32-63, q rows 0-31, 32-63); in each, every
        // lane reads its row's codes before any lane writes. A pass writes over
        // codes only of rows already converted or of its own pass (q rows 0-31
        // land on k's codes, q rows 32-63 on q's codes of rows 0-63).
        if constexpr (FP8) {
            bool alive = true;
            for (int n = 0; n < NC; ++n) {
                const int b = n % NSLOT, kk = n / NSLOT;
                const int64_t tok0 = t_begin + (int64_t)n * C;
                const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
                uint32_t ksw[2], qsw[2];  // the rows' scale words, loaded before the wait
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = lane + 32 * u;
                    ksw[u] = qsw[u] = 0x7f7f7f7fu;
                    if (r < L) {
                        ksw[u] = __ldg(reinterpret_cast<const uint32_t *>(p.ks) + (tok0 + r) * H + h);
                        qsw[u] = __ldg(reinterpret_cast<const uint32_t *>(p.qs) + (tok0 + r) * H + h);
                    }
                }
                alive = alive && s.flags()[1] == 0;
                const bool ok = __all_sync(0xffffffffu, alive && wait_bar(s, p, B_QK_FULL + b, kk & 1));
                unsigned char *ah = s.base + SM_A0 + b * 32768 + rank * 16384;
                if (ok) {
#pragma unroll 1
                    for (int tu = 0; tu < 4; ++tu) {  // k rows lane, lane + 32, then q rows lane, lane + 32
                        const int t = tu >> 1, r = lane + 32 * (tu & 1);
                        const uint32_t sw = t ? ((tu & 1) ? qsw[1] : qsw[0]) : ((tu & 1) ? ksw[1] : ksw[0]);
                        const unsigned char *src = ah + 8192 + 4096 * t + r * 64;
                        uint4 w0 = *reinterpret_cast<const uint4 *>(src), w1 = *reinterpret_cast<const uint4 *>(src + 16),
                              w2 = *reinterpret_cast<const uint4 *>(src + 32), w3 = *reinterpret_cast<const uint4 *>(src + 48);
                        __syncwarp();  // q rows 32-63 land on codes other lanes read in this pass
                        unsigned char *dst = ah + 8192 * t + r * 128;
#pragma unroll 1
                        for (int c2 = 0; c2 < 4; ++c2) {  // 16 channels: codes 16 c2 .. 16 c2 + 15, in w0
                            const float sc = e8m0((uint8_t)(sw >> (8 * (2 * (int)rank + (c2 >> 1)))));
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                float f[4], g[4];
                                e4m3x4_to_f32(hh ? w0.z : w0.x, sc, f);
                                e4m3x4_to_f32(hh ? w0.w : w0.y, sc, g);
                                *reinterpret_cast<uint4 *>(dst + (((2 * c2 + hh) ^ (r & 7)) << 4)) =
                                    make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(g[0], g[1]),
                                               pack_bf16(g[2], g[3]));
                            }
                            w0 = w1;
                            w1 = w2;
                            w2 = w3;
                        }
                        __syncwarp();
                    }
                    fence_proxy_async();  // before the slot returns to the copy engine
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(s.bar(B_DQ_FULL + b));
                alive = ok;
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        regs_inc<REGS_EPI>();
        // Group discipline (here and in the gate / solve groups): a failed
        // wait never leaves the loop; the thread keeps passing the same
        // barriers with its work switched off, and the next waits return at
        // once (abort flag). TMEM loads and stores are warp-collective, so the
        // conditions around them are warp-uniform.
        const int l = tid;  // TMEM lane: key channel (state) or token row
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // The v slice is single-buffered and refilled by this group as soon
        // as E1 has read it (thread 0 issues the copy).
        if (tid == 0) {
            mbar_arrive_expect_tx(s.bar(B_V_FULL), FP8 ? 4096 : 8192);
            tma_load_3d(s.base + SM_V, &tm_v, s.bar(B_V_FULL), v0, h, (int)t_begin);
        }
        const uint32_t tm_d = tmem + lane_off + TM_D;
        uint32_t r32[32];
        bool ok = wait_bar(s, p, B_TAB_FULL, 0);
        // The chunk's slow flag and mu are read once, as soon as its tables
        // exist, and kept in registers: the gate of chunk n + 3 overwrites them.
        bool slow_cur = s.slow(0);
        float mu_cur = (ok && !slow_cur) ? s.mu(0)[l] : 1.f;
        bool slow_prev = false;
        // St_0 = Diag(mu_0) S0 -> TMEM (fp32 accumulator base) and the bf16 operand
        {
            const float *src = (ok && s0) ? s0 + state_off + (int64_t)l * DV + v0 : nullptr;
            unsigned char *st = s.base + SM_ST;
#pragma unroll 1
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

        for (int n = 0; n <= NC; ++n) {
            const int b = n & 1;
            if (warp >= 2 && n >= 1) {
                // Outputs of chunk n-1 (token rows 64-127 of XY and UO): O = Y + P U.
                // Off the state chain: MMA1 of chunk n+1 waits for this read.
                const int m = n - 1, bm = m & 1;
                const int Lm = (int)((T - (int64_t)m * C) < C ? (T - (int64_t)m * C) : C);
                const int r = l - 64;
                if (__all_sync(0xffffffffu, ok && !slow_prev)) {
                    __nv_bfloat16 *dst = p.o + ((t_begin + (int64_t)m * C + r) * H + h) * DV + v0;
                    uint32_t y32[32];
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        tmem_ld32(tmem + lane_off + TM_XY + 64 * bm + 32 * hf, y32);
                        tmem_ld32(tmem + lane_off + TM_UO + 64 * bm + 32 * hf, r32);
                        tmem_wait_ld();
                        if (r < Lm) {
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                uint32_t w[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int j = 8 * c4 + 2 * e;
                                    w[e] = f2_to_bf2(f2_add((uint64_t)y32[j] | ((uint64_t)y32[j + 1] << 32),
                                                            (uint64_t)r32[j] | ((uint64_t)r32[j + 1] << 32)));
                                }
                                *reinterpret_cast<uint4 *>(dst + 32 * hf + 8 * c4) = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(s.bar(B_O_READ + bm));
            }
            if (n == NC) break;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            const int64_t tok0 = t_begin + (int64_t)n * C;
            ok = ok && s.flags()[1] == 0;  // stop waiting once the CTA gave up
            if (warp < 2) {
                // E1: R = beta (V - X) for token rows 0-63
                float vsc2[2] = {1.f, 1.f};  // FP8: this row's two block scales, loaded before the waits
                if constexpr (FP8) {
                    if (l < L) {
                        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(p.vs) + (tok0 + l) * H + h);
                        vsc2[0] = e8m0((uint8_t)(w >> (8 * (v0 / 32))));
                        vsc2[1] = e8m0((uint8_t)(w >> (8 * (v0 / 32 + 1))));
                    }
                }
                ok = ok && wait_bar(s, p, B_XY_FULL, n & 1);
                ok = ok && wait_bar(s, p, B_V_FULL, n & 1);
                tc_fence_after();
                const bool act = __all_sync(0xffffffffu, ok && !slow_cur);
                unsigned char *ru = s.base + SM_RU;
                if (act) {
                    const float bt = s.beta(n % NSLOT)[l];
                    const uint64_t bt2 = f2_make(bt, bt);
                    const unsigned char *vt = s.base + SM_V;
#pragma unroll 1
                    for (int qq = 0; qq < 4; ++qq) {  // 16 columns at a time
                        uint4 vrow[2];  // the v row first: no load waits behind an R store
                        float vsc = 1.f;
                        if constexpr (FP8) {  // 16 E4M3 codes of the 64-byte row (64B swizzle) and their scale
                            vrow[0] = *reinterpret_cast<const uint4 *>(vt + l * 64 + 16 * (qq ^ ((l >> 1) & 3)));
                            vsc = (qq >> 1) ? vsc2[1] : vsc2[0];
                        } else {
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2)
                                vrow[c2] = *reinterpret_cast<const uint4 *>(vt + row128_chunk(l, 2 * qq + c2));
                        }
                        uint32_t x16[16];
                        tmem_ld16(tmem + lane_off + TM_XY + 64 * b + 16 * qq, x16);
                        tmem_wait_ld();
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
                            uint64_t vp[4];  // 8 values of v as 4 fp32 pairs
                            if constexpr (FP8) {
                                float f[8];
                                e4m3x4_to_f32(c2 ? vrow[0].z : vrow[0].x, vsc, *reinterpret_cast<float (*)[4]>(f));
                                e4m3x4_to_f32(c2 ? vrow[0].w : vrow[0].y, vsc, *reinterpret_cast<float (*)[4]>(f + 4));
#pragma unroll
                                for (int e = 0; e < 4; ++e) vp[e] = f2_make(f[2 * e], f[2 * e + 1]);
                            } else {
                                const uint32_t vw[4] = {vrow[c2].x, vrow[c2].y, vrow[c2].z, vrow[c2].w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) vp[e] = bf2_to_f2(vw[e]);
                            }
                            uint32_t ow[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint64_t x2 = (uint64_t)x16[8 * c2 + 2 * e] | ((uint64_t)x16[8 * c2 + 2 * e + 1] << 32);
                                ow[e] = f2_to_bf2(f2_mul(f2_sub(vp[e], x2), bt2));
                            }
                            *reinterpret_cast<uint4 *>(ru + row128_chunk(l, 2 * qq + c2)) =
                                make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(s.bar(B_R_FULL));
                named_bar(4, 64);  // both E1 warps have read v: load the next chunk's
                if (tid == 0 && n + 1 < NC && ok) {  // (no new copies once this thread gave up)
                    mbar_arrive_expect_tx(s.bar(B_V_FULL), FP8 ? 4096 : 8192);
                    tma_load_3d(s.base + SM_V, &tm_v, s.bar(B_V_FULL), v0, h, (int)(tok0 + C));
                }
                // E2: U -> bf16 operand (replaces R, which MMA2 has consumed)
                ok = ok && wait_bar(s, p, B_U_FULL, n & 1);
                tc_fence_after();
                if (__all_sync(0xffffffffu, act && ok)) {
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        tmem_ld32(tmem + lane_off + TM_UO + 64 * b + 32 * hf, r32);
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
            }
            // E3: the state S_{n+1} = mu_n D -> St_{n+1} = mu_{n+1} S_{n+1}
            const bool last = n == NC - 1;
            float mu_next = 1.f;
            bool slow_next = false;
            if (!last) {  // the next chunk's tables exist long before D_FULL
                ok = ok && wait_bar(s, p, B_TAB_FULL + (n + 1) % NTAB, ((n + 1) / NTAB) & 1);
                // every thread reads the same slot: it changes only once the
                // state update of chunk n+1 released it, or never after an abort
                slow_next = s.slow((n + 1) % NSLOT);
                if (ok && !slow_next) mu_next = s.mu((n + 1) % NSLOT)[l];
            }
            ok = ok && wait_bar(s, p, B_D_FULL, n & 1);
            tc_fence_after();
            bool go = s.flags()[1] == 0;
            if (slow_cur) {  // group-uniform (every thread read the same votes)
                // one decision for the whole group: the slow path has group barriers
                go = !named_bar_or(2, EPI_THREADS, !go);
                if (go)
                    slow_chunk(p.alpha, p.gate, p.k, p.q, p.v, FP8 ? p.ks : nullptr, FP8 ? p.qs : nullptr,
                               FP8 ? p.vs : nullptr, p.beta, p.o, reinterpret_cast<float *>(s.base + SM_RED), tm_d,
                               l, warp, lane, tok0, L, H, h, v0);
            }
            unsigned char *st = s.base + SM_ST;
            float *fin = p.sT ? p.sT + state_off + (int64_t)l * DV + v0 : nullptr;
            // one scale per row: mu_n mu_{n+1} (the state) or mu_n (the final state)
            const float sc = last ? mu_cur : mu_cur * mu_next;
            const uint64_t sc2 = f2_make(sc, sc);
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                tmem_ld32(tm_d + 32 * hf, r32);
                tmem_wait_ld();
                uint64_t x2[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    x2[j] = f2_mul((uint64_t)r32[2 * j] | ((uint64_t)r32[2 * j + 1] << 32), sc2);
                if (last) {
                    if (go && fin)
#pragma unroll
                        for (int j = 0; j < 16; j += 2)
                            *reinterpret_cast<float4 *>(fin + 32 * hf + 2 * j) =
                                make_float4(f2_lo(x2[j]), f2_hi(x2[j]), f2_lo(x2[j + 1]), f2_hi(x2[j + 1]));
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        r32[2 * j] = (uint32_t)x2[j];
                        r32[2 * j + 1] = (uint32_t)(x2[j] >> 32);
                    }
                    tmem_st32(tm_d + 32 * hf, r32);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(st + row128_chunk(l, 4 * hf + c4)) =
                            make_uint4(f2_to_bf2(x2[4 * c4]), f2_to_bf2(x2[4 * c4 + 1]), f2_to_bf2(x2[4 * c4 + 2]),
                                       f2_to_bf2(x2[4 * c4 + 3]));
                }
            }
            if (!last) {
                tmem_wait_st();
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(s.bar(B_S_FULL));
            }
            slow_prev = slow_cur;
            mu_cur = mu_next;
            slow_cur = slow_next;
        }
    } else if ((warp & 3) >= 2) {
        // ------------------------------------------------------------ gate group (warps 6, 7, 10, 11)
        // Thread: key channels c0 + 4cq .. c0 + 4cq + 3; token rows 8rg .. 8rg+7.
        // (SM sub-partitions 2 and 3; TMEM lanes 64-127, the P rows of [A; P])
        const int gw = ((warp >> 3) << 1) | (warp & 1);  // 6, 7, 10, 11 -> 0..3
        const int pt = 32 * gw + lane;
        const int cq = pt & 15, rg = pt >> 4;
        float4 *scan = reinterpret_cast<float4 *>(s.base + SM_SCAN);
        // Byte offset of this thread's 8 bytes in row 8 rg + j of a 128B-swizzled
        // 64-column tile: rg * 1024 + j * 128 + ((c8 ^ j) << 4) + sub.
        const uint32_t c8 = (uint32_t)cq >> 1, sub = ((uint32_t)cq & 1u) * 8u;
        const uint32_t rowbase = (uint32_t)rg * 1024u + sub;
        // alpha of this thread's channels in rows 8 rg .. 8 rg + 7 goes from
        // global memory straight into registers, loaded before the chunk's
        // waits (rows past the sequence end are not read). (An L2 prefetch
        // one chunk ahead gained nothing and cost 1.4 KB of hot code.)
        // (one gate per token-head, broadcast over the channels, for the
        // scalar kind; none at all for the delta rule)
        auto alpha_src = [&](int n) {
            const int64_t th = (t_begin + (int64_t)n * C + 8 * rg) * H + h;
            return GATE == KDA_GATE_CHANNEL ? p.alpha + th * DK + c0 + 4 * cq : p.alpha + th;
        };
        bool alive = true;
        for (int n = 0; n <= NC; ++n) {
          if (n < NC) {
            const int b = n % NSLOT, kk = n / NSLOT;
            const int64_t tok0 = t_begin + (int64_t)n * C;
            const int L = (int)((T - (int64_t)n * C) < C ? (T - (int64_t)n * C) : C);
            // beta and alpha of this chunk, loaded before the waits so their
            // latency is hidden
            const float beta_r = pt < L ? p.beta[(tok0 + pt) * H + h] : 0.f;
            float4 arow[8];
            {
                const float *src = alpha_src(n);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 a = make_float4(1.f, 1.f, 1.f, 1.f);
                    if (8 * rg + j < L) {
                        if constexpr (GATE == KDA_GATE_CHANNEL) {
                            a = __ldg(reinterpret_cast<const float4 *>(src + (int64_t)j * H * DK));
                        } else if constexpr (GATE == KDA_GATE_SCALAR) {
                            const float x = __ldg(src + (int64_t)j * H);
                            a = make_float4(x, x, x, x);
                        }
                    }
                    arow[j] = a;
                }
            }
            const int b3 = b;  // A0 and B0 slots go together
            alive = alive && s.flags()[1] == 0;  // stop waiting once the CTA gave up
            // (FP8: the bf16 tiles warp 15 made from the codes)
            bool ok = alive && wait_bar(s, p, (FP8 ? B_DQ_FULL : B_QK_FULL) + b, kk & 1);
            // products of this thread's 8 rows, then the 8 group products
            float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 a = arow[j];
                g.x *= a.x; g.y *= a.y; g.z *= a.z; g.w *= a.w;
            }
            scan[rg * 16 + cq] = g;
            named_bar(1, GATE_THREADS);
            float4 before = make_float4(1.f, 1.f, 1.f, 1.f), after = before;
#pragma unroll
            for (int gi = 0; gi < 8; ++gi) {
                const float4 x = scan[gi * 16 + cq];
                if (gi < rg) { before.x *= x.x; before.y *= x.y; before.z *= x.z; before.w *= x.w; }
                if (gi > rg) { after.x *= x.x; after.y *= x.y; after.z *= x.z; after.w *= x.w; }
            }
            const float gm[4] = {before.x * g.x * after.x, before.y * g.y * after.y, before.z * g.z * after.z,
                                 before.w * g.w * after.w};
            bool bad = false;
#pragma unroll
            for (int c = 0; c < 4; ++c) bad |= !(gm[c] >= kMinGamma);
            // vote of this key half (the barrier also keeps the scan slots
            // from being overwritten while others still read them)
            const bool slow = named_bar_or(1, GATE_THREADS, bad);
            float inv[4], mu[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                inv[c] = slow ? 1.f : rsqrtf(gm[c]);
                mu[c] = gm[c] * inv[c];
            }
            // Kc, mu, beta and the votes go to slot n % 3 once the state update
            // of chunk n-3 released it in both CTAs
            if (n >= NSLOT) ok = ok && wait_bar(s, p, B_B0_EMPTY + b3, (kk - 1) & 1);
            unsigned char *ah = s.base + SM_A0 + b * 32768 + rank * 16384;  // [k; q] rows of this key half
            unsigned char *kch = s.base + SM_B0 + b3 * 16384 + rank * 8192;  // Kc rows of this key half
            if (ok && !slow) {
                // One pass over the rows with the running product p_r:
                // Kr = k p / mu and Qr = q p / mu in place, Kc = k mu / p (the
                // gates after row r over mu). Rows past the sequence end read
                // as k = q = 0, alpha = 1.
                const uint64_t inv01 = f2_make(inv[0], inv[1]), inv23 = f2_make(inv[2], inv[3]);
                const uint64_t mu01 = f2_make(mu[0], mu[1]), mu23 = f2_make(mu[2], mu[3]);
                uint64_t pr01 = f2_make(before.x, before.y), pr23 = f2_make(before.z, before.w);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t off = rowbase + (uint32_t)j * 128u + ((c8 ^ (uint32_t)j) << 4);
                    const bool in = 8 * rg + j < L;
                    const uint2 kw = in ? *reinterpret_cast<const uint2 *>(ah + off) : make_uint2(0u, 0u);
                    const uint2 qw = in ? *reinterpret_cast<const uint2 *>(ah + 8192 + off) : make_uint2(0u, 0u);
                    const uint64_t k01 = bf2_to_f2(kw.x), k23 = bf2_to_f2(kw.y);
                    const uint64_t q01 = bf2_to_f2(qw.x), q23 = bf2_to_f2(qw.y);
                    pr01 = f2_mul(pr01, f2_make(arow[j].x, arow[j].y));
                    pr23 = f2_mul(pr23, f2_make(arow[j].z, arow[j].w));
                    const uint64_t e01 = f2_mul(pr01, inv01), e23 = f2_mul(pr23, inv23);
                    const uint64_t c01 = f2_mul(f2_make(rcp_approx(f2_lo(pr01)), rcp_approx(f2_hi(pr01))), mu01);
                    const uint64_t c23 = f2_mul(f2_make(rcp_approx(f2_lo(pr23)), rcp_approx(f2_hi(pr23))), mu23);
                    *reinterpret_cast<uint2 *>(ah + off) =
                        make_uint2(f2_to_bf2(f2_mul(k01, e01)), f2_to_bf2(f2_mul(k23, e23)));
                    *reinterpret_cast<uint2 *>(ah + 8192 + off) =
                        make_uint2(f2_to_bf2(f2_mul(q01, e01)), f2_to_bf2(f2_mul(q23, e23)));
                    *reinterpret_cast<uint2 *>(kch + off) =
                        make_uint2(f2_to_bf2(f2_mul(k01, c01)), f2_to_bf2(f2_mul(k23, c23)));
                }
            }
            // (after an abort nothing more is written: slots that others may
            // still read stay as they are)
            float *mu_b = s.mu(b3) + c0;
            if (ok && rg == 0) *reinterpret_cast<float4 *>(mu_b + 4 * cq) = make_float4(mu[0], mu[1], mu[2], mu[3]);
            if (ok && pt < 64) s.beta(b3)[pt] = beta_r;
            int *vslot = s.vote(b3) + 4 * rank;
            if (ok && pt == 0) vslot[0] = slow ? 1 : 0;
            fence_proxy_async();
            named_bar(1, GATE_THREADS);
            if (ok && pt == 0) {
                // this key half into the peer (its slot n % 3 was released with
                // QK_EMPTY and B0_EMPTY of chunk n-3, in both CTAs)
                const uint32_t rbar = s.remote(s.bar(B_TAB_FULL + n % NTAB));
                bulk_s2c(s.remote(ah), ah, 16384, rbar);
                bulk_s2c(s.remote(kch), kch, 8192, rbar);
                bulk_s2c(s.remote(mu_b), mu_b, 256, rbar);
                bulk_s2c(s.remote(vslot), vslot, 16, rbar);
                // own tables are written; the peer's arrive as copies
                mbar_arrive_expect_tx(s.bar(B_TAB_FULL + n % NTAB), PUSH_TAB);
            }
            alive = ok;
          }
            // ---- P read-out of chunk m = n - 1 when this CTA solves it: by now
            // its [A; P] product has long completed (it waited only for the
            // tables of m, which preceded the gate of n)
            const int m = n - 1;
            if (m < 0 || (m & 1) != (int)rank) continue;
            const int bm = m & 1, im = m >> 1;
            const int Lm = (int)((T - (int64_t)m * C) < C ? (T - (int64_t)m * C) : C);
            bool okp = alive && wait_bar(s, p, B_AP_FULL + (im & 1), (im >> 1) & 1);
            tc_fence_after();
            const bool gop = !named_bar_or(1, GATE_THREADS, s.flags()[1] != 0);
            const bool workp = gop && !s.slow(m % NSLOT);
            // P row r (masked: j <= r, rows past the sequence end zero), columns
            // 32 hq .. 32 hq + 31, into slot bm of the P tiles once MMA4 of chunk
            // m-2 released it in both CTAs, then to the peer
            if (m >= 2) okp = okp && wait_bar(s, p, B_P_EMPTY + bm, ((m >> 1) - 1) & 1);
            const bool wr = __all_sync(0xffffffffu, okp && workp);
            unsigned char *ptile = s.base + SM_TP + 8192 * (bm + 1);
            if (wr) {
                const int hq = gw >> 1, r = 32 * ((warp & 3) - 2) + lane;
                const int lim = r < Lm ? r : -1;  // last unmasked column
                uint32_t r32[32];
                tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + TM_AP + 64 * (im & 1) + 32 * hq, r32);
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 32 * hq + 8 * c4 + 2 * e;
                        w[e] = pack_bf16(j <= lim ? __uint_as_float(r32[8 * c4 + 2 * e]) : 0.f,
                                         j + 1 <= lim ? __uint_as_float(r32[8 * c4 + 2 * e + 1]) : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(ptile + kmajor_chunk(r, 4 * hq + c4, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async();
            }
            tc_fence_before();
            const bool pushed = named_bar_or(1, GATE_THREADS, wr);
            if (pt == 0) {
                const uint32_t rbar = s.remote(s.bar(B_P_FULL + bm));
                if (pushed) {
                    mbar_arrive_remote_tx(rbar, PUSH_TILE);
                    bulk_s2c(s.remote(ptile), ptile, PUSH_TILE, rbar);
                } else {
                    mbar_arrive_remote_tx(rbar, 0);
                }
                mbar_arrive(s.bar(B_P_FULL + bm));
            }
            alive = okp;
        }
    } else {
        // ------------------------------------------------------------ solve group (warps 4, 5, 8, 9)
        // Chunks n = rank, rank + 2, ...
        // (SM sub-partitions 0 and 1; TMEM lanes 0-63, the A rows of [A; P])
        const int gw = ((warp >> 3) << 1) | (warp & 1);  // 4, 5, 8, 9 -> 0..3
        const int qt = 32 * gw + lane;
        const int q4 = warp & 3;           // TMEM lane quarter (0 or 1)
        const int R = 32 * q4 + lane;      // row of A
        const int hq = gw >> 1;            // column half of the A read-out
        // One fp32 64x64 scratch holds A and is overwritten by T block by block
        // (16x16 blocks (I, J)): the read-out writes A's strictly lower blocks
        // and zeros above the block diagonal; each step below writes a block
        // of T only once the A block in its place has been read.
        float *tsc = reinterpret_cast<float *>(s.base + SM_SOLVE);
        const int g8 = lane >> 2, t4 = lane & 3;
        bool alive = true;
        for (int n = (int)rank, i = 0; n < NC; n += 2, ++i) {
            const int b3 = n % NSLOT;
            alive = alive && s.flags()[1] == 0;  // stop waiting once the CTA gave up
            bool ok = alive && wait_bar(s, p, B_TAB_FULL + n % NTAB, (n / NTAB) & 1);  // beta and the votes
            ok = ok && wait_bar(s, p, B_AP_FULL + (i & 1), (i >> 1) & 1);
            tc_fence_after();
            // group-uniform decisions: step 2 and the TMEM loads are warp-collective
            const bool go = !named_bar_or(3, SOLVE_THREADS, s.flags()[1] != 0);
            // every thread of the group is past this chunk's TAB_FULL and
            // AP_FULL phases: A0 slot b3 may be refilled in both CTAs
            if (qt == 0) {
                mbar_arrive(s.bar(B_QK_EMPTY + b3));
                mbar_arrive_remote_tx(s.remote(s.bar(B_QK_EMPTY + b3)), 0);
            }
            const bool work = go && !s.slow(b3);
            if (work) {
                // A row R, columns 32 hq .. 32 hq + 31, beta-scaled, zero from
                // the block after the diagonal block on (the diagonal block's
                // upper part is never read)
                uint32_t r32[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + TM_AP + 64 * (i & 1) + 32 * hq, r32);
                tmem_wait_ld();
                tc_fence_before();
                const float bt = s.beta(b3)[R];
                const int cend = 16 * (R >> 4) + 16 - 32 * hq;  // first zero column of this half
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float f = 4 * j4 < cend ? bt : 0.f;
                    *reinterpret_cast<float4 *>(tsc + swz(R, 32 * hq + 4 * j4)) =
                        make_float4(f * __uint_as_float(r32[4 * j4]), f * __uint_as_float(r32[4 * j4 + 1]),
                                    f * __uint_as_float(r32[4 * j4 + 2]), f * __uint_as_float(r32[4 * j4 + 3]));
                }
            }
            named_bar(3, SOLVE_THREADS);
            if (work && gw < 2) {
                // T step 1: the four 16x16 diagonal blocks, one thread per column
                // (x_r -= A[r][s] x_s for s < r); rows are compile-time so the A
                // loads take immediate offsets from two base pointers (the
                // swizzle flips bit 4 of the column for rows with r & 7 >= 4).
                const int blk = 2 * gw + (lane >> 4), col = lane & 15;
                const float *rowp = tsc + (16 * blk) * 64;
                const float *b0p = rowp + 16 * blk, *b1p = rowp + ((16 * blk) ^ 16);
                float x[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) x[i2] = i2 == col ? 1.f : 0.f;
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
                __syncwarp();  // the block's A entries are read (its 16 columns are this warp's lanes)
#pragma unroll
                for (int rl = 0; rl < 16; ++rl) tsc[swz(16 * blk + rl, 16 * blk + col)] = x[rl];
            }
            named_bar(3, SOLVE_THREADS);
            // T step 2, two levels of 32-row blocks (tf32 mma.sync, all four warps):
            //   T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22 (one 8-column half each)
            //   T[32:64, 0:32] = -T[32:64, 32:64] (A[32:64, 0:32] T[0:32, 0:32])
            // (the scratch's blocks above the block diagonal are zero; the
            // product A21 T1 is staged in its upper-right quadrant, which the
            // T tile below writes as zeros).
            if (work) {
                // level A: warps gw 0, 1 -> T_10, gw 2, 3 -> T_32; 8-column half nt
                const int I = gw < 2 ? 1 : 3, J = I - 1, nt = gw & 1;
                float *ms = reinterpret_cast<float *>(s.base + SM_MSCR) + gw * 128;  // 16 x 8
                float mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int k8 = 0; k8 < 16; k8 += 8) {
                    const int r0 = 16 * I + g8, cc0 = 16 * J + k8 + t4;
                    const uint32_t af[4] = {to_tf32(tsc[swz(r0, cc0)]), to_tf32(tsc[swz(r0 + 8, cc0)]),
                                            to_tf32(tsc[swz(r0, cc0 + 4)]), to_tf32(tsc[swz(r0 + 8, cc0 + 4)])};
                    const int br = 16 * J + k8 + t4, bc = 16 * J + 8 * nt + g8;
                    mma_tf32(mq, af, to_tf32(tsc[swz(br, bc)]), to_tf32(tsc[swz(br + 4, bc)]));
                }
                ms[g8 * 8 + 2 * t4] = mq[0];
                ms[g8 * 8 + 2 * t4 + 1] = mq[1];
                ms[(g8 + 8) * 8 + 2 * t4] = mq[2];
                ms[(g8 + 8) * 8 + 2 * t4 + 1] = mq[3];
                named_bar(3, SOLVE_THREADS);  // A_10 and A_32 are read: T_10, T_32 go in their place
                float tq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int k8 = 0; k8 < 16; k8 += 8) {
                    const int r0 = 16 * I + g8, cc0 = 16 * I + k8 + t4;
                    const uint32_t af[4] = {to_tf32(tsc[swz(r0, cc0)]), to_tf32(tsc[swz(r0 + 8, cc0)]),
                                            to_tf32(tsc[swz(r0, cc0 + 4)]), to_tf32(tsc[swz(r0 + 8, cc0 + 4)])};
                    mma_tf32(tq, af, to_tf32(ms[(k8 + t4) * 8 + g8]), to_tf32(ms[(k8 + t4 + 4) * 8 + g8]));
                }
                const int c = 16 * J + 8 * nt + 2 * t4;
                tsc[swz(16 * I + g8, c)] = -tq[0];
                tsc[swz(16 * I + g8, c + 1)] = -tq[1];
                tsc[swz(16 * I + g8 + 8, c)] = -tq[2];
                tsc[swz(16 * I + g8 + 8, c + 1)] = -tq[3];
            }
            named_bar(3, SOLVE_THREADS);
            // levels B and C: warp gw owns rows 32 + 16 (gw >> 1) .. +15 and the
            // 8-column tiles 2 (gw & 1), 2 (gw & 1) + 1 of a 32 x 32 result
            const int mt = gw >> 1, ntb = 2 * (gw & 1);
            if (work) {  // level B: M2 = A[32:64, 0:32] T[0:32, 0:32] -> scratch [0:32, 32:64]
                float mq[2][4] = {};
#pragma unroll 1
                for (int k8 = 0; k8 < 32; k8 += 8) {
                    const int r0 = 32 + 16 * mt + g8, cc0 = k8 + t4;
                    const uint32_t af[4] = {to_tf32(tsc[swz(r0, cc0)]), to_tf32(tsc[swz(r0 + 8, cc0)]),
                                            to_tf32(tsc[swz(r0, cc0 + 4)]), to_tf32(tsc[swz(r0 + 8, cc0 + 4)])};
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int bc = 8 * (ntb + u) + g8;
                        mma_tf32(mq[u], af, to_tf32(tsc[swz(k8 + t4, bc)]), to_tf32(tsc[swz(k8 + t4 + 4, bc)]));
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = 16 * mt + g8, c = 32 + 8 * (ntb + u) + 2 * t4;
                    tsc[swz(r, c)] = mq[u][0];
                    tsc[swz(r, c + 1)] = mq[u][1];
                    tsc[swz(r + 8, c)] = mq[u][2];
                    tsc[swz(r + 8, c + 1)] = mq[u][3];
                }
            }
            named_bar(3, SOLVE_THREADS);
            if (work) {  // level C: T[32:64, 0:32] = -T[32:64, 32:64] M2
                float tq[2][4] = {};
#pragma unroll 1
                for (int k8 = 0; k8 < 32; k8 += 8) {
                    const int r0 = 32 + 16 * mt + g8, cc0 = 32 + k8 + t4;
                    const uint32_t af[4] = {to_tf32(tsc[swz(r0, cc0)]), to_tf32(tsc[swz(r0 + 8, cc0)]),
                                            to_tf32(tsc[swz(r0, cc0 + 4)]), to_tf32(tsc[swz(r0 + 8, cc0 + 4)])};
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int bc = 32 + 8 * (ntb + u) + g8;
                        mma_tf32(tq[u], af, to_tf32(tsc[swz(k8 + t4, bc)]), to_tf32(tsc[swz(k8 + t4 + 4, bc)]));
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = 32 + 16 * mt + g8, c = 8 * (ntb + u) + 2 * t4;
                    tsc[swz(r, c)] = -tq[u][0];
                    tsc[swz(r, c + 1)] = -tq[u][1];
                    tsc[swz(r + 8, c)] = -tq[u][2];
                    tsc[swz(r + 8, c + 1)] = -tq[u][3];
                }
            }
            named_bar(3, SOLVE_THREADS);
            // T -> the bf16 operand tile of both CTAs, once MMA2 of the previous
            // chunk completed in both
            if (n >= 1) ok = ok && wait_bar(s, p, B_T_EMPTY + ((n - 1) & 1), ((n - 1) >> 1) & 1);
            const bool wr = __all_sync(0xffffffffu, ok && work);
            if (wr) {
                unsigned char *tpt = s.base + SM_TP;
                const int r = qt >> 1, hc = qt & 1;  // T row r, columns 32hc .. 32hc+31 (exact: unit
                                                     // diagonal, zeros above)
                const bool zero = r < 32 && hc == 1;  // T[0:32, 32:64] = 0 (the scratch holds M2 there)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (!zero) {
                        const float4 x0 = *reinterpret_cast<const float4 *>(tsc + swz(r, 8 * (4 * hc + c4)));
                        const float4 x1 = *reinterpret_cast<const float4 *>(tsc + swz(r, 8 * (4 * hc + c4) + 4));
                        w = make_uint4(pack_bf16(x0.x, x0.y), pack_bf16(x0.z, x0.w), pack_bf16(x1.x, x1.y),
                                       pack_bf16(x1.z, x1.w));
                    }
                    *reinterpret_cast<uint4 *>(tpt + kmajor_chunk(r, 4 * hc + c4, 64)) = w;
                }
                fence_proxy_async();
            }
            const bool pushed = named_bar_or(3, SOLVE_THREADS, wr);
            if (qt == 0) {
                const uint32_t rbar = s.remote(s.bar(B_T_FULL));
                if (pushed) {
                    mbar_arrive_remote_tx(rbar, PUSH_TILE);
                    bulk_s2c(s.remote(s.base + SM_TP), s.base + SM_TP, PUSH_TILE, rbar);
                } else {
                    mbar_arrive_remote_tx(rbar, 0);
                }
                mbar_arrive(s.bar(B_T_FULL));
            }
            alive = ok;
        }
    }

    if (tid == 0 && (s.flags()[1] & 2)) atomicOr(p.err ? p.err : &g_tc_error, 2);  // a wait here timed out
    __syncthreads();  // every thread of this CTA is done: its abort flag is final
    if (tid == 0) st_cluster_u32(s.remote(s.base + SM_FLAGS + 8), (uint32_t)s.flags()[1]);  // the peer's flags[2]
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the other may still write into it
    // After a timeout some groups skipped the waits that would have seen their
    // last copies land (bulk copies into the peer, a v refill). Every thread of
    // both CTAs is past its last copy here, so a pause of some 50 us, far
    // longer than any such copy takes, lets them land before either CTA
    // leaves. Both CTAs take the same decision (either one's abort flag).
    if ((s.flags()[1] | s.flags()[2]) != 0) {
        const long long t0 = clock64();
        while (clock64() - t0 < 100000) {
        }
        cluster_sync();
    }
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
    return (a.dt == KDA_BF16 || a.fp8) && a.dk == DK && a.dv == DV;
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
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    CUtensorMap mk, mq, mv;
    // A map needs a non-empty extent; an empty token range never issues a copy.
    const int64_t ext = tokens > 0 ? tokens : 1;
    // bf16: 128-byte rows with the 128B swizzle the tensor core reads; FP8
    // codes: 64-byte rows (the gate and E1 dequantise them)
    const CUtensorMapDataType et = a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int es = a.fp8 ? 1 : 2;
    // (v codes: 64B swizzle, so that E1's row-per-thread reads hit distinct banks)
    const CUtensorMapSwizzle sw = a.fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapSwizzle swv = a.fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map(&mk, et, es, a.k, DK, a.H, ext, 64, sw) || !make_map(&mq, et, es, a.q, DK, a.H, ext, 64, sw) ||
        !make_map(&mv, et, es, a.v, DV, a.H, ext, 64, swv))
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
    p.slots = a.slots;
    p.gate = a.gate;
    p.qs = a.qs;
    p.ks = a.ks;
    p.vs = a.vs;
    p.N = a.N;
    p.T = a.T;
    p.H = a.H;
    p.stall1 = a.stall1;
    auto pick = [&](auto fp8) {
        constexpr bool F = decltype(fp8)::value;
        return a.gate == KDA_GATE_SCALAR ? kda_prefill_tc_kernel<KDA_GATE_SCALAR, F>
               : a.gate == KDA_GATE_NONE ? kda_prefill_tc_kernel<KDA_GATE_NONE, F>
                                         : kda_prefill_tc_kernel<KDA_GATE_CHANNEL, F>;
    };
    auto kern = a.fp8 ? pick(std::true_type{}) : pick(std::false_type{});
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // blocks is even: one cluster of NSLICE CTAs per (sequence, head)
    kern<<<(unsigned)blocks, NTHREADS, SMEM_BYTES, stream>>>(p, mk, mq, mv);
    return cudaGetLastError();
}

}  // namespace kda
