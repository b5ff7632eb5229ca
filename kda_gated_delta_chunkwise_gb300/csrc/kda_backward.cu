// KDA chunkwise backward (fp32 arithmetic, products on the tensor cores): the
// gradients of L = sum_t <do_t, o_t> + <dS_T, S_T> with respect to q, k, v,
// alpha, beta and the initial state, for equal-length or packed batches and
// every gate kind.
//
// Source of the map: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
// (pwwt.cn), the K3 essay: §四 (the KDA update), §二.1 (the read-out o = S^T q),
// §六.1 (chunks: recursion between chunks) and §六.2 (the WY form). The pages
// give no gradients; the chain rule applied to the chunk algebra below does.
//
// Chunk algebra (as in the forward; C = 64 rows r, j; key channels c; value
// columns v; St = Diag(mu) S the centred start state; the tables of
// kda_chunk_simt.cuh, built here by the tables pass):
//   X = Kr St,  R = Diag(beta) (V - X),  U = T R,  O = Qr St + P U,
//   S_next = Diag(mu) (St + Kc^T U).
// Reverse, with G = dL/dS_next and Gt = Diag(mu) G:
//   dU  = Kc Gt + P^T dO           dR = T^T dU        dX = -Diag(beta) dR
//   dV  = Diag(beta) dR            dbeta_r = sum_v dR (V - X) + sum_j dA Kr Kc^T
//   dSt = Gt + Qr^T dO + Kr^T dX   dS = Diag(mu) dSt  (the state chain)
//   dP  = lower(dO U^T)            dT = dU R^T        dA = strict-lower(-T^T dT T^T)
//   dQr = dO St^T + dP Kc          dKr = dX St^T + Diag(beta) dA Kc
//   dKc = U Gt^T + (Diag(beta) dA)^T Kr + dP^T Qr
//   dq = dQr (.) p/mu,  dk = dKr (.) p/mu + dKc (.) mu/p
// and the gates through logs: d log p_r = dKr Kr + dQr Qr - dKc Kc (per
// channel), d log mu = 2 sum_v Gt St + sum_r [Qr (dO St^T) + Kr (dX St^T) +
// Kc (U Gt^T)] - sum_r d log p_r, d log p_{L-1} += d log mu / 2 (gamma is the
// last row's product), d log alpha_m = sum_{r>=m} d log p_r and
// dalpha = d log alpha / alpha. Chunks that the forward runs token by token
// (a channel decays past e^-80) take the token-level reverse steps instead:
//   G += q do^T; w = G^T k; dv = beta w; dbeta = w.e; dk = beta (G e - S' w);
//   dS' = G - beta k w^T; dalpha = rowsum(dS' (.) S_{t-1}); G = Diag(alpha) dS'
// with S_{t-1} replayed from the chunk's start state.
//
// Four launches:
//   tables one CTA per (sequence, head, chunk), all chunks at once: the
//          chunk's gate products and WY tables (Kr, Qr, Kc, T, P, mu, beta)
//          into the workspace, so no serial pass rebuilds them;
//   states one CTA per (sequence, head, 64-column value slice): the forward
//          state chain, writing the state before every chunk and the chunk's
//          U and V - X;
//   chain  one CTA per (sequence, head, 64-column value slice), chunks in
//          reverse: writes dL/dS after every chunk, the chunk's dU and dR,
//          dv, and the initial state's gradient (it needs no forward state,
//          so it does not wait for the states pass's results);
//   local  one CTA per (sequence, head, chunk), all chunks at once: dq, dk,
//          dalpha, dbeta of the chunk's tokens from the chunk's tables, its
//          states and the four work tiles, each written once (the value
//          columns are taken 32 at a time, double-buffered in shared memory,
//          and the sums over them accumulate in registers), so the result is
//          deterministic.
// The products run on the tensor cores (mma.sync tf32; with a hi/lo split of
// every operand for fp32 inputs: fp32 accuracy).
#include <type_traits>

#include "kda_chunk_simt.cuh"

namespace kda {
namespace {

using simt::C;
using simt::ld_in;
using simt::NT;
using simt::VS;

constexpr int LDC = C + 4;

struct BwdParams {
    const void *q, *k, *v, *d_o;
    const float *alpha, *beta, *dsT;
    float *dq, *dk, *dv, *dalpha, *dbeta, *ds0;
    float *states;        // [N, H, NC, DK, DV]: the state before every chunk
    float *gnext;         // [N, H, NC, DK, DV]: dL/dS after every chunk
    float *tabs;          // [N, H, NC, TabLayout<DK>::FLOATS]: every chunk's tables
    float *work;          // [N, H, NC, 4, C, DV]: U and V - X (states pass), dU and dR (chain pass)
    int gate;             // kda_gate_t: dalpha per channel, per token-head, or none
    int N, T, H, DV, NC;  // T, NC: tokens and chunks of every sequence (equal lengths)
    const int32_t *cu;    // nullable: sequences packed by cu_seqlens [N + 1] (T is then T_total)
    const int32_t *coff;  // packed: first chunk of every sequence [N + 1]
    const int32_t *status;  // packed: nonzero = bad cu_seqlens, nothing runs
};

// Sequence n: first token, length and first chunk. The workspace holds every
// chunk of every sequence at (chunk * H + head).
__device__ __forceinline__ void seq_of(const BwdParams &p, int n, int64_t &t_begin, int64_t &T, int64_t &cbase) {
    if (p.cu) {
        t_begin = p.cu[n];
        T = (int64_t)p.cu[n + 1] - t_begin;
        cbase = p.coff[n];
    } else {
        t_begin = (int64_t)n * p.T;
        T = p.T;
        cbase = (int64_t)n * p.NC;
    }
}
// The workspace slot of a sequence's chunks: slot(ci) = base + ci * stride.
// Equal lengths keep each (sequence, head)'s chunks together ((n H + h) NC +
// ci); packed batches go by chunk, then head (c H + h).
__device__ __forceinline__ void slots_of(const BwdParams &p, int n, int h, int64_t cbase, int64_t &base,
                                         int64_t &stride) {
    if (p.cu) {
        base = cbase * p.H + h;
        stride = p.H;
    } else {
        base = ((int64_t)n * p.H + h) * p.NC;
        stride = 1;
    }
}
// The chunk and head of a CTA of the chunk-parallel passes, in the order of
// the workspace slots (its index is the slot).
__device__ __forceinline__ void cta_chunk(const BwdParams &p, int64_t bid, int64_t &c, int &h) {
    if (p.cu) {
        c = bid / p.H;
        h = (int)(bid % p.H);
    } else {
        const int64_t nh = bid / p.NC;
        h = (int)(nh % p.H);
        c = (nh / p.H) * p.NC + bid % p.NC;
    }
}
// Flat chunk c: its sequence, first token and length; false past the last
// chunk (packed launches are sized by an upper bound).
__device__ __forceinline__ bool chunk_of(const BwdParams &p, int64_t c, int &n, int64_t &tok0, int &L) {
    if (p.cu) {
        if (c >= p.coff[p.N]) return false;
        int lo = 0, hi = p.N - 1;  // the last n with coff[n] <= c (empty sequences own no chunk)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.coff[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        n = lo;
    } else {
        n = (int)(c / p.NC);
    }
    int64_t t_begin, T, cbase;
    seq_of(p, n, t_begin, T, cbase);
    const int64_t t0 = (c - cbase) * C;
    tok0 = t_begin + t0;
    L = (int)((T - t0) < C ? (T - t0) : (int64_t)C);
    return true;
}

// Every chunk's tables, computed once by kda_bwd_tables_kernel (all chunks at
// once) and read by the three passes that follow, so the serial chains do
// not rebuild them: Kr, Qr, Kc [C][DK], T, P [C][C], mu [DK], beta [C], the
// slow flag (its bits in a float), unpadded, in fp32.
template <int DK> struct TabLayout {
    static constexpr int KR = 0, QR = C * DK, KC = 2 * C * DK, T = 3 * C * DK, P = T + C * C, MU = P + C * C,
                         BETA = MU + DK, SLOW = BETA + C, FLOATS = SLOW + 4;
};

// 16 bytes global -> shared without a register round trip (cp.async), so
// that every thread has all its loads of a table in flight at once.
__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}

// 16 bytes global -> shared, or 16 zero bytes when n = 0 (src is then not read).
__device__ __forceinline__ void cp16z(void *dst, const void *src, uint32_t n) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src),
                 "r"(n)
                 : "memory");
}
// A [C][VS] tile of per-token rows (v or dO of value columns v0 ..) into
// shared memory (rows of ld elements), rows past the sequence as zeros;
// cp.async, not committed.
template <typename TIn>
__device__ __forceinline__ void load_rows(TIn *dst, int ld, const TIn *src, int64_t tok0, int L, int H, int h, int DV,
                                          int v0) {
    constexpr int E = 16 / (int)sizeof(TIn), Q = VS / E;  // elements per 16 bytes; 16-byte pieces of a row
    for (int e = threadIdx.x; e < C * Q; e += NT) {
        const int r = e / Q, cc = E * (e % Q);
        cp16z(dst + r * ld + cc, src + ((tok0 + (r < L ? r : 0)) * H + h) * DV + v0 + cc, r < L ? 16u : 0u);
    }
}
// Pulls the rows of such a tile into L2 ahead of their use.
template <typename TIn>
__device__ __forceinline__ void prefetch_rows(const TIn *src, int64_t tok0, int L, int H, int h, int DV, int v0) {
    if ((int)threadIdx.x < L)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src + ((tok0 + threadIdx.x) * H + h) * DV + v0));
}
// Two consecutive elements (the first at an even index) as floats.
__device__ __forceinline__ float2 ld2(const float *x) { return *reinterpret_cast<const float2 *>(x); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16 *x) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(x));
}

// Pulls a chunk's tables into L2 ahead of their use (128-byte lines).
template <int DK> __device__ __forceinline__ void prefetch_tables(const float *src) {
    constexpr int LINES = (TabLayout<DK>::FLOATS * 4 + 127) / 128;
    for (int l = threadIdx.x; l < LINES; l += NT) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 32 * l));
}

// ---- warp-level products on the tensor cores (mma.sync, m16n8k8, tf32) with
// fp32 accuracy: every operand x is split into hi = tf32(x) and lo =
// tf32(x - hi), and a b = a_lo b_hi + a_hi b_lo + a_hi b_hi (the lo lo term is
// below fp32 rounding). Fragment layout (lane = 4 g + t): A rows g, g + 8 and
// columns t, t + 4; B rows t, t + 4 and column g; C rows g, g + 8 and columns
// 2 t, 2 t + 1 of each 16 x 8 tile.
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_bits(x);
    lo = tf32_bits(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc[nt] (the 16 x 8 tile at rows r0.., columns c0 + 8 nt ..) += sum_{k < K} a(r, k) b(k, c)
// SPLIT = false takes one tf32 product per product (for bf16 inputs, whose
// tolerance is that of bf16: about 1e-3 relative instead of fp32's 1e-7).
template <int K, int NT8, bool SPLIT = true, typename FA, typename FB>
__device__ __forceinline__ void wmm(float (&acc)[NT8][4], FA a, FB b, int r0, int c0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 1
    for (int k = 0; k < K; k += 8) {
        uint32_t ah[4], al[4];
        const float av[4] = {a(r0 + g, k + t), a(r0 + g + 8, k + t), a(r0 + g, k + t + 4), a(r0 + g + 8, k + t + 4)};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (SPLIT) split_tf32(av[u], ah[u], al[u]);
            else ah[u] = tf32_bits(av[u]);
        }
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) {
            const float b0 = b(k + t, c0 + 8 * nt + g), b1 = b(k + t + 4, c0 + 8 * nt + g);
            if (SPLIT) {
                uint32_t bh0, bl0, bh1, bl1;
                split_tf32(b0, bh0, bl0);
                split_tf32(b1, bh1, bl1);
                mma8(acc[nt], al, bh0, bh1);
                mma8(acc[nt], ah, bl0, bl1);
                mma8(acc[nt], ah, bh0, bh1);
            } else {
                mma8(acc[nt], ah, tf32_bits(b0), tf32_bits(b1));
            }
        }
    }
}
template <int NT8> __device__ __forceinline__ void fzero(float (&acc)[NT8][4]) {
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
}
// f(r, c, value&) for each accumulator element of the tile at (r0, c0)
template <int NT8, typename F> __device__ __forceinline__ void ffor(float (&acc)[NT8][4], int r0, int c0, F f) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) f(r0 + g + 8 * (e >> 1), c0 + 8 * nt + 2 * t + (e & 1), acc[nt][e]);
}
// The tile at (r0, c0) into row-major global memory of row stride ld, two
// columns per store.
template <int NT8>
__device__ __forceinline__ void gstore(const float (&acc)[NT8][4], int r0, int c0, float *dst, int64_t ld) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int c = c0 + 8 * nt + 2 * t;
        *reinterpret_cast<float2 *>(dst + (int64_t)(r0 + g) * ld + c) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2 *>(dst + (int64_t)(r0 + g + 8) * ld + c) = make_float2(acc[nt][2], acc[nt][3]);
    }
}

// tf32 operands of one m16n8k8 step (hi, and lo when split).
struct BFrag {
    uint32_t h0, h1, l0, l1;
};
template <bool SPLIT> __device__ __forceinline__ BFrag bfrag(float b0, float b1) {
    BFrag f;
    if (SPLIT) {
        split_tf32(b0, f.h0, f.l0);
        split_tf32(b1, f.h1, f.l1);
    } else {
        f.h0 = tf32_bits(b0);
        f.h1 = tf32_bits(b1);
        f.l0 = f.l1 = 0u;
    }
    return f;
}
// A fragment of the 16 x 8 block at rows r0.., columns k.. of a row-major tile.
template <bool SPLIT, typename TS>
__device__ __forceinline__ void afrag(const TS *x, int ld, int r0, int k, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float v[4] = {to_f32(x[(r0 + g) * ld + k + t]), to_f32(x[(r0 + g + 8) * ld + k + t]),
                        to_f32(x[(r0 + g) * ld + k + t + 4]), to_f32(x[(r0 + g + 8) * ld + k + t + 4])};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (SPLIT) split_tf32(v[u], hi[u], lo[u]);
        else hi[u] = tf32_bits(v[u]), lo[u] = 0u;
    }
}
template <bool SPLIT>
__device__ __forceinline__ void mma_f(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], const BFrag &b) {
    if (SPLIT) {
        mma8(d, al, b.h0, b.h1);
        mma8(d, ah, b.l0, b.l1);
    }
    mma8(d, ah, b.h0, b.h1);
}

// Four 8 x 8 b16 matrices from shared memory (ldmatrix); this lane's row
// address is p.
__device__ __forceinline__ void ldsm_x4(const float *p, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
// A fragment of a row-major fp32 tile through ldmatrix (this lane's row address p).
template <bool SPLIT> __device__ __forceinline__ void afrag_ldsm(const float *p, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    uint32_t r[4];
    ldsm_x4(p, r);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float v = __uint_as_float(r[u]);
        if (SPLIT) split_tf32(v, hi[u], lo[u]);
        else hi[u] = tf32_bits(v), lo[u] = 0u;
    }
}

// This lane's row and column offsets of the ldmatrix addresses: of an A
// fragment (rows r0 .. r0 + 15, columns k .. k + 7) and of the B fragments of
// two 8-column tiles stored [n][k] (rows n0 .. n0 + 15, columns k .. k + 7).
__device__ __forceinline__ int ldsm_arow() { return (threadIdx.x & 7) + 8 * ((threadIdx.x >> 3) & 1); }
__device__ __forceinline__ int ldsm_acol() { return 4 * ((threadIdx.x >> 4) & 1); }
__device__ __forceinline__ int ldsm_brow() { return (threadIdx.x & 7) + 8 * ((threadIdx.x >> 4) & 1); }
__device__ __forceinline__ int ldsm_bcol() { return 4 * ((threadIdx.x >> 3) & 1); }

// ---------------------------------------------------------------- tables
// The key channels are taken in two halves of CH = DK / 2, so that the
// shared memory of a CTA (one half of Kr, Qr, Kc, plus A and T: about 88 KB
// for d_k = 128) lets two CTAs share an SM and hide each other's loads. Per
// half, thread (channel cl, segment seg) owns TPS consecutive tokens of one
// channel.
template <int DK> struct GateSplit {
    static constexpr int CH = DK / 2, SEG = NT / CH, TPS = C / SEG, LDH = CH + 4;
};

template <int DK> struct TabSmem {
    float Kr[C * GateSplit<DK>::LDH];  // one half of the channels
    float Qr[C * GateSplit<DK>::LDH];
    float Kc[C * GateSplit<DK>::LDH];
    float A[C * LDC];
    float T[C * LDC];
    float beta[C];
    float part[NT];  // segment products
    int slow;
};

// The gate factors of every row and channel of the chunk, with the arithmetic
// of the tables pass, so the same bits: p / mu (the factor that made Kr and
// Qr) into E2 and mu / p (that of Kc: the later gates over mu) into E3, both
// [C][ld] floats. Needs the chunk's mu ([DK], shared memory); uses part
// ([NT], shared memory) as scratch. Ends with a barrier.
// This thread's gates as gate_factor_table takes them: both halves of the
// channels, every load in flight at once.
template <int DK>
__device__ __forceinline__ void gate_factor_loads(float (&alh)[2][GateSplit<DK>::TPS], const float *alpha, int gate,
                                                  int64_t tok0, int L, int H, int h) {
    using GS = GateSplit<DK>;
    const int tid = threadIdx.x, cl = tid % GS::CH, seg = tid / GS::CH;
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) {
            const int r = seg * GS::TPS + i;
            alh[half][i] = r < L ? gate_at(alpha, gate, (tok0 + r) * H + h, half * GS::CH + cl, DK) : 1.f;
        }
}
template <int DK>
__device__ void gate_factor_table(float *part, const float *mu, float *E2, float *E3, int ld,
                                  const float (&alh)[2][GateSplit<DK>::TPS]) {
    using GS = GateSplit<DK>;
    const int tid = threadIdx.x, cl = tid % GS::CH, seg = tid / GS::CH;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int c = half * GS::CH + cl;
        const float(&al)[GS::TPS] = alh[half];
        float prod = 1.f;
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) prod *= al[i];
        __syncthreads();  // earlier readers of part are done
        part[seg * GS::CH + cl] = prod;
        __syncthreads();
        float before = 1.f, after = 1.f;
#pragma unroll
        for (int s2 = 0; s2 < GS::SEG; ++s2) {
            const float pt = part[s2 * GS::CH + cl];
            if (s2 < seg) before *= pt;
            if (s2 > seg) after *= pt;
        }
        const float inv_mu = 1.f / mu[c];
        float s_acc = after;
#pragma unroll
        for (int i = GS::TPS - 1; i >= 0; --i) {
            E3[(seg * GS::TPS + i) * ld + c] = s_acc * inv_mu;
            s_acc *= al[i];
        }
        float pre = before;
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) {
            pre *= al[i];
            E2[(seg * GS::TPS + i) * ld + c] = pre * inv_mu;
        }
    }
    __syncthreads();
}

// One CTA per (sequence, head, chunk): the chunk's tables into the workspace.
// Per half of the channels: the gate products (p_r running products, gamma,
// mu = sqrt(gamma), the slow flag), Kr = k p / mu, Qr = q p / mu, Kc = k
// (gamma / p) / mu written straight to the workspace and kept in shared
// memory for the half's share of A = Diag(beta) Kr Kc^T and P = Qr Kc^T (tensor
// cores; the sums over both halves stay in registers); then P to the
// workspace, T = (I + A)^{-1}.
template <int DK, typename TIn>
__global__ void __launch_bounds__(NT, 2) kda_bwd_tables_kernel(BwdParams p) {
    using GS = GateSplit<DK>;
    using TL = TabLayout<DK>;
    constexpr bool SPLIT = std::is_same<TIn, float>::value;  // fp32 inputs: fp32 accuracy
    constexpr int LDH = GS::LDH;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TabSmem<DK> &sm = *reinterpret_cast<TabSmem<DK> *>(smem_raw);
    const int64_t idx = blockIdx.x;  // the chunk's workspace slot
    int64_t c0;
    int h, n, L;
    int64_t tok0;
    cta_chunk(p, idx, c0, h);
    if ((p.status && *p.status) || !chunk_of(p, c0, n, tok0, L)) return;
    const int H = p.H;
    const TIn *q = (const TIn *)p.q, *k = (const TIn *)p.k;
    float *dst = p.tabs + idx * TL::FLOATS;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int cl = tid % GS::CH, seg = tid / GS::CH;
    const int R0 = 16 * (warp & 3), C0 = 32 * (warp >> 2);
    // the chunk's rows of alpha, k and q into L2: the second half of the
    // channels is read after the first half's products
    {
        constexpr int LA = DK * 4 / 128, LK = DK * (int)sizeof(TIn) / 128;  // 128-byte lines per row
        const int la = p.gate == KDA_GATE_CHANNEL ? LA : 0, per = la + 2 * LK;
        for (int l = tid; l < L * per; l += NT) {
            const int r = l / per, u = l % per;
            const int64_t th = (tok0 + r) * H + h;
            const void *a = u < la ? (const void *)(p.alpha + th * DK + 32 * u)
                            : u < la + LK ? (const void *)(k + th * DK + (128 / sizeof(TIn)) * (u - la))
                                          : (const void *)(q + th * DK + (128 / sizeof(TIn)) * (u - la - LK));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
    }
    if (tid == 0) sm.slow = 0;
    if (tid < C) sm.beta[tid] = tid < L ? p.beta[(tok0 + tid) * H + h] : 0.f;
    float accA[4][4], accP[4][4];
    fzero<4>(accA);
    fzero<4>(accP);
    for (int half = 0; half < 2; ++half) {
        const int c = half * GS::CH + cl;
        float al[GS::TPS], kk[GS::TPS], qq[GS::TPS];  // every load of the thread in flight at once
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) {
            const int r = seg * GS::TPS + i;
            const int64_t th = (tok0 + r) * H + h;
            const bool in = r < L;
            al[i] = in ? gate_at(p.alpha, p.gate, th, c, DK) : 1.f;
            kk[i] = in ? ld_in(k, th * DK + c) : 0.f;
            qq[i] = in ? ld_in(q, th * DK + c) : 0.f;
        }
        float prod = 1.f;
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) prod *= al[i];
        __syncthreads();  // the previous half's products are done with the tiles
        sm.part[seg * GS::CH + cl] = prod;
        __syncthreads();
        float before = 1.f, after = 1.f, gamma = 1.f;
#pragma unroll
        for (int s2 = 0; s2 < GS::SEG; ++s2) {
            const float pt = sm.part[s2 * GS::CH + cl];
            if (s2 < seg) before *= pt;
            if (s2 > seg) after *= pt;
            gamma *= pt;
        }
        if (gamma < simt::kMinGamma) sm.slow = 1;
        const float mu = sqrtf(gamma), inv_mu = 1.f / mu;
        if (seg == 0) dst[TL::MU + c] = mu;
        // Kc from the exclusive suffix products (within the segment, times the
        // later segments), last row first; then Kr, Qr from the prefix products
        float s_acc = after;
#pragma unroll
        for (int i = GS::TPS - 1; i >= 0; --i) {
            const int r = seg * GS::TPS + i;
            const float kc = kk[i] * (s_acc * inv_mu);
            s_acc *= al[i];
            sm.Kc[r * LDH + cl] = kc;
            dst[TL::KC + r * DK + c] = kc;
        }
        float pre = before;
#pragma unroll
        for (int i = 0; i < GS::TPS; ++i) {
            const int r = seg * GS::TPS + i;
            pre *= al[i];
            const float e2 = pre * inv_mu;
            const float kr = kk[i] * e2, qr = qq[i] * e2;
            sm.Kr[r * LDH + cl] = kr;
            sm.Qr[r * LDH + cl] = qr;
            dst[TL::KR + r * DK + c] = kr;
            dst[TL::QR + r * DK + c] = qr;
        }
        __syncthreads();
        // this half's share of [A; P] = [Kr; Qr] Kc^T (the two share the Kc fragments)
#pragma unroll 2
        for (int kx = 0; kx < GS::CH; kx += 8) {
            uint32_t kh[4], kl[4], qh[4], ql[4];
            const int ao = (R0 + ldsm_arow()) * LDH + kx + ldsm_acol();
            afrag_ldsm<SPLIT>(sm.Kr + ao, kh, kl);
            afrag_ldsm<SPLIT>(sm.Qr + ao, qh, ql);
#pragma unroll
            for (int np = 0; np < 2; ++np) {  // two 8-column tiles of Kc^T per load
                uint32_t k4[4];
                ldsm_x4(sm.Kc + (C0 + 16 * np + ldsm_brow()) * LDH + kx + ldsm_bcol(), k4);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const BFrag b = bfrag<SPLIT>(__uint_as_float(k4[2 * u]), __uint_as_float(k4[2 * u + 1]));
                    mma_f<SPLIT>(accA[2 * np + u], kh, kl, b);
                    mma_f<SPLIT>(accP[2 * np + u], qh, ql, b);
                }
            }
        }
    }
    if (tid < C) dst[TL::BETA + tid] = sm.beta[tid];
    const int slow = sm.slow;  // (set before the last barrier)
    if (tid == 0) dst[TL::SLOW] = __int_as_float(slow);
    if (slow) return;  // the chunk runs token by token: no T or P
    ffor<4>(accA, R0, C0, [&](int r, int j, float &x) { sm.A[r * LDC + j] = j < r ? sm.beta[r] * x : 0.f; });
    ffor<4>(accP, R0, C0, [&](int r, int j, float &x) { x = j <= r ? x : 0.f; });
    gstore<4>(accP, R0, C0, dst + TL::P, C);
    __syncthreads();
    simt::invert_unit_lower(simt::TPair{sm.A, sm.T});
    for (int e = tid; e < C * C / 4; e += NT) {
        const int r = e / (C / 4), cc = 4 * (e % (C / 4));
        *reinterpret_cast<float4 *>(dst + TL::T + r * C + cc) = *reinterpret_cast<const float4 *>(&sm.T[r * LDC + cc]);
    }
}

// ---------------------------------------------------------------- chains
// The two serial passes keep every tile in shared memory with a row stride
// picked for the way the mma fragments read it: = 4 (mod 32) floats for a
// tile read along its rows (A operands, row-major; B operands stored
// [n][k]), = 8 (mod 32) for a tile read down its columns (transposed A
// operands; B operands stored [k][n]; accumulator tiles written two columns
// at a time). Either way the 32 lanes of a fragment load hit 32 banks.
constexpr int LR = C + 4;   // a [C][C] tile read along rows
constexpr int LS = VS + 8;  // a [rows][VS] value tile read down its columns / written as accumulators
template <int DK> struct Ld {
    static constexpr int ROW = DK + 4, COL = DK + 8;  // [C][DK] tiles read along rows / down columns
};
// dO or v tile (qkv type) read down its columns: 16-byte rows, conflict-free.
template <typename TIn> struct ColTile { static constexpr int LD = sizeof(TIn) == 4 ? VS + 8 : VS + 16; };

// cp.async of a [rows][cols] fp32 tile (cols a multiple of 4) from rows of
// sld floats into shared rows of ld floats; not committed.
__device__ __forceinline__ void cp_tile(float *dst, int ld, const float *src, int sld, int rows, int cols) {
    const int q4 = cols / 4;
    for (int e = threadIdx.x; e < rows * q4; e += NT) {
        const int r = e / q4, c = 4 * (e % q4);
        cp16(dst + r * ld + c, src + (int64_t)r * sld + c);
    }
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed cp.async groups are pending.
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A fragment of a transposed operand: A(m, k) = x[k][m].
template <bool SPLIT, typename TS>
__device__ __forceinline__ void afragT(const TS *x, int ld, int r0, int k, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float v[4] = {to_f32(x[(k + t) * ld + r0 + g]), to_f32(x[(k + t) * ld + r0 + g + 8]),
                        to_f32(x[(k + t + 4) * ld + r0 + g]), to_f32(x[(k + t + 4) * ld + r0 + g + 8])};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (SPLIT) split_tf32(v[u], hi[u], lo[u]);
        else hi[u] = tf32_bits(v[u]), lo[u] = 0u;
    }
}
// acc[nt] += A B over K for the warp tile at (r0, c0): A from fa(k, hi, lo)
// (a fragment loader), B(k, n) = x[k][n] times the row factor f[k] (or 1
// when f is null). Even and odd k-steps go to two accumulator sets (summed at
// the end), so twice as many products are in flight.
template <int K, int NT8, bool SPLIT, typename FA, typename TS>
__device__ __forceinline__ void mm_kn(float (&acc)[NT8][4], FA fa, const TS *x, int ld, const float *f, int r0, int c0) {
    static_assert(K % 16 == 0, "K in steps of 16");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float acc2[NT8][4];
    fzero<NT8>(acc2);
    auto step = [&](int k, float(&d)[NT8][4]) {
        uint32_t ah[4], al[4];
        fa(k, ah, al);
        const float f0 = f ? f[k + t] : 1.f, f1 = f ? f[k + t + 4] : 1.f;
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) {
            const int n = c0 + 8 * nt + g;
            const BFrag b = bfrag<SPLIT>(f0 * to_f32(x[(k + t) * ld + n]), f1 * to_f32(x[(k + t + 4) * ld + n]));
            mma_f<SPLIT>(d[nt], ah, al, b);
        }
    };
#pragma unroll 1
    for (int k = 0; k < K; k += 16) {
        step(k, acc);
        step(k + 8, acc2);
    }
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
}
// Accumulator tile (r0, c0) into shared rows of ld floats, two columns per store.
template <int NT8> __device__ __forceinline__ void sstore(const float (&acc)[NT8][4], int r0, int c0, float *dst, int ld) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int c = c0 + 8 * nt + 2 * t;
        *reinterpret_cast<float2 *>(dst + (r0 + g) * ld + c) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2 *>(dst + (r0 + g + 8) * ld + c) = make_float2(acc[nt][2], acc[nt][3]);
    }
}
// x[r][c] <- mu[r] (mu[r] x[r][c] + acc) for the accumulator tile (r0, c0) of
// shared rows of ld floats: the state and state-gradient updates.
template <int NT8>
__device__ __forceinline__ void state_update(const float (&acc)[NT8][4], int r0, int c0, float *x, int ld, const float *mu) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float m0 = mu[r0 + g], m1 = mu[r0 + g + 8];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int c = c0 + 8 * nt + 2 * t;
        float2 *a = reinterpret_cast<float2 *>(x + (r0 + g) * ld + c), *b = reinterpret_cast<float2 *>(x + (r0 + g + 8) * ld + c);
        float2 va = *a, vb = *b;
        va.x = m0 * (m0 * va.x + acc[nt][0]);
        va.y = m0 * (m0 * va.y + acc[nt][1]);
        vb.x = m1 * (m1 * vb.x + acc[nt][2]);
        vb.y = m1 * (m1 * vb.y + acc[nt][3]);
        *a = va;
        *b = vb;
    }
}

// A rows x VS fp32 slice from shared rows of LS floats to global rows of DV
// floats, and back (zeros for a null source); 16-byte moves.
__device__ __forceinline__ void slice_store(float *g, const float *s, int rows, int DV) {
    for (int e = threadIdx.x; e < rows * (VS / 4); e += NT) {
        const int r = e / (VS / 4), c = 4 * (e % (VS / 4));
        *reinterpret_cast<float4 *>(g + (int64_t)r * DV + c) = *reinterpret_cast<const float4 *>(s + r * LS + c);
    }
}
__device__ __forceinline__ void slice_load(float *s, const float *g, int rows, int DV) {
    for (int e = threadIdx.x; e < rows * (VS / 4); e += NT) {
        const int r = e / (VS / 4), c = 4 * (e % (VS / 4));
        *reinterpret_cast<float4 *>(s + r * LS + c) =
            g ? *reinterpret_cast<const float4 *>(g + (int64_t)r * DV + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Warp tiles of a DK x 64 product (the state slice): DK = 128 gives each warp
// 16 rows and all 64 columns, DK = 64 16 rows and 32 columns.
template <int DK> struct StateTile {
    static constexpr int N8 = DK == 128 ? 8 : 4;
    __device__ static int r0(int warp) { return 16 * (DK == 128 ? warp : (warp & 3)); }
    __device__ static int c0(int warp) { return DK == 128 ? 0 : 32 * (warp >> 2); }
};

// The per-chunk scalars of a chain step (double-buffered with its token tile).
template <int DK> struct ChunkScalars {
    float mu[DK];
    float beta[C];
    float flag[4];  // [0]: the slow flag's bits
};
// Issues the cp.async of a chunk's mu, beta and slow flag (not committed).
template <int DK> __device__ __forceinline__ void cp_scalars(ChunkScalars<DK> &d, const float *tab) {
    using TL = TabLayout<DK>;
    const int tid = threadIdx.x;
    if (tid < DK / 4) cp16(&d.mu[4 * tid], tab + TL::MU + 4 * tid);
    else if (tid < DK / 4 + C / 4) cp16(&d.beta[4 * (tid - DK / 4)], tab + TL::BETA + 4 * (tid - DK / 4));
    else if (tid == DK / 4 + C / 4) cp16(d.flag, tab + TL::SLOW);
}

// ---------------------------------------------------------------- states
// The forward chain only: one CTA per (sequence, head, value slice) writes the
// state before every chunk (S_{n+1} = Diag(mu) (Diag(mu) S_n + Kc^T U), U =
// T Diag(beta) (V - Kr Diag(mu) S_n)) and the chunk's U and V - X, reading the
// chunk's tables; slow chunks go token by token (the §四 update) and write no
// U or V - X. Products on the tensor cores. Each table of the next chunk is
// copied in (cp.async) as soon as this chunk is done with it, so the copies
// run under this chunk's products: Kr after X, T after U, Kc after the state
// update; mu, beta, the flag and v are double-buffered.
template <int DK, typename TIn> struct StatesSmem {
    float S[DK * LS];  // the state slice
    float Kr[C * Ld<DK>::ROW];
    float Kc[C * Ld<DK>::COL];
    float T[C * LR];
    float R[C * LS];
    float U[C * LS];
    TIn V[2][C * ColTile<TIn>::LD];
    ChunkScalars<DK> sc[2];
};

// 16-byte offsets for cp.async (every tile and row is a multiple of 16 bytes)
template <int DK, typename TIn> constexpr bool states_layout_ok() {
    using S = StatesSmem<DK, TIn>;
    return offsetof(S, Kr) % 16 == 0 && offsetof(S, Kc) % 16 == 0 && offsetof(S, T) % 16 == 0 &&
           offsetof(S, R) % 16 == 0 && offsetof(S, U) % 16 == 0 && offsetof(S, V) % 16 == 0 &&
           offsetof(S, sc) % 16 == 0 && sizeof(ChunkScalars<DK>) % 16 == 0 && (C * ColTile<TIn>::LD * sizeof(TIn)) % 16 == 0;
}
static_assert(states_layout_ok<128, float>() && states_layout_ok<128, __nv_bfloat16>() && states_layout_ok<64, float>() &&
                  states_layout_ok<64, __nv_bfloat16>(),
              "16-byte offsets");

template <int DK, typename TIn>
__global__ void __launch_bounds__(NT, 1) kda_bwd_states_kernel(BwdParams p, const float *s0) {
    constexpr bool SPLIT = std::is_same<TIn, float>::value;  // fp32 inputs: fp32 accuracy
    using TL = TabLayout<DK>;
    using ST = StateTile<DK>;
    constexpr int LKR = Ld<DK>::ROW, LKC = Ld<DK>::COL, LV = ColTile<TIn>::LD;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StatesSmem<DK, TIn> &sm = *reinterpret_cast<StatesSmem<DK, TIn> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nslices = p.DV / VS;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % p.H;
    const int n = blockIdx.x / (nslices * p.H);
    const int H = p.H, DV = p.DV, v0 = slice * VS;
    if (p.status && *p.status) return;
    int64_t t_begin, T, cbase;
    seq_of(p, n, t_begin, T, cbase);
    const int NC = (int)((T + C - 1) / C);
    const int64_t sh = (int64_t)n * H + h;
    const TIn *k = (const TIn *)p.k, *v = (const TIn *)p.v;
    int64_t wbase, wstride;
    slots_of(p, n, h, cbase, wbase, wstride);
    float *st = p.states + wbase * DK * DV;  // chunk i at slot wbase + i wstride
    float *wkb = p.work + wbase * 4 * C * DV;
    const float *tabs = p.tabs + wbase * TL::FLOATS;
    auto tab = [&](int i) { return tabs + (int64_t)i * wstride * TL::FLOATS; };
    auto len = [&](int i) { return (int)((T - (int64_t)i * C) < C ? (T - (int64_t)i * C) : (int64_t)C); };
    const int R0 = 16 * (warp & 3), C0 = 32 * (warp >> 2);
    const int SR0 = ST::r0(warp), SC0 = ST::c0(warp);
    // chunk i's copies, in three groups: (scalars, v, Kr), (T), (Kc)
    auto issue_a = [&](int i) {
        if (i < NC) {
            cp_scalars<DK>(sm.sc[i & 1], tab(i));
            load_rows<TIn>(sm.V[i & 1], LV, v, t_begin + (int64_t)i * C, len(i), H, h, DV, v0);
            cp_tile(sm.Kr, LKR, tab(i) + TL::KR, DK, C, DK);
        }
        cp_commit();
    };
    auto issue_b = [&](int i) {
        if (i < NC) cp_tile(sm.T, LR, tab(i) + TL::T, C, C, C);
        cp_commit();
    };
    auto issue_c = [&](int i) {
        if (i < NC) cp_tile(sm.Kc, LKC, tab(i) + TL::KC, DK, C, DK);
        cp_commit();
    };
    slice_load(sm.S, s0 ? s0 + sh * DK * DV + v0 : nullptr, DK, DV);
    issue_a(0);
    issue_b(0);
    issue_c(0);
    for (int ci = 0; ci < NC; ++ci) {
        const int64_t t0 = (int64_t)ci * C, tok0 = t_begin + t0;
        const int L = len(ci);
        ChunkScalars<DK> &cs = sm.sc[ci & 1];
        const TIn *Vt = sm.V[ci & 1];
        cp_wait<1>();  // this chunk's scalars, v, Kr and T (Kc may still be on its way)
        __syncthreads();
        slice_store(st + ci * wstride * DK * DV + v0, sm.S, DK, DV);
        if (ci + 2 < NC) {  // two chunks ahead into L2
            prefetch_tables<DK>(tab(ci + 2));
            prefetch_rows<TIn>(v, tok0 + 2 * C, len(ci + 2), H, h, DV, v0);
        }
        if (__float_as_int(cs.flag[0])) {
            const int j = tid % VS, part = tid / VS;
            for (int r = 0; r < L; ++r) {
                const int64_t tk = (tok0 + r) * H + h;
                float vh = 0.f;
                for (int c = part; c < DK; c += NT / VS)
                    vh += gate_at(p.alpha, p.gate, tk, c, DK) * ld_in(k, tk * DK + c) * sm.S[c * LS + j];
                sm.R[part * LS + j] = vh;
                __syncthreads();
                float vs = 0.f;
#pragma unroll
                for (int p2 = 0; p2 < NT / VS; ++p2) vs += sm.R[p2 * LS + j];
                const float be = p.beta[tk] * (ld_in(v, tk * DV + v0 + j) - vs);
                __syncthreads();
                for (int c = part; c < DK; c += NT / VS)
                    sm.S[c * LS + j] = gate_at(p.alpha, p.gate, tk, c, DK) * sm.S[c * LS + j] + ld_in(k, tk * DK + c) * be;
                __syncthreads();
            }
            cp_wait<0>();  // nothing of this chunk's copies is in flight before the slots are refilled
            __syncthreads();
            issue_a(ci + 1);
            issue_b(ci + 1);
            issue_c(ci + 1);
            continue;
        }
        float *wk = wkb + ci * wstride * 4 * C * DV + v0;  // this chunk's U, V - X (the slice's columns)
        float acc[4][4];
        // X = Kr St (St = Diag(mu) S); V - X into the workspace; R = Diag(beta) (V - X)
        fzero<4>(acc);
        mm_kn<DK, 4, SPLIT>(acc, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afrag_ldsm<SPLIT>(sm.Kr + (R0 + ldsm_arow()) * LKR + kx + ldsm_acol(), hi, lo); },
                            sm.S, LS, cs.mu, R0, C0);
        {  // V - X, two columns per load
            const int lane = tid & 31, g = lane >> 2, t4 = lane & 3;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float2 vv = ld2(Vt + (R0 + g + 8 * u) * LV + C0 + 8 * nt + 2 * t4);
                    acc[nt][2 * u] = vv.x - acc[nt][2 * u];
                    acc[nt][2 * u + 1] = vv.y - acc[nt][2 * u + 1];
                }
        }
        gstore<4>(acc, R0, C0, wk + C * DV, DV);
        ffor<4>(acc, R0, C0, [&](int r, int c, float &x) { x *= cs.beta[r]; });
        sstore<4>(acc, R0, C0, sm.R, LS);
        __syncthreads();
        issue_a(ci + 1);  // Kr is free
        // U = T R, also into the workspace
        fzero<4>(acc);
        mm_kn<C, 4, SPLIT>(acc, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afrag_ldsm<SPLIT>(sm.T + (R0 + ldsm_arow()) * LR + kx + ldsm_acol(), hi, lo); },
                           sm.R, LS, (const float *)nullptr, R0, C0);
        sstore<4>(acc, R0, C0, sm.U, LS);
        gstore<4>(acc, R0, C0, wk, DV);
        cp_wait<1>();  // Kc (the group of the next chunk's scalars, v and Kr may be pending)
        __syncthreads();
        issue_b(ci + 1);  // T is free
        // S <- Diag(mu) (Diag(mu) S + Kc^T U)
        float acc2[ST::N8][4];
        fzero<ST::N8>(acc2);
        mm_kn<C, ST::N8, SPLIT>(acc2, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afragT<SPLIT>(sm.Kc, LKC, SR0, kx, hi, lo); },
                                sm.U, LS, (const float *)nullptr, SR0, SC0);
        state_update<ST::N8>(acc2, SR0, SC0, sm.S, LS, cs.mu);
        __syncthreads();
        issue_c(ci + 1);  // Kc is free
    }
    cp_wait<0>();
}

// ---------------------------------------------------------------- chain
// The reverse chain: one CTA per (sequence, head, value slice), chunks last to
// first; writes dL/dS after every chunk, the chunk's dU and dR, dv, and dS_0.
// The next chunk's tables are copied in as this chunk frees them: Kc and P
// after dU, T after dR, Qr and Kr after the state-gradient update; mu, beta
// and the flag are double-buffered, and so is dO for bf16 inputs (for fp32
// inputs a second fp32 dO tile does not fit: it comes with Qr and Kr).
template <typename TIn> struct ChainDo { static constexpr int BUFS = sizeof(TIn) == 4 ? 1 : 2; };
template <int DK, typename TIn> struct ChainSmem {
    float G[DK * LS];  // dL/dS slice
    float Kc[C * Ld<DK>::ROW];
    float P[C * LS];   // read transposed
    float T[C * LS];   // read transposed
    float dU[C * LS];
    float Qr[C * Ld<DK>::COL];
    float Kr[C * Ld<DK>::COL];
    TIn dO[ChainDo<TIn>::BUFS][C * ColTile<TIn>::LD];
    ChunkScalars<DK> sc[2];
    float red[4 * VS];
};

template <int DK, typename TIn> constexpr bool chain_layout_ok() {
    using S = ChainSmem<DK, TIn>;
    return offsetof(S, Kc) % 16 == 0 && offsetof(S, P) % 16 == 0 && offsetof(S, T) % 16 == 0 &&
           offsetof(S, dU) % 16 == 0 && offsetof(S, Qr) % 16 == 0 && offsetof(S, Kr) % 16 == 0 &&
           offsetof(S, dO) % 16 == 0 && offsetof(S, sc) % 16 == 0;
}
static_assert(chain_layout_ok<128, float>() && chain_layout_ok<128, __nv_bfloat16>() && chain_layout_ok<64, float>() &&
                  chain_layout_ok<64, __nv_bfloat16>(),
              "16-byte offsets");

template <int DK, typename TIn>
__global__ void __launch_bounds__(NT, 1) kda_bwd_chain_kernel(BwdParams p) {
    constexpr bool SPLIT = std::is_same<TIn, float>::value;  // fp32 inputs: fp32 accuracy
    using TL = TabLayout<DK>;
    using ST = StateTile<DK>;
    constexpr int LKR = Ld<DK>::ROW, LQK = Ld<DK>::COL, LD = ColTile<TIn>::LD, LP = LS;
    constexpr bool DB = ChainDo<TIn>::BUFS == 2;  // dO double-buffered
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ChainSmem<DK, TIn> &sm = *reinterpret_cast<ChainSmem<DK, TIn> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nslices = p.DV / VS;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % p.H;
    const int n = blockIdx.x / (nslices * p.H);
    const int H = p.H, DV = p.DV, v0 = slice * VS;
    if (p.status && *p.status) return;
    int64_t t_begin, T, cbase;
    seq_of(p, n, t_begin, T, cbase);
    const int NC = (int)((T + C - 1) / C);
    const TIn *q = (const TIn *)p.q, *k = (const TIn *)p.k, *dO = (const TIn *)p.d_o;
    const int64_t sh = (int64_t)n * H + h;
    int64_t wbase, wstride;
    slots_of(p, n, h, cbase, wbase, wstride);
    float *gn = p.gnext + wbase * DK * DV;  // chunk i at slot wbase + i wstride
    float *wkb = p.work + wbase * 4 * C * DV;
    const float *tabs = p.tabs + wbase * TL::FLOATS;
    auto tab = [&](int i) { return tabs + (int64_t)i * wstride * TL::FLOATS; };
    auto len = [&](int i) { return (int)((T - (int64_t)i * C) < C ? (T - (int64_t)i * C) : (int64_t)C); };
    const int R0 = 16 * (warp & 3), C0 = 32 * (warp >> 2);
    const int SR0 = ST::r0(warp), SC0 = ST::c0(warp);
    // chunk i's copies, in three groups: (scalars, dO, Kc, P), (T), (Qr, Kr)
    // (a single dO tile comes with Qr and Kr)
    auto issue_a = [&](int i) {
        if (i >= 0) {
            cp_scalars<DK>(sm.sc[i & 1], tab(i));
            if (DB) load_rows<TIn>(sm.dO[i & 1], LD, dO, t_begin + (int64_t)i * C, len(i), H, h, DV, v0);
            cp_tile(sm.Kc, LKR, tab(i) + TL::KC, DK, C, DK);
            cp_tile(sm.P, LP, tab(i) + TL::P, C, C, C);
        }
        cp_commit();
    };
    auto issue_b = [&](int i) {
        if (i >= 0) cp_tile(sm.T, LS, tab(i) + TL::T, C, C, C);
        cp_commit();
    };
    auto issue_c = [&](int i) {
        if (i >= 0) {
            cp_tile(sm.Qr, LQK, tab(i) + TL::QR, DK, C, DK);
            cp_tile(sm.Kr, LQK, tab(i) + TL::KR, DK, C, DK);
            if (!DB) load_rows<TIn>(sm.dO[0], LD, dO, t_begin + (int64_t)i * C, len(i), H, h, DV, v0);
        }
        cp_commit();
    };

    slice_load(sm.G, p.dsT ? p.dsT + sh * DK * DV + v0 : nullptr, DK, DV);
    issue_a(NC - 1);
    issue_b(NC - 1);
    issue_c(NC - 1);

    for (int ci = NC - 1; ci >= 0; --ci) {
        const int64_t t0 = (int64_t)ci * C;
        const int L = len(ci);
        const int64_t tok0 = t_begin + t0;
        ChunkScalars<DK> &cs = sm.sc[ci & 1];
        const TIn *dOt = sm.dO[DB ? (ci & 1) : 0];
        if (DB) cp_wait<2>();  // this chunk's scalars, dO, Kc and P (T, Qr and Kr may still be on their way)
        else cp_wait<0>();
        __syncthreads();
        slice_store(gn + ci * wstride * DK * DV + v0, sm.G, DK, DV);  // dL/dS after this chunk
        if (ci >= 2) {  // two chunks ahead into L2
            prefetch_tables<DK>(tab(ci - 2));
            prefetch_rows<TIn>(dO, tok0 - 2 * C, C, H, h, DV, v0);
        }
        if (__float_as_int(cs.flag[0])) {
            // token by token, last token first: G += q do^T; w = G^T k; G = Diag(alpha)(G - beta k w^T)
            const int j = tid % VS, part = tid / VS;
            for (int r = L - 1; r >= 0; --r) {
                const int64_t tk = (tok0 + r) * H + h;
                const float dj = to_f32(dOt[r * LD + j]);
                float wp = 0.f;
                for (int c = part; c < DK; c += NT / VS) {
                    const float g = sm.G[c * LS + j] + ld_in(q, tk * DK + c) * dj;
                    sm.G[c * LS + j] = g;
                    wp += ld_in(k, tk * DK + c) * g;
                }
                sm.red[part * VS + j] = wp;
                __syncthreads();
                float w = 0.f;
#pragma unroll
                for (int p2 = 0; p2 < NT / VS; ++p2) w += sm.red[p2 * VS + j];
                const float bt = p.beta[tk];
                for (int c = part; c < DK; c += NT / VS)
                    sm.G[c * LS + j] = gate_at(p.alpha, p.gate, tk, c, DK) * (sm.G[c * LS + j] - bt * ld_in(k, tk * DK + c) * w);
                __syncthreads();
            }
            cp_wait<0>();  // nothing of this chunk's copies is in flight before the slots are refilled
            __syncthreads();
            issue_a(ci - 1);
            issue_b(ci - 1);
            issue_c(ci - 1);
            continue;
        }
        float *wk = wkb + ci * wstride * 4 * C * DV + v0;  // this chunk's dU, dR (the slice's columns)
        float acc[4][4];
        // dU = Kc Gt + P^T dO (Gt = Diag(mu) G), also into the workspace
        fzero<4>(acc);
        mm_kn<DK, 4, SPLIT>(acc, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afrag_ldsm<SPLIT>(sm.Kc + (R0 + ldsm_arow()) * LKR + kx + ldsm_acol(), hi, lo); },
                            sm.G, LS, cs.mu, R0, C0);
        mm_kn<C, 4, SPLIT>(acc, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afragT<SPLIT>(sm.P, LP, R0, kx, hi, lo); },
                           dOt, LD, (const float *)nullptr, R0, C0);
        sstore<4>(acc, R0, C0, sm.dU, LS);
        gstore<4>(acc, R0, C0, wk + 2 * C * DV, DV);
        cp_wait<1>();  // T (the group of Qr and Kr may be pending)
        __syncthreads();
        issue_a(ci - 1);  // Kc and P are free
        // dR = T^T dU into the workspace; dv = Diag(beta) dR; dX = -Diag(beta) dR (into dU's place)
        fzero<4>(acc);
        mm_kn<C, 4, SPLIT>(acc, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afragT<SPLIT>(sm.T, LS, R0, kx, hi, lo); },
                           sm.dU, LS, (const float *)nullptr, R0, C0);
        gstore<4>(acc, R0, C0, wk + 3 * C * DV, DV);
        {  // dv = Diag(beta) dR (two columns per store), then dX = -Diag(beta) dR
            const int lane = tid & 31, g = lane >> 2, t4 = lane & 3;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = R0 + g + 8 * u;
                const float br = cs.beta[r];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    float &x0 = acc[nt][2 * u], &x1 = acc[nt][2 * u + 1];
                    if (r < L)
                        *reinterpret_cast<float2 *>(p.dv + ((tok0 + r) * H + h) * DV + v0 + C0 + 8 * nt + 2 * t4) =
                            make_float2(br * x0, br * x1);
                    x0 *= -br;
                    x1 *= -br;
                }
            }
        }
        cp_wait<1>();  // Qr and Kr (the next chunk's first group may be pending)
        __syncthreads();  // every read of dU is done; Qr and Kr have landed
        sstore<4>(acc, R0, C0, sm.dU, LS);
        issue_b(ci - 1);  // T is free
        __syncthreads();
        // G <- Diag(mu) (Gt + Qr^T dO + Kr^T dX)
        float acc2[ST::N8][4];
        fzero<ST::N8>(acc2);
        mm_kn<C, ST::N8, SPLIT>(acc2, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afragT<SPLIT>(sm.Qr, LQK, SR0, kx, hi, lo); },
                                dOt, LD, (const float *)nullptr, SR0, SC0);
        mm_kn<C, ST::N8, SPLIT>(acc2, [&](int kx, uint32_t(&hi)[4], uint32_t(&lo)[4]) { afragT<SPLIT>(sm.Kr, LQK, SR0, kx, hi, lo); },
                                sm.dU, LS, (const float *)nullptr, SR0, SC0);
        state_update<ST::N8>(acc2, SR0, SC0, sm.G, LS, cs.mu);
        __syncthreads();
        issue_c(ci - 1);  // Qr and Kr are free
    }
    cp_wait<0>();
    __syncthreads();
    if (p.ds0)
        slice_store(p.ds0 + sh * DK * DV + v0, sm.G, DK, DV);
}

// ---------------------------------------------------------------- local
constexpr int VP = 32;       // value columns per piece of the local pass
constexpr int LDP = VP + 4;  // padded row of a piece tile (fp32): conflict-free fragments
// padded row of the dO tile (elements): 16-byte rows, conflict-free fragments
template <typename TIn> struct DoRow { static constexpr int LD = sizeof(TIn) == 4 ? LDP : VP + 8; };

// One piece of value columns [v0, v0 + VP) of everything the local pass sums
// over the value columns.
template <int DK, typename TIn> struct LocalPiece {
    float S[DK * LDP];  // the state before the chunk (rows: key channels)
    float G[DK * LDP];  // dL/dS after the chunk
    float U[C * LDP];
    float VmX[C * LDP];  // V - X
    float dU[C * LDP];
    float dR[C * LDP];
    TIn dO[C * DoRow<TIn>::LD];
};
// What the last part of the local pass reads, in the pieces' place.
template <int DK> struct LocalFinal {
    float Kr[C * (DK + 8)];
    float Qr[C * (DK + 8)];
    float W[4][C * LS];  // work tiles: rows of LDC floats when read along rows, LS when read down columns
};
// The token path's buffers (local_slow), in the pieces' place.
template <int DK> constexpr int slow_floats() { return 2 * DK * 128 + 2 * NT + 2 * 128 + 4 * NT + DK; }

template <int DK, typename TIn> struct LocalSmem {
    union Front {
        LocalPiece<DK, TIn> piece[2];  // double-buffered pieces
        LocalFinal<DK> fin;
        float slow[slow_floats<DK>()];
    } u;
    float Kc[C * (DK + 8)];
    float T[C * LDC];
    float mu[DK];
    float beta[C];
    float part[(NT / DK) * DK];
    float red[8 * DK + 3 * C];  // column sums by row block; dbeta parts by row
};

// 16-byte tiles and offsets (cp.async and float4 accesses)
template <int DK, typename TIn> constexpr bool local_layout_ok() {
    using P = LocalPiece<DK, TIn>;
    using S = LocalSmem<DK, TIn>;
    return sizeof(P) % 16 == 0 && offsetof(P, dO) % 16 == 0 && offsetof(P, U) % 16 == 0 && offsetof(S, Kc) % 16 == 0 &&
           offsetof(S, T) % 16 == 0 && offsetof(S, mu) % 16 == 0 && offsetof(S, beta) % 16 == 0 &&
           offsetof(LocalFinal<DK>, Qr) % 16 == 0 && offsetof(LocalFinal<DK>, W) % 16 == 0;
}
static_assert(local_layout_ok<128, float>() && local_layout_ok<128, __nv_bfloat16>() && local_layout_ok<64, float>() &&
                  local_layout_ok<64, __nv_bfloat16>(),
              "16-byte tiles and offsets");

// The local pass of a chunk that the forward runs token by token (a channel
// decays past e^-80), in `buf` (slow_floats<DK>() floats of shared memory).
template <int DK, typename TIn, int GATE>
__device__ __noinline__ void local_slow(float *buf, const BwdParams &p, const float *Sg, const float *Gg, int64_t tok0,
                                        int L, int h) {
    // Token-level reverse steps over every value column; the state before
    // token r is replayed from the chunk's start state for every r (the chunk
    // is rare: this is written for size).
    const int H = p.H, DV = p.DV, tid = threadIdx.x;
    const int NP = NT / DV;      // key-row parts of the column mapping
    constexpr int NH = NT / DK;  // column parts of the row mapping
    const TIn *q = (const TIn *)p.q, *k = (const TIn *)p.k, *v = (const TIn *)p.v, *dO = (const TIn *)p.d_o;
    float *Sb = buf, *G = buf + DK * DV;
    float *redv = G + DK * DV, *redw = redv + NP * DV, *ev = redw + NP * DV, *wv = ev + DV;
    float *redc = wv + DV;          // [NH][4][DK]
    float *das = redc + 4 * NH * DK;  // [DK]: a token's dalpha by channel
    const int j = tid % DV, part = tid / DV;
    for (int e = tid; e < DK * DV; e += NT) G[e] = Gg[e];
    for (int r = L - 1; r >= 0; --r) {
        // Sb = S_{r-1}
        for (int e = tid; e < DK * DV; e += NT) Sb[e] = Sg[e];
        __syncthreads();
        for (int m = 0; m < r; ++m) {
            const int64_t tk = (tok0 + m) * H + h;
            float vp = 0.f;
            for (int c = part; c < DK; c += NP) vp += gate_at(p.alpha, GATE, tk, c, DK) * ld_in(k, tk * DK + c) * Sb[c * DV + j];
            redv[part * DV + j] = vp;
            __syncthreads();
            float vh = 0.f;
            for (int p2 = 0; p2 < NP; ++p2) vh += redv[p2 * DV + j];
            const float be = p.beta[tk] * (ld_in(v, tk * DV + j) - vh);
            for (int c = part; c < DK; c += NP)
                Sb[c * DV + j] = gate_at(p.alpha, GATE, tk, c, DK) * Sb[c * DV + j] + ld_in(k, tk * DK + c) * be;
            __syncthreads();
        }
        // reverse step of token r
        const int64_t tk = (tok0 + r) * H + h;
        const float bt = p.beta[tk];
        {
            const float dj = ld_in(dO, tk * DV + j);
            float vp = 0.f, wp = 0.f;
            for (int c = part; c < DK; c += NP) {
                const float kc = ld_in(k, tk * DK + c);
                const float g = G[c * DV + j] + ld_in(q, tk * DK + c) * dj;
                G[c * DV + j] = g;
                vp += gate_at(p.alpha, GATE, tk, c, DK) * kc * Sb[c * DV + j];
                wp += kc * g;
            }
            redv[part * DV + j] = vp;
            redw[part * DV + j] = wp;
            __syncthreads();
            if (part == 0) {
                float vh = 0.f, w = 0.f;
                for (int p2 = 0; p2 < NP; ++p2) {
                    vh += redv[p2 * DV + j];
                    w += redw[p2 * DV + j];
                }
                ev[j] = ld_in(v, tk * DV + j) - vh;
                wv[j] = w;
                p.dv[tk * DV + j] = bt * w;
            }
            __syncthreads();
        }
        {
            // row mapping: channel c, value columns of part hp
            const int c = tid % DK, hp = tid / DK, cw = DV / NH;
            const float ac = gate_at(p.alpha, GATE, tk, c, DK), kc = ld_in(k, tk * DK + c);
            float dq = 0.f, ge = 0.f, sw = 0.f, da = 0.f;
            for (int jj = hp * cw; jj < (hp + 1) * cw; ++jj) {
                const float sv = Sb[c * DV + jj], g = G[c * DV + jj], e = ev[jj], w = wv[jj];
                dq += (ac * sv + bt * kc * e) * ld_in(dO, tk * DV + jj);
                ge += g * e;
                sw += ac * sv * w;
                da += (g - bt * kc * w) * sv;
            }
            redc[(hp * 4 + 0) * DK + c] = dq;
            redc[(hp * 4 + 1) * DK + c] = ge;
            redc[(hp * 4 + 2) * DK + c] = sw;
            redc[(hp * 4 + 3) * DK + c] = da;
            __syncthreads();
            if (tid < DK) {
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
                for (int h2 = 0; h2 < NH; ++h2)
#pragma unroll
                    for (int u = 0; u < 4; ++u) s4[u] += redc[(h2 * 4 + u) * DK + tid];
                p.dq[tk * DK + tid] = s4[0];
                p.dk[tk * DK + tid] = bt * (s4[1] - s4[2]);
                if (GATE == KDA_GATE_CHANNEL) p.dalpha[tk * DK + tid] = s4[3];
                das[tid] = s4[3];
            }
            if (tid == 0) {
                float db = 0.f;
                for (int jj = 0; jj < DV; ++jj) db += wv[jj] * ev[jj];
                p.dbeta[tk] = db;
            }
            __syncthreads();
            if (tid == 0 && GATE == KDA_GATE_SCALAR) {  // one gate for every channel: the sum over them
                float da = 0.f;
                for (int c = 0; c < DK; ++c) da += das[c];
                p.dalpha[tk] = da;
            }
        }
        // G = Diag(alpha)(G - beta k w^T)
        for (int c = part; c < DK; c += NP)
            G[c * DV + j] = gate_at(p.alpha, GATE, tk, c, DK) * (G[c * DV + j] - bt * ld_in(k, tk * DK + c) * wv[j]);
        __syncthreads();
    }
}

template <int DK, typename TIn, int GATE>
__global__ void __launch_bounds__(NT, 1) kda_bwd_local_kernel(BwdParams p) {
    constexpr bool SPLIT = std::is_same<TIn, float>::value;  // fp32 inputs: fp32 accuracy
    extern __shared__ __align__(16) unsigned char smem_raw[];
    LocalSmem<DK, TIn> &sm = *reinterpret_cast<LocalSmem<DK, TIn> *>(smem_raw);
    using TL = TabLayout<DK>;
    constexpr int LDK = DK + 8;  // [C][DK] tables: read down their columns by the chunk-wide products
    constexpr int NK = DK / 16;  // 8-column tiles of a warp's half of a 64 x DK product
    constexpr int DLD = DoRow<TIn>::LD;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int64_t idx = blockIdx.x;  // the chunk's workspace slot
    int64_t c;
    int h, n, L;
    int64_t tok0;
    cta_chunk(p, idx, c, h);
    const int H = p.H, DV = p.DV;
    if ((p.status && *p.status) || !chunk_of(p, c, n, tok0, L)) return;
    const TIn *dO = (const TIn *)p.d_o;
    const float *Sg = p.states + idx * DK * DV, *Gg = p.gnext + idx * DK * DV;
    const float *tab = p.tabs + idx * TL::FLOATS;
    const float *wk = p.work + idx * 4 * C * DV;  // U, V - X, dU, dR: [4][C][DV]
    if (__float_as_int(tab[TL::SLOW])) {
        local_slow<DK, TIn, GATE>(sm.u.slow, p, Sg, Gg, tok0, L, h);
        return;
    }
    // Kr and Qr are read last, into the pieces' place, and the gates near the
    // end: pull them into L2 now
    for (int l = tid; l < 2 * C * DK / 32; l += NT) asm volatile("prefetch.global.L2 [%0];" ::"l"(tab + TL::KR + 32 * l));
    if (GATE == KDA_GATE_CHANNEL)
        for (int l = tid; l < L * (DK / 32); l += NT)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.alpha + ((tok0 + l / (DK / 32)) * H + h) * DK + 32 * (l % (DK / 32))));
    // Kc, T, mu, beta, then the first piece
    for (int e = tid; e < C * DK / 4; e += NT) {
        const int r = e / (DK / 4), cc = 4 * (e % (DK / 4));
        cp16(&sm.Kc[r * LDK + cc], tab + TL::KC + r * DK + cc);
    }
    for (int e = tid; e < C * C / 4; e += NT) {
        const int r = e / (C / 4), cc = 4 * (e % (C / 4));
        cp16(&sm.T[r * LDC + cc], tab + TL::T + r * C + cc);
    }
    for (int e = tid; e < DK / 4; e += NT) cp16(&sm.mu[4 * e], tab + TL::MU + 4 * e);
    for (int e = tid; e < C / 4; e += NT) cp16(&sm.beta[4 * e], tab + TL::BETA + 4 * e);
    auto load_piece = [&](int v0, LocalPiece<DK, TIn> &P) {
        constexpr int Q = VP / 4;  // 16-byte pieces of a fp32 row
        for (int e = tid; e < DK * Q; e += NT) {
            const int r = e / Q, cc = 4 * (e % Q);
            cp16(&P.S[r * LDP + cc], Sg + (int64_t)r * DV + v0 + cc);
            cp16(&P.G[r * LDP + cc], Gg + (int64_t)r * DV + v0 + cc);
        }
        for (int e = tid; e < C * Q; e += NT) {
            const int r = e / Q, cc = 4 * (e % Q);
            const float *src = wk + (int64_t)r * DV + v0 + cc;
            cp16(&P.U[r * LDP + cc], src);
            cp16(&P.VmX[r * LDP + cc], src + C * DV);
            cp16(&P.dU[r * LDP + cc], src + 2 * C * DV);
            cp16(&P.dR[r * LDP + cc], src + 3 * C * DV);
        }
        constexpr int EO = 16 / (int)sizeof(TIn), QO = VP / EO;  // elements per 16 bytes; 16-byte pieces of a row
        for (int e = tid; e < C * QO; e += NT) {
            const int r = e / QO, cc = EO * (e % QO);
            const TIn *src = dO + ((tok0 + (r < L ? r : 0)) * H + h) * DV + v0 + cc;
            cp16z(&P.dO[r * DLD + cc], src, r < L ? 16u : 0u);  // rows past the sequence: zeros
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    load_piece(0, sm.u.piece[0]);

    // warp tile: rows R0 .. R0 + 15; columns C0 .. C0 + 31 of a 64-wide product,
    // CK .. CK + DK/2 - 1 of a DK-wide one
    const int R0 = 16 * (warp & 3), C0 = 32 * (warp >> 2), CK = (DK / 2) * (warp >> 2);
    // Sums over the value columns, accumulated piece by piece (the diagonal
    // factors that do not depend on the column are applied after the loop):
    float dT[4][4], dP[4][4];                  // dU (V - X)^T, dO U^T
    float dKc[NK][4], dQr[NK][4], dKr[NK][4];  // U G^T, dO S^T, dR S^T
    float db1 = 0.f;                           // sum_v dR (V - X) of row tid / 4 (a quarter of the columns)
    float s0 = 0.f;                            // sum_v S G of channel tid % DK (part tid / DK)
    fzero<4>(dT);
    fzero<4>(dP);
    fzero<NK>(dKc);
    fzero<NK>(dQr);
    fzero<NK>(dKr);
    const int npieces = DV / VP;
    for (int it = 0; it < npieces; ++it) {
        if (it + 1 < npieces) {
            load_piece((it + 1) * VP, sm.u.piece[(it + 1) & 1]);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const LocalPiece<DK, TIn> &P = sm.u.piece[it & 1];
#pragma unroll 2
        for (int k = 0; k < VP; k += 8) {
            uint32_t oh[4], ol[4], rh[4], rl[4], uh[4], ul[4], dh[4], dl[4];
            afrag<SPLIT>(P.dO, DLD, R0, k, oh, ol);
            // the fp32 tiles' fragments by ldmatrix: an 8 x 8 b16 matrix is 8 rows of
            // 4 floats, and lane 4 g + t receives row g, float t of each
            const int arow = R0 + ldsm_arow(), acol = k + ldsm_acol();
            afrag_ldsm<SPLIT>(P.dR + arow * LDP + acol, rh, rl);
            afrag_ldsm<SPLIT>(P.U + arow * LDP + acol, uh, ul);
            afrag_ldsm<SPLIT>(P.dU + arow * LDP + acol, dh, dl);
            const int brow = ldsm_brow(), bcol = k + ldsm_bcol();
#pragma unroll
            for (int np = 0; np < NK / 2; ++np) {  // two 8-column tiles per load
                const int o = (CK + 16 * np + brow) * LDP + bcol;
                uint32_t s4[4], g4[4];
                ldsm_x4(P.S + o, s4);
                ldsm_x4(P.G + o, g4);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const BFrag bs = bfrag<SPLIT>(__uint_as_float(s4[2 * u]), __uint_as_float(s4[2 * u + 1]));
                    const BFrag bg = bfrag<SPLIT>(__uint_as_float(g4[2 * u]), __uint_as_float(g4[2 * u + 1]));
                    mma_f<SPLIT>(dQr[2 * np + u], oh, ol, bs);
                    mma_f<SPLIT>(dKr[2 * np + u], rh, rl, bs);
                    mma_f<SPLIT>(dKc[2 * np + u], uh, ul, bg);
                }
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int o = (C0 + 16 * np + brow) * LDP + bcol;
                uint32_t u4[4], v4[4];
                ldsm_x4(P.U + o, u4);
                ldsm_x4(P.VmX + o, v4);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const BFrag bu = bfrag<SPLIT>(__uint_as_float(u4[2 * u]), __uint_as_float(u4[2 * u + 1]));
                    const BFrag bv = bfrag<SPLIT>(__uint_as_float(v4[2 * u]), __uint_as_float(v4[2 * u + 1]));
                    mma_f<SPLIT>(dP[2 * np + u], oh, ol, bu);
                    mma_f<SPLIT>(dT[2 * np + u], dh, dl, bv);
                }
            }
        }
        {
            constexpr int NH = NT / DK, CW = VP / NH;
            const int cc = tid % DK, hp = tid / DK;
#pragma unroll
            for (int j = 0; j < CW; j += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&P.S[cc * LDP + hp * CW + j]);
                const float4 g4 = *reinterpret_cast<const float4 *>(&P.G[cc * LDP + hp * CW + j]);
                s0 += a4.x * g4.x + a4.y * g4.y + a4.z * g4.z + a4.w * g4.w;
            }
            const int r = tid >> 2, j0 = (VP / 4) * (tid & 3);
#pragma unroll
            for (int j = 0; j < VP / 4; j += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&P.dR[r * LDP + j0 + j]);
                const float4 e4 = *reinterpret_cast<const float4 *>(&P.VmX[r * LDP + j0 + j]);
                db1 += a4.x * e4.x + a4.y * e4.y + a4.z * e4.z + a4.w * e4.w;
            }
        }
        __syncthreads();  // this piece's buffer is refilled two pieces on
    }
    // Kr, Qr into the pieces' place; meanwhile the column and row factors:
    // dQr = dO St^T, dKr = dX St^T (dX = -Diag(beta) dR), dKc = U Gt^T with
    // St = Diag(mu) S, Gt = Diag(mu) G; dT = dU R^T with R = Diag(beta) (V - X)
    LocalFinal<DK> &F = sm.u.fin;
    float alh[2][GateSplit<DK>::TPS];  // the gates of the chunk's gate factors, loaded under the products
    gate_factor_loads<DK>(alh, p.alpha, GATE, tok0, L, H, h);
    for (int e = tid; e < C * DK / 4; e += NT) {
        const int r = e / (DK / 4), cc = 4 * (e % (DK / 4));
        cp16(&F.Kr[r * LDK + cc], tab + TL::KR + r * DK + cc);
        cp16(&F.Qr[r * LDK + cc], tab + TL::QR + r * DK + cc);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = R0 + g + 8 * (e >> 1), cc = CK + 8 * nt + 2 * t4 + (e & 1);
            const float m = sm.mu[cc];
            dQr[nt][e] *= m;
            dKc[nt][e] *= m;
            dKr[nt][e] *= -sm.beta[r] * m;
        }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dT[nt][e] *= sm.beta[C0 + 8 * nt + 2 * t4 + (e & 1)];
    db1 += __shfl_xor_sync(0xffffffffu, db1, 1);
    db1 += __shfl_xor_sync(0xffffffffu, db1, 2);
    float *dbr = sm.red + 8 * DK;  // [3][C]: dbeta's second part by column half, its first part
    if ((tid & 3) == 0) dbr[2 * C + (tid >> 2)] = db1;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // W[0]: dT, then dA (rows of LDC); W[1]: lower(dP), then dA (rows of LS,
    // for the transposed reads); W[2]: lower(dP) (rows of LDC); W[3]: Z (rows of LS)
    float *WA = F.W[0], *WP = F.W[1], *WC = F.W[2], *WD = F.W[3];
    float acc[4][4];
    float db[2] = {0.f, 0.f};  // dbeta's second part, rows R0 + g, R0 + g + 8
    // the first parts of d log mu's column sums: Kc (U Gt^T), Qr (dO St^T), Kr (dX St^T)
    float s123[NK][2];
#pragma unroll
    for (int nt = 0; nt < NK; ++nt) {
        const int cc = CK + 8 * nt + 2 * t4, a0 = (R0 + g) * LDK + cc, a1 = (R0 + g + 8) * LDK + cc;
        const float2 kc0 = *reinterpret_cast<const float2 *>(sm.Kc + a0), kc1 = *reinterpret_cast<const float2 *>(sm.Kc + a1);
        const float2 qr0 = *reinterpret_cast<const float2 *>(F.Qr + a0), qr1 = *reinterpret_cast<const float2 *>(F.Qr + a1);
        const float2 kr0 = *reinterpret_cast<const float2 *>(F.Kr + a0), kr1 = *reinterpret_cast<const float2 *>(F.Kr + a1);
        s123[nt][0] = kc0.x * dKc[nt][0] + kc1.x * dKc[nt][2] + qr0.x * dQr[nt][0] + qr1.x * dQr[nt][2] +
                      kr0.x * dKr[nt][0] + kr1.x * dKr[nt][2];
        s123[nt][1] = kc0.y * dKc[nt][1] + kc1.y * dKc[nt][3] + qr0.y * dQr[nt][1] + qr1.y * dQr[nt][3] +
                      kr0.y * dKr[nt][1] + kr1.y * dKr[nt][3];
    }
    ffor<4>(dP, R0, C0, [&](int r, int cc, float &x) { x = cc <= r ? x : 0.f; });  // lower(dP)
    sstore<4>(dP, R0, C0, WC, LDC);
    sstore<4>(dP, R0, C0, WP, LS);
    sstore<4>(dT, R0, C0, WA, LDC);
    __syncthreads();
    // dQr += dP Kc;  dKc += dP^T Qr
    wmm<C, NK, SPLIT>(dQr, [&](int r, int m) { return WC[r * LDC + m]; }, [&](int m, int cc) { return sm.Kc[m * LDK + cc]; }, R0,
                      CK);
    wmm<C, NK, SPLIT>(dKc, [&](int r, int m) { return WP[m * LS + r]; }, [&](int m, int cc) { return F.Qr[m * LDK + cc]; }, R0,
                      CK);
    // dA = strict-lower(-T^T dT T^T): Z = dT T^T -> WD, then -T^T Z -> WA (and WP)
    fzero<4>(acc);
    wmm<C, 4, SPLIT>(acc, [&](int r, int m) { return WA[r * LDC + m]; }, [&](int m, int cc) { return sm.T[cc * LDC + m]; }, R0,
                     C0);
    sstore<4>(acc, R0, C0, WD, LS);
    __syncthreads();
    fzero<4>(acc);
    wmm<C, 4, SPLIT>(acc, [&](int r, int m) { return sm.T[m * LDC + r]; }, [&](int m, int cc) { return WD[m * LS + cc]; }, R0,
                     C0);
    __syncthreads();  // every read of dT in WA and of lower(dP) in WP is done
    ffor<4>(acc, R0, C0, [&](int r, int cc, float &x) { x = cc < r ? -x : 0.f; });
    sstore<4>(acc, R0, C0, WA, LDC);
    sstore<4>(acc, R0, C0, WP, LS);
    __syncthreads();
    // dKr += Diag(beta) dA Kc (and dbeta's second part Kr . (dA Kc));  dKc += (Diag(beta) dA)^T Kr
    {
        float tmp[NK][4];
        fzero<NK>(tmp);
        wmm<C, NK, SPLIT>(tmp, [&](int r, int m) { return WA[r * LDC + m]; }, [&](int m, int cc) { return sm.Kc[m * LDK + cc]; },
                          R0, CK);
#pragma unroll
        for (int nt = 0; nt < NK; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int r = R0 + g + 8 * (e >> 1), cc = CK + 8 * nt + 2 * t4;
                const float2 kr = *reinterpret_cast<const float2 *>(F.Kr + r * LDK + cc);
                const float br = sm.beta[r];
                db[e >> 1] += kr.x * tmp[nt][e] + kr.y * tmp[nt][e + 1];
                dKr[nt][e] += br * tmp[nt][e];
                dKr[nt][e + 1] += br * tmp[nt][e + 1];
            }
    }
    wmm<C, NK, SPLIT>(dKc, [&](int r, int m) { return sm.beta[m] * WP[m * LS + r]; },
                      [&](int m, int cc) { return F.Kr[m * LDK + cc]; }, R0, CK);
    // dbeta's second part: sums over this warp's columns (the 4 lanes of a
    // row), then the two column halves of each row and the first part, in a
    // fixed order
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        db[u] += __shfl_xor_sync(0xffffffffu, db[u], 1);
        db[u] += __shfl_xor_sync(0xffffffffu, db[u], 2);
    }
    if (t4 == 0) {
        dbr[(warp >> 2) * C + R0 + g] = db[0];
        dbr[(warp >> 2) * C + R0 + g + 8] = db[1];
    }
    // the chunk's gate factors p / mu (as in the forward tables) into the free
    // work tiles; dq, dk, and d log p into Qr's place
    float *E2 = F.W[0], *E3 = F.W[2];  // [C][LDK] each: W[0..1] and W[2..3]
    static_assert(C * LDK <= 2 * C * LS, "E2 and E3 fit in two work tiles each");
    gate_factor_table<DK>(sm.part, sm.mu, E2, E3, LDK, alh);
    sm.part[(tid / DK) * DK + tid % DK] = sm.mu[tid % DK] * sm.mu[tid % DK] * s0;
    if (tid < L) p.dbeta[(tok0 + tid) * H + h] = dbr[tid] + dbr[C + tid] + dbr[2 * C + tid];
    float dlogp[NK][4];
#pragma unroll
    for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {  // the two columns of a row together (8-byte accesses)
            const int r = R0 + g + 8 * (e >> 1), cc = CK + 8 * nt + 2 * t4, rc = r * LDK + cc;
            const float2 e2 = *reinterpret_cast<const float2 *>(E2 + rc);  // p / mu
            const float2 e3 = *reinterpret_cast<const float2 *>(E3 + rc);  // mu / p
            if (r < L) {
                const int64_t th = (tok0 + r) * H + h;
                *reinterpret_cast<float2 *>(p.dq + th * DK + cc) = make_float2(dQr[nt][e] * e2.x, dQr[nt][e + 1] * e2.y);
                *reinterpret_cast<float2 *>(p.dk + th * DK + cc) =
                    make_float2(dKr[nt][e] * e2.x + dKc[nt][e] * e3.x, dKr[nt][e + 1] * e2.y + dKc[nt][e + 1] * e3.y);
            }
            const float2 kr = *reinterpret_cast<const float2 *>(F.Kr + rc), qr = *reinterpret_cast<const float2 *>(F.Qr + rc),
                         kc = *reinterpret_cast<const float2 *>(sm.Kc + rc);
            dlogp[nt][e] = dKr[nt][e] * kr.x + dQr[nt][e] * qr.x - dKc[nt][e] * kc.x;
            dlogp[nt][e + 1] = dKr[nt][e + 1] * kr.y + dQr[nt][e + 1] * qr.y - dKc[nt][e + 1] * kc.y;
        }
    // s123: sums over the 16 rows of this warp (lanes with the same t), then by warp row block
#pragma unroll
    for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float x = s123[nt][u];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            s123[nt][u] = x;
        }
    __syncthreads();  // every read of Qr is done
    if (g == 0)
#pragma unroll
        for (int nt = 0; nt < NK; ++nt)
#pragma unroll
            for (int u = 0; u < 2; ++u) sm.red[(warp & 3) * DK + CK + 8 * nt + 2 * t4 + u] = s123[nt][u];
    ffor<NK>(dlogp, R0, CK, [&](int r, int cc, float &x) { F.Qr[r * LDK + cc] = x; });
    __syncthreads();
    // per channel: d log mu, then d log alpha by a reverse running sum over
    // the rows; NT / DK threads per channel, each over a block of RH rows
    {
        constexpr int NH = NT / DK, RH = C / NH;
        const int cc = tid % DK, hp = tid / DK, rb = hp * RH;
        float al[RH];  // this block's gates, every load in flight at once
#pragma unroll
        for (int i = 0; i < RH; ++i)
            al[i] = rb + i < L ? gate_at(p.alpha, GATE, (tok0 + rb + i) * H + h, cc, DK) : 1.f;
        float *psum = F.W[0];  // [NH][DK]: d log p summed over each row block (E2 is read no more)
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < RH; ++i)
            if (rb + i < L) ps += F.Qr[(rb + i) * LDK + cc];
        psum[hp * DK + cc] = ps;
        __syncthreads();
        float s0c = 0.f, colsum = 0.f, later = 0.f;  // (sums in block order)
        for (int h2 = 0; h2 < NH; ++h2) {
            s0c += sm.part[h2 * DK + cc];
            const float x = psum[h2 * DK + cc];
            colsum += x;
            if (h2 > hp) later += x;
        }
        float s123c = 0.f;
        for (int t2 = 0; t2 < 4; ++t2) s123c += sm.red[t2 * DK + cc];
        const float dlogmu = 2.f * s0c + s123c - colsum;
        float run = 0.5f * dlogmu + later;  // d log p_{L-1} += d log mu / 2, plus the later blocks
#pragma unroll
        for (int i = RH - 1; i >= 0; --i) {
            const int r = rb + i;
            if (r < L) {
                run += F.Qr[r * LDK + cc];
                const int64_t th = (tok0 + r) * H + h;
                const float da = run / al[i];
                if (GATE == KDA_GATE_CHANNEL) p.dalpha[th * DK + cc] = da;
                else F.Qr[r * LDK + cc] = da;  // (this thread's own rows and column, read only by itself)
            }
        }
    }
    if (GATE == KDA_GATE_SCALAR) {  // one gate for every channel: the sum over them, in channel order
        __syncthreads();
        if (tid < L) {
            float da = 0.f;
            for (int cc = 0; cc < DK; ++cc) da += F.Qr[tid * LDK + cc];
            p.dalpha[(tok0 + tid) * H + h] = da;
        }
    }
}

constexpr size_t kMaxSmem = 232448;  // dynamic shared memory one CTA may have
static_assert(sizeof(StatesSmem<128, float>) <= kMaxSmem && sizeof(StatesSmem<128, __nv_bfloat16>) <= kMaxSmem &&
                  sizeof(ChainSmem<128, float>) <= kMaxSmem && sizeof(ChainSmem<128, __nv_bfloat16>) <= kMaxSmem &&
                  sizeof(LocalSmem<128, float>) <= kMaxSmem && sizeof(LocalSmem<128, __nv_bfloat16>) <= kMaxSmem &&
                  2 * sizeof(TabSmem<128>) + 2048 <= kMaxSmem,  // two tables CTAs per SM
              "shared memory per CTA");

// Packed batches: checks cu_seqlens (starts at 0, never decreases, ends at
// T_total) and lists the first chunk of every sequence (coff, an exclusive
// sum of ceil(L_n / 64)); on a bad cu_seqlens it writes the status and an
// empty chunk list, and every later kernel skips its work.
constexpr int kPrepThreads = 1024;
__global__ void __launch_bounds__(kPrepThreads) kda_bwd_varlen_prep_kernel(const int32_t *__restrict__ cu, int N,
                                                                          int T_total, int32_t *__restrict__ coff,
                                                                          int32_t *__restrict__ status) {
    __shared__ int bad;
    __shared__ int32_t part[kPrepThreads];
    __shared__ int32_t total;
    const int tid = threadIdx.x;
    if (tid == 0) bad = (cu[0] != 0 || cu[N] != T_total) ? 1 : 0;
    __syncthreads();
    const int per = (N + kPrepThreads - 1) / kPrepThreads, lo = tid * per, hi = lo + per < N ? lo + per : N;
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) {
        const int32_t L = cu[i + 1] - cu[i];
        if (L < 0) atomicOr(&bad, 1);
        else local += (L + C - 1) / C;
    }
    part[tid] = local;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int t = 0; t < kPrepThreads; ++t) {
            const int32_t x = part[t];
            part[t] = run;
            run += x;
        }
        total = run;
    }
    __syncthreads();
    int32_t run = part[tid];
    for (int i = lo; i < hi; ++i) {
        coff[i] = run;
        const int32_t L = cu[i + 1] - cu[i];
        run += L > 0 ? (L + C - 1) / C : 0;
    }
    if (tid == 0) {
        coff[N] = bad ? 0 : total;
        *status = bad ? KDA_DEV_BAD_CU_SEQLENS : KDA_DEV_OK;
    }
}

// Chunks the workspace must hold: every chunk of equal-length sequences, or
// for a packed batch an upper bound (each sequence adds at most one partial
// chunk to ceil(T_total / 64)).
int64_t chunk_bound(bool packed, int N, int T) {
    return packed ? ((int64_t)T + C - 1) / C + N : (int64_t)N * ((T + C - 1) / C);
}

template <int DK, typename TIn>
cudaError_t launch_t(const BackwardArgs &b, cudaStream_t s) {
    const bool packed = b.cu_seqlens != nullptr;
    const int NC = packed ? 0 : (b.T + C - 1) / C;
    const int nslices = b.d_v / VS;
    const int64_t chunks = chunk_bound(packed, b.N, b.T);
    BwdParams p;
    p.q = b.q; p.k = b.k; p.v = b.v; p.d_o = b.d_o; p.alpha = b.alpha; p.beta = b.beta; p.dsT = b.dsT;
    p.dq = b.dq; p.dk = b.dk; p.dv = b.dvv; p.dalpha = b.dalpha; p.dbeta = b.dbeta; p.ds0 = b.ds0;
    float *ws = static_cast<float *>(b.workspace);
    const int64_t slab = chunks * b.H * DK * b.d_v;
    p.states = ws;
    p.gnext = ws + slab;
    p.tabs = ws + 2 * slab;
    p.work = p.tabs + chunks * b.H * TabLayout<DK>::FLOATS;
    p.N = b.N; p.T = b.T; p.H = b.H; p.DV = b.d_v; p.NC = NC; p.gate = b.gate;
    p.cu = b.cu_seqlens;
    p.coff = nullptr;
    p.status = nullptr;
    cudaError_t e;
    if (packed) {
        int32_t *tail = reinterpret_cast<int32_t *>(p.work + chunks * b.H * 4 * C * b.d_v);
        int32_t *coff = tail + 4;  // tail[0]: the status word when the caller gives none
        int32_t *status = b.dev_status ? b.dev_status : tail;
        kda_bwd_varlen_prep_kernel<<<1, kPrepThreads, 0, s>>>(b.cu_seqlens, b.N, b.T, coff, status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        p.coff = coff;
        p.status = status;
    }
    const unsigned heads = (unsigned)((int64_t)b.N * b.H * nslices);
    const unsigned chunk_ctas = (unsigned)(chunks * b.H);
    if (chunks > 0) {  // 1. every chunk's tables, all chunks at once
        auto tabk = kda_bwd_tables_kernel<DK, TIn>;
        const size_t st = sizeof(TabSmem<DK>);
        if ((e = cudaFuncSetAttribute(tabk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st)) != cudaSuccess)
            return e;
        tabk<<<chunk_ctas, NT, st, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // 2. the state before every chunk
        auto stk = kda_bwd_states_kernel<DK, TIn>;
        const size_t ss = sizeof(StatesSmem<DK, TIn>);
        if ((e = cudaFuncSetAttribute(stk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss)) != cudaSuccess)
            return e;
        stk<<<heads, NT, ss, s>>>(p, b.s0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 3. the reverse state-gradient chain (also for empty sequences: dS_0 = dS_T)
    auto chain = kda_bwd_chain_kernel<DK, TIn>;
    const size_t sc = sizeof(ChainSmem<DK, TIn>);
    if ((e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc)) != cudaSuccess) return e;
    chain<<<heads, NT, sc, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (chunks == 0) return cudaSuccess;
    // 4. every chunk's gradients
    // (the gate kind is a template parameter here: this pass runs at the
    // register limit, where run-time branches on it cost 7 %)
    auto local = b.gate == KDA_GATE_SCALAR ? kda_bwd_local_kernel<DK, TIn, KDA_GATE_SCALAR>
                 : b.gate == KDA_GATE_NONE ? kda_bwd_local_kernel<DK, TIn, KDA_GATE_NONE>
                                           : kda_bwd_local_kernel<DK, TIn, KDA_GATE_CHANNEL>;
    const size_t sl = sizeof(LocalSmem<DK, TIn>);
    if ((e = cudaFuncSetAttribute(local, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl)) != cudaSuccess) return e;
    local<<<chunk_ctas, NT, sl, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_bytes(int N, int T, int H, int dk, int dv, bool packed) {
    const size_t chunks = (size_t)chunk_bound(packed, N, T) * H;
    const size_t tab = dk == 128 ? TabLayout<128>::FLOATS : TabLayout<64>::FLOATS;
    const size_t tail = packed ? (4 + (size_t)N + 1) * sizeof(int32_t) : 0;  // status, chunk offsets
    return (2 * chunks * dk * dv + chunks * tab + chunks * 4 * C * dv) * sizeof(float) + tail;
}

cudaError_t launch_backward(const BackwardArgs &b, cudaStream_t s) {
    if (b.d_v % VS) return cudaErrorInvalidValue;
    if (b.d_k == 128) return b.dt == KDA_BF16 ? launch_t<128, __nv_bfloat16>(b, s) : launch_t<128, float>(b, s);
    if (b.d_k == 64) return b.dt == KDA_BF16 ? launch_t<64, __nv_bfloat16>(b, s) : launch_t<64, float>(b, s);
    return cudaErrorInvalidValue;
}

}  // namespace kda
