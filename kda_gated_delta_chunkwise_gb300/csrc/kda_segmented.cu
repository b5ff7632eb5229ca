// Prefill of one long sequence split into segments that run at the same time
// (kda_prefill_segmented in include/kda.h).
//
// The K3 essay (pwwt.cn/news/3763336) writes the update as an affine map of
// the state, S_t = A_t S_{t-1} + B_t (§六), with the transition from position
// j to t the product A_t ... A_{j+1} (§五). Over a stretch of tokens the map
// is therefore S_end = Phi S_start + b, where Phi is the stretch's transition
// product and b the state the stretch reaches from zero; inside the stretch
// the state at token t is Phi_t S_start + S_loc,t, so its output is
//
//     o_t = S_t^T q_t = S_loc,t^T q_t + S_start^T (Phi_t^T q_t).
//
// Both Phi_t^T q_t and Phi come out of the ordinary prefill run on the
// stretch with v = 0 and the identity as the initial state (every value
// column of that run carries one column of Phi_t): its outputs are
// z_t = Phi_t^T q_t and its final state is Phi. So a sequence of n chunks is
// cut into segment 0 (true initial state) and G - 1 later segments, and
//
//   - segment 0 runs from S0 (stream `hi`, highest priority, so its clusters
//     are placed first: it is the longest);
//   - each later segment g runs twice on stream `a`: from zero with the true
//     v (outputs o_loc into o, final state b_g), then with v = 0 from the
//     identity (outputs Z, final state Phi_g);
//   - combine: S_start,1 = S_end,0 and S_start,g+1 = Phi_g S_start,g + b_g in
//     float32; the final state is the last of these;
//   - correct: o_t += S_start,g^T z_t for every token of segment g >= 1, a
//     bf16 tensor-core product with float32 accumulation (the same operand
//     precision as the prefill's own chunk products).
//
// Segment 0 runs n - (G-1)L chunks and the others L each; the plan picks G and
// L so that segment 0 ends about when the later segments' two runs do, the
// later runs filling the kResidentClusters - H cluster slots that segment 0
// leaves free.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kC = 64;               // tokens per chunk
constexpr int kD = 128;              // d_k = d_v of the tensor-core prefill
constexpr int kResidentClusters = 76; // two-CTA prefill clusters the 152 SMs hold at once
constexpr int kMaxSegments = 16;     // automatic plans
constexpr int kMaxForced = 4096;     // a forced count
constexpr int kMinSegChunks = 8;     // automatic plans: shortest later segment
// Start-up and drain of one launch wave of the prefill (launch, barrier and
// TMEM set-up, the first chunk through the gate-solve-chain pipeline, the
// last one out), in chunk steps; fitted to measured splits of 1 x 16 x 16384,
// 1 x 16 x 131072 and 1 x 32 x 131072 (about 50 us).
constexpr int kStartupChunks = 16;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

kda_status_t fail(kda_status_t st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
kda_status_t fail(kda_status_t st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return kda::set_error(st, buf);
}

kda_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// G segments: segment 0 has `first` chunks, segments 1..G-1 `len` chunks each
// (the last may end in a partial chunk: it stops at T).
struct Plan {
    int G, first, len;
};

bool splittable(int B, int d_k, int d_v, kda_dtype_t dt) { return B == 1 && dt == KDA_BF16 && d_k == kD && d_v == kD; }

// Launch waves of the later segments' runs (in units of one segment's run)
// while segment 0 holds H cluster slots: their 2 (G-1) H runs come as two
// launches over the remaining kResidentClusters - H slots.
int waves(int G, int H) {
    const int free_slots = kResidentClusters - H > H ? kResidentClusters - H : H;
    const int per_launch = (H * (G - 1) + free_slots - 1) / free_slots;
    return 2 * per_launch;
}

Plan make_plan(int B, int T, int H, int d_k, int d_v, kda_dtype_t dt, int segments) {
    const int n = T > 0 ? (T + kC - 1) / kC : 0;
    if (!splittable(B, d_k, d_v, dt) || n < 2 || segments == 1) return {1, n, 0};
    // Segment 0 takes n - (G-1)L chunk steps (+ one launch's start-up), the
    // later runs w (L + start-up); L balances the two.
    auto split = [&](int G, int startup) {
        const int w = waves(G, H);
        int L = (n + startup - w * startup) / (w + G - 1);
        return Plan{G, n - (G - 1) * L, L};
    };
    if (segments >= 2) {  // a forced count: an even balance, no start-up term
        int G = segments < n ? segments : n;
        while (G > 1 && split(G, 0).len < 1) --G;
        return G > 1 ? split(G, 0) : Plan{1, n, 0};
    }
    // automatic: only while segment 0's clusters leave room for the others
    if (2 * H > kResidentClusters) return {1, n, 0};
    Plan best{1, n, 0};
    for (int G = 2; G <= kMaxSegments; ++G) {
        const Plan p = split(G, kStartupChunks);
        if (p.len < kMinSegChunks) continue;
        if (p.first < best.first) best = p;
    }
    // a split pays only when it saves a fifth of the chunk steps
    return 5 * (best.first + kStartupChunks) <= 4 * n ? best : Plan{1, n, 0};
}

struct Layout {
    size_t cu, vlws, fs0, fs1, ident, phi, sst, zv, z, total;
    int64_t T1;  // tokens of segments 1..G-1
};

Layout layout(const Plan &p, int T, int H) {
    Layout l{};
    if (p.G < 2) return l;
    const size_t g1 = (size_t)(p.G - 1);
    l.T1 = (int64_t)T - (int64_t)p.first * kC;
    const size_t mat = (size_t)kD * kD;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align_up(bytes);
        return at;
    };
    l.cu = take((size_t)p.G * sizeof(int32_t));
    l.vlws = take(kda_varlen_workspace_bytes(p.G - 1, H, kD, kD));
    l.fs0 = take((size_t)H * mat * sizeof(float));
    l.fs1 = take(g1 * H * mat * sizeof(float));
    l.ident = take(g1 * H * mat * sizeof(float));
    l.phi = take(g1 * H * mat * sizeof(float));
    l.sst = take(g1 * H * mat * sizeof(__nv_bfloat16));
    l.zv = take((size_t)l.T1 * H * kD * sizeof(__nv_bfloat16));
    l.z = take((size_t)l.T1 * H * kD * sizeof(__nv_bfloat16));
    l.total = off;
    return l;
}

// ---------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------

// cu_seqlens of segments 1..G-1 (relative to their first token) and the
// identity initial state of every (segment, head) of the transition runs.
__global__ void seg_setup_kernel(int32_t *__restrict__ cu, int G, int len_tokens, int T1,
                                 float4 *__restrict__ ident, int64_t n_vec4) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < G) cu[i] = i == G - 1 ? T1 : (int32_t)(i * len_tokens);
    if (i < n_vec4) {
        const int r = (int)(i % (kD * kD / 4));  // float4 index inside one 128 x 128 matrix
        const int row = r / (kD / 4), c0 = (r % (kD / 4)) * 4;
        float4 x;
        x.x = row == c0 ? 1.f : 0.f;
        x.y = row == c0 + 1 ? 1.f : 0.f;
        x.z = row == c0 + 2 ? 1.f : 0.f;
        x.w = row == c0 + 3 ? 1.f : 0.f;
        ident[i] = x;
    }
}

constexpr int kCombThreads = 256;
constexpr int kPhiLd = kD + 1;           // padded row of Phi in shared memory
template <int COLS> constexpr size_t comb_smem() { return (size_t)(2 * kD * kPhiLd + kD * (COLS + 1)) * sizeof(float); }

__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void cp4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}

// Start states of segments 1..G-1 and the final state, COLS state columns
// of one head per CTA (columns of the state never mix: Phi acts on the left;
// 16 columns when that keeps more SMs busy, else 32). Thread (row i, COLS / 2
// columns); Phi of the next step is copied in (cp.async) while this step
// multiplies. sst[g - 1][h] receives S_start,g^T in bf16 (row = value
// column, k fastest): the B operand of the correction's products.
template <int COLS>
__global__ void __launch_bounds__(kCombThreads)
seg_combine_kernel(const float *__restrict__ fs0, const float *__restrict__ fs1, const float *__restrict__ phi,
                   __nv_bfloat16 *__restrict__ sst, float *__restrict__ final_state, int G, int H) {
    extern __shared__ float sm[];
    float *Ps = sm;                      // [2][kD][kPhiLd]
    constexpr int NC = COLS / 2, LD = COLS + 1;
    float *Ss = sm + 2 * kD * kPhiLd;    // [kD][LD]
    const int h = blockIdx.x, j0 = blockIdx.y * COLS, tid = threadIdx.x;
    const int i = tid & (kD - 1), jh = (tid >> 7) * NC;  // output row, first of NC columns
    const size_t mat = (size_t)kD * kD;
    auto issue = [&](int g, int buf) {  // Phi of segment g + 1 (phi[g]) into buffer buf
        const float *src = phi + ((size_t)g * H + h) * mat;
        float *dst = Ps + buf * kD * kPhiLd;
        for (int e = tid; e < kD * kD; e += kCombThreads) cp4(dst + (e / kD) * kPhiLd + e % kD, src + e);
        cp_commit();
    };
    float acc[NC];
    for (int c = 0; c < NC; ++c) acc[c] = fs0[(size_t)h * mat + (size_t)i * kD + j0 + jh + c];
    if (G > 1) issue(0, 0);
    for (int g = 1; g < G; ++g) {
        const size_t at = ((size_t)(g - 1) * H + h) * mat;
        // S_start,g: to shared memory (this step's operand) and, as bf16, to
        // the correction's operand
        for (int c = 0; c < NC; ++c) {
            Ss[i * LD + jh + c] = acc[c];
            sst[at + (size_t)(j0 + jh + c) * kD + i] = __float2bfloat16_rn(acc[c]);
        }
        if (g + 1 < G) issue(g, g & 1);
        else cp_commit();
        cp_wait1();  // Phi of this step landed (this thread's part)
        __syncthreads();
        const float *P = Ps + ((g - 1) & 1) * kD * kPhiLd + i * kPhiLd;
        for (int c = 0; c < NC; ++c) acc[c] = fs1[at + (size_t)i * kD + j0 + jh + c];
        for (int kk = 0; kk < kD; ++kk) {
            const float p = P[kk];
            const float *sr = Ss + kk * LD + jh;
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c] = fmaf(p, sr[c], acc[c]);
        }
        __syncthreads();  // Ss and this Phi buffer are rewritten next step
    }
    if (final_state)
        for (int c = 0; c < NC; ++c) final_state[(size_t)h * mat + (size_t)i * kD + j0 + jh + c] = acc[c];
}

constexpr int kCorrWarps = 12;          // one CTA per SM: 12 warps share the S_start tile
constexpr int kCorrRows = 768;           // token rows of one segment per CTA (4 strips per warp)
constexpr int kStrip = 16 * kD;          // one 16-row strip of z or o in shared memory (bf16)
constexpr size_t kCorrSmem = (size_t)(kD * kD + kCorrWarps * 4 * kStrip) * sizeof(__nv_bfloat16);

// Shared-memory tiles of 128 bf16 per row (16 chunks of 16 bytes) store
// chunk c of row r at chunk c ^ (r & 7): the 8 rows an ldmatrix phase or a
// fragment read touches then sit in 8 different bank groups.
__device__ __forceinline__ int swz(int r, int c8) { return r * kD + ((((c8 >> 3) ^ r) & 7) | ((c8 >> 3) & 8)) * 8 + (c8 & 7); }

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(const __nv_bfloat16 *p, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}

// o_t += S_start,g^T z_t for the tokens of segments 1..G-1: per head a
// [rows x 128] x [128 x 128] product. CTA (x, g - 1, h) takes rows
// [x * kCorrRows, +kCorrRows) of segment g and holds S_start,g^T in shared
// memory; each warp takes 16-row strips. The z and o rows of the next strip
// are copied in (cp.async, 16 bytes a lane) while the current strip is
// multiplied; the products accumulate in float32 onto o, are rounded to bf16
// once, and leave through shared memory as 16-byte stores. Segments start at
// multiples of 64 tokens, so a strip never spans two. Rows past the segment
// are neither copied nor stored (each output row depends on its own z row
// only).
__global__ void __launch_bounds__(kCorrWarps * 32)
seg_correct_kernel(const __nv_bfloat16 *__restrict__ z, const __nv_bfloat16 *__restrict__ sst,
                   __nv_bfloat16 *__restrict__ o, int H, int len_tokens, int T1) {
    extern __shared__ __align__(16) unsigned char corr_smem[];
    __nv_bfloat16 *Bs = reinterpret_cast<__nv_bfloat16 *>(corr_smem);  // [128 value columns][128], swizzled
    const int g1 = blockIdx.y, h = blockIdx.z;
    const int seg_lo = g1 * len_tokens;
    const int seg_hi = min(T1, seg_lo + len_tokens);
    const int row_lo = seg_lo + blockIdx.x * kCorrRows;
    if (row_lo >= seg_hi) return;
    const int row_hi = min(seg_hi, row_lo + kCorrRows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    // this warp's buffers: z strips [2], o strips [2]
    __nv_bfloat16 *Zs = Bs + kD * kD + warp * 4 * kStrip;
    __nv_bfloat16 *Os = Zs + 2 * kStrip;
    const size_t row_stride = (size_t)H * kD;  // elements from one token to the next
    const __nv_bfloat16 *zh = z + (size_t)h * kD;
    __nv_bfloat16 *oh = o + (size_t)h * kD;

    const __nv_bfloat16 *src = sst + ((size_t)g1 * H + h) * kD * kD;
    for (int e = threadIdx.x; e < kD * kD / 8; e += kCorrWarps * 32) {
        const int r = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
        cp16(&Bs[swz(r, c8)], &src[r * kD + c8]);
    }
    cp_commit();

    auto issue = [&](int r0, int buf) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = lane + 32 * j, r = c >> 4, c8 = (c & 15) * 8;
            if (r0 + r < row_hi) {
                const size_t at = (size_t)(r0 + r) * row_stride + c8;
                cp16(Zs + buf * kStrip + swz(r, c8), zh + at);
                cp16(Os + buf * kStrip + swz(r, c8), oh + at);
            }
        }
        cp_commit();
    };
    const int first = row_lo + warp * 16;
    if (first < row_hi) issue(first, 0);
    else cp_commit();
    cp_wait1();  // S_start^T landed (this thread's part)
    __syncthreads();

    int buf = 0;
    for (int r0 = first; r0 < row_hi; r0 += kCorrWarps * 16, buf ^= 1) {
        const int rn = r0 + kCorrWarps * 16;
        if (rn < row_hi) issue(rn, buf ^ 1);
        else cp_commit();
        cp_wait1();
        __syncwarp();
        __nv_bfloat16 *ob = Os + buf * kStrip;
        // the accumulators start from o
        float acc[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = nt * 8 + 2 * tq;
            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(ob + swz(gq, c)));
            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(ob + swz(gq + 8, c)));
            acc[nt][0] = fa.x;
            acc[nt][1] = fa.y;
            acc[nt][2] = fb.x;
            acc[nt][3] = fb.y;
        }
        const __nv_bfloat16 *zb = Zs + buf * kStrip;
        const int ar = lane & 15, ak = (lane >> 4) * 8;                         // A: this lane's row, k offset
        const int br = (lane >> 4) * 8 + (lane & 7), bk = ((lane >> 3) & 1) * 8;  // B: row (value column), k offset
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(zb + swz(ar, ks * 16 + ak), a);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t b[4];
                ldsm_x4(Bs + swz(np * 16 + br, ks * 16 + bk), b);
                mma_bf16_16816(acc[2 * np], a, b[0], b[1]);
                mma_bf16_16816(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = nt * 8 + 2 * tq;
            *reinterpret_cast<__nv_bfloat162 *>(ob + swz(gq, c)) = __floats2bfloat162_rn(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<__nv_bfloat162 *>(ob + swz(gq + 8, c)) = __floats2bfloat162_rn(acc[nt][2], acc[nt][3]);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = lane + 32 * j, r = c >> 4, c8 = (c & 15) * 8;
            if (r0 + r < row_hi)
                *reinterpret_cast<uint4 *>(oh + (size_t)(r0 + r) * row_stride + c8) =
                    *reinterpret_cast<const uint4 *>(ob + swz(r, c8));
        }
        __syncwarp();  // both buffers of this strip are refilled two strips on
    }
}

// ---------------------------------------------------------------------------
// Streams of the split (created once per device)
// ---------------------------------------------------------------------------

struct Streams {
    bool ready = false;
    cudaStream_t hi = nullptr, a = nullptr, b = nullptr;
    cudaEvent_t fork = nullptr, hi_done = nullptr, a_done = nullptr, b_done = nullptr;
};

std::mutex g_mu;
Streams g_streams[kMaxDevices];

cudaError_t make_streams(Streams &s) {
    cudaError_t e;
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&s.hi, cudaStreamNonBlocking, greatest)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&s.a, cudaStreamNonBlocking, least)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&s.b, cudaStreamNonBlocking, least)) != cudaSuccess) return e;
    cudaEvent_t *evs[] = {&s.fork, &s.hi_done, &s.a_done, &s.b_done};
    for (cudaEvent_t *ev : evs)
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    s.ready = true;
    return cudaSuccess;
}

}  // namespace

extern "C" {

kda_status_t kda_prefill_segment_plan(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype, int segments,
                                      int *n_segments, int *first_tokens, int *segment_tokens) {
    if (!n_segments || !first_tokens || !segment_tokens)
        return fail(KDA_ERR_INVALID_ARG, "n_segments, first_tokens, segment_tokens must not be NULL");
    if (B < 0 || T < 0 || H <= 0 || segments < 0)
        return fail(KDA_ERR_INVALID_ARG, "B, T, segments must be >= 0 and H > 0");
    if (segments > 1 && !splittable(B, d_k, d_v, qkv_dtype))
        return fail(KDA_ERR_UNSUPPORTED, "a split needs B = 1, bf16 q/k/v and d_k = d_v = 128");
    // (the correction's grid holds the heads in z and the segments in y)
    if (segments > 1 && (H > 65535 || segments > kMaxForced))
        return fail(KDA_ERR_UNSUPPORTED, "a split needs H <= 65535 and at most %d segments", kMaxForced);
    const Plan p = make_plan(B, T, H, d_k, d_v, qkv_dtype, segments);
    *n_segments = p.G;
    *first_tokens = p.G > 1 ? p.first * kC : T;
    *segment_tokens = p.G > 1 ? p.len * kC : 0;
    return KDA_OK;
}

size_t kda_prefill_segmented_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype,
                                             int segments) {
    if (B < 0 || T < 0 || H <= 0 || segments < 0) return 0;
    return layout(make_plan(B, T, H, d_k, d_v, qkv_dtype, segments), T, H).total;
}

kda_status_t kda_prefill_segmented(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                   const float *alpha, kda_gate_t gate, const float *beta,
                                   const float *initial_state, void *o, float *final_state, int B, int T, int H,
                                   int d_k, int d_v, int segments, void *workspace, size_t workspace_bytes,
                                   kda_stream_t stream) {
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_SCALAR && gate != KDA_GATE_NONE)
        return fail(KDA_ERR_INVALID_ARG, "unknown gate kind %d", (int)gate);
    int G = 1, first = 0, seg = 0;
    kda_status_t st = kda_prefill_segment_plan(B, T, H, d_k, d_v, qkv_dtype, segments, &G, &first, &seg);
    if (st != KDA_OK) return st;
    if (G < 2)
        return kda_prefill_gate(q, k, v, qkv_dtype, alpha, gate, beta, initial_state, o, final_state, B, T, H, d_k,
                                d_v, KDA_ALGO_AUTO, stream);
    // the pointer checks of the plain call
    const void *need16[] = {q, k, v, o};
    const char *names[] = {"q", "k", "v", "o"};
    for (int i = 0; i < 4; ++i) {
        if (!need16[i]) return fail(KDA_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
        if (reinterpret_cast<uintptr_t>(need16[i]) & 15u)
            return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned", names[i]);
    }
    if (gate != KDA_GATE_NONE) {
        if (!alpha) return fail(KDA_ERR_INVALID_ARG, "alpha must not be NULL");
        if (reinterpret_cast<uintptr_t>(alpha) & (gate == KDA_GATE_CHANNEL ? 15u : 3u))
            return fail(KDA_ERR_INVALID_ARG, "alpha must be %d-byte aligned", gate == KDA_GATE_CHANNEL ? 16 : 4);
    }
    if (!beta) return fail(KDA_ERR_INVALID_ARG, "beta must not be NULL");
    if (reinterpret_cast<uintptr_t>(beta) & 3u) return fail(KDA_ERR_INVALID_ARG, "beta must be 4-byte aligned");
    if ((reinterpret_cast<uintptr_t>(initial_state) | reinterpret_cast<uintptr_t>(final_state)) & 15u)
        return fail(KDA_ERR_INVALID_ARG, "initial_state and final_state must be 16-byte aligned");
    const Plan p = make_plan(B, T, H, d_k, d_v, qkv_dtype, segments);
    const Layout L = layout(p, T, H);
    if (!workspace || workspace_bytes < L.total)
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", L.total, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return fail(KDA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KDA_ERR_UNSUPPORTED, "device index %d out of range", dev);

    std::lock_guard<std::mutex> lock(g_mu);
    Streams &S = g_streams[dev];
    if (!S.ready && (e = make_streams(S)) != cudaSuccess) return cuda_fail(e, "creating the segment streams");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    char *ws = static_cast<char *>(workspace);
    int32_t *cu = reinterpret_cast<int32_t *>(ws + L.cu);
    float *fs0 = reinterpret_cast<float *>(ws + L.fs0);
    float *fs1 = reinterpret_cast<float *>(ws + L.fs1);
    float *ident = reinterpret_cast<float *>(ws + L.ident);
    float *phi = reinterpret_cast<float *>(ws + L.phi);
    __nv_bfloat16 *sst = reinterpret_cast<__nv_bfloat16 *>(ws + L.sst);
    __nv_bfloat16 *zv = reinterpret_cast<__nv_bfloat16 *>(ws + L.zv);
    __nv_bfloat16 *zz = reinterpret_cast<__nv_bfloat16 *>(ws + L.z);
    const int64_t t1 = (int64_t)first;  // first token of segment 1
    const size_t row = (size_t)H * kD;  // elements per token row of q, k, v, o, alpha
    const char *q1 = static_cast<const char *>(q) + t1 * row * sizeof(__nv_bfloat16);
    const char *k1 = static_cast<const char *>(k) + t1 * row * sizeof(__nv_bfloat16);
    const char *v1 = static_cast<const char *>(v) + t1 * row * sizeof(__nv_bfloat16);
    char *o1 = static_cast<char *>(o) + t1 * row * sizeof(__nv_bfloat16);
    const float *a1 = gate == KDA_GATE_CHANNEL ? alpha + t1 * row : gate == KDA_GATE_SCALAR ? alpha + t1 * H : nullptr;
    const float *b1 = beta + t1 * H;
    const int G1 = G - 1, T1 = (int)L.T1;

    // every step is checked; after a failure the joins still run, so the
    // caller's stream waits for whatever was queued
    st = KDA_OK;
    auto q_ok = [&](cudaError_t err, const char *what) {
        if (err != cudaSuccess && st == KDA_OK) st = cuda_fail(err, what);
        return st == KDA_OK;
    };
    auto k_ok = [&](kda_status_t r) {
        if (r != KDA_OK && st == KDA_OK) st = r;
        return st == KDA_OK;
    };
    if (q_ok(cudaEventRecord(S.fork, s), "event record") && q_ok(cudaStreamWaitEvent(S.hi, S.fork, 0), "wait") &&
        q_ok(cudaStreamWaitEvent(S.a, S.fork, 0), "wait") && q_ok(cudaStreamWaitEvent(S.b, S.fork, 0), "wait")) {
        // segment 0 from the caller's initial state
        k_ok(kda_prefill_gate(q, k, v, KDA_BF16, alpha, gate, beta, initial_state, o, fs0, 1, first, H, kD, kD,
                              KDA_ALGO_TC, reinterpret_cast<kda_stream_t>(S.hi)));
        // the transition runs' v: zeros
        if (st == KDA_OK)
            q_ok(cudaMemsetAsync(zv, 0, (size_t)T1 * row * sizeof(__nv_bfloat16), S.b), "zeroing v");
        // segments 1..G-1: cu_seqlens and identities, then the local runs, then
        // the transition runs
        if (st == KDA_OK) {
            const int64_t nv4 = (int64_t)G1 * H * kD * kD / 4;
            const int64_t n = nv4 > G ? nv4 : G;
            seg_setup_kernel<<<(unsigned)((n + 255) / 256), 256, 0, S.a>>>(cu, G1 + 1, seg, T1,
                                                                          reinterpret_cast<float4 *>(ident), nv4);
            q_ok(cudaGetLastError(), "segment setup launch");
        }
        void *vlws = ws + L.vlws;
        const size_t vlbytes = kda_varlen_workspace_bytes(G1, H, kD, kD);
        if (st == KDA_OK)
            k_ok(kda::varlen_prefill_gate(q1, k1, v1, KDA_BF16, a1, gate, b1, nullptr, o1, fs1, cu, G1, T1, H, kD,
                                          kD, vlws, vlbytes, nullptr, S.a));
        if (st == KDA_OK) q_ok(cudaEventRecord(S.b_done, S.b), "event record");
        if (st == KDA_OK) q_ok(cudaStreamWaitEvent(S.a, S.b_done, 0), "wait");
        if (st == KDA_OK)
            k_ok(kda::varlen_prefill_gate(q1, k1, zv, KDA_BF16, a1, gate, b1, ident, zz, phi, cu, G1, T1, H, kD,
                                          kD, vlws, vlbytes, nullptr, S.a));
    }
    // joins (always, so that nothing queued outlives the call's stream order)
    cudaError_t j1 = cudaEventRecord(S.hi_done, S.hi);
    cudaError_t j2 = cudaEventRecord(S.a_done, S.a);
    cudaError_t j3 = cudaEventRecord(S.b_done, S.b);
    if (j1 == cudaSuccess) j1 = cudaStreamWaitEvent(s, S.hi_done, 0);
    if (j2 == cudaSuccess) j2 = cudaStreamWaitEvent(s, S.a_done, 0);
    if (j3 == cudaSuccess) j3 = cudaStreamWaitEvent(s, S.b_done, 0);
    q_ok(j1, "join");
    q_ok(j2, "join");
    q_ok(j3, "join");
    if (st != KDA_OK) return st;

    {
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "SM count");
        // one CTA per SM (two Phi buffers): 16 columns per CTA while H x 8 CTAs fit at once
        const bool narrow = (int64_t)H * (kD / 16) <= sms;
        auto kern = narrow ? seg_combine_kernel<16> : seg_combine_kernel<32>;
        const size_t smem = narrow ? comb_smem<16>() : comb_smem<32>();
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e, "combine attribute");
        kern<<<dim3(H, narrow ? kD / 16 : kD / 32), kCombThreads, smem, s>>>(fs0, fs1, phi, sst, final_state, G, H);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "combine launch");
    e = cudaFuncSetAttribute(seg_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCorrSmem);
    if (e != cudaSuccess) return cuda_fail(e, "correction attribute");
    const unsigned xs = (unsigned)((seg + kCorrRows - 1) / kCorrRows);
    seg_correct_kernel<<<dim3(xs, G1, H), kCorrWarps * 32, kCorrSmem, s>>>(
        zz, sst, static_cast<__nv_bfloat16 *>((void *)o1), H, seg, T1);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "correction launch");
    return KDA_OK;
}

}  // extern "C"
