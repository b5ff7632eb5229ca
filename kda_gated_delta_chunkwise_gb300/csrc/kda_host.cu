// Prefill on host buffers (kda_prefill_host): the tokens travel to the GPU in
// pieces along T and the outputs come back piece by piece, so the host link,
// the kernels and the copies back overlap. The state between pieces stays on
// the device; each piece is one kda_prefill_gate call that starts from the
// state the previous piece left (the chunk-to-chunk passing of the K3 essay
// §六.1, carried across calls).
//
// Streams: the kernels run on the caller's stream; the copies to the device run
// on one internal stream and the copies back on another (created once per
// device). Events tie them: a piece's kernel waits for its inputs, its inputs
// wait for the kernel that last used their ring slot, its copy back waits for
// its kernel. The caller's stream waits for the last copy back, so the call is
// ordered on the caller's stream like any kernel launch.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "kda_internal.cuh"

namespace {

constexpr int kRing = 3;                      // piece buffers in flight
constexpr size_t kAlign = 256;
constexpr int64_t kPieceBytes = 32ll << 20;   // input bytes per piece when the caller leaves it open
constexpr size_t kMaxPitch = size_t(1) << 30;  // larger row pitches are copied row by row
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

// Bytes of one token row (all heads) of each tensor.
struct Rows {
    size_t qk, v, a, b, o;
};

Rows row_bytes(int H, int dk, int dv, kda_dtype_t dt, kda_gate_t gate) {
    const size_t es = dt == KDA_BF16 ? 2 : 4;
    Rows r;
    r.qk = (size_t)H * dk * es;
    r.v = (size_t)H * dv * es;
    r.a = gate == KDA_GATE_CHANNEL ? (size_t)H * dk * 4 : gate == KDA_GATE_SCALAR ? (size_t)H * 4 : 0;
    r.b = (size_t)H * 4;
    r.o = (size_t)H * dv * es;
    return r;
}

// Tokens per piece: the caller's choice, else about kPieceBytes of input per
// piece, in whole chunks.
int64_t piece_tokens_for(int B, int T, const Rows &r, int piece_tokens) {
    if (T <= 0) return 0;
    int64_t pt = piece_tokens;
    if (pt == 0) {
        const int64_t per_tok = (int64_t)B * (int64_t)(2 * r.qk + r.v + r.a + r.b);
        const int64_t pieces = (T * per_tok + kPieceBytes - 1) / kPieceBytes;
        const int64_t len = (T + (pieces > 0 ? pieces : 1) - 1) / (pieces > 0 ? pieces : 1);
        pt = (len + 63) / 64 * 64;
    }
    return pt < T ? pt : T;  // buffers hold at most T tokens
}

struct Layout {
    size_t q, k, v, a, b, o, slot, state, total;
};

Layout layout(int B, int64_t cap, int H, int dk, int dv, const Rows &r) {
    Layout l;
    const size_t n = (size_t)B * (size_t)cap;
    l.q = 0;
    l.k = l.q + align_up(n * r.qk);
    l.v = l.k + align_up(n * r.qk);
    l.a = l.v + align_up(n * r.v);
    l.b = l.a + align_up(n * r.a);
    l.o = l.b + align_up(n * r.b);
    l.slot = l.o + align_up(n * r.o);
    l.state = kRing * l.slot;
    l.total = l.state + align_up((size_t)B * H * dk * dv * sizeof(float));
    return l;
}

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, copied[kRing] = {}, ran[kRing] = {}, sent[kRing] = {};
};

std::mutex g_mu;
Pipe g_pipe[kMaxDevices];

cudaError_t make_pipe(Pipe &p) {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t *evs[] = {&p.start, &p.done};
    for (cudaEvent_t *ev : evs)
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < kRing; ++i) {
        if ((e = cudaEventCreateWithFlags(&p.copied[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.ran[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.sent[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    p.ready = true;
    return cudaSuccess;
}

// `rows` rows of `width` bytes; one 2D copy when the pitches allow it.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, int rows,
                      cudaStream_t s) {
    if (width == 0 || rows == 0) return cudaSuccess;
    if (rows > 1 && dpitch <= kMaxPitch && spitch <= kMaxPitch)
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, cudaMemcpyDefault, s);
    for (int r = 0; r < rows; ++r) {
        cudaError_t e = cudaMemcpyAsync(static_cast<char *>(dst) + r * dpitch,
                                        static_cast<const char *>(src) + r * spitch, width, cudaMemcpyDefault, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// A caller buffer that must live in host memory (pinned, registered or pageable).
kda_status_t need_host(const void *p, const char *name) {
    if (!p) return KDA_OK;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) return cuda_fail(e, "pointer query");
    if (at.type == cudaMemoryTypeDevice)
        return fail(KDA_ERR_INVALID_ARG, "%s must be a host pointer (got device memory)", name);
    return KDA_OK;
}

bool valid_args(kda_dtype_t dt, kda_gate_t gate, int B, int T, int H, int dk, int dv, int piece_tokens) {
    return (dt == KDA_F32 || dt == KDA_BF16) &&
           (gate == KDA_GATE_CHANNEL || gate == KDA_GATE_SCALAR || gate == KDA_GATE_NONE) && B >= 0 && T >= 0 &&
           H > 0 && (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && piece_tokens >= 0 &&
           piece_tokens % 64 == 0 && (int64_t)B * T <= INT32_MAX;
}

}  // namespace

extern "C" {

size_t kda_prefill_host_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype,
                                        kda_gate_t gate, int piece_tokens) {
    if (!valid_args(qkv_dtype, gate, B, T, H, d_k, d_v, piece_tokens)) return 0;
    const Rows r = row_bytes(H, d_k, d_v, qkv_dtype, gate);
    return layout(B, piece_tokens_for(B, T, r, piece_tokens), H, d_k, d_v, r).total;
}

kda_status_t kda_prefill_host(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                              const float *alpha, kda_gate_t gate, const float *beta,
                              const float *initial_state, void *o, float *final_state, int B, int T,
                              int H, int d_k, int d_v, kda_algo_t algo, int piece_tokens, void *workspace,
                              size_t workspace_bytes, kda_stream_t stream) {
    // ---- argument checks, before any CUDA call
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16)
        return fail(KDA_ERR_INVALID_ARG, "unknown qkv dtype %d", (int)qkv_dtype);
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_SCALAR && gate != KDA_GATE_NONE)
        return fail(KDA_ERR_INVALID_ARG, "unknown gate kind %d", (int)gate);
    if (algo != KDA_ALGO_AUTO && algo != KDA_ALGO_SIMT && algo != KDA_ALGO_TC)
        return fail(KDA_ERR_INVALID_ARG, "unknown algo %d", (int)algo);
    if (H <= 0 || d_k <= 0 || d_v <= 0) return fail(KDA_ERR_INVALID_ARG, "H, d_k, d_v must be positive");
    if ((d_k != 64 && d_k != 128) || (d_v != 64 && d_v != 128))
        return fail(KDA_ERR_UNSUPPORTED, "d_k, d_v must be 64 or 128 (got %d, %d)", d_k, d_v);
    if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B and T must be >= 0 (got %d, %d)", B, T);
    if ((int64_t)B * T > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "B * T must fit in int32");
    if (piece_tokens < 0 || piece_tokens % 64 != 0)
        return fail(KDA_ERR_INVALID_ARG, "piece_tokens must be 0 or a positive multiple of 64 (got %d)",
                    piece_tokens);
    const bool any = (int64_t)B * T > 0;
    if (any) {
        if (!q || !k || !v || !beta || !o) return fail(KDA_ERR_INVALID_ARG, "q, k, v, beta and o must not be NULL");
        if (gate != KDA_GATE_NONE && !alpha) return fail(KDA_ERR_INVALID_ARG, "alpha must not be NULL");
    }
    if (B == 0 || (T == 0 && !final_state)) return KDA_OK;
    const Rows r = row_bytes(H, d_k, d_v, qkv_dtype, gate);
    const int64_t piece = piece_tokens_for(B, T, r, piece_tokens);
    const Layout L = layout(B, piece, H, d_k, d_v, r);
    if (!workspace || workspace_bytes < L.total)
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes needed (kda_prefill_host_workspace_bytes)", L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return fail(KDA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    // ---- buffers: host inputs and outputs, device workspace
    kda_status_t st;
    const void *hosts[] = {q, k, v, alpha, beta, initial_state, o, final_state};
    const char *names[] = {"q", "k", "v", "alpha", "beta", "initial_state", "o", "final_state"};
    for (int i = 0; i < 8; ++i)
        if ((st = need_host(hosts[i], names[i])) != KDA_OK) return st;
    cudaPointerAttributes wat;
    cudaError_t e = cudaPointerGetAttributes(&wat, workspace);
    if (e != cudaSuccess) return cuda_fail(e, "pointer query");
    if (wat.type != cudaMemoryTypeDevice) return fail(KDA_ERR_INVALID_ARG, "workspace must be device memory");
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KDA_ERR_UNSUPPORTED, "device index %d out of range", dev);
    if (wat.device != dev) return fail(KDA_ERR_INVALID_ARG, "workspace is not on the current device");

    std::lock_guard<std::mutex> lock(g_mu);
    Pipe &p = g_pipe[dev];
    if (!p.ready && (e = make_pipe(p)) != cudaSuccess) return cuda_fail(e, "creating the copy streams");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    float *state = reinterpret_cast<float *>(ws + L.state);
    const size_t state_bytes = (size_t)B * H * d_k * d_v * sizeof(float);

    // every queued step below is checked; on a failure the caller's stream
    // still waits for what was queued, so the workspace stays owned until then
    st = KDA_OK;
    auto q_ok = [&](cudaError_t err, const char *what) {
        if (err != cudaSuccess && st == KDA_OK) st = cuda_fail(err, what);
        return st == KDA_OK;
    };
    if (q_ok(cudaEventRecord(p.start, s), "event record") && q_ok(cudaStreamWaitEvent(p.in, p.start, 0), "wait") &&
        q_ok(cudaStreamWaitEvent(p.out, p.start, 0), "wait") && initial_state)
        q_ok(cudaMemcpyAsync(state, initial_state, state_bytes, cudaMemcpyDefault, p.in), "initial state copy");
    const int64_t npieces = T > 0 ? (T + piece - 1) / piece : 1;
    for (int64_t i = 0; i < npieces && st == KDA_OK; ++i) {
        const int slot = (int)(i % kRing);
        const int64_t t0 = i * piece;
        const int len = (int)(T > 0 ? (T - t0 < piece ? T - t0 : piece) : 0);
        char *b = ws + slot * L.slot;
        // inputs of piece i into ring slot i % kRing, once the kernel that read
        // that slot before (piece i - kRing) is done
        if (i >= kRing && !q_ok(cudaStreamWaitEvent(p.in, p.ran[slot], 0), "wait")) break;
        const struct {
            size_t off;
            const void *src;
            size_t row;
        } ins[] = {{L.q, q, r.qk}, {L.k, k, r.qk}, {L.v, v, r.v}, {L.a, alpha, r.a}, {L.b, beta, r.b}};
        for (const auto &x : ins)
            if (x.src && x.row && !q_ok(copy_rows(b + x.off, (size_t)len * x.row,
                                                  static_cast<const char *>(x.src) + t0 * x.row, (size_t)T * x.row,
                                                  (size_t)len * x.row, B, p.in),
                                        "host-to-device copy"))
                break;
        if (!q_ok(cudaEventRecord(p.copied[slot], p.in), "event record")) break;
        // the kernel of piece i: from the state the previous piece left (or the
        // caller's initial state), into the same state buffer
        if (!q_ok(cudaStreamWaitEvent(s, p.copied[slot], 0), "wait")) break;
        if (i >= kRing && !q_ok(cudaStreamWaitEvent(s, p.sent[slot], 0), "wait")) break;
        const float *s0 = (i == 0 && !initial_state) ? nullptr : state;
        st = kda_prefill_gate(b + L.q, b + L.k, b + L.v, qkv_dtype, gate == KDA_GATE_NONE ? nullptr : (const float *)(b + L.a),
                              gate, (const float *)(b + L.b), s0, b + L.o, state, B, len, H, d_k, d_v, algo, stream);
        if (st != KDA_OK) break;
        if (!q_ok(cudaEventRecord(p.ran[slot], s), "event record")) break;
        // outputs of piece i back to the host
        if (!q_ok(cudaStreamWaitEvent(p.out, p.ran[slot], 0), "wait")) break;
        if (!q_ok(copy_rows(static_cast<char *>(o) + t0 * r.o, (size_t)T * r.o, b + L.o, (size_t)len * r.o,
                            (size_t)len * r.o, B, p.out),
                  "device-to-host copy"))
            break;
        if (i == npieces - 1 && final_state &&
            !q_ok(cudaMemcpyAsync(final_state, state, state_bytes, cudaMemcpyDefault, p.out), "final state copy"))
            break;
        if (!q_ok(cudaEventRecord(p.sent[slot], p.out), "event record")) break;
    }
    // the caller's stream continues once the last copy back is done
    cudaError_t e1 = cudaEventRecord(p.done, p.out);
    cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(s, p.done, 0) : e1;
    if (st != KDA_OK) return st;
    if (e2 != cudaSuccess) return cuda_fail(e2, "joining the copy streams");
    return KDA_OK;
}

}  // extern "C"
