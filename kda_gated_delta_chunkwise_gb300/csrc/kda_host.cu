// Prefill on host buffers (kda_prefill_host, kda_prefill_fp8_host): the tokens
// travel to the GPU in pieces along T and the outputs come back piece by
// piece, so the host link, the kernels and the copies back overlap. The state
// between pieces stays on the device; each piece is one device prefill call
// that starts from the state the previous piece left (the chunk-to-chunk
// passing of the K3 essay §六.1, carried across calls).
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

#include "kda_internal.cuh"

namespace {

constexpr int kRing = 3;                       // piece buffers in flight
constexpr size_t kAlign = 256;
constexpr int64_t kPieceBytes = 32ll << 20;    // input bytes per piece when the caller leaves it open
constexpr size_t kMaxPitch = size_t(1) << 30;  // larger row pitches are copied row by row
constexpr int kMaxDevices = 64;
constexpr int kMaxInputs = 8;

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

// One host-to-device stream of token rows: the caller's host tensor and the
// bytes of one token row (all heads). A tensor the call does not use has
// row = 0 (no buffer, no copy).
struct In {
    const void *src;
    size_t row;
};

// The tensors of one call: inputs in the order the launcher expects them,
// the output row (o), the state size.
struct Plan {
    In in[kMaxInputs];
    int nin;
    size_t orow, state_bytes;
};

// Tokens per piece: the caller's choice, else about kPieceBytes of input per
// piece, in whole chunks.
int64_t piece_tokens_for(const Plan &pl, int B, int T, int piece_tokens) {
    if (T <= 0) return 0;
    int64_t pt = piece_tokens;
    if (pt == 0) {
        size_t row = 0;
        for (int i = 0; i < pl.nin; ++i) row += pl.in[i].row;
        const int64_t per_tok = (int64_t)B * (int64_t)row;
        int64_t pieces = (T * per_tok + kPieceBytes - 1) / kPieceBytes;
        if (pieces < 1) pieces = 1;
        const int64_t len = (T + pieces - 1) / pieces;
        pt = (len + 63) / 64 * 64;
    }
    return pt < T ? pt : T;  // buffers hold at most T tokens
}

// Workspace: kRing slots of [inputs..., o], then the state.
struct Layout {
    size_t in[kMaxInputs], o, slot, state, total;
};

Layout layout(const Plan &pl, int B, int64_t cap) {
    Layout l;
    const size_t n = (size_t)B * (size_t)cap;
    size_t off = 0;
    for (int i = 0; i < pl.nin; ++i) {
        l.in[i] = off;
        off += align_up(n * pl.in[i].row);
    }
    l.o = off;
    l.slot = off + align_up(n * pl.orow);
    l.state = kRing * l.slot;
    l.total = l.state + align_up(pl.state_bytes);
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

// Launch of one piece: device buffers of the inputs (in Plan order), the
// piece's tokens, the state to start from (NULL: zeros) and the state buffer
// to write, on the caller's stream.
struct Launcher {
    virtual kda_status_t operator()(char *const in[], void *o, int len, const float *s0, float *state,
                                    kda_stream_t s) const = 0;
};

// The pipeline shared by the host entry points; arguments already checked
// except the workspace and the memory kinds.
kda_status_t run_host(const Plan &pl, const char *const *names, const float *initial_state, void *o,
                      float *final_state, int B, int T, int piece_tokens, void *workspace, size_t workspace_bytes,
                      kda_stream_t stream, const Launcher &launch) {
    const int64_t piece = piece_tokens_for(pl, B, T, piece_tokens);
    const Layout L = layout(pl, B, piece);
    if (!workspace || workspace_bytes < L.total)
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes needed (the call's workspace_bytes function)", L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return fail(KDA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    kda_status_t st;
    for (int i = 0; i < pl.nin; ++i)
        if ((st = need_host(pl.in[i].src, names[i])) != KDA_OK) return st;
    if ((st = need_host(initial_state, "initial_state")) != KDA_OK) return st;
    if ((st = need_host(o, "o")) != KDA_OK) return st;
    if ((st = need_host(final_state, "final_state")) != KDA_OK) return st;
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

    // every queued step below is checked; on a failure the caller's stream
    // still waits for what was queued, so the workspace stays owned until then
    st = KDA_OK;
    auto q_ok = [&](cudaError_t err, const char *what) {
        if (err != cudaSuccess && st == KDA_OK) st = cuda_fail(err, what);
        return st == KDA_OK;
    };
    if (q_ok(cudaEventRecord(p.start, s), "event record") && q_ok(cudaStreamWaitEvent(p.in, p.start, 0), "wait") &&
        q_ok(cudaStreamWaitEvent(p.out, p.start, 0), "wait") && initial_state)
        q_ok(cudaMemcpyAsync(state, initial_state, pl.state_bytes, cudaMemcpyDefault, p.in), "initial state copy");
    const int64_t npieces = T > 0 ? (T + piece - 1) / piece : 1;
    for (int64_t i = 0; i < npieces && st == KDA_OK; ++i) {
        const int slot = (int)(i % kRing);
        const int64_t t0 = i * piece;
        const int len = (int)(T > 0 ? (T - t0 < piece ? T - t0 : piece) : 0);
        char *b = ws + slot * L.slot;
        // inputs of piece i into ring slot i % kRing, once the kernel that read
        // that slot before (piece i - kRing) is done
        if (i >= kRing && !q_ok(cudaStreamWaitEvent(p.in, p.ran[slot], 0), "wait")) break;
        char *bufs[kMaxInputs];
        for (int j = 0; j < pl.nin; ++j) {
            const In &x = pl.in[j];
            bufs[j] = x.row ? b + L.in[j] : nullptr;
            if (x.src && x.row &&
                !q_ok(copy_rows(bufs[j], (size_t)len * x.row, static_cast<const char *>(x.src) + t0 * x.row,
                                (size_t)T * x.row, (size_t)len * x.row, B, p.in),
                      "host-to-device copy"))
                break;
        }
        if (!q_ok(cudaEventRecord(p.copied[slot], p.in), "event record")) break;
        // the kernel of piece i: from the state the previous piece left (or the
        // caller's initial state), into the same state buffer
        if (!q_ok(cudaStreamWaitEvent(s, p.copied[slot], 0), "wait")) break;
        if (i >= kRing && !q_ok(cudaStreamWaitEvent(s, p.sent[slot], 0), "wait")) break;
        const float *s0 = (i == 0 && !initial_state) ? nullptr : state;
        if ((st = launch(bufs, b + L.o, len, s0, state, stream)) != KDA_OK) break;
        if (!q_ok(cudaEventRecord(p.ran[slot], s), "event record")) break;
        // outputs of piece i back to the host
        if (!q_ok(cudaStreamWaitEvent(p.out, p.ran[slot], 0), "wait")) break;
        if (!q_ok(copy_rows(static_cast<char *>(o) + t0 * pl.orow, (size_t)T * pl.orow, b + L.o,
                            (size_t)len * pl.orow, (size_t)len * pl.orow, B, p.out),
                  "device-to-host copy"))
            break;
        if (i == npieces - 1 && final_state &&
            !q_ok(cudaMemcpyAsync(final_state, state, pl.state_bytes, cudaMemcpyDefault, p.out), "final state copy"))
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

bool valid_gate(int gate) { return gate == KDA_GATE_CHANNEL || gate == KDA_GATE_SCALAR || gate == KDA_GATE_NONE; }

size_t alpha_row(kda_gate_t gate, int H, int dk) {
    return gate == KDA_GATE_CHANNEL ? (size_t)H * dk * 4 : gate == KDA_GATE_SCALAR ? (size_t)H * 4 : 0;
}

// ---- kda_prefill_host: q, k, v in qkv_dtype
Plan plan_plain(const void *q, const void *k, const void *v, kda_dtype_t dt, const float *alpha, kda_gate_t gate,
                const float *beta, int B, int H, int dk, int dv) {
    const size_t es = dt == KDA_BF16 ? 2 : 4;
    Plan pl{};
    pl.nin = 5;
    pl.in[0] = {q, (size_t)H * dk * es};
    pl.in[1] = {k, (size_t)H * dk * es};
    pl.in[2] = {v, (size_t)H * dv * es};
    pl.in[3] = {alpha, alpha_row(gate, H, dk)};
    pl.in[4] = {beta, (size_t)H * 4};
    pl.orow = (size_t)H * dv * es;
    pl.state_bytes = (size_t)B * H * dk * dv * sizeof(float);
    return pl;
}
const char *const kPlainNames[] = {"q", "k", "v", "alpha", "beta"};

struct PlainLauncher : Launcher {
    kda_dtype_t dt;
    kda_gate_t gate;
    kda_algo_t algo;
    int B, H, dk, dv;
    kda_status_t operator()(char *const in[], void *o, int len, const float *s0, float *state,
                            kda_stream_t s) const override {
        return kda_prefill_gate(in[0], in[1], in[2], dt, reinterpret_cast<const float *>(in[3]), gate,
                                reinterpret_cast<const float *>(in[4]), s0, o, state, B, len, H, dk, dv, algo, s);
    }
};

bool valid_plain(kda_dtype_t dt, kda_gate_t gate, int B, int T, int H, int dk, int dv, int piece_tokens) {
    return (dt == KDA_F32 || dt == KDA_BF16) && valid_gate(gate) && B >= 0 && T >= 0 && H > 0 &&
           (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && piece_tokens >= 0 && piece_tokens % 64 == 0 &&
           (int64_t)B * T <= INT32_MAX;
}

// ---- kda_prefill_fp8_host: E4M3 codes and E8M0 block scales
Plan plan_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *qs, const uint8_t *ks,
              const uint8_t *vs, const float *alpha, kda_gate_t gate, const float *beta, int B, int H, int dk,
              int dv) {
    Plan pl{};
    pl.nin = 8;
    pl.in[0] = {q, (size_t)H * dk};
    pl.in[1] = {k, (size_t)H * dk};
    pl.in[2] = {v, (size_t)H * dv};
    pl.in[3] = {qs, (size_t)H * (dk / 32)};
    pl.in[4] = {ks, (size_t)H * (dk / 32)};
    pl.in[5] = {vs, (size_t)H * (dv / 32)};
    pl.in[6] = {alpha, alpha_row(gate, H, dk)};
    pl.in[7] = {beta, (size_t)H * 4};
    pl.orow = (size_t)H * dv * 2;  // o is bf16
    pl.state_bytes = (size_t)B * H * dk * dv * sizeof(float);
    return pl;
}
const char *const kFp8Names[] = {"q", "k", "v", "q_scale", "k_scale", "v_scale", "alpha", "beta"};

struct Fp8Launcher : Launcher {
    kda_gate_t gate;
    int B, H, dk, dv;
    kda_status_t operator()(char *const in[], void *o, int len, const float *s0, float *state,
                            kda_stream_t s) const override {
        auto u8 = [&](int i) { return reinterpret_cast<const uint8_t *>(in[i]); };
        return kda_prefill_fp8(u8(0), u8(1), u8(2), u8(3), u8(4), u8(5), reinterpret_cast<const float *>(in[6]),
                               gate, reinterpret_cast<const float *>(in[7]), s0, o, state, B, len, H, dk, dv, s);
    }
};

bool valid_fp8(kda_gate_t gate, int B, int T, int H, int dk, int dv, int piece_tokens) {
    return valid_gate(gate) && B >= 0 && T >= 0 && H > 0 && dk == 128 && dv == 128 && piece_tokens >= 0 &&
           piece_tokens % 64 == 0 && (int64_t)B * T <= INT32_MAX;
}

kda_status_t check_common(kda_gate_t gate, int B, int T, int H, int d_k, int d_v, int piece_tokens) {
    if (!valid_gate(gate)) return fail(KDA_ERR_INVALID_ARG, "unknown gate kind %d", (int)gate);
    if (H <= 0 || d_k <= 0 || d_v <= 0) return fail(KDA_ERR_INVALID_ARG, "H, d_k, d_v must be positive");
    if ((d_k != 64 && d_k != 128) || (d_v != 64 && d_v != 128))
        return fail(KDA_ERR_UNSUPPORTED, "d_k, d_v must be 64 or 128 (got %d, %d)", d_k, d_v);
    if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B and T must be >= 0 (got %d, %d)", B, T);
    if ((int64_t)B * T > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "B * T must fit in int32");
    if (piece_tokens < 0 || piece_tokens % 64 != 0)
        return fail(KDA_ERR_INVALID_ARG, "piece_tokens must be 0 or a positive multiple of 64 (got %d)",
                    piece_tokens);
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_prefill_host_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_dtype_t qkv_dtype,
                                        kda_gate_t gate, int piece_tokens) {
    if (!valid_plain(qkv_dtype, gate, B, T, H, d_k, d_v, piece_tokens)) return 0;
    const Plan pl = plan_plain(nullptr, nullptr, nullptr, qkv_dtype, nullptr, gate, nullptr, B, H, d_k, d_v);
    return layout(pl, B, piece_tokens_for(pl, B, T, piece_tokens)).total;
}

kda_status_t kda_prefill_host(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                              const float *alpha, kda_gate_t gate, const float *beta,
                              const float *initial_state, void *o, float *final_state, int B, int T,
                              int H, int d_k, int d_v, kda_algo_t algo, int piece_tokens, void *workspace,
                              size_t workspace_bytes, kda_stream_t stream) {
    // ---- argument checks, before any CUDA call
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16)
        return fail(KDA_ERR_INVALID_ARG, "unknown qkv dtype %d", (int)qkv_dtype);
    if (algo != KDA_ALGO_AUTO && algo != KDA_ALGO_SIMT && algo != KDA_ALGO_TC)
        return fail(KDA_ERR_INVALID_ARG, "unknown algo %d", (int)algo);
    kda_status_t st;
    if ((st = check_common(gate, B, T, H, d_k, d_v, piece_tokens)) != KDA_OK) return st;
    if ((int64_t)B * T > 0) {
        if (!q || !k || !v || !beta || !o) return fail(KDA_ERR_INVALID_ARG, "q, k, v, beta and o must not be NULL");
        if (gate != KDA_GATE_NONE && !alpha) return fail(KDA_ERR_INVALID_ARG, "alpha must not be NULL");
    }
    if (B == 0 || (T == 0 && !final_state)) return KDA_OK;
    const Plan pl = plan_plain(q, k, v, qkv_dtype, gate == KDA_GATE_NONE ? nullptr : alpha, gate, beta, B, H, d_k,
                               d_v);
    PlainLauncher launch;
    launch.dt = qkv_dtype; launch.gate = gate; launch.algo = algo;
    launch.B = B; launch.H = H; launch.dk = d_k; launch.dv = d_v;
    return run_host(pl, kPlainNames, initial_state, o, final_state, B, T, piece_tokens, workspace, workspace_bytes,
                    stream, launch);
}

size_t kda_prefill_fp8_host_workspace_bytes(int B, int T, int H, int d_k, int d_v, kda_gate_t gate,
                                            int piece_tokens) {
    if (!valid_fp8(gate, B, T, H, d_k, d_v, piece_tokens)) return 0;
    const Plan pl = plan_fp8(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, gate, nullptr, B, H,
                             d_k, d_v);
    return layout(pl, B, piece_tokens_for(pl, B, T, piece_tokens)).total;
}

kda_status_t kda_prefill_fp8_host(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *q_scale,
                                  const uint8_t *k_scale, const uint8_t *v_scale, const float *alpha,
                                  kda_gate_t gate, const float *beta, const float *initial_state, void *o,
                                  float *final_state, int B, int T, int H, int d_k, int d_v, int piece_tokens,
                                  void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    kda_status_t st;
    if ((st = check_common(gate, B, T, H, d_k, d_v, piece_tokens)) != KDA_OK) return st;
    if (d_k != 128 || d_v != 128)
        return fail(KDA_ERR_UNSUPPORTED, "FP8 inputs need d_k = d_v = 128 (the tensor-core kernel)");
    if ((int64_t)B * T > 0) {
        if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !beta || !o)
            return fail(KDA_ERR_INVALID_ARG, "q, k, v, their scales, beta and o must not be NULL");
        if (gate != KDA_GATE_NONE && !alpha) return fail(KDA_ERR_INVALID_ARG, "alpha must not be NULL");
    }
    if (B == 0 || (T == 0 && !final_state)) return KDA_OK;
    const Plan pl = plan_fp8(q, k, v, q_scale, k_scale, v_scale, gate == KDA_GATE_NONE ? nullptr : alpha, gate, beta,
                             B, H, d_k, d_v);
    Fp8Launcher launch;
    launch.gate = gate;
    launch.B = B; launch.H = H; launch.dk = d_k; launch.dv = d_v;
    return run_host(pl, kFp8Names, initial_state, o, final_state, B, T, piece_tokens, workspace, workspace_bytes,
                    stream, launch);
}

}  // extern "C"
