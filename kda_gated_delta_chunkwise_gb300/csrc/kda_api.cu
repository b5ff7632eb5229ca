// Host side of the C ABI declared in include/kda.h: argument checks, kernel
// choice and launches. Nothing here allocates, synchronises or reads device
// memory; every check happens before the first launch of a call.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "kda_internal.cuh"

namespace {

thread_local std::string g_last_error;

kda_status_t fail(kda_status_t st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kda_status_t ok() {
    g_last_error.clear();
    return KDA_OK;
}

kda_status_t cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return ok();
    return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status_t check_dims(int H, int dk, int dv) {
    if (H <= 0) return fail(KDA_ERR_INVALID_ARG, "H must be positive (got %d)", H);
    if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARG, "d_k, d_v must be positive");
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128))
        return fail(KDA_ERR_UNSUPPORTED, "d_k, d_v must be 64 or 128 (got %d, %d)", dk, dv);
    return KDA_OK;
}

kda_status_t check_dtype(kda_dtype_t dt) {
    if (dt != KDA_F32 && dt != KDA_BF16) return fail(KDA_ERR_INVALID_ARG, "unknown qkv dtype %d", (int)dt);
    return KDA_OK;
}

#define KDA_REQUIRE_PTR(p)                                                                  \
    do {                                                                                    \
        if (!(p)) return fail(KDA_ERR_INVALID_ARG, "%s must not be NULL", #p);              \
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned", #p); \
    } while (0)
#define KDA_OPTIONAL_PTR(p)                                                                 \
    do {                                                                                    \
        if ((p) && !aligned16(p))                                                           \
            return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned", #p);             \
    } while (0)

// Every prefill kernel launches one CTA per (sequence, head, value slice),
// at most two slices of 64 columns for d_v = 128: the grid must stay within
// the 2^31 - 1 blocks of one launch.
kda_status_t check_grid(int64_t n_seqs, int H) {
    if (n_seqs * H * 2 > INT32_MAX)
        return fail(KDA_ERR_UNSUPPORTED, "N * H * 2 must fit in int32 (got N = %lld, H = %d)", (long long)n_seqs, H);
    return KDA_OK;
}

kda_status_t check_gate(int gate) {
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_SCALAR && gate != KDA_GATE_NONE)
        return fail(KDA_ERR_INVALID_ARG, "unknown gate kind %d", gate);
    return KDA_OK;
}

kda_status_t check_tensors(const void *q, const void *k, const void *v, const float *alpha,
                           const float *beta, const void *o, const float *s0, const float *sT,
                           bool any_tokens, int gate = KDA_GATE_CHANNEL) {
    if (any_tokens) {
        KDA_REQUIRE_PTR(q);
        KDA_REQUIRE_PTR(k);
        KDA_REQUIRE_PTR(v);
        if (gate == KDA_GATE_CHANNEL) KDA_REQUIRE_PTR(alpha);
        if (gate == KDA_GATE_SCALAR) {
            if (!alpha) return fail(KDA_ERR_INVALID_ARG, "alpha must not be NULL");
            if (reinterpret_cast<uintptr_t>(alpha) & 3u)
                return fail(KDA_ERR_INVALID_ARG, "alpha must be 4-byte aligned");
        }
        if (!beta) return fail(KDA_ERR_INVALID_ARG, "beta must not be NULL");
        if (reinterpret_cast<uintptr_t>(beta) & 3u) return fail(KDA_ERR_INVALID_ARG, "beta must be 4-byte aligned");
        KDA_REQUIRE_PTR(o);
    }
    KDA_OPTIONAL_PTR(s0);
    KDA_OPTIONAL_PTR(sT);
    return KDA_OK;
}

kda_status_t run_prefill(const kda::PrefillArgs &a, kda_algo_t algo, cudaStream_t s) {
    bool use_tc;
    switch (algo) {
        case KDA_ALGO_AUTO: use_tc = kda::prefill_tc_supported(a); break;
        case KDA_ALGO_SIMT: use_tc = false; break;
        case KDA_ALGO_TC:
            if (!kda::prefill_tc_supported(a))
                return fail(KDA_ERR_UNSUPPORTED,
                            "the tensor-core prefill needs bf16 q/k/v and d_k = d_v = 128");
            use_tc = true;
            break;
        default: return fail(KDA_ERR_INVALID_ARG, "unknown algo %d", (int)algo);
    }
    return cuda_status(use_tc ? kda::launch_prefill_tc(a, s) : kda::launch_prefill_simt(a, s),
                       use_tc ? "tensor-core prefill launch" : "prefill launch");
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

kda_status_t kda::set_error(kda_status_t st, const char *msg) { return fail(st, "%s", msg); }

extern "C" {

const char *kda_last_error(void) { return g_last_error.c_str(); }

int kda_abi_version(void) { return KDA_ABI_VERSION; }

kda_status_t kda_device_errors(int *errors, int reset) {
    if (!errors) return fail(KDA_ERR_INVALID_ARG, "errors must not be NULL");
    return cuda_status(kda::read_device_error(errors, reset != 0), "reading the device error word");
}

kda_status_t kda_prefill_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                              const float *alpha, kda_gate_t gate, const float *beta,
                              const float *initial_state, void *o, float *final_state, int B, int T,
                              int H, int d_k, int d_v, kda_algo_t algo, kda_stream_t stream) {
    kda_status_t st;
    if ((st = check_dtype(qkv_dtype)) != KDA_OK) return st;
    if ((st = check_gate(gate)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B and T must be >= 0 (got %d, %d)", B, T);
    if ((int64_t)B * T > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "B * T must fit in int32");
    if ((st = check_grid(B, H)) != KDA_OK) return st;
    if ((st = check_tensors(q, k, v, alpha, beta, o, initial_state, final_state,
                            (int64_t)B * T > 0, gate)) != KDA_OK)
        return st;
    kda::PrefillArgs a{};
    a.dt = qkv_dtype; a.dk = d_k; a.dv = d_v;
    if (algo == KDA_ALGO_TC && !kda::prefill_tc_supported(a))
        return fail(KDA_ERR_UNSUPPORTED, "the tensor-core prefill needs bf16 q/k/v and d_k = d_v = 128");
    if (B == 0) return ok();
    if (T == 0 && !final_state) return ok();
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.s0 = initial_state;
    a.o = o; a.sT = final_state; a.cu_seqlens = nullptr;
    a.gate = gate; a.slots = nullptr;
    a.N = B; a.T = T; a.H = H; a.dk = d_k; a.dv = d_v; a.dt = qkv_dtype;
    a.order = nullptr; a.counter = nullptr; a.dev_status = nullptr;
    return run_prefill(a, algo, reinterpret_cast<cudaStream_t>(stream));
}

kda_status_t kda_prefill_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *q_scale,
                             const uint8_t *k_scale, const uint8_t *v_scale, const float *alpha,
                             kda_gate_t gate, const float *beta, const float *initial_state, void *o,
                             float *final_state, int B, int T, int H, int d_k, int d_v, kda_stream_t stream) {
    kda_status_t st;
    if ((st = check_gate(gate)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (d_k != 128 || d_v != 128)
        return fail(KDA_ERR_UNSUPPORTED, "FP8 inputs need d_k = d_v = 128 (the tensor-core kernel)");
    if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B and T must be >= 0 (got %d, %d)", B, T);
    if ((int64_t)B * T > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "B * T must fit in int32");
    if ((st = check_grid(B, H)) != KDA_OK) return st;
    if ((st = check_tensors(q, k, v, alpha, beta, o, initial_state, final_state, (int64_t)B * T > 0, gate)) !=
        KDA_OK)
        return st;
    if ((int64_t)B * T > 0) {
        if (!q_scale || !k_scale || !v_scale) return fail(KDA_ERR_INVALID_ARG, "q_scale, k_scale, v_scale must not be NULL");
        if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
             reinterpret_cast<uintptr_t>(v_scale)) & 3u)
            return fail(KDA_ERR_INVALID_ARG, "the scale arrays must be 4-byte aligned");
    }
    if (B == 0) return ok();
    if (T == 0 && !final_state) return ok();
    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.s0 = initial_state;
    a.o = o; a.sT = final_state; a.cu_seqlens = nullptr;
    a.gate = gate; a.slots = nullptr;
    a.fp8 = true; a.qs = q_scale; a.ks = k_scale; a.vs = v_scale;
    a.N = B; a.T = T; a.H = H; a.dk = d_k; a.dv = d_v; a.dt = KDA_BF16;
    a.order = nullptr; a.counter = nullptr; a.dev_status = nullptr;
    return cuda_status(kda::launch_prefill_tc(a, reinterpret_cast<cudaStream_t>(stream)), "FP8 prefill launch");
}

kda_status_t kda_prefill_ex(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                            const float *alpha, const float *beta, const float *initial_state,
                            void *o, float *final_state, int B, int T, int H, int d_k, int d_v,
                            kda_algo_t algo, kda_stream_t stream) {
    return kda_prefill_gate(q, k, v, qkv_dtype, alpha, KDA_GATE_CHANNEL, beta, initial_state, o, final_state, B,
                            T, H, d_k, d_v, algo, stream);
}

kda_status_t kda_prefill(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                         const float *alpha, const float *beta, const float *initial_state,
                         void *o, float *final_state, int B, int T, int H, int d_k, int d_v,
                         kda_stream_t stream) {
    return kda_prefill_ex(q, k, v, qkv_dtype, alpha, beta, initial_state, o, final_state, B, T, H,
                          d_k, d_v, KDA_ALGO_AUTO, stream);
}

size_t kda_prefill_workspace_bytes(int B, int T, int H, int d_k, int d_v) {
    (void)B; (void)T; (void)H; (void)d_k; (void)d_v;
    return 0;  // the equal-length prefill keeps everything on chip
}

size_t kda_varlen_workspace_bytes(int N, int H, int d_k, int d_v) {
    (void)H; (void)d_k; (void)d_v;
    const size_t n = N > 0 ? (size_t)N : 0;
    return align_up(n * sizeof(int32_t)) + kAlign;  // order[N] | counter, status
}

}  // extern "C"

namespace {

kda_status_t varlen_prefill(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                            const float *alpha, int gate, const float *beta, const float *initial_state,
                            void *o, float *final_state, const int32_t *slots, int pool_size,
                            const int32_t *cu_seqlens, int N, int T_total, int H, int d_k, int d_v,
                            void *workspace, size_t workspace_bytes, int32_t *device_status,
                            cudaStream_t s) {
    kda_status_t st;
    if ((st = check_dtype(qkv_dtype)) != KDA_OK) return st;
    if ((st = check_gate(gate)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (N < 0 || T_total < 0) return fail(KDA_ERR_INVALID_ARG, "N and T_total must be >= 0");
    if (N == 0) return ok();
    if ((st = check_grid(N, H)) != KDA_OK) return st;
    if (!cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
    if ((st = check_tensors(q, k, v, alpha, beta, o, initial_state, final_state, T_total > 0, gate)) != KDA_OK)
        return st;
    const size_t need = kda_varlen_workspace_bytes(N, H, d_k, d_v);
    if (!workspace || workspace_bytes < need)
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return fail(KDA_ERR_WORKSPACE, "workspace must be 256-byte aligned");

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *order = reinterpret_cast<int32_t *>(ws);
    int32_t *tail = reinterpret_cast<int32_t *>(ws + align_up((size_t)N * sizeof(int32_t)));
    int32_t *counter = tail;
    int32_t *status = device_status ? device_status : tail + 1;

    cudaError_t e = kda::launch_varlen_prep(cu_seqlens, N, T_total, order, counter, status, slots, pool_size, s);
    if (e != cudaSuccess) return cuda_status(e, "varlen prep launch");

    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.s0 = initial_state;
    a.o = o; a.sT = final_state; a.cu_seqlens = cu_seqlens;
    a.gate = gate; a.slots = slots;
    a.N = N; a.T = T_total; a.H = H; a.dk = d_k; a.dv = d_v; a.dt = qkv_dtype;
    a.order = order; a.counter = counter; a.dev_status = status;
    return run_prefill(a, KDA_ALGO_AUTO, s);
}

}  // namespace

kda_status_t kda::varlen_prefill_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                      const float *alpha, int gate, const float *beta, const float *initial_state,
                                      void *o, float *final_state, const int32_t *cu_seqlens, int N, int T_total,
                                      int H, int d_k, int d_v, void *workspace, size_t workspace_bytes,
                                      int32_t *device_status, cudaStream_t s) {
    return varlen_prefill(q, k, v, qkv_dtype, alpha, gate, beta, initial_state, o, final_state, nullptr, 0,
                          cu_seqlens, N, T_total, H, d_k, d_v, workspace, workspace_bytes, device_status, s);
}

extern "C" {

kda_status_t kda_varlen_prefill(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                const float *alpha, const float *beta,
                                const float *initial_state, void *o, float *final_state,
                                const int32_t *cu_seqlens, int N, int T_total, int H, int d_k,
                                int d_v, void *workspace, size_t workspace_bytes,
                                int32_t *device_status, kda_stream_t stream) {
    return varlen_prefill(q, k, v, qkv_dtype, alpha, KDA_GATE_CHANNEL, beta, initial_state, o, final_state,
                          nullptr, 0, cu_seqlens, N, T_total, H, d_k, d_v, workspace, workspace_bytes,
                          device_status, reinterpret_cast<cudaStream_t>(stream));
}

kda_status_t kda_varlen_prefill_slots(const void *q, const void *k, const void *v,
                                      kda_dtype_t qkv_dtype, const float *alpha, kda_gate_t gate,
                                      const float *beta, float *state_pool, const int32_t *slots,
                                      int pool_size, void *o, const int32_t *cu_seqlens, int N,
                                      int T_total, int H, int d_k, int d_v, void *workspace,
                                      size_t workspace_bytes, int32_t *device_status,
                                      kda_stream_t stream) {
    if (N > 0) {
        KDA_REQUIRE_PTR(state_pool);
        if (!slots) return fail(KDA_ERR_INVALID_ARG, "slots must not be NULL");
        if (reinterpret_cast<uintptr_t>(slots) & 3u) return fail(KDA_ERR_INVALID_ARG, "slots must be 4-byte aligned");
        if (pool_size <= 0) return fail(KDA_ERR_INVALID_ARG, "pool_size must be positive");
    }
    return varlen_prefill(q, k, v, qkv_dtype, alpha, gate, beta, state_pool, o, state_pool, slots, pool_size,
                          cu_seqlens, N, T_total, H, d_k, d_v, workspace, workspace_bytes, device_status,
                          reinterpret_cast<cudaStream_t>(stream));
}

size_t kda_prefill_backward_workspace_bytes(int B, int T, int H, int d_k, int d_v) {
    if (B < 0 || T < 0 || H <= 0 || d_k <= 0 || d_v <= 0) return 0;
    return kda::backward_workspace_bytes(B, T, H, d_k, d_v, false);
}

size_t kda_varlen_prefill_backward_workspace_bytes(int N, int T_total, int H, int d_k, int d_v) {
    if (N < 0 || T_total < 0 || H <= 0 || d_k <= 0 || d_v <= 0) return 0;
    return kda::backward_workspace_bytes(N, T_total, H, d_k, d_v, true);
}

}  // extern "C"

namespace {

// The checks and the launch shared by the equal-length and the packed backward
// (cu_seqlens == NULL: B sequences of T tokens; else N = B packed sequences of
// T = T_total tokens in all).
kda_status_t backward(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype, const float *alpha,
                      kda_gate_t gate, const float *beta, const float *initial_state, const void *d_o,
                      const float *d_final_state, float *dq, float *dk, float *dv, float *dalpha, float *dbeta,
                      float *d_initial_state, const int32_t *cu_seqlens, int B, int T, int H, int d_k, int d_v,
                      void *workspace, size_t workspace_bytes, int32_t *device_status, kda_stream_t stream) {
    kda_status_t st;
    const bool packed = cu_seqlens != nullptr;
    if ((st = check_dtype(qkv_dtype)) != KDA_OK) return st;
    if ((st = check_gate(gate)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B (N) and T (T_total) must be >= 0 (got %d, %d)", B, T);
    const int64_t tokens = packed ? (int64_t)T : (int64_t)B * T;
    if (tokens > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "the token count must fit in int32");
    const int64_t chunks = packed ? ((int64_t)T + 63) / 64 + B : (int64_t)B * (((int64_t)T + 63) / 64);
    if ((chunks > 0 ? chunks : 1) * H * 2 > INT32_MAX)
        return fail(KDA_ERR_UNSUPPORTED, "the chunks of all sequences times H times 2 must fit in int32");
    const bool any = tokens > 0;
    if ((st = check_tensors(q, k, v, alpha, beta, d_o, initial_state, d_final_state, any, gate)) != KDA_OK) return st;
    if (any) {
        KDA_REQUIRE_PTR(dq);
        KDA_REQUIRE_PTR(dk);
        KDA_REQUIRE_PTR(dv);
        if (gate == KDA_GATE_CHANNEL) KDA_REQUIRE_PTR(dalpha);
        if (gate == KDA_GATE_SCALAR) {
            if (!dalpha) return fail(KDA_ERR_INVALID_ARG, "dalpha must not be NULL");
            if (reinterpret_cast<uintptr_t>(dalpha) & 3u)
                return fail(KDA_ERR_INVALID_ARG, "dalpha must be 4-byte aligned");
        }
        if (!dbeta) return fail(KDA_ERR_INVALID_ARG, "dbeta must not be NULL");
        if (reinterpret_cast<uintptr_t>(dbeta) & 3u) return fail(KDA_ERR_INVALID_ARG, "dbeta must be 4-byte aligned");
    }
    KDA_OPTIONAL_PTR(d_initial_state);
    if (packed) {
        if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
        if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
            return fail(KDA_ERR_INVALID_ARG, "device_status must be 4-byte aligned");
    }
    if (B == 0) return ok();
    const size_t need = kda::backward_workspace_bytes(B, T, H, d_k, d_v, packed);
    if (need && (!workspace || workspace_bytes < need))
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, workspace_bytes);
    if (need && !aligned16(workspace)) return fail(KDA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    kda::BackwardArgs b{};
    b.q = q; b.k = k; b.v = v; b.d_o = d_o; b.dt = qkv_dtype;
    b.alpha = alpha; b.beta = beta; b.s0 = initial_state; b.dsT = d_final_state;
    b.dq = dq; b.dk = dk; b.dvv = dv; b.dalpha = dalpha; b.dbeta = dbeta; b.ds0 = d_initial_state;
    b.workspace = workspace;
    b.gate = gate;
    b.N = B; b.T = T; b.H = H; b.d_k = d_k; b.d_v = d_v;
    b.cu_seqlens = cu_seqlens;
    b.dev_status = device_status;
    return cuda_status(kda::launch_backward(b, reinterpret_cast<cudaStream_t>(stream)), "backward launch");
}

}  // namespace

extern "C" {

kda_status_t kda_prefill_backward_gate(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                       const float *alpha, kda_gate_t gate, const float *beta,
                                       const float *initial_state, const void *d_o, const float *d_final_state,
                                       float *dq, float *dk, float *dv, float *dalpha, float *dbeta,
                                       float *d_initial_state, int B, int T, int H, int d_k, int d_v,
                                       void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    return backward(q, k, v, qkv_dtype, alpha, gate, beta, initial_state, d_o, d_final_state, dq, dk, dv, dalpha,
                    dbeta, d_initial_state, nullptr, B, T, H, d_k, d_v, workspace, workspace_bytes, nullptr, stream);
}

kda_status_t kda_prefill_backward(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                  const float *alpha, const float *beta, const float *initial_state,
                                  const void *d_o, const float *d_final_state, float *dq, float *dk, float *dv,
                                  float *dalpha, float *dbeta, float *d_initial_state, int B, int T, int H,
                                  int d_k, int d_v, void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    return kda_prefill_backward_gate(q, k, v, qkv_dtype, alpha, KDA_GATE_CHANNEL, beta, initial_state, d_o,
                                     d_final_state, dq, dk, dv, dalpha, dbeta, d_initial_state, B, T, H, d_k, d_v,
                                     workspace, workspace_bytes, stream);
}

kda_status_t kda_varlen_prefill_backward(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                         const float *alpha, kda_gate_t gate, const float *beta,
                                         const float *initial_state, const void *d_o, const float *d_final_state,
                                         float *dq, float *dk, float *dv, float *dalpha, float *dbeta,
                                         float *d_initial_state, const int32_t *cu_seqlens, int N, int T_total,
                                         int H, int d_k, int d_v, void *workspace, size_t workspace_bytes,
                                         int32_t *device_status, kda_stream_t stream) {
    if (N > 0 && !cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    if (N == 0) return ok();
    return backward(q, k, v, qkv_dtype, alpha, gate, beta, initial_state, d_o, d_final_state, dq, dk, dv, dalpha,
                    dbeta, d_initial_state, cu_seqlens, N, T_total, H, d_k, d_v, workspace, workspace_bytes,
                    device_status, stream);
}

kda_status_t kda_selftest_bounded_wait(const void *q, const void *k, const void *v, const float *alpha,
                                       const float *beta, void *o, float *final_state, int T, int stall_chunk,
                                       kda_stream_t stream) {
    kda_status_t st;
    if (T <= 0) return fail(KDA_ERR_INVALID_ARG, "T must be positive (got %d)", T);
    if (stall_chunk < 0 || (int64_t)stall_chunk * 64 >= T)
        return fail(KDA_ERR_INVALID_ARG, "stall_chunk must name one of the %d chunks", (T + 63) / 64);
    if ((st = check_tensors(q, k, v, alpha, beta, o, nullptr, final_state, true)) != KDA_OK) return st;
    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.s0 = nullptr;
    a.o = o; a.sT = final_state; a.cu_seqlens = nullptr;
    a.gate = KDA_GATE_CHANNEL; a.slots = nullptr;
    a.N = 1; a.T = T; a.H = 1; a.dk = 128; a.dv = 128; a.dt = KDA_BF16;
    a.order = nullptr; a.counter = nullptr; a.dev_status = nullptr;
    a.stall1 = stall_chunk + 1;
    return cuda_status(kda::launch_prefill_tc(a, reinterpret_cast<cudaStream_t>(stream)), "self-test launch");
}

kda_status_t kda_decode_step(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                             const float *alpha, const float *beta, float *state, void *o,
                             int N, int H, int d_k, int d_v, kda_stream_t stream) {
    kda_status_t st;
    if ((st = check_dtype(qkv_dtype)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (N < 0) return fail(KDA_ERR_INVALID_ARG, "N must be >= 0");
    if (N == 0) return ok();
    if ((int64_t)N * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "N * H must fit in int32");
    if ((st = check_tensors(q, k, v, alpha, beta, o, nullptr, nullptr, true)) != KDA_OK) return st;
    KDA_REQUIRE_PTR(state);
    return cuda_status(kda::launch_decode(q, k, v, qkv_dtype, alpha, KDA_GATE_CHANNEL, beta, state, nullptr, 0,
                                          nullptr, o, N, H, d_k, d_v, reinterpret_cast<cudaStream_t>(stream)),
                       "decode launch");
}

kda_status_t kda_decode_step_slots(const void *q, const void *k, const void *v, kda_dtype_t qkv_dtype,
                                   const float *alpha, kda_gate_t gate, const float *beta,
                                   float *state_pool, const int32_t *slots, int pool_size, void *o,
                                   int N, int H, int d_k, int d_v, int32_t *device_status,
                                   kda_stream_t stream) {
    kda_status_t st;
    if ((st = check_dtype(qkv_dtype)) != KDA_OK) return st;
    if ((st = check_gate(gate)) != KDA_OK) return st;
    if ((st = check_dims(H, d_k, d_v)) != KDA_OK) return st;
    if (N < 0) return fail(KDA_ERR_INVALID_ARG, "N must be >= 0");
    if (N == 0) return ok();
    if ((int64_t)N * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "N * H must fit in int32");
    if ((st = check_tensors(q, k, v, alpha, beta, o, nullptr, nullptr, true, gate)) != KDA_OK) return st;
    KDA_REQUIRE_PTR(state_pool);
    if (!slots) return fail(KDA_ERR_INVALID_ARG, "slots must not be NULL");
    if (reinterpret_cast<uintptr_t>(slots) & 3u) return fail(KDA_ERR_INVALID_ARG, "slots must be 4-byte aligned");
    if (pool_size <= 0) return fail(KDA_ERR_INVALID_ARG, "pool_size must be positive");
    if ((int64_t)pool_size * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "pool_size * H must fit in int32");
    if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
        return fail(KDA_ERR_INVALID_ARG, "device_status must be 4-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (device_status) {  // KDA_DEV_OK unless a head finds a bad slot
        const cudaError_t e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_status(e, "status reset");
    }
    return cuda_status(kda::launch_decode(q, k, v, qkv_dtype, alpha, gate, beta, state_pool, slots, pool_size,
                                          device_status, o, N, H, d_k, d_v, s),
                       "decode launch");
}

}  // extern "C"
