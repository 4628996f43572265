// C ABI of liblinattn.so: argument validation, kernel selection and launch.
// The declarations and their contracts are in include/linattn.h.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "la_internal.h"
#include "la_tc.h"
#include "la_tc_host.h"

namespace la {

// Per-device status words.  A kernel that gives up on a bounded wait stores a
// non-zero la_status in word 0 and where it gave up in word 1 (block index in
// the high 12 bits, the wait's identifier in the low 20 bits: a barrier's
// shared-memory address, or 0x80000 | a flag's word address);
// la_check_device_status reads and clears both.
__device__ int g_status_word[2];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices] = {};
thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_launches{0};

la_status fail(la_status s, const char *msg) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
    return s;
}

la_status cuda_fail(cudaError_t e, const char *where) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where,
                  cudaGetErrorString(e));
    return LA_ERR_CUDA;
}

bool valid_dtype(la_dtype t) { return t == LA_F32 || t == LA_BF16; }
}  // namespace

int *device_status_word(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_status_word);
        if (*err != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

void note_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

void set_last_error(const char *msg) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

}  // namespace la

using namespace la;

namespace {

la_status validate_forward(const void *q, const void *k, const void *v,
                           const void *out, int B, int H, int N, int d,
                           int causal, const float *decay, la_dtype dtype,
                           DecayArgs *dk) {
    if (B < 0 || H < 0 || N < 0)
        return fail(LA_ERR_INVALID_ARG, "la_forward: negative B, H or N");
    // an empty problem reads and writes no tensor element, so its pointers
    // may be NULL (zero-size framework tensors have no storage)
    const bool empty = (long long)B * H * N == 0;
    if (!empty && (!q || !k || !v || !out))
        return fail(LA_ERR_INVALID_ARG, "la_forward: null tensor pointer");
    if (d < 1 || d > LA_MAX_D)
        return fail(LA_ERR_INVALID_ARG, "la_forward: d must be in 1..256");
    if (causal != 0 && causal != 1)
        return fail(LA_ERR_INVALID_ARG, "la_forward: causal must be 0 or 1");
    if (!valid_dtype(dtype))
        return fail(LA_ERR_INVALID_ARG, "la_forward: unknown dtype");
    if (!empty && (out == q || out == k || out == v))
        return fail(LA_ERR_INVALID_ARG, "la_forward: out aliases an input");
    dk->has = 0;
    dk->H = H > 0 ? H : 1;
    if (decay) {
        if (!causal)
            return fail(LA_ERR_INVALID_ARG,
                        "la_forward: decay is defined for the causal form only");
        if (H > LA_MAX_DECAY_HEADS)
            return fail(LA_ERR_UNSUPPORTED,
                        "la_forward: decay given for more than 1024 heads");
        for (int h = 0; h < H; ++h) {
            float g = decay[h];
            if (!(g >= 0.f && g <= 1.f))  // also rejects NaN
                return fail(LA_ERR_INVALID_ARG,
                            "la_forward: decay values must lie in [0, 1]");
            dk->g[h] = g;
        }
        dk->has = 1;
    }
    return LA_OK;
}

}  // namespace

extern "C" {

__attribute__((visibility("default")))
la_status la_forward_ex(const void *q, const void *k, const void *v,
                        void *out, int B, int H, int N, int d, int causal,
                        const float *decay, la_dtype dtype, int path,
                        int segment_chunks, la_stream_t stream) {
    return la::forward_with_workspace(q, k, v, out, B, H, N, d, causal, decay,
                                      dtype, path, segment_chunks, nullptr, 0,
                                      nullptr, nullptr, nullptr, nullptr, stream);
}

__attribute__((visibility("default")))
la_status la_forward_variant(const void *q, const void *k, const void *v,
                             void *out, int B, int H, int N, int d, int causal,
                             const float *decay, la_dtype dtype,
                             const la_variant *variant, la_stream_t stream) {
    return la::forward_with_workspace(q, k, v, out, B, H, N, d, causal, decay,
                                      dtype, 0, 0, nullptr, 0, nullptr, nullptr,
                                      variant, nullptr, stream);
}

__attribute__((visibility("default")))
la_status la_forward_causal_state(const void *q, const void *k, const void *v,
                                  void *out, float *S, float *z, int B, int H,
                                  int N, int d, const float *decay,
                                  la_dtype dtype, la_stream_t stream) {
    if (!S || !z)
        return fail(LA_ERR_INVALID_ARG, "la_forward_causal_state: null state pointer");
    if ((reinterpret_cast<uintptr_t>(S) & 15u) != 0)
        return fail(LA_ERR_INVALID_ARG, "la_forward_causal_state: S must be 16-byte aligned");
    return la::forward_with_workspace(q, k, v, out, B, H, N, d, 1, decay, dtype,
                                      0, 0, nullptr, 0, S, z, nullptr, nullptr, stream);
}

__attribute__((visibility("default")))
la_status la_forward(const void *q, const void *k, const void *v, void *out,
                     int B, int H, int N, int d, int causal,
                     const float *decay, la_dtype dtype, la_stream_t stream) {
    return la_forward_ex(q, k, v, out, B, H, N, d, causal, decay, dtype, 0, 0,
                         stream);
}

}  // extern "C"

la_status la::forward_with_workspace(const void *q, const void *k, const void *v,
                                     void *out, int B, int H, int N, int d,
                                     int causal, const float *decay,
                                     la_dtype dtype, int path, int segment_chunks,
                                     void *ws, size_t ws_bytes, float *S_out,
                                     float *z_out, const la_variant *variant,
                                     const float *gates, la_stream_t stream) {
    if (variant && ((variant->feature_map != LA_PHI_ELU1 &&
                     variant->feature_map != LA_PHI_IDENTITY) ||
                    (variant->normalise != 0 && variant->normalise != 1)))
        return fail(LA_ERR_INVALID_ARG, "la_forward_variant: unknown variant");
    DecayArgs dk;
    la_status st = validate_forward(q, k, v, out, B, H, N, d, causal, decay,
                                    dtype, &dk);
    if (st != LA_OK) return st;
    if (path < 0 || path > 2)
        return fail(LA_ERR_INVALID_ARG, "la_forward_ex: path must be 0, 1 or 2");
    if (segment_chunks < 0)
        return fail(LA_ERR_INVALID_ARG, "la_forward_ex: segment_chunks < 0");
    FwdShape sh{B, H, N, d};
    if (variant) {
        sh.phi = variant->feature_map == LA_PHI_ELU1 ? 1 : 0;
        sh.norm = variant->normalise;
    }
    if (sh.BH() == 0) return LA_OK;
    if (sh.BH() > 2147483647LL || (long long)N * d > (1LL << 40))
        return fail(LA_ERR_UNSUPPORTED, "la_forward: problem too large");
    if (N == 0) {
        // no tokens: the final state is the zero state
        if (!S_out) return LA_OK;
        cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t e0 = cudaMemsetAsync(S_out, 0, sizeof(float) * sh.BH() * d * d, s0);
        if (e0 == cudaSuccess)
            e0 = cudaMemsetAsync(z_out, 0, sizeof(float) * sh.BH() * d, s0);
        return e0 == cudaSuccess ? LA_OK : cuda_fail(e0, "la_forward: zero state");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (gates && !causal)
        return fail(LA_ERR_INVALID_ARG, "la_forward_gated: gates are defined for the causal form only");
    if (gates && decay)
        return fail(LA_ERR_INVALID_ARG, "la_forward_gated: give gates or a decay, not both");
    // gates run on the tensor cores as their third mode (no final state)
    const bool tc_ok = tc_supported(sh, dtype, causal, q, k, v, out) &&
                       !(gates && S_out);
    if (path == 2 && !tc_ok)
        return fail(LA_ERR_UNSUPPORTED,
                    "la_forward_ex: tensor-core path needs bf16, d in {64,128} and 16-byte aligned tensors");
    if (tc_ok && path != 1) {
        cudaError_t ce;
        int *status = device_status_word(&ce);
        if (!status) return cuda_fail(ce, "la_forward: status word");
        TcResult r = tc_forward(q, k, v, out, sh, causal, dk, segment_chunks,
                                status, ws, ws_bytes, S_out, z_out, gates, s);
        if (r.status != LA_OK) {
            if (r.status == LA_ERR_CUDA) return cuda_fail(r.cuda, r.where);
            return fail(r.status, r.where);
        }
        return LA_OK;
    }
    int launches = 0;
    TcResult r = launch_simt_forward(q, k, v, out, sh, causal, dk, dtype, S_out, z_out,
                                     gates, segment_chunks, s, &launches);
    note_launches(launches);
    if (r.status != LA_OK) {
        if (r.status == LA_ERR_CUDA) return cuda_fail(r.cuda, r.where);
        return fail(r.status, r.where);
    }
    return LA_OK;
}

size_t la::forward_workspace_bytes(int B, int H, int N, int d, int causal,
                                   bool decay, la_dtype dtype) {
    FwdShape sh{B, H, N, d};
    if (dtype != LA_BF16 || (d != 64 && d != 128)) return 0;  // CUDA-core path
    int sms = 0;
    if (tchost::sm_count(&sms) != cudaSuccess || sms <= 0) sms = 1;
    return tc_workspace_bytes(sh, causal, decay, 0, sms);
}

la_status la::decode_common(float *S, float *z, const void *q, const void *k,
                           const void *v, void *out, int B, int H, int d,
                           const float *decay, const float *gates, la_dtype dtype,
                           const la_variant *variant, la_stream_t stream) {
    if (gates && decay)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_gated: give gates or a decay, not both");
    if (variant && ((variant->feature_map != LA_PHI_ELU1 &&
                     variant->feature_map != LA_PHI_IDENTITY) ||
                    (variant->normalise != 0 && variant->normalise != 1)))
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_variant: unknown variant");
    const int phi = (!variant || variant->feature_map == LA_PHI_ELU1) ? 1 : 0;
    const int norm = variant ? variant->normalise : 1;
    if (!S || !z || !q || !k || !v || !out)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step: null pointer");
    if (B < 0 || H < 0)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step: negative B or H");
    if (d < 1 || d > LA_MAX_D)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step: d must be in 1..256");
    if (!valid_dtype(dtype))
        return fail(LA_ERR_INVALID_ARG, "la_decode_step: unknown dtype");
    DecayArgs dk;
    dk.has = 0;
    dk.H = H > 0 ? H : 1;
    if (decay) {
        if (H > LA_MAX_DECAY_HEADS)
            return fail(LA_ERR_UNSUPPORTED,
                        "la_decode_step: decay given for more than 1024 heads");
        for (int h = 0; h < H; ++h) {
            const float g = decay[h];
            if (!(g >= 0.f && g <= 1.f))  // also rejects NaN
                return fail(LA_ERR_INVALID_ARG,
                            "la_decode_step: decay values must lie in [0, 1]");
            dk.g[h] = g;
        }
        dk.has = 1;
    }
    long long BH = (long long)B * H;
    if (BH == 0) return LA_OK;
    if (BH > 2147483647LL)
        return fail(LA_ERR_UNSUPPORTED, "la_decode_step: too many heads");
    cudaError_t e = launch_decode_step(S, z, q, k, v, out, BH, d, dk, phi, norm,
                                       gates, dtype, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "la_decode_step");
    note_launches(1);
    return LA_OK;
}

extern "C" {

__attribute__((visibility("default")))
la_status la_decode_step_variant(float *S, float *z, const void *q,
                                 const void *k, const void *v, void *out, int B,
                                 int H, int d, const float *decay,
                                 la_dtype dtype, const la_variant *variant,
                                 la_stream_t stream) {
    return la::decode_common(S, z, q, k, v, out, B, H, d, decay, nullptr, dtype,
                             variant, stream);
}

__attribute__((visibility("default")))
la_status la_decode_step_gated(float *S, float *z, const void *q, const void *k,
                               const void *v, void *out, const float *gates,
                               int B, int H, int d, la_dtype dtype,
                               const la_variant *variant, la_stream_t stream) {
    if (!gates) return fail(LA_ERR_INVALID_ARG, "la_decode_step_gated: null gates");
    return la::decode_common(S, z, q, k, v, out, B, H, d, nullptr, gates, dtype,
                             variant, stream);
}

__attribute__((visibility("default")))
la_status la_forward_gated(const void *q, const void *k, const void *v,
                           void *out, const float *gates, int B, int H, int N,
                           int d, la_dtype dtype, const la_variant *variant,
                           la_stream_t stream) {
    if (!gates && (long long)B * H * N > 0)
        return fail(LA_ERR_INVALID_ARG, "la_forward_gated: null gates");
    return la::forward_with_workspace(q, k, v, out, B, H, N, d, 1, nullptr, dtype,
                                      0, 0, nullptr, 0, nullptr, nullptr, variant,
                                      gates, stream);
}

__attribute__((visibility("default")))
la_status la_decode_step_delta(float *S, const void *q, const void *k,
                               const void *v, void *out, const float *beta,
                               const float *alpha, int B, int H, int d,
                               la_dtype dtype, la_stream_t stream) {
    if (!S || !q || !k || !v || !out || !beta)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_delta: null pointer");
    if (B < 0 || H < 0)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_delta: negative B or H");
    if (d < 1 || d > LA_MAX_D)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_delta: d must be in 1..256");
    if (!valid_dtype(dtype))
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_delta: unknown dtype");
    const long long BH = (long long)B * H;
    if (BH == 0) return LA_OK;
    if (BH > 2147483647LL)
        return fail(LA_ERR_UNSUPPORTED, "la_decode_step_delta: too many heads");
    cudaError_t e = launch_delta_step(S, q, k, v, out, beta, alpha, BH, d, dtype,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "la_decode_step_delta");
    note_launches(1);
    return LA_OK;
}

__attribute__((visibility("default")))
la_status la_forward_delta(const void *q, const void *k, const void *v, void *out,
                           const float *beta, const float *alpha, float *S, int B,
                           int H, int N, int d, la_dtype dtype, la_stream_t stream) {
    if (B < 0 || H < 0 || N < 0)
        return fail(LA_ERR_INVALID_ARG, "la_forward_delta: negative B, H or N");
    if (d < 1 || d > LA_MAX_D)
        return fail(LA_ERR_INVALID_ARG, "la_forward_delta: d must be in 1..256");
    if (!valid_dtype(dtype))
        return fail(LA_ERR_INVALID_ARG, "la_forward_delta: unknown dtype");
    const long long BH = (long long)B * H;
    if (BH == 0 || N == 0) return LA_OK;
    if (!q || !k || !v || !out || !beta)
        return fail(LA_ERR_INVALID_ARG, "la_forward_delta: null pointer");
    if (BH > 2147483647LL || (long long)N * d > (1LL << 40))
        return fail(LA_ERR_UNSUPPORTED, "la_forward_delta: problem too large");
    cudaError_t e = launch_delta_forward(q, k, v, out, beta, alpha, S, BH, N, d, dtype,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_delta");
    note_launches(1);
    return LA_OK;
}

__attribute__((visibility("default")))
la_status la_decode_step_ex(float *S, float *z, const void *q, const void *k,
                            const void *v, void *out, int B, int H, int d,
                            const float *decay, la_dtype dtype,
                            la_stream_t stream) {
    return la_decode_step_variant(S, z, q, k, v, out, B, H, d, decay, dtype,
                                  nullptr, stream);
}

__attribute__((visibility("default")))
la_status la_decode_step(float *S, float *z, const void *q, const void *k,
                         const void *v, void *out, int B, int H, int d,
                         la_dtype dtype, la_stream_t stream) {
    return la_decode_step_ex(S, z, q, k, v, out, B, H, d, nullptr, dtype, stream);
}

__attribute__((visibility("default")))
la_status la_check_device_status(la_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "la_check_device_status: sync");
    int *p = device_status_word(&e);
    if (!p) return cuda_fail(e, "la_check_device_status: status word");
    int word[2] = {0, 0};
    e = cudaMemcpy(word, p, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "la_check_device_status: read");
    if (word[0] != 0) {
        int zero[2] = {0, 0};
        e = cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "la_check_device_status: clear");
        char msg[160];
        if (word[0] == (int)LA_ERR_INTERNAL)
            std::snprintf(msg, sizeof(msg),
                          "a device-side index check failed (debug build, source line %d)",
                          word[1]);
        else
            std::snprintf(msg, sizeof(msg),
                          "a kernel reported a device-side failure (block %d, wait 0x%05x)",
                          (word[1] >> 20) & 0xFFF, word[1] & 0xFFFFF);
        return fail(static_cast<la_status>(word[0]), msg);
    }
    return LA_OK;
}

__attribute__((visibility("default")))
const char *la_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
        case LA_ERR_CUDA: return "LA_ERR_CUDA";
        case LA_ERR_NO_MEMORY: return "LA_ERR_NO_MEMORY";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
        case LA_ERR_INTERNAL: return "LA_ERR_INTERNAL";
    }
    return "LA_ERR_UNKNOWN";
}

__attribute__((visibility("default")))
const char *la_last_error(void) { return g_last_error; }

__attribute__((visibility("default")))
int la_abi_version(void) { return 1; }

__attribute__((visibility("default")))
unsigned long long la_kernel_launch_count(void) { return g_launches.load(); }

__attribute__((visibility("default")))
la_status la_debug_inject_timeout(long long wait_cycles, int hold_segment) {
    if (wait_cycles < 4096)
        return fail(LA_ERR_INVALID_ARG, "la_debug_inject_timeout: wait_cycles below 4096");
    la::tc_debug_set_timeout(wait_cycles, hold_segment);
    return LA_OK;
}

__attribute__((visibility("default")))
la_status la_debug_fail_next_allocs(int n) {
    if (n < 0) return fail(LA_ERR_INVALID_ARG, "la_debug_fail_next_allocs: negative n");
    la::tc_debug_fail_allocs(n);
    return LA_OK;
}

}  // extern "C"
