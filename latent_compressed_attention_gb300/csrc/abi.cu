// C ABI of the library (declared in include/mla.h): host-side validation,
// dispatch to the kernels, and the per-device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/mla.h"
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

// Device error word: kernels record the first device-side failure here.
__device__ int g_device_error = 0;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int *err_word = nullptr;
    int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;
std::atomic<unsigned long long> g_launches{0};

cudaError_t device_info(DeviceInfo *&out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        d.err_word = static_cast<int *>(p);
        d.num_sms = sms;
        d.ready = true;
    }
    out = &d;
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool mul_fits(long long a, long long b, long long limit) { return a == 0 || b <= limit / a; }

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void *tensor_map_encode_fn() {
    static void *fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    });
    return fn;
}

// One thread waits, with the library's bounded wait, for a barrier phase that
// nothing completes: the wait gives up after `limit_ns` and records
// kDevErrTimeout in the device error word, exactly as a stalled pipeline would.
__global__ void wait_timeout_probe_kernel(int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait(b, 0, err, nullptr, limit_ns);
}

}  // namespace mla

using namespace mla;

extern "C" {

MLA_API const char *mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_NULL: return "a required pointer is NULL";
        case MLA_ERR_SHAPE: return "invalid size";
        case MLA_ERR_DTYPE: return "unknown dtype";
        case MLA_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_UNSUPPORTED: return "shape or dtype not supported by this build";
        case MLA_ERR_CUDA: return "CUDA call failed";
        case MLA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case MLA_ERR_DEVICE_BOUNDS: return "device-side bounds check failed";
        default: return "unknown status";
    }
}

MLA_API int mla_version(void) { return 100; }

MLA_API unsigned long long mla_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

MLA_API size_t mla_absorbed_attn_fwd_workspace_size(int B, int T, int H, int d_q, int d_v, int r, int dtype) {
    if ((dtype != MLA_DTYPE_F32 && dtype != MLA_DTYPE_BF16) || B < 0 || T < 0 || H <= 0) return 0;
    if (static_cast<long long>(B) * T > INT_MAX || !mul_fits(static_cast<long long>(B) * T, r, LLONG_MAX / 8)) return 0;
    return prefill_workspace_bytes(B, T, r, d_q, d_v, dtype == MLA_DTYPE_F32);
}

namespace {
int fwd_impl(const void *q, const void *c, const void *w_uk, const void *w_uv, const void *gate, float scale, void *out,
             float *lse, int B, int T, int H, int d_q, int d_v, int r, int dtype, void *workspace,
             size_t workspace_bytes, void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || d_q <= 0 || d_v <= 0 || r <= 0) return MLA_ERR_SHAPE;
    const long long rows = static_cast<long long>(B) * T;
    if (!mul_fits(rows, static_cast<long long>(H) * (d_q > d_v ? d_q : d_v), LLONG_MAX / 8) ||
        !mul_fits(rows, r, LLONG_MAX / 8) || rows > INT_MAX)
        return MLA_ERR_SHAPE;
    if (!q || !c || !w_uk || !w_uv || !out) return MLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(c) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(out) ||
        (gate && !aligned16(gate)))
        return MLA_ERR_ALIGN;
    const bool f32 = dtype == MLA_DTYPE_F32;
    const bool ok_shape = f32 ? prefill_f32_simt_supports(r, d_q, d_v)
                              : (prefill_bf16_r512_supports(r, d_q, d_v) || prefill_bf16_small_supports(r, d_q, d_v));
    if (!ok_shape || (f32 && T > kPrefillF32MaxT)) return MLA_ERR_UNSUPPORTED;
    if (lse && (f32 || !prefill_bf16_r512_supports(r, d_q, d_v))) return MLA_ERR_UNSUPPORTED;
    if (lse && !aligned16(lse)) return MLA_ERR_ALIGN;
    if (rows == 0) return MLA_OK;
    const size_t need = prefill_workspace_bytes(B, T, r, d_q, d_v, f32);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MLA_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return MLA_ERR_ALIGN;

    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    PrefillArgs a{q, c, w_uk, w_uv, gate, out, scale, B, T, H, d_q, d_v, r, dev->err_word, dev->num_sms,
                  workspace, workspace_bytes};
    a.lse = lse;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (f32)
        e = launch_prefill_f32_simt(a, s);
    else if (prefill_bf16_r512_supports(r, d_q, d_v))
        e = launch_prefill_bf16_r512(a, s);
    else
        e = launch_prefill_bf16_small(a, s);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
}  // namespace

MLA_API int mla_absorbed_attn_fwd(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                  const void *gate, float scale, void *out, int B, int T, int H, int d_q,
                                  int d_v, int r, int dtype, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    return fwd_impl(q, c, w_uk, w_uv, gate, scale, out, nullptr, B, T, H, d_q, d_v, r, dtype, workspace,
                    workspace_bytes, stream);
}

MLA_API int mla_absorbed_attn_fwd_lse(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                      const void *gate, float scale, void *out, float *lse, int B, int T, int H,
                                      int d_q, int d_v, int r, int dtype, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    if (!lse) return MLA_ERR_NULL;
    return fwd_impl(q, c, w_uk, w_uv, gate, scale, out, lse, B, T, H, d_q, d_v, r, dtype, workspace,
                    workspace_bytes, stream);
}

MLA_API size_t mla_absorbed_attn_bwd_workspace_size(int B, int T, int H, int d_q, int d_v, int r, int dtype) {
    if ((dtype != MLA_DTYPE_F32 && dtype != MLA_DTYPE_BF16) || B <= 0 || T <= 0 || H <= 0) return 0;
    if (dtype == MLA_DTYPE_BF16 && backward_bf16_r512_supports(r, d_q, d_v)) {
        if (static_cast<long long>(B) * T > INT_MAX || !mul_fits(static_cast<long long>(B) * H * T, T + 128LL, LLONG_MAX / 8))
            return 0;
        return backward_bf16_r512_workspace_bytes(B, T, H);
    }
    if (!backward_f32_supports(r, d_q, d_v)) return 0;
    if (!mul_fits(static_cast<long long>(B) * T, static_cast<long long>(H) * (2 * r + 4), LLONG_MAX / 8)) return 0;
    return backward_f32_workspace_bytes(B, T, H, r);
}

namespace {
int bwd_impl(const void *q, const void *c, const void *w_uk, const void *w_uv, const void *gate, float scale,
             const void *dout, const void *out_fwd, const float *lse, void *dq, void *dc, void *dw_uk, void *dw_uv,
             void *dgate, int B, int T, int H, int d_q, int d_v, int r, int dtype, void *workspace,
             size_t workspace_bytes, void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || d_q <= 0 || d_v <= 0 || r <= 0) return MLA_ERR_SHAPE;
    const long long rows = static_cast<long long>(B) * T;
    if (!mul_fits(rows, static_cast<long long>(H) * (2 * r + 4 > d_q + d_v ? 2 * r + 4 : d_q + d_v), LLONG_MAX / 8) ||
        rows > INT_MAX)
        return MLA_ERR_SHAPE;
    if (!q || !c || !w_uk || !w_uv || !dout || !dq || !dc || !dw_uk || !dw_uv) return MLA_ERR_NULL;
    if ((gate == nullptr) != (dgate == nullptr)) return MLA_ERR_NULL;   // a gate and its gradient go together
    if (!aligned16(q) || !aligned16(c) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dc) || !aligned16(dw_uk) || !aligned16(dw_uv) || (gate && !aligned16(gate)) ||
        (dgate && !aligned16(dgate)))
        return MLA_ERR_ALIGN;
    const bool r512 = dtype == MLA_DTYPE_BF16 && backward_bf16_r512_supports(r, d_q, d_v);
    if (lse && !r512) return MLA_ERR_UNSUPPORTED;
    if (lse && (!aligned16(lse) || !aligned16(out_fwd))) return MLA_ERR_ALIGN;
    if (r512) {
        if (!mul_fits(rows * H, T + 128LL, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
        if (rows == 0) return MLA_OK;
        if (!workspace) return MLA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MLA_ERR_ALIGN;
        if (workspace_bytes < backward_bf16_r512_workspace_bytes(B, T, H)) return MLA_ERR_WORKSPACE;
        DeviceInfo *dev = nullptr;
        if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
        BackwardR512Args a{q, c, w_uk, w_uv, gate, dout, static_cast<float *>(dq), static_cast<float *>(dc),
                           static_cast<float *>(dw_uk), static_cast<float *>(dw_uv), static_cast<float *>(dgate),
                           scale, B, T, H, d_q, d_v, r, workspace, workspace_bytes, dev->err_word, dev->num_sms};
        a.out_fwd = out_fwd;
        a.lse = lse;
        const cudaError_t e = launch_backward_bf16_r512(a, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
    }
    if (!backward_f32_supports(r, d_q, d_v) || T > kBackwardMaxT) return MLA_ERR_UNSUPPORTED;
    if (rows == 0) return MLA_OK;
    if (!workspace) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    if (workspace_bytes < backward_f32_workspace_bytes(B, T, H, r)) return MLA_ERR_WORKSPACE;
    BackwardArgs a{q, c, w_uk, w_uv, gate, dout, dq, dc, dw_uk, dw_uv, dgate, scale, B, T, H, d_q, d_v, r, workspace,
                   dtype == MLA_DTYPE_BF16};
    const cudaError_t e = launch_backward_f32(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
}  // namespace

MLA_API int mla_absorbed_attn_bwd(const void *q, const void *c, const void *w_uk, const void *w_uv, const void *gate,
                                  float scale, const void *dout, void *dq, void *dc, void *dw_uk, void *dw_uv,
                                  void *dgate, int B, int T, int H, int d_q, int d_v, int r, int dtype,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    return bwd_impl(q, c, w_uk, w_uv, gate, scale, dout, nullptr, nullptr, dq, dc, dw_uk, dw_uv, dgate, B, T, H, d_q,
                    d_v, r, dtype, workspace, workspace_bytes, stream);
}

MLA_API int mla_absorbed_attn_bwd_lse(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                      const void *gate, float scale, const void *dout, const void *out,
                                      const float *lse, void *dq, void *dc, void *dw_uk, void *dw_uv, void *dgate,
                                      int B, int T, int H, int d_q, int d_v, int r, int dtype, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    if (!out || !lse) return MLA_ERR_NULL;
    return bwd_impl(q, c, w_uk, w_uv, gate, scale, dout, out, lse, dq, dc, dw_uk, dw_uv, dgate, B, T, H, d_q, d_v, r,
                    dtype, workspace, workspace_bytes, stream);
}

MLA_API size_t mla_latent_decode_workspace_size(int B, int H, int r, int max_len) {
    if (B <= 0 || H <= 0 || r <= 0 || max_len < 0) return 0;
    if (!decode_bf16_supports(H, 128, r)) return 0;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return 0;
    return decode_bf16_workspace_bytes(B, H, r, max_len, dev->num_sms);
}

MLA_API int mla_latent_decode(const void *q_abs, const void *c_cache, long long ld_cache, const int *lens,
                              int max_len, const void *w_uv, const void *gate, float scale, void *out, int B,
                              int H, int d_v, int r, int dtype, void *workspace, size_t workspace_bytes,
                              void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || H <= 0 || d_v <= 0 || r <= 0 || max_len < 0 || ld_cache < r) return MLA_ERR_SHAPE;
    if (!mul_fits(static_cast<long long>(B) * max_len, ld_cache, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (!q_abs || !c_cache || !lens || !w_uv || !out) return MLA_ERR_NULL;
    if (!aligned16(q_abs) || !aligned16(c_cache) || !aligned16(w_uv) || !aligned16(out) ||
        !aligned16(lens) || (gate && !aligned16(gate)) || (ld_cache % 8) != 0)
        return MLA_ERR_ALIGN;
    if (dtype != MLA_DTYPE_BF16 || !decode_bf16_supports(H, d_v, r)) return MLA_ERR_UNSUPPORTED;
    if (B == 0) return MLA_OK;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    const size_t need = decode_bf16_workspace_bytes(B, H, r, max_len, dev->num_sms);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MLA_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return MLA_ERR_ALIGN;
    DecodeArgs a{q_abs, c_cache, w_uv, gate, lens, out, ld_cache, max_len, scale, B, H, d_v, r,
                 workspace, workspace_bytes, dev->err_word, dev->num_sms};
    const cudaError_t e = launch_decode_bf16(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_latent_decode_fp8_workspace_size(int B, int H, int r, int max_len) {
    if (B <= 0 || H <= 0 || r <= 0 || max_len < 0) return 0;
    if (!decode_bf16_supports(H, 128, r)) return 0;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return 0;
    return decode_fp8_workspace_bytes(B, H, r, max_len, dev->num_sms);
}

MLA_API int mla_latent_decode_fp8(const void *q_abs, const void *c8_cache, long long ld_cache, const int *lens,
                                  int max_len, float cache_scale, const void *w_uv, const void *gate, float scale,
                                  void *out, int B, int H, int d_v, int r, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (B < 0 || H <= 0 || d_v <= 0 || r <= 0 || max_len < 0 || ld_cache < r) return MLA_ERR_SHAPE;
    if (!(cache_scale > 0.f) || cache_scale > 3.0e38f) return MLA_ERR_SHAPE;   // positive and finite
    if (!mul_fits(static_cast<long long>(B) * max_len, ld_cache, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (!q_abs || !c8_cache || !lens || !w_uv || !out) return MLA_ERR_NULL;
    if (!aligned16(q_abs) || !aligned16(c8_cache) || !aligned16(w_uv) || !aligned16(out) || !aligned16(lens) ||
        (gate && !aligned16(gate)) || (ld_cache % 16) != 0)
        return MLA_ERR_ALIGN;
    if (!decode_bf16_supports(H, d_v, r)) return MLA_ERR_UNSUPPORTED;
    if (B == 0) return MLA_OK;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    const size_t need = decode_fp8_workspace_bytes(B, H, r, max_len, dev->num_sms);
    if (!workspace || workspace_bytes < need) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    DecodeArgs a{q_abs, c8_cache, w_uv, gate, lens, out, ld_cache, max_len, scale, B, H, d_v, r,
                 workspace, workspace_bytes, dev->err_word, dev->num_sms, cache_scale};
    const cudaError_t e = launch_decode_fp8(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_quantize_latent_fp8(const void *c, long long ld_c, void *c8, long long ld_c8, long long rows, int r,
                                    float cache_scale, void *stream) {
    if (rows < 0 || r <= 0 || (r % 8) != 0 || ld_c < r || ld_c8 < r) return MLA_ERR_SHAPE;
    if (!(cache_scale > 0.f) || cache_scale > 3.0e38f) return MLA_ERR_SHAPE;
    if (!mul_fits(rows, ld_c, LLONG_MAX / 8) || !mul_fits(rows, ld_c8, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (rows == 0) return MLA_OK;
    if (!c || !c8) return MLA_ERR_NULL;
    if (!aligned16(c) || !aligned16(c8) || (ld_c % 8) != 0 || (ld_c8 % 16) != 0) return MLA_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    const float inv_scale = 1.0f / cache_scale;
    const cudaError_t e = launch_quantize_latent_e4m3(c, ld_c, c8, ld_c8, rows, r, inv_scale,
                                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_latent_decode_noalloc(const void *q_abs, const void *c_cache, long long ld_cache, const int *lens,
                                      int max_len, const void *w_uv, const void *gate, float scale, void *out,
                                      int B, int H, int d_v, int r, int dtype, void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || H <= 0 || d_v <= 0 || r <= 0 || max_len < 0 || ld_cache < r) return MLA_ERR_SHAPE;
    if (!mul_fits(static_cast<long long>(B) * max_len, ld_cache, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (!q_abs || !c_cache || !lens || !w_uv || !out) return MLA_ERR_NULL;
    if (!aligned16(q_abs) || !aligned16(c_cache) || !aligned16(w_uv) || !aligned16(out) ||
        !aligned16(lens) || (gate && !aligned16(gate)) || (ld_cache % 8) != 0)
        return MLA_ERR_ALIGN;
    if (dtype != MLA_DTYPE_BF16 || !decode_bf16_supports(H, d_v, r)) return MLA_ERR_UNSUPPORTED;
    if (B == 0) return MLA_OK;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    const size_t need = decode_bf16_workspace_bytes(B, H, r, max_len, dev->num_sms);
    if (need > decode_noalloc_scratch_capacity()) return MLA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (decode_noalloc_scratch(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
    DecodeArgs a{q_abs, c_cache, w_uv, gate, lens, out, ld_cache, max_len, scale, B, H, d_v, r,
                 scratch, decode_noalloc_scratch_capacity(), dev->err_word, dev->num_sms};
    const cudaError_t e = launch_decode_bf16(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_gated_layer_workspace_size(int B, int T, int D, int H, int d_q, int d_v, int r, int r_q,
                                              int dtype) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return 0;
    if (B < 0 || T < 0) return 0;
    const bool f32 = dtype == MLA_DTYPE_F32;
    if (!gated_layer_supports(D, H, d_q, d_v, r, r_q, f32)) return 0;
    const long long M = static_cast<long long>(B) * T;
    if (M > INT_MAX) return 0;
    return gated_layer_workspace_bytes(M, D, H, d_q, d_v, r, r_q, f32);
}

MLA_API int mla_gated_layer_fwd(const void *x, const void *w_q_down, const void *w_q_up, const void *w_kv_down,
                                const void *w_kv_up, const void *w_gate, const void *w_o, float scale, void *y,
                                int B, int T, int D, int H, int d_q, int d_v, int r, int r_q, int dtype,
                                void *workspace, size_t workspace_bytes, void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || T < 0 || D <= 0 || H <= 0 || d_q <= 0 || d_v <= 0 || r <= 0 || r_q <= 0) return MLA_ERR_SHAPE;
    const long long M = static_cast<long long>(B) * T;
    const long long widest = static_cast<long long>(H) * (d_q + d_v) > D ? static_cast<long long>(H) * (d_q + d_v)
                                                                          : static_cast<long long>(D);
    if (M > INT_MAX || !mul_fits(M, widest > r_q ? widest : r_q, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (!x || !w_q_down || !w_q_up || !w_kv_down || !w_kv_up || !w_gate || !w_o || !y) return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_q_down) || !aligned16(w_q_up) || !aligned16(w_kv_down) ||
        !aligned16(w_kv_up) || !aligned16(w_gate) || !aligned16(w_o) || !aligned16(y))
        return MLA_ERR_ALIGN;
    const bool f32 = dtype == MLA_DTYPE_F32;
    if (!gated_layer_supports(D, H, d_q, d_v, r, r_q, f32) || (f32 && T > kPrefillF32MaxT)) return MLA_ERR_UNSUPPORTED;
    if (M == 0) return MLA_OK;
    const size_t need = gated_layer_workspace_bytes(M, D, H, d_q, d_v, r, r_q, f32);
    if (!workspace || workspace_bytes < need) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    LayerArgs a{x, w_q_down, w_q_up, w_kv_down, w_kv_up, w_gate, w_o, y, scale, B, T, D, H, d_q, d_v, r, r_q,
                f32, workspace, workspace_bytes, dev->err_word, dev->num_sms};
    const cudaError_t e = launch_gated_layer(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_gated_layer_decode_workspace_size(int B, int D, int H, int d_q, int d_v, int r, int r_q,
                                                     int max_len, int dtype) {
    if (dtype != MLA_DTYPE_BF16 || B <= 0 || max_len < 0) return 0;
    if (!gated_layer_decode_supports(D, H, d_q, d_v, r, r_q)) return 0;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return 0;
    return gated_layer_decode_workspace_bytes(B, D, H, d_q, d_v, r, r_q, max_len, dev->num_sms);
}

MLA_API int mla_gated_layer_decode(const void *x, const void *w_q_down, const void *w_q_up, const void *w_kv_down,
                                   const void *w_kv_up, const void *w_gate, const void *w_o, float scale, void *y,
                                   void *c_cache, long long ld_cache, const int *lens, int max_len, int B, int D,
                                   int H, int d_q, int d_v, int r, int r_q, int dtype, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_F32) return MLA_ERR_DTYPE;
    if (B < 0 || D <= 0 || H <= 0 || d_q <= 0 || d_v <= 0 || r <= 0 || r_q <= 0 || max_len < 0 || ld_cache < r)
        return MLA_ERR_SHAPE;
    if (!mul_fits(static_cast<long long>(B) * max_len, ld_cache, LLONG_MAX / 8)) return MLA_ERR_SHAPE;
    if (!x || !w_q_down || !w_q_up || !w_kv_down || !w_kv_up || !w_gate || !w_o || !y || !c_cache || !lens)
        return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_q_down) || !aligned16(w_q_up) || !aligned16(w_kv_down) ||
        !aligned16(w_kv_up) || !aligned16(w_gate) || !aligned16(w_o) || !aligned16(y) || !aligned16(c_cache) ||
        !aligned16(lens) || (ld_cache % 8) != 0)
        return MLA_ERR_ALIGN;
    if (dtype != MLA_DTYPE_BF16 || !gated_layer_decode_supports(D, H, d_q, d_v, r, r_q)) return MLA_ERR_UNSUPPORTED;
    if (B == 0) return MLA_OK;
    if (!workspace) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (workspace_bytes < gated_layer_decode_workspace_bytes(B, D, H, d_q, d_v, r, r_q, max_len, dev->num_sms))
        return MLA_ERR_WORKSPACE;
    LayerDecodeArgs a{x, w_q_down, w_q_up, w_kv_down, w_kv_up, w_gate, w_o, y, c_cache, ld_cache, lens, max_len,
                      scale, B, D, H, d_q, d_v, r, r_q, workspace, workspace_bytes, dev->err_word, dev->num_sms};
    const cudaError_t e = launch_gated_layer_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_debug_wait_timeout(unsigned int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 2000000u) return MLA_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    note_launch();
    wait_timeout_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(dev->err_word,
                                                                             uint64_t(limit_us) * 1000u);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_get_device_error(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
    DeviceInfo *dev = nullptr;
    if (device_info(dev) != cudaSuccess) return MLA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, dev->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    return word;
}

}  // extern "C"
