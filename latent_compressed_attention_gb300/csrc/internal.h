// Internal host-side interface between the C ABI (abi.cu) and the kernel
// translation units.  Not exported from the shared library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mla {

struct PrefillArgs {
    const void *q, *c, *w_uk, *w_uv, *gate;
    void *out;
    float scale;
    int B, T, H, d_q, d_v, r;
    int *dev_err;  // device error word of the current device
    int num_sms;
    void *workspace = nullptr;   // prefill_workspace_bytes() bytes (none for the fp32 and small-rank kernels)
    size_t workspace_bytes = 0;
    // optional (r = 512 kernel): each row's log-sum-exp of the scaled scores, [B, H, T] fp32, natural log:
    // lse = ln sum_u exp(scale q_abs . c_u), so attn = exp(scale q_abs . c_u - lse)
    float *lse = nullptr;
};

struct DecodeArgs {
    const void *q_abs, *c_cache, *w_uv, *gate;
    const int *lens;
    void *out;
    long long ld_cache;
    int max_len;
    float scale;
    int B, H, d_v, r;
    void *workspace;
    size_t workspace_bytes;
    int *dev_err;
    int num_sms;
    float cache_scale = 1.f;   // e4m3 cache: it holds c / cache_scale
};

struct BackwardArgs {
    const void *q, *c, *w_uk, *w_uv, *gate, *dout;
    void *dq, *dc, *dw_uk, *dw_uv, *dgate;
    float scale;
    int B, T, H, d_q, d_v, r;
    void *workspace;   // backward_f32_workspace_bytes(B, T, H, r)
    bool bf16;         // inputs bf16 (else fp32); the gradients are fp32 either way
};

// Each launcher validates nothing the ABI already checked; it returns a
// cudaError_t from the launch (or cudaErrorInvalidValue for an internal
// precondition) and never synchronises.
cudaError_t launch_prefill_f32_simt(const PrefillArgs &a, cudaStream_t s);
bool prefill_f32_simt_supports(int r, int d_q, int d_v);
// Longest sequences of the fp32 prefill and of the backward: their grids put the tile rank (16 or 64
// tokens) on the y index, at most 65535.
constexpr long long kPrefillF32MaxT = 65535LL * 16;
constexpr long long kBackwardMaxT = 65535LL * 64;

cudaError_t launch_prefill_bf16_r512(const PrefillArgs &a, cudaStream_t s);
bool prefill_bf16_r512_supports(int r, int d_q, int d_v);
size_t prefill_bf16_r512_workspace_bytes(long long B, long long T);
// Device workspace a prefill call of these sizes needs (0 for the kernels that need none).
inline size_t prefill_workspace_bytes(long long B, long long T, int r, int d_q, int d_v, bool f32) {
    return (!f32 && prefill_bf16_r512_supports(r, d_q, d_v)) ? prefill_bf16_r512_workspace_bytes(B, T) : 0;
}

cudaError_t launch_prefill_bf16_small(const PrefillArgs &a, cudaStream_t s);

// Gradients of the attention at r = 512, d_q = d_v = 128, bf16 inputs, fp32 gradients (tensor cores).
struct BackwardR512Args {
    const void *q, *c, *w_uk, *w_uv, *gate, *dout;
    float *dq, *dc, *dw_uk, *dw_uv, *dgate;
    float scale;
    int B, T, H, d_q, d_v, r;
    void *workspace;
    size_t workspace_bytes;
    int *dev_err;
    int num_sms;
    // optional: the forward's output (after the gate) and each row's log-sum-exp from a forward call with
    // lse; given both, the forward is not run again
    const void *out_fwd = nullptr;
    const float *lse = nullptr;
};
bool backward_bf16_r512_supports(int r, int d_q, int d_v);
size_t backward_bf16_r512_workspace_bytes(long long B, long long T, long long H);
cudaError_t launch_backward_bf16_r512(const BackwardR512Args &a, cudaStream_t s);

// fp32 gradients of the attention (steps 2-4); r, d_q, d_v <= 64.
bool backward_f32_supports(int r, int d_q, int d_v);
size_t backward_f32_workspace_bytes(long long B, long long T, long long H, int r);
cudaError_t launch_backward_f32(const BackwardArgs &a, cudaStream_t s);
bool prefill_bf16_small_supports(int r, int d_q, int d_v);

size_t decode_bf16_workspace_bytes(int B, int H, int r, int max_len, int num_sms);
cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s);
// The same decode over an e4m3 latent cache (c_cache holds bytes, ld_cache in bytes).
size_t decode_fp8_workspace_bytes(int B, int H, int r, int max_len, int num_sms);
cudaError_t launch_decode_fp8(const DecodeArgs &a, cudaStream_t s);
// c [rows][r] bf16 -> e4m3(c * inv_scale) [rows][r] bytes.
cudaError_t launch_quantize_latent_e4m3(const void *c, long long ld_c, void *c8, long long ld_c8, long long rows, int r,
                                        float inv_scale, cudaStream_t s);
bool decode_bf16_supports(int H, int d_v, int r);

// Scratch of the no-alloc decode entry point: capacity in bytes, and its
// device address on the current device (set up once per device).
size_t decode_noalloc_scratch_capacity();
cudaError_t decode_noalloc_scratch(void **ptr);

// bf16 tensor-core GEMM C[M,N] = A[M,K] . B[N,K]^T (both row-major, K-major operands), fp32
// accumulation, bf16 output, with the epilogues the layer's projections need.
enum GemmEpilogue { kGemmPlain = 0, kGemmSumSq = 1, kGemmRowScale = 2, kGemmRmsNorm = 3 };
struct GemmArgs {
    const void *A, *B;
    void *C;
    float *ss;   // row sums of squares: accumulated (kGemmSumSq) or read (kGemmRowScale)
    int M, N, K;
    long long lda, ldb, ldc;   // elements
    int epilogue;
    float n_norm, eps;         // RMSNorm divisor (columns of the normalised row) and epsilon
    int *dev_err;
    int num_sms;
    // Split K (few row tiles): zeroed scratch of gemm_bf16_split_bytes() bytes, or NULL = never split
    float *split_acc;
};
bool gemm_bf16_supports(int N, int K, int epilogue);
size_t gemm_bf16_split_bytes(const GemmArgs &g);   // 0: this product does not split
cudaError_t launch_gemm_bf16(const GemmArgs &g, cudaStream_t s);

// The whole Gated-MLA layer: step-1 projections, the absorbed attention, W_o.
struct LayerArgs {
    const void *x, *w_q_down, *w_q_up, *w_kv_down, *w_kv_up, *w_gate, *w_o;
    void *y;
    float scale;
    int B, T, D, H, d_q, d_v, r, r_q;
    bool f32;
    void *workspace;
    size_t workspace_bytes;
    int *dev_err;
    int num_sms;
};
bool gated_layer_supports(int D, int H, int d_q, int d_v, int r, int r_q, bool f32);
// The layer's five bf16 projections in the order they run, and the zeroed split-K
// scratch each reserves: slice i is [off[i], off[i + 1]) (empty = never splits), sized
// for any device of up to 256 SMs; off[kLayerGemms] is the total.
enum LayerGemm { kQDown = 0, kQUp, kKvDown, kGate, kOProj, kLayerGemms };
size_t layer_split_plan(long long M, int D, int H, int d_q, int d_v, int r, int r_q, size_t off[kLayerGemms + 1]);
size_t gated_layer_workspace_bytes(long long M, int D, int H, int d_q, int d_v, int r, int r_q, bool f32);
cudaError_t launch_gated_layer(const LayerArgs &a, cudaStream_t s);

// One decode step of the whole layer: the new token's latent is appended to the cache at
// row lens[b], then the sequence attends to rows [0, lens[b]].
struct LayerDecodeArgs {
    const void *x, *w_q_down, *w_q_up, *w_kv_down, *w_kv_up, *w_gate, *w_o;
    void *y;
    void *c_cache;
    long long ld_cache;
    const int *lens;
    int max_len;
    float scale;
    int B, D, H, d_q, d_v, r, r_q;
    void *workspace;
    size_t workspace_bytes;
    int *dev_err;
    int num_sms;
};
bool gated_layer_decode_supports(int D, int H, int d_q, int d_v, int r, int r_q);
size_t gated_layer_decode_workspace_bytes(int B, int D, int H, int d_q, int d_v, int r, int r_q, int max_len,
                                          int num_sms);
cudaError_t launch_gated_layer_decode(const LayerDecodeArgs &a, cudaStream_t s);

// Driver entry point for cuTensorMapEncodeTiled, resolved once through the runtime.
void *tensor_map_encode_fn();

// Count one kernel launch of this library (read by mla_kernel_launches).
void note_launch();

}  // namespace mla
