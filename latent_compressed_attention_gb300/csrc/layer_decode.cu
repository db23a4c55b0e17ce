// One decode step of the whole Gated-MLA layer with the latent-cache append
// (page "Gated MLA（矩阵吸收版）": section "低秩压缩" — only the rank-r latent c is
// cached; section "完整计算流（四步）" steps 1-4; W_o from the listing of section
// "代码对照"):
//
//   per sequence b, one new token x_b [D] at position lens[b]:
//     c_b     = RMSNorm(x_b . W_kv_down^T)                 written to cache row lens[b]
//     q_abs_b = (RMSNorm(x_b . W_q_down^T) . W_q_up^T) . W_UK  per head (step 2's absorb)
//     g_b     = x_b . W_gate^T
//     o_b     = decode attention of q_abs_b over cache rows [0, lens[b]] (the new row included)
//     y_b     = o_b . W_o^T
//
// The projections reuse the tensor-core GEMM (M = B rows), the attention reuses
// the cached-latent decode kernels; two small kernels here append the latents
// and absorb W_UK into the queries.  lens is read, not advanced: the caller
// moves it on after the step.  A position outside [0, max_len) is reported as
// MLA_ERR_DEVICE_BOUNDS and that sequence's latent is not written.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr float kRmsEps = 1e-6f;
constexpr int kAbsorbRows = 16;   // sequences per absorb CTA

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecLayout {
    size_t q, c, g, qa, o, yq, ss, lens1, dec, end;
};

DecLayout dec_layout(int B, int H, int d_q, int d_v, int r, int r_q, size_t dec_bytes) {
    DecLayout L;
    const size_t es = 2;
    L.q = 0;
    L.c = L.q + align256(static_cast<size_t>(B) * H * d_q * es);
    L.g = L.c + align256(static_cast<size_t>(B) * r * es);
    L.qa = L.g + align256(static_cast<size_t>(B) * H * d_v * es);
    L.o = L.qa + align256(static_cast<size_t>(B) * H * r * es);
    L.yq = L.o + align256(static_cast<size_t>(B) * H * d_v * es);
    L.ss = L.yq + align256(static_cast<size_t>(B) * r_q * es);
    L.lens1 = L.ss + align256(static_cast<size_t>(B) * sizeof(float));
    L.dec = L.lens1 + align256(static_cast<size_t>(B) * sizeof(int));
    L.end = L.dec + align256(dec_bytes);
    return L;
}

// Cache row lens[b] of sequence b <- c[b] (r bf16), and lens1[b] = rows the step attends to.
__global__ void append_latent_kernel(const __nv_bfloat16 *c, __nv_bfloat16 *cache, long long ld, const int *lens,
                                     int *lens1, int max_len, int r, int *err) {
    const int b = blockIdx.x;
    const int pos = __ldg(lens + b);
    const bool ok = pos >= 0 && pos < max_len;
    if (threadIdx.x == 0) {
        if (!ok) record_error(err, kDevErrBounds);
        lens1[b] = ok ? pos + 1 : min(max(pos, 0), max_len);
    }
    if (!ok) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(c + static_cast<size_t>(b) * r);
    uint4 *dst = reinterpret_cast<uint4 *>(cache + (static_cast<size_t>(b) * max_len + pos) * ld);
    for (int i = threadIdx.x; i < r / 8; i += blockDim.x) dst[i] = src[i];
}

// q_abs[b, h, :] = q[b, h, :] . W_UK[h] (d_q -> r), fp32 accumulation, bf16 out.
__global__ void absorb_query_kernel(const __nv_bfloat16 *q, const __nv_bfloat16 *w_uk, __nv_bfloat16 *q_abs, int B,
                                    int H, int d_q, int r) {
    extern __shared__ float qs[];   // [kAbsorbRows][d_q]
    const int h = blockIdx.x, b0 = blockIdx.y * kAbsorbRows;
    const int nb = min(kAbsorbRows, B - b0);
    for (int i = threadIdx.x; i < kAbsorbRows * d_q; i += blockDim.x) {
        const int bb = i / d_q, d = i % d_q;
        qs[i] = bb < nb ? __bfloat162float(q[(static_cast<size_t>(b0 + bb) * H + h) * d_q + d]) : 0.f;
    }
    __syncthreads();
    const __nv_bfloat16 *w = w_uk + static_cast<size_t>(h) * d_q * r;
    for (int j = threadIdx.x; j < r; j += blockDim.x) {
        float acc[kAbsorbRows];
#pragma unroll
        for (int bb = 0; bb < kAbsorbRows; ++bb) acc[bb] = 0.f;
        for (int d = 0; d < d_q; ++d) {
            const float wv = __bfloat162float(w[static_cast<size_t>(d) * r + j]);
#pragma unroll
            for (int bb = 0; bb < kAbsorbRows; ++bb) acc[bb] = fmaf(qs[bb * d_q + d], wv, acc[bb]);
        }
        for (int bb = 0; bb < nb; ++bb)
            q_abs[(static_cast<size_t>(b0 + bb) * H + h) * r + j] = __float2bfloat16_rn(acc[bb]);
    }
}

}  // namespace

bool gated_layer_decode_supports(int D, int H, int d_q, int d_v, int r, int r_q) {
    return gated_layer_supports(D, H, d_q, d_v, r, r_q, false) && decode_bf16_supports(H, d_v, r);
}

size_t gated_layer_decode_workspace_bytes(int B, int H, int d_q, int d_v, int r, int r_q, int max_len,
                                          int num_sms) {
    return dec_layout(B, H, d_q, d_v, r, r_q, decode_bf16_workspace_bytes(B, H, r, max_len, num_sms)).end;
}

cudaError_t launch_gated_layer_decode(const LayerDecodeArgs &a, cudaStream_t s) {
    const size_t dec_bytes = decode_bf16_workspace_bytes(a.B, a.H, a.r, a.max_len, a.num_sms);
    const DecLayout L = dec_layout(a.B, a.H, a.d_q, a.d_v, a.r, a.r_q, dec_bytes);
    if (a.workspace_bytes < L.end) return cudaErrorInvalidValue;
    char *ws = static_cast<char *>(a.workspace);
    auto *q = reinterpret_cast<__nv_bfloat16 *>(ws + L.q);
    auto *c = reinterpret_cast<__nv_bfloat16 *>(ws + L.c);
    auto *g = reinterpret_cast<__nv_bfloat16 *>(ws + L.g);
    auto *qa = reinterpret_cast<__nv_bfloat16 *>(ws + L.qa);
    auto *o = reinterpret_cast<__nv_bfloat16 *>(ws + L.o);
    auto *yq = reinterpret_cast<__nv_bfloat16 *>(ws + L.yq);
    auto *ss = reinterpret_cast<float *>(ws + L.ss);
    auto *lens1 = reinterpret_cast<int *>(ws + L.lens1);
    const int Hq = a.H * a.d_q, Hv = a.H * a.d_v;
    const auto *w_uk = static_cast<const __nv_bfloat16 *>(a.w_kv_up);
    const __nv_bfloat16 *w_uv = w_uk + static_cast<size_t>(Hq) * a.r;
    cudaError_t e;
    if ((e = cudaMemsetAsync(ss, 0, static_cast<size_t>(a.B) * sizeof(float), s)) != cudaSuccess) return e;
    GemmArgs gm{};
    gm.M = a.B;
    gm.dev_err = a.dev_err;
    gm.num_sms = a.num_sms;
    gm.eps = kRmsEps;
    gm.ss = ss;
    auto run = [&](const void *A, long long lda, const void *Bw, void *C, int N, int K, int epi, float n_norm) {
        gm.A = A;
        gm.lda = lda;
        gm.B = Bw;
        gm.ldb = K;
        gm.C = C;
        gm.ldc = N;
        gm.N = N;
        gm.K = K;
        gm.epilogue = epi;
        gm.n_norm = n_norm;
        return launch_gemm_bf16(gm, s);
    };
    if ((e = run(a.x, a.D, a.w_q_down, yq, a.r_q, a.D, kGemmSumSq, 0.f)) != cudaSuccess) return e;
    if ((e = run(yq, a.r_q, a.w_q_up, q, Hq, a.r_q, kGemmRowScale, static_cast<float>(a.r_q))) != cudaSuccess)
        return e;
    if ((e = run(a.x, a.D, a.w_kv_down, c, a.r, a.D, kGemmRmsNorm, static_cast<float>(a.r))) != cudaSuccess)
        return e;
    if ((e = run(a.x, a.D, a.w_gate, g, Hv, a.D, kGemmPlain, 0.f)) != cudaSuccess) return e;
    append_latent_kernel<<<a.B, 64, 0, s>>>(c, static_cast<__nv_bfloat16 *>(a.c_cache), a.ld_cache, a.lens, lens1,
                                            a.max_len, a.r, a.dev_err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 agrid(a.H, (a.B + kAbsorbRows - 1) / kAbsorbRows);
    absorb_query_kernel<<<agrid, 256, kAbsorbRows * a.d_q * sizeof(float), s>>>(q, w_uk, qa, a.B, a.H, a.d_q, a.r);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    DecodeArgs da{qa, a.c_cache, w_uv, g, lens1, o, a.ld_cache, a.max_len, a.scale, a.B, a.H, a.d_v, a.r,
                  ws + L.dec, dec_bytes, a.dev_err, a.num_sms};
    if ((e = launch_decode_bf16(da, s)) != cudaSuccess) return e;
    return run(o, Hv, a.w_o, a.y, a.D, Hv, kGemmPlain, 0.f);
}

}  // namespace mla
