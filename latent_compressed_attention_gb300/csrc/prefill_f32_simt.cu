// fp32 causal absorbed Gated-MLA prefill on the CUDA cores (true fp32 FMA, no
// TF32), for the toy layer sizes (r, d_q, d_v <= 64).
//
// Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）", steps 2-4, fused
// into one kernel: each thread owns one (b, t, h) query row, absorbs W_UK into
// its query (step 2), streams the latent rows u <= t through shared memory
// with an online softmax (scores and the latent weighting of step 3 share the
// same c rows), then applies W_UV^T and the sigmoid gate (step 4).
//
// One CTA = one (b, h) and 128 consecutive tokens.  Work per token grows with
// t, so the grid is ordered heaviest tile first.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kMaxDim = 64;   // r, d_q, d_v limit of this kernel
constexpr int kRows = 128;    // tokens per CTA (one per thread)
constexpr int kKeys = 64;     // latent rows staged per shared-memory tile

__global__ void __launch_bounds__(kRows) prefill_f32_kernel(const float *__restrict__ q,
                                                            const float *__restrict__ c,
                                                            const float *__restrict__ w_uk,
                                                            const float *__restrict__ w_uv,
                                                            const float *__restrict__ gate,
                                                            float *__restrict__ out, float scale, int T,
                                                            int H, int d_q, int d_v, int r) {
    __shared__ float s_wuk[kMaxDim * kMaxDim];
    __shared__ float s_wuv[kMaxDim * kMaxDim];
    __shared__ float s_c[kKeys * kMaxDim];

    const int n_tiles = (T + kRows - 1) / kRows;
    const int tile = n_tiles - 1 - static_cast<int>(blockIdx.x);   // heaviest first
    const int h = blockIdx.y, b = blockIdx.z;
    const int t = tile * kRows + static_cast<int>(threadIdx.x);
    const bool active = t < T;

    for (int i = threadIdx.x; i < d_q * r; i += kRows) s_wuk[i] = w_uk[(size_t)h * d_q * r + i];
    for (int i = threadIdx.x; i < d_v * r; i += kRows) s_wuv[i] = w_uv[(size_t)h * d_v * r + i];
    __syncthreads();

    // step 2: q_abs = q_h . W_UK,h
    float qa[kMaxDim];
#pragma unroll
    for (int j = 0; j < kMaxDim; ++j) qa[j] = 0.f;
    if (active) {
        const float *qrow = q + (((size_t)b * T + t) * H + h) * d_q;
        for (int d = 0; d < d_q; ++d) {
            const float qd = qrow[d];
#pragma unroll
            for (int j = 0; j < kMaxDim; ++j)
                if (j < r) qa[j] = fmaf(qd, s_wuk[d * r + j], qa[j]);
        }
    }

    float o[kMaxDim];
#pragma unroll
    for (int j = 0; j < kMaxDim; ++j) o[j] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int last_key = min(T, (tile + 1) * kRows);   // keys this CTA needs: [0, last_key)
    const float *cb = c + (size_t)b * T * r;
    for (int k0 = 0; k0 < last_key; k0 += kKeys) {
        const int nk = min(kKeys, last_key - k0);
        __syncthreads();
        for (int i = threadIdx.x; i < nk * r; i += kRows) s_c[i] = cb[(size_t)k0 * r + i];
        __syncthreads();
        if (!active) continue;
        const int n_vis = min(nk, t - k0 + 1);   // keys u <= t in this tile
        for (int u = 0; u < n_vis; ++u) {
            const float *cu = s_c + u * r;
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxDim; ++j)
                if (j < r) s = fmaf(qa[j], cu[j], s);
            s *= scale;
            if (s > m) {   // online softmax: rescale the running sums to the new maximum
                const float corr = expf(m - s);
                l *= corr;
#pragma unroll
                for (int j = 0; j < kMaxDim; ++j) o[j] *= corr;
                m = s;
            }
            const float p = expf(s - m);
            l += p;
#pragma unroll
            for (int j = 0; j < kMaxDim; ++j)
                if (j < r) o[j] = fmaf(p, cu[j], o[j]);
        }
    }
    if (!active) return;

    // step 3 (W_UV^T) and step 4 (gate)
    const float inv_l = 1.f / l;
    float *orow = out + ((size_t)b * T + t) * H * d_v + (size_t)h * d_v;
    const float *grow = gate ? gate + ((size_t)b * T + t) * H * d_v + (size_t)h * d_v : nullptr;
    for (int v = 0; v < d_v; ++v) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxDim; ++j)
            if (j < r) acc = fmaf(o[j], s_wuv[v * r + j], acc);
        acc *= inv_l;
        if (grow) acc = acc / (1.f + expf(-grow[v]));
        orow[v] = acc;
    }
}

}  // namespace

bool prefill_f32_simt_supports(int r, int d_q, int d_v) {
    return r >= 1 && r <= kMaxDim && d_q >= 1 && d_q <= kMaxDim && d_v >= 1 && d_v <= kMaxDim;
}

cudaError_t launch_prefill_f32_simt(const PrefillArgs &a, cudaStream_t s) {
    if (!prefill_f32_simt_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    const dim3 grid((a.T + kRows - 1) / kRows, a.H, a.B);
    note_launch();
    prefill_f32_kernel<<<grid, kRows, 0, s>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.c), static_cast<const float *>(a.w_uk),
        static_cast<const float *>(a.w_uv), static_cast<const float *>(a.gate), static_cast<float *>(a.out),
        a.scale, a.T, a.H, a.d_q, a.d_v, a.r);
    return cudaGetLastError();
}

}  // namespace mla
