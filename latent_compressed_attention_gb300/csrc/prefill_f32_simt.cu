// fp32 causal absorbed Gated-MLA prefill on the CUDA cores (true fp32 FMA, no
// TF32), for the toy layer sizes (r, d_q, d_v <= 64).
//
// Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）", steps 2-4, fused
// into one kernel.  One CTA = one (b, h) and 16 consecutive tokens (so even a
// short sequence fills the GPU); each of its 8 warps owns 2 of those query
// rows.  Per row the warp
//   absorbs W_UK into the query (step 2, lane j computes latent column j),
//   walks the latent rows u <= t in chunks of 32 that the CTA stages in
//   shared memory: lane u scores key u against q_abs (step 2), the warp takes
//   the chunk maximum and the sum with shuffles (online softmax, step 2),
//   and lane j adds sum_u p_u c[u, j] to its latent column (step 3, the same c
//   rows as the scores),
//   then applies W_UV^T and the sigmoid gate (steps 3-4, lane v computes
//   output column v).
// Short dependency chains per lane and no bank conflicts (the staged rows are
// padded to r + 1 floats) keep the warps busy; heavy tiles launch first, over all heads.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kMaxDim = 64;   // r, d_q, d_v limit of this kernel
constexpr int kRows = 16;     // tokens per CTA
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRows / kWarps;
constexpr int kKeys = 32;     // latent rows staged per chunk: one per lane
constexpr int kPad = kMaxDim + 1;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kWarps * 32) prefill_f32_kernel(const float *__restrict__ q,
                                                                  const float *__restrict__ c,
                                                                  const float *__restrict__ w_uk,
                                                                  const float *__restrict__ w_uv,
                                                                  const float *__restrict__ gate,
                                                                  float *__restrict__ out, float scale, int T,
                                                                  int H, int d_q, int d_v, int r) {
    __shared__ float s_c[kKeys * kPad];                         // staged latent rows, padded
    __shared__ float s_qa[kWarps][kRowsPerWarp][kMaxDim];       // q_abs of each warp's rows
    __shared__ float s_p[kWarps][kKeys];                        // one chunk's softmax weights
    __shared__ float s_wk[kMaxDim * kMaxDim];                   // W_UK[h] as [d_q][r]
    __shared__ float s_wv[kMaxDim * kPad];                      // W_UV[h] as [d_v][r], rows padded

    const int n_tiles = (T + kRows - 1) / kRows;
    const int tile = n_tiles - 1 - static_cast<int>(blockIdx.y);   // heaviest first, over all heads
    const int b = static_cast<int>(blockIdx.x) / H, h = static_cast<int>(blockIdx.x) % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = tile * kRows;
    const float *wuk = w_uk + static_cast<size_t>(h) * d_q * r;
    const float *wuv = w_uv + static_cast<size_t>(h) * d_v * r;
    // this head's weights, read once per CTA with coalesced loads
    for (int i = threadIdx.x; i < d_q * r; i += kWarps * 32) s_wk[i] = __ldg(wuk + i);
    for (int i = threadIdx.x; i < d_v * r; i += kWarps * 32) {
        const int v = i / r, j = i - v * r;
        s_wv[v * kPad + j] = __ldg(wuv + i);
    }
    __syncthreads();

    // step 2, absorb: q_abs[t, j] = sum_d q[b, t, h, d] W_UK[h, d, j]; lane j holds columns j and j + 32
    float o[kRowsPerWarp][2], m[kRowsPerWarp], l[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int t = t0 + i * kWarps + warp;
        o[i][0] = o[i][1] = 0.f;
        m[i] = -INFINITY;
        l[i] = 0.f;
        if (t >= T) continue;
        const float *qrow = q + ((static_cast<size_t>(b) * T + t) * H + h) * d_q;
        float a0 = 0.f, a1 = 0.f;
        for (int d = 0; d < d_q; ++d) {
            const float qd = __ldg(qrow + d);
            if (lane < r) a0 = fmaf(qd, s_wk[d * r + lane], a0);
            if (lane + 32 < r) a1 = fmaf(qd, s_wk[d * r + lane + 32], a1);
        }
        s_qa[warp][i][lane] = a0;
        s_qa[warp][i][lane + 32] = a1;
    }
    __syncwarp();

    const int last_key = min(T, t0 + kRows);   // keys this CTA needs: [0, last_key)
    const float *cb = c + static_cast<size_t>(b) * T * r;
    for (int k0 = 0; k0 < last_key; k0 += kKeys) {
        __syncthreads();
        for (int i = threadIdx.x; i < kKeys * r; i += kWarps * 32) {
            const int u = i / r, j = i - u * r;
            s_c[u * kPad + j] = k0 + u < T ? __ldg(cb + static_cast<size_t>(k0 + u) * r + j) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int t = t0 + i * kWarps + warp;
            if (t >= T || k0 > t) continue;   // warp-uniform
            const int n_vis = min(kKeys, t - k0 + 1);   // keys u <= t of this chunk
            // scores: lane u against key k0 + u
            float s = -INFINITY;
            if (lane < n_vis) {
                float acc0 = 0.f, acc1 = 0.f;
                const float *cu = s_c + lane * kPad;
                const float *qa = s_qa[warp][i];
                int j = 0;
                for (; j + 1 < r; j += 2) {
                    acc0 = fmaf(qa[j], cu[j], acc0);
                    acc1 = fmaf(qa[j + 1], cu[j + 1], acc1);
                }
                if (j < r) acc0 = fmaf(qa[j], cu[j], acc0);
                s = (acc0 + acc1) * scale;
            }
            // online softmax over the chunk
            const float m_new = fmaxf(m[i], warp_max(s));
            const float corr = expf(m[i] - m_new);   // 0 on the first chunk (m = -inf)
            const float p = lane < n_vis ? expf(s - m_new) : 0.f;
            l[i] = l[i] * corr + warp_sum(p);
            m[i] = m_new;
            s_p[warp][lane] = p;
            __syncwarp();
            // step 3, latent weighting: lane j adds sum_u p_u c[u, j]
            float a0 = 0.f, a1 = 0.f;
            for (int u = 0; u < n_vis; ++u) {
                const float pu = s_p[warp][u];
                a0 = fmaf(pu, s_c[u * kPad + lane], a0);
                a1 = fmaf(pu, s_c[u * kPad + lane + 32], a1);
            }
            o[i][0] = fmaf(o[i][0], corr, a0);
            o[i][1] = fmaf(o[i][1], corr, a1);
            __syncwarp();
        }
    }

    // step 3 (W_UV^T) and step 4 (gate): lane v computes output columns v and v + 32
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int t = t0 + i * kWarps + warp;
        if (t >= T) continue;
        const float inv_l = 1.f / l[i];
        float *ol = s_qa[warp][i];   // this row's q_abs is no longer needed: reuse it for o_lat / l
        ol[lane] = o[i][0] * inv_l;
        ol[lane + 32] = o[i][1] * inv_l;
        __syncwarp();
        float *orow = out + (static_cast<size_t>(b) * T + t) * H * d_v + static_cast<size_t>(h) * d_v;
        const float *grow = gate ? gate + (static_cast<size_t>(b) * T + t) * H * d_v + static_cast<size_t>(h) * d_v
                                 : nullptr;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int v = lane + 32 * half;
            if (v >= d_v) continue;
            const float *wv = s_wv + v * kPad;   // lanes read rows kPad apart: distinct banks
            float acc = 0.f;
            for (int j = 0; j < r; ++j) acc = fmaf(ol[j], wv[j], acc);
            if (grow) acc = acc / (1.f + expf(-grow[v]));
            orow[v] = acc;
        }
        __syncwarp();
    }
}

}  // namespace

bool prefill_f32_simt_supports(int r, int d_q, int d_v) {
    return r >= 1 && r <= kMaxDim && d_q >= 1 && d_q <= kMaxDim && d_v >= 1 && d_v <= kMaxDim;
}

cudaError_t launch_prefill_f32_simt(const PrefillArgs &a, cudaStream_t s) {
    if (!prefill_f32_simt_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    // (b, h) is the fastest grid index, so the heaviest tiles of every head are dispatched first
    const unsigned tiles = static_cast<unsigned>((a.T + kRows - 1) / kRows);
    if (tiles > 65535u) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(a.B) * static_cast<unsigned>(a.H), tiles);
    note_launch();
    prefill_f32_kernel<<<grid, kWarps * 32, 0, s>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.c), static_cast<const float *>(a.w_uk),
        static_cast<const float *>(a.w_uv), static_cast<const float *>(a.gate), static_cast<float *>(a.out),
        a.scale, a.T, a.H, a.d_q, a.d_v, a.r);
    return cudaGetLastError();
}

}  // namespace mla
