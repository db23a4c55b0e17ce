// fp32 gradients of the causal absorbed Gated-MLA attention (steps 2-4) on the
// CUDA cores (true fp32 FMA, no TF32), for the toy sizes (r, d_q, d_v <= 64);
// inputs fp32 or bf16 (read and widened to fp32), gradients fp32.
//
// The page "Gated MLA（矩阵吸收版）" gives the forward (section "完整计算流（四步）":
// q_abs = q W_UK, s = scale q_abs c^T masked to u <= t, a = softmax(s),
// o_lat = a c, o = o_lat W_UV^T, out = sigmoid(g) o).  The backward takes the
// chain rule back through those steps:
//   step 4   dg = dout o sg (1 - sg),  do = dout sg                   (sg = sigmoid(g))
//   step 3   dW_UV += do^T o_lat,  do_lat = do W_UV,  da = do_lat c^T,  dc += a^T do_lat
//   softmax  ds = a (da - delta),  delta_t = sum_u a_tu da_tu = do_lat_t . o_lat_t
//   step 2   dq_abs = scale ds c,  dc += scale ds^T q_abs,  dq = dq_abs W_UK^T,  dW_UK += q^T dq_abs
// Two kernels:
//   query kernel: one CTA per (b, h, 16 tokens), a warp per query row (two rows per warp).  It
//     recomputes q_abs and the softmax statistics and o_lat over the keys u <= t (staged 32 at a time,
//     rows padded to r + 1 floats), forms do, do_lat, delta and dgate, and in a second pass over the keys
//     dq_abs; it writes dq and dgate, and q_abs, do_lat and (m, l, delta) for the key kernel.  dW_UK and
//     dW_UV are summed per CTA in shared memory and added to global memory once per CTA.
//   key kernel: one CTA per (b, h, 16 keys), a warp per key (two per warp).  For the queries t >= u
//     (staged 32 at a time) it recomputes a_tu and ds_tu and adds this head's part of
//     dc_u = sum_t a_tu do_lat_t + scale ds_tu q_abs_t.
// dc, dW_UK and dW_UV are sums over blocks, so they are zeroed first and added with atomics.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kMaxDim = 64;    // r, d_q, d_v limit
constexpr int kRows = 16;      // query rows (query kernel) or keys (key kernel) per CTA
constexpr int kWarps = 8;
constexpr int kPerWarp = kRows / kWarps;   // 2
constexpr int kChunk = 32;     // staged keys (query kernel) or queries (key kernel)
constexpr int kPad = kMaxDim + 1;

template <typename In>
struct BwdParams {
    const In *q, *c, *w_uk, *w_uv, *gate, *dout;
    float *dq, *dc, *dw_uk, *dw_uv, *dgate;
    float *ws_qa, *ws_dol, *ws_st;   // [B,T,H,r], [B,T,H,r], [B,T,H,4] = (m, l, delta, 0)
    float scale;
    int B, T, H, d_q, d_v, r;
};

__device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }

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

// Shared memory of the query kernel, in floats.
constexpr int kQC = 0;                                        // [kChunk][kPad] staged latent rows
constexpr int kQQa = kQC + kChunk * kPad;                     // [kWarps][kPerWarp][kMaxDim] q_abs
constexpr int kQDol = kQQa + kWarps * kPerWarp * kMaxDim;     // [kWarps][kPerWarp][kMaxDim] do_lat
constexpr int kQVec = kQDol + kWarps * kPerWarp * kMaxDim;    // [kWarps][kMaxDim] per-warp vector
constexpr int kQP = kQVec + kWarps * kMaxDim;                 // [kWarps][kChunk] per-key weights
constexpr int kQDwuk = kQP + kWarps * kChunk;                 // [kMaxDim][kMaxDim] dW_UK partial (d, j)
constexpr int kQDwuv = kQDwuk + kMaxDim * kMaxDim;            // [kMaxDim][kMaxDim] dW_UV partial (v, j)
constexpr int kQFloats = kQDwuv + kMaxDim * kMaxDim;
constexpr size_t kQSmem = kQFloats * sizeof(float);

template <typename In>
__global__ void __launch_bounds__(kWarps * 32) bwd_query_kernel(const BwdParams<In> p) {
    extern __shared__ float sm[];
    float *s_c = sm + kQC, *s_qa = sm + kQQa, *s_dol = sm + kQDol, *s_vec = sm + kQVec, *s_p = sm + kQP;
    float *s_dwuk = sm + kQDwuk, *s_dwuv = sm + kQDwuv;
    const int T = p.T, H = p.H, r = p.r, dq_dim = p.d_q, dv = p.d_v;
    const int n_tiles = (T + kRows - 1) / kRows;
    const int tile = n_tiles - 1 - static_cast<int>(blockIdx.x);   // heaviest first
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = tile * kRows;
    const In *wuk = p.w_uk + static_cast<size_t>(h) * dq_dim * r;
    const In *wuv = p.w_uv + static_cast<size_t>(h) * dv * r;
    float *vec = s_vec + warp * kMaxDim;
    float *pw = s_p + warp * kChunk;

    for (int i = threadIdx.x; i < 2 * kMaxDim * kMaxDim; i += kWarps * 32) s_dwuk[i] = 0.f;   // both partials

    // step 2 absorb: q_abs[t, j] = sum_d q[b, t, h, d] W_UK[h, d, j]; lane j holds columns j and j + 32
    float m[kPerWarp], l[kPerWarp], ol[kPerWarp][2], delta[kPerWarp], dqa[kPerWarp][2];
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int t = t0 + i * kWarps + warp;
        m[i] = -INFINITY;
        l[i] = 0.f;
        ol[i][0] = ol[i][1] = delta[i] = dqa[i][0] = dqa[i][1] = 0.f;
        float a0 = 0.f, a1 = 0.f;
        if (t < T) {
            const In *qrow = p.q + ((static_cast<size_t>(b) * T + t) * H + h) * dq_dim;
            for (int d = 0; d < dq_dim; ++d) {
                const float qd = ld(qrow + d);
                if (lane < r) a0 = fmaf(qd, ld(wuk + d * r + lane), a0);
                if (lane + 32 < r) a1 = fmaf(qd, ld(wuk + d * r + lane + 32), a1);
            }
        }
        s_qa[(warp * kPerWarp + i) * kMaxDim + lane] = a0;
        s_qa[(warp * kPerWarp + i) * kMaxDim + lane + 32] = a1;
    }
    __syncwarp();

    const int last_key = min(T, t0 + kRows);   // keys this CTA needs: [0, last_key)
    const In *cb = p.c + static_cast<size_t>(b) * T * r;
    auto stage = [&](int k0) {
        __syncthreads();
        for (int i = threadIdx.x; i < kChunk * r; i += kWarps * 32) {
            const int u = i / r, j = i - u * r;
            s_c[u * kPad + j] = k0 + u < T ? ld(cb + static_cast<size_t>(k0 + u) * r + j) : 0.f;
        }
        __syncthreads();
    };
    auto score = [&](const float *qa, int u) {   // q_abs . c_u over the latent columns
        const float *cu = s_c + u * kPad;
        float acc0 = 0.f, acc1 = 0.f;
        int j = 0;
        for (; j + 1 < r; j += 2) {
            acc0 = fmaf(qa[j], cu[j], acc0);
            acc1 = fmaf(qa[j + 1], cu[j + 1], acc1);
        }
        if (j < r) acc0 = fmaf(qa[j], cu[j], acc0);
        return acc0 + acc1;
    };

    // pass 1: the softmax statistics and o_lat (the forward, recomputed)
    for (int k0 = 0; k0 < last_key; k0 += kChunk) {
        stage(k0);
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int t = t0 + i * kWarps + warp;
            if (t >= T || k0 > t) continue;   // warp-uniform
            const int n_vis = min(kChunk, t - k0 + 1);
            const float s = lane < n_vis ? score(s_qa + (warp * kPerWarp + i) * kMaxDim, lane) * p.scale : -INFINITY;
            const float m_new = fmaxf(m[i], warp_max(s));
            const float corr = expf(m[i] - m_new);
            const float e = lane < n_vis ? expf(s - m_new) : 0.f;
            l[i] = l[i] * corr + warp_sum(e);
            m[i] = m_new;
            pw[lane] = e;
            __syncwarp();
            float a0 = 0.f, a1 = 0.f;
            for (int u = 0; u < n_vis; ++u) {
                a0 = fmaf(pw[u], s_c[u * kPad + lane], a0);
                a1 = fmaf(pw[u], s_c[u * kPad + lane + 32], a1);
            }
            ol[i][0] = fmaf(ol[i][0], corr, a0);
            ol[i][1] = fmaf(ol[i][1], corr, a1);
            __syncwarp();
        }
    }

    // steps 4 and 3 backward, per row
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int t = t0 + i * kWarps + warp;
        if (t >= T) continue;
        const size_t row = (static_cast<size_t>(b) * T + t) * H + h;
        const float inv_l = 1.f / l[i];
        ol[i][0] *= inv_l;
        ol[i][1] *= inv_l;
        vec[lane] = ol[i][0];
        vec[lane + 32] = ol[i][1];
        __syncwarp();
        float dov[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {   // lane v: o_v, dgate_v, do_v
            const int v = lane + 32 * half;
            dov[half] = 0.f;
            if (v >= dv) continue;
            float o = 0.f;
            for (int j = 0; j < r; ++j) o = fmaf(vec[j], ld(wuv + v * r + j), o);
            const float dout = ld(p.dout + row * dv + v);
            if (p.gate) {
                const float sg = 1.f / (1.f + expf(-ld(p.gate + row * dv + v)));
                p.dgate[row * dv + v] = dout * o * sg * (1.f - sg);
                dov[half] = dout * sg;
            } else {
                dov[half] = dout;
            }
        }
        __syncwarp();
        vec[lane] = dov[0];
        vec[lane + 32] = dov[1];
        __syncwarp();
        // do_lat_j = sum_v do_v W_UV[h, v, j]; dW_UV[v, j] += do_v o_lat_j
        float dl0 = 0.f, dl1 = 0.f;
        for (int v = 0; v < dv; ++v) {
            const float dv_ = vec[v];
            if (lane < r) {
                dl0 = fmaf(dv_, ld(wuv + v * r + lane), dl0);
                atomicAdd(s_dwuv + v * kMaxDim + lane, dv_ * ol[i][0]);
            }
            if (lane + 32 < r) {
                dl1 = fmaf(dv_, ld(wuv + v * r + lane + 32), dl1);
                atomicAdd(s_dwuv + v * kMaxDim + lane + 32, dv_ * ol[i][1]);
            }
        }
        float *dol = s_dol + (warp * kPerWarp + i) * kMaxDim;
        dol[lane] = dl0;
        dol[lane + 32] = dl1;
        delta[i] = warp_sum(dl0 * ol[i][0] + dl1 * ol[i][1]);
        // for the key kernel: q_abs, do_lat and (m, l, delta) of this row
        const float *qa = s_qa + (warp * kPerWarp + i) * kMaxDim;
        if (lane < r) {
            p.ws_qa[row * r + lane] = qa[lane];
            p.ws_dol[row * r + lane] = dl0;
        }
        if (lane + 32 < r) {
            p.ws_qa[row * r + lane + 32] = qa[lane + 32];
            p.ws_dol[row * r + lane + 32] = dl1;
        }
        if (lane == 0) {
            p.ws_st[row * 4 + 0] = m[i];
            p.ws_st[row * 4 + 1] = l[i];
            p.ws_st[row * 4 + 2] = delta[i];
            p.ws_st[row * 4 + 3] = 0.f;
        }
        __syncwarp();
    }

    // pass 2: dq_abs = scale sum_u ds_tu c_u with ds_tu = a_tu (do_lat_t . c_u - delta_t)
    for (int k0 = 0; k0 < last_key; k0 += kChunk) {
        stage(k0);
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int t = t0 + i * kWarps + warp;
            if (t >= T || k0 > t) continue;   // warp-uniform
            const int n_vis = min(kChunk, t - k0 + 1);
            float ds = 0.f;
            if (lane < n_vis) {
                const float a = expf(score(s_qa + (warp * kPerWarp + i) * kMaxDim, lane) * p.scale - m[i]) / l[i];
                const float da = score(s_dol + (warp * kPerWarp + i) * kMaxDim, lane);
                ds = a * (da - delta[i]);
            }
            pw[lane] = ds;
            __syncwarp();
            float a0 = 0.f, a1 = 0.f;
            for (int u = 0; u < n_vis; ++u) {
                a0 = fmaf(pw[u], s_c[u * kPad + lane], a0);
                a1 = fmaf(pw[u], s_c[u * kPad + lane + 32], a1);
            }
            dqa[i][0] = fmaf(p.scale, a0, dqa[i][0]);
            dqa[i][1] = fmaf(p.scale, a1, dqa[i][1]);
            __syncwarp();
        }
    }

    // absorb backward: dq = dq_abs W_UK^T, dW_UK[d, j] += q_d dq_abs_j
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int t = t0 + i * kWarps + warp;
        if (t >= T) continue;
        const size_t row = (static_cast<size_t>(b) * T + t) * H + h;
        vec[lane] = dqa[i][0];
        vec[lane + 32] = dqa[i][1];
        __syncwarp();
        const In *qrow = p.q + row * dq_dim;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int d = lane + 32 * half;
            if (d >= dq_dim) continue;
            float acc = 0.f;
            for (int j = 0; j < r; ++j) acc = fmaf(vec[j], ld(wuk + d * r + j), acc);
            p.dq[row * dq_dim + d] = acc;
        }
        for (int d = 0; d < dq_dim; ++d) {
            const float qd = ld(qrow + d);
            if (lane < r) atomicAdd(s_dwuk + d * kMaxDim + lane, qd * dqa[i][0]);
            if (lane + 32 < r) atomicAdd(s_dwuk + d * kMaxDim + lane + 32, qd * dqa[i][1]);
        }
        __syncwarp();
    }

    // this CTA's parts of dW_UK[h] and dW_UV[h]
    __syncthreads();
    for (int i = threadIdx.x; i < dq_dim * r; i += kWarps * 32) {
        const int d = i / r, j = i - d * r;
        atomicAdd(p.dw_uk + static_cast<size_t>(h) * dq_dim * r + i, s_dwuk[d * kMaxDim + j]);
    }
    for (int i = threadIdx.x; i < dv * r; i += kWarps * 32) {
        const int v = i / r, j = i - v * r;
        atomicAdd(p.dw_uv + static_cast<size_t>(h) * dv * r + i, s_dwuv[v * kMaxDim + j]);
    }
}

// Shared memory of the key kernel, in floats.
constexpr int kKC = 0;                                   // [kRows][kPad] this CTA's keys' latents
constexpr int kKQa = kKC + kRows * kPad;                 // [kChunk][kPad] staged q_abs
constexpr int kKDol = kKQa + kChunk * kPad;              // [kChunk][kPad] staged do_lat
constexpr int kKSt = kKDol + kChunk * kPad;              // [kChunk][4] staged (m, l, delta, 0)
constexpr int kKA = kKSt + kChunk * 4;                   // [kWarps][kChunk] a_tu
constexpr int kKDs = kKA + kWarps * kChunk;              // [kWarps][kChunk] scale ds_tu
constexpr int kKFloats = kKDs + kWarps * kChunk;
constexpr size_t kKSmem = kKFloats * sizeof(float);

template <typename In>
__global__ void __launch_bounds__(kWarps * 32) bwd_key_kernel(const BwdParams<In> p) {
    extern __shared__ float sm[];
    float *s_ck = sm + kKC, *s_qa = sm + kKQa, *s_dol = sm + kKDol, *s_st = sm + kKSt;
    const int T = p.T, H = p.H, r = p.r;
    const int k0 = static_cast<int>(blockIdx.x) * kRows;   // this CTA's keys [k0, k0 + 16)
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *pa = sm + kKA + warp * kChunk, *pds = sm + kKDs + warp * kChunk;
    const In *cb = p.c + static_cast<size_t>(b) * T * r;
    for (int i = threadIdx.x; i < kRows * r; i += kWarps * 32) {
        const int u = i / r, j = i - u * r;
        s_ck[u * kPad + j] = k0 + u < T ? ld(cb + static_cast<size_t>(k0 + u) * r + j) : 0.f;
    }
    float acc[kPerWarp][2] = {};
    for (int tq0 = (k0 / kChunk) * kChunk; tq0 < T; tq0 += kChunk) {   // queries t >= k0, 32 at a time
        __syncthreads();
        for (int i = threadIdx.x; i < kChunk * r; i += kWarps * 32) {
            const int tl = i / r, j = i - tl * r;
            const bool in = tq0 + tl < T;
            const size_t row = (static_cast<size_t>(b) * T + tq0 + tl) * H + h;
            s_qa[tl * kPad + j] = in ? p.ws_qa[row * r + j] : 0.f;
            s_dol[tl * kPad + j] = in ? p.ws_dol[row * r + j] : 0.f;
        }
        for (int i = threadIdx.x; i < kChunk * 4; i += kWarps * 32) {
            const int tl = i >> 2;
            const size_t row = (static_cast<size_t>(b) * T + tq0 + tl) * H + h;
            s_st[i] = tq0 + tl < T ? p.ws_st[row * 4 + (i & 3)] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int ul = i * kWarps + warp, u = k0 + ul;
            if (u >= T) continue;   // warp-uniform
            const int t = tq0 + lane;
            float a = 0.f, ds = 0.f;
            if (t < T && t >= u) {   // query t sees key u
                const float *cu = s_ck + ul * kPad, *qa = s_qa + lane * kPad, *dl = s_dol + lane * kPad;
                float s0 = 0.f, s1 = 0.f;
                for (int j = 0; j < r; ++j) {
                    s0 = fmaf(qa[j], cu[j], s0);
                    s1 = fmaf(dl[j], cu[j], s1);
                }
                a = expf(s0 * p.scale - s_st[lane * 4 + 0]) / s_st[lane * 4 + 1];
                ds = p.scale * a * (s1 - s_st[lane * 4 + 2]);
            }
            pa[lane] = a;
            pds[lane] = ds;
            __syncwarp();
            float a0 = 0.f, a1 = 0.f;
            for (int tl = 0; tl < kChunk; ++tl) {
                const float w = pa[tl], wd = pds[tl];
                a0 = fmaf(w, s_dol[tl * kPad + lane], fmaf(wd, s_qa[tl * kPad + lane], a0));
                a1 = fmaf(w, s_dol[tl * kPad + lane + 32], fmaf(wd, s_qa[tl * kPad + lane + 32], a1));
            }
            acc[i][0] += a0;
            acc[i][1] += a1;
            __syncwarp();
        }
    }
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int u = k0 + i * kWarps + warp;
        if (u >= T) continue;
        float *dcu = p.dc + (static_cast<size_t>(b) * T + u) * r;
        if (lane < r) atomicAdd(dcu + lane, acc[i][0]);
        if (lane + 32 < r) atomicAdd(dcu + lane + 32, acc[i][1]);
    }
}

}  // namespace

bool backward_f32_supports(int r, int d_q, int d_v) {
    return r >= 1 && r <= kMaxDim && d_q >= 1 && d_q <= kMaxDim && d_v >= 1 && d_v <= kMaxDim;
}

size_t backward_f32_workspace_bytes(long long B, long long T, long long H, int r) {
    return static_cast<size_t>(B * T * H) * (2 * static_cast<size_t>(r) + 4) * sizeof(float);
}

template <typename In>
static cudaError_t launch_typed(const BackwardArgs &a, cudaStream_t s) {
    BwdParams<In> p;
    p.q = static_cast<const In *>(a.q);
    p.c = static_cast<const In *>(a.c);
    p.w_uk = static_cast<const In *>(a.w_uk);
    p.w_uv = static_cast<const In *>(a.w_uv);
    p.gate = static_cast<const In *>(a.gate);
    p.dout = static_cast<const In *>(a.dout);
    p.dq = static_cast<float *>(a.dq);
    p.dc = static_cast<float *>(a.dc);
    p.dw_uk = static_cast<float *>(a.dw_uk);
    p.dw_uv = static_cast<float *>(a.dw_uv);
    p.dgate = static_cast<float *>(a.dgate);
    const size_t rows = static_cast<size_t>(a.B) * a.T * a.H;
    p.ws_qa = static_cast<float *>(a.workspace);
    p.ws_dol = p.ws_qa + rows * a.r;
    p.ws_st = p.ws_dol + rows * a.r;
    p.scale = a.scale;
    p.B = a.B;
    p.T = a.T;
    p.H = a.H;
    p.d_q = a.d_q;
    p.d_v = a.d_v;
    p.r = a.r;
    // sums over CTAs start from zero
    cudaError_t e;
    if ((e = cudaMemsetAsync(a.dc, 0, static_cast<size_t>(a.B) * a.T * a.r * sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dw_uk, 0, static_cast<size_t>(a.H) * a.d_q * a.r * sizeof(float), s)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(a.dw_uv, 0, static_cast<size_t>(a.H) * a.d_v * a.r * sizeof(float), s)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(bwd_query_kernel<In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kQSmem))) != cudaSuccess)
        return e;
    const unsigned tiles = static_cast<unsigned>((a.T + kRows - 1) / kRows);
    note_launch();
    bwd_query_kernel<In><<<dim3(tiles, a.H, a.B), kWarps * 32, kQSmem, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
    bwd_key_kernel<In><<<dim3(tiles, a.H, a.B), kWarps * 32, kKSmem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_backward_f32(const BackwardArgs &a, cudaStream_t s) {
    if (!backward_f32_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    return a.bf16 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace mla
