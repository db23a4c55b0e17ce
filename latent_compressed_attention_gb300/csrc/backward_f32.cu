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
// Two kernels, each a register-tiled SIMT loop over 64 x 32 blocks of (query, key) pairs:
//   query kernel: one CTA per (b, h, 64 query rows).  Pass 1 recomputes q_abs, the softmax statistics
//     and o_lat over the keys u <= t (32 keys staged at a time); the per-row epilogue forms o, dgate, do,
//     do_lat, delta and this CTA's part of dW_UV.  Pass 2 walks the keys again for dq_abs, and the
//     epilogue forms dq and this CTA's part of dW_UK.  q_abs, do_lat and (m, 1/l, delta) go to the
//     workspace for the key kernel.
//   key kernel: one CTA per (b, h, 64 keys).  For the queries t >= u (32 staged at a time) it recomputes
//     a_tu and ds_tu and accumulates this head's part of dc_u = sum_t a_tu do_lat_t + scale ds_tu q_abs_t.
// A CTA is 128 threads.  Each thread owns a 4 x 4 block of pairs (4 rows of the CTA's 64, 4 of the
// chunk's 32) for the score products and a 4 x (RP/8) block of the [64, RP] accumulator; both operands of
// a step are 128-bit loads of transposed shared buffers, so two loads feed 16 FMAs.  The chunk after the
// current one is loaded into registers while the current one is in use, and stored into the other of two
// buffers, one barrier per chunk.  RP is r rounded up to 16, 32 or 64; the padding columns are zero.  dc, dW_UK and dW_UV are sums over blocks, so they are zeroed first and added with atomics; dq
// and dgate are written once (no atomics).
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kMaxDim = 64;          // r, d_q, d_v limit
constexpr int kTile = 64;            // query rows (query kernel) or keys (key kernel) per CTA
constexpr int kChunk = 32;           // keys (query kernel) or queries (key kernel) staged per step
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTP = kTile + 4;       // row of a transposed [., kTile] buffer, padded (16-byte multiple)
constexpr int kCP = kChunk + 4;      // row of a transposed [., kChunk] buffer, padded (16-byte multiple)

template <typename In>
struct BwdParams {
    const In *q, *c, *w_uk, *w_uv, *gate, *dout;
    float *dq, *dc, *dw_uk, *dw_uv, *dgate;
    float *ws_qa, *ws_dol, *ws_st;   // [B,H,T,r], [B,H,T,r], [B,H,T,4] = (m, 1 / l, delta, 0)
    float scale;
    float scale_log2;                // scale log2(e): the scores in base 2, m in the same units
    int B, T, H, d_q, d_v, r;
};

__device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }

// max / sum over the 8 lanes that share a row block (lane bits 0-2)
__device__ __forceinline__ float oct_max(float v) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float oct_sum(float v) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Offset of rows 4 ty .. 4 ty + 3 of row u in a [kChunk][kTile] weight buffer.  The 16-byte groups are
// swizzled (group ty ^ ((u >> 2) & 7)), so the eight threads that store one row group for keys
// 4 tx .. 4 tx + 3 (tx = 0..7) and the warp that reads four row groups of one key both hit distinct banks.
__device__ __forceinline__ int wsw(int u, int ty) { return u * kTile + 4 * (ty ^ ((u >> 2) & 7)); }
__device__ __forceinline__ void st4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// NC consecutive floats of a shared row (NC = 1, 2, 4 or 8; the address is min(NC, 4)-float aligned)
template <int NC>
__device__ __forceinline__ void ldn(const float *p, float (&v)[NC]) {
    if constexpr (NC == 8) {
        const float4 t = ld4(p), u = ld4(p + 4);
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w, v[4] = u.x, v[5] = u.y, v[6] = u.z, v[7] = u.w;
    } else if constexpr (NC == 4) {
        const float4 t = ld4(p);
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    } else if constexpr (NC == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x, v[1] = t.y;
    } else {
        v[0] = *p;
    }
}

// Shared memory of the query kernel, in floats (every float4-read buffer starts on a 4-float boundary).
struct QLayout {
    int qaT, dolT, c, pT, ol, cT, wuk, wuv, q, dO, st, total;
    __host__ __device__ QLayout(int RP, int dq, int dv) {
        int o = 0;
        qaT = o, o += RP * kTP;             // [RP][kTP]  q_abs, transposed
        dolT = o, o += RP * kTP;            // [RP][kTP]  do_lat, transposed
        c = o, o += 2 * kChunk * (RP + 4);  // 2 x [kChunk][RP + 4]  staged latent rows (double-buffered)
        ol = c;                             // [kTile][RP + 4]  o_lat, later dq_abs: the same memory, used
                                            //   only between the passes and after pass 2
        pT = o, o += kChunk * kTile;        // [kChunk][kTile]  p (pass 1) or scale ds (pass 2), swizzled
        cT = o, o += 2 * RP * kCP;          // 2 x [RP][kCP]  staged latent rows, transposed
        wuk = o, o += dq * (RP + 1);        // [d_q][RP + 1]  W_UK[h], zero-padded
        wuv = o, o += dv * (RP + 1);        // [d_v][RP + 1]  W_UV[h], zero-padded
        q = o, o += kTile * (dq + 1);       // [kTile][d_q + 1]  the tile's q rows
        if (kTile * (dv + 1) <= kChunk * kTile) {
            dO = pT;                        // [kTile][d_v + 1]  do: only between the passes, when pT is idle
        } else {
            dO = o, o += kTile * (dv + 1);
        }
        st = o, o += 3 * kTile;             // m, l, delta of each row
        total = o;
    }
};

// Shared memory of the key kernel, in floats.
struct KLayout {
    int ckT, qa, dol, aT, dsT, qaT, dolT, st, total;
    __host__ __device__ explicit KLayout(int RP) {
        int o = 0;
        ckT = o, o += RP * kTP;             // [RP][kTP]  this CTA's keys' latents, transposed
        qa = o, o += 2 * kChunk * (RP + 4);   // 2 x [kChunk][RP + 4]  staged q_abs rows (double-buffered)
        dol = o, o += 2 * kChunk * (RP + 4);  // 2 x [kChunk][RP + 4]  staged do_lat rows
        aT = o, o += kChunk * kTile;        // [kChunk][kTile]  a, swizzled
        dsT = o, o += kChunk * kTile;       // [kChunk][kTile]  scale ds, swizzled
        qaT = o, o += 2 * RP * kCP;         // 2 x [RP][kCP]  staged q_abs, transposed
        dolT = o, o += 2 * RP * kCP;        // 2 x [RP][kCP]  staged do_lat, transposed
        st = o, o += 2 * 3 * kChunk;        // 2 x m, 1 / l, delta of the staged queries
        total = o;
    }
};

// Rows first .. first + 31 of a [., r] source, staged through registers (loaded while the previous chunk
// is in use, stored after) into rows [kChunk][RP + 4] and rowsT [RP][kCP]; zero past T and past r.  A
// thread holds column j of 4 consecutive rows, so the loads coalesce over j, and the transposed copy is
// one 16-byte store per (column, 4 rows), conflict-free with the kCP padding.
template <typename In, int RP>
struct RowStage {
    static constexpr int kPairs = RP * (kChunk / 4) / kThreads;   // (column, 4 rows) per thread: 1, 2 or 4
    static constexpr int kRows = kChunk * (RP + 4), kRowsT = RP * kCP;   // one buffer of each layout
    float v[kPairs][4];
    __device__ __forceinline__ void load(const In *src, int first, int T, int r) {
#pragma unroll
        for (int e = 0; e < kPairs; ++e) {
            const int q = static_cast<int>(threadIdx.x) + e * kThreads, g = q / RP, j = q - g * RP;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = first + 4 * g + k;
                v[e][k] = (u < T && j < r) ? ld(src + static_cast<size_t>(u) * r + j) : 0.f;
            }
        }
    }
    __device__ __forceinline__ void store(float *rows, float *rowsT) const {
#pragma unroll
        for (int e = 0; e < kPairs; ++e) {
            const int q = static_cast<int>(threadIdx.x) + e * kThreads, g = q / RP, j = q - g * RP;
#pragma unroll
            for (int k = 0; k < 4; ++k) rows[(4 * g + k) * (RP + 4) + j] = v[e][k];
            st4(rowsT + j * kCP + 4 * g, v[e][0], v[e][1], v[e][2], v[e][3]);
        }
    }
};

// s[i][k] += a_i b_k
__device__ __forceinline__ void outer4(float (&s)[4][4], const float4 &a, const float4 &b) {
    const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) s[i][k] = fmaf(av[i], bv[k], s[i][k]);
}

// s[i][k] += sum_j aT[j][4 ty + i] bT[j][4 tx + k]
template <int RP>
__device__ __forceinline__ void dot_4x4(const float *aT, const float *bT, int ty, int tx, float (&s)[4][4]) {
#pragma unroll 8
    for (int j = 0; j < RP; ++j) outer4(s, ld4(aT + j * kTP + 4 * ty), ld4(bT + j * kCP + 4 * tx));
}

// the same for two row operands sharing bT: s += aT . bT, e += eT . bT
template <int RP>
__device__ __forceinline__ void dot2_4x4(const float *aT, const float *eT, const float *bT, int ty, int tx,
                                         float (&s)[4][4], float (&e)[4][4]) {
#pragma unroll 4
    for (int j = 0; j < RP; ++j) {
        const float4 b = ld4(bT + j * kCP + 4 * tx);
        outer4(s, ld4(aT + j * kTP + 4 * ty), b);
        outer4(e, ld4(eT + j * kTP + 4 * ty), b);
    }
}

// and for one row operand against two column operands: s += aT . bT, e += aT . fT
template <int RP>
__device__ __forceinline__ void dot_4x4x2(const float *aT, const float *bT, const float *fT, int ty, int tx,
                                          float (&s)[4][4], float (&e)[4][4]) {
#pragma unroll 4
    for (int j = 0; j < RP; ++j) {
        const float4 a = ld4(aT + j * kTP + 4 * ty);
        outer4(s, a, ld4(bT + j * kCP + 4 * tx));
        outer4(e, a, ld4(fT + j * kCP + 4 * tx));
    }
}

// acc[i][c] += sum_u pT[u][4 ty + i] rows[u][tx NC + c]
template <int RP>
__device__ __forceinline__ void acc_4xn(const float *pT, const float *rows, int ty, int tx,
                                        float (&acc)[4][RP / 8]) {
    constexpr int NC = RP / 8;
#pragma unroll 8
    for (int u = 0; u < kChunk; ++u) {
        const float4 w = ld4(pT + wsw(u, ty));
        float v[NC];
        ldn<NC>(rows + u * (RP + 4) + tx * NC, v);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            acc[0][c] = fmaf(w.x, v[c], acc[0][c]);
            acc[1][c] = fmaf(w.y, v[c], acc[1][c]);
            acc[2][c] = fmaf(w.z, v[c], acc[2][c]);
            acc[3][c] = fmaf(w.w, v[c], acc[3][c]);
        }
    }
}

// acc += pT . rows + qT . rows2
template <int RP>
__device__ __forceinline__ void acc2_4xn(const float *pT, const float *rows, const float *qT, const float *rows2,
                                         int ty, int tx, float (&acc)[4][RP / 8]) {
    constexpr int NC = RP / 8;
#pragma unroll 4
    for (int u = 0; u < kChunk; ++u) {
        const float4 w = ld4(pT + wsw(u, ty)), x = ld4(qT + wsw(u, ty));
        float v[NC], y[NC];
        ldn<NC>(rows + u * (RP + 4) + tx * NC, v);
        ldn<NC>(rows2 + u * (RP + 4) + tx * NC, y);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            acc[0][c] = fmaf(w.x, v[c], fmaf(x.x, y[c], acc[0][c]));
            acc[1][c] = fmaf(w.y, v[c], fmaf(x.y, y[c], acc[1][c]));
            acc[2][c] = fmaf(w.z, v[c], fmaf(x.z, y[c], acc[2][c]));
            acc[3][c] = fmaf(w.w, v[c], fmaf(x.w, y[c], acc[3][c]));
        }
    }
}

template <typename In, int RP>
__global__ void __launch_bounds__(kThreads, RP <= 32 ? 4 : 3) bwd_query_kernel(const BwdParams<In> p) {
    constexpr int NC = RP / 8;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int T = p.T, H = p.H, r = p.r, dqd = p.d_q, dvd = p.d_v;
    const QLayout L(RP, dqd, dvd);
    float *s_qaT = sm + L.qaT, *s_dolT = sm + L.dolT, *s_c = sm + L.c, *s_pT = sm + L.pT, *s_ol = sm + L.ol;
    float *s_cT = sm + L.cT, *s_wuk = sm + L.wuk, *s_wuv = sm + L.wuv, *s_q = sm + L.q, *s_do = sm + L.dO;
    float *s_m = sm + L.st, *s_l = s_m + kTile, *s_dl = s_l + kTile;
    const int n_tiles = (T + kTile - 1) / kTile;
    const int tile = n_tiles - 1 - static_cast<int>(blockIdx.y);   // heaviest first, over all heads
    const int b = static_cast<int>(blockIdx.x) / p.H, h = static_cast<int>(blockIdx.x) % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tx = tid & 7, ty = tid >> 3;   // rows 4 ty .. 4 ty + 3; a warp owns rows 16 warp .. 16 warp + 15
    const int t0 = tile * kTile;
    const In *wuk = p.w_uk + static_cast<size_t>(h) * dqd * r;
    const In *wuv = p.w_uv + static_cast<size_t>(h) * dvd * r;
    const In *cb = p.c + static_cast<size_t>(b) * T * r;
    auto grow = [&](int t) { return (static_cast<size_t>(b) * T + t) * H + h; };   // row of q, dq, gate, dout

    // W_UK[h] and W_UV[h] (zero past r) and the tile's q rows (zero past T)
    for (int i = tid; i < dqd * RP; i += kThreads) {
        const int d = i / RP, j = i - d * RP;
        s_wuk[d * (RP + 1) + j] = j < r ? ld(wuk + d * r + j) : 0.f;
    }
    for (int i = tid; i < dvd * RP; i += kThreads) {
        const int v = i / RP, j = i - v * RP;
        s_wuv[v * (RP + 1) + j] = j < r ? ld(wuv + v * r + j) : 0.f;
    }
    for (int i = tid; i < kTile * dqd; i += kThreads) {
        const int row = i / dqd, d = i - row * dqd;
        s_q[row * (dqd + 1) + d] = t0 + row < T ? ld(p.q + grow(t0 + row) * dqd + d) : 0.f;
    }
    __syncthreads();
    // step 2 absorb: q_abs[row, j] = sum_d q[row, d] W_UK[d, j], kept transposed
    for (int i = tid; i < RP * kTile; i += kThreads) {
        const int j = i / kTile, row = i - j * kTile;
        float acc = 0.f;
        for (int d = 0; d < dqd; ++d) acc = fmaf(s_q[row * (dqd + 1) + d], s_wuk[d * (RP + 1) + j], acc);
        s_qaT[j * kTP + row] = acc;
    }

    // pass 1: the softmax statistics and o_lat (the forward, recomputed)
    float m[4], l[4], o[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) o[i][c] = 0.f;
    }
    using Stage = RowStage<In, RP>;
    const int n_chunks = (min(T, t0 + kTile) + kChunk - 1) / kChunk;   // keys this CTA needs: [0, t0 + 64)
    Stage stg;
    stg.load(cb, 0, T, r);
    stg.store(s_c, s_cT);
    __syncthreads();   // chunk 0 and q_abs are written
    for (int ck = 0; ck < n_chunks; ++ck) {
        const int k0 = ck * kChunk;
        const float *c_ = s_c + (ck & 1) * Stage::kRows, *cT_ = s_cT + (ck & 1) * Stage::kRowsT;
        if (ck + 1 < n_chunks) stg.load(cb, k0 + kChunk, T, r);
        float s[4][4] = {};
        dot_4x4<RP>(s_qaT, cT_, ty, tx, s);
        float corr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = min(t0 + 4 * ty + i, T - 1);   // rows past T take row T - 1's mask (never stored)
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[i][k] = k0 + 4 * tx + k <= t ? s[i][k] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[i][k]);
            }
            const float m_new = fmaxf(m[i], oct_max(mx));   // finite: key 0 is in chunk 0
            corr[i] = exp2f(m[i] - m_new);   // 0 on the first chunk
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) sum += (s[i][k] = exp2f(s[i][k] - m_new));   // s now holds p
            l[i] = fmaf(l[i], corr[i], oct_sum(sum));
            m[i] = m_new;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) st4(s_pT + wsw(4 * tx + k, ty), s[0][k], s[1][k], s[2][k], s[3][k]);
        __syncwarp();   // a warp reads only its own rows' weights
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < NC; ++c) o[i][c] *= corr[i];
        acc_4xn<RP>(s_pT, c_, ty, tx, o);
        if (ck + 1 < n_chunks) stg.store(s_c + ((ck + 1) & 1) * Stage::kRows, s_cT + ((ck + 1) & 1) * Stage::kRowsT);
        __syncthreads();   // the next chunk is written; this chunk's buffers and weights are consumed
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // o_lat = o / l, row-major; the statistics
        const int row = 4 * ty + i;
        const float inv = 1.f / l[i];
#pragma unroll
        for (int c = 0; c < NC; ++c) s_ol[row * (RP + 4) + tx * NC + c] = o[i][c] * inv;
        if (tx == 0) s_m[row] = m[i], s_l[row] = l[i];
    }
    __syncthreads();

    // steps 4 and 3 backward, per row: o, dgate and do
    for (int i = tid; i < kTile * dvd; i += kThreads) {
        const int row = i / dvd, v = i - row * dvd, t = t0 + row;
        float d = 0.f;
        if (t < T) {
            float o_ = 0.f;
            for (int j = 0; j < RP; ++j) o_ = fmaf(s_ol[row * (RP + 4) + j], s_wuv[v * (RP + 1) + j], o_);
            const size_t gi = grow(t) * dvd + v;
            const float dout = ld(p.dout + gi);
            if (p.gate) {
                const float sg = 1.f / (1.f + expf(-ld(p.gate + gi)));
                p.dgate[gi] = dout * o_ * sg * (1.f - sg);
                d = dout * sg;
            } else {
                d = dout;
            }
        }
        s_do[row * (dvd + 1) + v] = d;
    }
    __syncthreads();
    // do_lat[row, j] = sum_v do[row, v] W_UV[v, j] (kept transposed); dW_UV[v, j] += sum_row do[row, v] o_lat[row, j]
    for (int i = tid; i < RP * kTile; i += kThreads) {
        const int j = i / kTile, row = i - j * kTile;
        float acc = 0.f;
        for (int v = 0; v < dvd; ++v) acc = fmaf(s_do[row * (dvd + 1) + v], s_wuv[v * (RP + 1) + j], acc);
        s_dolT[j * kTP + row] = acc;
    }
    for (int i = tid; i < dvd * r; i += kThreads) {
        const int v = i / r, j = i - v * r;
        float acc = 0.f;
        for (int row = 0; row < kTile; ++row) acc = fmaf(s_do[row * (dvd + 1) + v], s_ol[row * (RP + 4) + j], acc);
        atomicAdd(p.dw_uv + static_cast<size_t>(h) * dvd * r + i, acc);
    }
    __syncthreads();
    // delta_t = do_lat_t . o_lat_t
    for (int rr = 0; rr < kTile / kWarps; ++rr) {
        const int row = warp * (kTile / kWarps) + rr;
        float acc = 0.f;
        for (int j = lane; j < RP; j += 32) acc = fmaf(s_dolT[j * kTP + row], s_ol[row * (RP + 4) + j], acc);
        acc = warp_sum(acc);
        if (lane == 0) s_dl[row] = acc;
    }
    __syncthreads();
    // q_abs, do_lat and (m, 1 / l, delta) of the tile's rows, for the key kernel (m in base-2 units)
    const size_t ws_row0 = (static_cast<size_t>(b) * H + h) * T + t0;
    for (int i = tid; i < kTile * r; i += kThreads) {
        const int row = i / r, j = i - row * r;
        if (t0 + row < T) {
            p.ws_qa[(ws_row0 + row) * r + j] = s_qaT[j * kTP + row];
            p.ws_dol[(ws_row0 + row) * r + j] = s_dolT[j * kTP + row];
        }
    }
    if (tid < kTile && t0 + tid < T) {
        float *st = p.ws_st + (ws_row0 + tid) * 4;
        st[0] = s_m[tid], st[1] = 1.f / s_l[tid], st[2] = s_dl[tid], st[3] = 0.f;
    }

    // pass 2: dq_abs = scale sum_u ds_tu c_u with ds_tu = a_tu (do_lat_t . c_u - delta_t)
    float dqa[4][NC], mr[4], linv[4], dr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 4 * ty + i;
        mr[i] = s_m[row], linv[i] = 1.f / s_l[row], dr[i] = s_dl[row];
#pragma unroll
        for (int c = 0; c < NC; ++c) dqa[i][c] = 0.f;
    }
    stg.load(cb, 0, T, r);
    stg.store(s_c, s_cT);   // pass 1's last reads of both buffers ended before the epilogue's barriers
    __syncthreads();
    for (int ck = 0; ck < n_chunks; ++ck) {
        const int k0 = ck * kChunk;
        const float *c_ = s_c + (ck & 1) * Stage::kRows, *cT_ = s_cT + (ck & 1) * Stage::kRowsT;
        if (ck + 1 < n_chunks) stg.load(cb, k0 + kChunk, T, r);
        float s[4][4] = {}, da[4][4] = {};
        dot2_4x4<RP>(s_qaT, s_dolT, cT_, ty, tx, s, da);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = min(t0 + 4 * ty + i, T - 1);
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // s becomes scale ds
                const float a = exp2f(s[i][k] * p.scale_log2 - mr[i]) * linv[i];
                s[i][k] = k0 + 4 * tx + k <= t ? p.scale * a * (da[i][k] - dr[i]) : 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) st4(s_pT + wsw(4 * tx + k, ty), s[0][k], s[1][k], s[2][k], s[3][k]);
        __syncwarp();
        acc_4xn<RP>(s_pT, c_, ty, tx, dqa);
        if (ck + 1 < n_chunks) stg.store(s_c + ((ck + 1) & 1) * Stage::kRows, s_cT + ((ck + 1) & 1) * Stage::kRowsT);
        __syncthreads();
    }
    // dq_abs into the o_lat buffer (last read before the pass-2 barriers)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) s_ol[(4 * ty + i) * (RP + 4) + tx * NC + c] = dqa[i][c];
    __syncthreads();
    // absorb backward: dq[row, d] = sum_j dq_abs[row, j] W_UK[d, j]; dW_UK[d, j] += sum_row q[row, d] dq_abs[row, j]
    for (int i = tid; i < kTile * dqd; i += kThreads) {
        const int row = i / dqd, d = i - row * dqd, t = t0 + row;
        if (t >= T) continue;
        float acc = 0.f;
        for (int j = 0; j < RP; ++j) acc = fmaf(s_ol[row * (RP + 4) + j], s_wuk[d * (RP + 1) + j], acc);
        p.dq[grow(t) * dqd + d] = acc;
    }
    for (int i = tid; i < dqd * r; i += kThreads) {
        const int d = i / r, j = i - d * r;
        float acc = 0.f;
        for (int row = 0; row < kTile; ++row) acc = fmaf(s_q[row * (dqd + 1) + d], s_ol[row * (RP + 4) + j], acc);
        atomicAdd(p.dw_uk + static_cast<size_t>(h) * dqd * r + i, acc);
    }
}

template <typename In, int RP>
__global__ void __launch_bounds__(kThreads, 3) bwd_key_kernel(const BwdParams<In> p) {
    constexpr int NC = RP / 8;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const KLayout L(RP);
    float *s_ckT = sm + L.ckT, *s_qa = sm + L.qa, *s_dol = sm + L.dol, *s_aT = sm + L.aT, *s_dsT = sm + L.dsT;
    float *s_qaT = sm + L.qaT, *s_dolT = sm + L.dolT, *s_st = sm + L.st;   // s_st: 2 x (m, 1 / l, delta) x kChunk
    const int T = p.T, H = p.H, r = p.r;
    const int u0 = static_cast<int>(blockIdx.y) * kTile;   // keys [u0, u0 + 64); the first tiles are the heaviest
    const int b = static_cast<int>(blockIdx.x) / p.H, h = static_cast<int>(blockIdx.x) % p.H;
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;   // keys u0 + 4 ty .. + 3; a warp owns 16 consecutive keys
    const In *cb = p.c + static_cast<size_t>(b) * T * r;
    const size_t ws0 = (static_cast<size_t>(b) * H + h) * T;   // workspace row of (b, h, token 0)
    for (int i = tid; i < kTile * RP; i += kThreads) {
        const int ul = i / RP, j = i - ul * RP;
        s_ckT[j * kTP + ul] = (u0 + ul < T && j < r) ? ld(cb + static_cast<size_t>(u0 + ul) * r + j) : 0.f;
    }
    float acc[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
    // the queries t >= u0, 32 at a time, staged through registers into two alternating buffers
    using Stage = RowStage<float, RP>;
    const float *qa_g = p.ws_qa + ws0 * r, *dol_g = p.ws_dol + ws0 * r;
    Stage sq, sd;
    float st3[3];
    auto load = [&](int tq0) {
        sq.load(qa_g, tq0, T, r);
        sd.load(dol_g, tq0, T, r);
        if (tid < kChunk) {
            st3[0] = 0.f, st3[1] = 1.f, st3[2] = 0.f;   // (m, 1 / l, delta) past T: never used
            if (tq0 + tid < T) {
                const float *st = p.ws_st + (ws0 + tq0 + tid) * 4;
                st3[0] = st[0], st3[1] = st[1], st3[2] = st[2];
            }
        }
    };
    auto store = [&](int buf) {
        sq.store(s_qa + buf * Stage::kRows, s_qaT + buf * Stage::kRowsT);
        sd.store(s_dol + buf * Stage::kRows, s_dolT + buf * Stage::kRowsT);
        if (tid < kChunk)
            for (int e = 0; e < 3; ++e) s_st[(buf * 3 + e) * kChunk + tid] = st3[e];
    };
    load(u0);
    store(0);
    __syncthreads();   // chunk 0 and this CTA's keys are written
    for (int ci = 0, tq0 = u0; tq0 < T; ++ci, tq0 += kChunk) {
        const int buf = ci & 1;
        const bool more = tq0 + kChunk < T;
        if (more) load(tq0 + kChunk);
        const float *qa_ = s_qa + buf * Stage::kRows, *dol_ = s_dol + buf * Stage::kRows;
        const float *sm_ = s_st + buf * 3 * kChunk;
        float s[4][4] = {}, da[4][4] = {};   // [key][query]
        dot_4x4x2<RP>(s_ckT, s_qaT + buf * Stage::kRowsT, s_dolT + buf * Stage::kRowsT, ty, tx, s, da);
        const float4 mq4 = ld4(sm_ + 4 * tx), lq4 = ld4(sm_ + kChunk + 4 * tx), dq4 = ld4(sm_ + 2 * kChunk + 4 * tx);
        const float mq[4] = {mq4.x, mq4.y, mq4.z, mq4.w}, linv[4] = {lq4.x, lq4.y, lq4.z, lq4.w};
        const float dq_[4] = {dq4.x, dq4.y, dq4.z, dq4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = tq0 + 4 * tx + k;
#pragma unroll
            for (int i = 0; i < 4; ++i) {   // s becomes a, da becomes scale ds
                const bool vis = t < T && u0 + 4 * ty + i <= t;   // query t sees key u
                const float a = vis ? exp2f(s[i][k] * p.scale_log2 - mq[k]) * linv[k] : 0.f;
                da[i][k] = p.scale * a * (da[i][k] - dq_[k]);
                s[i][k] = a;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            st4(s_aT + wsw(4 * tx + k, ty), s[0][k], s[1][k], s[2][k], s[3][k]);
            st4(s_dsT + wsw(4 * tx + k, ty), da[0][k], da[1][k], da[2][k], da[3][k]);
        }
        __syncwarp();   // a warp reads only its own keys' weights
        acc2_4xn<RP>(s_aT, dol_, s_dsT, qa_, ty, tx, acc);
        if (more) store(buf ^ 1);
        __syncthreads();   // the next chunk is written; this chunk's buffers and weights are consumed
    }
    // this head's part of dc
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = u0 + 4 * ty + i;
        if (u >= T) continue;
        float *dcu = p.dc + (static_cast<size_t>(b) * T + u) * r;
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (tx * NC + c < r) atomicAdd(dcu + tx * NC + c, acc[i][c]);
    }
}

template <typename In, int RP>
cudaError_t launch_rp(const BwdParams<In> &p, cudaStream_t s) {
    const int qsm = QLayout(RP, p.d_q, p.d_v).total * static_cast<int>(sizeof(float));
    const int ksm = KLayout(RP).total * static_cast<int>(sizeof(float));
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bwd_query_kernel<In, RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, qsm)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(bwd_key_kernel<In, RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, ksm)) !=
        cudaSuccess)
        return e;
    // (b, h) is the fastest grid index and the tile rank the next, so every head's heaviest tiles start first
    const unsigned tiles = static_cast<unsigned>((p.T + kTile - 1) / kTile);
    const dim3 grid(static_cast<unsigned>(p.B) * static_cast<unsigned>(p.H), tiles);
    if (tiles > 65535u) return cudaErrorInvalidValue;
    note_launch();
    bwd_query_kernel<In, RP><<<grid, kThreads, qsm, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
    bwd_key_kernel<In, RP><<<grid, kThreads, ksm, s>>>(p);
    return cudaGetLastError();
}

template <typename In>
cudaError_t launch_typed(const BackwardArgs &a, cudaStream_t s) {
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
    p.scale_log2 = a.scale * 1.4426950408889634f;
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
    if (a.r <= 16) return launch_rp<In, 16>(p, s);
    if (a.r <= 32) return launch_rp<In, 32>(p, s);
    return launch_rp<In, 64>(p, s);
}

}  // namespace

bool backward_f32_supports(int r, int d_q, int d_v) {
    return r >= 1 && r <= kMaxDim && d_q >= 1 && d_q <= kMaxDim && d_v >= 1 && d_v <= kMaxDim;
}

size_t backward_f32_workspace_bytes(long long B, long long T, long long H, int r) {
    return static_cast<size_t>(B * T * H) * (2 * static_cast<size_t>(r) + 4) * sizeof(float);
}

cudaError_t launch_backward_f32(const BackwardArgs &a, cudaStream_t s) {
    if (!backward_f32_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    return a.bf16 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace mla
