// The whole Gated-MLA layer forward (page "Gated MLA（矩阵吸收版）", section
// "完整计算流（四步）", steps 1-4, and the listing of section "代码对照"):
//
//   step 1  c = RMSNorm(x . W_kv_down^T)                      [B,T,r]
//           q = RMSNorm(x . W_q_down^T) . W_q_up^T            [B,T,H,d_q]
//           g = x . W_gate^T                                  [B,T,H d_v]  (gate logits)
//   2-4     o = sigmoid(g) * (absorbed causal attention)      [B,T,H d_v]  (the hot path)
//   out     y = o . W_o^T                                     [B,T,D]
//
// RMSNorm has unit gain and eps 1e-6; every projection is bias-free.  kv_up's
// weight splits as a block: all heads' W_UK rows, then all heads' W_UV rows.
//
// bf16: the projections run on the tensor-core GEMM; the RMSNorm of the latent
// is fused into its GEMM's epilogue (the 512-column row fits one tile), and the
// RMSNorm of the query's low-rank projection moves past W_q_up as a row scale,
// from row sums of squares accumulated by the W_q_down GEMM.
// fp32 (the toy layer): plain SIMT kernels with fp32 FMAs (no TF32).
//
// Workspace, in this order, each part starting on a 256-byte boundary:
// q [M, H d_q], c [M, r], g [M, H d_v], o [M, H d_v] (the layer's intermediate
// results, in the input dtype), then the low-rank query [M, r_q] (input dtype),
// the row sums of squares [M] (fp32) and (bf16) the fp32 split-K scratch of the
// projections with too few row tiles to fill the GPU; M = B T.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr float kRmsEps = 1e-6f;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
    size_t q, c, g, o, yq, pre, ss, acc, end;
};

}  // namespace

size_t layer_split_plan(long long M, int D, int H, int d_q, int d_v, int r, int r_q, size_t off[kLayerGemms + 1]) {
    const int n[kLayerGemms] = {r_q, H * d_q, r, H * d_v, D};
    const int k[kLayerGemms] = {D, r_q, D, D, H * d_v};
    const int epi[kLayerGemms] = {kGemmSumSq, kGemmRowScale, kGemmRmsNorm, kGemmPlain, kGemmPlain};
    off[0] = 0;
    for (int i = 0; i < kLayerGemms; ++i) {
        GemmArgs g{};
        g.M = static_cast<int>(M);
        g.N = n[i];
        g.K = k[i];
        g.epilogue = epi[i];
        g.num_sms = 256;
        off[i + 1] = off[i] + gemm_bf16_split_bytes(g);
    }
    return off[kLayerGemms];
}

namespace {

Layout layout(long long M, int D, int H, int d_q, int d_v, int r, int r_q, size_t es) {
    Layout L;
    L.q = 0;
    L.c = L.q + align256(static_cast<size_t>(M) * H * d_q * es);
    L.g = L.c + align256(static_cast<size_t>(M) * r * es);
    L.o = L.g + align256(static_cast<size_t>(M) * H * d_v * es);
    L.yq = L.o + align256(static_cast<size_t>(M) * H * d_v * es);
    // the prefill's own workspace, sized for B = M sequences of one token: a bound for every B * T = M
    L.pre = L.yq + align256(static_cast<size_t>(M) * r_q * es);
    L.ss = L.pre + align256(prefill_workspace_bytes(M, 1, r, d_q, d_v, es == 4));
    L.acc = L.ss + align256(static_cast<size_t>(M) * sizeof(float));   // split-K scratch, right after ss
    size_t off[kLayerGemms + 1];
    L.end = L.acc + (es == 2 ? layer_split_plan(M, D, H, d_q, d_v, r, r_q, off) : 0);
    return L;
}

// ---------------------------------------------------------------- fp32 SIMT kernels
constexpr int kT = 16;    // output tile edge
constexpr int kKT = 64;   // K step: few dependent global round trips for the toy layer's short K

// C[M,N] = A[M,K] . B[N,K]^T in fp32, 16 x 16 output tiles.  Each K step stages 16 x 64 of A and of B
// in shared memory (coalesced along K); the next step's values are loaded into registers while the
// current one is used, so a call of K = 256 makes four global round trips, not sixteen.
__global__ void __launch_bounds__(kT *kT) gemm_f32_kernel(const float *A, const float *B, float *C, int M, int N,
                                                          int K) {
    constexpr int kPer = kT * kKT / (kT * kT);   // staged values of each operand per thread: 4
    __shared__ float sa[kT][kKT + 1], sb[kT][kKT + 1];
    const int tx = threadIdx.x % kT, ty = threadIdx.x / kT;
    const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
    float va[kPer], vb[kPer];
    auto load = [&](int k0) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = static_cast<int>(threadIdx.x) + e * kT * kT, row = i / kKT, k = k0 + i % kKT;
            va[e] = (m0 + row < M && k < K) ? A[static_cast<size_t>(m0 + row) * K + k] : 0.f;
            vb[e] = (n0 + row < N && k < K) ? B[static_cast<size_t>(n0 + row) * K + k] : 0.f;
        }
    };
    float acc = 0.f;
    load(0);
    for (int k0 = 0; k0 < K; k0 += kKT) {
        __syncthreads();   // the previous step's tiles are consumed
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = static_cast<int>(threadIdx.x) + e * kT * kT;
            sa[i / kKT][i % kKT] = va[e];
            sb[i / kKT][i % kKT] = vb[e];
        }
        __syncthreads();
        if (k0 + kKT < K) load(k0 + kKT);
#pragma unroll 16
        for (int k = 0; k < kKT; ++k) acc = fmaf(sa[ty][k], sb[tx][k], acc);
    }
    const int m = m0 + ty, n = n0 + tx;
    if (m < M && n < N) C[static_cast<size_t>(m) * N + n] = acc;
}

// Row-wise RMSNorm in place: z / sqrt(mean(z^2) + eps), one warp per row.
__global__ void rmsnorm_rows_f32_kernel(float *Z, int M, int N, float eps) {
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
    if (row >= M) return;
    float *z = Z + static_cast<size_t>(row) * N;
    float s = 0.f;
    for (int j = lane; j < N; j += 32) s = fmaf(z[j], z[j], s);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float inv = 1.f / sqrtf(s / N + eps);
    for (int j = lane; j < N; j += 32) z[j] *= inv;
}

cudaError_t gemm_f32(const void *A, const void *B, void *C, long long M, int N, int K, cudaStream_t s) {
    const dim3 grid((N + kT - 1) / kT, static_cast<unsigned>((M + kT - 1) / kT));
    note_launch();
    gemm_f32_kernel<<<grid, kT * kT, 0, s>>>(static_cast<const float *>(A), static_cast<const float *>(B),
                                               static_cast<float *>(C), static_cast<int>(M), N, K);
    return cudaGetLastError();
}

cudaError_t rmsnorm_f32(void *Z, long long M, int N, cudaStream_t s) {
    note_launch();
    rmsnorm_rows_f32_kernel<<<static_cast<unsigned>((M + 7) / 8), 256, 0, s>>>(static_cast<float *>(Z),
                                                                              static_cast<int>(M), N, kRmsEps);
    return cudaGetLastError();
}

}  // namespace

bool gated_layer_supports(int D, int H, int d_q, int d_v, int r, int r_q, bool f32) {
    if (D <= 0 || H <= 0 || d_q <= 0 || d_v <= 0 || r <= 0 || r_q <= 0) return false;
    if (f32) return prefill_f32_simt_supports(r, d_q, d_v);
    return prefill_bf16_r512_supports(r, d_q, d_v) && gemm_bf16_supports(r_q, D, kGemmSumSq) &&
           gemm_bf16_supports(H * d_q, r_q, kGemmRowScale) && gemm_bf16_supports(r, D, kGemmRmsNorm) &&
           gemm_bf16_supports(H * d_v, D, kGemmPlain) && gemm_bf16_supports(D, H * d_v, kGemmPlain);
}

size_t gated_layer_workspace_bytes(long long M, int D, int H, int d_q, int d_v, int r, int r_q, bool f32) {
    return layout(M, D, H, d_q, d_v, r, r_q, f32 ? 4 : 2).end;
}

cudaError_t launch_gated_layer(const LayerArgs &a, cudaStream_t s) {
    const long long M = static_cast<long long>(a.B) * a.T;
    const size_t es = a.f32 ? 4 : 2;
    const Layout L = layout(M, a.D, a.H, a.d_q, a.d_v, a.r, a.r_q, es);
    if (a.workspace_bytes < L.end) return cudaErrorInvalidValue;
    char *ws = static_cast<char *>(a.workspace);
    void *q = ws + L.q, *c = ws + L.c, *g = ws + L.g, *o = ws + L.o, *yq = ws + L.yq;
    float *ss = reinterpret_cast<float *>(ws + L.ss);
    const int Hq = a.H * a.d_q, Hv = a.H * a.d_v;
    const char *w_uv = static_cast<const char *>(a.w_kv_up) + static_cast<size_t>(Hq) * a.r * es;
    cudaError_t e;
    if (a.f32) {
        if ((e = gemm_f32(a.x, a.w_q_down, yq, M, a.r_q, a.D, s)) != cudaSuccess) return e;
        if ((e = rmsnorm_f32(yq, M, a.r_q, s)) != cudaSuccess) return e;
        if ((e = gemm_f32(yq, a.w_q_up, q, M, Hq, a.r_q, s)) != cudaSuccess) return e;
        if ((e = gemm_f32(a.x, a.w_kv_down, c, M, a.r, a.D, s)) != cudaSuccess) return e;
        if ((e = rmsnorm_f32(c, M, a.r, s)) != cudaSuccess) return e;
        if ((e = gemm_f32(a.x, a.w_gate, g, M, Hv, a.D, s)) != cudaSuccess) return e;
    } else {
        // one memset zeroes the row sums of squares and every split-K slice
        if ((e = cudaMemsetAsync(ss, 0, L.end - L.ss, s)) != cudaSuccess) return e;
        size_t off[kLayerGemms + 1];
        layer_split_plan(M, a.D, a.H, a.d_q, a.d_v, a.r, a.r_q, off);
        GemmArgs gm{};
        gm.M = static_cast<int>(M);
        gm.dev_err = a.dev_err;
        gm.num_sms = a.num_sms;
        gm.eps = kRmsEps;
        auto run = [&](int which, const void *A, long long lda, const void *B, void *C, int N, int K, int epi,
                       float n_norm) {
            gm.A = A;
            gm.lda = lda;
            gm.B = B;
            gm.ldb = K;
            gm.C = C;
            gm.ldc = N;
            gm.N = N;
            gm.K = K;
            gm.epilogue = epi;
            gm.ss = ss;
            gm.n_norm = n_norm;
            gm.split_acc = nullptr;
            const size_t need = gemm_bf16_split_bytes(gm);
            if (need != 0 && need <= off[which + 1] - off[which])
                gm.split_acc = reinterpret_cast<float *>(ws + L.acc + off[which]);
            return launch_gemm_bf16(gm, s);
        };
        if ((e = run(kQDown, a.x, a.D, a.w_q_down, yq, a.r_q, a.D, kGemmSumSq, 0.f)) != cudaSuccess) return e;
        if ((e = run(kQUp, yq, a.r_q, a.w_q_up, q, Hq, a.r_q, kGemmRowScale, static_cast<float>(a.r_q))) !=
            cudaSuccess)
            return e;
        if ((e = run(kKvDown, a.x, a.D, a.w_kv_down, c, a.r, a.D, kGemmRmsNorm, static_cast<float>(a.r))) !=
            cudaSuccess)
            return e;
        if ((e = run(kGate, a.x, a.D, a.w_gate, g, Hv, a.D, kGemmPlain, 0.f)) != cudaSuccess) return e;
    }
    PrefillArgs pa{q, c, a.w_kv_up, w_uv, g, o, a.scale, a.B, a.T, a.H, a.d_q, a.d_v, a.r, a.dev_err, a.num_sms,
                   ws + L.pre, L.ss - L.pre};
    e = a.f32 ? launch_prefill_f32_simt(pa, s) : launch_prefill_bf16_r512(pa, s);
    if (e != cudaSuccess) return e;
    if (a.f32) return gemm_f32(o, a.w_o, a.y, M, a.D, Hv, s);
    GemmArgs go{};
    go.A = o;
    go.lda = Hv;
    go.B = a.w_o;
    go.ldb = Hv;
    go.C = a.y;
    go.ldc = a.D;
    go.M = static_cast<int>(M);
    go.N = a.D;
    go.K = Hv;
    go.epilogue = kGemmPlain;
    go.dev_err = a.dev_err;
    go.num_sms = a.num_sms;
    size_t off[kLayerGemms + 1];
    layer_split_plan(M, a.D, a.H, a.d_q, a.d_v, a.r, a.r_q, off);
    const size_t need = gemm_bf16_split_bytes(go);
    if (need != 0 && need <= off[kOProj + 1] - off[kOProj])
        go.split_acc = reinterpret_cast<float *>(ws + L.acc + off[kOProj]);
    return launch_gemm_bf16(go, s);
}

}  // namespace mla
