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
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr float kRmsEps = 1e-6f;
constexpr int kAbsThreads = 128;
constexpr int kAbsCols = 256;                     // latent columns (fp32 TMEM accumulator columns) per CTA
constexpr uint32_t kAbsASlab = 128 * 128;         // [128 sequences x 64 d] bf16, 128-byte swizzle
constexpr uint32_t kAbsWBox = 64 * 128;           // [64 d x 64 latent columns] bf16
constexpr uint32_t kAbsIdesc = make_idesc_bf16(128, 256, 0, 1);   // q (K-major) x W_UK (MN-major)

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecLayout {
    size_t q, c, g, qa, o, yq, lens1, ss, acc, dec, end;
};

DecLayout dec_layout(int B, int D, int H, int d_q, int d_v, int r, int r_q, size_t dec_bytes) {
    DecLayout L;
    const size_t es = 2;
    L.q = 0;
    L.c = L.q + align256(static_cast<size_t>(B) * H * d_q * es);
    L.g = L.c + align256(static_cast<size_t>(B) * r * es);
    L.qa = L.g + align256(static_cast<size_t>(B) * H * d_v * es);
    L.o = L.qa + align256(static_cast<size_t>(B) * H * r * es);
    L.yq = L.o + align256(static_cast<size_t>(B) * H * d_v * es);
    L.lens1 = L.yq + align256(static_cast<size_t>(B) * r_q * es);
    L.ss = L.lens1 + align256(static_cast<size_t>(B) * sizeof(int));
    L.acc = L.ss + align256(static_cast<size_t>(B) * sizeof(float));   // split-K scratch, right after ss
    size_t off[kLayerGemms + 1];
    L.dec = L.acc + layer_split_plan(B, D, H, d_q, d_v, r, r_q, off);
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

// q_abs[b, h, :] = q[b, h, :] . W_UK[h] (d_q -> r) on the tensor cores, fp32
// accumulation in TMEM, bf16 out.  A CTA takes one head, up to 128 sequences
// and 256 of the latent columns (two CTAs per head at r = 512, so 192 CTAs
// share the W_UK stream): A = the sequences' q rows of that head (K-major,
// rows past B read as zeros), B = its 256 columns of W_UK[h] [d_q, r] as stored
// (latent columns contiguous, so an MN-major operand), D = [128, 256] in 256
// TMEM columns.  One thread issues every copy and product; the four warps then
// drain their 32 TMEM lanes.
__global__ void __launch_bounds__(kAbsThreads, 1)
    absorb_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w,
                        __nv_bfloat16 *q_abs, int B, int H, int d_q, int r, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int n_kh = d_q / 64, n_ns = kAbsCols / 64;
    const int nh = blockIdx.z;   // this CTA's 256 latent columns
    const uint32_t w_off = n_kh * kAbsASlab, bar_off = w_off + n_kh * n_ns * kAbsWBox;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + (base - raw) + bar_off);
    uint64_t *done = full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, b0 = blockIdx.y * 128;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(full), 1);
        mbar_init(smem_u32(done), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kAbsCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        const uint32_t bar = smem_u32(full);
        mbar_arrive_expect_tx(bar, n_kh * kAbsASlab + n_kh * n_ns * kAbsWBox);
        for (int kh = 0; kh < n_kh; ++kh) {
            tma_load_3d(base + kh * kAbsASlab, &tm_q, bar, kh * 64, h, b0);
            for (int ns = 0; ns < n_ns; ++ns)
                tma_load_3d(base + w_off + (kh * n_ns + ns) * kAbsWBox, &tm_w, bar, (nh * n_ns + ns) * 64, kh * 64,
                            h);
        }
        if (mbar_wait(bar, 0, err)) {
            tc_fence_after();
            for (int kh = 0; kh < n_kh; ++kh)
#pragma unroll
                for (int j = 0; j < 4; ++j) {   // K steps of 16 within a 64-wide slab
                    const uint64_t ad = make_smem_desc(base + kh * kAbsASlab + j * 32, 16, 1024);
                    const uint64_t bd = make_smem_desc(base + w_off + kh * n_ns * kAbsWBox + j * 2048, kAbsWBox, 1024);
                    umma_bf16(tmem, ad, bd, kAbsIdesc, (kh | j) != 0);
                }
            umma_commit(smem_u32(done));
        } else {
            *abort_flag = 1;
        }
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done), 0, err, abort_flag));
    if (ok) {   // warp-uniform: the TMEM loads below are warp-collective
        tc_fence_after();
        const int b = b0 + warp * 32 + lane;
        uint4 *dst = reinterpret_cast<uint4 *>(q_abs + (static_cast<size_t>(b < B ? b : 0) * H + h) * r + nh * kAbsCols);
#pragma unroll 1
        for (int cc = 0; cc < kAbsCols / 32; ++cc) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
            tmem_wait_ld();
            if (b < B)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    dst[cc * 4 + q4] = make_uint4(pack_bf16x2(v[8 * q4], v[8 * q4 + 1]),
                                                  pack_bf16x2(v[8 * q4 + 2], v[8 * q4 + 3]),
                                                  pack_bf16x2(v[8 * q4 + 4], v[8 * q4 + 5]),
                                                  pack_bf16x2(v[8 * q4 + 6], v[8 * q4 + 7]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kAbsCols);
}

size_t absorb_smem_bytes(int d_q, int r) {
    (void)r;   // each CTA takes 256 latent columns
    return static_cast<size_t>(d_q / 64) * (kAbsASlab + static_cast<size_t>(kAbsCols / 64) * kAbsWBox) + 64 + 1024;
}

CUresult encode_bf16_3d(CUtensorMap *m, const void *ptr, const cuuint64_t *dims, const cuuint64_t *strides,
                        const cuuint32_t *box) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool gated_layer_decode_supports(int D, int H, int d_q, int d_v, int r, int r_q) {
    return gated_layer_supports(D, H, d_q, d_v, r, r_q, false) && decode_bf16_supports(H, d_v, r) &&
           d_q % 64 == 0 && r % kAbsCols == 0 && absorb_smem_bytes(d_q, r) <= 227u * 1024;
}

size_t gated_layer_decode_workspace_bytes(int B, int D, int H, int d_q, int d_v, int r, int r_q, int max_len,
                                          int num_sms) {
    return dec_layout(B, D, H, d_q, d_v, r, r_q, decode_bf16_workspace_bytes(B, H, r, max_len, num_sms)).end;
}

cudaError_t launch_gated_layer_decode(const LayerDecodeArgs &a, cudaStream_t s) {
    const size_t dec_bytes = decode_bf16_workspace_bytes(a.B, a.H, a.r, a.max_len, a.num_sms);
    const DecLayout L = dec_layout(a.B, a.D, a.H, a.d_q, a.d_v, a.r, a.r_q, dec_bytes);
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
    // one memset zeroes the row sums of squares and every split-K slice
    if ((e = cudaMemsetAsync(ss, 0, L.dec - L.ss, s)) != cudaSuccess) return e;
    size_t off[kLayerGemms + 1];
    layer_split_plan(a.B, a.D, a.H, a.d_q, a.d_v, a.r, a.r_q, off);
    GemmArgs gm{};
    gm.M = a.B;
    gm.dev_err = a.dev_err;
    gm.num_sms = a.num_sms;
    gm.eps = kRmsEps;
    gm.ss = ss;
    auto run = [&](int which, const void *A, long long lda, const void *Bw, void *C, int N, int K, int epi,
                   float n_norm) {
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
        gm.split_acc = nullptr;
        const size_t need = gemm_bf16_split_bytes(gm);
        if (need != 0 && need <= off[which + 1] - off[which])
            gm.split_acc = reinterpret_cast<float *>(ws + L.acc + off[which]);
        return launch_gemm_bf16(gm, s);
    };
    if ((e = run(kQDown, a.x, a.D, a.w_q_down, yq, a.r_q, a.D, kGemmSumSq, 0.f)) != cudaSuccess) return e;
    if ((e = run(kQUp, yq, a.r_q, a.w_q_up, q, Hq, a.r_q, kGemmRowScale, static_cast<float>(a.r_q))) != cudaSuccess)
        return e;
    if ((e = run(kKvDown, a.x, a.D, a.w_kv_down, c, a.r, a.D, kGemmRmsNorm, static_cast<float>(a.r))) !=
        cudaSuccess)
        return e;
    if ((e = run(kGate, a.x, a.D, a.w_gate, g, Hv, a.D, kGemmPlain, 0.f)) != cudaSuccess) return e;
    note_launch();
    append_latent_kernel<<<a.B, 64, 0, s>>>(c, static_cast<__nv_bfloat16 *>(a.c_cache), a.ld_cache, a.lens, lens1,
                                            a.max_len, a.r, a.dev_err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CUtensorMap tm_q, tm_w;
    {
        const cuuint64_t qd[3] = {static_cast<cuuint64_t>(a.d_q), static_cast<cuuint64_t>(a.H),
                                  static_cast<cuuint64_t>(a.B)};
        const cuuint64_t qs[2] = {static_cast<cuuint64_t>(a.d_q) * 2, static_cast<cuuint64_t>(Hq) * 2};
        const cuuint32_t qb[3] = {64, 1, 128};
        const cuuint64_t wd[3] = {static_cast<cuuint64_t>(a.r), static_cast<cuuint64_t>(a.d_q),
                                  static_cast<cuuint64_t>(a.H)};
        const cuuint64_t wstr[2] = {static_cast<cuuint64_t>(a.r) * 2, static_cast<cuuint64_t>(a.d_q) * a.r * 2};
        const cuuint32_t wb[3] = {64, 64, 1};
        if (encode_bf16_3d(&tm_q, q, qd, qs, qb) != CUDA_SUCCESS ||
            encode_bf16_3d(&tm_w, w_uk, wd, wstr, wb) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t asmem = absorb_smem_bytes(a.d_q, a.r);
    if ((e = cudaFuncSetAttribute(absorb_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(asmem))) != cudaSuccess)
        return e;
    note_launch();
    absorb_query_kernel<<<dim3(a.H, (a.B + 127) / 128, a.r / kAbsCols), kAbsThreads, asmem, s>>>(
        tm_q, tm_w, qa, a.B, a.H, a.d_q, a.r, a.dev_err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    DecodeArgs da{qa, a.c_cache, w_uv, g, lens1, o, a.ld_cache, a.max_len, a.scale, a.B, a.H, a.d_v, a.r,
                  ws + L.dec, dec_bytes, a.dev_err, a.num_sms};
    if ((e = launch_decode_bf16(da, s)) != cudaSuccess) return e;
    return run(kOProj, o, Hv, a.w_o, a.y, a.D, Hv, kGemmPlain, 0.f);
}

}  // namespace mla
