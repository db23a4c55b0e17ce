// bf16 GEMM on the sm_103a tensor cores for the Gated-MLA layer's projections
// (page "Gated MLA（矩阵吸收版）": section "低秩压缩", c = RMSNorm(W_down x); section
// "完整计算流（四步）" step 1, q = W_q_up RMSNorm(W_q_down x), and step 4, the gate
// logits W_g x and the output projection W_o):
//
//   C[M, N] = A[M, K] . B[N, K]^T
//
// A is the activation matrix (row-major), B an nn.Linear weight [out, in]
// (row-major), both K-major operands; fp32 accumulation in TMEM, bf16 output.
// Epilogues (a thread owns one row of the 128-row tile):
//   kPlain     C = A B^T
//   kSumSq     C = A B^T, and ss[m] += sum_n (A B^T)[m, n]^2 in fp32 before
//              rounding (atomics across the N tiles of a row)
//   kRowScale  C = (A B^T)[m, :] / sqrt(ss[m] / n_norm + eps): RMSNorm of the
//              previous product moved past this right-multiplication, since
//              RMSNorm(y) W^T = (y W^T) / rms(y) row by row
//   kRmsNorm   C = RMSNorm(A B^T) with a whole 512-column row in one tile
//
// Persistent: one CTA per SM walks tiles of 128 x 256 (two TMEM accumulators,
// so one tile's epilogue overlaps the next tile's products) or 128 x 512
// (kRmsNorm, one accumulator), grouped 8 row-tiles at a time so the A and B
// tiles a wave touches stay in L2.  K steps of 64 through a TMA ring.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kGroupM = 8;
constexpr int kThreads = 256;   // warp 0 TMA, warp 1 MMA (and TMEM), warps 4-7 epilogue
constexpr uint32_t kASlab = 128 * 128;   // [128 rows x 64 bf16], 128-byte swizzle
constexpr uint32_t kBSlab = 256 * 128;   // [256 rows x 64 bf16]

enum Mode { kPlain = 0, kSumSq = 1, kRowScale = 2, kRmsNorm = 3 };

template <int kMode>
struct Cfg {
    static constexpr int kSub = kMode == kRmsNorm ? 2 : 1;            // 256-column halves per tile
    static constexpr int kBN = 256 * kSub;
    static constexpr int kAcc = kMode == kRmsNorm ? 1 : 2;            // TMEM accumulators
    static constexpr uint32_t kStage = kASlab + kSub * kBSlab;
    static constexpr int kStages = kMode == kRmsNorm ? 2 : 4;
    static constexpr uint32_t kBars = kStages * kStage;
    static constexpr uint32_t kSmem = kBars + 256 + 1024;
};

struct GemmParams {
    __nv_bfloat16 *C;
    float *ss;   // kSumSq: accumulated; kRowScale: read
    int *err;
    int M, N, K;
    long long ldc;
    float n_norm, eps;
};

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int &m, int &n) {
    const int group = kGroupM * n_tiles;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(m_tiles - first_m, kGroupM);
    const int in = t % group;
    m = first_m + in % gm;
    n = in / gm;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const GemmParams p) {
    using C = Cfg<kMode>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + C::kBars);
    uint64_t *empty = full + C::kStages;
    uint64_t *acc_full = empty + C::kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (p.M + kBM - 1) / kBM, n_tiles = p.N / C::kBN, k_steps = p.K / kBK;
    const int n_all = m_tiles * n_tiles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(acc_full + i), 1);
            mbar_init(smem_u32(acc_empty + i), 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < n_all; t += gridDim.x) {
            int mt, nt;
            tile_coords(t, m_tiles, n_tiles, mt, nt);
            for (int ks = 0; ks < k_steps; ++ks, ++it) {
                const int st = it % C::kStages;
                if (it >= static_cast<uint32_t>(C::kStages) &&
                    !(ok = mbar_wait(smem_u32(empty + st), ((it / C::kStages) - 1) & 1, p.err, abort_flag)))
                    break;
                const uint32_t bar = smem_u32(full + st);
                const uint32_t dst = base + st * C::kStage;
                mbar_arrive_expect_tx(bar, C::kStage);
                tma_load_2d(dst, &tm_a, bar, ks * kBK, mt * kBM);
                for (int sub = 0; sub < C::kSub; ++sub)
                    tma_load_2d(dst + kASlab + sub * kBSlab, &tm_b, bar, ks * kBK, nt * C::kBN + sub * 256);
            }
        }
        if (!ok) *abort_flag = 1;
        for (uint32_t k = (it > static_cast<uint32_t>(C::kStages) ? it - C::kStages : 0); k < it; ++k)
            mbar_wait(smem_u32(full + k % C::kStages), (k / C::kStages) & 1, p.err);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = make_idesc_bf16(128, 256, 0, 0);
        uint32_t it = 0, at = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < n_all; t += gridDim.x, ++at) {
            const int buf = at % C::kAcc;
            if (at >= static_cast<uint32_t>(C::kAcc) &&
                !(ok = mbar_wait(smem_u32(acc_empty + buf), ((at / C::kAcc) - 1) & 1, p.err, abort_flag)))
                break;
            tc_fence_after();
            for (int ks = 0; ks < k_steps; ++ks, ++it) {
                const int st = it % C::kStages;
                if (!(ok = mbar_wait(smem_u32(full + st), (it / C::kStages) & 1, p.err, abort_flag))) break;
                tc_fence_after();
                const uint32_t a0 = base + st * C::kStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = make_smem_desc(a0 + kk * 32, 16, 1024);
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub) {
                        const uint64_t bd = make_smem_desc(a0 + kASlab + sub * kBSlab + kk * 32, 16, 1024);
                        umma_bf16(tmem + buf * 256 + sub * 256, ad, bd, idesc, (ks | kk) != 0);
                    }
                }
                umma_commit(smem_u32(empty + st));
            }
            if (!ok) break;
            umma_commit(smem_u32(acc_full + buf));
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 4) {
        // ---- epilogue: thread `row` owns TMEM lane `row` = row m0 + row of the tile
        const int row = (warp & 3) * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        uint32_t at = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_all; t += gridDim.x, ++at) {
            int mt, nt;
            tile_coords(t, m_tiles, n_tiles, mt, nt);
            const int buf = at % C::kAcc;
            const bool fail = !mbar_wait(smem_u32(acc_full + buf), (at / C::kAcc) & 1, p.err, abort_flag);
            if (__any_sync(0xffffffffu, fail)) { ok = false; break; }
            tc_fence_after();
            const int m = mt * kBM + row;
            const bool live = m < p.M;
            const uint32_t tacc = trow + buf * 256;
            float scale = 1.f;
            if (kMode == kRowScale) scale = live ? rsqrtf(p.ss[m] / p.n_norm + p.eps) : 1.f;
            if (kMode == kRmsNorm) {   // first pass over the row: its mean square
                float acc = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < C::kBN / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tacc + cc * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc = fmaf(v[i], v[i], acc);
                }
                scale = rsqrtf(acc / p.n_norm + p.eps);
            }
            float ssq = 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.C + static_cast<size_t>(live ? m : 0) * p.ldc + nt * C::kBN);
#pragma unroll 1
            for (int cc = 0; cc < C::kBN / 32; ++cc) {
                float v[32];
                tmem_ld32(tacc + cc * 32, v);
                tmem_wait_ld();
                if (kMode == kSumSq)
#pragma unroll
                    for (int i = 0; i < 32; ++i) ssq = fmaf(v[i], v[i], ssq);
                if (live)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[cc * 4 + q] = make_uint4(pack_bf16x2(v[8 * q] * scale, v[8 * q + 1] * scale),
                                                     pack_bf16x2(v[8 * q + 2] * scale, v[8 * q + 3] * scale),
                                                     pack_bf16x2(v[8 * q + 4] * scale, v[8 * q + 5] * scale),
                                                     pack_bf16x2(v[8 * q + 6] * scale, v[8 * q + 7] * scale));
            }
            if (kMode == kSumSq && live) atomicAdd(p.ss + m, ssq);
            tc_fence_before();
            mbar_arrive(smem_u32(acc_empty + buf));   // the accumulator may take the next tile
        }
        if (!ok) *abort_flag = 1;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

CUresult encode_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems,
                   uint32_t box_outer) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld_elems * 2};
    const cuuint32_t box[2] = {64, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int kMode>
cudaError_t launch_mode(const GemmArgs &g, cudaStream_t s) {
    using C = Cfg<kMode>;
    if (g.N % C::kBN != 0 || g.K % kBK != 0 || g.M < 0) return cudaErrorInvalidValue;
    if (g.M == 0) return cudaSuccess;
    CUtensorMap tm_a, tm_b;
    if (encode_2d(&tm_a, g.A, g.K, g.M, g.lda, kBM) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_2d(&tm_b, g.B, g.K, g.N, g.ldb, 256) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmem));
    if (e != cudaSuccess) return e;
    GemmParams p;
    p.C = static_cast<__nv_bfloat16 *>(g.C);
    p.ss = g.ss;
    p.err = g.dev_err;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.ldc = g.ldc;
    p.n_norm = g.n_norm;
    p.eps = g.eps;
    const long long tiles = static_cast<long long>((g.M + kBM - 1) / kBM) * (g.N / C::kBN);
    const int grid = static_cast<int>(tiles < g.num_sms ? tiles : g.num_sms);
    gemm_bf16_kernel<kMode><<<grid, kThreads, C::kSmem, s>>>(tm_a, tm_b, p);
    return cudaGetLastError();
}

}  // namespace

bool gemm_bf16_supports(int N, int K, int epilogue) {
    const int bn = epilogue == kGemmRmsNorm ? 512 : 256;
    return N > 0 && K > 0 && N % bn == 0 && K % kBK == 0;
}

cudaError_t launch_gemm_bf16(const GemmArgs &g, cudaStream_t s) {
    switch (g.epilogue) {
        case kGemmPlain: return launch_mode<kPlain>(g, s);
        case kGemmSumSq: return launch_mode<kSumSq>(g, s);
        case kGemmRowScale: return launch_mode<kRowScale>(g, s);
        case kGemmRmsNorm: return launch_mode<kRmsNorm>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mla
