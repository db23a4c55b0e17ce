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
//
// When those tiles cannot fill the SMs (few rows):
// - M <= 128 (a decode step): the operands swap roles.  The weight streams as
//   the 128-row MMA operand (128 output columns per tile, every byte of the
//   stage useful) and the few activation rows are the narrow one; the ring
//   deepens to up to 8 stages to keep the weight stream busy, and tiles cut
//   their K range into chunks for more CTAs.  Thread n of the epilogue holds
//   output column n for every row: a plain product without chunks stores bf16
//   directly, everything else adds into a zeroed fp32 buffer (vector-free
//   atomics, coalesced across the warp) that a row pass finishes.
// - otherwise: tiles narrow to 128 or 64 columns and, if still too few, cut K
//   into chunks that add into the fp32 buffer; the CTA that finishes a tile's
//   last chunk (a per-tile ticket) reads the sums back and applies the
//   epilogue (kRmsNorm, which needs whole rows, leaves it to the row pass).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kGroupM = 8;
constexpr int kThreads = 256;   // warp 0 TMA, warp 1 MMA (and TMEM), warps 4-7 epilogue
constexpr int kMaxStages = 8;
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
    static constexpr uint32_t kBars = kStages * kStage;   // the ring; narrower stages fit more of them
    static constexpr uint32_t kSmem = kBars + 256 + 1024;
};

struct GemmParams {
    __nv_bfloat16 *C;
    float *ss;    // kSumSq: accumulated; kRowScale: read
    float *acc;   // split K: fp32 [M, N] partial sums (zeroed before the launch)
    int *sem;     // split K: per-tile count of finished K chunks (zeroed before the launch)
    int *err;
    int M, N, K;
    long long ldc;
    float n_norm, eps;
    int swap;                 // 1: A operand = 128 weight rows, B operand = the (<= 128) activation rows
    int bn;                   // B-operand rows per tile: output columns, or the padded activation rows
    int k_split, steps_per;   // K chunks per tile and 64-wide steps per chunk
    int stages;               // ring depth (<= kMaxStages)
    int rotate;               // 1: each tile starts its K walk at its own offset (few rows: the CTAs
                              //    then read different activation tiles at a time, not one hot tile)
    uint32_t stage_bytes;     // ring stride (a multiple of 1024)
};

__device__ __forceinline__ void red_add(float *addr, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int &m, int &n) {
    const int group = kGroupM * n_tiles;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(m_tiles - first_m, kGroupM);
    const int in = t % group;
    m = first_m + in % gm;
    n = in / gm;
}

// kFew: the few-rows regimes take their cut from the parameters; the default
// path keeps it in compile-time constants.
template <int kMode, bool kFew>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const GemmParams p) {
    using C = Cfg<kMode>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + C::kBars);
    uint64_t *empty = full + kMaxStages;
    uint64_t *acc_full = empty + kMaxStages;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ticket = reinterpret_cast<volatile int *>(tmem_slot + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile grid: rows of the A operand in 128-blocks x rows of the B operand in bn-blocks
    const bool swap = kFew && p.swap, rotate = kFew && p.rotate;
    const int bn = kFew ? p.bn : C::kBN, ksplit = kFew ? p.k_split : 1, nst = kFew ? p.stages : C::kStages;
    const uint32_t sbytes = kFew ? p.stage_bytes : C::kStage;
    const int m_tiles = swap ? p.N / kBM : (p.M + kBM - 1) / kBM, n_tiles = swap ? 1 : p.N / bn;
    const int k_steps = p.K / kBK, steps_per = kFew ? p.steps_per : k_steps;
    const int n_sub = bn > 256 ? 2 : 1, mma_n = bn > 256 ? 256 : bn;   // products of <= 256 columns
    const int n_all = m_tiles * n_tiles * ksplit;   // work items: (tile, K chunk)
    // K steps of work item w: ks0 .. ks1-1, walked from ks0 + rot (mod the range)
    auto k_range = [&](int w, int &ks0, int &ks1, int &rot) {
        ks0 = (w % ksplit) * steps_per;
        ks1 = min(ks0 + steps_per, k_steps);
        rot = rotate ? static_cast<int>((static_cast<unsigned>(w / ksplit) * 13u) % (ks1 - ks0)) : 0;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < nst; ++i) {
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
    grid_launch_dependents();   // a row pass launched after this grid may get ready meanwhile

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < n_all; t += gridDim.x) {
            int mt, nt, ks0, ks1, rot;
            tile_coords(t / ksplit, m_tiles, n_tiles, mt, nt);
            k_range(t, ks0, ks1, rot);
            for (int j = 0; j < ks1 - ks0; ++j, ++it) {
                const int ks = ks0 + (j + rot) % (ks1 - ks0);
                const int st = it % nst;
                if (it >= static_cast<uint32_t>(nst) &&
                    !(ok = mbar_wait(smem_u32(empty + st), ((it / nst) - 1) & 1, p.err, abort_flag)))
                    break;
                const uint32_t bar = smem_u32(full + st);
                const uint32_t dst = base + st * sbytes;
                mbar_arrive_expect_tx(bar, kASlab + n_sub * mma_n * 128);
                tma_load_2d(dst, &tm_a, bar, ks * kBK, mt * kBM);
                for (int sub = 0; sub < n_sub; ++sub)
                    tma_load_2d(dst + kASlab + sub * kBSlab, &tm_b, bar, ks * kBK, nt * bn + sub * 256);
            }
        }
        if (!ok) *abort_flag = 1;
        for (uint32_t k = (it > static_cast<uint32_t>(nst) ? it - nst : 0); k < it; ++k)
            mbar_wait(smem_u32(full + k % nst), (k / nst) & 1, p.err);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = make_idesc_bf16(128, mma_n, 0, 0);
        uint32_t it = 0, at = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < n_all; t += gridDim.x, ++at) {
            const int buf = at % C::kAcc;
            if (at >= static_cast<uint32_t>(C::kAcc) &&
                !(ok = mbar_wait(smem_u32(acc_empty + buf), ((at / C::kAcc) - 1) & 1, p.err, abort_flag)))
                break;
            tc_fence_after();
            int ks0, ks1, rot;
            k_range(t, ks0, ks1, rot);
            for (int j = 0; j < ks1 - ks0; ++j, ++it) {
                const int st = it % nst;
                if (!(ok = mbar_wait(smem_u32(full + st), (it / nst) & 1, p.err, abort_flag))) break;
                tc_fence_after();
                const uint32_t a0 = base + st * sbytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = make_smem_desc(a0 + kk * 32, 16, 1024);
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub) {
                        if (sub >= n_sub) break;
                        const uint64_t bd = make_smem_desc(a0 + kASlab + sub * kBSlab + kk * 32, 16, 1024);
                        umma_bf16(tmem + buf * 256 + sub * 256, ad, bd, idesc, j > 0 || kk != 0);
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
            tile_coords(t / ksplit, m_tiles, n_tiles, mt, nt);
            const int buf = at % C::kAcc;
            const bool fail = !mbar_wait(smem_u32(acc_full + buf), (at / C::kAcc) & 1, p.err, abort_flag);
            if (named_bar_or(1, 128, fail)) { ok = false; break; }   // uniform over the epilogue warps
            tc_fence_after();
            const uint32_t tacc = trow + buf * 256;
            if (swap) {   // thread `row` holds output column n for the activation rows 0..bn-1
                const int n = mt * kBM + row;
                const bool direct = kMode == kPlain && ksplit == 1;
#pragma unroll 1
                for (int cc = 0; cc < bn / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tacc + cc * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int m = cc * 32 + i;
                        if (m < p.M) {
                            if (direct)
                                p.C[static_cast<size_t>(m) * p.ldc + n] = __float2bfloat16_rn(v[i]);
                            else
                                red_add(p.acc + static_cast<size_t>(m) * p.N + n, v[i]);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(acc_empty + buf));
                continue;
            }
            const int m = mt * kBM + row;
            const bool live = m < p.M;
            const float *gsum = p.acc + static_cast<size_t>(live ? m : 0) * p.N + nt * bn;
            bool from_global = false;
            if (ksplit > 1) {   // a K chunk: add the partial tile into the fp32 buffer
#pragma unroll 1
                for (int cc = 0; cc < bn / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tacc + cc * 32, v);
                    tmem_wait_ld();
                    if (live)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            red_add_v4(const_cast<float *>(gsum) + cc * 32 + 4 * q, v[4 * q], v[4 * q + 1],
                                       v[4 * q + 2], v[4 * q + 3]);
                }
                tc_fence_before();
                mbar_arrive(smem_u32(acc_empty + buf));
                if (kMode == kRmsNorm) continue;   // the row pass normalises the sums
                __threadfence();
                named_bar_sync(1, 128);
                if (threadIdx.x == 128) *ticket = atomicAdd(p.sem + t / ksplit, 1);
                named_bar_sync(1, 128);
                if (*ticket != ksplit - 1) continue;   // another chunk of this tile is still running
                __threadfence();
                from_global = true;
            }
            // the tile's sums: TMEM, or (split K, last chunk) the fp32 buffer every chunk added into
            auto load = [&](int cc, float(&v)[32]) {
                if (from_global) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = __ldcg(reinterpret_cast<const float4 *>(gsum + cc * 32) + q);
                        v[4 * q] = f.x;
                        v[4 * q + 1] = f.y;
                        v[4 * q + 2] = f.z;
                        v[4 * q + 3] = f.w;
                    }
                } else {
                    tmem_ld32(tacc + cc * 32, v);
                    tmem_wait_ld();
                }
            };
            float scale = 1.f;
            if (kMode == kRowScale) scale = live ? rsqrtf(p.ss[m] / p.n_norm + p.eps) : 1.f;
            if (kMode == kRmsNorm) {   // first pass over the row: its mean square
                float acc = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < bn / 32; ++cc) {
                    float v[32];
                    load(cc, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc = fmaf(v[i], v[i], acc);
                }
                scale = rsqrtf(acc / p.n_norm + p.eps);
            }
            float ssq = 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.C + static_cast<size_t>(live ? m : 0) * p.ldc + nt * bn);
#pragma unroll 1
            for (int cc = 0; cc < bn / 32; ++cc) {
                float v[32];
                load(cc, v);
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
            if (from_global) continue;                  // the accumulator was released above
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

// Row pass over the fp32 sums: C = the epilogue of `kMode` applied to them.
// Grid (M, column chunks of 2048); kSumSq and kRmsNorm, which need the whole
// row's sum of squares, take one chunk per row.  Launched as a dependent of
// the GEMM grid, it waits for that grid before reading.
template <int kMode>
__global__ void __launch_bounds__(256) finish_sums_kernel(const GemmParams p) {
    __shared__ float red[8];
    grid_dependency_wait();
    const int m = blockIdx.x;
    const float *row = p.acc + static_cast<size_t>(m) * p.N;
    float scale = 1.f;
    if (kMode == kSumSq || kMode == kRmsNorm) {
        float s = 0.f;
        for (int n = threadIdx.x * 4; n < p.N; n += blockDim.x * 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(row + n));
            s = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, s))));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += red[w];
        if (kMode == kSumSq && threadIdx.x == 0) atomicAdd(p.ss + m, tot);
        if (kMode == kRmsNorm) scale = rsqrtf(tot / p.n_norm + p.eps);
    }
    if (kMode == kRowScale) scale = rsqrtf(p.ss[m] / p.n_norm + p.eps);
    const int n1 = (kMode == kSumSq || kMode == kRmsNorm) ? p.N : min(p.N, (blockIdx.y + 1) * 2048);
    for (int n = blockIdx.y * 2048 + threadIdx.x * 8; n < n1; n += blockDim.x * 8) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(row + n));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(row + n + 4));
        *reinterpret_cast<uint4 *>(p.C + static_cast<size_t>(m) * p.ldc + n) =
            make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                       pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
    }
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

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// How a product is cut.
struct Plan {
    int swap, bn, k_split, steps_per, stages;
    uint32_t stage_bytes;
    bool scratch;   // adds into the fp32 buffer (which must be zeroed)
    bool finish;    // a row pass turns the sums into C
};

int clamp_split(long long per, int k_steps) {
    return per < 1 ? 1 : (per > k_steps ? k_steps : static_cast<int>(per));
}

template <int kMode>
Plan make_plan(const GemmArgs &g, bool have_scratch) {
    using C = Cfg<kMode>;
    const long long m_tiles = (g.M + kBM - 1) / kBM;
    const int k_steps = g.K / kBK;
    Plan pl{0, C::kBN, 1, k_steps, C::kStages, C::kStage, false, false};
    if (m_tiles * (g.N / C::kBN) * 2 > g.num_sms) return pl;   // enough tiles as they are
    if (g.M <= kBM && g.N % kBM == 0) {
        // swapped operands: 128 weight rows x the activation rows padded to 32
        const int bt = (g.M + 31) / 32 * 32;
        // K chunks per tile: the fewest weight-plus-atomic bytes on the busiest SM
        // (waves of work items x bytes of one item), counted per 64-wide K step
        const long long tiles = g.N / kBM;
        int ks = 1;
        double best = 0.0;
        for (int cand = 1; cand <= k_steps && cand <= 64; ++cand) {
            const int per = (k_steps + cand - 1) / cand;
            const int chunks = (k_steps + per - 1) / per;
            if (chunks != cand) continue;   // the same cut as a smaller count
            const long long waves = (tiles * chunks + g.num_sms - 1) / g.num_sms;
            const bool adds = kMode != kPlain || chunks > 1;
            const double cost = static_cast<double>(waves) *
                                (static_cast<double>(kBM) * per * kBK * 2 + (adds ? 4.0 * g.M * kBM : 0.0));
            if (cand == 1 || cost < best) {
                best = cost;
                ks = cand;
            }
        }
        const bool scratch = kMode != kPlain || ks > 1;
        if (!scratch || have_scratch) {
            Plan sp{1, bt, ks, (k_steps + ks - 1) / ks, 0, kASlab + static_cast<uint32_t>(bt) * 128, scratch,
                    scratch};
            sp.k_split = (k_steps + sp.steps_per - 1) / sp.steps_per;
            sp.stages = static_cast<int>(C::kBars / sp.stage_bytes);
            if (sp.stages > kMaxStages) sp.stages = kMaxStages;
            return sp;
        }
    }
    // the widest narrower tile that gives half the SMs a tile, else 64 columns
    int bn = 64;
    if (kMode != kRmsNorm)
        for (int cand = 128; cand > 64; cand >>= 1)
            if (m_tiles * (g.N / cand) * 2 >= g.num_sms) {
                bn = cand;
                break;
            }
    int ks = clamp_split(g.num_sms / (m_tiles * (g.N / bn)), k_steps);
    if (kMode == kRmsNorm && ks == 1) {   // a narrow tile alone cannot normalise a row: keep whole rows
        bn = C::kBN;
        ks = clamp_split(g.num_sms / m_tiles, k_steps);
    }
    if (ks > 1 && !have_scratch) ks = 1;
    if (kMode == kRmsNorm && ks == 1) return pl;
    pl.bn = bn;
    pl.steps_per = (k_steps + ks - 1) / ks;
    pl.k_split = (k_steps + pl.steps_per - 1) / pl.steps_per;
    pl.scratch = pl.k_split > 1;
    pl.finish = kMode == kRmsNorm;
    return pl;
}

// Zeroed scratch a launch needs when it adds into the fp32 buffer: the sums, then a
// ticket per 64-column tile (the count for the narrowest tiles, so the size does not
// depend on the cut); 0 when it does not.
template <int kMode>
size_t split_bytes(const GemmArgs &g) {
    using C = Cfg<kMode>;
    if (g.M <= 0 || g.N % C::kBN != 0 || g.K % kBK != 0) return 0;
    if (!make_plan<kMode>(g, true).scratch) return 0;
    const size_t tiles64 = static_cast<size_t>((g.M + kBM - 1) / kBM) * (g.N / 64);
    return align256(static_cast<size_t>(g.M) * g.N * sizeof(float)) + align256(tiles64 * sizeof(int));
}

template <int kMode>
cudaError_t launch_mode(const GemmArgs &g, cudaStream_t s) {
    using C = Cfg<kMode>;
    if (g.N % C::kBN != 0 || g.K % kBK != 0 || g.M < 0) return cudaErrorInvalidValue;
    if (g.M == 0) return cudaSuccess;
    CUtensorMap tm_a, tm_b;
    if (encode_2d(&tm_a, g.A, g.K, g.M, g.lda, kBM) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const Plan pl = make_plan<kMode>(g, g.split_acc != nullptr);
    if (pl.swap) {   // A operand = the weight, B operand = the activation rows
        if (encode_2d(&tm_a, g.B, g.K, g.N, g.ldb, kBM) != CUDA_SUCCESS ||
            encode_2d(&tm_b, g.A, g.K, g.M, g.lda, pl.bn) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else if (encode_2d(&tm_b, g.B, g.K, g.N, g.ldb, pl.bn > 256 ? 256 : pl.bn) != CUDA_SUCCESS) {
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<kMode, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_bf16_kernel<kMode, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    p.swap = pl.swap;
    p.bn = pl.bn;
    p.k_split = pl.k_split;
    p.steps_per = pl.steps_per;
    p.stages = pl.stages;
    p.rotate = pl.swap || pl.bn != C::kBN;
    p.stage_bytes = pl.stage_bytes;
    p.acc = nullptr;
    p.sem = nullptr;
    if (pl.scratch) {
        p.acc = g.split_acc;
        p.sem = reinterpret_cast<int *>(reinterpret_cast<char *>(g.split_acc) +
                                        align256(static_cast<size_t>(g.M) * g.N * sizeof(float)));
    }
    const long long tiles = pl.swap ? g.N / kBM : static_cast<long long>((g.M + kBM - 1) / kBM) * (g.N / pl.bn);
    const long long work = tiles * pl.k_split;
    const int grid = static_cast<int>(work < g.num_sms ? work : g.num_sms);
    const bool few = pl.swap || pl.bn != C::kBN || pl.k_split > 1 || pl.stages != C::kStages;
    if (few)
        gemm_bf16_kernel<kMode, true><<<grid, kThreads, C::kSmem, s>>>(tm_a, tm_b, p);
    else
        gemm_bf16_kernel<kMode, false><<<grid, kThreads, C::kSmem, s>>>(tm_a, tm_b, p);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess || !pl.finish) return e;
    cudaLaunchConfig_t cfg{};
    const bool whole_rows = kMode == kSumSq || kMode == kRmsNorm;
    cfg.gridDim = dim3(g.M, whole_rows ? 1 : (g.N + 2047) / 2048);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, finish_sums_kernel<kMode>, p);
}

}  // namespace

bool gemm_bf16_supports(int N, int K, int epilogue) {
    if (epilogue == kGemmRmsNorm) return N == 512 && K > 0 && K % kBK == 0;   // a whole row per tile
    return N > 0 && K > 0 && N % 256 == 0 && K % kBK == 0;
}

size_t gemm_bf16_split_bytes(const GemmArgs &g) {
    switch (g.epilogue) {
        case kGemmPlain: return split_bytes<kPlain>(g);
        case kGemmSumSq: return split_bytes<kSumSq>(g);
        case kGemmRowScale: return split_bytes<kRowScale>(g);
        case kGemmRmsNorm: return split_bytes<kRmsNorm>(g);
        default: return 0;
    }
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
