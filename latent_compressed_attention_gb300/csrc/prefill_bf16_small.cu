// bf16 causal absorbed Gated-MLA prefill for small latent ranks (r = 32 or
// 64, d_q and d_v in {16, 32, 48, 64}) on the sm_103a tensor cores, one fused
// kernel; the toy sizes of the course notes (r = 32, d = 16) are the target.
//
// Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）", steps 2-4, as in
// the r = 512 kernel: W_UK absorb prologue, scores against the latent c,
// causal online softmax, latent weighting by the same c tile, W_UV^T and gate
// epilogue.  At these ranks the tensor work per score is tiny (4r FLOPs) and
// the exponentials bound the kernel, so the design aims at many softmax warps
// per SM: one CTA per 128-token tile, 256 TMEM columns and about 100 KB of
// shared memory, two CTAs per SM, and two softmax threads per query row (each
// owns 64 keys of a block; the row maximum and the row sums are exchanged
// through shared memory), with tree reductions to keep dependency chains short.
//
// The score operand q_abs * scale * log2(e) is rounded to a pair of bf16 values
// (hi + lo, about 16 significant bits): one bf16 rounding alone puts a relative
// error of 2^-9 on every score, which at a score spread of ~25 natural-log
// units moves the softmax weights by a few percent.  hi sits in the q tile, lo
// in spare TMEM columns, and S = hi . c^T + lo . c^T; at r = 32 the four K
// steps of one 64-column product are exactly the two of hi and the two of lo.
//
// Narrow rows (r = 32: 64 bytes; d = 16: 32 bytes) are widened to the 128-byte
// swizzled layout by TMA's zero fill past the tensor's inner extent: every
// operand is a [rows x 64] bf16 tile, the padding columns are zero, and they
// add nothing to any product.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kBM = 128;        // tokens per tile
constexpr int kBN = 128;        // keys per block
constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-5 and 6-9: two softmax / epilogue groups
constexpr int kMath = 256;      // softmax threads (two per query row)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

constexpr uint32_t kTile = 16384;   // [128 rows x 64 bf16], 128B swizzle
constexpr uint32_t QT = 0;          // q tile, then q_abs, then the epilogue's o_lat
constexpr uint32_t WK = QT + kTile;             // W_UK[h] [d_q rows x 64]
constexpr uint32_t WV = WK + 8192;              // W_UV[h] [d_v rows x 64]
// c tiles [128 keys x r]: at r = 64 two stages of 128-byte-swizzled rows; at r = 32 the rows are 64 bytes and
// four stages of 64-byte-swizzled tiles fit the same bytes, so the loads run further ahead of the products
constexpr uint32_t RING = WV + 8192;
constexpr int kMaxStages = 4;
constexpr uint32_t kRingBytes = 2 * kTile;
constexpr uint32_t PT = RING + kRingBytes;      // P [128 rows x 128 keys] = 2 tiles
constexpr uint32_t BARS = PT + 2 * kTile;
constexpr uint32_t PMAX = BARS + 256;            // [2 parities][2 groups][128 rows] partial row maxima
constexpr uint32_t LSUM = PMAX + 2 * 2 * kBM * 4;   // [2 groups][128 rows] partial row sums
constexpr uint32_t kSmemBytes = LSUM + 2 * kBM * 4 + 1024;   // + alignment slack
static_assert(RING % 1024 == 0 && PT % 1024 == 0, "alignment");

// TMEM columns: S (128 keys), o_lat (the absorb's output first), and the low bf16 part of the score operand
// (packed pairs, r / 2 columns)
constexpr uint32_t S_COL = 0, O_COL = 128, LO_COL = 192;

struct Bars {
    uint64_t pro_full, absorb_done, qabs_ready;
    uint64_t c_full[kMaxStages], c_empty[kMaxStages];
    uint64_t s_full, s_free, p_full, pv_done, olat_ready, ep_done;
    uint32_t tmem_base;
    int abort;
};

// Pairwise (tree) reductions over 64 values: short dependency chains.
__device__ __forceinline__ float tree_max64(const float (&s)[2][32]) {
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(fmaxf(s[0][i], s[0][i + 16]), fmaxf(s[1][i], s[1][i + 16]));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}
__device__ __forceinline__ float tree_sum64(const float (&s)[2][32]) {
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = (s[0][i] + s[0][i + 16]) + (s[1][i] + s[1][i + 16]);
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] += m[i + w];
    return m[0];
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Barrier of the two softmax warps (one per group) that share TMEM lanes 32 pair .. 32 pair + 31; the ids
// are literals so the kernel reserves barriers 0-5 only.
__device__ __forceinline__ void pair_bar_sync(int pair) {
    switch (pair) {
        case 0: named_bar_sync(2, 64); break;
        case 1: named_bar_sync(3, 64); break;
        case 2: named_bar_sync(4, 64); break;
        default: named_bar_sync(5, 64); break;
    }
}

// Opt-in timeline (build with MLA_NVCC_FLAGS=-DMLA_TRACE): per key block of CTA 0 (a heaviest tile), the
// cycle at which each role passed its waits, and every CTA's start and end on the global timer.
#ifdef MLA_TRACE
constexpr int kSTEv = 9, kSTBlk = 64;
__device__ long long g_stl[kSTEv][kSTBlk];
__device__ unsigned long long g_scta[3][4096];   // start ns, end ns, SM id
#define STL(ev, j) do { if (blockIdx.x == 0 && (j) < kSTBlk) g_stl[ev][j] = clock64() - st_t0; } while (0)
#else
#define STL(ev, j) (void)0
#endif

struct Params {
    const __nv_bfloat16 *gate;
    __nv_bfloat16 *out;
    int *err;
    int T, H, d_q, d_v, r, n_qtiles, bh_count;
    float qk_scale_log2;
};

__global__ void __launch_bounds__(kThreads, 2)
    prefill_small_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                         const __grid_constant__ CUtensorMap tm_wuk, const __grid_constant__ CUtensorMap tm_wuv,
                         const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    Bars *bars = reinterpret_cast<Bars *>(smem_raw + (base - raw) + BARS);
    volatile int *abort_flag = &bars->abort;
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.bh_count;   // heaviest tiles first
    const int bh = static_cast<int>(blockIdx.x) % p.bh_count;
    const int b = bh / p.H, h = bh % p.H;
    const int t0 = qt * kBM;
    const int nkv = qt + 1;
    const bool narrow = p.r == 32;   // 64-byte latent rows
    const int n_stages = narrow ? 4 : 2;
    const uint32_t st_bytes = kRingBytes / static_cast<uint32_t>(n_stages);
#ifdef MLA_TRACE
    const long long st_t0 = clock64();
    if (threadIdx.x == 0 && blockIdx.x < 4096) {
        g_scta[0][blockIdx.x] = globaltimer_ns();
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_scta[2][blockIdx.x] = smid;
    }
#endif

    if (threadIdx.x == 0) {
        mbar_init(B_(bars->pro_full), 1);
        mbar_init(B_(bars->absorb_done), 1);
        mbar_init(B_(bars->qabs_ready), 1);
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(B_(bars->c_full[i]), 1);
            mbar_init(B_(bars->c_empty[i]), 1);
        }
        mbar_init(B_(bars->s_full), 1);
        mbar_init(B_(bars->s_free), kMath);
        mbar_init(B_(bars->p_full), kMath);   // every softmax thread arrives after storing its part of P
        mbar_init(B_(bars->pv_done), 1);
        mbar_init(B_(bars->olat_ready), 1);
        mbar_init(B_(bars->ep_done), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_c);
        const uint32_t pro = B_(bars->pro_full);
        mbar_arrive_expect_tx(pro, kTile + (p.d_q + p.d_v) * 128u);
        tma_load_4d(base + QT, &tm_q, pro, 0, h, t0, b);
        tma_load_2d(base + WK, &tm_wuk, pro, 0, h * p.d_q);
        tma_load_2d(base + WV, &tm_wuv, pro, 0, h * p.d_v);
        bool ok = true;
        int j = 0;
        for (; ok && j < nkv; ++j) {
            const int st = j % n_stages;
            if (j >= n_stages &&
                !(ok = mbar_wait(B_(bars->c_empty[st]), ((j / n_stages) - 1) & 1, p.err, abort_flag)))
                break;
            mbar_arrive_expect_tx(B_(bars->c_full[st]), st_bytes);
            tma_load_3d(base + RING + st * st_bytes, &tm_c, B_(bars->c_full[st]), 0, j * kBN, b);
            STL(7, j);
        }
        if (!ok) *abort_flag = 1;
        mbar_wait(pro, 0, p.err);
        for (int k = (j > n_stages ? j - n_stages : 0); k < j; ++k)
            mbar_wait(B_(bars->c_full[k % n_stages]), (k / n_stages) & 1, p.err);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t id_absorb = make_idesc_bf16(128, 64, 0, 1);
        const uint32_t id_qk = make_idesc_bf16(128, kBN, 0, 0);
        const uint32_t id_pv = make_idesc_bf16(128, p.r, 0, 1);
        const uint32_t id_ep = make_idesc_bf16(128, p.d_v, 0, 0);
        bool ok = mbar_wait(B_(bars->pro_full), 0, p.err, abort_flag);
        if (ok) {
            tc_fence_after();
            for (int kk = 0; kk < p.d_q / 16; ++kk)
                umma_bf16(tmem + O_COL, make_smem_desc(base + QT + kk * 32, 16, 1024),
                          make_smem_desc(base + WK + kk * 2048, 8192, 1024), id_absorb, kk > 0);
            umma_commit(B_(bars->absorb_done));
            ok = mbar_wait(B_(bars->qabs_ready), 0, p.err, abort_flag);
        }
        // S(j + 1) is issued as soon as the softmax has read S(j) out of TMEM, so the next block's scores are
        // ready when the softmax finishes block j; then P(j) . c(j).  The score operand is the pair hi + lo
        // (hi from the q tile, lo from TMEM): S = hi . c^T + lo . c^T, over the r latent columns only.
        // Descriptors: built once per block from the stage's base and advanced by adding offsets, with no
        // branch between two MMAs, so the issuing thread keeps up with these short products.  The latent tile
        // is the score product's K-major operand (latent columns = K) and P . c's MN-major one.
        const uint64_t q_desc = make_smem_desc(base + QT, 16, 1024);
        auto c_desc = [&](int st) {   // K step kk at + 32 kk bytes (K-major); 16 keys at + kv_step (MN-major)
            const uint32_t a = base + RING + st * st_bytes;
            return narrow ? make_smem_desc_sw64(a, 16, 512) : make_smem_desc(a, 16, 1024);
        };
        const uint32_t kv_step = narrow ? 1024u : 2048u;
        const uint64_t pv_b_lbo = static_cast<uint64_t>((8192u - 16u) >> 4) << 16;   // leading offset 16 -> 8192
        auto issue_scores = [&](int j) {
            const uint64_t cb = c_desc(j % n_stages);
            tc_fence_after();
            if (narrow) {   // r = 32: two K steps of hi, two of lo
                umma_bf16(tmem + S_COL, q_desc, cb, id_qk, 0);
                umma_bf16(tmem + S_COL, desc_add(q_desc, 32), desc_add(cb, 32), id_qk, 1);
                umma_bf16_tmem_a(tmem + S_COL, tmem + LO_COL, cb, id_qk, 1);
                umma_bf16_tmem_a(tmem + S_COL, tmem + LO_COL + 8, desc_add(cb, 32), id_qk, 1);
            } else {        // r = 64: four of each
    #pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + S_COL, desc_add(q_desc, kk * 32), desc_add(cb, kk * 32), id_qk, kk > 0);
    #pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16_tmem_a(tmem + S_COL, tmem + LO_COL + kk * 8, desc_add(cb, kk * 32), id_qk, 1);
            }
            umma_commit(B_(bars->s_full));
            STL(0, j);
        };
        if (ok && (ok = mbar_wait(B_(bars->c_full[0]), 0, p.err, abort_flag))) issue_scores(0);
        for (int j = 0; ok && j < nkv; ++j) {
            if (j + 1 < nkv) {
                const int sn = (j + 1) % n_stages;
                if (!(ok = mbar_wait(B_(bars->c_full[sn]), ((j + 1) / n_stages) & 1, p.err, abort_flag))) break;
                if (!(ok = mbar_wait(B_(bars->s_free), j & 1, p.err, abort_flag))) break;
                issue_scores(j + 1);
            }
            if (!(ok = mbar_wait(B_(bars->p_full), j & 1, p.err, abort_flag))) break;
            STL(1, j);
            tc_fence_after();
            const int st = j % n_stages;
            // the MN-major view of the tile: leading byte offset 8192 (the next 64 latent columns, read at r = 64)
            const uint64_t cv = c_desc(st) + pv_b_lbo;
            const uint64_t pa = make_smem_desc(base + PT, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                umma_bf16(tmem + O_COL, desc_add(pa, (kk >> 2) * kTile + (kk & 3) * 32), desc_add(cv, kk * kv_step), id_pv,
                          (j > 0 || kk > 0));
            umma_commit(B_(bars->c_empty[st]));
            umma_commit(B_(bars->pv_done));
            STL(2, j);
        }
        if (ok && (ok = mbar_wait(B_(bars->olat_ready), 0, p.err, abort_flag))) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < p.r / 16; ++kk)   // o_lat's columns past r are not products
                umma_bf16(tmem + S_COL, make_smem_desc(base + QT + kk * 32, 16, 1024),
                          make_smem_desc(base + WV + kk * 32, 16, 1024), id_ep, kk > 0);
            umma_commit(B_(bars->ep_done));
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 2) {
        // ---- softmax / epilogue: group g (warps 2-5 or 6-9) owns keys [64 g, 64 g + 64) of every block and
        // 32-column chunk g of the 64-column q_abs / o_lat tiles; thread `row` owns TMEM lane `row`
        const int g = (warp - 2) >> 2;
        const int row = (warp & 3) * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int t = t0 + row;
        const bool leader = threadIdx.x == 64;   // arrives on the barriers the MMA warp waits for
        bool fail = !mbar_wait(B_(bars->absorb_done), 0, p.err, abort_flag);
        bool ok = !named_bar_or(1, kMath, fail);
        if (ok) {   // q_abs (fp32 TMEM) -> x = q_abs * scale * log2(e) as hi = bf16(x) into the q tile and
                    // lo = bf16(x - hi) packed into TMEM: the score operand keeps about 16 significant bits
            tc_fence_after();
            float v[32], lo[16];
            tmem_ld32(trow + O_COL + g * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x0 = v[2 * i] * p.qk_scale_log2, x1 = v[2 * i + 1] * p.qk_scale_log2;
                const uint32_t hw = pack_bf16x2(x0, x1);
                lo[i] = __uint_as_float(pack_bf16x2(x0 - __uint_as_float(hw << 16), x1 - __uint_as_float(hw & 0xFFFF0000u)));
                v[2 * i] = x0;
                v[2 * i + 1] = x1;
            }
            store_row32_bf16(base + QT, kTile, row, g, v, 1.f);
            tmem_st16(trow + LO_COL + g * 16, lo);
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
        }
        named_bar_sync(1, kMath);
        if (leader && ok) mbar_arrive(B_(bars->qabs_ready));
        if (!ok) *abort_flag = 1;   // every later wait then returns at once

        float m_run = -INFINITY, l_run = 0.f;   // l_run: this group's part of the row sum
        // Per block the only barrier is between the two warps (one per group) that share these rows.  A wait
        // that fails sets the abort flag, after which every wait returns at once: all threads still run the
        // same barrier sequence, and one vote after the loop settles the outcome.
        const int pair = warp & 3;
        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait(B_(bars->s_full), j & 1, p.err, abort_flag)) ok = false, *abort_flag = 1;
            if (leader) STL(3, j);
            tc_fence_after();
            float s[2][32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) tmem_ld32(trow + S_COL + g * 64 + c2 * 32, s[c2]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(B_(bars->s_free));
            if (j == nkv - 1) {   // diagonal block: keys after the query or past the sequence
                const int lim = min(t, p.T - 1) - j * kBN - g * 64;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c2 * 32 + i > lim) s[c2][i] = -INFINITY;
            }
            st_shared_f32(base + PMAX + ((j & 1) * 2 + g) * kBM * 4 + row * 4, tree_max64(s));
            pair_bar_sync(pair);   // publishes both groups' partial maxima of these rows
            const float mx = fmaxf(ld_shared_f32(base + PMAX + ((j & 1) * 2 + 0) * kBM * 4 + row * 4),
                                   ld_shared_f32(base + PMAX + ((j & 1) * 2 + 1) * kBM * 4 + row * 4));
            float factor = 1.f;
            if (mx > m_run + kRescaleLog2) {
                factor = fast_exp2(m_run - mx);
                m_run = mx;
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c2][i] = fast_exp2(s[c2][i] - m_run);
            l_run = l_run * factor + tree_sum64(s);
            if (leader) STL(4, j);
            if (j > 0) {   // P and o_lat are free once the previous block's product completed
                if (!mbar_wait(B_(bars->pv_done), (j - 1) & 1, p.err, abort_flag)) ok = false, *abort_flag = 1;
                if (leader) STL(5, j);
                if (__any_sync(0xffffffffu, factor != 1.f)) {   // this warp's rows of o_lat (warp-collective)
                    tc_fence_after();
                    float v[32];
                    tmem_ld32(trow + O_COL + g * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= factor;
                    tmem_st32(trow + O_COL + g * 32, v);
                    tmem_wait_st();
                    tc_fence_before();
                }
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) store_row32_bf16(base + PT, kTile, row, 2 * g + c2, s[c2], 1.f);
            fence_proxy_async_smem();
            mbar_arrive(B_(bars->p_full));
            if (leader) STL(6, j);
        }
        if (!mbar_wait(B_(bars->pv_done), (nkv - 1) & 1, p.err, abort_flag)) ok = false, *abort_flag = 1;
        ok = !named_bar_or(1, kMath, !ok);
        // the row sum: both groups' parts
        st_shared_f32(base + LSUM + g * kBM * 4 + row * 4, l_run);
        named_bar_sync(1, kMath);
        const float l_row = ld_shared_f32(base + LSUM + row * 4) + ld_shared_f32(base + LSUM + kBM * 4 + row * 4);
        if (ok) {   // o_lat / l -> bf16 into the (now free) q tile for the W_UV product
            tc_fence_after();
            float v[32];
            tmem_ld32(trow + O_COL + g * 32, v);
            tmem_wait_ld();
            store_row32_bf16(base + QT, kTile, row, g, v, 1.f / l_row);
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(1, kMath);
            if (leader) mbar_arrive(B_(bars->olat_ready));
            fail = !mbar_wait(B_(bars->ep_done), 0, p.err, abort_flag);
            ok = !named_bar_or(1, kMath, fail);
        }
        if (ok) {
            tc_fence_after();
            const size_t off = ((static_cast<size_t>(b) * p.T + t) * p.H + h) * p.d_v;
            for (int v16 = g; v16 < p.d_v / 16; v16 += 2) {
                float o[16];
                tmem_ld16(trow + S_COL + v16 * 16, o);
                tmem_wait_ld();
                if (t < p.T) {
                    if (p.gate) {
                        const uint4 *g4 = reinterpret_cast<const uint4 *>(p.gate + off + v16 * 16);
#pragma unroll
                        for (int q2 = 0; q2 < 2; ++q2) {
                            const uint4 gv = __ldg(g4 + q2);
                            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                o[8 * q2 + 2 * k] *=
                                    __fdividef(1.f, 1.f + fast_exp2(-__uint_as_float(gw[k] << 16) * kLog2e));
                                o[8 * q2 + 2 * k + 1] *=
                                    __fdividef(1.f, 1.f + fast_exp2(-__uint_as_float(gw[k] & 0xFFFF0000u) * kLog2e));
                            }
                        }
                    }
                    uint4 *o4 = reinterpret_cast<uint4 *>(p.out + off + v16 * 16);
                    o4[0] = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                       pack_bf16x2(o[6], o[7]));
                    o4[1] = make_uint4(pack_bf16x2(o[8], o[9]), pack_bf16x2(o[10], o[11]),
                                       pack_bf16x2(o[12], o[13]), pack_bf16x2(o[14], o[15]));
                }
            }
        }
        if (!ok) *abort_flag = 1;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
#ifdef MLA_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 4096) g_scta[1][blockIdx.x] = globaltimer_ns();
#endif
    if (warp == 1) tmem_dealloc(tmem, 256);
}

CUresult encode_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool dim_ok(int d) { return d == 16 || d == 32 || d == 48 || d == 64; }

}  // namespace

#ifdef MLA_TRACE
// Diagnostic build only: the timeline of CTA 0 ([9][64] cycles) and every CTA's [start, end, SM] ([3][4096]).
extern "C" __attribute__((visibility("default"))) int mla_debug_small_trace(long long *tl, unsigned long long *ctas) {
    if (cudaMemcpyFromSymbol(tl, g_stl, sizeof(g_stl)) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(ctas, g_scta, sizeof(g_scta)) != cudaSuccess) return -1;
    return 0;
}
#endif

bool prefill_bf16_small_supports(int r, int d_q, int d_v) { return (r == 32 || r == 64) && dim_ok(d_q) && dim_ok(d_v); }

cudaError_t launch_prefill_bf16_small(const PrefillArgs &a, cudaStream_t s) {
    if (!prefill_bf16_small_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    const cuuint64_t B = a.B, T = a.T, H = a.H, dq = a.d_q, dv = a.d_v, r = a.r;
    CUtensorMap tm_q, tm_c, tm_wuk, tm_wuv;
    {
        const cuuint64_t dims[4] = {dq, H, T, B};
        const cuuint64_t strides[3] = {dq * 2, H * dq * 2, T * H * dq * 2};
        const cuuint32_t box[4] = {64, 1, kBM, 1};
        if (encode_map(&tm_q, a.q, 4, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {r, T, B};
        const cuuint64_t strides[2] = {r * 2, T * r * 2};
        // r = 32: rows of 64 bytes, staged with 64-byte swizzle; r = 64: 128-byte rows and swizzle
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(r), kBN, 1};
        if (encode_map(&tm_c, a.c, 3, dims, strides, box,
                       r == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {r, H * dq};
        const cuuint64_t strides[1] = {r * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(dq)};
        if (encode_map(&tm_wuk, a.w_uk, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {r, H * dv};
        const cuuint64_t strides[1] = {r * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(dv)};
        if (encode_map(&tm_wuv, a.w_uv, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    Params p;
    p.gate = static_cast<const __nv_bfloat16 *>(a.gate);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.err = a.dev_err;
    p.T = a.T;
    p.H = a.H;
    p.d_q = a.d_q;
    p.d_v = a.d_v;
    p.r = a.r;
    p.n_qtiles = (a.T + kBM - 1) / kBM;
    p.bh_count = a.B * a.H;
    p.qk_scale_log2 = a.scale * kLog2e;
    cudaError_t e = cudaFuncSetAttribute(prefill_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const long long n = static_cast<long long>(p.n_qtiles) * p.bh_count;
    if (n > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    note_launch();
    prefill_small_kernel<<<static_cast<unsigned>(n), kThreads, kSmemBytes, s>>>(tm_q, tm_c, tm_wuk, tm_wuv, p);
    return cudaGetLastError();
}

}  // namespace mla
