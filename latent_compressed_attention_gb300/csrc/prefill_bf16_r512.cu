// bf16 causal absorbed Gated-MLA prefill for r = 512, d_q = d_v = 128 on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA), one fused kernel.
//
// Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）":
//   step 2  q_abs = q . W_UK (prologue), score = q_abs . c^T, causal softmax
//   step 3  o_lat = attn . c, then o = o_lat . W_UV^T (epilogue)
//   step 4  out = sigmoid(gate) * o (epilogue)
// K and V are never decompressed: the same TMA-staged latent tile c serves as
// the key operand of the score product and the value operand of the latent
// weighting.
//
// A work tile is 128 consecutive tokens of one (batch, head).  Its fp32
// latent accumulator o_lat is 128 x 512 = all 512 TMEM columns of an SM, so
// the tile runs on a cluster of two CTAs:
//   rank 0, the score CTA: absorbs W_UK into q (tcgen05, fp32 in TMEM),
//     stores q_abs * scale * log2(e) as bf16 in smem, computes S = q_abs c^T
//     per 128-key block into a double-buffered TMEM accumulator, and runs the
//     online softmax (one thread per row).  P (bf16) and per-row (rescale
//     factor, running sum) go to the value CTA by a DSMEM bulk copy.
//   rank 1, the value CTA: accumulates o_lat += P . c in TMEM (512 columns),
//     rescales o_lat when a row maximum grew (lazily: only when it grew by
//     more than 2^8), then divides by the row sum, projects with W_UV^T on
//     the tensor cores and applies the sigmoid gate.
// Each CTA loads its own c tiles (no multicast); both read them from L2.
// Every wait is bounded; a CTA that gives up records an error, stops issuing
// work and still meets its partner at the final cluster barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kR = 512;      // latent rank
constexpr int kD = 128;      // d_q = d_v
constexpr int kBM = 128;     // query tokens per tile
constexpr int kBN = 128;     // keys per block
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale row maximum until the new one exceeds it by this

constexpr uint32_t kSlab = 16384;  // [128 rows x 64 bf16] with 128-byte swizzle
// score CTA
constexpr uint32_t S_QABS = 0;                       // 8 slabs: W_UK during the absorb, then q_abs
constexpr uint32_t S_QP = 8 * kSlab;                 // 2 slabs: q tile, then the P staging tile
constexpr uint32_t S_RING = S_QP + 2 * kSlab;        // c ring
constexpr int kSStages = 4;
constexpr uint32_t S_ROWINFO = S_RING + kSStages * kSlab;
constexpr uint32_t kRowInfoBytes = kBM * 8 + 16;     // (factor, l) per row + block rescale flag
constexpr uint32_t kRowInfoStride = 1056;
// value CTA
constexpr uint32_t O_RING = 0;
constexpr int kOStages = 2;
constexpr uint32_t kOStage = 4 * kSlab;              // 256 latent columns x 128 keys
constexpr uint32_t O_P = kOStages * kOStage;         // 2 P tiles (also the epilogue's o_lat staging)
constexpr uint32_t kPBytes = 2 * kSlab;
constexpr uint32_t O_ROWINFO = O_P + 2 * kPBytes;
constexpr uint32_t BARS = S_ROWINFO + kRowInfoStride;
constexpr uint32_t kSmemBytes = BARS + 512 + 1024;   // + barriers + alignment slack

static_assert(O_ROWINFO + 2 * kRowInfoStride <= BARS, "value-CTA layout overlaps the barriers");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB shared-memory limit");

constexpr uint32_t kIdescAbsorb = make_idesc_bf16(128, 256, 0, 1);  // q (K-major) x W_UK (MN-major)
constexpr uint32_t kIdescQK = make_idesc_bf16(128, 128, 0, 0);      // q_abs (K-major) x c (K-major)
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 256, 0, 1);      // P (K-major) x c (MN-major)
constexpr uint32_t kIdescEp = make_idesc_bf16(128, 128, 0, 0);      // o_lat (K-major) x W_UV (K-major)

struct Bars {
    uint64_t pro_full, absorb_done, qabs_ready;   // score CTA
    uint64_t sc_full[kSStages], sc_empty[kSStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_free[2];                           // arrivals from the value CTA
    uint64_t oc_full[kOStages], oc_empty[kOStages];  // value CTA
    uint64_t p_full[2];                           // bulk-copy transactions from the score CTA
    uint64_t pv_done[2], ri_read[2], corr_done;
    uint64_t olat_ready[2], ep_done[2];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

struct Params {
    const __nv_bfloat16 *gate;
    __nv_bfloat16 *out;
    int *err;
    int T, H, n_qtiles, bh_count;
    float qk_scale_log2;
};

__device__ __forceinline__ void st_shared_v2f(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_r512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                        const __grid_constant__ CUtensorMap tm_wuk, const __grid_constant__ CUtensorMap tm_wuv,
                        const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    Bars *bars = reinterpret_cast<Bars *>(smem_raw + (base - raw) + BARS);
    volatile int *abort_flag = &bars->abort;
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int qt = p.n_qtiles - 1 - cluster_id / p.bh_count;   // heaviest tiles first
    const int bh = cluster_id % p.bh_count;
    const int b = bh / p.H, h = bh % p.H;
    const int t0 = qt * kBM;
    const int nkv = qt + 1;   // 128-key blocks covering keys [0, min(T, t0 + 128))

    if (threadIdx.x == 0) {
        mbar_init(B_(bars->pro_full), 1);
        mbar_init(B_(bars->absorb_done), 1);
        mbar_init(B_(bars->qabs_ready), 1);
        for (int i = 0; i < kSStages; ++i) {
            mbar_init(B_(bars->sc_full[i]), 1);
            mbar_init(B_(bars->sc_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B_(bars->s_full[i]), 1);
            mbar_init(B_(bars->s_free[i]), 128);
            mbar_init(B_(bars->p_free[i]), 1);
            mbar_init(B_(bars->p_full[i]), 1);
            mbar_init(B_(bars->pv_done[i]), 1);
            mbar_init(B_(bars->ri_read[i]), 128);
            mbar_init(B_(bars->olat_ready[i]), 1);
            mbar_init(B_(bars->ep_done[i]), 1);
        }
        for (int i = 0; i < kOStages; ++i) {
            mbar_init(B_(bars->oc_full[i]), 1);
            mbar_init(B_(bars->oc_empty[i]), 1);
        }
        mbar_init(B_(bars->corr_done), 128);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers exist before any remote arrival or copy
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (rank == 0) {
        // =========================================================== score CTA
        if (warp == 0 && lane == 0) {
            // ---- TMA producer: q tile + W_UK[h], then the c ring
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_c);
            tma_prefetch_desc(&tm_wuk);
            const uint32_t pro = B_(bars->pro_full);
            mbar_arrive_expect_tx(pro, 10 * kSlab);
            for (int s = 0; s < 2; ++s) tma_load_4d(base + S_QP + s * kSlab, &tm_q, pro, s * 64, h, t0, b);
            for (int s = 0; s < 8; ++s) tma_load_2d(base + S_QABS + s * kSlab, &tm_wuk, pro, s * 64, h * kD);
            int it = 0;
            bool ok = true;
            for (int j = 0; ok && j < nkv; ++j) {
                for (int kc = 0; kc < 8; ++kc, ++it) {
                    const int st = it % kSStages;
                    if (it >= kSStages &&
                        !(ok = mbar_wait(B_(bars->sc_empty[st]), ((it / kSStages) - 1) & 1, p.err, abort_flag)))
                        break;
                    mbar_arrive_expect_tx(B_(bars->sc_full[st]), kSlab);
                    tma_load_3d(base + S_RING + st * kSlab, &tm_c, B_(bars->sc_full[st]), kc * 64, j * kBN, b);
                }
            }
            if (!ok) *abort_flag = 1;
            // no load may still be landing when the CTA exits
            mbar_wait(pro, 0, p.err);
            for (int k = (it > kSStages ? it - kSStages : 0); k < it; ++k)
                mbar_wait(B_(bars->sc_full[k % kSStages]), (k / kSStages) & 1, p.err);
        } else if (warp == 1 && lane == 0) {
            // ---- MMA issuer: absorb, then S = q_abs . c^T per key block
            bool ok = mbar_wait(B_(bars->pro_full), 0, p.err, abort_flag);
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t a = make_smem_desc(base + S_QP + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        const uint64_t bd = make_smem_desc(base + S_QABS + nh * 4 * kSlab + kk * 2048, kSlab, 1024);
                        umma_bf16(tmem + nh * 256, a, bd, kIdescAbsorb, kk > 0);
                    }
                }
                umma_commit(B_(bars->absorb_done));
                ok = mbar_wait(B_(bars->qabs_ready), 0, p.err, abort_flag);
            }
            int it = 0;
            for (int j = 0; ok && j < nkv; ++j) {
                const int sb = j & 1;
                if (j >= 2 && !(ok = mbar_wait(B_(bars->s_free[sb]), ((j >> 1) - 1) & 1, p.err, abort_flag))) break;
                tc_fence_after();
                for (int kc = 0; kc < 8; ++kc, ++it) {
                    const int st = it % kSStages;
                    if (!(ok = mbar_wait(B_(bars->sc_full[st]), (it / kSStages) & 1, p.err, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = make_smem_desc(base + S_QABS + kc * kSlab + kk * 32, 16, 1024);
                        const uint64_t bd = make_smem_desc(base + S_RING + st * kSlab + kk * 32, 16, 1024);
                        umma_bf16(tmem + sb * kBN, a, bd, kIdescQK, (kc | kk) != 0);
                    }
                    umma_commit(B_(bars->sc_empty[st]));
                }
                if (!ok) break;
                umma_commit(B_(bars->s_full[sb]));
            }
            if (!ok) *abort_flag = 1;
        } else if (warp >= 4) {
            // ---- softmax warpgroup: thread `row` owns TMEM lane `row`
            const int row = threadIdx.x - 128;
            const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const int t = t0 + row;
            bool fail = false;
            fail = !mbar_wait(B_(bars->absorb_done), 0, p.err, abort_flag);
            bool ok = !named_bar_or(1, 128, fail);
            if (ok) {
                // q_abs (fp32, TMEM) -> q_abs * scale * log2(e) as bf16 into the q_abs tile
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < kR / 32; ++cc) {
                    float v[32];
                    tmem_ld32(trow + cc * 32, v);
                    tmem_wait_ld();
                    store_row32_bf16(base + S_QABS, kSlab, row, cc, v, p.qk_scale_log2);
                }
                fence_proxy_async_smem();
                tc_fence_before();
            }
            named_bar_sync(1, 128);
            if (row == 0 && ok) mbar_arrive(B_(bars->qabs_ready));

            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; ok && j < nkv; ++j) {
                const int sb = j & 1, pb = j & 1;
                fail = false;
                fail = !mbar_wait(B_(bars->s_full[sb]), (j >> 1) & 1, p.err, abort_flag);
                if (named_bar_or(1, 128, fail)) { ok = false; break; }
                tc_fence_after();
                float s[4][32];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(trow + sb * kBN + c4 * 32, s[c4]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(B_(bars->s_free[sb]));

                const int key0 = j * kBN;
                if (j == nkv - 1) {   // the diagonal block: mask keys after the query and past the sequence
                    const int lim = min(t, p.T - 1) - key0;   // last visible column
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c4 * 32 + i > lim) s[c4][i] = -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, s[c4][i]);
                float factor = 1.f;
                if (mx > m_run + kRescaleLog2) {
                    factor = fast_exp2(m_run - mx);
                    m_run = mx;
                }
                float sum = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[c4][i] = fast_exp2(s[c4][i] - m_run);
                        sum += s[c4][i];
                    }
                l_run = l_run * factor + sum;

                // the staging tile is free once the previous copy has read it, and the
                // value CTA's P buffer `pb` once its block j-2 product completed
                fail = false;
                if (row == 0) {
                    bulk_wait_read_all();
                    if (j >= 2) fail = !mbar_wait<true>(B_(bars->p_free[pb]), ((j >> 1) - 1) & 1, p.err, abort_flag);
                }
                if (named_bar_or(1, 128, fail)) { ok = false; break; }
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) store_row32_bf16(base + S_QP, kSlab, row, c4, s[c4], 1.f);
                st_shared_v2f(base + S_ROWINFO + row * 8, factor, l_run);
                fence_proxy_async_smem();
                const bool any = named_bar_or(1, 128, factor != 1.f);
                if (row == 0) {
                    st_shared_u32(base + S_ROWINFO + kBM * 8, any ? 1u : 0u);
                    fence_proxy_async_smem();
                    const uint32_t dst_bar = mapa_shared(B_(bars->p_full[pb]), 1);
                    bulk_copy_s2cluster(mapa_shared(base + O_P + pb * kPBytes, 1), base + S_QP, kPBytes, dst_bar);
                    bulk_copy_s2cluster(mapa_shared(base + O_ROWINFO + pb * kRowInfoStride, 1), base + S_ROWINFO,
                                        kRowInfoBytes, dst_bar);
                    bulk_commit_group();
                }
            }
            if (!ok) *abort_flag = 1;
            if (row == 0) bulk_wait_all();
        }
    } else {
        // =========================================================== value CTA
        if (warp == 0 && lane == 0) {
            // ---- TMA producer: c tiles as the MN-major value operand, then W_UV[h]
            tma_prefetch_desc(&tm_c);
            tma_prefetch_desc(&tm_wuv);
            int it = 0;
            bool ok = true;
            for (int j = 0; ok && j < nkv + 1; ++j) {   // j == nkv: the W_UV tile
                for (int nh = 0; nh < 2; ++nh, ++it) {
                    const int st = it % kOStages;
                    if (it >= kOStages &&
                        !(ok = mbar_wait(B_(bars->oc_empty[st]), ((it / kOStages) - 1) & 1, p.err, abort_flag)))
                        break;
                    const uint32_t full = B_(bars->oc_full[st]);
                    mbar_arrive_expect_tx(full, kOStage);
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint32_t dst = base + O_RING + st * kOStage + q4 * kSlab;
                        if (j < nkv)
                            tma_load_3d(dst, &tm_c, full, (nh * 4 + q4) * 64, j * kBN, b);
                        else
                            tma_load_2d(dst, &tm_wuv, full, (nh * 4 + q4) * 64, h * kD);
                    }
                }
            }
            if (!ok) *abort_flag = 1;
            for (int k = (it > kOStages ? it - kOStages : 0); k < it; ++k)
                mbar_wait(B_(bars->oc_full[k % kOStages]), (k / kOStages) & 1, p.err);
        } else if (warp == 1 && lane == 0) {
            // ---- MMA issuer: o_lat += P . c, then o = o_lat . W_UV^T
            int it = 0, ncorr = 0;
            bool ok = true;
            for (int j = 0; ok && j < nkv; ++j) {
                const int pb = j & 1;
                mbar_arrive_expect_tx(B_(bars->p_full[pb]), kPBytes + kRowInfoBytes);
                if (!(ok = mbar_wait<true>(B_(bars->p_full[pb]), (j >> 1) & 1, p.err, abort_flag))) break;
                const uint32_t flag = ld_shared_u32(base + O_ROWINFO + pb * kRowInfoStride + kBM * 8);
                if (j > 0 && flag) {
                    if (!(ok = mbar_wait(B_(bars->corr_done), ncorr & 1, p.err, abort_flag))) break;
                    ++ncorr;
                }
                tc_fence_after();
                for (int nh = 0; nh < 2; ++nh, ++it) {
                    const int st = it % kOStages;
                    if (!(ok = mbar_wait(B_(bars->oc_full[st]), (it / kOStages) & 1, p.err, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t a =
                            make_smem_desc(base + O_P + pb * kPBytes + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = make_smem_desc(base + O_RING + st * kOStage + kk * 2048, kSlab, 1024);
                        umma_bf16(tmem + nh * 256, a, bd, kIdescPV, (j > 0 || kk > 0));
                    }
                    umma_commit(B_(bars->oc_empty[st]));
                }
                if (!ok) break;
                umma_commit(B_(bars->pv_done[pb]));
            }
            for (int kh = 0; ok && kh < 2; ++kh, ++it) {
                if (!(ok = mbar_wait(B_(bars->olat_ready[kh]), 0, p.err, abort_flag))) break;
                const int st = it % kOStages;
                if (!(ok = mbar_wait(B_(bars->oc_full[st]), (it / kOStages) & 1, p.err, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t a = make_smem_desc(base + O_P + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        make_smem_desc(base + O_RING + st * kOStage + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
                    umma_bf16(tmem, a, bd, kIdescEp, (kh > 0 || kk > 0));
                }
                umma_commit(B_(bars->oc_empty[st]));
                umma_commit(B_(bars->ep_done[kh]));
            }
            if (!ok) *abort_flag = 1;
        } else if (warp == 2 && lane == 0) {
            // ---- relay: P buffer pb is free again once its product completed and its row info was read
            for (int j = 0; j < nkv; ++j) {
                const int pb = j & 1;
                if (!mbar_wait(B_(bars->pv_done[pb]), (j >> 1) & 1, p.err, abort_flag) ||
                    !mbar_wait(B_(bars->ri_read[pb]), (j >> 1) & 1, p.err, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_remote(B_(bars->p_free[pb]), 0);
            }
        } else if (warp >= 4) {
            // ---- correction + epilogue warpgroup: thread `row` owns TMEM lane `row`
            const int row = threadIdx.x - 128;
            const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const int t = t0 + row;
            float l_fin = 1.f;
            bool ok = true, fail;
            for (int j = 0; j < nkv; ++j) {
                const int pb = j & 1;
                fail = false;
                fail = !mbar_wait<true>(B_(bars->p_full[pb]), (j >> 1) & 1, p.err, abort_flag);
                if (named_bar_or(2, 128, fail)) { ok = false; break; }
                const uint32_t ri = base + O_ROWINFO + pb * kRowInfoStride;
                const float2 fl = ld_shared_v2f(ri + row * 8);
                const uint32_t flag = ld_shared_u32(ri + kBM * 8);
                mbar_arrive(B_(bars->ri_read[pb]));
                l_fin = fl.y;
                if (j > 0 && flag) {
                    fail = false;
                    fail = !mbar_wait(B_(bars->pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, p.err, abort_flag);
                    if (named_bar_or(2, 128, fail)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, fl.x != 1.f)) {
#pragma unroll 1
                        for (int cc = 0; cc < kR / 32; ++cc) {
                            float v[32];
                            tmem_ld32(trow + cc * 32, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] *= fl.x;
                            tmem_st32(trow + cc * 32, v);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    mbar_arrive(B_(bars->corr_done));
                }
            }
            if (ok) {
                fail = false;
                fail = !mbar_wait(B_(bars->pv_done[(nkv - 1) & 1]), ((nkv - 1) >> 1) & 1, p.err, abort_flag);
                ok = !named_bar_or(2, 128, fail);
            }
            const float inv_l = 1.f / l_fin;
            for (int kh = 0; ok && kh < 2; ++kh) {
                if (kh == 1) {   // the staging tile is free once the first half's product completed
                    fail = false;
                    fail = !mbar_wait(B_(bars->ep_done[0]), 0, p.err, abort_flag);
                    if (named_bar_or(2, 128, fail)) { ok = false; break; }
                }
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    float v[32];
                    tmem_ld32(trow + kh * 256 + cc * 32, v);
                    tmem_wait_ld();
                    store_row32_bf16(base + O_P, kSlab, row, cc, v, inv_l);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(2, 128);
                if (row == 0) mbar_arrive(B_(bars->olat_ready[kh]));
            }
            if (ok) {
                fail = false;
                fail = !mbar_wait(B_(bars->ep_done[1]), 0, p.err, abort_flag);
                ok = !named_bar_or(2, 128, fail);
            }
            if (ok) {
                tc_fence_after();
                float o[4][32];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(trow + c4 * 32, o[c4]);
                tmem_wait_ld();
                if (t < p.T) {
                    const size_t off = ((static_cast<size_t>(b) * p.T + t) * p.H + h) * kD;
                    const uint4 *g4 = p.gate ? reinterpret_cast<const uint4 *>(p.gate + off) : nullptr;
                    uint4 *o4 = reinterpret_cast<uint4 *>(p.out + off);
#pragma unroll
                    for (int v8 = 0; v8 < kD / 8; ++v8) {
                        float y[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) y[i] = o[(v8 * 8 + i) >> 5][(v8 * 8 + i) & 31];
                        if (g4) {
                            const uint4 gv = __ldg(g4 + v8);
                            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float g_lo = __uint_as_float(gw[i] << 16);
                                const float g_hi = __uint_as_float(gw[i] & 0xFFFF0000u);
                                y[2 * i] *= __fdividef(1.f, 1.f + fast_exp2(-g_lo * kLog2e));
                                y[2 * i + 1] *= __fdividef(1.f, 1.f + fast_exp2(-g_hi * kLog2e));
                            }
                        }
                        o4[v8] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                            pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                    }
                }
            }
            if (!ok) *abort_flag = 1;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster_sync_all();   // the partner no longer touches this CTA's shared memory
}

CUresult encode_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool prefill_bf16_r512_supports(int r, int d_q, int d_v) { return r == kR && d_q == kD && d_v == kD; }

cudaError_t launch_prefill_bf16_r512(const PrefillArgs &a, cudaStream_t s) {
    if (!prefill_bf16_r512_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    const cuuint64_t B = a.B, T = a.T, H = a.H;
    CUtensorMap tm_q, tm_c, tm_wuk, tm_wuv;
    {
        const cuuint64_t dims[4] = {kD, H, T, B};
        const cuuint64_t strides[3] = {kD * 2, H * kD * 2, T * H * kD * 2};
        const cuuint32_t box[4] = {64, 1, kBM, 1};
        if (encode_map(&tm_q, a.q, 4, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {kR, T, B};
        const cuuint64_t strides[2] = {kR * 2, T * kR * 2};
        const cuuint32_t box[3] = {64, kBN, 1};
        if (encode_map(&tm_c, a.c, 3, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {kR, H * kD};
        const cuuint64_t strides[1] = {kR * 2};
        const cuuint32_t box[2] = {64, kD};
        if (encode_map(&tm_wuk, a.w_uk, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
        if (encode_map(&tm_wuv, a.w_uv, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    Params p;
    p.gate = static_cast<const __nv_bfloat16 *>(a.gate);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.err = a.dev_err;
    p.T = a.T;
    p.H = a.H;
    p.n_qtiles = (a.T + kBM - 1) / kBM;
    p.bh_count = a.B * a.H;
    p.qk_scale_log2 = a.scale * kLog2e;
    cudaError_t e = cudaFuncSetAttribute(prefill_r512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const long long n_ctas = 2LL * p.n_qtiles * p.bh_count;
    if (n_ctas > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    prefill_r512_kernel<<<static_cast<unsigned>(n_ctas), kThreads, kSmemBytes, s>>>(tm_q, tm_c, tm_wuk, tm_wuv, p);
    return cudaGetLastError();
}

}  // namespace mla
