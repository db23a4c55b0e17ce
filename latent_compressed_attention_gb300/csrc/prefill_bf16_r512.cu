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
//   rank 0, the score CTA: absorbs W_UK into q (tcgen05, fp32 in TMEM), packs
//     q_abs * scale * log2(e) as f16 into TMEM columns 0-255, where it is the
//     A operand of S = q_abs c^T against an f16 copy of c (times a power of two
//     per sequence); S sits in columns 256-511.
//     Two warpgroups run the online softmax (64 columns of each row each; the
//     row maximum is exchanged through smem).  P (bf16) and per-row (rescale
//     factor, partial sums) are staged in double-buffered smem and shipped to
//     the value CTA by asynchronous DSMEM bulk copies.
//   rank 1, the value CTA: accumulates o_lat += P . c in TMEM (512 columns),
//     rescales o_lat when a row maximum grew (lazily: only when it grew by
//     more than 2^16), then divides by the row sum, packing o_lat/l as bf16 in
//     place in TMEM, where it is the A operand of the W_UV^T product, and
//     applies the sigmoid gate.
// Each CTA loads its own c tiles (no multicast); both read them from L2.
//
// Precision of the score: a bf16 operand (8 significant bits) would put a
// relative error of 2^-9 on every score, a few percent of the softmax weights
// once scores spread over ~25 natural-log units.  The score product therefore
// runs in f16 (11 significant bits) on both sides: latent_amax_kernel and
// latent_f16_kernel convert c once per call into the workspace, each sequence
// scaled by the power of two that brings its largest |c| into [2^13, 2^14);
// f16 keeps 11 significant bits between 2^-14 and 2^15, so the score CTA
// packs the query operand unscaled and only a row whose largest element is
// outside [2^-10, 2^15) (recomputed on a rare slow path) gets a power of two.  The powers of two are folded back
// into the softmax's one FMA per score (exp2(s * F - m)): exact and free.  The value product keeps the bf16 latent and bf16 weights P.
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
constexpr int kBN = 128;     // keys per value-CTA unit
constexpr int kBS = 256;     // keys per score block (two units)
constexpr int kThreads = 384;   // warps 0 TMA, 1 MMA, 2 relay (value CTA), 4-7 and 8-11: two row warpgroups
// Register split: the control warpgroup (warps 0-3) gives registers to the two row warpgroups.
// 4 x 32 x 72 + 8 x 32 x 208 = 62,464 <= 384 x 168 launched; the launcher checks the kernel's count.
#ifndef MLA_TRACE
constexpr uint32_t kRegsCtl = 72, kRegsMath = 208, kRegsLaunch = 168;
#else   // the wait accounting needs more registers in the control warps
constexpr uint32_t kRegsCtl = 88, kRegsMath = 200, kRegsLaunch = 168;
#endif
static_assert(128 * kRegsCtl + 256 * kRegsMath <= kThreads * kRegsLaunch, "register split exceeds the launch");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Keep a stale row maximum until the new one exceeds it by this (log2 units):
// p <= 2^16, far inside the fp32 range of the row sums and the accumulator.
constexpr float kRescaleLog2 = 16.0f;
// Range of a row's largest |x| in which the score operand is packed as f16 directly: below 2^15 nothing
// overflows, and from 2^-10 up the large elements keep f16's 11 significant bits (the elements that fall into
// f16's subnormals are 2^-4 or less of the largest and err by 2^-25 at most).  A row outside it (other than an
// all-zero row) is recomputed times a power of two.
constexpr float kF16Limit = 32768.0f, kF16Floor = 0.0009765625f;

constexpr uint32_t kSlab = 16384;  // [128 rows x 64 bf16] with 128-byte swizzle
// score CTA
constexpr uint32_t kSStage = 2 * kSlab;              // c ring stage: [256 keys x 64 latent columns]
constexpr uint32_t S_RING = 0;                       // W_UK fills the ring for the absorb
constexpr int kSStages = 4;
constexpr uint32_t kPBytes = 2 * kSlab;              // one unit of P: [128 rows x 128 keys]
constexpr uint32_t kRowInfoBytes = kBM * 8;          // {rescale factor, running sum} per row
constexpr uint32_t kPUnit = kPBytes + kRowInfoBytes; // staging per warpgroup (the first also holds the q tile)
constexpr uint32_t S_PST = S_RING + kSStages * kSStage;
// value CTA
constexpr uint32_t O_RING = 0;
constexpr int kOStages = 2;
constexpr uint32_t kOStage = 4 * kSlab;              // 256 latent columns x 128 keys
constexpr uint32_t O_P = kOStages * kOStage;         // 2 P tiles
constexpr uint32_t O_ROWINFO = O_P + 2 * kPBytes;    // 2 row-info blocks
constexpr uint32_t BARS = S_PST + 2 * kPUnit;
constexpr uint32_t PMAX = BARS + 512;                // [2 parities][2 warpgroups][128 rows] partial maxima
constexpr uint32_t QMAX = PMAX + 2 * 2 * kBM * 4;    // [2 warpgroups][128 rows] half-row maxima of |x|
constexpr uint32_t LSUM = QMAX + 2 * kBM * 4;        // [128 rows] the second warpgroup's row sums at a tile's end
constexpr uint32_t kSmemUsed = LSUM + kBM * 4;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;    // + alignment slack
// TMEM columns of the score CTA
constexpr uint32_t S_QCOL = 0;     // packed f16 q_abs: K step ks (16 latent columns) at columns 8 ks .. 8 ks + 7
constexpr uint32_t S_SCOL = 256;   // S for one 256-key block
static_assert(O_ROWINFO + 2 * kRowInfoBytes <= BARS, "value-CTA layout overlaps the barriers");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB shared-memory limit");
static_assert(S_PST % 1024 == 0 && (S_PST + kPUnit) % 1024 == 0 && O_P % 1024 == 0, "alignment");

constexpr uint32_t kIdescAbsorb = make_idesc_bf16(128, 256, 0, 1);  // q (K-major) x W_UK (MN-major)
constexpr uint32_t kIdescQK = make_idesc_f16(128, 256, 0, 0);       // f16 q_abs (TMEM) x f16 c (K-major), 256 keys
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 256, 0, 1);      // P (K-major) x c (MN-major)
constexpr uint32_t kIdescEp = make_idesc_bf16(128, 128, 0, 0);      // o_lat/l (TMEM) x W_UV (K-major)
// TMEM columns of the value CTA in the epilogue: o_lat/l packed as bf16 pairs in place, latent columns
// 0-255 into columns 0-127 and 256-511 into columns 384-511 (K step ks of 16 latent columns at
// ep_acol(ks)); the product o = (o_lat/l) . W_UV^T lands in columns 128-255.
__device__ __forceinline__ uint32_t ep_acol(int ks) { return ks < 16 ? 8 * ks : 384 + 8 * (ks - 16); }
constexpr uint32_t O_EPCOL = 128;

struct Bars {
    uint64_t pro_full, absorb_done, qabs_ready, q_free;   // score CTA
    uint64_t sc_full[kSStages], sc_empty[kSStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_free[2];                           // arrivals from the value CTA
    uint64_t oc_full[kOStages], oc_empty[kOStages];  // value CTA
    uint64_t p_full[2];                           // bulk-copy transactions from the score CTA
    uint64_t pv_done[2], ri_read[2], corr_done;
    uint64_t olat_ready, ep_done, ep_read;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

// Opt-in wait accounting (build with MLA_NVCC_FLAGS=-DMLA_TRACE): cycles each
// role spends at its waits and in its loop, summed over all CTAs.
enum TraceSlot {
    TR_S_MMA_LOOP, TR_S_MMA_SFREE, TR_S_MMA_SCFULL, TR_S_SM_LOOP, TR_S_SM_SFULL, TR_S_SM_XBAR, TR_S_SM_PFREE,
    TR_S_SM_STORE, TR_O_MMA_LOOP, TR_O_MMA_PFULL, TR_O_MMA_OCFULL, TR_O_MMA_CORR, TR_O_COR_LOOP, TR_S_PROD_EMPTY,
    TR_O_PROD_EMPTY, TR_TILES, TR_BLOCKS, TR_CORRECTIONS, TR_S_PROLOGUE, TR_O_EPILOGUE, TR_S_TOTAL, TR_O_TOTAL,
    TR_S_SM_RELEASE, TR_O_EP_PACK, TR_O_EP_WAIT, TR_O_EP_OUT, TR_COUNT
};
#ifdef MLA_TRACE
__device__ unsigned long long g_trace[TR_COUNT];
#define TR(...) __VA_ARGS__
#define TR_ADD(slot, v) atomicAdd(&g_trace[slot], static_cast<unsigned long long>(v))
// Per-block event times (cycles since the start barrier) of cluster 0's first tile (the heaviest).
constexpr int kTLMax = 128, kTLEvents = 12;
__device__ long long g_ptl[kTLEvents][kTLMax];
#define TL(ev, idx, val) \
    do { if (static_cast<int>(idx) < kTLMax) g_ptl[ev][idx] = (val); } while (0)
#else
#define TR(...)
#define TR_ADD(slot, v) (void)0
#endif

struct Params {
    const __nv_bfloat16 *gate;
    __nv_bfloat16 *out;
    const float *sscale;   // [B]: 2^-e_b, the scale of sequence b's f16 latent copy
    const __nv_bfloat16 *w_uk;   // [H, d_q, r], read only by the rare recompute of a row beyond f16's range
    float *lse;                  // optional [B, H, T]: each row's log-sum-exp of the scaled scores (natural log)
    int *err;
    int T, H, n_qtiles, bh_count;
    int n_tiles;   // n_qtiles * bh_count work tiles, numbered heaviest first
    int G;         // clusters of the persistent grid
    float qk_scale_log2;
};

// Work tile `tile` (heaviest first): 128 query tokens of one (batch, head) and the key blocks they see.
struct TileInfo {
    int b, h, t0;
    int nblk;   // 256-key score blocks covering keys [0, min(T, t0 + 128))
    int nkv;    // 128-key value units (the last may be entirely masked)
};
__device__ __forceinline__ TileInfo tile_info(int tile, const Params &p) {
    const int qt = p.n_qtiles - 1 - tile / p.bh_count;
    const int bh = tile % p.bh_count;
    TileInfo ti;
    ti.b = bh / p.H;
    ti.h = bh % p.H;
    ti.t0 = qt * kBM;
    ti.nblk = (qt + 2) / 2;
    ti.nkv = 2 * ti.nblk;
    return ti;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_shared_bf16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_v2f(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// Pairwise (tree) reductions over 64 values: short dependency chains.
__device__ __forceinline__ float tree_max128(const float (&s)[4][32]) {
    float m[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) m[i] = fmaxf(fmaxf(s[0][i], s[1][i]), fmaxf(s[2][i], s[3][i]));
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}
__device__ __forceinline__ float tree_sum128(const float (&s)[4][32]) {
    float m[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) m[i] = (s[0][i] + s[1][i]) + (s[2][i] + s[3][i]);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] += m[i + w];
    return m[0];
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_r512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                        const __grid_constant__ CUtensorMap tm_c256, const __grid_constant__ CUtensorMap tm_wuk,
                        const __grid_constant__ CUtensorMap tm_wuv, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    Bars *bars = reinterpret_cast<Bars *>(smem_raw + (base - raw) + BARS);
    volatile int *abort_flag = &bars->abort;
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cl = static_cast<int>(blockIdx.x >> 1);   // this cluster; it walks the tiles of tile_of(k)
    // Tile k of this cluster: a snake over the heavy-first tile order, so every cluster's work adds up the same.
    auto tile_of = [&](int k) { return k * p.G + ((k & 1) ? p.G - 1 - cl : cl); };

    if (threadIdx.x == 0) {
        mbar_init(B_(bars->pro_full), 1);
        mbar_init(B_(bars->absorb_done), 1);
        mbar_init(B_(bars->qabs_ready), 1);
        mbar_init(B_(bars->q_free), 1);
        for (int i = 0; i < kSStages; ++i) {
            mbar_init(B_(bars->sc_full[i]), 1);
            mbar_init(B_(bars->sc_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B_(bars->s_full[i]), 1);
            mbar_init(B_(bars->s_free[i]), 256);
            mbar_init(B_(bars->p_free[i]), 1);
            mbar_init(B_(bars->p_full[i]), 1);   // the value CTA's expect-tx arrival
            mbar_init(B_(bars->pv_done[i]), 1);
            mbar_init(B_(bars->ri_read[i]), 256);
        }
        for (int i = 0; i < kOStages; ++i) {
            mbar_init(B_(bars->oc_full[i]), 1);
            mbar_init(B_(bars->oc_empty[i]), 1);
        }
        mbar_init(B_(bars->corr_done), 256);
        mbar_init(B_(bars->olat_ready), 1);
        mbar_init(B_(bars->ep_done), 1);
        mbar_init(B_(bars->ep_read), 256);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers exist before any remote arrival or store
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    TR(const long long t_start = clock64();)
    if (warp < 4) {
        regs_release<kRegsCtl>();   // warpgroup-uniform
        if (rank == 0) {
            // =========================================================== score CTA: control
            if (warp == 0 && lane == 0) {
                // ---- ring producer.  Per tile: W_UK[h] into four ring positions, then c tiles [256 keys x 64] for
                // every score block, streaming on into the next tile as slots free up.  A tile takes 4 + 8 nblk
                // ring positions, a multiple of the 4 stages, so W_UK always fills slots 0-3 in order.  (One
                // [256 x 64] load per position: one thread issues them fast enough.)
                tma_prefetch_desc(&tm_c256);
                tma_prefetch_desc(&tm_wuk);
                int it = 0, k = 0;
                bool ok = true, converted = false;
                for (; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    const int n_pos = 4 + 8 * ti.nblk;
                    for (int i = 0; i < n_pos; ++i, ++it) {
                        const int st = it % kSStages;
                        TR(const long long _a = clock64();)
                        if (it >= kSStages &&
                            !(ok = mbar_wait(B_(bars->sc_empty[st]), ((it / kSStages) - 1) & 1, p.err, abort_flag)))
                            break;
                        TR(TR_ADD(TR_S_PROD_EMPTY, clock64() - _a);)
                        const uint32_t full = B_(bars->sc_full[st]);
                        mbar_arrive_expect_tx(full, kSStage);
                        if (i < 4) {
                            for (int s = 0; s < 2; ++s)
                                tma_load_2d(base + S_RING + st * kSStage + s * kSlab, &tm_wuk, full, (2 * i + s) * 64,
                                            ti.h * kD);
                        } else {
                            if (!converted) {   // launched as a dependent of the latent's conversion: its copy
                                grid_dependency_wait();   // is complete and visible only after this
                                converted = true;
                            }
                            const int q = i - 4;
                            tma_load_3d(base + S_RING + st * kSStage, &tm_c256, full, (q & 7) * 64, (q >> 3) * kBS, ti.b);
                        }
                    }
                }
                if (!ok) *abort_flag = 1;
                // no load may still be landing when the CTA exits
                for (int q = (it > kSStages ? it - kSStages : 0); q < it; ++q)
                    mbar_wait(B_(bars->sc_full[q % kSStages]), (q / kSStages) & 1, p.err);
            } else if (warp == 2 && lane == 0) {
                // ---- q producer: each tile's q tile into the first P staging buffer, once the previous tile's last
                // P copy has read it (apart from the ring, so the ring streams across tile boundaries)
                tma_prefetch_desc(&tm_q);
                const uint32_t pro = B_(bars->pro_full);
                int k = 0;
                bool ok = true;
                for (; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    if (k >= 1 && !(ok = mbar_wait(B_(bars->q_free), (k - 1) & 1, p.err, abort_flag))) break;
                    mbar_arrive_expect_tx(pro, 2 * kSlab);
                    for (int s = 0; s < 2; ++s) tma_load_4d(base + S_PST + s * kSlab, &tm_q, pro, s * 64, ti.h, ti.t0, ti.b);
                }
                if (!ok) *abort_flag = 1;
                if (k > 0) mbar_wait(pro, (k - 1) & 1, p.err);   // no load may still be landing when the CTA exits
            } else if (warp == 1 && lane == 0) {
                // ---- MMA issuer: per tile the absorb, then S = q_abs . c^T per 256-key block (q_abs from TMEM)
                int it = 0, gb = 0;   // ring positions consumed, score blocks issued (all tiles)
                bool ok = true;
                TR(long long tl0 = clock64(), w_free = 0, w_full = 0;)
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    TR(const bool tl_on = cl == 0 && k == 0;)
                    ok = mbar_wait(B_(bars->pro_full), k & 1, p.err, abort_flag);
                    for (int i = 0; ok && i < 4; ++i)
                        ok = mbar_wait(B_(bars->sc_full[(it + i) % kSStages]), ((it + i) / kSStages) & 1, p.err, abort_flag);
                    // the absorb writes all 512 TMEM columns: the previous tile's last S must have been read
                    if (ok && gb >= 1) ok = mbar_wait(B_(bars->s_free[0]), (gb - 1) & 1, p.err, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    {
                        const uint64_t aq = make_smem_desc(base + S_PST, 16, 1024);
                        const uint64_t bw = make_smem_desc(base + S_RING, kSlab, 1024);
    #pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t a = desc_add(aq, (kk >> 2) * kSlab + (kk & 3) * 32);
    #pragma unroll
                            for (int nh = 0; nh < 2; ++nh)
                                umma_bf16(tmem + nh * 256, a, desc_add(bw, nh * 2 * kSStage + kk * 2048), kIdescAbsorb,
                                          kk > 0);
                        }
                    }
                    umma_commit(B_(bars->absorb_done));
                    for (int i = 0; i < 4; ++i, ++it) umma_commit(B_(bars->sc_empty[it % kSStages]));   // W_UK's slots
                    if (!(ok = mbar_wait(B_(bars->qabs_ready), k & 1, p.err, abort_flag))) break;
                    for (int j = 0; ok && j < ti.nblk; ++j, ++gb) {
                        TR(long long _a = clock64();)
                        if (j >= 1 && !(ok = mbar_wait(B_(bars->s_free[0]), (gb - 1) & 1, p.err, abort_flag))) break;
                        TR(w_free += clock64() - _a; if (tl_on) TL(0, j, clock64() - t_start); long long w_blk = 0;)
                        tc_fence_after();
                        for (int kc = 0; kc < 8; ++kc, ++it) {
                            const int st = it % kSStages;
                            TR(long long _b = clock64();)
                            if (!(ok = mbar_wait(B_(bars->sc_full[st]), (it / kSStages) & 1, p.err, abort_flag))) break;
                            TR(w_full += clock64() - _b; w_blk += clock64() - _b;)
                            tc_fence_after();
                            const uint64_t b0 = make_smem_desc(base + S_RING + st * kSStage, 16, 1024);
                            const uint32_t a0 = tmem + S_QCOL + kc * 32;
    #pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_bf16_tmem_a(tmem + S_SCOL, a0 + kk * 8, desc_add(b0, kk * 32), kIdescQK, (kc | kk) != 0);
                            umma_commit(B_(bars->sc_empty[st]));
                        }
                        if (!ok) break;
                        umma_commit(B_(bars->s_full[0]));
                        TR(if (tl_on) { TL(1, j, clock64() - t_start); TL(7, j, w_blk); })
                    }
                }
                TR(TR_ADD(TR_S_MMA_LOOP, clock64() - tl0); TR_ADD(TR_S_MMA_SFREE, w_free); TR_ADD(TR_S_MMA_SCFULL, w_full);)
                if (!ok) *abort_flag = 1;
            }
        } else {
            // =========================================================== value CTA: control
            if ((warp == 0 || warp == 3) && lane == 0) {
                // ---- TMA producers (warps 0 and 3, on alternate ring positions: a position is four [128 x 64] loads,
                // more than one thread issues in the products' time): per tile, c tiles as the MN-major value
                // operand for every unit, then W_UV[h]
                const int pi = warp == 3 ? 1 : 0;
                if (pi == 0) {
                    tma_prefetch_desc(&tm_c);
                    tma_prefetch_desc(&tm_wuv);
                }
                int it = 0;
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    for (int j = 0; ok && j < ti.nkv + 1; ++j) {   // j == nkv: the W_UV tile
                        for (int nh = 0; nh < 2; ++nh, ++it) {
                            if ((it & 1) != pi) continue;
                            const int st = it % kOStages;
                            TR(const long long _a = clock64();)
                            if (it >= kOStages &&
                                !(ok = mbar_wait(B_(bars->oc_empty[st]), ((it / kOStages) - 1) & 1, p.err, abort_flag)))
                                break;
                            TR(TR_ADD(TR_O_PROD_EMPTY, clock64() - _a);)
                            const uint32_t full = B_(bars->oc_full[st]);
                            mbar_arrive_expect_tx(full, kOStage);
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const uint32_t dst = base + O_RING + st * kOStage + q4 * kSlab;
                                if (j < ti.nkv)
                                    tma_load_3d(dst, &tm_c, full, (nh * 4 + q4) * 64, j * kBN, ti.b);
                                else
                                    tma_load_2d(dst, &tm_wuv, full, (nh * 4 + q4) * 64, ti.h * kD);
                            }
                        }
                    }
                }
                if (!ok) *abort_flag = 1;
                for (int q = (it > kOStages ? it - kOStages : 0); q < it; ++q)
                    if ((q & 1) == pi) mbar_wait(B_(bars->oc_full[q % kOStages]), (q / kOStages) & 1, p.err);
            } else if (warp == 1) {
                // ---- MMA warp: per tile o_lat += P . c, then o = o_lat . W_UV^T; lane 0 issues
                const bool leader = lane == 0;
                auto wait_all = [&](uint64_t &bar, uint32_t parity, bool cluster) {
                    return __all_sync(0xffffffffu, cluster ? mbar_wait<true>(B_(bar), parity, p.err, abort_flag)
                                                           : mbar_wait(B_(bar), parity, p.err, abort_flag));
                };
                int it = 0, ncorr = 0, gu = 0;   // ring positions, corrections, units (all tiles)
                bool ok = true;
                TR(long long tl0 = clock64(), w_pfull = 0, w_oc = 0, w_corr = 0;)
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    TR(const bool tl_on = cl == 0 && k == 0;)
                    // o_lat's TMEM columns are free once the previous tile's epilogue has read its output
                    if (k >= 1 && !(ok = wait_all(bars->ep_read, (k - 1) & 1, false))) break;
                    for (int j = 0; ok && j < ti.nkv; ++j, ++gu) {
                        const int pb = gu & 1;
                        TR(long long _a = clock64();)
                        if (leader) mbar_arrive_expect_tx(B_(bars->p_full[pb]), kPBytes + kRowInfoBytes);
                        if (!(ok = wait_all(bars->p_full[pb], (gu >> 1) & 1, true))) break;
                        TR(w_pfull += clock64() - _a; if (leader && tl_on) TL(8, j, clock64() - t_start); long long w_u = 0;)
                        // any row whose maximum grew needs o_lat rescaled before this unit's product
                        const uint32_t rinfo = base + O_ROWINFO + pb * kRowInfoBytes;
                        bool grew = false;
    #pragma unroll
                        for (int q = 0; q < 4; ++q) grew |= ld_shared_f32(rinfo + (lane + 32 * q) * 8) != 1.f;
                        if (j > 0 && __any_sync(0xffffffffu, grew)) {
                            TR(long long _c = clock64();)
                            if (!(ok = wait_all(bars->corr_done, ncorr & 1, false))) break;
                            TR(w_corr += clock64() - _c;)
                            ++ncorr;
                        }
                        tc_fence_after();
                        for (int nh = 0; nh < 2; ++nh, ++it) {
                            const int st = it % kOStages;
                            TR(long long _o = clock64();)
                            if (!(ok = wait_all(bars->oc_full[st], (it / kOStages) & 1, false))) break;
                            TR(w_oc += clock64() - _o; w_u += clock64() - _o;)
                            tc_fence_after();
                            if (leader) {
                                const uint64_t a0 = make_smem_desc(base + O_P + pb * kPBytes, 16, 1024);
                                const uint64_t b0 = make_smem_desc(base + O_RING + st * kOStage, kSlab, 1024);
    #pragma unroll
                                for (int kk = 0; kk < kBN / 16; ++kk)
                                    umma_bf16(tmem + nh * 256, desc_add(a0, (kk >> 2) * kSlab + (kk & 3) * 32),
                                              desc_add(b0, kk * 2048), kIdescPV, (j > 0 || kk > 0));
                                umma_commit(B_(bars->oc_empty[st]));
                            }
                            __syncwarp();
                        }
                        if (!ok) break;
                        if (leader) umma_commit(B_(bars->pv_done[pb]));
                        TR(if (leader && tl_on) { TL(9, j, clock64() - t_start); TL(10, j, w_u); })
                    }
                    // the epilogue: o = (o_lat/l) . W_UV^T with A from TMEM (packed in place by the correction
                    // warpgroups) and W_UV[h] in the ring's next two stages
                    if (ok) ok = wait_all(bars->olat_ready, k & 1, false);
                    for (int kh = 0; ok && kh < 2; ++kh, ++it) {
                        const int st = it % kOStages;
                        if (!(ok = wait_all(bars->oc_full[st], (it / kOStages) & 1, false))) break;
                        tc_fence_after();
                        if (leader) {
                            const uint64_t b0 = make_smem_desc(base + O_RING + st * kOStage, 16, 1024);
    #pragma unroll
                            for (int kk = 0; kk < 16; ++kk)
                                umma_bf16_tmem_a(tmem + O_EPCOL, tmem + ep_acol(kh * 16 + kk),
                                                 desc_add(b0, (kk >> 2) * kSlab + (kk & 3) * 32), kIdescEp, (kh > 0 || kk > 0));
                            umma_commit(B_(bars->oc_empty[st]));
                            if (kh == 1) umma_commit(B_(bars->ep_done));
                        }
                        __syncwarp();
                    }
                }
                TR(if (leader) {
                    TR_ADD(TR_O_MMA_LOOP, clock64() - tl0); TR_ADD(TR_O_MMA_PFULL, w_pfull); TR_ADD(TR_O_MMA_OCFULL, w_oc);
                    TR_ADD(TR_O_MMA_CORR, w_corr); TR_ADD(TR_CORRECTIONS, ncorr);
                })
                if (!ok && leader) *abort_flag = 1;
            } else if (warp == 2 && lane == 0) {
                // ---- relay: P buffer pb is free again once its product completed and its row info was read
                int gu = 0;
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    for (int j = 0; j < ti.nkv; ++j, ++gu) {
                        const int pb = gu & 1;
                        if (!mbar_wait(B_(bars->pv_done[pb]), (gu >> 1) & 1, p.err, abort_flag) ||
                            !mbar_wait(B_(bars->ri_read[pb]), (gu >> 1) & 1, p.err, abort_flag)) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(B_(bars->p_free[pb]), 0);
                    }
                }
            }
        }
    } else {
        regs_acquire<kRegsMath>();
        if (rank == 0) {
            // =========================================================== score CTA: softmax
                // ---- softmax: warpgroup `wg` owns keys [128 wg, 128 wg + 128) of each 256-key block, i.e. the
                // value CTA's unit 2j + wg; thread `row` owns TMEM lane `row`
                const int wg = (warp - 4) >> 2;
                const int row = (warp & 3) * 32 + lane;
                const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
                const bool issuer = (threadIdx.x & 127) == 0;   // issues this warpgroup's bulk copies
                const uint32_t ptile = base + S_PST + wg * kPUnit;   // this warpgroup's staging unit
                const uint32_t ri = ptile + kPBytes;
                int gb = 0, nu = 0;   // score blocks (all tiles), units this warpgroup has sent
                bool ok = true, fail = false;
                TR(long long tl0 = clock64(), w_sfull = 0, w_xbar = 0, w_pfree = 0, w_store = 0, w_rel = 0;)
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    TR(const bool tl_on = cl == 0 && k == 0;)
                    const int t = ti.t0 + row;
                    fail = fail || !mbar_wait(B_(bars->absorb_done), k & 1, p.err, abort_flag);
                    if (named_bar_or(1, 256, fail)) { ok = false; break; }
                    // the score operand x = q_abs * scale * log2(e) is packed as f16 pairs by warpgroup 0: chunk kc
                    // (fp32 columns 64kc .. 64kc+63) lands in columns 32kc .. 32kc+31, which this thread has already
                    // read, so the compaction is in place, chunk by chunk in increasing order.  The thread tracks
                    // its row's largest |x|; a row whose largest |x| is outside [2^-10, 2^15) is recomputed below.
                    tc_fence_after();
                    uint32_t hmax = 0;   // the two halves' largest |f16| bit patterns
                    if (wg == 0) {
    #pragma unroll 1
                        for (int kc = 0; kc < kR / 64; ++kc) {
                            float v[2][32], w[32];
                            tmem_ld32(trow + kc * 64, v[0]);
                            tmem_ld32(trow + kc * 64 + 32, v[1]);
                            tmem_wait_ld();
    #pragma unroll
                            for (int q = 0; q < 32; ++q) {
                                const uint32_t h2 = pack_f16x2(v[q >> 4][2 * (q & 15)] * p.qk_scale_log2,
                                                               v[q >> 4][2 * (q & 15) + 1] * p.qk_scale_log2);
                                hmax = __vmaxu2(hmax, h2 & 0x7FFF7FFFu);   // |f16| bit patterns order as magnitudes
                                w[q] = __uint_as_float(h2);
                            }
                            tmem_st32(trow + S_QCOL + kc * 32, w);
                            tmem_wait_st();
                        }
                    }
                    // largest |x| as f16: 0x7800 = 2^15 (0x7C00 and up: the packing overflowed), 0x1400 = 2^-10
                    const uint32_t hm = max(hmax & 0xFFFFu, hmax >> 16);
                    const float amax = hm >= 0x7800u ? kF16Limit : (hm == 0u ? 0.f : (hm < 0x1400u ? kF16Floor * 0.5f : 1.f));
                    tc_fence_before();
                    int e_row = 0;
                    if (named_bar_or(1, 256, amax >= kF16Limit || (amax > 0.f && amax < kF16Floor))) {
                        // rare: some row's largest |x| is outside [2^-10, 2^15).  Every warp recomputes its rows' x
                        // from the q tile and W_UK (fp32 SIMT) in two passes over this warpgroup's half of the row:
                        // the largest |x| (both halves through shared memory), then x * 2^e_row (e_row = 0 for rows
                        // inside the range) packed into this half's columns (tcgen05.st is warp-collective)
                        const __nv_bfloat16 *wk = p.w_uk + static_cast<size_t>(ti.h) * kD * kR + wg * 256;
                        float xm = 0.f;
    #pragma unroll 1
                        for (int pass = 0; pass < 2; ++pass) {
                            const float up = exp2_int(e_row);
    #pragma unroll 1
                            for (int jb = 0; jb < 8; ++jb) {
                                float acc[32];
    #pragma unroll
                                for (int q = 0; q < 32; ++q) acc[q] = 0.f;
    #pragma unroll 1
                                for (int d = 0; d < kD; ++d) {
                                    const uint32_t qa = base + S_PST + (d >> 6) * kSlab + sw128_offset(row, (d & 63) >> 3) +
                                                        (d & 7) * 2;
                                    const float qd = ld_shared_bf16(qa);
                                    const uint4 *w4 = reinterpret_cast<const uint4 *>(wk + static_cast<size_t>(d) * kR + jb * 32);
    #pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        const uint4 wv = __ldg(w4 + u);
                                        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    #pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            acc[u * 8 + 2 * e] = fmaf(qd, __uint_as_float(ww[e] << 16), acc[u * 8 + 2 * e]);
                                            acc[u * 8 + 2 * e + 1] =
                                                fmaf(qd, __uint_as_float(ww[e] & 0xFFFF0000u), acc[u * 8 + 2 * e + 1]);
                                        }
                                    }
                                }
                                if (pass == 0) {
    #pragma unroll
                                    for (int q = 0; q < 32; ++q) xm = fmaxf(xm, fabsf(acc[q] * p.qk_scale_log2));
                                    continue;
                                }
                                float pk[16];
    #pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    pk[q] = __uint_as_float(pack_f16x2((acc[2 * q] * p.qk_scale_log2) * up,
                                                                       (acc[2 * q + 1] * p.qk_scale_log2) * up));
                                tc_fence_after();
                                tmem_st16(trow + S_QCOL + wg * 128 + jb * 16, pk);
                            }
                            if (pass == 0) {
                                st_shared_f32(base + QMAX + wg * kBM * 4 + row * 4, xm);
                                named_bar_sync(1, 256);
                                const float xmax = fmaxf(ld_shared_f32(base + QMAX + row * 4),
                                                         ld_shared_f32(base + QMAX + kBM * 4 + row * 4));
                                e_row = (xmax >= kF16Limit || xmax < kF16Floor) ? f16_range_exponent(xmax) : 0;
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        named_bar_sync(1, 256);
                    }
                    // the score in log2 units is the product times F = 2^-e_row * 2^-e_b (the latent copy's scale)
                    if (k == 0) grid_dependency_wait();   // the conversion's sequence scale
                    const float F = exp2_int(-e_row) * __ldg(p.sscale + ti.b);
                    if (threadIdx.x == 128) mbar_arrive(B_(bars->qabs_ready));
                    TR(if (threadIdx.x == 128) { TR_ADD(TR_S_PROLOGUE, clock64() - t_start); TR_ADD(TR_TILES, 1);
                                                 TR_ADD(TR_BLOCKS, ti.nkv); })

                    float m_run = -INFINITY, l_part = 0.f;
                    for (int j = 0; j < ti.nblk; ++j, ++gb) {
                        TR(long long _a = clock64();)
                        fail = fail || !mbar_wait(B_(bars->s_full[0]), gb & 1, p.err, abort_flag);
                        TR(w_sfull += clock64() - _a;
                           if (tl_on && (threadIdx.x & 127) == 0) TL(2 + 3 * wg, j, clock64() - t_start);)
                        float s[4][32];
                        if (!fail) {
                            tc_fence_after();
    #pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(trow + S_SCOL + wg * 128 + c4 * 32, s[c4]);
                            tmem_wait_ld();
                            tc_fence_before();
                            mbar_arrive(B_(bars->s_free[0]));
                            if (j == ti.nblk - 1) {   // the last block: keys after the query or past the sequence
                                const int lim = min(t, p.T - 1) - j * kBS - wg * 128;   // last visible column
    #pragma unroll
                                for (int c4 = 0; c4 < 4; ++c4)
    #pragma unroll
                                    for (int i = 0; i < 32; ++i)
                                        if (c4 * 32 + i > lim) s[c4][i] = -INFINITY;
                            }
                            st_shared_f32(base + PMAX + ((gb & 1) * 2 + wg) * kBM * 4 + row * 4, tree_max128(s) * F);
                        }
                        TR(long long _x = clock64();)
                        if (named_bar_or(1, 256, fail)) { ok = false; break; }   // also publishes the partial maxima
                        TR(w_xbar += clock64() - _x; if (tl_on && threadIdx.x == 128) TL(3, j, clock64() - t_start);)
                        const float mx = fmaxf(ld_shared_f32(base + PMAX + ((gb & 1) * 2 + 0) * kBM * 4 + row * 4),
                                               ld_shared_f32(base + PMAX + ((gb & 1) * 2 + 1) * kBM * 4 + row * 4));
                        float factor = 1.f;
                        if (mx > m_run + kRescaleLog2) {
                            factor = fast_exp2(m_run - mx);
                            m_run = mx;
                        }
    #pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
    #pragma unroll
                            for (int i = 0; i < 32; ++i) s[c4][i] = fast_exp2(fmaf(s[c4][i], F, -m_run));
                        l_part = l_part * factor + tree_sum128(s);

                        TR(long long _s = clock64();)
                        // the staging unit is free once this warpgroup's previous copy has read it
                        if (issuer) bulk_wait_read_all();
                        named_bar_sync(2 + wg, 128);
    #pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
    #pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float *v = &s[c4][8 * q4];
                                st_shared_v4(ptile + (c4 >> 1) * kSlab + sw128_offset(row, (c4 & 1) * 4 + q4),
                                             pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                             pack_bf16x2(v[6], v[7]));
                            }
                        // unit 2j carries the block's rescale factor; unit 2j+1 shares its maximum (factor 1)
                        st_shared_v2f(ri + row * 8, wg == 0 ? factor : 1.f, l_part);
                        fence_proxy_async_smem();
                        named_bar_sync(2 + wg, 128);
                        TR(w_store += clock64() - _s;)
                        if (issuer) {
                            // the value CTA's P buffer `wg` is free once the product of this warpgroup's previous
                            // unit completed (and, after a tile's last units, once the epilogue's staging is done)
                            TR(long long _f = clock64();)
                            if (nu >= 1) fail = !mbar_wait<true>(B_(bars->p_free[wg]), (nu - 1) & 1, p.err, abort_flag);
                            TR(w_pfree += clock64() - _f;)
                            if (!fail) {
                                const uint32_t dst_bar = mapa_shared(B_(bars->p_full[wg]), 1);
                                bulk_copy_s2cluster(mapa_shared(base + O_P + wg * kPBytes, 1), ptile, kPBytes, dst_bar);
                                bulk_copy_s2cluster(mapa_shared(base + O_ROWINFO + wg * kRowInfoBytes, 1), ri,
                                                    kRowInfoBytes, dst_bar);
                                bulk_commit_group();
                                TR(if (tl_on) TL(wg == 0 ? 4 : 6, j, clock64() - t_start);)
                            }
                        }
                        ++nu;
                    }
                    if (!ok) break;
                    if (p.lse) {   // ln sum_u exp(scale s_u) = ln 2 (m + log2 l), l = both warpgroups' sums
                        if (wg == 1) st_shared_f32(base + LSUM + row * 4, l_part);
                        named_bar_sync(1, 256);
                        if (wg == 0 && t < p.T)
                            p.lse[(static_cast<size_t>(ti.b) * p.H + ti.h) * p.T + t] =
                                kLn2 * (m_run + log2f(l_part + ld_shared_f32(base + LSUM + row * 4)));
                    }
                    // the first staging buffer takes the next tile's q tile once this tile's last copy has read it
                    if (issuer) bulk_wait_read_all();
                    if (issuer && wg == 0) mbar_arrive(B_(bars->q_free));
                }
                TR(if (threadIdx.x == 128) {
                    TR_ADD(TR_S_SM_LOOP, clock64() - tl0); TR_ADD(TR_S_SM_SFULL, w_sfull); TR_ADD(TR_S_SM_XBAR, w_xbar);
                    TR_ADD(TR_S_SM_PFREE, w_pfree); TR_ADD(TR_S_SM_STORE, w_store); TR_ADD(TR_S_SM_RELEASE, w_rel);
                })
                if (issuer) bulk_wait_all();
                if (!ok || fail) *abort_flag = 1;
        } else {
            // =========================================================== value CTA: corrections, epilogue
                // ---- correction + epilogue: thread `row` of warpgroup `wg` owns TMEM lane `row`,
                // latent columns [256 wg, 256 wg + 256) for rescaling
                const int wg = (warp - 4) >> 2;
                const int row = (warp & 3) * 32 + lane;
                const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
                int gu = 0;
                bool ok = true, fail;
                TR(long long tl0 = clock64();)
                for (int k = 0; ok; ++k) {
                    const int tile = tile_of(k);
                    if (tile >= p.n_tiles) break;
                    const TileInfo ti = tile_info(tile, p);
                    const int t = ti.t0 + row;
                    float l_even = 0.f, l_odd = 0.f;
                    for (int j = 0; j < ti.nkv; ++j, ++gu) {
                        const int pb = gu & 1;
                        fail = !mbar_wait<true>(B_(bars->p_full[pb]), (gu >> 1) & 1, p.err, abort_flag);
                        if (named_bar_or(4, 256, fail)) { ok = false; break; }
                        const float2 fl = ld_shared_v2f(base + O_ROWINFO + pb * kRowInfoBytes + row * 8);
                        mbar_arrive(B_(bars->ri_read[pb]));
                        // the two warpgroups of the score CTA keep separate sums (even and odd units)
                        if (j & 1)
                            l_odd = fl.y;
                        else
                            l_even = fl.y;
                        if (named_bar_or(4, 256, j > 0 && fl.x != 1.f)) {
                            const int pu = gu - 1;
                            fail = !mbar_wait(B_(bars->pv_done[pu & 1]), (pu >> 1) & 1, p.err, abort_flag);
                            if (named_bar_or(4, 256, fail)) { ok = false; break; }
                            tc_fence_after();
                            if (__any_sync(0xffffffffu, fl.x != 1.f)) {
    #pragma unroll 1
                                for (int cc = 0; cc < 8; ++cc) {
                                    float v[32];
                                    const uint32_t ta = trow + wg * 256 + cc * 32;
                                    tmem_ld32(ta, v);
                                    tmem_wait_ld();
    #pragma unroll
                                    for (int i = 0; i < 32; ++i) v[i] *= fl.x;
                                    tmem_st32(ta, v);
                                }
                                tmem_wait_st();
                            }
                            tc_fence_before();
                            mbar_arrive(B_(bars->corr_done));
                        }
                    }
                    if (!ok) break;
                    {
                        const int pu = gu - 1;   // this tile's last unit
                        fail = !mbar_wait(B_(bars->pv_done[pu & 1]), (pu >> 1) & 1, p.err, abort_flag);
                        if (named_bar_or(4, 256, fail)) { ok = false; break; }
                    }
                    TR(const long long t_ep = clock64();)
                    // this row's gate values (read once, from DRAM) are requested now: their latency runs under
                    // the packing and the W_UV product
                    const size_t off = ((static_cast<size_t>(ti.b) * p.T + t) * p.H + ti.h) * kD + wg * 64;
                    uint4 gv[8];
                    if (p.gate && t < p.T) {
    #pragma unroll
                        for (int v2 = 0; v2 < 4; ++v2)
                            ld_global_32B(reinterpret_cast<const uint4 *>(p.gate + off) + 2 * v2, gv[2 * v2], gv[2 * v2 + 1]);
                    } else {
    #pragma unroll
                        for (int v8 = 0; v8 < 8; ++v8) gv[v8] = make_uint4(0, 0, 0, 0);
                    }
                    const float inv_l = 1.f / (l_even + l_odd);
                    // o_lat/l packed as bf16 pairs in place, the A operand of the W_UV product: warpgroup 0 takes
                    // latent columns 0-255 into TMEM columns 0-127 (chunks in increasing order), warpgroup 1
                    // latent columns 256-511 into columns 384-511 (decreasing order), so no column is written
                    // before it has been read
                    tc_fence_after();
    #pragma unroll 1
                    for (int i = 0; i < 8; ++i) {
                        const int c = wg == 0 ? i : 7 - i;
                        float v[32], w[16];
                        tmem_ld32(trow + wg * 256 + c * 32, v);
                        tmem_wait_ld();
    #pragma unroll
                        for (int q = 0; q < 16; ++q) w[q] = __uint_as_float(pack_bf16x2(v[2 * q] * inv_l, v[2 * q + 1] * inv_l));
                        tmem_st16(trow + (wg == 0 ? 16 * c : 384 + 16 * c), w);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar_sync(4, 256);
                    if (threadIdx.x == 128) mbar_arrive(B_(bars->olat_ready));
                    TR(const long long t_pk = clock64(); if (threadIdx.x == 128) TR_ADD(TR_O_EP_PACK, t_pk - t_ep);)
                    fail = !mbar_wait(B_(bars->ep_done), k & 1, p.err, abort_flag);
                    if (named_bar_or(4, 256, fail)) { ok = false; break; }
                    TR(const long long t_md = clock64(); if (threadIdx.x == 128) TR_ADD(TR_O_EP_WAIT, t_md - t_pk);)
                    tc_fence_after();
                    float o[2][32];
    #pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) tmem_ld32(trow + O_EPCOL + wg * 64 + c2 * 32, o[c2]);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(B_(bars->ep_read));   // the next tile may overwrite these TMEM columns
                    if (t < p.T) {
                        uint4 *o4 = reinterpret_cast<uint4 *>(p.out + off);
                        uint4 ov[8];
    #pragma unroll
                        for (int v8 = 0; v8 < 8; ++v8) {
                            float y[8];
    #pragma unroll
                            for (int i = 0; i < 8; ++i) y[i] = o[(v8 * 8 + i) >> 5][(v8 * 8 + i) & 31];
                            if (p.gate) {
                                const uint32_t gw[4] = {gv[v8].x, gv[v8].y, gv[v8].z, gv[v8].w};
    #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float g_lo = __uint_as_float(gw[i] << 16);
                                    const float g_hi = __uint_as_float(gw[i] & 0xFFFF0000u);
                                    y[2 * i] *= __fdividef(1.f, 1.f + fast_exp2(-g_lo * kLog2e));
                                    y[2 * i + 1] *= __fdividef(1.f, 1.f + fast_exp2(-g_hi * kLog2e));
                                }
                            }
                            ov[v8] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                        }
    #pragma unroll
                        for (int v2 = 0; v2 < 4; ++v2) st_global_32B(o4 + 2 * v2, ov[2 * v2], ov[2 * v2 + 1]);
                    }
                    TR(if (threadIdx.x == 128) { TR_ADD(TR_O_EPILOGUE, clock64() - t_ep); TR_ADD(TR_O_EP_OUT, clock64() - t_md); })
                }
                TR(if (threadIdx.x == 128) TR_ADD(TR_O_COR_LOOP, clock64() - tl0);)
                if (!ok) *abort_flag = 1;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    TR(if (threadIdx.x == 0) TR_ADD(rank == 0 ? TR_S_TOTAL : TR_O_TOTAL, clock64() - t_start);)
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster_sync_all();   // the partner no longer touches this CTA's shared memory
}

// The f16 copy of the latent for the score product, in two passes over c [B, T, 512] bf16 (one CTA per
// 32-key group g of sequence b in each): latent_amax_kernel writes the group's largest |c| to gmax[b][g];
// latent_f16_kernel takes the sequence's maximum over its groups, the power of two 2^e_b that brings it into
// [2^13, 2^14), and writes c16 = c * 2^e_b (f16, round to nearest even) and sscale[b] = 2^-e_b.
constexpr int kCvtThreads = 256;
constexpr int kCvtRows = 32;                                   // keys per conversion CTA
constexpr int kCvtChunks = kCvtRows * kR / 8 / kCvtThreads;    // 16-byte chunks per thread

__device__ __forceinline__ float block_max(float v, float *wmax) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = v;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kCvtThreads / 32; ++i) v = fmaxf(v, wmax[i]);
    return v;
}

__global__ void __launch_bounds__(kCvtThreads) latent_amax_kernel(const uint4 *__restrict__ c, float *__restrict__ gmax,
                                                                  int T, int n_groups) {
    __shared__ float wmax[kCvtThreads / 32];
    const int b = static_cast<int>(blockIdx.x) / n_groups, g = static_cast<int>(blockIdx.x) % n_groups;
    grid_launch_dependents();
    const size_t first = (static_cast<size_t>(b) * T + static_cast<size_t>(g) * kCvtRows) * (kR / 8);
    const int n = min(kCvtRows, T - g * kCvtRows) * (kR / 8);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kCvtChunks; ++k) {
        const int u = static_cast<int>(threadIdx.x) + k * kCvtThreads;
        if (u < n) {
            const uint4 v = __ldg(c + first + u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
    }
    amax = block_max(amax, wmax);
    if (threadIdx.x == 0) gmax[blockIdx.x] = amax;
}

__global__ void __launch_bounds__(kCvtThreads) latent_f16_kernel(const uint4 *__restrict__ c, const float *__restrict__ gmax,
                                                                 uint4 *__restrict__ c16, float *__restrict__ sscale,
                                                                 int T, int n_groups) {
    __shared__ float wmax[kCvtThreads / 32];
    const int b = static_cast<int>(blockIdx.x) / n_groups, g = static_cast<int>(blockIdx.x) % n_groups;
    grid_launch_dependents();   // the prefill may take SMs as they free up; it waits for this grid before use
    grid_dependency_wait();     // launched as a dependent of latent_amax_kernel: gmax is complete after this
    float amax = 0.f;
    for (int i = static_cast<int>(threadIdx.x); i < n_groups; i += kCvtThreads)
        amax = fmaxf(amax, gmax[static_cast<size_t>(b) * n_groups + i]);
    amax = block_max(amax, wmax);
    const int e = f16_range_exponent(amax);
    const float up = exp2_int(e);
    if (g == 0 && threadIdx.x == 0) sscale[b] = exp2_int(-e);
    const size_t first = (static_cast<size_t>(b) * T + static_cast<size_t>(g) * kCvtRows) * (kR / 8);
    const int n = min(kCvtRows, T - g * kCvtRows) * (kR / 8);
#pragma unroll 8
    for (int k = 0; k < kCvtChunks; ++k) {
        const int u = static_cast<int>(threadIdx.x) + k * kCvtThreads;
        if (u < n) {
            const uint4 v = __ldg(c + first + u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = pack_f16x2(__uint_as_float(w[i] << 16) * up, __uint_as_float(w[i] & 0xFFFF0000u) * up);
            c16[first + u] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

CUresult encode_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, type, rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool prefill_bf16_r512_supports(int r, int d_q, int d_v) { return r == kR && d_q == kD && d_v == kD; }

// Workspace of the r = 512 prefill: the f16 latent copy [B, T, 512], the group maxima [B][ceil(T / 32)] and
// the sequence scales [B].
size_t prefill_bf16_r512_workspace_bytes(long long B, long long T) {
    const size_t c16 = (static_cast<size_t>(B) * T * kR * 2 + 255) & ~static_cast<size_t>(255);
    return c16 + static_cast<size_t>(B) * ((T + kCvtRows - 1) / kCvtRows + 1) * sizeof(float);
}

#ifdef MLA_TRACE
// Diagnostic build only: copy (and optionally clear) the wait-accounting slots.
extern "C" __attribute__((visibility("default"))) int mla_debug_prefill_trace(unsigned long long *host, int n,
                                                                                int clear) {
    if (n > TR_COUNT) n = TR_COUNT;
    if (cudaMemcpyFromSymbol(host, g_trace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
    if (clear) {
        static const unsigned long long zeros[TR_COUNT] = {};
        if (cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) != cudaSuccess) return -1;
    }
    return n;
}
// Diagnostic build only: copy the per-block event times of the traced cluster.
extern "C" __attribute__((visibility("default"))) int mla_debug_prefill_timeline(long long *host) {
    if (cudaMemcpyFromSymbol(host, g_ptl, sizeof(g_ptl)) != cudaSuccess) return -1;
    return kTLEvents * kTLMax;
}
#endif

cudaError_t launch_prefill_bf16_r512(const PrefillArgs &a, cudaStream_t s) {
    if (!prefill_bf16_r512_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    if (!a.workspace || a.workspace_bytes < prefill_bf16_r512_workspace_bytes(a.B, a.T)) return cudaErrorInvalidValue;
    const cuuint64_t B = a.B, T = a.T, H = a.H;
    const int n_groups = (a.T + kCvtRows - 1) / kCvtRows;   // conversion groups of 32 keys
    void *c16 = a.workspace;
    float *gmax = reinterpret_cast<float *>(static_cast<char *>(a.workspace) +
                                            ((static_cast<size_t>(a.B) * a.T * kR * 2 + 255) & ~static_cast<size_t>(255)));
    float *sscale = gmax + static_cast<size_t>(a.B) * n_groups;
    CUtensorMap tm_q, tm_c, tm_c256, tm_wuk, tm_wuv;
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
        const cuuint32_t box256[3] = {64, kBS, 1};
        if (encode_map(&tm_c256, c16, 3, dims, strides, box256, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
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
    p.sscale = sscale;
    p.w_uk = static_cast<const __nv_bfloat16 *>(a.w_uk);
    p.lse = a.lse;
    p.err = a.dev_err;
    p.T = a.T;
    p.H = a.H;
    p.n_qtiles = (a.T + kBM - 1) / kBM;
    p.bh_count = a.B * a.H;
    p.qk_scale_log2 = a.scale * kLog2e;
    const long long n_tiles = static_cast<long long>(p.n_qtiles) * p.bh_count;
    if (n_tiles > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
    p.n_tiles = static_cast<int>(n_tiles);
    // persistent grid: one cluster per SM pair, each walking its share of the tiles
    p.G = static_cast<int>(n_tiles < a.num_sms / 2 ? n_tiles : (a.num_sms / 2 > 0 ? a.num_sms / 2 : 1));
    cudaError_t e = cudaFuncSetAttribute(prefill_r512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    if (n_tiles == 0) return cudaSuccess;
    {   // the kernel's register split assumes this launch budget
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, prefill_r512_kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    note_launch();
    latent_amax_kernel<<<static_cast<unsigned>(a.B * n_groups), kCvtThreads, 0, s>>>(
        static_cast<const uint4 *>(a.c), gmax, a.T, n_groups);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the conversion and the prefill are programmatic dependents of the kernel before them: their prologues
    // overlap it, and each waits (griddepcontrol.wait) before reading what it wrote
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * n_groups));
    cfg.blockDim = dim3(kCvtThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    note_launch();
    e = cudaLaunchKernelEx(&cfg, latent_f16_kernel, static_cast<const uint4 *>(a.c), static_cast<const float *>(gmax),
                           static_cast<uint4 *>(c16), sscale, static_cast<int>(a.T), n_groups);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * p.G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    note_launch();
    return cudaLaunchKernelEx(&cfg, prefill_r512_kernel, tm_q, tm_c, tm_c256, tm_wuk, tm_wuv, p);
}

}  // namespace mla
