// bf16 cached-latent decode (one query per sequence) on the sm_103a tensor
// cores: r = 512, d_v = 128, 1 <= H <= 96.
//
// Only the latent c is cached (page "Gated MLA（矩阵吸收版）", KV-cache table in
// section "形状与参数对比": r values per token).  Sequence b's absorbed query
// q_abs[b] (all H heads) attends to its cache rows [0, lens[b]); steps 2-4 of
// section "完整计算流（四步）" follow: scores against c itself, softmax, the
// latent weighting by c itself, W_UV^T, gate.
//
// Pair kernel (persistent, one cluster of two CTAs per SM pair): the
// concatenation of all sequences' cache rows (plus a fixed charge per
// sequence start) is cut into one contiguous, equal share per cluster, so
// ragged lengths balance by construction.  A
// cluster walks its share as segments (one per sequence it touches) in blocks
// of 256 rows.  Heads are the M = 128 rows of every product (zero-padded):
//   rank 0, the score CTA: q_abs[b] sits in TMEM as packed bf16 (columns
//     0-255) and is the A operand of S = q_abs . c_blk^T (N = 256 cache rows,
//     K = r) into columns 256-511.  Two warpgroups run the online softmax, one
//     per 128-row half of the block (thread = head); P (bf16) and per-head
//     (rescale factor, partial sum) go to the value CTA by DSMEM bulk copies.
//   rank 1, the value CTA: o_lat += P . c_unit (M = heads, N = 2 x 256 latent
//     columns, K = 128 cache rows), fp32 in all 512 TMEM columns, rescaled
//     lazily when a head's maximum grew by more than 2^16.
// Per segment the cluster writes (o_lat unnormalised, running max, sum) to a
// workspace slot.  Each cache row is read from HBM once by the score CTA,
// which keeps it in L2 (evict_last) for the value CTA's second read
// (evict_first).
// Merge kernel: one CTA per (head, 32 sequences), launched as a programmatic
// dependent of the pair kernel, combines the segments of a sequence with the
// log-sum-exp rule, rounds o_lat to bf16 and applies W_UV^T on the tensor
// cores, then the sigmoid gate.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kR = 512;
constexpr int kDV = 128;
constexpr int kBS = 256;      // cache rows per score block
constexpr int kBN = 128;      // cache rows per value unit (two per block)
constexpr int kHMax = 96;
constexpr int kThreads = 384;   // warps 0 TMA, 1 MMA, 2 relay (value CTA), 4-7 and 8-11: two warpgroups
// Register split: the control warpgroup (warps 0-3) gives registers to the two
// math warpgroups.  4 x 32 x 56 + 8 x 32 x 216 = 62,464 <= 384 x 168 launched.
#ifndef MLA_TRACE
constexpr uint32_t kRegsCtl = 56, kRegsMath = 216, kRegsLaunch = 168;
#else   // the wait accounting needs more registers in the control warps
constexpr uint32_t kRegsCtl = 88, kRegsMath = 200, kRegsLaunch = 168;
#endif
static_assert(128 * kRegsCtl + 256 * kRegsMath <= kThreads * kRegsLaunch, "register split exceeds the launch");
constexpr float kLog2e = 1.4426950408889634f;
// Keep a stale maximum until the new one exceeds it by this (log2 units):
// p <= 2^16, far inside the fp32 range of the sums and the accumulator.
constexpr float kRescaleLog2 = 16.0f;
// Largest scratch the no-alloc decode entry point can use (48 MiB: the K3 decode
// workload, B = 64 and H = 96 on 152 SMs, needs 13.9 MB).
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

constexpr uint32_t kSlab = 16384;                    // [128 rows x 64 bf16] with 128-byte swizzle
// P travels compactly: only the H <= 96 head rows of each [128 x 64] swizzled
// slab are stored and copied.  The value CTA's M = 128 operand read of a slab
// runs 4 KB into the following memory; those rows (heads >= H) only feed
// accumulator rows nobody reads.
constexpr uint32_t kPSlab = kHMax * 128;             // compact P slab: [96 heads x 64 rows]
constexpr uint32_t kPBytes = 2 * kPSlab;             // one unit of P: [96 heads x 128 rows]
constexpr uint32_t kRowInfoBytes = 128 * 8;          // {rescale factor, running sum} per head
// score CTA
constexpr uint32_t kSStage = 2 * kSlab;              // c ring stage: [256 rows x 64 latent columns]
constexpr int kSStages = 5;
constexpr uint32_t S_RING = 0;
constexpr uint32_t kPUnit = kPBytes + kRowInfoBytes; // staging per warpgroup
constexpr uint32_t S_PST = S_RING + kSStages * kSStage;
constexpr uint32_t S_END = S_PST + 2 * kPUnit;
// value CTA
constexpr uint32_t O_RING = 0;
constexpr int kVRows = 64;                           // cache rows per value ring stage (half a unit)
constexpr uint32_t kVSlab = kVRows * 128;            // [64 rows x 64 latent columns], 128-byte swizzle
constexpr int kOStages = 4;
constexpr uint32_t kOStage = 4 * kVSlab;             // 256 latent columns x 64 rows
constexpr int kPBufs = 3;                            // P units in flight to the value CTA
constexpr uint32_t O_P = kOStages * kOStage;         // kPBufs P tiles, then the operand over-read pad
constexpr uint32_t O_ROWINFO = O_P + kPBufs * kPBytes + (kSlab - kPSlab);
constexpr uint32_t O_END = O_ROWINFO + kPBufs * kRowInfoBytes;
constexpr uint32_t BARS = S_END > O_END ? S_END : O_END;
constexpr uint32_t PMAX = BARS + 512;                // [2 parities][2 warpgroups][128 heads] partial maxima
constexpr uint32_t kSmemPair = PMAX + 2 * 2 * 128 * 4 + 1024;   // + alignment slack
static_assert(BARS % 16 == 0, "barrier alignment");
static_assert(kSmemPair <= 232448, "pair kernel exceeds shared memory");
static_assert(S_PST % 1024 == 0 && kPUnit % 1024 == 0 && kPSlab % 1024 == 0 && O_P % 1024 == 0, "alignment");
// TMEM columns of the score CTA
constexpr uint32_t S_QCOL = 0;     // packed bf16 q_abs: K step ks (16 latent columns) at columns 8 ks .. 8 ks + 7
constexpr uint32_t S_SCOL = 256;   // S for one 256-row block

constexpr uint32_t kIdescQK = make_idesc_bf16(128, 256, 0, 0);   // q_abs (TMEM) x c (K-major), 256 rows
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 256, 0, 1);   // P (K-major) x c (MN-major)
// The e4m3 cache (kF8): the same products as kind::f8f6f4 (K = 32 per instruction, twice the bf16 rate), each
// 16-bit operand split into e4m3 hi + lo parts that both multiply the cache tile.  TMEM: q_abs hi in columns
// 0-127 and lo in 128-255 (four e4m3 per column, 8 columns per K step of 32).
constexpr uint32_t S_QLO = 128;
constexpr uint32_t kIdescQK8 = make_idesc_e4m3(128, 256, 0, 0);
constexpr uint32_t kIdescPV8 = make_idesc_e4m3(128, 256, 0, 1);
// kF8 softmax weights: p' = exp2(s - m + 4), rescaled once the maximum grows by more than 4, so p' <= 2^8
// (inside e4m3's 448) and weights down to 2^-13 of the maximum keep their lo part.
constexpr float kRescaleLog2F8 = 4.0f, kPBiasF8 = 4.0f;

struct PairBars {
    uint64_t qabs_ready;                              // score CTA
    uint64_t sc_full[kSStages], sc_empty[kSStages];
    uint64_t s_full, s_free;
    uint64_t p_free[kPBufs];                          // arrivals from the value CTA
    uint64_t oc_full[kOStages], oc_empty[kOStages];   // value CTA
    uint64_t p_full[kPBufs];                          // bulk-copy transactions from the score CTA
    uint64_t pv_done[kPBufs], ri_read[kPBufs], corr_done, o_drained;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PairBars) <= 512, "barrier block too large");

// Opt-in wait accounting (build with MLA_NVCC_FLAGS=-DMLA_TRACE): cycles each
// role spends at its waits and in its loop, summed over all CTAs.
enum DecodeTraceSlot {
    DT_S_MMA_LOOP, DT_S_MMA_SFREE, DT_S_MMA_SCFULL, DT_S_MMA_QREADY, DT_S_SM_LOOP, DT_S_SM_SFULL, DT_S_SM_XBAR,
    DT_S_SM_PFREE, DT_S_SM_QLOAD, DT_O_MMA_LOOP, DT_O_MMA_PFULL, DT_O_MMA_OCFULL, DT_O_MMA_CORR, DT_O_MMA_DRAINED,
    DT_O_COR_LOOP, DT_O_DRAIN, DT_S_PROD_EMPTY, DT_O_PROD_EMPTY, DT_SEGMENTS, DT_BLOCKS, DT_CORRECTIONS,
    DT_S_TOTAL, DT_O_TOTAL, DT_COUNT
};
#ifdef MLA_TRACE
__device__ unsigned long long g_dtrace[DT_COUNT];
#define TR(...) __VA_ARGS__
#define TR_ADD(slot, v) atomicAdd(&g_dtrace[slot], static_cast<unsigned long long>(v))
// Per-block event times (cycles since the start barrier) of one cluster, for timelines.
constexpr int kTLMax = 256, kTLEvents = 14, kTLCluster = 10;
__device__ long long g_dtl[kTLEvents][kTLMax];
__device__ long long g_dclu[2][512];   // per cluster: value CTA's total cycles, segments
__device__ long long g_mtrace[8][1024];   // per merge CTA: phase end times (cycles since its start)
#define MT(ph) do { if (threadIdx.x == 0) { const int _c = blockIdx.y * gridDim.x + blockIdx.x; \
    if (_c < 1024) g_mtrace[ph][_c] = clock64() - mt0; } } while (0)
#define TL(ev, idx, val) \
    do { if (cl == kTLCluster && static_cast<int>(idx) < kTLMax) g_dtl[ev][idx] = (val); } while (0)
#else
#define TR(...)
#define TR_ADD(slot, v) (void)0
#define MT(ph) (void)0
#endif

struct PairParams {
    const int *lens;
    const __nv_bfloat16 *q_abs;   // kF8: [B][H] rows of 1024 bytes, e4m3 hi (512) then lo (512)
    const float *qmul;            // kF8: [B][H], the power of two that undoes q_abs's split scale
    float cache_scale;            // kF8: the cache holds c / cache_scale
    __nv_bfloat16 *ws_o;   // [slots][H][r], unnormalised o_lat rounded to bf16
    float *ws_m;   // [slots][H]
    float *ws_l;   // [slots][H]
    int *err;
    int B, H, max_len;
    float qk_scale_log2;
};

__device__ __forceinline__ int clamp_len(int x, int max_len) { return min(max(x, 0), max_len); }

// Work is split on a virtual row axis: each non-empty sequence occupies
// kSeqOverhead virtual rows (the cost of starting a segment: loading its
// query, draining its accumulator, refilling the pipeline) followed by its
// cache rows.  Cluster c of G owns the virtual rows [share_lo(c), share_lo(c+1)).
constexpr long long kSeqOverhead = 1024;
__device__ __forceinline__ long long share_lo(long long total, int c, int G) { return (total * c) / G; }

// Walks the (sequence, [k0, k1)) segments of one cluster's share in order.
// Every role of both CTAs runs the same walk, so their counters agree.
struct SegWalk {
    const int *lens;
    int B, max_len;
    long long lo, hi, pre;   // pre = first virtual row of sequence b
    int b;
    __device__ void init(const int *lens_, int B_, int max_len_, long long lo_, long long hi_) {
        lens = lens_;
        B = B_;
        max_len = max_len_;
        lo = lo_;
        hi = hi_;
        pre = 0;
        b = 0;
    }
    // Next non-empty segment; false when the share is exhausted.
    __device__ bool next(int &seq, int &k0, int &k1) {
        while (b < B && pre < hi) {
            const int len = clamp_len(__ldg(lens + b), max_len);
            const long long base = pre + kSeqOverhead;   // virtual row of cache row 0
            const long long s0 = max(base, lo), s1 = min(base + len, hi);
            const int cur = b;
            if (len > 0) pre = base + len;
            ++b;
            if (s1 > s0) {
                seq = cur;
                k0 = static_cast<int>(s0 - base);
                k1 = static_cast<int>(s1 - base);
                return true;
            }
        }
        return false;
    }
};

__device__ __forceinline__ long long total_rows(const int *lens, int B, int max_len, int *err, bool report) {
    long long t = 0;
    for (int b = 0; b < B; ++b) {
        const int x = __ldg(lens + b);
        if (report && (x < 0 || x > max_len)) record_error(err, kDevErrBounds);
        const int len = clamp_len(x, max_len);
        if (len > 0) t += kSeqOverhead + len;
    }
    return t;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_v2f(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// Reductions over 128 values as 8 interleaved chains: short dependency chains
// without holding 32 extra temporaries next to the 128 values.
__device__ __forceinline__ float max128(const float (&s)[4][32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = s[0][i];
#pragma unroll
    for (int k = 8; k < 128; ++k) m[k & 7] = fmaxf(m[k & 7], s[k >> 5][k & 31]);
    return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}
__device__ __forceinline__ float min128(const float (&s)[4][32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = s[0][i];
#pragma unroll
    for (int k = 8; k < 128; ++k) m[k & 7] = fminf(m[k & 7], s[k >> 5][k & 31]);
    return fminf(fminf(fminf(m[0], m[1]), fminf(m[2], m[3])), fminf(fminf(m[4], m[5]), fminf(m[6], m[7])));
}
__device__ __forceinline__ float sum128(const float (&s)[4][32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = s[0][i];
#pragma unroll
    for (int k = 8; k < 128; ++k) m[k & 7] = m[k & 7] + s[k >> 5][k & 31];
    return ((m[0] + m[1]) + (m[2] + m[3])) + ((m[4] + m[5]) + (m[6] + m[7]));
}

// Absorbed-query rows into TMEM: a head's packed bf16 pairs are its row's
// 32-bit words in memory order.  Warpgroup wg owns latent columns
// [256 wg, 256 wg + 256) of head `row` (zeros for padding heads), in two
// halves of 16 x 16 bytes.
__device__ __forceinline__ void q_issue(const __nv_bfloat16 *q_abs, int sq, int H, int row, bool head, int wg, int half,
                                        uint4 (&v)[16]) {
    const uint4 *src =
        reinterpret_cast<const uint4 *>(q_abs + (static_cast<size_t>(sq) * H + (head ? row : 0)) * kR) + wg * 32 +
        half * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = head ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void q_store(uint32_t trow, int wg, int half, const uint4 (&v)[16]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w[4 * i + 0] = __uint_as_float(v[8 * k + i].x);
            w[4 * i + 1] = __uint_as_float(v[8 * k + i].y);
            w[4 * i + 2] = __uint_as_float(v[8 * k + i].z);
            w[4 * i + 3] = __uint_as_float(v[8 * k + i].w);
        }
        tmem_st32(trow + S_QCOL + wg * 128 + (half * 2 + k) * 32, w);
    }
}

template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap tm_c256, const __grid_constant__ CUtensorMap tm_c,
                       const PairParams p) {
    // a score stage holds 256 rows x 128 bytes: 64 bf16 or 128 e4m3 latent columns
    constexpr int kStagesPerBlock = kF8 ? 4 : 8;
    constexpr int kStageCols = kF8 ? 128 : 64;
    // a value stage holds 64 rows x 256 latent columns: 4 slabs of 64 bf16 or 2 of 128 e4m3 columns
    constexpr int kVSlabs = kF8 ? 2 : 4;
    constexpr uint32_t kOStageBytes = kVSlabs * kVSlab;
    constexpr float kRescale = kF8 ? kRescaleLog2F8 : kRescaleLog2;
    constexpr float kPBias = kF8 ? kPBiasF8 : 0.f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    PairBars *bars = reinterpret_cast<PairBars *>(smem_raw + (base - raw) + BARS);
    volatile int *abort_flag = &bars->abort;
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int G = static_cast<int>(gridDim.x >> 1), cl = static_cast<int>(blockIdx.x >> 1);
    const int H = p.H;

    if (threadIdx.x == 0) {
        mbar_init(B_(bars->qabs_ready), 1);
        for (int i = 0; i < kSStages; ++i) {
            mbar_init(B_(bars->sc_full[i]), 1);
            mbar_init(B_(bars->sc_empty[i]), 1);
        }
        mbar_init(B_(bars->s_full), 1);
        mbar_init(B_(bars->s_free), 256);
        for (int i = 0; i < kPBufs; ++i) {
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
        mbar_init(B_(bars->o_drained), 1);
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
    TR(const long long t_start = clock64();)
    grid_launch_dependents();   // the merge may take SMs as clusters finish; it waits for the whole grid

    const long long total = total_rows(p.lens, p.B, p.max_len, p.err, cl == 0 && rank == 0 && threadIdx.x == 0);
    SegWalk walk;
    walk.init(p.lens, p.B, p.max_len, share_lo(total, cl, G), share_lo(total, cl + 1, G));
    int seq, k0, k1;

    if (warp < 4) {
        regs_release<kRegsCtl>();
        if (rank == 0) {
            // =========================================================== score CTA
            if (warp == 0 && lane == 0) {
                // ---- TMA producer: c tiles [256 rows x 64 latent columns]; the next segment's absorbed
                // query is prefetched into L2 near the end of this one
                tma_prefetch_desc(&tm_c256);
                const uint64_t keep = l2_policy_evict_last();   // the value CTA reads these rows again
                uint32_t it = 0;
                bool ok = true;
                while (ok && walk.next(seq, k0, k1)) {
                    const int nblk = (k1 - k0 + kBS - 1) / kBS;
                    SegWalk nx = walk;
                    int n_seq, n_k0, n_k1;
                    const bool has_next = nx.next(n_seq, n_k0, n_k1);
                    for (int j = 0; ok && j < nblk; ++j) {
                        const int key = k0 + j * kBS;
                        if (has_next && j + 2 >= nblk)   // the softmax loads it one to two blocks from now
                            bulk_prefetch_l2(p.q_abs + static_cast<size_t>(n_seq) * H * kR, static_cast<uint32_t>(H) * kR * 2);
                        for (int kc = 0; kc < kStagesPerBlock; ++kc, ++it) {
                            const int st = it % kSStages;
                            TR(const long long _a = clock64();)
                            if (it >= kSStages &&
                                !(ok = mbar_wait(B_(bars->sc_empty[st]), ((it / kSStages) - 1) & 1, p.err, abort_flag)))
                                break;
                            TR(TR_ADD(DT_S_PROD_EMPTY, clock64() - _a);)
                            mbar_arrive_expect_tx(B_(bars->sc_full[st]), kSStage);
                            tma_load_3d_hint(base + S_RING + st * kSStage, &tm_c256, B_(bars->sc_full[st]),
                                             kc * kStageCols, key, seq, keep);
                        }
                    }
                }
                if (!ok) *abort_flag = 1;
                // no load may still be landing when the CTA exits
                for (uint32_t k = (it > kSStages ? it - kSStages : 0); k < it; ++k)
                    mbar_wait(B_(bars->sc_full[k % kSStages]), (k / kSStages) & 1, p.err);
            } else if (warp == 1 && lane == 0) {
                // ---- MMA issuer: S = q_abs . c^T per 256-row block (q_abs from TMEM, N = 256)
                uint32_t it = 0, jb = 0, nseg = 0;
                bool ok = true;
                TR(long long tl0 = clock64(), w_free = 0, w_full = 0, w_q = 0;)
                while (ok && walk.next(seq, k0, k1)) {
                    const int nblk = (k1 - k0 + kBS - 1) / kBS;
                    TR(long long _q = clock64();)
                    if (!(ok = mbar_wait(B_(bars->qabs_ready), nseg & 1, p.err, abort_flag))) break;
                    TR(w_q += clock64() - _q; TL(13, jb, clock64() - t_start);)
                    ++nseg;
                    for (int j = 0; ok && j < nblk; ++j, ++jb) {
                        TR(long long _a = clock64();)
                        if (jb >= 1 && !(ok = mbar_wait(B_(bars->s_free), (jb - 1) & 1, p.err, abort_flag))) break;
                        TR(w_free += clock64() - _a; TL(0, jb, clock64() - t_start); long long w_blk = 0;)
                        tc_fence_after();
                        for (int kc = 0; kc < kStagesPerBlock; ++kc, ++it) {
                            const int st = it % kSStages;
                            TR(long long _b = clock64();)
                            if (!(ok = mbar_wait(B_(bars->sc_full[st]), (it / kSStages) & 1, p.err, abort_flag))) break;
                            TR(w_full += clock64() - _b; w_blk += clock64() - _b;)
                            tc_fence_after();
    #pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t bd = make_smem_desc(base + S_RING + st * kSStage + kk * 32, 16, 1024);
                                if constexpr (kF8) {   // S = hi . c^T + lo . c^T
                                    umma_f8_tmem_a(tmem + S_SCOL, tmem + S_QCOL + (kc * 4 + kk) * 8, bd, kIdescQK8,
                                                   (kc | kk) != 0);
                                    umma_f8_tmem_a(tmem + S_SCOL, tmem + S_QLO + (kc * 4 + kk) * 8, bd, kIdescQK8, 1);
                                } else {
                                    umma_bf16_tmem_a(tmem + S_SCOL, tmem + S_QCOL + (kc * 4 + kk) * 8, bd, kIdescQK,
                                                     (kc | kk) != 0);
                                }
                            }
                            umma_commit(B_(bars->sc_empty[st]));
                        }
                        if (!ok) break;
                        umma_commit(B_(bars->s_full));
                        TR(TL(1, jb, clock64() - t_start); TL(7, jb, w_blk);)
                    }
                }
                TR(TR_ADD(DT_S_MMA_LOOP, clock64() - tl0); TR_ADD(DT_S_MMA_SFREE, w_free);
                   TR_ADD(DT_S_MMA_SCFULL, w_full); TR_ADD(DT_S_MMA_QREADY, w_q);)
                if (!ok) *abort_flag = 1;
            }
        } else {
            // =========================================================== value CTA
            if (warp == 0 && lane == 0) {
                // ---- TMA producer: c tiles as the MN-major value operand, 4 x [64 rows x 256 latent columns] a unit
                tma_prefetch_desc(&tm_c);
                const uint64_t done_with = l2_policy_evict_first();   // the last read of these rows
                uint32_t it = 0;
                bool ok = true;
                while (ok && walk.next(seq, k0, k1)) {
                    const int nunits = 2 * ((k1 - k0 + kBS - 1) / kBS);
                    for (int u = 0; ok && u < nunits; ++u) {
                        const int key = k0 + u * kBN;
                        if (key >= k1) continue;   // a unit past the segment's end: nothing to load
                        for (int nq = 0; ok && nq < 4; ++nq, ++it) {   // latent half nq >> 1, row half nq & 1
                            const int st = it % kOStages;
                            TR(const long long _a = clock64();)
                            if (it >= kOStages &&
                                !(ok = mbar_wait(B_(bars->oc_empty[st]), ((it / kOStages) - 1) & 1, p.err, abort_flag)))
                                break;
                            TR(TR_ADD(DT_O_PROD_EMPTY, clock64() - _a);)
                            const uint32_t full = B_(bars->oc_full[st]);
                            mbar_arrive_expect_tx(full, kOStageBytes);
                            for (int q4 = 0; q4 < kVSlabs; ++q4)
                                tma_load_3d_hint(base + O_RING + st * kOStage + q4 * kVSlab, &tm_c, full,
                                                 ((nq >> 1) * kVSlabs + q4) * (kF8 ? 128 : 64), key + (nq & 1) * kVRows,
                                                 seq, done_with);
                        }
                    }
                }
                if (!ok) *abort_flag = 1;
                for (uint32_t k = (it > kOStages ? it - kOStages : 0); k < it; ++k)
                    mbar_wait(B_(bars->oc_full[k % kOStages]), (k / kOStages) & 1, p.err);
            } else if (warp == 1) {
                // ---- MMA warp: o_lat += P . c; lane 0 issues.  All lanes zero the cache rows at or past
                // lens[b] in a sequence's last unit (those rows may hold anything; p = 0 times them must stay 0).
                const bool leader = lane == 0;
                auto wait_all = [&](uint64_t &bar, uint32_t parity, bool cluster) {
                    return __all_sync(0xffffffffu, cluster ? mbar_wait<true>(B_(bar), parity, p.err, abort_flag)
                                                           : mbar_wait(B_(bar), parity, p.err, abort_flag));
                };
                uint32_t it = 0, jj = 0, ncorr = 0, nseg = 0;
                bool ok = true;
                TR(long long tl0 = clock64(), w_pfull = 0, w_oc = 0, w_corr = 0, w_dr = 0;)
                while (ok && walk.next(seq, k0, k1)) {
                    const int nunits = 2 * ((k1 - k0 + kBS - 1) / kBS);
                    const int len = clamp_len(__ldg(p.lens + seq), p.max_len);
                    for (int u = 0; ok && u < nunits; ++u, ++jj) {
                        const uint32_t pb = jj % kPBufs;
                        TR(long long _a = clock64();)
                        if (leader) mbar_arrive_expect_tx(B_(bars->p_full[pb]), 2u * H * 128u + kRowInfoBytes);
                        if (!(ok = wait_all(bars->p_full[pb], (jj / kPBufs) & 1, true))) break;
                        TR(w_pfull += clock64() - _a; if (leader) TL(8, jj, clock64() - t_start); long long w_u = 0;)
                        if (u == 0 && nseg > 0) {   // the previous segment's o_lat has been drained
                            TR(long long _d = clock64();)
                            if (!(ok = wait_all(bars->o_drained, (nseg - 1) & 1, false))) break;
                            TR(w_dr += clock64() - _d;)
                        }
                        // any head whose maximum grew needs o_lat rescaled before this unit's product
                        const uint32_t ri = base + O_ROWINFO + pb * kRowInfoBytes;
                        bool grew = false;
    #pragma unroll
                        for (int k = 0; k < 4; ++k) grew |= ld_shared_f32(ri + (lane + 32 * k) * 8) != 1.f;
                        if (u > 0 && __any_sync(0xffffffffu, grew)) {
                            TR(long long _c = clock64();)
                            if (!(ok = wait_all(bars->corr_done, ncorr & 1, false))) break;
                            TR(w_corr += clock64() - _c;)
                            ++ncorr;
                        }
                        const int key = k0 + u * kBN;
                        if (key < k1) {
                            for (int nq = 0; ok && nq < 4; ++nq, ++it) {   // latent half nq >> 1, row half nq & 1
                                const int st = it % kOStages, hr = nq & 1;
                                const int nvalid = len - key - hr * kVRows;   // rows of this stage inside the sequence
                                TR(long long _o = clock64();)
                                if (!(ok = wait_all(bars->oc_full[st], (it / kOStages) & 1, false))) break;
                                TR(w_oc += clock64() - _o; w_u += clock64() - _o;)
                                if (nvalid < kVRows) {
                                    for (int sl = 0; sl < kVSlabs; ++sl) {
                                        const uint32_t tile = base + O_RING + st * kOStage + sl * kVSlab;
                                        for (int r = max(nvalid, 0) + lane; r < kVRows; r += 32)
#pragma unroll
                                            for (int ch = 0; ch < 8; ++ch)
                                                st_shared_v4(tile + (r >> 3) * 1024 + (r & 7) * 128 + ch * 16, 0, 0, 0, 0);
                                    }
                                    fence_proxy_async_smem();
                                    __syncwarp();
                                }
                                tc_fence_after();
                                if (leader) {
                                    if constexpr (kF8) {
                                        // P hi and lo slabs [heads x 128 rows], 128 bytes a head; K steps of 32 rows
#pragma unroll
                                        for (int j = 0; j < kVRows / 32; ++j) {
                                            const int kk = hr * 2 + j;   // K step within the unit's 128 rows
                                            const uint32_t pa = base + O_P + pb * kPBytes + kk * 32;
                                            const uint64_t bd =
                                                make_smem_desc(base + O_RING + st * kOStage + j * 4096, kVSlab, 1024);
                                            umma_f8(tmem + (nq >> 1) * 256, make_smem_desc(pa, 16, 1024), bd, kIdescPV8,
                                                    (u > 0 || kk > 0));
                                            umma_f8(tmem + (nq >> 1) * 256, make_smem_desc(pa + kPSlab, 16, 1024), bd,
                                                    kIdescPV8, 1);
                                        }
                                    } else {
#pragma unroll
                                        for (int j = 0; j < kVRows / 16; ++j) {
                                            const int kk = hr * 4 + j;   // K step within the unit's 128 rows
                                            const uint64_t a = make_smem_desc(
                                                base + O_P + pb * kPBytes + hr * kPSlab + j * 32, 16, 1024);
                                            const uint64_t bd =
                                                make_smem_desc(base + O_RING + st * kOStage + j * 2048, kVSlab, 1024);
                                            umma_bf16(tmem + (nq >> 1) * 256, a, bd, kIdescPV, (u > 0 || kk > 0));
                                        }
                                    }
                                    umma_commit(B_(bars->oc_empty[st]));
                                }
                                __syncwarp();
                            }
                            if (!ok) break;
                        }
                        if (leader) umma_commit(B_(bars->pv_done[pb]));
                        TR(if (leader) { TL(9, jj, clock64() - t_start); TL(10, jj, w_u); })
                    }
                    ++nseg;
                }
                TR(if (leader) {
                    TR_ADD(DT_O_MMA_LOOP, clock64() - tl0); TR_ADD(DT_O_MMA_PFULL, w_pfull); TR_ADD(DT_O_MMA_OCFULL, w_oc);
                    TR_ADD(DT_O_MMA_CORR, w_corr); TR_ADD(DT_O_MMA_DRAINED, w_dr); TR_ADD(DT_CORRECTIONS, ncorr);
                    TR_ADD(DT_SEGMENTS, nseg);
                    if (cl < 512) g_dclu[1][cl] = nseg;
                })
                if (!ok && leader) *abort_flag = 1;
            } else if (warp == 2 && lane == 0) {
                // ---- relay: P buffer pb is free again once its product completed and its row info was read
                uint32_t jj = 0;
                bool ok = true;
                while (ok && walk.next(seq, k0, k1)) {
                    const int nunits = 2 * ((k1 - k0 + kBS - 1) / kBS);
                    for (int u = 0; u < nunits; ++u, ++jj) {
                        const uint32_t pb = jj % kPBufs;
                        if (!mbar_wait(B_(bars->pv_done[pb]), (jj / kPBufs) & 1, p.err, abort_flag) ||
                            !mbar_wait(B_(bars->ri_read[pb]), (jj / kPBufs) & 1, p.err, abort_flag)) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(B_(bars->p_free[pb]), 0);
                        TR(TL(11, jj, clock64() - t_start);)
                    }
                }
            }
        }
    } else {
        regs_acquire<kRegsMath>();
        if (rank == 0) {
            // ---- softmax: warpgroup `wg` owns rows [128 wg, 128 wg + 128) of each 256-row block, i.e. the
            // value CTA's unit 2j + wg; thread `row` owns TMEM lane `row`, which is head `row`
            const int wg = (warp - 4) >> 2;
            const int row = (warp & 3) * 32 + lane;
            const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const bool head = row < H;
            const uint32_t ptile = base + S_PST + wg * kPUnit;
            const uint32_t ri = ptile + kPBytes;
            float c_log2 = p.qk_scale_log2;
            uint32_t jb = 0;
            bool ok = true, fail = false;
            TR(long long tl0 = clock64(), w_sfull = 0, w_xbar = 0, w_pfree = 0, w_q = 0;)
            // q_abs[sq] -> TMEM columns 0-255: a head's packed bf16 pairs are its row's 32-bit words in
            // memory order.  Warpgroup wg owns latent columns [256 wg, 256 wg + 256); its loads are all
            // issued at once, and the stores wait until the previous segment's score products completed.
            bool first = true;
            while (ok && walk.next(seq, k0, k1)) {
                const int nblk = (k1 - k0 + kBS - 1) / kBS;
                if (first) {   // later segments' queries are stored during the previous segment's last block
                    TR(long long _q = clock64();)
                    uint4 v[16], v2[16];
                    q_issue(p.q_abs, seq, H, row, head, wg, 0, v);
                    q_issue(p.q_abs, seq, H, row, head, wg, 1, v2);
                    q_store(trow, wg, 0, v);
                    q_store(trow, wg, 1, v2);
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar_sync(1, 256);
                    if (threadIdx.x == 128) mbar_arrive(B_(bars->qabs_ready));
                    first = false;
                    TR(w_q += clock64() - _q;)
                }
                if constexpr (kF8)   // the score product's units: (q_abs * 2^e) . (c / cache_scale)
                    c_log2 = p.qk_scale_log2 * p.cache_scale * __ldg(p.qmul + static_cast<size_t>(seq) * H + (head ? row : 0));
                float m_run = -INFINITY, l_part = 0.f;
                for (int j = 0; j < nblk; ++j, ++jb) {
                    // in the segment's last block the next segment's query goes into TMEM as soon as this
                    // block's score products have completed, so its first products overlap this softmax
                    bool q_next = false;
                    int n_seq = 0;
                    if (j == nblk - 1) {
                        SegWalk nx = walk;
                        int n_k0, n_k1;
                        q_next = nx.next(n_seq, n_k0, n_k1);
                    }
                    TR(long long _a = clock64();)
                    if (q_next) {
                        uint4 qv[16];   // half the query rides across the wait (registers allow no more)
                        q_issue(p.q_abs, n_seq, H, row, head, wg, 0, qv);
                        fail = fail || !mbar_wait(B_(bars->s_full), jb & 1, p.err, abort_flag);
                        if (!fail) {
                            tc_fence_after();
                            q_store(trow, wg, 0, qv);
                            q_issue(p.q_abs, n_seq, H, row, head, wg, 1, qv);
                            q_store(trow, wg, 1, qv);
                            tmem_wait_st();
                        }
                    } else {
                        fail = fail || !mbar_wait(B_(bars->s_full), jb & 1, p.err, abort_flag);
                    }
                    TR(w_sfull += clock64() - _a; if ((threadIdx.x & 127) == 0) TL(2 + 3 * wg, jb, clock64() - t_start);)
                    float s[4][32];
                    const int lim = k1 - (k0 + j * kBS + wg * 128);   // columns < lim are inside the segment
                    if (!fail) {
                        tc_fence_after();
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(trow + S_SCOL + wg * 128 + c4 * 32, s[c4]);
                        tmem_wait_ld();
                        tc_fence_before();
                        mbar_arrive(B_(bars->s_free));
                        // rows at or past the segment's end are masked (only the segment's last block has
                        // any).  The scale multiplies inside the exponent: max(c s) = c max(s) for c >= 0,
                        // c min(s) otherwise.  Padding heads (q_abs = 0) compute finite values nobody reads.
                        if (lim < 128) {
                            const float fill = c_log2 >= 0.f ? -INFINITY : INFINITY;
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (c4 * 32 + i >= lim) s[c4][i] = fill;
                        }
                        const float mraw = c_log2 >= 0.f ? max128(s) : min128(s);
                        st_shared_f32(base + PMAX + ((jb & 1) * 2 + wg) * 512 + row * 4,
                                      fabsf(mraw) == INFINITY ? -INFINITY : c_log2 * mraw);
                    }
                    TR(long long _x = clock64();)
                    if (named_bar_or(1, 256, fail)) { ok = false; break; }   // also publishes the partial maxima
                    TR(w_xbar += clock64() - _x; if (threadIdx.x == 128) TL(3, jb, clock64() - t_start);)
                    if (q_next && threadIdx.x == 128) {
                        mbar_arrive(B_(bars->qabs_ready));
                        TR(TL(12, jb, clock64() - t_start);)
                    }
                    const float mx = fmaxf(ld_shared_f32(base + PMAX + ((jb & 1) * 2 + 0) * 512 + row * 4),
                                           ld_shared_f32(base + PMAX + ((jb & 1) * 2 + 1) * 512 + row * 4));
                    float factor = 1.f;
                    if (mx > m_run + kRescale) {
                        factor = fast_exp2(m_run - mx);
                        m_run = mx;
                    }
                    const float neg_m = kPBias - m_run;
                    if (lim < 128) {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                s[c4][i] = c4 * 32 + i < lim ? fast_exp2(fmaf(s[c4][i], c_log2, neg_m)) : 0.f;
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                            for (int i = 0; i < 32; ++i) s[c4][i] = fast_exp2(fmaf(s[c4][i], c_log2, neg_m));
                    }
                    l_part = l_part * factor + sum128(s);

                    // the staging unit is free once this warpgroup's previous copy has read it
                    if ((threadIdx.x & 127) == 0) bulk_wait_read_all();
                    named_bar_sync(2 + wg, 128);
                    if (head) {
                        if constexpr (kF8) {   // hi slab, then lo slab: 16 rows (bytes) per 16-byte chunk
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                const float *v = &s[ch >> 1][(ch & 1) * 16];
                                uint32_t hw[4], lw[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const uint32_t a = split_e4m3x2(v[4 * k], v[4 * k + 1]);
                                    const uint32_t b = split_e4m3x2(v[4 * k + 2], v[4 * k + 3]);
                                    hw[k] = (a & 0xFFFFu) | (b << 16);
                                    lw[k] = (a >> 16) | (b & 0xFFFF0000u);
                                }
                                st_shared_v4(ptile + sw128_offset(row, ch), hw[0], hw[1], hw[2], hw[3]);
                                st_shared_v4(ptile + kPSlab + sw128_offset(row, ch), lw[0], lw[1], lw[2], lw[3]);
                            }
                        } else {
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const float *v = &s[c4][8 * k];
                                    st_shared_v4(ptile + (c4 >> 1) * kPSlab + sw128_offset(row, (c4 & 1) * 4 + k),
                                                 pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                 pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                                }
                        }
                    }
                    // unit 2j carries the block's rescale factor; unit 2j+1 shares its maximum (factor 1)
                    st_shared_v2f(ri + row * 8, wg == 0 ? factor : 1.f, l_part);
                    fence_proxy_async_smem();
                    named_bar_sync(2 + wg, 128);
                    if ((threadIdx.x & 127) == 0) {
                        // unit u = 2 jb + wg goes to the value CTA's P buffer u mod 3, free once the product
                        // of unit u - 3 completed
                        const uint32_t u = 2 * jb + wg, pb = u % kPBufs;
                        TR(long long _f = clock64();)
                        if (u >= kPBufs)
                            fail = !mbar_wait<true>(B_(bars->p_free[pb]), (u / kPBufs - 1) & 1, p.err, abort_flag);
                        TR(w_pfree += clock64() - _f;)
                        if (!fail) {
                            const uint32_t p_rows_bytes = static_cast<uint32_t>(H) * 128;
                            const uint32_t dst_bar = mapa_shared(B_(bars->p_full[pb]), 1);
                            const uint32_t dst = mapa_shared(base + O_P + pb * kPBytes, 1);
                            bulk_copy_s2cluster(dst, ptile, p_rows_bytes, dst_bar);
                            bulk_copy_s2cluster(dst + kPSlab, ptile + kPSlab, p_rows_bytes, dst_bar);
                            bulk_copy_s2cluster(mapa_shared(base + O_ROWINFO + pb * kRowInfoBytes, 1), ri,
                                                kRowInfoBytes, dst_bar);
                            bulk_commit_group();
                            TR(TL(wg == 0 ? 4 : 6, jb, clock64() - t_start);)
                        }
                    }
                }
                if (!ok) break;
                if (wg == 0 && head) p.ws_m[static_cast<size_t>(cl + seq) * H + row] = m_run - kPBias;
            }
            TR(if (threadIdx.x == 128) {
                TR_ADD(DT_S_SM_LOOP, clock64() - tl0); TR_ADD(DT_S_SM_SFULL, w_sfull); TR_ADD(DT_S_SM_XBAR, w_xbar);
                TR_ADD(DT_S_SM_PFREE, w_pfree); TR_ADD(DT_S_SM_QLOAD, w_q); TR_ADD(DT_BLOCKS, jb);
            })
            if ((threadIdx.x & 127) == 0) bulk_wait_all();
            if (!ok || fail) *abort_flag = 1;
        } else {
            // ---- correction + drain: thread `row` of warpgroup `wg` owns TMEM lane `row` (head `row`),
            // latent columns [256 wg, 256 wg + 256)
            const int wg = (warp - 4) >> 2;
            const int row = (warp & 3) * 32 + lane;
            const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const bool head = row < H;
            uint32_t jj = 0;
            bool ok = true, fail;
            TR(long long tl0 = clock64(), w_drain = 0;)
            while (ok && walk.next(seq, k0, k1)) {
                const int nunits = 2 * ((k1 - k0 + kBS - 1) / kBS);
                float l_even = 0.f, l_odd = 0.f;
                for (int u = 0; u < nunits; ++u, ++jj) {
                    const uint32_t pb = jj % kPBufs;
                    fail = !mbar_wait<true>(B_(bars->p_full[pb]), (jj / kPBufs) & 1, p.err, abort_flag);
                    if (named_bar_or(4, 256, fail)) { ok = false; break; }
                    const float2 fl = ld_shared_v2f(base + O_ROWINFO + pb * kRowInfoBytes + row * 8);
                    mbar_arrive(B_(bars->ri_read[pb]));
                    // the two warpgroups of the score CTA keep separate sums (even and odd units)
                    if (u & 1)
                        l_odd = fl.y;
                    else
                        l_even = fl.y;
                    if (named_bar_or(4, 256, u > 0 && fl.x != 1.f)) {
                        const uint32_t prev = jj - 1;
                        fail = !mbar_wait(B_(bars->pv_done[prev % kPBufs]), (prev / kPBufs) & 1, p.err, abort_flag);
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
                // segment end: o_lat (unnormalised) and the sum into the workspace slot
                TR(long long _d = clock64();)
                const uint32_t last = jj - 1;
                fail = !mbar_wait(B_(bars->pv_done[last % kPBufs]), (last / kPBufs) & 1, p.err, abort_flag);
                if (named_bar_or(4, 256, fail)) { ok = false; break; }
                tc_fence_after();
                const size_t slot = static_cast<size_t>(cl + seq);
                uint4 *dst = reinterpret_cast<uint4 *>(p.ws_o + (slot * H + (head ? row : 0)) * kR + wg * 256);
                const uint64_t ws_keep = l2_policy_evict_last();   // the merge reads it right after this kernel
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    float v[32];
                    tmem_ld32(trow + wg * 256 + cc * 32, v);
                    tmem_wait_ld();
                    if constexpr (kF8)
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= p.cache_scale;
                    if (head)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            st_global_v4_hint(dst + cc * 4 + q,
                                              make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]),
                                                         pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                                         pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                                                         pack_bf16x2(v[8 * q + 6], v[8 * q + 7])),
                                              ws_keep);
                }
                if (wg == 0 && head) p.ws_l[slot * H + row] = l_even + l_odd;
                tc_fence_before();
                named_bar_sync(4, 256);
                if (threadIdx.x == 128) mbar_arrive(B_(bars->o_drained));
                TR(w_drain += clock64() - _d;)
            }
            TR(if (threadIdx.x == 128) { TR_ADD(DT_O_COR_LOOP, clock64() - tl0); TR_ADD(DT_O_DRAIN, w_drain); })
            if (!ok) *abort_flag = 1;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    TR(if (threadIdx.x == 0) TR_ADD(rank == 0 ? DT_S_TOTAL : DT_O_TOTAL, clock64() - t_start);
       if (threadIdx.x == 0 && rank == 1 && cl < 512) g_dclu[0][cl] = clock64() - t_start;)
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster_sync_all();   // the partner no longer touches this CTA's shared memory or barriers
}

// ----------------------------------------------------------------------------- merge
constexpr int kMRows = 32;                          // sequences per merge CTA
constexpr int kMergeThreads = 512;
constexpr int kMaxClusters = 128;                   // share boundaries the merge keeps in shared memory
constexpr uint32_t kASlab = kMRows * 128;           // o_lat tile [32 rows x 64 latent columns]
constexpr uint32_t MA_OFF = 0;
constexpr uint32_t MA_BYTES = 7 * kASlab + kSlab;   // an M=128 operand read of the last slab stays inside
constexpr uint32_t MW_OFF = MA_BYTES;               // W_UV[h] ring: 2 stages x [128 x 128 latent] (2 slabs)
constexpr uint32_t kWStage = 2 * kSlab;
constexpr uint32_t MBAR_OFF = MW_OFF + 2 * kWStage;
constexpr uint32_t kSmemMerge = MBAR_OFF + 64 + 1024;   // two CTAs fit on an SM
static_assert(MW_OFF % 1024 == 0, "alignment");

struct MergeParams {
    const int *lens;
    const __nv_bfloat16 *ws_o;
    const float *ws_m, *ws_l;
    const __nv_bfloat16 *gate;
    __nv_bfloat16 *out;
    int *err;
    int B, H, max_len, G;
};

__global__ void __launch_bounds__(kMergeThreads, 2)
    decode_merge_kernel(const __grid_constant__ CUtensorMap tm_wuv, const MergeParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    uint64_t *w_full = reinterpret_cast<uint64_t *>(gbase + MBAR_OFF);   // [2]
    uint64_t *w_empty = w_full + 2;                                      // [2]
    uint64_t *mma_done = w_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(w_full + 5);
    __shared__ long long s_pre[kMRows + 1];
    __shared__ long long s_lo[kMaxClusters + 1];
    __shared__ long long s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, b0 = blockIdx.y * kMRows;
    const int H = p.H, G = p.G;
    TR(const long long mt0 = clock64();)

    if (threadIdx.x == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(smem_u32(w_full + i), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto load_w_chunk = [&](int k) {   // latent columns [128 k, 128 k + 128) of W_UV[h] into stage k % 2
        const uint32_t bar = smem_u32(w_full + (k & 1));
        mbar_arrive_expect_tx(bar, kWStage);
        for (int sl = 0; sl < 2; ++sl)
            tma_load_2d(base + MW_OFF + (k & 1) * kWStage + sl * kSlab, &tm_wuv, bar, k * 128 + sl * 64, h * kDV);
    };
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_wuv);
        load_w_chunk(0);
        load_w_chunk(1);
        for (int k = 2; k < 4; ++k)
            for (int sl = 0; sl < 2; ++sl) tma_prefetch_l2_2d(&tm_wuv, k * 128 + sl * 64, h * kDV);
    }
    if (warp == 1) {
        // virtual row offsets of this CTA's sequences (the pair kernel's work axis): a warp-wide scan
        long long run = 0;
        for (int c0 = 0; c0 < p.B; c0 += 32) {
            const int b = c0 + lane;
            const int x = b < p.B ? __ldg(p.lens + b) : 0;
            if (x < 0 || x > p.max_len) record_error(p.err, kDevErrBounds);
            const int len = clamp_len(x, p.max_len);
            long long v = len > 0 ? kSeqOverhead + len : 0, incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long n = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += n;
            }
            const long long excl = run + incl - v;   // virtual start of sequence b
            if (b < p.B && b >= b0 && b <= b0 + kMRows) s_pre[b - b0] = excl;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        for (int b = max(p.B, b0) + lane; b <= b0 + kMRows; b += 32) s_pre[b - b0] = run;
        if (lane == 0) s_total = run;
    }
    __syncthreads();
    const long long total = s_total;
    for (int c = threadIdx.x; c <= G && c <= kMaxClusters; c += kMergeThreads) s_lo[c] = share_lo(total, c, G);
    __syncthreads();
    // launched as a programmatic dependent of the pair kernel: everything above overlapped its
    // tail; its workspace writes are complete and visible after this
    MT(0);
    grid_dependency_wait();
    MT(1);

    // log-sum-exp combine of the segments of each sequence; o_lat -> bf16 tile row.
    // A warp takes a row at a time: lane j holds segment j's (m, l) and weight;
    // every lane accumulates its 16 latent columns, two segments' loads in flight.
    for (int i = warp; i < kMRows; i += kMergeThreads / 32) {
        const int b = b0 + i;
        float o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k] = 0.f;
        // the sequence's cache rows on the virtual axis (none for an empty sequence)
        const long long r0 = s_pre[i] + kSeqOverhead, r1 = s_pre[i + 1];
        if (b < p.B && r1 > r0) {
            const int c_first = min(static_cast<int>(((r0 + 1) * G - 1) / total), G - 1);
            // cluster c wrote slot c + b iff its share [lo_c, lo_c+1) overlaps [r0, r1)
            auto overlaps = [&](int c) { return c < G && min(s_lo[c + 1], r1) > max(s_lo[c], r0); };
            int n_seg = 0;   // consecutive clusters from c_first whose shares start before r1
            while (c_first + n_seg < G && s_lo[c_first + n_seg] < r1) ++n_seg;
            float M = -INFINITY, L = 0.f, wl = 0.f;
            for (int s0 = 0; s0 < n_seg; s0 += 32) {
                const int c = c_first + s0 + lane;
                const bool has = s0 + lane < n_seg && overlaps(c);
                const size_t slot = static_cast<size_t>(c + b);
                const float m = has ? __ldg(p.ws_m + slot * H + h) : -INFINITY;
                const float l = has ? __ldg(p.ws_l + slot * H + h) : 0.f;
                float mw = m;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
                const float M_new = fmaxf(M, mw);
                float lw = has ? fast_exp2(m - M_new) * l : 0.f;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
                L = (M == -INFINITY ? 0.f : L * fast_exp2(M - M_new)) + lw;
                M = M_new;
                wl = has ? fast_exp2(m - M) : 0.f;   // final when all segments fit one pass
            }
            if (i == 0) MT(6);
            for (int s0 = 0; s0 < n_seg; s0 += 32) {
                if (n_seg > 32) {   // more segments than lanes: weights against the final maximum
                    const int c = c_first + s0 + lane;
                    const bool has = s0 + lane < n_seg && overlaps(c);
                    wl = has ? fast_exp2(__ldg(p.ws_m + static_cast<size_t>(c + b) * H + h) - M) : 0.f;
                }
                const int cnt = min(32, n_seg - s0);
                for (int j = 0; j < cnt; j += 2) {
                    const bool two = j + 1 < cnt;
                    const float w0 = __shfl_sync(0xffffffffu, wl, j);
                    const float w1 = __shfl_sync(0xffffffffu, wl, two ? j + 1 : j);
                    const size_t slot0 = static_cast<size_t>(c_first + s0 + j + b);
                    // a segment with weight 0 (empty share) is not read; its slot may hold anything
                    const uint4 *src0 = reinterpret_cast<const uint4 *>(p.ws_o + (slot0 * H + h) * kR + lane * 16);
                    const uint4 *src1 = src0 + static_cast<size_t>(H) * kR / 8;
                    uint4 v0[2], v1[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        v0[q] = w0 != 0.f ? __ldg(src0 + q) : make_uint4(0, 0, 0, 0);
                        v1[q] = two && w1 != 0.f ? __ldg(src1 + q) : make_uint4(0, 0, 0, 0);
                    }
                    const float u1 = two ? w1 : 0.f;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint32_t a[4] = {v0[q].x, v0[q].y, v0[q].z, v0[q].w};
                        const uint32_t c[4] = {v1[q].x, v1[q].y, v1[q].z, v1[q].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {   // bf16 pair -> two fp32: the bits are the upper half
                            o[8 * q + 2 * k] += w0 * __uint_as_float(a[k] << 16) + u1 * __uint_as_float(c[k] << 16);
                            o[8 * q + 2 * k + 1] +=
                                w0 * __uint_as_float(a[k] & 0xFFFF0000u) + u1 * __uint_as_float(c[k] & 0xFFFF0000u);
                        }
                    }
                }
            }
            const float inv = 1.f / L;
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] *= inv;
            if (i == 0) MT(7);
        }
        const uint32_t slab = base + MA_OFF + (lane >> 2) * kASlab;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float *v = &o[8 * half];
            st_shared_v4(slab + sw128_offset(i, (lane & 3) * 2 + half), pack_bf16x2(v[0], v[1]),
                         pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    MT(2);
    if (threadIdx.x == 0) {
        // o = o_lat . W_UV^T over four 128-column chunks of the latent, two in flight
        const uint32_t idesc = make_idesc_bf16(128, kDV, 0, 0);
        bool ok = true;
        int loaded = 2;   // chunks whose loads were issued
        for (int k = 0; ok && k < 4; ++k) {
            const int st = k & 1;
            if (!(ok = mbar_wait(smem_u32(w_full + st), (k >> 1) & 1, p.err))) break;
            if (k == 0) MT(3);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int ks = 8 * k + kk;   // K step of 16 latent columns
                const uint64_t a = make_smem_desc(base + MA_OFF + (ks >> 2) * kASlab + (ks & 3) * 32, 16, 1024);
                const uint64_t bd =
                    make_smem_desc(base + MW_OFF + st * kWStage + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
                umma_bf16(tmem, a, bd, idesc, ks > 0);
            }
            umma_commit(smem_u32(w_empty + st));
            if (k + 2 < 4) {   // the stage is refilled once its products completed
                if (!(ok = mbar_wait(smem_u32(w_empty + st), 0, p.err))) break;
                load_w_chunk(k + 2);
                ++loaded;
            }
        }
        if (ok) umma_commit(smem_u32(mma_done));
        // no load may still be landing when the CTA exits
        if (!ok)
            for (int k = 0; k < loaded; ++k) mbar_wait(smem_u32(w_full + (k & 1)), (k >> 1) & 1, p.err);
    }
    __syncwarp();
    const bool done = mbar_wait(smem_u32(mma_done), 0, p.err);
    tc_fence_after();
    MT(4);
    static_assert(kMRows % 32 == 0, "epilogue warps own 32 rows each");
    if (warp < kMRows / 32 && __all_sync(0xffffffffu, done)) {
        const int i = warp * 32 + lane;
        const int b = b0 + i;
        const size_t off = (static_cast<size_t>(b) * H + h) * kDV;
        const uint4 *g4 = p.gate ? reinterpret_cast<const uint4 *>(p.gate + off) : nullptr;
        uint4 *o4 = reinterpret_cast<uint4 *>(p.out + off);
#pragma unroll 1
        for (int c4 = 0; c4 < kDV / 32; ++c4) {   // 32 output columns at a time
            float o[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c4 * 32, o);
            tmem_wait_ld();
            if (b >= p.B) continue;
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8) {
                float y[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) y[k] = o[v8 * 8 + k];
                if (g4) {
                    const uint4 gv = __ldg(g4 + c4 * 4 + v8);
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        y[2 * k] *= __fdividef(1.f, 1.f + fast_exp2(-__uint_as_float(gw[k] << 16) * kLog2e));
                        y[2 * k + 1] *= __fdividef(1.f, 1.f + fast_exp2(-__uint_as_float(gw[k] & 0xFFFF0000u) * kLog2e));
                    }
                }
                o4[c4 * 4 + v8] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                             pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    MT(5);
    if (warp == 0) tmem_dealloc(tmem, 128);
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

size_t slot_count(int B, int G) { return static_cast<size_t>(G) + static_cast<size_t>(B); }

}  // namespace

// ----------------------------------------------------------------------------- no-alloc scratch
// Scratch for mla_latent_decode_noalloc: callers that cannot call cudaMalloc
// (all device memory is owned by a host framework that hands the library only
// its inputs and outputs, or no allocation may happen after start-up) get the
// decode's partial results kept here instead of in a caller workspace.  Every
// device that loads the library holds this array until the process exits.
// Calls share it: two calls whose kernels overlap on the GPU race on it.
// Nothing in it needs to start at zero: the merge reads only the slots the
// split kernel of the same call wrote.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
constexpr int kMaxDevices = 64;
void *g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;
}  // namespace

size_t decode_noalloc_scratch_capacity() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  Resolved once
// per device (the first call on a device does it), with that device current;
// in host code the array's name is only a stand-in, not a device address.
cudaError_t decode_noalloc_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            // a failed lookup (the module cannot be loaded on this device, or the first call came
            // inside a stream capture) must not leave an error pending for the caller's next CUDA call
            (void)cudaGetLastError();
            return e;
        }
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return cudaSuccess;
}


bool decode_bf16_supports(int H, int d_v, int r) { return r == kR && d_v == kDV && H >= 1 && H <= kHMax; }

namespace {
// Clusters of the pair kernel that run at once on this device, at most one per
// two SMs (a GPC with an odd SM count leaves one SM out).  Queried once per device.
int pair_clusters(int num_sms) {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cached[kMaxDev];
    const int cap = num_sms / 2 > 0 ? num_sms / 2 : 1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = -1;
    if (dev >= 0) {
        const int v = cached[dev].load();
        if (v > 0) return v < cap ? v : cap;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * cap);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemPair;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<false>, &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = cap;
    }
    if (n > cap) n = cap;
    if (dev >= 0) cached[dev].store(n);
    return n;
}
}  // namespace

size_t decode_bf16_workspace_bytes(int B, int H, int r, int, int num_sms) {
    if (r != kR || H < 1 || H > kHMax || B < 1 || num_sms < 1) return 0;
    const size_t slots = slot_count(B, num_sms / 2 > 0 ? num_sms / 2 : 1);
    return slots * static_cast<size_t>(H) * (kR * sizeof(__nv_bfloat16) + 2 * sizeof(float));
}

#ifdef MLA_TRACE
// Diagnostic build only: copy (and optionally clear) the decode wait-accounting slots.
extern "C" __attribute__((visibility("default"))) int mla_debug_decode_trace(unsigned long long *host, int n,
                                                                               int clear) {
    if (n > DT_COUNT) n = DT_COUNT;
    if (cudaMemcpyFromSymbol(host, g_dtrace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
    if (clear) {
        static const unsigned long long zeros[DT_COUNT] = {};
        if (cudaMemcpyToSymbol(g_dtrace, zeros, sizeof(zeros)) != cudaSuccess) return -1;
    }
    return n;
}
// Diagnostic build only: copy the per-block event times of the traced cluster.
extern "C" __attribute__((visibility("default"))) int mla_debug_decode_timeline(long long *host) {
    if (cudaMemcpyFromSymbol(host, g_dtl, sizeof(g_dtl)) != cudaSuccess) return -1;
    return kTLEvents * kTLMax;
}
extern "C" __attribute__((visibility("default"))) int mla_debug_decode_merge(long long *host) {
    if (cudaMemcpyFromSymbol(host, g_mtrace, sizeof(g_mtrace)) != cudaSuccess) return -1;
    return 8 * 1024;
}
extern "C" __attribute__((visibility("default"))) int mla_debug_decode_clusters(long long *host) {
    if (cudaMemcpyFromSymbol(host, g_dclu, sizeof(g_dclu)) != cudaSuccess) return -1;
    return 1024;
}
#endif

namespace {
// q_abs [B][H][512] bf16 -> per row (b, h): 2^e scaling its largest |q_abs| into [128, 256), then e4m3 hi and lo
// parts (hi = e4m3(x), lo = e4m3(x - hi)) as a 1024-byte row [hi | lo], and qmul[b][h] = 2^-e.  A warp per row,
// lane j holds latent columns 16j .. 16j + 15.
__global__ void __launch_bounds__(256) qabs_split_e4m3_kernel(const __nv_bfloat16 *__restrict__ q_abs, uint8_t *__restrict__ q8,
                                                              float *__restrict__ qmul, int rows) {
    const int r = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(q_abs + static_cast<size_t>(r) * kR) + lane * 2;
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16], amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // f16_range_exponent brings the maximum into [2^13, 2^14); 6 fewer gives [2^7, 2^8), inside e4m3's 448
    const int e = amax > 0.f && amax < 3.0e38f ? f16_range_exponent(amax) - 6 : 0;
    const float up = exp2_int(e);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t a = split_e4m3x2(x[4 * k] * up, x[4 * k + 1] * up);
        const uint32_t b = split_e4m3x2(x[4 * k + 2] * up, x[4 * k + 3] * up);
        hw[k] = (a & 0xFFFFu) | (b << 16);
        lw[k] = (a >> 16) | (b & 0xFFFF0000u);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q8 + static_cast<size_t>(r) * 1024);
    dst[lane] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    dst[32 + lane] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    if (lane == 0) qmul[r] = exp2_int(-e);
}

// c [rows][r] bf16 (row stride ld_c) -> c8 = e4m3(c * inv_scale) [rows][r] (row stride ld_c8 bytes): 8 values
// (16 bytes in, 8 out) per thread.
__global__ void __launch_bounds__(256) quantize_latent_e4m3_kernel(const __nv_bfloat16 *__restrict__ c, long long ld_c,
                                                                   uint8_t *__restrict__ c8, long long ld_c8,
                                                                   long long rows, int r, float inv_scale) {
    const long long per_row = r / 8;
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * per_row) return;
    const long long row = i / per_row, g = i % per_row;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(c + row * ld_c) + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t a = cvt_e4m3x2(__uint_as_float(w[2 * k] << 16) * inv_scale,
                                      __uint_as_float(w[2 * k] & 0xFFFF0000u) * inv_scale);
        const uint32_t b = cvt_e4m3x2(__uint_as_float(w[2 * k + 1] << 16) * inv_scale,
                                      __uint_as_float(w[2 * k + 1] & 0xFFFF0000u) * inv_scale);
        o[k] = a | (b << 16);
    }
    *reinterpret_cast<uint2 *>(c8 + row * ld_c8 + g * 8) = make_uint2(o[0], o[1]);
}

CUresult encode_map_u8(CUtensorMap *m, const void *ptr, const cuuint64_t *dims, const cuuint64_t *strides,
                       const cuuint32_t *box) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

size_t partials_bytes(int B, int H, int G) {
    return slot_count(B, G) * static_cast<size_t>(H) * (kR * sizeof(__nv_bfloat16) + 2 * sizeof(float));
}

// The pair kernel (bf16 or e4m3 cache) and the merge, on workspace partials laid out as [o | m | l].
template <bool kF8>
cudaError_t launch_pair_and_merge(const DecodeArgs &a, const void *q_rows, const float *qmul, int G, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<kF8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemPair));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemMerge));
    if (e != cudaSuccess) return e;
    {   // the kernel's register split assumes this launch budget
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, decode_pair_kernel<kF8>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    const size_t slots = slot_count(a.B, G);
    __nv_bfloat16 *ws_o = static_cast<__nv_bfloat16 *>(a.workspace);
    float *ws_m = reinterpret_cast<float *>(ws_o + slots * a.H * kR);
    float *ws_l = ws_m + slots * a.H;
    CUtensorMap tm_c256, tm_c, tm_wuv;
    {
        const cuuint64_t rows = static_cast<cuuint64_t>(a.max_len > 0 ? a.max_len : 1);
        const cuuint64_t es = kF8 ? 1 : 2;   // bytes per cache element
        const cuuint64_t dims[3] = {kR, rows, static_cast<cuuint64_t>(a.B)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.ld_cache) * es, rows * a.ld_cache * es};
        const cuuint32_t box256[3] = {kF8 ? 128u : 64u, kBS, 1};
        const cuuint32_t box64[3] = {kF8 ? 128u : 64u, kVRows, 1};
        if (kF8) {
            if (encode_map_u8(&tm_c256, a.c_cache, dims, strides, box256) != CUDA_SUCCESS ||
                encode_map_u8(&tm_c, a.c_cache, dims, strides, box64) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        } else {
            if (encode_map(&tm_c256, a.c_cache, 3, dims, strides, box256) != CUDA_SUCCESS ||
                encode_map(&tm_c, a.c_cache, 3, dims, strides, box64) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    {
        const cuuint64_t dims[2] = {kR, static_cast<cuuint64_t>(a.H) * kDV};
        const cuuint64_t strides[1] = {kR * 2};
        const cuuint32_t box[2] = {64, kDV};
        if (encode_map(&tm_wuv, a.w_uv, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    PairParams pp;
    pp.lens = a.lens;
    pp.q_abs = static_cast<const __nv_bfloat16 *>(q_rows);
    pp.qmul = qmul;
    pp.cache_scale = a.cache_scale;
    pp.ws_o = ws_o;
    pp.ws_m = ws_m;
    pp.ws_l = ws_l;
    pp.err = a.dev_err;
    pp.B = a.B;
    pp.H = a.H;
    pp.max_len = a.max_len;
    pp.qk_scale_log2 = a.scale * kLog2e;
    decode_pair_kernel<kF8><<<2 * G, kThreads, kSmemPair, s>>>(tm_c256, tm_c, pp);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    MergeParams mp;
    mp.lens = a.lens;
    mp.ws_o = ws_o;
    mp.ws_m = ws_m;
    mp.ws_l = ws_l;
    mp.gate = static_cast<const __nv_bfloat16 *>(a.gate);
    mp.out = static_cast<__nv_bfloat16 *>(a.out);
    mp.err = a.dev_err;
    mp.B = a.B;
    mp.H = a.H;
    mp.max_len = a.max_len;
    mp.G = G;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H, (a.B + kMRows - 1) / kMRows);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = kSmemMerge;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel, tm_wuv, mp);
}
}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
    if (!decode_bf16_supports(a.H, a.d_v, a.r)) return cudaErrorInvalidValue;
    const int G = pair_clusters(a.num_sms);
    if (G > kMaxClusters) return cudaErrorInvalidConfiguration;
    if (partials_bytes(a.B, a.H, G) > a.workspace_bytes) return cudaErrorInvalidValue;
    return launch_pair_and_merge<false>(a, a.q_abs, nullptr, G, s);
}

// Workspace of the e4m3-cache decode: the partials (as for bf16), then the split query rows [B][H][1024 bytes]
// and their multipliers [B][H].
size_t decode_fp8_workspace_bytes(int B, int H, int r, int max_len, int num_sms) {
    const size_t part = decode_bf16_workspace_bytes(B, H, r, max_len, num_sms);
    if (part == 0) return 0;
    const size_t aligned = (part + 255) & ~static_cast<size_t>(255);
    return aligned + static_cast<size_t>(B) * H * (1024 + sizeof(float));
}

cudaError_t launch_decode_fp8(const DecodeArgs &a, cudaStream_t s) {
    if (!decode_bf16_supports(a.H, a.d_v, a.r)) return cudaErrorInvalidValue;
    const int G = pair_clusters(a.num_sms);
    if (G > kMaxClusters) return cudaErrorInvalidConfiguration;
    if (decode_fp8_workspace_bytes(a.B, a.H, a.r, a.max_len, a.num_sms) > a.workspace_bytes)
        return cudaErrorInvalidValue;
    // the split rows start after the largest partials any cluster count needs (G <= num_sms / 2)
    const size_t part = (decode_bf16_workspace_bytes(a.B, a.H, a.r, a.max_len, a.num_sms) + 255) & ~static_cast<size_t>(255);
    uint8_t *q8 = static_cast<uint8_t *>(a.workspace) + part;
    float *qmul = reinterpret_cast<float *>(q8 + static_cast<size_t>(a.B) * a.H * 1024);
    const int rows = a.B * a.H;
    note_launch();
    qabs_split_e4m3_kernel<<<(rows + 7) / 8, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(a.q_abs), q8, qmul, rows);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pair_and_merge<true>(a, q8, qmul, G, s);
}

cudaError_t launch_quantize_latent_e4m3(const void *c, long long ld_c, void *c8, long long ld_c8, long long rows, int r,
                                        float inv_scale, cudaStream_t s) {
    const long long n = rows * (r / 8);
    if (n <= 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    note_launch();
    quantize_latent_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(c), ld_c, static_cast<uint8_t *>(c8), ld_c8, rows, r, inv_scale);
    return cudaGetLastError();
}

}  // namespace mla
