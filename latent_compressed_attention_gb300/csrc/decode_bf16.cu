// bf16 cached-latent decode (one query per sequence) on the sm_103a tensor
// cores: r = 512, d_v = 128, 1 <= H <= 96.
//
// Only the latent c is cached (page "Gated MLA（矩阵吸收版）", KV-cache table in
// section "形状与参数对比": r values per token).  Sequence b's absorbed query
// q_abs[b] (all H heads) attends to its cache rows [0, lens[b]); steps 2-4 of
// section "完整计算流（四步）" follow: scores against c itself, softmax, the
// latent weighting by c itself, W_UV^T, gate.
//
// Split kernel (one CTA per SM, persistent): the concatenation of all
// sequences' cache rows is cut into one contiguous, equal share per CTA, so
// ragged lengths balance by construction.  A CTA walks its share as segments
// (one per sequence it touches) in blocks of 128 rows:
//   S  = q_abs[b] . c_blk^T          M = 128 (heads, zero-padded), N = 128 rows, K = r
//   O^T += c_blk^T . P^T             M = r (4 x 128), N = heads, K = 128 rows
// Heads are rows of S, so the online softmax is one thread per head; the
// latent accumulator is kept transposed (TMEM lanes = latent index, columns =
// heads: 4 x 96 columns), which leaves 128 TMEM columns for S.  Each cache
// row is read from HBM once for all heads; the value product re-reads the
// block's tiles from L2.  Per segment the CTA writes (O^T, running max, sum).
// Merge kernel: one CTA per (head, 64 sequences) combines the segments of a
// sequence with the log-sum-exp rule, rounds o_lat to bf16 and applies W_UV^T
// on the tensor cores, then the sigmoid gate.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kR = 512;
constexpr int kDV = 128;
constexpr int kBN = 128;      // cache rows per block
constexpr int kHMax = 96;
constexpr int kThreads = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
// Largest scratch the no-alloc decode entry point can use (48 MiB: the K3 decode
// workload, B = 64 and H = 96 on 152 SMs, needs 42.6 MB).
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

constexpr uint32_t kSlab = 16384;            // c tile [128 rows x 64 latent columns], 128B swizzle
constexpr uint32_t kQSlab = kHMax * 128;     // q_abs tile [96 heads x 64 latent columns]
constexpr uint32_t kPSlab = kHMax * 128;     // P^T tile [96 heads x 64 cache rows]
constexpr uint32_t Q_OFF = 0;
constexpr uint32_t Q_BYTES = 7 * kQSlab + kSlab;   // an M=128 operand read of the last slab stays inside
constexpr uint32_t RING_OFF = Q_BYTES;
constexpr int kUnits = 3;                    // ring of units, 2 tiles each
constexpr uint32_t kUnit = 2 * kSlab;
constexpr uint32_t P_OFF = RING_OFF + kUnits * kUnit;
constexpr uint32_t FAC_OFF = P_OFF + 2 * kPSlab;
constexpr uint32_t BAR_OFF = FAC_OFF + 128 * 4;
constexpr uint32_t kSmemSplit = BAR_OFF + 256 + 1024;
static_assert(kSmemSplit <= 232448, "split kernel exceeds shared memory");
static_assert(RING_OFF % 1024 == 0 && P_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");

constexpr uint32_t S_COL = 0;     // TMEM columns of S
constexpr uint32_t O_COL = 128;   // TMEM columns of O^T (4 blocks x Hp)

struct SplitBars {
    uint64_t q_full, q_free;
    uint64_t u_full[kUnits], u_empty[kUnits];
    uint64_t s_full, s_free, p_full, pv_done, o_drained;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(SplitBars) <= 256, "barrier block too large");

struct SplitParams {
    const int *lens;
    float *ws_o;   // [slots][H][r]
    float *ws_m;   // [slots][H]
    float *ws_l;   // [slots][H]
    int *err;
    int B, H, Hp, max_len;
    float qk_scale_log2;
};

__device__ __forceinline__ int clamp_len(int x, int max_len) { return min(max(x, 0), max_len); }

// The share of the concatenated cache rows that CTA c of G owns: [lo, hi).
__device__ __forceinline__ long long share_lo(long long total, int c, int G) { return (total * c) / G; }

// Walks the (sequence, [k0, k1)) segments of one CTA's share in order.  All
// roles of the CTA run the same walk, so their ring and barrier counters agree.
struct SegWalk {
    const int *lens;
    int B, max_len;
    long long lo, hi, pre;   // pre = first concatenated row of sequence b
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
            const long long s0 = max(pre, lo), s1 = min(pre + len, hi);
            const long long base = pre;
            const int cur = b;
            pre += len;
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
        t += clamp_len(x, max_len);
    }
    return t;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                        const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    SplitBars *bars = reinterpret_cast<SplitBars *>(gbase + BAR_OFF);
    float *fac = reinterpret_cast<float *>(gbase + FAC_OFF);
    volatile int *abort_flag = &bars->abort;
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int H = p.H, Hp = p.Hp;

    if (threadIdx.x == 0) {
        mbar_init(B_(bars->q_full), 1);
        mbar_init(B_(bars->q_free), 1);
        for (int i = 0; i < kUnits; ++i) {
            mbar_init(B_(bars->u_full[i]), 1);
            mbar_init(B_(bars->u_empty[i]), 1);
        }
        mbar_init(B_(bars->s_full), 1);
        mbar_init(B_(bars->s_free), 128);
        mbar_init(B_(bars->p_full), 1);
        mbar_init(B_(bars->pv_done), 1);
        mbar_init(B_(bars->o_drained), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    const long long total = total_rows(p.lens, p.B, p.max_len, p.err, cta == 0 && threadIdx.x == 0);
    const long long lo = share_lo(total, cta, G), hi = share_lo(total, cta + 1, G);
    SegWalk walk;
    walk.init(p.lens, p.B, p.max_len, lo, hi);
    int seq, k0, k1;

    if (warp == 0 && lane == 0) {
        // ---- producer: q_abs per segment, then ring units in consumption order
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_c);
        uint32_t u = 0, nq = 0;
        bool ok = true;
        while (ok && walk.next(seq, k0, k1)) {
            const int nblk = (k1 - k0 + kBN - 1) / kBN;
            if (nq > 0 && !(ok = mbar_wait(B_(bars->q_free), (nq - 1) & 1, p.err, abort_flag))) break;
            mbar_arrive_expect_tx(B_(bars->q_full), 8u * H * 128u);
            for (int s = 0; s < 8; ++s) tma_load_3d(base + Q_OFF + s * kQSlab, &tm_q, B_(bars->q_full), s * 64, 0, seq);
            ++nq;
            for (int step = 0; ok && step <= nblk; ++step) {
                for (int pass = 0; ok && pass < 2; ++pass) {
                    const bool value = pass == 1;
                    const int blk = value ? step - 1 : step;
                    if (blk < 0 || blk >= nblk) continue;
                    const int key = k0 + blk * kBN;
                    for (int un = 0; un < 4; ++un, ++u) {
                        const int st = u % kUnits;
                        if (u >= kUnits &&
                            !(ok = mbar_wait(B_(bars->u_empty[st]), ((u / kUnits) - 1) & 1, p.err, abort_flag)))
                            break;
                        mbar_arrive_expect_tx(B_(bars->u_full[st]), kUnit);
                        for (int i = 0; i < 2; ++i)
                            tma_load_3d(base + RING_OFF + st * kUnit + i * kSlab, &tm_c, B_(bars->u_full[st]),
                                        (2 * un + i) * 64, key, seq);
                    }
                }
            }
        }
        if (!ok) *abort_flag = 1;
        for (uint32_t k = (u > kUnits ? u - kUnits : 0); k < u; ++k)
            mbar_wait(B_(bars->u_full[k % kUnits]), (k / kUnits) & 1, p.err);
        if (nq > 0) mbar_wait(B_(bars->q_full), (nq - 1) & 1, p.err);
    } else if (warp == 1) {
        // ---- MMA warp: lane 0 issues the tensor-core work; all 32 lanes wait on the
        // ring and, in a sequence's last block, zero the cache rows at or past lens[b]
        // in the value tiles (those rows may hold anything; p = 0 times them must stay 0)
        const uint32_t idesc_s = make_idesc_bf16(128, kBN, 0, 0);
        const uint32_t idesc_o = make_idesc_bf16(128, Hp, 1, 0);
        const bool leader = lane == 0;
        uint32_t u = 0, nq = 0, ns = 0, np = 0, nseg = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t &bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(B_(bar), parity, p.err, abort_flag));
        };
        while (ok && walk.next(seq, k0, k1)) {
            const int nblk = (k1 - k0 + kBN - 1) / kBN;
            const int len = clamp_len(__ldg(p.lens + seq), p.max_len);
            if (!(ok = wait_all(bars->q_full, nq & 1))) break;
            ++nq;
            tc_fence_after();
            for (int step = 0; ok && step <= nblk; ++step) {
                if (step < nblk) {   // S = q_abs . c_blk^T
                    if (ns > 0 && !(ok = wait_all(bars->s_free, (ns - 1) & 1))) break;
                    tc_fence_after();
                    for (int un = 0; ok && un < 4; ++un, ++u) {
                        const int st = u % kUnits;
                        if (!(ok = wait_all(bars->u_full[st], (u / kUnits) & 1))) break;
                        tc_fence_after();
                        if (leader) {
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int kc = 2 * un + i;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t a = make_smem_desc(base + Q_OFF + kc * kQSlab + kk * 32, 16, 1024);
                                    const uint64_t bd =
                                        make_smem_desc(base + RING_OFF + st * kUnit + i * kSlab + kk * 32, 16, 1024);
                                    umma_bf16(tmem + S_COL, a, bd, idesc_s, (kc | kk) != 0);
                                }
                            }
                            umma_commit(B_(bars->u_empty[st]));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (leader) {
                        umma_commit(B_(bars->s_full));
                        if (step == nblk - 1) umma_commit(B_(bars->q_free));
                    }
                    ++ns;
                }
                if (step >= 1) {   // O^T += c_blk^T . P^T for block step-1
                    const int blk = step - 1;
                    const int nvalid = len - (k0 + blk * kBN);   // rows of this block inside the sequence
                    if (step == 1 && nseg > 0 &&   // the previous segment's O^T has been drained
                        !(ok = wait_all(bars->o_drained, (nseg - 1) & 1)))
                        break;
                    if (!(ok = wait_all(bars->p_full, np & 1))) break;
                    ++np;
                    tc_fence_after();
                    for (int rb = 0; ok && rb < 4; ++rb, ++u) {
                        const int st = u % kUnits;
                        if (!(ok = wait_all(bars->u_full[st], (u / kUnits) & 1))) break;
                        if (nvalid < kBN) {
                            for (int i = 0; i < 2; ++i) {
                                const uint32_t tile = base + RING_OFF + st * kUnit + i * kSlab;
                                for (int row = nvalid + lane; row < kBN; row += 32)
#pragma unroll
                                    for (int ch = 0; ch < 8; ++ch)
                                        st_shared_v4(tile + (row >> 3) * 1024 + (row & 7) * 128 + ch * 16, 0, 0, 0, 0);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        tc_fence_after();
                        if (leader) {
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; ++kk) {
                                const uint64_t a =
                                    make_smem_desc(base + RING_OFF + st * kUnit + kk * 2048, kSlab, 1024);
                                const uint64_t bd =
                                    make_smem_desc(base + P_OFF + (kk >> 2) * kPSlab + (kk & 3) * 32, 16, 1024);
                                umma_bf16(tmem + O_COL + rb * Hp, a, bd, idesc_o, (blk > 0 || kk > 0));
                            }
                            umma_commit(B_(bars->u_empty[st]));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (leader) umma_commit(B_(bars->pv_done));
                }
            }
            ++nseg;
        }
        if (!ok && leader) *abort_flag = 1;
    } else if (warp >= 4) {
        // ---- softmax (thread = head row of S) / correction and drain (thread = TMEM lane of O^T)
        const int tid = threadIdx.x - 128;
        const uint32_t tq = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const bool head = tid < H;
        uint32_t ns = 0, npv = 0, nseg = 0;
        bool ok = true;
        const int slot_base = cta;   // segment slot = cta + sequence index
        while (ok && walk.next(seq, k0, k1)) {
            const int nblk = (k1 - k0 + kBN - 1) / kBN;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nblk; ++j) {
                bool fail = !mbar_wait(B_(bars->s_full), ns & 1, p.err, abort_flag);
                if (named_bar_or(1, 128, fail)) { ok = false; break; }
                ++ns;
                tc_fence_after();
                float s[4][32];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(tmem + tq + S_COL + c4 * 32, s[c4]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(B_(bars->s_free));

                const int lim = k1 - (k0 + j * kBN);   // columns < lim are inside the segment
                float factor = 1.f;
                if (head) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            s[c4][i] = c4 * 32 + i < lim ? s[c4][i] * p.qk_scale_log2 : -INFINITY;
                            mx = fmaxf(mx, s[c4][i]);
                        }
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
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int i = 0; i < 32; ++i) s[c4][i] = 0.f;
                }
                // P^T and O^T are free once the previous block's value product completed
                if (j > 0) {
                    fail = !mbar_wait(B_(bars->pv_done), npv & 1, p.err, abort_flag);
                    ++npv;
                }
                fac[tid] = factor;
                if (named_bar_or(1, 128, fail)) { ok = false; break; }
                const bool any = named_bar_or(1, 128, j > 0 && factor != 1.f);
                if (any) {   // rescale columns h of O^T by fac[h]
                    tc_fence_after();
                    for (int rb = 0; rb < 4; ++rb)
                        for (int hc = 0; hc < Hp / 16; ++hc) {
                            float v[16];
                            const uint32_t ta = tmem + tq + O_COL + rb * Hp + hc * 16;
                            tmem_ld16(ta, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] *= fac[hc * 16 + i];
                            tmem_st16(ta, v);
                        }
                    tmem_wait_st();
                    tc_fence_before();
                }
                if (tid < Hp) {   // P^T row `tid` (zeros for padding heads)
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint32_t slab = base + P_OFF + (c4 >> 1) * kPSlab;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float *v = &s[c4][8 * k];
                            st_shared_v4(slab + sw128_offset(tid, (c4 & 1) * 4 + k), pack_bf16x2(v[0], v[1]),
                                         pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                        }
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (tid == 0) mbar_arrive(B_(bars->p_full));
            }
            if (!ok) break;
            // segment end: drain O^T and (m, l) into the workspace slot
            bool fail = !mbar_wait(B_(bars->pv_done), npv & 1, p.err, abort_flag);
            ++npv;
            if (named_bar_or(1, 128, fail)) { ok = false; break; }
            tc_fence_after();
            const size_t slot = static_cast<size_t>(slot_base + seq);
            float *wo = p.ws_o + slot * H * kR;
            for (int rb = 0; rb < 4; ++rb)
                for (int hc = 0; hc < Hp / 16; ++hc) {
                    float v[16];
                    tmem_ld16(tmem + tq + O_COL + rb * Hp + hc * 16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int h = hc * 16 + i;
                        if (h < H) wo[static_cast<size_t>(h) * kR + rb * 128 + tid] = v[i];
                    }
                }
            if (head) {
                p.ws_m[slot * H + tid] = m_run;
                p.ws_l[slot * H + tid] = l_run;
            }
            tc_fence_before();
            named_bar_sync(1, 128);
            if (tid == 0) mbar_arrive(B_(bars->o_drained));
            ++nseg;
        }
        if (!ok) *abort_flag = 1;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------- merge
constexpr int kMRows = 64;                          // sequences per merge CTA
constexpr int kMergeThreads = 512;
constexpr uint32_t kASlab = kMRows * 128;           // o_lat tile [64 rows x 64 latent columns]
constexpr uint32_t MA_OFF = 0;
constexpr uint32_t MA_BYTES = 7 * kASlab + kSlab;   // an M=128 operand read of the last slab stays inside
constexpr uint32_t MW_OFF = MA_BYTES;               // W_UV[h]: 8 tiles [128 x 64]
constexpr uint32_t MBAR_OFF = MW_OFF + 8 * kSlab;
constexpr uint32_t kSmemMerge = MBAR_OFF + 64 + 1024;
static_assert(MW_OFF % 1024 == 0, "alignment");

struct MergeParams {
    const int *lens;
    const float *ws_o, *ws_m, *ws_l;
    const __nv_bfloat16 *gate;
    __nv_bfloat16 *out;
    int *err;
    int B, H, max_len, G;
};

__global__ void __launch_bounds__(kMergeThreads, 1)
    decode_merge_kernel(const __grid_constant__ CUtensorMap tm_wuv, const MergeParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    uint64_t *w_full = reinterpret_cast<uint64_t *>(gbase + MBAR_OFF);
    uint64_t *mma_done = w_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(w_full + 2);
    __shared__ long long s_pre[kMRows + 1];
    __shared__ long long s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, b0 = blockIdx.y * kMRows;
    const int H = p.H;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(w_full), 1);
        mbar_init(smem_u32(mma_done), 1);
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
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_wuv);
        mbar_arrive_expect_tx(smem_u32(w_full), 8 * kSlab);
        for (int s = 0; s < 8; ++s) tma_load_2d(base + MW_OFF + s * kSlab, &tm_wuv, smem_u32(w_full), s * 64, h * kDV);
        // row offsets of this CTA's sequences in the concatenated cache
        long long total = 0;
        for (int b = 0; b < p.B; ++b) {
            const int x = __ldg(p.lens + b);
            if (x < 0 || x > p.max_len) record_error(p.err, kDevErrBounds);
            if (b >= b0 && b <= b0 + kMRows) s_pre[b - b0] = total;
            total += clamp_len(x, p.max_len);
        }
        for (int b = max(p.B, b0); b <= b0 + kMRows; ++b) s_pre[b - b0] = total;
        s_total = total;
    }
    __syncthreads();
    const long long total = s_total;

    // log-sum-exp combine of the segments of each sequence; o_lat -> bf16 tile row.
    // A warp takes a row at a time: lane i fetches segment i's (m, l), the warp
    // reduces them with shuffles, then every lane accumulates its 16 latent
    // columns over the segments, issuing a segment's loads together.
    for (int i = warp; i < kMRows; i += kMergeThreads / 32) {
        const int b = b0 + i;
        float o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k] = 0.f;
        const long long r0 = s_pre[i], r1 = s_pre[i + 1];
        if (b < p.B && r1 > r0) {
            const int G = p.G;
            const int c_first = min(static_cast<int>(((r0 + 1) * G - 1) / total), G - 1);
            // CTA c wrote slot c + b iff its share [lo_c, lo_c+1) overlaps [r0, r1)
            auto overlaps = [&](int c) {
                return c < G && min(share_lo(total, c + 1, G), r1) > max(share_lo(total, c, G), r0);
            };
            int n_seg = 0;   // consecutive CTAs from c_first whose shares start before r1
            while (c_first + n_seg < G && share_lo(total, c_first + n_seg, G) < r1) ++n_seg;
            float M = -INFINITY, L = 0.f;
            for (int s0 = 0; s0 < n_seg; s0 += 32) {
                const int c = c_first + s0 + lane;
                const bool has = s0 + lane < n_seg && overlaps(c);
                const size_t slot = static_cast<size_t>(c + b);
                const float m = has ? __ldg(p.ws_m + slot * H + h) : -INFINITY;
                float mw = m;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
                const float M_new = fmaxf(M, mw);
                float lw = has ? fast_exp2(m - M_new) * __ldg(p.ws_l + slot * H + h) : 0.f;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
                L = (M == -INFINITY ? 0.f : L * fast_exp2(M - M_new)) + lw;
                M = M_new;
            }
            for (int si = 0; si < n_seg; ++si) {
                const int c = c_first + si;
                if (!overlaps(c)) continue;
                const size_t slot = static_cast<size_t>(c + b);
                const float w = fast_exp2(__ldg(p.ws_m + slot * H + h) - M);
                const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + (slot * H + h) * kR + lane * 16);
                float4 v[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) v[q4] = __ldg(src + q4);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    o[4 * q4 + 0] += w * v[q4].x;
                    o[4 * q4 + 1] += w * v[q4].y;
                    o[4 * q4 + 2] += w * v[q4].z;
                    o[4 * q4 + 3] += w * v[q4].w;
                }
            }
            const float inv = 1.f / L;
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] *= inv;
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
    if (threadIdx.x == 0) {
        if (mbar_wait(smem_u32(w_full), 0, p.err)) {
            tc_fence_after();
            const uint32_t idesc = make_idesc_bf16(128, kDV, 0, 0);
#pragma unroll 1
            for (int kk = 0; kk < kR / 16; ++kk) {
                const uint64_t a = make_smem_desc(base + MA_OFF + (kk >> 2) * kASlab + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = make_smem_desc(base + MW_OFF + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
                umma_bf16(tmem, a, bd, idesc, kk > 0);
            }
            umma_commit(smem_u32(mma_done));
        }
    }
    __syncwarp();
    const bool done = mbar_wait(smem_u32(mma_done), 0, p.err);
    tc_fence_after();
    if (warp < 2 && __all_sync(0xffffffffu, done)) {
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
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return cudaSuccess;
}

bool decode_bf16_supports(int H, int d_v, int r) { return r == kR && d_v == kDV && H >= 1 && H <= kHMax; }

size_t decode_bf16_workspace_bytes(int B, int H, int r, int, int num_sms) {
    if (r != kR || H < 1 || H > kHMax || B < 1 || num_sms < 1) return 0;
    const size_t slots = slot_count(B, num_sms);
    return slots * static_cast<size_t>(H) * (kR + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
    if (!decode_bf16_supports(a.H, a.d_v, a.r)) return cudaErrorInvalidValue;
    const int G = a.num_sms;
    const size_t slots = slot_count(a.B, G);
    float *ws_o = static_cast<float *>(a.workspace);
    float *ws_m = ws_o + slots * a.H * kR;
    float *ws_l = ws_m + slots * a.H;
    CUtensorMap tm_q, tm_c, tm_wuv;
    {
        const cuuint64_t dims[3] = {kR, static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.B)};
        const cuuint64_t strides[2] = {kR * 2, static_cast<cuuint64_t>(a.H) * kR * 2};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(a.H), 1};
        if (encode_map(&tm_q, a.q_abs, 3, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {kR, static_cast<cuuint64_t>(a.max_len > 0 ? a.max_len : 1),
                                    static_cast<cuuint64_t>(a.B)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.ld_cache) * 2,
                                       static_cast<cuuint64_t>(a.max_len > 0 ? a.max_len : 1) * a.ld_cache * 2};
        const cuuint32_t box[3] = {64, kBN, 1};
        if (encode_map(&tm_c, a.c_cache, 3, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {kR, static_cast<cuuint64_t>(a.H) * kDV};
        const cuuint64_t strides[1] = {kR * 2};
        const cuuint32_t box[2] = {64, kDV};
        if (encode_map(&tm_wuv, a.w_uv, 2, dims, strides, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    SplitParams sp;
    sp.lens = a.lens;
    sp.ws_o = ws_o;
    sp.ws_m = ws_m;
    sp.ws_l = ws_l;
    sp.err = a.dev_err;
    sp.B = a.B;
    sp.H = a.H;
    sp.Hp = (a.H + 15) / 16 * 16;
    sp.max_len = a.max_len;
    sp.qk_scale_log2 = a.scale * kLog2e;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemSplit));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemMerge));
    if (e != cudaSuccess) return e;
    decode_split_kernel<<<G, kThreads, kSmemSplit, s>>>(tm_q, tm_c, sp);
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
    const dim3 grid(a.H, (a.B + kMRows - 1) / kMRows);
    decode_merge_kernel<<<grid, kMergeThreads, kSmemMerge, s>>>(tm_wuv, mp);
    return cudaGetLastError();
}

}  // namespace mla
