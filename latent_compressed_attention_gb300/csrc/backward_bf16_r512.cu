// Gradients of the absorbed Gated-MLA attention at r = 512, d_q = d_v = 128 on the sm_103a tensor cores.
//
// The page "Gated MLA（矩阵吸收版）" gives the forward only (section "完整计算流（四步）", steps 2-4); this is
// the chain rule back through it, for L = sum(dout * out):
//   sigma = sigmoid(g), do = dout * sigma, dgate = dout * o * sigma * (1 - sigma)   (step 4, o before the gate)
//   do_lat = do . W_UV[h], dW_UV[h] = sum do^T o_lat                                 (step 3, W_UV)
//   dA[t,u] = do_lat_t . c_u, delta_t = sum_u A dA                                     (step 3, A . c)
//   dS = A * (dA - delta) * scale                                                     (softmax, step 2)
//   dq_abs = dS . c, dc += dS^T . q_abs + A^T . do_lat (summed over heads)            (step 2, both uses of c)
//   dq = dq_abs . W_UK[h]^T, dW_UK[h] = sum q^T dq_abs                                (step 2, the absorb)
//
// Design: the forward's output and each row's log-sum-exp lse of the scaled scores are given by the caller
// (saved from its forward) or recomputed by the forward kernel; every product above is then one launch of a
// batched tcgen05 GEMM over materialised per-head matrices: the attention matrix P and the score gradient dS
// ([T, T] per head, bf16, only the causal tiles written or read), q_abs, do_lat, o_lat and dq_abs ([T, r] per
// head, bf16).  The GEMM takes each operand K-major or MN-major through its own TMA tensor map, skips tiles
// above the diagonal, limits K to the causal range of each tile, runs K over a second index (heads for dc,
// sequences for the weight gradients), and fuses the softmax (P = exp2(S scale log2 e - lse log2 e)) and the
// dS epilogues.  fp32 accumulation in TMEM; the gradients are written in fp32, the intermediate matrices in
// bf16.  Two persistent kernels run the products: bwd_gemm_kernel (128-row tiles, one CTA) and
// bwd_gemm2_kernel (256 x 256 tiles on a CTA pair, which halves each SM's shared-memory traffic per product).
//
// delta is the mean of dA under the rounded attention matrix the products use, delta_t = sum_u P dA / sum_u P
// (the numerator is do_lat_t . o_lat_t with o_lat = P . c; both sums come from the P and o_lat epilogues),
// so sum_u P (dA - delta) = 0 holds for the rows as computed.  Taking delta from the rounded output instead
// (do . o) makes dA - delta cancel catastrophically where one key dominates a row.  The partial sums of each
// tile go to slots of their own and are added in a fixed order, so the gradients are the same bits on every
// call.  The scores that rebuild P use q_abs as a bf16 pair hi + lo (about 16 significant bits), as the
// forward's statistics came from a score operand more precise than bf16.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <initializer_list>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kR = 512, kD = 128;
constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr uint32_t kOpBytes = 128 * 128;            // an operand's stage: [128 x 64] K-major or 2 x [64 x 64] MN-major
// warps 0 and 2 TMA (alternate ring positions), warp 1 MMA, then the epilogue warps (thread = row)
constexpr float kLog2e = 1.4426950408889634f;

// The products of the backward.  Operand layouts: "K" = K-major (K contiguous), "MN" = M or N contiguous.
enum Problem : int {
    kQAbs = 0,   // q_abs[z]   = q[b,:,h,:] . W_UK[h]          M=T  N=r   K=d        A K   B MN   bf16 hi, lo [z,T,r]
    kDoLat,      // do_lat[z]  = do[z] . W_UV[h]                M=T  N=r   K=d_v      A K   B MN   bf16
    kP,          // P[z]       = exp2(S - lse), S = q_abs.c^T    M=T  N=T   K=(hi,lo)r A K   B K    bf16 [z,T,Tp]
                 //              (+ this tile's row sums of the rounded P)
    kDS,         // dS[z]      = scale P (do_lat . c^T - delta)  M=T  N=T   K=r        A K   B K    bf16
    kOLat,       // o_lat[z]   = P . c                          M=T  N=r   K=u<=t     A K   B MN   bf16
                 //              (+ this tile's do_lat . o_lat; N tile 0 also adds up P's row sums)
    kDqAbs,      // dq_abs[z]  = dS . c                         M=T  N=r   K=u<=t     A K   B MN   bf16
    kDc,         // dc[b]      = sum_h P^T do_lat + dS^T q_abs   M=T  N=r   K=(h,t>=u) A MN  B MN   f32 [B,T,r]
    kDq,         // dq[b,:,h,:] = dq_abs . W_UK[h]^T             M=T  N=d   K=r        A K   B K    f32 [B,T,H,d]
    kDWuk,       // dW_UK[h]   = sum_b q^T . dq_abs             M=d  N=r   K=(b,t)    A MN  B MN   f32 [H,d,r]
    kDWuv,       // dW_UV[h]   = sum_b do^T . o_lat             M=d_v N=r  K=(b,t)    A MN  B MN   f32 [H,d_v,r]
};

struct GemmP {
    int problem;
    int B, T, H, Tp;      // Tp: row stride of P and dS (T rounded up to 128)
    int M, N;             // output extent of one batch item
    float scale_log2;     // kP: softmax scale * log2(e)
    float scale;          // kDS: softmax scale
    const float *lse;                   // [z, T]: each row's log-sum-exp of the scaled scores (natural log)
    float *psum;                        // [z, T]: row sums of P (o_lat's N tile 0 adds up psum_part)
    float *psum_part;                   // [Tp / 128][z, T]: P's row sums, one slot per key tile
    float *dnum_part;                   // [4][z, T]: do_lat . o_lat, one slot per o_lat N tile
    long long rows;                     // B * H * T
    void *out2;                         // kQAbs: the lo part
    const __nv_bfloat16 *p_in;          // kDS: P
    const __nv_bfloat16 *dl_in;         // kOLat: do_lat
    void *out;
    float *part;                        // split K: part k of a tile's sum at part + k * part_n, out's layout
    long long part_n;                   // elements of one part
    int tile_m;                         // rows of an output tile: 128, or 256 for a CTA pair
    int tile_n;                         // columns of an output tile: 128 or 256
    int nmt, nnt, nz;                   // row tiles, column tiles, batch items
    int ksplit;                         // dc and the weight gradients: parts each tile's K steps are cut into
    int items;                          // work items of the launch
    int *err;
};

__device__ __forceinline__ bool a_mn(int pr) { return pr == kDc || pr == kDWuk || pr == kDWuv; }
__device__ __forceinline__ bool b_mn(int pr) { return pr == kQAbs || pr == kDoLat || pr == kOLat || pr == kDqAbs ||
                                                      pr == kDc || pr == kDWuk || pr == kDWuv; }
__device__ __forceinline__ bool causal_tiles(int pr) { return pr == kP || pr == kDS; }

// The K walk of output tile (m0, z): `outer` runs over a second index (heads for dc, sequences for the weight
// gradients), the inner K over [lo, hi) in steps of 64; dc takes two operand pairs per step.
struct KWalk {
    int outer, lo, hi, pairs;
};
__device__ __forceinline__ KWalk k_walk(const GemmP &p, int m0) {
    switch (p.problem) {
        case kQAbs: case kDoLat: return {1, 0, kD, 1};
        case kP: return {1, 0, kR, 1};                                             // hi and lo in one step
        case kDS: case kDq: return {1, 0, kR, 1};
        case kOLat: case kDqAbs: return {1, 0, min(p.T, m0 + p.tile_m), 1};      // u <= t
        case kDc: return {p.H, m0, p.T, 2};                                        // t >= u, every head
        default: return {p.B, 0, p.T, 1};                                          // kDWuk, kDWuv: every sequence
    }
}

// A work item: output tile (mt, nt) of batch item z, and for a split K the part ks of the tile's K steps.
// The order puts the longest items first where K depends on the row tile, and keeps the items that share
// an operand next to each other (the column tiles of one row tile run side by side).
struct Item {
    int mt, nt, z, ks;
};
__device__ __forceinline__ Item item_of(const GemmP &p, int idx) {
    Item t{0, 0, 0, 0};
    if (causal_tiles(p.problem)) {
        if (p.tile_m == 128 && p.tile_n == 256) {
            // 128-row tiles by 256-column blocks, the lower triangle (block nt starts at or left of the diagonal:
            // nt <= mt / 2) of one batch item after another; row tile mt starts at item C(mt) of its batch item,
            // C(2a) = a (a + 1), C(2a + 1) = (a + 1)^2.  At even mt the diagonal block's right half is zeros.
            const int ntri = p.nmt % 2 == 0 ? (p.nmt / 2) * (p.nmt / 2 + 1) : (p.nmt / 2 + 1) * (p.nmt / 2 + 1);
            t.z = idx / ntri;
            const int r = idx - t.z * ntri;
            int a = static_cast<int>((sqrtf(4.f * static_cast<float>(r) + 1.f) - 1.f) * 0.5f);
            while ((a + 1) * (a + 2) <= r) ++a;
            while (a > 0 && a * (a + 1) > r) --a;
            if (r < a * (a + 1) + a + 1) {
                t.mt = 2 * a;
                t.nt = r - a * (a + 1);
            } else {
                t.mt = 2 * a + 1;
                t.nt = r - (a + 1) * (a + 1);
            }
            return t;
        }
        // The lower triangle (nt <= mt) of one batch item after another.  With 128-row tiles, the items after
        // those are the tiles just above the diagonal at even mt (no K steps: zeros), which the 256-row dc
        // products read.
        const int ntri = p.nmt * (p.nmt + 1) / 2;
        if (p.tile_m == 128 && idx >= p.nz * ntri) {
            const int j = idx - p.nz * ntri, nzt = p.nmt / 2;
            t.z = j / nzt;
            t.mt = 2 * (j % nzt);
            t.nt = t.mt + 1;
            return t;
        }
        t.z = idx / ntri;
        const int r = idx - t.z * ntri;
        int mt = static_cast<int>((sqrtf(8.f * static_cast<float>(r) + 1.f) - 1.f) * 0.5f);
        while ((mt + 1) * (mt + 2) / 2 <= r) ++mt;
        while (mt > 0 && mt * (mt + 1) / 2 > r) --mt;
        t.mt = mt;
        t.nt = r - mt * (mt + 1) / 2;
        return t;
    }
    t.nt = idx % p.nnt;
    const int r = idx / p.nnt;
    switch (p.problem) {
        case kOLat: case kDqAbs:   // K = the causal prefix of the row tile: the last row tiles first
            t.z = r % p.nz;
            t.mt = p.nmt - 1 - r / p.nz;
            break;
        case kDc: {                // K = keys t >= u: the first row tiles first
            const int zk = r % (p.nz * p.ksplit);
            t.mt = r / (p.nz * p.ksplit);
            t.z = zk % p.nz;
            t.ks = zk / p.nz;
            break;
        }
        case kDWuk: case kDWuv:    // a single row tile
            t.z = r % p.nz;
            t.ks = r / p.nz;
            break;
        default:
            t.mt = r % p.nmt;
            t.z = r / p.nmt;
            break;
    }
    return t;
}

// The K steps of an item: steps s_lo .. s_hi - 1 of the tile's walk, step s = (outer o, inner k, pair pr)
// with pr = s % pairs, k = lo + 64 ((s / pairs) % inner), o = s / (pairs inner).
struct Walk {
    int lo, inner, pairs, s_lo, s_hi;
};
__device__ __forceinline__ Walk walk_of(const GemmP &p, const Item &t) {
    const KWalk kw = k_walk(p, t.mt * p.tile_m);
    Walk w;
    w.lo = kw.lo;
    w.pairs = kw.pairs;
    w.inner = kw.hi > kw.lo ? (kw.hi - kw.lo + kBK - 1) / kBK : 0;
    long long total = static_cast<long long>(kw.outer) * w.inner * kw.pairs;
    if (causal_tiles(p.problem) && t.nt * p.tile_n >= (t.mt + 1) * p.tile_m) total = 0;   // a tile of zeros
    w.s_lo = static_cast<int>(total * t.ks / p.ksplit);
    w.s_hi = static_cast<int>(total * (t.ks + 1) / p.ksplit);
    return w;
}

// The item of turn n of a persistent loop for slot `slot` of `slots` (a CTA, or a CTA pair).  Where K depends
// on the row tile (o_lat, dq_abs, dc: heavy-first orders), turn 0 deals items 0 .. slots - 1 in slot order,
// turn 1 the next slots items in reverse order, and so on, so every slot's total comes out about the same (a
// plain stride gives slot 0 the heaviest item of every turn); items of equal K keep the plain stride.
__device__ __forceinline__ int turn_item(const GemmP &p, int n, int slot, int slots) {
    const bool back = (n & 1) && (p.problem == kOLat || p.problem == kDqAbs || p.problem == kDc);
    return n * slots + (back ? slots - 1 - slot : slot);
}

// TMA loads of one K step into stage memory: A at sa, B at sb (each 16 KB).  z: batch item of the output tile,
// o: the outer K index, k: the inner K offset, pair: which operand pair (dc).
template <bool kPair>
__device__ __forceinline__ void tl3(uint32_t dst, const CUtensorMap *m, uint32_t bar, int x, int y, int z) {
    if constexpr (kPair) tma2_load_3d(dst, m, bar, x, y, z);
    else tma_load_3d(dst, m, bar, x, y, z);
}
template <bool kPair>
__device__ __forceinline__ void tl4(uint32_t dst, const CUtensorMap *m, uint32_t bar, int x, int y, int z, int w) {
    if constexpr (kPair) tma2_load_4d(dst, m, bar, x, y, z, w);
    else tma_load_4d(dst, m, bar, x, y, z, w);
}

// (kPair: the loads of one CTA of a pair, completing on the pair's even CTA's barrier `bar`.  nbp: B's columns
// in parts of 128, part j at sb + 16 KB j: MN-major 64-column slabs stay 8 KB apart, K-major rows 128 B apart.)
template <bool kPair>
__device__ __forceinline__ void load_step(const GemmP &p, const CUtensorMap *ta, const CUtensorMap *tb,
                                          const CUtensorMap *ta2, const CUtensorMap *tb2, uint32_t sa, uint32_t sb,
                                          uint32_t bar, int z, int o, int k, int pair, int m0, int n0, int nbp = 1) {
    const int b = p.problem == kDWuk || p.problem == kDWuv ? o : (p.problem == kDc ? z : z / p.H);
    const int h = p.problem == kDc ? o : (p.problem == kDWuk || p.problem == kDWuv ? z : z % p.H);
    const int zz = b * p.H + h;   // head-major batch item of the per-head matrices
    switch (p.problem) {
        case kQAbs:   // A = q [B,T,H,d] (K-major), B = W_UK [H,d,r] (MN-major)
            tl4<kPair>(sa, ta, bar, k, h, m0, b);
            for (int j = 0; j < nbp; ++j)
                for (int s = 0; s < 2; ++s) tl3<kPair>(sb + j * 16384 + s * 8192, tb, bar, n0 + 128 * j + 64 * s, k, h);
            break;
        case kDoLat:  // A = do [z,T,d_v], B = W_UV [H,d_v,r]
            tl3<kPair>(sa, ta, bar, k, m0, zz);
            for (int j = 0; j < nbp; ++j)
                for (int s = 0; s < 2; ++s) tl3<kPair>(sb + j * 16384 + s * 8192, tb, bar, n0 + 128 * j + 64 * s, k, h);
            break;
        case kP:   // A = q_abs [z,T,r] (K-major): hi at sa, lo at sa + 16 KB; B = c [B,T,r] (K-major, rows u)
            tl3<kPair>(sa, ta, bar, k, m0, zz);
            tl3<kPair>(sa + kOpBytes, ta2, bar, k, m0, zz);
            for (int j = 0; j < nbp; ++j) tl3<kPair>(sb + j * 16384, tb, bar, k, n0 + 128 * j, b);
            break;
        case kDS:   // A = do_lat [z,T,r] (K-major), B = c [B,T,r] (K-major, rows u)
            tl3<kPair>(sa, ta, bar, k, m0, zz);
            for (int j = 0; j < nbp; ++j) tl3<kPair>(sb + j * 16384, tb, bar, k, n0 + 128 * j, b);
            break;
        case kOLat: case kDqAbs:   // A = P or dS [z,T,Tp] (K-major over u), B = c [B,T,r] (MN-major: rows u;
                                   // slab map: both 64-column slabs of a part in one box)
            tl3<kPair>(sa, ta, bar, k, m0, zz);
            for (int j = 0; j < nbp; ++j) tl4<kPair>(sb + j * 16384, tb, bar, 0, k, (n0 + 128 * j) / 64, b);
            break;
        case kDc: {   // A = P^T or dS^T (MN-major: rows t, u contiguous), B = do_lat or q_abs (MN-major: rows t);
                      // slab maps: both 64-column slabs of an operand part in one box
            const CUtensorMap *a = pair ? ta2 : ta, *bm = pair ? tb2 : tb;
            tl4<kPair>(sa, a, bar, 0, k, m0 / 64, zz);
            for (int j = 0; j < nbp; ++j) tl4<kPair>(sb + j * 16384, bm, bar, 0, k, (n0 + 128 * j) / 64, zz);
            break;
        }
        case kDq:   // A = dq_abs [z,T,r] (K-major), B = W_UK [H,d,r] (K-major: rows d)
            tl3<kPair>(sa, ta, bar, k, m0, zz);
            for (int j = 0; j < nbp; ++j) tl3<kPair>(sb + j * 16384, tb, bar, k, n0 + 128 * j, h);
            break;
        case kDWuk:   // A = q^T (MN-major: rows t, d contiguous), B = dq_abs (MN-major: rows t)
            for (int s = 0; s < 2; ++s) tl4<kPair>(sa + s * 8192, ta, bar, m0 + 64 * s, h, k, b);
            for (int j = 0; j < nbp; ++j)
                for (int s = 0; s < 2; ++s) tl3<kPair>(sb + j * 16384 + s * 8192, tb, bar, n0 + 128 * j + 64 * s, k, zz);
            break;
        default:   // kDWuv: A = do^T (MN-major: rows t), B = o_lat (MN-major: rows t)
            for (int s = 0; s < 2; ++s) tl3<kPair>(sa + s * 8192, ta, bar, m0 + 64 * s, k, zz);
            for (int j = 0; j < nbp; ++j)
                for (int s = 0; s < 2; ++s) tl3<kPair>(sb + j * 16384 + s * 8192, tb, bar, n0 + 128 * j + 64 * s, k, zz);
            break;
    }
}

// The epilogue's per-row inputs of an item, read before its sums are ready: the softmax statistics (P) or
// delta (dS).
struct RowIn {
    float mrow, inv_l, drow;
};
__device__ __forceinline__ void read_row_stats(const GemmP &p, int z, int m, RowIn &r) {
    const int pr = p.problem;
    r.mrow = r.inv_l = r.drow = 0.f;
    if (m >= p.M) return;
    const size_t ri = static_cast<size_t>(z) * p.T + m;
    if (pr == kP) {
        r.mrow = __ldg(p.lse + ri) * kLog2e;   // P = exp2(s scale log2 e - lse log2 e)
        r.inv_l = 1.f;
    } else if (pr == kDS) {   // written by earlier launches, added in a fixed order
        float num = 0.f;
#pragma unroll
        for (int q = 0; q < kR / kBN; ++q) num += p.dnum_part[q * p.rows + ri];
        r.drow = num / p.psum[ri];
    }
}
// 32 bf16 of row m's P (dS) or do_lat (o_lat) from column nb, for the chunk of the epilogue that needs them.
__device__ __forceinline__ void read_chunk_input(const GemmP &p, int z, int m, int nb, uint4 (&in)[4]) {
    const int pr = p.problem;
    if (m >= p.M || (pr != kDS && pr != kOLat)) return;
    const size_t ri = static_cast<size_t>(z) * p.T + m;
    const uint4 *src = reinterpret_cast<const uint4 *>(pr == kDS ? p.p_in + ri * p.Tp + nb : p.dl_in + ri * kR + nb);
    ld_global_32B(src, in[0], in[1]);
    ld_global_32B(src + 2, in[2], in[3]);
}

// One 32-column chunk of an item's epilogue: row m of batch item z, columns nb .. nb + 31, the fp32 sums v.
// (mrow, inv_l: the row's softmax statistics for P; drow: its delta for dS; rsum: the row's running sum of
// P as rounded, or of do_lat . o_lat; ks: the K part of a split item; in: the chunk's 32 bf16 of P (dS) or of
// do_lat (o_lat).)
__device__ __forceinline__ void epilogue_chunk(const GemmP &p, int z, int m, int nb, int ks, float (&v)[32], float mrow,
                                               float inv_l, float drow, float &rsum, const uint4 (&in)[4]) {
    const int pr = p.problem;
    // P and dS rows are written out to their padded width Tp (zeros past the diagonal): the products
    // that read them take K in steps of 64 up to the end of the diagonal tile
    if (m >= p.M || nb >= ((pr == kP || pr == kDS) ? p.Tp : p.N)) return;
    if (pr == kP || pr == kDS) {
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + (static_cast<size_t>(z) * p.T + m) * p.Tp + nb;
        float pv[32];
        if (pr == kDS) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = in[q];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pv[8 * q + 2 * e] = __uint_as_float(ww[e] << 16);
                    pv[8 * q + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const bool vis = nb + i <= m;   // causal: key u <= query t
            if (pr == kP)
                v[i] = vis ? fast_exp2(fmaf(v[i], p.scale_log2, -mrow)) * inv_l : 0.f;
            else
                v[i] = vis ? p.scale * pv[i] * (v[i] - drow) : 0.f;
        }
        uint4 *o4 = reinterpret_cast<uint4 *>(o);
        uint4 w4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t wq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                wq[e] = pack_bf16x2(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
                if (pr == kP)   // the row sum of P as rounded
                    rsum += __uint_as_float(wq[e] << 16) + __uint_as_float(wq[e] & 0xFFFF0000u);
            }
            w4[q] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
        st_global_32B(o4, w4[0], w4[1]);
        st_global_32B(o4 + 2, w4[2], w4[3]);
    } else if (pr <= kDqAbs) {   // bf16 [z, T, r]
        if (pr == kQAbs) {   // the lo part: bf16(x - bf16(x))
            uint4 *l4 = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out2) +
                                                  (static_cast<size_t>(z) * p.T + m) * kR + nb);
            uint4 lo4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = v[8 * q + 2 * e], x1 = v[8 * q + 2 * e + 1];
                    const uint32_t hw = pack_bf16x2(x0, x1);
                    lw[e] = pack_bf16x2(x0 - __uint_as_float(hw << 16), x1 - __uint_as_float(hw & 0xFFFF0000u));
                }
                lo4[q] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            st_global_32B(l4, lo4[0], lo4[1]);
            st_global_32B(l4 + 2, lo4[2], lo4[3]);
        }
        if (pr == kOLat) {   // do_lat . o_lat over these 32 columns
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = in[q];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    rsum += v[8 * q + 2 * e] * __uint_as_float(ww[e] << 16) +
                            v[8 * q + 2 * e + 1] * __uint_as_float(ww[e] & 0xFFFF0000u);
            }
        }
        uint4 *o4 = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                              (static_cast<size_t>(z) * p.T + m) * kR + nb);
        uint4 b4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            b4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        st_global_32B(o4, b4[0], b4[1]);
        st_global_32B(o4 + 2, b4[2], b4[3]);
    } else {   // fp32 gradients
        size_t off;
        if (pr == kDc) off = (static_cast<size_t>(z) * p.T + m) * kR + nb;
        else if (pr == kDq) off = ((static_cast<size_t>(z / p.H) * p.T + m) * p.H + z % p.H) * kD + nb;
        else off = (static_cast<size_t>(z) * p.M + m) * kR + nb;   // dW_UK, dW_UV [H, 128, r]
        float *dst = p.ksplit > 1 ? p.part + static_cast<size_t>(ks) * p.part_n : static_cast<float *>(p.out);
        float *o = dst + off;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            st_global_32B(o + 8 * q,
                          make_uint4(__float_as_uint(v[8 * q]), __float_as_uint(v[8 * q + 1]), __float_as_uint(v[8 * q + 2]),
                                     __float_as_uint(v[8 * q + 3])),
                          make_uint4(__float_as_uint(v[8 * q + 4]), __float_as_uint(v[8 * q + 5]),
                                     __float_as_uint(v[8 * q + 6]), __float_as_uint(v[8 * q + 7])));
    }
}

// After the chunks of a row: the row sum of the rounded P over one 128-column key tile (slot = the key tile),
// or do_lat . o_lat over one 128-column tile of o_lat (slot = that tile); the o_lat tile of columns 0-127 also
// adds up P's slots of key tiles 0 .. m / 128, in order.
__device__ __forceinline__ void epilogue_row(const GemmP &p, int z, int m, int slot, float rsum) {
    const int pr = p.problem;
    if (m >= p.M) return;
    const size_t ri = static_cast<size_t>(z) * p.T + m;
    if (pr == kP && slot < p.Tp / kBM) p.psum_part[static_cast<size_t>(slot) * p.rows + ri] = rsum;
    if (pr == kOLat) {
        p.dnum_part[static_cast<size_t>(slot) * p.rows + ri] = rsum;
        if (slot == 0) {   // the P launch has finished
            float ps = 0.f;
            for (int j = 0; j <= m / kBM; ++j) ps += p.psum_part[static_cast<size_t>(j) * p.rows + ri];
            p.psum[ri] = ps;
        }
    }
}

// Persistent: CTA i takes item i, then 2G - 1 - i or i + G, ... (G = the grid; turn_item).  The TMA ring runs on
// across items, and the accumulator alternates between two kW-column halves of the CTA's TMEM, so one item's
// epilogue overlaps the next item's products.  kW = 128: 128 x 128 tiles, two CTAs per SM; kW = 256: 128 x 256
// tiles (B staged as two 128-column parts, 87 instead of 64 FLOPs per staged byte), one CTA per SM, two epilogue
// column groups.
// kNA: A operands of a K step (2 for P: the hi and lo parts of q_abs against one c tile, so c is staged once
// for both products).  kPIn (dS): the item's tile of P [128 x kW] is staged in shared memory by TMA for the
// epilogue, which would otherwise wait on its rows' global loads.
template <int kW, int kNA = 1, bool kPIn = false>
struct Shape {
    static constexpr int kStagesW = kW == 256 && kNA == 1 && !kPIn ? 4 : 3;
    static constexpr uint32_t kBOff = kNA * kOpBytes;          // B's offset in a stage
    static constexpr uint32_t kStageW = kBOff + kW * 128;      // A [128 x 64] (kNA of them) + B [kW x 64]
    static constexpr uint32_t kPOff = kStagesW * kStageW;      // the P tile: kW / 64 boxes [128 x 64]
    static constexpr uint32_t kPBytes = kPIn ? 128 * kW * 2 : 0;
    static constexpr uint32_t kBarOffW = kPOff + kPBytes;
    static constexpr uint32_t kSmemW = kBarOffW + 256 + 1024;
    static constexpr int kGroups = kW / 128;                   // epilogue column groups of four warps
    static constexpr int kThreadsW = 96 + 128 * kGroups;       // warps 0 and 2 TMA, warp 1 MMA, then the epilogue
    static constexpr int kMinBlocks = kW == 256 ? 1 : 2;
};
static_assert(Shape<256>::kSmemW <= 232448 && Shape<256, 2>::kSmemW <= 232448 &&
                  Shape<256, 1, true>::kSmemW <= 232448 && 2 * Shape<128>::kSmemW <= 233472,
              "shared memory");

template <int kW, int kNA, bool kPIn>
__global__ void __launch_bounds__(Shape<kW, kNA, kPIn>::kThreadsW, Shape<kW, kNA, kPIn>::kMinBlocks)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_b2,
                    const GemmP p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    using S = Shape<kW, kNA, kPIn>;
    constexpr int kStages = S::kStagesW;
    constexpr uint32_t kStageBytes = S::kStageW;
    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + S::kBarOffW);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;     // [2] the accumulator holds an item's finished sums
    uint64_t *acc_empty = acc_full + 2;       // [2] the epilogue has read them out
    uint64_t *p_full = acc_empty + 2;         // kPIn: the P tile has landed
    uint64_t *p_empty = p_full + 1;           // kPIn: every epilogue warp has read it
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(p_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(acc_full + i), 1);
            mbar_init(smem_u32(acc_empty + i), 128 * S::kGroups);
        }
        mbar_init(smem_u32(p_full), 1);
        mbar_init(smem_u32(p_empty), 4 * S::kGroups);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 2 * kW);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if ((warp == 0 || warp == 2) && lane == 0) {
        // two producers, on alternate ring positions: one thread's TMA issues are too slow to keep the ring full
        const int pi = warp >> 1;
        if (pi == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
        }
        bool ok = true;
        int it = 0;
        const int slot = static_cast<int>(blockIdx.x);
        for (int turn = 0, idx = slot; ok && idx < p.items; idx = turn_item(p, ++turn, slot, G)) {
            const Item t = item_of(p, idx);
            const Walk w = walk_of(p, t);
            for (int s = w.s_lo; s < w.s_hi; ++s, ++it) {
                if ((it & 1) != pi) continue;
                const int st = it % kStages;
                if (it >= kStages && !(ok = mbar_wait(smem_u32(empty + st), ((it / kStages) - 1) & 1, p.err, abort_flag)))
                    break;
                const int pr = s % w.pairs, s2 = s / w.pairs;
                const uint32_t bar = smem_u32(full + st);
                mbar_arrive_expect_tx(bar, kStageBytes);
                load_step<false>(p, &tm_a, &tm_b, &tm_a2, &tm_b2, base + st * kStageBytes, base + st * kStageBytes + S::kBOff,
                                 bar, t.z, s2 / w.inner, w.lo + (s2 % w.inner) * kBK, pr, t.mt * kBM, t.nt * kW,
                                 S::kGroups);
            }
        }
        if (!ok) *abort_flag = 1;
        for (int q = (it > kStages ? it - kStages : 0); q < it; ++q)   // no load may still be landing at exit
            if ((q & 1) == pi) mbar_wait(smem_u32(full + q % kStages), (q / kStages) & 1, p.err);
    } else if (warp == 1 && lane == 0) {
        const bool amn = a_mn(p.problem), bmn = b_mn(p.problem);
        const uint32_t idesc = make_idesc_bf16(128, kW, amn ? 1 : 0, bmn ? 1 : 0);
        // descriptors of stage 0; a stage and a K step of 16 move them by constant offsets (MN-major operands:
        // two 64-wide slabs 8 KB apart, 2 KB per K step; K-major: 32 bytes per K step), so the issue loop is
        // one add per operand per MMA
        const uint64_t a0 = make_smem_desc(base, amn ? 8192 : 16, 1024);
        const uint64_t b0 = make_smem_desc(base + S::kBOff, bmn ? 8192 : 16, 1024);
        const uint32_t a_step = amn ? 2048u : 32u, b_step = bmn ? 2048u : 32u;
        bool ok = true;
        int it = 0, lt = 0;
        const int slot = static_cast<int>(blockIdx.x);
        for (int turn = 0, idx = slot; ok && idx < p.items; idx = turn_item(p, ++turn, slot, G), ++lt) {
            const Walk w = walk_of(p, item_of(p, idx));
            const int acc = lt & 1;
            if (!(ok = mbar_wait(smem_u32(acc_empty + acc), ((lt >> 1) & 1) ^ 1, p.err, abort_flag))) break;
            tc_fence_after();
            const uint32_t d = tmem + acc * kW;
            const int n = w.s_hi - w.s_lo;
            for (int j = 0; j < n; ++j, ++it) {
                const int st = it % kStages;
                if (!(ok = mbar_wait(smem_u32(full + st), (it / kStages) & 1, p.err, abort_flag))) break;
                tc_fence_after();
                const uint64_t as = desc_add(a0, st * kStageBytes), bs = desc_add(b0, st * kStageBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    umma_bf16(d, desc_add(as, kk * a_step), desc_add(bs, kk * b_step), idesc, (j | kk) != 0);
                    if constexpr (kNA == 2)   // the lo part against the same B slice
                        umma_bf16(d, desc_add(as, kOpBytes + kk * a_step), desc_add(bs, kk * b_step), idesc, true);
                }
                umma_commit(smem_u32(empty + st));
            }
            if (!ok) break;
            if (n > 0) umma_commit(smem_u32(acc_full + acc));
            else mbar_arrive(smem_u32(acc_full + acc));   // nothing to add up: the epilogue writes zeros
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 3) {
        // epilogue: thread `row` owns TMEM lane row (warp w reads lanes 32 (w % 4) .. + 31) and columns
        // 128 g .. 128 g + 127 of the accumulator, g = (w - 3) / 4
        const int g = (warp - 3) >> 2;
        const int row = (warp & 3) * 32 + lane;
        // kPIn: thread (warp 3, lane 0) loads each item's P tile, the first before the loop and the next one once
        // every epilogue warp has read the current one
        const bool p_loader = kPIn && warp == 3 && lane == 0;
        const uint32_t p_base = base + S::kPOff;
        int p_loads = 0, p_landed = 0;
        auto load_p = [&](int pidx) {
            const Item u = item_of(p, pidx);
            const uint32_t bar = smem_u32(p_full);
            mbar_arrive_expect_tx(bar, S::kPBytes);
#pragma unroll
            for (int j = 0; j < kW / 64; ++j)
                tma_load_3d(p_base + j * 16384, &tm_a2, bar, u.nt * kW + 64 * j, u.mt * kBM, u.z);
            ++p_loads;
        };
        if (p_loader && static_cast<int>(blockIdx.x) < p.items) load_p(static_cast<int>(blockIdx.x));
        int lt = 0;
        const int slot = static_cast<int>(blockIdx.x);
        for (int turn = 0, idx = slot; idx < p.items; idx = turn_item(p, ++turn, slot, G), ++lt) {
            const Item t = item_of(p, idx);
            const Walk w = walk_of(p, t);
            const bool any = w.s_hi > w.s_lo;
            const int acc = lt & 1;
            const int z = t.z;
            const int m = t.mt * kBM + row, n0 = t.nt * kW + 128 * g;
            const uint32_t trow = tmem + acc * kW + 128 * g + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            RowIn rin;
            uint4 cur[4], nxt[4];
            read_row_stats(p, z, m, rin);   // in flight while the products finish
            if constexpr (!kPIn) read_chunk_input(p, z, m, n0, cur);
            bool ok = mbar_wait(smem_u32(acc_full + acc), (lt >> 1) & 1, p.err, abort_flag);
            if constexpr (kPIn) {
                ok = ok && mbar_wait(smem_u32(p_full), lt & 1, p.err, abort_flag);
                if (ok && p_loader) ++p_landed;
            }
            if (!ok) *abort_flag = 1;   // every later wait of every role then returns at once
            tc_fence_after();
            if (!__all_sync(0xffffffffu, ok)) break;
            float rsum = 0.f;
            if (!any) {   // the accumulator was not touched: release it now
                tc_fence_before();
                mbar_arrive(smem_u32(acc_empty + acc));
            }
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                if constexpr (kPIn) {   // this chunk's 64 bytes of the row, from the 128-byte-swizzled boxes
                    const int cb = 128 * g + 32 * c4;
                    const uint32_t rb = p_base + (cb >> 6) * 16384 + row * 128;
                    const int j0 = (cb & 63) >> 3;
#pragma unroll
                    for (int q = 0; q < 4; ++q) cur[q] = ld_shared_v4(rb + (((j0 + q) ^ (row & 7)) << 4));
                    if (c4 == 3) {   // this warp is done with the P tile
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(p_empty));
                        __syncwarp();   // converged again for the TMEM load
                    }
                } else if (c4 < 3) {
                    read_chunk_input(p, z, m, n0 + (c4 + 1) * 32, nxt);   // one chunk ahead
                }
                float v[32];
                if (any) {
                    tmem_ld32(trow + c4 * 32, v);
                    tmem_wait_ld();
                    if (c4 == 3) {   // every column is in registers: the next item may accumulate here
                        tc_fence_before();
                        mbar_arrive(smem_u32(acc_empty + acc));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                epilogue_chunk(p, z, m, n0 + c4 * 32, t.ks, v, rin.mrow, rin.inv_l, rin.drow, rsum, cur);
                if constexpr (!kPIn) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
                }
            }
            epilogue_row(p, z, m, t.nt * S::kGroups + g, rsum);
            if (p_loader && turn_item(p, turn + 1, slot, G) < p.items) {
                if (!mbar_wait(smem_u32(p_empty), lt & 1, p.err, abort_flag)) {
                    *abort_flag = 1;
                } else {
                    fence_proxy_async_smem();   // the warps' reads of the tile come before the TMA overwrites it
                    load_p(turn_item(p, turn + 1, slot, G));
                }
            }
        }
        if (p_loader)   // no load of the P tile may still be landing at exit
            for (int q = p_landed; q < p_loads; ++q) mbar_wait(smem_u32(p_full), q & 1, p.err);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * kW);
}

// The pair form: a cluster of two CTAs, one per SM, computes 256 x 256 tiles with cta_group::2 MMAs.  CTA r of
// the pair stages rows 128 r .. 128 r + 127 of the tile's A and columns 128 r .. 128 r + 127 of its B, so each SM
// loads 32 KB per K step of 64 for twice the products of a 128 x 128 tile, and holds rows 128 r .. 128 r + 127 of
// the 256 x 256 sums in TMEM (two 256-column accumulators).  Per SM the tensor core reads 8 KB of shared memory
// per 16-deep product instead of the 12 KB of a 128 x 256 tile, which with the TMA writes keeps the SM's
// shared-memory traffic under its bandwidth at the full product rate.  The even CTA issues the MMAs; both CTAs'
// loads complete on its barriers, its commits arrive on both CTAs' barriers, and both CTAs' epilogue warps report
// to it when an accumulator is read.  kNA = 2 (P): each CTA stages both q_abs parts with its half of the c tile.
template <int kNA>
struct Shape2 {
    static constexpr int kStages = kNA == 2 ? 4 : 6;
    static constexpr uint32_t kBOff = kNA * kOpBytes;
    static constexpr uint32_t kStage = kBOff + kOpBytes;
    static constexpr uint32_t kSmem = kStages * kStage + 256 + 1024;   // one CTA per SM
};
constexpr int kThreads2 = 352;   // warps 0 and 2 TMA, warp 1 MMA (even CTA), warps 3-10 epilogue (two column halves)
static_assert(Shape2<1>::kSmem <= 232448 && Shape2<2>::kSmem <= 232448, "exceeds the 227 KB shared-memory limit");

template <int kNA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads2, 1)
    bwd_gemm2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_b2,
                     const GemmP p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    using S2 = Shape2<kNA>;
    constexpr int kStages2 = S2::kStages;
    constexpr uint32_t kStageBytes = S2::kStage;
    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + kStages2 * kStageBytes);   // even CTA: both CTAs' loads
    uint64_t *empty = full + kStages2;         // each CTA's own: the stage's products completed
    uint64_t *acc_full = empty + kStages2;     // [2] each CTA's own: the accumulator holds an item's sums
    uint64_t *acc_empty = acc_full + 2;        // [2] even CTA: every epilogue warp of both CTAs has read it out
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0: the pair's MMA issuer
    const int pair_id = static_cast<int>(blockIdx.x) >> 1, n_pairs = static_cast<int>(gridDim.x) >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages2; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(acc_full + i), 1);
            mbar_init(smem_u32(acc_empty + i), 16);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {   // one warp of each CTA of the pair, together
        tmem_alloc2(smem_u32(tmem_slot), 512);
        tmem_relinquish2();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers exist before any remote arrival or load
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if ((warp == 0 || warp == 2) && lane == 0) {
        const int pi = warp >> 1;   // two producers, on alternate ring positions
        if (pi == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
        }
        bool ok = true;
        int it = 0;
        for (int turn = 0, idx = pair_id;
             ok && idx < p.items; idx = turn_item(p, ++turn, pair_id, n_pairs)) {
            const Item t = item_of(p, idx);
            const Walk w = walk_of(p, t);
            for (int s = w.s_lo; s < w.s_hi; ++s, ++it) {
                if ((it & 1) != pi) continue;
                const int st = it % kStages2;
                if (it >= kStages2 &&
                    !(ok = mbar_wait(smem_u32(empty + st), ((it / kStages2) - 1) & 1, p.err, abort_flag)))
                    break;
                const int pr = s % w.pairs, s2 = s / w.pairs;
                if (rank == 0) mbar_arrive_expect_tx(smem_u32(full + st), 2 * kStageBytes);
                load_step<true>(p, &tm_a, &tm_b, &tm_a2, &tm_b2, base + st * kStageBytes,
                                base + st * kStageBytes + S2::kBOff, mapa_shared(smem_u32(full + st), 0), t.z,
                                s2 / w.inner, w.lo + (s2 % w.inner) * kBK, pr, t.mt * 256 + 128 * rank,
                                t.nt * 256 + 128 * rank);
            }
        }
        if (!ok) *abort_flag = 1;
        if (rank == 0)   // no load of either CTA may still be landing at exit
            for (int q = (it > kStages2 ? it - kStages2 : 0); q < it; ++q)
                if ((q & 1) == pi) mbar_wait(smem_u32(full + q % kStages2), (q / kStages2) & 1, p.err);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        const bool amn = a_mn(p.problem), bmn = b_mn(p.problem);
        const uint32_t idesc = make_idesc_bf16(256, 256, amn ? 1 : 0, bmn ? 1 : 0);
        const uint64_t a0 = make_smem_desc(base, amn ? 8192 : 16, 1024);
        const uint64_t b0 = make_smem_desc(base + S2::kBOff, bmn ? 8192 : 16, 1024);
        const uint32_t a_step = amn ? 2048u : 32u, b_step = bmn ? 2048u : 32u;
        bool ok = true;
        int it = 0, lt = 0;
        for (int turn = 0, idx = pair_id;
             ok && idx < p.items; idx = turn_item(p, ++turn, pair_id, n_pairs), ++lt) {
            const Walk w = walk_of(p, item_of(p, idx));
            const int acc = lt & 1;
            if (!(ok = mbar_wait(smem_u32(acc_empty + acc), ((lt >> 1) & 1) ^ 1, p.err, abort_flag))) break;
            tc_fence_after();
            const uint32_t d = tmem + acc * 256;
            const int n = w.s_hi - w.s_lo;
            for (int j = 0; j < n; ++j, ++it) {
                const int st = it % kStages2;
                if (!(ok = mbar_wait(smem_u32(full + st), (it / kStages2) & 1, p.err, abort_flag))) break;
                tc_fence_after();
                const uint64_t as = desc_add(a0, st * kStageBytes), bs = desc_add(b0, st * kStageBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    umma2(d, desc_add(as, kk * a_step), desc_add(bs, kk * b_step), idesc, (j | kk) != 0);
                    if constexpr (kNA == 2)   // the lo part against the same B slice
                        umma2(d, desc_add(as, kOpBytes + kk * a_step), desc_add(bs, kk * b_step), idesc, true);
                }
                umma2_commit(smem_u32(empty + st), 0x3);
            }
            if (!ok) break;
            if (n > 0) {
                umma2_commit(smem_u32(acc_full + acc), 0x3);
            } else {   // nothing to add up: both CTAs' epilogues write zeros
                mbar_arrive(smem_u32(acc_full + acc));
                mbar_arrive_remote(smem_u32(acc_full + acc), 1);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 3) {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (this CTA's rows of the tile) and columns
        // 128 g .. 128 g + 127 of the accumulator, g = (w - 3) / 4
        const int g = (warp - 3) >> 2;
        const int row = (warp & 3) * 32 + lane;
        int lt = 0;
        for (int turn = 0, idx = pair_id;
             idx < p.items; idx = turn_item(p, ++turn, pair_id, n_pairs), ++lt) {
            const Item t = item_of(p, idx);
            const Walk w = walk_of(p, t);
            const bool any = w.s_hi > w.s_lo;
            const int acc = lt & 1;
            const int z = t.z;
            const int m = t.mt * 256 + 128 * static_cast<int>(rank) + row, n0 = t.nt * 256 + 128 * g;
            const uint32_t trow = tmem + acc * 256 + 128 * g + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            RowIn rin;
            uint4 cur[4], nxt[4];
            read_row_stats(p, z, m, rin);   // in flight while the products finish
            read_chunk_input(p, z, m, n0, cur);
            const bool ok = mbar_wait(smem_u32(acc_full + acc), (lt >> 1) & 1, p.err, abort_flag);
            if (!ok) *abort_flag = 1;
            tc_fence_after();
            if (!__all_sync(0xffffffffu, ok)) break;
            float rsum = 0.f;
            auto release = [&]() {   // this warp has read its part of the accumulator
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(smem_u32(acc_empty + acc));
                    else mbar_arrive_remote(smem_u32(acc_empty + acc), 0);
                }
            };
            if (!any) release();
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                if (c4 < 3) read_chunk_input(p, z, m, n0 + (c4 + 1) * 32, nxt);   // one chunk ahead
                float v[32];
                if (any) {
                    tmem_ld32(trow + c4 * 32, v);
                    tmem_wait_ld();
                    if (c4 == 3) release();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                epilogue_chunk(p, z, m, n0 + c4 * 32, t.ks, v, rin.mrow, rin.inv_l, rin.drow, rsum, cur);
#pragma unroll
                for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
            }
            epilogue_row(p, z, m, 2 * t.nt + g, rsum);
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();   // no pair product is in flight and neither CTA reads the other's barriers any more
    if (warp == 1) tmem_dealloc2(tmem, 512);
    cluster_sync_all();
}

// do = dout * sigmoid(g) (head-major [z, T, d_v] bf16) and dgate = dout * o * sigmoid(g) (1 - sigmoid(g)) (fp32,
// [B, T, H d_v]), o the output before the gate; given the output after the gate instead (gated: out = o sigmoid(g)),
// dgate = dout * out * (1 - sigmoid(g)).  One warp per (b, t, h), lane j holds columns 4j .. 4j + 3.
__global__ void __launch_bounds__(256) bwd_gate_kernel(const __nv_bfloat16 *__restrict__ dout, const __nv_bfloat16 *__restrict__ g,
                                                       const __nv_bfloat16 *__restrict__ o, __nv_bfloat16 *__restrict__ do_hm,
                                                       float *__restrict__ dgate, int B, int T, int H, bool gated) {
    const long long w = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= static_cast<long long>(B) * T * H) return;
    const int h = static_cast<int>(w % H);
    const long long bt = w / H;
    const int b = static_cast<int>(bt / T), t = static_cast<int>(bt % T);
    const size_t off = static_cast<size_t>(w) * kD + lane * 4;
    const uint2 dv = __ldg(reinterpret_cast<const uint2 *>(dout + off));
    const uint2 ov = __ldg(reinterpret_cast<const uint2 *>(o + off));
    const uint2 gv = g ? __ldg(reinterpret_cast<const uint2 *>(g + off)) : make_uint2(0u, 0u);
    const uint32_t dw[2] = {dv.x, dv.y}, ow[2] = {ov.x, ov.y}, gw[2] = {gv.x, gv.y};
    float dov[4], dg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t sh = (i & 1) ? 0u : 16u;
        const float d = __uint_as_float((dw[i >> 1] << sh) & 0xFFFF0000u);
        const float ov_ = __uint_as_float((ow[i >> 1] << sh) & 0xFFFF0000u);
        const float sg = g ? 1.f / (1.f + expf(-__uint_as_float((gw[i >> 1] << sh) & 0xFFFF0000u))) : 1.f;
        dov[i] = d * sg;
        dg[i] = gated ? d * ov_ * (1.f - sg) : d * ov_ * sg * (1.f - sg);
    }
    const size_t hm = ((static_cast<size_t>(b) * H + h) * T + t) * kD + lane * 4;
    *reinterpret_cast<uint2 *>(do_hm + hm) = make_uint2(pack_bf16x2(dov[0], dov[1]), pack_bf16x2(dov[2], dov[3]));
    if (dgate) *reinterpret_cast<float4 *>(dgate + off) = make_float4(dg[0], dg[1], dg[2], dg[3]);

}

// out = part[0] + part[1] + ... + part[parts - 1], in that order (the gradients are the same bits on every call).
__global__ void __launch_bounds__(256) split_sum_kernel(const float4 *__restrict__ part, int parts, long long n4,
                                                        float4 *__restrict__ out) {
    const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
    if (i >= n4) return;
    float4 acc = __ldg(part + i);
    for (int k = 1; k < parts; ++k) {
        const float4 v = __ldg(part + static_cast<long long>(k) * n4 + i);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    out[i] = acc;
}

CUresult enc(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
             const cuuint32_t *box) {
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides_bytes, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

size_t al(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct BwdLayout {
    size_t o, pre, lse, psum, psum_part, dnum_part, do_hm, qa, qlo, dl, ol, dqa, P, dS, part, end;
};
// dc and the weight gradients cut each tile's K steps into up to this many parts (fp32 partial sums in the
// workspace, added in a fixed order afterwards), so that their few long tiles spread over the SMs
constexpr int kMaxSplit = 8;
BwdLayout bwd_layout(long long B, long long T, long long H) {
    const long long Tp = (T + 127) / 128 * 128;
    const size_t rows = static_cast<size_t>(B) * H * T;
    BwdLayout L;
    L.o = 0;
    L.pre = L.o + al(static_cast<size_t>(B) * T * H * kD * 2);
    L.lse = L.pre + al(prefill_bf16_r512_workspace_bytes(B, T));
    L.psum = L.lse + al(rows * 4);
    L.psum_part = L.psum + al(rows * 4);
    L.dnum_part = L.psum_part + al(rows * 4 * static_cast<size_t>(Tp / 128));
    L.do_hm = L.dnum_part + al(rows * 4 * (kR / kBN));
    L.qa = L.do_hm + al(rows * kD * 2);
    L.qlo = L.qa + al(rows * kR * 2);
    L.dl = L.qlo + al(rows * kR * 2);
    L.ol = L.dl + al(rows * kR * 2);
    L.dqa = L.ol + al(rows * kR * 2);
    L.P = L.dqa + al(rows * kR * 2);
    L.dS = L.P + al(rows * Tp * 2);
    L.part = L.dS + al(rows * Tp * 2);
    L.end = L.part + al(static_cast<size_t>(kMaxSplit) * static_cast<size_t>(B * T > H * kD ? B * T : H * kD) * kR * 4);
    return L;
}

}  // namespace

bool backward_bf16_r512_supports(int r, int d_q, int d_v) { return r == kR && d_q == kD && d_v == kD; }

size_t backward_bf16_r512_workspace_bytes(long long B, long long T, long long H) { return bwd_layout(B, T, H).end; }

cudaError_t launch_backward_bf16_r512(const BackwardR512Args &a, cudaStream_t s) {
    if (!backward_bf16_r512_supports(a.r, a.d_q, a.d_v)) return cudaErrorInvalidValue;
    const int B = a.B, T = a.T, H = a.H;
    const int Tp = (T + 127) / 128 * 128;
    const BwdLayout L = bwd_layout(B, T, H);
    if (a.workspace_bytes < L.end) return cudaErrorInvalidValue;
    char *ws = static_cast<char *>(a.workspace);
    auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16 *>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
    const size_t rowsz = static_cast<size_t>(B) * H;   // head-major batch items

    // 1. the forward without the gate: o, and each row's log-sum-exp; or both given by the caller's forward
    const bool saved = a.lse != nullptr && a.out_fwd != nullptr;
    const float *lse = saved ? a.lse : f32(L.lse);
    cudaError_t e = cudaSuccess;
    if (!saved) {
        PrefillArgs pa{a.q, a.c, a.w_uk, a.w_uv, nullptr, bf(L.o), a.scale, B, T, H, kD, kD, kR, a.dev_err, a.num_sms,
                       ws + L.pre, L.lse - L.pre};
        pa.lse = f32(L.lse);
        if ((e = launch_prefill_bf16_r512(pa, s)) != cudaSuccess) return e;
    }
    // 2. the gate's backward, do and delta
    {
        const long long warps = static_cast<long long>(B) * T * H;
        note_launch();
        bwd_gate_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(a.dout), static_cast<const __nv_bfloat16 *>(a.gate),
            saved ? static_cast<const __nv_bfloat16 *>(a.out_fwd) : bf(L.o), bf(L.do_hm), static_cast<float *>(a.dgate),
            B, T, H, saved);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // tensor maps (dims innermost first, strides in bytes)
    const cuuint64_t uT = T, uH = H, uB = B, uZ = rowsz, uTp = Tp;
    CUtensorMap mq_k, mq_mn, mwuk_mn, mwuk_k, mwuv_mn, mdo_k, mdo_mn, mqa_k, mqlo_k, mdl_k, mol_mn, mdqa_k, mdqa_mn,
        mc_k, mP_k, mdS_k, mc_sl, mP_sl, mdS_sl, mdl_sl, mqa_sl;
    bool okm = true;
    auto E = [&](CUtensorMap *m, const void *ptr, int rank, std::initializer_list<cuuint64_t> d,
                 std::initializer_list<cuuint64_t> st, std::initializer_list<cuuint32_t> bx) {
        cuuint64_t dd[5], ss[4];
        cuuint32_t bb[5];
        int i = 0;
        for (auto v : d) dd[i++] = v;
        i = 0;
        for (auto v : st) ss[i++] = v;
        i = 0;
        for (auto v : bx) bb[i++] = v;
        okm = okm && enc(m, ptr, rank, dd, ss, bb) == CUDA_SUCCESS;
    };
    const cuuint64_t hd2 = static_cast<cuuint64_t>(H) * kD * 2;
    E(&mq_k, a.q, 4, {kD, uH, uT, uB}, {kD * 2, hd2, hd2 * T}, {64, 1, 128, 1});
    E(&mq_mn, a.q, 4, {kD, uH, uT, uB}, {kD * 2, hd2, hd2 * T}, {64, 1, 64, 1});
    E(&mwuk_mn, a.w_uk, 3, {kR, kD, uH}, {kR * 2, kR * kD * 2}, {64, 64, 1});
    E(&mwuk_k, a.w_uk, 3, {kR, kD, uH}, {kR * 2, kR * kD * 2}, {64, 128, 1});
    E(&mwuv_mn, a.w_uv, 3, {kR, kD, uH}, {kR * 2, kR * kD * 2}, {64, 64, 1});
    E(&mdo_k, bf(L.do_hm), 3, {kD, uT, uZ}, {kD * 2, kD * 2 * uT}, {64, 128, 1});
    E(&mdo_mn, bf(L.do_hm), 3, {kD, uT, uZ}, {kD * 2, kD * 2 * uT}, {64, 64, 1});
    auto EK = [&](CUtensorMap *mk, size_t off) {   // a [z, T, r] matrix, K-major boxes [128 rows x 64]
        E(mk, bf(off), 3, {kR, uT, uZ}, {kR * 2, kR * 2 * uT}, {64, 128, 1});
    };
    EK(&mqa_k, L.qa);
    EK(&mqlo_k, L.qlo);
    EK(&mdl_k, L.dl);
    EK(&mdqa_k, L.dqa);
    E(&mdqa_mn, bf(L.dqa), 3, {kR, uT, uZ}, {kR * 2, kR * 2 * uT}, {64, 64, 1});   // dW_UK's B: MN-major
    E(&mol_mn, bf(L.ol), 3, {kR, uT, uZ}, {kR * 2, kR * 2 * uT}, {64, 64, 1});
    E(&mc_k, a.c, 3, {kR, uT, uB}, {kR * 2, kR * 2 * uT}, {64, 128, 1});
    // slab maps of MN-major operands: [64 columns] x [rows] x [column slab of 64] x [batch], so one box
    // {64, 64, 2, 1} brings two 64-column slabs, 8 KB apart in shared memory (the MN-major operand layout),
    // in one TMA instruction instead of two
    auto ESL = [&](CUtensorMap *m, const void *ptr, cuuint64_t cols, cuuint64_t nz) {
        E(m, ptr, 4, {64, uT, cols / 64, nz}, {cols * 2, 128, cols * 2 * uT}, {64, 64, 2, 1});
    };
    ESL(&mc_sl, a.c, kR, uB);
    ESL(&mdl_sl, bf(L.dl), kR, uZ);
    ESL(&mqa_sl, bf(L.qa), kR, uZ);
    E(&mP_k, bf(L.P), 3, {uTp, uT, uZ}, {uTp * 2, uTp * 2 * uT}, {64, 128, 1});
    E(&mdS_k, bf(L.dS), 3, {uTp, uT, uZ}, {uTp * 2, uTp * 2 * uT}, {64, 128, 1});
    ESL(&mP_sl, bf(L.P), uTp, uZ);
    ESL(&mdS_sl, bf(L.dS), uTp, uZ);
    if (!okm) return cudaErrorInvalidValue;
    if ((e = cudaFuncSetAttribute(bwd_gemm_kernel<128, 1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape<128>::kSmemW))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_gemm_kernel<256, 1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape<256>::kSmemW))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_gemm_kernel<256, 2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape<256, 2>::kSmemW))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_gemm_kernel<256, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape<256, 1, true>::kSmemW))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_gemm2_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape2<1>::kSmem))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_gemm2_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(Shape2<2>::kSmem))) != cudaSuccess)
        return e;
    const int sms = a.num_sms > 1 ? a.num_sms : 2;
    auto split_for = [&](long long base_items, int slots) {   // parts per tile: about four items per slot
        const long long k = (4LL * slots + base_items - 1) / base_items;
        return static_cast<int>(k < 1 ? 1 : (k > kMaxSplit ? kMaxSplit : k));
    };
    // kind 0: 128 x 128 tiles, two CTAs per SM; 1: 128 x 256 tiles, one CTA per SM; 2: 256 x 256 tiles on CTA
    // pairs (one CTA per SM)
    auto gemm = [&](int pr, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ta2,
                    const CUtensorMap &tb2, int M, int N, int Z, void *out, int kind) {
        if (pr == kP && kind == 0) return cudaErrorInvalidValue;   // P's staging (hi and lo together): 128 x 256 or pairs
        const int tm = kind == 2 ? 256 : 128, tn = kind == 0 ? 128 : 256;
        const int slots = kind == 0 ? 2 * sms : (kind == 1 ? sms : sms / 2);   // CTAs, or pairs, resident at once
        GemmP gp{};
        gp.problem = pr;
        gp.B = B;
        gp.T = T;
        gp.H = H;
        gp.Tp = Tp;
        gp.M = M;
        gp.N = N;
        gp.scale_log2 = a.scale * kLog2e;
        gp.scale = a.scale;
        gp.lse = lse;
        gp.psum = f32(L.psum);
        gp.psum_part = f32(L.psum_part);
        gp.dnum_part = f32(L.dnum_part);
        gp.rows = static_cast<long long>(rowsz) * T;
        gp.out2 = bf(L.qlo);
        gp.p_in = bf(L.P);
        gp.dl_in = bf(L.dl);
        gp.out = out;
        gp.err = a.dev_err;
        gp.tile_m = tm;
        gp.tile_n = tn;
        gp.nmt = (M + tm - 1) / tm;
        gp.nnt = (N + tn - 1) / tn;
        gp.nz = Z;
        gp.ksplit = 1;
        gp.part = f32(L.part);
        gp.part_n = static_cast<long long>(Z) * M * N;
        long long items;
        if (pr == kP || pr == kDS) {
            const long long n = gp.nmt, h2 = n / 2;
            const long long tri = kind == 1 ? (n % 2 == 0 ? h2 * (h2 + 1) : (h2 + 1) * (h2 + 1))
                                            : n * (n + 1) / 2 + (kind == 0 ? h2 : 0);
            items = static_cast<long long>(Z) * tri;
        } else {
            if (pr == kDc || pr == kDWuk || pr == kDWuv)
                gp.ksplit = split_for(static_cast<long long>(gp.nmt) * gp.nnt * Z, slots);
            items = static_cast<long long>(gp.nmt) * gp.nnt * Z * gp.ksplit;
        }
        if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
        gp.items = static_cast<int>(items);
        const unsigned grid = static_cast<unsigned>(items < slots ? items : slots);
        note_launch();
        if (kind == 2 && pr == kP) bwd_gemm2_kernel<2><<<2 * grid, kThreads2, Shape2<2>::kSmem, s>>>(ta, tb, ta2, tb2, gp);
        else if (kind == 2) bwd_gemm2_kernel<1><<<2 * grid, kThreads2, Shape2<1>::kSmem, s>>>(ta, tb, ta2, tb2, gp);
        else if (pr == kP)
            bwd_gemm_kernel<256, 2, false><<<grid, Shape<256, 2>::kThreadsW, Shape<256, 2>::kSmemW, s>>>(ta, tb, ta2, tb2, gp);
        else if (pr == kDS && kind == 1)   // ta2: P [z, T, Tp] in [128 x 64] boxes
            bwd_gemm_kernel<256, 1, true><<<grid, Shape<256, 1, true>::kThreadsW, Shape<256, 1, true>::kSmemW, s>>>(
                ta, tb, ta2, tb2, gp);
        else if (kind == 1)
            bwd_gemm_kernel<256, 1, false><<<grid, Shape<256>::kThreadsW, Shape<256>::kSmemW, s>>>(ta, tb, ta2, tb2, gp);
        else bwd_gemm_kernel<128, 1, false><<<grid, Shape<128>::kThreadsW, Shape<128>::kSmemW, s>>>(ta, tb, ta2, tb2, gp);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess || gp.ksplit == 1) return err;
        const long long n4 = gp.part_n / 4;   // N = r: a multiple of 4
        note_launch();
        split_sum_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, s>>>(
            reinterpret_cast<const float4 *>(gp.part), gp.ksplit, n4, static_cast<float4 *>(out));
        return cudaGetLastError();
    };
    const int Z = static_cast<int>(rowsz);
    // 3. q_abs and do_lat; 4. P (and its row sums), o_lat (and do_lat . o_lat), then dS (reads P and both sums);
    // 5. dq_abs; 6. dc and dq; 7. the weight gradients
    if ((e = gemm(kQAbs, mq_k, mwuk_mn, mq_k, mwuk_mn, T, kR, Z, bf(L.qa), 1)) != cudaSuccess) return e;
    if ((e = gemm(kDoLat, mdo_k, mwuv_mn, mdo_k, mwuv_mn, T, kR, Z, bf(L.dl), 1)) != cudaSuccess) return e;
    if ((e = gemm(kP, mqa_k, mc_k, mqlo_k, mc_k, T, T, Z, bf(L.P), 2)) != cudaSuccess) return e;
    if ((e = gemm(kOLat, mP_k, mc_sl, mP_k, mc_sl, T, kR, Z, bf(L.ol), 2)) != cudaSuccess) return e;
    if ((e = gemm(kDS, mdl_k, mc_k, mP_k, mc_k, T, T, Z, bf(L.dS), 1)) != cudaSuccess) return e;
    if ((e = gemm(kDqAbs, mdS_k, mc_sl, mdS_k, mc_sl, T, kR, Z, bf(L.dqa), 2)) != cudaSuccess) return e;
    if ((e = gemm(kDc, mP_sl, mdl_sl, mdS_sl, mqa_sl, T, kR, B, a.dc, 2)) != cudaSuccess) return e;
    if ((e = gemm(kDq, mdqa_k, mwuk_k, mdqa_k, mwuk_k, T, kD, Z, a.dq, 0)) != cudaSuccess) return e;
    if ((e = gemm(kDWuk, mq_mn, mdqa_mn, mq_mn, mdqa_mn, kD, kR, H, a.dw_uk, 1)) != cudaSuccess) return e;
    return gemm(kDWuv, mdo_mn, mol_mn, mdo_mn, mol_mn, kD, kR, H, a.dw_uv, 1);
}

}  // namespace mla
