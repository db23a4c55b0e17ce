/*
 * mla.h - C ABI of the GB300 (sm_103a) absorbed, NoPE, causal Gated MLA forward.
 *
 * The method is the one on the course-notes page "Gated MLA（矩阵吸收版）"
 * (Gated MLA with matrix absorption): keys and values are never decompressed;
 * each head's query is absorbed into the latent space, q_abs = q . W_UK,
 * scored directly against the shared rank-r latent c, softmax-weighted sums
 * are taken over c itself, and only then are they up-projected by W_UV^T and
 * gated by sigmoid(W_g x) (section "完整计算流（四步）", steps 2-4; shapes from
 * the symbol-table page "符号表", table "MLA 变量").
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or retains them past the call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Nothing is launched when a status other than MLA_OK is returned.
 *  - Layouts are dense row-major (C order) with the shapes given; all float
 *    tensors of one call share one dtype; accumulation is fp32; `out` has the
 *    input dtype.
 *  - Arguments are validated on the host before any launch.  Errors raised on
 *    the device (a bounded wait that gave up) are recorded in a per-device
 *    error word read by mla_get_device_error().
 *  - There is no CPU fallback and no silent slow path: a shape outside the
 *    supported set returns MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define MLA_API
#else
#define MLA_API __attribute__((visibility("default")))
#endif

/* Element types. */
typedef enum {
    MLA_DTYPE_BF16 = 0, /* bfloat16 inputs and output, fp32 accumulation */
    MLA_DTYPE_F32 = 1   /* fp32 inputs and output, fp32 FMA (no TF32)    */
} mla_dtype_t;

/* Status codes (0 = success, negative = error). */
typedef enum {
    MLA_OK = 0,
    MLA_ERR_NULL = -1,           /* a required pointer is NULL                       */
    MLA_ERR_SHAPE = -2,          /* a size is negative, zero where it may not be, or overflows */
    MLA_ERR_DTYPE = -3,          /* unknown dtype                                   */
    MLA_ERR_ALIGN = -4,          /* a pointer or stride is not 16-byte aligned      */
    MLA_ERR_WORKSPACE = -5,      /* workspace missing or smaller than required      */
    MLA_ERR_UNSUPPORTED = -6,    /* valid shape that no kernel of this build serves  */
    MLA_ERR_CUDA = -7,           /* a CUDA runtime/driver call failed               */
    MLA_ERR_DEVICE_TIMEOUT = -8, /* a bounded device-side wait gave up              */
    MLA_ERR_DEVICE_BOUNDS = -9   /* a device-side bounds check rejected an index    */
} mla_status_t;

/*
 * mla_absorbed_attn_fwd - causal prefill of the absorbed Gated MLA.
 * mla_absorbed_attn_fwd_workspace_size - bytes of workspace it needs for these
 * sizes (0 when none; also 0 for invalid or unsupported sizes).
 *
 * Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）":
 *   step 2  q_abs[b,t,h,:] = q[b,t,h,:] . W_UK[h]                  [B,T,H,r]
 *           score[b,h,t,u] = scale * q_abs[b,t,h,:] . c[b,u,:]     (u <= t)
 *           attn = softmax over u of the causally masked score
 *   step 3  o_lat[b,h,t,:] = sum_u attn[b,h,t,u] * c[b,u,:]        [B,H,T,r]
 *           o[b,h,t,v]     = o_lat[b,h,t,:] . W_UV[h,v,:]
 *   step 4  out[b,t,h*d_v+v] = sigmoid(gate[b,t,h*d_v+v]) * o[b,h,t,v]
 * The output projection W_o of step 4 is not part of this call.
 *
 * Arguments (shapes in elements, dense row-major):
 *   q     [B,T,H,d_q]   queries (the step-1 low-rank query path's output)
 *   c     [B,T,r]       shared latent, used as both key and value
 *   w_uk  [H,d_q,r]     key up-projection W_UK (first block of kv_up.weight)
 *   w_uv  [H,d_v,r]     value up-projection W_UV (second block of kv_up.weight)
 *   gate  [B,T,H*d_v]   pre-sigmoid gate logits W_g x, or NULL for no gate
 *   scale               softmax scale applied to the score (1.0 = the page's listing)
 *   out   [B,T,H*d_v]   result, flat index h*d_v + v; must not alias an input
 *   workspace           device buffer of >= mla_absorbed_attn_fwd_workspace_size(...)
 *                       bytes, 16-byte aligned, not used by any other call in flight;
 *                       may be NULL when that size is 0.  The r = 512 kernel keeps an
 *                       f16 copy of c there (see precision below).
 * Masking: token t attends to tokens 0..t of its own sequence.
 * Precision (BF16): the score operand q_abs * scale is not rounded to bf16.  At
 * r = 512 the score product runs on f16 copies of q_abs and c, each scaled by a
 * power of two (per query row, per sequence) into the f16 range and scaled back
 * exactly in the softmax; at r <= 64 q_abs is split into two bf16 parts.  The
 * softmax weights, o_lat / l and the output are rounded to bf16.
 * Supported: F32 with r, d_q, d_v <= 64 and T <= 1,048,560; BF16 with (r, d_q, d_v) = (512, 128, 128),
 * or r in {32, 64} with d_q, d_v in {16, 32, 48, 64}.  B*T == 0 is a no-op
 * returning MLA_OK.
 * Alignment: every pointer 16-byte aligned.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API size_t mla_absorbed_attn_fwd_workspace_size(int B, int T, int H, int d_q, int d_v, int r, int dtype);
MLA_API int mla_absorbed_attn_fwd(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                  const void *gate, float scale, void *out,
                                  int B, int T, int H, int d_q, int d_v, int r,
                                  int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_absorbed_attn_fwd_lse - mla_absorbed_attn_fwd that also writes each row's
 * log-sum-exp of the scaled, causally masked scores, for mla_absorbed_attn_bwd_lse:
 *   lse[b,h,t] = ln sum_{u<=t} exp(scale * q_abs[b,t,h,:] . c[b,u,:])   [B,H,T] fp32
 * so that attn[b,h,t,u] = exp(scale * q_abs . c_u - lse[b,h,t]) (page "Gated MLA
 * （矩阵吸收版）", section "完整计算流（四步）", step 2: the softmax's normaliser).
 * Arguments, workspace (mla_absorbed_attn_fwd_workspace_size) and precision as
 * for mla_absorbed_attn_fwd; lse is caller-owned device memory, 16-byte aligned,
 * overwritten.  Supported: BF16 with (r, d_q, d_v) = (512, 128, 128); others
 * return MLA_ERR_UNSUPPORTED.  lse NULL returns MLA_ERR_NULL.
 */
MLA_API int mla_absorbed_attn_fwd_lse(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                      const void *gate, float scale, void *out, float *lse, int B, int T, int H,
                                      int d_q, int d_v, int r, int dtype, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * mla_absorbed_attn_bwd - gradients of the attention (steps 2-4 of section
 * "完整计算流（四步）" of the page "Gated MLA（矩阵吸收版）", which gives the forward
 * only; this takes the chain rule back through it).  For
 * L = sum(dout * out) with out = mla_absorbed_attn_fwd(q, c, w_uk, w_uv, gate,
 * scale) it writes (fp32 whatever the input dtype, caller-owned device memory,
 * overwritten):
 *   dq     [B,T,H,d_q]   dL/dq
 *   dc     [B,T,r]       dL/dc (summed over heads and over the queries that see each key)
 *   dw_uk  [H,d_q,r]     dL/dW_UK (summed over batch and tokens)
 *   dw_uv  [H,d_v,r]     dL/dW_UV
 *   dgate  [B,T,H*d_v]   dL/dgate (the pre-sigmoid logits); NULL exactly when gate is NULL
 * Inputs as for mla_absorbed_attn_fwd, plus dout [B,T,H*d_v], all of dtype
 * `dtype` (MLA_DTYPE_F32 or MLA_DTYPE_BF16; bf16 values are widened to fp32).
 * workspace: >= mla_absorbed_attn_bwd_workspace_size(...) bytes, 16-byte
 * aligned (per-row q_abs, do_lat and softmax statistics between the kernels).
 * Supported:
 *  - r, d_q, d_v <= 64 (the toy sizes), F32 or BF16, T <= 4,194,240: fp32
 *    arithmetic throughout (SIMT).  dc, dw_uk and dw_uv are sums over thread
 *    blocks formed with atomics, so their last bits may differ between calls.
 *  - BF16 with (r, d_q, d_v) = (512, 128, 128): tensor cores.  The call runs the
 *    forward once more (its output before the gate and each row's softmax
 *    statistics), then every product of the chain rule as a batched bf16 GEMM
 *    with fp32 accumulation over per-head matrices kept in the workspace: the
 *    attention matrix and its gradient ([T, T] per head, bf16, causal tiles
 *    only), q_abs, do_lat, o_lat and dq_abs ([T, r] per head, bf16).  The
 *    workspace is therefore O(B H T^2): about 2 B H T^2 + 9 B H T r bytes.
 *    Deterministic (no atomics).
 * Other shapes return MLA_ERR_UNSUPPORTED.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API size_t mla_absorbed_attn_bwd_workspace_size(int B, int T, int H, int d_q, int d_v, int r, int dtype);
MLA_API int mla_absorbed_attn_bwd(const void *q, const void *c, const void *w_uk, const void *w_uv, const void *gate,
                                  float scale, const void *dout, void *dq, void *dc, void *dw_uk, void *dw_uv,
                                  void *dgate, int B, int T, int H, int d_q, int d_v, int r, int dtype,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_absorbed_attn_bwd_lse - mla_absorbed_attn_bwd given what a forward call
 * mla_absorbed_attn_fwd_lse(q, c, w_uk, w_uv, gate, scale) on the same inputs
 * returned: its output `out` [B,T,H*d_v] (after the gate) and `lse` [B,H,T].  The
 * forward is not run again: the attention matrix is rebuilt from lse, and with a
 * gate dgate = dout * out * (1 - sigmoid(gate)).  Outputs, workspace
 * (mla_absorbed_attn_bwd_workspace_size) and determinism as for mla_absorbed_attn_bwd.
 * Supported: BF16 with (r, d_q, d_v) = (512, 128, 128); others return
 * MLA_ERR_UNSUPPORTED.  out or lse NULL returns MLA_ERR_NULL; both 16-byte aligned.
 */
MLA_API int mla_absorbed_attn_bwd_lse(const void *q, const void *c, const void *w_uk, const void *w_uv,
                                      const void *gate, float scale, const void *dout, const void *out,
                                      const float *lse, void *dq, void *dc, void *dw_uk, void *dw_uv, void *dgate,
                                      int B, int T, int H, int d_q, int d_v, int r, int dtype, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * mla_latent_decode_workspace_size - bytes of device workspace mla_latent_decode
 * needs for these sizes on the CURRENT device (it depends on the SM count).
 * Returns 0 for sizes that are invalid or unsupported.
 */
MLA_API size_t mla_latent_decode_workspace_size(int B, int H, int r, int max_len);

/*
 * mla_latent_decode - one decode step over the cached latent.
 *
 * Only the latent c is cached (page "Gated MLA（矩阵吸收版）", sections
 * "标准 MHA 的 KV cache 问题" and "形状与参数对比", KV-cache table: r values
 * per token instead of 2*H*d).  Each sequence b has one new query, already
 * absorbed (q_abs = q . W_UK, step 2), that attends, without a mask, to its
 * cache rows 0 .. lens[b]-1 (the caller has appended the new token's own
 * latent first).  Steps 2-4 then follow as in the prefill.
 *
 * Arguments:
 *   q_abs     [B,H,r]         absorbed queries
 *   c_cache   element (b,u,j) at b*max_len*ld_cache + u*ld_cache + j
 *   ld_cache  row stride of the cache in elements (>= r, multiple of 8)
 *   lens      int32 [B] on the device, 0 <= lens[b] <= max_len;
 *             lens[b] == 0 writes a zero output row.  Rows at or beyond
 *             lens[b] are never used, whatever they hold.
 *   max_len   rows allocated per sequence
 *   w_uv      [H,d_v,r]       value up-projection
 *   gate      [B,H*d_v]       pre-sigmoid gate logits, or NULL
 *   scale     softmax scale
 *   out       [B,H*d_v]
 *   workspace device buffer of >= mla_latent_decode_workspace_size(...) bytes,
 *             16-byte aligned, not used by any other call in flight
 * Supported: BF16 with r = 512, d_v = 128, 1 <= H <= 96.
 * A lens[b] outside [0, max_len] found on the device is clamped to that
 * range and reported as MLA_ERR_DEVICE_BOUNDS by mla_get_device_error().
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API int mla_latent_decode(const void *q_abs, const void *c_cache, long long ld_cache, const int *lens,
                              int max_len, const void *w_uv, const void *gate, float scale, void *out,
                              int B, int H, int d_v, int r, int dtype,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_latent_decode_fp8 - mla_latent_decode over a latent cache stored in
 * 8-bit floating point (e4m3: 1 sign, 4 exponent, 3 mantissa bits; largest
 * finite value 448), half the bytes per cached token of the bf16 cache.
 *
 * This carries the cache-size argument of the page "Gated MLA（矩阵吸收版）"
 * (sections "标准 MHA 的 KV cache 问题" and "形状与参数对比": only r values per
 * token are cached) one step further; the page itself caches bf16/fp32 c.
 * The cache holds c / cache_scale: cache row u of sequence b dequantises to
 * cache_scale * e4m3(c8_cache[b, u, :]), and the call computes exactly
 * mla_latent_decode over those dequantised rows.
 *
 * Arguments as for mla_latent_decode, except:
 *   c8_cache     e4m3 bytes; element (b,u,j) at byte b*max_len*ld_cache + u*ld_cache + j
 *   ld_cache     row stride in bytes (>= r, multiple of 16)
 *   cache_scale  positive, finite
 *   q_abs, w_uv, gate, out  bf16 as in mla_latent_decode (there is no dtype argument)
 *   workspace    >= mla_latent_decode_fp8_workspace_size(...) bytes, 16-byte
 *                aligned, not used by any other call in flight
 * Precision: both products run on the 8-bit tensor cores.  The query q_abs is
 * split into two e4m3 parts (after a power-of-two scale per head) and so are
 * the softmax weights, which keeps about 8 significant bits of each, as a
 * bf16 operand would; the cache values themselves are exact.
 * Supported: r = 512, d_v = 128, 1 <= H <= 96.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API size_t mla_latent_decode_fp8_workspace_size(int B, int H, int r, int max_len);
MLA_API int mla_latent_decode_fp8(const void *q_abs, const void *c8_cache, long long ld_cache, const int *lens,
                                  int max_len, float cache_scale, const void *w_uv, const void *gate, float scale,
                                  void *out, int B, int H, int d_v, int r, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * mla_quantize_latent_fp8 - fill an e4m3 latent cache from bf16 latent rows:
 * c8[i, j] = e4m3(c[i, j] * (1 / cache_scale)), the product formed in fp32
 * (1 / cache_scale rounded to fp32 first), rounded to the nearest e4m3 value
 * (ties to even) and clamped to +-448.  Same section as mla_latent_decode_fp8.
 *   c      bf16 [rows, r] with row stride ld_c elements (multiple of 8)
 *   c8     bytes [rows, r] with row stride ld_c8 bytes (multiple of 16)
 * r a multiple of 8; both pointers 16-byte aligned; rows == 0 is a no-op.
 * Latent rows from RMSNorm with unit gain have |c| <= sqrt(r) (22.6 at
 * r = 512), so cache_scale = 1/16 maps them inside e4m3's range.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API int mla_quantize_latent_fp8(const void *c, long long ld_c, void *c8, long long ld_c8, long long rows, int r,
                                    float cache_scale, void *stream);

/*
 * mla_latent_decode_noalloc - mla_latent_decode for callers that cannot
 * allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc: a host framework that owns all device memory
 * and hands the library only its inputs and outputs, or a service that must
 * not allocate (or pay cudaMalloc's synchronisation) once it is running.  It
 * computes exactly what mla_latent_decode computes, with the same arguments
 * except that there is no workspace: the partial results live in a scratch
 * array that the library reserves in device memory when it is loaded, 48 MiB
 * on every device that loads the library, held until the process exits.
 *
 * - Sizes whose scratch need (mla_latent_decode_workspace_size) exceeds
 *   48 MiB return MLA_ERR_WORKSPACE and launch nothing.  The K3 decode
 *   workload (B = 64, H = 96, r = 512 on a 152-SM GB300) needs 13.9 MB.
 * - The call allocates and frees nothing, on the host or the device.
 * - The first call on a device looks up the scratch array's device address
 *   on that device (cudaGetSymbolAddress); make that first call before any
 *   stream capture.  If that lookup fails (for example inside a capture, or
 *   when the library's device code cannot be loaded on the device) the call
 *   returns MLA_ERR_CUDA, clears the runtime's pending error and launches
 *   nothing; a later call retries the lookup.
 * - Every call uses the same scratch array: calls whose kernels can overlap
 *   on the GPU (different streams, no ordering between them) race on it and
 *   give wrong results.  Calls on one stream, or otherwise ordered, are safe.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API int mla_latent_decode_noalloc(const void *q_abs, const void *c_cache, long long ld_cache, const int *lens,
                                      int max_len, const void *w_uv, const void *gate, float scale, void *out,
                                      int B, int H, int d_v, int r, int dtype, void *stream);

/*
 * mla_gated_layer_workspace_size - bytes of device workspace mla_gated_layer_fwd
 * needs for these sizes (0 if the shape or dtype is not supported).
 */
MLA_API size_t mla_gated_layer_workspace_size(int B, int T, int D, int H, int d_q, int d_v, int r, int r_q,
                                              int dtype);

/*
 * mla_gated_layer_fwd - the whole Gated-MLA layer (page "Gated MLA（矩阵吸收版）",
 * section "完整计算流（四步）", steps 1-4, plus the output projection of the
 * listing in section "代码对照"):
 *
 *   c   = RMSNorm(x . w_kv_down^T)                         [B,T,r]
 *   q   = RMSNorm(x . w_q_down^T) . w_q_up^T                 [B,T,H,d_q]
 *   g   = x . w_gate^T                                       [B,T,H*d_v]
 *   o   = mla_absorbed_attn_fwd(q, c, W_UK, W_UV, g, scale)  [B,T,H*d_v]
 *   y   = o . w_o^T                                          [B,T,D]
 *
 * RMSNorm: z / sqrt(mean(z^2) + 1e-6), unit gain.  No biases.  Weights are
 * nn.Linear weights [out_features, in_features], row-major:
 *   w_q_down [r_q, D]   w_q_up [H*d_q, r_q]   w_kv_down [r, D]
 *   w_kv_up  [H*(d_q+d_v), r]: all heads' W_UK rows first (W_UK = w_kv_up as
 *            [H,d_q,r]), then all heads' W_UV rows ([H,d_v,r])
 *   w_gate   [H*d_v, D]   w_o [D, H*d_v]
 * x [B,T,D] and y [B,T,D], row-major.  All tensors share `dtype`.
 *
 * Supported: MLA_DTYPE_F32 with r, d_q, d_v <= 64 and T <= 1,048,560 (SIMT fp32, no TF32);
 * MLA_DTYPE_BF16 with r = 512, d_q = d_v = 128, H even, D and r_q multiples of
 * 256 (tensor-core GEMMs, fp32 accumulation, bf16 intermediate results).
 *
 *   workspace  device buffer of >= mla_gated_layer_workspace_size(...) bytes,
 *              16-byte aligned, caller-owned.  On return (in stream order) it
 *              holds, each part starting on a 256-byte boundary and in the
 *              input dtype: q [B*T, H*d_q], c [B*T, r], g [B*T, H*d_v] and o
 *              [B*T, H*d_v], followed by internal scratch.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API int mla_gated_layer_fwd(const void *x, const void *w_q_down, const void *w_q_up, const void *w_kv_down,
                                const void *w_kv_up, const void *w_gate, const void *w_o, float scale, void *y,
                                int B, int T, int D, int H, int d_q, int d_v, int r, int r_q, int dtype,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_gated_layer_decode_workspace_size - bytes of device workspace
 * mla_gated_layer_decode needs on the CURRENT device (0 if unsupported).
 */
MLA_API size_t mla_gated_layer_decode_workspace_size(int B, int D, int H, int d_q, int d_v, int r, int r_q,
                                                     int max_len, int dtype);

/*
 * mla_gated_layer_decode - one decode step of the whole layer with the
 * latent-cache append (page "Gated MLA（矩阵吸收版）": only the latent c is
 * cached, section "低秩压缩"; steps 1-4 of section "完整计算流（四步）"; W_o).
 * For each sequence b, the new token x[b] (position lens[b]):
 *
 *   c_cache[b, lens[b], :] = RMSNorm(x[b] . w_kv_down^T)          (the append)
 *   q_abs = (RMSNorm(x[b] . w_q_down^T) . w_q_up^T) . W_UK          per head
 *   o     = mla_latent_decode(q_abs, c_cache, lens[b] + 1 rows, W_UV, g = x[b] . w_gate^T, scale)
 *   y[b]  = o . w_o^T
 *
 *   x [B, D], y [B, D]; weights as in mla_gated_layer_fwd.
 *   c_cache    [B, max_len, r] with row stride ld_cache (elements, multiple of
 *              8, >= r); row lens[b] of each sequence is written.
 *   lens       int32 [B] on the device: the new token's position, in
 *              [0, max_len).  Read only; the caller advances it after the
 *              step.  A position outside the range is reported as
 *              MLA_ERR_DEVICE_BOUNDS (mla_get_device_error) and that row is
 *              not written.
 *   workspace  >= mla_gated_layer_decode_workspace_size(...) bytes, 16-byte
 *              aligned.
 * Supported: MLA_DTYPE_BF16 with r = 512, d_q = d_v = 128, 1 <= H <= 96 and
 * even, D and r_q multiples of 256.
 * Returns MLA_OK or a negative mla_status_t; nothing is launched on error.
 */
MLA_API int mla_gated_layer_decode(const void *x, const void *w_q_down, const void *w_q_up, const void *w_kv_down,
                                   const void *w_kv_up, const void *w_gate, const void *w_o, float scale, void *y,
                                   void *c_cache, long long ld_cache, const int *lens, int max_len, int B, int D,
                                   int H, int d_q, int d_v, int r, int r_q, int dtype, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * mla_get_device_error - synchronise `stream`, then read and clear the current
 * device's error word.  Returns MLA_OK, MLA_ERR_DEVICE_TIMEOUT,
 * MLA_ERR_DEVICE_BOUNDS, or MLA_ERR_CUDA if the synchronisation itself failed.
 */
MLA_API int mla_get_device_error(void *stream);

/*
 * mla_debug_wait_timeout - exercise the device-side failure path.  The pages
 * have no counterpart: this is a diagnostic of the library's own error
 * handling.  Launches one thread on `stream` that waits, with the same bounded
 * wait every kernel of this library uses, for an mbarrier phase that nothing
 * completes; after `limit_us` microseconds (1 .. 2,000,000) the wait gives up
 * and records MLA_ERR_DEVICE_TIMEOUT in the current device's error word, which
 * mla_get_device_error() then returns.  Nothing faults or traps; the context
 * stays usable.  Returns MLA_OK when launched, MLA_ERR_SHAPE for a limit out
 * of range (nothing launched), MLA_ERR_CUDA if the launch failed.
 */
MLA_API int mla_debug_wait_timeout(unsigned int limit_us, void *stream);

/* mla_status_string - static, NUL-terminated description of a status code. */
MLA_API const char *mla_status_string(int status);

/* mla_version - library version as major*10000 + minor*100 + patch. */
MLA_API int mla_version(void);

/*
 * mla_kernel_launches - kernels this library has launched in this process
 * (every entry point, device and stream; a diagnostic counter, never reset).
 */
MLA_API unsigned long long mla_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
