/*
 * sageattn.h -- C ABI of the GB300 (sm_103a) attention forward library.
 *
 * Three operations, each defined on the pages this library restates:
 *
 *   attn_fwd_bf16   O = softmax(scale * Q K^T) V, non-causal self-attention,
 *                   BF16 [B, S, H, 128] in and out, computed tile by tile with
 *                   an online softmax so the S x S score matrix is never
 *                   stored.  (ai-infra handbook, "Kernel acceleration:
 *                   attention, compilation and fusion", section "Attention:
 *                   from O(N^2) memory to blocks"; the RDNA2 DiT flash kernel
 *                   note, Contribution.)
 *   sage_prepare    the input stage of the SageAttention-style forward: INT8
 *                   codes for Q and K, every 32 rows of a (batch, head) sharing
 *                   one FP32 scale (Q's scales also hold softmax_scale * log2 e);
 *                   e4m3 codes for V stored channel-major, [B, H, 128, S_pad],
 *                   each channel with its own FP32 scale; optionally an RMSNorm and a
 *                   rotate-half RoPE of Q and K beforehand, with the BF16
 *                   rounding points of PyTorch's eager sequence.  (aiter pull
 *                   request "gfx1201_sage_prepare / gfx1201_sage_attention",
 *                   commit message of gfx1201_sage_prepare; Technical Details.)
 *   sage_attn_fwd   the attention kernel by itself, on tensors a prepare wrote: Q K^T on
 *                   the INT8 codes, P V with P and V in FP8 e4m3, FP32
 *                   accumulation, online softmax, BF16 output.  (Same pull
 *                   request, commit message of gfx1201_sage_attention, whose
 *                   op also exposes the kernel on its own for inputs already
 *                   prepared.)
 *   sage_attention  prepare + kernel as one call (that pull request's
 *                   gfx1201_sage_attention op), the prepared tensors kept in
 *                   the caller's workspace.
 *
 * Beyond those: sage_prepare_smooth_k (K smoothing before the INT8
 * quantisation), sage_prepare_smoothed with sage_attn_fwd_smooth_q and
 * sage_attn_fwd_pv16_smooth_q (Q smoothing with its correction term) and
 * sage_attn_fwd_pv16 (P V in 16 bits with V unquantised), all from the
 * handbook's SageAttention section; sage_prepare_noalloc (no
 * workspace argument); attn_selftest_wait_timeout (exercises the failure path);
 * attn_sm_clock_sample (SM clock counters, for timing); sage_e4m3_encode (the
 * e4m3 conversion the prepare and the FP8 P V use, on its own);
 * sizes and status helpers.
 *
 * Conventions shared by every call
 *   - D (head dimension) must be 128; S >= 1 (attention over no keys is undefined:
 *     S = 0 is ATTN_ERR_INVALID_ARG).  B = 0 or H = 0 is an empty problem: every call
 *     returns ATTN_OK at once, writing and reading nothing (its pointers may be NULL).
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller; the library never allocates, frees or keeps them.
 *     Every pointer must be 16-byte aligned (sage_e4m3_encode's arrays need only
 *     their element alignment).  A call's outputs and workspace must not overlap
 *     its inputs or one another.
 *   - BF16 tensors are addressed as [B, S, H, 128] with element strides given
 *     as int64_t str[3] = {stride_b, stride_s, stride_h}; the channel stride is
 *     1.  Each stride must be a positive multiple of 8 elements (16 bytes);
 *     the stride of a dimension of extent 1 is ignored.  Views such as the
 *     [B, H, S, D] storage seen through its [B, S, H, D] permutation are
 *     accepted as they are.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and enqueue kernels and memsets only (except
 *     attn_get_device_status and attn_selftest_wait_timeout, which
 *     synchronise).  Argument errors are found on the host before anything is
 *     enqueued.
 *   - Each call returns ATTN_OK or an error; attn_last_error() gives the
 *     message of the calling thread's last failed call.
 *   - Device-side pipeline waits are bounded (about 2 s).  A wait that runs
 *     out makes its kernel stop early and records the fact in a device error
 *     word; attn_get_device_status() reports and clears it.
 *   - The library runs on sm_103 devices only; elsewhere every call returns
 *     ATTN_ERR_UNSUPPORTED.
 *   - Sizes: B * H * S_pad / 128 must stay below 2^31 (S_pad = the padded
 *     length, sage_padded_len(S) where the call takes none); the prepare
 *     stages also take at most 65535 heads per batch entry (H <= 65535).
 *     Larger calls return ATTN_ERR_INVALID_ARG.
 *   - Host-side state (the device check, kernel attributes, the SM count) is
 *     set up on first use in each CUDA context, under a lock: calls may come
 *     from several host threads.
 */
#ifndef SAGEATTN_H_
#define SAGEATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* == cudaStream_t */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null pointer, bad extent, bad stride, bad option */
  ATTN_ERR_ALIGNMENT = 2,      /* pointer not 16-byte aligned, stride not a multiple of 8 elements */
  ATTN_ERR_UNSUPPORTED = 3,    /* not an sm_103 device, or D != 128 */
  ATTN_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (message has the CUDA error) */
  ATTN_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up on a bounded wait (from attn_get_device_status) */
} attn_status;

/*
 * attn_fwd_bf16 -- O = softmax(softmax_scale * Q K^T) V over all S keys.
 *   q, k, v : const BF16 [B, S, H, 128], strides q_str/k_str/v_str
 *   o       : BF16 [B, S, H, 128] output, stride o_str; must not overlap q/k/v
 *   softmax_scale : any finite float (1/sqrt(128) for the usual attention)
 * Result is FP32-accumulated and rounded to BF16 once.  No mask, no causal
 * variant, no dropout.
 */
ATTN_API attn_status attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, int B, int S, int H, int D,
                          const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                          const int64_t o_str[3], float softmax_scale, attn_stream_t stream);

/* sage_padded_len -- S rounded up to a multiple of 128: the smallest valid S_pad. */
ATTN_API int64_t sage_padded_len(int64_t S);

/*
 * sage_prepare_workspace_size -- bytes of device scratch sage_prepare needs
 * for B x H heads (the per-channel V maxima, reduced across the sequence
 * before any V element can be encoded).  The caller allocates it.
 */
ATTN_API size_t sage_prepare_workspace_size(int B, int H);

/*
 * sage_prepare -- quantise Q, K and V for sage_attn_fwd.
 *   q, k, v    : const BF16 [B, S, H, 128] with strides q_str/k_str/v_str
 *   softmax_scale : folded, with log2(e), into q_scale:
 *                   c = (float)((double)softmax_scale * log2(e))
 *   q_norm_w, k_norm_w : BF16 [128] RMSNorm weights, both given or both NULL.
 *                   When given, each 128-channel head row x of Q (resp. K) is
 *                   replaced by bf16(bf16(x * r) * w), r = 1/sqrt(mean(x^2) + rms_eps),
 *                   all in binary32 (sum of squares: eight partial sums over
 *                   channels [16L, 16L+16) added left to right, combined
 *                   pairwise like an XOR butterfly at distances 4, 2, 1; sqrt
 *                   and the division each rounded once).
 *   rope_cos, rope_sin : BF16 [S, rope_dim] tables (contiguous), both given
 *                   when rope_dim > 0; rope_dim in {0, 32, 64, 96, 128}.
 *                   Channels c < rope_dim of Q and K (after the norm) become
 *                   bf16(bf16(x[c] cos[s,c]) + bf16(rot[c] sin[s,c])) with
 *                   rot[c] = -x[c + rope_dim/2] for c < rope_dim/2 and
 *                   x[c - rope_dim/2] otherwise; other channels pass through.
 *   S_pad      : padded length, a multiple of 128 and >= S
 *   outputs (caller-allocated device memory, every byte written, padding zero):
 *     q_i8, k_i8 : int8 [B, H, S_pad, 128], code = clamp(rint(x * (127/a)), -127, 127)
 *                  with a = max |x| over the valid rows of the 32-row block
 *     q_scale    : float [B, H, S_pad/32], (a/127) * c   (0 for an all-zero or padding block)
 *     k_scale    : float [B, H, S_pad/32], a/127
 *     v_fp8      : e4m3 bytes [B, H, 128, S_pad], code = e4m3_rn_satfinite(v * (448/a_ch)),
 *                  a_ch = max over s < S of |v[b, s, h, ch]|
 *     v_scale    : float [B, H, 128], a_ch / 448
 *   workspace  : device scratch of at least sage_prepare_workspace_size(B, H)
 *                bytes, 16-byte aligned; its contents on entry do not matter.
 * Every binary32 operation above is rounded once to nearest-even (no fused
 * multiply-add), so the outputs are a deterministic function of the inputs.
 * Enqueues a memset and two kernels on `stream`.
 */
ATTN_API attn_status sage_prepare(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                         const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                         float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                         const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad, int8_t* q_i8,
                         int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale, float* v_scale,
                         void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * sage_prepare_smooth_k_workspace_size -- bytes of device scratch
 * sage_prepare_smooth_k needs: the V maxima of sage_prepare plus one float per
 * (b, h, 32-row block, channel) of block sums of K.
 */
ATTN_API size_t sage_prepare_smooth_k_workspace_size(int B, int H, int64_t S_pad);

/*
 * sage_prepare_smooth_k -- sage_prepare with K smoothing.  SageAttention
 * subtracts the mean of K before quantising it, which removes K's outlier
 * channels (ai-infra handbook, "Kernel acceleration: attention, compilation
 * and fusion", section "SageAttention: quantizing attention too"); read here
 * as one mean per (batch, head, channel) over the S tokens.  In exact
 * arithmetic the attention output is unchanged: every score of a query row
 * moves by the same q . k_mean, which the softmax cancels, so the result goes
 * to sage_attn_fwd as it is.
 *   All arguments as sage_prepare, plus
 *   k_mean     : float [B, H, 128] output (caller-allocated, 16-byte aligned):
 *                k_mean[b,h,c] = (sum over s < S of K'[b,s,h,c]) / S, K' being
 *                K after the optional RMSNorm + RoPE.  The sum is taken in a
 *                fixed binary32 order: per 32-row block j, four partial sums
 *                P_g over rows 32j+4t+g (t = 0..7, ascending, from 0; rows >= S
 *                skipped), B_j = (P_0 + P_1) + (P_2 + P_3), then the B_j added in
 *                ascending j from 0, then divided by S.
 *   k_i8, k_scale : as sage_prepare, of fl32(K' - k_mean[b,h,c]) in place of K'.
 *   workspace  : at least sage_prepare_smooth_k_workspace_size(B, H, S_pad)
 *                bytes, 16-byte aligned; its contents on entry do not matter.
 * q_i8, q_scale, v_fp8 and v_scale are those of sage_prepare, bit for bit.
 * Enqueues a memset and four kernels on `stream`.  Errors as sage_prepare;
 * k_mean NULL -> ATTN_ERR_INVALID_ARG, misaligned -> ATTN_ERR_ALIGNMENT.
 */
ATTN_API attn_status sage_prepare_smooth_k(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                  const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                  float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                  const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad,
                                  int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale,
                                  float* v_scale, float* k_mean, void* workspace, size_t workspace_bytes,
                                  attn_stream_t stream);

/*
 * sage_prepare_smoothed -- sage_prepare with Q smoothing, K smoothing or both.
 * SageAttention subtracts the block means of Q as well as of K before the INT8
 * quantisation (ai-infra handbook, "Kernel acceleration: attention, compilation
 * and fusion", section "SageAttention: quantizing attention too").  K's mean
 * cancels in the softmax (sage_prepare_smooth_k).  Q's does not: with
 * q = (q - qbar) + qbar, q . k_j = (q - qbar) . k_j + qbar . k_j, and the
 * correction term qbar . k_j differs from key to key, so the mean is kept with
 * its block and added back in the score product (sage_attn_fwd_smooth_q).
 *   All arguments as sage_prepare_smooth_k, plus
 *   smooth_q, smooth_k : 0 or 1 each.
 *   q_mean     : with smooth_q, binary16 [B, H, S_pad/32, 128] output (16-byte
 *                aligned): each 32-row block's per-channel mean of Q' (Q after
 *                the optional RMSNorm + RoPE), in units of the block's step,
 *                m[c] = f16(fl32(qbar[c] * inv)).  qbar[c] is the block sum in
 *                k_mean's fixed order (four partial sums over rows 32j+4t+g,
 *                (P_0 + P_1) + (P_2 + P_3)) divided by the block's valid rows.
 *   q_i8, q_scale : with smooth_q, the codes of d = fl32(Q' - qbar[c]); the step
 *                is a_eff / 127 with a_eff = max(max |d|, max_c |qbar[c]| / 256)
 *                (so |m| <= 32512 stays in binary16), inv = fl32(127 / a_eff),
 *                q_scale = fl32(fl32(a_eff / 127) * c).  An all-zero block, or
 *                one whose 127 / a_eff overflows (every |Q'| below about
 *                3.7e-37), is stored as zero codes, zero means and scale 0.
 *   k_mean     : with smooth_k, as sage_prepare_smooth_k (else not written).
 *   workspace  : sage_prepare_smooth_k_workspace_size(B, H, S_pad) bytes with
 *                smooth_k, else sage_prepare_workspace_size(B, H).
 * Outputs not affected by a flag are those of sage_prepare, bit for bit.
 * Errors as sage_prepare_smooth_k; a flag other than 0/1, or a NULL q_mean
 * (k_mean) with smooth_q (smooth_k) -> ATTN_ERR_INVALID_ARG.
 */
ATTN_API attn_status sage_prepare_smoothed(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                           const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                           float softmax_scale, const void* q_norm_w, const void* k_norm_w,
                                           float rms_eps, const void* rope_cos, const void* rope_sin, int rope_dim,
                                           int64_t S_pad, int smooth_q, int smooth_k, int8_t* q_i8, int8_t* k_i8,
                                           uint8_t* v_fp8, float* q_scale, float* k_scale, float* v_scale,
                                           void* q_mean, float* k_mean, void* workspace, size_t workspace_bytes,
                                           attn_stream_t stream);

/*
 * sage_prepare_noalloc -- sage_prepare without a workspace argument.  None of the
 * pages has a counterpart; it exists for callers that cannot allocate device
 * memory when they call us: code whose device memory is owned and budgeted by
 * a host framework or engine, code that must not risk an out-of-memory failure
 * or the device-wide synchronisation cudaMalloc/cudaFree can cause in the middle
 * of a step, and plug-ins that are handed input and output buffers only.
 *   Arguments, layouts, results and errors are those of sage_prepare (the outputs
 *   are bit-identical); the scratch it needs (the per-channel maxima of |V|) is a
 *   1 MiB array inside this library instead:
 *   - limit: B * H <= 2048 heads; larger calls return ATTN_ERR_INVALID_ARG without
 *     launching anything (use sage_prepare for them);
 *   - the array lives on every device that loads the library, until the process
 *     exits; this function never calls cudaMalloc, cudaFree or any allocating
 *     routine;
 *   - its first call in a CUDA context looks the array's device address up
 *     (a runtime query, once per context: the address belongs to the module as
 *     loaded in that context, so a reset device or a second context of the
 *     same device looks it up again); make that first call before capturing
 *     a stream;
 *   - all calls on a device share the array: the call clears it on `stream`
 *     before use, so what an earlier call left does not matter, but two calls
 *     whose work can overlap on the GPU (different streams without ordering)
 *     race on it -- order them.
 */
ATTN_API attn_status sage_prepare_noalloc(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                          const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                          float softmax_scale, const void* q_norm_w, const void* k_norm_w,
                                          float rms_eps, const void* rope_cos, const void* rope_sin, int rope_dim,
                                          int64_t S_pad, int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8,
                                          float* q_scale, float* k_scale, float* v_scale, attn_stream_t stream);

/*
 * sage_attn_workspace_size -- bytes of device scratch sage_attn_fwd needs:
 * the INT8 Q and K codes widened to FP16, 2 * 2 * B * H * S_pad * 128 bytes.
 * (sm_103a has no INT8 tensor-core MMA; the codes are widened exactly and the
 * Q K^T product runs on the FP16 MMA, which is exact for these integers.)
 */
ATTN_API size_t sage_attn_workspace_size(int B, int H, int64_t S_pad);

/*
 * sage_attn_fwd -- attention on prepared tensors (layouts as sage_prepare writes them):
 *   t[r, j] = (q_i8[r] . k_i8[j]) * q_scale[r/32] * k_scale[j/32]   (exact integer dot
 *             product; Q's scale carries softmax_scale * log2 e, so t is in log2 units),
 *             keys j >= S are masked out;
 *   O[r, d] = v_scale[d] * sum_j e4m3(p'[r,j]) v_fp8[d, j] / sum_j p'[r,j],
 *             p'[r,j] = 448 * 2^-4 * 2^(t[r,j] - m_r), m_r a running row maximum that
 *             is raised whenever a tile's maximum exceeds it by more than 4; the
 *             constant cancels in the ratio.  FP32 accumulation, one BF16 rounding.
 *   o          : BF16 [B, S, H, 128] output with element strides o_str.
 *   workspace  : device scratch of at least sage_attn_workspace_size(B, H, S_pad) bytes,
 *                16-byte aligned; overwritten, contents on entry do not matter.
 * Enqueues two kernels on `stream`.
 */
ATTN_API attn_status sage_attn_fwd(const int8_t* q_i8, const int8_t* k_i8, const uint8_t* v_fp8, const float* q_scale,
                          const float* k_scale, const float* v_scale, void* o, const int64_t o_str[3], int B,
                          int S, int H, int D, int64_t S_pad, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream);

/*
 * sage_attn_fwd_pv16 -- the Sage forward with a 16-bit P V product: Q K^T on
 * the INT8 codes exactly as sage_attn_fwd, then P (BF16) times V taken from the
 * BF16 input itself, FP32 accumulation, BF16 output.  The handbook's
 * SageAttention section has P and V "in FP8 or FP16" (ai-infra handbook,
 * "Kernel acceleration: attention, compilation and fusion", section
 * "SageAttention: quantizing attention too"); this is the 16-bit choice,
 * with BF16 because V arrives in BF16.  It trades the FP8 product's speed for
 * accuracy: V is not quantised and P carries 8 significant bits instead of 4.
 *   O[r, d] = sum_j p[r, j] v[j, d] / sum_j p[r, j],  p = bf16(2^(t - m_r)),
 *   t as in sage_attn_fwd, m_r the row's reference maximum (moved only when a
 *   tile's maximum passes it by more than 32 log2 units), the denominator summed
 *   from the unrounded p in FP32.
 *   q_i8, k_i8, q_scale, k_scale : from sage_prepare or sage_prepare_smooth_k
 *                (its v_fp8 / v_scale outputs are not read)
 *   v          : const BF16 [B, S, H, 128] with element strides v_str
 *   o, o_str, B, S, H, D, S_pad, workspace, workspace_bytes : as sage_attn_fwd
 * Enqueues two kernels on `stream`.  Errors as sage_attn_fwd, plus v's
 * checks (NULL, alignment, strides) as attn_fwd_bf16.
 */
ATTN_API attn_status sage_attn_fwd_pv16(const int8_t* q_i8, const int8_t* k_i8, const float* q_scale,
                                        const float* k_scale, const void* v, const int64_t v_str[3], void* o,
                                        const int64_t o_str[3], int B, int S, int H, int D, int64_t S_pad,
                                        void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * sage_attn_fwd_smooth_q, sage_attn_fwd_pv16_smooth_q -- sage_attn_fwd and
 * sage_attn_fwd_pv16 on tensors prepared with Q smoothing (sage_prepare_smoothed,
 * smooth_q = 1).  Q's operand of the score product is the binary16 value
 * f16(q_i8[r, d] + q_mean[r/32, d]) -- the code and the block mean in step
 * units, summed and rounded once -- so that
 *   t[r, j] = (sum_d f16(q_i8[r,d] + q_mean[r/32,d]) k_i8[j,d]) * q_scale[r/32] * k_scale[j/32]
 * carries the correction term qbar . k_j; the FP32 accumulation of that sum is
 * exact while it stays below 2^24 in magnitude.  The rest is as sage_attn_fwd
 * (resp. sage_attn_fwd_pv16).
 *   q_mean : const binary16 [B, H, S_pad/32, 128], 16-byte aligned
 * Enqueues three kernels on `stream`.  Errors as sage_attn_fwd (resp.
 * sage_attn_fwd_pv16); q_mean NULL -> ATTN_ERR_INVALID_ARG.
 */
ATTN_API attn_status sage_attn_fwd_smooth_q(const int8_t* q_i8, const void* q_mean, const int8_t* k_i8,
                                            const uint8_t* v_fp8, const float* q_scale, const float* k_scale,
                                            const float* v_scale, void* o, const int64_t o_str[3], int B, int S,
                                            int H, int D, int64_t S_pad, void* workspace, size_t workspace_bytes,
                                            attn_stream_t stream);
ATTN_API attn_status sage_attn_fwd_pv16_smooth_q(const int8_t* q_i8, const void* q_mean, const int8_t* k_i8,
                                                 const float* q_scale, const float* k_scale, const void* v,
                                                 const int64_t v_str[3], void* o, const int64_t o_str[3], int B,
                                                 int S, int H, int D, int64_t S_pad, void* workspace,
                                                 size_t workspace_bytes, attn_stream_t stream);

/*
 * sage_attention_workspace_size -- bytes of device scratch sage_attention needs
 * (0 for an empty problem).  smooth_k, pv_bf16 and q_on_load as given to
 * sage_attention (the size does not depend on smooth_q).
 */
ATTN_API size_t sage_attention_workspace_size(int B, int H, int64_t S_pad, int smooth_k, int pv_bf16,
                                              int q_on_load);

/*
 * sage_attention -- the SageAttention-style forward as one call: the prepare
 * stage followed by the forward, as the aiter pull request's
 * gfx1201_sage_attention op does it (commit message of gfx1201_sage_attention:
 * prepare + kernel).  The prepared tensors never leave `workspace`: the Q/K codes
 * are written there as FP16 (the exact values of the INT8 codes, the operand the
 * Q K^T MMA reads), which spares the INT8 round trip and the widening pass of
 * sage_prepare + sage_attn_fwd.  With q_on_load = 1, Q is instead quantised
 * inside the attention kernel as it is loaded (each row after its optional
 * RMSNorm and RoPE, the same arithmetic as sage_prepare), so Q's codes never
 * reach memory; on a GB300 that measured slower (the coding sits on every CTA's
 * path to its first product, while the prepare's Q pass overlaps its K and V
 * passes), so it is not the default.  Either way the output is bit-identical to
 * the two-call sequence.
 *   q, k, v, strides, softmax_scale, RMSNorm and RoPE arguments : as sage_prepare
 *   smooth_q   : 0 or 1 -- Q smoothing as sage_prepare_smoothed (the FP16 Q operand
 *                written to the workspace is then f16(code + block mean)); not
 *                with q_on_load (ATTN_ERR_UNSUPPORTED)
 *   smooth_k   : 0 or 1 -- K smoothing as sage_prepare_smooth_k
 *   pv_bf16    : 0 -- P and V in e4m3 (sage_attn_fwd); 1 -- P in BF16 times the
 *                BF16 V input (sage_attn_fwd_pv16; V is then not quantised)
 *   q_on_load  : 0 -- Q and K coded by the prepare; 1 -- Q coded by the forward as
 *                it is loaded; 2 -- Q and K coded by the forward as they are loaded
 *                (each K tile by a softmax warpgroup while its next S product runs;
 *                the block scales stay in shared memory; with pv_bf16 = 1 no prepare
 *                kernel runs at all).  Every CTA of a head then codes all of the
 *                head's K tiles, so on a GB300 level 2 measured slower at every size
 *                (3x at 76112 tokens); levels 1 and 2 exist for callers that must not
 *                write codes to memory.  Not with smooth_q (1, 2) or smooth_k (2):
 *                ATTN_ERR_UNSUPPORTED
 *   o, o_str   : BF16 [B, S, H, 128] output, element strides (as sage_attn_fwd)
 *   workspace  : at least sage_attention_workspace_size(B, H, sage_padded_len(S),
 *                smooth_k, pv_bf16, q_on_load) bytes, 16-byte aligned; contents
 *                on entry do not matter.  May be NULL when that size is 0
 *                (pv_bf16 = 1 with q_on_load = 2: nothing is prepared).
 * Enqueues the prepare kernels (one to four) and the attention kernel on
 * `stream`.  Errors as sage_prepare and sage_attn_fwd; smooth_q, smooth_k or
 * pv_bf16 other than 0/1, q_on_load other than 0/1/2 -> ATTN_ERR_INVALID_ARG.
 */
ATTN_API attn_status sage_attention(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                    const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                    float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                    const void* rope_cos, const void* rope_sin, int rope_dim, int smooth_q,
                                    int smooth_k, int pv_bf16, int q_on_load, void* o, const int64_t o_str[3],
                                    void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_get_device_status -- synchronise `stream`, then read and clear the
 * device error words of all kernels.  ATTN_OK if no bounded wait ran out
 * since the last call, ATTN_ERR_DEVICE_TIMEOUT otherwise, ATTN_ERR_CUDA if
 * the synchronisation itself failed.
 */
ATTN_API attn_status attn_get_device_status(attn_stream_t stream);

/*
 * attn_selftest_wait_timeout -- exercises the failure path described above on
 * this GPU.  It launches the BF16 attention kernel on a [1, 128, 1, 128] problem
 * with its tile loads withheld, so that the MMA warp's first wait (for Q) runs
 * out after the kernels' wait limit (2 s of %globaltimer); the kernel then
 * raises its abort flag, the other roles leave their loops, TMEM is freed and
 * the kernel returns.  The call synchronises `stream` and returns what
 * attn_get_device_status reports for that launch: ATTN_ERR_DEVICE_TIMEOUT when
 * the failure path works.  The context stays usable afterwards.
 *   q, k, v, o : BF16 [1, 128, 1, 128] contiguous device buffers (nothing is read
 *                from q, k, v; o is not written)
 * Takes about 2 s.  Errors: bad pointers -> ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_ALIGNMENT; not an sm_103 device -> ATTN_ERR_UNSUPPORTED.
 */
ATTN_API attn_status attn_selftest_wait_timeout(const void* q, const void* k, const void* v, void* o,
                                                attn_stream_t stream);

/*
 * attn_sm_clock_sample -- an instrumentation helper for timing, not part of the
 * method: enqueues on `stream` a clear of `out` and a small kernel whose CTAs
 * record, for the SM each runs on, that SM's cycle counter (%clock64) and the
 * GPU's nanosecond timer (%globaltimer).  Two samples around a region give each
 * SM's average clock over it: (cycles_b - cycles_a) / (ns_b - ns_a) GHz.
 *   out     : device uint64 [n_slots][2] = {cycles, ns} per SM index (%smid);
 *             slots of SMs that ran no CTA stay 0
 *   n_slots : >= the device's SM count (SM indices past it are not recorded)
 * Errors: NULL or misaligned out, n_slots < 1 -> ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_ALIGNMENT; launch failure -> ATTN_ERR_CUDA.
 */
ATTN_API attn_status attn_sm_clock_sample(uint64_t* out, int n_slots, attn_stream_t stream);

/*
 * sage_e4m3_encode -- FP8 e4m3 codes of n binary32 values: round to nearest,
 * ties to the even code, magnitudes beyond 448 saturate to +-448, NaN gives
 * 0x7f (the V format of the aiter pull request "gfx1201_sage_prepare /
 * gfx1201_sage_attention", Technical Details, with the rounding sage_prepare
 * documents).  It runs the same packing as sage_prepare's V codes and the FP8
 * P of the Sage forward, so the conversion they share can be checked on its
 * own, and serves callers that quantise other tensors the same way.
 *   x : device float32 [n] (4-byte aligned);  y : device uint8 [n], written (any
 *       alignment); the two ranges must not overlap
 *   n : number of values; 0 returns ATTN_OK at once
 * Enqueues one kernel on `stream`.  Errors: n < 0, NULL x or y (n > 0) ->
 * ATTN_ERR_INVALID_ARG; launch failure -> ATTN_ERR_CUDA.
 */
ATTN_API attn_status sage_e4m3_encode(const float* x, uint8_t* y, int64_t n, attn_stream_t stream);

/* attn_last_error -- message of the calling thread's last failed call ("" if none). */
ATTN_API const char* attn_last_error(void);

/* attn_status_name -- the enumerator's name, e.g. "ATTN_ERR_ALIGNMENT". */
ATTN_API const char* attn_status_name(attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* SAGEATTN_H_ */
