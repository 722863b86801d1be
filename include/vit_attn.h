/*
 * vit_attn.h -- C ABI of the GB300 (sm_103a) varlen ViT encoder attention library.
 *
 * The hot path of a multimodal vision encoder's attention layer: several images
 * packed into one token stream delimited by cu_seqlens, every token attending
 * only to the tokens of its own image, after 2D vision RoPE and optional
 * per-head Q/K RMSNorm.
 *
 * Sources of the operations (web pages):
 *   [Dots]  vLLM docs, vllm.models.dots3_note.nvidia.vision_attention:
 *           VisionAttention (dense block-diagonal mask), VisionAttentionV2
 *           (per-segment loop), VisionRotaryEmbedding, _RMSNorm,
 *           _VisionAttentionBase._qkv_with_rope.
 *   [TS]    tokenspeed mm_encoder_attention.py: _varlen_metadata, the varlen
 *           backends, MultimodalEncoderAttention.forward (cos/sin duplication).
 *
 * Conventions shared by every call:
 *   - All pointers named *_dev or documented "device" are CUDA device pointers
 *     on the current device. The caller owns every buffer; the library never
 *     allocates or frees device memory and keeps no device state between
 *     calls (apart from the fixed array behind vit_varlen_attn_noalloc).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise, except vit_read_status and vit_kernel_timing_read.
 *   - bf16 tensors are raw 16-bit bfloat16 values ("const void*"), row-major,
 *     laid out [T, H, D] with a caller-given token stride (in elements) and a
 *     head stride of exactly D. Strides of 3*H*D (packed qkv views) are fine.
 *   - Errors the host can see (null pointers, bad sizes, strides, alignment,
 *     a too-small workspace) return a negative vit_status_t at once and launch
 *     nothing. Errors only the device can see (malformed cu_seqlens, a segment
 *     longer than max_seqlen, a grid that does not sum to T, a wait that timed
 *     out) are written into *status_dev when status_dev is non-NULL: kernels
 *     only ever store a negative code there and the first error wins, so the
 *     caller zeroes the word once and reads it with vit_read_status. For
 *     malformed offsets or lengths and a grid that does not sum to T, the
 *     affected call computes nothing and leaves its outputs untouched; after
 *     an expired wait (VIT_ERR_TIMEOUT) or a token position outside the rope
 *     table (VIT_ERR_POSITION_RANGE) its outputs are undefined, but nothing is
 *     read or written out of bounds. No kernel traps or waits without a bound.
 *   - Every call that launches or synchronises opens an NVTX range named after
 *     itself in the "vitattn" domain and closes it on every return, so a
 *     profiler shows each kernel launch under the call that made it.
 */
#ifndef VIT_ATTN_H
#define VIT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *vit_stream_t; /* same type as cudaStream_t */
typedef int vit_status_t;

enum {
    VIT_OK = 0,
    VIT_ERR_NULL_POINTER = -1,       /* a required pointer is NULL */
    VIT_ERR_BAD_HEAD_DIM = -2,       /* head_dim not in {32, 64, 80, 96, 128} */
    VIT_ERR_BAD_SHAPE = -3,          /* T < 0, H < 1, B < 1, T too large, ... */
    VIT_ERR_BAD_STRIDE = -4,         /* token stride < H*D or not a multiple of 8 elements */
    VIT_ERR_MISALIGNED = -5,         /* a tensor pointer is not 16-byte aligned */
    VIT_ERR_WORKSPACE_TOO_SMALL = -6,/* workspace smaller than vit_varlen_attn_workspace_size */
    VIT_ERR_TOO_MANY_SEGMENTS = -7,  /* B (or n_img) above VIT_MAX_SEGMENTS */
    VIT_ERR_CUDA = -8,               /* a CUDA runtime call failed (launch, attribute, ...) */
    VIT_ERR_UNSUPPORTED_DEVICE = -9, /* current device is not compute capability 10.3 */
    VIT_ERR_BAD_SEQLENS = -10,       /* device: cu[0] != 0, cu decreasing, or cu[B] != T */
    VIT_ERR_SEQLEN_EXCEEDS_MAX = -11,/* device: some segment longer than max_seqlen */
    VIT_ERR_GRID_MISMATCH = -12,     /* device: sum of h*w over the grid != T, or h, w < 0 */
    VIT_ERR_TIMEOUT = -13,           /* device: a bounded wait inside a kernel gave up */
    VIT_ERR_BAD_ARGUMENT = -14,      /* any other invalid scalar argument */
    VIT_ERR_POSITION_RANGE = -15     /* device: a token position lies outside the rope table */
};

#define VIT_MAX_SEGMENTS 8192

/* Library version string (never NULL). */
const char *vit_version(void);

/* Human-readable text of a status code (never NULL). */
const char *vit_status_string(vit_status_t status);

/* VIT_OK when `device` is a compute capability 10.3 GPU this library was built for. */
vit_status_t vit_device_supported(int device);

/*
 * 2D vision RoPE frequency table and patch positions.
 *
 * [Dots] VisionRotaryEmbedding(dim, theta): inv_freq[j] = 1 / theta^(2j/dim)
 * for j < dim/2, in fp32; _compute_freqs multiplies positions 0..seqlen-1 by
 * it. For 2D RoPE the table is built with dim = head_dim/2 and used once for
 * the row position and once for the column position of every patch.
 *
 *   dim         rotary table dimension = head_dim / 2 (even, >= 2, <= 256).
 *   theta       base (10000 in the Dots and tokenspeed encoders); > 0.
 *   grid_hw     device int32 [n_img, 2]: patch grid (h, w) of each image, in
 *               packing order.
 *   n_img       number of images, 0 <= n_img <= VIT_MAX_SEGMENTS.
 *   T           total tokens the caller packed; must equal sum(h*w) (checked
 *               on the device, VIT_ERR_GRID_MISMATCH otherwise).
 *   inv_freq    device fp32 [dim/2] output, or NULL.
 *   pos_hw      device int32 [T, 2] output, or NULL: (row, col) of each token
 *               inside its image, row-major (col fastest), restarting at 0 for
 *               every image.
 *   cu_seqlens  device int32 [n_img + 1] output, or NULL: 0, h0*w0, ... (the
 *               offsets VisionAttention and the varlen backends take).
 *   status_dev  device int32 [1] or NULL (see conventions).
 */
vit_status_t vit_rope_freqs(int dim, float theta, const int32_t *grid_hw, int n_img, int64_t T,
                            float *inv_freq, int32_t *pos_hw, int32_t *cu_seqlens,
                            int32_t *status_dev, vit_stream_t stream);

/*
 * Fused QK-RMSNorm + 2D rotate-half RoPE prologue (one pass over q and k).
 *
 * [Dots] _RMSNorm: y = bf16(fp32(x) * rsqrt(mean(fp32(x)^2) + eps)) * weight,
 * applied to q with the q weight and to k with the k weight
 * (_VisionAttentionBase._qkv_with_rope), then RoPE. [TS] forward duplicates a
 * half-width cos/sin table over both halves of the head (rotate-half / NeoX
 * layout). For m < D/2 with angle a_m = row * inv_freq[m] (m < D/4) or
 * col * inv_freq[m - D/4] (m >= D/4):
 *   y[m]       = x[m] cos a_m - x[m + D/2] sin a_m
 *   y[m + D/2] = x[m + D/2] cos a_m + x[m] sin a_m
 * computed in fp32 and rounded to bf16 once.
 *
 *   q_in, k_in     device bf16 [T, H, D], token strides q_in_stride, k_in_stride.
 *   q_out, k_out   device bf16 [T, H, D], token strides q_out_stride,
 *                  k_out_stride; may equal q_in / k_in (in place, same stride).
 *   pos_hw         device int32 [T, 2] from vit_rope_freqs.
 *   inv_freq       device fp32 [D/4] from vit_rope_freqs(dim = D/2).
 *   norm_w         device bf16 [2, D] (row 0 = q weight, row 1 = k weight), or
 *                  NULL for no QK-norm.
 *   eps            RMSNorm epsilon (>= 0), added inside the rsqrt.
 * D must be in {32, 64, 80, 96, 128}; pointers 16-byte aligned; strides
 * multiples of 8 elements and >= H*D.
 */
vit_status_t vit_qk_norm_rope(const void *q_in, void *q_out, const void *k_in, void *k_out,
                              int64_t T, int H, int D,
                              int64_t q_in_stride, int64_t q_out_stride,
                              int64_t k_in_stride, int64_t k_out_stride,
                              const int32_t *pos_hw, const float *inv_freq,
                              const void *norm_w, float eps, vit_stream_t stream);

/* Rotary pairings of vit_qk_norm_rope_ex. */
enum {
    VIT_ROPE_ROTATE_HALF = 0,   /* pairs (m, m + D/2): the NeoX layout of vit_qk_norm_rope */
    VIT_ROPE_INTERLEAVED = 1    /* pairs (2m, 2m + 1) */
};

/*
 * vit_qk_norm_rope with a choice of rotary pairing.
 *
 * [TS] MultimodalEncoderAttention accepts position_embedding_mode
 * "complex_rope" and then rotates q and k with packed_qkv_complex_rotary; the
 * page does not print that routine. It is read here as the complex form of
 * the same rotation: element pair m is (x[2m], x[2m + 1]), one complex number
 * turned by the same angle a_m as in the rotate-half mode:
 *   y[2m]     = x[2m] cos a_m - x[2m + 1] sin a_m
 *   y[2m + 1] = x[2m + 1] cos a_m + x[2m] sin a_m
 * RMSNorm (if norm_w is given) is the same in both modes.
 *
 * Arguments as for vit_qk_norm_rope, plus:
 *   rope_mode   VIT_ROPE_ROTATE_HALF or VIT_ROPE_INTERLEAVED (else
 *               VIT_ERR_BAD_ARGUMENT).
 *   status_dev  device int32 [1] or NULL (see conventions): rows may move
 *               through shared memory with bulk copies whose waits are
 *               bounded; one that expires stores VIT_ERR_TIMEOUT. (The plain
 *               vit_qk_norm_rope passes NULL.)
 * In both calls either half may be left out: q_in and q_out both NULL skip q
 * (its strides are then ignored), k_in and k_out both NULL skip k. Passing
 * only one pointer of a pair, or leaving out both halves, is
 * VIT_ERR_NULL_POINTER.
 */
vit_status_t vit_qk_norm_rope_ex(const void *q_in, void *q_out, const void *k_in, void *k_out,
                                 int64_t T, int H, int D,
                                 int64_t q_in_stride, int64_t q_out_stride,
                                 int64_t k_in_stride, int64_t k_out_stride,
                                 const int32_t *pos_hw, const float *inv_freq,
                                 const void *norm_w, float eps, int rope_mode, int32_t *status_dev,
                                 vit_stream_t stream);

/*
 * Rotary cos/sin table over positions, for the attention call that rotates Q
 * itself (vit_varlen_attn_fused_q).
 *
 * [Dots] VisionRotaryEmbedding builds freqs = outer(arange(max_grid_size),
 * inv_freq) once and the tower indexes it by each patch's (row, col). Same
 * here, with cos and sin already taken:
 *   cos_sin[p][f/2] = {cos a, cos a', sin a, sin a'},  a = p * inv_freq[f],
 *                     a' = p * inv_freq[f + 1],  f = 0, 2, .., D/4 - 2,
 * in fp32, the same product and sincosf the prologue evaluates per token, so
 * both paths rotate with the same bits.
 *
 *   inv_freq   device fp32 [head_dim/4] from vit_rope_freqs(dim = head_dim/2).
 *   head_dim   D, one of {32, 64, 80, 96, 128}.
 *   max_pos    number of positions, >= 1: larger than every row and column
 *              index a token will have (max over images of max(h, w)).
 *   cos_sin    device fp32 output of max_pos * head_dim/2 floats, 16-byte
 *              aligned.
 */
vit_status_t vit_rope_table(const float *inv_freq, int head_dim, int max_pos, float *cos_sin,
                            vit_stream_t stream);

/*
 * Workspace bytes vit_varlen_attn needs for these sizes (an upper bound
 * independent of the segment lengths). Returns 0 for invalid sizes, including
 * sizes whose work list could exceed 2^31 - 1 items (H * (T/64 + B)); the
 * attention calls then return VIT_ERR_BAD_SHAPE.
 */
size_t vit_varlen_attn_workspace_size(int64_t T, int H, int B, int D);

/*
 * Non-causal variable-length packed multi-head attention.
 *
 * [Dots] VisionAttention / VisionAttentionV2: for each segment i of the packed
 * stream, rows [cu[i], cu[i+1]), and each head h:
 *   out[t, h, :] = softmax_j(scale * <q[t, h], k[j, h]>) v[j, h], j in segment i
 * (a block-diagonal mask; no token ever attends across segments), softmax in
 * fp32, bf16 inputs, fp32 accumulation, bf16 output.
 *
 *   q, k, v       device bf16 [T, H, D], token strides q_stride, k_stride, v_stride.
 *   cu_seqlens    device int32 [B + 1] segment offsets, or NULL for B uniform
 *                 segments of T/B tokens ([TS] _varlen_metadata); zero-length
 *                 segments are allowed. Validated on the device.
 *   B             number of segments, 1 <= B <= VIT_MAX_SEGMENTS.
 *   max_seqlen    an upper bound on the segment lengths (may be padded to a
 *                 CUDA-graph bucket, [TS] round_up_to_bucket); a segment longer
 *                 than it is a device error. 0 = not given: T is taken as the
 *                 bound (where [TS] _varlen_metadata reads the exact maximum back
 *                 to the host, this needs no synchronisation). Used for
 *                 validation and to skip the long-segment kernel when no segment
 *                 can be long; never for the results. Negative: VIT_ERR_BAD_ARGUMENT.
 *   scale         softmax scale; <= 0 selects 1/sqrt(D) ([TS] head_size**-0.5).
 *   out           device bf16 [T, H, D] with token stride out_stride (the
 *                 [T, H*D] layout the output projection takes).
 *   workspace     device scratch of >= vit_varlen_attn_workspace_size(T, H, B, D)
 *                 bytes, 16-byte aligned, owned by the caller, overwritten by
 *                 every call (calls sharing one workspace must not overlap).
 * D must be in {32, 64, 80, 96, 128}; T < 2^31.
 */
vit_status_t vit_varlen_attn(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                             int64_t q_stride, int64_t k_stride, int64_t v_stride,
                             const int32_t *cu_seqlens, int B, int max_seqlen, float scale,
                             void *out, int64_t out_stride, void *workspace, size_t workspace_bytes,
                             int32_t *status_dev, vit_stream_t stream);

/*
 * vit_varlen_attn that also returns each row's log-sum-exp.
 *
 * [TS] vision_attn_fa4 notes that the FA4 kernel returns (output, lse) and
 * vision_attn_flashinfer_cudnn calls cuDNN with return_lse=True; the value is
 * what lets a caller merge partial attentions or recompute the softmax. Here:
 *   lse[t, h] = ln( sum_j exp(scale * <q[t, h], k[j, h]>) ), j in t's segment,
 * computed from the kernels' fp32 running max and row sum.
 *
 * Arguments as for vit_varlen_attn, plus:
 *   lse   device fp32 [T, H] (token-major, contiguous, 4-byte aligned), or
 *         NULL (then identical to vit_varlen_attn). Rows of zero-length
 *         segments do not exist; every other row is written.
 */
vit_status_t vit_varlen_attn_lse(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                 int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                 const int32_t *cu_seqlens, int B, int max_seqlen, float scale,
                                 void *out, int64_t out_stride, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, vit_stream_t stream);

/* How vit_varlen_attn_fused_q normalises and rotates Q (all pointers device). */
typedef struct vit_q_rope {
    const int32_t *pos_hw;   /* int32 [T, 2] (row, col) of every token, from vit_rope_freqs */
    const float *cos_sin;    /* table from vit_rope_table(inv_freq, D, max_pos, .) */
    int max_pos;             /* positions in the table */
    const void *norm_w;      /* bf16 [D] q weight (row 0 of the prologue's [2, D]), 16-byte
                                aligned, or NULL for no QK-norm */
    float eps;               /* RMSNorm epsilon, >= 0 */
    int rope_mode;           /* VIT_ROPE_ROTATE_HALF or VIT_ROPE_INTERLEAVED */
} vit_q_rope_t;

/*
 * vit_varlen_attn_lse with the Q half of the prologue fused into the kernels'
 * Q load: `q` holds the raw projections, and every Q tile is normalised and
 * rotated in shared memory after it arrives, before its first product. K must
 * already be normalised and rotated (vit_qk_norm_rope_ex with the q half left
 * out: a one-tensor pre-stage). This removes one write and one read of q from
 * HBM; the result is bit-identical to running vit_qk_norm_rope_ex on q and k
 * and then vit_varlen_attn_lse.
 *
 * Arguments as for vit_varlen_attn_lse, plus:
 *   q_rope   host pointer to the Q normalisation and rotation (see above).
 * Device-detected: a token whose row or column is outside [0, max_pos)
 * stores VIT_ERR_POSITION_RANGE; the table is never read out of range, but
 * the outputs of such a call are undefined.
 */
vit_status_t vit_varlen_attn_fused_q(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                     int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                     const vit_q_rope_t *q_rope,
                                     const int32_t *cu_seqlens, int B, int max_seqlen, float scale,
                                     void *out, int64_t out_stride, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *status_dev, vit_stream_t stream);

/*
 * Attention over a padded layout: segment i is the rows [seq_start[i],
 * seq_start[i] + seq_len[i]) of q, k, v and out, and the rows between
 * segments are padding that is neither read nor written.
 *
 * [TS] vision_attn_flashinfer_cudnn takes per-sequence element offsets for
 * q/k, v and o plus the real (un-padded) sequence_lengths, with max_seqlen as
 * the bucketed budget, so a CUDA graph captured for one bucket of sizes can be
 * replayed for any batch that fits it. Here the offsets are token rows shared
 * by all four tensors (each tensor keeps its own token stride, which is what
 * the page's per-tensor element offsets encode for packed qkv), and nothing
 * on the host depends on the lengths: capture once with the bucket's T, B and
 * max_seqlen, then replay after writing new starts and lengths on the device.
 *
 * Arguments as for vit_varlen_attn_lse, except:
 *   seq_start   device int32 [B]: first row of each segment, ascending.
 *   seq_len     device int32 [B]: real length of each segment (0 allowed).
 *               Checked on the device: every segment inside [0, T), after the
 *               previous segment's end, and no longer than max_seqlen (0:
 *               not given, T is the bound, as in vit_varlen_attn);
 *               otherwise VIT_ERR_BAD_SEQLENS / VIT_ERR_SEQLEN_EXCEEDS_MAX and
 *               nothing is computed.
 *   B           0 <= B <= VIT_MAX_SEGMENTS (0: nothing to do).
 *   q_rope      NULL, or the fused Q normalisation of vit_varlen_attn_fused_q.
 * The workspace size is vit_varlen_attn_workspace_size(T, H, B, D).
 */
vit_status_t vit_varlen_attn_padded(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                    int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                    const int32_t *seq_start, const int32_t *seq_len, int B,
                                    int max_seqlen, float scale, void *out, int64_t out_stride,
                                    float *lse, const vit_q_rope_t *q_rope,
                                    void *workspace, size_t workspace_bytes,
                                    int32_t *status_dev, vit_stream_t stream);

/* Size of the fixed device scratch array behind vit_varlen_attn_noalloc (per GPU). */
#define VIT_NOALLOC_WORKSPACE_BYTES (4u << 20)

/*
 * vit_varlen_attn for callers that cannot allocate device memory. The pages
 * have no counterpart of this call: it exists for code that runs where new
 * device allocations are not allowed or not possible, such as a serving loop
 * whose memory pool is frozen after warm-up, a plugin that is handed only its
 * input and output pointers, or a C caller with no allocator of its own.
 *
 * Arguments, layouts and results are those of vit_varlen_attn without the
 * workspace pair: the scheduler's work list lives instead in a static device
 * array of VIT_NOALLOC_WORKSPACE_BYTES (4 MiB) inside this library, which
 * every GPU that loads the library keeps while its CUDA context lives (until
 * process exit, unless the context is reset; with CUDA's lazy module loading
 * the array is placed when the first call looks it up). The call itself allocates
 * nothing (no cudaMalloc, no cudaFree, no library allocator), and its output
 * is bit-identical to vit_varlen_attn's on the same inputs.
 *   - Limit: sizes whose work list needs more than VIT_NOALLOC_WORKSPACE_BYTES
 *     (vit_varlen_attn_workspace_size(T, H, B, D) > 4 MiB; roughly
 *     H * (T/64 + B) > 262000 work items) return VIT_ERR_WORKSPACE_TOO_SMALL
 *     and launch nothing; use vit_varlen_attn with your own workspace there.
 *     Every other argument is checked first, exactly as vit_varlen_attn does.
 *   - The first call in each CUDA context (the device's primary context, and
 *     again after cudaDeviceReset or any other re-creation of it) looks up the
 *     array's device address (cudaGetSymbolAddress, with that device current).
 *     Make that call before any stream capture: a call that would need the
 *     lookup while `stream` is being captured returns VIT_ERR_BAD_ARGUMENT and
 *     touches nothing; later calls only launch.
 *   - All calls on a device share the one array, and it keeps whatever the
 *     previous call left there; every call rewrites what it reads, so nothing
 *     needs clearing, but two calls that overlap on the GPU (different streams
 *     without ordering between them) race on it and must not be issued.
 */
vit_status_t vit_varlen_attn_noalloc(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                     int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                     const int32_t *cu_seqlens, int B, int max_seqlen, float scale,
                                     void *out, int64_t out_stride, int32_t *status_dev, vit_stream_t stream);

/*
 * Per-call options of vit_varlen_attn_ex. Every field has a "library default"
 * value; a NULL options pointer means all defaults. The options only choose
 * how the work is spread over the kernels: results agree within the output
 * tolerance for every setting, and the workspace size does not depend on them.
 *
 *   short_segment_max   kernel split: segments of at most
 *                       min(short_segment_max, 64) tokens run on the
 *                       tiny-segment (warp-MMA) kernel, one item per segment
 *                       and a few heads; longer ones on the tcgen05/TMEM
 *                       long-segment kernel. 0 sends every segment to the long
 *                       kernel; values above 64 act as 64 (the tiny kernel's
 *                       bound; above it the long kernel is the faster one on
 *                       GB300). -1 = library default (64). Below -1:
 *                       VIT_ERR_BAD_ARGUMENT.
 */
typedef struct vit_attn_options {
    int short_segment_max;
} vit_attn_options_t;

/*
 * The general attention call: every option of the calls above in one place.
 * The segments come either from cu_seqlens (packed, as vit_varlen_attn; seq_start
 * and seq_len NULL) or from seq_start and seq_len (a padded layout, as
 * vit_varlen_attn_padded; cu_seqlens NULL); giving both is VIT_ERR_BAD_ARGUMENT.
 * lse (vit_varlen_attn_lse) and q_rope (vit_varlen_attn_fused_q) may be NULL.
 * opts: host pointer to per-call options, or NULL for the defaults. Nothing of
 * a call's configuration is kept between calls, so threads that issue calls
 * with different options do not affect one another.
 */
vit_status_t vit_varlen_attn_ex(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                const int32_t *cu_seqlens, const int32_t *seq_start, const int32_t *seq_len,
                                int B, int max_seqlen, float scale,
                                void *out, int64_t out_stride, float *lse, const vit_q_rope_t *q_rope,
                                const vit_attn_options_t *opts, void *workspace, size_t workspace_bytes,
                                int32_t *status_dev, vit_stream_t stream);

/*
 * Synchronise `stream`, then read the status word. Returns VIT_OK, the first
 * device-detected error code stored there, or VIT_ERR_CUDA when the stream or
 * the copy failed. The only call of the compute path that blocks the host.
 */
vit_status_t vit_read_status(const int32_t *status_dev, vit_stream_t stream);

/* ---- instrumentation (benchmarks and tests) ---- */

/* Total number of kernels this library has launched since it was loaded. */
int64_t vit_launch_count(void);

typedef struct {
    const char *name;   /* kernel name (static string) */
    int64_t launches;   /* launches recorded since the last read */
    double total_ms;    /* sum of their device durations (CUDA events on the launch stream) */
} vit_kernel_time_t;

/* Turn per-launch CUDA-event timing of every kernel on (1) or off (0). Returns the previous state. */
int vit_kernel_timing(int enable);

/*
 * Wait for the recorded events, aggregate per kernel name into out[0..max_entries),
 * clear the record, and return the number of entries written (< 0 on error).
 */
int vit_kernel_timing_read(vit_kernel_time_t *out, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* VIT_ATTN_H */
