/*
 * fp64 CPU oracle for varlen ViT encoder attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, and where each step is defined (vLLM docs page
 * "vllm.models.dots3_note.nvidia.vision_attention" = p1; tokenspeed
 * "mm_encoder_attention.py" = p3):
 *
 *   vo_rope_inv_freq   inverse frequencies 1/theta^(2j/dim), j < dim/2
 *                      (p1, VisionRotaryEmbedding.__init__); the table is
 *                      built for dim = head_dim/2 (one half of the head for
 *                      the h angles, the other for the w angles).
 *   vo_grid_positions  0-based (row, col) of every packed token inside its
 *                      image, row-major, plus the segment offsets; positions
 *                      start at 0 like arange(seqlen) in
 *                      VisionRotaryEmbedding._compute_freqs (p1).
 *   vo_norm_rope       per (token, head) row: optional RMSNorm
 *                      w * x / sqrt(mean(x^2) + eps) (p1, _RMSNorm.forward /
 *                      _norm) followed by 2D rotate-half RoPE with cos/sin
 *                      duplicated over both halves of the head (p3,
 *                      MultimodalEncoderAttention.forward, the
 *                      cat([cos, cos]) step); norm before RoPE as in p1
 *                      _VisionAttentionBase._qkv_with_rope.
 *                      The interleaved mode pairs x[2m] with x[2m+1]
 *                      instead (p3's "complex_rope" position-embedding mode,
 *                      MultimodalEncoderAttention.__init__ and the
 *                      packed_qkv_complex_rotary call in forward: each pair is
 *                      one complex number turned by the same angle a_m).
 *   vo_attention       per segment of the packed stream and per head:
 *                      softmax(scale * q k^T) v over that segment's keys only
 *                      (p1, VisionAttentionV2.forward: split by segment
 *                      lengths, plain attention per segment, concatenate),
 *                      and optionally the natural-log sum of exp(scale * s)
 *                      per row (the lse that p3's FA4 and cuDNN backends
 *                      return next to the output, vision_attn_fa4 and
 *                      vision_attn_flashinfer_cudnn with return_lse=True).
 *
 * Everything is evaluated in double precision from the exact bf16 inputs
 * (bf16 -> fp64 is exact). No blocking, fusion or reordering beyond the plain
 * definition: scores for one query row, their maximum, exp, sum, weighted V.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int vo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* inv_freq[j] = 1 / theta^(2j/dim) for j = 0 .. dim/2 - 1. */
void vo_rope_inv_freq(int dim, double theta, double *inv_freq)
{
    for (int j = 0; j < dim / 2; ++j)
        inv_freq[j] = 1.0 / pow(theta, (2.0 * j) / (double)dim);
}

/*
 * grid_hw: n_img pairs (h, w). Writes cu[n_img + 1] (segment offsets) and
 * pos[2 * T] with pos[2t] = row, pos[2t + 1] = col of token t inside its
 * image, row-major (col fastest). Returns T.
 */
int64_t vo_grid_positions(const int32_t *grid_hw, int n_img, int32_t *cu, int32_t *pos)
{
    int64_t t = 0;
    cu[0] = 0;
    for (int i = 0; i < n_img; ++i) {
        int h = grid_hw[2 * i], w = grid_hw[2 * i + 1];
        for (int r = 0; r < h; ++r)
            for (int c = 0; c < w; ++c) {
                if (pos) {
                    pos[2 * t] = r;
                    pos[2 * t + 1] = c;
                }
                ++t;
            }
        cu[i + 1] = (int32_t)t;
    }
    return t;
}

/*
 * x: bf16 bits, row (t, h) starts at x + t * tok_stride + h * D.
 * w: bf16 bits [D] or NULL (unit weight); use_norm selects RMSNorm.
 * pos: [T, 2] (row, col). out: fp64 [T, H, D] contiguous.
 *
 * Angles, for pair index m < D/2 (dim = D/2, table of D/4 frequencies):
 *   m <  D/4 : a_m = row * inv_freq[m]
 *   m >= D/4 : a_m = col * inv_freq[m - D/4]
 * Rotate-half with duplicated cos/sin (interleaved == 0):
 *   y[m]       = x[m] cos a_m - x[m + D/2] sin a_m
 *   y[m + D/2] = x[m + D/2] cos a_m + x[m] sin a_m
 * Interleaved pairs (interleaved != 0):
 *   y[2m]      = x[2m] cos a_m - x[2m + 1] sin a_m
 *   y[2m + 1]  = x[2m + 1] cos a_m + x[2m] sin a_m
 */
void vo_norm_rope(const uint16_t *x, int64_t T, int H, int D, int64_t tok_stride,
                  const int32_t *pos, double theta, const uint16_t *w, int use_norm,
                  double eps, int interleaved, double *out)
{
    const int half = D / 2, quarter = D / 4;
    double *inv_freq = (double *)malloc(sizeof(double) * (size_t)(quarter > 0 ? quarter : 1));
    vo_rope_inv_freq(half, theta, inv_freq);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double xh[512];
        double ang[256];
        for (int m = 0; m < half; ++m)
            ang[m] = (m < quarter) ? pos[2 * t] * inv_freq[m] : pos[2 * t + 1] * inv_freq[m - quarter];
        for (int h = 0; h < H; ++h) {
            const uint16_t *row = x + t * tok_stride + (int64_t)h * D;
            for (int d = 0; d < D; ++d)
                xh[d] = bf16_to_f64(row[d]);
            if (use_norm) {
                double ss = 0.0;
                for (int d = 0; d < D; ++d)
                    ss += xh[d] * xh[d];
                double inv_rms = 1.0 / sqrt(ss / D + eps);
                for (int d = 0; d < D; ++d)
                    xh[d] = xh[d] * inv_rms * (w ? bf16_to_f64(w[d]) : 1.0);
            }
            double *o = out + (t * H + h) * (int64_t)D;
            for (int m = 0; m < half; ++m) {
                double c = cos(ang[m]), s = sin(ang[m]);
                int i0 = interleaved ? 2 * m : m;           /* the two elements of pair m */
                int i1 = interleaved ? 2 * m + 1 : m + half;
                o[i0] = xh[i0] * c - xh[i1] * s;
                o[i1] = xh[i1] * c + xh[i0] * s;
            }
        }
    }
    free(inv_freq);
}

/*
 * q, k, v: fp64 [T, H, D] contiguous. cu: [B + 1] segment offsets.
 * rows: optional list of n_rows query tokens to evaluate (NULL = all T).
 * out: fp64 [n_rows or T, H, D]; row r of out belongs to rows[r] (or token r).
 * lse: fp64 [n_rows or T, H] or NULL: log(sum_j exp(scale * <q, k_j>)) over
 * the row's segment, natural log.
 * A token outside [cu[0], cu[B]) gets NaN (the packing does not cover it).
 */
void vo_attention(const double *q, const double *k, const double *v, int64_t T, int H, int D,
                  const int32_t *cu, int B, double scale, const int64_t *rows, int64_t n_rows,
                  double *out, double *lse)
{
    int64_t n = rows ? n_rows : T;
#pragma omp parallel
    {
        int64_t maxlen = 0;
        for (int i = 0; i < B; ++i)
            if (cu[i + 1] - cu[i] > maxlen)
                maxlen = cu[i + 1] - cu[i];
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < n * H; ++u) {
            int64_t r = u / H;
            int h = (int)(u % H);
            int64_t t = rows ? rows[r] : r;
            double *o = out + (r * H + h) * (int64_t)D;
            int seg = -1;
            for (int i = 0; i < B; ++i)
                if (t >= cu[i] && t < cu[i + 1]) {
                    seg = i;
                    break;
                }
            if (seg < 0) {
                for (int d = 0; d < D; ++d)
                    o[d] = NAN;
                if (lse)
                    lse[r * H + h] = NAN;
                continue;
            }
            int64_t lo = cu[seg], len = cu[seg + 1] - cu[seg];
            const double *qr = q + (t * H + h) * (int64_t)D;
            double mx = -INFINITY;
            for (int64_t j = 0; j < len; ++j) {
                const double *kr = k + ((lo + j) * H + h) * (int64_t)D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += qr[d] * kr[d];
                s[j] = scale * acc;
                if (s[j] > mx)
                    mx = s[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < len; ++j) {
                s[j] = exp(s[j] - mx);
                sum += s[j];
            }
            if (lse)
                lse[r * H + h] = mx + log(sum);
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t j = 0; j < len; ++j) {
                const double *vr = v + ((lo + j) * H + h) * (int64_t)D;
                double p = s[j] / sum;
                for (int d = 0; d < D; ++d)
                    o[d] += p * vr[d];
            }
        }
        free(s);
    }
}
