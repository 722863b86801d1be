// QK-RMSNorm + 2D RoPE arithmetic on 8-element chunks of one head row, shared by
// the prologue kernel and the attention kernels that normalise and rotate Q
// while loading it, so both produce the same bits.
//
// vLLM Dots vision_attention page, _RMSNorm.forward/_norm: sum of squares in
// fp32, x * rsqrt(mean + eps) cast back to bf16, then times the bf16 weight
// (rounded to bf16). tokenspeed mm_encoder_attention.py: rotate-half pairs
// (m, m + D/2) with cos/sin duplicated over both halves, or adjacent pairs
// (2m, 2m + 1) in the "complex_rope" mode; the rotation runs in fp32 and rounds
// once to bf16.
//
// A head row of D elements is seen as chunk pairs: chunk c (< D/16) holds
// elements [8c, 8c + 8) (xa) and [D/2 + 8c, D/2 + 8c + 8) (xb). The sum of
// squares is folded per chunk pair in a fixed order and the (at most 8)
// partial sums are combined as a fixed tree, which is what an 8-lane xor
// shuffle reduction produces, so a one-thread-per-row caller and an
// 8-lanes-per-row caller agree to the bit.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "vit_attn.h"

namespace vit {
namespace rope {

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---- packed pairs: f32x2 arithmetic
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t v;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(v) : "f"(lo), "f"(hi));
    return v;
}
__device__ __forceinline__ void f2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// sum of squares of one chunk pair, in the fixed order every caller uses
__device__ __forceinline__ float chunk_sumsq(const float *xa, const float *xb) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(xa[i], xa[i], fmaf(xb[i], xb[i], ss));
    return ss;
}

// the tree an xor-shuffle reduction over 8 lanes computes (offsets 1, 2, 4)
__device__ __forceinline__ float combine8(const float *s) {
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

__device__ __forceinline__ float inv_rms(float ss, int D, float eps) {
    return rsqrtf(ss / (float)D + eps);
}

// bf16(bf16(x0*inv) * w0), bf16(bf16(x1*inv) * w1) as two floats: the product of two bf16
// values is exact in fp32, so one bf16x2 multiply rounds exactly like the scalar form
__device__ __forceinline__ void norm_pair(float &x0, float &x1, float inv, uint32_t w2) {
    const uint32_t t = pack2(x0 * inv, x1 * inv);
    __nv_bfloat162 y = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&t),
                               *reinterpret_cast<const __nv_bfloat162 *>(&w2));
    const uint32_t u = *reinterpret_cast<uint32_t *>(&y);
    x0 = __uint_as_float(u << 16);
    x1 = __uint_as_float(u & 0xffff0000u);
}

// normalise 8 elements with their 8 bf16 weights (4 bf16x2 words)
__device__ __forceinline__ void norm8(float *x, float inv, const uint4 &w) {
    const uint32_t w_[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 8; i += 2) norm_pair(x[i], x[i + 1], inv, w_[i / 2]);
}

// Rotate-half: pair m = 8c + i of chunk c rotates xa[i] with xb[i]. cs[i/2] =
// {cos a_m, cos a_m+1, sin a_m, sin a_m+1} for i = 0, 2, 4, 6.
__device__ __forceinline__ void rotate_half8(const float *xa, const float *xb, const float4 *cs, uint4 &oa,
                                             uint4 &ob) {
    uint32_t a_[4], b_[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float4 t = cs[i / 2];
        const uint64_t cc = f2(t.x, t.y), sn = f2(t.z, t.w);
        const uint64_t a = f2(xa[i], xa[i + 1]), b = f2(xb[i], xb[i + 1]);
        float ya0, ya1, yb0, yb1;
        f2_split(f2_sub(f2_mul(a, cc), f2_mul(b, sn)), ya0, ya1);     // x cos - x' sin
        f2_split(f2_fma(a, sn, f2_mul(b, cc)), yb0, yb1);             // x' cos + x sin
        a_[i / 2] = pack2(ya0, ya1);
        b_[i / 2] = pack2(yb0, yb1);
    }
    oa = make_uint4(a_[0], a_[1], a_[2], a_[3]);
    ob = make_uint4(b_[0], b_[1], b_[2], b_[3]);
}

// Interleaved: the 8 elements hold pairs (x[2p], x[2p+1]), p = 0..3, with angles
// {cos, cos', sin, sin'} of pairs (0, 1) in cs[0] and (2, 3) in cs[1].
__device__ __forceinline__ uint4 interleaved8(const float *x, const float4 *cs) {
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float4 t = cs[p >> 1];
        const float c = (p & 1) ? t.y : t.x, s = (p & 1) ? t.w : t.z;
        float y0, y1;
        // (x0 cos - x1 sin, x1 cos + x0 sin) = (x0, x1) * cos + (x1, x0) * (-sin, sin)
        f2_split(f2_fma(f2(x[2 * p + 1], x[2 * p]), f2(-s, s), f2_mul(f2(x[2 * p], x[2 * p + 1]), f2(c, c))), y0, y1);
        o[p] = pack2(y0, y1);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Parameters of the Q normalisation + rotation that an attention kernel applies while
// loading Q (all device pointers; the table is the one vit_rope_table writes).
struct QRope {
    const int2 *pos_hw;        // [T] (row, col)
    const float4 *cos_sin;     // [max_pos][D/8] float4 {cos a_f, cos a_f+1, sin a_f, sin a_f+1}, f even
    const uint4 *norm_w;       // bf16 [D] q weight, or NULL for no norm
    int max_pos;
    float eps;
    int interleaved;
    int32_t *status;
};

// Normalise and rotate one head row of D bf16 values in place, reading and writing its
// chunks through `chunk(q)` (q = 0 .. D/8 - 1: a pointer to elements [8q, 8q + 8)).
// Positions outside the table are reported and clamped, so nothing is read out of range.
template <int D, typename ChunkPtr>
__device__ __forceinline__ void transform_row(const QRope &qr, int64_t token, ChunkPtr chunk) {
    constexpr int CH = D / 16;                 // chunk pairs
    constexpr int QUART = D / 4;
    int2 p = qr.pos_hw[token];
    if (p.x < 0 || p.y < 0 || p.x >= qr.max_pos || p.y >= qr.max_pos) {
        if (qr.status) atomicCAS(qr.status, 0, VIT_ERR_POSITION_RANGE);
        p.x = min(max(p.x, 0), qr.max_pos - 1);
        p.y = min(max(p.y, 0), qr.max_pos - 1);
    }
    const float4 *row_cs = qr.cos_sin + (int64_t)p.x * (QUART / 2);
    const float4 *col_cs = qr.cos_sin + (int64_t)p.y * (QUART / 2);
    float inv = 1.f;
    if (qr.norm_w) {
        float s[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) s[c] = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float xa[8], xb[8];
            unpack8(*chunk(c), xa);
            unpack8(*chunk(c + CH), xb);
            s[c] = chunk_sumsq(xa, xb);
        }
        inv = inv_rms(combine8(s), D, qr.eps);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        float xa[8], xb[8];
        uint4 *pa = chunk(c), *pb = chunk(c + CH);
        unpack8(*pa, xa);
        unpack8(*pb, xb);
        if (qr.norm_w) {
            norm8(xa, inv, qr.norm_w[c]);
            norm8(xb, inv, qr.norm_w[c + CH]);
        }
        uint4 oa, ob;
        if (!qr.interleaved) {
            float4 cs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * c + 2 * i;       // even; m and m + 1 share row/column
                cs[i] = m < QUART ? row_cs[m / 2] : col_cs[(m - QUART) / 2];
            }
            rotate_half8(xa, xb, cs, oa, ob);
        } else {
            // chunk c of the first half: pairs 4c .. 4c+3 (row angles); chunk c of the second
            // half: pairs D/4 + 4c .. (column angles, table entries 4c ..)
            const float4 ca[2] = {row_cs[2 * c], row_cs[2 * c + 1]};
            const float4 cb[2] = {col_cs[2 * c], col_cs[2 * c + 1]};
            oa = interleaved8(xa, ca);
            ob = interleaved8(xb, cb);
        }
        *pa = oa;
        *pb = ob;
    }
}

}  // namespace rope
}  // namespace vit
