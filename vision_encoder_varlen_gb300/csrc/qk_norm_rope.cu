// Fused QK-RMSNorm + 2D rotate-half RoPE prologue: one read and one write of q and k.
//
// vLLM Dots vision_attention page, _RMSNorm.forward/_norm: the norm is reduced
// in fp32 over head_dim, the normalised value is cast back to the input dtype
// (bf16) and then multiplied by the weight (bf16 x bf16 -> bf16); q and k each
// have their own weight (_VisionAttentionBase). _qkv_with_rope applies the norm
// before RoPE. tokenspeed mm_encoder_attention.py, MultimodalEncoderAttention.
// forward: a half-width cos/sin table is duplicated over both halves of the
// head (rotate-half / NeoX pairing of element m with m + D/2).
//
// Layout of the work: a block takes 8 tokens at a time, builds their D/2
// cos/sin values once in shared memory (shared by all heads and by q and k),
// then 8-lane groups each own (token, head, q-or-k) rows; lane c holds the
// 16-byte chunk c of the first half and the matching chunk of the second half,
// so every rotation pair lives in one thread and the RMS reduction is a
// three-step shuffle inside the group. Each group issues the loads of four rows
// before it computes on any of them, to keep enough bytes in flight.
// HBM-bound: 8*T*H*D bytes move in total.
#include "internal.h"

namespace vit {
namespace {

constexpr int kThreads = 256;
constexpr int kTokensPerIter = 8;
constexpr int kRowBatch = 4;                           // rows per group whose loads are in flight together
constexpr int kGroup = 8;                              // lanes per row
constexpr int kGroupsPerBlock = kThreads / kGroup;     // 32

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

__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

template <int D>
__global__ void __launch_bounds__(kThreads)
qk_norm_rope_kernel(const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out,
                    const __nv_bfloat16 *k_in, __nv_bfloat16 *k_out, int64_t T, int H,
                    int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride, int64_t k_out_stride,
                    const int2 *__restrict__ pos_hw, const float *__restrict__ inv_freq,
                    const __nv_bfloat16 *__restrict__ norm_w, float eps)
{
    constexpr int HALF = D / 2, QUART = D / 4, CHUNKS = HALF / 8;
    static_assert(HALF % 8 == 0 && CHUNKS <= kGroup, "head_dim must split into 16-byte chunks");
    __shared__ float s_cos[kTokensPerIter][HALF];
    __shared__ float s_sin[kTokensPerIter][HALF];
    __shared__ float s_w[2][D];

    const int tid = threadIdx.x;
    const int grp = tid / kGroup, c = tid % kGroup;
    const bool use_norm = norm_w != nullptr;
    if (use_norm)
        for (int i = tid; i < 2 * D; i += kThreads) s_w[i / D][i % D] = __bfloat162float(norm_w[i]);

    const int rows_per_tok = 2 * H;
    for (int64_t t0 = (int64_t)blockIdx.x * kTokensPerIter; t0 < T; t0 += (int64_t)gridDim.x * kTokensPerIter) {
        __syncthreads();                                // previous iteration done with s_cos/s_sin
        const int ntok = (int)(T - t0 < kTokensPerIter ? T - t0 : kTokensPerIter);
        for (int i = tid; i < ntok * HALF; i += kThreads) {
            const int tt = i / HALF, m = i % HALF;
            const int2 p = pos_hw[t0 + tt];
            const float ang = (float)(m < QUART ? p.x : p.y) * inv_freq[m < QUART ? m : m - QUART];
            float sn, cs;
            sincosf(ang, &sn, &cs);
            s_cos[tt][m] = cs;
            s_sin[tt][m] = sn;
        }
        __syncthreads();

        const int nrows = ntok * rows_per_tok;
        constexpr int STEP = kGroupsPerBlock * kRowBatch;
        const int nrows_pad = (nrows + STEP - 1) / STEP * STEP;
        for (int r0 = 0; r0 < nrows_pad; r0 += STEP) {            // same trip count for every group
            uint4 va[kRowBatch], vb[kRowBatch];
            __nv_bfloat16 *dst[kRowBatch];
            int tt_[kRowBatch], which_[kRowBatch];
            bool act[kRowBatch];
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                const int r = r0 + k * kGroupsPerBlock + grp;
                const bool row_ok = r < nrows;
                const int tt = row_ok ? r / rows_per_tok : 0;
                const int rem = row_ok ? r % rows_per_tok : 0;
                const int which = rem >= H;             // 0 = q, 1 = k
                const int h = rem - which * H;
                const int64_t t = t0 + tt;
                act[k] = row_ok && c < CHUNKS;
                tt_[k] = tt;
                which_[k] = which;
                const __nv_bfloat16 *src = (which ? k_in + t * k_in_stride : q_in + t * q_in_stride) + (int64_t)h * D + c * 8;
                dst[k] = (which ? k_out + t * k_out_stride : q_out + t * q_out_stride) + (int64_t)h * D + c * 8;
                if (act[k]) {
                    va[k] = *reinterpret_cast<const uint4 *>(src);
                    vb[k] = *reinterpret_cast<const uint4 *>(src + HALF);
                } else {
                    va[k] = vb[k] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                float xa[8], xb[8];
                unpack8(va[k], xa);
                unpack8(vb[k], xb);
                if (use_norm) {
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) ss = fmaf(xa[i], xa[i], fmaf(xb[i], xb[i], ss));
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    const float inv = rsqrtf(ss / (float)D + eps);
                    const float *w = s_w[which_[k]];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int m = c * 8 + i;
                        if (act[k]) {
                            xa[i] = round_bf16(round_bf16(xa[i] * inv) * w[m]);
                            xb[i] = round_bf16(round_bf16(xb[i] * inv) * w[m + HALF]);
                        }
                    }
                }
                if (act[k]) {
                    const float *cs_ = s_cos[tt_[k]], *sn_ = s_sin[tt_[k]];
                    uint32_t oa[4], ob[4];
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const int m = c * 8 + i;
                        const float c0 = cs_[m], s0 = sn_[m];
                        const float c1 = cs_[m + 1], s1 = sn_[m + 1];
                        oa[i / 2] = pack2(xa[i] * c0 - xb[i] * s0, xa[i + 1] * c1 - xb[i + 1] * s1);
                        ob[i / 2] = pack2(xb[i] * c0 + xa[i] * s0, xb[i + 1] * c1 + xa[i + 1] * s1);
                    }
                    *reinterpret_cast<uint4 *>(dst[k]) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
                    *reinterpret_cast<uint4 *>(dst[k] + HALF) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                }
            }
        }
    }
}

template <int D>
cudaError_t launch_d(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T, int H,
                     int64_t qis, int64_t qos, int64_t kis, int64_t kos, const int32_t *pos_hw,
                     const float *inv_freq, const void *norm_w, float eps, int num_sms, cudaStream_t stream)
{
    const int64_t want = (T + kTokensPerIter - 1) / kTokensPerIter;
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("qk_norm_rope", stream);
    qk_norm_rope_kernel<D><<<blocks, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q_in), static_cast<__nv_bfloat16 *>(q_out),
        static_cast<const __nv_bfloat16 *>(k_in), static_cast<__nv_bfloat16 *>(k_out), T, H, qis, qos, kis, kos,
        reinterpret_cast<const int2 *>(pos_hw), inv_freq, static_cast<const __nv_bfloat16 *>(norm_w), eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T,
                                int H, int D, int64_t q_in_stride, int64_t q_out_stride,
                                int64_t k_in_stride, int64_t k_out_stride, const int32_t *pos_hw,
                                const float *inv_freq, const void *norm_w, float eps, int num_sms,
                                cudaStream_t stream)
{
#define VIT_QKNR(DD)                                                                                   \
    case DD:                                                                                           \
        return launch_d<DD>(q_in, q_out, k_in, k_out, T, H, q_in_stride, q_out_stride, k_in_stride,   \
                            k_out_stride, pos_hw, inv_freq, norm_w, eps, num_sms, stream);
    switch (D) {
        VIT_QKNR(32)
        VIT_QKNR(64)
        VIT_QKNR(80)
        VIT_QKNR(96)
        VIT_QKNR(128)
        default: return cudaErrorInvalidValue;
    }
#undef VIT_QKNR
}

}  // namespace vit
