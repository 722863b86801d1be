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
// Two layouts of the work, both HBM-bound (8*T*H*D bytes move in total):
//   - head_dim <= 80: a block takes as many tokens at a time as give one
//     (token, head, q-or-k) row per thread; each thread issues the loads of its
//     whole row first, the block builds the tokens' D/2 cos/sin values in
//     shared memory (shared by all heads and by q and k) while those loads are
//     in flight, and the thread normalises and rotates its row in registers.
//   - head_dim 96 and 128 (and more than 128 heads): a block takes 8 tokens at
//     a time and 8-lane groups own rows, lane c holding the 16-byte chunk c of
//     the first half and the matching chunk of the second half, so every
//     rotation pair lives in one thread and the RMS reduction is a three-step
//     shuffle; each group has four rows' loads in flight. At head_dim 128 every
//     lane of a group is busy and a whole row per thread would not fit the
//     registers of two blocks per SM; at 80 three of the eight lanes would idle.
// Measured on GB300 (head_dim 80, 16 heads, 67792 tokens): 0.175 ms with one
// row per thread, 0.203 ms with 8-lane groups; at head_dim 128 the groups are
// faster (0.109 against 0.160 ms).
//
// The interleaved mode (tokenspeed mm_encoder_attention.py, the "complex_rope"
// position-embedding mode and packed_qkv_complex_rotary) pairs x[2m] with
// x[2m+1] and turns the pair by the same angle a_m; a lane then rotates pairs
// inside each of its two chunks. Either q or k may be left out (its pointers
// NULL), which turns the pass into a one-tensor pre-stage.
#include "internal.h"
#include "rope_math.cuh"

namespace vit {
namespace {

using namespace rope;

constexpr int kThreads = 256;
constexpr int kTokensPerIter = 8;
constexpr int kRowBatch = 4;                           // rows per group whose loads are in flight together
constexpr int kGroup = 8;                              // lanes per row
constexpr int kGroupsPerBlock = kThreads / kGroup;     // 32

template <int D, bool IL>
__global__ void __launch_bounds__(kThreads)
qk_norm_rope_kernel(const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out,
                    const __nv_bfloat16 *k_in, __nv_bfloat16 *k_out, int64_t T, int H,
                    int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride, int64_t k_out_stride,
                    const int2 *__restrict__ pos_hw, const float *__restrict__ inv_freq,
                    const __nv_bfloat16 *__restrict__ norm_w, float eps)
{
    constexpr int HALF = D / 2, QUART = D / 4, CHUNKS = HALF / 8;
    static_assert(HALF % 8 == 0 && CHUNKS <= kGroup, "head_dim must split into 16-byte chunks");
    // per token and pair (m, m+1): {cos a_m, cos a_m+1, sin a_m, sin a_m+1}, one 16-byte read
    __shared__ float4 s_cs[kTokensPerIter][HALF / 2];
    __shared__ __align__(16) uint32_t s_w[2][D / 2];      // bf16x2 weight pairs (q row, k row)

    const int tid = threadIdx.x;
    const int grp = tid / kGroup, c = tid % kGroup;
    const bool use_norm = norm_w != nullptr;
    if (use_norm)
        for (int i = tid; i < D; i += kThreads)
            s_w[i / (D / 2)][i % (D / 2)] = reinterpret_cast<const uint32_t *>(norm_w)[i];

    const int nq = q_in ? H : 0;                        // q rows per token (0 = q left out)
    const int rows_per_tok = nq + (k_in ? H : 0);
    for (int64_t t0 = (int64_t)blockIdx.x * kTokensPerIter; t0 < T; t0 += (int64_t)gridDim.x * kTokensPerIter) {
        __syncthreads();                                // previous iteration done with s_cos/s_sin
        const int ntok = (int)(T - t0 < kTokensPerIter ? T - t0 : kTokensPerIter);
        for (int i = tid; i < ntok * (HALF / 2); i += kThreads) {
            const int tt = i / (HALF / 2), m = 2 * (i % (HALF / 2));
            const int2 p = pos_hw[t0 + tt];
            // m is even and D/4 is even, so m and m + 1 are both row angles or both column angles
            const float pos = (float)(m < QUART ? p.x : p.y);
            const int f = m < QUART ? m : m - QUART;
            float s0, c0, s1, c1;
            sincosf(pos * inv_freq[f], &s0, &c0);
            sincosf(pos * inv_freq[f + 1], &s1, &c1);
            s_cs[tt][m / 2] = make_float4(c0, c1, s0, s1);
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
                const int which = rem >= nq;            // 0 = q, 1 = k
                const int h = rem - which * nq;
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
                    // per-lane chunk sums combined by the xor tree of combine8 (idle lanes add 0)
                    float ss = chunk_sumsq(xa, xb);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    const float inv = inv_rms(ss, D, eps);
                    if (act[k]) {                                // idle lanes (c >= CHUNKS) read nothing
                        norm8(xa, inv, *reinterpret_cast<const uint4 *>(&s_w[which_[k]][c * 4]));
                        norm8(xb, inv, *reinterpret_cast<const uint4 *>(&s_w[which_[k]][HALF / 2 + c * 4]));
                    }
                }
                if (act[k]) {
                    uint4 oa, ob;
                    if constexpr (!IL) {
                        rotate_half8(xa, xb, s_cs[tt_[k]] + c * 4, oa, ob);
                    } else {
                        // chunk c of the first half holds pairs 4c..4c+3, the second half's chunk c
                        // pairs D/4 + 4c .. D/4 + 4c + 3 (D/4 is even, so both start a float4 entry)
                        oa = interleaved8(xa, s_cs[tt_[k]] + 2 * c);
                        ob = interleaved8(xb, s_cs[tt_[k]] + D / 8 + 2 * c);
                    }
                    *reinterpret_cast<uint4 *>(dst[k]) = oa;
                    *reinterpret_cast<uint4 *>(dst[k] + HALF) = ob;
                }
            }
        }
    }
}

constexpr int kRowThreads = 256;

template <int D, bool IL>
__global__ void __launch_bounds__(kRowThreads, 2)
qk_norm_rope_row_kernel(const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out,
                        const __nv_bfloat16 *k_in, __nv_bfloat16 *k_out, int64_t T, int H,
                        int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride, int64_t k_out_stride,
                        const int2 *__restrict__ pos_hw, const float *__restrict__ inv_freq,
                        const __nv_bfloat16 *__restrict__ norm_w, float eps, int tpi)
{
    constexpr int HALF = D / 2, QUART = D / 4, CH = D / 16, NCH = D / 8;
    extern __shared__ float4 s_cs[];                      // [tpi][HALF / 2], as in the group kernel
    __shared__ uint4 s_w[2][NCH];                         // weight chunks (q row, k row)

    const int tid = threadIdx.x;
    const bool use_norm = norm_w != nullptr;
    if (use_norm)
        for (int i = tid; i < 2 * NCH; i += kRowThreads)
            s_w[i / NCH][i % NCH] = reinterpret_cast<const uint4 *>(norm_w)[i];

    const int nq = q_in ? H : 0;                          // q rows per token (0 = q left out)
    const int rpt = nq + (k_in ? H : 0);                  // rows per token; tpi * rpt <= kRowThreads
    for (int64_t t0 = (int64_t)blockIdx.x * tpi; t0 < T; t0 += (int64_t)gridDim.x * tpi) {
        const int ntok = (int)(T - t0 < tpi ? T - t0 : tpi);
        const bool act = tid < ntok * rpt;
        const int tt = act ? tid / rpt : 0, rem = act ? tid % rpt : 0;
        const int which = rem >= nq, h = rem - which * nq;
        const int64_t t = t0 + tt;
        // the row's loads go out before anything waits
        uint4 x[NCH];
        __nv_bfloat16 *dst = nullptr;
        if (act) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                (which ? k_in + t * k_in_stride : q_in + t * q_in_stride) + (int64_t)h * D);
            dst = (which ? k_out + t * k_out_stride : q_out + t * q_out_stride) + (int64_t)h * D;
#pragma unroll
            for (int c = 0; c < NCH; ++c) x[c] = src[c];
        }
        __syncthreads();                                  // the previous tokens' table is no longer read
        for (int i = tid; i < ntok * (HALF / 2); i += kRowThreads) {
            const int ti = i / (HALF / 2), m = 2 * (i % (HALF / 2));
            const int2 p = pos_hw[t0 + ti];
            // m is even and D/4 is even, so m and m + 1 are both row angles or both column angles
            const float pos = (float)(m < QUART ? p.x : p.y);
            const int f = m < QUART ? m : m - QUART;
            float s0, c0, s1, c1;
            sincosf(pos * inv_freq[f], &s0, &c0);
            sincosf(pos * inv_freq[f + 1], &s1, &c1);
            s_cs[ti * (HALF / 2) + m / 2] = make_float4(c0, c1, s0, s1);
        }
        __syncthreads();
        if (!act) continue;
        float inv = 1.f;
        if (use_norm) {
            float ss[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) ss[c] = 0.f;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                float xa[8], xb[8];
                unpack8(x[c], xa);
                unpack8(x[c + CH], xb);
                ss[c] = chunk_sumsq(xa, xb);
            }
            inv = inv_rms(combine8(ss), D, eps);
        }
        const float4 *cs = s_cs + tt * (HALF / 2);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float xa[8], xb[8];
            unpack8(x[c], xa);
            unpack8(x[c + CH], xb);
            if (use_norm) {
                norm8(xa, inv, s_w[which][c]);
                norm8(xb, inv, s_w[which][c + CH]);
            }
            uint4 oa, ob;
            if constexpr (!IL) {
                rotate_half8(xa, xb, cs + c * 4, oa, ob);
            } else {
                oa = interleaved8(xa, cs + 2 * c);
                ob = interleaved8(xb, cs + D / 8 + 2 * c);
            }
            reinterpret_cast<uint4 *>(dst)[c] = oa;
            reinterpret_cast<uint4 *>(dst)[c + CH] = ob;
        }
    }
}

template <int D>
cudaError_t launch_d(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T, int H,
                     int64_t qis, int64_t qos, int64_t kis, int64_t kos, const int32_t *pos_hw,
                     const float *inv_freq, const void *norm_w, float eps, bool interleaved, int num_sms,
                     cudaStream_t stream)
{
    const int rpt = (q_in ? H : 0) + (k_in ? H : 0);
    if (D <= 80 && rpt <= kRowThreads) {
        // one row per thread: as many tokens per block iteration as fill the block
        const int tpi = kRowThreads / rpt;
        const size_t smem = sizeof(float4) * (size_t)tpi * (D / 4);
        auto kern = interleaved ? qk_norm_rope_row_kernel<D, true> : qk_norm_rope_row_kernel<D, false>;
        static DeviceOnce once[2];
        cudaError_t e = once[interleaved ? 1 : 0].run([&] {
            // the largest table: 256 tokens (one row each)
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(sizeof(float4) * kRowThreads * (D / 4)));
        });
        if (e != cudaSuccess) return e;
        const int64_t want = (T + tpi - 1) / tpi;
        const int64_t cap = (int64_t)num_sms * 2;
        const unsigned blocks = (unsigned)(want < cap ? want : cap);
        if (blocks == 0) return cudaSuccess;
        LaunchScope scope("qk_norm_rope", stream);
        kern<<<blocks, kRowThreads, smem, stream>>>(
            static_cast<const __nv_bfloat16 *>(q_in), static_cast<__nv_bfloat16 *>(q_out),
            static_cast<const __nv_bfloat16 *>(k_in), static_cast<__nv_bfloat16 *>(k_out), T, H, qis, qos, kis, kos,
            reinterpret_cast<const int2 *>(pos_hw), inv_freq, static_cast<const __nv_bfloat16 *>(norm_w), eps, tpi);
        return cudaGetLastError();
    }
    const int64_t want = (T + kTokensPerIter - 1) / kTokensPerIter;
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("qk_norm_rope", stream);
    auto kern = interleaved ? qk_norm_rope_kernel<D, true> : qk_norm_rope_kernel<D, false>;
    kern<<<blocks, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q_in), static_cast<__nv_bfloat16 *>(q_out),
        static_cast<const __nv_bfloat16 *>(k_in), static_cast<__nv_bfloat16 *>(k_out), T, H, qis, qos, kis, kos,
        reinterpret_cast<const int2 *>(pos_hw), inv_freq, static_cast<const __nv_bfloat16 *>(norm_w), eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T,
                                int H, int D, int64_t q_in_stride, int64_t q_out_stride,
                                int64_t k_in_stride, int64_t k_out_stride, const int32_t *pos_hw,
                                const float *inv_freq, const void *norm_w, float eps, bool interleaved,
                                int num_sms, cudaStream_t stream)
{
#define VIT_QKNR(DD)                                                                                   \
    case DD:                                                                                           \
        return launch_d<DD>(q_in, q_out, k_in, k_out, T, H, q_in_stride, q_out_stride, k_in_stride,   \
                            k_out_stride, pos_hw, inv_freq, norm_w, eps, interleaved, num_sms, stream);
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
