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
//   - staged (head_dim <= 80, when one token's rows fit one iteration): a block
//     takes up to 256 rows' worth of tokens at a time, warp 0 copies their q
//     and k rows into one of two shared-memory
//     buffers with bulk asynchronous copies (whole contiguous token rows) while
//     the block computes on the other buffer, builds the tokens' D/2 cos/sin
//     values meanwhile, every thread normalises and rotates one row in place,
//     and warp 0 copies the buffer back out with bulk stores;
//   - grouped (head_dim 96 and 128, or more than 128 heads): a block takes 8
//     tokens at a time and 8-lane groups own rows,
//     lane c holding the 16-byte chunk c of the first half and the matching
//     chunk of the second half, so every rotation pair lives in one thread and
//     the RMS reduction is a three-step shuffle; each group keeps four rows'
//     loads in flight.
// Both compute each row with the same functions in the same order, so they
// agree bit for bit. Measured on GB300 (16 heads, 67792 tokens, head_dim 80):
// staged 0.125 ms (5.55 TB/s), one row per thread straight from HBM 0.175 ms,
// 8-lane groups 0.203 ms; at head_dim 128 (31934 tokens) the groups take 0.110
// ms, where a staged layout of 128 rows per iteration took 0.205 ms.
//
// The interleaved mode (tokenspeed mm_encoder_attention.py, the "complex_rope"
// position-embedding mode and packed_qkv_complex_rotary) pairs x[2m] with
// x[2m+1] and turns the pair by the same angle a_m; a lane then rotates pairs
// inside each of its two chunks. Either q or k may be left out (its pointers
// NULL), which turns the pass into a one-tensor pre-stage.
#include "internal.h"
#include "rope_math.cuh"
#include "sm100.cuh"

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
                const __nv_bfloat16 *src =
                    (which ? k_in + t * k_in_stride : q_in + t * q_in_stride) + (int64_t)h * D + c * 8;
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

// ---------------------------------------------------------------- staged layout
//
// Each iteration takes up to kStageTok tokens (at most NT rows, one per thread). Warp 0
// copies their q rows (H * D contiguous values per token) and k rows into one of two
// shared-memory buffers with bulk asynchronous copies, one per token and tensor, while the
// block works on the other buffer; every thread rotates its row in place in shared memory;
// warp 0 copies the buffer back out with bulk stores. HBM sees only whole contiguous token
// rows, and nothing in flight occupies registers.
constexpr int kStageTok = 64;
constexpr long long kStageWait = 2000000000ll;        // clock cycles before a copy wait gives up

// rows (= threads) per iteration: two blocks of two row buffers each per SM at head_dim <= 80
template <int D> __host__ __device__ constexpr int stage_rows() { return 256; }

template <int D>
__host__ __device__ constexpr size_t staged_smem_bytes() {
    return 2 * (size_t)stage_rows<D>() * D * 2 + sizeof(float4) * kStageTok * (D / 4);
}

template <int D, bool IL>
__global__ void __launch_bounds__(stage_rows<D>(), 2)
qk_norm_rope_staged_kernel(const __nv_bfloat16 *q_in, __nv_bfloat16 *q_out,
                           const __nv_bfloat16 *k_in, __nv_bfloat16 *k_out, int64_t T, int H,
                           int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride, int64_t k_out_stride,
                           const int2 *__restrict__ pos_hw, const float *__restrict__ inv_freq,
                           const __nv_bfloat16 *__restrict__ norm_w, float eps, int tpi, int32_t *status)
{
    using namespace sm100;
    constexpr int NT = stage_rows<D>();
    constexpr int HALF = D / 2, QUART = D / 4, CH = D / 16, NCH = D / 8, ROW = 2 * D;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *bufs = smem;                                         // [2][NT][ROW]
    float4 *s_cs = reinterpret_cast<float4 *>(smem + 2 * NT * ROW);   // [tpi][HALF / 2]
    __shared__ uint4 s_w[2][NCH];
    __shared__ __align__(8) uint64_t s_full[2];
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool use_norm = norm_w != nullptr;
    const int nq = q_in ? H : 0, nk = k_in ? H : 0, rpt = nq + nk;
    const uint32_t half_bytes = (uint32_t)H * ROW;                      // one token's q (or k) rows
    const int64_t n_it = (T + tpi - 1) / tpi;
    if (tid == 0) {
        mbar_init(smem_addr(&s_full[0]), 1);
        mbar_init(smem_addr(&s_full[1]), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (use_norm)
        for (int i = tid; i < 2 * NCH; i += NT) s_w[i / NCH][i % NCH] = reinterpret_cast<const uint4 *>(norm_w)[i];
    __syncthreads();

    // warp 0: bulk copies of the q and k rows of tokens [t0, t0 + ntok) into buffer b
    auto issue_loads = [&](int64_t t0, int ntok, int b) {
        unsigned char *buf = bufs + (size_t)b * NT * ROW;
        if (lane == 0) mbar_arrive_expect_tx(smem_addr(&s_full[b]), (uint32_t)ntok * rpt * ROW);
        __syncwarp();
        const int halves = (nq ? 1 : 0) + (nk ? 1 : 0);
        for (int l = lane; l < ntok * halves; l += 32) {
            const int tt = l / halves, which = (halves == 2) ? (l & 1) : (nq ? 0 : 1);
            const int64_t t = t0 + tt;
            const void *src = which ? (const void *)(k_in + t * k_in_stride) : (const void *)(q_in + t * q_in_stride);
            const int row0 = tt * rpt + (which ? nq : 0);
            bulk_load(smem_addr(buf + (size_t)row0 * ROW), src, half_bytes, smem_addr(&s_full[b]));
        }
    };
    auto issue_stores = [&](int64_t t0, int ntok, int b) {
        const unsigned char *buf = bufs + (size_t)b * NT * ROW;
        const int halves = (nq ? 1 : 0) + (nk ? 1 : 0);
        for (int l = lane; l < ntok * halves; l += 32) {
            const int tt = l / halves, which = (halves == 2) ? (l & 1) : (nq ? 0 : 1);
            const int64_t t = t0 + tt;
            void *dst = which ? (void *)(k_out + t * k_out_stride) : (void *)(q_out + t * q_out_stride);
            const int row0 = tt * rpt + (which ? nq : 0);
            bulk_store(dst, smem_addr(buf + (size_t)row0 * ROW), half_bytes);
        }
        bulk_commit();
    };

    int64_t it = blockIdx.x;
    if (warp == 0 && it < n_it) issue_loads(it * tpi, (int)min((int64_t)tpi, T - it * tpi), 0);
    int n = 0;
    for (; it < n_it; it += gridDim.x, ++n) {
        const int b = n & 1;
        const int64_t t0 = it * tpi;
        const int ntok = (int)min((int64_t)tpi, T - t0);
        const int64_t nx = it + gridDim.x;
        if (warp == 0 && nx < n_it) {
            bulk_wait_read_all();          // buffer b ^ 1's stores (last iteration) have read it
            __syncwarp();
            issue_loads(nx * tpi, (int)min((int64_t)tpi, T - nx * tpi), b ^ 1);
        }
        // this iteration's cos/sin while its rows are on the way
        for (int i = tid; i < ntok * (HALF / 2); i += NT) {
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
        if (!mbar_wait(smem_addr(&s_full[b]), (n >> 1) & 1, (const volatile int *)&s_abort, kStageWait))
            s_abort = 1;
        __syncthreads();                   // table ready, rows landed (or the wait gave up)
        if (s_abort) {
            // let the copies already issued land before this block's shared memory is released
            if (tid == 0) {
                const int never = 0;
                report_error(status, VIT_ERR_TIMEOUT);
                mbar_wait(smem_addr(&s_full[b]), (n >> 1) & 1, &never, 20000000ll);
                if (nx < n_it) mbar_wait(smem_addr(&s_full[b ^ 1]), ((n + 1) >> 1) & 1, &never, 20000000ll);
            }
            break;
        }
        const int r = tid;
        if (r < ntok * rpt) {
            const int rem = r % rpt, which = rem >= nq;
            uint4 *row = reinterpret_cast<uint4 *>(bufs + ((size_t)b * NT + r) * ROW);
            float inv = 1.f;
            if (use_norm) {
                float ss[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) ss[c] = 0.f;
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    float xa[8], xb[8];
                    unpack8(row[c], xa);
                    unpack8(row[c + CH], xb);
                    ss[c] = chunk_sumsq(xa, xb);
                }
                inv = inv_rms(combine8(ss), D, eps);
            }
            const float4 *cs = s_cs + (r / rpt) * (HALF / 2);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                float xa[8], xb[8];
                unpack8(row[c], xa);
                unpack8(row[c + CH], xb);
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
                row[c] = oa;
                row[c + CH] = ob;
            }
        }
        fence_proxy_async_smem();          // the rows are read next by the bulk stores
        __syncthreads();                   // every row done; the table may be rebuilt
        if (warp == 0) issue_stores(t0, ntok, b);
    }
    if (warp == 0) bulk_wait_all();        // the stores have completed
}

template <int D>
cudaError_t launch_d(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T, int H,
                     int64_t qis, int64_t qos, int64_t kis, int64_t kos, const int32_t *pos_hw,
                     const float *inv_freq, const void *norm_w, float eps, bool interleaved, int num_sms,
                     int32_t *status, cudaStream_t stream)
{
    const int rpt = (q_in ? H : 0) + (k_in ? H : 0);
    constexpr int NT = stage_rows<D>();
    if (D <= 80 && rpt <= NT) {
        // staged: bulk copies through shared memory, one row per thread
        const int tpi = NT / rpt < kStageTok ? NT / rpt : kStageTok;
        constexpr size_t smem = staged_smem_bytes<D>();
        auto kern = interleaved ? qk_norm_rope_staged_kernel<D, true> : qk_norm_rope_staged_kernel<D, false>;
        static DeviceOnce once[2];
        cudaError_t e = once[interleaved ? 1 : 0].run(
            [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); });
        if (e != cudaSuccess) return e;
        const int64_t want = (T + tpi - 1) / tpi;
        const int64_t cap = (int64_t)num_sms * 2;
        const unsigned blocks = (unsigned)(want < cap ? want : cap);
        if (blocks == 0) return cudaSuccess;
        LaunchScope scope("qk_norm_rope", stream);
        kern<<<blocks, NT, smem, stream>>>(
            static_cast<const __nv_bfloat16 *>(q_in), static_cast<__nv_bfloat16 *>(q_out),
            static_cast<const __nv_bfloat16 *>(k_in), static_cast<__nv_bfloat16 *>(k_out), T, H, qis, qos, kis, kos,
            reinterpret_cast<const int2 *>(pos_hw), inv_freq, static_cast<const __nv_bfloat16 *>(norm_w), eps, tpi,
            status);
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
                                int num_sms, int32_t *status, cudaStream_t stream)
{
#define VIT_QKNR(DD)                                                                                   \
    case DD:                                                                                           \
        return launch_d<DD>(q_in, q_out, k_in, k_out, T, H, q_in_stride, q_out_stride, k_in_stride,   \
                            k_out_stride, pos_hw, inv_freq, norm_w, eps, interleaved, num_sms, status, stream);
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
