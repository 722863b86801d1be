// 2D vision RoPE frequency table, patch positions and segment offsets.
//
// vLLM Dots vision_attention page, VisionRotaryEmbedding: inv_freq[j] =
// 1 / theta^(2j/dim) (fp32), positions 0..seqlen-1 multiplied by it. For 2D
// RoPE one table of dim = head_dim/2 serves the row and the column position
// of each patch; tokens of an image are packed row-major and every image
// restarts at position (0, 0). The segment offsets are the cu_seqlens of
// VisionAttention.forward.
//
// One kernel: every block scans the (small) grid list in shared memory, so no
// cross-block pass or scratch buffer is needed; block 0 also writes the
// frequency table and the offsets.
#include "internal.h"

namespace vit {
namespace {

constexpr int kThreads = 256;
constexpr int kTokensPerBlock = 2048;

__global__ void __launch_bounds__(kThreads)
rope_freqs_kernel(int dim, float theta, const int32_t *__restrict__ grid_hw, int n_img, int64_t T,
                  float *__restrict__ inv_freq, int2 *__restrict__ pos_hw, int32_t *__restrict__ cu_out,
                  int32_t *status)
{
    extern __shared__ int64_t s_cu[];          // [n_img + 1] inclusive-prefix offsets
    __shared__ int64_t s_part[kThreads];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // each thread sums a contiguous chunk of images, then a block scan of the partials
    const int per = (n_img + kThreads - 1) / kThreads;
    const int lo = min(tid * per, n_img), hi = min(lo + per, n_img);
    int64_t local = 0;
    for (int i = lo; i < hi; ++i) {
        const int h = grid_hw[2 * i], w = grid_hw[2 * i + 1];
        if (h < 0 || w < 0) s_bad = 1;
        local += (int64_t)max(h, 0) * max(w, 0);
    }
    s_part[tid] = local;
    __syncthreads();
    for (int off = 1; off < kThreads; off <<= 1) {     // Hillis-Steele inclusive scan, 256 entries
        const int64_t add = tid >= off ? s_part[tid - off] : 0;
        __syncthreads();
        s_part[tid] += add;
        __syncthreads();
    }
    int64_t run = s_part[tid] - local;                  // exclusive prefix of this chunk
    if (tid == 0) s_cu[0] = 0;
    for (int i = lo; i < hi; ++i) {
        run += (int64_t)max(grid_hw[2 * i], 0) * max(grid_hw[2 * i + 1], 0);
        s_cu[i + 1] = run;
    }
    __syncthreads();
    const int64_t total = s_cu[n_img];
    if (s_bad || total != T) {
        if (blockIdx.x == 0 && tid == 0) report_error(status, VIT_ERR_GRID_MISMATCH);
        return;
    }

    if (blockIdx.x == 0) {
        if (inv_freq)
            for (int j = tid; j < dim / 2; j += kThreads)
                inv_freq[j] = 1.0f / powf(theta, (float)(2 * j) / (float)dim);
        if (cu_out)
            for (int i = tid; i <= n_img; i += kThreads) cu_out[i] = (int32_t)s_cu[i];
    }
    if (!pos_hw) return;

    for (int64_t t = (int64_t)blockIdx.x * kTokensPerBlock + tid;
         t < T && t < (int64_t)(blockIdx.x + 1) * kTokensPerBlock; t += kThreads) {
        // last image i with s_cu[i] <= t (skips empty images)
        int a = 0, b = n_img;                          // invariant: s_cu[a] <= t < s_cu[b]
        while (b - a > 1) {
            const int m = (a + b) >> 1;
            if (s_cu[m] <= t) a = m; else b = m;
        }
        const int w = grid_hw[2 * a + 1];
        const int off = (int)(t - s_cu[a]);
        pos_hw[t] = make_int2(off / w, off % w);
    }
}

// cos/sin of p * inv_freq[f] for every position p < max_pos and frequency f < n_freq
// (VisionRotaryEmbedding's table over positions, indexed later by each token's row and
// column): entry (p, f/2) = {cos a_f, cos a_f+1, sin a_f, sin a_f+1}, the same fp32
// product and sincosf the prologue kernel evaluates per token.
__global__ void __launch_bounds__(kThreads)
rope_table_kernel(const float *__restrict__ inv_freq, int n_freq, int max_pos, float4 *__restrict__ cs)
{
    const int per = n_freq / 2;
    const int64_t n = (int64_t)max_pos * per;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        const int p = (int)(i / per), f = 2 * (int)(i % per);
        const float pos = (float)p;
        float s0, c0, s1, c1;
        sincosf(pos * inv_freq[f], &s0, &c0);
        sincosf(pos * inv_freq[f + 1], &s1, &c1);
        cs[i] = make_float4(c0, c1, s0, s1);
    }
}

}  // namespace

cudaError_t launch_rope_table(const float *inv_freq, int n_freq, int max_pos, float *cos_sin, cudaStream_t stream)
{
    const int64_t n = (int64_t)max_pos * (n_freq / 2);
    if (n == 0) return cudaSuccess;
    const int64_t want = (n + kThreads - 1) / kThreads;
    const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
    LaunchScope scope("rope_table", stream);
    rope_table_kernel<<<blocks, kThreads, 0, stream>>>(inv_freq, n_freq, max_pos, reinterpret_cast<float4 *>(cos_sin));
    return cudaGetLastError();
}

cudaError_t launch_rope_freqs(int dim, float theta, const int32_t *grid_hw, int n_img, int64_t T,
                              float *inv_freq, int32_t *pos_hw, int32_t *cu_seqlens, int32_t *status,
                              cudaStream_t stream)
{
    const int64_t blocks = T > 0 ? (T + kTokensPerBlock - 1) / kTokensPerBlock : 1;
    const size_t smem = sizeof(int64_t) * (size_t)(n_img + 1);
    static DeviceOnce once;                              // the limit for the largest grid list, set once
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(rope_freqs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(sizeof(int64_t) * (VIT_MAX_SEGMENTS + 1)));
    });
    if (e != cudaSuccess) return e;
    LaunchScope scope("rope_freqs", stream);
    rope_freqs_kernel<<<(unsigned)blocks, kThreads, smem, stream>>>(
        dim, theta, grid_hw, n_img, T, inv_freq, reinterpret_cast<int2 *>(pos_hw), cu_seqlens, status);
    return cudaGetLastError();
}

}  // namespace vit
