// Tiny-segment varlen attention (segments of at most 64 tokens) on warp-level MMA.
//
// Same result as the other two attention kernels: for each (segment, head) the
// plain softmax(scale * q k^T) v over that segment's keys only (vLLM Dots
// vision_attention page, VisionAttentionV2.forward / VisionAttention.forward),
// softmax in fp32, P rounded to bf16 for the P.V product, fp32 accumulation,
// bf16 output.
//
// A segment of L <= 64 tokens moves 4 * L * D * 2 bytes per head and does
// 4 * L^2 * D flops: about L / 2 flops per byte, so it is bound by HBM and by
// latency, not by arithmetic. The design therefore keeps many bytes in flight:
//   - one work item = one (segment, head): Q, K and V are at most 64 rows;
//   - each CTA (4 warps) holds two items' K and V in shared memory and loads
//     the next item with cp.async while it computes the current one; each
//     warp takes its 16 query rows straight from HBM into MMA fragments, so
//     four CTAs share an SM;
//   - warp w owns query rows [16w, 16w + 16) as one MMA tile; the whole key
//     range is one tile, so the softmax is a single pass (exact row max, no
//     running rescale);
//   - rows past the segment end are zero-filled on load and 16-key groups past
//     it are skipped, so no other segment's values (finite or not) enter.
#include "internal.h"
#include "warp_mma.cuh"

namespace vit {
namespace {

using namespace wmma16;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int TM = 64;                       // rows of Q, K and V per item (segment length bound)

// Shared memory holds K and V of two items; Q goes straight from HBM into each warp's MMA
// fragments (16 rows per warp), except when Q arrives raw and is rotated in shared memory (FQ).
template <int D, bool FQ> struct TinyCfg {
    static constexpr int PITCH = D + 8;                          // padded row pitch: conflict-free ldmatrix
    static constexpr int TILE = TM * PITCH;                      // elements of one 64-row tile
    static constexpr int NT = FQ ? 3 : 2;                        // tiles per item: (Q,) K, V
    static constexpr int BUF = NT * TILE;
    static constexpr size_t SMEM = sizeof(__nv_bfloat16) * 2 * BUF;   // two items
    // CTAs per SM: shared memory, then registers (at most 128 per thread for four)
    static constexpr int MIN_BLOCKS = (!FQ && D <= 96) ? 4 : (D <= 96 ? 3 : 2);
};

template <int D, bool FQ>
__device__ __forceinline__ void load_item(__nv_bfloat16 *buf, const Item &item, const __nv_bfloat16 *q,
                                          const __nv_bfloat16 *k, const __nv_bfloat16 *v, int64_t qs, int64_t ks,
                                          int64_t vs) {
    using C = TinyCfg<D, FQ>;
    const int L = item.y, rows = (L + 15) & ~15;
    const int64_t row0 = item.x;
    const int64_t hoff = (int64_t)item.w * D;
    if constexpr (FQ) load_rows<D, C::PITCH, kThreads>(buf + 2 * C::TILE, q + hoff, qs, row0, rows, L);
    load_rows<D, C::PITCH, kThreads>(buf, k + hoff, ks, row0, rows, L);
    load_rows<D, C::PITCH, kThreads>(buf + C::TILE, v + hoff, vs, row0, rows, L);
}

template <int D, bool FQ>
__global__ void __launch_bounds__(kThreads, TinyCfg<D, FQ>::MIN_BLOCKS)
attn_tiny_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, int64_t q_stride, int64_t k_stride, int64_t v_stride,
                 __nv_bfloat16 *__restrict__ out, int64_t out_stride, float *__restrict__ lse, int H,
                 float scale_log2, const WsHeader *__restrict__ hdr, const Item *__restrict__ items,
                 const rope::QRope qr)
{
    using C = TinyCfg<D, FQ>;
    constexpr int PITCH = C::PITCH;
    constexpr int KSTEPS = D / 16;       // QK^T reduction steps
    constexpr int DN = D / 8;            // output n-blocks of 8 columns
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16 *smem = reinterpret_cast<__nv_bfloat16 *>(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int n_items = hdr->n_tiny, first = hdr->n_long + hdr->n_short;
    const int r_base = warp * 16;

    int it = blockIdx.x;
    if (it < n_items) load_item<D, FQ>(smem, items[first + it], q, k, v, q_stride, k_stride, v_stride);
    cp_async_commit();
    for (int n = 0; it < n_items; ++n, it += gridDim.x) {
        // the next item goes into the other buffer while this one is computed; that buffer's
        // previous item finished before the barrier that closed the last iteration
        const int nxt = it + gridDim.x;
        if (nxt < n_items)
            load_item<D, FQ>(smem + ((n + 1) & 1) * C::BUF, items[first + nxt], q, k, v, q_stride, k_stride,
                             v_stride);
        cp_async_commit();
        const Item item = items[first + it];
        const int seg0 = item.x, L = item.y, head = item.w;
        // this warp's 16 query rows as MMA A fragments, loaded while K and V land: fragment e of
        // k-step kk holds row g (e even) or g + 8, columns 2 tig, 2 tig + 1 (+ 8 for e >= 2)
        uint32_t qa[KSTEPS][4];
        if constexpr (!FQ) {
            const __nv_bfloat16 *q0r = q + (int64_t)(seg0 + r_base + g) * q_stride + (int64_t)head * D + 2 * tig;
            const __nv_bfloat16 *q8r = q0r + 8 * q_stride;
            const bool ok0 = r_base + g < L, ok8 = r_base + g + 8 < L;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                qa[kk][0] = ok0 ? *reinterpret_cast<const uint32_t *>(q0r + kk * 16) : 0u;
                qa[kk][1] = ok8 ? *reinterpret_cast<const uint32_t *>(q8r + kk * 16) : 0u;
                qa[kk][2] = ok0 ? *reinterpret_cast<const uint32_t *>(q0r + kk * 16 + 8) : 0u;
                qa[kk][3] = ok8 ? *reinterpret_cast<const uint32_t *>(q8r + kk * 16 + 8) : 0u;
            }
        }
        cp_async_wait_one();                                 // this item's group has landed
        __syncthreads();

        __nv_bfloat16 *sK = smem + (n & 1) * C::BUF, *sV = sK + C::TILE, *sQ = sV + C::TILE;
        if constexpr (FQ) {
            // raw Q: thread r normalises and rotates row r (the prologue kernel's arithmetic)
            const int r = threadIdx.x;
            if (r < L)
                rope::transform_row<D>(qr, (int64_t)seg0 + r, [&](int c) {
                    return reinterpret_cast<uint4 *>(sQ + r * PITCH + 8 * c);
                });
            __syncthreads();
        }

        if (r_base < L) {                                    // warp-uniform
            const int n16 = (L + 15) >> 4;                   // 16-key groups holding a key of the segment
            // S = Q K^T for 16 rows x up to 64 keys
            float s[8][4];
#pragma unroll
            for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t a[4];
                if constexpr (FQ) {
                    ldsm_x4(smem_u32(sQ + (r_base + (lane & 7) + ((lane >> 3) & 1) * 8) * PITCH + kk * 16 +
                                     (lane >> 4) * 8),
                            a[0], a[1], a[2], a[3]);
                } else {
                    a[0] = qa[kk][0];
                    a[1] = qa[kk][1];
                    a[2] = qa[kk][2];
                    a[3] = qa[kk][3];
                }
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np < n16) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(smem_u32(sK + (np * 16 + (lane & 7) + (lane >> 4) * 8) * PITCH + kk * 16 +
                                         ((lane >> 3) & 1) * 8),
                                b0, b1, b2, b3);
                        mma16816(s[2 * np], a, b0, b1);
                        mma16816(s[2 * np + 1], a, b2, b3);
                    }
                }
            }
            // softmax over the whole key range in one pass (log2 domain); keys past the end -> -inf
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = nb * 8 + tig * 2 + (e & 1);
                    const float x = c < L ? s[nb][e] * scale_log2 : -INFINITY;
                    s[nb][e] = x;
                    mx[e >> 1] = fmaxf(mx[e >> 1], x);
                }
            float l[2] = {0.f, 0.f};
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            }
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
                if (nb < 2 * n16)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p = ex2(s[nb][e] - mx[e >> 1]);
                        s[nb][e] = p;
                        l[e >> 1] += p;
                    }
            // O = P V over the 16-key groups of the segment
            float o[DN][4];
#pragma unroll
            for (int nd = 0; nd < DN; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np < n16) {
                    uint32_t pa[4];
                    pa[0] = pack_bf16(s[2 * np][0], s[2 * np][1]);
                    pa[1] = pack_bf16(s[2 * np][2], s[2 * np][3]);
                    pa[2] = pack_bf16(s[2 * np + 1][0], s[2 * np + 1][1]);
                    pa[3] = pack_bf16(s[2 * np + 1][2], s[2 * np + 1][3]);
                    const int row = np * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int nd = 0; nd < DN; nd += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(sV + row * PITCH + nd * 8 + (lane >> 4) * 8), b0, b1, b2, b3);
                        mma16816(o[nd], pa, b0, b1);
                        mma16816(o[nd + 1], pa, b2, b3);
                    }
                }
            }
            // normalise and store the rows of the segment
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
            }
            const float inv0 = 1.f / l[0], inv1 = 1.f / l[1];
            const int r0 = r_base + g, r1 = r0 + 8;
            if (lse && tig == 0) {                           // ln(sum exp(scale * s)) = (m + log2 l) ln 2
                if (r0 < L) lse[(int64_t)(seg0 + r0) * H + head] = (mx[0] + log2f(l[0])) * 0.6931471805599453f;
                if (r1 < L) lse[(int64_t)(seg0 + r1) * H + head] = (mx[1] + log2f(l[1])) * 0.6931471805599453f;
            }
            __nv_bfloat16 *oh = out + (int64_t)head * D;
#pragma unroll
            for (int nd = 0; nd < DN; ++nd) {
                const int col = nd * 8 + tig * 2;
                if (r0 < L)
                    *reinterpret_cast<uint32_t *>(oh + (int64_t)(seg0 + r0) * out_stride + col) =
                        pack_bf16(o[nd][0] * inv0, o[nd][1] * inv0);
                if (r1 < L)
                    *reinterpret_cast<uint32_t *>(oh + (int64_t)(seg0 + r1) * out_stride + col) =
                        pack_bf16(o[nd][2] * inv1, o[nd][3] * inv1);
            }
        }
        __syncthreads();                                     // this buffer is free for the item after next
    }
    cp_async_wait_all();                                     // nothing in flight when the CTA exits
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, int64_t max_items, int num_sms, cudaStream_t stream)
{
    const size_t smem = a.fuse_q ? TinyCfg<D, true>::SMEM : TinyCfg<D, false>::SMEM;
    static_assert(TinyCfg<D, true>::SMEM <= 227 * 1024, "shared memory budget");
    auto kern = a.fuse_q ? attn_tiny_kernel<D, true> : attn_tiny_kernel<D, false>;
    static DeviceOnce once[2];                           // per fused-Q variant
    static int per_sm_of[2][64];                         // resident CTAs per SM, per variant and device
    const int var = a.fuse_q ? 1 : 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = once[var].run([&] {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r != cudaSuccess) return r;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_of[var][dev], kern, kThreads, smem);
    });
    if (e != cudaSuccess) return e;
    const int per_sm = per_sm_of[var][dev];
    const int64_t cap = (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
    const unsigned blocks = (unsigned)(max_items < cap ? max_items : cap);
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("attn_tiny", stream);
    kern<<<blocks, kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.q_stride, a.k_stride, a.v_stride,
        static_cast<__nv_bfloat16 *>(a.out), a.out_stride, a.lse, a.H, a.scale_log2, a.hdr, a.items, a.qr);
    return cudaGetLastError();
}

}  // namespace

int attn_tiny_max() { return TM; }

cudaError_t launch_attn_tiny(const AttnArgs &a, int64_t max_items_tiny, int num_sms, cudaStream_t stream)
{
    switch (a.D) {
        case 32: return launch_d<32>(a, max_items_tiny, num_sms, stream);
        case 64: return launch_d<64>(a, max_items_tiny, num_sms, stream);
        case 80: return launch_d<80>(a, max_items_tiny, num_sms, stream);
        case 96: return launch_d<96>(a, max_items_tiny, num_sms, stream);
        case 128: return launch_d<128>(a, max_items_tiny, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace vit
