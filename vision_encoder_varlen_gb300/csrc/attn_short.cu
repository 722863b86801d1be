// Short-segment varlen attention on warp-level MMA.
//
// Computes, for each work item (segment, head, 128-row query block) of the
// scheduler's list, out = softmax(scale * q k^T) v over the keys of that
// segment only (vLLM Dots vision_attention page, VisionAttentionV2.forward:
// plain attention per segment; VisionAttention.forward: the same result
// through a block-diagonal mask). Softmax in fp32 (F.softmax(..., dtype=
// float32) on the same page), probabilities rounded to bf16 for the P.V
// product, fp32 accumulation, bf16 output.
//
// Segments of up to ~128 tokens are HBM-bound (arithmetic intensity ~L/2
// flop/byte), so the design aims at touching every byte once and wasting
// little arithmetic on padding:
//   - one item covers 128 query rows, so a segment of <= 128 tokens is one
//     item per head and its K and V are read from HBM exactly once;
//   - 4 warps, each owning 32 query rows as two 16-row MMA tiles that share
//     every K and V fragment loaded from shared memory;
//   - keys in 64-key sub-chunks with an online softmax; 16-key groups past the
//     segment end and 16-row tiles past it are skipped, so padding costs at
//     most 15 rows and 15 keys;
//   - rows outside the segment are zero-filled on load and never read from
//     HBM, so no other segment is ever touched; several CTAs per SM overlap
//     one item's loads with another's arithmetic.
// Any segment length works (longer ones loop over 128-key tiles). With the
// default split it has no work: segments of at most 64 tokens go to the
// tiny-segment kernel and longer ones to the tcgen05 kernel; it takes the band
// between 64 tokens and a split a caller raises through vit_varlen_attn_ex.
#include "internal.h"
#include "warp_mma.cuh"

namespace vit {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int BM = 128;   // query rows per item (32 per warp = two 16-row tiles)
constexpr int BN = 128;   // keys per shared-memory tile
constexpr int SUB = 64;   // keys per softmax sub-chunk

template <int D> struct ShortCfg {
    static constexpr int PITCH = D + 8;                          // smem row pitch (elements): conflict-free ldmatrix
    static constexpr int ELEMS = 128 * PITCH;                    // one 128-row tile
    static constexpr size_t SMEM = sizeof(__nv_bfloat16) * 3 * ELEMS;   // Q, K, V
    static constexpr int MIN_BLOCKS = D <= 32 ? 3 : 2;          // CTAs per SM the register budget allows
};

using namespace wmma16;

// Copy rows [0, rows) of a tile into shared memory with the padded pitch (zero fill past valid_rows).
template <int D>
__device__ __forceinline__ void load_rows(__nv_bfloat16 *s, const __nv_bfloat16 *g, int64_t stride, int64_t row0,
                                          int rows, int valid_rows) {
    wmma16::load_rows<D, ShortCfg<D>::PITCH, kThreads>(s, g, stride, row0, rows, valid_rows);
}

template <int D, bool FQ>
__global__ void __launch_bounds__(kThreads, ShortCfg<D>::MIN_BLOCKS)
attn_short_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                  const __nv_bfloat16 *__restrict__ v, int64_t q_stride, int64_t k_stride, int64_t v_stride,
                  __nv_bfloat16 *__restrict__ out, int64_t out_stride, float *__restrict__ lse, int H,
                  float scale_log2, const WsHeader *__restrict__ hdr, const Item *__restrict__ items,
                  const rope::QRope qr)
{
    using C = ShortCfg<D>;
    constexpr int PITCH = C::PITCH;
    constexpr int KSTEPS = D / 16;       // QK^T reduction steps
    constexpr int DN = D / 8;            // output n-blocks of 8 columns
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    __nv_bfloat16 *sK = sQ + C::ELEMS;
    __nv_bfloat16 *sV = sK + C::ELEMS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int n_items = hdr->n_short, first = hdr->n_long;
    const int r_base = warp * 32;

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item item = items[first + it];
        const int seg0 = item.x, seg_len = item.y, q0 = item.z, head = item.w;
        const int seg_end = seg0 + seg_len;
        const int q_valid = min(BM, seg_end - q0);
        const int n_tiles = (seg_len + BN - 1) / BN;
        const __nv_bfloat16 *qh = q + head * D, *kh = k + head * D, *vh = v + head * D;
        // 16-row tiles of this warp that hold at least one query row of the segment
        const bool act0 = r_base < q_valid, act1 = r_base + 16 < q_valid;

        __syncthreads();                                     // smem of the previous item is free
        load_rows<D>(sQ, qh, q_stride, q0, (q_valid + 15) & ~15, q_valid);
        if constexpr (FQ) cp_async_commit();                // Q in a group of its own

        float o[2][DN][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < DN; ++i) o[mt][i][0] = o[mt][i][1] = o[mt][i][2] = o[mt][i][3] = 0.f;
        float m_r[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
        float l_r[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

        for (int j = 0; j < n_tiles; ++j) {
            const int kv0 = seg0 + j * BN;
            const int kv_valid = min(BN, seg_end - kv0);
            if (j > 0) __syncthreads();                      // every warp is done with the previous K/V tile
            load_rows<D>(sK, kh, k_stride, kv0, (kv_valid + 15) & ~15, kv_valid);
            load_rows<D>(sV, vh, v_stride, kv0, (kv_valid + 15) & ~15, kv_valid);
            cp_async_commit();
            if constexpr (FQ) {
                // raw Q: once its group has landed, thread r normalises and rotates row r in shared
                // memory (the prologue kernel's arithmetic, in the same order) while the first K/V
                // tile is still on its way
                if (j == 0) {
                    cp_async_wait_one();
                    __syncthreads();
                    const int r = threadIdx.x;
                    if (r < q_valid)
                        rope::transform_row<D>(qr, (int64_t)q0 + r, [&](int c) {
                            return reinterpret_cast<uint4 *>(sQ + r * PITCH + 8 * c);
                        });
                }
            }
            cp_async_wait_all();
            __syncthreads();
            if (!act0) continue;                             // warp-uniform: nothing of the segment in its rows

            for (int sc = 0; sc * SUB < kv_valid; ++sc) {
                const int k0 = sc * SUB;
                const int nvalid = min(SUB, kv_valid - k0);  // valid keys of this sub-chunk
                const int npairs = (nvalid + 15) >> 4;       // 16-key groups that hold a valid key

                // S = Q K^T for 32 rows x 64 keys (skipping empty 16-key groups / row tiles)
                float s[2][SUB / 8][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nb = 0; nb < SUB / 8; ++nb) s[mt][nb][0] = s[mt][nb][1] = s[mt][nb][2] = s[mt][nb][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    uint32_t a[2][4];
                    const int col = kk * 16 + (lane >> 4) * 8;
                    const int row = r_base + (lane & 7) + ((lane >> 3) & 1) * 8;
                    ldsm_x4(smem_u32(sQ + row * PITCH + col), a[0][0], a[0][1], a[0][2], a[0][3]);
                    if (act1) ldsm_x4(smem_u32(sQ + (row + 16) * PITCH + col), a[1][0], a[1][1], a[1][2], a[1][3]);
#pragma unroll
                    for (int np = 0; np < SUB / 16; ++np) {
                        if (np < npairs) {
                            const int n = k0 + np * 16 + (lane & 7) + (lane >> 4) * 8;
                            const int kc = kk * 16 + ((lane >> 3) & 1) * 8;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(smem_u32(sK + n * PITCH + kc), b0, b1, b2, b3);
                            mma16816(s[0][2 * np], a[0], b0, b1);
                            mma16816(s[0][2 * np + 1], a[0], b2, b3);
                            if (act1) {
                                mma16816(s[1][2 * np], a[1], b0, b1);
                                mma16816(s[1][2 * np + 1], a[1], b2, b3);
                            }
                        }
                    }
                }

                // online softmax in the log2 domain; keys past the segment end -> -inf
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    if (mt == 1 && !act1) break;             // warp-uniform
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int nb = 0; nb < SUB / 8; ++nb) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = nb * 8 + tig * 2 + (e & 1);
                            float x = s[mt][nb][e] * scale_log2;
                            if (c >= nvalid) x = -INFINITY;
                            s[mt][nb][e] = x;
                            mx[e >> 1] = fmaxf(mx[e >> 1], x);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                        const float m_new = fmaxf(m_r[mt][r], mx[r]);
                        const float alpha = ex2(m_r[mt][r] - m_new);
                        m_r[mt][r] = m_new;
                        l_r[mt][r] *= alpha;
#pragma unroll
                        for (int nd = 0; nd < DN; ++nd) {
                            o[mt][nd][2 * r] *= alpha;
                            o[mt][nd][2 * r + 1] *= alpha;
                        }
                    }
#pragma unroll
                    for (int nb = 0; nb < SUB / 8; ++nb) {
                        if (nb < 2 * npairs) {                   // groups past the segment end stay 0
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float p = ex2(s[mt][nb][e] - m_r[mt][e >> 1]);
                                s[mt][nb][e] = p;
                                l_r[mt][e >> 1] += p;
                            }
                        }
                    }
                }

                // O += P V over the 16-key groups that hold valid keys
#pragma unroll
                for (int np = 0; np < SUB / 16; ++np) {
                    if (np < npairs) {
                        uint32_t pa[2][4];
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            pa[mt][0] = pack_bf16(s[mt][2 * np][0], s[mt][2 * np][1]);
                            pa[mt][1] = pack_bf16(s[mt][2 * np][2], s[mt][2 * np][3]);
                            pa[mt][2] = pack_bf16(s[mt][2 * np + 1][0], s[mt][2 * np + 1][1]);
                            pa[mt][3] = pack_bf16(s[mt][2 * np + 1][2], s[mt][2 * np + 1][3]);
                        }
                        const int row = k0 + np * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                        for (int nd = 0; nd < DN; nd += 2) {
                            const int col = nd * 8 + (lane >> 4) * 8;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(smem_u32(sV + row * PITCH + col), b0, b1, b2, b3);
                            mma16816(o[0][nd], pa[0], b0, b1);
                            mma16816(o[0][nd + 1], pa[0], b2, b3);
                            if (act1) {
                                mma16816(o[1][nd], pa[1], b0, b1);
                                mma16816(o[1][nd + 1], pa[1], b2, b3);
                            }
                        }
                    }
                }
            }
        }

        // normalise and store the rows that belong to the segment
        if (act0) {
            __nv_bfloat16 *oh = out + head * D;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt == 1 && !act1) break;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    l_r[mt][r] += __shfl_xor_sync(0xffffffffu, l_r[mt][r], 1);
                    l_r[mt][r] += __shfl_xor_sync(0xffffffffu, l_r[mt][r], 2);
                }
                const float inv0 = 1.f / l_r[mt][0], inv1 = 1.f / l_r[mt][1];
                const int r0 = r_base + mt * 16 + g, r1 = r0 + 8;
                if (lse && tig == 0) {                       // ln(sum exp(scale * s)) = (m + log2 l) ln 2
                    if (r0 < q_valid)
                        lse[(int64_t)(q0 + r0) * H + head] = (m_r[mt][0] + log2f(l_r[mt][0])) * 0.6931471805599453f;
                    if (r1 < q_valid)
                        lse[(int64_t)(q0 + r1) * H + head] = (m_r[mt][1] + log2f(l_r[mt][1])) * 0.6931471805599453f;
                }
#pragma unroll
                for (int nd = 0; nd < DN; ++nd) {
                    const int col = nd * 8 + tig * 2;
                    if (r0 < q_valid)
                        *reinterpret_cast<uint32_t *>(oh + (int64_t)(q0 + r0) * out_stride + col) =
                            pack_bf16(o[mt][nd][0] * inv0, o[mt][nd][1] * inv0);
                    if (r1 < q_valid)
                        *reinterpret_cast<uint32_t *>(oh + (int64_t)(q0 + r1) * out_stride + col) =
                            pack_bf16(o[mt][nd][2] * inv1, o[mt][nd][3] * inv1);
                }
            }
        }
    }
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, int64_t max_items, int num_sms, cudaStream_t stream)
{
    constexpr size_t smem = ShortCfg<D>::SMEM;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    auto kern = a.fuse_q ? attn_short_kernel<D, true> : attn_short_kernel<D, false>;
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
    LaunchScope scope("attn_short", stream);
    kern<<<blocks, kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.q_stride, a.k_stride, a.v_stride,
        static_cast<__nv_bfloat16 *>(a.out), a.out_stride, a.lse, a.H, a.scale_log2, a.hdr, a.items, a.qr);
    return cudaGetLastError();
}

}  // namespace

int attn_short_bm() { return BM; }

cudaError_t launch_attn_short(const AttnArgs &a, int64_t max_items_short, int num_sms, cudaStream_t stream)
{
    switch (a.D) {
        case 32: return launch_d<32>(a, max_items_short, num_sms, stream);
        case 64: return launch_d<64>(a, max_items_short, num_sms, stream);
        case 80: return launch_d<80>(a, max_items_short, num_sms, stream);
        case 96: return launch_d<96>(a, max_items_short, num_sms, stream);
        case 128: return launch_d<128>(a, max_items_short, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace vit
