// Short-segment varlen attention: 64-query-row tiles on warp-level MMA.
//
// Computes, for each work item (segment, head, 64-row query block) of the
// scheduler's list, out = softmax(scale * q k^T) v over the keys of that
// segment only (vLLM Dots vision_attention page, VisionAttentionV2.forward:
// plain attention per segment; VisionAttention.forward: the same result
// through a block-diagonal mask). Softmax in fp32 (F.softmax(..., dtype=
// float32) on the same page), probabilities rounded to bf16 for the P.V
// product, fp32 accumulation, bf16 output.
//
// Segments up to a few hundred tokens are HBM/latency bound (arithmetic
// intensity ~L/2 flop/byte), so this path favours many small independent
// CTAs: 4 warps x 16 query rows, 64-key tiles double-buffered with cp.async,
// online softmax in registers (exp2 with the scale folded in), and rows
// outside the segment zero-filled on load so no other segment is ever read.
#include "internal.h"

namespace vit {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int BM = 64;   // query rows per item (16 per warp)
constexpr int BN = 64;   // keys per tile

template <int D> struct ShortCfg {
    static constexpr int PITCH = D + 8;                          // smem row pitch (elements): conflict-free ldmatrix
    static constexpr int Q_ELEMS = BM * PITCH;
    static constexpr int KV_ELEMS = BN * PITCH;
    static constexpr size_t SMEM = sizeof(__nv_bfloat16) * (Q_ELEMS + 4 * KV_ELEMS);
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;                                // 0 source bytes -> 16 zero bytes
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma16816(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Copy `rows` rows of D bf16 (row r of the tile = token row0 + r) into smem with
// the padded pitch; rows >= valid_rows are zero-filled and never read from HBM.
template <int D>
__device__ __forceinline__ void load_tile(__nv_bfloat16 *s, const __nv_bfloat16 *g, int64_t stride, int64_t row0,
                                          int rows, int valid_rows) {
    constexpr int CH = D / 8;                                    // 16-byte chunks per row
    for (int i = threadIdx.x; i < rows * CH; i += kThreads) {
        const int r = i / CH, c = i - r * CH;
        const bool ok = r < valid_rows;
        const __nv_bfloat16 *src = g + (ok ? (row0 + r) * stride : 0) + c * 8;
        cp_async16(smem_u32(s + r * ShortCfg<D>::PITCH + c * 8), src, ok);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
attn_short_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                  const __nv_bfloat16 *__restrict__ v, int64_t q_stride, int64_t k_stride, int64_t v_stride,
                  __nv_bfloat16 *__restrict__ out, int64_t out_stride, float scale_log2,
                  const WsHeader *__restrict__ hdr, const Item *__restrict__ items)
{
    using C = ShortCfg<D>;
    constexpr int PITCH = C::PITCH;
    constexpr int KSTEPS = D / 16;       // QK^T reduction steps
    constexpr int DN = D / 8;            // output n-blocks of 8 columns
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    __nv_bfloat16 *sK = sQ + C::Q_ELEMS;                     // [2][BN][PITCH]
    __nv_bfloat16 *sV = sK + 2 * C::KV_ELEMS;                // [2][BN][PITCH]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int n_items = hdr->n_short, first = hdr->n_long;

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item item = items[first + it];
        const int seg0 = item.x, seg_len = item.y, q0 = item.z, head = item.w;
        const int seg_end = seg0 + seg_len;
        const int q_valid = min(BM, seg_end - q0);
        const int n_tiles = (seg_len + BN - 1) / BN;
        const __nv_bfloat16 *qh = q + head * D, *kh = k + head * D, *vh = v + head * D;

        __syncthreads();                                     // smem of the previous item is free
        load_tile<D>(sQ, qh, q_stride, q0, BM, q_valid);
        load_tile<D>(sK, kh, k_stride, seg0, BN, min(BN, seg_len));
        load_tile<D>(sV, vh, v_stride, seg0, BN, min(BN, seg_len));
        cp_async_commit();

        float o[DN][4];
#pragma unroll
        for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
        uint32_t qf[KSTEPS][4];

        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            if (j + 1 < n_tiles) {
                const int kv0 = seg0 + (j + 1) * BN;
                const int valid = min(BN, seg_end - kv0);
                load_tile<D>(sK + (st ^ 1) * C::KV_ELEMS, kh, k_stride, kv0, BN, valid);
                load_tile<D>(sV + (st ^ 1) * C::KV_ELEMS, vh, v_stride, kv0, BN, valid);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();

            if (j == 0) {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = kk * 16 + (lane >> 4) * 8;
                    ldsm_x4(smem_u32(sQ + row * PITCH + col), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
                }
            }

            // S = Q K^T for this warp's 16 rows x 64 keys
            const __nv_bfloat16 *sKs = sK + st * C::KV_ELEMS;
            float s[BN / 8][4];
#pragma unroll
            for (int nb = 0; nb < BN / 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
                for (int nb = 0; nb < BN / 8; nb += 2) {
                    const int n = nb * 8 + (lane & 7) + (lane >> 4) * 8;
                    const int kc = kk * 16 + ((lane >> 3) & 1) * 8;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(sKs + n * PITCH + kc), b0, b1, b2, b3);
                    mma16816(s[nb], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                    mma16816(s[nb + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
                }
            }

            // scale into the log2 domain, mask keys past the segment end, online softmax
            const int kv_valid = min(BN, seg_end - (seg0 + j * BN));
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nb = 0; nb < BN / 8; ++nb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = nb * 8 + tig * 2 + (e & 1);
                    float x = s[nb][e] * scale_log2;
                    if (col >= kv_valid) x = -INFINITY;
                    s[nb][e] = x;
                    mx[e >> 1] = fmaxf(mx[e >> 1], x);
                }
            }
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float m_new = fmaxf(m_r[r], mx[r]);
                alpha[r] = ex2(m_r[r] - m_new);
                m_r[r] = m_new;
                l_r[r] *= alpha[r];
            }
#pragma unroll
            for (int nb = 0; nb < DN; ++nb) {
                o[nb][0] *= alpha[0];
                o[nb][1] *= alpha[0];
                o[nb][2] *= alpha[1];
                o[nb][3] *= alpha[1];
            }
            uint32_t pf[BN / 16][4];
#pragma unroll
            for (int nb = 0; nb < BN / 8; ++nb) {
                const float p0 = ex2(s[nb][0] - m_r[0]), p1 = ex2(s[nb][1] - m_r[0]);
                const float p2 = ex2(s[nb][2] - m_r[1]), p3 = ex2(s[nb][3] - m_r[1]);
                l_r[0] += p0 + p1;
                l_r[1] += p2 + p3;
                pf[nb >> 1][(nb & 1) * 2 + 0] = pack_bf16(p0, p1);
                pf[nb >> 1][(nb & 1) * 2 + 1] = pack_bf16(p2, p3);
            }

            // O += P V
            const __nv_bfloat16 *sVs = sV + st * C::KV_ELEMS;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
#pragma unroll
                for (int nd = 0; nd < DN; nd += 2) {
                    const int row = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = nd * 8 + (lane >> 4) * 8;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(sVs + row * PITCH + col), b0, b1, b2, b3);
                    mma16816(o[nd], pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3], b0, b1);
                    mma16816(o[nd + 1], pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3], b2, b3);
                }
            }
            __syncthreads();                                 // stage st may be refilled next iteration
        }

        // normalise and store the rows that belong to the segment
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
            l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
        }
        const float inv0 = 1.f / l_r[0], inv1 = 1.f / l_r[1];
        const int r0 = warp * 16 + g, r1 = r0 + 8;
        __nv_bfloat16 *oh = out + head * D;
#pragma unroll
        for (int nd = 0; nd < DN; ++nd) {
            const int col = nd * 8 + tig * 2;
            if (r0 < q_valid)
                *reinterpret_cast<uint32_t *>(oh + (int64_t)(q0 + r0) * out_stride + col) =
                    pack_bf16(o[nd][0] * inv0, o[nd][1] * inv0);
            if (r1 < q_valid)
                *reinterpret_cast<uint32_t *>(oh + (int64_t)(q0 + r1) * out_stride + col) =
                    pack_bf16(o[nd][2] * inv1, o[nd][3] * inv1);
        }
    }
}

template <int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, int64_t qs, int64_t ks, int64_t vs, void *out,
                     int64_t os, float scale_log2, const WsHeader *hdr, const Item *items, int64_t max_items,
                     int num_sms, cudaStream_t stream)
{
    constexpr size_t smem = ShortCfg<D>::SMEM;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(attn_short_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_short_kernel<D>, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int64_t cap = (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
    const unsigned blocks = (unsigned)(max_items < cap ? max_items : cap);
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("attn_short", stream);
    attn_short_kernel<D><<<blocks, kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), qs, ks, vs, static_cast<__nv_bfloat16 *>(out), os, scale_log2, hdr,
        items);
    return cudaGetLastError();
}

}  // namespace

int attn_short_bm() { return BM; }

cudaError_t launch_attn_short(const void *q, const void *k, const void *v, int64_t q_stride, int64_t k_stride,
                              int64_t v_stride, void *out, int64_t out_stride, int D, float scale_log2,
                              const WsHeader *hdr, const Item *items, int64_t max_items_short, int num_sms,
                              cudaStream_t stream)
{
    switch (D) {
        case 32: return launch_d<32>(q, k, v, q_stride, k_stride, v_stride, out, out_stride, scale_log2, hdr, items, max_items_short, num_sms, stream);
        case 64: return launch_d<64>(q, k, v, q_stride, k_stride, v_stride, out, out_stride, scale_log2, hdr, items, max_items_short, num_sms, stream);
        case 80: return launch_d<80>(q, k, v, q_stride, k_stride, v_stride, out, out_stride, scale_log2, hdr, items, max_items_short, num_sms, stream);
        case 96: return launch_d<96>(q, k, v, q_stride, k_stride, v_stride, out, out_stride, scale_log2, hdr, items, max_items_short, num_sms, stream);
        case 128: return launch_d<128>(q, k, v, q_stride, k_stride, v_stride, out, out_stride, scale_log2, hdr, items, max_items_short, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace vit
