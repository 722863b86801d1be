// Warp-level MMA building blocks of the warp-MMA attention kernels (short and tiny
// segments): cp.async row loads with zero fill, ldmatrix fragment loads, the
// m16n8k16 bf16 MMA with fp32 accumulation, exp2 and bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace vit {
namespace wmma16 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;                                // 0 source bytes -> 16 zero bytes
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;\n" ::); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// Copy rows [0, rows) of a tile (row r = token row0 + r) into shared memory with row pitch
// PITCH elements, NT threads cooperating; rows >= valid_rows are zero-filled and never read
// from HBM, so nothing outside the segment is touched.
template <int D, int PITCH, int NT>
__device__ __forceinline__ void load_rows(__nv_bfloat16 *s, const __nv_bfloat16 *g, int64_t stride, int64_t row0,
                                          int rows, int valid_rows) {
    constexpr int CH = D / 8;                                    // 16-byte chunks per row
    for (int i = threadIdx.x; i < rows * CH; i += NT) {
        const int r = i / CH, c = i - r * CH;
        const bool ok = r < valid_rows;
        const __nv_bfloat16 *src = g + (ok ? (row0 + r) * stride : 0) + c * 8;
        cp_async16(smem_u32(s + r * PITCH + c * 8), src, ok);
    }
}

}  // namespace wmma16
}  // namespace vit
