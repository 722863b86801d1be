// Tiny-segment varlen attention (segments of at most 64 tokens) on warp-level MMA.
//
// Same result as the tcgen05 long-segment kernel: for each (segment, head) the
// plain softmax(scale * q k^T) v over that segment's keys only (vLLM Dots
// vision_attention page, VisionAttentionV2.forward / VisionAttention.forward),
// softmax in fp32, P rounded to bf16 for the P.V product, fp32 accumulation,
// bf16 output.
//
// A segment of L <= 64 tokens moves 4 * L * D * 2 bytes per head and does
// 4 * L^2 * D flops: about L / 2 flops per byte, so it is bound by HBM, and the
// way to reach HBM speed is to keep enough bytes in flight on every SM, in few
// wide requests. The design streams items through one large shared-memory ring
// per SM:
//   - one work item = one segment and HG consecutive heads (2 at head_dim 32,
//     80 and 96 when the head count is even, 4 at head_dim 80 when no segment
//     can exceed 24 tokens and the head count allows, else 1), so that a token's
//     row of the item is HG * D * 2 contiguous bytes; one persistent CTA per SM;
//   - a producer warp copies each item's Q, K and V with tiled TMA loads of 16
//     rows each into the next free bytes of the ring: an item takes ceil16(L)
//     rows per tensor, not the 64 rows of the longest segment. Rows are stored
//     densely under the TMA swizzle whose span makes ldmatrix reads of eight
//     rows conflict-free (a 32-byte span for 160-byte rows, 64 for 64-, 192-
//     and 320-byte rows, 128 for rows of an odd number of 128-byte spans; a
//     single head at head_dim 128 is two 128-byte slabs);
//   - consumer groups of four warps take the CTA's items in turn; a unit of work
//     is one head and 16 query rows, taken by the group's warps in turn, with the
//     whole key range as one MMA tile, so the softmax is a single pass (exact row
//     max, no running rescale). The warps of a group do not wait for each other
//     (except to rotate raw Q), and each releases its item's ring bytes once its
//     last shared-memory read is done, before its last output stores;
//   - the ring is allocated in item order and freed in item order: the producer
//     waits for the oldest unreleased item until the next one fits or the ring
//     is empty;
//   - shared-memory rows past the segment end hold the next tokens' rows (or
//     zeros past the last token): keys past it get score -inf by a select, V rows
//     past it are zeroed in registers before the P.V product, and query rows past
//     it are never stored, so no other segment's values (finite or not) enter a
//     result;
//   - the output leaves in whole 16-byte pieces of a row: the MMA accumulator
//     gives each lane two columns of every 8-column block, and the four lanes
//     of a quad exchange words (two shuffle stages) so that each holds one
//     block (not at head_dim 128, where 4-byte stores measured faster).
// Every wait is bounded: one that gives up records VIT_ERR_TIMEOUT, all roles
// leave their loops, and the producer waits (with a short limit) for its copies
// in flight before the CTA exits.
#include "internal.h"
#include "sm100.cuh"
#include "warp_mma.cuh"

#include <type_traits>

namespace vit {
namespace {

using namespace wmma16;
using sm100::mbar_arrive;
using sm100::mbar_arrive_expect_tx;
using sm100::mbar_init;
using sm100::mbar_try_wait;

constexpr int TM = 64;                       // segment length bound (rows of Q, K and V per item)
constexpr int kSlots = 32;                   // items in the ring at most (descriptor ring)
constexpr long long kWaitBudget = 4000000000ll;   // clock cycles before a wait gives up (~2 s)
constexpr long long kDrainBudget = 200000000ll;   // for copies in flight after an abort

template <int D, bool FQ, int HG> struct TinyCfg {
    // consumer groups of four warps, plus the producer warp (the last one). Registers are split
    // between the SM's four sub-partitions: with 13 warps one of them holds four warps, which caps
    // a thread at 16384 / (4 * 32) = 128 registers (at head_dim 128 and single-head 96, P.V runs
    // in 32-column chunks to stay below).
    static constexpr int GROUPS = 3;
    static constexpr int PV_CHUNK = (D == 128 || (D == 96 && HG == 1)) ? 4 : D / 8;   // 8-column blocks
    // output stores of 16 bytes per lane (the lanes of a quad exchange words) except at head_dim
    // 128, where the 32-column P.V chunks measured faster with plain 4-byte stores between them
    static constexpr bool WIDE_STORES = D != 128;
    // one copy of a unit's code per count of 16-key groups: measured faster at head_dim 80 with
    // several heads per item (16-64 tokens: -9 %, 9-24 tokens: -16 %), slower at 64 and 128, where
    // the copies also no longer fit the registers without spilling
    static constexpr bool PER_N16 = D == 80 && HG >= 2 && !FQ;
    static constexpr int CONSUMERS = 4 * GROUPS;
    static constexpr int THREADS = 32 * (CONSUMERS + 1);
    // An item is one segment and HG consecutive heads. A tensor tile of an item holds its rows
    // (16 * n16 of them) of the HG heads side by side, as SLABS slabs of SLAB_BYTES per row, each
    // slab written by TMA boxes of {W elements, CHUNKS, 16 rows} under the swizzle of span 2 * W
    // bytes. The spans are chosen so that the eight rows of an ldmatrix read fall in eight
    // different bank groups: a row of 160 bytes under the 32-byte span, 64, 192 or 320 under the
    // 64-byte span, and an odd number of 128-byte spans under the 128-byte span.
    static constexpr int SLABS = D == 128 ? 2 : 1;
    static constexpr int SLAB_BYTES = HG * D * 2 / SLABS;
    static constexpr int W =
        SLAB_BYTES == 160 ? 16 : ((SLAB_BYTES == 64 || SLAB_BYTES == 192 || SLAB_BYTES == 320) ? 32 : 64);
    static constexpr int CHUNKS = SLAB_BYTES / (2 * W);
    static constexpr uint32_t SWZ = W == 16 ? 1 : (W == 32 ? 3 : 7);   // 16-byte chunk bits flipped
    static constexpr int RING = 220 * 1024;                      // bytes of the item ring
    static constexpr int SMEM = RING + 1024;                     // + alignment of the ring start
    static constexpr int MAX_ITEM = 3 * 1024 * ((SLABS * TM * SLAB_BYTES + 1023) / 1024);
    static_assert(SLABS == 1 || HG == 1, "two slabs only for single heads");
    static_assert(SLAB_BYTES % (2 * W) == 0 && (W != 64 || CHUNKS % 2 == 1), "slab of an odd number of spans");
    static_assert(RING % 1024 == 0, "1024-byte tiles");
    static_assert(MAX_ITEM <= RING, "the largest item fits in the empty ring");
    // bytes of one tensor tile of n16 16-row groups: tiles start on 1024-byte boundaries, so the
    // swizzle (a function of the address bits) is the same for TMA and for the readers below
    static __host__ __device__ constexpr uint32_t tile_bytes(int n16) {
        return (uint32_t)(SLABS * 16 * n16 * SLAB_BYTES + 1023) / 1024 * 1024;
    }
    // shared-memory address of element column `col` of row `r` of a tile at `base`
    static __device__ __forceinline__ uint32_t at(uint32_t base, int n16, int r, int col) {
        const int cb = col * 2;
        const int s = SLABS == 1 ? 0 : cb / SLAB_BYTES;
        const uint32_t a = base + (uint32_t)(s * 16 * n16 * SLAB_BYTES + r * SLAB_BYTES + cb - s * SLAB_BYTES);
        return a ^ (((a >> 7) & SWZ) << 4);
    }
};

struct TinyShared {
    uint64_t full[kSlots];                   // producer -> consumers: the item's rows have landed
    uint64_t empty[kSlots];                  // consumers -> producer: four warps are done reading
    int4 item[kSlots];                       // {first token, length, first head, tile address in shared memory}
    unsigned long long end[kSlots];          // ring position (bytes since the start) after the item
    volatile int abort;
};

// true for every thread of the 128-thread group on named barrier `id` when `ok` holds for all of them
__device__ __forceinline__ bool group_all(bool ok, int id) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 128, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r) : "r"((uint32_t)ok), "r"(id) : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t bar_addr(const uint64_t *b) { return smem_u32(b); }

// V fragment of keys k0, k0 + 1 (low, high half) with keys at or past L zeroed
__device__ __forceinline__ uint32_t keep_keys(uint32_t b, int k0, int L) {
    return b & ((k0 < L ? 0x0000ffffu : 0u) | (k0 + 1 < L ? 0xffff0000u : 0u));
}

template <int D, bool FQ, int HG>
__global__ void __launch_bounds__(TinyCfg<D, FQ, HG>::THREADS, 1)
attn_tiny_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ out, int64_t out_stride,
                 float *__restrict__ lse, int H,
                 float scale_log2, const WsHeader *__restrict__ hdr, const Item *__restrict__ items,
                 int32_t *__restrict__ status, const rope::QRope qr)
{
    using C = TinyCfg<D, FQ, HG>;
    constexpr int KSTEPS = D / 16;       // QK^T reduction steps
    constexpr int DN = D / 8;            // output n-blocks of 8 columns
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ TinyShared sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a tiny segment has one work item per head, in head order: HG of them make one item here
    const int n_items = hdr->n_tiny / HG, first = hdr->n_long;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(bar_addr(&sh.full[i]), 1);
            mbar_init(bar_addr(&sh.empty[i]), 4);
        }
        sh.abort = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();

    // bounded wait; the first role to give up records the timeout and tells the others
    auto wait = [&](const uint64_t *b, uint32_t parity) -> bool {
        if (mbar_try_wait(bar_addr(b), parity)) return true;
        const long long t0 = clock64();
        while (true) {
            if (mbar_try_wait(bar_addr(b), parity)) return true;
            if (sh.abort) return false;
            if (clock64() - t0 > kWaitBudget) {
                if (!sh.abort) {
                    sh.abort = 1;
                    report_error(status, VIT_ERR_TIMEOUT);
                }
                return false;
            }
        }
    };

    if (warp == C::CONSUMERS) {
        // ---------------------------------------------------------------- producer warp
        const uint32_t ring_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
        if (lane == 0) {
            sm100::tma_prefetch_desc(&tm_q);
            sm100::tma_prefetch_desc(&tm_k);
            sm100::tma_prefetch_desc(&tm_v);
        }
        unsigned long long head = 0, freed = 0;    // ring positions: next free byte, end of the released
        int released = 0, n = 0;
        bool ok = true;
        // item descriptors are read 32 at a time, one per lane, the next 32 while these are placed
        auto fetch = [&](int n0) {
            const int it = blockIdx.x + (n0 + lane) * gridDim.x;
            return it < n_items ? items[first + it * HG] : make_int4(0, 0, 0, 0);
        };
        Item batch = fetch(0), ahead = fetch(32);
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
            if ((n & 31) == 0 && n > 0) {
                batch = ahead;
                ahead = fetch(n + 32);
            }
            Item item;
            item.x = __shfl_sync(0xffffffffu, batch.x, n & 31);
            item.y = __shfl_sync(0xffffffffu, batch.y, n & 31);
            item.w = __shfl_sync(0xffffffffu, batch.w, n & 31);
            const int L = item.y, n16 = (L + 15) >> 4, hd = item_head(item);
            const uint32_t tb = C::tile_bytes(n16);
            const unsigned long long sz = 3ull * tb;
            unsigned long long start = head;
            if (start % C::RING + sz > C::RING) start += C::RING - start % C::RING;   // wrap to the ring start
            // free the oldest items until this one fits (or the ring is empty) and its descriptor
            // slot is free
            while (n - released >= kSlots || (released < n && start + sz > freed + C::RING)) {
                const int s = released % kSlots;
                bool got = true;
                if (lane == 0) got = wait(&sh.empty[s], (released / kSlots) & 1);
                if (!(ok = __shfl_sync(0xffffffffu, got, 0))) break;
                freed = sh.end[s];
                ++released;
            }
            if (!ok) break;
            if (released == n) freed = start;                 // empty ring: all of it is free
            const int slot = n % kSlots;
            const uint32_t off = (uint32_t)(start % C::RING);
            head = start + sz;
            if (lane == 0) {
                sh.item[slot] = make_int4(item.x, L, hd, (int)(ring_base + off));
                sh.end[slot] = head;
                // whole boxes land, rows past the segment included (past the last token: zeros)
                mbar_arrive_expect_tx(bar_addr(&sh.full[slot]), 3u * 16u * n16 * HG * D * 2);
            }
            __syncwarp();
            // one box per (tensor, 16-row group, slab): at most 3 * 4 * 2 = 24, one per lane
            const int boxes = 3 * n16 * C::SLABS;
            if (lane < boxes) {
                const int t = lane / (n16 * C::SLABS), rest = lane - t * n16 * C::SLABS;
                const int j = rest / C::SLABS, sl = rest - j * C::SLABS;
                const CUtensorMap *map = t == 0 ? &tm_q : (t == 1 ? &tm_k : &tm_v);
                const uint32_t dst = ring_base + off + t * tb + (uint32_t)(sl * 16 * n16 + 16 * j) * C::SLAB_BYTES;
                sm100::tma_load_3d(dst, map, 0, (hd * D + sl * (C::SLAB_BYTES / 2)) / C::W, item.x + 16 * j,
                                   bar_addr(&sh.full[slot]));
            }
        }
        // after an abort, the copies already issued must land before the CTA may exit
        // (nothing is in flight in the normal path once the consumers are done)
        if (!ok || sh.abort) {
            for (int m = released; m < n; ++m) {
                const long long t0 = clock64();
                while (!mbar_try_wait(bar_addr(&sh.full[m % kSlots]), (m / kSlots) & 1) &&
                       clock64() - t0 < kDrainBudget) {
                }
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumer warps
    const int grp = warp >> 2, wr = warp & 3;
    const int g = lane >> 2, tig = lane & 3;
    for (int n = grp;; n += C::GROUPS) {
        const int it = blockIdx.x + n * gridDim.x;
        if (it >= n_items) break;
        const int slot = n % kSlots;
        bool ok = __all_sync(0xffffffffu, wait(&sh.full[slot], (n / kSlots) & 1));
        if constexpr (FQ) ok = group_all(ok, grp + 1);   // the group's warps go on (or stop) together
        if (!ok) break;
        const int4 ti = sh.item[slot];
        const int seg0 = ti.x, L = ti.y, head0 = ti.z;
        const int n16 = (L + 15) >> 4;                   // 16-key groups holding a key of the segment
        const uint32_t tb = C::tile_bytes(n16);
        const uint32_t sQ0 = (uint32_t)ti.w, sK0 = sQ0 + tb, sV0 = sK0 + tb;

        if constexpr (FQ) {
            // raw Q: the group's threads normalise and rotate its rows (the prologue kernel's arithmetic)
            for (int p = threadIdx.x - grp * 128; p < L * HG; p += 128) {
                const int r = p / HG, hl = p - r * HG;
                rope::transform_row<D>(qr, (int64_t)seg0 + r, [&](int c) {
                    return reinterpret_cast<uint4 *>(smem_raw +
                                                     (C::at(sQ0, n16, r, hl * D + 8 * c) - smem_u32(smem_raw)));
                });
            }
            asm volatile("bar.sync %0, 128;\n" ::"r"(grp + 1) : "memory");
        }

        // the item's units (head hl, 16 query rows from 16 rt) go to the group's warps in turn; a
        // warp releases the item's ring bytes after the shared-memory reads of its last unit
        const int units = HG * n16;
        auto release = [&] {
            __syncwarp();
            if constexpr (FQ) sm100::fence_proxy_async_smem();   // its Q writes precede the next copy there
            if (lane == 0) mbar_arrive(bar_addr(&sh.empty[slot]));
        };
        // the first unit of this warp: the group's warps start one place further on each item, so
        // that the items whose unit count is not a multiple of four load them evenly over time
        const int u0 = (wr + n / C::GROUPS) & 3;
        if (u0 >= units) release();
        // (one head: at most four units, so a warp has at most one)
        constexpr int kStep = HG == 1 ? TM : 4;
#pragma unroll 1
        for (int u = u0; u < units; u += kStep) {
            const int rt = u / HG, hl = u - rt * HG;
            const int r_base = rt * 16, cq = hl * D, head = head0 + hl;
            // at head_dim 80 (several heads per item) the unit's code is compiled once per count of
            // 16-key groups (1 to 4), so every loop over key groups has a fixed trip count; N16 = 0
            // is the one copy for any count
            auto unit = [&](auto n16c) {
                constexpr int N16 = decltype(n16c)::value;
                const int nk = N16 > 0 ? N16 : n16;
                // the tile addresses are re-derived in each unit: hoisting the K and V fragment
                // addresses out of the loop would hold dozens of registers across it
                uint32_t sQ = sQ0, sK = sK0, sV = sV0;
                asm volatile("" : "+r"(sQ), "+r"(sK), "+r"(sV));
                float s[8][4];
                float mx[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
                // S = Q K^T for 16 rows x up to 64 keys
#pragma unroll
                for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(C::at(sQ, nk, r_base + (lane & 7) + ((lane >> 3) & 1) * 8, cq + kk * 16 + (lane >> 4) * 8),
                            a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        if (np < nk) {
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(C::at(sK, nk, np * 16 + (lane & 7) + (lane >> 4) * 8,
                                          cq + kk * 16 + ((lane >> 3) & 1) * 8),
                                    b0, b1, b2, b3);
                            mma16816(s[2 * np], a, b0, b1);
                            mma16816(s[2 * np + 1], a, b2, b3);
                        }
                    }
                }
                // softmax over the whole key range in one pass: the row max of the raw scores (the
                // scale is positive), then p = 2^(s * scale*log2(e) - max * scale*log2(e)) with one FMA
                // per score; keys past the end -> -inf
#pragma unroll
                for (int nb = 0; nb < 8; ++nb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = nb * 8 + tig * 2 + (e & 1);
                        const float x = c < L ? s[nb][e] : -INFINITY;
                        s[nb][e] = x;
                        mx[e >> 1] = fmaxf(mx[e >> 1], x);
                    }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                    mx[r] *= scale_log2;                         // the row max in the log2 domain
                }
#pragma unroll
                for (int nb = 0; nb < 8; ++nb)
                    if (nb < 2 * nk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p = ex2(fmaf(s[nb][e], scale_log2, -mx[e >> 1]));
                            s[nb][e] = p;
                            l[e >> 1] += p;
                        }
                // P as bf16 A fragments, one per 16-key group (S is dead after this)
                uint32_t pa[4][4];
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    pa[np][0] = pack_bf16(s[2 * np][0], s[2 * np][1]);
                    pa[np][1] = pack_bf16(s[2 * np][2], s[2 * np][3]);
                    pa[np][2] = pack_bf16(s[2 * np + 1][0], s[2 * np + 1][1]);
                    pa[np][3] = pack_bf16(s[2 * np + 1][2], s[2 * np + 1][3]);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
                }
                // l >= 1 (the row max contributes 2^0): the fast reciprocal is within an ulp or two
                const float inv0 = __fdividef(1.f, l[0]), inv1 = __fdividef(1.f, l[1]);
                const int r0 = r_base + g, r1 = r0 + 8;
                if (lse && tig == 0) {                           // ln(sum exp(scale * s)) = (m + log2 l) ln 2
                    if (r0 < L) lse[(int64_t)(seg0 + r0) * H + head] = (mx[0] + log2f(l[0])) * 0.6931471805599453f;
                    if (r1 < L) lse[(int64_t)(seg0 + r1) * H + head] = (mx[1] + log2f(l[1])) * 0.6931471805599453f;
                }
                __nv_bfloat16 *oh = out + (int64_t)head * D;
                // O = P V over the 16-key groups of the segment, in chunks of NC 8-column blocks that
                // are normalised and stored before the next: at the widest rows, 16 accumulators
                // instead of D / 2 keep the unit within 128 registers
                constexpr int NC = C::PV_CHUNK;
#pragma unroll
                for (int c0 = 0; c0 < DN; c0 += NC) {
                    float o[NC][4];
#pragma unroll
                    for (int j = 0; j < NC; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        if (np < nk) {
                            const int row = np * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                            // fragments b0/b2 hold keys 16 np + 2 tig (+1), b1/b3 the same + 8
                            const int k0 = np * 16 + 2 * tig, k1 = k0 + 8;
                            const bool tail = np * 16 + 16 > L;
#pragma unroll
                            for (int j = 0; j < NC; j += 2) {
                                if (c0 + j < DN) {
                                    uint32_t b0, b1, b2, b3;
                                    ldsm_x4_t(C::at(sV, nk, row, cq + (c0 + j) * 8 + (lane >> 4) * 8), b0, b1, b2, b3);
                                    if (tail) {
                                        b0 = keep_keys(b0, k0, L);
                                        b1 = keep_keys(b1, k1, L);
                                        b2 = keep_keys(b2, k0, L);
                                        b3 = keep_keys(b3, k1, L);
                                    }
                                    mma16816(o[j], pa[np], b0, b1);
                                    mma16816(o[j + 1], pa[np], b2, b3);
                                }
                            }
                        }
                    }
                    // this warp's reads of the ring are done after the last chunk of its last unit
                    if (c0 + NC >= DN && u + kStep >= units) release();
                    if constexpr (C::WIDE_STORES) {
                        // the four lanes of a quad hold, per row, one word (two columns) of each 8-column
                        // block; a 4 x 4 transpose across the quad (two shuffle stages) gives each lane a
                        // whole block of a row, written with one 16-byte store; a trailing pair of blocks
                        // (head_dim 80) swaps one word between the lanes of a pair for 8-byte stores
                        static_assert(DN % NC == 0 && NC % 2 == 0, "whole chunks of paired blocks");
                        const bool lo = tig & 1, hi = tig & 2;
                        __nv_bfloat16 *row0 = oh + (int64_t)(seg0 + r0) * out_stride;
                        __nv_bfloat16 *row1 = oh + (int64_t)(seg0 + r1) * out_stride;
                        // x[i]: this lane's word of block j + i in one row; returns the words of block
                        // j + tig in column order
                        auto transpose4 = [&](uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
                            // lanes two apart swap halves: keep the columns of block pair `hi`
                            const uint32_t k0 = hi ? x2 : x0, k1 = hi ? x3 : x1;
                            const uint32_t g0 = __shfl_xor_sync(0xffffffffu, hi ? x0 : x2, 2);
                            const uint32_t g1 = __shfl_xor_sync(0xffffffffu, hi ? x1 : x3, 2);
                            // neighbours swap: z[m] = word of lane tig ^ m for block j + tig
                            const uint32_t z1 = __shfl_xor_sync(0xffffffffu, lo ? k0 : k1, 1);
                            const uint32_t z3 = __shfl_xor_sync(0xffffffffu, lo ? g0 : g1, 1);
                            const uint32_t z0 = lo ? k1 : k0, z2 = lo ? g1 : g0;
                            // y[e] = z[e ^ tig]
                            const uint32_t w0 = lo ? z1 : z0, w1 = lo ? z0 : z1, w2 = lo ? z3 : z2, w3 = lo ? z2 : z3;
                            return hi ? make_uint4(w2, w3, w0, w1) : make_uint4(w0, w1, w2, w3);
                        };
#pragma unroll
                        for (int j = 0; j + 4 <= NC; j += 4) {
                            uint32_t x[2][4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                x[0][i] = pack_bf16(o[j + i][0] * inv0, o[j + i][1] * inv0);
                                x[1][i] = pack_bf16(o[j + i][2] * inv1, o[j + i][3] * inv1);
                            }
                            const uint4 y0 = transpose4(x[0][0], x[0][1], x[0][2], x[0][3]);
                            const uint4 y1 = transpose4(x[1][0], x[1][1], x[1][2], x[1][3]);
                            const int col = (c0 + j + tig) * 8;
                            if (r0 < L) *reinterpret_cast<uint4 *>(row0 + col) = y0;
                            if (r1 < L) *reinterpret_cast<uint4 *>(row1 + col) = y1;
                        }
                        if constexpr (NC % 4 == 2) {
                            constexpr int j = NC - 2;
                            const uint32_t a0 = pack_bf16(o[j][0] * inv0, o[j][1] * inv0);
                            const uint32_t a1 = pack_bf16(o[j][2] * inv1, o[j][3] * inv1);
                            const uint32_t b0 = pack_bf16(o[j + 1][0] * inv0, o[j + 1][1] * inv0);
                            const uint32_t b1 = pack_bf16(o[j + 1][2] * inv1, o[j + 1][3] * inv1);
                            const uint32_t t0 = __shfl_xor_sync(0xffffffffu, lo ? a0 : b0, 1);
                            const uint32_t t1 = __shfl_xor_sync(0xffffffffu, lo ? a1 : b1, 1);
                            const int col = (c0 + j + (lo ? 1 : 0)) * 8 + (tig & 2) * 2;
                            if (r0 < L)
                                *reinterpret_cast<uint2 *>(row0 + col) = lo ? make_uint2(t0, b0) : make_uint2(a0, t0);
                            if (r1 < L)
                                *reinterpret_cast<uint2 *>(row1 + col) = lo ? make_uint2(t1, b1) : make_uint2(a1, t1);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < NC; ++j) {
                            if (c0 + j < DN) {
                                const int col = (c0 + j) * 8 + tig * 2;
                                if (r0 < L)
                                    *reinterpret_cast<uint32_t *>(oh + (int64_t)(seg0 + r0) * out_stride + col) =
                                        pack_bf16(o[j][0] * inv0, o[j][1] * inv0);
                                if (r1 < L)
                                    *reinterpret_cast<uint32_t *>(oh + (int64_t)(seg0 + r1) * out_stride + col) =
                                        pack_bf16(o[j][2] * inv1, o[j][3] * inv1);
                            }
                        }
                    }
                }
            };
            if constexpr (C::PER_N16) {
                switch (n16) {
                case 1: unit(std::integral_constant<int, 1>{}); break;
                case 2: unit(std::integral_constant<int, 2>{}); break;
                case 3: unit(std::integral_constant<int, 3>{}); break;
                default: unit(std::integral_constant<int, 4>{}); break;
                }
            } else {
                unit(std::integral_constant<int, 0>{});
            }
        }
    }
}

template <int D, int HG>
cudaError_t launch_hg(const AttnArgs &a, int64_t max_items, int num_sms, cudaStream_t stream)
{
    using C = TinyCfg<D, false, HG>;
    using CF = TinyCfg<D, true, HG>;                     // the variant that rotates raw Q
    const size_t smem = a.fuse_q ? CF::SMEM : C::SMEM;
    static_assert(C::SMEM + sizeof(TinyShared) <= 227 * 1024 && CF::SMEM + sizeof(TinyShared) <= 227 * 1024,
                  "shared memory budget");
    // [T, H*D] rows seen as {W elements, H*D/W chunks, T rows}; boxes of {W, CHUNKS, 16}
    if ((int64_t)a.H * D % C::W != 0) return cudaErrorInvalidValue;
    CUtensorMap maps[3];
    const void *ptrs[3] = {a.q, a.k, a.v};
    const int64_t strides[3] = {a.q_stride, a.k_stride, a.v_stride};
    for (int t = 0; t < 3; ++t) {
        const uint64_t dims[3] = {(uint64_t)C::W, (uint64_t)a.H * D / C::W, (uint64_t)(a.T > 0 ? a.T : 1)};
        const uint64_t st[2] = {(uint64_t)C::W * 2, (uint64_t)strides[t] * 2};
        const uint32_t box[3] = {(uint32_t)C::W, (uint32_t)C::CHUNKS, 16u};
        if (!encode_tiled_map(&maps[t], ptrs[t], 3, dims, st, box, C::W * 2)) return cudaErrorInvalidValue;
    }
    auto kern = a.fuse_q ? attn_tiny_kernel<D, true, HG> : attn_tiny_kernel<D, false, HG>;
    const int threads = a.fuse_q ? CF::THREADS : C::THREADS;
    static DeviceOnce once[2];                           // per fused-Q variant
    cudaError_t e = once[a.fuse_q ? 1 : 0].run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    const int64_t items = max_items / HG;
    const unsigned blocks = (unsigned)(items < num_sms ? items : num_sms);   // one CTA per SM
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("attn_tiny", stream);
    kern<<<blocks, threads, smem, stream>>>(maps[0], maps[1], maps[2], static_cast<__nv_bfloat16 *>(a.out),
                                            a.out_stride, a.lse, a.H, a.scale_log2, a.hdr, a.items, a.status, a.qr);
    return cudaGetLastError();
}

// Heads per item: as many as make the copied rows wide (several heads side by side) while the
// row still falls under a conflict-free swizzle, and divide the head count. Four at head_dim 80
// when no segment can exceed 24 tokens (an item is then at most 61 KB; measured 1.6x faster
// than two on 4-16-token images and 1.1x on 9-24-token ones, even at 17-32 tokens and slower
// on 16-64-token ones, whose items would leave the ring room for two).
template <int D>
cudaError_t launch_d(const AttnArgs &a, int64_t max_items, int num_sms, cudaStream_t stream)
{
    if constexpr (D == 80) {
        if (a.H % 4 == 0 && a.max_len <= 24) return launch_hg<D, 4>(a, max_items, num_sms, stream);
    }
    if constexpr (D == 32 || D == 80 || D == 96) {
        if (a.H % 2 == 0) return launch_hg<D, 2>(a, max_items, num_sms, stream);
    }
    return launch_hg<D, 1>(a, max_items, num_sms, stream);
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
