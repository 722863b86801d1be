// Long-segment varlen attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Same result as the tiny-segment kernel: for each (segment, head) the plain
// softmax(scale * q k^T) v over that segment's keys only (vLLM Dots
// vision_attention page, VisionAttentionV2.forward / VisionAttention.forward
// with its block-diagonal mask), softmax in fp32, P rounded to bf16 for the
// P.V product, fp32 accumulation in TMEM, bf16 output.
//
// One work item = (segment, head, 256 query rows) = two 128-row Q tiles that
// share every K/V tile the TMA warp streams in; or, flagged split, (segment,
// head, 128 query rows): one Q tile whose key tiles alternate between the two
// halves of the CTA, which merge their partial results at the end (the
// segment's last block when it has at most 128 rows, and every block of a
// batch too small to occupy the GPU otherwise). Persistent CTAs (one per SM)
// take the scheduler's longest-first list in order: each CTA its own index
// first, then the next unclaimed item from a device counter, which the
// producer passes to the other roles through a small shared-memory item ring
// (CTAs that draw short items take more of them). Three warpgroups (384 threads,
// launched at 168 registers; setmaxnreg lowers the control warpgroup to 88
// and raises the two softmax warpgroups to 208, or 96 and 200 in the variant
// that rotates raw Q in warp 3):
//   warp 0      TMA producer: Q tiles per item, K and V tiles into a ring of
//               STAGES slots, each tile's V after the next tile's K. Q and K
//               in 64-column slabs with 128-byte swizzle plus a 16- or
//               32-column remainder slab (wide boxes stream faster); V in
//               16-column slabs with 32-byte swizzle (the P.V operand's N is
//               the head dim, whole swizzle atoms per instruction).
//   warp 1      TMEM owner; lane 0 issues the MMAs of Q tile 0
//   warp 2      lane 0 issues the MMAs of Q tile 1
//                 S_i = Q_i K^T     (SS MMA, M=128, N=BN, K=D)   into TMEM
//                 O_i += P V        (TS MMA, A=P from TMEM, B=V MN-major)
//               each issuer orders QK(j+1) before PV(j), so S of the next key
//               tile is computed while its softmax group turns S into P.
//   warp 3      idle (completes the control warpgroup); when Q arrives raw, it
//               normalises and rotates each Q pair in shared memory between
//               the TMA landing and the first MMA (fence to the async proxy,
//               then q_ready), one row per lane at a time
//   warps 4-7   softmax group 0 (tile 0), one TMEM lane = one query row per
//   warps 8-11  softmax group 1 (tile 1)  thread: row max, lazy rescaling of
//               O (only when the max grows by more than 2^8), exp2 with the
//               scale folded in, row sum, P -> bf16 into the tile's own P
//               region of TMEM, and the epilogue O / l -> bf16 -> HBM (for a
//               split item, both groups combine O0 and O1 with their maxima
//               and sums, each writing half of the head's columns).
// TMEM (512 columns): S0 | S1 | O0 | O1 | P0 | P1; the key tile BN is the
// largest that fits (128 for head_dim <= 64, 112 for 80, 96 for 96, 80 for
// 128), so the two tiles never wait for each other. Keys past the segment end are
// masked to -inf; the last tile of a segment that ends inside it runs only the
// 16-key steps holding its keys, with the leftover V rows zeroed, so no value
// outside the segment (finite or not) enters a result; query rows past it are
// never stored, rows past T are zero-filled by TMA. Template switches add the
// per-row log-sum-exp store (LSE) and the Q rotation in warp 3 (FQ) without
// touching the plain kernel's code. Every wait is bounded; a wait that expires
// sets VIT_ERR_TIMEOUT, and all roles drain and free TMEM before exiting.
#include <cudaTypedefs.h>

#include <type_traits>

#include "internal.h"
#include "sm100.cuh"

namespace vit {
namespace {

using namespace sm100;

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;              // 65536 / 384, rounded down to a multiple of 8
constexpr int kCtrlRegs = 88;                 // control warpgroup after setmaxnreg.dec
constexpr int kSoftmaxRegs = 208;             // softmax warpgroups after setmaxnreg.inc
// the variant that rotates raw Q in warp 3 gives the control warpgroup more room
constexpr int kCtrlRegsFQ = 96;
constexpr int kSoftmaxRegsFQ = 200;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split exceeds the launch pool");
static_assert(128 * kCtrlRegsFQ + 256 * kSoftmaxRegsFQ <= kThreads * kLaunchRegs, "register split exceeds the launch pool");
constexpr int BM = 128;                       // rows per Q tile; two tiles per item
constexpr long long kWaitBudget = 4000000000ll;   // clock cycles before a wait gives up (~2 s)
constexpr int kMaxStages = 4;                 // K/V ring slots the barrier arrays hold
constexpr int kItemRing = 4;                  // items the producer may publish ahead of the other roles
constexpr int kItemReaders = 11;              // the two issuers, warp 3 and the eight softmax warps

template <int D> struct LongCfg {
    // keys per tile: the largest multiple of 16 (at most 128) with S0, S1 (BN columns each),
    // O0, O1 (D each) and separate P0, P1 (BN/2 each) inside the 512 TMEM columns
    static constexpr int BN = ((512 - 2 * D) / 3 / 16 * 16 > 128) ? 128 : (512 - 2 * D) / 3 / 16 * 16;
    // K/V ring of 3 slots; the next item's Q pair is prefetched into a second Q buffer where that
    // fits in shared memory (every head dim but 128: there a third K/V slot measured 1.8 % faster
    // than a second Q buffer, since a K tile lands thousands of cycles after its copy is issued)
    static constexpr int STAGES = 3;
    // Q and K (K-major operands of QK) sit in 64-column slabs with 128-byte swizzle, the columns
    // past the last multiple of 64 (16 or 32) in one slab with 32- or 64-byte swizzle: a wide TMA box
    // moves a tile at about 1.6x the rate of 16-column boxes. V (the MN-major operand of P.V, whose
    // N = head_dim must be whole swizzle atoms in one instruction) keeps 16-column slabs.
    static constexpr int N128 = D / 64;                     // 64-column slabs
    static constexpr int REM = D % 64;                      // columns of the remainder slab: 0, 16, 32
    static constexpr int REM_SW = REM == 32 ? 64 : 32;      // its swizzle width in bytes
    static constexpr int NK = D / 16;                       // K steps of QK (16 columns each)
    static constexpr int Q_SLAB128 = BM * 128;
    static constexpr int K_SLAB128 = BN * 128;
    static constexpr int Q_TILE = BM * D * 2;
    static constexpr int K_TILE = BN * D * 2;
    static constexpr int K_STRIDE = (K_TILE + 1023) / 1024 * 1024;   // ring slots stay 1024-aligned
    static constexpr int NSLAB = D / 16;                    // 16-column slabs of a V tile
    static constexpr int KV_SLAB = BN * 32;                 // bytes of one 16-column V slab
    static constexpr int KV_TILE = NSLAB * KV_SLAB;         // bytes of one V tile
    static constexpr int QBUF = (4 * Q_TILE + STAGES * (K_STRIDE + KV_TILE) + 1024 <= 227 * 1024) ? 2 : 1;
    static constexpr int OFF_Q = 0;                        // QBUF buffers x two tiles
    static constexpr int OFF_K = OFF_Q + QBUF * 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + STAGES * K_STRIDE;
    static constexpr int DATA = OFF_V + STAGES * KV_TILE;
    // > half of the SM's shared memory: exactly one CTA (one TMEM owner) per SM
    static constexpr int SMEM = (DATA + 1024 > 118 * 1024) ? DATA + 1024 : 118 * 1024;
    // TMEM columns
    // TMEM columns; every region starts on a 16-column boundary, P1 on an 8-column one,
    // and every TMEM access below is naturally aligned to its own width
    static constexpr int TS0 = 0, TS1 = BN, TO0 = 2 * BN, TO1 = 2 * BN + D, TP0 = 2 * BN + 2 * D;
    static constexpr int TP1 = (TP0 + BN / 2 + 7) / 8 * 8;
    static_assert(TP1 + BN / 2 <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory per block (227 KB opt-in limit)");
    static_assert(STAGES >= 2 && STAGES <= kMaxStages, "ring slots the barrier arrays hold");
    static_assert(D % 16 == 0 && BN % 16 == 0 && (BN / 2) % 8 == 0, "tile shapes");
    static_assert(Q_TILE % 1024 == 0 && K_SLAB128 % 1024 == 0 && OFF_V % 1024 == 0,
                  "128-byte-swizzle slabs start on 1024-byte boundaries");
    // byte offset of K step kk (16 columns) inside a Q or K tile of `rows` rows, and whether it
    // lies in a 128-byte-swizzle slab (else in the remainder slab)
    __host__ __device__ static constexpr bool wide_step(int kk) { return kk < 4 * N128; }
    __host__ __device__ static constexpr int step_off(int kk, int rows)
    {
        return wide_step(kk) ? (kk / 4) * rows * 128 + (kk % 4) * 32 : N128 * rows * 128 + (kk - 4 * N128) * 32;
    }
};

// Shared-memory matrix descriptor of a K-major operand slab: 128-byte swizzle (8-row groups of
// 1024 B) for the 64-column slabs, the remainder slab's own swizzle otherwise.
template <int SW> __device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr)
{
    static_assert(SW == 128 || SW == 64 || SW == 32, "swizzle width");
    return smem_desc(addr, 16, 8 * SW, SW == 128 ? 2 : (SW == 64 ? 4 : 6));
}

struct Bars {
    uint64_t q_full[2], q_empty[2], q_ready[2];
    uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages], v_empty[kMaxStages];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_free[2];
    uint64_t drain[2];
    uint64_t merge;          // split items: the eight softmax warps meet twice at the item's end
    uint64_t item_full[kItemRing], item_empty[kItemRing];   // the producer's item ring
};

__device__ __forceinline__ uint32_t bar_addr(const uint64_t &b) { return smem_addr(&b); }

// P.V of the last tile of a segment that ends inside the tile: only the 16-key steps that hold a
// key of the segment, with the rows of the last step past the segment's end zeroed first. Those
// rows get P = 0, but 0 * (Inf or NaN) is NaN, so without this a non-finite value in the next
// segment or in padding would reach this segment's output. V has landed (v_full) when this runs,
// and both issuers write the same zeros, so their order does not matter. Called only from the copy
// of the issuer's tile step that follows its loop over full tiles (inlined there: measured as fast
// as before on the full tiles, where an out-of-line call was 0.5 % slower).
template <int NSLAB, int SLAB, int D>
__device__ __forceinline__ void pv_tail(uint32_t tO, uint32_t tP, uint64_t dv, unsigned char *vt, uint32_t acc,
                                     int kv_valid, uint32_t bar_done)
{
    constexpr uint32_t ID_PV = idesc_bf16(128, D, 0, 1);
    const int n16 = (kv_valid + 15) >> 4;
    if (kv_valid & 15) {
        for (int r = kv_valid; r < 16 * n16; ++r)
            for (int s = 0; s < NSLAB; ++s) {
                uint4 *p = reinterpret_cast<uint4 *>(vt + s * SLAB + 32 * r);
                p[0] = make_uint4(0u, 0u, 0u, 0u);
                p[1] = make_uint4(0u, 0u, 0u, 0u);
            }
        fence_proxy_async_smem();
    }
    for (int kk = 0; kk < n16; ++kk)
        mma_ts(tO, tP + kk * 8, dv + (uint64_t)(kk * (512 >> 4)), ID_PV, kk > 0 ? 1u : acc);
    mma_commit(bar_done);
}

template <int D, bool LSE, bool FQ>
__global__ void __launch_bounds__(kThreads, 1)
attn_long_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kr,
                 const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ out, int64_t out_stride,
                 float *__restrict__ lse, int H, float scale_log2, WsHeader *__restrict__ hdr,
                 const Item *__restrict__ items, int32_t *status, int stall_v, const rope::QRope qr)
{
    using C = LongCfg<D>;
    constexpr int BN = C::BN, ST = C::STAGES, NSLAB = C::NSLAB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ Bars bars;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ float s_m[2][BM], s_l[2][BM];   // split items: each half's running max and row sum per row
    __shared__ Item s_items[kItemRing];        // the item ring (y < 0: the end of this CTA's list)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = hdr->n_long;                   // read by the producer; the others take items from it

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(bars.q_full[b]), 1);
            mbar_init(bar_addr(bars.q_empty[b]), 2);     // one commit from each MMA issuer
            mbar_init(bar_addr(bars.q_ready[b]), 1);     // warp 3 after rotating raw Q
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_addr(bars.k_full[s]), 1);
            mbar_init(bar_addr(bars.v_full[s]), 1);
            mbar_init(bar_addr(bars.k_empty[s]), 2);     // one commit from each MMA issuer after its QK
            mbar_init(bar_addr(bars.v_empty[s]), 2);     // and after its P.V
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(bars.s_full[i]), 1);
            mbar_init(bar_addr(bars.s_free[i]), 4);
            mbar_init(bar_addr(bars.p_full[i]), 4);
            mbar_init(bar_addr(bars.pv_done[i]), 1);
            mbar_init(bar_addr(bars.o_free[i]), 4);
        }
        mbar_init(bar_addr(bars.drain[0]), 1);
        mbar_init(bar_addr(bars.drain[1]), 1);
        mbar_init(bar_addr(bars.merge), 8);
        for (int r = 0; r < kItemRing; ++r) {
            mbar_init(bar_addr(bars.item_full[r]), 1);
            mbar_init(bar_addr(bars.item_empty[r]), kItemReaders);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    auto fail = [&]() {
        if (!s_abort) {
            s_abort = 1;
            report_error(status, VIT_ERR_TIMEOUT);
        }
    };
    auto wait = [&](const uint64_t &b, uint32_t parity) -> bool {
        if (mbar_wait(bar_addr(b), parity, (const volatile int *)&s_abort, kWaitBudget)) return true;
        fail();
        return false;
    };
    // softmax warps run warp-collective tcgen05.ld/st after their waits: all 32 lanes
    // either go on together or give up together
    auto wait_warp = [&](const uint64_t &b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(b, parity)) != 0;
    };
    // The k-th item of this CTA from the producer's ring: false at the end of the list or when a
    // wait gave up. Called by one thread (issuers) or by a whole warp (warp_wide); one arrival per
    // caller frees the slot once its item has been copied out.
    auto take_item = [&](uint32_t k, Item &x, bool warp_wide, bool &ok_) -> bool {
        const uint32_t slot = k % kItemRing, par = (k / kItemRing) & 1;
        if (!(ok_ = warp_wide ? wait_warp(bars.item_full[slot], par) : wait(bars.item_full[slot], par))) return false;
        x = s_items[slot];
        if (warp_wide) __syncwarp();
        if (!warp_wide || lane == 0) mbar_arrive(bar_addr(bars.item_empty[slot]));
        return x.y >= 0;
    };

    if (warp < 4) regs_dec<FQ ? kCtrlRegsFQ : kCtrlRegs>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_qr);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_kr);
            tma_prefetch_desc(&tm_v);
            // one Q or K tile: its 64-column slabs (128-byte swizzle), then the remainder slab
            auto load_qk_tile = [&](unsigned char *dst, const CUtensorMap *wide, const CUtensorMap *rem, int rows,
                                    int head, int row, uint32_t bar) {
#pragma unroll
                for (int s = 0; s < C::N128; ++s)
                    tma_load_2d(smem_addr(dst + s * rows * 128), wide, head * D + 64 * s, row, bar);
                if constexpr (C::REM > 0)
                    tma_load_2d(smem_addr(dst + C::N128 * rows * 128), rem, head * D + 64 * C::N128, row, bar);
            };
            uint32_t g = 0, q_it = 0;
            // parity + 1 of the last load issued on each barrier (0 = none), for the abort drain;
            // two bits per stage, kept in registers
            uint32_t q_pend = 0, k_pend = 0, v_pend = 0;     // q_pend: two bits per Q buffer
            bool ok = true;
            // a split item has one Q tile, the other items two
            auto load_q = [&](uint32_t qb, uint32_t qn, int q0, int head, bool split) {
                const int nt = split ? 1 : 2;
                mbar_arrive_expect_tx(bar_addr(bars.q_full[qb]), nt * C::Q_TILE);
                for (int i = 0; i < nt; ++i)
                    load_qk_tile(base + C::OFF_Q + (2 * qb + i) * C::Q_TILE, &tm_q, &tm_qr, BM, head, q0 + BM * i,
                                 bar_addr(bars.q_full[qb]));
                q_pend = (q_pend & ~(3u << (2 * qb))) | (((qn & 1) + 1) << (2 * qb));
            };
            // K and V of a tile go into separate halves of a ring slot: a slot's K half is free once
            // its QK has completed, its V half only once its P.V has. So each tile's V is issued
            // after the next tile's K: that K load waits on an earlier event than this V load would,
            // and the K of the tile after next reaches shared memory well before its QK.
            uint32_t v_g = 0;                                // pending V: ring index, first row, head
            int v_row = -1, v_head = 0;
            auto load_v = [&]() -> bool {
                const int st = v_g % ST;
                if (v_g >= (uint32_t)ST && !(ok = wait(bars.v_empty[st], (v_g / ST - 1) & 1))) return false;
                if (stall_v) return true;       // test hook: V never arrives, the MMA wait expires
                mbar_arrive_expect_tx(bar_addr(bars.v_full[st]), C::KV_TILE);
                for (int s = 0; s < NSLAB; ++s)
                    tma_load_2d(smem_addr(base + C::OFF_V + st * C::KV_TILE + s * C::KV_SLAB), &tm_v,
                                v_head * D + 16 * s, v_row, bar_addr(bars.v_full[st]));
                v_pend = (v_pend & ~(3u << (2 * st))) | ((((v_g / ST) & 1) + 1) << (2 * st));
                return true;
            };
            // raw Q needs time for warp 3 to rotate it, so with two Q buffers the next item's Q
            // goes out as soon as its buffer is free rather than after this item's last K/V tile
            bool q_early = false;                            // Q of item q_it already issued
            // Items: the CTA's first is its block index; each later one is taken from a device-wide
            // counter, so a CTA that finishes early takes the next item of the longest-first list
            // (greedy list scheduling). Each is published to the other roles through the ring.
            uint32_t k_pub = 0;
            auto publish = [&](const Item &x) -> bool {
                const uint32_t slot = k_pub % kItemRing;
                if (k_pub >= kItemRing && !(ok = wait(bars.item_empty[slot], (k_pub / kItemRing - 1) & 1)))
                    return false;
                s_items[slot] = x;
                mbar_arrive(bar_addr(bars.item_full[slot]));
                ++k_pub;
                return true;
            };
            const Item kEnd = make_int4(0, -1, 0, 0);
            int it = blockIdx.x;
            Item item = it < n_items ? items[it] : kEnd;
            for (; ok && it < n_items; ++q_it) {
                if (!publish(item)) break;
                const int it_next = (int)gridDim.x + atomicAdd(&hdr->next_long, 1);
                const Item nx = it_next < n_items ? items[it_next] : kEnd;
                const int seg0 = item.x, seg_len = item.y, q0 = item.z, head = item_head(item);
                const int n_kv = (seg_len + BN - 1) / BN;
                // Q pairs alternate between two buffers, so the next item's Q is loaded while
                // the current item still runs
                const uint32_t qb = q_it % C::QBUF, qn = q_it / C::QBUF;   // buffer, its use count
                if (!q_early) {
                    if (qn > 0 && !(ok = wait(bars.q_empty[qb], (qn - 1) & 1))) break;
                    load_q(qb, qn, q0, head, item_split(item));
                }
                q_early = false;
                for (int j = 0; j < n_kv; ++j, ++g) {
                    if constexpr (FQ && C::QBUF == 2) {
                        if (!q_early && it_next < n_items) {
                            const uint32_t qb1 = (q_it + 1) & 1, qn1 = (q_it + 1) >> 1;
                            if (qn1 == 0 || mbar_test(bar_addr(bars.q_empty[qb1]), (qn1 - 1) & 1)) {
                                load_q(qb1, qn1, nx.z, item_head(nx), item_split(nx));
                                q_early = true;
                            }
                        }
                    }
                    const int st = g % ST;
                    if (g >= (uint32_t)ST && !(ok = wait(bars.k_empty[st], (g / ST - 1) & 1))) break;
                    const int row = seg0 + j * BN;
                    mbar_arrive_expect_tx(bar_addr(bars.k_full[st]), C::K_TILE);
                    load_qk_tile(base + C::OFF_K + st * C::K_STRIDE, &tm_k, &tm_kr, BN, head, row,
                                 bar_addr(bars.k_full[st]));
                    k_pend = (k_pend & ~(3u << (2 * st))) | ((((g / ST) & 1) + 1) << (2 * st));
                    if (v_row >= 0 && !load_v()) break;
                    v_g = g;
                    v_row = row;
                    v_head = head;
                }
                it = it_next;
                item = nx;
            }
            if (ok && v_row >= 0) load_v();                 // the last tile's V
            if (ok) publish(kEnd);                           // the other roles stop at this entry
            if (!ok) {
                // let every copy already issued land before this CTA's shared memory is released
                // (loads that completed earlier return at once; short budget, abort flag ignored)
                const int never = 0;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint32_t qp = (q_pend >> (2 * b)) & 3u;
                    if (qp) mbar_wait(bar_addr(bars.q_full[b]), qp - 1, &never, 20000000ll);
                }
#pragma unroll
                for (int s = 0; s < ST; ++s) {
                    const uint32_t kp = (k_pend >> (2 * s)) & 3u, vp = (v_pend >> (2 * s)) & 3u;
                    if (kp) mbar_wait(bar_addr(bars.k_full[s]), kp - 1, &never, 20000000ll);
                    if (vp) mbar_wait(bar_addr(bars.v_full[s]), vp - 1, &never, 20000000ll);
                }
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues every MMA of Q tile 0, warp 2 every MMA of Q tile 1. A single issuer's
        // serial chain (barrier checks of ~100 cycles each, fences, commits, the MMAs) per key
        // tile is about as long as the tensor work of that tile at head_dim 80, so one thread
        // per tile halves it. Descriptors are precomputed 64-bit bases plus compile-time offsets
        // (the address field is the low 14 bits and never carries); every barrier parity derives
        // from one global key-tile counter. The two issuers share nothing but the K/V stage
        // barriers (two-arrival k_empty / v_empty / q_empty); each softmax group rewrites its tile's P
        // region only after that tile's previous P.V has completed.
        if (lane == 0) {
            const int ti = warp - 1;                              // Q tile of this issuer
            constexpr uint32_t ID_QK = idesc_bf16(128, BN, 0, 0);
            constexpr uint32_t ID_PV = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t STAGE_STEP = C::KV_TILE >> 4;         // V ring slot, descriptor units
            constexpr uint32_t K_STEP = C::K_STRIDE >> 4;             // K ring slot
            const uint32_t tS = tmem + (ti ? C::TS1 : C::TS0);
            const uint32_t tO = tmem + (ti ? C::TO1 : C::TO0);
            const uint32_t tP = tmem + (ti ? C::TP1 : C::TP0);
            // descriptor bases (128-byte-swizzle form and remainder form) of this issuer's Q tile, of
            // tile 0 (split items), and of K ring slot 0; K steps add their offsets in 16-byte units
            const uint32_t a_q = smem_addr(base + C::OFF_Q), a_k = smem_addr(base + C::OFF_K);
            const uint64_t dqw_own = kmajor_desc<128>(a_q + ti * C::Q_TILE);
            const uint64_t dqr_own = kmajor_desc<C::REM_SW>(a_q + ti * C::Q_TILE);
            const uint64_t dqw_tile0 = kmajor_desc<128>(a_q), dqr_tile0 = kmajor_desc<C::REM_SW>(a_q);
            const uint64_t dkw0 = kmajor_desc<128>(a_k), dkr0 = kmajor_desc<C::REM_SW>(a_k);
            const uint64_t dv0 = smem_desc(smem_addr(base + C::OFF_V), C::KV_SLAB, 256, 6);
            const uint64_t &b_sfree = bars.s_free[ti], &b_pfull = bars.p_full[ti], &b_ofree = bars.o_free[ti];
            const uint32_t a_sfull = bar_addr(bars.s_full[ti]), a_pvdone = bar_addr(bars.pv_done[ti]);
            // t: key tiles this CTA has passed through the K/V ring (every one, own or not: stage
            // and phase of each); c: S tiles this issuer has computed (parity of s_free, p_full)
            uint32_t t = 0, c = 0, item_cnt = 0;
            bool ok = true;

            // S = Q K^T over the K steps: each step's A and B descriptors in the form of its slab
            auto qk = [&](uint64_t dqw, uint64_t dqr, uint64_t dkw, uint64_t dkr) {
#pragma unroll
                for (int kk = 0; kk < C::NK; ++kk) {
                    const uint64_t a = (C::wide_step(kk) ? dqw : dqr) + (uint64_t)(C::step_off(kk, BM) >> 4);
                    const uint64_t b = (C::wide_step(kk) ? dkw : dkr) + (uint64_t)(C::step_off(kk, BN) >> 4);
                    mma_ss(tS, a, b, ID_QK, kk > 0 ? 1u : 0u);
                }
                mma_commit(a_sfull);
            };
            auto pv = [&](uint64_t dv, uint32_t acc) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tO, tP + kk * 8, dv + (uint64_t)(kk * (512 >> 4)), ID_PV, kk > 0 ? 1u : acc);
                mma_commit(a_pvdone);
            };

            for (Item item; take_item(item_cnt, item, false, ok); ++item_cnt) {
                const int n_kv = (item.y + BN - 1) / BN;
                const int n_full = item.y / BN;                  // tiles with BN keys of the segment
                uint32_t st = t % ST, ph = (t / ST) & 1;
                const uint32_t qb = item_cnt % C::QBUF;         // Q buffer of this item
                if (!(ok = wait(FQ ? bars.q_ready[qb] : bars.q_full[qb], (item_cnt / C::QBUF) & 1))) break;
                if (!item_split(item)) {
                    const uint64_t qoff = qb * ((2 * C::Q_TILE) >> 4);
                    const uint64_t dqw = dqw_own + qoff, dqr = dqr_own + qoff;
                    // prologue: S of the item's first key tile
                    if (!(ok = wait(bars.k_full[st], ph))) break;
                    if (c > 0 && !(ok = wait(b_sfree, (c - 1) & 1))) break;
                    tc_fence_after();
                    qk(dqw, dqr, dkw0 + st * K_STEP, dkr0 + st * K_STEP);
                    mma_commit(bar_addr(bars.k_empty[st]));
                    if (n_kv == 1) mma_commit(bar_addr(bars.q_empty[qb]));
                    // one key tile: QK of the next tile, then P.V of this one; the tail variant (the
                    // last tile of a segment that ends inside it) is a separate copy after the loop,
                    // so the loop over full tiles carries no test for it
                    auto step = [&](int j, auto tail) -> bool {
                        const uint32_t u = c + j;                 // this issuer's S count of this tile
                        const uint32_t st1 = (st + 1 == (uint32_t)ST) ? 0u : st + 1;
                        const uint32_t ph1 = (st + 1 == (uint32_t)ST) ? ph ^ 1u : ph;
                        if (j + 1 < n_kv) {                        // next tile's S as soon as this S was read
                            if (!(ok = wait(bars.k_full[st1], ph1))) return false;
                            if (!(ok = wait(b_sfree, u & 1))) return false;
                            tc_fence_after();
                            qk(dqw, dqr, dkw0 + st1 * K_STEP, dkr0 + st1 * K_STEP);
                            mma_commit(bar_addr(bars.k_empty[st1]));
                            if (j + 2 == n_kv) mma_commit(bar_addr(bars.q_empty[qb]));
                        }
                        if (!(ok = wait(bars.v_full[st], ph))) return false;
                        if (j == 0 && item_cnt > 0 && !(ok = wait(b_ofree, (item_cnt - 1) & 1))) return false;
                        if (!(ok = wait(b_pfull, u & 1))) return false;
                        tc_fence_after();
                        if constexpr (decltype(tail)::value)
                            pv_tail<NSLAB, C::KV_SLAB, D>(tO, tP, dv0 + st * STAGE_STEP,
                                                          base + C::OFF_V + st * C::KV_TILE, j > 0 ? 1u : 0u,
                                                          item.y - j * BN, a_pvdone);
                        else
                            pv(dv0 + st * STAGE_STEP, j > 0 ? 1u : 0u);
                        mma_commit(bar_addr(bars.v_empty[st]));
                        st = st1;
                        ph = ph1;
                        return true;
                    };
                    for (int j = 0; j < n_full; ++j)
                        if (!step(j, std::false_type{})) break;
                    if (ok && n_full < n_kv) step(n_full, std::true_type{});
                    t += n_kv;
                    c += n_kv;
                    continue;
                }
                // Split item: one Q tile (tile 0 of the buffer), this issuer takes the key tiles
                // j = ti, ti + 2, ...; it still waits for the K and V of every tile as they pass, so
                // that each of its parity waits is at most one phase ahead of its barrier.
                const uint64_t qoff = qb * ((2 * C::Q_TILE) >> 4);
                const uint64_t dqw = dqw_tile0 + qoff, dqr = dqr_tile0 + qoff;
                int prev_j = -1;                                  // own tile whose P.V is pending
                uint32_t prev_st = 0, prev_ph = 0, prev_c = 0;
                bool first_pv = true;
                auto pv_of_prev = [&]() -> bool {
                    if (!(ok = wait(bars.v_full[prev_st], prev_ph))) return false;
                    if (first_pv && item_cnt > 0 && !(ok = wait(b_ofree, (item_cnt - 1) & 1))) return false;
                    if (!(ok = wait(b_pfull, prev_c & 1))) return false;
                    tc_fence_after();
                    const uint32_t acc = first_pv ? 0u : 1u;
                    if (prev_j < n_full)
                        pv(dv0 + prev_st * STAGE_STEP, acc);
                    else
                        pv_tail<NSLAB, C::KV_SLAB, D>(tO, tP, dv0 + prev_st * STAGE_STEP,
                                                      base + C::OFF_V + prev_st * C::KV_TILE, acc,
                                                      item.y - prev_j * BN, a_pvdone);
                    mma_commit(bar_addr(bars.v_empty[prev_st]));
                    first_pv = false;
                    return true;
                };
                // as in the two-tile path, the next own tile's QK goes out before the pending P.V: its
                // K half of the ring slot is released by QKs only, never by a P.V
                // the other issuer's tiles: this issuer passes each phase of their K and V as well
                // and adds its arrival to the slot's release, so the producer never refills a slot
                // this issuer has not yet seen (its V phase is taken after this issuer's next QK)
                bool skip_v = false;
                uint32_t skip_st = 0, skip_ph = 0;
                auto pass_skipped_v = [&]() -> bool {
                    if (!skip_v) return true;
                    if (!(ok = wait(bars.v_full[skip_st], skip_ph))) return false;
                    mbar_arrive(bar_addr(bars.v_empty[skip_st]));
                    skip_v = false;
                    return true;
                };
                for (int j = 0; j < n_kv; ++j) {
                    if ((j & 1) != ti) {
                        if (!(ok = wait(bars.k_full[st], ph))) break;
                        mbar_arrive(bar_addr(bars.k_empty[st]));
                        skip_v = true;
                        skip_st = st;
                        skip_ph = ph;
                    } else {
                        if (!(ok = wait(bars.k_full[st], ph))) break;
                        if (c > 0 && !(ok = wait(b_sfree, (c - 1) & 1))) break;
                        tc_fence_after();
                        qk(dqw, dqr, dkw0 + st * K_STEP, dkr0 + st * K_STEP);
                        mma_commit(bar_addr(bars.k_empty[st]));
                        if (j + 2 >= n_kv) mma_commit(bar_addr(bars.q_empty[qb]));   // last own QK
                        if (!pass_skipped_v()) break;
                        if (prev_j >= 0 && !pv_of_prev()) break;
                        prev_j = j;
                        prev_st = st;
                        prev_ph = ph;
                        prev_c = c++;
                    }
                    if (++st == (uint32_t)ST) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // no key tile of this item is this issuer's (a single-tile segment): release the Q
                // buffer at once (the producer may be waiting for it before it issues the V that
                // the line below waits for)
                if (prev_j < 0) mbar_arrive(bar_addr(bars.q_empty[qb]));
                if (!pass_skipped_v()) break;                  // the item's last tile was the other's
                if (prev_j >= 0) {
                    if (!pv_of_prev()) break;
                } else if (item_cnt > 0 && !(ok = wait(b_ofree, (item_cnt - 1) & 1))) {
                    break;                                     // keep o_free's phase count in step
                }
                t += n_kv;
            }
            // drain: nothing this thread issued may still be running when TMEM is freed
            mma_commit(bar_addr(bars.drain[ti]));
            mbar_wait(bar_addr(bars.drain[ti]), 0, (const volatile int *)&s_abort, ok ? kWaitBudget : 200000000ll);
        }
    } else if (warp == 3) {
        if constexpr (FQ) {
            // -------------------------------------------------------- raw Q -> normalised, rotated Q
            // Lane l takes rows l, l + 32, .. of the item's 256; each row is read and rewritten in
            // place through its 32-byte-swizzled slabs (16-byte chunk index XOR bit 2 of the row,
            // the layout the TMA wrote and the MMA descriptors read). Rows past the segment end
            // belong to no result and are left as loaded.
            uint32_t item_cnt = 0;
            bool ok = true;
            for (Item item; take_item(item_cnt, item, true, ok); ++item_cnt) {
                const int64_t seg_end = (int64_t)item.x + item.y, q0 = item.z;
                const uint32_t qb = item_cnt % C::QBUF;
                if (!(ok = wait_warp(bars.q_full[qb], (item_cnt / C::QBUF) & 1))) break;
                unsigned char *qbuf = base + C::OFF_Q + 2 * qb * C::Q_TILE;
                const int n_rows = item_split(item) ? BM : 2 * BM;   // a split item has one Q tile
#pragma unroll 1
                for (int k = 0; k < n_rows / 32; ++k) {
                    const int row = lane + 32 * k;
                    if (q0 + row >= seg_end) continue;
                    const int r = row % BM;
                    unsigned char *tile = qbuf + (row / BM) * C::Q_TILE;
                    // 16-byte chunk c (columns 8c .. 8c + 7) of row r, through the swizzle the TMA wrote
                    // (chunk index XOR the row's bits 0-2, 1-2 or 2 for 128-, 64- or 32-byte swizzle)
                    unsigned char *wide_row = tile + 128 * r;                    // row r of slab 0
                    unsigned char *rem_row = tile + C::N128 * C::Q_SLAB128 + 2 * C::REM * r;
                    const int wx = r & 7, rx = C::REM == 32 ? (r >> 1) & 3 : (r >> 2) & 1;
                    rope::transform_row<D>(qr, q0 + row, [&](int c) -> uint4 * {
                        if (C::REM == 0 || c < 8 * C::N128)
                            return reinterpret_cast<uint4 *>(wide_row + (c >> 3) * C::Q_SLAB128 + (((c & 7) ^ wx) << 4));
                        return reinterpret_cast<uint4 *>(rem_row + (((c - 8 * C::N128) ^ rx) << 4));
                    });
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_addr(bars.q_ready[qb]));
            }
        } else if (lane == 0) {
            // nothing to do but free its share of every item ring slot
            bool ok = true;
            Item item;
            for (uint32_t k = 0; take_item(k, item, false, ok); ++k) {
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax groups
        regs_inc<FQ ? kSoftmaxRegsFQ : kSoftmaxRegs>();
        const int grp = (warp - 4) >> 2;                       // 0 or 1: which Q tile
        const int quarter = warp & 3;                          // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;                   // row of the tile = TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tS = t_lane + (grp ? C::TS1 : C::TS0);
        const uint32_t tO = t_lane + (grp ? C::TO1 : C::TO0);
        const uint32_t tP = t_lane + (grp ? C::TP1 : C::TP0);
        // P tiles this group has written; at the top of the tile loop it also counts the S tiles read
        uint32_t p_cnt = 0, item_cnt = 0;
        bool ok = true;
        // At head_dim 128 a two-tile item's output is written after the group has stored the
        // first P of its next item (or at the end): the exponentials of that tile hide the wait
        // for the item's last P.V and the longer O read-out. Until then O stays reserved (o_free
        // not yet arrived), so the next item's first P.V cannot overwrite it. Measured: 2 % faster
        // at head_dim 128, 1-6 % slower at 80 (where the epilogue is short), so only there.
        constexpr bool kDeferOut = D >= 128;
        bool pend = false, pend_store = false;
        int pend_row = 0, pend_head = 0;
        float pend_m = 0.f, pend_l = 1.f;
        auto write_out = [&]() {               // O / l -> bf16 -> HBM, then O is free
            tc_fence_after();
            const float inv_l = 1.f / pend_l;
            // l sums exp2(s * scale*log2(e) - m), so ln(sum exp(scale * s)) = (m + log2 l) ln 2
            if (LSE && pend_store)
                lse[(int64_t)pend_row * H + pend_head] = (pend_m + log2f(pend_l)) * 0.6931471805599453f;
            __nv_bfloat16 *dst = out + (int64_t)pend_row * out_stride + (int64_t)pend_head * D;
#pragma unroll
            for (int c = 0; c < D; c += 16) {
                uint32_t r[16];
                tmem_ld16(tO + c, r);
                tmem_wait_ld();
                reg_fence(r);
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
                if (pend_store) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
                    d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(bars.o_free[grp]));
            pend = false;
        };

        for (Item item; take_item(item_cnt, item, true, ok); ++item_cnt) {
            const int seg0 = item.x, seg_len = item.y, q0 = item.z, head = item_head(item);
            const int n_kv = (seg_len + BN - 1) / BN;
            // own key tiles: every one, or in a split item every other one starting at this group's
            const int dj = item_split(item) ? 2 : 1;
            float m_run = -INFINITY, l_run = 0.f;

            for (int j = dj == 2 ? grp : 0; j < n_kv && ok; j += dj) {
                if (!(ok = wait_warp(bars.s_full[grp], p_cnt & 1))) break;
                tc_fence_after();
                // S row -> registers: all loads in flight, one wait
                uint32_t sr[BN];
#pragma unroll
                for (int c = 0; c < BN; c += 16) tmem_ld16(tS + c, *reinterpret_cast<uint32_t(*)[16]>(sr + c));
                tmem_wait_ld();
                reg_fence(sr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_addr(bars.s_free[grp]));

                // the previous P.V of this tile has almost always finished by now: probe it
                // without blocking, so its barrier latency overlaps the arithmetic below
                const bool pv_probe = p_cnt == 0 || mbar_test(bar_addr(bars.pv_done[grp]), (p_cnt - 1) & 1);
                const int kv_valid = seg_len - j * BN;         // keys of this tile inside the segment
                if (kv_valid < BN) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c >= kv_valid) sr[c] = __float_as_uint(-INFINITY);
                }
                // row max: 8 independent chains of 3-input max, then a tree
                static_assert(BN % 16 == 0, "row max consumes 16 columns per step");
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmaxf(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
#pragma unroll
                for (int c = 16; c < BN; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m8[i] = max3(m8[i], __uint_as_float(sr[c + 2 * i]), __uint_as_float(sr[c + 2 * i + 1]));
                const float mx = fmaxf(max3(m8[0], m8[1], m8[2]), max3(max3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
                const float m_tile = mx * scale_log2;
                float alpha = 1.f;
                if (m_tile > m_run + 8.f) {                    // lazy rescale: only when the max grows by > 2^8
                    alpha = ex2(m_run - m_tile);
                    m_run = m_tile;
                }
                // the first own tile of an item (l_run still 0) overwrites O: its P.V does not accumulate
                const bool rescale = (l_run != 0.f) && (alpha != 1.f);
                // p = exp2(s * scale*log2(e) - m): pairs through the f32x2 FMA, row sum in f32x2 adds
                uint32_t pk[BN / 2];
                const uint64_t sc2 = f2_splat(scale_log2), nm2 = f2_splat(-m_run);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    float x0, x1;
                    f2_split(f2_fma(f2_from_u32(sr[c], sr[c + 1]), sc2, nm2), x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    uint64_t pp;
                    asm("mov.b64 %0, {%1, %2};\n" : "=l"(pp) : "f"(p0), "f"(p1));
                    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], pp);
                    pk[c / 2] = pack_bf16x2(p0, p1);
                }
                float a0, a1;
                f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                l_run = l_run * alpha + (a0 + a1);

                // this tile's P region is free, and its O holds every earlier P.V product, once
                // the previous P.V of this tile has completed
                if (!__all_sync(0xffffffffu, pv_probe) && !(ok = wait_warp(bars.pv_done[grp], (p_cnt - 1) & 1))) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
                    const float a = rescale ? alpha : 1.f;
#pragma unroll
                    for (int c = 0; c < D; c += 16) {
                        uint32_t r[16];
                        tmem_ld16(tO + c, r);
                        tmem_wait_ld();
                        reg_fence(r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a);
                        tmem_st16(tO + c, r);
                    }
                }
#pragma unroll
                for (int c = 0; c < BN / 2; c += 8) tmem_st8(tP + c, *reinterpret_cast<const uint32_t(*)[8]>(pk + c));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_addr(bars.p_full[grp]));
                ++p_cnt;
                // the previous item's last P.V completed before this P was stored (the wait above)
                if constexpr (kDeferOut) {
                    if (pend) write_out();
                }
            }
            if (!ok) break;

            if (kDeferOut && dj == 1) {
                // the output of this item waits for the first P of the next one (or the end)
                pend = true;
                pend_row = q0 + grp * BM + row;
                pend_store = pend_row < seg0 + seg_len;
                pend_head = head;
                pend_m = m_run;
                pend_l = l_run;
                continue;
            }
            if (dj == 1) {
                // epilogue: wait for this tile's last P.V, then O / l -> bf16 -> HBM
                if (!(ok = wait_warp(bars.pv_done[grp], (p_cnt - 1) & 1))) break;
                tc_fence_after();
                const int q_row = q0 + grp * BM + row;
                const bool store = q_row < seg0 + seg_len;
                const float inv_l = 1.f / l_run;
                // l_run sums exp2(s * scale*log2(e) - m_run), so ln(sum exp(scale * s)) = (m_run + log2 l_run) ln 2
                if (LSE && store) lse[(int64_t)q_row * H + head] = (m_run + log2f(l_run)) * 0.6931471805599453f;
                __nv_bfloat16 *dst = out + (int64_t)q_row * out_stride + (int64_t)head * D;
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                    uint32_t r[16];
                    tmem_ld16(tO + c, r);
                    tmem_wait_ld();
                    reg_fence(r);
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
                    if (store) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
                        d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_addr(bars.o_free[grp]));
                continue;
            }
            // a split item in which this group owns no key tile: the pending output goes first
            if (kDeferOut && pend) {
                if (!(ok = wait_warp(bars.pv_done[grp], (p_cnt - 1) & 1))) break;
                write_out();
            }

            // split item: the two groups hold partial results of the same 128 rows over disjoint
            // key tiles (group g: O_g, running max m_g, row sum l_g, all relative to m_g). Each
            // group waits for its last P.V, publishes (m_g, l_g), and after the first meeting
            // writes half of the head's columns of
            //   out = (2^(m_0 - M) O_0 + 2^(m_1 - M) O_1) / (2^(m_0 - M) l_0 + 2^(m_1 - M) l_1),
            // M = max(m_0, m_1), reading both groups' O. A group with no tile of this item (a
            // one-tile segment) contributes nothing: its O is never read. The second meeting
            // keeps either O region from being overwritten before both groups have read it.
            const int n_own1 = n_kv >> 1;                     // key tiles of group 1 (group 0 has >= 1)
            const bool mine = grp ? n_own1 > 0 : true;
            if (mine && !(ok = wait_warp(bars.pv_done[grp], (p_cnt - 1) & 1))) break;
            s_m[grp][row] = m_run;
            s_l[grp][row] = l_run;
            tc_fence_before();
            __syncwarp();
            // every split item takes the merge barrier through two phases: parity 0, then 1
            if (lane == 0) mbar_arrive(bar_addr(bars.merge));
            if (!(ok = wait_warp(bars.merge, 0))) break;
            tc_fence_after();
            // this group's (m, l) are still in registers; the other group's come from shared memory
            const float m_oth = s_m[grp ^ 1][row], l_oth = s_l[grp ^ 1][row];
            const bool oth_has = grp ? true : n_own1 > 0;     // group 0 always has a tile
            const float M = oth_has ? fmaxf(m_run, m_oth) : m_run;
            const float w_own = mine ? ex2(m_run - M) : 0.f, w_oth = oth_has ? ex2(m_oth - M) : 0.f;
            const float l_sum = w_own * l_run + w_oth * l_oth;
            const float inv_l = 1.f / l_sum;
            const float c0 = (grp ? w_oth : w_own) * inv_l, c1 = (grp ? w_own : w_oth) * inv_l;
            const int q_row = q0 + row;
            const bool store = q_row < seg0 + seg_len;
            if (LSE && store && grp == 0) lse[(int64_t)q_row * H + head] = (M + log2f(l_sum)) * 0.6931471805599453f;
            constexpr int HALF = D / 2;                        // columns of the head this group writes
            static_assert(HALF % 8 == 0, "each group writes whole 16-byte pieces");
            static_assert(C::TO1 == C::TO0 + D, "O1 follows O0");
            const uint32_t tO0 = tO - grp * HALF, tO1 = tO0 + D;     // this group's columns of O0 and O1
            __nv_bfloat16 *dst = out + (int64_t)q_row * out_stride + (int64_t)head * D + grp * HALF;
#pragma unroll
            for (int c = 0; c < HALF; c += 8) {
                uint32_t r0[8], r1[8];
                tmem_ld8(tO0 + c, r0);
                if (n_own1 > 0) tmem_ld8(tO1 + c, r1);
                tmem_wait_ld();
                reg_fence(r0);
                if (n_own1 > 0) reg_fence(r1);
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x0 = __uint_as_float(r0[2 * e]) * c0, x1 = __uint_as_float(r0[2 * e + 1]) * c0;
                    if (n_own1 > 0) {
                        x0 = fmaf(__uint_as_float(r1[2 * e]), c1, x0);
                        x1 = fmaf(__uint_as_float(r1[2 * e + 1]), c1, x1);
                    }
                    o[e] = pack_bf16x2(x0, x1);
                }
                if (store) *reinterpret_cast<uint4 *>(dst + c) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(bars.merge));
            if (!(ok = wait_warp(bars.merge, 1))) break;
            if (lane == 0) mbar_arrive(bar_addr(bars.o_free[grp]));
        }
        // the last item's output, once its last P.V has completed
        if (kDeferOut && pend && ok && (ok = wait_warp(bars.pv_done[grp], (p_cnt - 1) & 1))) write_out();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

// [T, H*D] bf16 rows with a token stride, read as boxes of `cols` columns x `rows` rows with the
// swizzle that matches the box width (128, 64 or 32 bytes).
bool make_map(CUtensorMap *m, const void *ptr, int64_t T, int H, int D, int64_t stride, int rows, int cols)
{
    const uint64_t dims[2] = {(uint64_t)H * D, (uint64_t)(T > 0 ? T : 1)};
    const uint64_t strides[1] = {(uint64_t)stride * 2};
    const uint32_t box[2] = {(uint32_t)cols, (uint32_t)rows};
    return encode_tiled_map(m, ptr, 2, dims, strides, box, cols * 2);
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, int64_t max_items, int num_sms, int stall_v, cudaStream_t stream)
{
    using C = LongCfg<D>;
    // Q and K: 64-column boxes and a remainder box (unused when head_dim is a multiple of 64);
    // V: 16-column boxes
    const int rem = C::REM > 0 ? C::REM : 64;
    CUtensorMap mq, mqr, mk, mkr, mv;
    if (!make_map(&mq, a.q, a.T, a.H, D, a.q_stride, BM, 64) || !make_map(&mqr, a.q, a.T, a.H, D, a.q_stride, BM, rem) ||
        !make_map(&mk, a.k, a.T, a.H, D, a.k_stride, C::BN, 64) ||
        !make_map(&mkr, a.k, a.T, a.H, D, a.k_stride, C::BN, rem) ||
        !make_map(&mv, a.v, a.T, a.H, D, a.v_stride, C::BN, 16))
        return cudaErrorInvalidValue;
    // the lse store is compiled in only where it is asked for: the plain kernel keeps its code unchanged
    auto kern = a.lse ? (a.fuse_q ? attn_long_kernel<D, true, true> : attn_long_kernel<D, true, false>)
                      : (a.fuse_q ? attn_long_kernel<D, false, true> : attn_long_kernel<D, false, false>);
    static DeviceOnce once[4];                           // per (lse, fused Q) variant
    cudaError_t e = once[(a.lse ? 2 : 0) + (a.fuse_q ? 1 : 0)].run([&] {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (r != cudaSuccess) return r;
        // the setmaxnreg split assumes exactly this launch budget; refuse anything else rather than wait on it
        cudaFuncAttributes fa;
        r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        return (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads) ? cudaErrorInvalidConfiguration
                                                                              : cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)(max_items < num_sms ? max_items : num_sms);
    if (blocks == 0) return cudaSuccess;
    LaunchScope scope("attn_long", stream);
    kern<<<blocks, kThreads, C::SMEM, stream>>>(mq, mqr, mk, mkr, mv, static_cast<__nv_bfloat16 *>(a.out),
                                                               a.out_stride, a.lse, a.H, a.scale_log2,
                                                               const_cast<WsHeader *>(a.hdr),
                                                               a.items, a.status, stall_v, a.qr);
    return cudaGetLastError();
}

}  // namespace

bool encode_tiled_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides,
                      const uint32_t *box, int swizzle_bytes)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                   ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p)
                   : nullptr;
    }();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), d, st, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int attn_long_bm() { return 2 * BM; }

bool attn_long_supports(int D) { return D == 32 || D == 64 || D == 80 || D == 96 || D == 128; }

cudaError_t launch_attn_long(const AttnArgs &a, int64_t max_items_long, int num_sms, int stall_v,
                             cudaStream_t stream)
{
    switch (a.D) {
        case 32: return launch_d<32>(a, max_items_long, num_sms, stall_v, stream);
        case 64: return launch_d<64>(a, max_items_long, num_sms, stall_v, stream);
        case 80: return launch_d<80>(a, max_items_long, num_sms, stall_v, stream);
        case 96: return launch_d<96>(a, max_items_long, num_sms, stall_v, stream);
        case 128: return launch_d<128>(a, max_items_long, num_sms, stall_v, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace vit
