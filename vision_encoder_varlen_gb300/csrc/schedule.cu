// Segment-aware work scheduler for the varlen attention kernels.
//
// From cu_seqlens alone, on the device (no host sync, so a caller can stay
// inside a CUDA graph: tokenspeed mm_encoder_attention.py, _varlen_metadata,
// keeps max_seqlen off the GPU->CPU path for the same reason), one block:
//   1. validates the offsets (cu[0] == 0, non-decreasing, cu[B] == T, every
//      length <= max_seqlen; max_seqlen may be a padded bucket bound,
//      round_up_to_bucket on the same page). A padded layout (per-segment
//      start and real length, as the cuDNN path's offsets and
//      sequence_lengths describe) is taken instead when seq_len is given:
//      starts ascending, segments inside [0, T) and not overlapping; the rows
//      between them are padding that nothing reads or writes;
//   2. orders the segments: those for the long-segment kernel longest first
//      (LPT, a bitonic sort of (length desc, index asc) keys, so the order is
//      deterministic and the persistent CTAs end together), then the tiny
//      ones in index order (a stable partition by block scans: their items
//      are small, so sorting them buys no balance and cost most of the
//      scheduler's time for thousands of small images);
//   3. expands every segment into (segment, head, q-block) work items: long
//      segments into blocks of bm_long query rows for the long-segment kernel
//      (a last block of at most bm_long / 2 rows, and every block of a batch
//      too small to give each SM two blocks' worth of items, as a split item
//      of bm_long / 2 rows whose two halves take alternate key tiles),
//      tiny ones (at most tiny_max tokens) into one item per head, in head
//      order, for the tiny-segment kernel. The two classes come out as two
//      contiguous runs of the item list.
//      Items never straddle two segments; the q-block is the fastest index,
//      so concurrently running CTAs share one head's K/V in L2.
// On invalid offsets it records the error and publishes zero items, so the
// attention kernels that follow compute nothing.
#include "internal.h"

namespace vit {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *s_warp, int64_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;                // inclusive over warps
    }
    __syncthreads();
    const int64_t before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kThreads)
schedule_kernel(const int32_t *__restrict__ cu_seqlens, const int32_t *__restrict__ seq_start,
                const int32_t *__restrict__ seq_len, int B, int64_t T, int H, int max_seqlen,
                SchedParams sp, WsHeader *hdr, Item *items, int32_t *status)
{
    extern __shared__ unsigned long long s_key[];      // [NP] sort keys of the long segments
    __shared__ int64_t s_warp[32];
    __shared__ int s_err;
    const int tid = threadIdx.x;
    int NP = 1;
    while (NP < B) NP <<= 1;
    int32_t *s_start = reinterpret_cast<int32_t *>(s_key + NP);   // [B] segment start by segment index
    int32_t *s_len = s_start + B;                                  // [B] segment length by segment index
    int32_t *s_off = s_len + B;                                    // [B] first item of position p
    int32_t *s_order = s_off + B;                                  // [B] segment index at position p

    if (tid == 0) s_err = 0;
    __syncthreads();

    // ---- 1. offsets and validation
    const int64_t uni = B > 0 ? T / B : 0;
    for (int i = tid; i < B; i += kThreads) {
        int64_t a, b;
        if (seq_len) {
            a = seq_start[i];
            b = a + seq_len[i];
            // inside [0, T), after the previous segment's end
            if (a < 0 || b > T || (i > 0 && a < (int64_t)seq_start[i - 1] + seq_len[i - 1]))
                atomicMax(&s_err, 1);
        } else {
            if (cu_seqlens) {
                a = cu_seqlens[i];
                b = cu_seqlens[i + 1];
            } else {
                a = uni * i;
                b = uni * (i + 1);
            }
            if (i == 0 && a != 0) atomicMax(&s_err, 1);
            if (i == B - 1 && b != T) atomicMax(&s_err, 1);
        }
        if (b < a) atomicMax(&s_err, 1);
        else if (b - a > (int64_t)max_seqlen) atomicMax(&s_err, 2);
        s_start[i] = (int32_t)a;
        s_len[i] = (int32_t)(b > a ? b - a : 0);
    }
    __syncthreads();
    if (s_err) {
        if (tid == 0) {
            hdr->n_long = 0;
            hdr->reserved = 0;
            hdr->n_tiny = 0;
            hdr->long_all_split = 0;
            hdr->next_long = 0;
            hdr->error = s_err == 1 ? VIT_ERR_BAD_SEQLENS : VIT_ERR_SEQLEN_EXCEEDS_MAX;
            report_error(status, hdr->error);
        }
        return;
    }

    // ---- 2. order: long class longest first, then tiny (index order)
    const int per = (B + kThreads - 1) / kThreads;
    const int lo = min(tid * per, B), hi = min(lo + per, B);
    auto seg_class = [&](int len) { return len > sp.tiny_max ? 0 : 1; };
    int64_t cnt[2] = {0, 0};
    for (int i = lo; i < hi; ++i) ++cnt[seg_class(s_len[i])];
    int64_t tot[2];
    int64_t pos[2];
    for (int c = 0; c < 2; ++c) pos[c] = block_exclusive_scan(cnt[c], s_warp, &tot[c]);
    const int n_lseg = (int)tot[0];
    pos[1] += tot[0];
    for (int i = lo; i < hi; ++i) {
        const int c = seg_class(s_len[i]);
        if (c == 0)      // ascending keys = descending length, then ascending index
            s_key[pos[0]++] = ((unsigned long long)(0x7fffffffu - (uint32_t)s_len[i]) << 32) | (uint32_t)i;
        else
            s_order[pos[c]++] = i;
    }
    int NPL = 1;
    while (NPL < n_lseg) NPL <<= 1;
    for (int i = n_lseg + tid; i < NPL; i += kThreads) s_key[i] = ~0ull;
    __syncthreads();
    for (int k = 2; k <= NPL; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < NPL; i += kThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = s_key[i], y = s_key[l];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) {
                        s_key[i] = y;
                        s_key[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int p = tid; p < n_lseg; p += kThreads) s_order[p] = (int32_t)(s_key[p] & 0xffffffffu);
    __syncthreads();

    // ---- 3. item counts per position, exclusive scan, expansion
    // (the block sizes are powers of two: shifts instead of divisions, which otherwise dominate
    // this single block's instruction count for thousands of segments)
    // Long blocks are bm_long rows (two Q tiles) unless the whole batch would give at most
    // num_sms / 2 of them: then every long block is cut to bm_long / 2 rows, twice as many items,
    // each split over its key tiles, so twice as many SMs work on the batch.
    const int lg_full = __ffs(sp.bm_long) - 1;
    int64_t local_full = 0, total_full;
    for (int p = lo; p < hi; ++p) {
        const int len = s_len[s_order[p]];
        if (len > sp.tiny_max) local_full += (int64_t)H * ((len + (1 << lg_full) - 1) >> lg_full);
    }
    block_exclusive_scan(local_full, s_warp, &total_full);
    const bool all_split = 2 * total_full <= (int64_t)sp.num_sms;
    const int lg_long = all_split ? lg_full - 1 : lg_full;
    auto n_blocks = [&](int len) {                      // a tiny segment is one block
        return len > sp.tiny_max ? (len + (1 << lg_long) - 1) >> lg_long : (len > 0 ? 1 : 0);
    };
    int64_t local = 0, local_long = 0;
    for (int p = lo; p < hi; ++p) {
        const int len = s_len[s_order[p]];
        const int64_t n = (int64_t)H * n_blocks(len);
        local += n;
        if (len > sp.tiny_max) local_long += n;
    }
    int64_t total, total_long;
    int64_t run = block_exclusive_scan(local, s_warp, &total);
    block_exclusive_scan(local_long, s_warp, &total_long);
    for (int p = lo; p < hi; ++p) {
        s_off[p] = (int32_t)run;
        run += (int64_t)H * n_blocks(s_len[s_order[p]]);
    }
    __syncthreads();
    // one warp per sorted segment (a whole-block loop over B segments would leave most threads idle)
    const int lane = tid & 31, warp = tid >> 5;
    for (int p = warp; p < B; p += kThreads / 32) {
        const int seg = s_order[p];
        const int len = s_len[seg];
        if (len == 0) continue;
        const bool is_long = len > sp.tiny_max;
        const int bm = 1 << lg_long;
        const int nq = n_blocks(len);             // 1 for a tiny segment
        const int start = s_start[seg];
        // a long item is split when every long item is, or when it is the segment's last block
        // and holds at most bm_long / 2 rows (its second Q tile would be empty)
        const int last_rows = len - (nq - 1) * bm;
        const int split_last = is_long && (all_split || 2 * last_rows <= sp.bm_long) ? kItemSplit : 0;
        const int split_rest = is_long && all_split ? kItemSplit : 0;
        Item *dst = items + s_off[p];
        if (nq == 1) {                                     // one query block: item i is head i
            for (int i = lane; i < H; i += 32) dst[i] = make_int4(start, len, start, i | split_last);
        } else {
            for (int i = lane; i < H * nq; i += 32) {
                const int h = i / nq, qb = i - h * nq;
                dst[i] = make_int4(start, len, start + qb * bm, h | (qb == nq - 1 ? split_last : split_rest));
            }
        }
    }
    if (tid == 0) {
        hdr->n_long = (int32_t)total_long;
        hdr->reserved = 0;
        hdr->n_tiny = (int32_t)(total - total_long);
        hdr->bm_long = 1 << lg_long;
        hdr->tiny_max = sp.tiny_max;
        hdr->error = 0;
        hdr->long_all_split = all_split ? 1 : 0;
        hdr->next_long = 0;
    }
}

}  // namespace

size_t schedule_smem_bytes(int B)
{
    int NP = 1;
    while (NP < B) NP <<= 1;
    return sizeof(unsigned long long) * (size_t)NP + sizeof(int32_t) * 4 * (size_t)B;
}

cudaError_t launch_schedule(const int32_t *cu_seqlens, const int32_t *seq_start, const int32_t *seq_len, int B,
                            int64_t T, int H, int max_seqlen, SchedParams sp, WsHeader *hdr, Item *items,
                            int32_t *status, cudaStream_t stream)
{
    const size_t smem = schedule_smem_bytes(B);
    static DeviceOnce once;                              // the limit for the largest B, set once
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)schedule_smem_bytes(VIT_MAX_SEGMENTS));
    });
    if (e != cudaSuccess) return e;
    LaunchScope scope("schedule", stream);
    schedule_kernel<<<1, kThreads, smem, stream>>>(cu_seqlens, seq_start, seq_len, B, T, H, max_seqlen, sp, hdr,
                                                   items, status);
    return cudaGetLastError();
}

}  // namespace vit
