// Internal declarations shared by the CUDA translation units of libvitattn.
#pragma once

#include <cuda.h>           // CUtensorMap (type only; the library never links libcuda)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "vit_attn.h"
#include "rope_math.cuh"

namespace vit {

// Work item of the attention kernels: one (segment, head, q-block).
//   x = first token of the segment, y = segment length,
//   z = first query token of the block, w = head | kItemSplit when set.
// A long-segment item covers 256 query rows as two 128-row Q tiles that share every key tile;
// with kItemSplit it covers 128 rows, and its two halves of the long kernel take alternate key
// tiles of the segment and merge their partial results at the end (used for a segment's last
// block of at most 128 rows, and for every block when a batch has too few items to fill the GPU).
using Item = int4;
constexpr int kItemSplit = 1 << 30;
constexpr int kMaxHeads = 1 << 24;            // heads fit below the flag bit
__host__ __device__ inline int item_head(const Item &it) { return it.w & (kItemSplit - 1); }
__host__ __device__ inline bool item_split(const Item &it) { return (it.w & kItemSplit) != 0; }

// Header at the start of the attention workspace, written by the scheduler.
struct WsHeader {
    int32_t n_long;      // items [0, n_long) go to the long-segment kernel
    int32_t reserved;    // 0
    int32_t bm_long;     // query rows per long item
    int32_t tiny_max;    // segments of at most this many tokens are tiny (one item per head)
    int32_t error;       // device-detected error of the last scheduling pass (0 = none)
    int32_t n_tiny;      // items [n_long, n_long + n_tiny) go to the tiny-segment kernel
    int32_t long_all_split;   // 1 when every long item is a split item of bm_long / 2 rows
    int32_t next_long;   // long items handed out so far beyond each CTA's first (zeroed by the scheduler)
    int32_t pad[8];
};
static_assert(sizeof(WsHeader) == 64, "header is 64 bytes");

// Scheduling parameters chosen by the host.
struct SchedParams {
    int tiny_max;    // segments with length <= tiny_max use the tiny-segment kernel (one item per
                     // head), longer ones the tcgen05 kernel
    int bm_long;     // q rows per long item
    int num_sms;     // SMs of the device: with at most num_sms / 2 long items of bm_long rows, every
                     // long block is cut to bm_long / 2 rows and split over its key tiles instead
};

// Upper bound on the number of items of one class for these sizes.
inline int64_t max_items(int64_t T, int H, int B, int bm) {
    return (int64_t)H * ((T + bm - 1) / bm + B);
}

// Record a device-side error (first error wins; never overwrites a stored code).
__device__ __forceinline__ void report_error(int32_t *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// One-time setup per device of a kernel's launch attributes (dynamic shared memory limit,
// register checks, occupancy). Done on the first launch on each device, so later calls,
// including ones made while a stream is being captured into a CUDA graph, only launch.
struct DeviceOnce {
    std::atomic<uint64_t> done{0};
    template <typename F> cudaError_t run(F &&fn) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
        if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        e = fn();
        if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }
};

// ---- launch bookkeeping (instrument.cpp) ----
struct LaunchScope {
    LaunchScope(const char *name, cudaStream_t stream);
    ~LaunchScope();
    const char *name_;
    cudaStream_t stream_;
    void *slot_;
};

// ---- launchers (one per translation unit) ----
cudaError_t launch_rope_freqs(int dim, float theta, const int32_t *grid_hw, int n_img, int64_t T,
                              float *inv_freq, int32_t *pos_hw, int32_t *cu_seqlens, int32_t *status,
                              cudaStream_t stream);

cudaError_t launch_rope_table(const float *inv_freq, int n_freq, int max_pos, float *cos_sin,
                              cudaStream_t stream);

// q_in/q_out or k_in/k_out may both be NULL (that half is skipped); interleaved selects adjacent pairs.
cudaError_t launch_qk_norm_rope(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T,
                                int H, int D, int64_t q_in_stride, int64_t q_out_stride,
                                int64_t k_in_stride, int64_t k_out_stride, const int32_t *pos_hw,
                                const float *inv_freq, const void *norm_w, float eps, bool interleaved,
                                int num_sms, int32_t *status, cudaStream_t stream);

// segments from cu_seqlens (contiguous; NULL = B uniform segments) or, when seq_len is
// given, from per-segment starts and lengths (a padded layout)
cudaError_t launch_schedule(const int32_t *cu_seqlens, const int32_t *seq_start, const int32_t *seq_len, int B,
                            int64_t T, int H, int max_seqlen, SchedParams sp, WsHeader *hdr, Item *items,
                            int32_t *status, cudaStream_t stream);

// Everything both attention kernels read, validated by the API layer.
struct AttnArgs {
    const void *q, *k, *v;      // bf16 [T, H, D] with token strides below
    void *out;                  // bf16 [T, H, D]
    float *lse;                 // fp32 [T, H] natural-log sum of exp(scale * s) per row, or NULL
    int64_t T;
    int H, D;
    int64_t max_len;            // upper bound on every segment's length (max_seqlen, or T / B uniform)
    int64_t q_stride, k_stride, v_stride, out_stride;   // token strides, elements
    float scale_log2;           // softmax scale * log2(e)
    const WsHeader *hdr;
    const Item *items;
    int32_t *status;
    bool fuse_q;                // q holds raw values: normalise and rotate each Q tile after it is loaded
    rope::QRope qr;             // how (when fuse_q)
};

cudaError_t launch_attn_tiny(const AttnArgs &a, int64_t max_items_tiny, int num_sms, cudaStream_t stream);

cudaError_t launch_attn_long(const AttnArgs &a, int64_t max_items_long, int num_sms, int stall_v,
                             cudaStream_t stream);

// Every host-side check of the attention calls except those of the workspace (api.cu).
// *nothing is set when the call has no work at all (no segments, no tokens).
vit_status_t check_varlen_attn_args(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                    int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                    const vit_q_rope_t *q_rope, const int32_t *cu_seqlens, const int32_t *seq_start,
                                    const int32_t *seq_len, int B, int max_seqlen, float scale, const void *out,
                                    int64_t out_stride, const float *lse, const vit_attn_options_t *opts,
                                    bool *nothing);

// A tiled TMA descriptor of a bf16 tensor (cuTensorMapEncodeTiled, reached through the runtime's
// driver entry point): `rank` dims innermost first, rank - 1 byte strides of the outer dims, the
// box, and the swizzle span in bytes (32, 64, 128; anything else: none). False when it fails.
bool encode_tiled_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides,
                      const uint32_t *box, int swizzle_bytes);

// VIT_OK when the current device is one this library was built for.
vit_status_t check_device();

}  // namespace vit
