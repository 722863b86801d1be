// vit_varlen_attn_noalloc: the varlen attention call without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code that runs under an allocator that forbids new allocations
// (a serving loop whose memory pool is frozen after warm-up), plugins handed
// only input and output pointers by a host framework, or C callers that have
// no allocator of their own. For them this entry point keeps the scheduler's
// work list in a fixed array that lives in the library's own device image
// (VIT_NOALLOC_WORKSPACE_BYTES per GPU, held from module load until process
// exit) and otherwise behaves exactly like vit_varlen_attn.
#include <mutex>

#include "internal.h"
#include "trace.h"

namespace {

// The scheduler's header and work items for calls without a caller workspace.
// Every GPU that loads this library holds one copy until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VIT_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device (NULL = not set up)
std::mutex g_scratch_mutex;

// Resolve the array's device address on the current device, once per device.
vit_status_t scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VIT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return VIT_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return VIT_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return VIT_OK;
}

}  // namespace

extern "C" vit_status_t vit_varlen_attn_noalloc(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                                int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                                const int32_t *cu_seqlens, int B, int max_seqlen, float scale,
                                                void *out, int64_t out_stride, int32_t *status_dev,
                                                vit_stream_t stream)
{
    vit::TraceRange trace("vit_varlen_attn_noalloc");
    // sizes whose work list does not fit the fixed array are refused before anything runs
    const size_t need = vit_varlen_attn_workspace_size(T, H, B, D);
    if (need > (size_t)VIT_NOALLOC_WORKSPACE_BYTES) return VIT_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    vit_status_t st = scratch_address(&scratch);
    if (st != VIT_OK) return st;
    // The scheduler rewrites the header and the whole item list on every call before the
    // attention kernels read them, so nothing in the array has to start at zero.
    return vit_varlen_attn(q, k, v, T, H, D, q_stride, k_stride, v_stride, cu_seqlens, B, max_seqlen, scale, out,
                           out_stride, scratch, (size_t)VIT_NOALLOC_WORKSPACE_BYTES, status_dev, stream);
}
