// vit_varlen_attn_noalloc: the varlen attention call without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code that runs under an allocator that forbids new allocations
// (a serving loop whose memory pool is frozen after warm-up), plugins handed
// only input and output pointers by a host framework, or C callers that have
// no allocator of their own. For them this entry point keeps the scheduler's
// work list in a fixed array that lives in the library's own device image
// (VIT_NOALLOC_WORKSPACE_BYTES per GPU, held while the context that loaded it
// lives) and otherwise behaves exactly like vit_varlen_attn.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "trace.h"

namespace {

// The scheduler's header and work items for calls without a caller workspace.
// Every GPU that loads this library holds one copy while its context lives.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VIT_NOALLOC_WORKSPACE_BYTES];

// The array's address belongs to the module loaded into one CUDA context. A context that is
// destroyed and made again (cudaDeviceReset, or the primary context released by every user and
// retained anew) loads the module again, possibly elsewhere, so the cache is keyed on the
// context's unique id, not on the device number.
struct ScratchCache {
    unsigned long long ctx_id;   // id of the context the address was looked up in (0 = none)
    void *ptr;
};
constexpr int kMaxDevices = 64;
ScratchCache g_cache[kMaxDevices];
std::mutex g_scratch_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Driver entry points for the current context's id (the library does not link libcuda).
bool current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// The array's device address in the current context: looked up on the first call in each
// context (with that context's device current), then taken from the cache. A lookup is refused
// while `stream` is being captured, since it may load the module and so break the capture.
vit_status_t scratch_address(cudaStream_t stream, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VIT_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return VIT_ERR_UNSUPPORTED_DEVICE;
    // (also binds the device's primary context to this thread if nothing has yet)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return VIT_ERR_BAD_ARGUMENT;
    }
    unsigned long long id = 0;
    if (!current_context_id(&id)) return VIT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchCache &c = g_cache[dev];
    if (c.ctx_id != id || !c.ptr) {
        if (cs != cudaStreamCaptureStatusNone) return VIT_ERR_BAD_ARGUMENT;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();               // leave no stale error for the next call to read
            return VIT_ERR_CUDA;
        }
        c.ctx_id = id;
        c.ptr = p;
    }
    *out = c.ptr;
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
    // every check vit_varlen_attn makes, then the device check, before the array is looked up
    bool nothing = false;
    vit_status_t st = vit::check_varlen_attn_args(q, k, v, T, H, D, q_stride, k_stride, v_stride, nullptr,
                                                  cu_seqlens, nullptr, nullptr, B, max_seqlen, scale, out,
                                                  out_stride, nullptr, nullptr, &nothing);
    if (st != VIT_OK || nothing) return st;
    // sizes whose work list does not fit the fixed array are refused before anything runs
    if (vit_varlen_attn_workspace_size(T, H, B, D) > (size_t)VIT_NOALLOC_WORKSPACE_BYTES)
        return VIT_ERR_WORKSPACE_TOO_SMALL;
    st = vit::check_device();
    if (st != VIT_OK) return st;
    void *scratch = nullptr;
    st = scratch_address((cudaStream_t)stream, &scratch);
    if (st != VIT_OK) return st;
    // The scheduler rewrites the header and the whole item list on every call before the
    // attention kernels read them, so nothing in the array has to start at zero.
    return vit_varlen_attn(q, k, v, T, H, D, q_stride, k_stride, v_stride, cu_seqlens, B, max_seqlen, scale, out,
                           out_stride, scratch, (size_t)VIT_NOALLOC_WORKSPACE_BYTES, status_dev, stream);
}
