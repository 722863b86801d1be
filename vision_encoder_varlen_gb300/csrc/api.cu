// C ABI of libvitattn: argument validation on the host, then kernel launches.
// Every check that can be made without reading device memory is made here and
// returns an error before anything is launched; device-side checks (segment
// offsets, grid sums) are made by the kernels and reported through status_dev.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "trace.h"

namespace vit {
size_t schedule_smem_bytes(int B);
int attn_long_bm();
int attn_tiny_max();
}  // namespace vit

using namespace vit;

namespace {

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];         // 0 = not queried yet
int g_supported[kMaxDevices];   // 0 = not queried, 1 = yes, -1 = no
std::mutex g_dev_mutex;

vit_status_t device_info(int *num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VIT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return VIT_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_supported[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return VIT_ERR_CUDA;
        g_supported[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_sms[dev] = sms;
    }
    if (g_supported[dev] < 0) return VIT_ERR_UNSUPPORTED_DEVICE;
    if (num_sms) *num_sms = g_sms[dev];
    return VIT_OK;
}

bool head_dim_ok(int D) { return D == 32 || D == 64 || D == 80 || D == 96 || D == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool stride_ok(int64_t s, int H, int D) { return s >= (int64_t)H * D && s % 8 == 0; }

vit_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? VIT_OK : VIT_ERR_CUDA; }

constexpr int64_t kMaxTokens = (int64_t)1 << 31;

// Segments longer than this run on the tcgen05 long-segment kernel, the others on the
// tiny-segment kernel, unless a call's options ask for a lower split (the tiny kernel takes at
// most 64 tokens). Measured on GB300: up to 64 tokens the tiny-segment kernel is 2-4x faster
// than the tcgen05 kernel.
constexpr int kDefaultShortMax = 64;

#ifdef VIT_TEST_HOOKS
// Test builds only: when set, the long-segment kernel never loads V, so its bounded waits expire.
std::atomic<int> g_stall_v{0};
int stall_v() { return g_stall_v.load(); }
#else
constexpr int stall_v() { return 0; }
#endif

}  // namespace

extern "C" {

const char *vit_version(void) { return "vitattn 0.1 (sm_103a)"; }

const char *vit_status_string(vit_status_t s)
{
    switch (s) {
        case VIT_OK: return "ok";
        case VIT_ERR_NULL_POINTER: return "a required pointer is NULL";
        case VIT_ERR_BAD_HEAD_DIM: return "head_dim must be one of 32, 64, 80, 96, 128";
        case VIT_ERR_BAD_SHAPE: return "invalid tensor shape (T, H, B)";
        case VIT_ERR_BAD_STRIDE: return "token stride must be >= H*D and a multiple of 8 elements";
        case VIT_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case VIT_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than vit_varlen_attn_workspace_size()";
        case VIT_ERR_TOO_MANY_SEGMENTS: return "more segments than VIT_MAX_SEGMENTS";
        case VIT_ERR_CUDA: return "a CUDA runtime call failed";
        case VIT_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
        case VIT_ERR_BAD_SEQLENS: return "cu_seqlens invalid: cu[0] != 0, decreasing, or cu[B] != T";
        case VIT_ERR_SEQLEN_EXCEEDS_MAX: return "a segment is longer than max_seqlen";
        case VIT_ERR_GRID_MISMATCH: return "patch grid does not sum to T (or has negative sides)";
        case VIT_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case VIT_ERR_BAD_ARGUMENT: return "invalid argument";
        case VIT_ERR_POSITION_RANGE: return "a token position lies outside the rope table";
        default: return "unknown status";
    }
}

vit_status_t vit_device_supported(int device)
{
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
        return VIT_ERR_CUDA;
    return (major == 10 && minor == 3) ? VIT_OK : VIT_ERR_UNSUPPORTED_DEVICE;
}

vit_status_t vit_rope_freqs(int dim, float theta, const int32_t *grid_hw, int n_img, int64_t T, float *inv_freq,
                            int32_t *pos_hw, int32_t *cu_seqlens, int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_rope_freqs");
    if (dim < 2 || dim % 2 != 0 || dim > 256) return VIT_ERR_BAD_ARGUMENT;
    if (!(theta > 0.f) || !isfinite(theta)) return VIT_ERR_BAD_ARGUMENT;
    if (n_img < 0 || T < 0 || T >= kMaxTokens) return VIT_ERR_BAD_SHAPE;
    if (n_img > VIT_MAX_SEGMENTS) return VIT_ERR_TOO_MANY_SEGMENTS;
    if (n_img > 0 && !grid_hw) return VIT_ERR_NULL_POINTER;
    if (pos_hw && ((uintptr_t)pos_hw & 7u)) return VIT_ERR_MISALIGNED;
    if (!inv_freq && !pos_hw && !cu_seqlens) return VIT_OK;
    vit_status_t st = device_info(nullptr);
    if (st != VIT_OK) return st;
    return from_cuda(launch_rope_freqs(dim, theta, grid_hw, n_img, T, inv_freq, pos_hw, cu_seqlens, status_dev,
                                       (cudaStream_t)stream));
}

static vit_status_t qk_norm_rope_impl(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T,
                                      int H, int D, int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride,
                                      int64_t k_out_stride, const int32_t *pos_hw, const float *inv_freq,
                                      const void *norm_w, float eps, int rope_mode, int32_t *status_dev,
                                      vit_stream_t stream)
{
    if (!head_dim_ok(D)) return VIT_ERR_BAD_HEAD_DIM;
    if (T < 0 || T >= kMaxTokens || H < 1) return VIT_ERR_BAD_SHAPE;
    if (!(eps >= 0.f) || !isfinite(eps)) return VIT_ERR_BAD_ARGUMENT;
    if (rope_mode != VIT_ROPE_ROTATE_HALF && rope_mode != VIT_ROPE_INTERLEAVED) return VIT_ERR_BAD_ARGUMENT;
    // each of the q and k halves is either fully given or fully absent; at least one is given
    const bool has_q = q_in || q_out, has_k = k_in || k_out;
    if ((has_q && (!q_in || !q_out)) || (has_k && (!k_in || !k_out)) || (!has_q && !has_k))
        return VIT_ERR_NULL_POINTER;
    if (T == 0) return VIT_OK;
    if (!pos_hw || !inv_freq) return VIT_ERR_NULL_POINTER;
    if ((has_q && (!stride_ok(q_in_stride, H, D) || !stride_ok(q_out_stride, H, D))) ||
        (has_k && (!stride_ok(k_in_stride, H, D) || !stride_ok(k_out_stride, H, D))))
        return VIT_ERR_BAD_STRIDE;
    if ((has_q && q_in == q_out && q_in_stride != q_out_stride) ||
        (has_k && k_in == k_out && k_in_stride != k_out_stride))
        return VIT_ERR_BAD_STRIDE;
    if ((has_q && (!aligned16(q_in) || !aligned16(q_out))) || (has_k && (!aligned16(k_in) || !aligned16(k_out))) ||
        ((uintptr_t)pos_hw & 7u) || ((uintptr_t)inv_freq & 3u) || ((uintptr_t)norm_w & 1u))
        return VIT_ERR_MISALIGNED;
    int sms = 0;
    vit_status_t st = device_info(&sms);
    if (st != VIT_OK) return st;
    return from_cuda(launch_qk_norm_rope(q_in, q_out, k_in, k_out, T, H, D, q_in_stride, q_out_stride, k_in_stride,
                                         k_out_stride, pos_hw, inv_freq, norm_w, eps,
                                         rope_mode == VIT_ROPE_INTERLEAVED, sms, status_dev, (cudaStream_t)stream));
}

vit_status_t vit_qk_norm_rope_ex(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T, int H,
                                 int D, int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride,
                                 int64_t k_out_stride, const int32_t *pos_hw, const float *inv_freq,
                                 const void *norm_w, float eps, int rope_mode, int32_t *status_dev,
                                 vit_stream_t stream)
{
    TraceRange trace("vit_qk_norm_rope_ex");
    return qk_norm_rope_impl(q_in, q_out, k_in, k_out, T, H, D, q_in_stride, q_out_stride, k_in_stride, k_out_stride,
                             pos_hw, inv_freq, norm_w, eps, rope_mode, status_dev, stream);
}

vit_status_t vit_qk_norm_rope(const void *q_in, void *q_out, const void *k_in, void *k_out, int64_t T, int H, int D,
                              int64_t q_in_stride, int64_t q_out_stride, int64_t k_in_stride, int64_t k_out_stride,
                              const int32_t *pos_hw, const float *inv_freq, const void *norm_w, float eps,
                              vit_stream_t stream)
{
    TraceRange trace("vit_qk_norm_rope");
    return qk_norm_rope_impl(q_in, q_out, k_in, k_out, T, H, D, q_in_stride, q_out_stride, k_in_stride, k_out_stride,
                             pos_hw, inv_freq, norm_w, eps, VIT_ROPE_ROTATE_HALF, nullptr, stream);
}

vit_status_t vit_rope_table(const float *inv_freq, int head_dim, int max_pos, float *cos_sin, vit_stream_t stream)
{
    TraceRange trace("vit_rope_table");
    if (!head_dim_ok(head_dim)) return VIT_ERR_BAD_HEAD_DIM;
    if (max_pos < 1) return VIT_ERR_BAD_ARGUMENT;
    if (!inv_freq || !cos_sin) return VIT_ERR_NULL_POINTER;
    if (((uintptr_t)inv_freq & 3u) || !aligned16(cos_sin)) return VIT_ERR_MISALIGNED;
    vit_status_t st = device_info(nullptr);
    if (st != VIT_OK) return st;
    return from_cuda(launch_rope_table(inv_freq, head_dim / 4, max_pos, cos_sin, (cudaStream_t)stream));
}

size_t vit_varlen_attn_workspace_size(int64_t T, int H, int B, int D)
{
    if (T < 0 || T >= kMaxTokens || H < 1 || B < 0 || B > VIT_MAX_SEGMENTS || !head_dim_ok(D)) return 0;
    // a tiny segment is one item per head and a long one at least 128 query rows per item, so
    // this bound holds for any kernel split; item indices are int32 on the device
    const int64_t items = max_items(T, H, B, 64);
    if (items >= ((int64_t)1 << 31)) return 0;
    return sizeof(WsHeader) + sizeof(Item) * (size_t)items;
}

}  // extern "C"

namespace vit {

// Every host-side check of the attention calls except those of the workspace.
// *nothing is set when the call has no work at all (no segments and no tokens).
vit_status_t check_varlen_attn_args(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                    int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                    const vit_q_rope_t *q_rope, const int32_t *cu_seqlens, const int32_t *seq_start,
                                    const int32_t *seq_len, int B, int max_seqlen, float scale, const void *out,
                                    int64_t out_stride, const float *lse, const vit_attn_options_t *opts,
                                    bool *nothing)
{
    const bool padded = seq_len != nullptr;
    *nothing = false;
    if (!head_dim_ok(D)) return VIT_ERR_BAD_HEAD_DIM;
    if (T < 0 || T >= kMaxTokens || H < 1 || H >= kMaxHeads || B < 0) return VIT_ERR_BAD_SHAPE;
    if (B > VIT_MAX_SEGMENTS) return VIT_ERR_TOO_MANY_SEGMENTS;
    if (B == 0) {
        *nothing = T == 0;
        return T == 0 ? VIT_OK : VIT_ERR_BAD_SHAPE;
    }
    if (max_seqlen < 0) return VIT_ERR_BAD_ARGUMENT;
    if (isnan(scale) || isinf(scale)) return VIT_ERR_BAD_ARGUMENT;
    if (padded) {
        if (!seq_start) return VIT_ERR_NULL_POINTER;
        if (((uintptr_t)seq_start & 3u) || ((uintptr_t)seq_len & 3u)) return VIT_ERR_MISALIGNED;
    } else if (!cu_seqlens && T % B != 0) {
        return VIT_ERR_BAD_ARGUMENT;
    }
    if ((uintptr_t)cu_seqlens & 3u) return VIT_ERR_MISALIGNED;
    if (T > 0) {
        if (!q || !k || !v || !out) return VIT_ERR_NULL_POINTER;
        if (!stride_ok(q_stride, H, D) || !stride_ok(k_stride, H, D) || !stride_ok(v_stride, H, D) ||
            !stride_ok(out_stride, H, D))
            return VIT_ERR_BAD_STRIDE;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return VIT_ERR_MISALIGNED;
        if ((uintptr_t)lse & 3u) return VIT_ERR_MISALIGNED;
    }
    if (q_rope && T > 0) {
        if (!q_rope->pos_hw || !q_rope->cos_sin) return VIT_ERR_NULL_POINTER;
        if (q_rope->max_pos < 1) return VIT_ERR_BAD_ARGUMENT;
        if (!(q_rope->eps >= 0.f) || !isfinite(q_rope->eps)) return VIT_ERR_BAD_ARGUMENT;
        if (q_rope->rope_mode != VIT_ROPE_ROTATE_HALF && q_rope->rope_mode != VIT_ROPE_INTERLEAVED)
            return VIT_ERR_BAD_ARGUMENT;
        if (((uintptr_t)q_rope->pos_hw & 7u) || !aligned16(q_rope->cos_sin) || !aligned16(q_rope->norm_w))
            return VIT_ERR_MISALIGNED;
    }
    if (opts && opts->short_segment_max < -1) return VIT_ERR_BAD_ARGUMENT;
    if (vit_varlen_attn_workspace_size(T, H, B, D) == 0) return VIT_ERR_BAD_SHAPE;
    return VIT_OK;
}

vit_status_t check_device() { return device_info(nullptr); }

}  // namespace vit

namespace {

vit_status_t varlen_attn_impl(const void *q, const void *k, const void *v, int64_t T, int H, int D, int64_t q_stride,
                              int64_t k_stride, int64_t v_stride, const vit_q_rope_t *q_rope,
                              const int32_t *cu_seqlens, const int32_t *seq_start, const int32_t *seq_len, int B,
                              int max_seqlen, float scale, void *out, int64_t out_stride, float *lse,
                              const vit_attn_options_t *opts, void *workspace, size_t workspace_bytes,
                              int32_t *status_dev, vit_stream_t stream)
{
    const bool padded = seq_len != nullptr;
    bool nothing = false;
    vit_status_t st = check_varlen_attn_args(q, k, v, T, H, D, q_stride, k_stride, v_stride, q_rope, cu_seqlens,
                                             seq_start, seq_len, B, max_seqlen, scale, out, out_stride, lse, opts,
                                             &nothing);
    if (st != VIT_OK || nothing) return st;
    // 0 = not given: every segment lies inside [0, T), so T bounds it. ([TS] _varlen_metadata
    // derives the exact maximum with a device-to-host read instead; a bound is all that is
    // needed here, and taking T keeps the call free of host synchronisation.)
    if (max_seqlen == 0) max_seqlen = (int)T;
    if (!workspace) return VIT_ERR_NULL_POINTER;
    if (!aligned16(workspace)) return VIT_ERR_MISALIGNED;
    if (workspace_bytes < vit_varlen_attn_workspace_size(T, H, B, D)) return VIT_ERR_WORKSPACE_TOO_SMALL;

    int sms = 0;
    st = device_info(&sms);
    if (st != VIT_OK) return st;
    if (scale <= 0.f) scale = 1.0f / sqrtf((float)D);
    cudaStream_t s = (cudaStream_t)stream;

    WsHeader *hdr = static_cast<WsHeader *>(workspace);
    Item *items = reinterpret_cast<Item *>(hdr + 1);
    SchedParams sp;
    const int split = (opts && opts->short_segment_max >= 0) ? opts->short_segment_max : kDefaultShortMax;
    sp.tiny_max = split < attn_tiny_max() ? split : attn_tiny_max();
    sp.bm_long = attn_long_bm();
    sp.num_sms = sms;
    // the scheduler divides by this with shifts
    if (sp.bm_long & (sp.bm_long - 1)) return VIT_ERR_BAD_ARGUMENT;
    cudaError_t e = launch_schedule(padded ? nullptr : cu_seqlens, seq_start, seq_len, B, T, H, max_seqlen, sp, hdr,
                                    items, status_dev, s);
    if (e != cudaSuccess) return VIT_ERR_CUDA;
    if (T == 0) return VIT_OK;
    AttnArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.T = T;
    a.H = H;
    a.D = D;
    a.q_stride = q_stride;
    a.k_stride = k_stride;
    a.v_stride = v_stride;
    a.out_stride = out_stride;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.hdr = hdr;
    a.items = items;
    a.status = status_dev;
    a.fuse_q = q_rope != nullptr;
    a.qr = rope::QRope{};
    if (q_rope) {
        a.qr.pos_hw = reinterpret_cast<const int2 *>(q_rope->pos_hw);
        a.qr.cos_sin = reinterpret_cast<const float4 *>(q_rope->cos_sin);
        a.qr.norm_w = static_cast<const uint4 *>(q_rope->norm_w);
        a.qr.max_pos = q_rope->max_pos;
        a.qr.eps = q_rope->eps;
        a.qr.interleaved = q_rope->rope_mode == VIT_ROPE_INTERLEAVED;
        a.qr.status = status_dev;
    }
    // a segment can only be long when the bound allows it
    const int64_t longest = (cu_seqlens || padded) ? (int64_t)max_seqlen : T / B;
    a.max_len = longest;
    if (longest > sp.tiny_max) {
        // split items cover bm_long / 2 rows, so that many more items may exist
        e = launch_attn_long(a, max_items(T, H, B, sp.bm_long / 2), sms, stall_v(), s);
        if (e != cudaSuccess) return VIT_ERR_CUDA;
    }
    // segments of at most tiny_max tokens on the tiny-segment kernel, launched only when that
    // class can be non-empty: the host knows the shortest segment only for one packed segment
    // (T tokens) and for uniform segments (T / B each); an empty launch still costs ~6 us
    const int64_t shortest = padded ? 0 : (!cu_seqlens ? T / B : (B == 1 ? T : 0));
    if (sp.tiny_max > 0 && shortest <= sp.tiny_max) e = launch_attn_tiny(a, (int64_t)H * B, sms, s);
    return from_cuda(e);
}

}  // namespace

extern "C" {

vit_status_t vit_varlen_attn_lse(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                 int64_t q_stride, int64_t k_stride, int64_t v_stride, const int32_t *cu_seqlens,
                                 int B, int max_seqlen, float scale, void *out, int64_t out_stride, float *lse,
                                 void *workspace, size_t workspace_bytes, int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_varlen_attn_lse");
    return varlen_attn_impl(q, k, v, T, H, D, q_stride, k_stride, v_stride, nullptr, cu_seqlens, nullptr, nullptr, B,
                            max_seqlen, scale, out, out_stride, lse, nullptr, workspace, workspace_bytes, status_dev,
                            stream);
}

vit_status_t vit_varlen_attn_fused_q(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                     int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                     const vit_q_rope_t *q_rope, const int32_t *cu_seqlens, int B, int max_seqlen,
                                     float scale, void *out, int64_t out_stride, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_varlen_attn_fused_q");
    if (!q_rope) return VIT_ERR_NULL_POINTER;
    return varlen_attn_impl(q, k, v, T, H, D, q_stride, k_stride, v_stride, q_rope, cu_seqlens, nullptr, nullptr, B,
                            max_seqlen, scale, out, out_stride, lse, nullptr, workspace, workspace_bytes, status_dev,
                            stream);
}

vit_status_t vit_varlen_attn_padded(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                    int64_t q_stride, int64_t k_stride, int64_t v_stride, const int32_t *seq_start,
                                    const int32_t *seq_len, int B, int max_seqlen, float scale, void *out,
                                    int64_t out_stride, float *lse, const vit_q_rope_t *q_rope, void *workspace,
                                    size_t workspace_bytes, int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_varlen_attn_padded");
    if (!head_dim_ok(D)) return VIT_ERR_BAD_HEAD_DIM;
    if (T < 0 || T >= kMaxTokens || H < 1 || B < 0) return VIT_ERR_BAD_SHAPE;
    if (B == 0) return VIT_OK;                           // every row is padding: nothing to compute
    if (!seq_len || !seq_start) return VIT_ERR_NULL_POINTER;
    return varlen_attn_impl(q, k, v, T, H, D, q_stride, k_stride, v_stride, q_rope, nullptr, seq_start, seq_len, B,
                            max_seqlen, scale, out, out_stride, lse, nullptr, workspace, workspace_bytes, status_dev,
                            stream);
}

vit_status_t vit_varlen_attn(const void *q, const void *k, const void *v, int64_t T, int H, int D, int64_t q_stride,
                             int64_t k_stride, int64_t v_stride, const int32_t *cu_seqlens, int B, int max_seqlen,
                             float scale, void *out, int64_t out_stride, void *workspace, size_t workspace_bytes,
                             int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_varlen_attn");
    return varlen_attn_impl(q, k, v, T, H, D, q_stride, k_stride, v_stride, nullptr, cu_seqlens, nullptr, nullptr, B,
                            max_seqlen, scale, out, out_stride, nullptr, nullptr, workspace, workspace_bytes,
                            status_dev, stream);
}

vit_status_t vit_varlen_attn_ex(const void *q, const void *k, const void *v, int64_t T, int H, int D,
                                int64_t q_stride, int64_t k_stride, int64_t v_stride, const int32_t *cu_seqlens,
                                const int32_t *seq_start, const int32_t *seq_len, int B, int max_seqlen, float scale,
                                void *out, int64_t out_stride, float *lse, const vit_q_rope_t *q_rope,
                                const vit_attn_options_t *opts, void *workspace, size_t workspace_bytes,
                                int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_varlen_attn_ex");
    if (seq_len || seq_start) {
        if (cu_seqlens) return VIT_ERR_BAD_ARGUMENT;   // one layout or the other
        if (!head_dim_ok(D)) return VIT_ERR_BAD_HEAD_DIM;
        if (T < 0 || T >= kMaxTokens || H < 1 || B < 0) return VIT_ERR_BAD_SHAPE;
        if (B == 0) return VIT_OK;
        if (!seq_len || !seq_start) return VIT_ERR_NULL_POINTER;
    }
    return varlen_attn_impl(q, k, v, T, H, D, q_stride, k_stride, v_stride, q_rope, cu_seqlens, seq_start, seq_len, B,
                            max_seqlen, scale, out, out_stride, lse, opts, workspace, workspace_bytes, status_dev,
                            stream);
}

#ifdef VIT_TEST_HOOKS
int vit_debug_stall_long_kernel(int enable)
{
    return g_stall_v.exchange(enable ? 1 : 0);
}
#endif

vit_status_t vit_read_status(const int32_t *status_dev, vit_stream_t stream)
{
    TraceRange trace("vit_read_status");
    if (!status_dev) return VIT_ERR_NULL_POINTER;
    int32_t h = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&h, status_dev, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return VIT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VIT_ERR_CUDA;
    return h;
}

}  // extern "C"
