// mhc_abi.cu -- the C ABI of libmhc.so (declared in include/mhc.h): host-side
// argument checks, launch-plan choice and the kernel launches.
#include "../../include/mhc.h"

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace mhc {
cudaError_t launch_post(const uint16_t* x, const uint16_t* y, const float* comb,
                        const float* post, int64_t T, int C, uint16_t* x_new,
                        cudaStream_t stream, int num_sms, bool overlap, bool broadcast);
cudaError_t launch_pre_cluster(const uint16_t* x, const float* pre_in, const float* fn,
                               const float* bias, const float* alpha, const uint16_t* norm_w,
                               int64_t T, int C, int iters, float rms_eps, float norm_eps,
                               float sk_eps, float* pre_out, float* post_out, float* comb_out,
                               uint16_t* layer_input, float* logits_out, cudaStream_t stream,
                               int max_clusters, bool overlap, const uint16_t* y, const float* comb_prev,
                               const float* post_prev, uint16_t* x_new, bool nondelayed, bool broadcast);
int pre_cluster_tile_tokens(int64_t T, int max_clusters);
int pre_cluster_max_tile();
int pre_cluster_ctas();
int pre_cluster_prepare(int C);
bool pre_tc_supports(int C);
int pre_tc_tile_tokens();
int pre_tc_prepare();
cudaError_t launch_pre_tc(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                          const float* alpha, const uint16_t* norm_w, int64_t T, int C, int iters,
                          float rms_eps, float norm_eps, float sk_eps, float* pre_out, float* post_out,
                          float* comb_out, uint16_t* layer_input, float* logits_out, void* workspace,
                          cudaStream_t stream, int max_clusters, bool broadcast, bool gates_only,
                          const void* packed);
size_t pre_tc_packed_bytes(int C);
cudaError_t launch_collapse_fold(const uint16_t* x, const float* pre, const uint16_t* norm_w, int64_t T, int C,
                                 bool broadcast, int clusters, float norm_eps, uint16_t* out, cudaStream_t stream,
                                 int num_sms);
cudaError_t launch_pre_tc_pack(const float* fn, int C, void* out, cudaStream_t stream);
cudaError_t read_device_status(unsigned int* status);
cudaError_t read_decode_status(unsigned int* status);
cudaError_t read_collapse_status(unsigned int* status);
}  // namespace mhc

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxC = 6144;
// From this many tokens on, the tensor-core kernel (128-token tiles) runs the
// pre block; below it the cluster kernel (tiles of up to 32 tokens, one per
// cluster, warp-level MMA) has lower latency.
constexpr int64_t kTcMinTokens = 256;

// Per-device cache: SM count, and the cluster kernel's set-up result per
// hidden size (the kernel instance, and with it the occupancy, depends on C
// only through the number of 8-column groups per CTA).
struct DeviceInfo {
    int num_sms = 0;
    int tc_clusters = -1;  // -1: not yet set up; 0: unavailable
    int cached_C[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int cached_clusters[8] = {0, 0, 0, 0, 0, 0, 0, 0};
};

std::mutex g_mutex;
// Programmatic dependent launch for the decode pre kernel and the post kernel
// (mhc_set_launch_overlap); off by default.
std::atomic<int> g_launch_overlap{0};
DeviceInfo g_dev[kMaxDevices];

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}

int num_sms(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev[dev].num_sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_dev[dev].num_sms = n;
    }
    return g_dev[dev].num_sms;
}

// Maximum co-resident clusters of the pre kernel for hidden size C on device
// dev, after its one-time set-up; cached for up to 8 hidden sizes per device
// (others are set up at every call).  0 on error.
int max_clusters(int dev, int C) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_dev[dev];
    for (int i = 0; i < 8; ++i)
        if (d.cached_C[i] == C) return d.cached_clusters[i];
    int n = mhc::pre_cluster_prepare(C);
    if (n <= 0) return 0;
    for (int i = 0; i < 8; ++i)
        if (d.cached_C[i] == 0) {
            d.cached_C[i] = C;
            d.cached_clusters[i] = n;
            break;
        }
    return n;
}

int tc_clusters(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev[dev].tc_clusters < 0) g_dev[dev].tc_clusters = mhc::pre_tc_prepare();
    return g_dev[dev].tc_clusters;
}

bool use_tc(int64_t T, int C) { return T >= kTcMinTokens && mhc::pre_tc_supports(C); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

// mhc_pre from 256 tokens: the first tensor-core pass's pre-mix [T][4]
size_t nondelayed_scratch_bytes(int64_t T) { return ((size_t)T * 16 + 255) / 256 * 256; }

mhc_status check_pre_shape(int64_t T, int n, int C, int iters) {
    if (T < 0 || n < 1 || C < 1 || iters < 1) return MHC_ERR_INVALID_ARGUMENT;
    if (n != 4 || C % 8 != 0 || C > kMaxC) return MHC_ERR_UNSUPPORTED;
    if (T > ((int64_t)1 << 40) / ((int64_t)n * C)) return MHC_ERR_UNSUPPORTED;
    return MHC_OK;
}

}  // namespace

extern "C" {

const char* mhc_status_string(mhc_status s) {
    switch (s) {
        case MHC_OK: return "MHC_OK";
        case MHC_ERR_INVALID_ARGUMENT: return "MHC_ERR_INVALID_ARGUMENT: null, misaligned or overlapping pointer, or bad count";
        case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: shape this library does not handle (n must be 4, C a multiple of 8 up to 6144)";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: a CUDA runtime call or kernel launch failed";
        case MHC_ERR_TIMEOUT: return "MHC_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "unknown mhc_status";
}

int mhc_version(void) { return (0 << 16) | 3; }

int mhc_set_launch_overlap(int enable) { return g_launch_overlap.exchange(enable ? 1 : 0); }

mhc_status mhc_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MHC_ERR_CUDA;
    unsigned int v = 0, w = 0, c = 0;
    if (mhc::read_device_status(&v) != cudaSuccess) return MHC_ERR_CUDA;
    if (mhc::read_decode_status(&w) != cudaSuccess) return MHC_ERR_CUDA;
    if (mhc::read_collapse_status(&c) != cudaSuccess) return MHC_ERR_CUDA;
    return (v | w | c) ? MHC_ERR_TIMEOUT : MHC_OK;
}

mhc_status mhc_pre_delayed_plan(int64_t T, int n, int C, int* kernel, int* grid, int* cluster,
                                int* tokens_per_tile) {
    mhc_status st = check_pre_shape(T, n, C, 1);
    if (st != MHC_OK) return st;
    const bool tc = use_tc(T, C);
    if (kernel) *kernel = tc ? 2 : 1;
    if (cluster) *cluster = mhc::pre_cluster_ctas();
    int dev = T > 0 && (grid || tokens_per_tile) ? current_device() : -1;
    int mc = dev < 0 ? 0 : (tc ? tc_clusters(dev) : max_clusters(dev, C));
    int tt = tc ? mhc::pre_tc_tile_tokens()
                : (mc > 0 ? mhc::pre_cluster_tile_tokens(T, mc)
                          : (int)(T < mhc::pre_cluster_max_tile() ? (T > 0 ? T : 1) : mhc::pre_cluster_max_tile()));
    if (tokens_per_tile) *tokens_per_tile = tt;
    if (grid) {
        *grid = 0;
        if (T > 0 && mc > 0) {
            int64_t tiles = (T + tt - 1) / tt;
            *grid = (int)((tiles < mc ? tiles : mc) * mhc::pre_cluster_ctas());
        }
    }
    return MHC_OK;
}

size_t mhc_pre_workspace_bytes(int64_t T, int n, int C) {
    if (check_pre_shape(T, n, C, 1) != MHC_OK || T == 0 || !use_tc(T, C)) return 0;
    int dev = current_device();
    if (dev < 0) return 0;
    int tcc = tc_clusters(dev);
    // one copy of fn's planes, then (mhc_pre only) the first pass's pre-mix
    return tcc > 0 ? mhc::pre_tc_packed_bytes(C) + nondelayed_scratch_bytes(T) : 0;
}

}  // extern "C"

namespace {

struct Span { const void* p; size_t n; };

// Host-side checks shared by the pre entry points, then the launch(es).
// fused: the previous seam's post runs first on x (into x_new) and the pre
// block reads x_new.  nondelayed: the collapse takes the token's own pre-mix
// (no pre_in).  bcast: x is [T, C], read as every one of the n streams.
mhc_status pre_entry(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                     const float* alpha, const uint16_t* norm_weight, int64_t T, int n, int C,
                     int sinkhorn_iters, float rms_eps, float norm_eps, float sinkhorn_eps, float* pre_out,
                     float* post_out, float* comb_out, uint16_t* layer_input, float* logits_out, void* workspace,
                     size_t workspace_bytes, void* stream, bool fused, const uint16_t* y, const float* comb_prev,
                     const float* post_prev, uint16_t* x_new, bool nondelayed = false, bool bcast = false,
                     const void* packed = nullptr, size_t packed_bytes = 0) {
    mhc_status st = check_pre_shape(T, n, C, sinkhorn_iters);
    if (st != MHC_OK) return st;
    if (!(rms_eps >= 0.f) || !(norm_eps >= 0.f) || !(sinkhorn_eps >= 0.f)) return MHC_ERR_INVALID_ARGUMENT;
    if (T == 0) return MHC_OK;
    const void* req[] = {x, nondelayed ? fn : pre_in, fn, bias, alpha, pre_out, post_out, comb_out, layer_input};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MHC_ERR_INVALID_ARGUMENT;
    if (fused) {
        const void* req2[] = {y, comb_prev, post_prev, x_new};
        for (const void* p : req2)
            if (!p || !aligned16(p)) return MHC_ERR_INVALID_ARGUMENT;
    }
    if ((norm_weight && !aligned16(norm_weight)) || (logits_out && !aligned16(logits_out)))
        return MHC_ERR_INVALID_ARGUMENT;
    const int M = 2 * n + n * n;
    if (fused && bcast) return MHC_ERR_INVALID_ARGUMENT;
    if (packed && (fused || bcast || nondelayed)) return MHC_ERR_INVALID_ARGUMENT;
    if (packed && (!mhc::pre_tc_supports(C) || packed_bytes < mhc::pre_tc_packed_bytes(C) ||
                   (reinterpret_cast<uintptr_t>(packed) & 255u)))
        return MHC_ERR_INVALID_ARGUMENT;
    const size_t xb = (size_t)T * (bcast ? 1 : n) * C * 2, pb = (size_t)T * n * 4, cb = (size_t)T * n * n * 4;
    const size_t lib = (size_t)T * C * 2, lob = (size_t)T * M * 4;
    const size_t fnb = (size_t)M * n * C * 4, bb = (size_t)M * 4, ab = 12, nwb = (size_t)C * 2;
    // Exact aliases allowed when fused: x_new == x, comb_out == comb_prev,
    // post_out == post_prev (each is read, for a token, before it is written).
    const Span ins[] = {{x, xb}, {nondelayed ? nullptr : pre_in, pb}, {fn, fnb}, {bias, bb}, {alpha, ab},
                        {norm_weight, nwb}, {packed, packed_bytes},
                        {fused ? y : nullptr, lib}, {fused ? comb_prev : nullptr, cb},
                        {fused ? post_prev : nullptr, pb}};
    const Span outs[] = {{pre_out, pb}, {post_out, pb}, {comb_out, cb}, {layer_input, lib}, {logits_out, lob},
                         {workspace, workspace_bytes}, {fused ? x_new : nullptr, xb}};
    for (const Span& o : outs) {
        for (const Span& i : ins) {
            const bool exact_alias = fused && o.p == i.p &&
                                     ((o.p == x_new && i.p == x) || (o.p == comb_out && i.p == comb_prev) ||
                                      (o.p == post_out && i.p == post_prev));
            if (!exact_alias && overlaps(o.p, o.n, i.p, i.n)) return MHC_ERR_INVALID_ARGUMENT;
        }
        for (const Span& o2 : outs)
            if (&o != &o2 && overlaps(o.p, o.n, o2.p, o2.n)) return MHC_ERR_INVALID_ARGUMENT;
    }
    int dev = current_device();
    if (dev < 0) return MHC_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool overlap = g_launch_overlap.load() != 0;
    if (use_tc(T, C)) {
        int tcc = tc_clusters(dev);
        if (tcc > 0) {
            // fn's planes: packed by the caller, or packed here into the
            // workspace by one launch over the whole GPU ahead of the kernel
            // (one shared copy instead of a conversion in every cluster's
            // prologue before its first MMA)
            const size_t planes = packed ? 0 : mhc::pre_tc_packed_bytes(C);
            const size_t need = planes + (nondelayed ? nondelayed_scratch_bytes(T) : 0);
            if (workspace_bytes < need || (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))))
                return MHC_ERR_INVALID_ARGUMENT;
            if (!packed) {
                if (mhc::launch_pre_tc_pack(fn, C, workspace, s) != cudaSuccess) return MHC_ERR_CUDA;
                packed = workspace;
            }
            if (nondelayed) {
                // pass 1: the gates only (no collapse, fold or layer_input),
                // its unused pre_in pointed at the workspace scratch; pass 2:
                // the collapse and fold with pass 1's pre as an HBM stream,
                // in the tensor-core kernel's order (so the same bits as the
                // delayed block fed that pre)
                float* scratch = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + planes);
                cudaError_t e = mhc::launch_pre_tc(x, scratch, fn, bias, alpha, norm_weight, T, C, sinkhorn_iters,
                                                   rms_eps, norm_eps, sinkhorn_eps, pre_out, post_out, comb_out,
                                                   layer_input, logits_out, workspace, s, tcc, bcast, true,
                                                   packed);
                if (e == cudaSuccess) {
                    const int64_t ntiles = (T + 127) / 128;
                    const int ncl = ntiles < tcc ? (int)ntiles : tcc;
                    const int sms = num_sms(dev);
                    e = sms > 0 ? mhc::launch_collapse_fold(x, pre_out, norm_weight, T, C, bcast, ncl, norm_eps,
                                                            layer_input, s, sms)
                                : cudaErrorInvalidValue;
                }
                return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
            }
            const uint16_t* xin = x;
            if (fused) {   // large T: the post kernel, then the tensor-core pre on x_new
                int sms = num_sms(dev);
                if (sms <= 0) return MHC_ERR_CUDA;
                if (mhc::launch_post(x, y, comb_prev, post_prev, T, C, x_new, s, sms, overlap, false) != cudaSuccess)
                    return MHC_ERR_CUDA;
                xin = x_new;
            }
            cudaError_t e = mhc::launch_pre_tc(xin, pre_in, fn, bias, alpha, norm_weight, T, C, sinkhorn_iters,
                                               rms_eps, norm_eps, sinkhorn_eps, pre_out, post_out, comb_out,
                                               layer_input, logits_out, workspace, s, tcc, bcast, false,
                                               packed);
            return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
        }
    }
    int mc = max_clusters(dev, C);
    if (mc <= 0) return MHC_ERR_CUDA;
    cudaError_t e = mhc::launch_pre_cluster(x, pre_in, fn, bias, alpha, norm_weight, T, C, sinkhorn_iters, rms_eps,
                                            norm_eps, sinkhorn_eps, pre_out, post_out, comb_out, layer_input,
                                            logits_out, s, mc, overlap, fused ? y : nullptr,
                                            fused ? comb_prev : nullptr, fused ? post_prev : nullptr,
                                            fused ? x_new : nullptr, nondelayed, bcast);
    return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}

}  // namespace

extern "C" {

mhc_status mhc_pre_delayed(const uint16_t* x, const float* pre_in, const float* fn,
                           const float* bias, const float* alpha, const uint16_t* norm_weight,
                           int64_t T, int n, int C, int sinkhorn_iters, float rms_eps,
                           float norm_eps, float sinkhorn_eps, float* pre_out, float* post_out,
                           float* comb_out, uint16_t* layer_input, float* logits_out,
                           void* workspace, size_t workspace_bytes, void* stream) {
    return pre_entry(x, pre_in, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, workspace, workspace_bytes,
                     stream, false, nullptr, nullptr, nullptr, nullptr);
}

size_t mhc_pre_packed_bytes(int n, int C) {
    if (n != 4 || C < 1 || C % 8 != 0 || C > kMaxC || !mhc::pre_tc_supports(C)) return 0;
    return mhc::pre_tc_packed_bytes(C);
}

mhc_status mhc_pre_pack(const float* fn, int n, int C, void* packed, size_t packed_bytes, void* stream) {
    if (n < 1 || C < 1) return MHC_ERR_INVALID_ARGUMENT;
    if (n != 4 || C % 8 != 0 || C > kMaxC || !mhc::pre_tc_supports(C)) return MHC_ERR_UNSUPPORTED;
    if (!fn || !packed || !aligned16(fn) || (reinterpret_cast<uintptr_t>(packed) & 255u)) return MHC_ERR_INVALID_ARGUMENT;
    const size_t need = mhc::pre_tc_packed_bytes(C);
    if (packed_bytes < need || overlaps(packed, need, fn, (size_t)24 * n * C * 4)) return MHC_ERR_INVALID_ARGUMENT;
    if (current_device() < 0) return MHC_ERR_CUDA;
    return mhc::launch_pre_tc_pack(fn, C, packed, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MHC_OK
                                                                                                    : MHC_ERR_CUDA;
}

mhc_status mhc_pre_delayed_packed(const uint16_t* x, const float* pre_in, const float* fn, const void* packed,
                                  size_t packed_bytes, const float* bias, const float* alpha,
                                  const uint16_t* norm_weight, int64_t T, int n, int C, int sinkhorn_iters,
                                  float rms_eps, float norm_eps, float sinkhorn_eps, float* pre_out, float* post_out,
                                  float* comb_out, uint16_t* layer_input, float* logits_out, void* stream) {
    if (!packed) return MHC_ERR_INVALID_ARGUMENT;
    return pre_entry(x, pre_in, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, nullptr, 0, stream, false,
                     nullptr, nullptr, nullptr, nullptr, false, false, packed, packed_bytes);
}

mhc_status mhc_pre(const uint16_t* x, const float* fn, const float* bias, const float* alpha,
                   const uint16_t* norm_weight, int64_t T, int n, int C, int sinkhorn_iters, float rms_eps,
                   float norm_eps, float sinkhorn_eps, float* pre_out, float* post_out, float* comb_out,
                   uint16_t* layer_input, float* logits_out, void* workspace, size_t workspace_bytes, void* stream) {
    return pre_entry(x, nullptr, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, workspace, workspace_bytes,
                     stream, false, nullptr, nullptr, nullptr, nullptr, true);
}

mhc_status mhc_post_pre_delayed(const uint16_t* x, const uint16_t* y, const float* comb, const float* post,
                                uint16_t* x_new, const float* pre_in, const float* fn, const float* bias,
                                const float* alpha, const uint16_t* norm_weight, int64_t T, int n, int C,
                                int sinkhorn_iters, float rms_eps, float norm_eps, float sinkhorn_eps,
                                float* pre_out, float* post_out, float* comb_out, uint16_t* layer_input,
                                float* logits_out, void* workspace, size_t workspace_bytes, void* stream) {
    return pre_entry(x, pre_in, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, workspace, workspace_bytes,
                     stream, true, y, comb, post, x_new);
}

mhc_status mhc_pre_delayed_broadcast(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                                     const float* alpha, const uint16_t* norm_weight, int64_t T, int n, int C,
                                     int sinkhorn_iters, float rms_eps, float norm_eps, float sinkhorn_eps,
                                     float* pre_out, float* post_out, float* comb_out, uint16_t* layer_input,
                                     float* logits_out, void* workspace, size_t workspace_bytes, void* stream) {
    return pre_entry(x, pre_in, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, workspace, workspace_bytes,
                     stream, false, nullptr, nullptr, nullptr, nullptr, false, true);
}

mhc_status mhc_pre_broadcast(const uint16_t* x, const float* fn, const float* bias, const float* alpha,
                             const uint16_t* norm_weight, int64_t T, int n, int C, int sinkhorn_iters,
                             float rms_eps, float norm_eps, float sinkhorn_eps, float* pre_out, float* post_out,
                             float* comb_out, uint16_t* layer_input, float* logits_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    return pre_entry(x, nullptr, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps, norm_eps,
                     sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, workspace, workspace_bytes,
                     stream, false, nullptr, nullptr, nullptr, nullptr, true, true);
}

}  // extern "C"

namespace {

// Host-side checks and the launch for mhc_post and mhc_post_broadcast
// (bcast: x is [T, C], every stream equal to it; x_new may not alias it).
mhc_status post_entry(const uint16_t* x, const uint16_t* y, const float* comb, const float* post,
                      int64_t T, int n, int C, uint16_t* x_new, void* stream, bool bcast) {
    if (T < 0 || n < 1 || C < 1) return MHC_ERR_INVALID_ARGUMENT;
    if (n != 4 || C % 8 != 0) return MHC_ERR_UNSUPPORTED;
    if (T == 0) return MHC_OK;
    const void* req[] = {x, y, comb, post, x_new};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MHC_ERR_INVALID_ARGUMENT;
    const size_t xb = (size_t)T * n * C * 2, xinb = bcast ? (size_t)T * C * 2 : xb;
    if ((bcast || (const void*)x_new != (const void*)x) && overlaps(x_new, xb, x, xinb))
        return MHC_ERR_INVALID_ARGUMENT;
    if (overlaps(x_new, xb, y, (size_t)T * C * 2) || overlaps(x_new, xb, comb, (size_t)T * n * n * 4) ||
        overlaps(x_new, xb, post, (size_t)T * n * 4))
        return MHC_ERR_INVALID_ARGUMENT;
    int dev = current_device();
    if (dev < 0) return MHC_ERR_CUDA;
    int sms = num_sms(dev);
    if (sms <= 0) return MHC_ERR_CUDA;
    cudaError_t e = mhc::launch_post(x, y, comb, post, T, C, x_new, static_cast<cudaStream_t>(stream), sms,
                                     g_launch_overlap.load() != 0, bcast);
    return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}

}  // namespace

extern "C" {

mhc_status mhc_post(const uint16_t* x, const uint16_t* y, const float* comb, const float* post,
                    int64_t T, int n, int C, uint16_t* x_new, void* stream) {
    return post_entry(x, y, comb, post, T, n, C, x_new, stream, false);
}

mhc_status mhc_post_broadcast(const uint16_t* x, const uint16_t* y, const float* comb, const float* post,
                              int64_t T, int n, int C, uint16_t* x_new, void* stream) {
    return post_entry(x, y, comb, post, T, n, C, x_new, stream, true);
}

}  // extern "C"
