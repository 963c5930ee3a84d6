// pre_noalloc.cu -- mhc_pre_delayed_noalloc: the delayed pre block for
// callers that cannot allocate device memory.
//
// Who needs this: mhc_pre_delayed takes a caller-provided workspace (the
// per-call copy of fn split into three bf16 planes that the tensor-core
// kernel streams from).  Some callers have no way to provide one: a serving
// engine that reserves all free device memory for its caches up front and
// forbids any later cudaMalloc, a plugin that only receives tensors from its
// host application and owns no allocator, or a latency-critical path where
// cudaMalloc's implicit device synchronisation is not acceptable.  This entry
// point runs the same tensor-core kernel with its scratch in a fixed array
// that lives in this file; it never calls cudaMalloc, cudaFree or any
// allocating routine.
//
// The array holds one copy of the fn planes (16 x 10 x 18 KB = 2,949,120
// bytes at C = 5120), packed by one launch over the whole GPU; the kernel
// then runs on every co-resident cluster, as mhc_pre_delayed does.  Every GPU
// that loads the library holds the array until the process exits.
#include "../../include/mhc.h"

#include <cuda_runtime.h>

#include <mutex>

namespace mhc {
bool pre_tc_supports(int C);
int pre_tc_prepare();
size_t pre_tc_packed_bytes(int C);
cudaError_t launch_pre_tc_pack(const float* fn, int C, void* out, cudaStream_t stream);
cudaError_t launch_pre_tc(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                          const float* alpha, const uint16_t* norm_w, int64_t T, int C, int iters,
                          float rms_eps, float norm_eps, float sk_eps, float* pre_out, float* post_out,
                          float* comb_out, uint16_t* layer_input, float* logits_out, void* workspace,
                          cudaStream_t stream, int max_clusters, bool broadcast, bool gates_only,
                          const void* packed);
}  // namespace mhc

namespace {

constexpr size_t kNoAllocBytes = MHC_NOALLOC_SCRATCH_BYTES;
// Every shape the entry point accepts fits: C is at most 5120 (the
// tensor-core kernel's limit, checked first), i.e. at most 10 stages of
// 18 KB of planes for each of the 16 CTA ranks.
static_assert((size_t)16 * 10 * 18432 <= kNoAllocBytes, "the scratch array holds the planes of every accepted shape");

// The scratch itself.  Its name is a host-side stand-in in host code, not a
// device address: host code uses the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
int g_clusters[kMaxDevices] = {};   // co-resident tensor-core clusters; 0 = not set up

// Once per device, with that device current: resolve the array's device
// address and set up the kernel (attributes, occupancy).  No allocation.
bool setup(int dev, void** scratch, int* clusters) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return false;
        const int n = mhc::pre_tc_prepare();
        if (n <= 0) return false;
        g_clusters[dev] = n;
        g_scratch_ptr[dev] = p;
    }
    *scratch = g_scratch_ptr[dev];
    *clusters = g_clusters[dev];
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" mhc_status mhc_pre_delayed_noalloc(const uint16_t* x, const float* pre_in, const float* fn,
                                              const float* bias, const float* alpha,
                                              const uint16_t* norm_weight, int64_t T, int n, int C,
                                              int sinkhorn_iters, float rms_eps, float norm_eps,
                                              float sinkhorn_eps, float* pre_out, float* post_out,
                                              float* comb_out, uint16_t* layer_input, float* logits_out,
                                              void* stream) {
    if (T < 0 || n < 1 || C < 1 || sinkhorn_iters < 1) return MHC_ERR_INVALID_ARGUMENT;
    if (n != 4 || !mhc::pre_tc_supports(C)) return MHC_ERR_UNSUPPORTED;
    if (!(rms_eps >= 0.f) || !(norm_eps >= 0.f) || !(sinkhorn_eps >= 0.f)) return MHC_ERR_INVALID_ARGUMENT;
    if (T == 0) return MHC_OK;
    if (T > ((int64_t)1 << 40) / ((int64_t)n * C)) return MHC_ERR_UNSUPPORTED;
    const void* req[] = {x, pre_in, fn, bias, alpha, pre_out, post_out, comb_out, layer_input};
    for (const void* p : req)
        if (!p || !aligned16(p)) return MHC_ERR_INVALID_ARGUMENT;
    if ((norm_weight && !aligned16(norm_weight)) || (logits_out && !aligned16(logits_out)))
        return MHC_ERR_INVALID_ARGUMENT;
    const int M = 2 * n + n * n;
    const size_t xb = (size_t)T * n * C * 2, pb = (size_t)T * n * 4, cb = (size_t)T * n * n * 4;
    const size_t lib = (size_t)T * C * 2, lob = (size_t)T * M * 4;
    const size_t fnb = (size_t)M * n * C * 4, bb = (size_t)M * 4, ab = 12, nwb = (size_t)C * 2;
    struct R { const void* p; size_t n; };
    const R ins[] = {{x, xb}, {pre_in, pb}, {fn, fnb}, {bias, bb}, {alpha, ab}, {norm_weight, nwb}};
    const R outs[] = {{pre_out, pb}, {post_out, pb}, {comb_out, cb}, {layer_input, lib}, {logits_out, lob}};
    for (const R& o : outs) {
        for (const R& i : ins)
            if (overlaps(o.p, o.n, i.p, i.n)) return MHC_ERR_INVALID_ARGUMENT;
        for (const R& o2 : outs)
            if (&o != &o2 && overlaps(o.p, o.n, o2.p, o2.n)) return MHC_ERR_INVALID_ARGUMENT;
    }
    // one copy of the planes fits the array (host arithmetic only: nothing
    // has been set up or launched yet)
    if (mhc::pre_tc_packed_bytes(C) > kNoAllocBytes) return MHC_ERR_UNSUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHC_ERR_CUDA;
    // The scratch address below belongs to the current device: x and the
    // stream must belong to it too, or the kernel would run on another GPU
    // with this one's address.  Checked before anything is set up or launched.
    cudaPointerAttributes pa = {};
    if (cudaPointerGetAttributes(&pa, x) != cudaSuccess) {
        (void)cudaGetLastError();
        return MHC_ERR_INVALID_ARGUMENT;
    }
    if ((pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged) || pa.device != dev)
        return MHC_ERR_INVALID_ARGUMENT;
    if (stream) {
        int sdev = -1;
        if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
            (void)cudaGetLastError();
            return MHC_ERR_INVALID_ARGUMENT;
        }
        if (sdev != dev) return MHC_ERR_INVALID_ARGUMENT;
    }
    void* scratch = nullptr;
    int clusters = 0;
    if (!setup(dev, &scratch, &clusters)) return MHC_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = mhc::launch_pre_tc_pack(fn, C, scratch, s);
    if (e == cudaSuccess)
        e = mhc::launch_pre_tc(x, pre_in, fn, bias, alpha, norm_weight, T, C, sinkhorn_iters, rms_eps, norm_eps,
                               sinkhorn_eps, pre_out, post_out, comb_out, layer_input, logits_out, nullptr, s,
                               clusters, false, false, scratch);
    return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}
