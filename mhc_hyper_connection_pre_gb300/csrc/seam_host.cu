// seam_host.cu -- mhc_seam_host: one seam (the delayed pre block, then the
// post block on the same residual) with its activations in page-locked HOST
// memory.  The tokens are cut into chunks; each chunk's host->device copies,
// its two kernels and its device->host copies go to three streams, so that
// both directions of the host link and the kernels overlap (chunk k's
// kernels run while chunk k+1 comes in and chunk k-1 goes out).  Every chunk
// takes the kernel the whole call would take, and tokens are independent,
// so the results are bit-identical to mhc_pre_delayed followed by mhc_post
// on device copies of the same inputs.
#include "../../include/mhc.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kChunkTokens = 1024;  // a multiple of the tensor-core kernel's 128-token tile
constexpr int64_t kTcMinTokens = 256;   // the pre block's tensor-core threshold
constexpr int kSets = 2;                // device buffer sets in rotation (three measured the same)

// Internal streams and events, created once per device on first use and
// kept for the life of the process.
struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start, in_done[kSets], comp_done[kSets], out_done[kSets], end_in, end_out;
};
std::mutex g_pipe_mutex;
Pipe g_pipe[kMaxDevices];

bool make_pipe(Pipe& p) {
    if (p.ready) return true;
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.end_in, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.end_out, ef) == cudaSuccess;
    for (int b = 0; ok && b < kSets; ++b)
        ok = cudaEventCreateWithFlags(&p.in_done[b], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.comp_done[b], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.out_done[b], ef) == cudaSuccess;
    p.ready = ok;
    return ok;
}

// The chunks of a call over T tokens.  No chunk falls under 256 tokens
// (unless T does), so a call under 256 tokens stays on the cluster kernel
// and every chunk of a larger one takes the tensor-core kernel:
//  * below 512 tokens, one chunk;
//  * below 2048, two: half of T rounded down to the tile, then the rest;
//  * from 2048, a 256-token head (the first copies in wait for no kernel,
//    so a short head starts the pipeline sooner), 1024-token chunks, then
//    512 tokens plus what does not fill a 1024-token chunk, then a 256-token
//    tail (the last copies out follow the last kernels, so a short tail ends
//    it sooner).
struct Chunk {
    int64_t t0, n;
};
int64_t num_chunks(int64_t T) {
    if (T <= 0) return 0;
    if (T < 2 * kTcMinTokens) return 1;
    if (T < 2 * kChunkTokens) return 2;
    return (T - kChunkTokens) / kChunkTokens + 3;
}
Chunk chunk_of(int64_t T, int64_t k) {
    const int64_t nch = num_chunks(T);
    if (nch == 1) return {0, T};
    if (nch == 2) {
        const int64_t c = (T / 2) / 128 * 128;
        return k == 0 ? Chunk{0, c} : Chunk{c, T - c};
    }
    const int64_t body = nch - 3;   // 1024-token chunks
    if (k == 0) return {0, kTcMinTokens};
    if (k <= body) return {kTcMinTokens + (k - 1) * kChunkTokens, kChunkTokens};
    if (k == body + 1) {
        const int64_t t0 = kTcMinTokens + body * kChunkTokens;
        return {t0, T - kTcMinTokens - t0};
    }
    return {T - kTcMinTokens, kTcMinTokens};
}
// the largest chunk (the buffers of both sets are sized for it)
int64_t max_chunk(int64_t T) {
    const int64_t nch = num_chunks(T);
    if (nch <= 2) return nch == 0 ? 0 : chunk_of(T, nch - 1).n;
    const int64_t before_tail = chunk_of(T, nch - 2).n;   // 512 .. 1535 tokens
    return before_tail > kChunkTokens ? before_tail : kChunkTokens;
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

// Device buffers of one chunk set, in workspace order.
struct SetLayout {
    size_t x, y, pre_in, x_new, pre, post, comb, li, total;
};
SetLayout set_layout(int64_t cap, int n, int C) {
    SetLayout L;
    size_t o = 0;
    L.x = o;      o += up256((size_t)cap * n * C * 2);
    L.y = o;      o += up256((size_t)cap * C * 2);
    L.pre_in = o; o += up256((size_t)cap * n * 4);
    L.x_new = o;  o += up256((size_t)cap * n * C * 2);
    L.pre = o;    o += up256((size_t)cap * n * 4);
    L.post = o;   o += up256((size_t)cap * n * 4);
    L.comb = o;   o += up256((size_t)cap * n * n * 4);
    L.li = o;     o += up256((size_t)cap * C * 2);
    L.total = o;
    return L;
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

bool pinned(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

size_t mhc_seam_host_workspace_bytes(int64_t T, int n, int C) {
    if (T <= 0 || n != 4 || C < 8 || C % 8 != 0) return 0;
    const int64_t cap = max_chunk(T);
    return up256(mhc_pre_workspace_bytes(cap, n, C)) + kSets * set_layout(cap, n, C).total;
}

mhc_status mhc_seam_host(const uint16_t* x_h, const uint16_t* y_h, const float* pre_in_h, const float* fn,
                         const float* bias, const float* alpha, const uint16_t* norm_weight, int64_t T, int n, int C,
                         int sinkhorn_iters, float rms_eps, float norm_eps, float sinkhorn_eps, uint16_t* x_new_h,
                         float* pre_out_h, float* post_out_h, float* comb_out_h, uint16_t* layer_input_h,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (T < 0 || n < 1 || C < 1 || sinkhorn_iters < 1) return MHC_ERR_INVALID_ARGUMENT;
    if (n != 4 || C % 8 != 0) return MHC_ERR_UNSUPPORTED;
    if (T == 0) return MHC_OK;
    const void* req[] = {x_h, y_h, pre_in_h, fn, bias, alpha, x_new_h, pre_out_h, workspace};
    for (const void* p : req)
        if (!p) return MHC_ERR_INVALID_ARGUMENT;
    // host ranges: outputs may not overlap inputs, except x_new == x exactly
    const size_t xb = (size_t)T * n * C * 2, yb = (size_t)T * C * 2, pb = (size_t)T * n * 4;
    struct R { const void* p; size_t b; };
    const R ins[] = {{x_h, xb}, {y_h, yb}, {pre_in_h, pb}};
    const R outs[] = {{x_new_h, xb}, {pre_out_h, pb}, {post_out_h, pb}, {comb_out_h, (size_t)T * n * n * 4},
                      {layer_input_h, yb}};
    for (const R& o : outs) {
        for (const R& i : ins)
            if (!(o.p == x_new_h && i.p == x_h && o.p == i.p) && overlaps(o.p, o.b, i.p, i.b))
                return MHC_ERR_INVALID_ARGUMENT;
        for (const R& o2 : outs)
            if (&o != &o2 && overlaps(o.p, o.b, o2.p, o2.b)) return MHC_ERR_INVALID_ARGUMENT;
    }
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHC_ERR_INVALID_ARGUMENT;
    const size_t need = mhc_seam_host_workspace_bytes(T, n, C);
    if (need == 0 || workspace_bytes < need) return MHC_ERR_INVALID_ARGUMENT;
    const void* host[] = {x_h, y_h, pre_in_h, x_new_h, pre_out_h, post_out_h, comb_out_h, layer_input_h};
    for (const void* p : host)
        if (p && !pinned(p)) return MHC_ERR_INVALID_ARGUMENT;   // page-locked host memory only

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);   // one enqueue at a time per process
    Pipe& p = g_pipe[dev];
    if (!make_pipe(p)) return MHC_ERR_CUDA;

    const int64_t nch = num_chunks(T), cap = max_chunk(T);
    const SetLayout L = set_layout(cap, n, C);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const size_t tc_bytes = up256(mhc_pre_workspace_bytes(cap, n, C));
    unsigned char* sets[kSets];
    for (int b = 0; b < kSets; ++b) sets[b] = ws + tc_bytes + b * L.total;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);

    mhc_status st = MHC_OK;
    auto cu = [&](cudaError_t e) {
        if (e != cudaSuccess && st == MHC_OK) st = MHC_ERR_CUDA;
        return e == cudaSuccess;
    };
    // fork: the copy streams start after what the caller's stream holds
    cu(cudaEventRecord(p.start, s));
    cu(cudaStreamWaitEvent(p.in, p.start, 0));
    cu(cudaStreamWaitEvent(p.out, p.start, 0));
    for (int64_t k = 0; k < nch && st == MHC_OK; ++k) {
        const int b = (int)(k % kSets);
        const Chunk ch = chunk_of(T, k);
        const int64_t t0 = ch.t0, nk = ch.n;
        unsigned char* S = sets[b];
        uint16_t* dx = reinterpret_cast<uint16_t*>(S + L.x);
        uint16_t* dy = reinterpret_cast<uint16_t*>(S + L.y);
        float* dpi = reinterpret_cast<float*>(S + L.pre_in);
        uint16_t* dxn = reinterpret_cast<uint16_t*>(S + L.x_new);
        float* dpre = reinterpret_cast<float*>(S + L.pre);
        float* dpost = reinterpret_cast<float*>(S + L.post);
        float* dcomb = reinterpret_cast<float*>(S + L.comb);
        uint16_t* dli = reinterpret_cast<uint16_t*>(S + L.li);
        // in: set b's inputs are free once chunk k-kSets's kernels are done
        if (k >= kSets) cu(cudaStreamWaitEvent(p.in, p.comp_done[b], 0));
        cu(cudaMemcpyAsync(dx, x_h + t0 * n * C, (size_t)nk * n * C * 2, cudaMemcpyHostToDevice, p.in));
        cu(cudaMemcpyAsync(dy, y_h + t0 * C, (size_t)nk * C * 2, cudaMemcpyHostToDevice, p.in));
        cu(cudaMemcpyAsync(dpi, pre_in_h + t0 * n, (size_t)nk * n * 4, cudaMemcpyHostToDevice, p.in));
        cu(cudaEventRecord(p.in_done[b], p.in));
        // kernels on the caller's stream: set b's outputs are free once chunk
        // k-kSets's results have left
        cu(cudaStreamWaitEvent(s, p.in_done[b], 0));
        if (k >= kSets) cu(cudaStreamWaitEvent(s, p.out_done[b], 0));
        if (st != MHC_OK) break;
        mhc_status r = mhc_pre_delayed(dx, dpi, fn, bias, alpha, norm_weight, nk, n, C, sinkhorn_iters, rms_eps,
                                       norm_eps, sinkhorn_eps, dpre, dpost, dcomb, dli, nullptr, ws, tc_bytes, s);
        if (r == MHC_OK) r = mhc_post(dx, dy, dcomb, dpost, nk, n, C, dxn, s);
        if (r != MHC_OK) {
            st = r;
            break;
        }
        cu(cudaEventRecord(p.comp_done[b], s));
        // out
        cu(cudaStreamWaitEvent(p.out, p.comp_done[b], 0));
        cu(cudaMemcpyAsync(x_new_h + t0 * n * C, dxn, (size_t)nk * n * C * 2, cudaMemcpyDeviceToHost, p.out));
        cu(cudaMemcpyAsync(pre_out_h + t0 * n, dpre, (size_t)nk * n * 4, cudaMemcpyDeviceToHost, p.out));
        if (post_out_h)
            cu(cudaMemcpyAsync(post_out_h + t0 * n, dpost, (size_t)nk * n * 4, cudaMemcpyDeviceToHost, p.out));
        if (comb_out_h)
            cu(cudaMemcpyAsync(comb_out_h + t0 * n * n, dcomb, (size_t)nk * n * n * 4, cudaMemcpyDeviceToHost,
                               p.out));
        if (layer_input_h)
            cu(cudaMemcpyAsync(layer_input_h + t0 * C, dli, (size_t)nk * C * 2, cudaMemcpyDeviceToHost, p.out));
        cu(cudaEventRecord(p.out_done[b], p.out));
    }
    // join: the caller's stream completes after every copy of the call
    cudaError_t e1 = cudaEventRecord(p.end_in, p.in);
    cudaError_t e2 = cudaEventRecord(p.end_out, p.out);
    cudaError_t e3 = cudaStreamWaitEvent(s, p.end_in, 0);
    cudaError_t e4 = cudaStreamWaitEvent(s, p.end_out, 0);
    if (st == MHC_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess))
        st = MHC_ERR_CUDA;
    return st;
}

}  // extern "C"
