// pre_cluster.cu -- delayed mHC pre block on CUDA cores, one cluster of 16
// CTAs per token tile (sm_103a).
//
// What it computes (vLLM page "Use AITER mHC for the delayed pre block":
// commit message, sections "Why V4.1 cannot just reuse MHCPreOp", "Approach"
// and "Result"; page "Fix TileLang mHC pre on 64-wide wavefronts",
// "Measurements" for the fold), per token t with K = 4C:
//   r = 1/sqrt(sum x_flat^2 / K + eps); l = r (x_flat . fn^T) alpha_seg + bias;
//   pre = sigmoid(l[0:4]); post = 2 sigmoid(l[4:8]); comb = Sinkhorn(l[8:24]);
//   h = fp32 collapse of x with the INCOMING pre-mix; layer_input = bf16(h)
//   or bf16(h * rsqrt(mean h^2 + eps) * w).
//
// Decomposition.  A cluster of 16 CTAs owns a tile of 8 tokens; CTA r owns a
// slice of C/16 columns of all four streams (so it can collapse them) and
// keeps the matching K-slice of fn in registers for the whole launch:
// warp w holds logits 2w and 2w+1, lane l holds 8-column groups
// q = l, l+32, ... of the slice.  Per tile:
//   1. the tile's x slice (and pre_in) arrives by cp.async, double-buffered
//      one tile ahead;
//   2. each warp forms its two partial dot products for the 8 tokens and
//      reduces them across lanes (a reduce-scatter butterfly, fixed order);
//      each thread collapses one (token, 8-column) item, keeping h in
//      registers, and forms its sum x^2 and sum h^2;
//   3. cluster barrier; CTA r < 8 sums the 16 CTAs' partials of token r over
//      distributed shared memory in rank order, computes r, the logits, the
//      gates and the Sinkhorn comb in one thread, writes them, and writes the
//      token's fold scale into every CTA of the cluster;
//   4. cluster barrier; every CTA writes its layer_input slice.
// No global scratch memory, no atomics, no spin waits: the only waits are
// hardware cluster barriers, and every reduction has a fixed order, so the
// results are deterministic.
#include "common.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace mhc {

constexpr int kClusterCtas = 16;   // CTAs per cluster = column slices of C
constexpr int kPreThreads = 384;   // 12 warps x 2 logits = 24 logits
constexpr int kTileTokens = 8;     // tokens per cluster tile
constexpr int kPartStride = 26;    // 24 dot products, sum x^2, sum h^2

struct PreArgs {
    const uint16_t* x;
    const float* pre_in;
    const float* fn;
    const float* bias;
    const float* alpha;
    const uint16_t* norm_w;
    int64_t T;
    int C;
    int iters;
    float rms_eps, norm_eps, sk_eps;
    float* pre_out;
    float* post_out;
    float* comb_out;
    uint16_t* layer_input;
    float* logits_out;
    int64_t ntiles;
    int lcmax;  // max 8-column groups per CTA slice
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    int n = valid ? 16 : 0;  // 0 bytes read: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Reduce 16 per-lane values over the 32 lanes of a warp.  After the call
// lane l holds in v[0] the full sum of value index (l >> 1) & 15.
__device__ __forceinline__ void warp_reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int half = 8 >> s, bit = 16 >> s;
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            float send = upper ? v[i] : v[i + half];
            float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
}

template <int JMAX>
__global__ void __launch_bounds__(kPreThreads, 1) pre_cluster_kernel(const PreArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int64_t cluster_id = blockIdx.x / kClusterCtas;
    const int64_t nclusters = gridDim.x / kClusterCtas;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = a.C, K = 4 * C, nch = C >> 3;
    const int ch0 = rank * nch / kClusterCtas;
    const int lc = (rank + 1) * nch / kClusterCtas - ch0;  // 8-column groups of this CTA
    const int qn = 4 * lc;                                  // (stream, group) pairs
    const bool fold = a.norm_w != nullptr;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int qstride = 4 * a.lcmax;
    uint4* xs = reinterpret_cast<uint4*>(smem_raw);                       // [2][TT][qstride]
    float* pin = reinterpret_cast<float*>(xs + 2 * kTileTokens * qstride);  // [2][TT][4]
    float* part = pin + 2 * kTileTokens * 4;                                // [TT][26]
    float* scale = part + kTileTokens * kPartStride;                        // [TT]
    float* red = scale + kTileTokens;                                       // [2][TT][lcmax]

    // ---- this warp's two rows of fn over this CTA's K-slice, in registers
    const int m0 = 2 * warp;
    float w[JMAX][2][8];
#pragma unroll
    for (int j = 0; j < JMAX; ++j) {
        const int q = lane + 32 * j;
        if (q < qn) {
            const int i = q / lc, cc = q - i * lc;
            const int64_t k = (int64_t)i * C + (int64_t)(ch0 + cc) * 8;
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                const float4* src = reinterpret_cast<const float4*>(a.fn + (int64_t)(m0 + mm) * K + k);
                float4 u = __ldg(src), v = __ldg(src + 1);
                w[j][mm][0] = u.x; w[j][mm][1] = u.y; w[j][mm][2] = u.z; w[j][mm][3] = u.w;
                w[j][mm][4] = v.x; w[j][mm][5] = v.y; w[j][mm][6] = v.z; w[j][mm][7] = v.w;
            }
        } else {
#pragma unroll
            for (int mm = 0; mm < 2; ++mm)
#pragma unroll
                for (int e = 0; e < 8; ++e) w[j][mm][e] = 0.f;
        }
    }

    auto issue_tile = [&](int64_t tile, int buf) {
        const int64_t t0 = tile * kTileTokens;
        for (int idx = threadIdx.x; idx < kTileTokens * qn; idx += kPreThreads) {
            const int tt = idx / qn, q = idx - tt * qn;
            const int i = q / lc, cc = q - i * lc;
            const int64_t t = t0 + tt;
            const bool ok = t < a.T;
            const uint16_t* src = a.x + ((ok ? t : 0) * 4 + i) * (int64_t)C + (int64_t)(ch0 + cc) * 8;
            cp_async16(xs + (buf * kTileTokens + tt) * qstride + q, src, ok);
        }
        if (threadIdx.x < kTileTokens) {
            const int64_t t = t0 + threadIdx.x;
            const bool ok = t < a.T;
            cp_async16(pin + (buf * kTileTokens + threadIdx.x) * 4, a.pre_in + (ok ? t : 0) * 4, ok);
        }
    };

    int64_t tile = cluster_id;
    int buf = 0;
    issue_tile(tile, 0);
    cp_async_commit();

    for (; tile < a.ntiles; tile += nclusters, buf ^= 1) {
        const int64_t t0 = tile * kTileTokens;
        const int64_t next = tile + nclusters;
        if (next < a.ntiles) issue_tile(next, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();  // this tile's group has landed (the next may be in flight)
        __syncthreads();

        const uint4* xb = xs + buf * kTileTokens * qstride;

        // ---- 2a. partial dot products of logits m0, m0+1 for the 8 tokens
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int tt = 0; tt < kTileTokens; ++tt) {
#pragma unroll
            for (int j = 0; j < JMAX; ++j) {
                const int q = lane + 32 * j;
                if (q < qn) {
                    float f[8];
                    unpack8(xb[tt * qstride + q], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acc[2 * tt + 0] = fmaf(w[j][0][e], f[e], acc[2 * tt + 0]);
                        acc[2 * tt + 1] = fmaf(w[j][1][e], f[e], acc[2 * tt + 1]);
                    }
                }
            }
        }
        warp_reduce_scatter16(acc, lane);
        if ((lane & 1) == 0) {
            const int idx = (lane >> 1) & 15;
            part[(idx >> 1) * kPartStride + m0 + (idx & 1)] = acc[0];
        }

        // ---- 2b. collapse one (token, 8-column) item per thread
        float h[8];
        const int item = threadIdx.x;
        const bool has_item = item < kTileTokens * lc;
        const int it_tt = has_item ? item / lc : 0;
        const int it_cc = has_item ? item - it_tt * lc : 0;
        if (has_item) {
            const float* p = pin + (buf * kTileTokens + it_tt) * 4;
            float xv[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) unpack8(xb[it_tt * qstride + i * lc + it_cc], xv[i]);
            float sx = 0.f, sh = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float v = __fmul_rn(p[0], xv[0][e]);
                v = __fadd_rn(v, __fmul_rn(p[1], xv[1][e]));
                v = __fadd_rn(v, __fmul_rn(p[2], xv[2][e]));
                v = __fadd_rn(v, __fmul_rn(p[3], xv[3][e]));
                h[e] = v;
                sh = fmaf(v, v, sh);
#pragma unroll
                for (int i = 0; i < 4; ++i) sx = fmaf(xv[i][e], xv[i][e], sx);
            }
            red[it_tt * a.lcmax + it_cc] = sx;
            red[(kTileTokens + it_tt) * a.lcmax + it_cc] = sh;
            const int64_t t = t0 + it_tt;
            if (!fold && t < a.T) {
                uint4* dst = reinterpret_cast<uint4*>(a.layer_input + t * C + (int64_t)(ch0 + it_cc) * 8);
                st_stream(dst, pack8(h));
            }
        }
        __syncthreads();

        // ---- 2c. this CTA's sum x^2 and sum h^2 per token (warp tt, fixed order)
        if (warp < kTileTokens) {
            float sx = 0.f, sh = 0.f;
            for (int cc = lane; cc < lc; cc += 32) {
                sx += red[warp * a.lcmax + cc];
                sh += red[(kTileTokens + warp) * a.lcmax + cc];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sx += __shfl_xor_sync(0xffffffffu, sx, o);
                sh += __shfl_xor_sync(0xffffffffu, sh, o);
            }
            if (lane == 0) {
                part[warp * kPartStride + 24] = sx;
                part[warp * kPartStride + 25] = sh;
            }
        }
        cluster.sync();  // A: every CTA's partials are visible cluster-wide

        // ---- 3. finalize token t0 + rank in CTA rank (rank < 8), warp 0: the fold
        //         scale is pushed first (it gates every CTA's stores), the gates and
        //         the Sinkhorn comb follow while the other CTAs wait at barrier B
        if (rank < kTileTokens && warp == 0) {
            const int64_t t = t0 + rank;
            float v = 0.f;
            if (lane < kPartStride) {
                float pv[kClusterCtas];
#pragma unroll
                for (int s = 0; s < kClusterCtas; ++s)
                    pv[s] = cluster.map_shared_rank(part, s)[rank * kPartStride + lane];
#pragma unroll
                for (int s = 0; s < kClusterCtas; ++s) v += pv[s];
            }
            const float sh = __shfl_sync(0xffffffffu, v, 25);
            if (fold && lane < kClusterCtas) {
                float* rs = cluster.map_shared_rank(scale, lane);
                rs[rank] = 1.0f / sqrtf(sh / (float)C + a.norm_eps);
            }
            float l[kLogits];
#pragma unroll
            for (int m = 0; m < kLogits; ++m) l[m] = __shfl_sync(0xffffffffu, v, m);
            const float sx = __shfl_sync(0xffffffffu, v, 24);
            if (lane == 0 && t < a.T) {
                const float r = 1.0f / sqrtf(sx / (float)K + a.rms_eps);
                const float al0 = __ldg(a.alpha), al1 = __ldg(a.alpha + 1), al2 = __ldg(a.alpha + 2);
#pragma unroll
                for (int m = 0; m < kLogits; ++m) {
                    const float al = m < 4 ? al0 : (m < 8 ? al1 : al2);
                    l[m] = (r * l[m]) * al + __ldg(a.bias + m);
                }
                if (a.logits_out) {
                    float4* lo = reinterpret_cast<float4*>(a.logits_out + t * kLogits);
#pragma unroll
                    for (int m = 0; m < kLogits; m += 4) lo[m / 4] = make_float4(l[m], l[m + 1], l[m + 2], l[m + 3]);
                }
                float pre[4], post[4], P[16];
                gates_and_comb(l, a.iters, a.sk_eps, pre, post, P);
                reinterpret_cast<float4*>(a.pre_out)[t] = make_float4(pre[0], pre[1], pre[2], pre[3]);
                reinterpret_cast<float4*>(a.post_out)[t] = make_float4(post[0], post[1], post[2], post[3]);
                float4* co = reinterpret_cast<float4*>(a.comb_out + t * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) co[i] = make_float4(P[4 * i], P[4 * i + 1], P[4 * i + 2], P[4 * i + 3]);
            }
        }
        cluster.sync();  // B: fold scales are in place; partial buffers may be reused

        // ---- 4. fold: scale h, round once, store this CTA's slice
        if (fold && has_item) {
            const int64_t t = t0 + it_tt;
            if (t < a.T) {
                const float s = scale[it_tt];
                const uint4 wv = __ldg(reinterpret_cast<const uint4*>(a.norm_w + (int64_t)(ch0 + it_cc) * 8));
                float wf[8], o[8];
                unpack8(wv, wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(h[e], s), wf[e]);
                uint4* dst = reinterpret_cast<uint4*>(a.layer_input + t * C + (int64_t)(ch0 + it_cc) * 8);
                st_stream(dst, pack8(o));
            }
        }
    }
    cp_async_wait<0>();
}

static size_t pre_cluster_smem(int lcmax) {
    return sizeof(uint4) * 2 * kTileTokens * 4 * lcmax + sizeof(float) * 2 * kTileTokens * 4 +
           sizeof(float) * kTileTokens * kPartStride + sizeof(float) * kTileTokens +
           sizeof(float) * 2 * kTileTokens * lcmax;
}

static cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kPreThreads, 1, 1);
    cfg.gridDim = dim3(kClusterCtas, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cfg;
}

static int lcmax_of(int C) { return (C / 8 + kClusterCtas - 1) / kClusterCtas; }

int pre_cluster_jmax(int C) {
    const int j = (4 * lcmax_of(C) + 31) / 32;
    if (j <= 2) return 2;
    if (j <= 4) return 4;
    if (j <= 5) return 5;
    if (j <= 6) return 6;
    return 0;
}

int pre_cluster_tile_tokens() { return kTileTokens; }
int pre_cluster_ctas() { return kClusterCtas; }

// One-time set-up for the current device and hidden size C: allows the
// non-portable cluster size and the dynamic shared memory of the kernel
// instance C uses, then returns the maximum number of co-resident clusters
// (the launch grid is min(tiles, that) clusters).  Returns 0 on error.
// Must run before any stream capture that records the kernel.
int pre_cluster_prepare(int C) {
    const size_t smem = pre_cluster_smem(lcmax_of(C));
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(attr, smem, nullptr);
    int n = 0;
    cudaError_t e = cudaSuccess;
    auto setup = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    };
    switch (pre_cluster_jmax(C)) {
        case 2: setup(pre_cluster_kernel<2>); break;
        case 4: setup(pre_cluster_kernel<4>); break;
        case 5: setup(pre_cluster_kernel<5>); break;
        case 6: setup(pre_cluster_kernel<6>); break;
        default: return 0;
    }
    return e == cudaSuccess ? n : 0;
}

cudaError_t launch_pre_cluster(const uint16_t* x, const float* pre_in, const float* fn,
                               const float* bias, const float* alpha, const uint16_t* norm_w,
                               int64_t T, int C, int iters, float rms_eps, float norm_eps,
                               float sk_eps, float* pre_out, float* post_out, float* comb_out,
                               uint16_t* layer_input, float* logits_out, cudaStream_t stream,
                               int max_clusters) {
    PreArgs a;
    a.x = x; a.pre_in = pre_in; a.fn = fn; a.bias = bias; a.alpha = alpha; a.norm_w = norm_w;
    a.T = T; a.C = C; a.iters = iters;
    a.rms_eps = rms_eps; a.norm_eps = norm_eps; a.sk_eps = sk_eps;
    a.pre_out = pre_out; a.post_out = post_out; a.comb_out = comb_out;
    a.layer_input = layer_input; a.logits_out = logits_out;
    a.ntiles = (T + kTileTokens - 1) / kTileTokens;
    a.lcmax = lcmax_of(C);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(attr, pre_cluster_smem(a.lcmax), stream);
    const int64_t nclusters = a.ntiles < max_clusters ? a.ntiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(nclusters * kClusterCtas), 1, 1);
    switch (pre_cluster_jmax(C)) {
        case 2: return cudaLaunchKernelEx(&cfg, pre_cluster_kernel<2>, a);
        case 4: return cudaLaunchKernelEx(&cfg, pre_cluster_kernel<4>, a);
        case 5: return cudaLaunchKernelEx(&cfg, pre_cluster_kernel<5>, a);
        case 6: return cudaLaunchKernelEx(&cfg, pre_cluster_kernel<6>, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
