// collapse.cu -- collapse and optional RMSNorm fold as a pure HBM stream,
// for the second pass of the non-delayed pre block from 256 tokens (its
// first pass, the tensor-core kernel's gates-only instance, has written each
// token's pre-mix).  The non-delayed block collapses with the token's own
// pre-mix (vLLM page "Use AITER mHC for the delayed pre block", "Why V4.1
// cannot just reuse MHCPreOp"); the fold is rounded once (page "Fix TileLang
// mHC pre on 64-wide wavefronts", "Measurements").
//
// The results must be the bits the tensor-core kernel would produce for the
// same pre-mix (the non-delayed call equals the delayed one fed its own
// pre), so this kernel repeats that kernel's arithmetic in the same order:
//  * h = ((p0 x0 + p1 x1) + p2 x2) + p3 x3, every product and sum rounded;
//  * sum h^2: the tensor-core kernel splits the C columns into 16 slices (one
//    per CTA of a cluster) of C/256 stages of 16 columns; a stage belongs to
//    token-row group (it * stages + stage) & 1, `it` being the tile's round
//    in its cluster (tile / clusters); each group accumulates its stages in
//    order with a packed fma (even and odd columns in the two lanes), adds
//    the two lanes, and the finaliser sums the 32 partials in (slice, group)
//    order.  Here lane q = 2 * slice + group of a warp forms partial q the
//    same way, and every lane sums the 32 partials in lane order;
//  * the fold (h * s) * w with s = 1 / sqrt(sum / C + eps), rounded to bf16.
// One warp per token: the collapse with the sum of squares, h parked in the
// warp's row of shared memory, then the fold from there.  Reads x and the
// pre-mix once, writes layer_input: 50 KB per token at C = 5120.
#include "common.cuh"

namespace mhc {

namespace {

constexpr int kThreads = 128;                  // 4 warps: 4 tokens per CTA at a time, 2 CTAs per SM
constexpr int kWarps = kThreads / 32;
constexpr int kPad = 4;                        // floats between slices of a parked row (bank spread)

// the collapse of one 16-column stage of slice r: h as 8 column pairs
__device__ __forceinline__ void collapse16(const uint16_t* __restrict__ xs, int64_t xsc, const float (&p)[4],
                                           f32x2 (&h)[8]) {
    uint4 w[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4* src = reinterpret_cast<const uint4*>(xs + i * xsc);
        w[i][0] = __ldg(src);
        w[i][1] = __ldg(src + 1);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float xl[4], xh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4& u = w[i][e >> 2];
            const uint32_t word = (e & 3) == 0 ? u.x : (e & 3) == 1 ? u.y : (e & 3) == 2 ? u.z : u.w;
            xl[i] = bf16lo(word);
            xh[i] = bf16hi(word);
        }
        float vl = __fmul_rn(p[0], xl[0]), vh = __fmul_rn(p[0], xh[0]);
        vl = __fadd_rn(vl, __fmul_rn(p[1], xl[1]));
        vh = __fadd_rn(vh, __fmul_rn(p[1], xh[1]));
        vl = __fadd_rn(vl, __fmul_rn(p[2], xl[2]));
        vh = __fadd_rn(vh, __fmul_rn(p[2], xh[2]));
        vl = __fadd_rn(vl, __fmul_rn(p[3], xl[3]));
        vh = __fadd_rn(vh, __fmul_rn(p[3], xh[3]));
        h[e] = make_f32x2(vl, vh);
    }
}

// One warp per token.  FOLD: pass 1 collapses the lane's stages, parks h in
// the warp's shared-memory row and accumulates the lane's sum of squares;
// pass 2 reads h back, folds and stores.  Without the fold one pass stores
// bf16(h) directly.
template <bool FOLD>
__global__ void __launch_bounds__(kThreads)
collapse_fold_kernel(const uint16_t* __restrict__ x, const float* __restrict__ pre,
                     const uint16_t* __restrict__ norm_w, int64_t T, int C, int64_t xtok, int64_t xsc,
                     int clusters, float norm_eps, uint16_t* __restrict__ out) {
    extern __shared__ __align__(16) float park[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = C / 16, stages = slice / 16, row = 16 * (slice + kPad);
    const int r = lane >> 1, par = lane & 1;
    float* hrow = park + (size_t)warp * row + (size_t)r * (slice + kPad);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < T; t += nwarps) {
        const float4 pv = __ldg(reinterpret_cast<const float4*>(pre) + t);
        const float p[4] = {pv.x, pv.y, pv.z, pv.w};
        const int64_t it = (t / 128) / clusters;
        const int first = (int)(((it * stages) & 1) != par);   // this lane's first stage of the slice
        const uint16_t* xt = x + t * xtok + (int64_t)r * slice;
        uint16_t* ot = out + t * C + (int64_t)r * slice;
        if (!FOLD) {
            for (int stg = first; stg < stages; stg += 2) {
                f32x2 h[8];
                collapse16(xt + 16 * stg, xsc, p, h);
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = f32x2_to_bf16x2(h[e]);
                uint4* dst = reinterpret_cast<uint4*>(ot + 16 * stg);
                st_stream(dst, make_uint4(o[0], o[1], o[2], o[3]));
                st_stream(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
            }
            continue;
        }
        f32x2 sh2 = make_f32x2(0.f, 0.f);
        int stg = first;
        // two stages per iteration: twice the loads in flight
        for (; stg + 2 < stages; stg += 4) {
            f32x2 h0[8], h1[8];
            collapse16(xt + 16 * stg, xsc, p, h0);
            collapse16(xt + 16 * (stg + 2), xsc, p, h1);
#pragma unroll
            for (int e = 0; e < 8; ++e) sh2 = fma_rn2(h0[e], h0[e], sh2);
#pragma unroll
            for (int e = 0; e < 8; ++e) sh2 = fma_rn2(h1[e], h1[e], sh2);
            float4* d0 = reinterpret_cast<float4*>(hrow + 16 * stg);
            float4* d1 = reinterpret_cast<float4*>(hrow + 16 * (stg + 2));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float a, b, cc, d;
                split_f32x2(h0[2 * c], a, b);
                split_f32x2(h0[2 * c + 1], cc, d);
                d0[c] = make_float4(a, b, cc, d);
                split_f32x2(h1[2 * c], a, b);
                split_f32x2(h1[2 * c + 1], cc, d);
                d1[c] = make_float4(a, b, cc, d);
            }
        }
        for (; stg < stages; stg += 2) {
            f32x2 h0[8];
            collapse16(xt + 16 * stg, xsc, p, h0);
#pragma unroll
            for (int e = 0; e < 8; ++e) sh2 = fma_rn2(h0[e], h0[e], sh2);
            float4* d0 = reinterpret_cast<float4*>(hrow + 16 * stg);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float a, b, cc, d;
                split_f32x2(h0[2 * c], a, b);
                split_f32x2(h0[2 * c + 1], cc, d);
                d0[c] = make_float4(a, b, cc, d);
            }
        }
        float a0, a1;
        split_f32x2(sh2, a0, a1);
        const float partial = a0 + a1;
        float total = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) total += __shfl_sync(0xffffffffu, partial, q);
        const float s = 1.0f / sqrtf(total / (float)C + norm_eps);
        const f32x2 s2 = make_f32x2(s, s);
        for (int sg = first; sg < stages; sg += 2) {
            const float4* src = reinterpret_cast<const float4*>(hrow + 16 * sg);
            const uint4* wv = reinterpret_cast<const uint4*>(norm_w + (int64_t)r * slice + 16 * sg);
            const uint4 w0 = __ldg(wv), w1 = __ldg(wv + 1);
            const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t o[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 v = src[c];
                o[2 * c] = f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v.x, v.y), s2), bf16x2_to_f32x2(ww[2 * c])));
                o[2 * c + 1] =
                    f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v.z, v.w), s2), bf16x2_to_f32x2(ww[2 * c + 1])));
            }
            uint4* dst = reinterpret_cast<uint4*>(ot + 16 * sg);
            st_stream(dst, make_uint4(o[0], o[1], o[2], o[3]));
            st_stream(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
        }
        __syncwarp();   // the row is reused by the warp's next token
    }
}

}  // namespace

// x: [T][4][C] (xtok = 4C, xsc = C) or the broadcast [T][C] (xtok = C,
// xsc = 0); C a multiple of 256; clusters: the number of clusters the
// tensor-core kernel ran with for this T (its tile -> round mapping).
cudaError_t launch_collapse_fold(const uint16_t* x, const float* pre, const uint16_t* norm_w, int64_t T, int C,
                                 bool broadcast, int clusters, float norm_eps, uint16_t* out, cudaStream_t stream,
                                 int num_sms) {
    if (T <= 0) return cudaSuccess;
    const int64_t xtok = broadcast ? C : 4 * (int64_t)C, xsc = broadcast ? 0 : C;
    int64_t blocks = (T + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms * 2;       // two CTAs per SM (shared memory)
    if (blocks > cap) blocks = cap;
    if (norm_w) {
        const size_t smem = (size_t)kWarps * 16 * (C / 16 + kPad) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(collapse_fold_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        collapse_fold_kernel<true><<<(unsigned)blocks, kThreads, smem, stream>>>(x, pre, norm_w, T, C, xtok, xsc,
                                                                                clusters, norm_eps, out);
    } else {
        collapse_fold_kernel<false><<<(unsigned)blocks, kThreads, 0, stream>>>(x, pre, norm_w, T, C, xtok, xsc,
                                                                              clusters, norm_eps, out);
    }
    return cudaGetLastError();
}

}  // namespace mhc
