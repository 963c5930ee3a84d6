// common.cuh -- device helpers shared by the seam kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mhc {

constexpr int kStreams = 4;                       // hc_mult n
constexpr int kLogits = 2 * kStreams + kStreams * kStreams;  // 24

// Two bf16 packed in a 32-bit word -> two exact fp32 values.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two fp32 to bf16 (nearest, ties to even) and pack lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// Two fp32 lanes in one 64-bit register for the packed .f32x2 instructions
// (each lane is rounded on its own, exactly like the scalar instruction).
struct f32x2 {
    unsigned long long v;
};
__device__ __forceinline__ f32x2 make_f32x2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void split_f32x2(f32x2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ f32x2 mul_rn2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f32x2 add_rn2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f32x2 fma_rn2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
// bf16 pair (low column in the low half) -> packed fp32 pair.
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) { return make_f32x2(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(f32x2 a) {
    float lo, hi;
    split_f32x2(a, lo, hi);
    return pack_bf16x2(lo, hi);
}

// Programmatic dependent launch (PTX griddepcontrol).  A kernel launched
// with the programmatic stream serialization attribute may start while the
// previous kernel in the stream is still running: griddep_wait() blocks until
// that kernel has completed and its writes are visible (without the
// attribute it returns at once); griddep_launch_dependents() allows the next
// such kernel to start before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// mHC post on 8 columns of one token: out[j][e] = sum_i cw[i][j] x[i][e]
// + pw[j] y[e] in fp32, the sum over i in order 0..3 (the first term a
// product, then fused multiply-adds), then + post * y, one rounding to bf16
// per output.  Taken one stream at a time (post_mix_first for i = 0,
// post_mix_next for i = 1..3, post_mix_last); the post kernel and the fused
// post + pre kernel both use these steps, so the two give the same bits.
// cw / pw: the coefficients of the NJ outputs taken (comb row i from the
// first of them, post of each).
// NE: elements (columns) per call: 8, or 4 / 2 where a caller splits an item.
template <int NJ, int NE = 8>
__device__ __forceinline__ void post_mix_first(float (&acc)[NJ][NE], const float (&x)[NE], const float* cw) {
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[j][e] = cw[j] * x[e];
}
template <int NJ, int NE = 8>
__device__ __forceinline__ void post_mix_next(float (&acc)[NJ][NE], const float (&x)[NE], const float* cw) {
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[j][e] = fmaf(cw[j], x[e], acc[j][e]);
}
template <int NJ>
__device__ __forceinline__ void post_mix_last(const float (&acc)[NJ][8], const float (&y)[8], const float* pw,
                                              uint4 (&out)[NJ]) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf(pw[j], y[e], acc[j][e]);
        out[j] = pack8(o);
    }
}

// post_mix_last on four columns: two packed bf16 pairs per output.
template <int NJ>
__device__ __forceinline__ void post_mix_last4(const float (&acc)[NJ][4], const float (&y)[4], const float* pw,
                                               uint2 (&out)[NJ]) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = fmaf(pw[j], y[e], acc[j][e]);
        out[j] = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
    }
}

// post_mix_last on two columns: one packed bf16 pair per output.
template <int NJ>
__device__ __forceinline__ void post_mix_last2(const float (&acc)[NJ][2], const float (&y)[2], const float* pw,
                                               uint32_t (&out)[NJ]) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) out[j] = pack_bf16x2(fmaf(pw[j], y[0], acc[j][0]), fmaf(pw[j], y[1], acc[j][1]));
}

// Streaming 16-byte global load / store (data touched once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }

// Hardware reciprocal (PTX rcp.approx.ftz: about 1 ulp, one instruction).
// The sums it inverts here are at least 4 * eps > 0, far from the
// subnormal range, so flushing subnormals changes nothing.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Sinkhorn on a 4x4 row-major matrix A that already holds iteration 1's row
// softmax plus eps: iteration 1 finishes with a column normalisation,
// iterations 2..iters normalise rows then columns.  One thread.  The matrix
// is carried as P_ij = A_ij R_i C_j: a row normalisation sets
// R_i = 1 / sum_j A_ij C_j, a column one C_j = 1 / sum_i A_ij R_i, and P is
// formed once at the end -- the same normalisations in exact arithmetic,
// with a shorter dependent chain per step than rescaling all 16 entries.
// The 2*iters steps are one dependent chain; two iterations per loop body
// keep the loop overhead low and the body small enough for the instruction
// cache (the kernels run the chain once per token: a fully unrolled chain
// is fetched cold every call and was slower in them).
__device__ __forceinline__ void sinkhorn_iterations(float (&P)[16], int iters) {
    float R[4] = {1.f, 1.f, 1.f, 1.f}, Cs[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) Cs[j] = rcp_approx(((P[j] + P[4 + j]) + P[8 + j]) + P[12 + j]);
    auto iteration = [&]() {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            R[i] = rcp_approx(
                fmaf(P[4 * i + 3], Cs[3], fmaf(P[4 * i + 2], Cs[2], fmaf(P[4 * i + 1], Cs[1], P[4 * i] * Cs[0]))));
#pragma unroll
        for (int j = 0; j < 4; ++j)
            Cs[j] = rcp_approx(fmaf(P[12 + j], R[3], fmaf(P[8 + j], R[2], fmaf(P[4 + j], R[1], P[j] * R[0]))));
    };
    int it = 1;
    for (; it + 1 < iters; it += 2) {
        iteration();
        iteration();
    }
    if (it < iters) iteration();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) P[4 * i + j] = (P[4 * i + j] * R[i]) * Cs[j];
}

// Iteration 1's row step of the comb's Sinkhorn, by one thread: the row
// softmax (max subtracted per row) of the 4x4 row-major comb logits l16,
// plus eps on every entry.  The exponentials take the hardware exp2 path
// (__expf): its arguments are <= 0, its relative error on every entry that
// survives next to eps is about 1e-6, and the four of a row are the head of
// the Sinkhorn chain on the decode path.
__device__ __forceinline__ void comb_softmax_eps(const float* l16, float eps, float (&P)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* l = l16 + 4 * i;
        float mx = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
        float e0 = __expf(l[0] - mx), e1 = __expf(l[1] - mx);
        float e2 = __expf(l[2] - mx), e3 = __expf(l[3] - mx);
        float inv = rcp_approx(((e0 + e1) + e2) + e3);
        P[4 * i + 0] = e0 * inv + eps;
        P[4 * i + 1] = e1 * inv + eps;
        P[4 * i + 2] = e2 * inv + eps;
        P[4 * i + 3] = e3 * inv + eps;
    }
}

// Per-token gates and comb from the 2n+n^2 logits, in fp32, by one thread.
// pre = sigmoid(l[0:4]), post = 2 sigmoid(l[4:8]); comb = Sinkhorn on the
// 4x4 row-major comb logits l[8:24]: iteration 1 is the row softmax (max
// subtracted per row) plus eps on every entry, then a column normalisation;
// iterations 2..iters normalise rows then columns.  Normalisations multiply
// by the hardware reciprocal of the sum: a relative error of a few fp32 ulps
// per step, far inside the 2e-5 gate tolerance.
__device__ __forceinline__ void gates_and_comb(const float (&l)[kLogits], int iters, float eps,
                                               float (&pre)[4], float (&post)[4],
                                               float (&P)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pre[i] = __fdividef(1.0f, 1.0f + expf(-l[i]));
        post[i] = __fdividef(2.0f, 1.0f + expf(-l[4 + i]));
    }
    comb_softmax_eps(l + 8, eps, P);
    sinkhorn_iterations(P, iters);
}

}  // namespace mhc
