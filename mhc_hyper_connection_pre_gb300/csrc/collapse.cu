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
//    per CTA of a cluster) of ceil(C/512) stages of 32 columns (the last one
//    16 when C/16 is an odd multiple of 16); a stage belongs to token-row
//    group (it * stages + stage) & 1, `it` being the tile's round in its
//    cluster (tile / clusters); each group accumulates its stages' columns
//    in order with a packed fma (even and odd columns in the two lanes), adds
//    the two lanes, and the finaliser sums the 32 partials in (slice, group)
//    order.  Here lane q = 2 * slice + group of a warp forms partial q the
//    same way, and every lane sums the 32 partials in lane order;
//  * the fold (h * s) * w with s = 1 / sqrt(sum / C + eps), rounded to bf16.
// Both kernels stream a CTA's tokens through a ring of shared-memory slots,
// one token's rows and its pre-mix per slot, filled by bulk copies that one
// producer thread keeps up to `slots` tokens ahead (the register-staged
// designs measured before kept too few bytes in flight).  Without the fold,
// eight warps per CTA collapse with coalesced lanes and store, two CTAs per
// SM.  With it, one CTA per SM pipelines the token: consumer warps collapse
// and park h in shared memory, a sum warp forms the sum of squares in the
// tensor-core kernel's order from the park, and the consumers fold the
// token before the previous one meanwhile.  Reads x and the pre-mix once,
// writes layer_input: 50 KB per token at C = 5120.
#include <algorithm>

#include "common.cuh"
#include "sm100.cuh"

// This translation unit has its own device status word (sm100.cuh), read
// and cleared by read_collapse_status().

namespace mhc {

namespace {

constexpr int kMaxSlots = 8;
constexpr int kConsumerBar = 1;                // named barrier of the fold kernel's consumer warps

// The producer thread: the CTA's k-th token (t = b + k G) into slot k % slots
// once every consumer warp has released the slot's previous token; then a
// bounded look at the last copy into each slot, which may still be in
// flight after an abort, before the thread exits.
template <bool BCAST>
__device__ __forceinline__ void produce(const uint16_t* x, const float* pre, int C, int b, int G, int K,
                                        int slots, uint32_t slot_bytes, unsigned char* ring, float4* pres,
                                        uint64_t* full, uint64_t* empty, volatile int* abort) {
    const uint64_t pol = policy_evict_first();
    int k = 0, s = 0;
    uint32_t n = 0;                               // the slot's round
    for (; k < K; ++k) {
        // consumers that timed out release slots without waiting for their
        // copies: nothing is issued once the flag is up (read after the
        // empty wait, which acquires the release that followed raising it),
        // so never two copies are in flight into one slot
        if (n > 0 && (!mbar_wait(&empty[s], (n - 1) & 1u, abort) || *abort)) break;
        const int64_t t = b + (int64_t)k * G;
        mbar_arrive_expect_tx(&full[s], slot_bytes + 16u);
        bulk_load_hint(ring + (size_t)s * slot_bytes, x + t * (BCAST ? (int64_t)C : 4 * (int64_t)C), slot_bytes,
                       &full[s], pol);
        bulk_load_hint(&pres[s], pre + 4 * t, 16u, &full[s], pol);
        if (++s == slots) s = 0, ++n;
    }
    // loads max(k - slots, 0) .. k - 1; load k - slots went to slot s in round n - 1
    int js = k < slots ? 0 : s;
    uint32_t jn = k < slots ? 0u : n - 1;
    for (int c = 0; c < (k < slots ? k : slots); ++c) {
        mbar_wait_drain(&full[js], jn & 1u);   // not cut short by a timeout
        if (++js == slots) js = 0, ++jn;
    }
}

// h for the 8 columns of chunk k of a staged token (rows 2C bytes apart;
// broadcast: one row read as all four streams), every product and sum rounded.
template <bool BCAST>
__device__ __forceinline__ void collapse8(const unsigned char* xs, uint32_t row_bytes, int k, const float (&p)[4],
                                          float (&h)[8]) {
    uint4 w[4];
    w[0] = reinterpret_cast<const uint4*>(xs)[k];
#pragma unroll
    for (int i = 1; i < 4; ++i) w[i] = BCAST ? w[0] : reinterpret_cast<const uint4*>(xs + i * row_bytes)[k];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float xl[4], xh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t word = e == 0 ? w[i].x : e == 1 ? w[i].y : e == 2 ? w[i].z : w[i].w;
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
        h[2 * e] = vl;
        h[2 * e + 1] = vh;
    }
}

// ---- without the fold: two CTAs per SM, eight warps collapse and store ----
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32 + 32;     // + the producer warp

// Shared memory: the slots' rows, the slots' pre-mix, full[] and empty[], the abort flag.
__host__ __device__ inline uint32_t ring_pre_off(int C, bool broadcast, int slots) {
    return (uint32_t)slots * (uint32_t)((broadcast ? 1 : 4) * 2 * C);
}
__host__ __device__ inline uint32_t ring_bytes(int C, bool broadcast, int slots) {
    return ring_pre_off(C, broadcast, slots) + 32u * (uint32_t)slots + 16u;
}

template <bool BCAST>
__global__ void __launch_bounds__(kThreads, 2)
collapse_kernel(const uint16_t* __restrict__ x, const float* __restrict__ pre, int T, int C, int slots,
                uint16_t* __restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t slot_bytes = (uint32_t)((BCAST ? 1 : 4) * 2 * C), row_bytes = 2u * (uint32_t)C;
    float4* pres = reinterpret_cast<float4*>(smem + ring_pre_off(C, BCAST, slots));
    uint64_t* full = reinterpret_cast<uint64_t*>(pres + slots);
    uint64_t* empty = full + slots;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + slots);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, chunks = C / 8;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int K = b < T ? (T - 1 - b) / G + 1 : 0;         // this CTA's tokens: b, b + G, ...

    if (tid == 0) {
        for (int s = 0; s < slots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        *abort = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();

    if (warp == kWarps) {
        if (lane == 0) produce<BCAST>(x, pre, C, b, G, K, slots, slot_bytes, smem, pres, full, empty, abort);
        return;
    }
    // each warp on its own: no barrier but the slots' mbarriers
    int s = 0;
    uint32_t ph = 0;                             // slot s's phase parity
    for (int k = 0; k < K; ++k) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort))) break;
        const float4 pv = pres[s];
        const float p[4] = {pv.x, pv.y, pv.z, pv.w};
        const unsigned char* xs = smem + (size_t)s * slot_bytes;
        uint16_t* ot = out + (b + (int64_t)k * G) * C;
        for (int c8 = tid; c8 < chunks; c8 += kWarps * 32) {
            float h[8];
            collapse8<BCAST>(xs, row_bytes, c8, p, h);
            st_stream(reinterpret_cast<uint4*>(ot) + c8,
                      make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                                 pack_bf16x2(h[6], h[7])));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);   // this warp is done with the slot
        if (++s == slots) s = 0, ph ^= 1u;
    }
}

template <bool BCAST>
cudaError_t launch_nofold(const uint16_t* x, const float* pre, int64_t T, int C, uint16_t* out,
                          cudaStream_t stream, int num_sms) {
    int dev = 0, per_sm = 0, per_block = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    // two CTAs per SM when each gets at least two slots, else one CTA with more
    int ctas_per_sm = 0, slots = 0;
    for (int cps = 2; cps >= 1 && !ctas_per_sm; --cps) {
        const int64_t budget = std::min<int64_t>(per_block, per_sm / cps - 1024);
        int sl = kMaxSlots;
        while (sl >= 2 && (int64_t)ring_bytes(C, BCAST, sl) > budget) --sl;
        if (sl >= 2) ctas_per_sm = cps, slots = sl;
    }
    if (!ctas_per_sm) return cudaErrorInvalidValue;
    const uint32_t smem = ring_bytes(C, BCAST, slots);
    e = cudaFuncSetAttribute(collapse_kernel<BCAST>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(T, (int64_t)num_sms * ctas_per_sm);
    collapse_kernel<BCAST><<<(unsigned)grid, kThreads, smem, stream>>>(x, pre, T, C, slots, out);
    return cudaGetLastError();
}

// ---- with the fold: one CTA per SM, the sum of squares pipelined ---------
// 20 consumer warps collapse token k into park k % 3 while the sum warp of
// park (k - 1) % 3 forms token k - 1's fold scale, and fold token k - 2
// meanwhile: each sum warp (one per park) has a whole token period for its
// dependent chain.  hfull[p] (20 warp arrivals: h parked) and sready[p] (the
// sum warp: scale written, park read) hand each park over; the producer
// thread keeps the ring `slots` tokens ahead as above.  Only consumer warp 0
// waits on an mbarrier; the others block on the consumers' named barrier,
// which takes no issue slots from the warps that work.
//
// A park holds h of chunk c8 (8 columns) as two float4 halves, A[pc] and
// B[pc], pc = c8 + c8 / (slice / 8): one float4 of padding per slice, so
// that the consumers' accesses (consecutive chunks) and the sum warp's
// (one slice per lane pair) are free of bank conflicts.
constexpr int kParks = 3;
constexpr int kPipeConsumerWarps = 20;
constexpr int kPipeConsumers = kPipeConsumerWarps * 32;
constexpr int kPipeThreads = kPipeConsumers + 32 * (kParks + 1);   // + the sum warps + the producer warp
constexpr int kPipeMaxChunks = 2;                   // chunks per consumer thread: C / 8 <= 2 * 640

struct PipeSmem {
    int slots;
    uint32_t slot_bytes, park_f4, park_off, pre_off, scale_off, bar_off, size;
};

__host__ __device__ inline PipeSmem pipe_layout(int C, bool broadcast, int slots) {
    PipeSmem m;
    m.slots = slots;
    m.slot_bytes = (uint32_t)((broadcast ? 1 : 4) * 2 * C);
    m.park_f4 = (uint32_t)(C / 8 + 16);                          // padded chunks per half
    m.park_off = (uint32_t)slots * m.slot_bytes;
    m.pre_off = m.park_off + (uint32_t)kParks * 2u * m.park_f4 * 16u;
    m.scale_off = m.pre_off + 16u * (uint32_t)slots;
    m.bar_off = m.scale_off + 16u;
    // full[slots], empty[slots], hfull[kParks], sready[kParks], the abort flag
    m.size = m.bar_off + 16u * (uint32_t)slots + 16u * (uint32_t)kParks + 16u;
    return m;
}

__device__ __forceinline__ bool pipe_consumers_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(r) : "r"((uint32_t)ok), "n"(kConsumerBar), "n"(kPipeConsumers) : "memory");
    return r != 0;
}

template <bool BCAST>
__global__ void __launch_bounds__(kPipeThreads, 1)
collapse_fold_pipe_kernel(const uint16_t* __restrict__ x, const float* __restrict__ pre,
                          const uint16_t* __restrict__ norm_w, int T, int C, int clusters, int slots,
                          float norm_eps, uint16_t* __restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    const PipeSmem m = pipe_layout(C, BCAST, slots);
    float4* parks = reinterpret_cast<float4*>(smem + m.park_off);   // park p, half q at (2p + q) * park_f4
    float4* pres = reinterpret_cast<float4*>(smem + m.pre_off);
    float* scale = reinterpret_cast<float*>(smem + m.scale_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.bar_off);
    uint64_t* empty = full + slots;
    uint64_t* hfull = empty + slots;
    uint64_t* sready = hfull + kParks;
    volatile int* abort = reinterpret_cast<volatile int*>(sready + kParks);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = C / 16, stages = (slice + 31) / 32, chunks = C / 8, spc = slice / 8;
    const uint32_t row_bytes = 2u * (uint32_t)C;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int K = b < T ? (T - 1 - b) / G + 1 : 0;         // this CTA's tokens: b, b + G, ...

    if (tid == 0) {
        for (int s = 0; s < slots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPipeConsumerWarps);
        }
        for (int p = 0; p < kParks; ++p) {
            mbar_init(&hfull[p], kPipeConsumerWarps);
            mbar_init(&sready[p], 1);
        }
        *abort = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();

    if (warp == kPipeConsumerWarps + kParks) {
        if (lane == 0)
            produce<BCAST>(x, pre, C, b, G, K, slots, m.slot_bytes, smem, pres, full, empty, abort);
        return;
    }

    if (warp >= kPipeConsumerWarps) {
        // sum warp pb (tokens k with k % 3 == pb, all in park pb): the sum of
        // squares in the tensor-core kernel's order, lane q = 2 r + group,
        // then the fold scale
        const int pb = warp - kPipeConsumerWarps;
        const int r = lane >> 1, par = lane & 1;
        const float4* hA = parks + (size_t)(2 * pb) * m.park_f4 + r * (spc + 1);
        const float4* hB = hA + m.park_f4;
        uint32_t n = 0;
        for (int k = pb; k < K; k += kParks, ++n) {
            if (!mbar_wait(&hfull[pb], n & 1u, abort)) break;
            const int it = ((b + k * G) >> 7) / clusters;   // the token's tile's round in its cluster
            const int first = (int)(((it * stages) & 1) != par);
            f32x2 sh2 = make_f32x2(0.f, 0.f);
#pragma unroll 2
            for (int stg = first; stg < stages; stg += 2) {
                // the stage's 32 columns (16 in a half last stage): chunks
                // 4 stg .. 4 stg + 3 of the slice, each as its two halves
                const int c8end = 4 * stg + (spc - 4 * stg < 4 ? spc - 4 * stg : 4);
                for (int c8 = 4 * stg; c8 < c8end; ++c8) {
                    const float4 v[2] = {hA[c8], hB[c8]};
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const f32x2 a = make_f32x2(v[c].x, v[c].y), bb = make_f32x2(v[c].z, v[c].w);
                        sh2 = fma_rn2(a, a, sh2);
                        sh2 = fma_rn2(bb, bb, sh2);
                    }
                }
            }
            float a0, a1;
            split_f32x2(sh2, a0, a1);
            const float partial = a0 + a1;
            float total = 0.f;
#pragma unroll
            for (int q = 0; q < 32; ++q) total += __shfl_sync(0xffffffffu, partial, q);
            __syncwarp();                        // every lane's reads of the park are done
            if (lane == 0) {
                scale[pb] = 1.0f / sqrtf(total / (float)C + norm_eps);
                mbar_arrive(&sready[pb]);
            }
        }
        return;
    }

    // consumers: this thread's chunks, their park positions and norm weights
    int pc[kPipeMaxChunks];
    uint4 wv[kPipeMaxChunks];
#pragma unroll
    for (int j = 0; j < kPipeMaxChunks; ++j) {
        const int c8 = tid + j * kPipeConsumers;
        pc[j] = c8 + c8 / spc;
        wv[j] = c8 < chunks ? __ldg(reinterpret_cast<const uint4*>(norm_w) + c8) : make_uint4(0, 0, 0, 0);
    }
    // iteration k collapses token k (k < K) and folds token k - 2 (k >= 2)
    int s = 0, pk = 0, pf = 0;                   // token k's slot and park, token k - 2's park
    uint32_t ph = 0, fph = 0;                    // slot s's and park pf's phase parities
    for (int k = 0; k < K + 2; ++k) {
        const bool have = k < K;
        // warp 0 waits for the slot; all consumers leave together on a failed
        // wait; the barrier also keeps the fold of token k - 3 (previous
        // iteration) ahead of the collapse into its park
        bool ok = true;
        if (warp == 0 && have) ok = mbar_wait(&full[s], ph, abort);
        if (!pipe_consumers_all(ok)) break;
        if (have) {
            const float4 pv = pres[s];
            const float p[4] = {pv.x, pv.y, pv.z, pv.w};
            const unsigned char* xs = smem + (size_t)s * m.slot_bytes;
            float4* pA = parks + (size_t)(2 * pk) * m.park_f4;
            float4* pB = pA + m.park_f4;
#pragma unroll
            for (int j = 0; j < kPipeMaxChunks; ++j) {
                const int c8 = tid + j * kPipeConsumers;
                if (c8 >= chunks) break;
                float h[8];
                collapse8<BCAST>(xs, row_bytes, c8, p, h);
                pA[pc[j]] = make_float4(h[0], h[1], h[2], h[3]);
                pB[pc[j]] = make_float4(h[4], h[5], h[6], h[7]);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);          // this warp is done with the slot
                mbar_arrive(&hfull[pk]);         // and its part of h is parked
            }
            if (++s == slots) s = 0, ph ^= 1u;
        }
        if (++pk == kParks) pk = 0;
        if (k < 2) continue;
        const int kf = k - 2;
        ok = true;
        if (warp == 0) ok = mbar_wait(&sready[pf], fph, abort);
        if (!pipe_consumers_all(ok)) break;
        const float sc = scale[pf];
        const f32x2 s2 = make_f32x2(sc, sc);
        const float4* pA = parks + (size_t)(2 * pf) * m.park_f4;
        const float4* pB = pA + m.park_f4;
        uint16_t* ot = out + (b + (int64_t)kf * G) * C;
#pragma unroll
        for (int j = 0; j < kPipeMaxChunks; ++j) {
            const int c8 = tid + j * kPipeConsumers;
            if (c8 >= chunks) break;
            const float4 v0 = pA[pc[j]], v1 = pB[pc[j]];
            st_stream(reinterpret_cast<uint4*>(ot) + c8,
                      make_uint4(
                          f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v0.x, v0.y), s2), bf16x2_to_f32x2(wv[j].x))),
                          f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v0.z, v0.w), s2), bf16x2_to_f32x2(wv[j].y))),
                          f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v1.x, v1.y), s2), bf16x2_to_f32x2(wv[j].z))),
                          f32x2_to_bf16x2(mul_rn2(mul_rn2(make_f32x2(v1.z, v1.w), s2), bf16x2_to_f32x2(wv[j].w)))));
        }
        if (++pf == kParks) pf = 0, fph ^= 1u;
    }
}

template <bool BCAST>
cudaError_t launch_pipe(const uint16_t* x, const float* pre, const uint16_t* norm_w, int64_t T, int C,
                        int clusters, float norm_eps, uint16_t* out, cudaStream_t stream, int num_sms) {
    int dev = 0, per_block = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    int slots = kMaxSlots;
    while (slots >= 2 && (int64_t)pipe_layout(C, BCAST, slots).size > per_block) --slots;
    if (slots < 2) return cudaErrorInvalidValue;
    const uint32_t smem = pipe_layout(C, BCAST, slots).size;
    e = cudaFuncSetAttribute(collapse_fold_pipe_kernel<BCAST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(T, (int64_t)num_sms);
    collapse_fold_pipe_kernel<BCAST><<<(unsigned)grid, kPipeThreads, smem, stream>>>(x, pre, norm_w, T, C, clusters,
                                                                                    slots, norm_eps, out);
    return cudaGetLastError();
}

}  // namespace

// x: [T][4][C] or the broadcast [T][C]; pre: [T][4]; C a multiple of 256;
// 16-byte aligned pointers; clusters: the number of clusters the tensor-core
// kernel ran with for this T (its tile -> round mapping).
cudaError_t launch_collapse_fold(const uint16_t* x, const float* pre, const uint16_t* norm_w, int64_t T, int C,
                                 bool broadcast, int clusters, float norm_eps, uint16_t* out, cudaStream_t stream,
                                 int num_sms) {
    if (T <= 0) return cudaSuccess;
    if (T > INT32_MAX) return cudaErrorInvalidValue;   // far beyond any device's memory
    // the slice and stage arithmetic needs C a multiple of 256, the fold
    // kernel at most two chunks per consumer thread, the round mapping a cluster
    if (C <= 0 || C % 256 != 0 || C / 8 > kPipeMaxChunks * kPipeConsumers || clusters < 1)
        return cudaErrorInvalidValue;
    if (norm_w)
        return broadcast ? launch_pipe<true>(x, pre, norm_w, T, C, clusters, norm_eps, out, stream, num_sms)
                         : launch_pipe<false>(x, pre, norm_w, T, C, clusters, norm_eps, out, stream, num_sms);
    return broadcast ? launch_nofold<true>(x, pre, T, C, out, stream, num_sms)
                     : launch_nofold<false>(x, pre, T, C, out, stream, num_sms);
}

// Host read-and-clear of this translation unit's device status word.
cudaError_t read_collapse_status(unsigned int* status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    *status = v;
    return e;
}

}  // namespace mhc
