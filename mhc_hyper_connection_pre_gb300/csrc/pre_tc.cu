// pre_tc.cu -- delayed mHC pre block with the projection on the tcgen05
// tensor cores (sm_103a), for prefill-sized token counts.
//
// Same method as pre_cluster.cu (vLLM page "Use AITER mHC for the delayed
// pre block": projection against fn plus row square-sums, gates, Sinkhorn,
// collapse with the previous seam's pre-mix; page "Fix TileLang mHC pre on
// 64-wide wavefronts", "Measurements": the fold rounded once).
//
// Why tensor cores: the projection is a dense contraction of 983,040 flop per
// token against 51 KB of HBM traffic, about 19 flop/B -- above the fp32
// CUDA-core ratio of GB300 (~74 TFLOP/s / 6.8 TB/s ~ 11 flop/B).  On tcgen05
// it is nearly free and the kernel becomes HBM-bound.  Exactness: x is bf16
// (exact as an MMA operand); fn (fp32) is split into three bf16 planes
// fn = hi + mid + lo (24 significant bits: the split is exact), stacked as
// the MMA's N = 72 rows (padded to 80), and the three accumulated planes are
// added in fp32 in the epilogue.
//
// Decomposition: a cluster of 16 CTAs owns a tile of 128 tokens (the MMA's
// M); CTA r owns C/16 columns of all four streams, holds the matching
// K-slice of the three fn planes in shared memory for the whole persistent
// launch (184 KB at C = 5120), and walks its slice in stages of
// 8 columns x 4 streams x 128 tokens (8 KB, one 3-D TMA box per stream).
// Warp roles (7 warps):
//   warp 0  TMA producer      -- 4-stage ring, mbarrier full/empty;
//   warp 1  MMA issuer        -- 2 x tcgen05.mma (M128 N80 K16) per stage into
//                                a double-buffered fp32 accumulator in TMEM;
//   warps 2-5  token rows     -- thread = token: collapse h (fp32, fixed order),
//                                sum x^2, sum h^2; h parked in TMEM columns
//                                while the fold scale is unknown; at the tile
//                                end read the 72 accumulator columns, add the
//                                planes, push 26 partials to the token's
//                                finalizer CTA over DSMEM; after the scale
//                                arrives, scale h, round once, store;
//   warp 6  finalizer         -- for its 8 tokens of the tile: sum the 16 CTAs'
//                                partials in rank order, push the fold scale
//                                to all 16 CTAs, then logits, gates and the
//                                Sinkhorn comb in registers, written to HBM.
// No global scratch; every wait is bounded (see sm100.cuh).
#include "common.cuh"
#include "sm100.cuh"

#include <cuda.h>

namespace mhc {
namespace tc {

constexpr int kCtas = 16;                         // CTAs per cluster = column slices
constexpr int kTile = 128;                        // tokens per tile = MMA M
constexpr int kStages = 4;                        // TMA ring depth
constexpr int kPrefetch = 16;                     // stages prefetched into L2 ahead of the ring
constexpr int kStageBytes = 4 * kTile * 16;       // 4 streams x 128 tokens x 8 bf16
constexpr int kMaxGroups = 40;                    // 8-column groups per CTA (C <= 5120)
constexpr int kWBlock = 2 * 9 * 128;              // per (group, k-step): 2 K-chunks x 9 row-groups
constexpr int kWBytes = kMaxGroups * 2 * kWBlock; // 184,320
constexpr int kN = 80;                            // MMA N: 72 plane rows + 8 ignored
constexpr int kPart = 26;                         // 24 dots, sum x^2, sum h^2
constexpr int kFinTok = kTile / kCtas;            // tokens finalized per CTA per tile
constexpr int kThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol0 = 0, kDCol1 = 96, kHCol = 192;  // accumulators, parked h

constexpr int kOffStages = 0;
constexpr int kOffW = kOffStages + kStages * kStageBytes;
constexpr int kOffInbox = kOffW + kWBytes;                      // [16 src][8 tok][26]
constexpr int kOffScale = kOffInbox + kCtas * kFinTok * kPart * 4;  // [128]
constexpr int kOffFinred = kOffScale + kTile * 4;               // [8][26]
constexpr int kOffBars = kOffFinred + kFinTok * kPart * 4;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1 + 1;       // full, empty, dfull, dempty, inbox, scale, drain
constexpr int kOffMisc = kOffBars + kNumBars * 8;               // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;

struct Args {
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
    int ntiles;
};

// Byte offset of the 16-byte row (8 k-values) of plane row n for 8-column
// group g, stream s, in the K-major no-swizzle B layout:
// [group][k-step j = s/2][K-chunk kk = s%2][row-group n/8][row n%8][16 B].
__device__ __forceinline__ int w_off(int g, int s, int n) {
    return ((((g * 2 + (s >> 1)) * 2 + (s & 1)) * 9 + (n >> 3)) * 8 + (n & 7)) * 16;
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
}

__global__ void __launch_bounds__(kThreads, 1)
pre_tc_kernel(const __grid_constant__ CUtensorMap xmap, const Args a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem + kOffStages;
    unsigned char* wsm = smem + kOffW;
    float* inbox = reinterpret_cast<float*>(smem + kOffInbox);
    float* scale = reinterpret_cast<float*>(smem + kOffScale);
    float* finred = reinterpret_cast<float*>(smem + kOffFinred);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* dfull = bars + 2 * kStages;
    uint64_t* dempty = dfull + 2;
    uint64_t* inbox_full = dempty + 2;
    uint64_t* scale_full = inbox_full + 1;
    uint64_t* drain = scale_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)ncluster_x();
    const int C = a.C, K = 4 * C, slice = C / kCtas, ngroups = slice / 8, c0 = (int)rank * slice;
    const bool fold = a.norm_w != nullptr;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 5);     // MMA commit + 4 token-row warps
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&dfull[d], 1);
            mbar_init(&dempty[d], 4);
        }
        mbar_init(inbox_full, kTile);    // one arrival per (source CTA, token) pair
        mbar_init(scale_full, kCtas);    // one arrival per finalizer CTA
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);

    // ---- fn K-slice -> three bf16 planes in shared memory (exact split)
    for (int idx = tid; idx < 24 * 4 * ngroups; idx += kThreads) {
        const int g = idx % ngroups, rest = idx / ngroups, s = rest & 3, m = rest >> 2;
        const float4* src = reinterpret_cast<const float4*>(a.fn + (int64_t)m * K + (int64_t)s * C + c0 + 8 * g);
        const float4 u = __ldg(src), v = __ldg(src + 1);
        const float w[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
        uint32_t pk[3][4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            uint16_t b[3][2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float w0 = w[e + q];
                const uint16_t h1 = bf16_bits_rn(w0);
                const float r1 = w0 - __uint_as_float((uint32_t)h1 << 16);
                const uint16_t h2 = bf16_bits_rn(r1);
                const float r2 = r1 - __uint_as_float((uint32_t)h2 << 16);
                b[0][q] = h1;
                b[1][q] = h2;
                b[2][q] = bf16_bits_rn(r2);
            }
#pragma unroll
            for (int p = 0; p < 3; ++p) pk[p][e >> 1] = (uint32_t)b[p][0] | ((uint32_t)b[p][1] << 16);
        }
#pragma unroll
        for (int p = 0; p < 3; ++p)
            *reinterpret_cast<uint4*>(wsm + w_off(g, s, p * 24 + m)) = make_uint4(pk[p][0], pk[p][1], pk[p][2], pk[p][3]);
    }
    fence_proxy_async_smem();  // generic-proxy writes of fn planes -> visible to the tensor core
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();        // barrier initialisation visible to the whole cluster
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================== TMA producer
        if (lane == 0) {
            // L2 prefetch of the first kPrefetch stages; afterwards each issued
            // stage prefetches the one kPrefetch later (the shared-memory ring
            // holds only 32 KB, the L2 keeps HBM requests in flight).
            auto prefetch = [&](uint32_t q) {
                const int tile_q = cid + (int)(q / ngroups) * ncl;
                if (tile_q >= a.ntiles) return;
                const int grp_q = (int)(q % ngroups);
#pragma unroll
                for (int st = 0; st < 4; ++st) tma_prefetch_3d(&xmap, c0 + 8 * grp_q, st, tile_q * kTile);
            };
            for (uint32_t q = 0; q < (uint32_t)kPrefetch; ++q) prefetch(q);
            uint32_t g = 0;
            for (int tile = cid; tile < a.ntiles && !*abort; tile += ncl) {
                for (int grp = 0; grp < ngroups; ++grp, ++g) {
                    prefetch(g + kPrefetch);
                    const int s = g % kStages;
                    const uint32_t ph = (g / kStages) & 1;
                    mbar_wait(&empty[s], ph ^ 1, abort);
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
#pragma unroll
                    for (int st = 0; st < 4; ++st)
                        tma_load_3d(stages + s * kStageBytes + st * (kTile * 16), &xmap, c0 + 8 * grp, st,
                                    tile * kTile, &full[s]);
                }
            }
            // drain: the last load of every slot has landed before the CTA exits
            for (uint32_t k = (g > (uint32_t)kStages ? g - kStages : 0); k < g; ++k)
                mbar_wait(&full[k % kStages], (k / kStages) & 1, abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTile, kN);
            const uint32_t wbase = smem_u32(wsm);
            const uint32_t sbase = smem_u32(stages);
            uint32_t g = 0;
            int it = 0;
            for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
                const int d = it & 1;
                mbar_wait(&dempty[d], ((it >> 1) & 1) ^ 1, abort);
                tc_fence_after();
                const uint32_t dt = tmem + (d ? kDCol1 : kDCol0);
                for (int grp = 0; grp < ngroups; ++grp, ++g) {
                    const int s = g % kStages;
                    mbar_wait(&full[s], (g / kStages) & 1, abort);
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint64_t ad = smem_desc(sbase + s * kStageBytes + j * 2 * (kTile * 16), kTile * 16, 128);
                        const uint64_t bd = smem_desc(wbase + (grp * 2 + j) * kWBlock, 9 * 128, 128);
                        mma_bf16(dt, ad, bd, idesc, (grp | j) != 0);
                    }
                    mma_commit(&empty[s]);
                }
                mma_commit(&dfull[d]);
            }
            mma_commit(drain);
            mbar_wait(drain, 0, abort);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================================================== token rows
        const int quad = warp & 3;
        const int trow = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const int fin = trow / kFinTok, slot = trow % kFinTok;
        const uint32_t inbox_dst = mapa(smem_u32(inbox + ((int)rank * kFinTok + slot) * kPart), fin);
        const uint32_t inbox_bar = mapa(smem_u32(inbox_full), fin);
        // The folded store of tile i is deferred into tile i+1's stage loop:
        // at group grp the thread first reads back tile i's parked h for that
        // group, scales, rounds and stores it, then parks tile i+1's new h in
        // the same TMEM columns.  The last tile is flushed after the loop.
        bool have_prev = false, valid_prev = false;
        int64_t t_prev = 0;
        float sc_prev = 1.f;
        auto store_folded = [&](int grp) {
            uint32_t r[8];
            tmem_ld8(tl + kHCol + 8 * grp, r);
            tmem_wait_ld();
            if (valid_prev) {
                float wf[8], o[8];
                unpack8(__ldg(reinterpret_cast<const uint4*>(a.norm_w + c0 + 8 * grp)), wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(__uint_as_float(r[e]), sc_prev), wf[e]);
                st_stream(reinterpret_cast<uint4*>(a.layer_input + t_prev * C + c0 + 8 * grp), pack8(o));
            }
        };
        uint32_t g = 0;
        int it = 0;
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            const int64_t t = (int64_t)tile * kTile + trow;
            const bool valid = t < a.T;
            float p[4] = {0.f, 0.f, 0.f, 0.f};
            if (valid) {
                const float4 pv = __ldg(reinterpret_cast<const float4*>(a.pre_in) + t);
                p[0] = pv.x; p[1] = pv.y; p[2] = pv.z; p[3] = pv.w;
            }
            float sx = 0.f, sh = 0.f;
            for (int grp = 0; grp < ngroups; ++grp, ++g) {
                const int s = g % kStages;
                mbar_wait(&full[s], (g / kStages) & 1, abort);
                const uint4* xb = reinterpret_cast<const uint4*>(stages + s * kStageBytes);
                float xv[4][8];
#pragma unroll
                for (int st = 0; st < 4; ++st) unpack8(xb[st * kTile + trow], xv[st]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                float h[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float v = __fmul_rn(p[0], xv[0][e]);
                    v = __fadd_rn(v, __fmul_rn(p[1], xv[1][e]));
                    v = __fadd_rn(v, __fmul_rn(p[2], xv[2][e]));
                    v = __fadd_rn(v, __fmul_rn(p[3], xv[3][e]));
                    h[e] = v;
                    sh = fmaf(v, v, sh);
#pragma unroll
                    for (int st = 0; st < 4; ++st) sx = fmaf(xv[st][e], xv[st][e], sx);
                }
                if (fold) {
                    if (have_prev) store_folded(grp);
                    uint32_t hb[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) hb[e] = __float_as_uint(h[e]);
                    tmem_st8(tl + kHCol + 8 * grp, hb);
                } else if (valid) {
                    st_stream(reinterpret_cast<uint4*>(a.layer_input + t * C + c0 + 8 * grp), pack8(h));
                }
            }
            if (fold) tmem_wait_st();

            // accumulated projection of this CTA's K-slice for the token
            const int d = it & 1;
            mbar_wait(&dfull[d], (it >> 1) & 1, abort);
            tc_fence_after();
            float acc[72];
#pragma unroll
            for (int c = 0; c < 72; c += 8) {
                uint32_t r[8];
                tmem_ld8(tl + (d ? kDCol1 : kDCol0) + c, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[c + e] = __uint_as_float(r[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[d]);
            float part[kPart];
#pragma unroll
            for (int m = 0; m < 24; ++m) part[m] = acc[m] + (acc[24 + m] + acc[48 + m]);
            part[24] = sx;
            part[25] = sh;
#pragma unroll
            for (int k = 0; k < kPart; k += 2) st_cluster_v2(inbox_dst + 4 * k, part[k], part[k + 1]);
            mbar_arrive_remote(inbox_bar);

            // this tile's fold scale from the finalizers (also: every finalizer
            // has read its inbox, so the next tile's partials may be pushed)
            mbar_wait<true>(scale_full, it & 1, abort);
            sc_prev = scale[trow];
            t_prev = t;
            valid_prev = valid;
            have_prev = true;
        }
        if (fold && have_prev)
            for (int grp = 0; grp < ngroups; ++grp) store_folded(grp);
    } else {
        // ================================================== finalizer
        const uint32_t scale_dst = mapa(smem_u32(scale + (int)rank * kFinTok), lane & (kCtas - 1));
        const uint32_t scale_bar = mapa(smem_u32(scale_full), lane & (kCtas - 1));
        int it = 0;
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            mbar_wait<true>(inbox_full, it & 1, abort);
            for (int q = lane; q < kFinTok * kPart; q += 32) {
                const int sl = q / kPart, v = q - sl * kPart;
                float s = 0.f;
#pragma unroll
                for (int src = 0; src < kCtas; ++src) s += inbox[(src * kFinTok + sl) * kPart + v];
                finred[q] = s;
            }
            __syncwarp();
            const int sl = lane & (kFinTok - 1);
            const float sx = finred[sl * kPart + 24], sh = finred[sl * kPart + 25];
            const float sfold = fold ? 1.0f / sqrtf(sh / (float)C + a.norm_eps) : 1.0f;
            float sv[kFinTok];
#pragma unroll
            for (int k = 0; k < kFinTok; ++k) sv[k] = __shfl_sync(0xffffffffu, sfold, k);
            if (lane < kCtas) {
                st_cluster_v4(scale_dst, sv[0], sv[1], sv[2], sv[3]);
                st_cluster_v4(scale_dst + 16, sv[4], sv[5], sv[6], sv[7]);
                mbar_arrive_remote(scale_bar);
            }
            const int64_t t = (int64_t)tile * kTile + (int)rank * kFinTok + lane;
            if (lane < kFinTok && t < a.T) {
                const float r = 1.0f / sqrtf(sx / (float)K + a.rms_eps);
                const float al0 = __ldg(a.alpha), al1 = __ldg(a.alpha + 1), al2 = __ldg(a.alpha + 2);
                float l[kLogits];
#pragma unroll
                for (int m = 0; m < kLogits; ++m) {
                    const float al = m < 4 ? al0 : (m < 8 ? al1 : al2);
                    l[m] = (r * finred[lane * kPart + m]) * al + __ldg(a.bias + m);
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
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
}

}  // namespace tc

using PFN_encodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
    static PFN_encodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    return fn;
}

bool pre_tc_supports(int C) { return C % (8 * tc::kCtas) == 0 && C / tc::kCtas <= 8 * tc::kMaxGroups; }
int pre_tc_tile_tokens() { return tc::kTile; }

// One-time set-up for the current device: cluster-size and shared-memory
// attributes, then the number of co-resident 16-CTA clusters (0 on error).
int pre_tc_prepare() {
    cudaError_t e = cudaFuncSetAttribute(tc::pre_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc::pre_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
    if (e != cudaSuccess || encode_fn() == nullptr) return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = tc::kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(tc::kThreads, 1, 1);
    cfg.gridDim = dim3(tc::kCtas, 1, 1);
    cfg.dynamicSmemBytes = tc::kSmemBytes;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, tc::pre_tc_kernel, &cfg);
    return e == cudaSuccess ? n : 0;
}

cudaError_t launch_pre_tc(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                          const float* alpha, const uint16_t* norm_w, int64_t T, int C, int iters,
                          float rms_eps, float norm_eps, float sk_eps, float* pre_out, float* post_out,
                          float* comb_out, uint16_t* layer_input, float* logits_out, cudaStream_t stream,
                          int max_clusters) {
    PFN_encodeTiled enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // x viewed as [T][4][C] bf16; box = 8 columns x 1 stream x 128 tokens.
    alignas(64) CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)C, 4, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)C * 8};
    const cuuint32_t box[3] = {8, 1, (cuuint32_t)tc::kTile};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    tc::Args a;
    a.x = x; a.pre_in = pre_in; a.fn = fn; a.bias = bias; a.alpha = alpha; a.norm_w = norm_w;
    a.T = T; a.C = C; a.iters = iters;
    a.rms_eps = rms_eps; a.norm_eps = norm_eps; a.sk_eps = sk_eps;
    a.pre_out = pre_out; a.post_out = post_out; a.comb_out = comb_out;
    a.layer_input = layer_input; a.logits_out = logits_out;
    a.ntiles = (int)((T + tc::kTile - 1) / tc::kTile);
    const int nclusters = a.ntiles < max_clusters ? a.ntiles : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = tc::kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(tc::kThreads, 1, 1);
    cfg.gridDim = dim3((unsigned)(nclusters * tc::kCtas), 1, 1);
    cfg.dynamicSmemBytes = tc::kSmemBytes;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, tc::pre_tc_kernel, map, a);
}

// Host read-and-clear of the device status word (synchronous).
cudaError_t read_device_status(unsigned int* status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    *status = v;
    return e;
}

}  // namespace mhc
