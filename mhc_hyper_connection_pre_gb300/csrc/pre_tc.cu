// pre_tc.cu -- delayed mHC pre block with the projection on the tcgen05
// tensor cores (sm_103a), for prefill-sized token counts.
//
// Same method as pre_cluster.cu (vLLM page "Use AITER mHC for the delayed
// pre block", "Approach": the projection with each row's sum of squares,
// the gates, the Sinkhorn iterations, the collapse with the previous seam's
// pre-mix; page "Fix TileLang mHC pre on
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
// M); CTA r owns C/16 columns of all four streams and walks its slice in
// stages of 32 columns x 4 streams x 128 tokens (32 KB: one 3-D TMA box --
// x described as (column, token, stream) -- of 64-byte rows, 64-byte
// swizzle, one instruction per stage).  The three fn planes (184 KB per CTA
// rank at C = 5120), in the MMA's operand layout, come packed ahead of the
// kernel by pre_tc_pack_stage_kernel (one copy of 16 rank regions that every
// cluster reads; the library packs them per call into the workspace, or the
// caller once with mhc_pre_pack).  The kernel can still write its own
// cluster's copy in its prologue when Args::packed is null, a path the
// library no longer takes (removing it changed code generation and made the
// kernel 1.4 us slower).  Every stage brings the matching 18 KB block with
// one bulk copy (L2 evict-last) next to the x box (default L2 policy;
// evict-first was 1.6 us slower).  A 4-slot ring of 50 KB
// slots keeps 200 KB in flight per SM.  Warp roles (16 warps):
//   warp 0       TMA producer;
//   warp 1       MMA issuer: per stage 8 x tcgen05.mma (M128 N80 K16: two K
//                steps per stream) into a double-buffered fp32 accumulator
//                in TMEM;
//   warps 2-9    collapse warps, two groups of four taking alternate stages
//                (thread = token, TMEM lane quadrant = warp % 4): collapse h
//                (fp32, fixed order), sum x^2, sum h^2, park h in the stage's
//                TMEM columns once the fold warps have read the previous
//                tile's h there; at the tile end push the sums to the
//                token's scale warp (st.async into its shared memory, bytes
//                counted on its mbarrier);
//   warps 10-13  fold warps, one per lane quadrant: the tile's accumulated
//                dot products to the token's finalizer, then the tile's fold
//                scale, then every stage's parked h as soon as it is parked:
//                folded, rounded once and stored through staging tiles by TMA;
//   warp 14      finalizer: for its 8 tokens of each tile sums the 16 CTAs'
//                dot products in rank order, then logits, gates and the
//                Sinkhorn comb in registers;
//   warp 15      scale warp: for the same 8 tokens sums the 16 CTAs' sums of
//                squares in rank order and pushes the fold scales to all 16
//                CTAs at once.
// A gates-only instance (GATES) serves the first of the non-delayed block's
// two passes: the token rows only sum x^2 (in the same order, so the gates
// are the same bits), with no collapse, fold or layer_input.
// The model-entry broadcast seam (x is [T][C], the same for all four
// streams) brings one x box per stage, which the MMA and the collapse read
// as every stream: the same operands, so the same bits as the four-stream
// call on a copied x, with a quarter of the x traffic.
// The only global scratch is the fn planes in the caller's workspace; every
// wait is bounded (see sm100.cuh).
#include "common.cuh"
#include "sm100.cuh"

#include <cuda.h>

namespace mhc {
namespace tc {

constexpr int kCtas = 16;                         // CTAs per cluster = column slices
constexpr int kTile = 128;                        // tokens per tile = MMA M
constexpr int kStages = 4;                        // shared-memory ring depth
static_assert(kStages % 2 == 0, "each ring slot must always belong to the same token-row group");
constexpr int kCols = 32;                         // columns per stream per stage (64-byte rows)
constexpr int kHalf = 16;                         // columns per K16 MMA step / per output store
constexpr int kBoxBytes = kTile * kCols * 2;      // 8 KB: one stream of one stage
constexpr int kXBytes = 4 * kBoxBytes;            // 32 KB of x per stage
constexpr int kMaxGroups = 10;                    // stages per tile (C <= 5120)
constexpr int kWBlock = 9 * 512;                  // per (stage, stream): 9 row-atoms of 8 x 64 B
constexpr int kWStage = 4 * kWBlock;              // 18 KB of fn planes per stage
constexpr int kSlotBytes = kXBytes + kWStage;     // 50 KB ring slot: x boxes, then fn blocks
constexpr int kN = 80;                            // MMA N: 72 plane rows + 8 ignored
constexpr int kDots = 24;                         // projection dot products per token
constexpr int kFinTok = kTile / kCtas;            // tokens finalized per CTA per tile
constexpr int kRowWarps = 8;                      // collapse warps: two groups of four
constexpr int kFoldWarps = 4;                     // fold warps: one per TMEM lane quadrant
constexpr int kFoldWarp0 = 2 + kRowWarps;
constexpr int kFinWarp = kFoldWarp0 + kFoldWarps;
constexpr int kScaleWarp = kFinWarp + 1;
constexpr int kThreads = 32 * (kScaleWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol0 = 0, kDCol1 = 96, kHCol = 192;  // accumulators, parked h (320 columns)

constexpr int kOffStages = 0;                                         // 1 KB aligned
// The last slot's ignored 10th B-operand atom reads 512 B past the ring: the
// dots inbox follows it, so that read stays inside shared memory.
constexpr int kOffDots = kOffStages + kStages * kSlotBytes;           // [16 src][8 tok][24] dots
constexpr int kOffSq = kOffDots + kCtas * kFinTok * kDots * 4;        // [16 src][8 tok][2 grp][2] sums
constexpr int kOffScale = kOffSq + kCtas * kFinTok * 2 * 2 * 4;       // [128] fold scales
constexpr int kOffSx = kOffScale + kTile * 4;                         // [2][8] Σx² handoff
constexpr int kOffNormW = kOffSx + 2 * kFinTok * 4;                   // [C/16] bf16
// [4 fold warps][2 halves][32 tok][16 col] bf16 staging tiles, 32-byte
// swizzled: the swizzle pattern follows address bit 7, so each tile starts
// 1 KB aligned
constexpr int kOutTile = 32 * kHalf * 2;                              // 1 KB
constexpr int kOffOut = (kOffNormW + kMaxGroups * kCols * 2 + 1023) / 1024 * 1024;
constexpr int kOffBars = kOffOut + kFoldWarps * 2 * kOutTile;
// full[4], empty[4], dfull[2], dempty[2], sq_full, dots_full, scale_full,
// dots_free, drain, hfull[10], hfree[10], sx_ready[2], sx_free[2]
constexpr int kNumBars = 2 * kStages + 2 + 2 + 5 + 2 * kMaxGroups + 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;                     // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kOffBars % 8 == 0, "mbarriers need 8-byte alignment");
static_assert(kSlotBytes % 1024 == 0 && kBoxBytes % 1024 == 0 && kXBytes % 512 == 0 && kWBlock % 512 == 0,
              "64-byte-swizzled TMA boxes and MMA operand atoms must stay 512-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory budget");

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
    unsigned char* ws;  // fn planes, one region of ngroups x 18 KB per (cluster, rank)
    const unsigned char* packed;  // or planes packed ahead (one region per rank, shared by the clusters)
    int ntiles;
};

// Byte offset, inside a CTA's fn-plane region, of 16-byte chunk c (k =
// 8c..8c+7 of the stage's 32 columns) of plane row n for stage g and stream
// s: blocks [g][s] of 9 atoms x 512 B, row n in atom n/8, 64-byte swizzle in
// the atom (the layout the MMA reads once the block sits in a ring slot).
__device__ __forceinline__ int w_off(int g, int s, int n, int c) {
    return (g * 4 + s) * kWBlock + (n >> 3) * 512 + sw64_off(n & 7, c);
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
}

// fn -> three bf16 planes (hi, mid, lo): an exact split of the fp32 value.
__device__ __forceinline__ void split3(const float (&w)[8], uint32_t (&pk)[3][4]) {
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
}

// fn K-slice [c0, c0 + slice) of all 24 rows and 4 streams -> the three
// bf16 planes in the MMA operand layout at wreg (ngroups x 18 KB), by the 352
// threads of a CTA.  A warp takes units of 8 rows x the 4 column chunks of
// one (stage, stream) (lane = row * 4 + chunk), so that a load covers 8 runs
// of 128 contiguous bytes of fn and a plane store one whole 512-byte row
// atom; every thread first loads all of its items (one latency), then splits
// and stores them.  Chunks past the slice (the second half of a 16-column
// last stage) are neither read nor written: the MMA skips that half.
__device__ __forceinline__ void write_planes(const float* __restrict__ fn, int C, int c0, int slice,
                                             int ngroups, unsigned char* wreg, int warp, int lane) {
    const int64_t K = 4 * (int64_t)C;
    constexpr int kUnitsMax = (kMaxGroups * 4 * 3 + kThreads / 32 - 1) / (kThreads / 32);
    const int nunits = ngroups * 4 * 3;
    const int mrow = lane >> 2, c = lane & 3;
    float w[kUnitsMax][8];
#pragma unroll
    for (int j = 0; j < kUnitsMax; ++j) {
        const int u = warp + j * (kThreads / 32);
        const int mo = u % 3, rest = u / 3, st = rest & 3, g = rest >> 2;
        if (u < nunits && kCols * g + 8 * c < slice) {
            const int m = 8 * mo + mrow;
            const float4* src = reinterpret_cast<const float4*>(fn + (int64_t)m * K + (int64_t)st * C + c0 +
                                                                kCols * g + 8 * c);
            const float4 u0 = __ldg(src), u1 = __ldg(src + 1);
            w[j][0] = u0.x; w[j][1] = u0.y; w[j][2] = u0.z; w[j][3] = u0.w;
            w[j][4] = u1.x; w[j][5] = u1.y; w[j][6] = u1.z; w[j][7] = u1.w;
        }
    }
#pragma unroll
    for (int j = 0; j < kUnitsMax; ++j) {
        const int u = warp + j * (kThreads / 32);
        const int mo = u % 3, rest = u / 3, st = rest & 3, g = rest >> 2;
        if (u < nunits && kCols * g + 8 * c < slice) {
            const int m = 8 * mo + mrow;
            uint32_t pk[3][4];
            split3(w[j], pk);
#pragma unroll
            for (int p = 0; p < 3; ++p)
                *reinterpret_cast<uint4*>(wreg + w_off(g, st, p * 24 + m, c)) =
                    make_uint4(pk[p][0], pk[p][1], pk[p][2], pk[p][3]);
        }
    }
}

template <bool BCAST, bool GATES>
__global__ void __launch_bounds__(kThreads, 1)
pre_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap omap, const Args a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem + kOffStages;
    float* dots_in = reinterpret_cast<float*>(smem + kOffDots);
    float* sq_in = reinterpret_cast<float*>(smem + kOffSq);
    float* scale = reinterpret_cast<float*>(smem + kOffScale);
    uint16_t* nw_s = reinterpret_cast<uint16_t*>(smem + kOffNormW);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* dfull = bars + 2 * kStages;
    uint64_t* dempty = dfull + 2;
    uint64_t* sq_full = dempty + 2;       // this CTA's finalizer: Σx², Σh² of its 8 tokens arrived
    uint64_t* dots_full = sq_full + 1;    // ... their dot products arrived
    uint64_t* scale_full = dots_full + 1; // this CTA's 128 fold scales arrived
    uint64_t* dots_free = scale_full + 1; // every finalizer has read this CTA's previous dots
    uint64_t* drain = dots_free + 1;
    uint64_t* hfull = drain + 1;          // [stage]: its h of the tile is parked (collapse warps)
    uint64_t* hfree = hfull + kMaxGroups; // [stage]: its parked h has been read (fold warps)
    uint64_t* sx_ready = hfree + kMaxGroups;  // [tile & 1]: the scale warp's Σx² of the tile's 8 tokens
    uint64_t* sx_free = sx_ready + 2;         // [tile & 1]: ... read by the finalizer
    float* sx_buf = reinterpret_cast<float*>(smem + kOffSx);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)ncluster_x();
    // a slice of C/16 columns (a multiple of 16) walks ceil(slice/32) stages;
    // an odd multiple of 16 ends in a half stage of 16 columns
    const int C = a.C, K = 4 * C, slice = C / kCtas, ngroups = (slice + kCols - 1) / kCols;
    const int c0 = (int)rank * slice;
    const bool fold = a.norm_w != nullptr;
    // broadcast seam: one x box per stage, read as all four streams
    constexpr int nbox = BCAST ? 1 : 4, xbox = BCAST ? 0 : kBoxBytes;
    constexpr uint32_t slot_bytes = (uint32_t)(kSlotBytes - (4 - nbox) * kBoxBytes);
    unsigned char* wreg = a.packed ? const_cast<unsigned char*>(a.packed) + (size_t)rank * ngroups * kWStage
                                   : a.ws + (size_t)(cid * kCtas + (int)rank) * ngroups * kWStage;
    // stages of this CTA in the whole launch, and those issued before the fn planes are ready
    const int my_tiles = cid < a.ntiles ? (a.ntiles - 1 - cid) / ncl + 1 : 0;
    const uint32_t total_stages = (uint32_t)my_tiles * ngroups;
    const uint32_t early = total_stages < (uint32_t)kStages ? total_stages : (uint32_t)kStages;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 5);     // MMA commit + the stage's 4 token-row warps
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&dfull[d], 1);
            mbar_init(&dempty[d], kFoldWarps);
        }
        for (int q = 0; q < kMaxGroups; ++q) {
            mbar_init(&hfull[q], 4);             // the 4 collapse warps of the stage's group
            mbar_init(&hfree[q], kFoldWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sx_ready[b], 1);
            mbar_init(&sx_free[b], 1);
        }
        // the three cluster exchanges complete by bytes (st.async); each has
        // one local arrival per phase that arms the expected byte count
        mbar_init(sq_full, 1);           // + 16 CTAs x 8 tokens x 2 groups x 8 B
        mbar_init(dots_full, 1);         // + 16 CTAs x 8 tokens x 96 B
        mbar_init(scale_full, 1);        // + 16 finalizers x 32 B
        mbar_init(dots_free, kCtas);     // one arrival per finalizer CTA
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init_cluster();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);

    // ---- fn K-slice -> three bf16 planes in the operand layout, written to
    //      this CTA's workspace region (unless packed ahead of the call)
    if (!a.packed) write_planes(a.fn, C, c0, slice, ngroups, wreg, warp, lane);
    // the first ring slots' x boxes do not depend on fn: start them now,
    // after this CTA's fn reads (issued at the start they slowed those by
    // 2 us) and still well before the planes can be loaded
    if (tid == 0) {
        for (uint32_t q = 0; q < early; ++q) {
            const int tile = cid + (int)(q / ngroups) * ncl, grp = (int)(q % ngroups);
            mbar_arrive_expect_tx(&full[q], slot_bytes);
            tma_load_3d(stages + q * kSlotBytes, &xmap, c0 + kCols * grp, tile * kTile, 0, &full[q]);
        }
    }
    if (fold)
        for (int i = tid; i < slice / 8; i += kThreads)
            reinterpret_cast<uint4*>(nw_s)[i] = __ldg(reinterpret_cast<const uint4*>(a.norm_w + c0) + i);
    fence_proxy_async_global();  // this thread's fn-plane writes -> visible to the bulk copies
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // barrier initialisation visible to the whole cluster
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================== TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_last();
            for (uint32_t q = 0; q < early; ++q)   // fn blocks of the slots started before the planes existed
                bulk_load_hint(stages + q * kSlotBytes + kXBytes, wreg + (q % ngroups) * kWStage, kWStage,
                               &full[q], pol_w);
            uint32_t g = early;
            for (; g < total_stages && !*abort; ++g) {
                const int tile = cid + (int)(g / ngroups) * ncl, grp = (int)(g % ngroups);
                const int s = g % kStages;
                // After a timeout consumers release slots without waiting for
                // their data: a second copy must never be in flight into one
                // slot, so nothing is issued once the flag is up.  (A consumer
                // raises the flag before any early release, and the empty
                // wait acquires that release, so the read below sees it.)
                if (!mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1, abort) || *abort) break;
                unsigned char* slot = stages + s * kSlotBytes;
                mbar_arrive_expect_tx(&full[s], slot_bytes);
                tma_load_3d(slot, &xmap, c0 + kCols * grp, tile * kTile, 0, &full[s]);
                bulk_load_hint(slot + kXBytes, wreg + grp * kWStage, kWStage, &full[s], pol_w);
            }
            // drain: the last load of every slot has landed before the CTA
            // exits (waits that a timeout does not cut short)
            for (uint32_t k = (g > (uint32_t)kStages ? g - kStages : 0); k < g; ++k)
                mbar_wait_drain(&full[k % kStages], (k / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTile, kN);
            const uint32_t sbase = smem_u32(stages);
            // descriptors of the ring's base: an operand's descriptor is this
            // plus its byte offset / 16 (the 14-bit address field cannot carry:
            // shared memory ends below 256 KB)
            const uint64_t adesc0 = smem_desc(sbase, 16, 512, kLayoutSwizzle64B);
            const uint64_t bdesc0 = smem_desc(sbase + kXBytes, 16, 512, kLayoutSwizzle64B);
            uint32_t g = 0;
            int it = 0;
            for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
                const int d = it & 1;
                mbar_wait(&dempty[d], ((it >> 1) & 1) ^ 1, abort);
                tc_fence_after();
                const uint32_t dt = tmem + (d ? kDCol1 : kDCol0);
                for (int grp = 0; grp < ngroups; ++grp, ++g) {
                    const int s = g % kStages;
                    // a stage is two K16 steps (the halves of its 64-byte rows),
                    // a half stage at the end of an odd slice one
                    const int nk = kCols * grp + kHalf < slice ? 2 : 1;
                    mbar_wait(&full[s], (g / kStages) & 1, abort);
                    tc_fence_after();
                    const uint32_t so = (uint32_t)(s * kSlotBytes) >> 4;
#pragma unroll
                    for (int st = 0; st < 4; ++st)
#pragma unroll
                        for (int k = 0; k < 2; ++k)
                            if (k < nk) {
                                const uint64_t ad = adesc0 + so + (uint32_t)((st * xbox + 32 * k) >> 4);
                                const uint64_t bd = bdesc0 + so + (uint32_t)((st * kWBlock + 32 * k) >> 4);
                                mma_bf16(dt, ad, bd, idesc, (grp | st | k) != 0);
                            }
                    mma_commit(&empty[s]);
                }
                mma_commit(&dfull[d]);
            }
            // every MMA has completed before TMEM is freed, also after a timeout
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
        __syncwarp();
    } else if (warp < kFoldWarp0) {
        // ================================================== collapse warps
        // Two groups of four taking alternate stages (thread = token, TMEM
        // lane quadrant = warp % 4): load the stage's x, collapse h (fp32,
        // fixed order), sum x^2 and h^2, park h in the stage's TMEM columns
        // once the fold warps have read the previous tile's h there.
        const int grpsel = (warp - 2) >> 2;   // 0 or 1: which stages this warp takes
        const int quad = warp & 3;
        const int trow = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const int fin = trow / kFinTok, fslot = trow % kFinTok;
        const uint32_t sq_dst = mapa(smem_u32(sq_in + (((int)rank * kFinTok + fslot) * 2 + grpsel) * 2), fin);
        const uint32_t sq_bar = mapa(smem_u32(sq_full), fin);
        // byte offsets of this token's four 16-byte chunks (8 columns each)
        // in an 8 KB stream box: 64-byte rows, 64-byte swizzle
        int xo[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) xo[c] = (trow >> 3) * 512 + sw64_off(trow & 7, c);
        // pair e (columns 2e, 2e+1) of a half's 16 columns: word e & 3 of chunk e >> 2
        auto pair_of = [](const uint4 (&ch)[2], int e) -> uint32_t {
            const uint4 v = ch[e >> 2];
            return (e & 3) == 0 ? v.x : (e & 3) == 1 ? v.y : (e & 3) == 2 ? v.z : v.w;
        };
        // collapse 16 columns in scalar fp32, every product and sum rounded
        // on its own, stream order (the bit-exact reference order); the sums
        // of squares use the packed pipe in a fixed order
        auto collapse16 = [&](const uint4 (&xr)[4][2], const float (&p)[4], f32x2 (&h)[8], f32x2& sx2,
                              f32x2& sh2) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                f32x2 xv[4];
#pragma unroll
                for (int st = 0; st < 4; ++st) xv[st] = bf16x2_to_f32x2(pair_of(xr[st], e));
                float x0l, x0h, x1l, x1h, x2l, x2h, x3l, x3h;
                split_f32x2(xv[0], x0l, x0h);
                split_f32x2(xv[1], x1l, x1h);
                split_f32x2(xv[2], x2l, x2h);
                split_f32x2(xv[3], x3l, x3h);
                float vl = __fmul_rn(p[0], x0l), vh = __fmul_rn(p[0], x0h);
                vl = __fadd_rn(vl, __fmul_rn(p[1], x1l));
                vh = __fadd_rn(vh, __fmul_rn(p[1], x1h));
                vl = __fadd_rn(vl, __fmul_rn(p[2], x2l));
                vh = __fadd_rn(vh, __fmul_rn(p[2], x2h));
                vl = __fadd_rn(vl, __fmul_rn(p[3], x3l));
                vh = __fadd_rn(vh, __fmul_rn(p[3], x3h));
                const f32x2 v = make_f32x2(vl, vh);
                h[e] = v;
                sh2 = fma_rn2(v, v, sh2);
#pragma unroll
                for (int st = 0; st < 4; ++st) sx2 = fma_rn2(xv[st], xv[st], sx2);
            }
        };
        auto park = [&](int grp, int hf, const f32x2 (&h)[8]) {
            uint32_t hb[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float lo, hi;
                split_f32x2(h[e], lo, hi);
                hb[2 * e] = __float_as_uint(lo);
                hb[2 * e + 1] = __float_as_uint(hi);
            }
            tmem_st16(tl + kHCol + kCols * grp + kHalf * hf, hb);
        };
        // the pre-mix of the next tile's token is loaded a tile ahead
        auto load_pre = [&](int tl_) {
            const int64_t tt = (int64_t)tl_ * kTile + trow;
            float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tl_ < a.ntiles && tt < a.T) pv = __ldg(reinterpret_cast<const float4*>(a.pre_in) + tt);
            return pv;
        };
        float4 pnext = load_pre(cid);
        uint32_t g = 0;
        int it = 0;
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            const float p[4] = {pnext.x, pnext.y, pnext.z, pnext.w};
            pnext = load_pre(tile + ncl);
            f32x2 sx2 = make_f32x2(0.f, 0.f), sh2 = make_f32x2(0.f, 0.f);
            for (int grp = 0; grp < ngroups; ++grp, ++g) {
                if ((int)(g & 1) != grpsel) continue;  // stages alternate between the two groups
                const int s = g % kStages;                // (kStages is even: slot s -> group s % 2)
                const bool two = kCols * grp + kHalf < slice;   // a full stage, or a half stage at the end
                mbar_wait(&full[s], (g / kStages) & 1, abort);
                const unsigned char* sb = stages + s * kSlotBytes;
                // x of the token: 4 streams x 32 (or 16) columns, raw bf16 pairs
                uint4 x0[4][2], x1[4][2];
#pragma unroll
                for (int st = 0; st < 4; ++st)
#pragma unroll
                    for (int c = 0; c < 2; ++c) x0[st][c] = *reinterpret_cast<const uint4*>(sb + st * xbox + xo[c]);
                if (two)
#pragma unroll
                    for (int st = 0; st < 4; ++st)
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            x1[st][c] = *reinterpret_cast<const uint4*>(sb + st * xbox + xo[2 + c]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (GATES) {
                    // gates only: the sums of squares in the same order as
                    // below (the same RMS scale, so the same gates)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
#pragma unroll
                        for (int st = 0; st < 4; ++st) {
                            const f32x2 v = bf16x2_to_f32x2(pair_of(x0[st], e));
                            sx2 = fma_rn2(v, v, sx2);
                        }
                    if (two)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
#pragma unroll
                            for (int st = 0; st < 4; ++st) {
                                const f32x2 v = bf16x2_to_f32x2(pair_of(x1[st], e));
                                sx2 = fma_rn2(v, v, sx2);
                            }
                    continue;
                }
                f32x2 h0[8], h1[8];
                collapse16(x0, p, h0, sx2, sh2);
                if (two) collapse16(x1, p, h1, sx2, sh2);
                // the fold warps have read the previous tile's h of this stage
                if (it > 0) {
                    mbar_wait(&hfree[grp], (uint32_t)(it - 1) & 1u, abort);
                    tc_fence_after();
                }
                park(grp, 0, h0);
                if (two) park(grp, 1, h1);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hfull[grp]);
            }
            float sx, sh;
            {
                float a0, a1;
                split_f32x2(sx2, a0, a1);
                sx = a0 + a1;
                split_f32x2(sh2, a0, a1);
                sh = a0 + a1;
            }
            // the finalizer has read this CTA's previous sums once their
            // scales are back (the sums inbox is single-buffered)
            if (it > 0) mbar_wait<true>(scale_full, (uint32_t)(it - 1) & 1u, abort);
            st_async_v2(sq_dst, sx, sh, sq_bar);
        }
    } else if (warp < kFinWarp) {
        // ================================================== fold warps
        // One warp per TMEM lane quadrant (thread = token).  Per tile: the
        // accumulated projection of this CTA's K-slice to the token's
        // finalizer, then the tile's fold scale, then every stage's parked h
        // as soon as it is parked: read, scaled, weighted, rounded once and
        // stored through a staging tile by TMA; the stage's TMEM columns are
        // released to the collapse warps right after the read.
        const int quad = warp & 3;
        const int trow = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const int fin = trow / kFinTok, fslot = trow % kFinTok;
        const uint32_t dots_dst = mapa(smem_u32(dots_in + ((int)rank * kFinTok + fslot) * kDots), fin);
        const uint32_t dots_bar = mapa(smem_u32(dots_full), fin);
        const bool armer = (warp == kFoldWarp0 && lane == 0);   // arms this CTA's scale_full
        // layer_input leaves through a per-warp pair of 32-token x 16-column
        // staging tiles (32-byte swizzle), one TMA tensor store each: full
        // 32-byte sectors instead of 32 scattered 16-byte stores per
        // instruction; rows past T are clipped by the store.
        unsigned char* ostage = smem + kOffOut + (warp - kFoldWarp0) * 2 * kOutTile;
        const int oo0 = (lane >> 3) * 256 + sw32_off(lane & 7, 0);
        const int oo1 = (lane >> 3) * 256 + sw32_off(lane & 7, 1);
        auto stage_out = [&](const uint32_t (&r)[16], unsigned char* stg, int col, float sc) {
            uint32_t o[8];
            if (fold) {
                const uint4* wv = reinterpret_cast<const uint4*>(nw_s + (col - c0));
                const f32x2 sc2 = make_f32x2(sc, sc);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 w4 = wv[c];
                    const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const f32x2 hv = make_f32x2(__uint_as_float(r[8 * c + 2 * e]),
                                                    __uint_as_float(r[8 * c + 2 * e + 1]));
                        o[4 * c + e] = f32x2_to_bf16x2(mul_rn2(mul_rn2(hv, sc2), bf16x2_to_f32x2(ww[e])));  // (h * s) * w
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
            }
            *reinterpret_cast<uint4*>(stg + oo0) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(stg + oo1) = make_uint4(o[4], o[5], o[6], o[7]);
        };
        if (armer && my_tiles > 0) mbar_arrive_expect_tx(scale_full, kCtas * kFinTok * 4);
        int it = 0;
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            const int64_t t = (int64_t)tile * kTile + trow;
            {
                // accumulated projection of this CTA's K-slice for the token:
                // planes mid + lo first, then hi (24 columns each)
                const int d = it & 1;
                const uint32_t acc_col = d ? kDCol1 : kDCol0;
                mbar_wait(&dfull[d], (it >> 1) & 1, abort);
                tc_fence_after();
                uint32_t rm[3][8], rl[3][8];
#pragma unroll
                for (int c = 0; c < 3; ++c) {
                    tmem_ld8(tl + acc_col + 24 + 8 * c, rm[c]);
                    tmem_ld8(tl + acc_col + 48 + 8 * c, rl[c]);
                }
                tmem_wait_ld();
                float dots[kDots];
#pragma unroll
                for (int c = 0; c < 3; ++c) {
                    tmem_regs_ready(rm[c]);
                    tmem_regs_ready(rl[c]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) dots[8 * c + e] = __uint_as_float(rm[c][e]) + __uint_as_float(rl[c][e]);
                }
                uint32_t rh[3][8];
#pragma unroll
                for (int c = 0; c < 3; ++c) tmem_ld8(tl + acc_col + 8 * c, rh[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 3; ++c) {
                    tmem_regs_ready(rh[c]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) dots[8 * c + e] = __uint_as_float(rh[c][e]) + dots[8 * c + e];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[d]);
                // the finalizers have read this CTA's previous dots
                mbar_wait<true>(dots_free, (it & 1) ^ 1, abort);
#pragma unroll
                for (int k = 0; k < kDots; k += 4)
                    st_async_v4(dots_dst + 4 * k, dots[k], dots[k + 1], dots[k + 2], dots[k + 3], dots_bar);
            }
            // this tile's fold scale (every phase is taken, with or without a
            // fold: the collapse warps' sums protocol relies on the arming
            // of the next phase that follows)
            mbar_wait<true>(scale_full, (uint32_t)it & 1u, abort);
            const float sc = scale[trow];
            // Every fold warp has taken this phase before the next one is
            // armed: a parity wait must never fall two phases behind, and
            // without a fold (the gates-only pass) nothing else keeps the
            // four warps within one phase of each other.
            named_bar_sync(1, 32 * kFoldWarps);
            if (armer && it + 1 < my_tiles) mbar_arrive_expect_tx(scale_full, kCtas * kFinTok * 4);
            if (GATES) continue;
            for (int grp = 0; grp < ngroups; ++grp) {
                const bool two = kCols * grp + kHalf < slice;
                mbar_wait(&hfull[grp], (uint32_t)it & 1u, abort);
                tc_fence_after();
                uint32_t r0[16], r1[16];
                tmem_ld16(tl + kHCol + kCols * grp, r0);
                if (two) tmem_ld16(tl + kHCol + kCols * grp + kHalf, r1);
                tmem_wait_ld();
                tmem_regs_ready(r0);
                if (two) tmem_regs_ready(r1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hfree[grp]);   // the collapse warps may park the next tile's h
                if (lane == 0) bulk_wait_read_all();        // the previous stores have read the staging tiles
                __syncwarp();
                stage_out(r0, ostage, c0 + kCols * grp, sc);
                if (two) stage_out(r1, ostage + kOutTile, c0 + kCols * grp + kHalf, sc);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && t - lane < a.T) {
                    tma_store_2d(&omap, ostage, c0 + kCols * grp, (int)(t - lane));
                    if (two) tma_store_2d(&omap, ostage + kOutTile, c0 + kCols * grp + kHalf, (int)(t - lane));
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_all();   // stores complete before the CTA exits
    } else if (warp == kScaleWarp) {
        // ================================================== scale warp
        // For its 8 tokens of each tile: sums the 16 CTAs' Σx², Σh² partials
        // in rank order and pushes the fold scales to all 16 CTAs at once
        // (nothing else runs in this warp, so no scale waits behind the
        // Sinkhorn chain); hands Σx² to the finalizer warp.
        const uint32_t peer = (uint32_t)(lane & (kCtas - 1));
        const uint32_t scale_dst = mapa(smem_u32(scale + (int)rank * kFinTok), peer);
        const uint32_t scale_bar = mapa(smem_u32(scale_full), peer);
        int it = 0;
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            if (lane == 0) mbar_arrive_expect_tx(sq_full, kCtas * kFinTok * 2 * 8);
            mbar_wait<true>(sq_full, it & 1, abort);
            float sum = 0.f;
            if (lane < 2 * kFinTok) {
                const int tk = lane & (kFinTok - 1), v = lane >> 3;
                float vals[2 * kCtas];
#pragma unroll
                for (int q = 0; q < 2 * kCtas; ++q) vals[q] = sq_in[(((q >> 1) * kFinTok + tk) * 2 + (q & 1)) * 2 + v];
#pragma unroll
                for (int q = 0; q < 2 * kCtas; ++q) sum += vals[q];
            }
            const float sx = __shfl_sync(0xffffffffu, sum, lane & (kFinTok - 1));
            const float sh = __shfl_sync(0xffffffffu, sum, kFinTok + (lane & (kFinTok - 1)));
            const float sfold = fold ? 1.0f / sqrtf(sh / (float)C + a.norm_eps) : 1.0f;
            float sv[kFinTok];
#pragma unroll
            for (int k = 0; k < kFinTok; ++k) sv[k] = __shfl_sync(0xffffffffu, sfold, k);
            if (lane < kCtas) {
                st_async_v4(scale_dst, sv[0], sv[1], sv[2], sv[3], scale_bar);
                st_async_v4(scale_dst + 16, sv[4], sv[5], sv[6], sv[7], scale_bar);
            }
            // Σx² to the finalizer: buffer it & 1, once it has read the tile
            // that used that buffer before
            const int b = it & 1;
            if (it >= 2) mbar_wait(&sx_free[b], (uint32_t)((it >> 1) - 1) & 1u, abort);
            if (lane < kFinTok) sx_buf[b * kFinTok + lane] = sx;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sx_ready[b]);
        }
    } else {
        // ================================================== finalizer
        const uint32_t peer = (uint32_t)(lane & (kCtas - 1));
        const uint32_t scale_dst = mapa(smem_u32(scale + (int)rank * kFinTok), peer);
        const uint32_t scale_bar = mapa(smem_u32(scale_full), peer);
        const uint32_t free_bar = mapa(smem_u32(dots_free), peer);
        float bias_r[kLogits], al_r[3];
#pragma unroll
        for (int m = 0; m < kLogits; ++m) bias_r[m] = __ldg(a.bias + m);
#pragma unroll
        for (int i = 0; i < 3; ++i) al_r[i] = __ldg(a.alpha + i);
        int it = 0;
        if (lane == 0 && my_tiles > 0) mbar_arrive_expect_tx(dots_full, kCtas * kFinTok * kDots * 4);
        for (int tile = cid; tile < a.ntiles; tile += ncl, ++it) {
            // the dot products of the tile's 8 tokens, off the tiles' critical path
            mbar_wait<true>(dots_full, it & 1, abort);
            float dsum[kDots];
#pragma unroll
            for (int m = 0; m < kDots; ++m) dsum[m] = 0.f;
            if (lane < kFinTok) {
#pragma unroll 4
                for (int src = 0; src < kCtas; ++src) {
                    const float4* row = reinterpret_cast<const float4*>(dots_in + (src * kFinTok + lane) * kDots);
#pragma unroll
                    for (int k = 0; k < kDots / 4; ++k) {
                        const float4 v4 = row[k];
                        dsum[4 * k] += v4.x;
                        dsum[4 * k + 1] += v4.y;
                        dsum[4 * k + 2] += v4.z;
                        dsum[4 * k + 3] += v4.w;
                    }
                }
            }
            __syncwarp();
            if (lane < kCtas) mbar_arrive_remote(free_bar);   // inbox read: sources may push again
            if (lane == 0 && it + 1 < my_tiles) mbar_arrive_expect_tx(dots_full, kCtas * kFinTok * kDots * 4);
            // the tokens' Σx² from the scale warp
            const int b = it & 1;
            mbar_wait(&sx_ready[b], (uint32_t)(it >> 1) & 1u, abort);
            const float sx = sx_buf[b * kFinTok + (lane & (kFinTok - 1))];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sx_free[b]);
            const int64_t t = (int64_t)tile * kTile + (int)rank * kFinTok + lane;
            if (lane < kFinTok && t < a.T) {
                const float r = 1.0f / sqrtf(sx / (float)K + a.rms_eps);
                float l[kLogits];
#pragma unroll
                for (int m = 0; m < kLogits; ++m) {
                    const float al = m < 4 ? al_r[0] : (m < 8 ? al_r[1] : al_r[2]);
                    l[m] = (r * dsum[m]) * al + bias_r[m];
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
    // After a timeout the waits above may have been cut short: before this
    // CTA leaves, the last phase of each inbox (every peer pushes its bytes
    // for every tile whatever happened) is waited for again, uncut.
    if (*abort && my_tiles > 0) {
        const uint32_t lp = (uint32_t)(my_tiles - 1) & 1u;
        if (warp == kFinWarp && lane == 0) {
            mbar_wait_drain<true>(sq_full, lp);
            mbar_wait_drain<true>(dots_full, lp);
        }
        if (warp == kFoldWarp0 && lane == 0) mbar_wait_drain<true>(scale_full, lp);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
}

// Planes packed ahead of the kernel: rank r's region holds the bytes the
// kernel's prologue would write into each cluster's region.  One stage of
// one rank per CTA (grid ngroups x 16), so the whole GPU converts fn at once
// (write_planes on a one-stage slice writes that stage's bytes).
__global__ void __launch_bounds__(kThreads, 1) pre_tc_pack_stage_kernel(const float* fn, int C, unsigned char* out) {
    const int slice = C / kCtas, ngroups = (slice + kCols - 1) / kCols, g = blockIdx.x, r = blockIdx.y;
    const int sl = slice - kCols * g < kCols ? slice - kCols * g : kCols;
    write_planes(fn, C, r * slice + kCols * g, sl, 1, out + ((size_t)r * ngroups + g) * kWStage, threadIdx.x >> 5,
                 threadIdx.x & 31);
}

// Stages (32 columns, the last possibly 16) of one CTA's slice.
static int stages_of(int C) { return (C / kCtas + kCols - 1) / kCols; }

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

size_t pre_tc_packed_bytes(int C) { return (size_t)tc::kCtas * (size_t)tc::stages_of(C) * tc::kWStage; }

cudaError_t launch_pre_tc_pack(const float* fn, int C, void* out, cudaStream_t stream) {
    tc::pre_tc_pack_stage_kernel<<<dim3((unsigned)tc::stages_of(C), tc::kCtas), tc::kThreads, 0, stream>>>(
        fn, C, static_cast<unsigned char*>(out));
    return cudaGetLastError();
}

bool pre_tc_supports(int C) {
    return C % (tc::kHalf * tc::kCtas) == 0 && C / tc::kCtas <= tc::kCols * tc::kMaxGroups;
}
int pre_tc_tile_tokens() { return tc::kTile; }

// One-time set-up for the current device: cluster-size and shared-memory
// attributes, then the number of co-resident 16-CTA clusters (0 on error).
int pre_tc_prepare() {
    cudaError_t e = cudaSuccess;
    for (auto k : {tc::pre_tc_kernel<false, false>, tc::pre_tc_kernel<true, false>, tc::pre_tc_kernel<false, true>,
                   tc::pre_tc_kernel<true, true>}) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
    }
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
    e = cudaOccupancyMaxActiveClusters(&n, tc::pre_tc_kernel<false, false>, &cfg);
    return e == cudaSuccess ? n : 0;
}

cudaError_t launch_pre_tc(const uint16_t* x, const float* pre_in, const float* fn, const float* bias,
                          const float* alpha, const uint16_t* norm_w, int64_t T, int C, int iters,
                          float rms_eps, float norm_eps, float sk_eps, float* pre_out, float* post_out,
                          float* comb_out, uint16_t* layer_input, float* logits_out, void* workspace,
                          cudaStream_t stream, int max_clusters, bool broadcast, bool gates_only,
                          const void* packed) {
    PFN_encodeTiled enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // x viewed as (column, token, stream) -- the token stride 4C and the
    // stream stride C elements (broadcast: one stream) -- so that one box of
    // 32 columns (64 B) x 128 tokens x all streams lands in shared memory as
    // one 8 KB tile per stream, 64-byte swizzled as the MMA reads it: a
    // single TMA instruction per stage (the producer's issue time per stage
    // is on the kernel's critical path).  Columns past C (a half last stage
    // of the last slice) read as zeros and are not used.  No L2 promotion:
    // a CTA's slice row is C/8 bytes (640 at C = 5120), so 256-byte
    // promotion fetched up to 128 bytes of the next CTA's columns with every
    // row, bytes that were evicted again before that CTA read them -- 20 %
    // more DRAM reads of x (T = 16384: 188.8 -> 175.3 us without it).
    alignas(64) CUtensorMap map;
    const cuuint64_t ns = broadcast ? 1 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)T, ns};
    const cuuint64_t strides[2] = {(cuuint64_t)C * 2 * ns, (cuuint64_t)C * 2};
    const cuuint32_t box[3] = {(cuuint32_t)tc::kCols, (cuuint32_t)tc::kTile, (cuuint32_t)ns};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // layer_input [T][C] bf16; box = 16 columns x 32 tokens (one warp's rows)
    alignas(64) CUtensorMap omap;
    const cuuint64_t odims[2] = {(cuuint64_t)C, (cuuint64_t)T};
    const cuuint64_t ostrides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t obox[2] = {(cuuint32_t)tc::kHalf, 32};
    const cuuint32_t oestr[2] = {1, 1};
    r = enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, layer_input, odims, ostrides, obox, oestr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    tc::Args a;
    a.x = x; a.pre_in = pre_in; a.fn = fn; a.bias = bias; a.alpha = alpha; a.norm_w = norm_w;
    a.T = T; a.C = C; a.iters = iters;
    a.rms_eps = rms_eps; a.norm_eps = norm_eps; a.sk_eps = sk_eps;
    a.pre_out = pre_out; a.post_out = post_out; a.comb_out = comb_out;
    a.layer_input = layer_input; a.logits_out = logits_out;
    a.ws = static_cast<unsigned char*>(workspace);
    a.packed = static_cast<const unsigned char*>(packed);
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
    if (gates_only)
        return broadcast ? cudaLaunchKernelEx(&cfg, tc::pre_tc_kernel<true, true>, map, omap, a)
                         : cudaLaunchKernelEx(&cfg, tc::pre_tc_kernel<false, true>, map, omap, a);
    return broadcast ? cudaLaunchKernelEx(&cfg, tc::pre_tc_kernel<true, false>, map, omap, a)
                     : cudaLaunchKernelEx(&cfg, tc::pre_tc_kernel<false, false>, map, omap, a);
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
