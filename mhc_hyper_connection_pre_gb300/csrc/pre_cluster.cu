// pre_cluster.cu -- delayed mHC pre block for small token counts (decode and
// short prefill): one cluster of 16 CTAs per tile of up to 32 tokens, the
// projection on the tensor cores through warp-level MMA (sm_103a).
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
// Decomposition.  CTA r of a cluster owns a slice of the columns (8-column
// groups spread as evenly as possible over the 16 CTAs) of all four streams:
// its K_r = 4 x ncols entries of x_flat, in 32-wide chunks.  Chunk q belongs
// to warp q mod 12, which keeps the 24 x 32 block of fn for it in registers
// (fp32) for the whole launch.  Per tile of TT tokens:
//   1. the tile's x slice and pre_in arrive by cp.async (the next tile's load
//      is issued as soon as this one's MMA is done);
//   2. all 12 warps collapse one token at a time (h to shared memory, or
//      straight to layer_input without the fold), the tokens dealt first to
//      the warps with one chunk fewer, and push the token's partial sum x^2
//      and sum h^2 to every CTA of the cluster;
//   3. every warp multiplies its chunks: up to 4 tokens with fp32 FMAs on
//      the fn registers, otherwise on the tensor cores with mma.sync m16n8k8
//      (tf32 inputs, fp32 accumulation, tokens as M in one or two 16-row
//      m-tiles, the 24 logits as three n-tiles of 8).  x (bf16) is exact in
//      tf32; fn is split into hi = fn with the low 13 mantissa bits cleared
//      (exactly a tf32 value) and lo = fn - hi (exact in fp32), two MMAs per
//      block; the MMA keeps 10 mantissa bits of lo, so each product carries
//      a relative error below 2^-20;
//   4. the 12 warps' partial dot products are summed in shared memory in a
//      fixed order and pushed to the finalising CTA, four logits per store;
//   5. CTA r finalises tokens r and r + 16 of the tile: it sums the 16
//      CTAs' partials in a fixed pairwise order and forms r and the logits;
//      warps 0 and 1 form the comb (row softmax and Sinkhorn in one lane,
//      the steps of the prefill kernels), warps 2 and 3 the gates;
//   6. meanwhile warps 2..11 form each token's fold scale from the 16 sum h^2
//      partials (the same sum, in rank order, in every CTA: the same bits),
//      fold h and store layer_input.
// Non-delayed (MODE kNonDelayed, the V4 form without an incoming pre-mix):
// the collapse needs this tile's own pre, so step 2 only sums x^2; the
// finalising CTA's gate warp sends each token's pre to all 16 CTAs as soon
// as it has the logits, then every CTA collapses with it and exchanges sum
// h^2 for the fold, while the comb warp runs the Sinkhorn chain.  The x tile is read by
// that collapse, so the next tile's x is fetched only after it.
//
// Fused with the previous seam's post (MODE kFusedPost): before step 2 every
// thread turns its share of the tile's x slice into x_new = post(x, y, comb,
// post) with the post kernel's arithmetic (the same bits), writes it out and
// leaves it in shared memory, where the pre block reads it in place of x.
//
// Every push is an st.async into the receiver's shared memory that completes
// bytes on the receiver's mbarrier, so no CTA waits at a cluster barrier for
// the slowest one inside a tile; all waits are bounded (a timeout sets the
// device status word).  Every reduction has a fixed order: results are
// deterministic.
#include "common.cuh"
#include "sm100.cuh"

namespace mhc {
namespace dec {

constexpr int kCtas = 16;                  // CTAs per cluster = column slices
constexpr int kWarps = 12;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxTile = 32;               // tokens per cluster tile
constexpr int kSlots = kMaxTile / kCtas;   // tokens each CTA finalises per tile
constexpr int kFfmaTile = 4;    // tiles of up to this many tokens project with FFMA (project_ffma)
constexpr int kRowWarp0 = kSlots;          // warps kRowWarp0.. fold (and run the non-delayed collapse);
                                            // the first kSlots of them also form the gates
constexpr int kRowWarps = kWarps - kRowWarp0;
constexpr int kSqBytes = kCtas * 2 * 4;            // per token: 16 x (sum x^2, sum h^2)
constexpr int kNumBars = 6 + 2 * kSlots;           // sq_full[p], dots_full[p][slot], pre_full[p], sh_full[p]
enum Mode { kDelayed = 0, kFusedPost = 1, kNonDelayed = 2 };
constexpr int kDotsBytes = kCtas * kLogits * 4;    // per token: 16 x 24 partial dots

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
    int64_t ntiles;
    int tile;      // tokens per tile (1..kMaxTile)
    int lcmax;     // max 8-column groups per CTA slice
    int xstride;   // bytes per token row of the x tile in shared memory
    int64_t xtok;  // elements between tokens of x: 4C, or C for the broadcast seam
    int64_t xsc;   // elements between streams of x: C, or 0 (all four read x[t])
    // previous seam's post, fused in front (y == nullptr: none)
    const uint16_t* y;
    const float* comb_prev;
    const float* post_prev;
    uint16_t* x_new;
};

// Shared-memory carve-up (bytes), in this order.
struct Layout {
    int xs, hs, red, pin, nw, sq, dots, ys, gates, prex, shin, ba, bars, abort_flag, total;
};
__host__ __device__ inline int dec_xstride(int lcmax) {
    // 64 bytes per group (4 streams x 8 bf16); rows an odd multiple of 64
    // bytes apart so that the MMA's row loads of 8 tokens hit distinct banks
    return ((64 * lcmax + 127) / 128) * 128 + 64;
}
__host__ __device__ inline Layout dec_layout(int lcmax, int mode) {
    Layout L;
    int o = 0;
    L.xs = o;    o += kMaxTile * dec_xstride(lcmax);
    L.hs = o;    o += kMaxTile * 8 * lcmax * 4;
    L.red = o;   o += kWarps * kMaxTile * kLogits * 4;
    L.pin = o;   o += kMaxTile * 16;
    L.nw = o;    o += ((8 * lcmax * 2 + 15) / 16) * 16;
    L.sq = o;    o += 2 * kMaxTile * kCtas * 2 * 4;
    L.dots = o;  o += 2 * kSlots * kCtas * kLogits * 4;
    // fused post inputs share memory with buffers first written after the
    // post step: the y slice with h, the gates with the warps' partials
    L.ys = L.hs;     // kMaxTile x 8 lcmax bf16 <= the h buffer
    L.gates = L.red; // kMaxTile x 20 fp32 <= the partials buffer
    // non-delayed: this tile's pre per token, sum h^2 partials [parity]
    L.prex = o;  o += mode == kNonDelayed ? 2 * kMaxTile * 16 : 0;
    L.shin = o;  o += mode == kNonDelayed ? 2 * kMaxTile * kCtas * 4 : 0;
    L.ba = o;    o += 2 * kLogits * 4;   // bias of each logit, then the three alphas
    L.bars = o;  o += kNumBars * 8;
    L.abort_flag = o; o += 16;
    L.total = o;
    return L;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// fp32 -> (hi, lo) with hi + lo == v exactly: hi keeps sign, exponent and
// the top 10 mantissa bits (a tf32 value as is), lo the rest.  (volatile: the
// split is redone at each use rather than hoisted into 192 live registers.)
__device__ __forceinline__ void split_tf32(float v, uint32_t& hi, uint32_t& lo) {
    asm volatile("and.b32 %0, %1, 0xffffe000;" : "=r"(hi) : "r"(__float_as_uint(v)));
    lo = __float_as_uint(v - __uint_as_float(hi));
}
// D += A (16x8, tf32, row) * B (8x8, tf32, col); fp32 accumulators.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ((q0 + q1) + (q2 + q3)) + ... : a fixed pairwise order, depth 4.
__device__ __forceinline__ float tree_sum16(const float (&q)[16]) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = q[2 * i] + q[2 * i + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = a[2 * i] + a[2 * i + 1];
    return (a[0] + a[1]) + (a[2] + a[3]);
}

// Projection of a tile of NT (<= 4) tokens with fp32 FMAs on the fn
// registers.  Lane (g, t4) sums logits g, g + 8, g + 16 over its 8 columns
// of each of its chunks, token by token; the four lanes of a group then add
// their sums (xor 1, then xor 2) and one of them stores the warp's partial.
template <int JMAX, int NT>
__device__ __forceinline__ void project_ffma(const float (&b)[JMAX][3][8], const unsigned char* xs, int xstride,
                                             int warp, int lc, int g, int t4, float* red) {
    float acc[NT][3];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
        for (int nt = 0; nt < 3; ++nt) acc[tt][nt] = 0.f;
#pragma unroll
    for (int j = 0; j < JMAX; ++j) {
        const int q = warp + kWarps * j;
        if (q < lc) {
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                float xv[8];
                unpack8(*reinterpret_cast<const uint4*>(xs + tt * xstride + (32 * q + 8 * t4) * 2), xv);
#pragma unroll
                for (int nt = 0; nt < 3; ++nt)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[tt][nt] = fmaf(b[j][nt][e], xv[e], acc[tt][nt]);
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
        for (int nt = 0; nt < 3; ++nt) {
            float v = acc[tt][nt];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (t4 == (tt & 3)) red[(warp * kMaxTile + tt) * kLogits + 8 * nt + g] = v;
        }
}

template <int JMAX, int MODE>
__global__ void __launch_bounds__(kThreads, 1) pre_decode_kernel(const Args a) {
    const int rank = (int)cluster_ctarank();
    const int64_t cid = cluster_id_x();
    const int64_t ncl = ncluster_x();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int C = a.C, K = 4 * C, nch = C >> 3;
    const float inv_k = 1.0f / (float)K;
    const int ch0 = rank * nch / kCtas;
    const int lc = (rank + 1) * nch / kCtas - ch0;   // 8-column groups of this CTA
    const int ncols = 8 * lc;
    const int c0 = 8 * ch0;
    const bool fold = a.norm_w != nullptr;
    constexpr bool fused = MODE == kFusedPost;     // the previous seam's post runs first
    constexpr bool nondel = MODE == kNonDelayed;   // collapse with this tile's own pre
    const int TT = a.tile;

    extern __shared__ __align__(128) unsigned char smem[];
    const Layout L = dec_layout(a.lcmax, MODE);
    unsigned char* xs = smem + L.xs;
    float* hs = reinterpret_cast<float*>(smem + L.hs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* pin = reinterpret_cast<float*>(smem + L.pin);
    uint16_t* nw = reinterpret_cast<uint16_t*>(smem + L.nw);
    float* inbox_sq = reinterpret_cast<float*>(smem + L.sq);      // [parity][token][src][2]
    float* inbox_dots = reinterpret_cast<float*>(smem + L.dots);  // [parity][slot][src][24]
    uint16_t* ys = reinterpret_cast<uint16_t*>(smem + L.ys);         // [token][8 lcmax]
    float* gts = reinterpret_cast<float*>(smem + L.gates);          // [token][comb 16, post 4]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* sq_full = bars;              // [parity]
    uint64_t* dots_full = bars + 2;        // [parity][slot]
    uint64_t* pre_full = bars + 2 + 2 * kSlots;   // [parity] (non-delayed)
    uint64_t* sh_full = pre_full + 2;             // [parity] (non-delayed)
    float* prex = reinterpret_cast<float*>(smem + L.prex);   // [parity][token][4]
    float* shin = reinterpret_cast<float*>(smem + L.shin);   // [parity][token][src]
    volatile int* abort = reinterpret_cast<volatile int*>(smem + L.abort_flag);
    const int hstride = 8 * a.lcmax;       // floats per token row of h

    auto tile_tokens = [&](int64_t tile) -> int {
        const int64_t left = a.T - tile * TT;
        return (int)(left < TT ? left : TT);
    };

    griddep_launch_dependents();  // the next kernel may set itself up meanwhile

    // ---- set-up: barriers armed for the first tile
    int64_t tile = cid;
    int nv = tile_tokens(tile);
    // Phases of tile k: sq_full[k & 1] (every token's 16 partials) and
    // dots_full[k & 1][slot] (the finalised tokens' 16 x 24 partials).  The
    // first tile's are armed here, tile k + 1's at the start of tile k:
    // before this CTA pushes tile k's dots, which every sender of tile
    // k + 1 bytes must have received first, and after tile k - 1's phases of
    // the same barriers completed.
    auto arm = [&](int parity, int n) {
        mbar_arrive_expect_tx(&sq_full[parity], kSqBytes * n);
        for (int s = 0; s < kSlots; ++s)
            if (kCtas * s + rank < n) mbar_arrive_expect_tx(&dots_full[parity * kSlots + s], kDotsBytes);
        if (nondel) {
            mbar_arrive_expect_tx(&pre_full[parity], 16 * n);          // every token's pre, once
            mbar_arrive_expect_tx(&sh_full[parity], kCtas * 4 * n);    // 16 x sum h^2 per token
        }
    };
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
        *abort = 0;
        fence_mbar_init_cluster();
        arm(0, nv);
    }
    // Relaxed: this arrival waits for none of the loads below.  The matching
    // wait comes before the first push into another CTA.
    cluster_arrive_relaxed();

    // ---- this warp's fn blocks, fp32 in registers: chunk q = warp + 12 j,
    //      n-tile nt (logits 8 nt .. 8 nt + 7), lane (g, t4) holds logit
    //      8 nt + g at local K 32 q + 8 t4 .. + 7
    float b[JMAX][3][8];
#pragma unroll
    for (int j = 0; j < JMAX; ++j) {
        const int q = warp + kWarps * j;
        if (q < lc) {
            const int kl = 32 * q + 8 * t4;
            const int i = kl / ncols, cc = kl - i * ncols;
            const float* src = a.fn + (int64_t)i * C + c0 + cc;
#pragma unroll
            for (int nt = 0; nt < 3; ++nt) {
                const float4* p = reinterpret_cast<const float4*>(src + (int64_t)(8 * nt + g) * K);
                const float4 u = __ldg(p), v = __ldg(p + 1);
                b[j][nt][0] = u.x; b[j][nt][1] = u.y; b[j][nt][2] = u.z; b[j][nt][3] = u.w;
                b[j][nt][4] = v.x; b[j][nt][5] = v.y; b[j][nt][6] = v.z; b[j][nt][7] = v.w;
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 3; ++nt)
#pragma unroll
                for (int e = 0; e < 8; ++e) b[j][nt][e] = 0.f;
        }
    }

    // x tile (and pre_in) of a tile into shared memory: row tt, local K order
    // (stream, column) so that local k = i * ncols + column
    auto issue_tile = [&](int64_t tl, int n) {
        const int64_t t0 = tl * TT;
        const int items = n * 4 * lc;
        for (int idx = tid; idx < items; idx += kThreads) {
            const int tt = idx / (4 * lc), r2 = idx - tt * 4 * lc;
            const int i = r2 / lc, cc = r2 - i * lc;
            // (the fused instance never takes a broadcast x)
            const int64_t xtok = fused ? 4 * (int64_t)C : a.xtok, xsc = fused ? (int64_t)C : a.xsc;
            const uint16_t* src = a.x + (t0 + tt) * xtok + i * xsc + c0 + 8 * cc;
            cp_async16(smem_u32(xs + tt * a.xstride + (i * ncols + 8 * cc) * 2), src);
        }
        if (!nondel && tid < n) cp_async16(smem_u32(pin + 4 * tid), a.pre_in + (t0 + tid) * 4);
    };
    // y slice and gates of a tile (fused post).  Their buffers double as h and
    // the partials later in a tile, so a later tile's are loaded at its start.
    auto issue_post_inputs = [&](int64_t tl, int n) {
        const int64_t t0 = tl * TT;
        {
            for (int idx = tid; idx < n * lc; idx += kThreads) {
                const int tt = idx / lc, cc = idx - tt * lc;
                cp_async16(smem_u32(ys + tt * 8 * a.lcmax + 8 * cc), a.y + (t0 + tt) * C + c0 + 8 * cc);
            }
            for (int idx = tid; idx < n * 5; idx += kThreads) {
                const int tt = idx / 5, k = idx - tt * 5;
                const float* src = k < 4 ? a.comb_prev + (t0 + tt) * 16 + 4 * k : a.post_prev + (t0 + tt) * 4;
                cp_async16(smem_u32(gts + tt * 20 + 4 * k), src);
            }
        }
    };
    if (fold)
        for (int cc = tid; cc < lc; cc += kThreads) cp_async16(smem_u32(nw + 8 * cc), a.norm_w + c0 + 8 * cc);

    // bias and alpha, read by the finalising warps (shared memory rather
    // than registers held through the whole tile).  Copied asynchronously:
    // a thread that stored a loaded value itself would wait here for the
    // load, which queues behind its warp's fn loads, and would then issue
    // its share of the x tile's copies that much later.
    float* ba = reinterpret_cast<float*>(smem + L.ba);
    if (tid < kLogits) cp_async4(smem_u32(ba + tid), a.bias + tid);
    else if (tid < kLogits + 3) cp_async4(smem_u32(ba + tid), a.alpha + (tid - kLogits));

    // Everything above reads only the weights (fn, bias, alpha, norm_w).
    // Under programmatic dependent launch it overlaps the previous kernel;
    // x and pre_in may be that kernel's output.
    griddep_wait();
    issue_tile(tile, nv);
    if (fused) issue_post_inputs(tile, nv);
    cp_async_commit();
    cluster_wait_acquire();  // every CTA's barriers are initialised before any push

    bool arrived = false;  // this thread's arrival at the final cluster barrier
    for (int round = 0; tile < a.ntiles; ++round, tile += ncl) {
        const int64_t t0 = tile * TT;
        nv = tile_tokens(tile);
        const bool last = tile + ncl >= a.ntiles;
        const int nv_next = last ? 0 : tile_tokens(tile + ncl);
        const int par = round & 1;
        cp_async_wait_all();
        __syncthreads();
        if (tid == 0 && nv_next > 0) arm(par ^ 1, nv_next);
        if (fused && round > 0) {   // h and the partials of the last tile are dead now
            issue_post_inputs(tile, nv);
            cp_async_commit();
            cp_async_wait_all();
            __syncthreads();
        }

        // ---- 1b. fused post of the previous seam: x_new for this CTA's
        //          slice of the tile, written out and kept in place of x
        if (fused) {
            if (4 * nv * lc <= kThreads) {
                // a few items (decode): four threads per item, two columns
                // each, all in one pass; every thread reads and overwrites
                // only its own columns, with the per-output order below
                for (int it = tid; it < 4 * nv * lc; it += kThreads) {
                    const int item = it >> 2, qq = it & 3;
                    const int tt = item / lc, cc = item - tt * lc;
                    const float* gt = gts + tt * 20;
                    unsigned char* xb = xs + tt * a.xstride + (8 * cc + 2 * qq) * 2;
                    float acc[4][2], v[2];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(xb + i * ncols * 2);
                        v[0] = bf16lo(w);
                        v[1] = bf16hi(w);
                        if (i == 0) post_mix_first<4, 2>(acc, v, gt);
                        else post_mix_next<4, 2>(acc, v, gt + 4 * i);
                    }
                    const uint32_t wy = *reinterpret_cast<const uint32_t*>(ys + tt * 8 * a.lcmax + 8 * cc + 2 * qq);
                    v[0] = bf16lo(wy);
                    v[1] = bf16hi(wy);
                    uint32_t o[4];
                    post_mix_last2<4>(acc, v, gt + 16, o);
#pragma unroll
                    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint32_t*>(xb + j * ncols * 2) = o[j];
                }
            } else {
                for (int it = tid; it < nv * lc; it += kThreads) {
                    const int tt = it / lc, cc = it - tt * lc;
                    const float* gt = gts + tt * 20;
                    // the item's four streams stay packed in registers, so each
                    // output can overwrite its stream in place; all four outputs
                    // are formed four columns at a time, so every element is
                    // widened from bf16 once
                    uint4 xp[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        xp[i] = *reinterpret_cast<const uint4*>(xs + tt * a.xstride + (i * ncols + 8 * cc) * 2);
                    const uint4 yp = *reinterpret_cast<const uint4*>(ys + tt * 8 * a.lcmax + 8 * cc);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float acc[4][4], v[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t w0 = hf ? xp[i].z : xp[i].x, w1 = hf ? xp[i].w : xp[i].y;
                            v[0] = bf16lo(w0); v[1] = bf16hi(w0); v[2] = bf16lo(w1); v[3] = bf16hi(w1);
                            if (i == 0) post_mix_first<4, 4>(acc, v, gt);
                            else post_mix_next<4, 4>(acc, v, gt + 4 * i);
                        }
                        {
                            const uint32_t w0 = hf ? yp.z : yp.x, w1 = hf ? yp.w : yp.y;
                            v[0] = bf16lo(w0); v[1] = bf16hi(w0); v[2] = bf16lo(w1); v[3] = bf16hi(w1);
                        }
                        uint2 o[4];
                        post_mix_last4<4>(acc, v, gt + 16, o);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint2*>(xs + tt * a.xstride + (j * ncols + 8 * cc + 4 * hf) * 2) = o[j];
                    }
                }
            }
            fence_proxy_async_smem();   // the tile's x_new is read by bulk copies below
            __syncthreads();
            // x_new out: one bulk copy per (token, stream) row of the slice
            if (tid < 4 * nv && ncols > 0) {
                const int tt = tid >> 2, i = tid & 3;
                bulk_store(a.x_new + ((t0 + tt) * 4 + i) * (int64_t)C + c0, xs + tt * a.xstride + i * ncols * 2,
                           (uint32_t)ncols * 2);
                bulk_commit_group();
            }
        }

        // ---- 2. collapse, one token per warp at a time, on all 12 warps
        //         (non-delayed: only sum x^2 here, the collapse follows the
        //         pre from the finaliser).  Warps lc % 12 .. 11 hold one fn
        //         chunk fewer than warps 0 .. lc % 12 - 1, so the tokens are
        //         dealt to them first: collapse plus projection then take
        //         about as long in every warp, and no warp idles at the
        //         barrier that ends the projection.
        const int tt0 = (warp - lc % kWarps + kWarps) % kWarps;
        if (nondel) {
            for (int tt = tt0; tt < nv; tt += kWarps) {
                float sx = 0.f;
                for (int cc = lane; cc < lc; cc += 32) {
                    float xv[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        unpack8(*reinterpret_cast<const uint4*>(xs + tt * a.xstride + (i * ncols + 8 * cc) * 2), xv[i]);
                    // the delayed block's order of accumulation, so that both
                    // blocks give the same RMS scale and gates bit for bit
#pragma unroll
                    for (int e = 0; e < 8; ++e)
#pragma unroll
                        for (int i = 0; i < 4; ++i) sx = fmaf(xv[i][e], xv[i][e], sx);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
                if (lane < kCtas)
                    st_async_v2(mapa(smem_u32(inbox_sq + ((par * kMaxTile + tt) * kCtas + rank) * 2), lane), sx, 0.f,
                                mapa(smem_u32(&sq_full[par]), lane));
            }
        }
        if (!nondel) {
            for (int tt = tt0; tt < nv; tt += kWarps) {
                const float p0 = pin[4 * tt], p1 = pin[4 * tt + 1], p2 = pin[4 * tt + 2], p3 = pin[4 * tt + 3];
                float sx = 0.f, sh = 0.f;
                for (int cc = lane; cc < lc; cc += 32) {
                    float xv[4][8], h[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        unpack8(*reinterpret_cast<const uint4*>(xs + tt * a.xstride + (i * ncols + 8 * cc) * 2), xv[i]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float v = __fmul_rn(p0, xv[0][e]);
                        v = __fadd_rn(v, __fmul_rn(p1, xv[1][e]));
                        v = __fadd_rn(v, __fmul_rn(p2, xv[2][e]));
                        v = __fadd_rn(v, __fmul_rn(p3, xv[3][e]));
                        h[e] = v;
                        sh = fmaf(v, v, sh);
#pragma unroll
                        for (int i = 0; i < 4; ++i) sx = fmaf(xv[i][e], xv[i][e], sx);
                    }
                    if (fold) {
                        float4* hp = reinterpret_cast<float4*>(hs + tt * hstride + 8 * cc);
                        hp[0] = make_float4(h[0], h[1], h[2], h[3]);
                        hp[1] = make_float4(h[4], h[5], h[6], h[7]);
                    } else {
                        st_stream(reinterpret_cast<uint4*>(a.layer_input + (t0 + tt) * C + c0 + 8 * cc), pack8(h));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sx += __shfl_xor_sync(0xffffffffu, sx, o);
                    sh += __shfl_xor_sync(0xffffffffu, sh, o);
                }
                if (lane < kCtas)   // every lane holds both sums; lane d sends them to CTA d
                    st_async_v2(mapa(smem_u32(inbox_sq + ((par * kMaxTile + tt) * kCtas + rank) * 2), lane), sx, sh,
                                mapa(smem_u32(&sq_full[par]), lane));
            }
        }

        // ---- 3. projection on the tensor cores.  Up to 16 tokens: one
        //         16-row m-tile, hi and lo products in separate accumulators.
        //         17..32 tokens: each fn fragment is split once and feeds
        //         both m-tiles, hi and lo products sharing one accumulator
        //         per m-tile so that the two tiles fit the registers of one
        //         (the lo products then round against the running hi sum:
        //         one more fp32 rounding per k-block, inside the fp32 dot
        //         bound).
        if (nv <= kFfmaTile) {
            // a few tokens: fp32 FMAs on the fn registers (a 16-row MMA
            // would spend most of its rows on absent tokens)
            switch (nv) {
                case 1: project_ffma<JMAX, 1>(b, xs, a.xstride, warp, lc, g, t4, red); break;
                case 2: project_ffma<JMAX, 2>(b, xs, a.xstride, warp, lc, g, t4, red); break;
                case 3: project_ffma<JMAX, 3>(b, xs, a.xstride, warp, lc, g, t4, red); break;
                default: project_ffma<JMAX, 4>(b, xs, a.xstride, warp, lc, g, t4, red); break;
            }
        } else if (nv <= 16) {
            float dh[3][4], dl[3][4];
#pragma unroll
            for (int nt = 0; nt < 3; ++nt)
#pragma unroll
                for (int k = 0; k < 4; ++k) dh[nt][k] = dl[nt][k] = 0.f;
#pragma unroll
            for (int j = 0; j < JMAX; ++j) {
                const int q = warp + kWarps * j;
                if (q < lc) {
                    const unsigned char* r0 = xs + g * a.xstride + (32 * q + 8 * t4) * 2;
                    const uint4 x0 = *reinterpret_cast<const uint4*>(r0);
                    const uint4 x1 = *reinterpret_cast<const uint4*>(r0 + 8 * a.xstride);
                    const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        // block blk: logical k = t4 <-> local 32q + 8 t4 + 2 blk,
                        // logical k = t4 + 4 <-> the next column
                        const uint32_t af[4] = {w0[blk] << 16, w1[blk] << 16, w0[blk] & 0xffff0000u,
                                                w1[blk] & 0xffff0000u};
#pragma unroll
                        for (int nt = 0; nt < 3; ++nt) {
                            uint32_t h0, l0, h1, l1;
                            split_tf32(b[j][nt][2 * blk], h0, l0);
                            split_tf32(b[j][nt][2 * blk + 1], h1, l1);
                            mma_tf32(dh[nt], af, h0, h1);
                            mma_tf32(dl[nt], af, l0, l1);
                        }
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 3; ++nt) {
                float* rr = red + (warp * kMaxTile + g) * kLogits + 8 * nt + 2 * t4;
                *reinterpret_cast<float2*>(rr) = make_float2(dh[nt][0] + dl[nt][0], dh[nt][1] + dl[nt][1]);
                *reinterpret_cast<float2*>(rr + 8 * kLogits) =
                    make_float2(dh[nt][2] + dl[nt][2], dh[nt][3] + dl[nt][3]);
            }
        } else {
            float d[2][3][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 3; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) d[mt][nt][k] = 0.f;
#pragma unroll
            for (int j = 0; j < JMAX; ++j) {
                const int q = warp + kWarps * j;
                if (q < lc) {
                    // rows g, g + 8 (m-tile 0) and g + 16, g + 24 (m-tile 1)
                    const unsigned char* r0 = xs + g * a.xstride + (32 * q + 8 * t4) * 2;
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        uint32_t w[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            w[r] = *reinterpret_cast<const uint32_t*>(r0 + 8 * r * a.xstride + 4 * blk);
                        const uint32_t af0[4] = {w[0] << 16, w[1] << 16, w[0] & 0xffff0000u, w[1] & 0xffff0000u};
                        const uint32_t af1[4] = {w[2] << 16, w[3] << 16, w[2] & 0xffff0000u, w[3] & 0xffff0000u};
#pragma unroll
                        for (int nt = 0; nt < 3; ++nt) {
                            uint32_t h0, l0, h1, l1;
                            split_tf32(b[j][nt][2 * blk], h0, l0);
                            split_tf32(b[j][nt][2 * blk + 1], h1, l1);
                            mma_tf32(d[0][nt], af0, h0, h1);
                            mma_tf32(d[1][nt], af1, h0, h1);
                            mma_tf32(d[0][nt], af0, l0, l1);
                            mma_tf32(d[1][nt], af1, l0, l1);
                        }
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 3; ++nt) {
                    float* rr = red + (warp * kMaxTile + 16 * mt + g) * kLogits + 8 * nt + 2 * t4;
                    *reinterpret_cast<float2*>(rr) = make_float2(d[mt][nt][0], d[mt][nt][1]);
                    *reinterpret_cast<float2*>(rr + 8 * kLogits) = make_float2(d[mt][nt][2], d[mt][nt][3]);
                }
        }
        if (fused && tid < 4 * nv) bulk_wait_read_all();   // x_new copies done reading the x tile
        __syncthreads();  // partials complete; the x tile (delayed: also pre_in) is free

        if (!last && !nondel) {
            issue_tile(tile + ncl, nv_next);
            cp_async_commit();
        }

        // ---- 4. sum the 12 warps' partials (warp order), push them to the
        //         finalising CTA, four logits per 16-byte store
        for (int pidx = tid; pidx < nv * (kLogits / 4); pidx += kThreads) {
            const int tok = pidx / (kLogits / 4), m = 4 * (pidx - tok * (kLogits / 4));
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(red + (w * kMaxTile + tok) * kLogits + m);
                s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
            }
            const uint32_t f = (uint32_t)(tok % kCtas), slot = (uint32_t)(tok / kCtas);
            st_async_v4(mapa(smem_u32(inbox_dots + ((par * kSlots + slot) * kCtas + rank) * kLogits + m), f),
                        s.x, s.y, s.z, s.w, mapa(smem_u32(&dots_full[par * kSlots + slot]), f));
        }

        if (last) {
            // every push of this CTA has been issued (relaxed: the receivers
            // count the bytes on their barriers; this barrier only keeps a
            // CTA from leaving while a peer may still push into it)
            cluster_arrive_relaxed();
            arrived = true;
        }

        // ---- 5. finalise token 16 * slot + rank.  Warp slot (0, 1) forms the
        //         comb: its 16 logits gathered into lane 0, which takes the
        //         row softmax and the Sinkhorn chain.  Warp kSlots + slot
        //         (2, 3) forms the pre and post gates (and stores the logits)
        //         meanwhile, so that none of that precedes the chain.
        if (warp < 2 * kSlots) {
            const bool comb_warp = warp < kSlots;
            const int slot = comb_warp ? warp : warp - kSlots;
            const int tok = kCtas * slot + rank;
            if (tok < nv) {
                const int64_t t = t0 + tok;
                bool ok = mbar_wait<true>(&dots_full[par * kSlots + slot], (round >> 1) & 1, abort);
                ok = ok && mbar_wait<true>(&sq_full[par], (round >> 1) & 1, abort);
                ok = __all_sync(0xffffffffu, ok);   // one outcome per warp (its shuffles below)
                if (ok) {
                    // sums over the 16 slices as fixed pairwise trees (four
                    // dependent adds instead of sixteen): x^2 in every lane,
                    // logit li in the lanes that form one
                    const float* sq = inbox_sq + (par * kMaxTile + tok) * kCtas * 2;
                    float q[kCtas];
#pragma unroll
                    for (int s2 = 0; s2 < kCtas; ++s2) q[s2] = sq[2 * s2];
                    const float sx = tree_sum16(q);
                    const int li = comb_warp ? 8 + lane : lane;
                    const int nl = comb_warp ? 16 : (a.logits_out ? kLogits : 8);
                    float l = 0.f;
                    if (lane < nl) {
                        const float* src = inbox_dots + (par * kSlots + slot) * kCtas * kLogits + li;
#pragma unroll
                        for (int s2 = 0; s2 < kCtas; ++s2) q[s2] = src[s2 * kLogits];
                        l = tree_sum16(q);
                        const float r = rsqrtf(sx * inv_k + a.rms_eps);
                        l = (r * l) * ba[kLogits + (li < 4 ? 0 : (li < 8 ? 1 : 2))] + ba[li];
                    }
                    if (comb_warp) {
                        float lc16[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) lc16[k] = __shfl_sync(0xffffffffu, l, k);
                        if (lane == 0) {
                            float P[16];
                            comb_softmax_eps(lc16, a.sk_eps, P);
                            sinkhorn_iterations(P, a.iters);
                            float4* co = reinterpret_cast<float4*>(a.comb_out + t * 16);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                co[i] = make_float4(P[4 * i], P[4 * i + 1], P[4 * i + 2], P[4 * i + 3]);
                        }
                    } else {
                        if (a.logits_out && lane < kLogits) a.logits_out[t * kLogits + lane] = l;
                        // gates: lanes 0..3 pre, 4..7 post
                        const float gate =
                            lane < 4 ? __fdividef(1.0f, 1.0f + expf(-l)) : __fdividef(2.0f, 1.0f + expf(-l));
                        if (lane < 4) a.pre_out[t * 4 + lane] = gate;
                        else if (lane < 8) a.post_out[t * 4 + lane - 4] = gate;
                        if (nondel) {   // this token's pre to every CTA, for their collapse
                            const float q0 = __shfl_sync(0xffffffffu, gate, 0), q1 = __shfl_sync(0xffffffffu, gate, 1);
                            const float q2 = __shfl_sync(0xffffffffu, gate, 2), q3 = __shfl_sync(0xffffffffu, gate, 3);
                            if (lane < kCtas)
                                st_async_v4(mapa(smem_u32(prex + (par * kMaxTile + tok) * 4), lane), q0, q1, q2, q3,
                                            mapa(smem_u32(&pre_full[par]), lane));
                        }
                    }
                }
            }
        }
        // ---- 5b. non-delayed: collapse with the tile's own pre, then send
        //          sum h^2 to every CTA (warps 2..11)
        if (nondel && warp >= kRowWarp0) {
            const bool ok = mbar_wait<true>(&pre_full[par], (round >> 1) & 1, abort);
            for (int tt = warp - kRowWarp0; ok && tt < nv; tt += kRowWarps) {
                const float* pp = prex + (par * kMaxTile + tt) * 4;
                const float p0 = pp[0], p1 = pp[1], p2 = pp[2], p3 = pp[3];
                float sh = 0.f;
                for (int cc = lane; cc < lc; cc += 32) {
                    float h[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float xv[8];
                        unpack8(*reinterpret_cast<const uint4*>(xs + tt * a.xstride + (i * ncols + 8 * cc) * 2), xv);
                        const float pi = i == 0 ? p0 : (i == 1 ? p1 : (i == 2 ? p2 : p3));
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            h[e] = i == 0 ? __fmul_rn(pi, xv[e]) : __fadd_rn(h[e], __fmul_rn(pi, xv[e]));
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) sh = fmaf(h[e], h[e], sh);
                    if (fold) {
                        float4* hp = reinterpret_cast<float4*>(hs + tt * hstride + 8 * cc);
                        hp[0] = make_float4(h[0], h[1], h[2], h[3]);
                        hp[1] = make_float4(h[4], h[5], h[6], h[7]);
                    } else {
                        st_stream(reinterpret_cast<uint4*>(a.layer_input + (t0 + tt) * C + c0 + 8 * cc), pack8(h));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sh += __shfl_xor_sync(0xffffffffu, sh, o);
                if (lane < kCtas)
                    st_async_f32(mapa(smem_u32(shin + (par * kMaxTile + tt) * kCtas + rank), lane), sh,
                                 mapa(smem_u32(&sh_full[par]), lane));
            }
        }
        if (nondel && !last) {   // the collapse above was the x tile's last reader
            __syncthreads();
            issue_tile(tile + ncl, nv_next);
            cp_async_commit();
        }

        // ---- 6. fold scales from the 16 sum h^2 partials; fold and store
        //         (warps 2..11)
        if (warp >= kRowWarp0) {
            const bool ok = nondel ? mbar_wait<true>(&sh_full[par], (round >> 1) & 1, abort)
                                   : mbar_wait<true>(&sq_full[par], (round >> 1) & 1, abort);
            if (nondel) mbar_wait<true>(&sq_full[par], (round >> 1) & 1, abort);   // every incoming byte seen
            if (fold && ok) {
                for (int tt = warp - kRowWarp0; tt < nv; tt += kRowWarps) {
                    float sh = 0.f;
                    if (nondel) {
                        const float* sp = shin + (par * kMaxTile + tt) * kCtas;
#pragma unroll
                        for (int s2 = 0; s2 < kCtas; ++s2) sh += sp[s2];
                    } else {
                        const float* sq = inbox_sq + (par * kMaxTile + tt) * kCtas * 2;
#pragma unroll
                        for (int s2 = 0; s2 < kCtas; ++s2) sh += sq[2 * s2 + 1];
                    }
                    const float s = 1.0f / sqrtf(sh / (float)C + a.norm_eps);
                    for (int cc = lane; cc < lc; cc += 32) {
                        const float4* hp = reinterpret_cast<const float4*>(hs + tt * hstride + 8 * cc);
                        const float4 h0 = hp[0], h1 = hp[1];
                        const float h[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                        float wf[8], o[8];
                        unpack8(*reinterpret_cast<const uint4*>(nw + 8 * cc), wf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(h[e], s), wf[e]);
                        st_stream(reinterpret_cast<uint4*>(a.layer_input + (t0 + tt) * C + c0 + 8 * cc), pack8(o));
                    }
                }
            }
        }
    }
    if (!arrived) cluster_arrive_relaxed();  // (a CTA with no tile)
    cp_async_wait_all();
    if (fused) bulk_wait_all();   // x_new copies complete before the CTA leaves
    // After a timeout the inbox waits above may have been cut short: the last
    // phase of each inbox barrier (peers push every tile's bytes whatever
    // happened) is waited for again, uncut, before this CTA leaves.
    __syncthreads();
    if (*abort && tid == 0) {
        const int64_t nrounds = cid < a.ntiles ? (a.ntiles - 1 - cid) / ncl + 1 : 0;
        bool seen[2 + 2 * kSlots] = {};
        for (int64_t r = nrounds - 1; r >= 0 && r >= nrounds - 4; --r) {
            const int p = (int)(r & 1);
            const uint32_t ph = (uint32_t)(r >> 1) & 1u;
            const int n = tile_tokens(cid + r * ncl);
            if (!seen[p]) {
                seen[p] = true;
                mbar_wait_drain<true>(&sq_full[p], ph);
                if (nondel) {
                    mbar_wait_drain<true>(&pre_full[p], ph);
                    mbar_wait_drain<true>(&sh_full[p], ph);
                }
            }
            for (int s = 0; s < kSlots; ++s)
                if (kCtas * s + rank < n && !seen[2 + p * kSlots + s]) {
                    seen[2 + p * kSlots + s] = true;
                    mbar_wait_drain<true>(&dots_full[p * kSlots + s], ph);
                }
        }
    }
    cluster_wait_acquire();  // no CTA leaves while a peer may still push into it
}

int lcmax_of(int C) { return (C / 8 + kCtas - 1) / kCtas; }

int jmax_of(int C) {
    const int j = (lcmax_of(C) + kWarps - 1) / kWarps;
    if (j <= 1) return 1;
    if (j <= 2) return 2;
    if (j <= 4) return 4;
    return 0;
}

cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.gridDim = dim3(kCtas, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cfg;
}

}  // namespace dec

int pre_cluster_ctas() { return dec::kCtas; }
int pre_cluster_max_tile() { return dec::kMaxTile; }

// Tokens per tile for T tokens and `max_clusters` co-resident clusters: the
// tokens spread evenly over the clusters, at most 32 per tile.
int pre_cluster_tile_tokens(int64_t T, int max_clusters) {
    if (T <= 0 || max_clusters <= 0) return 1;
    int64_t tt = (T + max_clusters - 1) / max_clusters;
    return (int)(tt < dec::kMaxTile ? tt : dec::kMaxTile);
}

// One-time set-up for the current device and hidden size C: allows the
// non-portable cluster size and the kernel's dynamic shared memory, then
// returns the maximum number of co-resident clusters (0 on error).  Must run
// before any stream capture that records the kernel.
int pre_cluster_prepare(int C) {
    // the attribute belongs to the kernel instance, which several hidden
    // sizes share: allow the largest slice that instance takes; the plan
    // uses the smaller of the two instances' co-resident cluster counts
    const int jmax = dec::jmax_of(C);
    int n_min = 0;
    cudaError_t e = cudaSuccess;
    auto setup = [&](auto kern, int mode) {
        const size_t smem = (size_t)dec::dec_layout(dec::lcmax_of(C), mode).total;
        const size_t smem_cap = (size_t)dec::dec_layout(dec::kWarps * jmax, mode).total;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = dec::cluster_config(attr, smem, nullptr);
        int n = 0;
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_cap);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        n_min = (n_min == 0 || n < n_min) ? n : n_min;
    };
    switch (jmax) {
        case 1:
            setup(dec::pre_decode_kernel<1, dec::kDelayed>, dec::kDelayed);
            setup(dec::pre_decode_kernel<1, dec::kFusedPost>, dec::kFusedPost);
            setup(dec::pre_decode_kernel<1, dec::kNonDelayed>, dec::kNonDelayed);
            break;
        case 2:
            setup(dec::pre_decode_kernel<2, dec::kDelayed>, dec::kDelayed);
            setup(dec::pre_decode_kernel<2, dec::kFusedPost>, dec::kFusedPost);
            setup(dec::pre_decode_kernel<2, dec::kNonDelayed>, dec::kNonDelayed);
            break;
        case 4:
            setup(dec::pre_decode_kernel<4, dec::kDelayed>, dec::kDelayed);
            setup(dec::pre_decode_kernel<4, dec::kFusedPost>, dec::kFusedPost);
            setup(dec::pre_decode_kernel<4, dec::kNonDelayed>, dec::kNonDelayed);
            break;
        default: return 0;
    }
    return e == cudaSuccess ? n_min : 0;
}

cudaError_t launch_pre_cluster(const uint16_t* x, const float* pre_in, const float* fn,
                               const float* bias, const float* alpha, const uint16_t* norm_w,
                               int64_t T, int C, int iters, float rms_eps, float norm_eps,
                               float sk_eps, float* pre_out, float* post_out, float* comb_out,
                               uint16_t* layer_input, float* logits_out, cudaStream_t stream,
                               int max_clusters, bool overlap, const uint16_t* y, const float* comb_prev,
                               const float* post_prev, uint16_t* x_new, bool nondelayed, bool broadcast) {
    if (broadcast && y != nullptr) return cudaErrorInvalidValue;   // no fused post on a broadcast x
    dec::Args a;
    a.y = y; a.comb_prev = comb_prev; a.post_prev = post_prev; a.x_new = x_new;
    a.x = x; a.pre_in = pre_in; a.fn = fn; a.bias = bias; a.alpha = alpha; a.norm_w = norm_w;
    a.T = T; a.C = C; a.iters = iters;
    a.rms_eps = rms_eps; a.norm_eps = norm_eps; a.sk_eps = sk_eps;
    a.pre_out = pre_out; a.post_out = post_out; a.comb_out = comb_out;
    a.layer_input = layer_input; a.logits_out = logits_out;
    a.tile = pre_cluster_tile_tokens(T, max_clusters);
    a.ntiles = (T + a.tile - 1) / a.tile;
    a.lcmax = dec::lcmax_of(C);
    a.xstride = dec::dec_xstride(a.lcmax);
    a.xtok = broadcast ? C : 4 * (int64_t)C;
    a.xsc = broadcast ? 0 : C;
    cudaLaunchAttribute attr[2];
    const int mode = nondelayed ? dec::kNonDelayed : (y != nullptr ? dec::kFusedPost : dec::kDelayed);
    cudaLaunchConfig_t cfg = dec::cluster_config(attr, (size_t)dec::dec_layout(a.lcmax, mode).total, stream);
    if (overlap) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    const int64_t nclusters = a.ntiles < max_clusters ? a.ntiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(nclusters * dec::kCtas), 1, 1);
    switch (dec::jmax_of(C) * 3 + mode) {
        case 3: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<1, dec::kDelayed>, a);
        case 4: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<1, dec::kFusedPost>, a);
        case 5: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<1, dec::kNonDelayed>, a);
        case 6: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<2, dec::kDelayed>, a);
        case 7: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<2, dec::kFusedPost>, a);
        case 8: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<2, dec::kNonDelayed>, a);
        case 12: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<4, dec::kDelayed>, a);
        case 13: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<4, dec::kFusedPost>, a);
        case 14: return cudaLaunchKernelEx(&cfg, dec::pre_decode_kernel<4, dec::kNonDelayed>, a);
        default: return cudaErrorInvalidValue;
    }
}

// Read and clear this kernel's device status word (bit 0: a bounded wait
// gave up).
cudaError_t read_decode_status(unsigned int* status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    *status = v;
    return e;
}

}  // namespace mhc
