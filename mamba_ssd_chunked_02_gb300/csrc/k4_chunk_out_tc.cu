// k4_chunk_out_tc.cu -- stage 4 on tcgen05 tensor cores: the fused output.
//
// Pages: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile" (brifing.si), section 9 "Fusing Operations in compute_out"
// (interaction matrix, carried-state term and skip term in one tiled kernel,
// the interaction matrix never in global memory) and section 11 "Causal
// Masking and Stability" (mask before exponentiating: every in-mask exponent
// is <= 0); "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
// "세 가지 핵심 커널 구현" (compute_out: the lower-triangular mask is generated
// from indices, decay by exp2) and "cuTile 기반 성능 최적화 기법" (the operand a
// kernel produces itself goes to tensor memory as MMA operand A, using
// (AB)^T = B^T A^T).
//
// For a 128-token query tile (rows t) of chunk c, keys s in [0, KS) of the same
// chunk (KS = 128 * (tile + 1)), and each head h of a block of heads that share
// the B/C group:
//   y[t,:] = sum_s M[t,s] x[s,:] + exp2(cum2_t) (C_t . Sprev_c^T) + D_h x[t,:]
//   M[t,s] = (C_t . B_s) * exp2(cum2_t - cum2_s) * dt_s  for s <= t, else 0.
// Tensor-memory plan (512 columns):
//   [0, KS/2)       CB = C_tile . B_keys^T as 16-bit pairs (GEMM1 once per CTA,
//                   in fp32 into [256, 256+KS), then packed by the epilogue:
//                   C.B^T does not depend on the head)
//   [128, 128+KS/2) M as 16-bit pairs, MMA operand A of GEMM2, in two K-halves
//                   (written by the epilogue warps with tcgen05.st)
//   [256, 384)      S: two 64-column fp32 accumulators of C . Sprev^T
//   [384, 512)      G: two 64-column fp32 accumulators of M . X
// Per head: GEMM3 S = C . Sprev^T (A = C tile, B = Sprev, both K-major in
// shared memory); the epilogue builds M from CB: the causal mask comes
// from the row/column indices; below the warp's diagonal 32x32 block the
// decay is split as exp2(cum2_t - cum2_r) * exp2(cum2_r - cum2_s) with r the
// warp's first row, so both factors are <= 1; on the fp16 path the two
// multiplies of a below-diagonal entry are packed fp16 multiplies, two keys
// per instruction.  The diagonal block takes its last key m as reference:
// exp2(cum2_t - cum2_m) in [1, 2^R] times exp2(cum2_m - cum2_s) in [2^-R, 1]
// times dt_s, packed fp16 and masked after the product, when its cum2 range R
// is at most 14 and every dt_s of the block is a normal fp16 number; otherwise
// one exp2 per element in fp32 with the mask applied before the exp2.  GEMM2 G = M . X in two
// K-halves (A from tensor memory, X MN-major in shared memory), so that the
// tensor core works on one half while
// the epilogue builds the other.  Once the next head's M is handed over, the
// epilogue finishes the previous head: y = exp2(cum2_t) S + G + D_h x_t,
// rounded to bf16, its 32x32 piece stored with a TMA store (rows past the
// sequence end are clipped by the tensor map).
//
// Precision of GEMM2.  M and X enter GEMM2 as fp16 (10-bit mantissa) rather
// than bf16 (7-bit): the worst-case error of a large output is then set by the
// final bf16 rounding of y alone.  The skip term rides along: D_h is added to
// M's diagonal, so G = M . X includes D_h x_t.  Per head the converter warps
// check that fp16 holds x and M without overflow and without their
// significant entries or factors falling to fp16 subnormals -- max|x| in
// [2^-6, 2^15], |M| <= max|C.B| max(dt) + |D_h| (every decay being <= 1) in
// [2^-4, 2^15], max|C.B| in [2^-8, 2^15], max dt >= 2^-10 -- and otherwise
// keep bf16 for that head (x stays untouched, M is packed as bf16).
//
// The fp32-output variants also carry the backward's options; one of them,
// anti-causal (a template parameter, for the backward's y' run in token order),
// takes for the rows [128 qt, 128 qt + 128) the keys [128 qt, L), builds M over
// keys at or after each row (the decay split at the warp's last row, the
// diagonal block's packed path referenced to its first key) and scales the
// carried-state term by exp2(cum2_last - cum2_t).
//
// Warp roles: 0, 1 = converters, 2 = TMA producer, 3 = MMA issuer (+ TMEM
// owner), 4 .. 4+4*EG-1 = epilogue (TMEM lane quadrant = warp % 4, column
// group (warp-4)/4).  Loads stream through a ring
// of NS stages: first the B blocks of GEMM1 (64 state dims each), then per
// head x (KS rows) and Sprev.  As soon as a head's stage lands, the converters
// copy its cum2 and dt rows into that stage's vector buffers, take the range
// check and convert the x tile to fp16 in place; the epilogue warps, which
// set the pace, only build M, rescale and write y.
#include <cuda_fp16.h>

#include <algorithm>
#include <array>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "tc5.cuh"
#include "tmap.h"

namespace m2 {
namespace {

using namespace tc;

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int EG = 2;                         // epilogue warp groups (4 warps each)
constexpr int kEpiWarps = 4 * EG;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kConvWarps = 2;                 // converter warps
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 64 + kEpiThreads + kConvThreads;
// Warp roles.  A warp issues from sub-partition (warp index % 4); the
// converters share theirs with the lightly loaded epilogue warps of lane
// quadrants 0 and 1, the producer and MMA warps (mostly waiting) with the
// busiest epilogue warps (quadrants 2 and 3, which own the most key blocks).
constexpr int kWarpProd = kConvWarps;            // converters: warps 0 .. kConvWarps-1
constexpr int kWarpMma = kConvWarps + 1;
constexpr int kEpiWarp0 = kConvWarps + 2;        // epilogue: kEpiWarp0 .. kEpiWarp0 + kEpiWarps - 1
static_assert(kEpiWarp0 % 4 == 0, "epilogue warp w accesses TMEM lane quadrant w % 4");
constexpr int PC = 64 / EG;                   // y columns per epilogue group
static_assert(PC == 32, "the epilogue moves one 32-column TMEM slice per thread");
// Tensor-memory columns: C.B^T as 16-bit pairs, M as 16-bit pairs, and two
// double-buffered fp32 accumulators (carried-state term S, intra-chunk term G).
// GEMM1 writes C.B^T in fp32 to [COL_S, COL_S + KS) before any S is live.
constexpr uint32_t COL_CB = 0, COL_MM = 128, COL_S = 256, COL_G = 384, COL_CB32 = COL_S;
constexpr uint32_t kF16MinX = 0x3c80u, kF16MaxX = 0x4700u;   // bf16 bits of 2^-6, 2^15
// C.B^T is packed as fp16 when max|C.B| lies in [2^-8, 2^15] (else bf16).
__device__ __forceinline__ bool cb_fits_f16(float cbmax) {
    return cbmax <= 32768.f && cbmax >= 0.00390625f;
}

// NA = N / 64; Y32: y stored in fp32; DOT: the backward's dot mode (no y stored:
// one y buffer, holding two 16 KB slots of staged dy, so that a third ring stage fits).
template <int L, int NA, bool Y32 = false, bool DOT = false>
struct K4Cfg {
    static constexpr int P = 64;
    static constexpr int C_BYTES = NA * 128 * 128;         // C tile: NA K-major atoms
    static constexpr int X_BYTES = L * 128;                 // x rows [0, L) (or a B block)
    static constexpr int S_BYTES = NA * 64 * 128;           // Sprev: NA K-major atoms, 64 rows
    static constexpr int STAGE = X_BYTES + S_BYTES;
    static constexpr int YW_BYTES = Y32 ? 32 * 128 : 32 * 64;   // one warp's 32x32 piece of y
    static constexpr int Y_BYTES = kEpiWarps * YW_BYTES;    // one y buffer for all warps
    // cumv[3][256], dtv[3][256] (per stage), vdt[4][256], red_x[3][kConvWarps][2], red_cb[warps]
    static constexpr int VEC_BYTES = (3 * 256 + 3 * 256 + 4 * 256 + 3 * kConvWarps * 2 + kEpiWarps) * 4;
    static constexpr int budget(int ns, int yb) {
        return 1024 + C_BYTES + ns * STAGE + yb * Y_BYTES + VEC_BYTES;
    }
    static constexpr int NS = budget(3, DOT ? 1 : 2) <= 220 * 1024 ? 3 : 2;
    static constexpr int YB = DOT ? 1 : (budget(NS, 2) <= 220 * 1024 ? 2 : 1);
    static constexpr int SMEM = budget(NS, YB);
};

struct K4Bars {
    uint64_t full[3], xfree[3];
    uint64_t cb_full;
    uint64_t cb_packed;     // C.B^T packed to 16 bits (fp32 copy may be overwritten)
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mm_ready[2], mm_free[2];   // per K-half of M
    uint64_t epi_sync;      // group barrier of the epilogue warps (abortable, unlike bar.sync)
    uint64_t drain;         // commit target used to drain in-flight MMAs on abort
    uint32_t tmem_base;
    int abort;
    uint64_t xready[3];     // per stage: x tile converted, decay vectors and flags written
    uint64_t conv_sync;     // group barrier of the converter warps (abortable)
    uint64_t cbinfo;        // max |C.B| published by the epilogue
    float cbmax;
    int use16s[3];          // per stage: GEMM2 operands of that head in fp16 (1) or bf16 (0)
    float dvals[3];         // per stage: D of that head
    uint64_t dfull[2], dfree[2];   // dx mode: the head's x and dy tiles in the y staging area
};

// Two bf16 (one word) -> f16x2, exactly when |v| is in the fp16 normal range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}


template <int L, int NA, bool kY32, bool kDot = false, bool kAnti = false>
__global__ void __launch_bounds__(kThreads, 1)
chunk_out_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_dxx,
                    const __grid_constant__ CUtensorMap tm_ddy, const float* __restrict__ cum2,
                    const float* __restrict__ dtT, const float* __restrict__ Dvec,
                    const uint32_t* __restrict__ xabs, int T, int H,
                    int G, int nc, int v1, int n1, int v2, int pts, int pst, int xdiv, int xmul, int xmod,
                    int yred, int st_mn, int dt1, const __nv_bfloat16* __restrict__ dyv,
                    float* __restrict__ ydot2, int yrev, float* __restrict__ yacc, int ycols,
                    const DxArgs dxa, int32_t* err) {
    using C = K4Cfg<L, NA, kY32, kDot>;
    constexpr int NS = C::NS, YB = C::YB, NQ = L / 128, N = NA * 64;
    // Staging slots of dx / dot mode in the y buffers: x at +0 and dy at +16384 of
    // a 32 KB slot (dx mode, TMA tiles from the producer), or dy alone in a 16 KB
    // slot (dot mode, each epilogue thread's own copies of its row).
    constexpr int kSlot = kDot ? 16384 : 32768, kSlotDy = kDot ? 0 : 16384;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sC = smem;
    uint8_t* sStage = sC + C::C_BYTES;
    uint8_t* sY = sStage + NS * C::STAGE;
    float* cumv = reinterpret_cast<float*>(sY + YB * C::Y_BYTES);    // [stage][256]
    float* dtv = cumv + 3 * 256;                                      // [stage][256]
    float* vdt = dtv + 3 * 256;                                       // [4][256]
    uint32_t* red_x = reinterpret_cast<uint32_t*>(vdt + 4 * 256);     // [stage][kConvWarps][2]
    uint32_t* red_cb = red_x + 3 * kConvWarps * 2;                    // [kEpiWarps]
    __shared__ K4Bars bars;
    volatile int* abort = &bars.abort;

    // Work item: (b, c, head block) outer; the query tiles of one item are
    // adjacent (heaviest first) so that they share x and Sprev through L2.  The
    // first n1 CTAs take blocks of v1 heads, the rest (the last (b, c) pairs)
    // blocks of v2 heads, so that the last wave of CTAs ends evenly.
    int rest = blockIdx.x, hpc = v1, bc0 = 0;
    if (rest >= n1) {
        rest -= n1;
        hpc = v2;
        bc0 = n1 / (NQ * (H / v1));
    }
    const int n_hblk = H / hpc;
    // Anti-causal mode (fp32-output variant only: the backward's y' run in token
    // order): the keys of a row are the tokens at or after it, so the tile of rows
    // [128 qt, 128 qt + 128) takes keys [128 qt, L) of the chunk.
    constexpr bool anti = kY32 && kAnti;
    const int qt = anti ? rest % NQ : NQ - 1 - rest % NQ; rest /= NQ;   // heaviest first
    const int hblk = rest % n_hblk; rest /= n_hblk;
    const int c = (bc0 + rest) % nc;
    const int b = (bc0 + rest) / nc;
    const int KS = anti ? L - 128 * qt : 128 * (qt + 1);   // keys of the tile
    const int kb = anti ? 128 * qt : 0;                    // its first key (chunk position)
    const int h0 = hblk * hpc;
    const int g = h0 / (H / G);
    const int nh = hpc;
    const int n_items = NA + nh;
    const int Lc = min(L, T - c * L);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (128 * qt >= Lc) return;       // tile entirely past the end of the sequence

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.xfree[i], 1);
        }
        mbar_init(&bars.cb_full, 1);
        mbar_init(&bars.cb_packed, kEpiThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.acc_full[i], 1);
            mbar_init(&bars.acc_empty[i], kEpiThreads);
            mbar_init(&bars.mm_ready[i], kEpiThreads);
            mbar_init(&bars.mm_free[i], 1);
        }
        mbar_init(&bars.epi_sync, kEpiThreads);
        for (int i = 0; i < NS; ++i) mbar_init(&bars.xready[i], kConvThreads);
        mbar_init(&bars.conv_sync, kConvThreads);
        mbar_init(&bars.cbinfo, 1);
        mbar_init(&bars.drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.dfull[i], 1);
            mbar_init(&bars.dfree[i], kEpiThreads);
        }
        bars.abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == kWarpProd) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            prefetch_tmap(&tm_s);
            prefetch_tmap(&tm_y);
            int issued = 0;
            for (int it = 0; it < n_items; ++it) {
                const int st = it % NS, k = it / NS;
                if (!mbar_wait_or_abort(&bars.xfree[st], (k & 1) ^ 1, abort, kWaitNs)) break;
                uint8_t* sx = sStage + st * C::STAGE;
                if (it < NA) {
                    // B block `it`: keys [kb, kb + KS) x state dims [64 it, 64 it + 64), K-major.
                    mbar_arrive_expect_tx(&bars.full[st], KS * 128 + (it == 0 ? C::C_BYTES : 0));
                    for (int r = 0; r < KS / 128; ++r)
                        tma_load_3d(sx + r * 16384, &tm_b, &bars.full[st], g * N + 64 * it,
                                    c * L + kb + 128 * r, b);
                    if (it == 0)
                        for (int a = 0; a < NA; ++a)
                            tma_load_3d(sC + a * 16384, &tm_c, &bars.full[st], g * N + 64 * a,
                                        c * L + 128 * qt, b);
                } else {
                    const int h = h0 + it - NA;
                    // The backward's options (x mapping, untransposed states, reduced or dotted
                    // output) come with fp32 y only: the forward's variant keeps none of them.
                    // pst: columns per head (32: the tile also holds the next head's columns)
                    const int xcol = kY32 ? (h / xdiv) * xmul + (h % xmod) * C::P : h * pst;
                    mbar_arrive_expect_tx(&bars.full[st], KS * 128 + C::S_BYTES);
                    for (int r = 0; r < KS / 128; ++r)
                        tma_load_3d(sx + r * 16384, &tm_x, &bars.full[st], xcol, c * L + kb + 128 * r, b);
                    // Sprev comes from stage 3: with programmatic dependent launch
                    // everything before this point ran while it was finishing.
                    if (it == NA) grid_dep_wait();
                    if (kY32 && st_mn) {   // untransposed state: N rows of (h / xmod), 64 columns
                        const int srow = (int)((((int64_t)b * nc + c) * (H / xmod) + h / xmod) * N);
                        for (int a = 0; a < NA; ++a)
                            tma_load_2d(sx + C::X_BYTES + a * 8192, &tm_s, &bars.full[st], (h % xmod) * 64,
                                        srow + 64 * a);
                    } else {
                        const int srow = (int)((((int64_t)b * nc + c) * H + h) * pst);
                        for (int a = 0; a < NA; ++a)
                            tma_load_2d(sx + C::X_BYTES + a * 8192, &tm_s, &bars.full[st], 64 * a, srow);
                    }
                }
                issued = it + 1;
            }
            if (*abort)
                for (int it = issued - 1; it >= 0 && it >= issued - NS; --it)
                    mbar_wait(&bars.full[it % NS], (it / NS) & 1, kWaitNs);
        } else if (lane == 1 && anti) {
            // dx mode (the anti-causal variant's only use): the staged tiles, from a
            // thread of their own so that the ring's loads never wait for a slot: the
            // head's x and dy rows of this tile's tokens (rows in token order) into
            // slot hi & 1.
            prefetch_tmap(&tm_dxx);
            prefetch_tmap(&tm_ddy);
            int dissued = 0;
            for (int hi = 0; hi < nh; ++hi) {
                const int sl = hi & 1, h = h0 + hi;
                if (!mbar_wait_or_abort(&bars.dfree[sl], ((hi >> 1) & 1) ^ 1, abort, kWaitNs)) break;
                uint8_t* ds = sY + sl * kSlot;
                const int row = c * L + 128 * qt;
                mbar_arrive_expect_tx(&bars.dfull[sl], 32768);
                tma_load_3d(ds, &tm_dxx, &bars.dfull[sl], h * C::P, row, b);
                tma_load_3d(ds + kSlotDy, &tm_ddy, &bars.dfull[sl], h * C::P, row, b);
                dissued = hi + 1;
            }
            if (*abort)   // the staged tiles of the last two heads issued
                for (int hi = dissued - 1; hi >= 0 && hi >= dissued - 2; --hi)
                    mbar_wait(&bars.dfull[hi & 1], (hi >> 1) & 1, kWaitNs);
        }
    } else if (warp == kWarpMma) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t c_addr = smem_u32(sC);
            const uint32_t id_cb = idesc_bf16_f32(128, KS, 0, 0);
            constexpr uint32_t id_s3 = idesc_bf16_f32(128, 64, 0, 0);
            constexpr uint32_t id_s3mn = idesc_bf16_f32(128, 64, 0, 1);   // B MN-major
            // Descriptors are formed once here; each MMA only adds a constant byte
            // offset / 16 to the start-address field: an MMA issue waits for the
            // scalar work in front of it, so that work is kept out of the chains
            // (chains of 8 N = 64 MMAs run at ~45 cycles per MMA this way, against
            // well over 100 with the descriptor rebuilt in front of each MMA).
            const uint64_t c_desc = smem_desc_sw128(c_addr, 16, 1024);                    // K-major
            const uint32_t st0 = smem_u32(sStage);
            const uint64_t bk_desc0 = smem_desc_sw128(st0, 16, 1024);                     // K-major rows
            const uint64_t xm_desc0 = smem_desc_sw128(st0, C::X_BYTES, 1024);             // MN-major x
            const uint64_t sk_desc0 = smem_desc_sw128(st0 + C::X_BYTES, 16, 1024);        // K-major Sprev
            constexpr uint64_t kStageD = C::STAGE >> 4;
            bool ok = true;
            // GEMM1: C . B^T, one 64-state-dim block per ring item.
            for (int it = 0; it < NA && ok; ++it) {
                const int st = it % NS, k = it / NS;
                const uint64_t bd0 = bk_desc0 + (uint64_t)st * kStageD;
                const uint64_t ad0 = c_desc + (uint64_t)it * (16384 >> 4);
                if (!(ok = mbar_wait_or_abort(&bars.full[st], k & 1, abort, kWaitNs))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + COL_CB32, ad0 + 2 * kk, bd0 + 2 * kk, id_cb, (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars.xfree[st]);
                if (it == NA - 1) mma_commit(&bars.cb_full);
            }
            // The fp32 C.B^T is overwritten by GEMM3: wait until the epilogue packed it.
            if (ok) {
                ok = mbar_wait_or_abort(&bars.cb_packed, 0, abort, kWaitNs);
                tc_fence_after();
            }
            // GEMM3 of head hh: S[hh & 1] = C . Sprev_hh^T.
            auto gemm3 = [&](int hh) -> bool {
                const int it = NA + hh, st = it % NS, k = it / NS, ab = hh & 1, ka = hh >> 1;
                if (!mbar_wait_or_abort(&bars.full[st], k & 1, abort, kWaitNs)) return false;
                if (!mbar_wait_or_abort(&bars.acc_empty[ab], (ka & 1) ^ 1, abort, kWaitNs)) return false;
                tc_fence_after();
                const uint64_t sd = sk_desc0 + (uint64_t)st * kStageD;
                const uint32_t acc = tmem + COL_S + 64 * ab;
                if (kY32 && st_mn) {   // B = the state tile as [K rows][64 columns], MN-major
#pragma unroll
                    for (int kk = 0; kk < N / 16; ++kk)
                        mma_ss(acc, c_desc + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                               sd + (uint64_t)(kk * (2048 >> 4)), id_s3mn, kk > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < N / 16; ++kk)
                        mma_ss(acc, c_desc + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                               sd + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id_s3, kk > 0 ? 1u : 0u);
                }
                return true;
            };
            if (ok && nh > 0) ok = gemm3(0);
            // Per head: GEMM2 as soon as the epilogue has M, then GEMM3 of the next
            // head (its S buffer frees up when the epilogue finished head hi-1).
            for (int hi = 0; hi < nh && ok; ++hi) {
                const int it = NA + hi, st = it % NS, ab = hi & 1;
                const uint64_t xd = xm_desc0 + (uint64_t)st * kStageD;
                const uint32_t acc = tmem + COL_G + 64 * ab;
                for (int half = 0; half < 2 && ok; ++half) {   // GEMM2: acc += M . X
                    if (!(ok = mbar_wait_or_abort(&bars.mm_ready[half], hi & 1, abort, kWaitNs))) break;
                    tc_fence_after();
                    const uint32_t id_s2 = bars.use16s[st] ? idesc_f16_f32(128, 64, 0, 1)
                                                              : idesc_bf16_f32(128, 64, 0, 1);
                    const int k0 = half * (KS / 32);
                    const uint32_t am = tmem + COL_MM + 8 * k0;
                    const uint64_t bd0 = xd + (uint64_t)(k0 * (2048 >> 4));
                    if (KS == 256) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(acc, am + 8 * kk, bd0 + (uint64_t)(kk * (2048 >> 4)), id_s2,
                                   (k0 + kk) > 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(acc, am + 8 * kk, bd0 + (uint64_t)(kk * (2048 >> 4)), id_s2,
                                   (k0 + kk) > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars.mm_free[half]);
                }
                if (!ok) break;
                mma_commit(&bars.acc_full[ab]);
                mma_commit(&bars.xfree[st]);
                if (hi + 1 < nh && !(ok = gemm3(hi + 1))) break;
            }
            if (*abort) {   // nothing may be in flight when TMEM is freed
                mma_commit(&bars.drain);
                mbar_wait(&bars.drain, 0, kWaitNs);
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpiWarp0;               // 0 .. kEpiWarps-1
        const int q = warp & 3;                        // TMEM lane quadrant
        const int grp = ew >> 2;                       // column group
        const int etid = threadIdx.x - 32 * kEpiWarp0; // 0 .. kEpiThreads-1
        const int tl = 32 * q + lane;                  // row within the tile
        const int tc_ = 128 * qt + tl;                 // row within the chunk
        const int jd = (128 * qt + 32 * q - kb) >> 5;  // this warp's diagonal key block
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int nblk = KS / 32, hblkn = KS / 64;    // key blocks, key blocks per K-half
        // In-mask key blocks: those up to the diagonal (causal) or from it (anti).
        const int jmin = anti ? jd : 0, jmax = anti ? nblk - 1 : jd;
        const int jown = jmin + ((grp - jmin) % EG + EG) % EG;   // first own in-mask block
        uint32_t sync_phase = 0;
        // Barrier of all epilogue threads; gives up (false) on abort or timeout.
        auto group_sync = [&]() -> bool {
            mbar_arrive(&bars.epi_sync);
            const bool r = mbar_wait_or_abort(&bars.epi_sync, sync_phase, abort, kWaitNs);
            sync_phase ^= 1u;
            return __all_sync(0xffffffffu, r);
        };
        // Key blocks outside the mask are zero for every head: write them once.
        {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            for (int j = 0; j < nblk; ++j)
                if ((j < jmin || j > jmax) && j % EG == grp) tmem_st16(tmem + lane_off + COL_MM + 16 * j, z);
            tmem_wait_st();
        }
        bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.cb_full, 0, abort, kWaitNs));
        tc_fence_after();
        // max |C.B| over the entries this tile uses (bounds |M| for the fp16 check).
        float cbmax = 0.f;
        if (ok) {
            for (int j = jown; j <= jmax; j += EG) {
                uint32_t r[32];
                tmem_ld32_sync(tmem + lane_off + COL_CB32 + 32 * j, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) cbmax = fmaxf(cbmax, fabsf(__uint_as_float(r[e])));
            }
            uint32_t m = __float_as_uint(cbmax);   // non-negative floats order as integers
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == 0) red_cb[ew] = m;
            ok = group_sync();
            const uint32_t mm = __reduce_max_sync(0xffffffffu, lane < kEpiWarps ? red_cb[lane] : 0u);
            cbmax = __uint_as_float(mm);
            if (etid == 0) {             // publish for the converter warps
                bars.cbmax = cbmax;
                mbar_arrive(&bars.cbinfo);
            }
        }
        // Pack C.B^T to 16-bit pairs: fp16 when it fits (every head may then take
        // the fp16 path), else bf16 (no head takes the fp16 path).
        const bool cb16 = cb_fits_f16(cbmax);
        if (ok) {
            for (int j = jown; j <= jmax; j += EG) {
                uint32_t r[32];
                tmem_ld32_sync(tmem + lane_off + COL_CB32 + 32 * j, r);
                uint32_t p[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    p[e] = cb16 ? pack_f16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]))
                                : pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                tmem_st16(tmem + lane_off + COL_CB + 16 * j, p);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bars.cb_packed);

        float e_prev = 0.f;
        // dx mode: dt of this thread's token and D for the head finish() handles
        // next, loaded one head ahead so that finish() does not wait for them.
        float pf_dt = 0.f, pf_D = 0.f;
        auto prefetch_dt = [&](int hp) {
            if (!anti || hp >= nh) return;
            const int k = 128 * qt + tl;
            if (k < Lc) pf_dt = __ldg(dxa.dt + ((int64_t)b * H + h0 + hp) * T + (int64_t)c * L + k);
            pf_D = dxa.D ? __ldg(dxa.D + h0 + hp) : 0.f;
        };
        prefetch_dt(0);
        // finish(hp): y rows of head hp = exp2(cum2_t) S + G (the skip term D x
        // is in G, through M's diagonal), bf16, TMA-stored per warp.
        auto finish = [&](int hp) -> bool {
            const int pb = hp & 1;
            if constexpr (kDot) {
                // Dot mode (the backward's y run): sum_p dy[t, h, p] y[t, p] over this
                // warp's 32 columns, one fp32 partial per (b, h, t, column group); y
                // itself is not written.  dy of this row first: this thread's own
                // copies into slot hp & 1 (row tl, 128-byte swizzled: 16-byte chunk cc
                // of row r at cc ^ (r & 7)), issued as head hp's iteration began (those
                // of head hp + 1 may still be in flight).  Then S and G in two 16-column
                // halves, each used before the next is loaded, so that fewer
                // accumulator words are live at once.
                if (hp + 1 < nh) cp_async_wait<1>();
                else cp_async_wait<0>();
                const uint8_t* dsr = sY + (hp & 1) * kSlot + kSlotDy + tl * 128;
                uint4 dw4[PC / 8];
#pragma unroll
                for (int k4 = 0; k4 < PC / 8; ++k4)
                    dw4[k4] = *reinterpret_cast<const uint4*>(dsr + (((grp * PC / 8 + k4) ^ (tl & 7)) << 4));
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(&bars.acc_full[pb], (hp >> 1) & 1, abort, kWaitNs)))
                    return false;
                tc_fence_after();
                float part = 0.f;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t g16[16], s16[16];
                    tmem_ld16(tmem + lane_off + COL_S + 64 * pb + grp * PC + 16 * hf, s16);
                    tmem_ld16(tmem + lane_off + COL_G + 64 * pb + grp * PC + 16 * hf, g16);
                    tmem_wait_ld_regs(s16);
                    tmem_wait_ld_regs(g16);
#pragma unroll
                    for (int k4 = 0; k4 < 2; ++k4) {
                        const uint4 w = dw4[2 * hf + k4];
                        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int e = 8 * k4 + 2 * e2;
                            part = fmaf(__uint_as_float(wv[e2] << 16),
                                        fmaf(e_prev, __uint_as_float(s16[e]), __uint_as_float(g16[e])), part);
                            part = fmaf(__uint_as_float(wv[e2] & 0xffff0000u),
                                        fmaf(e_prev, __uint_as_float(s16[e + 1]), __uint_as_float(g16[e + 1])), part);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.acc_empty[pb]);
                const int64_t t = (int64_t)c * L + 128 * qt + tl;
                if (t < T) ydot2[(((int64_t)b * H + h0 + hp) * T + t) * 2 + grp] = part;
                return true;   // the slot is next written by this thread's own copies
            }
            if constexpr (anti) {
                // dx mode (the backward's y' run, rows in token order): write
                // dx = dt y' + D dy for this row's token and the partial dots x . y' and
                // dy . x over this warp's 32 columns, from the x and dy tiles the
                // producer staged in slot hp & 1 (row tl, 128-byte swizzled: 16-byte
                // chunk cc of row r at cc ^ (r & 7)).  S and G in two 16-column halves,
                // each used before the next is loaded, so that fewer accumulator words
                // are live at once.
                const int sl = hp & 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(&bars.dfull[sl], (hp >> 1) & 1, abort, kWaitNs)))
                    return false;
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(&bars.acc_full[pb], (hp >> 1) & 1, abort, kWaitNs)))
                    return false;
                tc_fence_after();
                const uint8_t* xs = sY + sl * kSlot + tl * 128;
                const int k = 128 * qt + tl;
                const bool live = k < Lc;
                const int hh = h0 + hp;
                const int64_t t = (int64_t)c * L + k;
                float4* op = reinterpret_cast<float4*>(
                    dxa.dx + ((int64_t)b * T + t) * ((int64_t)H * C::P) + (int64_t)hh * C::P + grp * PC);
                const float dtj = pf_dt, dh = pf_D;
                float xy = 0.f, dyx = 0.f;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t g16[16], s16[16];
                    tmem_ld16(tmem + lane_off + COL_S + 64 * pb + grp * PC + 16 * hf, s16);
                    tmem_ld16(tmem + lane_off + COL_G + 64 * pb + grp * PC + 16 * hf, g16);
                    tmem_wait_ld_regs(s16);
                    tmem_wait_ld_regs(g16);
#pragma unroll
                    for (int k4 = 0; k4 < 2; ++k4) {
                        const int kc = 2 * hf + k4;   // 16-byte chunk of the row's 32 columns
                        const int cc = (grp * PC / 8 + kc) ^ (tl & 7);
                        const uint4 xw = *reinterpret_cast<const uint4*>(xs + (cc << 4));
                        const uint4 dw = *reinterpret_cast<const uint4*>(xs + kSlotDy + (cc << 4));
                        const uint32_t xv[4] = {xw.x, xw.y, xw.z, xw.w};
                        const uint32_t dv[4] = {dw.x, dw.y, dw.z, dw.w};
                        float o[8];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int e = 8 * k4 + 2 * e2;
                            const float y0 = fmaf(e_prev, __uint_as_float(s16[e]), __uint_as_float(g16[e]));
                            const float y1 = fmaf(e_prev, __uint_as_float(s16[e + 1]), __uint_as_float(g16[e + 1]));
                            const float x0 = __uint_as_float(xv[e2] << 16), x1 = __uint_as_float(xv[e2] & 0xffff0000u);
                            const float d0 = __uint_as_float(dv[e2] << 16), d1 = __uint_as_float(dv[e2] & 0xffff0000u);
                            o[2 * e2] = fmaf(dtj, y0, dh * d0);
                            o[2 * e2 + 1] = fmaf(dtj, y1, dh * d1);
                            xy = fmaf(x0, y0, fmaf(x1, y1, xy));
                            dyx = fmaf(d0, x0, fmaf(d1, x1, dyx));
                        }
                        if (live) {
                            op[2 * kc] = make_float4(o[0], o[1], o[2], o[3]);
                            op[2 * kc + 1] = make_float4(o[4], o[5], o[6], o[7]);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.acc_empty[pb]);
                // Release the slot to the next head's TMA loads: this thread's reads
                // (generic proxy) are ordered before those writes (async proxy).
                fence_proxy_async_smem();
                mbar_arrive(&bars.dfree[sl]);
                if (live) {
                    const int64_t po = (((int64_t)b * H + hh) * T + t) * 2 + grp;
                    dxa.xy[po] = xy;
                    dxa.dyx[po] = dyx;
                }
                prefetch_dt(hp + 1);
                return true;
            }
            if (!__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bars.acc_full[pb], (hp >> 1) & 1, abort, kWaitNs)))
                return false;
            tc_fence_after();
            uint32_t r[32], rs[32];
            tmem_ld32(tmem + lane_off + COL_S + 64 * pb + grp * PC, rs);
            tmem_ld32(tmem + lane_off + COL_G + 64 * pb + grp * PC, r);
            tmem_wait_ld_regs(rs);
            tmem_wait_ld_regs(r);
            tc_fence_before();
            mbar_arrive(&bars.acc_empty[pb]);
            uint8_t* yw = sY + (hp % YB) * C::Y_BYTES + ew * C::YW_BYTES;
            // Reversed rows (yrev, with yred): the run's row k of the chunk is token
            // Lc - 1 - k, so this warp's 32 rows are 32 consecutive tokens in reverse
            // order, starting at row0; a block that would start before token 0 (only
            // when T < L) is added element by element instead.
            const bool rev = kY32 && yrev;
            const int row0 = rev ? c * L + Lc - 32 - (128 * qt + 32 * q) : c * L + 128 * qt + 32 * q;
            const int rr = rev ? 31 - lane : lane;           // staging row of this lane
            if constexpr (kY32) {
                // fp32 piece: 128-byte rows, 128-byte swizzled (16-byte chunk k
                // of row r at k ^ (r & 7); the buffer is 1024-byte aligned).
                uint32_t yv[PC];
#pragma unroll
                for (int e = 0; e < PC; ++e)
                    yv[e] = __float_as_uint(fmaf(e_prev, __uint_as_float(rs[e]), __uint_as_float(r[e])));
                if (rev && row0 < 0) {
                    const int k = 128 * qt + 32 * q + lane;
                    if (k < Lc) {
                        const int hy = h0 + hp;
                        float* dst = yacc + ((int64_t)b * T + (c * L + Lc - 1 - k)) * ycols +
                                     (hy / xdiv) * xmul + (hy % xmod) * C::P + grp * PC;
#pragma unroll
                        for (int e = 0; e < PC; ++e) atomicAdd(dst + e, __uint_as_float(yv[e]));
                    }
                    return true;
                }
                if (lane == 0) bulk_wait_read<YB - 1>();   // this warp's store from YB heads ago
                __syncwarp();
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4*>(yw + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
                        make_uint4(yv[4 * cc], yv[4 * cc + 1], yv[4 * cc + 2], yv[4 * cc + 3]);
            } else {
                uint32_t yv[PC / 2];
#pragma unroll
                for (int e = 0; e < PC / 2; ++e)
                    yv[e] = pack_bf16x2(fmaf(e_prev, __uint_as_float(rs[2 * e]), __uint_as_float(r[2 * e])),
                                        fmaf(e_prev, __uint_as_float(rs[2 * e + 1]), __uint_as_float(r[2 * e + 1])));
                // This warp's 32 x 32 piece, 64-byte swizzled (16-byte chunk k of
                // row r at k ^ ((r >> 1) & 3)), stored by one lane with TMA.
                if (lane == 0) bulk_wait_read<YB - 1>();   // this warp's store from YB heads ago
                __syncwarp();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    *reinterpret_cast<uint4*>(yw + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(yv[4 * cc], yv[4 * cc + 1], yv[4 * cc + 2], yv[4 * cc + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int hy = h0 + hp;
                if (kY32 && yred)   // add into the head's columns of the summed tensor
                    tma_reduce_add_3d(&tm_y, yw, (hy / xdiv) * xmul + (hy % xmod) * C::P + grp * PC, row0, b);
                else if (grp * PC < pst)   // P = 32: the second group's columns are the next head's
                    tma_store_3d(&tm_y, yw, hy * pst + grp * PC, c * L + 128 * qt + 32 * q, b);
                bulk_commit();
            }
            return true;
        };
        for (int hi = 0; hi < nh && ok; ++hi) {
            const int it = NA + hi, st = it % NS;
            if constexpr (kDot) {
                // Dot mode: this row's dy (this thread's 32 columns of the head, 64
                // bytes) into slot hi & 1, one group per head.  finish(hi), about a
                // head later, reads it; the slot's last reader was this thread's
                // finish(hi - 2), in the previous iteration.
                const int64_t t = (int64_t)c * L + 128 * qt + tl;
                if (t < T) {
                    const __nv_bfloat16* src =
                        dyv + ((int64_t)b * T + t) * ((int64_t)H * C::P) + (int64_t)(h0 + hi) * C::P + grp * PC;
                    uint8_t* dst = sY + (hi & 1) * kSlot + kSlotDy + tl * 128;
#pragma unroll
                    for (int k4 = 0; k4 < PC / 8; ++k4)
                        cp_async16(smem_u32(dst + (((grp * PC / 8 + k4) ^ (tl & 7)) << 4)), src + 8 * k4);
                }
                cp_async_commit();
            }
            // ---- x tile, decay vectors and range decision come from the converters
            // (phase of xready[st]: one per head item of that stage).
            ok = __all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bars.xready[st], (hi / NS) & 1, abort, kWaitNs));
            if (!ok) break;
            const float* ck = cumv + st * 256;
            const float* dk = dtv + st * 256;
            const bool use16 = bars.use16s[st] != 0;
            const float dh = bars.dvals[st];           // D of this head: added to M[t, t]
            // Every load of the row's vectors first, so that their latencies overlap.
            // (ck, dk index keys from kb: the tile's rows are keys tc_ - kb.)
            const float ct = ck[tc_ - kb];
            const float cfirst = ck[32 * jd], clast = ck[32 * jd + 31];
            // Off the diagonal block the decay splits at the warp's first row (causal:
            // keys before it) or last row (anti: keys after it); the diagonal block's
            // packed path takes its last key (causal) or first key (anti).
            const float cr = anti ? clast : cfirst;
            const float cml = anti ? cfirst : clast;
            const float ckd = ck[32 * jd + lane];
            const float dsd = dk[32 * jd + lane];
            constexpr int kMaxOwn = (L / 32 + EG - 1) / EG;   // own blocks off the diagonal
            float cj[kMaxOwn], dj[kMaxOwn];
#pragma unroll
            for (int i = 0; i < kMaxOwn; ++i) {
                const int j = grp + EG * i;
                const bool off = anti ? (j > jd && j < nblk) : j < jd;
                cj[i] = off ? ck[32 * j + lane] : 0.f;
                dj[i] = off ? dk[32 * j + lane] : 0.f;
            }
            // State term's row factor: exp2(cum2_t) (anti: exp2(cum2_last - cum2_t)).
            const float e_t = anti ? ex2(ck[KS - 1] - ct) : ex2(ct);
            const float u_t = anti ? ex2(cr - ct) : ex2(ct - cr);
            float* vq = vdt + q * 256;
            __half* vh = reinterpret_cast<__half*>(vq);
#pragma unroll
            for (int i = 0; i < kMaxOwn; ++i) {
                const int j = grp + EG * i;
                if (anti ? (j > jd && j < nblk) : j < jd) {
                    const float v = (anti ? ex2(cj[i] - cr) : ex2(cr - cj[i])) * dj[i];
                    if (use16) vh[32 * j + lane] = __float2half_rn(v);
                    else vq[32 * j + lane] = v;
                }
            }
            // Diagonal block on the fp16 path, with its last key m as reference:
            // exp2(cum2_t - cum2_s) = u_t w_s, u_t = exp2(cum2_t - cum2_m) in [1, 2^R],
            // w_s = exp2(cum2_m - cum2_s) in [2^-R, 1] (R = the block's cum2 range),
            // then times dt_s.  All three stay normal fp16 numbers when R <= 14 and
            // every dt_s of the block is >= 2^-14; otherwise the fp32 path below.
            // The causal mask is applied to the final product.
            const bool owner = jd % EG == grp;
            const bool dpack = use16 && cfirst - clast <= 14.f &&
                               !__any_sync(0xffffffffu, owner && dsd < 6.1035156e-5f);
            // The block's dt goes to the slot of block jd + 1, outside the causal
            // mask; in anti mode that block is inside it, so to halves 256.., which
            // the packed key factors (halves 0 .. 32 nblk - 1) never use.
            constexpr int kNoSlot = 256;
            const int dslot = anti ? kNoSlot : 32 * jd + 32;
            if (dpack && owner) {
                vh[32 * jd + lane] = __float2half_rn(anti ? ex2(ckd - cml) : ex2(cml - ckd));
                vh[dslot + lane] = __float2half_rn(dsd);
            }
            __syncwarp();
            const __half2 u2 = __float2half2_rn(u_t);
            const __half2 ud2 = __float2half2_rn(anti ? ex2(cml - ct) : ex2(ct - cml));
            const __half2 dd2 = (lane & 1) ? __floats2half2_rn(0.f, dh) : __floats2half2_rn(dh, 0.f);

            // ---- M, in two K-halves.
            for (int half = 0; half < 2 && ok; ++half) {
                // The half's M columns are free once the previous head's GEMM2 half completed.
                if (hi > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.mm_free[half], (hi - 1) & 1,
                                                                    abort, kWaitNs));
                    if (!ok) break;
                    tc_fence_after();
                }
                const int jlo = max(half * hblkn, jmin), jhi = min(jmax, half * hblkn + hblkn - 1);
                int j = jlo + ((grp - jlo) % EG + EG) % EG;    // first own in-mask block >= jlo
                uint32_t r[16];
                if (j <= jhi) tmem_ld16(tmem + lane_off + COL_CB + 16 * j, r);
                for (; j <= jhi; j += EG) {
                    tmem_wait_ld_regs(r);
                    uint32_t m[16];
                    if (j != jd && use16) {
                        const uint4* v4 = reinterpret_cast<const uint4*>(vh + 32 * j);
#pragma unroll
                        for (int e8 = 0; e8 < 4; ++e8) {
                            const uint4 vv = v4[e8];
                            const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                            for (int k2 = 0; k2 < 4; ++k2) {
                                const __half2 cb2 = *reinterpret_cast<const __half2*>(&r[4 * e8 + k2]);
                                const __half2 uv = __hmul2(u2, *reinterpret_cast<const __half2*>(&vw[k2]));
                                const __half2 mm2 = __hmul2(cb2, uv);
                                m[4 * e8 + k2] = *reinterpret_cast<const uint32_t*>(&mm2);
                            }
                        }
                        if (j + EG <= jhi) tmem_ld16(tmem + lane_off + COL_CB + 16 * (j + EG), r);
                    } else if (j == jd && dpack) {
                        const uint4* w4 = reinterpret_cast<const uint4*>(vh + 32 * j);
                        const uint4* d4 = reinterpret_cast<const uint4*>(vh + dslot);
#pragma unroll
                        for (int e8 = 0; e8 < 4; ++e8) {
                            const uint4 ww = w4[e8], dd = d4[e8];
                            const uint32_t wv[4] = {ww.x, ww.y, ww.z, ww.w};
                            const uint32_t dv[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                            for (int k2 = 0; k2 < 4; ++k2) {
                                const int e = 4 * e8 + k2;          // keys 2e, 2e+1 of the block
                                const __half2 cb2 = *reinterpret_cast<const __half2*>(&r[e]);
                                const __half2 uw = __hmul2(ud2, *reinterpret_cast<const __half2*>(&wv[k2]));
                                const __half2 cd = __hmul2(cb2, *reinterpret_cast<const __half2*>(&dv[k2]));
                                __half2 mm2 = __hmul2(cd, uw);
                                if (e == (lane >> 1)) mm2 = __hadd2(mm2, dd2);   // key t: + D
                                const uint32_t mw = *reinterpret_cast<const uint32_t*>(&mm2);
                                // keys 2e (low half) and 2e + 1 against row lane
                                m[e] = anti ? (2 * e >= lane ? mw : (2 * e + 1 >= lane ? (mw & 0xffff0000u) : 0u))
                                            : (2 * e + 1 <= lane ? mw : (2 * e <= lane ? (mw & 0xffffu) : 0u));
                            }
                        }
                        if (j + EG <= jhi) tmem_ld16(tmem + lane_off + COL_CB + 16 * (j + EG), r);
                    } else {
                        float cbv[32];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (cb16) {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r[e]));
                                cbv[2 * e] = f.x;
                                cbv[2 * e + 1] = f.y;
                            } else {
                                cbv[2 * e] = __uint_as_float(r[e] << 16);
                                cbv[2 * e + 1] = __uint_as_float(r[e] & 0xffff0000u);
                            }
                        }
                        float mv[32];
                        if (j != jd) {
                            const float4* v4 = reinterpret_cast<const float4*>(vq + 32 * j);
#pragma unroll
                            for (int e4 = 0; e4 < 8; ++e4) {
                                const float4 v = v4[e4];
                                mv[4 * e4 + 0] = cbv[4 * e4 + 0] * (u_t * v.x);
                                mv[4 * e4 + 1] = cbv[4 * e4 + 1] * (u_t * v.y);
                                mv[4 * e4 + 2] = cbv[4 * e4 + 2] * (u_t * v.z);
                                mv[4 * e4 + 3] = cbv[4 * e4 + 3] * (u_t * v.w);
                            }
                        } else {
                            const float4* c4 = reinterpret_cast<const float4*>(ck + 32 * j);
                            const float4* d4 = reinterpret_cast<const float4*>(dk + 32 * j);
#pragma unroll
                            for (int e4 = 0; e4 < 8; ++e4) {
                                const float4 cv = c4[e4], dv = d4[e4];
                                const float cs[4] = {cv.x, cv.y, cv.z, cv.w};
                                const float ds[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int e = 4 * e4 + u;   // key 32 j + e, row 32 j + lane
                                    mv[e] = anti ? (e >= lane ? cbv[e] * ex2(cs[u] - ct) * ds[u] : 0.f)
                                                 : (e <= lane ? cbv[e] * ex2(ct - cs[u]) * ds[u] : 0.f);
                                    if (e == lane) mv[e] += dh;          // key t: + D
                                }
                            }
                        }
                        if (j + EG <= jhi) tmem_ld16(tmem + lane_off + COL_CB + 16 * (j + EG), r);
                        if (use16) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) m[e] = pack_f16x2(mv[2 * e], mv[2 * e + 1]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) m[e] = pack_bf16x2(mv[2 * e], mv[2 * e + 1]);
                        }
                    }
                    tmem_st16(tmem + lane_off + COL_MM + 16 * j, m);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars.mm_ready[half]);
            }
            if (!ok) break;
            // ---- previous head's output while the tensor core works on this one.
            if (hi > 0 && !(ok = finish(hi - 1))) break;
            e_prev = e_t;
        }
        if (ok && nh > 0) ok = finish(nh - 1);
        if constexpr (kDot) cp_async_wait<0>();   // none of this thread's copies outlive it
        if (lane == 0) bulk_wait<0>();
    }
    else {
        // ----------------------------------------------------------- converters
        // Per head: decay vectors of the chunk into the stage's vector buffers,
        // the range check (max |x| over the x tile, max dt) and, when fp16 cannot
        // overflow, the x tile converted to fp16 in place.  They run ahead of the
        // epilogue warps, which then only build M and write y.
        const int ctid = threadIdx.x;                  // 0 .. kConvThreads-1
        const int cw = ctid >> 5;
        uint32_t sync_phase = 0;
        auto conv_sync = [&]() -> bool {
            mbar_arrive(&bars.conv_sync);
            const bool r = mbar_wait_or_abort(&bars.conv_sync, sync_phase, abort, kWaitNs);
            sync_phase ^= 1u;
            return __all_sync(0xffffffffu, r);
        };
        const int64_t row0 = (int64_t)b * (H >> pts) * T + (int64_t)c * L;  // chunk c of batch b
        constexpr int KPT = L / kConvThreads;                  // keys per thread (at most)
        float pc[KPT], pd[KPT], plast = 0.f, pD = 0.f;
#pragma unroll
        for (int i = 0; i < KPT; ++i) { pc[i] = 0.f; pd[i] = 0.f; }
        uint4 pX = make_uint4(0u, 0u, 0u, 0u), pX2 = pX;
        auto prefetch = [&](int hh) {
            const float* crow = cum2 + row0 + (int64_t)((h0 + hh) >> pts) * T;   // the head's rows
            const float* drow = dtT + row0 + (int64_t)((h0 + hh) >> pts) * T;
            plast = __ldg(crow + Lc - 1);
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                const int s = ctid + kConvThreads * i;   // key kb + s of the chunk
                if (s < KS && kb + s < Lc) {
                    pc[i] = __ldg(crow + kb + s);
                    pd[i] = (kY32 && dt1) ? 1.f : __ldg(drow + kb + s);
                }
            }
            pD = Dvec ? __ldg(Dvec + ((h0 + hh) >> pts)) : 0.f;
            if (xabs) {   // stage 2's max |x| of the chunk (eight words, bf16 bits)
                const uint4* xw = reinterpret_cast<const uint4*>(xabs) + 2 * (((int64_t)b * nc + c) * H + h0 + hh);
                pX = __ldg(xw);
                pX2 = __ldg(xw + 1);
            }
        };
        if (nh > 0) prefetch(0);
        // The C.B^T bound comes from the epilogue (after GEMM1); by then every
        // C.B^T block item of the ring has landed, so only head items remain.
        bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.cbinfo, 0, abort, kWaitNs));
        const float cbmax = bars.cbmax;        // C.B^T packed as fp16 iff cb_fits_f16(cbmax)
        for (int hi = 0; hi < nh && ok; ++hi) {
            const int it = NA + hi, st = it % NS, k = it / NS;
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.full[st], k & 1, abort, kWaitNs));
            if (!ok) break;
            float* ck = cumv + st * 256;
            float* dk = dtv + st * 256;
            float dloc = 0.f;
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                const int s = ctid + kConvThreads * i;
                if (s < KS) {
                    const bool in = kb + s < Lc;
                    ck[s] = in ? pc[i] : plast;
                    dk[s] = in ? pd[i] : 0.f;
                    if (in) dloc = fmaxf(dloc, pd[i]);
                }
            }
            const float dval = pD;
            const uint32_t xknown = max(max(max(pX.x, pX.y), max(pX.z, pX.w)),
                                        max(max(pX2.x, pX2.y), max(pX2.z, pX2.w)));
            if (hi + 1 < nh) prefetch(hi + 1);
            uint8_t* xs = sStage + st * C::STAGE;
            const int nch = KS * 8 / kConvThreads;
            __nv_bfloat162 xm2 = __floats2bfloat162_rn(0.f, 0.f);
            // max |x| over the tile: from stage 2 (over the whole chunk, a bound)
            // when available, else one pass over the tile.
#pragma unroll 8
            for (int i = 0; i < (xabs ? 0 : nch); ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(xs + (ctid + kConvThreads * i) * 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t a = w4[e] & 0x7fff7fffu;   // |x|, two at a time
                    xm2 = __hmax2(xm2, *reinterpret_cast<const __nv_bfloat162*>(&a));
                }
            }
            const uint32_t xm2u = *reinterpret_cast<const uint32_t*>(&xm2);
            const uint32_t xmax = __reduce_max_sync(0xffffffffu, max(xm2u & 0xffffu, xm2u >> 16));
            const uint32_t dmax = __reduce_max_sync(0xffffffffu, __float_as_uint(dloc));
            if (lane == 0) {
                red_x[(st * kConvWarps + cw) * 2 + 0] = xmax;
                red_x[(st * kConvWarps + cw) * 2 + 1] = dmax;
            }
            if (!(ok = conv_sync())) break;
            const uint32_t gx = xabs ? xknown : __reduce_max_sync(
                0xffffffffu, lane < kConvWarps ? red_x[(st * kConvWarps + lane) * 2 + 0] : 0u);
            const uint32_t gd = __reduce_max_sync(
                0xffffffffu, lane < kConvWarps ? red_x[(st * kConvWarps + lane) * 2 + 1] : 0u);
            // fp16 for the head when fp16 holds x and M without overflow and
            // without their significant entries or factors falling to fp16
            // subnormals: C.B^T packed as fp16, max|x| in [2^-6, 2^15], the bound
            // max|C.B| max(dt) + |D| of |M| in [2^-4, 2^15], max dt >= 2^-10.
            const float mb = cbmax * __uint_as_float(gd) + fabsf(dval);
            const bool use16 = cb_fits_f16(cbmax) && gx >= kF16MinX && gx <= kF16MaxX &&
                               mb <= 32768.f && mb >= 0.0625f && __uint_as_float(gd) >= 0.0009765625f;
            if (use16) {
#pragma unroll 8
                for (int i = 0; i < nch; ++i) {
                    uint4* p = reinterpret_cast<uint4*>(xs + (ctid + kConvThreads * i) * 16);
                    const uint4 v = *p;
                    *p = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                    bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
                }
            }
            // The tile's generic-proxy accesses (the range check's reads, the fp16
            // rewrite) before the async proxy's: GEMM2 reads it, the next TMA load
            // into this stage overwrites it.
            fence_proxy_async_smem();
            if (ctid == 0) {
                bars.use16s[st] = use16 ? 1 : 0;
                bars.dvals[st] = dval;
            }
            mbar_arrive(&bars.xready[st]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && bars.abort) record_error(err, kErrTimeoutK4);
}

// Head blocks per CTA.  One CTA per SM at a time, each with a fixed cost (the
// C.B^T product and its packing, the pipeline's fill and drain) of about two
// heads; the second query tile costs about 1.25 times the first per head.  The
// grid is cut in two regions: the first n1 CTAs take blocks of v1 heads (the
// first (b, c) pairs), the rest blocks of v2 heads, both dividing H/G.  The
// choice minimises the makespan of a simulation of greedy CTA scheduling over
// the SMs: single sizes, and mixes whose first region fills whole waves.  At
// b8 T4096 H80 it takes 40 heads for 114 of the 128 (b, c) pairs and 16 for the
// rest (1 024 CTAs of 20 heads simulate to 179 head units, the mix to 168).

double makespan4(int64_t bc, int64_t n1_bc, int v1, int v2, int64_t H, int NQ, int sms) {
    std::priority_queue<double, std::vector<double>, std::greater<double>> q;
    for (int i = 0; i < sms; ++i) q.push(0.0);
    double mk = 0.0;
    auto run = [&](int64_t nbc, int v) {
        for (int64_t i = 0; i < nbc * (H / v); ++i)
            for (int qt = NQ - 1; qt >= 0; --qt) {
                const double t = q.top() + v * (qt ? 1.25 : 1.0) + 2.0;
                q.pop();
                q.push(t);
                mk = std::max(mk, t);
            }
    };
    run(n1_bc, v1);
    run(bc - n1_bc, v2);
    return mk;
}

Split4 pick_split4(const Dims& d, int NQ) {
    static std::mutex mu;
    static std::map<std::array<int64_t, 5>, Split4> cache;
    const int sms = sm_count();
    const std::array<int64_t, 5> key = {d.b * d.nc, d.H, d.G, NQ, sms};
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int64_t bc = d.b * d.nc, hpg = d.H / d.G, cap = 32LL * sms;   // CTAs simulated at most
    std::vector<int> divs;
    for (int64_t v = 1; v <= hpg; ++v)
        if (hpg % v == 0 && bc * NQ * (d.H / v) <= cap) divs.push_back((int)v);
    if (divs.empty()) divs.push_back((int)hpg);
    Split4 best{divs.back(), divs.back(), bc * NQ * (d.H / divs.back()), bc * NQ * (d.H / divs.back()), bc,
                kFromModel};
    double best_t = -1.0;
    auto consider = [&](int64_t n1_bc, int v1, int v2) {
        const double t = makespan4(bc, n1_bc, v1, v2, d.H, NQ, sms);
        const int64_t n1 = n1_bc * NQ * (d.H / v1), ctas = n1 + (bc - n1_bc) * NQ * (d.H / v2);
        if (best_t < 0.0 || t < best_t * 0.999 || (t <= best_t * 1.001 && ctas < best.ctas)) {
            best_t = t;
            best = {v1, v2, n1, ctas, n1_bc, kFromModel};
        }
    };
    int vsingle = divs.front();
    double tsingle = -1.0;
    for (int v : divs) {
        const double t = makespan4(bc, bc, v, v, d.H, NQ, sms);
        if (tsingle < 0.0 || t <= tsingle) { tsingle = t; vsingle = v; }
        consider(bc, v, v);
    }
    for (int v1 : divs) {
        if (v1 < vsingle) continue;
        const int64_t per_bc = NQ * (d.H / v1);
        for (int64_t k = 1; k <= 32; ++k) {
            const int64_t n1_bc = k * sms / per_bc;
            if (n1_bc <= 0) continue;
            if (n1_bc >= bc) break;
            for (int v2 : divs)
                if (v2 < v1) consider(n1_bc, v1, v2);
        }
    }
    cache[key] = best;
    return best;
}

template <int L, int NA, bool kY32, bool kDot = false, bool kAnti = false>
cudaError_t launch_k4(const Dims& d, const void* x, const void* B, const void* Cm,
                      const float* cum2, const float* dtT, const void* Sprev, const float* D,
                      void* y, int32_t* err, cudaStream_t st, const uint32_t* xabs, bool pdl) {
    using C = K4Cfg<L, NA, kY32, kDot>;
    if constexpr (C::SMEM > 232448) {   // the fp32 y staging does not fit (L = 256, N = 256)
        return cudaErrorNotSupported;
    } else {
    CUtensorMap tm_x, tm_b, tm_c, tm_s, tm_y, tm_dxx, tm_ddy;
    const uint64_t xd[3] = {(uint64_t)(d.H * d.P), (uint64_t)d.T, (uint64_t)d.b};     // y
    const uint64_t xin[3] = {(uint64_t)(d.xcols ? d.xcols : d.H * d.P), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t xs[2] = {(uint64_t)(d.sx[1] * 2), (uint64_t)(d.sx[0] * 2)};   // token, batch
    constexpr uint64_t ye = kY32 ? 4 : 2;   // bytes per y element
    const uint64_t ys[2] = {(uint64_t)(d.sy[1] * ye), (uint64_t)(d.sy[0] * ye)};
    const uint32_t box[3] = {64, 128, 1};
    const uint32_t ybox[3] = {32, 32, 1};
    const uint64_t bd[3] = {(uint64_t)(d.G * d.N), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t bs[2] = {(uint64_t)(d.sB[1] * 2), (uint64_t)(d.sB[0] * 2)};
    const uint64_t cs[2] = {(uint64_t)(d.sC[1] * 2), (uint64_t)(d.sC[0] * 2)};
    // state rows of 64 x 64 tiles: [(b, c, h, p)][n], or untransposed (st_mn)
    const uint64_t scols = d.st_mn ? (uint64_t)(d.xmod * 64) : (uint64_t)d.N;
    const uint64_t srows = d.st_mn ? (uint64_t)(d.b * d.nc * (d.H / d.xmod) * d.N) : (uint64_t)(d.b * d.nc * d.H * d.P);
    const uint64_t sd[2] = {scols, srows};
    const uint64_t ss[1] = {scols * 2};
    const uint32_t sbox[2] = {64, 64};
    if (!make_tmap_bf16(&tm_x, x, 3, xin, xs, box) || !make_tmap_bf16(&tm_b, B, 3, bd, bs, box) ||
        !make_tmap_bf16(&tm_c, Cm, 3, bd, cs, box) || !make_tmap_bf16(&tm_s, Sprev, 2, sd, ss, sbox) ||
        !(kY32 ? make_tmap(&tm_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y, 3, d.yred ? xin : xd, ys, ybox,
                           CU_TENSOR_MAP_SWIZZLE_128B)
               : make_tmap_bf16(&tm_y, y, 3, xd, ys, ybox, CU_TENSOR_MAP_SWIZZLE_64B)))
        return cudaErrorInvalidValue;
    // dx / dot mode: x and dy rows (contiguous [b, T, H, 64] bf16) staged in the two
    // y buffers; dx mode is the anti-causal variant's, dot mode the dot variant's.
    if ((d.dxm_dx || d.ydot_dy) &&
        (!kY32 || (d.ydot_dy && !kDot) || (d.dxm_dx && !kAnti) ||
         C::YB * C::Y_BYTES < 2 * (kDot ? 16384 : 32768)))
        return cudaErrorNotSupported;
    if ((kAnti && !d.dxm_dx) || (kDot && !d.ydot_dy)) return cudaErrorNotSupported;
    if (d.dxm_dx) {   // dx mode: the producer's TMA tiles (dot mode's rows are per-thread copies)
        const uint64_t dd[3] = {(uint64_t)(d.H * 64), (uint64_t)d.T, (uint64_t)d.b};
        const uint64_t ds[2] = {(uint64_t)(d.H * 64 * 2), (uint64_t)(d.T * d.H * 64 * 2)};
        if (!make_tmap_bf16(&tm_dxx, d.dxm_x, 3, dd, ds, box) || !make_tmap_bf16(&tm_ddy, d.dxm_dy, 3, dd, ds, box))
            return cudaErrorInvalidValue;
    } else {
        tm_dxx = tm_x;   // unused
        tm_ddy = tm_x;
    }
    const Split4 sp = k4_split(d);
    const int64_t grid = sp.ctas;
    auto k = chunk_out_tc_kernel<L, NA, kY32, kDot, kAnti>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, dim3((unsigned)grid), dim3(kThreads), C::SMEM, st, pdl, tm_x, tm_b, tm_c,
                         tm_s, tm_y, tm_dxx, tm_ddy, cum2, dtT, D, xabs, (int)d.T, (int)d.H, (int)d.G, (int)d.nc,
                         sp.v1, (int)sp.n1, sp.v2, d.pts, (int)d.P, d.xdiv, (int)(d.xmul ? d.xmul : d.P), d.xmod,
                         d.yred, d.st_mn, d.dt1, static_cast<const __nv_bfloat16*>(d.ydot_dy), d.ydot_out,
                         d.yrev, static_cast<float*>(y), (int)(d.xcols ? d.xcols : d.H * d.P),
                         DxArgs{d.dxm_x, d.dxm_dy, d.dxm_dt, d.dxm_D, d.dxm_dx, d.dxm_xy, d.dxm_dyx}, err);
    }
}

template <int L, bool kY32>
cudaError_t launch_k4_n(const Dims& d, const void* x, const void* B, const void* Cm,
                        const float* cum2, const float* dtT, const void* Sprev, const float* D,
                        void* y, int32_t* err, cudaStream_t st, const uint32_t* xabs, bool pdl) {
    switch (d.N) {
        case 64:
            if constexpr (kY32) {
                if (d.ydot_dy) return launch_k4<L, 1, true, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
                if (d.antic) return launch_k4<L, 1, true, false, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
            }
            return launch_k4<L, 1, kY32>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
        case 128:
            if constexpr (kY32) {
                if (d.ydot_dy) return launch_k4<L, 2, true, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
                if (d.antic) return launch_k4<L, 2, true, false, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
            }
            return launch_k4<L, 2, kY32>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
        case 256:
            if constexpr (kY32) {
                if (d.ydot_dy) return launch_k4<L, 4, true, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
                if (d.antic) return launch_k4<L, 4, true, false, true>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
            }
            return launch_k4<L, 4, kY32>(d, x, B, Cm, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
    }
    return cudaErrorInvalidValue;
}

template <int L, int NA>
constexpr bool dx_fits() {
    using C = K4Cfg<L, NA, true>;
    return C::SMEM <= 232448 && C::YB * C::Y_BYTES >= 65536;
}

}  // namespace

bool k4_dx_fits(const Dims& dq) {
    const Dims d = tc_view(dq);
    const int64_t na = d.N / 64;
    if (d.L == 256) return na == 1 ? dx_fits<256, 1>() : na == 2 ? dx_fits<256, 2>() : na == 4 && dx_fits<256, 4>();
    if (d.L == 128) return na == 1 ? dx_fits<128, 1>() : na == 2 ? dx_fits<128, 2>() : na == 4 && dx_fits<128, 4>();
    return false;
}

// A forced or tabled split: v1 and v2 divide H/G, and the v1 region takes the
// (b, c) pairs that fill `waves` waves of the SMs (all pairs when waves is 0).
bool fixed_split4(const Dims& d, int v1, int v2, int waves, int src, Split4* out) {
    const int64_t hpg = d.H / d.G, bc = d.b * d.nc, NQ = d.L / 128;
    if (v1 <= 0 || hpg % v1) return false;
    if (waves > 0 && (v2 <= 0 || hpg % v2)) return false;
    int64_t n1_bc = bc;
    if (waves > 0) n1_bc = std::min<int64_t>(bc, (int64_t)waves * sm_count() / (NQ * (d.H / v1)));
    if (n1_bc == bc) v2 = v1;
    const int64_t n1 = n1_bc * NQ * (d.H / v1);
    *out = {v1, v2, n1, n1 + (bc - n1_bc) * NQ * (d.H / v2), n1_bc, src};
    return true;
}

Split4 k4_split(const Dims& d) {
    if (d.H == 0 || d.b * d.nc == 0) return {1, 1, 0, 0, 0, kFromModel};   // nothing to launch
    Split4 sp;
    const int o1 = tile_override(1);
    if (fixed_split4(d, o1, tile_override(2), tile_override(3), kFromOverride, &sp)) return sp;
    const TileChoice* t = o1 < 0 ? nullptr : find_tile(d);   // -1: the cost model only
    if (t && fixed_split4(d, t->k4_v1, t->k4_v2, t->k4_waves1, kFromTable, &sp)) return sp;
    return pick_split4(d, (int)(d.L / 128));
}

cudaError_t launch_chunk_out_tc(const Dims& dq, const void* x, const void* B, const void* C,
                                const float* cum2, const float* dtT, const void* Sprev,
                                const float* D, void* y, int32_t* err, cudaStream_t st,
                                const uint32_t* xabs, bool pdl, bool y32) {
    const Dims d = tc_view(dq);
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    if (!tc_supported(d)) return cudaErrorInvalidValue;
    if (y32)
        return d.L == 256 ? launch_k4_n<256, true>(d, x, B, C, cum2, dtT, Sprev, D, y, err, st, xabs, pdl)
                          : launch_k4_n<128, true>(d, x, B, C, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
    return d.L == 256 ? launch_k4_n<256, false>(d, x, B, C, cum2, dtT, Sprev, D, y, err, st, xabs, pdl)
                      : launch_k4_n<128, false>(d, x, B, C, cum2, dtT, Sprev, D, y, err, st, xabs, pdl);
}

}  // namespace m2
