// bwd_bc_tc.cu -- the backward's dC and dB on tcgen05 tensor cores, summed over
// each group's heads inside the kernel.
//
// The pages give no backward method ("NVIDIA、cuTileでMamba-2フォワードパスを高速化"
// (ai.newsbites.today), "開発現場への影響と未確認事項"): these are the chain rule
// applied to the chunked forward of "Accelerating Mamba-2 with High-Performance
// Forward Pass Kernels in NVIDIA CUDA Tile" (brifing.si), sections 4, 5 and 9,
// for one chunk (chunk-local tokens, c2 the log2-space decay cumsum, c2_last its
// last entry, Sprev the state entering the chunk, Gn the adjoint of the state
// leaving it), summed over the heads h of group g:
//
//   dC_t[n] = sum_h [ sum_{s<=t} (dy_t.x_s) 2^(c2_t - c2_s) dt_s B_s[n]
//                     + 2^(c2_t) sum_p dy_t[p] Sprev[p,n] ]
//   dB_s[n] = sum_h [ sum_{t>=s} (x_s.dy_t) 2^(c2_t - c2_s) dt_s C_t[n]
//                     + dt_s 2^(c2_last - c2_s) sum_p x_s[p] Gn[p,n] ]
//
// Both have one shape: rows r, keys k, a row operand Q, a key operand K, an
// output operand O shared by the group's heads and a per-head state S:
//   out_r = sum_h [ sum_k W_h[r,k] O_k + f_r (Q_r . S_h) ]
//   W_h[r,k] = (Q_r . K_k) 2^-|c2_r - c2_k| times dt of the earlier token,
// causal (k <= r) for dC with (Q, K, O, S) = (dy, x, B, Sprev) and f = 2^c2,
// anti-causal (k >= r) for dB with (Q, K, O, S) = (x, dy, C, Gn) and
// f = dt 2^(c2_last - c2).  Because O does not depend on the head, the head sum
// happens in the accumulator: one CTA takes a 128-row tile of one (b, chunk)
// and a block of heads of one group, and per head issues
//   GEMM1  D1 = Q_h . K_h^T          (tensor memory, fp32, two key halves)
//   GEMM2  acc += W_h . O            (W_h built from D1 by the epilogue warps)
//   GEMM3  acc += (f . Q_h) . S_h    (Q_h rescaled in place by the converters)
// and only at the end adds its 128 x NO accumulator into dC or dB with TMA
// reduce-add copies (several head blocks of one group add into the same rows).
//
// W is built as in the forward's output kernel (section 11 "Causal Masking and
// Stability"): the mask comes from the indices, and outside the warp's diagonal
// 32 x 32 block the decay splits at the warp's first row (causal) or last row
// (anti-causal) into two factors that are both at most 1; the diagonal block
// masks the exponent before exp2.  W, f . Q and the operands are bf16, the
// accumulation fp32.
//
// Tensor memory (512 columns): D1 in [0, 256) (key k at column k), W as bf16
// pairs in [256, 384) (the MMA's A operand), the accumulator in [384, 384 + NO).
// Warp roles: 0, 1 converters (decay vectors, f . Q), 2 TMA producer, 3 MMA
// issuer (and tensor-memory owner), 4 .. 11 epilogue (lane quadrant warp % 4,
// column group (warp - 4) / 4).  Every wait is bounded: on a timeout the CTA
// raises its abort flag, drains what is in flight and returns with an error bit.
#include "common.cuh"
#include "internal.h"
#include "tc5.cuh"
#include "tmap.h"

namespace m2 {
namespace {

using namespace tc;

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kConvThreads = 64;                        // warps 0, 1
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kConvThreads + kEpiThreads;
constexpr int kWarpProd = 2, kWarpMma = 3, kEpiWarp0 = 4;
constexpr uint32_t COL_D1 = 0, COL_W = 256, COL_ACC = 384;

template <int L, int NO>   // NO: output columns per CTA (64 or 128)
struct BCCfg {
    static constexpr int Q_BYTES = 128 * 128;            // 128 rows x 64 p, K-major
    static constexpr int K_BYTES = L * 128;              // up to L keys x 64 p, K-major
    static constexpr int S_BYTES = (NO / 64) * 8192;     // 64 p rows x NO n, MN-major blocks
    static constexpr int STAGE = Q_BYTES + K_BYTES + S_BYTES;
    static constexpr int O_BLK = L * 128;                // one 64-column block of O
    static constexpr int O_BYTES = (NO / 64) * O_BLK;
    static constexpr int VEC_BYTES = (2 * 3 * 256 + 4 * 256) * 4;   // c2, dt per stage; key factors
    static constexpr int budget(int ns) { return 1024 + O_BYTES + ns * STAGE + VEC_BYTES; }
    static constexpr int NS = budget(3) <= 225 * 1024 ? 3 : 2;
    static constexpr int SMEM = budget(NS);
    static_assert(NS * STAGE >= kEpiWarps * (NO / 64) * 4096, "the drain's staging fits the stages");
};

struct BCBars {
    uint64_t full[3], xfree[3];     // stage landed / stage free (after GEMM3)
    uint64_t vready[3];             // decay vectors of the stage's head written
    uint64_t g1done[3];             // GEMM1 of the stage's head complete (Q may be rescaled)
    uint64_t qready[3];             // f . Q written
    uint64_t o_full;
    uint64_t d1_full[2];            // per key half: D1 written
    uint64_t w_ready[2], w_free[2]; // per key half: W built / W read by GEMM2 (and D1 free)
    uint64_t acc_full;
    uint64_t drain;                 // commit target used to drain in-flight MMAs on abort
    uint32_t tmem_base;
    int abort;
};

// Eight bf16 (one 16-byte chunk) times f, rounded to bf16.
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float f) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(f * __uint_as_float(w[e] << 16), f * __uint_as_float(w[e] & 0xffff0000u));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int L, int NO, bool kRev>
__global__ void __launch_bounds__(kThreads, 1)
bwd_bc_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_s,
                 const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ cum2,
                 const float* __restrict__ dtT, int T, int H, int G, int N, int nc, int hpc,
                 int32_t* err) {
    using C = BCCfg<L, NO>;
    constexpr int NS = C::NS, NQ = L / 128, NB = NO / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sO = smem;
    uint8_t* sStage = sO + C::O_BYTES;
    float* cv = reinterpret_cast<float*>(sStage + NS * C::STAGE);   // [stage][256] c2
    float* dv = cv + 3 * 256;                                        // [stage][256] dt
    float* vqa = dv + 3 * 256;                                       // [quadrant][256] key factors
    __shared__ BCBars bars;
    volatile int* abort = &bars.abort;

    // Work item: (b, c) outer, then group, head block, query tile (heaviest
    // first: the tiles of one head block share Q, K and S through L2), column block.
    const int ncb = N / NO, hpg = H / G, nhb = hpg / hpc;
    int rest = blockIdx.x;
    const int cb = rest % ncb; rest /= ncb;
    const int qi = rest % NQ; rest /= NQ;
    const int hb = rest % nhb; rest /= nhb;
    const int g = rest % G; rest /= G;
    const int c = rest % nc;
    const int b = rest / nc;
    const int qt = kRev ? qi : NQ - 1 - qi;
    const int h0 = g * hpg + hb * hpc, nh = hpc;
    const int Lc = min(L, T - c * L);
    if (128 * qt >= Lc) return;                   // tile entirely past the end of the sequence
    const int kb = kRev ? 128 * qt : 0;           // first key of the tile
    const int KS = kRev ? L - 128 * qt : 128 * (qt + 1);
    const int kh = KS / 2;                        // keys per half
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.xfree[i], 1);
            mbar_init(&bars.vready[i], kConvThreads);
            mbar_init(&bars.g1done[i], 1);
            mbar_init(&bars.qready[i], kConvThreads);
        }
        mbar_init(&bars.o_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.d1_full[i], 1);
            mbar_init(&bars.w_ready[i], kEpiThreads);
            mbar_init(&bars.w_free[i], 1);
        }
        mbar_init(&bars.acc_full, 1);
        mbar_init(&bars.drain, 1);
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
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_o);
            prefetch_tmap(&tm_s);
            prefetch_tmap(&tm_out);
            const int ocol = g * N + cb * NO;
            mbar_arrive_expect_tx(&bars.o_full, NB * KS * 128);
            for (int blk = 0; blk < NB; ++blk)
                for (int r = 0; r < KS / 128; ++r)
                    tma_load_3d(sO + blk * C::O_BLK + r * 16384, &tm_o, &bars.o_full, ocol + 64 * blk,
                                c * L + kb + 128 * r, b);
            auto srow = [&](int h) { return (int)((((int64_t)b * nc + c) * H + h) * 64); };
            // The ring is shallow (two stages of 64 KB at L = 256): each head's tiles
            // are prefetched into L2 when the head NS places earlier is loaded, so
            // that its own loads, issued once a stage frees, find them there.
            auto prefetch = [&](int hi) {
                const int h = h0 + hi;
                tma_prefetch_3d(&tm_q, h * 64, c * L + 128 * qt, b);
                for (int r = 0; r < KS / 128; ++r) tma_prefetch_3d(&tm_k, h * 64, c * L + kb + 128 * r, b);
                for (int blk = 0; blk < NB; ++blk) tma_prefetch_2d(&tm_s, cb * NO + 64 * blk, srow(h));
            };
            int issued = 0;
            for (int hi = 0; hi < nh; ++hi) {
                const int st = hi % NS, k = hi / NS, h = h0 + hi;
                if (!mbar_wait_or_abort(&bars.xfree[st], (k & 1) ^ 1, abort, kWaitNs)) break;
                uint8_t* sq = sStage + st * C::STAGE;
                mbar_arrive_expect_tx(&bars.full[st], C::Q_BYTES + KS * 128 + C::S_BYTES);
                tma_load_3d(sq, &tm_q, &bars.full[st], h * 64, c * L + 128 * qt, b);
                for (int r = 0; r < KS / 128; ++r)
                    tma_load_3d(sq + C::Q_BYTES + r * 16384, &tm_k, &bars.full[st], h * 64,
                                c * L + kb + 128 * r, b);
                for (int blk = 0; blk < NB; ++blk)
                    tma_load_2d(sq + C::Q_BYTES + C::K_BYTES + blk * 8192, &tm_s, &bars.full[st],
                                cb * NO + 64 * blk, srow(h));
                if (hi + NS < nh) prefetch(hi + NS);
                issued = hi + 1;
            }
            if (*abort) {   // let every copy already issued land before the CTA exits
                mbar_wait(&bars.o_full, 0, kWaitNs);
                for (int it = issued - 1; it >= 0 && it >= issued - NS; --it)
                    mbar_wait(&bars.full[it % NS], (it / NS) & 1, kWaitNs);
            }
        }
    } else if (warp == kWarpMma) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            // GEMM2 and GEMM3: one MMA over all NO output columns; B is MN-major in
            // 64-column blocks LBO bytes apart (O: O_BLK, S: 8192).
            constexpr uint32_t id_out = idesc_bf16_f32(128, NO, 0, 1);
            const uint32_t id_g1 = idesc_bf16_f32(128, kh, 0, 0);        // both K-major
            const uint32_t st0 = smem_u32(sStage);
            // Descriptors formed once; each MMA adds a constant offset / 16.
            const uint64_t q_desc0 = smem_desc_sw128(st0, 16, 1024);
            const uint64_t k_desc0 = smem_desc_sw128(st0 + C::Q_BYTES, 16, 1024);
            const uint64_t s_desc0 = smem_desc_sw128(st0 + C::Q_BYTES + C::K_BYTES, 8192, 1024);
            const uint64_t o_desc0 = smem_desc_sw128(smem_u32(sO), C::O_BLK, 1024);
            constexpr uint64_t kStageD = C::STAGE >> 4;
            // GEMM1 of head hi, key half `half`: D1[:, half keys] = Q . K^T.
            auto gemm1 = [&](int hi, int half) {
                const int st = hi % NS;
                const uint64_t qd = q_desc0 + (uint64_t)st * kStageD;
                const uint64_t kd = k_desc0 + (uint64_t)st * kStageD + (uint64_t)((half * kh * 128) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + COL_D1 + half * kh, qd + 2 * kk, kd + 2 * kk, id_g1, kk > 0 ? 1u : 0u);
                mma_commit(&bars.d1_full[half]);
            };
            bool ok = nh > 0 && mbar_wait_or_abort(&bars.full[0], 0, abort, kWaitNs);
            if (ok) {
                tc_fence_after();
                gemm1(0, 0);
                gemm1(0, 1);
                mma_commit(&bars.g1done[0]);
                ok = mbar_wait_or_abort(&bars.o_full, 0, abort, kWaitNs);
                tc_fence_after();
            }
            // Per head: GEMM2 of each key half as soon as its W is built, then
            // GEMM3 once the converters rescaled Q (freeing the head's stage).  The
            // next head's GEMM1 goes in between, half by half (its D1 columns are
            // free once W is built), when its tiles have already landed; otherwise
            // after GEMM3, so that waiting for them never holds up this head.
            auto gemm2 = [&](int hi, int half) {
                const int s0 = half * (kh / 16);   // first 16-key step of the half
                for (int kk = 0; kk < kh / 16; ++kk)
                    mma_ts(tmem + COL_ACC, tmem + COL_W + 8 * (s0 + kk),
                           o_desc0 + (uint64_t)((s0 + kk) * (2048 >> 4)), id_out,
                           (hi > 0 || half > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars.w_free[half]);
            };
            for (int hi = 0; hi < nh && ok; ++hi) {
                const int st = hi % NS, st1 = (hi + 1) % NS;
                const uint32_t ph1 = ((hi + 1) / NS) & 1;
                const bool nxt = hi + 1 < nh;
                if (!(ok = mbar_wait_or_abort(&bars.w_ready[0], hi & 1, abort, kWaitNs))) break;
                tc_fence_after();
                gemm2(hi, 0);
                const bool early = nxt && mbar_test_wait(smem_u32(&bars.full[st1]), ph1);
                if (early) {
                    tc_fence_after();
                    gemm1(hi + 1, 0);
                }
                if (!(ok = mbar_wait_or_abort(&bars.w_ready[1], hi & 1, abort, kWaitNs))) break;
                tc_fence_after();
                gemm2(hi, 1);
                if (early) {
                    gemm1(hi + 1, 1);
                    mma_commit(&bars.g1done[st1]);
                }
                if (!(ok = mbar_wait_or_abort(&bars.qready[st], (hi / NS) & 1, abort, kWaitNs))) break;
                tc_fence_after();
                const uint64_t qd = q_desc0 + (uint64_t)st * kStageD;
                const uint64_t sd = s_desc0 + (uint64_t)st * kStageD;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + COL_ACC, qd + 2 * kk, sd + (uint64_t)(kk * (2048 >> 4)), id_out, 1u);
                mma_commit(&bars.xfree[st]);
                if (nxt && !early) {
                    if (!(ok = mbar_wait_or_abort(&bars.full[st1], ph1, abort, kWaitNs))) break;
                    tc_fence_after();
                    gemm1(hi + 1, 0);
                    gemm1(hi + 1, 1);
                    mma_commit(&bars.g1done[st1]);
                }
            }
            if (ok) mma_commit(&bars.acc_full);
            if (*abort) {   // nothing may be in flight when TMEM is freed
                mma_commit(&bars.drain);
                mbar_wait(&bars.drain, 0, kWaitNs);
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpiWarp0;              // 0 .. kEpiWarps-1
        const int q = warp & 3;                       // TMEM lane quadrant
        const int grp = ew >> 2;                      // key-block parity / column group
        const int R0 = 128 * qt + 32 * q;             // first row of the warp (chunk-local)
        const int tr = R0 + lane;                     // this thread's row
        const int jd = (R0 - kb) >> 5;                // the warp's diagonal key block
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int nbh = KS / 64;                      // key blocks per half (even)
        float* vq = vqa + q * 256;
        // Key blocks outside the mask are zero for every head: written once.
        {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            for (int j = grp; j < KS / 32; j += 2)
                if (kRev ? j < jd : j > jd) tmem_st16(tmem + lane_off + COL_W + 16 * j, z);
            tmem_wait_st();
        }
        bool ok = true;
        for (int hi = 0; hi < nh && ok; ++hi) {
            const int st = hi % NS;
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.vready[st], (hi / NS) & 1, abort, kWaitNs));
            if (!ok) break;
            const float* ck = cv + st * 256;
            const float* dk = dv + st * 256;
            // Off the diagonal block, 2^-|c2_r - c2_k| = u_r v_k with the warp's
            // first row (causal) or last row (anti-causal) as reference: both <= 1.
            const float cr = ck[tr], drow = dk[tr];
            const float cref = kRev ? ck[R0 + 31] : ck[R0];
            const float u = kRev ? ex2(cref - cr) * drow : ex2(cr - cref);
            for (int j = grp; j < KS / 32; j += 2)
                if (kRev ? j > jd : j < jd) {
                    const int k = kb + 32 * j + lane;
                    vq[32 * j + lane] = kRev ? ex2(ck[k] - cref) : ex2(cref - ck[k]) * dk[k];
                }
            __syncwarp();
            for (int half = 0; half < 2 && ok; ++half) {
                ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.d1_full[half], hi & 1, abort, kWaitNs));
                if (ok && hi > 0)
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait_or_abort(&bars.w_free[half], (hi - 1) & 1, abort, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                for (int j = half * nbh + grp; j < (half + 1) * nbh; j += 2) {
                    if (kRev ? j < jd : j > jd) continue;   // zero block
                    uint32_t r[32];
                    tmem_ld32_sync(tmem + lane_off + COL_D1 + 32 * j, r);
                    uint32_t m[16];
                    if (j != jd) {
                        const float4* v4 = reinterpret_cast<const float4*>(vq + 32 * j);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 v = v4[e4];
                            m[2 * e4] = pack_bf16x2(__uint_as_float(r[4 * e4]) * (u * v.x),
                                                    __uint_as_float(r[4 * e4 + 1]) * (u * v.y));
                            m[2 * e4 + 1] = pack_bf16x2(__uint_as_float(r[4 * e4 + 2]) * (u * v.z),
                                                        __uint_as_float(r[4 * e4 + 3]) * (u * v.w));
                        }
                    } else {
                        // Diagonal block: key R0 + e against row R0 + lane; the
                        // exponent is masked before exp2 (in the mask it is <= 0).
                        const float4* c4 = reinterpret_cast<const float4*>(ck + R0);
                        const float4* d4 = reinterpret_cast<const float4*>(dk + R0);
                        float mv[32];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 cvv = c4[e4], dvv = d4[e4];
                            const float cs[4] = {cvv.x, cvv.y, cvv.z, cvv.w};
                            const float ds[4] = {dvv.x, dvv.y, dvv.z, dvv.w};
#pragma unroll
                            for (int uu = 0; uu < 4; ++uu) {
                                const int e = 4 * e4 + uu;
                                const float d1 = __uint_as_float(r[e]);
                                if (kRev)
                                    mv[e] = d1 * ex2(e >= lane ? cs[uu] - cr : -INFINITY) * drow;
                                else
                                    mv[e] = d1 * ex2(e <= lane ? cr - cs[uu] : -INFINITY) * ds[uu];
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) m[e] = pack_bf16x2(mv[2 * e], mv[2 * e + 1]);
                    }
                    tmem_st16(tmem + lane_off + COL_W + 16 * j, m);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars.w_ready[half]);
            }
        }
        // Drain: add the accumulator into the output, one 32 x 32 fp32 piece per
        // TMA reduce-add (128-byte swizzled rows; the stages are free by now).
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.acc_full, 0, abort, kWaitNs));
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int pc = 0; pc < NB; ++pc) {
                const int col = grp * (NO / 2) + 32 * pc;
                uint32_t r[32];
                tmem_ld32_sync(tmem + lane_off + COL_ACC + col, r);
                uint8_t* buf = sStage + (ew * NB + pc) * 4096;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4*>(buf + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                        make_uint4(r[4 * cc], r[4 * cc + 1], r[4 * cc + 2], r[4 * cc + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_3d(&tm_out, buf, g * N + cb * NO + col, c * L + R0, b);
                    bulk_commit();
                }
            }
            if (lane == 0) bulk_wait<0>();
        }
    } else {
        // ----------------------------------------------------------- converters
        // Per head: the chunk's c2 and dt into the stage's vector buffers (c2 of
        // the last token and dt = 0 past the sequence end), then, once GEMM1 has
        // read Q, Q's rows rescaled in place by f.  Lane l of converter warp w
        // owns the factors of rows 64 w + l and 64 w + 32 + l; each pass of the
        // warp rescales four whole rows (conflict-free 16-byte accesses).
        const int ctid = threadIdx.x;                 // 0 .. kConvThreads-1
        const int cw = ctid >> 5;
        constexpr int KPT = L / kConvThreads;
        const int64_t row0 = (int64_t)b * H * T + (int64_t)c * L;
        float pc[KPT], pd[KPT], plast = 0.f, prc[2], prd[2];
        auto prefetch = [&](int hi) {
            const float* crow = cum2 + row0 + (int64_t)(h0 + hi) * T;
            const float* drow = dtT + row0 + (int64_t)(h0 + hi) * T;
            plast = __ldg(crow + Lc - 1);
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                const int s = ctid + kConvThreads * i;
                pc[i] = s < Lc ? __ldg(crow + s) : plast;
                pd[i] = s < Lc ? __ldg(drow + s) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = 128 * qt + 64 * cw + 32 * i + lane;
                prc[i] = r < Lc ? __ldg(crow + r) : plast;
                prd[i] = r < Lc ? __ldg(drow + r) : 0.f;
            }
        };
        if (nh > 0) prefetch(0);
        bool ok = true;
        for (int hi = 0; hi < nh && ok; ++hi) {
            const int st = hi % NS, k = hi / NS;
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.full[st], k & 1, abort, kWaitNs));
            if (!ok) break;
            float* ck = cv + st * 256;
            float* dk = dv + st * 256;
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                ck[ctid + kConvThreads * i] = pc[i];
                dk[ctid + kConvThreads * i] = pd[i];
            }
            float f[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) f[i] = kRev ? prd[i] * ex2(plast - prc[i]) : ex2(prc[i]);
            mbar_arrive(&bars.vready[st]);
            if (hi + 1 < nh) prefetch(hi + 1);
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.g1done[st], k & 1, abort, kWaitNs));
            if (!ok) break;
            uint8_t* sq = sStage + st * C::STAGE;
#pragma unroll 4
            for (int m = 0; m < 16; ++m) {
                const int ro = 4 * m + (lane >> 3);   // row within this warp's 64
                const float f0 = __shfl_sync(0xffffffffu, f[0], ro & 31);
                const float f1 = __shfl_sync(0xffffffffu, f[1], ro & 31);
                uint4* p = reinterpret_cast<uint4*>(sq + (64 * cw + ro) * 128 + (lane & 7) * 16);
                *p = scale_bf16x8(*p, ro < 32 ? f0 : f1);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars.qready[st]);
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

template <int L, int NO, bool kRev>
cudaError_t launch_bc(const Dims& d, const void* q, const void* k, const void* o, const void* s,
                      const float* cum2, const float* dtT, float* out, int hpc, int32_t* err,
                      cudaStream_t st) {
    using C = BCCfg<L, NO>;
    CUtensorMap tm_q, tm_k, tm_o, tm_s, tm_out;
    // Q and K: [b][T][H * 64] bf16; O and out: [b][T][G * N] (bf16 / fp32); S: rows
    // (b, c, h, p) of N columns, bf16.
    const uint64_t xd[3] = {(uint64_t)(d.H * 64), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t xs[2] = {(uint64_t)(d.H * 64 * 2), (uint64_t)(d.T * d.H * 64 * 2)};
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t od[3] = {(uint64_t)(d.G * d.N), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t os[2] = {(uint64_t)(d.G * d.N * 2), (uint64_t)(d.T * d.G * d.N * 2)};
    const uint64_t ys[2] = {(uint64_t)(d.G * d.N * 4), (uint64_t)(d.T * d.G * d.N * 4)};
    const uint32_t ybox[3] = {32, 32, 1};
    const uint64_t sd[2] = {(uint64_t)d.N, (uint64_t)(d.b * d.nc * d.H * 64)};
    const uint64_t ss[1] = {(uint64_t)(d.N * 2)};
    const uint32_t sbox[2] = {64, 64};
    if (!make_tmap_bf16(&tm_q, q, 3, xd, xs, box) || !make_tmap_bf16(&tm_k, k, 3, xd, xs, box) ||
        !make_tmap_bf16(&tm_o, o, 3, od, os, box) || !make_tmap_bf16(&tm_s, s, 2, sd, ss, sbox) ||
        !make_tmap(&tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, 3, od, ys, ybox,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t grid = d.b * d.nc * (d.H / hpc) * (L / 128) * (d.N / NO);
    auto kern = bwd_bc_tc_kernel<L, NO, kRev>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), C::SMEM, st, false, tm_q, tm_k,
                         tm_o, tm_s, tm_out, cum2, dtT, (int)d.T, (int)d.H, (int)d.G, (int)d.N,
                         (int)d.nc, hpc, err);
}

template <bool kRev>
cudaError_t launch_bc_l(const Dims& d, const void* q, const void* k, const void* o, const void* s,
                        const float* cum2, const float* dtT, float* out, int hpc, int32_t* err,
                        cudaStream_t st) {
    if (d.L == 256)
        return d.N == 64 ? launch_bc<256, 64, kRev>(d, q, k, o, s, cum2, dtT, out, hpc, err, st)
                         : launch_bc<256, 128, kRev>(d, q, k, o, s, cum2, dtT, out, hpc, err, st);
    return d.N == 64 ? launch_bc<128, 64, kRev>(d, q, k, o, s, cum2, dtT, out, hpc, err, st)
                     : launch_bc<128, 128, kRev>(d, q, k, o, s, cum2, dtT, out, hpc, err, st);
}

}  // namespace

bool bwd_bc_tc_supported(const Dims& d) {
    return d.dtype == 1 && d.P == 64 && (d.L == 128 || d.L == 256) &&
           (d.N == 64 || d.N == 128 || d.N == 256) && d.G > 0 && d.H % d.G == 0 &&
           d.T < (int64_t(1) << 31) && d.b * d.nc * d.H * 64 < (int64_t(1) << 31);
}

// Heads per CTA: the largest divisor of the heads per group that still gives
// four waves of CTAs (each CTA pays a fixed cost of about two heads: O's load,
// the pipeline's fill and the accumulator's drain).
int bwd_bc_heads_per_cta(const Dims& d) {
    const int64_t hpg = d.H / d.G;
    const int64_t per = d.b * d.nc * d.G * (d.L / 128) * (d.N > 128 ? d.N / 128 : 1);
    const int64_t want = 4 * (int64_t)sm_count();
    for (int64_t v = hpg; v >= 1; --v)
        if (hpg % v == 0 && per * (hpg / v) >= want) return (int)v;
    return 1;
}

cudaError_t launch_bwd_bc_tc(const Dims& d, bool rev, const void* q, const void* k, const void* o,
                             const void* s, const float* cum2, const float* dtT, float* out,
                             int32_t* err, cudaStream_t st) {
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    if (!bwd_bc_tc_supported(d)) return cudaErrorInvalidValue;
    const int hpc = bwd_bc_heads_per_cta(d);
    if (d.b * d.nc * (d.H / hpc) * (d.L / 128) * (d.N > 128 ? 2 : 1) >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    return rev ? launch_bc_l<true>(d, q, k, o, s, cum2, dtT, out, hpc, err, st)
               : launch_bc_l<false>(d, q, k, o, s, cum2, dtT, out, hpc, err, st);
}

}  // namespace m2
