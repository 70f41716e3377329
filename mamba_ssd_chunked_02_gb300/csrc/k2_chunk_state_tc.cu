// k2_chunk_state_tc.cu -- stage 2 on tcgen05 tensor cores: chunk states by the
// jump formula.
//
// Pages: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile" (brifing.si), section 4 "Mathematical Jump Formula
// Implementation" (stacking a chunk's B and X turns the state update into one
// matrix product) and section 5 "Handling Exponential Decay Terms" (rows are
// pre-multiplied by their decay so that tensor cores still apply);
// "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr), "세 가지 핵심
// 커널 구현" (fwd_pass_state uses tensor-core MMA for the chunk states).
//
//   dS[b,c,h,p,n] = sum_{s in chunk c} B[s,n] * w_s * x[s,p],
//   w_s = dtT[s] * exp2(cum2[last token of c] - cum2[s])
//
// The same contraction with w_s = exp2(cum2[s]), x = dy and B = C is the
// backward pass's chunk adjoint sum_s exp2(cum2_s) dy_s C_s^T (weight mode 1).
//
// As a GEMM per (b, c, h): D[n, p] = A[n, s] * X~[s, p] with M = n (a 128-wide
// tile of the state dimension), N = P = 64, K = L (the chunk).
//   * A = B_chunk^T straight from HBM: B is [s][n] with n contiguous, i.e. an
//     MN-major operand; it is shared by every head of the group, so one CTA
//     loads it once (TMA, 128-byte swizzle) and reuses it for `hpc` heads.
//   * X~ = diag(w) X: x is [s][p] with p contiguous (MN-major); TMA brings the
//     chunk into a stage buffer and four warps scale each 128-byte row s by w_s
//     in place (a row of the swizzled tile is one s, so the swizzle does not
//     matter), then hand it to the tensor core.  The decay is thus folded into
//     the operand the kernel produces itself; the pages route that operand to
//     tensor memory instead, to avoid shared-memory contention, which does not
//     limit this HBM-bound kernel.
//   * D accumulates in tensor memory (fp32), double buffered across heads; four
//     warps read it back (tcgen05.ld) into a shared [p][n] tile and one TMA
//     store per head writes it to dS, in fp32 or, on the whole-path call, in
//     bf16 (the stage-3 kernel reads it back at once; half the bytes).
// Warp roles: 0 = TMA producer, 1 = MMA issuer (+ TMEM owner), then L / 32
// scaling warps (one x row per thread: two per sub-partition at L = 256, so that
// one warp's load latency hides behind the other's), then 4 epilogue warps.
// Stage ring of NS x-buffers; every wait is bounded.
//
// Fused variant (stages 2 and 3 in one kernel, used by the whole-path call):
// the epilogue does not store dS.  Per head it takes the state entering its
// chunk, Sprev_c, from the CTA that handled chunk c-1 (published through a
// two-slot fp32 ring in global memory plus one flag word per (b, h, n-tile,
// chunk) written with release semantics): one TMA load brings the [P x n-tile]
// tile into shared memory, each lane n updates its column in place
// (decay_c * Sprev_c + dS_c, with dS_c from tensor memory) and writes the bf16
// copy of Sprev_c beside it, and two TMA stores write Sprev_c (for stage 4) and
// the next state (for chunk c+1, or the final state after the last chunk).
// The CTA raises its heads' flags once all its stores have completed (a CTA of
// chunk c+1 normally starts a wave later, when they are long set).  Pages: "Accelerating
// Mamba-2 ..." section 8 (fwd_pass_state walks the chunks in order, combining
// the decayed carried state with the chunk's own contribution).  The carried
// state never goes to HBM as a whole tensor: each ring slot is read shortly
// after it is written, while it is still in L2.  CTAs take their work item from
// a global ticket counter in chunk-major order, so every CTA a CTA waits for has
// already started (no dependence on the hardware's CTA launch order); waits are
// bounded, and a CTA that gives up marks its flags so that its successors stop
// at once.
#include "common.cuh"
#include "internal.h"
#include "tc5.cuh"
#include "tmap.h"

namespace m2 {
namespace {

using namespace tc;

constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait

template <int L, bool kFuse, bool kDS16>
struct K2Cfg {
    static constexpr int P = 64;
    static constexpr int kSW = L / 32;                    // scaling warps: one x row per thread
    static constexpr int kThreads = 64 + 32 * kSW + 128;  // producer, MMA, scaling, epilogue
    // x stages: shared memory left after B^T and the dS staging tiles (the
    // fused variant spends it on its state tiles instead).
    static constexpr int NS = L == 256 ? (kFuse ? 2 : (kDS16 ? 4 : 3)) : 6;
    static constexpr int ATOM = L * 128;                  // one 64-wide MN block, L rows
    static constexpr int BT_BYTES = 2 * ATOM;             // two 64-n blocks = M of 128
    static constexpr int X_BYTES = ATOM;                  // P = 64: one block
    static constexpr int D_BYTES = 64 * 128 * (kDS16 ? 2 : 4);   // one dS tile [p][n-tile]
    // fused: two buffers of {carried state fp32 [64][128], Sprev bf16 [64][128]}
    static constexpr int F_BYTES = 2 * (64 * 128 * 4 + 64 * 128 * 2);
    static constexpr int SMEM = 1024 + BT_BYTES + NS * X_BYTES + (kFuse ? F_BYTES : 2 * D_BYTES);
    // Tensor memory: 2 accumulators x 64 columns, then B^T as the MMA's A operand
    // (lane = state dim n, L keys as 16-bit pairs: L / 2 columns); the plain
    // variant keeps two B^T slots, so that the next group segment's B^T is copied
    // in while the MMAs of the current one still read theirs.
    static constexpr uint32_t COL_BT = 128;
    static constexpr uint32_t BT_COLS = L / 2;
    static constexpr int TMEM_COLS = (kFuse || L == 128) ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, 64, 0, 1);   // A in tensor memory, B MN-major
};

struct K2Bars {
    uint64_t bt_full;
    uint64_t bt_tmem[2];    // B^T copied into tensor-memory slot 0 / 1 by the epilogue warps
    uint64_t full[6], scaled[6], xfree[6];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;         // commit target used to drain in-flight MMAs on abort
    uint64_t cfull[2];      // fused: carried-state tile landed (per tile buffer)
    uint64_t epi_sync;      // group barrier of the 4 epilogue warps (abortable)
    uint32_t tmem_base;
    int abort;
    int item;               // work item (ticket on the fused path)
};

// Arguments used by the fused variant only (null on the plain one).
struct FuseArgs {
    const float* init;        // [b][H][P][N] fp32 or null (zero initial state)
    float* carry;             // [2][b][H][P][N] fp32 ring
    int32_t* flags;           // [b][H][n_tiles][nc]
    int32_t* ticket;          // work-item counter
    __nv_bfloat16* Sprev;     // [b][nc][H][P][N]
    float* fin;               // [b][H][P][N]
    int nb;                   // batch
    int adj = 0;              // weight mode: 0 = w_s above, 1 = w_s = exp2(cum2[s])
};

// Plain variant's work order: unit u = ((b * nc + c) * n_tiles + nt) * H + h, one
// head of one (b, chunk, state tile); a CTA takes units [u0, u0 + upc).  The heads
// of one group with the same (b, c, nt) form a segment, which shares B^T.
struct UnitIt {
    int b, c, nt, h;
    __device__ void init(int64_t u, int H, int n_tiles, int nc) {
        h = (int)(u % H);
        u /= H;
        nt = (int)(u % n_tiles);
        u /= n_tiles;
        c = (int)(u % nc);
        b = (int)(u / nc);
    }
    __device__ void next(int H, int n_tiles, int nc) {   // carries instead of divisions
        if (++h < H) return;
        h = 0;
        if (++nt < n_tiles) return;
        nt = 0;
        if (++c < nc) return;
        c = 0;
        ++b;
    }
};

template <int L, bool kFuse, bool kDS16>
__global__ void __launch_bounds__(K2Cfg<L, kFuse, kDS16>::kThreads, 1)
chunk_state_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_d,
                      const __grid_constant__ CUtensorMap tm_ring,   // fused: [2 b H P][N] f32
                      const __grid_constant__ CUtensorMap tm_init,   // fused: [b H P][N] f32
                      const __grid_constant__ CUtensorMap tm_fin,    // fused: [b H P][N] f32
                      const __grid_constant__ CUtensorMap tm_sp,     // fused: [b nc H P][N] bf16
                      const float* __restrict__ cum2, const float* __restrict__ dtT,
                      int T, int H, int N, int G, int nc, int n_tiles, int pts, int pst,
                      int hpc, int n_hblk, int upc, int64_t units, int32_t* err,
                      const FuseArgs fa, uint32_t* __restrict__ xabs) {
    using C = K2Cfg<L, kFuse, kDS16>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sBt = smem;
    uint8_t* sX = smem + C::BT_BYTES;
    float* sD = reinterpret_cast<float*>(sX + NS * C::X_BYTES);   // [2][64][128]
    __shared__ K2Bars bars;
    volatile int* abort = &bars.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars.bt_full, 1);
        mbar_init(&bars.bt_tmem[0], 128);
        mbar_init(&bars.bt_tmem[1], 128);
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.scaled[i], 32 * C::kSW);
            mbar_init(&bars.xfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.acc_full[i], 1);
            mbar_init(&bars.acc_empty[i], 128);
        }
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.cfull[0], 1);
        mbar_init(&bars.cfull[1], 1);
        mbar_init(&bars.epi_sync, 128);
        bars.abort = 0;
        bars.item = kFuse ? atomicAdd(fa.ticket, 1) : (int)blockIdx.x;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars.tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    // Work item.  Plain: units [u0, u0 + nh) in unit order (the first unit's
    // position below; later ones from UnitIt).  Fused: a block of hpc heads of one
    // (b, c, n-tile), chunk outermost, in ticket order.
    const int hpg = H / G;
    int b, c, nt, h0, nh;
    int64_t u0 = 0;
    if (kFuse) {
        int rest = bars.item;
        const int per_chunk = fa.nb * n_tiles * n_hblk;
        c = rest / per_chunk; rest %= per_chunk;
        b = rest / (n_tiles * n_hblk); rest %= n_tiles * n_hblk;
        nt = rest / n_hblk;
        h0 = (rest % n_hblk) * hpc;
        nh = hpc;
    } else {
        u0 = (int64_t)bars.item * upc;
        nh = (int)(units - u0 < upc ? units - u0 : upc);
        UnitIt first;
        first.init(u0, H, n_tiles, nc);
        b = first.b; c = first.c; nt = first.nt; h0 = first.h;
    }
    const int g = h0 / hpg;

    if (c >= nc) {
        // A ticket past the grid (the counter was not cleared): do nothing.
        if (threadIdx.x == 0) record_error(err, kErrLaunchCfg);
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            if (!kFuse) prefetch_tmap(&tm_d);
            if (kFuse) {
                prefetch_tmap(&tm_ring);
                prefetch_tmap(&tm_sp);
            }
            mbar_arrive_expect_tx(&bars.bt_full, C::BT_BYTES);
            for (int a = 0; a < 2; ++a) {
                // N = 64: both halves of the 128-row M tile hold n in [0, 64).
                const int n_off = (N == 64) ? 0 : nt * 128 + 64 * a;
                tma_load_3d(sBt + a * C::ATOM, &tm_b, &bars.bt_full, g * N + n_off, c * L, b);
            }
            int issued = 0;
            UnitIt it;
            it.init(u0, H, n_tiles, nc);   // plain: the unit's head and chunk
            for (int i = 0; i < nh; ++i) {
                const int st = i % NS, k = i / NS;
                if (!mbar_wait_or_abort(&bars.xfree[st], (k & 1) ^ 1, abort, kWaitNs)) break;
                mbar_arrive_expect_tx(&bars.full[st], C::X_BYTES);
                if (kFuse)
                    tma_load_3d(sX + st * C::X_BYTES, &tm_x, &bars.full[st], (h0 + i) * C::P, c * L, b);
                else
                    tma_load_3d(sX + st * C::X_BYTES, &tm_x, &bars.full[st], it.h * pst, it.c * L, it.b);
                issued = i + 1;
                if (!kFuse) it.next(H, n_tiles, nc);
            }
            if (*abort) {
                // Let every copy already issued land before the CTA can exit (plain:
                // the epilogue warps wait for the B^T loads, which they also issue).
                if (kFuse) mbar_wait(&bars.bt_full, 0, kWaitNs);
                for (int i = issued - 1; i >= 0 && i >= issued - NS; --i)
                    mbar_wait(&bars.full[i % NS], (i / NS) & 1, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            int last = -1;
            // Descriptors formed once; each MMA adds a constant offset / 16 (an MMA
            // issue waits for the scalar work in front of it).
            const uint64_t x_desc0 = smem_desc_sw128(smem_u32(sX), C::ATOM, 1024);
            int seg = -1;                  // segment of head i (its B^T slot: seg & 1)
            int hh = kFuse ? 0 : h0;       // head of unit i (plain), to find segment starts
            for (int i = 0; i < nh; ++i) {
                if (i == 0 || (!kFuse && hh % hpg == 0)) {
                    ++seg;
                    if (!mbar_wait_or_abort(&bars.bt_tmem[seg & 1], (seg >> 1) & 1, abort, kWaitNs)) break;
                    tc_fence_after();
                }
                if (!kFuse && ++hh == H) hh = 0;
                const int st = i % NS, k = i / NS, ab = i & 1, ka = i >> 1;
                if (!mbar_wait_or_abort(&bars.scaled[st], k & 1, abort, kWaitNs)) break;
                if (!mbar_wait_or_abort(&bars.acc_empty[ab], (ka & 1) ^ 1, abort, kWaitNs)) break;
                tc_fence_after();
                const uint64_t xd = x_desc0 + (uint64_t)st * (C::X_BYTES >> 4);
                const uint32_t d = tmem + ab * C::P;
                const uint32_t a = tmem + C::COL_BT + (uint32_t)(seg & 1) * C::BT_COLS;
#pragma unroll
                for (int kk = 0; kk < L / 16; ++kk)
                    mma_ts(d, a + 8 * kk, xd + (uint64_t)(kk * (2048 >> 4)), C::IDESC, kk > 0 ? 1u : 0u);
                mma_commit(&bars.acc_full[ab]);
                mma_commit(&bars.xfree[st]);
                last = i;
            }
            if (last >= 0 && *abort) {   // nothing may be in flight when TMEM is freed
                mma_commit(&bars.drain);
                mbar_wait(&bars.drain, 0, kWaitNs);
            }
        }
    } else if (warp < 2 + C::kSW) {
        // ------------------------------------------------------------- scaling
        constexpr int kST = 32 * C::kSW;                 // scaling threads
        constexpr int RPT = L / kST;                     // x rows per thread (1)
        const int idx = threadIdx.x - 64;                // 0 .. kST - 1
        // Raw decay inputs of the next head, fetched one head ahead.
        float pc[RPT], pd[RPT], plast = 0.f;
        auto prefetch = [&](int bb, int cc, int hh) {
            const int Lc = min(L, T - cc * L);
            const int64_t bh = (int64_t)bb * (H >> pts) + (hh >> pts);   // the head's cum2 / dt row
            const float* crow = cum2 + bh * T + (int64_t)cc * L;
            const float* drow = dtT + bh * T + (int64_t)cc * L;
            plast = __ldg(crow + Lc - 1);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int s = idx + kST * r;
                pc[r] = s < Lc ? __ldg(crow + s) : 0.f;
                pd[r] = s < Lc ? __ldg(drow + s) : 0.f;
            }
        };
        // cum2 and dtT come from stage 1: with programmatic dependent launch the
        // producer's loads of B and x already run; wait for stage 1 here, then
        // let stage 3 start launching.
        grid_dep_wait();
        if (idx == 0) grid_dep_launch();
        // Plain: (b, c, h) of unit i and of unit i + 1; fused: h0 + i of (b, c).
        UnitIt cur, nxt;
        cur.init(u0, H, n_tiles, nc);
        if (kFuse) {
            cur.b = b;
            cur.c = c;
            cur.nt = nt;
            cur.h = h0;
        }
        nxt = cur;
        prefetch(nxt.b, nxt.c, nxt.h);
        for (int i = 0; i < nh; ++i) {
            const int st = i % NS, k = i / NS;
            float w[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r)   // 0 past Lc (the x rows there are zero-filled)
                w[r] = fa.adj ? ex2(pc[r]) : pd[r] * ex2(plast - pc[r]);
            if (kFuse) ++nxt.h;
            else nxt.next(H, n_tiles, nc);
            if (i + 1 < nh) prefetch(nxt.b, nxt.c, nxt.h);
            const bool ok = __all_sync(0xffffffffu,
                                       mbar_wait_or_abort(&bars.full[st], k & 1, abort, kWaitNs));
            if (!ok) break;
            uint8_t* xs = sX + st * C::X_BYTES;
            __nv_bfloat162 xm2 = __floats2bfloat162_rn(0.f, 0.f);   // max |x| (raw), two lanes
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int s = idx + kST * r;
                uint4* row = reinterpret_cast<uint4*>(xs + s * 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    // Lanes own consecutive rows (128 bytes apart); visiting chunk
                    // (q + s) mod 8 spreads a warp's accesses over all 32 banks.
                    const int qc = (q + s) & 7;
                    uint4 v = row[qc];
                    uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (xabs) {
                            const uint32_t a = u[e] & 0x7fff7fffu;
                            xm2 = __hmax2(xm2, *reinterpret_cast<const __nv_bfloat162*>(&a));
                        }
                        const float lo = __uint_as_float(u[e] << 16) * w[r];
                        const float hi = __uint_as_float(u[e] & 0xffff0000u) * w[r];
                        u[e] = pack_bf16x2(lo, hi);
                    }
                    row[qc] = v;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars.scaled[st]);
            if (xabs) {   // this warp's share of max |x| over the chunk, as bf16 bits
                const uint32_t m2u = *reinterpret_cast<const uint32_t*>(&xm2);
                const uint32_t m = __reduce_max_sync(0xffffffffu, max(m2u & 0xffffu, m2u >> 16));
                if (lane == 0) {   // eight words per head; with four scaling warps the rest are 0
                    uint32_t* xw = xabs + ((((int64_t)cur.b * nc + cur.c) * H + cur.h) << 3);
                    xw[warp - 2] = m;
                    if (C::kSW == 4) xw[warp + 2] = 0u;
                }
            }
            cur = nxt;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Plain variant: D[n, p] (lane = n) goes to a shared [p][n] fp32 tile
        // (conflict-free: a warp writes 32 consecutive n of one p), then one TMA
        // store per head writes the tile to dS[b, c, h, :, n-tile].  Fused
        // variant: lane n reads Sprev_c[p, n] for every p (a warp covers 128
        // consecutive bytes), stores it as bf16 and passes the next state on.
        const int q = warp & 3;                          // TMEM lane quadrant
        const int ep = threadIdx.x - 64 - 32 * C::kSW;   // 0..127
        const int NT = N < 128 ? N : 128;                // n-tile width = tile row pitch
        const int nl = 32 * q + lane;                    // n within the tile
        uint32_t sync_phase = 0;
        auto group_sync = [&]() -> bool {
            mbar_arrive(&bars.epi_sync);
            const bool r = mbar_wait_or_abort(&bars.epi_sync, sync_phase, abort, kWaitNs);
            sync_phase ^= 1u;
            return __all_sync(0xffffffffu, r);
        };
        // B^T into tensor memory, once per CTA: lane n takes B[s][n] for every key s
        // from the TMA-loaded tile (64-wide MN blocks, 128-byte swizzled: piece k
        // of row s at k ^ (s & 7)) and writes the pairs (s, s+1) as 32-bit
        // columns.  The tensor core then reads only x~ from shared memory: an
        // M128 N64 MMA with both operands there would take the whole shared-memory
        // bandwidth, which the scaling warps also need.
        auto copy_bt = [&](uint32_t col) {
            const uint8_t* base = sBt + (nl >> 6) * C::ATOM + ((nl & 7) << 1);
            const int k16 = (nl & 63) >> 3;                 // this n's 16-byte piece of a row
#pragma unroll 1
            for (int s0 = 0; s0 < L; s0 += 64) {
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int sa = s0 + 2 * e, sb = sa + 1;
                    const uint32_t lo = *reinterpret_cast<const uint16_t*>(
                        base + sa * 128 + ((k16 ^ (sa & 7)) << 4));
                    const uint32_t hi = *reinterpret_cast<const uint16_t*>(
                        base + sb * 128 + ((k16 ^ (sb & 7)) << 4));
                    w[e] = lo | (hi << 16);
                }
                tmem_st32(tmem + ((uint32_t)(32 * q) << 16) + col + (s0 >> 1), w);
            }
            tmem_wait_st();
        };
        if constexpr (kFuse) {
            {
                const bool okb = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.bt_full, 0, abort, kWaitNs));
                if (okb) copy_bt(C::COL_BT);
                tc_fence_before();
                mbar_arrive(&bars.bt_tmem[0]);
            }
            const int64_t bH = (int64_t)fa.nb * H;
            const int Lc = min(L, T - c * L);
            const bool own = nl < NT;
            const bool has_in = c > 0 || fa.init != nullptr;   // else Sprev_0 = 0
            const bool last = c == nc - 1;
            float* sCT = reinterpret_cast<float*>(sX + NS * C::X_BYTES);          // [2][64][NT]
            __nv_bfloat16* sSP = reinterpret_cast<__nv_bfloat16*>(sCT + 2 * 64 * 128);  // [2][64][NT]
            auto flag_of = [&](int i) {
                return fa.flags + (((int64_t)b * H + h0 + i) * n_tiles + nt) * nc + c;
            };
            int published = 0;            // ep == 0: heads whose flag is raised (at the end)
            int pending[2] = {-1, -1};    // ep == 0: head whose tile load is in flight, per buffer
            for (int i = 0; i < nh; ++i) {
                const int ab = i & 1, ka = i >> 1, buf = i & 1;
                const int64_t bh = (int64_t)b * H + h0 + i;
                float* ct = sCT + buf * (64 * 128);
                __nv_bfloat16* spt = sSP + buf * (64 * 128);
                if (ep == 0) {
                    bulk_wait_read<1>();      // stores of head i-2 (same buffers) have read them
                    bool go = true;
                    if (c > 0) go = wait_flag(flag_of(i) - 1, abort, kWaitNs);
                    if (go && has_in) {
                        fence_proxy_async();  // the acquire above before the async-proxy read
                        mbar_arrive_expect_tx(&bars.cfull[buf], (uint32_t)(NT * 64 * 4));
                        if (c > 0)
                            tma_load_2d(ct, &tm_ring, &bars.cfull[buf], nt * 128,
                                        (int)((((int64_t)(c & 1)) * bH + bh) * C::P));
                        else
                            tma_load_2d(ct, &tm_init, &bars.cfull[buf], nt * 128, (int)(bh * C::P));
                        pending[buf] = i;
                    }
                }
                // Without an incoming tile nothing else orders the writes below after
                // ep 0's wait for the stores that last read these buffers.
                if (!has_in && i >= 2 && !group_sync()) break;
                bool ok = __all_sync(0xffffffffu,
                                     mbar_wait_or_abort(&bars.acc_full[ab], ka & 1, abort, kWaitNs));
                if (ok && has_in)
                    ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bars.cfull[buf], (i >> 1) & 1,
                                                                    abort, kWaitNs));
                if (!ok) break;
                if (ep == 0) pending[buf] = -1;
                tc_fence_after();
                const int64_t bho = (int64_t)b * (H >> pts) + ((h0 + i) >> pts);
                const float dec = ex2(__ldg(cum2 + bho * T + (int64_t)c * L + Lc - 1));
#pragma unroll
                for (int cc = 0; cc < C::P / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld32_sync(tmem + ((uint32_t)(32 * q) << 16) + ab * C::P + 32 * cc, r);
                    if (own) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int o = (32 * cc + j) * NT + nl;
                            const float sv = has_in ? ct[o] : 0.f;
                            spt[o] = __float2bfloat16_rn(sv);
                            ct[o] = fmaf(dec, sv, __uint_as_float(r[j]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.acc_empty[ab]);
                fence_proxy_async_smem();
                if (!group_sync()) break;
                if (ep == 0) {
                    tma_store_2d(&tm_sp, spt, nt * 128, (int)((((int64_t)b * nc + c) * H + h0 + i) * C::P));
                    if (last)
                        tma_store_2d(&tm_fin, ct, nt * 128, (int)(bh * C::P));
                    else
                        tma_store_2d(&tm_ring, ct, nt * 128,
                                     (int)((((int64_t)((c + 1) & 1)) * bH + bh) * C::P));
                    bulk_commit();
                }
            }
            if (ep == 0) {
                bulk_wait<0>();
                if (!last) {
                    fence_proxy_async();
                    __threadfence();
                    // Heads completed without an abort get their flag; after an abort
                    // the rest are marked so that the next chunk's CTA stops at once.
                    const int done = *abort ? published : nh;
                    for (; published < done; ++published) st_release_gpu(flag_of(published), 1);
                    for (int i = published; i < nh; ++i) st_release_gpu(flag_of(i), -1);
                }
                // A tile load still in flight after an abort must land before exit.
                for (int k = 0; k < 2; ++k)
                    if (pending[k] >= 0) mbar_wait(&bars.cfull[k], (pending[k] >> 1) & 1, kWaitNs);
            }
        } else {
            // B^T per segment (the heads of one group of one (b, c, n-tile) in this
            // CTA's range): segment k's tile is copied into tensor-memory slot k & 1
            // after the epilogue has finished head f_k - 2 (f_k: the segment's first
            // head), when the MMAs of segment k - 2 -- the slot's last user -- have
            // completed; the shared tile is then free, and segment k + 1's B^T is
            // loaded into it at once, so the MMAs never wait for a reload.
            const int64_t seg0 = u0 / hpg;
            const int nseg = (int)((u0 + nh - 1) / hpg - seg0) + 1;
            auto seg_first = [&](int k) { return k == 0 ? 0 : (int)((seg0 + k) * hpg - u0); };
            int bt_issued = 1, bt_done = 0;   // B^T loads issued (the producer's first) / landed
            auto copy_seg = [&](int k) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bars.bt_full, k & 1, abort, kWaitNs)))
                    return false;
                bt_done = k + 1;
                copy_bt(C::COL_BT + (uint32_t)(k & 1) * C::BT_COLS);
                tc_fence_before();
                mbar_arrive(&bars.bt_tmem[k & 1]);
                if (k + 1 < nseg) {
                    if (!group_sync()) return false;           // every lane has read the tile
                    if (ep == 0) {
                        int64_t sg = seg0 + k + 1;
                        const int gg = (int)(sg % G);
                        sg /= G;
                        const int tt = (int)(sg % n_tiles);
                        sg /= n_tiles;
                        const int cc = (int)(sg % nc), bb = (int)(sg / nc);
                        mbar_arrive_expect_tx(&bars.bt_full, C::BT_BYTES);
                        for (int a = 0; a < 2; ++a) {
                            const int n_off = (N == 64) ? 0 : tt * 128 + 64 * a;
                            tma_load_3d(sBt + a * C::ATOM, &tm_b, &bars.bt_full, gg * N + n_off, cc * L, bb);
                        }
                    }
                    bt_issued = k + 2;
                }
                return true;
            };
            bool run = copy_seg(0);
            int kc = 1;
            while (run && kc < nseg && seg_first(kc) <= 1) run = copy_seg(kc++);
            UnitIt it;
            it.init(u0, H, n_tiles, nc);
            for (int i = 0; run && i < nh; ++i) {
                const int ab = i & 1, ka = i >> 1;
                const bool ok = __all_sync(0xffffffffu,
                                           mbar_wait_or_abort(&bars.acc_full[ab], ka & 1, abort, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                float* tile = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sD) + ab * C::D_BYTES);
                if (ep == 0) bulk_wait_read<1>();            // the store that used this tile is done
                if (!group_sync()) break;                    // ... before any warp writes it
#pragma unroll
                for (int cc = 0; cc < C::P / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld32_sync(tmem + ((uint32_t)(32 * q) << 16) + ab * C::P + 32 * cc, r);
                    if (kDS16 && nl < NT) {
                        __nv_bfloat16* t16 = reinterpret_cast<__nv_bfloat16*>(tile);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            t16[(32 * cc + j) * NT + nl] = __float2bfloat16_rn(__uint_as_float(r[j]));
                    } else if (nl < NT) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) tile[(32 * cc + j) * NT + nl] = __uint_as_float(r[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.acc_empty[ab]);
                fence_proxy_async_smem();
                if (!group_sync()) break;
                if (ep == 0) {
                    const int row = (int)((((int64_t)it.b * nc + it.c) * H + it.h) * pst);
                    tma_store_2d(&tm_d, tile, it.nt * 128, row);
                    bulk_commit();
                }
                it.next(H, n_tiles, nc);
                while (run && kc < nseg && seg_first(kc) - 2 <= i) run = copy_seg(kc++);
            }
            if (ep == 0) {
                bulk_wait<0>();
                // After an abort: B^T loads still in flight land before the CTA exits.
                for (int k = bt_done; k < bt_issued; ++k) mbar_wait(&bars.bt_full, k & 1, kWaitNs);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && bars.abort) record_error(err, kFuse ? (kErrTimeoutK2 | kErrChainK23) : kErrTimeoutK2);
}

// Heads per CTA in blocks of one group (one CTA per SM at a time): the divisor
// v of H/G that minimises (waves of CTAs) x (v + 4), i.e. per-SM time in head
// units with a CTA's fixed work (loading B^T, filling and draining the x ring)
// counted as about four heads (fitted to measurements: at b8 T4096 H80 N128
// whole-path times of 440, 437, 429 and 423 us for 10, 20, 40 and 80 heads per
// CTA).  *cost receives the minimum.
int pick_hpc(const Dims& d, int64_t outer, int64_t* cost) {
    const int64_t hpg = d.H / d.G, sms = sm_count();
    int best = 1;
    int64_t best_cost = -1;
    for (int64_t v = 1; v <= hpg; ++v) {
        if (hpg % v) continue;
        const int64_t ctas = outer * (d.H / v);
        const int64_t c = (ctas + sms - 1) / sms * (v + 4);
        if (best_cost < 0 || c <= best_cost) {
            best_cost = c;
            best = (int)v;
        }
    }
    *cost = best_cost;
    return best;
}

// One wave of CTAs over all units: ceil(U / SMs) units each.
int even_upc(const Dims& d, int64_t units) {
    const int64_t sms = sm_count();
    return (int)std::max<int64_t>(1, (units + sms - 1) / sms);
}

// Fused variant: the largest divisor of H/G (at most 16) for which one chunk's
// CTAs, b * n_tiles * H / hpc, still cover every SM.
int pick_hpc_fused(const Dims& d, int64_t n_tiles) {
    const int hpg = (int)(d.H / d.G);
    for (int v = 16; v >= 1; --v)
        if (hpg % v == 0 && d.b * n_tiles * (d.H / v) >= sm_count()) return v;
    return 1;
}

template <int L, bool kFuse, bool kDS16>
cudaError_t launch_k2(const Dims& d, const void* x, const void* B, const float* cum2,
                      const float* dtT, void* dS, const FuseArgs& fa, int32_t* err,
                      cudaStream_t st, uint32_t* xabs = nullptr, bool pdl = false) {
    using C = K2Cfg<L, kFuse, kDS16>;
    constexpr bool ds16 = kDS16;
    CUtensorMap tm_x, tm_b;
    const uint64_t xd[3] = {(uint64_t)(d.H * d.P), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t xs[2] = {(uint64_t)(d.sx[1] * 2), (uint64_t)(d.sx[0] * 2)};   // token, batch
    const uint32_t box[3] = {64, (uint32_t)L, 1};
    const uint64_t bd[3] = {(uint64_t)(d.G * d.N), (uint64_t)d.T, (uint64_t)d.b};
    const uint64_t bs[2] = {(uint64_t)(d.sB[1] * 2), (uint64_t)(d.sB[0] * 2)};
    if (!make_tmap_bf16(&tm_x, x, 3, xd, xs, box) || !make_tmap_bf16(&tm_b, B, 3, bd, bs, box))
        return cudaErrorInvalidValue;
    CUtensorMap tm_d = tm_x;   // the fused variant stores no dS
    CUtensorMap tm_ring = tm_x, tm_init = tm_x, tm_fin = tm_x, tm_sp = tm_x;   // plain: unused
    if (kFuse) {
        const uint32_t tbox[2] = {(uint32_t)(d.N < 128 ? d.N : 128), 64};
        const uint64_t rs[1] = {(uint64_t)(d.N * 4)};
        const uint64_t ring_d[2] = {(uint64_t)d.N, (uint64_t)(2 * d.b * d.H * d.P)};
        const uint64_t st_d[2] = {(uint64_t)d.N, (uint64_t)(d.b * d.H * d.P)};
        const uint64_t sp_d[2] = {(uint64_t)d.N, (uint64_t)(d.b * d.nc * d.H * d.P)};
        const uint64_t sps[1] = {(uint64_t)(d.N * 2)};
        const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        const auto NONE = CU_TENSOR_MAP_SWIZZLE_NONE;
        if (!make_tmap(&tm_ring, F32, fa.carry, 2, ring_d, rs, tbox, NONE) ||
            !make_tmap(&tm_fin, F32, fa.fin, 2, st_d, rs, tbox, NONE) ||
            (fa.init && !make_tmap(&tm_init, F32, fa.init, 2, st_d, rs, tbox, NONE)) ||
            !make_tmap(&tm_sp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, fa.Sprev, 2, sp_d, sps, tbox, NONE))
            return cudaErrorInvalidValue;
    }
    if (!kFuse) {
        const uint64_t dd[2] = {(uint64_t)d.N, (uint64_t)(d.b * d.nc * d.H * d.P)};
        const uint64_t ds[1] = {(uint64_t)(d.N * (ds16 ? 2 : 4))};
        // P = 32: the 64-column x tile also holds the next head's columns; only
        // the head's own 32 rows of the dS tile are stored.
        const uint32_t dbox[2] = {(uint32_t)(d.N < 128 ? d.N : 128), (uint32_t)(d.P < 64 ? d.P : 64)};
        if (!make_tmap(&tm_d, ds16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       dS, 2, dd, ds, dbox,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    const int n_tiles = d.N > 128 ? (int)(d.N / 128) : 1;
    const int64_t outer = d.b * d.nc * n_tiles, units = outer * d.H;
    // Fused: one chunk's CTAs should fill the GPU, so that the CTA of chunk c
    // typically starts after the one of chunk c-1 has finished (no waiting).
    // Plain: contiguous ranges of upc units.
    int hpc = 0, n_hblk = 0, upc = 0;
    int64_t grid;
    if (kFuse) {
        hpc = pick_hpc_fused(d, n_tiles);
        n_hblk = (int)(d.H / hpc);
        grid = outer * n_hblk;
    } else {
        int src = kFromModel;
        upc = k2_units_per_cta(d, &src);
        grid = (units + upc - 1) / upc;
    }
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    auto k = chunk_state_tc_kernel<L, kFuse, kDS16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, dim3((unsigned)grid), dim3(C::kThreads), C::SMEM, st, pdl, tm_x, tm_b, tm_d,
                         tm_ring, tm_init, tm_fin, tm_sp, cum2, dtT, (int)d.T, (int)d.H, (int)d.N,
                         (int)d.G, (int)d.nc, n_tiles, d.pts, (int)d.P, hpc, n_hblk, upc, units, err, fa,
                         xabs);
}

}  // namespace

int k2_units_per_cta(const Dims& d, int* src) {
    const int64_t n_tiles = d.N > 128 ? d.N / 128 : 1, outer = d.b * d.nc * n_tiles;
    const int64_t units = outer * d.H, hpg = d.H / d.G;
    if (units == 0) {
        *src = kFromModel;
        return 1;
    }
    const int o = tile_override(0);
    if (o > 0 || o == kEvenSplit) {
        *src = kFromOverride;
        return o > 0 ? (int)std::min<int64_t>(o, units) : even_upc(d, units);
    }
    const TileChoice* t = o == -1 ? nullptr : find_tile(d);   // -1: the cost model only
    if (t && t->k2_hpc >= 0) {
        *src = kFromTable;
        return t->k2_hpc > 0 ? (int)std::min<int64_t>(t->k2_hpc, units) : even_upc(d, units);
    }
    // Cost model: blocks of one group's heads against one wave of even ranges.
    // A range of u units touches at most 1 + ceil((u - 1) / (H/G)) segments; the
    // B^T of each further segment is loaded behind the MMAs and its copy into
    // tensor memory costs about one head.
    *src = kFromModel;
    int64_t cost_blk = 0;
    const int hpc = pick_hpc(d, outer, &cost_blk);
    const int upc = even_upc(d, units);
    const int64_t segs = 1 + (upc - 1 + hpg - 1) / hpg;
    const int64_t cost_even = upc + 4 + (segs - 1);
    return cost_even < cost_blk ? upc : hpc;
}

bool tc_supported(const Dims& d) {
    return d.dtype == 1 && (d.L == 128 || d.L == 256) && (d.P == 32 || d.P == 64 || d.P == 128) &&
           (d.N == 64 || d.N == 128 || d.N == 256) && d.T < (int64_t(1) << 31) &&
           d.b * d.nc * d.H * d.P < (int64_t(1) << 31) &&      // TMA row coordinate of Sprev
           d.H * d.P < (int64_t(1) << 31) && d.G * d.N < (int64_t(1) << 31);
}

// The fused stages 2+3 keep a head's 64 columns to itself: P >= 64.
bool tc_fused_supported(const Dims& d) { return tc_supported(d) && d.P >= 64; }

cudaError_t launch_chunk_state_tc(const Dims& dq, const void* x, const void* B, const float* cum2,
                                  const float* dtT, void* dS, bool ds16, int32_t* err,
                                  cudaStream_t st, uint32_t* xabs, bool pdl, bool adj) {
    const Dims d = tc_view(dq);
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    if (!tc_supported(d)) return cudaErrorInvalidValue;
    FuseArgs none{};
    none.adj = adj ? 1 : 0;
    if (ds16)
        return d.L == 256
                   ? launch_k2<256, false, true>(d, x, B, cum2, dtT, dS, none, err, st, xabs, pdl)
                   : launch_k2<128, false, true>(d, x, B, cum2, dtT, dS, none, err, st, xabs, pdl);
    return d.L == 256
               ? launch_k2<256, false, false>(d, x, B, cum2, dtT, dS, none, err, st, xabs, pdl)
               : launch_k2<128, false, false>(d, x, B, cum2, dtT, dS, none, err, st, xabs, pdl);
}

int64_t fused_flag_words(const Dims& dq) {
    const Dims d = tc_view(dq);
    const int64_t n_tiles = d.N > 128 ? d.N / 128 : 1;
    return d.b * d.H * n_tiles * d.nc;
}

cudaError_t launch_chunk_state_pass_tc(const Dims& dq, const void* x, const void* B,
                                       const float* cum2, const float* dtT, const float* init,
                                       float* carry, int32_t* flags, int32_t* ticket,
                                       void* Sprev, float* final_state, int32_t* err,
                                       cudaStream_t st) {
    const Dims d = tc_view(dq);
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    if (!tc_fused_supported(d) || d.b > (1 << 20)) return cudaErrorInvalidValue;
    FuseArgs fa;
    fa.init = init;
    fa.carry = carry;
    fa.flags = flags;
    fa.ticket = ticket;
    fa.Sprev = static_cast<__nv_bfloat16*>(Sprev);
    fa.fin = final_state;
    fa.nb = (int)d.b;
    return d.L == 256 ? launch_k2<256, true, false>(d, x, B, cum2, dtT, nullptr, fa, err, st)
                      : launch_k2<128, true, false>(d, x, B, cum2, dtT, nullptr, fa, err, st);
}

}  // namespace m2
