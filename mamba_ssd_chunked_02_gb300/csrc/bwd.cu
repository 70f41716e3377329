// bwd.cu -- backward pass of the SSD in the chunked form: the orchestration
// around the forward's stage 2 and stage 4 kernels, and the kernels between them.
//
// The pages give no backward method; they only note that end-to-end training
// speed also depends on one ("NVIDIA、cuTileでMamba-2フォワードパスを高速化"
// (ai.newsbites.today), "開発現場への影響と未確認事項"; "NVIDIA CUDA Tile로 Mamba-2
// 순방향 전달 커널 가속화" (devin.kr), "성능 벤치마크 결과 및 활용").  What is
// computed here is the chain rule applied to the chunked forward of the same
// pages ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile" (brifing.si), sections 4, 5, 8 and 9), so that it equals
// the gradient of the token-by-token recurrence.
//
// Notation for one (b, h) and chunk c with Lc tokens i, j (chunk-local), the
// forward's log2-scaled chunk-local cumsum c2_i, e_i = exp2(c2_i), the chunk
// decay E = exp2(c2_last), w_j = dt_j exp2(c2_last - c2_j), the state entering
// the chunk Sprev, the state leaving it S_after, and Gn, the adjoint of S_after:
//
//   forward:  y_i = sum_{j<=i} CB_ij exp2(c2_i - c2_j) dt_j x_j + e_i Sprev C_i + D x_i
//             S_after = E Sprev + sum_j w_j x_j B_j^T
//   adjoint of the state entering chunk c (reverse pass over chunks):
//             dSprev_c = sum_i e_i dy_i C_i^T + E_c dSprev_{c+1},  dSprev_nc = dfinal
//             Gn_c = dSprev_{c+1},  dinitial_state = dSprev_0
//   dx and the decay terms come from the forward's own output kernel run
//   backwards in time, with B and C swapped, dt' = 1 and Gn as the carried state:
//             y'_j = sum_{i>=j} (B_j.C_i) exp2(c2_i - c2_j) dy_i + exp2(c2_last - c2_j) Gn B_j
//   On the tensor cores (dx mode) stage 4 runs this anti-causal form directly,
//   in token order; elsewhere it runs causally on each chunk's tokens reversed
//   (cum2' = c2_last - c2).  Then
//     dx_j   = dt_j y'_j + D dy_j
//     ddt_j  = x_j.y'_j + A sum_{i>=j} dcum_i
//     dcum_i = dy_i.(y_i - D x_i) - dt_i x_i.y'_i + [i = last] <Gn, S_after>
//     dA     = sum over (b, chunks, j) of dt_j sum_{i>=j} dcum_i
//     dD     = sum over (b, t) of dy . x
//   (dcum is the gradient with respect to the natural-log cumsum, cum_t = A sum dt:
//   the row and column sums of dCB (.) CB (.) decay collapse into the two dots.)
//   The group gradients (summed over the group's heads) are forward-output
//   runs too, with the state
//   transposed: dC_i = sum_h S_i^T dy_i (S_i the state after token i) is stage 4
//   with x'' = B, B'' = x, C'' = dy and carried state Sprev^T; dB_j =
//   sum_h dt_j G_j^T x_j (G_j the adjoint of S_j) is the reversed run with
//   x'' = C, B'' = dy, C'' = x and carried state Gn^T.  In both, the N columns of
//   the output are split into Q = N/64 heads of 64 (the tensor-core shape), so a
//   run has Q*H heads in H groups of Q, and the head sum follows.  On the
//   tensor-core path (bf16, P = 64) dC and dB instead come from bwd_bc_tc.cu:
//   B (or C) is shared by the group's heads, so one kernel loops over the heads
//   and sums them in its accumulator, reading x, dy, B, C, Sprev and Gn as they
//   are (dB anti-causal, in token order).
//
// Kernels, after the forward's stages 1-3 recompute cum2, dtT, Sprev and the
// final state:
//   (stage 4)           y without the skip term
//   (stage 2)           sum_i e_i dy_i C_i^T per (b, c, h) -> dSout: stage 2's
//                       tensor-core kernel in its adjoint weight mode, or
//                       bwd_chunk_adjoint where the shape does not allow it
//   bwd_state_pass_rev  reverse pass over chunks, in place            -> Gn, dinit
//   bwd_prep            the reordered inputs of the runs that need them (reversed
//                       chunks, per-head copies of B and C, cum2' and dt' rows;
//                       none in dx mode with dC / dB from bwd_bc_tc)
//   bwd_transpose       Sprev^T and Gn^T
//   (stage 4)           y' (fp32), or on the tensor cores (dx mode, anti-causal in
//                       token order) dx itself and the per-token dots x . y', dy . x
//   bwd_bc_tc (2 runs)  dC and dB, summed over the heads in the kernel (tensor
//                       cores: bf16, P = 64, L in {128, 256}, N in {64, 128, 256})
//   (stage 4, 2 runs)   otherwise the dC run and the dB run (per-head outputs in
//                       the I/O type, or added into dC / dB on the tensor cores)
//   bwd_token           per (b, c, h): dx (unless the y' run wrote it), ddt, and
//                       dA, dD partial sums
//   bwd_bc_reduce       dC and dB summed over each group's heads (CUDA-core runs)
// bwd_chunk_adjoint's contraction goes through mm_tile, a 64x64 fp32 tile on
// 256 threads (4x4 outputs each) with operands staged through shared memory.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kT = 64;         // tile edge (tokens, p, n)
constexpr int kK = 16;         // k per shared-memory stage
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 outputs each

struct MMSmem {
    float a[2][kK][kT + 4];
    float b[2][kK][kT + 4];
};

// acc[r][q] += sum_{k in [k0, k1)} A(4 ty + r, k) * B(k, 4 tx + q), with
// ty = threadIdx.x / 16, tx = threadIdx.x % 16.  fa(m, k) / fb(k, n) return the
// operand elements (0 outside the operand); AK / BK: the operand is contiguous
// in memory along k (else along m / n), which sets the load order so that
// neighbouring threads read neighbouring addresses.  Two shared-memory stages:
// the next 16 k are fetched into registers while the current ones are used.
// Every thread of the block must call it; it synchronises on entry (after the
// first fetch) and on exit, so shared memory the functors read may be written
// right before the call and rewritten right after it.
template <bool AK, bool BK, class FA, class FB>
__device__ __forceinline__ void mm_tile(float (&acc)[4][4], MMSmem& s, int k0, int k1, FA fa,
                                        FB fb) {
    if (k0 >= k1) return;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float ra[4], rb[4];
    auto fetch = [&](int kb) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = tid + kThreads * r;
            const int am = AK ? (e >> 4) : (e & 63), ak = AK ? (e & 15) : (e >> 6);
            const int bn = BK ? (e >> 4) : (e & 63), bk = BK ? (e & 15) : (e >> 6);
            ra[r] = (kb + ak < k1) ? fa(am, kb + ak) : 0.f;
            rb[r] = (kb + bk < k1) ? fb(kb + bk, bn) : 0.f;
        }
    };
    auto put = [&](int buf) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = tid + kThreads * r;
            const int am = AK ? (e >> 4) : (e & 63), ak = AK ? (e & 15) : (e >> 6);
            const int bn = BK ? (e >> 4) : (e & 63), bk = BK ? (e & 15) : (e >> 6);
            s.a[buf][ak][am] = ra[r];
            s.b[buf][bk][bn] = rb[r];
        }
    };
    fetch(k0);
    put(0);
    __syncthreads();
    int buf = 0;
    for (int kb = k0; kb < k1; kb += kK) {
        const bool more = kb + kK < k1;
        if (more) fetch(kb + kK);
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(&s.a[buf][k][4 * ty]);
            const float4 b = *reinterpret_cast<const float4*>(&s.b[buf][k][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
        }
        if (more) put(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }
}

__device__ __forceinline__ void zero(float (&acc)[4][4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
}

// Sum over the block (256 threads); `red` holds 8 floats; the result is
// returned to every thread.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    return s;
}

// Suffix sum over the block: thread j gets sum_{k >= j} v_k.  `red` holds 8 floats.
__device__ __forceinline__ float block_suffix_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_down_sync(0xffffffffu, s, o);
        if (lane + o < 32) s += n;
    }
    __syncthreads();
    if (lane == 0) red[warp] = s;   // the warp's total
    __syncthreads();
    for (int w = warp + 1; w < kThreads / 32; ++w) s += red[w];
    return s;
}

struct BwdArgs {
    const void* x;      // [b,T,H,P] TI
    const void* B;      // [b,T,G,N] TI
    const void* C;      // [b,T,G,N] TI
    const void* dy;     // [b,T,H,P] TI
    const float* A;     // [H]
    const float* D;     // [H] or null
    const float* cum2;  // [b,H,T]
    const float* dtT;   // [b,H,T]
    const void* Sprev;  // [b,nc,H,P,N] TI (the state entering each chunk)
    const float* fin;   // [b,H,P,N] fp32 (the final state)
    float* Gn;          // [b,nc,H,P,N] fp32: dSout, then Gn
    void* GnIO;         // [b,nc,H,P,N] TI copy of Gn (stage 4's carried-state operand)
    const float* yno;   // [b,T,H,P] fp32: y without the skip term (or null: ydot2)
    const float* ydot2; // [b,H,T,2] fp32: partial sums of dy . y without the skip term, or null
    const float* yr;    // [b,T,H,P] fp32: y' with each chunk's tokens reversed (or null:
                        // the y' run wrote dx and the dots below itself)
    float* xyd;         // [b,H,T,2] fp32: partial sums of x . y' (with ydot2), or null
    float* dyxd;        // [b,H,T,2] fp32: partial sums of dy . x (with ydot2), or null
    float* dx;          // [b,T,H,P]
    float* ddt;         // [b,T,H]
    float* dA;          // [H] (accumulated)
    float* dD;          // [H] (accumulated) or null
    float* dB;          // [b,T,G,N]
    float* dC;          // [b,T,G,N]
    int T, H, P, N, G, L, nc;
    int gn16;           // tensor-core path: adjoints in bf16 in Gn's buffer, Gn only in GnIO
};

// --- dSout[b,c,h] = sum_i e_i dy_i C_i^T  (P x N).  Grid: b*nc*H * ceil(P/64) * ceil(N/64).
template <typename TI>
__global__ void __launch_bounds__(kThreads) bwd_chunk_adjoint(BwdArgs a) {
    __shared__ MMSmem sm;
    __shared__ float s_e[256];
    const int npt = (a.P + kT - 1) / kT, nnt = (a.N + kT - 1) / kT;
    int id = blockIdx.x;
    const int nt = id % nnt; id /= nnt;
    const int pt = id % npt; id /= npt;
    const int h = id % a.H; id /= a.H;
    const int c = id % a.nc, b = id / a.nc;
    const int g = h / (a.H / a.G);
    const int64_t t0 = (int64_t)c * a.L;
    const int Lc = (int)min((int64_t)a.L, a.T - t0);
    const float* c2 = a.cum2 + ((int64_t)b * a.H + h) * a.T + t0;
    for (int i = threadIdx.x; i < a.L; i += kThreads) s_e[i] = i < Lc ? ex2(c2[i]) : 0.f;
    __syncthreads();
    const TI* dy = static_cast<const TI*>(a.dy) + ((int64_t)b * a.T + t0) * a.H * a.P + (int64_t)h * a.P;
    const TI* C = static_cast<const TI*>(a.C) + ((int64_t)b * a.T + t0) * a.G * a.N + (int64_t)g * a.N;
    const int64_t sdy = (int64_t)a.H * a.P, sC = (int64_t)a.G * a.N;
    const int P = a.P, N = a.N;
    float acc[4][4];
    zero(acc);
    mm_tile<false, false>(
        acc, sm, 0, Lc,
        [&](int m, int k) {
            const int p = pt * kT + m;
            return p < P ? s_e[k] * to_f32(dy[k * sdy + p]) : 0.f;
        },
        [&](int k, int n) {
            const int nn = nt * kT + n;
            return nn < N ? to_f32(C[k * sC + nn]) : 0.f;
        });
    float* out = a.Gn + (((int64_t)b * a.nc + c) * a.H + h) * (int64_t)P * N;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int p = pt * kT + 4 * ty + r;
        if (p >= P) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int nn = nt * kT + 4 * tx + q;
            if (nn < N) out[(int64_t)p * N + nn] = acc[r][q];
        }
    }
}

// --- Reverse pass over chunks, in place: buf[c] holds dSout_c on entry and
// Gn_c = dSprev_{c+1} on exit (and in the I/O type in gio, unless TI is fp32);
// dinit = dSprev_0.  One thread per (b, h) and four consecutive (p, n); the
// loads of four chunks are issued before their values are used (the chain
// through the chunks is the only dependence).
template <typename TI>
__global__ void __launch_bounds__(kThreads)
bwd_state_pass_rev(float4* __restrict__ buf, TI* __restrict__ gio, const float* __restrict__ cum2,
                   const float4* __restrict__ dfinal, float4* __restrict__ dinit, int64_t total4,
                   int H, int64_t PN4, int T, int L, int nc, const uint2* __restrict__ adj16) {
    // adj16: the chunk adjoints in bf16 (four per 8 bytes); then only the I/O-type
    // copy of Gn is written (buf unused).  Else adjoints and Gn in fp32 in buf.
    constexpr int kU = 4;
    for (int64_t idx = blockIdx.x * (int64_t)kThreads + threadIdx.x; idx < total4;
         idx += (int64_t)gridDim.x * kThreads) {
        const int64_t k = idx % PN4, bh = idx / PN4;
        const int64_t b = bh / H, h = bh % H;
        float4 gv = dfinal ? dfinal[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float* c2 = cum2 + bh * T;
        for (int c0 = nc - 1; c0 >= 0; c0 -= kU) {
            float4 v[kU];
            float dec[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = c0 - u;
                if (c >= 0) {
                    const int64_t o = ((b * nc + c) * H + h) * PN4 + k;
                    if (adj16) {
                        const uint2 q = adj16[o];
                        v[u] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                           __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
                    } else {
                        v[u] = buf[o];
                    }
                    dec[u] = ex2(c2[min(T, (c + 1) * L) - 1]);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = c0 - u;
                if (c >= 0) {
                    const int64_t o = ((b * nc + c) * H + h) * PN4 + k;
                    if (!adj16) buf[o] = gv;
                    if constexpr (sizeof(TI) == 2) {   // one 8-byte store of the four bf16
                        TI q[4] = {from_f32<TI>(gv.x), from_f32<TI>(gv.y), from_f32<TI>(gv.z),
                                   from_f32<TI>(gv.w)};
                        *reinterpret_cast<uint2*>(gio + 4 * o) = *reinterpret_cast<const uint2*>(q);
                    }
                    gv.x = fmaf(dec[u], gv.x, v[u].x);
                    gv.y = fmaf(dec[u], gv.y, v[u].y);
                    gv.z = fmaf(dec[u], gv.z, v[u].z);
                    gv.w = fmaf(dec[u], gv.w, v[u].w);
                }
            }
        }
        if (dinit) dinit[idx] = gv;
    }
}

// The same reverse pass for bf16 chunk adjoints and a bf16 Gn (the tensor-core
// path), laid out like the forward's state pass: one thread owns 8 consecutive
// state elements (16 bytes of bf16) of one (b, h) for the whole chain, and keeps
// kDepth chunks of adjoint loads in flight (a rolling prefetch, issued for chunk
// c - kDepth as chunk c is consumed), so the pass is one HBM stream of adjoints
// in and Gn out.
constexpr int kRevDepth = 4;

__global__ void __launch_bounds__(kThreads)
bwd_state_pass_rev16(const __nv_bfloat16* __restrict__ adj, __nv_bfloat16* __restrict__ gio,
                     const float* __restrict__ cum2, const float* __restrict__ dfinal,
                     float* __restrict__ dinit, int T, int H, int L, int nc, int64_t PN,
                     int64_t blocks_per_bh) {
    const int64_t bh = blockIdx.x / blocks_per_bh;
    const int64_t e = ((blockIdx.x % blocks_per_bh) * kThreads + threadIdx.x) * 8;
    if (e >= PN) return;
    const int64_t b = bh / H, h = bh % H;
    float S[8];
    if (dfinal) {
        const float4 f0 = *reinterpret_cast<const float4*>(dfinal + bh * PN + e);
        const float4 f1 = *reinterpret_cast<const float4*>(dfinal + bh * PN + e + 4);
        S[0] = f0.x; S[1] = f0.y; S[2] = f0.z; S[3] = f0.w;
        S[4] = f1.x; S[5] = f1.y; S[6] = f1.z; S[7] = f1.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) S[k] = 0.f;
    }
    const float* crow = cum2 + bh * T;
    const int64_t cstride = (int64_t)H * PN;                       // chunk stride
    const int64_t base = ((b * nc + (nc - 1)) * H + h) * PN + e;   // [b, c = nc-1, h, e]
    // Chunk c's decay is exp2 of its last token's cum2 (the sequence end for a ragged last chunk).
    auto last_c2 = [&](int c) { return __ldg(crow + (min(T, (c + 1) * L) - 1)); };
    uint4 buf[kRevDepth];
    float cl[kRevDepth];
#pragma unroll
    for (int u = 0; u < kRevDepth; ++u) {
        const int c = nc - 1 - u;
        if (c >= 0) {
            buf[u] = __ldcs(reinterpret_cast<const uint4*>(adj + base - u * cstride));
            cl[u] = last_c2(c);
        }
    }
    for (int c0 = nc - 1; c0 >= 0; c0 -= kRevDepth) {
#pragma unroll
        for (int u = 0; u < kRevDepth; ++u) {
            const int c = c0 - u;
            if (c >= 0) {
                const uint4 q = buf[u];
                const float dec = ex2(cl[u]);
                const int64_t o = base - (int64_t)(nc - 1 - c) * cstride;
                if (c - kRevDepth >= 0) {
                    buf[u] = __ldcs(reinterpret_cast<const uint4*>(adj + o - kRevDepth * cstride));
                    cl[u] = last_c2(c - kRevDepth);
                }
                // Gn of chunk c: the adjoint of the state leaving it, before chunk c's own term.
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __nv_bfloat162 t = __floats2bfloat162_rn(S[2 * k], S[2 * k + 1]);
                    w[k] = *reinterpret_cast<uint32_t*>(&t);
                }
                *reinterpret_cast<uint4*>(gio + o) = make_uint4(w[0], w[1], w[2], w[3]);
                const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    S[2 * k] = fmaf(dec, S[2 * k], __uint_as_float(qv[k] << 16));
                    S[2 * k + 1] = fmaf(dec, S[2 * k + 1], __uint_as_float(qv[k] & 0xffff0000u));
                }
            }
        }
    }
    if (dinit) {
        *reinterpret_cast<float4*>(dinit + bh * PN + e) = make_float4(S[0], S[1], S[2], S[3]);
        *reinterpret_cast<float4*>(dinit + bh * PN + e + 4) = make_float4(S[4], S[5], S[6], S[7]);
    }
}

// --- Inputs of the three stage-4 runs, one CTA per (token t, b).  Token k of
// chunk c (Lc tokens) is reversed to position Lc-1-k of the same chunk.
//   y' run (H heads):         dyr = dy reversed, Br = C reversed, Cr = B reversed,
//                             cum2r = c2_last - c2 (reversed), ones
//   dC run (Q*H heads of N/Q): xB[h] = B of the head's group
//   dB run (Q*H heads, reversed): xCr[h] = C of the group reversed, xr = x reversed
//   per (Q*H)-head rows: cum2d, dtTd (natural order), cum2rd, onesd (reversed).
struct PrepArgs {
    const void *dy, *B, *C, *x;
    const float *cum2, *dtT;
    void *dyr, *Br, *Cr, *xB, *xCr, *xr;
    float *cum2r, *ones, *cum2d, *dtTd, *cum2rd, *onesd;
    int T, H, G, P, N, L, Q;
    int copies;   // write xB, xCr and the per-(Q*H)-head rows (the CUDA-core dC / dB runs)
    int with_xr;  // write xr (not needed when dC and dB come from bwd_bc_tc)
    int with_cr;  // write cum2r and ones, and dyr, Br, Cr (the reversed y' run; not in dx mode,
                  // whose y' run is anti-causal on dy, B and C as they are)
};

template <typename TI>
__global__ void __launch_bounds__(kThreads) bwd_prep(PrepArgs a) {
    const int t = blockIdx.x, b = blockIdx.y;
    const int c = t / a.L, k = t - c * a.L;
    const int Lc = min(a.L, a.T - c * a.L);
    const int ts = c * a.L + (Lc - 1 - k);   // the source token of reversed position t
    const int hpg = a.H / a.G;
    // Rows are 16-byte multiples (P, N >= 16 elements) at 16-byte aligned starts.
    // Four of a thread's 16-byte loads are in flight before their stores.
    auto copy = [&](const void* src, int64_t srow, void* dst, int64_t drow, int64_t n16) {
        const uint4* __restrict__ s4 = reinterpret_cast<const uint4*>(static_cast<const TI*>(src) + srow);
        uint4* __restrict__ d4 = reinterpret_cast<uint4*>(static_cast<TI*>(dst) + drow);
        for (int64_t i0 = threadIdx.x; i0 < n16; i0 += 4 * kThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * kThreads < n16) v[u] = s4[i0 + u * kThreads];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * kThreads < n16) d4[i0 + u * kThreads] = v[u];
        }
    };
    const int64_t rowx = (int64_t)a.H * a.P, rowbc = (int64_t)a.G * a.N, rowhn = (int64_t)a.H * a.N;
    const int64_t E = sizeof(TI);
    const int64_t bt = (int64_t)b * a.T;
    if (a.with_cr) copy(a.dy, (bt + ts) * rowx, a.dyr, (bt + t) * rowx, rowx * E / 16);
    if (a.copies) {
        copy(a.x, (bt + ts) * rowx, a.xr, (bt + t) * rowx, rowx * E / 16);
    } else if (a.with_xr) {
        // The tensor-core dB run adds dt_h[t] * (its row) into dB: its C operand is
        // x reversed, each head's row scaled by dt of the source token.
        constexpr int V = 16 / sizeof(TI);
        const int pv = a.P / V;                          // 16-byte pieces per head row
        const uint4* s4 = reinterpret_cast<const uint4*>(static_cast<const TI*>(a.x) + (bt + ts) * rowx);
        uint4* d4 = reinterpret_cast<uint4*>(static_cast<TI*>(a.xr) + (bt + t) * rowx);
        for (int64_t i = threadIdx.x; i < rowx / V; i += kThreads) {
            const int h = (int)(i / pv);
            const float w = a.dtT[((int64_t)b * a.H + h) * a.T + ts];
            uint4 q = s4[i];
            TI* e = reinterpret_cast<TI*>(&q);
#pragma unroll
            for (int v = 0; v < V; ++v) e[v] = from_f32<TI>(w * to_f32(e[v]));
            d4[i] = q;
        }
    }
    if (a.with_cr) {
        copy(a.C, (bt + ts) * rowbc, a.Br, (bt + t) * rowbc, rowbc * E / 16);
        copy(a.B, (bt + ts) * rowbc, a.Cr, (bt + t) * rowbc, rowbc * E / 16);
    }
    for (int h = threadIdx.x; a.with_cr && h < a.H; h += kThreads) {
        const float* c2 = a.cum2 + ((int64_t)b * a.H + h) * a.T;
        const int64_t o = ((int64_t)b * a.H + h) * a.T + t;
        a.cum2r[o] = c2[c * a.L + Lc - 1] - c2[ts];
        a.ones[o] = 1.f;
    }
    if (!a.copies) return;   // the tensor-core runs read B, Br, cum2, dtT, cum2r, ones directly
    // Per-head copies of the group's B (natural order) and C (reversed).
    {
        const int64_t n16 = (int64_t)a.N * E / 16;
        const uint4* Bs = reinterpret_cast<const uint4*>(static_cast<const TI*>(a.B) + (bt + t) * rowbc);
        const uint4* Cs = reinterpret_cast<const uint4*>(static_cast<const TI*>(a.C) + (bt + ts) * rowbc);
        uint4* xb = reinterpret_cast<uint4*>(static_cast<TI*>(a.xB) + (bt + t) * rowhn);
        uint4* xc = reinterpret_cast<uint4*>(static_cast<TI*>(a.xCr) + (bt + t) * rowhn);
        for (int64_t i = threadIdx.x; i < a.H * n16; i += kThreads) {
            const int64_t h = i / n16, e = i - h * n16;
            const int64_t src = (h / hpg) * n16 + e;
            xb[i] = Bs[src];
            xc[i] = Cs[src];
        }
    }
    for (int hq = threadIdx.x; hq < a.Q * a.H; hq += kThreads) {
        const int h = hq / a.Q;
        const float* c2 = a.cum2 + ((int64_t)b * a.H + h) * a.T;
        const int64_t o = ((int64_t)b * a.Q * a.H + hq) * a.T + t;
        a.cum2d[o] = c2[t];
        a.dtTd[o] = a.dtT[((int64_t)b * a.H + h) * a.T + t];
        a.cum2rd[o] = c2[c * a.L + Lc - 1] - c2[ts];
        a.onesd[o] = 1.f;
    }
}

// --- Batched transpose of P x N blocks into N x P blocks (I/O type out).
// One CTA per (block, 32 x 32 tile).
template <typename TS, typename TI>
__global__ void __launch_bounds__(kThreads)
bwd_transpose(const TS* __restrict__ in, TI* __restrict__ out, int P, int N) {
    __shared__ float tile[32][33];
    const int ntn = (N + 31) / 32, ntp = (P + 31) / 32;
    const int64_t blk = blockIdx.x / (ntn * ntp);
    const int tn = (blockIdx.x % (ntn * ntp)) % ntn, tp = (blockIdx.x % (ntn * ntp)) / ntn;
    const TS* src = in + blk * (int64_t)P * N;
    TI* dst = out + blk * (int64_t)P * N;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (int r = ty; r < 32; r += 8) {
        const int p = tp * 32 + r, n = tn * 32 + tx;
        if (p < P && n < N) tile[r][tx] = to_f32(src[(int64_t)p * N + n]);
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int n = tn * 32 + r, p = tp * 32 + tx;
        if (p < P && n < N) dst[(int64_t)n * P + p] = from_f32<TI>(tile[tx][r]);
    }
}

// --- dC and dB from the two transposed-state runs (their per-head outputs in
// the I/O type), summed over each group's heads in fp32: dC[t] = sum_h yC[h, t];
// dB[t] = sum_h dt_h[t] zB[h, reversed t].  One CTA per (token, b).
template <typename TI>
__global__ void __launch_bounds__(kThreads)
bwd_bc_reduce(const TI* __restrict__ yC, const TI* __restrict__ zB,
              const float* __restrict__ dtT, float* __restrict__ dB, float* __restrict__ dC,
              int T, int H, int G, int N, int L, int with_dc) {
    const int t = blockIdx.x, b = blockIdx.y;
    const int c = t / L, k = t - c * L;
    const int Lc = min(L, T - c * L);
    const int tr = c * L + (Lc - 1 - k);   // where the reversed run wrote token t
    const int hpg = H / G;
    const int64_t rowhn = (int64_t)H * N, bt = (int64_t)b * T;
    const TI* yc = yC + (bt + t) * rowhn;
    const TI* zb = zB + (bt + tr) * rowhn;
    for (int e = threadIdx.x; e < G * N; e += kThreads) {
        const int g = e / N, n = e - g * N;
        float sc = 0.f, sb = 0.f;
        for (int hh = 0; hh < hpg; ++hh) {
            const int h = g * hpg + hh;
            if (with_dc) sc += to_f32(yc[(int64_t)h * N + n]);
            sb = fmaf(dtT[((int64_t)b * H + h) * T + t], to_f32(zb[(int64_t)h * N + n]), sb);
        }
        if (with_dc) dC[(bt + t) * (int64_t)G * N + e] = sc;
        dB[(bt + t) * (int64_t)G * N + e] = sb;
    }
}


// Elements 2 pp and 2 pp + 1 of a row, as floats (4- or 8-byte load).
__device__ __forceinline__ float2 load_pair(const float* __restrict__ p, int pp) {
    return reinterpret_cast<const float2*>(p)[pp];
}
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* __restrict__ p, int pp) {
    return __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(p)[pp]);
}

// --- Per (b, c, h): dx, ddt and the dA, dD partial sums from y' (reversed) and
// y without the skip term.  A warp per token, lanes over p.  Grid: b*nc*H.
template <typename TI>
__global__ void __launch_bounds__(kThreads) bwd_token(BwdArgs a) {
    __shared__ float s_dt[256], s_dcum[256], s_ddt[256];
    __shared__ float red[kThreads / 32];
    int id = blockIdx.x;
    const int h = id % a.H; id /= a.H;
    const int c = id % a.nc, b = id / a.nc;
    const int P = a.P, N = a.N, L = a.L;
    const int64_t t0 = (int64_t)c * L;
    const int Lc = (int)min((int64_t)L, a.T - t0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t PN = (int64_t)P * N;
    // This thread's token (L <= kThreads: one token per thread): its dt and, when
    // the y' run wrote them, its three dot pairs, loaded before the chunk dot below
    // so that their latency overlaps it.
    const float* dth = a.dtT + ((int64_t)b * a.H + h) * a.T + t0;
    const float pre_dt = tid < Lc ? dth[tid] : 0.f;
    float2 pre_xy = make_float2(0.f, 0.f), pre_dyx = pre_xy, pre_yd = pre_xy;
    if (a.xyd && tid < Lc) {
        const int64_t po = (((int64_t)b * a.H + h) * a.T + t0) * 2;
        pre_xy = reinterpret_cast<const float2*>(a.xyd + po)[tid];
        pre_dyx = reinterpret_cast<const float2*>(a.dyxd + po)[tid];
        pre_yd = reinterpret_cast<const float2*>(a.ydot2 + po)[tid];
    }
    // <Gn_c, S_after_c>: S_after is the next chunk's Sprev, or the final state.
    float gs = 0.f;
    {
        const int64_t go = (((int64_t)b * a.nc + c) * a.H + h) * PN;
        const float* Gn = a.Gn + go;
        const TI* G16 = static_cast<const TI*>(a.GnIO) + go;   // when only the I/O-type Gn exists
        bool done = false;
        if constexpr (sizeof(TI) == 2) {
            if (a.gn16) {   // 16-byte loads: eight bf16 of Gn (and of Sprev) at a time (PN % 8 == 0)
                const uint4* g4 = reinterpret_cast<const uint4*>(G16);
                auto dot8 = [](uint4 g, const float (&s)[8], float acc) {
                    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc = fmaf(__uint_as_float(gw[e] << 16), s[2 * e], acc);
                        acc = fmaf(__uint_as_float(gw[e] & 0xffff0000u), s[2 * e + 1], acc);
                    }
                    return acc;
                };
                if (c + 1 < a.nc) {
                    const uint4* s4 = reinterpret_cast<const uint4*>(
                        static_cast<const TI*>(a.Sprev) + (((int64_t)b * a.nc + c + 1) * a.H + h) * PN);
#pragma unroll 4
                    for (int64_t k8 = tid; k8 < PN / 8; k8 += kThreads) {
                        const uint4 sv = s4[k8];
                        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
                        float sf[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            sf[2 * e] = __uint_as_float(sw[e] << 16);
                            sf[2 * e + 1] = __uint_as_float(sw[e] & 0xffff0000u);
                        }
                        gs = dot8(g4[k8], sf, gs);
                    }
                } else {
                    const float4* f4 = reinterpret_cast<const float4*>(a.fin + ((int64_t)b * a.H + h) * PN);
                    for (int64_t k8 = tid; k8 < PN / 8; k8 += kThreads) {
                        const float4 f0 = f4[2 * k8], f1 = f4[2 * k8 + 1];
                        const float sf[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                        gs = dot8(g4[k8], sf, gs);
                    }
                }
                done = true;
            }
        }
        if (!done) {
            auto gn = [&](int64_t k) { return a.gn16 ? to_f32(G16[k]) : Gn[k]; };
            if (c + 1 < a.nc) {
                const TI* Sa = static_cast<const TI*>(a.Sprev) + (((int64_t)b * a.nc + c + 1) * a.H + h) * PN;
                for (int64_t k = tid; k < PN; k += kThreads) gs = fmaf(gn(k), to_f32(Sa[k]), gs);
            } else {
                const float* Sa = a.fin + ((int64_t)b * a.H + h) * PN;
                for (int64_t k = tid; k < PN; k += kThreads) gs = fmaf(gn(k), Sa[k], gs);
            }
        }
    }
    s_dt[tid] = pre_dt;   // kThreads = 256 slots
    __syncthreads();
    const float Dh = a.D ? a.D[h] : 0.f;
    const int64_t sxy = (int64_t)a.H * P;
    const int64_t base = ((int64_t)b * a.T + t0) * sxy + (int64_t)h * P;
    const TI* __restrict__ x = static_cast<const TI*>(a.x) + base;
    const TI* __restrict__ dy = static_cast<const TI*>(a.dy) + base;
    const float* __restrict__ yno = a.ydot2 ? nullptr : a.yno + base;
    const float* __restrict__ yd = a.ydot2 ? a.ydot2 + (((int64_t)b * a.H + h) * a.T + t0) * 2 : nullptr;
    float yx = 0.f;
    if (a.xyd) {
        // The y' run wrote dx and the per-token dots x . y' and dy . x (this
        // thread's token's, loaded above).
        if (tid < Lc) {
            const float xy = pre_xy.x + pre_xy.y;
            s_ddt[tid] = xy;
            s_dcum[tid] = (pre_yd.x + pre_yd.y) - pre_dt * xy;
            yx += pre_dyx.x + pre_dyx.y;
        }
    } else {
    const float* __restrict__ yr = a.yr + base;
    float* __restrict__ dx = a.dx + base;
    // Four tokens per warp per iteration (j0 + 8 u), p in pairs (8-byte loads),
    // all of an iteration's loads issued before their values are used.
    constexpr int kW = kThreads / 32, kU = 4;
    const int P2 = P / 2;   // P is even
    for (int j0 = warp; j0 < Lc; j0 += kU * kW) {
        float xy[kU], dyy[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            xy[u] = 0.f;
            dyy[u] = 0.f;
            const int j = j0 + u * kW;
            if (j >= Lc) continue;
            const int jr = Lc - 1 - j;   // where the reversed run wrote token j
            const float dtj = s_dt[j];
            for (int pp = lane; pp < P2; pp += 32) {
                const float2 yp = reinterpret_cast<const float2*>(yr + jr * sxy)[pp];
                const float2 yn = yno ? reinterpret_cast<const float2*>(yno + j * sxy)[pp] : make_float2(0.f, 0.f);
                const float2 xv = load_pair(x + j * sxy, pp);
                const float2 dv = load_pair(dy + j * sxy, pp);
                reinterpret_cast<float2*>(dx + j * sxy)[pp] =
                    make_float2(fmaf(dtj, yp.x, Dh * dv.x), fmaf(dtj, yp.y, Dh * dv.y));
                xy[u] = fmaf(xv.x, yp.x, fmaf(xv.y, yp.y, xy[u]));
                dyy[u] = fmaf(dv.x, yn.x, fmaf(dv.y, yn.y, dyy[u]));
                yx = fmaf(dv.x, xv.x, fmaf(dv.y, xv.y, yx));
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                xy[u] += __shfl_xor_sync(0xffffffffu, xy[u], o);
                dyy[u] += __shfl_xor_sync(0xffffffffu, dyy[u], o);
            }
            const int j = j0 + u * kW;
            if (lane == 0 && j < Lc) {
                s_ddt[j] = xy[u];
                const float dsum = yd ? yd[2 * j] + yd[2 * j + 1] : dyy[u];
                s_dcum[j] = dsum - s_dt[j] * xy[u];
            }
        }
    }
    }
    gs = block_sum(gs, red);
    yx = block_sum(yx, red);   // (its barriers also publish s_ddt / s_dcum)
    if (tid == 0) s_dcum[Lc - 1] += gs;
    __syncthreads();
    const int j = tid;
    const float rcs = block_suffix_sum(j < Lc ? s_dcum[j] : 0.f, red);
    float da = 0.f;
    if (j < Lc) {
        a.ddt[((int64_t)b * a.T + t0 + j) * a.H + h] = fmaf(a.A[h], rcs, s_ddt[j]);
        da = s_dt[j] * rcs;
    }
    da = block_sum(da, red);
    if (tid == 0) {
        atomicAdd(a.dA + h, da);
        if (a.dD) atomicAdd(a.dD + h, yx);
    }
}

template <typename TI>
cudaError_t launch_t(const Dims& d, const BwdArgs& a, const BwdWork& w, bool tc,
                     const float* dfinal, float* dinit, int32_t* err, cudaStream_t st) {
    const int64_t bnc = d.b * d.nc;
    const int npt = (int)((d.P + kT - 1) / kT), nnt = (int)((d.N + kT - 1) / kT);
    const int64_t g1 = bnc * d.H * npt * nnt;
    const int64_t g4 = bnc * d.H;
    const int64_t ntile = ((d.P + 31) / 32) * ((d.N + 31) / 32);
    const int64_t gt = bnc * d.H * ntile;
    if (g1 >= (int64_t(1) << 31) || g4 >= (int64_t(1) << 31) || gt >= (int64_t(1) << 31) ||
        d.T >= (int64_t(1) << 31) || d.b >= 65536)
        return cudaErrorInvalidValue;
    // Stage 4 with y in fp32 (y32) or the I/O type (tensor cores where the shape
    // allows them; the CUDA-core kernel otherwise or where the fp32 variant's
    // staging does not fit).
    auto out4 = [&](const Dims& dd, const void* x4, const void* B4, const void* C4, const float* c4,
                    const float* d4, const void* S4, const void* y4, bool y32) {
        void* yo = const_cast<void*>(y4);
        if (tc && tc_supported(dd)) {
            const cudaError_t r = launch_chunk_out_tc(dd, x4, B4, C4, c4, d4, S4, nullptr, yo, err,
                                                      st, nullptr, false, y32);
            if (r != cudaErrorNotSupported) return r;
        }
        return launch_chunk_out_simt(dd, x4, B4, C4, c4, d4, S4, nullptr, yo, err, st, y32);
    };
    // y without the skip term (fp32: its dots with dy set the decay gradients).
    cudaError_t e;
    if (a.ydot2) {   // the tensor-core y run writes only the dots dy . y the per-token kernel needs
        Dims dd = d;
        dd.ydot_dy = a.dy;
        dd.ydot_out = const_cast<float*>(a.ydot2);
        e = launch_chunk_out_tc(dd, a.x, a.B, a.C, a.cum2, a.dtT, a.Sprev, nullptr, dd.ydot_out, err, st,
                                w.xabs_x, false, true);
    } else {
        e = out4(d, a.x, a.B, a.C, a.cum2, a.dtT, a.Sprev, a.yno, true);
    }
    if (e != cudaSuccess) return e;
    // Chunk adjoints sum_i e_i dy_i C_i^T: stage 2's tensor-core contraction in
    // its adjoint weight mode where the shape allows it.
    if (tc && tc_supported(d)) {
        e = launch_chunk_state_tc(d, a.dy, a.C, a.cum2, a.dtT, a.Gn, a.gn16 != 0, err, st, w.xabs_dy,
                                  false, true);
        if (e != cudaSuccess) return e;
    } else {
        bwd_chunk_adjoint<TI><<<(unsigned)g1, kThreads, 0, st>>>(a);
    }
    bool rev_done = false;
    if constexpr (sizeof(TI) == 2) {
        if (a.gn16) {   // bf16 adjoints in, bf16 Gn out: 8 state elements per thread
            const int64_t PN = d.P * d.N;   // a multiple of 256
            const int64_t bpb = (PN / 8 + kThreads - 1) / kThreads;
            bwd_state_pass_rev16<<<(unsigned)(d.b * d.H * bpb), kThreads, 0, st>>>(
                reinterpret_cast<const __nv_bfloat16*>(a.Gn), reinterpret_cast<__nv_bfloat16*>(a.GnIO), a.cum2,
                dfinal, dinit, (int)d.T, (int)d.H, (int)d.L, (int)d.nc, PN, bpb);
            rev_done = true;
        }
    }
    if (!rev_done) {
        const int64_t total4 = d.b * d.H * d.P * d.N / 4;   // N is a multiple of 16
        const int64_t blocks = std::min<int64_t>((total4 + kThreads - 1) / kThreads, 152 * 16);
        bwd_state_pass_rev<TI><<<(unsigned)blocks, kThreads, 0, st>>>(
            reinterpret_cast<float4*>(a.Gn), static_cast<TI*>(a.GnIO), a.cum2,
            reinterpret_cast<const float4*>(dfinal), reinterpret_cast<float4*>(dinit), total4,
            (int)d.H, d.P * d.N / 4, (int)d.T, (int)d.L, (int)d.nc,
            a.gn16 ? reinterpret_cast<const uint2*>(a.Gn) : nullptr);
    }
    // The dC / dB runs: Q heads of N/Q columns per head (64 wide when N >= 64).
    const int Q = d.N >= 64 ? (int)(d.N / 64) : 1;
    const Dims d2 = bwd_run_dims(d);
    const bool tc2 = tc && tc_supported(d2);
    // dC and dB straight from the inputs, summed over the heads in the kernel.
    const bool bc = tc2 && bwd_bc_tc_supported(d);
    PrepArgs pa{a.dy, a.B, a.C, a.x, a.cum2, a.dtT, w.dyr, w.Br, w.Cr, w.xB, w.xCr, w.xr,
                w.cum2r, w.ones, w.cum2d, w.dtTd, w.cum2rd, w.onesd,
                (int)d.T, (int)d.H, (int)d.G, (int)d.P, (int)d.N, (int)d.L, Q, tc2 ? 0 : 1,
                bc ? 0 : 1, a.xyd ? 0 : 1};
    if (pa.with_cr || pa.with_xr || pa.copies)   // dx mode with dC / dB from bwd_bc_tc needs none
        bwd_prep<TI><<<dim3((unsigned)d.T, (unsigned)d.b), kThreads, 0, st>>>(pa);
    if (!tc2) {   // the tensor-core runs read Sprev and Gn untransposed
        bwd_transpose<TI, TI><<<(unsigned)gt, kThreads, 0, st>>>(static_cast<const TI*>(a.Sprev),
                                                                 static_cast<TI*>(w.SprevT),
                                                                 (int)d.P, (int)d.N);
        bwd_transpose<float, TI><<<(unsigned)gt, kThreads, 0, st>>>(a.Gn, static_cast<TI*>(w.GnT),
                                                                    (int)d.P, (int)d.N);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // y' = stage 4 on the reversed inputs: x' = dy, B' = C, C' = B, Gn carried.
    const void* gio = sizeof(TI) == 2 ? a.GnIO : static_cast<const void*>(a.Gn);
    if (a.xyd) {   // dx mode: the run writes dx and the dots x . y', dy . x instead of y'
        Dims dd = d;
        dd.dxm_x = a.x;
        dd.dxm_dy = a.dy;
        dd.dxm_dt = a.dtT;
        dd.dxm_D = a.D;
        dd.dxm_dx = a.dx;
        dd.dxm_xy = a.xyd;
        dd.dxm_dyx = a.dyxd;
        // Anti-causal in token order: y'_j = sum_{i >= j} (B_j . C_i) exp2(c2_i - c2_j)
        // dy_i + exp2(c2_last - c2_j) Gn B_j, i.e. x'' = dy, B'' = C, C'' = B, dt' = 1.
        dd.dt1 = 1;
        dd.antic = 1;
        e = launch_chunk_out_tc(dd, a.dy, a.C, a.B, a.cum2, a.dtT, gio, nullptr, a.dx, err, st,
                                w.xabs_dy, false, true);
    } else {
        e = out4(d, w.dyr, w.Br, w.Cr, w.cum2r, w.ones, gio, a.yr, true);
    }
    if (e != cudaSuccess) return e;
    // The per-head outputs in the I/O type: the head sum that follows is in fp32.
    const size_t bcbytes = sizeof(float) * (size_t)(d.b * d.T * d.G * d.N);
    if (bc) {
        e = cudaMemsetAsync(a.dC, 0, bcbytes, st);
        if (e == cudaSuccess)
            e = launch_bwd_bc_tc(d, false, a.dy, a.x, a.B, a.Sprev, a.cum2, a.dtT, a.dC, err, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.dB, 0, bcbytes, st);
        if (e == cudaSuccess)
            e = launch_bwd_bc_tc(d, true, a.x, a.dy, a.C, a.GnIO, a.cum2, a.dtT, a.dB, err, st);
    } else if (tc2) {
        // Run head h*Q + q reads columns 64 q .. of its group's B (dC run) or of Br,
        // the group's C reversed (dB run), and cum2 / dt rows of head h.
        Dims dm = d2;
        dm.st_mn = 1;   // Sprev / Gn untransposed: rows of head h, columns 64 q ..
        dm.pts = Q == 4 ? 2 : (Q == 2 ? 1 : 0);
        dm.xcols = d.G * d.N;
        dm.xdiv = Q * (int)(d.H / d.G);
        dm.xmul = d.N;
        dm.xmod = Q;
        dm.sx[1] = d.G * d.N;
        dm.sx[0] = d.T * d.G * d.N;
        // dC = sum over the group's heads of S^T dy: each run head adds its fp32
        // output straight into dC (columns 64 q .. of its group).  The fp32-output
        // variant fits shared memory here (N'' = P <= 128).
        Dims dr = dm;
        dr.yred = 1;
        dr.sy[1] = d.G * d.N;
        dr.sy[0] = d.T * d.G * d.N;
        e = cudaMemsetAsync(a.dC, 0, sizeof(float) * (size_t)(d.b * d.T * d.G * d.N), st);
        if (e == cudaSuccess)
            e = launch_chunk_out_tc(dr, a.B, a.x, a.dy, a.cum2, a.dtT, a.Sprev, nullptr, a.dC, err, st,
                                    nullptr, false, true);
        // dB = sum over the group's heads of dt G^T x: C'' = dt x reversed (bwd_prep), and
        // each run head adds its fp32 rows, reversed back to token order, into dB.
        Dims db = dm;
        db.yred = 1;
        db.yrev = 1;
        db.sy[1] = d.G * d.N;
        db.sy[0] = d.T * d.G * d.N;
        if (e == cudaSuccess)
            e = cudaMemsetAsync(a.dB, 0, sizeof(float) * (size_t)(d.b * d.T * d.G * d.N), st);
        if (e == cudaSuccess)
            e = launch_chunk_out_tc(db, w.Br, w.dyr, w.xr, w.cum2r, w.ones, a.GnIO, nullptr, a.dB, err, st,
                                    nullptr, false, true);
    } else {
        e = out4(d2, w.xB, a.x, a.dy, w.cum2d, w.dtTd, w.SprevT, w.yC, false);        // S^T dy
        if (e == cudaSuccess)
            e = out4(d2, w.xCr, w.dyr, w.xr, w.cum2rd, w.onesd, w.GnT, w.zB, false); // G^T x
    }
    if (e != cudaSuccess) return e;
    bwd_token<TI><<<(unsigned)g4, kThreads, 0, st>>>(a);
    if (!tc2)
        bwd_bc_reduce<TI><<<dim3((unsigned)d.T, (unsigned)d.b), kThreads, 0, st>>>(
            static_cast<const TI*>(w.yC), static_cast<const TI*>(w.zB), a.dtT, a.dB, a.dC, (int)d.T,
            (int)d.H, (int)d.G, (int)d.N, (int)d.L, 1);
    return cudaGetLastError();
}

}  // namespace

bool bwd_dot_mode(const Dims& d, bool tc) {
    return tc && tc_supported(d) && d.P == 64 && k4_dx_fits(d);   // the fp32-y variant and dx mode fit
}

Dims bwd_run_dims(const Dims& d) {
    const int64_t Q = d.N >= 64 ? d.N / 64 : 1;
    Dims d2 = d;   // Q*H heads of N/Q, H groups of Q, state dimension P
    d2.H = Q * d.H;
    d2.P = d.N / Q;
    d2.N = d.P;
    d2.G = d.H;
    set_contiguous(d2);
    return d2;
}

cudaError_t launch_backward(const Dims& d, bool tc, const void* x, const void* B, const void* C,
                            const void* dy, const float* A, const float* D, const float* cum2,
                            const float* dtT, const void* Sprev, const float* fin,
                            const BwdWork& w, const float* dfinal, float* dx, float* ddt,
                            float* dA, float* dB, float* dC, float* dD, float* dinit,
                            int32_t* err, cudaStream_t st) {
    if (d.b == 0 || d.H == 0 || d.T == 0) return cudaSuccess;
    if (d.L > 256) return cudaErrorInvalidValue;   // bwd_token's tokens: one per thread
    const bool dot = bwd_dot_mode(d, tc);
    BwdArgs a{x, B, C, dy, A, D, cum2, dtT, Sprev, fin, w.Gn, w.GnIO,
              static_cast<const float*>(w.yno), dot ? w.ydot2 : nullptr,
              dot ? nullptr : static_cast<const float*>(w.yr), dot ? w.xyd2 : nullptr,
              dot ? w.dyxd2 : nullptr, dx, ddt, dA, dD, dB, dC, (int)d.T, (int)d.H, (int)d.P, (int)d.N, (int)d.G,
              (int)d.L, (int)d.nc, tc ? 1 : 0};
    return d.dtype == 1 ? launch_t<__nv_bfloat16>(d, a, w, tc, dfinal, dinit, err, st)
                        : launch_t<float>(d, a, w, tc, dfinal, dinit, err, st);
}

}  // namespace m2
