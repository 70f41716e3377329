// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernels.
// Not part of the public interface (include/mamba2_ssd.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace m2 {

// Problem dimensions of one call, after validation.
struct Dims {
    int64_t b, T, H, P, N, G, L, nc;
    int dtype;   // 0 = f32, 1 = bf16 (element type of x, B, C, y, Sprev)
    // Element strides {batch, token} of x, y ([.., H*P] contiguous per token),
    // B, C ([.., G*N]) and dt ([.., H]); contiguous unless set by the strided
    // whole-path call (the stage entry points take contiguous tensors).
    int64_t sx[2], sy[2], sB[2], sC[2], sdt[2];
    // Tensor-core view only (tc_view): each head is split into 2^pts heads of 64
    // of its P dimension; per-head inputs (cum2, dtT, D) are read at head >> pts.
    int pts = 0;
    // Tensor-core output stage only: x of head h starts at column
    // (h / xdiv) * xmul + (h % xmod) * 64 of an x tensor xcols wide (0: xmul = P,
    // xcols = H * P, i.e. x laid out [.., H, P]).  The backward's runs read B and C
    // of a head's group this way instead of per-head copies.
    int xdiv = 1, xmod = 1;
    int64_t xmul = 0, xcols = 0;
    // Tensor-core output stage with fp32 y only: add y of head h into the fp32
    // tensor y (xcols wide, element strides sy) at the x column of head h,
    // instead of storing it (the backward's head sums).
    int yred = 0;
    // Tensor-core output stage only: the carried state of head h is read
    // untransposed, as GEMM3's operand in MN-major form: rows (h / xmod) * N .. of
    // a [.., P' = N, N' = xmod * 64] state tensor (P', N' the state's own sizes), the
    // 64 columns from (h % xmod) * 64 (the backward's runs on transposed states).
    int st_mn = 0;
    // Tensor-core output stage with fp32 y only (dot mode): instead of y, write
    // ydot_out[((b * H + h) * T + t) * 2 + g] = sum over the 32 columns of group g
    // of dy[b, t, h, p] * y[b, t, h, p] (dy bf16, contiguous [b, T, H, P]).
    const void* ydot_dy = nullptr;
    float* ydot_out = nullptr;
    // With yred: the run's rows are each chunk's tokens in reverse order (row k of
    // a chunk of Lc tokens adds into token Lc - 1 - k).
    int yrev = 0;
    // Tensor-core output stage with fp32 y only (dx mode, the backward's y' run,
    // whose row k of a chunk of Lc tokens is token j = Lc - 1 - k): instead of y',
    // write dx[b, t, h, :] = dt[b, h, t] y' + D[h] dy[b, t, h, :] (fp32) and the
    // partial dots dxm_xy[((b * H + h) * T + t) * 2 + g] = sum over the 32 columns
    // of group g of x y', dxm_dyx[...] = the same of dy x (x, dy bf16, contiguous
    // [b, T, H, 64]; dt [b, H, T]; D [H] or null).
    // Tensor-core output stage with fp32 y only: dt is 1 everywhere (the
    // backward's y' run); dtT is not read.
    int dt1 = 0;
    // Tensor-core output stage with fp32 y only (the backward's y' run in token
    // order): anti-causal, y_t = sum_{s >= t} M[t, s] x_s + exp2(cum2_last - cum2_t)
    // (C_t . Sprev^T), M[t, s] = (C_t . B_s) exp2(cum2_s - cum2_t) dt_s.
    int antic = 0;
    const void* dxm_x = nullptr;
    const void* dxm_dy = nullptr;
    const float* dxm_dt = nullptr;
    const float* dxm_D = nullptr;
    float* dxm_dx = nullptr;
    float* dxm_xy = nullptr;
    float* dxm_dyx = nullptr;
};

// The dx-mode pointers of Dims, as one kernel argument.
struct DxArgs {
    const void* x;    // bf16
    const void* dy;   // bf16
    const float* dt;
    const float* D;
    float* dx;
    float* xy;
    float* dyx;
};

// Contiguous strides for the sizes in d.
inline void set_contiguous(Dims& d) {
    d.sx[1] = d.sy[1] = d.H * d.P;
    d.sx[0] = d.sy[0] = d.T * d.H * d.P;
    d.sB[1] = d.sC[1] = d.G * d.N;
    d.sB[0] = d.sC[0] = d.T * d.G * d.N;
    d.sdt[1] = d.H;
    d.sdt[0] = d.T * d.H;
}

// Element counts and byte sizes of the intermediates.
inline int64_t n_cum(const Dims& d) { return d.b * d.H * d.T; }
inline int64_t n_state(const Dims& d) { return d.b * d.nc * d.H * d.P * d.N; }
inline int64_t esize(const Dims& d) { return d.dtype == 1 ? 2 : 4; }

// Stage 1: chunk-local log2-scaled cumsum + [b,h,t] transpose of dt.  When
// `zero` is given, the kernel also sets zero[0 .. nzero) to 0 (the ticket and
// flag words of the fused stage 2+3 kernel that follows on the same stream).
cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, float* cum2,
                                float* dtT, int32_t* err, cudaStream_t st,
                                int32_t* zero = nullptr, int64_t nzero = 0, bool pdl = false);

// Stage 2: chunk states.  CUDA-core variant (any supported shape / dtype).
cudaError_t launch_chunk_state_simt(const Dims& d, const void* x, const void* B,
                                    const float* cum2, const float* dtT, float* dS,
                                    int32_t* err, cudaStream_t st);
// Stage 2: tcgen05 variant (bf16, shapes accepted by tc_supported()); dS is
// written in fp32, or in bf16 when ds16 (the whole-path call).
// When xabs is given it also records max |x| per (b, chunk, head): eight words
// per head ([b][nc][H][8], bf16 bit patterns of |x|; their max is the bound).
// pdl: launched with programmatic dependent launch after stage 1 (the
// whole-path call): x and B are read before stage 1 completes.
// adj: weight mode of the backward's chunk adjoint, w_s = exp2(cum2_s) (dtT unused).
cudaError_t launch_chunk_state_tc(const Dims& d, const void* x, const void* B,
                                  const float* cum2, const float* dtT, void* dS, bool ds16,
                                  int32_t* err, cudaStream_t st, uint32_t* xabs = nullptr,
                                  bool pdl = false, bool adj = false);

// Stages 2 and 3 fused (tcgen05, bf16, tc_supported() shapes): each CTA
// computes its chunk's dS in tensor memory, then, head by head, takes the state
// entering its chunk from the CTA of the previous chunk (a two-slot ring `carry`
// [2][b][H][P][N] fp32 and one flag per (b, h, n-tile, chunk)), writes Sprev
// (bf16) and passes decay * Sprev + dS on (or writes final_state).  CTAs take
// their work item from `ticket` in chunk order, so a CTA only waits for CTAs
// that started before it.  flags[0 .. fused_flag_words(d)) and *ticket must be
// zero at launch.
int64_t fused_flag_words(const Dims& d);
cudaError_t launch_chunk_state_pass_tc(const Dims& d, const void* x, const void* B,
                                       const float* cum2, const float* dtT, const float* init,
                                       float* carry, int32_t* flags, int32_t* ticket,
                                       void* Sprev, float* final_state, int32_t* err,
                                       cudaStream_t st);

// Stage 3: sequential state pass over chunks (dS in fp32, or bf16 when ds16).
// pdl: launched with programmatic dependent launch after stage 2.
cudaError_t launch_state_pass(const Dims& d, const void* dS, bool ds16, const float* cum2,
                              const float* init, void* Sprev, float* final_state,
                              int32_t* err, cudaStream_t st, bool pdl = false);

// Stage 4: fused output.  CUDA-core variant.
// y32: y is written in fp32 whatever the input type (the backward pass's use).
cudaError_t launch_chunk_out_simt(const Dims& d, const void* x, const void* B, const void* C,
                                  const float* cum2, const float* dtT, const void* Sprev,
                                  const float* D, void* y, int32_t* err, cudaStream_t st,
                                  bool y32 = false);
// Stage 4: tcgen05 variant; xabs: stage 2's max |x| words, or null (then the
// kernel scans each x tile for its fp16 range check itself).
// pdl: launched with programmatic dependent launch after stage 3 (the
// whole-path call): everything but Sprev is read before stage 3 completes.
// y32: y is written in fp32 (the backward pass's use); cudaErrorNotSupported
// when that variant's staging does not fit in shared memory (L = 256, N = 256).
cudaError_t launch_chunk_out_tc(const Dims& d, const void* x, const void* B, const void* C,
                                const float* cum2, const float* dtT, const void* Sprev,
                                const float* D, void* y, int32_t* err, cudaStream_t st,
                                const uint32_t* xabs = nullptr, bool pdl = false,
                                bool y32 = false);

// One recurrent step per (b, h): S <- exp(dt A) S + dt x B^T in place, y = S C + D x.
// A bounded wait that runs out sets kErrTimeoutDecode in *err.
cudaError_t launch_decode(const Dims& d, float* S, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, void* y, int32_t* err,
                          cudaStream_t st);

// Backward pass, after the forward's stages 1-3 (cum2, dtT, Sprev in the I/O
// type, the final state in fp32).  Scratch, all in the workspace:
struct BwdWork {
    float* Gn;      // [b,nc,H,P,N] fp32 (chunk adjoints, then Gn)
    void* GnIO;     // [b,nc,H,P,N] I/O type copy of Gn (unused when the I/O type is fp32)
    void* yno;      // [b,T,H,P] fp32: y without the skip term
    void* yr;       // [b,T,H,P] fp32: y' of the reversed run
    void* dyr;      // [b,T,H,P] dy, each chunk's tokens reversed
    void* Br;       // [b,T,G,N] C reversed (the reversed run's B)
    void* Cr;       // [b,T,G,N] B reversed (the reversed run's C)
    float* cum2r;   // [b,H,T]
    float* ones;    // [b,H,T]
    void* xB;       // [b,T,H,N] the group's B per head (the dC run's x)
    void* xCr;      // [b,T,H,N] the group's C per head, reversed (the dB run's x)
    void* xr;       // [b,T,H,P] x reversed (the dB run's C)
    void* SprevT;   // [b,nc,H,N,P] Sprev transposed (the dC run's carried state)
    void* GnT;      // [b,nc,H,N,P] Gn transposed (the dB run's carried state)
    float* cum2d;   // [b,Q*H,T] cum2 per run head (Q = N/64, or 1 when N < 64)
    float* dtTd;    // [b,Q*H,T]
    float* cum2rd;  // [b,Q*H,T]
    float* onesd;   // [b,Q*H,T]
    void* yC;       // [b,T,H,N] S^T dy per head (I/O type)
    void* zB;       // [b,T,H,N] G^T x per head, reversed chunks (I/O type)
    float* ydot2;   // [b,H,T,2] dy . y partial sums (dot mode, bwd_dot_mode)
    float* xyd2;    // [b,H,T,2] x . y' partial sums (the y' run in dx mode, same condition)
    float* dyxd2;   // [b,H,T,2] dy . x partial sums (same)
    uint32_t* xabs_x;    // [b,nc,H][8] max |x| per chunk from stage 2 (tensor-core path), or null
    uint32_t* xabs_dy;   // [b,nc,H][8] max |dy| per chunk from the adjoint stage-2 run, or null
};
// The backward's dC (rev = false: Q = dy, K = x, O = B, S = Sprev) or dB (rev =
// true: Q = x, K = dy, O = C, S = Gn) on tcgen05, summed over each group's heads
// in the kernel and added into out (fp32 [b,T,G,N]: zero it first).  bf16, P = 64,
// L in {128, 256}, N in {64, 128, 256} (bwd_bc_tc_supported).
bool bwd_bc_tc_supported(const Dims& d);
int bwd_bc_heads_per_cta(const Dims& d);
cudaError_t launch_bwd_bc_tc(const Dims& d, bool rev, const void* q, const void* k, const void* o,
                             const void* s, const float* cum2, const float* dtT, float* out,
                             int32_t* err, cudaStream_t st);
// The dC / dB runs of the backward: Q = N/64 heads of 64 columns per head (one
// when N < 64), H groups of Q, state dimension P.
Dims bwd_run_dims(const Dims& d);
// True when the backward's y run takes the tensor cores in dot mode (no fp32 y)
// and its y' run in dx mode (no fp32 y').
bool bwd_dot_mode(const Dims& d, bool tc);
// True when the fp32-output stage-4 variant for d's shape can stage dx mode's x
// and dy tiles (two 32 KB slots in its y buffers).
bool k4_dx_fits(const Dims& d);
// tc: run stage 4 on the tensor cores (the shapes tc_supported() accepts).
// dA and dD (if given) are accumulated into (zero them first); dinit may be null.
cudaError_t launch_backward(const Dims& d, bool tc, const void* x, const void* B, const void* C,
                            const void* dy, const float* A, const float* D, const float* cum2,
                            const float* dtT, const void* Sprev, const float* fin,
                            const BwdWork& w, const float* dfinal, float* dx, float* ddt,
                            float* dA, float* dB, float* dC, float* dD, float* dinit,
                            int32_t* err, cudaStream_t st);

// Diagnostic: waits that nothing releases, bounded by limit_ns; sets kErrSelfTest.
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* err, cudaStream_t st);

// True when the tcgen05 kernels handle this shape.  P = 32 runs on 64-column
// tiles that also hold the next head's columns (only the head's own outputs are
// kept): stages 2 and 4, not the fused stages 2+3.
bool tc_supported(const Dims& d);
bool tc_fused_supported(const Dims& d);

// The shape the tcgen05 kernels run: P = 128 as twice the heads of P = 64.  x, y
// ([.., H, P] per token), Sprev and dS ([.., H, P, N]) hold the same bytes in
// either view; only cum2, dtT and D stay per original head (read at h >> pts).
inline Dims tc_view(const Dims& d) {
    Dims v = d;
    if (d.P == 128) {
        v.H = 2 * d.H;
        v.P = 64;
        v.pts = 1;
    }
    return v;
}

// SMs of the current device (cached per device); kFallbackSMs, a GB300's
// count, when no device can be queried.
constexpr int kFallbackSMs = 152;
int sm_count();

// Per-shape launch choices found by the offline sweep (tiles.cu, tile_table.inc).
struct TileChoice {
    int32_t N, P, L, hpg;      // state size, head dim, chunk size, heads per group
    int64_t bnc_lo, bnc_hi;    // range of b * nc the entry covers
    int32_t k2_hpc;            // stage 2: units per CTA (0: one wave of even ranges)
    int32_t k4_v1, k4_v2;      // stage 4: head-block sizes of the two grid regions
    int32_t k4_waves1;         // stage 4: SM waves the v1 region fills (0: v1 everywhere)
};
// The table entry for this shape, or null.
const TileChoice* find_tile(const Dims& d);
// Tuning override k (0: stage-2 units per CTA, 1/2: stage-4 v1/v2, 3: stage-4
// v1-region waves), 0 when not set (mamba2_ssd_tile_override); -1 bypasses the
// table, kEvenSplit (stage 2 only) forces one wave of even ranges.
int tile_override(int k);
constexpr int kEvenSplit = -2;

// Where a launch choice comes from.
enum : int { kFromModel = 0, kFromTable = 1, kFromOverride = 2 };
// Stage 2 (tensor-core, unfused): units per CTA (a unit is one head of one
// (b, chunk, 128-wide state tile); a CTA takes a contiguous range) and its source.
int k2_units_per_cta(const Dims& d, int* src);
// Stage 4 (tensor-core): head-block sizes v1, v2, CTAs of the v1 region (n1),
// all CTAs, the (b, c) pairs of the v1 region and the source.
struct Split4 {
    int v1, v2;
    int64_t n1, ctas, n1_bc;
    int src;
};
Split4 k4_split(const Dims& d);

// Device-side error bits (OR-ed into the library's error word).
enum : int32_t {
    kErrTimeoutK2 = 1 << 0,    // a bounded wait ran out in the tcgen05 chunk-state kernel
    kErrTimeoutK4 = 1 << 1,    // ... in the tcgen05 chunk-output kernel
    kErrLaunchCfg = 1 << 2,    // a kernel saw a launch configuration it does not support
    kErrChainK23 = 1 << 3,     // the fused stage 2+3 kernel gave up waiting for the previous chunk
    kErrSelfTest = 1 << 4,     // the wait self-test's waits ran out (expected)
    kErrTimeoutDecode = 1 << 5,  // a bounded wait ran out in the decode kernel
};

}  // namespace m2
