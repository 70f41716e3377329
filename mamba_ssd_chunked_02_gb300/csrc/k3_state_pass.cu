// k3_state_pass.cu -- stage 3: carry the state across chunks.
//
// Pages: "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
// "세 가지 핵심 커널 구현" (fwd_pass_state: a sequential loop over chunks that
// produces the state at the start of every chunk and the final state, reading
// the chunk's last cumsum value and decaying with exp2); "Accelerating Mamba-2
// ..." (brifing.si), section 8 "Advancing States with fwd_pass_state".
//
//   S = initial_state (or 0)
//   for c in 0..nc-1:  Sprev[c] = S;  S = exp2(cum2[last token of c]) * S + dS[c]
//   final_state = S
//
// Sequential over chunks, parallel over (b, h, slices of the P x N state): one
// thread owns 16 bytes' worth of dS elements of the state (4 for fp32 dS, 8 for
// bf16 dS) for the whole chain.  The dS
// loads do not depend on the chain, so each thread keeps a few chunks of loads
// in flight (a rolling prefetch) while it walks the chain: a pure HBM stream of
// dS (fp32, or bf16 on the whole-path call) in and Sprev out per state element
// per chunk.
#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kThreads = 256;
// Chunks of dS loads in flight per thread: 4 for bf16 dS (48 registers, five
// blocks per SM), 8 for fp32 dS (measured best for each).
template <typename TD>
struct Depth {
    static constexpr int value = sizeof(TD) == 2 ? 4 : 8;
};

// A thread owns EPT consecutive state elements, EPT = 16 bytes of dS: one
// 16-byte load of dS and one store of Sprev per chunk.
template <typename TD>
struct Ept {
    static constexpr int value = 16 / (int)sizeof(TD);
};

// 16 bytes of dS stay packed while in flight (4 registers) and are widened to
// fp32 when consumed.
__device__ __forceinline__ uint4 load16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void widen(const uint4& u, float (&v)[4]) {   // fp32 dS
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void widen(const uint4& u, float (&v)[8]) {   // bf16 dS
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
template <int E>
__device__ __forceinline__ void store_state(float* p, const float (&S)[E]) {
#pragma unroll
    for (int k = 0; k < E; k += 4)
        *reinterpret_cast<float4*>(p + k) = make_float4(S[k], S[k + 1], S[k + 2], S[k + 3]);
}
template <int E>
__device__ __forceinline__ void store_state(__nv_bfloat16* p, const float (&S)[E]) {
    uint32_t w[E / 2];
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        __nv_bfloat162 t = __floats2bfloat162_rn(S[2 * k], S[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&t);
    }
    if constexpr (E == 8)
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
}

template <typename TS, typename TD>
__global__ void __launch_bounds__(kThreads)
state_pass_kernel(const TD* __restrict__ dS, const float* __restrict__ cum2,
                  const float* __restrict__ init, TS* __restrict__ Sprev,
                  float* __restrict__ fin, int64_t T, int64_t H, int64_t L, int64_t nc,
                  int64_t PN, int64_t blocks_per_bh) {
    constexpr int E = Ept<TD>::value;
    constexpr int kDepth = Depth<TD>::value;
    // dS comes from stage 2 (programmatic dependent launch on the whole-path
    // call): wait for it, then let stage 4 start launching.
    grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_launch();
    const int64_t bh = blockIdx.x / blocks_per_bh;
    const int64_t iv = (blockIdx.x % blocks_per_bh) * kThreads + threadIdx.x;
    const int64_t e = iv * E;
    if (e >= PN) return;
    const int64_t b = bh / H, h = bh % H;

    float S[E];
#pragma unroll
    for (int k = 0; k < E; ++k) S[k] = init ? __ldg(init + bh * PN + e + k) : 0.f;

    const float* crow = cum2 + bh * T;
    const int64_t cstride = H * PN;                       // chunk stride in dS / Sprev
    const int64_t base = (b * nc * H + h) * PN + e;       // [b, c=0, h, e]

    // Rolling prefetch: the loads of chunk c + kDepth are issued when chunk c is
    // consumed, so kDepth chunks of dS stay in flight for the whole chain.
    // Addresses advance by running pointers (one chunk = cstride elements).
    const TD* pd = dS + base;                    // next chunk of dS to fetch
    const float* pl = crow + L - 1;              // its last token's cum2 (clamped below)
    const float* const plend = crow + T - 1;
    TS* ps = Sprev + base;
    uint4 buf[kDepth];
    float cl[kDepth];
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
        if (u < nc) {
            buf[u] = load16(pd);
            cl[u] = __ldg(pl < plend ? pl : plend);
            pd += cstride;
            pl += L;
        }
    }
    for (int64_t c0 = 0; c0 < nc; c0 += kDepth) {
#pragma unroll
        for (int u = 0; u < kDepth; ++u) {
            if (c0 + u < nc) {
                float d[E];
                widen(buf[u], d);
                const float dec = ex2(cl[u]);
                if (c0 + u + kDepth < nc) {
                    buf[u] = load16(pd);
                    cl[u] = __ldg(pl < plend ? pl : plend);
                    pd += cstride;
                    pl += L;
                }
                store_state(ps, S);
                ps += cstride;
#pragma unroll
                for (int k = 0; k < E; ++k) S[k] = fmaf(dec, S[k], d[k]);
            }
        }
    }
    store_state(fin + bh * PN + e, S);
}

}  // namespace

cudaError_t launch_state_pass(const Dims& d, const void* dS, bool ds16, const float* cum2,
                              const float* init, void* Sprev, float* final_state,
                              int32_t* /*err*/, cudaStream_t st, bool pdl) {
    const int64_t PN = d.P * d.N;   // multiple of 256 for every supported P, N
    if (d.b == 0 || d.H == 0) return cudaSuccess;
    if (d.nc == 0) {
        // Empty sequence: the final state is the initial state.
        const size_t bytes = (size_t)(d.b * d.H * PN) * sizeof(float);
        return init ? cudaMemcpyAsync(final_state, init, bytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(final_state, 0, bytes, st);
    }
    const int64_t ept = ds16 ? Ept<__nv_bfloat16>::value : Ept<float>::value;
    const int64_t blocks_per_bh = (PN / ept + kThreads - 1) / kThreads;
    const int64_t grid = d.b * d.H * blocks_per_bh;
    using bf16 = __nv_bfloat16;
    const dim3 g((unsigned)grid), blk(kThreads);
    if (d.dtype == 1 && ds16)
        return launch_kernel(state_pass_kernel<bf16, bf16>, g, blk, 0, st, pdl,
                             static_cast<const bf16*>(dS), cum2, init, static_cast<bf16*>(Sprev),
                             final_state, d.T, d.H, d.L, d.nc, PN, blocks_per_bh);
    if (d.dtype == 1)
        return launch_kernel(state_pass_kernel<bf16, float>, g, blk, 0, st, pdl,
                             static_cast<const float*>(dS), cum2, init, static_cast<bf16*>(Sprev),
                             final_state, d.T, d.H, d.L, d.nc, PN, blocks_per_bh);
    return launch_kernel(state_pass_kernel<float, float>, g, blk, 0, st, pdl,
                         static_cast<const float*>(dS), cum2, init, static_cast<float*>(Sprev),
                         final_state, d.T, d.H, d.L, d.nc, PN, blocks_per_bh);
}

}  // namespace m2
