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
// Sequential over chunks, parallel over (b, h, 4-element slices of the P x N
// state): one thread owns a float4 of the state for the whole chain.  The dS
// loads do not depend on the chain, so each thread keeps kDepth chunks of loads
// in flight (a rolling prefetch) while it walks the chain: a pure HBM stream of
// 4 + esize bytes per state element per chunk.
#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kThreads = 256;
constexpr int kDepth = 8;   // chunks of dS loads in flight per thread

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

template <typename TS>
__global__ void __launch_bounds__(kThreads)
state_pass_kernel(const float* __restrict__ dS, const float* __restrict__ cum2,
                  const float* __restrict__ init, TS* __restrict__ Sprev,
                  float* __restrict__ fin, int64_t T, int64_t H, int64_t L, int64_t nc,
                  int64_t PN, int64_t blocks_per_bh) {
    const int64_t bh = blockIdx.x / blocks_per_bh;
    const int64_t i4 = (blockIdx.x % blocks_per_bh) * kThreads + threadIdx.x;
    const int64_t e = i4 * 4;
    if (e >= PN) return;
    const int64_t b = bh / H, h = bh % H;

    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init) S = __ldg(reinterpret_cast<const float4*>(init + bh * PN + e));

    const float* crow = cum2 + bh * T;
    const int64_t cstride = H * PN;                       // chunk stride in dS / Sprev
    const int64_t base = (b * nc * H + h) * PN + e;       // [b, c=0, h, e]

    // Rolling prefetch: the loads of chunk c + kDepth are issued when chunk c is
    // consumed, so kDepth chunks of dS stay in flight for the whole chain.
    // Addresses advance by running pointers (one chunk = cstride elements).
    const float* pd = dS + base;                 // next chunk of dS to fetch
    const float* pl = crow + L - 1;              // its last token's cum2 (clamped below)
    const float* const plend = crow + T - 1;
    TS* ps = Sprev + base;
    float4 buf[kDepth];
    float cl[kDepth];
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
        if (u < nc) {
            buf[u] = __ldcs(reinterpret_cast<const float4*>(pd));
            cl[u] = __ldg(pl < plend ? pl : plend);
            pd += cstride;
            pl += L;
        }
    }
    for (int64_t c0 = 0; c0 < nc; c0 += kDepth) {
#pragma unroll
        for (int u = 0; u < kDepth; ++u) {
            if (c0 + u < nc) {
                const float4 d = buf[u];
                const float dec = ex2(cl[u]);
                if (c0 + u + kDepth < nc) {
                    buf[u] = __ldcs(reinterpret_cast<const float4*>(pd));
                    cl[u] = __ldg(pl < plend ? pl : plend);
                    pd += cstride;
                    pl += L;
                }
                store4(ps, S);
                ps += cstride;
                S.x = fmaf(dec, S.x, d.x);
                S.y = fmaf(dec, S.y, d.y);
                S.z = fmaf(dec, S.z, d.z);
                S.w = fmaf(dec, S.w, d.w);
            }
        }
    }
    *reinterpret_cast<float4*>(fin + bh * PN + e) = S;
}

}  // namespace

cudaError_t launch_state_pass(const Dims& d, const float* dS, const float* cum2,
                              const float* init, void* Sprev, float* final_state,
                              int32_t* /*err*/, cudaStream_t st) {
    const int64_t PN = d.P * d.N;   // multiple of 256 for every supported P, N
    if (d.b == 0 || d.H == 0) return cudaSuccess;
    if (d.nc == 0) {
        // Empty sequence: the final state is the initial state.
        const size_t bytes = (size_t)(d.b * d.H * PN) * sizeof(float);
        return init ? cudaMemcpyAsync(final_state, init, bytes, cudaMemcpyDeviceToDevice, st)
                    : cudaMemsetAsync(final_state, 0, bytes, st);
    }
    const int64_t blocks_per_bh = (PN / 4 + kThreads - 1) / kThreads;
    const int64_t grid = d.b * d.H * blocks_per_bh;
    if (d.dtype == 1)
        state_pass_kernel<__nv_bfloat16><<<(unsigned)grid, kThreads, 0, st>>>(
            dS, cum2, init, static_cast<__nv_bfloat16*>(Sprev), final_state, d.T, d.H, d.L,
            d.nc, PN, blocks_per_bh);
    else
        state_pass_kernel<float><<<(unsigned)grid, kThreads, 0, st>>>(
            dS, cum2, init, static_cast<float*>(Sprev), final_state, d.T, d.H, d.L, d.nc, PN,
            blocks_per_bh);
    return cudaGetLastError();
}

}  // namespace m2
