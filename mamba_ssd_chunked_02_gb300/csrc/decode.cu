// decode.cu -- one recurrent step per (b, h): the single-token form of the model.
//
// Pages: "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr), "Mamba-2
// 아키텍처의 핵심 연산" (the recurrent read-out of the state), with the state update
// of the chunked path (decay exp(dt A) on the state, dt x B^T as the input):
//
//   S <- exp2(log2(e) dt A) S + dt x B^T        (S: P x N, fp32, updated in place)
//   y  = S C + D x
//
// One CTA per (b, h); a warp walks state rows p (warp, warp + 8, ...), four rows'
// loads in flight at a time, each lane holding the state elements n = lane + 32 k
// of a row: rows are read and written with 128-byte coalesced accesses, B and C of the head's group are held
// in registers, and y_p is the warp-sum of S_p . C plus D x_p.  A pure stream of
// the state: 8 bytes per state element (read + write).
#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kThreads = 256;

template <typename TI, int NK>   // NK = ceil(N / 32) state elements per lane
__global__ void __launch_bounds__(kThreads)
decode_kernel(float* __restrict__ S, const TI* __restrict__ x, const float* __restrict__ dt,
              const float* __restrict__ A, const TI* __restrict__ B, const TI* __restrict__ C,
              const float* __restrict__ D, TI* __restrict__ y, int H, int P, int N, int G) {
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float dth = __ldg(dt + bh);
    const float a = ex2(dth * __ldg(A + h) * kLog2e);
    const float dh = D ? __ldg(D + h) : 0.f;
    float bn[NK], cn[NK];
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const int n = lane + 32 * k;
        bn[k] = n < N ? to_f32(B[((int64_t)b * G + g) * N + n]) : 0.f;
        cn[k] = n < N ? to_f32(C[((int64_t)b * G + g) * N + n]) : 0.f;
    }
    float* Sh = S + (int64_t)bh * P * N;
    // Rows p = warp + 8 r; kRows rows' loads are issued before any is used.
    constexpr int kRows = 4;
    for (int p0 = warp; p0 < P; p0 += kRows * (kThreads / 32)) {
        float sv[kRows][NK];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int p = p0 + r * (kThreads / 32);
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                const int n = lane + 32 * k;
                sv[r][k] = (p < P && n < N) ? Sh[(int64_t)p * N + n] : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int p = p0 + r * (kThreads / 32);
            if (p >= P) break;
            const float xp = to_f32(x[(int64_t)bh * P + p]);
            const float u = dth * xp;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                const int n = lane + 32 * k;
                if (n < N) {
                    const float v = fmaf(a, sv[r][k], u * bn[k]);
                    Sh[(int64_t)p * N + n] = v;
                    acc = fmaf(v, cn[k], acc);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) y[(int64_t)bh * P + p] = from_f32<TI>(fmaf(dh, xp, acc));
        }
    }
}

template <typename TI>
cudaError_t launch_t(const Dims& d, float* S, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* D, void* y, cudaStream_t st) {
    const unsigned grid = (unsigned)(d.b * d.H);
    const int nk = (int)((d.N + 31) / 32);
    auto args = [&](auto k) {
        k<<<grid, kThreads, 0, st>>>(S, static_cast<const TI*>(x), dt, A, static_cast<const TI*>(B),
                                     static_cast<const TI*>(C), D, static_cast<TI*>(y), (int)d.H,
                                     (int)d.P, (int)d.N, (int)d.G);
    };
    switch (nk) {
        case 1: args(decode_kernel<TI, 1>); break;
        case 2: args(decode_kernel<TI, 2>); break;
        case 4: args(decode_kernel<TI, 4>); break;
        case 8: args(decode_kernel<TI, 8>); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Dims& d, float* S, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, void* y, cudaStream_t st) {
    if (d.b == 0 || d.H == 0) return cudaSuccess;
    if (d.b * d.H >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    return d.dtype == 1 ? launch_t<__nv_bfloat16>(d, S, x, dt, A, B, C, D, y, st)
                        : launch_t<float>(d, S, x, dt, A, B, C, D, y, st);
}

}  // namespace m2
