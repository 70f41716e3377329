// simt.cu -- CUDA-core versions of stage 2 (chunk states) and stage 4 (fused
// output).  They serve the fp32 dtype (whose tolerance rules out reduced-
// precision tensor-core operands) and every supported shape the tcgen05
// kernels do not cover; all arithmetic is fp32 FMA.
//
// Pages: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile" (brifing.si), section 4 (jump formula: the chunk state is a
// matrix product of stacked B and X), section 9 (compute_out fuses the
// interaction term, the carried-state term and the skip term), section 11
// (causal masking before exponentiation).  "NVIDIA CUDA Tile로 Mamba-2 순방향
// 전달 커널 가속화" (devin.kr), "세 가지 핵심 커널 구현" (the lower-triangular mask
// is generated from indices, never stored).
#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------------ stage 2 ---
// dS[b,c,h,p,n] = sum_{s in chunk c} w_s x[s,p] B[s,n],
// w_s = dtT[s] * exp2(cum2[last] - cum2[s]).
// Element strides {batch, token} of x, y, B and C (a token's H*P or G*N
// elements are contiguous).
struct IoStrides {
    int64_t xb, xt, yb, yt, Bb, Bt, Cb, Ct;
};
IoStrides io_strides(const Dims& d) {
    return {d.sx[0], d.sx[1], d.sy[0], d.sy[1], d.sB[0], d.sB[1], d.sC[0], d.sC[1]};
}

// CTA per (b, c, h) x (64-wide p tile) x (64-wide n tile); each thread owns a
// 4 x 4 register tile; s is consumed in blocks of 32 staged in shared memory.
template <typename T>
__global__ void __launch_bounds__(kThreads)
chunk_state_simt_kernel(const T* __restrict__ x, const T* __restrict__ B,
                        const float* __restrict__ cum2, const float* __restrict__ dtT,
                        float* __restrict__ dS, int64_t Tlen, int64_t H, int64_t P, int64_t N,
                        int64_t G, int64_t L, int64_t nc, IoStrides io) {
    constexpr int TP = 64, TN = 64, SB = 32;
    __shared__ float xs[SB][TP];
    __shared__ float bs[SB][TN];
    __shared__ float ws[SB];

    const int64_t bch = blockIdx.x;
    const int64_t h = bch % H, c = (bch / H) % nc, b = bch / (H * nc);
    const int64_t g = h / (H / G);
    const int64_t p0 = (int64_t)blockIdx.y * TP, n0 = (int64_t)blockIdx.z * TN;
    const int64_t t0 = c * L, t1 = min(t0 + L, Tlen);
    const float* crow = cum2 + (b * H + h) * Tlen;
    const float* drow = dtT + (b * H + h) * Tlen;
    const float last = crow[t1 - 1];

    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[4][4] = {};

    for (int64_t s0 = t0; s0 < t1; s0 += SB) {
        if (threadIdx.x < SB) {
            const int64_t s = s0 + threadIdx.x;
            ws[threadIdx.x] = s < t1 ? drow[s] * ex2(last - crow[s]) : 0.f;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < SB * TP; idx += kThreads) {
            const int i = idx / TP, j = idx % TP;
            const int64_t s = s0 + i, p = p0 + j;
            xs[i][j] = (s < t1 && p < P) ? ws[i] * to_f32(x[b * io.xb + s * io.xt + h * P + p]) : 0.f;
        }
        for (int idx = threadIdx.x; idx < SB * TN; idx += kThreads) {
            const int i = idx / TN, j = idx % TN;
            const int64_t s = s0 + i, n = n0 + j;
            bs[i][j] = (s < t1 && n < N) ? to_f32(B[b * io.Bb + s * io.Bt + g * N + n]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int i = 0; i < SB; ++i) {
            const float4 a = *reinterpret_cast<const float4*>(&xs[i][ty * 4]);
            const float4 v = *reinterpret_cast<const float4*>(&bs[i][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
        }
        __syncthreads();
    }
    float* out = dS + ((b * nc + c) * H + h) * P * N;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t p = p0 + ty * 4 + r;
        if (p >= P) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t n = n0 + tx * 4 + q;
            if (n < N) out[p * N + n] = acc[r][q];
        }
    }
}

// ------------------------------------------------------------------ stage 4 ---
// CTA per (b, c, h) x (32-token tile of the chunk).  For each 32-token block of
// keys s <= the tile's last query: G = C_t . B_s (fp32 dot products in shared
// memory), masked with s <= t from the indices before exp2, scaled by
// exp2(cum2_t - cum2_s) dt_s, then accumulated against x_s.  The carried term
// exp2(cum2_t) Sprev C_t and the skip term D x_t are added before the store.
template <typename T, typename TY>   // TY: element type of y (T, or fp32)
__global__ void __launch_bounds__(kThreads)
chunk_out_simt_kernel(const T* __restrict__ x, const T* __restrict__ B, const T* __restrict__ C,
                      const float* __restrict__ cum2, const float* __restrict__ dtT,
                      const T* __restrict__ Sprev, const float* __restrict__ D,
                      TY* __restrict__ y, int64_t Tlen, int64_t H, int64_t P, int64_t N,
                      int64_t G, int64_t L, int64_t nc, IoStrides io) {
    constexpr int TT = 32, SB = 32;
    extern __shared__ float smem[];
    const int NP = (int)N + 1;                 // padded rows (bank spread)
    const int XP = (int)P + 1;
    float* Cs = smem;                          // [TT][N]
    float* Bs = Cs + TT * N;                   // [SB][N+1]
    float* Xs = Bs + SB * NP;                  // [SB][P+1]  (also Sprev^T staging)
    float* Gs = Xs + SB * XP;                  // [TT][SB+1]
    float* ct = Gs + TT * (SB + 1);            // cum2 of the query rows
    float* cs = ct + TT;                       // cum2 of the key block
    float* dsv = cs + SB;                      // dt of the key block

    const int64_t bch = blockIdx.x;
    const int64_t h = bch % H, c = (bch / H) % nc, b = bch / (H * nc);
    const int64_t g = h / (H / G);
    const int64_t cs0 = c * L, ce = min(cs0 + L, Tlen);
    const int64_t q0 = cs0 + (int64_t)blockIdx.y * TT;      // first query token
    if (q0 >= ce) return;
    const int64_t q1 = min(q0 + TT, ce);                   // one past the last query
    const float* crow = cum2 + (b * H + h) * Tlen;
    const float* drow = dtT + (b * H + h) * Tlen;

    for (int idx = threadIdx.x; idx < TT * N; idx += kThreads) {
        const int i = idx / (int)N, n = idx % (int)N;
        const int64_t t = q0 + i;
        Cs[idx] = t < q1 ? to_f32(C[b * io.Cb + t * io.Ct + g * N + n]) : 0.f;
    }
    if (threadIdx.x < TT) ct[threadIdx.x] = (q0 + threadIdx.x < q1) ? crow[q0 + threadIdx.x] : 0.f;

    // Output ownership: thread owns column p = tid % P and rows r0 + k * rs.
    const int p = threadIdx.x % (int)P;
    const int r0 = threadIdx.x / (int)P, rs = kThreads / (int)P;
    const int nrow = TT / rs;                  // 2 .. 16
    float acc[16], accs[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) { acc[k] = 0.f; accs[k] = 0.f; }

    for (int64_t s0 = cs0; s0 < q1; s0 += SB) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < SB * N; idx += kThreads) {
            const int j = idx / (int)N, n = idx % (int)N;
            const int64_t s = s0 + j;
            Bs[j * NP + n] = s < q1 ? to_f32(B[b * io.Bb + s * io.Bt + g * N + n]) : 0.f;
        }
        for (int idx = threadIdx.x; idx < SB * P; idx += kThreads) {
            const int j = idx / (int)P, pp = idx % (int)P;
            const int64_t s = s0 + j;
            Xs[j * XP + pp] = s < q1 ? to_f32(x[b * io.xb + s * io.xt + h * P + pp]) : 0.f;
        }
        if (threadIdx.x < SB) {
            const int64_t s = s0 + threadIdx.x;
            cs[threadIdx.x] = s < q1 ? crow[s] : 0.f;
            dsv[threadIdx.x] = s < q1 ? drow[s] : 0.f;
        }
        __syncthreads();
        // G[i][j] for the 32 x 32 block: thread -> j = tid % 32, i = tid / 32 + 8k.
        {
            const int j = threadIdx.x % SB;
            for (int i = threadIdx.x / SB; i < TT; i += kThreads / SB) {
                const int64_t t = q0 + i, s = s0 + j;
                float v = 0.f;
                if (s <= t && t < q1) {            // causal mask from indices, before exp2
                    float dot = 0.f;
                    for (int n = 0; n < (int)N; ++n) dot = fmaf(Cs[i * N + n], Bs[j * NP + n], dot);
                    v = dot * ex2(ct[i] - cs[j]) * dsv[j];
                }
                Gs[i * (SB + 1) + j] = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k >= nrow) break;
            const int i = r0 + k * rs;
            float a = acc[k];
#pragma unroll 8
            for (int j = 0; j < SB; ++j) a = fmaf(Gs[i * (SB + 1) + j], Xs[j * XP + p], a);
            acc[k] = a;
        }
    }

    // Carried-state term: sum_n C[t,n] Sprev[p,n], Sprev^T staged in 32-wide n blocks.
    const T* Sp = Sprev + ((b * nc + c) * H + h) * P * N;
    for (int64_t n0 = 0; n0 < N; n0 += SB) {
        const int nb = (int)min((int64_t)SB, N - n0);   // 16 when N == 16
        __syncthreads();
        for (int idx = threadIdx.x; idx < SB * P; idx += kThreads) {
            const int pp = idx / SB, j = idx % SB;    // coalesced along n
            Xs[j * XP + pp] = j < nb ? to_f32(Sp[pp * N + n0 + j]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k >= nrow) break;
            const int i = r0 + k * rs;
            float a = accs[k];
            for (int j = 0; j < nb; ++j) a = fmaf(Cs[i * N + n0 + j], Xs[j * XP + p], a);
            accs[k] = a;
        }
    }

    const float Dh = D ? D[h] : 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if (k >= nrow) break;
        const int i = r0 + k * rs;
        const int64_t t = q0 + i;
        if (t >= q1) continue;
        const float v = acc[k] + ex2(ct[i]) * accs[k] + Dh * to_f32(x[b * io.xb + t * io.xt + h * P + p]);
        y[b * io.yb + t * io.yt + h * P + p] = from_f32<TY>(v);
    }
}

size_t chunk_out_smem(const Dims& d) {
    constexpr int TT = 32, SB = 32;
    return sizeof(float) * (TT * d.N + SB * (d.N + 1) + SB * (d.P + 1) + TT * (SB + 1) + TT + 2 * SB);
}

}  // namespace

cudaError_t launch_chunk_state_simt(const Dims& d, const void* x, const void* B,
                                    const float* cum2, const float* dtT, float* dS,
                                    int32_t* /*err*/, cudaStream_t st) {
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    const dim3 grid((unsigned)(d.b * d.nc * d.H), (unsigned)((d.P + 63) / 64),
                    (unsigned)((d.N + 63) / 64));
    if (d.dtype == 1)
        chunk_state_simt_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(B), cum2,
            dtT, dS, d.T, d.H, d.P, d.N, d.G, d.L, d.nc, io_strides(d));
    else
        chunk_state_simt_kernel<float><<<grid, kThreads, 0, st>>>(
            static_cast<const float*>(x), static_cast<const float*>(B), cum2, dtT, dS, d.T, d.H,
            d.P, d.N, d.G, d.L, d.nc, io_strides(d));
    return cudaGetLastError();
}

cudaError_t launch_chunk_out_simt(const Dims& d, const void* x, const void* B, const void* C,
                                  const float* cum2, const float* dtT, const void* Sprev,
                                  const float* D, void* y, int32_t* /*err*/, cudaStream_t st,
                                  bool y32) {
    if (d.b == 0 || d.H == 0 || d.nc == 0) return cudaSuccess;
    const size_t smem = chunk_out_smem(d);
    const dim3 grid((unsigned)(d.b * d.nc * d.H), (unsigned)(d.L / 32));
    cudaError_t e;
    if (d.dtype == 1 && y32) {
        auto k = chunk_out_simt_kernel<__nv_bfloat16, float>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kThreads, smem, st>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(B),
            static_cast<const __nv_bfloat16*>(C), cum2, dtT,
            static_cast<const __nv_bfloat16*>(Sprev), D, static_cast<float*>(y), d.T,
            d.H, d.P, d.N, d.G, d.L, d.nc, io_strides(d));
    } else if (d.dtype == 1) {
        auto k = chunk_out_simt_kernel<__nv_bfloat16, __nv_bfloat16>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kThreads, smem, st>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(B),
            static_cast<const __nv_bfloat16*>(C), cum2, dtT,
            static_cast<const __nv_bfloat16*>(Sprev), D, static_cast<__nv_bfloat16*>(y), d.T,
            d.H, d.P, d.N, d.G, d.L, d.nc, io_strides(d));
    } else {
        auto k = chunk_out_simt_kernel<float, float>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kThreads, smem, st>>>(
            static_cast<const float*>(x), static_cast<const float*>(B),
            static_cast<const float*>(C), cum2, dtT, static_cast<const float*>(Sprev), D,
            static_cast<float*>(y), d.T, d.H, d.P, d.N, d.G, d.L, d.nc, io_strides(d));
    }
    return cudaGetLastError();
}

}  // namespace m2
