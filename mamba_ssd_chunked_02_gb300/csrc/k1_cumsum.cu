// k1_cumsum.cu -- stage 1: chunk-local decay cumsum in log2 space, [b,h,t] layout.
//
// Pages: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile" (brifing.si), section 7 "Optimizing chunk_cumsum Kernel":
// per-token, per-head cumulative sums of the decay term, scaled by log2(e) so
// that later stages use exp2.  "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널
// 가속화" (devin.kr), "cuTile 기반 성능 최적화 기법": dt and the decay cumsum are
// stored in a [batch, head, token] layout so that later loads are contiguous.
//
// cum2[b,h,t] = log2(e) * sum_{r = chunk start}^{t} dt[b,r,h] * A[h]   (inclusive)
// dtT[b,h,t]  = dt[b,t,h]
//
// One CTA per (chunk, batch, block of 16 heads; more CTAs than with 32 hide
// more of the load latency of this one-wave kernel).  The [L x 16] dt tile is
// read with coalesced 64-byte rows (16 heads of one token; 16-byte loads, all of
// a thread's loads issued before any is stored), transposed into shared memory,
// scanned by one warp per head (each lane owns L/32 consecutive tokens; lane
// totals are combined with a shuffle scan), and each lane writes its tokens of
// the [h][t] rows straight from registers (16-byte stores).  The shared tile
// keeps one padding word per 32 tokens, which keeps a warp's reads of one row
// free of bank conflicts, and a row pitch of 2 mod 8 words: a warp's
// transposing stores cover 8 tokens of 4 heads, and heads 4 apart then sit 8
// banks apart, so those stores are conflict-free too.  HBM-bound: 12 bytes per
// (token, head).
// On the fused path the kernel also clears the next kernel's ticket and flag
// words.
#include "common.cuh"
#include "internal.h"

namespace m2 {
namespace {

constexpr int kHB = 16;        // heads per CTA
constexpr int kThreads = 256;  // 8 warps

// Token i of a head's row sits at i + i / 32; rows are `pitch` words apart.
__device__ __forceinline__ int tpos(int i) { return i + (i >> 5); }

template <int L>
__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const float* __restrict__ dt, const float* __restrict__ A,
                    float* __restrict__ cum2, float* __restrict__ dtT, int64_t T, int64_t H,
                    int64_t sb, int64_t stt, int32_t* __restrict__ zero, int64_t nzero) {
    constexpr int kRow = L + L / 32;
    constexpr int kPitch = kRow + ((2 - kRow) & 7);   // 2 mod 8
    __shared__ float tile[kHB * kPitch];
    const int64_t c = blockIdx.x, b = blockIdx.y, h0 = (int64_t)blockIdx.z * kHB;
    // Launched as a programmatic dependent (the whole-path call), this grid may
    // start while the stream's previous kernel drains: nothing here runs before
    // that kernel has completed.  Then stage 2 may start its loads of x and B (the
    // call's inputs, complete by now); it waits for this grid before reading
    // cum2/dtT.
    grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_launch();
    // Clear the next kernel's synchronisation words (grid-stride).
    if (zero) {
        const int64_t cta = c + (int64_t)gridDim.x * (b + (int64_t)gridDim.y * blockIdx.z);
        const int64_t stride = (int64_t)gridDim.x * gridDim.y * gridDim.z * kThreads;
        for (int64_t i = cta * kThreads + threadIdx.x; i < nzero; i += stride) zero[i] = 0;
    }
    const int64_t t0 = c * L;
    const int nt = (int)min((int64_t)L, T - t0);
    const int nh = (int)min((int64_t)kHB, H - h0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* src = dt + b * sb + t0 * stt + h0;   // dt[b, t, h]: strides sb, stt, 1

    // Load [nt x nh] (token-major in HBM) and transpose into tile[head][token].
    if (nh == kHB && (H & 3) == 0 && (stt & 3) == 0 && (sb & 3) == 0) {
        // kHB/4 float4 per token row; element (token i, quad q) of item idx = i * kQ + q.
        constexpr int kQ = kHB / 4;
        constexpr int kPer = L * kHB / 4 / kThreads;
        float4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + kThreads * k, i = idx / kQ, q = idx % kQ;
            v[k] = i < nt ? __ldg(reinterpret_cast<const float4*>(src + (int64_t)i * stt) + q)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + kThreads * k, i = idx / kQ, j = 4 * (idx % kQ);
            tile[(j + 0) * kPitch + tpos(i)] = v[k].x;
            tile[(j + 1) * kPitch + tpos(i)] = v[k].y;
            tile[(j + 2) * kPitch + tpos(i)] = v[k].z;
            tile[(j + 3) * kPitch + tpos(i)] = v[k].w;
        }
    } else {
        for (int idx = threadIdx.x; idx < L * kHB; idx += kThreads) {
            const int i = idx / kHB, j = idx % kHB;
            tile[j * kPitch + tpos(i)] = (i < nt && j < nh) ? __ldg(src + (int64_t)i * stt + j) : 0.f;
        }
    }
    __syncthreads();

    // One warp per head.  L >= 128: the row is cut into L/128 segments of 128
    // tokens, lane l owning tokens 4l .. 4l+3 of each; the segments are scanned in
    // order (a 4-token local sum per lane, a shuffle scan of the lane totals, the
    // running total carried to the next segment), so that each lane writes its
    // four dtT and cum2 values of a segment with one 16-byte store each and a
    // warp's stores cover 512 contiguous bytes.  L = 64: two tokens per lane.
    constexpr int kSeg = L >= 128 ? L / 128 : 1, kPer = L >= 128 ? 4 : L / 32;
    const bool vec = L >= 128 && (T & 3) == 0;   // row starts (b H + h) T + c L 16-byte aligned
    for (int j = warp; j < nh; j += kThreads / 32) {
        const int64_t row = (b * H + h0 + j) * T + t0;
        const float* trow = tile + j * kPitch;
        const float a2 = __ldg(A + h0 + j) * kLog2e;
        float carry = 0.f;
#pragma unroll
        for (int sg = 0; sg < kSeg; ++sg) {
            const int i0 = sg * 128 + lane * kPer;
            float dv[kPer], sv[kPer];
            float run = 0.f;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                dv[k] = trow[tpos(i0 + k)];   // tokens past T hold 0
                run += dv[k] * a2;
                sv[k] = run;
            }
            float tot = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, tot, o);
                if (lane >= o) tot += n;
            }
            const float excl = carry + tot - run;
#pragma unroll
            for (int k = 0; k < kPer; ++k) sv[k] += excl;
            carry += __shfl_sync(0xffffffffu, tot, 31);
            if (vec && i0 + kPer <= nt) {
                *reinterpret_cast<float4*>(dtT + row + i0) = make_float4(dv[0], dv[1], dv[2], dv[3 % kPer]);
                *reinterpret_cast<float4*>(cum2 + row + i0) = make_float4(sv[0], sv[1], sv[2], sv[3 % kPer]);
            } else {
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                    if (i0 + k < nt) {
                        dtT[row + i0 + k] = dv[k];
                        cum2[row + i0 + k] = sv[k];
                    }
            }
        }
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, float* cum2,
                                float* dtT, int32_t* /*err*/, cudaStream_t st, int32_t* zero,
                                int64_t nzero, bool pdl) {
    if (d.b == 0 || d.H == 0 || d.T == 0) return cudaSuccess;
    const dim3 grid((unsigned)d.nc, (unsigned)d.b, (unsigned)((d.H + kHB - 1) / kHB));
    switch (d.L) {
        case 64:
            return launch_kernel(chunk_cumsum_kernel<64>, grid, dim3(kThreads), 0, st, pdl, dt, A, cum2, dtT,
                                 (int64_t)d.T, (int64_t)d.H, (int64_t)d.sdt[0], (int64_t)d.sdt[1], zero, nzero);
        case 128:
            return launch_kernel(chunk_cumsum_kernel<128>, grid, dim3(kThreads), 0, st, pdl, dt, A, cum2, dtT,
                                 (int64_t)d.T, (int64_t)d.H, (int64_t)d.sdt[0], (int64_t)d.sdt[1], zero, nzero);
        case 256:
            return launch_kernel(chunk_cumsum_kernel<256>, grid, dim3(kThreads), 0, st, pdl, dt, A, cum2, dtT,
                                 (int64_t)d.T, (int64_t)d.H, (int64_t)d.sdt[0], (int64_t)d.sdt[1], zero, nzero);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m2
