// decode.cu -- one recurrent step per (b, h): the single-token form of the model.
//
// Pages: "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr), "Mamba-2
// 아키텍처의 핵심 연산" (the recurrent read-out of the state), with the state update
// of the chunked path (decay exp(dt A) on the state, dt x B^T as the input):
//
//   S <- exp2(log2(e) dt A) S + dt x B^T        (S: P x N, fp32, updated in place)
//   y  = S C + D x
//
// A pure stream of the state: 8 bytes per state element (read + write), with a
// few hundred bytes of x, B, C and y per head beside it.  At the 2.7B layer's
// state (640 heads of 32 KB) the whole state of the step fits in the GPU's
// shared memory at once, so the kernel is one wave whose speed is set by how
// many bytes each SM has in flight.
//
// N = 128 or 256 (staged kernel): a head's P rows are split over `nsplit` CTAs
// of four warps (about 16 KB of state each, which balances the SMs better than
// one CTA per head).  One thread copies each warp's contiguous slice of rows into
// shared memory with a bulk copy (cp.async.bulk) on the warp's own mbarrier, so
// the whole slice is in flight at once with no registers held; the warp then
// updates its rows from shared memory, lane l owning the float4s n = 4 l + 128 j,
// and writes them back with 512-byte coalesced stores.  The wait is bounded: a
// wait that runs out sets kErrTimeoutDecode and the warp returns.
//
// Other N (scalar kernel): one CTA per (b, h), a warp per state row (rows warp,
// warp + 8, ...), four rows' loads in flight, lane l holding n = l + 32 k.
//
// Both: B and C of the head's group are held in registers and y_p is the
// warp-sum of S_p . C plus D x_p.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc5.cuh"

namespace m2 {
namespace {
using namespace tc;

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

constexpr int kSW = 4;                        // warps of the staged kernel
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr int kSliceBytes = 16 * 1024;        // target state bytes per CTA

// CTA s of head bh (blockIdx.x = bh * nsplit + s) owns rows [s R, min(P, s R + R));
// warp w owns the contiguous slice of rw = ceil(R / 4) rows starting at s R + w rw.
template <typename TI, int NV>
__global__ void __launch_bounds__(kSW * 32)
decode_staged_kernel(float* __restrict__ S, const TI* __restrict__ x, const float* __restrict__ dt,
                     const float* __restrict__ A, const TI* __restrict__ B,
                     const TI* __restrict__ C, const float* __restrict__ D, TI* __restrict__ y,
                     int H, int P, int G, int R, int nsplit, int32_t* err) {
    constexpr int N = 128 * NV, kRowV = N / 4;   // float4s per row
    extern __shared__ __align__(128) float4 rows[];
    __shared__ uint64_t bars[kSW];
    const int bh = blockIdx.x / nsplit, s = blockIdx.x % nsplit;
    const int b = bh / H, h = bh % H;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pa = s * R, pb = min(P, pa + R);
    const int rw = (R + kSW - 1) / kSW;
    float4* Sh = reinterpret_cast<float4*>(S + (int64_t)bh * P * N);
    if (threadIdx.x == 0) {
        for (int w = 0; w < kSW; ++w) mbar_init(&bars[w], 1);
        fence_barrier_init();
        for (int w = 0; w < kSW; ++w) {
            const int a = pa + w * rw, e = min(pb, a + rw);
            if (e <= a) break;
            const uint32_t bytes = (uint32_t)(e - a) * (uint32_t)(N * 4);
            mbar_arrive_expect_tx(&bars[w], bytes);
            bulk_load(rows + (a - pa) * kRowV, Sh + (int64_t)a * kRowV, bytes, &bars[w]);
        }
    }
    const float dth = __ldg(dt + bh);
    const float decay = ex2(dth * __ldg(A + h) * kLog2e);
    const float dh = D ? __ldg(D + h) : 0.f;
    float bn[NV][4], cn[NV][4];
    const TI* Bg = B + ((int64_t)b * G + g) * N;
    const TI* Cg = C + ((int64_t)b * G + g) * N;
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bn[j][e] = to_f32(Bg[4 * lane + 128 * j + e]);
            cn[j][e] = to_f32(Cg[4 * lane + 128 * j + e]);
        }
    __syncthreads();   // the barriers are initialised before any warp waits on one
    const int wa = pa + warp * rw, wb = min(pb, wa + rw);
    if (wb <= wa) return;
    if (!mbar_wait(&bars[warp], 0, kWaitNs)) {
        if (lane == 0) record_error(err, kErrTimeoutDecode);
        return;
    }
    for (int p = wa; p < wb; ++p) {
        const float xp = to_f32(x[(int64_t)bh * P + p]);
        const float u = dth * xp;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float4 v = rows[(p - pa) * kRowV + lane + 32 * j];
            v.x = fmaf(decay, v.x, u * bn[j][0]);
            v.y = fmaf(decay, v.y, u * bn[j][1]);
            v.z = fmaf(decay, v.z, u * bn[j][2]);
            v.w = fmaf(decay, v.w, u * bn[j][3]);
            Sh[(int64_t)p * kRowV + lane + 32 * j] = v;
            acc = fmaf(v.x, cn[j][0], acc);
            acc = fmaf(v.y, cn[j][1], acc);
            acc = fmaf(v.z, cn[j][2], acc);
            acc = fmaf(v.w, cn[j][3], acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) y[(int64_t)bh * P + p] = from_f32<TI>(fmaf(dh, xp, acc));
    }
}

template <typename TI, int NV>
cudaError_t launch_staged(const Dims& d, float* S, const void* x, const float* dt, const float* A,
                          const void* B, const void* C, const float* D, void* y, int32_t* err,
                          cudaStream_t st) {
    const int64_t head_bytes = d.P * d.N * 4;
    int nsplit = (int)std::min<int64_t>(d.P, std::max<int64_t>(1, (head_bytes + kSliceBytes - 1) / kSliceBytes));
    const int R = (int)((d.P + nsplit - 1) / nsplit);
    nsplit = (int)((d.P + R - 1) / R);   // no CTA without rows
    const size_t smem = (size_t)R * d.N * 4;   // <= kSliceBytes + one row: under the 48 KB default
    if (d.b * d.H * nsplit >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    auto k = decode_staged_kernel<TI, NV>;
    k<<<(unsigned)(d.b * d.H * nsplit), kSW * 32, smem, st>>>(
        S, static_cast<const TI*>(x), dt, A, static_cast<const TI*>(B), static_cast<const TI*>(C), D,
        static_cast<TI*>(y), (int)d.H, (int)d.P, (int)d.G, R, nsplit, err);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t launch_t(const Dims& d, float* S, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* D, void* y, int32_t* err,
                     cudaStream_t st) {
    if (d.N == 128) return launch_staged<TI, 1>(d, S, x, dt, A, B, C, D, y, err, st);
    if (d.N == 256) return launch_staged<TI, 2>(d, S, x, dt, A, B, C, D, y, err, st);
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
                          const void* B, const void* C, const float* D, void* y, int32_t* err,
                          cudaStream_t st) {
    if (d.b == 0 || d.H == 0) return cudaSuccess;
    if (d.b * d.H >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    return d.dtype == 1 ? launch_t<__nv_bfloat16>(d, S, x, dt, A, B, C, D, y, err, st)
                        : launch_t<float>(d, S, x, dt, A, B, C, D, y, err, st);
}

}  // namespace m2
