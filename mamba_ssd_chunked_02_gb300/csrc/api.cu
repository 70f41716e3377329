// api.cu -- the C ABI declared in include/mamba2_ssd.h: argument validation,
// workspace carving and the launch sequence of the four stages.
//
// Pages: "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
// "세 가지 핵심 커널 구현" (chunk_cumsum -> fwd_pass_state -> compute_out);
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile" (brifing.si), section 6 "The Three Custom Kernels".  The pages'
// state kernel is split here into a parallel chunk-state contraction (stage 2)
// and a sequential pass over chunks (stage 3).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "mamba2_ssd.h"

using m2::Dims;

namespace {

// Device-side error word (see mamba2_ssd_device_error).  Kernels receive its
// device address; it is read back only on request.
__device__ int32_t g_device_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_sym_mu;
int32_t* g_sym_addr[kMaxDevices] = {};

int32_t* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_sym_mu);
    if (!g_sym_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
            cudaGetLastError();   // the failed lookup must not surface in a later launch check
            return nullptr;
        }
        g_sym_addr[dev] = static_cast<int32_t*>(p);
    }
    return g_sym_addr[dev];
}

bool in_set(int64_t v, std::initializer_list<int64_t> s) {
    for (int64_t e : s)
        if (v == e) return true;
    return false;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mamba2_status check(const mamba2_ssd_shape* s) {
    if (!s) return MAMBA2_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 0) return MAMBA2_ERR_INVALID_ARG;
    if (s->headdim <= 0 || s->dstate <= 0 || s->ngroups <= 0 || s->chunk_size <= 0)
        return MAMBA2_ERR_INVALID_ARG;
    if (s->dtype != MAMBA2_F32 && s->dtype != MAMBA2_BF16) return MAMBA2_ERR_INVALID_ARG;
    if (s->flags & ~(MAMBA2_FLAG_FORCE_SIMT | MAMBA2_FLAG_FUSED_STATE | MAMBA2_FLAG_DS_BF16 |
                     MAMBA2_FLAG_SERIAL))
        return MAMBA2_ERR_INVALID_ARG;
    if (s->nheads % s->ngroups != 0) return MAMBA2_ERR_INVALID_ARG;
    if (!in_set(s->headdim, {16, 32, 64, 128})) return MAMBA2_ERR_UNSUPPORTED;
    if (!in_set(s->dstate, {16, 32, 64, 128, 256})) return MAMBA2_ERR_UNSUPPORTED;
    if (!in_set(s->chunk_size, {64, 128, 256})) return MAMBA2_ERR_UNSUPPORTED;
    // Launch-grid limits (grid y/z dimensions and 32-bit grid x products).
    if (s->batch > 65535) return MAMBA2_ERR_UNSUPPORTED;
    if (s->seqlen > (int64_t(1) << 31) || s->nheads > 65535) return MAMBA2_ERR_UNSUPPORTED;
    const int64_t nc = (s->seqlen + s->chunk_size - 1) / s->chunk_size;
    if (s->batch * nc * s->nheads >= (int64_t(1) << 31)) return MAMBA2_ERR_UNSUPPORTED;
    return MAMBA2_OK;
}

Dims dims_of(const mamba2_ssd_shape* s) {
    Dims d;
    d.b = s->batch; d.T = s->seqlen; d.H = s->nheads; d.P = s->headdim; d.N = s->dstate;
    d.G = s->ngroups; d.L = s->chunk_size; d.nc = (d.T + d.L - 1) / d.L;
    d.dtype = s->dtype == MAMBA2_BF16 ? 1 : 0;
    m2::set_contiguous(d);
    return d;
}

// Strides of mamba2_ssd_fwd_strided into d: each token stride at least the
// token's extent, each batch stride at least T token strides (batch strides are
// not used with one batch entry and are set to that then), T token strides and
// each batch stride below 2^40 elements.
mamba2_status set_strides(Dims& d, const mamba2_ssd_strides* st) {
    auto one = [&](const int64_t (&in)[2], int64_t extent, int64_t (&out)[2]) -> bool {
        const int64_t lim = int64_t(1) << 40;
        if (in[1] < extent || in[1] <= 0) return false;
        if (d.T > 0 && in[1] > (lim - 1) / d.T) return false;
        const int64_t bs = d.b > 1 ? in[0] : d.T * in[1];
        if (bs < d.T * in[1] || bs >= lim) return false;
        out[0] = bs;
        out[1] = in[1];
        return true;
    };
    if (!st) return MAMBA2_ERR_INVALID_ARG;
    return one(st->x, d.H * d.P, d.sx) && one(st->y, d.H * d.P, d.sy) && one(st->B, d.G * d.N, d.sB) &&
                   one(st->C, d.G * d.N, d.sC) && one(st->dt, d.H, d.sdt)
               ? MAMBA2_OK
               : MAMBA2_ERR_INVALID_ARG;
}

// The tensor-core kernels move x, y, B and C with tensor-memory-accelerator
// copies, whose global strides must be multiples of 16 bytes.
bool tma_strides(const Dims& d) {
    const int64_t es = m2::esize(d);
    for (const int64_t* v : {d.sx, d.sy, d.sB, d.sC})
        if ((v[0] * es) % 16 || (v[1] * es) % 16) return false;
    return true;
}

bool use_tc(const mamba2_ssd_shape* s, const Dims& d) {
    return !(s->flags & MAMBA2_FLAG_FORCE_SIMT) && m2::tc_supported(d);
}

// The dimensions the whole-path call runs with.  A chunk length of 64 on a shape
// the tensor cores take at 128 runs as 128-token chunks: y and the final state
// do not depend on the chunk length (only the intermediates do, and the
// whole-path call does not return them), and a 64-row query tile would leave
// half of every tcgen05 MMA's rows idle.  The workspace this needs is never
// larger than the one mamba2_ssd_workspace_size reports for the shape.
Dims whole_dims(const mamba2_ssd_shape* s) {
    Dims d = dims_of(s);
    if (d.L == 64 && !(s->flags & MAMBA2_FLAG_FORCE_SIMT)) {
        Dims e = d;
        e.L = 128;
        e.nc = (d.T + 127) / 128;
        if (m2::tc_supported(e)) return e;
    }
    return d;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct Carve {
    size_t cum2, dtT, dS, Sprev, xabs, total;
};

Carve carve(const Dims& d) {
    Carve c;
    c.cum2 = 0;
    c.dtT = c.cum2 + align256(sizeof(float) * (size_t)m2::n_cum(d));
    c.dS = c.dtT + align256(sizeof(float) * (size_t)m2::n_cum(d));
    c.Sprev = c.dS + align256(sizeof(float) * (size_t)m2::n_state(d));
    c.xabs = c.Sprev + align256((size_t)m2::esize(d) * (size_t)m2::n_state(d));
    // max |x| per (b, chunk, tensor-core head): H heads, or 2H at P = 128 (tc_view)
    c.total = c.xabs + align256(8 * sizeof(uint32_t) * (size_t)(d.b * d.nc * m2::tc_view(d).H));
    return c;
}

// Workspace of the backward pass: the forward's cum2, dtT, dS (fp32; reused for
// the chunk adjoints dSout / Gn), Sprev in the I/O type, the final state, an
// I/O-type copy of Gn, y without the skip term and y' (fp32; on the tensor-core
// path instead three per-token dots: dy . y, x . y' and dy . x), the reordered
// inputs of the output runs, Sprev^T and Gn^T, the per-run-head cum2 / dt rows,
// and the dC / dB runs' per-head outputs (I/O type).
struct BwdCarve {
    size_t cum2, dtT, dS, Sprev, fin, GnIO, yno, yr, dyr, Br, Cr, cum2r, ones, xB, xCr, xr,
        SprevT, GnT, cum2d, dtTd, cum2rd, onesd, yC, zB, ydot2, xyd2, dyxd2, xabs_x, xabs_dy, total;
};

// copies: the dC / dB runs take the CUDA cores and read per-head copies (xB,
// xCr) and per-run-head rows (cum2d, dtTd, cum2rd, onesd); the tensor-core runs
// read B, C reversed and the per-head rows directly.
// half: the tensor-core path, where dS and then the chunk adjoints are held in
// bf16 (the forward's hand-off of R15; Gn itself only in the I/O type).
// xr: the dB run reads x reversed (not when dC and dB come from bwd_bc_tc).
BwdCarve bwd_carve(const Dims& d, bool copies, bool dot, bool half, bool xr) {
    BwdCarve c;
    const size_t E = (size_t)m2::esize(d);
    const size_t Q = d.N >= 64 ? (size_t)(d.N / 64) : 1;
    const size_t cum = align256(sizeof(float) * (size_t)m2::n_cum(d));
    const size_t cumq = align256(sizeof(float) * Q * (size_t)m2::n_cum(d));
    const size_t st32 = align256(sizeof(float) * (size_t)m2::n_state(d));
    const size_t stE = align256(E * (size_t)m2::n_state(d));
    const size_t xyE = align256(E * (size_t)(d.b * d.T * d.H * d.P));
    const size_t xy32 = align256(sizeof(float) * (size_t)(d.b * d.T * d.H * d.P));
    const size_t bcE = align256(E * (size_t)(d.b * d.T * d.G * d.N));
    const size_t hnE = align256(E * (size_t)(d.b * d.T * d.H * d.N));
    size_t o = 0;
    auto take = [&](size_t& f, size_t n) { f = o; o += n; };
    take(c.cum2, cum);
    take(c.dtT, cum);
    take(c.dS, half ? stE : st32);
    take(c.Sprev, stE);
    take(c.fin, align256(sizeof(float) * (size_t)(d.b * d.H * d.P * d.N)));
    take(c.GnIO, stE);
    take(c.yno, dot ? 0 : xy32);   // dot mode: the y run writes only dy . y (ydot2)
    take(c.yr, dot ? 0 : xy32);   // dot mode: the y' run writes dx and two dots per token
    // the reversed inputs of the y' run (dot mode: the run is anti-causal on the inputs)
    take(c.dyr, dot ? 0 : xyE);
    take(c.Br, dot ? 0 : bcE);
    take(c.Cr, dot ? 0 : bcE);
    take(c.cum2r, dot ? 0 : cum);
    take(c.ones, dot ? 0 : cum);   // dot mode: the y' run takes dt' = 1 without rows
    take(c.xB, copies ? hnE : 0);
    take(c.xCr, copies ? hnE : 0);
    take(c.xr, xr ? xyE : 0);
    take(c.SprevT, copies ? stE : 0);   // the tensor-core runs read them untransposed
    take(c.GnT, copies ? stE : 0);
    take(c.cum2d, copies ? cumq : 0);
    take(c.dtTd, copies ? cumq : 0);
    take(c.cum2rd, copies ? cumq : 0);
    take(c.onesd, copies ? cumq : 0);
    take(c.yC, copies ? hnE : 0);   // the tensor-core dC run adds into dC directly
    take(c.zB, copies ? hnE : 0);   // the tensor-core dB run adds into dB directly
    const size_t dots = dot ? align256(sizeof(float) * 2 * (size_t)(d.b * d.H * d.T)) : 0;
    take(c.ydot2, dots);
    take(c.xyd2, dots);
    take(c.dyxd2, dots);
    // max |x| and max |dy| per (b, chunk, head) from the stage-2 runs, for the y and
    // y' runs' fp16 range check (the forward's hand-off of the same bound)
    const size_t xab = half ? align256(8 * sizeof(uint32_t) * (size_t)(d.b * d.nc * d.H)) : 0;
    take(c.xabs_x, xab);
    take(c.xabs_dy, xab);
    c.total = o;
    return c;
}

mamba2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MAMBA2_OK : MAMBA2_ERR_CUDA; }

// The backward's tensor-core choices: its own runs (P = 64 only), and whether
// its dC / dB runs take the tensor cores (then without per-head copies).
bool bwd_tc(const mamba2_ssd_shape* s, const Dims& d) { return use_tc(s, d) && d.P == 64; }
bool bwd_copies(const mamba2_ssd_shape* s, const Dims& d) {
    return !(bwd_tc(s, d) && m2::tc_supported(m2::bwd_run_dims(d)));
}
// dC and dB from their own tensor-core kernel (no reversed copy of x).
bool bwd_bc(const mamba2_ssd_shape* s, const Dims& d) {
    return !bwd_copies(s, d) && m2::bwd_bc_tc_supported(d);
}

// A required pointer: non-null and 16-byte aligned, unless the tensor is empty.
bool req(const void* p, bool empty) { return empty || (p && aligned16(p)); }
// An optional pointer: null, or 16-byte aligned.
bool opt(const void* p) { return !p || aligned16(p); }

}  // namespace

extern "C" {

mamba2_status mamba2_ssd_check_shape(const mamba2_ssd_shape* shape) { return check(shape); }

int32_t mamba2_ssd_path(const mamba2_ssd_shape* shape) {
    if (check(shape) != MAMBA2_OK) return -1;
    return use_tc(shape, whole_dims(shape)) ? MAMBA2_PATH_TCGEN05 : MAMBA2_PATH_SIMT;
}

size_t mamba2_ssd_workspace_size(const mamba2_ssd_shape* shape) {
    if (check(shape) != MAMBA2_OK) return 0;
    return carve(dims_of(shape)).total;
}

mamba2_status mamba2_ssd_chunk_cumsum(const mamba2_ssd_shape* shape, const float* dt,
                                      const float* A, float* cum2, float* dtT, void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(dt, empty) || !req(A, empty) || !req(cum2, empty) || !req(dtT, empty))
        return MAMBA2_ERR_INVALID_ARG;
    return from_cuda(m2::launch_chunk_cumsum(d, dt, A, cum2, dtT, error_word(),
                                             static_cast<cudaStream_t>(stream)));
}

mamba2_status mamba2_ssd_chunk_state(const mamba2_ssd_shape* shape, const void* x, const void* B,
                                     const float* cum2, const float* dtT, void* dS,
                                     void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    const bool ds16 = shape->flags & MAMBA2_FLAG_DS_BF16;
    if (ds16 && !use_tc(shape, d)) return MAMBA2_ERR_UNSUPPORTED;
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(x, empty) || !req(B, empty) || !req(cum2, empty) || !req(dtT, empty) ||
        !req(dS, empty))
        return MAMBA2_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = use_tc(shape, d)
                        ? m2::launch_chunk_state_tc(d, x, B, cum2, dtT, dS, ds16, error_word(), s)
                        : m2::launch_chunk_state_simt(d, x, B, cum2, dtT, static_cast<float*>(dS),
                                                      error_word(), s);
    return from_cuda(e);
}

mamba2_status mamba2_ssd_state_pass(const mamba2_ssd_shape* shape, const void* dS,
                                    const float* cum2, const float* initial_state, void* Sprev,
                                    float* final_state, void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    const bool ds16 = shape->flags & MAMBA2_FLAG_DS_BF16;
    if (ds16 && d.dtype != 1) return MAMBA2_ERR_UNSUPPORTED;
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(dS, empty) || !req(cum2, empty) || !opt(initial_state) || !req(Sprev, empty) ||
        !req(final_state, d.b * d.H == 0))
        return MAMBA2_ERR_INVALID_ARG;
    return from_cuda(m2::launch_state_pass(d, dS, ds16, cum2, initial_state, Sprev, final_state,
                                           error_word(), static_cast<cudaStream_t>(stream)));
}

size_t mamba2_ssd_chunk_state_pass_workspace_size(const mamba2_ssd_shape* shape) {
    if (check(shape) != MAMBA2_OK) return 0;
    const Dims d = dims_of(shape);
    if (!use_tc(shape, d) || !m2::tc_fused_supported(d)) return 0;
    return align256(2 * sizeof(float) * (size_t)(d.b * d.H * d.P * d.N)) +
           align256(sizeof(int32_t) * (size_t)(m2::fused_flag_words(d) + 1));
}

mamba2_status mamba2_ssd_chunk_state_pass(const mamba2_ssd_shape* shape, const void* x,
                                          const void* B, const float* cum2, const float* dtT,
                                          const float* initial_state, void* Sprev,
                                          float* final_state, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    if (!use_tc(shape, d) || !m2::tc_fused_supported(d)) return MAMBA2_ERR_UNSUPPORTED;
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(x, empty) || !req(B, empty) || !req(cum2, empty) || !req(dtT, empty) ||
        !opt(initial_state) || !req(Sprev, empty) || !req(final_state, d.b * d.H == 0))
        return MAMBA2_ERR_INVALID_ARG;
    if (d.b * d.H == 0) return MAMBA2_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d.T == 0)
        return from_cuda(m2::launch_state_pass(d, nullptr, false, nullptr, initial_state, nullptr,
                                               final_state, error_word(), s));
    const size_t ring = align256(2 * sizeof(float) * (size_t)(d.b * d.H * d.P * d.N));
    const size_t nflag = (size_t)m2::fused_flag_words(d);
    if (!workspace || workspace_bytes < mamba2_ssd_chunk_state_pass_workspace_size(shape) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MAMBA2_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    int32_t* flags = reinterpret_cast<int32_t*>(ws + ring);
    cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(int32_t) * (nflag + 1), s);
    if (e == cudaSuccess)
        e = m2::launch_chunk_state_pass_tc(d, x, B, cum2, dtT, initial_state,
                                           reinterpret_cast<float*>(ws), flags, flags + nflag,
                                           Sprev, final_state, error_word(), s);
    return from_cuda(e);
}

mamba2_status mamba2_ssd_chunk_out(const mamba2_ssd_shape* shape, const void* x, const void* B,
                                   const void* C, const float* cum2, const float* dtT,
                                   const void* Sprev, const float* D, void* y, void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(x, empty) || !req(B, empty) || !req(C, empty) || !req(cum2, empty) ||
        !req(dtT, empty) || !req(Sprev, empty) || !opt(D) || !req(y, empty))
        return MAMBA2_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = use_tc(shape, d)
                        ? m2::launch_chunk_out_tc(d, x, B, C, cum2, dtT, Sprev, D, y, error_word(), s)
                        : m2::launch_chunk_out_simt(d, x, B, C, cum2, dtT, Sprev, D, y, error_word(), s);
    return from_cuda(e);
}

}  // extern "C"

namespace {

// The whole path; events (five cudaEvent_t or null) are recorded before stage 1,
// after each stage and after stage 4 (stages 2 and 3 share one event when fused).
mamba2_status fwd_impl(const mamba2_ssd_shape* shape, const void* x, const float* dt,
                       const float* A, const void* B, const void* C, const float* D,
                       const float* initial_state, void* y, float* final_state, void* workspace,
                       size_t workspace_bytes, void* stream, void* const* events,
                       const mamba2_ssd_strides* strides = nullptr) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    Dims d = whole_dims(shape);
    if (strides && (st = set_strides(d, strides)) != MAMBA2_OK) return st;
    const bool empty = d.b * d.T * d.H == 0;
    if (!req(x, empty) || !req(dt, empty) || !req(A, empty) || !req(B, empty) ||
        !req(C, empty) || !opt(D) || !opt(initial_state) || !req(y, empty) ||
        !req(final_state, d.b * d.H == 0))
        return MAMBA2_ERR_INVALID_ARG;
    const Carve cv = carve(d);
    if (d.b * d.H == 0) return MAMBA2_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* err = error_word();
    if (d.T == 0)   // final_state = initial_state (or 0); nothing else to write
        return from_cuda(m2::launch_state_pass(d, nullptr, false, nullptr, initial_state, nullptr,
                                               final_state, err, s));
    if (!workspace || workspace_bytes < cv.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MAMBA2_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    float* cum2 = reinterpret_cast<float*>(ws + cv.cum2);
    float* dtT = reinterpret_cast<float*>(ws + cv.dtT);
    float* dS = reinterpret_cast<float*>(ws + cv.dS);
    void* Sprev = ws + cv.Sprev;
    uint32_t* xabs = reinterpret_cast<uint32_t*>(ws + cv.xabs);   // stage 2 -> stage 4: max |x|
    const bool tc = use_tc(shape, d) && tma_strides(d);
    // Fused stages 2+3 (opt-in): the two-slot carried-state ring, the flag words
    // and the ticket live in the dS region, which holds them from three chunks on.
    const size_t ring = 2 * sizeof(float) * (size_t)(d.b * d.H * d.P * d.N);
    const size_t nflag = tc ? (size_t)m2::fused_flag_words(d) : 0;
    const bool fuse = tc && m2::tc_fused_supported(d) && d.nc >= 3 && (shape->flags & MAMBA2_FLAG_FUSED_STATE) &&
                      ring + sizeof(int32_t) * (nflag + 1) <= cv.Sprev - cv.dS;
    int32_t* flags = reinterpret_cast<int32_t*>(ws + cv.dS + ring);
    // Programmatic dependent launch of stages 1-4 (not across recorded events).
    // Stage 1 waits for the stream's previous kernel before anything else and
    // only then lets stage 2 start, so everything queued before this call has
    // completed before any stage reads its inputs; its launch overlaps the tail
    // of that kernel.
    const bool pdl = !(shape->flags & MAMBA2_FLAG_SERIAL) && !events;

    auto mark = [&](int k) -> cudaError_t {
        return (events && events[k]) ? cudaEventRecord(static_cast<cudaEvent_t>(events[k]), s)
                                     : cudaSuccess;
    };
    cudaError_t e = mark(0);
    if (e == cudaSuccess)
        e = fuse ? m2::launch_chunk_cumsum(d, dt, A, cum2, dtT, err, s, flags, (int64_t)nflag + 1)
                 : m2::launch_chunk_cumsum(d, dt, A, cum2, dtT, err, s, nullptr, 0, pdl);
    if (e == cudaSuccess) e = mark(1);
    if (fuse) {
        if (e == cudaSuccess)
            e = m2::launch_chunk_state_pass_tc(d, x, B, cum2, dtT, initial_state, dS, flags,
                                               flags + nflag, Sprev, final_state, err, s);
        if (e == cudaSuccess) e = mark(2);
    } else {
        if (e == cudaSuccess)
            e = tc ? m2::launch_chunk_state_tc(d, x, B, cum2, dtT, dS, true, err, s, xabs, pdl)
                   : m2::launch_chunk_state_simt(d, x, B, cum2, dtT, dS, err, s);
        if (e == cudaSuccess) e = mark(2);
        // On the tensor-core path dS travels between stages 2 and 3 in bf16.
        if (e == cudaSuccess)
            e = m2::launch_state_pass(d, dS, tc, cum2, initial_state, Sprev, final_state, err, s,
                                      pdl);
    }
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess)
        e = tc ? m2::launch_chunk_out_tc(d, x, B, C, cum2, dtT, Sprev, D, y, err, s,
                                         fuse ? nullptr : xabs, pdl && !fuse)
               : m2::launch_chunk_out_simt(d, x, B, C, cum2, dtT, Sprev, D, y, err, s);
    if (e == cudaSuccess) e = mark(4);
    return from_cuda(e);
}

}  // namespace

extern "C" {

mamba2_status mamba2_ssd_fwd(const mamba2_ssd_shape* shape, const void* x, const float* dt,
                             const float* A, const void* B, const void* C, const float* D,
                             const float* initial_state, void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(shape, x, dt, A, B, C, D, initial_state, y, final_state, workspace,
                    workspace_bytes, stream, nullptr);
}

mamba2_status mamba2_ssd_fwd_strided(const mamba2_ssd_shape* shape,
                                     const mamba2_ssd_strides* strides, const void* x,
                                     const float* dt, const float* A, const void* B, const void* C,
                                     const float* D, const float* initial_state, void* y,
                                     float* final_state, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    if (!strides) return MAMBA2_ERR_INVALID_ARG;
    return fwd_impl(shape, x, dt, A, B, C, D, initial_state, y, final_state, workspace,
                    workspace_bytes, stream, nullptr, strides);
}

mamba2_status mamba2_ssd_fwd_timed(const mamba2_ssd_shape* shape, const void* x, const float* dt,
                                   const float* A, const void* B, const void* C, const float* D,
                                   const float* initial_state, void* y, float* final_state,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   void* const* events) {
    return fwd_impl(shape, x, dt, A, B, C, D, initial_state, y, final_state, workspace,
                    workspace_bytes, stream, events);
}

size_t mamba2_ssd_bwd_workspace_size(const mamba2_ssd_shape* shape) {
    if (check(shape) != MAMBA2_OK) return 0;
    const Dims d = dims_of(shape);
    return bwd_carve(d, bwd_copies(shape, d), m2::bwd_dot_mode(d, bwd_tc(shape, d)), bwd_tc(shape, d),
                     !bwd_bc(shape, d)).total;
}

mamba2_status mamba2_ssd_bwd(const mamba2_ssd_shape* shape, const void* x, const float* dt,
                             const float* A, const void* B, const void* C, const float* D,
                             const float* initial_state, const void* dy,
                             const float* dfinal_state, float* dx, float* ddt, float* dA,
                             float* dB, float* dC, float* dD, float* dinitial_state,
                             void* workspace, size_t workspace_bytes, void* stream) {
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    if (shape->flags & ~MAMBA2_FLAG_FORCE_SIMT) return MAMBA2_ERR_INVALID_ARG;
    const Dims d = dims_of(shape);
    const bool empty = d.b * d.T * d.H == 0;
    const bool nostate = d.b * d.H == 0;
    if (!req(x, empty) || !req(dt, empty) || !req(A, d.H == 0) || !req(B, empty) ||
        !req(C, empty) || !opt(D) || !opt(initial_state) || !req(dy, empty) ||
        !opt(dfinal_state) || !req(dx, empty) || !req(ddt, empty) || !req(dA, d.H == 0) ||
        !req(dB, empty) || !req(dC, empty) || !opt(dD) || !opt(dinitial_state))
        return MAMBA2_ERR_INVALID_ARG;
    if (D && !dD) return MAMBA2_ERR_INVALID_ARG;
    if (d.L > 256 || d.P > 128) return MAMBA2_ERR_UNSUPPORTED;
    const BwdCarve cv = bwd_carve(d, bwd_copies(shape, d), m2::bwd_dot_mode(d, bwd_tc(shape, d)),
                                  bwd_tc(shape, d), !bwd_bc(shape, d));
    if (!empty && (!workspace || workspace_bytes < cv.total ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return MAMBA2_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (d.H > 0) e = cudaMemsetAsync(dA, 0, sizeof(float) * (size_t)d.H, s);
    if (e == cudaSuccess && dD && d.H > 0) e = cudaMemsetAsync(dD, 0, sizeof(float) * (size_t)d.H, s);
    if (e != cudaSuccess || nostate) return from_cuda(e);
    const size_t sbytes = sizeof(float) * (size_t)(d.b * d.H * d.P * d.N);
    if (d.T == 0) {   // dinitial_state = dfinal_state (or 0)
        if (!dinitial_state) return MAMBA2_OK;
        return from_cuda(dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, sbytes,
                                                        cudaMemcpyDeviceToDevice, s)
                                      : cudaMemsetAsync(dinitial_state, 0, sbytes, s));
    }
    char* ws = static_cast<char*>(workspace);
    float* cum2 = reinterpret_cast<float*>(ws + cv.cum2);
    float* dtT = reinterpret_cast<float*>(ws + cv.dtT);
    float* dS = reinterpret_cast<float*>(ws + cv.dS);
    void* Sprev = ws + cv.Sprev;
    float* fin = reinterpret_cast<float*>(ws + cv.fin);
    int32_t* err = error_word();
    // Forward stages 1-3: cum2, dtT, dS (fp32), the state entering each chunk (in
    // the I/O type, stage 4's operand) and the final state.  P = 128 runs the
    // whole backward on the CUDA cores: with the tensor-core kernels (16-bit
    // operands, each head as two heads of 64) dA, a signed sum over every token,
    // missed the fp32 reading by 1.4e-2 relative L2 on a two-head case.
    const bool tc = bwd_tc(shape, d);
    e = m2::launch_chunk_cumsum(d, dt, A, cum2, dtT, err, s);
    if (e == cudaSuccess)
        e = tc ? m2::launch_chunk_state_tc(d, x, B, cum2, dtT, dS, true, err, s,   // bf16 dS
                                           reinterpret_cast<uint32_t*>(ws + cv.xabs_x))
               : m2::launch_chunk_state_simt(d, x, B, cum2, dtT, dS, err, s);
    if (e == cudaSuccess)
        e = m2::launch_state_pass(d, dS, tc, cum2, initial_state, Sprev, fin, err, s);
    auto at = [&](size_t off) { return static_cast<void*>(ws + off); };
    auto atf = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    m2::BwdWork w{dS,           at(cv.GnIO),     at(cv.yno),      at(cv.yr),    at(cv.dyr),
                  at(cv.Br),    at(cv.Cr),       atf(cv.cum2r),   atf(cv.ones), at(cv.xB),
                  at(cv.xCr),   at(cv.xr),       at(cv.SprevT),   at(cv.GnT),   atf(cv.cum2d),
                  atf(cv.dtTd), atf(cv.cum2rd),  atf(cv.onesd),   at(cv.yC),    at(cv.zB),
                  atf(cv.ydot2),  atf(cv.xyd2),    atf(cv.dyxd2),
                  tc ? reinterpret_cast<uint32_t*>(ws + cv.xabs_x) : nullptr,
                  tc ? reinterpret_cast<uint32_t*>(ws + cv.xabs_dy) : nullptr};
    if (e == cudaSuccess)
        e = m2::launch_backward(d, tc, x, B, C, dy, A, D, cum2, dtT, Sprev, fin, w, dfinal_state,
                                dx, ddt, dA, dB, dC, dD, dinitial_state, err, s);
    return from_cuda(e);
}

mamba2_status mamba2_ssd_device_error(int32_t* code, int32_t clear) {
    if (!code) return MAMBA2_ERR_INVALID_ARG;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return MAMBA2_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return MAMBA2_ERR_CUDA;
    if (clear && v) {
        const int32_t zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
            return MAMBA2_ERR_CUDA;
    }
    *code = v;
    return v ? MAMBA2_ERR_DEVICE : MAMBA2_OK;
}

mamba2_status mamba2_ssd_decode(const mamba2_ssd_shape* shape, float* state, const void* x,
                                const float* dt, const float* A, const void* B, const void* C,
                                const float* D, void* y, void* stream) {
    if (!shape) return MAMBA2_ERR_INVALID_ARG;
    if (shape->seqlen != 1 || shape->flags != 0) return MAMBA2_ERR_INVALID_ARG;
    mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    const Dims d = dims_of(shape);
    const bool empty = d.b * d.H == 0;
    if (!req(state, empty) || !req(x, empty) || !req(dt, empty) || !req(A, empty) ||
        !req(B, empty) || !req(C, empty) || !opt(D) || !req(y, empty))
        return MAMBA2_ERR_INVALID_ARG;
    return from_cuda(m2::launch_decode(d, state, x, dt, A, B, C, D, y, error_word(),
                                       static_cast<cudaStream_t>(stream)));
}

mamba2_status mamba2_ssd_selftest_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 100000) return MAMBA2_ERR_INVALID_ARG;
    return from_cuda(m2::launch_wait_timeout_selftest((uint64_t)limit_us * 1000, error_word(),
                                                      static_cast<cudaStream_t>(stream)));
}

mamba2_status mamba2_ssd_tile_choice(const mamba2_ssd_shape* shape, int32_t* out) {
    const mamba2_status st = check(shape);
    if (st != MAMBA2_OK) return st;
    if (!out) return MAMBA2_ERR_INVALID_ARG;
    const Dims d0 = whole_dims(shape);
    if (!use_tc(shape, d0)) return MAMBA2_ERR_UNSUPPORTED;
    const Dims d = m2::tc_view(d0);   // the launchers choose on this view
    int src2 = 0;
    out[0] = m2::k2_units_per_cta(d, &src2);
    out[1] = src2;
    const m2::Split4 sp = m2::k4_split(d);
    out[2] = sp.v1;
    out[3] = sp.v2;
    out[4] = (int32_t)sp.n1_bc;
    out[5] = sp.src;
    return MAMBA2_OK;
}

const char* mamba2_status_string(mamba2_status status) {
    switch (status) {
        case MAMBA2_OK: return "ok";
        case MAMBA2_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer or bad dimension)";
        case MAMBA2_ERR_UNSUPPORTED: return "unsupported shape (see mamba2_ssd_shape)";
        case MAMBA2_ERR_CUDA: return "CUDA runtime error or launch failure";
        case MAMBA2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MAMBA2_ERR_DEVICE: return "a kernel recorded a device-side error";
    }
    return "unknown status";
}

const char* mamba2_ssd_version(void) { return "0.1.0"; }

}  // extern "C"
