/*
 * mamba2_ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked forward pass.
 *
 * Pages cited (by title and section):
 *   [P1] "NVIDIA、cuTileでMamba-2フォワードパスを高速化" (ai.newsbites.today),
 *        "cuTileによるMamba-2フォワードパスの3段階カーネル設計" and the
 *        optimisation table.
 *   [P2] "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
 *        "Mamba-2 아키텍처의 핵심 연산", "세 가지 핵심 커널 구현",
 *        "cuTile 기반 성능 최적화 기법".
 *   [P3] "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 *        NVIDIA CUDA Tile" (brifing.si), sections 4, 5, 7, 8, 9, 11.
 *
 * The operation.  Per batch b and head h, with state S in R^{P x N} and
 * a_t = dt[b,t,h] * A[h] (A[h] < 0):
 *     S_t = exp(a_t) S_{t-1} + dt[b,t,h] x[b,t,h,:] B[b,t,g,:]^T
 *     y[b,t,h,:] = S_t C[b,t,g,:] + D[h] x[b,t,h,:]
 * S_{-1} = initial_state[b,h] (or 0), final_state[b,h] = S_{T-1}; head h reads
 * group g = h / (H/G).  [P2 "핵심 연산"] prints the read-out
 * y_t = c_t^T h_t + D x_t; the update is the standard Mamba-2 discretisation
 * that the pages' log-space cumulative sum of a_t presumes.  It is evaluated
 * chunk by chunk (chunk length L) in four steps [P2 "세 가지 핵심 커널 구현",
 * P3 sections 4-9]: a log2-scaled chunk-local cumsum, per-chunk states by the
 * jump formula, a sequential pass over chunks, and a fused three-term output.
 *
 * Conventions for every entry point.
 *   - All tensors are dense, row-major, contiguous device memory, owned by the
 *     caller.  The library allocates nothing and keeps no per-call host state;
 *     it may be called concurrently from several host threads on different
 *     streams with disjoint buffers.  The one piece of state it shares between
 *     calls is the device error word (mamba2_ssd_device_error): one 32-bit
 *     word per device, into which every kernel of every call on that device
 *     ORs its error bits.  A bounded wait that runs out in one stream's call is
 *     therefore seen by every caller that reads the word, and reading it with
 *     `clear` set clears it for all of them; callers that run several streams
 *     at once should read and clear it from one place.
 *   - Every pointer must be 16-byte aligned (tensor-memory-accelerator copies).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronise.  Argument errors are detected on the host,
 *     before any launch, and nothing is launched when a call fails.
 *   - Outputs must not alias inputs or each other.
 *   - `dtype` selects the element type of x, B, C, y (and of the Sprev
 *     intermediate): MAMBA2_F32 (float) or MAMBA2_BF16 (__nv_bfloat16).
 *     dt, A, D, initial_state, final_state and the other intermediates are
 *     always float.
 *
 * Layouts (nc = ceil(T / L)):
 *   x, y           [b, T, H, P]     dtype
 *   dt             [b, T, H]        float, dt > 0 (taken as given: no softplus)
 *   A              [H]              float, A < 0
 *   B, C           [b, T, G, N]     dtype
 *   D              [H]              float, or NULL (= 0)
 *   initial_state  [b, H, P, N]     float, or NULL (= 0)
 *   final_state    [b, H, P, N]     float
 *   cum2, dtT      [b, H, T]        float (chunk-local cumsum * log2(e); dt transposed)
 *   dS             [b, nc, H, P, N] float (state each chunk builds from zero)
 *   Sprev          [b, nc, H, P, N] dtype (state entering each chunk)
 */
#ifndef MAMBA2_SSD_H
#define MAMBA2_SSD_H

#include <stddef.h>
#include <stdint.h>

#if defined(MAMBA2_SSD_BUILD) && defined(__GNUC__)
#define MAMBA2_API __attribute__((visibility("default")))
#else
#define MAMBA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mamba2_status {
    MAMBA2_OK = 0,
    MAMBA2_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad dimension       */
    MAMBA2_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shape set      */
    MAMBA2_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed           */
    MAMBA2_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required        */
    MAMBA2_ERR_DEVICE = 5         /* a kernel recorded a device-side error (timeout) */
} mamba2_status;

typedef enum mamba2_dtype { MAMBA2_F32 = 0, MAMBA2_BF16 = 1 } mamba2_dtype;

/* Force the CUDA-core (SIMT) chunk-state and chunk-output kernels even where
 * the tcgen05 tensor-core kernels apply (cross-checks and debugging). */
#define MAMBA2_FLAG_FORCE_SIMT 1
/* In mamba2_ssd_fwd on the tensor-core path, run stages 2 and 3 as the one
 * fused kernel of mamba2_ssd_chunk_state_pass instead of two kernels with dS in
 * HBM.  Same results bit for bit; slower on GB300 at the 2.7B layer shape
 * (0.321 ms against 0.244 ms for the pair), so it is not the default. */
#define MAMBA2_FLAG_FUSED_STATE 2
/* dS is bf16 (not fp32) in mamba2_ssd_chunk_state (output) and
 * mamba2_ssd_state_pass (input): the hand-off mamba2_ssd_fwd uses on the
 * tensor-core path (half the bytes; each chunk's dS rounded to bf16).  Needs
 * the tensor-core path for chunk_state and dtype BF16 for state_pass; other
 * shapes return MAMBA2_ERR_UNSUPPORTED. */
#define MAMBA2_FLAG_DS_BF16 4
/* In mamba2_ssd_fwd, launch the stages strictly one after another.  By default
 * stages 2, 3 and 4 of the tensor-core path use programmatic dependent launch:
 * each may start while the previous stage finishes and reads that stage's
 * outputs only after it has completed (stage 2 loads x and B early, stage 4
 * computes C.B^T and prepares x early).  Same results either way. */
#define MAMBA2_FLAG_SERIAL 8

/* Shape of one call.  Supported set:
 *   batch, seqlen, nheads >= 0 (a zero batch or head count is a no-op; seqlen 0
 *   writes final_state = initial_state, or 0);
 *   headdim P in {16, 32, 64, 128}; dstate N in {16, 32, 64, 128, 256};
 *   ngroups G >= 1 with nheads % G == 0; chunk_size L in {64, 128, 256};
 *   seqlen need not be a multiple of L (the last chunk is shorter).
 * The tensor-core path is used for dtype BF16 with L in {128, 256},
 * P in {32, 64, 128} and N in {64, 128, 256} (P = 128 runs as twice the heads
 * of 64: the tensors hold the same bytes in either view; P = 32 runs on
 * 64-column tiles that also hold the next head's columns, of which only the
 * head's own outputs are kept); every other supported shape runs on the
 * CUDA-core kernels (mamba2_ssd_path reports which).  mamba2_ssd_bwd keeps
 * P in {32, 128} on the CUDA-core kernels.
 * The whole-path calls (mamba2_ssd_fwd, _fwd_strided, _fwd_timed,
 * _fwd_noalloc) run chunk_size 64 as 128-token chunks on shapes the tensor
 * cores take at 128: y and final_state do not depend on the chunk length.
 * The stage entry points, whose intermediates are laid out per chunk, keep
 * L = 64 on the CUDA cores. */
typedef struct mamba2_ssd_shape {
    int64_t batch;
    int64_t seqlen;
    int64_t nheads;
    int64_t headdim;
    int64_t dstate;
    int64_t ngroups;
    int64_t chunk_size;
    int32_t dtype;   /* mamba2_dtype */
    int32_t flags;   /* MAMBA2_FLAG_* */
} mamba2_ssd_shape;

/* Paths reported by mamba2_ssd_path. */
#define MAMBA2_PATH_SIMT 0
#define MAMBA2_PATH_TCGEN05 1

/* Validate a shape without touching any pointer or the GPU. */
MAMBA2_API mamba2_status mamba2_ssd_check_shape(const mamba2_ssd_shape* shape);

/* Which kernels mamba2_ssd_fwd would launch for this shape (MAMBA2_PATH_*),
 * or -1 for an invalid / unsupported shape.  Host-only. */
MAMBA2_API int32_t mamba2_ssd_path(const mamba2_ssd_shape* shape);

/* Bytes of workspace mamba2_ssd_fwd needs: cum2, dtT, dS and Sprev, each
 * 256-byte aligned.  0 for an invalid shape.  Host-only. */
MAMBA2_API size_t mamba2_ssd_workspace_size(const mamba2_ssd_shape* shape);

/* The whole forward pass: the four stages below, in order, on `stream`
 * (stages 2 and 3 as one kernel with MAMBA2_FLAG_FUSED_STATE, tensor-core path,
 * three or more chunks; successive stages overlap their start and end unless
 * MAMBA2_FLAG_SERIAL is set).  Everything queued on `stream` before the call
 * has completed before the first stage reads anything.  On the tensor-core path dS goes from stage 2 to
 * stage 3 in bf16 (as with MAMBA2_FLAG_DS_BF16); the carried states themselves
 * are accumulated in fp32.
 *   workspace: device buffer of at least mamba2_ssd_workspace_size(shape)
 *   bytes, 256-byte aligned, owned by the caller, contents ignored on entry.
 * Returns MAMBA2_OK once the launches are queued. */
MAMBA2_API mamba2_status mamba2_ssd_fwd(const mamba2_ssd_shape* shape,
                             const void* x, const float* dt, const float* A,
                             const void* B, const void* C, const float* D,
                             const float* initial_state,
                             void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream);

/* mamba2_ssd_fwd that also records stage boundaries, for profiling (the stages
 * then run strictly one after another, as with MAMBA2_FLAG_SERIAL): events[k]
 * (a cudaEvent_t created by the caller, or NULL to skip) is recorded on `stream`
 * before stage 1 (k = 0), after stages 1, 2, 3 (k = 1, 2, 3; with
 * MAMBA2_FLAG_FUSED_STATE events[2] and events[3] mark the same point) and after
 * stage 4 (k = 4).  `events` may be NULL. */
MAMBA2_API mamba2_status mamba2_ssd_fwd_timed(const mamba2_ssd_shape* shape,
                             const void* x, const float* dt, const float* A,
                             const void* B, const void* C, const float* D,
                             const float* initial_state,
                             void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* const* events);

/* Element strides of the large input/output tensors for mamba2_ssd_fwd_strided:
 * for each tensor, {batch stride, token stride} in elements.  Within one token
 * the data stay contiguous: H*P elements (head-major) for x and y, G*N for B and
 * C, H for dt.  Contiguous tensors have x = y = {T*H*P, H*P}, B = C = {T*G*N,
 * G*N}, dt = {T*H, H}, with which the call equals mamba2_ssd_fwd.  The typical
 * use is x, B and C as column slices of one projection output [b, T, H*P +
 * 2*G*N] (token stride H*P + 2*G*N) and y written into a wider buffer.
 * Requirements (else MAMBA2_ERR_INVALID_ARG): token stride >= the token's
 * extent, batch stride >= T * token stride, both > 0 (batch stride ignored when
 * batch == 1); y must not overlap any input.  Strides whose byte size is not a
 * multiple of 16 take the CUDA-core kernels (the tensor-memory-accelerator
 * copies of the tensor-core kernels need 16-byte strides); results are the same
 * as for contiguous tensors either way. */
typedef struct mamba2_ssd_strides {
    int64_t x[2], dt[2], B[2], C[2], y[2];
} mamba2_ssd_strides;

/* mamba2_ssd_fwd on strided x, dt, B, C and y (see mamba2_ssd_strides);
 * initial_state and final_state stay contiguous [b, H, P, N]. */
MAMBA2_API mamba2_status mamba2_ssd_fwd_strided(const mamba2_ssd_shape* shape,
                             const mamba2_ssd_strides* strides,
                             const void* x, const float* dt, const float* A,
                             const void* B, const void* C, const float* D,
                             const float* initial_state,
                             void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Stage 1, chunk_cumsum [P3 section 7; P2 "세 가지 핵심 커널 구현"]:
 *   cum2[b,h,t] = log2(e) * sum_{r = chunk start of t}^{t} dt[b,r,h] * A[h]
 *   dtT[b,h,t]  = dt[b,t,h]
 * (inclusive, restarting at every chunk start; the [b,h,t] layout is the
 * transposed layout of the optimisation table of [P1] / [P2 "성능 최적화"]). */
MAMBA2_API mamba2_status mamba2_ssd_chunk_cumsum(const mamba2_ssd_shape* shape,
                                      const float* dt, const float* A,
                                      float* cum2, float* dtT, void* stream);

/* Stage 2, chunk states by the jump formula [P3 sections 4, 8]:
 *   dS[b,c,h,p,n] = sum_{s in chunk c} exp2(cum2_last(c) - cum2[s]) dtT[s] x[s,p] B[s,n]
 * (tcgen05 tensor cores where the shape allows).  dS is fp32 (float*), or bf16
 * with MAMBA2_FLAG_DS_BF16. */
MAMBA2_API mamba2_status mamba2_ssd_chunk_state(const mamba2_ssd_shape* shape,
                                     const void* x, const void* B,
                                     const float* cum2, const float* dtT,
                                     void* dS, void* stream);

/* Stage 3, sequential pass over chunks [P2 "세 가지 핵심 커널 구현", fwd_pass_state]:
 *   S = initial_state (or 0); for c: Sprev[c] = S; S = exp2(cum2_last(c)) S + dS[c];
 *   final_state = S.
 * Sprev is rounded to `dtype` (it is the tensor-core operand of stage 4); S is
 * fp32.  dS is fp32, or bf16 with MAMBA2_FLAG_DS_BF16. */
MAMBA2_API mamba2_status mamba2_ssd_state_pass(const mamba2_ssd_shape* shape,
                                    const void* dS, const float* cum2,
                                    const float* initial_state,
                                    void* Sprev, float* final_state, void* stream);

/* Stages 2 and 3 fused (tensor-core path only) [P3 section 8: fwd_pass_state
 * walks the chunks in order, combining the decayed carried state with each
 * chunk's own contribution]: Sprev and final_state exactly as
 * mamba2_ssd_chunk_state followed by mamba2_ssd_state_pass compute them (same
 * fp32 operations in the same order), without writing dS.  Each chunk's CTA
 * computes dS_c on the tensor cores and takes the state entering its chunk
 * from the CTA of the previous chunk.
 *   workspace: mamba2_ssd_chunk_state_pass_workspace_size(shape) bytes,
 *   256-byte aligned, owned by the caller: a two-slot fp32 ring of states per
 *   (b, h) and the synchronisation words, which the call clears on `stream`
 *   first.  Calls sharing one workspace must not overlap on the GPU.
 * Shapes without the tensor-core path (mamba2_ssd_path), and P = 32, return
 * MAMBA2_ERR_UNSUPPORTED (workspace size 0); they run mamba2_ssd_chunk_state +
 * _state_pass. */
MAMBA2_API size_t mamba2_ssd_chunk_state_pass_workspace_size(const mamba2_ssd_shape* shape);
MAMBA2_API mamba2_status mamba2_ssd_chunk_state_pass(const mamba2_ssd_shape* shape,
                                          const void* x, const void* B,
                                          const float* cum2, const float* dtT,
                                          const float* initial_state,
                                          void* Sprev, float* final_state,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream);

/* Stage 4, fused output [P3 sections 9, 11; P2 "세 가지 핵심 커널 구현", compute_out]:
 *   y[t,p] = sum_{s<=t in chunk} (C_t . B_s) exp2(cum2_t - cum2_s) dtT_s x[s,p]
 *          + exp2(cum2_t) (Sprev[c] C_t)[p] + D[h] x[t,p]
 * The causal mask is generated from indices and applied before exp2; the
 * L x L interaction matrix never leaves the chip. */
MAMBA2_API mamba2_status mamba2_ssd_chunk_out(const mamba2_ssd_shape* shape,
                                   const void* x, const void* B, const void* C,
                                   const float* cum2, const float* dtT,
                                   const void* Sprev, const float* D,
                                   void* y, void* stream);

/* Single-token decode step, the recurrent form of the same model
 * [P2 "Mamba-2 아키텍처의 핵심 연산": y_t = c_t^T h_t + D x_t], on the state layout of
 * mamba2_ssd_fwd's final_state, for each (b, h):
 *   state <- exp(dt A) state + dt x B^T   (in place, fp32)
 *   y      = state C + D x
 * shape: batch, nheads, headdim, dstate, ngroups, dtype as for mamba2_ssd_fwd;
 * seqlen must be 1; chunk_size is not used (any supported value); flags 0.
 *   state [b,H,P,N] fp32, read and written; x [b,H,P] (dtype); dt [b,H] fp32;
 *   A [H] fp32; B, C [b,G,N] (dtype); D [H] fp32 or NULL (= 0); y [b,H,P] (dtype).
 * Feeding the final_state of a prefix to this call token by token continues the
 * sequence (tested against mamba2_ssd_fwd over the whole sequence).
 * Pointers are device memory, 16-byte aligned, owned by the caller; state must
 * not overlap the other arrays.  Returns MAMBA2_OK once queued on `stream`,
 * MAMBA2_ERR_INVALID_ARG for a bad shape or pointer.  For dstate 128 and 256 the
 * kernel stages the state through shared memory behind a bounded wait; a wait
 * that runs out sets MAMBA2_DEVERR_TIMEOUT_DECODE in the device error word. */
MAMBA2_API mamba2_status mamba2_ssd_decode(const mamba2_ssd_shape* shape, float* state,
                                const void* x, const float* dt, const float* A,
                                const void* B, const void* C, const float* D,
                                void* y, void* stream);

/* Backward pass: gradients of a scalar loss given dL/dy and dL/dfinal_state.
 *
 * The pages give no backward method; they only note that end-to-end training
 * speed also depends on one [P1 "開発現場への影響と未確認事項"; P2 "성능 벤치마크 결과
 * 및 활용"].  This call computes the chain rule applied to the same chunked
 * forward [P3 sections 4, 5, 8, 9], which equals the gradient of the
 * token-by-token recurrence of mamba2_ssd_fwd (tested against an fp64 reverse
 * sweep of the recurrence).  It recomputes the forward's chunk states itself,
 * so it takes the forward's inputs, not its outputs.
 *
 * shape: as for mamba2_ssd_fwd; flags 0 or MAMBA2_FLAG_FORCE_SIMT (the forward
 *   recompute on CUDA cores); headdim <= 128.
 * Inputs (device, 16-byte aligned, caller-owned, read only): x, dt, A, B, C, D
 *   (or NULL = 0), initial_state (or NULL = 0) in the layouts and types of
 *   mamba2_ssd_fwd; dy [b,T,H,P] in x's type; dfinal_state [b,H,P,N] fp32 or
 *   NULL (= 0).
 * Outputs (device, 16-byte aligned, fp32 whatever the input type, fully written):
 *   dx [b,T,H,P], ddt [b,T,H], dA [H], dB and dC [b,T,G,N] (summed over the
 *   heads of each group), dD [H] (required when D is given, else may be NULL),
 *   dinitial_state [b,H,P,N] (NULL when not wanted).
 * workspace: mamba2_ssd_bwd_workspace_size(shape) bytes, 256-byte aligned.
 * Asynchronous on `stream`; argument errors are returned before any launch
 * (MAMBA2_ERR_INVALID_ARG, MAMBA2_ERR_UNSUPPORTED, MAMBA2_ERR_WORKSPACE);
 * MAMBA2_ERR_CUDA for a failed launch.  dA and dD are accumulated with atomic
 * adds across chunks, and on the tensor-core path dB and dC with fp32
 * reduce-adds across blocks of heads, so their last bits may vary from run to
 * run. */
MAMBA2_API size_t mamba2_ssd_bwd_workspace_size(const mamba2_ssd_shape* shape);
MAMBA2_API mamba2_status mamba2_ssd_bwd(const mamba2_ssd_shape* shape,
                                        const void* x, const float* dt, const float* A,
                                        const void* B, const void* C, const float* D,
                                        const float* initial_state, const void* dy,
                                        const float* dfinal_state,
                                        float* dx, float* ddt, float* dA, float* dB,
                                        float* dC, float* dD, float* dinitial_state,
                                        void* workspace, size_t workspace_bytes,
                                        void* stream);

/* Bits of the device-side error word. */
#define MAMBA2_DEVERR_TIMEOUT_CHUNK_STATE 1   /* a wait ran out in the stage-2 kernel */
#define MAMBA2_DEVERR_TIMEOUT_CHUNK_OUT 2     /* ... in the stage-4 kernel or the
                                                 backward's dB / dC kernel */
#define MAMBA2_DEVERR_LAUNCH_CONFIG 4         /* a kernel saw a launch it does not support */
#define MAMBA2_DEVERR_CHAIN 8                 /* the fused stage 2+3 kernel gave up waiting
                                                 for the previous chunk's state */
#define MAMBA2_DEVERR_SELFTEST 16             /* mamba2_ssd_selftest_wait_timeout ran out */
#define MAMBA2_DEVERR_TIMEOUT_DECODE 32       /* a wait ran out in the decode kernel */

/* Device-side error word.  The tensor-core kernels bound every wait; a wait
 * that runs out sets a bit here and the kernel returns early (its outputs are
 * then invalid).  This call synchronises the current device, reads the word
 * into *code (0 = no error) and clears it when `clear` is nonzero.  Returns
 * MAMBA2_ERR_DEVICE when the word was nonzero, MAMBA2_ERR_CUDA on a CUDA
 * failure, MAMBA2_OK otherwise. */
MAMBA2_API mamba2_status mamba2_ssd_device_error(int32_t* code, int32_t clear);

/* Diagnostic (no counterpart on the pages): launches one small kernel whose
 * bounded waits -- on an mbarrier nothing arrives at and on a global flag
 * nothing sets, the two kinds of wait the kernels use -- run out after
 * `limit_us` microseconds (1 .. 100000).  The kernel then sets
 * MAMBA2_DEVERR_SELFTEST in the device error word and returns normally; the
 * context stays usable.  Lets a caller check the failure path without a fault.
 * Returns MAMBA2_OK once queued, MAMBA2_ERR_INVALID_ARG for a limit out of range. */
MAMBA2_API mamba2_status mamba2_ssd_selftest_wait_timeout(uint32_t limit_us, void* stream);

/* Forward pass for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this is a convenience of this library.  Some
 * callers have no way to obtain device memory of their own -- code running
 * where cudaMalloc is forbidden or unavailable (for example inside a host
 * framework that owns every allocation, or a plug-in whose host may not call
 * the CUDA allocator), or code that must not allocate on its hot path.  For
 * them this entry point runs exactly mamba2_ssd_fwd, but with the workspace
 * taken from a fixed device array compiled into this library,
 * MAMBA2_NOALLOC_SCRATCH_BYTES (64 MiB) large; every GPU that loads the
 * library keeps that array until the process exits.  The caller still passes
 * every input and output buffer.
 *   - Shapes whose mamba2_ssd_workspace_size exceeds the array are rejected
 *     with MAMBA2_ERR_WORKSPACE before anything is launched.
 *   - The call allocates nothing: no cudaMalloc, cudaFree or allocating
 *     library routine.  The first call on each device looks up the array's
 *     device address (cudaGetSymbolAddress, with that device current); make
 *     that first call before any stream capture on the device.  The address
 *     is kept for the life of the process and belongs to the device's primary
 *     context (the one the CUDA runtime uses): do not call this entry point
 *     after cudaDeviceReset, or with another context current on the device.
 *   - Every call on a device shares the one array.  Nothing in it needs to
 *     start at zero (each stage writes what the next reads), but two calls
 *     that overlap on the GPU (different streams, no ordering between them)
 *     race on it and produce wrong results: order such calls. */
#define MAMBA2_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
MAMBA2_API mamba2_status mamba2_ssd_fwd_noalloc(const mamba2_ssd_shape* shape,
                             const void* x, const float* dt, const float* A,
                             const void* B, const void* C, const float* D,
                             const float* initial_state,
                             void* y, float* final_state, void* stream);

/* Per-shape launch choices of the tensor-core kernels.
 *
 * [P1] optimisation table and [P2] "cuTile 기반 성능 최적화 기법": the pages
 * pick block sizes and occupancy per input shape by searching them.  Here the
 * search runs offline (mamba_ssd_chunked_02_gb300/tune.py, which times every
 * candidate on the GPU through mamba2_ssd_tile_override) and its winners are
 * compiled into the library as a table keyed by (N, P, L, H/G, a range of
 * b * nc).  Two choices are tabled: the work per CTA of the chunk-state
 * kernel (stage 2: a CTA takes a contiguous range of units, a unit being one
 * head of one (b, chunk, 128-wide state tile), in the order b, chunk, state
 * tile, head; either blocks of heads of one group, or one wave of CTAs over
 * ceil(units / SMs)-unit ranges), and the head-block sizes of the output kernel (stage 4),
 * whose grid has two regions -- the first (b, c) pairs, filling `waves1` whole
 * waves of the SMs, take blocks of v1 heads, the rest blocks of v2.  A shape
 * with no table entry (or an entry that does not divide its H/G) takes the
 * launch-time cost models.  Neither choice changes any result bit: they only
 * regroup independent work.
 *
 * mamba2_ssd_tile_choice writes, for a shape on the tensor-core path,
 *   out[0] stage-2 units per CTA, out[1] its source,
 *   out[2] stage-4 v1, out[3] v2, out[4] (b, c) pairs in the v1 region,
 *   out[5] its source,
 * with source 0 = cost model, 1 = table, 2 = override.  `out` holds 6 words
 * owned by the caller.  Returns MAMBA2_ERR_INVALID_ARG for an invalid shape or
 * a NULL `out`, MAMBA2_ERR_UNSUPPORTED for a shape off the tensor-core path
 * (mamba2_ssd_path() == MAMBA2_PATH_SIMT), MAMBA2_OK otherwise.  Host only.
 *
 * mamba2_ssd_tile_override forces choices for every later launch in the
 * process (all threads, all devices) until it is called again with zeros:
 * stage2_units > 0 forces the units per CTA (capped at the shape's units), -2
 * one wave of even ranges; stage4_v1 > 0 forces stage 4's
 * split, v1 for the pairs of the first stage4_waves1 waves and stage4_v2 for
 * the rest (stage4_waves1 = 0: v1 for every pair, stage4_v2 ignored).  A
 * forced head-block size that does not divide a shape's H/G is ignored for
 * that shape.  stage2_units = -1 or stage4_v1 = -1 bypasses the table for that stage (the
 * cost model decides), so that the sweep can time the model's choice.  Meant
 * for the offline sweep, not for concurrent use with other callers.  Returns
 * MAMBA2_ERR_INVALID_ARG for stage2_units below -2, stage4_v1 below -1,
 * stage4_v2 or stage4_waves1 below 0, or v2 / waves1 set without a positive v1, MAMBA2_OK
 * otherwise. */
MAMBA2_API mamba2_status mamba2_ssd_tile_choice(const mamba2_ssd_shape* shape, int32_t* out);
MAMBA2_API mamba2_status mamba2_ssd_tile_override(int32_t stage2_units, int32_t stage4_v1,
                                                  int32_t stage4_v2, int32_t stage4_waves1);

/* Static description of a status code. */
MAMBA2_API const char* mamba2_status_string(mamba2_status status);

/* Library version, e.g. "0.1.0". */
MAMBA2_API const char* mamba2_ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA2_SSD_H */
