/*
 * msc.h -- C ABI of libmsc, the B300 (sm_103a) Mamba selective scan.
 *
 * Three operations, as the pages state the problem.  Pages are cited by title:
 * "Mamba — 选择性状态空间模型" (study note), bqwf survey (the Mamba survey
 * article on bqwf.cn, whose title did not survive extraction),
 * "Mamba前世今生全挖掘", "Review: Mamba — Linear-Time Sequence Modeling with
 * Selective State Spaces", and "Mamba 解密".
 *
 *  - S6 forward.  Selection Delta_t = softplus(delta_t + Delta_bias) (bqwf survey sec. 2.2;
 *    "Mamba 解密" sec. 5), exponential-Euler recurrence
 *    h_t = exp(Delta_t A) (.) h_{t-1} + Delta_t B_t u_t ("Mamba 解密" sec. 6.3:
 *    Mamba-1/2 are exponential-Euler), readout y_t = C_t . h_t + D u_t ("Mamba 解密"
 *    sec. 3, D feed-through), gated by silu(z_t) ("Mamba前世今生全挖掘" sec. 二,
 *    selective SSM + gating).
 *  - S6 backward by recomputation (bqwf survey sec. 2.2): a forward pass keeps
 *    the fp32 state entering every 8-step group of every row in the workspace
 *    (1/8 of h), and the reverse pass recomputes the steps in between in
 *    registers; no other state is stored.
 *  - Mamba-2 SSD chunked forward: scalar A per head (A_t = alpha_t I), the
 *    semiseparable form Y = M (X . B^T) C with M_ij = a_{j+1}...a_i (bqwf
 *    survey sec. 3.2; "Mamba 解密" sec. 6.2), computed by the block
 *    decomposition on tcgen05 tensor cores.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned.  The library allocates no device memory: any
 *    scratch comes from the caller's `workspace`, whose size is given by the
 *    matching *_workspace_size() query (0 means NULL may be passed).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; the host returns after enqueueing.
 *  - Outputs are fully overwritten, including gradients that are sums.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns MSC_ERR_INVALID_ARG / MSC_ERR_UNSUPPORTED with a message in
 *    msc_last_error() and launches nothing.  Launch failures return MSC_ERR_CUDA.
 *  - bf16 applies to the streamed inputs (u, delta, z, B, C, dy, x).  A, D and
 *    Delta_bias are always fp32; outputs and gradients are always fp32.
 *  - NaN and Inf propagate unchecked.  No C++ exception crosses this boundary.
 */
#ifndef MSC_H_
#define MSC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MSC_OK = 0,
    MSC_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, misalignment */
    MSC_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels cover */
    MSC_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    MSC_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out (see msc_check_device_status) */
    MSC_ERR_WORKSPACE = 5      /* workspace NULL or smaller than the query returned */
} msc_status;

typedef enum { MSC_F32 = 0, MSC_BF16 = 1 } msc_dtype;

/* ------------------------------------------------------------------ S6 forward
 * Shapes: u, delta, z: [batch, dim, seqlen]; B, C: [batch, dstate, seqlen]
 * (shared by all channels of a batch entry); A: [dim, dstate] fp32;
 * D, delta_bias: [dim] fp32; h0, h_last: [batch, dim, dstate] fp32;
 * y: [batch, dim, seqlen] fp32.
 * Optional (may be NULL): D (no feed-through), z (no gate), delta_bias (0),
 * h0 (zero initial state), h_last (final state not returned).
 * Limits: batch, dim, seqlen >= 1; 1 <= dstate <= MSC_S6_FWD_MAX_DSTATE (64).
 * Above 16 states the fused conv front end and the training pair are not
 * offered (MSC_S6_MAX_DSTATE, 16); the backward and the decode step take 64
 * like the forward, the SSD entry points
 * dstate 128.  Each row holds its states in 16, 32 or 64 slots (the next of
 * these at or above dstate); the slots past dstate carry zeros.  Above 16
 * states, rows that TMA cannot stream as they are (seqlen not a multiple of 8
 * with bf16 inputs, of 4 with fp32) are copied to a padded pitch inside the
 * workspace, which the size query then includes and which is REQUIRED: the
 * padded steps take delta = -inf, so that Delta = 0 there and the state passes
 * them unchanged.  The trapezoidal form cannot take padded steps and returns
 * MSC_ERR_UNSUPPORTED for such rows.
 * Workspace (256-byte aligned, size from msc_selective_scan_fwd_workspace_size):
 *  - long sequences with few rows are split into segments whose carries are
 *    combined in the workspace (three launches); there it is REQUIRED and a
 *    smaller one returns MSC_ERR_WORKSPACE;
 *  - otherwise one pass; for sequences of 512 steps or more the workspace lets
 *    persistent CTAs hand each 32-row block's state from one time chunk to the
 *    next (a ticket counter, per-block flags and the states, cleared by the
 *    call itself), which balances the load across SMs.  There it is OPTIONAL:
 *    with NULL or a smaller one the pass runs one CTA per row block.
 *  - a workspace must not be shared by calls that overlap on the GPU.
 * Rows whose byte stride (seqlen * element size) is a multiple of 16 are
 * streamed with TMA; other lengths take a plain-load kernel with identical
 * arithmetic for dstate <= 16, and the padded copies above. */
#define MSC_S6_FWD_MAX_DSTATE 64
#define MSC_S6_MAX_DSTATE 16

size_t msc_selective_scan_fwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen,
                                             int64_t dstate);

msc_status msc_selective_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                  msc_dtype in_dtype,
                                  const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D,
                                  const void* z, const float* delta_bias, const float* h0,
                                  float* y, float* h_last,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------- S6 forward, other discretisations
 * The same forward with the input term of h_t = abar_t h_{t-1} + b_t chosen by
 * `disc` (abar_t = exp(Delta_t A) in every form):
 *  - MSC_DISC_EULER: b_t = Delta_t B_t u_t, exactly msc_selective_scan_fwd
 *    ("Mamba 解密" sec. 6.3: Mamba-1/2 are exponential-Euler);
 *  - MSC_DISC_ZOH: zero-order hold, b_t = (Delta_t A)^-1 (exp(Delta_t A) - 1)
 *    Delta_t B_t u_t ("Mamba 解密" sec. 3 and sec. 5);
 *  - MSC_DISC_TRAPEZOID: exponential-trapezoidal (Mamba-3, "Mamba 解密" sec. 6.3),
 *    b_t = 1/2 (Delta_t B_t u_t + abar_t Delta_{t-1} B_{t-1} u_{t-1}), with no
 *    input term before t = 0 (h0, if given, is the state only).
 * Arguments, workspace (msc_selective_scan_fwd_workspace_size) and errors as
 * msc_selective_scan_fwd, including rows of any length (up to 16 states the
 * plain-load kernel takes every form; above, the padded copies take the
 * zero-order hold but not the trapezoid, which returns MSC_ERR_UNSUPPORTED for
 * rows TMA cannot stream).  No backward is provided for these forms.
 */
typedef enum { MSC_DISC_EULER = 0, MSC_DISC_ZOH = 1, MSC_DISC_TRAPEZOID = 2 } msc_discretization;

msc_status msc_selective_scan_fwd_ex(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                     msc_dtype in_dtype, msc_discretization disc,
                                     const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D,
                                     const void* z, const float* delta_bias, const float* h0,
                                     float* y, float* h_last,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* -------------------------------------------- S6 forward without allocation
 * No counterpart on the pages: an interface for callers that cannot allocate
 * device memory -- a plugin inside a host framework that owns every device
 * allocation and exposes no allocator to it, or a latency-critical serving loop
 * that must not call cudaMalloc on its hot path (cudaMalloc can synchronise the
 * device).  Same arguments, results and errors as msc_selective_scan_fwd()
 * without the workspace: the segment scratch of long sequences comes from a
 * library-owned array of MSC_STATIC_SCRATCH_BYTES in device global memory,
 * present on every device that loads the library until the process exits.
 * - A problem whose REQUIRED workspace (the segment scratch of long sequences
 *   with few rows, see msc_selective_scan_fwd) exceeds MSC_STATIC_SCRATCH_BYTES
 *   returns MSC_ERR_WORKSPACE and launches nothing; the optional load-balancing
 *   scratch is used when it fits in the array and left out when it does not.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and caches it; make that
 *   first call before any stream capture.  The cache is kept per device
 *   ordinal for the life of the process: after cudaDeviceReset the module is
 *   loaded again and the array may move, so a process that resets a device
 *   must not call this entry point on it afterwards.
 * - All calls share the one array and its contents persist between calls:
 *   calls that overlap on the GPU (other streams, other host threads) race.
 * - Allocates nothing itself (no cudaMalloc / cudaFree). */
#define MSC_STATIC_SCRATCH_BYTES (4u << 20)

msc_status msc_selective_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                          msc_dtype in_dtype,
                                          const void* u, const void* delta, const float* A,
                                          const void* B, const void* C, const float* D,
                                          const void* z, const float* delta_bias, const float* h0,
                                          float* y, float* h_last, void* stream);

/* ------------------------------------------- S6 forward from host memory
 * The forward of msc_selective_scan_fwd for inputs and outputs that live in
 * HOST memory: u, delta, z (optional), B, C and y are host pointers (pinned
 * memory lets the copies overlap the scan; pageable memory works but
 * serialises); A, D, delta_bias are device pointers as in
 * msc_selective_scan_fwd (zero initial state, no final state).  The batch runs
 * in chunks of chunk_batch entries through a three-stream pipeline: the upload
 * of chunk i + 1, the scan of chunk i on `stream` and the download of chunk
 * i - 1 proceed together.  staging: caller-owned device memory, 256-byte
 * aligned, of msc_selective_scan_fwd_host_staging_size(...) bytes (two chunk
 * slots and the forward's workspace); the library allocates nothing (it keeps
 * two CUDA streams per device for the copies).  The call returns once the work
 * is queued; `stream` waits for the last download, so synchronising it makes
 * y complete.  Rows are independent, so y equals msc_selective_scan_fwd over
 * the whole batch whenever both take the same segment plan. */
size_t msc_selective_scan_fwd_host_staging_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                                msc_dtype in_dtype, int has_z, int64_t chunk_batch);

msc_status msc_selective_scan_fwd_host(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                       const void* B, const void* C, const float* D, const void* z,
                                       const float* delta_bias, float* y, int64_t chunk_batch, void* staging,
                                       size_t staging_bytes, void* stream);

/* ------------------------------- S6 forward with the conv1d front end fused
 * The Mamba block's causal depthwise conv1d + SiLU (bqwf survey sec. 3.1: the
 * convolution gives local context before the selective SSM), formed inside the
 * scan so that its output u never goes through memory:
 *   u[b, d, t] = silu(conv_bias[d] + sum_{k < width} conv_weight[d, k] x[b, d, t - (width - 1) + k])
 * (x = 0 before t = 0), then exactly msc_selective_scan_fwd on u.  x: [batch,
 * dim, seqlen] in in_dtype; conv_weight [dim, width] fp32 (width 1..4);
 * conv_bias [dim] fp32 or NULL; the other arguments, the workspace
 * (msc_selective_scan_fwd_workspace_size) and the errors as
 * msc_selective_scan_fwd.  u is kept in fp32 (not rounded to in_dtype), so
 * the result equals msc_causal_conv1d_fwd (fp32 out) followed by
 * msc_selective_scan_fwd with fp32 u up to rounding.  Any seqlen >= 1: rows
 * TMA can stream (seqlen a multiple of 8 with bf16 inputs, of 4 with fp32,
 * seqlen and dim below 2^31) take the TMA kernel, the rest the plain-load
 * kernel, which reads the three inputs before each segment from memory.
 * Exponential-Euler form and 1 <= dstate <= 16 only (else
 * MSC_ERR_UNSUPPORTED); no backward. */
msc_status msc_selective_scan_fwd_conv(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       int64_t conv_width, msc_dtype in_dtype, const void* x,
                                       const float* conv_weight, const float* conv_bias, const void* delta,
                                       const float* A, const void* B, const void* C, const float* D,
                                       const void* z, const float* delta_bias, const float* h0, float* y,
                                       float* h_last, void* workspace, size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------- S6 backward
 * Same shapes and dtype as the forward (zero initial state), plus the upstream
 * gradient dy [batch, dim, seqlen] (in_dtype).  Outputs (fp32, overwritten):
 * du, ddelta: [batch, dim, seqlen]; dA: [dim, dstate]; dB, dC: [batch, dstate, seqlen];
 * dD [dim] (required iff D != NULL); dz [batch, dim, seqlen] (required iff z != NULL);
 * ddelta_bias [dim] (required iff delta_bias != NULL).  dstate <= 64
 * (MSC_S6_FWD_MAX_DSTATE, as the forward), else MSC_ERR_UNSUPPORTED.  Above 16
 * states the backward runs once per slice of 16 (every gradient is a sum of
 * per-state terms or is per state): the slices' du, ddelta and dz add up in
 * the outputs, and the workspace also holds one slice of A and of dA.
 * The forward states are recomputed from checkpoints kept every 8 steps in the
 * workspace (16 fp32 per row and group: 8 bytes per element); dB, dC, dA, dD and
 * ddelta_bias are sums accumulated with fp32 atomics, so their low bits depend
 * on the order in which blocks finish.  seqlen (rounded up to a 16-byte row)
 * and dim must be below 2^31, else MSC_ERR_UNSUPPORTED. */
size_t msc_selective_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen,
                                             int64_t dstate);

msc_status msc_selective_scan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                  msc_dtype in_dtype,
                                  const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D,
                                  const void* z, const float* delta_bias, const void* dy,
                                  float* du, float* ddelta, float* dA, float* dB, float* dC,
                                  float* dD, float* dz, float* ddelta_bias,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* -------------------------------------------------------- S6 training pair
 * For training, the forward can keep what the backward otherwise recomputes
 * first: the state entering every 8-step group of every row, the checkpoints
 * the backward runs its adjoint from (1/8 of the states, fp32; bqwf survey
 * sec. 2.2: the backward recomputes the states rather than storing them all).
 *  - msc_selective_scan_fwd_train is msc_selective_scan_fwd (zero initial
 *    state, no final state, same workspace rules) that also writes ckpt
 *    [batch * dim, seqlen / 8, 16] fp32, msc_selective_scan_ckpt_size() bytes:
 *    state n entering group g of row r at ckpt[(r * (seqlen / 8) + g) * 16 + n],
 *    zero for n >= dstate.  y equals msc_selective_scan_fwd's bit for bit.
 *  - msc_selective_scan_bwd_ckpt is msc_selective_scan_bwd run from those
 *    checkpoints: it skips its own checkpoint pass and takes no workspace.
 *    When the forward runs as one pass or in chained chunks (sequences under
 *    512 steps, or enough rows to fill the GPU) the checkpoints equal the ones
 *    msc_selective_scan_bwd computes bit for bit, and the gradients agree up
 *    to the order of the atomic sums; with segments (few rows, long
 *    sequences) each segment starts from a carry that combines the states in
 *    another order, so checkpoints and gradients differ by rounding.
 * Limits: dstate 1..16 (MSC_S6_MAX_DSTATE: a checkpoint holds 16 states), seqlen
 * a multiple of 8 and seqlen, dim below 2^31, else MSC_ERR_UNSUPPORTED; the checkpoints must come from
 * msc_selective_scan_fwd_train on the same inputs. */
size_t msc_selective_scan_ckpt_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate);

msc_status msc_selective_scan_fwd_train(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                        msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                        const void* B, const void* C, const float* D, const void* z,
                                        const float* delta_bias, float* y, float* ckpt, void* workspace,
                                        size_t workspace_bytes, void* stream);

msc_status msc_selective_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                       const void* B, const void* C, const float* D, const void* z,
                                       const float* delta_bias, const void* dy, const float* ckpt, float* du,
                                       float* ddelta, float* dA, float* dB, float* dC, float* dD, float* dz,
                                       float* ddelta_bias, void* stream);

/* ------------------------------------------------------------ S6 decode step
 * One token of the same recurrence for every channel row, the state carried
 * from call to call ("Mamba — 选择性状态空间模型", 实践案例 1: what happens when
 * one token is read -- the fixed-size state h is updated once and read out;
 * 核心要点: training runs the parallel scan, inference runs this step-by-step
 * recurrence).  Per row (b, d), with Delta = softplus(delta + Delta_bias[d]):
 *   state[n] <- exp(Delta A[d, n]) state[n] + Delta B[b, n] u
 *   y = (sum_n C[b, n] state[n] + D[d] u) * silu(z)
 * Shapes: u, delta, z, y: [batch, dim]; B, C: [batch, dstate]; A: [dim, dstate];
 * D, delta_bias: [dim]; state: [batch, dim, dstate] fp32, read and overwritten
 * in place.  dstate 1..64 (MSC_S6_FWD_MAX_DSTATE, as the forward); no
 * workspace.  Calling it seqlen times on tokens t = 0.. reproduces
 * msc_selective_scan_fwd with h0 = the initial state, up to fp32 rounding.
 * Each thread moves 8 states of a row with one 32-byte load and store (two,
 * four or eight threads per row up to 16, 32 or 64 states).
 */
msc_status msc_selective_state_update(int64_t batch, int64_t dim, int64_t dstate, msc_dtype in_dtype,
                                      const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, const float* D,
                                      const void* z, const float* delta_bias,
                                      float* state, float* y, void* stream);

/* ------------------------------------------------ causal conv1d front end
 * The short causal convolution that gives the selective SSM its local context
 * in every Mamba block (bqwf survey sec. 3.1: causal 1-D convolution, then the
 * selective SSM), depthwise per channel, followed by SiLU:
 *   out[b, d, t] = silu(bias[d] + sum_{k < width} w[d, k] x[b, d, t - (width - 1) + k])
 * with x = 0 before t = 0 (width 1..8; 4 in Mamba).  Shapes: x, out
 * [batch, dim, seqlen]; weight [dim, width] fp32; bias [dim] fp32 or NULL.
 * `silu` = 0 skips the activation.  x is fp32 or bf16 (in_dtype); out is
 * fp32 or bf16 (out_dtype; bf16 rounds to nearest even), so the result can be
 * passed to msc_selective_scan_fwd as u.  No workspace.
 */
msc_status msc_causal_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                                 msc_dtype in_dtype, msc_dtype out_dtype, const void* x,
                                 const float* weight, const float* bias, int silu, void* out,
                                 void* stream);

/* Backward of msc_causal_conv1d_fwd for an upstream gradient dout (the chain
 * rule through its definition): with pre the pre-activation and g = dout *
 * silu'(pre) (g = dout when silu = 0),
 *   dx[b, d, s]   = sum_k weight[d, k] g[b, d, s + (width - 1) - k]
 *   dweight[d, k] = sum_{b, t} g[b, d, t] x[b, d, t - (width - 1) + k]
 *   dbias[d]      = sum_{b, t} g[b, d, t]
 * x, weight, bias, silu as the forward (x in in_dtype); dout, dx [batch, dim,
 * seqlen] fp32 (dout is what msc_selective_scan_bwd returns as du); dweight
 * [dim, width] and dbias [dim] fp32 (dbias may be NULL), overwritten.  The sums
 * over batch and steps use fp32 atomics.  No workspace. */
msc_status msc_causal_conv1d_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width, msc_dtype in_dtype,
                                 const void* x, const float* weight, const float* bias, int silu,
                                 const float* dout, float* dx, float* dweight, float* dbias, void* stream);

/* Decode step of the same convolution (study note "Mamba — 选择性状态空间模型",
 * 踩过的坑: with no attention cache, the convolution still keeps the last
 * few inputs).  conv_state [batch, dim, width - 1] fp32 holds the previous
 * width - 1 inputs, oldest first; it is read, shifted by one and written back
 * with x appended.  x, out: [batch, dim].  Calling it seqlen times reproduces
 * msc_causal_conv1d_fwd from a zero state.
 */
msc_status msc_causal_conv1d_update(int64_t batch, int64_t dim, int64_t width, msc_dtype in_dtype,
                                    msc_dtype out_dtype, const void* x, const float* weight,
                                    const float* bias, int silu, float* conv_state, void* out,
                                    void* stream);

/* ------------------------------------------------------------- SSD chunked fwd
 * Shapes: x, z: [batch, seqlen, nheads, headdim]; delta: [batch, seqlen, nheads];
 * A, D, delta_bias: [nheads] fp32; B, C: [batch, seqlen, ngroups, dstate];
 * y: [batch, seqlen, nheads, headdim] fp32; final_state: [batch, nheads, headdim, dstate] fp32.
 * Optional (may be NULL): D, z, delta_bias, final_state.
 * Limits: in_dtype == MSC_BF16; headdim == 64; dstate == 128; ngroups divides
 * nheads; chunk in {64, 128, 256}; seqlen >= 1 (ragged last chunk allowed).
 * The result does not depend on `chunk` beyond rounding: it only sets where
 * the chunk states are materialised.  A device-side bounded wait that runs out
 * is reported by msc_check_device_status().
 * Workspace: REQUIRED, of msc_ssd_chunked_fwd_workspace_size() bytes and
 * 1024-byte aligned (it holds the chunk states as tensor-core operand tiles
 * with a 128-byte swizzle, whose atoms are 1024 bytes): a smaller one returns
 * MSC_ERR_WORKSPACE, a misaligned one MSC_ERR_INVALID_ARG. */
size_t msc_ssd_chunked_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads,
                                          int64_t headdim, int64_t dstate, int64_t ngroups,
                                          int64_t chunk);

msc_status msc_ssd_chunked_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t dstate, int64_t ngroups, int64_t chunk,
                               msc_dtype in_dtype,
                               const void* x, const void* delta, const float* A,
                               const void* B, const void* C, const float* D, const void* z,
                               const float* delta_bias, float* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------- SSD chunked bwd
 * Gradients of msc_ssd_chunked_fwd (zero initial state; final_state is not an
 * output here), derived from the same chunk decomposition (bqwf survey sec. 3.2:
 * scalar A_t = alpha_t I; "Mamba 解密" sec. 6.2: the SSD as the masked matrix
 * Y = M (X . B^T) C).  Inputs as the forward, plus dy [batch, seqlen, nheads,
 * headdim] bf16.  Outputs (fp32, overwritten): dx [batch, seqlen, nheads,
 * headdim]; ddelta [batch, seqlen, nheads]; dA [nheads]; dB, dC [batch, seqlen,
 * ngroups, dstate]; dD [nheads] (required iff D != NULL); dz like dx (required
 * iff z != NULL); ddelta_bias [nheads] (required iff delta_bias != NULL).
 * Limits as the forward, and nheads / ngroups a multiple of 16 when ngroups > 1.
 * With z the pre-gate output is recomputed by the forward into the workspace
 * (has_z selects the larger workspace).  dB, dC, dA, dD, ddelta_bias and the
 * cumulative-sum gradients are fp32 atomic sums: their low bits depend on the
 * order in which blocks finish.  Workspace: required, of
 * msc_ssd_chunked_bwd_workspace_size() bytes, 1024-byte aligned (as the
 * forward's). */
size_t msc_ssd_chunked_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads,
                                          int64_t headdim, int64_t dstate, int64_t ngroups,
                                          int64_t chunk, int has_z);

msc_status msc_ssd_chunked_bwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t dstate, int64_t ngroups, int64_t chunk,
                               msc_dtype in_dtype,
                               const void* x, const void* delta, const float* A,
                               const void* B, const void* C, const float* D, const void* z,
                               const float* delta_bias, const void* dy, float* dx, float* ddelta,
                               float* dA, float* dB, float* dC, float* dD, float* dz,
                               float* ddelta_bias, void* workspace, size_t workspace_bytes,
                               void* stream);

/* ------------------------------------------------------------------- utilities
 * msc_check_device_status: synchronises `stream`, then reads and clears the
 * device status words that the library's kernels keep on the current device
 * (one per kernel module, in device global memory).  A kernel whose bounded
 * wait on an mbarrier ran out (about one second) records MSC_ERR_TIMEOUT and
 * the site there, and returns instead of hanging.  Returns MSC_OK,
 * MSC_ERR_TIMEOUT, or MSC_ERR_CUDA if the stream itself reports an error. */
msc_status msc_check_device_status(void* stream);

/* Static English name of a status code. */
const char* msc_status_string(msc_status status);

/* Message of the last failing call on this host thread ("" if none).  The
 * pointer stays valid until the next library call on the same thread. */
const char* msc_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int msc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSC_H_ */
