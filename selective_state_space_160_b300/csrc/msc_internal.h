// msc_internal.h -- launcher interfaces between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "msc.h"

namespace msc_host {

struct S6Plan {
    int G = 1;            // independent segments per row (1: no segment pass)
    int64_t seg_len = 0;  // timesteps per segment
    int chunks = 1;       // chained chunks per row block (1: one item per row block)
    int64_t chunk = 0;    // timesteps per chained chunk
    size_t workspace = 0; // bytes the plan uses
    bool workspace_required = false;  // segmented plans cannot run without it
    size_t seg_state_off = 0, seg_dsum_off = 0, ctrl_off = 0, ctrl_bytes = 0, chain_state_off = 0, bc_off = 0;
    // More than 16 states with rows that are not a multiple of 8 steps: the rows
    // are copied to a pitch of padded_len steps in the workspace (from pad_off)
    // and the fields above plan the padded problem.  0: no padding.
    int64_t padded_len = 0;
    size_t pad_off = 0;
};

// max_required: the largest required (segment) scratch the plan may use.
S6Plan s6_fwd_plan(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, size_t max_required = SIZE_MAX);

struct S6FwdArgs {
    int64_t batch, dim, L;
    int N;
    bool bf16;
    const void *u, *delta, *z, *B, *C;
    const float *A, *D, *delta_bias, *h0;
    float *y, *h_last;
    void* workspace;
    size_t workspace_bytes = 0;
    int disc = 0;  // msc_discretization
    // fused causal conv1d + SiLU front end: u holds its input x when conv_w is set
    const float* conv_w = nullptr;  // [dim, conv_k]
    const float* conv_b = nullptr;  // [dim] or null
    int conv_k = 0;
    // training forward: also the state entering every 8-step group, [rows, L / 8, 16]
    float* ckpt = nullptr;
    // checkpoint pass on a slice of the states: B and C point at the slice's
    // first state row, bc_rows state rows apart per batch entry (0: N)
    int bc_rows = 0;
};

msc_status s6_fwd_launch(const S6FwdArgs& a, const S6Plan& plan, cudaStream_t stream);

// The S6 forward entry point's validation, plan and launch; disc is an
// msc_discretization; max_required caps the plan's required scratch.
msc_status s6_fwd_entry(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, msc_dtype in_dtype, int disc,
                        const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, const float* h0, float* y,
                        float* h_last, void* workspace, size_t workspace_bytes, void* stream,
                        size_t max_required);

// Checkpoint pass used by the backward: writes the state entering every
// 8-step group of every row to ckpt [batch * dim, ceil(L / 8), 16] (fp32).
msc_status s6_fwd_checkpoints(const S6FwdArgs& a, float* ckpt, cudaStream_t stream);

// Each translation unit with bounded device-side waits keeps its own status
// word (code, site); these read and clear it.
msc_status s6_fwd_take_status(unsigned int* code, unsigned int* site);
msc_status s6_bwd_take_status(unsigned int* code, unsigned int* site);
msc_status ssd_take_status(unsigned int* code, unsigned int* site);
msc_status ssd_bwd_take_status(unsigned int* code, unsigned int* site);

size_t s6_bwd_workspace(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate);

struct S6BwdArgs {
    int64_t batch, dim, L;
    int N;
    bool bf16;
    const void *u, *delta, *z, *B, *C, *dy;
    const float *A, *D, *delta_bias;
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *ddelta_bias;
    void* workspace;
    // checkpoints from the training forward ([rows, L / 8, 16], L a multiple of
    // 8); when set the backward skips its own checkpoint pass and needs no workspace
    const float* ckpt_in = nullptr;
};

msc_status s6_bwd_launch(const S6BwdArgs& a, cudaStream_t stream);

// Decode step: one token per row, state [batch * dim, N] updated in place.
struct S6StepArgs {
    int64_t batch, dim;
    int N;
    bool bf16;
    const void *u, *delta, *z, *B, *C;
    const float *A, *D, *delta_bias;
    float *state, *y;
};

msc_status s6_step_launch(const S6StepArgs& a, cudaStream_t stream);

// Causal depthwise conv1d (+ SiLU) front end and its decode step.
struct Conv1dArgs {
    int64_t batch, dim, L;
    int K, silu;
    bool in_bf16, out_bf16;
    const void* x;
    const float *weight, *bias;
    float* state;
    void* out;
};

msc_status conv1d_fwd_launch(const Conv1dArgs& a, cudaStream_t stream);
msc_status conv1d_update_launch(const Conv1dArgs& a, cudaStream_t stream);
// dout, dx: [batch, dim, L] fp32; dweight [dim, K], dbias [dim] (may be null) fp32, overwritten.
msc_status conv1d_bwd_launch(const Conv1dArgs& a, const float* dout, float* dx, float* dweight, float* dbias,
                             cudaStream_t stream);

struct SsdArgs {
    int64_t batch, L, H, P, N, G, Q;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias;
    float *y, *final_state;
    void* workspace;
    // optional, for the backward: the state entering every chunk in fp32
    // [b, nc, H, P, N], written by the forward's state pass
    float* Hin32 = nullptr;
};

size_t ssd_workspace(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                     int64_t Q);
msc_status ssd_launch(const SsdArgs& a, cudaStream_t stream);
// For the backward: Delta and in-chunk cumsum cs [b, H, nc * Q], chunk states
// S and the state entering every chunk Hin32 [b, nc, H, P, N] (all fp32), and
// the same states as bf16 hi + lo tile images Himg [b, nc, H][2][64 x 128]
// (K-major, 128-byte swizzle) for the tensor cores.
msc_status ssd_states(const SsdArgs& a, float* dt, float* cs, float* S, float* Hin32, uint16_t* Himg,
                      cudaStream_t stream);
// U_c [b, nc, H, P, N] = sum over the chunk of exp(cs_i) g_i (x) C_i, g = dy
// (times silu(z) when a.z is set), on the chunk-state tensor-core kernel; cs from
// ssd_states or from the forward's workspace.
msc_status ssd_ugrad(const SsdArgs& a, const void* dy, const float* cs, float* U, cudaStream_t stream);

// SSD backward: the forward's inputs in f (y, final_state, workspace unused),
// the upstream gradient dy (bf16, shaped like x) and fp32 gradients.
struct SsdBwdArgs {
    SsdArgs f;
    const void* dy;
    float *dx, *ddelta, *dA, *dB, *dC, *dD, *dz, *ddelta_bias;
    void* workspace;
};

size_t ssd_bwd_workspace(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t Q, bool has_z);
msc_status ssd_bwd_launch(const SsdBwdArgs& a, cudaStream_t stream);

}  // namespace msc_host
