// msc_api.cu -- extern "C" entry points of libmsc: argument validation,
// workspace sizing, status reporting; the work itself is in the kernels.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tma.cuh"

namespace msc_host {

static thread_local char g_last_error[512] = "";

msc_status fail(msc_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { g_last_error[0] = 0; }

msc_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return MSC_OK;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) {
        fail(MSC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        fail(MSC_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return false;
    }
    return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MSC_REQUIRE(cond, ...)                                          \
    do {                                                                \
        if (!(cond)) return fail(MSC_ERR_INVALID_ARG, __VA_ARGS__);     \
    } while (0)

#define MSC_PTR(p, name)                                                \
    do {                                                                \
        MSC_REQUIRE((p) != nullptr, "%s must not be NULL", name);       \
        MSC_REQUIRE(aligned16(p), "%s must be 16-byte aligned", name);  \
    } while (0)

#define MSC_OPT_PTR(p, name)                                            \
    do {                                                                \
        if ((p) != nullptr) MSC_REQUIRE(aligned16(p), "%s must be 16-byte aligned", name); \
    } while (0)

// max_dstate: 64 for the forward scan (exponential Euler, zero-order hold,
// trapezoid), 16 for the backward, the decode step and the fused conv front end.
static msc_status check_s6_dims(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                msc_dtype dt, int64_t max_dstate = 16) {
    MSC_REQUIRE(batch >= 1 && dim >= 1 && seqlen >= 1, "batch, dim and seqlen must be >= 1 (got %lld, %lld, %lld)",
                (long long)batch, (long long)dim, (long long)seqlen);
    MSC_REQUIRE(dt == MSC_F32 || dt == MSC_BF16, "in_dtype must be MSC_F32 or MSC_BF16");
    if (dstate < 1 || dstate > max_dstate)
        return fail(MSC_ERR_UNSUPPORTED, "dstate must be in [1, %lld] (got %lld)", (long long)max_dstate,
                    (long long)dstate);
    if (batch > 65535) return fail(MSC_ERR_UNSUPPORTED, "batch must be <= 65535");
    if (dim > (int64_t)1 << 36) return fail(MSC_ERR_UNSUPPORTED, "dim too large");
    // the largest element index must fit comfortably in int64 arithmetic
    MSC_REQUIRE(batch * dim <= ((int64_t)1 << 40) && seqlen <= ((int64_t)1 << 40) / (batch * dim) * ((int64_t)1 << 20),
                "batch * dim * seqlen too large");
    return MSC_OK;
}

}  // namespace msc_host

using namespace msc_host;

extern "C" {

int msc_version(void) { return 100; }

const char* msc_status_string(msc_status s) {
    switch (s) {
        case MSC_OK: return "MSC_OK";
        case MSC_ERR_INVALID_ARG: return "MSC_ERR_INVALID_ARG";
        case MSC_ERR_UNSUPPORTED: return "MSC_ERR_UNSUPPORTED";
        case MSC_ERR_CUDA: return "MSC_ERR_CUDA";
        case MSC_ERR_TIMEOUT: return "MSC_ERR_TIMEOUT";
        case MSC_ERR_WORKSPACE: return "MSC_ERR_WORKSPACE";
    }
    return "MSC_ERR_UNKNOWN";
}

const char* msc_last_error(void) { return g_last_error; }

size_t msc_selective_scan_fwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen,
                                             int64_t dstate) {
    if (batch < 1 || dim < 1 || seqlen < 1 || dstate < 1 || dstate > MSC_S6_FWD_MAX_DSTATE) return 0;
    return s6_fwd_plan(batch, dim, seqlen, dstate).workspace;
}

msc_status msc_selective_scan_fwd_ex(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                     msc_dtype in_dtype, msc_discretization disc, const void* u,
                                     const void* delta, const float* A, const void* B, const void* C,
                                     const float* D, const void* z, const float* delta_bias, const float* h0,
                                     float* y, float* h_last, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    return msc_host::s6_fwd_entry(batch, dim, seqlen, dstate, in_dtype, (int)disc, u, delta, A, B, C, D, z,
                                  delta_bias, h0, y, h_last, workspace, workspace_bytes, stream, SIZE_MAX);
}

}  // extern "C"

namespace msc_host {

msc_status s6_fwd_entry(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, msc_dtype in_dtype, int disc,
                        const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, const float* h0, float* y,
                        float* h_last, void* workspace, size_t workspace_bytes, void* stream,
                        size_t max_required) {
    clear_error();
    msc_status s = check_s6_dims(batch, dim, seqlen, dstate, in_dtype, MSC_S6_FWD_MAX_DSTATE);
    if (s != MSC_OK) return s;
    MSC_REQUIRE(disc == MSC_DISC_EULER || disc == MSC_DISC_ZOH || disc == MSC_DISC_TRAPEZOID,
                "disc must be MSC_DISC_EULER, MSC_DISC_ZOH or MSC_DISC_TRAPEZOID");
    MSC_PTR(u, "u"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B");
    MSC_PTR(C, "C"); MSC_PTR(y, "y");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    MSC_OPT_PTR(h0, "h0"); MSC_OPT_PTR(h_last, "h_last");
    S6Plan plan = s6_fwd_plan(batch, dim, seqlen, dstate, max_required);
    if (plan.workspace_required && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", plan.workspace,
                    workspace ? workspace_bytes : (size_t)0);
    if (workspace != nullptr)
        MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
    S6FwdArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.delta_bias = delta_bias; a.h0 = h0; a.y = y; a.h_last = h_last;
    a.workspace = workspace;
    a.workspace_bytes = workspace ? workspace_bytes : 0;
    a.disc = disc;
    return s6_fwd_launch(a, plan, static_cast<cudaStream_t>(stream));
}

}  // namespace msc_host

extern "C" {

msc_status msc_selective_scan_fwd_conv(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       int64_t conv_width, msc_dtype in_dtype, const void* x,
                                       const float* conv_weight, const float* conv_bias, const void* delta,
                                       const float* A, const void* B, const void* C, const float* D,
                                       const void* z, const float* delta_bias, const float* h0, float* y,
                                       float* h_last, void* workspace, size_t workspace_bytes, void* stream) {
    clear_error();
    msc_status s = check_s6_dims(batch, dim, seqlen, dstate, in_dtype);
    if (s != MSC_OK) return s;
    if (conv_width < 1 || conv_width > 4)
        return fail(MSC_ERR_UNSUPPORTED, "conv_width must be 1..4 (got %lld)", (long long)conv_width);
    MSC_PTR(x, "x"); MSC_PTR(conv_weight, "conv_weight"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A");
    MSC_PTR(B, "B"); MSC_PTR(C, "C"); MSC_PTR(y, "y");
    MSC_OPT_PTR(conv_bias, "conv_bias"); MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z");
    MSC_OPT_PTR(delta_bias, "delta_bias"); MSC_OPT_PTR(h0, "h0"); MSC_OPT_PTR(h_last, "h_last");
    S6Plan plan = s6_fwd_plan(batch, dim, seqlen, dstate);
    if (plan.workspace_required && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", plan.workspace,
                    workspace ? workspace_bytes : (size_t)0);
    if (workspace != nullptr)
        MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
    S6FwdArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = x; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.delta_bias = delta_bias; a.h0 = h0; a.y = y; a.h_last = h_last;
    a.workspace = workspace;
    a.workspace_bytes = workspace ? workspace_bytes : 0;
    a.conv_w = conv_weight; a.conv_b = conv_bias; a.conv_k = (int)conv_width;
    return s6_fwd_launch(a, plan, static_cast<cudaStream_t>(stream));
}

msc_status msc_selective_state_update(int64_t batch, int64_t dim, int64_t dstate, msc_dtype in_dtype,
                                      const void* u, const void* delta, const float* A, const void* B,
                                      const void* C, const float* D, const void* z, const float* delta_bias,
                                      float* state, float* y, void* stream) {
    clear_error();
    msc_status s = check_s6_dims(batch, dim, 1, dstate, in_dtype, MSC_S6_FWD_MAX_DSTATE);
    if (s != MSC_OK) return s;
    MSC_PTR(u, "u"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B");
    MSC_PTR(C, "C"); MSC_PTR(state, "state"); MSC_PTR(y, "y");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    S6StepArgs a{};
    a.batch = batch; a.dim = dim; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.delta_bias = delta_bias; a.state = state; a.y = y;
    return s6_step_launch(a, static_cast<cudaStream_t>(stream));
}

static msc_status check_conv_dims(int64_t batch, int64_t dim, int64_t seqlen, int64_t width, msc_dtype in_dt,
                                  msc_dtype out_dt) {
    MSC_REQUIRE(batch >= 1 && dim >= 1 && seqlen >= 1, "batch, dim and seqlen must be >= 1 (got %lld, %lld, %lld)",
                (long long)batch, (long long)dim, (long long)seqlen);
    MSC_REQUIRE(in_dt == MSC_F32 || in_dt == MSC_BF16, "in_dtype must be MSC_F32 or MSC_BF16");
    MSC_REQUIRE(out_dt == MSC_F32 || out_dt == MSC_BF16, "out_dtype must be MSC_F32 or MSC_BF16");
    if (width < 1 || width > 8) return fail(MSC_ERR_UNSUPPORTED, "width must be in [1, 8] (got %lld)", (long long)width);
    MSC_REQUIRE(batch * dim <= ((int64_t)1 << 40) && seqlen <= ((int64_t)1 << 40) / (batch * dim) * ((int64_t)1 << 20),
                "batch * dim * seqlen too large");
    return MSC_OK;
}

msc_status msc_causal_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width, msc_dtype in_dtype,
                                 msc_dtype out_dtype, const void* x, const float* weight, const float* bias, int silu,
                                 void* out, void* stream) {
    clear_error();
    msc_status s = check_conv_dims(batch, dim, seqlen, width, in_dtype, out_dtype);
    if (s != MSC_OK) return s;
    MSC_PTR(x, "x"); MSC_PTR(weight, "weight"); MSC_PTR(out, "out");
    MSC_OPT_PTR(bias, "bias");
    Conv1dArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.K = (int)width; a.silu = silu != 0;
    a.in_bf16 = in_dtype == MSC_BF16; a.out_bf16 = out_dtype == MSC_BF16;
    a.x = x; a.weight = weight; a.bias = bias; a.out = out;
    return conv1d_fwd_launch(a, static_cast<cudaStream_t>(stream));
}

msc_status msc_causal_conv1d_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width, msc_dtype in_dtype,
                                 const void* x, const float* weight, const float* bias, int silu, const float* dout,
                                 float* dx, float* dweight, float* dbias, void* stream) {
    clear_error();
    msc_status s = check_conv_dims(batch, dim, seqlen, width, in_dtype, MSC_F32);
    if (s != MSC_OK) return s;
    MSC_PTR(x, "x"); MSC_PTR(weight, "weight"); MSC_PTR(dout, "dout"); MSC_PTR(dx, "dx");
    MSC_PTR(dweight, "dweight");
    MSC_OPT_PTR(bias, "bias"); MSC_OPT_PTR(dbias, "dbias");
    Conv1dArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.K = (int)width; a.silu = silu != 0;
    a.in_bf16 = in_dtype == MSC_BF16; a.out_bf16 = false;
    a.x = x; a.weight = weight; a.bias = bias;
    return conv1d_bwd_launch(a, dout, dx, dweight, dbias, static_cast<cudaStream_t>(stream));
}

msc_status msc_causal_conv1d_update(int64_t batch, int64_t dim, int64_t width, msc_dtype in_dtype,
                                    msc_dtype out_dtype, const void* x, const float* weight, const float* bias,
                                    int silu, float* conv_state, void* out, void* stream) {
    clear_error();
    msc_status s = check_conv_dims(batch, dim, 1, width, in_dtype, out_dtype);
    if (s != MSC_OK) return s;
    MSC_PTR(x, "x"); MSC_PTR(weight, "weight"); MSC_PTR(out, "out");
    MSC_OPT_PTR(bias, "bias");
    if (width > 1) MSC_PTR(conv_state, "conv_state");
    Conv1dArgs a{};
    a.batch = batch; a.dim = dim; a.L = 1; a.K = (int)width; a.silu = silu != 0;
    a.in_bf16 = in_dtype == MSC_BF16; a.out_bf16 = out_dtype == MSC_BF16;
    a.x = x; a.weight = weight; a.bias = bias; a.out = out; a.state = conv_state;
    return conv1d_update_launch(a, static_cast<cudaStream_t>(stream));
}

msc_status msc_selective_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                  msc_dtype in_dtype, const void* u, const void* delta,
                                  const float* A, const void* B, const void* C, const float* D,
                                  const void* z, const float* delta_bias, const float* h0,
                                  float* y, float* h_last, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return msc_selective_scan_fwd_ex(batch, dim, seqlen, dstate, in_dtype, MSC_DISC_EULER, u, delta, A, B, C, D,
                                     z, delta_bias, h0, y, h_last, workspace, workspace_bytes, stream);
}

size_t msc_selective_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen,
                                             int64_t dstate) {
    if (batch < 1 || dim < 1 || seqlen < 1 || dstate < 1 || dstate > MSC_S6_FWD_MAX_DSTATE) return 0;
    return s6_bwd_workspace(batch, dim, seqlen, dstate);
}

msc_status msc_selective_scan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                  msc_dtype in_dtype, const void* u, const void* delta,
                                  const float* A, const void* B, const void* C, const float* D,
                                  const void* z, const float* delta_bias, const void* dy,
                                  float* du, float* ddelta, float* dA, float* dB, float* dC,
                                  float* dD, float* dz, float* ddelta_bias, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    clear_error();
    msc_status s = check_s6_dims(batch, dim, seqlen, dstate, in_dtype, MSC_S6_FWD_MAX_DSTATE);
    if (s != MSC_OK) return s;
    MSC_PTR(u, "u"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B");
    MSC_PTR(C, "C"); MSC_PTR(dy, "dy");
    MSC_PTR(du, "du"); MSC_PTR(ddelta, "ddelta"); MSC_PTR(dA, "dA"); MSC_PTR(dB, "dB"); MSC_PTR(dC, "dC");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    MSC_REQUIRE((D == nullptr) == (dD == nullptr), "dD must be given exactly when D is given");
    MSC_REQUIRE((z == nullptr) == (dz == nullptr), "dz must be given exactly when z is given");
    MSC_REQUIRE((delta_bias == nullptr) == (ddelta_bias == nullptr),
                "ddelta_bias must be given exactly when delta_bias is given");
    MSC_OPT_PTR(dD, "dD"); MSC_OPT_PTR(dz, "dz"); MSC_OPT_PTR(ddelta_bias, "ddelta_bias");
    const size_t need = s6_bwd_workspace(batch, dim, seqlen, dstate);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                        workspace ? workspace_bytes : (size_t)0);
        MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
    }
    S6BwdArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C; a.dy = dy;
    a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.du = du; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz;
    a.ddelta_bias = ddelta_bias; a.workspace = workspace;
    return s6_bwd_launch(a, static_cast<cudaStream_t>(stream));
}

// The training pair's common limits: dstate <= 16 (a checkpoint holds 16
// states), seqlen a multiple of 8 (whole checkpoint groups, 16-byte rows in both dtypes) and
// seqlen, dim below 2^31 (32-bit TMA tile coordinates).
static msc_status check_train_dims(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, msc_dtype dt) {
    msc_status s = check_s6_dims(batch, dim, seqlen, dstate, dt);
    if (s != MSC_OK) return s;
    if (seqlen % 8 != 0)
        return fail(MSC_ERR_UNSUPPORTED, "the training pair needs seqlen a multiple of 8 (got %lld)",
                    (long long)seqlen);
    constexpr int64_t kMaxCoord = ((int64_t)1 << 31) - 64;
    if (seqlen > kMaxCoord || dim > kMaxCoord)
        return fail(MSC_ERR_UNSUPPORTED, "the training pair needs seqlen and dim below 2^31");
    return MSC_OK;
}

size_t msc_selective_scan_ckpt_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate) {
    if (batch < 1 || dim < 1 || seqlen < 1 || dstate < 1 || dstate > 16 || seqlen % 8 != 0) return 0;
    return (size_t)batch * (size_t)dim * (size_t)(seqlen / 8) * 16 * sizeof(float);
}

msc_status msc_selective_scan_fwd_train(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                        msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                        const void* B, const void* C, const float* D, const void* z,
                                        const float* delta_bias, float* y, float* ckpt, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    clear_error();
    msc_status s = check_train_dims(batch, dim, seqlen, dstate, in_dtype);
    if (s != MSC_OK) return s;
    MSC_PTR(u, "u"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B");
    MSC_PTR(C, "C"); MSC_PTR(y, "y"); MSC_PTR(ckpt, "ckpt");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    S6Plan plan = s6_fwd_plan(batch, dim, seqlen, dstate);
    if (plan.workspace_required && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", plan.workspace,
                    workspace ? workspace_bytes : (size_t)0);
    if (workspace != nullptr)
        MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
    S6FwdArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.delta_bias = delta_bias; a.h0 = nullptr; a.y = y; a.h_last = nullptr;
    a.workspace = workspace;
    a.workspace_bytes = workspace ? workspace_bytes : 0;
    a.ckpt = ckpt;
    return s6_fwd_launch(a, plan, static_cast<cudaStream_t>(stream));
}

msc_status msc_selective_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                       const void* B, const void* C, const float* D, const void* z,
                                       const float* delta_bias, const void* dy, const float* ckpt, float* du,
                                       float* ddelta, float* dA, float* dB, float* dC, float* dD, float* dz,
                                       float* ddelta_bias, void* stream) {
    clear_error();
    msc_status s = check_train_dims(batch, dim, seqlen, dstate, in_dtype);
    if (s != MSC_OK) return s;
    MSC_PTR(u, "u"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B");
    MSC_PTR(C, "C"); MSC_PTR(dy, "dy"); MSC_PTR(ckpt, "ckpt");
    MSC_PTR(du, "du"); MSC_PTR(ddelta, "ddelta"); MSC_PTR(dA, "dA"); MSC_PTR(dB, "dB"); MSC_PTR(dC, "dC");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    MSC_REQUIRE((D == nullptr) == (dD == nullptr), "dD must be given exactly when D is given");
    MSC_REQUIRE((z == nullptr) == (dz == nullptr), "dz must be given exactly when z is given");
    MSC_REQUIRE((delta_bias == nullptr) == (ddelta_bias == nullptr),
                "ddelta_bias must be given exactly when delta_bias is given");
    MSC_OPT_PTR(dD, "dD"); MSC_OPT_PTR(dz, "dz"); MSC_OPT_PTR(ddelta_bias, "ddelta_bias");
    S6BwdArgs a{};
    a.batch = batch; a.dim = dim; a.L = seqlen; a.N = (int)dstate; a.bf16 = in_dtype == MSC_BF16;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C; a.dy = dy;
    a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.du = du; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz;
    a.ddelta_bias = ddelta_bias; a.workspace = nullptr; a.ckpt_in = ckpt;
    return s6_bwd_launch(a, static_cast<cudaStream_t>(stream));
}

size_t msc_ssd_chunked_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads,
                                          int64_t headdim, int64_t dstate, int64_t ngroups,
                                          int64_t chunk) {
    if (batch < 1 || seqlen < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        nheads % ngroups != 0 || chunk < 1)
        return 0;
    return ssd_workspace(batch, seqlen, nheads, headdim, dstate, ngroups, chunk);
}

msc_status msc_ssd_chunked_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t dstate, int64_t ngroups, int64_t chunk, msc_dtype in_dtype,
                               const void* x, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, float* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream) {
    clear_error();
    MSC_REQUIRE(batch >= 1 && seqlen >= 1 && nheads >= 1 && headdim >= 1 && dstate >= 1 && ngroups >= 1,
                "all sizes must be >= 1");
    MSC_REQUIRE(nheads % ngroups == 0, "ngroups (%lld) must divide nheads (%lld)", (long long)ngroups,
                (long long)nheads);
    MSC_REQUIRE(in_dtype == MSC_F32 || in_dtype == MSC_BF16, "in_dtype must be MSC_F32 or MSC_BF16");
    if (in_dtype != MSC_BF16) return fail(MSC_ERR_UNSUPPORTED, "SSD supports bf16 inputs only");
    if (headdim != 64 || dstate != 128)
        return fail(MSC_ERR_UNSUPPORTED, "SSD supports headdim 64 and dstate 128 (got %lld, %lld)",
                    (long long)headdim, (long long)dstate);
    if (chunk != 64 && chunk != 128 && chunk != 256)
        return fail(MSC_ERR_UNSUPPORTED, "chunk must be 64, 128 or 256 (got %lld)", (long long)chunk);
    if (batch > 65535 || nheads > 65535) return fail(MSC_ERR_UNSUPPORTED, "batch and nheads must be <= 65535");
    MSC_REQUIRE(seqlen <= ((int64_t)1 << 31), "seqlen too large");
    MSC_PTR(x, "x"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B"); MSC_PTR(C, "C");
    MSC_PTR(y, "y");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    MSC_OPT_PTR(final_state, "final_state");
    const size_t need = ssd_workspace(batch, seqlen, nheads, headdim, dstate, ngroups, chunk);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    workspace ? workspace_bytes : (size_t)0);
    MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 1023u) == 0, "workspace must be 1024-byte aligned");
    SsdArgs a{};
    a.batch = batch; a.L = seqlen; a.H = nheads; a.P = headdim; a.N = dstate; a.G = ngroups; a.Q = chunk;
    a.x = x; a.delta = delta; a.B = B; a.C = C; a.z = z; a.A = A; a.D = D; a.delta_bias = delta_bias;
    a.y = y; a.final_state = final_state; a.workspace = workspace;
    return ssd_launch(a, static_cast<cudaStream_t>(stream));
}

size_t msc_ssd_chunked_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads,
                                          int64_t headdim, int64_t dstate, int64_t ngroups,
                                          int64_t chunk, int has_z) {
    if (batch < 1 || seqlen < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        nheads % ngroups != 0 || chunk < 1)
        return 0;
    return ssd_bwd_workspace(batch, seqlen, nheads, ngroups, chunk, has_z != 0);
}

msc_status msc_ssd_chunked_bwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                               int64_t dstate, int64_t ngroups, int64_t chunk, msc_dtype in_dtype,
                               const void* x, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, const void* dy, float* dx, float* ddelta,
                               float* dA, float* dB, float* dC, float* dD, float* dz,
                               float* ddelta_bias, void* workspace, size_t workspace_bytes,
                               void* stream) {
    clear_error();
    MSC_REQUIRE(batch >= 1 && seqlen >= 1 && nheads >= 1 && headdim >= 1 && dstate >= 1 && ngroups >= 1,
                "all sizes must be >= 1");
    MSC_REQUIRE(nheads % ngroups == 0, "ngroups (%lld) must divide nheads (%lld)", (long long)ngroups,
                (long long)nheads);
    MSC_REQUIRE(in_dtype == MSC_F32 || in_dtype == MSC_BF16, "in_dtype must be MSC_F32 or MSC_BF16");
    if (in_dtype != MSC_BF16) return fail(MSC_ERR_UNSUPPORTED, "SSD supports bf16 inputs only");
    if (headdim != 64 || dstate != 128)
        return fail(MSC_ERR_UNSUPPORTED, "SSD supports headdim 64 and dstate 128 (got %lld, %lld)",
                    (long long)headdim, (long long)dstate);
    if (chunk != 64 && chunk != 128 && chunk != 256)
        return fail(MSC_ERR_UNSUPPORTED, "chunk must be 64, 128 or 256 (got %lld)", (long long)chunk);
    if (batch > 65535 || nheads > 65535) return fail(MSC_ERR_UNSUPPORTED, "batch and nheads must be <= 65535");
    if (ngroups != 1 && (nheads / ngroups) % 16 != 0)
        return fail(MSC_ERR_UNSUPPORTED, "heads per group must be a multiple of 16 when ngroups > 1");
    MSC_REQUIRE(seqlen <= ((int64_t)1 << 31), "seqlen too large");
    MSC_PTR(x, "x"); MSC_PTR(delta, "delta"); MSC_PTR(A, "A"); MSC_PTR(B, "B"); MSC_PTR(C, "C");
    MSC_PTR(dy, "dy"); MSC_PTR(dx, "dx"); MSC_PTR(ddelta, "ddelta"); MSC_PTR(dA, "dA");
    MSC_PTR(dB, "dB"); MSC_PTR(dC, "dC");
    MSC_OPT_PTR(D, "D"); MSC_OPT_PTR(z, "z"); MSC_OPT_PTR(delta_bias, "delta_bias");
    MSC_REQUIRE((D == nullptr) == (dD == nullptr), "dD must be given exactly when D is");
    MSC_REQUIRE((z == nullptr) == (dz == nullptr), "dz must be given exactly when z is");
    MSC_REQUIRE((delta_bias == nullptr) == (ddelta_bias == nullptr),
                "ddelta_bias must be given exactly when delta_bias is");
    const size_t need = ssd_bwd_workspace(batch, seqlen, nheads, ngroups, chunk, z != nullptr);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(MSC_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    workspace ? workspace_bytes : (size_t)0);
    MSC_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 1023u) == 0, "workspace must be 1024-byte aligned");
    SsdBwdArgs a{};
    a.f.batch = batch; a.f.L = seqlen; a.f.H = nheads; a.f.P = headdim; a.f.N = dstate; a.f.G = ngroups;
    a.f.Q = chunk;
    a.f.x = x; a.f.delta = delta; a.f.B = B; a.f.C = C; a.f.z = z; a.f.A = A; a.f.D = D;
    a.f.delta_bias = delta_bias;
    a.dy = dy; a.dx = dx; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz;
    a.ddelta_bias = ddelta_bias; a.workspace = workspace;
    return ssd_bwd_launch(a, static_cast<cudaStream_t>(stream));
}

msc_status msc_check_device_status(void* stream) {
    clear_error();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned int code = 0, site = 0;
    msc_status s = s6_fwd_take_status(&code, &site);
    if (s != MSC_OK) return s;
    if (code == 0) {
        s = s6_bwd_take_status(&code, &site);
        if (s != MSC_OK) return s;
    }
    if (code == 0) {
        s = ssd_take_status(&code, &site);
        if (s != MSC_OK) return s;
    }
    if (code == 0) {
        s = ssd_bwd_take_status(&code, &site);
        if (s != MSC_OK) return s;
    }
    if (code == 0) return MSC_OK;
    if (code == MSC_ERR_TIMEOUT) return fail(MSC_ERR_TIMEOUT, "device-side wait ran out (site %u)", site);
    return fail((msc_status)code, "device status %u (site %u)", code, site);
}

}  // extern "C"
