// C ABI of liblla.so: argument validation and dispatch to the kernels.
// Declarations, layouts and error behaviour: include/lla.h.
#include <stdint.h>

#include "bwd_simt.cuh"
#include "decode.cuh"
#include "gdn.cuh"
#include "fwd_simt.cuh"
#include "fwd_tc.cuh"
#include "lambda_mlp.cuh"
#include "lla_common.cuh"

using namespace lla;

namespace {

constexpr long long kMaxGridY = 65535;

bool is_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool is_chunk(int c) { return c == 16 || c == 32 || c == 64 || c == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

lla_status fwd_shape_status(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt)
{
    if (B < 0 || H < 0 || T < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (!is_chunk(chunk) || !is_dim(dk) || !is_dim(dv)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (T % chunk != 0 || T > (1 << 24)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > kMaxGridY) return LLA_ERR_UNSUPPORTED_SHAPE;
    return LLA_OK;
}

}  // namespace

namespace lla {

// Every check lla_fwd makes before it looks at the workspace: shape and
// dtype, the empty case (LLA_OK with *empty set), pointers and alignment.
lla_status fwd_args_status(const void *q, const void *k, const void *v, const float *g,
                           const float *lambda, const void *out, int B, int H, int T, int dk,
                           int dv, int chunk, lla_dtype in_dt, lla_dtype out_dt, bool *empty)
{
    *empty = false;
    lla_status st = fwd_shape_status(B, H, T, dk, dv, chunk, in_dt);
    if (st != LLA_OK) return st;
    if (out_dt != LLA_F32 && out_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt == LLA_F32 && out_dt != LLA_F32) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H * T == 0) {
        *empty = true;
        return LLA_OK;
    }
    if (!q || !k || !v || !g || !lambda || !out) return LLA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(lambda) ||
        !aligned16(out))
        return LLA_ERR_INVALID_ARGUMENT;
    return LLA_OK;
}

}  // namespace lla

namespace {

SimtFwdArgs simt_args(const void *q, const void *k, const void *v, const float *g,
                      const float *lambda, void *out, int B, int H, int T, int dk, int dv,
                      int chunk, lla_dtype in_dt, lla_dtype out_dt, void *ws, void *stream)
{
    SimtFwdArgs A;
    A.q = q; A.k = k; A.v = v; A.g = g; A.lam = lambda; A.out = out;
    A.B = B; A.H = H; A.T = T; A.dk = dk; A.dv = dv; A.C = chunk;
    A.L = lla_num_levels(T);
    A.in_dt = in_dt; A.out_dt = out_dt; A.workspace = ws; A.stream = stream;
    return A;
}

}  // namespace

extern "C" {

const char *lla_status_string(lla_status s)
{
    switch (s) {
    case LLA_OK: return "LLA_OK";
    case LLA_ERR_INVALID_ARGUMENT: return "LLA_ERR_INVALID_ARGUMENT";
    case LLA_ERR_UNSUPPORTED_SHAPE: return "LLA_ERR_UNSUPPORTED_SHAPE";
    case LLA_ERR_WORKSPACE_TOO_SMALL: return "LLA_ERR_WORKSPACE_TOO_SMALL";
    case LLA_ERR_CUDA: return "LLA_ERR_CUDA";
    case LLA_ERR_DEVICE_REPORTED: return "LLA_ERR_DEVICE_REPORTED";
    }
    return "LLA_UNKNOWN_STATUS";
}

int lla_version(void) { return 100; }

int lla_num_levels(int T)
{
    if (T <= 0) return 0;
    return 1 + bit_length_u32((uint32_t)(T - 1));
}

size_t lla_fwd_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt)
{
    if (fwd_shape_status(B, H, T, dk, dv, chunk, in_dt) != LLA_OK) return 0;
    if ((long long)B * H * T == 0) return 0;
    if (tc_supported(dk, dv, in_dt)) return tc_workspace_bytes(B, H, T, dk);
    SimtFwdArgs A = simt_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, T,
                              dk, dv, chunk, in_dt, LLA_F32, nullptr, nullptr);
    return simt_workspace_bytes(A);
}

int lla_fwd_launches(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt,
                     lla_dtype out_dt)
{
    if (fwd_shape_status(B, H, T, dk, dv, chunk, in_dt) != LLA_OK) return 0;
    if (out_dt != LLA_F32 && out_dt != LLA_BF16) return 0;
    if (in_dt == LLA_F32 && out_dt != LLA_F32) return 0;
    if ((long long)B * H * T == 0) return 0;
    if (tc_supported(dk, dv, in_dt)) return tc_launches(T);
    return T / chunk > 1 ? 4 : 3;
}

lla_status lla_device_error_check(const int32_t *device_error, int32_t *code, void *stream)
{
    if (device_error == nullptr) return LLA_ERR_INVALID_ARGUMENT;
    int32_t h = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&h, device_error, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return LLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LLA_ERR_CUDA;
    if (code) *code = h;
    return h == 0 ? LLA_OK : LLA_ERR_DEVICE_REPORTED;
}

void lla_debug_withhold_first_product(int enable) { lla::tc_set_withhold_first_product(enable); }

lla_status lla_fwd(const void *q, const void *k, const void *v, const float *g,
                   const float *lambda, void *out, int B, int H, int T, int dk, int dv,
                   int chunk, lla_dtype in_dt, lla_dtype out_dt, void *workspace,
                   size_t workspace_bytes, int32_t *device_error, void *stream)
{
    bool empty = false;
    lla_status st = fwd_args_status(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt,
                                    out_dt, &empty);
    if (st != LLA_OK || empty) return st;
    const size_t need = lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt);
    if (workspace_bytes < need) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0))
        return LLA_ERR_INVALID_ARGUMENT;
    if (tc_supported(dk, dv, in_dt)) {
        TcFwdArgs A;
        A.q = q; A.k = k; A.v = v; A.g = g; A.lam = lambda; A.out = out;
        A.B = B; A.H = H; A.T = T; A.L = lla_num_levels(T); A.dk = dk; A.out_dt = out_dt;
        A.workspace = workspace; A.device_error = device_error; A.stream = stream;
        return tc_fwd(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
    }
    SimtFwdArgs A = simt_args(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt, out_dt,
                              workspace, stream);
    if (simt_max_smem_bytes(A) > 227 * 1024) return LLA_ERR_UNSUPPORTED_SHAPE;
    return simt_fwd(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

size_t lla_fwd_lambda_mlp_workspace_bytes(int B, int H, int T, int dk, int dv, int Dd, int chunk,
                                          lla_dtype in_dt)
{
    if (Dd < 1 || Dd > 256) return 0;
    const size_t fwd = lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt);
    if (fwd == 0) return 0;
    // lambda staged in the workspace when it cannot be computed in the read-out
    const size_t lam = align_up((size_t)B * H * T * lla_num_levels(T) * sizeof(float), 256);
    return lam + fwd;
}

lla_status lla_fwd_lambda_mlp(const void *q, const void *k, const void *v, const float *g,
                              const void *d, const float *W1, const float *W2, const float *b,
                              void *out, int B, int H, int T, int dk, int dv, int Dd, int chunk,
                              lla_dtype in_dt, lla_dtype out_dt, void *workspace,
                              size_t workspace_bytes, int32_t *device_error, void *stream)
{
    // lla_fwd's checks with a stand-in lambda pointer (lambda is not an input here)
    bool empty = false;
    lla_status st = fwd_args_status(q, k, v, g, g, out, B, H, T, dk, dv, chunk, in_dt, out_dt,
                                    &empty);
    if (st != LLA_OK || empty) return st;
    const int L = lla_num_levels(T);
    if (Dd < 1 || Dd > 256 || L > 32) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (!d || !W1 || !W2 || !b || !aligned16(d)) return LLA_ERR_INVALID_ARGUMENT;
    const size_t need = lla_fwd_lambda_mlp_workspace_bytes(B, H, T, dk, dv, Dd, chunk, in_dt);
    if (workspace_bytes < need) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0) return LLA_ERR_INVALID_ARGUMENT;
    if (d == k && Dd == dk && tc_mlp_supported(dk, dv, in_dt, L)) {
        TcFwdArgs A;
        A.q = q; A.k = k; A.v = v; A.g = g; A.lam = nullptr; A.out = out;
        A.B = B; A.H = H; A.T = T; A.L = L; A.dk = dk; A.out_dt = out_dt;
        A.W1 = W1; A.W2 = W2; A.bmlp = b;
        A.workspace = workspace; A.device_error = device_error; A.stream = stream;
        return tc_fwd(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
    }
    float *lam = (float *)workspace;
    const size_t lam_bytes = align_up((size_t)B * H * T * L * sizeof(float), 256);
    st = lla_lambda_mlp(d, W1, W2, b, lam, B, H, T, Dd, L, in_dt, device_error, stream);
    if (st != LLA_OK) return st;
    return lla_fwd(q, k, v, g, lam, out, B, H, T, dk, dv, chunk, in_dt, out_dt,
                   (char *)workspace + lam_bytes, workspace_bytes - lam_bytes, device_error, stream);
}

size_t lla_decode_state_bytes(int B, int H, int dk, int dv, int Ls)
{
    if (B < 0 || H < 0 || dk < 0 || dv < 0 || Ls < 0) return 0;
    return (size_t)B * H * Ls * dk * dv * sizeof(float);
}

lla_status lla_decode_step(float *state_levels, float *state_logdecay, const void *q,
                           const void *k, const void *v, const float *g, const float *lambda,
                           float *out, const int64_t *pos, int B, int H, int dk, int dv, int Ls,
                           lla_dtype in_dt, int32_t *device_error, void *stream)
{
    if (B < 0 || H < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (!is_dim(dk) || !is_dim(dv) || Ls < 1 || Ls > 40) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (B > kMaxGridY || H > (1 << 30)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H == 0) return LLA_OK;
    if (!state_levels || !state_logdecay || !q || !k || !v || !g || !lambda || !out || !pos)
        return LLA_ERR_INVALID_ARGUMENT;
    if (!aligned16(state_levels) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out))
        return LLA_ERR_INVALID_ARGUMENT;
    DecodeArgs A;
    A.S = state_levels; A.D = state_logdecay; A.q = q; A.k = k; A.v = v; A.g = g;
    A.lam = lambda; A.out = out; A.pos = pos; A.B = B; A.H = H; A.dk = dk; A.dv = dv;
    A.Ls = Ls; A.in_dt = in_dt; A.err = device_error; A.stream = stream;
    return decode_step(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

size_t lla_prefill_workspace_bytes(int B, int H, int T)
{
    if (B < 0 || H < 0 || T < 0) return 0;
    return prefill_workspace_bytes(B, H, T);
}

lla_status lla_prefill_state(const void *k, const void *v, const float *g, float *state_levels,
                             float *state_logdecay, int B, int H, int T, int dk, int dv, int Ls,
                             lla_dtype in_dt, void *workspace, size_t workspace_bytes,
                             int32_t *device_error, void *stream)
{
    if (B < 0 || H < 0 || T < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (!is_dim(dk) || !is_dim(dv) || Ls < 1 || Ls > 40) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (T > (1 << 30) || bit_length_u32((uint32_t)T) > Ls) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > kMaxGridY) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H == 0) return LLA_OK;
    if (!state_levels || !state_logdecay) return LLA_ERR_INVALID_ARGUMENT;
    if (T > 0 && (!k || !v || !g)) return LLA_ERR_INVALID_ARGUMENT;
    const size_t need = lla_prefill_workspace_bytes(B, H, T);
    if (workspace_bytes < need) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0) return LLA_ERR_INVALID_ARGUMENT;
    PrefillArgs A;
    A.k = k; A.v = v; A.g = g; A.S = state_levels; A.D = state_logdecay;
    A.B = B; A.H = H; A.T = T; A.dk = dk; A.dv = dv; A.Ls = Ls; A.in_dt = in_dt;
    A.workspace = workspace; A.device_error = device_error; A.stream = stream;
    return prefill_state(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

lla_status lla_lambda_mlp(const void *d, const float *W1, const float *W2, const float *b,
                          float *lambda, int B, int H, int T, int Dd, int L, lla_dtype in_dt,
                          int32_t *device_error, void *stream)
{
    if (B < 0 || H < 0 || T < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (Dd < 1 || Dd > 256 || L < 1 || L > 32) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H * T == 0) return LLA_OK;
    if ((long long)B * H * T > (1LL << 38)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (!d || !W1 || !W2 || !b || !lambda) return LLA_ERR_INVALID_ARGUMENT;
    LambdaMlpArgs A;
    A.d = d; A.W1 = W1; A.W2 = W2; A.bias = b; A.lam = lambda;
    A.B = B; A.H = H; A.T = T; A.Dd = Dd; A.L = L; A.in_dt = in_dt;
    A.device_error = device_error; A.stream = stream;
    return lambda_mlp(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

size_t lla_bwd_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt)
{
    if (fwd_shape_status(B, H, T, dk, dv, chunk, in_dt) != LLA_OK || chunk > 64) return 0;
    if ((long long)B * H * T == 0) return 0;
    lla::BwdArgs A{};
    A.B = B; A.H = H; A.T = T; A.dk = dk; A.dv = dv; A.C = chunk;
    A.L = lla_num_levels(T); A.in_dt = in_dt;
    return lla::bwd_workspace_bytes(A);
}

lla_status lla_bwd(const void *q, const void *k, const void *v, const float *g, const float *lambda,
                   const float *dout, float *dq, float *dk, float *dv, float *dg, float *dlambda,
                   int B, int H, int T, int dk_dim, int dv_dim, int chunk, lla_dtype in_dt,
                   void *workspace, size_t workspace_bytes, int32_t *device_error, void *stream)
{
    lla_status st = fwd_shape_status(B, H, T, dk_dim, dv_dim, chunk, in_dt);
    if (st != LLA_OK) return st;
    if (chunk > 64) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H * T == 0) return LLA_OK;
    if (!q || !k || !v || !g || !lambda || !dout || !dq || !dk || !dv || !dg || !dlambda)
        return LLA_ERR_INVALID_ARGUMENT;
    lla::BwdArgs A{};
    A.B = B; A.H = H; A.T = T; A.dk = dk_dim; A.dv = dv_dim; A.C = chunk;
    A.L = lla_num_levels(T); A.in_dt = in_dt;
    if (workspace_bytes < lla::bwd_workspace_bytes(A)) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0) return LLA_ERR_INVALID_ARGUMENT;
    if (lla::bwd_smem_bytes(A) > 227 * 1024) return LLA_ERR_UNSUPPORTED_SHAPE;
    A.q = q; A.k = k; A.v = v; A.g = g; A.lam = lambda; A.dout = dout;
    A.dq = dq; A.dkey = dk; A.dval = dv; A.dg = dg; A.dlam = dlambda;
    A.workspace = workspace; A.device_error = device_error; A.stream = stream;
    return lla::bwd(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

size_t lla_gdn_fwd_workspace_bytes(int B, int H, int T, int dk, int dv)
{
    if (B <= 0 || H <= 0 || T <= 0 || !is_dim(dk) || !is_dim(dv) || T > (1 << 24)) return 0;
    return lla::gdn_fwd_workspace_bytes(B, H, T, dk, dv);
}

lla_status lla_gdn_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const float *lambda, float *out, float *state_out, int B, int H, int T, int dk,
                       int dv, int Ls_out, lla_dtype in_dt, void *workspace, size_t workspace_bytes,
                       void *stream)
{
    if (B < 0 || H < 0 || T < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (!is_dim(dk) || !is_dim(dv) || T > (1 << 24) || B > 65535 || H > 65535)
        return LLA_ERR_UNSUPPORTED_SHAPE;
    const int need_slots = T > 0 ? bit_length_u32((uint32_t)T) : 0;
    if (state_out && (Ls_out < need_slots || Ls_out > 40)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H * T == 0) return LLA_OK;
    const int L = lla_num_levels(T);
    const int tin_bytes = in_dt == LLA_F32 ? 4 : 2;
    if (!lla::gdn_fwd_fits(T, dk, dv, L, tin_bytes)) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k || !v || !g || !beta || !lambda || !out || !workspace) return LLA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || ((uintptr_t)workspace & 255u) != 0 ||
        workspace_bytes < lla::gdn_fwd_workspace_bytes(B, H, T, dk, dv))
        return LLA_ERR_INVALID_ARGUMENT;
    lla::GdnFwdArgs A;
    A.q = q; A.k = k; A.v = v; A.g = g; A.beta = beta; A.lam = lambda; A.out = out;
    A.state_out = state_out; A.B = B; A.H = H; A.T = T; A.dk = dk; A.dv = dv; A.L = L;
    A.Ls_out = state_out ? Ls_out : 0; A.in_dt = in_dt; A.workspace = workspace; A.stream = stream;
    return lla::gdn_fwd(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

lla_status lla_gdn_decode_step(float *state, const void *q, const void *k, const void *v, const float *g,
                               const float *beta, const float *lambda, float *out, const int64_t *pos,
                               int B, int H, int dk, int dv, int Ls, lla_dtype in_dt,
                               int32_t *device_error, void *stream)
{
    if (B < 0 || H < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (in_dt != LLA_F32 && in_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if (!is_dim(dk) || !is_dim(dv) || Ls < 1 || Ls > 40) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (B > 65535 || H > 65535) return LLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H == 0) return LLA_OK;
    if (!state || !q || !k || !v || !g || !beta || !lambda || !out || !pos)
        return LLA_ERR_INVALID_ARGUMENT;
    lla::GdnDecodeArgs A;
    A.S = state; A.q = q; A.k = k; A.v = v; A.g = g; A.beta = beta; A.lam = lambda; A.out = out;
    A.pos = pos; A.B = B; A.H = H; A.dk = dk; A.dv = dv; A.Ls = Ls; A.in_dt = in_dt;
    A.err = device_error; A.stream = stream;
    return lla::gdn_decode_step(A) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

}  // extern "C"
