// Internal interface of Log-Linear Gated DeltaNet (chunkwise forward, decode step).
#pragma once

#include <stddef.h>

#include "lla_common.cuh"

namespace lla {

struct GdnFwdArgs {
    const void *q, *k, *v;
    const float *g, *beta, *lam;
    float *out, *state_out;
    int B, H, T, dk, dv, L, Ls_out;
    lla_dtype in_dt;
    void *workspace;  // gdn_fwd_workspace_bytes(...) bytes, 256-byte aligned
    void *stream;
};

struct GdnDecodeArgs {
    float *S;
    const void *q, *k, *v;
    const float *g, *beta, *lam;
    float *out;
    const int64_t *pos;
    int B, H, dk, dv, Ls;
    lla_dtype in_dt;
    int32_t *err;
    void *stream;
};

size_t gdn_fwd_workspace_bytes(int B, int H, int T, int dk, int dv);
// Whether both forward kernels' shared memory fits one CTA at this shape.
bool gdn_fwd_fits(int T, int dk, int dv, int L, int tin_bytes);
cudaError_t gdn_fwd(const GdnFwdArgs &A);
cudaError_t gdn_decode_step(const GdnDecodeArgs &A);

}  // namespace lla
