// Internal interface of Log-Linear Gated DeltaNet (recurrent form).
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

size_t gdn_fwd_smem_bytes(int T, int dk, int L);
cudaError_t gdn_fwd(const GdnFwdArgs &A);
cudaError_t gdn_decode_step(const GdnDecodeArgs &A);

}  // namespace lla
