// Internal interface of the lambda producer (two-layer MLP + softplus).
#pragma once

#include "lla_common.cuh"

namespace lla {

struct LambdaMlpArgs {
    const void *d;
    const float *W1, *W2, *bias;
    float *lam;
    int B, H, T, Dd, L;
    lla_dtype in_dt;
    int32_t *device_error;  // caller's word, or nullptr (a library word is used)
    void *stream;
};

cudaError_t lambda_mlp(const LambdaMlpArgs &A);

}  // namespace lla
