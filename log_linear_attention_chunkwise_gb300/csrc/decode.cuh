// Internal interface of the decode step and the prefill state builder.
#pragma once

#include <stddef.h>

#include "lla_common.cuh"

namespace lla {

struct DecodeArgs {
    float *S, *D;
    const void *q, *k, *v;
    const float *g, *lam;
    float *out;
    const int64_t *pos;
    int B, H, dk, dv, Ls;
    lla_dtype in_dt;
    int32_t *err;
    void *stream;
};

struct PrefillArgs {
    const void *k, *v;
    const float *g;
    float *S, *D;
    int B, H, T, dk, dv, Ls;
    lla_dtype in_dt;
    void *workspace;
    int32_t *device_error;  // caller's word, or nullptr (a workspace word is used)
    void *stream;
};

cudaError_t decode_step(const DecodeArgs &A);
size_t prefill_workspace_bytes(int B, int H, int T);
cudaError_t prefill_state(const PrefillArgs &A);
// Tensor-core bucket states (bf16, dk = dv = 128): after the tail kernel and
// the zeroing of the state; err is a zeroed device word.
bool prefill_tc_supported(const PrefillArgs &A);
cudaError_t prefill_tc(const PrefillArgs &A, const float *tail, int *err);

}  // namespace lla
