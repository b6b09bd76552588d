// Internal interface of the tensor-core (tcgen05) forward.
#pragma once

#include <stddef.h>

#include "lla_common.cuh"

namespace lla {

struct TcFwdArgs {
    const void *q, *k, *v;
    const float *g, *lam;
    void *out;
    int B, H, T, L;
    int dk;  // = dv, 64 or 128
    lla_dtype out_dt;
    // non-null: lambda is computed in the read-out from the key tile,
    // softplus((k W1) W2 + b), and lam is not read
    const float *W1 = nullptr, *W2 = nullptr, *bmlp = nullptr;
    void *workspace;
    int32_t *device_error;  // caller's word, or nullptr (the workspace word is used)
    void *stream;
};

bool tc_supported(int dk, int dv, lla_dtype in_dt);
// The in-kernel lambda MLP: the tensor-core shapes with 2L <= 32 (T <= 32768).
bool tc_mlp_supported(int dk, int dv, lla_dtype in_dt, int L);
size_t tc_workspace_bytes(int B, int H, int T, int D);
int tc_launches(int T);
cudaError_t tc_fwd(const TcFwdArgs &A);
// Test hook: withhold each tile's first product and shorten the waits.
void tc_set_withhold_first_product(int enable);

}  // namespace lla
