// Internal interface of the CUDA-core forward (fp32 arithmetic).
#pragma once

#include <stddef.h>

#include "lla_common.cuh"

namespace lla {

struct SimtFwdArgs {
    const void *q, *k, *v;
    const float *g, *lam;
    void *out;
    int B, H, T, dk, dv, C, L;
    lla_dtype in_dt, out_dt;
    void *workspace;
    void *stream;
};

size_t simt_ws_offset_P(const SimtFwdArgs &A);
size_t simt_ws_offset_nodes(const SimtFwdArgs &A);
size_t simt_workspace_bytes(const SimtFwdArgs &A);
size_t simt_max_smem_bytes(const SimtFwdArgs &A);
cudaError_t simt_fwd(const SimtFwdArgs &A);
// Chunk states, chunk-gate prefix and Fenwick nodes only (the backward reads
// them): P at simt_ws_offset_P, Node_j at slot j of simt_ws_offset_nodes.
cudaError_t simt_build_nodes(const SimtFwdArgs &A);
// The same with the chunk states and chunk gate totals already in place
// (totals [BH][N] fp32 at the workspace start, H_{j-1} in node slot j):
// only the prefix and the Fenwick scan run.
cudaError_t simt_nodes_from_states(const SimtFwdArgs &A);

}  // namespace lla
