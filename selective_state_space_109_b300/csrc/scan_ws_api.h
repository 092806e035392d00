// scan_ws_api.h -- host-side interface of the warp-specialised scan kernels
// (scan_ws.cuh), which are compiled in their own translation units, one per
// I/O type (scan_ws_bf16.cu, scan_ws_f32.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace ssm {

struct WsScanParams {
    const float* A;
    const float* D;        // nullable
    const float* dt_bias;  // nullable
    const float* h0;       // nullable
    float* h_final;        // nullable
    void* y;               // [batch, dim, seqlen] in the I/O type
    unsigned int* status;  // nullable caller status word (timeouts)
    int batch, dim, seqlen, ngroups, dim_per_group;
    int blocks_per_group;  // CTAs along the channels of one group
    int ntiles;            // ceil(seqlen / TS)
    int has_z;
    // Failure injection for the tests of the bounded waits: the producer
    // stops issuing loads at this tile (-1: never), and every wait gives up
    // after wait_budget_ns.
    int stop_tile;
    unsigned long long wait_budget_ns;
    // Time chunks (grid y; 1: the whole sequence).  Chunk c > 0 starts from
    // the state carried into it, at carry[((c - 1) * batch * dim + b * dim +
    // d) * 2 * dstate + dstate ...] (the summary layout after the carry pass),
    // read once the previous kernel in the stream has completed.
    const float* carry;
    int nchunks;
};

// TMA descriptors of one call: the [batch * ngroups, dim_per_group, seqlen]
// activation views (box: one tile row times the CTA's channels) and the
// [batch * ngroups * dstate, seqlen] B and C views (box: one tile row times
// dstate rows).
struct WsMaps {
    CUtensorMap u, d, z, B, C;
};

// Dynamic shared memory of one kernel variant, or 0 if that variant is not
// built.  seg = 1: the plain pass; seg > 1: the time-segmented variant (a tile
// row of 16 * seg bytes, one 16-byte chunk per segment).
int ws_smem_bytes_bf16(int dstate, int lanes, int nw, int seg);
int ws_smem_bytes_f32(int dstate, int lanes, int nw, int seg);

// Enqueues the pass (grid: blocks_per_group * ngroups * batch CTAs, times
// nchunks; a chunked pass is launched to overlap the previous kernel's tail).
// cudaErrorInvalidValue if the variant is not built.
cudaError_t ws_launch_bf16(int dstate, int lanes, int nw, int seg, const WsMaps& m, const WsScanParams& p,
                           cudaStream_t st);
cudaError_t ws_launch_f32(int dstate, int lanes, int nw, int seg, const WsMaps& m, const WsScanParams& p,
                          cudaStream_t st);

}  // namespace ssm
