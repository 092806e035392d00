// scan_ws_bf16.cu -- the warp-specialised fused scan pass for bf16 I/O.
#include <cuda_bf16.h>

#include "scan_ws_inst.cuh"

namespace ssm {

int ws_smem_bytes_bf16(int dstate, int lanes, int nw, int seg) {
    return ws_detail::smem_any<__nv_bfloat16>(dstate, lanes, nw, seg);
}

cudaError_t ws_launch_bf16(int dstate, int lanes, int nw, int seg, const WsMaps& m, const WsScanParams& p,
                           cudaStream_t st) {
    return ws_detail::launch_any<__nv_bfloat16>(dstate, lanes, nw, seg, m, p, st);
}

}  // namespace ssm
