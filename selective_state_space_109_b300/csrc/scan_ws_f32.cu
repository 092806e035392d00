// scan_ws_f32.cu -- the warp-specialised fused scan pass for fp32 I/O.
#include "scan_ws_inst.cuh"

namespace ssm {

int ws_smem_bytes_f32(int dstate, int lanes, int nw, int seg) {
    return ws_detail::smem_any<float>(dstate, lanes, nw, seg);
}

cudaError_t ws_launch_f32(int dstate, int lanes, int nw, int seg, const WsMaps& m, const WsScanParams& p,
                           cudaStream_t st) {
    return ws_detail::launch_any<float>(dstate, lanes, nw, seg, m, p, st);
}

}  // namespace ssm
