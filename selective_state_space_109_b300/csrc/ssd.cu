// ssd.cu -- host side of the SSD (Mamba-2) layer: argument checks, the TMA
// descriptors and the launch of ssd_fwd_kernel (ssd.cuh); ssm_ssd_fwd of the
// C ABI.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/ssm_scan.h"
#include "ssd.cuh"

// Records a CUDA error for ssm_last_cuda_error (ssm_scan.cu).
ssm_status_t ssm_note_cuda_error(cudaError_t e);

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// [rows, L] bf16 view, box = 64 steps x box_rows rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* ptr, long long rows, int seqlen, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(seqlen), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(seqlen) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [planes, dstate, L] bf16 view of B or C, box = 64 steps x the tile's N rows
// x 1 plane, 128-byte swizzle: rows past dstate are filled with zeros.
bool encode_bc_planes(CUtensorMap* m, const void* ptr, long long planes, int dstate, int seqlen) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(seqlen), static_cast<cuuint64_t>(dstate),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(seqlen) * 2,
                                   static_cast<cuuint64_t>(seqlen) * 2 * static_cast<cuuint64_t>(dstate)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(ssm::ssd::N), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void ssd_copy_state_kernel(const float* h0, float* h_final, long long n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i < n) h_final[i] = h0 ? h0[i] : 0.f;
}

}  // namespace

extern "C" ssm_status_t ssm_ssd_fwd(const void* x, const void* delta, const void* z, const float* A,
                                    const void* B, const void* C, const float* Dskip, const float* dt_bias,
                                    const float* h0, void* y, float* h_final, int batch, int nheads, int headdim,
                                    int dstate, int seqlen, int ngroups, ssm_dtype_t io, void* stream) {
    if (batch < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0)
        return SSM_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (headdim != ssm::ssd::P) return SSM_ERR_UNSUPPORTED;
    if (dstate != 16 && dstate != 32 && dstate != 64 && dstate != ssm::ssd::N) return SSM_ERR_UNSUPPORTED;
    if ((static_cast<long long>(seqlen) * 2) % 16 != 0) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!A) return SSM_ERR_INVALID_ARG;
    if (seqlen > 0 && (!x || !delta || !B || !C || !y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long dim = static_cast<long long>(nheads) * headdim;
    if (seqlen == 0) {
        if (h_final) {
            const long long n = static_cast<long long>(batch) * dim * dstate;
            ssd_copy_state_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(h0, h_final, n);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return ssm_note_cuda_error(e);
        }
        return SSM_OK;
    }
    if (!encode_tiled_fn()) return SSM_ERR_CUDA;
    CUtensorMap mx, mb, mc, mz, my;
    // z's map is encoded on x when there is no z (the kernel then never uses it).
    const bool ok = encode_rows(&mx, x, batch * dim, seqlen, ssm::ssd::P) &&
                    encode_rows(&mz, z ? z : x, batch * dim, seqlen, ssm::ssd::P) &&
                    encode_rows(&my, y, batch * dim, seqlen, ssm::ssd::P) &&
                    encode_bc_planes(&mb, B, static_cast<long long>(batch) * ngroups, dstate, seqlen) &&
                    encode_bc_planes(&mc, C, static_cast<long long>(batch) * ngroups, dstate, seqlen);
    if (!ok) return SSM_ERR_CUDA;
    ssm::SsdParams p{};
    p.delta = static_cast<const __nv_bfloat16*>(delta);
    p.A = A; p.D = Dskip; p.dt_bias = dt_bias; p.h0 = h0; p.h_final = h_final;
    p.y = static_cast<__nv_bfloat16*>(y); p.z = static_cast<const __nv_bfloat16*>(z); p.status = nullptr;
    p.batch = batch; p.nheads = nheads; p.seqlen = seqlen; p.ngroups = ngroups; p.dstate = dstate;
    p.has_z = z != nullptr;

    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(ssm::ssd_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   ssm::ssd::SMEM_BYTES);
        if (e != cudaSuccess) return ssm_note_cuda_error(e);
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = static_cast<long long>(batch) * nheads;
    if (grid > 0x7fffffffLL) return SSM_ERR_INVALID_ARG;
    // Launched with programmatic stream serialization, so that its launch
    // overlaps the tail of the previous kernel in the stream.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(ssm::ssd::THREADS);
    cfg.dynamicSmemBytes = ssm::ssd::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, ssm::ssd_fwd_kernel, mx, mb, mc, mz, my, p);
    return e == cudaSuccess ? SSM_OK : ssm_note_cuda_error(e);
}
