// ssm_scan.cu -- host side of libssmscan.so: the C ABI of include/ssm_scan.h.
//
// Each entry point validates its arguments without touching the GPU, picks a
// kernel variant for the shape (lanes per channel, chunking), and enqueues the
// launch on the caller's stream.  Nothing here computes on the host.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/ssm_scan.h"
#include "scan_fwd.cuh"
#include "state_update.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

ssm_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return SSM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dstate(int n) { return n == 4 || n == 8 || n == 16; }

int env_int(const char* name, int fallback) {
    const char* s = std::getenv(name);
    if (!s || !*s) return fallback;
    return std::atoi(s);
}

// Argument checks shared by the scan entry points (no CUDA calls).
ssm_status_t check_scan_args(const void* u, const void* delta, const void* z, const float* A,
                             const void* B, const void* C, const float* Dskip,
                             const float* dt_bias, const void* y, const float* h0,
                             const float* h_final, int batch, int dim, int dstate, int seqlen,
                             int ngroups, ssm_dtype_t io) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0) return SSM_ERR_INVALID_ARG;
    if (dim % ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!A) return SSM_ERR_INVALID_ARG;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    // (batch * dim * seqlen) must index within 63 bits; rows are addressed in 64-bit.
    return SSM_OK;
}

// Lanes that split one channel's N states.  Enough lanes to give every SM
// about eight warps, no more (more lanes mean more reduce-scatter work).
int choose_lanes(int channels, int dstate, int num_sms) {
    const int max_lanes = dstate / 2;  // each lane keeps at least one fp32x2 pair
    const long long want = static_cast<long long>(num_sms) * 8 * 32;
    int lanes = 1;
    while (lanes < max_lanes && static_cast<long long>(channels) * lanes < want) lanes *= 2;
    return lanes;
}

int device_sm_count() {
    static thread_local int cached_dev = -1;
    static thread_local int cached_sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cached_sms;
    if (dev != cached_dev) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            cached_sms = sms;
        cached_dev = dev;
    }
    return cached_sms;
}

constexpr int kScanWarps = 4;
constexpr int kScanTile = 64;

template <typename T, int N, int LANES>
cudaError_t launch_scan_variant(ssm::ScanParams p, cudaStream_t st) {
    constexpr int CH = kScanWarps * (32 / LANES);
    constexpr int V = ssm::ScanShape<T, LANES>::V;
    constexpr int VE = ssm::Elem<T>::kPer16B;
    p.blocks_per_group = (p.dim_per_group + CH - 1) / CH;
    p.vec_ok = (p.seqlen % V) == 0;
    p.bc_vec_ok = (p.seqlen % VE) == 0;
    const long long blocks = static_cast<long long>(p.blocks_per_group) * p.ngroups * p.batch;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    constexpr bool kAccurate = sizeof(T) == 4;
    ssm::scan_fwd_kernel<T, N, LANES, kScanWarps, kScanTile, kAccurate>
        <<<static_cast<unsigned>(blocks), kScanWarps * 32, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_scan_n(const ssm::ScanParams& p, int lanes, cudaStream_t st) {
    switch (lanes) {
        case 1: return launch_scan_variant<T, N, 1>(p, st);
        case 2: return launch_scan_variant<T, N, 2>(p, st);
        case 4: if constexpr (N >= 8) return launch_scan_variant<T, N, 4>(p, st); break;
        case 8: if constexpr (N >= 16) return launch_scan_variant<T, N, 8>(p, st); break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_scan_t(const ssm::ScanParams& p, int dstate, int lanes, cudaStream_t st) {
    switch (dstate) {
        case 4: return launch_scan_n<T, 4>(p, lanes, st);
        case 8: return launch_scan_n<T, 8>(p, lanes, st);
        case 16: return launch_scan_n<T, 16>(p, lanes, st);
        default: return cudaErrorInvalidValue;
    }
}

// Writes h_final = h0 (or zeros) for an empty sequence.
__global__ void copy_or_zero_state_kernel(const float* __restrict__ h0, float* __restrict__ hf, long long n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i < n) hf[i] = h0 ? h0[i] : 0.f;
}

ssm_status_t run_scan(const void* u, const void* delta, const void* z, const float* A,
                      const void* B, const void* C, const float* Dskip, const float* dt_bias,
                      const float* h0, void* y, float* h_final, int batch, int dim, int dstate,
                      int seqlen, int ngroups, ssm_dtype_t io, cudaStream_t st) {
    if (batch == 0) return SSM_OK;
    if (seqlen == 0) {
        if (h_final) {
            const long long n = static_cast<long long>(batch) * dim * dstate;
            copy_or_zero_state_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(h0, h_final, n);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return SSM_OK;
    }
    ssm::ScanParams p{};
    p.u = u; p.delta = delta; p.z = z; p.A = A; p.B = B; p.C = C; p.D = Dskip;
    p.dt_bias = dt_bias; p.y = y; p.h0 = h0; p.h_final = h_final;
    p.batch = batch; p.dim = dim; p.seqlen = seqlen; p.ngroups = ngroups;
    p.dim_per_group = dim / ngroups;
    int lanes = choose_lanes(batch * dim, dstate, device_sm_count());
    const int forced = env_int("SSM_FORCE_LANES", 0);
    if (forced == 1 || forced == 2 || forced == 4 || forced == 8) lanes = forced;
    if (lanes > dstate / 2) lanes = dstate / 2;
    const cudaError_t e = (io == SSM_F32) ? launch_scan_t<float>(p, dstate, lanes, st)
                                          : launch_scan_t<__nv_bfloat16>(p, dstate, lanes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

// Workspace header: a device-side status word written by kernels that wait.
constexpr size_t kWorkspaceHeader = 256;

}  // namespace

extern "C" {

int ssm_abi_version(void) { return SSM_ABI_VERSION; }

const char* ssm_status_string(ssm_status_t s) {
    switch (s) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
        case SSM_ERR_MISALIGNED: return "SSM_ERR_MISALIGNED";
        case SSM_ERR_WORKSPACE_TOO_SMALL: return "SSM_ERR_WORKSPACE_TOO_SMALL";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    }
    return "SSM_ERR_UNKNOWN";
}

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const void* z, const float* A,
                          const void* B, const void* C, const float* Dskip, const float* dt_bias,
                          void* y, int batch, int dim, int dstate, int seqlen, int ngroups,
                          ssm_dtype_t io, void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, nullptr, nullptr,
                                           batch, dim, dstate, seqlen, ngroups, io);
    if (s != SSM_OK) return s;
    return run_scan(u, delta, z, A, B, C, Dskip, dt_bias, nullptr, y, nullptr, batch, dim, dstate,
                    seqlen, ngroups, io, static_cast<cudaStream_t>(stream));
}

size_t ssm_scan_fwd_chunked_workspace_size(int batch, int dim, int dstate, int seqlen, int ngroups,
                                           ssm_dtype_t io) {
    if (batch < 0 || dim <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups != 0) return 0;
    if (!supported_dstate(dstate) || (io != SSM_F32 && io != SSM_BF16)) return 0;
    return kWorkspaceHeader;
}

ssm_status_t ssm_scan_fwd_chunked(const void* u, const void* delta, const void* z, const float* A,
                                  const void* B, const void* C, const float* Dskip,
                                  const float* dt_bias, const float* h0, void* y, float* h_final,
                                  int batch, int dim, int dstate, int seqlen, int ngroups,
                                  ssm_dtype_t io, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final,
                                           batch, dim, dstate, seqlen, ngroups, io);
    if (s != SSM_OK) return s;
    if (workspace && !aligned16(workspace)) return SSM_ERR_MISALIGNED;
    const size_t need = ssm_scan_fwd_chunked_workspace_size(batch, dim, dstate, seqlen, ngroups, io);
    if (workspace_bytes < need || (need > 0 && !workspace)) return SSM_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (workspace) {
        const cudaError_t e = cudaMemsetAsync(workspace, 0, kWorkspaceHeader, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return run_scan(u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final, batch, dim, dstate,
                    seqlen, ngroups, io, st);
}

ssm_status_t ssm_workspace_status(const void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kWorkspaceHeader) return SSM_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return SSM_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == 0 ? SSM_OK : SSM_ERR_TIMEOUT;
}

ssm_status_t ssm_state_update(float* state, const void* u, const void* delta, const void* z,
                              const float* A, const void* B, const void* C, const float* Dskip,
                              const float* dt_bias, void* y, int batch, int dim, int dstate,
                              int ngroups, ssm_dtype_t io, void* stream) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || ngroups <= 0 || dim % ngroups != 0)
        return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!state || !u || !delta || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {state, u, delta, z, A, B, C, Dskip, dt_bias, y};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;

    ssm::DecodeParams p{};
    p.state = state; p.u = u; p.delta = delta; p.z = z; p.A = A; p.B = B; p.C = C;
    p.D = Dskip; p.dt_bias = dt_bias; p.y = y;
    p.batch = batch; p.dim = dim; p.ngroups = ngroups; p.dim_per_group = dim / ngroups;
    constexpr int kBPT = 8;
    constexpr int kThreads = 128;
    const long long threads_x = static_cast<long long>(dim) * (dstate / 4);
    dim3 grid(static_cast<unsigned>((threads_x + kThreads - 1) / kThreads),
              static_cast<unsigned>((batch + kBPT - 1) / kBPT));
    if (grid.y > 65535u) return SSM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define SSM_DECODE_LAUNCH(T, N, ACC) ssm::state_update_kernel<T, N, kBPT, ACC><<<grid, kThreads, 0, st>>>(p)
    if (io == SSM_F32) {
        if (dstate == 4) SSM_DECODE_LAUNCH(float, 4, true);
        else if (dstate == 8) SSM_DECODE_LAUNCH(float, 8, true);
        else SSM_DECODE_LAUNCH(float, 16, true);
    } else {
        if (dstate == 4) SSM_DECODE_LAUNCH(__nv_bfloat16, 4, false);
        else if (dstate == 8) SSM_DECODE_LAUNCH(__nv_bfloat16, 8, false);
        else SSM_DECODE_LAUNCH(__nv_bfloat16, 16, false);
    }
#undef SSM_DECODE_LAUNCH
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

}  // extern "C"
