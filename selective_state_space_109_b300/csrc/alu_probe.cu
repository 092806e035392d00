// alu_probe.cu -- measures the two arithmetic pipes that bound the scan: the
// MUFU.EX2 rate (one per state update: the decay exp(Delta A)) and the fp32
// FMA-pipe rate (four operations per state update: Delta*A, (Delta u)*B, the
// recurrence's FMA and the readout's FMA).  Each kernel runs long chains of
// independent operations with every SM fully occupied; the result is the
// rate per SM per nanosecond, which the benchmark turns into the scan's
// arithmetic roofline.  Not part of the scan itself.
#include <cuda_runtime.h>

#include "../../include/ssm_scan.h"

namespace {

constexpr int kChains = 8;
constexpr int kThreads = 1024;  // 32 warps per SM: 8 per scheduler

__device__ __forceinline__ float ex2_op(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x <- 2^-x keeps every chain in (0, 1]; the negation is an operand modifier.
__global__ void __launch_bounds__(kThreads, 1) probe_ex2_kernel(float* sink, int iters) {
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) v[i] = 1e-3f * static_cast<float>(threadIdx.x + i);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = ex2_op(-v[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += v[i];
    if (s == -1.f) sink[0] = s;  // never true: keeps the chains live
}

__global__ void __launch_bounds__(kThreads, 1) probe_ffma_kernel(float* sink, int iters) {
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) v[i] = 1e-3f * static_cast<float>(threadIdx.x + i);
    const float a = 0.999f, b = 1e-4f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = fmaf(v[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += v[i];
    if (s == -1.f) sink[0] = s;
}

// Mean device time (ms) of `reps` launches after one warm-up launch.
template <typename K>
cudaError_t time_kernel(K kern, int blocks, float* sink, int iters, int reps, cudaStream_t st, float* ms) {
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) {
        kern<<<blocks, kThreads, 0, st>>>(sink, iters);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e0, st);
    for (int r = 0; r < reps && e == cudaSuccess; ++r) {
        kern<<<blocks, kThreads, 0, st>>>(sink, iters);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (e == cudaSuccess) *ms /= static_cast<float>(reps);
    return e;
}

}  // namespace

extern "C" ssm_status_t ssm_probe_alu_rates(float* sink, double* ex2_per_sm_ns, double* ffma_per_sm_ns,
                                            void* stream) {
    if (!sink || !ex2_per_sm_ns || !ffma_per_sm_ns) return SSM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SSM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int iters = 8192, reps = 5;
    const double ops = static_cast<double>(sms) * kThreads * iters * kChains;  // per launch
    float ms = 0.f;
    if (time_kernel(probe_ex2_kernel, sms, sink, iters, reps, st, &ms) != cudaSuccess) return SSM_ERR_CUDA;
    *ex2_per_sm_ns = ops / sms / (static_cast<double>(ms) * 1e6);
    if (time_kernel(probe_ffma_kernel, sms, sink, iters, reps, st, &ms) != cudaSuccess) return SSM_ERR_CUDA;
    *ffma_per_sm_ns = ops / sms / (static_cast<double>(ms) * 1e6);
    return SSM_OK;
}
