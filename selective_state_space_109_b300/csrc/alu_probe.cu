// alu_probe.cu -- measures the two arithmetic pipes that bound the scan: the
// MUFU.EX2 rate (one per state update: the decay exp(Delta A)) and the fp32
// FMA-pipe rate (four operations per state update: Delta*A, (Delta u)*B, the
// recurrence's FMA and the readout's FMA).  Each kernel runs long chains of
// independent operations with every SM fully occupied; the result is the
// rate per SM per nanosecond, which the benchmark turns into the scan's
// arithmetic roofline; a third kernel runs the scan's own per-state
// instruction mix for comparison.  Not part of the scan itself.
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

// The scan's own per-state instruction mix, for comparison with the two pipe
// rates: per state pair and step FMUL2 Delta*A, two MUFU.EX2, FMUL2
// (Delta u)*B, FFMA2 of the recurrence and FFMA2 of the readout, B and C read
// from shared memory as one 16-byte quad per pair; eight pairs per thread,
// eight steps per iteration.
__global__ void __launch_bounds__(kThreads, 1) probe_mix_kernel(float* sink, int iters) {
    __shared__ float4 bc[64 * 8];
    for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x)
        bc[i] = make_float4(0.01f * static_cast<float>(i & 63), 0.02f, 0.03f, 0.04f);
    __syncthreads();
    float2 h[8], a2[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = make_float2(0.f, 0.f);
        a2[k] = make_float2(-1.4f * static_cast<float>(k + 1), -1.4f * (static_cast<float>(k) + 1.5f));
    }
    float dt = 0.01f + 1e-4f * static_cast<float>(threadIdx.x), du = 0.5f, ysum = 0.f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const float2 dt2 = make_float2(dt, dt), du2 = make_float2(du, du);
            float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 q = bc[((it & 7) * 8 + kk) * 8 + k];
                const float2 x = __fmul2_rn(dt2, a2[k]);
                const float2 ab = make_float2(ex2_op(x.x), ex2_op(x.y));
                h[k] = __ffma2_rn(ab, h[k], __fmul2_rn(du2, make_float2(q.x, q.y)));
                y2 = __ffma2_rn(make_float2(q.z, q.w), h[k], y2);
            }
            ysum += y2.x + y2.y;
            dt += 1e-7f;
            du -= 1e-7f;
        }
    }
    if (ysum == -1.f) sink[0] = ysum;
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
                                            double* mix_updates_per_sm_ns, void* stream) {
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
    if (mix_updates_per_sm_ns) {
        const int mix_iters = 512;
        const double upd = static_cast<double>(sms) * kThreads * mix_iters * 8 * 16;  // steps x states
        if (time_kernel(probe_mix_kernel, sms, sink, mix_iters, reps, st, &ms) != cudaSuccess) return SSM_ERR_CUDA;
        *mix_updates_per_sm_ns = upd / sms / (static_cast<double>(ms) * 1e6);
    }
    return SSM_OK;
}
