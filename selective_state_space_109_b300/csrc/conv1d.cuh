// conv1d.cuh -- the short causal depthwise convolution (+ silu) in front of the
// scan, and its decode step.
//
// The pages place a short local convolution between the input projection and
// the selective SSM (eightmm.github.io "Mamba", Block Structure;
// aipedia.org "Mamba: State Space Models", What a Mamba Block Contains).  Read
// as: one filter of W taps per channel, causal, a per-channel bias, then silu:
//
//     out[b,d,l] = act(bias[d] + sum_{k<W} w[d,k] * x[b,d,l-(W-1)+k]),
//
// where times before 0 read the caller's history (the W-1 inputs that preceded
// the sequence, oldest first) or zero.
//
// The step reads x once and writes out once, so it is bound by HBM.  One thread
// owns one 16-byte chunk of a row (VPC steps): a warp reads and writes 512
// contiguous bytes per group of 32 chunks.  The W-1 inputs before a chunk are
// the last ones of the chunk held by the lane before it (a shuffle); the first
// lane of a warp's first group reloads them from the previous chunk (an L1/L2
// hit), and the first chunk of a row takes them from the history.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_device.cuh"
#include "tma.cuh"

namespace ssm {

struct ConvParams {
    const void* x;        // [rows, L]
    const float* w;       // [dim, W]
    const float* bias;    // [dim] or null
    const void* x_prev;   // [rows, W-1] or null (history)
    void* out;            // [rows, L]
    void* x_last;         // [rows, W-1] or null (history of the next segment)
    long long rows;       // batch * dim
    int dim, seqlen;
    int silu;             // apply silu
};

template <typename T>
__device__ __forceinline__ float conv_ld(const T* p, long long i) {
    if constexpr (sizeof(T) == 4) return __ldg(reinterpret_cast<const float*>(p) + i);
    else return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p) + i));
}

template <typename T>
__device__ __forceinline__ void conv_st(T* p, long long i, float v) {
    if constexpr (sizeof(T) == 4) reinterpret_cast<float*>(p)[i] = v;
    else reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// silu: the accurate form for fp32 I/O, the MUFU form for bf16 I/O (its error
// is far below bf16's rounding).
//
// Vector path: L * sizeof(T) is a multiple of 16 and x, out are 16-byte aligned.
// A warp takes U groups of 32 consecutive chunks per iteration and issues all
// U loads before it computes, so that every lane has U x 16 bytes in flight.
// Five resident CTAs per SM (48 registers, a few spilled): measured 303.7 us
// against 323.5 us at four (60 registers) on b1 d5120 L65536 bf16, and 65.6
// against 67.9 us on b8 d2048 L4096; six (40 registers) and loading the next
// iteration's packets ahead (84 registers) were slower.
template <typename T, int W, typename Idx>
__global__ void __launch_bounds__(256, 5)
conv1d_vec_kernel(const ConvParams p) {
    // Programmatic dependent launch (when launched with it): let the next
    // kernel begin launching, and wait for the previous kernel's writes
    // before the first global access.
    grid_dep_launch();
    grid_dep_wait();
    constexpr int VPC = 16 / static_cast<int>(sizeof(T));
    constexpr int H = W - 1;  // history length
    constexpr int U = 4;      // 32-chunk groups per warp iteration
    const long long cpr = p.seqlen / VPC;  // chunks per row
    const long long total = p.rows * cpr;
    const int lane = threadIdx.x & 31;
    const T* __restrict__ x = static_cast<const T*>(p.x);
    T* __restrict__ out = static_cast<T*>(p.out);
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long g0 = warp * (U * 32); g0 < total; g0 += nwarps * (U * 32)) {
        float v[U][VPC];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long q = g0 + u * 32 + lane;
            Packet<T, VPC> pk;
            if (q < total) pk.load_cached(x + q * VPC);
            else pk.zero();
            pk.to_float(v[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long q = g0 + u * 32 + lane;
            const bool valid = q < total;
            // Row and chunk within the row in Idx arithmetic (32-bit whenever
            // the chunk count fits: a 64-bit division costs tens of
            // instructions per 16 bytes).
            const Idx row = valid ? static_cast<Idx>(q) / static_cast<Idx>(cpr) : 0;
            const Idx c = valid ? static_cast<Idx>(q) - row * static_cast<Idx>(cpr) : 0;
            // The H inputs before this chunk are the last of the previous
            // chunk: the lane before, or for lane 0 lane 31 of the previous
            // group (group 0: a reload from memory); the first chunk of a row
            // takes them from the history.
            float hist[H > 0 ? H : 1];
#pragma unroll
            for (int k = 0; k < H; ++k) {
                const float up = __shfl_up_sync(0xffffffffu, v[u][VPC - H + k], 1);
                const float wrap = u > 0 ? __shfl_sync(0xffffffffu, v[u > 0 ? u - 1 : 0][VPC - H + k], 31) : 0.f;
                hist[k] = lane == 0 ? wrap : up;
            }
            if (valid && (c == 0 || (lane == 0 && u == 0))) {
                if (c == 0) {
#pragma unroll
                    for (int k = 0; k < H; ++k)
                        hist[k] = p.x_prev ? conv_ld(static_cast<const T*>(p.x_prev), static_cast<long long>(row) * H + k) : 0.f;
                } else {
#pragma unroll
                    for (int k = 0; k < H; ++k) hist[k] = conv_ld(x, q * VPC - H + k);
                }
            }
            if (!valid) continue;
            const int d = static_cast<int>(row % static_cast<Idx>(p.dim));
            float wk[W];
#pragma unroll
            for (int k = 0; k < W; ++k) wk[k] = __ldg(p.w + static_cast<long long>(d) * W + k);
            const float b0 = p.bias ? __ldg(p.bias + d) : 0.f;
            float o[VPC];
#pragma unroll
            for (int t = 0; t < VPC; ++t) {
                float acc = b0;
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    const int s = t - H + k;  // input position relative to the chunk start
                    const float xv = s >= 0 ? v[u][s] : hist[H + s];
                    acc = fmaf(wk[k], xv, acc);
                }
                o[t] = p.silu ? silu<sizeof(T) == 4>(acc) : acc;
            }
            store_row<T, VPC>(out + q * VPC, o, VPC, true);
            if (p.x_last && c == static_cast<Idx>(cpr - 1)) {
                // The row's last H inputs: the chunk holds VPC >= H of them.
#pragma unroll
                for (int k = 0; k < H; ++k)
                    conv_st(static_cast<T*>(p.x_last), static_cast<long long>(row) * H + k, v[u][VPC - H + k]);
            }
        }
    }
}

// Element path (any L): one thread per output element, W loads each.
template <typename T, int W>
__global__ void __launch_bounds__(256)
conv1d_elem_kernel(const ConvParams p) {
    constexpr int H = W - 1;
    const long long total = p.rows * p.seqlen;
    const T* __restrict__ x = static_cast<const T*>(p.x);
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / p.seqlen;
        const long long l = i - row * p.seqlen;
        const int d = static_cast<int>(row % p.dim);
        float acc = p.bias ? __ldg(p.bias + d) : 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const long long t = l - H + k;
            float xv;
            if (t >= 0) xv = conv_ld(x, row * p.seqlen + t);
            else xv = p.x_prev ? conv_ld(static_cast<const T*>(p.x_prev), row * H + (H + t)) : 0.f;
            acc = fmaf(__ldg(p.w + static_cast<long long>(d) * W + k), xv, acc);
        }
        conv_st(static_cast<T*>(p.out), i, p.silu ? silu<sizeof(T) == 4>(acc) : acc);
    }
}

// History of the next segment for rows shorter than what the vector path
// covers: the last H inputs of history + sequence, one thread per row.
template <typename T, int W>
__global__ void __launch_bounds__(256)
conv1d_last_kernel(const ConvParams p) {
    constexpr int H = W - 1;
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const long long t = static_cast<long long>(p.seqlen) - H + k;
        float v;
        if (t >= 0) v = conv_ld(static_cast<const T*>(p.x), row * p.seqlen + t);
        else v = p.x_prev ? conv_ld(static_cast<const T*>(p.x_prev), row * H + (H + t)) : 0.f;
        conv_st(static_cast<T*>(p.x_last), row * H + k, v);
    }
}

// Decode: one token per (b, d).  conv_state [rows, W-1] holds the last W-1
// inputs, oldest first; it drops the oldest and appends x.
template <typename T, int W>
__global__ void __launch_bounds__(256)
conv1d_update_kernel(void* conv_state, const void* xin, const float* w, const float* bias, void* out,
                     long long rows, int dim, int silu_act) {
    constexpr int H = W - 1;
    grid_dep_launch();  // programmatic dependent launch, as in conv1d_vec_kernel
    grid_dep_wait();
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const int d = static_cast<int>(row % dim);
    T* st = static_cast<T*>(conv_state);
    float win[W];
#pragma unroll
    for (int k = 0; k < H; ++k) win[k] = conv_ld(static_cast<const T*>(conv_state), row * H + k);
    win[H] = conv_ld(static_cast<const T*>(xin), row);
    float acc = bias ? __ldg(bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) acc = fmaf(__ldg(w + static_cast<long long>(d) * W + k), win[k], acc);
    conv_st(static_cast<T*>(out), row, silu_act ? silu<sizeof(T) == 4>(acc) : acc);
#pragma unroll
    for (int k = 0; k < H; ++k) conv_st(st, row * H + k, win[k + 1]);
}

}  // namespace ssm
