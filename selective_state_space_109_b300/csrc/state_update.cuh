// state_update.cuh -- single-token decode step of the selective SSM.
//
// Per (sequence b, channel d): read the fp32 state h[b,d,:], advance it by one
// token, h = exp(Delta A) h + Delta B u, write it back in place, and emit
// y = (C.h + D u) silu(z).  Inference runs this recurrence one token at a
// time with a state whose size does not depend on the context length
// (cuishuaiwen.com "Mamba & State-Space Sequence Models", Core mechanics;
// intvml.com "DL0170 Mamba Selective SSM vs Attention", point (5)).
//
// The step is bound by HBM traffic on the state (read + write once).  N/4
// lanes share one (b,d) with four states each (one 16-byte state packet per
// lane, so a warp moves 512 contiguous bytes; at N = 256, 32 lanes of eight
// states); a thread walks BPT sequences of the batch so that its A row is
// loaded once and reused.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

struct DecodeParams {
    float* state;
    const void* u;
    const void* delta;
    const void* z;        // nullable
    const float* A;
    const void* B;
    const void* C;
    const float* D;       // nullable
    const float* dt_bias; // nullable
    void* y;
    const int* slots;     // nullable: row b uses state slot slots[b] (outside [0, nslots): padding)
    int nslots;
    int batch, dim, ngroups, dim_per_group;
};

template <typename T, int N, int BPT, bool ACCURATE>
__global__ void __launch_bounds__(128)
state_update_kernel(const DecodeParams p) {
    constexpr int SPL = N > 128 ? 8 : 4;  // states per lane (whole 16-byte packets)
    constexpr int NV4 = SPL / 4;          // float4 packets per lane
    constexpr int QL = N / SPL;           // lanes per (b, d)
    static_assert(N % SPL == 0 && (QL == 1 || QL == 2 || QL == 4 || QL == 8 || QL == 16 || QL == 32),
                  "N in {4, ..., 256}");

    const int gx = blockIdx.x * blockDim.x + threadIdx.x;
    const int d = gx / QL;
    const int q = gx % QL;
    // Lanes past the last channel still take part in the shuffles below.
    const bool active = d < p.dim;
    const int dc = active ? d : p.dim - 1;
    const int g = dc / p.dim_per_group;

    constexpr float sc = decay_scale<ACCURATE>();
    float a2[SPL];
#pragma unroll
    for (int v = 0; v < NV4; ++v) {
        const float4 av = __ldg(reinterpret_cast<const float4*>(p.A + static_cast<long long>(dc) * N) + q * NV4 + v);
        a2[4 * v] = av.x * sc; a2[4 * v + 1] = av.y * sc; a2[4 * v + 2] = av.z * sc; a2[4 * v + 3] = av.w * sc;
    }
    const float bias = p.dt_bias ? __ldg(p.dt_bias + dc) : 0.f;
    const float dsk = p.D ? __ldg(p.D + dc) : 0.f;

    const T* __restrict__ up = static_cast<const T*>(p.u);
    const T* __restrict__ dp = static_cast<const T*>(p.delta);
    const T* __restrict__ zp = static_cast<const T*>(p.z);
    const T* __restrict__ Bp = static_cast<const T*>(p.B);
    const T* __restrict__ Cp = static_cast<const T*>(p.C);
    T* __restrict__ yp = static_cast<T*>(p.y);

#pragma unroll 1
    for (int i = 0; i < BPT; ++i) {
        const int b = blockIdx.y * BPT + i;
        if (b >= p.batch) break;  // uniform over the CTA
        const int slot = p.slots ? __ldg(p.slots + b) : b;
        if (slot < 0 || slot >= p.nslots) continue;  // a padding row (uniform over the CTA)
        const long long bd = static_cast<long long>(b) * p.dim + dc;
        float4* sp = reinterpret_cast<float4*>(p.state + (static_cast<long long>(slot) * p.dim + dc) * N) + q * NV4;
        float s[SPL];
#pragma unroll
        for (int v = 0; v < NV4; ++v) {
            const float4 sv = active ? sp[v] : make_float4(0.f, 0.f, 0.f, 0.f);
            s[4 * v] = sv.x; s[4 * v + 1] = sv.y; s[4 * v + 2] = sv.z; s[4 * v + 3] = sv.w;
        }
        const float uv = Elem<T>::load(up + bd);
        const float dt = softplus<ACCURATE>(Elem<T>::load(dp + bd) + bias);
        const float du = dt * uv;
        const long long bc = (static_cast<long long>(b) * p.ngroups + g) * N + q * SPL;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            s[k] = fmaf(decay<ACCURATE>(dt * a2[k]), s[k], du * Elem<T>::load(Bp + bc + k));
            acc = fmaf(Elem<T>::load(Cp + bc + k), s[k], acc);
        }
        if (active) {
#pragma unroll
            for (int v = 0; v < NV4; ++v) sp[v] = make_float4(s[4 * v], s[4 * v + 1], s[4 * v + 2], s[4 * v + 3]);
        }
#pragma unroll
        for (int m = QL / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (active && q == 0) {
            float yv = acc + dsk * uv;
            if (zp) yv *= silu<ACCURATE>(Elem<T>::load(zp + bd));
            Elem<T>::store(yp + bd, yv);
        }
    }
}

}  // namespace ssm
