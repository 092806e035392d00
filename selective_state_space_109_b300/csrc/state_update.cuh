// state_update.cuh -- single-token decode step of the selective SSM.
//
// Per (sequence b, channel d): read the fp32 state h[b,d,:], advance it by one
// token, h = exp(Delta A) h + Delta B u, write it back in place, and emit
// y = (C.h + D u) silu(z).  Inference runs this recurrence one token at a
// time with a state whose size does not depend on the context length
// (cuishuaiwen.com "Mamba & State-Space Sequence Models", Core mechanics;
// intvml.com "DL0170 Mamba Selective SSM vs Attention", point (5)).
//
// The step is bound by HBM traffic on the state (read + write once).  Four
// lanes share one (b,d) with four states each (one 16-byte state packet per
// lane, so a warp moves 512 contiguous bytes); a thread walks BPT sequences
// of the batch so that its A row is loaded once and reused.
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
    constexpr int SPL = 4;          // states per lane
    constexpr int QL = N / SPL;     // lanes per (b, d)
    static_assert(N % SPL == 0 && (QL == 1 || QL == 2 || QL == 4 || QL == 8 || QL == 16 || QL == 32),
                  "N in {4, ..., 128}");

    const int gx = blockIdx.x * blockDim.x + threadIdx.x;
    const int d = gx / QL;
    const int q = gx % QL;
    // Lanes past the last channel still take part in the shuffles below.
    const bool active = d < p.dim;
    const int dc = active ? d : p.dim - 1;
    const int g = dc / p.dim_per_group;

    const float4 av = __ldg(reinterpret_cast<const float4*>(p.A + static_cast<long long>(dc) * N) + q);
    constexpr float sc = decay_scale<ACCURATE>();
    const float4 a2 = make_float4(av.x * sc, av.y * sc, av.z * sc, av.w * sc);
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
        float4* sp = reinterpret_cast<float4*>(p.state + (static_cast<long long>(slot) * p.dim + dc) * N) + q;
        const float4 s = active ? *sp : make_float4(0.f, 0.f, 0.f, 0.f);
        const float uv = Elem<T>::load(up + bd);
        const float dt = softplus<ACCURATE>(Elem<T>::load(dp + bd) + bias);
        const float du = dt * uv;
        const long long bc = (static_cast<long long>(b) * p.ngroups + g) * N + q * SPL;
        float bv[4], cv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            bv[k] = Elem<T>::load(Bp + bc + k);
            cv[k] = Elem<T>::load(Cp + bc + k);
        }
        float4 hn;
        hn.x = fmaf(decay<ACCURATE>(dt * a2.x), s.x, du * bv[0]);
        hn.y = fmaf(decay<ACCURATE>(dt * a2.y), s.y, du * bv[1]);
        hn.z = fmaf(decay<ACCURATE>(dt * a2.z), s.z, du * bv[2]);
        hn.w = fmaf(decay<ACCURATE>(dt * a2.w), s.w, du * bv[3]);
        if (active) *sp = hn;
        float acc = cv[0] * hn.x + cv[1] * hn.y + cv[2] * hn.z + cv[3] * hn.w;
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
