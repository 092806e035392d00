// ssm_device.cuh -- device-side helpers shared by the scan and decode kernels:
// MUFU wrappers, the softplus / silu forms used by each I/O type, and 8/16-byte
// vector loads and stores of fp32 or bf16 rows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// MUFU.EX2 / RCP (approximate, denormals flushed).  Not volatile, so the
// compiler may schedule them freely.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// The same MUFU.EX2, never merged with an identical earlier one: where a
// value is deliberately recomputed instead of kept in a register.
__device__ __forceinline__ float ex2_approx_again(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// MUFU.TANH (approximate: relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// e^x to about 1 ulp on the FMA pipe (used where the I/O type is fp32):
// Cody & Waite's argument reduction x = k ln2 + r with |r| <= ln2/2 (ln2 split
// into a short head and a tail so that k * head is exact), e^r from its
// degree-7 Taylor polynomial (truncation < 6e-9 relative), and the factor 2^k
// added into the exponent bits.  x is clamped to [-86, 88] so the result stays
// a normal float (e^-86 ~ 4e-38 stands in for a decay that has underflowed).
__device__ __forceinline__ float exp_cody_waite(float x) {
    x = fminf(fmaxf(x, -86.0f), 88.0f);
    const float t = fmaf(x, kLog2e, 12582912.0f);  // 1.5 * 2^23: rounds x log2(e) to an integer
    const float k = t - 12582912.0f;
    float r = fmaf(k, -0.693145751953125f, x);      // ln2 head: 15 significant bits, so k * head is exact for |k| < 2^9
    r = fmaf(k, -1.4286068203094172e-6f, r);        // ln2 tail
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const int ki = __float_as_int(t) - 0x4B400000;  // k as an integer
    return __int_as_float(__float_as_int(p) + (ki << 23));
}

// Per-state decay factor Abar = exp(x) where x = Delta * a and a is the
// prepared per-state constant: a = A (ACCURATE, base e) or A * log2(e)
// (fast, MUFU.EX2 in base 2).
template <bool ACCURATE>
__host__ __device__ constexpr float decay_scale() { return ACCURATE ? 1.0f : kLog2e; }

template <bool ACCURATE>
__device__ __forceinline__ float decay(float x) {
    return ACCURATE ? exp_cody_waite(x) : ex2_approx(x);
}

// decay() evaluated again for a value computed earlier, without keeping the
// earlier result live (fp32 I/O: the FMA-pipe exp may still be merged).
template <bool ACCURATE>
__device__ __forceinline__ float decay_again(float x) {
    return ACCURATE ? exp_cody_waite(x) : ex2_approx_again(x);
}

// log1p(w) / w on [0, 1]: a degree-8 polynomial, the interpolant of that
// function at the nine Chebyshev nodes of the interval (computed in fp64 and
// rounded to fp32), evaluated by Horner's rule; its relative error in fp32 is
// below 2e-7 over [0, 1] (the function is analytic there, its nearest
// singularity at w = -1).  Scalar and fp32x2 forms, the same operations.
__device__ __forceinline__ float log1p_over_w(float w) {
    float q = fmaf(w, 0.005126102f, -0.029074065f);
    q = fmaf(w, q, 0.07751609f);
    q = fmaf(w, q, -0.13602248f);
    q = fmaf(w, q, 0.19076881f);
    q = fmaf(w, q, -0.24835399f);
    q = fmaf(w, q, 0.3331812f);
    q = fmaf(w, q, -0.49999446f);
    return fmaf(w, q, 0.99999994f);
}
__device__ __forceinline__ float2 log1p_over_w2(float2 w) {
    float2 q = __ffma2_rn(w, make_float2(0.005126102f, 0.005126102f), make_float2(-0.029074065f, -0.029074065f));
    q = __ffma2_rn(w, q, make_float2(0.07751609f, 0.07751609f));
    q = __ffma2_rn(w, q, make_float2(-0.13602248f, -0.13602248f));
    q = __ffma2_rn(w, q, make_float2(0.19076881f, 0.19076881f));
    q = __ffma2_rn(w, q, make_float2(-0.24835399f, -0.24835399f));
    q = __ffma2_rn(w, q, make_float2(0.3331812f, 0.3331812f));
    q = __ffma2_rn(w, q, make_float2(-0.49999446f, -0.49999446f));
    return __ffma2_rn(w, q, make_float2(0.99999994f, 0.99999994f));
}

// softplus(v) = max(v, 0) + log1p(exp(-|v|)).
// ACCURATE (fp32 I/O): the CUDA math library's expf / log1pf.
// fast (bf16 I/O): w = exp(-|v|) from MUFU.EX2, log1p(w) = w * log1p_over_w(w)
// (relative error below 2e-7 for every w in [0, 1]; one MUFU operation).
template <bool ACCURATE>
__device__ __forceinline__ float softplus(float v) {
    if (ACCURATE) {
        return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
    } else {
        const float w = ex2_approx(-fabsf(v) * kLog2e);
        return fmaf(w, log1p_over_w(w), fmaxf(v, 0.f));
    }
}

// silu(z) = z / (1 + exp(-z)).
template <bool ACCURATE>
__device__ __forceinline__ float silu(float z) {
    if (ACCURATE) {
        return z / (1.f + expf(-z));
    } else {
        return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
    }
}

// silu through the identity z sigmoid(z) = h + h tanh(h), h = z / 2: one
// MUFU operation instead of an exponential and a reciprocal.  Its relative
// error (about 2^-11) is below the bf16 rounding of the outputs it gates; the
// scan's fused passes and the SSD output use it for bf16 I/O, whose outputs
// are held to the bf16 rel-L2 tolerance.
__device__ __forceinline__ float silu_tanh(float z) {
    const float h = 0.5f * z;
    return fmaf(h, tanh_approx(h), h);
}

// Two-lane (fp32x2) forms of the fast softplus and of silu_tanh above, for
// two steps at once: the same operations element by element, issued as packed
// FMA-pipe instructions where the operation has a packed form.
__device__ __forceinline__ float2 softplus2_fast(float2 v) {
    const float w0 = ex2_approx(fabsf(v.x) * -kLog2e);
    const float w1 = ex2_approx(fabsf(v.y) * -kLog2e);
    const float2 w = make_float2(w0, w1);
    // max(v, 0) + w * (log1p(w) / w): no second MUFU operation, no branch
    return __ffma2_rn(w, log1p_over_w2(w), make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f)));
}

__device__ __forceinline__ float2 silu2_fast(float2 z) {
    const float2 h = __fmul2_rn(z, make_float2(0.5f, 0.5f));
    return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kPer16B = 4;
    __device__ static __forceinline__ float load(const float* p) { return __ldg(p); }
    __device__ static __forceinline__ float load_stream(const float* p) { return __ldcs(p); }
    __device__ static __forceinline__ void store(float* p, float v) { __stcs(p, v); }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPer16B = 8;
    __device__ static __forceinline__ float load(const __nv_bfloat16* p) {
        const unsigned short r = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(r) << 16);
    }
    __device__ static __forceinline__ float load_stream(const __nv_bfloat16* p) {
        const unsigned short r = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(r) << 16);
    }
    __device__ static __forceinline__ void store(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

// V consecutive elements of type T held as raw 32-bit words (8 or 16 bytes).
template <typename T, int V>
struct Packet {
    static constexpr int kWords = V * static_cast<int>(sizeof(T)) / 4;
    static_assert(kWords == 2 || kWords == 4, "packets are 8 or 16 bytes");
    uint32_t w[kWords];

    // Streaming (evict-first) load of V aligned elements.
    __device__ __forceinline__ void load_stream(const T* p) {
        if constexpr (kWords == 4) {
            const uint4 r = __ldcs(reinterpret_cast<const uint4*>(p));
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else {
            const uint2 r = __ldcs(reinterpret_cast<const uint2*>(p));
            w[0] = r.x; w[1] = r.y;
        }
    }
    // Cached load (data re-read by other CTAs).
    __device__ __forceinline__ void load_cached(const T* p) {
        if constexpr (kWords == 4) {
            const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else {
            const uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
            w[0] = r.x; w[1] = r.y;
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < kWords; ++i) w[i] = 0u;
    }
    // Element-wise load of the first `valid` elements (rest zero), any alignment.
    __device__ __forceinline__ void load_partial(const T* p, int valid) {
        float f[V];
#pragma unroll
        for (int k = 0; k < V; ++k) f[k] = (k < valid) ? Elem<T>::load_stream(p + k) : 0.f;
        from_float(f);
    }
    __device__ __forceinline__ void to_float(float (&f)[V]) const {
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int k = 0; k < V; ++k) f[k] = __uint_as_float(w[k]);
        } else {
#pragma unroll
            for (int k = 0; k < kWords; ++k) {
                f[2 * k] = __uint_as_float(w[k] << 16);
                f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
            }
        }
    }
    // Round to T (bf16: nearest even) and pack.
    __device__ __forceinline__ void from_float(const float (&f)[V]) {
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int k = 0; k < V; ++k) w[k] = __float_as_uint(f[k]);
        } else {
#pragma unroll
            for (int k = 0; k < kWords; ++k) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
        }
    }
    __device__ __forceinline__ void store_stream(T* p) const {
        if constexpr (kWords == 4) {
            __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
        } else {
            __stcs(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
        }
    }
};

// Load V elements at p: one vector load when the whole packet is in range and
// aligned, element-wise otherwise (`valid` = elements in range, may be <= 0).
template <typename T, int V>
__device__ __forceinline__ void load_row(Packet<T, V>& pk, const T* p, int valid, bool vec_ok) {
    if (vec_ok && valid >= V) {
        pk.load_stream(p);
    } else if (valid > 0) {
        pk.load_partial(p, valid);
    } else {
        pk.zero();
    }
}

template <typename T, int V>
__device__ __forceinline__ void store_row(T* p, const float (&f)[V], int valid, bool vec_ok) {
    if (vec_ok && valid >= V) {
        Packet<T, V> pk;
        pk.from_float(f);
        pk.store_stream(p);
    } else {
#pragma unroll
        for (int k = 0; k < V; ++k)
            if (k < valid) Elem<T>::store(p + k, f[k]);
    }
}

// Butterfly reduce-scatter over the LANES lanes of a channel: on entry slot
// q*V+v of lane j holds its partial readout of step q*V+v; on exit slots
// [0, V) hold the full sum (over all lanes) of steps j*V + [0, V).
template <int LANES, int V>
__device__ __forceinline__ void reduce_scatter(float (&acc)[LANES * V], int j) {
#pragma unroll
    for (int m = LANES / 2; m >= 1; m >>= 1) {
        const bool upper = (j & m) != 0;
#pragma unroll
        for (int q = 0; q < m; ++q) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float lo = acc[q * V + v];
                const float hi = acc[(q + m) * V + v];
                const float send = upper ? lo : hi;
                const float keep = upper ? hi : lo;
                acc[q * V + v] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
    }
}

}  // namespace ssm
