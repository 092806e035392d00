// scan_bwd.cuh -- backward pass of the selective scan: the gradients of a
// loss with respect to u, delta, z, A, B, C, D, dt_bias and h0, given dy (and
// optionally the gradient with respect to the final state).
//
// The pages keep the states on chip and recompute them in the backward pass
// instead of storing them (intvml.com "DL0170 Mamba Selective SSM vs
// Attention", the paragraphs after the key points).  The gradients are the
// chain rule through the forward definition.  With s_t the ungated output,
// g_t = dy_t silu(z_t) and lam_t[n] = dLoss/dh_t[n]:
//
//   lam_t[n] = g_t C_t[n] + Abar_{t+1}[n] lam_{t+1}[n]
//   dC_t[n] = g_t h_t[n]            dB_t[n] = lam_t[n] Delta_t u_t
//   du_t = g_t D + Delta_t sum_n lam_t[n] B_t[n]
//   dDelta_t = sum_n lam_t[n] (B_t[n] u_t + A[n] Abar_t[n] h_{t-1}[n])
//   ddelta_t = dDelta_t sigmoid(delta_t + dt_bias),  dz_t = dy_t s_t silu'(z_t)
//   dA[n] += lam_t[n] Delta_t Abar_t[n] h_{t-1}[n],  dD += g_t u_t,
//   ddt_bias += ddelta_t,  dh0[n] = Abar_0[n] lam_0[n].
//
// Structure.  Time is cut into chunks of p.chunk_steps steps; a CTA owns
// CH channels of one (sequence, group) and one chunk.  Both recurrences run
// across chunks through summaries, as in the forward pass:
//   1. summary pass: per chunk, from a zero state, the decay product P and
//      end state E; and, from a zero adjoint at the chunk's end, the adjoint
//      M that leaves the chunk at its start (mu = Abar_t lam_t after the
//      chunk's first step), accumulated forwards in the same walk;
//   2. carry pass: h entering chunk c+1 = P_c h + E_c (from h0), and the
//      adjoint entering chunk c-1 from the right = P_c mu + M_c (from dh_final);
//   3. main pass: from the state entering its chunk, a forward sweep stores
//      the state at every tile start in shared memory; then the tiles are
//      walked backwards: each tile's states are recomputed into registers from
//      its checkpoint, and the adjoint runs back over the tile, producing every
//      gradient of the tile's steps.
//
// Lanes: LN = N/S consecutive lanes share a channel, S = 4 states each (8 at
// N = 256).  The per-step sums over states (the readout, du, dDelta) are
// butterfly-reduced over the LN lanes; dB and dC sum over the channels of the group: a
// reduce-scatter over the channels of a warp, a sum over the CTA's warps in
// shared memory, then one atomic add per (state, step) per CTA into fp32
// buffers (vector adds of four steps when the rows keep 16-byte alignment).
// dA, dD and ddt_bias collect in registers and are added atomically once per
// CTA.
#pragma once

#include "ssm_device.cuh"
#include "tma.cuh"

namespace ssm {

constexpr int kBwdTT = 8;       // steps per tile
constexpr int kBwdWarps = 4;
// States per lane of the main pass: 4 (N/4 lanes a channel), 8 at N = 256 so
// that a channel stays within a warp.
__host__ __device__ constexpr int bwd_states_per_lane(int n) { return n > 128 ? 8 : 4; }

// Tiles per time chunk: their start states are held in shared memory (16 KB
// per 8 tiles at 4 states a lane).  The chunk length is chosen per call (see
// bwd_chunk_tiles_for in the host code) up to bwd_chunk_tiles_max tiles: 20,
// or 8 from N = 64 on, whose dB/dC staging is larger.
__host__ __device__ constexpr int bwd_chunk_tiles_max(int n) { return n >= 64 ? 8 : 20; }

struct BwdParams {
    const void *u, *delta, *z, *dy, *B, *C;
    const float *A, *D, *dt_bias, *h0, *dhf;
    void *du, *ddelta, *dz;
    float *dA, *dB, *dC, *dD, *ddt_bias, *dh0;
    float* fagg;  // [nchunks][batch*dim][2][N]: P, then E (replaced by the state entering chunk c+1)
    float* bagg;  // [nchunks][batch*dim][N]: M (replaced by the adjoint entering chunk c-1 from the right)
    int batch, dim, seqlen, ngroups, dim_per_group, blocks_per_group, nchunks;
    int chunk_steps;  // steps per time chunk: a multiple of kBwdTT, at most kBwdTT * bwd_chunk_tiles_max(N)
    int vec_ok;   // every row may be read and written as aligned 16-byte packets
};

template <bool ACCURATE>
__device__ __forceinline__ float sigmoid_f(float v) {
    if (ACCURATE) {
        const float w = expf(-fabsf(v));
        const float r = 1.f / (1.f + w);
        return v >= 0.f ? r : w * r;
    } else {
        const float w = ex2_approx(-fabsf(v) * kLog2e);
        const float r = rcp_approx(1.f + w);
        return v >= 0.f ? r : w * r;
    }
}

// Asynchronous 16-byte global -> shared copies (L1 bypassed).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory"); }

template <typename T>
__device__ __forceinline__ float bwd_to_f(T v) {
    if constexpr (sizeof(T) == 4) return v;
    else return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T bwd_zero() {
    if constexpr (sizeof(T) == 4) return 0.f;
    else return __float2bfloat16_rn(0.f);
}

// Stages kBwdTT elements of a row (from src, `valid` of them in range) into
// shared memory: cp.async when the whole segment is in range and aligned,
// element copies (zero past the end) otherwise.
template <typename T>
__device__ __forceinline__ void bwd_stage_row(T* dst, const T* src, int valid, bool vec) {
    constexpr int VP = 16 / static_cast<int>(sizeof(T));
    if (vec && valid >= kBwdTT) {
#pragma unroll
        for (int q = 0; q < kBwdTT / VP; ++q) cp_async16(dst + q * VP, src + q * VP);
    } else {
#pragma unroll
        for (int k = 0; k < kBwdTT; ++k) dst[k] = k < valid ? src[k] : bwd_zero<T>();
    }
}

// softplus(v) and sigmoid(v) from one exp(-|v|).
template <bool ACCURATE>
__device__ __forceinline__ void softplus_sigmoid(float v, float& sp, float& sg) {
    if (ACCURATE) {
        const float w = expf(-fabsf(v));
        sp = fmaxf(v, 0.f) + log1pf(w);
        const float r = 1.f / (1.f + w);
        sg = v >= 0.f ? r : w * r;
    } else {
        sp = softplus<false>(v);
        sg = sigmoid_f<false>(v);
    }
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

template <bool ACCURATE>
__device__ __forceinline__ float2 decay2(float2 x) {
    return make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
}

// Tensors of the activation rows staged per tile, in this order.
enum BwdAct { kU = 0, kDelta = 1, kZ = 2, kDy = 3 };

// Butterfly all-reduce over the LN lanes of a channel.
template <int LN>
__device__ __forceinline__ float lane_sum(float v) {
#pragma unroll
    for (int m = LN / 2; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// Sum over the channels of a warp (lane bits M..LN): a reduce-scatter while
// more than one value is left, then plain sums.  On exit a lane holds the
// values id0 + [0, CNT_left) of its list (see xchan_first_id).
template <int M, int LN, int CNT>
__device__ __forceinline__ void xchan_reduce(float* v, int lane) {
    if constexpr (M >= LN) {
        if constexpr (CNT > 1) {
            constexpr int H = CNT / 2;
            const bool upper = (lane & M) != 0;
#pragma unroll
            for (int q = 0; q < H; ++q) {
                const float send = upper ? v[q] : v[q + H];
                const float keep = upper ? v[q + H] : v[q];
                v[q] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            xchan_reduce<M / 2, LN, H>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
            xchan_reduce<M / 2, LN, 1>(v, lane);
        }
    }
}

// First list index held by `lane` after xchan_reduce<16, LN, CNT>, the count
// held, and whether the lane is the one copy that should write them.
template <int LN, int CNT>
__device__ __forceinline__ int xchan_first_id(int lane, bool& writer) {
    int id0 = 0, cnt = CNT;
    writer = true;
#pragma unroll
    for (int m = 16; m >= LN; m >>= 1) {
        if (cnt > 1) {
            cnt /= 2;
            if (lane & m) id0 += cnt;
        } else if (lane & m) {
            writer = false;
        }
    }
    return id0;
}

template <int N>
struct BwdShape {
    static constexpr int S = bwd_states_per_lane(N);
    static constexpr int LN = N / S;          // lanes per channel
    static constexpr int CPW = 32 / LN;       // channels per warp
    static constexpr int CH = kBwdWarps * CPW;
    static constexpr int NQP = N / 2 + 1;     // widened B/C row (state pairs + one pad)
    static constexpr int P2 = S / 2;          // state pairs per lane
    static constexpr int NV = 2 * S;          // dB, dC values per lane and step
    static constexpr int CF = NV / CPW > 1 ? NV / CPW : 1;  // values left per lane after the channel sum
    static_assert(N % S == 0 && LN >= 1 && LN <= 32, "N in {4, 8, 16, 32, 64, 128, 256}");
};

// The main pass's widened B/C entry of a state pair, (B_n, B_n+1, C_n,
// C_n+1): fp32 for fp32 I/O; for bf16 I/O the four bf16 values as they
// arrive (8 bytes: half the shared-memory traffic of the reads, which is a
// co-bound of that pass), widened where they are read.
template <typename T>
struct BwdBcf {
    using type = float4;
    static __device__ __forceinline__ float4 get(const float4& v) { return v; }
};
template <>
struct BwdBcf<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ float4 get(const uint2& v) {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
};

// Channel (b, d) and chunk of this thread; inactive lanes (past the group's
// last channel) compute on a valid channel but write nothing.
struct BwdLane {
    int lane, warp, j, r, b, g, bg, d;
    bool active;
    long long bd, row;
};

template <int N>
__device__ __forceinline__ BwdLane bwd_lane(const BwdParams& p) {
    using Sh = BwdShape<N>;
    BwdLane l;
    l.lane = threadIdx.x & 31;
    l.warp = threadIdx.x >> 5;
    l.j = l.lane % Sh::LN;
    l.r = l.warp * Sh::CPW + l.lane / Sh::LN;
    const int cb = blockIdx.x % p.blocks_per_group;
    l.bg = blockIdx.x / p.blocks_per_group;
    l.g = l.bg % p.ngroups;
    l.b = l.bg / p.ngroups;
    const int dloc = cb * Sh::CH + l.r;
    l.active = dloc < p.dim_per_group;
    l.d = l.g * p.dim_per_group + (l.active ? dloc : 0);
    l.bd = static_cast<long long>(l.b) * p.dim + l.d;
    l.row = l.bd * p.seqlen;
    return l;
}

// ---------------------------------------------------------------------------
// 1. Chunk summaries, both in one forward walk over the chunk [s, e):
//      P_c = prod_t Abar_t,  E_c = the end state from a zero state,
//      M_c = the adjoint leaving the chunk at its start when none enters at
//            its end = sum_t (prod_{r=s..t} Abar_r) g_t C_t,
//    the last accumulated forwards with the running product, so the decays
//    are computed once for both.  No exchange between lanes is needed; a lane
//    holds up to 8 states (two lanes per channel at N = 16: at 16 the grid of
//    the benchmark shape had too few CTAs to hide latency).  The per-step
//    scalars (Delta, Delta u, g) are computed once per (channel, step) into
//    shared memory.
// ---------------------------------------------------------------------------
template <int N>
struct BwdSumShape {
    static constexpr int S = N < 8 ? N : 8;     // states per lane
    static constexpr int LN = N / S;            // lanes per channel
    static constexpr int CH = kBwdWarps * 32 / LN;
    static constexpr int P = S / 2;             // state pairs per lane
    static constexpr int NQP = N / 2 + 1;
};

template <typename T, int N>
struct BwdSumLayout {
    using Sh = BwdSumShape<N>;
    static constexpr int TT = kBwdTT;
    static constexpr int ACT = 0;                                                        // T [2][4][CH][TT]
    static constexpr int BC = ACT + 2 * 4 * Sh::CH * TT * static_cast<int>(sizeof(T));  // T [2][2][N][TT]
    static constexpr int SC = BC + 2 * 2 * N * TT * static_cast<int>(sizeof(T));        // float4 [TT][CH]
    static constexpr int BCF = SC + TT * Sh::CH * 16;                                    // float4 [TT][NQP]
    static constexpr int BYTES = BCF + TT * Sh::NQP * 16;
};

// Six resident CTAs per SM (80 registers; 96 and five CTAs without the bound):
// the b2 d1536 L2048 backward call measured 362.9 us against 369.9 us.
template <typename T, int N, bool ACCURATE>
__global__ void __launch_bounds__(kBwdWarps * 32, 6)
scan_bwd_summary_kernel(const BwdParams p) {
    using Sh = BwdSumShape<N>;
    using Lay = BwdSumLayout<T, N>;
    constexpr int S = Sh::S, LN = Sh::LN, CH = Sh::CH, TT = kBwdTT;
    constexpr int THREADS = kBwdWarps * 32;
    extern __shared__ __align__(16) unsigned char smem[];
    T (*act_s)[4][CH][TT] = reinterpret_cast<T (*)[4][CH][TT]>(smem + Lay::ACT);
    T (*bc_s)[2][N][TT] = reinterpret_cast<T (*)[2][N][TT]>(smem + Lay::BC);
    float4 (*sc)[CH] = reinterpret_cast<float4 (*)[CH]>(smem + Lay::SC);
    float4 (*bcf)[Sh::NQP] = reinterpret_cast<float4 (*)[Sh::NQP]>(smem + Lay::BCF);

    const int c = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int j = lane % LN;
    const int r = threadIdx.x / LN;  // channel row within the CTA
    const int cb = blockIdx.x % p.blocks_per_group;
    const int bg = blockIdx.x / p.blocks_per_group;
    const int g = bg % p.ngroups;
    const int b = bg / p.ngroups;
    const int dloc0 = cb * CH;
    const bool active = dloc0 + r < p.dim_per_group;
    const int d = g * p.dim_per_group + (active ? dloc0 + r : 0);
    const long long bd = static_cast<long long>(b) * p.dim + d;
    const int L = p.seqlen;
    const int s0 = c * p.chunk_steps;
    const int s1 = min(L, s0 + p.chunk_steps);
    const int ntile = (s1 - s0 + TT - 1) / TT;
    const long long BD = static_cast<long long>(p.batch) * p.dim;
    const bool vec = p.vec_ok != 0;
    const bool gated = p.z != nullptr;

    auto act_ptr = [&](int x) -> const T* {
        return static_cast<const T*>(x == kU ? p.u : (x == kDelta ? p.delta : (x == kZ ? p.z : p.dy)));
    };
    auto fetch = [&](int tile, int buf) {
        const int t0 = s0 + tile * TT;
        const int valid = L - t0;
        constexpr int na = 4 * CH;
        for (int item = threadIdx.x; item < na + 2 * N; item += THREADS) {
            if (item < na) {
                const int x = item / CH, rr = item % CH;
                if (x == kZ && !gated) continue;
                const int dl = min(dloc0 + rr, p.dim_per_group - 1);
                const long long row = (static_cast<long long>(b) * p.dim + g * p.dim_per_group + dl) * L + t0;
                bwd_stage_row<T>(&act_s[buf][x][rr][0], act_ptr(x) + row, valid, vec);
            } else {
                const int k = item - na;
                const int isC = k / N, n = k % N;
                const T* src = static_cast<const T*>(isC ? p.C : p.B) + (static_cast<long long>(bg) * N + n) * L + t0;
                bwd_stage_row<T>(&bc_s[buf][isC][n][0], src, valid, vec);
            }
        }
        cp_async_commit();
    };

    float2 a2[Sh::P], hs[Sh::P], pr[Sh::P], ms[Sh::P];
#pragma unroll
    for (int k = 0; k < Sh::P; ++k) {
        const float2 av = __ldg(reinterpret_cast<const float2*>(p.A + static_cast<long long>(d) * N + j * S) + k);
        a2[k] = f2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
        hs[k] = f2(0.f);
        pr[k] = f2(1.f);
        ms[k] = f2(0.f);
    }

    fetch(0, 0);
    for (int i = 0; i < ntile; ++i) {
        const int buf = i & 1;
        if (i + 1 < ntile) {
            fetch(i + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int t0 = s0 + i * TT;
        // Per-(channel, step) scalars and the widened B, C rows.
        for (int item = threadIdx.x; item < TT * CH; item += THREADS) {
            const int t = item / CH, rr = item % CH;
            const bool live = dloc0 + rr < p.dim_per_group;
            const int dl = live ? dloc0 + rr : p.dim_per_group - 1;
            const float bias = p.dt_bias ? __ldg(p.dt_bias + g * p.dim_per_group + dl) : 0.f;
            const bool in = t0 + t < L;
            const float dt = in ? softplus<ACCURATE>(bwd_to_f(act_s[buf][kDelta][rr][t]) + bias) : 0.f;
            float gg = live ? bwd_to_f(act_s[buf][kDy][rr][t]) : 0.f;
            if (gated) {
                const float zv = bwd_to_f(act_s[buf][kZ][rr][t]);
                gg *= zv * sigmoid_f<ACCURATE>(zv);
            }
            sc[t][rr] = make_float4(dt, dt * bwd_to_f(act_s[buf][kU][rr][t]), gg, 0.f);
        }
        for (int item = threadIdx.x; item < 2 * N * TT; item += THREADS) {
            const int t = item % TT, n = (item / TT) % N, isC = item / (TT * N);
            const int q = n >> 1;
            const int slot = (q % Sh::P) * LN + q / Sh::P;
            reinterpret_cast<float*>(&bcf[t][slot])[isC * 2 + (n & 1)] = bwd_to_f(bc_s[buf][isC][n][t]);
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float4 q = sc[t][r];
#pragma unroll
            for (int k = 0; k < Sh::P; ++k) {
                const float4 bq = bcf[t][k * LN + j];
                const float2 a = decay2<ACCURATE>(__fmul2_rn(f2(q.x), a2[k]));
                hs[k] = __ffma2_rn(a, hs[k], __fmul2_rn(f2(q.y), f2(bq.x, bq.y)));
                pr[k] = __fmul2_rn(pr[k], a);
                ms[k] = __ffma2_rn(pr[k], __fmul2_rn(f2(q.z), f2(bq.z, bq.w)), ms[k]);
            }
        }
    }
    if (active) {
        float* fo = p.fagg + (static_cast<long long>(c) * BD + bd) * (2 * N) + j * S;
        float* bo = p.bagg + (static_cast<long long>(c) * BD + bd) * N + j * S;
#pragma unroll
        for (int k = 0; k < Sh::P; ++k) {
            reinterpret_cast<float2*>(fo)[k] = pr[k];
            reinterpret_cast<float2*>(fo + N)[k] = hs[k];
            reinterpret_cast<float2*>(bo)[k] = ms[k];
        }
    }
}

// ---------------------------------------------------------------------------
// 2. Carry across chunks.  blockIdx.y = 0: states, forward from h0; 1:
// adjoints, backward from dh_final.  One thread per (channel, state); the
// chunk summaries are fetched eight at a time ahead of the dependent chain.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256)
scan_bwd_carry_kernel(float* __restrict__ fagg, float* __restrict__ bagg, const float* __restrict__ h0,
                      const float* __restrict__ dhf, long long BD, int nchunks) {
    constexpr int G = 8;
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i >= BD * N) return;
    const long long bd = i / N;
    const int n = static_cast<int>(i % N);
    if (blockIdx.y == 0) {
        float h = h0 ? __ldg(h0 + i) : 0.f;
        for (int c0 = 0; c0 < nchunks - 1; c0 += G) {
            float P[G], E[G];
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int c = c0 + q;
                if (c < nchunks - 1) {
                    const float* a = fagg + (static_cast<long long>(c) * BD + bd) * (2 * N) + n;
                    P[q] = __ldcg(a);
                    E[q] = __ldcg(a + N);
                }
            }
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int c = c0 + q;
                if (c < nchunks - 1) {
                    h = fmaf(P[q], h, E[q]);
                    fagg[(static_cast<long long>(c) * BD + bd) * (2 * N) + N + n] = h;
                }
            }
        }
    } else {
        float mu = dhf ? __ldg(dhf + i) : 0.f;
        for (int c0 = nchunks - 1; c0 >= 1; c0 -= G) {
            float P[G], M[G];
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int c = c0 - q;
                if (c >= 1) {
                    P[q] = __ldcg(fagg + (static_cast<long long>(c) * BD + bd) * (2 * N) + n);
                    M[q] = __ldcg(bagg + (static_cast<long long>(c) * BD + bd) * N + n);
                }
            }
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int c = c0 - q;
                if (c >= 1) {
                    mu = fmaf(P[q], mu, M[q]);
                    bagg[(static_cast<long long>(c) * BD + bd) * N + n] = mu;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 3. Main pass: checkpoints, then the tiles backwards.  Each tile's rows are
// staged by cp.async one tile ahead; the per-(channel, step) scalars are
// computed once into shared memory; the lanes run the state loops on packed
// fp32 pairs.
// ---------------------------------------------------------------------------
template <typename T, int N>
struct BwdLayout {
    using Sh = BwdShape<N>;
    static constexpr int TT = kBwdTT;
    static constexpr int THREADS = kBwdWarps * 32;
    static constexpr int CKPT = 0;                                                  // float4 [tiles * S/4][THREADS]
    static constexpr int ACT = CKPT + bwd_chunk_tiles_max(N) * (Sh::S / 4) * THREADS * 16;  // T [2][4][CH][TT]
    static constexpr int BC = ACT + 2 * 4 * Sh::CH * TT * static_cast<int>(sizeof(T));  // T [2][2][N][TT]
    static constexpr int SC = BC + 2 * 2 * N * TT * static_cast<int>(sizeof(T));   // float4 [TT][CH]
    static constexpr int SC2 = SC + TT * Sh::CH * 16;                               // float2 [TT][CH]
    static constexpr int BCF = SC2 + TT * Sh::CH * 8;                               // float4 [TT][NQP]
    // dB/dC staging per warp: the whole tile, or at N = 256 (512 values a
    // step) half of it, flushed twice a tile, so that two CTAs fit on an SM.
    static constexpr int RED_STEPS = N >= 256 ? TT / 2 : TT;
    static constexpr int RED = BCF + TT * Sh::NQP * 16;                             // float [WARPS][RED_STEPS][2N]
    static constexpr int OUTS = RED + kBwdWarps * RED_STEPS * 2 * N * 4;            // float [3][CH][TT + 1]
    static constexpr int BYTES = OUTS + 3 * Sh::CH * (TT + 1) * 4;
};

// Three CTAs per SM at most: at four the register cap (128) spills the
// tile's recomputed states, which measured 40% slower on B300.  Where the
// shared-memory footprint leaves fewer resident CTAs (N = 256: one), the
// bound follows it, so the registers that occupancy leaves free hold the
// 8 states a lane instead of spilling them.
template <typename T, int N>
constexpr int bwd_min_blocks() {
    constexpr int b = (228 * 1024) / (BwdLayout<T, N>::BYTES + 1024);
    return b < 1 ? 1 : (b > 3 ? 3 : b);
}

template <typename T, int N, bool ACCURATE>
__global__ void __launch_bounds__(kBwdWarps * 32, (bwd_min_blocks<T, N>()))
scan_bwd_kernel(const BwdParams p) {
    using Sh = BwdShape<N>;
    using Lay = BwdLayout<T, N>;
    constexpr int S = Sh::S;
    constexpr int LN = Sh::LN;
    constexpr int CH = Sh::CH;
    constexpr int TT = kBwdTT;
    constexpr int P2 = Sh::P2;
    constexpr int THREADS = kBwdWarps * 32;
    extern __shared__ __align__(16) unsigned char smem[];
    float4 (*ckpt)[THREADS] = reinterpret_cast<float4 (*)[THREADS]>(smem + Lay::CKPT);
    T (*act_s)[4][CH][TT] = reinterpret_cast<T (*)[4][CH][TT]>(smem + Lay::ACT);
    T (*bc_s)[2][N][TT] = reinterpret_cast<T (*)[2][N][TT]>(smem + Lay::BC);
    float4 (*sc)[CH] = reinterpret_cast<float4 (*)[CH]>(smem + Lay::SC);
    float2 (*sc2)[CH] = reinterpret_cast<float2 (*)[CH]>(smem + Lay::SC2);
    using Bcf = BwdBcf<T>;
    typename Bcf::type (*bcf)[Sh::NQP] = reinterpret_cast<typename Bcf::type (*)[Sh::NQP]>(smem + Lay::BCF);
    constexpr int TR = Lay::RED_STEPS;
    float (*red)[TR][2 * N] = reinterpret_cast<float (*)[TR][2 * N]>(smem + Lay::RED);
    float (*outs)[CH][TT + 1] = reinterpret_cast<float (*)[CH][TT + 1]>(smem + Lay::OUTS);

    const BwdLane l = bwd_lane<N>(p);
    const int c = blockIdx.y;
    const int L = p.seqlen;
    const int s0 = c * p.chunk_steps;
    const int s1 = min(L, s0 + p.chunk_steps);
    const int ntile = (s1 - s0 + TT - 1) / TT;
    const long long BD = static_cast<long long>(p.batch) * p.dim;
    const bool vec = p.vec_ok != 0;
    const bool gated = p.z != nullptr;
    const int dloc0 = (blockIdx.x % p.blocks_per_group) * CH;

    float2 a2[P2], Ar[P2], h[P2], mu[P2];
#pragma unroll
    for (int k = 0; k < P2; ++k) {
        const long long sidx = l.j * S + 2 * k;
        Ar[k] = __ldg(reinterpret_cast<const float2*>(p.A + static_cast<long long>(l.d) * N + sidx));
        a2[k] = __fmul2_rn(Ar[k], f2(decay_scale<ACCURATE>()));
        const long long st = l.bd * N + sidx;
        if (c == 0) h[k] = p.h0 ? __ldg(reinterpret_cast<const float2*>(p.h0 + st)) : f2(0.f);
        else h[k] = __ldcg(reinterpret_cast<const float2*>(p.fagg + (static_cast<long long>(c - 1) * BD + l.bd) * (2 * N) + N + sidx));
        if (c == p.nchunks - 1) mu[k] = p.dhf ? __ldg(reinterpret_cast<const float2*>(p.dhf + st)) : f2(0.f);
        else mu[k] = __ldcg(reinterpret_cast<const float2*>(p.bagg + (static_cast<long long>(c + 1) * BD + l.bd) * N + sidx));
        if (!l.active) mu[k] = f2(0.f);
    }
    const float dsk = p.D ? __ldg(p.D + l.d) : 0.f;

    auto act_ptr = [&](int x) -> const T* {
        return static_cast<const T*>(x == kU ? p.u : (x == kDelta ? p.delta : (x == kZ ? p.z : p.dy)));
    };
    // Stage tile `tile` into buffer `buf`: the activation rows (u, delta, and
    // for the backward walk z, dy) and the B (and C) rows.
    auto fetch = [&](int tile, int buf, bool main) {
        const int t0 = s0 + tile * TT;
        const int valid = L - t0;
        const int na = (main ? 4 : 2) * CH;
        const int nb = (main ? 2 : 1) * N;
        for (int item = threadIdx.x; item < na + nb; item += THREADS) {
            if (item < na) {
                const int x = item / CH, rr = item % CH;
                if (x == kZ && !gated) continue;
                const int dl = min(dloc0 + rr, p.dim_per_group - 1);
                const long long row = (static_cast<long long>(l.b) * p.dim + l.g * p.dim_per_group + dl) * L + t0;
                bwd_stage_row<T>(&act_s[buf][x][rr][0], act_ptr(x) + row, valid, vec);
            } else {
                const int k = item - na;
                const int isC = k / N, n = k % N;
                const T* src = static_cast<const T*>(isC ? p.C : p.B) + (static_cast<long long>(l.bg) * N + n) * L + t0;
                bwd_stage_row<T>(&bc_s[buf][isC][n][0], src, valid, vec);
            }
        }
        cp_async_commit();
    };
    // Per-(channel, step) scalars of the staged tile and the widened B/C rows.
    auto prepare = [&](int t0, int buf, bool main) {
        for (int item = threadIdx.x; item < TT * CH; item += THREADS) {
            const int t = item / CH, rr = item % CH;
            const bool live = dloc0 + rr < p.dim_per_group;
            const int dl = live ? dloc0 + rr : p.dim_per_group - 1;
            const float bias = p.dt_bias ? __ldg(p.dt_bias + l.g * p.dim_per_group + dl) : 0.f;
            const bool in = t0 + t < L;
            const float uv = bwd_to_f(act_s[buf][kU][rr][t]);
            float dt = 0.f, sg = 0.f;
            if (in) softplus_sigmoid<ACCURATE>(bwd_to_f(act_s[buf][kDelta][rr][t]) + bias, dt, sg);
            if (!main) {
                sc[t][rr] = make_float4(dt, dt * uv, 0.f, uv);
                continue;
            }
            const float dy = live ? bwd_to_f(act_s[buf][kDy][rr][t]) : 0.f;
            float gg = dy, dzf = 0.f;
            if (gated) {
                const float zv = bwd_to_f(act_s[buf][kZ][rr][t]);
                const float sz = sigmoid_f<ACCURATE>(zv);
                gg = dy * zv * sz;
                dzf = dy * sz * fmaf(zv, 1.f - sz, 1.f);
            }
            sc[t][rr] = make_float4(dt, dt * uv, gg, uv);
            sc2[t][rr] = make_float2(sg, dzf);
        }
        for (int item = threadIdx.x; item < (main ? 2 : 1) * N * TT; item += THREADS) {
            const int t = item % TT, n = (item / TT) % N, isC = item / (TT * N);
            const int q = n >> 1;
            const int slot = (q % P2) * LN + q / P2;
            reinterpret_cast<T*>(&bcf[t][slot])[isC * 2 + (n & 1)] = bc_s[buf][isC][n][t];
        }
    };

    // ---- forward sweep: the state at every tile start ----
    fetch(0, 0, false);
    for (int i = 0; i < ntile; ++i) {
        const int buf = i & 1;
        if (i + 1 < ntile) {
            fetch(i + 1, buf ^ 1, false);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        prepare(s0 + i * TT, buf, false);
        __syncthreads();
#pragma unroll
        for (int v = 0; v < S / 4; ++v)
            ckpt[i * (S / 4) + v][threadIdx.x] = make_float4(h[2 * v].x, h[2 * v].y, h[2 * v + 1].x, h[2 * v + 1].y);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float4 q = sc[t][l.r];
#pragma unroll
            for (int k = 0; k < P2; ++k) {
                const float4 bq = Bcf::get(bcf[t][k * LN + l.j]);
                h[k] = __ffma2_rn(decay2<ACCURATE>(__fmul2_rn(f2(q.x), a2[k])), h[k], __fmul2_rn(f2(q.y), f2(bq.x, bq.y)));
            }
        }
    }

    bool xw;
    const int xid0 = xchan_first_id<LN, Sh::NV>(l.lane, xw);
    float2 dA_acc[P2];
#pragma unroll
    for (int k = 0; k < P2; ++k) dA_acc[k] = f2(0.f);
    float dD_acc = 0.f, db_acc = 0.f;

    // ---- the tiles backwards ----
    fetch(ntile - 1, 0, true);
    for (int ii = 0; ii < ntile; ++ii) {
        const int i = ntile - 1 - ii;
        const int buf = ii & 1;
        const int t0 = s0 + i * TT;
        if (i > 0) {
            fetch(i - 1, buf ^ 1, true);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        prepare(t0, buf, true);
        __syncthreads();

        // Recompute the tile's states from its checkpoint: hist[t] = state
        // before step t; ys[t] = the ungated output s_t.
        float2 hist[TT][P2];
        float ys[TT];
        float2 hh[P2];
#pragma unroll
        for (int v = 0; v < S / 4; ++v) {
            const float4 c4 = ckpt[i * (S / 4) + v][threadIdx.x];
            hh[2 * v] = f2(c4.x, c4.y);
            hh[2 * v + 1] = f2(c4.z, c4.w);
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float4 q = sc[t][l.r];
            float2 y2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < P2; ++k) {
                const float4 bq = Bcf::get(bcf[t][k * LN + l.j]);
                hist[t][k] = hh[k];
                hh[k] = __ffma2_rn(decay2<ACCURATE>(__fmul2_rn(f2(q.x), a2[k])), hh[k], __fmul2_rn(f2(q.y), f2(bq.x, bq.y)));
                y2 = __ffma2_rn(f2(bq.z, bq.w), hh[k], y2);
            }
            ys[t] = fmaf(dsk, q.w, lane_sum<LN>(y2.x + y2.y));
        }

        // dB, dC of steps tb .. tb + TR - 1 of the tile: sum over warps, one
        // atomic add per CTA -- four steps per vector add when the rows keep
        // 16-byte alignment.
        auto flush_red = [&](int tb) {
            if (L % 4 == 0) {
                for (int e = threadIdx.x; e < 2 * N * (TR / 4); e += THREADS) {
                    const int t = (e % (TR / 4)) * 4;
                    const int k = e / (TR / 4);  // tensor * N + n
                    if (t0 + tb + t < L) {
                        float v[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            v[q] = 0.f;
#pragma unroll
                            for (int w = 0; w < kBwdWarps; ++w) v[q] += red[w][t + q][k];
                        }
                        float* dst = ((k / N) ? p.dC : p.dB) + (static_cast<long long>(l.bg) * N + k % N) * L + t0 + tb + t;
                        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v[0]), "f"(v[1]),
                                     "f"(v[2]), "f"(v[3])
                                     : "memory");
                    }
                }
            } else {
                for (int e = threadIdx.x; e < 2 * N * TR; e += THREADS) {
                    const int t = e % TR;
                    const int k = e / TR;  // tensor * N + n
                    if (t0 + tb + t < L) {
                        float v = 0.f;
#pragma unroll
                        for (int w = 0; w < kBwdWarps; ++w) v += red[w][t][k];
                        float* dst = (k / N) ? p.dC : p.dB;
                        atomicAdd(dst + (static_cast<long long>(l.bg) * N + k % N) * L + t0 + tb + t, v);
                    }
                }
            }
        };

        // The adjoint, backwards over the tile.
#pragma unroll
        for (int t = TT - 1; t >= 0; --t) {
            const float4 q = sc[t][l.r];   // Delta, Delta u, g, u
            const float2 q2 = sc2[t][l.r]; // sigmoid(delta + bias), dz factor
            float vals[Sh::NV];
            float2 sb2 = f2(0.f), sd2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < P2; ++k) {
                const float4 bq = Bcf::get(bcf[t][k * LN + l.j]);
                const float2 Bv = f2(bq.x, bq.y), Cv = f2(bq.z, bq.w);
                const float2 hcur = (t == TT - 1) ? hh[k] : hist[t + 1 < TT ? t + 1 : t][k];
                const float2 a = decay2<ACCURATE>(__fmul2_rn(f2(q.x), a2[k]));
                const float2 lam = __ffma2_rn(f2(q.z), Cv, mu[k]);
                const float2 db = __fmul2_rn(lam, f2(q.y));
                const float2 dc = __fmul2_rn(f2(q.z), hcur);
                vals[2 * k] = db.x;
                vals[2 * k + 1] = db.y;
                vals[S + 2 * k] = dc.x;
                vals[S + 2 * k + 1] = dc.y;
                sb2 = __ffma2_rn(lam, Bv, sb2);
                const float2 ah = __fmul2_rn(a, hist[t][k]);
                sd2 = __ffma2_rn(lam, __ffma2_rn(Bv, f2(q.w), __fmul2_rn(Ar[k], ah)), sd2);
                dA_acc[k] = __ffma2_rn(__fmul2_rn(lam, f2(q.x)), ah, dA_acc[k]);
                mu[k] = __fmul2_rn(a, lam);
            }
            const float sb = lane_sum<LN>(sb2.x + sb2.y);
            const float sd = lane_sum<LN>(sd2.x + sd2.y);
            const float duv = fmaf(q.z, dsk, q.x * sb);
            const float ddv = sd * q2.x;
            dD_acc = fmaf(q.z, q.w, dD_acc);
            db_acc += ddv;
            if (l.j == 0 % LN) outs[0][l.r][t] = duv;
            if (l.j == 1 % LN) outs[1][l.r][t] = ddv;
            if (l.j == 2 % LN) outs[2][l.r][t] = q2.y * ys[t];  // dz_t = dy_t s_t silu'(z_t)

            // dB, dC: sum over the warp's channels, then stage per warp.
            xchan_reduce<16, LN, Sh::NV>(vals, l.lane);
            if (xw) {
#pragma unroll
                for (int qq = 0; qq < Sh::CF; ++qq) {
                    const int id = xid0 + qq;
                    red[l.warp][t % TR][(id / S) * N + l.j * S + id % S] = vals[qq];
                }
            }
            if constexpr (TR < TT) {
                if (t % TR == 0 && t > 0) {  // the upper steps' staging is full: flush it
                    __syncthreads();
                    flush_red(t);
                    __syncthreads();
                }
            }
        }
        __syncthreads();

        flush_red(0);
        // du, ddelta, dz rows of the tile.
        {
            constexpr int VP = 16 / static_cast<int>(sizeof(T));
            for (int e = threadIdx.x; e < 3 * CH * (TT / VP); e += THREADS) {
                const int part = e % (TT / VP);
                const int rr = (e / (TT / VP)) % CH;
                const int x = e / (TT / VP) / CH;
                if (x == 2 && !gated) continue;
                if (dloc0 + rr >= p.dim_per_group) continue;
                const long long orow = (static_cast<long long>(l.b) * p.dim + l.g * p.dim_per_group + dloc0 + rr) * L;
                T* dst = static_cast<T*>(x == 0 ? p.du : (x == 1 ? p.ddelta : p.dz)) + orow + t0 + part * VP;
                float f[VP];
#pragma unroll
                for (int k = 0; k < VP; ++k) f[k] = outs[x][rr][part * VP + k];
                store_row<T, VP>(dst, f, L - t0 - part * VP, vec);
            }
        }
    }

    // dh0 (the adjoint leaving the first step of the sequence).
    if (c == 0 && p.dh0 && l.active) {
#pragma unroll
        for (int k = 0; k < P2; ++k)
            *reinterpret_cast<float2*>(p.dh0 + l.bd * N + l.j * S + 2 * k) = mu[k];
    }
    if (l.active) {
        // dA of this lane's S states (16-byte aligned: S is 4 or 8 floats), four per vector add.
        static_assert(S % 4 == 0, "vector adds of dA take whole groups of four states");
#pragma unroll
        for (int k = 0; k < P2; k += 2) {
            float* da = p.dA + static_cast<long long>(l.d) * N + l.j * S + 2 * k;
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(da), "f"(dA_acc[k].x),
                         "f"(dA_acc[k].y), "f"(dA_acc[k + 1].x), "f"(dA_acc[k + 1].y)
                         : "memory");
        }
        if (l.j == 0) {
            if (p.dD) atomicAdd(p.dD + l.d, dD_acc);
            if (p.ddt_bias) atomicAdd(p.ddt_bias + l.d, db_acc);
        }
    }
}

}  // namespace ssm
