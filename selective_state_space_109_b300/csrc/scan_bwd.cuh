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
// Structure.  Time is cut into chunks of bwd_chunk_steps(N) steps; a CTA owns CH
// channels of one (sequence, group) and one chunk.  Both recurrences run
// across chunks through summaries, as in the forward pass:
//   1. summary pass (two modes in one launch): forward, from a zero state,
//      the chunk's decay product P and end state E; backward, from a zero
//      adjoint, the adjoint M that leaves the chunk at its start
//      (mu = Abar_t lam_t after the chunk's first step);
//   2. carry pass: h entering chunk c+1 = P_c h + E_c (from h0), and the
//      adjoint entering chunk c-1 from the right = P_c mu + M_c (from dh_final);
//   3. main pass: from the state entering its chunk, a forward sweep stores
//      the state at every tile start in shared memory; then the tiles are
//      walked backwards: each tile's states are recomputed into registers from
//      its checkpoint, and the adjoint runs back over the tile, producing every
//      gradient of the tile's steps.
//
// Lanes: LN = N/4 consecutive lanes share a channel, 4 states each.  The
// per-step sums over states (the readout, du, dDelta) are butterfly-reduced
// over the LN lanes; dB and dC sum over the channels of the group: a
// reduce-scatter over the channels of a warp, a sum over the CTA's warps in
// shared memory, then one atomic add per (state, step) per CTA into fp32
// buffers.  dA, dD and ddt_bias collect in registers and are added atomically
// once per CTA.
#pragma once

#include "ssm_device.cuh"

namespace ssm {

constexpr int kBwdTT = 8;       // steps per tile
constexpr int kBwdWarps = 4;
constexpr int kBwdStates = 4;   // states per lane

// Tiles per time chunk: their start states are held in shared memory (16 KB
// per 8 tiles); fewer at N = 64, whose dB/dC staging is larger.
__host__ __device__ constexpr int bwd_chunk_tiles(int n) { return n >= 64 ? 8 : 16; }
__host__ __device__ constexpr int bwd_chunk_steps(int n) { return kBwdTT * bwd_chunk_tiles(n); }

struct BwdParams {
    const void *u, *delta, *z, *dy, *B, *C;
    const float *A, *D, *dt_bias, *h0, *dhf;
    void *du, *ddelta, *dz;
    float *dA, *dB, *dC, *dD, *ddt_bias, *dh0;
    float* fagg;  // [nchunks][batch*dim][2][N]: P, then E (replaced by the state entering chunk c+1)
    float* bagg;  // [nchunks][batch*dim][N]: M (replaced by the adjoint entering chunk c-1 from the right)
    int batch, dim, seqlen, ngroups, dim_per_group, blocks_per_group, nchunks;
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

// kBwdTT consecutive elements of a row starting at p (valid = elements in
// range; the rest read as zero); cached loads (the rows are read twice).
template <typename T>
__device__ __forceinline__ void bwd_load_steps(const T* p, int valid, bool vec_ok, float (&f)[kBwdTT]) {
    constexpr int VP = 16 / static_cast<int>(sizeof(T));
#pragma unroll
    for (int q = 0; q < kBwdTT / VP; ++q) {
        Packet<T, VP> pk;
        const int v = valid - q * VP;
        if (vec_ok && v >= VP) {
            pk.load_cached(p + q * VP);
        } else {
            float g[VP];
#pragma unroll
            for (int k = 0; k < VP; ++k) g[k] = k < v ? Elem<T>::load(p + q * VP + k) : 0.f;
            pk.from_float(g);
        }
        float g[VP];
        pk.to_float(g);
#pragma unroll
        for (int k = 0; k < VP; ++k) f[q * VP + k] = g[k];
    }
}

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
    static constexpr int S = kBwdStates;
    static constexpr int LN = N / S;          // lanes per channel
    static constexpr int CPW = 32 / LN;       // channels per warp
    static constexpr int CH = kBwdWarps * CPW;
    static constexpr int NQP = N / 2 + 1;     // widened B/C row (state pairs + one pad)
    static constexpr int P2 = S / 2;          // state pairs per lane
    static constexpr int NV = 2 * S;          // dB, dC values per lane and step
    static constexpr int CF = NV / CPW > 1 ? NV / CPW : 1;  // values left per lane after the channel sum
    static_assert(N % S == 0 && LN >= 1 && LN <= 16, "N in {4, 8, 16, 32, 64}");
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

// Loads the B (and/or C) rows of the tile at t0 and widens them into
// bcf[t][pair slot] = (B_2q, B_2q+1, C_2q, C_2q+1); pair q of sub-lane j sits
// at slot (q % P2) * LN + q / P2 so that a channel's lanes read adjacent
// entries.  Called by every thread; synchronises before and after.
template <typename T, int N>
__device__ __forceinline__ void bwd_stage_bc(const BwdParams& p, int bg, int t0, bool withB, bool withC,
                                             float4 (*bcf)[BwdShape<N>::NQP]) {
    using Sh = BwdShape<N>;
    __syncthreads();
    const long long base = static_cast<long long>(bg) * N * p.seqlen + t0;
    for (int item = threadIdx.x; item < 2 * N; item += kBwdWarps * 32) {
        const int isC = item / N;
        const int n = item % N;
        if ((isC && !withC) || (!isC && !withB)) continue;
        const T* src = static_cast<const T*>(isC ? p.C : p.B) + base + static_cast<long long>(n) * p.seqlen;
        float f[kBwdTT];
        bwd_load_steps<T>(src, p.seqlen - t0, p.vec_ok != 0, f);
        const int q = n >> 1;
        const int slot = (q % Sh::P2) * Sh::LN + q / Sh::P2;
        float* dst = reinterpret_cast<float*>(&bcf[0][slot]) + isC * 2 + (n & 1);
#pragma unroll
        for (int t = 0; t < kBwdTT; ++t) dst[t * Sh::NQP * 4] = f[t];
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// 1. Chunk summaries.  blockIdx.z = 0: forward (P_c, E_c); 1: backward M_c.
// ---------------------------------------------------------------------------
template <typename T, int N, bool ACCURATE>
__global__ void __launch_bounds__(kBwdWarps * 32)
scan_bwd_summary_kernel(const BwdParams p) {
    using Sh = BwdShape<N>;
    constexpr int S = Sh::S;
    constexpr int TT = kBwdTT;
    __shared__ __align__(16) float4 bcf[TT][Sh::NQP];
    const BwdLane l = bwd_lane<N>(p);
    const int c = blockIdx.y;
    const bool fwd = blockIdx.z == 0;
    if (!fwd && c == 0) return;  // M_0 is not needed (uniform over the CTA)
    const int L = p.seqlen;
    const int s0 = c * bwd_chunk_steps(N);
    const int s1 = min(L, s0 + bwd_chunk_steps(N));
    const int ntile = (s1 - s0 + TT - 1) / TT;
    const long long BD = static_cast<long long>(p.batch) * p.dim;

    float a2[S];
#pragma unroll
    for (int s = 0; s < S; ++s) a2[s] = __ldg(p.A + static_cast<long long>(l.d) * N + l.j * S + s) * decay_scale<ACCURATE>();
    const float bias = p.dt_bias ? __ldg(p.dt_bias + l.d) : 0.f;
    const bool vec = p.vec_ok != 0;
    const T* drow = static_cast<const T*>(p.delta) + l.row;

    if (fwd) {
        const T* urow = static_cast<const T*>(p.u) + l.row;
        float h[S], pr[S];
#pragma unroll
        for (int s = 0; s < S; ++s) { h[s] = 0.f; pr[s] = 1.f; }
        for (int i = 0; i < ntile; ++i) {
            const int t0 = s0 + i * TT;
            bwd_stage_bc<T, N>(p, l.bg, t0, true, false, bcf);
            float uu[TT], dv[TT];
            bwd_load_steps<T>(urow + t0, L - t0, vec, uu);
            bwd_load_steps<T>(drow + t0, L - t0, vec, dv);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const float dt = (t0 + t < L) ? softplus<ACCURATE>(dv[t] + bias) : 0.f;
                const float dtu = dt * uu[t];
#pragma unroll
                for (int k = 0; k < Sh::P2; ++k) {
                    const float4 q = bcf[t][k * Sh::LN + l.j];
                    const float e0 = decay<ACCURATE>(dt * a2[2 * k]);
                    const float e1 = decay<ACCURATE>(dt * a2[2 * k + 1]);
                    pr[2 * k] *= e0;
                    pr[2 * k + 1] *= e1;
                    h[2 * k] = fmaf(e0, h[2 * k], dtu * q.x);
                    h[2 * k + 1] = fmaf(e1, h[2 * k + 1], dtu * q.y);
                }
            }
        }
        if (l.active) {
            float* out = p.fagg + (static_cast<long long>(c) * BD + l.bd) * (2 * N) + l.j * S;
#pragma unroll
            for (int s = 0; s < S; ++s) {
                out[s] = pr[s];
                out[N + s] = h[s];
            }
        }
    } else {
        const T* zrow = p.z ? static_cast<const T*>(p.z) + l.row : nullptr;
        const T* yrow = static_cast<const T*>(p.dy) + l.row;
        float mu[S];
#pragma unroll
        for (int s = 0; s < S; ++s) mu[s] = 0.f;
        for (int i = ntile - 1; i >= 0; --i) {
            const int t0 = s0 + i * TT;
            bwd_stage_bc<T, N>(p, l.bg, t0, false, true, bcf);
            float dv[TT], zz[TT], gy[TT];
            bwd_load_steps<T>(drow + t0, L - t0, vec, dv);
            bwd_load_steps<T>(yrow + t0, L - t0, vec, gy);
            if (zrow) bwd_load_steps<T>(zrow + t0, L - t0, vec, zz);
#pragma unroll
            for (int t = TT - 1; t >= 0; --t) {
                const bool in = t0 + t < L;
                const float dt = in ? softplus<ACCURATE>(dv[t] + bias) : 0.f;
                const float g = zrow ? gy[t] * silu<ACCURATE>(zz[t]) : gy[t];
#pragma unroll
                for (int k = 0; k < Sh::P2; ++k) {
                    const float4 q = bcf[t][k * Sh::LN + l.j];
                    const float l0 = fmaf(g, q.z, mu[2 * k]);
                    const float l1 = fmaf(g, q.w, mu[2 * k + 1]);
                    mu[2 * k] = decay<ACCURATE>(dt * a2[2 * k]) * l0;
                    mu[2 * k + 1] = decay<ACCURATE>(dt * a2[2 * k + 1]) * l1;
                }
            }
        }
        if (l.active) {
            float* out = p.bagg + (static_cast<long long>(c) * BD + l.bd) * N + l.j * S;
#pragma unroll
            for (int s = 0; s < S; ++s) out[s] = mu[s];
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
// 3. Main pass: checkpoints, then the tiles backwards.
// ---------------------------------------------------------------------------
template <typename T, int N, bool ACCURATE>
__global__ void __launch_bounds__(kBwdWarps * 32, 3)
scan_bwd_kernel(const BwdParams p) {
    using Sh = BwdShape<N>;
    constexpr int S = Sh::S;
    constexpr int LN = Sh::LN;
    constexpr int CH = Sh::CH;
    constexpr int TT = kBwdTT;
    constexpr int THREADS = kBwdWarps * 32;
    __shared__ __align__(16) float4 ckpt[bwd_chunk_tiles(N)][THREADS];
    __shared__ __align__(16) float4 bcf[TT][Sh::NQP];
    __shared__ float red[kBwdWarps][TT][2 * N];
    __shared__ float outs[3][CH][TT + 1];

    const BwdLane l = bwd_lane<N>(p);
    const int c = blockIdx.y;
    const int L = p.seqlen;
    const int s0 = c * bwd_chunk_steps(N);
    const int s1 = min(L, s0 + bwd_chunk_steps(N));
    const int ntile = (s1 - s0 + TT - 1) / TT;
    const long long BD = static_cast<long long>(p.batch) * p.dim;
    const bool vec = p.vec_ok != 0;
    const bool gated = p.z != nullptr;

    float a2[S], Ar[S], h[S], mu[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        Ar[s] = __ldg(p.A + static_cast<long long>(l.d) * N + l.j * S + s);
        a2[s] = Ar[s] * decay_scale<ACCURATE>();
        const long long st = l.bd * N + l.j * S + s;
        if (c == 0) h[s] = p.h0 ? __ldg(p.h0 + st) : 0.f;
        else h[s] = __ldcg(p.fagg + (static_cast<long long>(c - 1) * BD + l.bd) * (2 * N) + N + l.j * S + s);
        if (c == p.nchunks - 1) mu[s] = p.dhf ? __ldg(p.dhf + st) : 0.f;
        else mu[s] = __ldcg(p.bagg + (static_cast<long long>(c + 1) * BD + l.bd) * N + l.j * S + s);
        if (!l.active) mu[s] = 0.f;
    }
    const float bias = p.dt_bias ? __ldg(p.dt_bias + l.d) : 0.f;
    const float dsk = p.D ? __ldg(p.D + l.d) : 0.f;
    const T* urow = static_cast<const T*>(p.u) + l.row;
    const T* drow = static_cast<const T*>(p.delta) + l.row;
    const T* zrow = gated ? static_cast<const T*>(p.z) + l.row : nullptr;
    const T* yrow = static_cast<const T*>(p.dy) + l.row;

    // ---- forward sweep: the state at every tile start ----
    for (int i = 0; i < ntile; ++i) {
        const int t0 = s0 + i * TT;
        ckpt[i][threadIdx.x] = make_float4(h[0], h[1], h[2], h[3]);
        bwd_stage_bc<T, N>(p, l.bg, t0, true, false, bcf);
        float uu[TT], dv[TT];
        bwd_load_steps<T>(urow + t0, L - t0, vec, uu);
        bwd_load_steps<T>(drow + t0, L - t0, vec, dv);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float dt = (t0 + t < L) ? softplus<ACCURATE>(dv[t] + bias) : 0.f;
            const float dtu = dt * uu[t];
#pragma unroll
            for (int k = 0; k < Sh::P2; ++k) {
                const float4 q = bcf[t][k * LN + l.j];
                h[2 * k] = fmaf(decay<ACCURATE>(dt * a2[2 * k]), h[2 * k], dtu * q.x);
                h[2 * k + 1] = fmaf(decay<ACCURATE>(dt * a2[2 * k + 1]), h[2 * k + 1], dtu * q.y);
            }
        }
    }

    bool xw;
    const int xid0 = xchan_first_id<LN, Sh::NV>(l.lane, xw);
    float dA_acc[S];
#pragma unroll
    for (int s = 0; s < S; ++s) dA_acc[s] = 0.f;
    float dD_acc = 0.f, db_acc = 0.f;

    // ---- the tiles backwards ----
    for (int i = ntile - 1; i >= 0; --i) {
        const int t0 = s0 + i * TT;
        bwd_stage_bc<T, N>(p, l.bg, t0, true, true, bcf);
        float uu[TT], dv[TT], zz[TT], gy[TT];
        bwd_load_steps<T>(urow + t0, L - t0, vec, uu);
        bwd_load_steps<T>(drow + t0, L - t0, vec, dv);
        bwd_load_steps<T>(yrow + t0, L - t0, vec, gy);
        if (gated) bwd_load_steps<T>(zrow + t0, L - t0, vec, zz);
        if (!l.active) {
#pragma unroll
            for (int t = 0; t < TT; ++t) gy[t] = 0.f;
        }

        // Recompute the tile's states from its checkpoint; hist[t] = state
        // before step t; the readout s_t is summed over the channel's lanes.
        float hist[TT][S], dts[TT], sg[TT], ys[TT];
        {
            const float4 c4 = ckpt[i][threadIdx.x];
            float hh[S] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const bool in = t0 + t < L;
                const float v = dv[t] + bias;
                const float dt = in ? softplus<ACCURATE>(v) : 0.f;
                dts[t] = dt;
                sg[t] = in ? sigmoid_f<ACCURATE>(v) : 0.f;
                const float dtu = dt * uu[t];
                float y = 0.f;
#pragma unroll
                for (int k = 0; k < Sh::P2; ++k) {
                    const float4 q = bcf[t][k * LN + l.j];
                    hist[t][2 * k] = hh[2 * k];
                    hist[t][2 * k + 1] = hh[2 * k + 1];
                    hh[2 * k] = fmaf(decay<ACCURATE>(dt * a2[2 * k]), hh[2 * k], dtu * q.x);
                    hh[2 * k + 1] = fmaf(decay<ACCURATE>(dt * a2[2 * k + 1]), hh[2 * k + 1], dtu * q.y);
                    y = fmaf(q.z, hh[2 * k], y);
                    y = fmaf(q.w, hh[2 * k + 1], y);
                }
                ys[t] = lane_sum<LN>(y) + dsk * uu[t];
            }
            // The state after the tile's last step (h_t of that step).
#pragma unroll
            for (int s = 0; s < S; ++s) h[s] = hh[s];
        }

        // The adjoint, backwards over the tile.
#pragma unroll
        for (int t = TT - 1; t >= 0; --t) {
            float g = gy[t], dzv = 0.f;
            if (gated) {
                const float sz = sigmoid_f<ACCURATE>(zz[t]);
                dzv = gy[t] * ys[t] * sz * fmaf(zz[t], 1.f - sz, 1.f);
                g = gy[t] * zz[t] * sz;
            }
            const float dt = dts[t];
            const float dtu = dt * uu[t];
            float vals[Sh::NV];
            float sb = 0.f, sd = 0.f;
#pragma unroll
            for (int k = 0; k < Sh::P2; ++k) {
                const float4 q = bcf[t][k * LN + l.j];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int s = 2 * k + e;
                    const float Bv = e ? q.y : q.x;
                    const float Cv = e ? q.w : q.z;
                    const float hcur = (t == TT - 1) ? h[s] : hist[t + 1 < TT ? t + 1 : t][s];
                    const float hprev = hist[t][s];
                    const float a = decay<ACCURATE>(dt * a2[s]);
                    const float lam = fmaf(g, Cv, mu[s]);
                    vals[s] = lam * dtu;
                    vals[S + s] = g * hcur;
                    sb = fmaf(lam, Bv, sb);
                    const float ah = a * hprev;
                    sd = fmaf(lam, fmaf(Bv, uu[t], Ar[s] * ah), sd);
                    dA_acc[s] = fmaf(lam * dt, ah, dA_acc[s]);
                    mu[s] = a * lam;
                }
            }
            sb = lane_sum<LN>(sb);
            sd = lane_sum<LN>(sd);
            const float duv = fmaf(g, dsk, dt * sb);
            const float ddv = sd * sg[t];
            dD_acc = fmaf(g, uu[t], dD_acc);
            db_acc += ddv;
            if (l.j == 0 % LN) outs[0][l.r][t] = duv;
            if (l.j == 1 % LN) outs[1][l.r][t] = ddv;
            if (l.j == 2 % LN) outs[2][l.r][t] = dzv;

            // dB, dC: sum over the warp's channels, then stage per warp.
            xchan_reduce<16, LN, Sh::NV>(vals, l.lane);
            if (xw) {
#pragma unroll
                for (int q = 0; q < Sh::CF; ++q) {
                    const int id = xid0 + q;
                    const int tensor = id / S;
                    const int n = l.j * S + id % S;
                    red[l.warp][t][tensor * N + n] = vals[q];
                }
            }
        }
        __syncthreads();

        // dB, dC of the tile: sum over warps, one atomic add per CTA.
        for (int e = threadIdx.x; e < 2 * N * TT; e += THREADS) {
            const int t = e % TT;
            const int k = e / TT;  // tensor * N + n
            if (t0 + t < L) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kBwdWarps; ++w) v += red[w][t][k];
                const int tensor = k / N;
                const int n = k % N;
                float* dst = tensor ? p.dC : p.dB;
                atomicAdd(dst + (static_cast<long long>(l.bg) * N + n) * L + t0 + t, v);
            }
        }
        // du, ddelta, dz rows of the tile.
        {
            constexpr int VP = 16 / static_cast<int>(sizeof(T));
            const int dloc0 = (blockIdx.x % p.blocks_per_group) * CH;
            for (int e = threadIdx.x; e < 3 * CH * (TT / VP); e += THREADS) {
                const int part = e % (TT / VP);
                const int rr = (e / (TT / VP)) % CH;
                const int x = e / (TT / VP) / CH;
                if (x == 2 && !gated) continue;
                if (dloc0 + rr >= p.dim_per_group) continue;
                const long long drow_out = (static_cast<long long>(l.b) * p.dim + l.g * p.dim_per_group + dloc0 + rr) * L;
                T* dst = static_cast<T*>(x == 0 ? p.du : (x == 1 ? p.ddelta : p.dz)) + drow_out + t0 + part * VP;
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
        for (int s = 0; s < S; ++s) p.dh0[l.bd * N + l.j * S + s] = mu[s];
    }
    if (l.active) {
#pragma unroll
        for (int s = 0; s < S; ++s) atomicAdd(p.dA + static_cast<long long>(l.d) * N + l.j * S + s, dA_acc[s]);
        if (l.j == 0) {
            if (p.dD) atomicAdd(p.dD + l.d, dD_acc);
            if (p.ddt_bias) atomicAdd(p.ddt_bias + l.d, db_acc);
        }
    }
}

}  // namespace ssm
