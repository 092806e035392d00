// scan_tma.cuh -- TMA-staged selective-scan kernels for sm_103a.
//
// The same kernel template runs two passes of the scan:
//
//   Full       softplus step -> zero-order-hold decay exp(Delta A) -> input
//              term Delta B u -> diagonal recurrence h = Abar h + Bbar x ->
//              readout C.h -> skip D u -> silu(z) gate -> y, with the state
//              in registers (eightmm.github.io "Mamba", Main Claim and Scan
//              View; intvml.com "DL0170 Mamba Selective SSM vs Attention",
//              Mathematical Formulation).  A time chunk c > 0 starts from the
//              state carried into it (computed by scan_carry_kernel from the
//              chunk summaries below).
//   Aggregate  the same recurrence over one time chunk from a zero state,
//              without readout: it writes the chunk's summary, the pair
//              (P, E) with P[n] = prod_t Abar_t[n] = exp(A[n] sum_t Delta_t)
//              and E[n] = the chunk's end state.  Because the recurrence is a
//              scan over the pairs (Abar_t, Bbar_t x_t) (eightmm.github.io
//              "Mamba", Scan View), the state entering chunk c is
//              h_c = P_{c-1} (... (P_0 h0 + E_0) ...) + E_{c-1}.
//
// Data movement: every operand tile arrives by TMA into shared memory.  A CTA
// owns CH consecutive channels of one (sequence, group) and one time chunk; it
// walks the chunk in tiles of TS steps (kScanRowBytes = 32 bytes of each
// channel row), through a 4-stage ring of mbarrier-tracked stages.  Activation
// tiles (u, delta, z) are [CH rows x 32 B] with the TMA swizzle of that row
// width, so that the lanes of a warp, each reading its own row, hit distinct
// banks.  Narrow rows keep a CTA's stages small (13 KB per stage of the full
// pass), so that four CTAs -- four warps per scheduler -- fit on an SM.  B and
// C tiles ([N rows x 32 B],
// shared by all channels of the group) are widened once per tile into fp32
// (B_n, B_n+1, C_n, C_n+1) quads that every lane reads by broadcast.  y is
// written back in place over the u tile and leaves by a TMA store.
//
// Lanes: LANES consecutive lanes share one channel, S = N / LANES states each.
// Per 16-byte chunk of a row (VPC steps) lane j computes Delta and Delta*u for
// H = VPC / LANES of the steps and posts them, as ready-made fp32 pairs, to a
// per-warp scratch row that all lanes of the channel read; after the chunk's
// recurrence a butterfly reduce-scatter leaves lane j with the full readout
// of its H steps, which it gates and stores.
#pragma once

#include <type_traits>

#include "ssm_device.cuh"
#include "tma.cuh"

namespace ssm {

struct TmaScanParams {
    const float* A;
    const float* D;        // nullable
    const float* dt_bias;  // nullable
    const float* h0;       // nullable
    float* h_final;        // nullable
    float* agg;            // chunk summaries [nchunks - 1][batch * dim][2][N] (P then E)
    unsigned int* status;  // nullable caller status word (timeouts)
    int batch, dim, seqlen, ngroups, dim_per_group;
    int blocks_per_group;  // CTAs along the channels of one group
    int nchunks;           // time chunks of the Full pass
    int ntiles;            // ceil(seqlen / TS)
    int has_z;
};

enum class ScanMode { Full, Aggregate };

// Bytes of each channel row in one tile: 32 (TMA 32-byte swizzle) or 64
// (64-byte swizzle).  The build may override it to compare the two.
#ifndef SSM_SCAN_ROW_BYTES
#define SSM_SCAN_ROW_BYTES 32
#endif
constexpr int kScanRowBytes = SSM_SCAN_ROW_BYTES;
static_assert(kScanRowBytes == 32 || kScanRowBytes == 64, "tile rows are 32 or 64 bytes");

// Byte offset of 16-byte chunk c of row r in an activation tile.
__device__ __forceinline__ uint32_t swz_act(int r, int c) {
    if constexpr (kScanRowBytes == 64) return swz64(r, c);
    else return swz32(r, c);
}

template <typename T>
struct TileShape {
    static constexpr int kRowBytes = kScanRowBytes;
    static constexpr int TS = kRowBytes / static_cast<int>(sizeof(T));  // steps per tile
    static constexpr int VPC = 16 / static_cast<int>(sizeof(T));        // steps per 16-byte chunk
    static constexpr int CHUNKS = kRowBytes / 16;
};

template <typename T, int N, int LANES, int WARPS, ScanMode MODE>
struct TmaScanLayout {
    static constexpr bool FULL = MODE == ScanMode::Full;
    static constexpr int CH = WARPS * 32 / LANES;
    static constexpr int ACT_BYTES = CH * TileShape<T>::kRowBytes;  // one activation tile
    static constexpr int BC_BYTES = N * TileShape<T>::kRowBytes;    // one B or C tile
    static constexpr int NACT = FULL ? 3 : 2;                       // u, delta (, z)
    static constexpr int NBC = FULL ? 2 : 1;                        // B (, C)
    // The full pass refills a stage only after its y store has read it, so it
    // runs STAGES - 2 tiles ahead; the summary pass runs STAGES - 1 ahead.
    static constexpr int STAGES = FULL ? 4 : 3;
    static constexpr int STAGE_BYTES = ((NACT * ACT_BYTES + NBC * BC_BYTES) + 1023) / 1024 * 1024;
    // Widened B (, C): one row of N/2 state pairs per step plus one pad pair,
    // so that the widening loop's stores (consecutive steps of one pair) fall
    // in different banks.
    static constexpr int BCF_ROW = N / 2 + 1;
    static constexpr int BCF_BYTES = TileShape<T>::TS * BCF_ROW * 8 * NBC;
    // Per-warp scratch through which the lanes of a channel share (Delta,
    // Delta u) for one 16-byte chunk: two buffers (alternating chunks) of one
    // padded row of VPC float4 per channel.
    static constexpr int XS_STRIDE = TileShape<T>::VPC * 16 + 16;
    static constexpr int XS_BUF = (32 / LANES) * XS_STRIDE;
    static constexpr int XS_BYTES = LANES > 1 ? WARPS * 2 * XS_BUF : 0;
    static constexpr int XS_OFFSET = STAGES * STAGE_BYTES + BCF_BYTES;
    static constexpr int BAR_OFFSET = XS_OFFSET + XS_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + STAGES * 8 + 1024;  // + alignment slack
    static_assert(ACT_BYTES % (8 * TileShape<T>::kRowBytes) == 0, "activation tiles must keep the swizzle phase");
};

// Loads H consecutive elements (H * sizeof(T) = 2, 4, 8 or 16 bytes) from shared memory.
template <typename T, int H>
__device__ __forceinline__ void lds_row(const unsigned char* p, float (&f)[H]) {
    constexpr int BYTES = H * static_cast<int>(sizeof(T));
    if constexpr (BYTES == 2) {
        f[0] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
    } else {
        uint32_t w[BYTES / 4];
        if constexpr (BYTES == 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        } else if constexpr (BYTES == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            w[0] = v.x; w[1] = v.y;
        } else {
            static_assert(BYTES == 4, "2, 4, 8 or 16 bytes");
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        }
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int k = 0; k < H; ++k) f[k] = __uint_as_float(w[k]);
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                f[2 * k] = __uint_as_float(w[k] << 16);
                f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
            }
        }
    }
}

// Rounds H floats to T (bf16: nearest even) and stores them to shared memory.
template <typename T, int H>
__device__ __forceinline__ void sts_row(unsigned char* p, const float (&f)[H]) {
    constexpr int BYTES = H * static_cast<int>(sizeof(T));
    if constexpr (BYTES == 2) {
        const __nv_bfloat16 h = __float2bfloat16_rn(f[0]);
        *reinterpret_cast<unsigned short*>(p) = *reinterpret_cast<const unsigned short*>(&h);
    } else {
        uint32_t w[BYTES / 4];
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int k = 0; k < H; ++k) w[k] = __float_as_uint(f[k]);
        } else {
#pragma unroll
            for (int k = 0; k < BYTES / 4; ++k) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
        }
        if constexpr (BYTES == 16) {
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        } else if constexpr (BYTES == 8) {
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<uint32_t*>(p) = w[0];
        }
    }
}

template <typename T>
__device__ __forceinline__ float lds_elem(const unsigned char* p) {
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float*>(p);
    } else {
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
    }
}

// Most CTAs of one kernel planned per SM: four (four warps per scheduler)
// saturate the update mix, and more would cut registers below 128 a thread.
constexpr int kMaxCtasPerSm = 4;

// CTAs that shared memory lets reside on one SM (228 KB, 1 KB reserved per
// CTA), at most kMaxCtasPerSm: passed to __launch_bounds__ so that ptxas may
// use every register that this residency leaves free.
template <typename T, int N, int LANES, int WARPS, ScanMode MODE>
constexpr int tma_min_blocks() {
    constexpr int per = TmaScanLayout<T, N, LANES, WARPS, MODE>::SMEM_BYTES + 1024;
    constexpr int b = (228 * 1024) / per;
    return b < 1 ? 1 : (b > kMaxCtasPerSm ? kMaxCtasPerSm : b);
}

template <typename T, int N, int LANES, int WARPS, ScanMode MODE, bool ACCURATE>
__global__ void __launch_bounds__(WARPS * 32, (tma_min_blocks<T, N, LANES, WARPS, MODE>()))
scan_tma_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_y,
                const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
                const TmaScanParams p) {
    using Lay = TmaScanLayout<T, N, LANES, WARPS, MODE>;
    using Sh = TileShape<T>;
    constexpr bool FULL = Lay::FULL;
    constexpr int TS = Sh::TS;
    constexpr int VPC = Sh::VPC;
    constexpr int S = N / LANES;       // states per lane
    constexpr int P = S / 2;           // fp32x2 state pairs per lane
    constexpr int NQ = N / 2;          // state pairs per step
    constexpr int NQP = Lay::BCF_ROW;  // widened row stride (pairs)
    // Steps a lane owns per 16-byte chunk.  With more lanes than steps
    // (N = 128: 8 lanes of 16 states), lanes j >= VPC own none.
    constexpr int H = VPC >= LANES ? VPC / LANES : 1;
    constexpr bool SPARE = LANES > VPC;
    // Per-step scalar work (softplus, Delta u, gate) in fp32x2 pairs of steps.
    constexpr bool PACKED = !ACCURATE && (H % 2 == 0);
    constexpr int CH = Lay::CH;
    constexpr int THREADS = WARPS * 32;
    constexpr int STAGES = Lay::STAGES;
    static_assert(S >= 2 && S % 2 == 0, "each lane holds an even number of states");
    static_assert(H >= 1, "a lane owns at least one step of each chunk");

    // Align the dynamic shared memory to 1024 bytes by offsetting the shared
    // array itself, so that every access below stays a shared-memory access.
    extern __shared__ __align__(16) unsigned char smem_raw[];  // aligned below at run time
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* bcf = reinterpret_cast<float*>(smem + STAGES * Lay::STAGE_BYTES);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFFSET);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int r = warp * (32 / LANES) + lane / LANES;  // channel row within the CTA
    const int j = lane % LANES;                        // sub-lane within the channel
    const int jj = SPARE ? j % VPC : j;                // its step slot in a chunk
    const bool own = !SPARE || j < VPC;                // it owns steps
    const int cw = lane / LANES;                       // channel within the warp
    unsigned char* xs_warp = smem + Lay::XS_OFFSET + warp * 2 * Lay::XS_BUF;

    const int cb = blockIdx.x % p.blocks_per_group;
    const int bg = blockIdx.x / p.blocks_per_group;  // b * ngroups + g
    const int g = bg % p.ngroups;
    const int b = bg / p.ngroups;
    const int dloc0 = cb * CH;
    const int dloc = dloc0 + r;
    const bool active = dloc < p.dim_per_group;
    const int d = g * p.dim_per_group + (active ? dloc : 0);
    const long long bd = static_cast<long long>(b) * p.dim + d;
    const long long BD = static_cast<long long>(p.batch) * p.dim;

    const int chunk = blockIdx.y;
    const int tb = static_cast<int>(static_cast<long long>(chunk) * p.ntiles / p.nchunks);
    const int te = static_cast<int>(static_cast<long long>(chunk + 1) * p.ntiles / p.nchunks);
    const int nt = te - tb;

    // ---- per-lane constants and the state entering this chunk ----
    float2 a2[P], h[P];
    {
        const float* Ad = p.A + static_cast<long long>(d) * N + j * S;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const float2 av = __ldg(reinterpret_cast<const float2*>(Ad) + k);
            a2[k] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
            h[k] = make_float2(0.f, 0.f);
        }
        if constexpr (FULL) {
            if (p.h0 && active) {
                const float2* h0v = reinterpret_cast<const float2*>(p.h0 + bd * N + j * S);
#pragma unroll
                for (int k = 0; k < P; ++k) h[k] = __ldg(h0v + k);
            }
        }
    }
    const float bias = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
    const float dsk = p.D ? __ldg(p.D + d) : 0.f;
    const bool has_z = FULL && p.has_z;

    // ---- barriers and the TMA prologue ----
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_d);
        prefetch_tensormap(&tm_B);
        if constexpr (FULL) {
            prefetch_tensormap(&tm_y);
            prefetch_tensormap(&tm_C);
            if (has_z) prefetch_tensormap(&tm_z);
        }
    }
    __syncthreads();

    const uint32_t stage_tx =
        static_cast<uint32_t>((2 + (has_z ? 1 : 0)) * Lay::ACT_BYTES + Lay::NBC * Lay::BC_BYTES);
    auto stage_ptr = [&](int s) { return smem + s * Lay::STAGE_BYTES; };
    auto issue = [&](int i) {  // thread 0 only: load tile tb + i into its stage
        const int s = i % STAGES;
        unsigned char* st = stage_ptr(s);
        const int x = (tb + i) * TS;
        mbar_arrive_expect_tx(&full_bar[s], stage_tx);
        tma_load_3d(st, &tm_u, x, dloc0, bg, &full_bar[s]);
        tma_load_3d(st + Lay::ACT_BYTES, &tm_d, x, dloc0, bg, &full_bar[s]);
        if (has_z) tma_load_3d(st + 2 * Lay::ACT_BYTES, &tm_z, x, dloc0, bg, &full_bar[s]);
        unsigned char* bc = st + Lay::NACT * Lay::ACT_BYTES;
        tma_load_2d(bc, &tm_B, x, bg * N, &full_bar[s]);
        if constexpr (FULL) tma_load_2d(bc + Lay::BC_BYTES, &tm_C, x, bg * N, &full_bar[s]);
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES && i < nt; ++i) issue(i);
    }
    if constexpr (FULL) {
        // A later chunk starts from the state carried into it, which the carry
        // pass left in the E slot of the previous chunk's summary.  This kernel
        // may have started while that pass still ran (its input tiles are
        // already on their way): wait for it before reading the carry.
        if (chunk > 0) {
            grid_dep_wait();
            if (active) {
                const float2* carry = reinterpret_cast<const float2*>(
                    p.agg + (static_cast<long long>(chunk - 1) * BD + bd) * (2 * N) + N + j * S);
#pragma unroll
                for (int k = 0; k < P; ++k) h[k] = __ldcg(carry + k);
            }
        }
    }

    float dsum = 0.f;   // sum of Delta over the chunk (Aggregate)
    float dcomp = 0.f;  // its running compensation (fp32 I/O)

#pragma unroll 1
    for (int i = 0; i < nt; ++i) {
        const int s = i % STAGES;
        unsigned char* st = stage_ptr(s);
        mbar_wait(&full_bar[s], static_cast<uint32_t>((i / STAGES) & 1), p.status);

        // Widen this tile's B (and C) rows into per-step fp32 pairs/quads.
        // Steps run fastest over the threads (a warp reads whole 32-byte rows:
        // no bank conflicts).  Within a step row, pair k of sub-lane j sits at
        // k * LANES + j, so that the lanes of a channel read adjacent entries.
        {
            const unsigned char* bsrc = st + Lay::NACT * Lay::ACT_BYTES;
            for (int item = threadIdx.x; item < TS * NQ; item += THREADS) {
                const int t = item % TS;
                const int q = item / TS;
                const int slot = t * NQP + (q % P) * LANES + q / P;
                const unsigned char* b0 = bsrc + (2 * q) * Sh::kRowBytes + t * static_cast<int>(sizeof(T));
                const float B0 = lds_elem<T>(b0);
                const float B1 = lds_elem<T>(b0 + Sh::kRowBytes);
                if constexpr (FULL) {
                    const unsigned char* c0 = b0 + Lay::BC_BYTES;
                    reinterpret_cast<float4*>(bcf)[slot] =
                        make_float4(B0, B1, lds_elem<T>(c0), lds_elem<T>(c0 + Sh::kRowBytes));
                } else {
                    reinterpret_cast<float2*>(bcf)[slot] = make_float2(B0, B1);
                }
            }
        }
        __syncthreads();

        const int t0 = (tb + i) * TS;
        unsigned char* u_t = st;
        const unsigned char* d_t = st + Lay::ACT_BYTES;
        const unsigned char* z_t = st + 2 * Lay::ACT_BYTES;

        // One 16-byte chunk (VPC steps) of this lane's channel row.  MASKED:
        // the tile runs past the sequence end, so steps beyond it get Delta = 0
        // (Abar = 1, no input: the state passes through unchanged).
        auto run_chunk = [&](const int c, auto masked) {
            constexpr bool MASKED = decltype(masked)::value;
            const uint32_t off = swz_act(r, c) + jj * H * static_cast<int>(sizeof(T));
            float uu[H], dt[H], du[H];
            {
                float dv[H];
                lds_row<T, H>(u_t + off, uu);
                lds_row<T, H>(d_t + off, dv);
                if constexpr (PACKED) {
#pragma unroll
                    for (int k = 0; k < H; k += 2) {
                        const float2 v = __fadd2_rn(make_float2(dv[k], dv[k + 1]), make_float2(bias, bias));
                        float2 d2 = softplus2_fast(v);
                        if constexpr (MASKED) {
                            const int t = t0 + c * VPC + jj * H + k;
                            if (t >= p.seqlen) d2.x = 0.f;
                            if (t + 1 >= p.seqlen) d2.y = 0.f;
                        }
                        const float2 u2 = __fmul2_rn(d2, make_float2(uu[k], uu[k + 1]));
                        dt[k] = d2.x; dt[k + 1] = d2.y;
                        du[k] = u2.x; du[k + 1] = u2.y;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < H; ++k) {
                        dt[k] = softplus<ACCURATE>(dv[k] + bias);
                        if constexpr (MASKED) {
                            if (t0 + c * VPC + jj * H + k >= p.seqlen) dt[k] = 0.f;
                        }
                        du[k] = dt[k] * uu[k];
                    }
                }
            }
            // The channel's lanes share (Delta, Delta, Delta u, Delta u) for
            // every step of the chunk through the warp's scratch rows.
            [[maybe_unused]] float4* xrow = nullptr;
            if constexpr (LANES > 1) {
                xrow = reinterpret_cast<float4*>(xs_warp + (c & 1) * Lay::XS_BUF + cw * Lay::XS_STRIDE);
                if (own) {
#pragma unroll
                    for (int k = 0; k < H; ++k) xrow[jj * H + k] = make_float4(dt[k], dt[k], du[k], du[k]);
                }
                __syncwarp();
            }

            [[maybe_unused]] float acc[VPC];
#pragma unroll
            for (int kk = 0; kk < VPC; ++kk) {
                float2 dt2, du2;
                if constexpr (LANES == 1) {
                    dt2 = make_float2(dt[kk], dt[kk]);
                    du2 = make_float2(du[kk], du[kk]);
                } else {
                    const float4 e = xrow[kk];
                    dt2 = make_float2(e.x, e.y);
                    du2 = make_float2(e.z, e.w);
                }
                const int row = c * VPC + kk;
                if constexpr (!FULL) {
                    if constexpr (ACCURATE) {
                        // Compensated (Kahan) sum: P = exp(A * sum Delta) must match
                        // the product of the per-step decays to fp32 accuracy.
                        const float yk = dt2.x - dcomp;
                        const float tk = dsum + yk;
                        dcomp = (tk - dsum) - yk;
                        dsum = tk;
                    } else {
                        dsum += dt2.x;
                    }
                }
                if constexpr (FULL) {
                    const float4* q4 = reinterpret_cast<const float4*>(bcf) + row * NQP + j;
                    float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < P; ++k) {
                        const float4 q = q4[k * LANES];
                        const float2 x = __fmul2_rn(dt2, a2[k]);
                        const float2 abar = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                        const float2 bx = __fmul2_rn(du2, make_float2(q.x, q.y));
                        h[k] = __ffma2_rn(abar, h[k], bx);
                        y2 = __ffma2_rn(make_float2(q.z, q.w), h[k], y2);
                    }
                    acc[kk] = y2.x + y2.y;
                } else {
                    const float2* q2 = reinterpret_cast<const float2*>(bcf) + row * NQP + j;
#pragma unroll
                    for (int k = 0; k < P; ++k) {
                        const float2 bq = q2[k * LANES];
                        const float2 x = __fmul2_rn(dt2, a2[k]);
                        const float2 abar = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                        h[k] = __ffma2_rn(abar, h[k], __fmul2_rn(du2, bq));
                    }
                }
            }

            if constexpr (FULL) {
                if constexpr (SPARE) {
                    // Sum over the lane bits above the chunk's steps, then a
                    // reduce-scatter over the owners' bits.
#pragma unroll
                    for (int m = LANES / 2; m >= VPC; m >>= 1) {
#pragma unroll
                        for (int kk = 0; kk < VPC; ++kk) acc[kk] += __shfl_xor_sync(0xffffffffu, acc[kk], m);
                    }
                    reduce_scatter<VPC, 1>(acc, j);
                } else {
                    reduce_scatter<LANES, H>(acc, j);
                }
                float zz[H];
                if (has_z) lds_row<T, H>(z_t + off, zz);
                float out[H];
                if constexpr (PACKED) {
#pragma unroll
                    for (int k = 0; k < H; k += 2) {
                        float2 y2 = __ffma2_rn(make_float2(dsk, dsk), make_float2(uu[k], uu[k + 1]),
                                               make_float2(acc[k], acc[k + 1]));
                        if (has_z) y2 = __fmul2_rn(y2, silu2_fast(make_float2(zz[k], zz[k + 1])));
                        out[k] = y2.x; out[k + 1] = y2.y;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < H; ++k) {
                        float yv = fmaf(dsk, uu[k], acc[k]);
                        if (has_z) yv *= silu<ACCURATE>(zz[k]);
                        out[k] = yv;
                    }
                }
                if (own) sts_row<T, H>(u_t + off, out);  // y in place of u
            }
        };

        if (t0 + TS <= p.seqlen) {
#pragma unroll
            for (int c = 0; c < Sh::CHUNKS; ++c) run_chunk(c, std::false_type{});
        } else {
#pragma unroll 1
            for (int c = 0; c < Sh::CHUNKS; ++c) run_chunk(c, std::true_type{});
        }

        if constexpr (FULL) fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            if constexpr (FULL) {
                tma_store_3d(&tm_y, t0, dloc0, bg, st);
                bulk_commit();
                // The stage of tile i-1 is free once its y store has read it.
                if (i >= 1 && i - 1 + STAGES < nt) {
                    bulk_wait_read<1>();
                    issue(i - 1 + STAGES);
                }
            } else {
                if (i + STAGES < nt) issue(i + STAGES);
            }
        }
    }
    // Let the kernel that follows in the stream begin launching (it waits for
    // this one's results before it reads them).
    grid_dep_launch();
    if constexpr (FULL) {
        if (threadIdx.x == 0) bulk_wait<0>();
    }

    if (!active) return;
    if constexpr (FULL) {
        if (p.h_final && chunk == p.nchunks - 1) {
            float2* hf = reinterpret_cast<float2*>(p.h_final + bd * N + j * S);
#pragma unroll
            for (int k = 0; k < P; ++k) hf[k] = h[k];
        }
    } else {
        float* agg = p.agg + (static_cast<long long>(chunk) * BD + bd) * (2 * N) + j * S;
        const float2 ds2 = make_float2(dsum, dsum);
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const float2 x = __fmul2_rn(ds2, a2[k]);
            reinterpret_cast<float2*>(agg)[k] = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
            reinterpret_cast<float2*>(agg + N)[k] = h[k];
        }
    }
}

// Carry pass between the summary pass and the full pass.  For every channel
// and state it turns the chunk summaries (P_c, E_c), c = 0..nchunks-2, into
// the state entering each chunk, h_{c+1} = P_c * h_c + E_c from h_0 = h0 (or
// zero), and stores h_{c+1} over E_c.  One thread per (channel, state pair)
// issues the loads of sixteen summaries before their short dependent chain
// of FMAs, so the chain costs one memory latency per sixteen chunks instead
// of one per chunk (and no register array grows with the chunk cap).
template <int N, int MAXC>
__global__ void __launch_bounds__(256)
scan_carry_kernel(float* __restrict__ agg, const float* __restrict__ h0, long long BD, int nchunks) {
    constexpr int NP = N / 2;
    grid_dep_launch();
    grid_dep_wait();  // the summaries of the summary pass
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i >= BD * NP) return;
    const long long bd = i / NP;
    const int k = static_cast<int>(i % NP);
    static_assert(MAXC >= 2, "at least two chunks");
    const int nc = nchunks - 1;
    float2 h = h0 ? __ldg(reinterpret_cast<const float2*>(h0 + bd * N) + k) : make_float2(0.f, 0.f);
    // Blocks of G summaries: all loads of a block in flight before its chain.
    constexpr int G = MAXC - 1 < 16 ? MAXC - 1 : 16;
    for (int c0 = 0; c0 < nc; c0 += G) {
        float2 Pc[G], Ec[G];
#pragma unroll
        for (int q = 0; q < G; ++q) {
            if (c0 + q < nc) {
                const float2* a = reinterpret_cast<const float2*>(agg + ((c0 + q) * BD + bd) * (2 * N));
                Pc[q] = __ldcg(a + k);
                Ec[q] = __ldcg(a + NP + k);
            }
        }
#pragma unroll
        for (int q = 0; q < G; ++q) {
            if (c0 + q < nc) {
                h = __ffma2_rn(Pc[q], h, Ec[q]);
                reinterpret_cast<float2*>(agg + ((c0 + q) * BD + bd) * (2 * N))[NP + k] = h;
            }
        }
    }
}

}  // namespace ssm
