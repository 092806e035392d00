// scan_ws.cuh -- warp-specialised fused selective-scan pass for sm_103a.
//
// The fused forward pass of scan_tma.cuh (softplus step, zero-order-hold
// decay exp(Delta A), input term Delta B u, the diagonal recurrence with the
// state in registers, readout C.h, skip D u, silu(z) gate; eightmm.github.io
// "Mamba", Main Claim and Scan View; intvml.com "DL0170 Mamba Selective SSM
// vs Attention", Mathematical Formulation) over a whole sequence, organised so
// that no thread of the CTA ever waits on the whole CTA inside the time loop:
//
//   * one producer warp issues the TMA loads of every tile (u, delta, z and the
//     group's B, C rows) into a ring of STAGES stages, and widens each landed
//     B/C tile into per-step fp32 (B_n, B_n+1, C_n, C_n+1) quads inside the
//     same stage;
//   * NW consumer warps each own 32 / LANES channels of the CTA.  A consumer
//     warp waits only on the stage it reads (TMA landed, quads ready), runs the
//     recurrence with the state in registers, writes y straight from registers
//     to global memory, and releases the stage.
//
// Stage hand-off uses three mbarriers per stage: `full` (TMA bytes landed),
// `ready` (the producer warp's 32 lanes widened B/C) and `empty` (every
// consumer thread finished reading the stage).  Consumer warps may drift up to
// STAGES tiles apart.  Every wait is bounded in wall time (tma.cuh); a thread
// whose wait gives up records the timeout and leaves its loop, and the
// producer waits for its own loads in flight before it exits.
//
// The library runs this kernel for plans that do not split time (one CTA
// walks the whole sequence of its channels); time-chunked plans use the
// CTA-synchronous passes of scan_tma.cuh.
#pragma once

#include <type_traits>

#include "scan_tma.cuh"
#include "scan_ws_api.h"
#include "ssm_device.cuh"
#include "tma.cuh"

namespace ssm {

// SEG > 1: the time-segmented variant (see the consumer section): a tile row
// is SEG 16-byte chunks, one per time segment.
template <typename T, int N, int LANES, int NW, int STAGES, int SEG = 1>
struct WsLayout {
    static constexpr int RB = SEG == 1 ? kScanRowBytes : 16 * SEG;    // bytes of a row per tile
    static constexpr int TS = RB / static_cast<int>(sizeof(T));       // steps per tile
    static constexpr int CH = NW * 32 / (LANES * SEG);                // channels per CTA
    static constexpr int ACT_BYTES = CH * RB;                         // one activation tile
    static constexpr int BC_BYTES = N * RB;                           // one raw B or C tile
    static constexpr int NACT = 3;                                    // u, delta, z
    static constexpr int NBC = 2;                                     // B, C
    static constexpr int NQP = N / 2 + 1;                             // widened row stride (pairs), one pad
    static constexpr int QBYTES = 16;                                 // bytes of one widened quad
    static constexpr int RAW_BYTES = NACT * ACT_BYTES + NBC * BC_BYTES;
    static constexpr int BCF_OFFSET = (RAW_BYTES + 15) / 16 * 16;     // widened B/C inside the stage
    static constexpr int BCF_BYTES = TS * NQP * QBYTES;
    static constexpr int STAGE_BYTES = (BCF_OFFSET + BCF_BYTES + 1023) / 1024 * 1024;
    // Per consumer warp: two alternating rows (one per 16-byte chunk) of
    // (Delta, Delta, Delta u, Delta u) per step per channel, for LANES > 1.
    static constexpr int VPC = 16 / static_cast<int>(sizeof(T));
    static constexpr int XS_STRIDE = VPC * 16 + 16;
    static constexpr int XS_BUF = (32 / LANES) * XS_STRIDE;  // one row per group of LANES lanes
    static constexpr int XS_BYTES = LANES > 1 ? NW * 2 * XS_BUF : 0;
    static constexpr int XS_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFFSET = XS_OFFSET + XS_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 3 * STAGES * 8 + 1024;  // + alignment slack
    static constexpr int THREADS = (NW + 1) * 32;
    static_assert(ACT_BYTES % (8 * RB) == 0, "activation tiles must keep the swizzle phase");
    static_assert(BC_BYTES % 128 == 0, "B/C tiles must stay 128-byte aligned");
};

// Stores H consecutive elements of a row to global memory (2 to 16 bytes,
// aligned to their size), rounding to T (bf16: nearest even).
template <typename T, int H>
__device__ __forceinline__ void stg_row(T* p, const float (&f)[H]) {
    constexpr int BYTES = H * static_cast<int>(sizeof(T));
    if constexpr (BYTES == 2) {
        const __nv_bfloat16 h = __float2bfloat16_rn(f[0]);
        __stcs(reinterpret_cast<unsigned short*>(p), *reinterpret_cast<const unsigned short*>(&h));
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
            __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
        } else if constexpr (BYTES == 8) {
            __stcs(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
        } else {
            __stcs(reinterpret_cast<unsigned int*>(p), w[0]);
        }
    }
}

// Resident CTAs per SM planned for a variant, passed to __launch_bounds__ so
// that ptxas keeps registers within what that residency leaves: enough CTAs
// for 16 consumer warps per SM (four per scheduler), at most what shared
// memory allows (228 KB, 1 KB reserved per CTA).
template <typename T, int N, int LANES, int NW, int STAGES, int SEG = 1>
constexpr int ws_min_blocks() {
    constexpr int per = WsLayout<T, N, LANES, NW, STAGES, SEG>::SMEM_BYTES + 1024;
    constexpr int by_smem = (228 * 1024) / per;
    constexpr int want = 16 / NW;
    constexpr int b = by_smem < want ? by_smem : want;
    return b < 1 ? 1 : b;
}

template <typename T, int N, int LANES, int NW, int STAGES, bool ACCURATE, int SEG = 1>
__global__ void __launch_bounds__((NW + 1) * 32, (ws_min_blocks<T, N, LANES, NW, STAGES, SEG>()))
scan_ws_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
               const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
               const __grid_constant__ CUtensorMap tm_C, const WsScanParams p) {
    using Lay = WsLayout<T, N, LANES, NW, STAGES, SEG>;
    constexpr int TS = Lay::TS;
    constexpr int VPC = Lay::VPC;             // steps per 16-byte chunk
    constexpr int CHUNKS = Lay::RB / 16;      // 16-byte chunks per tile row
    constexpr int S = N / LANES;              // states per lane
    constexpr int P = S / 2;                  // fp32x2 state pairs per lane
    constexpr int NQ = N / 2;                 // state pairs per step
    constexpr int NQP = Lay::NQP;
    constexpr int H = VPC >= LANES ? VPC / LANES : 1;  // steps a lane owns per chunk
    constexpr bool SPARE = LANES > VPC;                // lanes that own no step of a chunk
    constexpr bool PACKED = !ACCURATE && (H % 2 == 0);
    constexpr int CONSUMERS = NW * 32;
    static_assert(S >= 2 && S % 2 == 0, "each lane holds an even number of states");
    static_assert(SEG == 1 || LANES > 1, "the time-segmented variant shares its scalars through the scratch rows");

    extern __shared__ __align__(16) unsigned char smem_raw[];  // aligned below at run time
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFFSET);
    uint64_t* ready_bar = full_bar + STAGES;
    uint64_t* empty_bar = ready_bar + STAGES;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    const int cb = blockIdx.x % p.blocks_per_group;
    const int bg = blockIdx.x / p.blocks_per_group;  // b * ngroups + g
    const int g = bg % p.ngroups;
    const int b = bg / p.ngroups;
    const int dloc0 = cb * Lay::CH;

    // This CTA's time chunk: tiles [tb, tb + nt).
    const int chunk = blockIdx.y;
    const int tb = static_cast<int>(static_cast<long long>(chunk) * p.ntiles / p.nchunks);
    const int nt = static_cast<int>(static_cast<long long>(chunk + 1) * p.ntiles / p.nchunks) - tb;
    const bool has_z = p.has_z;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&ready_bar[s], 32);
            mbar_init(&empty_bar[s], CONSUMERS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    auto stage_ptr = [&](int s) { return smem + s * Lay::STAGE_BYTES; };

    if (warp == NW) {
        // ------------------------------------------------------------------
        // Producer warp: TMA loads, then B/C widening one tile behind.
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tm_u);
            prefetch_tensormap(&tm_d);
            prefetch_tensormap(&tm_B);
            prefetch_tensormap(&tm_C);
            if (has_z) prefetch_tensormap(&tm_z);
        }
        const uint32_t stage_tx =
            static_cast<uint32_t>((2 + (has_z ? 1 : 0)) * Lay::ACT_BYTES + Lay::NBC * Lay::BC_BYTES);
        int issued = 0;   // tiles whose loads were issued
        int widened = 0;  // tiles widened (their loads have landed)
        bool ok = true;
        // Widens tile i: waits for its bytes, converts the raw B and C rows
        // into per-step fp32 quads, and arrives on its ready barrier.
        auto widen = [&](int i) {
            const int s = i % STAGES;
            unsigned char* st = stage_ptr(s);
            if (!mbar_wait(&full_bar[s], static_cast<uint32_t>((i / STAGES) & 1), p.status, p.wait_budget_ns)) {
                ok = false;  // its consumers give up on the ready barrier in turn
                return;
            }
            const unsigned char* bsrc = st + Lay::NACT * Lay::ACT_BYTES;
            float* bcf = reinterpret_cast<float*>(st + Lay::BCF_OFFSET);
#pragma unroll 2
            for (int item = lane; item < TS * NQ; item += 32) {
                const int t = item % TS;
                const int q = item / TS;
                // Pair q of the step belongs to sub-lane q / P (slot k = q % P):
                // the lanes of a channel read adjacent entries.
                const int slot = t * NQP + (q % P) * LANES + q / P;
                const unsigned char* b0 = bsrc + (2 * q) * Lay::RB + t * static_cast<int>(sizeof(T));
                const unsigned char* c0 = b0 + Lay::BC_BYTES;
                reinterpret_cast<float4*>(bcf)[slot] =
                    make_float4(lds_elem<T>(b0), lds_elem<T>(b0 + Lay::RB), lds_elem<T>(c0), lds_elem<T>(c0 + Lay::RB));
            }
            mbar_arrive(&ready_bar[s]);
            widened = i + 1;
        };
#pragma unroll 1
        for (int k = 0; k < nt && ok; ++k) {
            if (k == p.stop_tile) break;  // failure injection: no load for this tile or any later one
            const int s = k % STAGES;
            if (k >= STAGES) {
                // Tile k - STAGES's consumers are done with this stage.
                if (!mbar_wait(&empty_bar[s], static_cast<uint32_t>(((k / STAGES) - 1) & 1), p.status, p.wait_budget_ns)) {
                    ok = false;
                    break;
                }
            }
            if (lane == 0) {
                unsigned char* st = stage_ptr(s);
                const int x = (tb + k) * TS;
                mbar_arrive_expect_tx(&full_bar[s], stage_tx);
                tma_load_3d(st, &tm_u, x, dloc0, bg, &full_bar[s]);
                tma_load_3d(st + Lay::ACT_BYTES, &tm_d, x, dloc0, bg, &full_bar[s]);
                if (has_z) tma_load_3d(st + 2 * Lay::ACT_BYTES, &tm_z, x, dloc0, bg, &full_bar[s]);
                unsigned char* bc = st + Lay::NACT * Lay::ACT_BYTES;
                tma_load_2d(bc, &tm_B, x, bg * N, &full_bar[s]);
                tma_load_2d(bc + Lay::BC_BYTES, &tm_C, x, bg * N, &full_bar[s]);
            }
            __syncwarp();
            issued = k + 1;
            if (k >= 1) widen(k - 1);
        }
        if (ok && widened < issued) widen(issued - 1);
        // Loads still in flight (a wait gave up): wait for them before the CTA
        // may exit, so that no copy lands in shared memory it no longer owns.
        for (int i = widened; i < issued; ++i) {
            mbar_wait(&full_bar[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.status, p.wait_budget_ns);
        }
        return;
    }

    // ----------------------------------------------------------------------
    // Consumer warps, time-segmented variant (SEG > 1): the warp's lanes are
    // (channel, segment, sub-lane) triples.  A tile row holds SEG 16-byte
    // chunks of time; the LANES lanes of segment j work on chunk j.  Each
    // segment first runs the recurrence from a zero state over its chunk
    // (the summary pair (P, E): P = exp(A * sum Delta), E = end state), then
    // the SEG pairs of a channel are combined by a warp-shuffle scan over
    // (Abar, Bbar x) pairs -- (P1, E1) then (P2, E2) gives (P2 P1, P2 E1 + E2)
    // (eightmm.github.io "Mamba", Scan View) -- into the state entering each
    // segment, and each segment runs the recurrence again from that state with
    // the readout.  Every decay is computed twice; the per-step scalars once.
    // ----------------------------------------------------------------------
    if constexpr (SEG > 1) {
        constexpr int CPW = 32 / (LANES * SEG);           // channels per warp
        const int j = lane % LANES;                       // sub-lane within the channel
        const int seg = (lane / LANES) % SEG;             // time segment = chunk of the tile
        const int cw = lane / (LANES * SEG);              // channel within the warp
        const int grp = lane / LANES;                     // (channel, segment) group
        const int r = warp * CPW + cw;                    // channel row within the CTA
        const int jj = SPARE ? j % VPC : j;
        const bool own = !SPARE || j < VPC;
        unsigned char* xs_warp = smem + Lay::XS_OFFSET + warp * 2 * Lay::XS_BUF;
        const int last_src = cw * LANES * SEG + (SEG - 1) * LANES + j;  // lane of the last segment

        const int dloc = dloc0 + r;
        const bool active = dloc < p.dim_per_group;
        const int d = g * p.dim_per_group + (active ? dloc : 0);
        const long long bd = static_cast<long long>(b) * p.dim + d;

        float2 a2[P], hc[P];  // decay constants; state entering the tile
        {
            const float* Ad = p.A + static_cast<long long>(d) * N + j * S;
#pragma unroll
            for (int k = 0; k < P; ++k) {
                const float2 av = __ldg(reinterpret_cast<const float2*>(Ad) + k);
                a2[k] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
                hc[k] = make_float2(0.f, 0.f);
            }
            if (p.h0 && active) {
                const float2* h0v = reinterpret_cast<const float2*>(p.h0 + bd * N + j * S);
#pragma unroll
                for (int k = 0; k < P; ++k) hc[k] = __ldg(h0v + k);
            }
        }
        const float bias = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
        const float dsk = p.D ? __ldg(p.D + d) : 0.f;
        T* yrow = static_cast<T*>(p.y) + bd * p.seqlen;

#pragma unroll 1
        for (int i = 0; i < nt; ++i) {
            const int s = i % STAGES;
            const uint32_t par = static_cast<uint32_t>((i / STAGES) & 1);
            if (!mbar_wait(&full_bar[s], par, p.status, p.wait_budget_ns) ||
                !mbar_wait(&ready_bar[s], par, p.status, p.wait_budget_ns))
                break;
            const unsigned char* st = stage_ptr(s);
            const float* bcf = reinterpret_cast<const float*>(st + Lay::BCF_OFFSET);
            const int c = seg;
            const int tl = i * TS + c * VPC + jj * H;  // first step of this lane's share
            const uint32_t off = swz_rows<Lay::RB>(r, c) + jj * H * static_cast<int>(sizeof(T));

            // Per-step scalars of the lane's share of its chunk, shared with the
            // other lanes of the (channel, segment) group through the scratch row.
            float uu[H], dt[H], du[H];
            {
                float dv[H];
                lds_row<T, H>(st + off, uu);
                lds_row<T, H>(st + Lay::ACT_BYTES + off, dv);
#pragma unroll
                for (int k = 0; k < H; ++k) {
                    dt[k] = softplus<ACCURATE>(dv[k] + bias);
                    if (tl + k >= p.seqlen) dt[k] = 0.f;  // past the end: Abar = 1, no input
                    du[k] = dt[k] * uu[k];
                }
            }
            float4* xrow = reinterpret_cast<float4*>(xs_warp + (i & 1) * Lay::XS_BUF + grp * Lay::XS_STRIDE);
            if (own) {
#pragma unroll
                for (int k = 0; k < H; ++k) xrow[jj * H + k] = make_float4(dt[k], dt[k], du[k], du[k]);
            }
            __syncwarp();

            // Walk 1: the segment's summary from a zero state.
            float2 pe[P], ee[P];
            {
                float dsum = 0.f, dcomp = 0.f;
#pragma unroll
                for (int k = 0; k < P; ++k) ee[k] = make_float2(0.f, 0.f);
                // Two steps at a time: unrolled further, ptxas hoists the decays
                // of every step (nothing else paces them) and spills.
#pragma unroll 2
                for (int kk = 0; kk < VPC; ++kk) {
                    const float4 e = xrow[kk];
                    const float2 dt2 = make_float2(e.x, e.y), du2 = make_float2(e.z, e.w);
                    if constexpr (ACCURATE) {
                        const float yk = e.x - dcomp;
                        const float tk = dsum + yk;
                        dcomp = (tk - dsum) - yk;
                        dsum = tk;
                    } else {
                        dsum += e.x;
                    }
                    const float4* q4 = reinterpret_cast<const float4*>(bcf) + (c * VPC + kk) * NQP + j;
#pragma unroll
                    for (int k = 0; k < P; ++k) {
                        const float4 q = q4[k * LANES];
                        const float2 x = __fmul2_rn(dt2, a2[k]);
                        const float2 abar = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                        ee[k] = __ffma2_rn(abar, ee[k], __fmul2_rn(du2, make_float2(q.x, q.y)));
                    }
                }
                const float2 ds2 = make_float2(dsum, dsum);
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const float2 x = __fmul2_rn(ds2, a2[k]);
                    pe[k] = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                }
            }
            // Inclusive scan of the summaries over the channel's segments.
#pragma unroll
            for (int o = 1; o < SEG; o <<= 1) {
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const float px = __shfl_up_sync(0xffffffffu, pe[k].x, o * LANES);
                    const float py = __shfl_up_sync(0xffffffffu, pe[k].y, o * LANES);
                    const float ex = __shfl_up_sync(0xffffffffu, ee[k].x, o * LANES);
                    const float ey = __shfl_up_sync(0xffffffffu, ee[k].y, o * LANES);
                    if (seg >= o) {
                        ee[k] = __ffma2_rn(pe[k], make_float2(ex, ey), ee[k]);
                        pe[k] = __fmul2_rn(pe[k], make_float2(px, py));
                    }
                }
            }
            // State entering this segment: the tile's incoming state through
            // the segments before it.
            float2 h[P];
#pragma unroll
            for (int k = 0; k < P; ++k) {
                const float px = __shfl_up_sync(0xffffffffu, pe[k].x, LANES);
                const float py = __shfl_up_sync(0xffffffffu, pe[k].y, LANES);
                const float ex = __shfl_up_sync(0xffffffffu, ee[k].x, LANES);
                const float ey = __shfl_up_sync(0xffffffffu, ee[k].y, LANES);
                h[k] = seg == 0 ? hc[k] : __ffma2_rn(make_float2(px, py), hc[k], make_float2(ex, ey));
            }
            // Walk 2: the recurrence from that state, with the readout.  The
            // decays are evaluated again rather than kept from walk 1 (holding
            // them would need a register per step and state).
            float acc[VPC];
#pragma unroll
            for (int kk = 0; kk < VPC; ++kk) {
                const float4 e = xrow[kk];
                const float2 dt2 = make_float2(e.x, e.y), du2 = make_float2(e.z, e.w);
                const float4* q4 = reinterpret_cast<const float4*>(bcf) + (c * VPC + kk) * NQP + j;
                float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const float4 q = q4[k * LANES];
                    const float2 x = __fmul2_rn(dt2, a2[k]);
                    const float2 abar = make_float2(decay_again<ACCURATE>(x.x), decay_again<ACCURATE>(x.y));
                    h[k] = __ffma2_rn(du2, make_float2(q.x, q.y), __fmul2_rn(abar, h[k]));
                    y2 = __ffma2_rn(make_float2(q.z, q.w), h[k], y2);
                }
                acc[kk] = y2.x + y2.y;
            }
            // The next tile starts from the last segment's end state.
#pragma unroll
            for (int k = 0; k < P; ++k) {
                hc[k].x = __shfl_sync(0xffffffffu, h[k].x, last_src);
                hc[k].y = __shfl_sync(0xffffffffu, h[k].y, last_src);
            }
            // Readout summed over the group's lanes, skip term, gate, store.
            if constexpr (SPARE) {
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
            if (has_z) lds_row<T, H>(st + 2 * Lay::ACT_BYTES + off, zz);
            float out[H];
#pragma unroll
            for (int k = 0; k < H; ++k) {
                float yv = fmaf(dsk, uu[k], acc[k]);
                if (has_z) yv *= silu<ACCURATE>(zz[k]);
                out[k] = yv;
            }
            if (own && active) {
                if (tl + H <= p.seqlen) {
                    stg_row<T, H>(yrow + tl, out);
                } else {
#pragma unroll
                    for (int k = 0; k < H; ++k)
                        if (tl + k < p.seqlen) Elem<T>::store(yrow + tl + k, out[k]);
                }
            }
            mbar_arrive(&empty_bar[s]);
        }
        if (active && p.h_final && seg == 0) {
            float2* hf = reinterpret_cast<float2*>(p.h_final + bd * N + j * S);
#pragma unroll
            for (int k = 0; k < P; ++k) hf[k] = hc[k];
        }
    } else {
        const int r = warp * (32 / LANES) + lane / LANES;  // channel row within the CTA
        const int j = lane % LANES;                        // sub-lane within the channel
        const int jj = SPARE ? j % VPC : j;                // its step slot in a chunk
        const bool own = !SPARE || j < VPC;                // it owns steps
        const int cw = lane / LANES;                       // channel within the warp
        unsigned char* xs_warp = smem + Lay::XS_OFFSET + warp * 2 * Lay::XS_BUF;

        const int dloc = dloc0 + r;
        const bool active = dloc < p.dim_per_group;
        const int d = g * p.dim_per_group + (active ? dloc : 0);
        const long long bd = static_cast<long long>(b) * p.dim + d;

        float2 a2[P], h[P];
        {
            const float* Ad = p.A + static_cast<long long>(d) * N + j * S;
#pragma unroll
            for (int k = 0; k < P; ++k) {
                const float2 av = __ldg(reinterpret_cast<const float2*>(Ad) + k);
                a2[k] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
                h[k] = make_float2(0.f, 0.f);
            }
            if (chunk > 0) {
                // The carry pass wrote the state entering this chunk; this
                // kernel may have started before it finished.
                grid_dep_wait();
                if (active) {
                    const long long BD = static_cast<long long>(p.batch) * p.dim;
                    const float2* cv = reinterpret_cast<const float2*>(
                        p.carry + (static_cast<long long>(chunk - 1) * BD + bd) * (2 * N) + N + j * S);
#pragma unroll
                    for (int k = 0; k < P; ++k) h[k] = __ldcg(cv + k);
                }
            } else if (p.h0 && active) {
                const float2* h0v = reinterpret_cast<const float2*>(p.h0 + bd * N + j * S);
#pragma unroll
                for (int k = 0; k < P; ++k) h[k] = __ldg(h0v + k);
            }
        }
        const float bias = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
        const float dsk = p.D ? __ldg(p.D + d) : 0.f;
        T* yrow = static_cast<T*>(p.y) + bd * p.seqlen;

#pragma unroll 1
        for (int i = 0; i < nt; ++i) {
            const int s = i % STAGES;
            const uint32_t par = static_cast<uint32_t>((i / STAGES) & 1);
            if (!mbar_wait(&full_bar[s], par, p.status, p.wait_budget_ns) ||
                !mbar_wait(&ready_bar[s], par, p.status, p.wait_budget_ns))
                break;
            const unsigned char* st = stage_ptr(s);
            const unsigned char* u_t = st;
            const unsigned char* d_t = st + Lay::ACT_BYTES;
            const unsigned char* z_t = st + 2 * Lay::ACT_BYTES;
            const float* bcf = reinterpret_cast<const float*>(st + Lay::BCF_OFFSET);
            const int t0 = (tb + i) * TS;

            // One 16-byte chunk (VPC steps) of this lane's channel row.  MASKED:
            // the tile runs past the sequence end, so steps beyond it get Delta = 0
            // (Abar = 1, no input: the state passes through unchanged).
            auto run_chunk = [&](const int c, auto masked) {
                constexpr bool MASKED = decltype(masked)::value;
                const uint32_t off = swz_rows<Lay::RB>(r, c) + jj * H * static_cast<int>(sizeof(T));
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

                float acc[VPC];
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
                }
                if constexpr (LANES > 1) __syncwarp();  // the scratch row is rewritten two chunks on

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
                const int tl = t0 + c * VPC + jj * H;  // first step of this lane's share
                if (own && active) {
                    if constexpr (MASKED) {
#pragma unroll
                        for (int k = 0; k < H; ++k)
                            if (tl + k < p.seqlen) Elem<T>::store(yrow + tl + k, out[k]);
                    } else {
                        stg_row<T, H>(yrow + tl, out);
                    }
                }
            };

            if (t0 + TS <= p.seqlen) {
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c) run_chunk(c, std::false_type{});
            } else {
#pragma unroll 1
                for (int c = 0; c < CHUNKS; ++c) run_chunk(c, std::true_type{});
            }
            mbar_arrive(&empty_bar[s]);
        }

        if (!active) return;
        if (p.h_final && chunk == p.nchunks - 1) {
            float2* hf = reinterpret_cast<float2*>(p.h_final + bd * N + j * S);
#pragma unroll
            for (int k = 0; k < P; ++k) hf[k] = h[k];
        }
    }
}

}  // namespace ssm
