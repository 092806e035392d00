// decode_tma.cuh -- TMA-staged single-token decode step (N = 16).
//
// Same arithmetic as state_update.cuh (inference runs the recurrence one token
// at a time on a state of constant size: cuishuaiwen.com "Mamba &
// State-Space Sequence Models", Core mechanics), laid out so that one thread
// owns one (sequence, channel) with all 16 states:
//
//   * the work is a list of tiles, one tile = one sequence b x CH = 128
//     consecutive channels of one group; a persistent grid gives every CTA a
//     contiguous run of tiles (channel-block major, so A / dt_bias / D rows
//     are reloaded only when the block changes);
//   * per tile, TMA brings the 8 KB state block ([128 rows x 64 B], 64-byte
//     swizzle so that each thread's four 16-byte reads hit distinct banks),
//     the 128 u / delta / z values and the B and C rows into one stage of a
//     4-stage mbarrier ring;
//   * each thread updates its 16 states as fp32x2 pairs, writes them back in
//     place, and the block leaves by a TMA store that clips at the channel
//     edge; y goes out as a coalesced store.
// One softplus, one gate and 16 decays per (b, d): no work is repeated across
// lanes, and the state moves at full HBM width without holding loads in
// registers.
#pragma once

#include "scan_tma.cuh"  // lds_elem
#include "ssm_device.cuh"
#include "state_update.cuh"
#include "tma.cuh"

namespace ssm {

template <typename T, int CH_ = 128, int STAGES_ = 4>
struct DecodeTmaLayout {
    static constexpr int N = 16;
    static constexpr int CH = CH_;                                    // channels per tile = threads
    static constexpr int STATE_BYTES = CH * N * 4;                    // [CH rows x 64 B]
    static constexpr int TOK_BYTES = (CH * static_cast<int>(sizeof(T)) + 127) / 128 * 128;
    static constexpr int BC_BYTES = 128;                              // one row of N elements, padded
    static constexpr int OFF_U = STATE_BYTES;
    static constexpr int OFF_D = OFF_U + TOK_BYTES;
    static constexpr int OFF_Z = OFF_D + TOK_BYTES;
    static constexpr int OFF_B = OFF_Z + TOK_BYTES;
    static constexpr int OFF_C = OFF_B + BC_BYTES;
    static constexpr int STAGE_BYTES = (OFF_C + BC_BYTES + 1023) / 1024 * 1024;
    static constexpr int STAGES = STAGES_;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGES * 8 + 1024;
};

struct DecodeTmaParams {
    const float* A;
    const float* D;        // nullable
    const float* dt_bias;  // nullable
    void* y;
    int batch, dim, ngroups, dim_per_group;
    int nblk;              // channel blocks per sequence
    long long ntiles;      // batch * nblk
    int has_z;
    const int* slots;      // nullable: row b uses state slot slots[b] (outside [0, nslots): padding)
    int nslots;
};

template <typename T, int CH_, int STAGES_, bool ACCURATE>
__global__ void __launch_bounds__(CH_)
decode_tma_kernel(const __grid_constant__ CUtensorMap tm_state, const __grid_constant__ CUtensorMap tm_u,
                  const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_z,
                  const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
                  const DecodeTmaParams p) {
    using Lay = DecodeTmaLayout<T, CH_, STAGES_>;
    constexpr int N = Lay::N;
    constexpr int CH = Lay::CH;
    constexpr int STAGES = Lay::STAGES;
    constexpr int P = N / 2;

    extern __shared__ __align__(16) unsigned char smem_raw[];  // aligned below at run time
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * Lay::STAGE_BYTES);

    // This CTA's contiguous run of tiles; tile t = cb * batch + b.
    const long long t_begin = p.ntiles * blockIdx.x / gridDim.x;
    const long long t_end = p.ntiles * (blockIdx.x + 1) / gridDim.x;
    const int nt = static_cast<int>(t_end - t_begin);
    const bool has_z = p.has_z != 0;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_state);
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_d);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        if (has_z) prefetch_tensormap(&tm_z);
    }
    __syncthreads();

    const uint32_t tx = static_cast<uint32_t>(Lay::STATE_BYTES + (2 + (has_z ? 1 : 0)) * CH * sizeof(T) +
                                              2 * N * sizeof(T));
    auto tile_of = [&](int k, int& b, int& cb) {
        const long long t = t_begin + k;
        cb = static_cast<int>(t / p.batch);
        b = static_cast<int>(t % p.batch);
    };
    // State slot of batch row b: b itself, or the caller's slot; -1 for a
    // padding row (an index outside [0, nslots)), which loads slot 0, computes
    // on it and stores nothing.
    auto slot_of = [&](int b) {
        const int sl = p.slots ? __ldg(p.slots + b) : b;
        return sl >= 0 && sl < p.nslots ? sl : -1;
    };
    auto issue = [&](int k) {  // thread 0 only
        int b, cb;
        tile_of(k, b, cb);
        const int s = k % STAGES;
        unsigned char* st = smem + s * Lay::STAGE_BYTES;
        const int d0 = cb * CH;
        const int g = d0 / p.dim_per_group;
        mbar_arrive_expect_tx(&full_bar[s], tx);
        tma_load_3d(st, &tm_state, 0, d0, max(slot_of(b), 0), &full_bar[s]);
        tma_load_2d(st + Lay::OFF_U, &tm_u, d0, b, &full_bar[s]);
        tma_load_2d(st + Lay::OFF_D, &tm_d, d0, b, &full_bar[s]);
        if (has_z) tma_load_2d(st + Lay::OFF_Z, &tm_z, d0, b, &full_bar[s]);
        tma_load_2d(st + Lay::OFF_B, &tm_B, 0, b * p.ngroups + g, &full_bar[s]);
        tma_load_2d(st + Lay::OFF_C, &tm_C, 0, b * p.ngroups + g, &full_bar[s]);
    };
    if (threadIdx.x == 0) {
        for (int k = 0; k < STAGES && k < nt; ++k) issue(k);
    }

    const int c = threadIdx.x;
    int cur_cb = -1;
    float2 a2[P];
    float bias = 0.f, dsk = 0.f;
    bool active = false;
    int d = 0;
    T* __restrict__ yp = static_cast<T*>(p.y);

#pragma unroll 1
    for (int k = 0; k < nt; ++k) {
        int b, cb;
        tile_of(k, b, cb);
        if (cb != cur_cb) {  // uniform over the CTA
            cur_cb = cb;
            d = cb * CH + c;
            active = d < p.dim;
            const int dc = active ? d : p.dim - 1;
            const float4* Ad = reinterpret_cast<const float4*>(p.A + static_cast<long long>(dc) * N);
#pragma unroll
            for (int q = 0; q < N / 4; ++q) {
                const float4 av = __ldg(Ad + q);
                a2[2 * q] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
                a2[2 * q + 1] = make_float2(av.z * decay_scale<ACCURATE>(), av.w * decay_scale<ACCURATE>());
            }
            bias = p.dt_bias ? __ldg(p.dt_bias + dc) : 0.f;
            dsk = p.D ? __ldg(p.D + dc) : 0.f;
        }
        const int s = k % STAGES;
        unsigned char* st = smem + s * Lay::STAGE_BYTES;
        mbar_wait(&full_bar[s], static_cast<uint32_t>((k / STAGES) & 1), nullptr);

        // B and C rows of this tile's (sequence, group): read by every thread.
        float2 bq[P], cq[P];
        {
            const T* Bs = reinterpret_cast<const T*>(st + Lay::OFF_B);
            const T* Cs = reinterpret_cast<const T*>(st + Lay::OFF_C);
            if constexpr (sizeof(T) == 4) {
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    bq[q] = reinterpret_cast<const float2*>(Bs)[q];
                    cq[q] = reinterpret_cast<const float2*>(Cs)[q];
                }
            } else {
#pragma unroll
                for (int q = 0; q < P / 4; ++q) {
                    const uint4 bw = reinterpret_cast<const uint4*>(Bs)[q];
                    const uint4 cw = reinterpret_cast<const uint4*>(Cs)[q];
                    const uint32_t bv[4] = {bw.x, bw.y, bw.z, bw.w};
                    const uint32_t cv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        bq[4 * q + r] = make_float2(__uint_as_float(bv[r] << 16), __uint_as_float(bv[r] & 0xffff0000u));
                        cq[4 * q + r] = make_float2(__uint_as_float(cv[r] << 16), __uint_as_float(cv[r] & 0xffff0000u));
                    }
                }
            }
        }
        const float uv = lds_elem<T>(st + Lay::OFF_U + c * sizeof(T));
        const float dv = lds_elem<T>(st + Lay::OFF_D + c * sizeof(T));
        const float dt = softplus<ACCURATE>(dv + bias);
        const float du = dt * uv;
        const float2 dt2 = make_float2(dt, dt);
        const float2 du2 = make_float2(du, du);

        float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            float4* hp = reinterpret_cast<float4*>(st + swz64(c, q));
            const float4 hv = *hp;
            float2 h0 = make_float2(hv.x, hv.y), h1 = make_float2(hv.z, hv.w);
            {
                const float2 x = __fmul2_rn(dt2, a2[2 * q]);
                const float2 ab = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                h0 = __ffma2_rn(ab, h0, __fmul2_rn(du2, bq[2 * q]));
                y2 = __ffma2_rn(cq[2 * q], h0, y2);
            }
            {
                const float2 x = __fmul2_rn(dt2, a2[2 * q + 1]);
                const float2 ab = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                h1 = __ffma2_rn(ab, h1, __fmul2_rn(du2, bq[2 * q + 1]));
                y2 = __ffma2_rn(cq[2 * q + 1], h1, y2);
            }
            *hp = make_float4(h0.x, h0.y, h1.x, h1.y);
        }
        const int slot = slot_of(b);
        if (active && slot >= 0) {
            float yv = fmaf(dsk, uv, y2.x + y2.y);
            if (has_z) yv *= silu<ACCURATE>(lds_elem<T>(st + Lay::OFF_Z + c * sizeof(T)));
            Elem<T>::store(yp + static_cast<long long>(b) * p.dim + d, yv);
        }

        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            // One bulk group per tile (empty for a padding row), so that
            // waiting for all but the newest covers the previous tile's store.
            if (slot >= 0) tma_store_3d(&tm_state, 0, cb * CH, slot, st);
            bulk_commit();
            if (k >= 1 && k - 1 + STAGES < nt) {
                bulk_wait_read<1>();
                issue(k - 1 + STAGES);
            }
        }
    }
    if (threadIdx.x == 0) bulk_wait<0>();
}


// Warp-specialised variant of the same step: CH / 32 consumer warps and one
// producer warp.  The producer issues each tile's TMA loads into a ring of
// stages (full barrier per stage) once the stage is empty; each consumer warp
// updates its 32 channels' states in place and sends its own 32 rows back by
// a TMA store (box of 32 rows), then releases the previous tile's stage on
// the empty barrier once that store has read it.  No CTA-wide barrier is left
// in the tile loop.
template <typename T, int CH_, int STAGES_>
struct DecodeWsLayout {
    using Base = DecodeTmaLayout<T, CH_, STAGES_>;
    static constexpr int STAGES = STAGES_;
    static constexpr int BAR_OFF = STAGES * Base::STAGE_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + 2 * STAGES * 8 + 1024;
};

template <typename T, int CH_, int STAGES_, bool ACCURATE>
__global__ void __launch_bounds__(CH_ + 32)
decode_ws_kernel(const __grid_constant__ CUtensorMap tm_state, const __grid_constant__ CUtensorMap tm_state_out,
                 const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
                 const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
                 const __grid_constant__ CUtensorMap tm_C, const DecodeTmaParams p) {
    using Lay = DecodeTmaLayout<T, CH_, STAGES_>;
    using WLay = DecodeWsLayout<T, CH_, STAGES_>;
    constexpr int N = Lay::N;
    constexpr int CH = Lay::CH;
    constexpr int STAGES = Lay::STAGES;
    constexpr int P = N / 2;
    constexpr int CW = CH / 32;  // consumer warps

    extern __shared__ __align__(16) unsigned char smem_raw[];  // aligned below at run time
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + WLay::BAR_OFF);
    uint64_t* empty_bar = full_bar + STAGES;

    const long long t_begin = p.ntiles * blockIdx.x / gridDim.x;
    const long long t_end = p.ntiles * (blockIdx.x + 1) / gridDim.x;
    const int nt = static_cast<int>(t_end - t_begin);
    const bool has_z = p.has_z != 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Programmatic dependent launch: the next kernel in the stream may start
    // its launch now (it waits in turn before touching memory), and this one
    // waits for the previous kernel's writes before its first global access,
    // so that launch and prologue overlap the previous step's tail.
    grid_dep_launch();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_wait();

    auto tile_of = [&](int k, int& b, int& cb) {
        const long long t = t_begin + k;
        cb = static_cast<int>(t / p.batch);
        b = static_cast<int>(t % p.batch);
    };
    auto slot_of = [&](int b) {
        const int sl = p.slots ? __ldg(p.slots + b) : b;
        return sl >= 0 && sl < p.nslots ? sl : -1;
    };

    if (warp == CW) {
        // ---- producer ----
        if (lane == 0) {
            prefetch_tensormap(&tm_state);
            prefetch_tensormap(&tm_state_out);
            prefetch_tensormap(&tm_u);
            prefetch_tensormap(&tm_d);
            prefetch_tensormap(&tm_B);
            prefetch_tensormap(&tm_C);
            if (has_z) prefetch_tensormap(&tm_z);
            const uint32_t tx = static_cast<uint32_t>(Lay::STATE_BYTES + (2 + (has_z ? 1 : 0)) * CH * sizeof(T) +
                                                      2 * N * sizeof(T));
            for (int k = 0; k < nt; ++k) {
                const int s = k % STAGES;
                if (k >= STAGES) mbar_wait(&empty_bar[s], static_cast<uint32_t>((k / STAGES - 1) & 1), nullptr);
                int b, cb;
                tile_of(k, b, cb);
                unsigned char* st = smem + s * Lay::STAGE_BYTES;
                const int d0 = cb * CH;
                const int g = d0 / p.dim_per_group;
                mbar_arrive_expect_tx(&full_bar[s], tx);
                tma_load_3d(st, &tm_state, 0, d0, max(slot_of(b), 0), &full_bar[s]);
                tma_load_2d(st + Lay::OFF_U, &tm_u, d0, b, &full_bar[s]);
                tma_load_2d(st + Lay::OFF_D, &tm_d, d0, b, &full_bar[s]);
                if (has_z) tma_load_2d(st + Lay::OFF_Z, &tm_z, d0, b, &full_bar[s]);
                tma_load_2d(st + Lay::OFF_B, &tm_B, 0, b * p.ngroups + g, &full_bar[s]);
                tma_load_2d(st + Lay::OFF_C, &tm_C, 0, b * p.ngroups + g, &full_bar[s]);
            }
        }
        return;
    }

    // ---- consumers: thread c owns channel cb * CH + c of the tile ----
    const int c = threadIdx.x;
    int cur_cb = -1;
    float2 a2[P];
    float bias = 0.f, dsk = 0.f;
    bool active = false;
    int d = 0;
    T* __restrict__ yp = static_cast<T*>(p.y);

#pragma unroll 1
    for (int k = 0; k < nt; ++k) {
        int b, cb;
        tile_of(k, b, cb);
        if (cb != cur_cb) {
            cur_cb = cb;
            d = cb * CH + c;
            active = d < p.dim;
            const int dc = active ? d : p.dim - 1;
            const float4* Ad = reinterpret_cast<const float4*>(p.A + static_cast<long long>(dc) * N);
#pragma unroll
            for (int q = 0; q < N / 4; ++q) {
                const float4 av = __ldg(Ad + q);
                a2[2 * q] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
                a2[2 * q + 1] = make_float2(av.z * decay_scale<ACCURATE>(), av.w * decay_scale<ACCURATE>());
            }
            bias = p.dt_bias ? __ldg(p.dt_bias + dc) : 0.f;
            dsk = p.D ? __ldg(p.D + dc) : 0.f;
        }
        const int s = k % STAGES;
        unsigned char* st = smem + s * Lay::STAGE_BYTES;
        mbar_wait(&full_bar[s], static_cast<uint32_t>((k / STAGES) & 1), nullptr);

        float2 bq[P], cq[P];
        {
            const T* Bs = reinterpret_cast<const T*>(st + Lay::OFF_B);
            const T* Cs = reinterpret_cast<const T*>(st + Lay::OFF_C);
            if constexpr (sizeof(T) == 4) {
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    bq[q] = reinterpret_cast<const float2*>(Bs)[q];
                    cq[q] = reinterpret_cast<const float2*>(Cs)[q];
                }
            } else {
#pragma unroll
                for (int q = 0; q < P / 4; ++q) {
                    const uint4 bw = reinterpret_cast<const uint4*>(Bs)[q];
                    const uint4 cw = reinterpret_cast<const uint4*>(Cs)[q];
                    const uint32_t bv[4] = {bw.x, bw.y, bw.z, bw.w};
                    const uint32_t cv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        bq[4 * q + r] = make_float2(__uint_as_float(bv[r] << 16), __uint_as_float(bv[r] & 0xffff0000u));
                        cq[4 * q + r] = make_float2(__uint_as_float(cv[r] << 16), __uint_as_float(cv[r] & 0xffff0000u));
                    }
                }
            }
        }
        const float uv = lds_elem<T>(st + Lay::OFF_U + c * sizeof(T));
        const float dv = lds_elem<T>(st + Lay::OFF_D + c * sizeof(T));
        const float dt = softplus<ACCURATE>(dv + bias);
        const float du = dt * uv;
        const float2 dt2 = make_float2(dt, dt);
        const float2 du2 = make_float2(du, du);

        float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            float4* hp = reinterpret_cast<float4*>(st + swz64(c, q));
            const float4 hv = *hp;
            float2 h0 = make_float2(hv.x, hv.y), h1 = make_float2(hv.z, hv.w);
            {
                const float2 x = __fmul2_rn(dt2, a2[2 * q]);
                const float2 ab = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                h0 = __ffma2_rn(ab, h0, __fmul2_rn(du2, bq[2 * q]));
                y2 = __ffma2_rn(cq[2 * q], h0, y2);
            }
            {
                const float2 x = __fmul2_rn(dt2, a2[2 * q + 1]);
                const float2 ab = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                h1 = __ffma2_rn(ab, h1, __fmul2_rn(du2, bq[2 * q + 1]));
                y2 = __ffma2_rn(cq[2 * q + 1], h1, y2);
            }
            *hp = make_float4(h0.x, h0.y, h1.x, h1.y);
        }
        const int slot = slot_of(b);
        if (active && slot >= 0) {
            float yv = fmaf(dsk, uv, y2.x + y2.y);
            if (has_z) yv *= silu<ACCURATE>(lds_elem<T>(st + Lay::OFF_Z + c * sizeof(T)));
            Elem<T>::store(yp + static_cast<long long>(b) * p.dim + d, yv);
        }

        // This warp's 32 rows leave by their own store; the previous tile's
        // stage is released once this warp's store from it has read it.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // One bulk group per tile (empty for a padding row).
            if (slot >= 0) tma_store_3d(&tm_state_out, 0, cb * CH + warp * 32, slot, st + warp * 32 * N * 4);
            bulk_commit();
            if (k >= 1) {
                bulk_wait_read<1>();
                mbar_arrive(&empty_bar[(k - 1) % STAGES]);
            }
        }
        __syncwarp();
    }
    if (lane == 0) bulk_wait<0>();
}

}  // namespace ssm
