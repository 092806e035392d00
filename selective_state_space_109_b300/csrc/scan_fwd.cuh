// scan_fwd.cuh -- fused selective-scan forward kernel for sm_103a.
//
// One kernel does the whole path for a block of channels over time:
// softplus step -> zero-order-hold decay exp(Delta A) -> input term
// Delta B u -> diagonal recurrence h = Abar h + Bbar x -> readout C.h ->
// skip D u -> silu(z) gate -> y.  The state never leaves registers.
// (Recurrence and readout: eightmm.github.io "Mamba", Main Claim / Scan
// View; discretisation: intvml.com "DL0170 Mamba Selective SSM vs
// Attention", Mathematical Formulation; the fused, state-in-on-chip-memory
// design goal: intvml.com, engineering paragraph after point (6).)
//
// Work decomposition
//   * A channel's N states are split over LANES consecutive lanes of a warp
//     (S = N / LANES states per lane, updated as fp32x2 pairs with FFMA2 /
//     FMUL2).  A warp holds 32 / LANES channels; a CTA holds WARPS warps.
//   * Time advances in warp blocks of TB = LANES * V steps.  In a block, lane
//     j of a channel owns steps [j*V, j*V + V): it loads delta/u/z for them,
//     computes Delta and Delta*u once (shared with the channel's other lanes
//     through shared memory), and after the scan it receives their full
//     readout through a butterfly reduce-scatter and writes y.
//   * B and C are shared by every channel of a group; the CTA stages them in
//     shared memory per tile of TT steps as fp32 quads (B_n, B_n+1, C_n,
//     C_n+1), double-buffered with one CTA barrier per tile.
//   * A time range [t_begin, t_end) and an initial state let the same kernel
//     run a whole sequence or one chunk of it.
#pragma once

#include "ssm_device.cuh"
#include "tma.cuh"  // the library's device error word

namespace ssm {

// Range guard of every global access of the kernel below: an access whose
// elements [lo, hi) are not inside its tensor [0, size) is skipped and
// reported in the library's device error word (ssm_device_status).  Valid
// arguments never trip it; it keeps packed offsets that do not describe the
// row, or any slip in the index arithmetic, from touching other memory.
__device__ __forceinline__ bool in_range(long long lo, long long hi, long long size) {
    if (lo >= 0 && lo <= hi && hi <= size) return true;
    atomicOr(&g_ssm_device_error, kDeviceErrRange);
    return false;
}

struct ScanParams {
    const void* u;
    const void* delta;
    const void* z;        // nullable
    const float* A;
    const void* B;
    const void* C;
    const float* D;       // nullable
    const float* dt_bias; // nullable
    void* y;
    const float* h0;      // nullable
    float* h_final;       // nullable
    int batch, dim, seqlen, ngroups;
    int dim_per_group;    // dim / ngroups
    int blocks_per_group; // CTAs along the channels of one group
    int vec_ok;           // seqlen is a multiple of the activation packet width
    int bc_vec_ok;        // seqlen is a multiple of the 16-byte B/C packet width
    // Packed variable-length batch (batch == 1): sequence s occupies times
    // [cu_seqlens[s], cu_seqlens[s+1]) of the row and starts from h0[s];
    // h_final[s] is its end state.  NULL: one sequence per batch row.
    const int* cu_seqlens;
    int nseq;
};

// The generic kernel keeps the widened B/C tile in dynamic shared memory
// (single-buffered) from N = 128 on.
__host__ __device__ constexpr bool scan_bc_dynamic(int n) { return n >= 128; }

template <typename T, int LANES>
struct ScanShape {
    // Steps owned by one lane per block: a 16-byte packet when few lanes share
    // a channel, 4 steps otherwise (keeps TB = LANES * V <= 32 registers).
    static constexpr int V = (LANES <= 2) ? (16 / static_cast<int>(sizeof(T))) : 4;
    static constexpr int TB = LANES * V;
};

template <typename T, int N, int LANES, int WARPS, int TT, bool ACCURATE>
__global__ void __launch_bounds__(WARPS * 32)
scan_fwd_kernel(const ScanParams p) {
    constexpr int S = N / LANES;   // states per lane
    constexpr int P = S / 2;       // fp32x2 state pairs per lane
    static_assert(S >= 2 && S % 2 == 0, "each lane holds an even number of states");
    constexpr int CPW = 32 / LANES;  // channels per warp
    constexpr int CH = WARPS * CPW;  // channels per CTA
    constexpr int V = ScanShape<T, LANES>::V;
    constexpr int TB = ScanShape<T, LANES>::TB;
    static_assert(TT % TB == 0, "tile must hold whole warp blocks");
    constexpr int NQ = N / 2;        // (B,B,C,C) quads per step
    constexpr int VE = Elem<T>::kPer16B;
    constexpr int THREADS = WARPS * 32;
    constexpr int BC_ITEMS = 2 * N * (TT / VE);  // 16-byte B/C packets per tile
    // N >= 128: the widened B/C tile (32 or 128 KB) lives in dynamic shared
    // memory, single-buffered and staged between two barriers at each tile
    // boundary (no register copy of the next tile).
    constexpr bool DYN = scan_bc_dynamic(N);
    constexpr int BUFS = DYN ? 1 : 2;
    constexpr int BC_PER_THREAD = DYN ? 1 : (BC_ITEMS + THREADS - 1) / THREADS;

    __shared__ __align__(16) float4 bc_static[DYN ? 1 : 2][DYN ? 1 : TT][DYN ? 1 : NQ];
    extern __shared__ __align__(16) float4 bc_dynamic[];
    float4 (*bc_s)[TT][NQ] = DYN ? reinterpret_cast<float4 (*)[TT][NQ]>(bc_dynamic)
                                 : reinterpret_cast<float4 (*)[TT][NQ]>(&bc_static[0][0][0]);
    // (Delta, Delta*u) per warp channel and step; one float2 of padding per
    // row spreads the rows of a warp over distinct banks.
    __shared__ __align__(16) float2 dd_s[WARPS][CPW][TB + 1];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cw = lane / LANES;  // channel within warp
    const int j = lane % LANES;   // sub-lane within channel

    const int cb = blockIdx.x % p.blocks_per_group;
    const int bg = blockIdx.x / p.blocks_per_group;
    const int g = bg % p.ngroups;
    const int b = bg / p.ngroups;  // sequence: a batch row, or one of the packed sequences
    const int dloc = cb * CH + warp * CPW + cw;
    const bool active = dloc < p.dim_per_group;
    const int d = g * p.dim_per_group + (active ? dloc : 0);
    // This CTA's run of time: a whole row, or one packed sequence of the
    // single row (its offsets clamped into the row, so that any offsets stay
    // in bounds).  Lst is the row stride of every [.., L] tensor.
    const long long Lst = p.seqlen;
    long long seg0 = 0;
    int L = p.seqlen;
    int lead = 0;  // masked steps before a packed sequence's first one
    const bool packed = p.cu_seqlens != nullptr;
    if (packed) {
        const int s0 = min(max(__ldg(p.cu_seqlens + b), 0), p.seqlen);
        const int s1 = min(max(__ldg(p.cu_seqlens + b + 1), s0), p.seqlen);
        // Start the run on the 16-byte boundary at or before the sequence's
        // first step, so that every load and store stays a whole packet; the
        // `lead` steps before it belong to the previous sequence: they get
        // Delta = 0 (the state passes through) and their y is not written.
        lead = s0 % VE;
        seg0 = s0 - lead;
        L = s1 - s0 + lead;
    }
    const long long rowb = packed ? 0 : b;  // the tensors' batch row
    const long long nrows = packed ? 1 : p.batch;
    const long long act_size = nrows * p.dim * Lst;                  // u, delta, z, y
    const long long bc_size = nrows * p.ngroups * N * Lst;           // B, C
    const long long st_size = (packed ? p.nseq : p.batch) * static_cast<long long>(p.dim) * N;  // h0, h_final
    const long long row = (rowb * p.dim + d) * Lst + seg0;
    const T* __restrict__ u_row = static_cast<const T*>(p.u) + row;
    const T* __restrict__ dl_row = static_cast<const T*>(p.delta) + row;
    const T* __restrict__ z_row = p.z ? static_cast<const T*>(p.z) + row : nullptr;
    T* __restrict__ y_row = static_cast<T*>(p.y) + row;
    const long long bc_off = (rowb * p.ngroups + g) * N * Lst + seg0;
    const T* __restrict__ Bg = static_cast<const T*>(p.B) + bc_off;
    const T* __restrict__ Cg = static_cast<const T*>(p.C) + bc_off;
    // Vector packets need the run to start on a packet boundary.
    const bool vec_ok = p.vec_ok != 0 && seg0 % V == 0;
    const bool bc_vec_ok = p.bc_vec_ok != 0 && seg0 % VE == 0;
    const bool has_z = z_row != nullptr;

    // Per-lane constants: A (scaled for the exp form in use) for this lane's
    // states, bias, skip.
    float2 a2[P], h[P];
    {
        const float* Ad = p.A + static_cast<long long>(d) * N + j * S;
        const float* h0 = p.h0 ? p.h0 + (static_cast<long long>(b) * p.dim + d) * N + j * S : nullptr;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const float2 av = __ldg(reinterpret_cast<const float2*>(Ad) + k);
            a2[k] = make_float2(av.x * decay_scale<ACCURATE>(), av.y * decay_scale<ACCURATE>());
            const long long hoff = (static_cast<long long>(b) * p.dim + d) * N + j * S + 2 * k;
            h[k] = (h0 && active && in_range(hoff, hoff + 2, st_size))
                       ? __ldg(reinterpret_cast<const float2*>(h0) + k) : make_float2(0.f, 0.f);
        }
    }
    const float bias = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
    const float dsk = p.D ? __ldg(p.D + d) : 0.f;

    // ---- B/C tile staging: global -> registers -> shared (fp32 quads) ----
    Packet<T, VE> bc_reg[BC_PER_THREAD];
    auto load_item = [&](int item, int t0, Packet<T, VE>& pk) {
        const int r = item % (2 * N);  // (n, B|C) row, fastest across threads
        const int tv = item / (2 * N);
        const int n = r >> 1;
        const T* src = ((r & 1) ? Cg : Bg) + static_cast<long long>(n) * Lst + t0 + tv * VE;
        const int valid = L - (t0 + tv * VE);
        const long long boff = bc_off + static_cast<long long>(n) * Lst + t0 + tv * VE;
        const long long bhi = boff + ((bc_vec_ok && valid >= VE) ? VE : min(max(valid, 0), VE));
        if (valid > 0 && !in_range(boff, bhi, bc_size)) pk.zero();
        else if (bc_vec_ok && valid >= VE) pk.load_cached(src);
        else if (valid > 0) pk.load_partial(src, valid);
        else pk.zero();
    };
    auto store_item = [&](int item, int buf, const Packet<T, VE>& pk) {
        float* base = reinterpret_cast<float*>(&bc_s[buf][0][0]);
        const int r = item % (2 * N);
        const int tv = item / (2 * N);
        const int n = r >> 1;
        const int isC = r & 1;
        // Pair k of sub-lane j sits at k * LANES + j: the lanes of a
        // channel read adjacent quads (no bank conflicts).
        const int q = n >> 1;
        const int off = ((q % P) * LANES + q / P) * 4 + isC * 2 + (n & 1);
        float f[VE];
        pk.to_float(f);
#pragma unroll
        for (int k = 0; k < VE; ++k) base[(tv * VE + k) * (2 * N) + off] = f[k];
    };
    auto load_bc = [&](int t0) {
#pragma unroll
        for (int i = 0; i < BC_PER_THREAD; ++i) {
            const int item = threadIdx.x + i * THREADS;
            if (item < BC_ITEMS) load_item(item, t0, bc_reg[i]);
        }
    };
    auto store_bc = [&](int buf) {
#pragma unroll
        for (int i = 0; i < BC_PER_THREAD; ++i) {
            const int item = threadIdx.x + i * THREADS;
            if (item < BC_ITEMS) store_item(item, buf, bc_reg[i]);
        }
    };
    // Single-buffered tiles: load and widen item by item.
    auto stage_bc = [&](int t0) {
#pragma unroll 2
        for (int item = threadIdx.x; item < BC_ITEMS; item += THREADS) {
            Packet<T, VE> pk;
            load_item(item, t0, pk);
            store_item(item, 0, pk);
        }
    };

    // ---- per-lane activation packets, prefetched one warp block ahead ----
    Packet<T, V> pd_cur, pu_cur, pz_cur, pd_nxt, pu_nxt, pz_nxt;
    auto load_act = [&](int tb0, Packet<T, V>& pd, Packet<T, V>& pu, Packet<T, V>& pz) {
        const int t = tb0 + j * V;
        int valid = active ? (L - t) : 0;
        {
            const long long lo = row + t, hi = lo + ((vec_ok && valid >= V) ? V : min(max(valid, 0), V));
            if (valid > 0 && !in_range(lo, hi, act_size)) valid = 0;
        }
        load_row<T, V>(pd, dl_row + t, valid, vec_ok);
        load_row<T, V>(pu, u_row + t, valid, vec_ok);
        if (has_z) load_row<T, V>(pz, z_row + t, valid, vec_ok);
        else pz.zero();
    };

    const int ntiles = (L + TT - 1) / TT;
    if (ntiles > 0) {
        if constexpr (DYN) {
            stage_bc(0);
        } else {
            load_bc(0);
            store_bc(0);
        }
        load_act(0, pd_cur, pu_cur, pz_cur);
    }
    __syncthreads();

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = BUFS == 2 ? (tile & 1) : 0;
        const int t0 = tile * TT;
        if constexpr (!DYN) {
            if (tile + 1 < ntiles) load_bc(t0 + TT);
        }

#pragma unroll 1
        for (int blk = 0; blk < TT / TB; ++blk) {
            const int tb0 = t0 + blk * TB;
            if (tb0 >= L) break;  // uniform over the CTA
            if (tb0 + TB < L) load_act(tb0 + TB, pd_nxt, pu_nxt, pz_nxt);

            // Prologue: Delta and Delta*u for this lane's V steps.
            float uu[V], zz[V];
            {
                float dv[V];
                pd_cur.to_float(dv);
                pu_cur.to_float(uu);
                pz_cur.to_float(zz);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const int tk = tb0 + j * V + k;
                    const bool in = active && tk < L && tk >= lead;
                    const float dt = in ? softplus<ACCURATE>(dv[k] + bias) : 0.f;
                    dd_s[warp][cw][j * V + k] = make_float2(dt, dt * uu[k]);
                }
            }
            __syncwarp();

            // Scan: every lane advances its S states through all TB steps.
            float acc[TB];
            const float4* bcq = &bc_s[buf][blk * TB][j];
#pragma unroll
            for (int st = 0; st < TB; ++st) {
                const float2 dd = dd_s[warp][cw][st];
                const float2 dt2 = make_float2(dd.x, dd.x);
                const float2 du2 = make_float2(dd.y, dd.y);
                float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const float4 q = bcq[st * NQ + k * LANES];
                    const float2 x = __fmul2_rn(dt2, a2[k]);
                    const float2 abar = make_float2(decay<ACCURATE>(x.x), decay<ACCURATE>(x.y));
                    const float2 bx = __fmul2_rn(du2, make_float2(q.x, q.y));
                    h[k] = __ffma2_rn(abar, h[k], bx);
                    y2 = __ffma2_rn(make_float2(q.z, q.w), h[k], y2);
                }
                acc[st] = y2.x + y2.y;
            }

            // Readout of the channel's other lanes -> owner lane; skip, gate, store.
            reduce_scatter<LANES, V>(acc, j);
            if (active) {
                float out[V];
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    float yv = acc[k] + dsk * uu[k];
                    if (has_z) yv *= silu<ACCURATE>(zz[k]);
                    out[k] = yv;
                }
                const int t = tb0 + j * V;
                if (t >= lead) {
                    const int valid = L - t;
                    const long long lo = row + t, hi = lo + ((vec_ok && valid >= V) ? V : min(max(valid, 0), V));
                    if (valid <= 0 || in_range(lo, hi, act_size)) store_row<T, V>(y_row + t, out, valid, vec_ok);
                } else {
#pragma unroll
                    for (int k = 0; k < V; ++k)
                        if (t + k >= lead && t + k < L && in_range(row + t + k, row + t + k + 1, act_size))
                            Elem<T>::store(y_row + t + k, out[k]);
                }
            }
            pd_cur = pd_nxt;
            pu_cur = pu_nxt;
            pz_cur = pz_nxt;
            __syncwarp();
        }

        if constexpr (DYN) {
            if (tile + 1 < ntiles) {
                __syncthreads();  // every lane has read this tile
                stage_bc(t0 + TT);
            }
        } else {
            if (tile + 1 < ntiles) store_bc(buf ^ 1);
        }
        __syncthreads();
    }

    if (p.h_final && active) {
        float* hf = p.h_final + (static_cast<long long>(b) * p.dim + d) * N + j * S;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const long long hoff = (static_cast<long long>(b) * p.dim + d) * N + j * S + 2 * k;
            if (in_range(hoff, hoff + 2, st_size)) reinterpret_cast<float2*>(hf)[k] = h[k];
        }
    }
}

}  // namespace ssm
