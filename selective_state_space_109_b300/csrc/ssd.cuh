// ssd.cuh -- the SSD (Mamba-2) layer on the tcgen05 tensor cores, sm_103a.
//
// The layer is the selective recurrence with a scalar decay per head
// (eightmm.github.io "Mamba", Relation to Mamba-2): head h owns P channels
// that share A[h], the step Delta_t = softplus(delta[b, h, t] + dt_bias[h]) and
// the skip Dskip[h]; B and C belong to the head's group.  Written as the causal
// matrix mixer of that section, y_t = sum_{s<=t} C_t (prod_{j=s+1..t} Abar_j)
// Bbar_s x_s, a chunk of Q = 128 steps splits into dense contractions:
//
//   G      = C B^T                         [Q x Q]   over the N states
//   M      = G o exp(cs_t - cs_s) Delta_s   (s <= t, else 0; cs = running sum of Delta A)
//   Ydiag  = M X                           [Q x P]   the chunk's own inputs
//   Yoff   = C H_prev, scaled by exp(cs_t) [Q x P]   the state carried in
//   S      = B^T (w o X),  w_s = exp(cs_end - cs_s) Delta_s     [N x P]
//   H      = exp(cs_end) H_prev + S                  the state carried out
//   y      = (Ydiag + Yoff + Dskip x) * silu(z)
//
// One CTA walks one (sequence, head) through its chunks in order, so the state
// H stays on chip (fp32 in registers, half a state row per thread; a bf16 copy
// in shared memory feeds the next chunk's Yoff).  Thread 0 issues the TMA
// loads of each chunk's C, B, x, z tiles (128-byte swizzled rows of 64 steps;
// x and z one chunk ahead, C and B as soon as the first contractions have read
// the current ones) and the tcgen05.mma contractions (bf16 operands from shared
// memory, fp32 accumulators in tensor memory).  The 256 threads -- two
// warpgroups, each owning the 128 tensor-memory lanes for half of every
// accumulator row's columns -- build the computed operands (M, w o X, H), read
// the accumulators back with tcgen05.ld and form y, which leaves by a TMA
// store.  Operand layouts are the 128-byte-swizzled K-major or MN-major tiles
// of the UMMA descriptors; every wait is bounded.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_device.cuh"
#include "tma.cuh"

namespace ssm {

struct SsdParams {
    const __nv_bfloat16* delta;  // [batch, nheads, L]
    const float* A;              // [nheads]
    const float* D;              // [nheads] or null
    const float* dt_bias;        // [nheads] or null
    const float* h0;             // [batch, nheads * P, N] or null
    float* h_final;              // [batch, nheads * P, N] or null
    unsigned int* status;        // null (device error word only)
    int batch, nheads, seqlen, ngroups;
    int has_z;
};

namespace ssd {

constexpr int Q = 128;   // chunk length (the MMA's M for the per-step rows)
constexpr int P = 64;    // head dimension
constexpr int N = 128;   // state size
constexpr int THREADS = 256;  // two warpgroups: each takes half the columns of every accumulator row

// Shared-memory layout (bytes from a 1024-aligned base).  Tiles of 128-byte
// rows, two halves of 64 steps along time where a row holds 128 steps.  x and
// z are double-buffered (the next chunk's tiles load during this chunk); C
// and B are reloaded as soon as the first contractions have read them.
constexpr int CS_OFF = 0;                     // C  [N rows][Q]   (2 halves of N x 128 B)
constexpr int BS_OFF = CS_OFF + N * 256;      // B  [N rows][Q]
constexpr int XS_OFF = BS_OFF + N * 256;      // x  [P rows][Q], two buffers
constexpr int ZS_OFF = XS_OFF + 2 * P * 256;  // z  [P rows][Q], two buffers
constexpr int XH_OFF = ZS_OFF + 2 * P * 256;  // w o x, bf16 head  [P rows][Q] (B operand of S); y staging
constexpr int XL_OFF = XH_OFF + P * 256;      // w o x, bf16 tail (the rounding error of the head)
constexpr int MS_OFF = XL_OFF + P * 256;      // M  [Q rows][Q]     (A operand of Ydiag)
constexpr int HS_OFF = MS_OFF + Q * 256;      // H  [N rows][P]     (bf16 copy, B operand of Yoff)
constexpr int F_OFF = HS_OFF + N * 128;       // floats: Delta[Q], cs[Q], w[Q], warp sums[8]
constexpr int BAR_OFF = F_OFF + (3 * Q + 8) * 4;
constexpr int SMEM_BYTES = BAR_OFF + 64 + 1024;  // four mbarriers, the TMEM address, alignment slack
constexpr int XBUF = P * 256;                     // bytes of one x (or z) buffer
constexpr int HALF_C = N * 128;                   // byte stride between the time halves of C, B
constexpr int HALF_X = P * 128;                   // ... of x, z, w o x, y
constexpr int HALF_M = Q * 128;                   // ... of M
constexpr uint32_t TX_BC = 2u * N * 256u;         // bytes of one chunk's C and B tiles
constexpr uint32_t TX_X = P * 256u;               // ... of its x (or z) tile
static_assert(SMEM_BYTES <= 227 * 1024, "the SSD kernel's shared memory exceeds a CTA's limit");

// Tensor-memory columns (512 allocated; lanes = rows of the accumulators).
constexpr uint32_t TM_G = 0;      // G      [Q lanes x Q]
constexpr uint32_t TM_YOFF = 128; // Yoff   [Q lanes x P]
constexpr uint32_t TM_YD = 192;   // Ydiag  [Q lanes x P]
constexpr uint32_t TM_S = 256;    // S      [N lanes x P]

// Byte offset of element c (0..63) of row r in a tile of 128-byte rows written
// with the 128-byte swizzle (16-byte unit index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_elem(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((((c * 2) >> 4) ^ (r & 7)) << 4) + ((c * 2) & 15));
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand tile:
// start address, leading and stride byte offsets, layout version 1, swizzle
// mode 128B.  K-major tiles: rows along M/N, 64 K elements per 128-byte row,
// stride 1024 bytes between 8-row groups.  MN-major tiles: rows along K, 64
// M/N elements per row, stride `lbo` between 64-element groups along M/N and
// 1024 bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of a dense bf16 x bf16 -> fp32 tcgen05.mma (kind::f16)
// of shape M x N, A and B each K-major (false) or MN-major (true).
__host__ __device__ constexpr uint32_t umma_idesc(int m, int n, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier once every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane.  The load
// and its wait are one asm statement, so that no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float bf_at(const unsigned char* tile, uint32_t off) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(tile + off)) << 16);
}

__device__ __forceinline__ void bf_put(unsigned char* tile, uint32_t off, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = b;
}

}  // namespace ssd

// One CTA per (sequence b, head h): blockIdx.x = b * nheads + h.
__global__ void __launch_bounds__(ssd::THREADS, 1)
ssd_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_B,
               const __grid_constant__ CUtensorMap tm_C, const SsdParams p) {
    using namespace ssd;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* Cs = smem + CS_OFF;
    unsigned char* Bs = smem + BS_OFF;
    unsigned char* Xh = smem + XH_OFF;
    unsigned char* Xl = smem + XL_OFF;
    unsigned char* Ys = Xh;  // y staging reuses the w o x head once the state contraction has read it
    unsigned char* Ms = smem + MS_OFF;
    unsigned char* Hs = smem + HS_OFF;
    float* dts = reinterpret_cast<float*>(smem + F_OFF);  // Delta_t
    float* css = dts + Q;                                 // cs_t: running sum of Delta A (log2 units)
    float* wss = css + Q;                                 // w_s = 2^(cs_end - cs_s) Delta_s
    float* wsum = wss + Q;                                // per-warp totals of the running sum
    uint64_t* bc_bar = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // C, B of the current chunk
    uint64_t* xz_bar = bc_bar + 1;                                   // x, z: one barrier per buffer
    uint64_t* mma_bar = bc_bar + 3;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 32);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r = tid & (Q - 1);  // accumulator row (tensor-memory lane) of this thread
    const int wg = tid >> 7;      // warpgroup: which half of the row's columns it takes
    const int bh = blockIdx.x;
    const int b = bh / p.nheads, h = bh % p.nheads;
    const int g = h / (p.nheads / p.ngroups);
    const int L = p.seqlen;
    const int nch = (L + Q - 1) / Q;
    const bool has_z = p.has_z != 0;
    const float a2 = __ldg(p.A + h) * kLog2e;  // decay exponent per unit of Delta, base 2
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    const float dsk = p.D ? __ldg(p.D + h) : 0.f;
    const long long dim = static_cast<long long>(p.nheads) * P;
    const int xrow = bh * P;                                 // first row of the head in the x/z/y maps
    const int bcrow = (b * p.ngroups + g) * N;               // first row of the group in the B/C maps

    // TMA loads: C and B of chunk c (one phase per chunk), x and z of chunk c
    // into buffer c % 2 (one phase per use of the buffer).
    auto load_bc = [&](int c) {
        mbar_arrive_expect_tx(bc_bar, TX_BC);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_2d(Cs + half * HALF_C, &tm_C, c * Q + half * 64, bcrow, bc_bar);
            tma_load_2d(Bs + half * HALF_C, &tm_B, c * Q + half * 64, bcrow, bc_bar);
        }
    };
    auto load_xz = [&](int c) {
        const int buf = c & 1;
        mbar_arrive_expect_tx(&xz_bar[buf], has_z ? 2 * TX_X : TX_X);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_2d(smem + XS_OFF + buf * XBUF + half * HALF_X, &tm_x, c * Q + half * 64, xrow, &xz_bar[buf]);
            if (has_z)
                tma_load_2d(smem + ZS_OFF + buf * XBUF + half * HALF_X, &tm_z, c * Q + half * 64, xrow,
                            &xz_bar[buf]);
        }
    };
    if (tid == 0) {
        mbar_init(bc_bar, 1);
        mbar_init(&xz_bar[0], 1);
        mbar_init(&xz_bar[1], 1);
        mbar_init(mma_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_y);
        if (has_z) prefetch_tensormap(&tm_z);
        load_bc(0);
        load_xz(0);
        if (nch > 1) load_xz(1);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(tslot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // The carried state: state row n = r, channels p = 32 wg .. 32 wg + 31 per
    // thread (fp32), and its bf16 copy in shared memory ([n rows][p], MN-major
    // operand of Yoff).
    constexpr int PH = P / 2;
    float H[PH];
    {
        const float* h0 = p.h0 ? p.h0 + (static_cast<long long>(b) * dim + static_cast<long long>(h) * P) * N : nullptr;
#pragma unroll
        for (int i = 0; i < PH; ++i) {
            const int q = wg * PH + i;
            H[i] = h0 ? __ldg(h0 + static_cast<long long>(q) * N + r) : 0.f;
            bf_put(Hs, sw128_elem(r, q), H[i]);
        }
    }
    // Raw step input of this thread's step (threads 0 .. Q-1), loaded a chunk ahead.
    const __nv_bfloat16* drow = p.delta + static_cast<long long>(bh) * L;
    float dnext = (tid < Q && tid < L) ? __bfloat162float(drow[tid]) : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes

    uint32_t mma_phase = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * Q;
        const int buf = c & 1;
        const unsigned char* Xs = smem + XS_OFF + buf * XBUF;
        const unsigned char* Zs = smem + ZS_OFF + buf * XBUF;
        // (1) the previous chunk's y store has read its staging tile (the w o x
        // head, rewritten below)
        if (tid == 0) bulk_wait_read<0>();
        // (2) step sizes and the running sum of Delta A (threads 0 .. Q-1: one step each)
        {
            float dt = 0.f, v = 0.f;
            if (tid < Q) {
                if (t0 + tid < L) dt = softplus<false>(dnext + bias);
                // the next chunk's step input, in flight while this chunk runs
                dnext = (t0 + Q + tid < L) ? __bfloat162float(drow[t0 + Q + tid]) : 0.f;
                v = dt * a2;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                if (lane == 31) wsum[warp] = v;
                dts[tid] = dt;
            }
            __syncthreads();
            if (tid < Q) {
                for (int w = 0; w < warp; ++w) v += wsum[w];
                css[tid] = v;
            }
            __syncthreads();
            if (tid < Q) wss[tid] = ex2_approx(css[Q - 1] - v) * dt;
            __syncthreads();
        }
        const float cs_end = css[Q - 1];
        // (3) the tiles have landed
        mbar_wait(bc_bar, static_cast<uint32_t>(c & 1), p.status);
        mbar_wait(&xz_bar[buf], static_cast<uint32_t>((c >> 1) & 1), p.status);
        // (4) w o x, the B operand of the state contraction (same layout as x),
        // as a bf16 head plus a bf16 tail holding the head's rounding error, so
        // that the carried state keeps fp32 accuracy through the contraction
#pragma unroll 2
        for (int item = tid; item < P * 16; item += THREADS) {
            const int row = item >> 4, unit = item & 15;
            const int half = unit >> 3, u8 = unit & 7;
            const uint32_t off = half * HALF_X + static_cast<uint32_t>(row * 128 + ((u8 ^ (row & 7)) << 4));
            const uint4 raw = *reinterpret_cast<const uint4*>(Xs + off);
            const uint32_t w32[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t oh[4], ol[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = half * 64 + u8 * 8 + 2 * k;
                const float v0 = __uint_as_float(w32[k] << 16) * wss[s];
                const float v1 = __uint_as_float(w32[k] & 0xffff0000u) * wss[s + 1];
                const __nv_bfloat162 ph = __floats2bfloat162_rn(v0, v1);
                const float2 fh = __bfloat1622float2(ph);
                const __nv_bfloat162 pl = __floats2bfloat162_rn(v0 - fh.x, v1 - fh.y);
                oh[k] = *reinterpret_cast<const uint32_t*>(&ph);
                ol[k] = *reinterpret_cast<const uint32_t*>(&pl);
            }
            *reinterpret_cast<uint4*>(Xh + off) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
            *reinterpret_cast<uint4*>(Xl + off) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // (5) G = C B^T, Yoff = C H_prev, S = B^T (w o x)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t cs_a = smem_addr(Cs), bs_a = smem_addr(Bs), hs_a = smem_addr(Hs);
            const uint32_t xh_a = smem_addr(Xh), xl_a = smem_addr(Xl);
            const uint32_t id_g = umma_idesc(Q, Q, true, true);
            const uint32_t id_off = umma_idesc(Q, P, true, true);
            const uint32_t id_s = umma_idesc(N, P, false, false);
#pragma unroll
            for (int ks = 0; ks < N / 16; ++ks) {  // K = the N states, 16 rows per step
                const uint64_t ca = umma_desc(cs_a + ks * 2048, HALF_C, 1024);
                umma_f16(tmem + TM_G, ca, umma_desc(bs_a + ks * 2048, HALF_C, 1024), id_g, ks > 0);
                umma_f16(tmem + TM_YOFF, ca, umma_desc(hs_a + ks * 2048, HALF_C, 1024), id_off, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < Q / 16; ++ks) {  // K = the chunk's steps
                const uint32_t koff = (ks & 3) * 32;  // 16 steps = 32 bytes into the 128-byte row
                const uint64_t ba = umma_desc(bs_a + (ks >> 2) * HALF_C + koff, 16, 1024);
                umma_f16(tmem + TM_S, ba, umma_desc(xh_a + (ks >> 2) * HALF_X + koff, 16, 1024), id_s, ks > 0);
                umma_f16(tmem + TM_S, ba, umma_desc(xl_a + (ks >> 2) * HALF_X + koff, 16, 1024), id_s, 1);
            }
            umma_commit(mma_bar);
        }
        mbar_wait(mma_bar, mma_phase & 1, p.status);
        ++mma_phase;
        tc_fence_after();
        // C and B of this chunk are read: the next chunk's tiles load meanwhile.
        if (tid == 0 && c + 1 < nch) load_bc(c + 1);
        // (6) M = G o 2^(cs_t - cs_s) Delta_s (s <= t), row t = r, columns
        // s = 64 wg .. 64 wg + 63
        const float cs_t = css[r];
#pragma unroll 1
        for (int j = 2 * wg; j < 2 * wg + 2; ++j) {
            float gv[32];
            tmem_ld32(tmem + lane_base + TM_G + j * 32, gv);
            const int half = j >> 1;
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {  // four 16-byte units of 8 steps
                uint32_t o32[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i0 = u4 * 8 + 2 * k;
                    const int s0 = j * 32 + i0;
                    const float m0 = s0 <= r ? gv[i0] * ex2_approx(cs_t - css[s0]) * dts[s0] : 0.f;
                    const float m1 = s0 + 1 <= r ? gv[i0 + 1] * ex2_approx(cs_t - css[s0 + 1]) * dts[s0 + 1] : 0.f;
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(m0, m1);
                    o32[k] = *reinterpret_cast<const uint32_t*>(&pr);
                }
                const int unit = ((j & 1) * 4 + u4);  // 16-byte unit within the 128-byte row of this half
                const uint32_t off = half * HALF_M + static_cast<uint32_t>(r * 128 + ((unit ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(Ms + off) = make_uint4(o32[0], o32[1], o32[2], o32[3]);
            }
        }
        // (7) H = 2^cs_end H + S, state row n = r, channels 32 wg .. 32 wg + 31,
        // and its bf16 copy (pairs of channels per 4-byte store)
        {
            const float decay_all = ex2_approx(cs_end);
            float sv[32];
            tmem_ld32(tmem + lane_base + TM_S + wg * PH, sv);
#pragma unroll
            for (int i = 0; i < PH; i += 2) {
                H[i] = fmaf(decay_all, H[i], sv[i]);
                H[i + 1] = fmaf(decay_all, H[i + 1], sv[i + 1]);
                const __nv_bfloat162 pr = __floats2bfloat162_rn(H[i], H[i + 1]);
                *reinterpret_cast<__nv_bfloat162*>(Hs + sw128_elem(r, wg * PH + i)) = pr;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // (8) Ydiag = M x
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ms_a = smem_addr(Ms), xs_a = smem_addr(Xs);
            const uint32_t id_d = umma_idesc(Q, P, false, false);
#pragma unroll
            for (int ks = 0; ks < Q / 16; ++ks) {
                const uint32_t koff = (ks & 3) * 32;
                umma_f16(tmem + TM_YD, umma_desc(ms_a + (ks >> 2) * HALF_M + koff, 16, 1024),
                         umma_desc(xs_a + (ks >> 2) * HALF_X + koff, 16, 1024), id_d, ks > 0);
            }
            umma_commit(mma_bar);
        }
        mbar_wait(mma_bar, mma_phase & 1, p.status);
        ++mma_phase;
        tc_fence_after();
        // (9) y = (Ydiag + 2^cs_t Yoff + D x) * silu(z), row t = r, channels
        // 32 wg .. 32 wg + 31, staged as [p rows][t]
        {
            const float e_t = ex2_approx(cs_t);
            const int half = r >> 6, tc = r & 63;
            float yd[32], yo[32];
            tmem_ld32(tmem + lane_base + TM_YD + wg * PH, yd);
            tmem_ld32(tmem + lane_base + TM_YOFF + wg * PH, yo);
#pragma unroll
            for (int i = 0; i < PH; ++i) {
                const int q = wg * PH + i;
                const uint32_t off = half * HALF_X + sw128_elem(q, tc);
                const float xv = bf_at(Xs, off);
                float yv = fmaf(dsk, xv, fmaf(e_t, yo[i], yd[i]));
                if (has_z) yv *= silu<false>(bf_at(Zs, off));
                bf_put(Ys, off, yv);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int half = 0; half < 2; ++half) tma_store_2d(&tm_y, t0 + half * 64, xrow, Ys + half * HALF_X);
            bulk_commit();
            // x and z of this buffer are read: chunk c + 2 loads into it.
            if (c + 2 < nch) load_xz(c + 2);
        }
    }
    if (tid == 0) bulk_wait<0>();
    if (p.h_final) {
        float* hf = p.h_final + (static_cast<long long>(b) * dim + static_cast<long long>(h) * P) * N;
#pragma unroll
        for (int i = 0; i < PH; ++i) hf[static_cast<long long>(wg * PH + i) * N + r] = H[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

}  // namespace ssm
