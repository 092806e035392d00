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
// State sizes below N = 128 run on the same tiles: the B and C tiles load
// through 3-D maps whose rows past the caller's state size are filled with
// zeros, so G, Yoff and S gain only zero terms and the padded state rows stay
// zero (h0 and h_final touch only the caller's rows).
//
// One CTA walks one (sequence, head) through its chunks in order, so the state
// H stays on chip (fp32 in registers, a 16-channel slice of a state row per
// thread; a bf16 copy in shared memory feeds the next chunk's Yoff).  A
// control warp issues the TMA loads of each chunk's C, B and x tiles
// (128-byte swizzled rows of 64 steps; x two chunks ahead, C and B as soon
// as the previous chunk's contractions have read them), the
// tcgen05.mma contractions (bf16 operands from shared memory, except M,
// which Ydiag reads from tensor memory; fp32 accumulators in tensor memory;
// issued by one thread), and computes the per-step scalars (Delta, the
// running sum of Delta A, the state weights w) two chunks ahead.  Sixteen
// compute warps -- four per quarter of the 128 tensor-memory lanes, each
// taking a quarter of every accumulator row's columns -- build the computed
// operands (M with tcgen05.st, w o X and H in shared memory), read the
// accumulators back with tcgen05.ld and form y in a shared-memory tile: z
// arrives there by TMA while the chunk's operands are built, each thread
// overwrites its own z elements with y, and the control warp stores the tile
// by TMA.  The chunks are software-pipelined so that the tensor cores run
// while the threads compute: Yd(c) = M X and G, Yoff of chunk c+1 run while
// the compute warps weight chunk c+1's x, and S of chunk c+1 while they form
// chunk c's output.  Only the lower triangle of M (s <= t) is computed; its
// upper blocks are written as zeros.  Shared-memory operands are the
// 128-byte-swizzled K-major or MN-major tiles of the UMMA descriptors; every
// wait is bounded.
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
    const float* h0;             // [batch, nheads * P, dstate] or null
    float* h_final;              // [batch, nheads * P, dstate] or null
    const __nv_bfloat16* z;      // [batch, nheads * P, L] or null
    __nv_bfloat16* y;            // [batch, nheads * P, L]
    unsigned int* status;        // null (device error word only)
    int batch, nheads, seqlen, ngroups;
    int dstate;                  // the caller's state size, at most N: the tiles' rows past it load as zeros
    int has_z;
};

namespace ssd {

constexpr int Q = 128;   // chunk length (the MMA's M for the per-step rows)
constexpr int P = 64;    // head dimension
constexpr int N = 128;   // state size
constexpr int COMPUTE = 512;          // sixteen compute warps: lane quarter = warp % 4, column group = warp / 4
constexpr int THREADS = COMPUTE + 32; // and one control warp (TMA, MMA issue, per-step scalars)
constexpr int CTRL = COMPUTE;         // the control warp's first thread
constexpr int CG = COMPUTE / 128;     // column groups (each a quarter of an accumulator row's columns)

// Shared-memory layout (bytes from a 1024-aligned base).  Tiles of 128-byte
// rows, two halves of 64 steps along time where a row holds 128 steps.  x has
// three buffers (its tile loads two chunks ahead); C and B are reloaded as
// soon as the contractions of the chunk have read them.  One z tile: loaded
// once the previous chunk's y (formed in the same tile) has been read out by
// its TMA store.
constexpr int XBUFS = 3;                      // x buffers
constexpr int CS_OFF = 0;                     // C  [N rows][Q]   (2 halves of N x 128 B)
constexpr int BS_OFF = CS_OFF + N * 256;      // B  [N rows][Q]
constexpr int XS_OFF = BS_OFF + N * 256;      // x  [P rows][Q], XBUFS buffers
constexpr int XW_OFF = XS_OFF + XBUFS * P * 256;  // w o x [2P rows][Q]: P rows of the bf16 head, then
                                              // P rows of its tail (the head's rounding error); B operand of S
constexpr int HS_OFF = XW_OFF + 2 * P * 256;  // H  [N rows][P]     (bf16 copy, B operand of Yoff)
constexpr int ZS_OFF = HS_OFF + N * 128;      // z, then y in place  [P rows][Q]
constexpr int F_OFF = ZS_OFF + P * 256;       // floats, two buffers of: (cs_t, Delta_t) pairs [Q], w_t [Q]
constexpr int F_BUF = 3 * Q;                  // floats per buffer
constexpr int BAR_OFF = F_OFF + 2 * F_BUF * 4;
constexpr int SMEM_BYTES = BAR_OFF + 64 + 1024;  // seven mbarriers, the TMEM address, alignment slack
constexpr int XBUF = P * 256;                     // bytes of one x buffer
constexpr int HALF_C = N * 128;                   // byte stride between the time halves of C, B
constexpr int HALF_X = P * 128;                   // ... of x
constexpr int HALF_W = 2 * P * 128;               // ... of w o x (head and tail rows)
constexpr uint32_t TX_BC = 2u * N * 256u;         // bytes of one chunk's C and B tiles
constexpr uint32_t TX_X = P * 256u;               // ... of its x tile
static_assert(SMEM_BYTES <= 227 * 1024, "the SSD kernel's shared memory exceeds a CTA's limit");
static_assert(COMPUTE == 4 * 128 && P == 16 * CG && Q == 32 * CG, "warp roles assume 16 warps, P 64, Q 128");

// Tensor-memory columns (512 allocated; lanes = rows of the accumulators).
constexpr uint32_t TM_G = 0;      // G      [Q lanes x Q]
constexpr uint32_t TM_S = 128;    // S      [N lanes x 2P]: B^T (head of w o x), then B^T (its tail)
constexpr uint32_t TM_YD = 256;   // Ydiag  [Q lanes x P]
constexpr uint32_t TM_YOFF = 320; // Yoff   [Q lanes x P], two buffers (chunk parity)
constexpr uint32_t TM_M = 448;    // M      [Q lanes x Q] bf16, two steps a column (A operand of Ydiag)

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

// The same contraction with the A operand in tensor memory: M rows in lanes,
// two bf16 K elements a 32-bit column (the lower K index in the low half).
__device__ __forceinline__ void umma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// 16 consecutive fp32 columns of this thread's tensor-memory lane (load and
// wait in one asm statement, as above).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&a)[16], float (&b)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        a[i] = __uint_as_float(r[i]);
        b[i] = __uint_as_float(r[16 + i]);
    }
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane, stored
// and waited for in one asm statement.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&pr);
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
ssd_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
               const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_y, const SsdParams p) {
    using namespace ssd;
    // Programmatic dependent launch: the next kernel may begin launching now;
    // this one waits for the previous kernel's writes before reading anything.
    grid_dep_launch();
    grid_dep_wait();
    extern __shared__ __align__(16) unsigned char smem_raw[];  // aligned below at run time
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* Cs = smem + CS_OFF;
    unsigned char* Bs = smem + BS_OFF;
    unsigned char* Xw = smem + XW_OFF;
    unsigned char* Hs = smem + HS_OFF;
    unsigned char* Zs = smem + ZS_OFF;
    float* fbase = reinterpret_cast<float*>(smem + F_OFF);  // per buffer: float2 (cs_t, Delta_t) [Q], w_t [Q]
    uint64_t* bc_bar = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // C, B of the current chunk
    uint64_t* x_bar = bc_bar + 1;                                    // x: one barrier per buffer
    uint64_t* mma1_bar = bc_bar + 1 + XBUFS;                         // G, S, Yoff of a chunk done
    uint64_t* mma2_bar = mma1_bar + 1;                               // Ydiag of a chunk done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 48);
    uint64_t* z_bar = bc_bar + 7;                                    // z of the current chunk
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3;      // tensor-memory lane quarter of this warp
    const int cg = warp >> 2;     // column group of this warp
    const int r = tid & (Q - 1);  // accumulator row (tensor-memory lane) of this thread: 32 qd + lane
    const int bh = blockIdx.x;
    const int b = bh / p.nheads, h = bh % p.nheads;
    const int g = h / (p.nheads / p.ngroups);
    const int L = p.seqlen;
    const int nch = (L + Q - 1) / Q;
    const bool has_z = p.has_z != 0 && p.z != nullptr;
    const float a2 = __ldg(p.A + h) * kLog2e;  // decay exponent per unit of Delta, base 2
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    const float dsk = p.D ? __ldg(p.D + h) : 0.f;
    const long long dim = static_cast<long long>(p.nheads) * P;
    const int xrow = bh * P;                    // first row of the head in the x/z/y maps
    const int bcg = b * p.ngroups + g;          // the (sequence, group) plane of the B/C maps
    const int NS = p.dstate;                    // state rows in memory (rows NS..N-1 of the tiles are zero)
    constexpr int PC = P / CG;                  // channels per column group (16)

    // TMA loads: C and B of chunk c (one phase per chunk), x of chunk c into
    // buffer c % XBUFS (one phase per use of the buffer).
    auto load_bc = [&](int c) {
        mbar_arrive_expect_tx(bc_bar, TX_BC);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(Cs + half * HALF_C, &tm_C, c * Q + half * 64, 0, bcg, bc_bar);
            tma_load_3d(Bs + half * HALF_C, &tm_B, c * Q + half * 64, 0, bcg, bc_bar);
        }
    };
    auto load_x = [&](int c) {
        const int buf = c % XBUFS;
        mbar_arrive_expect_tx(&x_bar[buf], TX_X);
#pragma unroll
        for (int half = 0; half < 2; ++half)
            tma_load_2d(smem + XS_OFF + buf * XBUF + half * HALF_X, &tm_x, c * Q + half * 64, xrow, &x_bar[buf]);
    };
    auto load_z = [&](int c) {
        mbar_arrive_expect_tx(z_bar, TX_X);
#pragma unroll
        for (int half = 0; half < 2; ++half) tma_load_2d(Zs + half * HALF_X, &tm_z, c * Q + half * 64, xrow, z_bar);
    };
    if (tid == CTRL) {
        mbar_init(bc_bar, 1);
#pragma unroll
        for (int i = 0; i < XBUFS; ++i) mbar_init(&x_bar[i], 1);
        mbar_init(mma1_bar, 1);
        mbar_init(mma2_bar, 1);
        mbar_init(z_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_y);
        load_bc(0);
        if (has_z) {
            prefetch_tensormap(&tm_z);
            load_z(0);
        }
        for (int c = 0; c < XBUFS && c < nch; ++c) load_x(c);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(tslot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    const bool compute = tid < COMPUTE;
    uint32_t tmem = 0;  // tensor-memory base (read after the first barrier)

    // The carried state (compute threads): state row n = r, channels
    // PC cg .. PC cg + PC - 1 (fp32), and its bf16 copy in shared memory
    // ([n rows][p], MN-major operand of Yoff): two 16-byte units of the row.
    float H[PC];
    auto store_hs = [&]() {
        uint32_t w[PC / 2];
#pragma unroll
        for (int i = 0; i < PC / 2; ++i) w[i] = pack_bf2(H[2 * i], H[2 * i + 1]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int unit = 2 * cg + u;
            *reinterpret_cast<uint4*>(Hs + r * 128 + ((unit ^ (r & 7)) << 4)) =
                make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
    };
    if (compute) {
        const float* h0 = p.h0 ? p.h0 + (static_cast<long long>(b) * dim + static_cast<long long>(h) * P) * NS : nullptr;
#pragma unroll
        for (int i = 0; i < PC; ++i) H[i] = h0 && r < NS ? __ldg(h0 + static_cast<long long>(cg * PC + i) * NS + r) : 0.f;
        store_hs();
    }

    // Per-step scalars of chunk c (control warp; lane l owns steps 4l .. 4l+3):
    // Delta_t, the running sum cs_t of Delta A (base 2) and
    // w_t = 2^(cs_end - cs_t) Delta_t, into float buffer c % 2.  The raw step
    // inputs of the next chunk are loaded one chunk ahead.
    const __nv_bfloat16* drow = p.delta + static_cast<long long>(bh) * L;
    auto load_raw = [&](int c, float (&raw)[4]) {
        const int t = c * Q + 4 * lane;
        if (t + 4 <= L) {
            const uint2 v = *reinterpret_cast<const uint2*>(drow + t);
            raw[0] = __uint_as_float(v.x << 16);
            raw[1] = __uint_as_float(v.x & 0xffff0000u);
            raw[2] = __uint_as_float(v.y << 16);
            raw[3] = __uint_as_float(v.y & 0xffff0000u);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) raw[k] = t + k < L ? __bfloat162float(drow[t + k]) : 0.f;
        }
    };
    float rawn[4] = {0.f, 0.f, 0.f, 0.f};
    auto chunk_scalars = [&](int c) {
        float* fb = fbase + (c & 1) * F_BUF;
        float2* cd = reinterpret_cast<float2*>(fb);
        float* wv = fb + 2 * Q;
        const int t = c * Q + 4 * lane;
        float dt[4], cs[4];
        float run = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            dt[k] = t + k < L ? softplus<false>(rawn[k] + bias) : 0.f;
            run = fmaf(dt[k], a2, run);
            cs[k] = run;
        }
        if (c + 1 < nch) load_raw(c + 1, rawn);  // in flight until the next call
        float v = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        const float before = v - run;  // the sum over the lanes before this one
        const float cs_end = __shfl_sync(0xffffffffu, v, 31);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float c_k = before + cs[k];
            cd[4 * lane + k] = make_float2(c_k, dt[k]);
            wv[4 * lane + k] = ex2_approx(cs_end - c_k) * dt[k];
        }
    };
    // w o x of chunk c (compute threads) as a bf16 head and a bf16 tail
    // holding the head's rounding error, so that the carried state keeps fp32
    // accuracy through the state contraction.
    auto weight_x = [&](int c) {
        const float* wv = fbase + (c & 1) * F_BUF + 2 * Q;
        mbar_wait(&x_bar[c % XBUFS], static_cast<uint32_t>((c / XBUFS) & 1), p.status);
        const unsigned char* Xs = smem + XS_OFF + (c % XBUFS) * XBUF;
#pragma unroll
        for (int item = tid; item < P * 16; item += COMPUTE) {
            const int row = item >> 4, unit = item & 15;
            const int half = unit >> 3, u8 = unit & 7;
            const uint32_t off = half * HALF_X + static_cast<uint32_t>(row * 128 + ((u8 ^ (row & 7)) << 4));
            const uint4 raw = *reinterpret_cast<const uint4*>(Xs + off);
            const int s0 = half * 64 + u8 * 8;
            const float4 wa = *reinterpret_cast<const float4*>(wv + s0);
            const float4 wb = *reinterpret_cast<const float4*>(wv + s0 + 4);
            const float ws[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            const uint32_t w32[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t oh[4], ol[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float v0 = __uint_as_float(w32[k] << 16) * ws[2 * k];
                const float v1 = __uint_as_float(w32[k] & 0xffff0000u) * ws[2 * k + 1];
                const __nv_bfloat162 ph = __floats2bfloat162_rn(v0, v1);
                const float2 fh = __bfloat1622float2(ph);
                oh[k] = *reinterpret_cast<const uint32_t*>(&ph);
                ol[k] = pack_bf2(v0 - fh.x, v1 - fh.y);
            }
            const uint32_t woff = half * HALF_W + static_cast<uint32_t>(row * 128 + ((u8 ^ (row & 7)) << 4));
            *reinterpret_cast<uint4*>(Xw + woff) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
            *reinterpret_cast<uint4*>(Xw + woff + P * 128) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
    };
    // G = C B^T and Yoff = C H_prev (into buffer c % 2) of chunk c, by the
    // control thread once C and B have landed (H_prev's bf16 copy written).
    auto issue_g_off = [&](int c) {
        mbar_wait(bc_bar, static_cast<uint32_t>(c & 1), p.status);
        tc_fence_after();
        const uint32_t cs_a = smem_addr(Cs), bs_a = smem_addr(Bs), hs_a = smem_addr(Hs);
        const uint32_t id_g = umma_idesc(Q, Q, true, true);
        const uint32_t id_off = umma_idesc(Q, P, true, true);
        const uint32_t tm_off = tmem + TM_YOFF + static_cast<uint32_t>((c & 1) * P);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {  // K = the N states, 16 rows per step
            const uint64_t ca = umma_desc(cs_a + ks * 2048, HALF_C, 1024);
            umma_f16(tmem + TM_G, ca, umma_desc(bs_a + ks * 2048, HALF_C, 1024), id_g, ks > 0);
            umma_f16(tm_off, ca, umma_desc(hs_a + ks * 2048, HALF_C, 1024), id_off, ks > 0);
        }
    };
    // S = B^T (w o x) of chunk c once its weighted x is written; the commit
    // covers every contraction of the chunk issued before it (G, Yoff, S).
    auto issue_s = [&](int c) {
        (void)c;
        tc_fence_after();
        const uint32_t bs_a = smem_addr(Bs);
        const uint32_t xw_a = smem_addr(Xw);
        const uint32_t id_s = umma_idesc(N, 2 * P, false, false);  // head and tail columns in one pass
#pragma unroll
        for (int ks = 0; ks < Q / 16; ++ks) {  // K = the chunk's steps
            const uint32_t koff = (ks & 3) * 32;  // 16 steps = 32 bytes into the 128-byte row
            const uint64_t ba = umma_desc(bs_a + (ks >> 2) * HALF_C + koff, 16, 1024);
            umma_f16(tmem + TM_S, ba, umma_desc(xw_a + (ks >> 2) * HALF_W + koff, 16, 1024), id_s, ks > 0);
        }
        umma_commit(mma1_bar);
    };

    if (!compute) {
        load_raw(0, rawn);
        chunk_scalars(0);
        if (nch > 1) chunk_scalars(1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = *tslot;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;  // this warp's TMEM lanes
    if (compute) weight_x(0);
    __syncthreads();
    if (tid == CTRL) {
        issue_g_off(0);
        issue_s(0);
    }

    for (int c = 0; c < nch; ++c) {
        const int t0 = c * Q;
        const int buf = c & 1;
        const float2* cd = reinterpret_cast<const float2*>(fbase + buf * F_BUF);
        const unsigned char* Xs = smem + XS_OFF + (c % XBUFS) * XBUF;
        // (B) G, S, Yoff of chunk c have landed; C and B are read, so the
        // next chunk's tiles load meanwhile.
        mbar_wait(mma1_bar, static_cast<uint32_t>(c & 1), p.status);
        tc_fence_after();
        float cs_t = 0.f;
        if (tid == CTRL) {
            if (c + 1 < nch) load_bc(c + 1);
            // The previous chunk's y has been read out of the z tile: this
            // chunk's z loads into it while the operands are built.
            if (c > 0) {
                bulk_wait_read<0>();
                if (has_z) load_z(c);
            }
        }
        if (compute) {
            cs_t = cd[r].x;
            // M = G o 2^(cs_t - cs_s) Delta_s (s <= t): rows t = r, columns
            // s = 32 cg .. 32 cg + 31 (a block above the diagonal is all
            // zero), into tensor-memory columns 16 cg .. 16 cg + 15 of M
            uint32_t m32[16];
            if (cg > qd) {
#pragma unroll
                for (int i = 0; i < 16; ++i) m32[i] = 0u;
            } else {
                float gv[32];
                tmem_ld32(tmem + lane_base + TM_G + cg * 32, gv);
                const bool diag = cg == qd;
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {  // four groups of 8 steps
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int i0 = u4 * 8 + 2 * k;
                        const int s0 = cg * 32 + i0;
                        const float4 cp = *reinterpret_cast<const float4*>(cd + s0);  // cs, Delta of s0, s0 + 1
                        float m0 = gv[i0] * ex2_approx(cs_t - cp.x) * cp.y;
                        float m1 = gv[i0 + 1] * ex2_approx(cs_t - cp.z) * cp.w;
                        if (diag) {
                            m0 = s0 <= r ? m0 : 0.f;
                            m1 = s0 + 1 <= r ? m1 : 0.f;
                        }
                        m32[u4 * 4 + k] = pack_bf2(m0, m1);
                    }
                }
            }
            tmem_st16(tmem + lane_base + TM_M + cg * 16, m32);
            // H = 2^cs_end H + S, state row n = r, channels PC cg .. PC cg + PC - 1,
            // and its bf16 copy
            const float decay_all = ex2_approx(cd[Q - 1].x);
            float sh[PC], sl[PC];
            tmem_ld16x2(tmem + lane_base + TM_S + cg * PC, tmem + lane_base + TM_S + P + cg * PC, sh, sl);
#pragma unroll
            for (int i = 0; i < PC; ++i) H[i] = fmaf(decay_all, H[i], sh[i] + sl[i]);
            store_hs();
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        // Ydiag = M x, then G and Yoff of the next chunk (G is read, H written),
        // by the control thread, and the step scalars of the chunk after it
        // (this chunk's scalars are read); meanwhile the compute threads
        // weight the next chunk's x
        if (tid == CTRL) {
            tc_fence_after();
            const uint32_t xs_a = smem_addr(Xs);
            const uint32_t id_d = umma_idesc(Q, P, false, false);
#pragma unroll
            for (int ks = 0; ks < Q / 16; ++ks) {  // M from tensor memory: 16 steps = 8 columns
                const uint32_t koff = (ks & 3) * 32;
                umma_f16_ta(tmem + TM_YD, tmem + TM_M + static_cast<uint32_t>(ks * 8),
                            umma_desc(xs_a + (ks >> 2) * HALF_X + koff, 16, 1024), id_d, ks > 0);
            }
            umma_commit(mma2_bar);
            if (c + 1 < nch) issue_g_off(c + 1);
        }
        if (c + 1 < nch) {
            if (compute) weight_x(c + 1);
            __syncthreads();
        }
        if (!compute) {
            // S of the next chunk while the compute threads form this chunk's
            // output; then the step scalars of the chunk after it
            if (tid == CTRL && c + 1 < nch) issue_s(c + 1);
            if (c + 2 < nch) chunk_scalars(c + 2);
        } else {
            // (C) y = (Ydiag + 2^cs_t Yoff + D x) * silu(z), row t = r, channels
            // PC cg .. PC cg + PC - 1, formed in the z tile in place (each
            // element is read and written by this thread only); steps past
            // the sequence's end are computed but not stored (the TMA store
            // clips them)
            const int half = r >> 6, tc = r & 63;
            float xv[PC];
#pragma unroll
            for (int i = 0; i < PC; ++i) xv[i] = bf_at(Xs, half * HALF_X + sw128_elem(cg * PC + i, tc));
            const float e_t = ex2_approx(cs_t);
            mbar_wait(mma2_bar, static_cast<uint32_t>(c & 1), p.status);
            tc_fence_after();
            float yd[PC], yo[PC];
            tmem_ld16x2(tmem + lane_base + TM_YD + cg * PC,
                        tmem + lane_base + TM_YOFF + static_cast<uint32_t>(buf * P + cg * PC), yd, yo);
            if (has_z) mbar_wait(z_bar, static_cast<uint32_t>(c & 1), p.status);
#pragma unroll
            for (int i = 0; i < PC; ++i) {
                const uint32_t off = half * HALF_X + sw128_elem(cg * PC + i, tc);
                float yv = fmaf(dsk, xv[i], fmaf(e_t, yo[i], yd[i]));
                if (has_z) yv *= silu_tanh(bf_at(Zs, off));
                bf_put(Zs, off, yv);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == CTRL) {
            // y of this chunk out of the z tile (the halves that start before
            // the sequence's end)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                if (t0 + half * 64 < L) tma_store_2d(&tm_y, t0 + half * 64, xrow, Zs + half * HALF_X);
            bulk_commit();
            // x of this buffer is read (Ydiag is done, and so is the output
            // step): chunk c + XBUFS loads into it.
            if (c + XBUFS < nch) load_x(c + XBUFS);
        }
    }
    if (tid == CTRL) bulk_wait<0>();
    if (p.h_final && compute && r < NS) {
        float* hf = p.h_final + (static_cast<long long>(b) * dim + static_cast<long long>(h) * P) * NS;
#pragma unroll
        for (int i = 0; i < PC; ++i) hf[static_cast<long long>(cg * PC + i) * NS + r] = H[i];
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

}  // namespace ssm
