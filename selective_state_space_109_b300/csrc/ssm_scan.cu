// ssm_scan.cu -- host side of libssmscan.so: the C ABI of include/ssm_scan.h.
//
// Each entry point validates its arguments without touching the GPU, picks a
// kernel variant for the shape (lanes per channel, chunking), and enqueues the
// launch on the caller's stream.  Nothing here computes on the host.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched from the driver at run time
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>
#include <cmath>
#include <mutex>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "../../include/ssm_scan.h"
#include "conv1d.cuh"
#include "scan_bwd.cuh"
#include "scan_fwd.cuh"
#include "decode_tma.cuh"
#include "scan_tma.cuh"
#include "scan_ws_api.h"
#include "state_update.cuh"

// The library's device error word (declared in tma.cuh): every kernel
// translation unit of the library shares this one definition.
namespace ssm {
__device__ unsigned int g_ssm_device_error = 0;
}

// Records a CUDA error for ssm_last_cuda_error (also used by the SSD
// translation unit) and returns the matching status.
ssm_status_t ssm_note_cuda_error(cudaError_t e);

namespace {

thread_local int g_last_cuda_error = 0;
// Events that scan calls from this host thread record around the launch of
// their fused pass (ssm_set_pass_timer); null when unset.
thread_local cudaEvent_t g_pass_begin = nullptr;
thread_local cudaEvent_t g_pass_end = nullptr;

void mark_pass_begin(cudaStream_t st) {
    if (g_pass_begin) cudaEventRecord(g_pass_begin, st);
}
void mark_pass_end(cudaStream_t st) {
    if (g_pass_end) cudaEventRecord(g_pass_end, st);
}

ssm_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return SSM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dstate(int n) { return n == 4 || n == 8 || n == 16 || n == 32 || n == 64 || n == 128 || n == 256; }


// Lanes that may share one channel's N states: each lane keeps an even number
// of them, at most 16 (the register budget of the update loop).
constexpr int min_lanes_for(int n) { return n > 16 ? n / 16 : 1; }

int env_int(const char* name, int fallback) {
    const char* s = std::getenv(name);
    if (!s || !*s) return fallback;
    return std::atoi(s);
}

// Argument checks shared by the scan entry points (no CUDA calls).
ssm_status_t check_scan_args(const void* u, const void* delta, const void* z, const float* A,
                             const void* B, const void* C, const float* Dskip,
                             const float* dt_bias, const void* y, const float* h0,
                             const float* h_final, int batch, int dim, int dstate, int seqlen,
                             int ngroups, ssm_dtype_t io) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0) return SSM_ERR_INVALID_ARG;
    if (dim % ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!A) return SSM_ERR_INVALID_ARG;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    // (batch * dim * seqlen) must index within 63 bits; rows are addressed in 64-bit.
    return SSM_OK;
}

// Lanes that split one channel's N states.  Enough lanes to give every SM
// about eight warps, no more (more lanes mean more reduce-scatter work).
int choose_lanes(int channels, int dstate, int num_sms) {
    const int max_lanes = dstate / 2;  // each lane keeps at least one fp32x2 pair
    const long long want = static_cast<long long>(num_sms) * 8 * 32;
    int lanes = 1;
    while (lanes < max_lanes && static_cast<long long>(channels) * lanes < want) lanes *= 2;
    return lanes;
}

int device_sm_count() {
    static thread_local int cached_dev = -1;
    static thread_local int cached_sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cached_sms;
    if (dev != cached_dev) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            cached_sms = sms;
        cached_dev = dev;
    }
    return cached_sms;
}

// Opts a kernel into its dynamic shared memory once per device.
template <typename K>
cudaError_t ensure_smem(K kern, int bytes, unsigned long long* done_mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
    return e;
}

constexpr int kScanWarps = 4;
// Steps per staged B/C tile of the generic kernel: 64, or 32 for N = 64 and
// 128 (fp32 B/C quads of 64 steps would not fit), 64 again at N = 256 (16
// lanes of 4 steps: one warp block).  From N = 128 on the tile is held in
// dynamic shared memory, single-buffered (32 KB at N = 128, 128 KB at 256).
template <int N>
constexpr int scan_tile() { return N >= 256 ? 64 : (N >= 64 ? 32 : 64); }

template <typename T, int N, int LANES>
cudaError_t launch_scan_variant(ssm::ScanParams p, cudaStream_t st) {
    constexpr int CH = kScanWarps * (32 / LANES);
    constexpr int V = ssm::ScanShape<T, LANES>::V;
    constexpr int VE = ssm::Elem<T>::kPer16B;
    p.blocks_per_group = (p.dim_per_group + CH - 1) / CH;
    p.vec_ok = (p.seqlen % V) == 0;
    p.bc_vec_ok = (p.seqlen % VE) == 0;
    const long long blocks = static_cast<long long>(p.blocks_per_group) * p.ngroups * p.batch;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    constexpr bool kAccurate = sizeof(T) == 4;
    auto kern = ssm::scan_fwd_kernel<T, N, LANES, kScanWarps, scan_tile<N>(), kAccurate>;
    int dyn = 0;
    if constexpr (ssm::scan_bc_dynamic(N)) {
        dyn = scan_tile<N>() * (N / 2) * 16;
        static unsigned long long done = 0;
        const cudaError_t e = ensure_smem(kern, dyn, &done);
        if (e != cudaSuccess) return e;
    }
    kern<<<static_cast<unsigned>(blocks), kScanWarps * 32, dyn, st>>>(p);
    return cudaGetLastError();
}

// Lanes per channel of the generic kernel: 2 to 16 states each.
template <typename T, int N>
cudaError_t launch_scan_n(const ssm::ScanParams& p, int lanes, cudaStream_t st) {
    switch (lanes) {
        case 1: if constexpr (N <= 16) return launch_scan_variant<T, N, 1>(p, st); break;
        case 2: if constexpr (N <= 32) return launch_scan_variant<T, N, 2>(p, st); break;
        case 4: if constexpr (N >= 8 && N <= 64) return launch_scan_variant<T, N, 4>(p, st); break;
        case 8: if constexpr (N >= 16 && N <= 128) return launch_scan_variant<T, N, 8>(p, st); break;
        case 16: if constexpr (N == 256) return launch_scan_variant<T, N, 16>(p, st); break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_scan_t(const ssm::ScanParams& p, int dstate, int lanes, cudaStream_t st) {
    switch (dstate) {
        case 4: return launch_scan_n<T, 4>(p, lanes, st);
        case 8: return launch_scan_n<T, 8>(p, lanes, st);
        case 16: return launch_scan_n<T, 16>(p, lanes, st);
        case 32: return launch_scan_n<T, 32>(p, lanes, st);
        case 64: return launch_scan_n<T, 64>(p, lanes, st);
        case 128: return launch_scan_n<T, 128>(p, lanes, st);
        case 256: return launch_scan_n<T, 256>(p, lanes, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// TMA-staged path
// ---------------------------------------------------------------------------

constexpr int kTmaWarps = 4;
// The time-chunk plan aims to fill a B300 (148 SMs).  It is a function of the
// problem's arguments only, so the workspace size query needs no device.
constexpr int kPlanSms = 148;
constexpr int kMaxChunks = 64;

// Workspace header: the device-side status word written by kernels that wait.
constexpr size_t kWorkspaceHeader = 256;

int tma_steps_per_tile(ssm_dtype_t io) { return ssm::kScanRowBytes / (io == SSM_F32 ? 4 : 2); }

// Rows of every tensor must start on 16-byte boundaries for TMA.
bool tma_eligible(int seqlen, ssm_dtype_t io) {
    const int es = io == SSM_F32 ? 4 : 2;
    return seqlen > 0 && (static_cast<long long>(seqlen) * es) % 16 == 0;
}

int max_chunks_for(int seqlen, ssm_dtype_t io) {
    const int ntiles = (seqlen + tma_steps_per_tile(io) - 1) / tma_steps_per_tile(io);
    return std::max(1, std::min(kMaxChunks, ntiles));
}

struct ScanPlan {
    int lanes;
    int chunks;
    int agg_lanes;  // lanes of the summary pass (chunks > 1)
};

template <typename T, int N, ssm::ScanMode MODE>
int tma_smem_bytes(int lanes) {
    constexpr int L1 = N <= 16 ? 1 : N / 16;  // lanes the TMA kernel is built with for this N
    switch (lanes) {
        case 1: return ssm::TmaScanLayout<T, N, L1, kTmaWarps, MODE>::SMEM_BYTES;
        case 2: return ssm::TmaScanLayout<T, N, (N <= 32 ? 2 : L1), kTmaWarps, MODE>::SMEM_BYTES;
        case 8: return ssm::TmaScanLayout<T, N, (N == 128 ? 8 : L1), kTmaWarps, MODE>::SMEM_BYTES;
        case 16: return ssm::TmaScanLayout<T, N, (N == 256 ? 16 : L1), kTmaWarps, MODE>::SMEM_BYTES;
        default: return ssm::TmaScanLayout<T, N, (N >= 8 ? (N <= 64 ? 4 : L1) : 2), kTmaWarps, MODE>::SMEM_BYTES;
    }
}

template <ssm::ScanMode MODE>
int tma_smem_for(ssm_dtype_t io, int dstate, int lanes) {
    if (io == SSM_F32) {
        if (dstate == 32) return tma_smem_bytes<float, 32, MODE>(lanes);
        if (dstate == 64) return tma_smem_bytes<float, 64, MODE>(lanes);
        if (dstate == 128) return tma_smem_bytes<float, 128, MODE>(lanes);
        if (dstate == 256) return tma_smem_bytes<float, 256, MODE>(lanes);
        return dstate == 4 ? tma_smem_bytes<float, 4, MODE>(lanes)
                           : dstate == 8 ? tma_smem_bytes<float, 8, MODE>(lanes) : tma_smem_bytes<float, 16, MODE>(lanes);
    }
    if (dstate == 32) return tma_smem_bytes<__nv_bfloat16, 32, MODE>(lanes);
    if (dstate == 64) return tma_smem_bytes<__nv_bfloat16, 64, MODE>(lanes);
    if (dstate == 128) return tma_smem_bytes<__nv_bfloat16, 128, MODE>(lanes);
    if (dstate == 256) return tma_smem_bytes<__nv_bfloat16, 256, MODE>(lanes);
    return dstate == 4 ? tma_smem_bytes<__nv_bfloat16, 4, MODE>(lanes)
                       : dstate == 8 ? tma_smem_bytes<__nv_bfloat16, 8, MODE>(lanes)
                                     : tma_smem_bytes<__nv_bfloat16, 16, MODE>(lanes);
}

// CTAs that fit on one SM by shared memory (228 KB per SM, 1 KB of it
// reserved per CTA), at most the kMaxCtasPerSm that the kernels' launch
// bounds plan registers for.
int ctas_per_sm(int smem_bytes) {
    return std::max(1, std::min(ssm::kMaxCtasPerSm, (228 * 1024) / (smem_bytes + 1024)));
}

// Relative SM throughput with c resident CTAs (c warps per scheduler), from a
// measurement of the scan's update mix on B300: one warp per scheduler
// reaches about half the saturated rate, two about 0.8, three 0.9.
double sm_efficiency(long long c) {
    static const double e[5] = {0.0, 0.48, 0.8, 0.9, 1.0};
    return c >= 4 ? 1.0 : e[c];
}

// Time (arbitrary units) of one pass: `ctas` CTAs of `work` each over kPlanSms
// SMs, `cap` resident per SM; the busiest SM runs full waves of `cap` CTAs and
// then its remainder.
double pass_time(long long ctas, int cap, double work) {
    const long long nmax = (ctas + kPlanSms - 1) / kPlanSms;
    const long long full = nmax / cap, rest = nmax % cap;
    double t = static_cast<double>(full) * cap * work / sm_efficiency(cap);
    if (rest > 0) t += static_cast<double>(rest) * work / sm_efficiency(rest);
    return t;
}

// Time of one step of a CTA whose lanes hold S states each (units below): a
// fixed part per step (softplus, the Delta exchange, the readout and gate)
// plus a part per state, plus the cross-lane reduction at 4 lanes.  Fitted to
// B300 timings at N = 16, 32 and 64 over 1, 2 and 4 lanes; the summary pass
// has no readout and a smaller fixed part.
double step_time(int S, int lanes, bool summary) {
    const double shared = lanes >= 4 ? 12.8 : 0.0;
    return summary ? 12.8 + 7.2 * S + shared : 25.6 + 6.4 * S + shared;
}

// Picks lanes per channel and time chunks by a wave model of the two passes,
// fitted to B300 timings of the bf16 scan workloads over plans of 1 to 32
// chunks and 1, 2 or 4 lanes.  The summary pass costs 0.9 of its step time;
// the two extra kernels cost about 2 us, and each chunk about 0.65 us more
// (every chunk's CTAs fetch their first tiles at once when the kernel starts).
ScanPlan plan_scan(int batch, int dim, int dstate, int seqlen, int ngroups, ssm_dtype_t io,
                   int chunk_cap) {
    const int dpg = dim / ngroups;
    const int kmax = std::max(1, std::min(chunk_cap, max_chunks_for(seqlen, io)));
    const int lmax = dstate >= 128 ? dstate / 16 : (dstate >= 8 ? 4 : 2);
    const int lmin = min_lanes_for(dstate);
    // Time units: ~0.54 ns of an SM each on B300 (one step of a CTA of
    // 16-state lanes is 128 units).
    const double launch_units = 2000.0 / 0.54;
    const double chunk_units = 650.0 / 0.54;
    ScanPlan best{lmin, 1, lmin};
    double best_cost = 1e300;
    for (int lanes = lmin; lanes <= lmax; lanes *= 2) {
        const int ch = kTmaWarps * 32 / lanes;
        const long long blocks = static_cast<long long>((dpg + ch - 1) / ch) * ngroups * batch;
        const int cap_full = ctas_per_sm(tma_smem_for<ssm::ScanMode::Full>(io, dstate, lanes));
        for (int k = 1; k <= kmax; ++k) {
            const double steps = static_cast<double>(seqlen) / k;
            double cost = pass_time(blocks * k, cap_full, step_time(dstate / lanes, lanes, false) * steps);
            int best_agg = lanes;
            if (k > 1) {
                // The summary pass picks its own lanes (no readout to reduce:
                // cheaper lane sharing).
                double agg_cost = 1e300;
                for (int la = lmin; la <= lmax; la *= 2) {
                    const int cha = kTmaWarps * 32 / la;
                    const long long blocks_a = static_cast<long long>((dpg + cha - 1) / cha) * ngroups * batch;
                    const int cap_agg = ctas_per_sm(tma_smem_for<ssm::ScanMode::Aggregate>(io, dstate, la));
                    const double c = pass_time(blocks_a * (k - 1), cap_agg, 0.9 * step_time(dstate / la, la, true) * steps);
                    if (c < agg_cost * 0.999) {
                        agg_cost = c;
                        best_agg = la;
                    }
                }
                cost += agg_cost + launch_units + chunk_units * k;
            }
            if (cost < best_cost * 0.999) {
                best_cost = cost;
                best = {lanes, k, best_agg};
            }
        }
    }
    // At N <= 16 the summary pass runs with the fewest lanes the states allow:
    // measured best on both chunked N = 16 plans (b2 d1536 L2048: 66.1 us
    // against 68.3 and 71.8 at 2 and 4 lanes; b1 d5120 L65536: 2226 us
    // against 2407 and 2618), where the cost model above preferred 2 lanes
    // for the first.
    if (best.chunks > 1 && dstate <= 16) best.agg_lanes = lmin;
    // At 16 lanes a channel (N = 256) the model prices the summary pass like
    // the fused pass, but it has no readout to reduce across the 16 lanes.
    // When one pass would leave SMs short of three resident CTAs (the fused
    // pass's 148 registers allow three), a split into three chunks measured
    // best: b2 d1536 L2048 bf16, 872 us against 938 us in one pass (884 at
    // two chunks, 903 at four, 878 at six).
    if (dstate >= 256 && io != SSM_F32 && best.chunks == 1 && kmax >= 3) {
        const int ch = kTmaWarps * 32 / best.lanes;
        const long long blocks = static_cast<long long>((dpg + ch - 1) / ch) * ngroups * batch;
        if (blocks < 3LL * kPlanSms) {
            best.chunks = 3;
            best.agg_lanes = best.lanes;
        }
    }
    const int fl = env_int("SSM_FORCE_LANES", 0);
    if ((fl == 1 || fl == 2 || fl == 4) && fl <= lmax && fl >= lmin) best.lanes = fl;
    const int fk = env_int("SSM_FORCE_CHUNKS", 0);
    if (fk >= 1) best.chunks = std::min(fk, kmax);
    if (fl || fk) best.agg_lanes = best.lanes;
    const int fa = env_int("SSM_FORCE_AGG_LANES", 0);
    if ((fa == 1 || fa == 2 || fa == 4) && fa <= lmax && fa >= lmin) best.agg_lanes = fa;
    return best;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

struct ScanMaps {
    CUtensorMap u, d, z, y, B, C;
};

// [batch * ngroups, dim_per_group, seqlen] activation view; box = one tile of
// kScanRowBytes per row times `rows` channels, swizzled at that row width.
bool encode_act(CUtensorMap* m, const void* ptr, ssm_dtype_t io, int seqlen, int dpg, long long bg, int rows,
                int row_bytes = ssm::kScanRowBytes) {
    const cuuint64_t es = io == SSM_F32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(seqlen), static_cast<cuuint64_t>(dpg),
                                static_cast<cuuint64_t>(bg)};
    const cuuint64_t strides[2] = {seqlen * es, seqlen * es * dpg};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(row_bytes / es), static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                     : CU_TENSOR_MAP_SWIZZLE_32B;
    return encode_tiled()(m, io == SSM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [batch * ngroups * dstate, seqlen] view of B or C; box = one tile x dstate rows.
bool encode_bc(CUtensorMap* m, const void* ptr, ssm_dtype_t io, int seqlen, long long rows, int dstate,
               int row_bytes = ssm::kScanRowBytes) {
    const cuuint64_t es = io == SSM_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(seqlen), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {seqlen * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes / es), static_cast<cuuint32_t>(dstate)};
    const cuuint32_t estr[2] = {1, 1};
    return encode_tiled()(m, io == SSM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


template <typename T, int N, int LANES, ssm::ScanMode MODE>
cudaError_t launch_tma(const ScanMaps& m, const ssm::TmaScanParams& p, int grid_y, cudaStream_t st) {
    using Lay = ssm::TmaScanLayout<T, N, LANES, kTmaWarps, MODE>;
    auto kern = ssm::scan_tma_kernel<T, N, LANES, kTmaWarps, MODE, sizeof(T) == 4>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem(kern, Lay::SMEM_BYTES, &done);
    if (e != cudaSuccess) return e;
    const long long gx = static_cast<long long>(p.blocks_per_group) * p.ngroups * p.batch;
    if (gx > 0x7fffffffLL || grid_y > 65535) return cudaErrorInvalidConfiguration;
    // The full pass of a chunked call follows the carry pass: launch it with
    // programmatic stream serialization so that its prologue (barriers, the
    // first input tiles) overlaps that pass; it waits before reading the carry.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(grid_y));
    cfg.blockDim = dim3(kTmaWarps * 32);
    cfg.dynamicSmemBytes = Lay::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    const bool pdl = MODE == ssm::ScanMode::Full && p.nchunks > 1;
    cfg.attrs = pdl ? &attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, m.u, m.d, m.z, m.y, m.B, m.C, p);
}

template <typename T, int N, ssm::ScanMode MODE>
cudaError_t launch_tma_lanes(const ScanMaps& m, const ssm::TmaScanParams& p, int lanes, int grid_y,
                             cudaStream_t st) {
    switch (lanes) {
        case 1: if constexpr (N <= 16) return launch_tma<T, N, 1, MODE>(m, p, grid_y, st); break;
        case 2: if constexpr (N <= 32) return launch_tma<T, N, 2, MODE>(m, p, grid_y, st); break;
        case 4: if constexpr (N >= 8 && N <= 64) return launch_tma<T, N, 4, MODE>(m, p, grid_y, st); break;
        case 8: if constexpr (N == 128) return launch_tma<T, N, 8, MODE>(m, p, grid_y, st); break;
        case 16: if constexpr (N == 256) return launch_tma<T, N, 16, MODE>(m, p, grid_y, st); break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <typename T, ssm::ScanMode MODE>
cudaError_t launch_tma_n(const ScanMaps& m, const ssm::TmaScanParams& p, int dstate, int lanes, int grid_y,
                         cudaStream_t st) {
    switch (dstate) {
        case 4: return launch_tma_lanes<T, 4, MODE>(m, p, lanes, grid_y, st);
        case 8: return launch_tma_lanes<T, 8, MODE>(m, p, lanes, grid_y, st);
        case 16: return launch_tma_lanes<T, 16, MODE>(m, p, lanes, grid_y, st);
        case 32: return launch_tma_lanes<T, 32, MODE>(m, p, lanes, grid_y, st);
        case 64: return launch_tma_lanes<T, 64, MODE>(m, p, lanes, grid_y, st);
        case 128: return launch_tma_lanes<T, 128, MODE>(m, p, lanes, grid_y, st);
        case 256: return launch_tma_lanes<T, 256, MODE>(m, p, lanes, grid_y, st);
        default: return cudaErrorInvalidValue;
    }
}

// The carry pass between the summary and fused passes: one thread per
// (channel, state pair); it waits for the summary pass in-kernel (programmatic
// stream serialization), so its launch overlaps that pass's tail.
cudaError_t launch_carry(float* agg, const float* h0, int batch, int dim, int dstate, int chunks, cudaStream_t st) {
    const long long BD = static_cast<long long>(batch) * dim;
    const long long threads = BD * (dstate / 2);
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    switch (dstate) {
        case 4: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<4, kMaxChunks>, agg, h0, BD, chunks);
        case 8: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<8, kMaxChunks>, agg, h0, BD, chunks);
        case 16: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<16, kMaxChunks>, agg, h0, BD, chunks);
        case 32: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<32, kMaxChunks>, agg, h0, BD, chunks);
        case 64: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<64, kMaxChunks>, agg, h0, BD, chunks);
        case 128: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<128, kMaxChunks>, agg, h0, BD, chunks);
        case 256: return cudaLaunchKernelEx(&cfg, ssm::scan_carry_kernel<256, kMaxChunks>, agg, h0, BD, chunks);
        default: return cudaErrorInvalidValue;
    }
}

int ws_smem(ssm_dtype_t io, int dstate, int lanes, int nw, int seg = 1);
bool ws_encode(ssm::WsMaps* m, const void* u, const void* delta, const void* z, const void* B, const void* C,
               ssm_dtype_t io, int seqlen, int dpg, long long bg, int dstate, int ch, int rb);

// SSM_FUSED_KERNEL=ws runs the fused pass of chunked plans on the
// warp-specialised kernel.
bool fused_ws_enabled() {
    const char* v = std::getenv("SSM_FUSED_KERNEL");
    return v && std::strcmp(v, "ws") == 0;
}

// Enqueues the staged scan: with plan.chunks > 1 the summary pass over all
// chunks but the last, then the full pass over every chunk.
ssm_status_t run_scan_tma(const void* u, const void* delta, const void* z, const float* A, const void* B,
                          const void* C, const float* Dskip, const float* dt_bias, const float* h0, void* y,
                          float* h_final, int batch, int dim, int dstate, int seqlen, int ngroups,
                          ssm_dtype_t io, const ScanPlan& plan, float* agg, unsigned int* status,
                          cudaStream_t st) {
    if (!encode_tiled()) return cuda_fail(cudaErrorNotSupported);
    const int dpg = dim / ngroups;
    const long long bg = static_cast<long long>(batch) * ngroups;
    const int ch = kTmaWarps * 32 / plan.lanes;
    ScanMaps m;
    const bool ok = encode_act(&m.u, u, io, seqlen, dpg, bg, ch) && encode_act(&m.d, delta, io, seqlen, dpg, bg, ch) &&
                    encode_act(&m.y, y, io, seqlen, dpg, bg, ch) &&
                    (z ? encode_act(&m.z, z, io, seqlen, dpg, bg, ch) : true) &&
                    encode_bc(&m.B, B, io, seqlen, bg * dstate, dstate) &&
                    encode_bc(&m.C, C, io, seqlen, bg * dstate, dstate);
    if (!ok) return cuda_fail(cudaErrorInvalidValue);
    if (!z) m.z = m.u;  // never read: has_z = 0

    ssm::TmaScanParams p{};
    p.A = A; p.D = Dskip; p.dt_bias = dt_bias; p.h0 = h0; p.h_final = h_final;
    p.agg = agg; p.status = status;
    p.batch = batch; p.dim = dim; p.seqlen = seqlen; p.ngroups = ngroups; p.dim_per_group = dpg;
    p.blocks_per_group = (dpg + ch - 1) / ch;
    p.nchunks = plan.chunks;
    p.ntiles = (seqlen + tma_steps_per_tile(io) - 1) / tma_steps_per_tile(io);
    p.has_z = z != nullptr;

    cudaError_t e = cudaSuccess;
    if (plan.chunks > 1) {
        // The summary pass may share a channel's states over more lanes than
        // the full pass (it has no readout to reduce): more resident warps.
        int agg_lanes = plan.agg_lanes;
        ScanMaps ma = m;
        ssm::TmaScanParams pa = p;
        if (agg_lanes != plan.lanes) {
            const int cha = kTmaWarps * 32 / agg_lanes;
            if (!encode_act(&ma.u, u, io, seqlen, dpg, bg, cha) || !encode_act(&ma.d, delta, io, seqlen, dpg, bg, cha))
                return cuda_fail(cudaErrorInvalidValue);
            pa.blocks_per_group = (dpg + cha - 1) / cha;
        }
        e = io == SSM_F32 ? launch_tma_n<float, ssm::ScanMode::Aggregate>(ma, pa, dstate, agg_lanes, plan.chunks - 1, st)
                          : launch_tma_n<__nv_bfloat16, ssm::ScanMode::Aggregate>(ma, pa, dstate, agg_lanes,
                                                                                  plan.chunks - 1, st);
        if (e != cudaSuccess) return cuda_fail(e);
        e = launch_carry(agg, h0, batch, dim, dstate, plan.chunks, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (plan.chunks > 1 && fused_ws_enabled() && ws_smem(io, dstate, plan.lanes, 4) > 0) {
        // The fused pass of the chunked call on the warp-specialised kernel.
        ssm::WsMaps wm;
        const int wch = 4 * 32 / plan.lanes;
        if (!ws_encode(&wm, u, delta, z, B, C, io, seqlen, dpg, bg, dstate, wch, ssm::kScanRowBytes))
            return cuda_fail(cudaErrorInvalidValue);
        ssm::WsScanParams wp{};
        wp.A = A; wp.D = Dskip; wp.dt_bias = dt_bias; wp.h0 = h0; wp.h_final = h_final; wp.y = y;
        wp.status = status;
        wp.batch = batch; wp.dim = dim; wp.seqlen = seqlen; wp.ngroups = ngroups; wp.dim_per_group = dpg;
        wp.blocks_per_group = (dpg + wch - 1) / wch;
        wp.ntiles = p.ntiles;
        wp.has_z = z != nullptr;
        wp.stop_tile = -1;
        wp.wait_budget_ns = ssm::kWaitBudgetNs;
        wp.carry = agg;
        wp.nchunks = plan.chunks;
        mark_pass_begin(st);
        e = io == SSM_F32 ? ssm::ws_launch_f32(dstate, plan.lanes, 4, 1, wm, wp, st)
                          : ssm::ws_launch_bf16(dstate, plan.lanes, 4, 1, wm, wp, st);
        if (e != cudaSuccess) return cuda_fail(e);
        mark_pass_end(st);
        return SSM_OK;
    }
    mark_pass_begin(st);
    e = io == SSM_F32 ? launch_tma_n<float, ssm::ScanMode::Full>(m, p, dstate, plan.lanes, plan.chunks, st)
                      : launch_tma_n<__nv_bfloat16, ssm::ScanMode::Full>(m, p, dstate, plan.lanes, plan.chunks, st);
    if (e != cudaSuccess) return cuda_fail(e);
    mark_pass_end(st);
    return SSM_OK;
}

// ---------------------------------------------------------------------------
// Warp-specialised scan (scan_ws.cuh): plan and launch
// ---------------------------------------------------------------------------

struct WsPlan {
    int lanes;  // lanes per channel (the state split)
    int nw;     // consumer warps per CTA
    int seg;    // time segments per channel inside a warp (1: none)
};

// Bytes of a tile row of the warp-specialised pass: 32, or 16 per segment.
int ws_row_bytes(int seg) { return seg > 1 ? 16 * seg : ssm::kScanRowBytes; }

int ws_smem(ssm_dtype_t io, int dstate, int lanes, int nw, int seg) {
    return io == SSM_F32 ? ssm::ws_smem_bytes_f32(dstate, lanes, nw, seg)
                         : ssm::ws_smem_bytes_bf16(dstate, lanes, nw, seg);
}

// Plans that run one pass over the whole sequence (no time split) take the
// warp-specialised kernel (scan_ws.cuh): measured 407 us against 455 us for
// the CTA-synchronous fused pass on bf16 b8 d2048 L4096 (2 lanes), and 1-4%
// faster at N = 128 (at N = 256 it measured 1.25 ms against 0.93 ms, so that
// state size keeps the CTA-synchronous pass).  Chunked plans keep the CTA-synchronous passes,
// which measured faster there (b1 d5120 L65536: 2.20 ms against 2.58 ms for
// the best chunked plan of the warp-specialised kernel).  Consumer warps per
// CTA: two when four would leave SMs without a CTA (four measured 399 us
// against 407 us for two on b8 d2048 L4096, 256 CTAs of four).
// SSM_SCAN_KERNEL=tma forces the CTA-synchronous kernel (for comparisons).
bool ws_single_pass(int batch, int dim, int dstate, int ngroups, ssm_dtype_t io, const ScanPlan& plan,
                    WsPlan* out) {
    const char* v = std::getenv("SSM_SCAN_KERNEL");
    if (v && std::strcmp(v, "tma") == 0) return false;
    if (plan.chunks != 1 || dstate > 128) return false;  // N = 256: the CTA-synchronous pass measured faster
    const int dpg = dim / ngroups;
    auto ctas = [&](int nw) {
        const int ch = nw * 32 / plan.lanes;
        return static_cast<long long>((dpg + ch - 1) / ch) * ngroups * batch;
    };
    int nw = ctas(4) < kPlanSms ? 2 : 4;
    const int fnw = env_int("SSM_FORCE_NW", 0);
    if (fnw == 2 || fnw == 4 || fnw == 8) nw = fnw;
    if (ws_smem(io, dstate, plan.lanes, nw) <= 0) nw = 4;
    if (ws_smem(io, dstate, plan.lanes, nw) <= 0) return false;
    *out = WsPlan{plan.lanes, nw, 1};
    return true;
}

// SSM_FORCE_SEG=s (with SSM_FORCE_LANES=l) runs the time-segmented variant of
// the warp-specialised pass -- the whole sequence in one kernel, time split
// inside each warp by an associative scan -- in place of any other plan.
bool ws_segmented_forced(ssm_dtype_t io, int dstate, WsPlan* out) {
    const int seg = env_int("SSM_FORCE_SEG", 0);
    if (seg <= 1) return false;
    const int lanes = env_int("SSM_FORCE_LANES", 2);
    if (ws_smem(io, dstate, lanes, 4, seg) <= 0) return false;
    *out = WsPlan{lanes, 4, seg};
    return true;
}

// Encodes the TMA views of one pass whose CTAs hold `ch` channels.
bool ws_encode(ssm::WsMaps* m, const void* u, const void* delta, const void* z, const void* B, const void* C,
               ssm_dtype_t io, int seqlen, int dpg, long long bg, int dstate, int ch, int rb) {
    const bool ok = encode_act(&m->u, u, io, seqlen, dpg, bg, ch, rb) &&
                    encode_act(&m->d, delta, io, seqlen, dpg, bg, ch, rb) &&
                    (z ? encode_act(&m->z, z, io, seqlen, dpg, bg, ch, rb) : true) &&
                    encode_bc(&m->B, B, io, seqlen, bg * dstate, dstate, rb) &&
                    encode_bc(&m->C, C, io, seqlen, bg * dstate, dstate, rb);
    if (ok && !z) m->z = m->u;  // never read: has_z = 0
    return ok;
}

// Enqueues the warp-specialised scan: one fused pass over the whole sequence
// (from h0, final state written when asked).
ssm_status_t run_scan_ws(const void* u, const void* delta, const void* z, const float* A, const void* B,
                         const void* C, const float* Dskip, const float* dt_bias, const float* h0, void* y,
                         float* h_final, int batch, int dim, int dstate, int seqlen, int ngroups,
                         ssm_dtype_t io, const WsPlan& plan, unsigned int* status, cudaStream_t st) {
    if (!encode_tiled()) return cuda_fail(cudaErrorNotSupported);
    const int dpg = dim / ngroups;
    const long long bg = static_cast<long long>(batch) * ngroups;
    const int ch = plan.nw * 32 / (plan.lanes * plan.seg);
    const int rb = ws_row_bytes(plan.seg);
    const int ts = rb / (io == SSM_F32 ? 4 : 2);
    ssm::WsMaps m;
    if (!ws_encode(&m, u, delta, z, B, C, io, seqlen, dpg, bg, dstate, ch, rb))
        return cuda_fail(cudaErrorInvalidValue);
    ssm::WsScanParams p{};
    p.A = A; p.D = Dskip; p.dt_bias = dt_bias; p.h0 = h0; p.h_final = h_final; p.y = y;
    p.status = status;
    p.batch = batch; p.dim = dim; p.seqlen = seqlen; p.ngroups = ngroups; p.dim_per_group = dpg;
    p.blocks_per_group = (dpg + ch - 1) / ch;
    p.ntiles = (seqlen + ts - 1) / ts;
    p.has_z = z != nullptr;
    // Failure injection for the tests of the bounded waits (off unless set):
    // the producer stops loading at tile SSM_DEBUG_STOP_LOADS_AT_TILE, and the
    // waits give up after SSM_DEBUG_WAIT_BUDGET_US microseconds.
    p.stop_tile = env_int("SSM_DEBUG_STOP_LOADS_AT_TILE", -1);
    const int budget_us = env_int("SSM_DEBUG_WAIT_BUDGET_US", 0);
    p.wait_budget_ns = budget_us > 0 ? static_cast<unsigned long long>(budget_us) * 1000ull : ssm::kWaitBudgetNs;
    p.carry = nullptr;
    p.nchunks = 1;
    mark_pass_begin(st);
    const cudaError_t e = io == SSM_F32 ? ssm::ws_launch_f32(dstate, plan.lanes, plan.nw, plan.seg, m, p, st)
                                        : ssm::ws_launch_bf16(dstate, plan.lanes, plan.nw, plan.seg, m, p, st);
    if (e != cudaSuccess) return cuda_fail(e);
    mark_pass_end(st);
    return SSM_OK;
}

// The TMA-staged decode needs N = 16, token rows that start on 16-byte
// boundaries, and channel blocks of 128 that stay inside one group.
bool decode_tma_eligible(int batch, int dim, int dstate, int ngroups, ssm_dtype_t io) {
    const int es = io == SSM_F32 ? 4 : 2;
    const int dpg = dim / ngroups;
    return batch > 0 && dstate == 16 && (static_cast<long long>(dim) * es) % 16 == 0 &&
           (ngroups == 1 || dpg % 128 == 0);
}

// The bulk-staged decode runs the warp-specialised kernel (decode_ws_kernel):
// measured 31.5-31.8 us against 32.8-33.0 us for the CTA-synchronous one on
// batch 256 x 5120 channels with the state cold in HBM (82% against 79% of
// the measured copy); with the state resident in L2 it is slower (27.2
// against 24.8 us).  SSM_DECODE_KERNEL=tma selects the CTA-synchronous kernel.
bool decode_ws_enabled() {
    const char* v = std::getenv("SSM_DECODE_KERNEL");
    return !(v && std::strcmp(v, "tma") == 0);
}

template <typename T, int CH, int STAGES>
cudaError_t launch_decode_tma_v(float* state, const int* slots, int nslots, const void* u, const void* delta,
                                const void* z, const float* A, const void* B, const void* C, const float* Dskip,
                                const float* dt_bias, void* y, int batch, int dim, int ngroups, cudaStream_t st) {
    using Lay = ssm::DecodeTmaLayout<T, CH, STAGES>;
    constexpr int N = Lay::N;
    if (!encode_tiled()) return cudaErrorNotSupported;
    const bool f32 = sizeof(T) == 4;
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t es = sizeof(T);
    const cuuint32_t e1[3] = {1, 1, 1};
    CUtensorMap ms, mu, md, mz, mB, mC;
    {  // state [nslots, dim, N] fp32, box [N, CH, 1], 64-byte swizzle
        const cuuint64_t dims[3] = {N, static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(nslots)};
        const cuuint64_t str[2] = {N * 4, static_cast<cuuint64_t>(dim) * N * 4};
        const cuuint32_t box[3] = {N, Lay::CH, 1};
        if (encode_tiled()(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, state, dims, str, box, e1,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    auto tok = [&](CUtensorMap* m, const void* ptr) {  // [batch, dim], box [CH, 1]
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(batch)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(dim) * es};
        const cuuint32_t box[2] = {Lay::CH, 1};
        return encode_tiled()(m, dt, 2, const_cast<void*>(ptr), dims, str, box, e1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto bc = [&](CUtensorMap* m, const void* ptr) {  // [batch * ngroups, N], box [N, 1]
        const cuuint64_t dims[2] = {N, static_cast<cuuint64_t>(batch) * ngroups};
        const cuuint64_t str[1] = {N * es};
        const cuuint32_t box[2] = {N, 1};
        return encode_tiled()(m, dt, 2, const_cast<void*>(ptr), dims, str, box, e1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (!tok(&mu, u) || !tok(&md, delta) || (z && !tok(&mz, z)) || !bc(&mB, B) || !bc(&mC, C))
        return cudaErrorInvalidValue;
    if (!z) mz = mu;  // never read: has_z = 0

    ssm::DecodeTmaParams p{};
    p.A = A; p.D = Dskip; p.dt_bias = dt_bias; p.y = y;
    p.batch = batch; p.dim = dim; p.ngroups = ngroups; p.dim_per_group = dim / ngroups;
    p.nblk = (dim + Lay::CH - 1) / Lay::CH;
    p.ntiles = static_cast<long long>(p.nblk) * batch;
    p.has_z = z != nullptr;
    p.slots = slots;
    p.nslots = nslots;

    if (decode_ws_enabled()) {
        // Warp-specialised kernel: the state block also leaves by 32-row boxes.
        using WLay = ssm::DecodeWsLayout<T, CH, STAGES>;
        CUtensorMap mso;
        const cuuint64_t dims[3] = {N, static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(nslots)};
        const cuuint64_t str[2] = {N * 4, static_cast<cuuint64_t>(dim) * N * 4};
        const cuuint32_t box[3] = {N, 32, 1};
        if (encode_tiled()(&mso, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, state, dims, str, box, e1,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        auto kern = ssm::decode_ws_kernel<T, CH, STAGES, sizeof(T) == 4>;
        static unsigned long long done_ws = 0;
        cudaError_t e = ensure_smem(kern, WLay::SMEM_BYTES, &done_ws);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, CH + 32, WLay::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        const long long grid =
            std::min<long long>(p.ntiles, static_cast<long long>(device_sm_count()) * std::max(1, per_sm));
        // Programmatic dependent launch: consecutive steps overlap one
        // kernel's launch and prologue with the previous one's tail (the
        // kernel waits for the previous writes before reading anything):
        // 30.8-31.1 us against 31.6-31.7 us per cold step on b256 d5120.
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(CH + 32);
        cfg.dynamicSmemBytes = WLay::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, ms, mso, mu, md, mz, mB, mC, p);
    }
    auto kern = ssm::decode_tma_kernel<T, CH, STAGES, sizeof(T) == 4>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem(kern, Lay::SMEM_BYTES, &done);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, CH, Lay::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long grid = std::min<long long>(p.ntiles, static_cast<long long>(device_sm_count()) * std::max(1, per_sm));
    kern<<<static_cast<unsigned>(grid), CH, Lay::SMEM_BYTES, st>>>(ms, mu, md, mz, mB, mC, p);
    return cudaGetLastError();
}

// Tile shape of the staged decode: channels per tile (= threads per CTA) and
// pipeline stages.  SSM_DECODE_TILE=<channels>x<stages> overrides the default
// for tuning.
template <typename T>
cudaError_t launch_decode_tma(float* state, const int* slots, int nslots, const void* u, const void* delta,
                              const void* z, const float* A, const void* B, const void* C, const float* Dskip,
                              const float* dt_bias, void* y, int batch, int dim, int ngroups, cudaStream_t st) {
    // 128 channels x 3 stages measured fastest on B300 for both kernels
    // (CTA-synchronous: 128x4, 64x4, 64x6 within 6%, 32x8 30% slower;
    // warp-specialised: 128x4 and 64x4 5% slower, 256x3 3%, 128x2 and 256x2
    // 30-40%).
    int ch = 128, stages = 3;
    if (const char* v = std::getenv("SSM_DECODE_TILE")) std::sscanf(v, "%dx%d", &ch, &stages);
#define SSM_DECODE_V(C_, S_) \
    if (ch == C_ && stages == S_) \
        return launch_decode_tma_v<T, C_, S_>(state, slots, nslots, u, delta, z, A, B, C, Dskip, dt_bias, y, batch, \
                                              dim, ngroups, st);
    SSM_DECODE_V(128, 4)
    SSM_DECODE_V(128, 2)
    SSM_DECODE_V(256, 2)
    SSM_DECODE_V(256, 3)
    SSM_DECODE_V(64, 4)
    SSM_DECODE_V(64, 6)
    SSM_DECODE_V(32, 8)
#undef SSM_DECODE_V
    return launch_decode_tma_v<T, 128, 3>(state, slots, nslots, u, delta, z, A, B, C, Dskip, dt_bias, y, batch, dim,
                                          ngroups, st);
}


bool force_generic() {
    const char* s = std::getenv("SSM_FORCE_PATH");
    return s && std::strcmp(s, "generic") == 0;
}

// Writes h_final = h0 (or zeros) for an empty sequence.
__global__ void copy_or_zero_state_kernel(const float* __restrict__ h0, float* __restrict__ hf, long long n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i < n) hf[i] = h0 ? h0[i] : 0.f;
}

// Time chunks whose summaries fit in `bytes` of workspace (at least 1).
int chunks_fitting(size_t bytes, int batch, int dim, int dstate) {
    if (bytes < kWorkspaceHeader) return 1;
    const size_t per = static_cast<size_t>(batch) * static_cast<size_t>(dim) * 2u * static_cast<size_t>(dstate) *
                       sizeof(float);
    const size_t k = 1 + (bytes - kWorkspaceHeader) / std::max<size_t>(per, 1);
    return static_cast<int>(std::min<size_t>(k, kMaxChunks));
}

// workspace == nullptr: single pass, no time split.  Otherwise the plan uses
// at most the chunks whose summaries fit in workspace_bytes.
ssm_status_t run_scan(const void* u, const void* delta, const void* z, const float* A,
                      const void* B, const void* C, const float* Dskip, const float* dt_bias,
                      const float* h0, void* y, float* h_final, int batch, int dim, int dstate,
                      int seqlen, int ngroups, ssm_dtype_t io, void* workspace, size_t workspace_bytes,
                      cudaStream_t st) {
    if (batch == 0) return SSM_OK;
    if (seqlen == 0) {
        if (h_final) {
            const long long n = static_cast<long long>(batch) * dim * dstate;
            copy_or_zero_state_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(h0, h_final, n);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return SSM_OK;
    }
    if (tma_eligible(seqlen, io) && !force_generic()) {
        const bool chunks_ok = workspace != nullptr;
        const int cap = chunks_ok ? chunks_fitting(workspace_bytes, batch, dim, dstate) : 1;
        float* agg = chunks_ok ? reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceHeader) : nullptr;
        unsigned int* status = chunks_ok ? static_cast<unsigned int*>(workspace) : nullptr;
        const ScanPlan plan = plan_scan(batch, dim, dstate, seqlen, ngroups, io, cap);
        WsPlan wplan{};
        if (ws_segmented_forced(io, dstate, &wplan) || ws_single_pass(batch, dim, dstate, ngroups, io, plan, &wplan))
            return run_scan_ws(u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final, batch, dim, dstate, seqlen,
                               ngroups, io, wplan, status, st);
        return run_scan_tma(u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final, batch, dim, dstate, seqlen,
                            ngroups, io, plan, agg, status, st);
    }
    ssm::ScanParams p{};
    p.u = u; p.delta = delta; p.z = z; p.A = A; p.B = B; p.C = C; p.D = Dskip;
    p.dt_bias = dt_bias; p.y = y; p.h0 = h0; p.h_final = h_final;
    p.batch = batch; p.dim = dim; p.seqlen = seqlen; p.ngroups = ngroups;
    p.dim_per_group = dim / ngroups;
    int lanes = choose_lanes(batch * dim, dstate, device_sm_count());
    const int forced = env_int("SSM_FORCE_LANES", 0);
    if (forced == 1 || forced == 2 || forced == 4 || forced == 8) lanes = forced;
    lanes = std::max(std::min({lanes, dstate / 2, 8}), min_lanes_for(dstate));
    const cudaError_t e = (io == SSM_F32) ? launch_scan_t<float>(p, dstate, lanes, st)
                                          : launch_scan_t<__nv_bfloat16>(p, dstate, lanes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}


// ---------------------------------------------------------------------------
// Scratch for the entry point that allocates nothing (ssm_scan_fwd_chunked_static)
// ---------------------------------------------------------------------------

// File-scope device array: loaded with the module on every device that uses the
// library, held until exit.  Host code must not pass its name to a kernel (in
// host code it is only a stand-in); the device address comes from
// cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_static_scratch[SSM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
struct StaticScratchEntry {
    CUcontext ctx;  // context the address was looked up in
    void* ptr;
};
StaticScratchEntry g_static_scratch_ptr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static const CtxGetCurrentFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetCurrentFn>(nullptr);
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    return fn;
}

// Device address of g_static_scratch in the current device's current context.
// It is looked up once per device with that device current, and again whenever
// the current context differs from the one it was looked up in (after a
// cudaDeviceReset, or under a caller's own driver context, where the module --
// and so the array -- is a different instance).
ssm_status_t static_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return SSM_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;  // null until the runtime has made a context current on this thread
    const CtxGetCurrentFn get = ctx_get_current();
    if (!get || get(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorNotSupported);
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    StaticScratchEntry& ent = g_static_scratch_ptr[dev];
    if (!ent.ptr || !ctx || ent.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);  // makes the device's context current if needed
        if (e != cudaSuccess) return cuda_fail(e);
        if (get(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorNotSupported);
        ent.ctx = ctx;
        ent.ptr = p;
    }
    *out = ent.ptr;
    return SSM_OK;
}

// ---------------------------------------------------------------------------
// Short causal convolution in front of the scan
// ---------------------------------------------------------------------------

// Launches a kernel with programmatic dependent launch (the kernel calls
// grid_dep_launch / grid_dep_wait): its launch overlaps the previous kernel's
// tail in the stream.  Errors surface through cudaGetLastError.
template <typename... KArgs, typename... Args>
void launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = st;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <typename T>
cudaError_t launch_conv_t(const ssm::ConvParams& p, int width, cudaStream_t st) {
    const int es = static_cast<int>(sizeof(T));
    const bool vec = (static_cast<long long>(p.seqlen) * es) % 16 == 0;
    // Vector path: 8 warps a block, each taking 4 x 32 chunks per iteration.
    const long long work = vec ? (p.rows * (p.seqlen / (16 / es)) + 3) / 4 : p.rows * p.seqlen;
    const long long want = (work + 255) / 256;
    const unsigned grid = static_cast<unsigned>(std::max(1LL, std::min(want, static_cast<long long>(device_sm_count()) * 8)));
    auto go = [&](auto wc) {
        constexpr int W = decltype(wc)::value;
        if (vec) {
            if (p.rows * (p.seqlen / (16 / es)) < (1LL << 31))
                launch_pdl(ssm::conv1d_vec_kernel<T, W, unsigned>, grid, 256, st, p);
            else
                launch_pdl(ssm::conv1d_vec_kernel<T, W, unsigned long long>, grid, 256, st, p);
        } else {
            ssm::conv1d_elem_kernel<T, W><<<grid, 256, 0, st>>>(p);
            if (p.x_last && W > 1)
                ssm::conv1d_last_kernel<T, W><<<static_cast<unsigned>((p.rows + 255) / 256), 256, 0, st>>>(p);
        }
    };
    switch (width) {
        case 1: go(std::integral_constant<int, 1>{}); break;
        case 2: go(std::integral_constant<int, 2>{}); break;
        case 3: go(std::integral_constant<int, 3>{}); break;
        case 4: go(std::integral_constant<int, 4>{}); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_update_t(void* state, const void* x, const float* w, const float* bias, void* out,
                                 long long rows, int dim, int width, int silu_act, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>((rows + 255) / 256);
    switch (width) {
        case 1: launch_pdl(ssm::conv1d_update_kernel<T, 1>, grid, 256, st, state, x, w, bias, out, rows, dim, silu_act); break;
        case 2: launch_pdl(ssm::conv1d_update_kernel<T, 2>, grid, 256, st, state, x, w, bias, out, rows, dim, silu_act); break;
        case 3: launch_pdl(ssm::conv1d_update_kernel<T, 3>, grid, 256, st, state, x, w, bias, out, rows, dim, silu_act); break;
        case 4: launch_pdl(ssm::conv1d_update_kernel<T, 4>, grid, 256, st, state, x, w, bias, out, rows, dim, silu_act); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward pass
// ---------------------------------------------------------------------------

// Tiles per time chunk of the backward pass.  The main pass runs three CTAs
// per SM, each owning one (channel block, chunk); the length is chosen among
// 16..20 tiles (8 from N = 64 on) so that its CTAs fill whole waves on 148
// SMs: minimum of ceil(CTAs / 444) x tiles, the shorter chunk on a tie.  b2
// d1536 L2048: 20 tiles (13 chunks, 2.81 waves) in place of 16 (16 chunks,
// 3.46 waves).  A function of the arguments only, so that the workspace size
// needs no device.
int bwd_chunk_tiles_for(int batch, int dim, int dstate, int seqlen, int ngroups) {
    const int tmax = ssm::bwd_chunk_tiles_max(dstate);
    if (dstate >= 64) return tmax;
    const int ch = ssm::kBwdWarps * 32 / (dstate / ssm::bwd_states_per_lane(dstate));
    const long long blocks = static_cast<long long>((dim / ngroups + ch - 1) / ch) * ngroups * batch;
    const long long slots = 148LL * 3;
    int best = 16;
    long long best_cost = -1;
    for (int t = 16; t <= tmax; ++t) {
        const long long steps = static_cast<long long>(ssm::kBwdTT) * t;
        const long long k = std::max(1LL, (seqlen + steps - 1) / steps);
        const long long cost = ((blocks * k + slots - 1) / slots) * t;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = t;
        }
    }
    return best;
}

int bwd_chunk_steps_for(int batch, int dim, int dstate, int seqlen, int ngroups) {
    return ssm::kBwdTT * bwd_chunk_tiles_for(batch, dim, dstate, seqlen, ngroups);
}

int bwd_nchunks(int batch, int dim, int dstate, int seqlen, int ngroups) {
    const int cs = bwd_chunk_steps_for(batch, dim, dstate, seqlen, ngroups);
    return std::max(1, (seqlen + cs - 1) / cs);
}

size_t bwd_workspace_bytes(int batch, int dim, int dstate, int seqlen, int ngroups) {
    const int k = bwd_nchunks(batch, dim, dstate, seqlen, ngroups);
    if (k <= 1 || batch <= 0) return 0;
    // fagg [k][BD][2][N] and bagg [k][BD][N], fp32
    return static_cast<size_t>(k) * static_cast<size_t>(batch) * static_cast<size_t>(dim) *
           static_cast<size_t>(dstate) * 3u * sizeof(float);
}

template <typename T, int N>
cudaError_t launch_bwd_n(const ssm::BwdParams& p, cudaStream_t st) {
    constexpr bool kAcc = sizeof(T) == 4;
    const dim3 grid(static_cast<unsigned>(static_cast<long long>(p.blocks_per_group) * p.batch * p.ngroups),
                    static_cast<unsigned>(p.nchunks), 1);
    const dim3 block(ssm::kBwdWarps * 32);
    if (p.nchunks > 1) {
        // The summary pass holds more states per lane: its own channel blocks.
        ssm::BwdParams ps = p;
        constexpr int sch = ssm::BwdSumShape<N>::CH;
        ps.blocks_per_group = (p.dim_per_group + sch - 1) / sch;
        const dim3 sgrid(static_cast<unsigned>(static_cast<long long>(ps.blocks_per_group) * p.batch * p.ngroups),
                         static_cast<unsigned>(p.nchunks), 1);
        auto skern = ssm::scan_bwd_summary_kernel<T, N, kAcc>;
        constexpr int ssmem = ssm::BwdSumLayout<T, N>::BYTES;
        static unsigned long long sdone = 0;
        cudaError_t e = ensure_smem(skern, ssmem, &sdone);
        if (e != cudaSuccess) return e;
        skern<<<sgrid, block, ssmem, st>>>(ps);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const long long BD = static_cast<long long>(p.batch) * p.dim;
        const long long n = BD * N;
        ssm::scan_bwd_carry_kernel<N><<<dim3(static_cast<unsigned>((n + 255) / 256), 2), 256, 0, st>>>(
            p.fagg, p.bagg, p.h0, p.dhf, BD, p.nchunks);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto kern = ssm::scan_bwd_kernel<T, N, kAcc>;
    constexpr int smem = ssm::BwdLayout<T, N>::BYTES;
    static unsigned long long done = 0;
    const cudaError_t e = ensure_smem(kern, smem, &done);
    if (e != cudaSuccess) return e;
    kern<<<grid, block, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_t(const ssm::BwdParams& p, int dstate, cudaStream_t st) {
    switch (dstate) {
        case 4: return launch_bwd_n<T, 4>(p, st);
        case 8: return launch_bwd_n<T, 8>(p, st);
        case 32: return launch_bwd_n<T, 32>(p, st);
        case 64: return launch_bwd_n<T, 64>(p, st);
        case 128: return launch_bwd_n<T, 128>(p, st);
        case 256: return launch_bwd_n<T, 256>(p, st);
        default: return launch_bwd_n<T, 16>(p, st);
    }
}

// Copies dh_final (or zeros) into dh0: the gradient of an empty sequence.
__global__ void copy_or_zero_kernel(const float* __restrict__ src, float* __restrict__ dst, long long n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i < n) dst[i] = src ? src[i] : 0.f;
}

}  // namespace

ssm_status_t ssm_note_cuda_error(cudaError_t e) { return cuda_fail(e); }

extern "C" {

size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int seqlen, int ngroups, ssm_dtype_t io) {
    (void)io;
    if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0 || ngroups <= 0 || dim % ngroups != 0) return 0;
    if (!supported_dstate(dstate)) return 0;
    return bwd_workspace_bytes(batch, dim, dstate, seqlen, ngroups);
}

ssm_status_t ssm_scan_bwd(const void* u, const void* delta, const void* z, const float* A, const void* B,
                          const void* C, const float* Dskip, const float* dt_bias, const float* h0,
                          const void* dy, const float* dh_final, void* du, void* ddelta, void* dz, float* dA,
                          float* dB, float* dC, float* dDskip, float* ddt_bias, float* dh0, int batch, int dim,
                          int dstate, int seqlen, int ngroups, ssm_dtype_t io, void* workspace,
                          size_t workspace_bytes, void* stream) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0) return SSM_ERR_INVALID_ARG;
    if (dim % ngroups != 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!A || !dA) return SSM_ERR_INVALID_ARG;
    if (seqlen > 0 && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)) return SSM_ERR_INVALID_ARG;
    if (z && seqlen > 0 && !dz) return SSM_ERR_INVALID_ARG;
    if ((Dskip && !dDskip) || (dt_bias && !ddt_bias)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {u, delta, z, A, B, C, Dskip, dt_bias, h0, dy, dh_final, du, ddelta, dz, dA, dB, dC,
                          dDskip, ddt_bias, dh0, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    const void* outs[] = {du, ddelta, dz, dB, dC};
    const void* ins[] = {u, delta, z, B, C, dy};
    for (const void* o : outs)
        for (const void* i : ins)
            if (o && o == i) return SSM_ERR_INVALID_ARG;
    const size_t need = ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, ngroups, io);
    if (workspace_bytes < need || (need > 0 && !workspace)) return SSM_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int es = io == SSM_F32 ? 4 : 2;
    const size_t nBC = static_cast<size_t>(batch) * ngroups * dstate * static_cast<size_t>(seqlen);
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(dim) * dstate, st);
    if (e == cudaSuccess && dDskip) e = cudaMemsetAsync(dDskip, 0, sizeof(float) * static_cast<size_t>(dim), st);
    if (e == cudaSuccess && ddt_bias) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * static_cast<size_t>(dim), st);
    if (e == cudaSuccess && nBC > 0) e = cudaMemsetAsync(dB, 0, sizeof(float) * nBC, st);
    if (e == cudaSuccess && nBC > 0) e = cudaMemsetAsync(dC, 0, sizeof(float) * nBC, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (seqlen == 0) {
        if (dh0) {
            const long long n = static_cast<long long>(batch) * dim * dstate;
            copy_or_zero_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(dh_final, dh0, n);
            e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return SSM_OK;
    }

    ssm::BwdParams p{};
    p.u = u; p.delta = delta; p.z = z; p.dy = dy; p.B = B; p.C = C;
    p.A = A; p.D = Dskip; p.dt_bias = dt_bias; p.h0 = h0; p.dhf = dh_final;
    p.du = du; p.ddelta = ddelta; p.dz = dz;
    p.dA = dA; p.dB = dB; p.dC = dC; p.dD = dDskip; p.ddt_bias = ddt_bias; p.dh0 = dh0;
    p.batch = batch; p.dim = dim; p.seqlen = seqlen; p.ngroups = ngroups;
    p.dim_per_group = dim / ngroups;
    const int ch = ssm::kBwdWarps * 32 / (dstate / ssm::bwd_states_per_lane(dstate));
    p.blocks_per_group = (p.dim_per_group + ch - 1) / ch;
    p.chunk_steps = bwd_chunk_steps_for(batch, dim, dstate, seqlen, ngroups);
    p.nchunks = bwd_nchunks(batch, dim, dstate, seqlen, ngroups);
    p.vec_ok = (static_cast<long long>(seqlen) * es) % 16 == 0;
    if (p.nchunks > 1) {
        const size_t BDN = static_cast<size_t>(batch) * dim * dstate;
        p.fagg = static_cast<float*>(workspace);
        p.bagg = p.fagg + static_cast<size_t>(p.nchunks) * BDN * 2u;
    }
    const long long grid_x = static_cast<long long>(p.blocks_per_group) * batch * ngroups;
    if (grid_x > 0x7fffffffLL || p.nchunks > 65535) return SSM_ERR_INVALID_ARG;
    e = io == SSM_F32 ? launch_bwd_t<float>(p, dstate, st) : launch_bwd_t<__nv_bfloat16>(p, dstate, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}


ssm_status_t ssm_scan_plan(int batch, int dim, int dstate, int seqlen, int ngroups, ssm_dtype_t io, int chunked,
                           int* lanes, int* chunks, int* kernels, int* staged) {
    if (!lanes || !chunks || !kernels || !staged) return SSM_ERR_INVALID_ARG;
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups != 0)
        return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    *lanes = 0; *chunks = 0; *kernels = 0; *staged = 0;
    if (batch == 0 || seqlen == 0) {
        *kernels = (batch > 0 && chunked) ? 1 : 0;  // h_final copy for an empty sequence
        return SSM_OK;
    }
    if (tma_eligible(seqlen, io) && !force_generic()) {
        const ScanPlan plan = plan_scan(batch, dim, dstate, seqlen, ngroups, io, chunked != 0 ? kMaxChunks : 1);
        *lanes = plan.lanes; *chunks = plan.chunks; *kernels = plan.chunks > 1 ? 3 : 1; *staged = 1;
    } else {
        *lanes = 0; *chunks = 1; *kernels = 1; *staged = 0;
    }
    return SSM_OK;
}

ssm_status_t ssm_scan_fwd_chunked_static(const void* u, const void* delta, const void* z, const float* A,
                                         const void* B, const void* C, const float* Dskip,
                                         const float* dt_bias, const float* h0, void* y, float* h_final,
                                         int batch, int dim, int dstate, int seqlen, int ngroups,
                                         ssm_dtype_t io, void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final,
                                           batch, dim, dstate, seqlen, ngroups, io);
    if (s != SSM_OK) return s;
    if (batch == 0) return SSM_OK;
    void* scratch = nullptr;
    const ssm_status_t a = static_scratch_address(&scratch);
    if (a != SSM_OK) return a;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = cudaMemsetAsync(scratch, 0, kWorkspaceHeader, st);  // status word starts at 0
    if (e != cudaSuccess) return cuda_fail(e);
    return run_scan(u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final, batch, dim, dstate, seqlen, ngroups,
                    io, scratch, SSM_STATIC_SCRATCH_BYTES, st);
}


int ssm_abi_version(void) { return SSM_ABI_VERSION; }

const char* ssm_status_string(ssm_status_t s) {
    switch (s) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
        case SSM_ERR_MISALIGNED: return "SSM_ERR_MISALIGNED";
        case SSM_ERR_WORKSPACE_TOO_SMALL: return "SSM_ERR_WORKSPACE_TOO_SMALL";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    }
    return "SSM_ERR_UNKNOWN";
}

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const void* z, const float* A,
                          const void* B, const void* C, const float* Dskip, const float* dt_bias,
                          void* y, int batch, int dim, int dstate, int seqlen, int ngroups,
                          ssm_dtype_t io, void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, nullptr, nullptr,
                                           batch, dim, dstate, seqlen, ngroups, io);
    if (s != SSM_OK) return s;
    return run_scan(u, delta, z, A, B, C, Dskip, dt_bias, nullptr, y, nullptr, batch, dim, dstate,
                    seqlen, ngroups, io, nullptr, 0, static_cast<cudaStream_t>(stream));
}

size_t ssm_scan_fwd_chunked_workspace_size(int batch, int dim, int dstate, int seqlen, int ngroups,
                                           ssm_dtype_t io) {
    if (batch < 0 || dim <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups != 0) return 0;
    if (!supported_dstate(dstate) || (io != SSM_F32 && io != SSM_BF16)) return 0;
    size_t bytes = kWorkspaceHeader;
    if (tma_eligible(seqlen, io)) {
        // Summaries (P, E) of up to kMaxChunks - 1 chunks for every channel.
        const size_t chunks = static_cast<size_t>(max_chunks_for(seqlen, io)) - 1;
        bytes += chunks * static_cast<size_t>(batch) * static_cast<size_t>(dim) * 2u * static_cast<size_t>(dstate) *
                 sizeof(float);
    }
    return bytes;
}

ssm_status_t ssm_scan_fwd_chunked(const void* u, const void* delta, const void* z, const float* A,
                                  const void* B, const void* C, const float* Dskip,
                                  const float* dt_bias, const float* h0, void* y, float* h_final,
                                  int batch, int dim, int dstate, int seqlen, int ngroups,
                                  ssm_dtype_t io, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final,
                                           batch, dim, dstate, seqlen, ngroups, io);
    if (s != SSM_OK) return s;
    if (workspace && !aligned16(workspace)) return SSM_ERR_MISALIGNED;
    const size_t need = ssm_scan_fwd_chunked_workspace_size(batch, dim, dstate, seqlen, ngroups, io);
    if (workspace_bytes < need || (need > 0 && !workspace)) return SSM_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (workspace) {
        const cudaError_t e = cudaMemsetAsync(workspace, 0, kWorkspaceHeader, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return run_scan(u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final, batch, dim, dstate,
                    seqlen, ngroups, io, workspace, workspace_bytes, st);
}

ssm_status_t ssm_workspace_status(const void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kWorkspaceHeader) return SSM_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return SSM_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == 0 ? SSM_OK : SSM_ERR_TIMEOUT;
}

ssm_status_t ssm_set_pass_timer(void* begin_event, void* end_event) {
    if ((begin_event == nullptr) != (end_event == nullptr)) return SSM_ERR_INVALID_ARG;
    g_pass_begin = static_cast<cudaEvent_t>(begin_event);
    g_pass_end = static_cast<cudaEvent_t>(end_event);
    return SSM_OK;
}

ssm_status_t ssm_device_status(int clear, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&word, ssm::g_ssm_device_error, sizeof(word), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && clear && word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(ssm::g_ssm_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (word & ssm::kDeviceErrTimeout) return SSM_ERR_TIMEOUT;
    return word == 0 ? SSM_OK : SSM_ERR_INVALID_ARG;
}

ssm_status_t ssm_state_update_pooled(float* state_pool, const int* state_indices, int nslots, const void* u,
                                     const void* delta, const void* z, const float* A, const void* B, const void* C,
                                     const float* Dskip, const float* dt_bias, void* y, int batch, int dim,
                                     int dstate, int ngroups, ssm_dtype_t io, void* stream) {
    float* state = state_pool;
    if (batch < 0 || dim <= 0 || dstate <= 0 || ngroups <= 0 || dim % ngroups != 0)
        return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (!supported_dstate(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!state || !u || !delta || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
    if (state_indices ? nslots < 1 : nslots != batch) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {state, state_indices, u, delta, z, A, B, C, Dskip, dt_bias, y};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;

    ssm::DecodeParams p{};
    p.state = state; p.u = u; p.delta = delta; p.z = z; p.A = A; p.B = B; p.C = C;
    p.D = Dskip; p.dt_bias = dt_bias; p.y = y; p.slots = state_indices; p.nslots = nslots;
    p.batch = batch; p.dim = dim; p.ngroups = ngroups; p.dim_per_group = dim / ngroups;
    cudaStream_t st0 = static_cast<cudaStream_t>(stream);
    if (decode_tma_eligible(batch, dim, dstate, ngroups, io) && !force_generic()) {
        const cudaError_t e = io == SSM_F32
            ? launch_decode_tma<float>(state, state_indices, nslots, u, delta, z, A, B, C, Dskip, dt_bias, y, batch,
                                       dim, ngroups, st0)
            : launch_decode_tma<__nv_bfloat16>(state, state_indices, nslots, u, delta, z, A, B, C, Dskip, dt_bias, y,
                                               batch, dim, ngroups, st0);
        if (e != cudaSuccess) return cuda_fail(e);
        return SSM_OK;
    }
    constexpr int kBPT = 8;
    constexpr int kThreads = 128;
    // One lane per 16-byte state packet (8 states at N = 256, 4 otherwise).
    const long long threads_x = static_cast<long long>(dim) * (dstate / (dstate > 128 ? 8 : 4));
    dim3 grid(static_cast<unsigned>((threads_x + kThreads - 1) / kThreads),
              static_cast<unsigned>((batch + kBPT - 1) / kBPT));
    if (grid.y > 65535u) return SSM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define SSM_DECODE_LAUNCH(T, N, ACC) ssm::state_update_kernel<T, N, kBPT, ACC><<<grid, kThreads, 0, st>>>(p)
    if (io == SSM_F32) {
        if (dstate == 4) SSM_DECODE_LAUNCH(float, 4, true);
        else if (dstate == 8) SSM_DECODE_LAUNCH(float, 8, true);
        else if (dstate == 32) SSM_DECODE_LAUNCH(float, 32, true);
        else if (dstate == 64) SSM_DECODE_LAUNCH(float, 64, true);
        else if (dstate == 128) SSM_DECODE_LAUNCH(float, 128, true);
        else if (dstate == 256) SSM_DECODE_LAUNCH(float, 256, true);
        else SSM_DECODE_LAUNCH(float, 16, true);
    } else {
        if (dstate == 4) SSM_DECODE_LAUNCH(__nv_bfloat16, 4, false);
        else if (dstate == 8) SSM_DECODE_LAUNCH(__nv_bfloat16, 8, false);
        else if (dstate == 32) SSM_DECODE_LAUNCH(__nv_bfloat16, 32, false);
        else if (dstate == 64) SSM_DECODE_LAUNCH(__nv_bfloat16, 64, false);
        else if (dstate == 128) SSM_DECODE_LAUNCH(__nv_bfloat16, 128, false);
        else if (dstate == 256) SSM_DECODE_LAUNCH(__nv_bfloat16, 256, false);
        else SSM_DECODE_LAUNCH(__nv_bfloat16, 16, false);
    }
#undef SSM_DECODE_LAUNCH
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

ssm_status_t ssm_state_update(float* state, const void* u, const void* delta, const void* z,
                              const float* A, const void* B, const void* C, const float* Dskip,
                              const float* dt_bias, void* y, int batch, int dim, int dstate,
                              int ngroups, ssm_dtype_t io, void* stream) {
    return ssm_state_update_pooled(state, nullptr, batch, u, delta, z, A, B, C, Dskip, dt_bias, y, batch, dim,
                                   dstate, ngroups, io, stream);
}


ssm_status_t ssm_scan_fwd_varlen(const void* u, const void* delta, const void* z, const float* A, const void* B,
                                 const void* C, const float* Dskip, const float* dt_bias, const float* h0,
                                 const int* cu_seqlens, void* y, float* h_final, int dim, int dstate, int total,
                                 int ngroups, int nseq, ssm_dtype_t io, void* stream) {
    const ssm_status_t s = check_scan_args(u, delta, z, A, B, C, Dskip, dt_bias, y, h0, h_final, 1, dim, dstate,
                                           total, ngroups, io);
    if (s != SSM_OK) return s;
    if (nseq < 1 || !cu_seqlens) return SSM_ERR_INVALID_ARG;
    if (!aligned16(cu_seqlens)) return SSM_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (total == 0) {
        if (h_final) {
            const long long n = static_cast<long long>(nseq) * dim * dstate;
            copy_or_zero_state_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(h0, h_final, n);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return SSM_OK;
    }
    ssm::ScanParams p{};
    p.u = u; p.delta = delta; p.z = z; p.A = A; p.B = B; p.C = C; p.D = Dskip;
    p.dt_bias = dt_bias; p.y = y; p.h0 = h0; p.h_final = h_final;
    p.batch = nseq;  // one CTA row per packed sequence
    p.dim = dim; p.seqlen = total; p.ngroups = ngroups;
    p.dim_per_group = dim / ngroups;
    p.cu_seqlens = cu_seqlens; p.nseq = nseq;
    // Two lanes a channel at least: measured faster than one for packed
    // batches of short sequences on B300 (52 vs 69 us for 64 sequences of
    // mean length 64 at 1536 channels).
    int lanes = std::max(choose_lanes(nseq * dim, dstate, device_sm_count()), std::min(2, dstate / 2));
    const int forced = env_int("SSM_FORCE_LANES", 0);
    if (forced == 1 || forced == 2 || forced == 4 || forced == 8) lanes = forced;
    lanes = std::max(std::min({lanes, dstate / 2, 8}), min_lanes_for(dstate));
    const cudaError_t e = (io == SSM_F32) ? launch_scan_t<float>(p, dstate, lanes, st)
                                          : launch_scan_t<__nv_bfloat16>(p, dstate, lanes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

ssm_status_t ssm_causal_conv1d_fwd(const void* x, const float* w, const float* bias, const void* x_prev,
                                   void* out, void* x_last, int batch, int dim, int seqlen, int width,
                                   int silu, ssm_dtype_t io, void* stream) {
    if (batch < 0 || dim <= 0 || seqlen < 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (width < 1 || width > SSM_CONV_MAX_WIDTH) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!w || (seqlen > 0 && (!x || !out))) return SSM_ERR_INVALID_ARG;
    if ((x && x == out) || (x_prev && x_prev == x_last)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w, bias, x_prev, out, x_last};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    ssm::ConvParams p{};
    p.x = x; p.w = w; p.bias = bias; p.x_prev = width > 1 ? x_prev : nullptr; p.out = out;
    p.x_last = width > 1 ? x_last : nullptr;
    p.rows = static_cast<long long>(batch) * dim;
    p.dim = dim; p.seqlen = seqlen; p.silu = silu != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (seqlen == 0) {
        // Nothing to convolve; the next segment's history is this one's.
        if (p.x_last) {
            const size_t bytes = static_cast<size_t>(p.rows) * (width - 1) * (io == SSM_F32 ? 4 : 2);
            e = p.x_prev ? cudaMemcpyAsync(p.x_last, p.x_prev, bytes, cudaMemcpyDeviceToDevice, st)
                         : cudaMemsetAsync(p.x_last, 0, bytes, st);
        }
    } else {
        e = io == SSM_F32 ? launch_conv_t<float>(p, width, st) : launch_conv_t<__nv_bfloat16>(p, width, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

ssm_status_t ssm_causal_conv1d_update(void* conv_state, const void* x, const float* w, const float* bias,
                                      void* out, int batch, int dim, int width, int silu, ssm_dtype_t io,
                                      void* stream) {
    if (batch < 0 || dim <= 0) return SSM_ERR_INVALID_ARG;
    if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (width < 1 || width > SSM_CONV_MAX_WIDTH) return SSM_ERR_UNSUPPORTED;
    if (batch == 0) return SSM_OK;
    if (!x || !w || !out || (width > 1 && !conv_state)) return SSM_ERR_INVALID_ARG;
    if (x == out) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {conv_state, x, w, bias, out};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_MISALIGNED;
    const long long rows = static_cast<long long>(batch) * dim;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        io == SSM_F32 ? launch_conv_update_t<float>(conv_state, x, w, bias, out, rows, dim, width, silu != 0, st)
                      : launch_conv_update_t<__nv_bfloat16>(conv_state, x, w, bias, out, rows, dim, width, silu != 0,
                                                            st);
    if (e != cudaSuccess) return cuda_fail(e);
    return SSM_OK;
}

}  // extern "C"
