// scan_ws_inst.cuh -- instantiates the warp-specialised fused scan pass for one
// I/O type T and provides the host launchers declared in scan_ws_api.h.
// Included once by scan_ws_bf16.cu and once by scan_ws_f32.cu.
#pragma once

#include <atomic>

#include "scan_ws.cuh"

namespace ssm {
namespace ws_detail {

// The (state size, lanes per channel, consumer warps, time segments) variants
// that are built.  SEG > 1 (the time-segmented variant) is built for N = 16
// with four consumer warps: 2 lanes x 2, 4 or 8 segments and 4 lanes x 2 or
// 4 segments (a tile row of 16 * SEG bytes keeps at least eight rows per CTA).
template <int N, int LANES, int NW, int SEG>
constexpr bool built() {
    if (SEG > 1) return N == 16 && NW == 4 && ((LANES == 2 && SEG <= 8) || (LANES == 4 && SEG <= 4));
    if (NW == 4) {
        switch (N) {
            case 4: return LANES == 1 || LANES == 2;
            case 8: return LANES == 1 || LANES == 2 || LANES == 4;
            case 16: return LANES == 1 || LANES == 2 || LANES == 4 || LANES == 8;
            case 32: return LANES == 2 || LANES == 4 || LANES == 8;
            case 64: return LANES == 4 || LANES == 8;
            case 128: return LANES == 8 || LANES == 16;
            case 256: return LANES == 16;
            default: return false;
        }
    }
    if (NW == 2) return (N == 16 || N == 32) && LANES >= N / 16 && LANES <= 8;
    return false;
}

// Ring depth: four stages while a stage stays small, fewer for the large
// widened B/C tiles of big state sizes.  (Three stages to fit a fourth CTA
// per SM measured slower: 400 -> 430 us on the b8 d2048 L4096 shape.)
template <typename T, int N, int LANES, int NW, int SEG>
constexpr int stages() {
    constexpr int bytes = WsLayout<T, N, LANES, NW, 4, SEG>::STAGE_BYTES;
    return bytes <= 24 * 1024 ? 4 : (bytes <= 48 * 1024 ? 3 : 2);
}

template <typename T, int N, int LANES, int NW, int SEG>
int smem_bytes() {
    if constexpr (built<N, LANES, NW, SEG>()) {
        return WsLayout<T, N, LANES, NW, stages<T, N, LANES, NW, SEG>(), SEG>::SMEM_BYTES;
    } else {
        return 0;
    }
}

template <typename T, int N, int LANES, int NW, int SEG>
cudaError_t launch(const WsMaps& m, const WsScanParams& p, cudaStream_t st) {
    if constexpr (built<N, LANES, NW, SEG>()) {
        constexpr int STAGES = stages<T, N, LANES, NW, SEG>();
        using Lay = WsLayout<T, N, LANES, NW, STAGES, SEG>;
        auto kern = scan_ws_kernel<T, N, LANES, NW, STAGES, sizeof(T) == 4, SEG>;
        // Opt in to the dynamic shared memory once per device.
        static std::atomic<unsigned long long> done{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(done.load(std::memory_order_acquire) & bit)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            done.fetch_or(bit, std::memory_order_acq_rel);
        }
        const long long gx = static_cast<long long>(p.blocks_per_group) * p.ngroups * p.batch;
        if (gx > 0x7fffffffLL || gx <= 0 || p.nchunks < 1 || p.nchunks > 65535) return cudaErrorInvalidConfiguration;
        if (SEG > 1 && p.nchunks != 1) return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(p.nchunks));
        cfg.blockDim = dim3(Lay::THREADS);
        cfg.dynamicSmemBytes = Lay::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = p.nchunks > 1 ? &attr : nullptr;
        cfg.numAttrs = p.nchunks > 1 ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kern, m.u, m.d, m.z, m.B, m.C, p);
    } else {
        (void)m; (void)p; (void)st;
        return cudaErrorInvalidValue;
    }
}

template <typename T, int N, int NW, int SEG>
int smem_lanes(int lanes) {
    switch (lanes) {
        case 1: return smem_bytes<T, N, 1, NW, SEG>();
        case 2: return smem_bytes<T, N, 2, NW, SEG>();
        case 4: return smem_bytes<T, N, 4, NW, SEG>();
        case 8: return smem_bytes<T, N, 8, NW, SEG>();
        case 16: return smem_bytes<T, N, 16, NW, SEG>();
        default: return 0;
    }
}

template <typename T, int N, int NW, int SEG>
cudaError_t launch_lanes(int lanes, const WsMaps& m, const WsScanParams& p, cudaStream_t st) {
    switch (lanes) {
        case 1: return launch<T, N, 1, NW, SEG>(m, p, st);
        case 2: return launch<T, N, 2, NW, SEG>(m, p, st);
        case 4: return launch<T, N, 4, NW, SEG>(m, p, st);
        case 8: return launch<T, N, 8, NW, SEG>(m, p, st);
        case 16: return launch<T, N, 16, NW, SEG>(m, p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int NW, int SEG>
int smem_n(int dstate, int lanes) {
    switch (dstate) {
        case 4: return smem_lanes<T, 4, NW, SEG>(lanes);
        case 8: return smem_lanes<T, 8, NW, SEG>(lanes);
        case 16: return smem_lanes<T, 16, NW, SEG>(lanes);
        case 32: return smem_lanes<T, 32, NW, SEG>(lanes);
        case 64: return smem_lanes<T, 64, NW, SEG>(lanes);
        case 128: return smem_lanes<T, 128, NW, SEG>(lanes);
        case 256: return smem_lanes<T, 256, NW, SEG>(lanes);
        default: return 0;
    }
}

template <typename T, int NW, int SEG>
cudaError_t launch_n(int dstate, int lanes, const WsMaps& m, const WsScanParams& p, cudaStream_t st) {
    switch (dstate) {
        case 4: return launch_lanes<T, 4, NW, SEG>(lanes, m, p, st);
        case 8: return launch_lanes<T, 8, NW, SEG>(lanes, m, p, st);
        case 16: return launch_lanes<T, 16, NW, SEG>(lanes, m, p, st);
        case 32: return launch_lanes<T, 32, NW, SEG>(lanes, m, p, st);
        case 64: return launch_lanes<T, 64, NW, SEG>(lanes, m, p, st);
        case 128: return launch_lanes<T, 128, NW, SEG>(lanes, m, p, st);
        case 256: return launch_lanes<T, 256, NW, SEG>(lanes, m, p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
int smem_any(int dstate, int lanes, int nw, int seg) {
    if (nw == 2 && seg == 1) return smem_n<T, 2, 1>(dstate, lanes);
    if (nw != 4) return 0;
    switch (seg) {
        case 1: return smem_n<T, 4, 1>(dstate, lanes);
        case 2: return smem_n<T, 4, 2>(dstate, lanes);
        case 4: return smem_n<T, 4, 4>(dstate, lanes);
        case 8: return smem_n<T, 4, 8>(dstate, lanes);
        default: return 0;
    }
}

template <typename T>
cudaError_t launch_any(int dstate, int lanes, int nw, int seg, const WsMaps& m, const WsScanParams& p,
                       cudaStream_t st) {
    if (nw == 2 && seg == 1) return launch_n<T, 2, 1>(dstate, lanes, m, p, st);
    if (nw != 4) return cudaErrorInvalidValue;
    switch (seg) {
        case 1: return launch_n<T, 4, 1>(dstate, lanes, m, p, st);
        case 2: return launch_n<T, 4, 2>(dstate, lanes, m, p, st);
        case 4: return launch_n<T, 4, 4>(dstate, lanes, m, p, st);
        case 8: return launch_n<T, 4, 8>(dstate, lanes, m, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ws_detail
}  // namespace ssm
