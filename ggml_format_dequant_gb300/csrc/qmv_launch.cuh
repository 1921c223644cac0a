// qmv_launch.cuh -- host-side launch plan for qmv_stream_kernel: lane groups,
// grid size, rows per pipeline stage, pipeline depth and the shared-memory
// layout, chosen per shape (or forced through qmv_cfg for tests).
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qmv.h"
#include "qmv_kernel.cuh"

namespace qmv {

constexpr int THREADS_MAX = 256;
constexpr long long STAGE_MAX_BYTES = 40 * 1024;   // rows per stage are capped by this
constexpr int STAGES_MAX = 6;
constexpr int MAX_DEVICES = 64;

// The last CUDA error seen by a launch on this thread (for qmv_last_cuda_error).
inline cudaError_t& last_cuda_error() {
    static thread_local cudaError_t e = cudaSuccess;
    return e;
}

inline int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess) return QMV_OK;
    last_cuda_error() = e;
    return QMV_ECUDA;
}

struct DevInfo {
    int nsm = 0;
    int smem_optin = 0;
};

inline int dev_info(DevInfo* out, int* dev_out) {
    static DevInfo cache[MAX_DEVICES];
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        last_cuda_error() = e;
        return QMV_ECUDA;
    }
    if (dev < 0 || dev >= MAX_DEVICES) return QMV_ECUDA;
    if (cache[dev].nsm == 0) {
        DevInfo d;
        if (cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return QMV_ECUDA;
        cache[dev] = d;
    }
    *out = cache[dev];
    if (dev_out) *dev_out = dev;
    return QMV_OK;
}

struct Plan {
    int T = 0, GS = 0, NG = 0, UPL = 1, RG = 1, G = 1, S = 1;
    int parts = 1;        // CTAs per matrix (grid.x)
    bool resident = true;
    size_t smem = 0;
};

inline int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

inline long long round_up(long long v, long long a) { return (v + a - 1) / a * a; }

// U: units per row; limbs: the format keeps integer activation limbs in shared
// memory; slots: MoE slot count (1 for dense).
inline int make_plan(int U, long long rowbytes, int rows, int k, bool limbs, int slots,
                     const qmv_cfg* cfg, KParams* kp, Plan* pl) {
    DevInfo di;
    int rc = dev_info(&di, nullptr);
    if (rc) return rc;
    Plan P;
    if (U <= 32) {
        P.GS = pow2ceil(U);
        P.NG = THREADS_MAX / P.GS;
        P.T = THREADS_MAX;
    } else if (U <= THREADS_MAX) {
        P.GS = static_cast<int>(round_up(U, 32));
        P.NG = THREADS_MAX / P.GS;
        P.T = P.NG * P.GS;
    } else {
        P.GS = THREADS_MAX;
        P.NG = 1;
        P.T = THREADS_MAX;
        P.UPL = (U + THREADS_MAX - 1) / THREADS_MAX;
        P.resident = false;
    }

    // CTAs per matrix: enough to cover every SM once (MoE: shared by the
    // slots), never fewer rows per CTA than the groups can take in one pass
    // unless the matrix is that small.
    const int by_groups = (rows + P.NG - 1) / P.NG;
    if (cfg && cfg->ctas > 0)
        P.parts = std::min(cfg->ctas, rows);
    else if (slots > 1)
        P.parts = std::min((di.nsm + slots - 1) / slots, by_groups);
    else
        P.parts = std::min(di.nsm, by_groups);
    P.parts = std::max(P.parts, 1);
    const int rpc = (rows + P.parts - 1) / P.parts;

    // Rows per stage: up to 4 per group, as many as the CTA has, capped by the
    // stage byte budget.
    long long G = std::min<long long>(4LL * P.NG, rpc);
    if (cfg && cfg->stage_rows > 0) G = std::min<long long>(G, cfg->stage_rows);
    G = std::min<long long>(G, (STAGE_MAX_BYTES - 32) / rowbytes);
    if (G < 1) return QMV_ETOOBIG;
    P.G = static_cast<int>(G);
    P.RG = pow2ceil((P.G + P.NG - 1) / P.NG);

    const long long stage_stride = round_up(P.G * rowbytes + 32, 128);
    const int nst_max = (rpc + P.G - 1) / P.G;

    // Shared-memory layout: limb tables, reduction buffer, stages, barriers.
    long long off = 0;
    kp->off_la = kp->off_lb = kp->off_lc = kp->off_xs = kp->off_xsum = 0;
    if (limbs) {
        kp->off_la = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_lb = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_lc = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_xs = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 32), 128);
        kp->off_xsum = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 16), 128);
    }
    kp->off_red = static_cast<uint32_t>(off);
    if (P.GS > 32) off = round_up(off + 2LL * P.G * (P.GS / 32) * 4, 128);
    const long long fixed = off + 8 * STAGES_MAX + 1024;   // + barriers + static shared memory
    const long long avail = di.smem_optin - fixed;
    int S = (cfg && cfg->stages > 0) ? std::min(cfg->stages, STAGES_MAX) : STAGES_MAX;
    S = std::min<long long>(S, nst_max);
    S = static_cast<int>(std::min<long long>(S, avail / stage_stride));
    if (S < 1) return QMV_ETOOBIG;
    P.S = S;
    kp->off_stage = static_cast<uint32_t>(off);
    kp->stage_stride = static_cast<uint32_t>(stage_stride);
    off += stage_stride * S;
    kp->off_bar = static_cast<uint32_t>(off);
    off += 8 * S;
    P.smem = static_cast<size_t>(off);

    kp->U = U;
    kp->GS = P.GS;
    kp->NG = P.NG;
    kp->G = P.G;
    kp->S = P.S;
    kp->UPL = P.UPL;
    *pl = P;
    return QMV_OK;
}

template <class F, int RG, bool RES, bool MOE, int MODE>
inline int launch_one(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    auto kern = qmv_stream_kernel<F, RG, RES, MOE, MODE>;
    // Dynamic shared memory above 48 KB must be opted into per kernel; the
    // attribute only ever grows, once per size class and device.
    static int configured[MAX_DEVICES] = {};
    int dev = 0;
    DevInfo di;
    if (dev_info(&di, &dev)) return QMV_ECUDA;
    if (static_cast<int>(pl.smem) > configured[dev]) {
        int rc = cuda_rc(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(pl.smem)));
        if (rc) return rc;
        configured[dev] = static_cast<int>(pl.smem);
    }
    kern<<<dim3(pl.parts, MOE ? slots : 1, 1), pl.T, pl.smem, stream>>>(kp);
    return cuda_rc(cudaGetLastError());
}

template <class F, bool MOE, int MODE>
inline int launch(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    if (pl.resident) {
        switch (pl.RG) {
        case 1: return launch_one<F, 1, true, MOE, MODE>(kp, pl, slots, stream);
        case 2: return launch_one<F, 2, true, MOE, MODE>(kp, pl, slots, stream);
        default: return launch_one<F, 4, true, MOE, MODE>(kp, pl, slots, stream);
        }
    }
    switch (pl.RG) {
    case 1: return launch_one<F, 1, false, MOE, MODE>(kp, pl, slots, stream);
    case 2: return launch_one<F, 2, false, MOE, MODE>(kp, pl, slots, stream);
    default: return launch_one<F, 4, false, MOE, MODE>(kp, pl, slots, stream);
    }
}

// Read (and optionally clear) this translation unit's device status word.
inline int status_rw(unsigned int* out, int clear) {
    unsigned int v = 0;
    int rc = cuda_rc(cudaMemcpyFromSymbol(&v, g_status, sizeof(v)));
    if (rc) return rc;
    if (clear) {
        const unsigned int z = 0;
        rc = cuda_rc(cudaMemcpyToSymbol(g_status, &z, sizeof(z)));
        if (rc) return rc;
    }
    *out = v;
    return QMV_OK;
}

}  // namespace qmv
