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

constexpr long long STAGE_MAX_BYTES = 32 * 1024;   // rows per stage are capped by this
constexpr int STAGES_MAX = 8;
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

// Process-wide opt-in: launch with programmatic stream serialization so a call
// streams its packed weights while the previous kernel on the stream finishes.
inline int& weight_prefetch_flag() {
    static int f = 0;
    return f;
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
    int T = 0;            // threads per CTA
    int parts = 1;        // CTAs per matrix (grid.x)
    int R = 1;            // row steps per slot (kernel template parameter)
    bool bulk = false;    // copy engine: bulk TMA (true) or warp-wide cp.async (false)
    size_t smem = 0;
};

inline int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

inline long long round_up(long long v, long long a) { return (v + a - 1) / a * a; }

// Target bytes in flight per SM. Measured on GB300 (tuning sweeps over the
// five workloads): two slots per warp, about 40-60 KB per SM, is as fast as or
// faster than deeper rings; more outstanding copies only delay the moment a
// CTA's first slot lands.
constexpr long long IN_FLIGHT_BYTES = 48 * 1024;
constexpr long long DEFER_MAX_BYTES = 48 * 1024;

// Launch plan of format F for `rows` x `k` (slots: MoE slot count, 1 dense).
template <class F>
inline int make_plan(int rows, int k, int slots, const qmv_cfg* cfg, KParams* kp, Plan* pl) {
    DevInfo di;
    int rc = dev_info(&di, nullptr);
    if (rc) return rc;
    const int nb = k / F::QK;
    const int U = F::units(nb);
    const int KS = (U + 31) / 32;
    const int GS = KS == 1 ? pow2ceil(U) : 32;
    const int rpw = 32 / GS;
    int nw_max = F::MAX_THREADS / 32;
    if (cfg && cfg->warps > 0) nw_max = std::min(nw_max, cfg->warps);
    if (KS > nw_max) return QMV_ETOOBIG;
    const long long rowbytes = static_cast<long long>(nb) * F::BLOCK_BYTES;

    Plan P;
    // CTAs per matrix: one per SM (MoE: the SMs are shared by the slots), but
    // not more than there are rows.
    if (cfg && cfg->ctas > 0)
        P.parts = std::min(cfg->ctas, rows);
    else if (slots > 1)
        P.parts = std::min((di.nsm + slots - 1) / slots, rows);
    else
        P.parts = std::min(di.nsm, rows);
    P.parts = std::max(P.parts, 1);
    const int rpc = (rows + P.parts - 1) / P.parts;

    // Row groups: as many as the thread budget holds, no more than the CTA's
    // rows can feed.
    int NG = std::max(1, nw_max / KS);
    NG = std::min(NG, (rpc + rpw - 1) / rpw);
    NG = std::max(NG, 1);
    const int nwarps = NG * KS;
    P.T = 32 * nwarps;
    const int rows_per_group = (rpc + NG - 1) / NG;

    // Slot = R row steps (KS == 1) or one row's slice (KS > 1).
    int R = 1;
    if (KS == 1 && cfg && cfg->stage_rows > 0) {
        const int want = std::max(1, cfg->stage_rows / rpw);
        R = want >= 4 ? 4 : (want >= 2 ? 2 : 1);
    }
    P.R = R;
    // Copy engine: bulk TMA from one lane per warp by default; 16-byte
    // cp.async from all 32 lanes stays selectable (measured equal or slower).
    P.bulk = !(cfg && cfg->copy == 2);
    const long long slot_bytes = KS == 1 ? static_cast<long long>(R) * rpw * rowbytes
                                         : static_cast<long long>(F::SLICE_BLOCKS) * F::BLOCK_BYTES;
    if (slot_bytes + 32 > 0x7fffffffLL) return QMV_ETOOBIG;
    const long long slot_stride = round_up(slot_bytes + 32, 128);
    const int steps = KS == 1 ? (rows_per_group + R * rpw - 1) / (R * rpw) : rows_per_group;

    // Shared-memory layout: limb tables, slice partials, slots, barriers.
    long long off = 0;
    kp->off_la = kp->off_lb = kp->off_lc = kp->off_xs = kp->off_xsum = 0;
    if (F::LIMBS) {
        kp->off_la = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_lb = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_lc = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->off_xs = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 32), 128);
        kp->off_xsum = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 16), 128);
    }
    // Row partials: park every lane's partial ([rows][KS * GS] floats) and
    // reduce once at the end when that fits comfortably; otherwise reduce each
    // slot with shuffles and keep only per-slice partials ([rows][KS]).
    const int W = KS * GS;
    const bool defer = 4LL * rpc * W <= DEFER_MAX_BYTES;
    kp->off_red = static_cast<uint32_t>(off);
    if (defer)
        off = round_up(off + 4LL * rpc * W, 128);
    else if (KS > 1)
        off = round_up(off + 4LL * rpc * KS, 128);
    const long long avail = di.smem_optin - 1024 - off;   // 1 KB for static shared memory
    const long long per_slot = nwarps * (slot_stride + 8);
    int S;
    if (cfg && cfg->stages > 0)
        S = cfg->stages;
    else
        S = static_cast<int>(std::min<long long>(8, std::max<long long>(2, IN_FLIGHT_BYTES / (nwarps * slot_bytes))));
    S = std::min(S, std::max(steps, 1));
    S = static_cast<int>(std::min<long long>(S, avail / per_slot));
    if (S < 1) return QMV_ETOOBIG;
    kp->off_slots = static_cast<uint32_t>(off);
    kp->slot_stride = static_cast<uint32_t>(slot_stride);
    off += static_cast<long long>(nwarps) * S * slot_stride;
    kp->off_bars = static_cast<uint32_t>(off);
    off += 8LL * nwarps * S;
    P.smem = static_cast<size_t>(off);

    kp->nb = nb;
    kp->rowbytes = rowbytes;
    kp->U = U;
    kp->KS = KS;
    kp->GS = GS;
    int lg = 0;
    while ((1 << lg) < GS) lg++;
    kp->lgGS = lg;
    kp->NG = NG;
    kp->R = R;
    kp->S = S;
    kp->defer = defer ? 1 : 0;
    kp->W = W;
    // Balanced splits, precomputed so the kernel only multiplies.
    kp->rq = rows / P.parts;
    kp->rrem = rows % P.parts;
    for (int b = 0; b < 2; b++) {
        const int n = kp->rq + b;
        kp->gq[b] = n / NG;
        kp->grem[b] = n % NG;
    }
    *pl = P;
    return QMV_OK;
}

template <class F, int R, bool MOE, int MODE, bool BULK>
inline int launch_one(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    auto kern = qmv_stream_kernel<F, R, MOE, MODE, BULK>;
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
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.parts, MOE ? slots : 1, 1);
    lc.blockDim = dim3(pl.T, 1, 1);
    lc.dynamicSmemBytes = pl.smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = __atomic_load_n(&weight_prefetch_flag(), __ATOMIC_RELAXED) ? 1 : 0;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, kp));
}

template <class F, bool MOE, int MODE, bool BULK>
inline int launch_r(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    switch (pl.R) {
    case 1: return launch_one<F, 1, MOE, MODE, BULK>(kp, pl, slots, stream);
    case 2: return launch_one<F, 2, MOE, MODE, BULK>(kp, pl, slots, stream);
    default: return launch_one<F, 4, MOE, MODE, BULK>(kp, pl, slots, stream);
    }
}

template <class F, bool MOE, int MODE>
inline int launch(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    return pl.bulk ? launch_r<F, MOE, MODE, true>(kp, pl, slots, stream)
                   : launch_r<F, MOE, MODE, false>(kp, pl, slots, stream);
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
