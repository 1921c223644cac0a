// qmv_launch.cuh -- host-side launch plan for qmv_stream_kernel: lane groups,
// row groups, grid size, rows per ring slot, ring depth and the shared-memory
// layout, chosen per shape (or forced through qmv_opts for tests and sweeps).
#pragma once

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/qmv.h"
#include "qmv_kernel.cuh"

namespace qmv {

constexpr int MAX_DEVICES = 64;
constexpr int MAX_WARPS = 16;               // kernel launch bound: 512 threads, <= 128 registers each
constexpr int WARPS_TWO_PER_SM = 8;         // default CTA size: two CTAs fit on one SM
constexpr long long PIECE_TARGET_BYTES = 16 * 1024;   // rows per ring slot: about this many bytes
constexpr long long RED_MAX_BYTES = 64 * 1024;        // parked slice sums per CTA, at most
constexpr long long MIN_CTA_BYTES = 4 * 1024;         // packed weights per CTA, at least (small matrices)

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

// Launch overlap of one call (qmv_opts.overlap): 0 plain launch;
// 1 programmatic dependent launch, packed weights requested before waiting for
// the previous kernel; 2 also x / ids read early (the caller guarantees that
// the previous kernel writes none of this call's inputs; y still waits).
// A call without options is a plain launch.
inline int overlap_of(const qmv_opts* o) {
    if (!o) return QMV_OVERLAP_NONE;
    return o->overlap <= QMV_OVERLAP_NONE ? QMV_OVERLAP_NONE
                                          : (o->overlap >= QMV_OVERLAP_INDEPENDENT ? QMV_OVERLAP_INDEPENDENT
                                                                                   : QMV_OVERLAP_CHAIN);
}

struct DevInfo {
    int nsm = 0;
    int smem_optin = 0;   // per CTA
    int smem_sm = 0;      // per SM
    int smem_reserved = 0;
};

// The current device's properties, queried once per device (under a lock, so
// that host threads calling concurrently see a complete record).
inline int dev_info(DevInfo* out, int* dev_out) {
    static DevInfo cache[MAX_DEVICES];
    static std::atomic<int> ready[MAX_DEVICES];
    static std::mutex mu;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        last_cuda_error() = e;
        return QMV_ECUDA;
    }
    if (dev < 0 || dev >= MAX_DEVICES) return QMV_ECUDA;
    if (!ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> g(mu);
        if (!ready[dev].load(std::memory_order_relaxed)) {
            DevInfo d;
            if (cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
                return QMV_ECUDA;
            cache[dev] = d;
            ready[dev].store(1, std::memory_order_release);
        }
    }
    *out = cache[dev];
    if (dev_out) *dev_out = dev;
    return QMV_OK;
}

// Dynamic shared memory above 48 KB must be opted into per kernel and device.
// The opted-in size only grows; it is raised under a lock so that concurrent
// first launches from several host threads cannot leave it below a size that
// one of them launches with.
struct SmemOptIn {
    std::atomic<int> bytes[MAX_DEVICES];
    std::mutex mu;
};

template <class K>
inline int ensure_smem(K kern, SmemOptIn& st, int dev, int smem) {
    if (smem <= st.bytes[dev].load(std::memory_order_acquire)) return QMV_OK;
    std::lock_guard<std::mutex> g(st.mu);
    if (smem <= st.bytes[dev].load(std::memory_order_relaxed)) return QMV_OK;
    const int rc = cuda_rc(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    if (rc) return rc;
    st.bytes[dev].store(smem, std::memory_order_release);
    return QMV_OK;
}

struct Plan {
    int T = 0;            // threads per CTA
    int parts = 1;        // CTAs per matrix (grid.x)
    int R = 1;            // rows per warp step (kernel template parameter)
    int CL = 1;           // cluster size along grid.x
    int overlap = 0;      // QMV_OVERLAP_* of the call
    size_t smem = 0;
};

// CTAs sharing one activation prep, by default none: on GB300 a GPC holds 19
// SMs, so clusters of 2 or more leave SMs idle in every wave; measured slower
// (clusters of 4: +23 % on Q4_K 4096 x 4096, +80 % on Q6_K 4096 x 14336).
constexpr int CLUSTER_DEFAULT = 1;
constexpr int CLUSTER_MAX = 8;       // portable cluster size limit

inline int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

inline long long round_up(long long v, long long a) { return (v + a - 1) / a * a; }

// Launch plan of format F for `rows` x `k` (slots: MoE slot count, 1 dense)
// on a device described by `di`, for a given (or the default) CTA count.
template <class F>
inline int make_plan_core(const DevInfo& di, int rows, int k, int slots, const qmv_opts* cfg, KParams* kp, Plan* pl,
                          long long smem_cap = -1) {
    const int nb = k / F::QK;
    const int U = F::units(nb);
    const int KS = (U + 31) / 32;
    const int GS = KS == 1 ? pow2ceil(U) : 32;
    const int rpw = 32 / GS;
    const long long rowbytes = static_cast<long long>(nb) * F::BLOCK_BYTES;
    if (KS > MAX_WARPS) return QMV_ETOOBIG;

    // Warps per CTA: by default 8, so that the next call's CTAs can fit beside
    // this call's on every SM; rows of more than 4 slices take up to 16 (a
    // single row group of 5..8 warps would leave too few warps to hide
    // latency).
    int nw_max = (cfg && cfg->warps > 0) ? std::min(cfg->warps, MAX_WARPS)
                                         : (KS > 4 ? MAX_WARPS : WARPS_TWO_PER_SM);
    if (KS > nw_max) return QMV_ETOOBIG;

    Plan P;
    // CTAs per matrix: one per SM (MoE: the SMs are shared by the slots), but
    // not more than there are rows, and enough that the parked partials fit.
    const int mode = overlap_of(cfg);
    P.overlap = mode;
    const int early = mode >= QMV_OVERLAP_INDEPENDENT ? 1 : 0;
    const int W = KS > 1 ? KS : early;   // parked slice sums per row
    if (cfg && cfg->ctas > 0) {
        P.parts = cfg->ctas;
    } else {
        P.parts = slots > 1 ? (di.nsm + slots - 1) / slots : di.nsm;
        // small matrices: at least MIN_CTA_BYTES of weights per CTA (a CTA
        // pays a fixed start-up cost, the activation prep among it)
        const long long by_bytes = std::max<long long>(1, static_cast<long long>(rows) * rowbytes / MIN_CTA_BYTES);
        if (by_bytes < P.parts) P.parts = static_cast<int>(by_bytes);
        const long long max_rows = std::max<long long>(1, RED_MAX_BYTES / (4LL * std::max(W, 1)));
        const long long need = (rows + max_rows - 1) / max_rows;
        if (need > P.parts) P.parts = static_cast<int>(std::min<long long>(need, 1 << 30));
    }
    P.parts = std::max(1, std::min(P.parts, rows));
    // Clusters share the activation prep: CL CTAs of one matrix each convert
    // 1/CL of x. CL divides the CTA count and half the 16-element groups.
    {
        int want = (cfg && cfg->cluster > 0) ? std::min(cfg->cluster, CLUSTER_MAX) : CLUSTER_DEFAULT;
        if (!F::LIMBS) want = 1;
        int cl = 1;
        for (int c = want; c > 1; c--) {
            if ((c & (c - 1)) == 0 && P.parts % c == 0 && (k / 16) % (2 * c) == 0) {
                cl = c;
                break;
            }
        }
        if (cfg && cfg->cluster > 0 && cl != std::min(cfg->cluster, CLUSTER_MAX) && F::LIMBS) {
            // a forced size the shape cannot take: round the CTA count down to it
            const int c = std::min(cfg->cluster, CLUSTER_MAX);
            if ((c & (c - 1)) == 0 && (k / 16) % (2 * c) == 0 && P.parts >= c) {
                P.parts = P.parts / c * c;
                cl = c;
            }
        }
        P.CL = cl;
    }
    const int rpc = (rows + P.parts - 1) / P.parts;

    // Row groups: as many as the warp budget holds, no more than the CTA's
    // rows can feed.
    int NG = std::max(1, nw_max / KS);
    NG = std::min(NG, (rpc + rpw - 1) / rpw);
    NG = std::max(NG, 1);
    const int nwarps = NG * KS;
    P.T = 32 * nwarps;
    const int gmax = (rpc + NG - 1) / NG;   // rows of the largest row group

    // Rows per warp step: 2 by default for the lighter decoders.
    int R = (cfg && cfg->unroll > 0) ? (cfg->unroll >= 2 ? 2 : 1) : F::DEFAULT_UNROLL;
    P.R = R;

    // Shared-memory layout: limb tables, parked partials, ring, barriers, counters.
    long long off = 0;
    kp->lt = LimbTables{0, 0, 0, 0, 0};
    if (F::LIMBS) {
        kp->lt.la = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->lt.lb = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->lt.lc = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->lt.xs = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 32), 128);
        kp->lt.xsum16 = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 16), 128);
    } else if (quantizes_x<F>::value) {
        // the CTA's own codes (k bytes) and scales (k/32 floats) of x
        kp->lt.la = static_cast<uint32_t>(off); off = round_up(off + k, 128);
        kp->lt.xs = static_cast<uint32_t>(off); off = round_up(off + 4LL * (k / 32), 128);
    }
    kp->off_red = static_cast<uint32_t>(off);
    off = round_up(off + 4LL * rpc * W, 128);   // W == 0: nothing parked
    const long long fixed = off;

    // Budget: half an SM's shared memory when two CTAs are meant to share it,
    // else all a CTA may take.
    const long long per_sm = di.smem_sm - 2LL * di.smem_reserved;
    const long long half = per_sm / 2;
    const long long full = smem_cap > 0 ? std::min<long long>(smem_cap, di.smem_optin) : di.smem_optin;

    auto slot_stride_of = [&](int cr) { return round_up(static_cast<long long>(cr) * rowbytes + 32 + F::SLACK, 128); };
    auto tail = [&](int s) { return 8LL * NG * s + 4LL * (NG * s + NG + 1); };
    auto fits = [&](int cr, int s, long long budget) { return fixed + NG * s * slot_stride_of(cr) + tail(s) <= budget; };
    const int step = R * rpw;   // rows of one unrolled warp step
    int CR = 0, S = 0;
    bool done = false;
    if (cfg && (cfg->chunk_rows > 0 || cfg->chunks > 0)) {
        // Forced pieces and/or depth: as asked, within the CTA's limit.
        CR = cfg->chunk_rows > 0 ? cfg->chunk_rows
                                 : static_cast<int>(std::max<long long>(step, PIECE_TARGET_BYTES / rowbytes));
        CR = std::max(1, std::min(CR, gmax));
        const int pieces = (gmax + CR - 1) / CR;
        S = cfg->chunks > 0 ? std::min(cfg->chunks, pieces) : pieces;
        while (S > 0 && !fits(CR, S, full)) S--;
        done = S >= 1;
    } else {
        // 1. The CTA's whole share at once, one piece per row group, next to a
        //    second CTA on the SM (small CTAs) or alone.
        const long long whole_budget = nwarps <= WARPS_TWO_PER_SM ? half : full;
        if (fits(gmax, 1, whole_budget)) {
            CR = gmax;
            S = 1;
            done = true;
        } else {
            // 2. A ring per row group: pieces of about PIECE_TARGET_BYTES (whole
            //    warp steps where possible), as deep as the SM's shared memory
            //    allows, at least two slots when a group has two pieces.
            CR = static_cast<int>(std::max<long long>(step, PIECE_TARGET_BYTES / rowbytes));
            CR = std::max(1, std::min(CR / step * step > 0 ? CR / step * step : CR, gmax));
            while (true) {
                const int pieces = (gmax + CR - 1) / CR;
                S = pieces;
                while (S > 0 && !fits(CR, S, full)) S--;
                if (S >= 2 || (S >= 1 && pieces == 1)) {
                    done = true;
                    break;
                }
                if (CR == 1) {
                    done = S >= 1;
                    break;
                }
                CR = (CR / 2 >= step) ? (CR / 2) / step * step : std::max(1, CR / 2);
            }
        }
    }
    if (!done) return QMV_ETOOBIG;
    const long long stride = slot_stride_of(CR);
    if (stride > 0x7fffffffLL) return QMV_ETOOBIG;

    kp->off_ring = static_cast<uint32_t>(off);
    off += static_cast<long long>(NG) * S * stride;
    kp->off_bars = static_cast<uint32_t>(off);
    off += 8LL * NG * S;
    kp->off_cnt = static_cast<uint32_t>(off);
    off += 4LL * (NG * S + NG + 1);
    P.smem = static_cast<size_t>(round_up(off, 16));
    if (static_cast<long long>(P.smem) > full) return QMV_ETOOBIG;

    kp->nb = nb;
    kp->rowbytes = static_cast<uint32_t>(rowbytes);
    kp->U = U;
    kp->KS = KS;
    kp->GS = GS;
    int lg = 0;
    while ((1 << lg) < GS) lg++;
    kp->lgGS = lg;
    kp->NG = NG;
    kp->CR = CR;
    kp->S = S;
    kp->W = W;
    kp->slot_stride = static_cast<uint32_t>(stride);
#ifdef QMV_BOUNDS_CHECK_PLANT
    // A planted fault for the checking build's own test: ring slots half as
    // long as the plan needs. The checks skip every copy that no longer fits;
    // all other accesses stay inside the (now shorter) ring.
    kp->slot_stride = static_cast<uint32_t>(stride / 2) & ~15u;
#endif
    kp->aligned8 = (rowbytes % 8 == 0) ? 1 : 0;
    kp->CL = P.CL;
    kp->early_inputs = early;
    // Balanced splits, precomputed so the kernel only multiplies.
    kp->rq = rows / P.parts;
    kp->rrem = rows % P.parts;
    for (int b = 0; b < 2; b++) {
        const int n = kp->rq + b;
        kp->gq[b] = n / NG;
        kp->grem[b] = n % NG;
        for (int l = 0; l < 2; l++) kp->npc4[2 * b + l] = (kp->gq[b] + l + CR - 1) / CR;
    }
    for (int w = 0; w < MAX_WARPS; w++)
        kp->wmap[w] = w < NG * KS ? static_cast<uint8_t>(((w / KS) << 4) | (w % KS)) : uint8_t{0xff};
    *pl = P;
    return QMV_OK;
}

// Independent calls (QMV_OVERLAP_INDEPENDENT): CTAs per call, as a divisor of
// the SM count (the CTAs of an MoE call are shared by its slots).
constexpr int INDEP_SM_DIV = 5;

// Launch plan of format F. Independent calls (QMV_OVERLAP_INDEPENDENT) take a
// few CTAs (about a fifth of the SM count) of at most WARPS_TWO_PER_SM warps
// in half an SM's shared memory, each streaming a long share of the rows
// through a two-slot ring of the largest pieces that fit: with two CTAs an SM,
// many calls are then in flight at once (ten for the Q4_K 4096 x 4096
// matvec), and a CTA's fixed costs (start-up, activation prep, the wait before
// it writes y) are spread over many rows. Measured on GB300, us a call in a
// stream of 256 independent calls (and of 20): Q4_K 4096 x 4096 with 103
// whole-share CTAs 2.12 (2.61), 38 ring CTAs 1.62 (2.24), 30 ring CTAs 1.56
// (2.24), 25 ring CTAs 1.56 (2.44), 16 ring CTAs 1.66 (2.82); Q6_K 4096 x
// 14336 with 152 CTAs 10.03 (10.7), 38 CTAs 8.65 (9.78), 30 CTAs 8.61 (9.68),
// 25 CTAs 8.61 (11.1); Q8_0 dp4a 14336 x 4096 with 38 CTAs 8.60 (9.7), 30
// CTAs 8.39 (8.6). Fewer CTAs stream faster in long streams but leave a
// longer tail in short ones. Chained and plain calls, and forced plans, keep
// the default plan (every SM).
template <class F>
inline int make_plan_for(const DevInfo& di, int rows, int k, int slots, const qmv_opts* cfg, KParams* kp, Plan* pl) {
    const int rc = make_plan_core<F>(di, rows, k, slots, cfg, kp, pl);
    if (rc || overlap_of(cfg) != QMV_OVERLAP_INDEPENDENT) return rc;
    if (cfg->ctas > 0 || cfg->chunk_rows > 0 || cfg->chunks > 0 || cfg->warps > 0 || cfg->unroll > 0 ||
        cfg->cluster > 0)
        return rc;   // a forced plan stays as forced
    const long long half = (di.smem_sm - 2LL * di.smem_reserved) / 2;
    const int per = slots > 1 ? slots : 1;
    const int want = std::max(1, (di.nsm / INDEP_SM_DIV + per - 1) / per);
    if (want >= pl->parts) return rc;   // small shapes: already few CTAs
    qmv_opts c = *cfg;
    c.ctas = want;
    c.warps = WARPS_TWO_PER_SM;
    c.chunks = 2;
    // the largest pieces (up to 8 rows) whose two-slot rings fit half an SM
    for (int cr = 8; cr >= 1; cr--) {
        c.chunk_rows = cr;
        KParams k2 = *kp;
        Plan p2;
        if (make_plan_core<F>(di, rows, k, slots, &c, &k2, &p2, half)) continue;
        // two slots (unless a row group has a single piece), so that a
        // piece is decoded while the next one lands
        const int most = std::max(k2.npc4[2], k2.npc4[3]);
        if (static_cast<long long>(p2.smem) <= half && p2.T <= 32 * WARPS_TWO_PER_SM && k2.S >= std::min(2, most)) {
            *kp = k2;
            *pl = p2;
            return QMV_OK;
        }
    }
    return rc;
}

// The same on the current device.
template <class F>
inline int make_plan(int rows, int k, int slots, const qmv_opts* cfg, KParams* kp, Plan* pl) {
    DevInfo di;
    const int rc = dev_info(&di, nullptr);
    return rc ? rc : make_plan_for<F>(di, rows, k, slots, cfg, kp, pl);
}

template <class F, int R, bool MOE, int MODE, bool WIDE>
inline int launch_one(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    auto kern = qmv_stream_kernel<F, R, MOE, MODE, WIDE>;
    static SmemOptIn opted;
    int dev = 0;
    DevInfo di;
    if (dev_info(&di, &dev)) return QMV_ECUDA;
    if (const int rc = ensure_smem(kern, opted, dev, static_cast<int>(pl.smem))) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.parts, MOE ? slots : 1, 1);
    lc.blockDim = dim3(pl.T, 1, 1);
    lc.dynamicSmemBytes = pl.smem;
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    int na = 0;
    if (pl.CL > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = static_cast<unsigned>(pl.CL);
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        na++;
    }
    if (pl.overlap != QMV_OVERLAP_NONE) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    lc.attrs = at;
    lc.numAttrs = na;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, kp));
}

template <class F, bool MOE, int MODE>
inline int launch(const KParams& kp, const Plan& pl, int slots, cudaStream_t stream) {
    // WIDE: a row's units fill whole warps (32 lanes per row).
    if (kp.GS == 32)
        return pl.R >= 2 ? launch_one<F, 2, MOE, MODE, true>(kp, pl, slots, stream)
                         : launch_one<F, 1, MOE, MODE, true>(kp, pl, slots, stream);
    return pl.R >= 2 ? launch_one<F, 2, MOE, MODE, false>(kp, pl, slots, stream)
                     : launch_one<F, 1, MOE, MODE, false>(kp, pl, slots, stream);
}

// Snapshot of this translation unit's status word, taken by status_xchg.
static __device__ unsigned int g_status_snap;

// One thread: read the status word (and clear it, in the same atomic
// exchange) into g_status_snap.
static __global__ void status_xchg(int clear) {
    g_status_snap = clear ? atomicExch(&g_status, 0u) : atomicOr(&g_status, 0u);
}

// Read (and optionally clear) this translation unit's device status word:
// wait for all work on the device, then read and clear it in one atomic
// exchange, so that no bit raised by a kernel of another host thread is lost
// between the read and the clear. Calls are serialised by a lock.
inline int status_rw(unsigned int* out, int clear) {
    static std::mutex mu;
    std::lock_guard<std::mutex> g(mu);
    int rc = cuda_rc(cudaDeviceSynchronize());
    if (rc) return rc;
    status_xchg<<<1, 1>>>(clear);
    rc = cuda_rc(cudaGetLastError());
    if (rc) return rc;
    unsigned int v = 0;
    rc = cuda_rc(cudaMemcpyFromSymbol(&v, g_status_snap, sizeof(v)));   // after the kernel (same stream)
    if (rc) return rc;
    *out = v;
    return QMV_OK;
}

}  // namespace qmv
