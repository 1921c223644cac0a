// qmm_q4k_tc5.cu -- host side of the fifth-generation tensor-core batch
// kernel (qmm_tc5.cuh) for Q4_K rows: plan, tensor map, cluster launch.
#include <mutex>

#include "qmv_internal.h"
#include "qmm_tc5s.cuh"

namespace qmv {

// Smallest dynamic shared memory a CTA asks for: with this much, at most two
// CTAs share an SM, so two allocations of T5_TMEM_COLS columns always fit in
// an SM's tensor memory (a third CTA would wait in tcgen05.alloc).
constexpr long long T5_MIN_SMEM = 80 * 1024;
// Room left for the kernel's static shared memory (a few words) under the
// per-CTA opt-in limit.
constexpr long long T5_STATIC_SMEM = 1024;

// The plan: k-chunks per tile (the cluster size), ring slots and the
// shared-memory layout of the CTA with the most super-blocks.
inline int make_t5_plan(const DevInfo& di, int rows, int k, int m, const qmv_opts* cfg, T5Params* tp, Plan* pl) {
    if (rows <= 0 || k <= 0 || k % T5_SB || m < 1 || m > T5_COLS) return QMV_EINVAL;
    const int nsb = k / T5_SB;
    // k-chunks: a power of two (so that each of the CL ranks adds up exactly
    // 128 / CL rows of the tile), at most the cluster limit, the super-blocks
    // of a row, and the size asked for
    const int want = std::min((cfg && cfg->cluster > 0) ? std::min(cfg->cluster, CLUSTER_MAX) : CLUSTER_MAX, nsb);
    int CL = 1;
    while (2 * CL <= want) CL *= 2;
    const int nq = (nsb + CL - 1) / CL;   // super-blocks of the largest chunk
    int S = (cfg && cfg->chunks > 0) ? cfg->chunks : 4;
    S = std::max(1, std::min(S, nq));
    const uint32_t slot = static_cast<uint32_t>(T5_ROWS * T5_SBBYTES);
    // the kernel's static shared memory comes on top of the dynamic part
    const long long limit = di.smem_optin - T5_STATIC_SMEM;
    long long smem = 0;
    for (;; S--) {
        long long off = 0;
        tp->off_ring = 0;
        off = static_cast<long long>(S) * slot;
        tp->off_b = static_cast<uint32_t>(round_up(off, 128));
        off = tp->off_b + static_cast<long long>(nq) * 32 * 256;   // 32 k-blocks of 256 bytes a super-block
        tp->off_bm = static_cast<uint32_t>(round_up(off, 128));
        off = tp->off_bm + static_cast<long long>(nq) * 512;
        tp->off_sc = static_cast<uint32_t>(round_up(off, 16));
        off = tp->off_sc + static_cast<long long>(nq) * T5_COLS * 2 * 4;
        tp->off_x = static_cast<uint32_t>(round_up(off, 128));
        off = tp->off_x + static_cast<long long>(m) * nq * T5_SB * 4;
        tp->off_in = static_cast<uint32_t>(round_up(off, 16));
        off = tp->off_in + static_cast<long long>(T5_ROWS) * T5_COLS * 4;
        tp->off_bars = static_cast<uint32_t>(round_up(off, 8));
        off = tp->off_bars + 8LL * (2 * S + 10);
        smem = std::max(round_up(off, 128), T5_MIN_SMEM);
        if (smem <= limit) break;
        if (S == 1) return QMV_ETOOBIG;   // the chunk's x and B alone do not fit: a larger cluster is needed
    }
    tp->rows = rows;
    tp->k = k;
    tp->m = m;
    tp->nsb = nsb;
    tp->CL = CL;
    tp->S = S;
    tp->slot_bytes = slot;
    const int mode = overlap_of(cfg);
    tp->early_inputs = mode >= QMV_OVERLAP_INDEPENDENT ? 1 : 0;
    tp->late_alloc = mode == QMV_OVERLAP_CHAIN ? 1 : 0;
    pl->T = T5_THREADS;
    pl->parts = ((rows + T5_ROWS - 1) / T5_ROWS) * CL;
    pl->R = 1;
    pl->CL = CL;
    pl->overlap = mode;
    pl->smem = static_cast<size_t>(smem);
    return QMV_OK;
}

// Shared memory the streaming plan asks for at least: enough that no second
// CTA of this plan (more than half an SM) and no CTA of the cluster plan (at
// least T5_MIN_SMEM) fits beside it, so its allocation of all 512
// tensor-memory columns never meets another holder on the SM.
constexpr long long T5S_MIN_SMEM = 148 * 1024;
static_assert(T5S_MIN_SMEM + T5_MIN_SMEM + 2 * T5_STATIC_SMEM > 228 * 1024, "cluster-plan CTA beside a streaming one");

// The streaming plan (independent calls): one CTA a 128-row tile for the
// whole of k, with rings of weight copies, of B, and of the rows' d / dmin.
inline int make_t5s_plan(const DevInfo& di, int rows, int k, int m, const qmv_opts* cfg, T5SParams* tp, Plan* pl) {
    if (rows <= 0 || k <= 0 || k % T5_SB || m < 1 || m > T5_COLS) return QMV_EINVAL;
    const int nsb = k / T5_SB;
    int S = (cfg && cfg->chunks > 0) ? cfg->chunks : 6;
    S = std::max(1, std::min(S, nsb));
    const uint32_t slot = static_cast<uint32_t>(T5_ROWS * T5_SBBYTES);
    const long long limit = di.smem_optin - T5_STATIC_SMEM;
    long long smem = 0;
    for (;; S--) {
        long long off = static_cast<long long>(S) * slot;
        tp->off_ring = 0;
        tp->off_b = static_cast<uint32_t>(round_up(off, 128));
        off = tp->off_b + static_cast<long long>(T5S_SB) * T5S_BSLOT;
        tp->off_bm = static_cast<uint32_t>(round_up(off, 128));
        off = tp->off_bm + static_cast<long long>(T5S_SB) * T5S_BMSLOT;
        tp->off_sc = static_cast<uint32_t>(round_up(off, 16));
        off = tp->off_sc + static_cast<long long>(T5S_SB) * T5_COLS * 2 * 4;
        tp->off_dm = static_cast<uint32_t>(round_up(off, 16));
        off = tp->off_dm + static_cast<long long>(T5S_SD) * T5_ROWS * 8;
        tp->off_bars = static_cast<uint32_t>(round_up(off, 8));
        off = tp->off_bars + 8LL * (2 * S + T5S_NBARS_FIXED);
        smem = std::max(round_up(off, 128), T5S_MIN_SMEM);
        if (smem <= limit) break;
        if (S == 1) return QMV_ETOOBIG;
    }
    tp->rows = rows;
    tp->k = k;
    tp->m = m;
    tp->nsb = nsb;
    tp->S = S;
    tp->slot_bytes = slot;
    const int mode = overlap_of(cfg);
    tp->early_inputs = mode >= QMV_OVERLAP_INDEPENDENT ? 1 : 0;
    pl->T = T5S_THREADS;
    pl->parts = (rows + T5_ROWS - 1) / T5_ROWS;
    pl->R = 1;
    pl->CL = 1;
    pl->overlap = mode;
    pl->smem = static_cast<size_t>(smem);
    return QMV_OK;
}

// Independent calls take the streaming plan, unless a cluster size is forced.
inline bool t5_streams(const qmv_opts* cfg) {
    return overlap_of(cfg) == QMV_OVERLAP_INDEPENDENT && !(cfg && cfg->cluster > 0);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
inline EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of the packed rows: 8-byte elements, rows x (row bytes / 8), a
// box of one super-block (18 elements) by 128 rows; rows past the end read as
// zeros.
inline int make_wmap(const void* w, int rows, int nsb, CUtensorMap* map) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return QMV_ECUDA;
    const cuuint64_t rowbytes = static_cast<cuuint64_t>(nsb) * T5_SBBYTES;
    const cuuint64_t dims[2] = {rowbytes / 8, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {rowbytes};
    const cuuint32_t box[2] = {T5_SBBYTES / 8, T5_ROWS};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(w), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QMV_OK : QMV_EINVAL;
}

inline int launch_t5(const CUtensorMap& map, const T5Params& tp, const Plan& pl, cudaStream_t stream) {
    auto kern = qmm_tc5_q4k_kernel;
    static SmemOptIn opted;
    int dev = 0;
    DevInfo di;
    if (dev_info(&di, &dev)) return QMV_ECUDA;
    if (const int rc = ensure_smem(kern, opted, dev, static_cast<int>(pl.smem))) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.parts, 1, 1);
    lc.blockDim = dim3(pl.T, 1, 1);
    lc.dynamicSmemBytes = pl.smem;
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = static_cast<unsigned>(pl.CL);
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    na++;
    if (pl.overlap != QMV_OVERLAP_NONE) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    lc.attrs = at;
    lc.numAttrs = na;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, map, tp));
}

inline int launch_t5s(const CUtensorMap& map, const T5SParams& tp, const Plan& pl, cudaStream_t stream) {
    auto kern = qmm_tc5s_q4k_kernel;
    static SmemOptIn opted;
    int dev = 0;
    DevInfo di;
    if (dev_info(&di, &dev)) return QMV_ECUDA;
    if (const int rc = ensure_smem(kern, opted, dev, static_cast<int>(pl.smem))) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.parts, 1, 1);
    lc.blockDim = dim3(pl.T, 1, 1);
    lc.dynamicSmemBytes = pl.smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    int na = 0;
    if (pl.overlap != QMV_OVERLAP_NONE) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    lc.attrs = at;
    lc.numAttrs = na;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, map, tp));
}

}  // namespace qmv

namespace qmvi {

using namespace qmv;

int qmm_q4k_tc5(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                cudaStream_t s, int force_timeout) {
    if (!w || !x || !y || rows <= 0 || k <= 0 || m <= 0 || k % T5_SB) return QMV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(x) & 15u)) return QMV_EINVAL;
    DevInfo di;
    int rc = dev_info(&di, nullptr);
    if (rc) return rc;
    CUtensorMap map;
    rc = make_wmap(w, rows, k / T5_SB, &map);
    if (rc) return rc;
    const int tiles = (m + T5_COLS - 1) / T5_COLS;
    for (int t0 = 0, m0 = 0; t0 < tiles; t0++) {
        const int mt = m / tiles + (t0 < m % tiles ? 1 : 0);
        if (t5_streams(cfg)) {
            T5SParams sp{};
            Plan spl;
            if (make_t5s_plan(di, rows, k, mt, cfg, &sp, &spl) == QMV_OK) {
                sp.x = x + static_cast<long long>(m0) * k;
                sp.y = y + static_cast<long long>(m0) * rows;
                sp.force_timeout = force_timeout;
                rc = launch_t5s(map, sp, spl, s);
                if (rc) return rc;
                m0 += mt;
                continue;
            }
        }
        T5Params tp{};
        Plan pl;
        rc = make_t5_plan(di, rows, k, mt, cfg, &tp, &pl);
        if (rc) return rc;
        tp.x = x + static_cast<long long>(m0) * k;
        tp.y = y + static_cast<long long>(m0) * rows;
        tp.force_timeout = force_timeout;
        rc = launch_t5(map, tp, pl, s);
        if (rc) return rc;
        m0 += mt;
    }
    return QMV_OK;
}

int status_qmm_q4k_tc5(unsigned int* out, int clear) { return status_rw(out, clear); }

int qmm_q4k_tc5_plan(const int* device, int rows, int k, int m, const qmv_opts* cfg, int* out) {
    DevInfo di;
    di.nsm = device[0];
    di.smem_optin = device[1];
    di.smem_sm = device[2];
    di.smem_reserved = device[3];
    if (di.nsm <= 0 || di.smem_optin <= 0 || di.smem_sm <= 0 || di.smem_reserved < 0) return QMV_EINVAL;
    if (t5_streams(cfg)) {
        T5SParams sp{};
        Plan spl;
        if (make_t5s_plan(di, rows, k, m, cfg, &sp, &spl) == QMV_OK) {
            const int v[13] = {spl.parts, spl.T, static_cast<int>(spl.smem), 1, sp.S, sp.nsb,
                               static_cast<int>(sp.off_b), static_cast<int>(sp.off_bm), static_cast<int>(sp.off_sc),
                               static_cast<int>(sp.off_dm), 0, static_cast<int>(sp.off_bars), 1};
            for (int i = 0; i < 13; i++) out[i] = v[i];
            return QMV_OK;
        }
    }
    T5Params tp{};
    Plan pl;
    const int rc = make_t5_plan(di, rows, k, m, cfg, &tp, &pl);
    if (rc) return rc;
    const int v[13] = {pl.parts, pl.T, static_cast<int>(pl.smem), tp.CL, tp.S, tp.nsb, static_cast<int>(tp.off_b),
                       static_cast<int>(tp.off_bm), static_cast<int>(tp.off_sc), static_cast<int>(tp.off_x),
                       static_cast<int>(tp.off_in), static_cast<int>(tp.off_bars), 0};
    for (int i = 0; i < 13; i++) out[i] = v[i];
    return QMV_OK;
}

}  // namespace qmvi
