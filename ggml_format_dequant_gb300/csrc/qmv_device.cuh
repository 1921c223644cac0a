// qmv_device.cuh -- device-side building blocks shared by the quantized matvec
// kernels: bulk-copy (TMA) staging with bounded mbarrier waits, the integer
// "limb" form of the f32 activation, and deterministic group reductions.
//
// Target: sm_103a only (GB300). Nothing here is used by the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qmv {

constexpr unsigned FULL = 0xffffffffu;

// Status bits a kernel may raise in its translation unit's device status word.
constexpr unsigned STATUS_BAD_EXPERT_ID = 1u;   // an MoE id outside [0, n_experts)
constexpr unsigned STATUS_WAIT_TIMEOUT = 2u;    // a staged copy did not land in time

// Bound on one wait for a staged copy. A bulk copy of a few tens of KB lands in
// microseconds; if it has not after this long the kernel records the fact and
// stops instead of spinning forever.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;   // 2 s

// ----------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make freshly initialized barriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One potentially blocking test of phase `parity`: the hardware suspends the
// thread until the phase completes or the hint (in ns) runs out, so waiting
// warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after
// WAIT_LIMIT_NS. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// Programmatic dependent launch. launch_dependents lets the next kernel on the
// stream be scheduled before this one ends; dependency_wait blocks until every
// kernel this one depends on has finished and its memory is visible. Both are
// no-ops for a kernel launched without the programmatic-serialization
// attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One bulk (non-tensor) TMA copy global -> shared, completing on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void tma_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 only (LDGSTS); both
// addresses 16-byte aligned. Completion is tracked with commit/wait groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most n of this thread's most recent groups are still pending.
__device__ __forceinline__ void cp_async_wait(int n) {
    switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// d = c + sum of the four (unsigned byte of a) * (signed byte of b) products.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = c + sum of the four signed-byte products.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float f16_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// 16 bytes starting at a shared-memory address that is only 2-byte aligned:
// five aligned 32-bit loads and a funnel shift by 0 or 16 bits. The caller
// guarantees 4 readable bytes past the run.
__device__ __forceinline__ uint4 lds16_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    uint4 r;
    r.x = __funnelshift_r(w0, w1, sh);
    r.y = __funnelshift_r(w1, w2, sh);
    r.z = __funnelshift_r(w2, w3, sh);
    r.w = __funnelshift_r(w3, w4, sh);
    return r;
}

// 8 bytes at a 2-byte aligned shared address (three aligned loads).
__device__ __forceinline__ uint2 lds8_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// The 16-bit little-endian value at a 2-byte aligned shared address.
__device__ __forceinline__ uint32_t lds_u16_a2(const uint8_t* p) {
    return *reinterpret_cast<const unsigned short*>(p);
}

// --------------------------------------------------------- activation limbs
//
// The f32 activation is carried into the integer dot products as three signed
// byte "limbs" per element. Per 32-element group g with m = max|x_i| < 2^e the
// group exponent is s = 21 - e, each element becomes the integer
// X_i = rne(x_i * 2^s) with |X_i| <= 2^21, and X_i = a*65536 + b*256 + c with
// a in [-32, 32] and b, c in [-128, 127]. A weight-code dot then is
// sum q*X = 65536*sum(q*a) + 256*sum(q*b) + sum(q*c), three dp4a chains, and the
// f32 value is that integer times 2^-s. X_i keeps 21 bits below the group
// maximum, so the representation error of any element is at most 2^-22 * m.
//
// The integer is formed with one f32 fma: t = x*2^s + (2^23 + 0x208080) lies in
// [2^23, 2^24) where the f32 spacing is 1, so the fma's rounding is the RNE
// rounding of x*2^s, and the low 23 bits of t are M = X + 0x208080 whose three
// bytes are c + 128, b + 128 and a + 32.
constexpr int LIMB_BITS = 21;
constexpr float LIMB_MAGIC = 10518656.0f;   // 2^23 + 0x208080

struct XPrepSmem {
    uint8_t* la;       // [k] limb a (signed byte)
    uint8_t* lb;       // [k] limb b
    uint8_t* lc;       // [k] limb c
    float* xs;         // [k/32] 2^-s of each 32-group
    float* xsum16;     // [k/16] (sum of X over 16 elements) * 2^-s
};

// Fill the limb tables for x[0, k) (k a multiple of 32) with all T threads of
// the block. Each thread owns float4 slots i = tid, tid + T, ...; a 32-element
// group is 8 consecutive float4 slots, i.e. 8 consecutive lanes of one warp
// (T is a multiple of 32). Loads are issued BATCH at a time before any use so
// the prologue costs one or two memory round trips, not one per group.
template <int BATCH>
__device__ __forceinline__ void prep_limbs(const float* __restrict__ x, int k, const XPrepSmem& P, int tid,
                                           int T) {
    const int nvec = k >> 2;
    const float4* __restrict__ x4 = reinterpret_cast<const float4*>(x);
    for (int base = 0; base < nvec; base += BATCH * T) {
        float4 v[BATCH];
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            const int i = base + b * T + tid;
            v[b] = (i < nvec) ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            if (base + b * T >= nvec) break;   // uniform: nvec is a multiple of 8 and T of 32
            const int i = base + b * T + tid;
            const uint32_t m4 = max(max(__float_as_uint(v[b].x) & 0x7fffffffu, __float_as_uint(v[b].y) & 0x7fffffffu),
                                    max(__float_as_uint(v[b].z) & 0x7fffffffu, __float_as_uint(v[b].w) & 0x7fffffffu));
            uint32_t mx = max(m4, __shfl_xor_sync(FULL, m4, 4));
            mx = max(mx, __shfl_xor_sync(FULL, mx, 2));
            mx = max(mx, __shfl_xor_sync(FULL, mx, 1));
            const int E = static_cast<int>(mx >> 23);   // biased exponent of the group maximum
            int s = LIMB_BITS - (E - 126);               // max < 2^(E-126) for a normal maximum
            s = s > 126 ? 126 : s;                       // zero / tiny groups
            const float p2s = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
            const float p2ms = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
            const uint32_t M0 = __float_as_uint(__fmaf_rn(v[b].x, p2s, LIMB_MAGIC)) & 0x7fffffu;
            const uint32_t M1 = __float_as_uint(__fmaf_rn(v[b].y, p2s, LIMB_MAGIC)) & 0x7fffffu;
            const uint32_t M2 = __float_as_uint(__fmaf_rn(v[b].z, p2s, LIMB_MAGIC)) & 0x7fffffu;
            const uint32_t M3 = __float_as_uint(__fmaf_rn(v[b].w, p2s, LIMB_MAGIC)) & 0x7fffffu;
            // byte 0 of M is c + 128, byte 1 is b + 128, byte 2 is a + 32
            const uint32_t cw = __byte_perm(__byte_perm(M0, M1, 0x0040), __byte_perm(M2, M3, 0x0040), 0x5410) ^ 0x80808080u;
            const uint32_t bw = __byte_perm(__byte_perm(M0, M1, 0x0051), __byte_perm(M2, M3, 0x0051), 0x5410) ^ 0x80808080u;
            const uint32_t a0 = static_cast<uint32_t>(static_cast<int>(M0 >> 16) - 32);
            const uint32_t a1 = static_cast<uint32_t>(static_cast<int>(M1 >> 16) - 32);
            const uint32_t a2 = static_cast<uint32_t>(static_cast<int>(M2 >> 16) - 32);
            const uint32_t a3 = static_cast<uint32_t>(static_cast<int>(M3 >> 16) - 32);
            const uint32_t aw = __byte_perm(__byte_perm(a0, a1, 0x0040), __byte_perm(a2, a3, 0x0040), 0x5410);
            int X = static_cast<int>(M0 + M1 + M2 + M3) - 4 * 0x208080;
            X += __shfl_xor_sync(FULL, X, 2);
            X += __shfl_xor_sync(FULL, X, 1);
            // A whole 8-lane group is either inside [0, nvec) or past it
            // (nvec is a multiple of 8), so the shuffles above stay in step.
            if (i < nvec) {
                reinterpret_cast<uint32_t*>(P.la)[i] = aw;
                reinterpret_cast<uint32_t*>(P.lb)[i] = bw;
                reinterpret_cast<uint32_t*>(P.lc)[i] = cw;
                if ((tid & 3) == 0) P.xsum16[i >> 2] = __int2float_rn(X) * p2ms;
                if ((tid & 7) == 0) P.xs[i >> 3] = p2ms;
            }
        }
    }
}

// Combine the three limb partial sums into the exact integer sum q*X. The
// callers bound |sum q*X| below 2^31, so the wrapped 32-bit arithmetic is exact.
__device__ __forceinline__ int limb_combine(int sa, int sb, int sc) {
    return sa * 65536 + sb * 256 + sc;
}

}  // namespace qmv
