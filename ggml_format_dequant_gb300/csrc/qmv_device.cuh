// qmv_device.cuh -- device-side building blocks shared by the quantized matvec
// kernels: bulk-copy (TMA) staging with bounded mbarrier waits, shared-memory
// loads by 32-bit address, and the integer "limb" form of the f32 activation.
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
constexpr unsigned STATUS_OUT_OF_BOUNDS = 4u;   // checking build only: an access outside its region

// The checking build (compiled with QMV_BOUNDS_CHECK) tests every shared- and
// global-memory access of the matvec kernel against the region the plan gives
// it; an access outside raises STATUS_OUT_OF_BOUNDS and is skipped or moved
// to the region's start. In the normal build the tests fold away.
#ifdef QMV_BOUNDS_CHECK
constexpr bool BOUNDS_CHECK = true;
#else
constexpr bool BOUNDS_CHECK = false;
#endif

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

// Order earlier generic-proxy shared-memory accesses (as seen by this thread)
// before its later bulk copies into the same memory.
__device__ __forceinline__ void fence_proxy_async() {
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

// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after
// limit_ns. Returns false on timeout. A phase that is already complete (the
// usual case when the data was requested long before) costs one test.
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The same with the kernels' limit, WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    return mbar_wait_bounded_ns(bar, parity, WAIT_LIMIT_NS);
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

// ------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address, in the cluster's shared window, of shared address `a` of CTA
// `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t a, const uint4& v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t a, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Every thread of every CTA of the cluster: writes before it (to any CTA's
// shared memory) are visible to all after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------- shared loads by 32-bit address
//
// The staged weights are read with explicit ld.shared on 32-bit addresses (the
// immediate offsets fold into the instruction). They are volatile so that they
// stay after the mbarrier wait that publishes the data.

template <int OFF>
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
    return v;
}

template <int OFF>
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
    return v;
}

template <int OFF>
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a), "n"(OFF));
    return v;
}

// 16 bytes of a run that starts `sh` bits (0 or 16) past the 4-byte-aligned
// address wa + OFF: five aligned loads and four funnel shifts. Reads up to 4
// bytes past the run.
template <int OFF>
__device__ __forceinline__ uint4 lds16_sh(uint32_t wa, uint32_t sh) {
    const uint32_t w0 = lds32<OFF>(wa), w1 = lds32<OFF + 4>(wa), w2 = lds32<OFF + 8>(wa),
                   w3 = lds32<OFF + 12>(wa), w4 = lds32<OFF + 16>(wa);
    uint4 r;
    r.x = __funnelshift_r(w0, w1, sh);
    r.y = __funnelshift_r(w1, w2, sh);
    r.z = __funnelshift_r(w2, w3, sh);
    r.w = __funnelshift_r(w3, w4, sh);
    return r;
}

// 8 bytes, same convention (reads up to 4 bytes past the run).
template <int OFF>
__device__ __forceinline__ uint2 lds8_sh(uint32_t wa, uint32_t sh) {
    const uint32_t w0 = lds32<OFF>(wa), w1 = lds32<OFF + 4>(wa), w2 = lds32<OFF + 8>(wa);
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// ---------------------------------------------------------------- integers

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

// Small integers reach f32 through the exponent field: for 0 <= v < 2^22 the
// bit pattern 0x4B000000 + v is the float 2^23 + v, so s*v = fma(s, that,
// -s*2^23) is the correctly rounded product in one instruction once -s*2^23 is
// known. The pattern 0x4B400000 (the float 1.5*2^23) plus a sign-extended v in
// [-2^22, 2^22) is 1.5*2^23 + v, used the same way with -s*1.5*2^23.
constexpr float TWO23 = 8388608.0f;
constexpr float THREE22 = 12582912.0f;   // 1.5 * 2^23

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
constexpr float LIMB_MAGIC = 10518656.0f;          // 2^23 + 0x208080
constexpr uint32_t LIMB_MAGIC_BITS = 0x4B208080u;  // its bit pattern

// Shared-memory limb tables of x[0, k), as byte offsets into dynamic shared
// memory: limb bytes la, lb, lc [k rounded up to 128]; the 2^-s of every
// 32-group (xs, [k/32] floats); and (sum of X over every 16 elements) * 2^-s
// (xsum16, [k/16]).
struct LimbTables {
    uint32_t la, lb, lc, xs, xsum16;
};

// The limb bytes of elements 16c .. 16c+15 (16-byte chunk c) are stored in
// chunk limb_chunk(c): bits 3..5 of c are XORed into bits 0..2, which permutes
// chunks within each aligned group of 8. Lanes that read chunks 4u + v or
// 2u + v (one unit of 64 or 32 activations each) then hit distinct banks.
__host__ __device__ __forceinline__ uint32_t limb_chunk(uint32_t c) { return c ^ ((c >> 3) & 7u); }

// Limb words of four consecutive elements from their fma bit patterns (see
// above): the words of limbs a, b and c, one signed byte per element.
__device__ __forceinline__ void limb_words(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3, uint32_t& aw,
                                           uint32_t& bw, uint32_t& cw) {
    // byte transpose: (c0 c1 b0 b1), (c2 c3 b2 b3), (a0 a1 . .), (a2 a3 . .)
    const uint32_t s01 = __byte_perm(t0, t1, 0x5140);
    const uint32_t s23 = __byte_perm(t2, t3, 0x5140);
    const uint32_t a01 = __byte_perm(t0, t1, 0x0062);
    const uint32_t a23 = __byte_perm(t2, t3, 0x0062);
    cw = __byte_perm(s01, s23, 0x5410) ^ 0x80808080u;
    bw = __byte_perm(s01, s23, 0x7632) ^ 0x80808080u;
    // bytes a + 32 lie in [0, 64], so (byte + 96) ^ 0x80 is a as a signed byte
    // and the word add never carries between bytes
    aw = (__byte_perm(a01, a23, 0x5410) + 0x60606060u) ^ 0x80808080u;
}

// Largest magnitude of 16 activations (four float4).
__device__ __forceinline__ float max_abs16(const float4* v) {
    float mx = 0.0f;
#pragma unroll
    for (int m = 0; m < 4; m++)
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[m].x), fabsf(v[m].y)), fmaxf(fabsf(v[m].z), fabsf(v[m].w))));
    return mx;
}

// The power-of-two scale of a 32-element group from its largest magnitude
// mx: p2s = 2^s puts the group maximum just below 2^21, p2ms = 2^-s.
__device__ __forceinline__ void group_scale(float mx, float& p2s, float& p2ms) {
    const int E = static_cast<int>(__float_as_uint(mx) >> 23);   // biased exponent of the group maximum
    int s = LIMB_BITS - (E - 126);                               // max < 2^(E-126) for a normal maximum
    s = s > 126 ? 126 : s;                                       // zero / tiny groups
    p2s = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
    p2ms = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}

// Limb words of 16 consecutive activations (four float4) under the group
// scale p2s: word m of each limb holds elements 4m .. 4m+3, one signed byte
// each. Returns the exact integer sum of the 16 X.
__device__ __forceinline__ int limbs16(const float4* v, float p2s, uint32_t* A, uint32_t* B, uint32_t* C) {
    uint32_t tsum = 0;
#pragma unroll
    for (int m = 0; m < 4; m++) {
        const uint32_t t0 = __float_as_uint(__fmaf_rn(v[m].x, p2s, LIMB_MAGIC));
        const uint32_t t1 = __float_as_uint(__fmaf_rn(v[m].y, p2s, LIMB_MAGIC));
        const uint32_t t2 = __float_as_uint(__fmaf_rn(v[m].z, p2s, LIMB_MAGIC));
        const uint32_t t3 = __float_as_uint(__fmaf_rn(v[m].w, p2s, LIMB_MAGIC));
        limb_words(t0, t1, t2, t3, A[m], B[m], C[m]);
        tsum += t0 + t1 + t2 + t3;
    }
    // sum of the 16 X: sum of the patterns minus 16 magic patterns (mod 2^32)
    return static_cast<int>(tsum - 16u * LIMB_MAGIC_BITS);
}

// Limb words, sum and scale of one 16-element half (elements 16h .. 16h+15)
// held as four float4 by this thread; its partner lane (lane ^ 1) holds the
// other half of the 32-element group and calls this at the same time (the
// group maximum is exchanged with one shuffle, so every lane of the warp must
// call it). Writes the half's 16-byte chunk of each limb table, its sum, and
// (even h) the group's scale into the CTA's own tables when `store` is set.
__device__ __forceinline__ void prep_half(const float4 (&v)[4], uint32_t h, bool store, uint8_t* smem,
                                          const LimbTables& L) {
    float mx = max_abs16(v);
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));    // the group's other half
    float p2s, p2ms;
    group_scale(mx, p2s, p2ms);
    uint4 A, B, C;
    const int X = limbs16(v, p2s, &A.x, &B.x, &C.x);
    if (store) {
        const uint32_t o = limb_chunk(h) << 4;
        *reinterpret_cast<uint4*>(smem + L.la + o) = A;
        *reinterpret_cast<uint4*>(smem + L.lb + o) = B;
        *reinterpret_cast<uint4*>(smem + L.lc + o) = C;
        reinterpret_cast<float*>(smem + L.xsum16)[h] = __int2float_rn(X) * p2ms;
        if ((h & 1u) == 0) reinterpret_cast<float*>(smem + L.xs)[h >> 1] = p2ms;
    }
}

// Fill the CTA's own limb tables for x[0, k) (k a multiple of 32) with all T
// threads (T even): thread t converts halves t, t + T, t + 2T, ..., BATCH at
// a time with all of a batch's loads issued before any use. A half and its
// group partner (h ^ 1) land in neighbouring lanes of one warp because T is
// even; lanes past the last half join the shuffle with zeros and store
// nothing. The caller makes the tables visible with a block barrier.
template <int BATCH>
__device__ __forceinline__ void prep_limbs_cta(const float* __restrict__ x, int k, uint8_t* smem,
                                               const LimbTables& L, int tid, int T) {
    const int nh = k >> 4;
    const float4* __restrict__ x4 = reinterpret_cast<const float4*>(x);
    for (int base = 0; base < nh; base += BATCH * T) {
        float4 v[BATCH][4];
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            const int h = base + b * T + tid;
#pragma unroll
            for (int m = 0; m < 4; m++) v[b][m] = h < nh ? __ldg(x4 + 4 * h + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            if (base + b * T >= nh) break;   // uniform across the block
            const int h = base + b * T + tid;
            prep_half(v[b], static_cast<uint32_t>(h), h < nh, smem, L);
        }
    }
}

// The activation quantization of the dp4a path for 16 values of a 32-element
// block whose largest magnitude is amax (exact in any order): inv = 127/amax
// and d = amax/127 as IEEE f32 divides, q = clamp(round_half_even(x * inv),
// -127, 127) with one f32 multiply; amax == 0 gives d = 0 and every q = 0.
// codes: the 16 int8 codes, four to a word (byte i of word j is code 4j + i).
// Returns d; sum receives the integer sum of the 16 codes.
__device__ __forceinline__ float quantize_half_q8(const float4* v, float amax, uint32_t* codes, int& sum) {
    float d = 0.0f, inv = 0.0f;
    if (amax != 0.0f) {
        inv = __fdiv_rn(127.0f, amax);
        d = __fdiv_rn(amax, 127.0f);
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int q = __float2int_rn(__fmul_rn(e[i], inv));
            q = q > 127 ? 127 : (q < -127 ? -127 : q);
            s += q;
            w |= (static_cast<uint32_t>(q) & 0xffu) << (8 * i);
        }
        codes[j] = w;
    }
    sum = s;
    return d;
}

// The same for a whole 32-element block held by one thread (v: its 32
// values; codes: 8 words). Returns d; sum receives the codes' integer sum.
__device__ __forceinline__ float quantize_block_q8(const float4 (&v)[8], uint32_t (&codes)[8], int& sum) {
    const float amax = fmaxf(max_abs16(v), max_abs16(v + 4));
    int s0, s1;
    const float d = quantize_half_q8(v, amax, codes, s0);
    quantize_half_q8(v + 4, amax, codes + 4, s1);
    sum = s0 + s1;
    return d;
}

// The activation quantization done by a CTA into its own shared memory: two
// threads per 32-element block (neighbouring lanes, 16 values each, one
// shuffle for the block maximum; all lanes of a warp take part), the steps
// of quantize_half_q8, so the codes and scales equal the standalone
// quantizer's bit for bit. T even. xq: k bytes (16-byte aligned), xs: k/32
// floats; the caller publishes them with a block barrier.
__device__ __forceinline__ void quantize_x_cta(const float* __restrict__ x, int k, int8_t* xq, float* xs, int tid,
                                               int T) {
    const int nh = k >> 4;
    const float4* __restrict__ x4 = reinterpret_cast<const float4*>(x);
    for (int base = 0; base < nh; base += T) {
        const int h = base + tid;
        const bool valid = h < nh;
        float4 v[4];
#pragma unroll
        for (int m = 0; m < 4; m++) v[m] = valid ? __ldg(x4 + 4 * h + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        float amax = max_abs16(v);
        amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));   // the block's other half
        uint32_t codes[4];
        int sum;
        const float d = quantize_half_q8(v, amax, codes, sum);
        if (valid) {
            *reinterpret_cast<uint4*>(xq + 16 * h) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            if ((h & 1) == 0) xs[h >> 1] = d;
        }
    }
}

// Fill the limb tables for x[0, k) (k a multiple of 32) with all T threads of
// the block (T even), shared among the CL CTAs of a cluster: CTA `rank`
// converts halves [rank * nh / CL, (rank + 1) * nh / CL) of the nh = k/16
// 16-element halves and writes them into the tables of every CTA of the
// cluster (CL == 1: its own tables only). The caller makes them visible with a
// cluster (or block) barrier. A 32-element group is converted by two
// neighbouring threads, 16 elements (one 16-byte chunk of each limb table)
// each: thread slot h covers elements 16h .. 16h+15 and its partner (lane ^ 1)
// the other half of the group. All of a thread's loads are issued before any
// use, BATCH halves at a time. nh / CL must be even.
template <int BATCH>
__device__ __forceinline__ void prep_limbs(const float* __restrict__ x, int k, uint8_t* smem, const LimbTables& L,
                                           int tid, int T, int CL, uint32_t rank) {
    const int nhc = (k >> 4) / CL;            // halves converted by this CTA
    const int h0 = static_cast<int>(rank) * nhc;
    // Every CTA reads the same x: start each one at a different (even) offset
    // so that their requests spread over the lines instead of all asking for
    // the same line at once.
    const int rot = static_cast<int>((blockIdx.x * 64u) % static_cast<unsigned>(nhc));
    const uint32_t sbase = smem_u32(smem);
    const float4* __restrict__ x4 = reinterpret_cast<const float4*>(x) + 4 * h0;
    for (int base = 0; base < nhc; base += BATCH * T) {
        float4 v[BATCH][4];
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            int hl = base + b * T + tid;
            hl = (hl < nhc) ? (hl + rot < nhc ? hl + rot : hl + rot - nhc) : nhc;
#pragma unroll
            for (int m = 0; m < 4; m++)
                v[b][m] = (hl < nhc) ? __ldg(x4 + 4 * hl + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < BATCH; b++) {
            if (base + b * T >= nhc) break;   // uniform: nhc and T are even, so partners stay together
            int hl = base + b * T + tid;      // rotated like the loads (rot even: partners stay partners)
            hl = (hl < nhc) ? (hl + rot < nhc ? hl + rot : hl + rot - nhc) : nhc;
            uint32_t mx = 0;
#pragma unroll
            for (int m = 0; m < 4; m++)
                mx = max(mx, max(max(__float_as_uint(v[b][m].x) & 0x7fffffffu, __float_as_uint(v[b][m].y) & 0x7fffffffu),
                                 max(__float_as_uint(v[b][m].z) & 0x7fffffffu, __float_as_uint(v[b][m].w) & 0x7fffffffu)));
            mx = max(mx, __shfl_xor_sync(FULL, mx, 1));   // the group's other half
            const int E = static_cast<int>(mx >> 23);     // biased exponent of the group maximum
            int s = LIMB_BITS - (E - 126);                 // max < 2^(E-126) for a normal maximum
            s = s > 126 ? 126 : s;                         // zero / tiny groups
            const float p2s = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
            const float p2ms = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
            uint4 A, B, C;
            uint32_t tsum = 0;
            uint32_t* Ap = &A.x;
            uint32_t* Bp = &B.x;
            uint32_t* Cp = &C.x;
#pragma unroll
            for (int m = 0; m < 4; m++) {
                // bit patterns 0x4B000000 | M; M's bytes are c + 128, b + 128, a + 32
                const uint32_t t0 = __float_as_uint(__fmaf_rn(v[b][m].x, p2s, LIMB_MAGIC));
                const uint32_t t1 = __float_as_uint(__fmaf_rn(v[b][m].y, p2s, LIMB_MAGIC));
                const uint32_t t2 = __float_as_uint(__fmaf_rn(v[b][m].z, p2s, LIMB_MAGIC));
                const uint32_t t3 = __float_as_uint(__fmaf_rn(v[b][m].w, p2s, LIMB_MAGIC));
                limb_words(t0, t1, t2, t3, Ap[m], Bp[m], Cp[m]);
                tsum += t0 + t1 + t2 + t3;
            }
            // sum of the 16 X: sum of the patterns minus 16 magic patterns (mod 2^32)
            const int X = static_cast<int>(tsum - 16u * LIMB_MAGIC_BITS);
            const float xsum = __int2float_rn(X) * p2ms;
            if (hl < nhc) {   // always true here; keeps the stores visibly in bounds
                const uint32_t h = static_cast<uint32_t>(h0 + hl);
                const uint32_t o = limb_chunk(h) << 4;
                if (CL == 1) {
                    *reinterpret_cast<uint4*>(smem + L.la + o) = A;
                    *reinterpret_cast<uint4*>(smem + L.lb + o) = B;
                    *reinterpret_cast<uint4*>(smem + L.lc + o) = C;
                    reinterpret_cast<float*>(smem + L.xsum16)[h] = xsum;
                    if ((h & 1u) == 0) reinterpret_cast<float*>(smem + L.xs)[h >> 1] = p2ms;
                } else {
                    for (int r = 0; r < CL; r++) {
                        const uint32_t rr = static_cast<uint32_t>(r);
                        st_cluster_v4(cluster_addr(sbase + L.la + o, rr), A);
                        st_cluster_v4(cluster_addr(sbase + L.lb + o, rr), B);
                        st_cluster_v4(cluster_addr(sbase + L.lc + o, rr), C);
                        st_cluster_f32(cluster_addr(sbase + L.xsum16 + 4u * h, rr), xsum);
                        if ((h & 1u) == 0) st_cluster_f32(cluster_addr(sbase + L.xs + 4u * (h >> 1), rr), p2ms);
                    }
                }
            }
        }
    }
}

}  // namespace qmv
