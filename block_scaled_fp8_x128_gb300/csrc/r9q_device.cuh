// Device-side building blocks of libr9q: PTX wrappers (mbarrier, TMA,
// clusters, tcgen05, mma.sync), the e4m3 conversions and the group-128
// quantiser.
// Everything here is sm_103a code; nothing is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace r9q {

constexpr int kBlock = 128;                 // scale block edge (K group and weight block)
// Bounds of the device waits (then an error is recorded and the kernel
// returns): an mbarrier try_wait without a hint suspends for ~3.7 us in
// hardware when the phase is not complete, so 2^18 tries last ~1 s; a counter
// poll with a 128 ns sleep takes ~0.2 us, so 2^22 polls last ~1 s.
constexpr uint32_t kSpinLimit = 1u << 18;
constexpr uint32_t kCountSpinLimit = 1u << 22;
constexpr int kErrTimeout = -6;             // R9Q_ERR_TIMEOUT

// ------------------------------------------------------------------ basics --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in bits 0..15
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_round(float v) {
    return bf16_lo(pack_bf16x2(v, 0.0f));
}

// two fp32 -> packed e4m3x2, round to nearest even, saturating to +-448
// (cvt .satfinite never yields the NaN code for finite input); `lo` -> bits 0..7
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// fl32(a / 448) without a division, by Markstein's correction of a quotient
// with a fused multiply-add (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): y0 = a * RN(1/448), the residual a - 448*y0 is exact in one FMA, and
// y0 + residual * RN(1/448) rounds to the IEEE quotient.  Checked against IEEE
// division for every finite bf16 a (the group maxima are bf16 values);
// tests/test_quant_arith.py.
__device__ __forceinline__ float div448(float a) {
    const float c = __uint_as_float(0x3B124925u);     // RN(1/448)
    const float y0 = __fmul_rn(a, c);
    const float r = __fmaf_rn(-448.0f, y0, a);
    return __fmaf_rn(r, c, y0);
}

// fl32(x / s) without a division, for bf16 x and a scale s = fl32(amax/448)
// of a bf16 amax, again by Markstein's FMA correction: with r = RN(1/s),
// y = RN(x*r), e = RN(x - s*y) (one FMA) and RN(y + e*r) (one FMA) is the
// IEEE quotient.  Rounding commutes with
// scaling by powers of two, so only the significands of x and amax matter:
// tests/test_quant_arith.py runs all 128 x 128 pairs in exact arithmetic.
// The reduction to significands needs no underflow in e, which holds for
// s >= 2^-90 whenever |x/s| >= 2^-11 (the lowest bit of s*y is at least
// 2^-147); smaller quotients give the e4m3 code 0 either way.  Callers send
// groups with smaller scales through the IEEE division.  The residual is
// formed as s*y - x and subtracted, so that x = -0 gives -0 (x - s*y would
// give +0 and the code 0x00 instead of 0x80).
constexpr float kQuotExactMinScale = 0x1p-90f;

__device__ __forceinline__ float quot_exact(float x, float s, float r) {
    const float y = __fmul_rn(x, r);
    const float e = __fmaf_rn(s, y, -x);
    return __fmaf_rn(-e, r, y);
}

// Group-128 quantisation of one group held by a full warp: lane l holds
// x[4l .. 4l+3].  scale = amax/448 (IEEE fp32 quotient); codes = e4m3(x/scale)
// with x/scale the IEEE fp32 quotient (see quot_exact); amax == 0 gives scale
// 0, codes 0.  Returns the lane's 4 codes packed little-endian (x[4l] in bits
// 0..7).
__device__ __forceinline__ uint32_t quant_group128_warp(float v0, float v1, float v2, float v3,
                                                        float& scale) {
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = div448(amax);
    scale = s;
    if (amax == 0.0f) return 0u;
    float t0, t1, t2, t3;
    if (s >= kQuotExactMinScale) {
        const float r = __frcp_rn(s);
        t0 = quot_exact(v0, s, r);
        t1 = quot_exact(v1, s, r);
        t2 = quot_exact(v2, s, r);
        t3 = quot_exact(v3, s, r);
    } else {
        t0 = __fdiv_rn(v0, s);
        t1 = __fdiv_rn(v1, s);
        t2 = __fdiv_rn(v2, s);
        t3 = __fdiv_rn(v3, s);
    }
    return cvt_e4m3x2(t0, t1) | (cvt_e4m3x2(t2, t3) << 16);
}

// Four groups per warp, eight lanes per group: lane l quantises values
// x[16*(l&7) .. 16*(l&7)+15] of group l>>3, given as 16 bf16 in v[0], v[1].
// Same results as quant_group128_warp, with three shuffle levels instead of
// five and sixteen independent quotients per lane.  Returns the lane's 16
// codes (x[16*(l&7)] in the low byte of .x).
__device__ __forceinline__ uint4 quant_group128_lane8(const uint4 (&v)[2], float& scale) {
    float x[16];
    const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w[i]);
        x[2 * i + 1] = bf16_hi(w[i]);
    }
    float a0 = fmaxf(fabsf(x[0]), fabsf(x[1])), a1 = fmaxf(fabsf(x[2]), fabsf(x[3]));
    float a2 = fmaxf(fabsf(x[4]), fabsf(x[5])), a3 = fmaxf(fabsf(x[6]), fabsf(x[7]));
    float a4 = fmaxf(fabsf(x[8]), fabsf(x[9])), a5 = fmaxf(fabsf(x[10]), fabsf(x[11]));
    float a6 = fmaxf(fabsf(x[12]), fabsf(x[13])), a7 = fmaxf(fabsf(x[14]), fabsf(x[15]));
    float amax = fmaxf(fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)), fmaxf(fmaxf(a4, a5), fmaxf(a6, a7)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float s = div448(amax);
    scale = s;
    const bool live = amax != 0.0f;
    float t[16];
    if (__any_sync(0xffffffffu, live && !(s >= kQuotExactMinScale))) {
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = __fdiv_rn(x[i], s);
    } else {
        const float r = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = quot_exact(x[i], s, r);
    }
    uint4 c;
    c.x = cvt_e4m3x2(t[0], t[1]) | (cvt_e4m3x2(t[2], t[3]) << 16);
    c.y = cvt_e4m3x2(t[4], t[5]) | (cvt_e4m3x2(t[6], t[7]) << 16);
    c.z = cvt_e4m3x2(t[8], t[9]) | (cvt_e4m3x2(t[10], t[11]) << 16);
    c.w = cvt_e4m3x2(t[12], t[13]) | (cvt_e4m3x2(t[14], t[15]) << 16);
    if (!live) c = make_uint4(0u, 0u, 0u, 0u);
    return c;
}

// e^x in fp32 with every rounding fixed, so that the SwiGLU result does not
// depend on a math library's implementation.  Method of Cody and Waite
// ("Software Manual for the Elementary Functions", 1980): k = rint(x log2 e);
// r = x - k ln2 with ln2 as an fp32 head plus an fp32 tail, one fused
// multiply-add each (the head step is exact); e^r = sum_{n=0..7} r^n / n!
// by Horner's rule in fused multiply-adds (|r| <= ln2/2); e^x = e^r 2^k.
// The scaling is two multiplies by 2^(k/2) and 2^(k - k/2): the first is
// exact, so the pair rounds once, like an exact ldexp.  x > 88.8 gives +inf,
// x < -104 gives +0 (e^x below half the smallest subnormal).  Under 1 ulp of
// the exponential over the fp32 range.
__device__ __forceinline__ float exp_cw(float x) {
    if (x > 88.8f) return __int_as_float(0x7F800000);
    if (x < -104.0f) return 0.0f;
    const float k = rintf(__fmul_rn(x, 0x1.715476p+0f));        // x / ln2
    float r = __fmaf_rn(-k, 0x1.62e430p-1f, x);                  // ln2 head
    r = __fmaf_rn(-k, -0x1.05c610p-29f, r);                      // ln2 tail
    float p = 0x1.a01a02p-13f;                                   // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);                        // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);                         // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);                         // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);                         // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = static_cast<int>(k);                          // -150 .. 128
    const int k1 = ki >> 1, k2 = ki - k1;                        // each in -75 .. 64
    const float s1 = __int_as_float((k1 + 127) << 23);
    const float s2 = __int_as_float((k2 + 127) << 23);
    return __fmul_rn(__fmul_rn(p, s1), s2);
}

// silu(g) * u in fp32 (g, u already bf16-rounded): e = exp(-g), g / (1 + e),
// times u, each step one IEEE rounding.  The separate-launch SwiGLU kernel and
// the fused gate_up epilogue both call this, so they agree bit for bit.
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float e = exp_cw(-g);
    const float sg = __fdiv_rn(g, __fadd_rn(1.0f, e));
    return __fmul_rn(sg, u);
}

// Exact e4m3 -> bf16 for four codes packed in w (byte i = code of element i).
// The code's 7 magnitude bits moved to bf16 bits 4..10 (sign to bit 15) are
// the bf16 encoding of value * 2^-120 (normal and subnormal codes alike, since
// both formats share the field layout); one bf16 multiply by 2^120 then gives
// the value exactly (bf16 arithmetic keeps subnormal inputs).  Outputs pair
// the elements as even = (x0, x2), odd = (x1, x3), low half first.
__device__ __forceinline__ void e4m3x4_to_bf16x2x2(uint32_t w, uint32_t& even, uint32_t& odd) {
    const uint32_t e = ((w << 4) & 0x07F007F0u) | ((w << 8) & 0x80008000u);
    const uint32_t o = ((w >> 4) & 0x07F007F0u) | (w & 0x80008000u);
    const uint32_t two120 = 0x7B807B80u;     // bf16 2^120 in both halves
    const uint32_t negz = 0x80008000u;       // -0 addend keeps x*y exact (and +0 for +0)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(even) : "r"(e), "r"(two120), "r"(negz));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(odd) : "r"(o), "r"(two120), "r"(negz));
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// generic-proxy shared-memory writes (e.g. mbarrier.init) become visible to the
// async proxy (TMA) of this CTA
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait that sleeps in hardware: each try_wait suspends the thread for up
// to `hint_ns` unless the phase completes first, so a waiting warp takes no
// issue slots from the warps that do the work.  False after `tries` attempts.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 20000,
                                                uint32_t tries = 1u << 16) {
    for (uint32_t i = 0; i < tries; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Bounded wait for the phase with the given parity; false after kSpinLimit
// tries.  try_wait itself suspends the thread for a while in hardware, so the
// loop polls without sleeping (a software sleep would oversleep the arrival).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Bounded wait (acquire, gpu scope) until *counter >= need; false after
// about a second.
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ bool wait_count(const int* counter, int need) {
    for (uint32_t i = 0; i < kCountSpinLimit; ++i) {
        if (ld_acquire(counter) >= need) return true;
        __nanosleep(128);
    }
    return false;
}

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled TMA prefetch of box {c0 (inner), c1} into L2: no shared memory, no
// completion to wait for; a later load of the same box then hits L2.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, multiple of 16).
// It only fills L2, so it never returns stale data: data another kernel writes
// afterwards replaces the lines in L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tiled TMA load of box {c0 (inner), c1} into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- clusters --

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrive without release semantics: enough where the only thing peers rely on
// is mbarrier initialisation, which fence_mbar_init (release at cluster
// scope) has already ordered before this arrive.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Asynchronous store of two floats into a cluster peer's shared memory (addr,
// from mapa); the 8 bytes count toward the transaction count of the mbarrier
// at `bar` (the peer's barrier, same address space) when they land.
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float x, float y, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(x), "f"(y), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

__device__ __forceinline__ float2 ld_dsmem_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// --------------------------------------------------- programmatic launches --

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mma.sync --

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// D(16x8 f32) += A(16x32 e4m3, row) * B(32x8 e4m3, col)
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ tcgen05 --

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle: rows of 128 bytes in 8-row atoms stacked every 1024 bytes (stride
// byte offset); the leading byte offset is unused for this layout (encoded as
// 16 bytes).  A step of 32 bytes of K inside the atom moves the start address.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;                     // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                     // SWIZZLE_128B
    return d;
}

// kind::f8f6f4 instruction descriptor: D fp32, A and B e4m3, both K-major.
constexpr uint32_t umma_idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one M x N x 32 e4m3 step; issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The barrier receives one arrival once every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void umma_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void umma_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole-warp TMEM allocation of `cols` columns (a power of two >= 32); the
// base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// NC consecutive TMEM columns of this thread's lane (NC = 8, 16 or 32).  The
// load is asynchronous: use the values only after tmem_wait_ld on them.
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&d)[NC]) {
    static_assert(NC == 8 || NC == 16 || NC == 32, "tcgen05.ld width");
    if constexpr (NC == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3]), "=f"(d[4]), "=f"(d[5]), "=f"(d[6]),
                       "=f"(d[7])
                     : "r"(taddr)
                     : "memory");
    } else if constexpr (NC == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15}, [%16];"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3]), "=f"(d[4]), "=f"(d[5]), "=f"(d[6]), "=f"(d[7]),
              "=f"(d[8]), "=f"(d[9]), "=f"(d[10]), "=f"(d[11]), "=f"(d[12]), "=f"(d[13]), "=f"(d[14]), "=f"(d[15])
            : "r"(taddr)
            : "memory");
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3]), "=f"(d[4]), "=f"(d[5]), "=f"(d[6]), "=f"(d[7]),
              "=f"(d[8]), "=f"(d[9]), "=f"(d[10]), "=f"(d[11]), "=f"(d[12]), "=f"(d[13]), "=f"(d[14]), "=f"(d[15]),
              "=f"(d[16]), "=f"(d[17]), "=f"(d[18]), "=f"(d[19]), "=f"(d[20]), "=f"(d[21]), "=f"(d[22]),
              "=f"(d[23]), "=f"(d[24]), "=f"(d[25]), "=f"(d[26]), "=f"(d[27]), "=f"(d[28]), "=f"(d[29]),
              "=f"(d[30]), "=f"(d[31])
            : "r"(taddr)
            : "memory");
    }
}
// Waits for this thread's TMEM loads; the values named count as written here,
// so no use of them moves above the wait.
template <int NC>
__device__ __forceinline__ void tmem_wait_ld(float (&d)[NC]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < NC; ++i) asm volatile("" : "+f"(d[i]));
}

// Asynchronous store of four floats into a cluster peer's shared memory (16
// bytes, 16-byte aligned), counted on the peer's mbarrier like st_async_f32x2.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float x, float y, float z, float w, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

}  // namespace r9q
