// Device-side building blocks of libr9q: PTX wrappers (mbarrier, TMA,
// clusters, mma.sync), the e4m3 conversions and the group-128 quantiser.
// Everything here is sm_103a code; nothing is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace r9q {

constexpr int kBlock = 128;                 // scale block edge (K group and weight block)
constexpr uint32_t kSpinLimit = 1u << 22;   // bounded waits: ~0.3 s with back-off, then error
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

// fl32(a / 448) without a division: y0 = a * RN(1/448), the residual
// a - 448*y0 is exact in one FMA, and y0 + residual * RN(1/448) rounds to
// the IEEE quotient.  Checked against IEEE division for every finite bf16 a
// (the group maxima are bf16 values); tests/test_quant_arith.py.
__device__ __forceinline__ float div448(float a) {
    const float c = __uint_as_float(0x3B124925u);     // RN(1/448)
    const float y0 = __fmul_rn(a, c);
    const float r = __fmaf_rn(-448.0f, y0, a);
    return __fmaf_rn(r, c, y0);
}

// q = e4m3(fl32(x / s)) without a division per element.  With r the hardware
// reciprocal of s (relative error below 2^-22) y = x*r lies within 6 fp32
// ulps of fl32(x/s).  The e4m3 rounding of a value only depends on which side
// of an e4m3 midpoint it lies, and for |v| >= 2^-6 those midpoints are exactly
// the fp32 values whose low 20 mantissa bits are 0x80000.  So y gives the same
// code unless it lies within 8 ulps of such a midpoint or in the e4m3
// subnormal range; those rare elements take the IEEE division.
__device__ __forceinline__ float quot_for_e4m3(float x, float s, float r) {
    const float y = __fmul_rn(x, r);
    const uint32_t lo = __float_as_uint(y) & 0xFFFFFu;
    if (fabsf(y) < 0x1p-6f || (lo - 0x7FFF8u) <= 16u) return __fdiv_rn(x, s);
    return y;
}

__device__ __forceinline__ float rcp_approx(float s) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
    return r;
}

// Group-128 quantisation of one group held by a full warp: lane l holds
// x[4l .. 4l+3].  scale = amax/448 (IEEE fp32 quotient); codes = e4m3(x/scale)
// exactly as one IEEE fp32 division per element would give (see
// quot_for_e4m3); amax == 0 gives scale 0, codes 0.  Returns the lane's 4
// codes packed little-endian (x[4l] in bits 0..7).
__device__ __forceinline__ uint32_t quant_group128_warp(float v0, float v1, float v2, float v3,
                                                        float& scale) {
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = div448(amax);
    scale = s;
    if (amax == 0.0f) return 0u;
    const float r = rcp_approx(s);
    float t0, t1, t2, t3;
    if (s >= 0x1p-125f) {          // reciprocal comfortably finite and normal
        t0 = quot_for_e4m3(v0, s, r);
        t1 = quot_for_e4m3(v1, s, r);
        t2 = quot_for_e4m3(v2, s, r);
        t3 = quot_for_e4m3(v3, s, r);
    } else {
        t0 = __fdiv_rn(v0, s);
        t1 = __fdiv_rn(v1, s);
        t2 = __fdiv_rn(v2, s);
        t3 = __fdiv_rn(v3, s);
    }
    return cvt_e4m3x2(t0, t1) | (cvt_e4m3x2(t2, t3) << 16);
}

// true when y = x * (1/s) might not give the code of fl32(x / s): y within 8
// ulps of an e4m3 rounding midpoint, or in the e4m3 subnormal range
__device__ __forceinline__ bool quot_risky(float y) {
    const uint32_t lo = __float_as_uint(y) & 0xFFFFFu;
    return fabsf(y) < 0x1p-6f || (lo - 0x7FFF8u) <= 16u;
}

// Four groups at once (independent chains interleaved for ILP): group j's
// lane values are the bf16 pairs in v[j]; same results as quant_group128_warp.
// The common case is branch-free; only when some lane of the warp holds a
// risky quotient (or a tiny scale) does the warp redo those elements with the
// IEEE division.
__device__ __forceinline__ void quant_group128_warp_x4(const uint2 (&v)[4], uint32_t (&codes)[4],
                                                       float (&scale)[4]) {
    float x[4][4], amax[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[j][0] = bf16_lo(v[j].x);
        x[j][1] = bf16_hi(v[j].x);
        x[j][2] = bf16_lo(v[j].y);
        x[j][3] = bf16_hi(v[j].y);
        amax[j] = fmaxf(fmaxf(fabsf(x[j][0]), fabsf(x[j][1])), fmaxf(fabsf(x[j][2]), fabsf(x[j][3])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
    float s[4], r[4], t[4][4];
    bool risky = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s[j] = div448(amax[j]);
        r[j] = rcp_approx(s[j]);
        scale[j] = s[j];
        const bool live = amax[j] != 0.0f;
        risky |= live && !(s[j] >= 0x1p-125f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            t[j][e] = __fmul_rn(x[j][e], r[j]);
            risky |= live && quot_risky(t[j][e]);
        }
    }
    if (__any_sync(0xffffffffu, risky)) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (amax[j] != 0.0f && (!(s[j] >= 0x1p-125f) || quot_risky(t[j][e]))) t[j][e] = __fdiv_rn(x[j][e], s[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t c = cvt_e4m3x2(t[j][0], t[j][1]) | (cvt_e4m3x2(t[j][2], t[j][3]) << 16);
        codes[j] = (amax[j] == 0.0f) ? 0u : c;
    }
}

// silu(g) * u in fp32 (g, u already bf16-rounded); the separate-launch SwiGLU
// kernel and the fused gate_up epilogue both call this, so they agree bit for bit.
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float e = expf(-g);
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

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
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

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

}  // namespace r9q
