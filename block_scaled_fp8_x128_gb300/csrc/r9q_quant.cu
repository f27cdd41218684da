// Standalone quantisation kernels of libr9q (sm_103a):
//   * fp32 -> e4m3 conversion (the codec every quantiser uses),
//   * per-token-group-128 activation quantisation (the separate pass of the
//     unfused W8A8 path; r9700-stack v0.3.1 notes: what runs when the fused
//     activation quant is switched off),
//   * weight quantisation with one fp32 scale per 128x128 block (set-up),
//   * the SwiGLU of the separate-launch expert MLP chain (releases page,
//     v0.3.3 "What changed": the three-launch path the fused one must match).
// All are bandwidth-bound elementwise/reduction kernels: 16-byte coalesced
// accesses, warp-shuffle reductions, grids sized to cover the SMs.
#include "r9q_device.cuh"
#include "r9q_kernels.h"

namespace r9q {

// ------------------------------------------------------------------ codec --

__global__ void __launch_bounds__(256) e4m3_from_f32_kernel(const float* __restrict__ x, int64_t n,
                                                            uint8_t* __restrict__ q) {
    const int64_t n4 = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = reinterpret_cast<const float4*>(x)[i];
        reinterpret_cast<uint32_t*>(q)[i] = cvt_e4m3x2(v.x, v.y) | (cvt_e4m3x2(v.z, v.w) << 16);
    }
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        q[i] = (uint8_t)cvt_e4m3x2(x[i], 0.0f);
}

cudaError_t launch_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, cudaStream_t st, int sms) {
    if (n == 0) return cudaSuccess;
    int64_t want = (n / 4 + 255) / 256;
    int grid = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
    e4m3_from_f32_kernel<<<grid, 256, 0, st>>>(x, n, q);
    return cudaGetLastError();
}

// ------------------------------------------------------ group-128 quant --

// Four groups per warp step, eight lanes per group (lane l: 16 values of group
// l >> 3, see quant_group128_lane8); a warp takes 16 consecutive groups of the
// flattened [M][KB] group array per iteration, all loads in flight before any
// is quantised.  K is a multiple of 128, so groups never straddle rows.
constexpr int kQGroupsPerWarp = 16;

__global__ void __launch_bounds__(256) quant_group128_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                             int64_t K, uint8_t* __restrict__ xq,
                                                             float* __restrict__ xs) {
    const int64_t groups = M * (K / kBlock);
    const int lane = threadIdx.x & 31;
    const int gl = lane >> 3, el = (lane & 7) * 16;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t g0 = ((int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kQGroupsPerWarp; g0 < groups;
         g0 += warps * kQGroupsPerWarp) {
        uint4 v[kQGroupsPerWarp / 4][2];
#pragma unroll
        for (int j = 0; j < kQGroupsPerWarp / 4; ++j) {
            const int64_t g = g0 + 4 * j + gl;
            if (g < groups) {
                const uint4* q = reinterpret_cast<const uint4*>(x + g * kBlock + el);
                v[j][0] = q[0];
                v[j][1] = q[1];
            } else {
                v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < kQGroupsPerWarp / 4; ++j) {
            if (g0 + 4 * j < groups) {
                const int64_t g = g0 + 4 * j + gl;
                float sc;
                const uint4 codes = quant_group128_lane8(v[j], sc);
                if (g < groups) {
                    *reinterpret_cast<uint4*>(xq + g * kBlock + el) = codes;
                    if ((lane & 7) == 0) xs[g] = sc;
                }
            }
        }
    }
}

cudaError_t launch_quant_group128(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                                  cudaStream_t st, int sms) {
    const int64_t groups = M * (K / kBlock);
    const int64_t per_block = 8 * kQGroupsPerWarp;                 // 8 warps
    int64_t blocks = (groups + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sms * 4;                           // 32 warps an SM
    int grid = (int)(blocks < cap ? blocks : cap);
    quant_group128_kernel<<<grid, 256, 0, st>>>(x, M, K, xq, xs);
    return cudaGetLastError();
}

// --------------------------------------------------- weight block quant --

// One CTA of 256 threads per 128x128 block; thread t handles rows t/8 + 32i
// (i = 0..3), 16 consecutive columns each (four float4 loads).
__global__ void __launch_bounds__(256) quant_weight_block128_kernel(const float* __restrict__ w,
                                                                    int64_t K, uint8_t* __restrict__ wq,
                                                                    float* __restrict__ ws) {
    __shared__ float red[8];
    const int kb = blockIdx.x, nb = blockIdx.y;
    const int KB = (int)(K / kBlock);
    const int t = threadIdx.x;
    const int col = (t & 7) * 16;
    float4 v[4][4];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = (int64_t)nb * kBlock + (t >> 3) + 32 * i;
        const float4* p = reinterpret_cast<const float4*>(w + row * K + (int64_t)kb * kBlock + col);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[i][j] = p[j];
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i][j].x), fabsf(v[i][j].y)),
                                     fmaxf(fabsf(v[i][j].z), fabsf(v[i][j].w))));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 448.0f);
    if (t == 0) ws[(int64_t)nb * KB + kb] = s;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = (int64_t)nb * kBlock + (t >> 3) + 32 * i;
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (amax == 0.0f) {
                out[j] = 0u;
            } else {
                out[j] = cvt_e4m3x2(__fdiv_rn(v[i][j].x, s), __fdiv_rn(v[i][j].y, s)) |
                         (cvt_e4m3x2(__fdiv_rn(v[i][j].z, s), __fdiv_rn(v[i][j].w, s)) << 16);
            }
        }
        *reinterpret_cast<uint4*>(wq + row * K + (int64_t)kb * kBlock + col) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

cudaError_t launch_quant_weight_block128(const float* w, int64_t N, int64_t K, uint8_t* wq, float* ws,
                                         cudaStream_t st) {
    dim3 grid((unsigned)(K / kBlock), (unsigned)(N / kBlock));
    quant_weight_block128_kernel<<<grid, 256, 0, st>>>(w, K, wq, ws);
    return cudaGetLastError();
}

// --------------------------------------------------------------- SwiGLU --

// h[m][128j + c] = bf16(silu(g) * u), g = gu[m][256j + c], u = gu[m][256j + 128 + c]
// (gu already bf16).  Two outputs per thread.
__global__ void __launch_bounds__(256) swiglu_interleaved_kernel(const uint16_t* __restrict__ gu, int64_t M,
                                                                 int64_t I, uint16_t* __restrict__ h) {
    const int64_t pairs = M * I / 2;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < pairs;
         p += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = (2 * p) / I, col = (2 * p) % I;
        const int64_t j = col / kBlock, c = col % kBlock;
        const uint32_t g = *reinterpret_cast<const uint32_t*>(gu + m * 2 * I + 2 * kBlock * j + c);
        const uint32_t u = *reinterpret_cast<const uint32_t*>(gu + m * 2 * I + 2 * kBlock * j + kBlock + c);
        const float h0 = silu_mul(bf16_lo(g), bf16_lo(u));
        const float h1 = silu_mul(bf16_hi(g), bf16_hi(u));
        *reinterpret_cast<uint32_t*>(h + m * I + col) = pack_bf16x2(h0, h1);
    }
}

cudaError_t launch_swiglu_interleaved(const uint16_t* gu, int64_t M, int64_t I, uint16_t* h,
                                      cudaStream_t st, int sms) {
    const int64_t pairs = M * I / 2;
    int64_t blocks = (pairs + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    swiglu_interleaved_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, st>>>(gu, M, I, h);
    return cudaGetLastError();
}

}  // namespace r9q
