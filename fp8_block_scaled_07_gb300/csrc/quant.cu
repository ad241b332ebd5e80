// quant.cu -- bandwidth-bound kernels of the FP8 block-scaled linear:
//   act_quant        bf16 activations -> e4m3 + one fp32 scale per 128 block
//                    ("Data flow -- deepseek-ai/DeepSeek-V3", bullet "FP8
//                    quantization data flow"; source tour, "FP8 with
//                    per-block scales": clamp the block max, divide by 448)
//   weight_quant     bf16 weight -> e4m3 + 128x128 block scales
//   weight_dequant   e4m3 weight * block scale -> bf16 ("Behavior traces",
//                    bullet "fp8->bf16 trace")
//   silu_mul_quant   the expert body silu(h1)*h3 fused with act_quant
//
// Layout: every 128-element activation block is 256 contiguous bytes of
// bf16, so a tensor [M, K] is a flat sequence of M*K/128 blocks whose scales
// are stored in the same order.  A half-warp owns one block: each lane loads
// 16 bytes (8 values), the block max is a 4-step shuffle reduction inside
// the half-warp, and each lane writes 8 codes (8 bytes).
#include "common.cuh"
#include <cuda_fp16.h>

namespace fp8bs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // independent 16-byte loads in flight per lane
constexpr int kActUnroll = 8;   // act_quant: 8 loads in flight per lane (measured faster than 4)

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }


__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}


template <bool UE8M0>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint4* __restrict__ x,
                                                             uint2* __restrict__ y,
                                                             float* __restrict__ s,
                                                             int64_t nblocks) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int sub = lane & 15;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    for (int64_t b0 = warp * (2 * kActUnroll); b0 < nblocks; b0 += nwarps * (2 * kActUnroll)) {
        uint4 v[kActUnroll];
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t blk = b0 + 2 * u + half;
            v[u] = blk < nblocks ? ld_stream(x + blk * 16 + sub) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t blk = b0 + 2 * u + half;
            float f[8];
            unpack_bf16x8(v[u], f);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = half_warp_max(amax);
            if (blk < nblocks) {
                const float sc = block_scale(amax, UE8M0);
                __stcs(y + blk * 16 + sub, quant8<UE8M0>(f, sc));   // streamed out: evict first
                if (sub == 0) s[blk] = sc;
            }
        }
    }
}

// One CTA per 128x128 weight block.  Thread t handles the 8-column chunk
// (t % 16) of rows t/16 + 16*i, i < 8.
template <bool UE8M0>
__global__ void __launch_bounds__(kThreads) weight_quant_kernel(const uint16_t* __restrict__ w,
                                                                uint8_t* __restrict__ q,
                                                                float* __restrict__ s,
                                                                int64_t N, int64_t K,
                                                                int64_t KB) {
    griddep_launch_dependents();
    griddep_wait();
    __shared__ float red[kThreads / 32];
    const int64_t nb = blockIdx.y, kb = blockIdx.x;
    const int chunk = threadIdx.x & 15;
    const int r0 = threadIdx.x >> 4;
    const int64_t col = kb * kBlock + chunk * 8;
    const bool col_ok = col < K;   // K % 8 == 0: a chunk is all in or all out
    float f[8][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = nb * kBlock + r0 + 16 * i;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < N && col_ok) v = *reinterpret_cast<const uint4*>(w + row * K + col);
        unpack_bf16x8(v, f[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[i][j]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float sc = block_scale(amax, UE8M0);
    if (threadIdx.x == 0) s[nb * KB + kb] = sc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = nb * kBlock + r0 + 16 * i;
        if (row < N && col_ok)
            *reinterpret_cast<uint2*>(q + row * K + col) = quant8<UE8M0>(f[i], sc);
    }
}

// Thread handles 16 consecutive codes of one row (16-byte load, 32-byte
// store), kDequantUnroll of them in flight; the bf16 output is written with
// streaming (evict-first) stores, since nothing here reads it back.
constexpr int kDequantUnroll = 8;
__global__ void __launch_bounds__(kThreads) weight_dequant_kernel(const uint4* __restrict__ w,
                                                                  const float* __restrict__ s,
                                                                  uint4* __restrict__ y,
                                                                  int64_t M, int64_t N,
                                                                  int64_t NB) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t chunks_per_row = N / 16;
    const int64_t total = M * chunks_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t c = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; c < total; c += stride * kDequantUnroll) {
        uint4 v[kDequantUnroll];
#pragma unroll
        for (int u = 0; u < kDequantUnroll; ++u) {
            const int64_t cc = c + u * stride;
            v[u] = cc < total ? ld_stream(w + cc) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kDequantUnroll; ++u) {
            const int64_t cc = c + u * stride;
            if (cc >= total) break;
            const int64_t row = cc / chunks_per_row;
            const int64_t col = (cc - row * chunks_per_row) * 16;
            const float sc = __ldg(s + (row / kBlock) * NB + col / kBlock);
            const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t out[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(words[i] & 0xFFFFu));
                const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(words[i] >> 16));
                const __nv_bfloat162 b0 = __floats2bfloat162_rn(lo.x * sc, lo.y * sc);
                const __nv_bfloat162 b1 = __floats2bfloat162_rn(hi.x * sc, hi.y * sc);
                out[2 * i] = *reinterpret_cast<const uint32_t*>(&b0);
                out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&b1);
            }
            uint4* dst = y + cc * 2;
            __stcs(dst, make_uint4(out[0], out[1], out[2], out[3]));
            __stcs(dst + 1, make_uint4(out[4], out[5], out[6], out[7]));
        }
    }
}

// silu(h1) * h3 in bf16 steps, then act_quant of the result, one half-warp
// per 128-block of a row of g [R, I].
template <bool UE8M0>
__global__ void __launch_bounds__(kThreads) silu_mul_quant_kernel(
    const uint16_t* __restrict__ h1, const uint16_t* __restrict__ h3, int64_t ld_h, int64_t R,
    int64_t I, uint2* __restrict__ y, float* __restrict__ s, uint4* __restrict__ g_out) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int sub = lane & 15;
    const int64_t IB = I / kBlock;
    const int64_t nblocks = R * IB;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    constexpr int U = 2;
    // the next iteration's loads are issued before this one's arithmetic
    auto load = [&](int64_t b0, uint4 (&v1)[U], uint4 (&v3)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t blk = b0 + 2 * u + half;
            if (blk < nblocks) {
                const int64_t r = blk / IB, ib = blk - r * IB;
                const int64_t off = r * ld_h + ib * kBlock + sub * 8;
                v1[u] = ld_stream(reinterpret_cast<const uint4*>(h1 + off));
                v3[u] = ld_stream(reinterpret_cast<const uint4*>(h3 + off));
            } else {
                v1[u] = make_uint4(0, 0, 0, 0);
                v3[u] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    uint4 n1[U], n3[U];
    load(warp * (2 * U), n1, n3);
    for (int64_t b0 = warp * (2 * U); b0 < nblocks; b0 += nwarps * (2 * U)) {
        uint4 v1[U], v3[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            v1[u] = n1[u];
            v3[u] = n3[u];
        }
        load(b0 + nwarps * (2 * U), n1, n3);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t blk = b0 + 2 * u + half;
            float a[8], b[8], gv[8];
            unpack_bf16x8(v1[u], a);
            unpack_bf16x8(v3[u], b);
            uint32_t gbits[4];
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                gbits[i / 2] = silu_mul_bf16x2(a[i], a[i + 1], b[i], b[i + 1]);
                gv[i] = __uint_as_float(gbits[i / 2] << 16);
                gv[i + 1] = __uint_as_float(gbits[i / 2] & 0xFFFF0000u);
                amax = fmaxf(amax, fmaxf(fabsf(gv[i]), fabsf(gv[i + 1])));
            }
            amax = half_warp_max(amax);
            if (blk < nblocks) {
                const float sc = block_scale(amax, UE8M0);
                y[blk * 16 + sub] = quant8<UE8M0>(gv, sc);
                if (sub == 0) s[blk] = sc;
                if (g_out != nullptr) g_out[blk * 16 + sub] = make_uint4(gbits[0], gbits[1], gbits[2], gbits[3]);
            }
        }
    }
}

int grid_for(int64_t work_items, int64_t items_per_cta) {
    int64_t g = (work_items + items_per_cta - 1) / items_per_cta;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8_status fp8_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K,
                                    int scale_fmt, void* stream) {
    if (M < 0 || K <= 0 || K % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!x || !y || !s || !aligned16(x) || !aligned16(y)) return FP8_ERR_INVALID_ARG;
    const int64_t nblocks = M * (K / kBlock);
    const int grid = grid_for(nblocks, (kThreads / 32) * 2 * kActUnroll);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (scale_fmt == FP8_SCALE_UE8M0)
        launch_pdl(act_quant_kernel<true>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint4*>(x), static_cast<uint2*>(y), s, nblocks);
    else
        launch_pdl(act_quant_kernel<false>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint4*>(x), static_cast<uint2*>(y), s, nblocks);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_weight_quant(const void* w, void* q, float* s, int64_t N, int64_t K,
                                       int scale_fmt, void* stream) {
    if (N < 0 || K <= 0 || K % 16 != 0) return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (N == 0) return FP8_OK;
    if (!w || !q || !s || !aligned16(w) || !aligned16(q)) return FP8_ERR_INVALID_ARG;
    const int64_t NB = (N + kBlock - 1) / kBlock, KB = (K + kBlock - 1) / kBlock;
    if (NB > 65535) return FP8_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(KB), static_cast<unsigned>(NB));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (scale_fmt == FP8_SCALE_UE8M0)
        launch_pdl(weight_quant_kernel<true>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t*>(w), static_cast<uint8_t*>(q), s, N, K, KB);
    else
        launch_pdl(weight_quant_kernel<false>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t*>(w), static_cast<uint8_t*>(q), s, N, K, KB);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_weight_dequant(const void* w, const float* s, void* y, int64_t M,
                                         int64_t N, void* stream) {
    if (M < 0 || N <= 0 || N % 16 != 0) return FP8_ERR_INVALID_ARG;
    if (M == 0) return FP8_OK;
    if (!w || !s || !y || !aligned16(w) || !aligned16(y)) return FP8_ERR_INVALID_ARG;
    const int64_t NB = (N + kBlock - 1) / kBlock;
    const int64_t chunks = M * (N / 16);
    const int grid = grid_for(chunks, static_cast<int64_t>(kThreads) * kDequantUnroll);
    weight_dequant_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(w), s, static_cast<uint4*>(y), M, N, NB);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_silu_mul_quant(const void* h1, const void* h3, int64_t ld_h, int64_t R,
                                         int64_t I, void* y, float* s, void* g_bf16,
                                         int scale_fmt, void* stream) {
    if (R < 0 || I <= 0 || I % kBlock != 0 || ld_h < I || ld_h % 8 != 0)
        return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (R == 0) return FP8_OK;
    if (!h1 || !h3 || !y || !s || !aligned16(h1) || !aligned16(h3) || !aligned16(y) ||
        (g_bf16 && !aligned16(g_bf16)))
        return FP8_ERR_INVALID_ARG;
    const int64_t nblocks = R * (I / kBlock);
    const int grid = grid_for(nblocks, (kThreads / 32) * 4);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (scale_fmt == FP8_SCALE_UE8M0)
        launch_pdl(silu_mul_quant_kernel<true>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t*>(h1), static_cast<const uint16_t*>(h3), ld_h, R, I,
            static_cast<uint2*>(y), s, static_cast<uint4*>(g_bf16));
    else
        launch_pdl(silu_mul_quant_kernel<false>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t*>(h1), static_cast<const uint16_t*>(h3), ld_h, R, I,
            static_cast<uint2*>(y), s, static_cast<uint4*>(g_bf16));
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
