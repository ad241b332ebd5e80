// moe.cu -- data movement around the grouped expert GEMM
// ("Behavior traces -- deepseek-ai/DeepSeek-V3", bullet "MoE trace": count
// the tokens per expert, take each expert's tokens in order, run the expert
// and add its output times the gate weight back into y).
//
//   route    stable counting sort of (token, slot) pairs by expert id; CTA e
//            counts, each warp over a contiguous range read 32 pairs at a
//            time, the pairs with id < e (its first packed row) and those
//            with id == e, and ranks the latter in pair order (warp ballots,
//            then the warps' counts in order), so the result is
//            deterministic and needs no atomics;
//   gather   packed row r <- quantised token row row_token[r] (+ scales);
//   quant_scatter  act_quant of each token row, written straight to its
//            topk packed rows: act_quant and gather in one pass over x;
//   combine  y[t] = sum_j w[t,j] * out[pair_row[t,j]] in fp32, one warp per
//            token, 16-byte loads.
#include "common.cuh"

namespace fp8bs {
namespace {

constexpr int kRouteThreads = 256;

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const int32_t* __restrict__ ids,
                                                              int64_t P, int32_t topk, int32_t E,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ pair_row,
                                                              int32_t* __restrict__ row_token) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int kWarps = kRouteThreads / 32;
    __shared__ int s_lt[kWarps];
    __shared__ int s_eq[kWarps];
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp w owns the contiguous pairs [lo, hi) (a multiple of 32 long),
    // read 32 at a time: one pass counts the pairs with id < e (expert e's
    // first packed row) and those with id == e
    const int64_t seg = ((P + kWarps - 1) / kWarps + 31) / 32 * 32;
    const int64_t lo = min(P, seg * warp), hi = min(P, lo + seg);
    int lt = 0, eq = 0;
    // (unrolled: eight loads in flight per lane, not one L2 round trip per step)
#pragma unroll 8
    for (int64_t i0 = lo; i0 < hi; i0 += 32) {
        const int64_t i = i0 + lane;
        const int v = i < hi ? __ldg(ids + i) : -1;
        lt += (i < hi && v < e) ? 1 : 0;
        eq += __popc(__ballot_sync(0xFFFFFFFFu, v == e));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lt += __shfl_xor_sync(0xFFFFFFFFu, lt, o);
    if (lane == 0) {
        s_lt[warp] = lt;
        s_eq[warp] = eq;
    }
    __syncthreads();
    int base = 0, before = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        base += s_lt[w];
        if (w < warp) before += s_eq[w];
    }
    if (threadIdx.x == 0) {
        offsets[e] = base;
        if (e == E - 1) offsets[E] = static_cast<int32_t>(P);
    }
    // the pairs with id == e take packed rows base + rank, in pair order
    int r = base + before;
#pragma unroll 8
    for (int64_t i0 = lo; i0 < hi; i0 += 32) {
        const int64_t i = i0 + lane;
        const bool hit = i < hi && __ldg(ids + i) == e;
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, hit);
        if (hit) {
            const int row = r + __popc(ball & ((1u << lane) - 1u));
            pair_row[i] = row;
            row_token[row] = static_cast<int32_t>(i / topk);
        }
        r += __popc(ball);
    }
}

// One warp per packed row: K bytes of codes + K/128 scales.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ xq,
                                                    const float* __restrict__ xs,
                                                    const int32_t* __restrict__ row_token,
                                                    int64_t R, int64_t K, uint4* __restrict__ aq,
                                                    float* __restrict__ as) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t chunks = K / 16, KB = K / kBlock;
    for (int64_t r = warp; r < R; r += nwarps) {
        const int64_t t = __ldg(row_token + r);
        const uint4* src = xq + t * chunks;
        uint4* dst = aq + r * chunks;
        for (int64_t c = lane; c < chunks; c += 32) dst[c] = __ldcs(src + c);
        for (int64_t c = lane; c < KB; c += 32) as[r * KB + c] = __ldg(xs + t * KB + c);
    }
}

// act_quant of token rows scattered to their packed rows: a half-warp per
// 128-block of a token row (as act_quant: 16 lanes x 8 values, the block max
// by shuffles, the library's quantisation routine), the codes and the scale
// written to each of the token's topk packed rows pair_row[t, j].  x is read
// once; the result equals fp8_act_quant followed by fp8_moe_gather.
template <bool UE8M0>
__global__ void __launch_bounds__(256) quant_scatter_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ pair_row, int64_t T,
                                                           int32_t topk, int64_t K, uint2* __restrict__ aq,
                                                           float* __restrict__ as) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    const int64_t KB = K / kBlock, nblocks = T * KB;
    const int64_t hw = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 2 + half;
    const int64_t nhw = ((static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) * 2;
    for (int64_t blk = hw; blk < nblocks; blk += nhw) {
        const int64_t t = blk / KB, kb = blk - t * KB;
        float f[8];
        unpack_bf16x8(__ldcs(x + blk * 16 + sub), f);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float sc = block_scale(amax, UE8M0);
        const uint2 q = quant8<UE8M0>(f, sc);
        for (int j = 0; j < topk; ++j) {
            const int64_t r = __ldg(pair_row + t * topk + j);
            aq[(r * KB + kb) * 16 + sub] = q;
            if (sub == 0) as[r * KB + kb] = sc;
        }
    }
}

// One warp per token; lane handles 8 consecutive columns per step.  TK > 0
// is the topk known at compile time: the token's rows and weights are read
// once and its TK row loads of a step are all in flight together (the same
// fp32 sums, in the same slot order, as the generic loop).
template <int TK>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ out,
                                                     const float* __restrict__ w,
                                                     const int32_t* __restrict__ pair_row,
                                                     int64_t T, int32_t topk, int64_t D,
                                                     uint4* __restrict__ y_bf16,
                                                     float4* __restrict__ y_fp32) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t chunks = D / 8;
    auto add = [](float (&acc)[8], float wj, const uint4& v) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(wj, __uint_as_float(u[i] << 16), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj, __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
        }
    };
    for (int64_t t = warp; t < T; t += nwarps) {
        int64_t rows[TK > 0 ? TK : 1];
        float wts[TK > 0 ? TK : 1];
        if constexpr (TK > 0) {
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                rows[j] = __ldg(pair_row + t * TK + j);
                wts[j] = __ldg(w + t * TK + j);
            }
        }
        for (int64_t c = lane; c < chunks; c += 32) {
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if constexpr (TK > 0) {
                uint4 v[TK];
#pragma unroll
                for (int j = 0; j < TK; ++j) v[j] = __ldcs(out + rows[j] * chunks + c);
#pragma unroll
                for (int j = 0; j < TK; ++j) add(acc, wts[j], v[j]);
            } else {
                for (int j = 0; j < topk; ++j) {
                    const int64_t r = __ldg(pair_row + t * topk + j);
                    add(acc, __ldg(w + t * topk + j), __ldcs(out + r * chunks + c));
                }
            }
            if (y_bf16) {
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
                    o[i] = *reinterpret_cast<uint32_t*>(&b);
                }
                y_bf16[t * chunks + c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            if (y_fp32) {
                y_fp32[(t * chunks + c) * 2] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                y_fp32[(t * chunks + c) * 2 + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        }
    }
}

int warps_grid(int64_t warps_needed) {
    int64_t g = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8_status fp8_moe_route(const int32_t* ids, int64_t T, int32_t topk, int32_t E,
                                    int32_t* offsets, int32_t* pair_row, int32_t* row_token,
                                    void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || E > 1024) return FP8_ERR_INVALID_ARG;
    if (!offsets) return FP8_ERR_INVALID_ARG;
    const int64_t P = T * topk;
    if (P > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    if (P > 0 && (!ids || !pair_row || !row_token)) return FP8_ERR_INVALID_ARG;
    route_kernel<<<E, kRouteThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        ids, P, topk, E, offsets, pair_row, row_token);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_moe_gather(const void* xq, const float* xs, const int32_t* row_token,
                                     int64_t R, int64_t K, void* aq, float* as, void* stream) {
    if (R < 0 || K <= 0 || K % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (R == 0) return FP8_OK;
    if (!xq || !xs || !row_token || !aq || !as || !aligned16(xq) || !aligned16(aq))
        return FP8_ERR_INVALID_ARG;
    gather_kernel<<<warps_grid(R), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(xq), xs, row_token, R, K, static_cast<uint4*>(aq), as);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_moe_quant_scatter(const void* x, const int32_t* pair_row, int64_t T, int32_t topk,
                                          int64_t K, void* aq, float* as, int scale_fmt, void* stream) {
    if (T < 0 || topk <= 0 || K <= 0 || K % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (T == 0) return FP8_OK;
    if (!x || !pair_row || !aq || !as || !aligned16(x) || !aligned16(aq)) return FP8_ERR_INVALID_ARG;
    const int64_t halfwarps = T * (K / kBlock);
    const int grid = warps_grid((halfwarps + 1) / 2);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (scale_fmt == FP8_SCALE_UE8M0)
        launch_pdl(quant_scatter_kernel<true>, dim3(grid), dim3(256), 0, st, static_cast<const uint4*>(x), pair_row,
                   T, topk, K, static_cast<uint2*>(aq), as);
    else
        launch_pdl(quant_scatter_kernel<false>, dim3(grid), dim3(256), 0, st, static_cast<const uint4*>(x), pair_row,
                   T, topk, K, static_cast<uint2*>(aq), as);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_moe_combine(const void* out, const float* w, const int32_t* pair_row,
                                      int64_t T, int32_t topk, int64_t D, void* y_bf16,
                                      float* y_fp32, void* stream) {
    if (T < 0 || topk <= 0 || D <= 0 || D % 8 != 0) return FP8_ERR_INVALID_ARG;
    if (T == 0) return FP8_OK;
    if (!out || !w || !pair_row || (!y_bf16 && !y_fp32) || !aligned16(out) ||
        (y_bf16 && !aligned16(y_bf16)) || (y_fp32 && !aligned16(y_fp32)))
        return FP8_ERR_INVALID_ARG;
    auto kernel = topk == 8 ? combine_kernel<8> : combine_kernel<0>;   // (the V3 routing: top-8)
    kernel<<<warps_grid(T), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(out), w, pair_row, T, topk, D, static_cast<uint4*>(y_bf16),
        reinterpret_cast<float4*>(y_fp32));
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
