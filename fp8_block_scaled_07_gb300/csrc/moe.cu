// moe.cu -- data movement around the grouped expert GEMM
// ("Behavior traces -- deepseek-ai/DeepSeek-V3", bullet "MoE trace": count
// the tokens per expert, take each expert's tokens in order, run the expert
// and add its output times the gate weight back into y).
//
//   route    stable counting sort of (token, slot) pairs by expert id; each
//            CTA owns a group of experts and reads the ids twice (16-byte
//            loads where they allow it): once to count, per warp, the pairs
//            below its group and those of each of its experts, once to
//            rank its experts' pairs in pair order (warp match groups, then
//            the warps' counts in order), so the result is deterministic
//            and needs no global atomics;
//   gather   packed row r <- quantised token row row_token[r] (+ scales);
//   quant_scatter  act_quant of each token row, written straight to its
//            topk packed rows: act_quant and gather in one pass over x;
//   combine  y[t] = sum_j w[t,j] * out[pair_row[t,j]] in fp32, one warp per
//            token, 16-byte loads.
#include "common.cuh"

namespace fp8bs {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteMaxOwn = 32;   // experts per CTA (E <= 1024 over at most 32 CTAs)

// CTA c owns experts [e0, e0 + ne).  Each warp takes a contiguous range of
// the pairs; one pass counts, per warp, the pairs with id < e0 and those of
// each owned expert; the CTA turns these into the owned experts' first
// packed rows (offsets) and each warp's first row per expert; a second pass
// ranks the owned pairs in pair order (match groups per 32 pairs, in order)
// and writes pair_row / row_token.  Integer counts only: deterministic, no
// global atomics.  VEC: a lane reads four consecutive ids with one 16-byte
// load (P % 4 == 0 and an aligned base); the second pass transposes each
// 128-pair step through shared memory so that it walks them in pair order.
template <bool VEC>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const int32_t* __restrict__ ids,
                                                              int64_t P, int32_t topk, int32_t E, int32_t epc,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ pair_row,
                                                              int32_t* __restrict__ row_token) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int kPer = VEC ? 4 : 1;      // ids per lane per step
    constexpr int kStep = 32 * kPer;       // pairs per warp per step
    constexpr int kU = 8;                  // steps whose loads are in flight together
    __shared__ int s_cnt[kRouteWarps][kRouteMaxOwn + 1];   // per warp and owned expert
    __shared__ int s_lt[kRouteWarps];
    __shared__ int s_tot[kRouteMaxOwn];
    __shared__ int s_ids[VEC ? kRouteWarps : 1][VEC ? kStep : 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e0 = blockIdx.x * epc;
    const int ne = min(epc, E - e0);
    for (int i = threadIdx.x; i < kRouteWarps * (kRouteMaxOwn + 1); i += kRouteThreads)
        (&s_cnt[0][0])[i] = 0;
    __syncthreads();
    const int64_t seg = ((P + kRouteWarps - 1) / kRouteWarps + kStep - 1) / kStep * kStep;
    const int64_t lo = min(P, seg * warp), hi = min(P, lo + seg);
    auto load = [&](int64_t i, int (&v)[kPer]) {   // -1: past the range
        if constexpr (VEC) {
            const int4 q = i < hi ? __ldg(reinterpret_cast<const int4*>(ids + i)) : make_int4(-1, -1, -1, -1);
            v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
            v[0] = i < hi ? __ldg(ids + i) : -1;
        }
    };
    // ---- pass 1: counts
    int lt = 0;
    for (int64_t c0 = lo; c0 < hi; c0 += kU * kStep) {
        int v[kU][kPer];
#pragma unroll
        for (int u = 0; u < kU; ++u) load(c0 + u * kStep + lane * kPer, v[u]);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t i = c0 + u * kStep + lane * kPer;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int id = v[u][j];
                if (i < hi) {
                    lt += id < e0 ? 1 : 0;
                    if (id >= e0 && id < e0 + ne) atomicAdd(&s_cnt[warp][id - e0], 1);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lt += __shfl_xor_sync(0xFFFFFFFFu, lt, o);
    if (lane == 0) s_lt[warp] = lt;
    __syncthreads();
    // per owned expert: the warps' counts become their exclusive prefix
    if (threadIdx.x < ne) {
        int run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            const int c = s_cnt[w][threadIdx.x];
            s_cnt[w][threadIdx.x] = run;
            run += c;
        }
        s_tot[threadIdx.x] = run;
    }
    __syncthreads();
    // first packed row of each owned expert; each warp's first row per expert
    if (warp == 0) {
        int below = 0;
        for (int w = 0; w < kRouteWarps; ++w) below += s_lt[w];
        const int tot = lane < ne ? s_tot[lane] : 0;
        int inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += n;
        }
        const int base = below + inc - tot;
        if (lane < ne) {
            offsets[e0 + lane] = base;
            s_tot[lane] = base;
        }
        if (lane == 0 && e0 + ne == E) offsets[E] = static_cast<int32_t>(P);
    }
    __syncthreads();
    if (lane < ne) s_cnt[warp][lane] += s_tot[lane];
    __syncwarp();
    // ---- pass 2: the owned pairs take their rows in pair order
    const unsigned below_me = (1u << lane) - 1u;
    auto place = [&](int64_t i, int id) {
        const bool own = i < hi && id >= e0 && id < e0 + ne;
        if (!__any_sync(0xFFFFFFFFu, own)) return;
        const unsigned m = __match_any_sync(0xFFFFFFFFu, own ? id : -1);
        int row = 0;
        if (own) {
            row = s_cnt[warp][id - e0] + __popc(m & below_me);
            pair_row[i] = row;
            row_token[row] = static_cast<int32_t>(i / topk);
        }
        __syncwarp();
        if (own && (m >> lane) == 1u) s_cnt[warp][id - e0] = row + 1;   // the group's last lane
        __syncwarp();
    };
    for (int64_t c0 = lo; c0 < hi; c0 += kU * kStep) {
        int v[kU][kPer];
#pragma unroll
        for (int u = 0; u < kU; ++u) load(c0 + u * kStep + lane * kPer, v[u]);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t s0 = c0 + u * kStep;
            if constexpr (VEC) {
                __syncwarp();   // the previous step's ids have been read
                *reinterpret_cast<int4*>(&s_ids[warp][lane * 4]) = make_int4(v[u][0], v[u][1], v[u][2], v[u][3]);
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j) place(s0 + j * 32 + lane, s_ids[warp][j * 32 + lane]);
            } else {
                place(s0 + lane, v[u][0]);
            }
        }
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
    // the two half-warps may run different numbers of blocks (an odd block
    // count), so each reduces over its own 16 lanes only
    const unsigned hmask = 0xFFFFu << (half * 16);
    for (int64_t blk = hw; blk < nblocks; blk += nhw) {
        const int64_t t = blk / KB, kb = blk - t * KB;
        float f[8];
        unpack_bf16x8(__ldcs(x + blk * 16 + sub), f);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, o));
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
    const bool vec = P % 4 == 0 && reinterpret_cast<uintptr_t>(ids) % 16 == 0;
    auto kernel = vec ? route_kernel<true> : route_kernel<false>;
    const int epc = (E + kRouteWarps - 1) / kRouteWarps;   // <= kRouteMaxOwn for E <= 1024
    const int grid = (E + epc - 1) / epc;
    kernel<<<grid, kRouteThreads, 0, static_cast<cudaStream_t>(stream)>>>(ids, P, topk, E, epc, offsets, pair_row,
                                                                           row_token);
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
