// decode.cu -- the FP8 block-scaled linear at decode batches (M <= 64 tokens).
//
// What it computes ("Data flow -- deepseek-ai/DeepSeek-V3", bullet "FP8
// quantization data flow"; source tour "DeepSeek-V3", paragraph "FP8 with
// per-block scales"):
//   C[m, n] = sum_kb a_s[m, kb] * b_s[n/128, kb] * sum_{k in kb} a[m,k] w[n,k]
// with e4m3 operands, fp32 scales and fp32 accumulation -- fp8_gemm for
// M <= 64 -- and, fused, the act_quant of the bf16 activations that feeds it
// (fp8_linear: codes and scales bit-identical to fp8_act_quant's).
//
// At these batches the weight bytes are the work: the kernel is a weight
// stream, and the design is about keeping HBM busy from the first byte of a
// launch to the last.
//   * Swapped operands: each MMA has the 128 weight rows of one output tile
//     on its M side and the BN in {16, 32, 64} tokens on its N side.
//   * Each output tile gets a thread-block cluster of c CTAs (c <= 16) that
//     split its K range; their fp32 partials meet on chip -- each CTA pushes
//     every row of its partial into the shared memory of the CTA owning that
//     row (st.async, counted as transaction bytes on the owner's barrier) --
//     and the owner sums them in rank order (deterministic).
//   * One 128-K slab per pipeline stage: three stages for 16-token tiles (3
//     CTAs per SM), four for 32 (2 per SM), four or three for 64 (1 or 2 per
//     SM, by the layer's tile count); a launch takes about three quarters of
//     the CTA slots: with programmatic dependent launch most of the next
//     launch's CTAs are resident and set up while this one runs, and they
//     pass griddepcontrol.wait together.
//   * Four "activation" warps feed the token side of each slab: they load
//     their values from global memory one slab ahead, quantise them (fused;
//     the library's act_quant routine) or take the e4m3 codes as they are,
//     write the codes into the stage in the layout the MMA reads (128-byte
//     swizzle) and the per-token scale products b_s * a_s into a small ring
//     read by the epilogue.
//   * Four epilogue warps (one per TMEM lane quarter) promote each finished
//     slab: acc += D * (b_s * a_s), the per-block scales applied in fp32
//     registers, so the tensor core never accumulates across scale blocks.
// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-3 and 8-9
// activation warps, 4-7 epilogue.  Every wait is bounded (common.cuh).
#include "common.cuh"

#include <algorithm>

namespace fp8bs {

__device__ int g_decode_status;   // FP8_OK or FP8_ERR_TIMEOUT, read by fp8_device_status

#ifdef FP8BS_TRACE_ENABLED
// per-CTA timeline (global timer, ns) for profiling builds only
__device__ unsigned long long g_dtrace[4][1024][8];
#define DEC_TRACE(slot)                                                      \
    do {                                                                     \
        if (blockIdx.x < 1024) {                                             \
            unsigned long long t_;                                           \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));          \
            g_dtrace[p.trace_slot & 3][blockIdx.x][slot] = t_;               \
        }                                                                    \
    } while (0)
#else
#define DEC_TRACE(slot) \
    do {                \
    } while (0)
#endif

namespace {

constexpr int kDecThreads = 320;
constexpr int kDecMaxCluster = 16;
#ifndef FP8BS_DEC_EVICT_FIRST
#define FP8BS_DEC_EVICT_FIRST 1   // weight loads marked evict-first in L2 (each byte is read once)
#endif

// Pipeline stages (one 128-K slab each).  16-token tiles: 3 (three CTAs per
// SM).  32-token tiles: 4 (still two per SM; decode step at M = 32 49.9 ->
// 48.8 us against 3).  64-token tiles: 4, one CTA per SM, when the layer's
// tiles fit one wave of that, else 3 (two per SM): at M = 64 wo took 37.4
// against 46.5 us and wq_a 12.8 against 15.8, but wq_b's 192 tiles 20.5
// against 18.5 us in two waves.
constexpr int kDecStages = 3;
constexpr int kS32 = 4;
constexpr int kS64Deep = 4;
// Percent of the device's CTA slots one launch may take.  16-token tiles
// (three CTAs per SM): three quarters -- enough bytes in flight for the
// long weight streams, and room left for most of the next launch's CTAs to
// be resident and waiting when this one ends (measured on GB300, decode
// step at M = 16 / the wo layer alone, back to back: 50% 41.4 / 28.2 us,
// 60% 41.4 / 28.2, 66% 42.7 / 24.6, 75% 40.0 / 22.7, 100% 50.4 / 29.7).
// 32- and 64-token tiles (two per SM): three quarters as well.  With all
// slots, wo's clusters of 5 could not all be placed while the previous
// layer's CTAs were still resident, and the last ones ran as a second wave
// (decode step at M = 32 / 48 / 64: all 56.5 / 82.2 / 86.9 us, 75% 49.8 /
// 75.7 / 78.8, 70% 52.2 / 86.8 / 91.1, half 85.4 at M = 64).
#ifndef FP8BS_DEC_FILL16
#define FP8BS_DEC_FILL16 75
#endif
#ifndef FP8BS_DEC_FILL
#define FP8BS_DEC_FILL 75
#endif

template <int BN, int S>
struct Dec {
    static constexpr int kStages = S;
    static constexpr int kWBytes = 128 * kBlock;           // weight slab: 128 rows x 128 e4m3
    static constexpr int kXBytes = BN * kBlock;            // token codes of a slab
    static constexpr int kRing = kStages + 2;              // scale-product slots (see the act role)
    // split-K receive buffer [c][ceil(128 / c)][BN] fp32: c * ceil(128 / c) < 128 + c
    static constexpr int kRecvFloats = (128 + kDecMaxCluster) * BN;
    static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes =
        1024 + kStages * (kWBytes + kXBytes) + kRecvFloats * 4 + kRing * BN * 4 + kBarBytes;
    // CTAs per SM the footprint allows (228 KB per SM, 1 KB reserved per CTA; at most 3)
    static constexpr int kFit = (228 * 1024) / (kSmemBytes + 1024);
    static constexpr int kMinBlocks = kFit > 3 ? 3 : (kFit < 1 ? 1 : kFit);
    static constexpr int TPR = kBlock / BN;   // activation threads per token row: 8, 4, 2
    static constexpr int VPT = BN;            // values of a row per thread and slab: 16, 32, 64
    static_assert(128 * VPT == BN * kBlock, "128 activation threads cover a slab");
};

struct DecParams {
    const uint8_t* xq;          // e4m3 codes [M, K] (fp8_gemm)
    const uint16_t* x;          // bf16 [M, K] (fp8_linear: quantised here)
    const float* a_s;           // [M, KB] (fp8_gemm)
    const float* b_s;           // [NB, KB]
    __nv_bfloat16* c_bf16;      // [M, N] or null
    float* c_fp32;              // [M, N] or null
    long long K;                // row stride of x / xq (elements)
    int M, N, KB;
    int c;                      // CTAs per output tile (the cluster)
    int ue8m0;                  // fused: activation scale format
    int debug_skip;             // test hook: the MMA issuer withholds slab 0's hand-off to the epilogue
    int trace_slot;             // profiling builds
};

__device__ __forceinline__ void dec_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(&g_decode_status, static_cast<int>(FP8_ERR_TIMEOUT));
}

__device__ __forceinline__ bool dec_warp_all(bool ok) { return __all_sync(0xFFFFFFFFu, ok) != 0; }

// First row owned by cluster rank o when c CTAs share 128 rows: ceil(128 o / c).
__device__ __forceinline__ int own_lo(int o, int c) { return (o * 128 + c - 1) / c; }

template <int BN, bool FUSED, int SS>
__global__ void __launch_bounds__(kDecThreads, (Dec<BN, SS>::kMinBlocks))
    decode_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const DecParams p) {
    using D = Dec<BN, SS>;
    constexpr int S = D::kStages, R = D::kRing;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                        // S x 16 KB
    uint8_t* sX = smem + S * D::kWBytes;                       // S x BN x 128 B
    float* s_recv = reinterpret_cast<float*>(sX + S * D::kXBytes);
    float* s_ring = s_recv + D::kRecvFloats;                   // R x BN scale products
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_ring + R * BN);
    uint64_t* full = bars;                 // S: the slab's operands are in the stage
    uint64_t* empty = bars + S;            // S: the slab's MMAs are done with the stage
    uint64_t* tfull = bars + 2 * S;        // 2: TMEM slab buffer written
    uint64_t* tempty = tfull + 2;          // 2: TMEM slab buffer promoted (four epilogue warps)
    uint64_t* rfull = tempty + 2;          // R: scale products of the ring slot written
    uint64_t* rempty = rfull + R;          // R: the epilogue is done with the ring slot
    uint64_t* red_bar = rempty + R;        // split-K: every partial row pushed to this CTA
    uint64_t* mma_done = red_bar + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    static_assert((2 * S + 4 + 2 * R + 2) * 8 + 8 <= D::kBarBytes, "barrier block");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = p.c;
    const int tile = static_cast<int>(blockIdx.x) / c, part = static_cast<int>(blockIdx.x) - tile * c;
    const int k0 = part * p.KB / c, k1 = (part + 1) * p.KB / c;   // this CTA's 128-K slabs
    const int nslab = k1 - k0;
    const int n0 = tile * 128;
    if (threadIdx.x == 0) DEC_TRACE(0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            // the producer's bytes (weights; and the token codes unless they
            // are quantised here, by the four activation warps)
            mbar_init(&full[i], FUSED ? 1 + 4 : 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        for (int i = 0; i < R; ++i) {
            mbar_init(&rfull[i], 4);
            mbar_init(&rempty[i], 4);
        }
        mbar_init(red_bar, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_w);
        if (!FUSED) tma_prefetch_desc(&tm_x);
        // (no global data is touched before griddepcontrol.wait: a prefetch
        // racing with an earlier grid's writes of the same lines can leave
        // stale data in GB300's L2)
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, D::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (c > 1) cluster_sync_all();   // every CTA's barriers exist before remote arrivals
    // dependents may launch once this CTA holds its tensor memory
    if (threadIdx.x == 32 * 4) griddep_launch_dependents();
    if (threadIdx.x == 0) DEC_TRACE(1);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = FP8BS_DEC_EVICT_FIRST ? l2_policy_evict_first() : l2_policy_evict_normal();
            int issued = 0;
            for (int i = 0; i < nslab; ++i) {
                const int st = i % S;
                if (!mbar_wait(&empty[st], ((i / S) & 1) ^ 1, abort_flag)) {
                    dec_abort(abort_flag);
                    break;
                }
                if (i == 0) {
                    griddep_wait();   // the weights may be written by an earlier grid
                    DEC_TRACE(2);
                }
                mbar_arrive_expect_tx(&full[st], FUSED ? D::kWBytes : D::kWBytes + D::kXBytes);
                tma_load_2d_hint(sW + st * D::kWBytes, &tm_w, &full[st], (k0 + i) * kBlock, n0, pol);
                // e4m3 token codes [BN rows x 128]: rows past M read as zero
                if (!FUSED) tma_load_2d(sX + st * D::kXBytes, &tm_x, &full[st], (k0 + i) * kBlock, 0);
                ++issued;
            }
            // every load issued must land before the CTA may exit
            const volatile int never = 0;
            for (int st = 0; st < S && st < issued; ++st) {
                const int uses = issued / S + (st < issued % S ? 1 : 0);
                if (!mbar_wait(&full[st], (uses - 1) & 1, &never)) dec_abort(abort_flag);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(128, BN);
            for (int i = 0; i < nslab; ++i) {
                const int st = i % S, buf = i & 1;
                const bool ok = mbar_wait(&tempty[buf], ((i >> 1) & 1) ^ 1, abort_flag) &&
                                mbar_wait(&full[st], (i / S) & 1, abort_flag);
                if (!ok) {
                    dec_abort(abort_flag);
                    break;
                }
                tc_fence_after();
                if (i == 0) DEC_TRACE(3);
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
                const uint64_t da = smem_desc_sw128(smem_u32(sW + st * D::kWBytes));
                const uint64_t db = smem_desc_sw128(smem_u32(sX + st * D::kXBytes));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // 4 x K=32 = one slab; +32 bytes per step
                    mma_e4m3(d, da + 2 * kk, db + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                mma_commit(&empty[st]);
                if (!(p.debug_skip && i == 0)) mma_commit(&tfull[buf]);
            }
            mma_commit(mma_done);
            const volatile int never = 0;
            if (!mbar_wait(mma_done, 0, &never)) dec_abort(abort_flag);
        }
    } else if (warp < 4 || warp >= 8) {
        // ---------------------------------------------------------- activation warps
        const int t = (warp < 4 ? warp - 2 : warp - 6) * 32 + lane;   // 0..127
        const float* bs_row = p.b_s + static_cast<int64_t>(n0 / 128) * p.KB;
        griddep_wait();   // the activations come from an earlier grid
        if constexpr (FUSED) {
            // thread (r, sub): values [VPT sub, VPT (sub + 1)) of token row r,
            // loaded one slab ahead, quantised with the row's block max
            constexpr int TPR = D::TPR, VPT = D::VPT;
            constexpr int NC = VPT / 16;                   // 16-byte code chunks per thread and slab
            constexpr int NL = VPT / 8;                    // 16-byte bf16 loads per thread and slab
            const int r = t / TPR, sub = t - r * TPR;
            const bool valid = r < p.M;
            uint4 cur[NL], nxt[NL];
            float cur_bs = 0.0f, nxt_bs = 0.0f;
            auto load = [&](int kb, uint4 (&v)[NL], float& bs) {
                if (valid) {
                    const uint4* src = reinterpret_cast<const uint4*>(p.x + r * p.K + kb * kBlock + sub * VPT);
#pragma unroll
                    for (int j = 0; j < NL; ++j) v[j] = __ldg(src + j);
                } else {
#pragma unroll
                    for (int j = 0; j < NL; ++j) v[j] = make_uint4(0, 0, 0, 0);
                }
                if (sub == 0) bs = __ldg(bs_row + kb);
            };
            if (nslab > 0) load(k0, cur, cur_bs);
            for (int i = 0; i < nslab; ++i) {
                const int st = i % S;
                if (i + 1 < nslab) load(k0 + i + 1, nxt, nxt_bs);   // in flight while this slab is worked
                uint4 codes[NC];
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < NL; ++j) {
                    float nx[8];
                    unpack_bf16x8_neg(cur[j], nx);
                    amax = fmaxf(amax, max_abs8(nx));
                }
#pragma unroll
                for (int o = 1; o < TPR; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                const float sc = block_scale(amax, p.ue8m0 != 0);
                const float rc = __frcp_rn(sc);
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    float nx0[8], nx1[8];
                    unpack_bf16x8_neg(cur[2 * j], nx0);
                    unpack_bf16x8_neg(cur[2 * j + 1], nx1);
                    const uint2 q0 = p.ue8m0 ? quant8n<true>(nx0, sc, rc) : quant8n<false>(nx0, sc, rc);
                    const uint2 q1 = p.ue8m0 ? quant8n<true>(nx1, sc, rc) : quant8n<false>(nx1, sc, rc);
                    codes[j] = valid ? make_uint4(q0.x, q0.y, q1.x, q1.y) : make_uint4(0, 0, 0, 0);
                }
                // the stage is free once the MMAs of slab i - S are done
                if (!dec_warp_all(mbar_wait(&empty[st], ((i / S) & 1) ^ 1, abort_flag))) {
                    dec_abort(abort_flag);
                    break;
                }
                uint8_t* row = sX + st * D::kXBytes + r * 128;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    const int chunk = sub * NC + j;
                    *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) * 16)) = codes[j];
                }
                if (sub == 0) s_ring[(i % R) * BN + r] = valid ? cur_bs * sc : 0.0f;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&full[st]);
                    mbar_arrive(&rfull[i % R]);
                }
                if (i == 0 && t == 0) DEC_TRACE(4);
                if (i + 1 < nslab) {
#pragma unroll
                    for (int j = 0; j < NL; ++j) cur[j] = nxt[j];
                    cur_bs = nxt_bs;
                }
            }
        } else {
            // the codes come by TMA with the weights; thread t < BN makes
            // token t's scale product b_s * a_s of each slab
            const bool valid = t < p.M && t < BN;
            const float* as_row = p.a_s + static_cast<int64_t>(valid ? t : 0) * p.KB;
            float cur_p = 0.0f;
            if (valid && nslab > 0) cur_p = __ldg(bs_row + k0) * __ldg(as_row + k0);
            for (int i = 0; i < nslab; ++i) {
                float nxt_p = 0.0f;
                if (valid && i + 1 < nslab) nxt_p = __ldg(bs_row + k0 + i + 1) * __ldg(as_row + k0 + i + 1);
                // ring slot i % R was last read for slab i - R; the epilogue
                // hands it back itself (the stage barriers would not do: the
                // MMAs do not wait for these warps, so a stage can complete
                // two phases while they lag one behind)
                if (!dec_warp_all(mbar_wait(&rempty[i % R], ((i / R) & 1) ^ 1, abort_flag))) {
                    dec_abort(abort_flag);
                    break;
                }
                if (t < BN) s_ring[(i % R) * BN + t] = cur_p;
                __syncwarp();
                if (lane == 0) mbar_arrive(&rfull[i % R]);
                if (i == 0 && t == 0) DEC_TRACE(4);
                cur_p = nxt_p;
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue (warps 4-7)
        const int q = warp & 3;                       // TMEM lane quarter
        const int e = q * 32 + lane;                  // weight row of the tile = output column n0 + e
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        griddep_wait();   // the output may still be read by an earlier grid
        float acc[BN];
#pragma unroll
        for (int j = 0; j < BN; ++j) acc[j] = 0.0f;
        bool ok = true;
        for (int i = 0; i < nslab; ++i) {
            const int buf = i & 1;
            // every lane waits on its own; the warp votes after the hand-back
            const bool got = mbar_wait(&tfull[buf], (i >> 1) & 1, abort_flag) &&
                             mbar_wait(&rfull[i % R], (i / R) & 1, abort_flag);
            tc_fence_after();
            const float* sc = s_ring + (i % R) * BN;
            const uint32_t taddr = tmem_base + lane_off + static_cast<uint32_t>(buf * BN);
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const float2 s2 = *reinterpret_cast<const float2*>(sc + c0 + j);
                    const float2 o = __ffma2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2,
                                                make_float2(acc[c0 + j], acc[c0 + j + 1]));
                    acc[c0 + j] = o.x;
                    acc[c0 + j + 1] = o.y;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tempty[buf]);
                mbar_arrive(&rempty[i % R]);   // (read by the plain kernel's activation warps only)
            }
            if (!dec_warp_all(got)) {
                dec_abort(abort_flag);
                ok = false;
                break;
            }
        }
        if (e == 0) DEC_TRACE(5);
        if (ok && c == 1) {
            const int n = n0 + e;
            if (n < p.N) {
#pragma unroll
                for (int j = 0; j < BN; ++j) {
                    if (j < p.M) {
                        const int64_t o = static_cast<int64_t>(j) * p.N + n;
                        if (p.c_bf16) p.c_bf16[o] = __float2bfloat16_rn(acc[j]);
                        if (p.c_fp32) p.c_fp32[o] = acc[j];
                    }
                }
            }
        } else if (ok) {
            // ---- split-K: row e goes to the CTA owning it (rows [own_lo(o),
            // own_lo(o + 1)) belong to rank o); the owner expects c partial
            // rows of each of its rows and sums them in rank order
            const int rank = static_cast<int>(cluster_rank());
            const int rmax = (128 + c - 1) / c;
            const int owner = (e * c) >> 7;
            const int local = e - own_lo(owner, c);
            const uint32_t dst =
                cluster_map(smem_u32(s_recv + (rank * rmax + local) * BN), static_cast<uint32_t>(owner));
            const uint32_t bar = cluster_map(smem_u32(red_bar), static_cast<uint32_t>(owner));
#pragma unroll
            for (int j = 0; j < BN; j += 4)
                st_async_f4(dst + j * 4, make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]), bar);
            const int my_lo = own_lo(rank, c), my_n = own_lo(rank + 1, c) - my_lo;
            if (e == 0) mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(c * my_n * BN * 4));
            if (!dec_warp_all(mbar_wait(red_bar, 0, abort_flag))) {
                dec_abort(abort_flag);
            } else {
                if (e == 0) DEC_TRACE(6);
                // consecutive threads take consecutive rows (= output columns)
                constexpr int G4 = BN / 4;
                for (int idx = e; idx < my_n * G4; idx += 128) {
                    const int lr = idx % my_n, g4 = idx / my_n;
                    float4 sum = *reinterpret_cast<const float4*>(s_recv + lr * BN + g4 * 4);
                    for (int src = 1; src < c; ++src) {
                        const float4 v = *reinterpret_cast<const float4*>(s_recv + (src * rmax + lr) * BN + g4 * 4);
                        sum.x += v.x;
                        sum.y += v.y;
                        sum.z += v.z;
                        sum.w += v.w;
                    }
                    const int n = n0 + my_lo + lr;
                    if (n < p.N) {
                        const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = g4 * 4 + u;
                            if (j < p.M) {
                                const int64_t o = static_cast<int64_t>(j) * p.N + n;
                                if (p.c_bf16) p.c_bf16[o] = __float2bfloat16_rn(vals[u]);
                                if (p.c_fp32) p.c_fp32[o] = vals[u];
                            }
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, D::kTmemCols);
    if (threadIdx.x == 0) DEC_TRACE(7);
}

// ------------------------------------------------------------------ host side
template <int BN, bool FUSED, int S>
bool configure(int dev) {
    static int done[64] = {0};   // 1 configured, 2 failed
    if (dev < 0 || dev >= 64) return false;
    if (done[dev] == 0) {
        const auto fn = decode_kernel<BN, FUSED, S>;
        const bool ok =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Dec<BN, S>::kSmemBytes) ==
                cudaSuccess &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        done[dev] = ok ? 1 : 2;
    }
    return done[dev] == 1;
}

// Largest cluster size (<= 16) the device can schedule for this kernel.
template <int BN, bool FUSED, int S>
int max_cluster(int dev) {
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64) return 8;
    if (cache[dev] == 0) {
        int best = 1;
        if (configure<BN, FUSED, S>(dev)) {
            for (int cl = kDecMaxCluster; cl >= 2; --cl) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(cl);
                cfg.blockDim = dim3(kDecThreads);
                cfg.dynamicSmemBytes = Dec<BN, S>::kSmemBytes;
                cudaLaunchAttribute attr;
                attr.id = cudaLaunchAttributeClusterDimension;
                attr.val.clusterDim.x = cl;
                attr.val.clusterDim.y = 1;
                attr.val.clusterDim.z = 1;
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<BN, FUSED, S>, &cfg) == cudaSuccess && n > 0) {
                    best = cl;
                    break;
                }
            }
            cudaGetLastError();   // a refused query leaves no sticky error
        }
        cache[dev] = best;
    }
    return cache[dev];
}

struct DecPlan {
    int bn, stages, tiles, c, grid;
};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

// c: the fewest CTAs per tile that minimise the slabs of the busiest CTA,
// within the launch's share of the device's CTA slots and the cluster limit.
void plan_split(DecPlan& pl, int KB, long long budget, int cmax) {
    int best_c = 1, best_max = KB;
    for (int c = 2; c <= std::min(cmax, KB); ++c) {
        if (static_cast<long long>(pl.tiles) * c > budget) break;
        const int m = (KB + c - 1) / c;
        if (m < best_max) {
            best_max = m;
            best_c = c;
        }
    }
    pl.c = best_c;
    pl.grid = pl.tiles * best_c;
}

// (the fused and plain kernels of a tile width need the same resources, so
// one cluster-size query serves both and their plans agree)
DecPlan decode_plan(int64_t M, int64_t N, int64_t K, int sms, int dev) {
    DecPlan pl{};
    pl.bn = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    pl.tiles = static_cast<int>((N + 127) / 128);
    const int KB = static_cast<int>(K / kBlock);
    const int fill = pl.bn == 16 ? FP8BS_DEC_FILL16 : FP8BS_DEC_FILL;
    auto budget = [&](int per_sm) { return std::max<long long>(1, static_cast<long long>(sms) * per_sm * fill / 100); };
    int per_sm = 1, cmax = 1;
    if (pl.bn == 16) {
        pl.stages = kDecStages;
        per_sm = Dec<16, kDecStages>::kMinBlocks;
        cmax = max_cluster<16, false, kDecStages>(dev);
    } else if (pl.bn == 32) {
        pl.stages = kS32;
        per_sm = Dec<32, kS32>::kMinBlocks;
        cmax = max_cluster<32, false, kS32>(dev);
    } else if (pl.tiles <= budget(Dec<64, kS64Deep>::kMinBlocks)) {
        pl.stages = kS64Deep;
        per_sm = Dec<64, kS64Deep>::kMinBlocks;
        cmax = max_cluster<64, false, kS64Deep>(dev);
    } else {
        pl.stages = kDecStages;
        per_sm = Dec<64, kDecStages>::kMinBlocks;
        cmax = max_cluster<64, false, kDecStages>(dev);
    }
    plan_split(pl, KB, budget(per_sm), cmax);
    return pl;
}

template <int BN, bool FUSED, int S>
cudaError_t launch_decode(const CUtensorMap& tw, const CUtensorMap& tx, const DecParams& prm, int grid,
                          unsigned cluster, cudaStream_t st) {
    const int dev = current_device();
    if (!configure<BN, FUSED, S>(dev)) return cudaErrorInvalidValue;
    return launch_pdl_cluster(decode_kernel<BN, FUSED, S>, dim3(grid), dim3(kDecThreads), Dec<BN, S>::kSmemBytes,
                              st, cluster, tw, tx, prm);
}

#ifdef FP8BS_TRACE_ENABLED
int g_dtrace_next = 0;
#endif

}  // namespace

// Shared by fp8_gemm (xq + a_s, M <= 64) and fp8_linear (x, M <= 16: the
// quantisation fused; larger batches stage act_quant first): the
// same plan for both, so their results agree bit for bit.
fp8_status decode_gemm(const void* x, const void* xq, const float* a_s, const void* w, const float* b_s,
                       void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K, int ue8m0,
                       int debug_skip, cudaStream_t st) {
    const int dev = current_device();
    if (dev < 0) return FP8_ERR_CUDA;
    const bool fused = x != nullptr;
    if (fused && M > kDecodeFusedMaxM) return FP8_ERR_UNSUPPORTED;
    const DecPlan pl = decode_plan(M, N, K, device_sm_count(), dev);
    if (static_cast<long long>(pl.tiles) * pl.c > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    DecParams prm{};
    prm.xq = static_cast<const uint8_t*>(xq);
    prm.x = static_cast<const uint16_t*>(x);
    prm.a_s = a_s;
    prm.b_s = b_s;
    prm.c_bf16 = static_cast<__nv_bfloat16*>(c_bf16);
    prm.c_fp32 = c_fp32;
    prm.K = K;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.KB = static_cast<int>(K / kBlock);
    prm.c = pl.c;
    prm.ue8m0 = ue8m0;
    prm.debug_skip = debug_skip;
#ifdef FP8BS_TRACE_ENABLED
    prm.trace_slot = g_dtrace_next++ & 3;
#endif
    CUtensorMap tw, tx;
    if (!make_map(&tw, w, N, K, 128)) return FP8_ERR_CUDA;
    if (fused) tx = tw;   // not read
    else if (!make_map(&tx, xq, M, K, pl.bn)) return FP8_ERR_CUDA;
    const unsigned cl = static_cast<unsigned>(pl.c);
    cudaError_t e;
    if (pl.bn == 16)
        e = fused ? launch_decode<16, true, kDecStages>(tw, tx, prm, pl.grid, cl, st)
                  : launch_decode<16, false, kDecStages>(tw, tx, prm, pl.grid, cl, st);
    else if (pl.bn == 32)
        e = launch_decode<32, false, kS32>(tw, tx, prm, pl.grid, cl, st);
    else if (pl.stages == kS64Deep)
        e = launch_decode<64, false, kS64Deep>(tw, tx, prm, pl.grid, cl, st);
    else
        e = launch_decode<64, false, kDecStages>(tw, tx, prm, pl.grid, cl, st);
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

bool decode_set_wait_limit(long long cycles) {
    return cudaMemcpyToSymbol(g_wait_limit_cycles, &cycles, sizeof(cycles)) == cudaSuccess;
}

int decode_read_and_clear_status(cudaStream_t st) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_decode_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return -1;
        if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace fp8bs

#ifdef FP8BS_TRACE_ENABLED
extern "C" int fp8_debug_clear_decode_trace(void) {
    static unsigned long long zero[4][1024][8];
    fp8bs::g_dtrace_next = 0;
    return cudaMemcpyToSymbol(fp8bs::g_dtrace, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
extern "C" int fp8_debug_read_decode_trace(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, fp8bs::g_dtrace, sizeof(unsigned long long) * 4 * 1024 * 8) == cudaSuccess ? 0
                                                                                                                 : 1;
}
#endif
