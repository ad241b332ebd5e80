// common.cuh -- shared device helpers for the sm_103a FP8 block-scaled
// linear library: status codes, inline-PTX wrappers for mbarrier, TMA
// (cp.async.bulk.tensor) and the 5th-generation tensor core (tcgen05), and
// the number-format conversions the kernels use.
//
// Every wait in this library is bounded: a wait that runs past its limit
// records FP8_ERR_TIMEOUT in the device status word of its translation unit
// and the kernel winds down instead of hanging.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/fp8bs.h"

namespace fp8bs {

constexpr int kBlock = 128;            // quantisation block (elements)
constexpr float kE4m3Max = 448.0f;     // largest finite float8_e4m3fn
constexpr float kAmaxFloor = 1e-4f;    // clamp on a block's max |x|

// ~1 s at 2 GHz: far above any legitimate wait inside one kernel.
constexpr long long kWaitLimitCycles = 2000000000LL;
// The limit the waits use (SM clock cycles).  Only the test hook
// fp8_debug_set_wait_limit changes it, so that a test of the failure path
// ends in milliseconds; one copy per translation unit (the GEMM's is the one
// that matters: its kernels are the ones that wait).
static __device__ long long g_wait_limit_cycles = kWaitLimitCycles;

#define FP8_CUDA_TRY(expr)                                   \
    do {                                                     \
        cudaError_t e_ = (expr);                             \
        if (e_ != cudaSuccess) return FP8_ERR_CUDA;          \
    } while (0)

// ---------------------------------------------------------------- scalar
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Two fp32 -> two e4m3 codes, round to nearest even, saturating to +-448.
// The first argument lands in the low byte (lower address).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 codes (low byte first) -> two f32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
    uint32_t h2;   // f16x2: low half = low byte
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

// Smallest power of two >= s, for finite normal s > 0 (bit-level).
__device__ __forceinline__ float pow2_ceil(float s) {
    uint32_t u = __float_as_uint(s);
    if ((u & 0x007FFFFFu) == 0u) return s;
    return __uint_as_float((u & 0x7F800000u) + 0x00800000u);
}

// The block scale: clamped max / 448 rounded to nearest (as an IEEE
// divide), optionally ue8m0.  amax is always the magnitude of a bf16 value
// (or below the floor); on that domain one Markstein correction of
// amax * RN(1/448) -- remainder by fma, then fma update (P. Markstein, IBM J.
// Res. Dev. 34(1), 1990) -- gives the correctly rounded quotient for every
// value, which the GPU tests check against the oracle's division block max by
// block max.
__device__ __forceinline__ float block_scale(float amax, bool ue8m0) {
    constexpr float r = 1.0f / kE4m3Max;   // RN(1/448), folded at compile time
    const float a = fmaxf(amax, kAmaxFloor);
    const float q0 = __fmul_rn(a, r);
    const float e = __fmaf_rn(-q0, kE4m3Max, a);
    const float s = __fmaf_rn(e, r, q0);
    return ue8m0 ? pow2_ceil(s) : s;
}

// max |f[i]| over 8 values as a tree (max is exact, so the order is free).
__device__ __forceinline__ float max_abs8(const float (&f)[8]) {
    const float m0 = fmaxf(fabsf(f[0]), fabsf(f[1])), m1 = fmaxf(fabsf(f[2]), fabsf(f[3]));
    const float m2 = fmaxf(fabsf(f[4]), fabsf(f[5])), m3 = fmaxf(fabsf(f[6]), fabsf(f[7]));
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// 8 bf16 (one 16-byte load) -> 8 fp32, exact.
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// x / s for 8 values, then RNE-satfinite e4m3, packed low byte first.  The
// one quantisation routine of the library: act_quant, the fused expert body
// and the fused decode linear all call it, so their codes agree bit for bit.
//
// The quotient must be the IEEE fp32 x / s rounded to nearest.  ue8m0 scales
// are powers of two, so x * (1/s) is that quotient exactly.  For fp32 scales
// the quotient is formed by Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): r = RN(1/s), q0 = RN(x r), the
// exact remainder e = x - q0 s by one fma, then q = RN(q0 + e r).  Here x is
// a bf16 value and s = RN(max(|x|max, 1e-4) / 448) of its block, so x/s
// depends only on the two 8-bit mantissas and their exponent gap; the
// parity tests enumerate that whole domain against the oracle's IEEE
// division.  The remainder is formed negated, e' = q0 s - x, and q = RN(q0 -
// e' r): the same roundings (nearest-even is symmetric), and a zero x keeps
// its sign with no test, as every sum of zeros then rounds to the sign of x.
// The core takes the negated values nx = -x and -r, so that every step is a
// packed two-lane multiply or fma with no negated operand: q0 = RN(nx (-r)),
// e' = RN(q0 s + nx), q = RN(e' (-r) + q0).
template <bool UE8M0>
__device__ __forceinline__ uint2 quant8n(const float (&nx)[8], float s, float r) {
    const float2 nr2 = make_float2(-r, -r), s2 = make_float2(s, s);
    float2 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 n2 = make_float2(nx[2 * i], nx[2 * i + 1]);
        const float2 q0 = __fmul2_rn(n2, nr2);
        if (UE8M0) {
            q[i] = q0;   // s is a power of two: x (1/s) is exact
        } else {
            const float2 en = __ffma2_rn(q0, s2, n2);
            q[i] = __ffma2_rn(en, nr2, q0);
        }
    }
    uint2 out;
    out.x = static_cast<uint32_t>(f32x2_to_e4m3x2(q[0].x, q[0].y)) |
            (static_cast<uint32_t>(f32x2_to_e4m3x2(q[1].x, q[1].y)) << 16);
    out.y = static_cast<uint32_t>(f32x2_to_e4m3x2(q[2].x, q[2].y)) |
            (static_cast<uint32_t>(f32x2_to_e4m3x2(q[3].x, q[3].y)) << 16);
    return out;
}

template <bool UE8M0>
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s) {
    float nx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) nx[i] = -f[i];
    return quant8n<UE8M0>(nx, s, __frcp_rn(s));
}

// 8 bf16 (one 16-byte load) -> their 8 negated fp32 values, exact (the sign
// bit flipped), for quant8n.
__device__ __forceinline__ void unpack_bf16x8_neg(const uint4& v, float (&nx)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        nx[2 * i] = __uint_as_float((w[i] << 16) ^ 0x80000000u);
        nx[2 * i + 1] = __uint_as_float((w[i] & 0xFFFF0000u) ^ 0x80000000u);
    }
}

// The expert body's gate for one element pair: g = bf16(bf16(silu(h1)) * h3)
// with silu(v) = v / (1 + exp(-v)) in fp32, from bf16 inputs given as fp32
// (exact).  The exponential and the quotient use the fast hardware
// approximations (__expf, __fdividef: relative errors of a few fp32 ulps,
// far below the bf16 rounding that follows; for v < -87 the quotient is
// +-0, as is the bf16 of the exact value).  The one routine of the library
// for it: the standalone silu*mul+act_quant kernel and the GEMM epilogue
// that fuses it both call it, so their results agree bit for bit.  Returns
// the two bf16 results packed (first in the low half).
__device__ __forceinline__ uint32_t silu_mul_bf16x2(float a0, float a1, float b0, float b1) {
    const float s0 = __fdividef(a0, 1.0f + __expf(-a0));
    const float s1 = __fdividef(a1, 1.0f + __expf(-a1));
    const float sb0 = __bfloat162float(__float2bfloat16_rn(s0));
    const float sb1 = __bfloat162float(__float2bfloat16_rn(s1));
    const __nv_bfloat162 g = __floats2bfloat162_rn(sb0 * b0, sb1 * b1);
    return *reinterpret_cast<const uint32_t*>(&g);
}

// Make this thread's generic-proxy shared-memory writes visible to the
// async proxy (the tensor core reading operands from shared memory).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of the given parity to complete.  Returns false
// (and leaves the barrier alone) if the limit passed or *abort became set.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (clock64() - t0 > g_wait_limit_cycles) return false;
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  x is the innermost (contiguous) coordinate in
// elements and must be a multiple of 16 for 1-byte data.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const void* tmap, uint64_t* bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled store of one box from shared memory to global memory, tracked
// as a bulk async-group of the issuing thread.  Coordinates beyond the
// tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(smem_u32(smem_src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the thread's committed bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// the thread's committed bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation: executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes (128 e4m3 values) written by TMA with the 128-byte swizzle:
// 8-row x 128-byte swizzle atoms stacked every 1024 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address / 16
    d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride offset: 8 rows * 128 B
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptor: D f32, A and B e4m3, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                       // D format f32
         | (0u << 7) | (0u << 10)                          // A, B: e4m3
         | (0u << 15) | (0u << 16)                         // K-major A and B
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one K=32 step of e4m3, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for the block-scaled kind (mxf8f6f4 with E8M0
// scales, one per 32 K values of each A row and each B column): D f32 is
// implied; A and B e4m3, K-major, shape M x N; sf_id picks the byte of each
// 32-bit scale word in tensor memory (the K=32 step within a 128-K slab).
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N, int sf_id) {
    return (static_cast<uint32_t>(sf_id) << 4)                // B scale byte
         | (0u << 7) | (0u << 10)                             // A, B: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (1u << 23)                                         // scales are E8M0
         | (static_cast<uint32_t>(M >> 4) << 24)
         | (static_cast<uint32_t>(sf_id) << 29);              // A scale byte
}

// D[tmem] (+)= (A * 2^sfa) (B * 2^sfb)^T, one K=32 step of e4m3 with E8M0
// block scales read from tensor memory: the scale of A row m at lane m,
// column sfa + m/32; the scale of B column n at column sfb + n/32, lane
// n % 32 of every lane quarter (rows of quarter q read quarter q's copy).
__device__ __forceinline__ void mma_mx_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 bit stores into tensor memory: thread i of the warp writes
// columns [col, col + 4) (x4) or [col, col + 8) (x8) of lane (lane_base + i).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t a, uint32_t b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2};" ::"r"(taddr),
                 "r"(a), "r"(b)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp receives
// columns [col, col+16) of TMEM lane (lane_base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Whole-cluster barrier (every thread of every CTA of the cluster).  Used
// only where every thread is known to arrive: right after set-up and at the
// very end of the kernel, never behind a data-dependent wait.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
    return r;
}

// Arrive (release at cluster scope) on an mbarrier of another CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Asynchronous 16-byte store into the shared memory of a CTA of the cluster,
// counted as 16 transaction bytes on that CTA's mbarrier remote_bar: the
// receiver's barrier completes once every such store has landed, with no
// fence or arrive on the sender's side.
__device__ __forceinline__ void st_async_f4(uint32_t remote_saddr, float4 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_saddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t remote_saddr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote_saddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t remote_saddr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote_saddr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// A pair of CTAs on two SMs shares one MMA of M = 256: the leader (rank 0)
// issues it, each CTA holds 128 rows of the accumulator in its own TMEM and
// stages its own halves of the operands; every tcgen05 instruction of such a
// kernel uses cta_group::2.

// Bounded wait with acquire at cluster scope, for barriers other CTAs arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (clock64() - t0 > g_wait_limit_cycles) return false;
        }
    }
}

// Relaxed arrive on a barrier of a CTA of the cluster.  Enough where the
// data handed over lives in tensor memory: tcgen05.wait::st / wait::ld and
// tcgen05.fence::before_thread_sync order it before the arrive, and the
// waiter's fence::after_thread_sync after its wait.  (A release at cluster
// scope here halved the pair kernel's speed.)
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Executed by one whole warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// The pair's block-scaled K=32 step (as mma_mx_e4m3, with M = 256): A rows
// 0-127 and B rows 0-127 are read from the leader's shared memory, rows
// 128-255 of each from the peer's at the same offsets; each CTA's scales come
// from its own TMEM (A: its 128 rows; B: all N columns, as in the 1-CTA form).
__device__ __forceinline__ void mma_mx_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at this offset in both CTAs of the pair when
// every tcgen05 operation issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted
// on the pair leader's barrier (`bar_cluster`, a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// ---------------------------------------------------------------- dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation: it lets the next kernel on the stream start launching at
// once and, before touching any global input or output, waits for the grids
// it depends on to finish (a no-op when it was launched without the
// attribute or after a kernel that never signals).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- host
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
#ifndef FP8BS_NO_PDL   // profiling builds only: plain stream order
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
#endif
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
    return launch_pdl_cluster(kernel, grid, block, smem, st, 1u, std::forward<Args>(args)...);
}

int device_sm_count();   // cached per device (api.cu)

// Batches the decode kernel (decode.cu) serves: fp8_gemm up to 64 tokens;
// fp8_linear quantises the activations inside it up to 16 tokens.
constexpr int64_t kDecodeMaxM = 64;
constexpr int64_t kDecodeFusedMaxM = 16;

// TMA tensor maps over row-major matrices [rows, K], 128-byte swizzle (gemm.cu):
// e4m3 with boxes of 128 x box_rows bytes; bf16 with boxes of 64 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows);
bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows);

}  // namespace fp8bs
