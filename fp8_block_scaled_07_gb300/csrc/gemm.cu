// gemm.cu -- block-scaled FP8 GEMM on sm_103a tensor cores.
//
// What it computes ("Data flow -- deepseek-ai/DeepSeek-V3", bullet "FP8
// quantization data flow"; source tour "DeepSeek-V3", paragraph "FP8 with
// per-block scales"):
//   C[m, n] = sum_kb a_s[m, kb] * b_s[n/128, kb] * sum_{k in kb} a[m,k] b[n,k]
// with e4m3 operands, fp32 scales and fp32 accumulation; the grouped form
// runs the same product per routed expert over packed rows ("Behavior
// traces", bullet "MoE trace"; source tour, "Honest Limits").
//
// How (GB300-native, not the pages' Triton design):
//   * one 128-K slab is one pipeline stage: TMA brings a 128x128 e4m3 tile
//     of the "P" operand and a BNx128 tile of the "Q" operand into shared
//     memory (128-byte swizzle); one thread issues four K=32
//     tcgen05.mma.kind::f8f6f4 into a fresh TMEM slab buffer (128 lanes x
//     BN fp32 columns);
//   * four epilogue warps read the finished slab from TMEM (tcgen05.ld),
//     multiply by the slab's scale product a_s*b_s and accumulate in fp32
//     registers ("promotion"), while the tensor core fills the other slab
//     buffer;
//   * warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
//     owner), warps 4.. = epilogue; persistent CTAs, one per SM;
//   * decode shapes (M <= 64) run on the kernel of decode.cu instead;
//   * few tiles -> stream-K: each CTA takes an equal run of (tile, slab)
//     units; tiles split across CTAs are reduced deterministically by the
//     CTA that finishes a tile last (fp32 partials in the caller's
//     workspace, one atomic ticket per tile, no spinning).
// Every mbarrier wait is bounded (see common.cuh).
#include "common.cuh"
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

namespace fp8bs {

__device__ int g_gemm_status;   // FP8_OK or FP8_ERR_TIMEOUT, read by fp8_device_status

// Optional per-CTA timeline (global timer, ns) for profiling builds only;
// compiles to nothing unless FP8BS_TRACE_ENABLED is defined.
#ifdef FP8BS_TRACE_ENABLED
__device__ unsigned long long g_trace[4][512][24];
#define FP8BS_TRACE_VAL(slot, v)                                                      \
    do {                                                                             \
        if (blockIdx.x < 512) g_trace[p.trace_slot & 3][blockIdx.x][slot] = (v);     \
    } while (0)
#define FP8BS_TIC(v) const long long v = clock64()
#define FP8BS_TOC(acc, v) acc += clock64() - (v)
#define FP8BS_TRACE(slot)                                                            \
    do {                                                                             \
        if (blockIdx.x < 512) {                                                      \
            unsigned long long t_;                                                   \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                    \
            g_trace[p.trace_slot & 3][blockIdx.x][slot] = t_;                        \
        }                                                                            \
    } while (0)
#else
#define FP8BS_TRACE(slot) \
    do {                  \
    } while (0)
#define FP8BS_TRACE_VAL(slot, v) \
    do {                         \
    } while (0)
#define FP8BS_TIC(v)
#define FP8BS_TOC(acc, v)
#endif

namespace {

constexpr int kNumThreads = 256;
constexpr int kEpiWarp0 = 4;               // epilogue warps 4..7 (warp % 4 = TMEM lane quarter)
constexpr int kPTileBytes = 128 * kBlock;  // 128 rows x 128 e4m3
constexpr int kMaxGroups = 1024;
// Workspace layout: a fixed block of stream-K tile counters (which must stay
// zero between calls, whatever shape used the workspace before), then the
// fp32 partial tiles (no requirement on their contents).
constexpr int kMaxSkTiles = 4096;
constexpr size_t kCounterBytes = kMaxSkTiles * sizeof(int);

enum Variant { kDense = 0, kGrouped = 2 };

// Register split of the 128x256 kernels (warpgroup 0 / epilogue warpgroups).
#ifndef FP8BS_REGS_LOW
#define FP8BS_REGS_LOW 120
#endif
#ifndef FP8BS_REGS_HIGH
#define FP8BS_REGS_HIGH 192
#endif


struct Params {
    const float* a_s;          // [rows_a, KB]
    const float* b_s;          // [G][NB][KB]
    const int32_t* offsets;    // grouped: [G+1] (device)
    __nv_bfloat16* c_bf16;     // [rows, N] or null
    float* c_fp32;             // [rows, N] or null
    float* partials;           // stream-K workspace
    int* counters;             // stream-K tickets, one per tile
    int M;                     // rows of A (grouped: rows covered by offsets <= R_max)
    int N;                     // columns of C (per expert when grouped)
    int KB;                    // K / 128
    int NB;                    // ceil(N / 128)
    int G;                     // experts (grouped)
    int tiles_p, tiles_q;      // dense tile grid (P rows / 128, Q rows / BN)
    int num_tiles;             // dense
    int stream_k;              // 1: stream-K schedule over total_units
    long long total_units;     // num_tiles * KB
    int trace_slot;            // profiling builds: which timeline buffer this launch fills
    int tma_store;             // dense, bf16 only: full tiles leave through shared memory and TMA
    int vec_scales;            // scale rows are 16-byte aligned (K/128 % 4 == 0, aligned bases)
    int debug_skip;            // test hook: the MMA issuer skips its arrive on slab 0's TMEM-full barrier
    // the kernels with the expert body fused into the epilogue of the w1|w3
    // product (128x256 tiles; weights interleaved so a tile holds h1 and h3
    // of one 128-wide block): g = bf16(bf16(silu(h1)) * h3) -> act_quant ->
    // gq [rows, N/2] e4m3, gs [rows, N/256] fp32, instead of storing h
    int ue8m0;                 // scale format of g's codes
    uint8_t* gq;
    float* gs;
};

struct Tile {
    int p_row0, q_row0;   // TMA row coordinates of the P and Q tiles
    int p_valid, q_valid; // rows of the tile that hold real data
    int group;            // expert (grouped) else 0
    int q_col0;           // grouped: first output column of the tile
};

struct Seg {
    int tile, k0, k1;
};

template <int BN, int V, bool SW = false>
struct Cfg {
    static constexpr int kQTileBytes = BN * kBlock;
    static constexpr int kStageBytes = kPTileBytes + kQTileBytes;
    // the expert body of a 128x256 tile runs on warps 2-3 ("gate warps"),
    // from the tile's bf16 h left in shared memory by the epilogue warps
    static constexpr bool kGate = SW && BN == 256;
    static constexpr int kHBytes = 128 * 256 * 2;
    static constexpr int kStages = BN == 256 ? (kGate ? 3 : 4) : 6;
    // 128x256 tiles: 8 epilogue warps, two per TMEM lane quarter, each owning
    // 128 of the 256 columns; their warpgroups take registers from warps 0-3
    static constexpr int kEpiWarps = BN == 256 ? 8 : 4;
    static constexpr int kThreads = 128 + 32 * kEpiWarps;
    static constexpr int kMinBlocks = 1;
    static constexpr int kCPT = BN * 4 / kEpiWarps;   // accumulator columns per epilogue thread
    static constexpr bool kSplitRegs = BN == 256;
    // the MMA issuer checks one barrier per slab (each check by the issuing
    // thread costs tensor time): a stage's full barrier also counts the
    // epilogue warps' release of the TMEM buffer the slab will write, i.e. of
    // the slab two before it
    static constexpr bool kMergeT = true;
    // the producer and MMA warps keep their tile state in registers (spills
    // there were reloaded every slab); 120*128 + 192*256 = 168*384
    static constexpr int kRegsLow = FP8BS_REGS_LOW, kRegsHigh = FP8BS_REGS_HIGH;
    static constexpr int kTmemCols = 2 * BN;   // two slab buffers
    static constexpr int kBarBytes = 1024;
    // grouped: per-expert tile prefix
    static constexpr int kExtraBytes = V == kGrouped ? (kMaxGroups + 1 + 16) * 4 : 0;
    // per epilogue warp a staging box (kStgRows rows x 64 bf16, 128-byte
    // swizzle) through which output tiles leave by TMA stores; 32 rows dense,
    // 16 grouped (whose expert-tile prefix takes the room)
    // (the gate kernels use the room for the h tile instead)
    static constexpr bool kTmaStore = true;
    static constexpr int kStgRows = V == kGrouped ? 16 : 32;
    static constexpr int kStgBytes = kGate ? kHBytes : kEpiWarps * kStgRows * 128;
    static constexpr int kSmemBytes =
        1024 /*align slack*/ + kStages * kStageBytes + kStgBytes + kBarBytes + kExtraBytes;
};

// ------------------------------------------------------------------ schedule
__device__ __forceinline__ long long sk_start(long long c, long long U, long long P) {
    return c * U / P;
}
__device__ __forceinline__ int sk_owner(long long u, long long U, int P) {
    long long c = u * P / U;
    while (c + 1 < P && sk_start(c + 1, U, P) <= u) ++c;
    while (c > 0 && sk_start(c, U, P) > u) --c;
    return static_cast<int>(c);
}

struct SegIter {
    // data-parallel: tiles blockIdx.x + i * gridDim.x; stream-K: units [lo, hi)
    long long u, hi;
    int t, stride, num_tiles, KB;
    bool sk;
    __device__ void init(const Params& p, int ntiles) {
        KB = p.KB;
        sk = p.stream_k != 0;
        num_tiles = ntiles;
        if (sk) {
            u = sk_start(blockIdx.x, p.total_units, gridDim.x);
            hi = sk_start(blockIdx.x + 1, p.total_units, gridDim.x);
        } else {
            t = blockIdx.x;
            stride = gridDim.x;
        }
    }
    __device__ bool next(Seg& s) {
        if (sk) {
            if (u >= hi) return false;
            s.tile = static_cast<int>(u / KB);
            s.k0 = static_cast<int>(u - static_cast<long long>(s.tile) * KB);
            long long end = static_cast<long long>(s.tile + 1) * KB;
            if (end > hi) end = hi;
            s.k1 = static_cast<int>(end - static_cast<long long>(s.tile) * KB);
            u = end;
            return true;
        }
        if (t >= num_tiles) return false;
        s.tile = t;
        s.k0 = 0;
        s.k1 = KB;
        t += stride;
        return true;
    }
};

// Whole tiles blockIdx.x + i * gridDim.x only: the 128x256 kernels, whose
// producer and MMA warps run on a small register budget, never split K.
struct DpIter {
    int t, stride, num_tiles, KB;
    __device__ void init(const Params& p, int ntiles) {
        t = blockIdx.x;
        stride = gridDim.x;
        num_tiles = ntiles;
        KB = p.KB;
    }
    __device__ bool next(Seg& s) {
        if (t >= num_tiles) return false;
        s.tile = t;
        s.k0 = 0;
        s.k1 = KB;
        t += stride;
        return true;
    }
    // the tile next() returns next, without advancing
    __device__ bool peek(Seg& s) const {
        if (t >= num_tiles) return false;
        s.tile = t;
        s.k0 = 0;
        s.k1 = KB;
        return true;
    }
};

// Grouped: per-expert m-tiles (ceil(rows/128)) x N/BN n-tiles; tile index
// runs m-fastest inside an expert so CTAs working at the same time share the
// expert's weight tile through L2.
template <int BN, int V>
__device__ __forceinline__ Tile tile_geom(const Params& p, int t, const int* s_prefix) {
    Tile g{};
    if (V == kDense) {
        const int tp = t % p.tiles_p, tq = t / p.tiles_p;
        g.p_row0 = tp * 128;
        g.q_row0 = tq * BN;
        g.p_valid = min(128, p.M - g.p_row0);
        g.q_valid = min(BN, p.N - g.q_row0);
    } else {
        int lo = 0, hi = p.G;        // largest g with s_prefix[g] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= t) lo = mid; else hi = mid;
        }
        const int grp = lo;
        const int r0 = p.offsets[grp], cnt = p.offsets[grp + 1] - r0;
        const int mt = (cnt + 127) / 128;
        const int local = t - s_prefix[grp];
        const int tp = local % mt, tq = local / mt;
        g.group = grp;
        g.p_row0 = r0 + tp * 128;
        g.p_valid = min(128, cnt - tp * 128);
        g.q_col0 = tq * BN;
        g.q_row0 = grp * p.N + tq * BN;
        g.q_valid = min(BN, p.N - tq * BN);
    }
    return g;
}

__device__ __noinline__ bool gate_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait(bar, parity, abort_flag);
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(&g_gemm_status, static_cast<int>(FP8_ERR_TIMEOUT));
}

// True on every lane of the warp iff it is true on all of them: the outcome
// of a bounded wait is made warp-uniform before any warp-collective step.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xFFFFFFFFu, ok) != 0; }

// Store the CPT accumulators of one output row starting at tile column cofs.
template <int BN, int V, int CPT>
__device__ __forceinline__ void store_tile(const Params& p, const Tile& tg, int e, int cofs,
                                           const float (&acc)[CPT]) {
    if (e >= tg.p_valid) return;
    const int64_t row = tg.p_row0 + e;
    const int col0 = ((V == kGrouped) ? tg.q_col0 : tg.q_row0) + cofs;
    const int valid = tg.q_valid - cofs;
    const bool vec = (p.N % 8 == 0);
#pragma unroll
    for (int j0 = 0; j0 < CPT; j0 += 8) {
        const int col = col0 + j0;
        if (vec && j0 + 8 <= valid) {
            if (p.c_bf16) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __nv_bfloat162 b = __floats2bfloat162_rn(acc[j0 + 2 * i], acc[j0 + 2 * i + 1]);
                    w[i] = *reinterpret_cast<uint32_t*>(&b);
                }
                *reinterpret_cast<uint4*>(p.c_bf16 + row * p.N + col) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (p.c_fp32) {
                float4* d = reinterpret_cast<float4*>(p.c_fp32 + row * p.N + col);
                d[0] = make_float4(acc[j0], acc[j0 + 1], acc[j0 + 2], acc[j0 + 3]);
                d[1] = make_float4(acc[j0 + 4], acc[j0 + 5], acc[j0 + 6], acc[j0 + 7]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (j0 + i < valid) {
                    if (p.c_bf16) p.c_bf16[row * p.N + col + i] = __float2bfloat16_rn(acc[j0 + i]);
                    if (p.c_fp32) p.c_fp32[row * p.N + col + i] = acc[j0 + i];
                }
            }
        }
    }
}

// Store this warp's 32 output rows x CPT columns as bf16 through its
// staging buffer: lane = row, one TMA box of ROWS rows x 64 columns at a
// time (ROWS = 32, or 16: the two halves of the warp in turn), in the
// 128-byte-swizzled layout of the store's tensor map (16-byte chunk c of row
// r sits at chunk c ^ (r % 8), so the writes are conflict free).  Boxes
// wholly outside the output (rows_valid or cols_valid used up) are skipped;
// the TMA unit clips partial ones at the tensor's edge.  With ROWS = 16 a
// half with fewer than 16 valid rows (a tile ending inside it, as grouped
// tiles do at expert boundaries) is not stored here: the caller stores those
// rows directly; the return value is that half's first row (or 32 if none).
template <int CPT, int ROWS>
__device__ __forceinline__ int store_tile_tma(const CUtensorMap* tm_c, uint8_t* stg, int lane, int col0, int row0,
                                              int rows_valid, int cols_valid, const float (&acc)[CPT]) {
    if (rows_valid <= 0) return 32;
#pragma unroll
    for (int h0 = 0; h0 < 32; h0 += ROWS) {
        if (h0 >= rows_valid) return 32;
        if (ROWS < 32 && rows_valid < h0 + ROWS) return h0;   // partial half: direct stores
        const bool mine = lane >= h0 && lane < h0 + ROWS;
        const int rr = lane - h0;                              // row within the box
#pragma unroll
        for (int h = 0; h < CPT / 64; ++h) {
            if (h * 64 >= cols_valid) break;
            if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
            __syncwarp();
            if (mine) {
                uint8_t* row = stg + rr * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        __nv_bfloat162 b =
                            __floats2bfloat162_rn(acc[h * 64 + c * 8 + 2 * i], acc[h * 64 + c * 8 + 2 * i + 1]);
                        w[i] = *reinterpret_cast<uint32_t*>(&b);
                    }
                    *reinterpret_cast<uint4*>(row + ((c ^ (rr & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tm_c, stg, col0 + h * 64, row0 + h0);
                bulk_commit();
            }
        }
    }
    return 32;
}

// Exclusive prefix over experts of their tile counts (m-tiles x tq), by the
// whole block: each thread takes up to 4 experts, then a block-wide scan.
// G <= kMaxGroups and NT >= 256, so 4 experts per thread always suffice.
template <int NT>
__device__ __forceinline__ void expert_tile_prefix(const int32_t* offsets, int G, int tq, int* s_prefix,
                                                   int* s_warp) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int per = (G + NT - 1) / NT;
    const int g0 = t * per;
    int vals[4];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = g0 + i;
        int v = 0;
        if (i < per && g < G) {
            const int cnt = __ldg(offsets + g + 1) - __ldg(offsets + g);
            v = ((cnt + 127) / 128) * tq;
        }
        vals[i] = v;
        local += v;
    }
    int inc = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    int run = inc - local;
    for (int i = 0; i < w; ++i) run += s_warp[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = g0 + i;
        if (i < per && g < G) {
            s_prefix[g] = run;
            run += vals[i];
            if (g == G - 1) s_prefix[G] = run;
        }
    }
}

// Promote one finished slab from TMEM into the fp32 accumulators:
// acc[j] += D[lane][j] * scale, the scale per column (smem, swapped layout)
// or uniform for the row.  Packed f32x2 FMAs (two IEEE round-to-nearest
// FMAs per instruction, so the same values as scalar fmaf) halve the issue
// slots of the promotion, which otherwise runs longer than the tensor core
// takes for the next slab.
template <int N, bool PER_COL>
__device__ __forceinline__ void fma_chunk(float* acc, const uint32_t* r, const float* sc_col, float sc) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        const float2 s2 = PER_COL ? *reinterpret_cast<const float2*>(sc_col + j) : make_float2(sc, sc);
        const float2 v = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), s2,
                                    make_float2(acc[j], acc[j + 1]));
        acc[j] = v.x;
        acc[j + 1] = v.y;
    }
}

template <int BN, bool PER_COL>
__device__ __forceinline__ void promote(uint32_t taddr, float (&acc)[BN], const float* sc_col, float sc) {
    if constexpr (BN == 16) {
        uint32_t r[16];
        tmem_ld16(taddr, r);
        tmem_wait_ld();
        fma_chunk<16, PER_COL>(acc, r, sc_col, sc);
    } else {
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + c0, r);
            tmem_wait_ld();
            fma_chunk<32, PER_COL>(acc + c0, r, PER_COL ? sc_col + c0 : nullptr, sc);
        }
    }
}

// Barrier of the epilogue threads on an mbarrier (one arrival per thread) so
// that a thread that gave up on a wait cannot leave the others blocked
// forever; the warp's outcome is uniform.
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& phase, const volatile int* abort_flag) {
    mbar_arrive(bar);
    const bool ok = warp_all(mbar_wait(bar, phase, abort_flag));
    phase ^= 1u;
    if (!ok) {
        *const_cast<volatile int*>(abort_flag) = 1;
        atomicExch(&g_gemm_status, static_cast<int>(FP8_ERR_TIMEOUT));
    }
    return ok;
}

// SW: the expert body fused into the w1|w3 product (a kernel of its own,
// so that the plain kernels' register allocation does not carry it): the
// epilogue warps leave each finished 128x256 tile in shared memory as bf16
// and go on to the next tile; warps 2-3, idle in the plain kernels, turn it
// into g's codes and scales meanwhile.
template <int BN, int V, bool SW>
__global__ void __launch_bounds__((Cfg<BN, V, SW>::kThreads), (Cfg<BN, V, SW>::kMinBlocks))
    gemm_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_c, const Params p) {
    using C = Cfg<BN, V, SW>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sP = smem;                                   // S x 16 KB
    uint8_t* sQ = smem + S * kPTileBytes;                 // S x BN*128
    uint8_t* sStg = smem + S * C::kStageBytes;           // kEpiWarps output staging boxes
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes + C::kStgBytes);
    uint64_t* full = bars;                 // S
    uint64_t* empty = bars + S;            // S
    uint64_t* tfull = bars + 2 * S;        // 2
    uint64_t* tempty = bars + 2 * S + 2;   // 2
    uint64_t* mma_done = bars + 2 * S + 4; // 1
    uint64_t* epi_bar = bars + 2 * S + 5;  // epilogue-group barrier
    uint64_t* h_full = bars + 2 * S + 6;   // gate kernels: the h tile is in shared memory
    uint64_t* h_empty = bars + 2 * S + 7;  // gate kernels: the gate warps have read it
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* ticket_box = reinterpret_cast<volatile int*>(tmem_holder + 2);
    int* s_prefix = reinterpret_cast<int*>(smem + S * C::kStageBytes + C::kStgBytes + C::kBarBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) FP8BS_TRACE(0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            // the producer's bytes + the epilogue warps' release of a TMEM buffer
            mbar_init(&full[i], 1 + C::kEpiWarps);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], C::kEpiWarps);   // one arrival per epilogue warp
        }
        if constexpr (C::kMergeT) {
            static_assert(S >= 3, "the release of slab k-2 must land in the phase of slab k");
            for (int w = 0; w < C::kEpiWarps; ++w) {   // slabs 0 and 1 find their TMEM buffers free
                mbar_arrive(&full[0]);
                mbar_arrive(&full[1]);
            }
        }
        mbar_init(mma_done, 1);
        mbar_init(epi_bar, 32 * C::kEpiWarps);
        mbar_init(h_full, 32 * C::kEpiWarps);   // one arrival per epilogue thread
        mbar_init(h_empty, 64);                 // one arrival per gate thread
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_p);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // dependents may launch only once this CTA holds its tensor memory (a
    // dependent CTA on the same SM must never take columns this one needs);
    // an otherwise idle warp signals, so the producer is not delayed
    if (threadIdx.x == 96) griddep_launch_dependents();
    // Inputs written by earlier launches are visible to a thread once it has
    // passed griddepcontrol.wait.  Each role waits just before its first
    // access to global memory, so the set-up before it overlaps the previous
    // launch: the producer before its first load, the epilogue before its
    // first scale load; the MMA issuer touches only
    // shared and tensor memory.  The grouped kernel's tile prefix reads the
    // offsets with the whole block, so it waits here.
    if constexpr (V == kGrouped) griddep_wait();
    int num_tiles = p.num_tiles;
    if constexpr (V == kGrouped)
        expert_tile_prefix<C::kThreads>(p.offsets, p.G, p.N / BN, s_prefix, s_prefix + kMaxGroups + 1);
    if constexpr (V == kGrouped) {
        __syncthreads();
        num_tiles = s_prefix[p.G];
    }
    if (threadIdx.x == 0) FP8BS_TRACE(1);

    using Iter = std::conditional_t<C::kSplitRegs, DpIter, SegIter>;
    Iter it;
    it.init(p, num_tiles);
    Seg sg;

    if (warp < 4) {
    // whole warpgroups change their register budgets: 0-3 give, 4-11 take
    if constexpr (C::kSplitRegs) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t iter = 0;
            bool ok = true;
#ifdef FP8BS_TRACE_ENABLED
            long long w_empty = 0;
#endif
            while (ok && it.next(sg)) {
                const Tile tg = tile_geom<BN, V>(p, sg.tile, s_prefix);
                for (int kb = sg.k0; kb < sg.k1; ++kb, ++iter) {
                    const int st = iter % S;
                    FP8BS_TIC(t0_);
                    if (!mbar_wait(&empty[st], ((iter / S) & 1) ^ 1, abort_flag)) {
                        set_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    FP8BS_TOC(w_empty, t0_);
                    if (iter == 0) {
                        griddep_wait();
                        FP8BS_TRACE(8);
                        FP8BS_TRACE(2);
                    }
                    mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                    tma_load_2d(sP + st * kPTileBytes, &tm_p, &full[st], kb * kBlock, tg.p_row0);
                    tma_load_2d(sQ + st * C::kQTileBytes, &tm_q, &full[st], kb * kBlock, tg.q_row0);
                }
            }
            FP8BS_TRACE_VAL(11, static_cast<unsigned long long>(w_empty));
            // drain: every load issued must land before the CTA may exit
            for (int st = 0; st < S && st < static_cast<int>(iter); ++st) {
                const uint32_t uses = iter / S + (static_cast<uint32_t>(st) < iter % S ? 1u : 0u);
                const volatile int never = 0;
                if (!mbar_wait(&full[st], (uses - 1) & 1, &never)) set_abort(abort_flag);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(128, BN);
            uint32_t iter = 0, slab = 0;
            bool ok = true;
#ifdef FP8BS_TRACE_ENABLED
            long long w_tempty = 0, w_full = 0;
#endif
            while (ok && it.next(sg)) {
                for (int kb = sg.k0; kb < sg.k1; ++kb, ++iter, ++slab) {
                    const int st = iter % S;
                    const int buf = slab & 1;
                    FP8BS_TIC(t1_);
                    FP8BS_TOC(w_tempty, t1_);
                    FP8BS_TIC(t2_);
                    // (the stage's barrier also carries the release of TMEM buffer `buf`)
                    const bool fu = mbar_wait(&full[st], (iter / S) & 1, abort_flag);
                    FP8BS_TOC(w_full, t2_);
                    if (!fu) {
                        set_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (iter == 0) FP8BS_TRACE(3);
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
                    const uint64_t da = smem_desc_sw128(smem_u32(sP + st * kPTileBytes));
                    const uint64_t db = smem_desc_sw128(smem_u32(sQ + st * C::kQTileBytes));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 4 x K=32 = one 128-K slab; +32 bytes each
                        mma_e4m3(d, da + 2 * kk, db + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                    mma_commit(&empty[st]);
                    // (a test of the failure path withholds slab 0's
                    // hand-off: the epilogue's wait must run out)
                    if (!(p.debug_skip && slab == 0)) mma_commit(&tfull[buf]);
                }
            }
            FP8BS_TRACE_VAL(12, static_cast<unsigned long long>(w_tempty));
            FP8BS_TRACE_VAL(13, static_cast<unsigned long long>(w_full));
            FP8BS_TRACE_VAL(14, static_cast<unsigned long long>(slab));
            mma_commit(mma_done);
            const volatile int never = 0;
            if (!mbar_wait(mma_done, 0, &never)) set_abort(abort_flag);
        }
    } else if constexpr (C::kGate) {
        // ---------------------------------------------------------- gate warps (2-3)
        // The expert body of each finished tile, while the epilogue warps
        // promote the next one: g = bf16(bf16(silu(h1)) * h3) from the
        // tile's bf16 h (h1 in columns 0-127, h3 in 128-255 of the same
        // 128-wide block of the intermediate dimension), then act_quant of
        // each row's 128 values.  Two rows per thread; the library's
        // silu*mul and quantisation routines, so the codes and scales equal
        // those of the unfused chain bit for bit.
        griddep_wait();   // before the first store of g
        const int gt = static_cast<int>(threadIdx.x) - 64;   // 0..63
        const int I = p.N / 2;
        uint32_t hn = 0;
        while (it.next(sg)) {
            const Tile tg = tile_geom<BN, V>(p, sg.tile, s_prefix);
            if (!mbar_wait(h_full, hn & 1, abort_flag)) {
                set_abort(abort_flag);
                break;
            }
            const int iblk = ((V == kGrouped) ? tg.q_col0 : tg.q_row0) / 256;
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int r = gt + 64 * pass;
                uint8_t* hrow = sStg + r * 512;
                // g over h1's place in the row (the row is this thread's alone)
                float amax = 0.0f;
#pragma unroll 4
                for (int c = 0; c < 16; ++c) {
                    // chunk c: eight columns of h1 (chunk c) and of h3 (chunk 16 + c)
                    uint4* pa = reinterpret_cast<uint4*>(hrow + ((c ^ (r & 7)) * 16));
                    const uint4 a = *pa;
                    const uint4 b = *reinterpret_cast<const uint4*>(hrow + (((16 + c) ^ (r & 7)) * 16));
                    const uint32_t u1[4] = {a.x, a.y, a.z, a.w}, u3[4] = {b.x, b.y, b.z, b.w};
                    uint32_t g[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        g[i] = silu_mul_bf16x2(__uint_as_float(u1[i] << 16), __uint_as_float(u1[i] & 0xFFFF0000u),
                                               __uint_as_float(u3[i] << 16), __uint_as_float(u3[i] & 0xFFFF0000u));
                        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(g[i] << 16)),
                                                 fabsf(__uint_as_float(g[i] & 0xFFFF0000u))));
                    }
                    *pa = make_uint4(g[0], g[1], g[2], g[3]);
                }
                const float sc = block_scale(amax, p.ue8m0 != 0);
                if (r < tg.p_valid) {
                    const int64_t row = static_cast<int64_t>(tg.p_row0) + r;
                    uint4* dst = reinterpret_cast<uint4*>(p.gq + row * I + iblk * 128);
#pragma unroll 2
                    for (int c = 0; c < 8; ++c) {   // 16 codes per store, from g chunks 2c and 2c + 1
                        uint2 qv[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 v = *reinterpret_cast<const uint4*>(hrow + (((2 * c + h) ^ (r & 7)) * 16));
                            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                            float f[8];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                f[2 * u] = __uint_as_float(w[u] << 16);
                                f[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
                            }
                            qv[h] = p.ue8m0 ? quant8<true>(f, sc) : quant8<false>(f, sc);
                        }
                        dst[c] = make_uint4(qv[0].x, qv[0].y, qv[1].x, qv[1].y);
                    }
                    p.gs[row * (I / 128) + iblk] = sc;
                }
            }
            mbar_arrive(h_empty);   // this thread's rows are done with
            ++hn;
        }
    }
    } else {
        if constexpr (C::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
        // ---------------------------------------------------------- epilogue
        griddep_wait();   // before its first scale load or output store
        constexpr int CPT = C::kCPT;
        const int q = warp & 3;                     // TMEM lane quarter
        const int e = q * 32 + lane;                // row of the tile (TMEM lane)
        const int cofs = ((warp - kEpiWarp0) >> 2) * CPT;   // first tile column of this thread
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        uint32_t slab = 0, epi_phase = 0;
        bool ok = true;
        // one finished slab: wait for it in TMEM, promote it, free the buffer
#ifdef FP8BS_TRACE_ENABLED
        long long w_tfull = 0, w_promote = 0, w_store = 0;
#endif
        // The buffer is handed back with one arrival per warp (a warp-wide
        // arrival is 32 barrier updates on the MMA warp's critical path).
        // Every lane takes its own bounded wait and then runs the
        // warp-collective loads whatever the outcome (a buffer read too early
        // only yields values that are discarded with the timeout status); the
        // warp votes once at the end, so its lanes always leave together.
        auto take_slab = [&](float (&acc)[CPT], const float* sc_col, float sc) -> bool {
            const int buf = slab & 1;
            FP8BS_TIC(t3_);
            const bool got = mbar_wait(&tfull[buf], (slab >> 1) & 1, abort_flag);
            FP8BS_TOC(w_tfull, t3_);
            tc_fence_after();
            if (slab == 0 && e == 0) FP8BS_TRACE(4);
            FP8BS_TIC(t4_);
            promote<CPT, false>(tmem_base + lane_off + static_cast<uint32_t>(buf * BN + cofs), acc, sc_col, sc);
            FP8BS_TOC(w_promote, t4_);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[(slab + 2) % S]);   // the buffer slab + 2 writes is free
            ++slab;
            if (!warp_all(got)) {
                set_abort(abort_flag);
                return false;
            }
            return true;
        };
        // per-row a_s and per-block b_s, prefetched PF slabs ahead in registers
        constexpr int PF = CPT >= 128 ? 4 : 8;   // prefetch distance (slabs)
        float cs[PF], na[PF], nb[PF];
        const float* ps = nullptr;
        const float* qs = nullptr;
        bool vec = false;
        int sk1 = 0;
        auto scale_rows = [&](const Tile& tg, const Seg& s) {
            ps = p.a_s + static_cast<int64_t>(e < tg.p_valid ? tg.p_row0 + e : 0) * p.KB;
            // (columns past N read the last block's scales; they are never stored)
            qs = (V == kDense) ? p.b_s + static_cast<int64_t>(min((tg.q_row0 + cofs) / 128, p.NB - 1)) * p.KB
                               : p.b_s + (static_cast<int64_t>(tg.group) * p.NB + (tg.q_col0 + cofs) / 128) * p.KB;
            // four slabs' scales per 16-byte load where the rows allow it
            vec = p.vec_scales && (s.k0 % 4) == 0;
            sk1 = s.k1;
        };
        auto load_next = [&](int base) {
#pragma unroll
            for (int i = 0; i < PF; i += 4) {
                if (vec && base + i + 4 <= sk1) {
                    const float4 va = __ldg(reinterpret_cast<const float4*>(ps + base + i));
                    const float4 vb = __ldg(reinterpret_cast<const float4*>(qs + base + i));
                    na[i] = va.x; na[i + 1] = va.y; na[i + 2] = va.z; na[i + 3] = va.w;
                    nb[i] = vb.x; nb[i + 1] = vb.y; nb[i + 2] = vb.z; nb[i + 3] = vb.w;
                } else {
#pragma unroll
                    for (int j = i; j < i + 4; ++j) {
                        const int kb = base + j;
                        na[j] = kb < sk1 ? __ldg(ps + kb) : 0.0f;
                        nb[j] = kb < sk1 ? __ldg(qs + kb) : 0.0f;
                    }
                }
            }
        };
        bool ahead = false;   // na/nb already hold this tile's first PF scales
        uint32_t hn = 0;      // gate kernels: tiles handed to the gate warps
        while (ok && it.next(sg)) {
            const Tile tg = tile_geom<BN, V>(p, sg.tile, s_prefix);
            float acc[CPT];
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
            if (!ahead) {
                scale_rows(tg, sg);
                load_next(sg.k0);
            }
#pragma unroll
            for (int i = 0; i < PF; ++i) cs[i] = na[i] * nb[i];
            load_next(sg.k0 + PF);
            for (int kc = sg.k0; kc < sg.k1 && ok; kc += PF) {
#pragma unroll
                for (int i = 0; i < PF; ++i) {
                    if (ok && kc + i < sg.k1) ok = take_slab(acc, nullptr, cs[i]);
                }
#pragma unroll
                for (int i = 0; i < PF; ++i) cs[i] = na[i] * nb[i];
                load_next(kc + 2 * PF);
            }
            ahead = false;
            // dense whole-tile schedule: fetch the next tile's first scales
            // now, so that their latency hides behind this tile's output
            // store (the grouped kernel measured slower with it)
            if constexpr (C::kSplitRegs && V == kDense) {
                Seg nx;
                if (ok && it.peek(nx)) {
                    scale_rows(tile_geom<BN, V>(p, nx.tile, s_prefix), nx);
                    load_next(nx.k0);
                    ahead = true;
                }
            }
            if (!ok) break;
            if (e == 0) FP8BS_TRACE(5);
            if (sg.k0 == 0 && sg.k1 == p.KB) {
                FP8BS_TIC(t5_);
                if constexpr (C::kGate) {
                    // hand the tile to the gate warps: row e's 128 columns of
                    // h (this thread's half: h1 or h3) as bf16, in 16-byte
                    // chunks whose order within each group of eight is
                    // swizzled by the row (conflict-free for both sides);
                    // first wait until the gate warps have read the last tile
                    // (the usual case, the gate warps long done, costs one
                    // try_wait; the bounded wait sits out of line so that
                    // its state does not compete with the accumulators)
                    bool hfree = mbar_try_wait(smem_u32(h_empty), (hn & 1) ^ 1);
                    if (!warp_all(hfree)) hfree = gate_wait_slow(h_empty, (hn & 1) ^ 1, abort_flag);
                    if (!warp_all(hfree)) {
                        set_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    const int half = (warp - kEpiWarp0) >> 2;
                    uint8_t* hrow = sStg + e * 512;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[8 * c + 2 * i], acc[8 * c + 2 * i + 1]);
                            w[i] = *reinterpret_cast<const uint32_t*>(&b);
                        }
                        *reinterpret_cast<uint4*>(hrow + (((half * 16 + c) ^ (e & 7)) * 16)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    mbar_arrive(h_full);
                    ++hn;
                    FP8BS_TOC(w_store, t5_);
                    continue;
                }
                if constexpr (C::kTmaStore) {
                    if (p.tma_store) {
                        const int col0 = ((V == kGrouped) ? tg.q_col0 : tg.q_row0) + cofs;
                        const int rest = store_tile_tma<CPT, C::kStgRows>(
                            &tm_c, sStg + (warp - kEpiWarp0) * (C::kStgRows * 128), lane, col0, tg.p_row0 + q * 32,
                            tg.p_valid - q * 32, tg.q_valid - cofs, acc);
                        // rows of a half the boxes left out (expert boundary): direct
                        if (lane >= rest) store_tile<BN, V, CPT>(p, tg, e, cofs, acc);
                        FP8BS_TOC(w_store, t5_);
                        continue;
                    }
                }
                store_tile<BN, V, CPT>(p, tg, e, cofs, acc);
                FP8BS_TOC(w_store, t5_);
                continue;
            }
            // ---- stream-K fixup: partial tile.  The 128x256 kernels only
            // ever run whole tiles (the host plans them so); compiled out there.
            if constexpr (C::kSplitRegs) {   // never planned for these
                set_abort(abort_flag);
                ok = false;
                break;
            } else {
            const long long U = p.total_units;
            const int P = gridDim.x;
            const long long u_first = static_cast<long long>(sg.tile) * p.KB;
            const int c_first = sk_owner(u_first, U, P);
            const int c_last = sk_owner(u_first + p.KB - 1, U, P);
            const int nseg = c_last - c_first + 1;
            auto slot_of = [&](int c) -> float* {
                const int first_tile = static_cast<int>(sk_start(c, U, P) / p.KB);
                const int which = (first_tile == sg.tile) ? 0 : 1;
                return p.partials + (static_cast<int64_t>(c) * 2 + which) * (128 * BN);
            };
            // partial tile layout: [row e][BN columns], 16-byte vectors per thread
            float* mine = slot_of(blockIdx.x) + e * BN + cofs;
#pragma unroll
            for (int j = 0; j < CPT; j += 4)
                __stcg(reinterpret_cast<float4*>(mine + j), make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]));
            __threadfence();
            if (!(ok = epi_sync(epi_bar, epi_phase, abort_flag))) break;
            if (e == 0) FP8BS_TRACE(9);
            if (e == 0 && cofs == 0) *ticket_box = atomicAdd(p.counters + sg.tile, 1);
            if (!(ok = epi_sync(epi_bar, epi_phase, abort_flag))) break;
            if (e == 0) FP8BS_TRACE(10);
            const int ticket = *ticket_box;
            if (!(ok = epi_sync(epi_bar, epi_phase, abort_flag))) break;
            if (ticket == nseg - 1) {
                __threadfence();
#pragma unroll
                for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
                // fixed summation order (segment 0, 1, ...): deterministic; each
                // batch keeps 8-16 vector loads in flight before adding them
                constexpr int kFloats = CPT <= 32 ? 32 : 64; // floats in flight per thread
                constexpr int CW = CPT < kFloats ? CPT : kFloats;  // columns per chunk
                constexpr int SB = kFloats / CW;                    // segments per batch
#pragma unroll
                for (int c0 = 0; c0 < CPT; c0 += CW) {
                    for (int s0 = 0; s0 < nseg; s0 += SB) {
                        float4 v[SB][CW / 4];
#pragma unroll
                        for (int b = 0; b < SB; ++b) {
                            if (s0 + b < nseg) {
                                const float4* src = reinterpret_cast<const float4*>(
                                    slot_of(c_first + s0 + b) + e * BN + cofs + c0);
#pragma unroll
                                for (int j = 0; j < CW / 4; ++j) v[b][j] = __ldcg(src + j);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < SB; ++b) {
                            if (s0 + b < nseg) {
#pragma unroll
                                for (int j = 0; j < CW / 4; ++j) {
                                    acc[c0 + 4 * j] += v[b][j].x;
                                    acc[c0 + 4 * j + 1] += v[b][j].y;
                                    acc[c0 + 4 * j + 2] += v[b][j].z;
                                    acc[c0 + 4 * j + 3] += v[b][j].w;
                                }
                            }
                        }
                    }
                }
                store_tile<BN, V, CPT>(p, tg, e, cofs, acc);
                if (e == 0 && cofs == 0) p.counters[sg.tile] = 0;
            }
            }
            if (e == 0) FP8BS_TRACE(6);
        }
#ifdef FP8BS_TRACE_ENABLED
        if (e == 0 && cofs == 0) {
            FP8BS_TRACE_VAL(15, static_cast<unsigned long long>(w_tfull));
            FP8BS_TRACE_VAL(16, static_cast<unsigned long long>(w_promote));
            FP8BS_TRACE_VAL(17, static_cast<unsigned long long>(w_store));
        }
#endif
        // the staging boxes must be read out before the CTA's shared memory goes
        if constexpr (C::kTmaStore) {
            if (lane == 0) bulk_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
    if (threadIdx.x == 0) FP8BS_TRACE(7);
}

// ------------------------------------------------------------------ ue8m0: block-scaled MMA
// When every scale is a power of two (scale_fmt ue8m0) the tensor core can
// apply the block scales itself: tcgen05.mma kind::mxf8f6f4 with one E8M0
// scale per 32 K values of each A row and each B column, read from tensor
// memory.  A 128-K block's scale is that scale for all four of its K=32
// steps.  A tile then accumulates over the whole of K in TMEM and its
// epilogue runs once, instead of promoting every 128-K slab in registers.
//
// 128x256 tiles, whole tiles per persistent CTA (m-fastest, as the dense
// kernel).  Warp 0: TMA producer; warp 1: MMA issuer; warps 2-5 (one per
// TMEM lane quarter): write each slab's scale factors into the TMEM slot of
// its pipeline stage, and run each tile's epilogue.  A stage's barrier
// counts the tiles' bytes and the four scale writers, so the MMA issuer
// checks one barrier per slab (each check by the issuing thread costs tensor
// time).  TMEM: the accumulator in columns [0, 256), the scale slot of stage
// s at 256 + 16 s (A's scales in its first 4 columns, B's in the next 8).
constexpr int kMxBN = 256;
constexpr int kMxStages = 4;
constexpr int kMxSfSlots = kMxStages;   // one scale slot per stage
constexpr int kMxThreads = 192;
constexpr int kMxSfCol0 = 256;
constexpr int kMxStageBytes = kPTileBytes + kMxBN * kBlock;   // A 16 KB + B 32 KB
constexpr int kMxStgBytes = 4 * 32 * 128;                     // per epilogue warp a 32 x 64 bf16 box
constexpr int kMxSmemBytes = 1024 + kMxStages * kMxStageBytes + kMxStgBytes + 1024;

// E8M0 code of a power-of-two fp32 scale (its biased exponent); `bad` is set
// for anything else (a mantissa, a sign, zero, a subnormal, inf or NaN).
__device__ __forceinline__ uint32_t e8m0_code(float s, bool& bad) {
    const uint32_t u = __float_as_uint(s);
    const uint32_t e = u >> 23;   // sign bit included: negative values land above 255
    bad |= (u & 0x7FFFFFu) != 0u || e == 0u || e >= 255u;
    return e & 0xFFu;
}

__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_c, const Params p) {
    constexpr int S = kMxStages, R = kMxSfSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                    // S x 16 KB
    uint8_t* sB = smem + S * kPTileBytes;                  // S x 32 KB
    uint8_t* sStg = smem + S * kMxStageBytes;              // 4 x 4 KB output staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kMxStgBytes);
    uint64_t* full = bars;                      // S: operand tiles landed and scales written
    uint64_t* empty = bars + S;                 // S: the MMAs have read them
    uint64_t* acc_full = bars + 2 * S;          // tile accumulated
    uint64_t* acc_empty = acc_full + 1;         // accumulator read out (4 warps)
    uint64_t* mma_done = acc_full + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1 + 4);   // the producer's bytes + the four scale writers
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        if (p.tma_store) tma_prefetch_desc(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (threadIdx.x == 64) griddep_launch_dependents();
    griddep_wait();

    // this CTA's tiles: blockIdx.x + i * gridDim.x
    const int my_tiles = static_cast<int>(blockIdx.x) < p.num_tiles
                             ? (p.num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                   static_cast<int>(gridDim.x)
                             : 0;
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    const uint32_t total = static_cast<uint32_t>(my_tiles) * KB;
    auto tile_of = [&](int ord) {
        return tile_geom<kMxBN, kDense>(p, static_cast<int>(blockIdx.x) + ord * static_cast<int>(gridDim.x),
                                        nullptr);
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t iter = 0;
            for (int ord = 0; ord < my_tiles && iter == static_cast<uint32_t>(ord) * KB; ++ord) {
                const Tile tg = tile_of(ord);
                for (uint32_t kb = 0; kb < KB; ++kb, ++iter) {
                    const int st = static_cast<int>(iter % S);
                    if (!mbar_wait(&empty[st], ((iter / S) & 1) ^ 1, abort_flag)) {
                        set_abort(abort_flag);
                        break;
                    }
                    mbar_arrive_expect_tx(&full[st], kMxStageBytes);
                    tma_load_2d(sA + st * kPTileBytes, &tm_a, &full[st], static_cast<int>(kb) * kBlock, tg.p_row0);
                    tma_load_2d(sB + st * (kMxBN * kBlock), &tm_b, &full[st], static_cast<int>(kb) * kBlock,
                                tg.q_row0);
                }
            }
            // every load issued must land before the CTA may exit
            const volatile int never = 0;
            for (int st = 0; st < S && st < static_cast<int>(iter); ++st) {
                const uint32_t uses = iter / S + (static_cast<uint32_t>(st) < iter % S ? 1u : 0u);
                if (!mbar_wait(&full[st], (uses - 1) & 1, &never)) set_abort(abort_flag);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t iter = 0;
            bool ok = true;
            for (int ord = 0; ok && ord < my_tiles; ++ord) {
                if (!mbar_wait(acc_empty, (static_cast<uint32_t>(ord) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (uint32_t kb = 0; kb < KB; ++kb, ++iter) {
                    const int st = static_cast<int>(iter % S);
                    if (!mbar_wait(&full[st], (iter / S) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(smem_u32(sA + st * kPTileBytes));
                    const uint64_t db = smem_desc_sw128(smem_u32(sB + st * (kMxBN * kBlock)));
                    const uint32_t sfa = tmem_base + static_cast<uint32_t>(kMxSfCol0 + 16 * st);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 4 x K=32, each with its byte of the scale words
                        mma_mx_e4m3(tmem_base, da + 2 * kk, db + 2 * kk, idesc_mx_e4m3(128, kMxBN, kk), sfa, sfa + 4,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[st]);
                }
                if (!ok) break;
                mma_commit(acc_full);
            }
            if (!ok) set_abort(abort_flag);
            mma_commit(mma_done);
            const volatile int never = 0;
            if (!mbar_wait(mma_done, 0, &never)) set_abort(abort_flag);
        }
    } else {
        // ---------------------------------------------------------- scales + epilogue
        const int q = warp & 3;                        // TMEM lane quarter
        const int e = q * 32 + lane;                   // tile row
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = sStg + (warp - 2) * (32 * 128);
        bool bad = false, ok = true;
        // scales of 4 slabs at a time (16-byte loads), the next group loaded
        // while the current one is written
        float4 ca{}, cb0{}, cb1{}, na{}, nb0{}, nb1{};
        auto load_group = [&](uint32_t slab, float4& a4, float4& b04, float4& b14) {
            if (slab >= total) return;
            const Tile tg = tile_of(static_cast<int>(slab / KB));
            const uint32_t kb = slab % KB;
            const int row = tg.p_row0 + min(e, max(tg.p_valid, 1) - 1);   // rows past M repeat a valid one
            const int nb = tg.q_row0 / 128;
            a4 = __ldg(reinterpret_cast<const float4*>(p.a_s + static_cast<int64_t>(row) * KB + kb));
            b04 = __ldg(reinterpret_cast<const float4*>(p.b_s + static_cast<int64_t>(nb) * KB + kb));
            b14 = __ldg(reinterpret_cast<const float4*>(p.b_s + static_cast<int64_t>(min(nb + 1, p.NB - 1)) * KB + kb));
        };
        load_group(0, na, nb0, nb1);
        uint32_t iter = 0;   // slabs whose scales are written
        for (int te = 0; ok && te < my_tiles; ++te) {
            // scales up to kMxSfSlots slabs into the next tile (their slots
            // were last read by this tile's MMAs, which need nothing more)
            const uint32_t limit = min(total, static_cast<uint32_t>(te + 1) * KB + min(KB, static_cast<uint32_t>(R)));
            for (; iter < limit; ++iter) {
                // KB % 4 == 0: a group of 4 slabs never straddles two tiles
                if (iter % 4 == 0) {
                    ca = na;
                    cb0 = nb0;
                    cb1 = nb1;
                    load_group(iter + 4, na, nb0, nb1);
                }
                const int j = static_cast<int>(iter % 4);
                const float sa = j == 0 ? ca.x : j == 1 ? ca.y : j == 2 ? ca.z : ca.w;
                const float s0 = j == 0 ? cb0.x : j == 1 ? cb0.y : j == 2 ? cb0.z : cb0.w;
                const float s1 = j == 0 ? cb1.x : j == 1 ? cb1.y : j == 2 ? cb1.z : cb1.w;
                const uint32_t wa = e8m0_code(sa, bad) * 0x01010101u;
                const uint32_t w0 = e8m0_code(s0, bad) * 0x01010101u;
                const uint32_t w1 = e8m0_code(s1, bad) * 0x01010101u;
                // the stage's slot is free once the MMAs of its previous slab are done
                const int r = static_cast<int>(iter % R);
                if (!warp_all(mbar_wait(&empty[r], ((iter / R) & 1) ^ 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = tmem_base + lane_off + static_cast<uint32_t>(kMxSfCol0 + 16 * r);
                tmem_st4(col, wa, wa, wa, wa);   // row e's scale in column e/32 (the others unused)
                tmem_st8(col + 4, w0, w1);        // columns n/32: n < 128 in the first four
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[r]);
            }
            if (!ok) break;
            // epilogue of tile te
            if (!warp_all(mbar_wait(acc_full, static_cast<uint32_t>(te) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const Tile tg = tile_of(te);
            const int row0 = tg.p_row0 + q * 32;
            const int64_t row = tg.p_row0 + e;
            if (p.tma_store) {
                // bf16 only: read the whole row out of TMEM as packed bf16
                // (128 registers), hand the accumulator back to the MMA, then
                // stage and store while the next tile accumulates
                uint32_t pk[kMxBN / 2];
#pragma unroll
                for (int h = 0; h < kMxBN / 64; ++h) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h), r0);
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h + 32), r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        __nv_bfloat162 v0 = __floats2bfloat162_rn(__uint_as_float(r0[2 * c]), __uint_as_float(r0[2 * c + 1]));
                        __nv_bfloat162 v1 = __floats2bfloat162_rn(__uint_as_float(r1[2 * c]), __uint_as_float(r1[2 * c + 1]));
                        pk[32 * h + c] = *reinterpret_cast<uint32_t*>(&v0);
                        pk[32 * h + 16 + c] = *reinterpret_cast<uint32_t*>(&v1);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                // 32 rows x 64 columns per box, 128-byte swizzle (16-byte chunk
                // c of row r at c ^ (r % 8)); the TMA unit clips at M and N
#pragma unroll
                for (int h = 0; h < kMxBN / 64; ++h) {
                    const int col0 = tg.q_row0 + 64 * h;
                    if (col0 >= p.N || tg.p_valid - q * 32 <= 0) break;
                    if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                    __syncwarp();
                    uint8_t* srow = stg + lane * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(srow + ((c ^ (lane & 7)) * 16)) =
                            make_uint4(pk[32 * h + 4 * c], pk[32 * h + 4 * c + 1], pk[32 * h + 4 * c + 2],
                                       pk[32 * h + 4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_c, stg, col0, row0);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll 1
                for (int h = 0; h < kMxBN / 64; ++h) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h), r0);
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h + 32), r1);
                    tmem_wait_ld();
                    const int col0 = tg.q_row0 + 64 * h;
                    const int cols = min(64, p.N - col0);
                    if (cols > 0 && e < tg.p_valid) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            if (c < cols) {
                                const float v = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
                                if (p.c_bf16) p.c_bf16[row * p.N + col0 + c] = __float2bfloat16_rn(v);
                                if (p.c_fp32) p.c_fp32[row * p.N + col0 + c] = v;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
        }
        if (!ok) set_abort(abort_flag);
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicExch(&g_gemm_status, static_cast<int>(FP8_ERR_INVALID_ARG));
        if (lane == 0) bulk_wait_all();   // staging boxes read out before shared memory goes
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// The same product on CTA pairs (thread-block clusters of 2 on two SMs):
// one 256x256 output tile per pair and tcgen05.mma.cta_group::2 of M = 256,
// issued by the leader, twice the work per MMA (and per barrier check) of
// the 1-SM form.  Each CTA stages its own 128 rows of A and its half of the
// B tile (32 KB per slab), so six stages fit; each writes the scales its own
// TMEM must hold (its 128 A rows; all 256 B columns) into its stage's slot
// and runs the epilogue of its 128 rows.  The leader's stage barrier counts
// both CTAs' tile bytes and all eight scale writers, so the issuer checks
// one barrier per slab; the MMA's commits reach both CTAs.
constexpr int kMx2Stages = 6;
constexpr int kMx2StageBytes = 2 * kPTileBytes;   // A 128 rows + B 128 rows
constexpr int kMx2SmemBytes = 1024 + kMx2Stages * kMx2StageBytes + kMxStgBytes + 1024;

__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const Params p) {
    constexpr int S = kMx2Stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                    // S x 16 KB
    uint8_t* sB = smem + S * kPTileBytes;                  // S x 16 KB
    uint8_t* sStg = smem + S * kMx2StageBytes;             // 4 x 4 KB output staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kMxStgBytes);
    uint64_t* full = bars;                      // S (leader): both CTAs' tiles landed and scales written
    uint64_t* empty = bars + S;                 // S: the pair's MMAs have read the stage
    uint64_t* acc_full = bars + 2 * S;          // tile accumulated
    uint64_t* acc_empty = acc_full + 1;         // (leader) both accumulators read out (8 warps)
    uint64_t* mma_done = acc_full + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1 + 8);   // the leader's producer (with both CTAs' bytes) + 8 scale writers
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        if (p.tma_store) tma_prefetch_desc(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers exist before either arrives on the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (threadIdx.x == 64) griddep_launch_dependents();
    griddep_wait();

    // this pair's tiles (256 x 256): cluster c takes c + i * clusters, m-fastest
    const int cid = static_cast<int>(blockIdx.x >> 1), nclus = static_cast<int>(gridDim.x >> 1);
    const int my_tiles = cid < p.num_tiles ? (p.num_tiles - cid + nclus - 1) / nclus : 0;
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    const uint32_t total = static_cast<uint32_t>(my_tiles) * KB;
    struct PT {
        int m0, valid, n0;   // this CTA's first row and its rows inside M; the pair's first column
    };
    auto tile_of = [&](int ord) {
        const int t = cid + ord * nclus;
        const int tp = t % p.tiles_p, tq = t / p.tiles_p;
        PT g;
        g.m0 = tp * 256 + static_cast<int>(rank) * 128;
        g.valid = min(128, p.M - g.m0);
        g.n0 = tq * 256;
        return g;
    };
    auto leader = [&](uint64_t* bar) { return cluster_map(smem_u32(bar), 0); };

    if (warp == 0) {
        // ---------------------------------------------------------- producer (each CTA)
        if (lane == 0) {
            uint32_t iter = 0;
            bool ok = true;
            for (int ord = 0; ok && ord < my_tiles; ++ord) {
                const PT tg = tile_of(ord);
                for (uint32_t kb = 0; kb < KB; ++kb, ++iter) {
                    const int st = static_cast<int>(iter % S);
                    if (!mbar_wait_cluster(&empty[st], ((iter / S) & 1) ^ 1, abort_flag)) {
                        set_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * kMx2StageBytes);
                    const uint32_t fb = leader(&full[st]);
                    tma_load_2d_pair(sA + st * kPTileBytes, &tm_a, fb, static_cast<int>(kb) * kBlock, tg.m0);
                    tma_load_2d_pair(sB + st * kPTileBytes, &tm_b, fb, static_cast<int>(kb) * kBlock,
                                     tg.n0 + static_cast<int>(rank) * 128);
                }
            }
            // the leader's barriers count both CTAs' loads: it waits for every
            // stage it armed before the pair may end
            if (rank == 0) {
                const volatile int never = 0;
                for (int st = 0; st < S && st < static_cast<int>(iter); ++st) {
                    const uint32_t uses = iter / S + (static_cast<uint32_t>(st) < iter % S ? 1u : 0u);
                    if (!mbar_wait_cluster(&full[st], (uses - 1) & 1, &never)) set_abort(abort_flag);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer (leader)
        if (lane == 0 && rank == 0) {
            uint32_t iter = 0;
            bool ok = true;
            for (int ord = 0; ok && ord < my_tiles; ++ord) {
                if (!mbar_wait_cluster(acc_empty, (static_cast<uint32_t>(ord) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (uint32_t kb = 0; kb < KB; ++kb, ++iter) {
                    const int st = static_cast<int>(iter % S);
                    if (!mbar_wait_cluster(&full[st], (iter / S) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(smem_u32(sA + st * kPTileBytes));
                    const uint64_t db = smem_desc_sw128(smem_u32(sB + st * kPTileBytes));
                    const uint32_t sfa = tmem_base + static_cast<uint32_t>(kMxSfCol0 + 16 * st);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mx_e4m3_pair(tmem_base, da + 2 * kk, db + 2 * kk, idesc_mx_e4m3(256, 256, kk), sfa,
                                         sfa + 4, (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair(&empty[st]);
                }
                if (!ok) break;
                mma_commit_pair(acc_full);
            }
            if (!ok) set_abort(abort_flag);
            mma_commit_pair(mma_done);
            const volatile int never = 0;
            if (!mbar_wait_cluster(mma_done, 0, &never)) set_abort(abort_flag);
        }
    } else {
        // ---------------------------------------------------------- scales + epilogue (each CTA)
        const int q = warp & 3;
        const int e = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = sStg + (warp - 2) * (32 * 128);
        bool bad = false, ok = true;
        float4 ca{}, cb0{}, cb1{}, na{}, nb0{}, nb1{};
        auto load_group = [&](uint32_t slab, float4& a4, float4& b04, float4& b14) {
            if (slab >= total) return;
            const PT tg = tile_of(static_cast<int>(slab / KB));
            const uint32_t kb = slab % KB;
            const int row = tg.valid > 0 ? tg.m0 + min(e, tg.valid - 1) : 0;   // rows past M repeat a valid one
            const int nb = tg.n0 / 128;
            a4 = __ldg(reinterpret_cast<const float4*>(p.a_s + static_cast<int64_t>(row) * KB + kb));
            b04 = __ldg(reinterpret_cast<const float4*>(p.b_s + static_cast<int64_t>(min(nb, p.NB - 1)) * KB + kb));
            b14 = __ldg(reinterpret_cast<const float4*>(p.b_s + static_cast<int64_t>(min(nb + 1, p.NB - 1)) * KB + kb));
        };
        load_group(0, na, nb0, nb1);
        const uint32_t full_l0 = leader(&full[0]);
        const uint32_t acc_empty_l = leader(acc_empty);
        uint32_t iter = 0;
        for (int te = 0; ok && te < my_tiles; ++te) {
            // scales up to S slabs into the next tile (their slots were last
            // read by this tile's MMAs, which need nothing more)
            const uint32_t limit = min(total, static_cast<uint32_t>(te + 1) * KB + min(KB, static_cast<uint32_t>(S)));
            for (; iter < limit; ++iter) {
                if (iter % 4 == 0) {   // KB % 4 == 0: a group never straddles two tiles
                    ca = na;
                    cb0 = nb0;
                    cb1 = nb1;
                    load_group(iter + 4, na, nb0, nb1);
                }
                const int j = static_cast<int>(iter % 4);
                const float sa = j == 0 ? ca.x : j == 1 ? ca.y : j == 2 ? ca.z : ca.w;
                const float s0 = j == 0 ? cb0.x : j == 1 ? cb0.y : j == 2 ? cb0.z : cb0.w;
                const float s1 = j == 0 ? cb1.x : j == 1 ? cb1.y : j == 2 ? cb1.z : cb1.w;
                const uint32_t wa = e8m0_code(sa, bad) * 0x01010101u;
                const uint32_t w0 = e8m0_code(s0, bad) * 0x01010101u;
                const uint32_t w1 = e8m0_code(s1, bad) * 0x01010101u;
                // the stage's slot is free once the pair's MMAs of its previous slab are done
                const int r = static_cast<int>(iter % S);
                if (!warp_all(mbar_wait_cluster(&empty[r], ((iter / S) & 1) ^ 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = tmem_base + lane_off + static_cast<uint32_t>(kMxSfCol0 + 16 * r);
                tmem_st4(col, wa, wa, wa, wa);
                tmem_st8(col + 4, w0, w1);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(full_l0 + static_cast<uint32_t>(r * 8));
            }
            if (!ok) break;
            if (!warp_all(mbar_wait_cluster(acc_full, static_cast<uint32_t>(te) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const PT tg = tile_of(te);
            const int row0 = tg.m0 + q * 32;
            const int64_t row = tg.m0 + e;
            if (p.tma_store) {
                uint32_t pk[128];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h), r0);
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h + 32), r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        __nv_bfloat162 v0 = __floats2bfloat162_rn(__uint_as_float(r0[2 * c]), __uint_as_float(r0[2 * c + 1]));
                        __nv_bfloat162 v1 = __floats2bfloat162_rn(__uint_as_float(r1[2 * c]), __uint_as_float(r1[2 * c + 1]));
                        pk[32 * h + c] = *reinterpret_cast<uint32_t*>(&v0);
                        pk[32 * h + 16 + c] = *reinterpret_cast<uint32_t*>(&v1);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(acc_empty_l);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int col0 = tg.n0 + 64 * h;
                    if (col0 >= p.N || tg.valid - q * 32 <= 0) break;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    uint8_t* srow = stg + lane * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(srow + ((c ^ (lane & 7)) * 16)) =
                            make_uint4(pk[32 * h + 4 * c], pk[32 * h + 4 * c + 1], pk[32 * h + 4 * c + 2],
                                       pk[32 * h + 4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_c, stg, col0, row0);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll 1
                for (int h = 0; h < 4; ++h) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h), r0);
                    tmem_ld32(tmem_base + lane_off + static_cast<uint32_t>(64 * h + 32), r1);
                    tmem_wait_ld();
                    const int col0 = tg.n0 + 64 * h;
                    const int cols = min(64, p.N - col0);
                    if (cols > 0 && e < tg.valid) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            if (c < cols) {
                                const float v = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
                                if (p.c_bf16) p.c_bf16[row * p.N + col0 + c] = __float2bfloat16_rn(v);
                                if (p.c_fp32) p.c_fp32[row * p.N + col0 + c] = v;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(acc_empty_l);
            }
        }
        if (!ok) set_abort(abort_flag);
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicExch(&g_gemm_status, static_cast<int>(FP8_ERR_INVALID_ARG));
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    cluster_sync_all();   // the peer's shared memory and TMEM stay until the pair's last MMA is done
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

}  // namespace

// ------------------------------------------------------------------ host side
// Tensor-map helpers, shared with the decode kernels (decode.cu).
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D map over a bf16 matrix [rows, K] (row stride 2K bytes), box 64 x box_rows
// (128-byte rows), 128-byte swizzle.
bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over an e4m3 matrix [rows, K] (row stride K bytes), box 128 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlock), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

bool wide_tiles_ok();

// Schedule of the dense kernel (M > 64; smaller batches run on the decode
// kernel): 128x256 tiles per persistent CTA when there are plenty of them,
// else 128x128 tiles, as whole tiles or as a stream-K split of (tile, slab)
// units when there are few.
struct Plan {
    int bn;
    int tiles_p, tiles_q, num_tiles;
    int stream_k;
    int grid;
    long long total_units;
    size_t ws_bytes;   // counters + partial slots
    size_t counters_bytes;
};

Plan make_plan(int64_t M, int64_t N, int64_t K, int sms) {
    Plan pl{};
    const int KB = static_cast<int>(K / kBlock);
    pl.bn = 128;
    pl.tiles_p = static_cast<int>((M + 127) / 128);
    pl.tiles_q = static_cast<int>((N + 127) / 128);
    // enough 128x256 tiles for whole-tile scheduling: use the wide tile
    const long long wide = static_cast<long long>(pl.tiles_p) * ((N + 255) / 256);
    if (wide >= 4LL * sms && wide <= (1LL << 30) && KB > 1 && wide_tiles_ok()) {
        pl.bn = 256;
        pl.tiles_q = static_cast<int>((N + 255) / 256);
    }
    pl.num_tiles = pl.tiles_p * pl.tiles_q;
    pl.total_units = static_cast<long long>(pl.num_tiles) * KB;
    if (pl.num_tiles >= 4 * sms || pl.num_tiles > kMaxSkTiles || KB == 1) {
        pl.stream_k = 0;
        pl.grid = static_cast<int>(std::min<long long>(pl.num_tiles, sms));
        pl.ws_bytes = 0;
    } else {
        pl.stream_k = 1;
        // at least 2 slabs per CTA so the pipeline has something to overlap,
        // and at most ~8 CTAs sharing one tile so its reduction stays short
        long long g = std::min<long long>(sms, std::max<long long>(1, pl.total_units / 2));
        g = std::min<long long>(g, std::max<long long>(1, 8LL * pl.num_tiles));
        pl.grid = static_cast<int>(g);
        pl.counters_bytes = kCounterBytes;
        pl.ws_bytes = pl.counters_bytes + static_cast<size_t>(pl.grid) * 2 * 128 * pl.bn * 4;
    }
    return pl;
}

template <int BN, int V, bool SW = false>
cudaError_t launch(const CUtensorMap& mp, const CUtensorMap& mq, const CUtensorMap& mc, const Params& prm,
                   int grid, cudaStream_t st) {
    using C = Cfg<BN, V, SW>;
    constexpr int smem = C::kSmemBytes;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, V, SW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return launch_pdl(gemm_kernel<BN, V, SW>, dim3(grid), dim3(C::kThreads), smem, st, mp, mq, mc, prm);
}

// The 128x256 kernels move registers between warpgroups with setmaxnreg;
// that is only safe if the kernel was built with the register count the
// split assumes (launch total >= the sum of the new per-warpgroup counts).
template <int V, bool SW>
bool split_regs_ok() {
    using C = Cfg<256, V, SW>;
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, gemm_kernel<256, V, SW>) != cudaSuccess) return false;
    return a.numRegs * C::kThreads >= C::kRegsLow * 128 + C::kRegsHigh * 32 * C::kEpiWarps;
}

bool wide_tiles_ok() {
    static int cache[64] = {0};   // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return false;
    if (cache[dev] == 0)
        cache[dev] = (split_regs_ok<kDense, false>() && split_regs_ok<kGrouped, false>() &&
                      split_regs_ok<kDense, true>() && split_regs_ok<kGrouped, true>())
                         ? 1
                         : 2;
    return cache[dev] == 1;
}

}  // namespace

int gemm_read_and_clear_status(cudaStream_t st) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_gemm_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_gemm_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return -1;
        if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace fp8bs

using namespace fp8bs;

#ifdef FP8BS_TRACE_ENABLED
static int g_trace_next = 0;
extern "C" int fp8_debug_clear_trace(void) {
    static unsigned long long zero[4][512][24];
    g_trace_next = 0;
    return cudaMemcpyToSymbol(g_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
extern "C" int fp8_debug_read_trace(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * 4 * 512 * 24) == cudaSuccess ? 0 : 1;
}
#endif

namespace fp8bs {
// decode.cu: the M <= 64 path of fp8_gemm (xq, a_s) and fp8_linear (x)
fp8_status decode_gemm(const void* x, const void* xq, const float* a_s, const void* w, const float* b_s,
                       void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K, int ue8m0, int debug_skip,
                       cudaStream_t st);
bool decode_set_wait_limit(long long cycles);
}  // namespace fp8bs

// Test hooks of the failure path (see fp8_debug_skip_one_arrive).
static std::atomic<int> g_debug_skip_next{0};

extern "C" fp8_status fp8_debug_set_wait_limit(long long cycles) {
    const long long v = cycles > 0 ? cycles : kWaitLimitCycles;
    if (cudaMemcpyToSymbol(g_wait_limit_cycles, &v, sizeof(v)) != cudaSuccess) return FP8_ERR_CUDA;
    return decode_set_wait_limit(v) ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" void fp8_debug_skip_one_arrive(void) { g_debug_skip_next.store(1); }

extern "C" size_t fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % kBlock != 0) return 0;
    if (M <= kDecodeMaxM) return 0;   // the decode kernel reduces on chip
    return make_plan(M, N, K, device_sm_count()).ws_bytes;
}

namespace {
// fp8_gemm's argument checks, shared with fp8_gemm_noalloc so that a call
// either of them rejects touches nothing on the device.  FP8_OK with M == 0
// or N == 0 means there is nothing to do.
fp8_status gemm_check_args(const void* a, const float* a_s, const void* b, const float* b_s, const void* c_bf16,
                           const float* c_fp32, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K <= 0 || K % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    if (!a || !a_s || !b || !b_s || (!c_bf16 && !c_fp32)) return FP8_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b)) return FP8_ERR_INVALID_ARG;
    if ((c_bf16 && (reinterpret_cast<uintptr_t>(c_bf16) & 1)) ||
        (c_fp32 && (reinterpret_cast<uintptr_t>(c_fp32) & 3)))
        return FP8_ERR_INVALID_ARG;
    if (N % 8 == 0 && ((c_bf16 && !aligned16(c_bf16)) || (c_fp32 && !aligned16(c_fp32))))
        return FP8_ERR_INVALID_ARG;
    return FP8_OK;
}
}  // namespace

extern "C" fp8_status fp8_gemm(const void* a, const float* a_s, const void* b, const float* b_s,
                               void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K,
                               void* workspace, size_t workspace_bytes, void* stream) {
    const fp8_status chk = gemm_check_args(a, a_s, b, b_s, c_bf16, c_fp32, M, N, K);
    if (chk != FP8_OK || M == 0 || N == 0) return chk;
    if (M <= kDecodeMaxM)
        return decode_gemm(nullptr, a, a_s, b, b_s, c_bf16, c_fp32, M, N, K, 0, g_debug_skip_next.exchange(0),
                           static_cast<cudaStream_t>(stream));
    const Plan pl = make_plan(M, N, K, device_sm_count());
    if (pl.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pl.ws_bytes))
        return FP8_ERR_WORKSPACE;

    Params prm{};
    prm.a_s = a_s;
    prm.b_s = b_s;
    prm.c_bf16 = static_cast<__nv_bfloat16*>(c_bf16);
    prm.c_fp32 = c_fp32;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.KB = static_cast<int>(K / kBlock);
    prm.NB = static_cast<int>((N + 127) / 128);
    prm.G = 1;
    prm.tiles_p = pl.tiles_p;
    prm.tiles_q = pl.tiles_q;
    prm.num_tiles = pl.num_tiles;
    prm.stream_k = pl.stream_k;
    prm.total_units = pl.total_units;
    prm.vec_scales = (prm.KB % 4 == 0 && aligned16(a_s) && aligned16(b_s)) ? 1 : 0;
    prm.debug_skip = g_debug_skip_next.exchange(0);
#ifdef FP8BS_TRACE_ENABLED
    prm.trace_slot = g_trace_next++ & 3;
#endif
    if (pl.ws_bytes > 0) {
        prm.counters = static_cast<int*>(workspace);
        prm.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.counters_bytes);
    }
    CUtensorMap mp, mq, mc;
    // P: 128-row tiles of the activations; Q: BN-row tiles of the weight
    if (!make_map(&mp, a, M, K, 128) || !make_map(&mq, b, N, K, pl.bn)) return FP8_ERR_CUDA;
    // C (bf16 only, 16-byte rows): staging-box-high x 64 boxes for the TMA tile store
    prm.tma_store = (c_bf16 && !c_fp32 && N % 8 == 0) ? 1 : 0;
    const int box_rows = pl.bn == 256 ? Cfg<256, kDense>::kStgRows : Cfg<128, kDense>::kStgRows;
    if (prm.tma_store && !make_map_bf16(&mc, c_bf16, M, N, box_rows)) return FP8_ERR_CUDA;
    if (!prm.tma_store) mc = mp;   // not read
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = pl.bn == 256 ? launch<256, kDense>(mp, mq, mc, prm, pl.grid, st)
                                       : launch<128, kDense>(mp, mq, mc, prm, pl.grid, st);
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_gemm_ue8m0(const void* a, const float* a_s, const void* b, const float* b_s,
                                     void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K, void* stream) {
    if (M < 0 || N < 0 || K <= 0 || K % (4 * kBlock) != 0) return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    if (!a || !a_s || !b || !b_s || (!c_bf16 && !c_fp32)) return FP8_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(a_s) || !aligned16(b_s)) return FP8_ERR_INVALID_ARG;
    if ((c_bf16 && (reinterpret_cast<uintptr_t>(c_bf16) & 1)) ||
        (c_fp32 && (reinterpret_cast<uintptr_t>(c_fp32) & 3)))
        return FP8_ERR_INVALID_ARG;
    if (N % 8 == 0 && ((c_bf16 && !aligned16(c_bf16)) || (c_fp32 && !aligned16(c_fp32))))
        return FP8_ERR_INVALID_ARG;
    Params prm{};
    prm.a_s = a_s;
    prm.b_s = b_s;
    prm.c_bf16 = static_cast<__nv_bfloat16*>(c_bf16);
    prm.c_fp32 = c_fp32;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.KB = static_cast<int>(K / kBlock);
    prm.NB = static_cast<int>((N + 127) / 128);
    prm.G = 1;
    // CTA pairs (256 x 256 tiles) once there are enough of them to give
    // every SM a tile; else one SM per 128 x 256 tile
    const int sms = device_sm_count();
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + kMxBN - 1) / kMxBN);
    const bool pairs = pair_tiles >= sms / 2 && sms >= 2;
    prm.tiles_p = static_cast<int>(pairs ? (M + 255) / 256 : (M + 127) / 128);
    prm.tiles_q = static_cast<int>((N + kMxBN - 1) / kMxBN);
    const int64_t tiles = static_cast<int64_t>(prm.tiles_p) * prm.tiles_q;
    if (tiles > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    prm.num_tiles = static_cast<int>(tiles);
    CUtensorMap ma, mb, mc;
    if (!make_map(&ma, a, M, K, 128) || !make_map(&mb, b, N, K, pairs ? 128 : kMxBN)) return FP8_ERR_CUDA;
    prm.tma_store = (c_bf16 && !c_fp32 && N % 8 == 0) ? 1 : 0;
    if (prm.tma_store && !make_map_bf16(&mc, c_bf16, M, N, 32)) return FP8_ERR_CUDA;
    if (!prm.tma_store) mc = ma;   // not read
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    static int configured[64][2] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev][pairs ? 1 : 0]) {
        const cudaError_t a1 =
            pairs ? cudaFuncSetAttribute(gemm_mx2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMx2SmemBytes)
                  : cudaFuncSetAttribute(gemm_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmemBytes);
        if (a1 != cudaSuccess) return FP8_ERR_CUDA;
        configured[dev][pairs ? 1 : 0] = 1;
    }
    cudaError_t e;
    if (pairs) {
        const int grid = 2 * static_cast<int>(std::min<int64_t>(tiles, sms / 2));
        e = launch_pdl_cluster(gemm_mx2_kernel, dim3(grid), dim3(kMxThreads), kMx2SmemBytes, st, 2u, ma, mb, mc, prm);
    } else {
        const int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
        e = launch_pdl_cluster(gemm_mx_kernel, dim3(grid), dim3(kMxThreads), kMxSmemBytes, st, 1u, ma, mb, mc, prm);
    }
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_grouped_gemm(const void* a, const float* a_s, const void* b,
                                       const float* b_s, const int32_t* offsets, int32_t G,
                                       int64_t R_max, void* c_bf16, float* c_fp32, int64_t N,
                                       int64_t K, void* stream) {
    if (G < 0 || G > kMaxGroups || R_max < 0 || N < 0 || K <= 0 || K % kBlock != 0)
        return FP8_ERR_INVALID_ARG;
    if (G == 0 || R_max == 0 || N == 0) return FP8_OK;
    if (N % 128 != 0) return FP8_ERR_INVALID_ARG;
    if (static_cast<int64_t>(G) * N > (1LL << 31) - 1 || R_max > (1LL << 31) - 1)
        return FP8_ERR_UNSUPPORTED;
    if (!a || !a_s || !b || !b_s || !offsets || (!c_bf16 && !c_fp32)) return FP8_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || (c_bf16 && !aligned16(c_bf16)) ||
        (c_fp32 && !aligned16(c_fp32)))
        return FP8_ERR_INVALID_ARG;
    Params prm{};
    prm.a_s = a_s;
    prm.b_s = b_s;
    prm.offsets = offsets;
    prm.c_bf16 = static_cast<__nv_bfloat16*>(c_bf16);
    prm.c_fp32 = c_fp32;
    prm.M = static_cast<int>(R_max);
    prm.N = static_cast<int>(N);
    prm.KB = static_cast<int>(K / kBlock);
    prm.NB = static_cast<int>(N / 128);
    prm.G = G;
    prm.stream_k = 0;
    prm.vec_scales = (prm.KB % 4 == 0 && aligned16(a_s) && aligned16(b_s)) ? 1 : 0;
    const bool wide = (N % 256 == 0) && wide_tiles_ok();
    CUtensorMap mp, mq, mc;
    if (!make_map(&mp, a, R_max, K, 128) ||
        !make_map(&mq, b, static_cast<int64_t>(G) * N, K, wide ? 256 : 128))
        return FP8_ERR_CUDA;
    // bf16-only output: 16 x 64 boxes for the TMA tile store
    prm.tma_store = (c_bf16 && !c_fp32) ? 1 : 0;
    if (prm.tma_store && !make_map_bf16(&mc, c_bf16, R_max, N, 16)) return FP8_ERR_CUDA;
    if (!prm.tma_store) mc = mp;   // not read
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = wide ? launch<256, kGrouped>(mp, mq, mc, prm, device_sm_count(), st)
                         : launch<128, kGrouped>(mp, mq, mc, prm, device_sm_count(), st);
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ------------------------------------------------------------------ expert body fused into w1|w3
namespace {
fp8_status swiglu_check(int64_t M, int64_t I, int64_t K, int scale_fmt) {
    if (M < 0 || I <= 0 || K <= 0 || K % kBlock != 0 || I % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (M > (1LL << 31) - 1 || 2 * I > (1LL << 31) - 1 || K > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    return FP8_OK;
}
}  // namespace

extern "C" fp8_status fp8_gemm_swiglu(const void* a, const float* a_s, const void* w13, const float* w13_s,
                                      void* g_q, float* g_s, int64_t M, int64_t I, int64_t K, int scale_fmt,
                                      void* stream) {
    const fp8_status chk = swiglu_check(M, I, K, scale_fmt);
    if (chk != FP8_OK || M == 0) return chk;
    if (!a || !a_s || !w13 || !w13_s || !g_q || !g_s || !aligned16(a) || !aligned16(w13) || !aligned16(g_q))
        return FP8_ERR_INVALID_ARG;
    if (!wide_tiles_ok()) return FP8_ERR_UNSUPPORTED;
    Params prm{};
    prm.a_s = a_s;
    prm.b_s = w13_s;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(2 * I);
    prm.KB = static_cast<int>(K / kBlock);
    prm.NB = static_cast<int>(2 * I / 128);
    prm.G = 1;
    prm.tiles_p = static_cast<int>((M + 127) / 128);
    prm.tiles_q = static_cast<int>(I / 128);   // one 128 x 256 tile per 128-wide block of I
    const int64_t tiles = static_cast<int64_t>(prm.tiles_p) * prm.tiles_q;
    if (tiles > (1LL << 30)) return FP8_ERR_UNSUPPORTED;
    prm.num_tiles = static_cast<int>(tiles);
    prm.vec_scales = (prm.KB % 4 == 0 && aligned16(a_s) && aligned16(w13_s)) ? 1 : 0;
    prm.ue8m0 = scale_fmt == FP8_SCALE_UE8M0 ? 1 : 0;
    prm.gq = static_cast<uint8_t*>(g_q);
    prm.gs = g_s;
    prm.debug_skip = g_debug_skip_next.exchange(0);
#ifdef FP8BS_TRACE_ENABLED
    prm.trace_slot = g_trace_next++ & 3;
#endif
    CUtensorMap mp, mq;
    if (!make_map(&mp, a, M, K, 128) || !make_map(&mq, w13, 2 * I, K, 256)) return FP8_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(tiles, device_sm_count()));
    const cudaError_t e = launch<256, kDense, true>(mp, mq, mp, prm, grid, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

extern "C" fp8_status fp8_moe_expert_up(const void* a, const float* a_s, const void* w13, const float* w13_s,
                                        const int32_t* offsets, int32_t G, int64_t R_max, void* g_q, float* g_s,
                                        int64_t I, int64_t K, int scale_fmt, void* stream) {
    const fp8_status chk = swiglu_check(R_max, I, K, scale_fmt);
    if (chk != FP8_OK) return chk;
    if (G < 0 || G > kMaxGroups) return FP8_ERR_INVALID_ARG;
    if (G == 0 || R_max == 0) return FP8_OK;
    if (static_cast<int64_t>(G) * 2 * I > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    if (!a || !a_s || !w13 || !w13_s || !offsets || !g_q || !g_s || !aligned16(a) || !aligned16(w13) ||
        !aligned16(g_q))
        return FP8_ERR_INVALID_ARG;
    if (!wide_tiles_ok()) return FP8_ERR_UNSUPPORTED;
    Params prm{};
    prm.a_s = a_s;
    prm.b_s = w13_s;
    prm.offsets = offsets;
    prm.M = static_cast<int>(R_max);
    prm.N = static_cast<int>(2 * I);
    prm.KB = static_cast<int>(K / kBlock);
    prm.NB = static_cast<int>(2 * I / 128);
    prm.G = G;
    prm.stream_k = 0;
    prm.vec_scales = (prm.KB % 4 == 0 && aligned16(a_s) && aligned16(w13_s)) ? 1 : 0;
    prm.ue8m0 = scale_fmt == FP8_SCALE_UE8M0 ? 1 : 0;
    prm.gq = static_cast<uint8_t*>(g_q);
    prm.gs = g_s;
    prm.debug_skip = g_debug_skip_next.exchange(0);
#ifdef FP8BS_TRACE_ENABLED
    prm.trace_slot = g_trace_next++ & 3;
#endif
    CUtensorMap mp, mq;
    if (!make_map(&mp, a, R_max, K, 128) || !make_map(&mq, w13, static_cast<int64_t>(G) * 2 * I, K, 256))
        return FP8_ERR_CUDA;
    const cudaError_t e =
        launch<256, kGrouped, true>(mp, mq, mp, prm, device_sm_count(), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot allocate device memory at the point where they run a
// linear layer: code that must not call cudaMalloc (which can synchronise the
// device) on a latency-critical path, code running under a fixed memory
// budget, or hosts that own the CUDA allocator and hand out no scratch.  For
// them fp8_gemm_noalloc runs fp8_gemm with the split-tile scratch taken from
// a fixed array that lives in this library's device image.
namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB per device, held until exit

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's name is only a host-side stand-in; its device address is looked
// up once per device (with that device current) and cached here.
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {nullptr};

fp8_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FP8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FP8_OK;
}

}  // namespace

extern "C" fp8_status fp8_gemm_noalloc(const void* a, const float* a_s, const void* b,
                                       const float* b_s, void* c_bf16, float* c_fp32, int64_t M,
                                       int64_t N, int64_t K, void* stream) {
    // every check fp8_gemm makes comes first: a rejected call leaves the
    // shared array alone (it may belong to a call running on another stream)
    const fp8_status chk = gemm_check_args(a, a_s, b, b_s, c_bf16, c_fp32, M, N, K);
    if (chk != FP8_OK || M == 0 || N == 0) return chk;
    const size_t need = fp8_gemm_workspace_size(M, N, K);
    if (need > kNoAllocScratchBytes) return FP8_ERR_WORKSPACE;   // beyond the fixed array
    void* scratch = nullptr;
    if (need > 0) {
        const fp8_status st = noalloc_scratch(&scratch);
        if (st != FP8_OK) return st;
        // the split-tile counters must start at zero; the array keeps whatever
        // the previous call (or an aborted one) left in it
        if (cudaMemsetAsync(scratch, 0, kCounterBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FP8_ERR_CUDA;
    }
    return fp8_gemm(a, a_s, b, b_s, c_bf16, c_fp32, M, N, K, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                    stream);
}

// ------------------------------------------------------------------ fused linear
namespace {
constexpr size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Batches up to 16 tokens quantise the activations inside the decode kernel
// (each CTA quantises its own K range; a 16-token slab is 2 KB of codes);
// larger batches stage act_quant's codes and scales in the workspace and
// run fp8_gemm on them.
bool linear_is_fused(int64_t M, int64_t, int64_t) { return M <= kDecodeFusedMaxM; }

// Staged fp8_linear workspace: [fp8_gemm's region][codes][scales].  The
// region in front is never shorter than the split-tile counters, which must
// stay zero for whichever later call shares the workspace, even when this
// shape's own GEMM needs no workspace.
size_t linear_gemm_region(int64_t M, int64_t N, int64_t K) {
    return align256(std::max(fp8_gemm_workspace_size(M, N, K), kCounterBytes));
}
}  // namespace

extern "C" size_t fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % kBlock != 0) return 0;
    if (linear_is_fused(M, N, K)) return 0;
    return linear_gemm_region(M, N, K) + align256(static_cast<size_t>(M) * K) +
           align256(static_cast<size_t>(M) * (K / kBlock) * 4);
}

extern "C" fp8_status fp8_linear(const void* x, const void* w, const float* w_s, void* c_bf16, float* c_fp32,
                                 int64_t M, int64_t N, int64_t K, int scale_fmt, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (M < 0 || N < 0 || K <= 0 || K % kBlock != 0) return FP8_ERR_INVALID_ARG;
    if (scale_fmt != FP8_SCALE_FP32 && scale_fmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!x || !w || !w_s || (!c_bf16 && !c_fp32) || !aligned16(x) || !aligned16(w)) return FP8_ERR_INVALID_ARG;
    if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1) return FP8_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!linear_is_fused(M, N, K)) {
        const size_t need = fp8_linear_workspace_size(M, N, K);
        if (!workspace || workspace_bytes < need) return FP8_ERR_WORKSPACE;
        // layout: [fp8_gemm region (zero-kept counters first)][codes][scales],
        // so a workspace shared with fp8_gemm keeps its counters in place
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        const size_t g_need = fp8_gemm_workspace_size(M, N, K);
        const size_t g_bytes = linear_gemm_region(M, N, K);
        const size_t q_bytes = align256(static_cast<size_t>(M) * K);
        uint8_t* xq = ws + g_bytes;
        float* xs = reinterpret_cast<float*>(xq + q_bytes);
        fp8_status r = fp8_act_quant(x, xq, xs, M, K, scale_fmt, stream);
        if (r != FP8_OK) return r;
        return fp8_gemm(xq, xs, w, w_s, c_bf16, c_fp32, M, N, K, g_need ? ws : nullptr, g_need ? g_bytes : 0,
                        stream);
    }
    if ((c_bf16 && (reinterpret_cast<uintptr_t>(c_bf16) & 1)) || (c_fp32 && (reinterpret_cast<uintptr_t>(c_fp32) & 3)))
        return FP8_ERR_INVALID_ARG;
    // decode batches: the quantisation runs inside the decode kernel, whose
    // plan is fp8_gemm's for the same shape (bit-identical results)
    return decode_gemm(x, nullptr, nullptr, w, w_s, c_bf16, c_fp32, M, N, K, scale_fmt == FP8_SCALE_UE8M0 ? 1 : 0, 0,
                       st);
}
