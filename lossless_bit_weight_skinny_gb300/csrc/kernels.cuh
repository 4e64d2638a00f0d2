// kernels.cuh -- arguments and shared device code of the W12 GEMM kernels:
// the stream-K work split, the deterministic split-K fix-up and the
// bounded-wait abort protocol.
#pragma once
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "w12.h"

namespace w12 {

// Device status codes (mirror w12_status values).
constexpr int kStatusTimeout = 8;
constexpr int kStatusCorrupt = 7;

// Matrices of one launch: a grouped launch runs several W12 matrices that
// read the same activations x; their row blocks are laid end to end, matrix i
// owning row blocks [rb0, next matrix's rb0).
constexpr int kMaxGroup = 4;

struct MatArgs {
    const uint8_t *ebase;          // [N] window base per row
    const uint32_t *tile_ptr;      // [T + 1]
    const uint32_t *esc;           // escape entries
    uint32_t n_esc;                // their count: every read of esc stays below it
    const uint16_t *gptr;          // [T][16]: entries of tile t in rows < 8g
    void *y;                       // [M][ldy]: FP32, or BF16 under kOutBF16
    int *status;                   // device status word of the handle
    const float *scale;            // [N] row scales of an INT8 copy (INT8 weights only)
    int N;                         // rows of the matrix
    int ldy;                       // elements per row of y: N, or N / 2 under kOutSiluMul
    int rb0;                       // its first row block in the launch
};

struct GemmArgs {
    MatArgs mat[kMaxGroup];
    int n_mat;                     // matrices of the launch (1 .. kMaxGroup)
    float *partials;               // [2 * grid][M][rows_blk] split-K partial sums
    unsigned long long *counters;  // [n_rowblk] arrivals (zero between launches)
    int M, K;
    int tiles_c;                   // ceil(K / 256): escape tiles per row band
    int n_rowblk;                  // row blocks of all matrices
    int n_kstep;                   // k steps per row block
    int total_iters;               // n_rowblk * n_kstep
    uint64_t limit_ns;             // bounded-wait limit
    int inject_stall;              // test hook: wait on a barrier nobody arrives on
    int x_ready;                   // x was complete before the previous launch: load it at once
    int out_mode;                  // kOutBF16 | kOutSiluMul
    int defer;                     // split row blocks: leave the partials to sk_reduce_kernel
    // 2^28, 2^24, 2^20: multipliers whose high product words are the B word
    // shifted right by 4, 8, 12 bits (a kernel argument, so that the shifts
    // run as multiplies on the FMA pipe beside the decode's logic operations)
    uint32_t bshift_mul[3];
};

// TMA maps of a launch: each matrix's AE and B planes, and the activations.
struct alignas(64) TmapSet {
    CUtensorMap ae[kMaxGroup];
    CUtensorMap b[kMaxGroup];
    CUtensorMap x;
};

// The matrix that owns row block rb of the launch.
__host__ __device__ __forceinline__ int mat_of(const GemmArgs &a, int rb)
{
    int g = 0;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        g += (i < a.n_mat && rb >= a.mat[i].rb0) ? 1 : 0;
    return g;
}

// Output modes.  kOutBF16: y holds BF16, each FP32 result rounded to the
// nearest BF16 (ties to even).  kOutSiluMul: the matrix's rows come in
// (gate, up) pairs -- row 2i is gate row i, row 2i+1 up row i -- and y[m][i]
// = silu(y2i) * y2i+1 with silu(g) = g / (1 + e^-g), the gated-MLP product
// of a dense layer, so that y[M][N/2] is the input of the down projection.
constexpr int kOutBF16 = 1;
constexpr int kOutSiluMul = 2;

__device__ __forceinline__ void put_y(const GemmArgs &a, const MatArgs &mm, int m, int col, float v)
{
    const size_t i = static_cast<size_t>(m) * mm.ldy + col;
    if (a.out_mode & kOutBF16)
        static_cast<__nv_bfloat16 *>(mm.y)[i] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(mm.y)[i] = v;
}

// The final value v of y[m][n] of matrix mm (n < mm.N); `next` is the final
// value of row n + 1 (read only under kOutSiluMul, where N is even and a gate
// row n is even).
__device__ __forceinline__ void emit_y(const GemmArgs &a, const MatArgs &mm, int m, int n, float v, float next)
{
    if (a.out_mode & kOutSiluMul) {
        if ((n & 1) == 0)
            put_y(a, mm, m, n >> 1, v / (1.0f + expf(-v)) * next);
    } else {
        put_y(a, mm, m, n, v);
    }
}

// One BF16x2 pair (weights 2i, 2i+1 of a group of 8) from the group's AE word
// holding those two bytes and its B word (SpecPilot, Figure 5(a) caption):
//   PRMT spreads the two AE bytes into two 16-bit lanes, replicating each
//   byte's sign into the lane's high byte; then per lane
//   sign (bit 15) | (ebase + E) << 7 | (A & 7) << 4 | B,
// with eb2 = ebase << 7 in both lanes.  Written as explicit PTX so that it
// stays PRMT + LOP3 + IMAD + LOP3 (+ SHF + LOP3 for the B nibbles).
template <int I, bool Q8>
__device__ __forceinline__ uint32_t decode_pair(uint32_t ae_word, uint32_t bw, uint32_t eb2)
{
    uint32_t p, t, r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(p) : "r"(ae_word), "n"((I & 1) ? 0xB3A2 : 0x9180));
    asm("and.b32 %0, %1, 0x000F000F;" : "=r"(t) : "r"(p));
    asm("mad.lo.u32 %0, %1, 128, %2;" : "=r"(t) : "r"(t), "r"(eb2));
    asm("lop3.b32 %0, %1, 0x80708070, %2, 0xEA;" : "=r"(r) : "r"(p), "r"(t)); // (p & m) | t
    if (!Q8) {
        uint32_t b = bw;
        if (I)
            asm("shr.b32 %0, %1, %2;" : "=r"(b) : "r"(bw), "n"(4 * I));
        asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(b), "r"(r)); // (b & m) | r
    }
    return r;
}

// 8 weights (AE bytes of the group as two words, its B word) -> 4 BF16x2 pairs.
template <bool Q8>
__device__ __forceinline__ void decode_group(uint32_t a_lo, uint32_t a_hi, uint32_t bw, uint32_t eb2,
                                             uint32_t *out)
{
    out[0] = decode_pair<0, Q8>(a_lo, bw, eb2);
    out[1] = decode_pair<1, Q8>(a_lo, bw, eb2);
    out[2] = decode_pair<2, Q8>(a_hi, bw, eb2);
    out[3] = decode_pair<3, Q8>(a_hi, bw, eb2);
}

// 8 INT8 weights (two words, two's complement, weight j in byte j) -> 4 BF16x2
// pairs, exactly: byte u = q + 128 (XOR 0x80) is placed under the exponent of
// 2^23 by one PRMT (fp32 2^23 + u), an FP32 subtraction of 2^23 + 128 leaves q
// exactly, and since |q| <= 127 needs at most 7 significant bits, the upper
// halves of two such floats are the two BF16 values.
__device__ __forceinline__ void decode_i8_group(uint32_t lo, uint32_t hi, uint32_t *out)
{
    const uint32_t w[2] = {lo ^ 0x80808080u, hi ^ 0x80808080u};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t src = w[p >> 1];
        uint32_t f0, f1;
        const uint32_t sel0 = 0x7650u | static_cast<uint32_t>((2 * p) & 3);
        const uint32_t sel1 = 0x7650u | static_cast<uint32_t>((2 * p + 1) & 3);
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(f0) : "r"(src), "r"(0x4B000000u), "r"(sel0));
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(f1) : "r"(src), "r"(0x4B000000u), "r"(sel1));
        const float q0 = __uint_as_float(f0) - 8388736.0f; // 2^23 + 128
        const float q1 = __uint_as_float(f1) - 8388736.0f;
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(out[p]) : "r"(__float_as_uint(q0)), "r"(__float_as_uint(q1)));
    }
}

// First iteration of CTA c when `iters` iterations are split over `grid` CTAs.
__host__ __device__ __forceinline__ int sk_begin(int c, int grid, int iters)
{
    return static_cast<int>((static_cast<long long>(c) * iters) / grid);
}

// The CTA that owns iteration i.
__host__ __device__ __forceinline__ int sk_owner(int i, int grid, int iters)
{
    return static_cast<int>((static_cast<long long>(i + 1) * grid + iters - 1) / iters) - 1;
}

// Partial slot of contributor c for row block rb (a CTA contributes to at most
// two row blocks partially: the one it starts in and the one it ends in).
__host__ __device__ __forceinline__ int sk_slot(int c, int rb, int grid, int iters, int n_kstep)
{
    const int first_rb = sk_begin(c, grid, iters) / n_kstep;
    return 2 * c + (rb == first_rb ? 0 : 1);
}

// Register one arrival for row block rb; returns true for the last of `n`
// contributors, which also resets the count to zero for the next launch (or a
// replay of this one from a CUDA graph).  One atomic per contributor, with
// acquire-release semantics at GPU scope: it publishes this CTA's partial
// sums (stored by its threads before the CTA barrier that precedes the call)
// and, for the last contributor, makes every other contributor's partials
// visible to the reads after the next CTA barrier.  No retry loop, so many
// CTAs sharing a row block do not serialise on the L2.  Every contributor
// arrives exactly once even after a timeout (the kernels keep their loop
// shape), so the count always completes and resets.
__device__ __forceinline__ bool sk_arrive(unsigned long long *ctr, uint32_t n)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
    if (old + 1 != n)
        return false;
    atomicExch(ctr, 0ull);
    return true;
}

// Escape-list bounds of the units it0 + first + lane (one per lane; units of
// 256 columns = one escape tile wide, row blocks of rows_blk <= 128 rows).
__device__ __forceinline__ void load_tile_window(const GemmArgs &a, int it0, int n_it, int first,
                                                 int lane, int rows_blk, uint32_t &lo, uint32_t &hi)
{
    if (first + lane < n_it) {
        const int u = it0 + first + lane;
        const int rb = u / a.n_kstep;
        const MatArgs &mm = a.mat[mat_of(a, rb)];
        const int t = ((rb - mm.rb0) * rows_blk / 128) * a.tiles_c + u % a.n_kstep;
        lo = __ldg(mm.tile_ptr + t);
        hi = __ldg(mm.tile_ptr + t + 1);
    }
}

// Record a device-side failure in the status word of every matrix of the launch.
__device__ __forceinline__ void report(const GemmArgs &a, int code)
{
    for (int g = 0; g < a.n_mat; ++g)
        atomicCAS(a.mat[g].status, 0, code);
}

// The last contributor sums every partial of row block rb and writes y.
// Threads [0, nthreads) of the CTA take part (nthreads a multiple of 32).  Each
// float4 group of (m, 4 rows) is given to P lanes of one warp (P a power of two,
// up to 32, as many as the contributors and threads allow): lane j sums
// contributors c_first + j, c_first + j + P, ... in order, with independent
// 16-byte loads, and the P lanes then combine by a fixed butterfly.  The order
// is fixed, so results are bitwise reproducible, and many contributors cost
// one round of loads instead of one per contributor.  EPI: the results go
// through the output mode (emit_y); otherwise y is FP32 [M][N].
#ifndef W12_SK_UNROLL
#define W12_SK_UNROLL 4 // partial loads in flight per lane
#endif
#ifndef W12_SK_NOINLINE
#define W12_SK_NOINLINE 0
#endif
#if W12_SK_NOINLINE
#define W12_SK_INL static __noinline__
#else
#define W12_SK_INL __forceinline__
#endif
template <bool EPI, int U = W12_SK_UNROLL>
__device__ W12_SK_INL void sk_reduce_range(const GemmArgs &a, int rb, int rows_blk, int grid, int c_first,
                                           int c_last, int tid, int nthreads, int g_lo, int g_hi)
{
    const MatArgs &mm = a.mat[mat_of(a, rb)];
    const int row0 = (rb - mm.rb0) * rows_blk; // first row of the block in its matrix
    const int groups = g_hi; // float4 groups [g_lo, g_hi) of the partial
    const size_t slot4 = static_cast<size_t>(a.M) * rows_blk / 4;
    const float4 *base = reinterpret_cast<const float4 *>(a.partials);
    const int n_contrib = c_last - c_first + 1;
    // the first contributor's slot index is 0 or 1; the others start in this
    // row block, so their slot is 2c
    const int slot_first = sk_slot(c_first, rb, grid, a.total_iters, a.n_kstep);
    int P = 1;
    while (P < 32 && P < n_contrib && 2 * P * (g_hi - g_lo) <= nthreads)
        P *= 2;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    const int gpw = 32 / P; // groups per warp and pass
    const int j = lane % P;
    for (int gbase = g_lo + warp * gpw; gbase < groups; gbase += nwarps * gpw) {
        const int g = gbase + lane / P;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g < groups) {
            for (int c0 = c_first + j; c0 <= c_last; c0 += U * P) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * P;
                    if (c <= c_last) {
                        const int slot = (c == c_first) ? slot_first : 2 * c;
                        v[u] = __ldcg(base + slot * slot4 + g);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (c0 + u * P <= c_last) {
                        acc.x += v[u].x;
                        acc.y += v[u].y;
                        acc.z += v[u].z;
                        acc.w += v[u].w;
                    }
                }
            }
        }
        for (int o = P >> 1; o >= 1; o >>= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
            acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
            acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
        }
        if (g < groups && j == 0) {
            const int m = (4 * g) / rows_blk, r = (4 * g) % rows_blk;
            const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (row0 + r + q < mm.N) {
                    if constexpr (EPI)
                        emit_y(a, mm, m, row0 + r + q, v4[q], v4[(q + 1) & 3]);
                    else
                        static_cast<float *>(mm.y)[static_cast<size_t>(m) * mm.N + row0 + r + q] = v4[q];
                }
            }
        }
    }
}

// The last contributor's fix-up with few threads: each thread takes GPT float4
// groups of (m, 4 rows) at a stride of nthreads and sums every contributor's
// partial of them in contributor order, two contributors' GPT loads in flight
// at a time.  The order is fixed, so results are bitwise reproducible.
template <bool EPI, int GPT>
__device__ __forceinline__ void sk_reduce_wide(const GemmArgs &a, int rb, int rows_blk, int grid, int c_first,
                                               int c_last, int tid, int nthreads)
{
    const MatArgs &mm = a.mat[mat_of(a, rb)];
    const int row0 = (rb - mm.rb0) * rows_blk; // first row of the block in its matrix
    const int groups = a.M * rows_blk / 4;
    const size_t slot4 = static_cast<size_t>(a.M) * rows_blk / 4;
    const float4 *base = reinterpret_cast<const float4 *>(a.partials);
    const int slot_first = sk_slot(c_first, rb, grid, a.total_iters, a.n_kstep);
    for (int g0 = tid; g0 < groups; g0 += GPT * nthreads) {
        float4 acc[GPT];
#pragma unroll
        for (int i = 0; i < GPT; ++i)
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = c_first; c <= c_last; c += 2) {
            const float4 *p0 = base + static_cast<size_t>(c == c_first ? slot_first : 2 * c) * slot4;
            const bool two = c + 1 <= c_last;
            const float4 *p1 = base + static_cast<size_t>(2 * (c + 1)) * slot4;
            float4 v0[GPT], v1[GPT];
#pragma unroll
            for (int i = 0; i < GPT; ++i) {
                const int g = g0 + i * nthreads;
                if (g < groups) {
                    v0[i] = __ldcg(p0 + g);
                    if (two)
                        v1[i] = __ldcg(p1 + g);
                }
            }
#pragma unroll
            for (int i = 0; i < GPT; ++i) {
                acc[i].x += v0[i].x;
                acc[i].y += v0[i].y;
                acc[i].z += v0[i].z;
                acc[i].w += v0[i].w;
                if (two) {
                    acc[i].x += v1[i].x;
                    acc[i].y += v1[i].y;
                    acc[i].z += v1[i].z;
                    acc[i].w += v1[i].w;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < GPT; ++i) {
            const int g = g0 + i * nthreads;
            if (g >= groups)
                continue;
            const int m = (4 * g) / rows_blk, r = (4 * g) % rows_blk;
            const float v4[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (row0 + r + j < mm.N) {
                    if constexpr (EPI)
                        emit_y(a, mm, m, row0 + r + j, v4[j], v4[(j + 1) & 3]);
                    else
                        static_cast<float *>(mm.y)[static_cast<size_t>(m) * mm.N + row0 + r + j] = v4[j];
                }
            }
        }
    }
}

// The whole row block: every float4 group of its M x rows_blk partial.
template <bool EPI>
__device__ __forceinline__ void sk_reduce_block(const GemmArgs &a, int rb, int rows_blk, int grid, int c_first,
                                                int c_last, int tid, int nthreads)
{
    sk_reduce_range<EPI>(a, rb, rows_blk, grid, c_first, c_last, tid, nthreads, 0, a.M * rows_blk / 4);
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream is finishing; it calls
// pdl_wait_prior_grid() before touching anything that kernel may write.
template <typename Kern>
cudaError_t launch_pdl(Kern kern, int grid, int threads, int smem, cudaStream_t st, const GemmArgs &a,
                       const TmapSet &tm)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, tm);
}

// Launchers (defined in gemm_fma.cu / gemm_tc.cu / decode.cu).
cudaError_t launch_gemm_fma(int mt, bool q8, const GemmArgs &a, const TmapSet &tm, int grid, cudaStream_t st);
// Split-K fix-up as a kernel of its own (reduce.cu), chained after a
// tensor-core GEMM launched with a.defer set; nothing is launched when no row
// block is split.  *launched tells whether it was.
cudaError_t launch_sk_reduce(const GemmArgs &a, int gemm_grid, int rows_blk, cudaStream_t st, bool *launched);
// INT8 copy of BF16 weights on the device (i8.cu): per row, scale = amax / 127
// over the finite weights, q = rint(w / scale) clamped to [-127, 127], Inf to
// +-127, NaN to 0, q = 0 where the scale is 0.
cudaError_t launch_i8_quantize(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *scale, cudaStream_t st);
// i8: the weights are an INT8 copy (mat[].scale set, tm.ae over its bytes).
cudaError_t launch_gemm_tc(int mt, bool q8, bool i8, const GemmArgs &a, const TmapSet &tm, int grid,
                           cudaStream_t st);
int fma_rows_blk(int mt);
int fma_ctas_per_sm(int mt);
int fma_smem_bytes(int mt, bool q8);
int tc_smem_bytes(int mt, bool q8);
#ifndef W12_FMA_MIN_ITERS
#define W12_FMA_MIN_ITERS 1 // fewest units per CTA the CUDA-core grid aims for
#endif
#ifndef W12_TC_MIN_M
#define W12_TC_MIN_M 3 // smallest M sent to the tensor-core kernel (at most 5)
#endif
static_assert(W12_TC_MIN_M >= 1 && W12_TC_MIN_M <= 5, "the CUDA-core kernel covers M <= 4");
constexpr int kFmaKStep = 256;
constexpr int kTcKStep = 256;
constexpr int kTcRows = 128;
// activation ring slots (one 64-column sub-tile each) of the 128-row kernel
#ifndef W12_TC_XST128
#define W12_TC_XST128 4
#endif

// Grid of one GEMM launch (host side).  The units (row block, k step) are
// split evenly over the CTAs, one CTA per SM at most; a CTA's time is about
// its unit count, plus the tail of combining partial row blocks.  Measured on
// GB300, that tail costs about three units when CTA boundaries fall inside row
// blocks at random (stream-K over every SM) and about one when every CTA holds
// an equal share of a single row block (n_rowblk * c CTAs, c dividing the k
// steps).  The cheaper of the two estimates is launched.
#ifndef W12_GRID_ALIGNED
#define W12_GRID_ALIGNED 1
#endif
// Smallest unit count per CTA of the tensor-core kernel: a 128 x 256 unit
// reads 48 KB of W12 and a CTA's partial of a row block is M x 512 bytes, so
// for large M fewer CTAs each stream several units per partial they write.
//
// Above W12_TC_DEFER_M rows, the tensor-core GEMM leaves split row blocks to
// the separate fix-up kernel (reduce.cu), which reads the partials with many
// CTAs; then the partials cost little and the unit floor is lower.  Measured
// on GB300: at M = 128 a 1024 x 5120 GEMM takes 10.3 us that way against 23.2
// us with the in-kernel fix-up; at M <= 32 the second launch costs 2-3 us
// more than it saves.
#ifndef W12_TC_DEFER_M
#define W12_TC_DEFER_M 64
#endif
#ifndef W12_TC_PART_RATIO
#define W12_TC_PART_RATIO 24
#endif
inline bool tc_defer(int M) { return M > W12_TC_DEFER_M; }
inline int64_t tc_min_iters(int M)
{
    const int64_t ratio = tc_defer(M) ? 64 : W12_TC_PART_RATIO;
    return std::max<int64_t>(1, (static_cast<int64_t>(M) + ratio - 1) / ratio);
}

// SMs the CUDA-core kernel leaves out of its grid (at most one in eight).  A
// launch's CTAs start as the previous kernel's CTAs free their SMs; with some
// SMs left out, the first CTAs start at once, and at 16 of 152 the grid is
// 136 CTAs, which holds two whole 128-row blocks of a 34816-row (gate/up)
// group per CTA with no split.  Measured on GB300 on the grouped single-row
// layer step: 4 / 8 / 12 / 16 / 24 SMs left out: 100.9 / 101.1 / 100.3 /
// 99.8 / 107.1 us.
// SMs the tensor-core kernel leaves out of its grid (at most one in eight):
// at 136 CTAs the gate/up group and 17408-row matrices split into whole row
// blocks, and the split-K tail goes.  Measured on GB300, grouped layer step
// at 16 / 32 / 64 / 128 rows: none left out 125.6 / 129.0 / 146.9 / - us;
// 8: 125.3 / 128.7 / 146.7 / 201.7; 16: 124.4 / 126.6 / 138.8 / 184.6;
// 24: 130.4 / 132.8 / 148.7 / 209.2.
#ifndef W12_TC_SM_RESERVE
#define W12_TC_SM_RESERVE 16
#endif
#ifndef W12_FMA_SM_RESERVE
#define W12_FMA_SM_RESERVE 16
#endif
inline int choose_grid(int64_t n_rowblk, int64_t n_kstep, int sms, int64_t min_iters)
{
    const int64_t iters = n_rowblk * n_kstep;
    const int64_t want = std::max<int64_t>(n_rowblk, iters / std::max<int64_t>(min_iters, 1));
    const int64_t plain = std::min<int64_t>(sms, std::min<int64_t>(iters, want));
    if (!W12_GRID_ALIGNED)
        return static_cast<int>(plain);
    const int64_t upc = (iters + plain - 1) / plain; // units per CTA, rounded up
    const bool plain_whole = iters % plain == 0 && (upc % n_kstep == 0 || n_kstep % upc == 0);
    int64_t best = plain, best_cost = upc + (plain_whole ? (upc < n_kstep ? 1 : 0) : 3);
    for (int64_t c = 1; c <= n_kstep && n_rowblk * c <= std::min<int64_t>(sms, want); ++c) {
        if (n_kstep % c != 0)
            continue;
        const int64_t cost = n_kstep / c + (c > 1 ? 1 : 0);
        if (cost < best_cost) {
            best = n_rowblk * c;
            best_cost = cost;
        }
    }
    return static_cast<int>(best);
}

// ---- host-side runtime shared by the entry points (runtime.cu) ----

constexpr size_t kCounterBytes = 1 << 16; // split-K arrival counters: room for 8192 row blocks

// The launch of one GEMM: kernel, tile rows, grid and split-K shape.
struct Plan {
    bool tc = false;
    int mt = 0, rows_blk = 0, kstep = 0, grid = 0;
    int64_t n_rowblk = 0, n_kstep = 0, iters = 0;
    bool defer = false;
    size_t part_bytes = 0; // split-K partial sums of the launch
};
w12_status make_plan(int M, int64_t N, int64_t K, int sms, Plan *p);
// The launch over several matrices of rows Ns[0..n) that read the same x.
w12_status make_plan_group(int M, const int64_t *Ns, int n, int64_t K, int sms, Plan *p);
// 2-D TMA map over a row-major [rows][cols] array of `esize`-byte elements.
bool make_tmap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t cols,
               uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);
// The activations' map of a GEMM launch with tile rows mt.
bool make_x_tmap(CUtensorMap *m, const void *x, int M, int K, bool tc, int mt);
int sm_count(int dev);
// The wall-time limit of bounded device waits and the stall test hook, as set
// by w12_set_spin_limit / w12_debug_inject_stall.
uint64_t spin_limit_ns();
int inject_stall();
// Record a CUDA error for w12_last_cuda_error and return W12_ERR_CUDA.
w12_status cuda_fail(cudaError_t e);
void set_last_error(const char *msg);

} // namespace w12

struct w12_dev;

namespace w12 {

// A device handle for an N x K matrix with room for n_esc escapes (runtime.cu):
// one allocation, status word cleared on `st`, GEMM tensor maps built.
w12_status dev_create(int64_t N, int64_t K, int64_t n_esc, cudaStream_t st, w12_dev **out);

cudaError_t launch_decode(const uint8_t *ebase, const uint8_t *ae, const uint8_t *b,
                          const uint32_t *tile_ptr, const uint32_t *esc, uint16_t *out, int64_t N,
                          int64_t K, cudaStream_t st);

} // namespace w12
