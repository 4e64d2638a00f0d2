// kernels.cuh -- arguments and shared device code of the W12 GEMM kernels:
// the stream-K work split, the deterministic split-K fix-up and the
// bounded-wait abort protocol.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace w12 {

// Device status codes (mirror w12_status values).
constexpr int kStatusTimeout = 8;
constexpr int kStatusCorrupt = 7;

struct GemmArgs {
    const uint8_t *ebase;          // [N] window base per row
    const uint32_t *tile_ptr;      // [T + 1]
    const uint32_t *esc;           // escape entries
    float *y;                      // [M][N]
    float *partials;               // [2 * grid][M][rows_blk] split-K partial sums
    unsigned long long *counters;  // [n_rowblk] epoch<<32 | arrivals
    int *status;                   // device status word of the handle
    int M, N, K;
    int tiles_c;                   // ceil(K / 256): escape tiles per row band
    int n_rowblk;                  // row blocks
    int n_kstep;                   // k steps per row block
    int total_iters;               // n_rowblk * n_kstep
    uint32_t epoch;                // unique per call on this workspace
    uint64_t limit_ns;             // bounded-wait limit
    int inject_stall;              // test hook: wait on a barrier nobody arrives on
};

// First iteration of CTA c when `iters` iterations are split over `grid` CTAs.
__device__ __forceinline__ int sk_begin(int c, int grid, int iters)
{
    return static_cast<int>((static_cast<long long>(c) * iters) / grid);
}

// The CTA that owns iteration i.
__device__ __forceinline__ int sk_owner(int i, int grid, int iters)
{
    return static_cast<int>((static_cast<long long>(i + 1) * grid + iters - 1) / iters) - 1;
}

// Partial slot of contributor c for row block rb (a CTA contributes to at most
// two row blocks partially: the one it starts in and the one it ends in).
__device__ __forceinline__ int sk_slot(int c, int rb, int grid, int iters, int n_kstep)
{
    const int first_rb = sk_begin(c, grid, iters) / n_kstep;
    return 2 * c + (rb == first_rb ? 0 : 1);
}

// Register one arrival for row block rb under this call's epoch; returns true
// for the last of `n` contributors.  Stale counts left by an earlier call that
// was aborted are discarded by the epoch compare.
__device__ __forceinline__ bool sk_arrive(unsigned long long *ctr, uint32_t epoch, uint32_t n)
{
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(ctr);
    for (;;) {
        const unsigned long long nxt = (static_cast<uint32_t>(cur >> 32) == epoch)
                                           ? cur + 1
                                           : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
        const unsigned long long prev = atomicCAS(ctr, cur, nxt);
        if (prev == cur) {
            if (static_cast<uint32_t>(nxt) != n)
                return false;
            // last one: zero the count (keeping the epoch) so that a replay of
            // the same launch -- e.g. from a CUDA graph -- counts from zero
            atomicExch(ctr, static_cast<unsigned long long>(epoch) << 32);
            return true;
        }
        cur = prev;
    }
}

__device__ __forceinline__ void report(int *status, int code)
{
    atomicCAS(status, 0, code);
}

// The last contributor sums every partial of row block rb in contributor
// order (fixed, so results are bitwise reproducible) and writes y.
// Threads [0, nthreads) of the CTA take part.
__device__ __forceinline__ void sk_reduce_block(const GemmArgs &a, int rb, int rows_blk, int grid,
                                                int c_first, int c_last, int tid, int nthreads)
{
    const int row0 = rb * rows_blk;
    const int total = a.M * rows_blk;
    for (int idx = tid; idx < total; idx += nthreads) {
        const int m = idx / rows_blk, r = idx % rows_blk;
        float s = 0.f;
        for (int c = c_first; c <= c_last; ++c) {
            const int slot = sk_slot(c, rb, grid, a.total_iters, a.n_kstep);
            s += __ldcg(a.partials + (static_cast<size_t>(slot) * a.M + m) * rows_blk + r);
        }
        if (row0 + r < a.N)
            a.y[static_cast<size_t>(m) * a.N + row0 + r] = s;
    }
}

// Launchers (defined in gemm_fma.cu / gemm_tc.cu / decode.cu).
cudaError_t launch_gemm_fma(int mt, bool q8, const GemmArgs &a, const CUtensorMap *tm_ae,
                            const CUtensorMap *tm_b, const CUtensorMap *tm_x, int grid,
                            cudaStream_t st);
cudaError_t launch_gemm_tc(int mt, bool q8, const GemmArgs &a, const CUtensorMap *tm_ae,
                           const CUtensorMap *tm_b, const CUtensorMap *tm_x, int grid,
                           cudaStream_t st);
int fma_rows_blk(int mt);
int fma_smem_bytes(int mt, bool q8);
int tc_smem_bytes(int mt, bool q8);
constexpr int kFmaKStep = 256;
constexpr int kTcKStep = 128;
constexpr int kTcRows = 128;

cudaError_t launch_decode(const uint8_t *ebase, const uint8_t *ae, const uint8_t *b,
                          const uint32_t *tile_ptr, const uint32_t *esc, uint16_t *out, int64_t N,
                          int64_t K, cudaStream_t st);

} // namespace w12
