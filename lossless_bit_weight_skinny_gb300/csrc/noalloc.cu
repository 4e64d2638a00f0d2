// noalloc.cu -- w12_gemm_noalloc: the same W12 GEMM as w12_gemm for callers
// that must not allocate device memory.
//
// w12_gemm keeps a workspace (split-K partial sums and arrival counters) per
// (device, stream) and allocates it with cudaMallocAsync on the first call on
// a stream.  Some callers cannot allow that: code running where the device
// allocator is off limits (a host that pre-reserves every byte of device
// memory for its own pool, a plug-in inside a framework whose allocator must
// own all device memory, a real-time loop that may not take allocator locks).
// This entry point runs the same kernels with the scratch taken from one
// fixed, statically sized array in device memory instead.
//
// Costs and limits:
//   * every GPU that loads this library reserves kNoAllocScratchBytes (16 MiB)
//     for the array until the process exits, whether or not it is used;
//   * the array holds the split-K arrival counters (64 KiB: 8192 row blocks)
//     and the launch's partial sums, 2 x CTAs x M x 128 FP32 values; a call
//     that needs more is rejected with W12_ERR_UNSUPPORTED.  On a 152-SM GB300
//     that is any tensor-core call above about 107 rows whose grid fills every
//     SM (e.g. 5120 x 5120 or 17408 x 5120 at 128 rows), and matrices of more
//     than 8192 row blocks;
//   * every call on a device shares the one array and leaves its contents
//     behind, so two calls whose kernels overlap on the GPU (different
//     streams, or different host threads) race and give wrong results --
//     serialise them on one stream;
//   * the first call on each device looks up the array's device address and
//     clears its counters, then synchronises the device; make that first call
//     before any stream capture.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "w12_internal.h"

using namespace w12;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20; // arrival counters + split-K partial sums
static_assert(kCounterBytes < kNoAllocScratchBytes, "scratch too small for the counters");

} // namespace

// The scratch itself.  Zero-initialised when the module loads; in host code
// this name is only a stand-in for the symbol, never a usable address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_na_mu;
void *g_na_ptr[64] = {nullptr}; // device address of the scratch, per device

// Once per device, with that device current: fetch the array's device address
// and clear the counters.
w12_status noalloc_setup(int dev, unsigned char **out)
{
    if (dev < 0 || dev >= 64)
        return W12_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return W12_ERR_CUDA;
        if (cudaMemset(p, 0, kCounterBytes) != cudaSuccess)
            return W12_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess)
            return W12_ERR_CUDA;
        g_na_ptr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_na_ptr[dev]);
    return W12_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

} // namespace

static w12_status noalloc_impl(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                               cudaStream_t st, bool x_ready)
{
    if (M == 0 || N == 0)
        return W12_OK;
    if (!x_bf16 || !y)
        return W12_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(y))
        return W12_ERR_ALIGNMENT;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev != w->device)
        return W12_ERR_INVALID_ARG;
    if (K == 0) {
        e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(M) * N, st);
        return e == cudaSuccess ? W12_OK : cuda_fail(e);
    }
    if (!w->gemm_ok)
        return W12_ERR_UNSUPPORTED;

    // the same launch as w12_gemm's (kernel, tile rows, grid, split-K shape)
    Plan pl;
    const w12_status ps = make_plan(M, N, K, sm_count(dev), &pl);
    if (ps != W12_OK)
        return ps;
    // the fixed array must hold the counters and the partial sums of this call
    if (static_cast<size_t>(pl.n_rowblk) * 8 > kCounterBytes || kCounterBytes + pl.part_bytes > kNoAllocScratchBytes)
        return W12_ERR_UNSUPPORTED;

    GemmArgs a{};
    MatArgs &mm = a.mat[0];
    mm.ebase = w->ebase;
    mm.tile_ptr = w->tile_ptr;
    mm.esc = w->esc;
    mm.n_esc = static_cast<uint32_t>(w->n_esc);
    mm.gptr = w->gptr;
    mm.y = y;
    mm.ldy = N;
    mm.status = w->status;
    mm.N = N;
    mm.rb0 = 0;
    a.n_mat = 1;
    for (int i = 1; i < kMaxGroup; ++i)
        a.mat[i] = a.mat[0];
    a.M = M;
    a.K = K;
    a.tiles_c = static_cast<int>(w->tiles_c);
    a.n_rowblk = static_cast<int>(pl.n_rowblk);
    a.n_kstep = static_cast<int>(pl.n_kstep);
    a.total_iters = static_cast<int>(pl.iters);
    a.limit_ns = spin_limit_ns();
    a.inject_stall = inject_stall();
    a.x_ready = x_ready ? 1 : 0;
    a.defer = pl.defer;

    unsigned char *scratch = nullptr;
    const w12_status s = noalloc_setup(dev, &scratch);
    if (s != W12_OK)
        return s;
    a.counters = reinterpret_cast<unsigned long long *>(scratch);
    a.partials = reinterpret_cast<float *>(scratch + kCounterBytes);

    TmapSet tm;
    if (!make_x_tmap(&tm.x, x_bf16, M, K, pl.tc, pl.mt)) {
        set_last_error("cuTensorMapEncodeTiled failed for x");
        return W12_ERR_CUDA;
    }
    const w12_tmap &tae = pl.tc ? w->tm_ae_tc : (pl.rows_blk == 128 ? w->tm_ae_fma128 : w->tm_ae_fma64);
    const w12_tmap &tb = pl.tc ? w->tm_b_tc : (pl.rows_blk == 128 ? w->tm_b_fma128 : w->tm_b_fma64);
    tm.ae[0] = *reinterpret_cast<const CUtensorMap *>(&tae);
    tm.b[0] = *reinterpret_cast<const CUtensorMap *>(&tb);
    e = pl.tc ? launch_gemm_tc(pl.mt, false, false, a, tm, pl.grid, st) : launch_gemm_fma(pl.mt, false, a, tm, pl.grid, st);
    bool red = false;
    if (e == cudaSuccess && a.defer)
        e = launch_sk_reduce(a, pl.grid, pl.rows_blk, st, &red);
    return e == cudaSuccess ? W12_OK : cuda_fail(e);
}

extern "C" w12_status w12_gemm_noalloc(const void *x_bf16, const w12_dev *w, float *y, int M, int N,
                                       int K, w12_stream_t stream)
{
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!w || M < 0)
        return W12_ERR_INVALID_ARG;
    if (N != w->N || K != w->K)
        return W12_ERR_SHAPE;
    if (M > 256)
        return W12_ERR_UNSUPPORTED;
    return noalloc_impl(x_bf16, w, y, M, N, K, st, false);
}
