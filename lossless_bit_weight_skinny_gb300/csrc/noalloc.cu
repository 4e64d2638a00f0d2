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
//   * calls that would need more scratch than that are rejected with
//     W12_ERR_UNSUPPORTED (only extreme shapes: more than 8192 row blocks, or a
//     GPU with so many SMs that 2 * SMs * M * 128 partial sums do not fit);
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

constexpr size_t kNoAllocCounterBytes = size_t(64) << 10; // arrival counters: 8192 row blocks
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20; // counters + split-K partial sums

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
        if (cudaMemset(p, 0, kNoAllocCounterBytes) != cudaSuccess)
            return W12_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess)
            return W12_ERR_CUDA;
        g_na_ptr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_na_ptr[dev]);
    return W12_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// TMA descriptor of the activations x[M][K] (BF16), as w12_gemm builds it.
bool x_tmap(CUtensorMap *m, const void *x, int M, int K, uint32_t box_k, uint32_t box_m,
            CUtensorMapSwizzle sw)
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {box_k, box_m};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    if (cudaGetDevice(&dev) != cudaSuccess)
        return W12_ERR_CUDA;
    if (dev != w->device)
        return W12_ERR_INVALID_ARG;
    if (K == 0)
        return cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(M) * N, st) == cudaSuccess
                   ? W12_OK
                   : W12_ERR_CUDA;
    if (!w->gemm_ok)
        return W12_ERR_UNSUPPORTED;

    const bool tc = M >= W12_TC_MIN_M;
    const int mt = tc ? (M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256)
                      : (M <= 1 ? 1 : M <= 2 ? 2 : 4);
    const int rows_blk = tc ? kTcRows : fma_rows_blk(mt);
    const int kstep = tc ? kTcKStep : kFmaKStep;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return W12_ERR_CUDA;

    GemmArgs a{};
    a.ebase = w->ebase;
    a.tile_ptr = w->tile_ptr;
    a.esc = w->esc;
    a.gptr = w->gptr;
    a.y = y;
    a.ldy = N;
    a.status = w->status;
    a.M = M;
    a.N = N;
    a.K = K;
    a.tiles_c = static_cast<int>(w->tiles_c);
    a.n_rowblk = static_cast<int>(ceil_div(N, rows_blk));
    a.n_kstep = static_cast<int>(ceil_div(K, kstep));
    const int64_t iters = static_cast<int64_t>(a.n_rowblk) * a.n_kstep;
    const int64_t min_iters = tc ? tc_min_iters(M) : W12_FMA_MIN_ITERS;
    const int grid = choose_grid(a.n_rowblk, a.n_kstep, tc ? sms : sms * fma_ctas_per_sm(mt) - W12_FMA_SM_RESERVE,
                                 min_iters);
    const size_t part_bytes = sizeof(float) * 2 * static_cast<size_t>(grid) * M * rows_blk;
    // the fixed array must hold the counters and the partial sums of this call
    if (iters > (int64_t(1) << 30) || static_cast<size_t>(a.n_rowblk) * 8 > kNoAllocCounterBytes ||
        kNoAllocCounterBytes + part_bytes > kNoAllocScratchBytes)
        return W12_ERR_UNSUPPORTED;
    a.total_iters = static_cast<int>(iters);
    a.limit_ns = 200ull * 1000 * 1000;
    a.inject_stall = 0;
    a.x_ready = x_ready ? 1 : 0;
    a.defer = tc && tc_defer(M);

    unsigned char *scratch = nullptr;
    const w12_status s = noalloc_setup(dev, &scratch);
    if (s != W12_OK)
        return s;
    a.counters = reinterpret_cast<unsigned long long *>(scratch);
    a.partials = reinterpret_cast<float *>(scratch + kNoAllocCounterBytes);

    CUtensorMap tmx;
    const bool okx = tc ? x_tmap(&tmx, x_bf16, M, K, 64, mt, CU_TENSOR_MAP_SWIZZLE_128B)
                        : x_tmap(&tmx, x_bf16, M, K, 256, mt, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!okx)
        return W12_ERR_CUDA;
    const w12_tmap &tae = tc ? w->tm_ae_tc : (rows_blk == 128 ? w->tm_ae_fma128 : w->tm_ae_fma64);
    const w12_tmap &tb = tc ? w->tm_b_tc : (rows_blk == 128 ? w->tm_b_fma128 : w->tm_b_fma64);
    const CUtensorMap *pae = reinterpret_cast<const CUtensorMap *>(&tae);
    const CUtensorMap *pb = reinterpret_cast<const CUtensorMap *>(&tb);
    cudaError_t e = tc ? launch_gemm_tc(mt, false, false, a, pae, pb, &tmx, grid, st)
                       : launch_gemm_fma(mt, false, a, pae, pb, &tmx, grid, st);
    bool red = false;
    if (e == cudaSuccess && a.defer)
        e = launch_sk_reduce(a, grid, rows_blk, st, &red);
    return e == cudaSuccess ? W12_OK : W12_ERR_CUDA;
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
