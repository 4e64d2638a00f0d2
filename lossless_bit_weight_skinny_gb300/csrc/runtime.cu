// runtime.cu -- device side of the C ABI: upload of encoded matrices, TMA
// descriptors, the per-stream GEMM workspace cache and kernel dispatch.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "w12_internal.h"

using namespace w12;

namespace {

std::atomic<uint64_t> g_limit_ns{200ull * 1000 * 1000}; // bounded waits: 200 ms
thread_local const char *g_last_error = "no error";
std::atomic<int> g_inject_stall{0};

} // namespace

namespace w12 {

w12_status cuda_fail(cudaError_t e)
{
    g_last_error = cudaGetErrorName(e);
    return W12_ERR_CUDA;
}
void set_last_error(const char *msg) { g_last_error = msg; }
uint64_t spin_limit_ns() { return g_limit_ns.load(); }
int inject_stall() { return g_inject_stall.load(); }

} // namespace w12

namespace {

// ---- TMA descriptor encoding through the driver entry point -----------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
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
    return fn;
}

} // namespace

namespace w12 {

// 2-D map over a row-major [rows][cols] array of `esize`-byte elements.
bool make_tmap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t cols,
               uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The activations' map of a GEMM launch: 64-column swizzled boxes of mt rows
// for the tensor-core kernel, 256-column plain boxes for the CUDA-core one.
bool make_x_tmap(CUtensorMap *m, const void *x, int M, int K, bool tc, int mt)
{
    return tc ? make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, M, 64, mt, CU_TENSOR_MAP_SWIZZLE_128B)
              : make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, M, 256, mt, CU_TENSOR_MAP_SWIZZLE_NONE);
}

CUtensorMap *tmap_of(w12_tmap &t) { return reinterpret_cast<CUtensorMap *>(&t); }
const CUtensorMap *tmap_of(const w12_tmap &t) { return reinterpret_cast<const CUtensorMap *>(&t); }
static_assert(sizeof(w12_tmap) == sizeof(CUtensorMap), "tensor map size");

int sm_count(int dev)
{
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64)
        return 148;
    if (!cache[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 148;
    }
    return cache[dev];
}

} // namespace w12

namespace {

// ---- workspace cache: one growable buffer per (device, stream) --------------

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
// Workspaces replaced by a larger one.  A CUDA graph captured earlier may
// still hold their addresses, so they are kept until w12_release_workspaces.
std::vector<std::pair<int, void *>> g_ws_retired;

// Returns partial-sum and counter pointers for a call that needs `part_bytes`
// of partial sums.
w12_status get_workspace(int dev, cudaStream_t st, size_t part_bytes, float **partials,
                         unsigned long long **counters)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace &w = g_ws[{dev, st}];
    const size_t need = kCounterBytes + ((part_bytes + 255) & ~static_cast<size_t>(255));
    if (w.bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return W12_ERR_UNSUPPORTED; // grow outside capture: make one call first
        // first use: room for the largest call (M = 128, one CTA per SM), so a
        // workspace never moves under a captured CUDA graph
        const size_t most = kCounterBytes + sizeof(float) * 2 * static_cast<size_t>(sm_count(dev)) * 128 * 128;
        const size_t grow = need < most ? most : need;
        if (w.ptr)
            g_ws_retired.emplace_back(dev, w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        void *p = nullptr;
        if (cudaMallocAsync(&p, grow, st) != cudaSuccess)
            return W12_ERR_OOM;
        if (cudaMemsetAsync(p, 0, kCounterBytes, st) != cudaSuccess)
            return W12_ERR_CUDA;
        w.ptr = p;
        w.bytes = grow;
    }
    *counters = static_cast<unsigned long long *>(w.ptr);
    *partials = reinterpret_cast<float *>(static_cast<char *>(w.ptr) + kCounterBytes);
    return W12_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr int kMaxM = 256;

} // namespace

namespace w12 {

// The launch of one GEMM: kernel, tile rows, grid and split-K shape.  Kernel
// choice is a function of M only (measured on GB300): the CUDA-core kernel for
// M <= 2; from 3 rows on, the tensor-core kernel (M padded to 16, 32, 64, 128
// or 256) is faster than four FMAs per weight.
w12_status make_plan(int M, int64_t N, int64_t K, int sms, Plan *p)
{
    return make_plan_group(M, &N, 1, K, sms, p);
}

// The launch over several matrices of rows Ns[0..n) read with the same x:
// their row blocks end to end.
w12_status make_plan_group(int M, const int64_t *Ns, int n, int64_t K, int sms, Plan *p)
{
    Plan q;
    q.tc = M >= W12_TC_MIN_M;
    q.mt = q.tc ? (M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256)
                : (M <= 1 ? 1 : M <= 2 ? 2 : 4);
    q.rows_blk = q.tc ? kTcRows : fma_rows_blk(q.mt);
    q.kstep = q.tc ? kTcKStep : kFmaKStep;
    q.n_rowblk = 0;
    for (int i = 0; i < n; ++i)
        q.n_rowblk += ceil_div(Ns[i], q.rows_blk);
    q.n_kstep = ceil_div(K, q.kstep);
    q.iters = q.n_rowblk * q.n_kstep;
    if (q.iters > (1ll << 30) || q.n_rowblk * 8 > static_cast<int64_t>(kCounterBytes))
        return W12_ERR_UNSUPPORTED;
    q.defer = q.tc && tc_defer(M);
    // one CTA per SM (four left out for the CUDA-core kernel); for large M on
    // few row blocks, fewer CTAs so that each streams several times the weight
    // bytes of the partial sums it writes (a 128 x 256 tensor-core unit reads
    // 48 KB of W12, its partial is M x 512 B)
    const int64_t min_iters = q.tc ? tc_min_iters(M) : W12_FMA_MIN_ITERS;
    const int fma_sms = std::max(1, sms * fma_ctas_per_sm(q.mt) - std::min(W12_FMA_SM_RESERVE, sms / 8));
    const int tc_sms = std::max(1, sms - std::min(W12_TC_SM_RESERVE, sms / 8));
    q.grid = choose_grid(q.n_rowblk, q.n_kstep, q.tc ? tc_sms : fma_sms, min_iters);
    q.part_bytes = sizeof(float) * 2 * static_cast<size_t>(q.grid) * M * q.rows_blk;
    *p = q;
    return W12_OK;
}

} // namespace w12

namespace {

// One launch over n matrices (1 <= n <= kMaxGroup) that read the same x:
// y_i[M][N_i] = x[M][K] . W_i^T.
w12_status gemm_group_impl(const void *x, const w12_dev *const *ws, void *const *ys, int n, int M, int K,
                           cudaStream_t st, bool q8, bool x_ready, int out_mode)
{
    if (n < 1 || n > kMaxGroup || !ws || !ys || M < 0)
        return W12_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (!ws[i])
            return W12_ERR_INVALID_ARG;
        if (K != ws[i]->K)
            return W12_ERR_SHAPE;
        if ((out_mode & kOutSiluMul) && (ws[i]->N & 1))
            return W12_ERR_SHAPE;
    }
    if (M > kMaxM)
        return W12_ERR_UNSUPPORTED;
    if (M == 0)
        return W12_OK;
    if (!x || !aligned16(x))
        return x ? W12_ERR_ALIGNMENT : W12_ERR_INVALID_ARG;
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess)
        return cuda_fail(e);
    int64_t Ns[kMaxGroup] = {0};
    for (int i = 0; i < n; ++i) {
        if (ws[i]->N > 0 && !ys[i])
            return W12_ERR_INVALID_ARG;
        if (ys[i] && !aligned16(ys[i]))
            return W12_ERR_ALIGNMENT;
        if (ws[i]->device != cur)
            return W12_ERR_INVALID_ARG;
        Ns[i] = ws[i]->N;
    }
    if (K == 0) {
        for (int i = 0; i < n; ++i) {
            const int64_t ldy = (out_mode & kOutSiluMul) ? Ns[i] / 2 : Ns[i];
            const size_t ybytes = ((out_mode & kOutBF16) ? 2 : 4) * static_cast<size_t>(M) * ldy;
            if (ybytes && (e = cudaMemsetAsync(ys[i], 0, ybytes, st)) != cudaSuccess)
                return cuda_fail(e);
        }
        return W12_OK;
    }
    for (int i = 0; i < n; ++i)
        if (Ns[i] > 0 && !ws[i]->gemm_ok)
            return W12_ERR_UNSUPPORTED;

    Plan pl;
    const w12_status ps = make_plan_group(M, Ns, n, K, sm_count(cur), &pl);
    if (ps != W12_OK)
        return ps;
    if (pl.n_rowblk == 0)
        return W12_OK;
    GemmArgs a{};
    TmapSet tm;
    int rb = 0, g = 0;
    for (int i = 0; i < n; ++i) {
        if (Ns[i] == 0)
            continue; // no rows: nothing to compute or store
        const w12_dev *w = ws[i];
        MatArgs &mm = a.mat[g];
        mm.ebase = w->ebase;
        mm.tile_ptr = w->tile_ptr;
        mm.esc = w->esc;
        mm.n_esc = static_cast<uint32_t>(w->n_esc);
        mm.gptr = w->gptr;
        mm.y = ys[i];
        mm.status = w->status;
        mm.N = static_cast<int>(Ns[i]);
        mm.ldy = (out_mode & kOutSiluMul) ? mm.N / 2 : mm.N;
        mm.rb0 = rb;
        rb += static_cast<int>(ceil_div(Ns[i], pl.rows_blk));
        const w12_tmap &tae = pl.tc ? w->tm_ae_tc : (pl.rows_blk == 128 ? w->tm_ae_fma128 : w->tm_ae_fma64);
        const w12_tmap &tb = pl.tc ? w->tm_b_tc : (pl.rows_blk == 128 ? w->tm_b_fma128 : w->tm_b_fma64);
        tm.ae[g] = *tmap_of(tae);
        tm.b[g] = *tmap_of(tb);
        ++g;
    }
    a.n_mat = g;
    for (int i = g; i < kMaxGroup; ++i)
        a.mat[i] = a.mat[0];
    a.out_mode = out_mode;
    a.M = M;
    a.K = K;
    a.tiles_c = static_cast<int>(ws[0]->tiles_c);
    a.n_rowblk = static_cast<int>(pl.n_rowblk);
    a.n_kstep = static_cast<int>(pl.n_kstep);
    a.total_iters = static_cast<int>(pl.iters);
    a.limit_ns = spin_limit_ns();
    a.inject_stall = inject_stall();
    a.x_ready = x_ready ? 1 : 0;
    a.defer = pl.defer;

    w12_status wst = get_workspace(cur, st, pl.part_bytes, &a.partials, &a.counters);
    if (wst != W12_OK)
        return wst;
    if (!make_x_tmap(&tm.x, x, M, K, pl.tc, pl.mt)) {
        g_last_error = "cuTensorMapEncodeTiled failed for x";
        return W12_ERR_CUDA;
    }
    if (pl.tc) {
        e = launch_gemm_tc(pl.mt, q8, false, a, tm, pl.grid, st);
        bool red = false;
        if (e == cudaSuccess && a.defer)
            e = launch_sk_reduce(a, pl.grid, pl.rows_blk, st, &red);
    } else {
        e = launch_gemm_fma(pl.mt, q8, a, tm, pl.grid, st);
    }
    return e == cudaSuccess ? W12_OK : cuda_fail(e);
}

w12_status gemm_impl(const void *x, const w12_dev *w, void *y, int M, int N, int K,
                     cudaStream_t st, bool q8, bool x_ready = false, int out_mode = 0)
{
    if (!w || M < 0)
        return W12_ERR_INVALID_ARG;
    if (N != w->N || K != w->K)
        return W12_ERR_SHAPE;
    if (M > kMaxM)
        return W12_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return W12_OK;
    if (!x || !y)
        return W12_ERR_INVALID_ARG;
    return gemm_group_impl(x, &w, &y, 1, M, K, st, q8, x_ready, out_mode);
}

} // namespace

namespace w12 {

// A device handle for an N x K matrix with n_esc escapes: one allocation
// holding every array (256-byte aligned), the status word cleared on
// `stream`, and the TMA descriptors of both GEMM kernels when K allows them
// (rows of both planes must start on 16-byte boundaries: K % 32 == 0).
w12_status dev_create(int64_t N, int64_t K, int64_t n_esc, cudaStream_t st, w12_dev **out)
{
    *out = nullptr;
    w12_dev *d = new (std::nothrow) w12_dev;
    if (!d)
        return W12_ERR_OOM;
    if (cudaGetDevice(&d->device) != cudaSuccess) {
        delete d;
        return W12_ERR_CUDA;
    }
    d->N = N;
    d->K = K;
    d->T = num_tiles(N, K);
    d->n_esc = n_esc;
    d->brow = b_row_bytes(K);
    d->tiles_c = ceil_div(K, kTileCols);
    auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    const size_t s_status = 256, s_ebase = up(static_cast<size_t>(N)), s_ae = up(static_cast<size_t>(N * K)),
                 s_b = up(static_cast<size_t>(N * d->brow)), s_ptr = up(4 * static_cast<size_t>(d->T + 1)),
                 s_esc = up(4 * static_cast<size_t>(n_esc)), s_gp = up(32 * static_cast<size_t>(d->T));
    d->bytes = s_status + s_ebase + s_ae + s_b + s_ptr + s_esc + s_gp;
    if (cudaMalloc(&d->base, d->bytes) != cudaSuccess) {
        cudaGetLastError();
        delete d;
        return W12_ERR_OOM;
    }
    char *p = static_cast<char *>(d->base);
    d->status = reinterpret_cast<int *>(p);
    p += s_status;
    d->ebase = reinterpret_cast<uint8_t *>(p);
    p += s_ebase;
    d->ae = reinterpret_cast<uint8_t *>(p);
    p += s_ae;
    d->b = reinterpret_cast<uint8_t *>(p);
    p += s_b;
    d->tile_ptr = reinterpret_cast<uint32_t *>(p);
    p += s_ptr;
    d->esc = reinterpret_cast<uint32_t *>(p);
    p += s_esc;
    d->gptr = reinterpret_cast<uint16_t *>(p);
    if (cudaMemsetAsync(d->status, 0, 256, st) != cudaSuccess) {
        cudaFree(d->base);
        delete d;
        return W12_ERR_CUDA;
    }
    if (N > 0 && K >= 32 && K % 32 == 0) {
        const uint64_t n = N, k = K;
        const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        bool t = make_tmap(tmap_of(d->tm_ae_fma128), U8, 1, d->ae, k, n, 256, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
        t = t && make_tmap(tmap_of(d->tm_ae_fma64), U8, 1, d->ae, k, n, 256, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
        t = t && make_tmap(tmap_of(d->tm_b_fma128), U8, 1, d->b, k / 2, n, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
        t = t && make_tmap(tmap_of(d->tm_b_fma64), U8, 1, d->b, k / 2, n, 128, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
        t = t && make_tmap(tmap_of(d->tm_ae_tc), U8, 1, d->ae, k, n, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        t = t && make_tmap(tmap_of(d->tm_b_tc), U8, 1, d->b, k / 2, n, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        d->gemm_ok = t;
    }
    *out = d;
    return W12_OK;
}

} // namespace w12

extern "C" {

w12_status w12_upload(const w12_host *h, w12_stream_t stream, w12_dev **out)
{
    if (!h || !out)
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    w12_dev *d = nullptr;
    w12_status s = w12::dev_create(h->N, h->K, static_cast<int64_t>(h->esc.size()), st, &d);
    if (s != W12_OK)
        return s;
    // row-group index of every escape tile: gp[t][g] = entries of tile t whose
    // row (within the tile) is below 8g, so the entries of rows [8g, 8g+8) are
    // [gp[t][g], gp[t][g+1]) (gp[t][16] being the tile's count)
    std::vector<uint16_t> gp;
    try {
        gp.assign(16 * static_cast<size_t>(d->T), 0);
    } catch (...) {
        w12_dev_free(d);
        return W12_ERR_OOM;
    }
    for (int64_t t = 0; t < d->T; ++t) {
        const uint32_t lo = h->tile_ptr[t], hi = h->tile_ptr[t + 1];
        uint32_t i = lo;
        for (int g = 0; g < 16; ++g) {
            while (i < hi && (h->esc[i] >> 24) < static_cast<uint32_t>(8 * g))
                ++i;
            gp[16 * t + g] = static_cast<uint16_t>(i - lo);
        }
    }
    bool ok = true;
    auto cp = [&](void *dst, const void *src, size_t n) {
        if (n)
            ok = ok && cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
    };
    cp(d->ebase, h->ebase.data(), h->ebase.size());
    cp(d->ae, h->ae.data(), h->ae.size());
    cp(d->b, h->b.data(), h->b.size());
    cp(d->tile_ptr, h->tile_ptr.data(), 4 * h->tile_ptr.size());
    cp(d->esc, h->esc.data(), 4 * h->esc.size());
    cp(d->gptr, gp.data(), 2 * gp.size());
    if (ok && !gp.empty())
        ok = cudaStreamSynchronize(st) == cudaSuccess; // gp is a local staging buffer
    if (!ok) {
        w12_dev_free(d);
        return W12_ERR_CUDA;
    }
    *out = d;
    return W12_OK;
}

void w12_dev_free(w12_dev *d)
{
    if (!d)
        return;
    cudaDeviceSynchronize();
    cudaFree(d->base);
    delete d;
}

w12_status w12_dev_info(const w12_dev *d, int64_t *N, int64_t *K, size_t *device_bytes)
{
    if (!d)
        return W12_ERR_INVALID_ARG;
    if (N)
        *N = d->N;
    if (K)
        *K = d->K;
    if (device_bytes)
        *device_bytes = d->bytes;
    return W12_OK;
}

w12_status w12_gemm(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                     w12_stream_t stream)
{
    return gemm_impl(x_bf16, w, y, M, N, K, reinterpret_cast<cudaStream_t>(stream), false);
}

w12_status w12_gemm_q8view(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                           w12_stream_t stream)
{
    return gemm_impl(x_bf16, w, y, M, N, K, reinterpret_cast<cudaStream_t>(stream), true);
}

w12_status w12_gemm_plan_grouped(int M, const int64_t *Ns, int n, int64_t K, int sm_count_arg,
                                 w12_gemm_plan_t *out)
{
    if (!out || !Ns || n < 1 || n > kMaxGroup || M < 0 || K < 0)
        return W12_ERR_INVALID_ARG;
    *out = w12_gemm_plan_t{};
    int64_t rows = 0;
    for (int i = 0; i < n; ++i) {
        if (Ns[i] < 0)
            return W12_ERR_INVALID_ARG;
        if (Ns[i] > (int64_t(1) << 31))
            return W12_ERR_UNSUPPORTED;
        rows += Ns[i];
    }
    if (M > kMaxM || K > (int64_t(1) << 31))
        return W12_ERR_UNSUPPORTED;
    if (M == 0 || rows == 0 || K == 0)
        return W12_OK; // nothing is launched
    if (K % 32 != 0)
        return W12_ERR_UNSUPPORTED;
    int sms = sm_count_arg;
    if (sms <= 0) {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess)
            return W12_ERR_CUDA;
        sms = sm_count(cur);
        if (sms <= 0)
            return W12_ERR_CUDA;
    }
    Plan pl;
    const w12_status ps = make_plan_group(M, Ns, n, K, sms, &pl);
    if (ps != W12_OK)
        return ps;
    out->kernel = pl.tc ? 2 : 1;
    out->tile_rows = pl.mt;
    out->block_rows = pl.rows_blk;
    out->grid = pl.grid;
    out->row_blocks = pl.n_rowblk;
    out->k_steps = pl.n_kstep;
    int64_t split = 0;
    const int it = static_cast<int>(pl.iters);
    for (int64_t rb = 0; rb < pl.n_rowblk; ++rb)
        if (sk_owner(static_cast<int>(rb * pl.n_kstep), pl.grid, it) !=
            sk_owner(static_cast<int>((rb + 1) * pl.n_kstep - 1), pl.grid, it))
            ++split;
    out->split_row_blocks = split;
    out->separate_fixup = pl.defer && split > 0 ? 1 : 0;
    out->partial_bytes = split > 0 ? pl.part_bytes : 0;
    return W12_OK;
}

w12_status w12_gemm_plan(int M, int64_t N, int64_t K, int sm_count_arg, w12_gemm_plan_t *out)
{
    if (!out || M < 0 || N < 0 || K < 0)
        return W12_ERR_INVALID_ARG;
    return w12_gemm_plan_grouped(M, &N, 1, K, sm_count_arg, out);
}

w12_status w12_gemm_ex(const void *x_bf16, const w12_dev *w, void *y, int M, int N, int K,
                       unsigned flags, w12_stream_t stream)
{
    if (flags & ~static_cast<unsigned>(W12_GEMM_Q8VIEW | W12_GEMM_INPUT_READY | W12_GEMM_OUT_BF16 |
                                       W12_GEMM_SILU_MUL))
        return W12_ERR_INVALID_ARG;
    const int out_mode = ((flags & W12_GEMM_OUT_BF16) ? kOutBF16 : 0) | ((flags & W12_GEMM_SILU_MUL) ? kOutSiluMul : 0);
    return gemm_impl(x_bf16, w, y, M, N, K, reinterpret_cast<cudaStream_t>(stream),
                     (flags & W12_GEMM_Q8VIEW) != 0, (flags & W12_GEMM_INPUT_READY) != 0, out_mode);
}

w12_status w12_gemm_grouped(const void *x_bf16, const w12_dev *const *ws, void *const *ys, int n, int M, int K,
                            unsigned flags, w12_stream_t stream)
{
    if (flags & ~static_cast<unsigned>(W12_GEMM_Q8VIEW | W12_GEMM_INPUT_READY | W12_GEMM_OUT_BF16))
        return W12_ERR_INVALID_ARG;
    const int out_mode = (flags & W12_GEMM_OUT_BF16) ? kOutBF16 : 0;
    return gemm_group_impl(x_bf16, ws, ys, n, M, K, reinterpret_cast<cudaStream_t>(stream),
                           (flags & W12_GEMM_Q8VIEW) != 0, (flags & W12_GEMM_INPUT_READY) != 0, out_mode);
}

w12_status w12_gemm_host(const uint16_t *x_host, void *x_dev, const w12_dev *w, float *y_dev,
                         float *y_host, int M, int N, int K, w12_stream_t stream)
{
    if (!w || M < 0 || N < 0 || K < 0)
        return W12_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return W12_OK;
    if (!x_host || !x_dev || !y_dev || !y_host)
        return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, sizeof(uint16_t) * static_cast<size_t>(M) * K,
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const w12_status s = gemm_impl(x_dev, w, y_dev, M, N, K, st, false);
    if (s != W12_OK)
        return s;
    e = cudaMemcpyAsync(y_host, y_dev, sizeof(float) * static_cast<size_t>(M) * N, cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? W12_OK : cuda_fail(e);
}

w12_status w12_gemm_grouped_host(const uint16_t *x_host, void *x_dev, const w12_dev *const *ws,
                                 void *const *ys_dev, void *const *ys_host, int n, int M, int K, unsigned flags,
                                 w12_stream_t stream)
{
    if (n < 1 || n > kMaxGroup || !ws || !ys_dev || !ys_host || M < 0 || K < 0)
        return W12_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!ws[i] || (M > 0 && ws[i]->N > 0 && !ys_host[i]))
            return W12_ERR_INVALID_ARG;
    if (M == 0)
        return W12_OK;
    if (!x_host || !x_dev)
        return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, sizeof(uint16_t) * static_cast<size_t>(M) * K,
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const w12_status s = w12_gemm_grouped(x_dev, ws, ys_dev, n, M, K, flags, stream);
    if (s != W12_OK)
        return s;
    // outputs that lie end to end both on the device and on the host go
    // back in one copy (a run of small copies costs a round trip each)
    const size_t elem = (flags & W12_GEMM_OUT_BF16) ? 2 : 4;
    for (int i = 0; i < n;) {
        char *dst = static_cast<char *>(ys_host[i]);
        const char *src = static_cast<const char *>(ys_dev[i]);
        size_t bytes = elem * static_cast<size_t>(M) * ws[i]->N;
        int j = i + 1;
        while (j < n && ys_host[j] == dst + bytes && ys_dev[j] == src + bytes) {
            bytes += elem * static_cast<size_t>(M) * ws[j]->N;
            ++j;
        }
        if (bytes && (e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
            return cuda_fail(e);
        i = j;
    }
    return W12_OK;
}

w12_status w12_decode(const w12_dev *w, uint16_t *out, w12_stream_t stream)
{
    if (!w || (!out && w->N * w->K > 0))
        return W12_ERR_INVALID_ARG;
    if (w->N * w->K == 0)
        return W12_OK;
    if (w->K % 8 == 0 && !aligned16(out))
        return W12_ERR_ALIGNMENT;
    return launch_decode(w->ebase, w->ae, w->b, w->tile_ptr, w->esc, out, w->N, w->K,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

w12_status w12_dev_status(const w12_dev *w, w12_stream_t stream)
{
    if (!w)
        return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cudaMemcpy(&v, w->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return W12_ERR_CUDA;
    if (v != 0 && cudaMemset(w->status, 0, sizeof v) != cudaSuccess)
        return W12_ERR_CUDA;
    return static_cast<w12_status>(v);
}

w12_status w12_release_workspaces(void)
{
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return W12_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto it = g_ws.begin(); it != g_ws.end();) {
        if (it->first.first == cur) {
            if (it->second.ptr)
                cudaFree(it->second.ptr);
            it = g_ws.erase(it);
        } else {
            ++it;
        }
    }
    for (auto it = g_ws_retired.begin(); it != g_ws_retired.end();) {
        if (it->first == cur) {
            cudaFree(it->second);
            it = g_ws_retired.erase(it);
        } else {
            ++it;
        }
    }
    return W12_OK;
}

void w12_set_spin_limit(uint32_t limit_ns)
{
    g_limit_ns.store(limit_ns ? limit_ns : 200ull * 1000 * 1000);
}

void w12_debug_inject_stall(int on) { g_inject_stall.store(on ? 1 : 0); }

const char *w12_last_cuda_error(void) { return g_last_error; }

} // extern "C"

// ---- INT8 copy for the Q pass ------------------------------------------------

namespace {

w12_status i8_create(int64_t N, int64_t K, cudaStream_t st, w12_i8 **out)
{
    *out = nullptr;
    w12_i8 *q = new (std::nothrow) w12_i8;
    if (!q)
        return W12_ERR_OOM;
    if (cudaGetDevice(&q->device) != cudaSuccess) {
        delete q;
        return W12_ERR_CUDA;
    }
    q->N = N;
    q->K = K;
    auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    const size_t s_status = 256, s_q = up(static_cast<size_t>(N * K)), s_sc = up(4 * static_cast<size_t>(N));
    q->bytes = s_status + s_q + s_sc;
    if (cudaMalloc(&q->base, q->bytes) != cudaSuccess) {
        cudaGetLastError();
        delete q;
        return W12_ERR_OOM;
    }
    char *p = static_cast<char *>(q->base);
    q->status = reinterpret_cast<int *>(p);
    q->q = reinterpret_cast<int8_t *>(p + s_status);
    q->scale = reinterpret_cast<float *>(p + s_status + s_q);
    if (cudaMemsetAsync(q->status, 0, 256, st) != cudaSuccess) {
        cudaFree(q->base);
        delete q;
        return W12_ERR_CUDA;
    }
    if (N > 0 && K >= 32 && K % 32 == 0)
        q->gemm_ok = make_tmap(tmap_of(q->tm_q_tc), CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q->q, K, N, 128, 128,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    *out = q;
    return W12_OK;
}

w12_status gemm_i8_impl(const void *x, const w12_i8 *q, void *y, int M, int N, int K, cudaStream_t st,
                        bool x_ready, int out_mode)
{
    if (!q || M < 0)
        return W12_ERR_INVALID_ARG;
    if (N != q->N || K != q->K)
        return W12_ERR_SHAPE;
    if ((out_mode & kOutSiluMul) && (N & 1))
        return W12_ERR_SHAPE;
    const int ldy = (out_mode & kOutSiluMul) ? N / 2 : N;
    const size_t esz = (out_mode & kOutBF16) ? 2 : 4;
    if (M > kMaxM)
        return W12_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return W12_OK;
    if (!x || !y)
        return W12_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y))
        return W12_ERR_ALIGNMENT;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cur != q->device)
        return W12_ERR_INVALID_ARG;
    if (K == 0)
        return cudaMemsetAsync(y, 0, esz * static_cast<size_t>(M) * ldy, st) == cudaSuccess ? W12_OK : W12_ERR_CUDA;
    if (!q->gemm_ok)
        return W12_ERR_UNSUPPORTED;
    // the tensor-core kernel for every M (M padded to 16, 32, 64, 128 or 256)
    const int mt = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    GemmArgs a{};
    MatArgs &mm = a.mat[0];
    mm.y = y;
    mm.ldy = ldy;
    mm.scale = q->scale;
    mm.status = q->status;
    mm.N = N;
    mm.rb0 = 0;
    a.n_mat = 1;
    for (int i = 1; i < kMaxGroup; ++i)
        a.mat[i] = a.mat[0];
    a.out_mode = out_mode;
    a.M = M;
    a.K = K;
    a.tiles_c = static_cast<int>(ceil_div(K, kTileCols));
    a.n_rowblk = static_cast<int>(ceil_div(N, kTcRows));
    a.n_kstep = static_cast<int>(ceil_div(K, kTcKStep));
    const int64_t iters = static_cast<int64_t>(a.n_rowblk) * a.n_kstep;
    if (iters > (1ll << 30) || a.n_rowblk * 8 > static_cast<int64_t>(kCounterBytes))
        return W12_ERR_UNSUPPORTED;
    a.total_iters = static_cast<int>(iters);
    a.limit_ns = spin_limit_ns();
    a.inject_stall = inject_stall();
    a.x_ready = x_ready ? 1 : 0;
    a.defer = tc_defer(M);
    const int grid = choose_grid(a.n_rowblk, a.n_kstep, sm_count(cur), tc_min_iters(M));
    const size_t part_bytes = sizeof(float) * 2 * static_cast<size_t>(grid) * M * kTcRows;
    w12_status ws = get_workspace(cur, st, part_bytes, &a.partials, &a.counters);
    if (ws != W12_OK)
        return ws;
    TmapSet tm;
    if (!make_x_tmap(&tm.x, x, M, K, true, mt)) {
        g_last_error = "cuTensorMapEncodeTiled failed for x";
        return W12_ERR_CUDA;
    }
    tm.ae[0] = *tmap_of(q->tm_q_tc);
    tm.b[0] = tm.ae[0];
    cudaError_t e = launch_gemm_tc(mt, true, true, a, tm, grid, st);
    bool red = false;
    if (e == cudaSuccess && a.defer)
        e = launch_sk_reduce(a, grid, kTcRows, st, &red);
    return e == cudaSuccess ? W12_OK : cuda_fail(e);
}

} // namespace

extern "C" {

w12_status w12_i8_encode_device(const void *w_bf16, int64_t N, int64_t K, w12_stream_t stream, w12_i8 **out)
{
    if (!out || N < 0 || K < 0 || (N * K > 0 && !w_bf16))
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return W12_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    w12_i8 *q = nullptr;
    w12_status r = i8_create(N, K, st, &q);
    if (r != W12_OK)
        return r;
    if (launch_i8_quantize(static_cast<const uint16_t *>(w_bf16), N, K, q->q, q->scale, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        w12_i8_free(q);
        return W12_ERR_CUDA;
    }
    *out = q;
    return W12_OK;
}

w12_status w12_i8_from_dev(const w12_dev *w, w12_stream_t stream, w12_i8 **out)
{
    if (!w || !out)
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *tmp = nullptr;
    const size_t bytes = 2 * static_cast<size_t>(w->N) * static_cast<size_t>(w->K);
    if (bytes && cudaMallocAsync(&tmp, bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return W12_ERR_OOM;
    }
    w12_status r = w12_decode(w, static_cast<uint16_t *>(tmp), stream);
    if (r == W12_OK)
        r = w12_i8_encode_device(tmp, w->N, w->K, stream, out);
    if (tmp)
        cudaFreeAsync(tmp, st);
    return r;
}

void w12_i8_free(w12_i8 *q)
{
    if (!q)
        return;
    cudaFree(q->base);
    delete q;
}

w12_status w12_i8_download(const w12_i8 *q, int8_t *q_host, float *scale_host, w12_stream_t stream)
{
    if (!q)
        return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool ok = true;
    if (q_host && q->N * q->K > 0)
        ok = cudaMemcpyAsync(q_host, q->q, static_cast<size_t>(q->N * q->K), cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && scale_host && q->N > 0)
        ok = cudaMemcpyAsync(scale_host, q->scale, 4 * static_cast<size_t>(q->N), cudaMemcpyDeviceToHost, st) ==
             cudaSuccess;
    return ok && cudaStreamSynchronize(st) == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

w12_status w12_i8_status(const w12_i8 *q, w12_stream_t stream)
{
    if (!q)
        return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cudaMemcpy(&v, q->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return W12_ERR_CUDA;
    if (v != 0 && cudaMemset(q->status, 0, sizeof v) != cudaSuccess)
        return W12_ERR_CUDA;
    return static_cast<w12_status>(v);
}

w12_status w12_gemm_i8(const void *x_bf16, const w12_i8 *q, void *y, int M, int N, int K, unsigned flags,
                       w12_stream_t stream)
{
    if (flags & ~static_cast<unsigned>(W12_GEMM_INPUT_READY | W12_GEMM_OUT_BF16 | W12_GEMM_SILU_MUL))
        return W12_ERR_INVALID_ARG;
    const int out_mode = ((flags & W12_GEMM_OUT_BF16) ? kOutBF16 : 0) | ((flags & W12_GEMM_SILU_MUL) ? kOutSiluMul : 0);
    return gemm_i8_impl(x_bf16, q, y, M, N, K, reinterpret_cast<cudaStream_t>(stream),
                        (flags & W12_GEMM_INPUT_READY) != 0, out_mode);
}

} // extern "C"
