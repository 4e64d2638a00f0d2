// encode.cu -- W12 encoding on the device: BF16 weights already in device
// memory become a device W12 handle without a round trip through the host.
//
// The format is the host encoder's (SpecPilot, Figure 5(a) caption): per BF16
// weight A = sign + mantissa bits 6..4, E = exponent offset inside the 16-binade
// window of its row (ebase = max(emax, 16) - 15, emax the row's largest finite
// exponent field), B = mantissa bits 3..0; zeros, subnormals, Inf, NaN and
// anything below the window are escapes, listed per 128 x 256 tile as
// (row % 128) << 24 | (k % 256) << 16 | bits in (row, k) order, their slot
// holding A = s << 3, E = 0, B = 0.  With W12_ENCODE_COUNT_MAX a row's window
// is the one holding the most finite normal weights (the highest such base at
// or below the max-anchored one), and weights above it escape with the
// saturated placeholder A = s << 3 | 7, E = 15, B = 15.  The arrays come out
// byte-identical to the host encoder's with the same flags.
//
// Three passes over the weights:
//   1. window bases: one warp per row, maximum exponent field below 255 (and
//      for count-maximising windows an exponent histogram in shared memory,
//      then the best 16-binade window sum, one candidate base per lane);
//   2. escape counts: one CTA per tile, counts per 8-row group;
//   3. (after an exclusive prefix of the tile counts, and the allocation of
//      the handle, whose size depends on the total) the AE and B planes and
//      the escape entries: one CTA per tile, a warp per row, a lane per group
//      of 8 weights; an entry's place is the tile's start + the escapes of the
//      tile's earlier rows + those of its row before it.
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

constexpr int kEncThreads = 256; // 8 warps

__device__ __forceinline__ bool is_escape(uint32_t bits, uint32_t eb)
{
    const uint32_t e = (bits >> 7) & 0xFFu;
    return e < eb || e > eb + 15u; // ebase >= 1 and ebase + 15 <= 254: exponent 0 and 255 always escape
}

// 1. ebase[n] for every row.
__global__ void __launch_bounds__(kEncThreads) enc_rows_kernel(const uint16_t *w, int64_t N, int64_t K,
                                                               uint8_t *ebase, int count_max)
{
    __shared__ uint32_t hist_s[kEncThreads / 32][256];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * (kEncThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N)
        return;
    const uint16_t *row = w + n * K;
    uint32_t *hist = hist_s[threadIdx.x >> 5];
    if (count_max) {
        for (int e = lane; e < 256; e += 32)
            hist[e] = 0;
        __syncwarp();
    }
    uint32_t emax = 16; // floor: ebase >= 1 even for rows without normals
    for (int64_t k = lane; k < K; k += 32) {
        const uint32_t e = (row[k] >> 7) & 0xFFu;
        if (e != 0xFFu && e > emax)
            emax = e;
        if (count_max && e != 0 && e != 0xFFu)
            atomicAdd(hist + e, 1u);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    uint32_t eb = emax - 15;
    if (count_max) {
        __syncwarp();
        // lane l tries bases l + 1, l + 33, ... up to the max-anchored one; the
        // best (count, base) pair wins, higher base on equal counts
        uint32_t best = 0, best_b = 0;
        for (uint32_t b = lane + 1; b <= eb; b += 32) {
            uint32_t c = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                c += hist[b + i];
            if (best_b == 0 || c >= best) {
                best = c;
                best_b = b;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const uint32_t oc = __shfl_xor_sync(0xffffffffu, best, o);
            const uint32_t ob = __shfl_xor_sync(0xffffffffu, best_b, o);
            if (ob != 0 && (best_b == 0 || oc > best || (oc == best && ob > best_b))) {
                best = oc;
                best_b = ob;
            }
        }
        eb = best_b;
    }
    if (lane == 0)
        ebase[n] = static_cast<uint8_t>(eb);
}

// Escape mask of the (up to) 8 weights of group g of row n (bit j: weight 8g+j),
// with the weights themselves.
__device__ __forceinline__ uint32_t group_escapes(const uint16_t *row, int64_t K, int64_t g, uint32_t eb,
                                                  uint16_t (&v)[8])
{
    uint32_t mask = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t k = 8 * g + j;
        v[j] = k < K ? row[k] : 0;
        if (k < K && is_escape(v[j], eb))
            mask |= 1u << j;
    }
    return mask;
}

// 2. escape count of every 8-row group of every tile: cnt[16 t + g].
__global__ void __launch_bounds__(kEncThreads) enc_count_kernel(const uint16_t *w, int64_t N, int64_t K,
                                                                int64_t tiles_c, const uint8_t *ebase,
                                                                uint32_t *cnt)
{
    const int64_t t = blockIdx.x;
    const int64_t r0 = (t / tiles_c) * kTileRows, g0 = (t % tiles_c) * (kTileCols / 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // warp w takes rows 16w .. 16w + 15 of the tile = row groups 2w and 2w + 1
    uint32_t c[2] = {0u, 0u};
    for (int r = 0; r < 16; ++r) {
        const int64_t n = r0 + 16 * warp + r;
        if (n >= N)
            break;
        const int64_t g = g0 + lane;
        uint32_t m = 0;
        if (8 * g < K) {
            uint16_t v[8];
            m = group_escapes(w + n * K, K, g, ebase[n], v);
        }
        c[r >> 3] += __popc(m);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            c[h] += __shfl_xor_sync(0xffffffffu, c[h], o);
    }
    if (lane == 0) {
        cnt[16 * t + 2 * warp] = c[0];
        cnt[16 * t + 2 * warp + 1] = c[1];
    }
}

// Exclusive prefix of the tile totals (one CTA): tile_ptr[t] = entries of
// tiles < t, tile_ptr[T] = all of them.
__global__ void __launch_bounds__(1024) enc_scan_kernel(const uint32_t *cnt, int64_t T, uint32_t *tile_ptr)
{
    __shared__ uint32_t part[32];
    __shared__ uint32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < T; base += 1024) {
        const int64_t t = base + tid;
        uint32_t v = 0;
        if (t < T) {
#pragma unroll
            for (int g = 0; g < 16; ++g)
                v += cnt[16 * t + g];
        }
        // inclusive scan inside the warp, then over the warps
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            part[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t p = part[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, p, o);
                if (lane >= o)
                    p += y;
            }
            part[lane] = p; // inclusive over warps
        }
        __syncthreads();
        const uint32_t before = carry + (warp ? part[warp - 1] : 0u) + x - v;
        if (t < T)
            tile_ptr[t] = before;
        __syncthreads();
        if (tid == 1023)
            carry = before + v;
        __syncthreads();
    }
    if (tid == 0)
        tile_ptr[T] = carry;
}

// 3. AE and B planes, escape entries and the row-group index of every tile.
__global__ void __launch_bounds__(kEncThreads) enc_fill_kernel(const uint16_t *w, int64_t N, int64_t K,
                                                               int64_t tiles_c, int64_t brow,
                                                               const uint8_t *ebase, const uint32_t *tile_ptr,
                                                               uint8_t *ae, uint8_t *bpl, uint32_t *esc,
                                                               uint16_t *gptr)
{
    __shared__ uint32_t row_cnt[kTileRows];
    const int64_t t = blockIdx.x;
    const int64_t r0 = (t / tiles_c) * kTileRows, g0 = (t % tiles_c) * (kTileCols / 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = g0 + lane; // this lane's group of 8 columns
    const bool gv = 8 * g < K;
    // escapes per row of the tile
    for (int r = warp; r < kTileRows; r += kEncThreads / 32) {
        const int64_t n = r0 + r;
        uint32_t m = 0;
        if (n < N && gv) {
            uint16_t v[8];
            m = group_escapes(w + n * K, K, g, ebase[n], v);
        }
        uint32_t c = __popc(m);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0)
            row_cnt[r] = c;
    }
    __syncthreads();
    // exclusive prefix over the tile's rows (warp 0), and the row-group index
    if (warp == 0) {
        uint32_t v[4], s = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = row_cnt[4 * lane + i];
            s += v[i];
        }
        uint32_t x = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        uint32_t before = x - s;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            row_cnt[4 * lane + i] = before;
            before += v[i];
        }
        __syncwarp();
        if (lane < 16)
            gptr[16 * t + lane] = static_cast<uint16_t>(row_cnt[8 * lane]);
    }
    __syncthreads();
    const uint32_t tbase = tile_ptr[t];
    for (int r = warp; r < kTileRows; r += kEncThreads / 32) {
        const int64_t n = r0 + r;
        if (n >= N)
            break;
        const uint32_t eb = ebase[n];
        uint16_t v[8];
        uint32_t m = 0;
        if (gv)
            m = group_escapes(w + n * K, K, g, eb, v);
        // this lane's escapes come after those of the row's lanes before it
        const uint32_t c = __popc(m);
        uint32_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        uint32_t pos = tbase + row_cnt[r] + x - c;
        if (!gv)
            continue;
        uint8_t a8[8];
        uint32_t bword = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t bits = v[j];
            const uint32_t s = bits >> 15;
            if ((m >> j) & 1u) {
                // placeholder A = s << 3, E = 0, B = 0; above the window (count-
                // maximising windows only) the saturated A = s << 3 | 7, E = 15, B = 15
                const uint32_t e = (bits >> 7) & 0xFFu;
                const bool above = e != 0xFFu && e > eb + 15u;
                a8[j] = static_cast<uint8_t>(above ? ((s << 7) | 0x7Fu) : ((s << 3) << 4));
                if (above)
                    bword |= 0xFu << (4 * ((j >> 1) + 4 * (j & 1)));
                esc[pos++] = (static_cast<uint32_t>(r) << 24) | (static_cast<uint32_t>((8 * g + j) % kTileCols) << 16) | bits;
            } else {
                const uint32_t e = (bits >> 7) & 0xFFu, mant = bits & 0x7Fu;
                a8[j] = static_cast<uint8_t>((((s << 3) | (mant >> 4)) << 4) | (e - eb));
                bword |= (mant & 0xFu) << (4 * ((j >> 1) + 4 * (j & 1)));
            }
        }
        uint8_t *ae_row = ae + n * K + 8 * g;
        const int64_t kend = K - 8 * g < 8 ? K - 8 * g : 8;
        for (int j = 0; j < kend; ++j)
            ae_row[j] = a8[j];
        *reinterpret_cast<uint32_t *>(bpl + n * brow + 4 * g) = bword;
    }
}

} // namespace
} // namespace w12

using namespace w12;

extern "C" w12_status w12_encode_device(const void *w_bf16, int64_t N, int64_t K, w12_stream_t stream,
                                         w12_dev **out)
{
    return w12_encode_device_ex(w_bf16, N, K, 0, stream, out);
}

extern "C" w12_status w12_encode_device_ex(const void *w_bf16, int64_t N, int64_t K, unsigned flags,
                                            w12_stream_t stream, w12_dev **out)
{
    if (!out || N < 0 || K < 0 || (N * K > 0 && !w_bf16) || (flags & ~static_cast<unsigned>(W12_ENCODE_COUNT_MAX)))
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return W12_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *w = static_cast<const uint16_t *>(w_bf16);
    const int64_t T = num_tiles(N, K), tiles_c = ceil_div(K, kTileCols), brow = b_row_bytes(K);
    // scratch: window bases, per-group counts, tile prefix
    uint8_t *eb_s = nullptr;
    uint32_t *cnt_s = nullptr, *ptr_s = nullptr;
    const size_t s_eb = (static_cast<size_t>(N) + 255) & ~static_cast<size_t>(255);
    const size_t s_cnt = 64 * static_cast<size_t>(T), s_ptr = 4 * static_cast<size_t>(T + 1);
    void *scratch = nullptr;
    if (cudaMallocAsync(&scratch, s_eb + s_cnt + s_ptr + 16, st) != cudaSuccess) {
        cudaGetLastError();
        return W12_ERR_OOM;
    }
    eb_s = static_cast<uint8_t *>(scratch);
    cnt_s = reinterpret_cast<uint32_t *>(static_cast<char *>(scratch) + s_eb);
    ptr_s = reinterpret_cast<uint32_t *>(static_cast<char *>(scratch) + s_eb + s_cnt);
    w12_status res = W12_OK;
    uint32_t total = 0;
    if (N > 0)
        enc_rows_kernel<<<static_cast<unsigned>(ceil_div(N, kEncThreads / 32)), kEncThreads, 0, st>>>(
            w, N, K, eb_s, (flags & W12_ENCODE_COUNT_MAX) ? 1 : 0);
    if (T > 0) {
        enc_count_kernel<<<static_cast<unsigned>(T), kEncThreads, 0, st>>>(w, N, K, tiles_c, eb_s, cnt_s);
        enc_scan_kernel<<<1, 1024, 0, st>>>(cnt_s, T, ptr_s);
        if (cudaMemcpyAsync(&total, ptr_s + T, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            res = W12_ERR_CUDA;
    } else if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
        res = W12_ERR_CUDA;
    }
    w12_dev *d = nullptr;
    if (res == W12_OK)
        res = dev_create(N, K, total, st, &d);
    if (res == W12_OK) {
        bool ok = true;
        if (N > 0)
            ok = cudaMemcpyAsync(d->ebase, eb_s, static_cast<size_t>(N), cudaMemcpyDeviceToDevice, st) == cudaSuccess;
        if (T > 0)
            ok = ok && cudaMemcpyAsync(d->tile_ptr, ptr_s, 4 * static_cast<size_t>(T + 1), cudaMemcpyDeviceToDevice,
                                       st) == cudaSuccess;
        else
            ok = ok && cudaMemsetAsync(d->tile_ptr, 0, 4, st) == cudaSuccess;
        if (ok && T > 0)
            enc_fill_kernel<<<static_cast<unsigned>(T), kEncThreads, 0, st>>>(w, N, K, tiles_c, brow, eb_s, ptr_s,
                                                                            d->ae, d->b, d->esc, d->gptr);
        ok = ok && cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess;
        if (!ok) {
            w12_dev_free(d);
            d = nullptr;
            res = W12_ERR_CUDA;
        }
    }
    cudaFreeAsync(scratch, st);
    *out = d;
    return res;
}

extern "C" w12_status w12_download(const w12_dev *d, w12_stream_t stream, w12_host **out)
{
    if (!d || !out)
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    w12_host *h = new (std::nothrow) w12_host;
    if (!h)
        return W12_ERR_OOM;
    try {
        h->N = d->N;
        h->K = d->K;
        h->ebase.resize(static_cast<size_t>(d->N));
        h->ae.resize(static_cast<size_t>(d->N * d->K));
        h->b.resize(static_cast<size_t>(d->N * d->brow));
        h->tile_ptr.resize(static_cast<size_t>(d->T + 1));
        h->esc.resize(static_cast<size_t>(d->n_esc));
    } catch (...) {
        delete h;
        return W12_ERR_OOM;
    }
    bool ok = true;
    auto cp = [&](void *dst, const void *src, size_t n) {
        if (n)
            ok = ok && cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    };
    cp(h->ebase.data(), d->ebase, h->ebase.size());
    cp(h->ae.data(), d->ae, h->ae.size());
    cp(h->b.data(), d->b, h->b.size());
    cp(h->tile_ptr.data(), d->tile_ptr, 4 * h->tile_ptr.size());
    cp(h->esc.data(), d->esc, 4 * h->esc.size());
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
    if (!ok) {
        delete h;
        return W12_ERR_CUDA;
    }
    *out = h;
    return W12_OK;
}
