// decode.cu -- lossless W12 -> BF16 decode on the device (round-trip checks).
//
// One CTA per 128 x 256 escape tile: 8 warps x 16 rows, lane l rebuilds
// columns 8l..8l+7 of a row from its AE bytes and B word (sign | (ebase + E)
// << 7 | top mantissa bits << 4 | B; SpecPilot, Figure 5(a) caption), then the
// CTA writes the tile's escapes over their placeholders.
#include "kernels.cuh"

namespace w12 {
namespace {

__global__ void __launch_bounds__(256) decode_kernel(const uint8_t *__restrict__ ebase,
                                                     const uint8_t *__restrict__ ae,
                                                     const uint8_t *__restrict__ bpl,
                                                     const uint32_t *__restrict__ tile_ptr,
                                                     const uint32_t *__restrict__ esc,
                                                     uint16_t *__restrict__ out, int64_t N,
                                                     int64_t K, int64_t tiles_c)
{
    const int64_t t = blockIdx.x;
    const int64_t n0 = (t / tiles_c) * 128, k0 = (t % tiles_c) * 256;
    const int64_t brow = 4 * ((K + 7) / 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t k = k0 + 8 * lane;
    const bool vec = (K % 8) == 0;
    for (int r = 0; r < 16; ++r) {
        const int64_t n = n0 + 16 * warp + r;
        if (n >= N || k >= K)
            break;
        const uint32_t eb = ebase[n];
        if (vec) {
            const uint2 aw = *reinterpret_cast<const uint2 *>(ae + n * K + k);
            const uint32_t bw = *reinterpret_cast<const uint32_t *>(bpl + n * brow + k / 2);
            const uint32_t eb2 = (eb << 7) | (eb << 23);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t src = (i < 2) ? aw.x : aw.y;
                uint32_t p;
                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(src), "r"(0u), "r"((i & 1) ? 0xB3A2u : 0x9180u));
                o[i] = (p & 0x80708070u) | ((p & 0x000F000Fu) * 128u + eb2) | ((bw >> (4 * i)) & 0x000F000Fu);
            }
            *reinterpret_cast<uint4 *>(out + n * K + k) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            const uint8_t *bw8 = bpl + n * brow + 4 * (k / 8);
            const uint32_t bw = bw8[0] | (bw8[1] << 8) | (bw8[2] << 16) | (static_cast<uint32_t>(bw8[3]) << 24);
            for (int j = 0; j < 8 && k + j < K; ++j) {
                const uint32_t a8 = ae[n * K + k + j];
                const int slot = (j & 1) ? 4 + (j >> 1) : (j >> 1);
                const uint32_t bn = (bw >> (4 * slot)) & 0xF;
                out[n * K + k + j] = static_cast<uint16_t>(((a8 >> 7) << 15) | ((eb + (a8 & 0xF)) << 7) |
                                                           (((a8 >> 4) & 7) << 4) | bn);
            }
        }
    }
    __syncthreads();
    const uint32_t lo = tile_ptr[t], hi = tile_ptr[t + 1];
    for (uint32_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const uint32_t e = esc[i];
        const int64_t n = n0 + (e >> 24), kk = k0 + ((e >> 16) & 0xFF);
        out[n * K + kk] = static_cast<uint16_t>(e & 0xFFFF);
    }
}

} // namespace

cudaError_t launch_decode(const uint8_t *ebase, const uint8_t *ae, const uint8_t *b,
                          const uint32_t *tile_ptr, const uint32_t *esc, uint16_t *out, int64_t N,
                          int64_t K, cudaStream_t st)
{
    const int64_t tiles_c = (K + 255) / 256;
    const int64_t T = ((N + 127) / 128) * tiles_c;
    if (T == 0)
        return cudaSuccess;
    decode_kernel<<<static_cast<unsigned>(T), 256, 0, st>>>(ebase, ae, b, tile_ptr, esc, out, N, K,
                                                             tiles_c);
    return cudaGetLastError();
}

} // namespace w12
