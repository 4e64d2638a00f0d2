// i8.cu -- the INT8 copy of a weight matrix for the Q pass.
//
// The pages keep a separate low-bit copy of the weights for the Q pass on the
// smaller GPU (INT6/INT8, RTX PRO 6000 section); this is its INT8 form: per
// output row n a scale = amax / 127 (FP32, amax the largest |w| over the row's
// finite weights) and q[n][k] = rint(w / scale) (FP32 division, round half to
// even) clamped to [-127, 127]; Inf goes to +-127, NaN to 0, and a row whose
// scale is 0 keeps q = 0.  The Q-pass product is then scale[n] * sum_k x q,
// computed by the tensor-core kernel with its INT8 weight mode.
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

constexpr int kQThreads = 256; // 8 warps, one row each

__global__ void __launch_bounds__(kQThreads) i8_quantize_kernel(const uint16_t *w, int64_t N, int64_t K,
                                                                int8_t *q, float *scale)
{
    const int64_t n = static_cast<int64_t>(blockIdx.x) * (kQThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N)
        return;
    const uint16_t *row = w + n * K;
    float amax = 0.f;
    for (int64_t k = lane; k < K; k += 32) {
        const uint32_t bits = row[k];
        if (((bits >> 7) & 0xFFu) != 0xFFu) // finite
            amax = fmaxf(amax, __uint_as_float((bits & 0x7FFFu) << 16));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = __fdiv_rn(amax, 127.0f);
    if (lane == 0)
        scale[n] = sc;
    int8_t *qrow = q + n * K;
    for (int64_t k = lane; k < K; k += 32) {
        const float v = __uint_as_float(static_cast<uint32_t>(row[k]) << 16);
        float t = 0.f;
        if (sc != 0.f && !isnan(v)) {
            t = rintf(__fdiv_rn(v, sc));
            t = fminf(fmaxf(t, -127.f), 127.f);
        }
        qrow[k] = static_cast<int8_t>(static_cast<int>(t));
    }
}

} // namespace

cudaError_t launch_i8_quantize(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *scale, cudaStream_t st)
{
    if (N == 0)
        return cudaSuccess;
    i8_quantize_kernel<<<static_cast<unsigned>(ceil_div(N, kQThreads / 32)), kQThreads, 0, st>>>(w, N, K, q,
                                                                                                    scale);
    return cudaGetLastError();
}

} // namespace w12
