// w12_internal.h -- library-internal layout of host and device handles.
#pragma once
#include <cstdint>
#include <vector>

#include "w12.h"

namespace w12 {

constexpr int kTileRows = 128;  // escape tile: rows
constexpr int kTileCols = 256;  // escape tile: columns
constexpr int kHeaderBytes = 40;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t b_row_bytes(int64_t K) { return 4 * ceil_div(K, 8); }
inline int64_t num_tiles(int64_t N, int64_t K)
{
    return ceil_div(N, kTileRows) * ceil_div(K, kTileCols);
}

} // namespace w12

struct w12_host {
    int64_t N = 0, K = 0;
    std::vector<uint8_t> ebase;     // [N]
    std::vector<uint8_t> ae;        // [N][K]
    std::vector<uint8_t> b;         // [N][b_row_bytes(K)]
    std::vector<uint32_t> tile_ptr; // [T + 1]
    std::vector<uint32_t> esc;      // [n_esc]
};

// Opaque 128-byte CUDA tensor map (CUtensorMap), kept as raw bytes here so that
// host-only translation units need no CUDA headers.
struct alignas(64) w12_tmap {
    uint64_t opaque[16];
};

struct w12_dev {
    int device = 0;
    int64_t N = 0, K = 0, T = 0, n_esc = 0;
    int64_t brow = 0, tiles_c = 0;
    void *base = nullptr; // the one device allocation
    size_t bytes = 0;
    uint8_t *ebase = nullptr;
    uint8_t *ae = nullptr;
    uint8_t *b = nullptr;
    uint32_t *tile_ptr = nullptr;
    uint32_t *esc = nullptr;
    uint16_t *gptr = nullptr; // [T][16] row-group offsets inside each escape tile
    int *status = nullptr; // device status word
    bool gemm_ok = false;  // K % 32 == 0 and tensor maps built
    // tensor maps over the planes: plain boxes for the FMA kernels, swizzled
    // boxes for the tensor-core kernels
    w12_tmap tm_ae_fma128, tm_ae_fma64, tm_b_fma128, tm_b_fma64;
    w12_tmap tm_ae_tc, tm_b_tc;
};

// INT8 copy of a weight matrix for the Q pass (one allocation).
struct w12_i8 {
    int device = 0;
    int64_t N = 0, K = 0;
    void *base = nullptr;
    size_t bytes = 0;
    int8_t *q = nullptr;   // [N][K]
    float *scale = nullptr; // [N]
    int *status = nullptr;  // device status word
    bool gemm_ok = false;   // K % 32 == 0 and the tensor map built
    w12_tmap tm_q_tc;       // swizzled 128 x 128 boxes, as the tensor-core kernel's AE plane
};
