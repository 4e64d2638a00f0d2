// host.cpp -- host side of the W12 library: the multithreaded encoder, the
// format validator, blob (de)serialisation, file IO and statistics.
//
// Format (SpecPilot, Figure 5(a) caption, thelatestinai.com page): per BF16
// weight three 4-bit fields -- A = sign + mantissa bits 6..4, E = exponent
// offset inside a 16-binade window of the output channel, B = mantissa bits
// 3..0 -- plus an exact list of the weights the window cannot hold.  The
// window of row n spans exponents [ebase, ebase + 15] with ebase anchored so
// that the row's largest finite normal exponent is the window top
// (ebase = max(emax, 16) - 15); zeros, subnormals, Inf, NaN and anything below
// the window are escapes, stored as (row % 128) << 24 | (k % 256) << 16 | bits
// in per-(128 x 256)-tile lists, each sorted; the escaped slot keeps A = s << 3,
// E = 0, B = 0.  Lossless by construction (AI summary page, Main Findings,
// "W12 compression").
//
// Encoder option W12_ENCODE_COUNT_MAX: the window of a row is instead the one
// holding the most finite normal weights (the highest such base at or below
// the max-anchored one); weights above it escape as well, their slot holding
// the saturated placeholder A = s << 3 | 7, E = 15, B = 15 (the window's
// largest magnitude with the weight's sign, what the 8-bit view then reads).
// Decoding is the same for both.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <thread>

#include "w12_internal.h"

using namespace w12;

namespace {

// Window base of one row: exponent bits of finite normal weights are 1..254.
int row_window_base(const uint16_t *row, int64_t K)
{
    uint32_t emax = 16; // floor: ebase >= 1 even for rows without normals
    for (int64_t k = 0; k < K; ++k) {
        const uint32_t e = (row[k] >> 7) & 0xFFu;
        if (e != 0xFFu && e > emax)
            emax = e;
    }
    return static_cast<int>(emax) - 15;
}

// Count-maximising window base: the base b <= the max-anchored one whose 16
// binades [b, b + 15] hold the most finite normal weights of the row, the
// highest on ties (a sliding sum over the exponent histogram).
int row_window_base_count_max(const uint16_t *row, int64_t K)
{
    uint32_t cnt[256] = {};
    uint32_t emax = 16;
    for (int64_t k = 0; k < K; ++k) {
        const uint32_t e = (row[k] >> 7) & 0xFFu;
        if (e != 0 && e != 0xFFu) {
            ++cnt[e];
            if (e > emax)
                emax = e;
        }
    }
    const int b1 = static_cast<int>(emax) - 15;
    uint64_t win = 0;
    for (int e = 1; e <= 16; ++e)
        win += cnt[e];
    uint64_t best = win;
    int best_b = 1;
    for (int b = 2; b <= b1; ++b) {
        win += cnt[b + 15];
        win -= cnt[b - 1];
        if (win >= best) {
            best = win;
            best_b = b;
        }
    }
    return best_b;
}

struct BlockOut {
    // escape entries of one 128-row block, one list per column tile
    std::vector<std::vector<uint32_t>> per_tile;
};

// Encode rows [r0, r1) (inside one 128-row block) of W into the planes.
void encode_block(const uint16_t *w, int64_t K, int64_t r0, int64_t r1, w12_host *h,
                  BlockOut *out, bool count_max)
{
    const int64_t brow = b_row_bytes(K);
    const int64_t groups = ceil_div(K, 8);
    for (int64_t n = r0; n < r1; ++n) {
        const uint16_t *row = w + n * K;
        const int eb = count_max ? row_window_base_count_max(row, K) : row_window_base(row, K);
        h->ebase[n] = static_cast<uint8_t>(eb);
        uint8_t *ae_row = h->ae.data() + n * K;
        uint8_t *b_row = h->b.data() + n * brow;
        for (int64_t g = 0; g < groups; ++g) {
            uint32_t bword = 0;
            const int64_t kend = std::min<int64_t>(8, K - 8 * g);
            for (int64_t j = 0; j < kend; ++j) {
                const int64_t k = 8 * g + j;
                const uint32_t bits = row[k];
                const uint32_t s = bits >> 15;
                const uint32_t e = (bits >> 7) & 0xFFu;
                const uint32_t off = e - static_cast<uint32_t>(eb); // wraps when e < eb
                if (e != 0 && e != 0xFFu && off < 16u) {
                    ae_row[k] = static_cast<uint8_t>((s << 7) | ((bits & 0x70u)) | off);
                    // evens -> nibble slots 0..3, odds -> 4..7
                    const uint32_t slot = (j & 1) ? 4 + (j >> 1) : (j >> 1);
                    bword |= (bits & 0xFu) << (4 * slot);
                } else {
                    // above the window (count-maximising windows only): the
                    // saturated placeholder; otherwise A = s << 3, E = 0, B = 0
                    const bool above = e != 0xFFu && e > static_cast<uint32_t>(eb) + 15u;
                    ae_row[k] = static_cast<uint8_t>(above ? ((s << 7) | 0x7Fu) : (s << 7));
                    if (above) {
                        const uint32_t slot = (j & 1) ? 4 + (j >> 1) : (j >> 1);
                        bword |= 0xFu << (4 * slot);
                    }
                    out->per_tile[k / kTileCols].push_back(
                        (static_cast<uint32_t>(n % kTileRows) << 24) |
                        (static_cast<uint32_t>(k % kTileCols) << 16) | bits);
                }
            }
            b_row[4 * g + 0] = static_cast<uint8_t>(bword);
            b_row[4 * g + 1] = static_cast<uint8_t>(bword >> 8);
            b_row[4 * g + 2] = static_cast<uint8_t>(bword >> 16);
            b_row[4 * g + 3] = static_cast<uint8_t>(bword >> 24);
        }
    }
}

uint32_t crc32_update(uint32_t crc, const uint8_t *p, size_t n)
{
    crc = ~crc;
    for (size_t i = 0; i < n; ++i) {
        crc ^= p[i];
        for (int b = 0; b < 8; ++b)
            crc = (crc >> 1) ^ (0xEDB88320u & (0u - (crc & 1u)));
    }
    return ~crc;
}

void wr32(uint8_t *p, uint32_t v)
{
    for (int i = 0; i < 4; ++i)
        p[i] = static_cast<uint8_t>(v >> (8 * i));
}

void wr64(uint8_t *p, uint64_t v)
{
    for (int i = 0; i < 8; ++i)
        p[i] = static_cast<uint8_t>(v >> (8 * i));
}

uint32_t rd32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i)
        v |= static_cast<uint32_t>(p[i]) << (8 * i);
    return v;
}

uint64_t rd64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i)
        v |= static_cast<uint64_t>(p[i]) << (8 * i);
    return v;
}

size_t blob_size(const w12_host *h)
{
    const int64_t T = num_tiles(h->N, h->K);
    return static_cast<size_t>(kHeaderBytes + h->N + h->N * h->K + h->N * b_row_bytes(h->K) +
                               4 * (T + 1) + 4 * static_cast<int64_t>(h->esc.size()));
}

} // namespace

extern "C" {

const char *w12_status_string(w12_status s)
{
    switch (s) {
    case W12_OK: return "ok";
    case W12_ERR_INVALID_ARG: return "invalid argument";
    case W12_ERR_SHAPE: return "shape does not match the encoded matrix";
    case W12_ERR_ALIGNMENT: return "device buffer not 16-byte aligned";
    case W12_ERR_UNSUPPORTED: return "unsupported size (M must be 0..256, K % 32 == 0)";
    case W12_ERR_OOM: return "out of memory";
    case W12_ERR_CUDA: return "CUDA error";
    case W12_ERR_CORRUPT: return "encoded matrix is corrupt";
    case W12_ERR_TIMEOUT: return "device wait timed out";
    case W12_ERR_IO: return "file IO error";
    }
    return "unknown status";
}

w12_status w12_encode(const uint16_t *w_bf16, int64_t N, int64_t K, int n_threads,
                      w12_host **out)
{
    return w12_encode_ex(w_bf16, N, K, n_threads, 0, out);
}

w12_status w12_encode_ex(const uint16_t *w_bf16, int64_t N, int64_t K, int n_threads, unsigned flags,
                         w12_host **out)
{
    if (!out || N < 0 || K < 0 || (!w_bf16 && N * K > 0) || (flags & ~static_cast<unsigned>(W12_ENCODE_COUNT_MAX)))
        return W12_ERR_INVALID_ARG;
    const bool count_max = (flags & W12_ENCODE_COUNT_MAX) != 0;
    *out = nullptr;
    w12_host *h = new (std::nothrow) w12_host;
    if (!h)
        return W12_ERR_OOM;
    const int64_t tiles_c = ceil_div(K, kTileCols);
    const int64_t blocks = ceil_div(N, kTileRows);
    std::vector<BlockOut> outs;
    try {
        h->N = N;
        h->K = K;
        h->ebase.assign(static_cast<size_t>(N), 0);
        h->ae.assign(static_cast<size_t>(N * K), 0);
        h->b.assign(static_cast<size_t>(N * b_row_bytes(K)), 0);
        outs.resize(static_cast<size_t>(blocks));
        for (auto &o : outs)
            o.per_tile.resize(static_cast<size_t>(tiles_c));
    } catch (...) {
        delete h;
        return W12_ERR_OOM;
    }

    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = n_threads > 0 ? n_threads : (hw ? hw : 1);
    nt = std::max<int64_t>(1, std::min<int64_t>(nt, blocks));
    std::atomic<int64_t> next{0};
    auto worker = [&]() {
        for (;;) {
            const int64_t blk = next.fetch_add(1);
            if (blk >= blocks)
                break;
            const int64_t r0 = blk * kTileRows;
            encode_block(w_bf16, K, r0, std::min<int64_t>(N, r0 + kTileRows), h, &outs[blk], count_max);
        }
    };
    try {
        std::vector<std::thread> pool;
        for (int64_t i = 1; i < nt; ++i)
            pool.emplace_back(worker);
        worker();
        for (auto &t : pool)
            t.join();
    } catch (...) {
        delete h;
        return W12_ERR_OOM;
    }

    // tile order: t = block * tiles_c + column tile
    const int64_t T = blocks * tiles_c;
    try {
        h->tile_ptr.assign(static_cast<size_t>(T + 1), 0);
        size_t total = 0;
        for (int64_t t = 0; t < T; ++t) {
            total += outs[t / tiles_c].per_tile[t % tiles_c].size();
            h->tile_ptr[t + 1] = static_cast<uint32_t>(total);
        }
        h->esc.resize(total);
        for (int64_t t = 0; t < T; ++t) {
            const auto &v = outs[t / tiles_c].per_tile[t % tiles_c];
            std::copy(v.begin(), v.end(), h->esc.begin() + h->tile_ptr[t]);
        }
    } catch (...) {
        delete h;
        return W12_ERR_OOM;
    }
    *out = h;
    return W12_OK;
}

void w12_host_free(w12_host *h) { delete h; }

w12_status w12_host_stats(const w12_host *h, w12_stats *o)
{
    if (!h || !o)
        return W12_ERR_INVALID_ARG;
    const int64_t T = num_tiles(h->N, h->K);
    o->N = h->N;
    o->K = h->K;
    o->n_escapes = static_cast<int64_t>(h->esc.size());
    o->n_tiles = T;
    int64_t mx = 0;
    for (int64_t t = 0; t < T; ++t)
        mx = std::max<int64_t>(mx, h->tile_ptr[t + 1] - h->tile_ptr[t]);
    o->max_escapes_per_tile = mx;
    o->bytes_total = blob_size(h);
    o->bytes_ae = h->ae.size();
    o->bytes_b = h->b.size();
    const double nk = static_cast<double>(h->N) * static_cast<double>(h->K);
    o->bits_per_weight = nk > 0 ? 8.0 * static_cast<double>(o->bytes_total) / nk : 0.0;
    o->escape_fraction = nk > 0 ? static_cast<double>(o->n_escapes) / nk : 0.0;
    return W12_OK;
}

w12_status w12_host_view(const w12_host *h, const uint8_t **ebase, const uint8_t **ae,
                         const uint8_t **b, const uint32_t **tile_ptr, const uint32_t **esc)
{
    if (!h)
        return W12_ERR_INVALID_ARG;
    if (ebase)
        *ebase = h->ebase.data();
    if (ae)
        *ae = h->ae.data();
    if (b)
        *b = h->b.data();
    if (tile_ptr)
        *tile_ptr = h->tile_ptr.data();
    if (esc)
        *esc = h->esc.data();
    return W12_OK;
}

w12_status w12_validate(const w12_host *h)
{
    if (!h)
        return W12_ERR_INVALID_ARG;
    const int64_t N = h->N, K = h->K;
    if (N < 0 || K < 0)
        return W12_ERR_CORRUPT;
    const int64_t brow = b_row_bytes(K);
    const int64_t tiles_c = ceil_div(K, kTileCols);
    const int64_t T = num_tiles(N, K);
    if (static_cast<int64_t>(h->ebase.size()) != N || static_cast<int64_t>(h->ae.size()) != N * K ||
        static_cast<int64_t>(h->b.size()) != N * brow ||
        static_cast<int64_t>(h->tile_ptr.size()) != T + 1)
        return W12_ERR_CORRUPT;
    for (int64_t n = 0; n < N; ++n)
        if (h->ebase[n] < 1 || h->ebase[n] > 239)
            return W12_ERR_CORRUPT;
    if (h->tile_ptr[0] != 0 || h->tile_ptr[T] != h->esc.size())
        return W12_ERR_CORRUPT;
    for (int64_t t = 0; t < T; ++t) {
        if (h->tile_ptr[t + 1] < h->tile_ptr[t])
            return W12_ERR_CORRUPT;
        const int64_t n0 = (t / tiles_c) * kTileRows, k0 = (t % tiles_c) * kTileCols;
        for (uint32_t i = h->tile_ptr[t]; i < h->tile_ptr[t + 1]; ++i) {
            const uint32_t e = h->esc[i];
            if (i > h->tile_ptr[t] && e <= h->esc[i - 1])
                return W12_ERR_CORRUPT; // not sorted / not unique
            const int64_t n = n0 + (e >> 24), k = k0 + ((e >> 16) & 0xFF);
            if (n >= N || k >= K)
                return W12_ERR_CORRUPT;
            const uint32_t bits = e & 0xFFFF;
            const uint32_t ex = (bits >> 7) & 0xFF;
            const int eb = h->ebase[n];
            if (ex != 0 && ex != 0xFF && static_cast<int>(ex) >= eb && static_cast<int>(ex) <= eb + 15)
                return W12_ERR_CORRUPT; // an in-window weight must not escape
            // placeholder: A = s<<3, E = 0, B = 0; above the window (a
            // count-maximising window) A = s<<3 | 7, E = 15, B = 15
            const bool above = ex != 0xFF && static_cast<int>(ex) > eb + 15;
            if (h->ae[n * K + k] != (((bits >> 15) << 7) | (above ? 0x7Fu : 0u)))
                return W12_ERR_CORRUPT;
            const int64_t j = k % 8;
            const int slot = (j & 1) ? 4 + static_cast<int>(j >> 1) : static_cast<int>(j >> 1);
            const uint32_t word = rd32(&h->b[n * brow + 4 * (k / 8)]);
            if (((word >> (4 * slot)) & 0xF) != (above ? 0xFu : 0u))
                return W12_ERR_CORRUPT;
        }
    }
    if (K % 8) {
        // padding nibbles past K are zero
        for (int64_t n = 0; n < N; ++n) {
            const uint32_t word = rd32(&h->b[n * brow + brow - 4]);
            for (int64_t j = K % 8; j < 8; ++j) {
                const int slot = (j & 1) ? 4 + static_cast<int>(j >> 1) : static_cast<int>(j >> 1);
                if ((word >> (4 * slot)) & 0xF)
                    return W12_ERR_CORRUPT;
            }
        }
    }
    return W12_OK;
}

w12_status w12_serialize(const w12_host *h, uint8_t *buf, size_t cap, size_t *len)
{
    if (!h || !len)
        return W12_ERR_INVALID_ARG;
    const size_t need = blob_size(h);
    *len = need;
    if (!buf)
        return W12_OK;
    if (cap < need)
        return W12_ERR_INVALID_ARG;
    const int64_t T = num_tiles(h->N, h->K);
    uint8_t *p = buf;
    std::memcpy(p, "W12", 4);
    wr32(p + 4, 1);
    wr64(p + 8, static_cast<uint64_t>(h->N));
    wr64(p + 16, static_cast<uint64_t>(h->K));
    wr64(p + 24, static_cast<uint64_t>(h->esc.size()));
    wr64(p + 32, static_cast<uint64_t>(T));
    p += kHeaderBytes;
    std::memcpy(p, h->ebase.data(), h->ebase.size());
    p += h->ebase.size();
    std::memcpy(p, h->ae.data(), h->ae.size());
    p += h->ae.size();
    std::memcpy(p, h->b.data(), h->b.size());
    p += h->b.size();
    for (uint32_t v : h->tile_ptr) {
        wr32(p, v);
        p += 4;
    }
    for (uint32_t v : h->esc) {
        wr32(p, v);
        p += 4;
    }
    return W12_OK;
}

w12_status w12_deserialize(const uint8_t *buf, size_t len, w12_host **out)
{
    if (!buf || !out)
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    if (len < static_cast<size_t>(kHeaderBytes) || std::memcmp(buf, "W12", 4) != 0 ||
        rd32(buf + 4) != 1)
        return W12_ERR_CORRUPT;
    const uint64_t N = rd64(buf + 8), K = rd64(buf + 16), n_esc = rd64(buf + 24), T = rd64(buf + 32);
    if (N > (1ull << 40) || K > (1ull << 40) || n_esc > (1ull << 40) ||
        T != static_cast<uint64_t>(num_tiles(static_cast<int64_t>(N), static_cast<int64_t>(K))))
        return W12_ERR_CORRUPT;
    const unsigned __int128 need = (unsigned __int128)kHeaderBytes + N + (unsigned __int128)N * K +
                                   (unsigned __int128)N * b_row_bytes(static_cast<int64_t>(K)) +
                                   4 * (unsigned __int128)(T + 1) + 4 * (unsigned __int128)n_esc;
    if (need != len)
        return W12_ERR_CORRUPT;
    w12_host *h = new (std::nothrow) w12_host;
    if (!h)
        return W12_ERR_OOM;
    try {
        h->N = static_cast<int64_t>(N);
        h->K = static_cast<int64_t>(K);
        const uint8_t *p = buf + kHeaderBytes;
        h->ebase.assign(p, p + N);
        p += N;
        h->ae.assign(p, p + N * K);
        p += N * K;
        const size_t bb = static_cast<size_t>(N * b_row_bytes(static_cast<int64_t>(K)));
        h->b.assign(p, p + bb);
        p += bb;
        h->tile_ptr.resize(T + 1);
        for (uint64_t i = 0; i <= T; ++i, p += 4)
            h->tile_ptr[i] = rd32(p);
        h->esc.resize(n_esc);
        for (uint64_t i = 0; i < n_esc; ++i, p += 4)
            h->esc[i] = rd32(p);
    } catch (...) {
        delete h;
        return W12_ERR_OOM;
    }
    const w12_status st = w12_validate(h);
    if (st != W12_OK) {
        delete h;
        return st;
    }
    *out = h;
    return W12_OK;
}

w12_status w12_save(const w12_host *h, const char *path)
{
    if (!h || !path)
        return W12_ERR_INVALID_ARG;
    size_t len = 0;
    w12_serialize(h, nullptr, 0, &len);
    std::vector<uint8_t> buf;
    try {
        buf.resize(len + 4);
    } catch (...) {
        return W12_ERR_OOM;
    }
    w12_serialize(h, buf.data(), len, &len);
    wr32(buf.data() + len, crc32_update(0, buf.data(), len));
    FILE *f = std::fopen(path, "wb");
    if (!f)
        return W12_ERR_IO;
    const bool ok = std::fwrite(buf.data(), 1, buf.size(), f) == buf.size();
    return (std::fclose(f) == 0 && ok) ? W12_OK : W12_ERR_IO;
}

w12_status w12_load(const char *path, w12_host **out)
{
    if (!path || !out)
        return W12_ERR_INVALID_ARG;
    *out = nullptr;
    FILE *f = std::fopen(path, "rb");
    if (!f)
        return W12_ERR_IO;
    std::vector<uint8_t> buf;
    std::fseek(f, 0, SEEK_END);
    const long sz = std::ftell(f);
    std::fseek(f, 0, SEEK_SET);
    if (sz < 4) {
        std::fclose(f);
        return W12_ERR_CORRUPT;
    }
    try {
        buf.resize(static_cast<size_t>(sz));
    } catch (...) {
        std::fclose(f);
        return W12_ERR_OOM;
    }
    const bool ok = std::fread(buf.data(), 1, buf.size(), f) == buf.size();
    std::fclose(f);
    if (!ok)
        return W12_ERR_IO;
    const size_t len = buf.size() - 4;
    if (crc32_update(0, buf.data(), len) != rd32(buf.data() + len))
        return W12_ERR_CORRUPT;
    return w12_deserialize(buf.data(), len, out);
}

} // extern "C"
