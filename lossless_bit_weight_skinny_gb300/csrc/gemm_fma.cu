// gemm_fma.cu -- W12 skinny GEMM for M <= 4 activation rows on the CUDA cores
// (the library sends it M <= 2; from 3 rows on the tensor-core kernel is faster).
//
// y[m][n] = sum_k x[m][k] * W[n][k], W decoded from its W12 planes to exact
// BF16 values (SpecPilot, Figure 5(a) caption) in registers and accumulated in
// FP32 with BF16 x BF16 -> FP32 FMAs (packed FP32 FMAs with W12_FMA_MIXED=0).
//
// Work split: the matrix is cut into blocks of RBLK rows x 256 columns (one
// escape tile wide); the (row block, k step) iterations are split evenly over
// one persistent CTA per SM (stream-K), and row blocks shared by several CTAs
// are combined by the last contributor in a fixed order.
//
// CTA = CW consumer warps + a producer warp + two escape warps.  The producer
// streams each block's AE bytes, B words and x slice with TMA into a ring of
// shared-memory stages, and copies the tile's escape entries next to them with
// cp.async.  Consumer warp w owns RW rows of the block; lane l owns columns
// 8l..8l+7 of the 256-column step and keeps the products of its rows in
// registers until the row block ends, then the warp reduces across lanes.
//
// Escapes: the main loop multiplies every slot as decoded -- an escaped slot
// holds the placeholder +-2^(ebase-127), or the saturated one above a
// count-maximising window -- and has no branches and no escape
// work at all.  The escape warps (even and odd units) walk each stage's list
// and keep, per output, the two correction sums sum(-x * placeholder) and
// sum(x * exact value) in shared memory; the consumers add them to the output
// in that order at the end of the row block.  With a single non-zero product
// (one-hot x) this gives the exact escaped value back, Inf/NaN escapes
// propagate, and otherwise the result is the same sum in another (fixed)
// order.  The final store goes through the output mode (FP32, BF16, SiLU*mul
// of interleaved gate/up rows).
#include "kernels.cuh"

namespace w12 {
namespace {

#ifndef W12_FMA_CW
#define W12_FMA_CW 0 // consumer warps (8 or 16); 0 = 16 for M = 1, 8 otherwise
#endif
#ifndef W12_FMA_MIXED
#define W12_FMA_MIXED 1 // M <= 2: BF16 x BF16 -> FP32 FMAs instead of packed FP32 FMAs
#endif

#ifndef W12_FMA_CPS
#define W12_FMA_CPS 1 // CTAs per SM of the M = 1 kernel (1 or 2)
#endif


template <int MT>
struct FmaShape {
    // CTAs resident per SM: two for M = 1, so that the next kernel's CTAs can
    // start streaming while this kernel's last ones finish; each then works
    // on blocks of 64 rows (half an escape tile)
    static constexpr int CPS = MT == 1 ? W12_FMA_CPS : 1;
    static constexpr int RBLK = CPS == 2 ? 64 : 128;          // rows per block
    static constexpr int CW = W12_FMA_CW ? W12_FMA_CW : (MT == 1 ? 16 / CPS : 8); // consumer warps
    static constexpr int NE = CPS == 2 ? 1 : 2;               // escape warps
    static constexpr int RW = RBLK / CW;                      // rows per consumer warp
    static constexpr int THREADS = (CW + 1 + NE) * 32;        // + producer + escape warps
    // registers per thread: each of the 4 SM sub-partitions has 16K registers
    // and holds ceil(warps / 4) of the resident CTAs' warps
    static constexpr int PER_SMSP = (CPS * (CW + 1 + NE) + 3) / 4;
    static constexpr int MAXREG_RAW = (16384 / (32 * PER_SMSP)) & ~7;
    static constexpr int MAXREG = MAXREG_RAW > 255 ? 255 : MAXREG_RAW;
    static_assert(RW % 8 == 0 && RBLK % CW == 0, "warps own whole 8-row escape groups");
};

constexpr int r128(int v) { return (v + 127) & ~127; }
constexpr int r1024(int v) { return (v + 1023) & ~1023; }

template <int MT, bool Q8>
struct FmaSmem {
    using S = FmaShape<MT>;
    static constexpr int AE = S::RBLK * 256;
    static constexpr int B = Q8 ? 0 : S::RBLK * 128;
    static constexpr int X = MT * 256 * 2;
    static constexpr int ESC_CAP = 256; // more entries in a tile are read from global memory
    // escape area: [lo, hi, -, -] u32 | entries
    static constexpr int ESC_LIST = 16;
    static constexpr int ESC = Q8 ? 0 : ESC_LIST + ESC_CAP * 4;
    static constexpr int OFF_AE = 0;
    static constexpr int OFF_B = r128(AE);
    static constexpr int OFF_X = OFF_B + r128(B);
    static constexpr int OFF_ESC = OFF_X + r128(X);
    static constexpr int STAGE = r1024(OFF_ESC + ESC);
    // per escape warp: correction sums [buffer][neg, pos][RBLK * MT], window bases
    static constexpr int CORR_W = 2 * 2 * S::RBLK * MT * 4 + S::RBLK;
    static constexpr int CORR = Q8 ? 0 : S::NE * CORR_W;
    static constexpr int BUDGET = (227 * 1024) / S::CPS - 2048;
    static constexpr int STAGES_RAW = (BUDGET - CORR) / STAGE;
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr int TX_BYTES = AE + B + X;
    static constexpr int OFF_CORR = STAGES * STAGE;
    static constexpr int BARS = OFF_CORR + CORR;         // barrier area offset
    static constexpr int NBARS = 2 * STAGES + 1 + 4;     // full, empty, stall, corr_full/empty
    static constexpr int TOTAL = BARS + 8 * NBARS + 16 + 1024; // + slack to align the base
    static_assert(STAGES >= 4 / S::CPS && TOTAL <= (227 * 1024) / S::CPS, "shared memory budget");
};

// Bounded wait that also gives up as soon as another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const GemmArgs &a,
                                              volatile int *abort_flag)
{
    // the flag (a shared-memory load, queued behind this warp's other loads)
    // is read only once the phase is found incomplete
    if (mbar_try_wait(bar, parity))
        return true;
    if (*abort_flag)
        return false;
    // each try suspends the warp until the phase completes (or the suspend
    // hint passes), so a waiting warp takes no issue slots from the others
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > a.limit_ns) {
            *abort_flag = 1;
            report(a, kStatusTimeout);
            return false;
        }
    }
}

// Decode 8 weights (AE bytes k..k+7, their B word) to FP32 values.
template <bool Q8>
__device__ __forceinline__ void decode8(uint2 ae, uint32_t bw, uint32_t eb2, float (&wf)[8])
{
    uint32_t r[4];
    decode_group<Q8>(ae.x, ae.y, bw, eb2, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        wf[2 * i] = __uint_as_float(r[i] << 16);
        wf[2 * i + 1] = __uint_as_float(r[i] & 0xFFFF0000u);
    }
}

// acc.x += lo(w) * lo(x), acc.y += hi(w) * hi(x) on BF16 halves with FP32
// accumulation and one rounding each (the BF16 product is exact in FP32, so
// this equals an FP32 FMA of the widened values).
__device__ __forceinline__ void fma_bf16x2_f32(float2 &acc, uint32_t w, uint32_t x)
{
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc.x), "+f"(acc.y)
        : "r"(w), "r"(x));
}

// Reduce V per-lane values across the warp.  Afterwards, for V >= 32, lane l
// holds the totals of indices l*(V/32) .. l*(V/32)+V/32-1 in v[0..V/32); for
// V < 32 it holds the total of index l >> (5 - log2 V) in v[0].
template <int N, int O>
struct XReduce {
    static __device__ __forceinline__ void run(float *v, int lane)
    {
        if constexpr (O > 0) {
            if constexpr (N > 1) {
                constexpr int H = N / 2;
                const bool up = (lane & O) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float keep = up ? v[i + H] : v[i];
                    const float send = up ? v[i] : v[i + H];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
                }
                XReduce<H, O / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
                XReduce<1, O / 2>::run(v, lane);
            }
        }
    }
};

// Escape warp: NC chunks of 32 list entries starting at j1, one entry per
// lane.  For each entry the products -x * placeholder and x * exact value of
// every activation row; a segmented scan over the lanes sums them per output
// row (the list is sorted by row), and each row's sum is added to its
// correction totals in shared memory.  The chunks' loads and scans are
// independent and interleaved; the additions happen in list order.
template <int MT, int RBLK, int NC>
__device__ __forceinline__ void esc_chunks(const MatArgs &mm, const uint32_t *list_s, bool big,
                                           uint32_t lo, uint32_t cnt, uint32_t j1, uint32_t rbase,
                                           int row0, const uint8_t *eb_s, const uint8_t *xs,
                                           float *cneg, float *cpos, int lane)
{
    uint32_t e4[NC];
#pragma unroll
    for (int u = 0; u < NC; ++u) {
        const uint32_t j = j1 + 32 * u + static_cast<uint32_t>(lane);
        e4[u] = 0u;
        if (j < cnt) {
            if (big)
                e4[u] = __ldg(mm.esc + lo + j);
            else
                e4[u] = list_s[j];
        }
    }
    float pn[NC][MT], pp[NC][MT];
    uint32_t key[NC], rr[NC];
    bool in[NC];
#pragma unroll
    for (int u = 0; u < NC; ++u) {
        const uint32_t j = j1 + 32 * u + static_cast<uint32_t>(lane);
        const uint32_t e = e4[u];
        const uint32_t r = (e >> 24) - rbase; // row in the block
        in[u] = j < cnt && r < static_cast<uint32_t>(RBLK) && row0 + static_cast<int>(r) < mm.N;
        rr[u] = r;
        const uint32_t k8 = (e >> 16) & 0xFFu;
        const uint32_t eb = in[u] ? eb_s[r] : 0u;
        // the slot's placeholder: +-2^(ebase-127), or, for a finite weight
        // above the window (count-maximising windows), the saturated
        // +-(2 - 2^-7) * 2^(ebase+15-127)
        const uint32_t ex = (e >> 7) & 0xFFu;
        const bool above = ex != 0xFFu && ex > eb + 15u;
        const float wph = __uint_as_float(((e & 0x8000u) << 16) |
                                          (above ? (((eb + 15u) << 23) | (0x7Fu << 16)) : (eb << 23)));
        const float wex = __uint_as_float((e & 0xFFFFu) << 16);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint32_t xb = *reinterpret_cast<const uint16_t *>(xs + m * 512 + k8 * 2);
            const float xv = __uint_as_float(xb << 16);
            pn[u][m] = in[u] ? -(xv * wph) : 0.f; // both products are exact in FP32
            pp[u][m] = in[u] ? xv * wex : 0.f;
        }
        key[u] = in[u] ? r : 256u + static_cast<uint32_t>(lane);
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int u = 0; u < NC; ++u) {
            const uint32_t kp = __shfl_up_sync(0xffffffffu, key[u], d);
            const bool take = lane >= d && kp == key[u];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float an = __shfl_up_sync(0xffffffffu, pn[u][m], d);
                const float ap = __shfl_up_sync(0xffffffffu, pp[u][m], d);
                if (take) {
                    pn[u][m] = an + pn[u][m];
                    pp[u][m] = ap + pp[u][m];
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NC; ++u) {
        if (j1 + 32 * u >= cnt)
            break;
        const uint32_t kn = __shfl_down_sync(0xffffffffu, key[u], 1);
        if (in[u] && (lane == 31 || kn != key[u])) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                cneg[rr[u] * MT + m] += pn[u][m];
                cpos[rr[u] * MT + m] += pp[u][m];
            }
        }
        __syncwarp();
    }
}

template <int MT, bool Q8>
__global__ void __maxnreg__(FmaShape<MT>::MAXREG)
    gemm_fma_kernel(const GemmArgs a, const __grid_constant__ TmapSet tm)
{
    using S = FmaShape<MT>;
    using L = FmaSmem<MT, Q8>;
    constexpr int RBLK = S::RBLK, CW = S::CW, RW = S::RW, STAGES = L::STAGES;
    constexpr int V = RW * MT;           // per-lane partial sums
    constexpr int VPL = V >= 32 ? V / 32 : 1;
    constexpr int LOGV = (V >= 64) ? 6 : (V >= 32) ? 5 : (V >= 16) ? 4 : 3;
    constexpr int NE = S::NE;
    constexpr int WARP_P = CW, WARP_E = CW + 1; // producer, escape warps WARP_E .. WARP_E + NE - 1
    // Weight units streamed ahead of the activation wait: one short of the
    // ring, so that a CTA that starts while the previous kernel ends adds
    // less traffic to that kernel's last loads (measured on GB300, the M = 1
    // grouped layer: 99.4 us with the whole ring of 4, 98.5 with 3 or 2,
    // 100.1 with 1)
    constexpr int kPreUnits = STAGES > 1 ? STAGES - 1 : 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    // full, empty [STAGES]; stall; corr_full, corr_empty [2]
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t stall_bar = smem_u32(bars + 2 * STAGES);
    const uint32_t corr_full0 = stall_bar + 8, corr_empty0 = stall_bar + 24;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + L::NBARS);
    volatile int *seg_last = abort_flag + 1;
    // escape corrections of the current row block, double buffered:
    // [buffer][neg, pos][RBLK * MT]
    // escape warp E's correction sums: corr_of(E) + db * 2 * RBLK * MT
    auto corr_of = [&](int e) { return reinterpret_cast<float *>(smem + L::OFF_CORR + e * L::CORR_W); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int it0 = sk_begin(cta, grid, a.total_iters);
    const int n_it = sk_begin(cta + 1, grid, a.total_iters) - it0;
    const int nk = a.n_kstep;

    // the tensor maps' descriptors are fetched while the CTA sets up
    if (warp == WARP_P) {
        if (lane < a.n_mat) {
            prefetch_tmap(&tm.ae[lane]);
            if (!Q8)
                prefetch_tmap(&tm.b[lane]);
        }
        if (lane == 0)
            prefetch_tmap(&tm.x);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, Q8 ? 1 : 33);
            mbar_init(empty0 + 8 * s, Q8 ? CW : CW + NE);
        }
        mbar_init(stall_bar, 1);
        for (int d = 0; d < 2; ++d) {
            mbar_init(corr_full0 + 8 * d, 32 * NE);
            mbar_init(corr_empty0 + 8 * d, CW);
        }
        *abort_flag = 0;
        *seg_last = 0;
        fence_barrier_init();
    }
    // escape-list bounds of the producer's first 64 units, loaded while the
    // CTA sets up
    uint32_t w_lo = 0, w_hi = 0, w_nlo = 0, w_nhi = 0;
    if (!Q8 && warp == WARP_P) {
        load_tile_window(a, it0, n_it, 0, lane, RBLK, w_lo, w_hi);
        load_tile_window(a, it0, n_it, 32, lane, RBLK, w_nlo, w_nhi);
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == WARP_P) {
        // ------------------------------ producer ------------------------------
        int issued = 0;
        int rb = it0 / nk, ks = it0 % nk, s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < n_it; ++it) {
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(empty0 + 8 * s, ph ^ 1, a, abort_flag));
            if (!ok)
                break;
            const int g = mat_of(a, rb);
            const MatArgs &mm = a.mat[g];
            const int row0 = (rb - mm.rb0) * RBLK, k0 = ks * 256; // rows of matrix g
            uint8_t *st = smem + s * L::STAGE;
            const uint32_t fb = full0 + 8 * s;
            // The first kPreUnits units' weights stream before the previous
            // kernel in the stream has finished; activations, which it may
            // have written, only after it has -- unless the caller declared
            // them complete before that kernel started.  (Writes wait for the
            // previous kernel in any case: see the row-block end.)
            const int pre = a.x_ready ? 0 : (n_it < kPreUnits ? n_it : kPreUnits);
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, L::TX_BYTES);
                tma_load_2d(smem_u32(st + L::OFF_AE), &tm.ae[g], k0, row0, fb);
                if (!Q8)
                    tma_load_2d(smem_u32(st + L::OFF_B), &tm.b[g], k0 / 2, row0, fb);
                if (it >= pre)
                    tma_load_2d(smem_u32(st + L::OFF_X), &tm.x, k0, 0, fb);
                if (it == pre - 1) {
                    pdl_wait_prior_grid();
                    for (int j = 0; j < pre; ++j)
                        tma_load_2d(smem_u32(smem + j * L::STAGE + L::OFF_X), &tm.x,
                                    ((it0 + j) % nk) * 256, 0, full0 + 8 * j);
                }
            }
            if (!Q8) {
                // the tile's entry range, then its entries (up to ESC_CAP)
                uint8_t *esc_area = st + L::OFF_ESC;
                if (lane < 2)
                    cp_async_4(smem_u32(esc_area + 4 * lane),
                               mm.tile_ptr + (row0 / 128) * a.tiles_c + ks + lane);
                if (it > 0 && (it & 31) == 0) { // next window; prefetch the one after
                    w_lo = w_nlo;
                    w_hi = w_nhi;
                    load_tile_window(a, it0, n_it, it + 32, lane, RBLK, w_nlo, w_nhi);
                }
                const uint32_t lo = __shfl_sync(0xffffffffu, w_lo, it & 31);
                const uint32_t hi = __shfl_sync(0xffffffffu, w_hi, it & 31);
                const uint32_t cnt = min(hi - lo, static_cast<uint32_t>(L::ESC_CAP));
                uint32_t *list = reinterpret_cast<uint32_t *>(esc_area + L::ESC_LIST);
                for (uint32_t idx = lane; idx < cnt; idx += 32)
                    cp_async_4(smem_u32(list + idx), mm.esc + lo + idx);
                cp_async_arrive_noinc(fb);
            }
            issued = it + 1;
            if (++ks == nk) {
                ks = 0;
                ++rb;
            }
            if (++s == STAGES) {
                s = 0;
                ph ^= 1;
            }
        }
        // drain: every copy this warp started must land before the CTA exits
        for (int it = issued - 1; it >= 0 && it >= issued - STAGES; --it) {
            const int s = it % STAGES;
            mbar_wait(full0 + 8 * s, (it / STAGES) & 1, 1000000000ull);
        }
    } else if (warp >= WARP_E && warp < WARP_E + NE) {
        // ---------------------------- escape warps ----------------------------
        // Escape warp E takes the units of parity E.  Per unit, the tile's
        // entries 32 at a time, one per lane: the two products -x * placeholder
        // and x * exact value for each activation row, summed per output row
        // by a segmented scan over the lanes (the list is sorted by row), then
        // added to the row's correction sums of this warp.  Fixed order
        // throughout, so results are reproducible.
        const int ew = warp - WARP_E;
        float *const corr = corr_of(ew);
        uint8_t *const eb_s = reinterpret_cast<uint8_t *>(corr + 2 * 2 * RBLK * MT); // window bases
        if (!Q8) {
            int seg = 0;
            int rb = it0 / nk, ks = it0 % nk, s = 0;
            uint32_t ph = 0;
            for (int it = 0; it < n_it; ++it) {
                const bool seg_start = (it == 0) || (ks == 0);
                const bool seg_end = (ks == nk - 1) || (it == n_it - 1);
                const int db = seg & 1;
                float *cneg = corr + db * (2 * RBLK * MT), *cpos = cneg + RBLK * MT;
                if (seg_start) {
                    // buffer db was last read by the consumers at the end of segment seg - 2
                    if (seg >= 2)
                        wait_or_abort(corr_empty0 + 8 * db, ((seg >> 1) - 1) & 1, a, abort_flag);
                    for (int i = lane; i < 2 * RBLK * MT; i += 32)
                        cneg[i] = 0.f;
                    const MatArgs &mm = a.mat[mat_of(a, rb)];
                    const int lr0 = (rb - mm.rb0) * RBLK;
                    for (int r = lane; r < RBLK; r += 32)
                        eb_s[r] = lr0 + r < mm.N ? __ldg(mm.ebase + lr0 + r) : 0;
                    __syncwarp();
                }
                bool ok = wait_or_abort(full0 + 8 * s, ph, a, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                const MatArgs &mm = a.mat[mat_of(a, rb)];
                const int row0 = (rb - mm.rb0) * RBLK; // rows of its matrix
                const uint8_t *st = smem + s * L::STAGE;
                if (ok && (NE == 1 || ((it0 + it) & 1) == ew)) {
                    const uint8_t *esc_area = st + L::OFF_ESC;
                    const uint2 lohi = *reinterpret_cast<const uint2 *>(esc_area);
                    // a stage read after an abort may hold another unit's
                    // bounds: keep every global read inside this matrix's list
                    const uint32_t lo_c = min(lohi.x, mm.n_esc);
                    const uint32_t cnt = min(lohi.y - lohi.x, mm.n_esc - lo_c);
                    const bool big = cnt > static_cast<uint32_t>(L::ESC_CAP);
                    const uint32_t *list_s = reinterpret_cast<const uint32_t *>(esc_area + L::ESC_LIST);
                    const uint32_t rbase = static_cast<uint32_t>(row0 & 127);
                    for (uint32_t j1 = 0; j1 < cnt; j1 += 128) {
                        if (cnt - j1 <= 32)
                            esc_chunks<MT, RBLK, 1>(mm, list_s, big, lo_c, cnt, j1, rbase, row0, eb_s,
                                                    st + L::OFF_X, cneg, cpos, lane);
                        else
                            esc_chunks<MT, RBLK, 4>(mm, list_s, big, lo_c, cnt, j1, rbase, row0, eb_s,
                                                    st + L::OFF_X, cneg, cpos, lane);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty0 + 8 * s);
                if (seg_end) {
                    mbar_arrive(corr_full0 + 8 * db); // every escape lane: its sums are visible
                    ++seg;
                }
                if (++ks == nk) {
                    ks = 0;
                    ++rb;
                }
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else {
        // ------------------------------ consumers -----------------------------
        const int wrow = warp * RW;
        float acc[MT <= 2 ? 1 : RW][MT <= 2 ? 1 : MT];
        float2 acc2[MT <= 2 ? RW : 1][MT <= 2 ? MT : 1];
        uint32_t eb2[RW];
        int cur_rb = -1, seg = 0;
        int rb = it0 / nk, ks = it0 % nk; // (row block, k step) of iteration it
        int s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < n_it; ++it) {
            // window bases of a new row block: start the load before waiting
            uint32_t e_pre = 1u;
            const MatArgs &mm = a.mat[mat_of(a, rb)];
            const int row0 = (rb - mm.rb0) * RBLK; // rows of its matrix
            if (rb != cur_rb) {
                const int n = row0 + wrow + lane;
                if (lane < RW && n < mm.N)
                    e_pre = __ldg(mm.ebase + n);
            }
            wait_or_abort(full0 + 8 * s, ph, a, abort_flag);
            if (a.inject_stall)
                wait_or_abort(stall_bar, 0, a, abort_flag);
            // After an abort the loop keeps its shape (every warp still meets
            // every barrier) but works on stale data.
            const uint8_t *st = smem + s * L::STAGE;

            if (rb != cur_rb) { // a new row block: reset the sums, fetch window bases
                cur_rb = rb;
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if constexpr (MT <= 2)
                            acc2[r][m] = make_float2(0.f, 0.f);
                        else
                            acc[r][m] = 0.f;
                    }
                const uint32_t e = e_pre;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    const uint32_t er = __shfl_sync(0xffffffffu, e, r);
                    eb2[r] = (er << 7) | (er << 23);
                }
            }

            // this lane's x[m][8l .. 8l+7]: raw BF16x2 words and FP32 pairs
            constexpr bool kMixed = W12_FMA_MIXED && MT <= 2;
            uint32_t xw[MT][4];
            float2 x2[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 v = *reinterpret_cast<const uint4 *>(st + L::OFF_X + m * 512 + lane * 16);
                xw[m][0] = v.x;
                xw[m][1] = v.y;
                xw[m][2] = v.z;
                xw[m][3] = v.w;
                if constexpr (!kMixed) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        x2[m][i] = make_float2(__uint_as_float(xw[m][i] << 16),
                                               __uint_as_float(xw[m][i] & 0xFFFF0000u));
                }
            }

            // For M = 1 the warp's raw planes fit in registers: load them all and
            // hand the stage back to the producer before computing on them, so
            // the refill overlaps the arithmetic.  Larger M reads them row by
            // row and releases the stage afterwards.
            constexpr bool kEarly = MT == 1;
            const uint8_t *ae_p = st + L::OFF_AE + wrow * 256 + lane * 8;
            const uint8_t *b_p = st + L::OFF_B + wrow * 128 + lane * 4;
            uint2 aw[RW];
            uint32_t bwr[RW];
            if constexpr (kEarly) {
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    aw[r] = *reinterpret_cast<const uint2 *>(ae_p + r * 256);
                    bwr[r] = Q8 ? 0u : *reinterpret_cast<const uint32_t *>(b_p + r * 128);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty0 + 8 * s);
            }
            // main loop: every row of this warp, no branches
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                if constexpr (!kEarly) {
                    aw[r] = *reinterpret_cast<const uint2 *>(ae_p + r * 256);
                    bwr[r] = Q8 ? 0u : *reinterpret_cast<const uint32_t *>(b_p + r * 128);
                }
                const uint32_t bw = bwr[r];
                if constexpr (kMixed) {
                    uint32_t wr[4];
                    decode_group<Q8>(aw[r].x, aw[r].y, bw, eb2[r], wr);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            fma_bf16x2_f32(acc2[r][m], wr[i], xw[m][i]);
                    continue;
                }
                float wf[8];
                decode8<Q8>(aw[r], bw, eb2[r], wf);
                const float2 w01 = make_float2(wf[0], wf[1]), w23 = make_float2(wf[2], wf[3]);
                const float2 w45 = make_float2(wf[4], wf[5]), w67 = make_float2(wf[6], wf[7]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if constexpr (MT <= 2) {
                        float2 t = acc2[r][m];
                        t = __ffma2_rn(x2[m][0], w01, t);
                        t = __ffma2_rn(x2[m][1], w23, t);
                        t = __ffma2_rn(x2[m][2], w45, t);
                        t = __ffma2_rn(x2[m][3], w67, t);
                        acc2[r][m] = t;
                    } else {
                        float2 t = __fmul2_rn(x2[m][0], w01);
                        t = __ffma2_rn(x2[m][1], w23, t);
                        t = __ffma2_rn(x2[m][2], w45, t);
                        t = __ffma2_rn(x2[m][3], w67, t);
                        acc[r][m] += t.x + t.y;
                    }
                }
            }
            if constexpr (!kEarly) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty0 + 8 * s);
            }

            if (ks == nk - 1 || it == n_it - 1) {
                // ---- the row block ends here for this CTA: reduce and store ----
                // nothing is written before the previous kernel in the stream
                // has completed (at once when the activation load waited for it)
                pdl_wait_prior_grid();
                float v[V];
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if constexpr (MT <= 2)
                            v[r * MT + m] = acc2[r][m].x + acc2[r][m].y;
                        else
                            v[r * MT + m] = acc[r][m];
                    }
                XReduce<V, 16>::run(v, lane);
                // this segment's escape corrections (complete once the escape
                // warp has passed the segment's last stage)
                const int db = seg & 1;
                if (!Q8)
                    wait_or_abort(corr_full0 + 8 * db, (seg >> 1) & 1, a, abort_flag);
                const float *cneg0 = corr_of(0) + db * (2 * RBLK * MT), *cpos0 = cneg0 + RBLK * MT;
                const float *cneg1 = corr_of(NE - 1) + db * (2 * RBLK * MT), *cpos1 = cneg1 + RBLK * MT;
                const int c_first = sk_owner(rb * nk, grid, a.total_iters);
                const int c_last = sk_owner((rb + 1) * nk - 1, grid, a.total_iters);
                const bool writer = (V >= 32) || ((lane & ((32 >> LOGV) - 1)) == 0);
                const bool direct = (c_first == c_last);
                const int slot = direct ? 0 : sk_slot(cta, rb, grid, a.total_iters, nk);
                float tot[VPL];
#pragma unroll
                for (int q = 0; q < VPL; ++q) {
                    const int idx = (V >= 32) ? lane * VPL + q : (lane >> (5 - LOGV));
                    const int r = idx / MT, m = idx % MT;
                    // the placeholder products out first, then the exact ones in
                    tot[q] = v[q];
                    if (!Q8) {
                        const int i = (wrow + r) * MT + m;
                        if constexpr (NE == 1)
                            tot[q] = (tot[q] + cneg0[i]) + cpos0[i];
                        else
                            tot[q] = (tot[q] + (cneg0[i] + cneg1[i])) + (cpos0[i] + cpos1[i]);
                    }
                }
                // under kOutSiluMul, the value of row r + 1 (value index idx + MT):
                // another lane's (same q) or, with several values a lane, this one's
                constexpr int PAIR_IN_LANE = (V >= 32 && VPL % (2 * MT) == 0) ? 1 : 0;
                constexpr int PAIR_DL = V < 32 ? (MT << (5 - LOGV)) : (PAIR_IN_LANE ? 0 : MT / VPL);
                static_assert(PAIR_IN_LANE || (V < 32) || (MT % VPL == 0), "gate/up pairing layout");
                const bool pair = direct && (a.out_mode & kOutSiluMul);
#pragma unroll
                for (int q = 0; q < VPL; ++q) {
                    const int idx = (V >= 32) ? lane * VPL + q : (lane >> (5 - LOGV));
                    const int r = idx / MT, m = idx % MT;
                    const float total = tot[q];
                    float next = 0.f;
                    if constexpr (PAIR_IN_LANE)
                        next = tot[(q + MT) % VPL];
                    else if (pair)
                        next = __shfl_down_sync(0xffffffffu, total, PAIR_DL);
                    const int n = row0 + wrow + r;
                    if (writer && m < a.M) {
                        if (direct) {
                            if (n < mm.N)
                                emit_y(a, mm, m, n, total, next);
                        } else {
                            a.partials[(static_cast<size_t>(slot) * a.M + m) * RBLK + wrow + r] = total;
                        }
                    }
                }
                if (!Q8) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(corr_empty0 + 8 * db);
                }
                ++seg;
                if (!direct) {
                    // the CTA barrier orders every thread's partial stores before
                    // thread 0's release-acquire arrival (cumulativity), and that
                    // arrival before everyone's reads of the other partials
                    named_bar_sync(1, CW * 32);
                    if constexpr (MT == 1) {
                        // one row's partials are 512 bytes a contributor: warp 0
                        // alone arrives and, if last, sums them (the warp barrier
                        // orders lane 0's acquire before its lanes' reads) while
                        // the other warps go on with the next stage (measured on
                        // GB300: a single-row layer step 108.9 -> 108.0 us; at
                        // two rows one warp is too few)
                        if (warp == 0) {
                            uint32_t last = 0u;
                            if (lane == 0)
                                last = sk_arrive(a.counters + rb, c_last - c_first + 1) ? 1u : 0u;
                            last = __shfl_sync(0xffffffffu, last, 0);
                            __syncwarp();
                            if (last)
                                sk_reduce_block<true>(a, rb, RBLK, grid, c_first, c_last, lane, 32);
                        }
                    } else {
                        if (threadIdx.x == 0)
                            *seg_last = sk_arrive(a.counters + rb, c_last - c_first + 1) ? 1 : 0;
                        named_bar_sync(1, CW * 32);
                        if (*seg_last)
                            sk_reduce_block<true>(a, rb, RBLK, grid, c_first, c_last, threadIdx.x, CW * 32);
                    }
                }
            }
            // next iteration: (row block, k step) and ring slot
            if (++ks == nk) {
                ks = 0;
                ++rb;
            }
            if (++s == STAGES) {
                s = 0;
                ph ^= 1;
            }
        }
    }
    __syncthreads();
}

template <int MT, bool Q8>
cudaError_t launch_one(const GemmArgs &a, const TmapSet &tm, int grid, cudaStream_t st)
{
    using L = FmaSmem<MT, Q8>;
    auto kern = gemm_fma_kernel<MT, Q8>;
    static bool attr_done = false; // per instantiation; benign race (same value)
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
    return launch_pdl(kern, grid, FmaShape<MT>::THREADS, L::TOTAL, st, a, tm);
}

} // namespace

int fma_rows_blk(int mt) { return mt == 1 ? FmaShape<1>::RBLK : FmaShape<2>::RBLK; }

int fma_ctas_per_sm(int mt) { return mt == 1 ? FmaShape<1>::CPS : 1; }

int fma_smem_bytes(int mt, bool q8)
{
    switch (mt) {
    case 1: return q8 ? FmaSmem<1, true>::TOTAL : FmaSmem<1, false>::TOTAL;
    case 2: return q8 ? FmaSmem<2, true>::TOTAL : FmaSmem<2, false>::TOTAL;
    case 4: return q8 ? FmaSmem<4, true>::TOTAL : FmaSmem<4, false>::TOTAL;
    default: return q8 ? FmaSmem<4, true>::TOTAL : FmaSmem<4, false>::TOTAL;
    }
}

cudaError_t launch_gemm_fma(int mt, bool q8, const GemmArgs &a, const TmapSet &tm, int grid, cudaStream_t st)
{
    switch (mt) {
    case 1: return q8 ? launch_one<1, true>(a, tm, grid, st) : launch_one<1, false>(a, tm, grid, st);
    case 2: return q8 ? launch_one<2, true>(a, tm, grid, st) : launch_one<2, false>(a, tm, grid, st);
    case 4: return q8 ? launch_one<4, true>(a, tm, grid, st) : launch_one<4, false>(a, tm, grid, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace w12
