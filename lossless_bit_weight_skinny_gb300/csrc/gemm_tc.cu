// gemm_tc.cu -- W12 skinny GEMM on the tcgen05 tensor cores (activation rows
// padded to MT = 16, 32, 64, 128 or 256).
//
// The product is computed transposed: D[n][m] = sum_k W[n][k] x[m][k], with the
// decoded weight tile as the MMA "A" operand (128 output channels x 16 k per
// instruction) and the activation tile as "B" (MT rows, zero padded), FP32
// accumulators in tensor memory.  This is the Blackwell form of decoding W12
// records on the fly and feeding them to the tensor cores (SpecPilot, Figure
// 5(b) caption): instead of a register operand, the decode warps write the
// exact BF16 weights straight into tensor memory with tcgen05.st and the MMA
// reads A from there, so decoded weights never touch shared memory.
//
// Work unit: 128 rows x 256 columns, exactly one escape tile.  The (row block,
// k step) units are split over one persistent CTA per SM (stream-K, or whole
// row blocks when that is cheaper); row blocks shared by several CTAs are
// combined in a fixed order, by the last contributor or, above 64 rows, by the
// separate fix-up kernel (reduce.cu).
//
// CTA = 16 decode warps + a weight-TMA warp + an activation-TMA warp + an MMA
// warp + an escape warp, over three rings:
//   * weights (AE and B planes) in shared memory, handed back by the decode
//     warps as soon as they hold their raw planes in registers;
//   * activations (the MMA's B operand) in shared memory, released by the MMA:
//     a unit's four 64-column sub-tiles per slot up to 64 rows, one sub-tile
//     per slot from 128 rows;
//   * decoded weights (the A operand, 128 TMEM columns per unit), released by
//     the MMA.
// Decode warp (q, c) owns rows 32q..32q+31 of the unit (its TMEM lane
// quadrant) and columns 64c..64c+63.  Each thread decodes 64 weights of its
// row into 32 BF16x2 registers.  The escape warp reads each unit's escape list
// from global memory, up to a ring ahead, and sorts it into one short list per
// decode warp; after decoding, a decode warp overwrites its escaped slots in
// registers (through a small per-warp scratch row) and stores the 32 registers
// with one tcgen05.st.  Accumulators are double buffered up to 128 rows, so
// the epilogue of one row block overlaps the first products of the next; at
// 256 rows there is one 256-column buffer.
//
// Template flags: Q8 (the Q pass over the AE plane alone), EPI (the output
// modes: BF16, SiLU*mul; the plain FP32 store is a kernel of its own) and I8
// (an INT8 copy's bytes in place of the AE plane, row scales at the end).
#include "kernels.cuh"

namespace w12 {
namespace {

constexpr int kDecodeWarps = 16;
constexpr int kWarpW = kDecodeWarps;     // weight producer
constexpr int kWarpX = kDecodeWarps + 1; // activation producer
constexpr int kWarpM = kDecodeWarps + 2; // MMA issuer, tensor-memory owner
constexpr int kWarpE = kDecodeWarps + 3; // escape warp: sorts each unit's escapes per decode warp
constexpr int kThreads = (kDecodeWarps + 4) * 32;
constexpr int kPCap = 24;                // escapes per decode warp and unit kept in its list
static_assert(kTcKStep == 256 && kTcRows == 128, "one unit = one escape tile");

constexpr int a1024(int v) { return (v + 1023) & ~1023; }

template <int MT, bool Q8>
struct TcSmem {
    // weight stage: AE as two 128-column halves and B, each 128 rows of 128
    // bytes with the 128-byte swizzle
    static constexpr int AE_HALF = 128 * 128;
    static constexpr int AE = 2 * AE_HALF;
    static constexpr int B = Q8 ? 0 : 128 * 128;
    static constexpr int OFF_AE = 0;
    static constexpr int OFF_B = AE;
    static constexpr int WSTAGE = a1024(AE + B);
    // the escape warp's per-unit output, in a ring as deep as the weights':
    // entry count per decode warp u32[16], the unit's list start and end
    // u32[2], then up to kPCap entries per decode warp (a larger count means
    // "read the list yourself")
    static constexpr int PL_LO = 64;
    static constexpr int PL_LIST = 80;
    static constexpr int PL = Q8 ? 0 : PL_LIST + 4 * kPCap * kDecodeWarps;
    // tensor memory (512 columns): NA decoded A tiles of 128 columns, then ND
    // FP32 accumulator buffers of DW columns (MT <= 64: 3 x 128 + 2 x 64;
    // MT = 128: 2 x 128 + 2 x 128; MT = 256: 2 x 128 + 1 x 256, so a row
    // block's MMAs wait for the previous one's epilogue)
    static constexpr int NA = MT >= 128 ? 2 : 3;
    static constexpr uint32_t DCOL = NA * 128;
    static constexpr uint32_t DW = MT <= 64 ? 64 : MT;
    static constexpr int ND = MT == 256 ? 1 : 2;
    // activations: a unit needs four 64-column sub-tiles of MT rows (128-byte
    // swizzle); a ring slot holds SPS of them -- the whole unit's (SPS = 4)
    // up to 64 rows, one sub-tile (SPS = 1) from 128 rows, where a unit's 64
    // or 128 KB would leave too little room for the weights (at 256 rows three
    // slots, fewer than a unit's four: a slot is reloaded within the unit as
    // soon as the MMAs that read it complete)
    static constexpr int XSUB = MT * 128;
    static constexpr int SPS = MT >= 128 ? 1 : 4;
    static constexpr int SPU = 4 / SPS;       // slots per unit
    static constexpr int XSLOT = SPS * XSUB;
    static constexpr int XST = MT <= 32 ? 3 : MT == 64 ? 2 : MT == 128 ? W12_TC_XST128 : 3; // activation slots
    // per decode warp: one row of 32 BF16 pairs, for patching escapes
    static constexpr int SCR_PITCH = 144;
    static constexpr int SCR = Q8 ? 0 : kDecodeWarps * SCR_PITCH;
    static constexpr int BUDGET = 227 * 1024 - 2048;
    static constexpr int WST_RAW = (BUDGET - XST * XSLOT - SCR) / (WSTAGE + PL);
    static constexpr int WST = WST_RAW > 6 ? 6 : WST_RAW; // weight slots
    static constexpr int OFF_X = WST * WSTAGE;
    static constexpr int OFF_SCR = OFF_X + XST * XSLOT;
    static constexpr int OFF_PL = OFF_SCR + SCR;
    static constexpr int BARS = (OFF_PL + WST * PL + 15) & ~15;
    // w_full, w_empty [WST]; x_full, x_empty [XST]; a_full, a_empty [NA];
    // acc_full, acc_empty [2]; final, stall; pl_full, pl_empty [WST]
    static constexpr int NBARS = 2 * WST + 2 * XST + 2 * NA + 4 + 2 + 2 * WST;
    static constexpr int TOTAL = BARS + 8 * NBARS + 32 + 1024; // + slack to align the base
    static constexpr int W_TX = AE + B;
    static_assert(DCOL + ND * DW <= 512 && DW >= MT, "tensor memory budget");
    static_assert(WST >= 3 || (MT >= 128 && WST >= 2), "weight ring too shallow");
    static_assert(XST >= 2, "activation ring too shallow");
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

// Bounded wait that also gives up as soon as another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const GemmArgs &a,
                                              volatile int *abort_flag)
{
    if (*abort_flag)
        return false;
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > a.limit_ns) {
            *abort_flag = 1;
            report(a.status, kStatusTimeout);
            return false;
        }
    }
}

// Patch escapes into a decode thread's 32 BF16 pairs v (columns kb..kb+63 of
// its row) before they go to tensor memory.  The list is sorted by row, so the
// entries of one row are consecutive: the owning lane parks its pairs in the
// warp's scratch row, the lanes holding that row's entries overwrite the
// escaped 16-bit slots there, and the owner takes the pairs back before the
// next row's lane parks its own.
struct EscPatcher {
    uint8_t *scr;   // this warp's scratch row
    uint32_t rlo;   // first row of the warp's quadrant
    uint32_t kb;    // first column of the warp's quarter
    int lane;
    int cur = -1;   // lane whose pairs are parked

    __device__ __forceinline__ void park(uint32_t (&v)[32]) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4 *>(scr + 16 * i) = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    __device__ __forceinline__ void take(uint32_t (&v)[32]) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 w = *reinterpret_cast<const uint4 *>(scr + 16 * i);
            v[4 * i] = w.x;
            v[4 * i + 1] = w.y;
            v[4 * i + 2] = w.z;
            v[4 * i + 3] = w.w;
        }
    }
    // One chunk of entries, one per lane (e); h: the lanes whose entry lies in
    // this warp's quarter.  Row by row in list order: the row's lane parks its
    // pairs, then every lane holding an entry of that row writes its slot.
    __device__ __forceinline__ void apply(uint32_t e, uint32_t h, uint32_t (&v)[32])
    {
        const int mine_row = static_cast<int>((e >> 24) - rlo);
        const bool hit = (h >> lane) & 1u;
        while (h) {
            const int owner = static_cast<int>((__shfl_sync(0xffffffffu, e, __ffs(h) - 1) >> 24) - rlo);
            if (owner != cur) {
                if (lane == cur)
                    take(v);
                __syncwarp();
                if (lane == owner)
                    park(v);
                __syncwarp();
                cur = owner;
            }
            const bool mine = hit && mine_row == owner;
            if (mine)
                *reinterpret_cast<uint16_t *>(scr + 2 * (((e >> 16) & 0xFFu) - kb)) =
                    static_cast<uint16_t>(e & 0xFFFFu);
            h &= ~__ballot_sync(0xffffffffu, mine);
            __syncwarp();
        }
    }
    __device__ __forceinline__ void finish(uint32_t (&v)[32])
    {
        __syncwarp();
        if (lane == cur)
            take(v);
        __syncwarp();
        cur = -1;
    }
};

// 19 warps: 5 per SM sub-partition, whose 16K registers allow 102 per thread
// EPI: the output goes through the output mode (BF16, SiLU*mul); the default
// FP32 store is a kernel of its own, whose registers that code leaves alone.
// I8 (with Q8's layout: one weight plane, no escapes): the plane holds an
// INT8 copy, converted to BF16 exactly, and the row scales apply at the end.
template <int MT, bool Q8, bool EPI, bool I8 = false>
__global__ void __maxnreg__(96)
    gemm_tc_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tm_ae,
                   const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_x)
{
    using L = TcSmem<MT, Q8>;
    constexpr int WST = L::WST, XST = L::XST, kNA = L::NA;
    constexpr uint32_t kDCol = L::DCOL;
    constexpr uint32_t IDESC = idesc_bf16_f32(128, MT);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA tiles need 1024-byte aligned shared addresses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    const uint32_t w_full0 = smem_u32(bars);
    const uint32_t w_empty0 = smem_u32(bars + WST);
    const uint32_t x_full0 = smem_u32(bars + 2 * WST);
    const uint32_t x_empty0 = smem_u32(bars + 2 * WST + XST);
    const uint32_t a_full0 = smem_u32(bars + 2 * WST + 2 * XST);
    const uint32_t a_empty0 = smem_u32(bars + 2 * WST + 2 * XST + kNA);
    const uint32_t acc_full0 = smem_u32(bars + 2 * WST + 2 * XST + 2 * kNA);
    const uint32_t acc_empty0 = acc_full0 + 16;
    const uint32_t final_bar = acc_full0 + 32;
    const uint32_t stall_bar = acc_full0 + 40;
    const uint32_t pl_full0 = acc_full0 + 48, pl_empty0 = pl_full0 + 8 * WST;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + L::NBARS);
    volatile int *seg_last = abort_flag + 1;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(abort_flag + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int it0 = sk_begin(cta, grid, a.total_iters);
    const int n_it = sk_begin(cta + 1, grid, a.total_iters) - it0;
    const int nk = a.n_kstep;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WST; ++s) {
            mbar_init(w_full0 + 8 * s, 1);
            mbar_init(w_empty0 + 8 * s, kDecodeWarps);
            mbar_init(pl_full0 + 8 * s, 32);
            mbar_init(pl_empty0 + 8 * s, 32 * kDecodeWarps);
        }
        for (int s = 0; s < XST; ++s) {
            mbar_init(x_full0 + 8 * s, 1);
            mbar_init(x_empty0 + 8 * s, 1);
        }
        for (int b = 0; b < kNA; ++b) {
            mbar_init(a_full0 + 8 * b, kDecodeWarps);
            mbar_init(a_empty0 + 8 * b, 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(acc_full0 + 8 * d, 1);
            mbar_init(acc_empty0 + 8 * d, kDecodeWarps);
        }
        mbar_init(final_bar, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        *seg_last = 0;
        fence_barrier_init();
    }
    // escape-list bounds of the producer's first 64 units, loaded while the
    // CTA sets up
    uint32_t w_lo = 0, w_hi = 0, w_nlo = 0, w_nhi = 0;
    if (!Q8 && warp == kWarpE) {
        load_tile_window(a, it0, n_it, 0, lane, 128, w_lo, w_hi);
        load_tile_window(a, it0, n_it, 32, lane, 128, w_nlo, w_nhi);
    }
    if (warp == kWarpM) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == kWarpW) {
        // --------------------------- weight producer ---------------------------
        if (lane == 0) {
            prefetch_tmap(&tm_ae);
            if (!Q8)
                prefetch_tmap(&tm_b);
        }
        int issued = 0;
        int rb = it0 / nk, ks = it0 % nk, s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < n_it; ++it) {
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(w_empty0 + 8 * s, ph ^ 1, a, abort_flag));
            if (!ok)
                break;
            const int row0 = rb * 128, k0 = ks * 256;
            uint8_t *st = smem + s * L::WSTAGE;
            const uint32_t fb = w_full0 + 8 * s;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, L::W_TX);
                tma_load_2d(smem_u32(st + L::OFF_AE), &tm_ae, k0, row0, fb);
                tma_load_2d(smem_u32(st + L::OFF_AE + L::AE_HALF), &tm_ae, k0 + 128, row0, fb);
                if (!Q8)
                    tma_load_2d(smem_u32(st + L::OFF_B), &tm_b, k0 / 2, row0, fb);
            }
            issued = it + 1;
            if (++ks == nk) {
                ks = 0;
                ++rb;
            }
            if (++s == WST) {
                s = 0;
                ph ^= 1;
            }
        }
        // drain: every copy this warp started must land before the CTA exits
        for (int it = issued - 1; it >= 0 && it >= issued - WST; --it)
            mbar_wait(w_full0 + 8 * (it % WST), (it / WST) & 1, 1000000000ull);
    } else if (warp == kWarpX) {
        // ------------------------- activation producer -------------------------
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            // weights stream before the previous kernel in the stream has
            // finished; activations, which it may have written, only after it
            // has -- unless the caller declared them complete before that
            // kernel started (writes wait for it in any case: see the epilogue)
            if (!a.x_ready)
                pdl_wait_prior_grid();
            int issued = 0; // slot loads started
            int ks = it0 % nk, s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = 0; it < n_it && ok; ++it) {
                const int k0 = ks * 256;
#pragma unroll
                for (int h = 0; h < L::SPU; ++h) {
                    if (!wait_or_abort(x_empty0 + 8 * s, ph ^ 1, a, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *xs = smem + L::OFF_X + s * L::XSLOT;
                    const uint32_t fb = x_full0 + 8 * s;
                    mbar_arrive_expect_tx(fb, L::XSLOT);
#pragma unroll
                    for (int j = 0; j < L::SPS; ++j)
                        tma_load_2d(smem_u32(xs + j * L::XSUB), &tm_x, k0 + 64 * (h * L::SPS + j), 0, fb);
                    ++issued;
                    if (++s == XST) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (++ks == nk)
                    ks = 0;
            }
            for (int it = issued - 1; it >= 0 && it >= issued - XST; --it)
                mbar_wait(x_full0 + 8 * (it % XST), (it / XST) & 1, 1000000000ull);
        }
        __syncwarp();
    } else if (warp == kWarpM) {
        // ------------------------------ MMA issuer -----------------------------
        if (lane == 0) {
            // shared-memory descriptor of the first activation slot; slot sx
            // adds sx * XSLOT / 16, and within a slot the K-steps of 16 columns
            // add a fixed offset (address field in 16-byte units: +2 per 16
            // columns, +XSUB/16 per 64-column sub-tile)
            const uint64_t xdesc0 = smem_desc_sw128(smem_u32(smem + L::OFF_X), 1024);
            int seg = 0;
            int ks = it0 % nk, sx = 0, b = 0;
            uint32_t phx = 0, pha = 0;
            for (int it = 0; it < n_it; ++it) {
                const bool seg_start = (it == 0) || (ks == 0);
                const bool seg_end = (ks == nk - 1) || (it == n_it - 1);
                const int db = seg % L::ND;
                bool ok = true;
                // accumulator buffer db was last read by the epilogue of segment seg - ND
                if (seg_start && seg >= L::ND)
                    ok = wait_or_abort(acc_empty0 + 8 * db, ((seg / L::ND) - 1) & 1, a, abort_flag);
                ok = wait_or_abort(a_full0 + 8 * b, pha, a, abort_flag) && ok;
                const uint32_t d = tmem + kDCol + L::DW * db;
                const uint32_t a0 = tmem + b * 128;
#pragma unroll
                for (int h = 0; h < L::SPU; ++h) {
                    const bool okx = wait_or_abort(x_full0 + 8 * sx, phx, a, abort_flag) && ok;
                    tc_fence_after();
                    if (okx) {
                        const uint64_t bdesc = xdesc0 + static_cast<uint64_t>(sx * (L::XSLOT >> 4));
#pragma unroll
                        for (int jj = 0; jj < 4 * L::SPS; ++jj) {
                            const int j = h * 4 * L::SPS + jj; // K-step of 16 columns in the unit
                            const uint64_t bj = bdesc + static_cast<uint64_t>((jj >> 2) * (L::XSUB >> 4) + (jj & 3) * 2);
                            if (j == 0)
                                tc_mma_ts(d, a0, bj, IDESC, seg_start ? 0u : 1u);
                            else
                                tc_mma_ts_acc(d, a0 + j * 8, bj, IDESC);
                        }
                    }
                    // each commit arrives once every MMA issued so far has completed
                    tc_commit(x_empty0 + 8 * sx);
                    if (++sx == XST) {
                        sx = 0;
                        phx ^= 1;
                    }
                }
                tc_commit(a_empty0 + 8 * b);
                if (seg_end) {
                    tc_commit(acc_full0 + 8 * db);
                    ++seg;
                }
                if (++ks == nk)
                    ks = 0;
                if (++b == kNA) {
                    b = 0;
                    pha ^= 1;
                }
            }
            tc_commit(final_bar);
            mbar_wait(final_bar, 0, 1000000000ull);
        }
        __syncwarp();
    } else if (warp == kWarpE) {
        // ------------------------------ escape warp ---------------------------
        // Per unit, every escape entry of the tile (read straight from global
        // memory, up to 512 in one round of loads) goes to the list of the
        // decode warp that owns its slot (row quadrant q = row / 32, column
        // quarter c = column / 64): 32 entries at a time, one per lane, ranked
        // within the lanes of the same target so that each list keeps the
        // order of the tile's list (rows ascending).  It needs nothing from the
        // weight stages and runs up to a ring ahead of the decode warps.
        if (!Q8) {
            int s = 0;
            uint32_t ph = 0;
            const uint32_t lt = (1u << lane) - 1u;
            for (int it = 0; it < n_it; ++it) {
                if (it > 0 && (it & 31) == 0) { // next window of tile bounds; prefetch the one after
                    w_lo = w_nlo;
                    w_hi = w_nhi;
                    load_tile_window(a, it0, n_it, it + 32, lane, 128, w_nlo, w_nhi);
                }
                const uint32_t lo = __shfl_sync(0xffffffffu, w_lo, it & 31);
                const uint32_t hi = __shfl_sync(0xffffffffu, w_hi, it & 31);
                const uint32_t cnt = hi >= lo ? hi - lo : 0u;
                bool ok = true;
                if (it >= WST)
                    ok = wait_or_abort(pl_empty0 + 8 * s, ph ^ 1, a, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                uint8_t *pl = smem + L::OFF_PL + s * L::PL;
                uint32_t *cnt_s = reinterpret_cast<uint32_t *>(pl);
                uint32_t *lists = reinterpret_cast<uint32_t *>(pl + L::PL_LIST);
                if (lane < kDecodeWarps)
                    cnt_s[lane] = 0u;
                if (lane == 0)
                    *reinterpret_cast<uint2 *>(pl + L::PL_LO) = make_uint2(lo, lo + cnt);
                __syncwarp();
                for (uint32_t j1 = 0; ok && j1 < cnt; j1 += 512) {
                    uint32_t e16[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const uint32_t j = j1 + 32 * u + static_cast<uint32_t>(lane);
                        e16[u] = j < cnt ? __ldg(a.esc + lo + j) : 0u;
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        if (j1 + 32 * u >= cnt)
                            break;
                        const bool valid = j1 + 32 * u + static_cast<uint32_t>(lane) < cnt;
                        const uint32_t e = e16[u];
                        const uint32_t w = ((e >> 22) & 3u) * 4u + ((e >> 29) & 3u); // quarter * 4 + quadrant
                        const uint32_t key = valid ? w : 64u + static_cast<uint32_t>(lane);
                        const uint32_t peers = __match_any_sync(0xffffffffu, key);
                        const uint32_t base = valid ? cnt_s[w] : 0u;
                        const uint32_t pos = base + __popc(peers & lt);
                        if (valid && pos < static_cast<uint32_t>(kPCap))
                            lists[w * kPCap + pos] = e;
                        __syncwarp();
                        if (valid && (peers & lt) == 0u)
                            cnt_s[w] = base + __popc(peers);
                        __syncwarp();
                    }
                }
                __syncwarp();
                mbar_arrive(pl_full0 + 8 * s); // every lane: its writes are visible
                if (++s == WST) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else {
        // ------------------------------ decode warps --------------------------
        const int q = warp & 3, c = warp >> 2;
        const int row = 32 * q + lane; // this thread's row in the unit = TMEM lane
        const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t rlo = static_cast<uint32_t>(32 * q);
        const uint32_t kb = static_cast<uint32_t>(64 * c);
        uint32_t eb2 = 0;
        int cur_rb = -1, seg = 0;
        int rb = it0 / nk, ks = it0 % nk, s = 0, b = 0;
        uint32_t ph = 0, pha = 0;
        for (int it = 0; it < n_it; ++it) {
            // window base of a new row block: start the load before waiting
            uint32_t e_pre = 1u;
            if (rb != cur_rb && rb * 128 + row < a.N)
                e_pre = I8 ? 1u : __ldg(a.ebase + rb * 128 + row);
            bool ok = wait_or_abort(w_full0 + 8 * s, ph, a, abort_flag);
            if (a.inject_stall)
                ok = wait_or_abort(stall_bar, 0, a, abort_flag) && ok;
            // After an abort the loop keeps its shape (every warp still meets
            // every barrier) but works on stale data and reads nothing
            // through addresses taken from shared memory.
            ok = __all_sync(0xffffffffu, ok);
            const int row0 = rb * 128;
            const uint8_t *st = smem + s * L::WSTAGE;
            if (rb != cur_rb) {
                cur_rb = rb;
                eb2 = (e_pre << 7) | (e_pre << 23);
            }

            // 1. raw planes of this row's 64 columns: four 16-byte AE chunks
            //    and two B chunks (128-byte swizzle: chunk j of row r sits at
            //    j ^ (r & 7))
            uint4 aq[4], bq[2];
            {
                const uint8_t *ae_row = st + L::OFF_AE + (c >> 1) * L::AE_HALF + row * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    aq[i] = *reinterpret_cast<const uint4 *>(ae_row + ((((c & 1) * 4 + i) ^ (row & 7)) << 4));
                if (!Q8) {
                    const uint8_t *b_row = st + L::OFF_B + row * 128;
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        bq[i] = *reinterpret_cast<const uint4 *>(b_row + (((2 * c + i) ^ (row & 7)) << 4));
                } else {
                    bq[0] = bq[1] = make_uint4(0u, 0u, 0u, 0u);
                }
            }

            // 2. the stage is no longer needed: hand it back (this warp's
            //    escapes come from the escape warp's list for it)
            __syncwarp();
            if (lane == 0)
                mbar_arrive(w_empty0 + 8 * s);

            // 3. decode to exact BF16 pairs (escaped slots hold their placeholder)
            uint32_t v[32];
            {
                const uint32_t bw[8] = {bq[0].x, bq[0].y, bq[0].z, bq[0].w,
                                        bq[1].x, bq[1].y, bq[1].z, bq[1].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (I8) {
                        decode_i8_group(aq[i].x, aq[i].y, v + 8 * i);
                        decode_i8_group(aq[i].z, aq[i].w, v + 8 * i + 4);
                    } else {
                        decode_group<Q8>(aq[i].x, aq[i].y, bw[2 * i], eb2, v + 8 * i);
                        decode_group<Q8>(aq[i].z, aq[i].w, bw[2 * i + 1], eb2, v + 8 * i + 4);
                    }
                }
            }

            // 4. escapes of this warp's rows and columns, patched in registers
            if (!Q8) {
                bool okp = wait_or_abort(pl_full0 + 8 * s, ph, a, abort_flag);
                okp = __all_sync(0xffffffffu, okp) && ok;
                const uint8_t *pl = smem + L::OFF_PL + s * L::PL;
                const uint32_t n = okp ? reinterpret_cast<const uint32_t *>(pl)[warp] : 0u;
                uint32_t my_e = 0u;
                uint2 lohi = make_uint2(0u, 0u);
                if (n <= static_cast<uint32_t>(kPCap)) {
                    if (static_cast<uint32_t>(lane) < n)
                        my_e = reinterpret_cast<const uint32_t *>(pl + L::PL_LIST)[warp * kPCap + lane];
                } else {
                    lohi = *reinterpret_cast<const uint2 *>(pl + L::PL_LO);
                }
                mbar_arrive(pl_empty0 + 8 * s); // every lane, after its own reads
                if (n != 0u) {
                    EscPatcher pt{smem + L::OFF_SCR + warp * L::SCR_PITCH, rlo, kb, lane};
                    if (n <= static_cast<uint32_t>(kPCap)) {
                        pt.apply(my_e, n >= 32u ? 0xffffffffu : (1u << n) - 1u, v);
                    } else {
                        // more than the list holds: this quadrant's entries of the
                        // tile from global memory, four chunks of 32 at a time
                        const size_t t = static_cast<size_t>(rb) * a.tiles_c + ks;
                        const uint32_t cnt = lohi.y - lohi.x;
                        const uint32_t q_lb = min(static_cast<uint32_t>(__ldg(a.gptr + 16 * t + 4 * q)), cnt);
                        const uint32_t q_ub =
                            q == 3 ? cnt : min(static_cast<uint32_t>(__ldg(a.gptr + 16 * t + 4 * q + 4)), cnt);
                        for (uint32_t j0 = q_lb; j0 < q_ub; j0 += 128) {
                            uint32_t e4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t idx = j0 + 32 * u + static_cast<uint32_t>(lane);
                                e4[u] = idx < q_ub ? __ldg(a.esc + lohi.x + idx) : 0u;
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const bool valid = j0 + 32 * u + static_cast<uint32_t>(lane) < q_ub;
                                pt.apply(e4[u],
                                         __ballot_sync(0xffffffffu, valid && ((e4[u] >> 16) & 0xFFu) - kb < 64u), v);
                            }
                        }
                    }
                    pt.finish(v);
                }
            }

            // 5. into tensor memory, once the MMA is done with this A buffer
            wait_or_abort(a_empty0 + 8 * b, pha ^ 1, a, abort_flag);
            __syncwarp();
            tc_fence_after();
            tmem_st32(tmem + static_cast<uint32_t>(b * 128) + t_lane + kb / 2, v);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(a_full0 + 8 * b);

            if (ks == nk - 1 || it == n_it - 1) {
                // ---- accumulators of this row block are final: read them out ----
                // nothing is written before the previous kernel in the stream
                // has completed (at once when the activation load waited for it)
                pdl_wait_prior_grid();
                const int db = seg % L::ND;
                wait_or_abort(acc_full0 + 8 * db, (seg / L::ND) & 1, a, abort_flag);
                __syncwarp();
                tc_fence_after();
                constexpr int PART = MT / 4;              // accumulator columns read by this warp
                constexpr int CH = PART < 16 ? PART : 16; // read and stored in chunks of CH
                const bool used = c * PART < a.M;
                const int c_first = sk_owner(rb * nk, grid, a.total_iters);
                const int c_last = sk_owner((rb + 1) * nk - 1, grid, a.total_iters);
                const bool direct = (c_first == c_last);
                const int slot = direct ? 0 : sk_slot(cta, rb, grid, a.total_iters, nk);
                const int n = row0 + row;
                float rs = 1.f; // an INT8 copy's row scale
                if constexpr (I8)
                    rs = n < a.N ? __ldg(a.scale + n) : 0.f;
                if (used) {
                    const uint32_t dcol = tmem + t_lane + kDCol + L::DW * db + c * PART;
                    const bool pair = EPI && direct && (a.out_mode & kOutSiluMul);
#pragma unroll
                    for (int h = 0; h < PART / CH; ++h) {
                        uint32_t d[CH];
                        if constexpr (CH == 4)
                            tmem_ld4(dcol, d);
                        else if constexpr (CH == 8)
                            tmem_ld8(dcol, d);
                        else
                            tmem_ld16(dcol + 16 * h, d);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < CH; ++j) {
                            const float v = I8 ? __uint_as_float(d[j]) * rs : __uint_as_float(d[j]);
                            const int m = c * PART + h * CH + j;
                            // row + 1 (the up row of an even gate row) is lane + 1
                            const float next = pair ? __shfl_down_sync(0xffffffffu, v, 1) : 0.f;
                            if (m < a.M) {
                                if (direct) {
                                    if (n < a.N) {
                                        if constexpr (EPI)
                                            emit_y(a, m, n, v, next);
                                        else
                                            static_cast<float *>(a.y)[static_cast<size_t>(m) * a.N + n] = v;
                                    }
                                } else {
                                    a.partials[(static_cast<size_t>(slot) * a.M + m) * 128 + row] = v;
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acc_empty0 + 8 * db);
                ++seg;

                if (!direct && !a.defer) {
                    // the CTA barrier orders every thread's partial stores before
                    // thread 0's release-acquire arrival (cumulativity), and that
                    // arrival before everyone's reads of the other partials
                    named_bar_sync(1, kDecodeWarps * 32);
                    if (threadIdx.x == 0)
                        *seg_last = sk_arrive(a.counters + rb, c_last - c_first + 1) ? 1 : 0;
                    named_bar_sync(1, kDecodeWarps * 32);
                    if (*seg_last)
                        sk_reduce_block<EPI>(a, rb, 128, grid, c_first, c_last, threadIdx.x, kDecodeWarps * 32);
                }
            }
            if (++ks == nk) {
                ks = 0;
                ++rb;
            }
            if (++s == WST) {
                s = 0;
                ph ^= 1;
            }
            if (++b == kNA) {
                b = 0;
                pha ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpM) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MT, bool Q8, bool EPI, bool I8 = false>
cudaError_t launch_one(const GemmArgs &a, const CUtensorMap *tm_ae, const CUtensorMap *tm_b,
                       const CUtensorMap *tm_x, int grid, cudaStream_t st)
{
    using L = TcSmem<MT, Q8>;
    auto kern = gemm_tc_kernel<MT, Q8, EPI, I8>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
    return launch_pdl(kern, grid, kThreads, L::TOTAL, st, a, *tm_ae, *tm_b, *tm_x);
}

} // namespace

int tc_smem_bytes(int mt, bool q8)
{
    switch (mt) {
    case 16: return q8 ? TcSmem<16, true>::TOTAL : TcSmem<16, false>::TOTAL;
    case 32: return q8 ? TcSmem<32, true>::TOTAL : TcSmem<32, false>::TOTAL;
    case 64: return q8 ? TcSmem<64, true>::TOTAL : TcSmem<64, false>::TOTAL;
    case 128: return q8 ? TcSmem<128, true>::TOTAL : TcSmem<128, false>::TOTAL;
    default: return q8 ? TcSmem<256, true>::TOTAL : TcSmem<256, false>::TOTAL;
    }
}

template <int MT>
cudaError_t launch_mt(bool q8, bool i8, const GemmArgs &a, const CUtensorMap *tm_ae, const CUtensorMap *tm_b,
                      const CUtensorMap *tm_x, int grid, cudaStream_t st)
{
    if (i8)
        return a.out_mode ? launch_one<MT, true, true, true>(a, tm_ae, tm_b, tm_x, grid, st)
                          : launch_one<MT, true, false, true>(a, tm_ae, tm_b, tm_x, grid, st);
    if (a.out_mode)
        return q8 ? launch_one<MT, true, true>(a, tm_ae, tm_b, tm_x, grid, st)
                  : launch_one<MT, false, true>(a, tm_ae, tm_b, tm_x, grid, st);
    return q8 ? launch_one<MT, true, false>(a, tm_ae, tm_b, tm_x, grid, st)
              : launch_one<MT, false, false>(a, tm_ae, tm_b, tm_x, grid, st);
}

cudaError_t launch_gemm_tc(int mt, bool q8, bool i8, const GemmArgs &a, const CUtensorMap *tm_ae,
                           const CUtensorMap *tm_b, const CUtensorMap *tm_x, int grid,
                           cudaStream_t st)
{
    switch (mt) {
    case 16: return launch_mt<16>(q8, i8, a, tm_ae, tm_b, tm_x, grid, st);
    case 32: return launch_mt<32>(q8, i8, a, tm_ae, tm_b, tm_x, grid, st);
    case 64: return launch_mt<64>(q8, i8, a, tm_ae, tm_b, tm_x, grid, st);
    case 128: return launch_mt<128>(q8, i8, a, tm_ae, tm_b, tm_x, grid, st);
    case 256: return launch_mt<256>(q8, i8, a, tm_ae, tm_b, tm_x, grid, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace w12
