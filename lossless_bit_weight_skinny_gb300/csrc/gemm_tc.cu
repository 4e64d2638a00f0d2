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
// CTA = two decode groups of eight warps + a weight-TMA warp + an
// activation-TMA warp + an MMA warp + an escape-list warp (640 threads).  The
// groups take the units in turn (group 0 the even ones of the CTA's range,
// group 1 the odd ones), so that one group's loads and waits overlap the
// other's decode, which is integer work on the ALU pipe.  Warp (q, h) of a
// group owns TMEM lanes 32q..32q+31, i.e. rows 32q..32q+31 of the unit, and
// columns 128h..128h+127: each thread decodes 128 weights of its row as two
// chunks of 64 (32 BF16x2 registers, one tcgen05.st each).  The helper
// warpgroup runs on 32 registers a thread and hands the rest to the decode
// warpgroups (setmaxnreg), which hold a row's raw planes and a chunk's
// pairs at once.
//
// Three rings:
//   * weights (AE and B planes, plus the unit's 128 window bases) in shared
//     memory, handed back once the decode warps' loads of them are done;
//   * activations (the MMA's B operand) in shared memory, released by the MMA:
//     a unit's four 64-column sub-tiles per slot up to 64 rows, one sub-tile
//     per slot from 128 rows;
//   * decoded weights (the A operand, 128 TMEM columns per unit), released by
//     the MMA.
// The escape-list warp copies each unit's escape entries (sorted by row, so
// the rows of a TMEM lane quadrant are one contiguous run) next to the
// quadrant bounds into a shared-memory ring that runs ahead of the decode
// groups.  A decode warp patches the escaped slots of a chunk in registers
// before storing it: the rows holding escapes park their pairs in a small
// per-warp scratch area, a few rows at a time, the lanes holding the entries
// overwrite the escaped 16-bit slots there, and the rows take their pairs
// back.  The MMA warp runs its loop on all lanes, so that descriptors and
// addresses stay warp-uniform, and one elected lane issues the MMAs.
// Accumulators are double buffered up to 128 rows, so the epilogue of one row
// block overlaps the products of the next; at 256 rows there is one 256-column
// buffer.  The epilogue of a row block is done by the group that decoded its
// last unit.
//
// Barrier phases: an mbarrier's parity wait cannot tell phase k + 2 from phase
// k, so every barrier must be waited on phase by phase by one waiter.  The
// barriers that the two groups wait on (weights full, A buffer free,
// accumulators full) therefore exist once per group, and the producers arrive
// on the copy of the group that takes (or next takes) the unit.

// Template flags: Q8 (the Q pass over the AE plane alone), EPI (the output
// modes: BF16, SiLU*mul; the plain FP32 store is a kernel of its own) and I8
// (an INT8 copy's bytes in place of the AE plane, row scales at the end).
#include "kernels.cuh"

namespace w12 {
namespace {

constexpr int kGroups = 2;                       // decode groups, taking units in turn
constexpr int kSplit = 2;                        // warps per TMEM lane quadrant in a group (column halves)
constexpr int kGroupWarps = 4 * kSplit;          // warps of a decode group
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kCols = 256 / kSplit;              // columns of a unit each decode thread owns
constexpr int kChunks = kCols / 64;              // 64-column chunks per thread and unit
constexpr int kDecodeWarps = kGroups * kGroupWarps;
constexpr int kWarpW = kDecodeWarps;             // weight producer
constexpr int kWarpX = kDecodeWarps + 1;         // activation producer
constexpr int kWarpM = kDecodeWarps + 2;         // MMA issuer, tensor-memory owner
constexpr int kWarpE = kDecodeWarps + 3;         // escape-list stager
constexpr int kThreads = (kDecodeWarps + 4) * 32;
// Registers.  The block is launched with kRegLaunch per thread; the helper
// warpgroup (the last four warps) gives registers back with setmaxnreg and
// the decode warpgroups take them: their shares add up to the launch total.
constexpr int kRegLaunch = (65536 / kThreads) & ~7;
constexpr int kRegHelper = 32;
constexpr int kRegDecode = ((kRegLaunch * kThreads - 128 * kRegHelper) / (kDecodeWarps * 32)) & ~7;
static_assert(kRegDecode * kDecodeWarps * 32 + kRegHelper * 128 <= kRegLaunch * kThreads,
              "register shares exceed the launch allocation");
static_assert(kDecodeWarps % 4 == 0 && kGroupWarps % 4 == 0, "warpgroups of one role");
#ifndef W12_TC_ESC_CAP
#define W12_TC_ESC_CAP 512
#endif
constexpr int kEscCap = W12_TC_ESC_CAP;          // entries of a unit staged in shared memory
constexpr int kPlSt = 2 * kGroups;               // escape-list stages (each serves one group)
// Rows a decode warp patches at once (per activation-tile height).  Up to 64
// activation rows every row of a warp has a parking slot, and a chunk takes
// one round (measured on GB300, 17408 x 5120 at 16 / 32 rows: 33.8 / 35.2 us
// with 4 rows a round, 30.9 / 31.7 with all 32; 64 rows: see the activation
// slots below); from 128 rows the 74 KB this takes would leave too little
// room for the weights, so 4 rows a round.
#ifndef W12_TC_PARK16
#define W12_TC_PARK16 32
#endif
#ifndef W12_TC_PARK32
#define W12_TC_PARK32 32
#endif
#ifndef W12_TC_PARK64
#define W12_TC_PARK64 32
#endif
// Batches of 32 escape entries per patch round when a quadrant's list is
// longer than a warp (32-row parking): measured on GB300 on 17408 x 5120 at
// 16 rows with a dense escape tail (9e-3, ~74 entries a quadrant): 63.8 us
// with one batch a round, 54.9 with 2, 51.1 with 4, 48.9 with 3 (the
// projection draw 31.5 -> 30.9 us with 3 against 4); at 32 rows, 31.3 us with
// 2 and 32.3 with 4.
#ifndef W12_TC_PATCH_BATCHES16
#define W12_TC_PATCH_BATCHES16 3
#endif
#ifndef W12_TC_PATCH_BATCHES
#define W12_TC_PATCH_BATCHES 2
#endif
// At 64 rows the exact pass holds half a unit's activations per ring slot
// (three slots of 16 KB instead of two of 32 KB), which leaves room for a
// parking slot per row: measured on GB300, 17408 x 5120: 36.4 us with whole-unit
// slots and 8 rows a round, 37.8 with half-unit slots alone, 33.3 with both
// (5120 x 17408: 40.1 -> 37.5); the Q pass keeps whole-unit slots (20.3 against
// 20.6 us).
#ifndef W12_TC_SPS64
#define W12_TC_SPS64 2 // 64-column activation sub-tiles per ring slot at 64 rows (exact pass)
#endif
#ifndef W12_TC_WST_MAX
#define W12_TC_WST_MAX 6 // most weight stages
#endif
template <int MT>
__host__ __device__ constexpr int park_rows()
{
    return MT == 16 ? W12_TC_PARK16 : MT == 32 ? W12_TC_PARK32 : MT == 64 ? W12_TC_PARK64 : 4;
}
constexpr int kParkPitch = 144;                  // bytes per parked row (128 + 16: banks spread)
static_assert(kTcKStep == 256 && kTcRows == 128, "one unit = one escape tile");

template <int MT, bool Q8>
struct TcSmem {
    // activations: a unit needs four 64-column sub-tiles of MT rows (128-byte
    // swizzle); a ring slot holds SPS of them -- the whole unit's (SPS = 4) up
    // to 64 rows, one sub-tile (SPS = 1) from 128 rows, where a unit's 64 or
    // 128 KB would leave too little room for the weights (at 256 rows three
    // slots, fewer than a unit's four: a slot is reloaded within the unit as
    // soon as the MMAs that read it complete)
    static constexpr int XSUB = MT * 128;
    static constexpr int SPS = MT >= 128 ? 1 : (MT == 64 && !Q8) ? W12_TC_SPS64 : 4;
    static constexpr int SPU = 4 / SPS; // slots per unit
    static constexpr int XSLOT = SPS * XSUB;
    static constexpr int XST = MT <= 32 ? 3 : MT == 64 ? (SPS == 4 ? 2 : 3) : MT == 128 ? W12_TC_XST128 : 3;
    // weight stage: AE as two 128-column halves and B, each 128 rows of 128
    // bytes with the 128-byte swizzle; the rows' window bases beside it
    static constexpr int AE_HALF = 128 * 128;
    static constexpr int AE = 2 * AE_HALF;
    static constexpr int B = Q8 ? 0 : 128 * 128;
    static constexpr int WSTAGE = AE + B;
    static constexpr int EB = 128;
    // escape list of a unit: header u32[8] = {first entry, count, quadrant
    // bounds[5], matrix}, then up to kEscCap entries
    static constexpr int PL_HDR = 32;
    static constexpr int PL = Q8 ? 0 : PL_HDR + 4 * kEscCap;
    static constexpr int SCR = Q8 ? 0 : kDecodeWarps * park_rows<MT>() * kParkPitch;
    // tensor memory (512 columns): NA decoded A tiles of 128 columns, then ND
    // FP32 accumulator buffers of DW columns (MT <= 64: 3 x 128 + 2 x 64;
    // MT = 128: 2 x 128 + 2 x 128; MT = 256: 2 x 128 + 1 x 256)
    static constexpr int NA = MT >= 128 ? 2 : 3;
    static constexpr uint32_t DCOL = NA * 128;
    static constexpr uint32_t DW = MT <= 64 ? 64 : MT;
    static constexpr int ND = MT == 256 ? 1 : 2;
    static constexpr int BUDGET = 227 * 1024 - 1024 - 640; // alignment slack, barriers
    static constexpr int WST_RAW = (BUDGET - XST * XSLOT - SCR - kPlSt * PL) / (WSTAGE + EB);
    static constexpr int WST = WST_RAW > W12_TC_WST_MAX ? W12_TC_WST_MAX : WST_RAW; // weight stages
    static constexpr int OFF_X = 0;
    static constexpr int OFF_W = XST * XSLOT;
    static constexpr int OFF_EB = OFF_W + WST * WSTAGE;
    static constexpr int OFF_PL = OFF_EB + WST * EB;
    static constexpr int OFF_SCR = OFF_PL + kPlSt * PL;
    static constexpr int BARS = (OFF_SCR + SCR + 15) & ~15;
    // w_full [WST][kGroups], w_empty [WST], pl_full [kPlSt], pl_empty [kPlSt],
    // x_full, x_empty [XST], a_full [NA], a_empty [NA][kGroups],
    // acc_full [2][kGroups], acc_empty [2], final, stall
    static constexpr int NBARS = (kGroups + 1) * WST + 2 * kPlSt + 2 * XST + (kGroups + 1) * NA + 2 * kGroups + 2 + 2;
    static constexpr int TOTAL = BARS + 8 * NBARS + 32 + 1024; // + flags (4 + kGroups ints), + slack to align the base
    static constexpr int W_TX = AE + B;
    static_assert(DCOL + ND * DW <= 512 && DW >= MT, "tensor memory budget");
    static_assert(WST >= 2, "weight ring too shallow");
    static_assert(XST >= 2, "activation ring too shallow");
    static_assert(OFF_W % 1024 == 0 && WSTAGE % 1024 == 0, "swizzled stages need 1024-byte alignment");
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

__host__ __device__ constexpr int gcd_c(int a, int b) { return b ? gcd_c(b, a % b) : a; }

// Use count of a weight stage by one group before unit `it` (stage it % WST,
// group it % kGroups): a (stage, group) pair recurs every lcm(WST, kGroups)
// units.
template <int WST>
__device__ __forceinline__ uint32_t stage_use(int it)
{
    constexpr int period = WST / gcd_c(WST, kGroups) * kGroups;
    return static_cast<uint32_t>(it / period);
}

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

// One BF16x2 pair (weights 2i, 2i+1 of a group of 8) from the group's AE word
// holding those two bytes and its B word (SpecPilot, Figure 5(a) caption):
// PRMT spreads the two AE bytes into two 16-bit lanes, replicating each
// byte's sign into the lane's high byte; then per lane
//   sign (bit 15) | (ebase + E) << 7 | (A & 7) << 4 | B,
// with eb2 = ebase << 7 in both lanes.  The B nibbles of pair i sit 4i bits up
// in the B word; the shift is the high word of a multiply by 2^(32 - 4i)
// (`bm`, passed in so that it stays a multiply): PRMT, LOP3, LOP3, LOP3 on
// the ALU pipe and two multiply-adds on the FMA pipe per pair.
template <int I, bool Q8>
__device__ __forceinline__ uint32_t dec_pair(uint32_t ae_word, uint32_t bw, uint32_t eb2, uint32_t bm)
{
    uint32_t p, t, r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(p) : "r"(ae_word), "n"((I & 1) ? 0xB3A2 : 0x9180));
    asm("and.b32 %0, %1, 0x000F000F;" : "=r"(t) : "r"(p));
    asm("mad.lo.u32 %0, %1, 128, %2;" : "=r"(t) : "r"(t), "r"(eb2));
    asm("lop3.b32 %0, %1, 0x80708070, %2, 0xEA;" : "=r"(r) : "r"(p), "r"(t)); // (p & m) | t
    if (!Q8) {
        uint32_t b = bw;
        if (I)
            asm("mul.hi.u32 %0, %1, %2;" : "=r"(b) : "r"(bw), "r"(bm));
        asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(b), "r"(r)); // (b & m) | r
    }
    return r;
}

// Escape-list bounds and quadrant splits of the units it0 + first + lane (one
// per lane): first entry, count, and the counts below rows 32, 64, 96 of the
// tile (from the row-group index), packed as g12 = rows<32 | rows<64 << 16,
// with the unit's matrix in the top byte of g3.
__device__ __forceinline__ void esc_window(const GemmArgs &a, int it0, int n_it, int first, int lane,
                                           uint32_t &lo, uint32_t &cnt, uint32_t &g12, uint32_t &g3)
{
    lo = cnt = g12 = g3 = 0u;
    if (first + lane < n_it) {
        const int u = it0 + first + lane;
        const int rb = u / a.n_kstep;
        const int g = mat_of(a, rb);
        const MatArgs &mm = a.mat[g];
        const size_t t = static_cast<size_t>(rb - mm.rb0) * a.tiles_c + u % a.n_kstep;
        lo = __ldg(mm.tile_ptr + t);
        const uint32_t hi = __ldg(mm.tile_ptr + t + 1);
        cnt = hi >= lo ? hi - lo : 0u;
        const uint16_t *gp = mm.gptr + 16 * t;
        g12 = static_cast<uint32_t>(__ldg(gp + 4)) | (static_cast<uint32_t>(__ldg(gp + 8)) << 16);
        g3 = static_cast<uint32_t>(__ldg(gp + 12)) | (static_cast<uint32_t>(g) << 24);
    }
}

// Overwrite the escaped slots of one chunk (64 columns) in the 32 BF16 pairs v
// of this thread's row.  e: one escape entry per lane, inj: it lies in this
// chunk.  The rows holding such entries park their pairs in the warp's
// scratch area, PARK rows at a time (in row order); every lane holding an
// entry of a parked row writes the exact 16 bits into the row's slot; the
// rows take their pairs back.
// With a parking slot for every row (PARK = 32): R batches of 32 entries in
// one round -- every row holding one of them parks once, all entries are
// written, the rows take their pairs back.
template <int R>
__device__ __forceinline__ void patch_rows(const uint32_t (&e)[R], const bool (&inj)[R], uint32_t q32, uint8_t *scr,
                                           int lane, uint32_t (&v)[32])
{
    uint32_t mine_rows = 0u;
#pragma unroll
    for (int r = 0; r < R; ++r)
        mine_rows |= inj[r] ? 1u << (((e[r] >> 24) - q32) & 31u) : 0u;
    const uint32_t rowmask = __reduce_or_sync(0xffffffffu, mine_rows);
    const bool mine = (rowmask >> lane) & 1u;
    uint8_t *const row_s = scr + lane * kParkPitch;
    if (mine) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4 *>(row_s + 16 * i) = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (inj[r])
            *reinterpret_cast<uint16_t *>(scr + (((e[r] >> 24) - q32) & 31u) * kParkPitch + 2 * ((e[r] >> 16) & 63u)) =
                static_cast<uint16_t>(e[r] & 0xFFFFu);
    __syncwarp();
    if (mine) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 w = *reinterpret_cast<const uint4 *>(row_s + 16 * i);
            v[4 * i] = w.x;
            v[4 * i + 1] = w.y;
            v[4 * i + 2] = w.z;
            v[4 * i + 3] = w.w;
        }
    }
    __syncwarp();
}

template <int PARK>
__device__ __forceinline__ void patch_chunk(uint32_t e, bool inj, uint32_t q32, uint8_t *scr, int lane,
                                            uint32_t (&v)[32])
{
    const uint32_t rl = ((e >> 24) - q32) & 31u; // the entry's row = lane within the quadrant
    const uint32_t rowmask = __reduce_or_sync(0xffffffffu, inj ? (1u << rl) : 0u);
    const uint32_t nrows = __popc(rowmask);
    const bool mine = (rowmask >> lane) & 1u;
    const uint32_t myrank = __popc(rowmask & ((1u << lane) - 1u));
    const uint32_t erank = __popc(rowmask & ((1u << rl) - 1u));
    uint8_t *const my_slot0 = scr + 2 * ((e >> 16) & 63u);
    for (uint32_t r0 = 0; r0 < nrows; r0 += PARK) {
        const bool park = mine && myrank - r0 < static_cast<uint32_t>(PARK);
        uint8_t *row_s = scr + (myrank - r0) * kParkPitch;
        if (park) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<uint4 *>(row_s + 16 * i) =
                    make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        __syncwarp();
        if (inj && erank - r0 < static_cast<uint32_t>(PARK))
            *reinterpret_cast<uint16_t *>(my_slot0 + (erank - r0) * kParkPitch) = static_cast<uint16_t>(e & 0xFFFFu);
        __syncwarp();
        if (park) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 w = *reinterpret_cast<const uint4 *>(row_s + 16 * i);
                v[4 * i] = w.x;
                v[4 * i + 1] = w.y;
                v[4 * i + 2] = w.z;
                v[4 * i + 3] = w.w;
            }
        }
        __syncwarp();
    }
}

// This thread's raw planes of a unit from its weight stage: AE in sixteen
// 16-byte chunks per row, split into two swizzled 128-column halves, B in
// eight (chunk j of row r sits at j ^ (r & 7)); the thread takes the NA AE
// and NB B chunks of its column half hh.
template <bool Q8, int NA, int NB>
__device__ __forceinline__ void load_raw(const uint8_t *st, int ae_half, int ae_bytes, int row, int hh,
                                         uint4 (&aq)[NA], uint4 (&bq)[NB])
{
#pragma unroll
    for (int i = 0; i < NA; ++i) {
        const int ci = hh * NA + i;
        aq[i] = *reinterpret_cast<const uint4 *>(st + (ci >> 3) * ae_half + row * 128 + (((ci & 7) ^ (row & 7)) << 4));
    }
#pragma unroll
    for (int i = 0; i < NB; ++i)
        bq[i] = Q8 ? make_uint4(0u, 0u, 0u, 0u)
                   : *reinterpret_cast<const uint4 *>(st + ae_bytes + row * 128 + (((hh * NB + i) ^ (row & 7)) << 4));
}

// A 64-column chunk j of a thread's raw planes (AE chunks 4j..4j+3, B chunks
// 2j, 2j+1) decoded to 32 BF16 pairs (escaped slots hold their placeholder).
template <bool Q8, bool I8, int NA, int NB>
__device__ __forceinline__ void decode_chunk(const uint4 (&aq)[NA], const uint4 (&bq)[NB], int j, uint32_t eb2,
                                             uint32_t bm1, uint32_t bm2, uint32_t bm3, uint32_t (&v)[32])
{
    const uint32_t bw[8] = {bq[2 * j].x, bq[2 * j].y, bq[2 * j].z, bq[2 * j].w,
                            bq[2 * j + 1].x, bq[2 * j + 1].y, bq[2 * j + 1].z, bq[2 * j + 1].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 w = aq[4 * j + i];
        uint32_t *o = v + 8 * i;
        if constexpr (I8) {
            decode_i8_group(w.x, w.y, o);
            decode_i8_group(w.z, w.w, o + 4);
        } else {
            o[0] = dec_pair<0, Q8>(w.x, bw[2 * i], eb2, 0u);
            o[1] = dec_pair<1, Q8>(w.x, bw[2 * i], eb2, bm1);
            o[2] = dec_pair<2, Q8>(w.y, bw[2 * i], eb2, bm2);
            o[3] = dec_pair<3, Q8>(w.y, bw[2 * i], eb2, bm3);
            o[4] = dec_pair<0, Q8>(w.z, bw[2 * i + 1], eb2, 0u);
            o[5] = dec_pair<1, Q8>(w.z, bw[2 * i + 1], eb2, bm1);
            o[6] = dec_pair<2, Q8>(w.w, bw[2 * i + 1], eb2, bm2);
            o[7] = dec_pair<3, Q8>(w.w, bw[2 * i + 1], eb2, bm3);
        }
    }
}

// Patch the escapes of 64-column chunk jc of the unit into v: the quadrant's
// entries qlo .. qlo + qn of list `esrc` (the first 32 already in e_first,
// one per lane).  (Gathering a chunk's entries across batches of 32 before a
// round was measured slower on GB300: 33.1 against 31.7 us at 16 rows, and no
// faster on a dense escape tail.)
template <int PARK, int R>
__device__ __forceinline__ void patch_entries(uint32_t qlo, uint32_t qn, uint32_t e_first, const uint32_t *esrc,
                                              int jc, uint32_t q32, uint8_t *scr, int lane, uint32_t (&v)[32])
{
    if constexpr (PARK >= 32) {
        if (qn <= 32u) { // one batch: the common case
            const uint32_t e[1] = {e_first};
            const bool inj[1] = {static_cast<uint32_t>(lane) < qn && ((e_first >> 22) & 3u) == static_cast<uint32_t>(jc)};
            if (__any_sync(0xffffffffu, inj[0]))
                patch_rows<1>(e, inj, q32, scr, lane, v);
            return;
        }
        for (uint32_t i0 = 0; i0 < qn; i0 += 32 * R) {
            uint32_t e[R];
            bool inj[R], any = false;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t idx = i0 + 32 * r + static_cast<uint32_t>(lane);
                e[r] = (r == 0 && i0 == 0) ? e_first : (idx < qn ? esrc[qlo + idx] : 0u);
                inj[r] = idx < qn && ((e[r] >> 22) & 3u) == static_cast<uint32_t>(jc);
                any = any || inj[r];
            }
            if (__any_sync(0xffffffffu, any))
                patch_rows<R>(e, inj, q32, scr, lane, v);
        }
    } else {
        for (uint32_t i0 = 0; i0 < qn; i0 += 32) {
            const uint32_t idx = i0 + static_cast<uint32_t>(lane);
            uint32_t e = e_first;
            if (i0 != 0)
                e = idx < qn ? esrc[qlo + idx] : 0u;
            const bool inj = idx < qn && ((e >> 22) & 3u) == static_cast<uint32_t>(jc);
            if (__any_sync(0xffffffffu, inj))
                patch_chunk<PARK>(e, inj, q32, scr, lane, v);
        }
    }
}

// EPI: the output goes through the output mode (BF16, SiLU*mul); the default
// FP32 store is a kernel of its own.  I8 (with Q8's layout: one weight plane,
// no escapes): the plane holds an INT8 copy, converted to BF16 exactly, and
// the row scales apply at the end.
template <int MT, bool Q8, bool EPI, bool I8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const GemmArgs a, const __grid_constant__ TmapSet tm)
{
    using L = TcSmem<MT, Q8>;
    constexpr int WST = L::WST, XST = L::XST, kNA = L::NA, ND = L::ND;
    constexpr uint32_t kDCol = L::DCOL;
    constexpr uint32_t IDESC = idesc_bf16_f32(128, MT);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA tiles need 1024-byte aligned shared addresses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    const uint32_t w_full0 = smem_u32(bars);                   // [WST][kGroups]
    const uint32_t w_empty0 = w_full0 + 8 * kGroups * WST;      // [WST]
    const uint32_t pl_full0 = w_empty0 + 8 * WST;               // [kPlSt]
    const uint32_t pl_empty0 = pl_full0 + 8 * kPlSt;            // [kPlSt]
    const uint32_t x_full0 = pl_empty0 + 8 * kPlSt;             // [XST]
    const uint32_t x_empty0 = x_full0 + 8 * XST;                // [XST]
    const uint32_t a_full0 = x_empty0 + 8 * XST;                // [NA]
    const uint32_t a_empty0 = a_full0 + 8 * kNA;                // [NA][kGroups]
    const uint32_t acc_full0 = a_empty0 + 8 * kGroups * kNA;    // [2][kGroups]
    const uint32_t acc_empty0 = acc_full0 + 16 * kGroups;       // [2]
    const uint32_t final_bar = acc_empty0 + 16;
    const uint32_t stall_bar = final_bar + 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + L::NBARS);
    volatile int *seg_last = abort_flag + 1; // [kGroups], one per group
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(abort_flag + 1 + kGroups);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int it0 = sk_begin(cta, grid, a.total_iters);
    const int n_it = sk_begin(cta + 1, grid, a.total_iters) - it0;
    const int nk = a.n_kstep;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WST; ++s) {
            for (int g = 0; g < kGroups; ++g)
                mbar_init(w_full0 + 8 * (kGroups * s + g), 1);
            mbar_init(w_empty0 + 8 * s, kGroupWarps);
        }
        for (int s = 0; s < kPlSt; ++s) {
            mbar_init(pl_full0 + 8 * s, 33); // 32 lanes' copies + the header
            mbar_init(pl_empty0 + 8 * s, kGroupThreads);
        }
        for (int s = 0; s < XST; ++s) {
            mbar_init(x_full0 + 8 * s, 1);
            mbar_init(x_empty0 + 8 * s, 1);
        }
        for (int b = 0; b < kNA; ++b) {
            mbar_init(a_full0 + 8 * b, kGroupWarps);
            for (int g = 0; g < kGroups; ++g)
                mbar_init(a_empty0 + 8 * (kGroups * b + g), 1);
        }
        for (int d = 0; d < 2; ++d) {
            for (int g = 0; g < kGroups; ++g)
                mbar_init(acc_full0 + 8 * (kGroups * d + g), 1);
            mbar_init(acc_empty0 + 8 * d, kGroupWarps);
        }
        mbar_init(final_bar, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        for (int g = 0; g < kGroups; ++g)
            seg_last[g] = 0;
        fence_barrier_init();
    }
    // escape-list bounds of the stager's first 64 units, loaded while the CTA
    // sets up
    uint32_t c_lo = 0, c_cnt = 0, c_g12 = 0, c_g3 = 0, n_lo = 0, n_cnt = 0, n_g12 = 0, n_g3 = 0;
    if (!Q8 && warp == kWarpE) {
        esc_window(a, it0, n_it, 0, lane, c_lo, c_cnt, c_g12, c_g3);
        esc_window(a, it0, n_it, 32, lane, n_lo, n_cnt, n_g12, n_g3);
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

    if (warp >= kDecodeWarps) {
    // the helper warpgroup hands registers to the decode warpgroups
    if constexpr (kRegHelper != kRegLaunch)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegHelper));
    if (warp == kWarpW) {
        // --------------------------- weight producer ---------------------------
        if (lane < a.n_mat) {
            prefetch_tmap(&tm.ae[lane]);
            if (!Q8)
                prefetch_tmap(&tm.b[lane]);
        }
        int issued = 0;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % WST;
            const uint32_t ph = static_cast<uint32_t>(it / WST) & 1u;
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(w_empty0 + 8 * s, ph ^ 1, a, abort_flag));
            if (!ok)
                break;
            const int u = it0 + it;
            const int rb = u / nk, g = mat_of(a, rb);
            const int row0 = (rb - a.mat[g].rb0) * 128, k0 = (u % nk) * 256; // rows of matrix g
            uint8_t *st = smem + L::OFF_W + s * L::WSTAGE;
            const uint32_t fb = w_full0 + 8 * (kGroups * s + it % kGroups);
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, L::W_TX + (I8 ? 0 : L::EB));
                tma_load_2d(smem_u32(st), &tm.ae[g], k0, row0, fb);
                tma_load_2d(smem_u32(st + L::AE_HALF), &tm.ae[g], k0 + 128, row0, fb);
                if (!Q8)
                    tma_load_2d(smem_u32(st + L::AE), &tm.b[g], k0 / 2, row0, fb);
                if (!I8)
                    bulk_load_1d(smem_u32(smem + L::OFF_EB + s * L::EB), a.mat[g].ebase + row0, L::EB, fb);
            }
            issued = it + 1;
        }
        // drain: every copy this warp started must land before the CTA exits
        for (int it = issued - 1; it >= 0 && it >= issued - WST; --it)
            mbar_wait(w_full0 + 8 * (kGroups * (it % WST) + it % kGroups), stage_use<WST>(it) & 1u, 1000000000ull);
    } else if (warp == kWarpX) {
        // ------------------------- activation producer -------------------------
        if (lane == 0) {
            prefetch_tmap(&tm.x);
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
                        tma_load_2d(smem_u32(xs + j * L::XSUB), &tm.x, k0 + 64 * (h * L::SPS + j), 0, fb);
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
        // The whole warp runs the loop, so that its descriptors and addresses
        // are warp-uniform values; one elected lane issues the MMAs and the
        // commits.
        const uint32_t leader = elect_one();
        // shared-memory descriptor of the first activation slot; slot sx adds
        // sx * XSLOT / 16, and within a slot the K-steps of 16 columns add a
        // fixed offset (address field in 16-byte units: +2 per 16 columns,
        // +XSUB/16 per 64-column sub-tile)
        const uint64_t xdesc0 = smem_desc_sw128(smem_u32(smem + L::OFF_X), 1024);
        int seg = 0;
        int ks = it0 % nk, sx = 0, b = 0;
        uint32_t phx = 0, pha = 0;
        for (int it = 0; it < n_it; ++it) {
            const bool seg_start = (it == 0) || (ks == 0);
            const bool seg_end = (ks == nk - 1) || (it == n_it - 1);
            const int db = seg % ND;
            bool ok = true;
            // accumulator buffer db was last read by the epilogue of segment seg - ND
            if (seg_start && seg >= ND)
                ok = wait_or_abort(acc_empty0 + 8 * db, ((seg / ND) - 1) & 1, a, abort_flag);
            ok = wait_or_abort(a_full0 + 8 * b, pha, a, abort_flag) && ok;
            const uint32_t d = tmem + kDCol + L::DW * db;
            const uint32_t a0 = tmem + b * 128;
#pragma unroll
            for (int h = 0; h < L::SPU; ++h) {
                const bool okx = __all_sync(0xffffffffu, wait_or_abort(x_full0 + 8 * sx, phx, a, abort_flag)) && ok;
                tc_fence_after();
                if (okx) {
                    const uint64_t bdesc = xdesc0 + static_cast<uint64_t>(sx * (L::XSLOT >> 4));
#pragma unroll
                    for (int jj = 0; jj < 4 * L::SPS; ++jj) {
                        const int j = h * 4 * L::SPS + jj; // K-step of 16 columns in the unit
                        const uint64_t bj = bdesc + static_cast<uint64_t>((jj >> 2) * (L::XSUB >> 4) + (jj & 3) * 2);
                        tc_mma_ts_lead(leader, d, a0 + j * 8, bj, IDESC, (j == 0 && seg_start) ? 0u : 1u);
                    }
                }
                // each commit arrives once every MMA issued so far has completed
                tc_commit_lead(leader, x_empty0 + 8 * sx);
                if (++sx == XST) {
                    sx = 0;
                    phx ^= 1;
                }
            }
            // the buffer's next user is unit it + NA, of group (it + NA) % kGroups
            tc_commit_lead(leader, a_empty0 + 8 * (kGroups * b + (it + kNA) % kGroups));
            if (seg_end) {
                // the epilogue belongs to the group that decoded this unit
                tc_commit_lead(leader, acc_full0 + 8 * (kGroups * db + it % kGroups));
                ++seg;
            }
            if (++ks == nk)
                ks = 0;
            if (++b == kNA) {
                b = 0;
                pha ^= 1;
            }
        }
        tc_commit_lead(leader, final_bar);
        mbar_wait(final_bar, 0, 1000000000ull);
        __syncwarp();
    } else if (warp == kWarpE) {
        // ---------------------------- escape lists ----------------------------
        // Per unit: the tile's entries (up to kEscCap) copied with cp.async,
        // and a header with the first entry, the count and the four quadrant
        // bounds.  Runs as far ahead of the decode groups as the ring allows.
        if (!Q8) {
            for (int it = 0; it < n_it; ++it) {
                if (it > 0 && (it & 31) == 0) { // next window of bounds; prefetch the one after
                    c_lo = n_lo;
                    c_cnt = n_cnt;
                    c_g12 = n_g12;
                    c_g3 = n_g3;
                    esc_window(a, it0, n_it, it + 32, lane, n_lo, n_cnt, n_g12, n_g3);
                }
                const int l = it & 31;
                const uint32_t lo = __shfl_sync(0xffffffffu, c_lo, l);
                const uint32_t cnt = __shfl_sync(0xffffffffu, c_cnt, l);
                const uint32_t g12 = __shfl_sync(0xffffffffu, c_g12, l);
                const uint32_t g3 = __shfl_sync(0xffffffffu, c_g3, l);
                const int s = it % kPlSt;
                const uint32_t ph = static_cast<uint32_t>(it / kPlSt) & 1u;
                const bool ok = __all_sync(0xffffffffu, wait_or_abort(pl_empty0 + 8 * s, ph ^ 1, a, abort_flag));
                uint8_t *pl = smem + L::OFF_PL + s * L::PL;
                const uint32_t fb = pl_full0 + 8 * s;
                const uint32_t ncp = ok ? min(cnt, static_cast<uint32_t>(kEscCap)) : 0u;
                const uint32_t *esc = a.mat[g3 >> 24].esc;
                for (uint32_t j = lane; j < ncp; j += 32)
                    cp_async_4(smem_u32(pl + L::PL_HDR + 4 * j), esc + lo + j);
                cp_async_arrive_noinc(fb);
                if (lane == 0) {
                    uint32_t *h = reinterpret_cast<uint32_t *>(pl);
                    h[0] = lo;
                    h[1] = cnt;
                    const uint32_t b1 = min(g12 & 0xFFFFu, cnt);
                    const uint32_t b2 = max(b1, min(g12 >> 16, cnt));
                    const uint32_t b3 = max(b2, min(g3 & 0xFFFFu, cnt));
                    h[2] = 0u;
                    h[3] = b1;
                    h[4] = b2;
                    h[5] = b3;
                    h[6] = cnt;
                    h[7] = g3 >> 24; // the unit's matrix
                    mbar_arrive(fb);
                }
            }
            cp_async_wait_all();
        }
    }
    } else {
        // ---------------------------- decode groups ----------------------------
        if constexpr (kRegDecode != kRegLaunch)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegDecode));
        const int grp = warp / kGroupWarps, q = warp & 3, hh = (warp / 4) % kSplit;
        const int gw = warp % kGroupWarps; // warp within the group
        const int row = 32 * q + lane; // this thread's row in the unit = TMEM lane
        const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t q32 = static_cast<uint32_t>(32 * q);
        uint8_t *const scr = smem + L::OFF_SCR + warp * park_rows<MT>() * kParkPitch;
        const uint32_t bm1 = a.bshift_mul[0], bm2 = a.bshift_mul[1], bm3 = a.bshift_mul[2];
        uint32_t acc_use0 = 0u, acc_use1 = 0u; // this group's epilogues per accumulator buffer
        constexpr int NA16 = kCols / 16, NB16 = kCols / 32; // 16-byte chunks of this thread's AE / B bytes

        uint4 aq[NA16], bq[NB16];         // raw planes of the current unit
        uint32_t eb2 = 0u;                // its window base, << 7 in both 16-bit lanes
        bool rok = true;                  // its stage wait succeeded
        uint32_t qlo = 0, qn = 0, e_first = 0; // its escapes (this quadrant)
        const uint32_t *esrc = nullptr;
        int sp = 0;                       // its escape-list stage
        // wait for unit it's stage; false after an abort (the loop then keeps
        // its shape -- every warp still meets every barrier -- but works on
        // stale data and reads nothing through addresses taken from shared
        // memory)
#define W12_WAIT_STAGE(it_, ok_)                                                                              \
    do {                                                                                                      \
        bool w_ = wait_or_abort(w_full0 + 8 * (kGroups * ((it_) % WST) + grp), stage_use<WST>(it_) & 1u, a,   \
                                abort_flag);                                                                  \
        if (a.inject_stall)                                                                                   \
            w_ = wait_or_abort(stall_bar, 0, a, abort_flag) && w_;                                            \
        ok_ = __all_sync(0xffffffffu, w_);                                                                    \
    } while (0)
#define W12_WINDOW_BASE(it_, eb2_)                                                                            \
    do {                                                                                                      \
        uint32_t e8_ = 1u;                                                                                    \
        if (!I8)                                                                                              \
            e8_ = smem[L::OFF_EB + ((it_) % WST) * L::EB + row];                                             \
        eb2_ = (e8_ << 7) | (e8_ << 23);                                                                      \
    } while (0)
        // this quadrant's escapes of unit it: a contiguous run of the unit's
        // list, the first 32 entries into e_first (one per lane)
#define W12_FETCH_HDR(it_, ok_, qlo_, qn_, e_first_, esrc_, sp_)                                             \
    do {                                                                                                      \
        qlo_ = qn_ = e_first_ = 0u;                                                                           \
        esrc_ = nullptr;                                                                                      \
        sp_ = (it_) % kPlSt;                                                                                  \
        if (!Q8) {                                                                                            \
            bool p_ = wait_or_abort(pl_full0 + 8 * sp_, ((it_) / kPlSt) & 1, a, abort_flag);                 \
            p_ = __all_sync(0xffffffffu, p_) && (ok_);                                                        \
            const uint32_t *hp_ = reinterpret_cast<const uint32_t *>(smem + L::OFF_PL + sp_ * L::PL);        \
            if (p_) {                                                                                         \
                /* a header read after an abort may mix two units: every read */                              \
                /* of the matrix's list stays below its entry count */                                        \
                const MatArgs &hm_ = a.mat[hp_[7] % kMaxGroup];                                                 \
                const uint32_t lo_ = min(hp_[0], hm_.n_esc), cnt_ = min(hp_[1], hm_.n_esc - lo_);             \
                qlo_ = min(hp_[2 + q], cnt_);                                                                 \
                const uint32_t qhi_ = min(hp_[3 + q], cnt_);                                                  \
                qn_ = qhi_ > qlo_ ? qhi_ - qlo_ : 0u;                                                         \
                esrc_ = cnt_ > static_cast<uint32_t>(kEscCap) ? hm_.esc + lo_                                \
                                                               : hp_ + L::PL_HDR / 4;                         \
                if (static_cast<uint32_t>(lane) < qn_)                                                        \
                    e_first_ = esrc_[qlo_ + lane];                                                            \
            }                                                                                                 \
        }                                                                                                     \
    } while (0)

        for (int it = grp; it < n_it; it += kGroups) {
            const int u = it0 + it;
            const int rb = u / nk, ks = u % nk;
            const int b = it % kNA;
            // this quadrant's escape header, then this row's raw planes and
            // window base
            W12_WAIT_STAGE(it, rok);
            W12_FETCH_HDR(it, rok, qlo, qn, e_first, esrc, sp);
            load_raw<Q8>(smem + L::OFF_W + (it % WST) * L::WSTAGE, L::AE_HALF, L::AE, row, hh, aq, bq);
            W12_WINDOW_BASE(it, eb2);
            // this warp's loads of the stages are done (they had the wait to
            // land): hand them back; the escape list too unless the run is
            // longer than a warp (its later entries are read as the chunks
            // need them)
            __syncwarp();
            if (lane == 0)
                mbar_arrive(w_empty0 + 8 * (it % WST));
            if (!Q8 && qn <= 32u)
                mbar_arrive(pl_empty0 + 8 * sp); // every lane, after its own reads
#pragma unroll
            for (int j = 0; j < kChunks; ++j) {
                uint32_t v[32];
                decode_chunk<Q8, I8>(aq, bq, j, eb2, bm1, bm2, bm3, v);
                if (!Q8)
                    patch_entries<park_rows<MT>(), MT == 16 ? W12_TC_PATCH_BATCHES16 : W12_TC_PATCH_BATCHES>(qlo, qn, e_first, esrc, hh * kChunks + j, q32, scr, lane, v);
                if (j == 0) {
                    // before the first store the MMA must be done with this A
                    // buffer (unit it - NA: the completions on this group's
                    // copy of the barrier are units it - NA, it - NA - P, ...
                    // for P = lcm(NA, kGroups)); the first chunk's decode
                    // overlaps the wait
                    if (it >= kNA) {
                        constexpr int P = kNA / gcd_c(kNA, kGroups) * kGroups;
                        wait_or_abort(a_empty0 + 8 * (kGroups * b + grp), static_cast<uint32_t>((it - kNA) / P) & 1u,
                                      a, abort_flag);
                    }
                    __syncwarp();
                    tc_fence_after();
                }
                tmem_st32(tmem + static_cast<uint32_t>(b * 128 + 32 * (hh * kChunks + j)) + t_lane, v);
            }
            if (!Q8 && qn > 32u)
                mbar_arrive(pl_empty0 + 8 * sp);
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
                const int seg = rb - it0 / nk;
                const int db = seg % ND;
                const uint32_t use = db ? acc_use1++ : acc_use0++;
                wait_or_abort(acc_full0 + 8 * (kGroups * db + grp), use & 1u, a, abort_flag);
                __syncwarp();
                tc_fence_after();
                const MatArgs &mm = a.mat[mat_of(a, rb)];
                const int row0 = (rb - mm.rb0) * 128; // rows of its matrix
                const int c_first = sk_owner(rb * nk, grid, a.total_iters);
                const int c_last = sk_owner((rb + 1) * nk - 1, grid, a.total_iters);
                const bool direct = (c_first == c_last);
                const int slot = direct ? 0 : sk_slot(cta, rb, grid, a.total_iters, nk);
                const int n = row0 + row;
                float rs = 1.f; // an INT8 copy's row scale
                if constexpr (I8)
                    rs = n < mm.N ? __ldg(mm.scale + n) : 0.f;
                const uint32_t dcol = tmem + t_lane + kDCol + L::DW * db;
                const bool pair = EPI && direct && (a.out_mode & kOutSiluMul);
                // this warp's share of the MT accumulator columns: half hh
                constexpr int PART = MT / kSplit;
                constexpr int CH = PART < 16 ? PART : 16;
#pragma unroll 1
                for (int h = 0; h < PART / CH; ++h) {
                    const int m0 = hh * PART + CH * h;
                    if (m0 >= a.M)
                        break;
                    uint32_t d[CH];
                    if constexpr (CH == 8)
                        tmem_ld8(dcol + m0, d);
                    else
                        tmem_ld16(dcol + m0, d);
                    tc_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < CH; ++jj) {
                        const float v = I8 ? __uint_as_float(d[jj]) * rs : __uint_as_float(d[jj]);
                        const int m = m0 + jj;
                        // row + 1 (the up row of an even gate row) is lane + 1
                        const float next = pair ? __shfl_down_sync(0xffffffffu, v, 1) : 0.f;
                        if (m < a.M) {
                            if (direct) {
                                if (n < mm.N) {
                                    if constexpr (EPI)
                                        emit_y(a, mm, m, n, v, next);
                                    else
                                        static_cast<float *>(mm.y)[static_cast<size_t>(m) * mm.N + n] = v;
                                }
                            } else {
                                a.partials[(static_cast<size_t>(slot) * a.M + m) * 128 + row] = v;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acc_empty0 + 8 * db);

                if (!direct && !a.defer) {
                    // the group barrier orders every thread's partial stores
                    // before one thread's release-acquire arrival (cumulativity),
                    // and that arrival before everyone's reads of the others
                    named_bar_sync(1 + grp, kGroupThreads);
                    if (gw == 0 && lane == 0)
                        seg_last[grp] = sk_arrive(a.counters + rb, c_last - c_first + 1) ? 1 : 0;
                    named_bar_sync(1 + grp, kGroupThreads);
                    if (seg_last[grp])
                        sk_reduce_wide<EPI, 4>(a, rb, 128, grid, c_first, c_last, 32 * gw + lane, kGroupThreads);
                }
            }
        }
#undef W12_WAIT_STAGE
#undef W12_WINDOW_BASE
#undef W12_FETCH_HDR
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpM) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MT, bool Q8, bool EPI, bool I8 = false>
cudaError_t launch_one(const GemmArgs &a, const TmapSet &tm, int grid, cudaStream_t st)
{
    using L = TcSmem<MT, Q8>;
    auto kern = gemm_tc_kernel<MT, Q8, EPI, I8>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess)
            return e;
        // the decode warpgroups raise their register count only as far as the
        // helper warpgroup's release and the launch allocation allow; a
        // shortfall would leave them waiting, so it is refused here
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs * kThreads < kRegDecode * kDecodeWarps * 32 + kRegHelper * 128)
            return cudaErrorInvalidConfiguration;
        attr_done = true;
    }
    GemmArgs b = a;
    b.bshift_mul[0] = 1u << 28;
    b.bshift_mul[1] = 1u << 24;
    b.bshift_mul[2] = 1u << 20;
    return launch_pdl(kern, grid, kThreads, L::TOTAL, st, b, tm);
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
cudaError_t launch_mt(bool q8, bool i8, const GemmArgs &a, const TmapSet &tm, int grid, cudaStream_t st)
{
    if (i8)
        return a.out_mode ? launch_one<MT, true, true, true>(a, tm, grid, st)
                          : launch_one<MT, true, false, true>(a, tm, grid, st);
    if (a.out_mode)
        return q8 ? launch_one<MT, true, true>(a, tm, grid, st) : launch_one<MT, false, true>(a, tm, grid, st);
    return q8 ? launch_one<MT, true, false>(a, tm, grid, st) : launch_one<MT, false, false>(a, tm, grid, st);
}

cudaError_t launch_gemm_tc(int mt, bool q8, bool i8, const GemmArgs &a, const TmapSet &tm, int grid,
                           cudaStream_t st)
{
    switch (mt) {
    case 16: return launch_mt<16>(q8, i8, a, tm, grid, st);
    case 32: return launch_mt<32>(q8, i8, a, tm, grid, st);
    case 64: return launch_mt<64>(q8, i8, a, tm, grid, st);
    case 128: return launch_mt<128>(q8, i8, a, tm, grid, st);
    case 256: return launch_mt<256>(q8, i8, a, tm, grid, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace w12
