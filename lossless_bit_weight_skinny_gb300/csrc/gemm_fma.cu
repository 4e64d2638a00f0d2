// gemm_fma.cu -- W12 skinny GEMM for M <= 8 activation rows on the CUDA cores.
//
// y[m][n] = sum_k x[m][k] * W[n][k], W decoded from its W12 planes to exact
// BF16 values (SpecPilot, Figure 5(a) caption) in registers and accumulated in
// FP32 with packed f32x2 FMAs.
//
// Work split: the matrix is cut into blocks of RBLK rows x 256 columns (one
// escape tile wide); the (row block, k step) iterations are split evenly over
// one persistent CTA per SM (stream-K), and row blocks shared by several CTAs
// are combined by the last contributor in a fixed order.
//
// CTA = 8 consumer warps + 1 producer warp.  The producer streams each
// block's AE bytes, B words and x slice with TMA into a ring of shared-memory
// stages, and copies the block's escape entries next to them with cp.async.
// Consumer warp w owns RW rows of the block; lane l owns columns 8l..8l+7 of
// the 256-column step and keeps the products of all its rows in registers
// until the row block ends, then the warp reduces across lanes.
#include "kernels.cuh"

namespace w12 {
namespace {

template <int MT>
struct FmaShape {
    static constexpr int RBLK = (MT <= 4) ? 128 : 64; // rows per block
    static constexpr int CW = 8;                      // consumer warps
    static constexpr int RW = RBLK / CW;              // rows per consumer warp
    static constexpr int THREADS = (CW + 1) * 32;
};

constexpr int r128(int v) { return (v + 127) & ~127; }
constexpr int r1024(int v) { return (v + 1023) & ~1023; }

template <int MT, bool Q8>
struct FmaSmem {
    using S = FmaShape<MT>;
    static constexpr int AE = S::RBLK * 256;
    static constexpr int B = Q8 ? 0 : S::RBLK * 128;
    static constexpr int X = MT * 256 * 2;
    static constexpr int ESC_CAP = 512;
    static constexpr int ESC = Q8 ? 0 : 16 + ESC_CAP * 4;
    static constexpr int OFF_AE = 0;
    static constexpr int OFF_B = r128(AE);
    static constexpr int OFF_X = OFF_B + r128(B);
    static constexpr int OFF_ESC = OFF_X + r128(X);
    static constexpr int STAGE = r1024(OFF_ESC + ESC);
    static constexpr int STAGES_RAW = (212 * 1024) / STAGE;
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr int TX_BYTES = AE + B + X;
    static constexpr int BARS = STAGES * STAGE;           // barrier area offset
    static constexpr int TOTAL = BARS + 8 * (2 * STAGES + 1) + 16 + 1024; // + slack to align the base
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

// Decode 8 weights (AE bytes k..k+7, their B word) to FP32 values.
// Per pair: PRMT spreads two AE bytes into two 16-bit lanes with the sign
// replicated into the high byte; then sign | (ebase + E) << 7 | A&7 << 4 | B.
template <bool Q8>
__device__ __forceinline__ void decode8(uint2 ae, uint32_t bw, uint32_t eb2, float (&wf)[8])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t src = (i < 2) ? ae.x : ae.y;
        uint32_t p;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(src), "r"(0u), "r"((i & 1) ? 0xB3A2u : 0x9180u));
        uint32_t r = (p & 0x80708070u) | ((p & 0x000F000Fu) * 128u + eb2);
        if (!Q8)
            r |= (bw >> (4 * i)) & 0x000F000Fu;
        wf[2 * i] = __uint_as_float(r << 16);
        wf[2 * i + 1] = __uint_as_float(r & 0xFFFF0000u);
    }
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

template <int MT, bool Q8>
__global__ void __launch_bounds__(FmaShape<MT>::THREADS, 1)
    gemm_fma_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tm_ae,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_x)
{
    using S = FmaShape<MT>;
    using L = FmaSmem<MT, Q8>;
    constexpr int RBLK = S::RBLK, CW = S::CW, RW = S::RW, STAGES = L::STAGES;
    constexpr int V = RW * MT;           // per-lane partial sums
    constexpr int VPL = V >= 32 ? V / 32 : 1;
    constexpr int LOGV = (V >= 64) ? 6 : (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : 2;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA tiles need 1024-byte aligned shared addresses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * STAGES + 1);
    volatile int *seg_last = abort_flag + 1;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t stall_bar = smem_u32(bars + 2 * STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int it0 = sk_begin(cta, grid, a.total_iters);
    const int n_it = sk_begin(cta + 1, grid, a.total_iters) - it0;
    const int nk = a.n_kstep;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, Q8 ? 1 : 33);
            mbar_init(empty0 + 8 * s, CW);
        }
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        *seg_last = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            prefetch_tmap(&tm_ae);
            prefetch_tmap(&tm_x);
            if (!Q8)
                prefetch_tmap(&tm_b);
        }
        int win = -1;
        uint32_t my_lo = 0, my_hi = 0;
        int issued = 0;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(empty0 + 8 * s, ph ^ 1, a, abort_flag));
            if (!ok)
                break;
            const int gi = it0 + it, rb = gi / nk, ks = gi % nk;
            const int row0 = rb * RBLK, k0 = ks * 256;
            uint8_t *st = smem + s * L::STAGE;
            const uint32_t fb = full0 + 8 * s;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, L::TX_BYTES);
                tma_load_2d(smem_u32(st + L::OFF_AE), &tm_ae, k0, row0, fb);
                if (!Q8)
                    tma_load_2d(smem_u32(st + L::OFF_B), &tm_b, k0 / 2, row0, fb);
                tma_load_2d(smem_u32(st + L::OFF_X), &tm_x, k0, 0, fb);
            }
            if (!Q8) {
                const int t = (row0 / 128) * a.tiles_c + ks;
                uint32_t *hdr = reinterpret_cast<uint32_t *>(st + L::OFF_ESC);
                if (lane < 2)
                    cp_async_4(smem_u32(hdr + lane), a.tile_ptr + t + lane);
                if (win < 0 || it - win >= 32) {
                    win = it;
                    const int gj = it0 + it + lane;
                    if (gj < it0 + n_it) {
                        const int tj = ((gj / nk) * RBLK / 128) * a.tiles_c + gj % nk;
                        my_lo = __ldg(a.tile_ptr + tj);
                        my_hi = __ldg(a.tile_ptr + tj + 1);
                    }
                }
                const uint32_t lo = __shfl_sync(0xffffffffu, my_lo, it - win);
                const uint32_t hi = __shfl_sync(0xffffffffu, my_hi, it - win);
                const uint32_t cnt = min(hi - lo, static_cast<uint32_t>(L::ESC_CAP));
                for (uint32_t idx = lane; idx < cnt; idx += 32)
                    cp_async_4(smem_u32(hdr + 4 + idx), a.esc + lo + idx);
                cp_async_arrive_noinc(fb);
            }
            issued = it + 1;
        }
        // drain: every copy this warp started must land before the CTA exits
        for (int it = issued - 1; it >= 0 && it >= issued - STAGES; --it) {
            const int s = it % STAGES;
            mbar_wait(full0 + 8 * s, (it / STAGES) & 1, 1000000000ull);
        }
    } else {
        // ------------------------------ consumers -----------------------------
        const int wrow = warp * RW;
        float acc[MT <= 2 ? 1 : RW][MT <= 2 ? 1 : MT];
        float2 acc2[MT <= 2 ? RW : 1][MT <= 2 ? MT : 1];
        uint32_t eb2[RW];
        int cur_rb = -1;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            bool ok = wait_or_abort(full0 + 8 * s, ph, a, abort_flag);
            if (a.inject_stall)
                ok = wait_or_abort(stall_bar, 0, a, abort_flag) && ok;
            // After an abort the loop keeps its shape (every warp still meets
            // every named barrier) but works on stale data and reads nothing
            // through addresses taken from shared memory.
            ok = __all_sync(0xffffffffu, ok);
            const int gi = it0 + it, rb = gi / nk, ks = gi % nk;
            const int row0 = rb * RBLK;
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
                const int n = row0 + wrow + lane;
                const uint32_t e = (lane < RW && n < a.N) ? __ldg(a.ebase + n) : 1u;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    const uint32_t er = __shfl_sync(0xffffffffu, e, r);
                    eb2[r] = (er << 7) | (er << 23);
                }
            }

            // this lane's x[m][8l .. 8l+7] as FP32 pairs
            float2 x2[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 v = *reinterpret_cast<const uint4 *>(st + L::OFF_X + m * 512 + lane * 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    x2[m][i] = make_float2(__uint_as_float(w4[i] << 16),
                                           __uint_as_float(w4[i] & 0xFFFF0000u));
            }

            // escapes of this warp's rows: [p, ub) in the tile's sorted list
            uint32_t mask = 0;
            uint32_t p = 0, ub = 0;
            const uint32_t *list = nullptr;
            const int base_row = (row0 & 127) + wrow;
            if (!Q8) {
                const uint32_t *hdr = reinterpret_cast<const uint32_t *>(st + L::OFF_ESC);
                const uint32_t lo = hdr[0], hi = hdr[1];
                const uint32_t cnt = ok ? hi - lo : 0u;
                list = (cnt <= static_cast<uint32_t>(L::ESC_CAP)) ? hdr + 4 : a.esc + lo;
                uint32_t n_in = 0;
                for (uint32_t j = 0; j < cnt; j += 32) {
                    const uint32_t idx = j + lane;
                    const uint32_t e = idx < cnt ? list[idx] : 0xFFFFFFFFu;
                    const int r7 = static_cast<int>(e >> 24);
                    const bool inr = idx < cnt && r7 >= base_row && r7 < base_row + RW;
                    p += __popc(__ballot_sync(0xffffffffu, idx < cnt && r7 < base_row));
                    n_in += __popc(__ballot_sync(0xffffffffu, inr));
                    mask |= __reduce_or_sync(0xffffffffu, inr ? (1u << (r7 - base_row)) : 0u);
                }
                ub = p + n_in;
            }

            const uint8_t *ae_p = st + L::OFF_AE + wrow * 256 + lane * 8;
            const uint8_t *b_p = st + L::OFF_B + wrow * 128 + lane * 4;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const uint2 aw = *reinterpret_cast<const uint2 *>(ae_p + r * 256);
                const uint32_t bw = Q8 ? 0u : *reinterpret_cast<const uint32_t *>(b_p + r * 128);
                float wf[8];
                decode8<Q8>(aw, bw, eb2[r], wf);
                if (!Q8 && ((mask >> r) & 1u)) {
                    const uint32_t rr = static_cast<uint32_t>(base_row + r);
                    while (p < ub) {
                        const uint32_t e = list[p];
                        if ((e >> 24) != rr)
                            break;
                        const uint32_t k8 = (e >> 16) & 0xFFu;
                        if ((k8 >> 3) == static_cast<uint32_t>(lane)) {
                            const float f = __uint_as_float((e & 0xFFFFu) << 16);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (static_cast<uint32_t>(j) == (k8 & 7u))
                                    wf[j] = f;
                        }
                        ++p;
                    }
                }
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
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * s);

            if (ks == nk - 1 || it == n_it - 1) {
                // ---- the row block ends here for this CTA: reduce and store ----
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
                const int c_first = sk_owner(rb * nk, grid, a.total_iters);
                const int c_last = sk_owner((rb + 1) * nk - 1, grid, a.total_iters);
                const bool writer = (V >= 32) || ((lane & ((32 >> LOGV) - 1)) == 0);
                const bool direct = (c_first == c_last);
                const int slot = direct ? 0 : sk_slot(cta, rb, grid, a.total_iters, nk);
#pragma unroll
                for (int q = 0; q < VPL; ++q) {
                    const int idx = (V >= 32) ? lane * VPL + q : (lane >> (5 - LOGV));
                    const int r = idx / MT, m = idx % MT;
                    const int n = row0 + wrow + r;
                    if (writer && m < a.M) {
                        if (direct) {
                            if (n < a.N)
                                a.y[static_cast<size_t>(m) * a.N + n] = v[q];
                        } else {
                            a.partials[(static_cast<size_t>(slot) * a.M + m) * RBLK + wrow + r] = v[q];
                        }
                    }
                }
                if (!direct) {
                    __threadfence();
                    named_bar_sync(1, CW * 32);
                    if (threadIdx.x == 0)
                        *seg_last = sk_arrive(a.counters + rb, a.epoch, c_last - c_first + 1) ? 1 : 0;
                    named_bar_sync(1, CW * 32);
                    if (*seg_last) {
                        __threadfence();
                        sk_reduce_block(a, rb, RBLK, grid, c_first, c_last, threadIdx.x, CW * 32);
                    }
                }
            }
        }
    }
    __syncthreads();
}

template <int MT, bool Q8>
cudaError_t launch_one(const GemmArgs &a, const CUtensorMap *tm_ae, const CUtensorMap *tm_b,
                       const CUtensorMap *tm_x, int grid, cudaStream_t st)
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
    kern<<<grid, FmaShape<MT>::THREADS, L::TOTAL, st>>>(a, *tm_ae, *tm_b, *tm_x);
    return cudaGetLastError();
}

} // namespace

int fma_rows_blk(int mt) { return mt <= 4 ? 128 : 64; }

int fma_smem_bytes(int mt, bool q8)
{
    switch (mt) {
    case 1: return q8 ? FmaSmem<1, true>::TOTAL : FmaSmem<1, false>::TOTAL;
    case 2: return q8 ? FmaSmem<2, true>::TOTAL : FmaSmem<2, false>::TOTAL;
    case 4: return q8 ? FmaSmem<4, true>::TOTAL : FmaSmem<4, false>::TOTAL;
    default: return q8 ? FmaSmem<8, true>::TOTAL : FmaSmem<8, false>::TOTAL;
    }
}

cudaError_t launch_gemm_fma(int mt, bool q8, const GemmArgs &a, const CUtensorMap *tm_ae,
                            const CUtensorMap *tm_b, const CUtensorMap *tm_x, int grid,
                            cudaStream_t st)
{
    switch (mt) {
    case 1: return q8 ? launch_one<1, true>(a, tm_ae, tm_b, tm_x, grid, st)
                      : launch_one<1, false>(a, tm_ae, tm_b, tm_x, grid, st);
    case 2: return q8 ? launch_one<2, true>(a, tm_ae, tm_b, tm_x, grid, st)
                      : launch_one<2, false>(a, tm_ae, tm_b, tm_x, grid, st);
    case 4: return q8 ? launch_one<4, true>(a, tm_ae, tm_b, tm_x, grid, st)
                      : launch_one<4, false>(a, tm_ae, tm_b, tm_x, grid, st);
    case 8: return q8 ? launch_one<8, true>(a, tm_ae, tm_b, tm_x, grid, st)
                      : launch_one<8, false>(a, tm_ae, tm_b, tm_x, grid, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace w12
