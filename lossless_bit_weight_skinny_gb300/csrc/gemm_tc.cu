// gemm_tc.cu -- W12 skinny GEMM for 9..64 activation rows on the tcgen05
// tensor cores.
//
// The product is computed transposed: D[n][m] = sum_k W[n][k] x[m][k], with the
// decoded weight tile as the MMA "A" operand (128 output channels x 16 k per
// instruction) and the activation tile as "B" (MT = 16, 32 or 64 rows, zero
// padded), FP32 accumulators in tensor memory.  This is the Blackwell form of
// decoding W12 records on the fly and feeding them to the tensor cores
// (SpecPilot, Figure 5(b) caption): instead of a register operand, the decode
// warps write the exact BF16 weights straight into tensor memory with
// tcgen05.st and the MMA reads A from there, so decoded weights never touch
// shared memory.
//
// CTA = 8 decode warps + 1 TMA producer warp + 1 MMA warp.  Work split and
// split-K fix-up are the stream-K scheme of the CUDA-core kernel, over blocks of
// 128 rows x 128 columns (half an escape tile).
#include "kernels.cuh"

namespace w12 {
namespace {

constexpr int kDecodeWarps = 8;
constexpr int kThreads = (kDecodeWarps + 2) * 32;
constexpr int kScrPitch = 144; // escape scratch row pitch (bytes): 64 BF16 + pad

constexpr int a128(int v) { return (v + 127) & ~127; }
constexpr int a1024(int v) { return (v + 1023) & ~1023; }

template <int MT, bool Q8>
struct TcSmem {
    static constexpr int AE = 128 * 128;        // SWIZZLE_128B
    static constexpr int B = Q8 ? 0 : 128 * 64; // SWIZZLE_64B
    static constexpr int XSUB = MT * 128;       // one 64-column sub-tile, SWIZZLE_128B
    static constexpr int X = 2 * XSUB;
    static constexpr int ESC_CAP = 512;
    static constexpr int ESC = Q8 ? 0 : 16 + 4 * ESC_CAP;
    static constexpr int OFF_AE = 0;
    static constexpr int OFF_B = AE;
    static constexpr int OFF_X = a1024(OFF_B + B);
    static constexpr int OFF_ESC = OFF_X + X;
    static constexpr int STAGE = a1024(OFF_ESC + ESC);
    static constexpr int SCR = Q8 ? 0 : kDecodeWarps * 32 * kScrPitch;
    static constexpr int ST_RAW = (212 * 1024 - SCR) / STAGE;
    static constexpr int STAGES = ST_RAW > 6 ? 6 : ST_RAW;
    static constexpr int OFF_SCR = STAGES * STAGE;
    static constexpr int BARS = a128(OFF_SCR + SCR);
    // full, aready, empty per stage; acc_full, acc_empty, final, stall
    static constexpr int NBARS = 3 * STAGES + 4;
    static constexpr int TOTAL = BARS + 8 * NBARS + 32 + 1024; // + slack to align the base
    static constexpr int TX_BYTES = AE + B + X;
    static constexpr uint32_t D_COL = STAGES * 64;
    static_assert(D_COL + MT <= 512, "tensor memory budget");
};

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

// Four BF16x2 words (k pairs 0..3 of a group of 8) from the group's two AE
// words and its B word.
template <bool Q8>
__device__ __forceinline__ void decode_group(uint32_t a_lo, uint32_t a_hi, uint32_t bw,
                                             uint32_t eb2, uint32_t *out)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t src = (i < 2) ? a_lo : a_hi;
        uint32_t p;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(src), "r"(0u), "r"((i & 1) ? 0xB3A2u : 0x9180u));
        uint32_t r = (p & 0x80708070u) | ((p & 0x000F000Fu) * 128u + eb2);
        if (!Q8)
            r |= (bw >> (4 * i)) & 0x000F000Fu;
        out[i] = r;
    }
}

template <int MT, bool Q8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tm_ae,
                   const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_x)
{
    using L = TcSmem<MT, Q8>;
    constexpr int STAGES = L::STAGES;
    constexpr uint32_t IDESC = idesc_bf16_f32(128, MT);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA tiles need 1024-byte aligned shared addresses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t aready0 = smem_u32(bars + STAGES);
    const uint32_t empty0 = smem_u32(bars + 2 * STAGES);
    const uint32_t acc_full = smem_u32(bars + 3 * STAGES);
    const uint32_t acc_empty = smem_u32(bars + 3 * STAGES + 1);
    const uint32_t final_bar = smem_u32(bars + 3 * STAGES + 2);
    const uint32_t stall_bar = smem_u32(bars + 3 * STAGES + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + L::NBARS);
    volatile int *seg_last = abort_flag + 1;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(abort_flag + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = gridDim.x, cta = blockIdx.x;
    const int it0 = sk_begin(cta, grid, a.total_iters);
    const int n_it = sk_begin(cta + 1, grid, a.total_iters) - it0;
    const int nk = a.n_kstep;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, Q8 ? 1 : 33);
            mbar_init(aready0 + 8 * s, kDecodeWarps);
            mbar_init(empty0 + 8 * s, kDecodeWarps + 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kDecodeWarps);
        mbar_init(final_bar, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        *seg_last = 0;
        fence_barrier_init();
    }
    if (warp == kDecodeWarps + 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kDecodeWarps) {
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
            const int row0 = rb * 128, k0 = ks * 128;
            uint8_t *st = smem + s * L::STAGE;
            const uint32_t fb = full0 + 8 * s;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, L::TX_BYTES);
                tma_load_2d(smem_u32(st + L::OFF_AE), &tm_ae, k0, row0, fb);
                if (!Q8)
                    tma_load_2d(smem_u32(st + L::OFF_B), &tm_b, k0 / 2, row0, fb);
                tma_load_2d(smem_u32(st + L::OFF_X), &tm_x, k0, 0, fb);
                tma_load_2d(smem_u32(st + L::OFF_X + L::XSUB), &tm_x, k0 + 64, 0, fb);
            }
            if (!Q8) {
                const int t = rb * a.tiles_c + (k0 >> 8);
                uint32_t *hdr = reinterpret_cast<uint32_t *>(st + L::OFF_ESC);
                if (lane < 2)
                    cp_async_4(smem_u32(hdr + lane), a.tile_ptr + t + lane);
                if (win < 0 || it - win >= 32) {
                    win = it;
                    const int gj = it0 + it + lane;
                    if (gj < it0 + n_it) {
                        const int tj = (gj / nk) * a.tiles_c + ((gj % nk) * 128 >> 8);
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
        for (int it = issued - 1; it >= 0 && it >= issued - STAGES; --it)
            mbar_wait(full0 + 8 * (it % STAGES), (it / STAGES) & 1, 1000000000ull);
    } else if (warp == kDecodeWarps + 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            int seg = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                const int gi = it0 + it, ks = gi % nk;
                const bool seg_start = (it == 0) || (ks == 0);
                const bool seg_end = (ks == nk - 1) || (it == n_it - 1);
                bool ok = true;
                if (seg_start && seg > 0)
                    ok = wait_or_abort(acc_empty, (seg - 1) & 1, a, abort_flag);
                ok = wait_or_abort(aready0 + 8 * s, ph, a, abort_flag) && ok;
                tc_fence_after();
                if (ok) {
                    const uint8_t *st = smem + s * L::STAGE;
                    const uint32_t xs = smem_u32(st + L::OFF_X);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t b_addr = xs + (j >> 2) * L::XSUB + (j & 3) * 32;
                        const uint64_t bdesc = smem_desc_sw128(b_addr, 1024);
                        tc_mma_ts(tmem + L::D_COL, tmem + s * 64 + j * 8, bdesc, IDESC,
                                  (j > 0 || !seg_start) ? 1u : 0u);
                    }
                }
                tc_commit(empty0 + 8 * s);
                if (seg_end) {
                    tc_commit(acc_full);
                    ++seg;
                }
            }
            tc_commit(final_bar);
            mbar_wait(final_bar, 0, 1000000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------ decode warps --------------------------
        const int q = warp & 3, h = warp >> 2;
        const int row = 32 * q + lane; // this thread's row in the block = TMEM lane
        const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
        uint32_t eb2 = 0;
        int cur_rb = -1, seg = 0;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            bool ok = wait_or_abort(full0 + 8 * s, ph, a, abort_flag);
            if (a.inject_stall)
                ok = wait_or_abort(stall_bar, 0, a, abort_flag) && ok;
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const int gi = it0 + it, rb = gi / nk, ks = gi % nk;
            const int row0 = rb * 128, k0 = ks * 128;
            const uint8_t *st = smem + s * L::STAGE;
            if (rb != cur_rb) {
                cur_rb = rb;
                const int n = row0 + row;
                const uint32_t e = (n < a.N) ? __ldg(a.ebase + n) : 1u;
                eb2 = (e << 7) | (e << 23);
            }

            // raw planes of this row, columns [64h, 64h + 64) of the step
            uint32_t v[32];
            {
                const uint8_t *ae_row = st + L::OFF_AE + row * 128;
                const uint8_t *b_row = st + L::OFF_B + row * 64;
                uint4 bq[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
                if (!Q8) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int c = (2 * h + i) ^ ((row >> 1) & 3);
                        bq[i] = *reinterpret_cast<const uint4 *>(b_row + c * 16);
                    }
                }
                const uint32_t bwords[8] = {bq[0].x, bq[0].y, bq[0].z, bq[0].w,
                                            bq[1].x, bq[1].y, bq[1].z, bq[1].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = (4 * h + i) ^ (row & 7);
                    const uint4 aq = *reinterpret_cast<const uint4 *>(ae_row + c * 16);
                    decode_group<Q8>(aq.x, aq.y, Q8 ? 0u : bwords[2 * i], eb2, v + 8 * i);
                    decode_group<Q8>(aq.z, aq.w, Q8 ? 0u : bwords[2 * i + 1], eb2, v + 8 * i + 4);
                }
            }

            if (!Q8) {
                // escapes inside this warp's 32 rows x 64 columns: patch through
                // a per-warp scratch tile in shared memory
                const uint32_t *hdr = reinterpret_cast<const uint32_t *>(st + L::OFF_ESC);
                const uint32_t lo = hdr[0], hi = hdr[1];
                const uint32_t cnt = ok ? hi - lo : 0u;
                const uint32_t *list = (cnt <= static_cast<uint32_t>(L::ESC_CAP)) ? hdr + 4 : a.esc + lo;
                const uint32_t kb = static_cast<uint32_t>((k0 & 255) + 64 * h);
                const uint32_t rlo = static_cast<uint32_t>(32 * q);
                bool any = false;
                for (uint32_t j = 0; j < cnt; j += 32) {
                    const uint32_t idx = j + lane;
                    const uint32_t e = idx < cnt ? list[idx] : 0xFFFFFFFFu;
                    const uint32_t r7 = e >> 24, k8 = (e >> 16) & 0xFFu;
                    const bool hit = idx < cnt && r7 - rlo < 32u && k8 - kb < 64u;
                    any |= __any_sync(0xffffffffu, hit);
                }
                if (any) {
                    uint8_t *scr = smem + L::OFF_SCR + warp * 32 * kScrPitch;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(scr + lane * kScrPitch + c * 16) =
                            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                    __syncwarp();
                    for (uint32_t j = 0; j < cnt; j += 32) {
                        const uint32_t idx = j + lane;
                        const uint32_t e = idx < cnt ? list[idx] : 0xFFFFFFFFu;
                        const uint32_t r7 = e >> 24, k8 = (e >> 16) & 0xFFu;
                        if (idx < cnt && r7 - rlo < 32u && k8 - kb < 64u)
                            *reinterpret_cast<uint16_t *>(scr + (r7 - rlo) * kScrPitch + (k8 - kb) * 2) =
                                static_cast<uint16_t>(e & 0xFFFFu);
                    }
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 w4 = *reinterpret_cast<const uint4 *>(scr + lane * kScrPitch + c * 16);
                        v[4 * c] = w4.x;
                        v[4 * c + 1] = w4.y;
                        v[4 * c + 2] = w4.z;
                        v[4 * c + 3] = w4.w;
                    }
                    __syncwarp();
                }
            }

            tmem_st32(tmem + t_lane + static_cast<uint32_t>(s * 64 + 32 * h), v);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(aready0 + 8 * s);
                mbar_arrive(empty0 + 8 * s);
            }

            if (ks == nk - 1 || it == n_it - 1) {
                // ---- accumulators of this row block are final: read them out ----
                wait_or_abort(acc_full, seg & 1, a, abort_flag);
                __syncwarp();
                tc_fence_after();
                constexpr int HALF = MT / 2;
                float out[HALF];
                const uint32_t dcol = tmem + t_lane + L::D_COL + h * HALF;
                if constexpr (HALF == 32) {
                    uint32_t d[32];
                    tmem_ld32(dcol, d);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        out[j] = __uint_as_float(d[j]);
                } else {
#pragma unroll
                    for (int c8 = 0; c8 < HALF / 8; ++c8) {
                        uint32_t d[8];
                        tmem_ld8(dcol + 8 * c8, d);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            out[8 * c8 + j] = __uint_as_float(d[j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acc_empty);
                ++seg;

                const int c_first = sk_owner(rb * nk, grid, a.total_iters);
                const int c_last = sk_owner((rb + 1) * nk - 1, grid, a.total_iters);
                const bool direct = (c_first == c_last);
                const int slot = direct ? 0 : sk_slot(cta, rb, grid, a.total_iters, nk);
                const int n = row0 + row;
#pragma unroll
                for (int j = 0; j < HALF; ++j) {
                    const int m = h * HALF + j;
                    if (m < a.M) {
                        if (direct) {
                            if (n < a.N)
                                a.y[static_cast<size_t>(m) * a.N + n] = out[j];
                        } else {
                            a.partials[(static_cast<size_t>(slot) * a.M + m) * 128 + row] = out[j];
                        }
                    }
                }
                if (!direct) {
                    named_bar_sync(1, kDecodeWarps * 32);
                    if (threadIdx.x == 0) {
                        __threadfence();
                        const bool last = sk_arrive(a.counters + rb, a.epoch, c_last - c_first + 1);
                        if (last)
                            __threadfence();
                        *seg_last = last ? 1 : 0;
                    }
                    named_bar_sync(1, kDecodeWarps * 32);
                    if (*seg_last)
                        sk_reduce_block(a, rb, 128, grid, c_first, c_last, threadIdx.x, kDecodeWarps * 32);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kDecodeWarps + 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MT, bool Q8>
cudaError_t launch_one(const GemmArgs &a, const CUtensorMap *tm_ae, const CUtensorMap *tm_b,
                       const CUtensorMap *tm_x, int grid, cudaStream_t st)
{
    using L = TcSmem<MT, Q8>;
    auto kern = gemm_tc_kernel<MT, Q8>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
    kern<<<grid, kThreads, L::TOTAL, st>>>(a, *tm_ae, *tm_b, *tm_x);
    return cudaGetLastError();
}

} // namespace

int tc_smem_bytes(int mt, bool q8)
{
    switch (mt) {
    case 16: return q8 ? TcSmem<16, true>::TOTAL : TcSmem<16, false>::TOTAL;
    case 32: return q8 ? TcSmem<32, true>::TOTAL : TcSmem<32, false>::TOTAL;
    default: return q8 ? TcSmem<64, true>::TOTAL : TcSmem<64, false>::TOTAL;
    }
}

cudaError_t launch_gemm_tc(int mt, bool q8, const GemmArgs &a, const CUtensorMap *tm_ae,
                           const CUtensorMap *tm_b, const CUtensorMap *tm_x, int grid,
                           cudaStream_t st)
{
    switch (mt) {
    case 16: return q8 ? launch_one<16, true>(a, tm_ae, tm_b, tm_x, grid, st)
                       : launch_one<16, false>(a, tm_ae, tm_b, tm_x, grid, st);
    case 32: return q8 ? launch_one<32, true>(a, tm_ae, tm_b, tm_x, grid, st)
                       : launch_one<32, false>(a, tm_ae, tm_b, tm_x, grid, st);
    case 64: return q8 ? launch_one<64, true>(a, tm_ae, tm_b, tm_x, grid, st)
                       : launch_one<64, false>(a, tm_ae, tm_b, tm_x, grid, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace w12
