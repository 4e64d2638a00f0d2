// reduce.cu -- the split-K fix-up of a tensor-core GEMM as a kernel of its own.
//
// With many activation rows a row block's partial sums are large (M x 512
// bytes per contributor), and summing them inside the GEMM leaves one CTA per
// row block reading them with the few loads in flight its register budget
// allows.  Launched after the GEMM (programmatic dependent launch: it waits for
// the GEMM grid to complete before reading), this kernel spreads each split
// row block over several CTAs with deep load pipelining.  The contributors are
// summed in a fixed order (sk_reduce_range), so the results are bitwise
// reproducible; the output mode (BF16, SiLU*mul) applies here.
#include "kernels.cuh"

namespace w12 {
namespace {

constexpr int kRedThreads = 256;
constexpr int kRedGroupsPerCta = 512; // float4 groups of a row block per CTA

__global__ void __launch_bounds__(kRedThreads) sk_reduce_kernel(const GemmArgs a, int gemm_grid,
                                                                 int rows_blk, int slices)
{
    // the next kernel may start (its own writes wait for this one to
    // complete); the GEMM's partial sums are complete once the GEMM has
    pdl_launch_dependents();
    pdl_wait_prior_grid();
    const int rb = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int nk = a.n_kstep;
    const int c_first = sk_owner(rb * nk, gemm_grid, a.total_iters);
    const int c_last = sk_owner((rb + 1) * nk - 1, gemm_grid, a.total_iters);
    if (c_first == c_last)
        return; // stored directly by its only contributor
    const int groups = a.M * rows_blk / 4;
    const int g_lo = sl * kRedGroupsPerCta;
    const int g_hi = g_lo + kRedGroupsPerCta < groups ? g_lo + kRedGroupsPerCta : groups;
    if (g_lo >= g_hi)
        return;
    sk_reduce_range<true, 8>(a, rb, rows_blk, gemm_grid, c_first, c_last, threadIdx.x, kRedThreads, g_lo, g_hi);
}

} // namespace

cudaError_t launch_sk_reduce(const GemmArgs &a, int gemm_grid, int rows_blk, cudaStream_t st, bool *launched)
{
    *launched = false;
    int n_split = 0;
    for (int rb = 0; rb < a.n_rowblk; ++rb)
        if (sk_owner(rb * a.n_kstep, gemm_grid, a.total_iters) !=
            sk_owner((rb + 1) * a.n_kstep - 1, gemm_grid, a.total_iters))
            ++n_split;
    if (n_split == 0)
        return cudaSuccess;
    const int groups = a.M * rows_blk / 4;
    const int slices = (groups + kRedGroupsPerCta - 1) / kRedGroupsPerCta;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_rowblk * slices);
    cfg.blockDim = dim3(kRedThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sk_reduce_kernel, a, gemm_grid, rows_blk, slices);
    *launched = e == cudaSuccess;
    return e;
}

} // namespace w12
