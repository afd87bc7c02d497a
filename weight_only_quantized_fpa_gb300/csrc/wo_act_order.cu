// wo_act_order.cu -- the activation side of the GPTQ act-order GEMM.
//
// A GPTQ checkpoint quantised with act-order ("desc_act", the has_g_idx case
// that "[Misc][Kernel]: Add GPTQAllSpark Quantization" leaves out) gives each
// input channel c its own group number g_idx[c].  Sorting the channels by
// group (stable) makes every group a contiguous run of group_size channels,
// and a sum over k does not depend on the order of its terms, so
//     sum_c A[:, c] * w[:, c] = sum_j A[:, perm[j]] * w[:, perm[j]].
// The codes are sorted once at load time (pack_kernel with perm); per call
// the activations' columns are gathered into the same order here, and the
// ordinary group-wise kernels run on the sorted operands.
#include "wo_internal.h"

namespace wo {
namespace {

constexpr int kGatherThreads = 256;

// A'[r, j] = A[r, perm[j]].  A thread owns 8 consecutive output columns
// (one 16-byte store per row) and walks rows r = blockIdx.y, += gridDim.y,
// keeping its 8 indices in registers.  An index outside [0, k) reads 0.
// Launched with programmatic stream serialisation: the indices are read
// before the wait on the previous grid (they are load-time data), A after it.
__global__ void __launch_bounds__(kGatherThreads)
    gather_cols_kernel(const uint16_t* __restrict__ A, const int32_t* __restrict__ perm,
                       uint16_t* __restrict__ Ap, int m, int k)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int nch = k >> 3;
    const int ch = blockIdx.x * kGatherThreads + threadIdx.x;
    int idx[8];
    if (ch < nch) {
        const int4 p0 = __ldg(reinterpret_cast<const int4*>(perm) + 2 * ch);
        const int4 p1 = __ldg(reinterpret_cast<const int4*>(perm) + 2 * ch + 1);
        idx[0] = p0.x, idx[1] = p0.y, idx[2] = p0.z, idx[3] = p0.w;
        idx[4] = p1.x, idx[5] = p1.y, idx[6] = p1.z, idx[7] = p1.w;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ch >= nch)
        return;
    for (int r = blockIdx.y; r < m; r += gridDim.y) {
        const uint16_t* a = A + (size_t)r * k;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = (unsigned)idx[2 * i] < (unsigned)k ? __ldg(a + idx[2 * i]) : 0u;
            const uint32_t hi =
                (unsigned)idx[2 * i + 1] < (unsigned)k ? __ldg(a + idx[2 * i + 1]) : 0u;
            w[i] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(Ap + (size_t)r * k + 8 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

cudaError_t launch_gather_cols(const void* A, const int32_t* perm, void* Ap, int m, int k,
                               cudaStream_t s)
{
    const int nch = k / 8;
    const int gx = (nch + kGatherThreads - 1) / kGatherThreads;
    // enough CTAs for a few per SM; each walks the rest of the rows
    int gy = (num_sms() * 8 + gx - 1) / gx;
    if (gy > m)
        gy = m;
    if (gy > 65535)
        gy = 65535;
    if (gy < 1)
        gy = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(gx, gy);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gather_cols_kernel, static_cast<const uint16_t*>(A), perm,
                              static_cast<uint16_t*>(Ap), m, k);
}

}  // namespace wo
