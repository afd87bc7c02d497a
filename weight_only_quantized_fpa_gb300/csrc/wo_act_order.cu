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
#include <atomic>

#include "wo_bounds.cuh"
#include "wo_internal.h"

namespace wo {
namespace {

constexpr int kGatherThreads = 256;

// Activation loads after griddepcontrol.wait go through L2 only (.cg): A may
// have been written by the previous grid while this one was already
// resident, so no read of it may be served by a non-coherent or L1 copy.
__device__ __forceinline__ uint16_t ld_cg_u16(const uint16_t* p)
{
    uint16_t v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// A'[r, j] = A[r, perm[j]].
//
// Few rows (the weight-streaming sizes): a thread owns 8 consecutive output columns
// (one 16-byte store per row) and walks rows r = blockIdx.y, += gridDim.y,
// keeping its 8 indices in registers.  An index outside [0, k) reads 0.
// Launched with programmatic stream serialisation: the indices are read
// before the wait on the previous grid (they are load-time data), A after it.
__global__ void __launch_bounds__(kGatherThreads)
    act_order_gather_kernel(const uint16_t* A, const int32_t* __restrict__ perm,
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
            const uint32_t lo =
                in_bounds((unsigned)idx[2 * i] < (unsigned)k, 0x601) ? ld_cg_u16(a + idx[2 * i]) : 0u;
            const uint32_t hi =
                in_bounds((unsigned)idx[2 * i + 1] < (unsigned)k, 0x601) ? ld_cg_u16(a + idx[2 * i + 1]) : 0u;
            w[i] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(Ap + (size_t)r * k + 8 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Many rows (the tensor-core sizes): a CTA stages whole rows in shared
// memory with 16-byte loads and gathers from there, instead of scattered
// 2-byte loads from global memory (each a separate L1 line for a random
// permutation).  The permutation is kept in shared memory as 16-bit
// positions for all the CTA's rows; an index outside [0, k) points at a zero
// slot after the row.  Requires k <= kGatherSmemMaxK (< 65536).
constexpr int kGatherSmemThreads = 512;
constexpr int kGatherSmemMaxK = 49152;

__host__ __device__ constexpr size_t gather_smem_bytes(int k) { return (size_t)(2 * k + 8) * 2; }

__global__ void __launch_bounds__(kGatherSmemThreads)
    act_order_gather_smem_kernel(const uint16_t* A, const int32_t* __restrict__ perm,
                                 uint16_t* __restrict__ Ap, int m, int k)
{
    extern __shared__ __align__(16) uint16_t gsm[];
    uint16_t* pos = gsm;     // [k]: source column of each output column
    uint16_t* row = gsm + k; // [k + 8]: the staged row, then 8 zeros
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int j = tid; j < k; j += kGatherSmemThreads) {
        const int v = __ldg(perm + j);
        pos[j] = (uint16_t)(in_bounds((unsigned)v < (unsigned)k, 0x602) ? v : k);
    }
    if (tid < 8)
        row[k + tid] = 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nch = k >> 3;
    for (int r = blockIdx.x; r < m; r += gridDim.x) {
        __syncthreads();  // the previous row's gathers are done (first pass: pos is written)
        const uint4* src = reinterpret_cast<const uint4*>(A + (size_t)r * k);
        uint4* srow = reinterpret_cast<uint4*>(row);
        // four 16-byte loads in flight per thread, then their stores
        for (int c0 = tid; c0 < nch; c0 += 4 * kGatherSmemThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c0 + u * kGatherSmemThreads < nch)
                    v[u] = ld_cg_v4(src + c0 + u * kGatherSmemThreads);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c0 + u * kGatherSmemThreads < nch)
                    srow[c0 + u * kGatherSmemThreads] = v[u];
        }
        __syncthreads();
        uint4* dst = reinterpret_cast<uint4*>(Ap + (size_t)r * k);
#pragma unroll 1
        for (int c = tid; c < nch; c += kGatherSmemThreads) {
            const uint4 pi = reinterpret_cast<const uint4*>(pos)[c];
            auto pair = [&](uint32_t w) {
                return (uint32_t)row[w & 0xFFFFu] | ((uint32_t)row[w >> 16] << 16);
            };
            dst[c] = make_uint4(pair(pi.x), pair(pi.y), pair(pi.z), pair(pi.w));
        }
    }
}

}  // namespace

cudaError_t launch_gather_cols(const void* A, const int32_t* perm, void* Ap, int m, int k,
                               cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (m >= kTcMinM && k <= kGatherSmemMaxK) {
        const size_t smem = gather_smem_bytes(k);
        static std::atomic<int> smem_set[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 0 || dev >= 64 || smem_set[dev].load() < (int)smem) {
            if ((e = cudaFuncSetAttribute(act_order_gather_smem_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem)) != cudaSuccess)
                return e;
            if (dev >= 0 && dev < 64)
                smem_set[dev].store((int)smem);
        }
        int grid = num_sms() * 2;
        if (grid > m)
            grid = m;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kGatherSmemThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, act_order_gather_smem_kernel, static_cast<const uint16_t*>(A), perm,
                                  static_cast<uint16_t*>(Ap), m, k);
    }
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
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, act_order_gather_kernel, static_cast<const uint16_t*>(A), perm,
                              static_cast<uint16_t*>(Ap), m, k);
}

unsigned bounds_take_act_order() { return bounds_take_local(); }

}  // namespace wo
