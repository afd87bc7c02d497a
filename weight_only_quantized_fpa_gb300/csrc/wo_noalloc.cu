// wo_noalloc.cu -- wo_gemm_tc_noalloc: the tensor-core GEMM with its scratch
// memory in a file-scope device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory themselves, for
// instance a plugin that runs inside an engine owning all device memory
// through its own pool, or latency-critical code that must not call
// cudaMalloc (which can synchronise the whole device).  They pass inputs and
// outputs only.
//
// The scratch (error word; for 4-bit weights the per-channel pre-scaled
// scale and zero pairs and column scales, and with bf16 activations the
// fp16 copy of A and its row scales) lives in g_scratch below; every GPU
// that loads this library keeps it (24.06 MiB) until the process exits.  Host code cannot use g_scratch's
// name as a device address: each call looks the address up with
// cudaGetSymbolAddress in the caller's current context (a host-side table
// lookup), so a context other than the device's primary one, or a primary
// context recreated after cudaDeviceReset, gets its own copy's address.  The
// first call that meets a new (context, address) pair zeroes that copy's
// error word with a blocking cudaMemset, so it should come before any stream
// capture.
//
// All calls share the one array: two calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "wo_internal.h"

namespace wo {
namespace {

// Size of the built-in scratch: the 64.25 KiB header area every tensor-core
// call uses, plus 24 MiB for the per-call scratch of 4-bit weights: the
// pre-scaled scale and zero pairs (n * (k / group) * 4 bytes), the column
// scales (n * 2 bytes) and, with bf16 activations, the fp16 copy of A
// (m * k * 2 bytes) and its row scales (m * 4 bytes), each rounded up to
// 256 bytes.  8-bit weights need none of it.
constexpr size_t kNoAllocExtra = (size_t)24 << 20;
constexpr size_t kNoAllocBytes = kWsScratch + kNoAllocExtra;

static __device__ __align__(256) unsigned char g_scratch[kNoAllocBytes];

// The current context (driver entry point fetched through the runtime, so
// the library needs no link-time libcuda); null when it cannot be read.
CUcontext current_context()
{
    static const PFN_cuCtxGetCurrent_v4000 fn = []() -> PFN_cuCtxGetCurrent_v4000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        cudaGetLastError();
        return nullptr;
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS)
        return nullptr;
    return c;
}

struct Cleared {
    CUcontext ctx;
    void* addr;
};

std::mutex g_mu;
std::vector<Cleared> g_cleared;  // (context, address) pairs whose error word was zeroed

// Device address of g_scratch in the current context; zeroes its error word
// the first time a (context, address) pair is seen.
cudaError_t scratch_address(void** out)
{
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess)
        return e;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    bool seen = false;
    for (const Cleared& c : g_cleared)
        seen = seen || (c.ctx == ctx && c.addr == p);
    if (!seen) {
        e = cudaMemset(p, 0, kWsHeader);  // error word starts at zero
        if (e != cudaSuccess)
            return e;
        try {
            g_cleared.push_back(Cleared{ctx, p});
        } catch (...) {
            // no record: the next call zeroes the word again, harmless
        }
    }
    *out = p;
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

}  // namespace
}  // namespace wo

using namespace wo;

extern "C" wo_status wo_gemm_tc_noalloc(const void* A, const uint8_t* B_packed,
                                        const void* scales, const void* zeros, const void* bias,
                                        void* C, int m, int n, int k, int group_size, int bits,
                                        wo_dtype act_dtype, void* stream)
{
    if (m < 0 || n < 0 || k <= 0 || (bits != 4 && bits != 8) || n % 64 != 0 || k % 64 != 0)
        return WO_ERR_INVALID_ARG;
    if (act_dtype != WO_F16 && act_dtype != WO_BF16)
        return WO_ERR_INVALID_ARG;
    const int g = (group_size == -1 || group_size == k) ? k : group_size;
    if (g <= 0 || k % g != 0)
        return WO_ERR_INVALID_ARG;
    if ((bits == 8 && (g != k || zeros)) || (bits == 4 && g != k && g % 64 != 0))
        return WO_ERR_UNSUPPORTED;
    if (m == 0 || n == 0)
        return WO_OK;
    if (!A || !B_packed || !scales || !C || !aligned16(A) || !aligned16(B_packed) ||
        !aligned16(C) || !aligned2(scales) || (zeros && !aligned2(zeros)) ||
        (bias && !aligned2(bias)))
        return WO_ERR_INVALID_ARG;
    const TcPlan plan = plan_tc(m, n, k, g, bits, act_dtype, false);  // no k split: no partial tiles
    if (plan.ws_bytes > kNoAllocBytes)
        return WO_ERR_WORKSPACE;  // the problem needs more scratch than is built in
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return WO_ERR_CUDA;

    GemmArgs a{};
    a.A = A;
    a.B = B_packed;
    a.scales = scales;
    a.zeros = zeros;
    a.bias = bias;
    a.C = C;
    a.m = m;
    a.n = n;
    a.k = k;
    a.group = g;
    a.bits = bits;
    a.act = act_dtype;
    a.ws = scratch;
    a.ws_bytes = kNoAllocBytes;
    return launch_tc(a, plan, static_cast<cudaStream_t>(stream)) == cudaSuccess ? WO_OK
                                                                                : WO_ERR_CUDA;
}

extern "C" wo_status wo_noalloc_check(void* stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return WO_ERR_CUDA;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return WO_ERR_CUDA;
    unsigned flag = 0;
    if (cudaMemcpy(&flag, scratch, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess)
        return WO_ERR_CUDA;
    if (flag == 0)
        return WO_OK;
    if (cudaMemset(scratch, 0, sizeof flag) != cudaSuccess)
        return WO_ERR_CUDA;
    return WO_ERR_TIMEOUT;
}

extern "C" wo_status wo_noalloc_selftest_wait_timeout(unsigned limit_us, void* stream)
{
    if (limit_us < 1 || limit_us > 1000000)
        return WO_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return WO_ERR_CUDA;
    return launch_wait_timeout(static_cast<unsigned*>(scratch), limit_us,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? WO_OK
               : WO_ERR_CUDA;
}
