// wo_api.cu -- the extern "C" entry points of libwo: argument checks, kernel
// choice and launch.  Every check runs before any CUDA call, so invalid
// arguments return a status with nothing enqueued.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "wo_internal.h"
#include "wo_stream.h"

namespace wo {

int num_sms()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            v <= 0) {
            cudaGetLastError();
            v = 152;
        }
        cached[dev] = v;
    }
    return cached[dev];
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Normalised group size: k for per-channel (-1 or k), else the value given.
int norm_group(int group_size, int k) { return (group_size == -1 || group_size == k) ? k : group_size; }

wo_status check_gemm_shape(int m, int n, int k, int group_size, int bits)
{
    if (m < 0 || n < 0 || k <= 0)
        return WO_ERR_INVALID_ARG;
    if ((long long)n > (long long)kWsCounters * 128)
        return WO_ERR_UNSUPPORTED;  // more output tiles than arrival counters
    if (bits != 4 && bits != 8)
        return WO_ERR_INVALID_ARG;
    if (n % 64 != 0 || k % 64 != 0)
        return WO_ERR_INVALID_ARG;
    const int g = norm_group(group_size, k);
    if (g <= 0 || k % g != 0)
        return WO_ERR_INVALID_ARG;
    if (bits == 8 && g != k)
        return WO_ERR_UNSUPPORTED;  // 8-bit weights are per channel
    if (bits == 4 && g != k && g % 64 != 0)
        return WO_ERR_UNSUPPORTED;
    return WO_OK;
}

wo_status cuda_status(cudaError_t e) { return e == cudaSuccess ? WO_OK : WO_ERR_CUDA; }

// Kernel choice by m: the weight-streaming kernel below kTcMinM rows (when
// its shared-memory ring fits), the tensor-core kernel otherwise.
// WO_MID_KERNEL overrides the choice at 17..64 rows for measurements:
// "stream" (the cluster-split streaming kernel), "tensor_core" (the m >= 65
// kernel); unset, 8-bit weights there take the swap-AB kernel.
int mid_override()
{
    static const int v = [] {
        const char* e = std::getenv("WO_MID_KERNEL");
        if (!e)
            return 0;
        if (std::strcmp(e, "stream") == 0)
            return 1;
        if (std::strcmp(e, "tensor_core") == 0)
            return 2;
        return 0;
    }();
    return v;
}

// 8-bit weights at 17..64 rows (between the decode sizes and the tensor-core
// kernel's) and at most one block of 128 channels per SM: the swap-AB
// tensor-core kernel, whose MMA rows are the output channels and whose
// columns are the activation rows.
bool use_mid(int m, int n, int k, int bits)
{
    return m > 16 && m < kTcMinM && mid_override() == 0 && plan_mid(m, n, k, bits).valid;
}

// 8-bit weights at 17..64 rows with more blocks of 128 channels than SMs:
// the m >= 65 tensor-core kernel (one MMA per 256 channels and 16 k, no k
// split needed to fill the SMs) streams them faster than either small-m
// kernel.
bool mid_wide(int m, int n, int k, int bits)
{
    return m > 16 && m < kTcMinM && bits == 8 && mid_override() == 0 && n % 128 == 0 && k % 64 == 0 &&
           n / 128 > num_sms();
}

// The tensor-core kernel: from kTcMinM rows, for the wide 8-bit shapes
// above, or below where neither the swap-AB kernel nor the streaming
// kernel's ring fits.
bool use_tc(int m, int n, int k, int group_size, int bits)
{
    if (m >= kTcMinM || (mid_override() == 2 && m > 16) || mid_wide(m, n, k, bits))
        return true;
    if (use_mid(m, n, k, bits))
        return false;
    return !stream_supported(m, n, k, norm_group(group_size, k), bits);
}

// Below the tensor-core sizes, 4-bit weights at decode-sized m (1..16) run
// the persistent kernel (wo_gemv.cu) where the cluster-split streaming
// kernel (wo_stream.cu) would need more than one resident wave of CTAs (2
// per SM): the wide lm_head-like shapes (131072 x 2048: 39 against 68 us at
// m = 1).  Everything else keeps the cluster kernel, long k with few
// channels included (320 x 16384: 13.5 against 27.7 us at m = 1; 1024 x
// 13312: 13.9 against 20.3 us; 2048 x 13312: 14.4 against 15.3 us).  The environment variable WO_DECODE_KERNEL
// overrides the choice for measurements and tests: "stream" forces the
// cluster kernel, "persistent" the persistent one wherever it applies (the
// two give results within tolerance of each other, not bit-identical ones).
int decode_override()
{
    static const int v = [] {
        const char* e = std::getenv("WO_DECODE_KERNEL");
        if (!e)
            return 0;
        if (std::strcmp(e, "stream") == 0)
            return 1;
        if (std::strcmp(e, "persistent") == 0)
            return 2;
        return 0;
    }();
    return v;
}

bool use_gemv_shape(int m, int n, int k, int group, int bits)
{
    if (m < 1 || m > 16 || decode_override() == 1 || !gemv_supported(m, n, k, group, bits))
        return false;
    if (decode_override() == 2)
        return true;
    const StreamPlan c = plan_stream(m, n, k, group, bits, OUT_PLAIN, 0);
    if (!c.valid)
        return true;
    const long long ctas = (long long)c.grid_x * c.splits;
    return ctas > 2LL * num_sms();
}

bool use_gemv(const GemmArgs& a)
{
    if (!use_gemv_shape(a.m, a.n, a.k, a.group, a.bits))
        return false;
    if (a.bits == 4 && a.group != a.k)
        return aligned(a.scales, 16) && (!a.zeros || aligned(a.zeros, 16));
    return true;
}

}  // namespace
}  // namespace wo

using namespace wo;

extern "C" {

const char* wo_status_string(wo_status s)
{
    switch (s) {
    case WO_OK: return "WO_OK";
    case WO_ERR_INVALID_ARG: return "WO_ERR_INVALID_ARG";
    case WO_ERR_UNSUPPORTED: return "WO_ERR_UNSUPPORTED";
    case WO_ERR_WORKSPACE: return "WO_ERR_WORKSPACE";
    case WO_ERR_CUDA: return "WO_ERR_CUDA";
    case WO_ERR_TIMEOUT: return "WO_ERR_TIMEOUT";
    case WO_ERR_BOUNDS: return "WO_ERR_BOUNDS";
    }
    return "WO_ERR_UNKNOWN";
}

wo_status wo_debug_bounds(unsigned* site)
{
#if !defined(WO_DEBUG_BOUNDS) || !WO_DEBUG_BOUNDS
    if (site)
        *site = 0;
    return WO_ERR_UNSUPPORTED;
#else
    if (site)
        *site = 0;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return WO_ERR_CUDA;
    // every translation unit's word is read (and so cleared); the first
    // non-zero one is reported
    const unsigned words[] = {bounds_take_stream(), bounds_take_gemv(),      bounds_take_gemm_tc(),
                              bounds_take_pack(),   bounds_take_act_order(), bounds_take_moe()};
    for (unsigned w : words)
        if (w) {
            if (site)
                *site = w;
            return WO_ERR_BOUNDS;
        }
    return WO_OK;
#endif
}

size_t wo_packed_bytes(int n, int k, int bits)
{
    if (n <= 0 || k <= 0 || n % 64 != 0 || k % 64 != 0 || (bits != 4 && bits != 8))
        return 0;
    return bits == 8 ? (size_t)n * (size_t)k : (size_t)n * (size_t)k / 2;
}

static wo_status pack_common(const uint8_t* src, uint8_t* dst, int n, int k, int bits,
                             bool unpack, void* stream)
{
    const size_t bytes = wo_packed_bytes(n, k, bits);
    if (bytes == 0 || !src || !dst || !aligned(src, 16) || !aligned(dst, 16))
        return WO_ERR_INVALID_ARG;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    if (s0 < d0 + bytes && d0 < s0 + bytes)
        return WO_ERR_INVALID_ARG;  // overlapping buffers
    return cuda_status(
        launch_pack(src, dst, n, k, bits, unpack, nullptr, static_cast<cudaStream_t>(stream)));
}

wo_status wo_pack(const uint8_t* B_rowmajor, uint8_t* B_packed, int n, int k, int bits,
                  void* stream)
{
    return pack_common(B_rowmajor, B_packed, n, k, bits, false, stream);
}

wo_status wo_unpack(const uint8_t* B_packed, uint8_t* B_rowmajor, int n, int k, int bits,
                    void* stream)
{
    return pack_common(B_packed, B_rowmajor, n, k, bits, true, stream);
}

size_t wo_workspace_size(int m, int n, int k, int group_size, int bits)
{
    if (check_gemm_shape(m, n, k, group_size, bits) != WO_OK || m == 0 || n == 0)
        return 0;
    if (use_tc(m, n, k, group_size, bits)) {
        // bf16 activations with 4-bit weights need an fp16 copy of A; size for
        // the larger of the two activation dtypes' needs
        return plan_tc(m, n, k, norm_group(group_size, k), bits, WO_BF16).ws_bytes;
    }
    if (use_mid(m, n, k, bits))
        return plan_mid(m, n, k, bits).ws_bytes;
    // either small-m kernel may run (the persistent one needs its partial sums)
    const size_t gv = use_gemv_shape(m, n, k, norm_group(group_size, k), bits)
                          ? gemv_workspace_bytes(m, n, k, norm_group(group_size, k), bits)
                          : 0;
    return gv > stream_workspace_bytes() ? gv : stream_workspace_bytes();
}

// Argument checks of wo_gemm, with `ws_need` the workspace the GEMM itself
// needs; fills `a` on success.  m == 0 or n == 0 returns WO_OK with a.m or
// a.n zero (nothing to launch).
static wo_status gemm_prepare(const void* A, const uint8_t* B_packed, const void* scales,
                              const void* zeros, const void* bias, void* C, int m, int n, int k,
                              int group_size, int bits, wo_dtype act_dtype, void* workspace,
                              size_t workspace_bytes, GemmArgs& a)
{
    a = GemmArgs{};
    wo_status st = check_gemm_shape(m, n, k, group_size, bits);
    if (st != WO_OK)
        return st;
    if (act_dtype != WO_F16 && act_dtype != WO_BF16)
        return WO_ERR_INVALID_ARG;
    if (bits == 8 && zeros)
        return WO_ERR_UNSUPPORTED;  // 8-bit weights are scale-only
    if (m == 0 || n == 0)
        return WO_OK;
    if (!A || !B_packed || !scales || !C)
        return WO_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B_packed, 16) || !aligned(C, 16) || !aligned(scales, 2) ||
        (zeros && !aligned(zeros, 2)) || (bias && !aligned(bias, 2)))
        return WO_ERR_INVALID_ARG;
    const size_t need = wo_workspace_size(m, n, k, group_size, bits);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return WO_ERR_WORKSPACE;
    a.A = A;
    a.B = B_packed;
    a.scales = scales;
    a.zeros = zeros;
    a.bias = bias;
    a.C = C;
    a.m = m;
    a.n = n;
    a.k = k;
    a.group = norm_group(group_size, k);
    a.bits = bits;
    a.act = act_dtype;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    return WO_OK;
}

static wo_status gemm_launch(const GemmArgs& a, cudaStream_t s)
{
    if (use_tc(a.m, a.n, a.k, a.group, a.bits))
        return cuda_status(launch_tc(a, plan_tc(a.m, a.n, a.k, a.group, a.bits, a.act), s));
    if (use_mid(a.m, a.n, a.k, a.bits))
        return cuda_status(launch_mid(a, s));
    if (use_gemv(a))
        return cuda_status(launch_gemv(a, s));
    return cuda_status(launch_stream_gemm(a, s));
}

wo_status wo_gemm(const void* A, const uint8_t* B_packed, const void* scales, const void* zeros,
                  const void* bias, void* C, int m, int n, int k, int group_size, int bits,
                  wo_dtype act_dtype, void* workspace, size_t workspace_bytes, void* stream)
{
    GemmArgs a;
    const wo_status st = gemm_prepare(A, B_packed, scales, zeros, bias, C, m, n, k, group_size,
                                      bits, act_dtype, workspace, workspace_bytes, a);
    if (st != WO_OK || a.m == 0 || a.n == 0)
        return st;
    return gemm_launch(a, static_cast<cudaStream_t>(stream));
}

wo_status wo_gemm_plan(int m, int n, int k, int group_size, int bits, wo_dtype act_dtype,
                       wo_gemm_plan_t* plan)
{
    if (!plan)
        return WO_ERR_INVALID_ARG;
    *plan = wo_gemm_plan_t{};
    const wo_status st = check_gemm_shape(m, n, k, group_size, bits);
    if (st != WO_OK)
        return st;
    if (act_dtype != WO_F16 && act_dtype != WO_BF16)
        return WO_ERR_INVALID_ARG;
    if (m == 0 || n == 0)
        return WO_OK;
    plan->workspace_bytes = wo_workspace_size(m, n, k, group_size, bits);
    const int g = norm_group(group_size, k);
    if (use_tc(m, n, k, g, bits)) {
        const TcPlan p = plan_tc(m, n, k, g, bits, act_dtype);
        const int tm = 128 * p.ms;
        const long long units =
            (long long)((m + tm - 1) / tm) * ((n + p.bn - 1) / p.bn) * p.splits;
        plan->kernel = WO_KERNEL_TENSOR_CORE;
        plan->tile_m = tm;
        plan->tile_n = p.bn;
        plan->k_splits = p.splits;
        plan->ctas = (int)(units < num_sms() ? units : num_sms());
        return WO_OK;
    }
    if (use_mid(m, n, k, bits)) {
        const MidPlan mp = plan_mid(m, n, k, bits);
        plan->kernel = WO_KERNEL_TENSOR_CORE_SWAP_AB;
        plan->tile_m = m;
        plan->tile_n = mp.ch;
        plan->k_splits = mp.ksplit;
        plan->ctas = mp.ctas;
        return WO_OK;
    }
    if (use_gemv_shape(m, n, k, g, bits)) {
        // (group-wise 4-bit with scales not 16-byte aligned runs WO_KERNEL_STREAM)
        const GemvInfo gi = gemv_info(m, n, k, g, bits);
        plan->kernel = WO_KERNEL_STREAM_PERSISTENT;
        plan->tile_m = m;
        plan->tile_n = gi.strip_channels;
        plan->k_splits = gi.max_pieces;
        plan->ctas = gi.ctas;
        plan->stages = gi.stages;
        return WO_OK;
    }
    const StreamPlan p = plan_stream(m, n, k, g, bits, OUT_PLAIN, 0);
    plan->kernel = WO_KERNEL_STREAM;
    plan->tile_m = m;
    plan->tile_n = p.nw * 32;  // each consumer warp owns two 16-channel blocks
    plan->k_splits = p.splits;
    plan->ctas = p.grid_x * p.splits;
    plan->stages = p.stages;
    return WO_OK;
}

// ---- GPTQ act-order ---------------------------------------------------------

wo_status wo_act_order_perm(const int32_t* g_idx, int k, int group_size, int32_t* perm)
{
    if (!g_idx || !perm || k <= 0)
        return WO_ERR_INVALID_ARG;
    const int g = norm_group(group_size, k);
    if (g <= 0 || k % g != 0)
        return WO_ERR_INVALID_ARG;
    const int G = k / g;
    // the group counters are the only host memory used; no exception may
    // leave a C entry point, so an allocation failure becomes a status
    std::vector<int> next;
    try {
        next.assign(G, 0);
    } catch (...) {
        return WO_ERR_INVALID_ARG;
    }
    for (int c = 0; c < k; ++c) {
        if (g_idx[c] < 0 || g_idx[c] >= G)
            return WO_ERR_INVALID_ARG;
        ++next[g_idx[c]];
    }
    for (int b = 0; b < G; ++b)
        if (next[b] != g)
            return WO_ERR_UNSUPPORTED;  // groups of unequal size
    // stable counting sort: group b's channels fill positions [b*g, (b+1)*g)
    for (int b = 0; b < G; ++b)
        next[b] = b * g;
    for (int c = 0; c < k; ++c)
        perm[next[g_idx[c]]++] = c;
    return WO_OK;
}

wo_status wo_pack_act_order(const uint8_t* B_rowmajor, uint8_t* B_packed, const int32_t* perm,
                            int n, int k, int bits, void* stream)
{
    const size_t bytes = wo_packed_bytes(n, k, bits);
    if (bytes == 0 || !B_rowmajor || !B_packed || !perm || !aligned(B_rowmajor, 16) ||
        !aligned(B_packed, 16) || !aligned(perm, 4))
        return WO_ERR_INVALID_ARG;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(B_rowmajor);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(B_packed);
    if (s0 < d0 + bytes && d0 < s0 + bytes)
        return WO_ERR_INVALID_ARG;  // overlapping buffers
    return cuda_status(launch_pack(B_rowmajor, B_packed, n, k, bits, false, perm,
                                   static_cast<cudaStream_t>(stream)));
}

// Offset of the gathered activations in an act-order workspace: after the
// GEMM's own workspace, and never inside the header and counter area that
// every call shares (the small-m GEMM itself needs only the header).
static size_t act_order_a_offset(int m, int n, int k, int group_size, int bits)
{
    const size_t g = wo_workspace_size(m, n, k, group_size, bits);
    return align_up(g > kWsScratch ? g : kWsScratch, 256);
}

size_t wo_act_order_workspace_size(int m, int n, int k, int group_size, int bits)
{
    if (check_gemm_shape(m, n, k, group_size, bits) != WO_OK || m == 0 || n == 0)
        return 0;
    return act_order_a_offset(m, n, k, group_size, bits) + align_up((size_t)m * k * 2, 256);
}

wo_status wo_gemm_act_order(const void* A, const uint8_t* B_packed, const int32_t* perm,
                            const void* scales, const void* zeros, const void* bias, void* C,
                            int m, int n, int k, int group_size, int bits, wo_dtype act_dtype,
                            void* workspace, size_t workspace_bytes, void* stream)
{
    GemmArgs a;
    wo_status st = gemm_prepare(A, B_packed, scales, zeros, bias, C, m, n, k, group_size, bits,
                                act_dtype, workspace, workspace_bytes, a);
    if (st != WO_OK || a.m == 0 || a.n == 0)
        return st;
    if (!perm || !aligned(perm, 16))
        return WO_ERR_INVALID_ARG;
    const size_t need = wo_act_order_workspace_size(m, n, k, group_size, bits);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return WO_ERR_WORKSPACE;
    const size_t off = act_order_a_offset(m, n, k, group_size, bits);
    void* Ap = static_cast<char*>(workspace) + off;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = cuda_status(launch_gather_cols(A, perm, Ap, m, k, s));
    if (st != WO_OK)
        return st;
    a.A = Ap;
    a.ws_bytes = off;
    return gemm_launch(a, s);
}

wo_status wo_embed(const int32_t* ids, int T, const uint8_t* B_packed, const void* scales,
                   const void* zeros, void* out, int vocab, int hidden, int group_size, int bits,
                   wo_dtype act_dtype, void* stream)
{
    // the table's shape rules are wo_gemm's with n = vocab, k = hidden
    if (T < 0 || vocab < 0 || hidden <= 0 || (bits != 4 && bits != 8) || vocab % 64 != 0 ||
        hidden % 64 != 0)
        return WO_ERR_INVALID_ARG;
    const int g = norm_group(group_size, hidden);
    if (g <= 0 || hidden % g != 0)
        return WO_ERR_INVALID_ARG;
    if ((bits == 8 && g != hidden) || (bits == 4 && g != hidden && g % 64 != 0))
        return WO_ERR_UNSUPPORTED;
    if (act_dtype != WO_F16 && act_dtype != WO_BF16)
        return WO_ERR_INVALID_ARG;
    if (bits == 8 && zeros)
        return WO_ERR_UNSUPPORTED;  // 8-bit weights are scale-only
    if (T == 0 || vocab == 0)
        return WO_OK;
    if (!ids || !B_packed || !scales || !out)
        return WO_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(B_packed, 16) || !aligned(scales, 2) || !aligned(out, 16) ||
        (zeros && !aligned(zeros, 2)))
        return WO_ERR_INVALID_ARG;
    return cuda_status(launch_embed(ids, T, B_packed, scales, zeros, out, vocab, hidden, g, bits,
                                    act_dtype, static_cast<cudaStream_t>(stream)));
}

wo_status wo_check_workspace(void* workspace, size_t workspace_bytes, void* stream)
{
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return WO_ERR_CUDA;
    if (!workspace || workspace_bytes < kWsHeader)
        return WO_OK;
    unsigned flag = 0;
    if (cudaMemcpy(&flag, workspace, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess)
        return WO_ERR_CUDA;
    if (flag == 0)
        return WO_OK;
    if (cudaMemset(workspace, 0, sizeof flag) != cudaSuccess)
        return WO_ERR_CUDA;
    return WO_ERR_TIMEOUT;
}

}  // extern "C"
