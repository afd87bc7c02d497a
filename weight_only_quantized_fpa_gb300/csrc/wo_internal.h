// wo_internal.h -- host-side declarations shared by the libwo translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "wo.h"  // include/wo.h, found through -I

namespace wo {

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)            header: word 0 = error flag written by kernels that
//                       gave up a bounded wait; the rest reserved
//   [256, 256 + 64 KiB) split-K arrival counters, one per output tile; every
//                       kernel returns the counters it used to zero, and no
//                       other data is ever written here, so calls of any
//                       shape can share one workspace
//   [256 + 64 KiB, ...) per-call scratch (fp32 partial sums, converted
//                       activations), planned per call
constexpr size_t kWsHeader = 256;
constexpr size_t kWsCounters = 16384;  // counters (4 bytes each)
constexpr size_t kWsScratch = kWsHeader + kWsCounters * 4;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int num_sms();  // SM count of the current device (152 when none is visible)

// ---- pack -----------------------------------------------------------------
cudaError_t launch_pack(const uint8_t* src, uint8_t* dst, int n, int k, int bits, bool unpack,
                        cudaStream_t s);

// ---- weight-streaming kernel (small m) -----------------------------------
struct GemvPlan {
    int mt;             // 8-row activation tiles per pass (1, 2, 4 or 8)
    int m_per_pass;     // rows per launch (8 * mt)
    int passes;         // launches needed to cover m
    int grid_x;         // CTAs along n (32 output channels each)
    int splits;         // CTAs along k, one thread-block cluster (<= 8)
    int ktiles;         // k / KT
    int ktiles_per_split;
    int a_rows;         // activation rows staged in shared memory per launch
    int a_stride;       // bytes per staged activation row
    int g_span;         // scale groups staged per channel (4-bit)
    bool valid;         // false when k is too long to stage even 8 rows
    size_t ws_bytes;    // workspace bytes (none: the reduction stays on chip)
};

GemvPlan plan_gemv(int m, int n, int k, int group, int bits);

struct GemmArgs {
    const void* A;
    const uint8_t* B;
    const void* scales;
    const void* zeros;
    const void* bias;
    void* C;
    int m, n, k;
    int group;  // codes per scale group along k (k for per-channel)
    int bits;
    int act;    // WO_F16 / WO_BF16
    void* ws;
    size_t ws_bytes;
};

cudaError_t launch_gemv(const GemmArgs& a, const GemvPlan& p, cudaStream_t s);

// ---- tensor-core kernel (large m) -----------------------------------------
constexpr int kTcMinM = 65;  // m at and above which wo_gemm uses the tensor-core kernel

struct TcPlan {
    size_t a16_bytes;       // fp16 copy of a bf16 A (4-bit weights only)
    size_t rowscale_bytes;  // its per-row power-of-two scales
    size_t ws_bytes;        // total, header and counter area included
};

TcPlan plan_tc(int m, int n, int k, int bits, int act);
cudaError_t launch_tc(const GemmArgs& a, const TcPlan& p, cudaStream_t s);

}  // namespace wo
