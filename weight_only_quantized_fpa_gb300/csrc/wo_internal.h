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

// bounded-wait self-test: one CTA waits on an mbarrier nothing completes,
// gives up after limit_us and records its code in *err (wo_selftest.cu)
cudaError_t launch_wait_timeout(unsigned* err, unsigned limit_us, cudaStream_t s);

// Index checks of the debug build (wo_bounds.cuh): each translation unit's
// first failed site since the last call, cleared; 0 for none (always 0 in a
// build without the checks).
unsigned bounds_take_stream();
unsigned bounds_take_gemv();
unsigned bounds_take_gemm_tc();
unsigned bounds_take_pack();
unsigned bounds_take_act_order();
unsigned bounds_take_moe();

// ---- pack -----------------------------------------------------------------
// perm (pack only, optional): packed column j takes row-major column perm[j]
cudaError_t launch_pack(const uint8_t* src, uint8_t* dst, int n, int k, int bits, bool unpack,
                        const int32_t* perm, cudaStream_t s);
// A' = A[:, perm] (act-order GEMM): rows of k 16-bit values, perm [k]
cudaError_t launch_gather_cols(const void* A, const int32_t* perm, void* Ap, int m, int k,
                               cudaStream_t s);
// rows ids[0..T) of a packed [vocab, hidden] table, dequantised (wo_embed)
cudaError_t launch_embed(const int32_t* ids, int T, const uint8_t* B, const void* scales,
                         const void* zeros, void* out, int vocab, int hidden, int group, int bits,
                         int act, cudaStream_t s);

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

// small m: the weight-streaming kernel (wo_stream.cu)
size_t stream_workspace_bytes();
bool stream_supported(int m, int n, int k, int group, int bits);
cudaError_t launch_stream_gemm(const GemmArgs& a, cudaStream_t s);

// decode-sized m (1..16): the persistent weight-streaming kernel (wo_gemv.cu)
struct GemvInfo {
    int ctas, stages, strip_channels, max_pieces;
};
bool gemv_supported(int m, int n, int k, int group, int bits);
size_t gemv_workspace_bytes(int m, int n, int k, int group, int bits);  // 0 when unsupported
GemvInfo gemv_info(int m, int n, int k, int group, int bits);
cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t s);

// ---- tensor-core kernel (large m) -----------------------------------------
constexpr int kTcMinM = 65;  // m at and above which wo_gemm uses the tensor-core kernel

struct TcPlan {
    int bn, ms;             // output tile: ms x 128 rows by bn columns
    int splits;             // k split (units per tile); 1: none
    size_t a16_bytes;       // fp16 copy of a bf16 A (4-bit weights only)
    size_t rowscale_bytes;  // its per-row power-of-two scales
    size_t sz_bytes;        // 4-bit: pre-scaled fp16 (scale, zero) pairs [n, G]
    size_t colscale_bytes;  // 4-bit: per-channel powers of two [n] (bf16 bits)
    size_t partial_bytes;   // k split: fp32 partial tiles
    size_t ws_bytes;        // total, header and counter area included
};

// allow_split = false plans without the k split (no partial-tile scratch).
// group: codes per scale group along k (k for per-channel).
TcPlan plan_tc(int m, int n, int k, int group, int bits, int act, bool allow_split = true);
cudaError_t launch_tc(const GemmArgs& a, const TcPlan& p, cudaStream_t s);

// 8-bit weights at 17..64 rows: the swap-AB expert kernel as a plain GEMM
// (channel blocks of 128 or 256 by k splits; wo_gemm_tc.cu)
struct MidPlan {
    int ch, nb;            // channels per block, blocks
    int ksplit, kps;       // k splits per block, k blocks per split
    int ctas;
    size_t partial_bytes;  // fp32 sums of the splits
    size_t ws_bytes;       // total, header and counter area included
    bool valid;
};
MidPlan plan_mid(int m, int n, int k, int bits);
cudaError_t launch_mid(const GemmArgs& a, cudaStream_t s);

// MoE expert GEMMs on the tensor cores (8-bit codes; hidden and inter
// multiples of 128): gated fc1 -> h [rows, inter] in the activation dtype,
// or fc2 -> fp32 [rows, n_out]; rows are in expert order, offsets[E + 1].
bool moe_tc_supported(int hidden, int inter);
cudaError_t launch_moe_tc(bool gated, int act, const void* rows, int total_rows, int k,
                          const uint8_t* codes, const void* scales, int experts, int n_out,
                          int inter, const int* offsets, void* out, unsigned* err, cudaStream_t s);

}  // namespace wo
