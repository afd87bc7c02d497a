// wo_stream.h -- host interface of the weight-streaming kernel (wo_stream.cu),
// shared by the small-m GEMM and the MoE expert GEMMs.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "wo_internal.h"

namespace wo {

enum { OUT_PLAIN = 0, OUT_GATED = 1, OUT_F32 = 2 };

struct StreamParams {
    const uint16_t* A;      // activation rows of K values (MoE: in expert order)
    int a_rows_total;       // rows of A
    const int* offsets;     // MoE: [E + 1] row ranges per expert (null: one group of m rows)
    int m;                  // rows when offsets is null (<= 64)
    const uint8_t* B;       // packed weights; expert e follows expert e - 1
    int w_block_rows;       // 16-channel block rows of B in all (all experts)
    int blocks_per_expert;  // block rows of one expert (MoE)
    const uint16_t* scales; // [N] or [N, G]; expert e at + e * s_stride
    size_t s_stride;
    const uint16_t* zeros;  // 4-bit only, [N, G] or null
    const uint16_t* bias;   // plain output only, [N] or null
    int N, K, ktiles;
    int G, tiles_per_group;
    int inter;              // gated output: channel distance between gate and up
    int kt_per_split, splits;
    int stages, g_span;
    uint16_t* C;            // plain [m, N] or gated [rows, inter]
    float* Y;               // fp32 output [rows, N]
    unsigned* err;          // error word (workspace header)
};

struct StreamPlan {
    int mt, nw, tps, grid_x, splits, kt_per_split, stages, g_span;
    size_t smem;
    bool valid;
};

StreamPlan plan_stream(int m, int n, int k, int group, int bits, int out, int inter);
cudaError_t launch_stream(const StreamParams& p, const StreamPlan& plan, int bits, int act, int out,
                          int grid_y, cudaStream_t s);

}  // namespace wo
