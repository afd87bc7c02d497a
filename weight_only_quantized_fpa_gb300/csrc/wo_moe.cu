// wo_moe.cu -- grouped weight-only MoE FFN ("acext User Guide (v1.7)" 1.2.3
// MoE GEMM: gating output -> top-k experts per row -> fc1 with a gated
// activation -> fc2 -> routing-weighted combine), 8-bit per-channel expert
// weights.
//
//   1. route_topk_kernel (a warp per token): top-k of the fp32 logits (ties
//      to the lower expert id, compared exactly as stored) and the softmax
//      probabilities of the chosen experts over all experts (renormalised
//      over the chosen ones on request); route_sort_kernel (one CTA): a
//      stable counting sort of the T*k (token, slot) pairs by expert, giving
//      each expert a contiguous range of rows.
//   2. gather_rows_kernel copies the activation rows into expert order;
//      then fc1 with the gated output: x1 = A[rows] . dequant(fc1_e)^T for
//      gate channels and the matching up channels (inter apart),
//      h = round(silu(g) * u) into [rows, inter];
//   3. fc2 to fp32: y = h[rows] . dequant(fc2_e)^T into [rows, hidden].
//      Steps 2 and 3 run on the tensor cores (moe_tc_kernel in
//      wo_gemm_tc.cu: the expert's dequantised weights are the MMA's
//      128-row operand, its rows the N operand) when hidden and inter are
//      multiples of 128, else on the weight-streaming kernel (wo_stream.cu,
//      one CTA row per expert, mma.sync).
//   4. combine_kernel: out[t] = round(sum_j p[t][j] * y[row(t, j)]), j in
//      ascending order.
// Every sum has a fixed order, so the result is bit-for-bit repeatable.
//
// The expert GEMMs run up to 64 rows per pass (chunk); experts with more rows
// take several passes over their weights.
#include <cuda_runtime.h>

#include "wo_bounds.cuh"
#include "wo_common.cuh"
#include "wo_internal.h"
#include "wo_stream.h"

namespace wo {
namespace {

constexpr int kTopkWarps = 8;   // tokens per top-k CTA
constexpr int kSortWarps = 32;  // warps of the sorting CTA

// ---------------------------------------------------------------- layout ---

struct MoeLayout {
    size_t ids, wts, pos, offsets, perm_tok, a_sorted, h, y, total;
};

MoeLayout moe_layout(int T, int hidden, int inter, int experts, int topk)
{
    MoeLayout L{};
    const size_t P = (size_t)T * topk;
    size_t off = kWsScratch;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.ids = take(P * 4);
    L.wts = take(P * 4);
    L.pos = take(P * 4);
    L.offsets = take((size_t)(experts + 1) * 4);
    L.perm_tok = take(P * 4);
    L.a_sorted = take(P * (size_t)hidden * 2);
    L.h = take(P * (size_t)inter * 2);
    L.y = take(P * (size_t)hidden * 4);
    L.total = off;
    return L;
}

// ------------------------------------------------------------- routing -----

// Top-k and softmax weights, one warp per token.
__global__ void __launch_bounds__(kTopkWarps * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int topk, int renorm,
                      int* __restrict__ ids, float* __restrict__ wts)
{
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (tok >= T)
        return;
    const float* lg = logits + (size_t)tok * E;
    float mx = -INFINITY;
    for (int e = lane; e < E; e += 32)
        mx = fmaxf(mx, lg[e]);
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
    for (int e = lane; e < E; e += 32)
        den += expf(lg[e] - mx);
    for (int o = 16; o > 0; o >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, o);
    int chosen[8];
    float w[8];
    float wsum = 0.f;
    for (int j = 0; j < topk; ++j) {
        // best remaining logit; on equal values the lower id wins
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int e = lane; e < E; e += 32) {
            bool taken = false;
            for (int q = 0; q < j; ++q)
                taken |= chosen[q] == e;
            const float v = lg[e];
            if (!taken && (v > bv || (v == bv && e < bi) || bi == 0x7fffffff)) {
                bv = v;
                bi = e;
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        chosen[j] = bi;
        w[j] = expf(bv - mx) / den;
        wsum += w[j];
    }
    if (lane == 0)
        for (int j = 0; j < topk; ++j) {
            ids[(size_t)tok * topk + j] = chosen[j];
            wts[(size_t)tok * topk + j] = renorm ? w[j] / wsum : w[j];
        }
}

// Stable counting sort of the P = T * topk (token, slot) pairs by expert in
// one CTA: warp v owns the slots [v L, (v + 1) L).  Per-warp counts per
// expert give each expert's total and offset and each warp's base inside
// the expert; each warp then places its slots in slot order, so an expert's
// rows keep the slot order (deterministic).
__global__ void __launch_bounds__(kSortWarps * 32)
    route_sort_kernel(const int* __restrict__ ids, int P, int E, int topk, int* __restrict__ pos,
                      int* __restrict__ offsets, int* __restrict__ perm_tok)
{
    extern __shared__ int sm[];
    int* base = sm;                      // [kSortWarps][E]: counts, then bases
    int* off = sm + kSortWarps * E;      // [E] expert offsets
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = (P + kSortWarps - 1) / kSortWarps;
    const int s0 = warp * L, s1 = min(P, s0 + L);
    for (int i = threadIdx.x; i < kSortWarps * E; i += blockDim.x)
        base[i] = 0;
    __syncthreads();
    for (int slot = s0 + lane; slot < s1; slot += 32)
        atomicAdd(&base[warp * E + ids[slot]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int v = 0; v < kSortWarps; ++v) {
            const int c = base[v * E + e];
            base[v * E + e] = run;
            run += c;
        }
        off[e] = run;  // the expert's total, for the scan below
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int b = 0; b < E; b += 32) {
            const int e = b + lane;
            const int c = e < E ? off[e] : 0;
            int incl = c;
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += x;
            }
            if (e < E) {
                off[e] = carry + incl - c;
                offsets[e] = carry + incl - c;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            offsets[E] = carry;
    }
    __syncthreads();
    int* my = base + warp * E;
    for (int b = s0; b < s1; b += 32) {
        const int slot = b + lane;
        const bool ok = slot < s1;
        const int e = ok ? ids[slot] : -1 - lane;  // unique dummies for idle lanes
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        int p = 0;
        if (ok && in_bounds(e >= 0 && e < E, 0x701))
            p = off[e] + my[e] + rank;
        __syncwarp();
        if (ok && in_bounds(e >= 0 && e < E && p < P, 0x702)) {
            pos[slot] = p;
            perm_tok[p] = slot / topk;
            if (rank == __popc(same) - 1)  // last lane of this expert's group
                my[e] += __popc(same);
        }
        __syncwarp();
    }
}

// A rows in expert order: a_sorted[p] = A[perm_tok[p]] (16-byte pieces).
__global__ void gather_rows_kernel(const uint4* __restrict__ A, const int* __restrict__ perm_tok,
                                   uint4* __restrict__ a_sorted, int row_vecs, int T)
{
    const int p = blockIdx.x;
    if (!in_bounds(perm_tok[p] >= 0 && perm_tok[p] < T, 0x703))
        return;
    const uint4* src = A + (size_t)perm_tok[p] * row_vecs;
    uint4* dst = a_sorted + (size_t)p * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x)
        dst[i] = src[i];
}

// A CTA per token; the token's rows and weights are read once into
// registers (topk <= kMaxTopk), and a thread takes 8 channels at a time: two
// 16-byte loads per row, one 16-byte store (hidden % 64 == 0, out 16-byte
// aligned).  Per channel the sum is the same chain of fused multiply-adds
// over j in ascending order.
constexpr int kMaxTopk = 8;

template <int ACT>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ Y, const int* __restrict__ pos,
                   const float* __restrict__ wts, uint16_t* __restrict__ out, int hidden, int topk,
                   int P)
{
    const int tok = blockIdx.x;
    int pj[kMaxTopk];
    float wj[kMaxTopk];
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
        pj[j] = -1;  // j >= topk, or a position outside the rows: skipped
        wj[j] = 0.f;
        if (j < topk) {
            const int p = pos[(size_t)tok * topk + j];
            if (in_bounds(p >= 0 && p < P, 0x704)) {
                pj[j] = p;
                wj[j] = wts[(size_t)tok * topk + j];
            }
        }
    }
    for (int c = threadIdx.x * 8; c < hidden; c += blockDim.x * 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
            if (pj[j] < 0)
                continue;
            const float4* y = reinterpret_cast<const float4*>(Y + (size_t)pj[j] * hidden + c);
            const float4 a = y[0], b = y[1];
            v[0] = fmaf(wj[j], a.x, v[0]);
            v[1] = fmaf(wj[j], a.y, v[1]);
            v[2] = fmaf(wj[j], a.z, v[2]);
            v[3] = fmaf(wj[j], a.w, v[3]);
            v[4] = fmaf(wj[j], b.x, v[4]);
            v[5] = fmaf(wj[j], b.y, v[5]);
            v[6] = fmaf(wj[j], b.z, v[6]);
            v[7] = fmaf(wj[j], b.w, v[7]);
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = (uint32_t)from_f32<ACT>(v[2 * i]) | ((uint32_t)from_f32<ACT>(v[2 * i + 1]) << 16);
        *reinterpret_cast<uint4*>(out + (size_t)tok * hidden + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int ACT>
cudaError_t launch_moe(const void* A, const float* logits, const uint8_t* fc1, const void* fc1_s,
                       const uint8_t* fc2, const void* fc2_s, void* out, int T, int H, int I,
                       int E, int topk, int renorm, char* ws, cudaStream_t s)
{
    const MoeLayout L = moe_layout(T, H, I, E, topk);
    int* ids = reinterpret_cast<int*>(ws + L.ids);
    float* wts = reinterpret_cast<float*>(ws + L.wts);
    int* pos = reinterpret_cast<int*>(ws + L.pos);
    int* offsets = reinterpret_cast<int*>(ws + L.offsets);
    int* perm_tok = reinterpret_cast<int*>(ws + L.perm_tok);
    uint16_t* a_sorted = reinterpret_cast<uint16_t*>(ws + L.a_sorted);
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
    float* y = reinterpret_cast<float*>(ws + L.y);

    route_topk_kernel<<<(T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, s>>>(
        logits, T, E, topk, renorm, ids, wts);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const int P = T * topk;
    const int sort_smem = (kSortWarps + 1) * E * (int)sizeof(int);
    if ((err = cudaFuncSetAttribute(route_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    sort_smem)) != cudaSuccess)
        return err;
    route_sort_kernel<<<1, kSortWarps * 32, sort_smem, s>>>(ids, P, E, topk, pos, offsets, perm_tok);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;

    gather_rows_kernel<<<P, 128, 0, s>>>(static_cast<const uint4*>(A), perm_tok,
                                         reinterpret_cast<uint4*>(a_sorted), H / 8, T);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;

    if (moe_tc_supported(H, I)) {
        // tensor-core expert GEMMs: fc1 (gated) into h, fc2 into fp32 y
        unsigned* errw = reinterpret_cast<unsigned*>(ws);
        if ((err = launch_moe_tc(true, ACT, a_sorted, P, H, fc1, fc1_s, E, 2 * I, I, offsets, h,
                                 errw, s)) != cudaSuccess)
            return err;
        if ((err = launch_moe_tc(false, ACT, h, P, I, fc2, fc2_s, E, H, 0, offsets, y, errw, s)) !=
            cudaSuccess)
            return err;
        combine_kernel<ACT><<<T, 256, 0, s>>>(y, pos, wts, static_cast<uint16_t*>(out), H, topk, P);
        return cudaGetLastError();
    }

    // fc1 with the gated activation, on the rows in expert order
    StreamPlan P1 = plan_stream(64, 2 * I, H, H, 8, OUT_GATED, I);
    if (!P1.valid)
        return cudaErrorInvalidValue;
    StreamParams p1{};
    p1.A = a_sorted;
    p1.a_rows_total = P;
    p1.offsets = offsets;
    p1.B = fc1;
    p1.w_block_rows = E * (2 * I / 16);
    p1.blocks_per_expert = 2 * I / 16;
    p1.scales = static_cast<const uint16_t*>(fc1_s);
    p1.s_stride = (size_t)2 * I;
    p1.N = 2 * I;
    p1.K = H;
    p1.ktiles = H / 32;
    p1.G = 1;
    p1.tiles_per_group = H / 32;
    p1.inter = I;
    p1.kt_per_split = H / 32;
    p1.splits = 1;
    p1.stages = P1.stages;
    p1.C = h;
    p1.err = reinterpret_cast<unsigned*>(ws);
    if ((err = launch_stream(p1, P1, 8, ACT, OUT_GATED, E, s)) != cudaSuccess)
        return err;

    // fc2 to fp32: the sorted rows of h
    StreamPlan P2 = plan_stream(64, H, I, I, 8, OUT_F32, 0);
    if (!P2.valid)
        return cudaErrorInvalidValue;
    StreamParams p2 = p1;
    p2.A = h;
    p2.B = fc2;
    p2.w_block_rows = E * (H / 16);
    p2.blocks_per_expert = H / 16;
    p2.scales = static_cast<const uint16_t*>(fc2_s);
    p2.s_stride = (size_t)H;
    p2.N = H;
    p2.K = I;
    p2.ktiles = I / 32;
    p2.tiles_per_group = I / 32;
    p2.inter = 0;
    p2.kt_per_split = I / 32;
    p2.stages = P2.stages;
    p2.C = nullptr;
    p2.Y = y;
    if ((err = launch_stream(p2, P2, 8, ACT, OUT_F32, E, s)) != cudaSuccess)
        return err;

    combine_kernel<ACT><<<T, 256, 0, s>>>(y, pos, wts, static_cast<uint16_t*>(out), H, topk, P);
    return cudaGetLastError();
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

unsigned bounds_take_moe() { return bounds_take_local(); }

}  // namespace wo

using namespace wo;

extern "C" {

size_t wo_moe_workspace_size(int T, int hidden, int inter, int experts, int topk)
{
    if (T <= 0 || hidden <= 0 || inter <= 0 || experts <= 0 || topk <= 0 || topk > experts)
        return 0;
    return moe_layout(T, hidden, inter, experts, topk).total;
}

wo_status wo_moe_ffn(const void* A, const float* gating_logits, const uint8_t* fc1_packed,
                     const void* fc1_scales, const uint8_t* fc2_packed, const void* fc2_scales,
                     void* out, int T, int hidden, int inter, int experts, int topk,
                     int renormalize, wo_dtype act_dtype, void* workspace,
                     size_t workspace_bytes, void* stream)
{
    if (T < 0 || hidden <= 0 || inter <= 0 || hidden % 64 != 0 || inter % 64 != 0)
        return WO_ERR_INVALID_ARG;
    if (experts < 1 || experts > 1024 || topk < 1 || topk > experts || topk > kMaxTopk)
        return WO_ERR_INVALID_ARG;
    if (act_dtype != WO_F16 && act_dtype != WO_BF16)
        return WO_ERR_INVALID_ARG;
    if (T == 0)
        return WO_OK;
    if (!A || !gating_logits || !fc1_packed || !fc1_scales || !fc2_packed || !fc2_scales || !out)
        return WO_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(gating_logits, 4) || !aligned(fc1_packed, 16) ||
        !aligned(fc2_packed, 16) || !aligned(out, 16) || !aligned(fc1_scales, 2) ||
        !aligned(fc2_scales, 2))
        return WO_ERR_INVALID_ARG;
    const size_t need = wo_moe_workspace_size(T, hidden, inter, experts, topk);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return WO_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = act_dtype == WO_F16
        ? launch_moe<ACT_F16>(A, gating_logits, fc1_packed, fc1_scales, fc2_packed, fc2_scales,
                              out, T, hidden, inter, experts, topk, renormalize, ws, s)
        : launch_moe<ACT_BF16>(A, gating_logits, fc1_packed, fc1_scales, fc2_packed, fc2_scales,
                               out, T, hidden, inter, experts, topk, renormalize, ws, s);
    return e == cudaSuccess ? WO_OK : WO_ERR_CUDA;
}

}  // extern "C"
