// wo_moe.cu -- grouped weight-only MoE FFN ("acext User Guide (v1.7)" 1.2.3
// MoE GEMM: gating output -> top-k experts per row -> fc1 with a gated
// activation -> fc2 -> routing-weighted combine), 8-bit per-channel expert
// weights.
//
//   1. route_sort_kernel (one CTA): per token, top-k of the fp32 logits
//      (ties to the lower expert id, compared exactly as stored) and the
//      softmax probabilities of the chosen experts over all experts
//      (renormalised over the chosen ones on request); then a stable
//      counting sort of the T*k (token, slot) pairs by expert, giving each
//      expert a contiguous range of rows.
//   2. expert_gemv_kernel<GATED = true>: per expert and 128 gate channels,
//      x1 = A[rows] . dequant(fc1_e)^T for the gate channels and the matching
//      up channels (inter apart), h = round(silu(g) * u) into [rows, inter].
//   3. expert_gemv_kernel<GATED = false>: y = h[rows] . dequant(fc2_e)^T in
//      fp32 into [rows, hidden].
//   4. combine_kernel: out[t] = round(sum_j p[t][j] * y[row(t, j)]), j in
//      ascending order.
// Every sum has a fixed order, so the result is bit-for-bit repeatable.
//
// The expert kernels stream packed 8-bit tiles exactly like the decode
// kernel (register dequant into mma.m16n8k16 fragments) but share the
// activation rows among all warps: the warps of a CTA own different channel
// blocks and walk k together, one 256-wide chunk at a time, reading the
// expert's gathered rows from a double-buffered shared-memory chunk.
#include <cuda_runtime.h>

#include "wo_common.cuh"
#include "wo_internal.h"

namespace wo {
namespace {

constexpr int kMoeWarps = 8;
constexpr int kChunk = 256;          // k per lockstep chunk (8 tiles of 32)
constexpr int kRowsPerPass = 64;     // activation rows per pass (8 n8-tiles)
constexpr int kMT = kRowsPerPass / 8;
constexpr int kDepth = 3;            // weight tiles in flight per block and warp
constexpr int kChunkTiles = kChunk / 32;
constexpr int kAStride = kChunk * 2 + 16;  // bytes per staged row (padded)
constexpr int kRouteThreads = 1024;

// ---------------------------------------------------------------- layout ---

struct MoeLayout {
    size_t ids, wts, pos, offsets, perm_tok, h, y, total;
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
    L.h = take(P * (size_t)inter * 2);
    L.y = take(P * (size_t)hidden * 4);
    L.total = off;
    return L;
}

// ------------------------------------------------------------- routing -----

__global__ void __launch_bounds__(kRouteThreads)
    route_sort_kernel(const float* __restrict__ logits, int T, int E, int topk, int renorm,
                      int* __restrict__ ids, float* __restrict__ wts, int* __restrict__ pos,
                      int* __restrict__ offsets, int* __restrict__ perm_tok)
{
    extern __shared__ int cnt[];  // [E] counts, then [E] running offsets
    int* run = cnt + E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt[e] = 0;
    __syncthreads();

    // ---- top-k and softmax weights, one warp per token ----
    for (int tok = warp; tok < T; tok += nwarps) {
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
            const float w = expf(bv - mx) / den;
            wsum += w;
            if (lane == 0) {
                ids[(size_t)tok * topk + j] = bi;
                wts[(size_t)tok * topk + j] = w;
            }
        }
        if (renorm && lane == 0)
            for (int j = 0; j < topk; ++j)
                wts[(size_t)tok * topk + j] /= wsum;
        if (lane == 0)
            for (int j = 0; j < topk; ++j)
                atomicAdd(&cnt[chosen[j]], 1);
    }
    __syncthreads();

    // ---- expert offsets (exclusive scan) and the stable counting sort ----
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? cnt[e] : 0;
            int incl = c;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (e < E) {
                offsets[e] = carry + incl - c;
                run[e] = carry + incl - c;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            offsets[E] = carry;
        __syncwarp();
        const int P = T * topk;
        for (int base = 0; base < P; base += 32) {
            const int slot = base + lane;
            const bool ok = slot < P;
            const int e = ok ? ids[slot] : -1 - lane;  // unique dummies for idle lanes
            const unsigned same = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(same & ((1u << lane) - 1u));
            int p = 0;
            if (ok)
                p = run[e] + rank;
            __syncwarp();
            if (ok) {
                pos[slot] = p;
                perm_tok[p] = slot / topk;
                if (rank == __popc(same) - 1)  // last lane of this expert's group
                    run[e] += __popc(same);
            }
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------- expert GEMV ----

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

struct ExpertParams {
    const uint16_t* A;      // GATED: tokens [T, K]; else sorted rows [P, K]
    const int* perm_tok;    // sorted row -> token (GATED only)
    const int* offsets;     // [E + 1]
    const uint8_t* W;       // packed weights, expert e at W + e * w_stride
    size_t w_stride;
    const uint16_t* scales; // [E, N]
    int N;                  // output channels of the weight (2*inter for fc1)
    int K;
    int inter;              // GATED: channel offset between gate and up
    uint16_t* H;            // GATED output [P, inter]
    float* Y;               // plain output [P, N]
};

// GATED: warp w of CTA x owns gate block (8x + w) and its up block
// (8x + w + inter/16).  Plain: warp w owns blocks 2(8x + w) and +1.
template <int ACT, bool GATED>
__global__ void __launch_bounds__(kMoeWarps * 32)
    expert_gemv_kernel(const ExpertParams p)
{
    extern __shared__ __align__(16) uint8_t a_sm[];  // [2][kRowsPerPass][kAStride]
    const int e = blockIdx.y;
    const int row0 = p.offsets[e];
    const int rows_e = p.offsets[e + 1] - row0;
    if (rows_e <= 0)
        return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int ktiles = p.K / 32;
    const int nblocks = p.N / 16;
    int blk[2];
    bool active;
    if constexpr (GATED) {
        blk[0] = blockIdx.x * kMoeWarps + warp;
        blk[1] = blk[0] + p.inter / 16;
        active = blk[0] < p.inter / 16;
    } else {
        blk[0] = 2 * (blockIdx.x * kMoeWarps + warp);
        blk[1] = blk[0] + 1;
        active = blk[1] < nblocks;
    }
    const uint8_t* Wexp = p.W + (size_t)e * p.w_stride;
    const uint16_t* sexp = p.scales + (size_t)e * p.N;
    const uint32_t a_base = static_cast<uint32_t>(__cvta_generic_to_shared(a_sm));
    const int nchunks = (p.K + kChunk - 1) / kChunk;

    for (int pass0 = 0; pass0 < rows_e; pass0 += kRowsPerPass) {
        const int rows = min(kRowsPerPass, rows_e - pass0);

        // stage chunk c of the pass's activation rows into buffer c & 1
        auto stage = [&](int c) {
            const int kc = c * kChunk;
            const int cols8 = min(kChunk, p.K - kc) / 8;
            const uint32_t buf = a_base + (uint32_t)((c & 1) * kRowsPerPass * kAStride);
            for (int idx = threadIdx.x; idx < rows * cols8; idx += blockDim.x) {
                const int r = idx / cols8, c8 = idx % cols8;
                const int srow = GATED ? p.perm_tok[row0 + pass0 + r] : row0 + pass0 + r;
                cp_async16(buf + r * kAStride + c8 * 16, p.A + (size_t)srow * p.K + kc + c8 * 8);
            }
            cp_async_commit();
        };

        float acc[2][kMT][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < kMT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[r][j][q] = 0.f;

        const uint8_t* wp[2];
#pragma unroll
        for (int r = 0; r < 2; ++r)
            wp[r] = Wexp + (size_t)(active ? blk[r] : 0) * ktiles * kTileBytes + lane * 16;
        uint4 buf[kDepth][2];
#pragma unroll
        for (int u = 0; u < kDepth; ++u)
#pragma unroll
            for (int r = 0; r < 2; ++r)
                if (active && u < ktiles)
                    buf[u][r] = ld_stream_v4(wp[r] + (size_t)u * kTileBytes);

        stage(0);
        int i = 0;  // tile index along k
        for (int c = 0; c < nchunks; ++c) {
            if (c + 1 < nchunks) {
                stage(c + 1);
                cp_async_wait_1();
            } else {
                cp_async_wait_0();
            }
            __syncthreads();
            const uint32_t abuf = a_base + (uint32_t)((c & 1) * kRowsPerPass * kAStride);
            const int ct1 = min((c + 1) * kChunkTiles, ktiles);
            if (active) {
                for (; i < ct1; i += kDepth) {
#pragma unroll
                    for (int u = 0; u < kDepth; ++u) {
                        const int ii = i + u;
                        if (ii < ct1) {
                            uint4 cur[2];
                            const int slot = ii % kDepth;
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                // slots rotate with the absolute tile index
                                cur[r] = slot == 0 ? buf[0][r] : slot == 1 ? buf[1][r] : buf[2][r];
                                if (ii + kDepth < ktiles) {
                                    const uint4 nv = ld_stream_v4(wp[r] + (size_t)(ii + kDepth) * kTileBytes);
                                    if (slot == 0) buf[0][r] = nv;
                                    else if (slot == 1) buf[1][r] = nv;
                                    else buf[2][r] = nv;
                                }
                            }
                            const uint32_t koff = (uint32_t)((ii - c * kChunkTiles) * 64);
#pragma unroll
                            for (int s = 0; s < 2; ++s) {
                                uint32_t a0[4], a1[4];
                                tile_frag<8, ACT>(cur[0], s, a0);
                                tile_frag<8, ACT>(cur[1], s, a1);
#pragma unroll
                                for (int j = 0; j < kMT; ++j) {
                                    if (8 * j < rows) {  // warp-uniform
                                        uint32_t b0 = 0u, b1 = 0u;
                                        if (8 * j + g < rows) {
                                            const uint32_t ap = abuf + (8 * j + g) * kAStride + koff + 32 * s + 4 * t;
                                            b0 = lds32(ap);
                                            b1 = lds32(ap + 16);
                                        }
                                        mma16816<ACT>(acc[0][j], a0, b0, b1);
                                        mma16816<ACT>(acc[1][j], a1, b0, b1);
                                    }
                                }
                            }
                        }
                    }
                }
                i = ct1;
            }
            __syncthreads();  // the buffer is restaged two chunks later
        }

        // ---- epilogue: element q of (r, j): channel blk[r]*16 + g + 8*(q>>1),
        // row 8j + 2t + (q & 1) of this pass ----
        if (active) {
#pragma unroll
            for (int j = 0; j < kMT; ++j) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int rr = 8 * j + 2 * t + (q & 1);
                    if (rr >= rows)
                        continue;
                    const size_t prow = (size_t)(row0 + pass0 + rr);
                    const int ch0 = blk[0] * 16 + g + 8 * (q >> 1);
                    const int ch1 = blk[1] * 16 + g + 8 * (q >> 1);
                    const float v0 = acc[0][j][q] * to_f32<ACT>(ld_nc_u16(sexp + ch0));
                    const float v1 = acc[1][j][q] * to_f32<ACT>(ld_nc_u16(sexp + ch1));
                    if constexpr (GATED) {
                        const float silu = v0 / (1.f + expf(-v0));
                        p.H[prow * p.inter + ch0] = from_f32<ACT>(silu * v1);
                    } else {
                        p.Y[prow * p.N + ch0] = v0;
                        p.Y[prow * p.N + ch1] = v1;
                    }
                }
            }
        }
    }
}

template <int ACT>
__global__ void combine_kernel(const float* __restrict__ Y, const int* __restrict__ pos,
                               const float* __restrict__ wts, uint16_t* __restrict__ out,
                               int hidden, int topk)
{
    const int tok = blockIdx.x;
    for (int c = threadIdx.x; c < hidden; c += blockDim.x) {
        float v = 0.f;
        for (int j = 0; j < topk; ++j) {
            const int p = pos[(size_t)tok * topk + j];
            v = fmaf(wts[(size_t)tok * topk + j], Y[(size_t)p * hidden + c], v);
        }
        out[(size_t)tok * hidden + c] = from_f32<ACT>(v);
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
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
    float* y = reinterpret_cast<float*>(ws + L.y);

    route_sort_kernel<<<1, kRouteThreads, 2 * E * (int)sizeof(int), s>>>(
        logits, T, E, topk, renorm, ids, wts, pos, offsets, perm_tok);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;

    const int smem = 2 * kRowsPerPass * kAStride;
    static int smem_set[64] = {0};
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess)
        return err;
    if (dev < 0 || dev >= 64 || smem_set[dev] < smem) {
        for (auto kern : {expert_gemv_kernel<ACT, true>, expert_gemv_kernel<ACT, false>})
            if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                cudaSuccess)
                return err;
        if (dev >= 0 && dev < 64)
            smem_set[dev] = smem;
    }

    ExpertParams p1{};
    p1.A = static_cast<const uint16_t*>(A);
    p1.perm_tok = perm_tok;
    p1.offsets = offsets;
    p1.W = fc1;
    p1.w_stride = (size_t)2 * I * H;
    p1.scales = static_cast<const uint16_t*>(fc1_s);
    p1.N = 2 * I;
    p1.K = H;
    p1.inter = I;
    p1.H = h;
    const dim3 g1((I / 16 + kMoeWarps - 1) / kMoeWarps, E);
    expert_gemv_kernel<ACT, true><<<g1, kMoeWarps * 32, smem, s>>>(p1);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;

    ExpertParams p2{};
    p2.A = h;
    p2.offsets = offsets;
    p2.W = fc2;
    p2.w_stride = (size_t)H * I;
    p2.scales = static_cast<const uint16_t*>(fc2_s);
    p2.N = H;
    p2.K = I;
    p2.Y = y;
    const dim3 g2((H / 32 + kMoeWarps - 1) / kMoeWarps, E);
    expert_gemv_kernel<ACT, false><<<g2, kMoeWarps * 32, smem, s>>>(p2);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;

    combine_kernel<ACT><<<T, 256, 0, s>>>(y, pos, wts, static_cast<uint16_t*>(out), H, topk);
    return cudaGetLastError();
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
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
    if (experts < 1 || experts > 1024 || topk < 1 || topk > experts || topk > 8)
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
