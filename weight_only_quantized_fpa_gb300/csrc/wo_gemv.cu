// wo_gemv.cu -- the persistent weight-streaming kernel for decode-sized m
// (1..16 rows) with 4-bit weights:
//
//   C[m, n] = A[m, k] . dequant(B)^T + bias[n],  w = (q - 8) s + z
//
// (acext User Guide (v1.7) 1.3.2 / 1.3.3 Int4 per-channel and group-wise;
// vLLM-Omni "cpu_int4.py", module docstring, for the group-64 rule).  At
// decode sizes every packed weight byte is read once per call and the
// arithmetic per byte is small, so the time is HBM time plus whatever the
// kernel fails to overlap with it (the same docstring: the bits per weight,
// not the FLOPs, set the decode rate).  4-bit codes carry twice the weights
// per byte of 8-bit ones, so per byte of HBM traffic this kernel has twice
// the conversion and multiply work: it is built to spend as few
// instructions per byte as possible.
//
// Work split ("stream-K" over the weight matrix): the output channels are
// cut into strips of 256 channels, each strip's k range into stages of 128
// codes; the strip-major sequence of (strip, stage) units is divided into P
// equal contiguous ranges, one per CTA, two CTAs per SM.  Every CTA streams
// the same number of weight bytes as one continuous pipeline across strip
// boundaries: no wave quantisation.  A CTA's range covers whole strips
// (their outputs are written directly) and up to two strip pieces; a
// piece's fp32 partial sums go to the workspace and the CTA whose piece of a
// strip arrives last sums the strip's pieces in k order and writes the
// outputs (no CTA ever waits for another; the order of every sum is fixed
// by the shape, so results are bit-for-bit repeatable).
//
// Per CTA: one producer warp whose lane 0 fills a ring of shared-memory
// stages with TMA tensor copies (the packed weights of the strip's 16
// channel blocks for 128 codes of k, the activation rows, and for
// group-wise weights the boxes of 8 groups of scales and zeros that cover
// them); 8 consumer warps each own two 16-channel blocks.  A lane reads its
// 16 bytes of a packed tile (its mma.m16n8k16 A fragments, see
// wo_common.cuh), converts them to fp16/bf16 pairs and multiplies them on
// the tensor cores against the activations, accumulating in fp32.
//
// Code conversion without removing the offset: a low nibble becomes fp16
// 1024 + q (bits 0x6400 | q) or bf16 128 + q (0x4300 | q), an fp16 high
// nibble 64 + q (0x5400 | q << 4: the spacing of fp16 at 64 is 1/16, so no
// shift is needed).  Every value is an exact integer; with P'' the partial
// sum of a * (off + q) over a tile and R the sum of its activations (an mma
// against a fragment of ones),
//   sum a * ((q - 8) s + z) = s * P'' + (z - (off + 8) s) * R,
// so the scale, the zero and the offset enter once per tile and channel in
// fp32 (the offset never meets more than 64 terms of cancellation).
//
// One activation row (m = 1): the mma's 8 output columns would hold one row
// and seven zero rows.  Instead tile t's activations go to column t mod 8
// (the other columns get zeros), so 8 consecutive tiles -- 8 groups of 64
// codes -- accumulate side by side, and every lane folds its two columns'
// groups once per 8 tiles; the four lanes of a row are summed at the end.
//
// Programmatic dependent launch: before waiting for the previous grid the
// producer fetches the weights and scales of the first ring stages and the
// consumers their channels' per-channel values; activations are read and
// outputs written after the wait.  Every mbarrier wait is bounded; a wait
// that runs out records an error word in the workspace and the CTA winds
// down without a hang (every consumer warp still passes every named
// barrier, skipping the work).
#include "wo_bounds.cuh"
#include "wo_common.cuh"
#include "wo_internal.h"
#include "wo_sm100.cuh"
#include "wo_tmap.h"

namespace wo {
namespace {

using namespace sm100;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr int kGvStageK = 128;                      // codes of k per stage
constexpr int kGvTps = kGvStageK / 64;              // packed 4-bit tiles per block per stage
static_assert(kGvTps % 2 == 0, "a stage starts at an even k tile");
constexpr int kGvNw = 8;                            // consumer warps
constexpr int kGvCh = kGvNw * 32;                   // channels per strip
constexpr int kSzGroups = 8;                        // groups per scale box (16 bytes of 16-bit values)
constexpr int kGvWBytes = 2 * kGvNw * kGvTps * kTileBytes;
constexpr int kGvSzBox = kGvCh * kSzGroups * 2;     // one box of scales (or zeros)

// ONE (m = 1): the stage's activations are one unswizzled box of 128
// values; else two boxes of 64 k by 8 * MT rows (rows past m read as zeros)
// with the 128-byte swizzle that ldmatrix reads conflict-free.
template <int MT, bool ONE>
struct GvGeom {
    static constexpr int ROWS = ONE ? 1 : 8 * MT;
    static constexpr int A_BOX = ONE ? 2 * kGvStageK : ROWS * 128;
    static constexpr int A_BYTES = ONE ? A_BOX : 2 * A_BOX;
    static constexpr int NV = 2 * MT * 4;     // accumulator values per lane
};

struct GvParams {
    int m, N, K;
    int ktiles;        // K / 64
    int nst;           // stages per strip
    int nstrips;
    long long T;       // units (strip, stage) in all
    int lg_tpg;        // log2(group / 64), group-wise
    int G;             // groups per channel
    int stages;        // ring stages
    int stage_bytes;
    int tx;            // bytes a stage receives
    int maxseg;        // partial slots per strip
    const uint16_t* scales;  // per channel: [N]
    const uint16_t* zeros;   // per channel: [N] or null
    const uint16_t* bias;    // [N] or null
    uint16_t* C;             // [m, N]
    float* partial;          // [nstrips][maxseg][256][NV]
    unsigned* counters;      // [nstrips], zero between calls
    unsigned* err;
};

// CTA whose range of units holds unit u: the largest w with
// floor(w T / P) <= u.
__device__ __forceinline__ int worker_of(long long u, long long T, int P)
{
    int w = (int)((u * P) / T);
    while (w + 1 < P && ((long long)(w + 1) * T) / P <= u)
        ++w;
    while (w > 0 && ((long long)w * T) / P > u)
        --w;
    return w;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// Shared-memory loads at byte offset `off` of the CTA's shared window
// (shared-space addresses: measured 10 % faster than C++ loads through the
// window's generic pointer).  Volatile, so they stay between the mbarrier
// wait that makes a stage's data visible and the arrive that releases it.
__device__ __forceinline__ uint16_t lds_u16(const uint8_t* smem, uint32_t off)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_addr(smem) + off));
    return v;
}

__device__ __forceinline__ uint4 lds_v4(const uint8_t* smem, uint32_t off)
{
    return lds128(smem_addr(smem) + off);
}

// d += a . b, and d = a . b with a zero accumulator (the first k-step of a
// tile).  Register-only operations, so not volatile: the compiler may
// interleave independent mma chains with the conversions around them.
template <int ACT>
__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if constexpr (ACT == ACT_F16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

template <int ACT>
__device__ __forceinline__ void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1)
{
    const float z = 0.f;
    if constexpr (ACT == ACT_F16) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
    }
}

// 4-bit codes of k-step s of a packed tile, offsets kept (see the file
// comment): a[0], a[2] rows g (low nibbles), a[1], a[3] rows g + 8 (high
// nibbles).  fp16: 1024 + q and 64 + q; bf16: 128 + q.
template <int ACT>
__device__ __forceinline__ void frag_u4_biased(uint32_t w, uint32_t (&a)[4])
{
    if constexpr (ACT == ACT_F16) {
        const uint32_t w8 = w >> 8;
        a[0] = and_or(w, 0x000F000Fu, 0x64006400u);
        a[1] = and_or(w, 0x00F000F0u, 0x54005400u);
        a[2] = and_or(w8, 0x000F000Fu, 0x64006400u);
        a[3] = and_or(w8, 0x00F000F0u, 0x54005400u);
    } else {
        a[0] = and_or(w, 0x000F000Fu, 0x43004300u);
        a[1] = and_or(w >> 4, 0x000F000Fu, 0x43004300u);
        a[2] = and_or(w >> 8, 0x000F000Fu, 0x43004300u);
        a[3] = and_or(w >> 12, 0x000F000Fu, 0x43004300u);
    }
}

// offset + 8 of the converted values of rows g (low nibbles) and g + 8
// (high nibbles)
template <int ACT>
struct U4Off {
    static constexpr float lo = ACT == ACT_F16 ? 1032.f : 136.f;
    static constexpr float hi = ACT == ACT_F16 ? 72.f : 136.f;
};

// MT: 8-row activation blocks (1 or 2); ONE: m == 1 (MT == 1), tiles spread
// over the 8 output columns; GROUPED: scales and zeros per group (boxes in
// the stage) rather than per channel; ZEROS: group-wise zeros given.
constexpr int kGvCtasPerSm = 2;
constexpr size_t kGvSmemBudget = 110 * 1024;  // per CTA: two CTAs per SM

template <int ACT, int MT, bool ONE, bool GROUPED, bool ZEROS>
__global__ void __launch_bounds__((kGvNw + 1) * 32, kGvCtasPerSm)
    gemv4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                 const GvParams p)
{
    using Gm = GvGeom<MT, ONE>;
    constexpr int NV = Gm::NV, NW = kGvNw, CH = kGvCh, TPS = kGvTps;
    // Group-wise scales and zeros: with every stage, the boxes of 8 groups by
    // the strip's channels that cover it (a separate ring of boxes loaded
    // once per 8 groups measured slower: with two slots the producer waits
    // for the consumers at every box change, which shortens the stage ring).
    static_assert(!ONE || MT == 1, "one row fits one row block");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const uint32_t zero_off = (uint32_t)(S * p.stage_bytes);  // 16 zero bytes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + zero_off + 16);
    uint64_t* empty = full + S;
    int* abort_flag = reinterpret_cast<int*>(empty + S);
    int* last_flag = abort_flag + 1;
    volatile int* abort = abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = (int)gridDim.x;
    const long long u0 = ((long long)blockIdx.x * p.T) / P;
    const long long u1 = ((long long)(blockIdx.x + 1) * p.T) / P;
    const int nunits = (int)(u1 - u0);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
        *last_flag = 0;
        *reinterpret_cast<uint4*>(smem + zero_off) = make_uint4(0u, 0u, 0u, 0u);
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        if constexpr (GROUPED) {
            tma_prefetch_desc(&tmS);
            if constexpr (ZEROS)
                tma_prefetch_desc(&tmZ);
        }
    }
    __syncthreads();
    if (nunits <= 0)
        return;

    if (warp == NW) {
        // ================= producer (one thread) =================
        if (lane == 0) {
            auto load_w = [&](int s, int strip, int st) {
                uint8_t* stage = smem + (size_t)s * p.stage_bytes;
                const int kt0 = st * TPS;
                tma_load_2d(stage + Gm::A_BYTES, &tmW, &full[s], kt0 * 64, strip * 2 * NW);
                if constexpr (GROUPED) {
                    const int x0 = ((kt0 >> p.lg_tpg) / kSzGroups) * kSzGroups;
                    uint8_t* sz = stage + Gm::A_BYTES + kGvWBytes;
                    tma_load_2d(sz, &tmS, &full[s], x0, strip * CH);
                    if constexpr (ZEROS)
                        tma_load_2d(sz + kGvSzBox, &tmZ, &full[s], x0, strip * CH);
                }
            };
            auto load_a = [&](int s, int st) {
                uint8_t* stage = smem + (size_t)s * p.stage_bytes;
                tma_load_2d(stage, &tmA, &full[s], st * kGvStageK, 0);
                if constexpr (!ONE)
                    tma_load_2d(stage + Gm::A_BOX, &tmA, &full[s], st * kGvStageK + 64, 0);
            };
            // the first ring's weights do not depend on the previous grid
            const int pre = nunits < S ? nunits : S;
            int strip = (int)(u0 / p.nst), st = (int)(u0 % p.nst);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], (uint32_t)p.tx);
                load_w(i, strip, st);
                if (++st == p.nst) {
                    st = 0;
                    ++strip;
                }
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            strip = (int)(u0 / p.nst);
            st = (int)(u0 % p.nst);
            bool ok = true;
            int i = 0;
            for (; i < nunits; ++i) {
                const int s = i % S;
                if (i >= pre) {
                    ok = mbar_wait_bounded(&empty[s], ((i / S) & 1) ^ 1, abort, p.err, 31, kWaitLimitNs);
                    if (!ok)
                        break;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)p.tx);
                    load_w(s, strip, st);
                }
                load_a(s, st);
                if (++st == p.nst) {
                    st = 0;
                    ++strip;
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA winds down
                // (the loop only gives up at i >= pre, with stages [0, i)
                // issued in full)
                volatile int never = 0;
                for (int j = i - S > 0 ? i - S : 0; j < i; ++j)
                    mbar_wait_bounded(&full[j % S], (j / S) & 1, &never, nullptr, 0, kWaitLimitNs);
            }
        }
        return;
    }

    // ================= consumers =================
    // Every consumer warp runs the same sequence of units, segments and named
    // barriers whatever happens: after a wait gives up (ok false) it still
    // passes every barrier, only skipping the work, so no warp is ever left
    // at a barrier the others do not reach.
    const int g = lane >> 2, t = lane & 3;
    const uint32_t w_lane0 = (uint32_t)(Gm::A_BYTES + (2 * warp) * TPS * kTileBytes + lane * 16);
    const uint32_t w_lane1 = w_lane0 + (uint32_t)(TPS * kTileBytes);
    const uint32_t a_row = (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * 128);
    const uint32_t a_hi = (uint32_t)((lane >> 3) & 1);
    const uint32_t a_xor = (uint32_t)(lane & 7);
    const int c_lo = 32 * warp + g;  // channel within the strip of the lane's row g, block 0

    float acc[2][MT][4];
    // ONE: the 8 tiles of a column window, accumulated column by column;
    // even and odd tiles in two register sets (two independent mma chains)
    float wp[2][2][4], wr[2][4];
    float ps[2][2], pz[2][2];  // per channel: s and z - (off + 8) s of the lane's 4 channels

    int strip = (int)(u0 / p.nst), st = (int)(u0 % p.nst);
    int seg_st0 = st;  // first stage of the current segment
    bool ok = true;

    auto clear_window = [&]() {
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                wp[e][0][q] = wp[e][1][q] = 0.f;
                wr[e][q] = 0.f;
            }
    };

    auto seg_begin = [&]() {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[r][j][q] = 0.f;
        if constexpr (ONE)
            clear_window();
        const int blk = strip * 2 * NW + 2 * warp;
        const bool active = blk + 1 < p.N / 16;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ch = (blk + r) * 16 + g + 8 * h;
                ps[r][h] = pz[r][h] = 0.f;
                if (!GROUPED && active && in_bounds(ch < p.N, 0x201)) {
                    const float sv = to_f32<ACT>(ld_nc_u16(p.scales + ch));
                    const float zv = p.zeros ? to_f32<ACT>(ld_nc_u16(p.zeros + ch)) : 0.f;
                    ps[r][h] = sv;
                    pz[r][h] = fmaf(-(h ? U4Off<ACT>::hi : U4Off<ACT>::lo), sv, zv);
                }
            }
    };

    // scale and folded zero of channel (r, h) of this lane for group box
    // column gi of the stage's scale boxes at sbox (per channel: registers)
    auto scale_zero = [&](uint32_t sbox, int gi, int r, int h, float& sv, float& zv) {
        if constexpr (GROUPED) {
            const uint32_t off = (uint32_t)(((c_lo + 16 * r + 8 * h) * kSzGroups + gi) * 2);
            sv = to_f32<ACT>(lds_u16(smem, sbox + off));
            const float z = ZEROS ? to_f32<ACT>(lds_u16(smem, sbox + (uint32_t)kGvSzBox + off)) : 0.f;
            zv = fmaf(-(h ? U4Off<ACT>::hi : U4Off<ACT>::lo), sv, z);
        } else {
            sv = ps[r][h];
            zv = pz[r][h];
        }
    };

    // ONE: fold the column window that tile kt closes (or the segment cuts):
    // column c of the window holds tile (kt & ~7) + c; this lane holds
    // columns 2t and 2t + 1
    auto fold_window = [&](uint32_t sbox, int kt, int x0) {
        const int wbase = kt & ~7;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int gi = GROUPED ? ((wbase + 2 * t + c) >> p.lg_tpg) - x0 : 0;
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float sv, zv;
                    scale_zero(sbox, gi, r, h, sv, zv);
                    // column 2t + c holds tiles of parity c only
                    const int q = 2 * h + c;
                    acc[r][0][q] = fmaf(sv, wp[c][r][q], fmaf(zv, wr[c][q], acc[r][0][q]));
                }
        }
        clear_window();
    };

    // output of the lane's values fin for strip `sp` (bias added, one
    // rounding, rows past m skipped)
    auto store_c = [&](int sp, const float (&fin)[2][MT][4]) {
        const int blk = sp * 2 * NW + 2 * warp;
        if (blk + 1 >= p.N / 16)
            return;  // this warp's blocks are past n (last strip)
        float bb[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                bb[r][h] = p.bias && in_bounds((blk + r) * 16 + g + 8 * h < p.N, 0x202)
                               ? to_f32<ACT>(ld_nc_u16(p.bias + (blk + r) * 16 + g + 8 * h))
                               : 0.f;
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int row = 8 * j + 2 * t + (q & 1);
                if (row >= p.m)
                    continue;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int ch = (blk + r) * 16 + g + 8 * (q >> 1);
                    if (in_bounds(ch < p.N, 0x203))
                        p.C[(size_t)row * p.N + ch] = from_f32<ACT>(fin[r][j][q] + bb[r][q >> 1]);
                }
            }
    };

    // the segment's sums -> C (a whole strip) or the workspace (a piece; the
    // CTA whose piece of the strip arrives last sums the strip's pieces in k
    // order and stores them)
    auto seg_end = [&](int st_last) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs: after the previous grid
        float fin[2][MT][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    fin[r][j][q] = acc[r][j][q];
        if constexpr (ONE) {
            // a channel's columns are spread over the 4 lanes of its row:
            // sum them (the same value in all 4 lanes), row 0 only
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float v = fin[r][0][2 * h] + fin[r][0][2 * h + 1];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    fin[r][0][2 * h] = v;
                    fin[r][0][2 * h + 1] = 0.f;
                }
        }
        if (seg_st0 == 0 && st_last == p.nst - 1) {
            if (ok)
                store_c(strip, fin);
            return;
        }
        const long long su0 = (long long)strip * p.nst;
        const int wf = worker_of(su0, p.T, P);
        const int nseg = worker_of(su0 + p.nst - 1, p.T, P) - wf + 1;
        const float* base = p.partial + ((size_t)strip * p.maxseg * CH + (size_t)(32 * warp + lane)) * NV;
        if (ok && in_bounds(strip < p.nstrips && (int)blockIdx.x - wf >= 0 && (int)blockIdx.x - wf < p.maxseg &&
                                nseg <= p.maxseg, 0x204)) {
            float4* dst = reinterpret_cast<float4*>(const_cast<float*>(base) + (size_t)((int)blockIdx.x - wf) * CH * NV);
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int j = 0; j < MT; ++j)
                    __stcg(dst + r * MT + j, make_float4(fin[r][j][0], fin[r][j][1], fin[r][j][2], fin[r][j][3]));
        }
        // every consumer's piece is written; the CTA barrier orders those
        // writes before thread 0's fence, which releases them at GPU scope
        // ahead of the arrival count
        asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
        if (threadIdx.x == 0) {
            int last = 0;
            if (!*abort && in_bounds(strip < p.nstrips, 0x206)) {
                __threadfence();
                last = atomicAdd(p.counters + strip, 1u) == (unsigned)(nseg - 1) ? 1 : 0;
                if (last)
                    __threadfence();  // acquire: every other piece is visible
            }
            *last_flag = last;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
        if (!*(volatile int*)last_flag)
            return;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    fin[r][j][q] = 0.f;
        // slot order = k order; RB pieces' loads in flight at a time
        constexpr int RB = MT == 1 ? 4 : 2;
        for (int j0 = 0; j0 < nseg; j0 += RB) {
            float4 x[RB][2 * MT];
#pragma unroll
            for (int b = 0; b < RB; ++b)
#pragma unroll
                for (int v = 0; v < 2 * MT; ++v)
                    x[b][v] = j0 + b < nseg && in_bounds(j0 + b < p.maxseg, 0x205)
                                  ? __ldcg(reinterpret_cast<const float4*>(base + (size_t)(j0 + b) * CH * NV) + v)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < RB; ++b)
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        fin[r][j][0] += x[b][r * MT + j].x;
                        fin[r][j][1] += x[b][r * MT + j].y;
                        fin[r][j][2] += x[b][r * MT + j].z;
                        fin[r][j][3] += x[b][r * MT + j].w;
                    }
        }
        store_c(strip, fin);
        if (threadIdx.x == 0)
            p.counters[strip] = 0u;  // ready for the next call
    };

    // one packed tile (both blocks) of the stage at offset `stage` of the
    // shared window, tile tl of it
    const uint32_t sbase = smem_addr(smem);  // shared-space address (ldmatrix)
    auto do_tile = [&](uint32_t stage, uint32_t sbox, int kt0, int tl, int x0, const uint4 v0,
                       const uint4 v1) {
        const uint32_t one = ones_x2<ACT>();
        const uint32_t ones[4] = {one, one, one, one};
        if constexpr (ONE) {
            // activations in column (kt0 + tl) mod 8 only: lanes of that
            // column (g) keep them, the others get zeros
            const int kt = kt0 + tl;
            // ldmatrix of the tile's 64 activations as the B fragments of its
            // four k-steps (matrix i = 8 values of k, row r = column r): the
            // rows of the tile's column r = kt mod 8 point at the activations,
            // every other row at 16 zero bytes, so the other columns get zeros
            const uint32_t act = sbase + stage + (uint32_t)(tl * 128 + (lane >> 3) * 16);
            const bool mine = (lane & 7) == (kt & 7);
            uint32_t bf[4][2];
            ldsm_x4(mine ? act : sbase + zero_off, bf[0][0], bf[0][1], bf[1][0], bf[1][1]);
            ldsm_x4(mine ? act + 64u : sbase + zero_off, bf[2][0], bf[2][1], bf[3][0], bf[3][1]);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t b0 = bf[ks][0], b1 = bf[ks][1];
                const uint32_t w0 = ks == 0 ? v0.x : ks == 1 ? v0.y : ks == 2 ? v0.z : v0.w;
                const uint32_t w1 = ks == 0 ? v1.x : ks == 1 ? v1.y : ks == 2 ? v1.z : v1.w;
                uint32_t a0[4], a1[4];
                frag_u4_biased<ACT>(w0, a0);
                frag_u4_biased<ACT>(w1, a1);
                // kt0 is a multiple of the (even) tiles per stage, so kt and tl
                // have the same parity: a compile-time choice after unrolling
                if ((tl & 1) == 0) {
                    mma_acc<ACT>(wp[0][0], a0, b0, b1);
                    mma_acc<ACT>(wp[0][1], a1, b0, b1);
                    mma_acc<ACT>(wr[0], ones, b0, b1);
                } else {
                    mma_acc<ACT>(wp[1][0], a0, b0, b1);
                    mma_acc<ACT>(wp[1][1], a1, b0, b1);
                    mma_acc<ACT>(wr[1], ones, b0, b1);
                }
            }
            if ((tl & 1) && (kt & 7) == 7)  // only an odd tile ends a window of 8
                fold_window(sbox, kt, x0);
        } else {
            float gp[2][MT][4], rs[MT][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int kk = tl * 64 + 16 * ks;
                const uint32_t box = sbase + stage + (uint32_t)((kk >> 6) * Gm::A_BOX);
                const uint32_t col = ((((uint32_t)(kk & 63) >> 3) + a_hi) ^ a_xor) << 4;
                uint32_t b[MT][2];
                if constexpr (MT == 1)
                    ldsm_x2(box + a_row + col, b[0][0], b[0][1]);
                else
                    ldsm_x4(box + a_row + col, b[0][0], b[0][1], b[1][0], b[1][1]);
                const uint32_t w0 = ks == 0 ? v0.x : ks == 1 ? v0.y : ks == 2 ? v0.z : v0.w;
                const uint32_t w1 = ks == 0 ? v1.x : ks == 1 ? v1.y : ks == 2 ? v1.z : v1.w;
                uint32_t a0[4], a1[4];
                frag_u4_biased<ACT>(w0, a0);
                frag_u4_biased<ACT>(w1, a1);
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    if (ks == 0) {
                        mma16816_z<ACT>(gp[0][j], a0, b[j][0], b[j][1]);
                        mma16816_z<ACT>(gp[1][j], a1, b[j][0], b[j][1]);
                        mma16816_z<ACT>(rs[j], ones, b[j][0], b[j][1]);
                    } else {
                        mma_acc<ACT>(gp[0][j], a0, b[j][0], b[j][1]);
                        mma_acc<ACT>(gp[1][j], a1, b[j][0], b[j][1]);
                        mma_acc<ACT>(rs[j], ones, b[j][0], b[j][1]);
                    }
                }
            }
            // fold the tile: acc += s P'' + (z - (off + 8) s) R per channel
            const int gi = GROUPED ? ((kt0 + tl) >> p.lg_tpg) - x0 : 0;
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float sv, zv;
                    scale_zero(sbox, gi, r, h, sv, zv);
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        acc[r][j][2 * h] = fmaf(sv, gp[r][j][2 * h], fmaf(zv, rs[j][2 * h], acc[r][j][2 * h]));
                        acc[r][j][2 * h + 1] =
                            fmaf(sv, gp[r][j][2 * h + 1], fmaf(zv, rs[j][2 * h + 1], acc[r][j][2 * h + 1]));
                    }
                }
        }
    };

    seg_begin();
    for (int i = 0; i < nunits; ++i) {
        const int s = i % S;
        const bool strip_end = st == p.nst - 1;
        const bool seg_last = strip_end || i == nunits - 1;
        const int x0 = GROUPED ? (((st * TPS) >> p.lg_tpg) / kSzGroups) * kSzGroups : 0;
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(&full[s], (i / S) & 1, abort, p.err, 32, kWaitLimitNs));
        if (ok) {
            const int kt0 = st * TPS;
            const uint32_t stage = (uint32_t)(s * p.stage_bytes);  // offset in the shared window
            const uint32_t sbox = stage + (uint32_t)(Gm::A_BYTES + kGvWBytes);
            const bool two = kt0 + 1 < p.ktiles;  // a strip's last stage may hold one tile
            const uint32_t t1 = (uint32_t)kTileBytes;
            if constexpr (MT == 1) {
                // both tiles' weight loads before the first tile's work, so
                // that the second tile's loads overlap it (more rows would
                // spill: their accumulators take the registers)
                const uint4 v00 = lds_v4(smem, stage + w_lane0), v01 = lds_v4(smem, stage + w_lane1);
                uint4 v10 = v00, v11 = v01;
                if (two) {
                    v10 = lds_v4(smem, stage + w_lane0 + t1);
                    v11 = lds_v4(smem, stage + w_lane1 + t1);
                }
                do_tile(stage, sbox, kt0, 0, x0, v00, v01);
                if (two)
                    do_tile(stage, sbox, kt0, 1, x0, v10, v11);
            } else {
                do_tile(stage, sbox, kt0, 0, x0, lds_v4(smem, stage + w_lane0), lds_v4(smem, stage + w_lane1));
                if (two)
                    do_tile(stage, sbox, kt0, 1, x0, lds_v4(smem, stage + w_lane0 + t1),
                            lds_v4(smem, stage + w_lane1 + t1));
            }
            if constexpr (ONE) {
                // a segment that ends inside a column window folds it now
                const int kt_last = kt0 + (two ? 1 : 0);
                if (seg_last && (kt_last & 7) != 7)
                    fold_window(sbox, kt_last, x0);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
        }
        // end of a segment: the strip's last stage, or this CTA's last unit
        if (seg_last) {
            seg_end(st);
            if (strip_end) {
                ++strip;
                st = 0;
            } else {
                ++st;
            }
            seg_st0 = st;
            if (i + 1 < nunits)
                seg_begin();
        } else {
            ++st;
        }
    }
}

}  // namespace

// ------------------------------------------------------------------ host ---

namespace {


struct GvPlan {
    int mt, stages, stage_bytes, grid, nstrips, nst, maxseg;
    long long T;
    size_t smem, partial_bytes;
    bool valid;
};

int ilog2_exact(int x)
{
    int l = 0;
    while ((1 << l) < x)
        ++l;
    return (1 << l) == x ? l : -1;
}

GvPlan plan_gemv(int m, int n, int k, int group, int bits)
{
    GvPlan P{};
    P.valid = false;
    if (bits != 4 || m < 1 || m > 16)
        return P;
    P.mt = m <= 8 ? 1 : 2;
    const bool one = m == 1;
    const int a_bytes = one ? 2 * kGvStageK : 2 * 8 * P.mt * 128;
    const bool grouped = group != k;
    if (grouped) {
        const int G = k / group;
        if (G % kSzGroups != 0 || ilog2_exact(group / 64) < 0)
            return P;  // scale boxes need 8-group-aligned rows; groups of 64 * 2^j
    }
    P.stage_bytes = (a_bytes + kGvWBytes + (grouped ? 2 * kGvSzBox : 0) + 1023) / 1024 * 1024;
    const size_t fixed = 1024 + 512;
    int stages = (int)((kGvSmemBudget - fixed) / P.stage_bytes);
    if (stages > 8)
        stages = 8;
    if (stages < 2)
        return P;
    P.stages = stages;
    P.smem = fixed + (size_t)stages * P.stage_bytes;
    P.nstrips = (n + kGvCh - 1) / kGvCh;
    P.nst = (k + kGvStageK - 1) / kGvStageK;
    P.T = (long long)P.nstrips * P.nst;
    const int workers = num_sms() * kGvCtasPerSm;
    P.grid = (int)(P.T < workers ? P.T : workers);
    const long long q = P.T / P.grid;  // units per CTA, at least
    P.maxseg = q == 0 ? P.nst : (int)((P.nst - 1 + q - 1) / q + 2);
    if (P.maxseg > P.nst)
        P.maxseg = P.nst;
    P.partial_bytes = align_up((size_t)P.nstrips * P.maxseg * kGvCh * (2 * P.mt * 4) * 4, 256);
    if ((size_t)P.nstrips > kWsCounters)
        return P;
    P.valid = true;
    return P;
}

template <int ACT, int MT, bool ONE, bool GROUPED, bool ZEROS>
cudaError_t launch_gemv_t(const GemmArgs& a, const GvPlan& plan, cudaStream_t s)
{
    using Gm = GvGeom<MT, ONE>;
    CUtensorMap ma, mw, ms, mz;
    const CUtensorMapDataType dt16 =
        ACT == ACT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tmap_2d(&ma, dt16, a.A, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2,
                      ONE ? kGvStageK : 64, Gm::ROWS,
                      ONE ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int ktiles = a.k / 64;
    if (!make_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT64, a.B, (uint64_t)ktiles * 64, (uint64_t)a.n / 16,
                      (uint64_t)ktiles * kTileBytes, kGvTps * 64, 2 * kGvNw, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    ms = mw;
    mz = mw;
    const int G = a.k / a.group;
    if (GROUPED) {
        if (!make_tmap_2d(&ms, dt16, a.scales, (uint64_t)G, (uint64_t)a.n, (uint64_t)G * 2, kSzGroups, kGvCh,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        if (ZEROS && !make_tmap_2d(&mz, dt16, a.zeros, (uint64_t)G, (uint64_t)a.n, (uint64_t)G * 2, kSzGroups,
                                   kGvCh, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    GvParams p{};
    p.m = a.m;
    p.N = a.n;
    p.K = a.k;
    p.ktiles = ktiles;
    p.nst = plan.nst;
    p.nstrips = plan.nstrips;
    p.T = plan.T;
    p.lg_tpg = GROUPED ? ilog2_exact(a.group / 64) : 0;
    p.G = G;
    p.stages = plan.stages;
    p.stage_bytes = plan.stage_bytes;
    p.tx = Gm::A_BYTES + kGvWBytes + (GROUPED ? kGvSzBox * (ZEROS ? 2 : 1) : 0);
    p.maxseg = plan.maxseg;
    p.scales = static_cast<const uint16_t*>(a.scales);
    p.zeros = static_cast<const uint16_t*>(a.zeros);
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.C = static_cast<uint16_t*>(a.C);
    char* ws = static_cast<char*>(a.ws);
    p.err = reinterpret_cast<unsigned*>(ws);
    p.counters = reinterpret_cast<unsigned*>(ws + kWsHeader);
    p.partial = reinterpret_cast<float*>(ws + kWsScratch);

    auto kern = gemv4_kernel<ACT, MT, ONE, GROUPED, ZEROS>;
    static int smem_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || smem_set[dev] < (int)plan.smem) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem)) !=
            cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            smem_set[dev] = (int)plan.smem;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3((kGvNw + 1) * 32);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mw, ms, mz, p);
}

template <int ACT, int MT, bool ONE>
cudaError_t launch_gemv_g(const GemmArgs& a, const GvPlan& plan, cudaStream_t s)
{
    if (a.group == a.k)
        return launch_gemv_t<ACT, MT, ONE, false, false>(a, plan, s);
    return a.zeros ? launch_gemv_t<ACT, MT, ONE, true, true>(a, plan, s)
                   : launch_gemv_t<ACT, MT, ONE, true, false>(a, plan, s);
}

template <int ACT>
cudaError_t launch_gemv_a(const GemmArgs& a, const GvPlan& plan, cudaStream_t s)
{
    if (a.m == 1)
        return launch_gemv_g<ACT, 1, true>(a, plan, s);
    return plan.mt == 1 ? launch_gemv_g<ACT, 1, false>(a, plan, s) : launch_gemv_g<ACT, 2, false>(a, plan, s);
}

}  // namespace

bool gemv_supported(int m, int n, int k, int group, int bits)
{
    return plan_gemv(m, n, k, group, bits).valid;
}

size_t gemv_workspace_bytes(int m, int n, int k, int group, int bits)
{
    const GvPlan P = plan_gemv(m, n, k, group, bits);
    return P.valid ? kWsScratch + P.partial_bytes : 0;
}

GemvInfo gemv_info(int m, int n, int k, int group, int bits)
{
    const GvPlan P = plan_gemv(m, n, k, group, bits);
    GemvInfo r{};
    if (P.valid) {
        r.ctas = P.grid;
        r.stages = P.stages;
        r.strip_channels = kGvCh;
        r.max_pieces = P.maxseg;
    }
    return r;
}

cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t s)
{
    const GvPlan plan = plan_gemv(a.m, a.n, a.k, a.group, a.bits);
    if (!plan.valid)
        return cudaErrorInvalidValue;
    return a.act == WO_F16 ? launch_gemv_a<ACT_F16>(a, plan, s) : launch_gemv_a<ACT_BF16>(a, plan, s);
}

unsigned bounds_take_gemv() { return bounds_take_local(); }

}  // namespace wo
