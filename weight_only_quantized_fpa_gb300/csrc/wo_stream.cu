// wo_stream.cu -- the weight-streaming kernel: small-m GEMM (decode) and the
// MoE expert GEMMs.
//
// At small m every packed weight byte is read once per call and the
// arithmetic per byte is tiny, so the kernel is bound by HBM bandwidth (the
// point of vLLM-Omni "cpu_int4.py"'s module docstring: the bits per weight,
// not the FLOPs, set the decode rate).  Design, per CTA:
//
//   - one producer thread streams the CTA's share of the packed weights and
//     the matching activation rows into a ring of shared-memory stages with
//     TMA tensor copies (cp.async.bulk.tensor, completion counted on an
//     mbarrier per stage): the packed weights are viewed as a 2-D tensor of
//     16-channel block rows by k, so one copy brings every block of the CTA
//     for a 64- or 128-wide k slice; the activations are a 2-D tensor of
//     rows by k, fetched 64 wide with the 128-byte swizzle (MoE rows are
//     first gathered into expert order so that an expert's rows are
//     contiguous); two or three copies per stage in all;
//   - NW consumer warps each own two channel blocks, so one staged slice of
//     activations serves NW * 32 channels.  A lane reads its 16 bytes of a
//     packed tile (exactly its mma.m16n8k16 A fragments, see wo_common.cuh),
//     turns the codes into exact (q - offset) fp16/bf16 pairs and multiplies
//     them on the tensor cores against activation fragments read from the
//     stage, accumulating in fp32; then it frees the stage;
//   - 4-bit group-wise weights (acext User Guide 1.3.3, w = (q - 8) s + z)
//     keep per-group partials P_g = sum a (q - 8) and activation sums R_g
//     (an mma against a ones fragment) and fold acc += s P_g + z R_g in fp32
//     at each group end, so the tensor cores only see exact integers; 8-bit
//     per-channel weights (1.3.1) apply scale[n] once at the end;
//   - when k is long for the number of channels, the k range is split across
//     a thread-block cluster of up to 8 CTAs: each consumer warp pushes its
//     partial sums into a slot in the shared memory of the rank that owns its
//     channels (rank = warp % splits) and arrives on that rank's mbarrier;
//     the owner sums the slots in rank order and writes the outputs.  A CTA
//     leaves as soon as its pushes are out and its own channels are done.
//   - 8-bit decode rows (m <= 16) accumulate even and odd k-steps in two sets
//     (summed at the end), two independent mma chains per channel block.
//   - launched with programmatic dependent launch: the producer fetches the
//     weights of the first stages (for decode, of the CTA's whole k range)
//     and the consumers their channels' scales and bias before waiting for
//     the previous grid; every read of activations or routing data and every
//     output write comes after that wait.
// Every sum has a fixed order: the result is bit-for-bit repeatable.  Every
// mbarrier wait is bounded; a wait that runs out records an error word and
// the CTA winds down (the producer first lets its copies in flight land).
#include <cooperative_groups.h>

#include "wo_bounds.cuh"
#include "wo_common.cuh"
#include "wo_internal.h"
#include "wo_sm100.cuh"
#include "wo_stream.h"
#include "wo_tmap.h"

namespace wo {
namespace {

namespace cg = cooperative_groups;
using namespace sm100;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Stage geometry of a configuration (k per stage = TPS packed tiles).
template <int BITS, int MT, int NW, int TPS>
struct StageGeom {
    static constexpr int KT = Geom<BITS>::KT;
    static constexpr int ROWS = 8 * MT;
    static constexpr int KSTAGE = TPS * KT;          // 64 or 128
    static constexpr int NHALF = KSTAGE / 64;        // activation boxes of 64 k
    static constexpr int A_BOX = ROWS * 128;         // one swizzled box: ROWS x 128 bytes
    static constexpr int A_BYTES = NHALF * A_BOX;
    static constexpr int W_BYTES = 2 * NW * TPS * kTileBytes;
    static constexpr int TX = A_BYTES + W_BYTES;     // bytes a stage receives
    static constexpr int STAGE = (TX + 1023) / 1024 * 1024;
};

__host__ inline int stage_bytes_host(int bits, int mt, int nw, int tps)
{
    const int kt = bits == 8 ? 32 : 64;
    const int tx = (tps * kt / 64) * 8 * mt * 128 + 2 * nw * tps * kTileBytes;
    return (tx + 1023) / 1024 * 1024;
}

// Tiles per stage of each configuration.  Consumer warps: 15 for the MoE
// experts (16 warps with the producer, so the register file splits evenly
// across the 4 schedulers), 8 or 4 for the plain GEMM (chosen by the plan).
__host__ __device__ inline int stream_tps(int mt, int bits, int out)
{
    const int k_stage = (out != OUT_PLAIN || mt >= 4) ? 64 : 128;
    return k_stage / (bits == 8 ? 32 : 64);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
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

// Consumer-warp block assignment: plain and fp32 outputs own blocks 2v and
// 2v + 1 of the weight (v = global warp index); the gated output owns gate
// block v and its up block v + inter / 16.
template <int OUT>
__device__ __forceinline__ void warp_blocks(const StreamParams& p, int v, int (&blk)[2], bool& active)
{
    if constexpr (OUT == OUT_GATED) {
        blk[0] = v;
        blk[1] = v + p.inter / 16;
        active = v < p.inter / 16;
    } else {
        blk[0] = 2 * v;
        blk[1] = 2 * v + 1;
        active = 2 * v + 1 < p.N / 16;
    }
}

// Scale (8-bit) and bias of the plain output's four channels per lane,
// blk[r] * 16 + g + 8 h.  They are inputs, so the CTA reads them at its
// start, before waiting for the previous grid, and their load latency stays
// off the end of the kernel.
struct PlainEpi {
    float s[2][2], b[2][2];
};

template <int ACT, bool GROUPED>
__device__ __forceinline__ PlainEpi load_plain_epi(const StreamParams& p, const int (&blk)[2],
                                                   const uint16_t* sx, int lane)
{
    PlainEpi e;
    const int g = lane >> 2;
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int ch = blk[r] * 16 + g + 8 * h;
            const bool ok = in_bounds(ch < p.N, 0x101);
            e.s[r][h] = GROUPED || !ok ? 1.f : to_f32<ACT>(ld_nc_u16(sx + ch));
            e.b[r][h] = p.bias && ok ? to_f32<ACT>(ld_nc_u16(p.bias + ch)) : 0.f;
        }
    return e;
}

// Output of one warp's accumulators: element q of (r, j) is channel
// blk[r] * 16 + g + 8 (q >> 1), row 8 j + 2 t + (q & 1) of the pass.
template <int ACT, int MT, int OUT, bool GROUPED>
__device__ __forceinline__ void stream_epilogue(const StreamParams& p, const float (&acc)[2][MT][4],
                                                const int (&blk)[2], int prow0, int rows,
                                                const uint16_t* sx, const PlainEpi& pe, int lane)
{
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int rr = 8 * j + 2 * t + (q & 1);
            if (rr >= rows)
                continue;
            const size_t row = (size_t)(prow0 + rr);
            if constexpr (OUT == OUT_GATED) {
                const int ch0 = blk[0] * 16 + g + 8 * (q >> 1);
                const int ch1 = blk[1] * 16 + g + 8 * (q >> 1);
                if (!in_bounds(ch0 < p.inter && ch1 < p.N && row < (size_t)p.a_rows_total, 0x102))
                    continue;
                const float gate = acc[0][j][q] * to_f32<ACT>(ld_nc_u16(sx + ch0));
                const float up = acc[1][j][q] * to_f32<ACT>(ld_nc_u16(sx + ch1));
                p.C[row * p.inter + ch0] = from_f32<ACT>(gate / (1.f + expf(-gate)) * up);
            } else {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int ch = blk[r] * 16 + g + 8 * (q >> 1);
                    if (!in_bounds(ch < p.N && row < (size_t)p.a_rows_total, 0x103))
                        continue;
                    float v = acc[r][j][q];
                    if constexpr (OUT == OUT_PLAIN) {
                        if constexpr (!GROUPED)
                            v *= pe.s[r][q >> 1];
                        if (p.bias)
                            v += pe.b[r][q >> 1];
                        p.C[row * p.N + ch] = from_f32<ACT>(v);
                    } else {
                        if constexpr (!GROUPED)
                            v *= to_f32<ACT>(ld_nc_u16(sx + ch));
                        p.Y[row * p.N + ch] = v;
                    }
                }
            }
        }
    }
}

template <int BITS, int ACT, int MT, int NW, int OUT, int TPS>
__global__ void __launch_bounds__((NW + 1) * 32)
    stream_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                  const StreamParams p)
{
    using SG = StageGeom<BITS, MT, NW, TPS>;
    constexpr int KT = SG::KT;
    constexpr int KS = Geom<BITS>::KSTEPS;
    constexpr bool GROUPED = BITS == 4;
    constexpr int ROWS = SG::ROWS;
    constexpr int NV = 2 * MT * 4;  // accumulator values per lane
    // decode rows (m <= 16): split each block's mma chain over even / odd k-steps
    constexpr bool DUAL = !GROUPED && OUT == OUT_PLAIN && MT <= 2;
    // full stages load all their weight tiles before the first mma step
    // (decode sizes only: more rows would spill the accumulators)
    constexpr bool LOADS_FIRST = MT <= 2;
    // ... and their activation fragments too
    constexpr bool ACT_FIRST = LOADS_FIRST && MT == 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled activation boxes
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    // k split across the cluster: rank r finishes the consumer warps w with
    // w % splits == r.  pbuf holds, per such warp, one slot per rank that the
    // ranks push their partial sums into; redbar counts the pushes.
    const int splits = p.splits;
    const int fin_warps = (NW + splits - 1) / splits;  // warps a rank finishes, at most
    float* pbuf = reinterpret_cast<float*>(smem + (size_t)S * SG::STAGE);
    const size_t pbuf_floats = splits > 1 ? (size_t)fin_warps * splits * 32 * NV : 0;
    uint64_t* full = reinterpret_cast<uint64_t*>(pbuf + pbuf_floats);
    uint64_t* empty = full + S;
    uint64_t* redbar = empty + S;
    int* abort_flag = reinterpret_cast<int*>(redbar + 1);
    uint16_t* s_sm = reinterpret_cast<uint16_t*>(abort_flag + 4);
    volatile int* abort = abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2;

    // Programmatic dependent launch: the next grid may start now (it waits
    // for this one before touching its outputs); this grid waits for the
    // previous one before reading anything that grid may produce.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool moe = p.offsets != nullptr;
    if (moe)  // the row ranges come from the routing kernel
        asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- work of this CTA ----
    const int e = moe ? blockIdx.y : 0;
    const int row0 = moe ? p.offsets[e] : 0;
    const int rows_total = moe ? p.offsets[e + 1] - row0 : p.m;
    const int c0 = moe ? 0 : blockIdx.y * p.kt_per_split;
    const int c1 = moe ? p.ktiles : min(c0 + p.kt_per_split, p.ktiles);
    const int nst = (c1 - c0 + TPS - 1) / TPS;
    const int passes = (rows_total + ROWS - 1) / ROWS;
    const uint16_t* sx = p.scales + (size_t)e * p.s_stride;

    // consumer warps of this CTA whose pushes this rank receives
    const int rank = splits > 1 ? (int)cg::this_cluster().block_rank() : 0;
    int fin_active = 0;
    if (splits > 1)
        for (int w = rank; w < NW; w += splits) {
            int b_[2];
            bool act_;
            warp_blocks<OUT>(p, blockIdx.x * NW + w, b_, act_);
            fin_active += act_ ? 1 : 0;
        }

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        if (fin_active > 0)
            mbar_init(redbar, (uint32_t)(fin_active * splits * 32));
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
    }
    __syncthreads();
    if (splits > 1)
        cluster_arrive_relaxed();  // barrier inits visible cluster-wide before any push
    if (p.splits == 1 && (rows_total <= 0 || nst <= 0))
        return;  // a whole CTA with nothing to do (an expert without rows)

    PlainEpi pe{};  // consumer lanes: their channels' scale and bias
    if (warp == NW) {
        // ================= producer (one thread) =================
        if (lane == 0) {
            // first weight block row of this CTA (and of its up blocks)
            const int brow = e * p.blocks_per_expert;
            const int wrow0 = OUT == OUT_GATED ? brow + blockIdx.x * NW : brow + blockIdx.x * 2 * NW;
            const int wrow1 = brow + p.inter / 16 + blockIdx.x * NW;
            auto load_w = [&](int s, int kt_s) {
                uint8_t* wdst = smem + (size_t)s * SG::STAGE + SG::A_BYTES;
                tma_load_2d(wdst, &tmW, &full[s], kt_s * 64, wrow0);
                if constexpr (OUT == OUT_GATED)
                    tma_load_2d(wdst + NW * TPS * kTileBytes, &tmW, &full[s], kt_s * 64, wrow1);
            };
            auto load_a = [&](int s, int kt_s, int prow0) {
                uint8_t* stage = smem + (size_t)s * SG::STAGE;
#pragma unroll
                for (int h = 0; h < SG::NHALF; ++h)
                    tma_load_2d(stage + h * SG::A_BOX, &tmA, &full[s], kt_s * KT + 64 * h, prow0);
            };
            // the first ring's weights do not depend on the previous grid:
            // fetch them before waiting for it
            const int pre = moe ? 0 : min(S, nst);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], SG::TX);
                load_w(i, c0 + i * TPS);
            }
            if (!moe)
                asm volatile("griddepcontrol.wait;" ::: "memory");
            int it = 0;
            bool ok = true;
            for (int pass = 0; pass < passes && ok; ++pass) {
                const int prow0 = row0 + pass * ROWS;
                for (int st = 0; st < nst; ++st, ++it) {
                    const int s = it % S;
                    const int kt_s = c0 + st * TPS;
                    if (it < pre) {  // weights already in flight
                        load_a(s, kt_s, prow0);
                        continue;
                    }
                    ok = mbar_wait_bounded(&empty[s], ((it / S) & 1) ^ 1, abort, p.err, 11, kWaitLimitNs);
                    if (!ok)
                        break;
                    mbar_arrive_expect_tx(&full[s], SG::TX);
                    load_a(s, kt_s, prow0);
                    load_w(s, kt_s);
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA winds down
                volatile int never = 0;
                for (int i = it - S > 0 ? it - S : 0; i < it; ++i)
                    mbar_wait_bounded(&full[i % S], (i / S) & 1, &never, nullptr, 0, kWaitLimitNs);
            }
        }
    } else {
        // ================= consumers =================
        int blk[2];
        bool active;
        warp_blocks<OUT>(p, blockIdx.x * NW + warp, blk, active);
        if (OUT == OUT_PLAIN && active)
            pe = load_plain_epi<ACT, GROUPED>(p, blk, sx, lane);
        // 4-bit: this warp's 32 channels' scales and zeros over its k range
        uint16_t* ws_s = s_sm + (size_t)warp * 2 * 32 * p.g_span;
        uint16_t* ws_z = ws_s + 32 * p.g_span;
        const int g_lo = GROUPED ? c0 / p.tiles_per_group : 0;
        if (GROUPED && active) {
            const int gc = (c1 - 1) / p.tiles_per_group - g_lo + 1;
            // batches of 8 per lane: all 16 loads in flight before the stores
            // (one memory round trip per batch, not two per value)
            constexpr int NB = 8;
            for (int base = 0; base < 32 * gc; base += 32 * NB) {
                uint16_t sv[NB], zv[NB];
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int idx = base + b * 32 + lane;
                    sv[b] = zv[b] = 0;
                    if (idx < 32 * gc) {
                        const int ch = idx / gc, gg = idx % gc;
                        const size_t src = (size_t)(blk[ch >> 4] * 16 + (ch & 15)) * p.G + g_lo + gg;
                        if (in_bounds(src < (size_t)p.N * p.G, 0x104)) {
                            sv[b] = ld_nc_u16(sx + src);
                            if (p.zeros)
                                zv[b] = ld_nc_u16(p.zeros + src);
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int idx = base + b * 32 + lane;
                    if (idx < 32 * gc) {
                        const int ch = idx / gc, gg = idx % gc;
                        ws_s[ch * p.g_span + gg] = sv[b];
                        ws_z[ch * p.g_span + gg] = zv[b];
                    }
                }
            }
            __syncwarp();
        }
        // per-lane shared-memory offsets: this warp's two weight block rows,
        // and the ldmatrix row of this lane (lane L gives row L & 7 of
        // matrix L >> 3; matrices alternate k halves, then the next 8 rows)
        const int wr0 = OUT == OUT_GATED ? warp : 2 * warp;
        const int wr1 = OUT == OUT_GATED ? NW + warp : 2 * warp + 1;
        const uint32_t w_lane0 = (uint32_t)(SG::A_BYTES + wr0 * TPS * kTileBytes + lane * 16);
        const uint32_t w_lane1 = (uint32_t)(SG::A_BYTES + wr1 * TPS * kTileBytes + lane * 16);
        const uint32_t a_row = (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * 128);
        const uint32_t a_hi = (uint32_t)((lane >> 3) & 1);
        const uint32_t a_xor = (uint32_t)(lane & 7);

        int it = 0;
        bool ok = true;
        float acc[2][MT][4];
        for (int pass = 0; pass < passes && ok; ++pass) {
            const int rows = min(ROWS, rows_total - pass * ROWS);
            float gp[2][MT][4];
            float rs[MT][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int j = 0; j < MT; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[r][j][q] = 0.f;
                        gp[r][j][q] = 0.f;
                    }
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    rs[j][q] = 0.f;

            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % S;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (it / S) & 1, abort, p.err,
                                                                12, kWaitLimitNs));
                if (!ok)
                    break;
                const int kt_s = c0 + st * TPS;
                const int ntile = min(TPS, c1 - kt_s);
                const uint32_t stage = smem_addr(smem + (size_t)s * SG::STAGE);
                // activation fragments of rows 8j..8j+7 for k step ks of tile
                // tl (ldmatrix through the 128-byte swizzle; rows past the
                // valid count only feed output columns that are never stored)
                auto load_b = [&](int tl, int ks, uint32_t (&b)[MT][2]) {
                    const int kk = tl * KT + 16 * ks;  // k within the stage
                    const uint32_t box = stage + (uint32_t)((kk >> 6) * SG::A_BOX);
                    const uint32_t chunk = (uint32_t)((kk & 63) >> 3);
                    const uint32_t col = (((chunk + a_hi) ^ a_xor) << 4);
                    if constexpr (MT == 1) {
                        ldsm_x2(box + a_row + col, b[0][0], b[0][1]);
                    } else {
#pragma unroll
                        for (int jp = 0; jp < MT / 2; ++jp)
                            if (jp == 0 || 16 * jp < rows)  // rows >= 1
                                ldsm_x4(box + a_row + (uint32_t)(jp * 16 * 128) + col, b[2 * jp][0],
                                        b[2 * jp][1], b[2 * jp + 1][0], b[2 * jp + 1][1]);
                    }
                };
                // one packed tile of each of the warp's two blocks: mma steps
                // (and, 4-bit, the group's scale and zero when it ends);
                // bpre: the tile's activation fragments, loaded earlier, or null
                auto do_tile = [&](const uint4 v0, const uint4 v1, int tl, const uint32_t (*bpre)[MT][2]) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        uint32_t a0[4], a1[4];
                        tile_frag<BITS, ACT>(v0, ks, a0);
                        tile_frag<BITS, ACT>(v1, ks, a1);
                        uint32_t b[MT][2];
                        if (bpre) {
#pragma unroll
                            for (int j = 0; j < MT; ++j)
                                b[j][0] = bpre[ks][j][0], b[j][1] = bpre[ks][j][1];
                        } else {
                            load_b(tl, ks, b);
                        }
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            if (j == 0 || 8 * j < rows) {  // warp-uniform; rows >= 1
                                if constexpr (GROUPED) {
                                    mma16816<ACT>(gp[0][j], a0, b[j][0], b[j][1]);
                                    mma16816<ACT>(gp[1][j], a1, b[j][0], b[j][1]);
                                    const uint32_t one = ones_x2<ACT>();
                                    const uint32_t ones[4] = {one, one, one, one};
                                    mma16816<ACT>(rs[j], ones, b[j][0], b[j][1]);
                                } else {
                                    // DUAL: odd k-steps into a second set (gp), so
                                    // two independent mma chains per block
                                    float (&d0)[4] = (DUAL && (ks & 1)) ? gp[0][j] : acc[0][j];
                                    float (&d1)[4] = (DUAL && (ks & 1)) ? gp[1][j] : acc[1][j];
                                    mma16816<ACT>(d0, a0, b[j][0], b[j][1]);
                                    mma16816<ACT>(d1, a1, b[j][0], b[j][1]);
                                }
                            }
                        }
                    }
                    if constexpr (GROUPED) {
                        const int ktile = kt_s + tl;
                        if (((ktile + 1) % p.tiles_per_group == 0) || (ktile + 1 == c1)) {
                            const int gl = ktile / p.tiles_per_group - g_lo;
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int ch = r * 16 + g;
                                const float s_lo = to_f32<ACT>(ws_s[ch * p.g_span + gl]);
                                const float s_hi = to_f32<ACT>(ws_s[(ch + 8) * p.g_span + gl]);
                                const float z_lo = to_f32<ACT>(ws_z[ch * p.g_span + gl]);
                                const float z_hi = to_f32<ACT>(ws_z[(ch + 8) * p.g_span + gl]);
#pragma unroll
                                for (int j = 0; j < MT; ++j) {
                                    acc[r][j][0] = fmaf(s_lo, gp[r][j][0], fmaf(z_lo, rs[j][0], acc[r][j][0]));
                                    acc[r][j][1] = fmaf(s_lo, gp[r][j][1], fmaf(z_lo, rs[j][1], acc[r][j][1]));
                                    acc[r][j][2] = fmaf(s_hi, gp[r][j][2], fmaf(z_hi, rs[j][2], acc[r][j][2]));
                                    acc[r][j][3] = fmaf(s_hi, gp[r][j][3], fmaf(z_hi, rs[j][3], acc[r][j][3]));
#pragma unroll
                                    for (int q = 0; q < 4; ++q)
                                        gp[r][j][q] = 0.f;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < MT; ++j)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    rs[j][q] = 0.f;
                        }
                    }
                };
                if (active) {
                    if (LOADS_FIRST && ntile == TPS) {
                        // a full stage: every weight load first, so that the
                        // conversions and mma steps of one tile overlap the
                        // loads of the next (one basic block for all tiles)
                        uint4 v0[TPS], v1[TPS];
#pragma unroll
                        for (int tl = 0; tl < TPS; ++tl) {
                            v0[tl] = lds128(stage + w_lane0 + (uint32_t)(tl * kTileBytes));
                            v1[tl] = lds128(stage + w_lane1 + (uint32_t)(tl * kTileBytes));
                        }
                        if constexpr (ACT_FIRST) {
                            uint32_t bb[TPS][KS][MT][2];
#pragma unroll
                            for (int tl = 0; tl < TPS; ++tl)
#pragma unroll
                                for (int ks = 0; ks < KS; ++ks)
                                    load_b(tl, ks, bb[tl][ks]);
#pragma unroll
                            for (int tl = 0; tl < TPS; ++tl)
                                do_tile(v0[tl], v1[tl], tl, bb[tl]);
                        } else {
#pragma unroll
                            for (int tl = 0; tl < TPS; ++tl)
                                do_tile(v0[tl], v1[tl], tl, nullptr);
                        }
                    } else {
#pragma unroll
                        for (int tl = 0; tl < TPS; ++tl)
                            if (tl < ntile)
                                do_tile(lds128(stage + w_lane0 + (uint32_t)(tl * kTileBytes)),
                                        lds128(stage + w_lane1 + (uint32_t)(tl * kTileBytes)), tl, nullptr);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[s]);
            }
            if constexpr (DUAL) {
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int j = 0; j < MT; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[r][j][q] += gp[r][j][q];
            }
            if (ok && p.splits == 1 && active) {
                asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs: after the previous grid
                stream_epilogue<ACT, MT, OUT, GROUPED>(p, acc, blk, row0 + pass * ROWS, rows, sx, pe, lane);
            }
        }
        if (splits > 1 && active) {
            // push this warp's partial sums into slot (w / splits, rank) of
            // rank w % splits, then arrive there (zeros if the loop gave up)
            cluster_wait();
            const uint32_t dst_rank = (uint32_t)(warp % splits);
            const int slot = (warp / splits) * splits + rank;
            const uint32_t dst =
                mapa_shared(smem_addr(pbuf + ((size_t)slot * 32 + lane) * NV), dst_rank);
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int j = 0; j < MT; ++j)
                    st_cluster_v4(dst + (uint32_t)((r * MT + j) * 16),
                                  ok ? make_float4(acc[r][j][0], acc[r][j][1], acc[r][j][2], acc[r][j][3])
                                     : make_float4(0.f, 0.f, 0.f, 0.f));
            mbar_arrive_cluster(mapa_shared(smem_addr(redbar), dst_rank));

            if (warp % splits == rank) {
                // finish this warp's channels: every rank's partials, in rank order
                // waits for every push even after an abort elsewhere, so that no rank
                // writes into this CTA's shared memory after it has exited
                volatile int never = 0;
                const bool got = __all_sync(0xffffffffu, mbar_wait_bounded<true>(redbar, 0, &never, p.err,
                                                                                13, kWaitLimitNs)) &&
                                 !*abort;
                if (got) {
                    const float4* src = reinterpret_cast<const float4*>(pbuf) +
                                        ((size_t)(warp / splits) * splits * 32 + lane) * (NV / 4);
                    float4 sum[NV / 4];
#pragma unroll
                    for (int v = 0; v < NV / 4; ++v)
                        sum[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int rk = 0; rk < splits; ++rk) {
#pragma unroll
                        for (int v = 0; v < NV / 4; ++v) {
                            const float4 x = src[(size_t)rk * 32 * (NV / 4) + v];
                            sum[v].x += x.x;
                            sum[v].y += x.y;
                            sum[v].z += x.z;
                            sum[v].w += x.w;
                        }
                    }
                    float fin[2][MT][4];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            fin[r][j][0] = sum[r * MT + j].x;
                            fin[r][j][1] = sum[r * MT + j].y;
                            fin[r][j][2] = sum[r * MT + j].z;
                            fin[r][j][3] = sum[r * MT + j].w;
                        }
                    asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs: after the previous grid
                    stream_epilogue<ACT, MT, OUT, GROUPED>(p, fin, blk, row0, min(ROWS, rows_total), sx, pe, lane);
                }
            }
        }
    }
}

}  // namespace

// ------------------------------------------------------------------ host ---

namespace {

template <int BITS, int ACT, int MT, int NW, int OUT, int TPS>
cudaError_t launch_t(const StreamParams& p, const StreamPlan& plan, int grid_y, cudaStream_t s)
{
    using SG = StageGeom<BITS, MT, NW, TPS>;
    CUtensorMap ma, mw;
    if (!make_tmap_2d(&ma, ACT == ACT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      p.A, (uint64_t)p.K, (uint64_t)p.a_rows_total, (uint64_t)p.K * 2, 64, SG::ROWS,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // packed weights: one row per 16-channel block, 512 bytes per k tile
    if (!make_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT64, p.B, (uint64_t)p.ktiles * 64,
                      (uint64_t)p.w_block_rows, (uint64_t)p.ktiles * kTileBytes, TPS * 64,
                      OUT == OUT_GATED ? NW : 2 * NW, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = stream_kernel<BITS, ACT, MT, NW, OUT, TPS>;
    static int smem_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || smem_set[dev] < (int)plan.smem) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)plan.smem)) != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            smem_set[dev] = (int)plan.smem;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid_x, grid_y);
    cfg.blockDim = dim3((NW + 1) * 32);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (plan.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = plan.splits;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, ma, mw, p);
}

// plain output: decode configurations (must agree with plan_stream / stream_tps)
template <int BITS, int ACT, int NW>
cudaError_t launch_plain_nw(const StreamParams& p, const StreamPlan& plan, int grid_y, cudaStream_t s)
{
    constexpr int T128 = BITS == 8 ? 4 : 2;  // tiles of 128 k
    constexpr int T64 = BITS == 8 ? 2 : 1;   // tiles of 64 k
    switch (plan.mt) {
    case 1: return launch_t<BITS, ACT, 1, NW, OUT_PLAIN, T128>(p, plan, grid_y, s);
    case 2: return launch_t<BITS, ACT, 2, NW, OUT_PLAIN, T128>(p, plan, grid_y, s);
    case 4: return launch_t<BITS, ACT, 4, NW, OUT_PLAIN, T64>(p, plan, grid_y, s);
    default: return launch_t<BITS, ACT, 8, NW, OUT_PLAIN, T64>(p, plan, grid_y, s);
    }
}

template <int BITS, int ACT>
cudaError_t launch_plain(const StreamParams& p, const StreamPlan& plan, int grid_y, cudaStream_t s)
{
    return plan.nw == 4 ? launch_plain_nw<BITS, ACT, 4>(p, plan, grid_y, s)
                        : launch_plain_nw<BITS, ACT, 8>(p, plan, grid_y, s);
}

constexpr int kMaxCluster = 8;

}  // namespace

// m: rows per launch (<= 64; the MoE uses 64).  out: OUT_*.  inter: gated
// channel distance.  The plan sizes the ring of stages to the shared memory
// budget (two CTAs per SM for decode, one for the MoE experts) and splits k
// across a cluster when the channels alone give too few CTAs; a split covers
// whole stages.
StreamPlan plan_stream(int m, int n, int k, int group, int bits, int out, int inter)
{
    StreamPlan P{};
    const int rows = m < 64 ? m : 64;
    P.mt = out != OUT_PLAIN ? 8 : rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;
    const int tps = stream_tps(P.mt, bits, out);
    const int KT = bits == 8 ? 32 : 64;
    const int ktiles = k / KT;
    const int tpg = group / KT;
    const int nst_all = (ktiles + tps - 1) / tps;
    const int warps_total = out == OUT_GATED ? inter / 16 : n / 32;
    if (out != OUT_PLAIN) {
        P.nw = 15;
    } else {
        // 8 consumer warps (256 channels per CTA) unless that leaves SMs idle
        // even with the largest k split; then 4 (128 channels per CTA)
        int cap = nst_all / 2;
        if (cap > kMaxCluster)
            cap = kMaxCluster;
        if (cap < 1)
            cap = 1;
        const int ctas8 = (warps_total + 7) / 8 * cap;
        P.nw = ctas8 >= num_sms() ? 8 : 4;
    }
    P.grid_x = (warps_total + P.nw - 1) / P.nw;
    const size_t budget = out == OUT_PLAIN ? 110 * 1024 : 215 * 1024;
    const size_t stage = (size_t)stage_bytes_host(bits, P.mt, P.nw, tps);
    const int nst_total = nst_all;
    int splits = 1;
    if (out == OUT_PLAIN) {
        // as many k splits as keep the grid within one resident wave (two
        // CTAs per SM): a second, partial wave would leave SMs idle
        splits = (2 * num_sms()) / P.grid_x;
        int cap = nst_total / 2;  // at least two stages per CTA
        if (cap > kMaxCluster)
            cap = kMaxCluster;
        if (splits > cap)
            splits = cap;
        if (splits < 1)
            splits = 1;
    }
    for (; splits <= kMaxCluster; ++splits) {
        const int kps = (nst_total + splits - 1) / splits * tps;  // whole stages
        const int nsplit = (ktiles + kps - 1) / kps;                 // CTAs along k
        const int gspan = bits == 4 ? (kps + tpg - 1) / tpg + 1 : 0;
        const size_t sz = (size_t)P.nw * 2 * 32 * gspan * 2;
        // push buffer of the cluster reduction (see stream_kernel)
        const size_t pb = nsplit > 1 ? (size_t)((P.nw + nsplit - 1) / nsplit) * nsplit * 32 * (8 * P.mt) * 4 : 0;
        const size_t fixed = 1024 + pb + sz + 16 + 2 * 8 * 8 + 8 + 128;
        if (fixed + 2 * stage > budget)
            continue;  // not even two stages fit: split k further
        int stages = (int)((budget - fixed) / stage);
        if (stages > 8)
            stages = 8;
        if (out == OUT_PLAIN && stages > kps / tps) {
            // no more stages than the CTA's k range has (every weight is then
            // fetched before the wait for the previous grid), keeping shared
            // memory free for the next grid's CTAs
            stages = kps / tps;
        }
        P.splits = nsplit;
        P.kt_per_split = kps;
        P.stages = stages;
        P.g_span = gspan;
        P.tps = tps;
        P.smem = 1024 + (size_t)stages * stage + pb + 2 * 8 * (size_t)stages + 8 + 16 + sz;
        P.valid = out == OUT_PLAIN || P.splits == 1;
        return P;
    }
    P.valid = false;
    return P;
}

cudaError_t launch_stream(const StreamParams& p, const StreamPlan& plan, int bits, int act, int out,
                          int grid_y, cudaStream_t s)
{
    if (out == OUT_PLAIN) {
        if (bits == 8)
            return act == WO_F16 ? launch_plain<8, ACT_F16>(p, plan, grid_y, s)
                                 : launch_plain<8, ACT_BF16>(p, plan, grid_y, s);
        return act == WO_F16 ? launch_plain<4, ACT_F16>(p, plan, grid_y, s)
                             : launch_plain<4, ACT_BF16>(p, plan, grid_y, s);
    }
    if (bits != 8)
        return cudaErrorInvalidValue;
    if (out == OUT_GATED)
        return act == WO_F16 ? launch_t<8, ACT_F16, 8, 15, OUT_GATED, 2>(p, plan, grid_y, s)
                             : launch_t<8, ACT_BF16, 8, 15, OUT_GATED, 2>(p, plan, grid_y, s);
    return act == WO_F16 ? launch_t<8, ACT_F16, 8, 15, OUT_F32, 2>(p, plan, grid_y, s)
                         : launch_t<8, ACT_BF16, 8, 15, OUT_F32, 2>(p, plan, grid_y, s);
}

size_t stream_workspace_bytes() { return kWsHeader; }

bool stream_supported(int m, int n, int k, int group, int bits)
{
    return m >= 1 && m <= 64 && plan_stream(m, n, k, group, bits, OUT_PLAIN, 0).valid;
}

cudaError_t launch_stream_gemm(const GemmArgs& a, cudaStream_t s)
{
    const StreamPlan P = plan_stream(a.m, a.n, a.k, a.group, a.bits, OUT_PLAIN, 0);
    if (!P.valid)
        return cudaErrorInvalidValue;
    StreamParams p{};
    p.A = static_cast<const uint16_t*>(a.A);
    p.a_rows_total = a.m;
    p.m = a.m;
    p.B = a.B;
    p.w_block_rows = a.n / 16;
    p.blocks_per_expert = 0;
    p.scales = static_cast<const uint16_t*>(a.scales);
    p.zeros = static_cast<const uint16_t*>(a.zeros);
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.N = a.n;
    p.K = a.k;
    const int KT = a.bits == 8 ? 32 : 64;
    p.ktiles = a.k / KT;
    p.G = a.k / a.group;
    p.tiles_per_group = a.group / KT;
    p.kt_per_split = P.kt_per_split;
    p.splits = P.splits;
    p.stages = P.stages;
    p.g_span = P.g_span;
    p.C = static_cast<uint16_t*>(a.C);
    p.err = static_cast<unsigned*>(a.ws);
    return launch_stream(p, P, a.bits, a.act, OUT_PLAIN, P.splits, s);
}

unsigned bounds_take_stream() { return bounds_take_local(); }

}  // namespace wo
