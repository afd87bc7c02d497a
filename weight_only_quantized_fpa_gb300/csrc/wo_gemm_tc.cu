// wo_gemm_tc.cu -- tensor-core kernel for large m:
//
//   C[m, n] = A[m, k] . dequant(B)^T + bias[n]
//
// The acext User Guide (v1.7) 1.3.4 describes fpA-intB as integer weights
// that are turned back into floating point before the multiply: here that
// happens per 64-wide k block on chip, right before tcgen05 MMAs that
// accumulate in tensor memory.
//
// Persistent kernel: one CTA per SM walks output tiles of MS x 128 (m) by BN
// (n) in the order tile_coords gives; tc_shape picks the shape (256 x 256
// unless narrower tiles fill the SMs in fewer waves, so that every A and
// code byte fetched from L2 feeds the most FLOPs).  With MS = 2 two M=128
// MMAs per k step share one dequantised B tile.  Roles (16 warps):
//   warp 0       TMA producer of the packed code tiles (BN channels x 64 k)
//                into the code ring;
//   warp 2       TMA producer of the A tiles (128 x 64, 128-byte swizzle)
//                into the A ring;
//   warp 1       allocates the TMEM accumulators (two when they fit); one lane
//                issues the MMAs (M=128, N=BN, K=16, four per k block) and
//                commits them to the ring barriers and, at a tile's end, to
//                the accumulator's "full" barrier;
//   warps 4-7    epilogue: drain a finished accumulator (tcgen05.ld, one TMEM
//                lane quadrant per warp), apply scale[n] (8-bit) or the
//                activation row scale (4-bit), add bias, round once, store C,
//                and hand the accumulator back -- while the MMAs already run
//                the next tile into the other accumulator; with one
//                accumulator (256 x 256, 8-bit) the dequantisation warps,
//                idle until it is handed back, drain two thirds of it;
//   warps 8-15   dequantisation: code ring -> registers -> exact (q - 128)
//                for 8-bit codes or fp16 round((q - 8) * s' + z') for 4-bit
//                group codes, written with stmatrix into the operand ring in
//                the K-major 128-byte-swizzled layout the MMA reads (4-bit
//                scale and zero pairs are loaded into registers a few k
//                blocks ahead).
// Every mbarrier wait is bounded: a wait that runs out records an error word
// in the workspace header and the CTA winds down (see the abort path).
//
// Programmatic dependent launch: a CTA sets up (barriers, TMEM, tensor-map
// prefetch) and starts fetching its weight codes while the previous kernel
// on the stream is still finishing; the roles that touch anything that
// kernel may produce or read -- activations (warp 2), the 4-bit prepass's
// pre-scaled scales (dequantisation warps), outputs, row scales and the
// workspace (epilogue, drain helpers) -- first wait for it to complete.
//
// Operand types: 8-bit codes run the MMA in the activation dtype, in which
// q - 128 is exact.  4-bit codes run it in fp16, with both operands brought
// into fp16's range by powers of two that the epilogue undoes: a prepass
// (tc_prep_kernel) picks for every output channel n a power of two 2^E_n
// that puts the channel's largest |scale| or |zero| in [2^10, 2^11) and
// writes the channel's scales and zeros times 2^-E_n as fp16 pairs
// (s', z'); for bf16 activations it also converts A to fp16 with a
// per-row power of two 2^E_r (row maximum in [2^14, 2^15); exact for bf16
// values within 2^24 of the row maximum).  The weight is then
// fp16 round((q - 8) * s' + z'), one fused multiply-add per pair from the
// exact fp16 (q - 8), at most 9 * 2^11 in magnitude, and the epilogue
// scales the fp32 sum by 2^(E_r + E_n).  So any finite bf16 scale, zero and
// activation is in range; only values more than 2^24 below their channel's
// (or row's) largest fall into fp16's subnormals, where their share of the
// sum is below the output's rounding.
#include "wo_bounds.cuh"
#include "wo_common.cuh"
#include "wo_internal.h"
#include "wo_sm100.cuh"
#include "wo_tmap.h"

namespace wo {
namespace {

using namespace sm100;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 512;       // 16 warps
constexpr int kEpilogueWarp0 = 4;   // warps 4..7
constexpr int kDequantWarp0 = 8;    // warps 8..15
constexpr int kDequantWarps = 8;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// MS: M=128 sub-tiles per output tile.  With MS = 2 (256 x BN tiles) two
// MMAs share each dequantised B tile, halving the dequantisation per FLOP.
template <int BITS, int BN, int MS = 1>
struct TcCfg {
    static constexpr int A_SUB = BM * BK * 2;                    // 16 KiB per sub-tile
    static constexpr int A_BYTES = MS * A_SUB;
    static constexpr int C_BYTES = BN * BK * BITS / 8;           // packed codes of a k block
    static constexpr int B_BYTES = BN * BK * 2;                  // dequantised operand
    // 256 x 256 8-bit tiles: the A tiles' TMA round trip paces the MMAs, so
    // the A ring gets four stages and the code ring, whose 16 KiB stages
    // arrive early enough, two.  4-bit tiles keep three and three: their
    // dequantisation reads the group scales through L1, which a fuller
    // shared memory would shrink.
    static constexpr int SA = MS == 2 ? (BN == 256 ? (BITS == 8 ? 4 : 3) : BITS == 4 ? 4 : 3) : BN == 256 ? 4 : 6;  // A ring
    static constexpr int SC = MS == 2 ? (BN == 256 ? (BITS == 8 ? 2 : 3) : 6) : (BITS == 8 ? 4 : 6) + (BN == 256 ? 0 : 2);  // codes
    static constexpr int S2 = MS == 2 && BN == 256 ? 2 : BN == 256 ? 3 : 4;  // operand ring stages
    static constexpr int TPN = BK / Geom<BITS>::KT;              // packed tiles per 16 rows
    static constexpr int NT = (BN / 16) * TPN;                   // packed tiles per k block
    static constexpr int R = NT / kDequantWarps;                 // tiles per dequant warp
    static constexpr int PF = 3;                                 // 4-bit scales loaded ahead
    // 128-row tiles (MS = 1) keep each accumulator as two partial sums, the
    // even and odd k blocks, issued by two MMA threads (one thread's per-k-
    // block work otherwise paces these tiles' k loop); the drain adds them.
    static constexpr int PARTS = MS == 1 ? 2 : 1;
    // accumulators of MS sub-tiles (x PARTS): two (the epilogue of one tile
    // overlaps the next tile's main loop) when they fit in the 512 TMEM
    // columns, else one
    static constexpr int NACC = 2 * MS * BN * PARTS <= 512 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = NACC * MS * BN * PARTS;
    static_assert(TMEM_COLS <= 512, "tensor memory");
    static constexpr int SMEM = SA * A_BYTES + SC * C_BYTES + S2 * B_BYTES;  // + barriers
    static_assert(NT % kDequantWarps == 0, "tiles per k block must split evenly");
    static_assert(SA <= 8 && SC <= 8 && S2 <= 4, "barrier arrays");
};

struct TcParams {
    int m, n, k;
    int num_kb;              // k / BK
    int m_tiles, n_tiles;    // output tiles along m and n
    const uint16_t* scales;  // 8-bit: [n]
    const uint32_t* sz;      // 4-bit: [n, G] fp16 pairs (s' low, z' high), pre-scaled by 2^-E_n
    const uint16_t* colscale;  // 4-bit: [n] 2^E_n as bf16 bits
    const uint16_t* bias;    // [n] or null
    const float* rowscale;   // 4-bit with a converted A: [m] powers of two; else null
    uint16_t* C;
    int G;                   // scale groups per channel row
    int group;               // codes per group
    int m_fast;              // tile walk: m fastest (else n fastest)
    int c_v8;                // C 32-byte aligned (and n % 16 == 0): 32-byte stores
    int splits;              // k split: units per output tile (1: none)
    float* partial;          // splits > 1: fp32 partial tiles, [tile * splits + s][h][BN / 32][128][32]
    size_t partial_floats;   // its extent (index checks of the debug build)
    unsigned* counters;      // splits > 1: per-tile arrival counters (kept at zero between calls)
    unsigned* err;           // workspace error word
};

struct Barriers {
    uint64_t fullA[8], emptyA[8];  // A ring (TMA -> MMA)
    uint64_t fullC[16], emptyC[16];  // code ring (TMA -> dequant warps)
    uint64_t full2[8], empty2[8];  // operand ring (dequant warps -> MMA)
    uint64_t tfull[2], tempty[2];  // the two TMEM accumulators (MMA <-> epilogue)
    uint64_t mma_done;             // every MMA issued has completed (teardown)
    uint32_t tmem_base;
    int abort;
    int is_last;                   // k split: this CTA reduces the tile
};

// Output tile `t` of the persistent walk.  The operand that is larger in
// bytes is streamed from HBM once: when A is the smaller one the walk goes m
// fastest (the CTAs running at the same time share each weight tile while
// every A row stays in L2), otherwise n fastest (they share A tiles while the
// weights stay in L2).
__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int bm, int bn, int& m0, int& n0)
{
    if (p.m_fast) {
        m0 = (t % p.m_tiles) * bm;
        n0 = (t / p.m_tiles) * bn;
    } else {
        m0 = (t / p.n_tiles) * bm;
        n0 = (t % p.n_tiles) * bn;
    }
}

// 4-bit: the pre-scaled (s', z') fp16 pairs of one dequant warp's tiles for
// one k block (channels g and g + 8 of each tile), loaded a few k blocks
// ahead of their use.
template <int BITS, int BN>
struct DqScales {
    static constexpr int R = BITS == 4 ? TcCfg<BITS, BN>::R : 1;
    uint32_t lo[R], hi[R];
};

template <int BITS, int BN>
__device__ __forceinline__ void load_scales(const TcParams& p, int n0, int kb, int dw, int lane,
                                            DqScales<BITS, BN>& c)
{
    if constexpr (BITS == 4) {
        using Cfg = TcCfg<BITS, BN>;
        const int g = lane >> 2;
        const int gi = (kb * BK) / p.group;
#pragma unroll
        for (int r = 0; r < Cfg::R; ++r) {
            const int nb = (dw + kDequantWarps * r) / Cfg::TPN;
            const int ch = n0 + nb * 16 + g;
            c.lo[r] = 0u;
            c.hi[r] = 0u;
            if (ch < p.n && in_bounds((size_t)(ch + 8) * p.G + gi < (size_t)p.n * p.G, 0x301)) {
                // n is a multiple of 16: row ch + 8 is in range too
                const size_t lo = (size_t)ch * p.G + gi;
                c.lo[r] = ld_nc_u32(p.sz + lo);
                c.hi[r] = ld_nc_u32(p.sz + lo + (size_t)8 * p.G);
            }
        }
    }
}

// Dequantise one warp's share of a k block: code stage at c_s -> operand
// stage at b_s.
template <int BITS, int OT, int ACT, int BN>
__device__ __forceinline__ void dequant_stage(uint32_t c_s, const DqScales<BITS, BN>& sc,
                                              uint32_t b_s, int dw, int lane)
{
    using Cfg = TcCfg<BITS, BN>;
    constexpr int KT = Geom<BITS>::KT;
    constexpr int KS = Geom<BITS>::KSTEPS;
    const int mi = lane >> 3, r8 = lane & 7;
    uint4 v[Cfg::R];
#pragma unroll
    for (int r = 0; r < Cfg::R; ++r)  // all shared loads first
        v[r] = lds128(c_s + (uint32_t)(dw + kDequantWarps * r) * kTileBytes + lane * 16);
#pragma unroll
    for (int r = 0; r < Cfg::R; ++r) {
        const int tile = dw + kDequantWarps * r;
        const int nb = tile / Cfg::TPN, tl = tile % Cfg::TPN;
        uint32_t slo = 0, shi = 0, zlo = 0, zhi = 0;
        if constexpr (BITS == 4) {  // s' and z' of channels g and g + 8, each doubled
            slo = prmt(sc.lo[r], 0u, 0x1010u);
            zlo = prmt(sc.lo[r], 0u, 0x3232u);
            shi = prmt(sc.hi[r], 0u, 0x1010u);
            zhi = prmt(sc.hi[r], 0u, 0x3232u);
        }
        // lane -> row address of stmatrix matrix mi: rows r8 (+8 for mi >= 2),
        // 16-byte chunk of 8 codes (+1 for mi odd); matrices 0 and 1 (and 2
        // and 3) are the two k chunks of the same rows, which the swizzle puts
        // in different banks
        const int row = nb * 16 + r8 + 8 * (mi >> 1);
        const uint32_t row_base = b_s + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            uint32_t a[4];
            if constexpr (BITS == 8) {
                tile_frag<8, OT>(v[r], s, a);
            } else {
                const uint32_t w = s == 0 ? v[r].x : s == 1 ? v[r].y : s == 2 ? v[r].z : v[r].w;
                const uint32_t w8 = w >> 8;
                a[0] = fma_f16x2(cvt_u4x2<ACT_F16>(w), slo, zlo);
                a[1] = fma_f16x2(cvt_u4x2_hi_f16(w), shi, zhi);
                a[2] = fma_f16x2(cvt_u4x2<ACT_F16>(w8), slo, zlo);
                a[3] = fma_f16x2(cvt_u4x2_hi_f16(w8), shi, zhi);
            }
            const int chunk = (tl * KT + 16 * s) / 8 + (mi & 1);
            stmatrix_x4(row_base + (uint32_t)((chunk ^ (row & 7)) << 4), a[0], a[2], a[1], a[3]);
        }
    }
}

// Sum of `splits` partial blocks (4 KB each: 32 rows x 32 fp32, block sp at
// blk0 + sp * stride floats) into this lane's row v[32], in split order.  Up
// to four blocks at a time are staged in shared memory at `stg` (16 KB) with
// cp.async, their 16-byte pieces swizzled by row so that each lane reads its
// row without bank conflicts.  Kept out of line: it is the cold k-split path
// and stays out of the register allocation of the main loop.
__device__ __noinline__ void split_sum(const float* blk0, size_t stride, int splits, uint32_t stg, int lane,
                                       float (&v)[32])
{
    for (int sp0 = 0; sp0 < splits; sp0 += 4) {
        const int nb = splits - sp0 < 4 ? splits - sp0 : 4;
        for (int b = 0; b < nb; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int pc = i * 32 + lane, r = pc >> 3, w = pc & 7;
                cp_async_16(stg + (uint32_t)(b * 4096 + r * 128 + ((w ^ (r & 7)) << 4)),
                            blk0 + (size_t)(sp0 + b) * stride + pc * 4);
            }
        cp_async_wait_all();
        __syncwarp();
        for (int b = 0; b < nb; ++b)
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint4 u = lds128(stg + (uint32_t)(b * 4096 + lane * 128 + ((w ^ (lane & 7)) << 4)));
                v[4 * w] += __uint_as_float(u.x);
                v[4 * w + 1] += __uint_as_float(u.y);
                v[4 * w + 2] += __uint_as_float(u.z);
                v[4 * w + 3] += __uint_as_float(u.w);
            }
        __syncwarp();  // reads done before the next batch lands
    }
}

template <int BITS, int OT, int ACT, int BN, int MS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                   const TcParams p)
{
    using Cfg = TcCfg<BITS, BN, MS>;
    constexpr int TM = BM * MS;  // output tile height
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ringA = smem;
    uint8_t* ring2 = ringA + Cfg::SA * Cfg::A_BYTES;
    uint8_t* ringC = ring2 + Cfg::S2 * Cfg::B_BYTES;
    Barriers* bars = reinterpret_cast<Barriers*>(ringC + Cfg::SC * Cfg::C_BYTES);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // work units: (output tile, k range); unit u is tile u / splits, k blocks
    // [(u % splits) kps, + kps)
    const int splits = p.splits, kps = p.num_kb / splits;
    const int total_units = p.m_tiles * p.n_tiles * splits;
    const int my_tiles =  // units this CTA runs
        (int)blockIdx.x < total_units ? (total_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * kps;  // k blocks this CTA runs, over all its units
    // one accumulator (its epilogue cannot overlap the next tile's MMAs): the
    // dequantisation warps, idle while it drains, drain two thirds of it
    const bool helpers = BITS == 8 && Cfg::NACC == 1 && splits == 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::SA; ++s) {
            mbar_init(&bars->fullA[s], 1);
            mbar_init(&bars->emptyA[s], 1);
        }
        for (int s = 0; s < Cfg::SC; ++s) {
            mbar_init(&bars->fullC[s], 1);
            mbar_init(&bars->emptyC[s], kDequantWarps);
        }
        for (int s = 0; s < Cfg::S2; ++s) {
            mbar_init(&bars->full2[s], kDequantWarps * 32);
            mbar_init(&bars->empty2[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->tfull[a], Cfg::PARTS);  // one commit per MMA issuer
            mbar_init(&bars->tempty[a], helpers ? 4 * 32 + kDequantWarps : 4 * 32);
        }
        mbar_init(&bars->mma_done, Cfg::PARTS);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // A tile's column scales (8-bit) and bias are fetched into registers
    // before its accumulator is ready, BN / 32 columns per lane (CW
    // column pairs), so that their latency hides behind the MMAs; the
    // drain gathers each 32-column chunk's values with shuffles.
    constexpr int CW = BN / 64;
    uint32_t csc[CW], cbi[CW];
    auto col_pair = [&](const uint16_t* v, int col) -> uint32_t {
        if (col >= p.n)
            return 0u;
        const uint32_t lo = __ldg(v + col);
        return col + 1 < p.n ? lo | ((uint32_t)__ldg(v + col + 1) << 16) : lo;
    };
    auto stage_cols = [&](int n0) {
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            const int col = n0 + 2 * (lane * CW + i);
            csc[i] = col_pair(BITS == 8 ? p.scales : p.colscale, col);
            cbi[i] = p.bias ? col_pair(p.bias, col) : 0u;
        }
    };
    // chunk cc's 32 scales and bias values, as 16 pairs (whole warp)
    auto gather = [&](int cc, uint32_t (&sc)[16], uint32_t (&bi)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int src = (cc * 16 + j) / CW;
            sc[j] = __shfl_sync(0xffffffffu, csc[j % CW], src);
            bi[j] = __shfl_sync(0xffffffffu, cbi[j % CW], src);
        }
    };
    // scale (8-bit) or row and column powers of two (4-bit), bias, one
    // rounding: 32 values of row `row`, columns nc..nc+31
    auto finish = [&](int row, int nc, float rs, const float (&v)[32], const uint32_t (&sc)[16],
                      const uint32_t (&bi)[16]) {
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float v0 = v[2 * j], v1 = v[2 * j + 1];
            if constexpr (BITS == 8) {
                v0 *= to_f32<ACT>((uint16_t)(sc[j] & 0xFFFFu));
                v1 *= to_f32<ACT>((uint16_t)(sc[j] >> 16));
            } else {
                v0 *= rs * to_f32<ACT_BF16>((uint16_t)(sc[j] & 0xFFFFu));
                v1 *= rs * to_f32<ACT_BF16>((uint16_t)(sc[j] >> 16));
            }
            if (p.bias) {
                v0 += to_f32<ACT>((uint16_t)(bi[j] & 0xFFFFu));
                v1 += to_f32<ACT>((uint16_t)(bi[j] >> 16));
            }
            packed[j] = (uint32_t)from_f32<ACT>(v0) | ((uint32_t)from_f32<ACT>(v1) << 16);
        }
        if (!in_bounds(row < p.m && nc >= 0 && nc + 32 <= p.n, 0x302))
            return;
        uint16_t* dst = p.C + (size_t)row * p.n + nc;
        if (p.c_v8) {  // two 32-byte stores: whole sectors
#pragma unroll
            for (int w = 0; w < 2; ++w)
                st_global_v8(dst + 16 * w, &packed[8 * w]);
        } else {
#pragma unroll
            for (int w = 0; w < 4; ++w)
                reinterpret_cast<uint4*>(dst)[w] =
                    make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2], packed[4 * w + 3]);
        }
    };
    // TMEM -> C for the chunks x = part, part + nparts, ... of unit `it`'s
    // accumulator (x walks the MS sub-tiles' 32-column chunks), rows of this
    // warp's TMEM lane quadrant; stage_cols(n0) of the tile came first
    // r += the 32 columns of TMEM at `col` (a second partial accumulator)
    auto add_partial = [&](uint32_t col, uint32_t (&r)[32]) {
        uint32_t r2[32];
        tmem_ld_32x32b_x32(col, r2);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
    };
    auto drain = [&](int it, int part, int nparts) {
        const int acc = it % Cfg::NACC, qd = warp & 3;
        int m0, n0;
        tile_coords(p, ((int)blockIdx.x + it * (int)gridDim.x) / splits, TM, BN, m0, n0);
        int rs_h = -1;  // sub-tile whose row scale rs holds
        float rs = 1.f;
#pragma unroll 1
        for (int x = part; x < MS * (BN / 32); x += nparts) {
            const int h = x / (BN / 32), cc = x % (BN / 32);
            const int nc = n0 + cc * 32;
            if (nc >= p.n)
                continue;
            const int row = m0 + h * BM + qd * 32 + lane;
            if (h != rs_h) {
                rs = (p.rowscale && row < p.m) ? p.rowscale[row] : 1.f;
                rs_h = h;
            }
            uint32_t r[32];
            const uint32_t col = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)((acc * MS * Cfg::PARTS + h) * BN + cc * 32);
            tmem_ld_32x32b_x32(col, r);
            tmem_ld_wait();
            if (Cfg::PARTS == 2 && kps > 1)  // the odd k blocks' partial sums
                add_partial(col + (uint32_t)BN, r);
            uint32_t sc[16], bi[16];
            gather(cc, sc, bi);
            if (row < p.m) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = __uint_as_float(r[j]);
                finish(row, nc, rs, v, sc, bi);
            }
        }
    };


    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // ---- TMA producers: codes (warp 0) and A tiles (warp 2) ----
            const bool codes = warp == 0;
            const int S = codes ? Cfg::SC : Cfg::SA;
            uint64_t* full = codes ? bars->fullC : bars->fullA;
            uint64_t* empty = codes ? bars->emptyC : bars->emptyA;
            int c = 0;  // k blocks issued, over all tiles
            int s = 0;  // c % S and the parity of c / S, kept as counters (no division per block)
            uint32_t ph = 0;
            bool ok = true;
            if (!codes)  // activations: after the previous kernel on the stream
                asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int it = 0; it < my_tiles && ok; ++it) {
                const int u = (int)blockIdx.x + it * (int)gridDim.x;
                int m0, n0;
                tile_coords(p, u / splits, TM, BN, m0, n0);
                const int kb0 = (u % splits) * kps;
                for (int kb = kb0; kb < kb0 + kps; ++kb, ++c, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort, p.err, codes ? 1 : 9, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    if (codes) {
                        mbar_arrive_expect_tx(&full[s], Cfg::C_BYTES);
                        // one row per 16-channel block, x in 32-bit words
                        tma_load_2d(ringC + s * Cfg::C_BYTES, &tmC, &full[s],
                                    kb * (Cfg::C_BYTES / (BN / 16) / 4), n0 / 16);
                    } else {
                        mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES);
#pragma unroll
                        for (int h = 0; h < MS; ++h)  // rows past m read as zeros
                            tma_load_2d(ringA + s * Cfg::A_BYTES + h * Cfg::A_SUB, &tmA, &full[s], kb * BK,
                                        m0 + h * BM);
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                volatile int never = 0;
                for (int i = c - S > 0 ? c - S : 0; i < c; ++i)
                    mbar_wait_bounded(&full[i % S], (i / S) & 1, &never, nullptr, 0, kWaitLimitNs);
            }
        }
        __syncwarp();  // the whole warp reaches the closing CTA barrier together
    } else if (warp == 1 || (Cfg::PARTS == 2 && warp == 3)) {
        if (lane == 0) {
            // ---- MMA issuers: warp 1 (and with two partial sums, warp 3 for the
            // odd k blocks of each unit, into the columns after the first) ----
            constexpr uint32_t idesc = idesc_f16(OT == ACT_BF16 ? 1u : 0u, BM, BN);
            const int pt = warp >> 1;  // partial sum of this issuer
            int c = 0;
            bool ok = true;
            for (int it = 0; it < my_tiles && ok; ++it) {
                const int acc = it % Cfg::NACC, use = it / Cfg::NACC;
                if (!mbar_wait_bounded(&bars->tempty[acc], (use & 1) ^ 1, abort, p.err, 7,
                                       kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)((acc * MS * Cfg::PARTS + pt) * BN);
                const int kb0 = (((int)blockIdx.x + it * (int)gridDim.x) % splits) * kps;
                bool first = true;
                for (int kb = kb0; kb < kb0 + kps; ++kb, ++c) {
                    if (Cfg::PARTS == 2 && ((kb - kb0) & 1) != pt)
                        continue;  // the other issuer's k block (c still counts it)
                    const int sa = c % Cfg::SA, s2 = c % Cfg::S2;
                    // sleeping waits: the MMA thread polling the ring barriers
                    // slows the arrivals on them (m = 256 / 1024: 4-7 % measured)
                    if (!mbar_wait_bounded<false, true>(&bars->fullA[sa], (c / Cfg::SA) & 1, abort, p.err, 2,
                                           kWaitLimitNs) ||
                        !mbar_wait_bounded<false, true>(&bars->full2[s2], (c / Cfg::S2) & 1, abort, p.err, 3,
                                           kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = desc_sw128(smem_addr(ring2 + s2 * Cfg::B_BYTES));
#pragma unroll
                    for (int h = 0; h < MS; ++h) {  // sub-tile h: TMEM columns [h BN, (h + 1) BN)
                        const uint64_t ad =
                            desc_sw128(smem_addr(ringA + sa * Cfg::A_BYTES + h * Cfg::A_SUB));
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j)  // +32 bytes per 16-wide k step
                            mma_f16(d + (uint32_t)(h * BN), ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j),
                                    idesc, (!first || j > 0) ? 1u : 0u);
                    }
                    first = false;
                    mma_commit(&bars->emptyA[sa]);
                    mma_commit(&bars->empty2[s2]);
                }
                if (ok)
                    mma_commit(&bars->tfull[acc]);
            }
            // every MMA issued must finish before TMEM is released (also on
            // abort); warp 1 frees it after the closing barrier
            mma_commit(&bars->mma_done);
            if (pt == 0) {
                volatile int never = 0;
                mbar_wait_bounded(&bars->mma_done, 0, &never, p.err, 8, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
        // ---- epilogue: TMEM lane quadrant q = warp % 4 ----
        const int q = warp - kEpilogueWarp0;
        volatile int* is_last = &bars->is_last;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs, row scales, workspace
        for (int it = 0; it < my_tiles; ++it) {
            const int u = (int)blockIdx.x + it * (int)gridDim.x;
            const int tile = u / splits;
            const int acc = it % Cfg::NACC, use = it / Cfg::NACC;
            int m0, n0;
            tile_coords(p, tile, TM, BN, m0, n0);
            stage_cols(n0);
            const bool got = mbar_wait_bounded(&bars->tfull[acc], use & 1, abort, p.err, 6,
                                               kWaitLimitNs);
            const bool live = __all_sync(0xffffffffu, got && !*abort);  // tcgen05.ld: whole warp
            if (splits == 1) {
                if (!live)
                    break;
                tc_fence_after();
                drain(it, 0, helpers ? 3 : 1);
                tc_fence_before();
                mbar_arrive(&bars->tempty[acc]);
                continue;
            }
            // ---- k split: this unit's accumulator -> its fp32 partial tile; the
            // unit that arrives last at the tile's counter sums the partials in
            // split order and writes C (deterministic, and no unit waits) ----
            float* part = p.partial + (size_t)u * TM * BN;
            if (live) {
                tc_fence_after();
                for (int h = 0; h < MS; ++h)
#pragma unroll 1
                    for (int cc = 0; cc < BN / 32; ++cc) {
                        if (n0 + cc * 32 >= p.n)
                            break;
                        uint32_t r[32];
                        const uint32_t col = tmem + ((uint32_t)(q * 32) << 16) +
                                             (uint32_t)((acc * MS * Cfg::PARTS + h) * BN + cc * 32);
                        tmem_ld_32x32b_x32(col, r);
                        tmem_ld_wait();
                        if (Cfg::PARTS == 2 && kps > 1)
                            add_partial(col + (uint32_t)BN, r);
                        // [h][cc][row of the sub-tile][32]: a warp writes 4 KiB contiguously
                        float4* dst = reinterpret_cast<float4*>(
                            part + ((size_t)(h * (BN / 32) + cc) * BM + q * 32 + lane) * 32);
                        if (!in_bounds((size_t)(reinterpret_cast<float*>(dst) - p.partial) + 32 <= p.partial_floats,
                                       0x303))
                            continue;
#pragma unroll
                        for (int w = 0; w < 8; ++w)
                            dst[w] = make_float4(__uint_as_float(r[4 * w]), __uint_as_float(r[4 * w + 1]),
                                                 __uint_as_float(r[4 * w + 2]), __uint_as_float(r[4 * w + 3]));
                    }
            }
            tc_fence_before();
            mbar_arrive(&bars->tempty[acc]);
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (warp == kEpilogueWarp0 && lane == 0) {
                if (*abort) {
                    *is_last = -1;
                } else {
                    const unsigned prev =
                        in_bounds(tile < (int)kWsCounters, 0x304) ? atomicAdd(p.counters + tile, 1u) : 0u;
                    *is_last = prev == (unsigned)(splits - 1) ? 1 : 0;
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int last = *is_last;
            if (last < 0)
                break;  // every epilogue warp read the same value
            if (last) {
                __threadfence();
                // A split plan gives every CTA one unit (launch_tc_t checks), so
                // here the A ring is idle: split_sum stages the partials in it
                // (up to four splits, 16 KB per warp, in flight at once instead
                // of 128 bytes per lane).
                static_assert(Cfg::SA * Cfg::A_BYTES >= 4 * 16384, "partial staging");
                const uint32_t stg = smem_addr(ringA) + (uint32_t)(q * 16384);
#pragma unroll 1
                for (int h = 0; h < MS; ++h) {
                    const int row = m0 + h * BM + q * 32 + lane;
                    const float rs = (p.rowscale && row < p.m) ? p.rowscale[row] : 1.f;
#pragma unroll 1
                    for (int cc = 0; cc < BN / 32; ++cc) {
                        const int nc = n0 + cc * 32;
                        if (nc >= p.n)
                            break;
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = 0.f;
                        // split 0's block: this warp's 32 rows x 32 floats, 4 KB
                        const size_t blk0 = (size_t)tile * splits * TM * BN +
                                            ((size_t)(h * (BN / 32) + cc) * BM + q * 32) * 32;
                        if (in_bounds(blk0 + (size_t)(splits - 1) * TM * BN + 32 * 32 <= p.partial_floats, 0x305))
                            split_sum(p.partial + blk0, (size_t)TM * BN, splits, stg, lane, v);
                        uint32_t sc[16], bi[16];
                        gather(cc, sc, bi);
                        if (row < p.m)
                            finish(row, nc, rs, v, sc, bi);
                    }
                }
                if (warp == kEpilogueWarp0 && lane == 0)
                    p.counters[tile] = 0u;  // ready for the next call
            }
        }
    } else if (warp >= kDequantWarp0) {
        // ---- dequantisation ----
        const int dw = warp - kDequantWarp0;
        if (BITS == 4 || helpers)  // the prepass's scales / the helpers' C stores
            asm volatile("griddepcontrol.wait;" ::: "memory");
        auto n0_of = [&](int c) {
            const int u = (int)blockIdx.x + (c / kps) * (int)gridDim.x;
            int m0, n0;
            tile_coords(p, u / splits, TM, BN, m0, n0);
            return n0;
        };
        auto kb_of = [&](int c) {  // k block of the CTA's c-th k block
            const int u = (int)blockIdx.x + (c / kps) * (int)gridDim.x;
            return (u % splits) * kps + c % kps;
        };
        DqScales<BITS, BN> buf[Cfg::PF];
        if constexpr (BITS == 4) {
#pragma unroll
            for (int j = 0; j < Cfg::PF; ++j)
                if (j < total)
                    load_scales<BITS, BN>(p, n0_of(j), kb_of(j), dw, lane, buf[j]);
        }
        // drain part 1 + dw / 4 of three of unit t's accumulator (helpers)
        auto help = [&](int t) {
            int m0, n0;
            tile_coords(p, ((int)blockIdx.x + t * (int)gridDim.x) / splits, TM, BN, m0, n0);
            stage_cols(n0);
            const bool got = mbar_wait_bounded(&bars->tfull[0], t & 1, abort, p.err, 13, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got && !*abort))
                return false;
            tc_fence_after();
            drain(t, 1 + dw / 4, 3);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->tempty[0]);
            return true;
        };
        int nd = 0;  // next unit to help drain
        bool ok = true;
        for (int c0 = 0; c0 < total && ok; c0 += Cfg::PF) {
            // unit nd's k blocks all dequantised (c0 >= B), and this group
            // reaches block B + S2, whose operand stage only frees once the
            // next unit's MMAs run, i.e. after unit nd's drain: help first
            // (a group never holds both B - 1 and B + S2, as PF <= S2 + 1)
            static_assert(Cfg::NACC == 2 || Cfg::PF <= Cfg::S2 + 1, "helper trigger");
            while (helpers && ok && nd < my_tiles && c0 >= (nd + 1) * kps &&
                   c0 + Cfg::PF - 1 >= (nd + 1) * kps + Cfg::S2)
                ok = help(nd++);
#pragma unroll
            for (int j = 0; j < Cfg::PF; ++j) {
                const int c = c0 + j;
                if (c >= total)
                    break;
                const int sc = c % Cfg::SC, s2 = c % Cfg::S2;
                // warp-uniform decisions: stmatrix below needs the whole warp
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&bars->fullC[sc], (c / Cfg::SC) & 1, abort, p.err,
                                                  4, kWaitLimitNs) &&
                                    mbar_wait_bounded(&bars->empty2[s2], ((c / Cfg::S2) & 1) ^ 1,
                                                      abort, p.err, 5, kWaitLimitNs))) {
                    ok = false;
                    break;
                }
                dequant_stage<BITS, OT, ACT, BN>(smem_addr(ringC + sc * Cfg::C_BYTES), buf[j],
                                                 smem_addr(ring2 + s2 * Cfg::B_BYTES), dw, lane);
                fence_proxy_async_smem();
                mbar_arrive(&bars->full2[s2]);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->emptyC[sc]);
                if constexpr (BITS == 4) {
                    if (c + Cfg::PF < total)
                        load_scales<BITS, BN>(p, n0_of(c + Cfg::PF), kb_of(c + Cfg::PF), dw,
                                              lane, buf[j]);
                }
            }
        }
        while (helpers && ok && nd < my_tiles)
            ok = help(nd++);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// The 4-bit prepass (one launch before the GEMM), in two kinds of CTA:
//   - CTAs [0, a_ctas), bf16 activations only: row r of A times 2^-E_r
//     (E_r chosen so max |a| * 2^-E_r lies in [2^14, 2^15)), which is exact,
//     rounded to fp16, which is exact for bf16 values whose scaled magnitude
//     is at least 2^-14; rowscale[r] = 2^E_r.  One CTA per row, 16-byte
//     loads and stores (k % 64 == 0 and A 16-byte aligned on this path); up
//     to kA16Cache chunks of 8 values per thread stay in registers between
//     the maximum and the conversion, so rows of up to 16384 values are read
//     once.
//   - the other CTAs, one warp per output channel n: M = the largest |scale|
//     or |zero| of the channel's groups, E_n with M * 2^-E_n in [2^10, 2^11)
//     (clamped to [-120, 120], so that 2^E_n and 2^-E_n are normal floats),
//     then every group's (fp16(s * 2^-E_n), fp16(z * 2^-E_n)) pair into sz
//     and 2^E_n into colscale (bf16 bits).  (q - 8) s' + z' is then at most
//     8 * 2^11 + 2^11 in magnitude.
constexpr int kPrepThreads = 256, kA16Cache = 8;

__device__ __forceinline__ float absmax_bf16x8(const uint4& v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mx = fmaxf(mx, fabsf(to_f32<ACT_BF16>((uint16_t)(w[i] & 0xFFFFu))));
        mx = fmaxf(mx, fabsf(to_f32<ACT_BF16>((uint16_t)(w[i] >> 16))));
    }
    return mx;
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v, float inv)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)from_f32<ACT_F16>(to_f32<ACT_BF16>((uint16_t)(w[i] & 0xFFFFu)) * inv) |
               ((uint32_t)from_f32<ACT_F16>(to_f32<ACT_BF16>((uint16_t)(w[i] >> 16)) * inv) << 16);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void prep_a_row(const uint16_t* __restrict__ A, uint16_t* __restrict__ A16,
                                           float* __restrict__ rowscale, int row, int k)
{
    const uint4* a = reinterpret_cast<const uint4*>(A + (size_t)row * k);
    uint4* o = reinterpret_cast<uint4*>(A16 + (size_t)row * k);
    const int nch = k >> 3;  // chunks of 8 values
    uint4 c[kA16Cache];
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < kA16Cache; ++i) {
        const int j = (int)threadIdx.x + i * kPrepThreads;
        if (j < nch) {
            c[i] = __ldg(a + j);
            mx = fmaxf(mx, absmax_bf16x8(c[i]));
        }
    }
    for (int j = (int)threadIdx.x + kA16Cache * kPrepThreads; j < nch; j += kPrepThreads)
        mx = fmaxf(mx, absmax_bf16x8(__ldg(a + j)));
    __shared__ float red[32];
    for (int s = 16; s > 0; s >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (kPrepThreads >> 5) ? red[threadIdx.x] : 0.f;
        for (int s = 16; s > 0; s >>= 1)
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
        if (threadIdx.x == 0)
            red[0] = v;
    }
    __syncthreads();
    mx = red[0];
    int E = 0;
    if (mx > 0.f && mx <= 3.0e38f) {
        int e2;
        frexpf(mx, &e2);  // mx = f * 2^e2, f in [0.5, 1)
        E = e2 - 15;      // mx * 2^-E in [2^14, 2^15)
    }
    const float inv = ldexpf(1.f, -E);
#pragma unroll
    for (int i = 0; i < kA16Cache; ++i) {
        const int j = (int)threadIdx.x + i * kPrepThreads;
        if (j < nch)
            o[j] = bf16x8_to_f16x8(c[i], inv);
    }
    for (int j = (int)threadIdx.x + kA16Cache * kPrepThreads; j < nch; j += kPrepThreads)
        o[j] = bf16x8_to_f16x8(__ldg(a + j), inv);
    if (threadIdx.x == 0)
        rowscale[row] = ldexpf(1.f, E);
}

template <int ACT>
__device__ __forceinline__ void prep_channel(const uint16_t* __restrict__ scales,
                                             const uint16_t* __restrict__ zeros, int ch, int G,
                                             uint32_t* __restrict__ sz, uint16_t* __restrict__ colscale,
                                             int lane)
{
    const uint16_t* s = scales + (size_t)ch * G;
    const uint16_t* z = zeros ? zeros + (size_t)ch * G : nullptr;
    float mx = 0.f;
    for (int g = lane; g < G; g += 32) {
        mx = fmaxf(mx, fabsf(to_f32<ACT>(ld_nc_u16(s + g))));
        if (z)
            mx = fmaxf(mx, fabsf(to_f32<ACT>(ld_nc_u16(z + g))));
    }
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int E = 0;
    if (mx > 0.f && mx <= 3.0e38f) {
        int e2;
        frexpf(mx, &e2);  // mx in [2^(e2 - 1), 2^e2)
        E = min(max(e2 - 11, -120), 120);
    }
    const float inv = __int_as_float((127 - E) << 23);  // 2^-E, a normal float
    for (int g = lane; g < G; g += 32) {
        const uint32_t sv = from_f32<ACT_F16>(to_f32<ACT>(ld_nc_u16(s + g)) * inv);
        const uint32_t zv = z ? from_f32<ACT_F16>(to_f32<ACT>(ld_nc_u16(z + g)) * inv) : 0u;
        sz[(size_t)ch * G + g] = sv | (zv << 16);
    }
    if (lane == 0)
        colscale[ch] = (uint16_t)((127 + E) << 7);  // 2^E as bf16
}

template <int ACT>
__global__ void __launch_bounds__(kPrepThreads)
    tc_prep_kernel(const uint16_t* __restrict__ A, uint16_t* __restrict__ A16, float* __restrict__ rowscale,
                   int a_ctas, int k, const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros,
                   int n, int G, uint32_t* __restrict__ sz, uint16_t* __restrict__ colscale)
{
    // the GEMM kernel behind this one may start its set-up now: it waits for
    // this grid before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x < a_ctas) {
        prep_a_row(A, A16, rowscale, (int)blockIdx.x, k);
        return;
    }
    const int ch = ((int)blockIdx.x - a_ctas) * (kPrepThreads / 32) + (int)(threadIdx.x >> 5);
    if (ch < n)
        prep_channel<ACT>(scales, zeros, ch, G, sz, colscale, (int)(threadIdx.x & 31));
}

// Output tile shape: MS sub-tiles of 128 rows by BN columns, the one whose
// waves of tiles over the SMs take the least time.  A tile's time is its
// shape's relative cost per k block, measured on GB300 with this kernel
// (one 256 x 256 tile = 1): the 256 x 256 tiles fetch the fewest A and code
// bytes per FLOP and dequantise each B tile for two MMAs, so they do the
// most work per unit time; narrower tiles win when they fill more SMs.
// 4-bit codes cost more to dequantise per weight, which weighs on the
// shapes with one M=128 MMA per B tile (MS = 1).
struct TcShape {
    int bn, ms;
};

TcShape tc_shape(int m, int n, int bits)
{
    struct Cand {
        int bn, ms;
        double cost;
    };
    // (8-bit 256 x 128 tiles, 0.66, never beat 128 x 256 ones at 0.61: the
    // two shapes give nearly the same tile counts)
    static constexpr Cand c8[3] = {{256, 2, 1.0}, {256, 1, 0.61}, {128, 1, 0.48}};
    static constexpr Cand c4[4] = {{256, 2, 1.0}, {128, 2, 0.70}, {128, 1, 0.63}, {256, 1, 0.99}};
    const Cand* cs = bits == 8 ? c8 : c4;
    const int nc = bits == 8 ? 3 : 4;
    TcShape best{cs[0].bn, cs[0].ms};
    double best_t = 0.0;
    for (int i = 0; i < nc; ++i) {
        const long long tiles =
            (long long)((m + BM * cs[i].ms - 1) / (BM * cs[i].ms)) * ((n + cs[i].bn - 1) / cs[i].bn);
        const double t = (double)((tiles + num_sms() - 1) / num_sms()) * cs[i].cost;
        if (i == 0 || t < best_t * 0.999) {
            best = {cs[i].bn, cs[i].ms};
            best_t = t;
        }
    }
    return best;
}

template <int BITS, int OT, int ACT, int BN, int MS>
cudaError_t launch_tc_t(const CUtensorMap& ma, const void* B, TcParams tp, cudaStream_t s)
{
    constexpr int smem = TcCfg<BITS, BN, MS>::SMEM + (int)sizeof(Barriers) + 1024;
    static_assert(smem <= 232448, "shared memory per CTA");
    auto kern = gemm_tc_kernel<BITS, OT, ACT, BN, MS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    tp.m_tiles = (tp.m + BM * MS - 1) / (BM * MS);
    tp.n_tiles = (tp.n + BN - 1) / BN;
    const long long units = (long long)tp.m_tiles * tp.n_tiles * tp.splits;
    if (tp.splits > 1 && units > num_sms())
        return cudaErrorInvalidConfiguration;  // the split reduction stages in the A ring of a one-unit CTA
    const int grid = (int)(units < num_sms() ? units : num_sms());
    // packed codes viewed as [n/16 rows] x [bytes per 16-channel row / 4] words;
    // one box = BN/16 rows x one k block
    CUtensorMap mc;
    const uint64_t row_bytes = (uint64_t)tp.k * 16 * BITS / 8;
    if (!make_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, B, row_bytes / 4, (uint64_t)tp.n / 16,
                      row_bytes, BK * 16 * BITS / 8 / 4, BN / 16, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mc, tp);
}

template <int BITS, int OT, int ACT>
cudaError_t launch_tc_bn(const CUtensorMap& ma, const void* B, const TcParams& tp, const TcPlan& sh,
                         cudaStream_t s)
{
    if (sh.ms == 2) {
        if constexpr (BITS == 4)  // tc_shape gives 256 x 128 tiles for 4-bit codes only
            if (sh.bn == 128)
                return launch_tc_t<BITS, OT, ACT, 128, 2>(ma, B, tp, s);
        return launch_tc_t<BITS, OT, ACT, 256, 2>(ma, B, tp, s);
    }
    return sh.bn == 128 ? launch_tc_t<BITS, OT, ACT, 128, 1>(ma, B, tp, s)
                        : launch_tc_t<BITS, OT, ACT, 256, 1>(ma, B, tp, s);
}


// ============================================================ MoE experts ===
//
// Grouped expert GEMMs of the MoE FFN (acext User Guide (v1.7) 1.2.3) on the
// tensor cores, "swap AB": an expert's 8-bit weights, dequantised exactly to
// (q - 128) in the activation dtype, are the MMA's 128-row operand (output
// channels), and the expert's token rows (in expert order, a chunk of up to
// kMoeNT at a time) are its N operand, so an expert's few dozen rows still
// fill the tensor pipe while its weights stream from HBM once per chunk.
// Work items: (expert, block of output channels).  For the gated fc1 an item
// carries the 128 gate channels and the matching 128 up channels (inter
// apart) so the epilogue can form h = silu(gate) * up; for fc2 it carries
// 256 consecutive output channels when they tile the output (else 128).
// An item's two 128-row weight halves are two MMAs on the same staged token
// tile: the token rows are copied once per 256 weight rows.  Roles as in
// gemm_tc_kernel: warp 0 codes TMA, warp 2 activation TMA, warp 1 MMA,
// warps 4-7 epilogue (TMEM lanes are channels, columns are tokens), warps
// 8-15 dequantisation.
//
// The same kernel serves wo_gemm between the decode sizes and the
// tensor-core kernel's (8-bit weights, 17..64 rows, at most one block of 128
// output channels per SM: PLAIN): one "expert" of m rows, items (block of
// 128 output channels, k split), the epilogue writing
// round(acc * scale[n] + bias[n]) in the activation dtype.  A channel
// block's k range is split so that the items fill the SMs, one item per SM;
// each split stores its fp32 sums in the workspace, one 128-byte line of
// channels per row, and the split that arrives last sums them in split
// order and writes the block (deterministic; no item waits for another).

constexpr int kMoeNT = 64;  // token rows per chunk (the MMA's N)

// TWO: an item carries two 128-row weight halves that share each token tile
// (the gated fc1's gate and up rows, or 256 consecutive fc2 channels).
// PLAIN: a plain GEMM of at most 64 rows.
template <bool TWO, bool PLAIN>
struct MoeCfg {
    static constexpr int WR = TWO ? 256 : 128;           // weight rows per item
    static constexpr int A_BYTES = kMoeNT * BK * 2;       // 8 KiB of token rows
    static constexpr int C_BYTES = WR * BK;               // packed codes of a k block
    static constexpr int B_BYTES = WR * BK * 2;           // dequantised operand
    // The codes stream from HBM, token rows come from L2, and the operand
    // ring covers the dequant -> MMA hand-off.  Measured: with two MMA
    // issuers the operand ring paces the items, so the plain GEMM's rings
    // take 12 code and 6 operand stages (224 KiB; 3584 x 18944 m = 24: 26.5
    // -> 24.5 us) and the two-half MoE items 6 and 3 (224 KiB; MoE step
    // +3 %).
    static constexpr int SA = 4;
    static constexpr int SC = PLAIN ? 12 : (TWO ? 6 : 16);
    static constexpr int S2 = PLAIN ? 6 : 3;
    static_assert(SC <= 16 && S2 <= 8 && SA <= 8, "barrier arrays");
    static constexpr int COLS = (TWO ? 2 : 1) * kMoeNT;   // TMEM columns per accumulator
    // two items in flight, each as two partial accumulators (even and odd k
    // blocks, issued by two threads)
    static constexpr uint32_t TMEM_COLS = 4 * COLS;
    static_assert(TMEM_COLS <= 512, "tensor memory");
    static constexpr int SMEM = SA * A_BYTES + SC * C_BYTES + S2 * B_BYTES;
};

struct MoeTcParams {
    const int* offsets;      // [E + 1] row ranges of the experts (rows in expert order); PLAIN: null
    int E, nb;               // experts, channel blocks (128 or 256 channels) per expert
    int num_kb;              // K / BK
    int inter;               // gated: channel distance gate -> up (and h row length)
    int n_out;               // plain: output row length (hidden)
    int rows_per_expert_w;   // weight rows of one expert (2 * inter or hidden)
    const uint16_t* scales;  // [E, rows_per_expert_w] in the activation dtype
    uint16_t* H;             // gated output h [rows, inter]
    float* Y;                // fp32 output [rows, n_out]
    unsigned* err;
    // PLAIN (one expert of m rows):
    int m;                   // rows (<= kMoeNT)
    int ksplit, kps;         // k splits per channel block, k blocks per split
    const uint16_t* bias;    // [n_out] or null
    uint16_t* C;             // [m, n_out]
    float* partial;          // ksplit > 1: [nb][ksplit][kMoeNT rows][128 channels] fp32
    size_t partial_floats;   // its extent (index checks of the debug build)
    int rows_total;          // rows of H / Y (MoE) or C (plain)
    unsigned* counters;      // ksplit > 1: [nb], zero between calls
};

// Chunks of expert e's rows: its row range and how many kMoeNT chunks it needs.
__device__ __forceinline__ void moe_rows(const MoeTcParams& p, int e, int& r0, int& cnt, int& chunks)
{
    r0 = p.offsets ? p.offsets[e] : 0;
    cnt = p.offsets ? p.offsets[e + 1] - r0 : p.m;
    chunks = cnt > 0 ? (cnt + kMoeNT - 1) / kMoeNT : 0;
}

// Item `it`: its expert, channel block, k split and k blocks [kb0, kb1).
__device__ __forceinline__ void moe_item(const MoeTcParams& p, int it, int& e, int& nb, int& ks, int& kb0,
                                         int& kb1)
{
    if (p.offsets) {
        e = it / p.nb;
        nb = it % p.nb;
        ks = 0;
        kb0 = 0;
        kb1 = p.num_kb;
    } else {
        e = 0;
        nb = it / p.ksplit;
        ks = it % p.ksplit;
        kb0 = ks * p.kps;
        kb1 = min(kb0 + p.kps, p.num_kb);
    }
}

template <bool GATED, bool WIDE, bool PLAIN, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    moe_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                  const MoeTcParams p)
{
    static_assert(!(PLAIN && (GATED || WIDE)), "plain GEMM items are 128 channels");
    constexpr bool TWO = GATED || WIDE;
    constexpr int CH = WIDE ? 256 : 128;  // output channels per item
    using Cfg = MoeCfg<TWO, PLAIN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ringA = smem;
    uint8_t* ring2 = ringA + Cfg::SA * Cfg::A_BYTES;
    uint8_t* ringC = ring2 + Cfg::S2 * Cfg::B_BYTES;
    Barriers* bars = reinterpret_cast<Barriers*>(ringC + Cfg::SC * Cfg::C_BYTES);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int items = PLAIN ? p.nb * p.ksplit : p.E * p.nb;
    if constexpr (PLAIN)  // a wo_gemm: the next kernel may start its set-up
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::SA; ++s) {
            mbar_init(&bars->fullA[s], 1);
            mbar_init(&bars->emptyA[s], 1);
        }
        for (int s = 0; s < Cfg::SC; ++s) {
            mbar_init(&bars->fullC[s], 1);
            mbar_init(&bars->emptyC[s], kDequantWarps);
        }
        for (int s = 0; s < Cfg::S2; ++s) {
            mbar_init(&bars->full2[s], kDequantWarps * 32);
            mbar_init(&bars->empty2[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->tfull[a], 2);  // the two MMA issuers
            mbar_init(&bars->tempty[a], 4 * 32);
        }
        mbar_init(&bars->mma_done, 2);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // ---- TMA producers: codes (warp 0) and token rows (warp 2) ----
            const bool codes = warp == 0;
            const int S = codes ? Cfg::SC : Cfg::SA;
            uint64_t* full = codes ? bars->fullC : bars->fullA;
            uint64_t* empty = codes ? bars->emptyC : bars->emptyA;
            int c = 0;
            int s = 0;  // c % S and the parity of c / S, kept as counters (no division per block)
            uint32_t ph = 0;
            bool ok = true;
            if (PLAIN && !codes)  // activations: after the previous kernel on the stream
                asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, nb, ks, kb0, kb1;
                moe_item(p, it, e, nb, ks, kb0, kb1);
                int r0, cnt, chunks;
                moe_rows(p, e, r0, cnt, chunks);
                const int wrow = (e * p.rows_per_expert_w + nb * CH) / 16;  // 16-channel block row
                for (int ch = 0; ch < chunks && ok; ++ch) {
                    for (int kb = kb0; kb < kb1; ++kb, ++c, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0) {
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort, p.err, codes ? 21 : 22, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        if (codes) {
                            mbar_arrive_expect_tx(&full[s], Cfg::C_BYTES);
                            uint8_t* dst = ringC + s * Cfg::C_BYTES;
                            tma_load_2d(dst, &tmC, &full[s], kb * (BK * 16 / 4), wrow);
                            if constexpr (TWO)  // the matching up channels, inter rows further,
                                                // or the next 128 channels
                                tma_load_2d(dst + 128 * BK, &tmC, &full[s], kb * (BK * 16 / 4),
                                            wrow + (GATED ? p.inter / 16 : 8));
                        } else {
                            mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES);
                            tma_load_2d(ringA + s * Cfg::A_BYTES, &tmA, &full[s], kb * BK,
                                        r0 + ch * kMoeNT);
                        }
                    }
                }
            }
            if (!ok) {
                volatile int never = 0;
                for (int i = c - S > 0 ? c - S : 0; i < c; ++i)
                    mbar_wait_bounded(&full[i % S], (i / S) & 1, &never, nullptr, 0, kWaitLimitNs);
            }
        }
        __syncwarp();  // the whole warp reaches the closing CTA barrier together
    } else if (warp == 1 || warp == 3) {
        if (lane == 0) {
            // ---- MMA issuers: D[channels, tokens] += W[channels, k] . X[tokens, k]^T.
            // Warp 1 takes an item's even k blocks into partial accumulator 0,
            // warp 3 its odd ones into partial 1: one thread's per-k-block work
            // (waits, MMA issue, commits) bounded the weight stream, two
            // threads on two schedulers halve it.  The epilogue adds the two
            // partials (in that order). ----
            const int part = warp >> 1;
            constexpr uint32_t idesc = idesc_f16(ACT == ACT_BF16 ? 1u : 0u, 128, kMoeNT);
            int c = 0, t = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, nb, ks, kb0, kb1;
                moe_item(p, it, e, nb, ks, kb0, kb1);
                int r0, cnt, chunks;
                moe_rows(p, e, r0, cnt, chunks);
                for (int ch = 0; ch < chunks && ok; ++ch, ++t) {
                    const int acc = t & 1;
                    if (!mbar_wait_bounded(&bars->tempty[acc], ((t >> 1) & 1) ^ 1, abort, p.err, 27,
                                           kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)((2 * acc + part) * Cfg::COLS);
                    bool first = true;
                    for (int kb = kb0; kb < kb1; ++kb, ++c) {
                        if (((kb - kb0) & 1) != part)
                            continue;  // the other issuer's k block (c still counts it)
                        const int sa = c % Cfg::SA, s2 = c % Cfg::S2;
                        // the MMA thread sleeps while it waits: polling the
                        // operand barrier slows the dequantisation warps'
                        // arrivals on it (3-10 % measured)
                        if (!mbar_wait_bounded<false, true>(&bars->fullA[sa], (c / Cfg::SA) & 1, abort, p.err, 23,
                                                            kWaitLimitNs) ||
                            !mbar_wait_bounded<false, true>(&bars->full2[s2], (c / Cfg::S2) & 1, abort, p.err, 24,
                                                            kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t w_s = smem_addr(ring2 + s2 * Cfg::B_BYTES);
                        const uint64_t wd = desc_sw128(w_s);
                        const uint64_t xd = desc_sw128(smem_addr(ringA + sa * Cfg::A_BYTES));
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j) {
                            mma_f16(d, wd + (uint64_t)(2 * j), xd + (uint64_t)(2 * j), idesc,
                                    (!first || j > 0) ? 1u : 0u);
                            if constexpr (TWO)  // second half: operand rows 128..255, 16 KiB on
                                mma_f16(d + kMoeNT, desc_sw128(w_s + 128 * 128) + (uint64_t)(2 * j),
                                        xd + (uint64_t)(2 * j), idesc, (!first || j > 0) ? 1u : 0u);
                        }
                        first = false;
                        mma_commit(&bars->emptyA[sa]);
                        mma_commit(&bars->empty2[s2]);
                    }
                    // (an issuer without a k block in the item arrives at once;
                    // the epilogue then reads only partial 0)
                    if (ok)
                        mma_commit(&bars->tfull[acc]);
                }
            }
            mma_commit(&bars->mma_done);
            if (part == 0) {  // warp 1 frees TMEM after the closing barrier
                volatile int never = 0;
                mbar_wait_bounded(&bars->mma_done, 0, &never, p.err, 28, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (PLAIN && warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
        // ---- plain GEMM epilogue: lane = channel (TMEM lane quadrant warp % 4),
        // column = row of C; one accumulator per item (m <= kMoeNT) ----
        const int q = warp - kEpilogueWarp0;
        volatile int* is_last = &bars->is_last;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and workspace
        const int cnt = p.m;
        // this lane's channel as round(v * s + b) into row `row` of C
        auto store_c = [&](int row, int ch, float v, float sc, float bi) {
            if (in_bounds(row < p.m && ch < p.n_out, 0x401))
                p.C[(size_t)row * p.n_out + ch] = from_f32<ACT>(v * sc + bi);
        };
        int t = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++t) {
            int e, nb, ks, kb0, kb1;
            moe_item(p, it, e, nb, ks, kb0, kb1);
            const int ch0 = nb * CH + q * 32 + lane;  // this lane's channel
            const bool ch_ok = in_bounds(ch0 < p.n_out, 0x402);
            const float s0 = ch_ok ? to_f32<ACT>(ld_nc_u16(p.scales + ch0)) : 0.f;
            const float b0 = p.bias && ch_ok ? to_f32<ACT>(ld_nc_u16(p.bias + ch0)) : 0.f;
            const int acc = t & 1;
            const bool got = mbar_wait_bounded(&bars->tfull[acc], (t >> 1) & 1, abort, p.err, 29, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got && !*abort))  // tcgen05.ld needs the whole warp
                break;
            // split ks's fp32 sums, [row][128 channels]: this lane's channel
            float* part = p.partial + ((size_t)nb * p.ksplit + ks) * CH * kMoeNT + q * 32 + lane;
            tc_fence_after();
            // the item's two partial accumulators (even and odd k blocks; a
            // one-block item has only the first)
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(2 * acc * Cfg::COLS);
            const bool two_parts = kb1 - kb0 > 1;
#pragma unroll 1
            for (int cc = 0; cc < kMoeNT / 32; ++cc) {
                const int tok0 = cc * 32;
                if (tok0 >= cnt)
                    break;  // warp-uniform
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(cc * 32), r);
                tmem_ld_wait();
                if (two_parts) {
                    uint32_t r2[32];
                    tmem_ld_32x32b_x32(tbase + (uint32_t)(Cfg::COLS + cc * 32), r2);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                }
                if (p.ksplit == 1) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (tok0 + j < cnt)
                            store_c(tok0 + j, ch0, __uint_as_float(r[j]), s0, b0);
                } else {
                    // one 128-byte row of channels per row of C: each store is a
                    // whole line for the warp
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (tok0 + j < cnt &&
                            in_bounds((size_t)(part - p.partial) + (size_t)(tok0 + j) * 128 < p.partial_floats, 0x403))
                            __stcg(part + (size_t)(tok0 + j) * 128, __uint_as_float(r[j]));
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->tempty[acc]);
            if (p.ksplit == 1)
                continue;
            // k split: the split that arrives last at the block's counter sums the
            // splits in order (the CTA barrier orders every epilogue thread's
            // stores before the fence that releases them with the count)
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (warp == kEpilogueWarp0 && lane == 0) {
                if (*abort) {
                    *is_last = -1;
                } else {
                    __threadfence();
                    const unsigned prev =
                        in_bounds(nb < (int)kWsCounters, 0x404) ? atomicAdd(p.counters + nb, 1u) : 0u;
                    *is_last = prev == (unsigned)(p.ksplit - 1) ? 1 : 0;
                    if (prev == (unsigned)(p.ksplit - 1))
                        __threadfence();
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int last = *is_last;
            if (last < 0)
                break;  // every epilogue warp read the same value
            if (!last)
                continue;
            const float* base = p.partial + (size_t)nb * p.ksplit * CH * kMoeNT + q * 32 + lane;
#pragma unroll 1
            for (int t0 = 0; t0 < cnt; t0 += 16) {
                const float* src = base + (size_t)t0 * 128;
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    v[j] = 0.f;
                // four splits' loads in flight at a time, summed in split order
#pragma unroll 1
                for (int sp = 0; sp < p.ksplit; sp += 4) {
                    float x[4][16];
#pragma unroll
                    for (int b = 0; b < 4; ++b)
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            x[b][j] = (sp + b < p.ksplit && t0 + j < cnt &&
                                       in_bounds((size_t)(src - p.partial) + (size_t)(sp + b) * CH * kMoeNT +
                                                         (size_t)j * 128 < p.partial_floats, 0x405))
                                          ? __ldcg(src + (size_t)(sp + b) * CH * kMoeNT + (size_t)j * 128)
                                          : 0.f;
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (sp + b < p.ksplit)
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                v[j] += x[b][j];
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (t0 + j < cnt)
                        store_c(t0 + j, ch0, v[j], s0, b0);
            }
            if (warp == kEpilogueWarp0 && lane == 0)
                p.counters[nb] = 0u;  // ready for the next call
        }
    } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
        // ---- epilogue: lane = channel (TMEM lane quadrant warp % 4), column = token ----
        const int q = warp - kEpilogueWarp0;
        int t = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            const int e = it / p.nb, nb = it % p.nb;
            int r0, cnt, chunks;
            moe_rows(p, e, r0, cnt, chunks);
            const int chl = nb * CH + q * 32 + lane;  // output channel within the expert
            const uint16_t* se = p.scales + (size_t)e * p.rows_per_expert_w;
            const bool ch_ok = in_bounds((GATED ? p.inter : 128) * (TWO ? 1 : 0) + chl < p.rows_per_expert_w, 0x406);
            const float s0 = ch_ok ? to_f32<ACT>(ld_nc_u16(se + chl)) : 0.f;
            const float s1 = TWO && ch_ok ? to_f32<ACT>(ld_nc_u16(se + (GATED ? p.inter : 128) + chl)) : 0.f;
            bool ok = true;
            for (int ch = 0; ch < chunks; ++ch, ++t) {
                const int acc = t & 1;
                const bool got = mbar_wait_bounded(&bars->tfull[acc], (t >> 1) & 1, abort, p.err, 26,
                                                   kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got && !*abort)) {  // tcgen05.ld needs the whole warp
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the chunk's two partial accumulators (even and odd k blocks)
                const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(2 * acc * Cfg::COLS);
                const bool two_parts = p.num_kb > 1;
#pragma unroll 1
                for (int cc = 0; cc < kMoeNT / 32; ++cc) {
                    const int tok0 = ch * kMoeNT + cc * 32;
                    if (tok0 >= cnt)
                        break;  // warp-uniform
                    uint32_t r[32], u[32];
                    tmem_ld_32x32b_x32(tbase + (uint32_t)(cc * 32), r);
                    if constexpr (TWO)
                        tmem_ld_32x32b_x32(tbase + (uint32_t)(kMoeNT + cc * 32), u);
                    tmem_ld_wait();
                    if (two_parts) {
                        uint32_t r2[32];
                        tmem_ld_32x32b_x32(tbase + (uint32_t)(Cfg::COLS + cc * 32), r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                        if constexpr (TWO) {
                            tmem_ld_32x32b_x32(tbase + (uint32_t)(Cfg::COLS + kMoeNT + cc * 32), r2);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                u[j] = __float_as_uint(__uint_as_float(u[j]) + __uint_as_float(r2[j]));
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (tok0 + j < cnt &&  // rows past the expert's range are not its own
                            in_bounds(r0 + tok0 + j < p.rows_total &&
                                          chl + (WIDE ? 128 : 0) < (GATED ? p.inter : p.n_out), 0x407)) {
                            const size_t row = (size_t)(r0 + tok0 + j);
                            const float g = __uint_as_float(r[j]) * s0;
                            if constexpr (GATED) {
                                const float up = __uint_as_float(u[j]) * s1;
                                p.H[row * p.inter + chl] = from_f32<ACT>(g / (1.f + expf(-g)) * up);
                            } else {
                                p.Y[row * p.n_out + chl] = g;
                                if constexpr (WIDE)
                                    p.Y[row * p.n_out + chl + 128] = __uint_as_float(u[j]) * s1;
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->tempty[acc]);
            }
            if (!ok)
                break;
        }
    } else if (warp >= kDequantWarp0) {
        // ---- dequantisation: exact (q - 128) in the activation dtype ----
        const int dw = warp - kDequantWarp0;
        const DqScales<8, Cfg::WR> none{};
        int c = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            int e, nb, ks, kb0, kb1;
            moe_item(p, it, e, nb, ks, kb0, kb1);
            int r0, cnt, chunks;
            moe_rows(p, e, r0, cnt, chunks);
            for (int ch = 0; ch < chunks && ok; ++ch) {
                for (int kb = kb0; kb < kb1; ++kb, ++c) {
                    const int sc = c % Cfg::SC, s2 = c % Cfg::S2;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_bounded(&bars->fullC[sc], (c / Cfg::SC) & 1, abort, p.err,
                                                      24, kWaitLimitNs) &&
                                        mbar_wait_bounded(&bars->empty2[s2], ((c / Cfg::S2) & 1) ^ 1,
                                                          abort, p.err, 25, kWaitLimitNs))) {
                        ok = false;
                        break;
                    }
                    dequant_stage<8, ACT, ACT, Cfg::WR>(smem_addr(ringC + sc * Cfg::C_BYTES), none,
                                                        smem_addr(ring2 + s2 * Cfg::B_BYTES), dw, lane);
                    fence_proxy_async_smem();
                    mbar_arrive(&bars->full2[s2]);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars->emptyC[sc]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <bool GATED, bool WIDE, bool PLAIN, int ACT>
cudaError_t launch_moe_tc_t(const CUtensorMap& ma, const CUtensorMap& mc, const MoeTcParams& mp,
                            cudaStream_t s)
{
    constexpr int smem = MoeCfg<GATED || WIDE, PLAIN>::SMEM + (int)sizeof(Barriers) + 1024;
    static_assert(smem <= 232448, "shared memory per CTA");
    auto kern = moe_tc_kernel<GATED, WIDE, PLAIN, ACT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    const int items = PLAIN ? mp.nb * mp.ksplit : mp.E * mp.nb;
    const int grid = items < num_sms() ? items : num_sms();
    if constexpr (!PLAIN) {
        kern<<<grid, kThreads, smem, s>>>(ma, mc, mp);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mc, mp);
}

}  // namespace

TcPlan plan_tc(int m, int n, int k, int group, int bits, int act, bool allow_split)
{
    TcPlan p{};
    const TcShape sh = tc_shape(m, n, bits);
    p.bn = sh.bn;
    p.ms = sh.ms;
    p.splits = 1;
    const int num_kb = k / BK;
    const long long tiles256 = (long long)((m + BM - 1) / BM) * ((n + 255) / 256);
    if (allow_split && sh.ms == 1) {
        // too few 128 x 256 tiles for the SMs and a long k: split k instead of
        // narrowing the tiles (each unit keeps at least 48 k blocks, so the
        // partial tiles' round trip through the workspace stays small; the
        // per-tile counters live in the workspace's counter area)
        for (int sp = 8; sp >= 2; sp /= 2)
            if (num_kb % sp == 0 && num_kb / sp >= 48 && tiles256 * sp <= num_sms() &&
                tiles256 <= (long long)kWsCounters) {
                p.bn = 256;
                p.splits = sp;
                break;
            }
        // 128 x 128 tiles that fill at most half the SMs: split k in two when
        // each half keeps at least 24 k blocks (the partial round trip of a
        // 128 x 128 tile is a quarter of a 128 x 256 one's with four splits)
        const long long tiles128 = (long long)((m + BM - 1) / BM) * ((n + 127) / 128);
        if (p.splits == 1 && sh.bn == 128 && num_kb % 2 == 0 && num_kb / 2 >= 24 &&
            tiles128 * 2 <= num_sms() && tiles128 <= (long long)kWsCounters)
            p.splits = 2;
    }
    const long long tiles = (long long)((m + BM * p.ms - 1) / (BM * p.ms)) * ((n + p.bn - 1) / p.bn);
    p.a16_bytes = (bits == 4 && act == WO_BF16) ? align_up((size_t)m * k * 2, 256) : 0;
    p.rowscale_bytes = p.a16_bytes ? align_up((size_t)m * 4, 256) : 0;
    p.sz_bytes = bits == 4 ? align_up((size_t)n * (size_t)(k / group) * 4, 256) : 0;
    p.colscale_bytes = bits == 4 ? align_up((size_t)n * 2, 256) : 0;
    p.partial_bytes =
        p.splits > 1 ? align_up((size_t)tiles * p.splits * BM * p.ms * p.bn * 4, 256) : 0;
    p.ws_bytes = kWsScratch + p.a16_bytes + p.rowscale_bytes + p.sz_bytes + p.colscale_bytes +
                 p.partial_bytes;
    return p;
}

cudaError_t launch_tc(const GemmArgs& a, const TcPlan& plan, cudaStream_t s)
{
    char* ws = static_cast<char*>(a.ws);
    TcParams tp{};
    tp.m = a.m;
    tp.n = a.n;
    tp.k = a.k;
    tp.num_kb = a.k / BK;
    tp.scales = static_cast<const uint16_t*>(a.scales);
    tp.bias = static_cast<const uint16_t*>(a.bias);
    tp.C = static_cast<uint16_t*>(a.C);
    tp.G = a.k / a.group;
    tp.group = a.group;
    tp.c_v8 = reinterpret_cast<uintptr_t>(a.C) % 32 == 0 && a.n % 16 == 0;
    tp.err = reinterpret_cast<unsigned*>(ws);
    tp.splits = plan.splits;
    tp.counters = reinterpret_cast<unsigned*>(ws + kWsHeader);
    // scratch after the header and counters: [A16][rowscale][sz][colscale][partials]
    char* const a16_at = ws + kWsScratch;
    char* const rs_at = a16_at + plan.a16_bytes;
    char* const sz_at = rs_at + plan.rowscale_bytes;
    char* const cs_at = sz_at + plan.sz_bytes;
    char* const part_at = cs_at + plan.colscale_bytes;
    tp.partial = plan.splits > 1 ? reinterpret_cast<float*>(part_at) : nullptr;
    tp.partial_floats = plan.splits > 1 ? plan.partial_bytes / 4 : 0;
    // stream the larger operand once (A: m*k*2 bytes, codes: n*k*bits/8)
    tp.m_fast = (double)a.m * 2.0 <= (double)a.n * a.bits / 8.0;

    const void* Aop = a.A;
    if (a.bits == 4) {
        // the prepass: channel scales into fp16 range (and bf16 A into fp16)
        const int a_ctas = plan.a16_bytes ? a.m : 0;
        uint16_t* A16 = reinterpret_cast<uint16_t*>(a16_at);
        float* rsc = reinterpret_cast<float*>(rs_at);
        tp.sz = reinterpret_cast<const uint32_t*>(sz_at);
        tp.colscale = reinterpret_cast<const uint16_t*>(cs_at);
        const int ctas = a_ctas + (a.n + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
        auto prep = a.act == WO_F16 ? tc_prep_kernel<ACT_F16> : tc_prep_kernel<ACT_BF16>;
        prep<<<ctas, kPrepThreads, 0, s>>>(static_cast<const uint16_t*>(a.A), A16, rsc, a_ctas, a.k,
                                            static_cast<const uint16_t*>(a.scales),
                                            static_cast<const uint16_t*>(a.zeros), a.n, tp.G,
                                            reinterpret_cast<uint32_t*>(sz_at),
                                            reinterpret_cast<uint16_t*>(cs_at));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        if (a_ctas) {
            Aop = A16;
            tp.rowscale = rsc;
        }
    }
    const int OT = a.bits == 4 ? WO_F16 : a.act;
    CUtensorMap ma;
    if (!make_tmap_2d(&ma, OT == WO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      Aop, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2, BK, BM,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (a.bits == 8)
        return a.act == WO_F16 ? launch_tc_bn<8, ACT_F16, ACT_F16>(ma, a.B, tp, plan, s)
                               : launch_tc_bn<8, ACT_BF16, ACT_BF16>(ma, a.B, tp, plan, s);
    return a.act == WO_F16 ? launch_tc_bn<4, ACT_F16, ACT_F16>(ma, a.B, tp, plan, s)
                           : launch_tc_bn<4, ACT_F16, ACT_BF16>(ma, a.B, tp, plan, s);
}

}  // namespace wo

namespace wo {

bool moe_tc_supported(int hidden, int inter) { return hidden % 128 == 0 && inter % 128 == 0; }

cudaError_t launch_moe_tc(bool gated, int act, const void* rows, int total_rows, int k,
                          const uint8_t* codes, const void* scales, int experts, int n_out,
                          int inter, const int* offsets, void* out, unsigned* err, cudaStream_t s)
{
    MoeTcParams mp{};
    mp.offsets = offsets;
    mp.E = experts;
    // fc2 items of 256 channels when they tile the output (two MMAs per token
    // tile, half the token-row copies per weight byte), else 128
    const bool wide = !gated && n_out % 256 == 0;
    mp.nb = gated ? inter / 128 : n_out / (wide ? 256 : 128);
    mp.num_kb = k / BK;
    mp.inter = inter;
    mp.n_out = n_out;
    mp.rows_per_expert_w = gated ? 2 * inter : n_out;
    mp.scales = static_cast<const uint16_t*>(scales);
    mp.H = gated ? static_cast<uint16_t*>(out) : nullptr;
    mp.Y = gated ? nullptr : static_cast<float*>(out);
    mp.rows_total = total_rows;
    mp.err = err;
    // token rows: [total_rows, k], kMoeNT x 64 boxes, 128-byte swizzle
    CUtensorMap ma, mc;
    if (!make_tmap_2d(&ma, act == WO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      rows, (uint64_t)k, (uint64_t)total_rows, (uint64_t)k * 2, BK, kMoeNT,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // all experts' packed codes: one row per 16-channel block, k * 16 bytes each
    const uint64_t row_bytes = (uint64_t)k * 16;
    const uint64_t block_rows = (uint64_t)experts * mp.rows_per_expert_w / 16;
    if (!make_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, codes, row_bytes / 4, block_rows, row_bytes,
                      BK * 16 / 4, 8, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (gated)
        return act == WO_F16 ? launch_moe_tc_t<true, false, false, ACT_F16>(ma, mc, mp, s)
                             : launch_moe_tc_t<true, false, false, ACT_BF16>(ma, mc, mp, s);
    if (wide)
        return act == WO_F16 ? launch_moe_tc_t<false, true, false, ACT_F16>(ma, mc, mp, s)
                             : launch_moe_tc_t<false, true, false, ACT_BF16>(ma, mc, mp, s);
    return act == WO_F16 ? launch_moe_tc_t<false, false, false, ACT_F16>(ma, mc, mp, s)
                         : launch_moe_tc_t<false, false, false, ACT_BF16>(ma, mc, mp, s);
}

// ---- 8-bit weights at 17..64 rows: the swap-AB expert kernel as a plain GEMM

MidPlan plan_mid(int m, int n, int k, int bits)
{
    MidPlan P{};
    P.valid = false;
    if (bits != 8 || m < 1 || m > kMoeNT || n % 128 != 0 || k % BK != 0)
        return P;
    // blocks of 128 channels, the MMA's rows.  With more blocks than SMs the
    // m >= 65 tensor-core kernel (128 x 256 tiles, one MMA per 256 channels
    // and 16 k) streams the weights faster: this kernel is for the shapes
    // whose blocks alone leave SMs idle, which it fills by splitting k.
    P.ch = 128;
    P.nb = n / P.ch;
    if (P.nb > num_sms())
        return P;
    const int num_kb = k / BK;
    // as many (block, split) items as fit the SMs one each: an SM that ran a
    // second item would hold back the block its split belongs to, and the
    // last split's reduction behind it.  Each split keeps at least 4 k blocks;
    // at most 8 splits (the last split to arrive reads them all back).
    int ks = num_sms() / P.nb;
    const int ks_max = num_kb / 4 > 1 ? num_kb / 4 : 1;
    if (ks > ks_max)
        ks = ks_max;
    if (ks > 8)
        ks = 8;
    if (ks < 1)
        ks = 1;
    P.kps = (num_kb + ks - 1) / ks;
    P.ksplit = (num_kb + P.kps - 1) / P.kps;
    P.ctas = P.nb * P.ksplit;
    P.partial_bytes = P.ksplit > 1 ? align_up((size_t)P.nb * P.ksplit * P.ch * kMoeNT * 4, 256) : 0;
    P.ws_bytes = kWsScratch + P.partial_bytes;
    P.valid = (size_t)P.nb <= kWsCounters;
    return P;
}

cudaError_t launch_mid(const GemmArgs& a, cudaStream_t s)
{
    const MidPlan P = plan_mid(a.m, a.n, a.k, a.bits);
    if (!P.valid)
        return cudaErrorInvalidValue;
    MoeTcParams mp{};
    mp.offsets = nullptr;
    mp.E = 1;
    mp.nb = P.nb;
    mp.num_kb = a.k / BK;
    mp.n_out = a.n;
    mp.rows_per_expert_w = a.n;
    mp.scales = static_cast<const uint16_t*>(a.scales);
    mp.err = static_cast<unsigned*>(a.ws);
    mp.m = a.m;
    mp.ksplit = P.ksplit;
    mp.kps = P.kps;
    mp.bias = static_cast<const uint16_t*>(a.bias);
    mp.C = static_cast<uint16_t*>(a.C);
    char* ws = static_cast<char*>(a.ws);
    mp.counters = reinterpret_cast<unsigned*>(ws + kWsHeader);
    mp.partial = P.ksplit > 1 ? reinterpret_cast<float*>(ws + kWsScratch) : nullptr;
    mp.partial_floats = P.ksplit > 1 ? P.partial_bytes / 4 : 0;
    mp.rows_total = a.m;
    CUtensorMap ma, mc;
    if (!make_tmap_2d(&ma, a.act == WO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      a.A, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2, BK, kMoeNT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t row_bytes = (uint64_t)a.k * 16;
    if (!make_tmap_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.B, row_bytes / 4, (uint64_t)a.n / 16, row_bytes,
                      BK * 16 / 4, 8, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    return a.act == WO_F16 ? launch_moe_tc_t<false, false, true, ACT_F16>(ma, mc, mp, s)
                           : launch_moe_tc_t<false, false, true, ACT_BF16>(ma, mc, mp, s);
}

unsigned bounds_take_gemm_tc() { return bounds_take_local(); }

}  // namespace wo
