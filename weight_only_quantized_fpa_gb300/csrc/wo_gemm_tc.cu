// wo_gemm_tc.cu -- tensor-core kernel for large m:
//
//   C[m, n] = A[m, k] . dequant(B)^T + bias[n]
//
// "fpAintB uses mixed-precision quantization where weights are integers but
// are dequantized back to floating-point numbers before computation" (acext
// User Guide 1.3.4): here the dequantisation happens tile by tile in shared
// memory, feeding tcgen05 MMAs that accumulate in tensor memory.
//
// One CTA computes a 128 (m) x 256 (n) tile of C:
//   warp 0      TMA producer: A tile (128 x 64, 128-byte swizzle) and the
//               packed code tiles of 256 channels x 64 k into ring 1;
//   warp 1      allocates 256 TMEM columns; one lane issues the MMAs
//               (M=128, N=256, K=16, four per 64-wide k block) and commits
//               them to the ring barriers;
//   warps 4-11  dequantise ring-1 codes into ring 2: exact (q - 128) for
//               8-bit codes, fp16 round((q - 8) * s + z) for 4-bit group
//               codes, written with stmatrix straight into the K-major
//               128-byte-swizzled operand layout the MMA reads;
//   warps 4-7   after the last k block: the epilogue reads the fp32
//               accumulator (tcgen05.ld, one TMEM lane quadrant per warp),
//               applies scale[n] (8-bit) or the activation row scale
//               (4-bit), adds bias, rounds once and stores C.
// Every mbarrier wait is bounded: a wait that runs out records an error
// word in the workspace header and the CTA winds down (see the abort path).
//
// Operand types: 8-bit codes run the MMA in the activation dtype, in which
// q - 128 is exact.  4-bit codes run it in fp16: A is first converted to
// fp16 by a prepass with a per-row power-of-two scale (exact for bf16 values
// of normal range), and the weight is fp16 round((q - 8) * s + z) computed
// by one fused multiply-add per pair from the exact fp16 (q - 8).
#include "wo_common.cuh"
#include "wo_internal.h"
#include "wo_sm100.cuh"
#include "wo_tmap.h"

namespace wo {
namespace {

using namespace sm100;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kThreads = 384;       // 12 warps
constexpr int kDequantWarp0 = 4;    // warps 4..11 dequantise
constexpr int kDequantWarps = 8;
constexpr int kEpilogueWarp0 = 4;   // warps 4..7 run the epilogue
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

template <int BITS>
struct TcCfg {
    static constexpr int S1 = BITS == 8 ? 4 : 5;                // ring-1 stages
    static constexpr int S2 = 3;                                // ring-2 stages
    static constexpr int A_BYTES = BM * BK * 2;                 // 16 KiB
    static constexpr int CODE_BYTES = BN * BK * BITS / 8;       // 16 / 8 KiB
    static constexpr int STAGE1 = A_BYTES + CODE_BYTES;
    static constexpr int B_BYTES = BN * BK * 2;                 // 32 KiB
    static constexpr int TILES_PER_NB = BK / Geom<BITS>::KT;    // packed tiles per 16 rows
    static constexpr int SMEM = S1 * STAGE1 + S2 * B_BYTES;     // + barriers, see below
};

struct TcParams {
    int m, n, k;
    int num_kb;              // k / BK
    const uint16_t* scales;  // 8-bit: [n]; 4-bit: [n, G]
    const uint16_t* zeros;   // 4-bit only, [n, G] or null
    const uint16_t* bias;    // [n] or null
    const float* rowscale;   // 4-bit with a converted A: [m] powers of two; else null
    uint16_t* C;
    int G;                   // scale groups per channel row
    int group;               // codes per group
    unsigned* err;           // workspace error word
};

// Per-stage smem: ring-1 stage s = [A tile | code tiles], ring-2 stage = B tile.
struct Barriers {
    uint64_t full1[8], empty1[8], full2[4], empty2[4], accum;
    uint32_t tmem_base;
    int abort;
};

template <int BITS, int OT, int ACT>
__device__ __forceinline__ void dequant_stage(const TcParams& p, uint32_t codes_s, uint32_t b_s,
                                              int n0, int kb, int dw, int lane)
{
    constexpr int KT = Geom<BITS>::KT;
    constexpr int KS = Geom<BITS>::KSTEPS;
    constexpr int TPN = TcCfg<BITS>::TILES_PER_NB;
    constexpr int NT = (BN / 16) * TPN;  // packed tiles per stage
    const int g = lane >> 2;
    const int mi = lane >> 3, r8 = lane & 7;
    for (int tile = dw; tile < NT; tile += kDequantWarps) {
        const int nb = tile / TPN;          // 16-row block within the 256-row tile
        const int tl = tile % TPN;          // tile within the 64-wide k block
        const uint4 v = lds128(codes_s + (uint32_t)(nb * TPN + tl) * kTileBytes + lane * 16);
        uint32_t s2lo = 0, s2hi = 0, z2lo = 0, z2hi = 0;
        if constexpr (BITS == 4) {
            // scale and zero of this lane's two rows for this k block's group,
            // as fp16 pairs (exact for values in fp16's normal range)
            const int gi = (kb * BK) / p.group;
            const int nlo = n0 + nb * 16 + g;
            float slo = 0.f, shi = 0.f, zlo = 0.f, zhi = 0.f;
            if (nlo < p.n) {
                slo = to_f32<ACT>(ld_nc_u16(p.scales + (size_t)nlo * p.G + gi));
                shi = to_f32<ACT>(ld_nc_u16(p.scales + (size_t)(nlo + 8) * p.G + gi));
                if (p.zeros) {
                    zlo = to_f32<ACT>(ld_nc_u16(p.zeros + (size_t)nlo * p.G + gi));
                    zhi = to_f32<ACT>(ld_nc_u16(p.zeros + (size_t)(nlo + 8) * p.G + gi));
                }
            }
            const uint32_t hs_lo = from_f32<ACT_F16>(slo), hs_hi = from_f32<ACT_F16>(shi);
            const uint32_t hz_lo = from_f32<ACT_F16>(zlo), hz_hi = from_f32<ACT_F16>(zhi);
            s2lo = hs_lo | (hs_lo << 16);
            s2hi = hs_hi | (hs_hi << 16);
            z2lo = hz_lo | (hz_lo << 16);
            z2hi = hz_hi | (hz_hi << 16);
        }
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            uint32_t a[4];
            if constexpr (BITS == 8) {
                tile_frag<8, OT>(v, s, a);
            } else {
                const uint32_t w = s == 0 ? v.x : s == 1 ? v.y : s == 2 ? v.z : v.w;
                a[0] = fma_f16x2(cvt_u4x2<ACT_F16>(w), s2lo, z2lo);
                a[1] = fma_f16x2(cvt_u4x2<ACT_F16>(w >> 4), s2hi, z2hi);
                a[2] = fma_f16x2(cvt_u4x2<ACT_F16>(w >> 8), s2lo, z2lo);
                a[3] = fma_f16x2(cvt_u4x2<ACT_F16>(w >> 12), s2hi, z2hi);
            }
            // lane -> row address of matrix mi: rows r8 (+8 for mi odd), k
            // chunk of 8 codes (+1 for mi >= 2)
            const int row = nb * 16 + r8 + 8 * (mi & 1);
            const int chunk = (tl * KT + 16 * s) / 8 + (mi >> 1);
            const uint32_t addr = b_s + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u +
                                  (uint32_t)((chunk ^ (row & 7)) << 4);
            stmatrix_x4(addr, a[0], a[1], a[2], a[3]);
        }
    }
}

template <int BITS, int OT, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p)
{
    using Cfg = TcCfg<BITS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ring1 = smem;
    uint8_t* ring2 = smem + Cfg::S1 * Cfg::STAGE1;
    Barriers* bars = reinterpret_cast<Barriers*>(ring2 + Cfg::S2 * Cfg::B_BYTES);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int num_kb = p.num_kb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::S1; ++s) {
            mbar_init(&bars->full1[s], 1);
            mbar_init(&bars->empty1[s], 1);
        }
        for (int s = 0; s < Cfg::S2; ++s) {
            mbar_init(&bars->full2[s], kDequantWarps * 32);
            mbar_init(&bars->empty2[s], 1);
        }
        mbar_init(&bars->accum, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            int issued = 0;
            for (int i = 0; i < num_kb; ++i) {
                const int s = i % Cfg::S1;
                if (!mbar_wait_bounded(&bars->empty1[s], ((i / Cfg::S1) & 1) ^ 1, abort, p.err, 1,
                                       kWaitLimitNs))
                    break;
                uint8_t* st = ring1 + s * Cfg::STAGE1;
                mbar_arrive_expect_tx(&bars->full1[s], Cfg::STAGE1);
                tma_load_2d(st, &tmA, &bars->full1[s], i * BK, m0);
                // codes: row = 16-channel block, x in 32-bit words
                tma_load_2d(st + Cfg::A_BYTES, &tmB, &bars->full1[s], i * (BK * BITS / 8 * 16 / 4),
                            n0 / 16);
                issued = i + 1;
            }
            if (*abort) {
                // let the copies already issued land before the CTA exits
                volatile int never = 0;
                for (int i = issued - Cfg::S1 > 0 ? issued - Cfg::S1 : 0; i < issued; ++i)
                    mbar_wait_bounded(&bars->full1[i % Cfg::S1], (i / Cfg::S1) & 1, &never,
                                      nullptr, 0, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            constexpr uint32_t idesc = idesc_f16(OT == ACT_BF16 ? 1u : 0u, BM, BN);
            for (int i = 0; i < num_kb; ++i) {
                const int s1 = i % Cfg::S1, s2 = i % Cfg::S2;
                if (!mbar_wait_bounded(&bars->full1[s1], (i / Cfg::S1) & 1, abort, p.err, 2,
                                       kWaitLimitNs))
                    break;
                if (!mbar_wait_bounded(&bars->full2[s2], (i / Cfg::S2) & 1, abort, p.err, 3,
                                       kWaitLimitNs))
                    break;
                tc_fence_after();
                const uint32_t a_s = smem_addr(ring1 + s1 * Cfg::STAGE1);
                const uint32_t b_s = smem_addr(ring2 + s2 * Cfg::B_BYTES);
                const uint64_t ad = desc_sw128(a_s), bd = desc_sw128(b_s);
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)  // +32 bytes per 16-wide k step
                    mma_f16(tmem, ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j), idesc,
                            (i > 0 || j > 0) ? 1u : 0u);
                mma_commit(&bars->empty1[s1]);
                mma_commit(&bars->empty2[s2]);
            }
            // accumulator complete (also on abort, so the epilogue and the
            // TMEM release wait for every MMA already issued)
            mma_commit(&bars->accum);
        }
    } else if (warp >= kDequantWarp0) {
        // ---- dequantisation ----
        const int dw = warp - kDequantWarp0;
        for (int i = 0; i < num_kb; ++i) {
            const int s1 = i % Cfg::S1, s2 = i % Cfg::S2;
            // warp-uniform decisions: stmatrix below needs the whole warp
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars->full1[s1], (i / Cfg::S1) & 1,
                                                           abort, p.err, 4, kWaitLimitNs)))
                break;
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(&bars->empty2[s2], ((i / Cfg::S2) & 1) ^ 1, abort,
                                              p.err, 5, kWaitLimitNs)))
                break;
            dequant_stage<BITS, OT, ACT>(p, smem_addr(ring1 + s1 * Cfg::STAGE1 + Cfg::A_BYTES),
                                         smem_addr(ring2 + s2 * Cfg::B_BYTES), n0, i, dw, lane);
            fence_proxy_async_smem();
            mbar_arrive(&bars->full2[s2]);
        }
        // ---- epilogue ----
        if (warp < kEpilogueWarp0 + 4) {
            const int q = warp - kEpilogueWarp0;  // TMEM lane quadrant
            bool ok = mbar_wait_bounded(&bars->accum, 0, abort, p.err, 6, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok && !*abort);  // tcgen05.ld needs the whole warp
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            float rs = 1.f;
            if (p.rowscale && row < p.m)
                rs = p.rowscale[row];
            if (ok) {
                for (int c = 0; c < BN / 32; ++c) {
                    const int nc = n0 + c * 32;
                    if (nc >= p.n)
                        break;
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), r);
                    tmem_ld_wait();
                    if (row < p.m) {
                        uint32_t packed[16];
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float v0 = __uint_as_float(r[j]), v1 = __uint_as_float(r[j + 1]);
                            if constexpr (BITS == 8) {
                                v0 *= to_f32<ACT>(ld_nc_u16(p.scales + nc + j));
                                v1 *= to_f32<ACT>(ld_nc_u16(p.scales + nc + j + 1));
                            } else {
                                v0 *= rs;
                                v1 *= rs;
                            }
                            if (p.bias) {
                                v0 += to_f32<ACT>(ld_nc_u16(p.bias + nc + j));
                                v1 += to_f32<ACT>(ld_nc_u16(p.bias + nc + j + 1));
                            }
                            packed[j / 2] = (uint32_t)from_f32<ACT>(v0) |
                                            ((uint32_t)from_f32<ACT>(v1) << 16);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(p.C + (size_t)row * p.n + nc);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                                packed[4 * v + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// A bf16 -> fp16 with a per-row power-of-two scale: row r is multiplied by
// 2^-E (E chosen so max |a| * 2^-E lies in [2^14, 2^15)), which is exact,
// then rounded to fp16, which is exact for bf16 values whose scaled
// magnitude is at least 2^-14; rowscale[r] = 2^E undoes it in the epilogue.
__global__ void a_to_f16_kernel(const uint16_t* __restrict__ A, uint16_t* __restrict__ A16,
                                float* __restrict__ rowscale, int m, int k)
{
    const int row = blockIdx.x;
    if (row >= m)
        return;
    const uint16_t* a = A + (size_t)row * k;
    float mx = 0.f;
    for (int c = threadIdx.x; c < k; c += blockDim.x)
        mx = fmaxf(mx, fabsf(to_f32<ACT_BF16>(a[c])));
    __shared__ float red[32];
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1)
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
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
    for (int c = threadIdx.x; c < k; c += blockDim.x)
        A16[(size_t)row * k + c] = from_f32<ACT_F16>(to_f32<ACT_BF16>(a[c]) * inv);
    if (threadIdx.x == 0)
        rowscale[row] = ldexpf(1.f, E);
}

template <int BITS, int OT, int ACT>
cudaError_t launch_tc_t(const CUtensorMap& ma, const CUtensorMap& mb, const TcParams& tp,
                        cudaStream_t s)
{
    constexpr int smem = TcCfg<BITS>::SMEM + (int)sizeof(Barriers) + 1024;
    auto kern = gemm_tc_kernel<BITS, OT, ACT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((tp.n + BN - 1) / BN, (tp.m + BM - 1) / BM);
    kern<<<grid, kThreads, smem, s>>>(ma, mb, tp);
    return cudaGetLastError();
}

}  // namespace

TcPlan plan_tc(int m, int n, int k, int bits, int act)
{
    TcPlan p{};
    p.a16_bytes = (bits == 4 && act == WO_BF16) ? align_up((size_t)m * k * 2, 256) : 0;
    p.rowscale_bytes = p.a16_bytes ? align_up((size_t)m * 4, 256) : 0;
    p.ws_bytes = kWsScratch + p.a16_bytes + p.rowscale_bytes;
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
    tp.zeros = static_cast<const uint16_t*>(a.zeros);
    tp.bias = static_cast<const uint16_t*>(a.bias);
    tp.C = static_cast<uint16_t*>(a.C);
    tp.G = a.k / a.group;
    tp.group = a.group;
    tp.err = reinterpret_cast<unsigned*>(ws);

    const void* Aop = a.A;
    if (plan.a16_bytes) {
        uint16_t* A16 = reinterpret_cast<uint16_t*>(ws + kWsScratch);
        float* rsc = reinterpret_cast<float*>(ws + kWsScratch + plan.a16_bytes);
        a_to_f16_kernel<<<a.m, 256, 0, s>>>(static_cast<const uint16_t*>(a.A), A16, rsc, a.m, a.k);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        Aop = A16;
        tp.rowscale = rsc;
    }
    const int OT = a.bits == 4 ? WO_F16 : a.act;
    CUtensorMap ma, mb;
    if (!make_tmap_2d(&ma, OT == WO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  Aop, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2, BK, BM,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // packed codes viewed as [n/16 rows] x [bytes per 16-channel row / 4] words
    const uint64_t row_bytes = (uint64_t)a.k * 16 * a.bits / 8;
    if (!make_tmap_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.B, row_bytes / 4, (uint64_t)a.n / 16,
                  row_bytes, BK * 16 * a.bits / 8 / 4, BN / 16, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (a.bits == 8)
        return a.act == WO_F16 ? launch_tc_t<8, ACT_F16, ACT_F16>(ma, mb, tp, s)
                               : launch_tc_t<8, ACT_BF16, ACT_BF16>(ma, mb, tp, s);
    return a.act == WO_F16 ? launch_tc_t<4, ACT_F16, ACT_F16>(ma, mb, tp, s)
                           : launch_tc_t<4, ACT_F16, ACT_BF16>(ma, mb, tp, s);
}

}  // namespace wo
