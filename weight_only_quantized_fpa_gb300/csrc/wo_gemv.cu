// wo_gemv.cu -- weight-streaming kernel for small m (decode):
//
//   C[m, n] = A[m, k] . dequant(B)^T + bias[n]      (m <= 64 per launch)
//
// At small m the whole packed weight matrix is read once per call and the
// arithmetic per weight byte is tiny, so the kernel is bound by HBM
// bandwidth (the point made in vLLM-Omni "cpu_int4.py"'s module docstring:
// the bits per weight, not the FLOPs, set the decode rate).
//
// Design:
//   - a warp owns kRpw blocks of 16 output channels and a slice of k; each
//     lane streams its 16 bytes of every 512-byte packed tile with 128-bit
//     non-caching loads (kUnroll tiles in flight per block);
//   - the codes are turned into exact (q - offset) fp16/bf16 pairs in
//     registers (wo_common.cuh) that are directly the A fragments of
//     mma.m16n8k16; activations form the B fragments (8 rows of A per mma,
//     zero rows past m), accumulation in fp32.  At m = 16 and 8-bit codes
//     the kernel needs 2*16 FLOP per weight byte, beyond the CUDA cores at
//     HBM rate, hence the tensor-core FMA;
//   - 4-bit group-wise weights (acext 1.3.3, w = (q - 8) s + z): each group's
//     partial sum P_g = sum a (q - 8) and the group's activation sum R_g
//     (an mma against a ones fragment) are folded as
//     acc += s[n][g] * P_g + z[n][g] * R_g in fp32, so the tensor cores only
//     ever see exact integers;
//   - 8-bit per-channel weights (acext 1.3.1) accumulate sum a (q - 128) and
//     apply scale[n] and bias[n] once at the end;
//   - split-K: CTAs along grid.y take slices of k; each writes its fp32
//     partials to the workspace, and the last CTA to arrive (an atomic
//     counter, no waiting) sums the slices in fixed order, applies the
//     epilogue and resets the counter.  The result does not depend on the
//     arrival order.
#include "wo_common.cuh"
#include "wo_internal.h"

namespace wo {
namespace {

constexpr int kWarps = 4;
constexpr int kRpw = 2;                      // 16-row channel blocks per warp
constexpr int kCtaCols = kWarps * kRpw * 16; // output channels per CTA

struct GemvParams {
    const uint16_t* A;
    const uint8_t* B;
    const uint16_t* scales;
    const uint16_t* zeros;
    const uint16_t* bias;
    uint16_t* C;
    int m, n, k;
    int G;               // scale columns per channel row
    int tiles_per_group; // k-tiles per scale group
    int ktiles, ktiles_per_split, splits;
    float* part;
    unsigned* counters;
};

template <int BITS, int ACT, int MT, bool GROUPED>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const GemvParams p)
{
    constexpr int KT = Geom<BITS>::KT;
    constexpr int KS = Geom<BITS>::KSTEPS;
    constexpr int kUnroll = MT >= 4 ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nblocks = p.n >> 4;
    const int nb0 = (blockIdx.x * kWarps + warp) * kRpw;
    // n % 64 == 0 makes nblocks a multiple of 4, so a warp is either wholly
    // inside or wholly past the last channel block.
    const bool active = nb0 < nblocks;
    const int kt0 = blockIdx.y * p.ktiles_per_split;
    const int kt1 = min(kt0 + p.ktiles_per_split, p.ktiles);

    float acc[kRpw][MT][4];
    float gp[kRpw][MT][4];
    float rs[MT][4];
#pragma unroll
    for (int r = 0; r < kRpw; ++r)
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[r][j][e] = 0.f;
                gp[r][j][e] = 0.f;
            }
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            rs[j][e] = 0.f;

    const uint16_t* arow[MT];
    bool aval[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        const int r = 8 * j + g;
        aval[j] = r < p.m;
        arow[j] = p.A + (size_t)(aval[j] ? r : 0) * p.k + 2 * t;
    }

    if (active) {
        const uint8_t* wp[kRpw];
#pragma unroll
        for (int r = 0; r < kRpw; ++r)
            wp[r] = p.B + ((size_t)(nb0 + r) * p.ktiles + kt0) * kTileBytes + lane * 16;

        for (int kt = kt0; kt < kt1; kt += kUnroll) {
            uint4 wv[kUnroll][kRpw];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int r = 0; r < kRpw; ++r)
                    if (kt + u < kt1)
                        wv[u][r] = ld_stream_v4(wp[r] + (size_t)(kt - kt0 + u) * kTileBytes);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int ktile = kt + u;
                if (ktile < kt1) {
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        uint32_t bf[MT][2];
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            if (aval[j]) {
                                const uint16_t* ap = arow[j] + ktile * KT + 16 * s;
                                bf[j][0] = ld_nc_u32(ap);
                                bf[j][1] = ld_nc_u32(ap + 8);
                            } else {
                                bf[j][0] = 0u;
                                bf[j][1] = 0u;
                            }
                        }
#pragma unroll
                        for (int r = 0; r < kRpw; ++r) {
                            uint32_t a[4];
                            tile_frag<BITS, ACT>(wv[u][r], s, a);
#pragma unroll
                            for (int j = 0; j < MT; ++j) {
                                if constexpr (GROUPED)
                                    mma16816<ACT>(gp[r][j], a, bf[j][0], bf[j][1]);
                                else
                                    mma16816<ACT>(acc[r][j], a, bf[j][0], bf[j][1]);
                            }
                        }
                        if constexpr (GROUPED) {
                            const uint32_t one = ones_x2<ACT>();
                            const uint32_t ones[4] = {one, one, one, one};
#pragma unroll
                            for (int j = 0; j < MT; ++j)
                                mma16816<ACT>(rs[j], ones, bf[j][0], bf[j][1]);
                        }
                    }
                    if constexpr (GROUPED) {
                        const bool flush =
                            ((ktile + 1) % p.tiles_per_group == 0) || (ktile + 1 == kt1);
                        if (flush) {
                            const int gi = ktile / p.tiles_per_group;
#pragma unroll
                            for (int r = 0; r < kRpw; ++r) {
                                const size_t nlo = (size_t)(nb0 + r) * 16 + g;
                                const float s_lo = to_f32<ACT>(ld_nc_u16(p.scales + nlo * p.G + gi));
                                const float s_hi =
                                    to_f32<ACT>(ld_nc_u16(p.scales + (nlo + 8) * p.G + gi));
                                float z_lo = 0.f, z_hi = 0.f;
                                if (p.zeros) {
                                    z_lo = to_f32<ACT>(ld_nc_u16(p.zeros + nlo * p.G + gi));
                                    z_hi = to_f32<ACT>(ld_nc_u16(p.zeros + (nlo + 8) * p.G + gi));
                                }
#pragma unroll
                                for (int j = 0; j < MT; ++j) {
                                    acc[r][j][0] = fmaf(s_lo, gp[r][j][0], fmaf(z_lo, rs[j][0], acc[r][j][0]));
                                    acc[r][j][1] = fmaf(s_lo, gp[r][j][1], fmaf(z_lo, rs[j][1], acc[r][j][1]));
                                    acc[r][j][2] = fmaf(s_hi, gp[r][j][2], fmaf(z_hi, rs[j][2], acc[r][j][2]));
                                    acc[r][j][3] = fmaf(s_hi, gp[r][j][3], fmaf(z_hi, rs[j][3], acc[r][j][3]));
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        gp[r][j][e] = 0.f;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < MT; ++j)
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    rs[j][e] = 0.f;
                        }
                    }
                }
            }
        }
    }

    // Accumulator element e of (r, j): channel n = 16*(nb0 + r) + g + 8*(e >> 1),
    // activation row m = 8*j + 2*t + (e & 1).
    if (p.splits == 1) {
        if (!active)
            return;
#pragma unroll
        for (int r = 0; r < kRpw; ++r)
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int nn = (nb0 + r) * 16 + g + 8 * (e >> 1);
                    const int mm = 8 * j + 2 * t + (e & 1);
                    if (mm < p.m) {
                        float v = acc[r][j][e];
                        if constexpr (!GROUPED)
                            v *= to_f32<ACT>(ld_nc_u16(p.scales + nn));
                        if (p.bias)
                            v += to_f32<ACT>(ld_nc_u16(p.bias + nn));
                        p.C[(size_t)mm * p.n + nn] = from_f32<ACT>(v);
                    }
                }
        return;
    }

    if (active) {
#pragma unroll
        for (int r = 0; r < kRpw; ++r)
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int nn = (nb0 + r) * 16 + g + 8 * (e >> 1);
                    const int mm = 8 * j + 2 * t + (e & 1);
                    if (mm < p.m)
                        p.part[((size_t)blockIdx.y * p.m + mm) * p.n + nn] = acc[r][j][e];
                }
    }
    __threadfence();
    __syncthreads();
    __shared__ unsigned s_prev;
    if (threadIdx.x == 0)
        s_prev = atomicAdd(&p.counters[blockIdx.x], 1u);
    __syncthreads();
    if (s_prev != (unsigned)(p.splits - 1))
        return;
    __threadfence();
    const int n0 = blockIdx.x * kCtaCols;
    for (int idx = threadIdx.x; idx < p.m * kCtaCols; idx += blockDim.x) {
        const int mm = idx / kCtaCols;
        const int nn = n0 + idx % kCtaCols;
        if (nn >= p.n)
            continue;
        float v = 0.f;
        for (int s = 0; s < p.splits; ++s)
            v += __ldcg(p.part + ((size_t)s * p.m + mm) * p.n + nn);
        if constexpr (!GROUPED)
            v *= to_f32<ACT>(ld_nc_u16(p.scales + nn));
        if (p.bias)
            v += to_f32<ACT>(ld_nc_u16(p.bias + nn));
        p.C[(size_t)mm * p.n + nn] = from_f32<ACT>(v);
    }
    if (threadIdx.x == 0)
        p.counters[blockIdx.x] = 0u;
}

template <int BITS, int ACT, bool GROUPED>
cudaError_t launch_mt(int mt, dim3 grid, const GemvParams& gp, cudaStream_t s)
{
    const dim3 block(kWarps * 32);
    switch (mt) {
    case 1: gemv_kernel<BITS, ACT, 1, GROUPED><<<grid, block, 0, s>>>(gp); break;
    case 2: gemv_kernel<BITS, ACT, 2, GROUPED><<<grid, block, 0, s>>>(gp); break;
    case 4: gemv_kernel<BITS, ACT, 4, GROUPED><<<grid, block, 0, s>>>(gp); break;
    default: gemv_kernel<BITS, ACT, 8, GROUPED><<<grid, block, 0, s>>>(gp); break;
    }
    return cudaGetLastError();
}

}  // namespace

GemvPlan plan_gemv(int m, int n, int k, int bits)
{
    GemvPlan p{};
    const int rows = m < 64 ? m : 64;
    p.mt = rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;
    p.m_per_pass = 8 * p.mt;
    p.passes = (m + p.m_per_pass - 1) / p.m_per_pass;
    p.grid_x = (n + kCtaCols - 1) / kCtaCols;
    const int KT = bits == 8 ? 32 : 64;
    p.ktiles = k / KT;
    const int target = num_sms() * 8;  // 128-thread CTAs that keep every SM streaming
    int splits = (target + p.grid_x - 1) / p.grid_x;
    int cap = p.ktiles / 4;
    if (cap < 1)
        cap = 1;
    if (cap > 64)
        cap = 64;
    if (splits > cap)
        splits = cap;
    if (splits < 1)
        splits = 1;
    p.ktiles_per_split = (p.ktiles + splits - 1) / splits;
    p.splits = (p.ktiles + p.ktiles_per_split - 1) / p.ktiles_per_split;
    const int prow = m < p.m_per_pass ? m : p.m_per_pass;
    p.ws_partials = p.splits > 1 ? align_up((size_t)p.splits * prow * n * 4, 256) : 0;
    p.ws_bytes = p.splits > 1 ? kWsScratch + p.ws_partials : 0;
    return p;
}

cudaError_t launch_gemv(const GemmArgs& a, const GemvPlan& p, cudaStream_t s)
{
    GemvParams gp{};
    gp.B = a.B;
    gp.scales = static_cast<const uint16_t*>(a.scales);
    gp.zeros = static_cast<const uint16_t*>(a.zeros);
    gp.bias = static_cast<const uint16_t*>(a.bias);
    gp.n = a.n;
    gp.k = a.k;
    gp.G = a.k / a.group;
    const int KT = a.bits == 8 ? 32 : 64;
    gp.tiles_per_group = a.group / KT;
    gp.ktiles = p.ktiles;
    gp.ktiles_per_split = p.ktiles_per_split;
    gp.splits = p.splits;
    char* ws = static_cast<char*>(a.ws);
    gp.counters = p.splits > 1 ? reinterpret_cast<unsigned*>(ws + kWsHeader) : nullptr;
    gp.part = p.splits > 1 ? reinterpret_cast<float*>(ws + kWsScratch) : nullptr;
    const dim3 grid(p.grid_x, p.splits);
    for (int pass = 0; pass < p.passes; ++pass) {
        const int m0 = pass * p.m_per_pass;
        const int rows = a.m - m0 < p.m_per_pass ? a.m - m0 : p.m_per_pass;
        gp.m = rows;
        gp.A = static_cast<const uint16_t*>(a.A) + (size_t)m0 * a.k;
        gp.C = static_cast<uint16_t*>(a.C) + (size_t)m0 * a.n;
        cudaError_t e;
        if (a.bits == 8) {
            e = a.act == WO_F16 ? launch_mt<8, ACT_F16, false>(p.mt, grid, gp, s)
                                : launch_mt<8, ACT_BF16, false>(p.mt, grid, gp, s);
        } else {
            e = a.act == WO_F16 ? launch_mt<4, ACT_F16, true>(p.mt, grid, gp, s)
                                : launch_mt<4, ACT_BF16, true>(p.mt, grid, gp, s);
        }
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace wo
