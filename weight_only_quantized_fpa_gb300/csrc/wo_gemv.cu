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
//     non-caching loads, kDepth tiles in flight per block (a rolling
//     register prefetch that never drains until the slice ends);
//   - the CTA's slice of the activations (and, for 4-bit weights, the scales
//     and zeros of its channels and groups) is staged in shared memory once,
//     after the first weight loads are in flight, so the inner loop waits on
//     weights only;
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
//   - split-K without a workspace: the 8 warps of a CTA share the same 32
//     channels and stream consecutive slices of the CTA's k range (each
//     keeping kDepth tiles in flight), then reduce through shared memory in
//     fixed warp order; when k is long relative to n, a thread-block cluster
//     of up to 8 CTAs along k splits it further and the leader CTA sums the
//     members' results through distributed shared memory, in rank order.
//     The result does not depend on timing: it is bit-for-bit repeatable.
#include <cooperative_groups.h>

#include "wo_common.cuh"
#include "wo_internal.h"

namespace wo {
namespace {

namespace cg = cooperative_groups;

constexpr int kWarps = 8;
constexpr int kRpw = 2;                 // 16-row channel blocks per CTA (all warps share them)
constexpr int kCtaCols = kRpw * 16;     // output channels per CTA
constexpr int kMaxCluster = 8;
constexpr int kAsmemBudget = 64 * 1024; // bytes of staged activations per CTA

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
    int a_stride;        // bytes per staged activation row (ktiles_per_split * KT * 2 + 16)
    int a_rows;          // staged activation rows (min(m, 8 * MT))
    int g_span;          // scale groups staged per channel (4-bit)
};

template <int MT>
__host__ __device__ constexpr int red_floats()  // accumulator floats of one warp
{
    return kRpw * MT * 4 * 32;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

template <int BITS, int ACT, int MT, bool GROUPED>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const GemvParams p)
{
    constexpr int KT = Geom<BITS>::KT;
    constexpr int KS = Geom<BITS>::KSTEPS;
    constexpr int kDepth = MT <= 2 ? 4 : 2;  // tiles in flight per warp
    constexpr int RF = red_floats<MT>();
    // shared memory: [kWarps + 1][RF] floats (reduction), the staged
    // activations [a_rows][a_stride bytes], then (4-bit) scales and zeros
    // [kCtaCols][g_span] each as 16-bit values
    extern __shared__ __align__(16) float red[];
    uint8_t* a_sm = reinterpret_cast<uint8_t*>(red + (kWarps + 1) * RF);
    uint16_t* s_sm = reinterpret_cast<uint16_t*>(a_sm + p.a_rows * p.a_stride);
    uint16_t* z_sm = s_sm + kCtaCols * p.g_span;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nb0 = blockIdx.x * kRpw;       // n % 64 == 0: both blocks exist
    // this CTA's k range, then this warp's slice of it
    const int c0 = blockIdx.y * p.ktiles_per_split;
    const int c1 = min(c0 + p.ktiles_per_split, p.ktiles);
    const int per_warp = (c1 - c0 + kWarps - 1) / kWarps;
    const int kt0 = min(c0 + warp * per_warp, c1);
    const int kt1 = min(kt0 + per_warp, c1);
    const int nt = kt1 - kt0;
    const int g_lo = GROUPED ? c0 / p.tiles_per_group : 0;

    const uint8_t* wp[kRpw];
#pragma unroll
    for (int r = 0; r < kRpw; ++r)
        wp[r] = p.B + ((size_t)(nb0 + r) * p.ktiles + kt0) * kTileBytes + lane * 16;

    // rolling prefetch: buf[u] holds tile (base + u) while it is consumed and
    // is refilled with tile (base + u + kDepth) right after
    uint4 buf[kDepth][kRpw];
#pragma unroll
    for (int u = 0; u < kDepth; ++u)
#pragma unroll
        for (int r = 0; r < kRpw; ++r)
            if (u < nt)
                buf[u][r] = ld_stream_v4(wp[r] + (size_t)u * kTileBytes);

    // ---- stage this CTA's activations (and 4-bit scales/zeros) ----
    {
        const int cols8 = (c1 - c0) * KT / 8;  // 16-byte pieces per row
        const int total = p.a_rows * cols8;
        const uint32_t a_base = static_cast<uint32_t>(__cvta_generic_to_shared(a_sm));
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int row = idx / cols8, c8 = idx % cols8;
            cp_async16(a_base + row * p.a_stride + c8 * 16,
                       p.A + (size_t)row * p.k + (size_t)c0 * KT + c8 * 8);
        }
        if constexpr (GROUPED) {
            const int g_hi = (c1 - 1) / p.tiles_per_group;
            const int gc = g_hi - g_lo + 1;
            for (int idx = threadIdx.x; idx < kCtaCols * gc; idx += blockDim.x) {
                const int ch = idx / gc, gg = idx % gc;
                const size_t src = (size_t)(nb0 * 16 + ch) * p.G + g_lo + gg;
                s_sm[ch * p.g_span + gg] = ld_nc_u16(p.scales + src);
                z_sm[ch * p.g_span + gg] = p.zeros ? ld_nc_u16(p.zeros + src) : (uint16_t)0;
            }
        }
        cp_async_wait_all();
        __syncthreads();
    }

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

    // B-fragment addresses in the staged activations: row 8j + g, k pair 2t
    uint32_t arow[MT];
    bool aval[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        const int r = 8 * j + g;
        aval[j] = r < p.m;
        arow[j] = static_cast<uint32_t>(__cvta_generic_to_shared(a_sm)) +
                  (aval[j] ? r : 0) * p.a_stride + 4 * t;
    }

    for (int base = 0; base < nt; base += kDepth) {
#pragma unroll
        for (int u = 0; u < kDepth; ++u) {
            const int i = base + u;
            if (i < nt) {
                uint4 cur[kRpw];
#pragma unroll
                for (int r = 0; r < kRpw; ++r) {
                    cur[r] = buf[u][r];
                    if (i + kDepth < nt)
                        buf[u][r] = ld_stream_v4(wp[r] + (size_t)(i + kDepth) * kTileBytes);
                }
                const int ktile = kt0 + i;
                const uint32_t koff = (uint32_t)((ktile - c0) * KT * 2);
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    uint32_t bf[MT][2];
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        if (aval[j]) {
                            const uint32_t ap = arow[j] + koff + 32 * s;
                            bf[j][0] = lds32(ap);
                            bf[j][1] = lds32(ap + 16);
                        } else {
                            bf[j][0] = 0u;
                            bf[j][1] = 0u;
                        }
                    }
#pragma unroll
                    for (int r = 0; r < kRpw; ++r) {
                        uint32_t a[4];
                        tile_frag<BITS, ACT>(cur[r], s, a);
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
                    if (((ktile + 1) % p.tiles_per_group == 0) || (i + 1 == nt)) {
                        const int gl = ktile / p.tiles_per_group - g_lo;
#pragma unroll
                        for (int r = 0; r < kRpw; ++r) {
                            const int ch = r * 16 + g;
                            const float s_lo = to_f32<ACT>(s_sm[ch * p.g_span + gl]);
                            const float s_hi = to_f32<ACT>(s_sm[(ch + 8) * p.g_span + gl]);
                            const float z_lo = to_f32<ACT>(z_sm[ch * p.g_span + gl]);
                            const float z_hi = to_f32<ACT>(z_sm[(ch + 8) * p.g_span + gl]);
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
    // ---- reduce the warps' accumulators in fixed order ----
    // element (r, j, e) of lane L is red[w][((r * MT + j) * 4 + e) * 32 + L]
#pragma unroll
    for (int r = 0; r < kRpw; ++r)
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                red[warp * RF + ((r * MT + j) * 4 + e) * 32 + lane] = acc[r][j][e];
    __syncthreads();
    float* cta = red + kWarps * RF;
    for (int idx = threadIdx.x; idx < RF; idx += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            v += red[w * RF + idx];
        cta[idx] = v;
    }

    // ---- across the cluster (k splits), in rank order ----
    const bool clustered = p.splits > 1;
    if (clustered) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every member's result is in its shared memory
        if (cluster.block_rank() == 0) {
            for (int idx = threadIdx.x; idx < RF; idx += blockDim.x) {
                float v = cta[idx];
                for (int rk = 1; rk < p.splits; ++rk)
                    v += cluster.map_shared_rank(cta, rk)[idx];
                cta[idx] = v;
            }
        }
        cluster.sync();  // members stay resident until the leader has read them
        if (cluster.block_rank() != 0)
            return;
    } else {
        __syncthreads();
    }

    // ---- epilogue: element idx -> channel n, activation row m ----
    for (int idx = threadIdx.x; idx < RF; idx += blockDim.x) {
        const int L = idx & 31;
        const int e = (idx >> 5) & 3;
        const int rj = idx >> 7;
        const int j = rj % MT, r = rj / MT;
        const int nn = (nb0 + r) * 16 + (L >> 2) + 8 * (e >> 1);
        const int mm = 8 * j + 2 * (L & 3) + (e & 1);
        if (mm >= p.m)
            continue;
        float v = cta[idx];
        if constexpr (!GROUPED)
            v *= to_f32<ACT>(ld_nc_u16(p.scales + nn));
        if (p.bias)
            v += to_f32<ACT>(ld_nc_u16(p.bias + nn));
        p.C[(size_t)mm * p.n + nn] = from_f32<ACT>(v);
    }
}

template <int BITS, int ACT, int MT, bool GROUPED>
cudaError_t launch_one(const GemvPlan& plan, const GemvParams& gp, cudaStream_t s)
{
    auto kern = gemv_kernel<BITS, ACT, MT, GROUPED>;
    const int smem = (kWarps + 1) * red_floats<MT>() * (int)sizeof(float) +
                     gp.a_rows * gp.a_stride + 2 * kCtaCols * gp.g_span * 2;
    static int smem_set[64] = {0};  // largest opt-in granted so far, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || smem > smem_set[dev])) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            smem_set[dev] = smem;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid_x, plan.splits);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (plan.splits > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = plan.splits;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, gp);
}

template <int BITS, int ACT, bool GROUPED>
cudaError_t launch_mt(const GemvPlan& plan, const GemvParams& gp, cudaStream_t s)
{
    switch (plan.mt) {
    case 1: return launch_one<BITS, ACT, 1, GROUPED>(plan, gp, s);
    case 2: return launch_one<BITS, ACT, 2, GROUPED>(plan, gp, s);
    case 4: return launch_one<BITS, ACT, 4, GROUPED>(plan, gp, s);
    default: return launch_one<BITS, ACT, 8, GROUPED>(plan, gp, s);
    }
}

// Shared memory a launch needs (mirrors launch_one).
size_t gemv_smem(int mt, int a_rows, int a_stride, int g_span)
{
    return (size_t)(kWarps + 1) * kRpw * mt * 4 * 32 * 4 + (size_t)a_rows * a_stride +
           (size_t)2 * kCtaCols * g_span * 2;
}

}  // namespace

GemvPlan plan_gemv(int m, int n, int k, int group, int bits)
{
    GemvPlan p{};
    const int KT = bits == 8 ? 32 : 64;
    p.ktiles = k / KT;
    p.grid_x = n / kCtaCols;
    const int tpg = group / KT;
    // enough CTAs for about two per SM; split k across a cluster when the
    // channel count alone does not provide them, keeping >= 2 tiles per warp
    const int target = num_sms() * 2;
    int want = (target + p.grid_x - 1) / p.grid_x;
    int cap = p.ktiles / (2 * kWarps);
    if (cap < 1)
        cap = 1;
    if (cap > kMaxCluster)
        cap = kMaxCluster;
    if (want > cap)
        want = cap;
    if (want < 1)
        want = 1;
    // the staged activation slice must fit: try 8-row tiles per pass from
    // the natural count down, and a larger shared-memory budget last
    const int rows = m < 64 ? m : 64;
    const int mt0 = rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;
    for (int budget : {kAsmemBudget, 160 * 1024}) {
        for (int mt = mt0; mt >= 1; mt /= 2) {
            const int prow = m < 8 * mt ? m : 8 * mt;
            int splits = want;
            for (; splits <= kMaxCluster; ++splits) {
                const int kps = (p.ktiles + splits - 1) / splits;
                const int gspan = bits == 4 ? (kps + tpg - 1) / tpg + 1 : 0;
                const size_t need = gemv_smem(mt, prow, kps * KT * 2 + 16, gspan);
                if (need <= (size_t)budget + (size_t)(kWarps + 1) * kRpw * mt * 4 * 32 * 4)
                    break;
            }
            if (splits <= kMaxCluster) {
                p.mt = mt;
                p.m_per_pass = 8 * mt;
                p.passes = (m + p.m_per_pass - 1) / p.m_per_pass;
                p.ktiles_per_split = (p.ktiles + splits - 1) / splits;
                p.splits = (p.ktiles + p.ktiles_per_split - 1) / p.ktiles_per_split;
                p.a_rows = prow;
                p.a_stride = p.ktiles_per_split * KT * 2 + 16;
                p.g_span = bits == 4 ? (p.ktiles_per_split + tpg - 1) / tpg + 1 : 0;
                p.valid = true;
                p.ws_bytes = 0;
                return p;
            }
        }
    }
    p.valid = false;  // k too long to stage even 8 rows per pass
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
    gp.a_stride = p.a_stride;
    gp.g_span = p.g_span;
    for (int pass = 0; pass < p.passes; ++pass) {
        const int m0 = pass * p.m_per_pass;
        const int rows = a.m - m0 < p.m_per_pass ? a.m - m0 : p.m_per_pass;
        gp.m = rows;
        gp.a_rows = rows;
        gp.A = static_cast<const uint16_t*>(a.A) + (size_t)m0 * a.k;
        gp.C = static_cast<uint16_t*>(a.C) + (size_t)m0 * a.n;
        cudaError_t e;
        if (a.bits == 8) {
            e = a.act == WO_F16 ? launch_mt<8, ACT_F16, false>(p, gp, s)
                                : launch_mt<8, ACT_BF16, false>(p, gp, s);
        } else {
            e = a.act == WO_F16 ? launch_mt<4, ACT_F16, true>(p, gp, s)
                                : launch_mt<4, ACT_BF16, true>(p, gp, s);
        }
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace wo
