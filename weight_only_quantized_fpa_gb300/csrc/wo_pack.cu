// wo_pack.cu -- offline repack of row-major weight codes into the tile layout
// of wo_common.cuh, and its inverse.  This is the load-time weight
// preprocessing step of "acext User Guide (v1.7)" 1.3.1-1.3.3
// (preprocess_weights_for_mixed_gemm), with a layout of our own: each lane's
// 16 bytes hold its mma fragments, so the GEMM kernels need no shuffles.
//
// Row-major input (vLLM-Omni "cpu_int4.py" module docstring):
//   8-bit: uint8 [n, k];  4-bit: uint8 [n, k/2], byte j = code 2j | code 2j+1 << 4.
//
// One thread builds (or scatters) one lane chunk of 16 bytes.  Every output
// byte is written by exactly one thread, in both directions: in the 4-bit
// inverse the two nibbles of a row-major byte (k even and k + 1) come from
// the same lane word (registers R and R + 4 of the layout), so no two threads
// share a destination byte.
#include "wo_bounds.cuh"
#include "wo_common.cuh"
#include "wo_internal.h"

namespace wo {
namespace {

// Row and k (within the tile) of byte b of lane (g, t), 8-bit layout.
__device__ __forceinline__ void u8_coord(int b, int g, int t, int& row, int& kk)
{
    const int s = b >> 3;        // k-step
    const int w = (b >> 2) & 1;  // word within the k-step
    const int j = b & 3;         // byte within the word
    row = g + 8 * (j >> 1);
    kk = 16 * s + 2 * t + 8 * w + (j & 1);
}

// Row and k (within the tile) of nibble p of word s, lane (g, t), 4-bit layout.
__device__ __forceinline__ void u4_coord(int s, int p, int g, int t, int& row, int& kk)
{
    const int R = p & 3, h = p >> 2;
    row = g + 8 * (R & 1);
    kk = 16 * s + 2 * t + 8 * (R >> 1) + h;
}

// perm (optional, [k]): packed column j takes row-major column perm[j] (a GPTQ
// act-order checkpoint's channels, sorted by group).  An entry outside
// [0, k) reads code 0, so a bad permutation cannot read out of bounds.
template <int BITS>
__global__ void pack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int n,
                            int k, long long chunks, const int32_t* __restrict__ perm)
{
    constexpr int KT = Geom<BITS>::KT;
    const int ktiles = k / KT;
    for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < chunks;
         c += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(c & 31);
        const long long tile = c >> 5;
        const int nb = (int)(tile / ktiles);
        const int kt = (int)(tile % ktiles);
        const int g = lane >> 2, t = lane & 3;
        uint32_t words[4];
        if constexpr (BITS == 8) {
            for (int wi = 0; wi < 4; ++wi) {
                uint32_t w = 0;
                for (int j = 0; j < 4; ++j) {
                    int row, kk;
                    u8_coord(4 * wi + j, g, t, row, kk);
                    int kg = kt * KT + kk;
                    if (perm)
                        kg = perm[kg];
                    const uint32_t v = (unsigned)kg < (unsigned)k && in_bounds(nb * 16 + row < n, 0x501)
                                           ? src[(size_t)(nb * 16 + row) * k + kg]
                                           : 0u;
                    w |= v << (8 * j);
                }
                words[wi] = w;
            }
        } else {
            const int kb = k / 2;
            for (int s = 0; s < 4; ++s) {
                uint32_t w = 0;
                for (int p = 0; p < 8; ++p) {
                    int row, kk;
                    u4_coord(s, p, g, t, row, kk);
                    int kg = kt * KT + kk;
                    if (perm)
                        kg = perm[kg];
                    const uint8_t byte = (unsigned)kg < (unsigned)k && in_bounds(nb * 16 + row < n, 0x501)
                                             ? src[(size_t)(nb * 16 + row) * kb + kg / 2]
                                             : 0;
                    const uint32_t q = (kg & 1) ? (byte >> 4) : (byte & 0x0F);
                    w |= q << (4 * p);
                }
                words[s] = w;
            }
        }
        uint4 out = make_uint4(words[0], words[1], words[2], words[3]);
        *reinterpret_cast<uint4*>(dst + c * 16) = out;
    }
}

template <int BITS>
__global__ void unpack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int n,
                              int k, long long chunks)
{
    constexpr int KT = Geom<BITS>::KT;
    const int ktiles = k / KT;
    for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < chunks;
         c += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(c & 31);
        const long long tile = c >> 5;
        const int nb = (int)(tile / ktiles);
        const int kt = (int)(tile % ktiles);
        const int g = lane >> 2, t = lane & 3;
        const uint4 in = *reinterpret_cast<const uint4*>(src + c * 16);
        const uint32_t words[4] = {in.x, in.y, in.z, in.w};
        if constexpr (BITS == 8) {
            for (int b = 0; b < 16; ++b) {
                int row, kk;
                u8_coord(b, g, t, row, kk);
                if (in_bounds(nb * 16 + row < n && kt * KT + kk < k, 0x502))
                    dst[(size_t)(nb * 16 + row) * k + kt * KT + kk] = (uint8_t)(words[b >> 2] >> (8 * (b & 3)));
            }
        } else {
            const int kb = k / 2;
            for (int s = 0; s < 4; ++s) {
                for (int p = 0; p < 4; ++p) {  // p and p + 4: the even and odd k of one byte
                    int row, kk;
                    u4_coord(s, p, g, t, row, kk);
                    const uint32_t lo = (words[s] >> (4 * p)) & 0xF;
                    const uint32_t hi = (words[s] >> (4 * (p + 4))) & 0xF;
                    if (in_bounds(nb * 16 + row < n && kt * KT + kk < k, 0x502))
                        dst[(size_t)(nb * 16 + row) * kb + (kt * KT + kk) / 2] = (uint8_t)(lo | (hi << 4));
                }
            }
        }
    }
}

// Embedding rows straight from the packed table (vLLM-Omni "cpu_int4.py",
// CPUInt4EmbeddingMethod.embedding: gather the rows of the token ids,
// dequantise w = (q - offset) * scale (+ zero) in fp32, round once to the
// activation dtype).  Row r of a 16-row block lives in lanes 4 (r % 8) + t,
// t = 0..3, of each of its block's tiles, and within a lane's words its
// codes are every other nibble (4-bit: the nibbles of registers R with
// R & 1 == r / 8) or every other byte pair (8-bit: bytes 2 (r / 8) and
// 2 (r / 8) + 1 of each word).  A warp takes one token and kEmbedTiles
// consecutive k tiles: lane L reads the 16-byte chunk t = L % 4 of tiles
// L / 4 + 8 j, shifts its row's codes into place, dequantises them and
// writes them as value pairs into a shared-memory copy of the row segment
// (tiles padded by 16 bytes, so the 32 lanes' pair stores hit 32 banks);
// the warp then stores the segment with 16-byte stores.  Ids outside
// [0, vocab) give a zero row (scale and zero 0; the codes are not read).
constexpr int kEmbedPerLane = 2;
constexpr int kEmbedTiles = 8 * kEmbedPerLane;
constexpr int kEmbedWarps = 8;

// (q - off) * s + z with one rounding, q = byte `sel` of x: the byte is
// placed in the low mantissa bits of 2^23, so the float is 2^23 + q exactly
// and the subtraction leaves q - off exactly; (q - off) * s is exact in fp32
// (at most 8 + 11 significant bits), so the fused multiply-add rounds the
// same sum as the product-then-add of the definition.
__device__ __forceinline__ float embed_dq(uint32_t x, uint32_t sel, float magic, float s, float z)
{
    const float q = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | sel)) - magic;
    return fmaf(q, s, z);
}

// Two values rounded to the activation dtype, `lo` in the low half.
template <int ACT>
__device__ __forceinline__ uint32_t embed_pack2(float lo, float hi)
{
    uint32_t r;
    if constexpr (ACT == ACT_BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int BITS, int ACT>
__global__ void __launch_bounds__(kEmbedWarps * 32, 6)
    embed_kernel(const int32_t* __restrict__ ids, int T, const uint8_t* __restrict__ B,
                 const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros,
                 uint16_t* __restrict__ out, int vocab, int hidden, int G, int group)
{
    constexpr int KT = Geom<BITS>::KT;
    constexpr int TS = KT + 8;                    // a tile's values in shared memory, padded
    constexpr float kMagic = 8388608.f + (BITS == 8 ? 128.f : 8.f);
    __shared__ __align__(16) uint16_t seg_sm[kEmbedWarps][kEmbedTiles * TS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint16_t* seg = seg_sm[warp];
    const int ktiles = hidden / KT;
    const int segs = (ktiles + kEmbedTiles - 1) / kEmbedTiles;  // segments per row
    const long long total = (long long)T * segs;
    const int t4 = lane & 3;
    for (long long w = (long long)blockIdx.x * kEmbedWarps + warp; w < total;
         w += (long long)gridDim.x * kEmbedWarps) {
        const int tok = (int)(w / segs), sg = (int)(w % segs);
        const int id = ids[tok];
        const bool valid = id >= 0 && id < vocab;
        const int r = valid ? id % 16 : 0;
        const int g = r & 7;
        const uint32_t hi_row = (uint32_t)(r >> 3);  // the row is the upper one of its lane pair
        uint4 vj[kEmbedPerLane];
        float scj[kEmbedPerLane], zcj[kEmbedPerLane];
#pragma unroll
        for (int j = 0; j < kEmbedPerLane; ++j) {
            const int kt = sg * kEmbedTiles + (lane >> 2) + 8 * j;
            vj[j] = make_uint4(0u, 0u, 0u, 0u);
            scj[j] = zcj[j] = 0.f;
            if (valid && kt < ktiles && in_bounds((size_t)id * G + (size_t)(kt * KT) / group < (size_t)vocab * G, 0x503)) {
                vj[j] = *reinterpret_cast<const uint4*>(
                    B + ((((size_t)(id / 16) * ktiles + kt) * 32 + 4 * g + t4) * 16));
                // one scale (and zero) per k tile: groups are whole tiles or more
                const size_t gi = (size_t)id * G + (size_t)(kt * KT) / group;
                scj[j] = to_f32<ACT>(scales[gi]);
                zcj[j] = zeros ? to_f32<ACT>(zeros[gi]) : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < kEmbedPerLane; ++j) {
            const int tl = (lane >> 2) + 8 * j;
            if (sg * kEmbedTiles + tl < ktiles) {
                const uint32_t words[4] = {vj[j].x, vj[j].y, vj[j].z, vj[j].w};
                const float sc = scj[j], zc = zcj[j];
                uint32_t* dst = reinterpret_cast<uint32_t*>(seg + tl * TS);
                if constexpr (BITS == 8) {
                    // word 2s + w: bytes 2h, 2h + 1 are k = 16 s + 2 t + 8 w and k + 1
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint32_t x = words[wi] >> (16 * hi_row);
                        const int k0 = 16 * (wi >> 1) + 2 * t4 + 8 * (wi & 1);
                        dst[k0 / 2] = embed_pack2<ACT>(embed_dq(x, 0, kMagic, sc, zc),
                                                       embed_dq(x, 1, kMagic, sc, zc));
                    }
                } else {
                    // word s, shifted to the row's registers: nibble 0 is k = 16 s + 2 t,
                    // nibble 4 is k + 1, nibble 2 is k + 8, nibble 6 is k + 9
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t x = (words[s] >> (4 * hi_row)) & 0x0F0F0F0Fu;
                        const int k0 = 16 * s + 2 * t4;
                        dst[k0 / 2] = embed_pack2<ACT>(embed_dq(x, 0, kMagic, sc, zc),
                                                       embed_dq(x, 2, kMagic, sc, zc));
                        dst[k0 / 2 + 4] = embed_pack2<ACT>(embed_dq(x, 1, kMagic, sc, zc),
                                                           embed_dq(x, 3, kMagic, sc, zc));
                    }
                }
            }
        }
        __syncwarp();
        // the segment's valid part: 16-byte stores, consecutive lanes
        constexpr int CPT = KT / 8;  // 16-byte chunks per tile
        const int ntiles = ktiles - sg * kEmbedTiles < kEmbedTiles ? ktiles - sg * kEmbedTiles : kEmbedTiles;
        uint4* dstg = reinterpret_cast<uint4*>(out + (size_t)tok * hidden + (size_t)sg * kEmbedTiles * KT);
        for (int i = lane; i < ntiles * CPT; i += 32)
            if (in_bounds(tok < T && (size_t)sg * kEmbedTiles * KT + (size_t)(i + 1) * 8 <= (size_t)hidden, 0x504))
                dstg[i] = *reinterpret_cast<const uint4*>(seg + (i / CPT) * TS + (i % CPT) * 8);
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_embed(const int32_t* ids, int T, const uint8_t* B, const void* scales,
                         const void* zeros, void* out, int vocab, int hidden, int group, int bits,
                         int act, cudaStream_t s)
{
    const int KT = bits == 8 ? 32 : 64;
    const long long segs = (hidden / KT + kEmbedTiles - 1) / kEmbedTiles;
    const long long total = (long long)T * segs;  // warps of work
    const int threads = kEmbedWarps * 32;
    long long blocks = (total + kEmbedWarps - 1) / kEmbedWarps;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const int G = hidden / group;
    const auto* sc = static_cast<const uint16_t*>(scales);
    const auto* zc = static_cast<const uint16_t*>(zeros);
    auto* o = static_cast<uint16_t*>(out);
    const unsigned nb = (unsigned)blocks;
    if (bits == 8) {
        if (act == WO_F16)
            embed_kernel<8, ACT_F16><<<nb, threads, 0, s>>>(ids, T, B, sc, zc, o, vocab, hidden, G, group);
        else
            embed_kernel<8, ACT_BF16><<<nb, threads, 0, s>>>(ids, T, B, sc, zc, o, vocab, hidden, G, group);
    } else {
        if (act == WO_F16)
            embed_kernel<4, ACT_F16><<<nb, threads, 0, s>>>(ids, T, B, sc, zc, o, vocab, hidden, G, group);
        else
            embed_kernel<4, ACT_BF16><<<nb, threads, 0, s>>>(ids, T, B, sc, zc, o, vocab, hidden, G, group);
    }
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* src, uint8_t* dst, int n, int k, int bits, bool unpack,
                        const int32_t* perm, cudaStream_t s)
{
    const long long bytes = bits == 8 ? (long long)n * k : (long long)n * k / 2;
    const long long chunks = bytes / 16;
    const int threads = 256;
    long long blocks = (chunks + threads - 1) / threads;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    if (bits == 8) {
        if (unpack)
            unpack_kernel<8><<<(unsigned)blocks, threads, 0, s>>>(src, dst, n, k, chunks);
        else
            pack_kernel<8><<<(unsigned)blocks, threads, 0, s>>>(src, dst, n, k, chunks, perm);
    } else {
        if (unpack)
            unpack_kernel<4><<<(unsigned)blocks, threads, 0, s>>>(src, dst, n, k, chunks);
        else
            pack_kernel<4><<<(unsigned)blocks, threads, 0, s>>>(src, dst, n, k, chunks, perm);
    }
    return cudaGetLastError();
}

unsigned bounds_take_pack() { return bounds_take_local(); }

}  // namespace wo
