// wo_common.cuh -- device helpers shared by the libwo kernels (sm_103a).
//
// Packed weight layout (produced by wo_pack, read by every GEMM kernel):
//   tiles of 16 output channels x KT codes (KT = 32 for 8-bit, 64 for 4-bit),
//   512 bytes each, ordered [n / 16][k / KT].  Lane L = 4*g + t of a warp owns
//   bytes 16L..16L+15 of a tile, which hold exactly the codes of its
//   mma.m16n8k16 A-operand fragments (rows g and g+8, columns 2t, 2t+1,
//   2t+8, 2t+9 of each 16-wide k-step), so one 128-bit load per lane feeds
//   KT/16 k-steps with no shuffles:
//     8-bit, k-step s (bytes 8s..8s+7): word 0 = rows (g, g, g+8, g+8) at
//       k (2t, 2t+1, 2t, 2t+1); word 1 = the same at k + 8.
//     4-bit, k-step s = 32-bit word s; nibble p (bits 4p..4p+3) holds
//       register R = p & 3, half h = p >> 2: row g + 8*(R & 1),
//       k = 16s + 2t + 8*(R >> 1) + h.  Shifting the word right by 4R and
//       masking 0x000F000F leaves the two codes of register R in the two
//       16-bit halves.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace wo {

constexpr int kTileBytes = 512;

template <int BITS>
struct Geom {
    static constexpr int KT = BITS == 8 ? 32 : 64;  // codes of k per tile
    static constexpr int KSTEPS = KT / 16;          // m16n8k16 k-steps per tile
};

enum { ACT_F16 = 0, ACT_BF16 = 1 };

// ---------------------------------------------------------------- loads ----

// Streaming 128-bit load of packed weights: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p)
{
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const void* p)
{
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ------------------------------------------------------- bit operations ----

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// (a & b) ^ c
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// a * b + c on fp16 pairs, one rounding
__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// ------------------------------------------- exact code -> 16-bit floats ----
//
// All conversions below produce the exact integer (q - offset) as a pair of
// fp16 or bf16 values; every intermediate is an exactly representable
// integer, so no rounding happens anywhere.
//
// fp16 with exponent field 25 (bits 0x6400) spans [1024, 2048) with spacing
// 1, so the bits 0x64XX encode 1024 + XX for any byte XX; subtracting
// 1024 + offset leaves q - offset.
// bf16 with exponent field 134 (bits 0x4300) spans [128, 256) with spacing 1,
// so 0x4300 | x encodes 128 + x for x < 128.  An 8-bit code q = 128*h + x
// gives q - 128 = (128 + x) - S with S = 256 - 128*h, i.e. S = 256 (bits
// 0x4380) when h = 0 and S = 128 (bits 0x4300) when h = 1: S's bits are
// 0x4380 ^ (h << 7).

// 8-bit codes: the two bytes of `w` picked by `sel` (a prmt selector whose
// odd nibbles are 4) -> (q - 128) pair.
template <int ACT>
__device__ __forceinline__ uint32_t cvt_u8x2(uint32_t w, uint32_t sel);

template <>
__device__ __forceinline__ uint32_t cvt_u8x2<ACT_F16>(uint32_t w, uint32_t sel)
{
    return sub_f16x2(prmt(w, 0x64646464u, sel), 0x64806480u);  // - 1152
}

template <>
__device__ __forceinline__ uint32_t cvt_u8x2<ACT_BF16>(uint32_t w, uint32_t sel)
{
    const uint32_t x = prmt(w, 0u, sel);                      // 0x00bb00aa
    const uint32_t lo = and_or(x, 0x007F007Fu, 0x43004300u);  // 128 + (q & 127)
    const uint32_t s = and_xor(x, 0x00800080u, 0x43804380u);  // 256 or 128
    return sub_bf16x2(lo, s);
}

// 4-bit codes: the two nibbles at bits (4R, 16 + 4R) of `w_shifted` (already
// shifted right by 4R) -> (q - 8) pair.
template <int ACT>
__device__ __forceinline__ uint32_t cvt_u4x2(uint32_t w_shifted);

template <>
__device__ __forceinline__ uint32_t cvt_u4x2<ACT_F16>(uint32_t ws)
{
    return sub_f16x2(and_or(ws, 0x000F000Fu, 0x64006400u), 0x64086408u);  // - 1032
}

template <>
__device__ __forceinline__ uint32_t cvt_u4x2<ACT_BF16>(uint32_t ws)
{
    return sub_bf16x2(and_or(ws, 0x000F000Fu, 0x43004300u), 0x43084308u);  // - 136
}

// fp16 only: the two nibbles at bits (4, 20) of `w` -> (q - 8) pair, no
// shift.  fp16 with exponent field 21 (bits 0x5400) spans [64, 128) with
// spacing 1/16, so mantissa bits 4..7 carry weight 1 and 0x54X0 encodes
// 64 + X exactly; subtracting 72 leaves q - 8.
__device__ __forceinline__ uint32_t cvt_u4x2_hi_f16(uint32_t w)
{
    return sub_f16x2(and_or(w, 0x00F000F0u, 0x54005400u), 0x54805480u);  // - 72
}

// The four A-operand registers of k-step s of a packed tile.
template <int BITS, int ACT>
__device__ __forceinline__ void tile_frag(const uint4& v, int s, uint32_t (&a)[4])
{
    if constexpr (BITS == 8) {
        const uint32_t w0 = s == 0 ? v.x : v.z;
        const uint32_t w1 = s == 0 ? v.y : v.w;
        a[0] = cvt_u8x2<ACT>(w0, 0x4140u);
        a[1] = cvt_u8x2<ACT>(w0, 0x4342u);
        a[2] = cvt_u8x2<ACT>(w1, 0x4140u);
        a[3] = cvt_u8x2<ACT>(w1, 0x4342u);
    } else {
        const uint32_t w = s == 0 ? v.x : s == 1 ? v.y : s == 2 ? v.z : v.w;
        a[0] = cvt_u4x2<ACT>(w);
        a[2] = cvt_u4x2<ACT>(w >> 8);
        if constexpr (ACT == ACT_F16) {
            a[1] = cvt_u4x2_hi_f16(w);
            a[3] = cvt_u4x2_hi_f16(w >> 8);
        } else {
            a[1] = cvt_u4x2<ACT>(w >> 4);
            a[3] = cvt_u4x2<ACT>(w >> 12);
        }
    }
}

// ----------------------------------------------------------------- mma -----

template <int ACT>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<ACT_F16>(float (&d)[4], const uint32_t (&a)[4],
                                                  uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<ACT_BF16>(float (&d)[4], const uint32_t (&a)[4],
                                                   uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A pair of ones, the A operand that turns an mma into a row sum of B.
template <int ACT>
__device__ __forceinline__ uint32_t ones_x2()
{
    return ACT == ACT_F16 ? 0x3C003C00u : 0x3F803F80u;
}

// ------------------------------------------------------- 16-bit values ----

template <int ACT>
__device__ __forceinline__ float to_f32(uint16_t v)
{
    if constexpr (ACT == ACT_BF16) {
        return __uint_as_float((uint32_t)v << 16);
    } else {
        float f;
        asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(v));
        return f;
    }
}

template <int ACT>
__device__ __forceinline__ uint16_t from_f32(float f)
{
    uint16_t r;
    if constexpr (ACT == ACT_BF16) {
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    } else {
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(f));
    }
    return r;
}

}  // namespace wo
