// wo_bounds.cuh -- index checks of the debug build.
//
// Built with -DWO_DEBUG_BOUNDS=1, every global access whose index a kernel
// computes (loads and stores that do not go through a TMA tensor map, whose
// box is clipped by the hardware) is checked against the extent of its
// buffer.  A failed check skips the access and records the check's site in
// this translation unit's bounds word (the first failure wins); nothing
// traps.  wo_debug_bounds (include/wo.h) reads and clears the words of all
// translation units.  Built without the flag, the checks compile to nothing
// and bounds_take_* return 0.
//
// Sites: 0x100 + i streaming kernel, 0x200 + i persistent 4-bit kernel,
// 0x300 + i tensor-core kernel and its prepass, 0x400 + i swap-AB kernel,
// 0x500 + i pack / unpack / embedding gather, 0x600 + i act-order gather,
// 0x700 + i MoE routing, gather and combine.
#pragma once

#include <cuda_runtime.h>

#ifndef WO_DEBUG_BOUNDS
#define WO_DEBUG_BOUNDS 0
#endif

namespace wo {
namespace {

#if WO_DEBUG_BOUNDS
__device__ unsigned g_bounds_word;  // one per translation unit
#endif

// True when the access may go ahead.  `ok` is the check (index < extent);
// in a normal build it is not even evaluated for its result.
__device__ __forceinline__ bool in_bounds(bool ok, unsigned site)
{
#if WO_DEBUG_BOUNDS
    if (!ok)
        atomicCAS(&g_bounds_word, 0u, site);
    return ok;
#else
    (void)ok;
    (void)site;
    return true;
#endif
}

// Host side: this translation unit's bounds word, cleared (0: no failure or
// a normal build).  Waits for the device first.
inline unsigned bounds_take_local()
{
#if WO_DEBUG_BOUNDS
    unsigned v = 0, z = 0;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return 0;
    if (cudaMemcpyFromSymbol(&v, g_bounds_word, sizeof(v)) != cudaSuccess)
        return 0;
    if (v)
        cudaMemcpyToSymbol(g_bounds_word, &z, sizeof(z));
    return v;
#else
    return 0;
#endif
}

}  // namespace
}  // namespace wo
