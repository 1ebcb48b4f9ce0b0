// moe_common.cuh -- small device helpers shared by the SIMT kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {

// Builds with MOE_DEBUG_BOUNDS check every expert and row index the routing
// and combine kernels use against its range, record
// MOE_DEVICE_INDEX_OUT_OF_RANGE in the status word and skip the access
// instead of performing it.
#ifdef MOE_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Builds with MOE_TIMELINE record, for CTA 0 of every routed CTA-pair GEMM
// launch, globaltimer stamps of each unit's MMA and epilogue phases
// (moe_timeline_read); other builds record nothing.
#ifdef MOE_TIMELINE
constexpr bool kTimeline = true;
#else
constexpr bool kTimeline = false;
#endif

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename TE>
__device__ __forceinline__ TE from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

// SiLU with the fast exponential and reciprocal (the result is rounded to
// bf16 or checked at 1e-4 relative, far above their error).
__device__ __forceinline__ float silu_f32(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their memory is visible (no-op when launched normally).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid in the stream to be scheduled (it still waits in
// griddep_wait for this grid to complete).
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Sum over the warp; every lane receives lane 0's result, so all lanes hold
// bit-identical values whatever order the butterfly used.
__device__ __forceinline__ float warp_sum_bcast(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return __shfl_sync(0xffffffffu, v, 0);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The balance loss of AuxArgs, by one warp: lane l sums the terms of
// experts l, l+32, ... in order, then a fixed butterfly; lane 0 writes it.
__device__ __forceinline__ void balance_loss_warp(const AuxArgs &a)
{
    const int lane = threadIdx.x & 31;
    double sum = 0.0;
    for (int e = lane; e < a.E; e += 32)
        sum += ((double)__ldcg(a.counts + e) / ((double)a.T * (double)a.k)) *
               (__ldcg(a.psum + e) / (double)a.T);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0)
        *a.out = (float)((double)a.alpha * (double)a.E * sum);
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t code)
{
    if (status)
        atomicCAS(status, 0, code);
}

}  // namespace moe
