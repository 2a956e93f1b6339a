// Device-side helpers shared by the libmoe kernels: element conversions,
// the workspace error word, and a nanosecond clock for bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;
typedef __half f16;

// ---------------------------------------------------------------- errors

// The error word: [0] first error code (moe_status), [1..3] diagnostics.
// The first writer wins; later errors are dropped.
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code, uint32_t a = 0, uint32_t b = 0,
                                             uint32_t c = 0) {
    if (err == nullptr) return;
    if (atomicCAS(err, 0u, code) == 0u) {
        err[1] = a;
        err[2] = b;
        err[3] = c;
        __threadfence();
    }
}

// Programmatic dependent launch: a kernel launched as a dependent of the
// previous kernel on its stream may start while that kernel finishes; it
// waits here before touching anything the earlier kernels write, then lets
// its own dependents start their prologue.  Without a programmatic
// dependency both are no-ops.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------- conversions

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(f16 v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ f16 from_f32<f16>(float v) { return __float2half_rn(v); }

// E4M3, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
// Two values to two E4M3 codes (round to nearest even, saturating): a in
// the low byte, b in the high byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t q) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)q, __NV_E4M3);
    return __half2float(__half(hr));
}

// SiLU(a) * u in fp32: a * u / (1 + e^-a), with the hardware exponential
// and the fast (reciprocal-based) division: a few ulp of fp32, far below the
// fp16 / E4M3 rounding of h that follows.  For a < -88, e^-a is infinite
// and the quotient is 0, SiLU's limit.
__device__ __forceinline__ float swiglu(float a, float u) { return __fdividef(a * u, 1.0f + __expf(-a)); }

__host__ __device__ constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Unpermutation of one 32-column chunk of token t inside a GEMM epilogue:
// a[i] holds the shared expert's output for columns n0.. (already rounded to
// y's 16-bit type); it takes w[t,j] * y[inv[t*k+j]] for j = 0..k-1 in order,
// in fp32 -- the unpermute kernel's order and rounding.  y is [TK, ldy];
// blob plane 1 (at TK) holds the fp32 weights.  Two slots' loads are in
// flight at a time.  A dropped pair (row out of range) records
// MOE_ERR_BOUNDS and contributes nothing.
template <typename TY>
__device__ __forceinline__ void combine_chunk32(const TY* __restrict__ y, int64_t ldy, const int32_t* __restrict__ inv,
                                                const int32_t* __restrict__ blob, int k, int64_t t, int64_t TK, int n0,
                                                float* a, uint32_t* err) {
    for (int j0 = 0; j0 < k; j0 += 2) {
        uint4 q[2][4];
        float w[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int j = j0 + s;
            int r = 0;
            w[s] = 0.0f;
            if (j < k) {
                r = __ldg(inv + t * k + j);
                w[s] = __int_as_float(__ldg(blob + TK + t * k + j));
                if ((unsigned)r >= (unsigned)TK) {
                    record_error(err, MOE_ERR_BOUNDS, (uint32_t)t, (uint32_t)j, 2);
                    r = 0;
                    w[s] = 0.0f;
                }
            }
            const uint4* src = (const uint4*)(y + (int64_t)r * ldy + n0);
#pragma unroll
            for (int v = 0; v < 4; ++v) q[s][v] = j < k ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (j0 + s >= k) break;
            const TY* e = (const TY*)q[s];
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = fmaf(w[s], to_f32(e[i]), a[i]);
        }
    }
}

// Group of a row tile: tiles[g] <= tile < tiles[g+1] (tiles has G+1 entries,
// nondecreasing).  Binary search, G <= 1025.
// The same over a copy of the prefix in shared memory.
__device__ __forceinline__ int find_group_smem(const int32_t* tiles, int G, int tile) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (tiles[mid] <= tile) lo = mid;
        else hi = mid;
    }
    return lo;
}
__device__ __forceinline__ int find_group(const int32_t* tiles, int G, int tile) {
    int lo = 0, hi = G;  // invariant: tiles[lo] <= tile < tiles[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(tiles + mid) <= tile) lo = mid;
        else hi = mid;
    }
    return lo;
}

}  // namespace moe
