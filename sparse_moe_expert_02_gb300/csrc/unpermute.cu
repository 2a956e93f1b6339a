// Unpermutation with the local reduction and the shared-expert add:
//   out[t] = y[T*k + t] + sum_j w[t,j] * y[inv[t*k + j]]
// ("Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU", English
// page, table in "Pallas Kernels, SparseCore Co-Design, and the Roofline":
// token unpermutation plus local reduction offloaded to SparseCore; the
// shared expert is the always-on path of the MoE bullet in "The
// Architectural Constraints That Break Naive Sharding").
//
// A gather-reduce: one block per token, each thread owns 16-byte vectors of
// the row, reads the k+1 source rows and accumulates in fp32 in slot order.
// The routing weights come from plane 1 of the blob.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// grid = (T, ceil(D / (blockDim*V))): one 16-byte vector of one token per
// thread.  The k+1 source rows are read in groups of 8 independent loads, so
// a token costs two round trips to memory instead of k+1.
template <typename TY, typename TO>
__global__ void __launch_bounds__(256) unpermute_kernel(const TY* __restrict__ y, const int32_t* __restrict__ blob,
                                                        const int32_t* __restrict__ inv, int T, int D, int k,
                                                        TO* __restrict__ out, uint32_t* err) {
    constexpr int V = 16 / sizeof(TY);  // elements per 16-byte vector of y
    pdl_wait_then_release();
    __shared__ int64_t rows[33];
    __shared__ float wts[33];
    const int t = blockIdx.x;
    const int64_t TK = (int64_t)T * k;
    if (threadIdx.x < k) {
        int r = __ldg(inv + (int64_t)t * k + threadIdx.x);
        float wj = __int_as_float(__ldg(blob + TK + (int64_t)t * k + threadIdx.x));
        if ((unsigned)r >= (unsigned)TK) {  // a pair the permutation dropped (bad expert id)
            record_error(err, MOE_ERR_BOUNDS, (uint32_t)t, (uint32_t)threadIdx.x, 2);
            r = 0;
            wj = 0.0f;
        }
        rows[1 + threadIdx.x] = (int64_t)r * D;
        wts[1 + threadIdx.x] = wj;
    }
    if (threadIdx.x == 0) {  // slot 0: the shared expert's row, weight 1
        rows[0] = (TK + t) * D;
        wts[0] = 1.0f;
    }
    __syncthreads();
    const int c = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c >= D) return;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    // slot order: shared expert first, then j = 0 .. k-1 (fp32 accumulation)
    for (int j0 = 0; j0 <= k; j0 += 8) {
        int4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (j0 + q <= k) v[q] = __ldg((const int4*)(y + rows[j0 + q] + c));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (j0 + q > k) break;
            const TY* e = (const TY*)&v[q];
            const float wj = wts[j0 + q];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(wj, to_f32(e[i]), acc[i]);
        }
    }
    // This thread owns out[t, c .. c+V-1]: V*sizeof(TO) bytes at a
    // multiple of that size (16 B for fp32 out, 8 or 16 B for bf16 out).
    TO* o = out + (int64_t)t * D + c;
    if constexpr (sizeof(TO) == 4) {
#pragma unroll
        for (int i = 0; i < V; i += 4) *(float4*)(o + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    } else if constexpr (V == 4) {
        uint2 p;
        __nv_bfloat162* pb = (__nv_bfloat162*)&p;
        pb[0] = __floats2bfloat162_rn(acc[0], acc[1]);
        pb[1] = __floats2bfloat162_rn(acc[2], acc[3]);
        *(uint2*)o = p;
    } else {
        static_assert(V == 8, "16-bit y carries 8 values per 16-byte vector");
        uint4 p;
        __nv_bfloat162* pb = (__nv_bfloat162*)&p;
#pragma unroll
        for (int q = 0; q < 4; ++q) pb[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        *(uint4*)o = p;
    }
}

cudaError_t launch_unpermute(const void* y, int y_elem, const int32_t* blob, const int32_t* inv, int T, int D, int k,
                             void* out, int out_elem, uint32_t* err, cudaStream_t stream) {
    if (T <= 0) return cudaGetLastError();
    const int V = (y_elem == kF32) ? 4 : 8;
    const int vecs = D / V;
    const int threads = std::min(256, ((vecs + 31) / 32) * 32);
    dim3 grid((unsigned)T, (unsigned)cdiv(vecs, threads));
    cudaError_t e = cudaSuccess;
#define MOE_UNPERMUTE(TY, TO)                                                                                \
    e = launch_kernel(unpermute_kernel<TY, TO>, grid, dim3(threads), 0, stream, 1, (const TY*)y, blob, inv, T, D, k, \
                      (TO*)out, err)
    const bool o32 = out_elem == kF32;
    if (y_elem == kF32) {
        if (o32) MOE_UNPERMUTE(float, float); else MOE_UNPERMUTE(float, bf16);
    } else if (y_elem == kF16) {
        if (o32) MOE_UNPERMUTE(f16, float); else MOE_UNPERMUTE(f16, bf16);
    } else {
        if (o32) MOE_UNPERMUTE(bf16, float); else MOE_UNPERMUTE(bf16, bf16);
    }
#undef MOE_UNPERMUTE
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Bounded-wait self-test: one thread waits on an mbarrier that expects an
// arrival nobody makes, polling %globaltimer, and gives up after limit_ns.
__global__ void selftest_timeout_kernel(uint32_t* err, int64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(1));
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t done = 0;
        while (!done) {
            asm volatile(
                "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                : "=r"(done)
                : "r"(a), "r"(0));
            if (!done && (int64_t)(globaltimer_ns() - t0) > limit_ns) {
                record_error(err, MOE_ERR_DEVICE_TIMEOUT, 0xFFFFu, 0, 0);
                break;
            }
        }
    }
}

cudaError_t launch_selftest_timeout(uint32_t* err, int64_t limit_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
