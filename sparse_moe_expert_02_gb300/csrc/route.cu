// Top-k routing over fp32 router logits, and the packed routing blob.
//
// "Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU" (aihot.vn
// translation, section 1.3 "Sparse Mixture-of-Experts"): the router gate
// picks the top 10 experts through a softmax distribution; English page,
// "Fusing Three Collectives Into Two": indices and weights, both [T, k],
// travel as one 32-bit integer blob.
//
// One warp per token.  Each lane keeps E/32 logits in registers; k rounds of
// a warp-wide argmax pick the experts.  Order: larger logit first, the lower
// expert index on equal logits -- the same total order in every lane and in
// the cross-lane reduction, so the choice is deterministic.  Weights are the
// softmax over the chosen logits (equal to the renormalised full softmax).
#include "common.cuh"
#include "internal.h"

namespace moe {

template <int J>  // J = ceil(E / 32) logits per lane
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                   int32_t* __restrict__ blob, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* zt = logits + (int64_t)t * E;
    float v[J];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        int e = lane + 32 * j;
        v[j] = (e < E) ? __ldg(zt + e) : 0.0f;
        if (e < E && !isfinite(v[j])) finite = false;
    }
    if (!__all_sync(0xffffffffu, finite)) {
        if (lane == 0) record_error(err, MOE_ERR_NONFINITE, (uint32_t)t, 0, 0);
        // Out of contract.  Non-finite logits become -inf so the order stays
        // total and the k chosen indices stay distinct and in range.
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (!isfinite(v[j])) v[j] = -INFINITY;
    }
    uint32_t taken = 0;  // bit j: this lane's slot j is chosen
    float zsel = 0.0f;   // lane r < k keeps the r-th chosen logit
    int isel = 0;
    for (int r = 0; r < k; ++r) {
        float bv = 0.0f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            int e = lane + 32 * j;
            bool ok = (e < E) && !((taken >> j) & 1u);
            // lanes scan j upwards, so e grows: strict '>' keeps the lowest e on ties
            if (ok && (bi == 0x7fffffff || v[j] > bv)) { bv = v[j]; bi = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            bool take = (oi != 0x7fffffff) &&
                        (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
            if (take) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == r) { zsel = bv; isel = bi; }
    }
    const float zmax = __shfl_sync(0xffffffffu, zsel, 0);
    float ex = (lane < k) ? expf(zsel - zmax) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        const int64_t TK = (int64_t)T * k;
        blob[(int64_t)t * k + lane] = isel;
        blob[TK + (int64_t)t * k + lane] = __float_as_int(ex / sum);
    }
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* blob, uint32_t* err,
                        cudaStream_t stream) {
    const int warps = 8;
    dim3 grid((unsigned)cdiv(T, warps)), block(32 * warps);
    int J = (int)cdiv(E, 32);
    if (J <= 1) topk_kernel<1><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    else if (J <= 2) topk_kernel<2><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    else if (J <= 4) topk_kernel<4><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    else if (J <= 8) topk_kernel<8><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    else if (J <= 16) topk_kernel<16><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    else topk_kernel<32><<<grid, block, 0, stream>>>(logits, T, E, k, blob, err);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
