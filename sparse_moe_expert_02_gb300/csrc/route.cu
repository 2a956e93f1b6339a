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
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

template <int J>  // J = ceil(E / 32) logits per lane
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int S,
                                                   const float* __restrict__ bias, float* __restrict__ logits_out,
                                                   int T, int E, int k, int32_t* __restrict__ blob, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int64_t TE = (int64_t)T * E;
    const float* zt = part + (int64_t)t * E;
    float v[J];
    bool finite = true;
    // K-split partial products of the router GEMM, added in slice order; the
    // loads of one slice are independent, so each slice costs one round trip
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = (lane + 32 * j < E) ? __ldg(zt + lane + 32 * j) : 0.0f;
    for (int s = 1; s < S; ++s) {
        float w[J];
#pragma unroll
        for (int j = 0; j < J; ++j) w[j] = (lane + 32 * j < E) ? __ldg(zt + s * TE + lane + 32 * j) : 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j) v[j] += w[j];
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            if (bias) v[j] += __ldg(bias + e);
            if (logits_out) logits_out[(int64_t)t * E + e] = v[j];
            if (!isfinite(v[j])) finite = false;
        }
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

cudaError_t launch_topk(const float* part, int S, const float* bias, float* logits_out, int T, int E, int k,
                        int32_t* blob, uint32_t* err, cudaStream_t stream) {
    const int warps = 8;
    dim3 grid((unsigned)cdiv(T, warps)), block(32 * warps);
    const int J = (int)cdiv(E, 32);
#define MOE_TOPK(JJ) topk_kernel<JJ><<<grid, block, 0, stream>>>(part, S, bias, logits_out, T, E, k, blob, err)
    if (J <= 1) MOE_TOPK(1);
    else if (J <= 2) MOE_TOPK(2);
    else if (J <= 4) MOE_TOPK(4);
    else if (J <= 8) MOE_TOPK(8);
    else if (J <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    count_launches(1);
    return cudaGetLastError();
}

// Compact routing word: one int32 per (t, j) holding the expert index in the
// low 16 bits and the bf16 (round to nearest even) of the routing weight in
// the high 16 -- the single dense 32-bit blob of the English page's
// "Fusing Three Collectives Into Two", at half the bytes of the two-plane
// blob (the weight keeps 8 significant bits).
__global__ void pack_words_kernel(const int32_t* __restrict__ blob, int64_t TK, int32_t* __restrict__ words) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < TK; i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t e = (uint32_t)__ldg(blob + i) & 0xFFFFu;
        const uint32_t w = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__int_as_float(__ldg(blob + TK + i))));
        words[i] = (int32_t)(e | (w << 16));
    }
}

cudaError_t launch_pack_words(const int32_t* blob, int64_t TK, int32_t* words, cudaStream_t stream) {
    const int blocks = (int)std::min<int64_t>(cdiv(TK, 256), 4096);
    pack_words_kernel<<<blocks, 256, 0, stream>>>(blob, TK, words);
    count_launches(1);
    return cudaGetLastError();
}

// K slices of the router GEMM: enough (up to 8) that the units of 32
// experts x 128 tokens x K/S cover the SMs when T is small.
int router_splits(int T, int E, int D, int num_sms) {
    const int units = (int)cdiv(T, 128) * std::max(1, E / 32);
    const int kblocks = D / 64;
    int S = 1;
    while (S < 8 && units * S * 2 <= num_sms && kblocks % (2 * S) == 0) S *= 2;
    return S;
}

}  // namespace moe
