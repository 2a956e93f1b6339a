// Top-k routing over fp32 router logits, and the packed routing blob.
//
// "Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU" (aihot.vn
// translation, section 1.3 "Sparse Mixture-of-Experts"): the router gate
// picks the top 10 experts through a softmax distribution; English page,
// "Fusing Three Collectives Into Two": indices and weights, both [T, k],
// travel as one 32-bit integer blob.
//
// One warp per token.  Each lane keeps E/32 logits in registers and its four
// best in order; k rounds of a warp-wide argmax over the lanes' heads pick
// the experts.  Order: larger logit first, the lower
// expert index on equal logits -- the same total order in every lane and in
// the cross-lane reduction, so the choice is deterministic.  Weights are the
// softmax over the chosen logits (equal to the renormalised full softmax).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Order-preserving map of an fp32 to uint32 (larger float -> larger key);
// -0 is folded onto +0 first so that the two compare equal, as floats do.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u >> 31) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k >> 31) ? (k & 0x7FFFFFFFu) : ~k);
}

// J = ceil(E / 32) logits per lane (a power of two); SB = K slices loaded per
// batch (1 when the router GEMM did not split K: fewer registers, more warps)
// hist (nullable): the permutation's per-chunk expert histograms
// ([chunks][E], zeroed by the caller; chunk = pairs per chunk), counted here
// as the experts are chosen, so that the permutation needs no pass of its
// own over the indices.
template <int J, int SB>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int S,
                                                   const float* __restrict__ bias, float* __restrict__ logits_out,
                                                   int T, int E, int k, int32_t* __restrict__ blob,
                                                   int32_t* __restrict__ hist, int chunk, uint32_t* err) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warps leave together
    const int64_t TE = (int64_t)T * E;
    const float* zt = part + (int64_t)t * E;
    // K-split partial products of the router GEMM (S slices): the loads of a
    // batch of SB slices are all issued before the first add, and the slices
    // are added in order
    float v[J];
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = 0.0f;
    for (int s0 = 0; s0 < S; s0 += SB) {
        float w[SB][J];
#pragma unroll
        for (int s = 0; s < SB; ++s)
#pragma unroll
            for (int j = 0; j < J; ++j)
                w[s][j] = (s0 + s < S && lane + 32 * j < E) ? __ldg(zt + (s0 + s) * TE + lane + 32 * j) : 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int s = 0; s < SB; ++s)
                if (s0 + s < S) v[j] = (s0 + s == 0) ? w[s][j] : v[j] + w[s][j];
    }
    bool finite = true;
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
    // Each lane keeps its H best (key, expert) pairs in order -- larger logit
    // first, the lower expert index among equals -- built by insertion over
    // its J logits.  Key 0 marks an empty slot: every real logit (even -inf)
    // has a larger key.
    uint32_t key[J];
    int id[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? order_key(v[j]) : 0u;
        id[j] = e;
    }
    constexpr int H = J < 4 ? J : 4;
    uint32_t hk[H];
    int hi[H];
    // the H best of this lane's pairs that come strictly after (ak, ai) in the
    // order (all of them when `all`)
    auto build = [&](bool all, uint32_t ak, int ai) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
            hk[h] = 0u;
            hi[h] = 0x7FFFFFFF;
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const uint32_t kj = key[j];
            const int ij = id[j];
            const bool after = all || kj < ak || (kj == ak && ij > ai);
            if (after && (kj > hk[H - 1] || (kj == hk[H - 1] && ij < hi[H - 1]))) {
                hk[H - 1] = kj;
                hi[H - 1] = ij;
#pragma unroll
                for (int h = H - 1; h > 0; --h) {
                    if (hk[h] > hk[h - 1] || (hk[h] == hk[h - 1] && hi[h] < hi[h - 1])) {
                        const uint32_t tk = hk[h]; hk[h] = hk[h - 1]; hk[h - 1] = tk;
                        const int ti = hi[h]; hi[h] = hi[h - 1]; hi[h - 1] = ti;
                    }
                }
            }
        }
    };
    build(true, 0u, 0);
    // k rounds: the largest head over the warp, the lowest index among the
    // lanes holding it; that lane drops its head (and, having used all H,
    // rebuilds its list from the pairs after the one it gave up).
    float zsel = 0.0f;
    int isel = 0;
    int used = 0;
    for (int r = 0; r < k; ++r) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, hk[0]);
        const uint32_t win = __reduce_min_sync(0xffffffffu, hk[0] == m ? (uint32_t)hi[0] : 0xFFFFFFFFu);
        if (lane == r) {
            zsel = key_value(m);
            isel = (int)win;
        }
        if (hk[0] == m && (uint32_t)hi[0] == win) {
            const uint32_t lk = hk[0];
            const int li = hi[0];
#pragma unroll
            for (int h = 0; h + 1 < H; ++h) {
                hk[h] = hk[h + 1];
                hi[h] = hi[h + 1];
            }
            hk[H - 1] = 0u;
            hi[H - 1] = 0x7FFFFFFF;
            if (++used == H) {
                build(false, lk, li);
                used = 0;
            }
        }
    }
    const float zmax = __shfl_sync(0xffffffffu, zsel, 0);
    float ex = (lane < k) ? expf(zsel - zmax) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        const int64_t TK = (int64_t)T * k;
        const int64_t a = (int64_t)t * k + lane;
        blob[a] = isel;
        blob[TK + a] = __float_as_int(ex / sum);
        if (hist) atomicAdd(hist + (a / chunk) * E + isel, 1);
    }
}

cudaError_t launch_topk(const float* part, int S, const float* bias, float* logits_out, int T, int E, int k,
                        int32_t* blob, uint32_t* err, cudaStream_t stream, int32_t* hist, int chunk) {
    const int warps = 8;
    dim3 grid((unsigned)cdiv(T, warps)), block(32 * warps);
    const int J = (int)cdiv(E, 32);
    cudaError_t e = cudaSuccess;
#define MOE_TOPK(JJ)                                                                                          \
    do {                                                                                                      \
        if (S == 1)                                                                                           \
            e = launch_kernel(topk_kernel<JJ, 1>, grid, block, 0, stream, 1, part, S, bias, logits_out, T, E, k, \
                              blob, hist, chunk, err);                                                        \
        else                                                                                                  \
            e = launch_kernel(topk_kernel<JJ, (JJ <= 16 ? 8 : 2)>, grid, block, 0, stream, 1, part, S, bias,  \
                              logits_out, T, E, k, blob, hist, chunk, err);                                   \
    } while (0)
    if (J <= 1) MOE_TOPK(1);
    else if (J <= 2) MOE_TOPK(2);
    else if (J <= 4) MOE_TOPK(4);
    else if (J <= 8) MOE_TOPK(8);
    else if (J <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
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

// K slices of the router GEMM: up to 8, while twice the units of 256 experts
// x 128 tokens x K/S still fit in one wave on the SMs (the GEMM then narrows
// its expert block only if even that leaves SMs idle: decode-sized T).
int router_splits(int T, int E, int D, int num_sms) {
    const int units = (int)cdiv(T, 128) * std::max(1, E / 256);
    const int kblocks = D / 64;
    int S = 1;
    while (S < 8 && units * S * 2 <= num_sms && kblocks % (2 * S) == 0) S *= 2;
    return S;
}

}  // namespace moe
