// Expert-contiguous permutation of the routed (token, slot) pairs, row
// gathers, and the E4M3 quantisers.
//
// The grouped layout is what the expert GEMMs stream over; its inverse is
// the unpermutation of "Systems engineering playbook: Qwen 3.5 MoE on
// Ironwood TPU" (English page, table in "Pallas Kernels, SparseCore
// Co-Design, and the Roofline").  The order inside each expert's segment is
// the row-major (t, j) order of the pairs -- a stable counting sort -- so the
// layout is deterministic and needs no atomics for positions:
//   1. hist:   per chunk of perm_chunk(T*k) pairs, a histogram over experts;
//   2. scan:   per expert, an exclusive scan over chunks; then counts,
//              offsets (with the shared expert's T rows appended) and the
//              prefix of 128-row tiles the GEMMs walk;
//   3. rank:   per chunk, one warp walks its pairs in order, ranking equal
//              experts inside each 32-pair step with __match_any_sync, and
//              writes inv[pair] and src_tok[row].
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

// SM count of the current device (looked up once per device): the grid cap
// of the grid-stride copy kernels below.
static int current_sms() {
    static const char key = 0;
    int v = 0;
    const cudaError_t e = per_device_value(&key, [](int* out) {
        int dev = 0;
        cudaError_t e2 = cudaGetDevice(&dev);
        return e2 != cudaSuccess ? e2 : cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    }, &v);
    return (e == cudaSuccess && v > 0) ? v : 1;
}

// ------------------------------------------------------------------ hist

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ idx, int64_t TK, int E,
                                                        int32_t* __restrict__ hist, uint32_t* err) {
    pdl_wait_then_release();
    extern __shared__ int32_t sh[];
    const int chunk = perm_chunk(TK);
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
    __syncthreads();
    const int64_t a0 = (int64_t)blockIdx.x * chunk;
    for (int i = threadIdx.x; i < chunk; i += blockDim.x) {
        int64_t a = a0 + i;
        if (a < TK) {
            int e = __ldg(idx + a);
            if ((unsigned)e < (unsigned)E) atomicAdd(&sh[e], 1);
            else record_error(err, MOE_ERR_BOUNDS, (uint32_t)a, (uint32_t)e, 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// ------------------------------------------------------------------ scan

// Warp-wide exclusive scan of n <= 32*33 values in smem `v` into `out`
// (out[n] = total).  Lane l owns a contiguous segment.
__device__ void warp_exclusive_scan(const int32_t* v, int n, int32_t* out) {
    const int lane = threadIdx.x & 31;
    const int seg = (n + 31) / 32;
    const int b = lane * seg, e = min(n, b + seg);
    int s = 0;
    for (int i = b; i < e; ++i) s += v[i];
    int incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    int run = incl - s;
    for (int i = b; i < e; ++i) { out[i] = run; run += v[i]; }
    if (lane == 31) out[n] = incl;
}

// Split expert GEMMs (bf16 layer at prefill sizes): for every group the
// whole 256-row pairs (CTA-pair launch) and the 128-row tiles of the rest
// (single-CTA launch, concurrent on the second stream).  pairs[0 .. E+1]:
// exclusive prefix of the pairs by group; pairs[2(E+2) .. +1]: the number of
// CTA pairs each GEMM's pair launch keeps (gate/up, down), in proportion to
// its share of the work; pairs[2(E+2)+2 .. 3E+4]: the order in which the
// single-CTA launch takes the groups (position -> group), and
// pairs[E+2 .. 2E+3] the exclusive prefix of the rest tiles over those
// positions.
//
// The work is counted in SM cycles per k-block as measured on the bf16
// prefill layer (T=8192, E=512): a pair k-block (256 rows, one on each SM)
// 626 / 633 cycles per SM (gate/up / down), a single-CTA 128-row k-block
// 703 / 889, a narrow (transposed) tail of at most 112 rows 1,063 (gate/up
// only; they stream the whole weight block for few rows).  A pair count off
// this balance leaves one launch waiting for the other: T=8192 took 2.67 ms
// with 56 pairs against 76, 2.14 with 48, 2.36 with 40, against 2.22 ms for
// the single-CTA kernel alone.  The pair side's work is weighted up by
// kPairBias: the single-CTA launch starts after the shared expert's GEMMs on
// its stream, and too few pairs cost far more than too many.  With the group
// order below, alternating runs on three boxes, against 1.1 (the fastest on
// each, 2.11 - 2.13 ms per layer): 1.0 3 % slower, 1.05 up to 2 %, 1.15
// 0.2 %, 1.2 0.5 - 0.9 %, 1.3 1.0 %, 1.45 1.3 %.  1.15 gives up 0.2 % for a
// step of margin from the steep side.
//
// The order: a group with both pairs and a rest has its weights read by both
// launches.  Taken in group order, the single-CTA launch (one or two tiles a
// group) runs far ahead of the pair launch and reads them again from DRAM.
// So a group with pairs comes where the pair launch is halfway through it
// (the midpoint of its pairs as a fraction of all routed pairs), a group with
// only a rest where its midpoint falls among those groups' rest tiles; the
// two lists are merged by that fraction (pair groups first on equal
// fractions), the routed groups without a rest follow in group order and the
// shared group comes last, so that positions [0, E) are the routed groups.
constexpr float kCostPairGU = 626.f, kCostPairDN = 633.f, kCostFullGU = 703.f, kCostFullDN = 889.f,
                kCostNarrowGU = 1063.f, kPairBias = 1.15f;
__device__ __forceinline__ int rest_tiles(int n) { return (n % (2 * kRowTile) + kRowTile - 1) / kRowTile; }
// Entries of sorted[0, n) below key (strict) or at most key (!strict).
__device__ __forceinline__ int count_below(const float* sorted, int n, float key, bool strict) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (strict ? sorted[mid] < key : sorted[mid] <= key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}
// cnt: [E+1] rows per group (shared group last) in shared memory; s_f, s_r:
// [E+2] shared scratch; s_x: [4 (E+2)] shared scratch; s_red: [32 * 4]
// floats.  Every thread of a block of at least 288 threads calls it.
__device__ void pair_split(const int32_t* cnt, int E, int32_t* s_f, int32_t* s_r, int32_t* s_x, float* s_red,
                           int32_t* pairs, int clusters, int narrow_gu) {
    const int S = E + 2;
    int32_t* x_rb = s_x;           // rest tiles of the groups with no pairs
    int32_t* x_cls = s_x + S;      // 1: pairs and a rest; 1 << 16: a rest only
    int32_t* x_rbp = s_x + 2 * S;  // exclusive prefix of x_rb
    int32_t* x_clp = s_x + 3 * S;  // exclusive prefix of x_cls: (pairs-and-rest, rest-only) groups before
    float w[4] = {0.f, 0.f, 0.f, 0.f};  // pair / rest work of gate/up, then down
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int n = cnt[e];
        const int f = n / (2 * kRowTile), r = n % (2 * kRowTile);
        const int rf = r / kRowTile, rt = r % kRowTile;
        const int rest = rf + (rt > 0);
        s_f[e] = f;
        const bool both = e < E && f > 0 && rest > 0, only = e < E && f == 0 && rest > 0;
        x_rb[e] = only ? rest : 0;
        x_cls[e] = (both ? 1 : 0) | (only ? 1 << 16 : 0);
        if (e < E) {
            w[0] += 2.f * kCostPairGU * f;
            w[1] += kCostFullGU * rf + (rt ? ((narrow_gu && rt <= 112) ? kCostNarrowGU : kCostFullGU) : 0.f);
            w[2] += 2.f * kCostPairDN * f;
            w[3] += kCostFullDN * rest;
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w[j] += __shfl_xor_sync(0xffffffffu, w[j], o);
        if (lane == 0) s_red[warp * 4 + j] = w[j];
    }
    __syncthreads();
    const int nw = blockDim.x >> 5;
    if (warp == 4) {
        warp_exclusive_scan(s_f, E + 1, pairs);
    } else if (warp == 5) {
        warp_exclusive_scan(x_rb, E + 1, x_rbp);
    } else if (warp == 6) {
        warp_exclusive_scan(x_cls, E + 1, x_clp);
    } else if (warp == 7) {
        warp_exclusive_scan(s_f, E + 1, s_r);  // the pair prefix, kept in shared memory
    } else if (threadIdx.x == 256) {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < nw; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) t[j] += s_red[i * 4 + j];
        for (int g = 0; g < 2; ++g) {
            const float a = t[2 * g] * kPairBias, b = t[2 * g + 1];
            const int c = (a + b > 0.f) ? (int)lrintf((float)clusters * a / (a + b)) : 0;
            pairs[2 * S + g] = min(clusters, max(0, c));
        }
    }
    __syncthreads();
    // the two lists' fractions, each ascending in group order (x_rb and
    // x_cls were consumed by the scans above)
    const int nA = x_clp[E] & 0xFFFF, nB = x_clp[E] >> 16;
    const float pf2 = 2.f * (float)max(1, s_r[E]), rb2 = 2.f * (float)max(1, x_rbp[E]);
    float* kA = (float*)x_rb;
    float* kB = (float*)x_cls;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int n = cnt[e], rest = rest_tiles(n);
        if (rest == 0) continue;
        if (n >= 2 * kRowTile) kA[x_clp[e] & 0xFFFF] = (2.f * (float)s_r[e] + (float)(n / (2 * kRowTile))) / pf2;
        else kB[x_clp[e] >> 16] = (2.f * (float)x_rbp[e] + (float)rest) / rb2;
    }
    __syncthreads();
    int32_t* order = pairs + 2 * S + 2;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int n = cnt[e], rest = rest_tiles(n);
        const int ia = x_clp[e] & 0xFFFF, ib = x_clp[e] >> 16;
        int pos;
        if (e == E) pos = E;
        else if (rest == 0) pos = nA + nB + (e - ia - ib);
        else if (n >= 2 * kRowTile) pos = ia + count_below(kB, nB, kA[ia], true);
        else pos = ib + count_below(kA, nA, kB[ib], false);
        order[pos] = e;
        s_f[pos] = rest;  // rest tiles by position (s_f's pair counts were scanned above)
    }
    __syncthreads();
    if (warp == 5) warp_exclusive_scan(s_f, E + 1, pairs + S);
}

__global__ void __launch_bounds__(512) perm_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E, int T,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ tiles, int32_t* __restrict__ tiles2,
                                                         int32_t* __restrict__ shared_src, int64_t TK,
                                                         int32_t* __restrict__ pairs, int clusters, int narrow_gu) {
    pdl_wait_then_release();
    __shared__ int32_t cnt[1025 + 1];
    __shared__ int32_t s_pf[1025 + 1], s_pr[1025 + 1];
    __shared__ float s_red[32 * 4];
    __shared__ int32_t s_px[4 * (1025 + 1)];
    __shared__ int32_t ntile[1025 + 1];
    __shared__ int32_t ntile2[1025 + 1];
    // the shared expert's rows: token t at grouped row T*k + t
    for (int t = threadIdx.x; t < T; t += blockDim.x) shared_src[TK + t] = t;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        // 32 independent loads in flight per step of the running sum (the
        // last step predicated): 3 round trips to L2 for the 80 chunks of
        // T*k = 81,920 pairs instead of 10
        constexpr int U = 32;
        int run = 0;
        for (int c = 0; c < nchunks; c += U) {
            int v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = (c + u < nchunks) ? hist[(int64_t)(c + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (c + u < nchunks) hist[(int64_t)(c + u) * E + e] = run;
                run += v[u];
            }
        }
        cnt[e] = run;
        ntile[e] = (run + kRowTile - 1) / kRowTile;
        ntile2[e] = (run + 2 * kRowTile - 1) / (2 * kRowTile);
    }
    if (threadIdx.x == 0) {
        cnt[E] = T;
        ntile[E] = (T + kRowTile - 1) / kRowTile;
        ntile2[E] = (T + 2 * kRowTile - 1) / (2 * kRowTile);
    }
    __syncthreads();
    if (pairs) pair_split(cnt, E, s_pf, s_pr, s_px, s_red, pairs, clusters, narrow_gu);
    for (int e = threadIdx.x; e <= E; e += blockDim.x) counts[e] = cnt[e];
    if (threadIdx.x < 32) warp_exclusive_scan(cnt, E + 1, offsets);
    else if (threadIdx.x < 64) warp_exclusive_scan(ntile, E + 1, tiles);
    else if (threadIdx.x < 96 && tiles2) warp_exclusive_scan(ntile2, E + 1, tiles2);
}

// ------------------------------------------------------------------ rank

// One block of 8 warps per chunk: warp w owns the w-th eighth of the chunk's
// pairs.  Each warp counts its pairs per expert, the block turns the counts
// into per-warp cursors (chunk start from the scan, plus the counts of the
// warps before), and each warp then ranks its pairs in order, 32 at a time,
// ranking equal experts inside a step with __match_any_sync.
constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(32 * kRankWarps) perm_rank_kernel(const int32_t* __restrict__ idx, int64_t TK,
                                                                    int k, int E,
                                                                    const int32_t* __restrict__ hist,
                                                                    const int32_t* __restrict__ offsets,
                                                                    int32_t* __restrict__ inv,
                                                                    int32_t* __restrict__ src_tok) {
    pdl_wait_then_release();
    extern __shared__ int32_t cur[];  // [kRankWarps][E]: counts, then cursors
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = perm_chunk(TK);
    const int per = chunk / kRankWarps;  // pairs per warp (16 or 128)
    const int64_t a0 = (int64_t)blockIdx.x * chunk + (int64_t)warp * per;
    constexpr int kSteps = kPermChunk / kRankWarps / 32;
    int ids[kSteps];
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        const int64_t a = a0 + 32 * s + lane;
        int e = (32 * s + lane < per && a < TK) ? __ldg(idx + a) : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;  // out-of-range ids were reported by hist
        ids[s] = e;
    }
    for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) cur[i] = 0;
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kSteps; ++s)
        if (ids[s] >= 0) atomicAdd(&cur[warp * E + ids[s]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = __ldg(offsets + e) + __ldg(hist + (int64_t)blockIdx.x * E + e);
#pragma unroll
        for (int w = 0; w < kRankWarps; ++w) {
            const int c = cur[w * E + e];
            cur[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    int32_t* cw = cur + warp * E;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        if (32 * s >= per) break;
        const int64_t a = a0 + 32 * s + lane;
        const int e = ids[s];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = cw[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && (peers >> lane) == 1u) cw[e] += __popc(peers);  // highest lane of the group
        __syncwarp();
        if (e >= 0) {
            inv[a] = pos;
            src_tok[pos] = (int32_t)(a / k);
        } else if (32 * s + lane < per && a < TK) {
            inv[a] = -1;  // a dropped pair (its expert id was out of range)
        }
    }
}

// ------------------------------------------------- small problems, one block
//
// The same stable counting sort for T*k <= kSmallPairs pairs in one launch of
// one 1024-thread block, everything in shared memory: warp w owns the w-th
// 32nd of the pairs (histogram, then its ranks), thread e scans expert e over
// the 32 warps.  Decode-sized routing (1280 pairs) spends ~5 us here instead
// of four dependent launches.
constexpr int kSmallPairs = 16384;
constexpr int kSmallMaxE = 512;
constexpr int kSmallSmem = (32 * kSmallMaxE + 10 * (kSmallMaxE + 2) + 32 * 4) * 4;

__global__ void __launch_bounds__(1024) perm_index_small_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                                int32_t* __restrict__ counts,
                                                                int32_t* __restrict__ offsets,
                                                                int32_t* __restrict__ tiles,
                                                                int32_t* __restrict__ tiles2, int32_t* __restrict__ inv,
                                                                int32_t* __restrict__ src_tok, uint32_t* err,
                                                                int32_t* __restrict__ pairs, int clusters,
                                                                int narrow_gu) {
    pdl_wait_then_release();
    extern __shared__ int32_t sm[];
    int32_t* hist = sm;                   // [32][E]: per-warp counts, then cursors
    int32_t* cnt = hist + 32 * E;         // [E+1]
    int32_t* nt = cnt + (E + 2);          // [E+1] 128-row tiles
    int32_t* nt2 = nt + (E + 2);          // [E+1] 256-row tiles
    int32_t* off = nt2 + (E + 2);         // [E+2]
    int32_t* s_pf = off + (E + 2);        // [E+1] pair split scratch
    int32_t* s_pr = s_pf + (E + 2);       // [E+1]
    float* s_red = (float*)(s_pr + (E + 2));  // [32 * 4]
    int32_t* s_px = (int32_t*)(s_red + 32 * 4);  // [4 (E+2)]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TK = T * k;
    const int per = (TK + 31) / 32;
    const int a0 = warp * per, a1 = min(TK, a0 + per);
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int a = a0 + lane; a < a1; a += 32) {
        const int e = __ldg(idx + a);
        if ((unsigned)e < (unsigned)E) atomicAdd(&hist[warp * E + e], 1);
        else record_error(err, MOE_ERR_BOUNDS, (uint32_t)a, (uint32_t)e, 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) {
            const int v = hist[w * E + e];
            hist[w * E + e] = run;
            run += v;
        }
        cnt[e] = run;
        nt[e] = (run + kRowTile - 1) / kRowTile;
        nt2[e] = (run + 2 * kRowTile - 1) / (2 * kRowTile);
    }
    if (threadIdx.x == 0) {
        cnt[E] = T;
        nt[E] = (T + kRowTile - 1) / kRowTile;
        nt2[E] = (T + 2 * kRowTile - 1) / (2 * kRowTile);
    }
    __syncthreads();
    if (pairs) pair_split(cnt, E, s_pf, s_pr, s_px, s_red, pairs, clusters, narrow_gu);
    if (warp == 0) warp_exclusive_scan(cnt, E + 1, off);
    else if (warp == 1) warp_exclusive_scan(nt, E + 1, tiles);
    else if (warp == 2 && tiles2) warp_exclusive_scan(nt2, E + 1, tiles2);
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) counts[e] = cnt[e];
    for (int e = threadIdx.x; e <= E + 1; e += blockDim.x) offsets[e] = off[e];
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) hist[i] += off[i % E];  // cursors
    for (int t = threadIdx.x; t < T; t += blockDim.x) src_tok[TK + t] = t;
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    int32_t* cur = hist + warp * E;
    for (int s = a0; s < a1; s += 32) {
        const int a = s + lane;
        int e = (a < a1) ? __ldg(idx + a) : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = cur[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && (peers >> lane) == 1u) cur[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            inv[a] = pos;
            src_tok[pos] = a / k;
        } else if (a < a1) {
            inv[a] = -1;  // a dropped pair (its expert id was out of range)
        }
    }
}

bool permute_uses_chunks(int64_t TK, int E) { return !(TK <= kSmallPairs && E <= kSmallMaxE); }

cudaError_t launch_permute_index(const int32_t* idx, int T, int E, int k, int32_t* hist, int32_t* counts,
                                 int32_t* offsets, int32_t* tiles, int32_t* tiles2, int32_t* inv, int32_t* src_tok,
                                 uint32_t* err, cudaStream_t stream, bool hist_ready, int32_t* pairs, int clusters,
                                 int narrow_gu) {
    const int64_t TK = (int64_t)T * k;
    if (!permute_uses_chunks(TK, E)) {
        cudaError_t e = ensure_smem_attr((const void*)perm_index_small_kernel, kSmallSmem);
        if (e != cudaSuccess) return e;
        const int smem = (32 * E + 10 * (E + 2) + 32 * 4) * 4;
        e = launch_kernel(perm_index_small_kernel, dim3(1), dim3(1024), smem, stream, 1, idx, T, E, k, counts, offsets,
                          tiles, tiles2, inv, src_tok, err, pairs, clusters, narrow_gu);
        count_launches(1);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int nch = (int)cdiv(TK, perm_chunk(TK));
    cudaError_t e = cudaSuccess;
    if (!hist_ready)
        e = launch_kernel(perm_hist_kernel, dim3(nch), dim3(256), E * sizeof(int32_t), stream, 1, idx, TK, E, hist, err);
    if (e == cudaSuccess)
        e = launch_kernel(perm_scan_kernel, dim3(1), dim3(512), 0, stream, 1, hist, nch, E, T, counts, offsets, tiles,
                          tiles2, src_tok, TK, pairs, clusters, narrow_gu);
    if (e != cudaSuccess) return e;
    const int rank_smem = kRankWarps * E * (int)sizeof(int32_t);
    if (rank_smem > 48 * 1024) {
        e = ensure_smem_attr((const void*)perm_rank_kernel, rank_smem);
        if (e != cudaSuccess) return e;
    }
    e = launch_kernel(perm_rank_kernel, dim3(nch), dim3(32 * kRankWarps), rank_smem, stream, 1, idx, TK, k, E,
                      (const int32_t*)hist, (const int32_t*)offsets, inv, src_tok);
    count_launches(hist_ready ? 2 : 3);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------- gather

// xp[p] = x[src_tok[p]] for p < rows; one warp per row, 16-byte vectors when
// the row size allows, else 4-byte words.  Each x row is read about top_k
// times, so x should stay in L2 while xp (top_k times larger) streams out:
// the stores carry the evict-first hint (st.global.cs).
template <typename V>
__global__ void __launch_bounds__(256) gather_rows_kernel(const V* __restrict__ x, int64_t row_vecs,
                                                          const int32_t* __restrict__ src_tok, int rows,
                                                          V* __restrict__ xp) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const V* src = x + (int64_t)__ldg(src_tok + r) * row_vecs;
        V* dst = xp + (int64_t)r * row_vecs;
        int64_t i = lane;
        for (; i + 32 * 7 < row_vecs; i += 32 * 8) {  // 8 independent loads per lane in flight
            V t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t[u] = __ldg(src + i + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) __stcs(dst + i + 32 * u, t[u]);
        }
        for (; i < row_vecs; i += 32) __stcs(dst + i, __ldg(src + i));
    }
}

// xp[inv[t*k + j]] = x[t] for every token t and slot j: one warp per token
// reads the row once (8 vectors per lane at a time) and writes it to its k
// rows of the grouped layout, with the evict-first hint.  Each x row is
// read from DRAM once, where a gather by output row reads it k times
// through an L2 that the k-times larger output keeps flushing.  Dropped
// pairs (inv < 0) are skipped.
template <typename V>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const V* __restrict__ x, int64_t row_vecs,
                                                           const int32_t* __restrict__ inv, int T, int k,
                                                           int64_t rows_out, V* __restrict__ xp) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
        const int my = lane < k ? __ldg(inv + (int64_t)t * k + lane) : -1;
        const V* src = x + (int64_t)t * row_vecs;
        for (int64_t i0 = 0; i0 < row_vecs; i0 += 32 * 8) {
            V v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + lane + 32 * u;
                if (i < row_vecs) v[u] = __ldg(src + i);
            }
            for (int j = 0; j < k; ++j) {
                const int r = __shfl_sync(0xffffffffu, my, j);
                if (r < 0 || r >= rows_out) continue;
                V* dst = xp + (int64_t)r * row_vecs;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t i = i0 + lane + 32 * u;
                    if (i < row_vecs) __stcs(dst + i, v[u]);
                }
            }
        }
    }
}

cudaError_t launch_scatter_rows(const void* x, int64_t row_bytes, const int32_t* inv, int T, int k, void* xp,
                                cudaStream_t stream) {
    if (T <= 0) return cudaGetLastError();
    const int blocks = (int)std::min<int64_t>(cdiv(T, 8), (int64_t)current_sms() * 16);
    const int64_t rows_out = (int64_t)T * k;
    cudaError_t e;
    if (row_bytes % 16 == 0)
        e = launch_kernel(scatter_rows_kernel<int4>, dim3(blocks), dim3(256), 0, stream, 1, (const int4*)x,
                          row_bytes / 16, inv, T, k, rows_out, (int4*)xp);
    else
        e = launch_kernel(scatter_rows_kernel<int32_t>, dim3(blocks), dim3(256), 0, stream, 1, (const int32_t*)x,
                          row_bytes / 4, inv, T, k, rows_out, (int32_t*)xp);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, int elem_bytes, int64_t row_bytes, const int32_t* src_tok, int rows,
                               void* xp, cudaStream_t stream) {
    (void)elem_bytes;
    if (rows <= 0) return cudaGetLastError();
    int blocks = (int)std::min<int64_t>(cdiv(rows, 8), (int64_t)current_sms() * 16);
    cudaError_t e;
    if (row_bytes % 16 == 0)
        e = launch_kernel(gather_rows_kernel<int4>, dim3(blocks), dim3(256), 0, stream, 1, (const int4*)x,
                          row_bytes / 16, src_tok, rows, (int4*)xp);
    else
        e = launch_kernel(gather_rows_kernel<int32_t>, dim3(blocks), dim3(256), 0, stream, 1, (const int32_t*)x,
                          row_bytes / 4, src_tok, rows, (int32_t*)xp);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------- quantisers

// Per row, per 128-column group: s = amax / 448 (1 if the group is all
// zero), code = E4M3_rne_satfinite(fp32(v * fp32(448 / amax))).  A half-warp
// per group (8 bf16 = one 16-byte load per lane, 8 codes = one 8-byte store),
// so a warp quantises two groups per step.
__device__ __forceinline__ void load8f(const bf16* p, float* v) {
    const uint4 raw = __ldg((const uint4*)p);
    const __nv_bfloat162* h = (const __nv_bfloat162*)&raw;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8f(const float* p, float* v) {
    const float4 a = __ldg((const float4*)p), b = __ldg((const float4*)p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(256) quant_rows_kernel(const T* __restrict__ x, int rows, int cols,
                                                         uint8_t* __restrict__ q, float* __restrict__ s) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const int gpr = cols / 128;
    const int64_t ngroups = (int64_t)rows * gpr;
    const int64_t halves = ((int64_t)gridDim.x * blockDim.x) >> 4;
    // every lane walks the same number of steps, so the shuffles below see
    // the whole warp; groups past the end compute on zeros and store nothing
    const int64_t steps = (ngroups + halves - 1) / halves;
    int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
    for (int64_t it = 0; it < steps; ++it, g += halves) {
        const bool ok = g < ngroups;
        const int64_t r = ok ? g / gpr : 0;
        const int64_t c0 = ok ? (g - r * gpr) * 128 + sub * 8 : 0;
        float v[8];
        if (ok) load8f(x + r * cols + c0, v);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        float sc = __fdiv_rn(amax, 448.0f), inv = __fdiv_rn(448.0f, amax);
        if (amax == 0.0f) { sc = 1.0f; inv = 1.0f; }
        if (ok) {
            uint2 packed;
            packed.x = (uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
                       ((uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
            packed.y = (uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv)) |
                       ((uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[6], inv), __fmul_rn(v[7], inv)) << 16);
            *(uint2*)(q + r * cols + c0) = packed;
            if (sub == 0) s[g] = sc;
        }
    }
}

cudaError_t launch_quant_rows(const void* x, int x_elem, int rows, int cols, uint8_t* q, float* s,
                              cudaStream_t stream) {
    if (rows <= 0) return cudaGetLastError();
    int64_t groups = (int64_t)rows * (cols / 128);
    int blocks = (int)std::min<int64_t>(cdiv(groups, 16), (int64_t)current_sms() * 32);
    if (x_elem == kBF16)
        quant_rows_kernel<bf16><<<blocks, 256, 0, stream>>>((const bf16*)x, rows, cols, q, s);
    else
        quant_rows_kernel<float><<<blocks, 256, 0, stream>>>((const float*)x, rows, cols, q, s);
    count_launches(1);
    return cudaGetLastError();
}

// The FP8 layer's permutation at scatter sizes: x is quantised and
// scattered in one pass.  One warp per token quantises its row two
// 128-column groups at a time (a half-warp per group, 8 values per lane,
// four steps of loads in flight) exactly as quant_rows_kernel does (same
// values, amax, scale and rounding: the codes and scales are
// bit-identical), into a per-warp copy of the code row and its scales in
// shared memory; then it writes that copy to each of the token's k rows of
// xp / xp_scale in 16-byte vectors.  Against quant_rows + scatter of the
// codes + gather of the scales this reads x once and skips the xq round
// trip and two launches.
constexpr int kSqMaxCols = 4096;  // shared row copy per warp (larger D: not supported here)
constexpr int kSqWarps = 8;
__global__ void __launch_bounds__(32 * kSqWarps) scatter_quant_rows_kernel(const bf16* __restrict__ x, int Tn, int cols,
                                                                           const int32_t* __restrict__ inv, int k,
                                                                           int64_t rows_out, uint8_t* __restrict__ xp,
                                                                           float* __restrict__ xp_scale) {
    pdl_wait_then_release();
    __shared__ __align__(16) uint8_t s_code[kSqWarps][kSqMaxCols];
    __shared__ float s_sc[kSqWarps][kSqMaxCols / 128];
    const int lane = threadIdx.x & 31, sub = lane & 15, hw = lane >> 4, w = threadIdx.x >> 5;
    const int gpr = cols / 128;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += warps) {
        const int my = lane < k ? __ldg(inv + (int64_t)t * k + lane) : -1;
        const bf16* row = x + (int64_t)t * cols;
        constexpr int B = 4;  // steps (pairs of groups) whose loads are in flight together
        for (int g0 = 0; g0 < gpr; g0 += 2 * B) {
            uint4 raw[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int g = g0 + 2 * b + hw;
                raw[b] = g < gpr ? __ldg((const uint4*)(row + (int64_t)g * 128 + sub * 8)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int g = g0 + 2 * b + hw;
                float v[8];
                const __nv_bfloat162* h2 = (const __nv_bfloat162*)&raw[b];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h2[i]);
                    v[2 * i] = f.x;
                    v[2 * i + 1] = f.y;
                }
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                float sc = __fdiv_rn(amax, 448.0f), iv = __fdiv_rn(448.0f, amax);
                if (amax == 0.0f) { sc = 1.0f; iv = 1.0f; }
                if (g < gpr) {
                    uint2 packed;
                    packed.x = (uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[0], iv), __fmul_rn(v[1], iv)) |
                               ((uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[2], iv), __fmul_rn(v[3], iv)) << 16);
                    packed.y = (uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[4], iv), __fmul_rn(v[5], iv)) |
                               ((uint32_t)f32x2_to_e4m3x2(__fmul_rn(v[6], iv), __fmul_rn(v[7], iv)) << 16);
                    *(uint2*)(&s_code[w][g * 128 + sub * 8]) = packed;
                    if (sub == 0) s_sc[w][g] = sc;
                }
            }
        }
        __syncwarp();
        const int nvec = cols / 16;  // 16-byte vectors of the code row
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(0xffffffffu, my, j);
            if (r < 0 || r >= rows_out) continue;
            uint8_t* dst = xp + (int64_t)r * cols;
            for (int i = lane; i < nvec; i += 32) __stcs((uint4*)(dst + 16 * i), *(const uint4*)(&s_code[w][16 * i]));
            for (int g = lane; g < gpr; g += 32) xp_scale[(int64_t)r * gpr + g] = s_sc[w][g];
        }
        __syncwarp();
    }
}

cudaError_t launch_scatter_quant_rows(const void* x, int x_elem, int T, int cols, const int32_t* inv, int k,
                                      uint8_t* xp, float* xp_scale, cudaStream_t stream) {
    if (T <= 0) return cudaGetLastError();
    const int blocks = (int)std::min<int64_t>(cdiv(T, 8), (int64_t)current_sms() * 16);
    const int64_t rows_out = (int64_t)T * k;
    if (x_elem != kBF16 || cols > kSqMaxCols || cols % 128) return cudaErrorInvalidValue;  // bf16 x, D <= 4096
    cudaError_t e = launch_kernel(scatter_quant_rows_kernel, dim3(blocks), dim3(32 * kSqWarps), 0, stream, 1, (const bf16*)x,
                                  T, cols, inv, k, rows_out, xp, xp_scale);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// One block per 128x128 weight block of a [groups, rows, cols] fp32 tensor.
__global__ void __launch_bounds__(256) quant_blocks_kernel(const float* __restrict__ w, int rows, int cols,
                                                           uint8_t* __restrict__ q, float* __restrict__ s) {
    __shared__ float red[8];
    const int nbr = rows / 128, nbc = cols / 128;
    const int64_t b = blockIdx.x;
    const int64_t g = b / (nbr * nbc);
    const int br = (int)((b / nbc) % nbr), bc = (int)(b % nbc);
    const float* base = w + g * (int64_t)rows * cols + (int64_t)br * 128 * cols + bc * 128;
    uint8_t* qb = q + g * (int64_t)rows * cols + (int64_t)br * 128 * cols + bc * 128;
    const int c4 = (threadIdx.x & 31) * 4, r0 = threadIdx.x >> 5;  // 8 rows per pass
    float amax = 0.0f;
    for (int r = r0; r < 128; r += 8) {
        float4 v = *(const float4*)(base + (int64_t)r * cols + c4);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    float sc = __fdiv_rn(amax, 448.0f), inv = __fdiv_rn(448.0f, amax);
    if (amax == 0.0f) { sc = 1.0f; inv = 1.0f; }
    if (threadIdx.x == 0) s[b] = sc;
    for (int r = r0; r < 128; r += 8) {
        float4 v = *(const float4*)(base + (int64_t)r * cols + c4);
        uint32_t packed = (uint32_t)f32_to_e4m3(__fmul_rn(v.x, inv)) | ((uint32_t)f32_to_e4m3(__fmul_rn(v.y, inv)) << 8) |
                          ((uint32_t)f32_to_e4m3(__fmul_rn(v.z, inv)) << 16) |
                          ((uint32_t)f32_to_e4m3(__fmul_rn(v.w, inv)) << 24);
        *(uint32_t*)(qb + (int64_t)r * cols + c4) = packed;
    }
}

// bf16 -> fp16 for the down projection's tensor-core copy.  Every bf16 of
// magnitude 2^-17 .. 65504 is an fp16 exactly (fp16 keeps 3 more mantissa
// bits); smaller magnitudes round to fp16's subnormal grid (2^-24).  A finite
// bf16 beyond 65504 has no fp16: it is recorded as MOE_ERR_BOUNDS.
__global__ void bf16_to_f16_kernel(const bf16* __restrict__ src, f16* __restrict__ dst, int64_t n, uint32_t* err) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = __bfloat162float(src[i]);
        if (isfinite(v) && fabsf(v) > 65504.0f) record_error(err, MOE_ERR_BOUNDS, (uint32_t)(i & 0xffffffff), 0, 3);
        dst[i] = __float2half_rn(v);
    }
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, uint32_t* err, cudaStream_t stream) {
    if (n <= 0) return cudaGetLastError();
    const int blocks = (int)std::min<int64_t>(cdiv(n, 256), 152 * 64);
    bf16_to_f16_kernel<<<blocks, 256, 0, stream>>>((const bf16*)src, (f16*)dst, n, err);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_quant_blocks(const float* w, int64_t groups, int rows, int cols, uint8_t* q, float* s,
                                cudaStream_t stream) {
    int64_t nb = groups * (rows / 128) * (cols / 128);
    if (nb <= 0) return cudaGetLastError();
    quant_blocks_kernel<<<(unsigned)nb, 256, 0, stream>>>(w, rows, cols, q, s);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe

// ------------------------------------------------- allocation-free variant
//
// Some callers cannot call cudaMalloc at all: a plugin inside a host
// framework that owns every byte of device memory through its own arena, or
// a serving loop that forbids allocation (and the device synchronisation it
// can imply) once it has started.  They still pass their inputs and outputs;
// the only extra memory the permutation index build needs -- the per-chunk
// expert histograms -- lives here, in one file-scope device array that every
// GPU loading this library holds until the process exits.

namespace moe {
namespace {

constexpr int kNoAllocHistInts = 1 << 18;  // 1 MiB: chunks * E <= 262144
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) int32_t g_noalloc_hist[kNoAllocHistInts];

std::mutex g_noalloc_mu;
int32_t* g_noalloc_addr[kNoAllocMaxDevices] = {};

}  // namespace

}  // namespace moe

extern "C" MOE_API moe_status moe_permute_index_noalloc(const int32_t* idx, int32_t T, int32_t E, int32_t top_k,
                                                        int32_t* counts, int32_t* offsets, int32_t* tiles,
                                                        int32_t* inv, int32_t* src_tok, void* stream) {
    using namespace moe;
    if (!idx || !counts || !offsets || !tiles || !inv || !src_tok) return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * (top_k + 1) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    const int64_t chunks = cdiv((int64_t)T * top_k, perm_chunk((int64_t)T * top_k));
    if (chunks * E > kNoAllocHistInts) return MOE_ERR_UNSUPPORTED;  // beyond the static scratch
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_CUDA;
    int32_t* hist = nullptr;
    {
        // First call on this device: look up the array's device address
        // (the host-side name is only a stand-in, not a device pointer).
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_hist) != cudaSuccess || !p) return MOE_ERR_CUDA;
            g_noalloc_addr[dev] = (int32_t*)p;
        }
        hist = g_noalloc_addr[dev];
    }
    // Every histogram entry a chunk uses is written by the hist kernel before
    // the scan reads it, so what an earlier call left in the array is never
    // read and nothing needs clearing.
    if (launch_permute_index(idx, T, E, top_k, hist, counts, offsets, tiles, nullptr, inv, src_tok, nullptr,
                             (cudaStream_t)stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
