// Grouped bf16 GEMM on CTA pairs: tcgen05.mma.cta_group::2, M = 256.
//
// Same computation and epilogues as gemm_tc.cu, for the prefill regime where
// groups hold hundreds of rows and the single-CTA tile (128 x 256) needs 48 KB
// of operands per 512 MMA cycles -- more than L2 keeps up with under load.
// Two CTAs of a cluster share one 256 x 256 tile: each loads its own 128 rows
// of A and half of the B tile (128 of the 256 weight rows), the pair's leader
// issues M=256 MMAs that read both CTAs' shared memory, and each CTA's TMEM
// receives its own 128 rows x 256 columns.  Per CTA that is 32 KB per 512
// cycles, and the ring deepens from 4 to 6 stages (hi/lo pair input: 4).
//   SwiGLU: CTA 0 holds the 128 gate rows, CTA 1 the 128 up rows of the same
//     features, so accumulator columns 0..127 are gate and 128..255 up in both.
//   Plain: CTA r holds weight rows nb*256 + r*128 .. +127.
// Synchronisation: both CTAs' copies complete on the leader's "full"
// barriers (the leader registers the pair's byte count); the leader's MMA
// commits arrive on "empty" and "TMEM full" barriers in both CTAs
// (multicast); both CTAs' epilogue warps arrive on the leader's "TMEM empty"
// barriers.  All waits are bounded as in gemm_tc.cu.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows);

namespace p2 {

constexpr int BM = 128;                 // rows per CTA; a pair covers 256
constexpr int BK = 64;
constexpr int kABytes = BM * BK * 2;    // 16 KB
constexpr int kBHalf = 128 * BK * 2;    // 16 KB: this CTA's half of the B tile
constexpr int kThreads = 192;
constexpr int kAccCols = 256;
constexpr int kBoxRowsA = 16;
constexpr int kRing = 196608;
constexpr uint32_t kSmemBytes = 1024 + kRing + 256;

template <bool PAIR> struct Geo {
    static constexpr int kAStage = PAIR ? 2 * kABytes : kABytes;
    static constexpr int kStages = kRing / (kAStage + kBHalf);  // 6, or 4 with the hi/lo pair
};

enum Epi : int { EPI_SWIGLU = 0, EPI_PLAIN = 1 };

struct Params {
    int G, shared_group;
    const int32_t* offsets;
    const int32_t* tiles2;  // prefix of ceil(rows/256)
    int NB, N, KB, a_lo_x, ldo, out_pair, out_f32, out_f16, in_f16;
    void* out;
    uint32_t* err;
    int64_t spin_ns;
};

struct Unit {
    int g, m0pair, row0, nrows, nb;
};

__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
    Unit r;
    const int rt = u / p.NB;
    r.nb = u - rt * p.NB;
    r.g = find_group(p.tiles2, p.G, rt);
    r.m0pair = (rt - __ldg(p.tiles2 + r.g)) * 2 * BM;
    r.row0 = __ldg(p.offsets + r.g);
    r.nrows = __ldg(p.offsets + r.g + 1) - r.row0;
    return r;
}

__device__ __forceinline__ int boxes_for(int nrows, int m0) {
    const int valid = max(0, min(BM, nrows - m0));
    return (valid + kBoxRowsA - 1) / kBoxRowsA;
}

__device__ __forceinline__ void store_f16x32(f16* dst, const float* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 pk;
        __half2* h2 = (__half2*)&pk;
#pragma unroll
        for (int i = 0; i < 4; ++i) h2[i] = __floats2half2_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        *(uint4*)(dst + 8 * q) = pk;
    }
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 pk;
        __nv_bfloat162* h2 = (__nv_bfloat162*)&pk;
#pragma unroll
        for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        *(uint4*)(dst + 8 * q) = pk;
    }
}

template <int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a_sh,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_b2,
                    const __grid_constant__ CUtensorMap tm_af, const __grid_constant__ CUtensorMap tm_a_shf,
                    const Params p) {
    constexpr int kStages = Geo<PAIR>::kStages;
    constexpr int kAStage = Geo<PAIR>::kAStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kAStage;
    uint64_t* bars = (uint64_t*)(smem + kRing);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kStages), tempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
    uint32_t* tmem_slot = (uint32_t*)(bars + 2 * kStages + 5);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 2 * 4);  // four epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), 2 * kAccCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nclusters = gridDim.x >> 1, cid = blockIdx.x >> 1;
    const int total_units = __ldg(p.tiles2 + p.G) * p.NB;
    const int64_t lim = p.spin_ns;
    bool aborted = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            for (int u = cid; u < total_units; u += nclusters) {
                const Unit un = decode_unit(p, u);
                const bool sh = un.g == p.shared_group;
                const CUtensorMap* ta = sh ? &tm_a_sh : &tm_a;
                const CUtensorMap* taf = sh ? &tm_a_shf : &tm_af;
                const int m0 = un.m0pair + (int)rank * BM;
                const int nbox = boxes_for(un.nrows, m0);
                const int a_y = sh ? m0 : un.row0 + m0;
                const uint32_t pair_bytes =
                    (PAIR ? 2u : 1u) * (uint32_t)(boxes_for(un.nrows, un.m0pair) + boxes_for(un.nrows, un.m0pair + BM)) *
                        kBoxRowsA * BK * 2 +
                    2u * kBHalf;
                const CUtensorMap* tb = (EPI == EPI_SWIGLU && rank == 1) ? &tm_b2 : &tm_b;
                const int b_y = un.g * p.N + ((EPI == EPI_SWIGLU) ? un.nb * 128 : un.nb * 256 + (int)rank * 128);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 21, blockIdx.x, u);
                        *abort_flag = 1;
                        aborted = true;
                        break;
                    }
                    const uint32_t fb_local = full0 + 8 * stage;
                    const uint32_t fb = mapa_shared(fb_local, 0);  // the leader's full barrier
                    if (leader) mbar_expect_tx(fb_local, pair_bytes);
                    const uint32_t a_dst = smem_u32(sA + stage * kAStage);
                    const uint32_t b_dst = smem_u32(sB + stage * kBHalf);
                    if (nbox * kBoxRowsA == BM) {  // full half-tile: one 128-row box
                        tma_load_2d_pair(a_dst, taf, fb, kb * BK, a_y);
                        if (PAIR) tma_load_2d_pair(a_dst + kABytes, taf, fb, p.a_lo_x + kb * BK, a_y);
                    } else {
                        for (int i = 0; i < nbox; ++i) {
                            tma_load_2d_pair(a_dst + i * kBoxRowsA * 128, ta, fb, kb * BK, a_y + i * kBoxRowsA);
                            if (PAIR)
                                tma_load_2d_pair(a_dst + kABytes + i * kBoxRowsA * 128, ta, fb,
                                                 p.a_lo_x + kb * BK, a_y + i * kBoxRowsA);
                        }
                    }
                    tma_load_2d_pair(b_dst, tb, fb, kb * BK, b_y);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (aborted) break;
            }
            if (aborted) sleep_ns(200000);  // copies already issued land before the CTA leaves
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------ MMA issuer (leader only)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t idesc = p.in_f16 ? idesc_f16(2 * BM, 256) : idesc_bf16(2 * BM, 256);
            for (int u = cid; u < total_units && !aborted; u += nclusters) {
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 22, blockIdx.x, u);
                    *abort_flag = 1;
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 23, blockIdx.x, u);
                        *abort_flag = 1;
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_desc(smem_u32(sA + stage * kAStage));
                    const uint64_t bd = umma_desc(smem_u32(sB + stage * kBHalf));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                    if (PAIR) {
                        const uint64_t al = umma_desc(smem_u32(sA + stage * kAStage + kABytes));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_pair(d, al + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, 1u);
                    }
                    umma_commit_pair(empty0 + 8 * stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (aborted) break;
                umma_commit_pair(tfull0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            umma_commit_pair(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, 1000000000LL, &never);
        }
    } else {
        // --------------------------------------------- epilogue (both CTAs)
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = cid; u < total_units; u += nclusters) {
            const Unit un = decode_unit(p, u);
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(tfull0 + 8 * acc, acc_phase, lim, abort_flag);
                if (!ok) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 24, blockIdx.x, u);
                    *abort_flag = 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int m = un.m0pair + (int)rank * BM + row;
            const bool valid = m < un.nrows;
            const int64_t orow = (int64_t)un.row0 + m;
            const uint32_t tb = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kAccCols);
            if (EPI == EPI_SWIGLU) {
                bf16* o = (bf16*)p.out + orow * p.ldo + un.nb * 128;
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(tb + c, gr);
                    tmem_ld32(tb + 128 + c, ur);
                    tmem_wait_ld();
                    if (valid) {
                        float h[32], lo[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) h[i] = swiglu(__uint_as_float(gr[i]), __uint_as_float(ur[i]));
                        if (p.out_f16) {
                            float m = 0.f;
#pragma unroll
                            for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(h[i]));
                            if (!(m <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 5, blockIdx.x, 0);
                            store_f16x32((f16*)o + c, h);
                            continue;
                        }
                        store_bf16x32(o + c, h);
                        if (p.out_pair) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) lo[i] = h[i] - __bfloat162float(__float2bfloat16_rn(h[i]));
                            store_bf16x32(o + p.N + c, lo);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    if (valid) {
                        const int n0 = un.nb * 256 + c;
                        if (p.out_f32) {
                            float* o = (float*)p.out + orow * p.ldo + n0;
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *(float4*)(o + i) = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                                __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                        } else {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                            if (p.out_f16) {
                                float m = 0.f;
#pragma unroll
                                for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
                                if (!(m <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 6, blockIdx.x, 0);
                                store_f16x32((f16*)p.out + orow * p.ldo + n0, v);
                            } else {
                                store_bf16x32((bf16*)p.out + orow * p.ldo + n0, v);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no cross-CTA arrivals or copies remain in flight
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 2 * kAccCols);
    }
}

template <int EPI, bool PAIR>
cudaError_t launch_one(const CUtensorMap& ma, const CUtensorMap& msh, const CUtensorMap& mb, const CUtensorMap& mb2,
                       const CUtensorMap& maf, const CUtensorMap& mshf, const Params& p, int max_units, int num_sms,
                       cudaStream_t stream) {
    auto kern = gemm_tc2_kernel<EPI, PAIR>;
    int max_clusters = 0;
    cudaError_t e0 = per_device_value((const void*)kern, [&](int* v) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(2 * std::max(1, num_sms / 2));
        qc.blockDim = dim3(kThreads);
        qc.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        qc.attrs = qa;
        qc.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, (void*)kern, &qc);
        if (e != cudaSuccess || n < 1) return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        *v = n;
        return cudaSuccess;
    }, &max_clusters);
    if (e0 != cudaSuccess) return e0;
    const int clusters = std::max(1, std::min(max_clusters, max_units));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, msh, mb, mb2, maf, mshf, p);
}

}  // namespace p2
}  // namespace tc

bool gemm_tc2_supported(const GroupedGemm& g) {
    if (!g.tiles2 || !g.offsets || !gemm_tc_supported(g)) return false;
    if (g.b2) return g.N % 128 == 0;
    return g.N % 256 == 0;
}

cudaError_t launch_gemm_tc2(const GroupedGemm& g, int num_sms, cudaStream_t stream) {
    using namespace tc::p2;
    const bool sw = g.b2 != nullptr;
    const bool pair = g.Ka == 2 * g.Kb;
    Params p = {};
    p.G = g.G;
    p.shared_group = g.shared_group;
    p.offsets = g.offsets;
    p.tiles2 = g.tiles2;
    p.NB = sw ? g.N / 128 : g.N / 256;
    p.N = g.N;
    p.KB = g.Kb / BK;
    p.a_lo_x = g.Kb;
    p.ldo = g.ldo;
    p.out_pair = g.out_pair;
    p.out_f32 = g.out_elem == kF32;
    p.out_f16 = g.out_elem == kF16;
    p.in_f16 = g.elem == kF16;
    p.out = g.out;
    p.err = g.err;
    p.spin_ns = g.spin_ns > 0 ? g.spin_ns : 2000000000LL;
    CUtensorMap ma, msh, mb, mb2, maf, mshf;
    if (!tc::make_map(&ma, g.a, g.a_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
    if (!tc::make_map(&maf, g.a, g.a_rows, g.Ka, BM)) return cudaErrorInvalidValue;
    if (g.a_shared) {
        if (!tc::make_map(&msh, g.a_shared, g.a_shared_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mshf, g.a_shared, g.a_shared_rows, g.Ka, BM)) return cudaErrorInvalidValue;
    } else {
        msh = ma;
        mshf = maf;
    }
    if (!tc::make_map(&mb, g.b, (int64_t)g.G * g.N, g.Kb, 128)) return cudaErrorInvalidValue;
    if (sw) {
        if (!tc::make_map(&mb2, g.b2, (int64_t)g.G * g.N, g.Kb, 128)) return cudaErrorInvalidValue;
    } else {
        mb2 = mb;
    }
    const int max_units = g.max_tiles2 * p.NB;
    if (max_units <= 0) return cudaGetLastError();
    cudaError_t e;
    if (sw) e = launch_one<EPI_SWIGLU, false>(ma, msh, mb, mb2, maf, mshf, p, max_units, num_sms, stream);
    else if (pair) e = launch_one<EPI_PLAIN, true>(ma, msh, mb, mb2, maf, mshf, p, max_units, num_sms, stream);
    else e = launch_one<EPI_PLAIN, false>(ma, msh, mb, mb2, maf, mshf, p, max_units, num_sms, stream);
    count_launches(1);
    return e;
}

}  // namespace moe
