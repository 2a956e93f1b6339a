// Grouped bf16 / fp16 GEMM on CTA pairs: tcgen05.mma.cta_group::2, M = 256.
//
// Same computation and epilogues as gemm_tc.cu, for the prefill regime where
// groups hold hundreds of rows.  A single CTA's 128 x 256 tile reads its
// whole 32 KB B tile (and 16 KB of A) from shared memory for every 64-wide
// k-block while TMA writes the same 48 KB in.  Two CTAs of a cluster share one
// 256 x 256 tile instead: each loads its own 128 rows of A and half of the B
// tile (128 of the 256 weight rows), the pair's leader issues M=256 MMAs that
// read both CTAs' shared memory, and each CTA's TMEM receives its own 128
// rows x 256 columns: each SM moves about two thirds of the operand bytes per
// MMA cycle, and the ring holds 6 stages.  A whole 256-row pair unit runs
// ~11 % (gate/up) to ~29 % (down) faster per SM than two single-CTA tiles,
// but ragged pair tiles cost more than single-CTA tails, so on its own the
// kernel is no faster at T=8192 and runs on request; at prefill sizes it
// takes the whole 256-row pairs of the split expert GEMMs (with `active`:
// only that many pairs work, the rest leave at once) while the single-CTA
// kernel takes the remainders on another stream.
//   SwiGLU: CTA 0 holds the 128 gate rows, CTA 1 the 128 up rows of the same
//     features, so accumulator columns 0..127 are gate and 128..255 up in both.
//   Plain: CTA r holds weight rows nb*256 + r*128 .. +127.
// Pair tiles are 256 rows of one group, so a group's ragged last pair tile
// (fewer than 256 rows) would waste up to 255 rows of MMA.  Narrow tails
// (where enabled) run it transposed instead: the 256 weight rows are the
// MMA's M side (CTA r holds 128 of them) and the tile's rows its N side,
// rounded up to 32 (CTA r holds half of them), so the tensor pipe works in
// proportion to the rows that exist.  The epilogue then holds one feature
// per TMEM lane and one row per column:
//   SwiGLU: CTA r's weight rows are gate features 64r..64r+63 (lanes 0-63)
//     and the up rows of the same features (lanes 64-127); the up warps hand
//     their values to the gate warps through shared memory (bounded
//     mbarriers), which form h and store it.
//   Plain: CTA r's lanes are output features nb*256 + 128r + lane.
// Stores of 16-bit outputs go through a per-warp staging block in shared
// memory, so one warp instruction writes several whole 64-byte row segments
// instead of 32 scattered ones.
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
constexpr int kTabEntries = 1056;       // shared copies of the pair-tile prefix and row offsets (G <= 1025)
constexpr int kStRow = 80;              // staging row stride: 32 16-bit values (64 B) + 16 (conflict-free)
constexpr int kXRow = 33;               // exchange row stride in floats (32 + 1: conflict-free)
constexpr uint32_t kTabOff = kRing + 256;
constexpr uint32_t kStageOff = kTabOff + 2 * kTabEntries * 4;
constexpr uint32_t kXchgOff = kStageOff + 4 * 32 * kStRow;
constexpr uint32_t kSmemBytes = 1024 + kXchgOff + 2 * 32 * kXRow * 4;
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");

template <bool PAIR> struct Geo {
    static constexpr int kAStage = PAIR ? 2 * kABytes : kABytes;
    static constexpr int kStages = kRing / (kAStage + kBHalf);  // 6, or 4 with the hi/lo pair
};

enum Epi : int { EPI_SWIGLU = 0, EPI_PLAIN = 1 };

struct Params {
    int G, shared_group;
    int g_end;              // units cover the pair tiles of groups [0, g_end)
    const int32_t* offsets;
    const int32_t* tiles2;  // prefix of ceil(rows/256)
    int NB, N, KB, a_lo_x, ldo, out_pair, out_f32, out_f16, in_f16;
    int narrow;             // ragged pair tiles run transposed (16-bit outputs only)
    const int32_t* active;  // split GEMMs: [1] CTA pairs that take units (the rest leave at once), or nullptr
    void* out;
    uint32_t* err;
    int64_t spin_ns;
};

struct Unit {
    int g, m0pair, row0, nrows, nb;
    int nv;   // valid rows of the pair tile (<= 256)
    int nn;   // narrow tail: the MMA's N (nv rounded up to 32); 0 = a full-orientation unit
};

__device__ __forceinline__ Unit decode_unit(const Params& p, int u, const int32_t* s_t2, const int32_t* s_off) {
    Unit r;
    const int rt = u / p.NB;
    r.nb = u - rt * p.NB;
    r.g = find_group_smem(s_t2, p.G, rt);
    r.m0pair = (rt - s_t2[r.g]) * 2 * BM;
    r.row0 = s_off[r.g];
    r.nrows = s_off[r.g + 1] - r.row0;
    r.nv = min(2 * BM, r.nrows - r.m0pair);
    r.nn = (p.narrow && r.nv < 2 * BM) ? ((r.nv + 31) & ~31) : 0;
    return r;
}

__device__ __forceinline__ int boxes_for(int nrows, int m0) {
    const int valid = max(0, min(BM, nrows - m0));
    return (valid + kBoxRowsA - 1) / kBoxRowsA;
}

// Narrow unit: the token rows CTA `rank` supplies (half of nn, those that exist).
__device__ __forceinline__ int narrow_boxes(const Unit& un, int rank) {
    const int half = un.nn >> 1;
    const int cnt = max(0, min(half, un.nv - rank * half));
    return (cnt + kBoxRowsA - 1) / kBoxRowsA;
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

__device__ __forceinline__ uint32_t pack16(float a, float b, bool f16) {
    if (f16) {
        __half2 h = __floats2half2_rn(a, b);
        return *(uint32_t*)&h;
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(uint32_t*)&h;
}

// Row-major staging: this lane's row of 32 16-bit values (v) goes to row
// `lane` of the warp's staging block; then each lane stores 16 B of row
// 8 it + lane/4 (rows < nv only) to dst + row * ld (dst: the block's first
// row and column).
__device__ __forceinline__ void staged_rows32(uint8_t* st, const float* v, bool f16, int nv, uint16_t* dst, int64_t ld) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *(uint4*)(st + lane * kStRow + 16 * q) =
            make_uint4(pack16(v[8 * q], v[8 * q + 1], f16), pack16(v[8 * q + 2], v[8 * q + 3], f16),
                       pack16(v[8 * q + 4], v[8 * q + 5], f16), pack16(v[8 * q + 6], v[8 * q + 7], f16));
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = 8 * it + (lane >> 2), ch = lane & 3;
        const uint4 pk = *(const uint4*)(st + rr * kStRow + 16 * ch);
        if (rr < nv) *(uint4*)(dst + rr * ld + 8 * ch) = pk;
    }
    __syncwarp();
}

// Transposed staging: this lane holds one feature (column `lane` of the
// block) for 32 rows (v[j] = row j); the block is written row-major and
// stored as in staged_rows32.
__device__ __forceinline__ void staged_cols32(uint8_t* st, const float* v, bool f16, int nv, uint16_t* dst, int64_t ld) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        uint16_t b;
        if (f16) {
            __half h = __float2half_rn(v[j]);
            b = *(uint16_t*)&h;
        } else {
            __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
            b = *(uint16_t*)&h;
        }
        *(uint16_t*)(st + j * kStRow + 2 * lane) = b;
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = 8 * it + (lane >> 2), ch = lane & 3;
        const uint4 pk = *(const uint4*)(st + rr * kStRow + 16 * ch);
        if (rr < nv) *(uint4*)(dst + rr * ld + 8 * ch) = pk;
    }
    __syncwarp();
}

template <int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a_sh,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_b2,
                    const __grid_constant__ CUtensorMap tm_af, const __grid_constant__ CUtensorMap tm_a_shf,
                    const __grid_constant__ CUtensorMap tm_bh, const __grid_constant__ CUtensorMap tm_b2h,
                    const Params p) {
    constexpr int kStages = Geo<PAIR>::kStages;
    constexpr int kAStage = Geo<PAIR>::kAStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kAStage;
    uint64_t* bars = (uint64_t*)(smem + kRing);
    // barriers: stage full/empty [kStages each], TMEM full/empty [2 each],
    // drain, narrow-SwiGLU exchange full/empty [2 each]; then the TMEM
    // address and the abort flag
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kStages), tempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
    const uint32_t xfull0 = smem_u32(bars + 2 * kStages + 5), xempty0 = smem_u32(bars + 2 * kStages + 7);
    uint32_t* tmem_slot = (uint32_t*)(bars + 2 * kStages + 9);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    static_assert((2 * 6 + 9) * 8 + 8 <= 256, "barrier block overflows");
    int32_t* s_t2 = (int32_t*)(smem + kTabOff);
    int32_t* s_off = s_t2 + kTabEntries;
    uint8_t* s_stage = smem + kStageOff;        // [4 epilogue warps][32 rows][kStRow]
    float* s_xchg = (float*)(smem + kXchgOff);  // [2 warp pairs][32 lanes][kXRow]
    pdl_wait_then_release();
    // split GEMMs: only the first `npairs` CTA pairs take units; the others
    // leave before touching a barrier, TMEM or the peer, and free their SMs
    const int npairs = p.active ? min(__ldg(p.active), (int)(gridDim.x >> 1)) : (int)(gridDim.x >> 1);
    if ((int)(blockIdx.x >> 1) >= npairs) return;
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
        s_t2[i] = __ldg(p.tiles2 + i);
        s_off[i] = __ldg(p.offsets + i);
    }

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
            mbar_init(xfull0 + 8 * b, 1);
            mbar_init(xempty0 + 8 * b, 1);
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

    const int nclusters = npairs, cid = blockIdx.x >> 1;
    const int total_units = s_t2[p.g_end] * p.NB;
    const int64_t lim = p.spin_ns;
    bool aborted = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            for (int u = cid; u < total_units; u += nclusters) {
                const Unit un = decode_unit(p, u, s_t2, s_off);
                const bool sh = un.g == p.shared_group;
                const CUtensorMap* ta = sh ? &tm_a_sh : &tm_a;
                const CUtensorMap* taf = sh ? &tm_a_shf : &tm_af;
                const int base_y = sh ? 0 : un.row0;  // A row of the group's row 0
                int nbox, a_y;
                uint32_t pair_bytes;
                if (un.nn) {  // narrow: this CTA's half of the tile's rows, 16-row boxes
                    nbox = narrow_boxes(un, (int)rank);
                    a_y = base_y + un.m0pair + (int)rank * (un.nn >> 1);
                    pair_bytes = (uint32_t)(narrow_boxes(un, 0) + narrow_boxes(un, 1)) * kBoxRowsA * BK * 2 + 2u * kBHalf;
                } else {
                    const int m0 = un.m0pair + (int)rank * BM;
                    nbox = boxes_for(un.nrows, m0);
                    a_y = base_y + m0;
                    pair_bytes = (PAIR ? 2u : 1u) *
                                     (uint32_t)(boxes_for(un.nrows, un.m0pair) + boxes_for(un.nrows, un.m0pair + BM)) *
                                     kBoxRowsA * BK * 2 +
                                 2u * kBHalf;
                }
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 21, blockIdx.x, u);
                        raise_abort_pair(abort_flag, rank);
                        aborted = true;
                        break;
                    }
                    const uint32_t fb_local = full0 + 8 * stage;
                    const uint32_t fb = mapa_shared(fb_local, 0);  // the leader's full barrier
                    if (leader) mbar_expect_tx(fb_local, pair_bytes);
                    const uint32_t a_dst = smem_u32(sA + stage * kAStage);
                    const uint32_t b_dst = smem_u32(sB + stage * kBHalf);
                    if (!un.nn && nbox * kBoxRowsA == BM) {  // full half-tile: one 128-row box
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
                    if (EPI == EPI_SWIGLU && un.nn) {
                        // narrow SwiGLU: gate then up rows of features nb*128 + 64 rank .. +63
                        const int wy = un.g * p.N + un.nb * 128 + 64 * (int)rank;
                        tma_load_2d_pair(b_dst, &tm_bh, fb, kb * BK, wy);
                        tma_load_2d_pair(b_dst + 64 * 128, &tm_b2h, fb, kb * BK, wy);
                    } else {
                        const CUtensorMap* tb = (EPI == EPI_SWIGLU && rank == 1) ? &tm_b2 : &tm_b;
                        const int b_y =
                            un.g * p.N + ((EPI == EPI_SWIGLU) ? un.nb * 128 : un.nb * 256 + (int)rank * 128);
                        tma_load_2d_pair(b_dst, tb, fb, kb * BK, b_y);
                    }
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
            for (int u = cid; u < total_units && !aborted; u += nclusters) {
                const Unit un = decode_unit(p, u, s_t2, s_off);
                const int n = un.nn ? un.nn : 256;
                const uint32_t idesc = p.in_f16 ? idesc_f16(2 * BM, n) : idesc_bf16(2 * BM, n);
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 22, blockIdx.x, u);
                    raise_abort_pair(abort_flag, rank);
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 23, blockIdx.x, u);
                        raise_abort_pair(abort_flag, rank);
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_desc(smem_u32(sA + stage * kAStage));
                    const uint64_t bd = umma_desc(smem_u32(sB + stage * kBHalf));
                    if (un.nn) {
                        // transposed: weights (sB) as the M side, the tile's rows (sA) as N
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_pair(d, bd + (uint64_t)(kk * 2), ad + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                        if (PAIR) {
                            const uint64_t al = umma_desc(smem_u32(sA + stage * kAStage + kABytes));
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                umma_bf16_pair(d, al + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, 1u);
                        }
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
        uint8_t* st = s_stage + (size_t)sub * 32 * kStRow;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t xphase = 0;  // narrow SwiGLU: exchanges so far (the same count in both warps of a pair)
        const int xp = sub & 1;  // exchange pair: quarters 0 and 2, 1 and 3
        for (int u = cid; u < total_units && !aborted; u += nclusters) {
            const Unit un = decode_unit(p, u, s_t2, s_off);
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(tfull0 + 8 * acc, acc_phase, lim, abort_flag);
                if (!ok) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 24, blockIdx.x, u);
                    raise_abort_pair(abort_flag, rank);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kAccCols);
            if (un.nn) {
                // ---------------- narrow tail: lane = feature, column = row of the tile
                const int64_t orow0 = (int64_t)un.row0 + un.m0pair;
                float mx = 0.f;
#pragma unroll 1
                for (int c = 0; c < un.nv && !aborted; c += 32) {
                    const int nvc = min(32, un.nv - c);
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (EPI == EPI_SWIGLU) {
                        float* xb = s_xchg + xp * 32 * kXRow;
                        if (sub >= 2) {  // up values: hand them to the gate warp of the same features
                            int w_ok = 1;
                            if (lane == 0) w_ok = mbar_wait(xempty0 + 8 * xp, (xphase & 1) ^ 1, lim, abort_flag);
                            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                            if (!w_ok) {
                                if (lane == 0) {
                                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 25, blockIdx.x, u);
                                    raise_abort_pair(abort_flag, rank);
                                }
                                aborted = true;
                                break;
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j) xb[lane * kXRow + j] = v[j];
                            __syncwarp();
                            if (lane == 0) mbar_arrive(xfull0 + 8 * xp);
                        } else {  // gate values: wait for the up values, form h, store it
                            int w_ok = 1;
                            if (lane == 0) w_ok = mbar_wait(xfull0 + 8 * xp, xphase & 1, lim, abort_flag);
                            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                            if (!w_ok) {
                                if (lane == 0) {
                                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 26, blockIdx.x, u);
                                    raise_abort_pair(abort_flag, rank);
                                }
                                aborted = true;
                                break;
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                v[j] = swiglu(v[j], xb[lane * kXRow + j]);
                                if (j < nvc) mx = fmaxf(mx, fabsf(v[j]));
                            }
                            __syncwarp();
                            if (lane == 0) mbar_arrive(xempty0 + 8 * xp);
                            // features nb*128 + 64 rank + 32 sub + lane, rows c..c+31
                            uint16_t* dst = (uint16_t*)p.out + (orow0 + c) * p.ldo + un.nb * 128 + 64 * (int)rank + 32 * sub;
                            staged_cols32(st, v, p.out_f16, nvc, dst, p.ldo);
                        }
                        ++xphase;
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nvc) mx = fmaxf(mx, fabsf(v[j]));
                        // features nb*256 + 128 rank + 32 sub + lane, rows c..c+31
                        uint16_t* dst = (uint16_t*)p.out + (orow0 + c) * p.ldo + un.nb * 256 + 128 * (int)rank + 32 * sub;
                        staged_cols32(st, v, p.out_f16, nvc, dst, p.ldo);
                    }
                }
                if (p.out_f16 && !(mx <= 65504.f))
                    record_error(p.err, MOE_ERR_NONFINITE, EPI == EPI_SWIGLU ? 5 : 6, blockIdx.x, 0);
                if (aborted) break;
            } else {
                const int m = un.m0pair + (int)rank * BM + row;
                const bool valid = m < un.nrows;
                const int64_t orow = (int64_t)un.row0 + m;
                const int nvw = min(32, max(0, un.nrows - (un.m0pair + (int)rank * BM + sub * 32)));  // warp's rows
                const int64_t orow_w = (int64_t)un.row0 + un.m0pair + (int)rank * BM + sub * 32;
                if (EPI == EPI_SWIGLU) {
                    bf16* o = (bf16*)p.out + orow * p.ldo + un.nb * 128;
#pragma unroll 1
                    for (int c = 0; c < 128; c += 32) {
                        uint32_t gr[32], ur[32];
                        tmem_ld32(tb + c, gr);
                        tmem_ld32(tb + 128 + c, ur);
                        tmem_wait_ld();
                        float h[32], lo[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) h[i] = swiglu(__uint_as_float(gr[i]), __uint_as_float(ur[i]));
                        if (!p.out_pair) {
                            if (p.out_f16) {
                                float mx = 0.f;
#pragma unroll
                                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(h[i]));
                                if (valid && !(mx <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 5, blockIdx.x, 0);
                            }
                            staged_rows32(st, h, p.out_f16, nvw, (uint16_t*)p.out + orow_w * p.ldo + un.nb * 128 + c,
                                          p.ldo);
                        } else if (valid) {
                            store_bf16x32(o + c, h);
#pragma unroll
                            for (int i = 0; i < 32; ++i) lo[i] = h[i] - __bfloat162float(__float2bfloat16_rn(h[i]));
                            store_bf16x32(o + p.N + c, lo);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < 256; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(tb + c, r);
                        tmem_wait_ld();
                        const int n0 = un.nb * 256 + c;
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        if (p.out_f32) {
                            if (valid) {
                                float* o = (float*)p.out + orow * p.ldo + n0;
#pragma unroll
                                for (int i = 0; i < 32; i += 4) *(float4*)(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                            }
                        } else {
                            if (p.out_f16) {
                                float mx = 0.f;
#pragma unroll
                                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
                                if (valid && !(mx <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 6, blockIdx.x, 0);
                            }
                            staged_rows32(st, v, p.out_f16, nvw, (uint16_t*)p.out + orow_w * p.ldo + n0, p.ldo);
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
                       const CUtensorMap& maf, const CUtensorMap& mshf, const CUtensorMap& mbh, const CUtensorMap& mb2h,
                       const Params& p, int max_units, int max_ctas, int num_sms, cudaStream_t stream) {
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
    int clusters = std::max(1, std::min(max_clusters, max_units));
    if (max_ctas > 0) clusters = std::max(1, std::min(clusters, max_ctas / 2));
    return launch_kernel(kern, dim3(2 * clusters), dim3(kThreads), kSmemBytes, stream, 2, ma, msh, mb, mb2, maf, mshf,
                         mbh, mb2h, p);
}

}  // namespace p2
}  // namespace tc

bool gemm_tc2_supported(const GroupedGemm& g) {
    using namespace tc::p2;
    if (!g.tiles2 || !g.offsets || g.cmb_out || !gemm_tc_supported(g)) return false;
    if (g.G + 1 > kTabEntries) return false;
    if (g.b2) return g.N % 128 == 0;
    return g.N % 256 == 0;
}

cudaError_t launch_gemm_tc2(const GroupedGemm& g, int num_sms, cudaStream_t stream) {
    using namespace tc::p2;
    const bool sw = g.b2 != nullptr;
    const bool pair = g.Ka == 2 * g.Kb;
    Params p = {};
    p.G = g.G;
    p.g_end = (g.g_end > 0 && g.g_end < g.G) ? g.g_end : g.G;
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
    // narrow tails: 16-bit outputs only (the transposed stores), not the hi/lo pair input
    p.narrow = g.narrow && !pair && !g.out_pair && g.out_elem != kF32;
    p.active = g.pair_active;
    p.out = g.out;
    p.err = g.err;
    p.spin_ns = g.spin_ns > 0 ? g.spin_ns : 2000000000LL;
    CUtensorMap ma, msh, mb, mb2, maf, mshf, mbh, mb2h;
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
        if (!tc::make_map(&mbh, g.b, (int64_t)g.G * g.N, g.Kb, 64)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mb2h, g.b2, (int64_t)g.G * g.N, g.Kb, 64)) return cudaErrorInvalidValue;
    } else {
        mb2 = mb;
        mbh = mb;
        mb2h = mb;
    }
    const int max_units = g.max_tiles2 * p.NB;
    if (max_units <= 0) return cudaGetLastError();
    cudaError_t e;
    if (sw) e = launch_one<EPI_SWIGLU, false>(ma, msh, mb, mb2, maf, mshf, mbh, mb2h, p, max_units, g.max_ctas, num_sms, stream);
    else if (pair) e = launch_one<EPI_PLAIN, true>(ma, msh, mb, mb2, maf, mshf, mbh, mb2h, p, max_units, g.max_ctas, num_sms, stream);
    else e = launch_one<EPI_PLAIN, false>(ma, msh, mb, mb2, maf, mshf, mbh, mb2h, p, max_units, g.max_ctas, num_sms, stream);
    count_launches(1);
    return e;
}

}  // namespace moe
