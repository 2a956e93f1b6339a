// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMA + TMEM).
//
// The expert FFNs of the routed-MoE layer are "Grouped GEMMs" in the sense of
// "Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU" (English page,
// intro and "Pallas Kernels, SparseCore Co-Design, and the Roofline"): one
// GEMM per expert over that expert's rows of the grouped layout.  Here one
// persistent kernel walks all of them.
//
// Work unit: 128 rows of one group (M, the TMEM lanes) x one block of output
// features (N <= 256, the TMEM columns).  Units are numbered row-tile major,
// feature block minor, so the CTAs that run at the same time share a row tile
// (A read once) and the row tiles of a group run back to back (its weight
// block is reused from L2).  The row tiles come from the device-built prefix
// of ceil(rows/128) per group (copied to shared memory); no host round trip.
// A CTA takes its units either in the static round-robin order or, given a
// counter, from a launch-wide atomic (so that CTAs which start late, behind a
// kernel on another stream, take fewer); the producer draws them and hands
// them to the other roles through a 4-slot ring in shared memory.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: A rows (one 128-row box for a full tile, else
//               16-row boxes, only those that hold valid rows) and the B
//               weight tile into a ring of 4-8 stages (as many as fit);
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M=128, N=BN, K=16, fp32 accumulation in TMEM;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (two TMEM buffers,
//               so the epilogue of one unit overlaps the MMAs of the next),
//               SwiGLU / bias / conversion, stores.
// Tile pairs (prefill): the CTAs run as 2-CTA clusters whose two CTAs share
// one operand tile through TMA multicast, so each SM pulls fewer operand
// bytes from L2 per MMA.  A cluster unit is either two row tiles of one
// group against one weight block (each CTA copies half of the 256-row B tile
// into both CTAs: 16 KB of A + 16 KB of B per CTA and stage instead of
// 16 + 32) or, for a group's odd last row tile, that tile against two weight
// blocks (each CTA copies half of the A rows into both: 8 + 32).  Row tiles
// stay 128 rows, so no padding is added.  Each CTA's stage is written by both
// CTAs, so both MMA issuers' commits release it (commit multicast), and the
// cluster synchronises before it exits.
// Narrow tails (where enabled): a unit whose tile holds at most 112 valid
// rows (a group's ragged last tile; every tile at decode sizes) is
// multiplied transposed: the weight rows are the MMA's M = 128 side (one MMA
// per 128 features) and the tile's rows its N side, rounded up to 16, so the
// tensor pipe spends time in proportion to the rows that exist instead of on
// 128.  The stage holds the same operands either way; the epilogue then
// reads a feature per TMEM lane and a row per column.
// Operands are K-major with the 128-byte swizzle on both sides (TMA writes
// it, the UMMA descriptor reads it).  Every mbarrier wait is bounded by
// spin_ns; on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT, drains its
// own copies and MMAs (again bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                   // rows per unit (TMEM lanes)
constexpr int BK = 64;                    // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kABytes = BM * BK * 2;      // 16 KB: one A tile
constexpr int kBBytesMax = 256 * BK * 2;  // 32 KB
constexpr int kThreads = 192;
constexpr int kAccCols = 256;             // TMEM columns per accumulator buffer
constexpr int kNarrowMax = 112;           // narrow-tail units: at most this many valid rows
constexpr int kBoxRowsA = 16;             // a ragged tile's A rows come in 16-row boxes (2 KB);
                                          // a full tile's in one 128-row box: the single
                                          // producer thread issues few TMA instructions
// Shared-memory copy of the group row-tile prefix and row offsets (G <= 1025
// groups), and for the split GEMMs' single-CTA launch the order it takes the
// groups in: a unit's group comes from a binary search that never leaves the SM.
constexpr int kTabEntries = 1056;
// Plain epilogue, 16-bit output: each epilogue warp stages 32 rows x 64
// columns (128 B per row, rows 144 B apart: conflict-free) in shared memory
// and stores them 4 rows x 128 B per warp instruction; from the row-per-lane
// layout every store touched 32 rows, and the down GEMM's 8 KB of y per row
// (0.74 ms at T=8192, 0.62 ms with the stores left out) waited on them.
constexpr int kStageRow = 144;
constexpr uint32_t kStagingBytes = 4 * 32 * kStageRow;
constexpr uint32_t kSmemBytes = 1024 + 196608 + 256 + 3 * kTabEntries * 4 + kStagingBytes;
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");

// Stage geometry.  PAIR: A is a bf16 hi/lo pair (hi in columns [0, Kb), lo in
// [Kb, 2Kb)); a stage holds the hi and lo tiles of one k-block next to one B
// tile, so the weights stream once and both halves multiply the same tile.
// The ring holds as many stages of A + B as fit in kRingBytes (at most
// kMaxStages): 4 for 256-wide B tiles, 6 for 128-wide, 8 for narrower.
constexpr int kRingBytes = 196608;
constexpr int kMaxStages = 8;
template <bool PAIR> struct Geo {
    static constexpr int kAStage = PAIR ? 2 * kABytes : kABytes;
    static_assert(3 * (kAStage + kBBytesMax) <= kRingBytes, "stage ring exceeds the smem budget");
};

enum Epi : int { EPI_SWIGLU = 0, EPI_PLAIN = 1 };

struct Params {
    int G, shared_group;
    int g_end;           // units cover the row tiles of groups [0, g_end)
    int* sched;          // [2] device: next-unit counter and finished-CTA count, or nullptr (static order)
    const int32_t* offsets;
    const int32_t* tiles;
    int rows;            // single-group row count (offsets == nullptr)
    int NB;              // feature blocks per row tile
    int BN;              // MMA N (SwiGLU: 128 gate + 128 up)
    int N;               // output features of a group
    int KB;              // k-blocks of B (Kb / 64); one stage per k-block
    int KS;              // K slices (single group only): slice s walks k-blocks [s*KB/KS, (s+1)*KB/KS)
    int64_t split_stride;  // elements between the outputs of two K slices
    int a_lo_x;          // PAIR: column where A's lo half starts (= Kb)
    int b_group_rows;    // rows of B per group
    int ldo;
    int out_pair;
    int out_f32;
    int out_f16;         // SwiGLU output as fp16 (single rounding) instead of bf16
    int in_f16;          // A and B are fp16 (else bf16)
    int narrow;          // units of <= kNarrowMax valid rows run transposed (narrow tails)
    int rem_only;        // split GEMMs: only the rows after each group's whole 256-row pairs
    const int32_t* order;  // split GEMMs: [G] group at each position of `tiles` (nullptr: position = group)
    int stages;          // ring depth (<= kMaxStages)
    int b_stage;         // bytes of one B stage
    void* out;
    const float* bias;
    uint32_t* err;
    int64_t spin_ns;
    // fused unpermutation (see GroupedGemm::cmb_out); cmb_out == nullptr: off
    void* cmb_out;
    int cmb_out_f32;
    const int32_t* cmb_blob;
    const int32_t* cmb_inv;
    const void* cmb_y;
    int cmb_k;
};

// ------------------------------------------------------------ unit decode

struct Unit {
    int g, m0, row0, nrows, nb, ks;
};

// Units: K slice major, then row tile, then feature block.  s_tiles/s_off/
// s_ord: shared copies of p.tiles and p.offsets (entries 0..G) and p.order.
__device__ __forceinline__ Unit decode_unit(const Params& p, int u, int total_tiles, const int32_t* s_tiles,
                                            const int32_t* s_off, const int32_t* s_ord) {
    Unit r;
    const int per_slice = total_tiles * p.NB;
    r.ks = u / per_slice;
    u -= r.ks * per_slice;
    const int rt = u / p.NB;
    r.nb = u - rt * p.NB;
    if (p.offsets) {
        const int pos = find_group_smem(s_tiles, p.G, rt);
        r.g = p.order ? min(max(s_ord[pos], 0), p.G - 1) : pos;  // clamped against a stale table
        r.m0 = (rt - s_tiles[pos]) * BM;
        r.row0 = s_off[r.g];
        r.nrows = s_off[r.g + 1] - r.row0;
        if (p.rem_only) r.m0 += 2 * BM * (r.nrows / (2 * BM));  // past the group's whole pairs
    } else {
        r.g = 0;
        r.m0 = rt * BM;
        r.row0 = 0;
        r.nrows = p.rows;
    }
    return r;
}

// Tile pairs: cluster unit v, seen from the CTA of rank `rank`.  A group of
// t row tiles has t * NB / 2 cluster units: first (t / 2) * NB "B-shared"
// ones (row tiles 2q + rank against weight block nb), then, when t is odd,
// NB / 2 "A-shared" ones (the last row tile against block 2w + rank).  So
// the units of groups [0, g) number NB / 2 * tiles[g], and the row-tile
// prefix finds a unit's group.
__device__ __forceinline__ Unit decode_cunit(const Params& p, int v, int rank, int total_tiles,
                                             const int32_t* s_tiles, const int32_t* s_off, int& a_shared) {
    Unit r;
    r.ks = 0;
    const int H = p.NB >> 1;
    const int q = v / H;
    int t0, t;
    if (p.offsets) {
        r.g = find_group_smem(s_tiles, p.G, q);
        t0 = s_tiles[r.g];
        t = s_tiles[r.g + 1] - t0;
        r.row0 = s_off[r.g];
        r.nrows = s_off[r.g + 1] - r.row0;
    } else {
        r.g = 0;
        t0 = 0;
        t = total_tiles;
        r.row0 = 0;
        r.nrows = p.rows;
    }
    const int w = v - H * t0;
    const int b_units = (t >> 1) * p.NB;
    if (w < b_units) {
        a_shared = 0;
        const int q2 = w / p.NB;
        r.nb = w - q2 * p.NB;
        r.m0 = (2 * q2 + rank) * BM;
    } else {
        a_shared = 1;
        r.nb = 2 * (w - b_units) + rank;
        r.m0 = (t - 1) * BM;
    }
    return r;
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

// ------------------------------------------------------------------ kernel

// CL: tile pairs on 2-CTA clusters (tm_ah / tm_a_shh: 64-row A boxes; for
// the plain epilogue tm_b2 then holds 128-row boxes of B).
template <int EPI, bool PAIR, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a_sh,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_b2,
                   const __grid_constant__ CUtensorMap tm_af, const __grid_constant__ CUtensorMap tm_a_shf,
                   const __grid_constant__ CUtensorMap tm_ah, const __grid_constant__ CUtensorMap tm_a_shh,
                   const Params p) {
    static_assert(!(CL && PAIR), "tile pairs take a single A input");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int kStages = p.stages;
    const int kBStage = p.b_stage;
    constexpr int kAStage = Geo<PAIR>::kAStage;
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kAStage;
    uint64_t* bars = (uint64_t*)(smem + kRingBytes);
    int32_t* s_tiles = (int32_t*)(smem + kRingBytes + 256);
    int32_t* s_off = s_tiles + kTabEntries;
    int32_t* s_ord = s_off + kTabEntries;
    uint8_t* s_stage = (uint8_t*)(s_ord + kTabEntries);  // [4 epilogue warps][32 rows][kStageRow]
    pdl_wait_then_release();
    if (p.offsets)
        for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
            s_tiles[i] = __ldg(p.tiles + i);
            s_off[i] = __ldg(p.offsets + i);
            if (p.order && i < p.G) s_ord[i] = __ldg(p.order + i);
        }
    // barrier block (256 bytes): stage full/empty [kMaxStages each], TMEM
    // full/empty [2 each], drain, unit-ring full/empty [4 each], then the
    // TMEM address, the abort flag and the 4-slot unit ring
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kMaxStages), tempty0 = smem_u32(bars + 2 * kMaxStages + 2);
    const uint32_t drain = smem_u32(bars + 2 * kMaxStages + 4);
    const uint32_t ufull0 = smem_u32(bars + 2 * kMaxStages + 5), uempty0 = smem_u32(bars + 2 * kMaxStages + 9);
    uint32_t* tmem_slot = (uint32_t*)(bars + 2 * kMaxStages + 13);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    volatile int* s_units = (volatile int*)(tmem_slot + 2);
    static_assert((2 * kMaxStages + 13) * 8 + 6 * 4 <= 256, "barrier block overflows");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = CL ? (int)cluster_rank() : 0;
    // a timed-out wait stops this CTA's roles, and under tile pairs the peer's
    auto abort_cta = [&](volatile int* f) {
        if (CL) raise_abort_pair(f, (uint32_t)rank);
        else *f = 1;
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, CL ? 2 : 1);  // tile pairs: both CTAs' MMAs read what fills it
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 4);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(ufull0 + 8 * i, 1);
            mbar_init(uempty0 + 8 * i, 1 + 4);  // the MMA issuer and the 4 epilogue warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(2 * kAccCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (CL) cluster_sync();  // the peer's barriers exist before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int total_tiles = p.offsets ? __ldg(p.tiles + p.g_end) : (p.rows + BM - 1) / BM;
    const int total_units = CL ? total_tiles * (p.NB >> 1) : total_tiles * p.NB * p.KS;
    const int kbs = p.KB / p.KS;  // k-blocks per unit
    const int64_t lim = p.spin_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            const uint32_t b_bytes = (EPI == EPI_SWIGLU) ? 2u * 128 * BK * 2 : (uint32_t)p.BN * BK * 2;
            bool ok = true;
            // units come from the launch-wide counter (CTAs that start late
            // take fewer units) or in the static round-robin order; each is
            // published to the MMA issuer and the epilogue through the unit
            // ring.  The counter is drawn one unit ahead to hide its latency.
            // (tile pairs: both CTAs of a cluster walk the same static order)
            const int ord0 = CL ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
            const int ordn = CL ? (int)(gridDim.x >> 1) : (int)gridDim.x;
            int next_u = p.sched ? atomicAdd(p.sched, 1) : ord0;
            for (int i = 0; ok; ++i) {
                int u = next_u;
                if (u >= total_units) u = -1;
                if (u >= 0) next_u = p.sched ? atomicAdd(p.sched, 1) : ord0 + (i + 1) * ordn;
                if (!mbar_wait(uempty0 + 8 * (i & 3), ((i >> 2) & 1) ^ 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 5, blockIdx.x, i);
                    abort_cta(abort_flag);
                    ok = false;
                    break;
                }
                s_units[i & 3] = u;
                mbar_arrive(ufull0 + 8 * (i & 3));
                if (u < 0) break;
                int a_sh = 0;
                const Unit un = CL ? decode_cunit(p, u, rank, total_tiles, s_tiles, s_off, a_sh)
                                   : decode_unit(p, u, total_tiles, s_tiles, s_off, s_ord);
                const bool sh = un.g == p.shared_group;
                const CUtensorMap* ta = sh ? &tm_a_sh : &tm_a;
                const CUtensorMap* taf = sh ? &tm_a_shf : &tm_af;
                const CUtensorMap* tah = sh ? &tm_a_shh : &tm_ah;
                const int a_y = sh ? un.m0 : un.row0 + un.m0;
                const int valid = min(BM, un.nrows - un.m0);
                const int nbox = (valid + kBoxRowsA - 1) / kBoxRowsA;
                // A-shared pair unit: this CTA copies rows [64 rank, 64 rank + 64) of
                // the tile into both CTAs.  Either way the stage receives the
                // tile's valid rows in 16-row units plus the whole B tile.
                const int hv = max(0, min(BM / 2, valid - (BM / 2) * rank));
                const int hbox = (hv + kBoxRowsA - 1) / kBoxRowsA;
                const uint32_t bytes = (PAIR ? 2u : 1u) * (uint32_t)nbox * kBoxRowsA * BK * 2 + b_bytes;
                const int b_y = un.g * p.b_group_rows + un.nb * ((EPI == EPI_SWIGLU) ? 128 : p.BN);
                for (int kb = un.ks * kbs; kb < (un.ks + 1) * kbs; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 1, blockIdx.x, u);
                        abort_cta(abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, bytes);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    const uint32_t a_dst = smem_u32(sA + stage * kAStage);
                    const uint32_t b_dst = smem_u32(sB + stage * kBStage);
                    if (CL && a_sh) {
                        const uint32_t h_dst = a_dst + (uint32_t)rank * (kABytes / 2);
                        const int h_y = a_y + (BM / 2) * rank;
                        if (hv == BM / 2) {
                            tma_load_2d_mc(h_dst, tah, fb, kb * BK, h_y, 3);
                        } else {
                            for (int i = 0; i < hbox; ++i)
                                tma_load_2d_mc(h_dst + i * kBoxRowsA * 128, ta, fb, kb * BK, h_y + i * kBoxRowsA, 3);
                        }
                    } else if (nbox * kBoxRowsA == BM) {  // (nearly) full tile: one 128-row box
                        tma_load_2d(a_dst, taf, fb, kb * BK, a_y);
                        if (PAIR) tma_load_2d(a_dst + kABytes, taf, fb, p.a_lo_x + kb * BK, a_y);
                    } else {
                        for (int i = 0; i < nbox; ++i) {
                            tma_load_2d(a_dst + i * kBoxRowsA * 128, ta, fb, kb * BK, a_y + i * kBoxRowsA);
                            if (PAIR)
                                tma_load_2d(a_dst + kABytes + i * kBoxRowsA * 128, ta, fb, p.a_lo_x + kb * BK,
                                            a_y + i * kBoxRowsA);
                        }
                    }
                    const int bx = kb * BK;
                    if (CL && !a_sh) {  // B-shared pair unit: this CTA copies half of the B tile into both
                        if (EPI == EPI_SWIGLU)
                            tma_load_2d_mc(b_dst + (uint32_t)rank * (128 * 128), rank ? &tm_b2 : &tm_b, fb, bx, b_y, 3);
                        else
                            tma_load_2d_mc(b_dst + (uint32_t)rank * (128 * 128), &tm_b2, fb, bx, b_y + 128 * rank, 3);
                    } else {
                        tma_load_2d(b_dst, &tm_b, fb, bx, b_y);
                        if (EPI == EPI_SWIGLU) tma_load_2d(b_dst + 128 * 128, &tm_b2, fb, bx, b_y);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {  // let every copy this thread started land before the CTA exits
                if (CL) {
                    // (a tile-pair stage also waits for the peer's half, which an
                    // aborted peer may never send: give this CTA's own copies,
                    // here and in the peer, time to land instead)
                    sleep_ns(200000);
                } else {
                    for (int s = 0; s < kStages; ++s)
                        if (armed & (1u << s)) {
                            volatile int never = 0;
                            mbar_wait(full0 + 8 * s, (armed_parity >> s) & 1u, 1000000000LL, &never);
                        }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t idesc = p.in_f16 ? idesc_f16(BM, p.BN) : idesc_bf16(BM, p.BN);
            bool ok = true;
            for (int i = 0; ok; ++i) {
                if (!mbar_wait(ufull0 + 8 * (i & 3), (i >> 2) & 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 6, blockIdx.x, i);
                    abort_cta(abort_flag);
                    break;
                }
                const int u = s_units[i & 3];
                mbar_arrive(uempty0 + 8 * (i & 3));
                if (u < 0) break;
                int nn = 0;  // narrow tail: N of the transposed MMAs (valid rows rounded up to 16), else 0
                if (p.narrow) {
                    int a_sh = 0;
                    const Unit un = CL ? decode_cunit(p, u, rank, total_tiles, s_tiles, s_off, a_sh)
                                       : decode_unit(p, u, total_tiles, s_tiles, s_off, s_ord);
                    const int valid = min(BM, un.nrows - un.m0);
                    if (valid <= kNarrowMax) nn = (valid + 15) & ~15;
                }
                const int n_t = nn > 0 ? nn : 16;
                const uint32_t idesc_n = p.in_f16 ? idesc_f16(BM, n_t) : idesc_bf16(BM, n_t);
                const int regions = (EPI == EPI_SWIGLU) ? 2 : p.BN / 128;
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 2, blockIdx.x, u);
                    abort_cta(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 3, blockIdx.x, u);
                        abort_cta(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_desc(smem_u32(sA + stage * kAStage));
                    const uint64_t bd = umma_desc(smem_u32(sB + stage * kBStage));
                    if (nn > 0) {
                        // transposed: weight rows [128 r, 128 r + 128) of the B tile as M, the
                        // tile's rows as N; region r accumulates at TMEM columns [128 r, ...)
                        for (int r = 0; r < regions; ++r) {
                            const uint64_t wd = umma_desc(smem_u32(sB + stage * kBStage + r * kABytes));
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                umma_bf16(d + (uint32_t)(r * 128), wd + (uint64_t)(kk * 2), ad + (uint64_t)(kk * 2),
                                          idesc_n, (kb | kk) != 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)  // K=16 per MMA: 32 bytes along the swizzled row
                            umma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                    }
                    if (PAIR) {
                        const uint64_t al = umma_desc(smem_u32(sA + stage * kAStage + kABytes));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16(d, al + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, 1u);
                    }
                    if (CL) umma_commit_mc(empty0 + 8 * stage, 3);  // the stage was filled by both CTAs
                    else umma_commit(empty0 + 8 * stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(tfull0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // every MMA this thread issued completes before TMEM is freed
            umma_commit(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, 1000000000LL, &never);
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int sub = warp & 3;  // TMEM lane quarter this warp may access
        const int row = sub * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int i = 0;; ++i) {
            int u = -1, got = 1;
            if (lane == 0) {
                got = mbar_wait(ufull0 + 8 * (i & 3), (i >> 2) & 1, lim, abort_flag);
                if (got) {
                    u = s_units[i & 3];
                    mbar_arrive(uempty0 + 8 * (i & 3));
                } else {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 7, blockIdx.x, i);
                    abort_cta(abort_flag);
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (!got || u < 0) break;
            int a_sh = 0;
            const Unit un = CL ? decode_cunit(p, u, rank, total_tiles, s_tiles, s_off, a_sh)
                               : decode_unit(p, u, total_tiles, s_tiles, s_off, s_ord);
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(tfull0 + 8 * acc, acc_phase, lim, abort_flag);
                if (!ok) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 4, blockIdx.x, u);
                    abort_cta(abort_flag);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int m = un.m0 + row;
            const bool valid = m < un.nrows;
            const int64_t orow = (int64_t)un.row0 + m;
            const uint32_t tb = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kAccCols);
            const int nvalid = min(BM, un.nrows - un.m0);
            if (p.narrow && nvalid <= kNarrowMax) {
                // narrow tail: this thread holds feature `row` of each 128-feature
                // region, one tile row per TMEM column
                const int64_t orow0 = (int64_t)un.row0 + un.m0;
                if (EPI == EPI_SWIGLU) {
                    f16* o = (f16*)p.out + orow0 * p.ldo + un.nb * 128 + row;
                    bf16* ob = (bf16*)p.out + orow0 * p.ldo + un.nb * 128 + row;
                    float mx = 0.f;
#pragma unroll 1
                    for (int c = 0; c < nvalid; c += 32) {
                        uint32_t gr[32], ur[32];
                        tmem_ld32(tb + c, gr);
                        tmem_ld32(tb + 128 + c, ur);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c + i < nvalid) {
                                const float h = swiglu(__uint_as_float(gr[i]), __uint_as_float(ur[i]));
                                if (p.out_f16) {
                                    mx = fmaxf(mx, fabsf(h));
                                    o[(int64_t)(c + i) * p.ldo] = __float2half_rn(h);
                                } else {
                                    ob[(int64_t)(c + i) * p.ldo] = __float2bfloat16_rn(h);
                                }
                            }
                    }
                    if (p.out_f16 && !(mx <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 5, blockIdx.x, 0);
                } else {
                    float mx = 0.f;
#pragma unroll 1
                    for (int r = 0; r < p.BN / 128; ++r) {
                        const int64_t col = (int64_t)un.nb * p.BN + r * 128 + row;
#pragma unroll 1
                        for (int c = 0; c < nvalid; c += 32) {
                            uint32_t v[32];
                            tmem_ld32(tb + r * 128 + c, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (c + i < nvalid) {
                                    const float y = __uint_as_float(v[i]);
                                    const int64_t at = (orow0 + c + i) * p.ldo + col;
                                    if (p.out_f16) {
                                        mx = fmaxf(mx, fabsf(y));
                                        ((f16*)p.out)[at] = __float2half_rn(y);
                                    } else {
                                        ((bf16*)p.out)[at] = __float2bfloat16_rn(y);
                                    }
                                }
                        }
                    }
                    if (p.out_f16 && !(mx <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 6, blockIdx.x, 0);
                }
            } else if (EPI == EPI_SWIGLU) {
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
            } else if (!p.out_f32 && !p.cmb_out && p.BN % 64 == 0) {
                // 16-bit y through this warp's staging block, 64 columns per pass
                uint8_t* st = s_stage + (size_t)sub * 32 * kStageRow;
                const int nv = min(32, max(0, un.nrows - (un.m0 + sub * 32)));  // valid rows of the warp
                const int64_t orow0 = (int64_t)un.row0 + un.m0 + sub * 32;
                float mx = 0.f;
#pragma unroll 1
                for (int c = 0; c < p.BN; c += 64) {
                    uint32_t r[64];
                    tmem_ld32x2(tb + c, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        uint4 pk;
                        if (p.out_f16) {
                            __half2* h2 = (__half2*)&pk;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float a = __uint_as_float(r[8 * v + 2 * j]), b = __uint_as_float(r[8 * v + 2 * j + 1]);
                                mx = fmaxf(mx, fmaxf(fabsf(a), fabsf(b)));
                                h2[j] = __floats2half2_rn(a, b);
                            }
                        } else {
                            __nv_bfloat162* h2 = (__nv_bfloat162*)&pk;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                h2[j] = __floats2bfloat162_rn(__uint_as_float(r[8 * v + 2 * j]),
                                                              __uint_as_float(r[8 * v + 2 * j + 1]));
                        }
                        *(uint4*)(st + lane * kStageRow + 16 * v) = pk;
                    }
                    __syncwarp();
                    const int n0 = un.nb * p.BN + c;
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = 4 * it + (lane >> 3), ch = lane & 7;
                        const uint4 pk = *(const uint4*)(st + rr * kStageRow + 16 * ch);
                        if (rr < nv) *(uint4*)((uint16_t*)p.out + (orow0 + rr) * p.ldo + n0 + 8 * ch) = pk;
                    }
                    __syncwarp();
                }
                // (rows past the group hold whatever the stage held: they are
                // neither stored nor range-checked)
                if (p.out_f16 && valid && !(mx <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 6, blockIdx.x, 0);
            } else {
#pragma unroll 1
                for (int c = 0; c < p.BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c, r);
                    tmem_wait_ld();
                    if (valid && p.cmb_out) {
                        // fused unpermutation: this row is token orow of the shared group
                        const int n0 = un.nb * p.BN + c;
                        const int64_t TK = (int64_t)p.rows * p.cmb_k;
                        float a[32];
                        float m = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float v = p.out_f16 ? __half2float(__float2half_rn(__uint_as_float(r[i])))
                                                      : __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[i])));
                            m = fmaxf(m, fabsf(__uint_as_float(r[i])));
                            a[i] = fmaf(1.0f, v, 0.0f);
                        }
                        if (p.out_f16 && !(m <= 65504.f)) record_error(p.err, MOE_ERR_NONFINITE, 6, blockIdx.x, 0);
                        if (p.out_f16)
                            combine_chunk32((const f16*)p.cmb_y, p.N, p.cmb_inv, p.cmb_blob, p.cmb_k, orow, TK, n0, a, p.err);
                        else
                            combine_chunk32((const bf16*)p.cmb_y, p.N, p.cmb_inv, p.cmb_blob, p.cmb_k, orow, TK, n0, a,
                                            p.err);
                        if (p.cmb_out_f32) {
                            float* o = (float*)p.cmb_out + orow * p.N + n0;
#pragma unroll
                            for (int i = 0; i < 32; i += 4) *(float4*)(o + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
                        } else {
                            store_bf16x32((bf16*)p.cmb_out + orow * p.N + n0, a);
                        }
                    } else if (valid) {
                        const int n0 = un.nb * p.BN + c;
                        if (p.out_f32) {
                            float* o = (float*)p.out + un.ks * p.split_stride + orow * p.ldo + n0;
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                float4 v = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                       __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                                if (p.bias) {
                                    v.x += __ldg(p.bias + n0 + i);
                                    v.y += __ldg(p.bias + n0 + i + 1);
                                    v.z += __ldg(p.bias + n0 + i + 2);
                                    v.w += __ldg(p.bias + n0 + i + 3);
                                }
                                *(float4*)(o + i) = v;
                            }
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
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * kAccCols)
                     : "memory");
    }
    if (p.sched && threadIdx.x == 0) {
        // the last CTA to finish (every CTA's counter draws are done) rewinds
        // the counters for the next launch on the stream
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(p.sched, 0);
            atomicExch(p.sched + 1, 0);
        }
    }
    if (CL) cluster_sync();  // no copy or commit of the peer still targets this CTA
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    });
    return fn;
}

// 2D tensor of 2-byte elements [rows, cols] row-major, box {64 cols,
// box_rows}, 128B swizzle.  TMA copies bytes without conversion, so the map
// serves bf16 and fp16 data alike.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn || rows < 1) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

int plain_bn(int N) {
    if (N % 256 == 0) return 256;
    if (N <= 256 && N % 32 == 0) return N;
    return 0;
}

struct Maps {
    CUtensorMap a, a_sh, b, b2, af, a_shf, ah, a_shh;
};

// Launch one instantiation.  grid: CTAs for a plain launch; with CL, the
// upper bound on CTAs (rounded down to whole clusters and capped at the
// clusters that fit on the GPU at once).
template <int EPI, bool PAIR, bool CL>
cudaError_t launch_one(int grid, const Maps& m, const Params& p, cudaStream_t stream) {
    auto kern = gemm_tc_kernel<EPI, PAIR, CL>;
    // per device: the shared-memory limit raised and (CL) the most
    // co-resident clusters
    int ready = 0;
    cudaError_t e0 = per_device_value((const void*)kern, [&](int* v) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        int n = 1;
        if (CL) {
            int dev = 0, sms = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaLaunchConfig_t qc = {};
            qc.gridDim = dim3(2 * std::max(1, sms / 2));
            qc.blockDim = dim3(kThreads);
            qc.dynamicSmemBytes = kSmemBytes;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 2;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            qc.attrs = qa;
            qc.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&n, (void*)kern, &qc);
            if (e != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
        }
        *v = n;
        return cudaSuccess;
    }, &ready);
    if (e0 != cudaSuccess) return e0;
    if (!CL)
        return launch_kernel(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, 1, m.a, m.a_sh, m.b, m.b2, m.af,
                             m.a_shf, m.ah, m.a_shh, p);
    return launch_kernel(kern, dim3(2 * std::max(1, std::min(ready, grid / 2))), dim3(kThreads), kSmemBytes, stream, 2,
                         m.a, m.a_sh, m.b, m.b2, m.af, m.a_shf, m.ah, m.a_shh, p);
}

}  // namespace tc

bool gemm_tc_supported(const GroupedGemm& g) {
    using namespace tc;
    if (g.cmb_out) {  // fused unpermutation: one plain group of 16-bit y, 16-byte row segments
        if (g.offsets || g.b2 || g.Ka != g.Kb || (g.out_elem != kF16 && g.out_elem != kBF16) || g.N % 256 ||
            g.cmb_k < 1 || !aligned16(g.cmb_out) || !aligned16(g.cmb_y))
            return false;
    }
    if (g.elem != kBF16 && g.elem != kF16) return false;
    if (g.b_elem > 0 && g.b_elem != g.elem) return false;  // the tensor cores take one type for A and B
    if (!encode_fn()) return false;
    if (g.offsets && g.G + 1 > kTabEntries) return false;
    if (g.Kb % BK || g.Kb < BK || (g.Ka != g.Kb && g.Ka != 2 * g.Kb)) return false;
    if (g.b2 && g.Ka != g.Kb) return false;  // the hi/lo pair is only the down GEMM's input
    if (!aligned16(g.a) || !aligned16(g.b) || !aligned16(g.out)) return false;
    if (g.b2) {  // SwiGLU
        if (g.N % 128 || (g.out_elem != kBF16 && g.out_elem != kF16) || g.bias) return false;
        if (g.out_elem == kF16 && g.out_pair) return false;
        if (!aligned16(g.b2) || (g.a_shared && !aligned16(g.a_shared))) return false;
    } else {
        if (!plain_bn(g.N) || g.out_pair) return false;
        if (g.out_elem != kBF16 && g.out_elem != kF32 && g.out_elem != kF16) return false;
        if (g.bias && g.out_elem != kF32) return false;
    }
    if (g.ldo % 8) return false;
    return true;
}


cudaError_t launch_gemm_tc(const GroupedGemm& g, int num_sms, cudaStream_t stream) {
    using namespace tc;
    const bool sw = g.b2 != nullptr;
    const bool pair = g.Ka == 2 * g.Kb;
    Params p = {};
    p.G = g.offsets ? g.G : 1;
    p.g_end = (g.offsets && g.g_end > 0 && g.g_end < g.G) ? g.g_end : p.G;
    p.sched = g.sched;
    p.shared_group = g.shared_group;
    p.offsets = g.offsets;
    p.tiles = g.tiles;
    p.rows = g.rows;
    p.BN = sw ? 256 : plain_bn(g.N);
    if (!sw && !g.offsets) {
        // single group (router): narrow the feature block while twice the
        // units (K slices included) still fit in one wave on the SMs (T=128 at
        // E=512 with 8 K slices: 16 x 8 units of 32 experts; T=1024: 2 x 8
        // units of 8 row tiles x 256 experts)
        const int row_tiles = (g.rows + BM - 1) / BM;
        const int ks = (g.ksplit > 1 && (g.Kb / BK) % g.ksplit == 0) ? g.ksplit : 1;
        while (p.BN > 32 && g.N % (p.BN / 2) == 0 && (p.BN / 2) % 32 == 0 &&
               row_tiles * (g.N / p.BN) * ks * 2 <= num_sms)
            p.BN /= 2;
    }
    p.NB = sw ? g.N / 128 : g.N / p.BN;
    p.N = g.N;
    p.KB = g.Kb / BK;
    p.KS = 1;
    if (!g.offsets && g.ksplit > 1 && p.KB % g.ksplit == 0) p.KS = g.ksplit;
    p.split_stride = g.split_stride;
    p.a_lo_x = g.Kb;
    p.b_group_rows = g.N;
    p.ldo = g.ldo;
    p.out_pair = g.out_pair;
    p.out_f32 = g.out_elem == kF32;
    p.out_f16 = g.out_elem == kF16;
    p.in_f16 = g.elem == kF16;
    p.b_stage = (sw ? 256 : p.BN) * BK * 2;
    p.stages = std::min(kMaxStages, kRingBytes / ((pair ? Geo<true>::kAStage : Geo<false>::kAStage) + p.b_stage));
    p.out = g.out;
    p.bias = g.bias;
    p.err = g.err;
    p.spin_ns = g.spin_ns > 0 ? g.spin_ns : 2000000000LL;
    p.cmb_out = g.cmb_out;
    p.cmb_out_f32 = g.cmb_out_f32;
    p.cmb_blob = g.cmb_blob;
    p.cmb_inv = g.cmb_inv;
    p.cmb_y = g.cmb_y;
    p.cmb_k = g.cmb_k;
    p.rem_only = g.rem_only && g.offsets;
    p.order = p.rem_only ? g.rem_order : nullptr;

    // tile pairs: whole weight blocks in pairs (SwiGLU: 128 gate + 128 up;
    // plain: 256-wide), no K split, one A input; static unit order
    const bool cl = g.mcast && !pair && p.KS == 1 && p.NB % 2 == 0 && (sw || p.BN == 256) && !p.rem_only;
    if (cl) p.sched = nullptr;
    // narrow tails: expert GEMMs with 16-bit outputs in whole 128-feature regions
    p.narrow = g.narrow && !pair && p.KS == 1 && !g.out_pair && !g.bias && g.out_elem != kF32 &&
               (sw || p.BN % 128 == 0) && !g.cmb_out;

    Maps m;
    const int G = g.offsets ? g.G : 1;
    if (!make_map(&m.a, g.a, g.a_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
    if (!make_map(&m.af, g.a, g.a_rows, g.Ka, BM)) return cudaErrorInvalidValue;
    if (cl && !make_map(&m.ah, g.a, g.a_rows, g.Ka, BM / 2)) return cudaErrorInvalidValue;
    if (!cl) m.ah = m.af;
    if (g.a_shared) {
        if (!make_map(&m.a_sh, g.a_shared, g.a_shared_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
        if (!make_map(&m.a_shf, g.a_shared, g.a_shared_rows, g.Ka, BM)) return cudaErrorInvalidValue;
        if (cl && !make_map(&m.a_shh, g.a_shared, g.a_shared_rows, g.Ka, BM / 2)) return cudaErrorInvalidValue;
        if (!cl) m.a_shh = m.a_shf;
    } else {
        m.a_sh = m.a;
        m.a_shf = m.af;
        m.a_shh = m.ah;
    }
    const int brow_box = sw ? 128 : p.BN;
    if (!make_map(&m.b, g.b, (int64_t)G * g.N, g.Kb, brow_box)) return cudaErrorInvalidValue;
    if (sw) {
        if (!make_map(&m.b2, g.b2, (int64_t)G * g.N, g.Kb, brow_box)) return cudaErrorInvalidValue;
    } else if (cl) {  // halves of the 256-row B tile
        if (!make_map(&m.b2, g.b, (int64_t)G * g.N, g.Kb, 128)) return cudaErrorInvalidValue;
    } else {
        m.b2 = m.b;
    }
    const int max_units = cl ? g.max_tiles * (p.NB / 2) * 2 : g.max_tiles * p.NB * p.KS;  // CTAs' worth
    if (max_units <= 0) return cudaGetLastError();
    const int grid = std::max(1, std::min(g.max_ctas > 0 ? std::min(num_sms, g.max_ctas) : num_sms, max_units));
    cudaError_t e;
    if (cl && sw) e = launch_one<EPI_SWIGLU, false, true>(grid, m, p, stream);
    else if (cl) e = launch_one<EPI_PLAIN, false, true>(grid, m, p, stream);
    else if (sw) e = launch_one<EPI_SWIGLU, false, false>(grid, m, p, stream);
    else if (pair) e = launch_one<EPI_PLAIN, true, false>(grid, m, p, stream);
    else e = launch_one<EPI_PLAIN, false, false>(grid, m, p, stream);
    count_launches(1);
    return e;
}

}  // namespace moe
