// Grouped GEMM with E4M3 operands and fp32 block scales on the tcgen05
// tensor cores (the FP8 layer's expert GEMMs).
//
// "Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU" (English page,
// "Roofline Validation"): FP8 scaling blocks, audited against a
// higher-precision path.  Here: weights carry one fp32 scale per 128x128
// block, activations one per token per 128 columns, so every 128-wide slice
// of K has its own product of scales.  tcgen05.mma kind::f8f6f4 multiplies
// one such slice (4 MMAs of K=32) into one of two TMEM chunk buffers; the
// epilogue warps read the chunk, multiply it by s_a[row] * s_w[block] and add
// it to fp32 accumulators held in registers, while the MMA fills the other
// buffer.  The scales are not powers of two, so they cannot ride in the
// MMA's own block-scale operands.
//
// Unit, ordering, ring and error handling follow gemm_tc.cu (128 rows x 256
// accumulator columns; A in 16-row TMA boxes; 4-stage ring of 16 KB A + 32 KB
// B; bounded waits).  384 threads in three warpgroups: warp 0 TMA, warp 1
// TMEM + MMA, warps 2-3 copy staged y out (down GEMM at prefill sizes) or
// idle; warps 4..11 epilogue (two per TMEM lane
// quarter, each owning half of the columns).  The block launches at 168
// registers per thread; warpgroup 0 gives back down to 40 and the two
// epilogue warpgroups take up to 232 (4*32*128 = 8*32*64 registers, so the
// split balances exactly) for their 128 fp32 accumulators.
//   SwiGLU (gate/up): columns 0..127 gate, 128..255 up, features nb*128..+127.
//     A thread owns 64 gate and the matching 64 up columns of its row; at the
//     end of the unit it forms h, the two halves of a row exchange their amax
//     through shared memory, and h is written as E4M3 codes with one fp32
//     scale per row and 128 features (the next GEMM's activation format).
//   Plain (down): 256 output features = two 128-row weight blocks, one per
//     column half; the result is written as bf16.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();  // gemm_tc.cu

namespace f8 {

constexpr int BM = 128;
constexpr int BKB = 128;                  // K per stage: 128 E4M3 = one 128-byte swizzle row
constexpr int kABytes = BM * BKB;         // 16 KB
constexpr int kBBytes = 256 * BKB;        // 32 KB
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;              // first epilogue warp (warpgroups 1 and 2)
constexpr int kThreads = 128 + 32 * kEpiWarps;
constexpr int kRegsLaunch = 168, kRegsLow = 40, kRegsHigh = 232;
static_assert(4 * (kRegsLaunch - kRegsLow) == kEpiWarps * (kRegsHigh - kRegsLaunch), "register split must balance");
static_assert(kThreads * kRegsLaunch <= 65536, "launch registers exceed the SM");
constexpr int kAccCols = 256;
constexpr int kBoxRowsA = 16;
constexpr uint32_t kBarBytes = 512;  // mbarriers, TMEM address, abort flag, unit ring
// Shared copies of the row-tile prefix and the row offsets (G <= 1025
// groups): the producer finds a unit's group without leaving the SM.
constexpr int kTabEntries = 1056;

enum Epi : int { EPI_SWIGLU = 0, EPI_PLAIN = 1 };

// Ring depth and shared-memory plan.  The plain (down) epilogue writes
// 256 B of bf16 y per thread and unit.  Stored straight from the
// row-per-lane layout every warp store touches 32 rows, and at prefill sizes
// those stores throttled the load/store unit (FP8 prefill down 1.20 ms).
// With STG the epilogue instead drops the unit's whole 128 x 256 y tile into
// shared memory (rows kYRow bytes apart) and goes straight on to the next
// unit; warps 2 and 3 (idle otherwise) copy the tile out, one 512-byte row
// per warp instruction, while the next unit's slices run, so the 64 KB per
// unit leave spread over the unit instead of in a burst that held the MMA
// (FP8 prefill down 1.02 -> 0.92 ms; the epilogue had spent a fifth of its
// time in the unit-end stores).  The space comes from a 3-stage ring.
// Decode-sized tiles hold a few rows, stream weights from HBM and want the
// 4-stage ring, so they keep the direct stores.
constexpr int kYRow = 528;  // y staging row stride: 512 B + 16 (conflict-free row-per-lane writes)
template <int EPI, bool STG> struct Cfg {
    static constexpr int kStages = (EPI == EPI_PLAIN && STG) ? 3 : 4;
    static constexpr uint32_t kStagingBytes = (EPI == EPI_PLAIN && STG) ? BM * kYRow : 0;
    static constexpr uint32_t kSmemBytes =
        1024 + kStages * (kABytes + kBBytes) + kBarBytes + 2 * 2 * 128 * 4 + 2 * kTabEntries * 4 + kStagingBytes;
    static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
};

struct Params {
    int G, shared_group;
    int g_end;            // grouped: units cover the row tiles of groups [0, g_end)
    int* sched;           // [2] device: next-unit counter and finished-CTA count, or nullptr (static order)
    int rows;             // single group (offsets == nullptr): its row count
    const int32_t* offsets;
    const int32_t* tiles;
    int NB;               // feature blocks per row tile
    int N;                // output features of a group
    int KB;               // 128-wide K chunks
    const float* a_scale;         // [rows of A, KB]
    const float* a_shared_scale;  // [rows of A_shared, KB]
    const float* b_scale;         // [G, N/128, KB]
    const float* b2_scale;
    void* out;
    int ldo;                      // output row stride in elements
    float* out_scale;             // SwiGLU: [R, N/128]
    uint32_t* err;
    int64_t spin_ns;
    // fused unpermutation (plain, single group; see GroupedGemm::cmb_out)
    void* cmb_out;
    int cmb_out_f32;
    const int32_t* cmb_blob;
    const int32_t* cmb_inv;
    const void* cmb_y;
    int cmb_k;
};

struct Unit {
    int g, m0, row0, nrows, nb;
};

// s_tiles / s_off: shared copies of p.tiles and p.offsets (entries 0..G).
__device__ __forceinline__ Unit decode_unit(const Params& p, int u, const int32_t* s_tiles, const int32_t* s_off) {
    Unit r;
    const int rt = u / p.NB;
    r.nb = u - rt * p.NB;
    if (p.offsets) {
        r.g = find_group_smem(s_tiles, p.G, rt);
        r.m0 = (rt - s_tiles[r.g]) * BM;
        r.row0 = s_off[r.g];
        r.nrows = s_off[r.g + 1] - r.row0;
    } else {
        r.g = 0;
        r.m0 = rt * BM;
        r.row0 = 0;
        r.nrows = p.rows;
    }
    return r;
}

// The per-slice hand-off waits (MMA <-> promotion) of the gate/up kernel
// poll instead of suspending: FP8 prefill gate/up 1.50 ms against 1.535 with
// try_wait; the down kernel measured 3-5 us slower with polling and keeps
// try_wait.
template <int EPI>
__device__ __forceinline__ bool hot_wait(uint32_t bar, uint32_t parity, int64_t lim, volatile int* abort) {
    return EPI == EPI_SWIGLU ? mbar_spin(bar, parity, lim, abort) : mbar_wait(bar, parity, lim, abort);
}

template <int EPI, bool STG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a_sh,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_b2,
                    const __grid_constant__ CUtensorMap tm_af, const __grid_constant__ CUtensorMap tm_a_shf,
                    const Params p) {
    constexpr int kStages = Cfg<EPI, STG>::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kABytes;
    uint64_t* bars = (uint64_t*)(sB + kStages * kBBytes);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t cfull0 = smem_u32(bars + 2 * kStages), cempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
    // [2 unit parities][4 lane quarters]: amax exchange between the two warps
    // that hold the two column halves of the same 32 rows
    const uint32_t xbar0 = smem_u32(bars + 2 * kStages + 5);
    // unit ring: full/empty [4 each] and 4 slots (see gemm_tc.cu)
    const uint32_t ufull0 = smem_u32(bars + 2 * kStages + 13), uempty0 = smem_u32(bars + 2 * kStages + 17);
    // y staging (plain, STG): tile written by the epilogue / copied out by warps 2-3
    const uint32_t yfull = smem_u32(bars + 2 * kStages + 21), yempty = smem_u32(bars + 2 * kStages + 22);
    uint32_t* tmem_slot = (uint32_t*)(bars + 2 * kStages + 23);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    // unit ring slots: [4][6] = unit number, then its decoded group, m0, row0,
    // nrows, nb (the producer decodes each unit once for every role)
    volatile int* s_units = (volatile int*)(tmem_slot + 2);
    // the staged y tile: first global row, valid rows (-1: no more tiles), first column
    volatile int* s_yinfo = s_units + 4 * 6;
    static_assert((2 * kStages + 23) * 8 + 8 + 4 * 6 * 4 + 3 * 4 <= kBarBytes, "barrier block overflows");
    float* s_amax = (float*)(smem + kStages * (kABytes + kBBytes) + kBarBytes);  // [2 units][2 halves][128 rows]
    int32_t* s_tiles = (int32_t*)(s_amax + 2 * 2 * 128);
    int32_t* s_off = s_tiles + kTabEntries;
    uint8_t* s_stage = (uint8_t*)(s_off + kTabEntries);  // plain, STG: [128 rows][kYRow]
    pdl_wait_then_release();
    if (p.offsets)
        for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
            s_tiles[i] = __ldg(p.tiles + i);
            s_off[i] = __ldg(p.offsets + i);
        }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(cfull0 + 8 * b, 1);
            mbar_init(cempty0 + 8 * b, kEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(yfull, kEpiWarps);
        mbar_init(yempty, 2);  // the two copy warps
        for (int b = 0; b < 8; ++b) mbar_init(xbar0 + 8 * b, 2 * 32);
        for (int i = 0; i < 4; ++i) {
            mbar_init(ufull0 + 8 * i, 1);
            mbar_init(uempty0 + 8 * i, 1 + kEpiWarps);  // the MMA issuer and the epilogue warps
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
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int total_units = (p.offsets ? __ldg(p.tiles + p.g_end) : (p.rows + BM - 1) / BM) * p.NB;
    const int64_t lim = p.spin_ns;

    if (warp < kEpiWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            constexpr uint32_t b_bytes = 256u * BKB;
            bool ok = true;
            // units from the launch-wide counter (drawn one ahead) or in the
            // static round-robin order, published through the unit ring
            int next_u = p.sched ? atomicAdd(p.sched, 1) : blockIdx.x;
            for (int i = 0; ok; ++i) {
                int u = next_u;
                if (u >= total_units) u = -1;
                if (u >= 0) next_u = p.sched ? atomicAdd(p.sched, 1) : blockIdx.x + (i + 1) * gridDim.x;
                if (!mbar_wait(uempty0 + 8 * (i & 3), ((i >> 2) & 1) ^ 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 15, blockIdx.x, i);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                Unit un = {};
                if (u >= 0) un = decode_unit(p, u, s_tiles, s_off);
                volatile int* slot = s_units + 6 * (i & 3);
                slot[0] = u;
                slot[1] = un.g;
                slot[2] = un.m0;
                slot[3] = un.row0;
                slot[4] = un.nrows;
                slot[5] = un.nb;
                mbar_arrive(ufull0 + 8 * (i & 3));
                if (u < 0) break;
                const bool sh = un.g == p.shared_group;
                const CUtensorMap* ta = sh ? &tm_a_sh : &tm_a;
                const CUtensorMap* taf = sh ? &tm_a_shf : &tm_af;
                const int a_y = sh ? un.m0 : un.row0 + un.m0;
                const int valid = min(BM, un.nrows - un.m0);
                const int nbox = (valid + kBoxRowsA - 1) / kBoxRowsA;
                const uint32_t bytes = (uint32_t)nbox * kBoxRowsA * BKB + b_bytes;
                const int b_y = un.g * p.N + un.nb * ((EPI == EPI_SWIGLU) ? 128 : 256);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 11, blockIdx.x, u);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, bytes);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    const uint32_t a_dst = smem_u32(sA + stage * kABytes);
                    const uint32_t b_dst = smem_u32(sB + stage * kBBytes);
                    if (nbox * kBoxRowsA == BM) {  // (nearly) full tile: one 128-row box
                        tma_load_2d(a_dst, taf, fb, kb * BKB, a_y);
                    } else {
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(a_dst + i * kBoxRowsA * BKB, ta, fb, kb * BKB, a_y + i * kBoxRowsA);
                    }
                    tma_load_2d(b_dst, &tm_b, fb, kb * BKB, b_y);
                    if (EPI == EPI_SWIGLU) tma_load_2d(b_dst + 128 * BKB, &tm_b2, fb, kb * BKB, b_y);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < kStages; ++s)
                    if (armed & (1u << s)) {
                        volatile int never = 0;
                        mbar_wait(full0 + 8 * s, (armed_parity >> s) & 1u, 1000000000LL, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ----------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0, chunk = 0;
            const uint32_t idesc = idesc_e4m3(BM, 256);
            bool ok = true;
            for (int i = 0; ok; ++i) {
                if (!mbar_wait(ufull0 + 8 * (i & 3), (i >> 2) & 1, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 16, blockIdx.x, i);
                    *abort_flag = 1;
                    break;
                }
                const int u = s_units[6 * (i & 3)];
                mbar_arrive(uempty0 + 8 * (i & 3));
                if (u < 0) break;
                for (int kb = 0; kb < p.KB; ++kb) {
                    const uint32_t buf = chunk & 1u, cpar = (chunk >> 1) & 1u;
                    if (!hot_wait<EPI>(full0 + 8 * stage, phase, lim, abort_flag) ||
                        !hot_wait<EPI>(cempty0 + 8 * buf, cpar ^ 1u, lim, abort_flag)) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 12, blockIdx.x, u);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * kAccCols;
                    const uint64_t ad = umma_desc(smem_u32(sA + stage * kABytes));
                    const uint64_t bd = umma_desc(smem_u32(sB + stage * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < BKB / 32; ++kk)  // K=32 E4M3 per MMA: 32 bytes along the row
                        umma_e4m3(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, kk != 0);
                    umma_commit(empty0 + 8 * stage);
                    umma_commit(cfull0 + 8 * buf);
                    ++chunk;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            umma_commit(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, 1000000000LL, &never);
        }
    } else if (EPI == EPI_PLAIN && STG) {
        // ------------------------------------- y copy-out (warps 2 and 3)
        // Each staged tile: rows of the group only, warp 2 the even rows,
        // warp 3 the odd; lane l moves bytes 16l..16l+15 of the row's 512.
        const int cw = warp - 2;
        for (uint32_t n = 0;; ++n) {
            int w_ok = 1;
            if (lane == 0) {
                w_ok = mbar_wait(yfull, n & 1u, lim, abort_flag);
                if (!w_ok) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 18, blockIdx.x, (int)n);
                    *abort_flag = 1;
                }
            }
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) break;
            const int64_t grow = (int64_t)s_yinfo[0];
            const int nv = s_yinfo[1], col0 = s_yinfo[2];
            if (nv < 0) break;
            for (int r = cw; r < nv; r += 2) {
                const uint4 v = *(const uint4*)(s_stage + r * kYRow + 16 * lane);
                *(uint4*)((bf16*)p.out + (grow + r) * p.ldo + col0 + 8 * lane) = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(yempty);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ----------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;
        const int sub = warp & 3;      // TMEM lane quarter
        const int half = ew >> 2;      // which half of the columns
        const int row = sub * 32 + lane;
        uint32_t chunk = 0;
        uint32_t ny = 0;  // y tiles staged so far (plain, STG)
        bool ok = true;
        for (int i = 0; ok; ++i) {
            int u = -1;  // -1: no more units (or a wait that ran out)
            Unit un = {};
            if (lane == 0) {
                if (mbar_wait(ufull0 + 8 * (i & 3), (i >> 2) & 1, lim, abort_flag)) {
                    const volatile int* slot = s_units + 6 * (i & 3);
                    u = slot[0];
                    un.g = slot[1];
                    un.m0 = slot[2];
                    un.row0 = slot[3];
                    un.nrows = slot[4];
                    un.nb = slot[5];
                    mbar_arrive(uempty0 + 8 * (i & 3));
                } else {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 17, blockIdx.x, i);
                    *abort_flag = 1;
                }
            }
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u < 0) break;
            un.g = __shfl_sync(0xffffffffu, un.g, 0);
            un.m0 = __shfl_sync(0xffffffffu, un.m0, 0);
            un.row0 = __shfl_sync(0xffffffffu, un.row0, 0);
            un.nrows = __shfl_sync(0xffffffffu, un.nrows, 0);
            un.nb = __shfl_sync(0xffffffffu, un.nb, 0);
            const int unit_par = i & 1;
            const bool sh = un.g == p.shared_group;
            const int m = un.m0 + row;
            const bool valid = m < un.nrows;
            const int64_t arow = valid ? (sh ? (int64_t)m : (int64_t)un.row0 + m) : 0;
            const float* asc = (sh ? p.a_shared_scale : p.a_scale) + arow * p.KB;
            const int nblocks = p.N / 128;
            float acc[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) acc[c] = 0.0f;
            // weight scale rows for this unit: [g][block][KB]
            const float* wsc1;
            const float* wsc2;
            if (EPI == EPI_SWIGLU) {
                wsc1 = p.b_scale + ((int64_t)un.g * nblocks + un.nb) * p.KB;
                wsc2 = p.b2_scale + ((int64_t)un.g * nblocks + un.nb) * p.KB;
            } else {
                wsc1 = p.b_scale + ((int64_t)un.g * nblocks + 2 * un.nb + half) * p.KB;
                wsc2 = wsc1;
            }
            float sa_next = __ldg(asc), s1_next = __ldg(wsc1), s2_next = __ldg(wsc2);
            for (int kb = 0; kb < p.KB; ++kb) {
                const float sa = sa_next, s1 = s1_next, s2 = s2_next;
                if (kb + 1 < p.KB) {  // next chunk's scales, fetched while this one is consumed
                    sa_next = __ldg(asc + kb + 1);
                    s1_next = __ldg(wsc1 + kb + 1);
                    s2_next = __ldg(wsc2 + kb + 1);
                }
                const uint32_t buf = chunk & 1u, cpar = (chunk >> 1) & 1u;
                int w_ok = 1;
                if (lane == 0) {
                    w_ok = hot_wait<EPI>(cfull0 + 8 * buf, cpar, lim, abort_flag);
                    if (!w_ok) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 13, blockIdx.x, u);
                        *abort_flag = 1;
                    }
                }
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem_base + ((uint32_t)(sub * 32) << 16) + buf * kAccCols;
                const float f1 = sa * s1, f2 = sa * s2;
                // Two 32-column TMEM loads per wait, then the promotion with
                // paired fp32 FMAs (two lanes of work per instruction).  The
                // buffer goes back to the MMA as soon as the second half is
                // in registers, before that half is promoted: the MMA can
                // then start the slice after next about 130 cycles sooner.
                // SwiGLU: q=0 -> gate columns 64*half.., q=1 -> up columns
                // 128+64*half..; plain: q -> columns 128*half + 64*q.
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t r[64];
                    const int col = (EPI == EPI_SWIGLU) ? (q == 0 ? 64 * half : 128 + 64 * half) : 128 * half + 64 * q;
                    tmem_ld32x2(tb + col, r);
                    tmem_wait_ld();
                    if (q == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(cempty0 + 8 * buf);
                    }
                    const float f = (EPI == EPI_SWIGLU && q == 1) ? f2 : f1;
                    const float2 ff = make_float2(f, f);
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        float2 a = make_float2(acc[64 * q + i], acc[64 * q + i + 1]);
                        a = __ffma2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), ff, a);
                        acc[64 * q + i] = a.x;
                        acc[64 * q + i + 1] = a.y;
                    }
                }
                ++chunk;
            }
            if (!ok) break;
            const int64_t orow = (int64_t)un.row0 + m;
            if (EPI == EPI_SWIGLU) {
                float amax = 0.0f;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    acc[c] = swiglu(acc[c], acc[64 + c]);
                    amax = fmaxf(amax, fabsf(acc[c]));
                }
                // the two column halves of a row meet in shared memory; an
                // mbarrier (bounded wait) rather than a named barrier, so an
                // aborting warp cannot strand the others
                float* sm = s_amax + unit_par * 256;
                sm[half * 128 + row] = amax;
                const uint32_t xb = xbar0 + 8 * (unit_par * 4 + sub);
                mbar_arrive(xb);
                if (!mbar_wait(xb, (i >> 1) & 1u, lim, abort_flag)) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 14, blockIdx.x, u);
                    *abort_flag = 1;
                    break;
                }
                amax = fmaxf(sm[row], sm[128 + row]);
                float sc = __fdiv_rn(amax, 448.0f), inv = __fdiv_rn(448.0f, amax);
                if (amax == 0.0f) {
                    sc = 1.0f;
                    inv = 1.0f;
                }
                if (valid) {
                    uint8_t* o = (uint8_t*)p.out + orow * p.ldo + un.nb * 128 + 64 * half;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int c = 16 * v + 4 * j;
                            w4[j] = (uint32_t)f32x2_to_e4m3x2(__fmul_rn(acc[c], inv), __fmul_rn(acc[c + 1], inv)) |
                                    ((uint32_t)f32x2_to_e4m3x2(__fmul_rn(acc[c + 2], inv), __fmul_rn(acc[c + 3], inv))
                                     << 16);
                        }
                        *(uint4*)(o + 16 * v) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    if (half == 0) p.out_scale[orow * nblocks + un.nb] = sc;
                }
            } else if (valid && p.cmb_out) {
                // fused unpermutation: this row is token orow of the shared group
                const int64_t TK = (int64_t)p.rows * p.cmb_k;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {  // (unrolled: acc stays in registers)
                    const int n0 = un.nb * 256 + 128 * half + 32 * cc;
                    float a[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        a[i] = fmaf(1.0f, __bfloat162float(__float2bfloat16_rn(acc[32 * cc + i])), 0.0f);
                    combine_chunk32((const bf16*)p.cmb_y, p.N, p.cmb_inv, p.cmb_blob, p.cmb_k, orow, TK, n0, a, p.err);
                    if (p.cmb_out_f32) {
                        float* o = (float*)p.cmb_out + orow * p.N + n0;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) *(float4*)(o + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
                    } else {
                        bf16* o = (bf16*)p.cmb_out + orow * p.N + n0;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 pk;
                            __nv_bfloat162* h2 = (__nv_bfloat162*)&pk;
#pragma unroll
                            for (int j = 0; j < 4; ++j) h2[j] = __floats2bfloat162_rn(a[8 * v + 2 * j], a[8 * v + 2 * j + 1]);
                            *(uint4*)(o + 8 * v) = pk;
                        }
                    }
                }
            } else if (EPI == EPI_PLAIN && STG) {
                // y: this thread's 128 values into row `row` of the staging
                // tile, once the copy warps are done with the previous one
                int w_ok = 1;
                if (lane == 0) {
                    w_ok = mbar_wait(yempty, (ny & 1u) ^ 1u, lim, abort_flag);
                    if (!w_ok) {
                        record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 19, blockIdx.x, u);
                        *abort_flag = 1;
                    }
                }
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) break;
                uint8_t* st = s_stage + row * kYRow + 256 * half;
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    uint4 pk;
                    __nv_bfloat162* h2 = (__nv_bfloat162*)&pk;
#pragma unroll
                    for (int j = 0; j < 4; ++j) h2[j] = __floats2bfloat162_rn(acc[8 * v + 2 * j], acc[8 * v + 2 * j + 1]);
                    *(uint4*)(st + 16 * v) = pk;
                }
                if (ew == 0 && lane == 0) {
                    s_yinfo[0] = un.row0 + un.m0;
                    s_yinfo[1] = min(BM, un.nrows - un.m0);
                    s_yinfo[2] = un.nb * 256;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(yfull);
                ++ny;
            } else if (valid) {
                bf16* o = (bf16*)p.out + orow * p.ldo + un.nb * 256 + 128 * half;
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    uint4 pk;
                    __nv_bfloat162* h2 = (__nv_bfloat162*)&pk;
#pragma unroll
                    for (int j = 0; j < 4; ++j) h2[j] = __floats2bfloat162_rn(acc[8 * v + 2 * j], acc[8 * v + 2 * j + 1]);
                    *(uint4*)(o + 8 * v) = pk;
                }
            }
        }
        if (EPI == EPI_PLAIN && STG && !*abort_flag) {
            // no more tiles: an empty one ends the copy warps' loop
            int w_ok = 1;
            if (lane == 0) {
                w_ok = mbar_wait(yempty, (ny & 1u) ^ 1u, lim, abort_flag);
                if (!w_ok) {
                    record_error(p.err, MOE_ERR_DEVICE_TIMEOUT, 19, blockIdx.x, -1);
                    *abort_flag = 1;
                }
            }
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (w_ok) {
                if (ew == 0 && lane == 0) s_yinfo[1] = -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(yfull);
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
    if (p.sched && threadIdx.x == 0) {  // the last CTA rewinds the counters (see gemm_tc.cu)
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(p.sched, 0);
            atomicExch(p.sched + 1, 0);
        }
    }
}

bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn || rows < 1) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)BKB, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, bool STG>
cudaError_t launch_one(int grid, const CUtensorMap& ma, const CUtensorMap& msh, const CUtensorMap& mb,
                       const CUtensorMap& mb2, const CUtensorMap& maf, const CUtensorMap& mshf, const Params& p,
                       cudaStream_t stream) {
    int ready = 0;
    cudaError_t e = per_device_value((const void*)gemm_fp8_kernel<EPI, STG>, [](int* v) {
        // The warpgroup register split (setmaxnreg) balances only at exactly
        // kRegsLaunch registers per thread; anything else could leave the
        // raising warpgroups waiting for registers that never come free.
        cudaFuncAttributes fa;
        cudaError_t e2 = cudaFuncGetAttributes(&fa, gemm_fp8_kernel<EPI, STG>);
        if (e2 != cudaSuccess) return e2;
        if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
        e2 = cudaFuncSetAttribute(gemm_fp8_kernel<EPI, STG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg<EPI, STG>::kSmemBytes);
        if (e2 == cudaSuccess) *v = 1;
        return e2;
    }, &ready);
    if (e != cudaSuccess) return e;
    e = launch_kernel(gemm_fp8_kernel<EPI, STG>, dim3(grid), dim3(kThreads), Cfg<EPI, STG>::kSmemBytes, stream, 1, ma,
                      msh, mb, mb2, maf, mshf, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace f8
}  // namespace tc

bool gemm_fp8_supported(const GroupedGemm& g) {
    using namespace tc::f8;
    if (g.elem != kE4M3 || !tc::encode_fn()) return false;
    if (!g.offsets && (g.rows < 1 || g.a_shared)) return false;  // single group: A only
    if (g.offsets && g.G + 1 > kTabEntries) return false;
    if (g.cmb_out && (g.offsets || g.b2 || g.cmb_k < 1 || ((uintptr_t)g.cmb_out & 15) || ((uintptr_t)g.cmb_y & 15)))
        return false;
    if (g.Ka != g.Kb || g.Kb % BKB || g.N % 128) return false;
    if (!g.a_scale || !g.b_scale) return false;
    if (g.b2) {
        if (!g.b2_scale || !g.out_scale || g.out_elem != kE4M3) return false;
        if (g.offsets && (!g.a_shared || !g.a_shared_scale)) return false;
    } else {
        if (g.N % 256 || g.out_elem != kBF16) return false;
    }
    return true;
}

cudaError_t launch_gemm_fp8(const GroupedGemm& g, int num_sms, cudaStream_t stream) {
    using namespace tc::f8;
    const bool sw = g.b2 != nullptr;
    Params p = {};
    p.G = g.G;
    p.shared_group = g.shared_group;
    p.offsets = g.offsets;
    p.rows = g.rows;
    p.sched = g.sched;
    p.g_end = (g.offsets && g.g_end > 0 && g.g_end < g.G) ? g.g_end : g.G;
    if (!g.offsets) p.G = 1;
    p.tiles = g.tiles;
    p.NB = sw ? g.N / 128 : g.N / 256;
    p.N = g.N;
    p.KB = g.Kb / BKB;
    p.a_scale = g.a_scale;
    p.a_shared_scale = g.a_shared_scale ? g.a_shared_scale : g.a_scale;
    p.b_scale = g.b_scale;
    p.b2_scale = g.b2_scale ? g.b2_scale : g.b_scale;
    p.out = g.out;
    p.ldo = g.ldo;
    p.out_scale = g.out_scale;
    p.err = g.err;
    p.spin_ns = g.spin_ns > 0 ? g.spin_ns : 2000000000LL;
    p.cmb_out = g.cmb_out;
    p.cmb_out_f32 = g.cmb_out_f32;
    p.cmb_blob = g.cmb_blob;
    p.cmb_inv = g.cmb_inv;
    p.cmb_y = g.cmb_y;
    p.cmb_k = g.cmb_k;
    CUtensorMap ma, msh, mb, mb2, maf, mshf;
    if (!make_map_u8(&ma, g.a, g.a_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
    if (!make_map_u8(&maf, g.a, g.a_rows, g.Ka, BM)) return cudaErrorInvalidValue;
    if (g.a_shared) {
        if (!make_map_u8(&msh, g.a_shared, g.a_shared_rows, g.Ka, kBoxRowsA)) return cudaErrorInvalidValue;
        if (!make_map_u8(&mshf, g.a_shared, g.a_shared_rows, g.Ka, BM)) return cudaErrorInvalidValue;
    } else {
        msh = ma;
        mshf = maf;
    }
    if (!make_map_u8(&mb, g.b, (int64_t)g.G * g.N, g.Kb, sw ? 128 : 256)) return cudaErrorInvalidValue;
    if (sw) {
        if (!make_map_u8(&mb2, g.b2, (int64_t)g.G * g.N, g.Kb, 128)) return cudaErrorInvalidValue;
    } else {
        mb2 = mb;
    }
    const int max_units = g.max_tiles * p.NB;
    if (max_units <= 0) return cudaGetLastError();
    const int grid = std::max(1, std::min(g.max_ctas > 0 ? std::min(num_sms, g.max_ctas) : num_sms, max_units));
    // staged y stores where tiles are full (many rows per expert), and in the
    // fused unpermutation (which writes out itself)
    const bool stg = !sw && g.many_rows && !g.cmb_out;
    cudaError_t e = sw ? launch_one<EPI_SWIGLU, false>(grid, ma, msh, mb, mb2, maf, mshf, p, stream)
                  : stg ? launch_one<EPI_PLAIN, true>(grid, ma, msh, mb, mb2, maf, mshf, p, stream)
                        : launch_one<EPI_PLAIN, false>(grid, ma, msh, mb, mb2, maf, mshf, p, stream);
    count_launches(1);
    return e;
}

}  // namespace moe
