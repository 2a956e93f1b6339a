// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>

#include "moe.h"

namespace moe {

constexpr int kRowTile = 128;      // rows of the grouped layout per GEMM tile
constexpr int kPermChunk = 1024;   // (t, j) pairs per permute chunk (largest size)

// Pairs per permute chunk for T*k pairs: 128 up to 16384 pairs (more, shorter
// chunks: the ranking walk is one warp per chunk), 1024 beyond (fewer
// per-chunk histograms for the scan to walk).
__host__ __device__ constexpr int perm_chunk(int64_t TK) { return TK <= 16384 ? 128 : kPermChunk; }

// Element kinds of the GEMM operands.
enum Elem : int { kF32 = 0, kBF16 = 1, kE4M3 = 2, kF16 = 3 };

// One grouped GEMM, C_g = A_g * B_g^T, over the groups of the expert-grouped
// row layout (or a single dense group).
//   rows of group g: offsets[g] .. offsets[g] + counts[g] - 1 of the output;
//   A row r of group g comes from a[r] (routed groups) or a_shared[r - offsets[g]]
//   (group == shared_group); B_g is b + g * N * K (and b2 likewise for the
//   SwiGLU "up" matrix).
struct GroupedGemm {
    int G;                       // groups
    int shared_group;            // group whose A rows come from a_shared (-1: none)
    const int32_t* offsets;      // [G+1] device (nullptr: single group of `rows` rows)
    const int32_t* tiles;        // [G+1] device prefix of ceil(rows/128) (nullptr with offsets)
    const int32_t* tiles2;       // [G+1] device prefix of ceil(rows/256), or nullptr
    int g_end;                   // grouped tensor-core kernel only: work on groups [0, g_end) (0: all G)
    int max_ctas;                // tensor-core kernels: at most this many CTAs (0: one per SM)
    int* sched;                  // tensor-core kernels: [2] zeroed device ints for dynamic unit order, or nullptr
    int max_tiles2;              // host bound on the total number of 256-row tiles
    int prefer_pairs;            // 1: run on CTA pairs (M=256) when a kernel for it exists
    int mcast;                   // bf16/fp16 tensor-core kernel: 1 = tile pairs (2-CTA clusters sharing
                                 // operand tiles by TMA multicast) where the shape allows them
    int narrow;                  // bf16/fp16 tensor-core kernel: 1 = tiles of <= 112 valid rows multiplied
                                 // transposed (weights as M, rows as N rounded up to 16)
    int rem_only;                // bf16 single-CTA kernel, split GEMMs: `tiles` counts the 128-row tiles
                                 // left after each group's whole 256-row pairs, which start its rows
    const int32_t* pair_active;  // CTA-pair kernel, split GEMMs: [1] device count of CTA pairs that work
                                 // (the rest exit at once); its units are whole 256-row pairs (tiles2)
    const int32_t* rem_order;    // with rem_only: [G] device group at each position of `tiles` (the
                                 // prefix runs over positions), or nullptr for group order
    int many_rows;               // FP8 kernel: groups hold many rows (prefill sizes): stage the down
                                 // GEMM's y stores through shared memory
    int rows;                    // single-group row count
    int max_tiles;               // host bound on the total number of row tiles
    int N;                       // output columns (features) of one group
    int Ka;                      // reduction length walked over A's row (= Kb, or 2*Kb for a hi/lo pair)
    int Kb;                      // row length of B; B's column for reduction index k is k % Kb
    int ldo;                     // output row stride in elements
    int out_pair;                // 1: bf16 output split as hi | lo halves (hi at col n, lo at col N+n)
    int a_rows, a_shared_rows;   // rows of the A tensors (tensor-map extents)
    int elem;                    // Elem of A (and of B when b_elem < 0)
    int b_elem;                  // Elem of B when it differs from A (SIMT only); 0 = same as A
    const void* a;               // [*, K]
    const void* a_shared;        // [*, K]
    const float* a_scale;        // FP8: [*, K/128] per-row group scales of a
    const float* a_shared_scale; // FP8: same for a_shared
    const void* b;               // [G, N, K]
    const void* b2;              // [G, N, K] (SwiGLU up) or nullptr
    const float* b_scale;        // FP8: [G, N/128, K/128]
    const float* b2_scale;
    void* out;                   // [*, N] (or [*, N] SwiGLU output)
    int out_elem;                // Elem of out (kE4M3: out_scale receives [*, N/128])
    float* out_scale;
    const float* bias;           // [N] added to the result (router) or nullptr
    int ksplit;                  // single group only: K split into this many slices (0/1: none);
                                 // slice s writes its partial product at out + s * split_stride
    int64_t split_stride;
    uint32_t* err;
    int64_t spin_ns;
    // Fused unpermutation (tensor-core plain epilogue of the shared expert's
    // down GEMM, single group, row t = token t): instead of storing y_s the
    // epilogue writes cmb_out[t] = y_s[t] + sum_j w[t,j] * y[cmb_inv[t*k+j]],
    // y_s rounded to out_elem first and the sum taken in fp32 in slot order,
    // exactly as the unpermute kernel does.  cmb_out == nullptr: off.
    void* cmb_out;               // [rows, N]: fp32 (cmb_out_f32) or bf16
    int cmb_out_f32;
    const int32_t* cmb_blob;     // [2, rows, k] routing blob (plane 1: fp32 weight bits)
    const int32_t* cmb_inv;      // [rows * k] grouped row of each (t, j)
    const void* cmb_y;           // routed expert outputs [rows * k, N], out_elem (fp16 or bf16)
    int cmb_k;
};

// Kernel launch accounting (moe_launch_count): every launcher adds the
// number of kernels it enqueued.
void count_launches(int n);

// One-time, per-device kernel set-up.  cudaFuncSetAttribute and occupancy
// queries act on the current device only, so their results are remembered
// per (key, current device), under a lock (launchers may run on several host
// threads and devices).
//   ensure_smem_attr: raise `func`'s dynamic shared-memory limit on the
//     current device to at least `bytes` (a no-op once it is that high).
//   per_device_value: `init` runs once per (key, device) with the lock held;
//     later calls on that device return the value it produced.
cudaError_t ensure_smem_attr(const void* func, int bytes);

// Kernels launched while a PdlScope(true) is alive on this host thread are
// launched as programmatic dependents of the previous kernel on their stream
// (moe_forward's main-stream chain): they may start their prologue while that
// kernel finishes and wait for it in pdl_wait_then_release().
extern thread_local bool t_pdl;
struct PdlScope {
    bool prev;
    explicit PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
    ~PdlScope() { t_pdl = prev; }
};
// Launch `kern` with the programmatic-dependency attribute when t_pdl is set
// (plus a cluster dimension when cluster > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    int n = 0;
    if (cluster > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = cluster;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    if (t_pdl) {
        at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}
cudaError_t per_device_value(const void* key, const std::function<cudaError_t(int*)>& init, int* value);

// Launchers (all asynchronous on `stream`; return cudaGetLastError()).
cudaError_t launch_gemm_simt(const GroupedGemm& g, cudaStream_t stream);
cudaError_t launch_gemm_tc(const GroupedGemm& g, int num_sms, cudaStream_t stream);
bool gemm_tc_supported(const GroupedGemm& g);
cudaError_t launch_gemm_tc2(const GroupedGemm& g, int num_sms, cudaStream_t stream);
bool gemm_tc2_supported(const GroupedGemm& g);
cudaError_t launch_gemm_fp8(const GroupedGemm& g, int num_sms, cudaStream_t stream);
bool gemm_fp8_supported(const GroupedGemm& g);

// Top-k over logits = sum_{s<S} part[s] (+ bias), summed in slice order;
// when S > 1 or bias is given the summed logits are written to logits_out.
// hist (nullable): also count the chosen experts into the permutation's
// per-chunk histograms ([chunks][E] with `chunk` pairs per chunk; the caller
// zeroes them first), which launch_permute_index then takes as given.
cudaError_t launch_topk(const float* part, int S, const float* bias, float* logits_out, int T, int E, int k,
                        int32_t* blob, uint32_t* err, cudaStream_t stream, int32_t* hist = nullptr, int chunk = 1);
int router_splits(int T, int E, int D, int num_sms);
cudaError_t launch_pack_words(const int32_t* blob, int64_t TK, int32_t* words, cudaStream_t stream);

// tiles2 (nullable): exclusive prefix of ceil(counts/256), the row-tile
// pairs of the two-CTA GEMM.
// hist_ready: the per-chunk histograms were already counted (by the top-k
// kernel) -- only meaningful where permute_uses_chunks().
// pairs (nullable): the split expert GEMMs' tile prefixes and CTA-pair counts
// ([2, E+2] + [2], see moe_ws_layout::pairs) for `clusters` CTA pairs at
// most; narrow_gu: the gate/up GEMM's ragged tiles run as narrow tails.
cudaError_t launch_permute_index(const int32_t* idx, int T, int E, int k, int32_t* hist, int32_t* counts,
                                 int32_t* offsets, int32_t* tiles, int32_t* tiles2, int32_t* inv, int32_t* src_tok,
                                 uint32_t* err, cudaStream_t stream, bool hist_ready = false, int32_t* pairs = nullptr,
                                 int clusters = 0, int narrow_gu = 0);
// Whether T*k pairs over E experts take the chunked permutation (per-chunk
// histograms in the workspace) rather than the single-block one.
bool permute_uses_chunks(int64_t TK, int E);
cudaError_t launch_scatter_rows(const void* x, int64_t row_bytes, const int32_t* inv, int T, int k, void* xp,
                                cudaStream_t stream);
cudaError_t launch_gather_rows(const void* x, int elem_bytes, int64_t row_bytes, const int32_t* src_tok,
                               int rows, void* xp, cudaStream_t stream);
// FP8 layer, scatter sizes: quantise x per row and 128 columns (as
// launch_quant_rows) straight into its k rows of xp / xp_scale (inv[t*k+j]).
cudaError_t launch_scatter_quant_rows(const void* x, int x_elem, int T, int cols, const int32_t* inv, int k,
                                      uint8_t* xp, float* xp_scale, cudaStream_t stream);
cudaError_t launch_quant_rows(const void* x, int x_elem, int rows, int cols, uint8_t* q, float* s,
                              cudaStream_t stream);
cudaError_t launch_quant_blocks(const float* w, int64_t groups, int rows, int cols, uint8_t* q, float* s,
                                cudaStream_t stream);
// bf16 -> fp16 (round to nearest even); values outside fp16's finite range
// record MOE_ERR_BOUNDS (their fp16 would not stand for the same weight).
cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, uint32_t* err, cudaStream_t stream);
cudaError_t launch_unpermute(const void* y, int y_elem, const int32_t* blob, const int32_t* inv, int T, int D,
                             int k, void* out, int out_elem, uint32_t* err, cudaStream_t stream);
cudaError_t launch_selftest_timeout(uint32_t* err, int64_t limit_ns, cudaStream_t stream);

}  // namespace moe
