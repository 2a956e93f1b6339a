// C ABI of libmoe: argument validation, workspace carving and the launch
// sequence of the routed-MoE layer.  Every entry point only enqueues work on
// the caller's stream; the only host synchronisation is in moe_check().
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace moe {
thread_local bool t_pdl = false;
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
std::mutex g_setup_mu;
std::map<std::pair<const void*, int>, int> g_smem_set;  // (kernel, device) -> bytes allowed
std::map<std::pair<const void*, int>, int> g_values;    // (key, device) -> value
}  // namespace

cudaError_t ensure_smem_attr(const void* func, int bytes) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    int& cur = g_smem_set[{func, dev}];
    if (cur >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) cur = bytes;
    return e;
}

cudaError_t per_device_value(const void* key, const std::function<cudaError_t(int*)>& init, int* value) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    auto it = g_values.find({key, dev});
    if (it != g_values.end()) {
        *value = it->second;
        return cudaSuccess;
    }
    int v = 0;
    e = init(&v);
    if (e != cudaSuccess) return e;
    g_values[{key, dev}] = v;
    *value = v;
    return cudaSuccess;
}
}  // namespace moe

struct moe_plan {
    moe_config cfg;
    int device;
    int num_sms;
    int64_t spin_ns;
    // moe_forward runs the shared expert on a second stream, forked from and
    // joined back into the caller's stream with these events
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    // split expert GEMMs: the permutation is done (the second stream starts
    // the single-CTA halves)
    cudaEvent_t ev_perm = nullptr;
};

namespace {

thread_local char g_detail[256];

moe_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_detail, sizeof(g_detail), "%.160s: %s", where, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}
moe_status arg_fail(moe_status s, const char* what) {
    snprintf(g_detail, sizeof(g_detail), "%s", what);
    return s;
}
#define MOE_CUDA(call)                                        \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
    } while (0)

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// bf16 layer: h as a bf16 hi/lo pair against the bf16 W_down (on request),
// else h as one fp16 against an fp16 copy of W_down.
bool hilo(const moe_config& c) { return c.dtype == MOE_BF16 && (c.flags & MOE_FLAG_DOWN_HILO); }
bool f16_down(const moe_config& c) { return c.dtype == MOE_BF16 && !(c.flags & MOE_FLAG_DOWN_HILO); }
// The split expert GEMMs can run for T tokens (bf16 layer at prefill sizes,
// not turned off): only then does the permutation write their tables.
bool split_sizes(const moe_config& c, int T) {
    if (c.flags & (MOE_FLAG_SPLIT_GEMM_OFF | MOE_FLAG_PAIR_CTA_ON | MOE_FLAG_FORCE_SIMT)) return false;
    return f16_down(c) && (int64_t)T * c.top_k >= 64LL * c.E;
}
// Expert outputs y: bf16 (FP8 layer), fp16 (bf16 layer, fp16 down path), else fp32.
int y_elem(const moe_config& c) {
    return c.dtype == MOE_FP8_E4M3_B128 ? moe::kBF16 : f16_down(c) ? moe::kF16 : moe::kF32;
}

// The first 256 bytes of the workspace: the error word (16 bytes), then from
// byte 64 one pair of unit-scheduling counters per GEMM launch of a forward
// (each rewound to zero by the kernel that used it).
constexpr size_t kErrBlock = 256;
enum SchedSlot : int { kSchedRouter = 0, kSchedGateup = 1, kSchedDown = 2, kSchedSharedGateup = 3, kSchedSharedDown = 4 };

int act_bytes(int dtype) { return dtype == MOE_F32 ? 4 : (dtype == MOE_BF16 ? 2 : 1); }
int act_elem(int dtype) { return dtype == MOE_F32 ? moe::kF32 : (dtype == MOE_BF16 ? moe::kBF16 : moe::kE4M3); }
int in_elem(int dtype) { return dtype == MOE_F32 ? moe::kF32 : moe::kBF16; }  // x and router

int route_splits(const moe_config& c, int T, int num_sms) {
    return c.dtype == MOE_F32 ? 1 : moe::router_splits(T, c.E, c.D, num_sms);
}

void layout(const moe_config& c, int num_sms, int T, moe_ws_layout* L) {
    const int64_t TK = (int64_t)T * c.top_k, R = TK + T;
    const bool fp8 = c.dtype == MOE_FP8_E4M3_B128;
    const int ab = act_bytes(c.dtype);
    const int64_t nch = moe::cdiv(TK, moe::perm_chunk(TK));
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += up256(bytes); return at; };
    memset(L, 0, sizeof(*L));
    L->err = take(kErrBlock);
    L->logits = take((size_t)T * c.E * 4);
    L->blob = take((size_t)2 * TK * 4);
    L->counts = take((size_t)(c.E + 1) * 4);
    L->offsets = take((size_t)(c.E + 2) * 4);
    L->tiles = take((size_t)(c.E + 2) * 4);
    L->inv = take((size_t)TK * 4);
    L->src_tok = take((size_t)R * 4);
    L->hist = take((size_t)nch * c.E * 4);
    L->xq = fp8 ? take((size_t)T * c.D) : 0;
    L->xq_scale = fp8 ? take((size_t)T * (c.D / 128) * 4) : 0;
    L->xp = take((size_t)TK * c.D * ab);
    L->xp_scale = fp8 ? take((size_t)TK * (c.D / 128) * 4) : 0;
    // bf16 layer: h in fp16 ([R, I]), or as a bf16 hi/lo pair ([R, 2I]) under
    // MOE_FLAG_DOWN_HILO; a single bf16 rounding of h alone would cost about
    // 1e-2 of the output rms.
    L->h = take((size_t)R * c.I * (hilo(c) ? 4 : ab));
    L->h_scale = fp8 ? take((size_t)R * (c.I / 128) * 4) : 0;
    // y: fp16 for the bf16 layer, bf16 for the FP8 layer, else fp32 (a bf16 y
    // in the bf16 layer would cost about 1.3e-2 of the output rms).
    L->y = take((size_t)R * c.D * (y_elem(c) == moe::kF32 ? 4 : 2));
    const int S = route_splits(c, T, num_sms);
    L->logits_part = S > 1 ? take((size_t)S * T * c.E * 4) : 0;
    L->tiles2 = take((size_t)(c.E + 2) * 4);
    L->pairs = take((size_t)(3 * (c.E + 2) + 2) * 4);
    L->total = o;
}

struct Ws {
    moe_ws_layout L;
    char* base;
    int* sched(int slot) { return (int*)(base + L.err + 64) + 2 * slot; }
    template <typename T> T* at(size_t off) const { return (T*)(base + off); }
};

moe_status check_call(const moe_plan* p, int32_t T, void* ws, size_t ws_bytes, Ws* out) {
    if (!p) return arg_fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (T < 1 || T > p->cfg.T_max) return arg_fail(MOE_ERR_INVALID_ARG, "T outside [1, T_max]");
    if (!ws || !aligned(ws, 256)) return arg_fail(MOE_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    layout(p->cfg, p->num_sms, T, &out->L);
    if (ws_bytes < out->L.total) return arg_fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_workspace_size()");
    out->base = (char*)ws;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != p->device)
        return arg_fail(MOE_ERR_INVALID_ARG, "current CUDA device is not the plan's device");
    return MOE_OK;
}

bool ptr_ok(const void* q) { return q != nullptr && aligned(q, 16); }

moe_status check_weights(const moe_plan* p, const moe_weights* w, bool router, bool experts) {
    if (!w) return arg_fail(MOE_ERR_INVALID_ARG, "weights is NULL");
    if (router) {
        if (!ptr_ok(w->w_router)) return arg_fail(MOE_ERR_INVALID_ARG, "w_router NULL or misaligned");
        if (p->cfg.has_router_bias && !ptr_ok(w->b_router))
            return arg_fail(MOE_ERR_INVALID_ARG, "b_router NULL or misaligned");
    }
    if (experts) {
        if (!ptr_ok(w->w_gate) || !ptr_ok(w->w_up))
            return arg_fail(MOE_ERR_INVALID_ARG, "expert weight NULL or misaligned");
        // the bf16 layer's tensor-core down GEMM reads only the fp16 copy, so
        // there the bf16 w_down may be NULL (its memory freed by the caller)
        const bool f16_only = f16_down(p->cfg) && !(p->cfg.flags & MOE_FLAG_FORCE_SIMT);
        if (f16_only && !ptr_ok(w->w_down_f16))
            return arg_fail(MOE_ERR_INVALID_ARG, "w_down_f16 NULL or misaligned (see moe_convert_down_weights)");
        if (f16_only ? (w->w_down && !aligned(w->w_down, 16)) : !ptr_ok(w->w_down))
            return arg_fail(MOE_ERR_INVALID_ARG, "w_down NULL or misaligned");
        if (p->cfg.dtype == MOE_FP8_E4M3_B128 && (!ptr_ok(w->s_gate) || !ptr_ok(w->s_up) || !ptr_ok(w->s_down)))
            return arg_fail(MOE_ERR_INVALID_ARG, "FP8 block scales NULL or misaligned");
    }
    return MOE_OK;
}

bool use_tc(const moe_plan* p, const moe::GroupedGemm& g) {
    if (p->cfg.flags & MOE_FLAG_FORCE_SIMT) return false;
    return moe::gemm_tc_supported(g);
}

moe_status run_gemm(const moe_plan* p, const moe::GroupedGemm& g, cudaStream_t s, const char* what) {
    if (g.elem == moe::kE4M3) {
        if (!moe::gemm_fp8_supported(g)) return arg_fail(MOE_ERR_UNSUPPORTED, "FP8 GEMM shape without a kernel");
        cudaError_t e = moe::launch_gemm_fp8(g, p->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e, what);
        return MOE_OK;
    }
    if (use_tc(p, g)) {
        if (g.prefer_pairs && moe::gemm_tc2_supported(g)) MOE_CUDA(moe::launch_gemm_tc2(g, p->num_sms, s));
        else MOE_CUDA(moe::launch_gemm_tc(g, p->num_sms, s));
        return MOE_OK;
    }
    if (g.elem == moe::kE4M3) return arg_fail(MOE_ERR_UNSUPPORTED, "FP8 GEMM shape without a tensor-core kernel");
    cudaError_t e = moe::launch_gemm_simt(g, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return MOE_OK;
}

// CTA pairs (256-row tiles) halve each CTA's operand traffic but pad every
// group to 256 rows: under skewed routing at T=8192 that is 31 % padded MMA
// rows against 18 % for 128-row tiles, and single CTAs measure faster.  So
// pairs run only on request.
int prefer_pairs(const moe_plan* p, int T) {
    (void)T;
    if (p->cfg.flags & MOE_FLAG_PAIR_CTA_OFF) return 0;
    return (p->cfg.flags & MOE_FLAG_PAIR_CTA_ON) ? 1 : 0;
}

// Tile pairs (2-CTA clusters sharing operand tiles) pay where groups hold
// several row tiles; at decode sizes the GEMMs stream weights from HBM and the
// clusters only couple the CTAs' progress.
int prefer_mcast(const moe_plan* p, int T) {
    const uint32_t f = p->cfg.flags;
    if (f & MOE_FLAG_MCAST_OFF) return 0;
    if (f & MOE_FLAG_MCAST_ON) return 1;
    return (int64_t)T * p->cfg.top_k >= 64 * (int64_t)p->cfg.E ? 1 : 0;
}

// Narrow tails save tensor time on ragged tiles; measured at T=8192 they
// take the gate/up GEMM from 1.264 to 1.247 ms, while in the down GEMM (y
// stored transposed, 2 bytes at a time) and at decode sizes they cost more
// than they save.
int prefer_narrow(const moe_plan* p, int T, bool gateup) {
    const uint32_t f = p->cfg.flags;
    if (f & MOE_FLAG_NARROW_TAILS_OFF) return 0;
    if (f & MOE_FLAG_NARROW_TAILS_ON) return 1;
    // the CTA-pair kernel stages its transposed stores: narrow tails in both GEMMs
    if (prefer_pairs(p, T)) return 1;
    return gateup && prefer_mcast(p, T) ? 1 : 0;
}

int grouped_max_tiles2(const moe_config& c, int T) {
    const int64_t R = (int64_t)T * (c.top_k + 1);
    return (int)(R / (2 * moe::kRowTile) + c.E + 2);
}

int grouped_max_tiles(const moe_config& c, int T) {
    const int64_t R = (int64_t)T * (c.top_k + 1);
    return (int)(R / moe::kRowTile + c.E + 2);
}

}  // namespace

extern "C" {

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_BOUNDS: return "device index check failed";
        case MOE_ERR_NONFINITE: return "non-finite router logit";
    }
    return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail; }

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

const char* moe_build_info(void) { return "libmoe sm_103a: tcgen05+TMA grouped GEMM, SIMT grouped GEMM, route/permute/unpermute"; }

moe_status moe_plan_create(const moe_config* cfg, int device, moe_plan** out) {
    if (!out) return arg_fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg) return arg_fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
    const moe_config& c = *cfg;
    if (c.dtype < MOE_F32 || c.dtype > MOE_FP8_E4M3_B128) return arg_fail(MOE_ERR_UNSUPPORTED, "dtype");
    if (c.out_dtype != MOE_F32 && c.out_dtype != MOE_BF16) return arg_fail(MOE_ERR_UNSUPPORTED, "out_dtype");
    if (c.E < 1 || c.E > 1024) return arg_fail(MOE_ERR_UNSUPPORTED, "E outside [1, 1024]");
    if (c.top_k < 1 || c.top_k > std::min(c.E, 32)) return arg_fail(MOE_ERR_UNSUPPORTED, "top_k outside [1, min(E,32)]");
    if (c.T_max < 1 || c.T_max > (1 << 20)) return arg_fail(MOE_ERR_UNSUPPORTED, "T_max outside [1, 2^20]");
    if ((int64_t)c.T_max * (c.top_k + 1) >= (int64_t)1 << 31) return arg_fail(MOE_ERR_UNSUPPORTED, "T_max*(top_k+1) >= 2^31");
    const int q = (c.dtype == MOE_F32) ? 64 : 128;
    if (c.D < q || c.D % q || c.I < q || c.I % q) return arg_fail(MOE_ERR_UNSUPPORTED, "D and I must be multiples of 128 (64 for fp32)");
    if (c.D > 65536 || c.I > 65536) return arg_fail(MOE_ERR_UNSUPPORTED, "D or I above 65536");
    if (c.dtype == MOE_FP8_E4M3_B128 && c.D % 256)  // the FP8 down GEMM's units are 256 output features wide
        return arg_fail(MOE_ERR_UNSUPPORTED, "the FP8 layer needs D a multiple of 256");
    if (c.spin_limit_ns < 0) return arg_fail(MOE_ERR_INVALID_ARG, "spin_limit_ns < 0");
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return arg_fail(MOE_ERR_INVALID_ARG, "no such CUDA device");
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return arg_fail(MOE_ERR_CUDA, "device query failed");
    moe_plan* p = new moe_plan;
    p->cfg = c;
    p->device = device;
    p->num_sms = sms;
    p->spin_ns = c.spin_limit_ns ? c.spin_limit_ns : 2000000000LL;
    int prev = 0;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_perm, cudaEventDisableTiming) != cudaSuccess) {
        moe_plan_destroy(p);
        cudaSetDevice(prev);
        return arg_fail(MOE_ERR_CUDA, "stream or event creation failed");
    }
    cudaSetDevice(prev);
    *out = p;
    return MOE_OK;
}

void moe_plan_destroy(moe_plan* p) {
    if (!p) return;
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->ev_perm) cudaEventDestroy(p->ev_perm);
    if (p->side) cudaStreamDestroy(p->side);
    delete p;
}

const moe_config* moe_plan_config(const moe_plan* p) { return p ? &p->cfg : nullptr; }

moe_status moe_workspace_layout(const moe_plan* p, int32_t T, moe_ws_layout* out) {
    if (!p || !out) return arg_fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (T < 1 || T > p->cfg.T_max) return arg_fail(MOE_ERR_INVALID_ARG, "T outside [1, T_max]");
    layout(p->cfg, p->num_sms, T, out);
    return MOE_OK;
}

moe_status moe_workspace_size(const moe_plan* p, int32_t T, size_t* bytes) {
    if (!bytes) return arg_fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    moe_ws_layout L;
    moe_status s = moe_workspace_layout(p, T, &L);
    if (s == MOE_OK) *bytes = L.total;
    return s;
}

moe_status moe_workspace_init(const moe_plan* p, void* ws, size_t ws_bytes, void* stream) {
    if (!p || !ws || !aligned(ws, 256) || ws_bytes < 256) return arg_fail(MOE_ERR_INVALID_ARG, "workspace");
    MOE_CUDA(cudaMemsetAsync(ws, 0, kErrBlock, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_quantize_weights(const moe_plan* p, const float* w, int64_t groups, int32_t rows, int32_t cols,
                                uint8_t* q, float* s, void* stream) {
    if (!p) return arg_fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (!ptr_ok(w) || !ptr_ok(q) || !ptr_ok(s)) return arg_fail(MOE_ERR_INVALID_ARG, "NULL or misaligned pointer");
    if (groups < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128)
        return arg_fail(MOE_ERR_UNSUPPORTED, "rows and cols must be positive multiples of 128");
    MOE_CUDA(moe::launch_quant_blocks(w, groups, rows, cols, q, s, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_topk(const moe_plan* p, int32_t T, void* ws, size_t ws_bytes, void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    const moe_config& c = p->cfg;
    MOE_CUDA(moe::launch_topk(W.at<float>(W.L.logits), 1, nullptr, nullptr, T, c.E, c.top_k,
                              W.at<int32_t>(W.L.blob), W.at<uint32_t>(W.L.err), (cudaStream_t)stream));
    return MOE_OK;
}

namespace {
// moe_forward's route: with fused_hist the top-k kernel also counts the
// permutation's per-chunk expert histograms (zeroed here first), so that the
// permutation skips its own histogram pass.
moe_status route_impl(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, Ws& W, void* stream,
                      bool fused_hist, bool pdl = false);
}  // namespace

moe_status moe_route(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, void* ws, size_t ws_bytes,
                     void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if ((st = check_weights(p, w, true, false)) != MOE_OK) return st;
    if (!ptr_ok(x)) return arg_fail(MOE_ERR_INVALID_ARG, "x NULL or misaligned");
    return route_impl(p, w, x, T, W, stream, false);
}

namespace {
bool fuse_topk_hist(const moe_plan* p, int32_t T) {
    return !(p->cfg.flags & MOE_FLAG_TOPK_HIST_OFF) && moe::permute_uses_chunks((int64_t)T * p->cfg.top_k, p->cfg.E);
}

// Zero the per-chunk histograms the fused top-k counts into.  moe_forward
// does this before it forks the shared-expert stream, so that the router
// GEMM is still the first kernel queued after the fork (a memset there let
// the shared GEMMs take the SMs first: 2.30 vs 2.25 ms at T=8192).
cudaError_t zero_topk_hist(const moe_plan* p, int32_t T, Ws& W, cudaStream_t s) {
    const int64_t TK = (int64_t)T * p->cfg.top_k;
    return cudaMemsetAsync(W.at<int32_t>(W.L.hist), 0, (size_t)moe::cdiv(TK, moe::perm_chunk(TK)) * p->cfg.E * 4, s);
}

moe_status route_impl(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, Ws& W, void* stream,
                      bool fused_hist, bool pdl) {
    moe_status st;
    const moe_config& c = p->cfg;
    moe::GroupedGemm g = {};
    g.G = 1;
    g.shared_group = -1;
    g.rows = T;
    g.max_tiles = (int)moe::cdiv(T, moe::kRowTile);
    g.N = c.E;
    g.Ka = g.Kb = c.D;
    g.ldo = c.E;
    g.a_rows = T;
    g.elem = in_elem(c.dtype);
    g.a = x;
    g.b = w->w_router;
    g.out = W.at<float>(W.L.logits);
    g.out_elem = moe::kF32;
    g.bias = c.has_router_bias ? w->b_router : nullptr;
    g.err = W.at<uint32_t>(W.L.err);
    g.sched = W.sched(kSchedRouter);
    g.spin_ns = p->spin_ns;
    // Small T: split K over several CTAs; the top-k kernel then adds the
    // slices in order (and the bias) and writes the logits.
    const int S = use_tc(p, g) ? route_splits(c, T, p->num_sms) : 1;
    if (S > 1) {
        g.ksplit = S;
        g.split_stride = (int64_t)T * c.E;
        g.out = W.at<float>(W.L.logits_part);
        g.bias = nullptr;
    }
    int32_t* hist = nullptr;
    int chunk = 1;
    if (fused_hist) {  // the caller zeroed the histograms (zero_topk_hist)
        chunk = moe::perm_chunk((int64_t)T * c.top_k);
        hist = W.at<int32_t>(W.L.hist);
    }
    if ((st = run_gemm(p, g, (cudaStream_t)stream, "router GEMM")) != MOE_OK) return st;
    moe::PdlScope scope(pdl);  // the top-k follows the router GEMM on this stream
    if (S > 1)
        MOE_CUDA(moe::launch_topk(W.at<float>(W.L.logits_part), S, c.has_router_bias ? w->b_router : nullptr,
                                  W.at<float>(W.L.logits), T, c.E, c.top_k, W.at<int32_t>(W.L.blob),
                                  W.at<uint32_t>(W.L.err), (cudaStream_t)stream, hist, chunk));
    else
        MOE_CUDA(moe::launch_topk(W.at<float>(W.L.logits), 1, nullptr, nullptr, T, c.E, c.top_k,
                                  W.at<int32_t>(W.L.blob), W.at<uint32_t>(W.L.err), (cudaStream_t)stream, hist,
                                  chunk));
    return MOE_OK;
}

// Permuted copy of x: from T >= 1024 tokens one warp per token reads its row
// once and writes its top_k copies (x leaves DRAM once); below that there
// are too few tokens to fill the GPU and one warp per output row gathers.
bool scatter_by_token(int32_t T) { return T >= 1024; }
// FP8 layer: quantise x on the way into xp (one kernel) where the scatter
// runs and a row fits the kernel's shared-memory copy
bool fused_quant_scatter(const moe_config& c, int32_t T) { return scatter_by_token(T) && c.D <= 4096; }

// quant_x: the FP8 layer quantises x into xq here (false when the caller
// already did).
// hist_ready: route_impl already counted the per-chunk histograms.
moe_status permute_impl(const moe_plan* p, const void* x, int32_t T, Ws& W, cudaStream_t s, bool quant_x,
                        bool hist_ready = false) {
    const moe_config& c = p->cfg;
    const int TK = T * c.top_k;
    MOE_CUDA(moe::launch_permute_index(W.at<int32_t>(W.L.blob), T, c.E, c.top_k, W.at<int32_t>(W.L.hist),
                                       W.at<int32_t>(W.L.counts), W.at<int32_t>(W.L.offsets),
                                       W.at<int32_t>(W.L.tiles), W.at<int32_t>(W.L.tiles2), W.at<int32_t>(W.L.inv),
                                       W.at<int32_t>(W.L.src_tok),
                                       W.at<uint32_t>(W.L.err), s, hist_ready,
                                       split_sizes(c, T) ? W.at<int32_t>(W.L.pairs) : nullptr,
                                       std::max(1, p->num_sms / 2), prefer_narrow(p, T, true)));
    if (c.dtype == MOE_FP8_E4M3_B128) {
        // xq (x quantised) is the shared expert's A operand; the routed rows
        // are quantised from x on the way into xp at scatter sizes
        if (quant_x)
            MOE_CUDA(moe::launch_quant_rows(x, moe::kBF16, T, c.D, W.at<uint8_t>(W.L.xq), W.at<float>(W.L.xq_scale), s));
        if (fused_quant_scatter(c, T)) {
            MOE_CUDA(moe::launch_scatter_quant_rows(x, moe::kBF16, T, c.D, W.at<int32_t>(W.L.inv), c.top_k,
                                                    W.at<uint8_t>(W.L.xp), W.at<float>(W.L.xp_scale), s));
        } else {
            if (scatter_by_token(T))
                MOE_CUDA(moe::launch_scatter_rows(W.at<uint8_t>(W.L.xq), c.D, W.at<int32_t>(W.L.inv), T, c.top_k,
                                                  W.at<uint8_t>(W.L.xp), s));
            else
                MOE_CUDA(moe::launch_gather_rows(W.at<uint8_t>(W.L.xq), 1, c.D, W.at<int32_t>(W.L.src_tok), TK,
                                                 W.at<uint8_t>(W.L.xp), s));
            MOE_CUDA(moe::launch_gather_rows(W.at<float>(W.L.xq_scale), 4, (int64_t)(c.D / 128) * 4,
                                             W.at<int32_t>(W.L.src_tok), TK, W.at<float>(W.L.xp_scale), s));
        }
    } else {
        const int eb = act_bytes(c.dtype);
        if (scatter_by_token(T))
            MOE_CUDA(moe::launch_scatter_rows(x, (int64_t)c.D * eb, W.at<int32_t>(W.L.inv), T, c.top_k,
                                              W.at<char>(W.L.xp), s));
        else
            MOE_CUDA(moe::launch_gather_rows(x, eb, (int64_t)c.D * eb, W.at<int32_t>(W.L.src_tok), TK,
                                             W.at<char>(W.L.xp), s));
    }
    return MOE_OK;
}
}  // namespace

moe_status moe_permute(const moe_plan* p, const void* x, int32_t T, void* ws, size_t ws_bytes, void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if (!ptr_ok(x)) return arg_fail(MOE_ERR_INVALID_ARG, "x NULL or misaligned");
    return permute_impl(p, x, T, W, (cudaStream_t)stream, true);
}

namespace {

moe::GroupedGemm gateup_gemm(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, Ws& W) {
    const moe_config& c = p->cfg;
    const bool fp8 = c.dtype == MOE_FP8_E4M3_B128;
    moe::GroupedGemm g = {};
    g.G = c.E + 1;
    g.shared_group = c.E;
    g.offsets = W.at<int32_t>(W.L.offsets);
    g.tiles = W.at<int32_t>(W.L.tiles);
    g.max_tiles = grouped_max_tiles(c, T);
    g.tiles2 = W.at<int32_t>(W.L.tiles2);
    g.max_tiles2 = grouped_max_tiles2(c, T);
    g.prefer_pairs = prefer_pairs(p, T);
    g.mcast = prefer_mcast(p, T);
    g.narrow = prefer_narrow(p, T, true);
    g.N = c.I;
    g.Ka = g.Kb = c.D;
    g.out_pair = hilo(c);
    g.ldo = g.out_pair ? 2 * c.I : c.I;
    g.a_rows = T * c.top_k;
    g.a_shared_rows = T;
    g.elem = act_elem(c.dtype);
    g.a = W.at<void>(W.L.xp);
    g.a_shared = fp8 ? (const void*)W.at<uint8_t>(W.L.xq) : x;
    g.a_scale = fp8 ? W.at<float>(W.L.xp_scale) : nullptr;
    g.a_shared_scale = fp8 ? W.at<float>(W.L.xq_scale) : nullptr;
    g.b = w->w_gate;
    g.b2 = w->w_up;
    g.b_scale = w->s_gate;
    g.b2_scale = w->s_up;
    g.out = W.at<void>(W.L.h);
    g.out_elem = f16_down(c) ? moe::kF16 : act_elem(c.dtype);
    g.out_scale = fp8 ? W.at<float>(W.L.h_scale) : nullptr;
    g.err = W.at<uint32_t>(W.L.err);
    g.sched = W.sched(kSchedGateup);
    g.spin_ns = p->spin_ns;
    return g;
}

moe::GroupedGemm down_gemm(const moe_plan* p, const moe_weights* w, int32_t T, Ws& W) {
    const moe_config& c = p->cfg;
    const bool fp8 = c.dtype == MOE_FP8_E4M3_B128;
    moe::GroupedGemm g = {};
    g.G = c.E + 1;
    g.shared_group = -1;
    g.offsets = W.at<int32_t>(W.L.offsets);
    g.tiles = W.at<int32_t>(W.L.tiles);
    g.max_tiles = grouped_max_tiles(c, T);
    g.tiles2 = W.at<int32_t>(W.L.tiles2);
    g.max_tiles2 = grouped_max_tiles2(c, T);
    g.prefer_pairs = prefer_pairs(p, T);
    g.mcast = prefer_mcast(p, T);
    g.narrow = prefer_narrow(p, T, false);
    g.many_rows = (int64_t)T * c.top_k >= 64 * (int64_t)c.E;
    g.N = c.D;
    g.Kb = c.I;
    g.Ka = hilo(c) ? 2 * c.I : c.I;  // the hi/lo pair walks W_down twice
    g.ldo = c.D;
    g.a_rows = T * (c.top_k + 1);
    g.elem = act_elem(c.dtype);
    g.a = W.at<void>(W.L.h);
    g.a_scale = fp8 ? W.at<float>(W.L.h_scale) : nullptr;
    g.b = w->w_down;
    if (f16_down(c)) {
        g.elem = moe::kF16;  // fp16 h
        if (c.flags & MOE_FLAG_FORCE_SIMT) g.b_elem = moe::kBF16;  // CUDA cores read the bf16 W_down
        else g.b = w->w_down_f16;                                   // tensor cores: one type for A and B
    }
    g.b_scale = w->s_down;
    g.out = W.at<void>(W.L.y);
    g.out_elem = y_elem(c);
    g.err = W.at<uint32_t>(W.L.err);
    // dynamic unit order measured slower for the bf16 down GEMM (0.80 vs
    // 0.78 ms at T=8192), faster for the FP8 one (1.42 vs 1.43 ms) and for
    // every gate/up GEMM
    g.sched = W.sched(kSchedDown);  // (tile pairs at prefill take the static order)
    g.spin_ns = p->spin_ns;
    return g;
}

int elem_bytes(int e) { return e == moe::kF32 ? 4 : e == moe::kE4M3 ? 1 : 2; }

// The shared expert alone, as a dense GEMM over its T rows (which sit after
// the T*k routed rows of the grouped layout).  Its A comes from x (gate/up)
// or from the shared rows of h (down); its B is group E of the weights.
moe::GroupedGemm shared_only(const moe::GroupedGemm& full, const moe_config& c, int32_t T, bool gateup,
                             const void* x, const float* x_scale) {
    moe::GroupedGemm g = full;
    const int64_t TK = (int64_t)T * c.top_k;
    g.G = 1;
    g.shared_group = -1;
    g.offsets = g.tiles = g.tiles2 = nullptr;
    g.prefer_pairs = 0;
    g.rows = T;
    g.max_tiles = (int)moe::cdiv(T, moe::kRowTile);
    g.a_rows = T;
    g.a_shared = nullptr;
    g.a_shared_rows = 0;
    const int eb = elem_bytes(g.elem);
    const int bb = elem_bytes(g.b_elem > 0 ? g.b_elem : g.elem);
    if (gateup) {
        g.a = x;
        g.a_scale = x_scale;
    } else {
        g.a = (const char*)full.a + TK * g.Ka * eb;
        if (full.a_scale) g.a_scale = full.a_scale + TK * (g.Ka / 128);
    }
    g.a_shared_scale = nullptr;
    const int64_t group = (int64_t)g.N * g.Kb * bb;
    g.b = (const char*)full.b + c.E * group;
    if (g.b2) g.b2 = (const char*)full.b2 + c.E * group;
    const int64_t sgroup = (int64_t)(g.N / 128) * (g.Kb / 128);  // FP8 block scales of one group
    if (full.b_scale) g.b_scale = full.b_scale + c.E * sgroup;
    if (full.b2_scale) g.b2_scale = full.b2_scale + c.E * sgroup;
    g.out = (char*)full.out + TK * g.ldo * elem_bytes(g.out_elem);
    if (full.out_scale) g.out_scale = full.out_scale + TK * (g.N / 128);
    return g;
}

// Split expert GEMMs (see moe_forward): the bf16 layer at prefill sizes,
// unless the caller asked for the plain CTA-pair kernel or turned the split
// off.  Fills the two launches of each GEMM: gp on CTA pairs over the whole
// 256-row pairs (pairs[0..E+1]), as many pairs as the permutation counted
// (pairs[2(E+2) + i]); gr on single CTAs over the rest of each group
// (pairs[E+2..], in the group order at pairs[2(E+2)+2..] that keeps it near
// the pair launch's progress), drawing units from the shared expert's
// counters (its GEMMs are done by then on the same stream).
bool split_wanted(const moe_plan* p, int T, Ws& W, const moe::GroupedGemm& gu, const moe::GroupedGemm& dn,
                  moe::GroupedGemm* gp, moe::GroupedGemm* gr) {
    const moe_config& c = p->cfg;
    if (!split_sizes(c, T)) return false;
    int32_t* pairs = W.at<int32_t>(W.L.pairs);
    for (int i = 0; i < 2; ++i) {
        const moe::GroupedGemm& base = i == 0 ? gu : dn;
        gp[i] = base;
        gp[i].prefer_pairs = 1;
        gp[i].tiles2 = pairs;
        gp[i].narrow = 0;
        gp[i].pair_active = pairs + 2 * (c.E + 2) + i;
        gr[i] = base;
        gr[i].tiles = pairs + (c.E + 2);
        gr[i].rem_only = 1;
        gr[i].rem_order = pairs + 2 * (c.E + 2) + 2;
        gr[i].mcast = 0;
        gr[i].prefer_pairs = 0;
        gr[i].sched = W.sched(i == 0 ? kSchedSharedGateup : kSchedSharedDown);
        if (!moe::gemm_tc2_supported(gp[i]) || !moe::gemm_tc_supported(gr[i])) return false;
    }
    return true;
}

// A stage entry point's expert GEMM (all groups, the shared one included),
// split as in moe_forward where that applies: the whole 256-row pairs on the
// caller's stream, the rest on the plan's second stream, joined back before
// returning.  which: 0 gate/up, 1 down.
moe_status run_stage_gemm(const moe_plan* p, const moe::GroupedGemm& g, int which, int32_t T, Ws& W, cudaStream_t s,
                          const char* what) {
    moe::GroupedGemm gp[2], gr[2];
    if (!split_wanted(p, T, W, g, g, gp, gr)) return run_gemm(p, g, s, what);
    MOE_CUDA(cudaEventRecord(p->ev_fork, s));
    MOE_CUDA(cudaStreamWaitEvent(p->side, p->ev_fork, 0));
    const moe_status st = run_gemm(p, gp[which], s, what);
    const moe_status st2 = run_gemm(p, gr[which], p->side, what);
    MOE_CUDA(cudaEventRecord(p->ev_join, p->side));
    MOE_CUDA(cudaStreamWaitEvent(s, p->ev_join, 0));  // joined even after an error (stream capture)
    return st != MOE_OK ? st : st2;
}

}  // namespace

moe_status moe_gemm_gateup(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, void* ws,
                           size_t ws_bytes, void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if ((st = check_weights(p, w, false, true)) != MOE_OK) return st;
    if (!ptr_ok(x)) return arg_fail(MOE_ERR_INVALID_ARG, "x NULL or misaligned");
    return run_stage_gemm(p, gateup_gemm(p, w, x, T, W), 0, T, W, (cudaStream_t)stream, "gate/up GEMM");
}

moe_status moe_gemm_down(const moe_plan* p, const moe_weights* w, int32_t T, void* ws, size_t ws_bytes,
                         void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if ((st = check_weights(p, w, false, true)) != MOE_OK) return st;
    return run_stage_gemm(p, down_gemm(p, w, T, W), 1, T, W, (cudaStream_t)stream, "down GEMM");
}

moe_status moe_unpermute(const moe_plan* p, int32_t T, void* out, void* ws, size_t ws_bytes, void* stream) {
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if (!ptr_ok(out)) return arg_fail(MOE_ERR_INVALID_ARG, "out NULL or misaligned");
    const moe_config& c = p->cfg;
    MOE_CUDA(moe::launch_unpermute(W.at<void>(W.L.y), y_elem(c),
                                   W.at<int32_t>(W.L.blob), W.at<int32_t>(W.L.inv), T, c.D, c.top_k, out,
                                   c.out_dtype == MOE_F32 ? moe::kF32 : moe::kBF16, W.at<uint32_t>(W.L.err),
                                   (cudaStream_t)stream));
    return MOE_OK;
}

namespace {
// moe_forward's optional copies of the routing blob and the logits.
moe_status copy_routing_out(const moe_plan* p, Ws& W, int32_t T, int32_t* blob_out, float* logits_out,
                            cudaStream_t s) {
    const moe_config& c = p->cfg;
    if (blob_out)
        MOE_CUDA(cudaMemcpyAsync(blob_out, W.at<int32_t>(W.L.blob), (size_t)2 * T * c.top_k * 4,
                                 cudaMemcpyDeviceToDevice, s));
    if (logits_out)
        MOE_CUDA(cudaMemcpyAsync(logits_out, W.at<float>(W.L.logits), (size_t)T * c.E * 4, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}
}  // namespace

moe_status moe_forward(const moe_plan* p, const moe_weights* w, const void* x, int32_t T, void* out,
                       int32_t* blob_out, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
    if (p && T == 0) return MOE_OK;  // an empty batch: nothing to read, write or launch
    Ws W;
    moe_status st = check_call(p, T, ws, ws_bytes, &W);
    if (st != MOE_OK) return st;
    if ((st = check_weights(p, w, true, true)) != MOE_OK) return st;
    if (!ptr_ok(x) || !ptr_ok(out)) return arg_fail(MOE_ERR_INVALID_ARG, "x or out NULL or misaligned");
    if ((blob_out && !aligned(blob_out, 16)) || (logits_out && !aligned(logits_out, 16)))
        return arg_fail(MOE_ERR_INVALID_ARG, "blob_out or logits_out misaligned");
    cudaStream_t s = (cudaStream_t)stream;
    const moe_config& cf = p->cfg;
    MOE_CUDA(cudaMemsetAsync(ws, 0, kErrBlock, s));
    const bool fh = fuse_topk_hist(p, T);
    if (fh) MOE_CUDA(zero_topk_hist(p, T, W, s));
    moe::GroupedGemm gu = gateup_gemm(p, w, x, T, W), dn = down_gemm(p, w, T, W);
    const bool fp8 = cf.dtype == MOE_FP8_E4M3_B128;
    moe::GroupedGemm sgu = shared_only(gu, cf, T, true, fp8 ? (const void*)W.at<uint8_t>(W.L.xq) : x,
                                       fp8 ? W.at<float>(W.L.xq_scale) : nullptr);
    moe::GroupedGemm sdn = shared_only(dn, cf, T, false, nullptr, nullptr);
    // The shared expert needs no routing: on the tensor-core path its two
    // GEMMs run on the plan's second stream while the router, top-k and
    // permutation run here; the routed GEMMs then skip the shared group.
    // (FP8: the shared GEMM reads xq, x quantised per row; see below.)
    const bool overlap =
        !(cf.flags & MOE_FLAG_FORCE_SIMT) &&
        (fp8 ? (moe::gemm_fp8_supported(gu) && moe::gemm_fp8_supported(dn) && moe::gemm_fp8_supported(sgu) &&
                moe::gemm_fp8_supported(sdn))
             : (cf.dtype == MOE_BF16 && moe::gemm_tc_supported(gu) && moe::gemm_tc_supported(dn) &&
                moe::gemm_tc_supported(sgu) && moe::gemm_tc_supported(sdn)));
    // Fused unpermutation (MOE_FLAG_FUSED_COMBINE, fp16 / bf16 y): the
    // shared expert's down GEMM runs last, on this stream, and its epilogue
    // writes out; the unpermute kernel is not launched.
    const bool fused_comb = overlap && (cf.flags & MOE_FLAG_FUSED_COMBINE) && (fp8 || f16_down(cf));
    if (fused_comb) {
        sdn.cmb_out = out;
        sdn.cmb_out_f32 = cf.out_dtype == MOE_F32;
        sdn.cmb_blob = W.at<int32_t>(W.L.blob);
        sdn.cmb_inv = W.at<int32_t>(W.L.inv);
        sdn.cmb_y = W.at<void>(W.L.y);
        sdn.cmb_k = cf.top_k;
        const bool ok = fp8 ? moe::gemm_fp8_supported(sdn) : moe::gemm_tc_supported(sdn);
        if (!ok) return arg_fail(MOE_ERR_UNSUPPORTED, "fused unpermutation: shape without a kernel");
    }
    // Programmatic dependent launch along the main-stream chain (top-k,
    // permutation, expert GEMMs) below prefill sizes: batched decode bf16,
    // T=1024, 0.880 ms per layer against 0.898 without.  At T*k >= 64E
    // (prefill) it cost 15-25 us, also with only the routing and permutation
    // kernels dependent: early-launched CTAs waiting on their predecessor
    // hold SMs that the shared expert's GEMMs would otherwise take.
    const bool pdl = (int64_t)T * cf.top_k < 64LL * cf.E;
    if (overlap) {
        gu.g_end = dn.g_end = cf.E;
        // The FP8 kernel's CTA holds all of an SM's registers, so nothing
        // else runs beside it: the shared GEMMs then take five eighths of the
        // SMs and leave the rest to the top-k and permutation kernels (FP8
        // prefill, T=16384: 2.880 ms per layer against 2.894 with half, 2.896
        // with 3/4, 2.930 with all; decode sizes unchanged).  The bf16
        // shared GEMMs take three quarters (prefill bf16, T=8192: 2.223 ms
        // per layer against 2.252 with all SMs, 2.233 with 5/8, 2.251 with
        // 7/8; decode sizes unchanged).
        if (fp8) sgu.max_ctas = sdn.max_ctas = std::max(1, p->num_sms * 5 / 8);
        else sgu.max_ctas = sdn.max_ctas = std::max(1, p->num_sms * 3 / 4);
        if (fused_comb) sdn.max_ctas = 0;  // it runs alone at the end
        sgu.sched = W.sched(kSchedSharedGateup);
        sdn.sched = W.sched(kSchedSharedDown);
        // FP8: xq (the shared expert's A) is made on the side stream at
        // scatter sizes, where the permutation quantises the routed rows
        // itself; below them the gather reads xq, so it is made here
        const bool side_quant = fp8 && fused_quant_scatter(cf, T);
        if (fp8 && !side_quant)
            MOE_CUDA(moe::launch_quant_rows(x, moe::kBF16, T, cf.D, W.at<uint8_t>(W.L.xq), W.at<float>(W.L.xq_scale), s));
        MOE_CUDA(cudaEventRecord(p->ev_fork, s));
        // the router GEMM is enqueued first so that it gets the SMs; the
        // shared GEMMs fill them as its CTAs retire and run beside the
        // top-k and permutation kernels
        st = route_impl(p, w, x, T, W, stream, fh, pdl);
        MOE_CUDA(cudaStreamWaitEvent(p->side, p->ev_fork, 0));
        if (side_quant)
            MOE_CUDA(moe::launch_quant_rows(x, moe::kBF16, T, cf.D, W.at<uint8_t>(W.L.xq), W.at<float>(W.L.xq_scale),
                                            p->side));
        moe_status side_st = run_gemm(p, sgu, p->side, "shared gate/up GEMM");
        if (side_st == MOE_OK && !fused_comb) side_st = run_gemm(p, sdn, p->side, "shared down GEMM");
        // Split expert GEMMs (MOE_FLAG_SPLIT_GEMM_OFF): each routed GEMM as the
        // whole 256-row pairs on CTA pairs here and the rest of every group on
        // single CTAs on the second stream, at the same time.  The two halves
        // write disjoint rows, and each down half reads only the h rows its
        // own gate/up half wrote.  Prefill bf16, T=8192: see the design notes.
        moe::GroupedGemm gp[2], gr[2];
        const bool split = !fp8 && !fused_comb && split_wanted(p, T, W, gu, dn, gp, gr);
        if (!split) MOE_CUDA(cudaEventRecord(p->ev_join, p->side));
        {
            // the main-stream chain after the top-k: each kernel a programmatic
            // dependent of the one before it
            moe::PdlScope scope(pdl);
            if (st == MOE_OK) st = permute_impl(p, x, T, W, s, !fp8, fh);
            if (split) {
                MOE_CUDA(cudaEventRecord(p->ev_perm, s));
                MOE_CUDA(cudaStreamWaitEvent(p->side, p->ev_perm, 0));
                for (int i = 0; i < 2; ++i) {
                    if (st == MOE_OK) st = run_gemm(p, gp[i], s, i == 0 ? "gate/up GEMM, 256-row pairs" : "down GEMM, 256-row pairs");
                    if (side_st == MOE_OK)
                        side_st = run_gemm(p, gr[i], p->side, i == 0 ? "gate/up GEMM, remaining rows" : "down GEMM, remaining rows");
                }
                MOE_CUDA(cudaEventRecord(p->ev_join, p->side));
            } else {
                if (st == MOE_OK) st = run_gemm(p, gu, s, "gate/up GEMM");
                if (st == MOE_OK) st = run_gemm(p, dn, s, "down GEMM");
            }
        }
        MOE_CUDA(cudaStreamWaitEvent(s, p->ev_join, 0));  // joined even after an error (stream capture)
        if (side_st != MOE_OK) return side_st;
        if (st != MOE_OK) return st;
        if (fused_comb) {
            if ((st = run_gemm(p, sdn, s, "shared down GEMM with the unpermutation")) != MOE_OK) return st;
            return copy_routing_out(p, W, T, blob_out, logits_out, s);
        }
    } else {
        if ((st = route_impl(p, w, x, T, W, stream, fh, pdl)) != MOE_OK) return st;
        moe::PdlScope scope(pdl);
        if ((st = permute_impl(p, x, T, W, s, true, fh)) != MOE_OK) return st;
        if ((st = run_gemm(p, gu, s, "gate/up GEMM")) != MOE_OK) return st;
        if ((st = run_gemm(p, dn, s, "down GEMM")) != MOE_OK) return st;
    }
    if ((st = moe_unpermute(p, T, out, ws, ws_bytes, stream)) != MOE_OK) return st;
    return copy_routing_out(p, W, T, blob_out, logits_out, s);
}

moe_status moe_pointer_kind(const void* ptr, int32_t* kind) {
    if (!kind) return arg_fail(MOE_ERR_INVALID_ARG, "kind is NULL");
    *kind = 0;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // unregistered host memory on older drivers
        return MOE_OK;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice: *kind = 2; break;
        case cudaMemoryTypeManaged: *kind = 3; break;
        case cudaMemoryTypeHost: *kind = (a.devicePointer == ptr) ? 1 : 0; break;
        default: *kind = 0; break;
    }
    return MOE_OK;
}

moe_status moe_convert_down_weights(const moe_plan* p, const void* w_down, void* w_down_f16, void* ws,
                                   size_t ws_bytes, void* stream) {
    if (!p) return arg_fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (p->cfg.dtype != MOE_BF16) return arg_fail(MOE_ERR_UNSUPPORTED, "only the bf16 layer has an fp16 W_down copy");
    if (!ptr_ok(w_down) || !ptr_ok(w_down_f16)) return arg_fail(MOE_ERR_INVALID_ARG, "NULL or misaligned pointer");
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return arg_fail(MOE_ERR_INVALID_ARG, "workspace");
    const int64_t n = (int64_t)(p->cfg.E + 1) * p->cfg.D * p->cfg.I;
    MOE_CUDA(moe::launch_bf16_to_f16(w_down, w_down_f16, n, (uint32_t*)ws, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_pack_routing_words(const moe_plan* p, int32_t T, const void* ws, size_t ws_bytes, int32_t* words,
                                  void* stream) {
    Ws W;
    moe_status st = check_call(p, T, const_cast<void*>(ws), ws_bytes, &W);
    if (st != MOE_OK) return st;
    if (!ptr_ok(words)) return arg_fail(MOE_ERR_INVALID_ARG, "words NULL or misaligned");
    MOE_CUDA(moe::launch_pack_words(W.at<int32_t>(W.L.blob), (int64_t)T * p->cfg.top_k, words, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_check(const moe_plan* p, const void* ws, void* stream) {
    if (!p || !ws) return arg_fail(MOE_ERR_INVALID_ARG, "NULL argument");
    uint32_t word[4] = {0, 0, 0, 0};
    MOE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    MOE_CUDA(cudaMemcpy(word, ws, sizeof(word), cudaMemcpyDeviceToHost));
    if (word[0] != 0) {
        snprintf(g_detail, sizeof(g_detail), "device error %u (%s), info %u %u %u", word[0],
                 moe_status_str((moe_status)word[0]), word[1], word[2], word[3]);
        return (moe_status)word[0];
    }
    return MOE_OK;
}

moe_status moe_selftest_wait_timeout(const moe_plan* p, void* ws, size_t ws_bytes, int64_t limit_ns, void* stream) {
    if (!p || !ws || !aligned(ws, 256) || ws_bytes < 256) return arg_fail(MOE_ERR_INVALID_ARG, "workspace");
    if (limit_ns < 0 || limit_ns > 10000000000LL) return arg_fail(MOE_ERR_INVALID_ARG, "limit_ns outside [0, 10 s]");
    MOE_CUDA(moe::launch_selftest_timeout((uint32_t*)ws, limit_ns, (cudaStream_t)stream));
    return MOE_OK;
}

}  // extern "C"
