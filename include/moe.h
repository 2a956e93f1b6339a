/*
 * moe.h -- C ABI of libmoe, a single-GPU (sm_103a) routed Mixture-of-Experts
 * FFN layer.
 *
 * The layer ("Systems engineering playbook: Qwen 3.5 MoE on Ironwood TPU",
 * English page, section "The Architectural Constraints That Break Naive
 * Sharding"; aihot.vn translation of the report, section 1.3 "Sparse
 * Mixture-of-Experts"): a router gate scores every token against E experts,
 * the top_k experts are chosen through a softmax distribution and their
 * weights renormalised, each chosen SwiGLU expert runs on the token, and an
 * always-on shared expert is added:
 *
 *     z      = x W_r^T + b                       (router logits, fp32)
 *     idx, w = top_k(z), softmax over the chosen z
 *     out[t] = shared(x_t) + sum_j w[t,j] * expert_{idx[t,j]}(x_t)
 *     expert_g(v) = W_down_g ( silu(W_gate_g v) * (W_up_g v) )
 *
 * Ties between equal logits go to the lower expert index; output slots are
 * ordered by descending logit.  Expert indices and weights are kept as one
 * int32 "blob" of two [T, top_k] planes (plane 0 the index, plane 1 the fp32
 * bit pattern of the weight), the packing of the English page's section
 * "Fusing Three Collectives Into Two".
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers on the plan's device, owned by
 *     the caller, at least 16-byte aligned, row-major and dense.  The library
 *     allocates no device memory; it uses the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work: nothing synchronises the host,
 *     so a sequence of calls can be captured into a CUDA graph.
 *   - Argument errors are returned synchronously before anything is enqueued.
 *     MOE_ERR_CUDA means a launch failed.  Conditions found on the device (a
 *     bounded wait that ran out, a non-finite router logit, an index out of
 *     range) are recorded in an error word inside the workspace and reported
 *     by moe_check().  No entry point prints, exits or traps.
 *   - A workspace must not be used by two calls in flight at the same time.
 *
 * Weight layout (E+1 groups; group E is the shared expert, whose
 * intermediate size equals I):
 *   w_router [E, D]         fp32 (MOE_F32 layer) or bf16 (all others)
 *   b_router [E]            fp32, or NULL when has_router_bias == 0
 *   w_gate   [E+1, I, D]    fp32 | bf16 | E4M3 codes (uint8)
 *   w_up     [E+1, I, D]    same
 *   w_down   [E+1, D, I]    same
 *   s_gate, s_up [E+1, I/128, D/128] and s_down [E+1, D/128, I/128]:
 *                           fp32 block scales, MOE_FP8_E4M3_B128 only.
 *   w_down_f16 [E+1, D, I]  fp16 copy of w_down (MOE_BF16 layer on tensor
 *                           cores, unless MOE_FLAG_DOWN_HILO); made once by
 *                           moe_convert_down_weights().  Where it is read
 *                           (MOE_BF16 without MOE_FLAG_DOWN_HILO or
 *                           MOE_FLAG_FORCE_SIMT) w_down itself is not, and
 *                           may be NULL: the caller can free the bf16 copy.
 * Every matrix is [out_features, in_features]: the reduction dimension is
 * innermost (K-major), which is what the tensor-core operand loads want.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every entry point is exported from the shared library. */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* NULL / misaligned pointer, T out of range */
    MOE_ERR_UNSUPPORTED = 2,    /* shape or dtype this build has no kernel for */
    MOE_ERR_WORKSPACE = 3,      /* workspace smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device wait ran out (moe_check) */
    MOE_ERR_BOUNDS = 6,         /* a device-side index check failed (moe_check) */
    MOE_ERR_NONFINITE = 7       /* a router logit was NaN or infinite, or an fp16 h value
                                   overflowed (diagnostic word 1 = 5 / 6) (moe_check) */
} moe_status;

/* Arithmetic type of the layer.
 *   MOE_F32: fp32 activations and weights, fp32 arithmetic throughout (no
 *     tensor cores).
 *   MOE_BF16: bf16 x and weights, fp32 accumulation; the permuted x is bf16.
 *     h = SiLU(gate)*up and the expert outputs y are each rounded once to
 *     fp16 (11 significant bits), and the down GEMM reads an fp16 copy of
 *     W_down (exact for every bf16 weight of magnitude 2^-14 .. 65504); an
 *     |h| or |y| above 65504 is reported as MOE_ERR_NONFINITE (diagnostic
 *     word 1 = 5 for h, 6 for y).  With MOE_FLAG_DOWN_HILO h is instead kept
 *     as a bf16 hi/lo pair against the bf16 W_down and y in fp32 (no range
 *     limit, twice the down-GEMM work).  Either way the layer stays within
 *     1e-2 of the output rms; fp32 or bf16 output.
 *   MOE_FP8_E4M3_B128: expert weights as E4M3 codes with one fp32 scale per
 *     128x128 block; both expert GEMM inputs (x and h) quantised to E4M3 per
 *     token per 128-column group with s = amax/448 and
 *     code = E4M3_rne_satfinite(fp32(v * fp32(448/amax))); fp32 accumulation
 *     with the block scales applied per 128-wide K chunk; router in bf16;
 *     bf16 or fp32 output. */
typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3_B128 = 2 } moe_dtype;

/* moe_config.flags */
#define MOE_FLAG_FORCE_SIMT 0x1u   /* expert GEMMs on the CUDA-core kernel (cross-check path) */
#define MOE_FLAG_PAIR_CTA_OFF 0x2u /* bf16 expert GEMMs never on CTA pairs (the default) */
#define MOE_FLAG_PAIR_CTA_ON 0x4u  /* bf16 expert GEMMs on CTA pairs (cta_group::2, 256-row tiles; a
                                      group's ragged last tile runs transposed unless
                                      MOE_FLAG_NARROW_TAILS_OFF) */
#define MOE_FLAG_DOWN_HILO 0x8u    /* bf16 layer: h as a bf16 hi/lo pair, bf16 W_down (no w_down_f16) */
/* Tile pairs: the bf16 layer's tensor-core expert GEMMs run on 2-CTA
 * clusters whose CTAs share one operand tile through TMA multicast (two
 * 128-row tiles of an expert against one weight block, or a group's odd last
 * tile against two weight blocks), so each SM reads fewer operand bytes from
 * L2 per MMA; results are identical.  By default they are used when
 * T * top_k >= 64 * E (at least 64 rows per expert on average: prefill). */
#define MOE_FLAG_MCAST_ON 0x10u    /* tile pairs whenever the shape allows them */
#define MOE_FLAG_MCAST_OFF 0x20u   /* never tile pairs */
/* Narrow tails: in the bf16 layer's tensor-core expert GEMMs a tile with at
 * most 112 valid rows (a group's ragged last tile, every tile at decode
 * sizes) is multiplied transposed, weights as the MMA's 128-wide side and the
 * rows as its N side rounded up to 16, so padding rows cost no tensor time.
 * By default only the gate/up GEMM uses them, and only where tile pairs are
 * on (T * top_k >= 64 * E); the down GEMM's transposed stores of y cost more
 * than the MMA time saved. */
#define MOE_FLAG_NARROW_TAILS_ON 0x40u   /* narrow tails in both expert GEMMs at every size */
#define MOE_FLAG_NARROW_TAILS_OFF 0x80u  /* every tile as 128 rows x N features */
/* Top-k + histogram: where the permutation works in chunks (more than 16384
 * (token, slot) pairs, or E > 512), moe_forward's top-k kernel also counts
 * the chosen experts into the permutation's per-chunk histograms, and the
 * permutation skips its own pass over the indices (English page, "The
 * Remaining Roadmap": fusing the top-k selection).  Results are identical
 * either way; this flag turns the fusion off. */
#define MOE_FLAG_TOPK_HIST_OFF 0x100u
/* Fused unpermutation (English page, "Pallas Kernels, SparseCore Co-Design,
 * and the Roofline": token unpermutation plus the local reduction folded
 * into the expert path): on the tensor-core paths (bf16 without
 * MOE_FLAG_DOWN_HILO, and FP8) moe_forward runs the shared expert's down
 * GEMM last and its epilogue writes out[t] = y_s[t] + sum_j w[t,j] *
 * y[inv[t*k+j]] directly -- the same order and rounding as the unpermute
 * kernel, so the output is bit-identical -- instead of storing y_s and
 * launching the unpermutation.  Off by default: the GEMM epilogue's few
 * warps keep far fewer loads in flight than the unpermute kernel, so the
 * gather is slower than the y_s round trip it saves. */
#define MOE_FLAG_FUSED_COMBINE 0x200u
/* Split expert GEMMs (bf16 layer, prefill sizes: T*top_k >= 64*E, on the
 * tensor-core path with the shared expert on the second stream): each routed
 * expert GEMM runs as two concurrent launches -- the whole 256-row pairs of
 * every group on CTA pairs (M=256 MMAs, which spend less time per k-block
 * waiting for operands than single CTAs), and the remaining rows of each
 * group as 128-row tiles on single CTAs on the second stream.  How many CTA
 * pairs take part is computed on the device from the group sizes (the rest
 * exit at once and leave their SMs to the single-CTA launch).  Results are
 * bit-identical either way; this flag turns the split off. */
#define MOE_FLAG_SPLIT_GEMM_OFF 0x400u

typedef struct moe_config {
    int32_t T_max;           /* largest token count a call may pass */
    int32_t D, E, I, top_k;  /* hidden size, routed experts, intermediate, experts per token */
    int32_t dtype;           /* moe_dtype */
    int32_t out_dtype;       /* MOE_F32 or MOE_BF16 */
    int32_t has_router_bias; /* 1: b_router is added to the logits */
    uint32_t flags;          /* MOE_FLAG_* */
    int64_t spin_limit_ns;   /* bound on every device-side wait; 0 = 2 s */
} moe_config;

typedef struct moe_weights {
    const void* w_router;
    const float* b_router;
    const void* w_gate;
    const void* w_up;
    const void* w_down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    const void* w_down_f16;  /* MOE_BF16 only (see above); NULL otherwise */
} moe_weights;

typedef struct moe_plan moe_plan;

/* Byte offsets of the workspace's parts for T tokens (all 256-byte aligned).
 * Stage entry points read and write these parts; tests may inspect them.
 * Rows of the expert-contiguous layout: routed pairs first (T*top_k rows,
 * grouped by expert), then the T rows of the shared expert. */
typedef struct moe_ws_layout {
    size_t total;      /* bytes needed */
    size_t err;        /* uint32[4]: first error code, then three diagnostic words; the rest of
                          this 256-byte block holds the GEMMs' unit-scheduling counters, which
                          the kernels rewind themselves (moe_workspace_init and moe_forward
                          zero the whole block) */
    size_t logits;     /* f32 [T, E] router logits (bias included) */
    size_t blob;       /* int32 [2, T, top_k]: expert index plane, fp32-weight-bits plane */
    size_t counts;     /* int32 [E+1]: rows per group; counts[E] = T */
    size_t offsets;    /* int32 [E+2]: exclusive prefix of counts; offsets[E] = T*top_k */
    size_t tiles;      /* int32 [E+2]: exclusive prefix of ceil(counts/128) (row tiles) */
    size_t inv;        /* int32 [T*top_k]: row of pair (t, j) in the grouped layout */
    size_t src_tok;    /* int32 [T*top_k + T]: token of each grouped row */
    size_t hist;       /* int32 [chunks, E]: per-chunk expert histograms (scratch) */
    size_t xq;         /* FP8: E4M3 [T, D] quantised x */
    size_t xq_scale;   /* FP8: f32 [T, D/128] */
    size_t xp;         /* [T*top_k, D] x gathered into grouped order (layer dtype; E4M3 for FP8) */
    size_t xp_scale;   /* FP8: f32 [T*top_k, D/128] */
    size_t h;          /* SwiGLU activations: f32 [R, I] (MOE_F32) | fp16 [R, I] (MOE_BF16) |
                          bf16 hi/lo pair [R, 2I] (MOE_BF16 + MOE_FLAG_DOWN_HILO: hi in
                          columns 0..I-1, lo = bf16(h - hi) in I..2I-1) | E4M3 [R, I];
                          R = T*top_k + T */
    size_t h_scale;    /* FP8: f32 [T*top_k + T, I/128] */
    size_t y;          /* [R, D] expert outputs: f32 (MOE_F32; MOE_BF16 + MOE_FLAG_DOWN_HILO),
                          fp16 (MOE_BF16) or bf16 (FP8 layer) */
    size_t logits_part;/* f32 [S, T, E] router K-slice partials when T is small (S > 1), else 0 */
    size_t tiles2;     /* int32 [E+2]: exclusive prefix of ceil(counts/256) (row-tile pairs) */
    size_t pairs;      /* int32 [2, E+2], [2], [E+2]: the exclusive prefix of floor(counts/256)
                          by group (whole 256-row pairs); the exclusive prefix of the 128-row
                          tiles of what remains of each group, taken over the positions of
                          the order below; the CTA-pair clusters the split expert GEMMs run
                          with (gate/up, down); the group at each position of the single-CTA
                          launch's order (a permutation of 0..E, the shared group E last).
                          Written by the permutation, and only where the split can run: bf16
                          layer, T*top_k >= 64*E (see MOE_FLAG_SPLIT_GEMM_OFF) */
} moe_ws_layout;

/* Validate a configuration and build a host-side plan for `device`.
 * Supported: D, I multiples of 128 (64 for MOE_F32; D a multiple of 256 for
 * MOE_FP8_E4M3_B128), E <= 1024,
 * 1 <= top_k <= min(E, 32), 1 <= T_max <= 2^20, T_max*(top_k+1) < 2^31.
 * The plan owns no device memory; it holds one CUDA stream and two events
 * on `device` (see moe_forward).  *out is NULL on error. */
MOE_API moe_status moe_plan_create(const moe_config* cfg, int device, moe_plan** out);
MOE_API void moe_plan_destroy(moe_plan* plan);
MOE_API const moe_config* moe_plan_config(const moe_plan* plan);

/* Workspace layout / size for T tokens (1 <= T <= T_max). */
MOE_API moe_status moe_workspace_layout(const moe_plan* plan, int32_t T, moe_ws_layout* out);
MOE_API moe_status moe_workspace_size(const moe_plan* plan, int32_t T, size_t* bytes);

/* Zero the workspace's error word and scheduling counters (moe_forward does
 * this itself; call it before stage entry points after an error). */
MOE_API moe_status moe_workspace_init(const moe_plan* plan, void* ws, size_t ws_bytes, void* stream);

/* Block-quantise fp32 weights to E4M3 (English page, "Roofline Validation":
 * FP8 scaling blocks audited against a higher-precision path).  w is
 * [groups, rows, cols] fp32; q receives [groups, rows, cols] E4M3 codes and s
 * [groups, rows/128, cols/128] fp32 scales, s = amax/448 of each 128x128
 * block (1 for an all-zero block).  rows and cols must be multiples of 128. */
MOE_API moe_status moe_quantize_weights(const moe_plan* plan, const float* w, int64_t groups, int32_t rows,
                                int32_t cols, uint8_t* q, float* s, void* stream);

/* The whole layer: route, permute, gate/up GEMM with SwiGLU, down GEMM,
 * unpermute with the shared-expert add.  x [T, D] (fp32 for MOE_F32, else
 * bf16); out [T, D] of cfg.out_dtype; 1 <= T <= T_max, or T = 0 (an empty
 * batch: MOE_OK at once, no pointer is read and nothing is launched).  blob_out (nullable) receives a copy of
 * the [2, T, top_k] routing blob; logits_out (nullable) a copy of the [T, E]
 * fp32 logits.  Clears the workspace error word first.
 * On the tensor-core paths (bf16 and FP8; not MOE_FLAG_FORCE_SIMT) the
 * shared expert's two GEMMs, which need no
 * routing, run on the plan's own stream, forked from `stream` with an event
 * at the start and joined back before the unpermute, so they overlap the
 * router, top-k and permutation; the call stays asynchronous and can be
 * captured into a CUDA graph.  A plan must therefore not be used by two host
 * threads calling moe_forward at the same time. */
MOE_API moe_status moe_forward(const moe_plan* plan, const moe_weights* w, const void* x, int32_t T, void* out,
                       int32_t* blob_out, float* logits_out, void* ws, size_t ws_bytes, void* stream);

/* Stage entry points: the same kernels moe_forward runs, one stage per call,
 * reading and writing the workspace parts named in moe_ws_layout. */

/* Router GEMM (logits, bias added) then moe_topk. */
MOE_API moe_status moe_route(const moe_plan* plan, const moe_weights* w, const void* x, int32_t T, void* ws,
                     size_t ws_bytes, void* stream);
/* From ws.logits: top_k with lowest-index tie-break, softmax over the chosen
 * logits, written into ws.blob.  Non-finite logits set MOE_ERR_NONFINITE. */
MOE_API moe_status moe_topk(const moe_plan* plan, int32_t T, void* ws, size_t ws_bytes, void* stream);
/* From ws.blob plane 0: counts, offsets, tiles, inv, src_tok (a stable
 * counting sort of the (t, j) pairs in row-major order), and xp = x rows in
 * grouped order (quantised to E4M3 for the FP8 layer, with xq for the shared
 * group). */
MOE_API moe_status moe_permute(const moe_plan* plan, const void* x, int32_t T, void* ws, size_t ws_bytes,
                       void* stream);
/* h[r] = silu(W_gate_g a_r) * (W_up_g a_r) for every grouped row r of group g,
 * a_r = xp[r] for routed rows and x[t] for the shared group. */
MOE_API moe_status moe_gemm_gateup(const moe_plan* plan, const moe_weights* w, const void* x, int32_t T, void* ws,
                           size_t ws_bytes, void* stream);
/* y[r] = W_down_g h[r]. */
MOE_API moe_status moe_gemm_down(const moe_plan* plan, const moe_weights* w, int32_t T, void* ws, size_t ws_bytes,
                         void* stream);
/* out[t] = y[T*top_k + t] + sum_j w[t,j] * y[inv[t*top_k + j]], fp32
 * accumulation in slot order (English page, table in "Pallas Kernels,
 * SparseCore Co-Design, and the Roofline": token unpermutation plus the local
 * reduction). */
MOE_API moe_status moe_unpermute(const moe_plan* plan, int32_t T, void* out, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free permutation index build (no counterpart in the paper:
 * it exists for callers of this library that cannot allocate device memory,
 * e.g. a plugin whose host framework owns every device allocation through
 * its own arena, or a serving loop that forbids cudaMalloc -- and the device
 * synchronisation it may cause -- after start-up).
 * Computes what moe_permute writes into counts, offsets, tiles, inv and
 * src_tok, from idx = the [T, top_k] expert-index plane, with the same
 * kernels; the caller passes those outputs ([E+1], [E+2], [E+2], [T*top_k],
 * [T*top_k + T] int32, device pointers).  No allocation of any kind: the
 * only scratch (per-chunk histograms) is one 1 MiB array in the library's
 * device memory, held by every GPU that loads the library until the process
 * exits; so ceil(T*top_k / 1024) * E must not exceed 262144 (e.g. E=512
 * allows T*top_k <= 524288), else MOE_ERR_UNSUPPORTED before any work.
 * E <= 1024, 1 <= top_k <= min(E, 32).
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current); make that first call
 * before any stream capture.  The address is kept for the life of the
 * process: after cudaDeviceReset (or anything else that replaces the
 * device's primary context) this entry point must not be called again.  Every call on a device shares the one array:
 * calls that overlap on the GPU (other streams, other threads) race and must
 * be serialised by the caller.  Out-of-range expert ids are skipped (their
 * pairs get no row); there is no error word.  The array keeps the last
 * call's histograms, which no later call reads before overwriting. */
MOE_API moe_status moe_permute_index_noalloc(const int32_t* idx, int32_t T, int32_t E, int32_t top_k,
                                             int32_t* counts, int32_t* offsets, int32_t* tiles, int32_t* inv,
                                             int32_t* src_tok, void* stream);

/* Compact routing word (English page, "Fusing Three Collectives Into Two":
 * indices and weights packed into one dense 32-bit blob).  From the
 * workspace blob of the last moe_route / moe_forward for T tokens, writes
 * words [T, top_k] int32: bits 0..15 the expert index, bits 16..31 the bf16
 * (round to nearest even) of the fp32 routing weight.  Half the bytes of the
 * two-plane blob; the weight keeps 8 significant bits. */
MOE_API moe_status moe_pack_routing_words(const moe_plan* plan, int32_t T, const void* ws, size_t ws_bytes,
                                          int32_t* words, void* stream);

/* One-time weight preparation of the bf16 layer: writes w_down_f16, the
 * fp16 copy of w_down ([E+1, D, I], both caller-allocated device buffers,
 * 16-byte aligned, not overlapping) that the down GEMM reads on tensor cores.
 * Each value is rounded to nearest even; bf16 values below 2^-14 in
 * magnitude lose low bits (fp16 subnormals), values above 65504 record
 * MOE_ERR_BOUNDS in the error word of `ws` (moe_check reports it).
 * MOE_ERR_UNSUPPORTED unless the plan's dtype is MOE_BF16. */
MOE_API moe_status moe_convert_down_weights(const moe_plan* plan, const void* w_down, void* w_down_f16, void* ws,
                                            size_t ws_bytes, void* stream);

/* Where a pointer lives, as the device sees it: *kind = 0 host memory the
 * device cannot address, 1 page-locked host memory mapped at the same address
 * (a kernel may read or write it directly, e.g. moe_forward's `out`, so the
 * result lands in host memory without a separate copy), 2 device memory,
 * 3 managed memory.  Synchronous, enqueues nothing. */
MOE_API moe_status moe_pointer_kind(const void* p, int32_t* kind);

/* Synchronise `stream`, read the workspace error word and return the first
 * device-side error recorded since the last clear (MOE_OK if none). */
MOE_API moe_status moe_check(const moe_plan* plan, const void* ws, void* stream);

/* Self-test of the bounded-wait machinery: one block waits on an mbarrier
 * that nothing arrives at, for at most limit_ns, then records
 * MOE_ERR_DEVICE_TIMEOUT in the error word and returns normally. */
MOE_API moe_status moe_selftest_wait_timeout(const moe_plan* plan, void* ws, size_t ws_bytes, int64_t limit_ns,
                                     void* stream);

MOE_API const char* moe_status_str(moe_status s);

/* Human-readable detail of the last error returned on this host thread
 * (which argument, which CUDA call); empty if none. */
MOE_API const char* moe_last_error_detail(void);

/* Number of kernels this library has launched in this process (all
 * devices, all streams), for launch accounting by benchmarks. */
MOE_API uint64_t moe_launch_count(void);

/* Build identification: "sm_103a tcgen05" plus the kernel set compiled in. */
MOE_API const char* moe_build_info(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
