// Grouped GEMM on the CUDA cores (fp32 arithmetic), C_g = A_g * B_g^T.
//
// This is the kernel of the fp32 layer ("fp32 throughout": no tensor-core
// rounding of the operands) and an independent cross-check of the
// tensor-core path for bf16.  128 x 64 output tiles, K in steps of 16,
// 256 threads each owning an 8 x 4 block (two of them for SwiGLU, whose
// gate and up products share the A tile).  Row tiles of the grouped layout
// are walked through the device-built tile prefix, so no host round trip
// is needed to learn the per-expert row counts.
#include <type_traits>
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {
constexpr int BM = 128, BN = 64, BK = 16;

template <typename T> __device__ __forceinline__ void load8(const T* p, float* v);
template <> __device__ __forceinline__ void load8<float>(const float* p, float* v) {
    float4 a = __ldg((const float4*)p), b = __ldg((const float4*)(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <> __device__ __forceinline__ void load8<bf16>(const bf16* p, float* v) {
    int4 r = __ldg((const int4*)p);
    const bf16* e = (const bf16*)&r;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(e[i]);
}
template <> __device__ __forceinline__ void load8<f16>(const f16* p, float* v) {
    int4 r = __ldg((const int4*)p);
    const f16* e = (const f16*)&r;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __half2float(e[i]);
}
template <typename T> __device__ __forceinline__ void load4(const T* p, float* v) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = to_f32(p[i]);
}
}  // namespace

template <typename TE, typename TB, typename TO, bool SWIGLU>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GroupedGemm g) {
    pdl_wait_then_release();
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ float Bs2[SWIGLU ? BK : 1][BN + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int N = g.N, Ka = g.Ka, Kb = g.Kb;
    const int n0 = blockIdx.y * BN;
    const int total = g.offsets ? __ldg(g.tiles + g.G) : (int)cdiv(g.rows, BM);
    const TE* A = (const TE*)g.a;
    const TE* As_ = (const TE*)g.a_shared;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int grp = 0, m0, nrows, out0;
        if (g.offsets) {
            grp = find_group(g.tiles, g.G, tile);
            m0 = (tile - __ldg(g.tiles + grp)) * BM;
            out0 = __ldg(g.offsets + grp);
            nrows = __ldg(g.offsets + grp + 1) - out0;
        } else {
            m0 = tile * BM;
            out0 = 0;
            nrows = g.rows;
        }
        const TE* abase = (grp == g.shared_group) ? As_ : A + (int64_t)out0 * Ka;
        const TB* b1 = (const TB*)g.b + (int64_t)grp * N * Kb;
        const TB* b2 = SWIGLU ? (const TB*)g.b2 + (int64_t)grp * N * Kb : nullptr;
        float acc[8][4], acc2[SWIGLU ? 8 : 1][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) { acc[i][j] = 0.f; if (SWIGLU) acc2[i][j] = 0.f; }
        // loader coordinates
        const int ar = tid >> 1, ak = (tid & 1) * 8;   // A: 128 rows x 16 k
        const int br = tid >> 2, bk = (tid & 3) * 4;   // B: 64 rows x 16 k
        const bool a_ok = (m0 + ar) < nrows;
        const bool b_ok = (n0 + br) < N;
        for (int k0 = 0; k0 < Ka; k0 += BK) {
            float av[8], bv[4], bv2[4];
            const int kb0 = k0 % Kb;  // a hi/lo pair of A walks B twice
            if (a_ok) load8<TE>(abase + (int64_t)(m0 + ar) * Ka + k0 + ak, av);
            else {
#pragma unroll
                for (int i = 0; i < 8; ++i) av[i] = 0.f;
            }
            if (b_ok) {
                load4<TB>(b1 + (int64_t)(n0 + br) * Kb + kb0 + bk, bv);
                if (SWIGLU) load4<TB>(b2 + (int64_t)(n0 + br) * Kb + kb0 + bk, bv2);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) { bv[i] = 0.f; bv2[i] = 0.f; }
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 8; ++i) As[ak + i][ar] = av[i];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Bs[bk + i][br] = bv[i];
                if (SWIGLU) Bs2[bk + i][br] = bv2[i];
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[8], b[4], b2v[4];
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = As[kk][ty * 8 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[j] = Bs[kk][tx * 4 + j];
                    if (SWIGLU) b2v[j] = Bs2[kk][tx * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                        if (SWIGLU) acc2[i][j] = fmaf(a[i], b2v[j], acc2[i][j]);
                    }
            }
        }
        TO* out = (TO*)g.out;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = m0 + ty * 8 + i;
            if (m >= nrows) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n >= N) continue;
                float v = SWIGLU ? swiglu(acc[i][j], acc2[i][j]) : acc[i][j];
                if (g.bias) v += __ldg(g.bias + n);
                const int64_t o = (int64_t)(out0 + m) * g.ldo + n;
                if (std::is_same<TO, f16>::value && !(fabsf(v) <= 65504.f))
                    record_error(g.err, MOE_ERR_NONFINITE, SWIGLU ? 5 : 6, blockIdx.x, 1);
                const TO hi = from_f32<TO>(v);
                out[o] = hi;
                if (g.out_pair) out[o + N] = from_f32<TO>(v - to_f32(hi));
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_gemm_simt(const GroupedGemm& g, cudaStream_t stream) {
    if (g.max_tiles <= 0) return cudaGetLastError();
    dim3 grid((unsigned)std::min(g.max_tiles, 4096), (unsigned)cdiv(g.N, BN)), block(256);
    const bool sw = g.b2 != nullptr;
    const int be = g.b_elem > 0 ? g.b_elem : g.elem;
    cudaError_t e = cudaSuccess;
#define MOE_SIMT(TA, TBB, TO)                                                                          \
    do {                                                                                              \
        if (sw) e = launch_kernel(gemm_simt_kernel<TA, TBB, TO, true>, grid, block, 0, stream, 1, g);  \
        else e = launch_kernel(gemm_simt_kernel<TA, TBB, TO, false>, grid, block, 0, stream, 1, g);    \
    } while (0)
    if (g.elem == kF32 && be == kF32 && g.out_elem == kF32) MOE_SIMT(float, float, float);
    else if (g.elem == kBF16 && be == kBF16 && g.out_elem == kF32) MOE_SIMT(bf16, bf16, float);
    else if (g.elem == kBF16 && be == kBF16 && g.out_elem == kBF16) MOE_SIMT(bf16, bf16, bf16);
    else if (g.elem == kBF16 && be == kBF16 && g.out_elem == kF16) MOE_SIMT(bf16, bf16, f16);
    else if (g.elem == kF16 && be == kBF16 && g.out_elem == kF32) MOE_SIMT(f16, bf16, float);
    else if (g.elem == kF16 && be == kBF16 && g.out_elem == kF16) MOE_SIMT(f16, bf16, f16);
    else if (g.elem == kF16 && be == kF16 && g.out_elem == kF32) MOE_SIMT(f16, f16, float);
    else if (g.elem == kF16 && be == kF16 && g.out_elem == kF16) MOE_SIMT(f16, f16, f16);
    else return cudaErrorInvalidValue;
#undef MOE_SIMT
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
