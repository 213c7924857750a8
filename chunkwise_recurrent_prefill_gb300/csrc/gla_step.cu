// One decode step of the gated recurrence on a resident state (the step after prefill):
//     S <- diag(exp(g)) . S + k^T v,    o = scale . q . S        (per batch and head)
// This is the token update of "Linear Attention 在 GPU 上到底慢在哪", section 学长的反馈,
// applied once, with the update before the read as in "线性注意力GPU算子库的定义与技术解析",
// section 四. The state is read and written once, so the step is bound by HBM bandwidth:
// plain coalesced loads and stores, fp32 arithmetic, no tensor cores.
#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kStepWarps = 8;
constexpr int kStepCols = 128;  // state columns (value dims) per CTA: four per lane
constexpr int kStepBatch = 16;  // state rows a warp loads before it stores them

template <typename T>
__device__ __forceinline__ float ld_io(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld_io<float>(const float *p, size_t i) {
    return p[i];
}
template <>
__device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_io(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// CTA = (head bh, block of 128 value columns). Warp w updates key rows w, w + 8, ...; lane l
// owns value columns c = 128 * blockIdx.y + 4 l .. c + 3 and moves them with 16-byte
// accesses, so every row access of a warp is one contiguous 512-byte segment of S. The
// per-column dot products q . S[:, v] are summed across warps in shared memory in a fixed
// order (no atomics: the result is deterministic). Dv is a multiple of 4.
template <typename T>
__global__ void __launch_bounds__(kStepWarps * 32, 2)
gla_step_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const float *__restrict__ g, float scale, float *__restrict__ S,
                T *__restrict__ o, int Dk, int Dv) {
    __shared__ float4 part[kStepWarps][kStepCols / 4];
    extern __shared__ float rows[];   // [3][Dk]: exp(g_d), k_d, q_d, shared by every lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    for (int d = threadIdx.x; d < Dk; d += blockDim.x) {
        rows[d] = expf(g[bh * Dk + d]);
        rows[Dk + d] = ld_io(k, bh * Dk + d);
        rows[2 * Dk + d] = ld_io(q, bh * Dk + d);
    }
    __syncthreads();
    const int col = blockIdx.y * kStepCols + 4 * lane;
    const bool in = col < Dv;
    float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in) {
        vv.x = ld_io(v, bh * Dv + col);
        vv.y = ld_io(v, bh * Dv + col + 1);
        vv.z = ld_io(v, bh * Dv + col + 2);
        vv.w = ld_io(v, bh * Dv + col + 3);
    }
    float *Sp = S + bh * (size_t)Dk * Dv + col;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // rows warp, warp + 8, ...: a batch of kStepBatch rows is loaded before any of it is
    // stored, so each warp keeps that many 512-byte loads in flight
    for (int d0 = warp; d0 < Dk; d0 += kStepWarps * kStepBatch) {
        float4 sv[kStepBatch];
#pragma unroll
        for (int j = 0; j < kStepBatch; ++j) {
            const int d = d0 + j * kStepWarps;
            sv[j] = (d < Dk && in) ? *reinterpret_cast<const float4 *>(Sp + (size_t)d * Dv)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kStepBatch; ++j) {
            const int d = d0 + j * kStepWarps;
            if (d < Dk && in) {
                const float al = rows[d], kd = rows[Dk + d], qd = rows[2 * Dk + d];
                float4 s4;
                s4.x = fmaf(al, sv[j].x, kd * vv.x);
                s4.y = fmaf(al, sv[j].y, kd * vv.y);
                s4.z = fmaf(al, sv[j].z, kd * vv.z);
                s4.w = fmaf(al, sv[j].w, kd * vv.w);
                *reinterpret_cast<float4 *>(Sp + (size_t)d * Dv) = s4;
                acc.x = fmaf(qd, s4.x, acc.x);
                acc.y = fmaf(qd, s4.y, acc.y);
                acc.z = fmaf(qd, s4.z, acc.z);
                acc.w = fmaf(qd, s4.w, acc.w);
            }
        }
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && in) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kStepWarps; ++w) {
            sum.x += part[w][lane].x;
            sum.y += part[w][lane].y;
            sum.z += part[w][lane].z;
            sum.w += part[w][lane].w;
        }
        st_io(o, bh * Dv + col, scale * sum.x);
        st_io(o, bh * Dv + col + 1, scale * sum.y);
        st_io(o, bh * Dv + col + 2, scale * sum.z);
        st_io(o, bh * Dv + col + 3, scale * sum.w);
    }
}

}  // namespace

bool step_supported(int64_t Dk, int64_t Dv) {
    return Dk >= 1 && Dk <= 1024 && Dv >= 4 && Dv <= 1024 && Dv % 4 == 0;
}

cudaError_t launch_step(const void *q, const void *k, const void *v, const float *g, float scale,
                        float *S, void *o, int64_t BH, int64_t Dk, int64_t Dv, int io,
                        cudaStream_t stream) {
    const dim3 grid((unsigned)BH, (unsigned)((Dv + kStepCols - 1) / kStepCols));
    const size_t smem = 3 * (size_t)Dk * sizeof(float);   // <= 12 KB
    if (io == 0) {
        gla_step_kernel<__nv_bfloat16><<<grid, kStepWarps * 32, smem, stream>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(v), g, scale, S, static_cast<__nv_bfloat16 *>(o),
            (int)Dk, (int)Dv);
    } else {
        gla_step_kernel<float><<<grid, kStepWarps * 32, smem, stream>>>(
            static_cast<const float *>(q), static_cast<const float *>(k),
            static_cast<const float *>(v), g, scale, S, static_cast<float *>(o), (int)Dk, (int)Dv);
    }
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace gla
