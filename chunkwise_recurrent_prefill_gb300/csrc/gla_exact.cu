// Exact fp32 CUDA-core chunkwise GLA forward.
//
// The chunk steps of "线性注意力GPU算子库的定义与技术解析", section 四, in plain fp32:
// per chunk of C = 64 tokens, b = in-chunk inclusive cumulative log-gate (a Dk vector
// per token; a scalar gate is the same value in every key dimension), then
//     P_ij   = sum_d q_id k_jd exp(b_id - b_jd)   for j <= i    (decay-masked q.k^T)
//     o_i    = scale * ( sum_{j<=i} P_ij v_j + (q_i * exp(b_i)) . S )
//     S     <- diag(exp(b_last)) S + sum_j (k_j * exp(b_last - b_j))^T v_j
// Every decay is evaluated as exp of a difference of cumulative log-gates, never as a
// product of exp(+b) and exp(-b), so no intermediate can overflow however strong the
// gates are (the page's chunk form with the in-chunk decay kept exact). This is the
// path for fp32 I/O; it is also a slow exact reference for bf16 I/O.
//
// One CTA per (batch*head, Dv slice of VB columns); the state slice lives in shared
// memory for the whole sequence. Packed sequences (cu offsets) are the batches of a single
// [T] token axis. The tail chunk is zero-padded: a padded token has
// k = v = 0 and g = 0, so it neither adds to nor decays the state.
#include <cuda_bf16.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kC = 64;        // chunk length
constexpr int kVB = 32;       // Dv columns per CTA
constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int DK, int DV>
constexpr size_t exact_smem_bytes() {
    // q, k, b tiles with a padded row (DK + 1) against bank conflicts, v slice, P, S.
    return sizeof(float) * (3 * kC * (DK + 1) + kC * kVB + kC * kC + DK * kVB);
}

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
gla_exact_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                 const float *__restrict__ g, float scale, const float *__restrict__ h0,
                 IO *__restrict__ o, float *__restrict__ hT, int64_t T, int64_t H,
                 int gate_scalar, const int *__restrict__ cu, int seq_filter,
                 unsigned *__restrict__ err) {
    constexpr int KS = DK + 1;
    extern __shared__ float sm[];
    float *qs = sm;                 // [C][KS]  q, later q * exp(b)
    float *ks = qs + kC * KS;       // [C][KS]  k, later k * exp(b_last - b)
    float *bs = ks + kC * KS;       // [C][KS]  g, then the cumulative log-gate b
    float *vs = bs + kC * KS;       // [C][VB]
    float *Ps = vs + kC * kVB;      // [C][C]
    float *Ss = Ps + kC * kC;       // [DK][VB] state slice

    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H, h = bh % H;
    const int v0 = blockIdx.y * kVB;
    // token rows [r0, r0 + Tb) of the flattened [B*T] (or packed) token axis
    int64_t r0 = b * T, Tb = T;
    if (cu) {
        const int s0 = cu[b], s1 = cu[b + 1];
        const bool bad = s0 < 0 || s1 < s0 || s1 > T;
        if (bad && tid == 0 && err) atomicOr(err, kDevErrInternal);
        r0 = bad ? 0 : s0;
        Tb = bad ? 0 : s1 - s0;
        if (bad) return;   // uniform across the block: nothing is written
        // sequences another launch of the call handles (uniform across the block)
        if ((seq_filter == kShortOnly && Tb >= kShortSeq) ||
            (seq_filter == kLongOnly && Tb < kShortSeq))
            return;
    }

    for (int i = tid; i < DK * kVB; i += kThreads) {
        const int d = i / kVB, e = i % kVB;
        Ss[i] = h0 ? h0[(bh * DK + d) * DV + v0 + e] : 0.f;
    }

    for (int64_t t0 = 0; t0 < Tb; t0 += kC) {
        const int L = (int)((Tb - t0) < kC ? (Tb - t0) : kC);
        __syncthreads();
        for (int i = tid; i < kC * DK; i += kThreads) {
            const int t = i / DK, d = i % DK;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (t < L) {
                const int64_t idx = ((r0 + t0 + t) * H + h) * DK + d;
                qv = to_f(q[idx]);
                kv = to_f(k[idx]);
                gv = gate_scalar ? g[(r0 + t0 + t) * H + h] : g[idx];
            }
            qs[t * KS + d] = qv;
            ks[t * KS + d] = kv;
            bs[t * KS + d] = gv;
        }
        for (int i = tid; i < kC * kVB; i += kThreads) {
            const int t = i / kVB, e = i % kVB;
            vs[i] = t < L ? to_f(v[((r0 + t0 + t) * H + h) * DV + v0 + e]) : 0.f;
        }
        __syncthreads();
        if (tid < DK) {  // inclusive cumulative log-gate along the chunk, per key dim
            float acc = 0.f;
            for (int t = 0; t < kC; ++t) {
                acc += bs[t * KS + tid];
                bs[t * KS + tid] = acc;
            }
        }
        __syncthreads();
        for (int p = tid; p < kC * kC; p += kThreads) {  // decay-masked q.k^T
            const int i = p / kC, j = p % kC;
            float acc = 0.f;
            if (j <= i) {
                const float *qi = qs + i * KS, *kj = ks + j * KS;
                const float *bi = bs + i * KS, *bj = bs + j * KS;
#pragma unroll 8
                for (int d = 0; d < DK; ++d) acc += qi[d] * kj[d] * expf(bi[d] - bj[d]);
            }
            Ps[p] = acc;
        }
        __syncthreads();
        for (int i = tid; i < kC * DK; i += kThreads) {  // q * exp(b), k * exp(b_last - b)
            const int t = i / DK, d = i % DK;
            const float bb = bs[t * KS + d];
            qs[t * KS + d] *= expf(bb);
            ks[t * KS + d] *= expf(bs[(kC - 1) * KS + d] - bb);
        }
        __syncthreads();
        for (int p = tid; p < kC * kVB; p += kThreads) {  // o = intra + inter
            const int i = p / kVB, e = p % kVB;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc += Ps[i * kC + j] * vs[j * kVB + e];
            const float *qi = qs + i * KS;
#pragma unroll 8
            for (int d = 0; d < DK; ++d) acc += qi[d] * Ss[d * kVB + e];
            if (i < L) o[((r0 + t0 + i) * H + h) * DV + v0 + e] = from_f<IO>(scale * acc);
        }
        __syncthreads();
        for (int p = tid; p < DK * kVB; p += kThreads) {  // state scan step
            const int d = p / kVB, e = p % kVB;
            float acc = expf(bs[(kC - 1) * KS + d]) * Ss[p];
#pragma unroll 8
            for (int j = 0; j < kC; ++j) acc += ks[j * KS + d] * vs[j * kVB + e];
            Ss[p] = acc;
        }
    }
    __syncthreads();
    if (hT) {
        for (int i = tid; i < DK * kVB; i += kThreads) {
            const int d = i / kVB, e = i % kVB;
            hT[(bh * DK + d) * DV + v0 + e] = Ss[i];
        }
    }
}

template <typename IO, int DK, int DV>
cudaError_t launch_typed(const Problem &p, unsigned *err, cudaStream_t s) {
    auto kern = gla_exact_kernel<IO, DK, DV>;
    const size_t smem = exact_smem_bytes<DK, DV>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.B * p.H), DV / kVB);
    kern<<<grid, kThreads, smem, s>>>(static_cast<const IO *>(p.q), static_cast<const IO *>(p.k),
                                      static_cast<const IO *>(p.v), p.g, p.scale, p.h0,
                                      static_cast<IO *>(p.o), p.hT, p.T, p.H, p.gate, p.cu,
                                      p.seq_filter, err);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

template <typename IO>
cudaError_t launch_io(const Problem &p, unsigned *err, cudaStream_t s) {
    if (p.Dk == 128 && p.Dv == 128) return launch_typed<IO, 128, 128>(p, err, s);
    if (p.Dk == 128 && p.Dv == 64) return launch_typed<IO, 128, 64>(p, err, s);
    if (p.Dk == 64 && p.Dv == 128) return launch_typed<IO, 64, 128>(p, err, s);
    if (p.Dk == 64 && p.Dv == 64) return launch_typed<IO, 64, 64>(p, err, s);
    return cudaErrorInvalidValue;
}

}  // namespace

bool exact_supported(int64_t Dk, int64_t Dv) {
    return (Dk == 64 || Dk == 128) && (Dv == 64 || Dv == 128);
}

cudaError_t launch_exact(const Problem &p, unsigned int *dev_err, cudaStream_t s) {
    if (p.B * p.H == 0) return cudaSuccess;
    if (p.io == 1) return launch_io<float>(p, dev_err, s);
    return launch_io<__nv_bfloat16>(p, dev_err, s);
}

}  // namespace gla
