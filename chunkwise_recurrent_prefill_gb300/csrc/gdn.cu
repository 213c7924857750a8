// Gated delta rule forward (prefill), chunkwise, fp32 CUDA cores.
//
// Per batch and head, with one log-gate g_t and one write strength beta_t per token:
//     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = scale q_t S_t
// (the gated-delta-network family named in "面向长序列大模型的线性注意力算子性能评测方法与
// 优化实践", section 三.3, and "线性注意力GPU算子库的定义与技术解析", section 三; the formula is
// the published gated delta rule, which the pages do not print).
//
// Chunk algebra (C = 64 tokens, start state S0, b_i the inclusive in-chunk cumulative
// log-gate): the new values the chunk writes are U = Ut - W S0, where (I + A) Ut = diag(beta) V,
// (I + A) W = diag(beta exp(b)) K and A_jm = beta_j exp(b_j - b_m) k_j.k_m for m < j. Then
//     O   = scale (diag(exp(b)) Q S0 + P U),   P_ij = exp(b_i - b_j) q_i.k_j for j <= i
//     S1  = exp(b_63) S0 + Kh^T U,             Kh_j = exp(b_63 - b_j) k_j.
// Substituting U, O = Oi + G S0 with Oi = scale P Ut and G = scale (diag(exp(b)) Q - P W).
// Everything that does not depend on S0 (A, the triangular solves, P, G, Oi, the decay
// factors) is computed for all chunks at once by gdn_prep_kernel and written to a workspace;
// the state then runs through the chunks in gdn_scan_kernel, one CTA per (batch, head, block
// of state columns), which forms U and O from S0 in one pass and then S1: the columns of S
// are independent under this recurrence (the transition acts on the key axis only), which is
// what lets B = 1 spread over many SMs.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kMaxD = 128;      // largest head dim
constexpr int kThreads = 256;
constexpr int kPrepStride = kC + 4;   // padded row of the transposed q/k tiles (see the loads)

__device__ __forceinline__ void st_io(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// 4 consecutive elements (8 or 16 bytes, aligned) as fp32
template <typename T>
__device__ __forceinline__ float4 ld4(const T *p);
template <>
__device__ __forceinline__ float4 ld4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Workspace of one (batch, head, chunk), in floats (every offset a multiple of 4):
//   Wt [Dk][64]  W transposed                    Ut [64][Dv] the solved values
//   Gt [Dk][64]  (Qh - P W) transposed, Qh = scale exp(b_i) q_i
//   Oi [64][Dv]  P Ut  (P carries the scale, zero above the diagonal)
//   Kh [64][Dk]  exp(b_63 - b_j) k_j
//   gc [4]       exp(b_63), 0, 0, 0
// so that the scan computes, per chunk, U = Ut - W S0, O = Oi + G S0 (both from S0 alone)
// and S1 = exp(b_63) S0 + Kh^T U.
struct WsLayout {
    int64_t oW, oU, oG, oO, oK, oC, total;
    __host__ __device__ WsLayout(int Dk, int Dv) {
        oW = 0;
        oU = oW + (int64_t)Dk * kC;
        oG = oU + (int64_t)kC * Dv;
        oO = oG + (int64_t)Dk * kC;
        oK = oO + (int64_t)kC * Dv;
        oC = oK + (int64_t)kC * Dk;
        total = oC + 4;
    }
};

struct GdnArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    float scale;
    const float *h0;
    void *o;
    float *hT;
    int64_t T;
    int H, Dk, Dv, nchunks;
    float *ws;
};

constexpr int kPieces = kC * kMaxD / 4 / kThreads;   // 4-element pieces of a tile per thread

// ---------------------------------------------------------------------------------------
// Chunk-parallel part: one CTA per (batch, head, chunk).
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) gdn_prep_kernel(GdnArgs a) {
    extern __shared__ __align__(16) float smp[];
    float *Qt = smp;                                  // [Dk][kPrepStride]; later v [64][Dv]
    float *Kt = Qt + kMaxD * kPrepStride;             // [Dk][kPrepStride]
    float *As = Kt + kMaxD * kPrepStride;             // [64][64] strictly lower A
    float *Ps = As + kC * kC;                         // [64][64] P (row i), zero for j > i
    float *bs = Ps + kC * kC;                         // [64] cumulative log-gate b_j
    float *be = bs + kC;                              // [64] beta_j
    float *eb = be + kC;                              // [64] exp(b_j)
    float *bg = eb + kC;                              // [64] beta_j exp(b_j)
    float *ek = bg + kC;                              // [64] exp(b_63 - b_j)
    const int tid = threadIdx.x;
    const int64_t blk = blockIdx.x;
    const int c = (int)(blk % a.nchunks);
    const int64_t bh = blk / a.nchunks;
    const int64_t bb = bh / a.H, h = bh % a.H;
    const int Dk = a.Dk, Dv = a.Dv;
    const int64_t t0 = (int64_t)c * kC;
    const int nval = (int)(a.T - t0 < kC ? a.T - t0 : kC);   // valid tokens of this chunk
    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    auto row = [&](int j) -> int64_t { return (bb * a.T + t0 + j) * a.H + h; };   // token row
    const WsLayout L(Dk, Dv);
    float *ws = a.ws + blk * L.total;

    // q and k in 4-element pieces (piece p: row j = p % 64, key dims 4 (p / 64) ..), all
    // loads of a thread in flight at once; then transposed into [d][j]. The 32 lanes of a
    // warp hold 32 consecutive rows of one piece column, so with the padded stride each
    // transposed store hits 32 different banks. Rows past the sequence end are zero.
    const int npk = kC * (Dk / 4);
    float4 qr[kPieces], kr[kPieces];
#pragma unroll
    for (int it = 0; it < kPieces; ++it) {
        const int p = tid + kThreads * it, j = p & (kC - 1), c4 = p >> 6;
        const bool in = p < npk && j < nval;
        qr[it] = in ? ld4(q + row(j) * Dk + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        kr[it] = in ? ld4(k + row(j) * Dk + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < kC) {
        const bool in = tid < nval;
        bs[tid] = in ? a.g[row(tid)] : 0.f;
        be[tid] = in ? a.beta[row(tid)] : 0.f;
    }
#pragma unroll
    for (int it = 0; it < kPieces; ++it) {
        const int p = tid + kThreads * it, j = p & (kC - 1), c4 = p >> 6;
        if (p < npk) {
            float *qd = Qt + 4 * c4 * kPrepStride + j, *kd = Kt + 4 * c4 * kPrepStride + j;
            qd[0] = qr[it].x; qd[kPrepStride] = qr[it].y;
            qd[2 * kPrepStride] = qr[it].z; qd[3 * kPrepStride] = qr[it].w;
            kd[0] = kr[it].x; kd[kPrepStride] = kr[it].y;
            kd[2 * kPrepStride] = kr[it].z; kd[3 * kPrepStride] = kr[it].w;
        }
    }
    __syncthreads();
    if (tid == 0) {   // inclusive cumulative sum, left to right
        float s = 0.f;
        for (int j = 0; j < kC; ++j) {
            s += bs[j];
            bs[j] = s;
        }
    }
    __syncthreads();
    if (tid < kC) {
        eb[tid] = expf(bs[tid]);
        bg[tid] = be[tid] * eb[tid];
        ek[tid] = expf(bs[kC - 1] - bs[tid]);
    }
    __syncthreads();
    // Kh = exp(b_63 - b_j) k_j straight from the pieces in registers; exp(b_63)
#pragma unroll
    for (int it = 0; it < kPieces; ++it) {
        const int p = tid + kThreads * it, j = p & (kC - 1), c4 = p >> 6;
        if (p < npk) {
            const float e = ek[j];
            *reinterpret_cast<float4 *>(ws + L.oK + (int64_t)j * Dk + 4 * c4) =
                make_float4(e * kr[it].x, e * kr[it].y, e * kr[it].z, e * kr[it].w);
        }
    }
    if (tid < 4) ws[L.oC + tid] = tid == 0 ? eb[kC - 1] : 0.f;

    // K K^T and Q K^T, one 4 x 4 tile of each per thread: rows 4 mg .., columns 4 ng ..
    {
        const int mg = tid >> 4, ng = tid & 15;
        float kk[16], qk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) kk[x] = qk[x] = 0.f;
#pragma unroll 4
        for (int d = 0; d < Dk; ++d) {
            const float4 ka = *reinterpret_cast<const float4 *>(Kt + d * kPrepStride + 4 * mg);
            const float4 qa = *reinterpret_cast<const float4 *>(Qt + d * kPrepStride + 4 * mg);
            const float4 kb = *reinterpret_cast<const float4 *>(Kt + d * kPrepStride + 4 * ng);
            const float ar[4] = {ka.x, ka.y, ka.z, ka.w}, qa4[4] = {qa.x, qa.y, qa.z, qa.w};
            const float bc[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    kk[r * 4 + cc] = fmaf(ar[r], bc[cc], kk[r * 4 + cc]);
                    qk[r * 4 + cc] = fmaf(qa4[r], bc[cc], qk[r * 4 + cc]);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * mg + r;   // row: j of A, i of P
            float av[4], pv[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int m = 4 * ng + cc;   // column: m of A, j of P
                // A_im = beta_i exp(b_i - b_m) k_i.k_m for m < i
                av[cc] = m < i ? be[i] * expf(bs[i] - bs[m]) * kk[r * 4 + cc] : 0.f;
                // P_im = scale exp(b_i - b_m) q_i.k_m for m <= i
                pv[cc] = m <= i ? a.scale * expf(bs[i] - bs[m]) * qk[r * 4 + cc] : 0.f;
            }
            *reinterpret_cast<float4 *>(As + i * kC + 4 * ng) = make_float4(av[0], av[1], av[2], av[3]);
            *reinterpret_cast<float4 *>(Ps + i * kC + 4 * ng) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        }
    }
    __syncthreads();

    // Qh = scale exp(b_i) q_i (transposed) goes to the workspace, where it becomes G below;
    // then the q tile's space takes v, rows j, for the right-hand sides of the solve
    for (int idx = tid; idx < Dk * kC; idx += kThreads) {
        const int d = idx / kC, i = idx % kC;
        ws[L.oG + idx] = a.scale * eb[i] * Qt[d * kPrepStride + i];
    }
    __syncthreads();
    float *Vs = Qt;   // [64][Dv]
    {
        const int npv = kC * (Dv / 4);
        float4 vr[kPieces];
#pragma unroll
        for (int it = 0; it < kPieces; ++it) {
            const int p = tid + kThreads * it, j = p / (Dv / 4), c4 = p % (Dv / 4);
            vr[it] = (p < npv && j < nval) ? ld4(v + row(j) * Dv + 4 * c4)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int it = 0; it < kPieces; ++it) {
            const int p = tid + kThreads * it;
            if (p < npv) *reinterpret_cast<float4 *>(Vs + 4 * p) = vr[it];
        }
    }
    __syncthreads();

    // Forward substitution, one right-hand-side column per thread:
    //   x_j = r_j - sum_{m<j} A_jm x_m,  r_j = beta_j exp(b_j) k_j[col]  (col < Dk: W)
    //                                     r_j = beta_j v_j[col - Dk]    (otherwise: Ut)
    // then y_i = sum_{j<=i} P_ij x_j, which gives the column of P W (for G) or of P Ut (Oi).
    const int col = tid;
    if (col < Dk + Dv) {
        const bool isk = col < Dk;
        const int cv = col - Dk;
        float x[kC];
#pragma unroll
        for (int j = 0; j < kC; ++j) {
            const float r = isk ? bg[j] * Kt[col * kPrepStride + j] : be[j] * Vs[j * Dv + cv];
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int m = 0; m + 3 < j; m += 4) {
                const float4 av = *reinterpret_cast<const float4 *>(As + j * kC + m);
                s0 = fmaf(av.x, x[m], s0);
                s1 = fmaf(av.y, x[m + 1], s1);
                s0 = fmaf(av.z, x[m + 2], s0);
                s1 = fmaf(av.w, x[m + 3], s1);
            }
#pragma unroll
            for (int m = j & ~3; m < j; ++m) s0 = fmaf(As[j * kC + m], x[m], s0);
            x[j] = r - (s0 + s1);
        }
        if (isk) {
            float *wt = ws + L.oW + (int64_t)col * kC;
#pragma unroll
            for (int j = 0; j < kC; j += 4)
                *reinterpret_cast<float4 *>(wt + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
        } else {
            float *ut = ws + L.oU + cv;
#pragma unroll
            for (int j = 0; j < kC; ++j) ut[(int64_t)j * Dv] = x[j];
        }
        // y = P x, four rows at a time
#pragma unroll
        for (int i0 = 0; i0 < kC; i0 += 4) {
            float y[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int m = 0; m <= i; m += 4) {   // P is zero past the diagonal
                    const float4 pv = *reinterpret_cast<const float4 *>(Ps + i * kC + m);
                    s0 = fmaf(pv.x, x[m], s0);
                    s1 = fmaf(pv.y, x[m + 1], s1);
                    s0 = fmaf(pv.z, x[m + 2], s0);
                    s1 = fmaf(pv.w, x[m + 3], s1);
                }
                y[r] = s0 + s1;
            }
            if (isk) {   // G = Qh - P W, in place of Qh (this thread's own row of it)
                float4 *gp = reinterpret_cast<float4 *>(ws + L.oG + (int64_t)col * kC + i0);
                const float4 qh = *gp;
                *gp = make_float4(qh.x - y[0], qh.y - y[1], qh.z - y[2], qh.w - y[3]);
            } else {
                float *op = ws + L.oO + cv;
#pragma unroll
                for (int r = 0; r < 4; ++r) op[(int64_t)(i0 + r) * Dv] = y[r];
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// Serial part: one CTA per (batch, head, block of NV state columns), through all chunks.

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// acc[r][c] += sum_{k in [k0,k1)} A[k][m0 + r] B[k][n0 + c]: every lane of a warp reads the
// same k row, so both float4 loads are conflict-free.
__device__ __forceinline__ void outer_acc(float acc[16], const float *A, int lda, const float *B,
                                          int ldb, int m0, int n0, int k0, int k1) {
#pragma unroll 4
    for (int kk = k0; kk < k1; ++kk) {
        const float4 av = *reinterpret_cast<const float4 *>(A + kk * lda + m0);
        const float4 bv = *reinterpret_cast<const float4 *>(B + kk * ldb + n0);
        const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(ar[r], br[c], acc[r * 4 + c]);
    }
}

// The same for two A operands sharing B: acc1 += A1^T B and acc2 += A2^T B.
__device__ __forceinline__ void outer_acc2(float acc1[16], float acc2[16], const float *A1,
                                           const float *A2, int lda, const float *B, int ldb,
                                           int m0, int n0, int k0, int k1) {
#pragma unroll 2
    for (int kk = k0; kk < k1; ++kk) {
        const float4 a1 = *reinterpret_cast<const float4 *>(A1 + kk * lda + m0);
        const float4 a2 = *reinterpret_cast<const float4 *>(A2 + kk * lda + m0);
        const float4 bv = *reinterpret_cast<const float4 *>(B + kk * ldb + n0);
        const float r1[4] = {a1.x, a1.y, a1.z, a1.w}, r2[4] = {a2.x, a2.y, a2.z, a2.w};
        const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc1[r * 4 + c] = fmaf(r1[r], br[c], acc1[r * 4 + c]);
                acc2[r * 4 + c] = fmaf(r2[r], br[c], acc2[r * 4 + c]);
            }
    }
}

// Sums the k-split partial tiles into the threads of split 0 (fixed order: deterministic).
// Every thread of the CTA calls it. Partial tiles are stored component-major (slot
// [split][x][tile] of a float4), so the 32 lanes of a warp (32 consecutive tiles) touch 32
// consecutive 16-byte slots.
__device__ __forceinline__ void reduce_splits(float acc[16], float *red, int ks, int KS, int nt,
                                              int tile) {
    if (KS == 1) return;
    if (ks > 0 && ks < KS) {
        float4 *dst = reinterpret_cast<float4 *>(red) + (ks - 1) * 4 * nt + tile;
#pragma unroll
        for (int x = 0; x < 4; ++x)
            dst[x * nt] = make_float4(acc[4 * x], acc[4 * x + 1], acc[4 * x + 2], acc[4 * x + 3]);
    }
    __syncthreads();
    if (ks == 0) {
        for (int s = 1; s < KS; ++s) {
            const float4 *src = reinterpret_cast<const float4 *>(red) + (s - 1) * 4 * nt + tile;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float4 p = src[x * nt];
                acc[4 * x] += p.x;
                acc[4 * x + 1] += p.y;
                acc[4 * x + 2] += p.z;
                acc[4 * x + 3] += p.w;
            }
        }
    }
}

// reduce_splits for a pair of tiles (32 partial values per thread).
__device__ __forceinline__ void reduce_splits2(float acc1[16], float acc2[16], float *red, int ks,
                                               int KS, int nt, int tile) {
    if (KS == 1) return;
    if (ks > 0 && ks < KS) {
        float4 *dst = reinterpret_cast<float4 *>(red) + (ks - 1) * 8 * nt + tile;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            dst[x * nt] = make_float4(acc1[4 * x], acc1[4 * x + 1], acc1[4 * x + 2], acc1[4 * x + 3]);
            dst[(4 + x) * nt] = make_float4(acc2[4 * x], acc2[4 * x + 1], acc2[4 * x + 2], acc2[4 * x + 3]);
        }
    }
    __syncthreads();
    if (ks == 0) {
        for (int sp = 1; sp < KS; ++sp) {
            const float4 *src = reinterpret_cast<const float4 *>(red) + (sp - 1) * 8 * nt + tile;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float4 p1 = src[x * nt], p2 = src[(4 + x) * nt];
                acc1[4 * x] += p1.x; acc1[4 * x + 1] += p1.y; acc1[4 * x + 2] += p1.z; acc1[4 * x + 3] += p1.w;
                acc2[4 * x] += p2.x; acc2[4 * x + 1] += p2.y; acc2[4 * x + 2] += p2.z; acc2[4 * x + 3] += p2.w;
            }
        }
    }
}

template <int NV>
struct ScanSmem {
    static constexpr int S = 0;                          // [Dk][NV] state block
    static constexpr int U = S + kMaxD * NV;             // [64][NV] new values
    static constexpr int W = U + kC * NV;                // [Dk][64]   group A
    static constexpr int G = W + kMaxD * kC;             // [Dk][64]   group A
    static constexpr int UT = G + kMaxD * kC;            // [64][NV]   group A
    static constexpr int OI = UT + kC * NV;              // [64][NV]   group A
    static constexpr int K = OI + kC * NV;               // [64][Dk]   group B
    static constexpr int C = K + kC * kMaxD;             // [4]        group B
    static constexpr int RED = C + 4;                    // k-split partial tiles
    static constexpr int kRedFloats = 3 * 64 * 32;       // at most (splits - 1) x tiles x 32
    static constexpr int kFloats = RED + kRedFloats;
};

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads, 1) gdn_scan_kernel(GdnArgs a) {
    using SM = ScanSmem<NV>;
    extern __shared__ __align__(16) float sm[];
    float *S = sm + SM::S, *U = sm + SM::U, *Wt = sm + SM::W, *Gt = sm + SM::G;
    float *Ut = sm + SM::UT, *Oi = sm + SM::OI, *Kh = sm + SM::K, *gc = sm + SM::C;
    float *red = sm + SM::RED;
    const int tid = threadIdx.x;
    const int nvb = a.Dv / NV;
    const int64_t bh = blockIdx.x / nvb;
    const int v0 = (int)(blockIdx.x % nvb) * NV;
    const int64_t bb = bh / a.H, h = bh % a.H;
    const int Dk = a.Dk, Dv = a.Dv, n = a.nchunks;
    const WsLayout L(Dk, Dv);
    const float *wsh = a.ws + bh * n * L.total;   // this head's chunks
    T *o = static_cast<T *>(a.o);

    auto issue_a = [&](int c) {
        if (c < n) {
            const float *src = wsh + (int64_t)c * L.total;
            for (int i = tid; i < Dk * kC / 4; i += kThreads) {
                cp16(Wt + 4 * i, src + L.oW + 4 * i);
                cp16(Gt + 4 * i, src + L.oG + 4 * i);
            }
            for (int i = tid; i < kC * NV / 4; i += kThreads) {
                const int j = i / (NV / 4), x = i % (NV / 4);
                cp16(Ut + j * NV + 4 * x, src + L.oU + (int64_t)j * Dv + v0 + 4 * x);
                cp16(Oi + j * NV + 4 * x, src + L.oO + (int64_t)j * Dv + v0 + 4 * x);
            }
        }
        cp_commit();
    };
    auto issue_b = [&](int c) {
        if (c < n) {
            const float *src = wsh + (int64_t)c * L.total;
            for (int i = tid; i < kC * Dk / 4; i += kThreads) cp16(Kh + 4 * i, src + L.oK + 4 * i);
            if (tid == 0) cp16(gc, src + L.oC);
        }
        cp_commit();
    };

    // state block from h0 (or zero)
    for (int i = tid; i < Dk * NV; i += kThreads) {
        const int d = i / NV, x = i % NV;
        S[i] = a.h0 ? a.h0[(bh * Dk + d) * Dv + v0 + x] : 0.f;
    }
    issue_a(0);
    issue_b(0);

    // tile maps: U and O are [64][NV] (nt1 tiles), the state is [Dk][NV] (nt3 tiles); a
    // tile's contraction is split over up to 4 groups of warps (the partial-tile buffer)
    const int nt1 = 16 * (NV / 4), ks1n = min(kThreads / nt1, 4);
    const int ks1 = tid / nt1, tile1 = tid % nt1;
    const int m1 = 4 * (tile1 / (NV / 4)), n1 = 4 * (tile1 % (NV / 4));
    const int nt3 = (Dk / 4) * (NV / 4), ks3n = min(kThreads / nt3, 4);
    const int ks3 = tid / nt3, tile3 = tid % nt3;
    const int m3 = 4 * (tile3 / (NV / 4)), n3 = 4 * (tile3 % (NV / 4));

    for (int c = 0; c < n; ++c) {
        // ---- U = Ut - W S and O = Oi + G S (one pass over the key dims of S)
        cp_wait1();
        __syncthreads();
        {
            float aw[16], ag[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) aw[x] = ag[x] = 0.f;
            if (ks1 < ks1n)
                outer_acc2(aw, ag, Wt, Gt, kC, S, NV, m1, n1, ks1 * Dk / ks1n, (ks1 + 1) * Dk / ks1n);
            reduce_splits2(aw, ag, red, ks1, ks1n, nt1, tile1);
            if (ks1 == 0) {
                const int64_t tbase = (int64_t)c * kC;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float4 ut = *reinterpret_cast<const float4 *>(Ut + (m1 + r) * NV + n1);
                    *reinterpret_cast<float4 *>(U + (m1 + r) * NV + n1) =
                        make_float4(ut.x - aw[4 * r], ut.y - aw[4 * r + 1], ut.z - aw[4 * r + 2],
                                    ut.w - aw[4 * r + 3]);
                    const int64_t t = tbase + m1 + r;
                    if (t < a.T) {
                        const float4 oi = *reinterpret_cast<const float4 *>(Oi + (m1 + r) * NV + n1);
                        const int64_t off = ((bb * a.T + t) * a.H + h) * Dv + v0 + n1;
                        st_io(o, off, oi.x + ag[4 * r]);
                        st_io(o, off + 1, oi.y + ag[4 * r + 1]);
                        st_io(o, off + 2, oi.z + ag[4 * r + 2]);
                        st_io(o, off + 3, oi.w + ag[4 * r + 3]);
                    }
                }
            }
        }
        __syncthreads();
        issue_a(c + 1);
        // ---- S = exp(b_63) S + Kh^T U
        cp_wait1();
        __syncthreads();
        {
            float acc[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = 0.f;
            if (ks3 < ks3n)
                outer_acc(acc, Kh, Dk, U, NV, m3, n3, ks3 * kC / ks3n, (ks3 + 1) * kC / ks3n);
            reduce_splits(acc, red, ks3, ks3n, nt3, tile3);
            if (ks3 == 0) {
                const float dec = gc[0];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    float4 *sp = reinterpret_cast<float4 *>(S + (m3 + r) * NV + n3);
                    const float4 s = *sp;
                    *sp = make_float4(fmaf(dec, s.x, acc[4 * r]), fmaf(dec, s.y, acc[4 * r + 1]),
                                      fmaf(dec, s.z, acc[4 * r + 2]), fmaf(dec, s.w, acc[4 * r + 3]));
                }
            }
        }
        __syncthreads();
        issue_b(c + 1);
    }
    cp_wait0();
    if (a.hT) {
        for (int i = tid; i < Dk * NV; i += kThreads) {
            const int d = i / NV, x = i % NV;
            a.hT[(bh * Dk + d) * Dv + v0 + x] = S[i];
        }
    }
}

constexpr size_t kPrepSmem = (size_t)(2 * kMaxD * kPrepStride + 2 * kC * kC + 5 * kC) * sizeof(float);

template <typename T>
cudaError_t launch_typed(const GdnArgs &a, int64_t BH, int num_sms, cudaStream_t s) {
    const int64_t nprep = BH * a.nchunks;
    cudaError_t e = cudaFuncSetAttribute(gdn_prep_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    gdn_prep_kernel<T><<<(unsigned)nprep, kThreads, kPrepSmem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 16 state columns per CTA where 32 would leave SMs idle
    const bool narrow = BH * (a.Dv / 32) < num_sms || a.Dv % 32 != 0;
    if (narrow) {
        const size_t smem = ScanSmem<16>::kFloats * sizeof(float);
        e = cudaFuncSetAttribute(gdn_scan_kernel<T, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        gdn_scan_kernel<T, 16><<<(unsigned)(BH * (a.Dv / 16)), kThreads, smem, s>>>(a);
    } else {
        const size_t smem = ScanSmem<32>::kFloats * sizeof(float);
        e = cudaFuncSetAttribute(gdn_scan_kernel<T, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        gdn_scan_kernel<T, 32><<<(unsigned)(BH * (a.Dv / 32)), kThreads, smem, s>>>(a);
    }
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(2);
    return e;
}

}  // namespace

bool gdn_supported(int64_t Dk, int64_t Dv) {
    return Dk >= 4 && Dk <= kMaxD && Dk % 4 == 0 && Dv >= 16 && Dv <= kMaxD && Dv % 16 == 0;
}

size_t gdn_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv) {
    const int64_t nchunks = (T + kC - 1) / kC;
    return (size_t)(B * H * nchunks) * (size_t)WsLayout((int)Dk, (int)Dv).total * sizeof(float);
}

cudaError_t launch_gdn(const GdnProblem &p, void *ws, int num_sms, cudaStream_t s) {
    GdnArgs a;
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.g = p.g;
    a.beta = p.beta;
    a.scale = p.scale;
    a.h0 = p.h0;
    a.o = p.o;
    a.hT = p.hT;
    a.T = p.T;
    a.H = (int)p.H;
    a.Dk = (int)p.Dk;
    a.Dv = (int)p.Dv;
    a.nchunks = (int)((p.T + kC - 1) / kC);
    a.ws = static_cast<float *>(ws);
    const int64_t BH = p.B * p.H;
    return p.io == 0 /* bf16 */ ? launch_typed<__nv_bfloat16>(a, BH, num_sms, s)
                     : launch_typed<float>(a, BH, num_sms, s);
}

}  // namespace gla
