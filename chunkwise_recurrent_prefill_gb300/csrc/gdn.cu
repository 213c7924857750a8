// Gated delta rule forward (prefill), chunkwise. bf16 I/O at head dims 128 runs on the
// tensor cores (gdn_tc_prep_kernel: tcgen05 bf16 products; gdn_tc_scan_kernel: tcgen05 tf32
// products with the fp32 state in TMEM); every other case runs the fp32 CUDA-core pair
// gdn_prep_kernel / gdn_scan_kernel, which take the same chunk algebra.
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
// factors) is computed for all chunks at once by the prep kernel and written to a workspace;
// the state then runs through the chunks in the scan kernel, which forms U and O from S0 in
// one pass and then S1. The fp32 scan runs one CTA per (batch, head, block of state columns):
// the columns of S are independent under this recurrence (the transition acts on the key
// axis only), which is what lets B = 1 spread over many SMs; the tensor-core scan keeps the
// whole 128 x 128 state of one (batch, head) in TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "gla_internal.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

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

// x -> (hi, lo) bf16 pairs with hi = bf16(x), lo = bf16(x - hi), two elements per word
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = tc::pack_bf16(x0, x1);
    const float2 f = tc::unpack_bf16(hi);
    lo = tc::pack_bf16(x0 - f.x, x1 - f.y);
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

// Workspace of the tensor-core scan (bf16 I/O, Dk = Dv = 128): one array per quantity, so
// that each is a plain 2-D tensor the scan can tile with TMA. For chunk blk = bh * nchunks + c:
//   W [blk][64][Dk]    G [blk][64][Dk]    U [blk][64][Dv]    O [blk][64][Dv]
//   EK [blk][64] (e^(b_63 - b_j), the decay from token j to the chunk's end)
//   C [blk] (b_63, the chunk's summed log-gate)
// (the scan takes k itself, in bf16, for the state update). It fits in the per-chunk layout
// above, which sizes the workspace of both routes.
struct SoA {
    float *W, *G, *U, *O, *EK, *C;
    __host__ __device__ SoA(float *ws, int64_t nblk, int Dk, int Dv) {
        W = ws;
        G = W + nblk * kC * Dk;
        U = G + nblk * kC * Dk;
        O = U + nblk * kC * Dv;
        EK = O + nblk * kC * Dv;
        C = EK + nblk * kC;
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
    int64_t nblk;            // B * H * nchunks (structure-of-arrays workspace)
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
            if (isk) {   // G = Qh - P W, in place of Qh (this thread's own column of it)
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

// ---------------------------------------------------------------------------------------
// Serial part on the tensor cores (bf16 I/O, Dk = Dv = 128): one CTA per (batch, head) and
// segment of its chunks (see ScanPlan), the fp32 state kept in TMEM across the segment's
// chunks, transposed (lane = value column v, column = key
// row d) and decay-normalised: S = 2^L S~ with one scalar L per head (the gate is one per
// token). Per chunk c, with the prep's W, G, Ut, Oi, e^(b_63 - b_j) and b_63, and k:
//   [W S | G S]^T = S~^T [W | G]^T 2^L    one MMA chain, A = S~^T straight from TMEM (tf32)
//   U = Ut - 2^L (W S~),  O = Oi + 2^L (G S~)                      (CUDA cores, fp32)
//   S~ += sum_j (2^-L' e^(b_63 - b_j) U_j)^T k_j,  L' = L + b_63 log2(e):  A = the scaled U^T
//   from TMEM as a bf16 hi / lo pair (about 16 significant bits), B = k exact in bf16
// The state is rescaled (S~ <- 2^L' S~, L' <- 0) when |L'| passes kRenormL2, before the
// update that would use it; a full-forgetting chunk (b_63 very negative) so zeroes S~.
// The tf32 products W S~ and G S~ (10-bit mantissa) keep the output far inside the bf16
// tolerance, and the split-precision update keeps the final state within about 1e-5 of the
// fp64 recurrence (mean relative error over every head of the full-size workloads).
namespace gt {
constexpr int kStages = 2;
// stage: four [W | G] slabs (dk 32 s .. 32 s + 31: W rows then G rows, 128 rows x 128 B,
// 128B-swizzled, one swizzle atom per 8 rows), the chunk's k (bf16, two 128B-swizzled
// [64 tokens x 64 dk] boxes) and its 64 decay factors e^(b_63 - b_j)
constexpr uint32_t WG = 0, WGSLAB = 16384, KB = 65536, EKO = 81920, STAGE = 82944;
constexpr uint32_t BAR = kStages * STAGE;
constexpr uint32_t NBAR = 12;
constexpr uint32_t TSLOT = BAR + NBAR * 8;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
// TMEM columns
constexpr uint32_t kS = 0;       // S~^T, 128 columns
constexpr uint32_t kWG = 128;    // [W S~ | G S~]^T, 2 x 128 columns (double buffered)
constexpr uint32_t kU = 384;     // scaled U^T as bf16 hi (32 columns) and lo (32 columns):
                                 // the A operand of the update
constexpr int kThreadsTC = 18 * 32;   // producer, MMA issuer, 8 U warps, 8 O warps
constexpr float kRenormL2 = 60.f;
enum { FULL = 0, EMPTY = 2, WGD = 4, WGF = 6, URDY = 8, FIN = 9 };
}  // namespace gt

// Sequence split of the tensor-core scan. The chunk map S1 = (e^(b_63) I - Kh^T W) S0 +
// Kh^T Ut is affine in the state, so a segment of chunks maps its start state S to M S + E,
// with E its end state from a zero start and M (Dk x Dk) its end state from the identity with
// Ut = 0 (the value columns of the state are independent, so M is the same recurrence with
// Dk columns). Segment 0 starts from h0, which is known: its outputs run in the first
// launch (mode 1), and its end state is the start state of segment 1. Beside them, two CTAs
// per segment compute E and M of segments 1 .. segs - 2. gdn_seg_scan_kernel then forms
// S_start(s + 1) = M_s S_start(s) + E_s, and the second launch (mode 0) runs the outputs of
// segments 1 .. segs - 1 from their start states. Segment 0 is half as long as the others:
// a transition chunk costs about half an output chunk.
struct ScanPlan {
    int segs;          // segments per (batch, head); 1 = no split
    int mode;          // 0: outputs of segments s0 .. segs - 1; 1: see above
    int s0;            // first segment of a mode-0 launch
    float *E;          // [BH][segs - 1][Dk][Dv] (entries 1 .. segs - 2 used)
    float *M;          // [BH][segs - 1][Dk][Dk] (entries 1 .. segs - 2 used)
    float *Ss;         // [BH][segs - 1][Dk][Dv]: start states of segments 1 .. segs - 1
};

// First chunk of segment s of a split into `segs` (s = segs gives n): segment 0 weighs 1,
// every other segment 2.
__device__ __host__ __forceinline__ int gdn_seg_bound(int s, int n, int segs) {
    if (segs <= 1) return s == 0 ? 0 : n;
    if (s <= 0) return 0;
    if (s >= segs) return n;
    return (int)((int64_t)n * (2 * s - 1) / (2 * segs - 1));
}

// tcgen05.mma kind::tf32 with A from TMEM: D (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for kind::tf32, fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format: f32
           | (2u << 7)          // A format: tf32
           | (2u << 10)         // B format: tf32
           | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 2-D tiled load (x = inner coordinate, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, uint64_t *bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(tc::smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__global__ void __launch_bounds__(gt::kThreadsTC, 1)
gdn_tc_scan_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tg,
                   const __grid_constant__ CUtensorMap tk4, const __grid_constant__ CUtensorMap tek,
                   GdnArgs a, ScanPlan sp, unsigned *err) {
    using namespace gt;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                              ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TSLOT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA -> (batch and head, segment, output or transition, and of a transition E or M)
    const int64_t BH = a.nblk / a.nchunks;
    bool trans = false;
    int seg = 0, part = 0;   // part 1: the linear part M
    int64_t bh = 0;
    if (sp.mode == 0) {
        const int nout = sp.segs - sp.s0;
        seg = sp.s0 + (int)(blockIdx.x % nout);
        bh = blockIdx.x / nout;
    } else if ((int64_t)blockIdx.x < BH) {
        bh = blockIdx.x;   // segment 0's outputs
    } else {
        const int64_t t = blockIdx.x - BH;
        trans = true;
        part = (int)(t & 1);
        seg = 1 + (int)((t >> 1) % (sp.segs - 2));
        bh = (t >> 1) / (sp.segs - 2);
    }
    const int64_t bb = bh / a.H, h = bh % a.H;
    const int cb = gdn_seg_bound(seg, a.nchunks, sp.segs);
    const int ce = gdn_seg_bound(seg + 1, a.nchunks, sp.segs);
    const int n = ce - cb;                     // chunks of this segment
    const int64_t blk0 = bh * a.nchunks + cb;  // workspace index of its first chunk
    const SoA so(a.ws, a.nblk, kMaxD, kMaxD);
    const bool lin = trans && part == 1;       // Ut = 0, no outputs
    // start state: h0, a segment start state, zero (E) or the identity (M)
    const float *init = trans ? nullptr
                      : seg == 0 ? (a.h0 ? a.h0 + bh * kMaxD * kMaxD : nullptr)
                                 : sp.Ss + (bh * (sp.segs - 1) + seg - 1) * kMaxD * kMaxD;
    // final state: hT after the last segment; the start state of segment 1 after segment 0;
    // E or M of a transition
    float *fin = trans ? (part ? sp.M : sp.E) + (bh * (sp.segs - 1) + seg) * kMaxD * kMaxD
               : seg == sp.segs - 1 ? (a.hT ? a.hT + bh * kMaxD * kMaxD : nullptr)
               : seg == 0 ? sp.Ss + bh * (sp.segs - 1) * kMaxD * kMaxD : nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&bars[FULL + i], 1);
            tc::mbar_init(&bars[EMPTY + i], 1);
            tc::mbar_init(&bars[WGD + i], 1);
            tc::mbar_init(&bars[WGF + i], 8);
        }
        tc::mbar_init(&bars[URDY], 8);
        tc::mbar_init(&bars[FIN], 1);
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&tw);
        tc::tma_prefetch_desc(&tg);
        tc::tma_prefetch_desc(&tk4);
        tc::tma_prefetch_desc(&tek);
    }
    if (warp == 1) tc::tmem_alloc(tslot, 512);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *tslot;
    // the initial state, transposed into TMEM (U warps: lane quarter j, key rows of their half)
    if (warp >= 2 && warp < 10) {
        const int j = warp & 3, half = (warp - 2) >> 2, v = j * 32 + lane;
#pragma unroll 1
        for (int d0 = 64 * half; d0 < 64 * half + 64; d0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int x = 0; x < 16; ++x)
                r[x] = lin ? (d0 + x == v ? 0x3f800000u : 0u)
                           : init ? __float_as_uint(init[(d0 + x) * kMaxD + v]) : 0u;
            tc::tmem_st16(tc::tmem_addr(tm, j, kS + d0), r);
        }
        tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    bool ok = true;

    if (warp == 0) {
        // ---- TMA producer: [W | G] slabs, k and the decay factors of each chunk
        if (lane == 0) {
            int issued = 0;
            // the fp32 Ut and Oi tiles the U and O warps read with plain loads: brought into L2
            // two chunks ahead, so their loads do not wait on DRAM
            constexpr uint32_t kTile = kC * kMaxD * sizeof(float);
            // (a transition reads no Oi, and its linear part no Ut)
            for (int c = 0; c < 2 && c < n; ++c) {
                if (!lin) prefetch_l2(so.U + (blk0 + c) * kC * kMaxD, kTile);
                if (!trans) prefetch_l2(so.O + (blk0 + c) * kC * kMaxD, kTile);
            }
            for (int c = 0; c < n && ok; ++c) {
                const int st = c % kStages;
                if (c + 2 < n) {
                    if (!lin) prefetch_l2(so.U + (blk0 + c + 2) * kC * kMaxD, kTile);
                    if (!trans) prefetch_l2(so.O + (blk0 + c + 2) * kC * kMaxD, kTile);
                }
                if (c >= kStages && !tc::mbar_wait(&bars[EMPTY + st], ((c / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &bars[FULL + st];
                // a transition multiplies by W only: no G slabs
                tc::mbar_arrive_expect_tx(fb, (trans ? 32768u : 65536u) + 16384u + 256u);
                uint8_t *base = sm + st * STAGE;
                const int row = (int)((blk0 + c) * kC);
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    tma_load_2d(base + WG + sl * WGSLAB, &tw, fb, 32 * sl, row);
                    if (!trans) tma_load_2d(base + WG + sl * WGSLAB + 8192, &tg, fb, 32 * sl, row);
                }
                // k of the chunk (rows past the sequence end read as zero) and its decay factors
                const int tk = (int)((int64_t)(cb + c) * kC);
                tc::tma_load_4d(base + KB, &tk4, fb, 0, (int)h, tk, (int)bb);
                tc::tma_load_4d(base + KB + 8192, &tk4, fb, 64, (int)h, tk, (int)bb);
                tma_load_2d(base + EKO, &tek, fb, 0, (int)(blk0 + c));
                ++issued;
            }
            // no bulk copy may still be landing when the CTA exits
            for (int i = 0; i < kStages && i < issued; ++i) {
                const int uses = (issued - 1 - i) / kStages + 1;
                if (!tc::mbar_wait(&bars[FULL + i], (uses - 1) & 1)) ok = false;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer (converged warp, one elected lane issues)
        // a transition needs W S~ only: N = 64 (the W rows of each slab)
        const uint32_t idWG = idesc_tf32(128, trans ? 64 : 128);
        const uint32_t idUP = tc::idesc_bf16(128, 128, 0, 1);   // A from TMEM, k MN-major
        for (int c = 0; c < n; ++c) {
            const int st = c % kStages, wb = c & 1;
            bool w = tc::mbar_wait(&bars[FULL + st], (c / kStages) & 1);
            if (w && c >= 2) w = tc::mbar_wait(&bars[WGF + wb], ((c >> 1) - 1) & 1);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc::tc_fence_after();
            const uint32_t base = tc::smem_u32(sm + st * STAGE);
            if (tc::elect_one()) {
                // [W S~ | G S~]^T: K = 128 key rows in 16 steps of 8 (32 bytes of a slab row)
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    mma_tf32_ts(tm + kWG + wb * 128, tm + kS + kk * 8,
                                tc::smem_desc(base + WG + (kk >> 2) * WGSLAB + (kk & 3) * 32, 16, 1024),
                                idWG, kk > 0);
                tc::mma_commit(&bars[WGD + wb]);
            }
            __syncwarp();
            w = tc::mbar_wait(&bars[URDY], c & 1);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc::tc_fence_after();
            if (tc::elect_one()) {
                // S~^T += (scaled U)^T k: K = 64 tokens in 4 steps of 16, U hi then U lo
#pragma unroll
                for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ts(tm + kS, tm + kU + hl * 32 + kk * 8,
                                   tc::smem_desc(base + KB + kk * 2048, 8192, 1024), idUP, 1);
                tc::mma_commit(&bars[EMPTY + st]);   // the stage's last reader
            }
            __syncwarp();
        }
        if (tc::elect_one()) tc::mma_commit(&bars[FIN]);
        __syncwarp();
        if (!tc::mbar_wait(&bars[FIN], 0)) ok = false;
    } else if (warp < 10) {
        // ---- U warps: U = Ut - 2^L (W S~), scaled by 2^-L' into TMEM; rescale S~ when due
        const int j = warp & 3, half = (warp - 2) >> 2, v = j * 32 + lane;
        const int t0 = 32 * half;
        float L = 0.f;
        float ut[32];
        auto load_ut = [&](int c) {
            const float *src = so.U + ((blk0 + c) * kC + t0) * kMaxD + v;
#pragma unroll
            for (int x = 0; x < 32; ++x) ut[x] = lin ? 0.f : src[x * kMaxD];
        };
        if (n > 0) load_ut(0);
        for (int c = 0; c < n; ++c) {
            const float bsum = so.C[blk0 + c];
            const bool w = tc::mbar_wait(&bars[WGD + (c & 1)], (c >> 1) & 1);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc::tc_fence_after();
            float acc[32];
            {
                uint32_t r0[16], r1[16];
                tc::tmem_ld16(tc::tmem_addr(tm, j, kWG + (c & 1) * 128 + t0), r0);
                tc::tmem_ld16(tc::tmem_addr(tm, j, kWG + (c & 1) * 128 + t0 + 16), r1);
                tc::tmem_wait_ld();
                tc::reg_fence(r0);
                tc::reg_fence(r1);
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    acc[x] = __uint_as_float(r0[x]);
                    acc[16 + x] = __uint_as_float(r1[x]);
                }
            }
            const float eL = ex2f(L);
            float Ln = L + bsum * 1.4426950408889634f;
            const bool ren = !(fabsf(Ln) <= kRenormL2);   // also on NaN
            if (ren) {
                // every MMA reading S~ for this chunk (the [W | G] chain) has completed: scale
                // this warp's lane quarter, key rows of its half, by 2^L'
                const float f = ex2f(Ln);
#pragma unroll 1
                for (int d0 = 64 * half; d0 < 64 * half + 64; d0 += 16) {
                    uint32_t r[16];
                    tc::tmem_ld16(tc::tmem_addr(tm, j, kS + d0), r);
                    tc::tmem_wait_ld();
                    tc::reg_fence(r);
#pragma unroll
                    for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * f);
                    tc::tmem_st16(tc::tmem_addr(tm, j, kS + d0), r);
                }
                Ln = 0.f;
            }
            const float su = ex2f(-Ln);
            // decay factors of the chunk's tokens, in its stage (live until the update completes;
            // the stage's barrier has completed, and cannot move on before this chunk's update)
            if (!tc::mbar_wait(&bars[FULL + c % kStages], (c / kStages) & 1)) ok = false;
            const float *eks = reinterpret_cast<const float *>(sm + (c % kStages) * STAGE + EKO) + t0;
            uint32_t uh[16], ul[16];   // tokens t0 .. t0 + 31 in pairs: bf16 hi and lo
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const float a0 = (ut[2 * x] - eL * acc[2 * x]) * su * eks[2 * x];
                const float a1 = (ut[2 * x + 1] - eL * acc[2 * x + 1]) * su * eks[2 * x + 1];
                split2(a0, a1, uh[x], ul[x]);
            }
            tc::tmem_st16(tc::tmem_addr(tm, j, kU + half * 16), uh);
            tc::tmem_st16(tc::tmem_addr(tm, j, kU + 32 + half * 16), ul);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[URDY]);
            L = Ln;
            if (c + 1 < n) load_ut(c + 1);
        }
        // final state 2^L S~ (transposed back: hT, or E / M of a transition), once every
        // update has completed
        if (ok && fin) {
            if (!tc::mbar_wait(&bars[FIN], 0)) {
                ok = false;
            } else {
                tc::tc_fence_after();
                const float eL = ex2f(L);
#pragma unroll 1
                for (int d0 = 64 * half; d0 < 64 * half + 64; d0 += 16) {
                    uint32_t r[16];
                    tc::tmem_ld16(tc::tmem_addr(tm, j, kS + d0), r);
                    tc::tmem_wait_ld();
                    tc::reg_fence(r);
#pragma unroll
                    for (int x = 0; x < 16; ++x)
                        fin[(d0 + x) * kMaxD + v] = __uint_as_float(r[x]) * eL;
                }
            }
        }
    } else {
        // ---- O warps: o = Oi + 2^L (G S~), rounded to bf16 and stored
        const int j = warp & 3, v = j * 32 + lane, th = 32 * ((warp - 10) >> 2);
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);
        float L = 0.f;
        float oi[32];
        auto load_oi = [&](int c) {
            const float *src = so.O + ((blk0 + c) * kC + th) * kMaxD + v;
#pragma unroll
            for (int x = 0; x < 32; ++x) oi[x] = src[x * kMaxD];
        };
        if (n > 0 && !trans) load_oi(0);
        for (int c = 0; c < n; ++c) {
            const float bsum = so.C[blk0 + c];
            const bool w = tc::mbar_wait(&bars[WGD + (c & 1)], (c >> 1) & 1);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc::tc_fence_after();
            if (trans) {   // no outputs: only hand the accumulator back
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[WGF + (c & 1)]);
                continue;
            }
            const float eL = ex2f(L);
            const int64_t tb = (int64_t)(cb + c) * kC;
            const int vr = (int)(a.T - tb < kC ? a.T - tb : kC);
            __nv_bfloat16 *op = o + ((bb * a.T + tb) * a.H + h) * kMaxD + v;
            const int64_t rs = (int64_t)a.H * kMaxD;
            {
                uint32_t r0[16], r1[16];
                tc::tmem_ld16(tc::tmem_addr(tm, j, kWG + (c & 1) * 128 + 64 + th), r0);
                tc::tmem_ld16(tc::tmem_addr(tm, j, kWG + (c & 1) * 128 + 64 + th + 16), r1);
                tc::tmem_wait_ld();
                tc::reg_fence(r0);
                tc::reg_fence(r1);
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[WGF + (c & 1)]);   // the accumulator is free
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int t = th + x;
                    if (t < vr) op[t * rs] = __float2bfloat16_rn(oi[x] + eL * __uint_as_float(r0[x]));
                }
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int t = th + 16 + x;
                    if (t < vr) op[t * rs] = __float2bfloat16_rn(oi[16 + x] + eL * __uint_as_float(r1[x]));
                }
            }
            float Ln = L + bsum * 1.4426950408889634f;
            if (!(fabsf(Ln) <= kRenormL2)) Ln = 0.f;   // the U warps rescaled S~ here
            L = Ln;
            if (c + 1 < n) load_oi(c + 1);
        }
    }

    if (!ok) atomicOr(err, kDevErrTimeout);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tm, 512);
    }
}

// ---------------------------------------------------------------------------------------
// Tensor-core prep (bf16 I/O, Dk = Dv = 128): one CTA per (batch, head, chunk), two CTAs per
// SM. The chunk's contractions run on tcgen05 with bf16 operands and fp32 accumulation in
// TMEM; the triangular inverse stays in fp32 on the CUDA cores:
//   [K K^T ; Q K^T]                       (K, Q exact in bf16)       -> A, P
//   T = (I + A)^-1                        forward substitution, one column per thread
//   [P Tw | P Tu]^T = [Tw | Tu]^T P^T     Tw = T diag(beta e^b),  Tu = T diag(beta)
//   [W ; -P W] = [Tw ; -P Tw] K           (W = Tw K solves (I + A) W = diag(beta e^b) K)
//   [Ut ; Oi]  = [Tu ;  P Tu] V           (Ut solves (I + A) Ut = diag(beta) V, Oi = P Ut)
// and G = scale diag(e^b) Q - P W is finished in the epilogue. Each fp32 coefficient matrix
// enters the tensor cores as two bf16 operands, hi = bf16(x) and lo = bf16(x - hi), and a
// product of two such matrices takes hi*hi + lo*hi + hi*lo: about 16 significant bits (the
// scan then reads these tiles as tf32, 11 bits). The results leave through 128B-swizzled
// shared-memory staging and TMA tensor stores, in the structure-of-arrays workspace layout.
namespace gp {
// shared memory (bytes from the 1024-aligned base); every operand tile is 64 rows x 128 B,
// 128B-swizzled (8 KB)
constexpr uint32_t KQ = 0;          // k d0..63 | q d0..63 | k d64..127 | q d64..127
constexpr uint32_t V = 32768;       // v d0..63 | v d64..127
constexpr uint32_t TT = 49152;      // T (fp32) and merge scratch; then
                                    // Tw^T hi | Tu^T hi | Tw^T lo | Tu^T lo   (row m, column j)
constexpr uint32_t AP = 81920;      // A (fp32, stride kAStride); then P hi | lo; then
                                    // (-P Tw)^T hi | lo; then (P Tu)^T hi | lo (row m, column i)
constexpr uint32_t SMALL = AP + 18432;   // b, beta, e^b, beta e^b, e^(b63 - b), b log2(e)
constexpr uint32_t BAR = SMALL + 6 * 256;
constexpr uint32_t NBAR = 5;
constexpr uint32_t TSLOT = BAR + NBAR * 8;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
constexpr uint32_t ST0 = 32768, ST1 = 65536;   // fp32 output staging once the MMAs are done
constexpr int kAStride = 68;
constexpr int kThreadsP = 256;
// TMEM columns (256 allocated): [KK^T ; QK^T] at 0 (64 columns), [P Tw | P Tu]^T at 64
// (64), [W ; -P W] at 128 (128), [Ut ; Oi] at 0 (128, after the first two are read)
constexpr uint32_t kD1 = 0, kD2 = 64, kD3 = 128, kD4 = 0;
enum { LOAD = 0, M1 = 1, M2 = 2, M3 = 3, M4 = 4 };
}  // namespace gp

// Load 64 consecutive TMEM columns of this warp's lane quarter as fp32 (one wait).
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&out)[64]) {
    uint32_t r0[16], r1[16], r2[16], r3[16];
    tc::tmem_ld16(taddr, r0);
    tc::tmem_ld16(taddr + 16, r1);
    tc::tmem_ld16(taddr + 32, r2);
    tc::tmem_ld16(taddr + 48, r3);
    tc::tmem_wait_ld();
    tc::reg_fence(r0);
    tc::reg_fence(r1);
    tc::reg_fence(r2);
    tc::reg_fence(r3);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        out[x] = __uint_as_float(r0[x]);
        out[16 + x] = __uint_as_float(r1[x]);
        out[32 + x] = __uint_as_float(r2[x]);
        out[48 + x] = __uint_as_float(r3[x]);
    }
}


// Row `row` of a 64-column bf16 operand tile pair (hi at `hi`, lo at `lo`, 128B-swizzled):
// the 64 values x[0..63] scaled by f.
__device__ __forceinline__ void store_split_row(uint8_t *hi, uint8_t *lo, int row,
                                                const float (&x)[64], float f) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) split2(f * x[8 * ch + 2 * p], f * x[8 * ch + 2 * p + 1], h[p], l[p]);
        const uint32_t off = tc::sw128_offset(row, 8 * ch);
        *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// 64 fp32 values of row `row` into a staged [rows x 128] fp32 tile held as four
// 128B-swizzled boxes of 32 columns (8 KB each for 64 rows), columns c0 .. c0 + 63.
__device__ __forceinline__ void stage_row64(uint8_t *tile, int row, int c0, const float (&v)[64]) {
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) {
        const int col = c0 + 4 * c4, box = col >> 5, ch = (col & 31) >> 2;
        *reinterpret_cast<float4 *>(tile + box * 8192 + row * 128 + ((ch ^ (row & 7)) << 4)) =
            make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
    }
}

// 2-D tiled bulk tensor store from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(tc::smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}

__global__ void __launch_bounds__(gp::kThreadsP, 2)
gdn_tc_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tw,
                   const __grid_constant__ CUtensorMap tg, const __grid_constant__ CUtensorMap tu,
                   const __grid_constant__ CUtensorMap to, GdnArgs a, unsigned *err) {
    using namespace gp;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                              ~uintptr_t(1023));
    float *bs = reinterpret_cast<float *>(sm + SMALL);   // cumulative log-gate b_j
    float *be = bs + kC;                                 // beta_j
    float *eb = be + kC;                                 // e^(b_j)
    float *bg = eb + kC;                                 // beta_j e^(b_j)
    float *ek = bg + kC;                                 // e^(b_63 - b_j)
    float *bl = ek + kC;                                 // b_j log2(e)
    float *As = reinterpret_cast<float *>(sm + AP);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TSLOT);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t blk = blockIdx.x;
    const int c = (int)(blk % a.nchunks);
    const int64_t bh = blk / a.nchunks;
    const int64_t bb = bh / a.H, h = bh % a.H;
    const int64_t t0 = (int64_t)c * kC;
    const int nval = (int)(a.T - t0 < kC ? a.T - t0 : kC);
    const uint32_t base = tc::smem_u32(sm);
    const SoA so(a.ws, a.nblk, kMaxD, kMaxD);
    bool ok = true;

    if (warp == 1) {
        if (lane == 0) {   // barriers, then the q, k, v tiles (rows past the end read as zero)
            for (int i = 0; i < (int)NBAR; ++i) tc::mbar_init(&bars[i], 1);
            tc::fence_mbar_init();
            uint64_t *lb = &bars[LOAD];
            tc::mbar_arrive_expect_tx(lb, 6 * 8192);
            const int tt = (int)t0, hh = (int)h, b4 = (int)bb;
            tc::tma_load_4d(sm + KQ, &tk, lb, 0, hh, tt, b4);
            tc::tma_load_4d(sm + KQ + 8192, &tq, lb, 0, hh, tt, b4);
            tc::tma_load_4d(sm + KQ + 16384, &tk, lb, 64, hh, tt, b4);
            tc::tma_load_4d(sm + KQ + 24576, &tq, lb, 64, hh, tt, b4);
            tc::tma_load_4d(sm + V, &tv, lb, 0, hh, tt, b4);
            tc::tma_load_4d(sm + V + 8192, &tv, lb, 64, hh, tt, b4);
        }
        // gates, two tokens per lane; rows past the sequence end decay by nothing and write
        // nothing. Inclusive cumulative sum: pair sums, then a warp scan.
        const int j0 = 2 * lane;
        float g0 = 0.f, g1 = 0.f, be0 = 0.f, be1 = 0.f;
        const int64_t r0 = (bb * a.T + t0 + j0) * a.H + h;
        if (j0 < nval) { g0 = a.g[r0]; be0 = a.beta[r0]; }
        if (j0 + 1 < nval) { g1 = a.g[r0 + a.H]; be1 = a.beta[r0 + a.H]; }
        float inc = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        float ex = __shfl_up_sync(0xffffffffu, inc, 1);
        if (lane == 0) ex = 0.f;
        const float c0 = ex + g0, c1 = c0 + g1;
        const float l63 = __shfl_sync(0xffffffffu, c1, 31) * 1.4426950408889634f;
        const float l0 = c0 * 1.4426950408889634f, l1 = c1 * 1.4426950408889634f;
        bs[j0] = c0;
        bs[j0 + 1] = c1;
        be[j0] = be0;
        be[j0 + 1] = be1;
        bl[j0] = l0;
        bl[j0 + 1] = l1;
        const float e0 = ex2f(l0), e1 = ex2f(l1);
        eb[j0] = e0;
        eb[j0 + 1] = e1;
        bg[j0] = be0 * e0;
        bg[j0 + 1] = be1 * e1;
        ek[j0] = ex2f(l63 - l0);
        ek[j0 + 1] = ex2f(l63 - l1);
    }
    if (warp == 0) tc::tmem_alloc(tslot, 256);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *tslot;
    if (warp == 0) {   // [K ; Q] K^T: M = 128 (k rows, then q rows), N = 64, K = 128 key dims
        const bool w = tc::mbar_wait(&bars[LOAD], 0);
        ok = __all_sync(0xffffffffu, w);
        tc::tc_fence_after();
        if (tc::elect_one()) {
            const uint32_t id1 = tc::idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = base + KQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                tc::mma_ss(tm + kD1, tc::smem_desc(off, 16, 1024), tc::smem_desc(off, 16, 1024),
                           id1, kk > 0);
            }
            tc::mma_commit(&bars[M1]);
        }
        __syncwarp();
    }

    // one 64-value row per thread of warps 0..3, reused through the steps below:
    // the A row or P row, then the column of T (threads 0..63), then a row of [P Tw | P Tu]^T
    float w[64];
    if (warp < 4) {
        ok &= tc::mbar_wait(&bars[M1], 0);
        tc::tc_fence_after();
        tmem_ld64f(tc::tmem_addr(tm, warp, kD1), w);
        const int r = tid & (kC - 1);
        const float lr = bl[r];
        if (tid < kC) {
            // A_rm = beta_r e^(b_r - b_m) k_r.k_m for m < r
            const float sr = be[r];
            float *ar = As + r * kAStride;
#pragma unroll
            for (int m4 = 0; m4 < 16; ++m4) {
                float av[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * m4 + e;
                    av[e] = m < r ? sr * ex2f(lr - bl[m]) * w[m] : 0.f;
                }
                *reinterpret_cast<float4 *>(ar + 4 * m4) = make_float4(av[0], av[1], av[2], av[3]);
            }
        } else {
            // P_rm = scale e^(b_r - b_m) q_r.k_m for m <= r (kept in registers)
#pragma unroll
            for (int m = 0; m < kC; ++m) w[m] = m <= r ? a.scale * ex2f(lr - bl[m]) * w[m] : 0.f;
        }
        tc::tc_fence_before();
        tc::named_bar_sync(1, 128);

        // T = (I + A)^-1 (unit lower triangular) in shared memory, blocked: the four 16 x 16
        // diagonal blocks by forward substitution, then pairs merged into 32 x 32 and 64 x 64
        // inverses through  [L0 0 ; A10 L1]^-1 = [L0^-1 0 ; -L1^-1 A10 L0^-1  L1^-1].
        float *Ts = reinterpret_cast<float *>(sm + TT);
        float *Ys = Ts + kC * kAStride;
        if (tid < kC) {
            const int b0 = (tid >> 4) * 16, m = tid & 15;
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float *ar = As + (b0 + j) * kAStride + b0;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int l = 0; l + 3 < j; l += 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(ar + l);
                    s0 = fmaf(av.x, x[l], s0);
                    s1 = fmaf(av.y, x[l + 1], s1);
                    s0 = fmaf(av.z, x[l + 2], s0);
                    s1 = fmaf(av.w, x[l + 3], s1);
                }
#pragma unroll
                for (int l = j & ~3; l < j; ++l) s0 = fmaf(ar[l], x[l], s0);
                x[j] = (j == m ? 1.f : 0.f) - (s0 + s1);
                Ts[(b0 + j) * kAStride + b0 + m] = x[j];
                // the zero block right of an even diagonal block, read by the 64 x 64 merge
                if (!(b0 & 16)) Ts[(b0 + j) * kAStride + b0 + 16 + m] = 0.f;
            }
        }
        tc::named_bar_sync(1, 128);
        {   // 16 -> 32: rows 16 .. 31 of each 32-block, columns 0 .. 15 (4 rows per thread)
            const int pr = (tid >> 6) * 32, i0 = ((tid >> 4) & 3) * 4, m = tid & 15;
            float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int l = 0; l < 16; ++l) {
                const float tv = Ts[(pr + l) * kAStride + pr + m];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = fmaf(As[(pr + 16 + i0 + e) * kAStride + pr + l], tv, y[e]);
            }
            float *yp = Ys + (tid >> 6) * 16 * 20;
#pragma unroll
            for (int e = 0; e < 4; ++e) yp[(i0 + e) * 20 + m] = y[e];
            tc::named_bar_sync(1, 128);
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = 0.f;
#pragma unroll
            for (int l = 0; l < 16; ++l) {
                const float yv = yp[l * 20 + m];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    y[e] = fmaf(Ts[(pr + 16 + i0 + e) * kAStride + pr + 16 + l], yv, y[e]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) Ts[(pr + 16 + i0 + e) * kAStride + pr + m] = -y[e];
        }
        tc::named_bar_sync(1, 128);
        {   // 32 -> 64: rows 32 .. 63, columns 0 .. 31 (8 rows per thread)
            const int i0 = (tid >> 5) * 8, m = tid & 31;
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 4
            for (int l = 0; l < 32; l += 4) {
                const float t0v = Ts[l * kAStride + m], t1v = Ts[(l + 1) * kAStride + m];
                const float t2v = Ts[(l + 2) * kAStride + m], t3v = Ts[(l + 3) * kAStride + m];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 av = *reinterpret_cast<const float4 *>(As + (32 + i0 + e) * kAStride + l);
                    y[e] = fmaf(av.x, t0v, fmaf(av.y, t1v, fmaf(av.z, t2v, fmaf(av.w, t3v, y[e]))));
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Ys[(i0 + e) * 36 + m] = y[e];
            tc::named_bar_sync(1, 128);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 4
            for (int l = 0; l < 32; l += 4) {
                const float y0 = Ys[l * 36 + m], y1 = Ys[(l + 1) * 36 + m];
                const float y2 = Ys[(l + 2) * 36 + m], y3 = Ys[(l + 3) * 36 + m];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 tv = *reinterpret_cast<const float4 *>(Ts + (32 + i0 + e) * kAStride + 32 + l);
                    y[e] = fmaf(tv.x, y0, fmaf(tv.y, y1, fmaf(tv.z, y2, fmaf(tv.w, y3, y[e]))));
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Ts[(32 + i0 + e) * kAStride + m] = -y[e];
        }
        tc::named_bar_sync(1, 128);
        if (tid < kC) {   // column m of T
#pragma unroll
            for (int j = 0; j < kC; ++j) w[j] = j >= tid ? Ts[j * kAStride + tid] : 0.f;
        }
    } else if (warp == 4) {
        // the decay factors e^(b_63 - b_j) of the chunk's tokens, for the scan's state update
        so.EK[blk * kC + lane] = ek[lane];
        so.EK[blk * kC + 32 + lane] = ek[32 + lane];
    }
    __syncthreads();   // A and T are dead from here
    if (tid < kC) {
        // row m of Tw^T and Tu^T: T_jm beta_m e^(b_m) and T_jm beta_m over j
        store_split_row(sm + TT, sm + TT + 16384, tid, w, bg[tid]);
        store_split_row(sm + TT + 8192, sm + TT + 24576, tid, w, be[tid]);
    } else if (tid < 2 * kC) {
        store_split_row(sm + AP, sm + AP + 8192, tid - kC, w, 1.f);   // row i of P
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
        // [Tw | Tu]^T P^T: M = 128 (Tw^T rows, then Tu^T rows), N = 64, K = 64 tokens j;
        // hi*hi, lo*hi, hi*lo
        __syncwarp();
        tc::tc_fence_after();
        if (tc::elect_one()) {
            const uint32_t id2 = tc::idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int t = 0; t < 3; ++t) {
                const uint32_t ao = base + TT + (t == 1 ? 16384 : 0);
                const uint32_t bo = base + AP + (t == 2 ? 8192 : 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ss(tm + kD2, tc::smem_desc(ao + kk * 32, 16, 1024),
                               tc::smem_desc(bo + kk * 32, 16, 1024), id2, (t | kk) > 0);
            }
            tc::mma_commit(&bars[M2]);
        }
        __syncwarp();
    }
    if (warp < 4) {
        // lane m < 64: (P Tw)_{i m} over i; lane 64 + m: (P Tu)_{i m} over i
        ok &= tc::mbar_wait(&bars[M2], 0);
        tc::tc_fence_after();
        tmem_ld64f(tc::tmem_addr(tm, warp, kD2), w);
        if (tid < kC) store_split_row(sm + AP, sm + AP + 8192, tid, w, -1.f);   // (-P Tw)^T
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // [Tw ; -P Tw] K: A MN-major (M atoms Tw^T and (-P Tw)^T), B = k MN-major (N = key
        // dims), K = 64 tokens m; A hi then A lo
        __syncwarp();
        tc::tc_fence_after();
        if (tc::elect_one()) {
            const uint32_t id3 = tc::idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
                const uint32_t ao = TT + hl * 16384, lbo = AP + hl * 8192 - ao;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ss(tm + kD3, tc::smem_desc(base + ao + kk * 2048, lbo, 1024),
                               tc::smem_desc(base + KQ + kk * 2048, 16384, 1024), id3, (hl | kk) > 0);
            }
            tc::mma_commit(&bars[M3]);
        }
        __syncwarp();
    }
    if (tid >= kC && tid < 2 * kC) {
        // (P Tu)^T replaces (-P Tw)^T once the MMAs reading it have completed
        ok &= tc::mbar_wait(&bars[M3], 0);
        store_split_row(sm + AP, sm + AP + 8192, tid - kC, w, 1.f);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // [Tu ; P Tu] V, into the columns of the two products read above
        __syncwarp();
        tc::tc_fence_after();
        if (tc::elect_one()) {
            const uint32_t id4 = tc::idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
                const uint32_t ao = TT + 8192 + hl * 16384, lbo = AP + hl * 8192 - ao;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ss(tm + kD4, tc::smem_desc(base + ao + kk * 2048, lbo, 1024),
                               tc::smem_desc(base + V + kk * 2048, 8192, 1024), id4, (hl | kk) > 0);
            }
            tc::mma_commit(&bars[M4]);
        }
        __syncwarp();
    }
    ok &= tc::mbar_wait(&bars[M4], 0);
    tc::tc_fence_after();

    // ---- epilogue: staged through shared memory (v, Tw/Tu and P areas are dead), TMA stores
    const int q4 = warp & 3, hc = warp >> 2, r = 32 * q4 + lane, rr = r & (kC - 1);
    const int yrow = (int)(blk * kC);
    {
        // W (lanes 0..63) and G = scale e^(b_i) q_i - P W (lanes 64..127), columns 64 hc ..
        float v[64];
        tmem_ld64f(tc::tmem_addr(tm, q4, kD3 + 64 * hc), v);
        if (r >= kC) {
            const float f = a.scale * eb[rr];
            const uint8_t *qt = sm + KQ + 8192 + hc * 16384;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint4 qq = *reinterpret_cast<const uint4 *>(qt + tc::sw128_offset(rr, 8 * ch));
                const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 qf = tc::unpack_bf16(qw[p]);
                    v[8 * ch + 2 * p] = fmaf(f, qf.x, v[8 * ch + 2 * p]);
                    v[8 * ch + 2 * p + 1] = fmaf(f, qf.y, v[8 * ch + 2 * p + 1]);
                }
            }
        }
        stage_row64(sm + (r < kC ? ST0 : ST1), rr, 64 * hc, v);
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) {
            tma_store_2d(&tw, sm + ST0 + bx * 8192, 32 * bx, yrow);
            tma_store_2d(&tg, sm + ST1 + bx * 8192, 32 * bx, yrow);
        }
        tc::bulk_commit();
        tc::bulk_wait_read_all();
    }
    __syncthreads();
    {
        // Ut (lanes 0..63) and Oi = P Ut (lanes 64..127)
        float v[64];
        tmem_ld64f(tc::tmem_addr(tm, q4, kD4 + 64 * hc), v);
        stage_row64(sm + (r < kC ? ST0 : ST1), rr, 64 * hc, v);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) {
            tma_store_2d(&tu, sm + ST0 + bx * 8192, 32 * bx, yrow);
            tma_store_2d(&to, sm + ST1 + bx * 8192, 32 * bx, yrow);
        }
        tc::bulk_commit();
        so.C[blk] = bs[kC - 1];
        tc::bulk_wait_all();
    }
    if (warp == 0) {   // TMEM is no longer read
        __syncwarp();
        tc::tc_fence_after();
        tc::tmem_dealloc(tm, 256);
    }
    if (!ok) atomicOr(err, kDevErrTimeout);
}

// Start states of the segments of a split scan: S_start(1) is segment 0's end state, and
// S_start(s + 1) = M_s S_start(s) + E_s for s = 1 .. segs - 2, in fp32. One CTA per (batch and
// head, block of 16 value columns); thread (v, r) owns value column v of key rows r + 16 i,
// i < 8, so each S element read from shared memory feeds eight products. Each M_s is first copied
// into shared memory with coalesced loads (rows padded against bank conflicts).
constexpr int kSegCols = 16;
constexpr int kSegMStride = kMaxD + 4;
constexpr size_t kSegSmem = (size_t)(kMaxD * kSegMStride + kMaxD * kSegCols) * sizeof(float);
__global__ void __launch_bounds__(256) gdn_seg_scan_kernel(ScanPlan sp) {
    extern __shared__ __align__(16) float segsm[];
    float *Ms = segsm;                       // [128][kSegMStride]
    float *S = segsm + kMaxD * kSegMStride;  // [128][kSegCols]
    const int64_t bh = blockIdx.x;
    const int c0 = blockIdx.y * kSegCols;
    // key rows rb + 16 i: the two row groups of a warp sit in different banks
    const int v = threadIdx.x & (kSegCols - 1), rb = threadIdx.x >> 4;
    const size_t step = (size_t)kMaxD * kMaxD;
    const size_t base = (size_t)bh * (sp.segs - 1) * step;
    // S_start(1): the end state of segment 0, written by its output CTA
#pragma unroll
    for (int i = 0; i < 8; ++i)
        S[(rb + 16 * i) * kSegCols + v] = sp.Ss[base + (size_t)(rb + 16 * i) * kMaxD + c0 + v];
    // M_s and E_s of the next step are loaded while the current step computes
    float4 mr[16];
    float er[8];
    auto load_step = [&](int sg) {
        const float4 *src = reinterpret_cast<const float4 *>(sp.M + base + sg * step);
#pragma unroll
        for (int x = 0; x < 16; ++x) mr[x] = src[threadIdx.x + 256 * x];
#pragma unroll
        for (int i = 0; i < 8; ++i) er[i] = sp.E[base + sg * step + (size_t)(rb + 16 * i) * kMaxD + c0 + v];
    };
    if (sp.segs > 2) load_step(1);
    for (int sg = 1; sg < sp.segs - 1; ++sg) {
#pragma unroll
        for (int x = 0; x < 16; ++x) {   // M_s into shared memory (4096 float4, coalesced)
            const int f = threadIdx.x + 256 * x, row = f >> 5, col = (f & 31) * 4;
            *reinterpret_cast<float4 *>(Ms + row * kSegMStride + col) = mr[x];
        }
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = er[i];
        __syncthreads();   // M_s (and the previous step's S) in shared memory
        if (sg + 1 < sp.segs - 1) load_step(sg + 1);
#pragma unroll 2
        for (int e = 0; e < kMaxD; e += 4) {
            const float s0 = S[e * kSegCols + v], s1v = S[(e + 1) * kSegCols + v];
            const float s2 = S[(e + 2) * kSegCols + v], s3 = S[(e + 3) * kSegCols + v];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 m = *reinterpret_cast<const float4 *>(Ms + (rb + 16 * i) * kSegMStride + e);
                acc[i] = fmaf(m.x, s0, fmaf(m.y, s1v, fmaf(m.z, s2, fmaf(m.w, s3, acc[i]))));
            }
        }
        __syncthreads();   // every thread has read S and M_s
        float *out = sp.Ss + base + sg * step;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            S[(rb + 16 * i) * kSegCols + v] = acc[i];
            out[(size_t)(rb + 16 * i) * kMaxD + c0 + v] = acc[i];
        }
    }
}

// Segments of the tensor-core scan: the most whose first launch (segment 0's outputs and two
// transition CTAs per middle segment) still fits one wave of one-CTA-per-SM launches, with
// segment 0 at least 4 chunks. Fewer than three segments gain nothing (segment 1 would wait
// for all of segment 0), so the split is then off.
int gdn_tc_segments(int64_t BH, int nchunks, int num_sms) {
    int64_t s = (num_sms / BH - 1) / 2 + 2;
    s = std::min<int64_t>(s, (nchunks / 4 + 1) / 2);
    s = std::min<int64_t>(s, 16);
    return s >= 3 ? (int)s : 1;
}

// Floats of the split scan's arrays (E, M, start states) behind the per-chunk workspace.
int64_t gdn_seg_floats(int64_t BH, int segs) {
    return segs > 1 ? 3 * BH * (segs - 1) * (int64_t)kMaxD * kMaxD : 0;
}

constexpr size_t kPrepSmem = (size_t)(2 * kMaxD * kPrepStride + 2 * kC * kC + 5 * kC) * sizeof(float);

// Shared-memory opt-in of the tensor-core scan, once per device.
std::mutex g_gdn_attr_mu;
bool g_gdn_attr_done[64];

cudaError_t launch_tc_scan(const GdnArgs &a, int64_t BH, int num_sms, unsigned *err,
                           cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_gdn_attr_mu);
        if (!g_gdn_attr_done[dev]) {
            e = cudaFuncSetAttribute(gdn_tc_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)gt::ALLOC);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(gdn_seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSegSmem);
            if (e != cudaSuccess) return e;
            g_gdn_attr_done[dev] = true;
        }
    }
    const SoA so(a.ws, a.nblk, kMaxD, kMaxD);
    CUtensorMap mw, mg, mk, me;
    if (!make_2d_map(&mw, so.W, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.nblk * kC, kMaxD, 32, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_2d_map(&mg, so.G, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.nblk * kC, kMaxD, 32, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH / a.H, a.T, a.H, kMaxD,
                       64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_2d_map(&me, so.EK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.nblk, kC, kC, 1,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidResourceHandle;   // a tensor map could not be encoded
    const int segs = gdn_tc_segments(BH, a.nchunks, num_sms);
    ScanPlan sp{segs, 0, 0, nullptr, nullptr, nullptr};
    if (segs > 1) {
        // the split's arrays follow the per-chunk workspace
        float *seg = a.ws + a.nblk * WsLayout(kMaxD, kMaxD).total;
        const int64_t per = BH * (segs - 1) * (int64_t)kMaxD * kMaxD;
        sp.E = seg;
        sp.M = seg + per;
        sp.Ss = seg + 2 * per;
        sp.mode = 1;
        gdn_tc_scan_kernel<<<(unsigned)(BH + BH * (segs - 2) * 2), gt::kThreadsTC, gt::ALLOC, s>>>(
            mw, mg, mk, me, a, sp, err);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        gdn_seg_scan_kernel<<<dim3((unsigned)BH, kMaxD / kSegCols), 256, kSegSmem, s>>>(sp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        count_launches(2);
        sp.mode = 0;
        sp.s0 = 1;
    }
    gdn_tc_scan_kernel<<<(unsigned)(BH * (segs - sp.s0)), gt::kThreadsTC, gt::ALLOC, s>>>(
        mw, mg, mk, me, a, sp, err);
    return cudaGetLastError();
}


std::mutex g_gdn_prep_attr_mu;
bool g_gdn_prep_attr_done[64];

cudaError_t launch_tc_prep(const GdnArgs &a, int64_t B, unsigned *err, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_gdn_prep_attr_mu);
        if (!g_gdn_prep_attr_done[dev]) {
            e = cudaFuncSetAttribute(gdn_tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)gp::ALLOC);
            if (e != cudaSuccess) return e;
            g_gdn_prep_attr_done[dev] = true;
        }
    }
    const SoA so(a.ws, a.nblk, kMaxD, kMaxD);
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap mq, mk, mv, mw, mg, mu, mo;
    if (!make_bthd_map(&mq, a.q, bf, 2, B, a.T, a.H, kMaxD, 64, kC, sw) ||
        !make_bthd_map(&mk, a.k, bf, 2, B, a.T, a.H, kMaxD, 64, kC, sw) ||
        !make_bthd_map(&mv, a.v, bf, 2, B, a.T, a.H, kMaxD, 64, kC, sw) ||
        !make_2d_map(&mw, so.W, f32, 4, a.nblk * kC, kMaxD, 32, kC, sw) ||
        !make_2d_map(&mg, so.G, f32, 4, a.nblk * kC, kMaxD, 32, kC, sw) ||
        !make_2d_map(&mu, so.U, f32, 4, a.nblk * kC, kMaxD, 32, kC, sw) ||
        !make_2d_map(&mo, so.O, f32, 4, a.nblk * kC, kMaxD, 32, kC, sw))
        return cudaErrorInvalidResourceHandle;   // a tensor map could not be encoded
    gdn_tc_prep_kernel<<<(unsigned)a.nblk, gp::kThreadsP, gp::ALLOC, s>>>(mq, mk, mv, mw, mg, mu,
                                                                         mo, a, err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const GdnArgs &a, int64_t BH, int num_sms, unsigned *err,
                         cudaStream_t s) {
    const int64_t nprep = BH * a.nchunks;
    // bf16 I/O at head dims 128: the tensor-core scan (tf32), with the structure-of-arrays
    // workspace; otherwise the fp32 CUDA-core scan
    const bool tc = std::is_same<T, __nv_bfloat16>::value && a.Dk == kMaxD && a.Dv == kMaxD;
    if (tc) {
        cudaError_t e = launch_tc_prep(a, BH / a.H, err, s);
        if (e != cudaSuccess) return e;
        e = launch_tc_scan(a, BH, num_sms, err, s);
        if (e == cudaSuccess) count_launches(2);
        return e;
    }
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

size_t gdn_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int num_sms) {
    const int64_t nchunks = (T + kC - 1) / kC;
    // head dims 128 may take the tensor-core scan, whose split adds its segment arrays
    const int64_t seg = (Dk == kMaxD && Dv == kMaxD)
                            ? gdn_seg_floats(B * H, gdn_tc_segments(B * H, (int)nchunks, num_sms))
                            : 0;
    return ((size_t)(B * H * nchunks) * (size_t)WsLayout((int)Dk, (int)Dv).total + (size_t)seg) *
           sizeof(float);
}

cudaError_t launch_gdn(const GdnProblem &p, void *ws, int num_sms, unsigned *err,
                       cudaStream_t s) {
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
    a.nblk = BH * a.nchunks;
    return p.io == 0 /* bf16 */ ? launch_typed<__nv_bfloat16>(a, BH, num_sms, err, s)
                     : launch_typed<float>(a, BH, num_sms, err, s);
}

}  // namespace gla
