// Tensor-core chunkwise GLA forward for sm_103a: TMA-staged tiles, tcgen05 MMAs with
// TMEM accumulators, fp32 state kept in TMEM across the chunk scan, warp-specialised
// roles. The chunk algebra is that of "线性注意力GPU算子库的定义与技术解析", section 四
// (blocks recurred locally, states carried block to block, in-block work as matrix
// products); the update it evaluates is the gated state update of "Linear Attention 在
// GPU 上到底慢在哪", section 学长的反馈.
//
// Per (batch, head) and chunk of C = 64 tokens with in-chunk inclusive cumulative
// log-gate b (a Dk vector per token) and chunk total Bc = b_63:
//     Q~ = q * exp(b)          K~ = k * exp(-b)         K^ = k * exp(Bc - b)
//     P  = (Q~ K~^T) masked to j <= i                                (M=64 MMA)
//     O^T = V^T P^T + S^T Q~^T       (S^T bf16 from TMEM as the A operand)   (M=128)
//     S^T <- diag-scaled S^T * exp(Bc) + V^T K^                              (M=128)
//     o  = scale * O
// The state is stored transposed in TMEM (lane = value column v, column = key row d),
// so every large MMA has M = 128.
//
// Range: K~ = k * exp(-b) is finite only while |b| stays below ~88. A chunk whose
// |cumulative log-gate| exceeds kExtreme anywhere is flagged by the gate warps, and its
// P is computed instead on CUDA cores from the raw inputs with exact per-element decays
// exp(b_i - b_j); the state update and the inter-chunk term use only factors <= 1 and
// stay on the tensor cores.
//
// Sequence parallelism (so that B*H = 16 heads still fill 152 SMs): each head's chunks
// are split into `splits` contiguous segments.
//   gla_tc_state_kernel : segment s < splits-1 -> its end state from a zero start, E_s,
//                         and its total decay Gamma_s = exp(sum of its log-gates).
//                         Chunks run last-to-first so that the per-chunk suffix decay is
//                         known and E_s accumulates in TMEM with a single MMA chain.
//   gla_tc_scan_kernel  : S_start(s+1) = Gamma_s * S_start(s) + E_s  (S_start(0) = h0).
//   gla_tc_out_kernel   : every segment from its start state: outputs, and hT from the
//                         last segment.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "gla_internal.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace tc;

constexpr int kC = 64;                 // chunk length (tokens)
constexpr int kD = 128;                // Dk = Dv
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kExtreme = 60.f;       // |b| beyond which a chunk takes the exact P route

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Per-role timeline tracing, compiled in only with -DGLA_TRACE: clock64() stamps of the
// first kTraceCtas CTAs into a device buffer [cta][event][chunk] set by the tracer.
#ifdef GLA_TRACE
constexpr int kTraceCtas = 4, kTraceEvents = 24, kTraceChunks = 256;
__device__ long long *g_trace_out;
__device__ long long *g_trace_state;
#define GLA_TRACE_AT(buf, ev, lc)                                                              \
    do {                                                                                       \
        if ((buf) && blockIdx.x < kTraceCtas && (lc) < kTraceChunks)                           \
            (buf)[((size_t)blockIdx.x * kTraceEvents + (ev)) * kTraceChunks + (lc)] = clock64(); \
    } while (0)
#else
#define GLA_TRACE_AT(buf, ev, lc) \
    do {                          \
    } while (0)
#endif
#define TRACE_OUT(ev, lc) GLA_TRACE_AT(g_trace_out, ev, lc)
#define TRACE_ST(ev, lc) GLA_TRACE_AT(g_trace_state, ev, lc)

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// TMEM column map of the output kernel (512 columns).
constexpr uint32_t kColS = 0;      // S^T fp32, 128 columns
constexpr uint32_t kColSB = 128;   // S^T bf16 (A operand), 2 x 64 columns
constexpr uint32_t kColP = 256;    // P fp32 (M=64 layout), 2 x 64 columns
constexpr uint32_t kColO = 384;    // O^T fp32, 2 x 64 columns

// Shared-memory map of the output kernel (bytes from a 1024-aligned base). A stage holds
// the raw q, k, v tiles (128B-swizzled [64 x 64] bf16 boxes, two per tile) and the fp32
// log-gate rows; the gate warps rewrite q -> Q~ and k -> K~ in place and write K^ over
// the first half of the gate rows once every gate row has been read.
namespace om {
constexpr uint32_t Q = 0, K = 16384, V = 32768, G = 49152, KH = G, STAGE = 81920;
constexpr uint32_t P = 2 * STAGE;      // 2 x [64 x 64] bf16 P tiles (128B swizzle)
constexpr uint32_t OST = P + 16384;    // [64 x 128] bf16 output staging (two boxes)
constexpr uint32_t GAM = OST + 16384;  // [2][128] f32 exp(Bc)
constexpr uint32_t BV = GAM + 1024;    // [2][128] f32 Bc (log2 units)
constexpr uint32_t XCH = BV + 1024;    // [4][128] f32 token-quarter totals
constexpr uint32_t XF = XCH + 2048;    // [2] u32 "extreme chunk" flags
constexpr uint32_t SCR = XF + 64;      // [4][64] f32 exact-path scratch
constexpr uint32_t BAR = SCR + 1024;   // mbarriers
constexpr uint32_t NBAR = 20;
constexpr uint32_t TSLOT = BAR + NBAR * 8;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
}  // namespace om

// mbarrier indices of the output kernel
enum {
    FULL = 0, EMPTY = 2, GDONE = 4, PFULL = 6, PFREE = 8, PBF = 10, SREADY = 12, UDONE = 13,
    OFULL = 14, OFREE = 16, FIN = 18,
};

constexpr int kOutThreads = 576;       // 18 warps
constexpr int kStateThreads = 320;     // 10 warps

struct OutArgs {
    const __nv_bfloat16 *q, *k;        // raw inputs (exact route of extreme chunks)
    const float *g;
    const float *h0;                   // [B,H,Dk,Dv] or null
    float *hT;                         // [B,H,Dk,Dv] or null
    const float *sstart;               // [BH][splits-1][Dk][Dv] start states of segments 1..
    int64_t T;
    int H, nchunks, splits;
    float scale;
    unsigned *err;
};

struct StateArgs {
    float *E;                          // [BH][splits-1][Dk][Dv]
    float *gam;                        // [BH][splits-1][Dk]
    int64_t T;
    int H, nchunks, splits;
    unsigned *err;
};

__device__ __forceinline__ void seg_range(int seg, int nchunks, int splits, int &cb, int &ce) {
    cb = (int)((int64_t)seg * nchunks / splits);
    ce = (int)((int64_t)(seg + 1) * nchunks / splits);
}

// Load 64 consecutive TMEM columns of this warp's lane quarter (one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&out)[64]) {
    uint32_t r0[16], r1[16], r2[16], r3[16];
    tmem_ld16(taddr, r0);
    tmem_ld16(taddr + 16, r1);
    tmem_ld16(taddr + 32, r2);
    tmem_ld16(taddr + 48, r3);
    tmem_wait_ld();
    reg_fence(r0);
    reg_fence(r1);
    reg_fence(r2);
    reg_fence(r3);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        out[x] = __uint_as_float(r0[x]);
        out[16 + x] = __uint_as_float(r1[x]);
        out[32 + x] = __uint_as_float(r2[x]);
        out[48 + x] = __uint_as_float(r3[x]);
    }
}

// In-chunk cumulative log-gate of one thread's column pair over 16 tokens, in log2 units,
// shared with the other token quarters through `xch` (named barrier `bar`, 256 threads).
// On return b0/b1 hold the chunk-inclusive cumulative log2-gates of the thread's tokens.
__device__ __forceinline__ void gate_cumsum(const float *gs, float *xch, int qq, int d,
                                            float (&b0)[16], float (&b1)[16], uint32_t bar) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        const float2 gv = *reinterpret_cast<const float2 *>(gs + (16 * qq + x) * kD + d);
        a0 = fmaf(gv.x, kLog2e, a0);
        a1 = fmaf(gv.y, kLog2e, a1);
        b0[x] = a0;
        b1[x] = a1;
    }
    *reinterpret_cast<float2 *>(xch + qq * kD + d) = make_float2(a0, a1);
    named_bar_sync(bar, 256);
    float o0 = 0.f, o1 = 0.f;
    for (int q2 = 0; q2 < qq; ++q2) {
        const float2 t = *reinterpret_cast<const float2 *>(xch + q2 * kD + d);
        o0 += t.x;
        o1 += t.y;
    }
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        b0[x] += o0;
        b1[x] += o1;
    }
}

// ======================================================================= output kernel
__global__ void __launch_bounds__(kOutThreads, 1)
gla_tc_out_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                  const __grid_constant__ CUtensorMap to, const OutArgs a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + om::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + om::TSLOT);
    float *gam_s = reinterpret_cast<float *>(sm + om::GAM);
    float *bv_s = reinterpret_cast<float *>(sm + om::BV);
    float *xch = reinterpret_cast<float *>(sm + om::XCH);
    uint32_t *xf = reinterpret_cast<uint32_t *>(sm + om::XF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x % a.splits;
    const int bh = blockIdx.x / a.splits;
    const int bidx = bh / a.H, h = bh % a.H;
    int cb, ce;
    seg_range(seg, a.nchunks, a.splits, cb, ce);
    const int n = ce - cb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[FULL + i], 1);
            mbar_init(&bars[EMPTY + i], 1);
            mbar_init(&bars[GDONE + i], 8);
            mbar_init(&bars[PFULL + i], 1);
            mbar_init(&bars[PFREE + i], 4);
            mbar_init(&bars[PBF + i], 4);
            mbar_init(&bars[OFULL + i], 1);
            mbar_init(&bars[OFREE + i], 4);
        }
        mbar_init(&bars[SREADY], 4);
        mbar_init(&bars[UDONE], 1);
        mbar_init(&bars[FIN], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tg);
        tma_prefetch_desc(&to);
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;
    if (threadIdx.x == 0) TRACE_OUT(14, 0);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued[2] = {0, 0};
            for (int lc = 0; lc < n; ++lc) {
                const int st = lc & 1;
                const uint32_t u = lc >> 1;
                if (lc >= 2 && !mbar_wait(&bars[EMPTY + st], (u - 1) & 1)) { ok = false; break; }
                uint8_t *base = sm + st * om::STAGE;
                uint64_t *fb = &bars[FULL + st];
                TRACE_OUT(0, lc);
                mbar_arrive_expect_tx(fb, 3 * 16384 + 32768);
                const int t = (cb + lc) * kC;
                tma_load_4d(base + om::G, &tg, fb, 0, h, t, bidx);
                tma_load_4d(base + om::Q, &tq, fb, 0, h, t, bidx);
                tma_load_4d(base + om::Q + 8192, &tq, fb, 64, h, t, bidx);
                tma_load_4d(base + om::K, &tk, fb, 0, h, t, bidx);
                tma_load_4d(base + om::K + 8192, &tk, fb, 64, h, t, bidx);
                tma_load_4d(base + om::V, &tv, fb, 0, h, t, bidx);
                tma_load_4d(base + om::V + 8192, &tv, fb, 64, h, t, bidx);
                ++issued[st];
            }
            // never leave with a bulk copy still landing in this CTA's shared memory
            for (int st = 0; st < 2; ++st)
                if (issued[st] > 0 && !mbar_wait(&bars[FULL + st], (issued[st] - 1) & 1)) ok = false;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // order per chunk c: U(c) [needs S_c ready], P(c+1) [needs gates of c+1], O(c)
        if (lane == 0) {
            const uint32_t idP = idesc_bf16(64, 64, 0, 0);
            const uint32_t idU = idesc_bf16(128, 128, 1, 1);
            const uint32_t idOi = idesc_bf16(128, 64, 1, 0);
            const uint32_t idOs = idesc_bf16(128, 64, 0, 0);
            auto issue_p = [&](int lc) -> bool {
                const int st = lc & 1;
                const uint32_t u = lc >> 1;
                if (!mbar_wait(&bars[GDONE + st], u & 1)) return false;
                if (lc >= 2 && !mbar_wait(&bars[PFREE + st], (u - 1) & 1)) return false;
                TRACE_OUT(3, lc);
                tc_fence_after();
                const uint32_t base = smem_u32(sm + st * om::STAGE);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_ss(tm + kColP + st * 64, smem_desc(base + om::Q + off, 16, 1024),
                           smem_desc(base + om::K + off, 16, 1024), idP, kk > 0);
                }
                mma_commit(&bars[PFULL + st]);
                TRACE_OUT(4, lc);
                return true;
            };
            if (n > 0 && !issue_p(0)) ok = false;
            for (int lc = 0; lc < n && ok; ++lc) {
                const int st = lc & 1;
                const uint32_t u = lc >> 1;
                const uint32_t base = smem_u32(sm + st * om::STAGE);
                // S^T += V^T K^   (128 x 128, K = 64 tokens)
                if (!mbar_wait(&bars[SREADY], lc & 1)) { ok = false; break; }
                TRACE_OUT(5, lc);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tm + kColS, smem_desc(base + om::V + kk * 2048, 8192, 1024),
                           smem_desc(base + om::KH + kk * 2048, 8192, 1024), idU, 1);
                mma_commit(&bars[UDONE]);
                if (lc + 1 < n && !issue_p(lc + 1)) { ok = false; break; }
                // O^T = V^T P^T + S^T Q~^T   (128 x 64)
                if (!mbar_wait(&bars[PBF + st], u & 1)) { ok = false; break; }
                if (lc >= 2 && !mbar_wait(&bars[OFREE + st], (u - 1) & 1)) { ok = false; break; }
                TRACE_OUT(6, lc);
                tc_fence_after();
                const uint32_t pbase = smem_u32(sm + om::P + st * 8192);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tm + kColO + st * 64, smem_desc(base + om::V + kk * 2048, 8192, 1024),
                           smem_desc(pbase + kk * 32, 16, 1024), idOi, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tm + kColO + st * 64, tm + kColSB + st * 64 + kk * 8,
                           smem_desc(base + om::Q + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                           idOs, 1);
                mma_commit(&bars[OFULL + st]);
                mma_commit(&bars[EMPTY + st]);
                TRACE_OUT(7, lc);
            }
            // all issued MMAs complete before the CTA tears down its TMEM
            mma_commit(&bars[FIN]);
            if (!mbar_wait(&bars[FIN], 0)) ok = false;
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P conversion + epilogue
        const int j = warp & 3;
        const int et = (warp - 4) * 32 + lane;      // 0..127
        const int v = j * 32 + lane;                // O^T lane = value column
        float *scr = reinterpret_cast<float *>(sm + om::SCR);
        uint8_t *ost = sm + om::OST + (v >> 6) * 8192;
        const uint32_t vcol = (uint32_t)(v & 63);
        for (int lc = 0; lc <= n && ok; ++lc) {
            if (lc < n) {
                const int st = lc & 1;
                const uint32_t u = lc >> 1;
                bool w = mbar_wait(&bars[GDONE + st], u & 1) && mbar_wait(&bars[PFULL + st], u & 1);
                if (named_bar_or(2, 128, !w)) { ok = false; break; }
                if (et == 0) TRACE_OUT(10, lc);
                tc_fence_after();
                const bool extreme = xf[st] != 0;
                float prow[64];
                const int i = 16 * j + lane;        // P row held by this lane (lane < 16)
                if (!extreme) {
                    tmem_ld64(tmem_addr(tm, j, kColP + st * 64), prow);
                } else {
                    // exact route: P_ij = sum_d q_id k_jd exp(b_id - b_jd), j <= i
#pragma unroll
                    for (int x = 0; x < 64; ++x) prow[x] = 0.f;
                    float *gcol = scr, *qcol = scr + 64, *kcol = scr + 128, *bcol = scr + 192;
                    const int64_t t0 = (int64_t)(cb + lc) * kC;
                    for (int d = 0; d < kD; ++d) {
                        if (et < 64) {
                            const int64_t t = t0 + et;
                            const bool in = t < a.T;
                            const int64_t idx = (((int64_t)bidx * a.T + t) * a.H + h) * kD + d;
                            gcol[et] = in ? a.g[idx] : 0.f;
                            qcol[et] = in ? __bfloat162float(a.q[idx]) : 0.f;
                            kcol[et] = in ? __bfloat162float(a.k[idx]) : 0.f;
                        }
                        named_bar_sync(2, 128);
                        if (et == 0) {
                            float s = 0.f;
                            for (int t = 0; t < 64; ++t) { s += gcol[t]; bcol[t] = s; }
                        }
                        named_bar_sync(2, 128);
                        if (lane < 16) {
                            const float qi = qcol[i], bi = bcol[i];
#pragma unroll
                            for (int x = 0; x < 64; ++x)
                                if (x <= i) prow[x] += qi * kcol[x] * ex2((bi - bcol[x]) * kLog2e);
                        }
                        named_bar_sync(2, 128);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[PFREE + st]);
                if (lane < 16) {
                    uint8_t *pt = sm + om::P + st * 8192;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        uint32_t wv[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int c = cc * 8 + 2 * x;
                            wv[x] = pack_bf16(c <= i ? prow[c] : 0.f, c + 1 <= i ? prow[c + 1] : 0.f);
                        }
                        *reinterpret_cast<uint4 *>(pt + sw128_offset(i, cc * 8)) =
                            make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[PBF + st]);
                if (et == 0) TRACE_OUT(11, lc);
            }
            if (lc >= 1) {
                const int pc = lc - 1;
                const int st = pc & 1;
                const uint32_t u = pc >> 1;
                const bool w = mbar_wait(&bars[OFULL + st], u & 1);
                if (named_bar_or(2, 128, !w)) { ok = false; break; }
                if (et == 0) TRACE_OUT(12, pc);
                tc_fence_after();
                float ov[64];
                tmem_ld64(tmem_addr(tm, j, kColO + st * 64), ov);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[OFREE + st]);
                // stage O (bf16, 128B-swizzled boxes) and write it with two bulk tensor stores
                if (et == 0) bulk_wait_read_all();
                named_bar_sync(2, 128);
#pragma unroll
                for (int x = 0; x < 64; ++x)
                    *reinterpret_cast<__nv_bfloat16 *>(ost + sw128_offset(x, vcol)) =
                        __float2bfloat16_rn(a.scale * ov[x]);
                fence_proxy_async_smem();
                named_bar_sync(2, 128);
                if (et == 0) {
                    const int t0 = (cb + pc) * kC;
                    tma_store_4d(&to, sm + om::OST, 0, h, t0, bidx);
                    tma_store_4d(&to, sm + om::OST + 8192, 64, h, t0, bidx);
                    bulk_commit();
                    TRACE_OUT(13, pc);
                }
            }
        }
        if (et == 0) bulk_wait_all();
        __syncwarp();
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ state scan (TMEM)
        const int j = warp & 3;
        const int v = j * 32 + lane;
        const float *init = nullptr;
        if (seg > 0)
            init = a.sstart + ((size_t)bh * (a.splits - 1) + (seg - 1)) * (kD * kD);
        else if (a.h0)
            init = a.h0 + (size_t)bh * (kD * kD);
#pragma unroll 1
        for (int d0 = 0; d0 < kD; d0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int x = 0; x < 16; ++x)
                r[x] = init ? __float_as_uint(init[(d0 + x) * kD + v]) : 0u;
            tmem_st16(tmem_addr(tm, j, kColS + d0), r);
        }
        tmem_wait_st();
        for (int lc = 0; lc < n; ++lc) {
            const int st = lc & 1;
            const uint32_t u = lc >> 1;
            if (lc >= 1 && !mbar_wait(&bars[UDONE], (lc - 1) & 1)) { ok = false; break; }
            if (!mbar_wait(&bars[GDONE + st], u & 1)) { ok = false; break; }
            if (v == 0) TRACE_OUT(8, lc);
            tc_fence_after();
            const float *gam = gam_s + st * 128;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float sv[64];
                tmem_ld64(tmem_addr(tm, j, kColS + half * 64), sv);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        pk[x] = pack_bf16(sv[16 * c + 2 * x], sv[16 * c + 2 * x + 1]);
                    tmem_st8(tmem_addr(tm, j, kColSB + st * 64 + half * 32 + c * 8), pk);
                    uint32_t r[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x)
                        r[x] = __float_as_uint(sv[16 * c + x] * gam[half * 64 + 16 * c + x]);
                    tmem_st16(tmem_addr(tm, j, kColS + half * 64 + 16 * c), r);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[SREADY]);
            if (v == 0) TRACE_OUT(9, lc);
        }
        if (ok && a.hT && seg == a.splits - 1) {
            if (!mbar_wait(&bars[UDONE], (n - 1) & 1)) {
                ok = false;
            } else {
                tc_fence_after();
                float *hp = a.hT + (size_t)bh * (kD * kD) + v;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float sv[64];
                    tmem_ld64(tmem_addr(tm, j, kColS + half * 64), sv);
#pragma unroll
                    for (int x = 0; x < 64; ++x) hp[(half * 64 + x) * kD] = sv[x];
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ gate warps (8)
        const int gw = warp < 4 ? warp - 2 : warp - 10;   // 0..7
        const int gt = gw * 32 + lane;                      // 0..255
        const int p = gt & 63, qq = gt >> 6;                // key-dim pair, token quarter
        const int d = 2 * p;
        const uint32_t boxo = (uint32_t)(p >> 5) * 8192;
        const uint32_t col = (uint32_t)(d & 63);
        const float lim = kExtreme * kLog2e;
        for (int lc = 0; lc < n; ++lc) {
            const int st = lc & 1;
            const uint32_t u = lc >> 1;
            const bool w = mbar_wait(&bars[FULL + st], u & 1);
            if (named_bar_or(1, 256, !w)) { ok = false; break; }
            if (gt == 0) TRACE_OUT(1, lc);
            uint8_t *base = sm + st * om::STAGE;
            float b0[16], b1[16];   // cumulative log2-gates of this thread's tokens
            gate_cumsum(reinterpret_cast<const float *>(base + om::G), xch, qq, d, b0, b1, 1);
            float mx = 0.f;
#pragma unroll
            for (int x = 0; x < 16; ++x) mx = fmaxf(mx, fmaxf(fabsf(b0[x]), fabsf(b1[x])));
            if (qq == 3) {   // chunk totals -> exp(Bc) for the state warps and K^
                bv_s[st * 128 + d] = b0[15];
                bv_s[st * 128 + d + 1] = b1[15];
                gam_s[st * 128 + d] = ex2(b0[15]);
                gam_s[st * 128 + d + 1] = ex2(b1[15]);
            }
            const bool extreme = named_bar_or(1, 256, mx > lim);
            // every gate row has been read (the barriers above): K^ may overwrite them
            const float G0 = gam_s[st * 128 + d], G1 = gam_s[st * 128 + d + 1];
            const float B0 = bv_s[st * 128 + d], B1 = bv_s[st * 128 + d + 1];
            uint8_t *qt = base + om::Q + boxo;
            uint8_t *kt = base + om::K + boxo;
            uint8_t *kh = base + om::KH + boxo;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const uint32_t off = sw128_offset(16 * qq + x, col);
                const float2 qv = unpack_bf16(*reinterpret_cast<const uint32_t *>(qt + off));
                const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(kt + off));
                const float ep0 = ex2(b0[x]), ep1 = ex2(b1[x]);
                const float em0 = ex2(-b0[x]), em1 = ex2(-b1[x]);
                *reinterpret_cast<uint32_t *>(qt + off) = pack_bf16(qv.x * ep0, qv.y * ep1);
                *reinterpret_cast<uint32_t *>(kt + off) = pack_bf16(kv.x * em0, kv.y * em1);
                float kh0, kh1;
                if (!extreme) {
                    kh0 = kv.x * em0 * G0;
                    kh1 = kv.y * em1 * G1;
                } else {
                    kh0 = kv.x * ex2(B0 - b0[x]);
                    kh1 = kv.y * ex2(B1 - b1[x]);
                }
                *reinterpret_cast<uint32_t *>(kh + off) = pack_bf16(kh0, kh1);
            }
            if (gt == 0) xf[st] = extreme ? 1u : 0u;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[GDONE + st]);
            if (gt == 0) TRACE_OUT(2, lc);
        }
        __syncwarp();
    }

    if (!ok) atomicOr(a.err, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) TRACE_OUT(15, 0);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// ======================================================================= state kernel
// Three-stage ring of k, v and gate rows; the suffix-decayed keys K^' overwrite the gate
// rows of their stage once all of them have been read.
namespace sm_ {
constexpr int NST = 3;
constexpr uint32_t K = 0, V = 16384, G = 32768, KH = G, STAGE = 65536;
constexpr uint32_t BV = NST * STAGE;   // [3][128] f32 chunk totals
constexpr uint32_t XCH = BV + 1536;    // [4][128] f32
constexpr uint32_t BAR = XCH + 2048;
constexpr uint32_t TSLOT = BAR + 80;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
}  // namespace sm_

enum { SFULL = 0, SEMPTY = 3, SGDONE = 6, SEDONE = 9 };

__global__ void __launch_bounds__(kStateThreads, 1)
gla_tc_state_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tg, const StateArgs a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + sm_::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + sm_::TSLOT);
    float *bv_s = reinterpret_cast<float *>(sm + sm_::BV);
    float *xch = reinterpret_cast<float *>(sm + sm_::XCH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nseg = a.splits - 1;
    const int seg = blockIdx.x % nseg;
    const int bh = blockIdx.x / nseg;
    const int bidx = bh / a.H, h = bh % a.H;
    int cb, ce;
    seg_range(seg, a.nchunks, a.splits, cb, ce);
    const int n = ce - cb;
    constexpr int NST = sm_::NST;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bars[SFULL + i], 1);
            mbar_init(&bars[SEMPTY + i], 1);
            mbar_init(&bars[SGDONE + i], 8);
        }
        mbar_init(&bars[SEDONE], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tg);
    }
    if (warp == 1) tmem_alloc(tslot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            int issued[NST] = {0, 0, 0};
            for (int lc = 0; lc < n; ++lc) {
                const int st = lc % NST;
                const uint32_t u = lc / NST;
                if (lc >= NST && !mbar_wait(&bars[SEMPTY + st], (u - 1) & 1)) { ok = false; break; }
                uint8_t *base = sm + st * sm_::STAGE;
                uint64_t *fb = &bars[SFULL + st];
                TRACE_ST(0, lc);
                mbar_arrive_expect_tx(fb, 2 * 16384 + 32768);
                const int t = (ce - 1 - lc) * kC;      // last chunk first
                tma_load_4d(base + sm_::G, &tg, fb, 0, h, t, bidx);
                tma_load_4d(base + sm_::K, &tk, fb, 0, h, t, bidx);
                tma_load_4d(base + sm_::K + 8192, &tk, fb, 64, h, t, bidx);
                tma_load_4d(base + sm_::V, &tv, fb, 0, h, t, bidx);
                tma_load_4d(base + sm_::V + 8192, &tv, fb, 64, h, t, bidx);
                ++issued[st];
            }
            for (int st = 0; st < NST; ++st)
                if (issued[st] > 0 && !mbar_wait(&bars[SFULL + st], (issued[st] - 1) & 1)) ok = false;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idU = idesc_bf16(128, 128, 1, 1);
            for (int lc = 0; lc < n; ++lc) {
                const int st = lc % NST;
                const uint32_t u = lc / NST;
                if (!mbar_wait(&bars[SGDONE + st], u & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t base = smem_u32(sm + st * sm_::STAGE);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tm, smem_desc(base + sm_::V + kk * 2048, 8192, 1024),
                           smem_desc(base + sm_::KH + kk * 2048, 8192, 1024), idU,
                           (lc > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars[SEMPTY + st]);
                TRACE_ST(3, lc);
            }
            mma_commit(&bars[SEDONE]);
            if (!mbar_wait(&bars[SEDONE], 0)) ok = false;
        }
        __syncwarp();
    } else {
        // gate warps 2..9: suffix-decayed keys k * exp(Bc - b + l), l = sum of later Bc
        const int gt = (warp - 2) * 32 + lane;
        const int p = gt & 63, qq = gt >> 6;
        const int d = 2 * p;
        const uint32_t boxo = (uint32_t)(p >> 5) * 8192;
        const uint32_t col = (uint32_t)(d & 63);
        float l0 = 0.f, l1 = 0.f;   // log2 of the decay from this chunk's end to the segment end
        for (int lc = 0; lc < n; ++lc) {
            const int st = lc % NST;
            const uint32_t u = lc / NST;
            const bool w = mbar_wait(&bars[SFULL + st], u & 1);
            if (named_bar_or(1, 256, !w)) { ok = false; break; }
            if (gt == 0) TRACE_ST(1, lc);
            uint8_t *base = sm + st * sm_::STAGE;
            float b0[16], b1[16];
            gate_cumsum(reinterpret_cast<const float *>(base + sm_::G), xch, qq, d, b0, b1, 1);
            if (qq == 3) {
                bv_s[st * 128 + d] = b0[15];
                bv_s[st * 128 + d + 1] = b1[15];
            }
            named_bar_sync(1, 256);
            const float s0 = bv_s[st * 128 + d] + l0, s1 = bv_s[st * 128 + d + 1] + l1;
            const uint8_t *kt = base + sm_::K + boxo;
            uint8_t *kh = base + sm_::KH + boxo;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const uint32_t off = sw128_offset(16 * qq + x, col);
                const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(kt + off));
                *reinterpret_cast<uint32_t *>(kh + off) =
                    pack_bf16(kv.x * ex2(s0 - b0[x]), kv.y * ex2(s1 - b1[x]));
            }
            l0 = s0;
            l1 = s1;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[SGDONE + st]);
            if (gt == 0) TRACE_ST(2, lc);
        }
        if (ok && qq == 0) {
            float *gp = a.gam + ((size_t)bh * (a.splits - 1) + seg) * kD;
            gp[d] = ex2(l0);
            gp[d + 1] = ex2(l1);
        }
        // E^T (lane = v, column = d) -> E[d][v]
        if (ok && warp >= 4 && warp < 8) {
            const int j = warp & 3;
            const int v = j * 32 + lane;
            if (!mbar_wait(&bars[SEDONE], 0)) {
                ok = false;
            } else {
                tc_fence_after();
                float *ep = a.E + ((size_t)bh * (a.splits - 1) + seg) * (kD * kD) + v;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float ev[64];
                    tmem_ld64(tmem_addr(tm, j, half * 64), ev);
#pragma unroll
                    for (int x = 0; x < 64; ++x) ep[(half * 64 + x) * kD] = ev[x];
                }
            }
        }
        __syncwarp();
    }

    if (!ok) atomicOr(a.err, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 128);
    }
}

// ======================================================================= scan kernel
// S_start(s+1) = Gamma_s (.) S_start(s) + E_s, rows scaled by Gamma_s[d]; S_start(0) = h0.
// Block (bh, 8-row slab of d), thread = value column v.
__global__ void __launch_bounds__(128)
gla_tc_scan_kernel(const float *__restrict__ E, const float *__restrict__ gam,
                   const float *__restrict__ h0, float *__restrict__ sstart, int splits) {
    const int bh = blockIdx.x;
    const int d0 = blockIdx.y * 8;
    const int v = threadIdx.x;
    const int nseg = splits - 1;
    float s[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) s[x] = h0 ? h0[((size_t)bh * kD + d0 + x) * kD + v] : 0.f;
    for (int r = 0; r < nseg; ++r) {
        const size_t base = ((size_t)bh * nseg + r) * (kD * kD) + (size_t)d0 * kD + v;
        const float *gp = gam + ((size_t)bh * nseg + r) * kD + d0;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            s[x] = gp[x] * s[x] + E[base + x * kD];
            sstart[base + x * kD] = s[x];
        }
    }
}

bool g_attr_done = false;

cudaError_t set_attrs() {
    if (g_attr_done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gla_tc_out_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, om::ALLOC);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gla_tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sm_::ALLOC);
    if (e != cudaSuccess) return e;
    g_attr_done = true;
    return cudaSuccess;
}

int clamp_splits(const Problem &p, int splits) {
    const int64_t nchunks = (p.T + kC - 1) / kC;
    int64_t s = std::max<int64_t>(1, std::min<int64_t>(splits, nchunks));
    return (int)std::min<int64_t>(s, 64);
}

}  // namespace

bool tc_supported(const Problem &p) {
    return p.io == 0 && p.Dk == kD && p.Dv == kD && p.T < (int64_t(1) << 30) &&
           p.B * p.H < (int64_t(1) << 24);
}

int tc_auto_splits(const Problem &p, int num_sms) {
    const int64_t nchunks = (p.T + kC - 1) / kC;
    const int64_t bh = p.B * p.H;
    if (nchunks <= 1 || bh <= 0) return 1;
    // modelled time: waves of the output pass x chunks per segment, plus the state
    // pass (about 0.4 of an output-pass chunk) for every segment but the last
    double best = 1e30;
    int best_s = 1;
    for (int s = 1; s <= 32 && s <= nchunks; ++s) {
        const double per = (double)((nchunks + s - 1) / s);
        const double out_waves = (double)((bh * s + num_sms - 1) / num_sms);
        const double st_waves = s > 1 ? (double)((bh * (s - 1) + num_sms - 1) / num_sms) : 0.0;
        const double cost = out_waves * per + 0.4 * st_waves * per + 2.0 * (s > 1);
        if (cost < best - 1e-9) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

size_t tc_workspace_bytes(const Problem &p, int splits) {
    const int s = clamp_splits(p, splits);
    if (s <= 1) return 0;
    const size_t bh = (size_t)(p.B * p.H);
    return bh * (size_t)(s - 1) * (2 * (size_t)kD * kD + kD) * sizeof(float);
}

cudaError_t launch_tc(const Problem &p, int splits, void *ws, size_t ws_bytes,
                      unsigned int *dev_err, cudaStream_t stream) {
    if (p.T == 0) return launch_exact(p, dev_err, stream);   // only hT = h0 to write
    const int s = clamp_splits(p, splits);
    cudaError_t e = set_attrs();
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mg, mo;
    if (!make_bthd_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, p.T, p.H, kD, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, p.T, p.H, kD, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, p.T, p.H, kD, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.B, p.T, p.H, kD, kD, kC,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_bthd_map(&mo, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, p.T, p.H, kD, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidResourceHandle;   // a tensor map could not be encoded
    const int nchunks = (int)((p.T + kC - 1) / kC);
    const int bh = (int)(p.B * p.H);
    float *E = nullptr, *gam = nullptr, *sstart = nullptr;
    if (s > 1) {
        if (!ws || ws_bytes < tc_workspace_bytes(p, s)) return cudaErrorInvalidValue;
        E = static_cast<float *>(ws);
        sstart = E + (size_t)bh * (s - 1) * kD * kD;
        gam = sstart + (size_t)bh * (s - 1) * kD * kD;
        StateArgs sa{E, gam, p.T, (int)p.H, nchunks, s, dev_err};
        gla_tc_state_kernel<<<bh * (s - 1), kStateThreads, sm_::ALLOC, stream>>>(mk, mv, mg, sa);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        gla_tc_scan_kernel<<<dim3(bh, kD / 8), 128, 0, stream>>>(E, gam, p.h0, sstart, s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launches(2);
    }
    OutArgs oa{static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
               p.g, p.h0, p.hT, sstart, p.T, (int)p.H, nchunks, s, p.scale, dev_err};
    gla_tc_out_kernel<<<bh * s, kOutThreads, om::ALLOC, stream>>>(mq, mk, mv, mg, mo, oa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    count_launches(1);
    return cudaSuccess;
}

}  // namespace gla
