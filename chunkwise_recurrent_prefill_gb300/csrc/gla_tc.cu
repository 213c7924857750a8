// Tensor-core chunkwise GLA forward for sm_103a: TMA-staged tiles, tcgen05 MMAs with
// TMEM accumulators, fp32 state kept in TMEM across the chunk scan, warp-specialised
// roles. The chunk algebra is that of "线性注意力GPU算子库的定义与技术解析", section 四
// (blocks recurred locally, states carried block to block, in-block work as matrix
// products); the update it evaluates is the gated state update of "Linear Attention 在
// GPU 上到底慢在哪", section 学长的反馈.
//
// Per (batch, head) and chunk of C = 64 tokens with in-chunk inclusive cumulative
// log-gate b (a Dk vector per token) and chunk total Bc = b_63:
//     P  = (Q~ K~^T) masked to j <= i,  Q~ = q exp(b), K~ = k exp(-b)      (M=64 MMA)
//     O^T = V^T P^T + S^T Q~^T       (S^T bf16 from TMEM as the A operand)   (M=128)
//     S  <- diag(exp(Bc)) S + (k exp(Bc - b))^T V                            (M=128)
//     o  = scale * O
// The state is stored transposed in TMEM (lane = value column v, column = key row d),
// so every large MMA has M = 128. The output kernel keeps it decay-normalised:
// S = diag(exp(L)) S~, with L the per-key-row cumulative log-decay since the last
// renormalisation. Then the update is a pure accumulation S~ += K'^T V with
// K' = k exp(-(b + L)) and the inter term is Q' S~ with Q' = q exp(b + L); since
// Q' K'^T = Q~ K~^T the same two tiles serve the intra term too. No CUDA-core pass
// touches the fp32 state between two chunks except a bf16 snapshot for the inter MMA;
// the state is rescaled back (S~ <- exp(L) S~, L <- 0) only when |L| grows past a bound.
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
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gla_internal.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace gla {
namespace {

using namespace tc;

constexpr int kC = 64;                 // chunk length (tokens)
constexpr int kMaxSplits = 256;        // sequence segments per head, at most
constexpr int kMaxPieces = 8;          // state-pass pieces per segment, at most
constexpr int kD = 128;                // Dk = Dv
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kExtreme2 = 50.f;      // |b| (log2 units) beyond which P takes the exact route
constexpr float kRenorm2 = 50.f;       // |L| (log2 units) beyond which the state is renormalised
constexpr int64_t kL2KeepBytes = 64ll << 20;  // state-pass reads kept in L2 for the output pass
constexpr int kGateBlock = 8;          // tokens per load/compute/store block of the gate warps
constexpr unsigned kProducerNapNs = 128;  // idle back-off of the TMA producer's polling loop
constexpr unsigned kIssuerNapNs = 32;     // idle back-off of the MMA issuers' polling loops

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
// Global-timer stamps of every CTA (kernel k, event ev < 4), for the cross-kernel timeline.
#ifdef GLA_TRACE
constexpr int kTraceGlobCtas = 1024;
__device__ long long *g_trace_glob;
#define TRACE_GLOB(k, ev)                                                                     \
    do {                                                                                      \
        if (g_trace_glob && blockIdx.x < kTraceGlobCtas)                                      \
            g_trace_glob[((size_t)(k) * kTraceGlobCtas + blockIdx.x) * 4 + (ev)] = global_ns(); \
    } while (0)
#else
#define TRACE_GLOB(k, ev) \
    do {                  \
    } while (0)
#endif

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// TMEM column map of the output kernel (512 columns).
constexpr uint32_t kColS = 0;      // S~^T fp32, 128 columns
constexpr uint32_t kColSB = 128;   // S~^T bf16 snapshot (A operand), 2 x 64 columns
constexpr uint32_t kColP = 256;    // P (M=64 layout), 64 columns
constexpr uint32_t kColO = 320;    // O^T = S~^T Q'^T + V^T P^T, 64 columns
// head pairs (two heads of dims 64 as one of 128): the second head's P and O^T
constexpr uint32_t kColP2 = 384;
constexpr uint32_t kColO2 = 448;

// Shared-memory map of the output kernel (bytes from a 1024-aligned base).
//   q/k/v ring (3 stages): raw tiles as 128B-swizzled [64 x 64] bf16 boxes, two per tile;
//     the gate warps rewrite q -> Q' and k -> K' (or K^ in an extreme chunk) in place. With
//     head pairs, once the chunk's P and U MMAs (the readers of K') have completed, the two
//     heads' masked bf16 P tiles are written over K' (one box each). The stage is released
//     once the chunk's O MMAs (its last readers) have completed.
//   g ring (2 slots): the chunk's log-gates, [64 tokens][128] f32, loaded by TMA and
//     released as soon as the gate warps have scaled the chunk.
namespace om {
constexpr int NQ = 3;                   // q/k/v stages (per-key gates)
constexpr int NQS = 4;                  // q/k/v stages with a scalar gate: the fourth stage
                                        // takes the log-gate ring's space
constexpr int NG = 2;                   // log-gate slots
constexpr int NR = 4;                   // per-chunk ring of scales and flags (written by the
                                        // gates of c, read before O(c) completes)
constexpr uint32_t Q = 0, K = 16384, V = 32768, QSTAGE = 49152;
constexpr uint32_t G = NQ * QSTAGE, GSLOT = 32768;
constexpr uint32_t P = G + NG * GSLOT;  // [64 x 64] bf16 P tile, 128B swizzle (not head pairs)
constexpr uint32_t GAM = P + 8192;      // [NR][128] f32 exp(L_c): renormalisation scale
constexpr uint32_t GAM2 = GAM + NR * 512; // [NR][128] f32 exp(Bc) (extreme chunks)
constexpr uint32_t ENDS = GAM2 + NR * 512; // [128] f32 exp(L) after the latest chunk
constexpr uint32_t XF = ENDS + 512;     // [NR] u32 chunk flags: 1 = extreme, 2 = renormalise
constexpr uint32_t XCH = XF + 64;       // [<=4][128] f32 token-range totals of the gate warps
constexpr uint32_t GSC = XCH + 2048;    // [2][64] f32 scalar gates of two chunks (scalar mode)
constexpr uint32_t SCR = GSC + 512;     // [4][64] f32 exact-path scratch
constexpr uint32_t BAR = SCR + 1024;    // mbarriers
constexpr uint32_t NBAR = 27;
constexpr uint32_t TSLOT = BAR + NBAR * 8;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
static_assert(ALLOC <= 232448, "output kernel shared memory");
constexpr uint32_t FAC = NQS * QSTAGE;  // [64] float2 per-token factors (scalar gate)
constexpr int NQF = 8;                  // scalar gate: ring of the output's per-token factors
constexpr uint32_t QFR = FAC + 512;     // [NQF][64] f32
constexpr uint32_t RTOK = QFR + NQF * 256;  // [64] f32 running log2-gate sums within the ranges
static_assert(RTOK + 256 <= P, "scalar-gate stages and factors fit below the P tile");
}  // namespace om

// mbarrier indices of the output kernel
// (q/k/v rings of up to 4 stages: 4 with a scalar gate, whose log-gate ring is unused).
// With head pairs, whose P tiles live in the stages, the state warps may write P(c + 1) before
// O(c) is issued, so PBF (P tiles of chunk c written) alternates between two barriers, and
// snapshot(c) may reuse bf16 snapshot buffer c % 2 only once O(c - 2) has read it (SBFREE,
// two barriers): no barrier is ever two phases ahead of its waiter. A single head uses PBF
// alone (its P conversion waits for the previous chunk's O).
enum {
    QFULL = 0, QEMPTY = 4, GFULL = 8, GEMPTY = 10, GDONE = 12, PFULL = 16, PFREE = 17,
    SREADY = 18, UDONE = 19, OFULL = 20, OFREE = 21, FIN = 22, PBF = 23, SBFREE = 25,
};
static_assert(SBFREE + 2 <= (int)om::NBAR, "output kernel barrier map");

constexpr int kGateWarps = 6;          // warps 10..15 (4 warps with 32-token ranges measured
                                       // 3-5% slower at B*H = 64 and 256, equal at 16)
constexpr int kOutThreads = (10 + kGateWarps) * 32;   // at most 4 warps per SM
                                                       // sub-partition: 128 registers
constexpr int kGateThreads = kGateWarps * 32;
constexpr int kGateParts = kGateThreads / 64;   // token ranges (one thread per key pair each)
// Token ranges [0, 24), [24, 56), [56, 64). Warp w runs on sub-partition w % 4: ranges 0 and 2
// share sub-partitions 2 and 3 (warps 10, 14 and 11, 15), range 1 has 0 and 1 (warps 12, 13),
// so every sub-partition scales 32 tokens of a chunk (equal ranges of 24, 24, 16 left 40 on
// two of them).
__host__ __device__ constexpr int gate_range_begin(int part) {
    return part == 0 ? 0 : part == 1 ? 24 : part == 2 ? 56 : 64;
}
static_assert(kGateParts == 3 && gate_range_begin(kGateParts) == 64,
              "gate token ranges must cover the chunk");
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
    int stall_chunk;                   // test hook: chunk whose q/k/v load is never issued (-1)
    int last16;                        // weight of the last segment in 16ths (see seg_bound)
    const int *cu;                     // packed sequences: offsets [B+1] along T, or null
    __nv_bfloat16 *o;                  // output (rows a TMA store may not cover)
    int Dk, Dv;                        // head dims of the caller's tensors (64 or 128); the
                                       // kernels work at 128, padding with zeros
    int long_only;                     // packed sequences: skip those shorter than one chunk
};

struct StateArgs {
    float *E;                          // [BH][splits-1][Dk][Dv]
    float *gam;                        // [BH][splits-1][Dk]
    int64_t T;
    int H, nchunks, splits;
    unsigned *err;
    int retain;                        // chunks per CTA (read last) loaded with evict_last
    int last16;                        // weight of the last segment in 16ths (see seg_bound)
    int pieces;                        // consecutive pieces per segment, one CTA each
    const float *g;                    // scalar log-gates [B,T,H] (scalar mode only)
};

// Chunk range [cb, ce) of segment `seg`. Every segment weighs 16 except the last, which
// weighs `last16`: it is the only one the state pass does not read, so none of its tiles are
// in L2 when the output pass reaches them, and it is made shorter in proportion to what the
// others gain from L2. Short segments (fewer than 8 chunks each) are split evenly, so no
// segment is ever empty.
__device__ __host__ __forceinline__ int seg_bound(int j, int nchunks, int splits, int last16) {
    if (j >= splits) return nchunks;
    if (nchunks < 8 * splits) return (int)((int64_t)j * nchunks / splits);
    return (int)((int64_t)j * nchunks * 16 / (16 * (splits - 1) + last16));
}

__device__ __forceinline__ void seg_range(int seg, int nchunks, int splits, int last16, int &cb,
                                          int &ce) {
    cb = seg_bound(seg, nchunks, splits, last16);
    ce = seg_bound(seg + 1, nchunks, splits, last16);
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
// On return b0/b1 hold the chunk-inclusive cumulative log2-gates of the thread's tokens,
// and every participating thread has finished reading `gs`.
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

// gate_cumsum for a scalar gate: gs holds the chunk's 64 per-token log-gates, the same in
// every key dimension (so both columns of the pair see them).
__device__ __forceinline__ void gate_cumsum_scalar(const float *gs, float *xch, int qq, int d,
                                                   float (&b0)[16], float (&b1)[16],
                                                   uint32_t bar) {
    float a0 = 0.f;
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        a0 = fmaf(gs[16 * qq + x], kLog2e, a0);
        b0[x] = a0;
        b1[x] = a0;
    }
    *reinterpret_cast<float2 *>(xch + qq * kD + d) = make_float2(a0, a0);
    named_bar_sync(bar, 256);
    float o0 = 0.f;
    for (int q2 = 0; q2 < qq; ++q2) o0 += xch[q2 * kD + d];
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        b0[x] += o0;
        b1[x] += o0;
    }
}

// Phase parity of the k-th use of a ring slot.
__device__ __forceinline__ uint32_t par(int use) { return (uint32_t)use & 1u; }

// ======================================================================= output kernel
// Warp roles (10 + kGateWarps warps): 0 TMA producer, 1 MMA scheduler (one thread), 2-5 epilogue,
// 6-9 state + P conversion, the rest gate warps.
// kScalar: one log-gate per token and head (g [B,T,H]) instead of one per key dimension; the
// gates are then read by the gate warps straight from global memory, a chunk ahead.
// kPacked: the batches are sequences packed along one token axis at offsets a.cu; the rows
// of a sequence's last chunk past its end are masked (batched tensors need no masking: the
// rows past T are zero-filled by the tensor copies and clipped by the stores).
// kPair: the tensors hold head pairs (2p, 2p + 1) of dims 64 as heads p of dims 128
// (adjacent heads are contiguous in [B,T,H,64], so the tiles are the same). The state of a
// pair is block diagonal; its off-diagonal blocks collect cross-head products that are never
// read: the bf16 snapshot (the only operand read from the state) zeroes them, and hT
// writes the diagonal blocks. P and the intra term are per head: P of the second head
// accumulates apart, each head's P tile fills one of the two boxes of the chunk's K' region,
// and the second head's O^T (its lanes are value columns 64..127) accumulates in a second
// column block.
template <bool kScalar, bool kPacked, bool kPair = false>
__global__ void __launch_bounds__(kOutThreads, 1)
gla_tc_out_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                  const OutArgs a) {
    using namespace om;
    constexpr int NQ = kScalar ? NQS : om::NQ;   // q/k/v stages of this instance
    // P tiles in the stage (head pairs: two per chunk, no wait for the previous chunk's O);
    // otherwise one P tile, rewritten once the previous chunk's O MMAs have completed (that
    // order measured 3-5 % faster for a single head, whose state warps would otherwise wait
    // for the chunk's own state update)
    constexpr bool kStageP = kPair;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TSLOT);
    float *gam_s = reinterpret_cast<float *>(sm + GAM);
    float *gam2_s = reinterpret_cast<float *>(sm + GAM2);
    float *ends_s = reinterpret_cast<float *>(sm + ENDS);
    uint32_t *xf = reinterpret_cast<uint32_t *>(sm + XF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x % a.splits;
    const int bh = blockIdx.x / a.splits;
    const int bidx = bh / a.H, h = bh % a.H;
    // Tokens of this CTA's sequence: [tbase, tend) along the T axis of the tensors, in batch
    // bmap. Packed sequences (a.cu) all live in batch 0 and are not split.
    int64_t tbase = 0, tend = a.T;
    int bmap = bidx;
    bool bad_seq = false;
    if (kPacked) {
        const int s0 = a.cu[bidx], s1 = a.cu[bidx + 1];
        bad_seq = s0 < 0 || s1 < s0 || s1 > a.T;
        tbase = bad_seq ? 0 : s0;
        tend = bad_seq ? 0 : s1;
        bmap = 0;
        // a sequence shorter than one chunk is left to the exact kernel of the same call
        // (uniform across the CTA, before any barrier or allocation)
        if (a.long_only && !bad_seq && tend - tbase < kC) return;
    }
    int cb, ce;
    if (kPacked) {
        cb = 0;
        ce = (int)((tend - tbase + kC - 1) / kC);
    } else {
        seg_range(seg, a.nchunks, a.splits, a.last16, cb, ce);
    }
    const int n = ce - cb;
    // valid rows of chunk c (64 except at the end of a sequence)
    auto valid_rows = [&](int c) -> int {
        const int64_t left = tend - tbase - (int64_t)(cb + c) * kC;
        return left >= kC ? kC : (int)left;
    };

    if (threadIdx.x < kD) reinterpret_cast<float *>(sm + ENDS)[threadIdx.x] = 1.f;  // L = 0
    if (threadIdx.x == 0) {
        if (bad_seq) atomicOr(a.err, kDevErrInternal);
        for (int i = 0; i < NQ; ++i) {
            mbar_init(&bars[QFULL + i], 1);
            mbar_init(&bars[QEMPTY + i], 1);
            mbar_init(&bars[GDONE + i], kGateWarps);
        }
        for (int i = 0; i < NG; ++i) {
            mbar_init(&bars[GFULL + i], 1);
            mbar_init(&bars[GEMPTY + i], kGateWarps);
        }
        mbar_init(&bars[PFULL], 1);
        mbar_init(&bars[PFREE], 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[PBF + i], 4);
            mbar_init(&bars[SBFREE + i], 1);
        }
        mbar_init(&bars[SREADY], 4);
        mbar_init(&bars[UDONE], 1);
        mbar_init(&bars[OFULL], 1);
        mbar_init(&bars[OFREE], 4);
        mbar_init(&bars[FIN], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tg);
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;
    if (threadIdx.x == 0) TRACE_OUT(14, 0);
    if (threadIdx.x == 0) TRACE_GLOB(0, 0);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // Two rings filled independently: the log-gate slots (freed early, by the gate
        // warps) and the q/k/v stages (freed after the chunk's output store read them).
        if (lane == 0) {
            // every tile is read here for the last time: do not let it displace the chunks
            // the state kernel left in L2 for this kernel
            const uint64_t pol = l2_policy_evict_first();
            int ng = kScalar ? n : 0, nq = 0;   // scalar gates are not staged by TMA
            uint32_t idle = 0;
            uint64_t t_idle = 0;
            while (ng < n || nq < n) {
                bool prog = false;
                if (ng < n && (ng < NG || mbar_test(&bars[GEMPTY + ng % NG], par(ng / NG - 1)))) {
                    uint64_t *fb = &bars[GFULL + ng % NG];
                    mbar_arrive_expect_tx(fb, GSLOT);
                    tma_load_4d_hint(sm + G + (ng % NG) * GSLOT, &tg, fb, 0, h,
                                     (int)(tbase + (cb + ng) * kC), bmap, pol);
                    ++ng;
                    prog = true;
                }
                if (nq < n && (nq < NQ || mbar_test(&bars[QEMPTY + nq % NQ], par(nq / NQ - 1)))) {
                    uint8_t *base = sm + (nq % NQ) * QSTAGE;
                    uint64_t *fb = &bars[QFULL + nq % NQ];
                    TRACE_OUT(0, nq);
                    const int t = (int)(tbase + (cb + nq) * kC);
                    mbar_arrive_expect_tx(fb, 3 * 16384);
                    if (nq == a.stall_chunk) {   // test hook: the stage never fills
                        ++nq;
                        prog = true;
                        continue;
                    }
                    tma_load_4d_hint(base + Q, &tq, fb, 0, h, t, bmap, pol);
                    tma_load_4d_hint(base + Q + 8192, &tq, fb, 64, h, t, bmap, pol);
                    tma_load_4d_hint(base + K, &tk, fb, 0, h, t, bmap, pol);
                    tma_load_4d_hint(base + K + 8192, &tk, fb, 64, h, t, bmap, pol);
                    tma_load_4d_hint(base + V, &tv, fb, 0, h, t, bmap, pol);
                    tma_load_4d_hint(base + V + 8192, &tv, fb, 64, h, t, bmap, pol);
                    ++nq;
                    prog = true;
                }
                if (prog) {
                    idle = 0;
                } else {
                    // yield the issue slots of this sub-partition to the compute warps
                    __nanosleep(kProducerNapNs);
                    if (++idle == 256) {
                        t_idle = global_ns();   // the timer is read only on long idle streaks
                    } else if ((idle & 1023) == 0 && global_ns() - t_idle > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            // never leave with a bulk copy still landing in this CTA's shared memory
            for (int i = 0; i < NQ; ++i) {
                const int uses = nq > i ? (nq - 1 - i) / NQ + 1 : 0;
                if (uses > 0 && !mbar_wait(&bars[QFULL + i], par(uses - 1))) ok = false;
            }
            for (int i = 0; i < NG && !kScalar; ++i) {
                const int uses = ng > i ? (ng - 1 - i) / NG + 1 : 0;
                if (uses > 0 && !mbar_wait(&bars[GFULL + i], par(uses - 1))) ok = false;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA scheduler
        // Three MMA groups per chunk c, each issued back to back once its inputs are ready:
        //   U(c): snapshot of S~_c taken            -> S~ += K'^T V                (4 steps)
        //   P(c): gates of c done, P(c-1) read      -> P1 (d 0..63), P2 (d 64..127) (2 x 4)
        //   O(c): P tile of c written, O(c-1) read  -> Os = S~^T Q'^T (8), Oi = V^T P^T (4)
        //         (head pairs: the same for the second head into its own column block)
        // MMAs that accumulate into TMEM run at their latency, one after another, so the
        // order only decides who waits: U first (the state chain), then P, then O.
        // The whole warp runs the loop converged: every lane polls, lane 0's view of each
        // barrier decides (broadcast), and one elected lane issues the MMAs and commits.
        {
            const uint32_t idP = idesc_bf16(64, 64, 0, 0);
            const uint32_t idU = idesc_bf16(128, 128, 1, 1);
            const uint32_t idOi = idesc_bf16(128, 64, 1, 0);
            const uint32_t idOs = idesc_bf16(128, 64, 0, 0);
            int np = 0, nu = 0, no = 0;
            uint32_t idle = 0;
            uint64_t t_idle = 0;
            while (no < n) {
                bool prog = false;
                const bool rU = __shfl_sync(0xffffffffu, nu < np && mbar_test(&bars[SREADY], par(nu)), 0);
                if (rU) {
                    tc_fence_after();
                    if (lane == 0) TRACE_OUT(5, nu);
                    const uint32_t base = smem_u32(sm + (nu % NQ) * QSTAGE);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tm + kColS, smem_desc(base + V + kk * 2048, 8192, 1024),
                                   smem_desc(base + K + kk * 2048, 8192, 1024), idU, 1);
                        mma_commit(&bars[UDONE]);
                    }
                    __syncwarp();
                    ++nu;
                    prog = true;
                }
                const bool rP = __shfl_sync(
                    0xffffffffu, np < n && mbar_test(&bars[GDONE + np % NQ], par(np / NQ)) &&
                                     (np == 0 || mbar_test(&bars[PFREE], par(np - 1))), 0);
                if (rP) {
                    tc_fence_after();
                    if (lane == 0) TRACE_OUT(3, np);
                    const uint32_t base = smem_u32(sm + (np % NQ) * QSTAGE);
                    if (elect_one()) {
#pragma unroll
                        for (int x = 0; x < 8; ++x) {   // key dims 16x .. 16x + 15
                            const uint32_t off = (x >> 2) * 8192 + (x & 3) * 32;
                            // head pairs: each head's P over its own 64 key dims
                            const uint32_t dst = (kPair && x >= 4) ? kColP2 : kColP;
                            mma_ss(tm + dst, smem_desc(base + Q + off, 16, 1024),
                                   smem_desc(base + K + off, 16, 1024), idP,
                                   kPair ? (x & 3) > 0 : x > 0);
                        }
                        mma_commit(&bars[PFULL]);
                    }
                    __syncwarp();
                    if (lane == 0) TRACE_OUT(4, np);
                    ++np;
                    prog = true;
                }
                const bool rO = __shfl_sync(
                    0xffffffffu, no < nu &&
                                     mbar_test(&bars[PBF + (kStageP ? no & 1 : 0)],
                                               kStageP ? par(no >> 1) : par(no)) &&
                                     (no == 0 || mbar_test(&bars[OFREE], par(no - 1))), 0);
                if (rO) {
                    tc_fence_after();
                    if (lane == 0) TRACE_OUT(6, no);
                    const uint32_t base = smem_u32(sm + (no % NQ) * QSTAGE);
                    const uint32_t pbase = kStageP ? base + K : smem_u32(sm + P);
                    if (elect_one()) {
                        // one accumulator per head: the inter term S~^T Q'^T, then the intra term
                        // V^T P^T with the head's P tile
#pragma unroll
                        for (int hp = 0; hp < (kPair ? 2 : 1); ++hp) {
                            const uint32_t dst = hp ? kColO2 : kColO;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                mma_ts(tm + dst, tm + kColSB + (no & 1) * 64 + kk * 8,
                                       smem_desc(base + Q + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                                       idOs, kk > 0);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(tm + dst, smem_desc(base + V + kk * 2048, 8192, 1024),
                                       smem_desc(pbase + hp * 8192 + kk * 32, 16, 1024), idOi, 1);
                        }
                        // U(no) and P(no) were issued before O(no)
                        mma_commit(&bars[OFULL]);
                        if (kStageP) mma_commit(&bars[SBFREE + (no & 1)]);
                    }
                    __syncwarp();
                    if (lane == 0) TRACE_OUT(7, no);
                    ++no;
                    prog = true;
                }
                if (prog) {
                    idle = 0;
                } else {
                    // yield the issue slots of this sub-partition to the compute warps
                    __nanosleep(kIssuerNapNs);
                    if (++idle == 256) {
                        t_idle = global_ns();   // the timer is read only on long idle streaks
                    } else if ((idle & 1023) == 0 &&
                               __shfl_sync(0xffffffffu, global_ns() - t_idle > kWaitLimitNs, 0)) {
                        ok = false;
                        break;
                    }
                }
            }
            // all issued MMAs complete before the CTA tears down its TMEM
            if (elect_one()) mma_commit(&bars[FIN]);
            __syncwarp();
            if (!mbar_wait(&bars[FIN], 0)) ok = false;
        }
        __syncwarp();
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------------------ epilogue
        // O^T(c) from TMEM (lane = value column v, column = token), rounded to bf16 and
        // stored straight to global memory: a warp writes 64 contiguous bytes of a token row
        // per store. Once O(c) has completed, every MMA of chunk c has (they complete in issue
        // order), so its q/k/v stage is released right away.
        const int j = warp & 3;
        const int et = (warp - 2) * 32 + lane;      // 0..127
        const int v = j * 32 + lane;                // O^T lane = value column
        const uint64_t pol = l2_policy_evict_first();
        const int64_t rs = (int64_t)a.H * a.Dv;     // row stride of o (elements)
        for (int c = 0; c < n; ++c) {
            const bool w = mbar_wait(&bars[OFULL], par(c));
            if (named_bar_or(2, 128, !w)) { ok = false; break; }
            if (et == 0) TRACE_OUT(12, c);
            tc_fence_after();
            if (et == 0) mbar_arrive(&bars[QEMPTY + c % NQ]);   // the stage may be refilled
            float ov[64];
            tmem_ld64(tmem_addr(tm, j, (kPair && j >= 2) ? kColO2 : kColO), ov);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[OFREE]);
            const int64_t t0 = tbase + (int64_t)(cb + c) * kC;
            const int64_t left = tend - t0;
            const int vr = left < kC ? (int)left : kC;   // rows of the sequence
            if (kScalar) {
                // a scalar gate's q is not scaled in place: O = f_t (S~^T q^T + V^T P'^T) with
                // f_t = scale 2^(b_t + L) (1 in an extreme chunk, whose q is scaled)
                const float *qf = reinterpret_cast<const float *>(sm + QFR) + (c & (NQF - 1)) * kC;
#pragma unroll
                for (int x = 0; x < kC; ++x) ov[x] *= qf[x];
            }
            if (v < a.Dv) {
                __nv_bfloat16 *op = a.o + ((((int64_t)bmap * a.T + t0) * a.H + h) * a.Dv) + v;
                if (vr == kC) {
#pragma unroll
                    for (int x = 0; x < kC; ++x)
                        st_global_bf16_hint(op + x * rs, __float2bfloat16_rn(ov[x]), pol);
                } else {
#pragma unroll
                    for (int x = 0; x < kC; ++x)
                        if (x < vr) st_global_bf16_hint(op + x * rs, __float2bfloat16_rn(ov[x]), pol);
                }
            }
            if (et == 0) TRACE_OUT(13, c);
        }
        __syncwarp();
    } else if (warp >= 6 && warp < 10) {
        // ------------------------------------------------------------ state + P conversion
        // The TMEM state is decay-normalised: S_c = diag(exp(L_c)) S~_c. Pass c takes the
        // bf16 snapshot of S~_c for O(c) (a renormalising chunk first restores S~ = S_c, an
        // extreme chunk also pre-scales by exp(Bc) before its U), then turns P(c) into the
        // masked bf16 P tile.
        const int j = warp & 3;
        const int v = j * 32 + lane;
        const int st_t = (warp - 6) * 32 + lane;     // 0..127
        float *scr = reinterpret_cast<float *>(sm + SCR);
        const float *init = nullptr;
        if (seg > 0) {
            // the start states come from the scan kernel, which may still be running: this
            // kernel is launched as its programmatic dependent
            pdl_wait_prerequisites();
            if (threadIdx.x == 6 * 32) TRACE_GLOB(0, 1);
            init = a.sstart + ((size_t)bh * (a.splits - 1) + (seg - 1)) * (kD * kD);
        } else if (a.h0) {
            // head pairs: this lane's value column belongs to head 2 bh + v / 64, whose 64 x 64
            // h0 fills the diagonal block of its key rows
            init = kPair ? a.h0 + ((size_t)2 * bh + (v >> 6)) * 4096
                         : a.h0 + (size_t)bh * a.Dk * a.Dv;
        }
        // start states are 128 x 128 internally; h0 has the caller's Dk x Dv (zero padded)
        const int irows = seg > 0 ? kD : a.Dk, icols = seg > 0 ? kD : a.Dv;
#pragma unroll 1
        for (int d0 = 0; d0 < kD; d0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int d = d0 + x;
                if (kPair && seg == 0)
                    r[x] = (init && (d >> 6) == (v >> 6))
                               ? __float_as_uint(init[(d & 63) * 64 + (v & 63)]) : 0u;
                else
                    r[x] = (init && d < irows && v < icols)
                               ? __float_as_uint(init[d * icols + v]) : 0u;
            }
            tmem_st16(tmem_addr(tm, j, kColS + d0), r);
        }
        tmem_wait_st();
        for (int c = 0; c < n; ++c) {
            // ---- snapshot of S~_c
            // (the snapshot buffer c % 2 is free once O(c - 2) has completed: without P tiles
            // in the stages, the P conversion of c - 1 below waited for it)
            bool w = (c == 0 || mbar_wait(&bars[UDONE], par(c - 1))) &&
                     mbar_wait(&bars[GDONE + c % NQ], par(c / NQ)) &&
                     (!kStageP || c < 2 ||
                      mbar_wait(&bars[SBFREE + (c & 1)], par((c >> 1) - 1)));
            if (named_bar_or(3, 128, !w)) { ok = false; break; }
            if (v == 0) TRACE_OUT(8, c);
            tc_fence_after();
            const uint32_t fl = xf[c & (NR - 1)];
            const bool ext = (fl & 1u) != 0, ren = (fl & 2u) != 0;
            const float *gl = gam_s + (c & (NR - 1)) * 128;    // exp(L_c)
            const float *gb = gam2_s + (c & (NR - 1)) * 128;   // exp(Bc)
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float sv[64];
                tmem_ld64(tmem_addr(tm, j, kColS + half * 64), sv);
                if (ren) {
#pragma unroll
                    for (int x = 0; x < 64; ++x) sv[x] *= gl[half * 64 + x];
                }
                // head pairs: the blocks across heads are not state; the snapshot holds zeros
                const bool cross = kPair && half != (j >> 1);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t pk[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        pk[x] = cross ? 0u : pack_bf16(sv[16 * cc + 2 * x], sv[16 * cc + 2 * x + 1]);
                    tmem_st8(tmem_addr(tm, j, kColSB + (c & 1) * 64 + half * 32 + cc * 8), pk);
                }
                if (ext) {
#pragma unroll
                    for (int x = 0; x < 64; ++x) sv[x] *= gb[half * 64 + x];
                }
                if (ren) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t r[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(sv[16 * cc + x]);
                        tmem_st16(tmem_addr(tm, j, kColS + half * 64 + 16 * cc), r);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[SREADY]);
            if (v == 0) TRACE_OUT(9, c);
            // ---- P(c) -> masked bf16 P tile: over K' of chunk c's stage once its readers (the P
            // and U MMAs of c) have completed, or in the P tile once O(c - 1) has read it
            w = mbar_wait(&bars[PFULL], par(c)) &&
                (kStageP ? mbar_wait(&bars[UDONE], par(c))
                         : (c == 0 || mbar_wait(&bars[OFULL], par(c - 1))));
            if (named_bar_or(3, 128, !w)) { ok = false; break; }
            if (v == 0) TRACE_OUT(10, c);
            tc_fence_after();
            // head pairs: one P tile per head, in the two boxes of the K' region
#pragma unroll 1
            for (int ph = 0; ph < (kPair ? 2 : 1); ++ph) {
                uint8_t *pt = kStageP ? sm + (c % NQ) * QSTAGE + K + ph * 8192 : sm + P;
                if (!kScalar && !ext) {
                    // the warp's 16 P rows (lanes 0..15 of its quarter) spread over all 32
                    // threads: rows ia = 16 j + lane / 4 and ia + 8, column pairs 8 k + 2 (lane % 4)
                    // (with a scalar gate this measured 4 % slower than one row per lane < 16)
                    uint32_t pr[32];
                    {
                        uint32_t r0[16], r1[16];
                        const uint32_t ta = tmem_addr(tm, j, ph ? kColP2 : kColP);
                        tmem_ld16x256b_x4(ta, r0);
                        tmem_ld16x256b_x4(ta + 32, r1);
                        tmem_wait_ld();
                        reg_fence(r0);
                        reg_fence(r1);
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            pr[x] = r0[x];
                            pr[16 + x] = r1[x];
                        }
                    }
                    if (!kPair || ph == 1) {   // every P accumulator of c has been read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[PFREE]);
                    }
                    const int ia = 16 * j + (lane >> 2), ib = ia + 8, c0 = 2 * (lane & 3);
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int col = 8 * k8 + c0;
                        const float *f = reinterpret_cast<const float *>(pr + 4 * k8);
                        *reinterpret_cast<uint32_t *>(pt + sw128_offset(ia, col)) =
                            pack_bf16(col <= ia ? f[0] : 0.f, col + 1 <= ia ? f[1] : 0.f);
                        *reinterpret_cast<uint32_t *>(pt + sw128_offset(ib, col)) =
                            pack_bf16(col <= ib ? f[2] : 0.f, col + 1 <= ib ? f[3] : 0.f);
                    }
                } else {
                    // one P row per lane < 16: the accumulator, or in an extreme chunk the exact
                    // route P_ij = scale sum_d q_id k_jd exp(b_id - b_jd), j <= i
                    float prow[64];
                    const int i = 16 * j + lane;
                    if (!ext) {
                        tmem_ld64(tmem_addr(tm, j, ph ? kColP2 : kColP), prow);
                    } else {
#pragma unroll
                        for (int x = 0; x < 64; ++x) prow[x] = 0.f;
                        float *gcol = scr, *qcol = scr + 64, *kcol = scr + 128, *bcol = scr + 192;
                        const int64_t t0 = tbase + (int64_t)(cb + c) * kC;
                        const int dlo = kPair ? 64 * ph : 0, dhi = kPair ? dlo + 64 : a.Dk;
                        for (int d = dlo; d < dhi; ++d) {   // padded key dims add nothing
                            if (st_t < 64) {
                                const int64_t t = t0 + st_t;
                                const bool in = t < tend;
                                const int64_t idx = (((int64_t)bmap * a.T + t) * a.H + h) * a.Dk + d;
                                gcol[st_t] = in ? (kScalar ? a.g[idx / a.Dk] : a.g[idx]) : 0.f;
                                qcol[st_t] = in ? __bfloat162float(a.q[idx]) : 0.f;
                                kcol[st_t] = in ? __bfloat162float(a.k[idx]) : 0.f;
                            }
                            named_bar_sync(3, 128);
                            if (st_t == 0) {
                                float s = 0.f;
                                for (int t = 0; t < 64; ++t) { s += gcol[t]; bcol[t] = s; }
                            }
                            named_bar_sync(3, 128);
                            if (lane < 16) {
                                const float qi = a.scale * qcol[i], bi = bcol[i];
#pragma unroll
                                for (int x = 0; x < 64; ++x)
                                    if (x <= i) prow[x] += qi * kcol[x] * ex2((bi - bcol[x]) * kLog2e);
                            }
                            named_bar_sync(3, 128);
                        }
                    }
                    if (!kPair || ph == 1) {   // every P accumulator of c has been read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[PFREE]);
                    }
                    if (lane < 16) {
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) {
                            uint32_t wv[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const int col = cc * 8 + 2 * x;
                                wv[x] = pack_bf16(col <= i ? prow[col] : 0.f,
                                                  col + 1 <= i ? prow[col + 1] : 0.f);
                            }
                            *reinterpret_cast<uint4 *>(pt + sw128_offset(i, cc * 8)) =
                                make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[PBF + (kStageP ? c & 1 : 0)]);
            if (v == 0) TRACE_OUT(11, c);
        }
        if (ok && !bad_seq && a.hT && seg == a.splits - 1) {
            if (n > 0 && !mbar_wait(&bars[UDONE], par(n - 1))) {
                ok = false;
            } else {
                tc_fence_after();
                if (kPair) {
                    // the diagonal block of this lane's head: key rows of the same half
                    const int hb = j >> 1;
                    float *hq = a.hT + ((size_t)2 * bh + hb) * 4096 + (v & 63);
                    float sv[64];
                    tmem_ld64(tmem_addr(tm, j, kColS + hb * 64), sv);
#pragma unroll
                    for (int x = 0; x < 64; ++x) hq[x * 64] = sv[x] * ends_s[hb * 64 + x];
                } else {
                    float *hp = a.hT + (size_t)bh * a.Dk * a.Dv + v;
#pragma unroll 1
                    for (int half = 0; half < a.Dk / 64; ++half) {
                        float sv[64];
                        tmem_ld64(tmem_addr(tm, j, kColS + half * 64), sv);
                        if (v < a.Dv) {
#pragma unroll
                            for (int x = 0; x < 64; ++x)
                                hp[(half * 64 + x) * a.Dv] = sv[x] * ends_s[half * 64 + x];
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ gate warps
        // Thread (part, dp) owns the key-dimension pair d = 2 dp, 2 dp + 1 over one of the
        // kGateParts token ranges of a chunk (gate_range_begin). Pass 1 sums the range's
        // log2-gates and records the range of the running sums; the ranges exchange totals,
        // and the warps agree on the chunk's flags (extreme, renormalise). Pass 2 recomputes
        // the running sums while scaling q and k in place, two dimensions per 32-bit access.
        const int gt = (warp - 10) * 32 + lane;             // 0 .. kGateThreads - 1
        const int dp = gt & 63, part = gt >> 6;
        const int tb = gate_range_begin(part);              // first token of the range
        const int tl = gate_range_begin(part + 1) - tb;     // tokens in the range
        const int d = 2 * dp;
        const uint32_t boxo = (uint32_t)(d >> 6) * 8192;
        const uint32_t col = (uint32_t)(d & 63);
        // byte offsets of this thread's column within each row of an 8-row swizzle atom
        // (blocks start on multiples of 8 rows, so row % 8 is the index within the block)
        static_assert(kGateBlock % 8 == 0 && gate_range_begin(1) % kGateBlock == 0 &&
                          gate_range_begin(2) % kGateBlock == 0,
                      "gate blocks must cover whole swizzle atoms");
        uint32_t swz[kGateBlock];
#pragma unroll
        for (int x = 0; x < kGateBlock; ++x) swz[x] = sw128_offset((uint32_t)x, col);
        const float sc = a.scale;
        const float lsc = log2f(sc);                        // folded into the q exponent
        float *xch = reinterpret_cast<float *>(sm + XCH);   // [3][128] range totals
        float L0 = 0.f, L1 = 0.f;   // log2 decay of the normalised state (S = 2^L S~)
        // scalar gates: thread gt < 64 fetches token gt of the next chunk into gpre; at the top
        // of each chunk they are published in gsc[c & 1] (two buffers: no thread is ever more
        // than one chunk behind another, the loop has several barriers per chunk)
        float *gsc = reinterpret_cast<float *>(sm + GSC);
        float *rtok = reinterpret_cast<float *>(sm + RTOK);
        auto fetch_scalar = [&](int c) -> float {
            const int64_t t = tbase + (int64_t)(cb + c) * kC + gt;
            return t < tend ? __ldg(a.g + ((int64_t)bmap * a.T + t) * a.H + h) : 0.f;
        };
        float gpre = (kScalar && gt < kC && n > 0) ? fetch_scalar(0) : 0.f;
        for (int c = 0; c < n; ++c) {
            const int gs = c % NG, qs = c % NQ, slot = c & (NR - 1);
            bool w = true;
            if (kScalar) {
                if (gt < kC) {
                    gsc[(c & 1) * kC + gt] = gpre;
                    if (c + 1 < n) gpre = fetch_scalar(c + 1);
                }
                named_bar_sync(1, kGateThreads);
            } else {
                w = mbar_wait(&bars[GFULL + gs], par(c / NG));
                if (named_bar_or(1, kGateThreads, !w)) { ok = false; break; }
            }
            if (gt == 0) TRACE_OUT(16, c);
            const float *grow = reinterpret_cast<const float *>(sm + G + gs * GSLOT) + tb * kD + d;
            const float *gsrow = gsc + (c & 1) * kC + tb;   // scalar gates of this thread's range
            const int vr = kPacked ? valid_rows(c) : kC;
            if (!kScalar && kPacked && vr < kC) {
                // rows past the sequence end hold another sequence's gates (packed sequences):
                // this thread's own elements of them become 0 (no decay) before it reads them
                for (int t = max(vr - tb, 0); t < tl; ++t)
                    *reinterpret_cast<float2 *>(const_cast<float *>(grow) + t * kD) =
                        make_float2(0.f, 0.f);
            }
            auto gpair = [&](int t) -> float2 {
                if (kScalar) {
                    const float x = gsrow[t];
                    return make_float2(x, x);
                }
                return *reinterpret_cast<const float2 *>(grow + t * kD);
            };
            const float2 l2e = make_float2(kLog2e, kLog2e);
            float2 rs = make_float2(0.f, 0.f);                   // running sums of the pair
            float lo0 = 0.f, hi0 = 0.f, lo1 = 0.f, hi1 = 0.f;   // range of the running sums
#pragma unroll 1
            for (int t0 = 0; t0 < tl; t0 += kGateBlock) {
                float2 gv[kGateBlock];
#pragma unroll
                for (int x = 0; x < kGateBlock; ++x) gv[x] = gpair(t0 + x);
#pragma unroll
                for (int x = 0; x < kGateBlock; ++x) {
                    rs = fma2(gv[x], l2e, rs);
                    lo0 = fminf(lo0, rs.x); hi0 = fmaxf(hi0, rs.x);
                    lo1 = fminf(lo1, rs.y); hi1 = fmaxf(hi1, rs.y);
                    // scalar gate: every key pair forms the same sums; the first pair of each
                    // range publishes them for the per-token factors below
                    if (kScalar && dp == 0) rtok[tb + t0 + x] = rs.x;
                }
            }
            *reinterpret_cast<float2 *>(xch + part * kD + d) = rs;
            // the exchange barrier also ORs the renormalisation test of the state so far
            const bool renL = named_bar_or(1, kGateThreads, fabsf(L0) > kRenorm2 || fabsf(L1) > kRenorm2);
            // b = off + (running sum within the range), with off the left-to-right sum of the
            // earlier ranges' totals; the chunk total is formed by the same additions, so that
            // b of the last token equals it exactly
            float off0 = 0.f, off1 = 0.f, B0 = 0.f, B1 = 0.f;
#pragma unroll
            for (int q = 0; q < kGateParts; ++q) {
                const float2 t = *reinterpret_cast<const float2 *>(xch + q * kD + d);
                if (q == part) { off0 = B0; off1 = B1; }
                B0 = q == 0 ? t.x : B0 + t.x;
                B1 = q == 0 ? t.y : B1 + t.y;
            }
            // largest |b| over this thread's tokens (attained at an end of the range)
            const float mx = fmaxf(fmaxf(fabsf(off0 + lo0), fabsf(off0 + hi0)),
                                   fmaxf(fabsf(off1 + lo1), fabsf(off1 + hi1)));
            const bool ext = named_bar_or(1, kGateThreads, mx > kExtreme2);
            const bool ren = renL || ext;
            if (gt == 0) TRACE_OUT(17, c);
            const float Lc0 = L0, Lc1 = L1;                     // before this chunk
            const float Lq0 = ren ? 0.f : L0, Lq1 = ren ? 0.f : L1;   // used by this chunk
            L0 = ext ? 0.f : Lq0 + B0;
            L1 = ext ? 0.f : Lq1 + B1;
            if (gt == 0) TRACE_OUT(18, c);
            // scalar gate: the factors are the same in every key dimension, so the 64 token
            // threads compute them once per chunk (two ex2 each) for pass 2 to multiply by, from
            // the running sums pass 1 published and the range offset formed as the key-pair
            // threads form it (so the numbers are the same). The barrier after the stage wait
            // below publishes them.
            float2 *fac = reinterpret_cast<float2 *>(sm + FAC);
            if (kScalar && gt < kC) {
                const int pt = (gt >= gate_range_begin(1)) + (gt >= gate_range_begin(2));
                const float rt = rtok[gt];
                float Bt = 0.f, offt = 0.f;
#pragma unroll
                for (int q = 0; q < kGateParts; ++q) {
                    const float tq = xch[q * kD];
                    if (q == pt) offt = Bt;
                    Bt = q == 0 ? tq : Bt + tq;
                }
                // the output's factor of this token, for the epilogue: q stays raw in a normal
                // chunk (its factor applies to O), and is scaled in place in an extreme one. The
                // ring slot of chunk c was last read by the epilogue of chunk c - NQF, which ended
                // before the stage of chunk c - NQF + NQ could arrive.
                float *qfr = reinterpret_cast<float *>(sm + QFR) + (c & (NQF - 1)) * kC;
                if (!ext) {
                    const float eq = offt + Lq0 + lsc, ek = -(offt + Lq0);
                    const float fq = ex2(rt + eq);
                    fac[gt] = make_float2(fq, ex2(ek - rt));
                    qfr[gt] = fq;
                } else {
                    const float bt = offt + rt;
                    fac[gt] = make_float2(sc * ex2(bt), ex2(B0 - bt));
                    qfr[gt] = 1.f;
                }
            }
            w = mbar_wait(&bars[QFULL + qs], par(c / NQ));
            if (named_bar_or(1, kGateThreads, !w)) { ok = false; break; }
            // ring entries of chunk c: written only now, after the stage of chunk c arrived
            // (which required the output of c - NQ stored, so pass c - NR has read the slot)
            if (part == 0) {
                *reinterpret_cast<float2 *>(gam_s + slot * 128 + d) = make_float2(ex2(Lc0), ex2(Lc1));
                if (ext)
                    *reinterpret_cast<float2 *>(gam2_s + slot * 128 + d) = make_float2(ex2(B0), ex2(B1));
                *reinterpret_cast<float2 *>(ends_s + d) = make_float2(ex2(L0), ex2(L1));
            }
            if (gt == 0) TRACE_OUT(1, c);
            uint8_t *qt = sm + qs * QSTAGE + Q + boxo;
            uint8_t *kt = sm + qs * QSTAGE + K + boxo;
            if (kPacked && vr < kC) {
                // and their keys become 0: they add nothing to P or to the state
                for (int t = max(vr - tb, 0); t < tl; ++t)
                    *reinterpret_cast<uint32_t *>(kt + sw128_offset((uint32_t)(tb + t), col)) = 0u;
            }
            float r0 = 0.f, r1 = 0.f;
            rs = make_float2(0.f, 0.f);
            // blocks of kGateBlock tokens: all loads of a block are issued before its stores, so a
            // block costs one shared-memory round trip
            if (!ext) {
                // Q' = scale q 2^(b + L), K' = k 2^-(b + L) with b = off + r: the per-chunk
                // constants (offset, L, log2 scale) are folded into two exponent biases. With a
                // scalar gate only k is scaled here (see the epilogue).
                const float2 eq = make_float2(off0 + Lq0 + lsc, off1 + Lq1 + lsc);
                const float2 ek = make_float2(-(off0 + Lq0), -(off1 + Lq1));
                const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll 1
                for (int t0 = 0; t0 < tl; t0 += kGateBlock) {
                    float2 gv[kGateBlock];
                    uint32_t qv[kGateBlock], kv[kGateBlock];
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const uint32_t off = (uint32_t)(tb + t0) * 128u + swz[x];
                        gv[x] = gpair(t0 + x);
                        if (!kScalar) qv[x] = *reinterpret_cast<const uint32_t *>(qt + off);
                        kv[x] = *reinterpret_cast<const uint32_t *>(kt + off);
                    }
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const float2 kf = unpack_bf16(kv[x]);
                        if (kScalar) {
                            // one gate for every key dimension: the token's precomputed factor
                            // (q stays raw: its factor multiplies the output in the epilogue)
                            const float fk = fac[tb + t0 + x].y;
                            kv[x] = pack_bf16(kf.x * fk, kf.y * fk);
                        } else {
                            // the pair's two lanes in packed fp32 instructions (ek - r as the exact
                            // fma(r, -1, ek))
                            rs = fma2(gv[x], l2e, rs);
                            const float2 aq = add2(rs, eq), ak = fma2(rs, neg1, ek);
                            const float2 pq = mul2(unpack_bf16(qv[x]), make_float2(ex2(aq.x), ex2(aq.y)));
                            const float2 pk = mul2(kf, make_float2(ex2(ak.x), ex2(ak.y)));
                            qv[x] = pack_bf16(pq.x, pq.y);
                            kv[x] = pack_bf16(pk.x, pk.y);
                        }
                    }
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const uint32_t off = (uint32_t)(tb + t0) * 128u + swz[x];
                        if (!kScalar) *reinterpret_cast<uint32_t *>(qt + off) = qv[x];
                        *reinterpret_cast<uint32_t *>(kt + off) = kv[x];
                    }
                }
            } else {
                // extreme chunk: K^ = k 2^(Bc - b) with b = off + r formed exactly as the chunk
                // total was, so that the last token's factor is exactly 1
#pragma unroll 1
                for (int t0 = 0; t0 < tl; t0 += kGateBlock) {
                    float2 gv[kGateBlock];
                    uint32_t qv[kGateBlock], kv[kGateBlock];
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const uint32_t off = (uint32_t)(tb + t0) * 128u + swz[x];
                        gv[x] = gpair(t0 + x);
                        qv[x] = *reinterpret_cast<const uint32_t *>(qt + off);
                        kv[x] = *reinterpret_cast<const uint32_t *>(kt + off);
                    }
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const float2 qf = unpack_bf16(qv[x]), kf = unpack_bf16(kv[x]);
                        if (kScalar) {
                            const float2 f = fac[tb + t0 + x];
                            qv[x] = pack_bf16(qf.x * f.x, qf.y * f.x);
                            kv[x] = pack_bf16(kf.x * f.y, kf.y * f.y);
                        } else {
                            r0 = fmaf(gv[x].x, kLog2e, r0);
                            r1 = fmaf(gv[x].y, kLog2e, r1);
                            const float b0 = off0 + r0, b1 = off1 + r1;
                            qv[x] = pack_bf16(sc * qf.x * ex2(b0), sc * qf.y * ex2(b1));
                            kv[x] = pack_bf16(kf.x * ex2(B0 - b0), kf.y * ex2(B1 - b1));
                        }
                    }
#pragma unroll
                    for (int x = 0; x < kGateBlock; ++x) {
                        const uint32_t off = (uint32_t)(tb + t0) * 128u + swz[x];
                        *reinterpret_cast<uint32_t *>(qt + off) = qv[x];
                        *reinterpret_cast<uint32_t *>(kt + off) = kv[x];
                    }
                }
            }
            __syncwarp();
            if (!kScalar && lane == 0) mbar_arrive(&bars[GEMPTY + gs]);   // the g slot may be refilled
            if (gt == 0) xf[slot] = (ext ? 1u : 0u) | (ren ? 2u : 0u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[GDONE + qs]);
            if (gt == 0) TRACE_OUT(2, c);
        }
        __syncwarp();
    }

    if (!ok) atomicOr(a.err, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) TRACE_OUT(15, 0);
    if (threadIdx.x == 0) TRACE_GLOB(0, 2);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// ======================================================================= state kernel
// k/v ring of four stages and a two-slot gate ring (released after the cumsum); the
// suffix-decayed keys K^' overwrite k in place.
namespace sm_ {
constexpr int NKV = 4, NG = 2;
constexpr uint32_t K = 0, V = 16384, KVSTAGE = 32768;
constexpr uint32_t G = NKV * KVSTAGE, GSLOT = 32768;
constexpr uint32_t BV = G + NG * GSLOT;  // [128] f32 chunk totals
constexpr uint32_t XCH = BV + 512;       // [4][128] f32
constexpr uint32_t GSC = XCH + 2048;     // [2][64] f32 scalar gates of two chunks (scalar mode)
constexpr uint32_t BAR = GSC + 512;
constexpr uint32_t NBAR = 17;
constexpr uint32_t TSLOT = BAR + NBAR * 8;
constexpr uint32_t ALLOC = TSLOT + 16 + 1024;
}  // namespace sm_

// The gate-done ring has as many slots as the k/v ring: gate(c + NKV) needs the k/v stage
// that U(c) releases, so the MMA thread has always observed gate-done(c) before its slot
// is reused (no phase can be lapped).
enum { SKFULL = 0, SKEMPTY = 4, SGFULL = 8, SGEMPTY = 10, SGDONE = 12, SEDONE = 16 };
static_assert(SGDONE + sm_::NKV <= SEDONE, "state-kernel barrier map");

template <bool kScalar>
__global__ void __launch_bounds__(kStateThreads, 1)
gla_tc_state_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tg, const StateArgs a) {
    using namespace sm_;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TSLOT);
    float *bv_s = reinterpret_cast<float *>(sm + BV);
    float *xch = reinterpret_cast<float *>(sm + XCH);
    pdl_launch_dependents();   // the scan kernel may be scheduled now; it waits for us
    if (threadIdx.x == 0) TRACE_GLOB(1, 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA = piece `sub` of segment `seg` of head `bh`: E and Gamma of that piece
    const int npc = (a.splits - 1) * a.pieces;   // pieces per head
    const int pi = blockIdx.x % npc;
    const int bh = blockIdx.x / npc;
    const int seg = pi / a.pieces, sub = pi % a.pieces;
    const int bidx = bh / a.H, h = bh % a.H;
    int cb, ce;
    seg_range(seg, a.nchunks, a.splits, a.last16, cb, ce);
    {
        const int len = ce - cb;
        const int c0 = cb + (int)((int64_t)sub * len / a.pieces);
        ce = cb + (int)((int64_t)(sub + 1) * len / a.pieces);
        cb = c0;
    }
    const int n = ce - cb;
    constexpr int NGD = NKV;   // gate-done ring

    if (threadIdx.x == 0) {
        for (int i = 0; i < NKV; ++i) {
            mbar_init(&bars[SKFULL + i], 1);
            mbar_init(&bars[SKEMPTY + i], 1);
        }
        for (int i = 0; i < NG; ++i) {
            mbar_init(&bars[SGFULL + i], 1);
            mbar_init(&bars[SGEMPTY + i], 1);
        }
        for (int i = 0; i < NGD; ++i) mbar_init(&bars[SGDONE + i], 8);
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
            // The chunks this CTA reads last (the first ones of its segment) are the ones the
            // output kernel reads first: keep them in L2 ahead of the rest.
            const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
            int ng = kScalar ? n : 0, nk = 0;   // scalar gates are not staged by TMA
            uint32_t idle = 0;
            uint64_t t_idle = 0;
            while (ng < n || nk < n) {
                bool prog = false;
                if (ng < n && (ng < NG || mbar_test(&bars[SGEMPTY + ng % NG], par(ng / NG - 1)))) {
                    uint64_t *fb = &bars[SGFULL + ng % NG];
                    TRACE_ST(0, ng);
                    mbar_arrive_expect_tx(fb, 32768);
                    tma_load_4d_hint(sm + G + (ng % NG) * GSLOT, &tg, fb, 0, h, (ce - 1 - ng) * kC,
                                     bidx, ng >= n - a.retain ? keep : drop);
                    ++ng;
                    prog = true;
                }
                if (nk < n && (nk < NKV || mbar_test(&bars[SKEMPTY + nk % NKV], par(nk / NKV - 1)))) {
                    uint8_t *base = sm + (nk % NKV) * KVSTAGE;
                    uint64_t *fb = &bars[SKFULL + nk % NKV];
                    mbar_arrive_expect_tx(fb, 2 * 16384);
                    const int t = (ce - 1 - nk) * kC;      // last chunk first
                    const uint64_t pol = nk >= n - a.retain ? keep : drop;
                    tma_load_4d_hint(base + K, &tk, fb, 0, h, t, bidx, pol);
                    tma_load_4d_hint(base + K + 8192, &tk, fb, 64, h, t, bidx, pol);
                    tma_load_4d_hint(base + V, &tv, fb, 0, h, t, bidx, pol);
                    tma_load_4d_hint(base + V + 8192, &tv, fb, 64, h, t, bidx, pol);
                    ++nk;
                    prog = true;
                }
                if (prog) {
                    idle = 0;
                } else {
                    // yield the issue slots of this sub-partition to the compute warps
                    __nanosleep(kIssuerNapNs);
                    if (++idle == 256) {
                        t_idle = global_ns();   // the timer is read only on long idle streaks
                    } else if ((idle & 1023) == 0 && global_ns() - t_idle > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            for (int i = 0; i < NG && !kScalar; ++i) {
                const int uses = ng > i ? (ng - 1 - i) / NG + 1 : 0;
                if (uses > 0 && !mbar_wait(&bars[SGFULL + i], par(uses - 1))) ok = false;
            }
            for (int i = 0; i < NKV; ++i) {
                const int uses = nk > i ? (nk - 1 - i) / NKV + 1 : 0;
                if (uses > 0 && !mbar_wait(&bars[SKFULL + i], par(uses - 1))) ok = false;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idU = idesc_bf16(128, 128, 1, 1);
            for (int c = 0; c < n; ++c) {
                if (!mbar_wait(&bars[SGDONE + c % NGD], par(c / NGD))) { ok = false; break; }
                tc_fence_after();
                const uint32_t base = smem_u32(sm + (c % NKV) * KVSTAGE);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tm, smem_desc(base + V + kk * 2048, 8192, 1024),
                           smem_desc(base + K + kk * 2048, 8192, 1024), idU,
                           (c > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars[SKEMPTY + c % NKV]);
                TRACE_ST(3, c);
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
        float l0 = 0.f, l1 = 0.f;   // log2 decay from this chunk's end to the segment end
        // scalar gates: thread gt < 64 fetches token gt of the next chunk (chunks run last to
        // first) and publishes it in gsc[c & 1] at the top of each chunk
        float *gsc = reinterpret_cast<float *>(sm + GSC);
        auto fetch_scalar = [&](int c) -> float {
            const int64_t t = (int64_t)(ce - 1 - c) * kC + gt;
            return t < a.T ? __ldg(a.g + ((int64_t)bidx * a.T + t) * a.H + h) : 0.f;
        };
        float gpre = (kScalar && gt < kC && n > 0) ? fetch_scalar(0) : 0.f;
        for (int c = 0; c < n; ++c) {
            if (kScalar) {
                if (gt < kC) {
                    gsc[(c & 1) * kC + gt] = gpre;
                    if (c + 1 < n) gpre = fetch_scalar(c + 1);
                }
                named_bar_sync(1, 256);
            } else {
                bool w = mbar_wait(&bars[SGFULL + c % NG], par(c / NG));
                if (named_bar_or(1, 256, !w)) { ok = false; break; }
            }
            if (gt == 0) TRACE_ST(1, c);
            float b0[16], b1[16];
            if (kScalar)
                gate_cumsum_scalar(gsc + (c & 1) * kC, xch, qq, d, b0, b1, 1);
            else
                gate_cumsum(reinterpret_cast<const float *>(sm + G + (c % NG) * GSLOT), xch, qq, d,
                            b0, b1, 1);
            if (!kScalar && gt == 0) mbar_arrive(&bars[SGEMPTY + c % NG]);
            if (qq == 3) {
                bv_s[d] = b0[15];
                bv_s[d + 1] = b1[15];
            }
            const bool w = mbar_wait(&bars[SKFULL + c % NKV], par(c / NKV));
            if (named_bar_or(1, 256, !w)) { ok = false; break; }   // also publishes bv_s
            const float s0 = bv_s[d] + l0, s1 = bv_s[d + 1] + l1;
            uint8_t *kt = sm + (c % NKV) * KVSTAGE + K + boxo;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const uint32_t off = sw128_offset(16 * qq + x, col);
                const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(kt + off));
                if (kScalar) {   // one gate for every key dimension: one factor per token
                    const float f = ex2(s0 - b0[x]);
                    *reinterpret_cast<uint32_t *>(kt + off) = pack_bf16(kv.x * f, kv.y * f);
                } else {
                    *reinterpret_cast<uint32_t *>(kt + off) =
                        pack_bf16(kv.x * ex2(s0 - b0[x]), kv.y * ex2(s1 - b1[x]));
                }
            }
            l0 = s0;
            l1 = s1;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[SGDONE + c % NGD]);
            if (gt == 0) TRACE_ST(2, c);
        }
        if (ok && qq == 0) {
            float *gp = a.gam + ((size_t)bh * npc + pi) * kD;
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
                float *ep = a.E + ((size_t)bh * npc + pi) * (kD * kD) + v;
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
    if (threadIdx.x == 0) TRACE_GLOB(1, 2);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 128);
    }
}

// ======================================================================= scan kernel
// S_start(s+1) = fold over the pieces of segment s of (Gamma (.) S + E), rows scaled by
// Gamma[d]; S_start(0) = h0. Each thread carries kScanPer state elements (d, v) of one head,
// 256 apart; the loads of a batch of pieces are issued together so the chain costs one
// memory round trip per batch, not per piece. The grid stays small (B*H x 16 CTAs) so that
// all of it can be resident while it waits for the state kernel.
constexpr int kScanThreads = 256;
constexpr int kScanPer = 4;
constexpr int kScanBatch = 4;

__global__ void __launch_bounds__(kScanThreads)
gla_tc_scan_kernel(const float *__restrict__ E, const float *__restrict__ gam,
                   const float *__restrict__ h0, float *__restrict__ sstart, int splits,
                   int pieces, int Dk, int Dv, int paired) {
    pdl_launch_dependents();    // the output kernel may be scheduled now; it waits for us
    if (threadIdx.x == 0 && blockIdx.y == 0) TRACE_GLOB(2, 0);
    pdl_wait_prerequisites();   // the end states of the state kernel
    if (threadIdx.x == 0 && blockIdx.y == 0) TRACE_GLOB(2, 1);
    const size_t bh = blockIdx.x;
    const int e0 = blockIdx.y * (kScanThreads * kScanPer) + threadIdx.x;   // d * kD + v
    const int nseg = splits - 1;
    const int npc = nseg * pieces;
    constexpr size_t kDD = (size_t)kD * kD;
    float s[kScanPer];
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
        const int e = e0 + i * kScanThreads, d = e / kD, v = e % kD;   // h0 is Dk x Dv
        if (paired)   // head pairs: the diagonal blocks are heads 2 bh and 2 bh + 1 (64 x 64)
            s[i] = (h0 && (d >> 6) == (v >> 6))
                       ? h0[(bh * 2 + (v >> 6)) * 4096 + (size_t)(d & 63) * 64 + (v & 63)] : 0.f;
        else
            s[i] = (h0 && d < Dk && v < Dv) ? h0[bh * (size_t)Dk * Dv + (size_t)d * Dv + v] : 0.f;
    }
    const float *Eb = E + bh * npc * kDD + e0;
    const float *gb = gam + bh * npc * kD;
    float *ob = sstart + bh * nseg * kDD + e0;
    for (int r0 = 0; r0 < npc; r0 += kScanBatch) {
        float ev[kScanBatch][kScanPer], gv[kScanBatch][kScanPer];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (r0 + j < npc) {
#pragma unroll
                for (int i = 0; i < kScanPer; ++i) {
                    const int e = e0 + i * kScanThreads;
                    ev[j][i] = Eb[(size_t)(r0 + j) * kDD + i * kScanThreads];
                    gv[j][i] = gb[(size_t)(r0 + j) * kD + e / kD];
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (r0 + j < npc) {
                const bool seg_end = (r0 + j + 1) % pieces == 0;
                const size_t os = (size_t)((r0 + j + 1) / pieces - 1) * kDD;
#pragma unroll
                for (int i = 0; i < kScanPer; ++i) {
                    s[i] = gv[j][i] * s[i] + ev[j][i];
                    if (seg_end) ob[os + i * kScanThreads] = s[i];
                }
            }
        }
    }
}

// Opt-in shared-memory sizes are a per-device setting of each kernel: set once per device,
// under a lock (several host threads may make their first call at the same time).
constexpr int kMaxDevices = 64;
std::mutex g_attr_mu;
bool g_attr_done[kMaxDevices];

cudaError_t set_attrs() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (g_attr_done[dev]) return cudaSuccess;
    const void *outs[5] = {(const void *)gla_tc_out_kernel<false, false>,
                           (const void *)gla_tc_out_kernel<true, false>,
                           (const void *)gla_tc_out_kernel<false, true>,
                           (const void *)gla_tc_out_kernel<true, true>,
                           (const void *)gla_tc_out_kernel<false, false, true>};
    const void *states[2] = {(const void *)gla_tc_state_kernel<false>,
                             (const void *)gla_tc_state_kernel<true>};
    for (int i = 0; i < 5; ++i) {
        e = cudaFuncSetAttribute(outs[i], cudaFuncAttributeMaxDynamicSharedMemorySize, om::ALLOC);
        if (e != cudaSuccess) return e;
        if (i < 2) {
            e = cudaFuncSetAttribute(states[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     sm_::ALLOC);
            if (e != cudaSuccess) return e;
        }
    }
    g_attr_done[dev] = true;
    return cudaSuccess;
}

// Test hook of the bounded waits. The environment is read once per process: with
// GLA_TEST_STALL_ONE_LOAD set, the first tensor-core launch of the process skips the q/k/v
// load of one chunk in every output CTA (later launches run normally), so its waits run out
// and the call reports GLA_ERR_DEVICE_TIMEOUT with the context intact.
std::atomic<int> g_stall_left{-1};   // -1: environment not read yet

bool take_stall_hook() {
    int left = g_stall_left.load(std::memory_order_relaxed);
    if (left < 0) {
        int init = std::getenv("GLA_TEST_STALL_ONE_LOAD") ? 1 : 0, expect = -1;
        g_stall_left.compare_exchange_strong(expect, init);
        left = g_stall_left.load(std::memory_order_relaxed);
    }
    while (left > 0) {
        if (g_stall_left.compare_exchange_weak(left, left - 1)) return true;
    }
    return false;
}

int clamp_splits(const Problem &p, int splits) {
    const int64_t nchunks = (p.T + kC - 1) / kC;
    int64_t s = std::max<int64_t>(1, std::min<int64_t>(splits, nchunks));
    return (int)std::min<int64_t>(s, kMaxSplits);
}

// Head pairs: bf16 I/O, per-key gates, head dims 64 x 64, an even number of heads and no
// packed sequences run as H / 2 heads of dims 128 (gla_tc_out_kernel<.., kPair>).
bool pair_heads(const Problem &p) {
    return p.io == 0 && p.Dk == 64 && p.Dv == 64 && p.H % 2 == 0 && p.gate != 1 && !p.cu;
}

// The problem as the tensor-core kernels see it.
Problem tc_view(const Problem &p) {
    if (!pair_heads(p)) return p;
    Problem q = p;
    q.H = p.H / 2;
    q.Dk = q.Dv = kD;
    return q;
}

}  // namespace

bool tc_supported(const Problem &p) {
    // head dims 64 run on the 128-wide kernels: the tensor copies read zeros past the
    // caller's last dimension, and zero keys and gates add nothing and decay nothing
    const auto dim_ok = [](int64_t d) { return d == kD || d == 64; };
    return p.io == 0 && dim_ok(p.Dk) && dim_ok(p.Dv) && p.T < (int64_t(1) << 30) &&
           p.B * p.H < (int64_t(1) << 24);
}

int tc_auto_splits(const Problem &pc, int num_sms) {
    const Problem p = tc_view(pc);
    const int64_t nchunks = (p.T + kC - 1) / kC;
    const int64_t bh = p.B * p.H;
    if (nchunks <= 1 || bh <= 0) return 1;
    // The output pass runs one CTA per SM; a second wave of CTAs costs a whole extra
    // segment of latency-bound chunks. So: the most segments per head that still fit in
    // one wave of output CTAs (which also keeps the state pass to one wave).
    int64_t s = std::max<int64_t>(1, num_sms / bh);
    s = std::min<int64_t>(s, nchunks);
    return (int)std::min<int64_t>(s, kMaxSplits);
}

int tc_state_pieces(const Problem &pc, int splits, int num_sms) {
    const Problem p = tc_view(pc);
    const int s = clamp_splits(p, splits);
    if (s <= 1) return 1;
    // Split each segment's state pass into consecutive pieces until its grid, like the output
    // pass, fills the GPU in one wave; every piece keeps at least four chunks.
    const int64_t bh = p.B * p.H;
    const int64_t nchunks = (p.T + kC - 1) / kC;
    int64_t k = num_sms / (bh * (s - 1));
    k = std::min<int64_t>(k, nchunks / (4 * (int64_t)s));
    return (int)std::max<int64_t>(1, std::min<int64_t>(k, kMaxPieces));
}

size_t tc_workspace_bytes(const Problem &pc, int splits, int num_sms) {
    const Problem p = tc_view(pc);
    const int s = clamp_splits(p, splits);
    if (s <= 1) return 0;
    const size_t bh = (size_t)(p.B * p.H);
    const size_t k = (size_t)tc_state_pieces(p, splits, num_sms);
    // E and Gamma of every piece, and the start state of every segment but the first
    return bh * (size_t)(s - 1) * (k * ((size_t)kD * kD + kD) + (size_t)kD * kD) * sizeof(float);
}

cudaError_t launch_tc(const Problem &pc, int splits, int num_sms, void *ws, size_t ws_bytes,
                      unsigned int *dev_err, cudaStream_t stream) {
    // Fewer tokens than one chunk (for packed sequences: in all of them together): the exact
    // kernel (each output is a handful of products of bf16-rounded decayed operands here,
    // with nothing to average their rounding). T = 0 only writes hT = h0.
    if (pc.T < kC) return launch_exact(pc, dev_err, stream);
    const bool paired = pair_heads(pc);
    const Problem p = tc_view(pc);
    const int s = p.cu ? 1 : clamp_splits(p, splits);   // packed sequences are not split
    const int64_t mB = p.cu ? 1 : p.B;                   // batch extent of the tensor maps
    const bool scalar = p.gate == 1;
    cudaError_t e = set_attrs();
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mg;
    if (!make_bthd_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, mB, p.T, p.H, p.Dk, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, mB, p.T, p.H, p.Dk, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_bthd_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, mB, p.T, p.H, p.Dv, 64, kC,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        // per-key gates are staged by TMA; scalar gates are read directly (the map is unused)
        !(scalar ? make_bthd_map(&mg, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, mB, p.T, p.H,
                                 p.Dk, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B)
                 : make_bthd_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, mB, p.T, p.H,
                                 p.Dk, kD, kC, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return cudaErrorInvalidResourceHandle;   // a tensor map could not be encoded
    const int nchunks = (int)((p.T + kC - 1) / kC);
    const int bh = (int)(p.B * p.H);
    float *E = nullptr, *gam = nullptr, *sstart = nullptr;
    const int pieces = tc_state_pieces(p, s, num_sms);
    // State-pass reads kept in L2 for the output pass, as a fraction of all of them; the last
    // segment (which gets none) is shortened by 15 % of that fraction.
    const int64_t per_chunk = 2 * 16384 + (scalar ? 0 : 32768);   // k, v, g bytes of a chunk
    const int64_t state_bytes = (int64_t)bh * (s - 1) * ((nchunks + s - 1) / s) * per_chunk;
    const double kept = s > 1 ? std::min(1.0, (double)kL2KeepBytes / (double)state_bytes) : 0.0;
    const int last16 = 16 - (int)(16.0 * 0.15 * kept + 0.5);
    if (s > 1) {
        if (!ws || ws_bytes < tc_workspace_bytes(p, s, num_sms)) return cudaErrorInvalidValue;
        E = static_cast<float *>(ws);
        gam = E + (size_t)bh * (s - 1) * pieces * kD * kD;
        sstart = gam + (size_t)bh * (s - 1) * pieces * kD;
        // keep about kL2KeepBytes of the state pass's last reads for the output kernel
        const int retain = (int)std::min<int64_t>(
            ((nchunks + s - 1) / s + pieces - 1) / pieces,
            kL2KeepBytes / ((int64_t)bh * (s - 1) * pieces * per_chunk));
        StateArgs sa{E, gam, p.T, (int)p.H, nchunks, s, dev_err, retain, last16, pieces, p.g};
        if (scalar)
            gla_tc_state_kernel<true><<<bh * (s - 1) * pieces, kStateThreads, sm_::ALLOC, stream>>>(
                mk, mv, mg, sa);
        else
            gla_tc_state_kernel<false><<<bh * (s - 1) * pieces, kStateThreads, sm_::ALLOC, stream>>>(
                mk, mv, mg, sa);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // scan and output kernels are programmatic dependents: each may be scheduled while its
        // predecessor (one of ours) still runs, and waits for it in griddepcontrol.wait
        // before reading what it wrote. The state kernel itself launches normally, so every
        // kernel of this call starts after the caller's preceding work has completed.
        cudaLaunchAttribute pdl[1];
        pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(bh, kD * kD / (kScanThreads * kScanPer));
        cfg.blockDim = dim3(kScanThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gla_tc_scan_kernel, (const float *)E, (const float *)gam,
                               p.h0, sstart, s, pieces, (int)p.Dk, (int)p.Dv, paired ? 1 : 0);
        if (e != cudaSuccess) return e;
        count_launches(2);
    }
    // test hook of the bounded waits (see take_stall_hook): one chunk's load is never issued
    const int stall = (!p.cu && take_stall_hook()) ? std::min(1, nchunks / s - 1) : -1;
    OutArgs oa{static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
               p.g, p.h0, p.hT, sstart, p.T, (int)p.H, nchunks, s, p.scale, dev_err, stall,
               last16, p.cu, static_cast<__nv_bfloat16 *>(p.o), (int)p.Dk, (int)p.Dv,
               p.cu ? 1 : 0};
    if (s > 1) {
        cudaLaunchAttribute pdl[1];
        pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(bh * s);
        cfg.blockDim = dim3(kOutThreads);
        cfg.dynamicSmemBytes = om::ALLOC;
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        e = scalar   ? cudaLaunchKernelEx(&cfg, gla_tc_out_kernel<true, false>, mq, mk, mv, mg, oa)
            : paired ? cudaLaunchKernelEx(&cfg, gla_tc_out_kernel<false, false, true>, mq, mk, mv,
                                          mg, oa)
                     : cudaLaunchKernelEx(&cfg, gla_tc_out_kernel<false, false>, mq, mk, mv, mg, oa);
    } else {
        auto kern = p.cu ? (scalar ? gla_tc_out_kernel<true, true> : gla_tc_out_kernel<false, true>)
                    : scalar ? gla_tc_out_kernel<true, false>
                    : paired ? gla_tc_out_kernel<false, false, true>
                             : gla_tc_out_kernel<false, false>;
        kern<<<bh * s, kOutThreads, om::ALLOC, stream>>>(mq, mk, mv, mg, oa);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    count_launches(1);
    if (p.cu) {
        // packed sequences shorter than one chunk: the exact kernel, on the same stream
        Problem ps = p;
        ps.seq_filter = kShortOnly;
        return launch_exact(ps, dev_err, stream);
    }
    return cudaSuccess;
}

}  // namespace gla
