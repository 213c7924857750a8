/*
 * gla.h — C ABI of libgla.so, the GB300 (sm_103a) gated-linear-attention prefill forward
 * (and the gated delta rule forward, gdn_fwd, declared at the end).
 *
 * What every entry point computes, per batch b and head h independently
 * ("Linear Attention 在 GPU 上到底慢在哪", section 学长的反馈: the state update
 * h <- h.g + k^T v with a D x D state; "线性注意力GPU算子库的定义与技术解析",
 * section 四: the state is updated with token t before o[t] is read):
 *
 *     S_0 = h0 (zero when h0 == NULL)
 *     S_t = diag(exp(g_t)) . S_{t-1} + k_t^T v_t          t = 0 .. T-1
 *     o_t = scale . q_t . S_t
 *     hT  = S_T                                            (written when hT != NULL)
 *
 * g_t is the log-gate (a Dk vector per token and head; expected <= 0, any finite value
 * is accepted and computed as given). The GPU evaluates this in the chunkwise form of
 * "线性注意力GPU算子库的定义与技术解析", section 四 (chunks of 64 tokens, in-chunk
 * cumulative log-gate, decay-masked in-chunk attention, a state scan across chunks,
 * matrix products for the in-chunk work). The result equals the recurrence up to
 * floating-point rounding.
 *
 * Layouts (all contiguous, row-major, element strides implied by the shape):
 *     q, k, g_log : [B, T, H, Dk]
 *     v, o        : [B, T, H, Dv]
 *     h0, hT      : [B, H, Dk, Dv]   float32
 * Supported head dims: Dk, Dv in {64, 128} on both paths. The tensor-core kernels work at
 * 128: with Dk = Dv = 64, an even H, per-key gates and no packed sequences, heads 2p and
 * 2p + 1 (adjacent, so one contiguous row of 128) run together as one head of 128 with a
 * block-diagonal state; any other head dim of 64 is padded with zeros. Results are the same
 * either way, within the stated tolerances. Any T >= 0 (a partial last chunk is handled).
 *
 * Ownership and memory: every tensor pointer is a DEVICE pointer owned by the caller
 * and must be 16-byte aligned. o and hT must not overlap any input. The library never
 * frees caller memory.
 *
 * Execution: every call is asynchronous and ordered on `stream` (NULL = the legacy
 * default stream). No call synchronises the host, except gla_last_device_status().
 * Calls may be captured into a CUDA graph (stream capture) once their scratch exists: pass a
 * caller workspace, or make one call on the capturing stream first (the library's own
 * workspace is allocated with cudaMalloc, which cannot happen during capture). A replay
 * reads whatever the captured buffers then hold.
 *
 * Errors: every entry point returns a gla_status and never aborts, traps or throws.
 * Argument errors are detected on the host before any launch; nothing is written then.
 */
#ifndef GLA_H_
#define GLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream, so either may be passed. */
typedef struct CUstream_st *gla_stream_t;

typedef enum {
    GLA_OK = 0,
    GLA_ERR_NULL_ARG = 1,          /* a required pointer is NULL                      */
    GLA_ERR_BAD_SHAPE = 2,         /* negative or overflowing B, T, H                 */
    GLA_ERR_UNSUPPORTED_DIM = 3,   /* Dk / Dv not supported by the requested path     */
    GLA_ERR_MISALIGNED = 4,        /* a pointer is not 16-byte aligned                */
    GLA_ERR_ALIAS = 5,             /* an output overlaps an input                     */
    GLA_ERR_LAUNCH = 6,            /* a CUDA call or kernel launch failed             */
    GLA_ERR_DEVICE_TIMEOUT = 7,    /* a kernel gave up waiting on a pipeline barrier  */
    GLA_ERR_UNSUPPORTED_DEVICE = 8,/* the current device is not sm_103                */
    GLA_ERR_WORKSPACE = 9,         /* caller workspace too small or misaligned        */
    GLA_ERR_BAD_OPTION = 10,       /* an option value is out of range                 */
    GLA_ERR_BAD_SEQLENS = 11       /* packed-sequence offsets were found inconsistent on
                                      the device (reported by gla_last_device_status)   */
} gla_status;

/* Which arithmetic path runs. */
typedef enum {
    GLA_PATH_AUTO = 0,   /* tensor-core path for bf16 I/O, exact path for fp32 I/O    */
    GLA_PATH_EXACT = 1,  /* fp32 CUDA-core chunkwise kernel (exact in-chunk decays)   */
    GLA_PATH_TC = 2      /* tcgen05 / TMEM / TMA kernel, bf16 operands, fp32 state     */
} gla_path;

typedef enum { GLA_IO_BF16 = 0, GLA_IO_F32 = 1 } gla_io;

/* Shape of the log-gate. GLA_GATE_KEY: g_log [B, T, H, Dk], one gate per key dimension (the
 * default, and what gla_fwd / gla_fwd_f32 take). GLA_GATE_SCALAR: g_log [B, T, H], one gate
 * per token and head applied to every key row, S_t = exp(g_t) S_{t-1} + k_t^T v_t (the
 * scalar-decay (SSD-style) variant, "Linear Attention 在 GPU 上到底慢在哪", section
 * 正确的 baseline 和下一步). */
typedef enum { GLA_GATE_KEY = 0, GLA_GATE_SCALAR = 1 } gla_gate;

typedef struct {
    int path;               /* gla_path                                                */
    int seq_splits;         /* tensor-core path: sequence segments per head; 0 = auto  */
    void *workspace;        /* device scratch owned by the caller, or NULL. With NULL the
                               library keeps one buffer per stream and device: allocated
                               by the first call on that stream that needs scratch,
                               replaced (cudaFree, which synchronises the device, then
                               cudaMalloc) only when a call needs more than that stream's
                               buffer holds; repeated calls of the same shape allocate
                               nothing. Calls on different streams never share it. A
                               caller buffer is the caller's to order: two calls whose
                               kernels overlap on the GPU must not be given the same one. */
    size_t workspace_bytes; /* size of `workspace` in bytes                            */
    int gate;               /* gla_gate (0 = GLA_GATE_KEY)                             */
} gla_options;

/*
 * gla_fwd — bf16 q, k, v, o; fp32 g_log, h0, hT; fp32 state and accumulation.
 * Arguments: q, k, v, g_log (inputs), scale (output multiplier, typically Dk^-0.5),
 * h0 (initial state or NULL), o (output), hT (final state or NULL), shape B, T, H, Dk,
 * Dv, and the stream. Runs the tensor-core path (T < 64 runs the exact kernel instead).
 * Scratch: when the sequence is split across CTAs the call uses the library's workspace
 * of `stream` (see gla_options.workspace): concurrent calls on different streams are safe;
 * the first call on a stream (or the first needing a larger workspace) allocates, so make it
 * before any stream capture begins.
 */
gla_status gla_fwd(const void *q, const void *k, const void *v, const float *g_log,
                   float scale, const float *h0, void *o, float *hT,
                   int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv,
                   gla_stream_t stream);

/* gla_fwd_f32 — same contract with fp32 q, k, v, o; runs the exact CUDA-core path. */
gla_status gla_fwd_f32(const float *q, const float *k, const float *v, const float *g_log,
                       float scale, const float *h0, float *o, float *hT,
                       int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv,
                       gla_stream_t stream);

/*
 * gla_fwd_ex — the general entry: io selects bf16 or fp32 q/k/v/o, opt (may be NULL)
 * selects the path, the sequence split, the workspace and the gate shape. The tensor-core
 * path needs bf16 I/O and Dk, Dv in {64, 128}; with fewer than 64 tokens it runs the exact
 * kernel (whose results it then returns), since a handful of bf16-rounded products is all
 * each output would be. Scratch as gla_fwd: opt->workspace, else the stream's own library
 * workspace.
 */
gla_status gla_fwd_ex(const void *q, const void *k, const void *v, const float *g_log,
                      float scale, const float *h0, void *o, float *hT,
                      int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv,
                      int io, const gla_options *opt, gla_stream_t stream);

/*
 * gla_step — one decode step on a resident state: the token update of the recurrence above,
 * applied once (update first, then the read), for every batch and head:
 *     S <- diag(exp(g_log)) . S + k^T v,    o = scale . q . S
 * It continues a prefill: pass the hT that gla_fwd wrote as S ("Linear Attention 在 GPU 上到底
 * 慢在哪", section 学长的反馈, names decoding as the step that follows the prefill).
 * Layouts (one token, contiguous): q, k, g_log [B, H, Dk]; v, o [B, H, Dv]; S [B, H, Dk, Dv]
 * fp32, read and overwritten in place. io = GLA_IO_BF16 (bf16 q, k, v, o) or GLA_IO_F32;
 * g_log and S are fp32 either way. 1 <= Dk <= 1024; 4 <= Dv <= 1024 with Dv a multiple of 4
 * (GLA_ERR_UNSUPPORTED_DIM otherwise). Device pointers, 16-byte aligned; o
 * and S must not overlap each other or any input. fp32 arithmetic; deterministic.
 */
gla_status gla_step(const void *q, const void *k, const void *v, const float *g_log, float scale,
                    float *S, void *o, int64_t B, int64_t H, int64_t Dk, int64_t Dv, int io,
                    gla_stream_t stream);

/*
 * gla_fwd_varlen — gla_fwd_ex over N sequences of different lengths packed along one token
 * axis (a T-ragged batch). Sequence i is tokens cu_seqlens[i] .. cu_seqlens[i+1]-1; each
 * runs the recurrence independently from h0[i] (or zero) and writes hT[i].
 * Layouts: q, k, g_log [T, H, Dk] (g_log [T, H] with GLA_GATE_SCALAR); v, o [T, H, Dv];
 * h0, hT [N, H, Dk, Dv] fp32; cu_seqlens: DEVICE int32 [N + 1], non-decreasing, cu_seqlens[0]
 * = 0 and cu_seqlens[N] = T. The offsets are read on the device only: violations are
 * reported by gla_last_device_status as GLA_ERR_BAD_SEQLENS. Sequences are not split
 * (opt->seq_splits is ignored): the tensor-core path runs one CTA per sequence and head for
 * every sequence of at least 64 tokens, and a second launch of the exact kernel on the same
 * stream computes the shorter ones.
 * Other arguments, options and errors as gla_fwd_ex. This serves the batch-efficiency concern
 * of "面向长序列大模型的线性注意力算子性能评测方法与优化实践", section 四、评测维度设计 (no
 * padding to the longest sequence of a batch); the pages define no varlen interface.
 */
gla_status gla_fwd_varlen(const void *q, const void *k, const void *v, const float *g_log,
                          float scale, const float *h0, void *o, float *hT,
                          const int32_t *cu_seqlens, int64_t N, int64_t T, int64_t H,
                          int64_t Dk, int64_t Dv, int io, const gla_options *opt,
                          gla_stream_t stream);

/* Bytes of device workspace gla_fwd_ex needs for this shape and options (0 if none).
 * Returns 0 as well for arguments it would reject. */
size_t gla_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv,
                              int io, const gla_options *opt);

/* The path gla_fwd_ex would run for this shape, io and options: GLA_PATH_EXACT or
 * GLA_PATH_TC, or -1 when it would reject them. Makes no CUDA call. */
int gla_path_for(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                 const gla_options *opt);

/*
 * gla_last_device_status — synchronises `stream`, then reads and clears the library's
 * device error word on the current device. Returns GLA_OK, GLA_ERR_DEVICE_TIMEOUT when
 * a kernel abandoned a bounded pipeline wait (its outputs are then undefined, the
 * context stays usable), GLA_ERR_BAD_SEQLENS when gla_fwd_varlen found offsets that are
 * not non-decreasing within [0, T] (the affected sequences are left unwritten), or
 * GLA_ERR_LAUNCH when the synchronisation itself failed.
 */
gla_status gla_last_device_status(gla_stream_t stream);

/* Text of the last CUDA error behind a GLA_ERR_LAUNCH / GLA_ERR_WORKSPACE returned to
 * this host thread ("" if none). Thread-local static storage; never NULL. */
const char *gla_last_error_detail(void);

/* Human-readable name of a status (static storage; never NULL). */
const char *gla_status_string(gla_status s);

/* Number of kernel launches this library has issued in this process (all devices),
 * counted on the host at each successful launch. Lets a caller verify how many of
 * the library's kernels ran inside a timed region. */
uint64_t gla_launch_counter(void);

/* Number of device allocations (cudaMalloc) the library has made for its own per-stream
 * workspaces in this process (all devices). A caller can check that its steady-state calls
 * allocate nothing. */
uint64_t gla_workspace_allocations(void);

/* Size in bytes of the fixed scratch array behind gla_fwd_noalloc (16 MiB). */
#define GLA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * gla_fwd_noalloc — gla_fwd (bf16 q, k, v, o; same arguments, same path choice, same
 * results) that never allocates device memory. The method itself has no counterpart to
 * this entry point; it serves callers that cannot call cudaMalloc: a host that has handed
 * all device memory to its own pool or arena and must account for every byte, and code
 * on a latency-critical path where the library's own workspace growth (cudaFree followed
 * by cudaMalloc, which synchronises the whole device) would stall other streams.
 *
 * Scratch: the tensor-core path's sequence split needs the bytes gla_fwd_workspace_size()
 * reports for the same shape and seq_splits (about B*H*(splits-1)*128 KiB, more where the
 * state pass is cut into pieces). This entry point takes it from one array of
 * GLA_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that runs this entry
 * point holds until the process exits. seq_splits = 0 picks the split gla_fwd would pick,
 * lowered to the largest count whose scratch fits; seq_splits > 0 whose scratch does not fit
 * returns GLA_ERR_WORKSPACE (gla_last_error_detail() gives the bytes needed) before anything
 * is launched. seq_splits < 0 returns GLA_ERR_BAD_OPTION.
 *
 * Set-up: the first call on a device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress and caches it; make that first call before
 * any stream capture begins. A failed lookup returns GLA_ERR_LAUNCH.
 *
 * Sharing: every call on a device uses the same array. Nothing in it needs to start at
 * zero (a call writes every scratch element before reading it), but calls whose kernels
 * overlap on the GPU (different streams, or several host threads without ordering) race
 * on it and give wrong results; order them on one stream or serialise them.
 * Errors otherwise as gla_fwd_ex.
 */
gla_status gla_fwd_noalloc(const void *q, const void *k, const void *v, const float *g_log,
                           float scale, const float *h0, void *o, float *hT,
                           int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv,
                           int seq_splits, gla_stream_t stream);

/*
 * gdn_fwd — forward (prefill) pass of the gated delta rule, the gated-delta-network kind of
 * linear attention the operator libraries on the pages target ("面向长序列大模型的线性注意力
 * 算子性能评测方法与优化实践", section 三.3: a gate and an incremental update of the recurrent
 * state; "线性注意力GPU算子库的定义与技术解析", section 三). The pages print no formula; this is
 * the published gated delta rule, per batch b and head h:
 *     S_0 = h0 (or 0)
 *     S_t = exp(g_t) (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t      (Dk x Dv, fp32)
 *     o_t = scale . q_t . S_t,     hT = S_T
 * with one log-gate g_t and one write strength beta_t per token and head (k_t a row vector).
 * Layouts (contiguous, row-major): q, k [B, T, H, Dk]; v, o [B, T, H, Dv] in bf16
 * (io = GLA_IO_BF16) or fp32 (io = GLA_IO_F32); g_log, beta [B, T, H] fp32; h0, hT
 * [B, H, Dk, Dv] fp32, either may be NULL (zero initial state / final state not written).
 * The keys are used as given; the recurrence is stable for beta_t |k_t|^2 <= 2, e.g. unit
 * keys and beta in [0, 1].
 * Dims: Dk a multiple of 4 in [4, 128], Dv a multiple of 16 in [16, 128]
 * (GLA_ERR_UNSUPPORTED_DIM otherwise). Pointers are device pointers, 16-byte aligned
 * (GLA_ERR_MISALIGNED); o and hT must not overlap an input or each other (GLA_ERR_ALIAS).
 * Workspace: gdn_fwd_workspace_size() bytes of device memory (the size depends on the
 * current device: with few (batch, head) pairs the tensor-core scan splits the sequence over
 * its SMs and keeps the segments' transitions there), 16-byte aligned; pass NULL
 * to use the library's workspace of `stream` (one per stream and device, shared with
 * gla_fwd_ex calls on that stream; see gla_options.workspace).
 * A caller workspace smaller than needed, misaligned, or overlapping an argument returns
 * GLA_ERR_WORKSPACE. Arithmetic: bf16 I/O with Dk = Dv = 128 runs on the tensor cores
 * (bf16 products of the inputs and split-precision bf16 coefficients in the chunk-parallel
 * part, tf32 products with an fp32 state in the serial part, fp32 accumulation throughout);
 * every other case runs fp32 arithmetic on CUDA cores. Deterministic (no atomics). Two
 * kernels, stream-ordered on `stream`; no host synchronisation. T = 0 writes hT = h0 (or
 * zero) and launches nothing.
 */
size_t gdn_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv);
gla_status gdn_fwd(const void *q, const void *k, const void *v, const float *g_log,
                   const float *beta, float scale, const float *h0, void *o, float *hT,
                   int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                   void *workspace, size_t workspace_bytes, gla_stream_t stream);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H_ */
