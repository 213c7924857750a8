// Host-side declarations shared by the translation units of libgla.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

namespace gla {

// One forward problem, already validated by the C ABI layer.
struct Problem {
    const void *q, *k, *v;   // [B,T,H,Dk] / [B,T,H,Dv], bf16 or fp32 (io)
    const float *g;          // [B,T,H,Dk] log-gates
    float scale;
    const float *h0;         // [B,H,Dk,Dv] or nullptr
    void *o;                 // [B,T,H,Dv]
    float *hT;               // [B,H,Dk,Dv] or nullptr
    int64_t B, T, H, Dk, Dv;
    int io;                  // GLA_IO_BF16 / GLA_IO_F32
    int gate;                // GLA_GATE_KEY: g [B,T,H,Dk]; GLA_GATE_SCALAR: g [B,T,H]
    const int *cu;           // packed sequences: B sequences at offsets cu[0..B] along a
                             // single batch of T tokens (device), or null
    int seq_filter;          // packed sequences only: 0 = every sequence; kShortOnly = only
                             // those shorter than one 64-token chunk; kLongOnly = only the others
};

// Packed-sequence filters (Problem::seq_filter): the tensor-core path runs the sequences of at
// least one chunk, and the exact kernel the shorter ones, whose few bf16-rounded products
// nothing averages.
constexpr int kShortOnly = 1;
constexpr int kLongOnly = 2;
constexpr int kShortSeq = 64;

// Bits of the device error word kernels may raise (never trap).
enum : unsigned int {
    kDevErrTimeout = 1u,     // a bounded mbarrier / flag wait ran out
    kDevErrInternal = 2u,    // an input the host could not check was inconsistent (packed-
                             // sequence offsets not non-decreasing from 0 to T)
};

// Status (a gla_status value) of the current device: GLA_OK for an sm_103 device, else the
// error gla_fwd_ex would return; probes the device once.
int current_device_status();

// Host-side count of kernel launches issued by the library (gla_launch_counter).
void count_launches(unsigned n);

// Sets the text gla_last_error_detail() returns on this host thread.
void set_error_detail(const char *text);

// Exact fp32 CUDA-core chunkwise kernel (any io, Dk/Dv in {64,128}).
bool exact_supported(int64_t Dk, int64_t Dv);
cudaError_t launch_exact(const Problem &p, unsigned int *dev_err, cudaStream_t s);

// One decode step on a resident state (any io, 1 <= Dk <= 1024, Dv a multiple of 4 <= 1024).
bool step_supported(int64_t Dk, int64_t Dv);
cudaError_t launch_step(const void *q, const void *k, const void *v, const float *g, float scale,
                        float *S, void *o, int64_t BH, int64_t Dk, int64_t Dv, int io,
                        cudaStream_t stream);

// tcgen05 path (bf16 io, Dk and Dv in {64, 128}).
bool tc_supported(const Problem &p);
int tc_auto_splits(const Problem &p, int num_sms);
// tc_auto_splits of a bf16 problem of this shape on the current device (152 SMs if it cannot
// be queried).
int tc_auto_splits_for(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv);
int tc_state_pieces(const Problem &p, int splits, int num_sms);
size_t tc_workspace_bytes(const Problem &p, int splits, int num_sms);
cudaError_t launch_tc(const Problem &p, int splits, int num_sms, void *ws, size_t ws_bytes,
                      unsigned int *dev_err, cudaStream_t s);

// Gated delta rule forward (fp32 CUDA cores): chunk-parallel prep, then the state scan.
struct GdnProblem {
    const void *q, *k, *v;   // [B,T,H,Dk] / [B,T,H,Dv], bf16 or fp32 (io)
    const float *g, *beta;   // [B,T,H] log-gates and write strengths
    float scale;
    const float *h0;         // [B,H,Dk,Dv] or nullptr
    void *o;                 // [B,T,H,Dv]
    float *hT;               // [B,H,Dk,Dv] or nullptr
    int64_t B, T, H, Dk, Dv;
    int io;
};
bool gdn_supported(int64_t Dk, int64_t Dv);
// Workspace of gdn_fwd on a device with num_sms SMs (the tensor-core scan's split depends on it).
size_t gdn_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int num_sms);
cudaError_t launch_gdn(const GdnProblem &p, void *ws, int num_sms, unsigned int *dev_err,
                       cudaStream_t s);

}  // namespace gla
