// gla_fwd_noalloc: the forward of gla_fwd with its scratch memory taken from a fixed
// array compiled into this library instead of from cudaMalloc. See include/gla.h.
//
// The array lives in this translation unit's own module, so with CUDA's lazy module
// loading a process that never calls gla_fwd_noalloc does not load it; a GPU on which it
// is called holds it until the process exits.
#include <mutex>
#include <stdio.h>

#include "gla.h"
#include "gla_internal.h"

// Scratch of the tensor-core path (segment end states, segment decays and segment start
// states of the sequence split). Every element a call reads is written earlier in the
// same call, so nothing in it has to start at zero and leftovers of a previous call are
// harmless; calls that overlap on the GPU would race on it.
static __device__ __align__(256) float g_noalloc_scratch[GLA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// The host-side name g_noalloc_scratch is only a stand-in for the array: its device
// address is looked up once per device, with that device current, and cached.
gla_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        gla::set_error_detail("gla_fwd_noalloc: no usable current device");
        return GLA_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            char msg[200];
            snprintf(msg, sizeof(msg), "gla_fwd_noalloc: cudaGetSymbolAddress of the static scratch: %s (%d)",
                     cudaGetErrorString(e), (int)e);
            gla::set_error_detail(msg);
            return GLA_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GLA_OK;
}

}  // namespace

extern "C" gla_status gla_fwd_noalloc(const void *q, const void *k, const void *v,
                                      const float *g_log, float scale, const float *h0, void *o,
                                      float *hT, int64_t B, int64_t T, int64_t H, int64_t Dk,
                                      int64_t Dv, int seq_splits, gla_stream_t stream) {
    if (seq_splits < 0) return GLA_ERR_BAD_OPTION;
    const size_t cap = GLA_NOALLOC_SCRATCH_BYTES;
    gla_options opt{GLA_PATH_AUTO, seq_splits, nullptr, 0, GLA_GATE_KEY};
    size_t need = gla_fwd_workspace_size(B, T, H, Dk, Dv, GLA_IO_BF16, &opt);
    if (need > cap) {
        if (seq_splits > 0) {
            char msg[200];
            snprintf(msg, sizeof(msg),
                     "gla_fwd_noalloc: seq_splits=%d needs %zu bytes of scratch; the static scratch "
                     "holds %zu",
                     seq_splits, need, cap);
            gla::set_error_detail(msg);
            return GLA_ERR_WORKSPACE;
        }
        // automatic split: from the count gla_fwd would pick, down to the largest whose scratch
        // fits (one segment needs none)
        int s = gla::tc_auto_splits_for(B, T, H, Dk, Dv);
        for (; s > 1; --s) {
            opt.seq_splits = s;
            if (gla_fwd_workspace_size(B, T, H, Dk, Dv, GLA_IO_BF16, &opt) <= cap) break;
        }
        opt.seq_splits = s < 1 ? 1 : s;
        need = gla_fwd_workspace_size(B, T, H, Dk, Dv, GLA_IO_BF16, &opt);
    }
    if (need > 0) {
        // an unsupported device is reported as gla_fwd_ex would, before the symbol lookup
        const int dev_rc = gla::current_device_status();
        if (dev_rc != GLA_OK) return (gla_status)dev_rc;
        const gla_status rc = scratch_address(&opt.workspace);
        if (rc != GLA_OK) return rc;
        opt.workspace_bytes = cap;
    }
    return gla_fwd_ex(q, k, v, g_log, scale, h0, o, hT, B, T, H, Dk, Dv, GLA_IO_BF16, &opt, stream);
}
