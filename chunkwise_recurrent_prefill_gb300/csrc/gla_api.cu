// C ABI of libgla.so: argument validation, path selection, workspace, status.
// See include/gla.h for the contract of every entry point.
#include <atomic>
#include <mutex>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gla.h"
#include "gla_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Error word raised by kernels (bounded waits that ran out); one per device.
__device__ unsigned int g_dev_err;

// A workspace the library keeps for one stream of one device.
struct StreamWorkspace {
    cudaStream_t stream = nullptr;
    void *ptr = nullptr;
    size_t bytes = 0;
    uint64_t last_use = 0;
};

// At most this many streams per device keep a library workspace; the least recently used
// one is freed (cudaFree synchronises the device, so nothing still uses it) to make room.
constexpr int kMaxStreamWorkspaces = 16;

struct DeviceState {
    std::atomic<bool> probed{false};
    bool sm103 = false;
    int num_sms = 0;
    unsigned int *err_word = nullptr;
    StreamWorkspace ws[kMaxStreamWorkspaces];
    uint64_t ws_clock = 0;
};

std::mutex g_mu;
thread_local char g_detail[256] = "";

void set_detail(const char *where, cudaError_t e) {
    snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
}
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_ws_allocs{0};
DeviceState g_dev[kMaxDevices];

// Probe the current device once (under the library lock): architecture, SM count, error
// word address.
gla_status current_device(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GLA_ERR_LAUNCH;
    }
    DeviceState &st = g_dev[dev];
    if (!st.probed.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!st.probed.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                return GLA_ERR_LAUNCH;
            }
            st.sm103 = (major == 10 && minor == 3);
            st.num_sms = sms;
            if (st.sm103) {
                void *p = nullptr;
                if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess) {
                    cudaGetLastError();
                    return GLA_ERR_LAUNCH;
                }
                st.err_word = static_cast<unsigned int *>(p);
            }
            st.probed.store(true, std::memory_order_release);
        }
    }
    *out = &st;
    return st.sm103 ? GLA_OK : GLA_ERR_UNSUPPORTED_DEVICE;
}

bool misaligned(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Multiply non-negative sizes, flagging overflow past 2^62.
bool mul_ok(int64_t a, int64_t b, int64_t *r) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > (int64_t(1) << 62) / a) return false;
    *r = a * b;
    return true;
}

struct Sizes {
    int64_t nqk, nv, nstate;  // element counts
};

gla_status validate_shape(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                          Sizes *sz) {
    if (io != GLA_IO_BF16 && io != GLA_IO_F32) return GLA_ERR_BAD_OPTION;
    if (B < 0 || T < 0 || H < 0) return GLA_ERR_BAD_SHAPE;
    if (Dk <= 0 || Dv <= 0) return GLA_ERR_UNSUPPORTED_DIM;
    int64_t bth, bh;
    if (!mul_ok(B, T, &bth) || !mul_ok(bth, H, &bth) || !mul_ok(B, H, &bh))
        return GLA_ERR_BAD_SHAPE;
    if (!mul_ok(bth, Dk, &sz->nqk) || !mul_ok(bth, Dv, &sz->nv) ||
        !mul_ok(bh, Dk * Dv, &sz->nstate) || bh > (int64_t(1) << 31) - 1)
        return GLA_ERR_BAD_SHAPE;
    return GLA_OK;
}

gla_status validate(const void *q, const void *k, const void *v, const float *g,
                    const float *h0, const void *o, const float *hT, int64_t B, int64_t T,
                    int64_t H, int64_t Dk, int64_t Dv, int io, int gate, Sizes *sz) {
    gla_status rc = validate_shape(B, T, H, Dk, Dv, io, sz);
    if (rc != GLA_OK) return rc;
    const bool empty = (sz->nqk == 0);
    if (!empty && (!q || !k || !v || !g || !o)) return GLA_ERR_NULL_ARG;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(g) || misaligned(h0) ||
        misaligned(o) || misaligned(hT))
        return GLA_ERR_MISALIGNED;
    const size_t es = io == GLA_IO_BF16 ? 2 : 4;
    const size_t bqk = (size_t)sz->nqk * es, bv = (size_t)sz->nv * es;
    const size_t bg = (size_t)(gate == GLA_GATE_SCALAR ? sz->nqk / Dk : sz->nqk) * 4;
    const size_t bs = (size_t)sz->nstate * 4;
    const void *ins[5] = {q, k, v, g, h0};
    const size_t nins[5] = {bqk, bqk, bv, bg, bs};
    for (int i = 0; i < 5; ++i) {
        if (overlap(o, bv, ins[i], nins[i]) || overlap(hT, bs, ins[i], nins[i]))
            return GLA_ERR_ALIAS;
    }
    if (overlap(o, bv, hT, bs)) return GLA_ERR_ALIAS;
    return GLA_OK;
}

// The library-owned workspace of `stream` on the current device. Each stream has its own, so
// calls on different streams never share scratch; a stream's buffer is allocated on its first
// call that needs one and replaced only when a call needs more (sizes are rounded up to a power
// of two), so repeated calls allocate nothing.
gla_status library_workspace(DeviceState *st, cudaStream_t stream, size_t need, void **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    StreamWorkspace *slot = nullptr;
    for (auto &w : st->ws)
        if (w.ptr && w.stream == stream) slot = &w;
    if (!slot) {
        for (auto &w : st->ws)
            if (!w.ptr) { slot = &w; break; }
        if (!slot) {   // every slot taken: reuse the least recently used one
            slot = &st->ws[0];
            for (auto &w : st->ws)
                if (w.last_use < slot->last_use) slot = &w;
        }
        if (slot->stream != stream && slot->ptr) {
            cudaFree(slot->ptr);   // synchronises the device: no call still uses it
            slot->ptr = nullptr;
            slot->bytes = 0;
        }
        slot->stream = stream;
    }
    if (slot->bytes < need) {
        if (slot->ptr) {
            cudaFree(slot->ptr);   // synchronises the device: no call still uses it
            slot->ptr = nullptr;
            slot->bytes = 0;
        }
        size_t bytes = 1 << 20;
        while (bytes < need) bytes <<= 1;
        void *p = nullptr;
        const cudaError_t e = cudaMalloc(&p, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            set_detail("workspace cudaMalloc", e);
            return GLA_ERR_WORKSPACE;
        }
        g_ws_allocs.fetch_add(1, std::memory_order_relaxed);
        slot->ptr = p;
        slot->bytes = bytes;
    }
    slot->last_use = ++st->ws_clock;
    *out = slot->ptr;
    return GLA_OK;
}

// AUTO: tensor cores for bf16 I/O, except sequences shorter than one 64-token chunk.
// There each output is a handful of bf16-rounded dot products with no averaging, and the
// exact fp32 kernel is both more accurate and as fast.
int resolve_path(const gla_options *opt, const gla::Problem &p) {
    const int path = opt ? opt->path : GLA_PATH_AUTO;
    if (path != GLA_PATH_AUTO) return path;
    return (p.io == GLA_IO_BF16 && p.T >= 64 && gla::tc_supported(p)) ? GLA_PATH_TC
                                                                       : GLA_PATH_EXACT;
}

}  // namespace

namespace gla {
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
int current_device_status() {
    DeviceState *st = nullptr;
    return (int)current_device(&st);
}
int tc_auto_splits_for(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv) {
    DeviceState *st = nullptr;
    const int sms = current_device(&st) == GLA_OK ? st->num_sms : 152;
    Problem p{};
    p.B = B; p.T = T; p.H = H; p.Dk = Dk; p.Dv = Dv;
    return tc_auto_splits(p, sms);
}
void set_error_detail(const char *text) { snprintf(g_detail, sizeof(g_detail), "%s", text); }
}  // namespace gla

extern "C" {

const char *gla_last_error_detail(void) { return g_detail; }

uint64_t gla_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t gla_workspace_allocations(void) { return g_ws_allocs.load(std::memory_order_relaxed); }

int gla_version(void) { return 100; }

const char *gla_status_string(gla_status s) {
    switch (s) {
        case GLA_OK: return "GLA_OK";
        case GLA_ERR_NULL_ARG: return "GLA_ERR_NULL_ARG";
        case GLA_ERR_BAD_SHAPE: return "GLA_ERR_BAD_SHAPE";
        case GLA_ERR_UNSUPPORTED_DIM: return "GLA_ERR_UNSUPPORTED_DIM";
        case GLA_ERR_MISALIGNED: return "GLA_ERR_MISALIGNED";
        case GLA_ERR_ALIAS: return "GLA_ERR_ALIAS";
        case GLA_ERR_LAUNCH: return "GLA_ERR_LAUNCH";
        case GLA_ERR_DEVICE_TIMEOUT: return "GLA_ERR_DEVICE_TIMEOUT";
        case GLA_ERR_UNSUPPORTED_DEVICE: return "GLA_ERR_UNSUPPORTED_DEVICE";
        case GLA_ERR_WORKSPACE: return "GLA_ERR_WORKSPACE";
        case GLA_ERR_BAD_OPTION: return "GLA_ERR_BAD_OPTION";
        case GLA_ERR_BAD_SEQLENS: return "GLA_ERR_BAD_SEQLENS";
    }
    return "GLA_ERR_UNKNOWN";
}

int gla_path_for(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                 const gla_options *opt) {
    Sizes sz;
    if (validate_shape(B, T, H, Dk, Dv, io, &sz) != GLA_OK) return -1;
    gla::Problem p{};
    p.B = B; p.T = T; p.H = H; p.Dk = Dk; p.Dv = Dv; p.io = io;
    const int path = resolve_path(opt, p);
    if (path == GLA_PATH_EXACT) return gla::exact_supported(Dk, Dv) ? path : -1;
    if (path == GLA_PATH_TC) return (io == GLA_IO_BF16 && gla::tc_supported(p)) ? path : -1;
    return -1;
}

size_t gla_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                              const gla_options *opt) {
    Sizes sz;
    if (validate_shape(B, T, H, Dk, Dv, io, &sz) != GLA_OK) return 0;
    gla::Problem p{};
    p.B = B; p.T = T; p.H = H; p.Dk = Dk; p.Dv = Dv; p.io = io;
    if (resolve_path(opt, p) != GLA_PATH_TC || !gla::tc_supported(p)) return 0;
    int splits = opt ? opt->seq_splits : 0;
    DeviceState *st = nullptr;
    const int sms = current_device(&st) == GLA_OK ? st->num_sms : 152;
    if (splits <= 0) splits = gla::tc_auto_splits(p, sms);
    return gla::tc_workspace_bytes(p, splits, sms);
}

gla_status gla_fwd_ex(const void *q, const void *k, const void *v, const float *g_log,
                      float scale, const float *h0, void *o, float *hT, int64_t B, int64_t T,
                      int64_t H, int64_t Dk, int64_t Dv, int io, const gla_options *opt,
                      gla_stream_t stream) {
    Sizes sz;
    const int gate = opt ? opt->gate : GLA_GATE_KEY;
    if (gate != GLA_GATE_KEY && gate != GLA_GATE_SCALAR) return GLA_ERR_BAD_OPTION;
    gla_status rc = validate(q, k, v, g_log, h0, o, hT, B, T, H, Dk, Dv, io, gate, &sz);
    if (rc != GLA_OK) return rc;
    gla::Problem p{q, k, v, g_log, scale, h0, o, hT, B, T, H, Dk, Dv, io, gate, nullptr, 0};
    const int path = resolve_path(opt, p);
    if (path != GLA_PATH_EXACT && path != GLA_PATH_TC) return GLA_ERR_BAD_OPTION;
    if (opt && opt->seq_splits < 0) return GLA_ERR_BAD_OPTION;
    if (path == GLA_PATH_EXACT && !gla::exact_supported(Dk, Dv)) return GLA_ERR_UNSUPPORTED_DIM;
    if (path == GLA_PATH_TC && (io != GLA_IO_BF16 || !gla::tc_supported(p)))
        return GLA_ERR_UNSUPPORTED_DIM;
    if (opt && opt->workspace && misaligned(opt->workspace)) return GLA_ERR_WORKSPACE;

    DeviceState *st = nullptr;
    rc = current_device(&st);
    if (rc != GLA_OK) return rc;
    if (B * H == 0) return GLA_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (path == GLA_PATH_EXACT) {
        e = gla::launch_exact(p, st->err_word, s);
    } else {
        int splits = (opt && opt->seq_splits > 0) ? opt->seq_splits
                                                  : gla::tc_auto_splits(p, st->num_sms);
        const size_t need = gla::tc_workspace_bytes(p, splits, st->num_sms);
        void *ws = nullptr;
        if (need > 0) {
            if (opt && opt->workspace) {
                if (opt->workspace_bytes < need) return GLA_ERR_WORKSPACE;
                ws = opt->workspace;
            } else {
                rc = library_workspace(st, reinterpret_cast<cudaStream_t>(stream), need, &ws);
                if (rc != GLA_OK) return rc;
            }
        }
        e = gla::launch_tc(p, splits, st->num_sms, ws, need, st->err_word, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_detail(path == GLA_PATH_EXACT ? "exact path launch" : "tensor-core path launch", e);
        return GLA_ERR_LAUNCH;
    }
    return GLA_OK;
}

gla_status gla_fwd_varlen(const void *q, const void *k, const void *v, const float *g_log,
                          float scale, const float *h0, void *o, float *hT,
                          const int32_t *cu_seqlens, int64_t N, int64_t T, int64_t H,
                          int64_t Dk, int64_t Dv, int io, const gla_options *opt,
                          gla_stream_t stream) {
    // the token tensors are one batch of T tokens; the states are N per head
    Sizes sz;
    const int gate = opt ? opt->gate : GLA_GATE_KEY;
    if (gate != GLA_GATE_KEY && gate != GLA_GATE_SCALAR) return GLA_ERR_BAD_OPTION;
    if (N < 0) return GLA_ERR_BAD_SHAPE;
    gla_status rc = validate(q, k, v, g_log, nullptr, o, nullptr, 1, T, H, Dk, Dv, io, gate, &sz);
    if (rc != GLA_OK) return rc;
    int64_t nstate;
    if (!mul_ok(N, H, &nstate) || !mul_ok(nstate, Dk * Dv, &nstate) || N * H > (int64_t(1) << 24))
        return GLA_ERR_BAD_SHAPE;
    if (N > 0 && !cu_seqlens) return GLA_ERR_NULL_ARG;
    if (misaligned(h0) || misaligned(hT) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return GLA_ERR_MISALIGNED;
    const size_t es = io == GLA_IO_BF16 ? 2 : 4;
    const size_t bqk = (size_t)sz.nqk * es, bv = (size_t)sz.nv * es;
    const size_t bg = (size_t)(gate == GLA_GATE_SCALAR ? sz.nqk / Dk : sz.nqk) * 4;
    const size_t bs = (size_t)nstate * 4, bcu = (size_t)(N + 1) * 4;
    const void *ins[6] = {q, k, v, g_log, h0, cu_seqlens};
    const size_t nins[6] = {bqk, bqk, bv, bg, bs, bcu};
    for (int i = 0; i < 6; ++i) {
        if (overlap(o, bv, ins[i], nins[i]) || overlap(hT, bs, ins[i], nins[i]))
            return GLA_ERR_ALIAS;
    }
    if (overlap(o, bv, hT, bs)) return GLA_ERR_ALIAS;
    gla::Problem p{q, k, v, g_log, scale, h0, o, hT, N, T, H, Dk, Dv, io, gate, cu_seqlens, 0};
    const int path = resolve_path(opt, p);
    if (path != GLA_PATH_EXACT && path != GLA_PATH_TC) return GLA_ERR_BAD_OPTION;
    if (path == GLA_PATH_EXACT && !gla::exact_supported(Dk, Dv)) return GLA_ERR_UNSUPPORTED_DIM;
    if (path == GLA_PATH_TC && (io != GLA_IO_BF16 || !gla::tc_supported(p)))
        return GLA_ERR_UNSUPPORTED_DIM;
    DeviceState *st = nullptr;
    rc = current_device(&st);
    if (rc != GLA_OK) return rc;
    if (N * H == 0) return GLA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = path == GLA_PATH_EXACT
                              ? gla::launch_exact(p, st->err_word, s)
                              : gla::launch_tc(p, 1, st->num_sms, nullptr, 0, st->err_word, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_detail(path == GLA_PATH_EXACT ? "exact path launch" : "tensor-core path launch", e);
        return GLA_ERR_LAUNCH;
    }
    return GLA_OK;
}

gla_status gla_fwd(const void *q, const void *k, const void *v, const float *g_log, float scale,
                   const float *h0, void *o, float *hT, int64_t B, int64_t T, int64_t H,
                   int64_t Dk, int64_t Dv, gla_stream_t stream) {
    return gla_fwd_ex(q, k, v, g_log, scale, h0, o, hT, B, T, H, Dk, Dv, GLA_IO_BF16, nullptr,
                      stream);
}

gla_status gla_fwd_f32(const float *q, const float *k, const float *v, const float *g_log,
                       float scale, const float *h0, float *o, float *hT, int64_t B, int64_t T,
                       int64_t H, int64_t Dk, int64_t Dv, gla_stream_t stream) {
    return gla_fwd_ex(q, k, v, g_log, scale, h0, o, hT, B, T, H, Dk, Dv, GLA_IO_F32, nullptr,
                      stream);
}

gla_status gla_step(const void *q, const void *k, const void *v, const float *g_log, float scale,
                    float *S, void *o, int64_t B, int64_t H, int64_t Dk, int64_t Dv, int io,
                    gla_stream_t stream) {
    // one token: the shapes of gla_fwd_ex with T = 1; S plays h0 (in) and hT (out)
    Sizes sz;
    gla_status rc = validate_shape(B, 1, H, Dk, Dv, io, &sz);
    if (rc != GLA_OK) return rc;
    if (!gla::step_supported(Dk, Dv)) return GLA_ERR_UNSUPPORTED_DIM;
    const bool empty = (sz.nqk == 0);
    if (!empty && (!q || !k || !v || !g_log || !S || !o)) return GLA_ERR_NULL_ARG;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(g_log) || misaligned(S) ||
        misaligned(o))
        return GLA_ERR_MISALIGNED;
    const size_t es = io == GLA_IO_BF16 ? 2 : 4;
    const size_t bqk = (size_t)sz.nqk * es, bv = (size_t)sz.nv * es;
    const size_t bg = (size_t)sz.nqk * 4, bs = (size_t)sz.nstate * 4;
    const void *ins[4] = {q, k, v, g_log};
    const size_t nins[4] = {bqk, bqk, bv, bg};
    for (int i = 0; i < 4; ++i) {
        if (overlap(o, bv, ins[i], nins[i]) || overlap(S, bs, ins[i], nins[i]))
            return GLA_ERR_ALIAS;
    }
    if (overlap(o, bv, S, bs)) return GLA_ERR_ALIAS;
    DeviceState *st = nullptr;
    rc = current_device(&st);
    if (rc != GLA_OK) return rc;
    if (empty) return GLA_OK;
    const cudaError_t e = gla::launch_step(q, k, v, g_log, scale, S, o, B * H, Dk, Dv, io,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_detail("decode step launch", e);
        return GLA_ERR_LAUNCH;
    }
    return GLA_OK;
}

size_t gdn_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv) {
    Sizes sz;
    if (validate_shape(B, T, H, Dk, Dv, GLA_IO_BF16, &sz) != GLA_OK) return 0;
    if (!gla::gdn_supported(Dk, Dv) || sz.nqk == 0) return 0;
    DeviceState *st = nullptr;
    const int sms = current_device(&st) == GLA_OK ? st->num_sms : 152;
    return gla::gdn_workspace_bytes(B, T, H, Dk, Dv, sms);
}

gla_status gdn_fwd(const void *q, const void *k, const void *v, const float *g_log,
                   const float *beta, float scale, const float *h0, void *o, float *hT,
                   int64_t B, int64_t T, int64_t H, int64_t Dk, int64_t Dv, int io,
                   void *workspace, size_t workspace_bytes, gla_stream_t stream) {
    Sizes sz;
    gla_status rc = validate_shape(B, T, H, Dk, Dv, io, &sz);
    if (rc != GLA_OK) return rc;
    if (!gla::gdn_supported(Dk, Dv)) return GLA_ERR_UNSUPPORTED_DIM;
    const bool empty = (sz.nqk == 0);
    if (!empty && (!q || !k || !v || !g_log || !beta || !o)) return GLA_ERR_NULL_ARG;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(g_log) || misaligned(beta) ||
        misaligned(h0) || misaligned(o) || misaligned(hT))
        return GLA_ERR_MISALIGNED;
    const size_t es = io == GLA_IO_BF16 ? 2 : 4;
    const size_t bqk = (size_t)sz.nqk * es, bv = (size_t)sz.nv * es;
    const size_t bg = (size_t)(sz.nqk / Dk) * 4, bs = (size_t)sz.nstate * 4;
    const void *ins[6] = {q, k, v, g_log, beta, h0};
    const size_t nins[6] = {bqk, bqk, bv, bg, bg, bs};
    for (int i = 0; i < 6; ++i) {
        if (overlap(o, bv, ins[i], nins[i]) || overlap(hT, bs, ins[i], nins[i]))
            return GLA_ERR_ALIAS;
    }
    if (overlap(o, bv, hT, bs)) return GLA_ERR_ALIAS;
    // the size the caller got from gdn_fwd_workspace_size on this device (the device itself is
    // checked below, after the caller's arguments)
    DeviceState *st = nullptr;
    const gla_status dev_rc = current_device(&st);
    const int sms = dev_rc == GLA_OK ? st->num_sms : 152;
    const size_t need = empty ? 0 : gla::gdn_workspace_bytes(B, T, H, Dk, Dv, sms);
    if (workspace) {
        if (misaligned(workspace) || workspace_bytes < need) return GLA_ERR_WORKSPACE;
        for (int i = 0; i < 6; ++i)
            if (overlap(workspace, need, ins[i], nins[i])) return GLA_ERR_WORKSPACE;
        if (overlap(workspace, need, o, bv) || overlap(workspace, need, hT, bs))
            return GLA_ERR_WORKSPACE;
    }
    if (dev_rc != GLA_OK) return dev_rc;
    if (empty) {
        // no tokens: the final state is the initial one (zero without h0)
        if (T == 0 && B * H > 0 && hT) {
            cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
            const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, bs, cudaMemcpyDeviceToDevice, s)
                                     : cudaMemsetAsync(hT, 0, bs, s);
            if (e != cudaSuccess) {
                cudaGetLastError();
                set_detail("gated delta rule: final state of an empty sequence", e);
                return GLA_ERR_LAUNCH;
            }
        }
        return GLA_OK;
    }
    void *ws = workspace;
    if (!ws) {
        rc = library_workspace(st, reinterpret_cast<cudaStream_t>(stream), need, &ws);
        if (rc != GLA_OK) return rc;
    }
    gla::GdnProblem p{q, k, v, g_log, beta, scale, h0, o, hT, B, T, H, Dk, Dv, io};
    const cudaError_t e = gla::launch_gdn(p, ws, st->num_sms, st->err_word,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_detail("gated delta rule launch", e);
        return GLA_ERR_LAUNCH;
    }
    return GLA_OK;
}

gla_status gla_last_device_status(gla_stream_t stream) {
    DeviceState *st = nullptr;
    gla_status rc = current_device(&st);
    if (rc != GLA_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_LAUNCH;
    }
    unsigned int word = 0;
    if (cudaMemcpy(&word, st->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_LAUNCH;
    }
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(st->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return GLA_ERR_LAUNCH;
        }
        return (word & gla::kDevErrTimeout) ? GLA_ERR_DEVICE_TIMEOUT : GLA_ERR_BAD_SEQLENS;
    }
    return GLA_OK;
}

}  // extern "C"
