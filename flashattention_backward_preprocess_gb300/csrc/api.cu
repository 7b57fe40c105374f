// api.cu -- the C ABI (include/fa.h): argument validation, the per
// (device, stream) workspace cache and the launch sequence of each entry
// point.  Validation mirrors the checks of boostr flash_bwd.rs
// (flash_attention_bwd_impl: dout / output / lse shapes, contiguity, dtype,
// window_size) and rustytorch backward.rs (flash_attention_backward: 4-D Q,
// grad_output shape == Q shape, LSE shape) for what a C ABI of raw pointers
// can check: pointers, sizes, alignment, dtype, scale, head dim.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <vector>
#include <string>
#include <utility>

#include "fa_internal.cuh"

namespace fa {
namespace {

thread_local std::string g_last_error;

int fail(int status, const char* arg, const std::string& reason) {
    g_last_error = std::string(arg) + ": " + reason;
    return status;
}

int cuda_fail(const char* where, cudaError_t e) {
    return fail(FA_ERR_CUDA, where, cudaGetErrorString(e));
}

bool debug_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("FA_DEBUG");
        v = (e && *e && *e != '0') ? 1 : 0;
    }
    return v == 1;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int pad_rows(int S_q) { return (S_q + kTileQ - 1) / kTileQ * kTileQ; }

struct WsLayout {
    size_t off_err, off_lse2, off_D, off_dq, off_sem, sem_bytes, total;
};

WsLayout ws_layout(int B, int H, int S_q, int d) {
    WsLayout L;
    const size_t rows_pad = (size_t)B * H * pad_rows(S_q);
    L.off_err = 0;
    L.off_lse2 = 256;
    L.off_D = align_up(L.off_lse2 + rows_pad * 4, 256);
    L.off_dq = align_up(L.off_D + rows_pad * 4, 256);
    L.off_sem = align_up(L.off_dq + (size_t)B * H * S_q * d * 4, 256);
    // turn counters, then the CTA ticket counter
    L.sem_bytes = ((size_t)B * H * ((S_q + kTileQ - 1) / kTileQ) + 1) * 4;
    L.total = align_up(L.off_sem + L.sem_bytes, 256);
    return L;
}

struct WsEntry {
    void* base = nullptr;
    size_t bytes = 0;
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws;

// Grow-only workspace of at least `bytes` for (current device, stream).
int get_workspace(cudaStream_t st, size_t bytes, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    WsEntry& w = g_ws[{dev, st}];
    if (w.bytes < bytes) {
        if (w.base) {
            // the old buffer may still be in use by work queued on this stream
            e = cudaStreamSynchronize(st);
            if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
            cudaFree(w.base);
            w.base = nullptr;
            w.bytes = 0;
        }
        void* p = nullptr;
        e = cudaMalloc(&p, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(FA_ERR_NOMEM, "workspace", std::string("cudaMalloc failed: ") + cudaGetErrorString(e));
        }
        e = cudaMemsetAsync(p, 0, 256, st);  // error words
        if (e != cudaSuccess) return cuda_fail("cudaMemsetAsync", e);
        w.base = p;
        w.bytes = bytes;
    }
    *out = w.base;
    return FA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_dims(int B, int H, int H_kv, int S_q, int S_k, int d, int dtype) {
    if (B <= 0) return fail(FA_ERR_INVALID_ARG, "B", "must be > 0, got " + std::to_string(B));
    if (H <= 0) return fail(FA_ERR_INVALID_ARG, "H", "must be > 0, got " + std::to_string(H));
    if (H_kv <= 0) return fail(FA_ERR_INVALID_ARG, "H_kv", "must be > 0, got " + std::to_string(H_kv));
    if (H % H_kv != 0)
        return fail(FA_ERR_INVALID_ARG, "H_kv",
                    "num_kv_heads " + std::to_string(H_kv) + " must divide num_heads " + std::to_string(H));
    if (S_q <= 0) return fail(FA_ERR_INVALID_ARG, "S_q", "must be > 0, got " + std::to_string(S_q));
    if (S_k <= 0) return fail(FA_ERR_INVALID_ARG, "S_k", "must be > 0, got " + std::to_string(S_k));
    if (d <= 0) return fail(FA_ERR_INVALID_ARG, "d", "must be > 0, got " + std::to_string(d));
    if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16)
        return fail(FA_ERR_INVALID_ARG, "dtype", "unsupported dtype " + std::to_string(dtype) +
                                                     " (expected FA_F32, FA_F16 or FA_BF16)");
    if (!head_dim_supported(d))
        return fail(FA_ERR_UNSUPPORTED, "d",
                    "head dim " + std::to_string(d) + " not supported (32, 64, 96, 128 or 256)");
    // every flattened index must fit the kernels' 32-bit row arithmetic
    const double rows_q = (double)B * H * (double)pad_rows(S_q);
    const double rows_k = (double)B * H_kv * (double)S_k;
    if (rows_q * d >= 9.0e18 || rows_q >= 2147483647.0 || rows_k >= 2147483647.0)
        return fail(FA_ERR_INVALID_ARG, "shape", "tensor too large");
    return FA_OK;
}

int check_scale(float scale) {
    if (!(isfinite(scale) && scale > 0.f))
        return fail(FA_ERR_INVALID_ARG, "scale", "must be finite and > 0");
    return FA_OK;
}

int check_ptr(const void* p, const char* name, size_t align) {
    if (p == nullptr) return fail(FA_ERR_INVALID_ARG, name, "null pointer");
    if (!aligned(p, align))
        return fail(FA_ERR_INVALID_ARG, name, "must be " + std::to_string(align) + "-byte aligned");
    return FA_OK;
}

Shape make_shape(int B, int H, int H_kv, int S_q, int S_k, int d, float scale, int causal,
                 int window = 0) {
    Shape s;
    s.B = B;
    s.H = H;
    s.H_kv = H_kv;
    s.S_q = S_q;
    s.S_k = S_k;
    s.d = d;
    s.scale = scale;
    s.causal = causal ? 1 : 0;
    s.window = window;
    s.S_q_pad = pad_rows(S_q);
    return s;
}

// ---- optional per-kernel event timing (fa_profile)
struct ProfRec {
    cudaEvent_t ev[4];
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_used;
std::vector<ProfRec> g_prof_free;

bool prof_begin(ProfRec* r) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return false;
    if (!g_prof_free.empty()) {
        *r = g_prof_free.back();
        g_prof_free.pop_back();
        return true;
    }
    for (int i = 0; i < 4; ++i)
        if (cudaEventCreate(&r->ev[i]) != cudaSuccess) return false;
    return true;
}
void prof_end(const ProfRec& r) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_used.push_back(r);
}

bool use_simt_for_16bit() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("FA_BWD_KERNEL");
        v = (e && std::string(e) == "simt") ? 1 : 0;
    }
    return v == 1;
}

// FA_FWD_KERNEL=simt: the forward helper on CUDA cores for f16 / bf16 too
bool fwd_simt_for_16bit() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("FA_FWD_KERNEL");
        v = (e && std::string(e) == "simt") ? 1 : 0;
    }
    return v == 1;
}

int check_window(int window) {
    if (window < 0) return fail(FA_ERR_INVALID_ARG, "window_size", "must be >= 0 (0 = no window)");
    return FA_OK;
}

int bwd_impl(const void* dO, const void* Q, const void* K, const void* V, const void* O,
             const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
             int S_k, int d, float scale, int causal, int window, int deterministic, int dtype,
             cudaStream_t st) {
    int rc;
    if ((rc = check_dims(B, H, H_kv, S_q, S_k, d, dtype))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal", "must be 0 or 1");
    if ((rc = check_window(window))) return rc;
    if (deterministic != 0 && deterministic != 1)
        return fail(FA_ERR_INVALID_ARG, "deterministic", "must be 0 or 1");
    if ((rc = check_ptr(dO, "dO", 16)) || (rc = check_ptr(Q, "Q", 16)) || (rc = check_ptr(K, "K", 16)) ||
        (rc = check_ptr(V, "V", 16)) || (rc = check_ptr(O, "O", 16)) || (rc = check_ptr(LSE, "LSE", 4)) ||
        (rc = check_ptr(dQ, "dQ", 16)) || (rc = check_ptr(dK, "dK", 16)) || (rc = check_ptr(dV, "dV", 16)))
        return rc;
    const Shape s = make_shape(B, H, H_kv, S_q, S_k, d, scale, causal, window);
    const WsLayout L = ws_layout(B, H, S_q, d);
    void* base = nullptr;
    if ((rc = get_workspace(st, L.total, &base))) return rc;
    Workspace ws;
    ws.err = reinterpret_cast<unsigned int*>(static_cast<char*>(base) + L.off_err);
    ws.lse2 = reinterpret_cast<float*>(static_cast<char*>(base) + L.off_lse2);
    ws.Dws = reinterpret_cast<float*>(static_cast<char*>(base) + L.off_D);
    ws.dqacc = reinterpret_cast<float*>(static_cast<char*>(base) + L.off_dq);
    ws.dq_sem = nullptr;
    ws.dq_ticket = nullptr;
    const int kind = bwd_kernel_for(dtype, d);
    const bool tc = kind == kBwdSm103;
    if (deterministic && tc) {
        ws.dq_sem = reinterpret_cast<unsigned int*>(static_cast<char*>(base) + L.off_sem);
        ws.dq_ticket = ws.dq_sem + L.sem_bytes / 4 - 1;
        cudaError_t me = cudaMemsetAsync(ws.dq_sem, 0, L.sem_bytes, st);
        if (me != cudaSuccess) return cuda_fail("turn counter reset", me);
    }
    if (debug_enabled())
        fprintf(stderr,
                "[fa] bwd B=%d H=%d H_kv=%d S_q=%d S_k=%d d=%d causal=%d window=%d det=%d dtype=%d kernel=%s "
                "grid=%d ws=%zu\n",
                B, H, H_kv, S_q, S_k, d, causal, window, deterministic, dtype,
                kind == kBwdSm103 ? "sm103" : (kind == kBwdD256 ? "d256" : "simt"),
                tc ? (S_k + kTileK - 1) / kTileK * B * H_kv : 0, L.total);
    ProfRec pr;
    const bool prof = prof_begin(&pr);
    if (prof) cudaEventRecord(pr.ev[0], st);
    cudaError_t e = launch_preprocess(dtype, dO, O, LSE, ws.Dws, ws.lse2, ws.dqacc, s, s.S_q_pad, st);
    if (e != cudaSuccess) return cuda_fail("preprocess launch", e);
    if (prof) cudaEventRecord(pr.ev[1], st);
    if (tc) {
        e = launch_bwd_sm103(dtype, Q, K, V, dO, ws, dK, dV, s, st);
    } else if (kind == kBwdD256) {
        // deterministic: dK, dV on the tensor cores, dQ summed in key order on CUDA cores
        e = launch_bwd_d256(dtype, Q, K, V, dO, ws, dK, dV, s, deterministic != 0, st);
        if (e == cudaSuccess && deterministic) e = launch_dq_simt(dtype, Q, K, V, dO, ws, s, st);
    } else {
        // CUDA-core path: deterministic dQ comes from its own kernel, which sums each row's
        // contributions in key order; the main kernel then leaves dQ alone
        e = launch_bwd_simt(dtype, Q, K, V, dO, ws, dK, dV, s, deterministic != 0, st);
        if (e == cudaSuccess && deterministic) e = launch_dq_simt(dtype, Q, K, V, dO, ws, s, st);
    }
    if (e != cudaSuccess) return cuda_fail("main kernel launch", e);
    if (prof) cudaEventRecord(pr.ev[2], st);
    e = launch_dq_finalize(dtype, ws.dqacc, dQ, s, st);
    if (e != cudaSuccess) return cuda_fail("dq finalize launch", e);
    if (prof) {
        cudaEventRecord(pr.ev[3], st);
        prof_end(pr);
    }
    return FA_OK;
}

int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
             int S_q, int S_k, int d, float scale, int causal, int window, int dtype, cudaStream_t st) {
    int rc;
    if ((rc = check_dims(B, H, H_kv, S_q, S_k, d, dtype))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal", "must be 0 or 1");
    if ((rc = check_window(window))) return rc;
    if ((rc = check_ptr(Q, "Q", 16)) || (rc = check_ptr(K, "K", 16)) || (rc = check_ptr(V, "V", 16)) ||
        (rc = check_ptr(O, "O", 16)) || (rc = check_ptr(LSE, "LSE", 4)))
        return rc;
    const Shape s = make_shape(B, H, H_kv, S_q, S_k, d, scale, causal, window);
    cudaError_t e;
    // f16 / bf16: the tensor-core forward at every supported head dim (d = 256 with 64-key
    // tiles); f32 (and FA_FWD_KERNEL=simt): the CUDA-core helper
    if (dtype == FA_F32 || fwd_simt_for_16bit()) {
        e = launch_fwd_simt(dtype, Q, K, V, O, LSE, s, st);
    } else {
        // the tensor-core forward reports bounded-wait timeouts in the stream's workspace
        // error words (fa_check_device reads them)
        void* base = nullptr;
        if ((rc = get_workspace(st, 256, &base))) return rc;
        e = launch_fwd_sm103(dtype, Q, K, V, O, LSE, static_cast<unsigned int*>(base), s, st);
    }
    if (e != cudaSuccess) return cuda_fail("forward launch", e);
    return FA_OK;
}

size_t elem_size(int dtype) { return dtype == FA_F32 ? 4 : 2; }

// Host-buffer staging for fa_bwd_host, per (device, stream): device buffers for every
// input and output, two copy streams (host -> device, device -> host) and one pair of
// events per chunk of the copy / compute pipeline.
constexpr int kHostMaxChunks = 4;
constexpr size_t kHostChunkBytes = 16u << 20;  // input bytes per pipeline chunk (target)
struct HostStage {
    void* base = nullptr;
    size_t bytes = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kHostMaxChunks] = {}, ev_done[kHostMaxChunks] = {};
};
std::map<std::pair<int, cudaStream_t>, HostStage> g_stage;

}  // namespace

// Argument checks of fa_bwd, shared with the other backward entry points.
int validate_bwd_args(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                      const float* LSE, const void* dQ, const void* dK, const void* dV, int B, int H,
                      int H_kv, int S_q, int S_k, int d, float scale, int causal, int dtype) {
    int rc;
    if ((rc = check_dims(B, H, H_kv, S_q, S_k, d, dtype))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal", "must be 0 or 1");
    if ((rc = check_ptr(dO, "dO", 16)) || (rc = check_ptr(Q, "Q", 16)) || (rc = check_ptr(K, "K", 16)) ||
        (rc = check_ptr(V, "V", 16)) || (rc = check_ptr(O, "O", 16)) || (rc = check_ptr(LSE, "LSE", 4)) ||
        (rc = check_ptr(dQ, "dQ", 16)) || (rc = check_ptr(dK, "dK", 16)) || (rc = check_ptr(dV, "dV", 16)))
        return rc;
    return FA_OK;
}

int set_error(int status, const char* arg, const char* reason) { return fail(status, arg, reason); }

int key_tile_split(const Shape& s, int bn, int bm) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 148;
    }
    const int n_key_tiles = (s.S_k + bn - 1) / bn;
    const long groups = (long)s.B * s.H_kv;
    const int g = s.H / s.H_kv;
    long total = 0, most = 0;
    for (int kt = 0; kt < n_key_tiles; ++kt) {
        int lo, hi;
        query_range(s, kt * bn, kt * bn + bn < s.S_k ? kt * bn + bn : s.S_k, lo, hi);
        const long its = hi > lo ? (long)g * ((hi + bm - 1) / bm - lo / bm) : 0;
        total += its * groups;
        most = its > most ? its : most;
    }
    // a grid of fewer CTAs than SMs is not split: clusters of two CTAs that each fill an SM
    // fit about 72 pairs at a time, so the halves ran in two waves (measured: the causal
    // S = 1024, d = 64 workload went from 24 to 33 us)
    if ((long)n_key_tiles * groups < sms) return 1;
    return (double)most > 1.05 * (double)total / sms ? 2 : 1;
}

int bwd_kernel_for(int dtype, int d) {
    if (dtype == FA_F32 || use_simt_for_16bit()) return kBwdSimt;
    if (tc_head_dim(d) != 0) return kBwdSm103;
    return d == 256 ? kBwdD256 : kBwdSimt;
}

void clear_error() { g_last_error.clear(); }

}  // namespace fa

using namespace fa;

extern "C" {

int fa_bwd(const void* dO, const void* Q, const void* K, const void* V, const void* O,
           const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
           int S_k, int d, float scale, int causal, int dtype, void* stream) {
    g_last_error.clear();
    return bwd_impl(dO, Q, K, V, O, LSE, dQ, dK, dV, B, H, H_kv, S_q, S_k, d, scale, causal, 0, 0, dtype,
                    static_cast<cudaStream_t>(stream));
}

int fa_bwd_ex(const void* dO, const void* Q, const void* K, const void* V, const void* O,
              const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
              int S_k, int d, float scale, int causal, int window_size, int deterministic, int dtype,
              void* stream) {
    g_last_error.clear();
    return bwd_impl(dO, Q, K, V, O, LSE, dQ, dK, dV, B, H, H_kv, S_q, S_k, d, scale, causal, window_size,
                    deterministic, dtype, static_cast<cudaStream_t>(stream));
}

int fa_bwd_preprocess(const void* dO, const void* O, float* D, int B, int H, int S_q, int d,
                      int dtype, void* stream) {
    g_last_error.clear();
    int rc;
    if ((rc = check_dims(B, H, H, S_q, 1, d, dtype))) return rc;
    if ((rc = check_ptr(dO, "dO", 16)) || (rc = check_ptr(O, "O", 16)) || (rc = check_ptr(D, "D", 4)))
        return rc;
    const Shape s = make_shape(B, H, H, S_q, 1, d, 1.f, 0);
    cudaError_t e = launch_preprocess(dtype, dO, O, nullptr, D, nullptr, nullptr, s, S_q,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("preprocess launch", e);
    return FA_OK;
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
           int H_kv, int S_q, int S_k, int d, float scale, int causal, int dtype, void* stream) {
    g_last_error.clear();
    return fwd_impl(Q, K, V, O, LSE, B, H, H_kv, S_q, S_k, d, scale, causal, 0, dtype,
                    static_cast<cudaStream_t>(stream));
}

int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
              int H_kv, int S_q, int S_k, int d, float scale, int causal, int window_size, int dtype,
              void* stream) {
    g_last_error.clear();
    return fwd_impl(Q, K, V, O, LSE, B, H, H_kv, S_q, S_k, d, scale, causal, window_size, dtype,
                    static_cast<cudaStream_t>(stream));
}

int fa_bwd_host(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int S_q,
                int S_k, int d, float scale, int causal, int dtype, void* stream) {
    g_last_error.clear();
    int rc;
    if ((rc = check_dims(B, H, H_kv, S_q, S_k, d, dtype))) return rc;
    if ((rc = check_ptr(dO, "dO", 1)) || (rc = check_ptr(Q, "Q", 1)) || (rc = check_ptr(K, "K", 1)) ||
        (rc = check_ptr(V, "V", 1)) || (rc = check_ptr(O, "O", 1)) || (rc = check_ptr(LSE, "LSE", 1)) ||
        (rc = check_ptr(dQ, "dQ", 1)) || (rc = check_ptr(dK, "dK", 1)) || (rc = check_ptr(dV, "dV", 1)))
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dtype);
    const int g = H / H_kv;
    // Work unit = one (batch, kv head) with its g query heads.  In every tensor the units are
    // stored one after another in (b, kv head) order, so a range of units is one contiguous
    // slice of each tensor and a backward problem of its own (B = 1, H_kv = units, H = g units).
    const size_t uq = (size_t)g * S_q * d * es;  // dO, Q, O, dQ bytes per unit
    const size_t uk = (size_t)S_k * d * es;      // K, V, dK, dV bytes per unit
    const size_t ul = (size_t)g * S_q * 4;       // LSE bytes per unit
    const int units = B * H_kv;
    const size_t nq = units * uq, nk = units * uk, nl = units * ul;
    // device layout: dO Q O dQ | K V dK dV | LSE, each 256-byte aligned
    size_t off[9], tot = 0;
    const size_t sz[9] = {nq, nq, nq, nq, nk, nk, nk, nk, nl};
    for (int i = 0; i < 9; ++i) {
        off[i] = tot;
        tot = align_up(tot + sz[i], 256);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    char* dbase = nullptr;
    HostStage* hs = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        hs = &g_stage[{dev, st}];
        if (!hs->ev_done[kHostMaxChunks - 1]) {  // created last: set once everything exists
            if ((!hs->s_in && (e = cudaStreamCreateWithFlags(&hs->s_in, cudaStreamNonBlocking)) != cudaSuccess) ||
                (!hs->s_out && (e = cudaStreamCreateWithFlags(&hs->s_out, cudaStreamNonBlocking)) != cudaSuccess))
                return cuda_fail("cudaStreamCreateWithFlags", e);
            for (int c = 0; c < kHostMaxChunks; ++c)
                if ((!hs->ev_in[c] && (e = cudaEventCreateWithFlags(&hs->ev_in[c], cudaEventDisableTiming)) != cudaSuccess) ||
                    (!hs->ev_done[c] && (e = cudaEventCreateWithFlags(&hs->ev_done[c], cudaEventDisableTiming)) != cudaSuccess))
                    return cuda_fail("cudaEventCreateWithFlags", e);
        }
        if (hs->bytes < tot) {
            if (hs->base) {
                cudaStreamSynchronize(st);
                cudaFree(hs->base);
                hs->base = nullptr;
                hs->bytes = 0;
            }
            e = cudaMalloc(&hs->base, tot);
            if (e != cudaSuccess) {
                cudaGetLastError();
                hs->base = nullptr;
                return fail(FA_ERR_NOMEM, "staging", cudaGetErrorString(e));
            }
            hs->bytes = tot;
        }
        dbase = static_cast<char*>(hs->base);
    }
    // Pipeline over chunks of units: chunk c's inputs are copied on s_in while chunk c-1 runs
    // on `stream` and chunk c-2's results are copied back on s_out.  Every chunk has its own
    // device buffers (the full-size staging above), so no chunk waits for another's copies.
    // (One stream per direction: splitting every copy over four streams per direction
    // measured slower.)
    const size_t in_bytes = 3 * nq + 2 * nk + nl;
    int n_chunks = (int)(in_bytes / kHostChunkBytes);
    n_chunks = n_chunks < 1 ? 1 : n_chunks > kHostMaxChunks ? kHostMaxChunks : n_chunks;
    if (n_chunks > units) n_chunks = units;
    const void* hin[6] = {dO, Q, O, K, V, LSE};
    const int in_slot[6] = {0, 1, 2, 4, 5, 8};
    void* hout[3] = {dQ, dK, dV};
    const int out_slot[3] = {3, 6, 7};
    auto unit_bytes = [&](int slot) { return slot < 4 ? uq : slot < 8 ? uk : ul; };
    for (int c = 0; c < n_chunks; ++c) {
        const int u0 = (int)((long)units * c / n_chunks), u1 = (int)((long)units * (c + 1) / n_chunks);
        const int nu = u1 - u0;
        for (int i = 0; i < 6; ++i) {
            const size_t ub = unit_bytes(in_slot[i]);
            e = cudaMemcpyAsync(dbase + off[in_slot[i]] + u0 * ub, static_cast<const char*>(hin[i]) + u0 * ub,
                                nu * ub, cudaMemcpyHostToDevice, hs->s_in);
            if (e != cudaSuccess) return cuda_fail("cudaMemcpyAsync H2D", e);
        }
        if ((e = cudaEventRecord(hs->ev_in[c], hs->s_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(st, hs->ev_in[c], 0)) != cudaSuccess)
            return cuda_fail("cudaEventRecord / cudaStreamWaitEvent", e);
        auto at = [&](int slot) { return dbase + off[slot] + u0 * unit_bytes(slot); };
        rc = bwd_impl(at(0), at(1), at(4), at(5), at(2), reinterpret_cast<const float*>(at(8)), at(3), at(6), at(7),
                      1, nu * g, nu, S_q, S_k, d, scale, causal, 0, 0, dtype, st);
        if (rc != FA_OK) return rc;
        if ((e = cudaEventRecord(hs->ev_done[c], st)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hs->s_out, hs->ev_done[c], 0)) != cudaSuccess)
            return cuda_fail("cudaEventRecord / cudaStreamWaitEvent", e);
        for (int i = 0; i < 3; ++i) {
            const size_t ub = unit_bytes(out_slot[i]);
            e = cudaMemcpyAsync(static_cast<char*>(hout[i]) + u0 * ub, dbase + off[out_slot[i]] + u0 * ub, nu * ub,
                                cudaMemcpyDeviceToHost, hs->s_out);
            if (e != cudaSuccess) return cuda_fail("cudaMemcpyAsync D2H", e);
        }
    }
    // s_out waited for the last chunk's compute, which waited for every input copy
    e = cudaStreamSynchronize(hs->s_out);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    return FA_OK;
}

size_t fa_bwd_workspace_bytes(int B, int H, int S_q, int d) {
    if (B <= 0 || H <= 0 || S_q <= 0 || d <= 0) return 0;
    return ws_layout(B, H, S_q, d).total;
}

int fa_check_device(void* stream) {
    g_last_error.clear();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, st});
        if (it != g_ws.end()) base = it->second.base;
    }
    unsigned int words[4] = {0, 0, 0, 0};
    if (base != nullptr) {
        e = cudaMemcpy(words, base, sizeof(words), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail("cudaMemcpy", e);
        if (words[0] != 0) {
            e = cudaMemset(base, 0, sizeof(words));
            if (e != cudaSuccess) return cuda_fail("cudaMemset", e);
        }
    }
    // fa_bwd_noalloc records its timeouts in its own scratch, shared by every stream
    unsigned int na_word = 0;
    const int rc = noalloc_take_error_word(&na_word);
    if (rc != FA_OK) return rc;
    const int status = status_from_error_words(words[0], na_word);
    if (status == FA_ERR_TIMEOUT) return fail(FA_ERR_TIMEOUT, "device", "a bounded wait in a kernel timed out");
    if (status != FA_OK)
        return fail(status, "device", "kernel error word " + std::to_string(words[0] | na_word));
    return FA_OK;
}

int fa_profile(int enable) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : g_prof_used) g_prof_free.push_back(r);
    g_prof_used.clear();
    g_prof_on = enable != 0;
    return FA_OK;
}

int fa_profile_read(float* ms, int* calls) {
    g_last_error.clear();
    if (ms == nullptr || calls == nullptr) return fail(FA_ERR_INVALID_ARG, "ms", "null pointer");
    std::lock_guard<std::mutex> lk(g_prof_mu);
    ms[0] = ms[1] = ms[2] = 0.f;
    for (auto& r : g_prof_used) {
        cudaError_t e = cudaEventSynchronize(r.ev[3]);
        if (e != cudaSuccess) return cuda_fail("cudaEventSynchronize", e);
        for (int k = 0; k < 3; ++k) {
            float t = 0.f;
            e = cudaEventElapsedTime(&t, r.ev[k], r.ev[k + 1]);
            if (e != cudaSuccess) return cuda_fail("cudaEventElapsedTime", e);
            ms[k] += t;
        }
    }
    *calls = (int)g_prof_used.size();
    return FA_OK;
}

int fa_selftest_timeout(unsigned long long limit_ns, void* stream) {
    g_last_error.clear();
    if (limit_ns == 0 || limit_ns > 1000000000ull)
        return fail(FA_ERR_INVALID_ARG, "limit_ns", "must be in (0, 1e9] nanoseconds");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    int rc = get_workspace(st, 256, &base);
    if (rc != FA_OK) return rc;
    cudaError_t e = launch_wait_selftest(static_cast<unsigned int*>(base), limit_ns, st);
    if (e != cudaSuccess) return cuda_fail("self-test launch", e);
    return FA_OK;
}

const char* fa_last_error(void) { return g_last_error.c_str(); }

void fa_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& kv : g_ws)
        if (kv.second.base) cudaFree(kv.second.base);
    g_ws.clear();
    for (auto& kv : g_stage) {
        HostStage& hs = kv.second;
        if (hs.s_in) cudaStreamSynchronize(hs.s_in);
        if (hs.s_out) cudaStreamSynchronize(hs.s_out);
        if (hs.base) cudaFree(hs.base);
        for (int c = 0; c < kHostMaxChunks; ++c) {
            if (hs.ev_in[c]) cudaEventDestroy(hs.ev_in[c]);
            if (hs.ev_done[c]) cudaEventDestroy(hs.ev_done[c]);
        }
        if (hs.s_in) cudaStreamDestroy(hs.s_in);
        if (hs.s_out) cudaStreamDestroy(hs.s_out);
    }
    g_stage.clear();
}

const char* fa_version(void) { return "fa-gb300 0.1.0 (sm_103a)"; }

}  // extern "C"
