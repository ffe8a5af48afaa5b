// C ABI entry points of libcssd: argument validation on the host, workspace
// handling, and the launches.  See include/cssd.h for the contract.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/cssd.h"
#include "cssd_internal.h"

namespace {

bool supported_n(int64_t n) { return n == 16 || n == 32 || n == 64 || n == 128; }
bool supported_p(int64_t p) { return p == 16 || p == 32 || p == 64; }
bool supported_chunk(int c) { return c == 64 || c == 128; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxGridYZ = 65535;
constexpr int64_t kMaxInt = 2147483647;

int check_dims(const cssd_dims* d, bool need_seq) {
    if (!d) return CSSD_ERR_NULL;
    if (d->batch <= 0 || d->nheads <= 0 || d->dstate <= 0 || d->headdim <= 0) return CSSD_ERR_DIMS;
    if (need_seq && d->seqlen <= 0) return CSSD_ERR_DIMS;
    if (!supported_n(d->dstate) || !supported_p(d->headdim)) return CSSD_ERR_UNSUPPORTED;
    if (d->batch > kMaxGridYZ || d->nheads > kMaxGridYZ) return CSSD_ERR_DIMS;
    if (d->batch * d->nheads > kMaxInt) return CSSD_ERR_DIMS;
    if (need_seq && d->seqlen > kMaxInt) return CSSD_ERR_DIMS;
    // the chunk kernels index (batch, head, 64-token tile) in 32 bits
    if (need_seq && (d->seqlen + 63) / 64 > kMaxInt / (d->batch * d->nheads)) return CSSD_ERR_DIMS;
    return CSSD_OK;
}

// Device of the stream (or the current device for the default stream).
int stream_device(cudaStream_t s, int* dev) {
    if (s == nullptr) return cudaGetDevice(dev) == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
    return cssd::stream_device_of(s, dev) == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}

// The pointer must be device (or managed) memory usable on `dev`.
int check_device_ptr(const void* p, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error this query may set
        return CSSD_ERR_DEVICE;
    }
    if (at.type == cudaMemoryTypeManaged) return CSSD_OK;
    if (at.type != cudaMemoryTypeDevice || at.device != dev) return CSSD_ERR_DEVICE;
    return CSSD_OK;
}

template <typename... Ts>
int check_all_device(int dev, Ts... ptrs) {
    const void* arr[] = {ptrs...};
    for (const void* p : arr) {
        if (!p) continue;
        const int s = check_device_ptr(p, dev);
        if (s != CSSD_OK) return s;
    }
    return CSSD_OK;
}

}  // namespace

namespace cssd {
// Measurement hook: events recorded around the dominant kernel of the next
// forward calls made from this host thread (both NULL = off).
thread_local cudaEvent_t g_prof_begin = nullptr;
thread_local cudaEvent_t g_prof_end = nullptr;
}  // namespace cssd

namespace {
__device__ unsigned g_status_word;  // one per device that loads the library; starts at 0
constexpr int kMaxStatusDevices = 128;
unsigned* g_status_ptr[kMaxStatusDevices] = {};
std::mutex g_status_mu;
}  // namespace

namespace cssd {
unsigned* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStatusDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<unsigned*>(q);
    }
    return g_status_ptr[dev];
}
}  // namespace cssd

namespace {
// Shared argument checks and launch of cssd_step (nsteps < 0), cssd_step_n
// (nsteps >= 0) and cssd_step_infinite (no state: with_h = false).
int step_common(const cssd_dims* d, void* h, const void* x, const float* dt, const void* A, const void* B,
                       const void* C, const float* D, void* y, int64_t nsteps, bool with_h, cssd_stream_t stream_) {
    int s = check_dims(d, false);
    if (s != CSSD_OK) return s;
    if ((with_h && !h) || !x || !dt || !A || !B || !C || !D || !y) return CSSD_ERR_NULL;
    if ((with_h && !aligned(h, 16)) || !aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) ||
        !aligned(A, 8) || !aligned(dt, 4) || !aligned(D, 4))
        return CSSD_ERR_ALIGN;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if ((s = stream_device(stream, &dev)) != CSSD_OK) return s;
    if ((s = check_all_device(dev, (const void*)h, x, (const void*)dt, A, B, C, (const void*)D, (const void*)y)) !=
        CSSD_OK)
        return s;
    cssd::StepArgs a;
    a.Bz = d->batch;
    a.H = d->nheads;
    a.N = d->dstate;
    a.P = d->headdim;
    a.nsteps = nsteps;
    a.h = static_cast<float2*>(h);
    a.x = static_cast<const float2*>(x);
    a.dt = dt;
    a.A = static_cast<const float2*>(A);
    a.B = static_cast<const float2*>(B);
    a.C = static_cast<const float2*>(C);
    a.D = D;
    a.y = static_cast<float2*>(y);
    const cudaError_t e = with_h ? cssd::launch_step(a, stream) : cssd::launch_step_infinite(a, stream);
    return e == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}
// Shared checks and launch of cssd_chunked_forward (h0 == NULL) and
// cssd_chunked_forward_h0.
int forward_common(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B, const void* C,
                   const float* D, const void* h0, void* y, void* h_final, int chunk, void* workspace,
                   size_t workspace_bytes, cssd_stream_t stream_, bool precise = false, bool tf32 = false) {
    int s = check_dims(d, true);
    if (s != CSSD_OK) return s;
    if (!supported_chunk(chunk)) return CSSD_ERR_UNSUPPORTED;
    if (!x || !dt || !A || !B || !C || !D || !y) return CSSD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) ||
        (h_final && !aligned(h_final, 16)) || (h0 && !aligned(h0, 16)) || (workspace && !aligned(workspace, 16)) ||
        !aligned(A, 8) || !aligned(dt, 4) || !aligned(D, 4))
        return CSSD_ERR_ALIGN;
    const size_t need =
        precise ? cssd::forward_precise_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk)
                : cssd::forward_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
    if (workspace && workspace_bytes < need) return CSSD_ERR_WORKSPACE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if ((s = stream_device(stream, &dev)) != CSSD_OK) return s;
    if ((s = check_all_device(dev, x, (const void*)dt, A, B, C, (const void*)D, h0, (const void*)y,
                              (const void*)h_final, (const void*)workspace)) != CSSD_OK)
        return s;

    void* ws = workspace;
    if (!ws) {
        if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) {
            cudaGetLastError();
            return CSSD_ERR_WORKSPACE;
        }
    }
    cssd::FwdArgs a;
    a.Bz = d->batch;
    a.T = d->seqlen;
    a.H = d->nheads;
    a.N = d->dstate;
    a.P = d->headdim;
    a.chunk = chunk;
    a.x = static_cast<const float2*>(x);
    a.dt = dt;
    a.A = static_cast<const float2*>(A);
    a.B = static_cast<const float2*>(B);
    a.C = static_cast<const float2*>(C);
    a.D = D;
    a.y = static_cast<float2*>(y);
    a.h_final = static_cast<float2*>(h_final);
    a.h0 = static_cast<const float2*>(h0);
    a.split_operands = precise;
    a.tf32_operands = tf32;
    const cudaError_t e = cssd::launch_forward(a, ws, stream);
    if (!workspace) cudaFreeAsync(ws, stream);
    return e == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}

}  // namespace

extern "C" {

int cssd_profile_events(void* ev_begin, void* ev_end) {
    if ((ev_begin == nullptr) != (ev_end == nullptr)) return CSSD_ERR_NULL;
    cssd::g_prof_begin = static_cast<cudaEvent_t>(ev_begin);
    cssd::g_prof_end = static_cast<cudaEvent_t>(ev_end);
    return CSSD_OK;
}

int cssd_selftest_handoff_timeout(long long wait_cycles, int* err_bits, cssd_stream_t stream) {
    if (!err_bits) return CSSD_ERR_NULL;
    if (wait_cycles <= 0) return CSSD_ERR_DIMS;
    const cudaError_t e =
        cssd::tc_selftest_handoff_timeout(wait_cycles, err_bits, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    return CSSD_OK;
}

int cssd_device_status(unsigned* bits, int clear, cssd_stream_t stream_) {
    if (!bits) return CSSD_ERR_NULL;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if (stream_device(stream, &dev) != CSSD_OK) return CSSD_ERR_CUDA;
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != dev) {
        cudaGetLastError();
        return CSSD_ERR_DEVICE;
    }
    unsigned* w = cssd::status_word();
    if (!w) return CSSD_ERR_CUDA;
    unsigned v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, w, sizeof(unsigned), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(w, 0, sizeof(unsigned), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    *bits = v;
    return CSSD_OK;
}

const char* cssd_status_string(int status) {
    switch (status) {
        case CSSD_OK: return "ok";
        case CSSD_ERR_NULL: return "a required pointer is NULL";
        case CSSD_ERR_DIMS: return "a size is zero, negative or too large";
        case CSSD_ERR_UNSUPPORTED: return "dstate, headdim or chunk outside the supported set";
        case CSSD_ERR_ALIGN: return "a pointer breaks the alignment rule";
        case CSSD_ERR_WORKSPACE: return "workspace too small or its allocation failed";
        case CSSD_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case CSSD_ERR_DEVICE: return "a pointer is not device memory of the stream's device";
    }
    return "unknown status";
}

size_t cssd_workspace_bytes(const cssd_dims* d, int chunk) {
    if (check_dims(d, true) != CSSD_OK || !supported_chunk(chunk)) return 0;
    return cssd::forward_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
}

size_t cssd_precise_workspace_bytes(const cssd_dims* d, int chunk) {
    if (check_dims(d, true) != CSSD_OK || !supported_chunk(chunk)) return 0;
    return cssd::forward_precise_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
}

int cssd_forward_launches(const cssd_dims* d, int chunk) {
    if (check_dims(d, true) != CSSD_OK || !supported_chunk(chunk)) return 0;
    return cssd::forward_launches(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
}

int cssd_chunked_forward(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                         const void* C, const float* D, void* y, void* h_final, int chunk, void* workspace,
                         size_t workspace_bytes, cssd_stream_t stream_) {
    return forward_common(d, x, dt, A, B, C, D, nullptr, y, h_final, chunk, workspace, workspace_bytes, stream_);
}

int cssd_chunked_forward_h0(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                            const void* C, const float* D, const void* h0, void* y, void* h_final, int chunk,
                            void* workspace, size_t workspace_bytes, cssd_stream_t stream_) {
    return forward_common(d, x, dt, A, B, C, D, h0, y, h_final, chunk, workspace, workspace_bytes, stream_);
}

int cssd_chunked_forward_precise(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                                 const void* C, const float* D, const void* h0, void* y, void* h_final, int chunk,
                                 void* workspace, size_t workspace_bytes, cssd_stream_t stream_) {
    return forward_common(d, x, dt, A, B, C, D, h0, y, h_final, chunk, workspace, workspace_bytes, stream_, true);
}

int cssd_chunked_forward_tf32(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                              const void* C, const float* D, const void* h0, void* y, void* h_final, int chunk,
                              void* workspace, size_t workspace_bytes, cssd_stream_t stream_) {
    return forward_common(d, x, dt, A, B, C, D, h0, y, h_final, chunk, workspace, workspace_bytes, stream_, false,
                          true);
}

int cssd_step(const cssd_dims* d, void* h, const void* x, const float* dt, const void* A, const void* B,
              const void* C, const float* D, void* y, cssd_stream_t stream_) {
    return step_common(d, h, x, dt, A, B, C, D, y, -1, true, stream_);
}

int cssd_step_n(const cssd_dims* d, void* h, const void* x, const float* dt, const void* A, const void* B,
                const void* C, const float* D, int64_t nsteps, void* y, cssd_stream_t stream_) {
    if (nsteps < 0) return CSSD_ERR_DIMS;
    return step_common(d, h, x, dt, A, B, C, D, y, nsteps, true, stream_);
}

int cssd_step_infinite(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                       const void* C, const float* D, void* y, cssd_stream_t stream_) {
    return step_common(d, nullptr, x, dt, A, B, C, D, y, 0, false, stream_);
}

int cssd_cayley_scan(const cssd_dims* d, const float* phi, const float* u, const void* b, const void* C,
                     const void* psi0, void* y, void* psi_final, int chunk, float log_clamp, cssd_stream_t stream_) {
    if (!d) return CSSD_ERR_NULL;
    if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->dstate <= 0) return CSSD_ERR_DIMS;
    if (d->seqlen > kMaxInt || d->nheads * d->dstate > kMaxInt || d->batch * d->nheads * d->dstate > kMaxInt)
        return CSSD_ERR_DIMS;
    if (chunk < 1) return CSSD_ERR_DIMS;
    if (!(log_clamp == -INFINITY || (log_clamp >= -80.f && log_clamp <= 0.f))) return CSSD_ERR_DIMS;
    if (!phi || !u || !b || !C || !y) return CSSD_ERR_NULL;
    if (!aligned(phi, 4) || !aligned(u, 4) || !aligned(b, 8) || !aligned(C, 8) || !aligned(y, 8) ||
        (psi0 && !aligned(psi0, 8)) || (psi_final && !aligned(psi_final, 8)))
        return CSSD_ERR_ALIGN;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    int s = stream_device(stream, &dev);
    if (s != CSSD_OK) return s;
    if ((s = check_all_device(dev, (const void*)phi, (const void*)u, b, C, psi0, (const void*)y,
                              (const void*)psi_final)) != CSSD_OK)
        return s;
    cssd::CayleyArgs a;
    a.Bz = d->batch;
    a.T = d->seqlen;
    a.H = d->nheads;
    a.N = d->dstate;
    a.phi = phi;
    a.u = u;
    a.b = static_cast<const float2*>(b);
    a.C = static_cast<const float2*>(C);
    a.psi0 = static_cast<const float2*>(psi0);
    a.y = static_cast<float2*>(y);
    a.psi_final = static_cast<float2*>(psi_final);
    a.chunk = chunk;
    a.log_clamp = log_clamp;
    return cssd::launch_cayley_scan(a, stream) == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}

size_t cssd_backward_workspace_bytes(const cssd_dims* d, int chunk) {
    if (check_dims(d, true) != CSSD_OK || !supported_chunk(chunk) || !cssd::backward_supported(d->dstate, d->headdim))
        return 0;
    return cssd::backward_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
}

int cssd_chunked_backward(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                          const void* C, const float* D, const void* dy, void* gx, float* gdt, void* gA, void* gB,
                          void* gC, float* gD, int chunk, void* workspace, size_t workspace_bytes,
                          cssd_stream_t stream_) {
    int s = check_dims(d, true);
    if (s != CSSD_OK) return s;
    if (!supported_chunk(chunk) || !cssd::backward_supported(d->dstate, d->headdim)) return CSSD_ERR_UNSUPPORTED;
    if (!x || !dt || !A || !B || !C || !D || !dy || !gx || !gdt || !gA || !gB || !gC || !gD) return CSSD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(dy, 16) || !aligned(gx, 16) ||
        !aligned(gB, 16) || !aligned(gC, 16) || (workspace && !aligned(workspace, 16)) ||
        !aligned(A, 8) || !aligned(gA, 8) || !aligned(dt, 4) || !aligned(gdt, 4) || !aligned(D, 4) ||
        !aligned(gD, 4))
        return CSSD_ERR_ALIGN;
    const size_t need = cssd::backward_workspace_bytes(d->batch, d->seqlen, d->nheads, d->dstate, d->headdim, chunk);
    if (workspace && workspace_bytes < need) return CSSD_ERR_WORKSPACE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if ((s = stream_device(stream, &dev)) != CSSD_OK) return s;
    if ((s = check_all_device(dev, x, (const void*)dt, A, B, C, (const void*)D, dy, gx, (const void*)gdt, gA, gB,
                              gC, (const void*)gD, (const void*)workspace)) != CSSD_OK)
        return s;
    void* ws = workspace;
    if (!ws) {
        if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) {
            cudaGetLastError();
            return CSSD_ERR_WORKSPACE;
        }
    }
    cssd::BwdArgs a;
    a.Bz = d->batch;
    a.T = d->seqlen;
    a.H = d->nheads;
    a.N = d->dstate;
    a.P = d->headdim;
    a.chunk = chunk;
    a.x = static_cast<const float2*>(x);
    a.dt = dt;
    a.A = static_cast<const float2*>(A);
    a.B = static_cast<const float2*>(B);
    a.C = static_cast<const float2*>(C);
    a.D = D;
    a.dy = static_cast<const float2*>(dy);
    a.gx = static_cast<float2*>(gx);
    a.gdt = gdt;
    a.gA = static_cast<float2*>(gA);
    a.gB = static_cast<float2*>(gB);
    a.gC = static_cast<float2*>(gC);
    a.gD = gD;
    const cudaError_t e = cssd::launch_backward(a, ws, stream);
    if (!workspace) cudaFreeAsync(ws, stream);
    return e == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}

int cssd_born_attention(const cssd_dims* d, const void* q, const void* k, const void* v, void* psi,
                        cssd_stream_t stream_) {
    if (!d) return CSSD_ERR_NULL;
    if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->dstate <= 0) return CSSD_ERR_DIMS;
    if (d->seqlen > kMaxInt || d->batch * d->nheads > kMaxInt ||
        d->batch * d->nheads * ((d->seqlen + 63) / 64) > kMaxInt)
        return CSSD_ERR_DIMS;
    if (!cssd::born_supported(d->dstate)) return CSSD_ERR_UNSUPPORTED;
    if (!q || !k || !v || !psi) return CSSD_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(psi, 16)) return CSSD_ERR_ALIGN;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    int s = stream_device(stream, &dev);
    if (s != CSSD_OK) return s;
    if ((s = check_all_device(dev, q, k, v, (const void*)psi)) != CSSD_OK) return s;
    cssd::BornArgs a;
    a.Bz = d->batch;
    a.T = d->seqlen;
    a.H = d->nheads;
    a.D = d->dstate;
    a.q = static_cast<const float2*>(q);
    a.k = static_cast<const float2*>(k);
    a.v = static_cast<const float2*>(v);
    a.psi = static_cast<float2*>(psi);
    return cssd::launch_born(a, stream) == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}

}  // extern "C"
