// cssd_chunked_forward_noalloc: the chunked forward for callers that cannot
// allocate device memory at the time of the call.
//
// Some callers run under a device-memory budget that another component owns
// outright (for example a host framework whose caching allocator has reserved
// the device heap, or an embedding runtime that forbids allocation after
// start-up), and some must never block on an allocator on a latency-critical
// path.  They cannot hand the forward a workspace of their own, and the
// ordinary entry point would otherwise allocate one with cudaMallocAsync.
// This entry point instead runs the same kernels on a fixed scratch array that
// is part of the library's device image (kNoAllocScratchBytes below), so the
// call itself allocates nothing.
//
// Properties a caller must know:
//   - Every device that loads this library holds the array until the process
//     exits, whether or not this entry point is ever called.
//   - The first call on a device looks up the array's device address (with
//     that device made current for the lookup) and caches it; that set-up
//     allocates nothing but is a runtime call, so make the first call on each
//     device before any stream capture.
//   - All calls share the one array and it keeps the last call's contents.
//     The kernels clear everything that must start at zero on every call, but
//     two calls whose executions overlap on the GPU (different streams, or
//     different host threads) race on it: serialise them.
//   - Sizes whose workspace exceeds the array return CSSD_ERR_WORKSPACE
//     without launching anything.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/cssd.h"
#include "cssd_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 128;  // the bound the library's other per-device caches use

// The scratch array.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `dev`, looked up once per device
// with that device current (the caller's current device is restored).
int scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return CSSD_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) return CSSD_ERR_CUDA;
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return CSSD_ERR_CUDA;
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (prev != dev) cudaSetDevice(prev);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CSSD_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CSSD_OK;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool device_pointer_on(const void* p, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

}  // namespace

extern "C" int cssd_chunked_forward_noalloc(const cssd_dims* d, const void* x, const float* dt, const void* A,
                                            const void* B, const void* C, const float* D, void* y, void* h_final,
                                            int chunk, cssd_stream_t stream_) {
    if (!d) return CSSD_ERR_NULL;
    if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->dstate <= 0 || d->headdim <= 0) return CSSD_ERR_DIMS;
    const int64_t N = d->dstate, P = d->headdim;
    if (!(N == 16 || N == 32 || N == 64 || N == 128) || !(P == 16 || P == 32 || P == 64) ||
        !(chunk == 64 || chunk == 128))
        return CSSD_ERR_UNSUPPORTED;
    if (d->batch > 65535 || d->nheads > 65535 || d->seqlen > 2147483647LL ||
        d->batch * d->nheads > 2147483647LL || (d->seqlen + 63) / 64 > 2147483647LL / (d->batch * d->nheads))
        return CSSD_ERR_DIMS;
    if (!x || !dt || !A || !B || !C || !D || !y) return CSSD_ERR_NULL;
    if (!is_aligned(x, 16) || !is_aligned(B, 16) || !is_aligned(C, 16) || !is_aligned(y, 16) ||
        (h_final && !is_aligned(h_final, 16)) || !is_aligned(A, 8) || !is_aligned(dt, 4) || !is_aligned(D, 4))
        return CSSD_ERR_ALIGN;
    const size_t need = cssd::forward_workspace_bytes(d->batch, d->seqlen, d->nheads, N, P, chunk);
    if (need > kNoAllocScratchBytes) return CSSD_ERR_WORKSPACE;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if (cssd::stream_device_of(stream, &dev) != cudaSuccess) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    const void* ptrs[] = {x, dt, A, B, C, D, y, h_final};
    for (const void* p : ptrs)
        if (p && !device_pointer_on(p, dev)) return CSSD_ERR_DEVICE;
    void* scratch = nullptr;
    const int s = scratch_address(dev, &scratch);
    if (s != CSSD_OK) return s;

    cssd::FwdArgs a;
    a.Bz = d->batch;
    a.T = d->seqlen;
    a.H = d->nheads;
    a.N = N;
    a.P = P;
    a.chunk = chunk;
    a.x = static_cast<const float2*>(x);
    a.dt = dt;
    a.A = static_cast<const float2*>(A);
    a.B = static_cast<const float2*>(B);
    a.C = static_cast<const float2*>(C);
    a.D = D;
    a.y = static_cast<float2*>(y);
    a.h_final = static_cast<float2*>(h_final);
    return cssd::launch_forward(a, scratch, stream) == cudaSuccess ? CSSD_OK : CSSD_ERR_CUDA;
}
