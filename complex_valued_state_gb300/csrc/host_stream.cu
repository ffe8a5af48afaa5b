// cssd_chunked_forward_host: the chunked forward over host-resident tensors,
// streamed through the device in pieces of whole tokens.
//
// Piece k covers tokens [k Tp, min((k + 1) Tp, T)) of every sequence.  Its
// inputs are copied into one of two device slots on an input stream, the
// forward runs on the caller's stream started from the state piece k - 1 left
// (the initial-state form of the chunked forward, so the pieces together equal
// one forward over the whole sequence), and its output is copied back on an
// output stream.  Slot k mod 2 is refilled only after piece k - 2's output has
// left it, so copies in both directions overlap the compute of the neighbouring
// pieces.  The host link moves ~210 GB/s host-to-device and ~190 GB/s back on
// GB300, far below HBM, so the overlap, not the kernels, sets the end-to-end
// rate.

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/cssd.h"
#include "cssd_internal.h"

namespace {

constexpr size_t kPieceTargetBytes = 48ull << 20;  // inputs per piece when the caller does not choose
constexpr int kMaxDevices = 128;

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

bool sizes_ok(const cssd_dims* d, int chunk) {
    if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0) return false;
    if (!(d->dstate == 16 || d->dstate == 32 || d->dstate == 64 || d->dstate == 128)) return false;
    if (!(d->headdim == 16 || d->headdim == 32 || d->headdim == 64)) return false;
    if (!(chunk == 64 || chunk == 128)) return false;
    return d->batch <= 65535 && d->nheads <= 65535 && d->seqlen <= 2147483647LL &&
           d->batch * d->nheads <= 2147483647LL &&
           (d->seqlen + 63) / 64 <= 2147483647LL / (d->batch * d->nheads);  // 32-bit tile index
}

// Device memory of one call: A and D, two state buffers, the forward
// workspace of one piece, and two slots each holding one piece's x, dt, B, C
// and y (dense [batch, piece, nheads, .] arrays).
struct Layout {
    int64_t Tp = 0;  // tokens per piece
    size_t x = 0, dt = 0, bc = 0, y = 0;  // bytes of one full piece's arrays
    size_t off_A = 0, off_D = 0, off_h[2] = {0, 0}, off_ws = 0, off_slot[2] = {0, 0};
    size_t ws = 0, state = 0, total = 0;
};

Layout make_layout(const cssd_dims* d, int chunk, int64_t piece_len) {
    Layout L;
    const int64_t Bz = d->batch, T = d->seqlen, H = d->nheads, N = d->dstate, P = d->headdim;
    const size_t per_token = (size_t)(Bz * H) * (size_t)(8 * P + 4 + 16 * N);
    if (piece_len > 0) {
        L.Tp = piece_len < T ? piece_len : T;
    } else {
        int64_t t = (int64_t)(kPieceTargetBytes / per_token) / chunk * chunk;
        if (t < chunk) t = chunk;
        L.Tp = t < T ? t : T;
    }
    const size_t rows = (size_t)(Bz * L.Tp * H);
    L.x = rows * (size_t)P * 8;
    L.dt = rows * 4;
    L.bc = rows * (size_t)N * 8;
    L.y = rows * (size_t)P * 8;
    L.state = (size_t)(Bz * H) * (size_t)(N * P) * 8;
    L.ws = cssd::forward_workspace_bytes(Bz, L.Tp, H, N, P, chunk);
    size_t off = 0;
    L.off_A = off;
    off += up256((size_t)H * 8);
    L.off_D = off;
    off += up256((size_t)H * 4);
    for (int i = 0; i < 2; ++i) {
        L.off_h[i] = off;
        off += up256(L.state);
    }
    L.off_ws = off;
    off += up256(L.ws);
    const size_t slot = up256(L.x) + up256(L.dt) + 2 * up256(L.bc) + up256(L.y);
    for (int i = 0; i < 2; ++i) {
        L.off_slot[i] = off;
        off += slot;
    }
    L.total = off;
    return L;
}

// Two non-blocking copy streams per device, created on first use and kept for
// the life of the process (calls from several host threads share them; every
// ordering between calls goes through events, so sharing only serialises
// their copies).
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_streams[kMaxDevices];
std::mutex g_streams_mu;

cudaError_t copy_streams(int dev, CopyStreams* cs) {
    std::lock_guard<std::mutex> lock(g_streams_mu);
    CopyStreams& s = g_streams[dev];
    if (!s.in) {
        cudaError_t e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
        e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            cudaStreamDestroy(s.in);
            s.in = nullptr;
            return e;
        }
    }
    *cs = s;
    return cudaSuccess;
}

// Rows [t0, t0 + tk) of every batch row of a host [Bz, T, H, w] array, as a
// dense [Bz, tk, H, w] device array (or back): one strided copy.
cudaError_t copy_rows_in(void* dst, const void* src, size_t row_bytes, int64_t Bz, int64_t T, int64_t H,
                         int64_t t0, int64_t tk, cudaStream_t s) {
    const size_t width = (size_t)(tk * H) * row_bytes;
    return cudaMemcpy2DAsync(dst, width, static_cast<const char*>(src) + (size_t)(t0 * H) * row_bytes,
                             (size_t)(T * H) * row_bytes, width, (size_t)Bz, cudaMemcpyDefault, s);
}
cudaError_t copy_rows_out(void* dst, const void* src, size_t row_bytes, int64_t Bz, int64_t T, int64_t H,
                          int64_t t0, int64_t tk, cudaStream_t s) {
    const size_t width = (size_t)(tk * H) * row_bytes;
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + (size_t)(t0 * H) * row_bytes, (size_t)(T * H) * row_bytes,
                             src, width, width, (size_t)Bz, cudaMemcpyDefault, s);
}

// Restores the calling thread's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" {

size_t cssd_host_forward_device_bytes(const cssd_dims* d, int chunk, int64_t piece_len) {
    if (!d || !sizes_ok(d, chunk) || piece_len < 0) return 0;
    return make_layout(d, chunk, piece_len).total;
}

int cssd_chunked_forward_host(const cssd_dims* d, const void* x, const float* dt, const void* A, const void* B,
                              const void* C, const float* D, const void* h0, void* y, void* h_final, int chunk,
                              int64_t piece_len, void* device_buffer, size_t device_bytes, cssd_stream_t stream_) {
    if (!d) return CSSD_ERR_NULL;
    if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->dstate <= 0 || d->headdim <= 0 || piece_len < 0)
        return CSSD_ERR_DIMS;
    if (!sizes_ok(d, chunk)) {
        if (d->batch > 65535 || d->nheads > 65535 || d->seqlen > 2147483647LL ||
            d->batch * d->nheads > 2147483647LL || (d->seqlen + 63) / 64 > 2147483647LL / (d->batch * d->nheads))
            return CSSD_ERR_DIMS;
        return CSSD_ERR_UNSUPPORTED;
    }
    if (!x || !dt || !A || !B || !C || !D || !y) return CSSD_ERR_NULL;
    if (device_buffer && (reinterpret_cast<uintptr_t>(device_buffer) & 255) != 0) return CSSD_ERR_ALIGN;
    const Layout L = make_layout(d, chunk, piece_len);
    if (device_buffer && device_bytes < L.total) return CSSD_ERR_WORKSPACE;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if (cssd::stream_device_of(stream, &dev) != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    if (device_buffer) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, device_buffer) != cudaSuccess) {
            cudaGetLastError();
            return CSSD_ERR_DEVICE;
        }
        if (!(at.type == cudaMemoryTypeManaged || (at.type == cudaMemoryTypeDevice && at.device == dev)))
            return CSSD_ERR_DEVICE;
    }
    DeviceGuard guard(dev);
    CopyStreams cs;
    if (copy_streams(dev, &cs) != cudaSuccess) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    unsigned char* buf = static_cast<unsigned char*>(device_buffer);
    if (!buf) {
        if (cudaMallocAsync(reinterpret_cast<void**>(&buf), L.total, stream) != cudaSuccess) {
            cudaGetLastError();
            return CSSD_ERR_WORKSPACE;
        }
    }

    // events: start, per slot inputs-in / computed / output-out, end
    cudaEvent_t ev[8] = {};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    cudaEvent_t ev_start = ev[0], ev_end = ev[7];
    cudaEvent_t* ev_in = ev + 1;    // [2]
    cudaEvent_t* ev_done = ev + 3;  // [2]
    cudaEvent_t* ev_free = ev + 5;  // [2]

    const int64_t Bz = d->batch, T = d->seqlen, H = d->nheads, N = d->dstate, P = d->headdim;
    float2* A_d = reinterpret_cast<float2*>(buf + L.off_A);
    float* D_d = reinterpret_cast<float*>(buf + L.off_D);
    float2* hbuf[2] = {reinterpret_cast<float2*>(buf + L.off_h[0]), reinterpret_cast<float2*>(buf + L.off_h[1])};
    void* ws = buf + L.off_ws;
    auto slot_ptr = [&](int s, int which) -> unsigned char* {  // 0 x, 1 dt, 2 B, 3 C, 4 y
        size_t off = L.off_slot[s];
        const size_t sizes[5] = {up256(L.x), up256(L.dt), up256(L.bc), up256(L.bc), up256(L.y)};
        for (int i = 0; i < which; ++i) off += sizes[i];
        return buf + off;
    };

    if (e == cudaSuccess) e = cudaEventRecord(ev_start, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_start, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(A_d, A, (size_t)H * 8, cudaMemcpyDefault, cs.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(D_d, D, (size_t)H * 4, cudaMemcpyDefault, cs.in);
    if (e == cudaSuccess && h0) e = cudaMemcpyAsync(hbuf[1], h0, L.state, cudaMemcpyDefault, cs.in);

    const int64_t npieces = (T + L.Tp - 1) / L.Tp;
    for (int64_t k = 0; k < npieces && e == cudaSuccess; ++k) {
        const int s = (int)(k & 1);
        const int64_t t0 = k * L.Tp, tk = (T - t0 < L.Tp) ? T - t0 : L.Tp;
        // inputs of piece k into slot s, once piece k - 2 has left it
        if (k >= 2) e = cudaStreamWaitEvent(cs.in, ev_free[s], 0);
        if (e == cudaSuccess) e = copy_rows_in(slot_ptr(s, 0), x, (size_t)P * 8, Bz, T, H, t0, tk, cs.in);
        if (e == cudaSuccess) e = copy_rows_in(slot_ptr(s, 1), dt, 4, Bz, T, H, t0, tk, cs.in);
        if (e == cudaSuccess) e = copy_rows_in(slot_ptr(s, 2), B, (size_t)N * 8, Bz, T, H, t0, tk, cs.in);
        if (e == cudaSuccess) e = copy_rows_in(slot_ptr(s, 3), C, (size_t)N * 8, Bz, T, H, t0, tk, cs.in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[s], cs.in);
        // the forward of piece k, continuing from the state of piece k - 1
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev_in[s], 0);
        if (e == cudaSuccess) {
            cssd::FwdArgs a;
            a.Bz = Bz;
            a.T = tk;
            a.H = H;
            a.N = N;
            a.P = P;
            a.chunk = chunk;
            a.x = reinterpret_cast<const float2*>(slot_ptr(s, 0));
            a.dt = reinterpret_cast<const float*>(slot_ptr(s, 1));
            a.A = A_d;
            a.B = reinterpret_cast<const float2*>(slot_ptr(s, 2));
            a.C = reinterpret_cast<const float2*>(slot_ptr(s, 3));
            a.D = D_d;
            a.y = reinterpret_cast<float2*>(slot_ptr(s, 4));
            a.h_final = hbuf[k & 1];
            a.h0 = (k == 0) ? (h0 ? hbuf[1] : nullptr) : hbuf[(k - 1) & 1];
            e = cssd::launch_forward(a, ws, stream);
        }
        if (e == cudaSuccess) e = cudaEventRecord(ev_done[s], stream);
        // its output back to the host
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_done[s], 0);
        if (e == cudaSuccess) e = copy_rows_out(y, slot_ptr(s, 4), (size_t)P * 8, Bz, T, H, t0, tk, cs.out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_free[s], cs.out);
    }
    if (e == cudaSuccess && h_final)
        e = cudaMemcpyAsync(h_final, hbuf[(npieces - 1) & 1], L.state, cudaMemcpyDefault, cs.out);
    // Whatever happened above, `stream` waits for everything already queued on
    // both copy streams before its next work (and before the buffer can be
    // released).  ev_start is reused for the input stream: the waits above
    // have captured its first record.
    if (ev_start && ev_end) {
        const cudaError_t e_in = cudaEventRecord(ev_start, cs.in);
        const cudaError_t e_out = cudaEventRecord(ev_end, cs.out);
        const cudaError_t w_in = e_in == cudaSuccess ? cudaStreamWaitEvent(stream, ev_start, 0) : e_in;
        const cudaError_t w_out = e_out == cudaSuccess ? cudaStreamWaitEvent(stream, ev_end, 0) : e_out;
        if (e == cudaSuccess) e = w_in != cudaSuccess ? w_in : w_out;
    }
    if (!device_buffer) cudaFreeAsync(buf, stream);
    for (int i = 0; i < 8; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);  // released once the work that uses them completes
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CSSD_ERR_CUDA;
    }
    return CSSD_OK;
}

}  // extern "C"
