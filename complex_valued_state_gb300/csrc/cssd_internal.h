// Launchers behind the C ABI (host side).  Arguments are validated by the
// entry points in cssd_api.cu before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/cssd.h"

namespace cssd {

// Device a stream belongs to, also while the stream is being captured into a
// CUDA graph: cudaStreamGetDevice is not permitted then, and work captured on
// a stream runs on the current device, which is what is returned.
inline cudaError_t stream_device_of(cudaStream_t s, int* dev) {
    if (s == nullptr) return cudaGetDevice(dev);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return e;
    if (cap != cudaStreamCaptureStatusNone) return cudaGetDevice(dev);
    return cudaStreamGetDevice(s, dev);
}

// Index and sign modes of a forward run, honoured by the tensor-core path only
// (the backward runs its adjoint recurrences through them instead of copying
// reversed or conjugated inputs).
constexpr unsigned kFwdReverse = 1u;   // token tau of the run reads and writes original token T - 1 - tau
constexpr unsigned kFwdShiftDt = 2u;   // with kFwdReverse: the step of token tau is that of original token
                                       // T - tau (none at tau = 0)
constexpr unsigned kFwdConjX = 4u;     // conj(x), also in the skip term
constexpr unsigned kFwdConjB = 8u;     // conj(B)
constexpr unsigned kFwdConjC = 16u;    // conj(C)
constexpr unsigned kFwdConjY = 32u;    // the output is conjugated
constexpr unsigned kFwdConjA = 64u;    // rate conj(A)
constexpr unsigned kFwdDump = 128u;    // write every published chunk state and its rotation (dump, rot_dump)

struct FwdArgs {
    int64_t Bz, T, H, N, P;
    int chunk;
    const float2* x;
    const float* dt;
    const float2* A;
    const float2* B;
    const float2* C;
    const float* D;
    float2* y;
    float2* h_final;             // may be null
    const float2* h0 = nullptr;  // state before the first token [Bz,H,N,P]; null = zero
    // Tensor-core path only: split-precision operands (each value as two half
    // parts, three products per product, about fp32 accuracy, one CTA per SM).
    bool split_operands = false;
    // Tensor-core path only: plain TF32 operands on every tensor-core shape
    // (dstate 64 otherwise runs half operands with per-tile scales).
    bool tf32_operands = false;
    unsigned mode = 0;  // kFwd* bits (tensor-core path only); D may be null (no skip) when set
    // kFwdDump (dstate = headdim = 64): the state chunk c hands to chunk c + 1,
    // in the rotated frame, at dump[(bh * (nc + 1) + c + 1) * 2 * 64 * 64 +
    // part * 64 * 64 + n * 64 + p] (part 0 real, 1 imaginary; nc = 64-token
    // chunks), and (cos, sin) of that frame's angle at
    // rot_dump[bh * (nc + 1) + c + 1].
    float* dump = nullptr;
    float2* rot_dump = nullptr;
};

struct StepArgs {
    int64_t Bz, H, N, P;
    int64_t nsteps = -1;  // < 0: one ordinary step; >= 0: that many steps of a constant input, in closed form
    float2* h;
    const float2* x;
    const float* dt;
    const float2* A;
    const float2* B;
    const float2* C;
    const float* D;
    float2* y;
};

// The library's device status word on the current device (null if its address
// cannot be had): kernels whose bounded waits give up OR a kStatus* bit into it,
// and cssd_device_status reads and clears it.
constexpr unsigned kStatusHandoff = 1u;   // chunk kernel: a state hand-off wait gave up
constexpr unsigned kStatusChunkMma = 2u;  // chunk kernel: a tensor-core completion wait gave up
constexpr unsigned kStatusBornMma = 4u;   // Born attention: a tensor-core completion wait gave up
unsigned* status_word();

// Events the forward records around its dominant kernel (null = off); set by
// cssd_profile_events for the calling host thread.
extern thread_local cudaEvent_t g_prof_begin;
extern thread_local cudaEvent_t g_prof_end;

// The chunked forward: the fused tensor-core kernel where its shape applies
// (headdim 64, dstate 64 or 128; split-precision operands when
// FwdArgs::split_operands, dstate 64 only), else the CUDA-core chunk kernels.
size_t forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk);
size_t forward_precise_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk);
int forward_launches(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk);
cudaError_t launch_forward(const FwdArgs& a, void* workspace, cudaStream_t stream);

// CUDA-core chunk kernels (forward_seq.cu).
size_t seq_forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk);
cudaError_t launch_seq_forward(const FwdArgs& a, void* workspace, cudaStream_t stream);

// Fused tensor-core kernel (forward_tc.cu).
bool tc_forward_supported(int64_t N, int64_t P, int chunk);
// The unpadded shapes (headdim 64, dstate 64 or 128): split precision, TF32
// operands and the index and sign modes need them; the other tensor-core
// shapes (dstate and headdim up to 64) run the half-operand kernel, padded.
bool tc_full_shape(int64_t N, int64_t P);
// Launches of one tensor-core forward: the prep (one kernel, or two for
// sequences of more than 64 chunks) and the chunk kernel.
int tc_forward_launches(int64_t T);
size_t tc_forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N);
cudaError_t launch_tc_forward(const FwdArgs& a, void* workspace, cudaStream_t stream);
cudaError_t tc_selftest_handoff_timeout(long long wait_cycles, int* err_bits, cudaStream_t stream);

// Decode step (step.cu).
struct CayleyArgs {
    int64_t Bz, T, H, N;
    const float* phi;
    const float* u;
    const float2* b;
    const float2* C;
    const float2* psi0;  // may be null (zero state)
    float2* y;
    float2* psi_final;   // may be null
    int chunk;
    float log_clamp;     // -inf: the recurrence step by step; finite: the clamped chunked scan
};

struct BornArgs {
    int64_t Bz, T, H, D;
    const float2* q;
    const float2* k;
    const float2* v;
    float2* psi;
};

cudaError_t launch_step(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_cayley_scan(const CayleyArgs& a, cudaStream_t stream);
// Gradients of the forward (backward.cu).
struct BwdArgs {
    int64_t Bz, T, H, N, P;
    int chunk;
    const float2* x;
    const float* dt;
    const float2* A;
    const float2* B;
    const float2* C;
    const float* D;
    const float2* dy;
    float2* gx;
    float* gdt;
    float2* gA;
    float2* gB;
    float2* gC;
    float* gD;
};
bool backward_supported(int64_t N, int64_t P);
size_t backward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk);
cudaError_t launch_backward(const BwdArgs& a, void* workspace, cudaStream_t stream);
// Causal Born attention (born.cu).
bool born_supported(int64_t D);
cudaError_t launch_born(const BornArgs& a, cudaStream_t stream);
// Output of a constant input held forever (h is not used).
cudaError_t launch_step_infinite(const StepArgs& a, cudaStream_t stream);

}  // namespace cssd
