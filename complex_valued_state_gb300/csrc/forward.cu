// Chooses the kernels of the chunked forward by shape: the fused tensor-core
// kernels for headdim 64 with dstate 64 or 128 and, padded to 64, for dstate
// and headdim up to 64; the CUDA-core chunk kernels for dstate 128 with a
// smaller headdim, for the split-precision and TF32 entry points on the
// padded shapes, and for the split-precision entry point at dstate 128 (its
// tensor-core instance is not built).  All compute the same chunkwise
// decomposition.

#include "cssd_internal.h"

namespace cssd {

size_t forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    if (!tc_forward_supported(N, P, chunk)) return seq_forward_workspace_bytes(Bz, T, H, N, P, chunk);
    const size_t tc = tc_forward_workspace_bytes(Bz, T, H, N);
    if (tc_full_shape(N, P) && N == 64) return tc;
    // padded shapes (split precision and TF32) and dstate 128 (split precision)
    // run the CUDA-core kernels
    const size_t seq = seq_forward_workspace_bytes(Bz, T, H, N, P, chunk);
    return tc > seq ? tc : seq;
}

// The split-precision entry point at dstate 128 runs the CUDA-core kernels,
// which keep every chunk's state: N P complex values per chunk and sequence.
size_t forward_precise_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    if (N == 2 * 64) return seq_forward_workspace_bytes(Bz, T, H, N, P, chunk);
    return forward_workspace_bytes(Bz, T, H, N, P, chunk);
}

// Tensor-core path: the prep and the chunk kernel (tc_forward_launches);
// CUDA-core path: chunk states, scan, readout.
int forward_launches(int64_t, int64_t T, int64_t, int64_t N, int64_t P, int chunk) {
    return tc_forward_supported(N, P, chunk) ? tc_forward_launches(T) : 3;
}

cudaError_t launch_forward(const FwdArgs& a, void* ws, cudaStream_t st) {
    const bool plain = a.mode == 0 && !a.split_operands && !a.tf32_operands;
    const bool tc_split = !a.split_operands || a.N == 64;  // split precision is built for dstate 64 only
    if (tc_forward_supported(a.N, a.P, a.chunk) && ((tc_full_shape(a.N, a.P) && tc_split) || plain))
        return launch_tc_forward(a, ws, st);
    if (a.mode != 0) return cudaErrorInvalidValue;  // index and sign modes: tensor-core path only
    return launch_seq_forward(a, ws, st);
}

}  // namespace cssd
