// Chooses the kernels of the chunked forward by shape: the fused tensor-core
// kernel for headdim 64 with dstate 64 or 128, the CUDA-core chunk kernels for
// every other supported shape.  Both compute the same chunkwise decomposition.

#include "cssd_internal.h"

namespace cssd {

size_t forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    if (tc_forward_supported(N, P, chunk)) return tc_forward_workspace_bytes(Bz, T, H, N);
    return seq_forward_workspace_bytes(Bz, T, H, N, P, chunk);
}

// Tensor-core path: two prep kernels and the chunk kernel; CUDA-core path:
// chunk states, scan, readout.
int forward_launches(int64_t, int64_t, int64_t, int64_t, int64_t, int) { return 3; }

cudaError_t launch_forward(const FwdArgs& a, void* ws, cudaStream_t st) {
    if (tc_forward_supported(a.N, a.P, a.chunk)) return launch_tc_forward(a, ws, st);
    if (a.mode != 0) return cudaErrorInvalidValue;  // index and sign modes: tensor-core path only
    return launch_seq_forward(a, ws, st);
}

}  // namespace cssd
