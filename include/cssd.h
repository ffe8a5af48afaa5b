/*
 * cssd.h — C ABI of libcssd, the complex SSD (complex-valued diagonal state
 * space) forward and decode step for NVIDIA GB300 (sm_103a).
 *
 * The operation (per batch b and head h, state h_t in C^{N x P}):
 *     a_t = exp(softplus(dt_t) * A)          softplus on the real dt, then the
 *                                            complex exponential
 *     h_t = a_t h_{t-1} + B_t x_t^T          outer product, no conjugate
 *     y_t = C_t^T h_t + D x_t                readout after the update, sum over
 *                                            the N state rows, no conjugate
 * Sources: "Complex-Valued State Spaces" (Mamba-3-Lite docs), sections
 * "Discretization" and "The discretization" (the sequential loop and
 * exp(softplus(dt) A)); "SSD Theory" section 2 (the recurrence) and the
 * readout C^T h + D x of the workload statement.  The forward evaluates it in
 * the chunkwise form of "The Chunkwise Complex SSD Algorithm" sections 4.1-4.5
 * (pad, within-chunk cumsum, segment matrix, per-chunk states, inter-chunk
 * scan, output combine), with the inter-chunk state taken from the theorem of
 * "SSD Theory" section 4.5.
 *
 * Conventions shared by every entry point:
 *   - Complex numbers are complex64: interleaved [re, im] float32 pairs.
 *   - Arrays are dense and row-major with the shapes given per argument.
 *   - Every array pointer is a DEVICE pointer on the device that `stream`
 *     belongs to (the current device when stream is NULL), except in
 *     cssd_chunked_forward_host, which takes host memory.  The caller owns
 *     all memory; apart from the measurement hook cssd_profile_events and the
 *     device status word (cssd_device_status) the library keeps no state
 *     between calls.
 *   - Execution is asynchronous on `stream`.  Argument errors are detected on
 *     the host before anything is launched and leave every output untouched.
 *     A launch failure returns CSSD_ERR_CUDA.  Faults during execution surface
 *     at the caller's next synchronisation.  Nothing aborts or traps.
 *   - CUDA graphs: every device-pointer entry point except
 *     cssd_chunked_forward_noalloc (about which this note says nothing) may
 *     be called while `stream` is being captured, and the graph's replays then redo the call's
 *     work on the captured buffers.  Make one call of the same entry point on
 *     the device before the capture (it fills per-device caches of kernel
 *     attributes and occupancy), and pass a workspace where the call takes
 *     one.  cssd_chunked_forward_host, cssd_device_status and
 *     cssd_selftest_handoff_timeout wait on the host and cannot be captured.
 *   - Alignment: x, B, C, y, h, h_final and the workspace must be 16-byte
 *     aligned; A 8-byte; dt and D 4-byte.
 *   - Supported sizes: dstate N in {16, 32, 64, 128}; headdim P in {16, 32, 64};
 *     chunk in {64, 128}; seqlen >= 1 (any length; the last chunk is padded
 *     internally); batch >= 1; nheads >= 1.  Other values return
 *     CSSD_ERR_UNSUPPORTED (or CSSD_ERR_DIMS for non-positive sizes).
 *   - y must not alias any input.
 */
#ifndef CSSD_H
#define CSSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* cssd_stream_t;

typedef enum {
    CSSD_OK = 0,
    CSSD_ERR_NULL = -1,        /* a required pointer is NULL */
    CSSD_ERR_DIMS = -2,        /* a size is zero/negative or too large */
    CSSD_ERR_UNSUPPORTED = -3, /* N, P or chunk outside the supported set */
    CSSD_ERR_ALIGN = -4,       /* a pointer breaks the alignment rule */
    CSSD_ERR_WORKSPACE = -5,   /* workspace too small, or allocating it failed */
    CSSD_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
    CSSD_ERR_DEVICE = -7       /* a pointer is not device memory of the stream's device */
} cssd_status;

/* Problem sizes.  seqlen is ignored by cssd_step. */
typedef struct {
    int64_t batch;   /* Bz */
    int64_t seqlen;  /* T  */
    int64_t nheads;  /* H  */
    int64_t dstate;  /* N  (state rows) */
    int64_t headdim; /* P  (state columns, the pages' head dimension D) */
} cssd_dims;

/* Bytes of device workspace cssd_chunked_forward needs for these sizes.
 * Returns 0 when the sizes or the chunk are invalid. */
size_t cssd_workspace_bytes(const cssd_dims* dims, int chunk);

/* Bytes of device workspace cssd_chunked_forward_precise needs for these
 * sizes: cssd_workspace_bytes, except at dstate 128, where that entry point
 * runs the CUDA-core chunk kernels and keeps every chunk's state (8 dstate
 * headdim bytes per chunk and sequence).  Returns 0 when the sizes or the
 * chunk are invalid. */
size_t cssd_precise_workspace_bytes(const cssd_dims* dims, int chunk);

/* Chunkwise forward over a whole sequence from a zero initial state.
 *
 * Kernels and precision: every shape except dstate 128 with headdim 16 or 32
 * runs on the tensor cores, rounding the GEMM operands to an 11-bit
 * significand and accumulating in fp32: IEEE half operands with a
 * power-of-two scale per tile and operand (dstate and headdim up to 64, tiles
 * below 64 padded with zeros to 64; dstate 128 with headdim 64 in two 64-row
 * state halves, the carried-in state scaled per half).  Decays,
 * rotations, the inter-chunk state and the output are fp32.  Measured errors
 * are 1e-4 to 5e-4 of the largest value of y and of h_final (the bar the
 * tests hold is 2e-3).  dstate 128 with headdim 16 or 32 runs the CUDA-core
 * kernels, fp32 throughout.  cssd_chunked_forward_precise gives about fp32
 * accuracy. */
/* Arguments:
 *   x       complex64 [batch, seqlen, nheads, headdim]   token content
 *   dt      float32   [batch, seqlen, nheads]            raw step (softplus applied inside)
 *   A       complex64 [nheads]                           per-head rate
 *   B       complex64 [batch, seqlen, nheads, dstate]    input coupling
 *   C       complex64 [batch, seqlen, nheads, dstate]    readout
 *   D       float32   [nheads]                           skip, broadcast over headdim
 *   y       complex64 [batch, seqlen, nheads, headdim]   output (written)
 *   h_final complex64 [batch, nheads, dstate, headdim]   state after the last
 *           token (written); may be NULL.  It is the h that cssd_step
 *           continues from.
 *   chunk   chunk length of the decomposition (64 or 128).  The result does
 *           not depend on it beyond rounding.
 *   workspace, workspace_bytes: device scratch of at least
 *           cssd_workspace_bytes(dims, chunk) bytes, owned by the caller and
 *           not read before it is written.  With workspace == NULL the
 *           library allocates and frees it stream-ordered on `stream`
 *           (cudaMallocAsync / cudaFreeAsync).
 * Returns a cssd_status. */
int cssd_chunked_forward(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                         const void* B, const void* C, const float* D, void* y, void* h_final,
                         int chunk, void* workspace, size_t workspace_bytes, cssd_stream_t stream);

/* Number of kernel launches one cssd_chunked_forward call makes for these
 * sizes (0 when they are invalid).  Informational, for launch accounting. */
int cssd_forward_launches(const cssd_dims* dims, int chunk);

/* cssd_chunked_forward for callers that cannot allocate device memory when
 * they call it: callers whose device heap is owned outright by another
 * allocator (a host framework's caching allocator, an embedding runtime that
 * forbids allocation after start-up) or that must not wait on an allocator on
 * a latency-critical path.  The paper has no counterpart to this entry point.
 * Arguments and results are those of cssd_chunked_forward without the
 * workspace: the scratch the kernels need lives in a 16 MiB array that is
 * part of the library's device image, so the call allocates nothing.
 *   - Every device that loads the library holds those 16 MiB until exit.
 *   - Sizes whose workspace (cssd_workspace_bytes) exceeds 16 MiB return
 *     CSSD_ERR_WORKSPACE without launching.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it.
 *   - All calls share the array and it keeps the last call's contents; the
 *     kernels clear what must start at zero on every call, but calls whose
 *     executions overlap on the GPU race on it and must be serialised. */
int cssd_chunked_forward_noalloc(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                                 const void* B, const void* C, const float* D, void* y, void* h_final,
                                 int chunk, cssd_stream_t stream);

/* cssd_chunked_forward started from a given state instead of zero: h_{-1} =
 * h0 in the recurrence above.  "The Chunkwise Complex SSD Algorithm" gives its
 * inter-chunk scan an initial-states input, which the chunked form takes as the
 * state entering the first chunk; the result equals the sequential recurrence
 * started from h0.  Continuing a sequence in pieces is exact: the forward over
 * tokens [0, T) equals the forward over [0, T1) followed by this call over
 * [T1, T) with h0 = the first call's h_final.
 *   h0  complex64 [batch, nheads, dstate, headdim], device, 16-byte aligned;
 *       NULL means zero (the call is then cssd_chunked_forward).  h0 and
 *       h_final may be the same buffer (continuation in place: every state
 *       element is read before it is overwritten) but must not otherwise
 *       overlap.
 * Every other argument, the workspace size and the status are those of
 * cssd_chunked_forward. */
int cssd_chunked_forward_h0(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                            const void* B, const void* C, const float* D, const void* h0, void* y,
                            void* h_final, int chunk, void* workspace, size_t workspace_bytes,
                            cssd_stream_t stream);

/* cssd_chunked_forward_h0 to about fp32 accuracy.  The chunked form is exact
 * up to rounding, and on the tensor-core path the rounding of
 * cssd_chunked_forward is that of operands with an 11-bit significand (~1e-4
 * of the largest |y| on the pages' workloads).  Here every operand, scaled by
 * its tile's power of two, is held as two IEEE half parts hi + lo (hi = the
 * value rounded to half, lo = the remainder rounded to half) and every product
 * is taken as hi.hi + hi.lo + lo.hi, which keeps ~22 significant bits per
 * product; the decay exponentials use the accurate expf and the within-chunk
 * cumulative log-steps are summed in double.  Measured ~1e-6 of the largest
 * |y|, at about 2x the time of cssd_chunked_forward (three times the
 * tensor-core work and twice the shared memory, one CTA per SM).  Built for
 * headdim 64 with dstate 64; every other
 * shape (dstate 128, and headdim or dstate 16 / 32) runs the fp32 CUDA-core
 * chunk kernels, fp32 throughout (~1e-6 too, slower).  The workspace is
 * cssd_precise_workspace_bytes(dims, chunk) bytes.  Arguments and status are
 * otherwise those of cssd_chunked_forward_h0; h0 may be NULL. */
int cssd_chunked_forward_precise(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                                 const void* B, const void* C, const float* D, const void* h0, void* y,
                                 void* h_final, int chunk, void* workspace, size_t workspace_bytes,
                                 cssd_stream_t stream);

/* cssd_chunked_forward_h0 with the tensor-core contractions taken on TF32
 * operands (10 explicit mantissa bits, the fp32 exponent range, rounded to
 * nearest) on every tensor-core shape, accumulation fp32.  The chunked form of
 * "The Chunkwise Complex SSD Algorithm" (sections 4.3-4.5) is exact up to
 * rounding; the pages fix no operand precision for its GEMMs.
 * cssd_chunked_forward takes half operands with a power-of-two scale per tile
 * and operand (the same 11-bit significand, a narrower exponent range covered
 * by the per-tile scales); this entry point keeps TF32 at dstate 64 and 128,
 * for callers and measurements that want the wider operand exponent range
 * without per-tile scaling.  The other shapes
 * (dstate or headdim below 64, and dstate 128 with a smaller headdim) run the
 * fp32 CUDA-core chunk kernels.
 * Arguments, workspace size (cssd_workspace_bytes) and status are those of
 * cssd_chunked_forward_h0; h0 may be NULL. */
int cssd_chunked_forward_tf32(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                              const void* B, const void* C, const float* D, const void* h0, void* y,
                              void* h_final, int chunk, void* workspace, size_t workspace_bytes,
                              cssd_stream_t stream);

/* Forward over tensors that live in HOST memory, streamed through the device
 * in pieces of `piece_len` tokens: while one piece computes, the next one's
 * inputs are copied in and the previous one's output copied out, and each
 * piece continues from the state the previous piece left on the device (the
 * initial-state identity of cssd_chunked_forward_h0), so the result equals one
 * cssd_chunked_forward over the whole sequence up to rounding.  The pages have
 * no counterpart: it serves callers whose sequences are produced and consumed
 * on the host.
 *   x, dt, A, B, C, D, y, h0, h_final: shapes and meaning as in
 *       cssd_chunked_forward_h0, but any memory cudaMemcpyAsync can address:
 *       page-locked host memory (cudaHostAlloc / cudaHostRegister) for copies
 *       that overlap the compute, pageable host memory (correct, but the
 *       driver stages those copies), or device memory.  h0 and h_final may be
 *       NULL.  Inputs must stay unchanged, and outputs are not complete, until
 *       `stream` has run past this call.
 *   piece_len  tokens per piece (>= 1); 0 lets the library choose (~48 MB of
 *       inputs per piece, a multiple of chunk).
 *   device_buffer, device_bytes: device scratch of at least
 *       cssd_host_forward_device_bytes(dims, chunk, piece_len) bytes on the
 *       stream's device, 256-byte aligned; NULL makes the library allocate and
 *       free it stream-ordered on `stream`.
 * The copies run on two library-owned streams of the device that are ordered
 * after the work already on `stream`, and `stream` waits for all of them
 * before its next work, so the call behaves as one operation on `stream`.
 * Host pointers are not checked for page-locking.  Returns a cssd_status. */
size_t cssd_host_forward_device_bytes(const cssd_dims* dims, int chunk, int64_t piece_len);
int cssd_chunked_forward_host(const cssd_dims* dims, const void* x, const float* dt, const void* A,
                              const void* B, const void* C, const float* D, const void* h0, void* y,
                              void* h_final, int chunk, int64_t piece_len, void* device_buffer,
                              size_t device_bytes, cssd_stream_t stream);

/* One decode token for every (batch, head): the same recurrence, one step.
 *   h   complex64 [batch, nheads, dstate, headdim]  state, read then updated in place
 *   x   complex64 [batch, nheads, headdim]
 *   dt  float32   [batch, nheads]
 *   A   complex64 [nheads]
 *   B   complex64 [batch, nheads, dstate]
 *   C   complex64 [batch, nheads, dstate]
 *   D   float32   [nheads]
 *   y   complex64 [batch, nheads, headdim]          output (written)
 * Returns a cssd_status. */
int cssd_step(const cssd_dims* dims, void* h, const void* x, const float* dt, const void* A,
              const void* B, const void* C, const float* D, void* y, cssd_stream_t stream);

/* `nsteps` decode steps that all feed the same token (x, dt, B, C), in
 * closed form: the result equals nsteps calls of cssd_step with these inputs
 * (up to rounding), at the cost of one.  This is the constant-input shortcut
 * of "Constant-input stepping shortcuts - step_n_approx / step_infinite"
 * (burn-mamba docs, module step_constant), which there is stated for a block
 * whose input rotates each step; in this recurrence the rotation is part of
 * the complex per-step factor a = exp(softplus(dt) A), so the n steps are the
 * scalar geometric series
 *     h <- a^n h + g_n B x^T,   g_n = 1 + a + ... + a^(n-1),
 *     y  = C^T h + D x          (the output of the n-th step).
 * a^n and g_n are formed per (batch, head) in double, with the angle reduced
 * mod 2 pi, so n may be large (up to 2^53 keeps n exact).
 *   Arguments and layouts are those of cssd_step; nsteps >= 0 (0 leaves h
 *   unchanged and returns C^T h + D x).  nsteps < 0 returns CSSD_ERR_DIMS.
 *   When |a| > 1 the state grows like |a|^n and overflows to inf for large n,
 *   as the step-by-step loop would.
 * Returns a cssd_status. */
int cssd_step_n(const cssd_dims* dims, void* h, const void* x, const float* dt, const void* A,
                const void* B, const void* C, const float* D, int64_t nsteps, void* y, cssd_stream_t stream);

/* Output of the same token held forever (the step_infinite shortcut of the
 * passage above): for |a| < 1 the state's dependence on its start decays like
 * |a|^n and y tends to
 *     y_inf = (C^T B) x / (1 - a) + D x,
 * which needs no state.  Arguments and layouts are those of cssd_step without
 * h.  The formula is evaluated as written for every a; it is a limit of the
 * recurrence only when |a| < 1 (Re A < 0), and a = 1 (A = 0) divides by zero.
 * Returns a cssd_status. */
int cssd_step_infinite(const cssd_dims* dims, const void* x, const float* dt, const void* A, const void* B,
                       const void* C, const float* D, void* y, cssd_stream_t stream);

/* Per-coordinate Cayley-phase recurrence ("Complex Phase-State Dynamics Reduce
 * the Optimization Steps of Sequence Models", section 5.2 equations (2)-(3),
 * section 5.5, Appendix A Algorithms 1-2).  Per (batch, head) a state psi in
 * C^N evolves coordinatewise:
 *     a_t   = sigmoid(u_t) (1 + i phi_t) / (1 - i phi_t)   (gate times unit Cayley phase)
 *     psi_t = a_t psi_{t-1} + b_t,    y_t = conj(C_t) psi_t  (readout after the update)
 * from psi0 (zero when NULL).
 *   dims     batch, seqlen, nheads, dstate = N (any N >= 1); headdim is ignored
 *   phi      float32   [batch, seqlen, nheads, N]  phase parameters
 *   u        float32   [batch, seqlen, nheads, N]  gate logits
 *   b        complex64 [batch, seqlen, nheads, N]  input projection
 *   C        complex64 [batch, seqlen, nheads, N]  readout projection
 *   psi0     complex64 [batch, nheads, N]          initial state, may be NULL
 *   y        complex64 [batch, seqlen, nheads, N]  output (written)
 *   psi_final complex64 [batch, nheads, N]         last state (written), may be NULL
 *   chunk    >= 1, the chunk length of the scan (the paper uses 64)
 *   log_clamp  -INFINITY evaluates the recurrence exactly (chunk then has no
 *            effect).  A finite value in [-80, 0] evaluates the paper's
 *            Algorithm 2 as published: per chunk, the cumulative log-gate is
 *            clamped to [log_clamp, 0] (the paper: -30) before the polar
 *            reassembly.  That equals the recurrence while no chunk's
 *            cumulative log-gate falls below log_clamp, and departs from it
 *            (inputs stop decaying) once one does.
 * Alignment: phi, u 4 bytes; b, C, y, psi0, psi_final 8 bytes.  Other
 * log_clamp values, chunk < 1 or non-positive sizes return CSSD_ERR_DIMS.
 * Returns a cssd_status. */
int cssd_cayley_scan(const cssd_dims* dims, const float* phi, const float* u, const void* b, const void* C,
                     const void* psi0, void* y, void* psi_final, int chunk, float log_clamp, cssd_stream_t stream);

/* Gradients of cssd_chunked_forward with respect to every input ("The
 * Chunkwise Complex SSD Algorithm", its backward section; the gradients are
 * those of the sequential recurrence of "Complex-Valued State Spaces", "The
 * discretization", which the chunked forward computes up to rounding).
 * Given the upstream gradient dy of a real loss L, with the convention
 *     dL = Re sum conj(g_w) dw      (complex w: g_w = dL/dRe w + i dL/dIm w;
 *                                    real w: g_w = dL/dw)
 * the call writes gx, gdt, gA, gB, gC, gD.  The adjoint state
 * G_t = conj(a_{t+1}) G_{t+1} + conj(C_t) dy_t^T is itself a run of the forward
 * recurrence (time reversed, rate conj(A)), so the gradients of x, B and C are
 * three runs of the forward kernels on reversed and conjugated inputs (read in
 * place through the kernels' indexing for headdim = dstate = 64, else copied);
 * those of dt and A follow from R_t = sum_{u >= t} sum_p (conj(dy_u) y_u -
 * x_u conj(gx_u)), since dL/dz_t = conj(R_t) for z_t = softplus(dt_t) A, and
 * R_t = a_t sum conj(G_t) h_{t-1}: for headdim = dstate = 64 and seqlen a
 * multiple of 64, R is taken at every 64-token boundary from that inner
 * product of the two runs' states and summed only within chunks, otherwise
 * summed over the sequence from its shorter end; gD = sum Re(conj(dy) x).
 * The forward output y is recomputed, and it and gx are computed to about
 * fp32 accuracy, because R_t is a small difference of large sums that
 * operands rounded to 11 significant bits would spoil: by the tensor-core
 * kernel with split-precision operands (each value as two half parts, three
 * products per product) where headdim is 64 and dstate 64, else by the fp32
 * CUDA-core chunk kernels
 * (dstate 128 among them).  gB and gC use the tensor-core forward where it
 * applies; with dstate 128 their runs (state transposed: headdim 128) take
 * the CUDA-core kernels.
 *   dims, x, dt, A, B, C, D, chunk   as cssd_chunked_forward; dstate in
 *            {16, 32, 64, 128}, headdim in {16, 32, 64} (else
 *            CSSD_ERR_UNSUPPORTED)
 *   dy       complex64 [batch, seqlen, nheads, headdim]  upstream gradient
 *   gx       complex64 like x;  gdt float32 like dt;  gA complex64 [nheads];
 *   gB, gC   complex64 like B, C;  gD float32 [nheads]     (all written)
 *   workspace  device memory of at least cssd_backward_workspace_bytes(dims,
 *            chunk) bytes, 16-byte aligned, or NULL (the library allocates and
 *            frees it stream-ordered)
 * Complex arrays 16-byte aligned, A and gA 8-byte, real ones 4-byte.  gA and gD
 * sum over batch and tokens in a fixed order (deterministic).  Errors as
 * cssd_chunked_forward.  Returns a cssd_status. */
size_t cssd_backward_workspace_bytes(const cssd_dims* dims, int chunk);
int cssd_chunked_backward(const cssd_dims* dims, const void* x, const float* dt, const void* A, const void* B,
                          const void* C, const float* D, const void* dy, void* gx, float* gdt, void* gA, void* gB,
                          void* gC, float* gD, int chunk, void* workspace, size_t workspace_bytes,
                          cssd_stream_t stream);

/* Causal Born attention ("Complex Phase-State Dynamics Reduce the
 * Optimization Steps of Sequence Models", section 5.5 equation (5), Appendix A
 * Algorithm 3).  Per (batch, head), for every query position i:
 *     s_ij  = |<q_i|k_j>|^2 / (D tau_i)   for j <= i,   <q|k> = sum_a conj(q_a) k_a
 *     psi_i = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij
 * The factor 1/(D tau_i) is common to numerator and denominator, so psi does
 * not depend on the temperature and it is not an argument.  A row whose scores
 * are all zero (q_i orthogonal to every k_j, j <= i) returns psi_i = 0.
 *   dims  batch, seqlen, nheads, dstate = D (head width: 16 or 32); headdim
 *         is ignored
 *   q, k, v  complex64 [batch, seqlen, nheads, D]  queries, keys, values
 *            (any phase rotation of q and k is applied by the caller)
 *   psi      complex64 [batch, seqlen, nheads, D]  output (written)
 * Queries, keys and values enter the tensor cores rounded to TF32 (round to
 * nearest); the squared scores are read by the tensor cores at TF32 precision
 * for the numerator and the score sum alike; accumulation is fp32.  All four pointers are device pointers, 16-byte
 * aligned.  Other D return CSSD_ERR_UNSUPPORTED.  Returns a cssd_status. */
int cssd_born_attention(const cssd_dims* dims, const void* q, const void* k, const void* v, void* psi,
                        cssd_stream_t stream);

/* Device status word.  Every wait a kernel of this library makes on other
 * threads or on the tensor cores is bounded; a wait that gives up lets the
 * kernel finish (its results are then invalid) and ORs a bit into a status word
 * the library keeps per device:
 *   1  the chunked forward: a state hand-off from the previous chunk timed out
 *   2  the chunked forward: a tensor-core completion wait timed out
 *   4  Born attention: a tensor-core completion wait timed out
 * The chunked forward's bits also cover cssd_chunked_backward, the precise
 * and host-streamed forwards, which run the same kernel.  This call reads the
 * word of the stream's device (which must be the current device) after the
 * work already on `stream`, clears it when `clear` is nonzero, and waits for
 * the stream.  The word starts at 0 and is never cleared by the library
 * itself.  Returns a cssd_status (CSSD_ERR_DEVICE when the stream belongs to
 * another device). */
int cssd_device_status(unsigned* bits, int clear, cssd_stream_t stream);

/* Measurement hook.  ev_begin / ev_end are cudaEvent_t handles created by
 * the caller on the device in use; every later cssd_chunked_forward call made
 * from the same host thread records ev_begin on its stream just before the
 * launch of its dominant kernel and ev_end just after it, so that the caller
 * can time that kernel alone with cudaEventElapsedTime.  Pass (NULL, NULL) to
 * turn it off.  This per-thread setting is the library's only state.
 * Returns CSSD_ERR_NULL if exactly one of the two is NULL. */
int cssd_profile_events(void* ev_begin, void* ev_end);

/* Failure-detection self-test of the forward's inter-chunk hand-off.  Runs
 * the tensor-core forward kernels (TF32 operands, half operands at dstate 64,
 * half operands at dstate 128) on a small internal problem (two sequences,
 * two 64-token chunks, zero inputs)
 * whose first chunk is never processed, so the second chunk's bounded wait for
 * its predecessor's state has to give up after `wait_cycles` SM clocks.  Each
 * kernel then records bit 0 in its error word, finishes, and frees its tensor
 * memory; the device stays usable.  The call allocates its buffers
 * stream-ordered, synchronises `stream`, and returns the three error words in
 * *err_bits: the TF32 kernel's in bits 0-7, the dstate-64 half-operand
 * kernel's in bits 8-15, the dstate-128 one's in bits 16-23 (in each, bit 0 =
 * a hand-off wait timed out, bit 1 = a tensor-core completion wait timed
 * out).  Returns CSSD_ERR_NULL / CSSD_ERR_DIMS for bad
 * arguments, CSSD_ERR_CUDA if a runtime call fails. */
int cssd_selftest_handoff_timeout(long long wait_cycles, int* err_bits, cssd_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* cssd_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CSSD_H */
