// Launchers shared between the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>

#include "la.h"

namespace la {

// Records a CUDA error for la_last_cuda_error() and returns LA_ERR_CUDA (or LA_OK).
la_status cuda_status(cudaError_t e);

// Stream-ordered scratch: cudaMallocAsync / cudaFreeAsync on the call's stream.
struct Scratch {
    void *ptr = nullptr;
    cudaStream_t stream = nullptr;
    la_status alloc(size_t bytes, cudaStream_t s);
    ~Scratch();
};

// Feature-map and normaliser variant ("Linear attention", What the pieces are
// for: ReLU; "Linear Attention -- Math + Variants", Feature-map families: ReLU
// and identity-plus-shift, Implementation reality: dropping the normaliser):
// map LA_PHI_ELU1 (elu + 1), LA_PHI_RELU (max(x, 0) + shift), LA_PHI_IDENTITY
// (x + shift); normalize 0: o = phi(q)^T S.
struct Variant {
    int map = LA_PHI_ELU1;
    float shift = 0.f;
    int normalize = 1;
    bool is_default() const { return map == LA_PHI_ELU1 && normalize == 1; }
};

struct Problem {
    const void *q, *k, *v;
    void *o;
    int BH, N, dk, dv, chunk;
    float eps;
    la_dtype dtype;
    cudaStream_t stream;
    // Decayed state (la_forward_causal_decay): gamma [H] on the device, head of
    // sequence bh = bh % H; null for the undecayed forms.
    const float *gamma = nullptr;
    int H = 1;
    Variant var;
};

// Backward pass of the causal form (la_backward.cu): inputs q, k, v, dout; outputs
// dq, dk (layout of q) and dv (layout of v); fp32 arithmetic on the CUDA cores.
struct BackwardProblem {
    const void *q, *k, *v, *dout;
    void *dq, *dk, *dv;
    int BH, N, dkd, dvd;
    float eps;
    la_dtype dtype;
    cudaStream_t stream;
};
la_status causal_backward(const BackwardProblem &p);
// Tensor-core backward (la_tc_backward.cu): bf16, dk, dv <= 64 (64-column tiles), N >= 128.
bool backward_tc_eligible(const BackwardProblem &p);
la_status causal_backward_tc(const BackwardProblem &p);

// SIMT kernels (la_simt.cu): fp32 CUDA-core arithmetic, any supported dtype.
la_status causal_simt(const Problem &p);
la_status noncausal_simt(const Problem &p);
// Same computation with the library's fixed scratch array (no allocation).
la_status noncausal_simt_noalloc(const Problem &p);
// S, z (fp32, [BH,dk,dv], [BH,dk]) = sums over N tokens; overwrites S and z.
// gamma (device, [H]): token t weighted by gamma[bh % H]^(N-1-t); null: unweighted.
la_status state_simt(const void *k, const void *v, float *S, float *z, int BH, int N, int dk,
                     int dv, la_dtype dtype, cudaStream_t stream, const float *gamma = nullptr,
                     int H = 1, const Variant &var = Variant());

// Gated state with one gate per key feature (la_gated.cu), fp32 on the CUDA cores:
// alpha [BH, N, dk] (decode: [BH, dk]) fp32 in device memory.
la_status causal_gated(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH, int N,
                       int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream);
// The chunked form of the gated causal forward (la_gated_chunk.cu), and the
// token-by-token recurrence it replaced for the forward (la_gated.cu).
la_status causal_gated_chunked(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH,
                               int N, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream);
la_status causal_gated_recurrent(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH,
                                 int N, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream);
la_status state_gated(const void *k, const void *v, const float *alpha, float *S, float *z, int BH, int N, int dk,
                      int dv, la_dtype dtype, cudaStream_t stream);
la_status decode_step_gated(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                            const float *alpha, int BH, int dk, int dv, float eps, la_dtype dtype,
                            cudaStream_t stream);

// Decode step (la_decode.cu).
// gamma (device, [H], head = bh % H): the decayed step S = g S + phi(k) v^T,
// z = g z + phi(k); null for the undecayed step.
la_status decode_step(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                      int BH, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream,
                      const float *gamma = nullptr, int H = 1, const Variant &var = Variant());

// Tensor-core (tcgen05) paths (la_tc_causal.cu); return LA_ERR_UNSUPPORTED when
// the problem is outside the shapes they are built for.
la_status causal_tc(const Problem &p);
// Chunk-parallel causal kernel (la_tc_causal_chunks.cu): bf16, dk = dv = 64, chunk
// 128, N >= 128, elu + 1 with the normaliser, no decay.
la_status causal_chunks_tc(const Problem &p);
// Cluster kernel (la_tc_causal_cluster.cu): bf16, dk = dv = 64, chunk 128,
// 128 <= N <= 2048, elu + 1 with the normaliser, no decay.
la_status causal_cluster_tc(const Problem &p);
// (la_tc_noncausal.cu)
la_status noncausal_tc(const Problem &p);
// The non-causal FAVOR+ form with the features computed in the kernel
// (la_tc_noncausal.cu): bf16, q, k [.., 64] and W [64, 64] (m = d = 64, device,
// 16-byte aligned), dv <= 64, N >= 128; LA_ERR_UNSUPPORTED otherwise.
la_status noncausal_tc_favor(const Problem &p, const void *w);
// S, z (fp32, [BH,dk,dv], [BH,dk]) = sums over N tokens on the tensor cores (bf16
// k, v; dk, dv multiples of 8 up to 128 (on tiles of 64 or 128 columns), N >= 128);
// overwrites S and z.  gamma (device, [H]): token t weighted by gamma[bh % H]^(N-1-t);
// null: unweighted.
la_status noncausal_tc_state(const void *k, const void *v, float *S, float *z, int BH, int N, int dk, int dv,
                             cudaStream_t stream, const float *gamma = nullptr, int H = 1,
                             const Variant &var = Variant());

// Device status words of translation units that run bounded waits: read and clear.
la_status tc_causal_read_status(cudaStream_t s, unsigned *bits);
la_status tc_noncausal_read_status(cudaStream_t s, unsigned *bits);
la_status favor_read_status(cudaStream_t s, unsigned *bits);
la_status tc_chunks_read_status(cudaStream_t s, unsigned *bits);
la_status tc_cluster_read_status(cudaStream_t s, unsigned *bits);
la_status tc_backward_read_status(cudaStream_t s, unsigned *bits);

// Failure-detection test hooks (la_test_set_wait_limit_ns, la_test_drop_publication):
// the limit of the chunk-parallel causal kernel's bounded waits (2 s unless a test
// set another) and the ticket whose state that kernel does not publish (-1: none).
unsigned long long test_wait_limit_ns();
long long test_drop_ticket();

// FAVOR+ features (la_favor.cu): oq = phi(xq) and, when xk is not null, ok =
// phi(xk), with phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m); x [BH, N, d],
// W [m, d] and the outputs [BH, N, m], all of element type dtype.  bf16 with d,
// m in {64, 128} and N >= 128 on the tensor cores, everything else on the CUDA
// cores in fp32.
la_status favor_features(const void *xq, const void *xk, const void *W, void *oq, void *ok, int BH, int N, int d,
                         int m, la_dtype dtype, cudaStream_t stream);

bool supported_dim(int d);

// Counts every kernel launch / memset the library enqueues (la_kernel_launches).
void count_launches(unsigned n = 1);

// Flag workspace of the ticketed kernels: kFlagWorkspaceBytes per (device,
// stream), zeroed once when it is created, and left zeroed by every kernel that
// uses it (the last CTA to finish clears what the launch used).  Layout: [0]
// work ticket, [1] CTAs done, flags from byte 16.  Returns LA_ERR_UNSUPPORTED
// when it cannot serve the call -- more bytes than it holds, or a stream under
// capture that has none yet (it is created only outside capture) -- and the
// caller then uses per-call scratch cleared by a memset.  Calls on one stream
// are ordered, so they never share the flags at the same time; a captured graph
// keeps the workspace of the stream it was captured on.
constexpr size_t kFlagWorkspaceBytes = 64 << 10;
la_status flag_workspace(cudaStream_t s, size_t bytes, void **out);

// Data workspace of the ticketed kernels (split partials, published states,
// state images; contents need no clearing): one buffer per (device, stream),
// grown outside capture to the largest request seen (at least doubling).  A
// buffer it outgrows is kept, not freed, until the process exits, so a graph
// captured against it stays valid.  Returns LA_ERR_UNSUPPORTED when it cannot
// serve the call (a stream under capture whose buffer is too small, or the
// allocation failed); the caller then uses per-call scratch.
la_status data_workspace(cudaStream_t s, size_t bytes, void **out);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and device,
// so that repeated calls (and stream capture) issue no attribute calls.
la_status ensure_smem(const void *kernel, int bytes);

}  // namespace la
