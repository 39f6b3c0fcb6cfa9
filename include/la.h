/*
 * la.h -- C ABI of the GB300 (sm_103a) causal kernelized attention library.
 *
 * The library computes linear attention with the feature map
 * phi(x) = elu(x) + 1 (alpha = 1; equal to x + 1 for x > 0 and exp(x) otherwise):
 *
 *   o_i = phi(q_i)^T S_i / max(phi(q_i)^T z_i, eps)
 *   S_i = sum_{j<=i} phi(k_j) v_j^T   (dk x dv),   z_i = sum_{j<=i} phi(k_j)   (dk)
 *
 * Definitions followed ("Linear attention", learn.pranaymahendrakar.com,
 * Researcher: Derivation, the recurrence S_i = S_{i-1} + phi(k_i) v_i^T and
 * o_i = S_i^T phi(q_i) / z_i^T phi(q_i); "Linear Attention",
 * aiwiki.thehackersbrain.dev, the chunked parallel form and its clamp of the
 * denominator).  No 1/sqrt(d) scaling is applied to q or k.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers to contiguous row-major memory,
 *    owned by the caller.  The library keeps no pointer after a call returns
 *    and never frees caller memory.
 *  - Each pointer must be 16-byte aligned (LA_ERR_MISALIGNED otherwise).
 *  - `dtype` is the element type of q, k, v and o (fp32 or bf16).  The states
 *    S and z are always fp32.  Arithmetic is fp32 (bf16 products on the tensor
 *    cores accumulate in fp32).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  The return value reports argument validation and
 *    launch errors only; call la_get_device_status() to learn whether a kernel
 *    gave up on a bounded wait.
 *  - Any of B, H, N, dk, dv equal to 0 is a valid empty problem: LA_OK, no work.
 *    Negative sizes, NULL pointers (for a non-empty problem) and a negative or
 *    non-finite eps give LA_ERR_INVALID_ARG.  Sizes the kernels are not built
 *    for give LA_ERR_UNSUPPORTED (see each function).
 *  - o must not overlap q, k or v.
 *  - Scratch memory.  The bf16 tensor-core forward paths keep two workspaces
 *    per (device, stream) -- the per-thread default stream
 *    (cudaStreamPerThread) of each host thread has its own -- : 64 KB of work
 *    tickets and flags, zeroed once and
 *    left zeroed by every launch, and a data buffer (split partials,
 *    published states) grown to the largest problem seen on that stream.
 *    Both are created or grown only outside stream capture, with cudaMalloc,
 *    and are kept until the process exits (a grown-out buffer too, so that a
 *    graph captured against it stays valid).  When a workspace cannot serve a
 *    call (first call during capture, or a larger problem during capture),
 *    that call allocates and frees its scratch stream-ordered
 *    (cudaMallocAsync / cudaFreeAsync on `stream`) instead, as every other
 *    path does.  Calls on one stream are ordered, so they never use a
 *    workspace at the same time; a graph replays with the workspaces of the
 *    stream it was captured on, so do not replay it while other work of this
 *    library runs on that stream, nor replay two of its instances at once.
 *  - The tensor-core forward kernels are launched with programmatic stream
 *    serialization: a launch may begin its set-up while the kernel before it
 *    on the stream finishes, and waits for that kernel to complete before it
 *    reads any global memory.
 */
#ifndef LA_H
#define LA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad eps, overlap */
    LA_ERR_UNSUPPORTED = 2,  /* size/dtype/chunk combination not built */
    LA_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    LA_ERR_CUDA = 4,         /* a CUDA runtime call failed (la_last_cuda_error) */
    LA_ERR_TIMEOUT = 5       /* a kernel's bounded wait expired (device status) */
} la_status;

typedef enum la_dtype {
    LA_F32 = 0,   /* IEEE binary32 q, k, v, o */
    LA_BF16 = 1   /* bfloat16 q, k, v, o */
} la_dtype;

/* Same type as cudaStream_t, declared here so this header needs no CUDA header. */
typedef struct CUstream_st *la_stream_t;

/*
 * Causal forward, chunked parallel form ("Linear Attention",
 * aiwiki.thehackersbrain.dev: quadratic inside a chunk, recurrent across
 * chunks; "Linear attention", learn.pranaymahendrakar.com, Implementation
 * reality: chunks of 64 or 128).
 *
 *   q, k : [B, H, N, dk]   v, o : [B, H, N, dv]
 *
 * o[b,h,i,:] = phi(q_i)^T S_i / max(phi(q_i)^T z_i, eps) with the sums over
 * j <= i of the same (b,h) (inclusive of i).  N need not be a multiple of
 * `chunk`; the last chunk is then shorter.  `chunk` must be 64 or 128.
 * Supported: dk, dv in {32, 64, 128}.  bf16 with N >= 128 runs on the
 * tensor cores, any dk and dv (with dk != dv, or 32, on tiles of the next
 * width, 64 or 128, whose extra columns are zero and drop out of every
 * product); it computes with chunks of 128 tokens whether `chunk` is 64 or
 * 128: the chunked form is the same function for every chunk length, only the
 * order of the roundings differs.  The CUDA-core path (fp32, N < 128) uses
 * `chunk` as given.
 */
la_status la_forward_causal(const void *q, const void *k, const void *v, void *o,
                            int B, int H, int N, int dk, int dv, int chunk, float eps,
                            la_dtype dtype, la_stream_t stream);

/*
 * Non-causal forward ("Linear attention: change the order.", implementation
 * you can check; "Linear Attention -- Math + Variants", o_i = phi(q_i)^T S /
 * phi(q_i)^T z with S, z summed over the whole sequence).
 *
 *   q, k : [B, H, N, dk]   v, o : [B, H, N, dv]
 *
 * o_i = phi(q_i)^T S / max(phi(q_i)^T z, eps), S = sum_j phi(k_j) v_j^T,
 * z = sum_j phi(k_j), j over all N positions of the same (b,h).
 * Supported: dk, dv in {32, 64, 128}.  bf16 with N >= 128 runs on the
 * tensor cores for every dk and dv (widths other than dk = dv in {64, 128}
 * on tiles of the next width, the extra columns zero); fp32 and shorter
 * sequences on the CUDA cores.
 */
la_status la_forward_noncausal(const void *q, const void *k, const void *v, void *o,
                               int B, int H, int N, int dk, int dv, float eps,
                               la_dtype dtype, la_stream_t stream);

/* Size of the scratch array built into the library for la_forward_noncausal_noalloc. */
#define LA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * Non-causal forward that allocates no device memory.  The pages have no
 * counterpart of this entry point: it is the same computation as
 * la_forward_noncausal (same arguments, layouts and results up to the order
 * of floating-point additions), offered for callers that cannot call
 * cudaMalloc or cudaMallocAsync -- for example a host program that has handed
 * all device memory to its own pool allocator (so a driver allocation would
 * fail or break its accounting), or a serving loop that forbids allocation
 * calls once it has started so that its latency and memory use stay fixed.
 *
 * Its scratch (the per-head S and z sums, B*H*dk*(dv+1) floats) lives in one
 * array of LA_NOALLOC_SCRATCH_BYTES bytes compiled into the library; every GPU
 * on which this part of the library has been loaded (see below) holds that
 * array until the process exits.  Problems
 * needing more than LA_NOALLOC_SCRATCH_BYTES bytes of scratch are rejected
 * with LA_ERR_UNSUPPORTED before any work is enqueued.
 *
 * The first call on a device that has work to do sets up: it looks up the
 * array's device address (cudaGetSymbolAddress, with that device current) and
 * caches it.  Under CUDA's lazy module loading (the default) the first calls
 * also load this part of the library onto the device -- the array when its
 * address is looked up, and each kernel when it is first launched (one pair
 * of kernels per dtype and dk) -- and loading is a device allocation.  So,
 * on each device, make one call of every dtype and dk you will use before
 * reserving the rest of device memory for a pool and before any stream
 * capture; later calls allocate nothing.  (A process may instead set
 * CUDA_MODULE_LOADING=EAGER, which loads everything when its CUDA context is
 * created.)  All calls share the one
 * array, and each call clears the part it uses before accumulating into it, so calls
 * whose work may overlap on the GPU (different streams, different host
 * threads) race with each other and must be serialised by the caller.
 */
la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v, void *o,
                                       int B, int H, int N, int dk, int dv, float eps,
                                       la_dtype dtype, la_stream_t stream);

/*
 * One recurrent decode step for B*H independent heads ("Linear Attention",
 * "It is a linear RNN": O(d^2) per token with a fixed-size state;
 * "26. Linear (Kernelized) Attention", Step-by-Step steps 3-4: update the
 * state, then read it).
 *
 *   S : [B, H, dk, dv] fp32, z : [B, H, dk] fp32   (read and updated in place)
 *   q, k : [B, H, dk]   v, o : [B, H, dv]            (element type `dtype`)
 *
 * S += phi(k) v^T;  z += phi(k);  o = phi(q)^T S / max(phi(q)^T z, eps).
 * S and z are the whole resumable memory of a sequence: passing them back in
 * continues it.  Supported: dk, dv in {32, 64, 128}.
 */
la_status la_decode_step(float *S, float *z, const void *q, const void *k, const void *v,
                         void *o, int B, int H, int dk, int dv, float eps,
                         la_dtype dtype, la_stream_t stream);

/*
 * Causal forward with a decayed state ("Linear Attention -- Math + Variants",
 * RetNet and gated linear attention: the recurrent state is multiplied by a
 * decay before each update, so old tokens fade).  One scalar decay per head:
 *
 *   S_i = g S_{i-1} + phi(k_i) v_i^T,   z_i = g z_{i-1} + phi(k_i),
 *   o_i = phi(q_i)^T S_i / max(phi(q_i)^T z_i, eps)
 *
 * i.e. o_i weights key j <= i by g^(i-j) in both the numerator and the
 * normaliser.  g = 1 gives la_forward_causal; g = 0 gives o_i = v_i wherever
 * phi(q_i).phi(k_i) >= eps.
 *
 *   q, k : [B, H, N, dk]   v, o : [B, H, N, dv]   gamma : [H] fp32, DEVICE memory
 *
 * Head h of every batch entry uses gamma[h].  gamma must be 4-byte aligned and
 * must not overlap o; its values are read by the kernel and not checked (the
 * method takes them in [0, 1]).  `chunk` (64 or 128) is the length of the
 * intra-chunk quadratic blocks on the CUDA cores.  bf16 with N >= 128 runs on
 * the tensor cores (128-token chunks, any dk, dv as la_forward_causal) (the kernel of la_forward_causal with the
 * decay weights in the intra-chunk mask, on the rows of phi(Q) and phi(K), on
 * the running state and in the scan across segments); other shapes run on the
 * CUDA cores in fp32.  Supported: dk, dv in {32, 64, 128}.
 */
la_status la_forward_causal_decay(const void *q, const void *k, const void *v, void *o,
                                  const float *gamma, int B, int H, int N, int dk, int dv,
                                  int chunk, float eps, la_dtype dtype, la_stream_t stream);

/*
 * One decode step with a decayed state (same source as la_forward_causal_decay):
 *
 *   S = g S + phi(k) v^T;  z = g z + phi(k);  o = phi(q)^T S / max(phi(q)^T z, eps)
 *
 * with g = gamma[h] (DEVICE memory, [H] fp32, 4-byte aligned, overlapping none
 * of S, z, o).  Arguments, layouts and in-place update as la_decode_step.
 */
la_status la_decode_step_decay(float *S, float *z, const void *q, const void *k, const void *v,
                               void *o, const float *gamma, int B, int H, int dk, int dv,
                               float eps, la_dtype dtype, la_stream_t stream);

/*
 * State of a prefix ("Linear Attention -- Math + Variants": S = sum_j
 * phi(k_j) v_j^T, z = sum_j phi(k_j)), used to start decoding after a causal
 * prefill of N tokens.
 *
 *   k : [B, H, N, dk]   v : [B, H, N, dv]   S : [B, H, dk, dv] fp32   z : [B, H, dk] fp32
 *
 * S and z are OVERWRITTEN (not accumulated).  N = 0 writes zeros.
 * Supported: dk, dv in {32, 64, 128}.  bf16 with N >= 128 runs on the tensor
 * cores (any dk, dv; other than dk = dv in {64, 128} on tiles of the next
 * width): phi(k) is evaluated in fp32 and split into
 * a bf16 high part and a bf16 low part (together accurate to about 2^-17), both
 * multiplied by v with fp32 accumulation; other shapes use fp32 CUDA-core
 * arithmetic.
 */
la_status la_prefill_state(const void *k, const void *v, float *S, float *z,
                           int B, int H, int N, int dk, int dv, la_dtype dtype,
                           la_stream_t stream);

/*
 * State of a prefix under the decayed recurrence of la_forward_causal_decay
 * (the recurrence unrolled over N tokens from a zero state):
 *
 *   S = sum_t g^(N-1-t) phi(k_t) v_t^T,   z = sum_t g^(N-1-t) phi(k_t),   g = gamma[h]
 *
 * so that la_decode_step_decay continues the sequence.  Layouts as
 * la_prefill_state; gamma as la_forward_causal_decay (DEVICE memory, [H] fp32,
 * 4-byte aligned, not overlapping S or z; may be NULL when N = 0).  S and z are
 * OVERWRITTEN; N = 0 writes zeros.  bf16 with N >= 128 runs on the tensor cores
 * as la_prefill_state does, for the same widths (phi(k) times its weight in fp32,
 * split into bf16 high and low parts); fp32 and shorter prefixes on the CUDA cores.
 */
la_status la_prefill_state_decay(const void *k, const void *v, const float *gamma, float *S,
                                 float *z, int B, int H, int N, int dk, int dv, la_dtype dtype,
                                 la_stream_t stream);

/*
 * Gated state with one gate per key feature ("Linear Attention",
 * aiwiki.thehackersbrain.dev, What is actually lost: gated variants insert a
 * decay, S_t = G_t (.) S_{t-1} + phi(k_t) v_t^T; "Linear Attention -- Math +
 * Variants", RetNet and gated linear attention: S_i = Diag(alpha_i) S_{i-1} +
 * k_i v_i^T, the decay computed from the token itself):
 *
 *   S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t (.) z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps)
 *
 * i.e. key j reaches query i >= j through feature r with weight
 * prod_{s=j+1..i} alpha_s[r], in the numerator and the normaliser alike.  The
 * gate values are the caller's (the layer that computes them from the token has
 * trained weights): alpha is fp32 DEVICE memory shaped like k, [B, H, N, dk]
 * ([B, H, dk] for a decode step), 16-byte aligned; its values are read as given
 * (the method takes them in [0, 1]).  Every alpha = gamma[h] reproduces
 * la_forward_causal_decay; every alpha = 1 reproduces la_forward_causal.
 *
 * la_forward_causal_gated: q, k : [B, H, N, dk]   v, o : [B, H, N, dv].  o must not
 *   overlap q, k, v or alpha.
 * la_prefill_state_gated: the state after N tokens from a zero state
 *   (S [B, H, dk, dv], z [B, H, dk] fp32, OVERWRITTEN; N = 0 writes zeros), so
 *   that la_decode_step_gated continues the sequence.
 * la_decode_step_gated: S, z read and updated in place; q, k : [B, H, dk],
 *   v, o : [B, H, dv], alpha : [B, H, dk].  S, z and o overlap nothing else.
 *
 * fp32 arithmetic on the CUDA cores: the recurrence itself, split over value
 * columns (each column of S evolves on its own).  Supported: dk, dv in
 * {32, 64, 128}.
 */
la_status la_forward_causal_gated(const void *q, const void *k, const void *v, void *o, const float *alpha,
                                  int B, int H, int N, int dk, int dv, float eps, la_dtype dtype,
                                  la_stream_t stream);
la_status la_prefill_state_gated(const void *k, const void *v, const float *alpha, float *S, float *z, int B,
                                 int H, int N, int dk, int dv, la_dtype dtype, la_stream_t stream);
la_status la_decode_step_gated(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                               const float *alpha, int B, int H, int dk, int dv, float eps, la_dtype dtype,
                               la_stream_t stream);

/*
 * Variants of the feature map and of the normaliser.
 *
 * Feature maps ("Linear attention", learn.pranaymahendrakar.com, What the
 * pieces are for: ReLU among the alternatives to elu + 1; "Linear Attention --
 * Math + Variants", Feature-map families: ReLU and identity-plus-shift; "26.
 * Linear (Kernelized) Attention", Key Functions & Tricks: relu(x) + eps):
 *   LA_PHI_ELU1      phi(x) = elu(x) + 1          (the default; shift ignored)
 *   LA_PHI_RELU      phi(x) = max(x, 0) + shift   (shift >= 0 keeps phi >= 0)
 *   LA_PHI_IDENTITY  phi(x) = x + shift
 * normalize = 1: o = phi(q)^T S / max(phi(q)^T z, eps) (the default);
 * normalize = 0: o = phi(q)^T S, the normaliser-free output that "Linear
 * Attention -- Math + Variants", Implementation reality, describes (a
 * normalisation layer after attention, which needs trained weights, is the
 * caller's).  A NULL variant pointer means the default.
 */
typedef enum { LA_PHI_ELU1 = 0, LA_PHI_RELU = 1, LA_PHI_IDENTITY = 2 } la_feature_map;

typedef struct {
    int feature_map; /* la_feature_map */
    float shift;     /* finite */
    int normalize;   /* 0 or 1 */
} la_variant;

/*
 * The general forms: any feature map, with or without the normaliser, with or
 * without the decayed state (gamma: DEVICE pointer to H fp32 values, one per
 * head, as la_forward_causal_decay; NULL = no decay).  Same layouts, checks
 * and results as the specialised entry points, which they reduce to:
 *   la_forward_causal_ex(..., NULL, NULL, ...)   = la_forward_causal
 *   la_forward_causal_ex(..., gamma, NULL, ...)  = la_forward_causal_decay
 * bf16 with N >= 128 runs on the tensor cores for every variant and every
 * dk, dv; fp32 and shorter sequences on the CUDA cores.
 * An invalid variant (unknown map, non-finite shift, normalize not 0 or 1)
 * returns LA_ERR_INVALID_ARG.
 */
la_status la_forward_causal_ex(const void *q, const void *k, const void *v, void *o,
                               const float *gamma, const la_variant *variant, int B, int H,
                               int N, int dk, int dv, int chunk, float eps, la_dtype dtype,
                               la_stream_t stream);
la_status la_forward_noncausal_ex(const void *q, const void *k, const void *v, void *o,
                                  const la_variant *variant, int B, int H, int N, int dk,
                                  int dv, float eps, la_dtype dtype, la_stream_t stream);
la_status la_decode_step_ex(float *S, float *z, const void *q, const void *k, const void *v,
                            void *o, const float *gamma, const la_variant *variant, int B,
                            int H, int dk, int dv, float eps, la_dtype dtype,
                            la_stream_t stream);
/* The prefix state under a feature map (normalize is ignored: S and z are the
 * same either way) and an optional decay. */
la_status la_prefill_state_ex(const void *k, const void *v, const float *gamma,
                              const la_variant *variant, float *S, float *z, int B, int H,
                              int N, int dk, int dv, la_dtype dtype, la_stream_t stream);

/*
 * Backward pass of the causal forward (elu + 1, with the normaliser): given
 * dout = dL/do, writes dq = dL/dq, dk = dL/dk, dv = dL/dv for L = sum dout . o.
 * The pages give no gradient ("Linear Attention -- Math + Variants", Chunkwise
 * parallelism: training runs the chunked form); it is the chain rule through
 * the recurrence: a forward scan of S, z for dq and a reverse scan of
 * R_j = sum_{i>=j} phi(q_i) dn_i^T, r_j = sum_{i>=j} dd_i phi(q_i) for dk, dv,
 * with dn_i = dout_i / d_i, dd_i = -(dout_i . o_i) / d_i and d_i the clamped
 * denominator (no gradient flows through the clamp where it binds).
 *
 *   q, k, dq, dk : [B, H, N, d_k]   v, dout, dv : [B, H, N, d_v]   (element type `dtype`)
 *
 * Outputs must not overlap any input or each other.  Recomputes the forward
 * quantities it needs (no saved activations).  bf16 with d_k, d_v in {32, 64}
 * and N >= 128 runs on the tensor cores: five launches over chunks of 128
 * tokens (chunk states, a forward scan, dq, a reverse scan, dk and dv), bf16
 * operands with fp32 accumulation, scratch from the stream's workspace.  Other
 * shapes and fp32: fp32 arithmetic on the CUDA cores, chunk-parallel (chunk
 * states, scans over chunks, per-chunk gradients); per-call scratch of
 * B*H*ceil(N/C)*d_k*(d_v+1) + B*H*N*(d_v+1) floats (C = 64, or 32 when d_k or
 * d_v is 128), stream-ordered.  Supported: d_k, d_v in {32, 64, 128}.
 */
la_status la_backward_causal(const void *q, const void *k, const void *v, const void *dout,
                             void *dq, void *dk, void *dv, int B, int H, int N, int d_k, int d_v,
                             float eps, la_dtype dtype, la_stream_t stream);

/*
 * FAVOR+ positive random features ("Linear Attention -- Math + Variants",
 * Performer: features whose inner products estimate the softmax kernel,
 * E[phi(q) . phi(k)] = exp(q . k) over Gaussian projections w_r):
 *
 *   phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m),   r = 0 .. m-1
 *
 *   x : [B, H, N, d]   w : [m, d] (row r is w_r)   phi : [B, H, N, m]
 *
 * All three of element type `dtype`.  The projections are the caller's: plain
 * Gaussian rows, or orthogonal blocks rescaled to Gaussian norms (the page's
 * variance reduction) -- the library only applies them.  No 1/sqrt(d) or other
 * scaling is applied to x.  phi must not overlap x or w.  Supported: d, m in
 * {32, 64, 128}.  bf16 with d, m in {64, 128} and N >= 128 runs on the tensor cores (x w^T
 * accumulated in fp32, the exponential in fp32, phi rounded to bf16 once);
 * other shapes and fp32 on the CUDA cores in fp32.  m = 0 is an empty output.
 */
la_status la_favor_features(const void *x, const void *w, void *phi, int B, int H, int N, int d, int m,
                            la_dtype dtype, la_stream_t stream);

/*
 * Causal and non-causal linear attention on FAVOR+ features (same page): the
 * forwards of la_forward_causal / la_forward_noncausal with phi(q), phi(k) of
 * la_favor_features in place of elu + 1, normalised by max(phi(q)^T z, eps):
 *
 *   q, k : [B, H, N, d]   v, o : [B, H, N, dv]   w : [m, d]   (element type `dtype`)
 *
 * The state has m rows (S is m x dv).  phi(q) and phi(k) are written to
 * per-call stream-ordered scratch (2 * B*H*N*m elements of `dtype`) and then
 * attended with the identity map, so each call is two launches or more;
 * except the non-causal form for bf16 with d = m = 64, dv <= 64 and N >= 128,
 * which computes the features inside its one attention launch (no scratch).
 * w must not overlap o.  Supported: d, dv, m in {32, 64, 128}; the attention
 * step runs on the tensor cores for bf16 with m = dv in {64, 128} (and, causal,
 * N >= 128), on the CUDA cores otherwise.  m outside the
 * supported set (0 included) gives LA_ERR_UNSUPPORTED.
 */
la_status la_forward_causal_favor(const void *q, const void *k, const void *v, void *o, const void *w, int B,
                                  int H, int N, int d, int dv, int m, int chunk, float eps, la_dtype dtype,
                                  la_stream_t stream);
la_status la_forward_noncausal_favor(const void *q, const void *k, const void *v, void *o, const void *w, int B,
                                     int H, int N, int d, int dv, int m, float eps, la_dtype dtype,
                                     la_stream_t stream);

/*
 * The prefix state and the decode step on FAVOR+ features (same page; the
 * recurrent form that every kernelized variant keeps): la_prefill_state and
 * la_decode_step with phi(k), phi(q) of la_favor_features in place of elu + 1.
 *
 *   prefill: k : [B, H, N, d]   v : [B, H, N, dv]   w : [m, d]
 *            S : [B, H, m, dv] fp32, z : [B, H, m] fp32 (OVERWRITTEN; N = 0 writes zeros)
 *   decode:  q, k : [B, H, d]   v, o : [B, H, dv]   w : [m, d]
 *            S : [B, H, m, dv], z : [B, H, m] fp32, read and updated in place:
 *            S += phi(k) v^T;  z += phi(k);  o = phi(q)^T S / max(phi(q)^T z, eps)
 *
 * The features go to per-call stream-ordered scratch (prefill: B*H*N*m
 * elements; decode: 2*B*H*m), then the identity-map forms run on them.  In the
 * decode step the B*H rows of q and k are featurised as one batch (the tensor-core
 * features kernel takes it from 128 rows).  w must not overlap S, z or o; S and
 * z must not overlap k (or q).  Supported: d, dv, m in {32, 64, 128} (B, H or
 * dv = 0 is an empty problem; another d or m gives LA_ERR_UNSUPPORTED).
 */
la_status la_prefill_state_favor(const void *k, const void *v, const void *w, float *S, float *z, int B, int H,
                                 int N, int d, int dv, int m, la_dtype dtype, la_stream_t stream);
la_status la_decode_step_favor(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                               const void *w, int B, int H, int d, int dv, int m, float eps, la_dtype dtype,
                               la_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *la_status_string(la_status s);

/* The cudaError_t of the most recent CUDA failure on this thread (0 if none). */
int la_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device: LA_ERR_TIMEOUT if a kernel abandoned a bounded
 * wait since the last call, LA_OK otherwise (LA_ERR_CUDA if the read failed).
 */
la_status la_get_device_status(la_stream_t stream);

/*
 * Hooks for the library's own failure-detection tests -- not for production use.
 * They act on the causal forward for bf16 with dk = dv = 64 (elu + 1 with the
 * normaliser, no decay): its chunk-parallel kernel (N > 2048 and 16 or more heads
 * in total), whose work items publish per-chunk states that later items wait
 * for, and -- the wait limit only -- its cluster kernel (N <= 2048).  Both
 * settings are process-wide and apply to launches made after the call.
 *
 * la_test_set_wait_limit_ns(ns): every bounded wait of those kernels gives up after
 * ns nanoseconds instead of 2 s (0 restores 2 s).  A wait that gives up records
 * LA_ERR_TIMEOUT for la_get_device_status() and raises the launch's abort word, so
 * every CTA of the launch stops taking work, drains its copies and tensor-core
 * operations in flight, frees its tensor memory and exits; the outputs of that
 * launch are then undefined, and the next launch starts clean.
 *
 * la_test_drop_publication(t): the work item with ticket t (ticket t is chunk
 * t / (B*H) of sequence t % (B*H)) computes as usual but never publishes its
 * chunk state, so the later chunks of its sequence wait until their limit runs
 * out -- a lost message, made on purpose.  -1 turns it off.
 */
void la_test_set_wait_limit_ns(unsigned long long ns);
void la_test_drop_publication(long long ticket);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int la_version(void);

/*
 * Number of kernel launches (and memset nodes) the library has enqueued in this
 * process since it was loaded, on all streams and devices.  Launches recorded
 * into a CUDA graph during stream capture are counted once, at capture time.
 */
unsigned long long la_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
