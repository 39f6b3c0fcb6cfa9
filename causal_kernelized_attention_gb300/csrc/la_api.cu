// C ABI entry points: argument validation, dispatch to the kernels, status codes.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <set>
#include <thread>
#include <tuple>
#include <utility>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {

static thread_local int t_last_cuda_error = 0;

la_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return LA_OK;
    t_last_cuda_error = (int)e;
    return LA_ERR_CUDA;
}

la_status Scratch::alloc(size_t bytes, cudaStream_t s)
{
    stream = s;
    return cuda_status(cudaMallocAsync(&ptr, bytes, s));
}

Scratch::~Scratch()
{
    if (ptr) {
        cudaError_t e = cudaFreeAsync(ptr, stream);
        if (e != cudaSuccess) t_last_cuda_error = (int)e;
    }
}

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

static std::atomic<unsigned long long> g_launches{0};

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

la_status ensure_smem(const void *kernel, int bytes)
{
    static std::mutex mu;
    static std::set<std::tuple<const void *, int, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(kernel, dev, bytes);
    if (done.count(key)) return LA_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_status(e);
    done.insert(key);
    return LA_OK;
}

// Key of a stream's workspaces: the device, the stream handle and, for the
// per-thread default stream, the host thread.  cudaStreamPerThread is one handle
// value in every host thread but a different stream in each, so two threads
// must not share its workspaces.  (The stream's unique id would tell streams
// apart too, but querying it is not permitted while a stream is being captured.)
typedef std::tuple<int, cudaStream_t, std::thread::id> StreamKey;
static la_status stream_key(cudaStream_t s, StreamKey *key)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    *key = std::make_tuple(dev, s, s == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id());
    return LA_OK;
}

la_status flag_workspace(cudaStream_t s, size_t bytes, void **out)
{
    *out = nullptr;
    if (bytes > kFlagWorkspaceBytes) return LA_ERR_UNSUPPORTED;
    StreamKey key;
    la_status st = stream_key(s, &key);
    if (st != LA_OK) return st;
    static std::mutex mu;
    static std::map<StreamKey, void *> spaces;  // kept until the process exits
    std::lock_guard<std::mutex> lock(mu);
    auto it = spaces.find(key);
    if (it != spaces.end()) {
        *out = it->second;
        return LA_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_status(e);
    if (cs != cudaStreamCaptureStatusNone) return LA_ERR_UNSUPPORTED;
    void *p = nullptr;
    e = cudaMalloc(&p, kFlagWorkspaceBytes);
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaMemsetAsync(p, 0, kFlagWorkspaceBytes, s);
    count_launches();
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_status(e);
    }
    spaces[key] = p;
    *out = p;
    return LA_OK;
}

la_status data_workspace(cudaStream_t s, size_t bytes, void **out)
{
    *out = nullptr;
    if (bytes == 0) return LA_OK;
    StreamKey key;
    la_status st = stream_key(s, &key);
    if (st != LA_OK) return st;
    static std::mutex mu;
    static std::map<StreamKey, std::pair<void *, size_t>> spaces;
    std::lock_guard<std::mutex> lock(mu);
    auto it = spaces.find(key);
    if (it != spaces.end() && it->second.second >= bytes) {
        *out = it->second.first;
        return LA_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_status(e);
    if (cs != cudaStreamCaptureStatusNone) return LA_ERR_UNSUPPORTED;
    size_t size = it != spaces.end() ? std::max(bytes, 2 * it->second.second) : bytes;
    size = (size + (2u << 20) - 1) / (2u << 20) * (2u << 20);
    void *p = nullptr;
    if (cudaMalloc(&p, size) != cudaSuccess) {
        (void)cudaGetLastError();  // not sticky: the caller's per-call scratch may still fit
        return LA_ERR_UNSUPPORTED;
    }
    spaces[key] = std::make_pair(p, size);  // an outgrown buffer stays allocated (see above)
    *out = p;
    return LA_OK;
}

static std::atomic<unsigned long long> g_test_wait_ns{0};
static std::atomic<long long> g_test_drop{-1};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s: far beyond any healthy wait

unsigned long long test_wait_limit_ns()
{
    const unsigned long long v = g_test_wait_ns.load(std::memory_order_relaxed);
    return v ? v : kDefaultWaitNs;
}
long long test_drop_ticket() { return g_test_drop.load(std::memory_order_relaxed); }

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

static size_t elem_size(la_dtype t) { return t == LA_F32 ? 4 : 2; }

// Common checks of the forward entry points.  Returns LA_OK and sets *empty when
// there is nothing to do.
static la_status check_forward(const void *q, const void *k, const void *v, const void *o, int B, int H,
                               int N, int dk, int dv, float eps, la_dtype dtype, bool *empty)
{
    *empty = false;
    if (B < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0 || dk == 0 || dv == 0) {
        *empty = true;
        return LA_OK;
    }
    if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_MISALIGNED;
    const size_t es = elem_size(dtype);
    const size_t nqk = (size_t)B * H * N * dk * es, nvo = (size_t)B * H * N * dv * es;
    if (overlaps(o, nvo, q, nqk) || overlaps(o, nvo, k, nqk) || overlaps(o, nvo, v, nvo))
        return LA_ERR_INVALID_ARG;
    return LA_OK;
}

// A variant of the feature map / normaliser (NULL: elu + 1 with the normaliser).
static la_status check_variant(const la_variant *v, Variant *out)
{
    *out = Variant();
    if (!v) return LA_OK;
    if (v->feature_map != LA_PHI_ELU1 && v->feature_map != LA_PHI_RELU && v->feature_map != LA_PHI_IDENTITY)
        return LA_ERR_INVALID_ARG;
    if (!isfinite(v->shift)) return LA_ERR_INVALID_ARG;
    if (v->normalize != 0 && v->normalize != 1) return LA_ERR_INVALID_ARG;
    out->map = v->feature_map;
    out->shift = v->feature_map == LA_PHI_ELU1 ? 0.f : v->shift;
    out->normalize = v->normalize;
    return LA_OK;
}

// Checks of the decode entry points; gamma null for the undecayed step.
static la_status decode_checked(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                                const float *gamma, int B, int H, int dk, int dv, float eps, la_dtype dtype,
                                cudaStream_t stream, const Variant &var)
{
    if (B < 0 || H < 0 || dk < 0 || dv < 0) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || dk == 0 || dv == 0) return LA_OK;
    if (!S || !z || !q || !k || !v || !o) return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return LA_ERR_MISALIGNED;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)B * H, es = elem_size(dtype);
    if (BH > 0x7fffffff) return LA_ERR_UNSUPPORTED;
    const size_t nS = BH * dk * dv * 4, nz = BH * dk * 4, nqk = BH * dk * es, nvo = BH * dv * es;
    if (overlaps(S, nS, z, nz) || overlaps(o, nvo, S, nS) || overlaps(o, nvo, z, nz) ||
        overlaps(o, nvo, q, nqk) || overlaps(o, nvo, k, nqk) || overlaps(o, nvo, v, nvo))
        return LA_ERR_INVALID_ARG;
    return decode_step(S, z, q, k, v, o, (int)BH, dk, dv, eps, dtype, stream, gamma, H, var);
}

}  // namespace la

using namespace la;

extern "C" {

la_status la_forward_causal_ex(const void *q, const void *k, const void *v, void *o, const float *gamma,
                               const la_variant *variant, int B, int H, int N, int dk, int dv, int chunk,
                               float eps, la_dtype dtype, la_stream_t stream)
{
    bool empty;
    la_status st = check_forward(q, k, v, o, B, H, N, dk, dv, eps, dtype, &empty);
    if (st != LA_OK) return st;
    Variant var;
    if ((st = check_variant(variant, &var)) != LA_OK) return st;
    if (chunk != 64 && chunk != 128) return LA_ERR_UNSUPPORTED;
    if (empty) return LA_OK;
    if (gamma && ((uintptr_t)gamma & 3u) != 0) return LA_ERR_MISALIGNED;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    if (gamma && overlaps(o, (size_t)B * H * N * dv * elem_size(dtype), gamma, (size_t)H * 4))
        return LA_ERR_INVALID_ARG;
    Problem p{q, k, v, o, B * H, N, dk, dv, chunk, eps, dtype, (cudaStream_t)stream, gamma, H, var};
    if (dtype == LA_BF16) {
        st = causal_tc(p);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    return causal_simt(p);
}

la_status la_forward_causal(const void *q, const void *k, const void *v, void *o, int B, int H, int N,
                            int dk, int dv, int chunk, float eps, la_dtype dtype, la_stream_t stream)
{
    return la_forward_causal_ex(q, k, v, o, nullptr, nullptr, B, H, N, dk, dv, chunk, eps, dtype, stream);
}

la_status la_forward_causal_decay(const void *q, const void *k, const void *v, void *o, const float *gamma,
                                  int B, int H, int N, int dk, int dv, int chunk, float eps, la_dtype dtype,
                                  la_stream_t stream)
{
    if (!gamma) {  // required unless there is nothing to do
        bool empty;
        la_status st = check_forward(q, k, v, o, B, H, N, dk, dv, eps, dtype, &empty);
        if (st != LA_OK) return st;
        if (chunk != 64 && chunk != 128) return LA_ERR_UNSUPPORTED;
        return empty ? LA_OK : LA_ERR_INVALID_ARG;
    }
    return la_forward_causal_ex(q, k, v, o, gamma, nullptr, B, H, N, dk, dv, chunk, eps, dtype, stream);
}

la_status la_forward_noncausal_ex(const void *q, const void *k, const void *v, void *o, const la_variant *variant,
                                  int B, int H, int N, int dk, int dv, float eps, la_dtype dtype,
                                  la_stream_t stream)
{
    bool empty;
    la_status st = check_forward(q, k, v, o, B, H, N, dk, dv, eps, dtype, &empty);
    if (st != LA_OK) return st;
    Variant var;
    if ((st = check_variant(variant, &var)) != LA_OK || empty) return st;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    Problem p{q, k, v, o, B * H, N, dk, dv, 0, eps, dtype, (cudaStream_t)stream, nullptr, H, var};
    if (dtype == LA_BF16) {
        st = noncausal_tc(p);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    return noncausal_simt(p);
}

la_status la_forward_noncausal(const void *q, const void *k, const void *v, void *o, int B, int H, int N,
                               int dk, int dv, float eps, la_dtype dtype, la_stream_t stream)
{
    return la_forward_noncausal_ex(q, k, v, o, nullptr, B, H, N, dk, dv, eps, dtype, stream);
}

la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v, void *o, int B, int H,
                                       int N, int dk, int dv, float eps, la_dtype dtype, la_stream_t stream)
{
    bool empty;
    la_status st = check_forward(q, k, v, o, B, H, N, dk, dv, eps, dtype, &empty);
    if (st != LA_OK || empty) return st;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    Problem p{q, k, v, o, B * H, N, dk, dv, 0, eps, dtype, (cudaStream_t)stream};
    return noncausal_simt_noalloc(p);
}

la_status la_decode_step_ex(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                            const float *gamma, const la_variant *variant, int B, int H, int dk, int dv, float eps,
                            la_dtype dtype, la_stream_t stream)
{
    Variant var;
    la_status st = check_variant(variant, &var);
    if (st != LA_OK) return st;
    if (gamma && B > 0 && H > 0 && dk > 0 && dv > 0) {
        if (((uintptr_t)gamma & 3u) != 0) return LA_ERR_MISALIGNED;
        const size_t BH = (size_t)B * H;
        if (overlaps(gamma, (size_t)H * 4, S, BH * dk * dv * 4) || overlaps(gamma, (size_t)H * 4, z, BH * dk * 4))
            return LA_ERR_INVALID_ARG;
        if (o && overlaps(gamma, (size_t)H * 4, o, BH * dv * elem_size(dtype))) return LA_ERR_INVALID_ARG;
    }
    return decode_checked(S, z, q, k, v, o, gamma, B, H, dk, dv, eps, dtype, (cudaStream_t)stream, var);
}

la_status la_decode_step(float *S, float *z, const void *q, const void *k, const void *v, void *o, int B,
                         int H, int dk, int dv, float eps, la_dtype dtype, la_stream_t stream)
{
    return la_decode_step_ex(S, z, q, k, v, o, nullptr, nullptr, B, H, dk, dv, eps, dtype, stream);
}

la_status la_decode_step_decay(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                               const float *gamma, int B, int H, int dk, int dv, float eps, la_dtype dtype,
                               la_stream_t stream)
{
    if (!gamma && B > 0 && H > 0 && dk > 0 && dv > 0) return LA_ERR_INVALID_ARG;
    return la_decode_step_ex(S, z, q, k, v, o, gamma, nullptr, B, H, dk, dv, eps, dtype, stream);
}

la_status la_prefill_state_ex(const void *k, const void *v, const float *gamma, const la_variant *variant, float *S,
                              float *z, int B, int H, int N, int dk, int dv, la_dtype dtype, la_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    Variant var;
    la_status st = check_variant(variant, &var);
    if (st != LA_OK) return st;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || dk == 0 || dv == 0) return LA_OK;
    if (!S || !z || (N > 0 && (!k || !v))) return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z) || (N > 0 && (!aligned16(k) || !aligned16(v))))
        return LA_ERR_MISALIGNED;
    if (N > 0 && gamma && ((uintptr_t)gamma & 3u) != 0) return LA_ERR_MISALIGNED;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)B * H;
    if (overlaps(S, BH * dk * dv * 4, z, BH * dk * 4)) return LA_ERR_INVALID_ARG;
    if (N > 0 && gamma &&
        (overlaps(gamma, (size_t)H * 4, S, BH * dk * dv * 4) || overlaps(gamma, (size_t)H * 4, z, BH * dk * 4)))
        return LA_ERR_INVALID_ARG;
    if (N == 0) gamma = nullptr;
    // bf16: the summary phase of the tensor-core non-causal kernel (the final causal
    // state is the non-causal state of the prefix).
    if (dtype == LA_BF16 && N >= 128) {
        st = noncausal_tc_state(k, v, S, z, (int)BH, N, dk, dv, (cudaStream_t)stream, gamma, H, var);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    return state_simt(k, v, S, z, (int)BH, N, dk, dv, dtype, (cudaStream_t)stream, gamma, H, var);
}

la_status la_prefill_state(const void *k, const void *v, float *S, float *z, int B, int H, int N, int dk,
                           int dv, la_dtype dtype, la_stream_t stream)
{
    return la_prefill_state_ex(k, v, nullptr, nullptr, S, z, B, H, N, dk, dv, dtype, stream);
}

la_status la_prefill_state_decay(const void *k, const void *v, const float *gamma, float *S, float *z, int B,
                                 int H, int N, int dk, int dv, la_dtype dtype, la_stream_t stream)
{
    if (!gamma && N > 0 && B > 0 && H > 0 && dk > 0 && dv > 0) return LA_ERR_INVALID_ARG;  // required
    return la_prefill_state_ex(k, v, gamma, nullptr, S, z, B, H, N, dk, dv, dtype, stream);
}

// ---------------------------------------------------------------- gated state
la_status la_forward_causal_gated(const void *q, const void *k, const void *v, void *o, const float *alpha, int B,
                                  int H, int N, int dk, int dv, float eps, la_dtype dtype, la_stream_t stream)
{
    bool empty;
    la_status st = check_forward(q, k, v, o, B, H, N, dk, dv, eps, dtype, &empty);
    if (st != LA_OK || empty) return st;
    if (!alpha) return LA_ERR_INVALID_ARG;
    if (!aligned16(alpha)) return LA_ERR_MISALIGNED;
    const size_t na = (size_t)B * H * N * dk * 4, no = (size_t)B * H * N * dv * elem_size(dtype);
    if (overlaps(alpha, na, o, no)) return LA_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return causal_gated(q, k, v, alpha, o, B * H, N, dk, dv, eps, dtype, (cudaStream_t)stream);
}

la_status la_prefill_state_gated(const void *k, const void *v, const float *alpha, float *S, float *z, int B, int H,
                                 int N, int dk, int dv, la_dtype dtype, la_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || dk == 0 || dv == 0) return LA_OK;
    if (!S || !z) return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z)) return LA_ERR_MISALIGNED;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)B * H;
    if (overlaps(S, BH * dk * dv * 4, z, BH * dk * 4)) return LA_ERR_INVALID_ARG;
    if (N > 0) {
        if (!k || !v || !alpha) return LA_ERR_INVALID_ARG;
        if (!aligned16(k) || !aligned16(v) || !aligned16(alpha)) return LA_ERR_MISALIGNED;
        const size_t es = elem_size(dtype), nk = BH * N * dk * es, nv = BH * N * dv * es, na = BH * N * dk * 4;
        const void *in[3] = {k, v, alpha};
        const size_t ins[3] = {nk, nv, na};
        for (int x = 0; x < 3; ++x)
            if (overlaps(S, BH * dk * dv * 4, in[x], ins[x]) || overlaps(z, BH * dk * 4, in[x], ins[x]))
                return LA_ERR_INVALID_ARG;
    }
    if (N == 0) {  // the empty prefix: zero state
        cudaError_t e = cudaMemsetAsync(S, 0, BH * dk * dv * 4, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, BH * dk * 4, (cudaStream_t)stream);
        count_launches(2);
        return cuda_status(e);
    }
    return state_gated(k, v, alpha, S, z, (int)BH, N, dk, dv, dtype, (cudaStream_t)stream);
}

la_status la_decode_step_gated(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                               const float *alpha, int B, int H, int dk, int dv, float eps, la_dtype dtype,
                               la_stream_t stream)
{
    if (B < 0 || H < 0 || dk < 0 || dv < 0) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || dk == 0 || dv == 0) return LA_OK;
    if (!S || !z || !q || !k || !v || !o || !alpha) return LA_ERR_INVALID_ARG;
    const void *all[7] = {S, z, q, k, v, o, alpha};
    for (const void *x : all)
        if (!aligned16(x)) return LA_ERR_MISALIGNED;
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)B * H, es = elem_size(dtype);
    const size_t sizes[7] = {BH * dk * dv * 4, BH * dk * 4, BH * dk * es, BH * dk * es, BH * dv * es, BH * dv * es,
                             BH * dk * 4};
    const int outs[3] = {0, 1, 5};  // S, z and o are written: they overlap nothing else
    for (int oi : outs)
        for (int x = 0; x < 7; ++x)
            if (x != oi && overlaps(all[oi], sizes[oi], all[x], sizes[x])) return LA_ERR_INVALID_ARG;
    return decode_step_gated(S, z, q, k, v, o, alpha, (int)BH, dk, dv, eps, dtype, (cudaStream_t)stream);
}

la_status la_backward_causal(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk,
                             void *dv, int B, int H, int N, int d_k, int d_v, float eps, la_dtype dtype,
                             la_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || d_k < 0 || d_v < 0) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0 || d_k == 0 || d_v == 0) return LA_OK;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return LA_ERR_INVALID_ARG;
    const void *all[7] = {q, k, v, dout, dq, dk, dv};
    for (const void *x : all)
        if (!aligned16(x)) return LA_ERR_MISALIGNED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return LA_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    const size_t nk = (size_t)B * H * N * d_k * es, nv = (size_t)B * H * N * d_v * es;
    const size_t sizes[7] = {nk, nk, nv, nv, nk, nk, nv};
    for (int o = 4; o < 7; ++o)  // an output overlaps no input and no other output
        for (int x = 0; x < 7; ++x)
            if (x != o && overlaps(all[o], sizes[o], all[x], sizes[x])) return LA_ERR_INVALID_ARG;
    const BackwardProblem p{q, k, v, dout, dq, dk, dv, B * H, N, d_k, d_v, eps, dtype, (cudaStream_t)stream};
    return causal_backward(p);
}

la_status la_favor_features(const void *x, const void *w, void *phi, int B, int H, int N, int d, int m,
                            la_dtype dtype, la_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || d < 0 || m < 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0 || d == 0 || m == 0) return LA_OK;
    if (!x || !w || !phi) return LA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(phi)) return LA_ERR_MISALIGNED;
    if (!supported_dim(d) || !supported_dim(m)) return LA_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype), rows = (size_t)B * H * N;
    if (overlaps(phi, rows * m * es, x, rows * d * es) || overlaps(phi, rows * m * es, w, (size_t)m * d * es))
        return LA_ERR_INVALID_ARG;
    return favor_features(x, nullptr, w, phi, nullptr, B * H, N, d, m, dtype, (cudaStream_t)stream);
}

// Shared steps of the FAVOR+ forwards: checks, then phi(q) and phi(k) into
// stream-ordered scratch (*fq, *fk; [B, H, N, m] each, freed with *s).
static la_status favor_check(const void *q, const void *k, const void *v, const void *o, const void *w, int B,
                             int H, int N, int d, int dv, int m, float eps, la_dtype dtype, bool *empty)
{
    if (m < 0) return LA_ERR_INVALID_ARG;
    la_status st = check_forward(q, k, v, o, B, H, N, d, dv, eps, dtype, empty);
    if (st != LA_OK || *empty) return st;
    if (!w) return LA_ERR_INVALID_ARG;
    if (!aligned16(w)) return LA_ERR_MISALIGNED;
    if (!supported_dim(d) || !supported_dim(dv) || !supported_dim(m)) return LA_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    if (overlaps(o, (size_t)B * H * N * dv * es, w, (size_t)m * d * es)) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

static la_status favor_prologue(const void *q, const void *k, const void *v, const void *o, const void *w, int B,
                                int H, int N, int d, int dv, int m, float eps, la_dtype dtype, cudaStream_t stream,
                                Scratch *s, void **fq, void **fk, bool *empty)
{
    la_status st = favor_check(q, k, v, o, w, B, H, N, d, dv, m, eps, dtype, empty);
    if (st != LA_OK || *empty) return st;
    const size_t es = elem_size(dtype);
    const size_t bytes = (size_t)B * H * N * m * es;  // a multiple of 64: both halves stay 16-byte aligned
    if ((st = s->alloc(2 * bytes, stream)) != LA_OK) return st;
    *fq = s->ptr;
    *fk = (char *)s->ptr + bytes;
    return favor_features(q, k, w, *fq, *fk, B * H, N, d, m, dtype, stream);
}

// The attention half of the FAVOR+ forwards: phi is already applied, so the
// feature map is the identity (shift 0), with the normaliser.
static Variant favor_attention_variant()
{
    Variant v;
    v.map = LA_PHI_IDENTITY;
    v.shift = 0.f;
    v.normalize = 1;
    return v;
}

la_status la_forward_causal_favor(const void *q, const void *k, const void *v, void *o, const void *w, int B, int H,
                                  int N, int d, int dv, int m, int chunk, float eps, la_dtype dtype,
                                  la_stream_t stream)
{
    if (chunk != 64 && chunk != 128) return LA_ERR_UNSUPPORTED;
    Scratch s;
    void *fq = nullptr, *fk = nullptr;
    bool empty;
    la_status st = favor_prologue(q, k, v, o, w, B, H, N, d, dv, m, eps, dtype, (cudaStream_t)stream, &s, &fq, &fk,
                                  &empty);
    if (st != LA_OK || empty) return st;
    Problem p{fq, fk, v, o, B * H, N, m, dv, chunk, eps, dtype, (cudaStream_t)stream, nullptr, H,
              favor_attention_variant()};
    if (dtype == LA_BF16) {
        st = causal_tc(p);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    return causal_simt(p);
}

la_status la_forward_noncausal_favor(const void *q, const void *k, const void *v, void *o, const void *w, int B,
                                     int H, int N, int d, int dv, int m, float eps, la_dtype dtype,
                                     la_stream_t stream)
{
    if (dtype == LA_BF16 && d == 64 && m == 64) {  // the features inside the attention kernel
        bool empty;
        la_status st = favor_check(q, k, v, o, w, B, H, N, d, dv, m, eps, dtype, &empty);
        if (st != LA_OK || empty) return st;
        Problem p{q, k, v, o, B * H, N, d, dv, 0, eps, dtype, (cudaStream_t)stream, nullptr, H, Variant()};
        st = noncausal_tc_favor(p, w);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    Scratch s;
    void *fq = nullptr, *fk = nullptr;
    bool empty;
    la_status st = favor_prologue(q, k, v, o, w, B, H, N, d, dv, m, eps, dtype, (cudaStream_t)stream, &s, &fq, &fk,
                                  &empty);
    if (st != LA_OK || empty) return st;
    Problem p{fq, fk, v, o, B * H, N, m, dv, 0, eps, dtype, (cudaStream_t)stream, nullptr, H,
              favor_attention_variant()};
    if (dtype == LA_BF16) {
        st = noncausal_tc(p);
        if (st != LA_ERR_UNSUPPORTED) return st;
    }
    return noncausal_simt(p);
}

la_status la_prefill_state_favor(const void *k, const void *v, const void *w, float *S, float *z, int B, int H,
                                 int N, int d, int dv, int m, la_dtype dtype, la_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || d < 0 || dv < 0 || m < 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return LA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || dv == 0) return LA_OK;
    if (!supported_dim(m) || !supported_dim(d)) return LA_ERR_UNSUPPORTED;
    const la_variant identity = {LA_PHI_IDENTITY, 0.f, 1};
    if (N == 0)  // no tokens: S and z are zero
        return la_prefill_state_ex(nullptr, nullptr, nullptr, &identity, S, z, B, H, 0, m, dv, dtype, stream);
    if (!k || !v || !w || !S || !z) return LA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(w)) return LA_ERR_MISALIGNED;
    const size_t BH = (size_t)B * H, es = elem_size(dtype), nw = (size_t)m * d * es;
    if (overlaps(S, BH * m * dv * 4, w, nw) || overlaps(z, BH * m * 4, w, nw) ||
        overlaps(S, BH * m * dv * 4, k, BH * N * d * es) || overlaps(z, BH * m * 4, k, BH * N * d * es))
        return LA_ERR_INVALID_ARG;
    const size_t bytes = BH * N * m * es;
    Scratch s;
    la_status st = s.alloc(bytes, (cudaStream_t)stream);
    if (st != LA_OK) return st;
    if ((st = favor_features(k, nullptr, w, s.ptr, nullptr, (int)BH, N, d, m, dtype, (cudaStream_t)stream)) != LA_OK)
        return st;
    return la_prefill_state_ex(s.ptr, v, nullptr, &identity, S, z, B, H, N, m, dv, dtype, stream);
}

la_status la_decode_step_favor(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                               const void *w, int B, int H, int d, int dv, int m, float eps, la_dtype dtype,
                               la_stream_t stream)
{
    if (B < 0 || H < 0 || d < 0 || dv < 0 || m < 0) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || dv == 0) return LA_OK;
    if (!supported_dim(m) || !supported_dim(d)) return LA_ERR_UNSUPPORTED;
    if (!q || !k || !w || !o || !S || !z) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w)) return LA_ERR_MISALIGNED;
    const long long BHl = (long long)B * H;
    if (BHl > 0x7fffffff) return LA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)BHl, es = elem_size(dtype), nw = (size_t)m * d * es;
    if (overlaps(S, BH * m * dv * 4, w, nw) || overlaps(z, BH * m * 4, w, nw) || overlaps(o, BH * dv * es, w, nw) ||
        overlaps(S, BH * m * dv * 4, q, BH * d * es) || overlaps(S, BH * m * dv * 4, k, BH * d * es) ||
        overlaps(z, BH * m * 4, q, BH * d * es) || overlaps(z, BH * m * 4, k, BH * d * es) ||
        overlaps(o, BH * dv * es, q, BH * d * es) || overlaps(o, BH * dv * es, k, BH * d * es))
        return LA_ERR_INVALID_ARG;
    // phi(q) and phi(k) of every head: the rows are independent, so the batch is one
    // sequence of B*H rows (the tensor-core features kernel takes it from 128 rows)
    const size_t bytes = BH * m * es;  // a multiple of 64: both halves stay 16-byte aligned
    Scratch s;
    la_status st = s.alloc(2 * bytes, (cudaStream_t)stream);
    if (st != LA_OK) return st;
    void *fq = s.ptr, *fk = (char *)s.ptr + bytes;
    if ((st = favor_features(q, k, w, fq, fk, 1, (int)BH, d, m, dtype, (cudaStream_t)stream)) != LA_OK) return st;
    const la_variant identity = {LA_PHI_IDENTITY, 0.f, 1};
    return la_decode_step_ex(S, z, fq, fk, v, o, nullptr, &identity, B, H, m, dv, eps, dtype, stream);
}

const char *la_status_string(la_status s)
{
    switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
    case LA_ERR_MISALIGNED: return "LA_ERR_MISALIGNED";
    case LA_ERR_CUDA: return "LA_ERR_CUDA";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
    }
    return "LA_ERR_UNKNOWN";
}

int la_last_cuda_error(void) { return t_last_cuda_error; }

la_status la_get_device_status(la_stream_t stream)
{
    la_status st = cuda_status(cudaStreamSynchronize((cudaStream_t)stream));
    if (st != LA_OK) return st;
    unsigned bits = 0, nc_bits = 0, fv_bits = 0;
    st = tc_causal_read_status((cudaStream_t)stream, &bits);
    if (st != LA_OK) return st;
    st = tc_noncausal_read_status((cudaStream_t)stream, &nc_bits);
    if (st != LA_OK) return st;
    st = favor_read_status((cudaStream_t)stream, &fv_bits);
    if (st != LA_OK) return st;
    unsigned cc_bits = 0, cl_bits = 0, bw_bits = 0;
    st = tc_chunks_read_status((cudaStream_t)stream, &cc_bits);
    if (st != LA_OK) return st;
    st = tc_cluster_read_status((cudaStream_t)stream, &cl_bits);
    if (st != LA_OK) return st;
    st = tc_backward_read_status((cudaStream_t)stream, &bw_bits);
    if (st != LA_OK) return st;
    return ((bits | nc_bits | fv_bits | cc_bits | cl_bits | bw_bits) & kStatusTimeout) ? LA_ERR_TIMEOUT : LA_OK;
}

int la_version(void) { return 100; }

void la_test_set_wait_limit_ns(unsigned long long ns) { g_test_wait_ns.store(ns, std::memory_order_relaxed); }

void la_test_drop_publication(long long ticket) { g_test_drop.store(ticket, std::memory_order_relaxed); }

unsigned long long la_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
