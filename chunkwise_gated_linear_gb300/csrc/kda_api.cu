// C ABI of the library (declared in include/kda.h): argument checks, dispatch to the
// kernels, status strings and the device error word.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "kda.h"
#include "kda_bwd.h"
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_fwd_bf16(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_pc(const FwdArgs &a, cudaStream_t stream, bool *launched);
cudaError_t launch_fwd_pc_static(const FwdArgs &a, cudaStream_t stream);
int pc_static_max_units();
cudaError_t launch_recurrent(const FwdArgs &a, bool f32, cudaStream_t stream);
cudaError_t launch_frontend(const FwdArgs &a, bool f32, FwdArgs *out, void **scratch, cudaStream_t stream);
}  // namespace kda

namespace {

// One error word per device; its device address is looked up once per device.
__device__ unsigned int g_device_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned int *g_err_ptr[kMaxDevices] = {};

thread_local cudaError_t t_last_cuda_error = cudaSuccess;
thread_local char t_msg[256];

cudaError_t device_error_ptr(unsigned int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_err_mu);
    if (g_err_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error_word);
        if (e != cudaSuccess) return e;
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_err_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the arguments and resolves them into `a` (and its device error word); returns a
// status other than KDA_OK, with nothing launched, when the call is rejected.
int prepare(const kda_fwd_params &p, kda::FwdArgs &a) {
    // With no tokens there is nothing to read or write but the states, so the token
    // tensors may be empty (NULL).
    // (beta may be NULL: the decay-only recurrence)
    if (p.T != 0 && (p.q == nullptr || p.k == nullptr || p.v == nullptr || p.g == nullptr || p.o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (p.B < 1 || p.T < 0 || p.H_k < 1 || p.H_v < 1 || p.H_v % p.H_k != 0) return KDA_ERR_INVALID_ARG;
    if ((p.flags & ~(KDA_FLAG_ONE_CTA_PER_UNIT | KDA_FLAG_UNFUSED_FRONTEND | KDA_FLAG_DEBUG_SHORT_WAITS)) != 0)
        return KDA_ERR_INVALID_ARG;
    if (p.dtype != KDA_DTYPE_BF16 && p.dtype != KDA_DTYPE_F32) return KDA_ERR_UNSUPPORTED;
    if (p.gate_mode != KDA_GATE_PER_CHANNEL && p.gate_mode != KDA_GATE_PER_HEAD) return KDA_ERR_UNSUPPORTED;
    if ((p.d_k != 64 && p.d_k != 128) || (p.d_v != 64 && p.d_v != 128) || p.C != kda::kChunk)
        return KDA_ERR_UNSUPPORTED;
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.o) || !aligned16(p.g) ||
        !aligned16(p.beta) || !aligned16(p.h0) || !aligned16(p.ht))
        return KDA_ERR_ALIGNMENT;
    // Sizes must fit the kernels' 32-bit grid dimensions and the int32 offsets.
    const int64_t N = p.B;
    const int64_t total_tokens = p.cu_seqlens ? (int64_t)p.T : N * p.T;
    if (total_tokens > INT32_MAX || N > 65535 || p.H_v > 65535) return KDA_ERR_UNSUPPORTED;

    a = kda::FwdArgs{};
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.g = p.g;
    a.beta = p.beta;
    a.h0 = p.h0;
    a.o = p.o;
    a.ht = p.ht;
    a.cu_seqlens = p.cu_seqlens;
    a.N = p.B;
    a.T = p.T;
    a.H_k = p.H_k;
    a.H_v = p.H_v;
    a.d_k = p.d_k;
    a.d_v = p.d_v;
    a.group = p.H_v / p.H_k;
    a.scale = p.scale;
    a.gate_per_head = p.gate_mode == KDA_GATE_PER_HEAD ? 1 : 0;
    a.decay_only = p.beta == nullptr ? 1 : 0;
    a.wait_cycles = (p.flags & KDA_FLAG_DEBUG_SHORT_WAITS) ? 1024 : kda::kDefaultWaitCycles;
    return KDA_OK;
}

// Adds the front-end `fe` to resolved arguments; a status other than KDA_OK rejects the
// call with nothing launched.
int prepare_frontend(const kda_frontend *fe, kda::FwdArgs &a) {
    if (fe == nullptr) return KDA_OK;
    if (fe->dt_bias != nullptr && fe->A_log == nullptr) return KDA_ERR_INVALID_ARG;
    if (fe->beta_sigmoid && a.beta == nullptr) return KDA_ERR_INVALID_ARG;
    if (!aligned16(fe->A_log) || !aligned16(fe->dt_bias)) return KDA_ERR_ALIGNMENT;
    a.fe_qk_l2norm = fe->qk_l2norm ? 1 : 0;
    a.fe_beta_sigmoid = fe->beta_sigmoid ? 1 : 0;
    a.fe_A_log = fe->A_log;
    a.fe_dt_bias = fe->dt_bias;
    return KDA_OK;
}

// The forward kernels (the d = 128 bf16 ones apply the fe_* fields themselves; the others
// are only called with them cleared).
cudaError_t dispatch(const kda_fwd_params &p, const kda::FwdArgs &a, cudaStream_t stream) {
    if (p.dtype == KDA_DTYPE_F32) return kda::launch_fwd_f32(a, stream);
    if (p.d_k == 128 && p.d_v == 128) {
        // few units: the persistent producer/consumer kernel, else one CTA per unit
        bool launched = false;
        cudaError_t e = cudaSuccess;
        if (!(p.flags & (KDA_FLAG_ONE_CTA_PER_UNIT | KDA_FLAG_DEBUG_SHORT_WAITS)))
            e = kda::launch_fwd_pc(a, stream, &launched);
        if (e == cudaSuccess && !launched) e = kda::launch_fwd_tc(a, stream);
        return e;
    }
    return kda::launch_fwd_bf16(a, stream);
}

int status_of(cudaError_t e) {
    if (e != cudaSuccess) {
        t_last_cuda_error = e;
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int run(const kda_fwd_params &p, const kda_frontend *fe, cudaStream_t stream) {
    kda::FwdArgs a;
    int st = prepare(p, a);
    if (st == KDA_OK) st = prepare_frontend(fe, a);
    if (st != KDA_OK) return st;
    cudaError_t e = device_error_ptr(&a.err);
    if (e != cudaSuccess) return status_of(e);
    if (!kda::fe_any(a)) return status_of(dispatch(p, a, stream));
    // the d = 128 bf16 kernels (persistent and one CTA per unit) apply the front-end
    // themselves
    if (!(p.flags & KDA_FLAG_UNFUSED_FRONTEND) && p.dtype == KDA_DTYPE_BF16 && p.d_k == 128 && p.d_v == 128)
        return status_of(dispatch(p, a, stream));
    // otherwise a separate pass prepares the inputs in scratch
    kda::FwdArgs b;
    void *scratch = nullptr;
    e = kda::launch_frontend(a, p.dtype == KDA_DTYPE_F32, &b, &scratch, stream);
    if (e == cudaSuccess) e = dispatch(p, b, stream);
    if (scratch != nullptr) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return status_of(e);
}

int run_recurrent(const kda_fwd_params *p, const kda_frontend *fe, cudaStream_t stream) {
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    kda_fwd_params r = *p;
    r.C = kda::kChunk;  // no chunks: C is not used
    kda::FwdArgs a;
    int st = prepare(r, a);
    if (st == KDA_OK) st = prepare_frontend(fe, a);
    if (st != KDA_OK) return st;
    cudaError_t e = device_error_ptr(&a.err);
    if (e != cudaSuccess) return status_of(e);
    const bool f32 = p->dtype == KDA_DTYPE_F32;
    if (!kda::fe_any(a) || !(p->flags & KDA_FLAG_UNFUSED_FRONTEND)) return status_of(kda::launch_recurrent(a, f32, stream));
    kda::FwdArgs b;
    void *scratch = nullptr;
    e = kda::launch_frontend(a, f32, &b, &scratch, stream);
    if (e == cudaSuccess) e = kda::launch_recurrent(b, f32, stream);
    if (scratch != nullptr) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return status_of(e);
}

}  // namespace

extern "C" {

int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const float *h0, void *o, float *ht, int B, int T, int H_k, int H_v, int d_k, int d_v,
                  int C, float scale, const int32_t *cu_seqlens, cudaStream_t stream) {
    kda_fwd_params p{q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale, cu_seqlens,
                     KDA_DTYPE_BF16, KDA_GATE_PER_CHANNEL, 0};
    return run(p, nullptr, stream);
}

int kda_chunk_fwd_f32(const float *q, const float *k, const float *v, const float *g, const float *beta,
                      const float *h0, float *o, float *ht, int B, int T, int H_k, int H_v, int d_k,
                      int d_v, int C, float scale, const int32_t *cu_seqlens, cudaStream_t stream) {
    kda_fwd_params p{q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale, cu_seqlens,
                     KDA_DTYPE_F32, KDA_GATE_PER_CHANNEL, 0};
    return run(p, nullptr, stream);
}

int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g, const float *beta,
                          const float *h0, void *o, float *ht, int B, int T, int H_k, int H_v, int d_k,
                          int d_v, int C, float scale, const int32_t *cu_seqlens, cudaStream_t stream) {
    kda_fwd_params p{q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale, cu_seqlens,
                     KDA_DTYPE_BF16, KDA_GATE_PER_CHANNEL, 0};
    kda::FwdArgs a;
    const int st = prepare(p, a);
    if (st != KDA_OK) return st;
    // only the persistent kernel's shapes, within the static scratch (unit count and head
    // sizes checked on the host before any CUDA call)
    if (d_k != 128 || d_v != 128 || (int64_t)a.N * a.H_v > kda::pc_static_max_units()) return KDA_ERR_UNSUPPORTED;
    cudaError_t e = device_error_ptr(&a.err);
    if (e == cudaSuccess) e = kda::launch_fwd_pc_static(a, stream);
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;  // from host-side checks only
    if (e != cudaSuccess) {
        t_last_cuda_error = e;
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int kda_recurrent_fwd_ex(const kda_fwd_params *p, cudaStream_t stream) { return run_recurrent(p, nullptr, stream); }

int kda_recurrent_fwd_fused(const kda_fwd_params *p, const kda_frontend *fe, cudaStream_t stream) {
    return run_recurrent(p, fe, stream);
}

int kda_recurrent_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                      const float *h0, void *o, float *ht, int B, int T, int H_k, int H_v, int d_k, int d_v,
                      float scale, const int32_t *cu_seqlens, cudaStream_t stream) {
    kda_fwd_params p{q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, kda::kChunk, scale, cu_seqlens,
                     KDA_DTYPE_BF16, KDA_GATE_PER_CHANNEL, 0};
    return kda_recurrent_fwd_ex(&p, stream);
}

int kda_chunk_fwd_ex(const kda_fwd_params *p, cudaStream_t stream) {
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    return run(*p, nullptr, stream);
}

int kda_chunk_bwd(const kda_bwd_params *p, cudaStream_t stream) {
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    // the forward arguments through the forward's own checks (dq stands where o does)
    kda_fwd_params f{p->q, p->k, p->v, p->g, p->beta, p->h0, p->dq, nullptr, p->B, p->T, p->H_k, p->H_v,
                     p->d_k, p->d_v, p->C, p->scale, p->cu_seqlens, p->dtype, p->gate_mode, 0};
    kda::FwdArgs a;
    const int st = prepare(f, a);
    if (st != KDA_OK) return st;
    if (p->flags != 0) return KDA_ERR_INVALID_ARG;
    if (p->T != 0 && (p->dO == nullptr || p->dk == nullptr || p->dv == nullptr || p->dg == nullptr))
        return KDA_ERR_INVALID_ARG;
    if ((p->beta == nullptr) != (p->dbeta == nullptr) && p->T != 0) return KDA_ERR_INVALID_ARG;
    if (!aligned16(p->dO) || !aligned16(p->dht) || !aligned16(p->dk) || !aligned16(p->dv) ||
        !aligned16(p->dg) || !aligned16(p->dbeta) || !aligned16(p->dh0))
        return KDA_ERR_ALIGNMENT;
    kda::BwdArgs b{};
    b.q = p->q;
    b.k = p->k;
    b.v = p->v;
    b.g = p->g;
    b.beta = p->beta;
    b.h0 = p->h0;
    b.dO = p->dO;
    b.dht = p->dht;
    b.dq = p->dq;
    b.dk = p->dk;
    b.dv = p->dv;
    b.dg = p->dg;
    b.dbeta = p->dbeta;
    b.dh0 = p->dh0;
    b.cu_seqlens = p->cu_seqlens;
    b.N = a.N;
    b.T = a.T;
    b.H_k = a.H_k;
    b.H_v = a.H_v;
    b.d_k = a.d_k;
    b.d_v = a.d_v;
    b.group = a.group;
    b.scale = a.scale;
    b.gate_per_head = a.gate_per_head;
    b.decay_only = a.decay_only;
    const cudaError_t e = device_error_ptr(&b.err);
    if (e != cudaSuccess) return status_of(e);
    return status_of(kda::launch_bwd(b, p->dtype == KDA_DTYPE_F32, stream));
}

int kda_chunk_fwd_fused(const kda_fwd_params *p, const kda_frontend *fe, cudaStream_t stream) {
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    return run(*p, fe, stream);
}

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK:
            return "KDA_OK";
        case KDA_ERR_INVALID_ARG:
            return "KDA_ERR_INVALID_ARG: a required pointer is NULL or a size is out of range";
        case KDA_ERR_UNSUPPORTED:
            return "KDA_ERR_UNSUPPORTED: d_k and d_v must be 64 or 128, C must be 64, and the dtype "
                   "and gate mode must be known";
        case KDA_ERR_ALIGNMENT:
            return "KDA_ERR_ALIGNMENT: every tensor pointer must be 16-byte aligned";
        case KDA_ERR_CUDA:
            std::snprintf(t_msg, sizeof(t_msg), "KDA_ERR_CUDA: %s (%s)", cudaGetErrorName(t_last_cuda_error),
                          cudaGetErrorString(t_last_cuda_error));
            return t_msg;
        default:
            return "unknown kda status";
    }
}

int kda_get_device_error(cudaStream_t stream) {
    unsigned int *ptr = nullptr;
    cudaError_t e = device_error_ptr(&ptr);
    unsigned int host = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, ptr, sizeof(host), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, sizeof(unsigned int), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        t_last_cuda_error = e;
        return KDA_ERR_CUDA;
    }
    return static_cast<int>(host);
}

}  // extern "C"
