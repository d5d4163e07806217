// Front-end as a separate pass: the per-token preparation of the forward pass's inputs
// ("Gated DeltaNet", the model's gate and write strength in "模型调用方式", and the
// recurrent kernel's in-kernel q/k normalisation in "Recurrent 算法代码解析"), written to
// stream-ordered scratch for the kernels that do not apply it in their own staging:
//   q, k  <- x / sqrt(sum_d x_d^2 + 1e-6)          per (token, key head), in the input dtype
//   g     <- -exp(A_log[h]) * softplus(a + dt_bias)  per (token, value head[, channel]), fp32
//   beta  <- 1 / (1 + exp(-b))                       per (token, value head), fp32
// Each part is an HBM-bound elementwise or row pass: coalesced loads and stores, grids
// sized in multiples of the SM count with grid-stride loops.
#include <algorithm>
#include <cstdint>

#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_f32(const T *p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float *p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_f32(T *p, float v);
template <>
__device__ __forceinline__ void st_f32<float>(float *p, float v) {
    *p = v;
}
template <>
__device__ __forceinline__ void st_f32<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

// One warp per row of DK elements; lane l holds elements l, l + 32, ... (coalesced).
template <typename T, int DK>
__global__ void __launch_bounds__(kThreads) l2norm_rows_kernel(const T *__restrict__ x, T *__restrict__ y,
                                                                int64_t rows) {
    constexpr int E = DK / 32;
    const int lane = threadIdx.x & 31;
    const int64_t step = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows; r += step) {
        const T *xr = x + r * DK;
        float v[E];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            v[i] = ld_f32<T>(xr + 32 * i + lane);
            ss = fmaf(v[i], v[i], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss + kL2NormEps);
        T *yr = y + r * DK;
#pragma unroll
        for (int i = 0; i < E; ++i) st_f32<T>(yr + 32 * i + lane, v[i] * inv);
    }
}

// g from the pre-activation, D gate values per (token, value head): D = d_k (per-channel,
// dt_bias [H_v][d_k], four at a time) or 1 (per-head, dt_bias [H_v]).
__global__ void __launch_bounds__(kThreads) gate_kernel(const float *__restrict__ a, float *__restrict__ g,
                                                         const float *__restrict__ A_log,
                                                         const float *__restrict__ dt_bias, int64_t n, int H_v,
                                                         int D) {
    const int64_t step = (int64_t)gridDim.x * kThreads;
    if (D % 4 == 0) {
        const int64_t n4 = n / 4;
        const float4 *a4 = reinterpret_cast<const float4 *>(a);
        float4 *g4 = reinterpret_cast<float4 *>(g);
        for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += step) {
            const int64_t e = 4 * i;
            const int d = (int)(e % D), h = (int)((e / D) % H_v);
            const float negA = -expf(__ldg(A_log + h));
            const float4 x = __ldg(a4 + i);
            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (dt_bias != nullptr) b = __ldg(reinterpret_cast<const float4 *>(dt_bias + (int64_t)h * D + d));
            g4[i] = make_float4(gate_f(negA, x.x, b.x), gate_f(negA, x.y, b.y), gate_f(negA, x.z, b.z),
                                gate_f(negA, x.w, b.w));
        }
    } else {
        for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += step) {
            const int h = (int)((i / D) % H_v);
            const float bias = dt_bias != nullptr ? __ldg(dt_bias + h) : 0.f;
            g[i] = gate_f(-expf(__ldg(A_log + h)), __ldg(a + i), bias);
        }
    }
}

__global__ void __launch_bounds__(kThreads) sigmoid_kernel(const float *__restrict__ b, float *__restrict__ beta,
                                                            int64_t n) {
    const int64_t step = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += step) beta[i] = sigmoid_f(__ldg(b + i));
}

int grid_for(int64_t work, int per_block, int sms) {
    const int64_t want = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 threads per SM
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

template <typename T>
cudaError_t launch_norm(const void *x, void *y, int64_t rows, int d_k, int sms, cudaStream_t stream) {
    const int grid = grid_for(rows, kThreads / 32, sms);
    if (d_k == 128)
        l2norm_rows_kernel<T, 128><<<grid, kThreads, 0, stream>>>(static_cast<const T *>(x), static_cast<T *>(y), rows);
    else
        l2norm_rows_kernel<T, 64><<<grid, kThreads, 0, stream>>>(static_cast<const T *>(x), static_cast<T *>(y), rows);
    return cudaGetLastError();
}

}  // namespace

// Runs the parts of the front-end that `a` switches on, into scratch allocated on `stream`
// from the library's pool (*scratch; nullptr when nothing was needed), and returns in
// *out the arguments of the forward pass over the prepared tensors (front-end switched
// off). The caller frees *scratch on the same stream after launching that pass.
cudaError_t launch_frontend(const FwdArgs &a, bool f32, FwdArgs *out, void **scratch, cudaStream_t stream) {
    *out = a;
    out->fe_qk_l2norm = 0;
    out->fe_beta_sigmoid = 0;
    out->fe_A_log = nullptr;
    out->fe_dt_bias = nullptr;
    *scratch = nullptr;
    const int64_t T = a.cu_seqlens ? (int64_t)a.T : (int64_t)a.N * a.T;
    const int D = a.gate_per_head ? 1 : a.d_k;
    const size_t esz = f32 ? 4 : 2;
    const size_t qk_bytes = a.fe_qk_l2norm ? round256((size_t)T * a.H_k * a.d_k * esz) : 0;
    const size_t g_bytes = a.fe_A_log ? round256((size_t)T * a.H_v * D * 4) : 0;
    const size_t b_bytes = (a.fe_beta_sigmoid && a.beta) ? round256((size_t)T * a.H_v * 4) : 0;
    const size_t total = 2 * qk_bytes + g_bytes + b_bytes;
    if (T == 0 || total == 0) return cudaSuccess;

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaMemPool_t pool = nullptr;
    if (e == cudaSuccess) e = scratch_pool(dev, &pool);
    void *buf = nullptr;
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&buf, total, pool, stream);
    if (e != cudaSuccess) return e;
    *scratch = buf;
    unsigned char *p = static_cast<unsigned char *>(buf);
    if (qk_bytes) {
        const int64_t rows = T * a.H_k;
        out->q = p;
        out->k = p + qk_bytes;
        if (f32) {
            e = launch_norm<float>(a.q, p, rows, a.d_k, sms, stream);
            if (e == cudaSuccess) e = launch_norm<float>(a.k, p + qk_bytes, rows, a.d_k, sms, stream);
        } else {
            e = launch_norm<__nv_bfloat16>(a.q, p, rows, a.d_k, sms, stream);
            if (e == cudaSuccess) e = launch_norm<__nv_bfloat16>(a.k, p + qk_bytes, rows, a.d_k, sms, stream);
        }
        if (e != cudaSuccess) return e;
        p += 2 * qk_bytes;
    }
    if (g_bytes) {
        const int64_t n = T * a.H_v * D;
        float *g = reinterpret_cast<float *>(p);
        gate_kernel<<<grid_for(D % 4 == 0 ? n / 4 : n, kThreads, sms), kThreads, 0, stream>>>(
            a.g, g, a.fe_A_log, a.fe_dt_bias, n, a.H_v, D);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        out->g = g;
        p += g_bytes;
    }
    if (b_bytes) {
        const int64_t n = T * a.H_v;
        float *beta = reinterpret_cast<float *>(p);
        sigmoid_kernel<<<grid_for(n, kThreads, sms), kThreads, 0, stream>>>(a.beta, beta, n);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        out->beta = beta;
    }
    return cudaSuccess;
}

}  // namespace kda
