// Recurrent KDA forward: the token-by-token step of the recurrence, for decoding a few
// tokens at a time from a state left by the chunkwise pass (or by an earlier call).
//
// Per token ("TileLang 实战：KDA 从零到一–Kimi Delta Attention", §0 and §3.1; the
// recurrent form of "Gated DeltaNet"):
//   S <- Diag(exp(g_t)) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;  o_t = scale S^T q_t
// (u = v_t without beta: the decay-only recurrence). S [d_k x d_v] fp32.
//
// One CTA of 128 threads runs one (sequence, value head, 32-wide slice of d_v) through
// all its tokens. Column j of the slice belongs to the four lanes 4 (j % 8) + qd of warp
// j / 8 (qd = 0..3); lane qd holds the rows d = qd, qd + 4, ... of S[:, j] in registers,
// so each reduction over d is a sum over the thread's rows and two shuffles. The next
// token's q, k, exp(g), v and beta are staged in shared memory (double-buffered) while
// the current one is computed.
//
// The front-end ("Gated DeltaNet", "Recurrent 算法代码解析") is applied while staging when
// switched on: q and k enter as x / sqrt(sum x^2 + 1e-6) — kept as the raw values and two
// per-token factors, from per-warp partial sums of squares reduced after the staging
// barrier — beta as sigmoid(b), and g as -exp(A_log) * softplus(a + dt_bias).
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kSlice = 32;  // d_v columns per CTA

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int DK, typename T, bool GATE_HEAD>
__global__ void __launch_bounds__(128) kda_recurrent_kernel(const FwdArgs a) {
    constexpr int R = DK / 4;  // rows of S per thread
    constexpr int NW = DK / 32;  // warps that stage q and k
    __shared__ float sq[2][DK], sk[2][DK], sa[2][DK], sv[2][kSlice], sb[2];
    __shared__ float sn[2][NW][2];  // per-warp sums of squares of q and k (front-end norm)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = 8 * warp + (lane >> 2), qd = lane & 3;  // column of the slice, row phase
    const int dv0 = blockIdx.x * kSlice;
    const int h = blockIdx.y, n = blockIdx.z, hk = h / a.group;
    int64_t bos;
    int len;
    if (!seq_bounds(a, n, bos, len)) return;

    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o);
    const int64_t sqk = (int64_t)a.H_k * DK, sv_ = (int64_t)a.H_v * a.d_v;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * DK;
    // front-end constants of this head: -exp(A_log[h]) and this thread's dt_bias
    const bool fe_norm = a.fe_qk_l2norm != 0, fe_gate = a.fe_A_log != nullptr;
    const float negA = fe_gate ? -expf(a.fe_A_log[h]) : 0.f;
    const float bias = (fe_gate && a.fe_dt_bias != nullptr)
                           ? a.fe_dt_bias[GATE_HEAD ? (int64_t)h : (int64_t)h * DK + (tid < DK ? tid : 0)]
                           : 0.f;

    // stage token t into buffer t & 1
    auto stage = [&](int t) {
        const int bsel = t & 1;
        const int64_t row = bos + t;
        if (tid < DK) {  // whole warps (DK is a multiple of 32)
            const float qv = to_f32<T>(q[row * sqk + (int64_t)hk * DK + tid]);
            const float kv = to_f32<T>(k[row * sqk + (int64_t)hk * DK + tid]);
            sq[bsel][tid] = qv;
            sk[bsel][tid] = kv;
            float gv = GATE_HEAD ? a.g[row * sg + h] : a.g[row * sg + (int64_t)h * DK + tid];
            if (fe_gate) gv = gate_f(negA, gv, bias);
            sa[bsel][tid] = exp2f(gv * kLog2e);
            if (fe_norm) {
                float ssq = qv * qv, ssk = kv * kv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
                    ssk += __shfl_xor_sync(0xffffffffu, ssk, o);
                }
                if (lane == 0) {
                    sn[bsel][warp][0] = ssq;
                    sn[bsel][warp][1] = ssk;
                }
            }
        }
        if (tid < kSlice) sv[bsel][tid] = to_f32<T>(v[row * sv_ + (int64_t)h * a.d_v + dv0 + tid]);
        if (tid == 0) {
            float bv = a.decay_only ? 1.f : a.beta[row * a.H_v + h];
            if (a.fe_beta_sigmoid && !a.decay_only) bv = sigmoid_f(bv);
            sb[bsel] = bv;
        }
    };

    // S[:, j] rows qd, qd + 4, ... (from h0, or zero)
    float s[R];
    const int64_t state = ((int64_t)n * a.H_v + h) * DK * a.d_v + dv0 + j;
#pragma unroll
    for (int i = 0; i < R; ++i) s[i] = a.h0 ? a.h0[state + (int64_t)(qd + 4 * i) * a.d_v] : 0.f;

    if (len > 0) stage(0);
    __syncthreads();
    for (int t = 0; t < len; ++t) {
        const int bsel = t & 1;
        if (t + 1 < len) stage(t + 1);  // the other buffer, read by no thread now
        const float *cq = sq[bsel], *ck = sk[bsel], *ca = sa[bsel];
        // the normalised q and k are the staged ones times rq and rk
        float rq = 1.f, rk = 1.f;
        if (fe_norm) {
            float nq = 0.f, nk = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                nq += sn[bsel][w][0];
                nk += sn[bsel][w][1];
            }
            rq = rsqrtf(nq + kL2NormEps);
            rk = rsqrtf(nk + kL2NormEps);
        }
        // decay, then the erase read S^T k
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int d = qd + 4 * i;
            s[i] *= ca[d];
            dot = fmaf(s[i], ck[d], dot);
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        // u scaled by rk once more: the write is k u^T with k = rk * (staged k)
        const float u = rk * (a.decay_only ? sv[bsel][j] : sb[bsel] * (sv[bsel][j] - rk * dot));
        // write, then the output read S^T q
        float oq = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int d = qd + 4 * i;
            s[i] = fmaf(ck[d], u, s[i]);
            oq = fmaf(s[i], cq[d], oq);
        }
        oq += __shfl_xor_sync(0xffffffffu, oq, 1);
        oq += __shfl_xor_sync(0xffffffffu, oq, 2);
        if (qd == 0) o[(bos + t) * sv_ + (int64_t)h * a.d_v + dv0 + j] = from_f32<T>(a.scale * rq * oq);
        __syncthreads();  // buffer t & 1 is free; token t + 1 is staged
    }
    if (a.ht != nullptr) {
#pragma unroll
        for (int i = 0; i < R; ++i) a.ht[state + (int64_t)(qd + 4 * i) * a.d_v] = s[i];
    }
}

template <int DK, typename T>
cudaError_t launch_dk(const FwdArgs &a, cudaStream_t stream) {
    const dim3 grid(a.d_v / kSlice, a.H_v, a.N);
    if (a.gate_per_head)
        kda_recurrent_kernel<DK, T, true><<<grid, 128, 0, stream>>>(a);
    else
        kda_recurrent_kernel<DK, T, false><<<grid, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

// bf16 (f32 = false) or fp32 q/k/v/o; d_k in {64, 128}, d_v a multiple of 32.
cudaError_t launch_recurrent(const FwdArgs &a, bool f32, cudaStream_t stream) {
    if (a.d_k == 128) return f32 ? launch_dk<128, float>(a, stream) : launch_dk<128, __nv_bfloat16>(a, stream);
    return f32 ? launch_dk<64, float>(a, stream) : launch_dk<64, __nv_bfloat16>(a, stream);
}

}  // namespace kda
