// Recurrent KDA forward: the token-by-token step of the recurrence, for decoding a few
// tokens at a time from a state left by the chunkwise pass (or by an earlier call).
//
// Per token ("TileLang 实战：KDA 从零到一–Kimi Delta Attention", §0 and §3.1; the
// recurrent form of "Gated DeltaNet"):
//   S <- Diag(exp(g_t)) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;  o_t = scale S^T q_t
// (u = v_t without beta: the decay-only recurrence). S [d_k x d_v] fp32.
//
// One CTA of 256 threads runs one (sequence, value head) through all its tokens, with the
// whole state in registers, laid out for streaming: thread t owns the four columns
// 4 (t % (d_v / 4)) .. + 3 of the rows r g, r g + 1, ... of its row group g = t / (d_v / 4),
// so that a warp reads and writes whole rows of h0 / ht as 16-byte vectors. The two
// reductions over d_k per token (S^T k and S^T q) are per-thread sums over its rows, then
// a sum over the row groups through shared memory. The next token's q, k, exp(g), v and
// beta are staged in shared memory (double-buffered) while the current one is computed.
//
// The front-end ("Gated DeltaNet", "Recurrent 算法代码解析") is applied while staging when
// switched on: q and k enter as x / sqrt(sum x^2 + 1e-6) — kept as the raw values and two
// per-token factors, from per-warp partial sums of squares reduced after the staging
// barrier — beta as sigmoid(b), and g as -exp(A_log) * softplus(a + dt_bias).
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kThreadsRec = 256;

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

template <int DK, int DV, typename T, bool GATE_HEAD>
__global__ void __launch_bounds__(kThreadsRec) kda_recurrent_kernel(const FwdArgs a) {
    constexpr int NCG = DV / 4;               // column groups of four
    constexpr int RG = kThreadsRec / NCG;     // row groups
    constexpr int RPT = DK / RG;              // rows per thread
    constexpr int NW = DK / 32;               // warps that stage q and k
    __shared__ float sq[2][DK], sk[2][DK], sa[2][DK], sv[2][DV], sb[2];
    __shared__ float sn[2][NW][2];            // per-warp sums of squares of q and k (front-end norm)
    __shared__ __align__(16) float red[RG][DV];  // per-row-group partial sums
    __shared__ __align__(16) float ucol[DV];     // u of the current token

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = tid % NCG, g = tid / NCG;  // column group and row group of this thread
    const int h = blockIdx.x, n = blockIdx.y, hk = h / a.group;
    int64_t bos;
    int len;
    if (!seq_bounds(a, n, bos, len)) return;

    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o);
    const int64_t sqk = (int64_t)a.H_k * DK, sv_ = (int64_t)a.H_v * DV;
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
                for (int o2 = 16; o2 > 0; o2 >>= 1) {
                    ssq += __shfl_xor_sync(0xffffffffu, ssq, o2);
                    ssk += __shfl_xor_sync(0xffffffffu, ssk, o2);
                }
                if (lane == 0) {
                    sn[bsel][warp][0] = ssq;
                    sn[bsel][warp][1] = ssk;
                }
            }
        }
        if (tid < DV) sv[bsel][tid] = to_f32<T>(v[row * sv_ + (int64_t)h * DV + tid]);
        if (tid == 0) {
            float bv = a.decay_only ? 1.f : a.beta[row * a.H_v + h];
            if (a.fe_beta_sigmoid && !a.decay_only) bv = sigmoid_f(bv);
            sb[bsel] = bv;
        }
    };

    // this thread's rows g RPT .. + RPT - 1 (contiguous) and columns 4 cg .. + 3 of S
    float s[RPT][4];
    const int64_t state = ((int64_t)n * a.H_v + h) * DK * DV;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = g * RPT + i;
        if (a.h0 != nullptr) {
            const float4 x = *reinterpret_cast<const float4 *>(a.h0 + state + (int64_t)r * DV + 4 * cg);
            s[i][0] = x.x; s[i][1] = x.y; s[i][2] = x.z; s[i][3] = x.w;
        } else {
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        }
    }

    if (len > 0) stage(0);
    __syncthreads();
    for (int t = 0; t < len; ++t) {
        const int bsel = t & 1;
        if (t + 1 < len) stage(t + 1);  // the other buffer, read by no thread now
        const float *cq = sq[bsel], *ck = sk[bsel], *ca = sa[bsel];
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
        // decay, then the partial erase read (S^T k over this thread's rows)
        float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = g * RPT + i;
            const float dec = ca[r], kr = ck[r];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                s[i][c] *= dec;
                w4[c] = fmaf(s[i][c], kr, w4[c]);
            }
        }
        if (!a.decay_only) {
            *reinterpret_cast<float4 *>(&red[g][4 * cg]) = make_float4(w4[0], w4[1], w4[2], w4[3]);
            __syncthreads();
            if (tid < DV) {
                float wsum = 0.f;
#pragma unroll
                for (int gg = 0; gg < RG; ++gg) wsum += red[gg][tid];
                // u scaled by rk once more: the write is k u^T with k = rk * (staged k)
                ucol[tid] = rk * sb[bsel] * (sv[bsel][tid] - rk * wsum);
            }
        } else if (tid < DV) {
            ucol[tid] = rk * sv[bsel][tid];
        }
        __syncthreads();
        // write, then the partial output read (S^T q over this thread's rows)
        const float4 u4 = *reinterpret_cast<const float4 *>(&ucol[4 * cg]);
        const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
        float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = g * RPT + i;
            const float kr = ck[r], qr = cq[r];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                s[i][c] = fmaf(kr, uu[c], s[i][c]);
                o4[c] = fmaf(s[i][c], qr, o4[c]);
            }
        }
        *reinterpret_cast<float4 *>(&red[g][4 * cg]) = make_float4(o4[0], o4[1], o4[2], o4[3]);
        __syncthreads();
        if (tid < DV) {
            float osum = 0.f;
#pragma unroll
            for (int gg = 0; gg < RG; ++gg) osum += red[gg][tid];
            o[(bos + t) * sv_ + (int64_t)h * DV + tid] = from_f32<T>(a.scale * rq * osum);
        }
        __syncthreads();  // red and buffer t & 1 are free; token t + 1 is staged
    }
    if (a.ht != nullptr) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = g * RPT + i;
            *reinterpret_cast<float4 *>(a.ht + state + (int64_t)r * DV + 4 * cg) =
                make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
        }
    }
}

template <int DK, typename T>
cudaError_t launch_dk(const FwdArgs &a, cudaStream_t stream) {
    const dim3 grid(a.H_v, a.N);
    if (a.d_v == 128) {
        if (a.gate_per_head)
            kda_recurrent_kernel<DK, 128, T, true><<<grid, kThreadsRec, 0, stream>>>(a);
        else
            kda_recurrent_kernel<DK, 128, T, false><<<grid, kThreadsRec, 0, stream>>>(a);
    } else {
        if (a.gate_per_head)
            kda_recurrent_kernel<DK, 64, T, true><<<grid, kThreadsRec, 0, stream>>>(a);
        else
            kda_recurrent_kernel<DK, 64, T, false><<<grid, kThreadsRec, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

// bf16 (f32 = false) or fp32 q/k/v/o; d_k and d_v in {64, 128}.
cudaError_t launch_recurrent(const FwdArgs &a, bool f32, cudaStream_t stream) {
    if (a.d_k == 128) return f32 ? launch_dk<128, float>(a, stream) : launch_dk<128, __nv_bfloat16>(a, stream);
    return f32 ? launch_dk<64, float>(a, stream) : launch_dk<64, __nv_bfloat16>(a, stream);
}

}  // namespace kda
