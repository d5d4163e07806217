// Chunkwise KDA forward in fp32 throughout (CUDA cores).
//
// The same per-chunk steps as the bf16 kernel, for inputs that must be matched to
// single-precision accuracy: every operand stays fp32 and every product is an FFMA
// loop, so nothing is rounded to 16 bits. One CTA of 256 threads runs one
// (sequence, value head, 64-wide slice of d_v) unit through all of its chunks; the
// state slice S [d_k x 64] lives in shared memory.
//
// Per chunk ("TileLang 实战：KDA 从零到一–Kimi Delta Attention", §3.2-3.3;
// "RNN的复兴04:线性注意力并行计算DPLR", §5.3.5):
//   gamma (natural-log gates, chunk-local cumulative sum, log2 domain),
//   Qp = scale Q e^gamma, Kp = K e^gamma, Km = K e^-gamma, Kbar = Km e^gamma_n,
//   M = Kp Km^T (i < r), Aqk = Qp Km^T (i <= r),
//   T = (I + diag(beta) M)^-1 by column-wise forward substitution, T_beta = T diag(beta),
//   W = T_beta Kp, U = T_beta V, Vt = U - W S,
//   O = Qp S + Aqk Vt,  S <- Diag(e^gamma_n) S + Kbar^T Vt.
#include "kda_common.cuh"

namespace kda {

namespace {

template <int DK>
struct F32Layout {
    // Km and W rows are DK + 1 floats apart: the Gram reads Km by row across the lanes of
    // a warp, which would otherwise put all 32 lanes on one shared-memory bank
    static constexpr int LDK = DK + 1;
    static constexpr int oQ = 0;                        // [64][DK]  raw Q, then Qp
    static constexpr int oK = oQ + 64 * DK * 4;         // [64][DK]  raw K, then Kp
    static constexpr int oKm = oK + 64 * DK * 4;        // [64][LDK] Km, then W
    static constexpr int oG = oKm + 64 * LDK * 4;       // [64][DK]  gamma, then Kbar
    static constexpr int oV = oG + 64 * DK * 4;         // [64][64]  V, then U, then Vt
    static constexpr int oS = oV + 64 * 64 * 4;         // [DK][64]  state slice
    static constexpr int oA = oS + DK * 64 * 4;         // [64][64]  Aqk (masked)
    static constexpr int oL = oA + 64 * 64 * 4;         // [64][64]  L
    static constexpr int oT = oL + 64 * 64 * 4;         // [64][64]  T, then T_beta
    static constexpr int oB = oT + 64 * 64 * 4;         // [64]      beta
    static constexpr int oGh = oB + 64 * 4;             // [64]      per-head gates
    static constexpr int oEg = oGh + 64 * 4;            // [DK]      e^gamma_n
    static constexpr int kBytes = oEg + DK * 4;
};

template <int DK, bool GATE_HEAD>
__global__ void __launch_bounds__(256, 1) kda_fwd_f32_kernel(const FwdArgs a) {
    using Lay = F32Layout<DK>;
    constexpr int LDK = Lay::LDK;
    extern __shared__ __align__(128) unsigned char smem[];
    float *Q = reinterpret_cast<float *>(smem + Lay::oQ);
    float *K = reinterpret_cast<float *>(smem + Lay::oK);
    float *Km = reinterpret_cast<float *>(smem + Lay::oKm);
    float *Gs = reinterpret_cast<float *>(smem + Lay::oG);
    float *V = reinterpret_cast<float *>(smem + Lay::oV);
    float *S = reinterpret_cast<float *>(smem + Lay::oS);
    float *A = reinterpret_cast<float *>(smem + Lay::oA);
    float *L = reinterpret_cast<float *>(smem + Lay::oL);
    float *T = reinterpret_cast<float *>(smem + Lay::oT);
    float *Bs = reinterpret_cast<float *>(smem + Lay::oB);
    float *Gh = reinterpret_cast<float *>(smem + Lay::oGh);
    float *Eg = reinterpret_cast<float *>(smem + Lay::oEg);

    const int tid = threadIdx.x;
    const int dv0 = blockIdx.x * 64;
    const int h = blockIdx.y, n = blockIdx.z;
    const int hk = h / a.group;
    int64_t bos;
    int len;
    if (!seq_bounds(a, n, bos, len)) return;
    const int nchunks = (len + kChunk - 1) / kChunk;

    const float *q = static_cast<const float *>(a.q);
    const float *k = static_cast<const float *>(a.k);
    const float *v = static_cast<const float *>(a.v);
    float *o = static_cast<float *>(a.o);
    const int64_t sq = (int64_t)a.H_k * DK;
    const int64_t sv = (int64_t)a.H_v * a.d_v;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * DK;

    for (int i = tid; i < DK * 64; i += 256) {
        const int d = i >> 6, c = i & 63;
        S[i] = a.h0 ? a.h0[((int64_t)n * a.H_v + h) * DK * a.d_v + (int64_t)d * a.d_v + dv0 + c] : 0.f;
    }

    for (int ch = 0; ch < nchunks; ++ch) {
        const int row0 = ch * kChunk;
        const int nvalid = min(kChunk, len - row0);
        __syncthreads();  // the previous chunk is done with every buffer

        for (int i = tid; i < 64 * (DK / 4); i += 256) {
            const int r = i / (DK / 4), c4 = (i % (DK / 4)) * 4;
            float4 zq = make_float4(0.f, 0.f, 0.f, 0.f), zk = zq, zg = zq;
            if (r < nvalid) {
                const int64_t t = bos + row0 + r;
                zq = *reinterpret_cast<const float4 *>(q + t * sq + (int64_t)hk * DK + c4);
                zk = *reinterpret_cast<const float4 *>(k + t * sq + (int64_t)hk * DK + c4);
                if (!GATE_HEAD) zg = *reinterpret_cast<const float4 *>(a.g + t * sg + (int64_t)h * DK + c4);
            }
            *reinterpret_cast<float4 *>(Q + r * DK + c4) = zq;
            *reinterpret_cast<float4 *>(K + r * DK + c4) = zk;
            if (!GATE_HEAD) *reinterpret_cast<float4 *>(Gs + r * DK + c4) = zg;
        }
        for (int i = tid; i < 64 * 16; i += 256) {
            const int r = i >> 4, c4 = (i & 15) * 4;
            float4 zv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nvalid)
                zv = *reinterpret_cast<const float4 *>(v + (bos + row0 + r) * sv + (int64_t)h * a.d_v + dv0 + c4);
            *reinterpret_cast<float4 *>(V + r * 64 + c4) = zv;
        }
        if (tid < 64) {
            const bool ok = tid < nvalid;
            Bs[tid] = ok ? (a.decay_only ? 1.f : a.beta[(bos + row0 + tid) * a.H_v + h]) : 0.f;
            if (GATE_HEAD) Gh[tid] = ok ? a.g[(bos + row0 + tid) * sg + h] : 0.f;
        }
        __syncthreads();

        // gate: one thread per channel walks the 64 rows
        if (tid < DK) {
            const int c = tid;
            float acc = 0.f;
            for (int r = 0; r < 64; ++r) {
                acc += (GATE_HEAD ? Gh[r] : Gs[r * DK + c]) * kLog2e;
                const float ep = exp2f(acc), em = exp2f(-acc);
                const float kv = K[r * DK + c];
                Km[r * LDK + c] = kv * em;
                K[r * DK + c] = a.decay_only ? 0.f : kv * ep;
                Q[r * DK + c] = a.scale * Q[r * DK + c] * ep;
            }
            const float eg = exp2f(acc);
            Eg[c] = eg;
            for (int r = 0; r < 64; ++r) Gs[r * DK + c] = Km[r * LDK + c] * eg;  // Kbar
        }
        __syncthreads();

        // Gram: L = beta_r (Kp Km^T)_ri for i < r, Aqk = (Qp Km^T)_ri for i <= r
        for (int i = tid; i < 64 * 64; i += 256) {
            const int r = i >> 6, c = i & 63;
            float m = 0.f, aq = 0.f;
            if (c <= r) {
                for (int d = 0; d < DK; ++d) {
                    const float km = Km[c * LDK + d];
                    m += K[r * DK + d] * km;
                    aq += Q[r * DK + d] * km;
                }
            }
            L[i] = c < r ? Bs[r] * m : 0.f;
            A[i] = c <= r ? aq : 0.f;
        }
        __syncthreads();

        // T = (I + L)^-1 as a block lower-triangular inverse of 16 x 16 blocks, all in fp32:
        // the diagonal blocks D_k by forward substitution (one column per thread), then
        //   T_{k+1,k} = -D_{k+1} L_{k+1,k} D_k   (k = 0, 2)
        //   T_BA = -T_BB L_BA T_AA                (32 x 32 blocks A = rows 0-31, B = 32-63)
        // with the intermediate products kept in T's unused upper triangle; then
        // T_beta = T diag(beta) on the lower triangle
        if (tid < 64) {
            const int b0 = 16 * (tid >> 4), j = tid & 15;
            float v[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float s = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) s -= L[(b0 + r) * 64 + b0 + m] * v[m];
                v[r] = s;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) T[(b0 + r) * 64 + b0 + j] = v[r];
        }
        __syncthreads();
        for (int e = tid; e < 512; e += 256) {  // P_k = L_{k+1,k} D_k -> upper block (k, k+1)
            const int k = 2 * (e >> 8), r = (e >> 4) & 15, c = e & 15;
            const int lo = 16 * k, hi = lo + 16;
            float s = 0.f;
            for (int m = c; m < 16; ++m) s += L[(hi + r) * 64 + lo + m] * T[(lo + m) * 64 + lo + c];
            T[(lo + r) * 64 + hi + c] = s;
        }
        __syncthreads();
        for (int e = tid; e < 512; e += 256) {  // T_{k+1,k} = -D_{k+1} P_k
            const int k = 2 * (e >> 8), r = (e >> 4) & 15, c = e & 15;
            const int lo = 16 * k, hi = lo + 16;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s += T[(hi + r) * 64 + hi + m] * T[(lo + m) * 64 + hi + c];
            T[(hi + r) * 64 + lo + c] = -s;
        }
        __syncthreads();
        for (int e = tid; e < 1024; e += 256) {  // Y = L_BA T_AA -> upper block rows 0-31, cols 32-63
            const int r = e >> 5, c = e & 31;
            float s = 0.f;
            for (int m = c; m < 32; ++m) s += L[(32 + r) * 64 + m] * T[m * 64 + c];
            T[r * 64 + 32 + c] = s;
        }
        __syncthreads();
        for (int e = tid; e < 1024; e += 256) {  // T_BA = -T_BB Y
            const int r = e >> 5, c = e & 31;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s += T[(32 + r) * 64 + 32 + m] * T[m * 64 + 32 + c];
            T[(32 + r) * 64 + c] = -s;
        }
        __syncthreads();
        for (int e = tid; e < 64 * 64; e += 256) {
            const int r = e >> 6, j = e & 63;
            if (j <= r) T[e] *= Bs[j];
        }
        __syncthreads();

        // W = T_beta Kp (into Km's buffer), U = T_beta V (into V, via registers)
        for (int i = tid; i < 64 * DK; i += 256) {
            const int r = i / DK, d = i % DK;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s += T[r * 64 + m] * K[m * DK + d];
            Km[r * LDK + d] = s;
        }
        float u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int i = tid + 256 * e, r = i >> 6, c = i & 63;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s += T[r * 64 + m] * V[m * 64 + c];
            u[e] = s;
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 16; ++e) V[tid + 256 * e] = u[e];
        __syncthreads();

        // Vt = U - W S (in place: each thread rewrites only the elements it reads)
        for (int i = tid; i < 64 * 64; i += 256) {
            const int r = i >> 6, c = i & 63;
            float s = V[i];
            for (int d = 0; d < DK; ++d) s -= Km[r * LDK + d] * S[d * 64 + c];
            V[i] = s;
        }
        __syncthreads();

        // O = Qp S + Aqk Vt
        for (int i = tid; i < 64 * 64; i += 256) {
            const int r = i >> 6, c = i & 63;
            if (r < nvalid) {
                float s = 0.f;
                for (int d = 0; d < DK; ++d) s += Q[r * DK + d] * S[d * 64 + c];
                for (int m = 0; m <= r; ++m) s += A[r * 64 + m] * V[m * 64 + c];
                o[(bos + row0 + r) * sv + (int64_t)h * a.d_v + dv0 + c] = s;
            }
        }
        __syncthreads();

        // S <- Diag(e^gamma_n) S + Kbar^T Vt
        for (int i = tid; i < DK * 64; i += 256) {
            const int d = i >> 6, c = i & 63;
            float s = Eg[d] * S[i];
            for (int m = 0; m < 64; ++m) s += Gs[m * DK + d] * V[m * 64 + c];
            S[i] = s;
        }
    }
    __syncthreads();
    if (a.ht != nullptr) {
        for (int i = tid; i < DK * 64; i += 256) {
            const int d = i >> 6, c = i & 63;
            a.ht[((int64_t)n * a.H_v + h) * DK * a.d_v + (int64_t)d * a.d_v + dv0 + c] = S[i];
        }
    }
}

template <int DK, bool GATE_HEAD>
cudaError_t launch_f32(const FwdArgs &a, cudaStream_t stream) {
    constexpr int kSmem = F32Layout<DK>::kBytes;
    auto kern = kda_fwd_f32_kernel<DK, GATE_HEAD>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    const dim3 grid(a.d_v / 64, a.H_v, a.N);
    kern<<<grid, 256, kSmem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t stream) {
    if (a.d_k == 128) return a.gate_per_head ? launch_f32<128, true>(a, stream) : launch_f32<128, false>(a, stream);
    return a.gate_per_head ? launch_f32<64, true>(a, stream) : launch_f32<64, false>(a, stream);
}

}  // namespace kda
