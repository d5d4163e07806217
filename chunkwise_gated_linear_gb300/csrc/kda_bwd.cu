// Chunkwise backward pass of the gated delta rule (fp32 arithmetic throughout).
//
// Gradients of sum(dO * O) + sum(dht * ht) with respect to q, k, v, g, beta and h0, in the
// chunk form that "Gated DeltaNet" lays out in "反向传播：状态伴随与三角变换梯度": the chunk
// factors are recomputed, the state adjoint runs backwards from dht through the chunks,
// and the gradients of the WY factors are carried back through the triangular inverse.
// With gamma the chunk-local cumulative log gate and Gn its value at the chunk's last
// token, the forward chunk is (all per unit, 64 tokens):
//   Qp = scale Q e^g, Kp = K e^g, Km = K e^-g, Kb = K e^(Gn - g), EG = e^Gn
//   M = strict_lower(Kp Km^T), A = lower(Qp Km^T), T = (I + diag(beta) M)^-1
//   W = T diag(beta) Kp, U = T diag(beta) V, Vt = U - W S, O = Qp S + A Vt,
//   S' = diag(EG) S + Kb^T Vt
// and, for the adjoint dS' of the chunk's exit state:
//   dVt = A^T dO + Kb dS',  dS = diag(EG) dS' + Qp^T dO - W^T dVt
//   dQp = dO S^T + dA Km (dA = lower(dO Vt^T)),  dKb = Vt dS'^T,  dW = -dVt S^T
//   dT = (dW Kp^T + dVt V^T) diag(beta),  dL = -T^T dT T^T (strictly lower)
//   dKp = diag(beta) T^T dW + diag(beta) dL Km,  dKm = (diag(beta) dL)^T Kp + dA^T Qp
//   dV = diag(beta) T^T dVt,  dbeta = rows of (T^T dW . Kp) + (T^T dVt . V) + (dL . M)
//   dQ = scale e^g dQp,  dK = e^g dKp + e^-g dKm + e^(Gn - g) dKb
//   dgamma = dQp.Qp + dKp.Kp - dKm.Km - dKb.Kb,  dGn = sum_t dKb.Kb + dEG.EG,
//   dg = reverse cumulative sum of dgamma over the chunk's tokens, plus dGn
// (decay-only: Kp = 0, beta = 1, so T = I, W = 0, U = V and dV = dVt).
//
// Five kernels, all on stream-ordered scratch from the library's pool:
//   prep     (chunk, unit) parallel: gamma, Qp, Kp, Km, Kb, EG, M, A, T, W, U, V, dO (and
//            the transposed copies the tcgen05 gradient kernel reads)
//   states   (unit, 64 columns of d_v): the forward state scan, storing S and Vt per chunk
//   adjoint  (unit, 64 columns of d_v): the reverse scan of dS, storing dS' and dVt per
//            chunk, and dh0
//   grads    (chunk, unit) parallel: every gradient above; dq and dk written directly when
//            each key head has one value head, else added atomically into fp32
//            accumulators (value heads that share a key head add into the same rows)
//   finish   the accumulators to the output dtype (grouped heads, bf16 outputs)
// For bf16 inputs with d_k = d_v = 128 the two scans run on tcgen05 (kind::tf32, the state
// or its adjoint in TMEM), and with beta the gradient kernel as well (bwd_*_tc_kernel). The
// other contractions go through one CTA-wide GEMM on tf32 mma.sync (block_gemm: 64 x 64
// output tiles, 32-deep k steps staged in shared memory, fp32 accumulation).
#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "kda_bwd.h"
#include "kda_common.cuh"
#include "tc5_tf32.cuh"
#include "tc_util.cuh"

namespace kda {

namespace {

constexpr int kT = 512;            // threads of every backward kernel
constexpr int kKS = 32;             // k step of the GEMM
constexpr int kLoads = 64 * kKS / kT;  // staged elements of each operand tile per thread and k step

// Per-slot scratch layout (floats). A slot holds one chunk of one unit. Every array starts
// on a multiple of 128 floats, so that the slot can be viewed as rows of 64 or 128 floats by
// the tensor maps of the tcgen05 gradient kernel. The transposed copies (qpt, kpt, kmt: [d][t];
// tt = T^T, tbt = diag(beta) T^T; dvtt = dVt^T [v][t]) are written only for that kernel.
struct Lay {
    int64_t qp, kp, km, kb, wm, gm, u, vf, dof, vt, dvt, m, a, t, eg, bt, se, dsx;
    int64_t qpt, kpt, kmt, tt, tbt, dvtt, total;
};
__host__ __device__ inline Lay make_lay(int K, int V) {
    Lay L;
    int64_t o = 0;
    auto take = [&](int64_t n) {
        const int64_t at = o;
        o += (n + 127) & ~(int64_t)127;
        return at;
    };
    L.qp = take(64 * K); L.kp = take(64 * K); L.km = take(64 * K); L.kb = take(64 * K);
    L.wm = take(64 * K); L.gm = take(64 * K);
    L.u = take(64 * V); L.vf = take(64 * V); L.dof = take(64 * V); L.vt = take(64 * V); L.dvt = take(64 * V);
    L.m = take(64 * 64); L.a = take(64 * 64); L.t = take(64 * 64);
    L.eg = take(K); L.bt = take(64);
    L.se = take((int64_t)K * V); L.dsx = take((int64_t)K * V);
    L.qpt = take(64 * K); L.kpt = take(64 * K); L.kmt = take(64 * K);
    L.tt = take(64 * 64); L.tbt = take(64 * 64); L.dvtt = take(64 * V);
    L.total = o;
    return L;
}

template <typename T>
__device__ __forceinline__ void stf(T *p, float v);
template <>
__device__ __forceinline__ void stf<float>(float *p, float v) {
    *p = v;
}
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Four consecutive elements of a tensor that nothing writes while the kernel runs, through
// the read-only path (so that the compiler may issue the loads of later iterations ahead of
// earlier stores), as floats; zeros when !ok. p is 16-byte (fp32) or 8-byte (bf16) aligned.
template <typename T>
__device__ __forceinline__ float4 ld4(const T *p, bool ok);
template <>
__device__ __forceinline__ float4 ld4<float>(const float *p, bool ok) {
    return ok ? __ldg(reinterpret_cast<const float4 *>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p, bool ok) {
    if (!ok) return make_float4(0.f, 0.f, 0.f, 0.f);
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));  // element 0 in the low half
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
// Four consecutive outputs (16-byte aligned fp32, 8-byte aligned bf16, rounded to nearest).
template <typename T>
__device__ __forceinline__ void st4(T *p, float4 v);
template <>
__device__ __forceinline__ void st4<float>(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ float4 ld4f(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4f(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// tf32 tensor-core product on split operands: x = hi + lo with hi = tf32(x), lo = tf32(x -
// hi); a b ~ hi_a hi_b + hi_a lo_b + lo_a hi_b ("3xTF32"), whose error is about that of an
// fp32 product (the dropped lo_a lo_b term is below 2^-22 relative).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// C(m, n) = alpha * sum_k A(m, k) B(k, n) (+ C(m, n) when acc), fp32, every matrix given by
// a base pointer (global or shared) and element strides: A(m, k) = A[m * am + k * ak],
// B(k, n) = B[k * bk + n * bn], C(m, n) = C[m * cm + n * cn]. M and N are multiples of 64,
// K of 32; C must not overlap A or B. Called by all kT threads; ends with a barrier.
// Each 64 x 64 output tile is split over the 16 warps as 16 x 16 blocks (two m16n8
// accumulators per warp) on tf32 mma.sync: with SPLIT the operands are split (3xTF32,
// fp32-grade products; fp32 inputs), else rounded to tf32 once (10-bit mantissa products,
// fp32 accumulation; bf16 inputs, whose gradients are rounded to bf16 or compared at that
// level; the rounding is done once per element, when it is staged). The operand tiles go
// through shared memory in 32-deep k steps, the next one fetched into registers while the
// current one is multiplied.
constexpr int kSP = 72;  // row stride of a tile staged [k][64] (conflict-free fragment reads)
constexpr int kSA = 36;  // row stride of a tile staged [64][k]
static_assert(64 * kSA <= kKS * kSP, "both layouts fit one stage");
constexpr int kStageFloats = 2 * kKS * kSP;
template <bool SPLIT>
__device__ void block_gemm(int M, int N, int K, float alpha, const float *A, int64_t am, int64_t ak,
                           const float *B, int64_t bk, int64_t bn, float *C, int64_t cm, int64_t cn, bool acc,
                           float *stage) {
    static_assert(kT == 512 && kKS == 32, "16 warps: 4 x 4 blocks of 16 x 16 per 64 x 64 tile");
    float *As = stage, *Bs = stage + kKS * kSP;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int mb = (warp & 3) * 16, nb = (warp >> 2) * 16;
    for (int m0 = 0; m0 < M; m0 += 64) {
        for (int n0 = 0; n0 < N; n0 += 64) {
            float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float ra[kLoads], rb[kLoads];
            // Element r of this thread's share of the staged tiles: e = tid + kT r. With the k
            // index fastest (ak == 1) k = lane and m = e / 32; else m = tid % 64 and k = e / 64.
            // Its global offset and shared-memory slot are a base plus r times a step, and
            // move by k0 * ak (k0 * bk) from one k step to the next. A tile is staged in the
            // order of its source, [m][k] (row stride kSA) when k is contiguous, else [k][m]
            // (row stride kSP), and B likewise: both the staging stores and the fragment reads
            // are then free of bank conflicts.
            const bool akf = ak == 1, bnf = bn == 1;
            const int sam = akf ? kSA : 1, sak = akf ? 1 : kSP;    // A(m, k) at As[m sam + k sak]
            const int sbk = bnf ? kSP : 1, sbn = bnf ? 1 : kSA;    // B(k, n) at Bs[k sbk + n sbn]
            const int ma = akf ? (tid >> 5) : (tid & 63), ka = akf ? lane : (tid >> 6);
            const int64_t a_base = (int64_t)(m0 + ma) * am + (int64_t)ka * ak;
            const int64_t a_step = akf ? 16 * am : 8 * ak;  // r -> r + 1 (kT = 512, kKS = 32)
            const int as_base = ma * sam + ka * sak, as_step = akf ? 16 * kSA : 8 * kSP;
            const int nb_ = bnf ? (tid & 63) : (tid >> 5), kb_ = bnf ? (tid >> 6) : lane;
            const int64_t b_base = (int64_t)kb_ * bk + (int64_t)(n0 + nb_) * bn;
            const int64_t b_step = bnf ? 8 * bk : 16 * bn;
            const int bs_base = kb_ * sbk + nb_ * sbn, bs_step = bnf ? 8 * kSP : 16 * kSA;
            // fragment offsets: A(mb + g, t), B(t, nb + g)
            const int fa = (mb + g) * sam + t * sak, fb = t * sbk + (nb + g) * sbn;
            auto fetch = [&](int k0) {
                const float *Ak = A + (int64_t)k0 * ak + a_base;
                const float *Bk = B + (int64_t)k0 * bk + b_base;
#pragma unroll
                for (int r = 0; r < kLoads; ++r) {
                    ra[r] = Ak[r * a_step];
                    rb[r] = Bk[r * b_step];
                }
            };
            fetch(0);
            for (int k0 = 0; k0 < K; k0 += kKS) {
                // without SPLIT the operands are rounded to tf32 here, once per element, and
                // the fragments below are read as they are
#pragma unroll
                for (int r = 0; r < kLoads; ++r) {
                    As[as_base + r * as_step] = SPLIT ? ra[r] : __uint_as_float(to_tf32(ra[r]));
                    Bs[bs_base + r * bs_step] = SPLIT ? rb[r] : __uint_as_float(to_tf32(rb[r]));
                }
                __syncthreads();
                if (k0 + kKS < K) fetch(k0 + kKS);
#pragma unroll
                for (int k8 = 0; k8 < kKS; k8 += 8) {
                    // A (16 x 8): rows mb + g, mb + g + 8; columns k8 + t, k8 + t + 4
                    const float *Af = As + fa + k8 * sak;
                    const float a0 = Af[0], a1 = Af[8 * sam], a2 = Af[4 * sak], a3 = Af[8 * sam + 4 * sak];
                    uint32_t ah[4], al[4];
                    if constexpr (SPLIT) {
                        split_tf32(a0, ah[0], al[0]);
                        split_tf32(a1, ah[1], al[1]);
                        split_tf32(a2, ah[2], al[2]);
                        split_tf32(a3, ah[3], al[3]);
                    } else {
                        ah[0] = __float_as_uint(a0);
                        ah[1] = __float_as_uint(a1);
                        ah[2] = __float_as_uint(a2);
                        ah[3] = __float_as_uint(a3);
                    }
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        // B (8 x 8): rows k8 + t, k8 + t + 4; column nb + 8 f + g
                        const float *Bf = Bs + fb + k8 * sbk + 8 * f * sbn;
                        const float b0 = Bf[0], b1 = Bf[4 * sbk];
                        if constexpr (SPLIT) {
                            uint32_t bh0, bl0, bh1, bl1;
                            split_tf32(b0, bh0, bl0);
                            split_tf32(b1, bh1, bl1);
                            mma_m16n8k8_tf32(c[f], al, bh0, bh1);
                            mma_m16n8k8_tf32(c[f], ah, bl0, bl1);
                            mma_m16n8k8_tf32(c[f], ah, bh0, bh1);
                        } else {
                            mma_m16n8k8_tf32(c[f], ah, __float_as_uint(b0), __float_as_uint(b1));
                        }
                    }
                }
                __syncthreads();
            }
            // The accumulators of a row half (c[f][2 hq + qi]: row mb + g + 8 hq, column nb +
            // 8 f + 2 t + qi) go out in four rounds; in round rr lane g writes choice (g + rr)
            // % 4 of (f, qi), so that one store touches 16 columns instead of 4 (C's rows are
            // often a multiple of 32 words apart in shared memory: 2-way instead of 8-way
            // bank conflicts).
#pragma unroll
            for (int hq = 0; hq < 2; ++hq)
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int j = (g + rr) & 3, f = j >> 1, qi = j & 1;
                    const float v0 = qi ? c[0][2 * hq + 1] : c[0][2 * hq];
                    const float v1 = qi ? c[1][2 * hq + 1] : c[1][2 * hq];
                    const float v = f ? v1 : v0;
                    const int m = m0 + mb + g + 8 * hq, n = n0 + nb + 8 * f + 2 * t + qi;
                    float *p = C + (int64_t)m * cm + (int64_t)n * cn;
                    *p = acc ? fmaf(alpha, v, *p) : alpha * v;
                }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// Sequence bounds (fixed-length batches or packed sequences); false, with the device error
// bit raised, when the offsets are malformed (the sequence is then skipped).
__device__ __forceinline__ bool bounds(const BwdArgs &a, int n, int64_t &bos, int &len) {
    if (a.cu_seqlens == nullptr) {
        bos = (int64_t)n * a.T;
        len = a.T;
        return true;
    }
    const int s = a.cu_seqlens[n], e = a.cu_seqlens[n + 1];
    if (s < 0 || e < s || e > a.T) {
        if (threadIdx.x == 0) atomicOr(a.err, kDeviceErrSeqlens);
        bos = 0;
        len = 0;
        return false;
    }
    bos = s;
    len = e - s;
    return true;
}
// Slot of chunk c of sequence n (value head h): (bos / 64 + c + n) * H_v + h. Chunks of
// different sequences never share a slot (there are at most T / 64 + N windows).
__device__ __forceinline__ int64_t slot_of(const BwdArgs &a, int64_t bos, int n, int c, int h) {
    return ((bos >> 6) + c + n) * a.H_v + h;
}
// The (sequence, chunk) that owns window s, or false when none does.
__device__ bool window_owner(const BwdArgs &a, int64_t s, int &n, int &c, int64_t &bos, int &len) {
    // the largest n with bos_n / 64 + n <= s (strictly increasing in n)
    int lo = 0, hi = a.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        int64_t b;
        int l;
        bounds(a, mid, b, l);
        if ((b >> 6) + mid <= s) lo = mid; else hi = mid - 1;
    }
    n = lo;
    if (!bounds(a, n, bos, len)) return false;
    const int64_t cc = s - (bos >> 6) - n;
    if (cc < 0 || cc * 64 >= len) return false;
    c = (int)cc;
    return true;
}

// ---- prep: the chunk factors -----------------------------------------------------------------
// Shared memory: GEMM stage, L and T [64][65], gamma [64][K].
size_t prep_smem(int K) { return sizeof(float) * ((size_t)kStageFloats + 2 * 64 * 65 + 64 * (size_t)K); }

// two CTAs per SM (64 registers a thread): the kernel is latency-bound
template <typename T, bool GATE_HEAD>
__global__ void __launch_bounds__(kT, 2) bwd_prep_kernel(const BwdArgs a) {
    constexpr bool SPLIT = std::is_same<T, float>::value;
    extern __shared__ __align__(16) float psm[];
    float *stage = psm, *Lsh = stage + kStageFloats, *Tsh = Lsh + 64 * 65;
    float *Gs = Tsh + 64 * 65;
    int n, c, len;
    int64_t bos;
    if (!window_owner(a, blockIdx.y, n, c, bos, len)) return;
    const int h = blockIdx.x, hk = h / a.group, K = a.d_k, V = a.d_v;
    const Lay L = make_lay(K, V);
    float *S = a.scratch + slot_of(a, bos, n, c, h) * L.total;
    const int row0 = c * 64, nv = min(64, len - row0);
    const int tid = threadIdx.x;
    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const T *dO = static_cast<const T *>(a.dO);
    const int64_t sqk = (int64_t)a.H_k * K, sv = (int64_t)a.H_v * V;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * K;

    // gamma (natural log), per channel: the gate tile into shared memory (rows past the end
    // zero, so that they keep the last valid value), then a running sum per channel. The
    // element loops below take four consecutive channels (or value columns) of one token per
    // step: e4 indexes float4 groups, 4 e4 = t K + i.
    const int pk = K / 4, pv = V / 4;
#pragma unroll 4
    for (int e4 = tid; e4 < 16 * K; e4 += kT) {
        const int t = e4 / pk, i = 4 * (e4 - t * pk);
        const int64_t r = bos + row0 + t;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nv) {
            if (GATE_HEAD) {
                const float x = __ldg(a.g + r * sg + h);
                gv = make_float4(x, x, x, x);
            } else {
                gv = __ldg(reinterpret_cast<const float4 *>(a.g + r * sg + (int64_t)h * K + i));
            }
        }
        st4f(Gs + 4 * e4, gv);
    }
    __syncthreads();
    for (int i = tid; i < K; i += kT) {
        float acc = 0.f;
        for (int t = 0; t < 64; ++t) {
            acc += Gs[t * K + i];
            Gs[t * K + i] = acc;
        }
        S[L.eg + i] = expf(acc);
    }
    __syncthreads();
    for (int e4 = tid; e4 < 16 * K; e4 += kT) st4f(S + L.gm + 4 * e4, ld4f(Gs + 4 * e4));
    for (int t = tid; t < 64; t += kT)
        S[L.bt + t] = t < nv ? (a.decay_only ? 1.f : a.beta[(bos + row0 + t) * a.H_v + h]) : 0.f;
    // Qp, Kp, Km, Kb, and diag(beta) Kp for the W product (in the dS' area, free until the
    // adjoint scan)
    float *Kbeta = S + L.dsx;
#pragma unroll 2
    for (int e4 = tid; e4 < 16 * K; e4 += kT) {
        const int t = e4 / pk, i = 4 * (e4 - t * pk);
        const int64_t r = bos + row0 + t;
        const bool ok = t < nv;
        const float4 k4 = ld4<T>(k + r * sqk + (int64_t)hk * K + i, ok);
        const float4 q4 = ld4<T>(q + r * sqk + (int64_t)hk * K + i, ok);
        const float bt = ok ? (a.decay_only ? 1.f : __ldg(a.beta + r * a.H_v + h)) : 0.f;
        const float4 g4 = ld4f(Gs + 4 * e4), n4 = ld4f(Gs + 63 * K + i);
        const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
        const float gam[4] = {g4.x, g4.y, g4.z, g4.w}, gn[4] = {n4.x, n4.y, n4.z, n4.w};
        float qp[4], kp[4], km[4], kb[4], kbt[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            qp[j] = a.scale * qv[j] * expf(gam[j]);
            kp[j] = a.decay_only ? 0.f : kv[j] * expf(gam[j]);
            km[j] = kv[j] * expf(-gam[j]);
            kb[j] = kv[j] * expf(gn[j] - gam[j]);
            kbt[j] = bt * kp[j];
        }
        st4f(S + L.qp + 4 * e4, make_float4(qp[0], qp[1], qp[2], qp[3]));
        st4f(S + L.kp + 4 * e4, make_float4(kp[0], kp[1], kp[2], kp[3]));
        st4f(S + L.km + 4 * e4, make_float4(km[0], km[1], km[2], km[3]));
        st4f(S + L.kb + 4 * e4, make_float4(kb[0], kb[1], kb[2], kb[3]));
        st4f(Kbeta + 4 * e4, make_float4(kbt[0], kbt[1], kbt[2], kbt[3]));
    }
    // V, dO, and diag(beta) V for the U product (in the dVt area, free until the adjoint scan)
    float *Vbeta = S + L.dvt;
#pragma unroll 2
    for (int e4 = tid; e4 < 16 * V; e4 += kT) {
        const int t = e4 / pv, j = 4 * (e4 - t * pv);
        const int64_t r = bos + row0 + t;
        const bool ok = t < nv;
        const float4 v4 = ld4<T>(v + r * sv + (int64_t)h * V + j, ok);
        const float4 o4 = ld4<T>(dO + r * sv + (int64_t)h * V + j, ok);
        const float bt = ok ? (a.decay_only ? 1.f : __ldg(a.beta + r * a.H_v + h)) : 0.f;
        st4f(S + L.vf + 4 * e4, v4);
        st4f(S + L.dof + 4 * e4, o4);
        st4f(Vbeta + 4 * e4, make_float4(bt * v4.x, bt * v4.y, bt * v4.z, bt * v4.w));
    }
    __syncthreads();
    // M = Kp Km^T (strictly lower), A = Qp Km^T (lower with the diagonal)
    block_gemm<SPLIT>(64, 64, K, 1.f, S + L.kp, K, 1, S + L.km, 1, K, S + L.m, 64, 1, false, stage);
    block_gemm<SPLIT>(64, 64, K, 1.f, S + L.qp, K, 1, S + L.km, 1, K, S + L.a, 64, 1, false, stage);
    for (int e = tid; e < 64 * 64; e += kT) {
        const int t = e >> 6, s = e & 63;
        if (s >= t) S[L.m + e] = 0.f;
        if (s > t) S[L.a + e] = 0.f;
        Lsh[t * 65 + s] = s < t ? S[L.bt + t] * S[L.m + e] : 0.f;  // L = diag(beta) M
    }
    __syncthreads();
    // T = (I + L)^-1 in 16 x 16 blocks. The four diagonal blocks at once: column c of block
    // b solves (I + L_bb) x = e_c by forward substitution over the block's rows, x_i = [i ==
    // c] - sum_{c <= k < i} L[i][k] x_k, eight lanes of one warp per column (k = c + sub,
    // c + sub + 8) adding their parts by shuffles. Then the blocks below the diagonal, one
    // sub-diagonal d at a time: T_(j+d) j = -T_(j+d)(j+d) sum_{j <= k < j+d} L_(j+d) k T_kj.
    {
        static_assert(kT == 512, "16 warps x 4 columns");
        const int lane = tid & 31, sub = lane & 7, c = 4 * (tid >> 5) + (lane >> 3);
        const int b0 = c & ~15;
        for (int i = b0; i < b0 + 16; ++i) {
            float part = 0.f;
            for (int kk = c + sub; kk < i; kk += 8) part = fmaf(Lsh[i * 65 + kk], Tsh[kk * 65 + c], part);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            if (sub == 0) Tsh[i * 65 + c] = (i == c ? 1.f : 0.f) - part;
            __syncwarp();
        }
        for (int e = tid; e < 4096; e += kT) {
            const int r = e >> 6, cc = e & 63;
            if ((r >> 4) < (cc >> 4)) Tsh[r * 65 + cc] = 0.f;
        }
        __syncthreads();
        float *P = stage;  // sum_k L_(j+d) k T_kj of each block of the sub-diagonal [j][16][16]
        for (int d = 1; d < 4; ++d) {
            const int nb = 4 - d;
            for (int e = tid; e < nb * 256; e += kT) {
                const int j = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                const int row = 16 * (j + d) + r, col = 16 * j + cc;
                float acc = 0.f;
                for (int kk = 16 * j; kk < 16 * (j + d); ++kk) acc = fmaf(Lsh[row * 65 + kk], Tsh[kk * 65 + col], acc);
                P[e] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nb * 256; e += kT) {
                const int j = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                const int row = 16 * (j + d) + r, col = 16 * j + cc;
                float acc = 0.f;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) acc = fmaf(Tsh[row * 65 + 16 * (j + d) + kk], P[(j << 8) + kk * 16 + cc], acc);
                Tsh[row * 65 + col] = -acc;
            }
            __syncthreads();
        }
    }
    float *Tm = S + L.t;
    for (int e = tid; e < 4096; e += kT) Tm[e] = Tsh[(e >> 6) * 65 + (e & 63)];
    if (a.tc) {
        // T^T and diag(beta) T^T ([t][r], r fastest: the shared-memory reads are 65 apart)
        for (int e = tid; e < 4096; e += kT) {
            const int t = e >> 6, r = e & 63;
            const float x = Tsh[r * 65 + t];
            S[L.tt + e] = x;
            S[L.tbt + e] = S[L.bt + t] * x;
        }
        // Qp^T, Kp^T, Km^T [d][t] from the row-major copies this CTA wrote above (plain
        // loads: they were written in this kernel), t fastest so that the stores coalesce
        for (int e = tid; e < 16 * K; e += kT) {
            const int t = e & 63, d0 = 4 * (e >> 6);
            const float4 x = ld4f(S + L.qp + t * K + d0), y = ld4f(S + L.kp + t * K + d0),
                         z = ld4f(S + L.km + t * K + d0);
            const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w}, zs[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                S[L.qpt + (d0 + j) * 64 + t] = xs[j];
                S[L.kpt + (d0 + j) * 64 + t] = ys[j];
                S[L.kmt + (d0 + j) * 64 + t] = zs[j];
            }
        }
    }
    // W = T diag(beta) Kp, U = T diag(beta) V (the row-scaled operands were written above)
    block_gemm<SPLIT>(64, V, 64, 1.f, Tsh, 65, 1, Vbeta, V, 1, S + L.u, V, 1, false, stage);
    block_gemm<SPLIT>(64, K, 64, 1.f, Tsh, 65, 1, Kbeta, K, 1, S + L.wm, K, 1, false, stage);
}

// Copy `rows` rows of `cols` floats (a multiple of 4; every row start 16-byte aligned)
// global -> shared with cp.async, all kT threads; global row stride `stride`, shared row
// stride `dstride`.
__device__ __forceinline__ void stage_rows(float *dst, int dstride, const float *src, int rows, int cols,
                                           int64_t stride) {
    const int per = cols / 4;
    for (int e = threadIdx.x; e < rows * per; e += kT) {
        const int r = e / per, c4 = e - r * per;
        cp_async_16(dst + r * dstride + 4 * c4, src + r * stride + 4 * c4, 16);
    }
}

// The scans' operands stay in shared memory with padded rows, and their products read the
// mma fragments from there directly (smem_gemm): no staging copy, no barrier per k step.
// A fragment read touches 8 rows x 4 consecutive k (row stride = 4 mod 32 words: row_k)
// when k runs along the rows, or 4 rows x 8 consecutive m or n (stride = 8 mod 32: row_m)
// otherwise; either way 32 different banks.
__host__ __device__ constexpr int row_k(int n) { return n + 4; }  // rows holding k
__host__ __device__ constexpr int row_m(int n) { return n + 8; }  // rows holding m or n
static_assert(row_k(64) % 32 == 4 && row_k(128) % 32 == 4, "k rows");
static_assert(row_m(64) % 32 == 8 && row_m(128) % 32 == 8, "m rows");

// C(m, n) = alpha * sum_k A(m, k) B(k, n) (+ C(m, n) when acc) with A, B and C in shared
// memory: A(m, k) = A[m * am + k * ak] and so on, M, N multiples of 64, K of 8, C apart
// from A and B. The same mma.sync split and precision as block_gemm (SPLIT: 3xTF32, else
// operands rounded to tf32); fragments are read in place. Called by all kT threads; ends
// with a barrier.
template <bool SPLIT>
__device__ void smem_gemm(int M, int N, int K, float alpha, const float *A, int am, int ak, const float *B, int bk,
                          int bn, float *C, int cm, int cn, bool acc) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int mb = (warp & 3) * 16, nb = (warp >> 2) * 16;
    for (int m0 = 0; m0 < M; m0 += 64) {
        for (int n0 = 0; n0 < N; n0 += 64) {
            float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const float *Ab = A + (m0 + mb + g) * am + t * ak;
            const float *Bb = B + t * bk + (n0 + nb + g) * bn;
#pragma unroll 2
            for (int k8 = 0; k8 < K; k8 += 8) {
                const float *Af = Ab + k8 * ak;
                const float a[4] = {Af[0], Af[8 * am], Af[4 * ak], Af[8 * am + 4 * ak]};
                uint32_t ah[4], al[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (SPLIT) split_tf32(a[i], ah[i], al[i]);
                    else ah[i] = to_tf32(a[i]);
                }
#pragma unroll
                for (int f = 0; f < 2; ++f) {
                    const float *Bf = Bb + k8 * bk + 8 * f * bn;
                    const float b0 = Bf[0], b1 = Bf[4 * bk];
                    if constexpr (SPLIT) {
                        uint32_t bh0, bl0, bh1, bl1;
                        split_tf32(b0, bh0, bl0);
                        split_tf32(b1, bh1, bl1);
                        mma_m16n8k8_tf32(c[f], al, bh0, bh1);
                        mma_m16n8k8_tf32(c[f], ah, bl0, bl1);
                        mma_m16n8k8_tf32(c[f], ah, bh0, bh1);
                    } else {
                        mma_m16n8k8_tf32(c[f], ah, to_tf32(b0), to_tf32(b1));
                    }
                }
            }
#pragma unroll
            for (int hq = 0; hq < 2; ++hq)
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int j = (g + rr) & 3, f = j >> 1, qi = j & 1;
                    const float v0 = qi ? c[0][2 * hq + 1] : c[0][2 * hq];
                    const float v1 = qi ? c[1][2 * hq + 1] : c[1][2 * hq];
                    const float v = f ? v1 : v0;
                    const int m = m0 + mb + g + 8 * hq, n = n0 + nb + 8 * f + 2 * t + qi;
                    float *p = C + m * cm + n * cn;
                    *p = acc ? fmaf(alpha, v, *p) : alpha * v;
                }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;\n" ::); }

// ---- states: the forward scan, S slice [K][64 columns] in shared memory -----------------------
// Per chunk the operands (W, Kb [64][K], U's 64 columns, e^Gn) are copied into shared memory,
// two buffers, the next chunk's copy in flight while the current chunk is computed. Row
// strides: S and U rs (m/n rows), W rw (k rows: W is A with k = d_k along its rows), Kb rkb
// (Kb^T is A with m = d_k along the rows of Kb).
size_t states_smem(int K) {
    const size_t rs = row_m(64), rw = row_k(K), rkb = row_m(K);
    return sizeof(float) * (K * rs + 2 * (64 * rw + 64 * rkb + 64 * rs + K));
}

template <bool SPLIT>
__global__ void __launch_bounds__(kT) bwd_states_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int K = a.d_k, V = a.d_v, tid = threadIdx.x;
    const int rs = row_m(64), rw = row_k(K), rkb = row_m(K);
    float *St = sm;                          // S [K][64]
    float *buf = St + K * rs;                // two buffers of the chunk operands
    const int bstride = 64 * rw + 64 * rkb + 64 * rs + K;
    const int j0 = blockIdx.x * 64, h = blockIdx.y, n = blockIdx.z;
    const Lay L = make_lay(K, V);
    int64_t bos;
    int len;
    if (!bounds(a, n, bos, len)) return;
    const int nch = (len + 63) / 64;
    // buffer b: W [64][K], Kb [64][K], U, then Vt [64][64], e^Gn [K]
    auto issue = [&](int c) {
        const float *S = a.scratch + slot_of(a, bos, n, c, h) * L.total;
        float *Ws = buf + (c & 1) * bstride, *Kbs = Ws + 64 * rw, *Us = Kbs + 64 * rkb, *EGs = Us + 64 * rs;
        stage_rows(Ws, rw, S + L.wm, 64, K, K);
        stage_rows(Kbs, rkb, S + L.kb, 64, K, K);
        stage_rows(Us, rs, S + L.u + j0, 64, 64, V);
        stage_rows(EGs, K, S + L.eg, 1, K, K);
        cp_async_commit();
    };
    if (nch > 0) issue(0);
    for (int e = tid; e < K * 64; e += kT) {
        const int i = e >> 6, j = e & 63;
        St[i * rs + j] = a.h0 ? a.h0[(((int64_t)n * a.H_v + h) * K + i) * V + j0 + j] : 0.f;
    }
    for (int c = 0; c < nch; ++c) {
        float *S = a.scratch + slot_of(a, bos, n, c, h) * L.total;
        float *Ws = buf + (c & 1) * bstride, *Kbs = Ws + 64 * rw, *Us = Kbs + 64 * rkb, *EGs = Us + 64 * rs;
        cp_async_wait_all();
        __syncthreads();
        if (c + 1 < nch) issue(c + 1);  // into the buffer chunk c - 1 used
        for (int e = tid; e < K * 64; e += kT)
            S[L.se + (int64_t)(e >> 6) * V + j0 + (e & 63)] = St[(e >> 6) * rs + (e & 63)];
        // Vt = U - W S (in U's place), stored for the gradient kernel
        smem_gemm<SPLIT>(64, 64, K, -1.f, Ws, rw, 1, St, rs, 1, Us, rs, 1, true);
        for (int e = tid; e < 64 * 64; e += kT)
            S[L.vt + (int64_t)(e >> 6) * V + j0 + (e & 63)] = Us[(e >> 6) * rs + (e & 63)];
        // S <- diag(EG) S + Kb^T Vt
        for (int e = tid; e < K * 64; e += kT) St[(e >> 6) * rs + (e & 63)] *= EGs[e >> 6];
        __syncthreads();
        smem_gemm<SPLIT>(K, 64, 64, 1.f, Kbs, 1, rkb, Us, rs, 1, St, rs, 1, true);
    }
}

// ---- states on tcgen05 (bf16 inputs, d_k = d_v = 128) ---------------------------------------
// One CTA per (sequence, value head, 64 columns of d_v) carries R = S^T [64 v][d_k] through
// the chunks in TMEM (fp32, an M = 64 accumulator: row r in lane 32 (r / 16) + r % 16, 128
// columns). Per chunk c:
//   D1 = R W^T          tf32 MMA, A = R read from TMEM, B = W [t][d] (K-major), which TMA
//                       loads with the 128-byte swizzle
//   element warps:      Vt^T = U^T - D1 into TMEM (the next product's A operand) and to the
//                       scratch; the entry state S_c to the scratch; R <- R diag(e^Gn)
//   R += Vt^T Kb        A = Vt^T from TMEM, B = Kb^T [d][t] (K-major), which the staging
//                       warps transpose from the scratch into shared memory
// Roles: warps 0-3 and 8-11 the element passes (lane quarter warp % 4, its 16 rows in lanes
// 0-15; column half warp / 8), warp 4 lane 0 the loads and MMAs, warps 5-7 and 12-15 the
// transposition of Kb. The loads, Kb^T, U and e^Gn alternate between two buffers by chunk
// parity. Every wait is bounded; a timeout raises the device error word and ends the CTA's
// roles, which then wait for their MMAs and copies in flight before TMEM is freed.
struct StTc {
    static constexpr int oW = 0;         // W [64 t][128 d]: 4 K-major atoms (32 d) of 64 x 128 B
    static constexpr int oKbT = 32768;   // Kb^T [128 d][64 t]: 2 K-major atoms (32 t) of 128 x 128 B
    static constexpr int oU = 65536;     // U [64 t][64 v] fp32, row-major (this CTA's columns)
    static constexpr int oEG = 98304;    // e^Gn [128]
    static constexpr int kBuf = 99328;   // one buffer (1024-byte multiple)
    static constexpr int oBar = 2 * kBuf;
    static constexpr int kBytes = oBar + 128 + 1024;  // + barriers, + alignment slack
};
constexpr uint32_t kStR = 0, kStD = 128, kStV = 192, kStCols = 256;  // TMEM columns
enum { SB_LD0 = 0, SB_LD1, SB_KB0, SB_KB1, SB_D1, SB_UP0, SB_UP1, SB_EL, SB_Z, kStBars };

// (the slow path out of line: the waits of a kernel share one copy of it)
__device__ __noinline__ bool st_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag, unsigned int *err) {
    const long long t0 = clock64();
    while (!tc5::mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kDefaultWaitCycles) {
            *abort_flag = 1;
            atomicOr(err, kDeviceErrTimeout);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool st_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, unsigned int *err) {
    return tc5::mbar_try_wait(bar, parity) || st_wait_slow(bar, parity, abort_flag, err);
}
// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// st_wait by every lane of a warp, with one outcome for all of them (the warp-collective TMEM
// accesses and __syncwarp that follow need the whole warp on the same branch).
__device__ __forceinline__ bool st_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag, unsigned int *err) {
    return __all_sync(0xffffffffu, st_wait(bar, parity, abort_flag, err));
}

__global__ void __launch_bounds__(kT, 1) bwd_states_tc_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap umap) {
    using namespace tc5;
    using tcu::mbar_arrive;
    using tcu::tmem_ld32;
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + StTc::oBar);
    __shared__ uint32_t tslot;
    __shared__ int abort_w;
    volatile int *abort_flag = &abort_w;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = 64 * blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    constexpr int K = 128, V = 128;
    const Lay L = make_lay(K, V);
    int64_t bos;
    int len;
    if (!bounds(a, n, bos, len)) return;
    const int nch = (len + 63) / 64;
    if (tid == 0) {
        for (int i = 0; i < kStBars; ++i) mbar_init(&bars[i], i == SB_EL ? 8 : 1);
        abort_w = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, kStCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tslot;
    const bool elem = warp < 4 || (warp >= 8 && warp < 12);
    const int q = warp & 3, hh = warp >> 3;  // element warps: lane quarter, column half
    const bool row_lane = lane < 16;         // lanes 0-15 of a quarter hold rows 16 q + lane
    const int v = j0 + 16 * q + (lane & 15);  // this lane's d_v column
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    // R = h0^T (or zero)
    if (elem) {
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            uint32_t r0[16], r1[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int d0 = 64 * hh + 32 * p + j, d1 = d0 + 16;
                const float *h0 = a.h0 ? a.h0 + (((int64_t)n * a.H_v + h) * K) * V + v : nullptr;
                r0[j] = __float_as_uint(h0 ? h0[(int64_t)d0 * V] : 0.f);
                r1[j] = __float_as_uint(h0 ? h0[(int64_t)d1 * V] : 0.f);
            }
            tmem_st16(tmem + lane_off + kStR + 64 * hh + 32 * p, r0);
            tmem_st16(tmem + lane_off + kStR + 64 * hh + 32 * p + 16, r1);
        }
        tmem_st_wait();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (warp == 4) {
        // ---- loads and MMAs (lane 0) ----
        if (lane == 0) {
            auto load = [&](int c) {
                const int b = c & 1;
                unsigned char *B = sm + b * StTc::kBuf;
                const int64_t slot = slot_of(a, bos, n, c, h);
                const float *S = a.scratch + slot * L.total;
                mbar_arrive_expect_tx(&bars[SB_LD0 + b], 32768 + 16384 + 512);
#pragma unroll
                for (int at = 0; at < 4; ++at) tma_load_3d(B + StTc::oW + at * 8192, &wmap, &bars[SB_LD0 + b], 32 * at, 0, (int)slot);
                tma_load_3d(B + StTc::oU, &umap, &bars[SB_LD0 + b], j0, 0, (int)slot);
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 smem_u32(B + StTc::oEG)), "l"(S + L.eg), "r"(512), "r"(smem_u32(&bars[SB_LD0 + b]))
                             : "memory");
            };
            const uint32_t id1 = idesc_tf32(64, 64), id2 = idesc_tf32(64, 128);
            bool ok = true;
            int issued[2] = {-1, -1}, waited[2] = {-1, -1};  // latest chunk loaded / waited per buffer
            if (nch > 0) {
                load(0);
                issued[0] = 0;
            }
            for (int c = 0; c < nch && ok; ++c) {
                const int b = c & 1;
                const uint32_t sB = smem_u32(sm + b * StTc::kBuf);
                // R = S_c^T (the previous update is complete); buffer (c + 1) & 1 is free
                if (c > 0) ok = st_wait(&bars[SB_UP0 + ((c - 1) & 1)], (uint32_t)(((c - 1) >> 1) & 1), abort_flag, a.err);
                if (ok && c + 1 < nch) {
                    load(c + 1);
                    issued[(c + 1) & 1] = c + 1;
                }
                if (ok) ok = st_wait(&bars[SB_LD0 + b], (uint32_t)((c >> 1) & 1), abort_flag, a.err);
                if (ok) waited[b] = c;
                if (!ok) break;
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    mma_tf32_ts(tmem + kStD, tmem + kStR + 8 * s,
                                desc_sw128(sB + StTc::oW + (s >> 2) * 8192 + (s & 3) * 32, 0, 1024), id1, s > 0);
                commit(&bars[SB_D1]);
                ok = st_wait(&bars[SB_EL], (uint32_t)(c & 1), abort_flag, a.err);
                if (ok) ok = st_wait(&bars[SB_KB0 + b], (uint32_t)((c >> 1) & 1), abort_flag, a.err);
                if (!ok) break;
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_tf32_ts(tmem + kStR, tmem + kStV + 8 * s,
                                desc_sw128(sB + StTc::oKbT + (s >> 2) * 16384 + (s & 3) * 32, 0, 1024), id2, 1);
                commit(&bars[SB_UP0 + b]);
            }
            // every MMA and load of this CTA lands before TMEM is freed
            commit(&bars[SB_Z]);
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[SB_Z], 0) && clock64() - t0 < kDefaultWaitCycles) {}
            for (int bb = 0; bb < 2; ++bb) {
                if (issued[bb] > waited[bb]) {
                    const long long t1 = clock64();
                    while (!mbar_try_wait(&bars[SB_LD0 + bb], (uint32_t)((issued[bb] >> 1) & 1)) &&
                           clock64() - t1 < kDefaultWaitCycles) {}
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (elem) {
        // ---- element passes ----
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const unsigned char *B = sm + b * StTc::kBuf;
            float *S = a.scratch + slot_of(a, bos, n, c, h) * L.total;
            if (!st_wait_warp(&bars[SB_D1], (uint32_t)(c & 1), abort_flag, a.err)) break;
            if (!st_wait_warp(&bars[SB_LD0 + b], (uint32_t)((c >> 1) & 1), abort_flag, a.err)) break;
            fence_after_sync();
            {
                // Vt^T = U^T - D1 for tokens 32 hh .. 32 hh + 31
                float d1[32];
                tmem_ld32(tmem + lane_off + kStD + 32 * hh, d1);
                const float *U = reinterpret_cast<const float *>(B + StTc::oU);
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = 32 * hh + j;
                    const float vt = U[t * 64 + (v - j0)] - d1[j];
                    if (row_lane) S[L.vt + (int64_t)t * V + v] = vt;
                    if (j < 16) w0[j] = __float_as_uint(vt); else w1[j - 16] = __float_as_uint(vt);
                }
                tmem_st16(tmem + lane_off + kStV + 32 * hh, w0);
                tmem_st16(tmem + lane_off + kStV + 32 * hh + 16, w1);
            }
            {
                // the entry state S_c to the scratch, then R <- R diag(e^Gn), channels 64 hh .. + 63
                const float *EG = reinterpret_cast<const float *>(B + StTc::oEG);
#pragma unroll 1
                for (int p = 0; p < 2; ++p) {
                    const int d0 = 64 * hh + 32 * p;
                    float r[32];
                    tmem_ld32(tmem + lane_off + kStR + d0, r);
                    uint32_t y0[16], y1[16];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (row_lane) S[L.se + (int64_t)(d0 + j) * V + v] = r[j];
                        const float y = r[j] * EG[d0 + j];
                        if (j < 16) y0[j] = __float_as_uint(y); else y1[j - 16] = __float_as_uint(y);
                    }
                    tmem_st16(tmem + lane_off + kStR + d0, y0);
                    tmem_st16(tmem + lane_off + kStR + d0 + 16, y1);
                }
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[SB_EL]);
        }
    } else {
        // ---- Kb^T staging: warps 5-7 and 12-15 (224 threads) ----
        const int tt = (warp < 8 ? warp - 5 : warp - 9) * 32 + lane;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            unsigned char *KbT = sm + b * StTc::kBuf + StTc::oKbT;
            const float4 *Kb = reinterpret_cast<const float4 *>(a.scratch + slot_of(a, bos, n, c, h) * L.total + L.kb);
            if (tt == 0 && c + 1 < nch) prefetch_l2(a.scratch + slot_of(a, bos, n, c + 1, h) * L.total + L.kb, 64 * K * 4);
            float4 r[10];
#pragma unroll
            for (int i = 0; i < 10; ++i) {
                const int e = tt + 224 * i;  // t = e % 64, 4 d = 4 (e / 64)
                if (e < 2048) r[i] = __ldg(Kb + (e & 63) * 32 + (e >> 6));
            }
            // the buffer's previous Kb^T (chunk c - 2) has been read by its update
            // (all 224 threads take the same branch, so that none is left at the named barrier)
            if (c >= 2 && tcu::bar_or(3, 224, !st_wait(&bars[SB_UP0 + b], (uint32_t)(((c >> 1) - 1) & 1), abort_flag, a.err)))
                break;
#pragma unroll
            for (int i = 0; i < 10; ++i) {
                const int e = tt + 224 * i;
                if (e < 2048) {
                    const int t = e & 63, d = 4 * (e >> 6);
                    unsigned char *atom = KbT + (t >> 5) * 16384;
                    const int k = t & 31;
                    const float x[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = d + j;
                        *reinterpret_cast<uint32_t *>(atom + row * 128 + (((k >> 2) ^ (row & 7)) << 4) + (k & 3) * 4) =
                            tcu::tf32(x[j]);
                    }
                }
            }
            fence_proxy_async();
            asm volatile("bar.sync 3, 224;" ::: "memory");
            if (tt == 0) mbar_arrive(&bars[SB_KB0 + b]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, kStCols);
    }
}

// ---- adjoint: the reverse scan, dS slice [K][64 columns] in shared memory -------------------
// The chunk's operands are copied into shared memory in two sets: A, Kb, e^Gn and dO for the
// first products, Qp and W for the second. Each set's buffer is refilled with the next chunk's
// set as soon as the current chunk is done with it (dO, used by both, has two buffers). Row
// strides: dS, A, dO, dVt rs; Kb rkb (k rows); Qp, W rq (Qp^T and W^T are A with m = d_k
// along their rows).
size_t adjoint_smem(int K) {
    const size_t rs = row_m(64), rkb = row_k(K), rq = row_m(K);
    return sizeof(float) * (K * rs + 64 * rkb + 2 * 64 * rq + 4 * 64 * rs + 2 * K);
}

template <bool SPLIT>
__global__ void __launch_bounds__(kT) bwd_adjoint_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int K = a.d_k, V = a.d_v, tid = threadIdx.x;
    const int rs = row_m(64), rkb = row_k(K), rq = row_m(K);
    float *dS = sm;                  // dS [K][64]
    float *Kbs = dS + K * rs;        // Kb [64][K]
    float *Qps = Kbs + 64 * rkb;     // Qp [64][K]
    float *Ws = Qps + 64 * rq;       // W [64][K]
    float *As = Ws + 64 * rq;        // A [64][64]
    float *dOb = As + 64 * rs;       // dO's 64 columns [64][64], two buffers
    float *dVs = dOb + 2 * 64 * rs;  // dVt [64][64]
    float *EGb = dVs + 64 * rs;      // e^Gn [K], two buffers
    const int j0 = blockIdx.x * 64, h = blockIdx.y, n = blockIdx.z;
    const Lay L = make_lay(K, V);
    int64_t bos;
    int len;
    if (!bounds(a, n, bos, len)) return;
    const int nch = (len + 63) / 64;
    auto slot = [&](int c) { return a.scratch + slot_of(a, bos, n, c, h) * L.total; };
    auto issue_first = [&](int c) {
        const float *S = slot(c);
        stage_rows(Kbs, rkb, S + L.kb, 64, K, K);
        stage_rows(As, rs, S + L.a, 64, 64, 64);
        stage_rows(dOb + (c & 1) * 64 * rs, rs, S + L.dof + j0, 64, 64, V);
        stage_rows(EGb + (c & 1) * K, K, S + L.eg, 1, K, K);
        cp_async_commit();
    };
    auto issue_second = [&](int c) {
        const float *S = slot(c);
        stage_rows(Qps, rq, S + L.qp, 64, K, K);
        stage_rows(Ws, rq, S + L.wm, 64, K, K);
        cp_async_commit();
    };
    if (nch > 0) {
        issue_first(nch - 1);
        issue_second(nch - 1);
    }
    for (int e = tid; e < K * 64; e += kT) {
        const int i = e >> 6, j = e & 63;
        dS[i * rs + j] = a.dht ? a.dht[(((int64_t)n * a.H_v + h) * K + i) * V + j0 + j] : 0.f;
    }
    for (int c = nch - 1; c >= 0; --c) {
        float *S = slot(c);
        float *dOs = dOb + (c & 1) * 64 * rs, *EGs = EGb + (c & 1) * K;
        // the groups in flight are this chunk's two sets, oldest first
        cp_async_wait_one();
        __syncthreads();
        for (int e = tid; e < K * 64; e += kT)
            S[L.dsx + (int64_t)(e >> 6) * V + j0 + (e & 63)] = dS[(e >> 6) * rs + (e & 63)];
        // dVt = A^T dO + Kb dS', stored for the gradient kernel
        smem_gemm<SPLIT>(64, 64, 64, 1.f, As, 1, rs, dOs, rs, 1, dVs, rs, 1, false);
        smem_gemm<SPLIT>(64, 64, K, 1.f, Kbs, rkb, 1, dS, rs, 1, dVs, rs, 1, true);
        // A and Kb are consumed: the previous chunk's first set (its dO into the other buffer)
        if (c > 0) {
            issue_first(c - 1);
            cp_async_wait_one();  // this chunk's second set
        } else {
            cp_async_wait_all();
        }
        for (int e = tid; e < 64 * 64; e += kT)
            S[L.dvt + (int64_t)(e >> 6) * V + j0 + (e & 63)] = dVs[(e >> 6) * rs + (e & 63)];
        // dS <- diag(EG) dS' + Qp^T dO - W^T dVt
        for (int e = tid; e < K * 64; e += kT) dS[(e >> 6) * rs + (e & 63)] *= EGs[e >> 6];
        __syncthreads();
        smem_gemm<SPLIT>(K, 64, 64, 1.f, Qps, 1, rq, dOs, rs, 1, dS, rs, 1, true);
        smem_gemm<SPLIT>(K, 64, 64, -1.f, Ws, 1, rq, dVs, rs, 1, dS, rs, 1, true);
        if (c > 0) issue_second(c - 1);  // Qp and W are consumed
    }
    if (a.dh0 != nullptr)
        for (int e = tid; e < K * 64; e += kT)
            a.dh0[(((int64_t)n * a.H_v + h) * K + (e >> 6)) * V + j0 + (e & 63)] = dS[(e >> 6) * rs + (e & 63)];
}

// ---- adjoint on tcgen05 (bf16 inputs, d_k = d_v = 128) --------------------------------------
// One CTA per (sequence, value head, 64 columns of d_v) carries Q = dS^T [64 v][d_k] backwards
// through the chunks in TMEM (an M = 64 fp32 accumulator, 128 columns). Per chunk c, last
// first:
//   element warps:  dS' (= Q on entry) to the scratch; dO^T [v][t] into TMEM (an A operand)
//   D2 = dO^T A^T^T + Q Kb^T = dVt^T [v][t]   (A^T as a K-major [s][t] tile, Kb by TMA)
//   element warps:  dVt to the scratch, -dVt^T into TMEM, Q <- Q diag(e^Gn)
//   Q += dO^T Qp - dVt^T W                     (Qp^T and W^T as K-major [d][t] tiles)
// The transposed tiles are made by the staging warps from the scratch, as in the states scan.
// Roles: warps 0-3 and 8-11 the element passes, warp 4 lane 0 the loads and MMAs, warps 5-7 and
// 12-15 the transposition. Kb, dO, e^Gn and A^T alternate between two buffers; Qp^T and W^T
// have one. Every wait is bounded, as in the states scan.
struct AdTc {
    static constexpr int oKb = 0;        // Kb [64 t][128 d]: 4 K-major atoms (32 d) of 64 x 128 B
    static constexpr int oAT = 32768;    // A^T [64 s][64 t]: 2 K-major atoms (32 t) of 64 x 128 B
    static constexpr int oDO = 49152;    // dO [64 t][64 v] fp32 row-major (this CTA's columns)
    static constexpr int oEG = 65536;    // e^Gn [128]
    static constexpr int kBuf = 66560;
    static constexpr int oQpT = 2 * kBuf;          // Qp^T [128 d][64 t]: 2 atoms (32 t) of 128 x 128 B
    static constexpr int oWT = oQpT + 32768;       // W^T likewise
    static constexpr int oBar = oWT + 32768;
    static constexpr int kBytes = oBar + 128 + 1024;
};
constexpr uint32_t kAdQ = 0, kAdD = 128, kAdO = 192, kAdN = 256, kAdCols = 512;  // TMEM columns
enum { AB_LD0 = 0, AB_LD1, AB_AT0, AB_AT1, AB_QW, AB_PRE, AB_D0, AB_D1, AB_EL, AB_UP, AB_Z, kAdBars };

// Transposed K-major tile: element (row, k) of a tile of 32-column atoms `atom_bytes` apart.
__device__ __forceinline__ void st_kmajor(unsigned char *tile, int atom_bytes, int row, int k, float x) {
    unsigned char *atom = tile + (k >> 5) * atom_bytes;
    const int kk = k & 31;
    *reinterpret_cast<uint32_t *>(atom + row * 128 + (((kk >> 2) ^ (row & 7)) << 4) + (kk & 3) * 4) = tcu::tf32(x);
}

__global__ void __launch_bounds__(kT, 1) bwd_adjoint_tc_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap kbmap,
                                                                const __grid_constant__ CUtensorMap domap) {
    using namespace tc5;
    using tcu::mbar_arrive;
    using tcu::tmem_ld32;
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + AdTc::oBar);
    __shared__ uint32_t tslot;
    __shared__ int abort_w;
    volatile int *abort_flag = &abort_w;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = 64 * blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    constexpr int K = 128, V = 128;
    const Lay L = make_lay(K, V);
    int64_t bos;
    int len;
    if (!bounds(a, n, bos, len)) return;
    const int nch = (len + 63) / 64;
    if (tid == 0) {
        for (int i = 0; i < kAdBars; ++i) mbar_init(&bars[i], (i == AB_PRE || i == AB_EL) ? 8 : 1);
        abort_w = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, kAdCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tslot;
    const bool elem = warp < 4 || (warp >= 8 && warp < 12);
    const int q = warp & 3, hh = warp >> 3;
    const bool row_lane = lane < 16;
    const int v = j0 + 16 * q + (lane & 15);
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    auto slot = [&](int c) { return a.scratch + slot_of(a, bos, n, c, h) * L.total; };
    // Q = dht^T (or zero)
    if (elem) {
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            uint32_t r0[16], r1[16];
            const float *dht = a.dht ? a.dht + (((int64_t)n * a.H_v + h) * K) * V + v : nullptr;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int d0 = 64 * hh + 32 * p + j;
                r0[j] = __float_as_uint(dht ? dht[(int64_t)d0 * V] : 0.f);
                r1[j] = __float_as_uint(dht ? dht[(int64_t)(d0 + 16) * V] : 0.f);
            }
            tmem_st16(tmem + lane_off + kAdQ + 64 * hh + 32 * p, r0);
            tmem_st16(tmem + lane_off + kAdQ + 64 * hh + 32 * p + 16, r1);
        }
        tmem_st_wait();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (warp == 4) {
        if (lane == 0) {
            // iteration i works on chunk nch - 1 - i, in buffer i & 1
            auto load = [&](int i) {
                const int b = i & 1, c = nch - 1 - i;
                unsigned char *B = sm + b * AdTc::kBuf;
                const int64_t sl = slot_of(a, bos, n, c, h);
                mbar_arrive_expect_tx(&bars[AB_LD0 + b], 32768 + 16384 + 512);
#pragma unroll
                for (int at = 0; at < 4; ++at) tma_load_3d(B + AdTc::oKb + at * 8192, &kbmap, &bars[AB_LD0 + b], 32 * at, 0, (int)sl);
                tma_load_3d(B + AdTc::oDO, &domap, &bars[AB_LD0 + b], j0, 0, (int)sl);
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 smem_u32(B + AdTc::oEG)), "l"(a.scratch + sl * L.total + L.eg), "r"(512),
                             "r"(smem_u32(&bars[AB_LD0 + b]))
                             : "memory");
            };
            const uint32_t id64 = idesc_tf32(64, 64), id128 = idesc_tf32(64, 128);
            const uint32_t sQW = smem_u32(sm + AdTc::oQpT), sWT = smem_u32(sm + AdTc::oWT);
            bool ok = true;
            int issued[2] = {-1, -1}, waited[2] = {-1, -1};
            if (nch > 0) {
                load(0);
                issued[0] = 0;
            }
            for (int i = 0; i < nch && ok; ++i) {
                const int b = i & 1;
                const uint32_t sB = smem_u32(sm + b * AdTc::kBuf);
                if (i > 0) ok = st_wait(&bars[AB_UP], (uint32_t)((i - 1) & 1), abort_flag, a.err);
                if (ok && i + 1 < nch) {
                    load(i + 1);
                    issued[(i + 1) & 1] = i + 1;
                }
                if (ok) ok = st_wait(&bars[AB_LD0 + b], (uint32_t)((i >> 1) & 1), abort_flag, a.err);
                if (ok) waited[b] = i;
                if (ok) ok = st_wait(&bars[AB_PRE], (uint32_t)(i & 1), abort_flag, a.err);
                if (ok) ok = st_wait(&bars[AB_AT0 + b], (uint32_t)((i >> 1) & 1), abort_flag, a.err);
                if (!ok) break;
                fence_after_sync();
                // dVt^T = dO^T (A^T)^T + Q Kb^T
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_tf32_ts(tmem + kAdD, tmem + kAdO + 8 * s,
                                desc_sw128(sB + AdTc::oAT + (s >> 2) * 8192 + (s & 3) * 32, 0, 1024), id64, s > 0);
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    mma_tf32_ts(tmem + kAdD, tmem + kAdQ + 8 * s,
                                desc_sw128(sB + AdTc::oKb + (s >> 2) * 8192 + (s & 3) * 32, 0, 1024), id64, 1);
                commit(&bars[AB_D0 + b]);
                ok = st_wait(&bars[AB_EL], (uint32_t)(i & 1), abort_flag, a.err);
                if (ok) ok = st_wait(&bars[AB_QW], (uint32_t)(i & 1), abort_flag, a.err);
                if (!ok) break;
                fence_after_sync();
                // Q += dO^T Qp - dVt^T W
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_tf32_ts(tmem + kAdQ, tmem + kAdO + 8 * s, desc_sw128(sQW + (s >> 2) * 16384 + (s & 3) * 32, 0, 1024),
                                id128, 1);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_tf32_ts(tmem + kAdQ, tmem + kAdN + 8 * s, desc_sw128(sWT + (s >> 2) * 16384 + (s & 3) * 32, 0, 1024),
                                id128, 1);
                commit(&bars[AB_UP]);
            }
            commit(&bars[AB_Z]);
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[AB_Z], 0) && clock64() - t0 < kDefaultWaitCycles) {}
            for (int bb = 0; bb < 2; ++bb) {
                if (issued[bb] > waited[bb]) {
                    const long long t1 = clock64();
                    while (!mbar_try_wait(&bars[AB_LD0 + bb], (uint32_t)((issued[bb] >> 1) & 1)) &&
                           clock64() - t1 < kDefaultWaitCycles) {}
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (elem) {
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int b = i & 1, c = nch - 1 - i;
            const unsigned char *B = sm + b * AdTc::kBuf;
            float *S = slot(c);
            if (i > 0 && !(ok = st_wait_warp(&bars[AB_UP], (uint32_t)((i - 1) & 1), abort_flag, a.err))) break;
            if (!(ok = st_wait_warp(&bars[AB_LD0 + b], (uint32_t)((i >> 1) & 1), abort_flag, a.err))) break;
            fence_after_sync();
            {
                // dO^T [v][t] for tokens 32 hh .. + 31 into TMEM
                const float *dO = reinterpret_cast<const float *>(B + AdTc::oDO);
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    w0[j] = __float_as_uint(dO[(32 * hh + j) * 64 + (v - j0)]);
                    w1[j] = __float_as_uint(dO[(32 * hh + 16 + j) * 64 + (v - j0)]);
                }
                tmem_st16(tmem + lane_off + kAdO + 32 * hh, w0);
                tmem_st16(tmem + lane_off + kAdO + 32 * hh + 16, w1);
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[AB_PRE]);
            }
            // dS' of this chunk (Q on entry) to the scratch, channels 64 hh .. + 63
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                const int d0 = 64 * hh + 32 * p;
                float r[32];
                tmem_ld32(tmem + lane_off + kAdQ + d0, r);
                if (row_lane) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) S[L.dsx + (int64_t)(d0 + j) * V + v] = r[j];
                }
            }
            if (!(ok = st_wait_warp(&bars[AB_D0 + b], (uint32_t)((i >> 1) & 1), abort_flag, a.err))) break;
            fence_after_sync();
            {
                // dVt to the scratch, -dVt^T into TMEM (tokens 32 hh .. + 31)
                float d2[32];
                tmem_ld32(tmem + lane_off + kAdD + 32 * hh, d2);
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (row_lane) S[L.dvt + (int64_t)(32 * hh + j) * V + v] = d2[j];
                    if (j < 16) w0[j] = __float_as_uint(-d2[j]); else w1[j - 16] = __float_as_uint(-d2[j]);
                }
                if (a.tc && row_lane) {
                    // dVt^T row v, tokens 32 hh .. + 31, for the gradient kernel
                    float4 *dst = reinterpret_cast<float4 *>(S + L.dvtt + (int64_t)v * 64 + 32 * hh);
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j] = make_float4(d2[4 * j], d2[4 * j + 1], d2[4 * j + 2], d2[4 * j + 3]);
                }
                tmem_st16(tmem + lane_off + kAdN + 32 * hh, w0);
                tmem_st16(tmem + lane_off + kAdN + 32 * hh + 16, w1);
            }
            {
                // Q <- Q diag(e^Gn)
                const float *EG = reinterpret_cast<const float *>(B + AdTc::oEG);
#pragma unroll 1
                for (int p = 0; p < 2; ++p) {
                    const int d0 = 64 * hh + 32 * p;
                    float r[32];
                    tmem_ld32(tmem + lane_off + kAdQ + d0, r);
                    uint32_t y0[16], y1[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        y0[j] = __float_as_uint(r[j] * EG[d0 + j]);
                        y1[j] = __float_as_uint(r[16 + j] * EG[d0 + 16 + j]);
                    }
                    tmem_st16(tmem + lane_off + kAdQ + d0, y0);
                    tmem_st16(tmem + lane_off + kAdQ + d0 + 16, y1);
                }
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[AB_EL]);
        }
        // dh0 = Q after the first chunk (dht when there is none)
        if (ok && nch > 0) ok = st_wait_warp(&bars[AB_UP], (uint32_t)((nch - 1) & 1), abort_flag, a.err);
        if (ok && a.dh0 != nullptr) {
            fence_after_sync();
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                const int d0 = 64 * hh + 32 * p;
                float r[32];
                tmem_ld32(tmem + lane_off + kAdQ + d0, r);
                if (row_lane) {
                    float *dh0 = a.dh0 + (((int64_t)n * a.H_v + h) * K) * V + v;
#pragma unroll
                    for (int j = 0; j < 32; ++j) dh0[(int64_t)(d0 + j) * V] = r[j];
                }
            }
        }
    } else {
        // ---- transposition: warps 5-7 and 12-15 (224 threads) ----
        const int tt = (warp < 8 ? warp - 5 : warp - 9) * 32 + lane;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1, c = nch - 1 - i;
            const float *S = slot(c);
            if (tt == 0 && c > 0) {
                // the next chunk's A, Qp and W into L2 while this one is staged
                const float *Sn = slot(c - 1);
                prefetch_l2(Sn + L.a, 64 * 64 * 4);
                prefetch_l2(Sn + L.qp, 64 * K * 4);
                prefetch_l2(Sn + L.wm, 64 * K * 4);
            }
            // A^T: element (s, t) = A[t][s]; A [64 t][64 s] as 1024 float4, t = e % 64, 4 s = 4 (e / 64)
            {
                float4 r[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    const int e = tt + 224 * k;
                    if (e < 1024) r[k] = __ldg(reinterpret_cast<const float4 *>(S + L.a) + (e & 63) * 16 + (e >> 6));
                }
                // the buffer's A^T (iteration i - 2) has been read by its D2
                // (all 224 threads take the same branch, so that none is left at the named barrier)
                if (i >= 2 && tcu::bar_or(3, 224, !st_wait(&bars[AB_D0 + b], (uint32_t)(((i >> 1) - 1) & 1), abort_flag, a.err)))
                    break;
                unsigned char *AT = sm + b * AdTc::kBuf + AdTc::oAT;
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    const int e = tt + 224 * k;
                    if (e < 1024) {
                        const int t = e & 63, s0 = 4 * (e >> 6);
                        st_kmajor(AT, 8192, s0, t, r[k].x);
                        st_kmajor(AT, 8192, s0 + 1, t, r[k].y);
                        st_kmajor(AT, 8192, s0 + 2, t, r[k].z);
                        st_kmajor(AT, 8192, s0 + 3, t, r[k].w);
                    }
                }
                fence_proxy_async();
                asm volatile("bar.sync 3, 224;" ::: "memory");
                if (tt == 0) mbar_arrive(&bars[AB_AT0 + b]);
            }
            // Qp^T and W^T: element (d, t) of [64 t][128 d] as 2048 float4, t = e % 64, 4 d = 4 (e / 64)
            float4 r[10];
#pragma unroll
            for (int k = 0; k < 10; ++k) {
                const int e = tt + 224 * k;
                if (e < 2048) r[k] = __ldg(reinterpret_cast<const float4 *>(S + L.qp) + (e & 63) * 32 + (e >> 6));
            }
            // the single Qp^T / W^T buffer has been read by the previous update
            if (i >= 1 && tcu::bar_or(3, 224, !st_wait(&bars[AB_UP], (uint32_t)((i - 1) & 1), abort_flag, a.err))) break;
#pragma unroll
            for (int k = 0; k < 10; ++k) {
                const int e = tt + 224 * k;
                if (e < 2048) {
                    const int t = e & 63, d0 = 4 * (e >> 6);
                    st_kmajor(sm + AdTc::oQpT, 16384, d0, t, r[k].x);
                    st_kmajor(sm + AdTc::oQpT, 16384, d0 + 1, t, r[k].y);
                    st_kmajor(sm + AdTc::oQpT, 16384, d0 + 2, t, r[k].z);
                    st_kmajor(sm + AdTc::oQpT, 16384, d0 + 3, t, r[k].w);
                }
            }
#pragma unroll
            for (int k = 0; k < 10; ++k) {
                const int e = tt + 224 * k;
                if (e < 2048) r[k] = __ldg(reinterpret_cast<const float4 *>(S + L.wm) + (e & 63) * 32 + (e >> 6));
            }
#pragma unroll
            for (int k = 0; k < 10; ++k) {
                const int e = tt + 224 * k;
                if (e < 2048) {
                    const int t = e & 63, d0 = 4 * (e >> 6);
                    st_kmajor(sm + AdTc::oWT, 16384, d0, t, r[k].x);
                    st_kmajor(sm + AdTc::oWT, 16384, d0 + 1, t, r[k].y);
                    st_kmajor(sm + AdTc::oWT, 16384, d0 + 2, t, r[k].z);
                    st_kmajor(sm + AdTc::oWT, 16384, d0 + 3, t, r[k].w);
                }
            }
            fence_proxy_async();
            asm volatile("bar.sync 3, 224;" ::: "memory");
            if (tt == 0) mbar_arrive(&bars[AB_QW]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, kAdCols);
    }
}

// ---- grads: every gradient of one chunk ---------------------------------------------------------
// Shared memory: dQp, dKp, dKm, dKb, dW (then T^T dVt) [64][K or V], dA, dT (then dL), X
// [64][64], small vectors and the GEMM stage.
template <typename T, bool GATE_HEAD>
__global__ void __launch_bounds__(kT) bwd_grads_kernel(const BwdArgs a) {
    constexpr bool SPLIT = std::is_same<T, float>::value;
    extern __shared__ __align__(16) float sm[];
    int n, c, len;
    int64_t bos;
    if (!window_owner(a, blockIdx.y, n, c, bos, len)) return;
    const int h = blockIdx.x, hk = h / a.group, K = a.d_k, V = a.d_v, tid = threadIdx.x;
    const int KV = K > V ? K : V;
    float *dQp = sm, *dKp = dQp + 64 * K, *dKm = dKp + 64 * K, *dKb = dKm + 64 * K;
    float *dW = dKb + 64 * K;  // [64][KV]
    float *dA = dW + 64 * KV, *dT = dA + 4096, *X = dA;  // X reuses dA once dA is consumed
    float *dEG = dT + 4096, *dGn = dEG + 128, *dbeta = dGn + 128;
    float *stage = dbeta + 64;
    const Lay L = make_lay(K, V);
    const float *S = a.scratch + slot_of(a, bos, n, c, h) * L.total;
    const float *Qp = S + L.qp, *Kp = S + L.kp, *Km = S + L.km, *Kb = S + L.kb;
    const float *Gm = S + L.gm, *Vf = S + L.vf, *dOf = S + L.dof, *Vt = S + L.vt, *dVt = S + L.dvt;
    const float *Mm = S + L.m, *Tm = S + L.t, *EG = S + L.eg, *Bt = S + L.bt;
    const float *Se = S + L.se, *dSx = S + L.dsx;
    const int row0 = c * 64, nv = min(64, len - row0);

    // dQp = dO S^T;  dA = lower(dO Vt^T);  dQp += dA Km
    block_gemm<SPLIT>(64, K, V, 1.f, dOf, V, 1, Se, 1, V, dQp, K, 1, false, stage);
    block_gemm<SPLIT>(64, 64, V, 1.f, dOf, V, 1, Vt, 1, V, dA, 64, 1, false, stage);
    for (int e = tid; e < 4096; e += kT)
        if ((e & 63) > (e >> 6)) dA[e] = 0.f;
    __syncthreads();
    block_gemm<SPLIT>(64, K, 64, 1.f, dA, 64, 1, Km, K, 1, dQp, K, 1, true, stage);
    // dKm = dA^T Qp (dA is not needed after this)
    block_gemm<SPLIT>(64, K, 64, 1.f, dA, 1, 64, Qp, K, 1, dKm, K, 1, false, stage);
    // dKb = Vt dS'^T;  dW = -dVt S^T;  dEG = rows of dS' . S
    block_gemm<SPLIT>(64, K, V, 1.f, Vt, V, 1, dSx, 1, V, dKb, K, 1, false, stage);
    block_gemm<SPLIT>(64, K, V, -1.f, dVt, V, 1, Se, 1, V, dW, K, 1, false, stage);
    const int warp = tid >> 5, lane = tid & 31;
    for (int i = warp; i < K; i += kT / 32) {  // a warp per row, lanes along it
        float s = 0.f;
        for (int j = lane; j < V; j += 32) s = fmaf(dSx[(int64_t)i * V + j], Se[(int64_t)i * V + j], s);
        s = warp_sum(s);
        if (lane == 0) dEG[i] = s;
    }
    for (int t = tid; t < 64; t += kT) dbeta[t] = 0.f;
    __syncthreads();
    if (!a.decay_only) {
        // dT = (dW Kp^T + dVt V^T) diag(beta)
        block_gemm<SPLIT>(64, 64, K, 1.f, dW, K, 1, Kp, 1, K, dT, 64, 1, false, stage);
        block_gemm<SPLIT>(64, 64, V, 1.f, dVt, V, 1, Vf, 1, V, dT, 64, 1, true, stage);
        for (int e = tid; e < 4096; e += kT) dT[e] *= __ldg(Bt + (e & 63));
        __syncthreads();
        // T^T dW -> dKp (then scaled by beta), dbeta += rows of (T^T dW) . Kp
        block_gemm<SPLIT>(64, K, 64, 1.f, Tm, 1, 64, dW, K, 1, dKp, K, 1, false, stage);
        // T^T dVt -> dW's area (dW is consumed)
        float *TtdU = dW;
        block_gemm<SPLIT>(64, V, 64, 1.f, Tm, 1, 64, dVt, V, 1, TtdU, V, 1, false, stage);
        for (int t = warp; t < 64; t += kT / 32) {
            float s = 0.f;
            for (int i = lane; i < K; i += 32) s = fmaf(dKp[t * K + i], Kp[t * K + i], s);
            for (int j = lane; j < V; j += 32) s = fmaf(TtdU[t * V + j], Vf[t * V + j], s);
            s = warp_sum(s);
            if (lane == 0) dbeta[t] = s;
        }
        __syncthreads();
        for (int e = tid; e < 64 * K; e += kT) dKp[e] *= __ldg(Bt + e / K);
        // dv = diag(beta) T^T dVt
        T *dv = static_cast<T *>(a.dv);
        for (int e4 = tid; e4 < 16 * V; e4 += kT) {
            const int t = e4 / (V / 4), j = 4 * e4 - t * V;
            const float b = __ldg(Bt + t);
            const float4 x = ld4f(TtdU + 4 * e4);
            if (t < nv)
                st4<T>(dv + (bos + row0 + t) * (int64_t)a.H_v * V + (int64_t)h * V + j,
                       make_float4(b * x.x, b * x.y, b * x.z, b * x.w));
        }
        // dL = -T^T dT T^T (strictly lower): X = dT T^T, dL = -T^T X into dT's area
        block_gemm<SPLIT>(64, 64, 64, 1.f, dT, 64, 1, Tm, 1, 64, X, 64, 1, false, stage);
        block_gemm<SPLIT>(64, 64, 64, -1.f, Tm, 1, 64, X, 64, 1, dT, 64, 1, false, stage);
        float *dL = dT;
        for (int e = tid; e < 4096; e += kT)
            if ((e & 63) >= (e >> 6)) dL[e] = 0.f;
        __syncthreads();
        // dbeta += rows of dL . M;  dM = diag(beta) dL (in place)
        for (int t = warp; t < 64; t += kT / 32) {
            float s = 0.f;
            for (int s2 = lane; s2 < t; s2 += 32) s = fmaf(dL[t * 64 + s2], Mm[t * 64 + s2], s);
            s = warp_sum(s);
            if (lane == 0) dbeta[t] += s;
        }
        __syncthreads();
        for (int e = tid; e < 4096; e += kT) dL[e] *= __ldg(Bt + (e >> 6));
        __syncthreads();
        // dKp += dM Km;  dKm += dM^T Kp
        block_gemm<SPLIT>(64, K, 64, 1.f, dL, 64, 1, Km, K, 1, dKp, K, 1, true, stage);
        block_gemm<SPLIT>(64, K, 64, 1.f, dL, 1, 64, Kp, K, 1, dKm, K, 1, true, stage);
    } else {
        // decay-only: U = V, W = 0: dv = dVt
        T *dv = static_cast<T *>(a.dv);
        for (int e4 = tid; e4 < 16 * V; e4 += kT) {
            const int t = e4 / (V / 4), j = 4 * e4 - t * V;
            if (t < nv) st4<T>(dv + (bos + row0 + t) * (int64_t)a.H_v * V + (int64_t)h * V + j, __ldg(
                                   reinterpret_cast<const float4 *>(dVt) + e4));
        }
        for (int e = tid; e < 64 * K; e += kT) dKp[e] = 0.f;
        __syncthreads();
    }

    // dq, dk (atomically when several value heads share a key head's rows, else written
    // once each), dgamma in dQp's area
    float *dqa = a.dq_acc, *dka = a.dk_acc;
    T *dq = static_cast<T *>(a.dq), *dk = static_cast<T *>(a.dk);
#pragma unroll 2
    for (int e4 = tid; e4 < 16 * K; e4 += kT) {
        const int t = e4 / (K / 4), i = 4 * e4 - t * K;
        const float4 g4 = __ldg(reinterpret_cast<const float4 *>(Gm) + e4);
        const float4 n4 = __ldg(reinterpret_cast<const float4 *>(Gm + 63 * K + i));
        const float4 qp4 = __ldg(reinterpret_cast<const float4 *>(Qp) + e4);
        const float4 kp4 = __ldg(reinterpret_cast<const float4 *>(Kp) + e4);
        const float4 km4 = __ldg(reinterpret_cast<const float4 *>(Km) + e4);
        const float4 kb4 = __ldg(reinterpret_cast<const float4 *>(Kb) + e4);
        const float4 vq4 = ld4f(dQp + 4 * e4), vkp4 = ld4f(dKp + 4 * e4), vkm4 = ld4f(dKm + 4 * e4),
                     vkb4 = ld4f(dKb + 4 * e4);
        const float gam[4] = {g4.x, g4.y, g4.z, g4.w}, gn[4] = {n4.x, n4.y, n4.z, n4.w};
        const float qp[4] = {qp4.x, qp4.y, qp4.z, qp4.w}, kp[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
        const float km[4] = {km4.x, km4.y, km4.z, km4.w}, kb[4] = {kb4.x, kb4.y, kb4.z, kb4.w};
        const float vq[4] = {vq4.x, vq4.y, vq4.z, vq4.w}, vkp[4] = {vkp4.x, vkp4.y, vkp4.z, vkp4.w};
        const float vkm[4] = {vkm4.x, vkm4.y, vkm4.z, vkm4.w}, vkb[4] = {vkb4.x, vkb4.y, vkb4.z, vkb4.w};
        float gq[4], gk[4], dgam[4], dkb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float ep = expf(gam[j]), em = expf(-gam[j]), eb = expf(gn[j] - gam[j]);
            gq[j] = a.scale * ep * vq[j];
            gk[j] = ep * vkp[j] + em * vkm[j] + eb * vkb[j];
            dgam[j] = vq[j] * qp[j] + vkp[j] * kp[j] - vkm[j] * km[j] - vkb[j] * kb[j];
            dkb[j] = vkb[j] * kb[j];
        }
        if (t < nv) {
            const int64_t o = ((bos + row0 + t) * a.H_k + hk) * K + i;
            if (a.direct_qk) {
                st4<T>(dq + o, make_float4(gq[0], gq[1], gq[2], gq[3]));
                st4<T>(dk + o, make_float4(gk[0], gk[1], gk[2], gk[3]));
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    atomicAdd(dqa + o + j, gq[j]);
                    atomicAdd(dka + o + j, gk[j]);
                }
            }
        }
        st4f(dQp + 4 * e4, make_float4(dgam[0], dgam[1], dgam[2], dgam[3]));  // dgamma
        st4f(dKb + 4 * e4, make_float4(dkb[0], dkb[1], dkb[2], dkb[3]));      // for dGn
    }
    __syncthreads();
    for (int i = tid; i < K; i += kT) {
        float s = dEG[i] * EG[i];
        for (int t = 0; t < 64; ++t) s += dKb[t * K + i];
        dGn[i] = s;
    }
    __syncthreads();
    // dg: reverse cumulative sum over the chunk's tokens, plus dGn
    float *dgamma = dQp;
    if (!GATE_HEAD) {
        for (int i = tid; i < K; i += kT) {
            float acc = dGn[i];
            for (int t = 63; t >= 0; --t) {
                acc += dgamma[t * K + i];
                if (t < nv) a.dg[((bos + row0 + t) * a.H_v + h) * K + i] = acc;
            }
        }
    } else {
        // one gate per (token, head): the channels' sums
        for (int i = tid; i < K; i += kT) {
            float acc = dGn[i];
            for (int t = 63; t >= 0; --t) {
                acc += dgamma[t * K + i];
                dgamma[t * K + i] = acc;
            }
        }
        __syncthreads();
        for (int t = warp; t < nv; t += kT / 32) {
            float s = 0.f;
            for (int i = lane; i < K; i += 32) s += dgamma[t * K + i];
            s = warp_sum(s);
            if (lane == 0) a.dg[(bos + row0 + t) * a.H_v + h] = s;
        }
    }
    if (!a.decay_only && a.dbeta != nullptr)
        for (int t = tid; t < nv; t += kT) a.dbeta[(bos + row0 + t) * a.H_v + h] = dbeta[t];
}

// ---- grads on tcgen05 (bf16 inputs, d_k = d_v = 128, with beta) -------------------------------
// One CTA per (value head, window): every product of the chunk's gradient is a kind::tf32
// MMA with its accumulator in TMEM. The four per-token gradients are kept transposed, as
// [d][t] accumulators of M = 128 rows (d) and N = 64 columns (t), so that they fill TMEM's
// lanes and the epilogue reads one channel per thread:
//   G1   S dO^T, S dVt^T      -> dQp^T (then += Km^T dA^T), -dW^T (negated in place)
//   GA   dO Vt^T, dVt V^T     -> dA, dT (64 x 64, M = 64)
//   dT  += dW Kp^T;  dT <- dT diag(beta), dbeta += column sums of T . dT (before the scaling)
//   X    dT T^T;  dL = -T^T X (strictly lower), dbeta += rows of dL . M, dM = diag(beta) dL
//   F12b Km^T [dA; dM]^T     -> dQp^T, dKp^T (one N = 128 product)
//   F3   [Qp^T | Kp^T] [dA^T | dM^T]^T -> dKm^T (one K = 128 product)
// and, off that chain,
//   G2   dS' Vt^T             -> dKb^T
//   F2a  dW^T (diag(beta) T^T)^T -> dKp^T (= (diag(beta) T^T dW)^T), dv^T = dVt^T (diag(beta) T^T)^T
// then dq, dk, dgamma and the reverse cumulative sum per channel. Operands come from the
// scratch by TMA (128-byte swizzle, K-major: the scratch holds the transposed copies these
// products need) or are written by the read-back warps in the same layout; two of them are
// read from TMEM. Shared memory is five regions whose tiles follow one another as the
// products retire (offsets in bytes):
//   R0 [0, 64K)       S_e -> dS' -> diag(beta) T^T, dVt^T -> [Qp^T | Kp^T]
//   R1 [64K, 128K)    [dVt; dO] -> [dA; dM] and [dA^T | dM^T]
//   R2 [128K, 160K)   Vt -> X^T (upper half) -> Km^T
//   R3 [160K, 192K)   V -> Kp -> T, T^T -> gamma [t][d]
//   R4 [192K, 224K)   dW -> read-back scratch, dbeta parts, exchanges
// and Kb [t][d] over [dA; dM] for the epilogue, which reads Qp, Kp and Km from the K-major
// tiles of the last products.
// Roles: warps 0-7 read back and run the epilogue (warp w: TMEM lanes 32 (w % 4) .., column
// half w / 4); warp 8 lane 0 issues every copy and MMA, the chain's products first. Each
// barrier completes once. (Bulk L2 prefetches of the later operands, issued early from a warp
// of their own, made the kernel slower: they delay the copies issued after them.)
// D[tmem] (+)= A[smem] * B[smem], tf32 (K = 8 per instruction); issued by one thread.
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// n tf32 MMAs along K (8 elements each) into D: A and B K-major in shared memory with their
// 32-element atoms a_atom / b_atom bytes apart (mma_run_ss), or A in TMEM, 8 columns per step
// (mma_run_ts); the first one overwrites D unless acc. Out of line: one copy serves every
// product of the kernel.
__device__ __noinline__ void mma_run_ss(uint32_t d, uint32_t a, uint32_t a_atom, uint32_t b, uint32_t b_atom,
                                        uint32_t idesc, int n, bool acc) {
#pragma unroll 1
    for (int s = 0; s < n; ++s) mma_tf32_ss(d, tcu::dK(a, a_atom, s), tcu::dK(b, b_atom, s), idesc, acc || s > 0);
}
__device__ __noinline__ void mma_run_ts(uint32_t d, uint32_t a_tmem, uint32_t b, uint32_t b_atom, uint32_t idesc, int n,
                                        bool acc) {
#pragma unroll 1
    for (int s = 0; s < n; ++s) tc5::mma_tf32_ts(d, a_tmem + 8 * s, tcu::dK(b, b_atom, s), idesc, acc || s > 0);
}

struct GrTc {
    static constexpr int R0 = 0, R1 = 65536, R2 = 131072, R3 = 163840, R4 = 196608;
    // in R4 once dW is consumed, past the read-back scratch ([64][65] floats)
    static constexpr int oDB1 = R4 + 16896;          // dbeta, T . dT part [64]
    static constexpr int oDB3 = oDB1 + 256;          // dbeta, dL . M part, by column half [2][64]
    static constexpr int oDGH = oDB3 + 512;          // per-head dg [64]
    static constexpr int oDEG = 229376;              // dEG [128]
    static constexpr int oBar = oDEG + 512;
    static constexpr int oBT = oBar + 8 * 24;        // beta [64]
    static constexpr int kBytes = oBT + 256 + 1024;  // + alignment slack
};
// (the kernel's static shared memory takes 1 KB of the 227 KB)
static_assert(GrTc::kBytes <= 232448 - 1024 && GrTc::oDGH + 256 <= GrTc::oDEG, "shared memory");
constexpr int kGrThreads = 288;
// TMEM columns
constexpr uint32_t tgA = 0, tgT = 64, tgKB = 128, tgKM = 192, tgW = 256, tgQP = 320, tgKP = 384, tgV = 448;
enum {
    GB_LA = 0, GB_LV, GB_LDS, GB_LKP, GB_LTB, GB_LTM, GB_LKMT, GB_LQ, GB_LG, GB_LKB,  // copies
    GB_G1, GB_GT, GB_GA, GB_G2, GB_DT, GB_DV, GB_X, GB_DL, GB_F,              // MMA commits
    GB_DW, GB_DTS, GB_XT, GB_DM,                                       // read-backs (8 warps)
    GB_Z, kGrBars
};
constexpr int kGrLoads = GB_LKB + 1;
static_assert(kGrBars <= 24, "barrier area");

// The four tensor maps view a slot as rows of 128 or 64 floats; boxes of 32 floats x 64 or
// 128 rows land as 128-byte-swizzled K-major atoms.
struct GrMaps {
    CUtensorMap w128r64, w128r128, w64r64, w64r128;
};

// Element (row, k) of a K-major tile of 32-column atoms `atom_bytes` apart: byte offset.
__device__ __forceinline__ uint32_t kmaj(int atom_bytes, int row, int k) {
    const int kk = k & 31;
    return (uint32_t)((k >> 5) * atom_bytes + row * 128 + (((kk >> 2) ^ (row & 7)) << 4) + (kk & 3) * 4);
}

template <bool GATE_HEAD>
__global__ void __launch_bounds__(kGrThreads, 1) bwd_grads_tc_kernel(const BwdArgs a,
                                                                      const __grid_constant__ GrMaps mp) {
    using namespace tc5;
    using tcu::tmem_ld32;
    using tcu::mbar_arrive;
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + GrTc::oBar);
    float *dEG = reinterpret_cast<float *>(sm + GrTc::oDEG);
    float *db1 = reinterpret_cast<float *>(sm + GrTc::oDB1);
    float *db3 = reinterpret_cast<float *>(sm + GrTc::oDB3);
    float *dgh = reinterpret_cast<float *>(sm + GrTc::oDGH);
    __shared__ uint32_t tslot;
    __shared__ int abort_w;
    volatile int *abort_flag = &abort_w;
    int n, c, len;
    int64_t bos;
    if (!window_owner(a, blockIdx.y, n, c, bos, len)) return;
    constexpr int K = 128, V = 128;
    const int h = blockIdx.x, hk = h / a.group, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Lay L = make_lay(K, V);
    const int64_t sl = slot_of(a, bos, n, c, h);
    const float *S = a.scratch + sl * L.total;
    const int row0 = c * 64, nv = min(64, len - row0);
    if (tid == 0) {
        for (int i = 0; i < kGrBars; ++i)
            mbar_init(&bars[i], (i >= GB_DW && i <= GB_DM) ? 8 : 1);
        abort_w = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tslot, sb = smem_u32(sm);

    if (warp == 8) {
        if (lane == 0) {
            bool ok = true;
            bool armed[kGrLoads] = {}, done[kGrLoads] = {};
            const int z = (int)sl;
            auto arm = [&](int b, uint32_t bytes) {
                mbar_arrive_expect_tx(&bars[b], bytes);
                armed[b] = true;
            };
            auto wait_load = [&](int b) {
                if (ok) ok = st_wait(&bars[b], 0, abort_flag, a.err);
                if (ok) done[b] = true;
            };
            auto wait_bar = [&](int b) {
                if (ok) ok = st_wait(&bars[b], 0, abort_flag, a.err);
            };
            // 128-float rows: S_e, [dVt; dO], Vt, V
            arm(GB_LA, 131072);
#pragma unroll
            for (int at = 0; at < 4; ++at) {
                tma_load_3d(sm + GrTc::R0 + at * 16384, &mp.w128r128, &bars[GB_LA], 32 * at, (int)(L.se / 128), z);
                tma_load_3d(sm + GrTc::R1 + at * 16384, &mp.w128r64, &bars[GB_LA], 32 * at, (int)(L.dvt / 128), z);
                tma_load_3d(sm + GrTc::R1 + at * 16384 + 8192, &mp.w128r64, &bars[GB_LA], 32 * at, (int)(L.dof / 128), z);
            }
            arm(GB_LV, 65536);
#pragma unroll
            for (int at = 0; at < 4; ++at) {
                tma_load_3d(sm + GrTc::R2 + at * 8192, &mp.w128r64, &bars[GB_LV], 32 * at, (int)(L.vt / 128), z);
                tma_load_3d(sm + GrTc::R3 + at * 8192, &mp.w128r64, &bars[GB_LV], 32 * at, (int)(L.vf / 128), z);
            }
            const uint32_t i128x128 = idesc_tf32(128, 128), i128x64 = idesc_tf32(128, 64), i64x64 = idesc_tf32(64, 64);
            // G1: [ -dW^T | dQp^T ] = S_e [dVt; dO]^T
            wait_load(GB_LA);
            if (ok) {
                fence_after_sync();
                mma_run_ss(tmem + tgW, sb + GrTc::R0, 16384, sb + GrTc::R1, 16384, i128x128, 16, false);
                commit(&bars[GB_G1]);
            }
            // dT = dVt V^T (V is then free for Kp), dA = dO Vt^T
            wait_load(GB_LV);
            if (ok) {
                mma_run_ss(tmem + tgT, sb + GrTc::R1, 16384, sb + GrTc::R3, 8192, i64x64, 16, false);
                commit(&bars[GB_GT]);
                mma_run_ss(tmem + tgA, sb + GrTc::R1 + 8192, 16384, sb + GrTc::R2, 8192, i64x64, 16, false);
                commit(&bars[GB_GA]);
            }
            // dS' over S_e; Kp over V
            wait_bar(GB_G1);
            if (ok) {
                arm(GB_LDS, 65536);
#pragma unroll
                for (int at = 0; at < 4; ++at)
                    tma_load_3d(sm + GrTc::R0 + at * 16384, &mp.w128r128, &bars[GB_LDS], 32 * at, (int)(L.dsx / 128), z);
            }
            wait_bar(GB_GT);
            if (ok) {
                arm(GB_LKP, 32768);
#pragma unroll
                for (int at = 0; at < 4; ++at)
                    tma_load_3d(sm + GrTc::R3 + at * 8192, &mp.w128r64, &bars[GB_LKP], 32 * at, (int)(L.kp / 128), z);
            }
            // dT += dW Kp^T
            wait_bar(GB_DW);
            wait_load(GB_LKP);
            if (ok) {
                fence_after_sync();
                mma_run_ss(tmem + tgT, sb + GrTc::R4, 8192, sb + GrTc::R3, 8192, i64x64, 16, true);
                commit(&bars[GB_DT]);
            }
            // G2: dKb^T = dS' Vt^T (runs while dT is read back)
            wait_load(GB_LDS);
            if (ok) {
                mma_run_ss(tmem + tgKB, sb + GrTc::R0, 16384, sb + GrTc::R2, 8192, i128x64, 16, false);
                commit(&bars[GB_G2]);
            }
            // T and T^T over Kp
            wait_bar(GB_DT);
            if (ok) {
                arm(GB_LTM, 32768);
#pragma unroll
                for (int at = 0; at < 2; ++at) {
                    tma_load_3d(sm + GrTc::R3 + at * 8192, &mp.w64r64, &bars[GB_LTM], 32 * at, (int)(L.t / 64), z);
                    tma_load_3d(sm + GrTc::R3 + 16384 + at * 8192, &mp.w64r64, &bars[GB_LTM], 32 * at, (int)(L.tt / 64), z);
                }
            }
            // diag(beta) T^T and dVt^T over dS'
            wait_bar(GB_G2);
            if (ok) {
                arm(GB_LTB, 49152);
#pragma unroll
                for (int at = 0; at < 2; ++at) {
                    tma_load_3d(sm + GrTc::R0 + at * 8192, &mp.w64r64, &bars[GB_LTB], 32 * at, (int)(L.tbt / 64), z);
                    tma_load_3d(sm + GrTc::R0 + 16384 + at * 16384, &mp.w64r128, &bars[GB_LTB], 32 * at,
                                (int)(L.dvtt / 64), z);
                }
            }
            // X = dT T^T (A: the scaled dT in TMEM; the read-back waited for T)
            wait_bar(GB_DTS);
            if (ok) {
                done[GB_LTM] = true;
                fence_after_sync();
                mma_run_ts(tmem + tgA, tmem + tgT, sb + GrTc::R3, 8192, i64x64, 8, false);
                commit(&bars[GB_X]);
            }
            // F2a: dKp^T = dW^T (diag(beta) T^T)^T (A: dW^T in TMEM); dv^T = dVt^T (diag(beta) T^T)^T
            wait_load(GB_LTB);
            if (ok) {
                mma_run_ts(tmem + tgKP, tmem + tgW, sb + GrTc::R0, 8192, i128x64, 8, false);
                mma_run_ss(tmem + tgV, sb + GrTc::R0 + 16384, 16384, sb + GrTc::R0, 8192, i128x64, 8, false);
                commit(&bars[GB_DV]);
            }
            // T^T X (dL = minus its strict lower part)
            wait_bar(GB_XT);
            if (ok) {
                fence_after_sync();
                mma_run_ss(tmem + tgA, sb + GrTc::R3 + 16384, 8192, sb + GrTc::R2 + 16384, 8192, i64x64, 8, false);
                commit(&bars[GB_DL]);
            }
            // [Qp^T | Kp^T] over diag(beta) T^T and dVt^T; Km^T over X^T
            wait_bar(GB_DV);
            if (ok) {
                arm(GB_LQ, 65536);
#pragma unroll
                for (int at = 0; at < 2; ++at) {
                    tma_load_3d(sm + GrTc::R0 + at * 16384, &mp.w64r128, &bars[GB_LQ], 32 * at, (int)(L.qpt / 64), z);
                    tma_load_3d(sm + GrTc::R0 + 32768 + at * 16384, &mp.w64r128, &bars[GB_LQ], 32 * at,
                                (int)(L.kpt / 64), z);
                }
            }
            wait_bar(GB_DL);
            if (ok) {
                arm(GB_LKMT, 32768);
#pragma unroll
                for (int at = 0; at < 2; ++at)
                    tma_load_3d(sm + GrTc::R2 + at * 16384, &mp.w64r128, &bars[GB_LKMT], 32 * at, (int)(L.kmt / 64), z);
                // gamma [t][d] for the epilogue over T and T^T
                arm(GB_LG, 32768);
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 sb + GrTc::R3),
                             "l"(S + L.gm), "r"(32768), "r"(smem_u32(&bars[GB_LG]))
                             : "memory");
            }
            // F12b: [dQp^T | dKp^T] += Km^T [dA; dM]^T;  F3: dKm^T = [Qp^T | Kp^T] [dA^T | dM^T]^T
            wait_bar(GB_DM);
            wait_load(GB_LQ);
            if (ok) {
                fence_after_sync();
                mma_run_ss(tmem + tgKM, sb + GrTc::R0, 16384, sb + GrTc::R1 + 32768, 8192, i128x64, 16, false);
            }
            wait_load(GB_LKMT);
            if (ok) {
                mma_run_ss(tmem + tgQP, sb + GrTc::R2, 16384, sb + GrTc::R1, 16384, i128x128, 8, true);
                commit(&bars[GB_F]);
            }
            // Kb [t][d] for the epilogue over [dA; dM]
            wait_bar(GB_F);
            if (ok) {
                arm(GB_LKB, 32768);
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 sb + GrTc::R1),
                             "l"(S + L.kb), "r"(32768), "r"(smem_u32(&bars[GB_LKB]))
                             : "memory");
            }
            // drain: every MMA issued, every copy armed
            commit(&bars[GB_Z]);
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[GB_Z], 0) && clock64() - t0 < kDefaultWaitCycles) {}
            for (int b = 0; b < kGrLoads; ++b) {
                if (armed[b] && !done[b]) {
                    const long long t1 = clock64();
                    while (!mbar_try_wait(&bars[b], 0) && clock64() - t1 < kDefaultWaitCycles) {}
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        // ---- read-back and epilogue: warps 0-7 ----
        const int q = warp & 3, hw = warp >> 2;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int t16 = 16 * q + (lane & 15);  // row of an M = 64 accumulator (lanes 0-15)
        const bool rl = lane < 16;
        const int dch = 32 * q + lane;          // row of an M = 128 accumulator
        float *Bt = reinterpret_cast<float *>(sm + GrTc::oBT);
        if (tid < 64) Bt[tid] = __ldg(S + L.bt + tid);
        tcu::bar_named(1, 256);
        bool ok = true;
        auto arrive = [&](int b) {
            fence_proxy_async();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[b]);
        };
        // every wait of the 256 threads ends the same way for all of them (named barrier 1)
        auto wait_all = [&](int b) { return !tcu::bar_or(1, 256, !st_wait(&bars[b], 0, abort_flag, a.err)); };
        do {
            // -dW^T -> dW^T in place (the A operand of F2a) and dW [t][d] into R4
            if (!(ok = wait_all(GB_G1))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgW + 32 * hw, v);
                uint32_t w0[16], w1[16];
                unsigned char *DW = sm + GrTc::R4;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float x = -v[j];
                    if (j < 16) w0[j] = __float_as_uint(x); else w1[j - 16] = __float_as_uint(x);
                    *reinterpret_cast<uint32_t *>(DW + kmaj(8192, 32 * hw + j, dch)) = tcu::tf32(x);
                }
                tmem_st16(tmem + lane_off + tgW + 32 * hw, w0);
                tmem_st16(tmem + lane_off + tgW + 32 * hw + 16, w1);
                tmem_st_wait();
            }
            arrive(GB_DW);
            // dA (lower, with the diagonal) -> [dA; .] rows 0-63 and [dA^T | .] atoms 0-1 in R1
            if (!(ok = wait_all(GB_GA))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgA + 32 * hw, v);
                if (rl) {
                    unsigned char *AM = sm + GrTc::R1, *AMT = sm + GrTc::R1 + 32768;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int s2 = 32 * hw + j;
                        const float x = s2 <= t16 ? v[j] : 0.f;
                        *reinterpret_cast<uint32_t *>(AM + kmaj(16384, t16, s2)) = tcu::tf32(x);
                        *reinterpret_cast<uint32_t *>(AMT + kmaj(8192, s2, t16)) = tcu::tf32(x);
                    }
                }
            }
            // dT: dbeta += column sums of T . dT, then dT <- dT diag(beta) in place
            if (!(ok = wait_all(GB_DT))) break;
            if (!(ok = wait_all(GB_LTM))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgT + 32 * hw, v);
                float *P = reinterpret_cast<float *>(sm + GrTc::R4);  // [64 r][65]
                const unsigned char *TM = sm + GrTc::R3;
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s2 = 32 * hw + j;
                    if (rl) P[t16 * 65 + s2] = v[j] * *reinterpret_cast<const float *>(TM + kmaj(8192, t16, s2));
                    const float y = v[j] * Bt[s2];
                    if (j < 16) w0[j] = __float_as_uint(y); else w1[j - 16] = __float_as_uint(y);
                }
                tmem_st16(tmem + lane_off + tgT + 32 * hw, w0);
                tmem_st16(tmem + lane_off + tgT + 32 * hw + 16, w1);
                tmem_st_wait();
            }
            arrive(GB_DTS);
            tcu::bar_named(1, 256);  // P is complete
            if (tid < 64) {
                float acc = 0.f;
                const float *P = reinterpret_cast<const float *>(sm + GrTc::R4);
                for (int r = 0; r < 64; ++r) acc += P[r * 65 + tid];
                db1[tid] = acc;
                dgh[tid] = 0.f;
            }
            // X -> X^T into R2's upper half (Vt is consumed: X follows G2)
            if (!(ok = wait_all(GB_X))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgA + 32 * hw, v);
                if (rl) {
                    unsigned char *XT = sm + GrTc::R2 + 16384;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        *reinterpret_cast<uint32_t *>(XT + kmaj(8192, 32 * hw + j, t16)) = tcu::tf32(v[j]);
                }
            }
            arrive(GB_XT);
            // dL = -(T^T X) strictly lower: dM = diag(beta) dL; then (off the chain) dbeta +=
            // rows of dL . M
            if (!(ok = wait_all(GB_DL))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgA + 32 * hw, v);
                if (rl) {
                    unsigned char *AM = sm + GrTc::R1, *AMT = sm + GrTc::R1 + 32768;
                    const float bt = Bt[t16];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int s2 = 32 * hw + j;
                        v[j] = s2 < t16 ? -v[j] : 0.f;
                        const float dm = bt * v[j];
                        *reinterpret_cast<uint32_t *>(AM + kmaj(16384, 64 + t16, s2)) = tcu::tf32(dm);
                        *reinterpret_cast<uint32_t *>(AMT + kmaj(8192, s2, 64 + t16)) = tcu::tf32(dm);
                    }
                }
                arrive(GB_DM);
                if (rl) {
                    const float4 *Mr = reinterpret_cast<const float4 *>(S + L.m + t16 * 64 + 32 * hw);
                    float part = 0.f;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 m4 = __ldg(Mr + j4);
                        part = fmaf(v[4 * j4], m4.x, part);
                        part = fmaf(v[4 * j4 + 1], m4.y, part);
                        part = fmaf(v[4 * j4 + 2], m4.z, part);
                        part = fmaf(v[4 * j4 + 3], m4.w, part);
                    }
                    db3[hw * 64 + t16] = part;
                }
            }
            // dv = rows of dv^T, bf16 (off the chain)
            if (!(ok = wait_all(GB_DV))) break;
            fence_after_sync();
            {
                float v[32];
                tmem_ld32(tmem + lane_off + tgV + 32 * hw, v);
                __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(a.dv) + (bos + row0) * (int64_t)a.H_v * V + (int64_t)h * V + dch;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = 32 * hw + j;
                    if (t < nv) dv[(int64_t)t * a.H_v * V] = __float2bfloat16_rn(v[j]);
                }
            }

            // dEG[d] = rows of dS' . S_e (a warp per row, eight rows' loads in flight)
#pragma unroll 1
            for (int d0 = 8 * warp; d0 < K; d0 += 64) {
                float4 x[8], y[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    x[i] = __ldg(reinterpret_cast<const float4 *>(S + L.dsx + (d0 + i) * V) + lane);
                    y[i] = __ldg(reinterpret_cast<const float4 *>(S + L.se + (d0 + i) * V) + lane);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float sdot = warp_sum(x[i].x * y[i].x + x[i].y * y[i].y + x[i].z * y[i].z + x[i].w * y[i].w);
                    if (lane == 0) dEG[d0 + i] = sdot;
                }
            }
            // ---- epilogue ----
            if (!(ok = wait_all(GB_F))) break;
            if (!(ok = wait_all(GB_LG))) break;
            if (!(ok = wait_all(GB_LKB))) break;
            fence_after_sync();
            const unsigned char *QKT = sm + GrTc::R0, *KMT = sm + GrTc::R2;
            const float *Ekb = reinterpret_cast<const float *>(sm + GrTc::R1);
            const float *Egm = reinterpret_cast<const float *>(sm + GrTc::R3);
            const float gn = Egm[63 * K + dch];
            float dgam[32];
            float kbsum = 0.f;
            float *dqa = a.dq_acc, *dka = a.dk_acc;
            __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(a.dq), *dk = static_cast<__nv_bfloat16 *>(a.dk);
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                const int tb = 32 * hw + 16 * p;
                float vq[16], vkp[16], vkm[16], vkb[16];
                tcu::tmem_ld16(tmem + lane_off + tgQP + tb, vq);
                tcu::tmem_ld16(tmem + lane_off + tgKP + tb, vkp);
                tcu::tmem_ld16(tmem + lane_off + tgKM + tb, vkm);
                tcu::tmem_ld16(tmem + lane_off + tgKB + tb, vkb);
                tcu::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = tb + j;
                    const int e = t * K + dch;
                    const float qp = *reinterpret_cast<const float *>(QKT + kmaj(16384, dch, t));
                    const float kp = *reinterpret_cast<const float *>(QKT + kmaj(16384, dch, 64 + t));
                    const float km = *reinterpret_cast<const float *>(KMT + kmaj(16384, dch, t));
                    const float kb = Ekb[e], gm = Egm[e];
                    const float ep = __expf(gm), em = __expf(-gm), eb = __expf(gn - gm);
                    const float gq = a.scale * ep * vq[j];
                    const float gk = ep * vkp[j] + em * vkm[j] + eb * vkb[j];
                    dgam[16 * p + j] = vq[j] * qp + vkp[j] * kp - vkm[j] * km - vkb[j] * kb;
                    kbsum = fmaf(vkb[j], kb, kbsum);
                    if (t < nv) {
                        const int64_t o = ((bos + row0 + t) * a.H_k + hk) * K + dch;
                        if (a.direct_qk) {
                            dq[o] = __float2bfloat16_rn(gq);
                            dk[o] = __float2bfloat16_rn(gk);
                        } else {
                            atomicAdd(dqa + o, gq);
                            atomicAdd(dka + o, gk);
                        }
                    }
                }
            }
            // dGn and the reverse cumulative sum over the two column halves (exchange in R4)
            float *ex = reinterpret_cast<float *>(sm + GrTc::R4);  // [2][128] kb sums, [128] dgamma totals
            float tot = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) tot += dgam[j];
            ex[hw * 128 + dch] = kbsum;
            if (hw == 1) ex[256 + dch] = tot;
            tcu::bar_named(1, 256);
            float acc = ex[dch] + ex[128 + dch] + dEG[dch] * __ldg(S + L.eg + dch);  // dGn
            if (hw == 0) acc += ex[256 + dch];
            float dgo[32];
#pragma unroll
            for (int j = 31; j >= 0; --j) {
                acc += dgam[j];
                dgo[j] = acc;
            }
            if (!GATE_HEAD) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = 32 * hw + j;
                    if (t < nv) a.dg[((bos + row0 + t) * a.H_v + h) * K + dch] = dgo[j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sdot = warp_sum(dgo[j]);
                    if (lane == 0) atomicAdd(&dgh[32 * hw + j], sdot);
                }
            }
            tcu::bar_named(1, 256);  // dgh and every dbeta part are complete
            if (tid < 64 && tid < nv) {
                const int t = tid;
                if (GATE_HEAD) a.dg[(bos + row0 + t) * a.H_v + h] = dgh[t];
                if (a.dbeta != nullptr) a.dbeta[(bos + row0 + t) * a.H_v + h] = db1[t] + db3[t] + db3[64 + t];
            }
        } while (false);
        if (!ok) *abort_flag = 1;
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T>
__global__ void __launch_bounds__(kT) bwd_finish_kernel(const float *acc, T *out, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x; i < n; i += (int64_t)gridDim.x * kT)
        stf<T>(out + i, acc[i]);
}

size_t grads_smem(int K, int V) {
    const int KV = K > V ? K : V;
    return sizeof(float) * ((size_t)4 * 64 * K + (size_t)64 * KV + 2 * 4096 + 128 + 128 + 64 + kStageFloats);
}

// The tensor map of one [64][cols] fp32 factor of every slot (at `off` floats into the slot):
// 3-D (column, token, slot), boxes of `box_cols` columns x 64 tokens, with the 128-byte
// swizzle (K-major MMA operand tiles) or without (plain row-major tiles).
bool encode_slot_map(CUtensorMap *m, const BwdArgs &a, const Lay &L, int64_t off, int cols, int box_cols, bool swizzle,
                     int64_t nslots) {
    auto enc = tcu::tensor_map_encoder();
    if (enc == nullptr || nslots <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, 64, (cuuint64_t)nslots};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * sizeof(float), (cuuint64_t)L.total * sizeof(float)};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(a.scratch + off), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The slot viewed as rows of `width` floats (64 or 128), boxes of 32 floats x `rows` rows,
// 128-byte swizzle (the gradient kernel's operand tiles).
bool encode_view(CUtensorMap *m, const BwdArgs &a, const Lay &L, int width, int rows, int64_t nslots) {
    auto enc = tcu::tensor_map_encoder();
    if (enc == nullptr || nslots <= 0 || L.total % width != 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)(L.total / width), (cuuint64_t)nslots};
    const cuuint64_t strides[2] = {(cuuint64_t)width * sizeof(float), (cuuint64_t)L.total * sizeof(float)};
    const cuuint32_t box[3] = {32, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.scratch, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool GATE_HEAD>
cudaError_t launch_typed(const BwdArgs &a0, cudaStream_t stream) {
    constexpr bool kSplit = std::is_same<T, float>::value;  // fp32-grade products for fp32 inputs
    BwdArgs a = a0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int K = a.d_k, V = a.d_v;
    const int64_t Ttot = a.cu_seqlens ? (int64_t)a.T : (int64_t)a.N * a.T;
    const int64_t windows = (Ttot + 63) / 64 + a.N;
    const Lay L = make_lay(K, V);
    const size_t slot_bytes = sizeof(float) * (size_t)L.total;
    const size_t scratch_bytes = slot_bytes * (size_t)(windows * a.H_v);
    const size_t acc_elems = (size_t)Ttot * a.H_k * K;
    a.direct_qk = a.group == 1 ? 1 : 0;  // each (token, key head) row then has one writer
    // grouped heads with bf16 outputs: fp32 accumulators, converted at the end
    const bool own_acc = !a.direct_qk && !std::is_same<T, float>::value;
    const size_t acc_bytes = own_acc ? 2 * sizeof(float) * acc_elems : 0;
    cudaMemPool_t pool = nullptr;
    e = scratch_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    void *buf = nullptr;
    e = cudaMallocFromPoolAsync(&buf, scratch_bytes + acc_bytes + 256, pool, stream);
    if (e != cudaSuccess) return e;
    a.scratch = static_cast<float *>(buf);
    if (own_acc) {
        a.dq_acc = reinterpret_cast<float *>(static_cast<unsigned char *>(buf) + scratch_bytes);
        a.dk_acc = a.dq_acc + acc_elems;
    } else {
        a.dq_acc = static_cast<float *>(a.dq);
        a.dk_acc = static_cast<float *>(a.dk);
    }
    if (acc_elems > 0 && !a.direct_qk) {
        e = cudaMemsetAsync(a.dq_acc, 0, sizeof(float) * acc_elems, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.dk_acc, 0, sizeof(float) * acc_elems, stream);
    }
    const size_t ssmem = states_smem(K), asmem = adjoint_smem(K);
    const size_t gsmem = grads_smem(K, V);
    const size_t psmem = prep_smem(K);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_grads_kernel<T, GATE_HEAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)gsmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_prep_kernel<T, GATE_HEAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)psmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_states_kernel<kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_adjoint_kernel<kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)asmem);
    if (e == cudaSuccess && windows > 0 && Ttot > 0) {
        const dim3 gw(a.H_v, (unsigned)windows);
        // tcgen05 scans for bf16 inputs with d = 128; the tcgen05 gradient kernel with them
        // when beta is given
        const int64_t nslots = windows * a.H_v;
        CUtensorMap wmap, umap, kbmap, domap;
        GrMaps gmaps;
        const bool scan_tc = !kSplit && K == 128 && V == 128 &&
                             encode_slot_map(&wmap, a, L, L.wm, K, 32, true, nslots) &&
                             encode_slot_map(&umap, a, L, L.u, V, 64, false, nslots) &&
                             encode_slot_map(&kbmap, a, L, L.kb, K, 32, true, nslots) &&
                             encode_slot_map(&domap, a, L, L.dof, V, 64, false, nslots);
        const bool grads_tc = scan_tc && !a.decay_only && encode_view(&gmaps.w128r64, a, L, 128, 64, nslots) &&
                              encode_view(&gmaps.w128r128, a, L, 128, 128, nslots) &&
                              encode_view(&gmaps.w64r64, a, L, 64, 64, nslots) &&
                              encode_view(&gmaps.w64r128, a, L, 64, 128, nslots);
        a.tc = grads_tc ? 1 : 0;
        bwd_prep_kernel<T, GATE_HEAD><<<gw, kT, psmem, stream>>>(a);
        e = cudaGetLastError();
        if (e == cudaSuccess) {
            if (scan_tc) {
                e = cudaFuncSetAttribute(bwd_states_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         StTc::kBytes);
                if (e == cudaSuccess) {
                    bwd_states_tc_kernel<<<dim3(2, a.H_v, a.N), kT, StTc::kBytes, stream>>>(a, wmap, umap);
                    e = cudaGetLastError();
                }
            } else {
                bwd_states_kernel<kSplit><<<dim3(V / 64, a.H_v, a.N), kT, ssmem, stream>>>(a);
                e = cudaGetLastError();
            }
        }
        if (e == cudaSuccess) {
            if (scan_tc) {
                e = cudaFuncSetAttribute(bwd_adjoint_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         AdTc::kBytes);
                if (e == cudaSuccess) {
                    bwd_adjoint_tc_kernel<<<dim3(2, a.H_v, a.N), kT, AdTc::kBytes, stream>>>(a, kbmap, domap);
                    e = cudaGetLastError();
                }
            } else {
                bwd_adjoint_kernel<kSplit><<<dim3(V / 64, a.H_v, a.N), kT, asmem, stream>>>(a);
                e = cudaGetLastError();
            }
        }
        if (e == cudaSuccess) {
            if (grads_tc) {
                e = cudaFuncSetAttribute(bwd_grads_tc_kernel<GATE_HEAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GrTc::kBytes);
                if (e == cudaSuccess) {
                    bwd_grads_tc_kernel<GATE_HEAD><<<gw, kGrThreads, GrTc::kBytes, stream>>>(a, gmaps);
                    e = cudaGetLastError();
                }
            } else {
                bwd_grads_kernel<T, GATE_HEAD><<<gw, kT, gsmem, stream>>>(a);
                e = cudaGetLastError();
            }
        }
        if (e == cudaSuccess && own_acc && acc_elems > 0) {
            const int grid = (int)std::min<int64_t>((int64_t)sms * 8, ((int64_t)acc_elems + kT - 1) / kT);
            bwd_finish_kernel<T><<<grid, kT, 0, stream>>>(a.dq_acc, static_cast<T *>(a.dq), (int64_t)acc_elems);
            bwd_finish_kernel<T><<<grid, kT, 0, stream>>>(a.dk_acc, static_cast<T *>(a.dk), (int64_t)acc_elems);
            e = cudaGetLastError();
        }
    } else if (e == cudaSuccess) {
        // no tokens: dh0 = dht (or zero)
        const size_t sb = sizeof(float) * (size_t)a.N * a.H_v * K * V;
        if (a.dh0 != nullptr)
            e = a.dht ? cudaMemcpyAsync(a.dh0, a.dht, sb, cudaMemcpyDeviceToDevice, stream)
                      : cudaMemsetAsync(a.dh0, 0, sb, stream);
    }
    const cudaError_t ef = cudaFreeAsync(buf, stream);
    return e != cudaSuccess ? e : ef;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, bool f32, cudaStream_t stream) {
    if (f32)
        return a.gate_per_head ? launch_typed<float, true>(a, stream) : launch_typed<float, false>(a, stream);
    return a.gate_per_head ? launch_typed<__nv_bfloat16, true>(a, stream)
                           : launch_typed<__nv_bfloat16, false>(a, stream);
}

}  // namespace kda
