// Chunkwise KDA forward for d_k = d_v = 128, bf16 operands, on the 5th-generation tensor
// cores (tcgen05) with accumulators in tensor memory (TMEM).
//
// One CTA of 256 threads runs one (sequence, value head) unit through all its chunks.
// Every product is arranged so that the tensor core's M dimension is 128 (the d_k or d_v
// axis, or the stacked [Kp; Qp] rows), so each MMA runs at full width:
//
//   Gram      D_G [128 x 64]  = [Kp; Qp] Km^T          rows 0-63: M, rows 64-127: Aqk
//   WY        D_W [128 x 64]  = Kp^T T_beta^T           (W^T, d_k x tokens)
//             D_V [128 x 64]  = V^T  T_beta^T           (U^T, d_v x tokens)
//   serial    D_V += -(S^T) W^T                          (Vt^T = U^T - S^T W^T)
//             D_O  = S^T Qp^T;  D_O += Vt^T Aqk^T        (O^T, d_v x tokens)
//             D_S  = Kbar^T Vt                           (the chunk's state increment)
//
// and S <- Diag(e^gamma_n) S + D_S is applied in fp32 registers by the 128 threads of
// warpgroup 0, thread d owning row d of S (d_k x d_v) across the whole sequence. Per chunk
// ("RNN的复兴04:线性注意力并行计算DPLR", §5.3.5; "TileLang 实战：KDA 从零到一–Kimi Delta
// Attention", §3.3): the cumulative log2 gate and the decayed operands (gate pass), the
// Gram matrix, the UT-transform inverse T = (I + diag(beta) M)^-1 (16x16 diagonal blocks by
// forward substitution, then block merges with tf32 mma.sync), T_beta = T diag(beta), the WY
// factors, and the serial step. All operands live in shared memory in the 128-byte-swizzled
// layouts the tensor core reads; nothing but q, k, v, g, beta, h0 (in) and o, ht (out)
// touches HBM.
//
// Every mbarrier wait is bounded (about one second); on a timeout the CTA raises
// KDA_DEVICE_ERR_TIMEOUT, waits (bounded) for its issued MMAs, frees its TMEM and returns.
#include "kda_common.cuh"
#include "tc5.cuh"

namespace kda {

namespace {

using bf16 = __nv_bfloat16;
using namespace tc5;

// Shared-memory plan (byte offsets from a 1024-byte aligned base).
struct TcLayout {
    static constexpr int oRQ = 0;       // raw Q [64][128] bf16 row-major
    static constexpr int oRK = 16384;   // raw K
    static constexpr int oRV = 32768;   // raw V, MN-major: [2 atoms (d_v)][64 token rows][128 B]
    static constexpr int oGA = 49152;   // [2 atoms (d_k)][128 rows][128 B]: rows 0-63 Kp, 64-127 Qp
    static constexpr int oKM = 81920;   // [2][64][128 B] Km; then Aqk (8 KB) + T_beta (8 KB); then O staging
    static constexpr int oAQ = oKM;
    static constexpr int oTB = oKM + 8192;
    static constexpr int oOS = oKM;     // O staging [64][128] bf16 row-major
    static constexpr int oKB = 98304;   // [2][64][128 B] Kbar
    static constexpr int oWB = 114688;  // [128 rows (d_k)][128 B] W, MN-major B operand
    static constexpr int oSB = 131072;  // [2 atoms (d_v)][128 rows (d_k)][128 B] S in bf16, MN-major A
    static constexpr int oVB = 163840;  // [128 rows (d_v)][128 B] Vt in bf16, K-major
    static constexpr int oG = 180224;   // raw G fp32 [64][128]; then L and T fp32 [64][68]
    static constexpr int oL = oG;
    static constexpr int oT = oG + 17408;
    static constexpr int oBeta = oG + 34816;
    static constexpr int oEg = oBeta + 256;
    static constexpr int oBar = oEg + 512;
    static constexpr int oTmemAddr = oBar + 64;
    static constexpr int kBytes = oTmemAddr + 16 + 1024;  // + slack to align the base
};
constexpr int LDF = 68;  // fp32 row stride of L and T

// TMEM columns
constexpr uint32_t tG = 0, tW = 64, tV = 128, tO = 192, tS = 256;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitCycles = 1ll << 31;  // about one second

enum { BAR_G = 0, BAR_W, BAR_V, BAR_S, BAR_Z };

__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// acc (16x16, two m16n8 tiles) += A (16x16) * B (16x16), both fp32 in smem (stride LDF).
__device__ __forceinline__ void mm16_tf32(float (&acc)[2][4], const float *A, const float *B, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a0 = tf32(A[g * LDF + 8 * ks + t]);
        const uint32_t a1 = tf32(A[(g + 8) * LDF + 8 * ks + t]);
        const uint32_t a2 = tf32(A[g * LDF + 8 * ks + t + 4]);
        const uint32_t a3 = tf32(A[(g + 8) * LDF + 8 * ks + t + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = tf32(B[(8 * ks + t) * LDF + 8 * nt + g]);
            const uint32_t b1 = tf32(B[(8 * ks + t + 4) * LDF + 8 * nt + g]);
            mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
        }
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]);
    u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]);
    u.w = pack_bf16(x[6], x[7]);
    return u;
}
__device__ __forceinline__ void unpack8(uint4 u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// K-major operand descriptor, K step s (16 elements) of a tile whose atoms are `atom_bytes` apart.
__device__ __forceinline__ uint64_t dK(uint32_t base, uint32_t atom_bytes, int s) {
    return desc_sw128(base + (uint32_t)(s >> 2) * atom_bytes + (uint32_t)(s & 3) * 32u, 0, 1024);
}
// MN-major operand descriptor, K step s (16 rows) of a tile whose MN atoms are `atom_bytes` apart.
__device__ __forceinline__ uint64_t dMN(uint32_t base, uint32_t atom_bytes, int s) {
    return desc_sw128(base + (uint32_t)s * 2048u, atom_bytes, 1024);
}

template <bool GATE_HEAD>
__global__ void __launch_bounds__(256, 1) kda_fwd_tc_kernel(const FwdArgs a) {
    using Lay = TcLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    float *G = reinterpret_cast<float *>(sm + Lay::oG);
    float *L = reinterpret_cast<float *>(sm + Lay::oL);
    float *Tm = reinterpret_cast<float *>(sm + Lay::oT);
    float *Bs = reinterpret_cast<float *>(sm + Lay::oBeta);
    float *Eg = reinterpret_cast<float *>(sm + Lay::oEg);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::oBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::oTmemAddr);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, n = blockIdx.z;
    const int hk = h / a.group;

    int64_t bos;
    int len;
    if (!seq_bounds(a, n, bos, len)) return;
    const int nchunks = (len + kChunk - 1) / kChunk;

    const bf16 *q = static_cast<const bf16 *>(a.q);
    const bf16 *k = static_cast<const bf16 *>(a.k);
    const bf16 *v = static_cast<const bf16 *>(a.v);
    bf16 *o = static_cast<bf16 *>(a.o);
    const int64_t sq = (int64_t)a.H_k * 128;
    const int64_t sv = (int64_t)a.H_v * 128;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * 128;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }

    // State: warpgroup 0, thread d owns row d of S (fp32, d_v = 128 values).
    float S[128];
    if (tid < 128) {
        if (a.h0 != nullptr) {
            const float4 *h0 = reinterpret_cast<const float4 *>(a.h0 + (((int64_t)n * a.H_v + h) * 128 + tid) * 128);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float4 x = h0[j];
                S[4 * j] = x.x;
                S[4 * j + 1] = x.y;
                S[4 * j + 2] = x.z;
                S[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 128; ++j) S[j] = 0.f;
        }
    }
    // S in bf16, MN-major A operand: element (m = dv, k = d) at atom dv/64, row d.
    auto write_SB = [&]() {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = S[8 * c + e];
            *reinterpret_cast<uint4 *>(sm + Lay::oSB + (c >> 3) * 16384 + sw128(tid, c & 7)) = pack8(x);
        }
    };
    if (tid < 128) write_SB();

    auto stage = [&](int c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        for (int i = tid; i < 1024; i += 256) {
            const int r = i >> 4, c8 = i & 15;
            const bool ok = r < nvalid;
            const int64_t t = bos + row0 + r;
            const int64_t oq = ok ? t * sq + (int64_t)hk * 128 + c8 * 8 : 0;
            const int64_t ov = ok ? t * sv + (int64_t)h * 128 + c8 * 8 : 0;
            cp_async_16(sm + Lay::oRQ + r * 256 + c8 * 16, q + oq, ok ? 16 : 0);
            cp_async_16(sm + Lay::oRK + r * 256 + c8 * 16, k + oq, ok ? 16 : 0);
            cp_async_16(sm + Lay::oRV + (c8 >> 3) * 8192 + sw128(r, c8 & 7), v + ov, ok ? 16 : 0);
        }
        if constexpr (!GATE_HEAD) {
            for (int i = tid; i < 2048; i += 256) {
                const int r = i >> 5, c4 = i & 31;
                const bool ok = r < nvalid;
                const int64_t og = ok ? (bos + row0 + r) * sg + (int64_t)h * 128 + c4 * 4 : 0;
                cp_async_16(sm + Lay::oG + r * 512 + c4 * 16, a.g + og, ok ? 16 : 0);
            }
        }
        cp_async_commit();
        if (tid < 64) {
            Bs[tid] = tid < nvalid ? a.beta[(bos + row0 + tid) * a.H_v + h] : 0.f;
        } else if (GATE_HEAD && tid < 128) {
            const int r = tid - 64;
            G[r] = r < nvalid ? a.g[(bos + row0 + r) * sg + h] : 0.f;
        }
    };

    if (nchunks > 0) stage(0);
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter
    bool failed = false;

    for (int c = 0; c < nchunks && !failed; ++c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        const uint32_t par = (uint32_t)(c & 1);
        cp_async_wait_all();
        __syncthreads();

        // ---- gate pass: cumulative log2 gate, then the decayed operands --------------------
        if constexpr (!GATE_HEAD) {
            if (tid < 128) {
                float acc = 0.f;
#pragma unroll 8
                for (int r = 0; r < 64; ++r) {
                    acc += G[r * 128 + tid] * kLog2e;
                    G[r * 128 + tid] = acc;
                }
                Eg[tid] = exp2f(acc);
            }
        } else {
            if (tid < 64) {
                float acc = 0.f;
                for (int s = 0; s <= tid; ++s) acc += G[s] * kLog2e;
                G[64 + tid] = acc;
            }
            __syncthreads();
            if (tid < 128) Eg[tid] = exp2f(G[64 + 63]);
        }
        __syncthreads();
        for (int i = tid; i < 1024; i += 256) {
            const int r = i >> 4, c8 = i & 15;
            float gm[8], kv[8], qv[8], eg[8];
            if constexpr (!GATE_HEAD) {
                const float4 g0 = *reinterpret_cast<const float4 *>(G + r * 128 + c8 * 8);
                const float4 g1 = *reinterpret_cast<const float4 *>(G + r * 128 + c8 * 8 + 4);
                gm[0] = g0.x; gm[1] = g0.y; gm[2] = g0.z; gm[3] = g0.w;
                gm[4] = g1.x; gm[5] = g1.y; gm[6] = g1.z; gm[7] = g1.w;
            } else {
                const float gr = G[64 + r];
#pragma unroll
                for (int e = 0; e < 8; ++e) gm[e] = gr;
            }
            unpack8(*reinterpret_cast<const uint4 *>(sm + Lay::oRK + r * 256 + c8 * 16), kv);
            unpack8(*reinterpret_cast<const uint4 *>(sm + Lay::oRQ + r * 256 + c8 * 16), qv);
            const float4 e0 = *reinterpret_cast<const float4 *>(Eg + c8 * 8);
            const float4 e1 = *reinterpret_cast<const float4 *>(Eg + c8 * 8 + 4);
            eg[0] = e0.x; eg[1] = e0.y; eg[2] = e0.z; eg[3] = e0.w;
            eg[4] = e1.x; eg[5] = e1.y; eg[6] = e1.z; eg[7] = e1.w;
            float kp[8], km[8], qp[8], kb[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float ep = exp2f(gm[e]), em = exp2f(-gm[e]);
                kp[e] = kv[e] * ep;
                km[e] = kv[e] * em;
                qp[e] = a.scale * qv[e] * ep;
                kb[e] = km[e] * eg[e];
            }
            const uint32_t sw = sw128(r, c8 & 7);
            const int atom = c8 >> 3;
            *reinterpret_cast<uint4 *>(sm + Lay::oGA + atom * 16384 + sw) = pack8(kp);
            *reinterpret_cast<uint4 *>(sm + Lay::oGA + atom * 16384 + 8192 + sw) = pack8(qp);
            *reinterpret_cast<uint4 *>(sm + Lay::oKM + atom * 8192 + sw) = pack8(km);
            *reinterpret_cast<uint4 *>(sm + Lay::oKB + atom * 8192 + sw) = pack8(kb);
        }
        fence_proxy_async();
        __syncthreads();

        // ---- Gram: D_G = [Kp; Qp] Km^T ------------------------------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, false, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + tG, dK(sbase + Lay::oGA, 16384, s), dK(sbase + Lay::oKM, 8192, s), id, s > 0);
            commit(&bars[BAR_G]);
        }
        failed = !mbar_wait(&bars[BAR_G], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid < 128) {
            // rows 0-63 of D_G: L = diag(beta) strict_lower(M), fp32; rows 64-127: Aqk (lower) in bf16
            const int r = tid & 63;
            const float br = Bs[r];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t16[16];
                tmem_ld16(tmem + lane_off + tG + 16 * j, t16);
                tmem_ld_wait();
                if (tid < 64) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int col = 16 * j + e;
                        float4 x;
                        x.x = col < r ? br * t16[e] : 0.f;
                        x.y = col + 1 < r ? br * t16[e + 1] : 0.f;
                        x.z = col + 2 < r ? br * t16[e + 2] : 0.f;
                        x.w = col + 3 < r ? br * t16[e + 3] : 0.f;
                        *reinterpret_cast<float4 *>(L + r * LDF + col) = x;
                    }
                } else {
                    float x0[8], x1[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x0[e] = (16 * j + e) <= r ? t16[e] : 0.f;
                        x1[e] = (16 * j + 8 + e) <= r ? t16[8 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sm + Lay::oAQ + sw128(r, 2 * j)) = pack8(x0);
                    *reinterpret_cast<uint4 *>(sm + Lay::oAQ + sw128(r, 2 * j + 1)) = pack8(x1);
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();

        // ---- solve: T = (I + L)^-1 -----------------------------------------------------------
        if (warp < 4 && lane < 16) {
            const int b0 = 16 * warp, j = lane;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float s = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) s -= L[(b0 + r) * LDF + b0 + m] * x[m];
                x[r] = s;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tm[(b0 + r) * LDF + b0 + j] = x[r];
        }
        __syncthreads();
        for (int d = 1; d <= 3; ++d) {
            if (warp < 4 - d) {
                const int bi = d + warp, bj = bi - d;
                const int g8 = lane >> 2, t4 = lane & 3;
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                for (int kb = bj; kb < bi; ++kb)
                    mm16_tf32(acc, L + (16 * bi) * LDF + 16 * kb, Tm + (16 * kb) * LDF + 16 * bj, lane);
                // park P in the unused upper block (bj, bi)
                float *P = Tm + (16 * bj) * LDF + 16 * bi;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    P[g8 * LDF + 8 * nt + 2 * t4] = acc[nt][0];
                    P[g8 * LDF + 8 * nt + 2 * t4 + 1] = acc[nt][1];
                    P[(g8 + 8) * LDF + 8 * nt + 2 * t4] = acc[nt][2];
                    P[(g8 + 8) * LDF + 8 * nt + 2 * t4 + 1] = acc[nt][3];
                }
                __syncwarp();
                float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                mm16_tf32(acc2, Tm + (16 * bi) * LDF + 16 * bi, P, lane);
                float *Tij = Tm + (16 * bi) * LDF + 16 * bj;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    Tij[g8 * LDF + 8 * nt + 2 * t4] = -acc2[nt][0];
                    Tij[g8 * LDF + 8 * nt + 2 * t4 + 1] = -acc2[nt][1];
                    Tij[(g8 + 8) * LDF + 8 * nt + 2 * t4] = -acc2[nt][2];
                    Tij[(g8 + 8) * LDF + 8 * nt + 2 * t4 + 1] = -acc2[nt][3];
                }
            }
            __syncthreads();
        }
        // T_beta = T diag(beta) (lower triangle) -> bf16, K-major B operand [token][token']
        for (int i = tid; i < 512; i += 256) {
            const int r = i >> 3, c8 = i & 7;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int col = 8 * c8 + e;
                x[e] = col <= r ? Tm[r * LDF + col] * Bs[col] : 0.f;
            }
            *reinterpret_cast<uint4 *>(sm + Lay::oTB + sw128(r, c8)) = pack8(x);
        }
        fence_proxy_async();
        __syncthreads();

        // ---- WY factors: D_W = Kp^T T_beta^T, D_V = V^T T_beta^T ------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t b = dK(sbase + Lay::oTB, 8192, s);
                mma(tmem + tW, dMN(sbase + Lay::oGA, 16384, s), b, id, s > 0);
                mma(tmem + tV, dMN(sbase + Lay::oRV, 8192, s), b, id, s > 0);
            }
            commit(&bars[BAR_W]);
        }
        failed = !mbar_wait(&bars[BAR_W], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid < 128) {
            // W^T row d (64 tokens) -> bf16, MN-major B operand: row k = d, columns = tokens
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t16[16];
                tmem_ld16(tmem + lane_off + tW + 16 * j, t16);
                tmem_ld_wait();
                float x0[8], x1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x0[e] = t16[e];
                    x1[e] = t16[8 + e];
                }
                *reinterpret_cast<uint4 *>(sm + Lay::oWB + sw128(tid, 2 * j)) = pack8(x0);
                *reinterpret_cast<uint4 *>(sm + Lay::oWB + sw128(tid, 2 * j + 1)) = pack8(x1);
            }
        }
        fence_before_sync();
        fence_proxy_async();
        __syncthreads();
        // every raw tile is consumed: stage the next chunk behind the serial step
        if (c + 1 < nchunks) stage(c + 1);

        // ---- serial step, part 1: Vt^T = U^T - S^T W^T;  O^T = S^T Qp^T -----------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idv = idesc_bf16(128, 64, true, true, true);
            const uint32_t ido = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t sa = dMN(sbase + Lay::oSB, 16384, s);
                mma(tmem + tV, sa, dMN(sbase + Lay::oWB, 16384, s), idv, 1);
                mma(tmem + tO, sa, dK(sbase + Lay::oGA + 8192, 16384, s), ido, s > 0);
            }
            commit(&bars[BAR_V]);
        }
        failed = !mbar_wait(&bars[BAR_V], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid < 128) {
            // Vt^T row dv (64 tokens) -> bf16, K-major [dv][token]
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t16[16];
                tmem_ld16(tmem + lane_off + tV + 16 * j, t16);
                tmem_ld_wait();
                float x0[8], x1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x0[e] = t16[e];
                    x1[e] = t16[8 + e];
                }
                *reinterpret_cast<uint4 *>(sm + Lay::oVB + sw128(tid, 2 * j)) = pack8(x0);
                *reinterpret_cast<uint4 *>(sm + Lay::oVB + sw128(tid, 2 * j + 1)) = pack8(x1);
            }
        }
        fence_before_sync();
        fence_proxy_async();
        __syncthreads();

        // ---- serial step, part 2: O^T += Vt^T Aqk^T;  D_S = Kbar^T Vt -----------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t ido = idesc_bf16(128, 64, false, false, false);
            const uint32_t ids = idesc_bf16(128, 128, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t vb = dK(sbase + Lay::oVB, 16384, s);
                mma(tmem + tO, vb, dK(sbase + Lay::oAQ, 8192, s), ido, 1);
                mma(tmem + tS, dMN(sbase + Lay::oKB, 8192, s), vb, ids, s > 0);
            }
            commit(&bars[BAR_S]);
        }
        failed = !mbar_wait(&bars[BAR_S], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid < 128) {
            // S <- Diag(e^gamma_n) S + D_S, then S in bf16 for the next chunk
            const float e = Eg[tid];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float t16[16];
                tmem_ld16(tmem + lane_off + tS + 16 * j, t16);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) S[16 * j + x] = fmaf(e, S[16 * j + x], t16[x]);
            }
            write_SB();
        } else {
            // O^T row dv (64 tokens) -> O staging [token][dv]
            const int dv = tid - 128;
            bf16 *OS = reinterpret_cast<bf16 *>(sm + Lay::oOS);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t16[16];
                tmem_ld16(tmem + lane_off + tO + 16 * j, t16);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) OS[(16 * j + x) * 128 + dv] = __float2bfloat16_rn(t16[x]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            for (int i = dv; i < 1024; i += 128) {
                const int r = i >> 4, c8 = i & 15;
                if (r < nvalid)
                    *reinterpret_cast<uint4 *>(o + (bos + row0 + r) * sv + (int64_t)h * 128 + c8 * 8) =
                        *reinterpret_cast<const uint4 *>(sm + Lay::oOS + r * 256 + c8 * 16);
            }
        }
        fence_before_sync();
        fence_proxy_async();
        __syncthreads();
    }

    if (failed) {
        if (tid == 0) {
            atomicOr(a.err, kDeviceErrTimeout);
            // wait (bounded) for every MMA this CTA issued before freeing TMEM
            fence_after_sync();
            commit(&bars[BAR_Z]);
            mbar_wait(&bars[BAR_Z], 0, kWaitCycles);
        }
        cp_async_wait_all();
    } else if (a.ht != nullptr && tid < 128) {
        float4 *ht = reinterpret_cast<float4 *>(a.ht + (((int64_t)n * a.H_v + h) * 128 + tid) * 128);
#pragma unroll
        for (int j = 0; j < 32; ++j) ht[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool GATE_HEAD>
cudaError_t launch_tc(const FwdArgs &a, cudaStream_t stream) {
    constexpr int kSmem = TcLayout::kBytes;
    auto kern = kda_fwd_tc_kernel<GATE_HEAD>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    const dim3 grid(1, a.H_v, a.N);
    kern<<<grid, 256, kSmem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t stream) {
    return a.gate_per_head ? launch_tc<true>(a, stream) : launch_tc<false>(a, stream);
}

}  // namespace kda
