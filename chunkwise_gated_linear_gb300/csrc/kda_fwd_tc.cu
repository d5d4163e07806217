// Chunkwise KDA forward for d_k = d_v = 128, bf16 operands, on the 5th-generation tensor
// cores (tcgen05) with accumulators in tensor memory (TMEM).
//
// One CTA of 256 threads runs one (sequence, value head) unit through all its chunks.
// Every product is arranged so that the tensor core's M dimension is 128 (the d_k or d_v
// axis, or the stacked [Kp; Qp] rows), so each MMA runs at full width:
//
//   Gram      D_G [128 x 64]  = [Qp; Kp] Km^T          rows 0-63: Aqk, rows 64-127: M
//   WY        D_W [128 x 64]  = Kp^T T_beta^T           (W^T, d_k x tokens)
//             D_U [128 x 64]  = V^T  T_beta^T           (U^T, d_v x tokens)
//   serial    D_X [128 x 128] = S^T [W^T | Qp^T]         (one pass over S)
//             Vt^T = U^T - D_X[:, :64]                   (in registers, then bf16)
//             D_X[:, 64:] += Vt^T Aqk^T                  (O^T, d_v x tokens)
//             D_S  = Kbar^T Vt                           (the chunk's state increment)
//
// and S <- Diag(e^gamma_n) S + D_S is applied in fp32 registers by the 128 threads of
// warpgroup 0, thread d owning row d of S (d_k x d_v) across the whole sequence. Per chunk
// ("RNN的复兴04:线性注意力并行计算DPLR", §5.3.5; "TileLang 实战：KDA 从零到一–Kimi Delta
// Attention", §3.3): the cumulative log2 gate and the decayed operands (gate pass), the
// Gram matrix, the UT-transform inverse T = (I + diag(beta) M)^-1 (16x16 diagonal blocks by
// forward substitution, then the off-diagonal blocks column by column with tf32 mma.sync,
// one warp per 8 columns), T_beta = T diag(beta), the WY
// factors, and the serial step. All operands live in shared memory in the 128-byte-swizzled
// layouts the tensor core reads; nothing but q, k, v, g, beta, h0 (in) and o, ht (out)
// touches HBM.
//
// Every mbarrier wait is bounded (about one second); on a timeout the CTA raises
// KDA_DEVICE_ERR_TIMEOUT, waits (bounded) for its issued MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "tc5.cuh"

namespace kda {

namespace {

using bf16 = __nv_bfloat16;
using namespace tc5;

// Shared-memory plan (byte offsets from a 1024-byte aligned base). Tiles named [d][tok]
// hold one row per d_k channel and 64 tokens per 128-byte row (one swizzle atom).
struct TcLayout {
    static constexpr int oRQ = 0;       // raw Q [64 tok][128] bf16 row-major
    static constexpr int oRK = 16384;   // raw K
    static constexpr int oRV = 32768;   // raw V, [2 atoms (d_v)][64 tok rows][128 B] (MN-major A of U^T)
    static constexpr int oWT = 49152;   // W^T [d][tok]    } one N = 128 B operand (W^T | Qp^T)
    static constexpr int oQP = 65536;   // Qp^T [d][tok]   } and one M = 128 A operand (Qp | Kp)
    static constexpr int oKP = 81920;   // Kp^T [d][tok]   }
    static constexpr int oKM = 98304;   // Km^T [d][tok]; then Aqk [tok][tok'] (8 KB) + T_beta (8 KB);
    static constexpr int oAQ = oKM;     //   then the O staging tile [64 tok][128] bf16
    static constexpr int oTB = oKM + 8192;
    static constexpr int oOS = oKM;
    static constexpr int oKB = 114688;  // Kbar^T [d][tok]
    static constexpr int oSB = 131072;  // S in bf16: [2 atoms (d_v)][128 rows (d_k)][128 B]
    static constexpr int oVB = 163840;  // Vt^T in bf16: [128 rows (d_v)][128 B (tok)]
    static constexpr int oG = 180224;   // raw G fp32 [64][128]; then L and T fp32 [64][68]
    static constexpr int oL = oG;
    static constexpr int oT = oG + 17408;
    static constexpr int oBeta = oG + 34816;  // [64] fp32 (raw per-head gates follow at +256)
    static constexpr int oGh = oBeta + 256;   // [64] fp32 per-head gates
    static constexpr int oTot = oGh + 256;    // [4][128] fp32 partial gate sums
    static constexpr int oEg = oTot + 2048;   // [128] fp32 e^gamma_n
    static constexpr int oBar = oEg + 512;
    static constexpr int oTmemAddr = oBar + 64;
    static constexpr int kBytes = oTmemAddr + 16 + 1024;  // + slack to align the base
};
constexpr int LDF = 68;  // fp32 row stride of L and T

// TMEM columns: Gram, W^T, U^T, [S^T W^T | O^T], state increment
constexpr uint32_t tG = 0, tW = 64, tU = 128, tX = 192, tO = 256, tS = 320;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitCycles = 1ll << 31;  // about one second

enum { BAR_G = 0, BAR_W, BAR_V, BAR_S, BAR_Z, BAR_L, kNumBars };

// Tensor maps of the per-chunk tiles (TMA): q, k [tokens][H_k*128] bf16 (box 128 x 64),
// v [tokens][H_v*128] bf16 (box 64 x 64, 128-byte swizzle), g [tokens][H_v*128] fp32 (box 128 x 64).
struct TcMaps {
    CUtensorMap q, k, v, g;
};

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
// acc (16x8) += A (16x16, stride lda) * B (16x8, stride ldb); fp32 in smem, tf32 products.
__device__ __forceinline__ void mm16x8_tf32(float (&acc)[4], const float *A, int lda, const float *B, int ldb,
                                            int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a0 = tf32(A[g * lda + 8 * ks + t]);
        const uint32_t a1 = tf32(A[(g + 8) * lda + 8 * ks + t]);
        const uint32_t a2 = tf32(A[g * lda + 8 * ks + t + 4]);
        const uint32_t a3 = tf32(A[(g + 8) * lda + 8 * ks + t + 4]);
        const uint32_t b0 = tf32(B[(8 * ks + t) * ldb + g]);
        const uint32_t b1 = tf32(B[(8 * ks + t + 4) * ldb + g]);
        mma_tf32(acc, a0, a1, a2, a3, b0, b1);
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

// K-major operand descriptor, K step s (16 elements) of a tile whose K atoms are `atom_bytes` apart.
__device__ __forceinline__ uint64_t dK(uint32_t base, uint32_t atom_bytes, int s) {
    return desc_sw128(base + (uint32_t)(s >> 2) * atom_bytes + (uint32_t)(s & 3) * 32u, 0, 1024);
}
// MN-major operand descriptor, K step s (16 rows) of a tile whose MN atoms are `atom_bytes` apart.
__device__ __forceinline__ uint64_t dMN(uint32_t base, uint32_t atom_bytes, int s) {
    return desc_sw128(base + (uint32_t)s * 2048u, atom_bytes, 1024);
}

// TMEM (this warp's 32 lanes, columns [col, col+32)) -> 32 floats.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
    }
}

template <bool GATE_HEAD>
__global__ void __launch_bounds__(256, 1) kda_fwd_tc_kernel(const FwdArgs a, const __grid_constant__ TcMaps maps) {
    using Lay = TcLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const bf16 *RQ = reinterpret_cast<const bf16 *>(sm + Lay::oRQ);
    const bf16 *RK = reinterpret_cast<const bf16 *>(sm + Lay::oRK);
    float *G = reinterpret_cast<float *>(sm + Lay::oG);
    float *L = reinterpret_cast<float *>(sm + Lay::oL);
    float *Tm = reinterpret_cast<float *>(sm + Lay::oT);
    float *Bs = reinterpret_cast<float *>(sm + Lay::oBeta);
    float *Gh = reinterpret_cast<float *>(sm + Lay::oGh);
    float *Tot = reinterpret_cast<float *>(sm + Lay::oTot);
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

    bf16 *o = static_cast<bf16 *>(a.o);
    const int64_t sv = (int64_t)a.H_v * 128;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * 128;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
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
    // S in bf16, MN-major A operand of S^T: element (m = dv, k = d) at atom dv/64, row d.
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

    // Stage chunk c: Q, K, V and G by TMA (thread 0), beta and per-head gates by cp.async.
    constexpr uint32_t kTileBytes = 3 * 16384 + (GATE_HEAD ? 0 : 32768);
    auto stage = [&](int c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        if (tid == 0) {
            const int y = (int)(bos + row0);
            mbar_arrive_expect_tx(&bars[BAR_L], kTileBytes);
            tma_load_2d(sm + Lay::oRQ, &maps.q, &bars[BAR_L], hk * 128, y);
            tma_load_2d(sm + Lay::oRK, &maps.k, &bars[BAR_L], hk * 128, y);
            tma_load_2d(sm + Lay::oRV, &maps.v, &bars[BAR_L], h * 128, y);
            tma_load_2d(sm + Lay::oRV + 8192, &maps.v, &bars[BAR_L], h * 128 + 64, y);
            if constexpr (!GATE_HEAD) tma_load_2d(sm + Lay::oG, &maps.g, &bars[BAR_L], h * 128, y);
        }
        if (tid < 64) {
            const bool ok = tid < nvalid;
            const int64_t ob = ok ? (bos + row0 + tid) * a.H_v + h : 0;
            cp_async_4(Bs + tid, a.beta + ob, ok ? 4 : 0);
        } else if (GATE_HEAD && tid < 128) {
            const int r = tid - 64;
            const bool ok = r < nvalid;
            const int64_t og = ok ? (bos + row0 + r) * sg + h : 0;
            cp_async_4(Gh + r, a.g + og, ok ? 4 : 0);
        }
        cp_async_commit();
    };

    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (nchunks > 0) stage(0);
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter
    const uint32_t half = (uint32_t)(warp >> 2) * 32u;              // column half of a 64-wide readback
    bool failed = false;

    for (int c = 0; c < nchunks && !failed; ++c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        const uint32_t par = (uint32_t)(c & 1);
        cp_async_wait_all();
        failed = !mbar_wait(&bars[BAR_L], par, kWaitCycles);
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (nvalid < kChunk) {
            // the boxes read on past the sequence end (the next sequence, or zeros past the
            // tensor): those rows must be zero in every operand
            const int nz = kChunk - nvalid;
            for (int i = tid; i < nz * 16; i += 256) {
                const int r = nvalid + (i >> 4), c16 = i & 15;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sm + Lay::oRQ + r * 256 + c16 * 16) = z;
                *reinterpret_cast<uint4 *>(sm + Lay::oRK + r * 256 + c16 * 16) = z;
                *reinterpret_cast<uint4 *>(sm + Lay::oRV + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16) = z;
                if constexpr (!GATE_HEAD) {
                    *reinterpret_cast<uint4 *>(sm + Lay::oG + r * 512 + c16 * 32) = z;
                    *reinterpret_cast<uint4 *>(sm + Lay::oG + r * 512 + c16 * 32 + 16) = z;
                }
            }
            fence_proxy_async();
            __syncthreads();
        }

        // ---- gate pass ---------------------------------------------------------------------
        // warp w: rows 16 (w >> 1) .. +15, channels c0 = 64 (w & 1) + lane and c1 = c0 + 32.
        {
            const int qr = warp >> 1;
            const int c0 = 64 * (warp & 1) + lane, c1 = c0 + 32;
            float gl0[16], gl1[16];
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = 16 * qr + e;
                if constexpr (!GATE_HEAD) {
                    acc0 += G[r * 128 + c0] * kLog2e;
                    acc1 += G[r * 128 + c1] * kLog2e;
                } else {
                    const float gr = Gh[r] * kLog2e;
                    acc0 += gr;
                    acc1 += gr;
                }
                gl0[e] = acc0;
                gl1[e] = acc1;
            }
            Tot[qr * 128 + c0] = acc0;
            Tot[qr * 128 + c1] = acc1;
            __syncthreads();
            float off0 = 0.f, off1 = 0.f, gn0 = 0.f, gn1 = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const float t0 = Tot[qq * 128 + c0], t1 = Tot[qq * 128 + c1];
                if (qq < qr) {
                    off0 += t0;
                    off1 += t1;
                }
                gn0 += t0;
                gn1 += t1;
            }
            const float eg0 = ex2(gn0), eg1 = ex2(gn1);
            if (qr == 0) {
                Eg[c0] = eg0;
                Eg[c1] = eg1;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tc = 2 * qr + j;  // 16-byte chunk (8 tokens) within a 64-token row
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int cc = ch ? c1 : c0;
                    const float off = ch ? off1 : off0, eg = ch ? eg1 : eg0;
                    float kp[8], km[8], qp[8], kb[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int r = 16 * qr + 8 * j + e;
                        const float gm = off + (ch ? gl1[8 * j + e] : gl0[8 * j + e]);
                        const float ep = ex2(gm), em = ex2(-gm);
                        const float kv = __bfloat162float(RK[r * 128 + cc]);
                        const float qv = __bfloat162float(RQ[r * 128 + cc]);
                        kp[e] = kv * ep;
                        km[e] = kv * em;
                        qp[e] = a.scale * qv * ep;
                        kb[e] = km[e] * eg;
                    }
                    const uint32_t sw = sw128(cc, tc);
                    *reinterpret_cast<uint4 *>(sm + Lay::oKP + sw) = pack8(kp);
                    *reinterpret_cast<uint4 *>(sm + Lay::oQP + sw) = pack8(qp);
                    *reinterpret_cast<uint4 *>(sm + Lay::oKM + sw) = pack8(km);
                    *reinterpret_cast<uint4 *>(sm + Lay::oKB + sw) = pack8(kb);
                }
            }
        }
        fence_proxy_async();
        __syncthreads();

        // ---- Gram: D_G = [Qp; Kp] Km^T  (rows 0-63: Aqk, rows 64-127: M) --------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, true, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + tG, dMN(sbase + Lay::oQP, 16384, s), dMN(sbase + Lay::oKM, 16384, s), id, s > 0);
            commit(&bars[BAR_G]);
        }
        failed = !mbar_wait(&bars[BAR_G], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        {
            // each warpgroup reads 32 of the 64 columns of its lane's row
            const int row = tid & 127;
            float x[32];
            tmem_ld32(tmem + lane_off + tG + half, x);
            if (row < 64) {
                // Aqk (lower, diagonal included) -> bf16 [tok][tok'], K-major B operand
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int col = (int)half + 8 * c8 + e;
                        y[e] = col <= row ? x[8 * c8 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sm + Lay::oAQ + sw128(row, (int)(half >> 3) + c8)) = pack8(y);
                }
            } else {
                // L = diag(beta) strict_lower(M), fp32
                const int r = row - 64;
                const float br = Bs[r];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int col = (int)half + e;
                    float4 y;
                    y.x = col < r ? br * x[e] : 0.f;
                    y.y = col + 1 < r ? br * x[e + 1] : 0.f;
                    y.z = col + 2 < r ? br * x[e + 2] : 0.f;
                    y.w = col + 3 < r ? br * x[e + 3] : 0.f;
                    *reinterpret_cast<float4 *>(L + r * LDF + col) = y;
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();

        // ---- solve: T = (I + L)^-1 -----------------------------------------------------------
        // D = blockdiag of the 16x16 diagonal inverses (forward substitution, one column per lane)
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
        // Off-diagonal blocks column by column: warp w owns the 8 columns col0..col0+7 of T
        // (column block j = w / 2). T_jj = D_j, and for i > j
        //   T_ij = -D_i sum_{k=j}^{i-1} L_ik T_kj
        // (tf32 mma.sync, fp32 accumulation). The warp then writes its columns of
        // T_beta = T diag(beta) (lower triangle) in bf16. No CTA-wide barrier is needed:
        // each warp only reads L, the diagonal blocks and its own columns.
        {
            const int j = warp >> 1, col0 = 16 * j + 8 * (warp & 1);
            const int g8 = lane >> 2, t4 = lane & 3;
            float *P = reinterpret_cast<float *>(sm + Lay::oRQ) + warp * 128;  // 16x8 scratch
            for (int i = j + 1; i < 4; ++i) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int kb = j; kb < i; ++kb)
                    mm16x8_tf32(acc, L + (16 * i) * LDF + 16 * kb, LDF, Tm + (16 * kb) * LDF + col0, LDF, lane);
                P[g8 * 8 + 2 * t4] = acc[0];
                P[g8 * 8 + 2 * t4 + 1] = acc[1];
                P[(g8 + 8) * 8 + 2 * t4] = acc[2];
                P[(g8 + 8) * 8 + 2 * t4 + 1] = acc[3];
                __syncwarp();
                float acc2[4] = {0.f, 0.f, 0.f, 0.f};
                mm16x8_tf32(acc2, Tm + (16 * i) * LDF + 16 * i, LDF, P, 8, lane);
                float *Tij = Tm + (16 * i) * LDF + col0;
                Tij[g8 * LDF + 2 * t4] = -acc2[0];
                Tij[g8 * LDF + 2 * t4 + 1] = -acc2[1];
                Tij[(g8 + 8) * LDF + 2 * t4] = -acc2[2];
                Tij[(g8 + 8) * LDF + 2 * t4 + 1] = -acc2[3];
                __syncwarp();
            }
            const float4 b0 = *reinterpret_cast<const float4 *>(Bs + col0);
            const float4 b1 = *reinterpret_cast<const float4 *>(Bs + col0 + 4);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                float x[8];
                if (r < 16 * j) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.f;
                } else {
                    const float4 t0 = *reinterpret_cast<const float4 *>(Tm + r * LDF + col0);
                    const float4 t1 = *reinterpret_cast<const float4 *>(Tm + r * LDF + col0 + 4);
                    const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = (col0 + e) <= r ? tv[e] * bv[e] : 0.f;
                }
                *reinterpret_cast<uint4 *>(sm + Lay::oTB + sw128(r, col0 >> 3)) = pack8(x);
            }
        }
        fence_proxy_async();
        __syncthreads();

        // ---- WY factors: D_W = Kp^T T_beta^T, D_U = V^T T_beta^T ------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idw = idesc_bf16(128, 64, false, false, false);
            const uint32_t idu = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t b = dK(sbase + Lay::oTB, 8192, s);
                mma(tmem + tW, dK(sbase + Lay::oKP, 16384, s), b, idw, s > 0);
                mma(tmem + tU, dMN(sbase + Lay::oRV, 8192, s), b, idu, s > 0);
            }
            commit(&bars[BAR_W]);
        }
        failed = !mbar_wait(&bars[BAR_W], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        {
            // W^T row d -> bf16 [d][tok] (MN-major B); each warpgroup writes 32 of the 64 tokens
            const int d = tid & 127;
            float x[32];
            tmem_ld32(tmem + lane_off + tW + half, x);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = x[8 * c8 + e];
                *reinterpret_cast<uint4 *>(sm + Lay::oWT + sw128(d, (int)(half >> 3) + c8)) = pack8(y);
            }
        }
        fence_before_sync();
        fence_proxy_async();
        __syncthreads();
        // every raw tile is consumed: stage the next chunk behind the serial step
        if (c + 1 < nchunks) stage(c + 1);

        // ---- serial step, part 1: D_X = S^T [W^T | Qp^T] -----------------------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 128, true, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + tX, dMN(sbase + Lay::oSB, 16384, s), dMN(sbase + Lay::oWT, 16384, s), id, s > 0);
            commit(&bars[BAR_V]);
        }
        failed = !mbar_wait(&bars[BAR_V], par, kWaitCycles);
        fence_after_sync();
        if (__syncthreads_or(failed)) { failed = true; break; }
        {
            // Vt^T = U^T - S^T W^T, row dv -> bf16 [dv][tok]; each warpgroup does 32 tokens
            const int dv = tid & 127;
            float u[32], p[32];
            tmem_ld32(tmem + lane_off + tU + half, u);
            tmem_ld32(tmem + lane_off + tX + half, p);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = u[8 * c8 + e] - p[8 * c8 + e];
                *reinterpret_cast<uint4 *>(sm + Lay::oVB + sw128(dv, (int)(half >> 3) + c8)) = pack8(y);
            }
        }
        fence_before_sync();
        fence_proxy_async();
        __syncthreads();

        // ---- serial step, part 2: O^T += Vt^T Aqk^T;  D_S = Kbar^T Vt -----------------------
        if (tid == 0) {
            fence_after_sync();
            const uint32_t ido = idesc_bf16(128, 64, false, false, false);
            const uint32_t ids = idesc_bf16(128, 128, false, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t vb = dK(sbase + Lay::oVB, 16384, s);
                mma(tmem + tO, vb, dK(sbase + Lay::oAQ, 8192, s), ido, 1);
                mma(tmem + tS, dK(sbase + Lay::oKB, 16384, s), vb, ids, s > 0);
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
            for (int j = 0; j < 2; ++j) {
                float t0[16], t1[16], t2[16], t3[16];
                tmem_ld16(tmem + lane_off + tS + 64 * j, t0);
                tmem_ld16(tmem + lane_off + tS + 64 * j + 16, t1);
                tmem_ld16(tmem + lane_off + tS + 64 * j + 32, t2);
                tmem_ld16(tmem + lane_off + tS + 64 * j + 48, t3);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    S[64 * j + x] = fmaf(e, S[64 * j + x], t0[x]);
                    S[64 * j + 16 + x] = fmaf(e, S[64 * j + 16 + x], t1[x]);
                    S[64 * j + 32 + x] = fmaf(e, S[64 * j + 32 + x], t2[x]);
                    S[64 * j + 48 + x] = fmaf(e, S[64 * j + 48 + x], t3[x]);
                }
            }
            write_SB();
        } else {
            // O^T row dv (64 tokens) -> O staging [token][dv] -> global, valid rows only
            const int dv = tid - 128;
            bf16 *OS = reinterpret_cast<bf16 *>(sm + Lay::oOS);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float t32[32];
                tmem_ld32(tmem + lane_off + tO + 32 * j, t32);
#pragma unroll
                for (int x = 0; x < 32; ++x) OS[(32 * j + x) * 128 + dv] = __float2bfloat16_rn(t32[x]);
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over a [rows][inner] row-major tensor with a (box0 x 64-row) box.
bool encode_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t rows,
                uint64_t elem_bytes, uint32_t box0, CUtensorMapSwizzle sw) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box0, 64};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool GATE_HEAD>
cudaError_t launch_tc(const FwdArgs &a, cudaStream_t stream) {
    constexpr int kSmem = TcLayout::kBytes;
    auto kern = kda_fwd_tc_kernel<GATE_HEAD>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    TcMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const uint64_t rows = a.cu_seqlens ? (uint64_t)a.T : (uint64_t)a.N * (uint64_t)a.T;
    if (rows > 0) {
        bool ok = encode_map(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, (uint64_t)a.H_k * 128, rows, 2, 128,
                             CU_TENSOR_MAP_SWIZZLE_NONE) &&
                  encode_map(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k, (uint64_t)a.H_k * 128, rows, 2, 128,
                             CU_TENSOR_MAP_SWIZZLE_NONE) &&
                  encode_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.v, (uint64_t)a.H_v * 128, rows, 2, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B);
        if (ok && !GATE_HEAD)
            ok = encode_map(&maps.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.g, (uint64_t)a.H_v * 128, rows, 4, 128,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!ok) return cudaErrorInvalidValue;
    }
    const dim3 grid(1, a.H_v, a.N);
    kern<<<grid, 256, kSmem, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t stream) {
    return a.gate_per_head ? launch_tc<true>(a, stream) : launch_tc<false>(a, stream);
}

}  // namespace kda
