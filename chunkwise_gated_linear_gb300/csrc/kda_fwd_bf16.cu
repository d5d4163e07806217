// Chunkwise KDA forward, bf16 operands with fp32 accumulation (tensor cores, mma.sync).
//
// One CTA runs one (sequence, value head, 64-wide slice of d_v) unit through all of its
// chunks. Per chunk of 64 tokens (the steps of "RNN的复兴04:线性注意力并行计算DPLR", §5.3.5,
// and "TileLang 实战：KDA 从零到一–Kimi Delta Attention", §3.3 and §4):
//
//   1. stage    Q, K [64 x d_k], V [64 x 64], G [64 x d_k] (fp32) and beta into shared
//               memory with 16-byte cp.async; rows past the end of the sequence are zero;
//   2. gate     gamma = chunk-local cumulative sum of the log gates (log2 domain), and the
//               decayed operands Qp = scale Q e^gamma, Kp = K e^gamma, Km = K e^-gamma,
//               Kbar = K e^(gamma_n - gamma), e^gamma_n (KDA page §1.2: the exponent
//               separates channel by channel);
//   3. Gram     M = Kp Km^T (strictly lower) and Aqk = Qp Km^T (lower, diagonal included),
//               masked by selection, never by multiplication ("TileLang 实战：KDA 从零到一
//               --标量衰减", §2.2);
//   4. solve    T = (I + diag(beta) M)^-1 from four 16x16 forward substitutions and the
//               block merges ("Gated DeltaNet", the 64x64 inverse from 16x16 blocks);
//               T_beta = T diag(beta);
//   5. WY       W = T_beta Kp [64 x d_k], U = T_beta V [64 x 64];
//   6. serial   per warp, its 16 rows of S^T (fp32, in registers across all chunks):
//               Vt^T = U^T - S^T W^T;  O^T = S^T Qp^T + Vt^T Aqk^T;
//               S^T <- S^T Diag(e^gamma_n) + Vt^T Kbar.
//
// Keeping S^T (rows = d_v, columns = d_k) as the accumulator lets each product of the
// serial step take the previous product's accumulator as its A operand directly, so the
// state never leaves the registers and the four warps never wait on one another inside
// the serial step. The next chunk's tiles are staged while the serial step runs.
#include "kda_common.cuh"

namespace kda {

namespace {

using bf16 = __nv_bfloat16;

template <int DK>
struct Bf16Layout {
    static constexpr int LDK = DK + 8;  // bf16 row stride of [64][DK] tiles
    static constexpr int LDV = 64 + 8;  // bf16 row stride of [64][64] tiles
    static constexpr int LDF = 64 + 4;  // fp32 row stride of [64][64] tiles
    static constexpr int kTileK = 64 * LDK * 2;
    static constexpr int kTileV = 64 * LDV * 2;
    static constexpr int kTileF = 64 * LDF * 4;
    static constexpr int oQraw = 0;
    static constexpr int oKraw = oQraw + kTileK;
    static constexpr int oVraw = oKraw + kTileK;
    static constexpr int oG = oVraw + kTileV;
    static constexpr int oBeta = oG + 64 * DK * 4;
    static constexpr int oQp = oBeta + 64 * 4;
    static constexpr int oKp = oQp + kTileK;
    static constexpr int oKm = oKp + kTileK;
    static constexpr int oKbar = oKm + kTileK;
    static constexpr int oW = oKbar + kTileK;
    static constexpr int oL = oW + kTileK;  // L (fp32), then U (fp32)
    static constexpr int oT = oL + kTileF;
    static constexpr int oTb = oT + kTileF;  // T_beta (bf16), then the O staging tile
    static constexpr int oA = oTb + kTileV;
    static constexpr int oEg = oA + kTileV;
    static constexpr int kBytes = oEg + DK * 4;
};

template <int DK, bool GATE_HEAD>
__global__ void __launch_bounds__(128, 1) kda_fwd_bf16_kernel(const FwdArgs a) {
    using Lay = Bf16Layout<DK>;
    constexpr int LDK = Lay::LDK, LDV = Lay::LDV, LDF = Lay::LDF;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *Qraw = reinterpret_cast<bf16 *>(smem + Lay::oQraw);
    bf16 *Kraw = reinterpret_cast<bf16 *>(smem + Lay::oKraw);
    bf16 *Vraw = reinterpret_cast<bf16 *>(smem + Lay::oVraw);
    float *G = reinterpret_cast<float *>(smem + Lay::oG);
    float *Bs = reinterpret_cast<float *>(smem + Lay::oBeta);
    bf16 *Qp = reinterpret_cast<bf16 *>(smem + Lay::oQp);
    bf16 *Kp = reinterpret_cast<bf16 *>(smem + Lay::oKp);
    bf16 *Km = reinterpret_cast<bf16 *>(smem + Lay::oKm);
    bf16 *Kbar = reinterpret_cast<bf16 *>(smem + Lay::oKbar);
    bf16 *Wb = reinterpret_cast<bf16 *>(smem + Lay::oW);
    float *Lf = reinterpret_cast<float *>(smem + Lay::oL);
    float *Uf = Lf;
    float *Tf = reinterpret_cast<float *>(smem + Lay::oT);
    bf16 *Tb = reinterpret_cast<bf16 *>(smem + Lay::oTb);
    bf16 *Ob = Tb;
    bf16 *Ab = reinterpret_cast<bf16 *>(smem + Lay::oA);
    float *Eg = reinterpret_cast<float *>(smem + Lay::oEg);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int dv0 = blockIdx.x * 64;
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
    const int64_t sq = (int64_t)a.H_k * DK;    // elements between tokens in q, k
    const int64_t sv = (int64_t)a.H_v * a.d_v;  // ... in v, o
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * DK;

    // S^T: this warp's 16 rows (d_v) x all d_k columns, m16n8 accumulator layout.
    const int r0 = warp * 16;
    float S[DK / 8][4];
    if (a.h0 != nullptr) {
        const float *h0 = a.h0 + ((int64_t)n * a.H_v + h) * DK * a.d_v + dv0 + r0 + g8;
#pragma unroll
        for (int j = 0; j < DK / 8; ++j) {
            const int d = 8 * j + 2 * t4;
            S[j][0] = h0[(int64_t)d * a.d_v];
            S[j][1] = h0[(int64_t)(d + 1) * a.d_v];
            S[j][2] = h0[(int64_t)d * a.d_v + 8];
            S[j][3] = h0[(int64_t)(d + 1) * a.d_v + 8];
        }
    } else {
#pragma unroll
        for (int j = 0; j < DK / 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
    }

    auto stage = [&](int c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        // q, k: DK/8 vectors of 16 bytes per row
        for (int i = tid; i < 64 * (DK / 8); i += 128) {
            const int r = i / (DK / 8), c8 = (i % (DK / 8)) * 8;
            const bool ok = r < nvalid;
            const int64_t off = ok ? (bos + row0 + r) * sq + (int64_t)hk * DK + c8 : 0;
            cp_async_16(Qraw + r * LDK + c8, q + off, ok ? 16 : 0);
            cp_async_16(Kraw + r * LDK + c8, k + off, ok ? 16 : 0);
        }
        // v: 8 vectors per row (64 values of this CTA's slice)
        for (int i = tid; i < 64 * 8; i += 128) {
            const int r = i >> 3, c8 = (i & 7) * 8;
            const bool ok = r < nvalid;
            const int64_t off = ok ? (bos + row0 + r) * sv + (int64_t)h * a.d_v + dv0 + c8 : 0;
            cp_async_16(Vraw + r * LDV + c8, v + off, ok ? 16 : 0);
        }
        if constexpr (!GATE_HEAD) {
            for (int i = tid; i < 64 * (DK / 4); i += 128) {
                const int r = i / (DK / 4), c4 = (i % (DK / 4)) * 4;
                const bool ok = r < nvalid;
                const int64_t off = ok ? (bos + row0 + r) * sg + (int64_t)h * DK + c4 : 0;
                cp_async_16(G + r * DK + c4, a.g + off, ok ? 16 : 0);
            }
        }
        cp_async_commit();
        if (tid < 64) {
            const bool ok = tid < nvalid;
            Bs[tid] = ok ? (a.decay_only ? 1.f : a.beta[(bos + row0 + tid) * a.H_v + h]) : 0.f;
        } else if (GATE_HEAD) {
            const int r = tid - 64;
            const bool ok = r < nvalid;
            G[r] = ok ? a.g[(bos + row0 + r) * sg + h] : 0.f;
        }
    };

    if (nchunks > 0) stage(0);

    for (int c = 0; c < nchunks; ++c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        cp_async_wait_all();
        __syncthreads();

        // ---- 2. gate: cumulative log2 gate and the decayed operands ---------------------
        if constexpr (!GATE_HEAD) {
            if (tid < DK) {
                const int ch = tid;
                float acc = 0.f;
                for (int r = 0; r < 64; ++r) {
                    acc += G[r * DK + ch] * kLog2e;
                    G[r * DK + ch] = acc;
                    const float ep = exp2f(acc), em = exp2f(-acc);
                    const float kv = __bfloat162float(Kraw[r * LDK + ch]);
                    const float qv = __bfloat162float(Qraw[r * LDK + ch]);
                    Kp[r * LDK + ch] = __float2bfloat16_rn(a.decay_only ? 0.f : kv * ep);
                    Km[r * LDK + ch] = __float2bfloat16_rn(kv * em);
                    Qp[r * LDK + ch] = __float2bfloat16_rn(a.scale * qv * ep);
                }
                Eg[ch] = exp2f(acc);
                for (int r = 0; r < 64; ++r) {
                    const float kv = __bfloat162float(Kraw[r * LDK + ch]);
                    Kbar[r * LDK + ch] = __float2bfloat16_rn(kv * exp2f(acc - G[r * DK + ch]));
                }
            }
        } else {
            // one gate per token: row factors, then an elementwise pass
            float *gam = G + 64, *ep = G + 128, *em = G + 192, *eb = G + 256;
            if (tid < 64) {
                float acc = 0.f;
                for (int s = 0; s <= tid; ++s) acc += G[s] * kLog2e;
                gam[tid] = acc;
            }
            __syncthreads();
            if (tid < 64) {
                const float gn = gam[63];
                ep[tid] = exp2f(gam[tid]);
                em[tid] = exp2f(-gam[tid]);
                eb[tid] = exp2f(gn - gam[tid]);
            }
            if (tid < DK) Eg[tid] = exp2f(gam[63]);
            __syncthreads();
            for (int i = tid; i < 64 * DK; i += 128) {
                const int r = i / DK, ch = i % DK;
                const float kv = __bfloat162float(Kraw[r * LDK + ch]);
                const float qv = __bfloat162float(Qraw[r * LDK + ch]);
                Kp[r * LDK + ch] = __float2bfloat16_rn(a.decay_only ? 0.f : kv * ep[r]);
                Km[r * LDK + ch] = __float2bfloat16_rn(kv * em[r]);
                Qp[r * LDK + ch] = __float2bfloat16_rn(a.scale * qv * ep[r]);
                Kbar[r * LDK + ch] = __float2bfloat16_rn(kv * eb[r]);
            }
        }
        __syncthreads();

        // ---- 3. Gram: M = Kp Km^T, Aqk = Qp Km^T for this warp's 16 rows ----------------
        {
            const int m0 = warp * 16;
            float accM[8][4], accA[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) accM[j][e] = accA[j][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t aK[4], aQ[4];
                ldsm_x4(aK, Kp + (m0 + (lane & 15)) * LDK + kk * 16 + (lane >> 4) * 8);
                ldsm_x4(aQ, Qp + (m0 + (lane & 15)) * LDK + kk * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (p <= warp) {
                        uint32_t b[4];
                        ldsm_x4(b, Km + (16 * p + (lane & 7) + ((lane >> 4) << 3)) * LDK + kk * 16 +
                                       ((lane >> 3) & 1) * 8);
                        mma_bf16(accM[2 * p], aK, b[0], b[1]);
                        mma_bf16(accM[2 * p + 1], aK, b[2], b[3]);
                        mma_bf16(accA[2 * p], aQ, b[0], b[1]);
                        mma_bf16(accA[2 * p + 1], aQ, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = m0 + g8 + 8 * hf;
                    const float br = Bs[r];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = 8 * j + 2 * t4 + e;
                        Lf[r * LDF + col] = col < r ? br * accM[j][2 * hf + e] : 0.f;
                        Ab[r * LDV + col] = __float2bfloat16_rn(col <= r ? accA[j][2 * hf + e] : 0.f);
                    }
                }
            }
        }
        __syncthreads();

        // ---- 4. solve: T = (I + L)^-1, 16x16 diagonal blocks then block merges ------------
        {
            const int jb = lane & 15;
            const int b0 = warp * 16;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float s = (r == jb) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) s -= Lf[(b0 + r) * LDF + b0 + m] * x[m];
                x[r] = s;
            }
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) Tf[(b0 + r) * LDF + b0 + jb] = x[r];
            }
        }
        __syncthreads();
        for (int d = 1; d <= 3; ++d) {
            const int nblk = 4 - d;
            // P_ij = sum_{kb=j}^{i-1} L_i,kb T_kb,j, parked in the unused upper block (j, i)
            for (int it = tid; it < nblk * 256; it += 128) {
                const int bi = d + it / 256, bj = bi - d;
                const int r = (it % 256) / 16, cc = it % 16;
                float s = 0.f;
                for (int kb = bj; kb < bi; ++kb)
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        s += Lf[(16 * bi + r) * LDF + 16 * kb + m] * Tf[(16 * kb + m) * LDF + 16 * bj + cc];
                Tf[(16 * bj + r) * LDF + 16 * bi + cc] = s;
            }
            __syncthreads();
            // T_ij = -T_ii P_ij
            for (int it = tid; it < nblk * 256; it += 128) {
                const int bi = d + it / 256, bj = bi - d;
                const int r = (it % 256) / 16, cc = it % 16;
                float s = 0.f;
                for (int m = 0; m <= r; ++m)
                    s += Tf[(16 * bi + r) * LDF + 16 * bi + m] * Tf[(16 * bj + m) * LDF + 16 * bi + cc];
                Tf[(16 * bi + r) * LDF + 16 * bj + cc] = -s;
            }
            __syncthreads();
        }
        // T_beta = T diag(beta), lower triangle, bf16
        for (int i = tid; i < 64 * 64; i += 128) {
            const int r = i >> 6, cc = i & 63;
            Tb[r * LDV + cc] = __float2bfloat16_rn(cc <= r ? Tf[r * LDF + cc] * Bs[cc] : 0.f);
        }
        __syncthreads();

        // ---- 5. WY factors: W = T_beta Kp, U = T_beta V -----------------------------------
        {
            const int m0 = warp * 16;
            float accW[DK / 8][4], accU[8][4];
#pragma unroll
            for (int j = 0; j < DK / 8; ++j) accW[j][0] = accW[j][1] = accW[j][2] = accW[j][3] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) accU[j][0] = accU[j][1] = accU[j][2] = accU[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (kk <= warp) {
                    uint32_t aT[4];
                    ldsm_x4(aT, Tb + (m0 + (lane & 15)) * LDV + kk * 16 + (lane >> 4) * 8);
                    const int krow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int p = 0; p < DK / 16; ++p) {
                        uint32_t b[4];
                        ldsm_x4_t(b, Kp + krow * LDK + p * 16 + (lane >> 4) * 8);
                        mma_bf16(accW[2 * p], aT, b[0], b[1]);
                        mma_bf16(accW[2 * p + 1], aT, b[2], b[3]);
                    }
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        uint32_t b[4];
                        ldsm_x4_t(b, Vraw + krow * LDV + p * 16 + (lane >> 4) * 8);
                        mma_bf16(accU[2 * p], aT, b[0], b[1]);
                        mma_bf16(accU[2 * p + 1], aT, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < DK / 8; ++j) {
                const int col = 8 * j + 2 * t4;
                *reinterpret_cast<uint32_t *>(Wb + (m0 + g8) * LDK + col) = pack_bf16(accW[j][0], accW[j][1]);
                *reinterpret_cast<uint32_t *>(Wb + (m0 + g8 + 8) * LDK + col) = pack_bf16(accW[j][2], accW[j][3]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = 8 * j + 2 * t4;
                *reinterpret_cast<float2 *>(Uf + (m0 + g8) * LDF + col) = make_float2(accU[j][0], accU[j][1]);
                *reinterpret_cast<float2 *>(Uf + (m0 + g8 + 8) * LDF + col) = make_float2(accU[j][2], accU[j][3]);
            }
        }
        __syncthreads();

        // the raw tiles are free: stage the next chunk while the serial step runs
        if (c + 1 < nchunks) stage(c + 1);

        // ---- 6. serial step on this warp's 16 rows of S^T -------------------------------
        {
            uint32_t sA[DK / 16][4];
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                sA[kk][0] = pack_bf16(S[2 * kk][0], S[2 * kk][1]);
                sA[kk][1] = pack_bf16(S[2 * kk][2], S[2 * kk][3]);
                sA[kk][2] = pack_bf16(S[2 * kk + 1][0], S[2 * kk + 1][1]);
                sA[kk][3] = pack_bf16(S[2 * kk + 1][2], S[2 * kk + 1][3]);
            }
            // Vt^T = U^T - S^T W^T
            float Vt[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tk = 8 * j + 2 * t4;
                Vt[j][0] = Uf[tk * LDF + r0 + g8];
                Vt[j][1] = Uf[(tk + 1) * LDF + r0 + g8];
                Vt[j][2] = Uf[tk * LDF + r0 + g8 + 8];
                Vt[j][3] = Uf[(tk + 1) * LDF + r0 + g8 + 8];
            }
            const int nrow = (lane & 7) + ((lane >> 4) << 3);
            const int kcol = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t na[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) na[e] = sA[kk][e] ^ 0x80008000u;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldsm_x4(b, Wb + (16 * p + nrow) * LDK + kk * 16 + kcol);
                    mma_bf16(Vt[2 * p], na, b[0], b[1]);
                    mma_bf16(Vt[2 * p + 1], na, b[2], b[3]);
                }
            }
            uint32_t vA[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                vA[kk][0] = pack_bf16(Vt[2 * kk][0], Vt[2 * kk][1]);
                vA[kk][1] = pack_bf16(Vt[2 * kk][2], Vt[2 * kk][3]);
                vA[kk][2] = pack_bf16(Vt[2 * kk + 1][0], Vt[2 * kk + 1][1]);
                vA[kk][3] = pack_bf16(Vt[2 * kk + 1][2], Vt[2 * kk + 1][3]);
            }
            // O^T = S^T Qp^T + Vt^T Aqk^T
            float O[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldsm_x4(b, Qp + (16 * p + nrow) * LDK + kk * 16 + kcol);
                    mma_bf16(O[2 * p], sA[kk], b[0], b[1]);
                    mma_bf16(O[2 * p + 1], sA[kk], b[2], b[3]);
                }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (kk <= p) {
                        uint32_t b[4];
                        ldsm_x4(b, Ab + (16 * p + nrow) * LDV + kk * 16 + kcol);
                        mma_bf16(O[2 * p], vA[kk], b[0], b[1]);
                        mma_bf16(O[2 * p + 1], vA[kk], b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tk = 8 * j + 2 * t4;
                Ob[tk * LDV + r0 + g8] = __float2bfloat16_rn(O[j][0]);
                Ob[(tk + 1) * LDV + r0 + g8] = __float2bfloat16_rn(O[j][1]);
                Ob[tk * LDV + r0 + g8 + 8] = __float2bfloat16_rn(O[j][2]);
                Ob[(tk + 1) * LDV + r0 + g8 + 8] = __float2bfloat16_rn(O[j][3]);
            }
            // S^T <- S^T Diag(e^gamma_n) + Vt^T Kbar
#pragma unroll
            for (int j = 0; j < DK / 8; ++j) {
                const float e0 = Eg[8 * j + 2 * t4], e1 = Eg[8 * j + 2 * t4 + 1];
                S[j][0] *= e0;
                S[j][1] *= e1;
                S[j][2] *= e0;
                S[j][3] *= e1;
            }
            const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int p = 0; p < DK / 16; ++p) {
                    uint32_t b[4];
                    ldsm_x4_t(b, Kbar + (16 * kk + krow) * LDK + 16 * p + (lane >> 4) * 8);
                    mma_bf16(S[2 * p], vA[kk], b[0], b[1]);
                    mma_bf16(S[2 * p + 1], vA[kk], b[2], b[3]);
                }
            }
        }
        __syncthreads();

        // O tile -> global, valid rows only, 16-byte stores
        for (int i = tid; i < 64 * 8; i += 128) {
            const int r = i >> 3, c8 = (i & 7) * 8;
            if (r < nvalid) {
                *reinterpret_cast<uint4 *>(o + (bos + row0 + r) * sv + (int64_t)h * a.d_v + dv0 + c8) =
                    *reinterpret_cast<const uint4 *>(Ob + r * LDV + c8);
            }
        }
    }

    if (a.ht != nullptr) {
        float *ht = a.ht + ((int64_t)n * a.H_v + h) * DK * a.d_v + dv0 + r0 + g8;
#pragma unroll
        for (int j = 0; j < DK / 8; ++j) {
            const int d = 8 * j + 2 * t4;
            ht[(int64_t)d * a.d_v] = S[j][0];
            ht[(int64_t)(d + 1) * a.d_v] = S[j][1];
            ht[(int64_t)d * a.d_v + 8] = S[j][2];
            ht[(int64_t)(d + 1) * a.d_v + 8] = S[j][3];
        }
    }
}

template <int DK, bool GATE_HEAD>
cudaError_t launch_bf16(const FwdArgs &a, cudaStream_t stream) {
    constexpr int kSmem = Bf16Layout<DK>::kBytes;
    auto kern = kda_fwd_bf16_kernel<DK, GATE_HEAD>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    const dim3 grid(a.d_v / 64, a.H_v, a.N);
    kern<<<grid, 128, kSmem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs &a, cudaStream_t stream) {
    if (a.d_k == 128) return a.gate_per_head ? launch_bf16<128, true>(a, stream) : launch_bf16<128, false>(a, stream);
    return a.gate_per_head ? launch_bf16<64, true>(a, stream) : launch_bf16<64, false>(a, stream);
}

}  // namespace kda
