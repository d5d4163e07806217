// Chunkwise KDA forward for d_k = d_v = 128, bf16 operands, on the 5th-generation tensor
// cores (tcgen05) with accumulators in tensor memory (TMEM), warp-specialised.
//
// One CTA of 384 threads runs one (sequence, value head) unit through all its chunks. Per
// chunk ("RNN的复兴04:线性注意力并行计算DPLR", §5.3.5; "TileLang 实战：KDA 从零到一–Kimi
// Delta Attention", §3.3) the work splits into a part that depends only on the chunk's own
// inputs ("prep") and the serial step that carries the state. Eight prep warps build
// chunk c + 1 while the four serial warps run chunk c:
//
//   prep (warps 4-11), chunk c:
//     TMA    Q, K [64 x 128], V [64 x 128] (128-byte swizzled), G [64 x 128] fp32
//     gate   gamma = chunk-local cumulative log2 gate; Qp = scale Q e^gamma, Kp = K e^gamma,
//            Km = K e^-gamma, Kbar = Km e^gamma_n, all stored transposed [d][tok] in bf16
//     Gram   D_G [128 x 64] = [Qp; Kp] Km^T   -> Aqk (lower) in bf16, L = diag(beta) M (strict)
//     solve  T = (I + L)^-1: 16x16 diagonal blocks by forward substitution, off-diagonal
//            blocks column by column on tf32 mma.sync; T_beta = T diag(beta) in bf16
//     WY     D_W = Kp^T T_beta^T (W^T), D_U = V^T T_beta^T (U^T, left in TMEM)
//   serial (warps 0-3, thread = d_v row), chunk c, state S^T [d_v x d_k] fp32 in TMEM:
//     D_X [128 x 128] = S^T [W^T | Qp^T]           (S^T as a bf16 TMEM operand)
//     S^T <- S^T Diag(e^gamma_n)                    (in TMEM, while D_X is computed)
//     Vt^T = U^T - D_X[:, :64]  -> bf16 TMEM operand
//     D_X[:, 64:] += Vt^T Aqk^T (= O^T);  S^T += Vt^T Kbar
//
// The prep -> serial hand-off (Qp^T, Kbar^T, Aqk, e^gamma_n, U^T) is double-buffered; W^T
// is single-buffered behind a release barrier. All operands stay in shared memory or TMEM;
// only q, k, v, g, beta, h0 (in) and o, ht (out) touch HBM.
//
// Every mbarrier wait is bounded (about one second); on a timeout the CTA raises
// KDA_DEVICE_ERR_TIMEOUT, waits (bounded) for the MMAs it issued, frees its TMEM and returns.
#include <cstring>

#include "tc_util.cuh"

namespace kda {

namespace {

using bf16 = __nv_bfloat16;
using namespace tc5;
using namespace tcu;

// Shared-memory plan (byte offsets from a 1024-byte aligned base). Tiles named [d][tok]
// hold one row per d_k channel and 64 tokens per 128-byte row (one swizzle atom).
struct WsLayout {
    static constexpr int oRQ = 0;        // raw Q [64 tok][128] bf16 row-major
    static constexpr int oRK = 16384;    // raw K
    static constexpr int oRV = 32768;    // raw V [2 atoms (d_v)][64 tok][128 B] (MN-major A of U^T)
    static constexpr int oG = 49152;     // raw G fp32 [64][128]; then L and T fp32 [64][68]
    static constexpr int oL = oG;
    static constexpr int oT = oG + 17408;
    static constexpr int oRN = oG;       // front-end norm factors [128] fp32 (between the gate
                                         // sums and the Gram read-back)
    static constexpr int oWT = 83968;    // W^T [d][tok]        } WT, QP0, QP1, KP in this order:
    static constexpr int oQP0 = 100352;  // Qp^T [d][tok], slot 0} serial B operand (WT | QP[b]),
    static constexpr int oQP1 = 116736;  // Qp^T, slot 1          } Gram A operand (QP[b] | KP)
    static constexpr int oKP = 133120;   // Kp^T [d][tok]
    static constexpr int oKM = 149504;   // Km^T [d][tok]; after the Gram, T_beta at +8192
    static constexpr int oTB = oKM + 8192;
    static constexpr int oKB0 = 165888;  // Kbar^T [d][tok], slots 0 and 1
    static constexpr int oKB1 = 182272;
    static constexpr int oAQ0 = 198656;  // Aqk [tok][tok'] bf16 (K-major B), slots 0 and 1
    static constexpr int oAQ1 = 206848;
    static constexpr int oBeta = 215040;  // [64] fp32
    static constexpr int oGh = oBeta + 256;   // [64] fp32 per-head gates
    static constexpr int oTot = oGh + 256;    // [4][128] fp32 partial gate sums
    static constexpr int oEG0 = oTot + 2048;  // [128] fp32 e^gamma_n, slots 0 and 1
    static constexpr int oEG1 = oEG0 + 512;
    static constexpr int oBar = oEG1 + 512;   // mbarriers
    static constexpr int oTmemAddr = oBar + 256;
    static constexpr int oFlag = oTmemAddr + 16;  // abort flag
    static constexpr int oPS = oFlag + 16;        // solve scratch, 8 warps x 16x8 fp32
    static constexpr int oOS = oPS + 4096;        // O staging [32 tok][128] bf16 (serial)
    static constexpr int kBytes = oOS + 8192 + 1024;  // + slack to align the base
};

// TMEM columns (512 allocated)
constexpr uint32_t tGW = 0;    // Gram D_G, then W^T (prep)
constexpr uint32_t tU0 = 64;   // U^T, slot 0 (64) ; slot 1 at tU1
constexpr uint32_t tX = 128;   // [S^T W^T | O^T] (128); Vt^T in bf16 overwrites cols 0-31
constexpr uint32_t tSA = 256;  // S^T in bf16 (64 packed columns)
constexpr uint32_t tS = 320;   // S^T fp32 (128)
constexpr uint32_t tU1 = 448;  // U^T, slot 1 (64)
constexpr uint32_t kTmemCols = 512;

enum {
    BAR_LQK = 0, // TMA tiles of a chunk: Q and K
    BAR_LG,      //   G
    BAR_LV,      //   V
    BAR_G,       // Gram MMA done
    BAR_W,       // WY MMAs done
    BAR_FULL0,   // hand-off slot 0 / 1 ready (prep -> serial)
    BAR_FULL1,
    BAR_FREE0,   // hand-off slot 0 / 1 consumed (serial -> prep)
    BAR_FREE1,
    BAR_WT,      // W^T consumed (serial -> prep)
    BAR_X,       // serial product D_X done
    BAR_S2,      // serial products O^T, S^T done
    BAR_Z0,      // drains after a timeout (one per MMA-issuing thread)
    BAR_Z1,
    BAR_NEVER,   // test aid: a phase that nothing completes (see FwdArgs::wait_cycles)
    kNumBars
};


__device__ __forceinline__ void bar_serial() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void bar_prep() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

// Bounded wait on an mbarrier phase; gives up early when the CTA is aborting. On its own
// timeout it marks the CTA as aborting. Returns false when the phase did not complete.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

struct Unit {
    unsigned char *sm;
    uint32_t sbase, tmem;
    int h, hk, n, len, nchunks;
    int64_t bos;
    uint64_t *bars;
    volatile int *abort_flag;
};

// ---------------------------------------------------------------------------------------
// prep warps (4-11): TMA staging, gate pass, Gram, solve, WY factors for every chunk.
// Returns the loads that may still be in flight (abort path): for Q/K, G and V, two bits
// each holding 1 + the parity of the pending chunk, or 0. With FE the front-end is applied
// on the way: beta and the per-head gates as they land, the per-channel gates before the
// cumulative sum, and the q / k norms as factors of the image rows (kept in the first 512
// bytes of the G region, free between the gate sums and the Gram read-back).
// ---------------------------------------------------------------------------------------
template <bool GATE_HEAD, bool FE>
__device__ __forceinline__ int prep_role(const FwdArgs &a, const TcMaps &maps, const Unit &u) {
    using Lay = WsLayout;
    unsigned char *sm = u.sm;
    const uint32_t sbase = u.sbase, tmem = u.tmem;
    uint64_t *bars = u.bars;
    const int ptid = threadIdx.x - 128, pw = ptid >> 5, lane = ptid & 31, warp = threadIdx.x >> 5;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter
    const uint32_t half = (uint32_t)(pw >> 2) * 32u;                // column half of a 64-wide readback
    const bf16 *RQ = reinterpret_cast<const bf16 *>(sm + Lay::oRQ);
    const bf16 *RK = reinterpret_cast<const bf16 *>(sm + Lay::oRK);
    float *G = reinterpret_cast<float *>(sm + Lay::oG);
    float *L = reinterpret_cast<float *>(sm + Lay::oL);
    float *Tm = reinterpret_cast<float *>(sm + Lay::oT);
    float *Bs = reinterpret_cast<float *>(sm + Lay::oBeta);
    float *Gh = reinterpret_cast<float *>(sm + Lay::oGh);
    float *Tot = reinterpret_cast<float *>(sm + Lay::oTot);
    const int h = u.h, hk = u.hk, len = u.len, nchunks = u.nchunks;
    const int64_t bos = u.bos;
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * 128;
    // TMA tiles that may still be in flight, as the parity of their chunk (or -1)
    int pend_qk = -1, pend_g = -1, pend_v = -1;
    // Stage chunk c's tiles, each as soon as its buffer is free: Q and K after the gate pass,
    // G (with beta and the per-head gates, by cp.async) after the solve, V after the WY MMAs.
    auto stage_qk = [&](int c) {
        if (ptid == 0) {
            const int y = (int)(bos + c * kChunk);
            mbar_arrive_expect_tx(&bars[BAR_LQK], 32768);
            tma_load_2d(sm + Lay::oRQ, &maps.q, &bars[BAR_LQK], hk * 128, y);
            tma_load_2d(sm + Lay::oRK, &maps.k, &bars[BAR_LQK], hk * 128, y);
        }
        pend_qk = c & 1;
    };
    auto stage_v = [&](int c) {
        if (ptid == 0) {
            const int y = (int)(bos + c * kChunk);
            mbar_arrive_expect_tx(&bars[BAR_LV], 16384);
            tma_load_2d(sm + Lay::oRV, &maps.v, &bars[BAR_LV], h * 128, y);
            tma_load_2d(sm + Lay::oRV + 8192, &maps.v, &bars[BAR_LV], h * 128 + 64, y);
        }
        pend_v = c & 1;
    };
    // front-end constants of this unit: -exp(A_log[h]) and this thread's channel biases
    float negA = 0.f, bias0 = 0.f, bias1 = 0.f;
    if constexpr (FE) {
        if (a.fe_A_log != nullptr) {
            negA = -expf(a.fe_A_log[h]);
            if (a.fe_dt_bias != nullptr) {
                if constexpr (GATE_HEAD) {
                    bias0 = a.fe_dt_bias[h];
                } else {
                    const int cb = 64 * (pw & 1) + lane;
                    bias0 = a.fe_dt_bias[h * 128 + cb];
                    bias1 = a.fe_dt_bias[h * 128 + cb + 32];
                }
            }
        }
    }
    auto stage_g = [&](int c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        if constexpr (!GATE_HEAD) {
            if (ptid == 0) {
                mbar_arrive_expect_tx(&bars[BAR_LG], 32768);
                tma_load_2d(sm + Lay::oG, &maps.g, &bars[BAR_LG], h * 128, (int)(bos + row0));
            }
            pend_g = c & 1;
        }
        if (ptid < 64) {
            const bool ok = ptid < nvalid;
            if (a.decay_only) {
                Bs[ptid] = ok ? 1.f : 0.f;
            } else {
                const int64_t ob = ok ? (bos + row0 + ptid) * a.H_v + h : 0;
                cp_async_4(Bs + ptid, a.beta + ob, ok ? 4 : 0);
            }
        } else if (GATE_HEAD && ptid < 128) {
            const int r = ptid - 64;
            const bool ok = r < nvalid;
            const int64_t og = ok ? (bos + row0 + r) * sg + h : 0;
            cp_async_4(Gh + r, a.g + og, ok ? 4 : 0);
        }
        cp_async_commit();
    };

    bool failed = false;
    if (nchunks > 0) {
        stage_g(0);
        stage_qk(0);
        stage_v(0);
    }
    for (int p = 0; p < nchunks; ++p) {
        const int row0 = p * kChunk;
        const int nvalid = min(kChunk, len - row0);
        const int b = p & 1;
        const uint32_t oQP = b ? Lay::oQP1 : Lay::oQP0;
        const uint32_t oKB = b ? Lay::oKB1 : Lay::oKB0;
        const uint32_t oAQ = b ? Lay::oAQ1 : Lay::oAQ0;
        float *EG = reinterpret_cast<float *>(sm + (b ? Lay::oEG1 : Lay::oEG0));
        const uint32_t tU = b ? tU1 : tU0;
        // rows past the sequence end hold the next sequence (or zeros past the tensor) and
        // must be zero in every operand
        const int nz = kChunk - nvalid;

        // G, beta of chunk p, and hand-off slot b released by the serial step of chunk p - 2
        cp_async_wait_all();
        if constexpr (FE) {
            // each thread transforms the values it loaded itself (rows past the end stay 0)
            if (ptid < 64) {
                if (a.fe_beta_sigmoid && !a.decay_only && ptid < nvalid) Bs[ptid] = sigmoid_fast(Bs[ptid]);
            } else if (GATE_HEAD && ptid < 128 && a.fe_A_log != nullptr && ptid - 64 < nvalid) {
                Gh[ptid - 64] = negA * softplus_fast(Gh[ptid - 64] + bias0);
            }
        }
        if constexpr (!GATE_HEAD) failed = !wait_bar(&bars[BAR_LG], (uint32_t)(p & 1), u.abort_flag, a.wait_cycles);
        if (!failed && p >= 2)
            failed = !wait_bar(&bars[b ? BAR_FREE1 : BAR_FREE0], (uint32_t)(((p >> 1) - 1) & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        pend_g = -1;
        if (!GATE_HEAD && nz > 0) {
            for (int i = ptid; i < nz * 32; i += 256) {
                const int r = nvalid + (i >> 5), c16 = i & 31;
                *reinterpret_cast<uint4 *>(sm + Lay::oG + r * 512 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            bar_prep();
        }

        // ---- gate pass ---------------------------------------------------------------------
        // prep warp pw: rows 16 (pw >> 1) .. +15, channels c0 = 64 (pw & 1) + lane and c0 + 32.
        {
            const int qr = pw >> 1;
            const int c0 = 64 * (pw & 1) + lane, c1 = c0 + 32;
            float gl0[16], gl1[16];
            bool gate_done = false;
            if constexpr (!GATE_HEAD && FE) {
                if (a.fe_A_log != nullptr) {
                    // every gate of the thread first (independent), then the running sums
                    const float nAl = negA * kLog2e;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = 16 * qr + e;
                        const float v0 = nAl * softplus_fast(G[r * 128 + c0] + bias0);
                        const float v1 = nAl * softplus_fast(G[r * 128 + c1] + bias1);
                        gl0[e] = r < nvalid ? v0 : 0.f;
                        gl1[e] = r < nvalid ? v1 : 0.f;
                    }
#pragma unroll
                    for (int e = 1; e < 16; ++e) {
                        gl0[e] += gl0[e - 1];
                        gl1[e] += gl1[e - 1];
                    }
                    Tot[qr * 128 + c0] = gl0[15];
                    Tot[qr * 128 + c1] = gl1[15];
                    gate_done = true;
                }
            }
            if (!gate_done) {
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
            }
            failed = !wait_bar(&bars[BAR_LQK], (uint32_t)(p & 1), u.abort_flag, a.wait_cycles);
            if (bar_or(2, 256, failed)) { failed = true; break; }
            pend_qk = -1;
            if (nz > 0) {
                for (int i = ptid; i < nz * 16; i += 256) {
                    const int r = nvalid + (i >> 4), c16 = i & 15;
                    *reinterpret_cast<uint4 *>(sm + Lay::oRQ + r * 256 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(sm + Lay::oRK + r * 256 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                bar_prep();
            }
            if constexpr (FE) {
                if (a.fe_qk_l2norm) {
                    qk_row_norms(sm + Lay::oRQ, sm + Lay::oRK, reinterpret_cast<float *>(sm + Lay::oRN), pw, lane,
                                 a.scale);
                    bar_prep();
                }
            }
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
                EG[c0] = eg0;
                EG[c1] = eg1;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tc = 2 * qr + j;  // 16-byte chunk (8 tokens) of a 64-token row
                // front-end: the factors of these 8 rows (q: scale / |q|, k: 1 / |k|)
                float fq[8], fk[8];
                if constexpr (FE) {
                    const bool nrm = a.fe_qk_l2norm != 0;
                    const float4 *RN4 = reinterpret_cast<const float4 *>(sm + Lay::oRN) + 4 * qr + 2 * j;
                    const float4 q0 = nrm ? RN4[0] : make_float4(a.scale, a.scale, a.scale, a.scale);
                    const float4 q1 = nrm ? RN4[1] : q0;
                    const float4 k0 = nrm ? RN4[16] : make_float4(1.f, 1.f, 1.f, 1.f);
                    const float4 k1 = nrm ? RN4[17] : k0;
                    fq[0] = q0.x; fq[1] = q0.y; fq[2] = q0.z; fq[3] = q0.w;
                    fq[4] = q1.x; fq[5] = q1.y; fq[6] = q1.z; fq[7] = q1.w;
                    fk[0] = k0.x; fk[1] = k0.y; fk[2] = k0.z; fk[3] = k0.w;
                    fk[4] = k1.x; fk[5] = k1.y; fk[6] = k1.z; fk[7] = k1.w;
                }
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
                        float kv = __bfloat162float(RK[r * 128 + cc]);
                        const float qv = __bfloat162float(RQ[r * 128 + cc]);
                        float qs = a.scale;
                        if constexpr (FE) {
                            qs = fq[e];
                            kv *= fk[e];
                        }
                        kp[e] = a.decay_only ? 0.f : kv * ep;
                        km[e] = kv * em;
                        qp[e] = qs * qv * ep;
                        kb[e] = km[e] * eg;
                    }
                    const uint32_t sw = sw128(cc, tc);
                    *reinterpret_cast<uint4 *>(sm + Lay::oKP + sw) = pack8(kp);
                    *reinterpret_cast<uint4 *>(sm + oQP + sw) = pack8(qp);
                    *reinterpret_cast<uint4 *>(sm + Lay::oKM + sw) = pack8(km);
                    *reinterpret_cast<uint4 *>(sm + oKB + sw) = pack8(kb);
                }
            }
        }
        fence_proxy_async();
        bar_prep();
        if (p + 1 < nchunks) stage_qk(p + 1);  // the raw Q and K tiles are consumed

        // ---- Gram: D_G = [Qp; Kp] Km^T  (rows 0-63: Aqk, rows 64-127: M) --------------------
        if (ptid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, true, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + tGW, dMN(sbase + oQP, (uint32_t)(Lay::oKP - oQP), s), dMN(sbase + Lay::oKM, 16384, s), id,
                    s > 0);
            commit(&bars[BAR_G]);
        }
        failed = !wait_bar(&bars[BAR_G], (uint32_t)(p & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        fence_after_sync();
        {
            // each warp half reads 32 of the 64 columns of its lane's row
            const int row = 32 * (warp & 3) + lane;
            float x[32];
            tmem_ld32(tmem + lane_off + tGW + half, x);
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
                    *reinterpret_cast<uint4 *>(sm + oAQ + sw128(row, (int)(half >> 3) + c8)) = pack8(y);
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
        bar_prep();

        // ---- solve: T = (I + L)^-1 -----------------------------------------------------------
        // the 16x16 diagonal inverses by forward substitution, one column per lane
        if (pw < 4 && lane < 16) {
            const int b0 = 16 * pw, j = lane;
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
        bar_prep();
        // Off-diagonal blocks column by column: prep warp pw owns the 8 columns col0..col0+7
        // of T (column block j = pw / 2). T_jj = D_j, and for i > j
        //   T_ij = -D_i sum_{k=j}^{i-1} L_ik T_kj
        // (tf32 mma.sync, fp32 accumulation, one accumulator per k so that the products of a
        // step run side by side). The warp then writes its columns of T_beta = T diag(beta)
        // (lower triangle) in bf16. Each warp reads only L, the diagonal blocks and its own
        // columns, so no CTA-wide barrier is needed inside.
        {
            const int j = pw >> 1, col0 = 16 * j + 8 * (pw & 1);
            const int g8 = lane >> 2, t4 = lane & 3;
            float *P = reinterpret_cast<float *>(sm + Lay::oPS) + pw * 128;  // 16x8 scratch
            for (int i = j + 1; i < 4; ++i) {
                float acc[3][4];
#pragma unroll
                for (int kk = 0; kk < 3; ++kk) acc[kk][0] = acc[kk][1] = acc[kk][2] = acc[kk][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 3; ++kk)
                    if (j + kk < i)
                        mm16x8_tf32(acc[kk], L + (16 * i) * LDF + 16 * (j + kk), LDF, Tm + (16 * (j + kk)) * LDF + col0,
                                    LDF, lane);
                P[g8 * 8 + 2 * t4] = acc[0][0] + acc[1][0] + acc[2][0];
                P[g8 * 8 + 2 * t4 + 1] = acc[0][1] + acc[1][1] + acc[2][1];
                P[(g8 + 8) * 8 + 2 * t4] = acc[0][2] + acc[1][2] + acc[2][2];
                P[(g8 + 8) * 8 + 2 * t4 + 1] = acc[0][3] + acc[1][3] + acc[2][3];
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
        bar_prep();
        if (p + 1 < nchunks) stage_g(p + 1);  // G, L, T and beta are consumed
        failed = !wait_bar(&bars[BAR_LV], (uint32_t)(p & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        pend_v = -1;
        if (nz > 0) {
            for (int i = ptid; i < nz * 16; i += 256) {
                const int r = nvalid + (i >> 4), c16 = i & 15;
                *reinterpret_cast<uint4 *>(sm + Lay::oRV + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async();
            bar_prep();
        }

        // ---- WY factors: D_W = Kp^T T_beta^T, D_U = V^T T_beta^T ------------------------------
        if (ptid == 0) {
            fence_after_sync();
            const uint32_t idw = idesc_bf16(128, 64, false, false, false);
            const uint32_t idu = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = dK(sbase + Lay::oTB, 8192, s);
                mma(tmem + tGW, dK(sbase + Lay::oKP, 16384, s), bd, idw, s > 0);
                mma(tmem + tU, dMN(sbase + Lay::oRV, 8192, s), bd, idu, s > 0);
            }
            commit(&bars[BAR_W]);
        }
        // W^T is single-buffered: the serial product of chunk p - 1 must have read it
        failed = !wait_bar(&bars[BAR_W], (uint32_t)(p & 1), u.abort_flag, a.wait_cycles);
        if (!failed && p >= 1) failed = !wait_bar(&bars[BAR_WT], (uint32_t)((p - 1) & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        if (p + 1 < nchunks) stage_v(p + 1);  // the U MMA has read V
        fence_after_sync();
        {
            // W^T row d -> bf16 [d][tok] (MN-major B); each warp half writes 32 of the 64 tokens
            const int d = 32 * (warp & 3) + lane;
            float x[32];
            tmem_ld32(tmem + lane_off + tGW + half, x);
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
        bar_prep();
        // hand chunk p to the serial warps
        if (ptid == 0) mbar_arrive(&bars[b ? BAR_FULL1 : BAR_FULL0]);
    }
    if (failed) *u.abort_flag = 1;
    return (pend_qk + 1) | ((pend_g + 1) << 2) | ((pend_v + 1) << 4);
}

// ---------------------------------------------------------------------------------------
// serial warps (0-3): thread dv owns row dv of S^T (fp32 in TMEM) for the whole sequence.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void serial_role(const FwdArgs &a, const Unit &u) {
    using Lay = WsLayout;
    unsigned char *sm = u.sm;
    const uint32_t sbase = u.sbase, tmem = u.tmem;
    uint64_t *bars = u.bars;
    const int dv = threadIdx.x, warp = dv >> 5;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int h = u.h, n = u.n, len = u.len, nchunks = u.nchunks;
    const int64_t bos = u.bos;
    const int64_t sv = (int64_t)a.H_v * 128;
    bf16 *o = static_cast<bf16 *>(a.o);

    // S^T row dv (from h0, or zero) -> TMEM fp32, and its bf16 copy (the MMA operand)
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int d = 32 * pass + e;
            x[e] = a.h0 ? a.h0[(((int64_t)n * a.H_v + h) * 128 + d) * 128 + dv] : 0.f;
        }
        uint32_t f0[16], f1[16], p16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            f0[e] = __float_as_uint(x[e]);
            f1[e] = __float_as_uint(x[16 + e]);
            p16[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        }
        tmem_st16(tmem + lane_off + tS + 32 * pass, f0);
        tmem_st16(tmem + lane_off + tS + 32 * pass + 16, f1);
        tmem_st16(tmem + lane_off + tSA + 16 * pass, p16);
    }
    tmem_st_wait();
    fence_before_sync();
    bar_serial();

    bool failed = false;
    if (a.wait_cycles < kDefaultWaitCycles) {
        // test aid (shortened waits): first wait on a phase that nothing completes, so that
        // the call takes the failure path every time
        failed = !wait_bar(&u.bars[BAR_NEVER], 0u, u.abort_flag, a.wait_cycles);
        failed = bar_or(1, 128, failed);
    }
    for (int c = 0; c < nchunks && !failed; ++c) {
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, len - row0);
        const int b = c & 1;
        const uint32_t oQP = b ? Lay::oQP1 : Lay::oQP0;
        const uint32_t oKB = b ? Lay::oKB1 : Lay::oKB0;
        const uint32_t oAQ = b ? Lay::oAQ1 : Lay::oAQ0;
        const float *EG = reinterpret_cast<const float *>(sm + (b ? Lay::oEG1 : Lay::oEG0));
        const uint32_t tU = b ? tU1 : tU0;

        failed = !wait_bar(&bars[b ? BAR_FULL1 : BAR_FULL0], (uint32_t)((c >> 1) & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(1, 128, failed)) { failed = true; break; }
        fence_after_sync();

        // D_X = S^T [W^T | Qp^T]  (A: S^T bf16 in TMEM; B: the W^T and Qp^T tiles, MN-major)
        if (dv == 0) {
            const uint32_t id = idesc_bf16(128, 128, false, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_ts(tmem + tX, tmem + tSA + 8 * s, dMN(sbase + Lay::oWT, (uint32_t)(oQP - Lay::oWT), s), id,
                       s > 0);
            commit(&bars[BAR_X]);
        }
        // meanwhile S^T <- S^T Diag(e^gamma_n): column d of S^T scales by e^gamma_n[d]
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            float x[32];
            tmem_ld32(tmem + lane_off + tS + 32 * pass, x);
            uint32_t y0[16], y1[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                y0[e] = __float_as_uint(x[e] * EG[32 * pass + e]);
                y1[e] = __float_as_uint(x[16 + e] * EG[32 * pass + 16 + e]);
            }
            tmem_st16(tmem + lane_off + tS + 32 * pass, y0);
            tmem_st16(tmem + lane_off + tS + 32 * pass + 16, y1);
        }
        tmem_st_wait();

        failed = !wait_bar(&bars[BAR_X], (uint32_t)(c & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(1, 128, failed)) { failed = true; break; }
        fence_after_sync();
        if (dv == 0) mbar_arrive(&bars[BAR_WT]);  // W^T is no longer needed
        // Vt^T = U^T - S^T W^T -> bf16 pairs over tokens, written over D_X columns 0-31
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            float uu[32], pp[32];
            tmem_ld32(tmem + lane_off + tU + 32 * pass, uu);
            tmem_ld32(tmem + lane_off + tX + 32 * pass, pp);
            uint32_t v16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v16[e] = pack_bf16(uu[2 * e] - pp[2 * e], uu[2 * e + 1] - pp[2 * e + 1]);
            tmem_st16(tmem + lane_off + tX + 16 * pass, v16);
        }
        tmem_st_wait();
        fence_before_sync();
        bar_serial();

        // O^T += Vt^T Aqk^T;  S^T += Vt^T Kbar  (A: Vt^T bf16 in TMEM)
        if (dv == 0) {
            fence_after_sync();
            const uint32_t ido = idesc_bf16(128, 64, false, false, false);
            const uint32_t ids = idesc_bf16(128, 128, false, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                mma_ts(tmem + tX + 64, tmem + tX + 8 * s, dK(sbase + oAQ, 8192, s), ido, 1);
                mma_ts(tmem + tS, tmem + tX + 8 * s, dK(sbase + oKB, 16384, s), ids, 1);
            }
            commit(&bars[BAR_S2]);
        }
        failed = !wait_bar(&bars[BAR_S2], (uint32_t)(c & 1), u.abort_flag, a.wait_cycles);
        if (bar_or(1, 128, failed)) { failed = true; break; }
        fence_after_sync();
        if (dv == 0) mbar_arrive(&bars[b ? BAR_FREE1 : BAR_FREE0]);  // hand-off slot b consumed

        // S^T -> bf16 operand for the next chunk
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            float x[32];
            tmem_ld32(tmem + lane_off + tS + 32 * pass, x);
            uint32_t p16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) p16[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
            tmem_st16(tmem + lane_off + tSA + 16 * pass, p16);
        }
        tmem_st_wait();
        // O^T row dv -> o[token][dv], valid tokens only: 32 tokens at a time through a
        // [32 tok][128 dv] staging tile so that global stores are 16 bytes wide
        bf16 *OS = reinterpret_cast<bf16 *>(sm + Lay::oOS);
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            float x[32];
            tmem_ld32(tmem + lane_off + tX + 64 + 32 * pass, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) OS[e * 128 + dv] = __float2bfloat16_rn(x[e]);
            bar_serial();
#pragma unroll
            for (int i = dv; i < 512; i += 128) {
                const int r = i >> 4, c16 = i & 15;
                const int tok = 32 * pass + r;
                if (tok < nvalid)
                    *reinterpret_cast<uint4 *>(o + (bos + row0 + tok) * sv + (int64_t)h * 128 + c16 * 8) =
                        *reinterpret_cast<const uint4 *>(sm + Lay::oOS + r * 256 + c16 * 16);
            }
            bar_serial();
        }
        fence_before_sync();
    }
    if (failed) {
        *u.abort_flag = 1;
        return;
    }
    if (a.ht != nullptr) {
        float *ht = a.ht + ((int64_t)n * a.H_v + h) * 128 * 128 + dv;
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            float x[32];
            tmem_ld32(tmem + lane_off + tS + 32 * pass, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) ht[(int64_t)(32 * pass + e) * 128] = x[e];
        }
    }
}

template <bool GATE_HEAD, bool FE>
__global__ void __launch_bounds__(384, 1) kda_fwd_tc_kernel(const FwdArgs a, const __grid_constant__ TcMaps maps) {
    using Lay = WsLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::oBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::oTmemAddr);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + Lay::oFlag);
    const int tid = threadIdx.x, warp = tid >> 5;

    Unit u;
    u.sm = sm;
    u.sbase = smem_u32(sm);
    u.h = blockIdx.y;
    u.n = blockIdx.z;
    if (a.cu_seqlens != nullptr && a.N <= 64) {
        // Packed sequences of different lengths: blocks start in index order, so block z
        // takes the z-th longest sequence (ties by index) and no long unit starts in the
        // last wave. The lengths are ranked in the (not yet used) solve scratch.
        int *len_s = reinterpret_cast<int *>(sm + Lay::oPS);
        if (tid < a.N) len_s[tid] = a.cu_seqlens[tid + 1] - a.cu_seqlens[tid];
        __syncthreads();
        if (tid < a.N) {
            const int ls = len_s[tid];
            int rank = 0;
            for (int t = 0; t < a.N; ++t) rank += (len_s[t] > ls) || (len_s[t] == ls && t < tid);
            if (rank == (int)blockIdx.z) len_s[64] = tid;
        }
        __syncthreads();
        u.n = len_s[64];
        __syncthreads();
    }
    u.hk = u.h / a.group;
    if (!seq_bounds(a, u.n, u.bos, u.len)) return;
    u.nchunks = (u.len + kChunk - 1) / kChunk;
    u.bars = bars;
    u.abort_flag = abort_flag;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    u.tmem = *tmem_slot;

    int tma_pending = 0;
    if (tid < 128)
        serial_role(a, u);
    else
        tma_pending = prep_role<GATE_HEAD, FE>(a, maps, u);

    fence_before_sync();
    __syncthreads();
    if (*abort_flag) {
        // drain: every MMA and TMA this CTA issued must land before TMEM is freed and the
        // CTA exits (bounded waits)
        if (tid == 0 || tid == 128) {
            atomicOr(a.err, kDeviceErrTimeout);
            fence_after_sync();
            uint64_t *z = &bars[tid == 0 ? BAR_Z0 : BAR_Z1];
            commit(z);
            mbar_wait(z, 0, kWaitCycles);
        }
        if (tid == 128) {
            const int pq = (tma_pending & 3) - 1, pg = ((tma_pending >> 2) & 3) - 1, pv = ((tma_pending >> 4) & 3) - 1;
            if (pq >= 0) mbar_wait(&bars[BAR_LQK], (uint32_t)pq, kWaitCycles);
            if (pg >= 0) mbar_wait(&bars[BAR_LG], (uint32_t)pg, kWaitCycles);
            if (pv >= 0) mbar_wait(&bars[BAR_LV], (uint32_t)pv, kWaitCycles);
        }
        cp_async_wait_all();
        fence_before_sync();
        __syncthreads();
    }
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(u.tmem, kTmemCols);
    }
}


template <bool GATE_HEAD, bool FE>
cudaError_t launch_tc(const FwdArgs &a, cudaStream_t stream) {
    constexpr int kSmem = WsLayout::kBytes;
    auto kern = kda_fwd_tc_kernel<GATE_HEAD, FE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    TcMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_tile_maps(&maps, a, GATE_HEAD)) return cudaErrorInvalidValue;
    const dim3 grid(1, a.H_v, a.N);
    kern<<<grid, 384, kSmem, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t stream) {
    if (fe_any(a))
        return a.gate_per_head ? launch_tc<true, true>(a, stream) : launch_tc<false, true>(a, stream);
    return a.gate_per_head ? launch_tc<true, false>(a, stream) : launch_tc<false, false>(a, stream);
}

}  // namespace kda
