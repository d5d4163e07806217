// Helpers shared by the tcgen05 kernels for d_k = d_v = 128: tile tensor maps, tf32
// mma.sync for the triangular solve, operand descriptors of 128-byte swizzled tiles,
// TMEM read-back, named barriers and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "tc5.cuh"

namespace kda {
namespace tcu {

using namespace tc5;

constexpr int LDF = 68;                       // fp32 row stride of the 64 x 64 L and T tiles
constexpr long long kWaitCycles = kDefaultWaitCycles;  // bounded waits: about one second

// Tensor maps of the per-chunk tiles (TMA): q, k [tokens][H_k*128] bf16 (box 128 x 64),
// v [tokens][H_v*128] bf16 (box 64 x 64, 128-byte swizzle), g [tokens][H_v*128] fp32 (box 128 x 64).
struct TcMaps {
    CUtensorMap q, k, v, g;
    CUtensorMap o;  // o [tokens][H_v*128] bf16 (box 128 x 64), written by the persistent kernel only
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

// ---- front-end arithmetic: one special-function op per value, the rest on the FMA pipe ----
// log(1 + t) for t in [0, 1] as t P(t), P a degree-7 least-squares fit of log(1 + t) / t on
// Chebyshev nodes of [0, 1] (fit_log1p.py beside this file; worst relative error 2.2e-7).
__device__ __forceinline__ float log1p_01(float t) {
    float p = -8.574675769e-03f;
    p = fmaf(p, t, 4.421419278e-02f);
    p = fmaf(p, t, -1.078536808e-01f);
    p = fmaf(p, t, 1.775702387e-01f);
    p = fmaf(p, t, -2.449961156e-01f);
    p = fmaf(p, t, 3.327617645e-01f);
    p = fmaf(p, t, -4.999744892e-01f);
    p = fmaf(p, t, 9.999998212e-01f);
    return p * t;
}
// softplus(x) = max(x, 0) + log(1 + e^-|x|), the exponential on the special-function unit
__device__ __forceinline__ float softplus_fast(float x) { return fmaxf(x, 0.f) + log1p_01(ex2(-fabsf(x) * kLog2e)); }
// 1 / (1 + e^-b)
__device__ __forceinline__ float sigmoid_fast(float b) { return __fdividef(1.f, 1.f + ex2(-b * kLog2e)); }

// Front-end norms of a chunk's raw Q and K tiles (64 rows each, row-major bf16, 256 B per
// row): rn[t] = scale / sqrt(|q_t|^2 + 1e-6), rn[64 + t] = 1 / sqrt(|k_t|^2 + 1e-6). Warp w of
// the 8 calling warps (pw = 0..7) sums rows 16 w .. 16 w + 15 of [Q; K]: in step i lane l reads the 16-byte
// chunk l & 15 of row 2 i + (l >> 4) (a quarter-warp reads 128 contiguous bytes), then the
// eight partial sums of each half-warp are reduced across its 16 lanes by halving, so that
// lane l ends with the sum of row 2 (l >> 1 & 7) + (l >> 4).
__device__ __forceinline__ void qk_row_norms(const unsigned char *rq, const unsigned char *rk, float *rn, int pw,
                                             int lane, float scale) {
    const unsigned char *base = pw < 4 ? rq + pw * 4096 : rk + (pw - 4) * 4096;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 w = *reinterpret_cast<const uint4 *>(base + (2 * i + (lane >> 4)) * 256 + (lane & 15) * 16);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(ws[j] << 16), hi = __uint_as_float(ws[j] & 0xffff0000u);
            acc = fmaf(lo, lo, acc);
            acc = fmaf(hi, hi, acc);
        }
        v[i] = acc;
    }
    // halving: after the step across lane bit 3, v[k] is row index 4 b3 + k; bit 2: 4 b3 + 2 b2 + k;
    // bit 1: 4 b3 + 2 b2 + b1; bit 0: both lanes of a pair hold the full sum
    const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = b3 ? v[k] : v[k + 4], keep = b3 ? v[k + 4] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = b2 ? v[k] : v[k + 2], keep = b2 ? v[k + 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const float send = b1 ? v[0] : v[1], keep = b1 ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    if ((lane & 1) == 0) {
        const int row = 16 * pw + 2 * ((lane >> 1) & 7) + (lane >> 4);  // 0..127 over [Q; K]
        rn[row] = (pw < 4 ? scale : 1.f) * rsqrtf(v[0] + kL2NormEps);
    }
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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bar_named(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// OR of `v` over the `count` threads of named barrier `id` (all of them take the same branch).
__device__ __forceinline__ bool bar_or(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t"
        "}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---- host: tensor maps ------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
inline bool encode_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t rows,
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

// The q, k, v (and, for per-channel gates, g) tile maps of one call.
inline bool encode_tile_maps(TcMaps *maps, const FwdArgs &a, bool gate_per_head) {
    const uint64_t rows = a.cu_seqlens ? (uint64_t)a.T : (uint64_t)a.N * (uint64_t)a.T;
    if (rows == 0) return true;
    bool ok = encode_map(&maps->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, (uint64_t)a.H_k * 128, rows, 2, 128,
                         CU_TENSOR_MAP_SWIZZLE_NONE) &&
              encode_map(&maps->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k, (uint64_t)a.H_k * 128, rows, 2, 128,
                         CU_TENSOR_MAP_SWIZZLE_NONE) &&
              encode_map(&maps->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.v, (uint64_t)a.H_v * 128, rows, 2, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && !gate_per_head)
        ok = encode_map(&maps->g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.g, (uint64_t)a.H_v * 128, rows, 4, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    return ok;
}

// The output map of the persistent kernel (box 128 x 64, no swizzle: 256-byte rows).
inline bool encode_o_map(TcMaps *maps, const FwdArgs &a) {
    const uint64_t rows = a.cu_seqlens ? (uint64_t)a.T : (uint64_t)a.N * (uint64_t)a.T;
    if (rows == 0) return true;
    return encode_map(&maps->o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.o, (uint64_t)a.H_v * 128, rows, 2, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace tcu
}  // namespace kda
