// Shared pieces of the CUDA path: launch parameters, device error word, and thin
// inline-PTX wrappers (cp.async, ldmatrix, bf16 mma.sync, exp2).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk (the only chunk length supported)

// Device error bits, the same values as KDA_DEVICE_ERR_* in kda.h.
constexpr unsigned int kDeviceErrSeqlens = 1u;
constexpr unsigned int kDeviceErrTimeout = 2u;

// Everything a forward kernel needs, resolved on the host.
struct FwdArgs {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    void *o;
    float *ht;
    const int32_t *cu_seqlens;  // device offsets, or nullptr for fixed-length batches
    int N;                      // number of sequences
    int T;                      // tokens per sequence (fixed) or total tokens (packed)
    int H_k, H_v, d_k, d_v;
    int group;                  // H_v / H_k
    float scale;
    int gate_per_head;
    int decay_only;             // beta == nullptr: S <- Diag(a_t) S + k_t v_t^T (no erase)
    unsigned int *err;          // device error word of the current device (KDA_DEVICE_ERR_*)
};

// Sequence bounds of sequence n; returns false (and raises the error bit) when the
// offsets are malformed.
__device__ __forceinline__ bool seq_bounds(const FwdArgs &a, int n, int64_t &bos, int &len) {
    if (a.cu_seqlens == nullptr) {
        bos = (int64_t)n * a.T;
        len = a.T;
        return true;
    }
    const int s = a.cu_seqlens[n], e = a.cu_seqlens[n + 1];
    if (s < 0 || e < s || e > a.T) {
        if (threadIdx.x == 0) atomicOr(a.err, kDeviceErrSeqlens);
        return false;
    }
    bos = s;
    len = e - s;
    return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; bytes past src_bytes (0 or 16) are zero-filled.
__device__ __forceinline__ void cp_async_16(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(src_bytes));
}
// 4-byte global->shared copy; zero-filled when src_bytes is 0.
__device__ __forceinline__ void cp_async_4(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace kda
