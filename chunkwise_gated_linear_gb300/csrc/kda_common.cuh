// Shared pieces of the CUDA path: launch parameters, device error word, and thin
// inline-PTX wrappers (cp.async, ldmatrix, bf16 mma.sync, exp2).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk (the only chunk length supported)
constexpr long long kDefaultWaitCycles = 1ll << 31;  // bounded waits inside kernels: about one second

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
    long long wait_cycles;      // limit of the one-CTA-per-unit kernel's bounded waits (SM cycles)
    // Fused front-end, read only by the kernels that apply it in their staging:
    int fe_qk_l2norm;           // q, k divided per (token, key head) by sqrt(sum of squares + 1e-6)
    int fe_beta_sigmoid;        // beta holds logits b: sigmoid(b) is used
    const float *fe_A_log;      // non-null: g holds the pre-activation a, and
                                //   g = -exp(A_log[h]) * softplus(a + dt_bias) is used
    const float *fe_dt_bias;    // [H_v] (per-head gate) or [H_v][d_k] (per-channel), or null
};

// True when any part of the front-end is switched on.
__host__ __device__ __forceinline__ bool fe_any(const FwdArgs &a) {
    return a.fe_qk_l2norm || a.fe_beta_sigmoid || a.fe_A_log != nullptr;
}

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

// ---- front-end arithmetic ("Gated DeltaNet": the model's gate and write strength, and the
// recurrent kernel's in-kernel q/k normalisation), from CUDA's own expf / log1pf -----------
constexpr float kL2NormEps = 1e-6f;  // added to the sum of squares, inside the square root

// log(1 + e^x); above 20 the correction e^-x is below half an ulp of x
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
// 1 / (1 + e^-b)
__device__ __forceinline__ float sigmoid_f(float b) { return 1.f / (1.f + expf(-b)); }
// natural-log gate from the pre-activation: -exp(A_log) * softplus(a + dt_bias), with
// negA = -exp(A_log) taken once per head
__device__ __forceinline__ float gate_f(float negA, float a, float bias) { return negA * softplus_f(a + bias); }

// Stream-ordered scratch: the library's memory pool of device `dev` (kept between calls).
cudaError_t scratch_pool(int dev, cudaMemPool_t *out);

}  // namespace kda
