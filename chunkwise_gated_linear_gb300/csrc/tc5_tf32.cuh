// tf32 tensor-core products and 3-D tensor copies for the backward kernels (kda_bwd.cu),
// beside the bf16 layer in tc5.cuh: the same descriptors and layouts, 32-bit elements.
#pragma once

#include <cstdint>

#include "tc5.cuh"

namespace kda {
namespace tc5 {

// ---- instruction descriptor: tf32 x tf32 -> fp32, dense, both operands K-major ----------
// (the tf32 kind reads shared-memory operands K-major only; an A operand in TMEM holds one
// element per 32-bit column)
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                          // D format: f32
           | (2u << 7)                        // A format: tf32
           | (2u << 10)                       // B format: tf32
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A[tmem] * B[smem], tf32 (K = 8 per instruction); issued by one thread.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// 3-D tiled load global -> shared, completion counted on an mbarrier (x innermost).
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace tc5
}  // namespace kda
