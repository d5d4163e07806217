// Arguments of the backward kernels (kda_bwd.cu), resolved on the host by kda_api.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kda {

struct BwdArgs {
    const void *q, *k, *v;     // forward inputs (bf16 or fp32, the dtype of the call)
    const float *g, *beta, *h0;
    const void *dO;            // [tokens][H_v][d_v], the dtype of q
    const float *dht;          // [N][H_v][d_k][d_v] or nullptr
    void *dq, *dk, *dv;        // outputs, the dtype of q
    float *dg, *dbeta, *dh0;   // fp32 outputs (dbeta nullptr without beta, dh0 optional)
    const int32_t *cu_seqlens; // packed sequences, or nullptr for fixed-length batches
    int N, T, H_k, H_v, d_k, d_v, group;
    float scale;
    int gate_per_head, decay_only;
    float *scratch;            // per-chunk factors (set by the launcher)
    float *dq_acc, *dk_acc;    // fp32 accumulators of dq, dk (set by the launcher)
    int direct_qk;             // one value head per key head: dq, dk written directly
    int tc;                    // the tcgen05 gradient kernel runs: prep and the adjoint scan
                               // also write the transposed factors it reads
    unsigned int *err;         // device error word (KDA_DEVICE_ERR_*)
};

// Runs the backward pass on `stream` with stream-ordered scratch from the library's pool.
cudaError_t launch_bwd(const BwdArgs &a, bool f32, cudaStream_t stream);

}  // namespace kda
