/*
 * kda.h — C ABI of the chunkwise forward pass of the gated delta rule with a
 * per-channel gate (Kimi Delta Attention, KDA), for NVIDIA GB300 (sm_103a).
 *
 * The operation ("TileLang 实战：KDA 从零到一–Kimi Delta Attention", §0 and §3.1):
 * for every sequence n and value head h, with state S in R^{d_k x d_v} (the transposed
 * layout the kernels keep; "TileLang 实战：KDA 从零到一--标量衰减", §4.0),
 *
 *     S <- Diag(exp(g_t)) S                     decay, before the erase read
 *     u <- beta_t (v_t - S^T k_t)               erase (delta rule)
 *     S <- S + k_t u^T                          write
 *     o_t = scale * S^T q_t
 *
 * i.e. S_t = S_{t-1} Diag(a_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T in the paper
 * layout, a_t = exp(g_t). The scalar-gate Gated DeltaNet ("Gated DeltaNet", section
 * "DeltaNet 与 Gated Delta Rule") is the case of one gate per (token, head) broadcast over
 * the d_k channels. The library computes it chunk by chunk (C tokens per chunk), with
 * the per-chunk equations of "RNN的复兴04:线性注意力并行计算DPLR", §5.3.5: a chunk-local
 * cumulative log-gate, the separable decay-weighted Gram matrix, the UT-transform
 * triangular solve giving the WY factors W and U, the serial chunk-to-chunk state step
 * and the chunk-parallel output. The result equals the token recurrence up to rounding.
 *
 * Layouts (all pointers are DEVICE pointers; tensors are contiguous, token-major):
 *   q, k   [B, T, H_k, d_k]     bf16 (kda_chunk_fwd) or fp32 (kda_chunk_fwd_f32)
 *   v, o   [B, T, H_v, d_v]     same dtype as q
 *   g      [B, T, H_v, d_k]     fp32 natural-log gates (g <= 0), per token, NOT cumsummed;
 *                               [B, T, H_v] fp32 in the per-head gate mode of _ex
 *   beta   [B, T, H_v]          fp32
 *   h0, ht [N, H_v, d_k, d_v]   fp32 initial / final state, N = number of sequences
 *   Value head h reads key head h / (H_v / H_k) (grouped heads; H_v % H_k == 0).
 *
 * Varlen packing ("Gated DeltaNet", chunk_local_cumsum: cu_seqlens and chunk indices):
 *   if cu_seqlens != NULL the tensors hold N = B sequences packed along the token axis
 *   with a physical batch of 1 ([1, T, ...], T = total tokens). cu_seqlens is a DEVICE
 *   int32 array of B + 1 non-decreasing offsets, cu_seqlens[0] = 0 and cu_seqlens[B] = T.
 *   Chunks never span two sequences. Its contents are read on the device only: a
 *   malformed array is a precondition violation; the kernels skip a sequence whose
 *   offsets are out of order or out of [0, T] and raise KDA_DEVICE_ERR_SEQLENS, which
 *   kda_get_device_error reports.
 *   if cu_seqlens == NULL the batch holds B sequences of T tokens each (N = B).
 *
 * NULL conventions: h0 == NULL means a zero initial state; ht == NULL means the final
 *   state is not written; beta == NULL selects the decay-only recurrence (gated linear
 *   attention: no erase, unit write; "07 · linear 路线（二）：衰减机制的演进", §1, and the
 *   KDA page, §3.4):
 *       S <- Diag(exp(g_t)) S + k_t v_t^T,   o_t = scale * S^T q_t
 *   (GLA with a per-channel gate; RetNet, Lightning or Mamba-2 SSD with one gate per
 *   head). q, k, v, g and o are required unless T == 0.
 *
 * Sizes supported: d_k, d_v in {64, 128}; C == 64; B >= 1; T >= 0; H_k >= 1; H_v >= 1.
 *   T == 0 (or empty sequences) is valid: no o rows, ht = h0 (or 0).
 *
 * Ownership and semantics: the caller owns every buffer; the library allocates no
 *   memory except the stream-ordered scratch of the persistent kernel (see
 *   KDA_FLAG_ONE_CTA_PER_UNIT), which it frees on the same stream. Calls are asynchronous on `stream` (no host synchronisation). o and ht are
 *   fully overwritten; o and ht must not alias any input. The same inputs give bitwise
 *   equal outputs (no atomics on outputs). The entry points are thread-safe.
 *
 * Errors: 0 (KDA_OK) on success, otherwise a negative status; nothing is launched when
 *   a status other than KDA_OK or KDA_ERR_CUDA is returned.
 */
#ifndef KDA_H
#define KDA_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_OK 0
#define KDA_ERR_INVALID_ARG (-1) /* a required pointer is NULL or a size is out of range */
#define KDA_ERR_UNSUPPORTED (-2) /* d_k, d_v, C, dtype or gate mode not supported */
#define KDA_ERR_ALIGNMENT (-3)   /* a tensor pointer is not 16-byte aligned */
#define KDA_ERR_CUDA (-4)        /* a CUDA call failed; kda_status_string says which */

#define KDA_DTYPE_BF16 0
#define KDA_DTYPE_F32 1

#define KDA_GATE_PER_CHANNEL 0 /* g [.., H_v, d_k] */
#define KDA_GATE_PER_HEAD 1    /* g [.., H_v], one gate per (token, value head) */

/* Device-side error bits returned by kda_get_device_error. */
#define KDA_DEVICE_ERR_SEQLENS 1 /* cu_seqlens out of order or out of [0, T] */
#define KDA_DEVICE_ERR_TIMEOUT 2 /* a bounded wait inside a kernel gave up (about 1 s) */

/*
 * kda_chunk_fwd — bf16 q, k, v, o with fp32 accumulation.
 *
 * q, k: [B, T, H_k, d_k] bf16; v: [B, T, H_v, d_v] bf16; g: [B, T, H_v, d_k] fp32 log
 * gates; beta: [B, T, H_v] fp32; h0: [N, H_v, d_k, d_v] fp32 or NULL; o: [B, T, H_v, d_v]
 * bf16 (written, rounded to nearest even); ht: [N, H_v, d_k, d_v] fp32 or NULL (written);
 * B: batch (or number of packed sequences when cu_seqlens != NULL); T: tokens per
 * sequence (or total tokens when packed); C: chunk length, must be 64; scale: multiplies
 * the output only (commonly d_k^-1/2); cu_seqlens: device int32 [B + 1] or NULL;
 * stream: CUDA stream the work is ordered on (0 = the legacy default stream).
 */
int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                  const float *beta, const float *h0, void *o, float *ht, int B, int T,
                  int H_k, int H_v, int d_k, int d_v, int C, float scale,
                  const int32_t *cu_seqlens, cudaStream_t stream);

/*
 * kda_chunk_fwd_f32 — the same operation and argument list with fp32 q, k, v and o,
 * computed in fp32 throughout (no bf16 rounding anywhere).
 */
int kda_chunk_fwd_f32(const float *q, const float *k, const float *v, const float *g,
                      const float *beta, const float *h0, float *o, float *ht, int B,
                      int T, int H_k, int H_v, int d_k, int d_v, int C, float scale,
                      const int32_t *cu_seqlens, cudaStream_t stream);

/* Every argument of the two calls above, plus the dtype and the gate mode. */
typedef struct kda_fwd_params {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    void *o;
    float *ht;
    int B, T, H_k, H_v, d_k, d_v, C;
    float scale;
    const int32_t *cu_seqlens;
    int dtype;     /* KDA_DTYPE_BF16 or KDA_DTYPE_F32 */
    int gate_mode; /* KDA_GATE_PER_CHANNEL or KDA_GATE_PER_HEAD */
    int flags;     /* 0, or KDA_FLAG_ONE_CTA_PER_UNIT and / or KDA_FLAG_UNFUSED_FRONTEND */
} kda_fwd_params;

/*
 * flags of kda_fwd_params. With d_k = d_v = 128 in bf16 and at most half as many
 * (sequence, value head) units as the device has SMs (and at most 76 units), the library
 * runs a persistent kernel that occupies every SM: the chunk-local factors of all units
 * are built in parallel on the SMs the units leave free and handed to one SM per unit
 * that runs the serial state step. It allocates about 220 KiB per unit of stream-ordered
 * scratch from a memory pool the library owns (one per device). The pool keeps up to
 * 64 MiB reserved between calls, enough for this scratch, and returns anything above that
 * (the backward's scratch, for instance) to the device when the device, a stream or an
 * event is next synchronised. KDA_FLAG_ONE_CTA_PER_UNIT
 * selects the kernel with one CTA per unit instead, which allocates nothing and leaves
 * the other SMs free for concurrent work. Both give the same result up to rounding.
 */
#define KDA_FLAG_ONE_CTA_PER_UNIT 1
/* With a front-end (kda_chunk_fwd_fused, kda_recurrent_fwd_fused): run it as a separate
 * pass into scratch even where the selected kernel can apply it itself (for comparison;
 * the result agrees up to rounding). Ignored by the other entry points. */
#define KDA_FLAG_UNFUSED_FRONTEND 2
/* Test aid for the failure path: the one-CTA-per-unit kernel is used (as with
 * KDA_FLAG_ONE_CTA_PER_UNIT, bf16 with d_k = d_v = 128), its waits give up after about 1,000
 * SM cycles instead of about one second, and its serial warps first wait on a barrier phase
 * that nothing completes, so that the wait runs out; the kernel then drains its copies and
 * tensor-core work, frees its tensor memory, leaves its outputs undefined and raises
 * KDA_DEVICE_ERR_TIMEOUT. Read by kda_chunk_fwd_ex and kda_chunk_fwd_fused; the recurrent
 * entry points accept and ignore it. */
#define KDA_FLAG_DEBUG_SHORT_WAITS 4

/*
 * kda_chunk_fwd_ex — the general entry point: dtype and gate mode chosen by the struct.
 * The per-head gate mode reads g as [B, T, H_v] (the scalar-gate Gated DeltaNet), so the
 * gate costs 4 bytes per (token, head) instead of 4 * d_k.
 */
int kda_chunk_fwd_ex(const kda_fwd_params *p, cudaStream_t stream);

/*
 * kda_chunk_fwd_noalloc — the arguments and result of kda_chunk_fwd, computed by the
 * persistent kernel with its scratch (the ring of chunk slots and its flags) in one
 * fixed array of device memory inside the library: 9,568,256 + 4,352 bytes, room for 16
 * (sequence, value head) units. The pages have no counterpart: it exists for callers
 * that must not allocate (nothing is allocated, on the device or the host) — for example a
 * process that hands all device memory to its own allocator at start-up, where an
 * allocation inside the library could fail in the middle of a run, or one that must keep
 * its peak device memory fixed and known in advance.
 *
 * Supported: bf16, d_k = d_v = 128, C = 64, at most 16 units (B * H_v, or N * H_v with
 * cu_seqlens) and at most half as many units as the device has SMs; anything else returns
 * KDA_ERR_UNSUPPORTED with nothing launched. The unit-count and head-size checks are made
 * on the host before any CUDA call; the checks of the SM count and of cooperative launch
 * follow cudaGetDevice and cudaDeviceGetAttribute. Each call first zeroes the flag words of
 * the array with cudaMemsetAsync on `stream`; the slots need no clearing. The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) and the device error
 * word, and later calls reuse both: they assume the device's primary context is not reset
 * (cudaDeviceReset) while the library stays loaded.
 *
 * The array is shared by every call of this entry point on a device: calls that overlap
 * in time (on any stream, from any thread) race on it and give wrong results. The caller
 * must order them (same stream, or events). Other entry points do not use the array.
 * Errors and the device error word are as for kda_chunk_fwd.
 */
int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, void *o, float *ht, int B,
                          int T, int H_k, int H_v, int d_k, int d_v, int C, float scale,
                          const int32_t *cu_seqlens, cudaStream_t stream);

/*
 * kda_recurrent_fwd — the same operation computed token by token (the recurrent form:
 * "TileLang 实战：KDA 从零到一–Kimi Delta Attention", §0, and the recurrent form of
 * "Gated DeltaNet"), for decoding: typically a few tokens per sequence, continuing from a
 * state h0 written by kda_chunk_fwd or by an earlier call. Arguments, layouts, NULL
 * conventions (beta == NULL: decay-only) and errors as kda_chunk_fwd, without C.
 * ht may equal h0: the state is then updated in place (each part of it is read before it
 * is written by the same thread). bf16 q/k/v/o; d_k, d_v in {64, 128}.
 */
int kda_recurrent_fwd(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, const float *h0, void *o, float *ht, int B, int T,
                      int H_k, int H_v, int d_k, int d_v, float scale,
                      const int32_t *cu_seqlens, cudaStream_t stream);

/* kda_recurrent_fwd with the dtype and gate mode of the struct (its C is ignored). */
int kda_recurrent_fwd_ex(const kda_fwd_params *p, cudaStream_t stream);

/*
 * The fused front-end: the per-token preparation that the Gated DeltaNet model applies to
 * its projections before the recurrence ("Gated DeltaNet", section "模型调用方式：Qwen3.5
 * GatedDeltaNet", and the recurrent kernel's in-kernel variants in "Recurrent 算法代码解析").
 * Each part is independent; a zeroed struct switches everything off.
 *
 *   qk_l2norm     nonzero: q and k are divided, per (token, key head), by
 *                 sqrt(sum over d_k of x^2 + 1e-6) before use; the scale then multiplies
 *                 the normalised q.
 *   beta_sigmoid  nonzero: the beta tensor holds logits b and beta = 1 / (1 + exp(-b)) is
 *                 used. Requires beta != NULL.
 *   A_log         non-NULL: the g tensor holds the gate pre-activation a (same layout as g)
 *                 and the log gate g = -exp(A_log[h]) * softplus(a + dt_bias) is used.
 *                 A_log: [H_v] fp32, device, 16-byte aligned.
 *   dt_bias       with A_log: [H_v] fp32 (per-head gate) or [H_v, d_k] fp32 (per-channel
 *                 gate: one bias per value head and channel), device, 16-byte aligned; NULL
 *                 means no bias. Must be NULL when A_log is NULL.
 *
 * The input tensors are only read; nothing is written back to them.
 */
typedef struct kda_frontend {
    int qk_l2norm;
    int beta_sigmoid;
    const float *A_log;
    const float *dt_bias;
} kda_frontend;

/*
 * kda_chunk_fwd_fused — kda_chunk_fwd_ex with the front-end `fe` applied to its inputs
 * (fe == NULL: exactly kda_chunk_fwd_ex). With bf16 and d_k = d_v = 128 the kernels apply it
 * while staging each chunk, so q, k, g and beta are read once; the d = 64 and fp32 kernels
 * get it as a separate pass that writes the prepared q and k (in the input dtype),
 * g and beta (fp32) to stream-ordered scratch from the library's pool (freed on the same
 * stream), about 2 * T * H_k * d_k * elem + T * H_v * (d_k or 1) * 4 + T * H_v * 4 bytes.
 * Errors as kda_chunk_fwd_ex, and KDA_ERR_INVALID_ARG for beta_sigmoid with beta == NULL or
 * dt_bias without A_log, KDA_ERR_ALIGNMENT for A_log or dt_bias not 16-byte aligned.
 */
int kda_chunk_fwd_fused(const kda_fwd_params *p, const kda_frontend *fe, cudaStream_t stream);

/* kda_recurrent_fwd_ex with the front-end `fe` (applied inside the recurrent kernel, or as a
 * separate pass with KDA_FLAG_UNFUSED_FRONTEND). */
int kda_recurrent_fwd_fused(const kda_fwd_params *p, const kda_frontend *fe, cudaStream_t stream);

/*
 * kda_chunk_bwd — the backward pass: gradients of L = sum(dO * o) + sum(dht * ht) with
 * respect to q, k, v, g, beta and h0, for the forward pass that kda_chunk_fwd_ex computes
 * with the same arguments ("Gated DeltaNet", "反向传播：状态伴随与三角变换梯度": the state
 * adjoint runs backwards from dht through the chunks and the WY factors' gradients go back
 * through the triangular inverse). The chunk factors and the chunk-entry states are
 * recomputed from the inputs; all arithmetic is fp32.
 *
 * Forward arguments (q, k, v, g, beta, h0, sizes, scale, cu_seqlens, dtype, gate_mode) as
 * in kda_fwd_params, and (all device pointers, contiguous, 16-byte aligned):
 *   dO     [B, T, H_v, d_v], the dtype of q
 *   dht    [N, H_v, d_k, d_v] fp32, or NULL (no gradient reaches the final state)
 *   dq, dk [B, T, H_k, d_k], dv [B, T, H_v, d_v], the dtype of q (dq and dk sum the value
 *          heads that share a key head)
 *   dg     the shape of g (fp32): gradient of the natural-log gates
 *   dbeta  [B, T, H_v] fp32; must be NULL when beta is NULL (decay-only)
 *   dh0    [N, H_v, d_k, d_v] fp32, or NULL when not wanted (also when h0 is NULL: it is
 *          then the gradient with respect to the zero initial state)
 * Malformed cu_seqlens (decreasing, negative, or past T) are caught on the device: the
 * sequence is skipped, its outputs are left undefined and KDA_DEVICE_ERR_SEQLENS is raised.
 * Outputs are fully overwritten. Scratch: about 540 KB per (64-token chunk, value head)
 * at d = 128 (the chunk factors, entry states and their adjoints; about 700 KB for bf16
 * inputs with d_k = d_v = 128 and beta, whose tensor-core path also keeps transposed copies
 * of the factors), plus fp32 accumulators
 * of dq and dk for bf16 outputs, all stream-ordered from the library's pool and freed on
 * the same stream; the pool gives it back to the device at the next synchronisation (it
 * keeps at most 64 MiB between calls). Errors as kda_chunk_fwd_ex (flags must be 0).
 */
typedef struct kda_bwd_params {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    const void *dO;
    const float *dht;
    void *dq, *dk, *dv;
    float *dg, *dbeta, *dh0;
    int B, T, H_k, H_v, d_k, d_v, C;
    float scale;
    const int32_t *cu_seqlens;
    int dtype;     /* KDA_DTYPE_BF16 or KDA_DTYPE_F32 */
    int gate_mode; /* KDA_GATE_PER_CHANNEL or KDA_GATE_PER_HEAD */
    int flags;     /* 0 */
} kda_bwd_params;

int kda_chunk_bwd(const kda_bwd_params *p, cudaStream_t stream);

/* A static, human-readable description of a status (and of the last CUDA error for
 * KDA_ERR_CUDA on this thread). */
const char *kda_status_string(int status);

/*
 * kda_get_device_error — synchronises `stream`, returns the device-side error bits
 * (KDA_DEVICE_ERR_*) raised by kernels of this library on the current device since the
 * last call, and clears them. Returns KDA_ERR_CUDA if the query itself fails.
 */
int kda_get_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
