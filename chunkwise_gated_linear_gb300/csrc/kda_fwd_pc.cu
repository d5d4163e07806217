// Chunkwise KDA forward for d_k = d_v = 128, bf16 operands: a persistent kernel in which
// some CTAs (producers) build the per-chunk factors of every (sequence, value head) unit
// in parallel, and one CTA per unit (its consumer) runs the serial chunk-to-chunk step.
//
// The chunk equations ("RNN的复兴04:线性注意力并行计算DPLR", §5.3.5; "TileLang 实战：KDA
// 从零到一–Kimi Delta Attention", §3.3) split into a part that depends only on the chunk's
// own inputs and the state recurrence. Only the second is serial, so with fewer units than
// SMs the first runs on the SMs that would otherwise idle:
//
//   producer CTA, one chunk job after another, two stages working on consecutive jobs:
//     front (warps 0-7)   TMA Q, K, G; gamma = chunk-local cumulative log2 gate;
//                         Qp = Q e^gamma, Kp = K e^gamma, Km = K e^-gamma
//                         (transposed, bf16; the scale is applied to the output);
//                         Gram D_G = [Qp; Kp] Km^T -> Aqk (lower), L = diag(beta) M (strict)
//     back  (warps 8-15)  T = (I + L)^-1 (16x16 diagonal blocks by substitution, the rest
//                         on tf32 mma.sync); D_W = Kp^T (T diag beta)^T, D_U = V^T (T diag beta)^T
//     -> the chunk's slot in a per-unit ring in global memory: W^T, Qp^T, Km^T, Aqk (bf16,
//        in the consumer's 128-byte swizzled shared-memory image), U^T (bf16), e^gamma_n.
//   consumer CTA (unit u), TMEM holds R [d_v x d_k] fp32 = S_c^T, thread = d_v row (Kbar =
//   Km Diag(e^gamma_n) is never formed: S_{c+1}^T = (S_c^T + Vt^T Km) Diag(e^gamma_n)):
//     bulk copies bring each slot into shared memory (three buffers, up to three chunks
//     ahead of the serial step), then
//     D_X = S_c^T [W^T | Qp^T] (A: the bf16 copy of S_c^T);
//     Vt^T = U^T - D_X[:, :64];  O^T = D_X[:, 64:] + Vt^T Aqk^T;  R += Vt^T Km;
//     R <- R Diag(e^gamma_n) = S_{c+1}^T, with its bf16 copy for the next chunk.
//   The MMAs are issued by one warp, the output leaves through an epilogue warp group.
//
// Hand-offs through global memory use per-slot sequence numbers: a producer publishes
// chunk c of unit u by a release store of c + 1 into ready[u][c % R] after its writes;
// the consumer releases the slot by storing c + 1 into done[u] once the bulk copy has
// landed. Producers take jobs in (chunk, unit) order (claimed from a global counter when
// the units have equal lengths), so the oldest unfinished job never waits on a later one. The launch is cooperative (every CTA resident). Every
// wait is bounded (about one second) and watches a global abort word, so a failure
// anywhere ends all CTAs with KDA_DEVICE_ERR_TIMEOUT.
#include <algorithm>
#include <cstring>

#include "tc_util.cuh"

namespace kda {

namespace {

using bf16 = __nv_bfloat16;
using namespace tc5;
using namespace tcu;

constexpr int kMaxUnits = 76;       // units served by one launch (at most half the SMs)
constexpr int kRing = 8;            // ring slots per unit, at least (a launch argument)
constexpr int kThreads = 512;

// Slot image (global ring and consumer shared memory). [d][tok] tiles hold one row per
// d_k channel and 64 tokens per 128-byte row (one swizzle atom).
struct Slot {
    static constexpr int oWT = 0;       // W^T [d][tok] bf16     } adjacent: one N = 128
    static constexpr int oQP = 16384;   // Qp^T [d][tok] bf16    } MN-major B operand
    static constexpr int oKM = 32768;   // Km^T [d][tok] bf16 (K-major B)
    static constexpr int oAQ = 49152;   // Aqk [tok][tok'] bf16 (K-major B)
    static constexpr int oEG = 57344;   // e^gamma_n [128] fp32
    static constexpr int oU = 57856;    // U^T as bf16 token pairs: u32 [tok / 2][d_v]
    static constexpr int kBytes = 74240;
    static constexpr int kStride = 74752;  // 1024-byte multiple
    // the front stage writes [oQP, oU) as one image, the back stage W^T and U^T
    static constexpr int kFrontBytes = oU - oQP;
};

// Producer shared memory (offsets from a 1024-byte aligned base).
struct Prod {
    static constexpr int oRQ = 0;          // raw Q [64 tok][128] bf16 row-major
    static constexpr int oRK = 16384;      // raw K
    static constexpr int oG = 32768;       // raw G fp32 [64][128]
    static constexpr int oIMG = 65536;     // the front part of the slot image (Slot::oQP ..
                                           // Slot::oU); its Qp^T is also the Gram A operand
    static constexpr int oQP = oIMG;
    static constexpr int oKM = oIMG + (Slot::oKM - Slot::oQP);  // also the Gram's B operand
    static constexpr int oAQ = oIMG + (Slot::oAQ - Slot::oQP);
    static constexpr int oEG = oIMG + (Slot::oEG - Slot::oQP);
    static constexpr int oKP0 = 107520;    // Kp^T [d][tok], hand-off slots 0 / 1 (Gram A atom 1);
                                           // then U^T staging of the back stage
    static constexpr int oKP1 = 123904;
    static constexpr int oL1 = 140288;     // L fp32 [64][68] (front -> back), job parity 1
    static constexpr int oL0 = 157696;     // the same, job parity 0
    static constexpr int oT = 175104;      // T fp32 [64][68]; then W^T staging [d][tok] bf16
    static constexpr int oTB = 192512;     // T_beta [tok][tok'] bf16 (K-major B)
    static constexpr int oRV = 200704;     // raw V [2 atoms (d_v)][64 tok][128 B]
    static constexpr int oBF0 = 217088;    // beta as loaded, job parity 0 / 1
    static constexpr int oBF1 = 217344;
    static constexpr int oBH0 = 217600;    // beta handed to the back stage, job parity 0 / 1
    static constexpr int oBH1 = 217856;
    static constexpr int oGh0 = 218112;    // per-head gates, job parity 0 / 1
    static constexpr int oGh1 = 218368;
    static constexpr int oTot = 218624;    // [4][128] fp32 partial gate sums
    static constexpr int oPS = 220672;     // solve scratch, 8 warps x 16x8 fp32
    static constexpr int oRN = oPS + 4096; // front-end: 1 / |q_t| [64], 1 / |k_t| [64]
    static constexpr int kEnd = oRN + 512;
};
static_assert(Prod::oEG + 512 <= Prod::oKP0, "image overlaps");
static_assert(Prod::oL1 + 64 * 68 * 4 <= Prod::oL0 && Prod::oL0 + 64 * 68 * 4 <= Prod::oT, "L buffers overlap");
static_assert(Prod::oTB % 1024 == 0 && Prod::oRV % 1024 == 0, "swizzled tiles are 1024-byte aligned");
// Consumer shared memory.
struct Cons {
    static constexpr int kBufs = 3;        // slot images in flight: loads have up to two
                                           // chunks of the serial step to land
    static constexpr int kEnd = kBufs * Slot::kStride;
};
// Both roles.
struct Common {
    static constexpr int oBar = Prod::kEnd > Cons::kEnd ? Prod::kEnd : Cons::kEnd;  // mbarriers
    static constexpr int oTmemAddr = oBar + 256;
    static constexpr int oFlag = oTmemAddr + 16;   // CTA abort flag
    static constexpr int oUnits = oFlag + 16;      // UnitInfo [kMaxUnits]
    static constexpr int oSeen = oUnits + 16 * kMaxUnits;  // producer: done[u] last observed
    static constexpr int oJobq = oSeen + 4 * kMaxUnits;    // producer: claimed jobs [4]
    static constexpr int oEGc = oJobq + 16;                // consumer: e^gamma_n of chunks, [2][128] fp32
                                                           // (16-byte aligned: read as float4)
    static constexpr int kEnd = oEGc + 1024;
    static constexpr int kBytes = kEnd + 1024;      // + slack to align the base
};

static_assert(Common::kBytes <= 232448, "shared memory");
static_assert(Common::oEGc % 16 == 0, "float4 reads of the e^gamma_n copies");
static_assert(Slot::kBytes % 128 == 0 && Slot::kStride % 128 == 0, "slots are whole 128-byte lines");

// TMEM columns
constexpr uint32_t tGram = 0, tW = 64, tU = 128, kTmemProd = 256;     // producer
// consumer: D_X / O^T in two buffers (by chunk parity), S^T bf16, Vt^T, S^T fp32
constexpr uint32_t tX0 = 0, tSA = 128, tV = 192, tS = 256, tX1 = 384, kTmemCons = 512;

enum {
    // producer
    B_LQK = 0, B_LG, B_LV,   // TMA tiles: Q and K, G, V
    B_GRAM, B_WMMA,          // MMA completion: Gram, WY
    B_HFULL0, B_HFULL1,      // front -> back hand-off slot 0 / 1 written
    B_HEMPTY0, B_HEMPTY1,    // back -> front: the Kp^T buffer of hand-off slot 0 / 1 is free
    B_LFREE0, B_LFREE1,      // back -> front: L and beta of job parity 0 / 1 consumed by the solve
    B_PZ0, B_PZ1,            // drains after a failure (one per MMA-issuing thread)
    // consumer
    B_FULL0, B_FULL1, B_FULL2,     // slot image in buffer 0 / 1 / 2 landed
    B_EMPTY0, B_EMPTY1, B_EMPTY2,  // buffer 0 / 1 / 2 consumed by the serial step
    B_X, B_R,                // consumer products: D_X, the state update
    B_O0, B_O1,              // the output of D_X buffer 0 / 1 is complete (one barrier per
                             // buffer: each completes again only after the epilogue freed it)
    B_XFREE0, B_XFREE1,      // the output half of D_X buffer 0 / 1 has been read out
    B_CZ,
    kNumBars
};

struct UnitInfo {
    long long bos;
    int len, nch;
};

// Ring and flags in global memory; ready/done/abort start at zero for every launch.
// Each unit's flags have a 128-byte line of their own: a unit's ready words are polled by its
// consumer, its done word by the producers waiting for one of its slots, and lines shared by
// several units would concentrate that polling on a few L2 slices.
constexpr int kFlagLine = 32;  // ints

struct PcArgs {
    unsigned char *ring;   // [U][R] slots of Slot::kStride bytes
    int *ready;            // [U][kFlagLine], R used: c + 1 once chunk c is in slot c % R
    int *done;             // [U][kFlagLine], 1 used: chunks whose slot image has been copied out
    int *abort;            // set by any CTA that gave up
    int *jobs;             // equal-length units: the next job not yet claimed by a producer
    int U, P;              // units (= consumer CTAs), producer CTAs
    int R;                 // ring slots per unit
};

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// 1-D bulk copy global -> shared, completing on an mbarrier of this CTA.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// 1-D bulk copy shared -> global (bulk async-group of the issuing thread).
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the issuing thread's bulk stores have completed (written) / have read their source
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Product of two bf16 pairs, rounded to the nearest bf16 pair.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t x, uint32_t y) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t x, uint32_t y, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(y), "r"(sel));
    return d;
}
// x[e] holds (channel ch, channel ch + 1) of token 8 tc + e; rows ra and rb (ch and ch + 1,
// in either order) of a [d][tok] 128-byte swizzled tile receive the eight tokens as 16 bytes
// each: selector 0x5410 gathers the low halves of a token pair, 0x7632 the high halves.
__device__ __forceinline__ void store_pairs_t(unsigned char *tile, const uint32_t (&x)[8], int ra, int rb, int tc,
                                              uint32_t sel_a, uint32_t sel_b) {
    uint4 A, B;
    A.x = prmt(x[0], x[1], sel_a);
    A.y = prmt(x[2], x[3], sel_a);
    A.z = prmt(x[4], x[5], sel_a);
    A.w = prmt(x[6], x[7], sel_a);
    B.x = prmt(x[0], x[1], sel_b);
    B.y = prmt(x[2], x[3], sel_b);
    B.z = prmt(x[4], x[5], sel_b);
    B.w = prmt(x[6], x[7], sel_b);
    *reinterpret_cast<uint4 *>(tile + sw128(ra, tc)) = A;
    *reinterpret_cast<uint4 *>(tile + sw128(rb, tc)) = B;
}

// Raise the abort word (once) and the device error bit.
__device__ __forceinline__ void raise_abort_w(int *abort_w, unsigned int *err, volatile int *cta_flag) {
    *cta_flag = 1;
    if (atomicExch(abort_w, 1) == 0) atomicOr(err, kDeviceErrTimeout);
}
// Whether another CTA has raised the abort word, read at most once every kAbortPollCycles
// of a wait: the word sits in one L2 line that every waiting thread of the grid would
// otherwise load every few tens of nanoseconds, and that load stream slows every other
// access served by the same L2 slice (the ring flags among them).
constexpr long long kAbortPollCycles = 8192;
__device__ __forceinline__ bool abort_due(long long now, long long &tpoll, int *abort_w) {
    if (now - tpoll < kAbortPollCycles) return false;
    tpoll = now;
    return *(volatile int *)abort_w != 0;
}
// mbarrier phase test that lets the hardware suspend the thread until the phase completes
// (or about `hint_ns` nanoseconds have passed), so that waiting threads take no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// The waits below keep their slow paths out of line: one copy of each loop serves every
// call site, which keeps the kernel's hot code small.
__device__ __noinline__ bool wait_bar_slow(uint64_t *bar, uint32_t parity, volatile int *cta_flag, int *abort_w,
                                           unsigned int *err) {
    const long long t0 = clock64();
    long long tpoll = t0;
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (*cta_flag) return false;
        const long long now = clock64();
        if (abort_due(now, tpoll, abort_w)) {
            *cta_flag = 1;
            return false;
        }
        if (now - t0 > kWaitCycles) {
            raise_abort_w(abort_w, err, cta_flag);
            return false;
        }
    }
    return true;
}
// Bounded wait on an mbarrier phase of this CTA; gives up when this CTA or any other is
// aborting.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *cta_flag, const FwdArgs &a,
                                         const PcArgs &pc) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, cta_flag, pc.abort, a.err);
}
__device__ __noinline__ bool wait_geq_slow(const int *p, int target, volatile int *cta_flag, int *abort_w,
                                           unsigned int *err, int *seen) {
    const long long t0 = clock64();
    long long tpoll = t0;
    unsigned nap = 64u;
    int v;
    while ((v = ld_acquire(p)) < target) {
        if (*cta_flag) return false;
        const long long now = clock64();
        if (abort_due(now, tpoll, abort_w)) {
            *cta_flag = 1;
            return false;
        }
        if (now - t0 > kWaitCycles) {
            raise_abort_w(abort_w, err, cta_flag);
            return false;
        }
        // back off (64 ns doubling to 512 ns): a long wait polls its line less often
        __nanosleep(nap);
        nap = nap < 512u ? 2u * nap : nap;
    }
    if (seen) *seen = v;
    return true;
}
// Bounded wait until the global word *p reaches at least `target` (acquire); the value
// read last goes to *seen.
__device__ __forceinline__ bool wait_geq(const int *p, int target, volatile int *cta_flag, const FwdArgs &a,
                                         const PcArgs &pc, int *seen = nullptr) {
    const int v = ld_acquire(p);
    if (seen) *seen = v;
    if (v >= target) return true;
    return wait_geq_slow(p, target, cta_flag, pc.abort, a.err, seen);
}

// Per-CTA context shared by the roles.
struct Ctx {
    unsigned char *sm;
    uint32_t sbase, tmem;
    uint64_t *bars;
    volatile int *flag;     // this CTA is aborting
    volatile int *stored;   // producer: jobs whose front image is written to the ring
    int *seen;              // producer, thread 0: done[u] as last acquired, per unit
    volatile int *jobq;     // producer, equal-length units: claimed job of ordinal jo at [jo % 4]
    const UnitInfo *units;  // [U]
    int maxc, uniform;      // over the units of this launch
    int p;                  // producer index (producer CTAs)
};

// Bounded wait until the shared-memory counter *p reaches at least `target`.
__device__ __noinline__ bool wait_count_slow(const volatile int *p, int target, volatile int *cta_flag, int *abort_w,
                                             unsigned int *err) {
    const long long t0 = clock64();
    long long tpoll = t0;
    while (*p < target) {
        if (*cta_flag) return false;
        const long long now = clock64();
        if (abort_due(now, tpoll, abort_w)) {
            *cta_flag = 1;
            return false;
        }
        if (now - t0 > kWaitCycles) {
            raise_abort_w(abort_w, err, cta_flag);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}
__device__ __forceinline__ bool wait_count(const volatile int *p, int target, volatile int *cta_flag,
                                           const FwdArgs &a, const PcArgs &pc) {
    if (*p >= target) return true;
    return wait_count_slow(p, target, cta_flag, pc.abort, a.err);
}

// The jobs of producer p: the (chunk c, unit u) pairs with c < nch[u], ordered by c then
// u, every P-th one starting at the p-th. Every thread of a stage steps its own copy.
struct JobIt {
    int c, u, k;  // current pair and its index among all jobs
};
// Jobs are taken in the order (chunk, unit). With units of equal length a producer claims
// its next job from a global counter (set_job), so that faster producers take more jobs and
// every producer stays near the common front of that order; otherwise producer p takes the
// jobs p, p + P, p + 2P, ... of the order (next_job), skipping the chunks a unit lacks.
__device__ __forceinline__ bool set_job(JobIt &it, int k, const Ctx &x, const PcArgs &pc) {
    it.k = k;
    it.c = k / pc.U;
    it.u = k - it.c * pc.U;
    return it.c < x.maxc;
}
__device__ __forceinline__ bool next_job(JobIt &it, const Ctx &x, const PcArgs &pc) {
    const int want = it.k < 0 ? x.p : it.k + pc.P;
    while (true) {
        if (++it.u == pc.U) {
            it.u = 0;
            if (++it.c >= x.maxc) return false;
        }
        if (x.units[it.u].nch > it.c && ++it.k == want) return true;
    }
}

__device__ __forceinline__ unsigned char *slot_ptr(const PcArgs &pc, int u, int c) {
    return pc.ring + ((int64_t)u * pc.R + c % pc.R) * Slot::kStride;
}

// ---------------------------------------------------------------------------------------
// producer, front stage (warps 0-7): tiles, gate pass, Gram; the front image of the slot
// goes to the ring by one bulk store. Returns the TMA loads that may still be in flight
// (abort path): bit 0 Q/K, bit 1 G; bits 4 and 5 their parities. With FE the front-end is
// applied on the way: beta and the per-head gates as they land, the per-channel gates
// before the cumulative sum, and the q / k norms as factors of the image rows.
// ---------------------------------------------------------------------------------------
template <bool GATE_HEAD, bool FE>
__device__ __forceinline__ uint32_t producer_front(const FwdArgs &a, const TcMaps &maps, const PcArgs &pc,
                                                   const Ctx &x) {
    unsigned char *sm = x.sm;
    uint64_t *bars = x.bars;
    const int ptid = threadIdx.x, pw = ptid >> 5, lane = ptid & 31;
    const uint32_t lane_off = (uint32_t)(32 * (pw & 3)) << 16;  // this warp's TMEM lane quarter
    const uint32_t half = (uint32_t)(pw >> 2) * 32u;             // column half of a 64-wide readback
    const bf16 *RQ = reinterpret_cast<const bf16 *>(sm + Prod::oRQ);
    const bf16 *RK = reinterpret_cast<const bf16 *>(sm + Prod::oRK);
    float *G = reinterpret_cast<float *>(sm + Prod::oG);
    float *Tot = reinterpret_cast<float *>(sm + Prod::oTot);
    float *EG = reinterpret_cast<float *>(sm + Prod::oEG);
    const int64_t sg = GATE_HEAD ? (int64_t)a.H_v : (int64_t)a.H_v * 128;
    uint32_t pend = 0;

    // Bulk copies issued by one thread are served one after another; the copies of a job
    // are spread over the lane 0 of different warps so that they overlap. The issuers are
    // threads that load nothing with cp.async (beta and the per-head gates come from threads
    // 0-127): a thread's cp.async wait was measured to also wait for its own bulk copies
    // still in flight, which held the whole stage at the next barrier.
    constexpr int kIssQ = 128, kIssK = 160, kIssG = 192, kIssImg = 224;
    auto stage_qk = [&](const JobIt &j, int jo) {
        if (ptid == kIssQ || ptid == kIssK) {
            const int hk = (j.u % a.H_v) / a.group;
            const int y = (int)(x.units[j.u].bos + (int64_t)j.c * kChunk);
            if (ptid == kIssQ) {
                // the barrier expects both tiles; K may land first (transaction counts may
                // run ahead of the expectation within a phase)
                mbar_arrive_expect_tx(&bars[B_LQK], 32768);
                tma_load_2d(sm + Prod::oRQ, &maps.q, &bars[B_LQK], hk * 128, y);
            } else {
                tma_load_2d(sm + Prod::oRK, &maps.k, &bars[B_LQK], hk * 128, y);
            }
        }
        pend = (pend & ~0x11u) | 1u | ((uint32_t)(jo & 1) << 4);
    };
    // G by TMA; beta (and the per-head gates) by cp.async into the job-parity buffers
    auto stage_g = [&](const JobIt &j, int jo) {
        const int h = j.u % a.H_v;
        const int64_t bos = x.units[j.u].bos;
        const int row0 = j.c * kChunk;
        const int nvalid = min(kChunk, x.units[j.u].len - row0);
        if constexpr (!GATE_HEAD) {
            if (ptid == kIssG) {
                mbar_arrive_expect_tx(&bars[B_LG], 32768);
                tma_load_2d(sm + Prod::oG, &maps.g, &bars[B_LG], h * 128, (int)(bos + row0));
            }
            pend = (pend & ~0x22u) | 2u | ((uint32_t)(jo & 1) << 5);
        }
        float *Bf = reinterpret_cast<float *>(sm + ((jo & 1) ? Prod::oBF1 : Prod::oBF0));
        float *Gh = reinterpret_cast<float *>(sm + ((jo & 1) ? Prod::oGh1 : Prod::oGh0));
        if (ptid < 64) {
            const bool ok = ptid < nvalid;
            if (a.decay_only) {
                Bf[ptid] = ok ? 1.f : 0.f;
            } else {
                const int64_t ob = ok ? (bos + row0 + ptid) * a.H_v + h : 0;
                cp_async_4(Bf + ptid, a.beta + ob, ok ? 4 : 0);
            }
        } else if (GATE_HEAD && ptid < 128) {
            const int r = ptid - 64;
            const bool ok = r < nvalid;
            const int64_t og = ok ? (bos + row0 + r) * sg + h : 0;
            cp_async_4(Gh + r, a.g + og, ok ? 4 : 0);
        }
        cp_async_commit();
    };

    JobIt it{0, -1, -1};
    bool have = x.uniform ? set_job(it, x.jobq[0], x, pc) : next_job(it, x, pc);
    if (have) {
        stage_g(it, 0);
        stage_qk(it, 0);
    }
    bool failed = false;
    int jo = 0;
    int claimed = 0;  // thread 0, equal lengths: the job claimed for ordinal jo + 2
    for (; have; ++jo) {
        const int u = it.u, c = it.c, b = jo & 1;
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, x.units[u].len - row0);
        const int nz = kChunk - nvalid;  // rows past the sequence end: zero in every operand
        // The next job (equal lengths): thread 0 claimed it at the top of the previous job
        // (the atomic's latency is then off the path) and publishes it here; every thread
        // reads it after the first barrier below, the back stage after this job's hand-off.
        JobIt nx = it;
        bool have_next = false;
        if (!x.uniform) {
            have_next = next_job(nx, x, pc);
        } else if (ptid == 0) {
            if (jo > 0) x.jobq[(jo + 1) & 3] = claimed;  // jobs 0 and 1 were claimed at the start
            claimed = atomicAdd(pc.jobs, 1);              // job jo + 2
        }
        const uint32_t oKP = b ? Prod::oKP1 : Prod::oKP0;
        float *Bf = reinterpret_cast<float *>(sm + (b ? Prod::oBF1 : Prod::oBF0));
        float *Gh = reinterpret_cast<float *>(sm + (b ? Prod::oGh1 : Prod::oGh0));
        const int h = u % a.H_v;
        // front-end: -exp(A_log[h]) and this thread's two channel biases
        float negA = 0.f, bias0 = 0.f, bias1 = 0.f;
        if constexpr (FE) {
            if (a.fe_A_log != nullptr) {
                negA = -expf(a.fe_A_log[h]);
                if (a.fe_dt_bias != nullptr) {
                    if constexpr (GATE_HEAD) {
                        bias0 = a.fe_dt_bias[h];
                    } else {
                        const int cb = 64 * (pw & 1) + 2 * lane;
                        bias0 = a.fe_dt_bias[h * 128 + cb];
                        bias1 = a.fe_dt_bias[h * 128 + cb + 1];
                    }
                }
            }
        }

        if (ptid < (GATE_HEAD ? 128 : 64)) cp_async_wait_all();  // this job's beta and per-head gates
        if constexpr (FE) {
            // each thread transforms the values it loaded itself (rows past the end stay 0)
            if (ptid < 64) {
                if (a.fe_beta_sigmoid && !a.decay_only && ptid < nvalid) Bf[ptid] = sigmoid_fast(Bf[ptid]);
            } else if (GATE_HEAD && ptid < 128 && a.fe_A_log != nullptr && ptid - 64 < nvalid) {
                Gh[ptid - 64] = negA * softplus_fast(Gh[ptid - 64] + bias0);
            }
        }
        if constexpr (!GATE_HEAD) failed = !wait_bar(&bars[B_LG], (uint32_t)(jo & 1), x.flag, a, pc);
        if (bar_or(1, 256, failed)) { failed = true; break; }
        if (x.uniform) have_next = set_job(nx, x.jobq[(jo + 1) & 3], x, pc);
        pend &= ~2u;
        if (!GATE_HEAD && nz > 0) {
            for (int i = ptid; i < nz * 32; i += 256) {
                const int r = nvalid + (i >> 5), c16 = i & 31;
                *reinterpret_cast<uint4 *>(sm + Prod::oG + r * 512 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            bar_named(1, 256);
        }

        // ---- gate pass ---------------------------------------------------------------------
        // thread: rows 16 qr .. 16 qr + 15 (qr = pw >> 1) of the channel pair c0, c0 + 1,
        // c0 = 64 (pw & 1) + 2 lane; gl0 / gl1 hold the two channels' running log2 sums.
        const int qr = pw >> 1;
        const int c0 = 64 * (pw & 1) + 2 * lane;
        float gl0[16], gl1[16];
        bool gate_done = false;
        if constexpr (!GATE_HEAD && FE) {
            if (a.fe_A_log != nullptr) {
                // every gate of the thread first (independent), then the running sums
                const float nAl = negA * kLog2e;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = 16 * qr + e;
                    const float2 gv = *reinterpret_cast<const float2 *>(G + r * 128 + c0);
                    const float v0 = nAl * softplus_fast(gv.x + bias0);
                    const float v1 = nAl * softplus_fast(gv.y + bias1);
                    gl0[e] = r < nvalid ? v0 : 0.f;
                    gl1[e] = r < nvalid ? v1 : 0.f;
                }
#pragma unroll
                for (int e = 1; e < 16; ++e) {
                    gl0[e] += gl0[e - 1];
                    gl1[e] += gl1[e - 1];
                }
                gate_done = true;
            }
        }
        if (!gate_done) {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = 16 * qr + e;
                if constexpr (!GATE_HEAD) {
                    const float2 gv = *reinterpret_cast<const float2 *>(G + r * 128 + c0);
                    acc0 += gv.x * kLog2e;
                    acc1 += gv.y * kLog2e;
                } else {
                    acc0 += Gh[r] * kLog2e;
                    acc1 = acc0;
                }
                gl0[e] = acc0;
                gl1[e] = acc1;
            }
        }
        *reinterpret_cast<float2 *>(Tot + qr * 128 + c0) = make_float2(gl0[15], gl1[15]);
        // G (and the per-head gates) are consumed: request the next job's right away
        bar_named(1, 256);
        if (have_next) stage_g(nx, jo + 1);
        failed = !wait_bar(&bars[B_LQK], (uint32_t)(jo & 1), x.flag, a, pc);
        if (!failed && ptid == kIssImg && jo > 0) {
            // the previous image is written (long since): the image buffer is free, and the
            // back stage may publish that job
            bulk_wait_done();
            *x.stored = jo;
        }
        // the ring slot holds chunk c - R until the consumer has copied it out; done[u] only
        // grows, so a value this CTA has already acquired that is large enough saves the
        // round trip to L2
        if (!failed && ptid == 0 && c >= pc.R && x.seen[u] < c - pc.R + 1)
            failed = !wait_geq(&pc.done[u * kFlagLine], c - pc.R + 1, x.flag, a, pc, &x.seen[u]);
        // hand-off slot b (Kp^T) is free once the back stage has multiplied job jo - 2
        if (!failed && jo >= 2)
            failed = !wait_bar(&bars[B_HEMPTY0 + b], (uint32_t)(((jo >> 1) - 1) & 1), x.flag, a, pc);
        if (bar_or(1, 256, failed)) { failed = true; break; }
        pend &= ~1u;
        if (nz > 0) {
            for (int i = ptid; i < nz * 16; i += 256) {
                const int r = nvalid + (i >> 4), c16 = i & 15;
                *reinterpret_cast<uint4 *>(sm + Prod::oRQ + r * 256 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sm + Prod::oRK + r * 256 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            bar_named(1, 256);
        }
        if constexpr (FE) {
            if (a.fe_qk_l2norm) {
                qk_row_norms(sm + Prod::oRQ, sm + Prod::oRK, reinterpret_cast<float *>(sm + Prod::oRN), pw, lane, 1.f);
                bar_named(1, 256);
            }
        }
        {
            float off0 = 0.f, off1 = 0.f, gn0 = 0.f, gn1 = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const float2 t = *reinterpret_cast<const float2 *>(Tot + qq * 128 + c0);
                if (qq < qr) {
                    off0 += t.x;
                    off1 += t.y;
                }
                gn0 += t.x;
                gn1 += t.y;
            }
            if (qr == 0) *reinterpret_cast<float2 *>(EG + c0) = make_float2(ex2(gn0), ex2(gn1));
            // The products are taken on bf16 pairs of the two channels of one token (the factor
            // e^{+-gamma} rounded to bf16 first), then each 2 x 2 block of (token, channel) is
            // transposed by byte permutes into the [d][tok] rows. Lanes whose (lane >> 2) is odd
            // store the odd channel's row first, so that each 16-byte store spans all eight
            // swizzle phases of its rows.
            const bool odd_first = (lane >> 2) & 1;
            const uint32_t sel_a = odd_first ? 0x7632u : 0x5410u, sel_b = odd_first ? 0x5410u : 0x7632u;
            const int ra = c0 + (odd_first ? 1 : 0), rb = c0 + (odd_first ? 0 : 1);
            const float *RN = reinterpret_cast<const float *>(sm + Prod::oRN);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tc = 2 * qr + j;  // 16-byte chunk (8 tokens) of a 64-token row
                uint32_t qp2[8], kp2[8], km2[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = 16 * qr + 8 * j + e;
                    const float gm0 = off0 + gl0[8 * j + e];
                    const float ep0 = ex2(gm0), em0 = ex2(-gm0);
                    float ep1 = ep0, em1 = em0;
                    if constexpr (!GATE_HEAD) {
                        const float gm1 = off1 + gl1[8 * j + e];
                        ep1 = ex2(gm1);
                        em1 = ex2(-gm1);
                    }
                    const uint32_t q2 = *reinterpret_cast<const uint32_t *>(RQ + r * 128 + c0);
                    const uint32_t k2 = *reinterpret_cast<const uint32_t *>(RK + r * 128 + c0);
                    uint32_t epq, epk, emk;
                    if constexpr (FE) {
                        // front-end: the row factors 1 / |q_r| and 1 / |k_r| (or 1)
                        const bool nrm = a.fe_qk_l2norm != 0;
                        const float fq = nrm ? RN[r] : 1.f, fk = nrm ? RN[64 + r] : 1.f;
                        epq = pack_bf16(ep0 * fq, ep1 * fq);
                        epk = pack_bf16(ep0 * fk, ep1 * fk);
                        emk = pack_bf16(em0 * fk, em1 * fk);
                    } else {
                        epq = epk = pack_bf16(ep0, ep1);
                        emk = pack_bf16(em0, em1);
                    }
                    qp2[e] = mul_bf16x2(q2, epq);
                    kp2[e] = a.decay_only ? 0u : mul_bf16x2(k2, epk);
                    km2[e] = mul_bf16x2(k2, emk);
                }
                store_pairs_t(sm + Prod::oQP, qp2, ra, rb, tc, sel_a, sel_b);
                store_pairs_t(sm + oKP, kp2, ra, rb, tc, sel_a, sel_b);
                store_pairs_t(sm + Prod::oKM, km2, ra, rb, tc, sel_a, sel_b);
            }
        }
        fence_proxy_async();
        bar_named(1, 256);
        if (have_next) stage_qk(nx, jo + 1);  // the raw Q and K tiles are consumed

        // ---- Gram: D_G = [Qp; Kp] Km^T  (rows 0-63: Aqk, rows 64-127: M) --------------------
        if (ptid == 0) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 64, true, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(x.tmem + tGram, dMN(x.sbase + Prod::oQP, oKP - (uint32_t)Prod::oQP, s),
                    dMN(x.sbase + Prod::oKM, 16384, s), id, s > 0);
            commit(&bars[B_GRAM]);
        }
        failed = !wait_bar(&bars[B_GRAM], (uint32_t)(jo & 1), x.flag, a, pc);
        // L and beta go to the buffer of this job's parity, which job jo - 2 used: its
        // solve is long done unless the back stage is two jobs behind
        if (!failed && jo >= 2)
            failed = !wait_bar(&bars[B_LFREE0 + b], (uint32_t)(((jo >> 1) - 1) & 1), x.flag, a, pc);
        if (bar_or(1, 256, failed)) { failed = true; break; }
        fence_after_sync();
        {
            // each warp half reads 32 of the 64 columns of its lane's row
            float *Lw = reinterpret_cast<float *>(sm + (b ? Prod::oL1 : Prod::oL0));
            const int row = 32 * (pw & 3) + lane;
            float v[32];
            tmem_ld32(x.tmem + lane_off + tGram + half, v);
            if (row < 64) {
                // Aqk (lower, diagonal included) -> bf16 [tok][tok'], K-major B operand
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int col = (int)half + 8 * c8 + e;
                        y[e] = col <= row ? v[8 * c8 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sm + Prod::oAQ + sw128(row, (int)(half >> 3) + c8)) = pack8(y);
                }
            } else {
                // L = diag(beta) strict_lower(M), fp32
                const int r = row - 64;
                const float br = Bf[r];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int col = (int)half + e;
                    float4 y;
                    y.x = col < r ? br * v[e] : 0.f;
                    y.y = col + 1 < r ? br * v[e + 1] : 0.f;
                    y.z = col + 2 < r ? br * v[e + 2] : 0.f;
                    y.w = col + 3 < r ? br * v[e + 3] : 0.f;
                    *reinterpret_cast<float4 *>(Lw + r * LDF + col) = y;
                }
            }
            if (ptid < 64) reinterpret_cast<float *>(sm + (b ? Prod::oBH1 : Prod::oBH0))[ptid] = Bf[ptid];
        }
        fence_proxy_async();
        fence_before_sync();
        bar_named(1, 256);
        if (ptid == 0) mbar_arrive(&bars[B_HFULL0 + b]);
        if (ptid == kIssImg) {
            // Qp^T, Km^T, Aqk, e^gamma_n -> the ring slot, one bulk store; once it is
            // written the image buffer is free and the back stage may publish the job
            fence_proxy_async_global();  // after the slot was seen free (and dropped from L2)
            bulk_store(slot_ptr(pc, u, c) + Slot::oQP, sm + Prod::oIMG, Slot::kFrontBytes);
            bulk_commit();
        }
        it = nx;
        have = have_next;
    }
    cp_async_wait_all();  // no copy into shared memory outlives the loop
    if (failed) {
        *x.flag = 1;
    } else if (ptid == kIssImg && jo > 0) {
        bulk_wait_done();
        *x.stored = jo;
    }
    return pend;
}

// ---------------------------------------------------------------------------------------
// producer, back stage (warps 8-15): solve, WY factors, publication of the slot.
// Returns 0, or 1 + the parity of a V load that may still be in flight (abort path).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int producer_back(const FwdArgs &a, const TcMaps &maps, const PcArgs &pc, const Ctx &x) {
    unsigned char *sm = x.sm;
    uint64_t *bars = x.bars;
    const int ptid = threadIdx.x - 256, pw = ptid >> 5, lane = ptid & 31, warp = threadIdx.x >> 5;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter
    const uint32_t half = (uint32_t)(pw >> 2) * 32u;                // column half of a 64-wide readback
    constexpr int kPublisher = 224;  // lane 0 of the last warp: stores and publishes the slot
    float *Tm = reinterpret_cast<float *>(sm + Prod::oT);
    int pend_v = -1;
    auto stage_v = [&](const JobIt &j, int jo) {
        if (ptid == 0 || ptid == 32) {  // the two d_v halves from two warps
            const int h = j.u % a.H_v;
            const int y = (int)(x.units[j.u].bos + (int64_t)j.c * kChunk);
            if (ptid == 0) {
                mbar_arrive_expect_tx(&bars[B_LV], 16384);
                tma_load_2d(sm + Prod::oRV, &maps.v, &bars[B_LV], h * 128, y);
            } else {
                tma_load_2d(sm + Prod::oRV + 8192, &maps.v, &bars[B_LV], h * 128 + 64, y);
            }
        }
        pend_v = jo & 1;
    };

    // Publication of chunk pcn of unit pu, job ordinal pjo of this producer, once its W^T and
    // U^T stores and its front image are written. It depends on nothing later than the job.
    auto publish = [&](int pu, int pcn, int pjo) -> bool {
        bulk_wait_done();
        if (!wait_count(x.stored, pjo + 1, x.flag, a, pc)) return false;
        fence_proxy_async_global();
        st_release(&pc.ready[pu * kFlagLine + pcn % pc.R], pcn + 1);
        return true;
    };

    JobIt it{0, -1, -1};
    bool have = x.uniform ? set_job(it, x.jobq[0], x, pc) : next_job(it, x, pc);
    if (have) stage_v(it, 0);
    bool failed = false;
    int prev_u = -1, prev_c = 0;
    int jo = 0;
    for (; have; ++jo) {
        const int u = it.u, c = it.c, b = jo & 1;
        const int row0 = c * kChunk;
        const int nvalid = min(kChunk, x.units[u].len - row0);
        const int nz = kChunk - nvalid;
        JobIt nx = it;
        bool have_next = x.uniform ? false : next_job(nx, x, pc);  // equal lengths: after the hand-off
        unsigned char *slot = slot_ptr(pc, u, c);
        const uint32_t oKP = b ? Prod::oKP1 : Prod::oKP0;
        const float *L = reinterpret_cast<const float *>(sm + (b ? Prod::oL1 : Prod::oL0));
        const float *Bs = reinterpret_cast<const float *>(sm + (b ? Prod::oBH1 : Prod::oBH0));

        // The previous job's W^T and U^T stores read the T buffer and its Kp^T buffer: the
        // publisher waits for those reads here, ahead of the barrier after the hand-off
        // (before which no thread of this stage writes either buffer), so that the wait
        // overlaps the wait for the front stage, and then returns the Kp^T buffer to it.
        if (ptid == kPublisher && jo > 0) {
            bulk_wait_read();
            mbar_arrive(&bars[B_HEMPTY0 + (b ^ 1)]);
        }
        // The previous job is published while this stage would wait for the front stage;
        // when the front stage is already done with this job, the publisher does it during
        // the diagonal solve instead (its warp is idle there). Either way it waits on
        // nothing later than that job.
        bool defer = false;
        if (ptid == kPublisher && jo > 0) {
            defer = mbar_try_wait(&bars[B_HFULL0 + b], (uint32_t)((jo >> 1) & 1));
            if (!defer) failed = !publish(prev_u, prev_c, jo - 1);
        }
        if (!failed) failed = !wait_bar(&bars[B_HFULL0 + b], (uint32_t)((jo >> 1) & 1), x.flag, a, pc);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        // the front stage claimed the next job before it handed this one off
        if (x.uniform) have_next = set_job(nx, x.jobq[(jo + 1) & 3], x, pc);

        // ---- solve: T = (I + L)^-1 -----------------------------------------------------------
        // Warps 0-3 invert (I + L) as a 2 x 2 block matrix of 32 x 32 blocks A (tokens 0-31)
        // and B (32-63), each itself 2 x 2 in 16 x 16 blocks:
        //   D_k = (I + L_kk)^-1                      forward substitution, one column per lane
        //   T_10 = -D_1 L_10 D_0,  T_32 = -D_3 L_32 D_2
        //   Y = L_BA T_AA,  T_BA = -T_BB Y
        // (tf32 mma.sync, fp32 accumulation; Y is kept in T's unused upper triangle). Warps
        // 4-7, the publisher's among them, meet them at the T_beta step.
        float *Y = Tm + 32;  // Y[r][c] at Tm[r * LDF + 32 + c], r, c < 32
        if (pw < 4) {
            if (lane < 16) {
                const int b0 = 16 * pw, j = lane;
                float v[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float s = (r == j) ? 1.f : 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) s -= L[(b0 + r) * LDF + b0 + m] * v[m];
                    v[r] = s;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(b0 + r) * LDF + b0 + j] = v[r];
            }
            bar_named(5, 128);
            const int g8 = lane >> 2, t4 = lane & 3;
            // T_10 (warps 0, 1) and T_32 (warps 2, 3), 8 columns each: P = L_ij D_j, T_ij = -D_i P
            {
                const int i = (pw < 2) ? 1 : 3, jb = i - 1, col0 = 16 * jb + 8 * (pw & 1);
                float *P = reinterpret_cast<float *>(sm + Prod::oPS) + pw * 128;  // 16x8 scratch
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                mm16x8_tf32(acc, L + (16 * i) * LDF + 16 * jb, LDF, Tm + (16 * jb) * LDF + col0, LDF, lane);
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
            }
            bar_named(5, 128);
            // Y = L_BA T_AA: warp pw takes row block rb = pw >> 1 of Y and the 8-column tiles
            // ct0 = 2 (pw & 1) and ct0 + 1; T_AA has D_0, T_10 in columns 0-15 and D_1 in 16-31
            {
                const int rb = pw >> 1, ct0 = 2 * (pw & 1);
                const float *Lr = L + (32 + 16 * rb) * LDF;
                float acc[2][4];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
                    const int col = 8 * (ct0 + q);
                    if (col < 16) mm16x8_tf32(acc[q], Lr, LDF, Tm + col, LDF, lane);  // L_B0 [D_0; T_10]
                    mm16x8_tf32(acc[q], Lr + 16, LDF, Tm + 16 * LDF + col, LDF, lane);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float *Yt = Y + (16 * rb) * LDF + 8 * (ct0 + q);
                    Yt[g8 * LDF + 2 * t4] = acc[q][0];
                    Yt[g8 * LDF + 2 * t4 + 1] = acc[q][1];
                    Yt[(g8 + 8) * LDF + 2 * t4] = acc[q][2];
                    Yt[(g8 + 8) * LDF + 2 * t4 + 1] = acc[q][3];
                }
            }
            bar_named(5, 128);
            // T_BA = -T_BB Y: row block rb of T_BA is -D_2 Y_0 (rb = 0) or -(T_32 Y_0 + D_3 Y_1)
            {
                const int rb = pw >> 1, ct0 = 2 * (pw & 1);
                const float *Tb = Tm + (32 + 16 * rb) * LDF + 32;  // [T_32 | D_3] or [D_2 | 0]
                float acc[2][4];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
                    const int col = 8 * (ct0 + q);
                    if (rb == 0) {
                        mm16x8_tf32(acc[q], Tb, LDF, Y + col, LDF, lane);
                    } else {
                        mm16x8_tf32(acc[q], Tb, LDF, Y + col, LDF, lane);
                        mm16x8_tf32(acc[q], Tb + 16, LDF, Y + 16 * LDF + col, LDF, lane);
                    }
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float *Tt = Tm + (32 + 16 * rb) * LDF + 8 * (ct0 + q);
                    Tt[g8 * LDF + 2 * t4] = -acc[q][0];
                    Tt[g8 * LDF + 2 * t4 + 1] = -acc[q][1];
                    Tt[(g8 + 8) * LDF + 2 * t4] = -acc[q][2];
                    Tt[(g8 + 8) * LDF + 2 * t4 + 1] = -acc[q][3];
                }
            }
        } else if (pw == 7 && defer) {
            failed = !publish(prev_u, prev_c, jo - 1);
        }
        bar_named(2, 256);
        // T_beta = T diag(beta), lower triangle, bf16 [tok][tok'] (K-major B): warp pw writes
        // the 8 columns col0 .. col0 + 7, col0 = 8 pw
        {
            const int col0 = 8 * pw, jb = pw >> 1;
            const float4 b0 = *reinterpret_cast<const float4 *>(Bs + col0);
            const float4 b1 = *reinterpret_cast<const float4 *>(Bs + col0 + 4);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                float v[8];
                if (r < 16 * jb) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.f;
                } else {
                    const float4 t0 = *reinterpret_cast<const float4 *>(Tm + r * LDF + col0);
                    const float4 t1 = *reinterpret_cast<const float4 *>(Tm + r * LDF + col0 + 4);
                    const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = (col0 + e) <= r ? tv[e] * bv[e] : 0.f;
                }
                *reinterpret_cast<uint4 *>(sm + Prod::oTB + sw128(r, col0 >> 3)) = pack8(v);
            }
        }
        failed = !wait_bar(&bars[B_LV], (uint32_t)(jo & 1), x.flag, a, pc);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        pend_v = -1;
        if (ptid == 0) mbar_arrive(&bars[B_LFREE0 + b]);  // L and beta of this parity are consumed
        if (nz > 0) {
            for (int i = ptid; i < nz * 16; i += 256) {
                const int r = nvalid + (i >> 4), c16 = i & 15;
                *reinterpret_cast<uint4 *>(sm + Prod::oRV + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async();
        bar_named(2, 256);

        // ---- WY factors: D_W = Kp^T T_beta^T, D_U = V^T T_beta^T ------------------------------
        if (ptid == 0) {
            fence_after_sync();
            const uint32_t idw = idesc_bf16(128, 64, false, false, false);
            const uint32_t idu = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = dK(x.sbase + Prod::oTB, 8192, s);
                mma(x.tmem + tW, dK(x.sbase + oKP, 16384, s), bd, idw, s > 0);
                mma(x.tmem + tU, dMN(x.sbase + Prod::oRV, 8192, s), bd, idu, s > 0);
            }
            commit(&bars[B_WMMA]);
        }
        failed = !wait_bar(&bars[B_WMMA], (uint32_t)(jo & 1), x.flag, a, pc);
        if (bar_or(2, 256, failed)) { failed = true; break; }
        // V is consumed: the next job's tile is requested before this job's stores, which
        // would otherwise hold it up in the SM's bulk-copy queue
        if (have_next) stage_v(nx, jo + 1);
        fence_after_sync();
        {
            // row d of W^T and of U^T; each warp half takes 32 of the 64 tokens. W^T goes to
            // the (now free) T buffer as the swizzled [d][tok] image, U^T to the job's Kp^T
            // buffer (consumed by the W MMA) as bf16 token pairs.
            const int d = 32 * (warp & 3) + lane;
            float v[32];
            tmem_ld32(x.tmem + lane_off + tW + half, v);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = v[8 * c8 + e];
                *reinterpret_cast<uint4 *>(sm + Prod::oT + sw128(d, (int)(half >> 3) + c8)) = pack8(y);
            }
            tmem_ld32(x.tmem + lane_off + tU + half, v);
            uint32_t *U2 = reinterpret_cast<uint32_t *>(sm + oKP);
#pragma unroll
            for (int e = 0; e < 16; ++e) U2[((int)(half >> 1) + e) * 128 + d] = pack_bf16(v[2 * e], v[2 * e + 1]);
        }
        fence_proxy_async();
        fence_before_sync();
        bar_named(2, 256);
        if (ptid == kPublisher) {
            fence_proxy_async_global();  // after the slot was seen free (and dropped from L2)
            bulk_store(slot + Slot::oWT, sm + Prod::oT, 16384);
            bulk_store(slot + Slot::oU, sm + oKP, 16384);
            bulk_commit();
        }
        prev_u = u;
        prev_c = c;
        it = nx;
        have = have_next;
    }
    if (!failed && ptid == kPublisher && prev_u >= 0) failed = !publish(prev_u, prev_c, jo - 1);
    if (failed) *x.flag = 1;
    return pend_v + 1;
}

// ---------------------------------------------------------------------------------------
// consumer, loader (warps 4-6): slot images of unit u into the three shared buffers, each
// as three bulk copies from three warps (so that they overlap); up to three in flight. A
// ring slot is released when its buffer comes round again. Returns, for thread 128, the
// copies that may still be in flight: bit b for buffer b, bit 4 + b its phase parity.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int consumer_loader(const FwdArgs &a, const PcArgs &pc, const Ctx &x, int u, int nch) {
    uint64_t *bars = x.bars;
    const int lt = threadIdx.x - 128, lw = lt >> 5, lane = lt & 31;
    static_assert(Slot::kBytes % 16 == 0, "16-byte parts");
    constexpr uint32_t kPart = ((Slot::kBytes / 16 + 2) / 3) * 16;  // parts 0, 1; part 2 is the rest
    const uint32_t off = lw * kPart, bytes = lw < 2 ? kPart : Slot::kBytes - 2 * kPart;
    int pend = 0;
    bool failed = false;
    for (int c = 0; c < nch; ++c) {
        const int b = c % Cons::kBufs, k = c / Cons::kBufs;  // buffer and its use count
        if (lt == 0 && !failed) {
            // buffer b held chunk c - 3 until its output left; that copy has long landed, so
            // the ring slot of chunk c - 3 is free for the producers
            if (c >= Cons::kBufs) {
                failed = !wait_bar(&bars[B_EMPTY0 + b], (uint32_t)((k - 1) & 1), x.flag, a, pc);
                if (!failed) st_release(&pc.done[u * kFlagLine], c - Cons::kBufs + 1);
            }
            if (!failed) failed = !wait_geq(&pc.ready[u * kFlagLine + c % pc.R], c + 1, x.flag, a, pc);
            if (!failed) mbar_arrive_expect_tx(&bars[B_FULL0 + b], Slot::kBytes);
        }
        if (bar_or(2, 96, failed)) {
            failed = true;
            break;
        }
        if (lane == 0) {
            fence_proxy_async_global();  // the producers' generic writes, before the async-proxy read
            bulk_load(x.sm + b * Slot::kStride + off, slot_ptr(pc, u, c) + off, bytes, &bars[B_FULL0 + b]);
        }
        pend = (pend & ~(0x11 << b)) | ((1 | ((k & 1) << 4)) << b);
    }
    return lt == 0 ? pend : 0;
}

// ---------------------------------------------------------------------------------------
// consumer: the MMAs of the serial step are issued by warp 7 (lane 0), which waits for the
// element warps at named barrier kBarIss; the element warps arrive there without waiting
// (bar.arrive), once when the bf16 copy of the state S_c^T is in TMEM and once when
// Vt^T is. Every exit of the element warps on a failure arrives once more, so that the
// issuer never waits for arrivals that will not come.
// ---------------------------------------------------------------------------------------
constexpr int kBarIss = 1, kIssCount = 288;  // warps 0-3, 8-11 arrive; warp 7 waits

__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------------------
// consumer, serial step (warps 0-3 and 8-11): row dv of S^T (fp32 in TMEM) belongs to lane
// dv % 32 of warps dv / 32 and 8 + dv / 32, which take the column halves 0-63 and 64-127
// of every element pass (the two warps reach the same TMEM lanes).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void consumer_serial(const FwdArgs &a, const PcArgs &pc, const Ctx &x, int u) {
    unsigned char *sm = x.sm;
    const uint32_t tmem = x.tmem;
    uint64_t *bars = x.bars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp >> 3;                 // column half
    const int dv = 32 * (warp & 3) + lane;     // row of S^T
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int n = u / a.H_v, h = u % a.H_v;
    const int nchunks = x.units[u].nch;
    const uint32_t tSc = tS + 64 * grp, tSAc = tSA + 32 * grp;  // this thread's columns
    // e^gamma_n of the chunks by parity: the slot buffer is released before the state's bf16
    // copy (and the next chunk's rescale) would read it
    float *egc = reinterpret_cast<float *>(sm + Common::oEGc);

    // S^T row dv, columns 64 grp .. +63 (from h0, or zero) -> TMEM fp32 and its bf16 copy
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int d = 64 * grp + 32 * pass + e;
            v[e] = a.h0 ? a.h0[(((int64_t)n * a.H_v + h) * 128 + d) * 128 + dv] : 0.f;
        }
        uint32_t f0[16], f1[16], p16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            f0[e] = __float_as_uint(v[e]);
            f1[e] = __float_as_uint(v[16 + e]);
            p16[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
        }
        tmem_st16(tmem + lane_off + tSc + 32 * pass, f0);
        tmem_st16(tmem + lane_off + tSc + 32 * pass + 16, f1);
        tmem_st16(tmem + lane_off + tSAc + 16 * pass, p16);
    }
    tmem_st_wait();
    fence_before_sync();
    if (nchunks > 0) bar_arrive(kBarIss, kIssCount);  // S_0^T is in TMEM

    bool failed = false;
    for (int c = 0; c < nchunks; ++c) {
        const int b = c % Cons::kBufs;  // slot buffer; the TMEM buffers go by c & 1
        const uint32_t oB = b * Slot::kStride;
        const float *EG = reinterpret_cast<const float *>(sm + oB + Slot::oEG);
        const uint32_t *U2 = reinterpret_cast<const uint32_t *>(sm + oB + Slot::oU);
        const uint32_t tX = (c & 1) ? tX1 : tX0;

        failed = !wait_bar(&bars[B_FULL0 + b], (uint32_t)((c / Cons::kBufs) & 1), x.flag, a, pc);
        if (bar_or(4, 256, failed)) { failed = true; break; }
        // this chunk's e^gamma_n is kept (the slot buffer may be released before the copy
        // pass below reads it)
        if ((warp & 3) == 0) {
            egc[(c & 1) * 128 + 64 * grp + lane] = EG[64 * grp + lane];
            egc[(c & 1) * 128 + 64 * grp + 32 + lane] = EG[64 * grp + 32 + lane];
        }

        failed = !wait_bar(&bars[B_X], (uint32_t)(c & 1), x.flag, a, pc);
        if (bar_or(4, 256, failed)) { failed = true; break; }
        fence_after_sync();
        // Vt^T = U^T - S^T W^T for tokens 32 grp .. +31 -> bf16 token pairs at tV
        {
            float pp[32];
            tmem_ld32(tmem + lane_off + tX + 32 * grp, pp);
            uint32_t v16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const uint32_t uw = U2[(16 * grp + e) * 128 + dv];  // tokens 32 grp + 2e, + 1
                const float u0 = __uint_as_float(uw << 16), u1 = __uint_as_float(uw & 0xffff0000u);
                v16[e] = pack_bf16(u0 - pp[2 * e], u1 - pp[2 * e + 1]);
            }
            tmem_st16(tmem + lane_off + tV + 16 * grp, v16);
        }
        tmem_st_wait();
        fence_before_sync();
        bar_arrive(kBarIss, kIssCount);  // Vt^T (and the rescaled R) are in TMEM

        failed = !wait_bar(&bars[B_R], (uint32_t)(c & 1), x.flag, a, pc);
        if (bar_or(4, 256, failed)) { failed = true; break; }
        fence_after_sync();
        // S_{c+1}^T = R Diag(e^gamma_n): back into R (fp32) and as the bf16 operand of the
        // next chunk
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            // the factors first, so that their loads overlap the TMEM load's wait
            float eg[32];
            const float4 *eg4 = reinterpret_cast<const float4 *>(egc + (c & 1) * 128 + 64 * grp + 32 * pass);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 t4 = eg4[q];
                eg[4 * q] = t4.x;
                eg[4 * q + 1] = t4.y;
                eg[4 * q + 2] = t4.z;
                eg[4 * q + 3] = t4.w;
            }
            float v[32];
            tmem_ld32(tmem + lane_off + tSc + 32 * pass, v);
            uint32_t p16[16], y0[16], y1[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float s0 = v[2 * e] * eg[2 * e], s1 = v[2 * e + 1] * eg[2 * e + 1];
                p16[e] = pack_bf16(s0, s1);
                if (e < 8) {
                    y0[2 * e] = __float_as_uint(s0);
                    y0[2 * e + 1] = __float_as_uint(s1);
                } else {
                    y1[2 * e - 16] = __float_as_uint(s0);
                    y1[2 * e - 15] = __float_as_uint(s1);
                }
            }
            tmem_st16(tmem + lane_off + tSAc + 16 * pass, p16);
            tmem_st16(tmem + lane_off + tSc + 32 * pass, y0);
            tmem_st16(tmem + lane_off + tSc + 32 * pass + 16, y1);
        }
        tmem_st_wait();
        fence_before_sync();
        if (c + 1 < nchunks) bar_arrive(kBarIss, kIssCount);  // S_{c+1}^T is in TMEM
    }
    if (failed) {
        *x.flag = 1;
        bar_arrive(kBarIss, kIssCount);  // the issuer may be waiting for this warp group
        return;
    }
    if (a.ht != nullptr) {
        // S_N^T = R (h0^T when there is no chunk)
        fence_after_sync();
        float *ht = a.ht + ((int64_t)n * a.H_v + h) * 128 * 128 + dv;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            float v[32];
            tmem_ld32(tmem + lane_off + tSc + 32 * pass, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) ht[(int64_t)(64 * grp + 32 * pass + e) * 128] = v[e];
        }
    }
}

// ---------------------------------------------------------------------------------------
// consumer, MMA issuer (warp 7; lane 0 issues): per chunk c, once its slot image has landed,
// the output half of its D_X buffer has been read out (chunk c - 2) and S_c^T is in TMEM:
//   D_X = S_c^T [W^T | Qp^T]   (A: S_c^T bf16 in TMEM; B: the W^T and Qp^T tiles, MN-major)
// then, once Vt^T is in TMEM:
//   R += Vt^T Km  (commit B_R: the next state's copy may start),
//   O^T = D_X[:, 64:] + Vt^T Aqk^T  (commit B_O0 / B_O1 by D_X buffer: the output may leave).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void consumer_issuer(const FwdArgs &a, const PcArgs &pc, const Ctx &x, int u) {
    uint64_t *bars = x.bars;
    const uint32_t tmem = x.tmem, sbase = x.sbase;
    const bool lead = (threadIdx.x & 31) == 0;
    const int nchunks = x.units[u].nch;
    bool failed = false;
    for (int c = 0; c < nchunks; ++c) {
        const int b = c % Cons::kBufs;
        const uint32_t oB = b * Slot::kStride;
        const uint32_t tX = (c & 1) ? tX1 : tX0;
        if (lead) {
            failed = !wait_bar(&bars[B_FULL0 + b], (uint32_t)((c / Cons::kBufs) & 1), x.flag, a, pc);
            if (!failed && c >= 2)
                failed = !wait_bar(&bars[B_XFREE0 + (c & 1)], (uint32_t)(((c >> 1) - 1) & 1), x.flag, a, pc);
        }
        if (__shfl_sync(0xffffffffu, (int)failed, 0)) { failed = true; break; }
        bar_named(kBarIss, kIssCount);  // S_c^T is in TMEM
        if (__shfl_sync(0xffffffffu, *x.flag, 0)) { failed = true; break; }
        if (lead) {
            fence_after_sync();
            const uint32_t id = idesc_bf16(128, 128, false, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_ts(tmem + tX, tmem + tSA + 8 * s, dMN(sbase + oB + Slot::oWT, Slot::oQP - Slot::oWT, s), id,
                       s > 0);
            commit(&bars[B_X]);
        }
        __syncwarp();
        bar_named(kBarIss, kIssCount);  // Vt^T (and the rescaled R) are in TMEM
        if (__shfl_sync(0xffffffffu, *x.flag, 0)) { failed = true; break; }
        if (lead) {
            fence_after_sync();
            const uint32_t ido = idesc_bf16(128, 64, false, false, false);
            const uint32_t ids = idesc_bf16(128, 128, false, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_ts(tmem + tS, tmem + tV + 8 * s, dK(sbase + oB + Slot::oKM, 16384, s), ids, 1);
            commit(&bars[B_R]);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_ts(tmem + tX + 64, tmem + tV + 8 * s, dK(sbase + oB + Slot::oAQ, 8192, s), ido, 1);
            commit(&bars[B_O0 + (c & 1)]);
        }
        __syncwarp();
    }
    if (failed) *x.flag = 1;
}

// Drop a 128-byte line from L2 without writing it back (its contents become undefined).
__device__ __forceinline__ void discard_l2(const void *p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// TMA 2-D store shared -> global (bulk async-group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const void *tmap, int x, int y, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}

// ---------------------------------------------------------------------------------------
// consumer, epilogue (warps 12-15): O^T of each chunk, scaled and rounded, leaves through the
// slot buffer of that chunk, whose W^T area (all its MMAs are complete) holds the [tok][d_v]
// tile for one TMA store; the buffer goes back to the loader once the store has read it. A
// chunk shorter than 64 tokens is written by plain stores of its valid rows.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void consumer_epilogue(const FwdArgs &a, const TcMaps &maps, const PcArgs &pc,
                                                  const Ctx &x, int u) {
    unsigned char *sm = x.sm;
    uint64_t *bars = x.bars;
    const int et = threadIdx.x - 384, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dv = 32 * (warp & 3) + lane;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int h = u % a.H_v;
    const int len = x.units[u].len, nchunks = x.units[u].nch;
    const int64_t bos = x.units[u].bos;
    const int64_t sv = (int64_t)a.H_v * 128;
    bf16 *o = static_cast<bf16 *>(a.o);
    bool failed = false;
    for (int c = 0; c < nchunks; ++c) {
        const int b = c % Cons::kBufs;
        unsigned char *stage = sm + b * Slot::kStride + Slot::oWT;  // [64 tok][128 d_v] bf16
        const int nvalid = min(kChunk, len - c * kChunk);
        const uint32_t tO = ((c & 1) ? tX1 : tX0) + 64;
        failed = !wait_bar(&bars[B_O0 + (c & 1)], (uint32_t)((c >> 1) & 1), x.flag, a, pc);
        if (bar_or(3, 128, failed)) { failed = true; break; }
        fence_after_sync();
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            float v[32];
            tmem_ld32(x.tmem + lane_off + tO + 32 * hh, v);
            if (nvalid == kChunk) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    *reinterpret_cast<bf16 *>(stage + (32 * hh + e) * 256 + dv * 2) = __float2bfloat16_rn(v[e] * a.scale);
            } else {
                bf16 *op = o + (bos + (int64_t)c * kChunk + 32 * hh) * sv + (int64_t)h * 128 + dv;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (32 * hh + e < nvalid) op[(int64_t)e * sv] = __float2bfloat16_rn(v[e] * a.scale);
            }
        }
        // The ring slot of this chunk was copied into shared memory long ago (its copy is
        // complete: B_O0 / B_O1 follow the MMAs that read it). Its lines are dropped from L2
        // without being written back to DRAM: the producer that reuses the slot
        // overwrites every byte, and only after this CTA releases it (B_EMPTY, then done[u]).
        {
            const unsigned char *slot = slot_ptr(pc, u, c);
            for (int i = et; i < Slot::kBytes / 128; i += 128) discard_l2(slot + (size_t)i * 128);
        }
        fence_before_sync();
        fence_proxy_async();
        bar_named(3, 128);
        if (et == 0) {
            mbar_arrive(&bars[B_XFREE0 + (c & 1)]);  // the issuer may reuse this D_X buffer
            if (nvalid == kChunk) {
                tma_store_2d(&maps.o, h * 128, (int)(bos + (int64_t)c * kChunk), stage);
                bulk_commit();
                bulk_wait_read();  // the tile has been read: the buffer may be refilled
            }
            mbar_arrive(&bars[B_EMPTY0 + b]);
        }
    }
    if (et == 0) bulk_wait_done();
    if (failed) *x.flag = 1;
}

template <bool GATE_HEAD, bool FE>
__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd_pc_kernel(const FwdArgs a, const __grid_constant__ TcMaps maps, const PcArgs pc) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Common::oBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Common::oTmemAddr);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + Common::oFlag);
    int *stats = reinterpret_cast<int *>(sm + Common::oFlag + 4);  // most chunks, uniform
    volatile int *stored = reinterpret_cast<volatile int *>(sm + Common::oFlag + 12);
    UnitInfo *units = reinterpret_cast<UnitInfo *>(sm + Common::oUnits);
    int *seen = reinterpret_cast<int *>(sm + Common::oSeen);
    volatile int *jobq = reinterpret_cast<volatile int *>(sm + Common::oJobq);
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool consumer = (int)blockIdx.x < pc.U;
    const uint32_t ncols = consumer ? kTmemCons : kTmemProd;

    // unit table: sequence bounds of every unit (a malformed entry becomes len = -1)
    for (int i = tid; i < pc.U; i += kThreads) {
        const int n = i / a.H_v;
        UnitInfo ui;
        if (a.cu_seqlens == nullptr) {
            ui.bos = (long long)n * a.T;
            ui.len = a.T;
        } else {
            const int s = a.cu_seqlens[n], e = a.cu_seqlens[n + 1];
            const bool ok = s >= 0 && e >= s && e <= a.T;
            ui.bos = ok ? s : 0;
            ui.len = ok ? e - s : -1;
        }
        ui.nch = ui.len > 0 ? (ui.len + kChunk - 1) / kChunk : 0;
        units[i] = ui;
    }
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
        *flag = 0;
        *stored = 0;
        for (int i = 0; i < kMaxUnits; ++i) seen[i] = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        int mx = 0, uni = 1;
        for (int i = 0; i < pc.U; ++i) mx = max(mx, units[i].nch);
        for (int i = 0; i < pc.U; ++i) uni &= units[i].nch == mx ? 1 : 0;
        stats[0] = mx;
        stats[1] = uni;
        if (uni && !consumer) {  // this producer's first two jobs
            jobq[0] = atomicAdd(pc.jobs, 1);
            jobq[1] = atomicAdd(pc.jobs, 1);
        }
    }
    __syncthreads();

    Ctx x;
    x.sm = sm;
    x.sbase = smem_u32(sm);
    x.tmem = *tmem_slot;
    x.bars = bars;
    x.flag = flag;
    x.stored = stored;
    x.seen = seen;
    x.jobq = jobq;
    x.units = units;
    x.maxc = stats[0];
    x.uniform = stats[1];
    x.p = (int)blockIdx.x - pc.U;

    uint32_t pend_front = 0;
    int pend_back = 0, pend_load = 0;
    if (consumer) {
        const int u = blockIdx.x;
        if (units[u].len < 0) {
            if (tid == 0) atomicOr(a.err, kDeviceErrSeqlens);  // the unit is skipped, as in every kernel
        } else if (warp < 4 || (warp >= 8 && warp < 12)) {
            consumer_serial(a, pc, x, u);
        } else if (warp < 7) {
            pend_load = consumer_loader(a, pc, x, u, units[u].nch);
        } else if (warp == 7) {
            consumer_issuer(a, pc, x, u);
        } else {
            consumer_epilogue(a, maps, pc, x, u);
        }
    } else if (tid < 256) {
        pend_front = producer_front<GATE_HEAD, FE>(a, maps, pc, x);
    } else {
        pend_back = producer_back(a, maps, pc, x);
    }

    fence_before_sync();
    if (__syncthreads_or(*flag != 0)) {
        // drain: every MMA and copy this CTA issued must land before TMEM is freed and the
        // CTA exits (bounded waits)
        const bool issuer = consumer ? tid == 224 : (tid == 0 || tid == 256);
        if (issuer) {
            fence_after_sync();
            uint64_t *z = &bars[consumer ? B_CZ : (tid == 0 ? B_PZ0 : B_PZ1)];
            commit(z);
            mbar_wait(z, 0, kWaitCycles);
        }
        if (consumer && tid == 128) {
#pragma unroll 1
            for (int bb = 0; bb < Cons::kBufs; ++bb)
                if ((pend_load >> bb) & 1) mbar_wait(&bars[B_FULL0 + bb], (uint32_t)((pend_load >> (4 + bb)) & 1), kWaitCycles);
        }
        if (!consumer && tid == 0) {
            if (pend_front & 1u) mbar_wait(&bars[B_LQK], (pend_front >> 4) & 1u, kWaitCycles);
            if (pend_front & 2u) mbar_wait(&bars[B_LG], (pend_front >> 5) & 1u, kWaitCycles);
        }
        if (!consumer && tid == 256 && pend_back > 0) mbar_wait(&bars[B_LV], (uint32_t)(pend_back - 1), kWaitCycles);
        cp_async_wait_all();
        bulk_wait_done();
        fence_before_sync();
        __syncthreads();
    }
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(x.tmem, ncols);
    }
}

}  // namespace

// Stream-ordered scratch (the ring and flags here, the front-end's prepared tensors, the
// backward's factors) from a pool owned by the library, one per device. The pool keeps up
// to 64 MiB reserved between calls and releases the rest when the device, a stream or an
// event of it is synchronised.
namespace {
constexpr int kMaxDevices = 64;
// Flag words of a launch: ready [U][kFlagLine], done [U][kFlagLine], the abort word and the
// job counter, each on a 128-byte line of its own (R <= kFlagLine).
struct FlagLayout {
    size_t done, abort, jobs, bytes;  // offsets in ints from the ready array; total bytes
};
constexpr FlagLayout flag_layout(size_t U) {
    return FlagLayout{U * kFlagLine, 2 * U * kFlagLine, 2 * U * kFlagLine + kFlagLine,
                      (2 * U * kFlagLine + 2 * kFlagLine) * sizeof(int)};
}
inline void set_flags(PcArgs &pc, int *base, const FlagLayout &f) {
    pc.ready = base;
    pc.done = base + f.done;
    pc.abort = base + f.abort;
    pc.jobs = base + f.jobs;
}

constexpr uint64_t kPoolKeepBytes = 64ull << 20;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};
}  // namespace

cudaError_t scratch_pool(int dev, cudaMemPool_t *out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (g_pool[dev] == nullptr) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        // keep up to kPoolKeepBytes reserved between calls (the forward's ring fits), and give
        // anything above it back at the next synchronisation, such as the backward's scratch
        uint64_t keep = kPoolKeepBytes;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pool[dev] = pool;
    }
    *out = g_pool[dev];
    return cudaSuccess;
}

namespace {

template <bool GATE_HEAD, bool FE>
cudaError_t launch_pc(const FwdArgs &a, cudaStream_t stream, bool *launched) {
    *launched = false;
    int dev = 0, sms = 0, coop = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) return e;
    const int64_t U = (int64_t)a.N * a.H_v;
    // worth it only when the units leave at least as many SMs idle as they occupy
    if (!coop || U < 1 || U > kMaxUnits || 2 * U > sms) return cudaSuccess;
    auto kern = kda_fwd_pc_kernel<GATE_HEAD, FE>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Common::kBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Common::kBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaSuccess;

    TcMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_tile_maps(&maps, a, GATE_HEAD) || !encode_o_map(&maps, a)) return cudaErrorInvalidValue;

    // ring depth: 8 slots per unit at least, deeper for fewer units (about 38 MB, well
    // inside L2), so that producers taking jobs in order rarely wait for a slow consumer
    const int R = (int)std::max<int64_t>(kRing, std::min<int64_t>(4 * kRing, 512 / U));
    static_assert(4 * kRing <= kFlagLine, "a unit's ready words fit its flag line");
    const size_t ring_bytes = (size_t)U * R * Slot::kStride;
    const FlagLayout fl = flag_layout((size_t)U);
    const size_t flag_bytes = (fl.bytes + 255) & ~(size_t)255;
    cudaMemPool_t pool = nullptr;
    e = scratch_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    void *buf = nullptr;
    e = cudaMallocFromPoolAsync(&buf, ring_bytes + flag_bytes, pool, stream);
    if (e != cudaSuccess) return e;
    PcArgs pc;
    pc.ring = static_cast<unsigned char *>(buf);
    set_flags(pc, reinterpret_cast<int *>(pc.ring + ring_bytes), fl);
    pc.U = (int)U;
    pc.P = sms - (int)U;
    pc.R = R;
    e = cudaMemsetAsync(pc.ready, 0, flag_bytes, stream);
    if (e == cudaSuccess) {
        void *args[] = {const_cast<FwdArgs *>(&a), &maps, &pc};
        e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(sms), dim3(kThreads), args,
                                        Common::kBytes, stream);
        if (e == cudaSuccess) *launched = true;
    }
    const cudaError_t ef = cudaFreeAsync(buf, stream);
    return e != cudaSuccess ? e : ef;
}

// ---- the variant without allocation: scratch in a file-scope device array ----------------
// Room for kStaticUnits units with kRing slots each, and their flags. Calls that use it must
// not overlap (on any stream or thread): they share this one array.
constexpr int kStaticUnits = 16;
constexpr size_t kStaticRingBytes = (size_t)kStaticUnits * kRing * Slot::kStride;      // 9,568,256 B
constexpr size_t kStaticFlagBytes = 4352;
static_assert(flag_layout((size_t)kStaticUnits).bytes <= kStaticFlagBytes, "flag room");
static __device__ __align__(256) unsigned char g_static_scratch[kStaticRingBytes + kStaticFlagBytes];

std::mutex g_static_mu;
unsigned char *g_static_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device, looked up once per device.
cudaError_t static_scratch(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_static_ptr[dev];
    return cudaSuccess;
}

template <bool GATE_HEAD>
cudaError_t launch_pc_static(const FwdArgs &a, cudaStream_t stream) {
    const int64_t U = (int64_t)a.N * a.H_v;
    if (U < 1 || U > kStaticUnits) return cudaErrorNotSupported;
    int dev = 0, sms = 0, coop = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) return e;
    if (!coop || 2 * U > sms) return cudaErrorNotSupported;
    auto kern = kda_fwd_pc_kernel<GATE_HEAD, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Common::kBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Common::kBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;

    TcMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_tile_maps(&maps, a, GATE_HEAD) || !encode_o_map(&maps, a)) return cudaErrorInvalidValue;

    unsigned char *base = nullptr;
    e = static_scratch(dev, &base);
    if (e != cudaSuccess) return e;
    PcArgs pc;
    pc.ring = base;
    set_flags(pc, reinterpret_cast<int *>(base + kStaticRingBytes), flag_layout((size_t)U));
    pc.U = (int)U;
    pc.P = sms - (int)U;
    pc.R = kRing;
    // the flags start at zero for every call; the slots need no clearing
    e = cudaMemsetAsync(pc.ready, 0, kStaticFlagBytes, stream);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<FwdArgs *>(&a), &maps, &pc};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(sms), dim3(kThreads), args,
                                       Common::kBytes, stream);
}

}  // namespace

// The persistent kernel when the call has at most half as many units as the device has
// SMs; *launched tells whether it ran (otherwise nothing was launched). The front-end
// parts that `a` switches on are applied inside the kernel.
cudaError_t launch_fwd_pc(const FwdArgs &a, cudaStream_t stream, bool *launched) {
    if (fe_any(a))
        return a.gate_per_head ? launch_pc<true, true>(a, stream, launched) : launch_pc<false, true>(a, stream, launched);
    return a.gate_per_head ? launch_pc<true, false>(a, stream, launched) : launch_pc<false, false>(a, stream, launched);
}

// The same kernel with its scratch in g_static_scratch (nothing allocated), per-channel
// gates only. Returns cudaErrorNotSupported, with nothing launched, when the call has more
// than kStaticUnits units, more units than half the SMs, per-head gates, or the device
// cannot launch it cooperatively.
cudaError_t launch_fwd_pc_static(const FwdArgs &a, cudaStream_t stream) {
    // the entry point that uses it always passes per-channel gates
    if (a.gate_per_head) return cudaErrorNotSupported;
    return launch_pc_static<false>(a, stream);
}

int pc_static_max_units() { return kStaticUnits; }

}  // namespace kda
