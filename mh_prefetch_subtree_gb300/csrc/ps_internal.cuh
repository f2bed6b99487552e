// Internal declarations shared by the libps translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ps.h"

namespace ps {

// ---------------------------------------------------------------------------
// Scoring kernel geometry (K1).  Each warp streams its own contiguous range of
// row chunks through a private ring of shared-memory stages filled by 1-D bulk
// copies, then takes tail blocks of the remaining chunks until none is left;
// see ps_score_rows.cu.
// ---------------------------------------------------------------------------
constexpr int kWarpsPerCta = 16;
constexpr int kStages = 2;
constexpr int kStageBytes = 4096;
constexpr int kMaxCtas = 2048;                        // workspace sizing bound
// chunk ranges (warps' own ranges and tail blocks, plus the claim counter)
// that a workspace holds split-row partials and counters for
constexpr int kMaxRanges = kMaxCtas * kWarpsPerCta;

// Partial log-sum-exp state of (part of) a row: with y = l*log2e - R, the
// sums of 2^y, 2^(g*y) and 2^y * y over the row's elements except the token,
// plus the token's logit when this part held it (a marker NaN otherwise).
struct __align__(16) RowPart {
    float R;
    float s1;
    float st;       // tau sum (multi-temperature: the sum of 2^(2y))
    float ltok;
    float y1;
    float st1;      // multi-temperature: sums of 2^(4y) and 2^(8y)
    float st2;
    float pad;
};

struct RowsParams {
    const uint8_t *logits;
    int64_t ld_bytes;
    int64_t n_logit_rows;
    const int64_t *row_index;
    const int32_t *tokens;
    int64_t n_rows;
    int32_t V;
    int32_t dtype;              // PS_BF16 / PS_F32
    int32_t flags;              // PS_FLAG_* hints of the batch
    int32_t row_bytes;          // V * elem rounded up to 16
    int32_t cpr;                // chunks per row
    int64_t n_chunks;           // n_rows * cpr
    int32_t n_vwarps;           // warps, each owning one static chunk range
    int64_t n_static;           // the static ranges cover chunks [0, n_static)
    int64_t tail_chunks;        // chunks per tail block (0 when there are none)
    int32_t n_tail;             // tail blocks over [n_static, n_chunks)
    int32_t *claim;             // tail blocks taken so far; zero at launch
    int32_t npow;               // 1/tau when it is 1, 2, 4 or 8; 16 (17): several
                                // temperatures with 1/tau in {1, 2, 4, 8} ({1, 2, 4}),
                                // listed in tau_pow; else 0
    float g;                    // 1/tau in float
    int32_t n_taus;             // multi-temperature: number of temperatures (1..4)
    int32_t tau_pow[4];         // multi-temperature: 1/tau of each
    double *lq_multi;           // multi-temperature: [n_taus][n_rows]
    double *lp0;
    double *lq;
    double *entropy;            // optional: entropy of p0 per row
    RowPart *parts;             // [2 * (n_vwarps + n_tail)], two per chunk range
    int32_t *counters;          // [n_vwarps + n_tail], one per chunk range
    int32_t *status;
};

struct AssembleParams {
    int32_t T;
    int32_t n_chains;
    int32_t n_seg;
    int64_t n_rows;
    double alpha;
    double eps;
    const int32_t *chain_seg0;
    const int64_t *seg_row0;
    const int32_t *seg_cut;
    const int32_t *seg_src;
    const double *lp0;
    const double *lq;
    const double *root_lp0;     // optional carried values of the roots [n_chains][T]
    const double *root_lq;
    double *lp_y, *lq_y, *lp_x, *lq_x, *log_ratio, *log_accept;
    int8_t *eps_class;
    int32_t *status;
};

struct CarryParams {
    int32_t T;
    int32_t n_chains;
    int32_t n_seg;
    int64_t n_rows;
    const int32_t *chain_seg0;
    const int64_t *seg_row0;
    const int32_t *seg_cut;
    const int32_t *seg_src;
    ps_carry_io io;
};

struct WalkParams {
    int32_t n_chains;
    int32_t n_nodes;
    int32_t n_seg;
    int32_t max_steps;
    const int32_t *chain_node0;
    const int32_t *chain_seg0;
    const int32_t *acc, *rej, *req;
    const double *u;
    const double *log_accept;
    int32_t *state_seg, *end_node, *k_delta, *path;
    int32_t *status;
};

// Launchers (host side, asynchronous on `stream`).  The assemble, walk and
// carry kernels are launched with programmatic stream serialization, so each
// may start while its predecessor in the stream finishes; they wait
// (griddepcontrol.wait) before their first load of any input, because the
// predecessor may be the caller's own kernel writing those inputs.
cudaError_t launch_score_rows(const RowsParams &p, int n_ctas, cudaStream_t stream);
cudaError_t launch_assemble(const AssembleParams &p, cudaStream_t stream);
// Suffix sums and log A, then each chain's walk by the last CTA of the chain to
// finish; chain_cnt [n_chains] must be zero at launch.  early: the previous
// kernel in the stream is libps's own scoring kernel of the same call, so the
// layout arrays may be read before griddepcontrol.wait.
cudaError_t launch_assemble_walk(const AssembleParams &p, const WalkParams &wp,
                                 int32_t *chain_cnt, bool early, cudaStream_t stream);
cudaError_t launch_walk(const WalkParams &p, cudaStream_t stream);
cudaError_t launch_carry(const CarryParams &p, cudaStream_t stream);
size_t score_rows_smem_bytes();
// Diagnostic: a bounded wait on an mbarrier that nothing completes.
cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t *status, cudaStream_t stream);
// Diagnostic: a plain streaming read of n_vec 16-byte words, folded into *sink.
cudaError_t launch_read_probe(const void *data, int64_t n_vec, uint32_t *sink, int sms,
                              cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: spins on try_wait (which itself suspends for a short,
// hardware-chosen time) and gives up after `limit_ns` of wall time, or after
// 2^28 polls whatever the timer says.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 28); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// L2 policy for data read exactly once: evict it first, so that the small
// arrays the next kernels read stay cached.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier, with an
// L2 cache policy.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Hardware base-2 exponential (MUFU), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

#endif  // __CUDACC__

}  // namespace ps
