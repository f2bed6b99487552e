// K1: per-token log p0 and log q_tau of every scored row, in one pass over
// the row's logits (PreSTO, Appendix B.1 last paragraph and Appendix D.3:
// both log-probabilities come from the same logits, without and with the
// temperature), and optionally the full-vocabulary entropy of p0 (Appendix
// D.3, quantity (iii)) from the same pass.
//
// Formulation.  For a row l_0..l_{V-1} with token k, and any reference R
// (log2 units), with L = log2(e), g = 1/tau and y_j = l_j L - R:
//     S1 = sum_{j != k} 2^y_j,   St = sum_{j != k} 2^(g y_j),
//     Y1 = sum_{j != k} 2^y_j y_j  (entropy only),   t = l_k L - R,
//     log p0(k)    = -ln(1 + S1 2^-t),  log q_tau(k) = -ln(1 + St 2^(-g t)),
//     H(p0)        = ln 2 (log2 Z - (Y1 + t 2^t) / Z),  Z = S1 + 2^t.
// This is log softmax written relative to the token itself, so the token is
// left out of the sums and the result keeps its relative accuracy when the
// token holds nearly all the mass (the sums are then tiny, never 1 + tiny).
// No maximum is needed: R only has to keep the exponentials in range.  Each
// lane starts with R = -inf; a chunk whose sums overflow (or are NaN) takes a
// slow path that raises R to the chunk's maximum and rescales.  (The entropy
// variant keeps one R per warp and raises it whenever a chunk holds a logit
// above it, so that a dominant logit is added close to R.)  When 1/tau is
// 1, 2, 4 or 8 the tau exponential is the first one squared, so each logit
// costs one MUFU ex2; the same squaring chain serves up to four such
// temperatures in one pass (multi-temperature scoring).
//
// Data movement.  The rows are cut into chunks of one stage (the last chunk of
// a row may be shorter).  The chunk sequence of all rows is split into
// contiguous ranges, one per warp, so every warp streams about the same number
// of bytes whatever the row count.  In the variants without entropy, on large
// batches, those ranges cover the first 15/16 of the sequence only; the rest
// is cut into small tail blocks, which the warps that finish their own range
// first take one at a time (an atomic counter), so that SMs that read a
// little slower than the others do not decide when the kernel ends.  Each
// warp owns a ring of shared-memory stages that its lane 0 fills with 1-D bulk
// copies (cp.async.bulk, completion on an mbarrier, L2 evict-first since every
// byte is read once); the warp consumes a stage, refills it, and moves on.
// There is no block-wide synchronisation.  Before a stage is read, lane 0
// overwrites the row's token logit (after saving it) and any padding beyond V
// with -inf (in the entropy variant with -1e30, which adds nothing either but
// keeps 2^y y finite on the clamp-free fast path).
//
// A row whose chunks all lie in one range is finalised by the warp that reads
// that range.  A row split across ranges leaves one partial per range in the
// workspace; the last warp to arrive (atomic counter) merges them in range
// order and finalises.  Results are deterministic: they do not depend on
// which warp read which tail block.
#include <math.h>

#include "ps_internal.cuh"

namespace ps {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLimit = 1.8446744073709552e19f;   // 2^64: largest chunk sum kept as is
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s for one bulk copy
constexpr uint64_t kDrainLimitNs = 1000000000ull;
constexpr uint32_t kAbsent = 0x7fc0deadu;           // "token not in this part" (a NaN payload
                                                    // no bf16/f32 logit converts to)
// Entropy variant: logits below -1e30 (that is, -inf) are raised to -1e30, so
// that 2^y * y is 0 * (finite) = 0 instead of 0 * (-inf) = NaN.  The exponential
// of such a value is 0 either way; NaN is kept (the max propagates it).
constexpr uint32_t kFloorBf16x2 = 0xf14af14au;      // (-1.0009e30, -1.0009e30) as bf16x2
constexpr float kFloorF32 = -1.0e30f;

// Warp w's chunk range is [range_begin(w), range_begin(w + 1)).
__device__ __forceinline__ int64_t range_begin(int64_t w, int64_t C, int64_t W) {
    return (w * C) / W;
}

// The warp whose chunk range holds chunk c (all ranges are non-empty: W <= C).
__device__ __forceinline__ int64_t warp_of_chunk(int64_t c, int64_t C, int64_t W) {
    int64_t w = (c * W) / C;
    if (w >= W) w = W - 1;
    while (w + 1 < W && range_begin(w + 1, C, W) <= c) ++w;
    while (w > 0 && range_begin(w, C, W) > c) --w;
    return w;
}

// Chunk ranges with tail blocks.  Ranges 0..W-1 (W = n_vwarps) split chunks
// [0, n_static) as above, one per warp; ranges W..W+n_tail-1 are the tail
// blocks of tail_chunks chunks each over [n_static, n_chunks), taken at run
// time by whichever warps finish their own range first.  Every range is
// non-empty, and tail_range_begin(W + n_tail) = n_chunks.
__device__ __forceinline__ int64_t tail_range_begin(const RowsParams &p, int64_t r) {
    const int64_t W = p.n_vwarps;
    if (r > W) return min(p.n_chunks, p.n_static + (r - W) * p.tail_chunks);
    return range_begin(r, p.n_static, W);
}

// The range that holds chunk c.
__device__ __forceinline__ int64_t tail_range_of_chunk(const RowsParams &p, int64_t c) {
    if (c >= p.n_static) return p.n_vwarps + (c - p.n_static) / p.tail_chunks;
    return warp_of_chunk(c, p.n_static, p.n_vwarps);
}

template <int DT>
struct Elem;
template <>
struct Elem<PS_BF16> {
    static constexpr int kSize = 2;
    static constexpr uint32_t kNegInfWord = 0xff80ff80u;
    static constexpr uint32_t kFloorWord = 0xf14af14au;   // two bf16 -1.0009e30
    static constexpr uint16_t kFloorElem = 0xf14au;
};
template <>
struct Elem<PS_F32> {
    static constexpr int kSize = 4;
    static constexpr uint32_t kNegInfWord = 0xff800000u;
    static constexpr uint32_t kFloorWord = 0xf149f2cau;   // -1.0e30f
};
// Values at or below this are taken as absent (-inf) when the maximum is sought.
constexpr float kAbsentBelow = -9.0e29f;

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// NP == kAllPowers or kPowersTo4: one pass serves several temperatures whose
// 1/tau is 1, 2, 4 or 8 (the MultiTryMH set {0.25, 0.5, 1} among them): from
// 2^y the powers 2^(2y), 2^(4y) (and, for kAllPowers, 2^(8y)) are squares,
// and their sums are kept side by side.
constexpr int kAllPowers = 16;     // sums of 2^(2y), 2^(4y), 2^(8y)
constexpr int kPowersTo4 = 17;     // sums of 2^(2y), 2^(4y)

template <int NP>
__host__ __device__ constexpr bool multi_tau() { return NP == kAllPowers || NP == kPowersTo4; }

template <int NP>
__host__ __device__ constexpr int n_tau_sums() {
    return NP == kAllPowers ? 3 : (NP == kPowersTo4 ? 2 : 1);
}

// Running sums of one lane (or one merged part) relative to reference R.
// st[k] is the tau sum (multi-temperature: the sum of 2^(2^(k+1) y)).
struct Acc {
    float R;
    float s1;
    float st[3];
    float y1;
};

__device__ __forceinline__ Acc acc_empty() { return Acc{-INFINITY, 0.f, {0.f, 0.f, 0.f}, 0.f}; }

// One pair of logits v: accumulate 2^x into a1, 2^(g x) into at[0] (or the
// three power sums into at[0..2]) and 2^x x into ay, with x = v L - R.  For a
// general g the tau exponent g x = v (g L) - g R is formed from v directly
// (GL2, nGR2), so that it does not wait for x.
template <int NP, bool ENT>
__device__ __forceinline__ void step2(float2 v, float2 L2, float2 nR2, float2 GL2, float2 nGR2,
                                      float2 &a1, float2 (&at)[3], float2 &ay) {
    const float2 x = __ffma2_rn(v, L2, nR2);
    const float2 e = make_float2(ex2(x.x), ex2(x.y));
    a1 = __fadd2_rn(a1, e);
    if constexpr (ENT) ay = __ffma2_rn(e, x, ay);
    if constexpr (NP == 2) {
        at[0] = __fadd2_rn(at[0], __fmul2_rn(e, e));
    } else if constexpr (NP == 4) {
        const float2 e2 = __fmul2_rn(e, e);
        at[0] = __fadd2_rn(at[0], __fmul2_rn(e2, e2));
    } else if constexpr (NP == 8) {
        const float2 e2 = __fmul2_rn(e, e);
        const float2 e4 = __fmul2_rn(e2, e2);
        at[0] = __fadd2_rn(at[0], __fmul2_rn(e4, e4));
    } else if constexpr (multi_tau<NP>()) {
        const float2 e2 = __fmul2_rn(e, e);
        const float2 e4 = __fmul2_rn(e2, e2);
        at[0] = __fadd2_rn(at[0], e2);
        at[1] = __fadd2_rn(at[1], e4);
        if constexpr (NP == kAllPowers) at[2] = __fadd2_rn(at[2], __fmul2_rn(e4, e4));
    } else if constexpr (NP == 0) {
        const float2 xt = __ffma2_rn(v, GL2, nGR2);
        at[0] = __fadd2_rn(at[0], make_float2(ex2(xt.x), ex2(xt.y)));
    }
}

__device__ __forceinline__ float hsum4(const float2 (&a)[4]) {
    const float2 s01 = __fadd2_rn(a[0], a[1]), s23 = __fadd2_rn(a[2], a[3]);
    const float2 s = __fadd2_rn(s01, s23);
    return s.x + s.y;
}

// Sums of one lane's VPL vectors relative to reference R: c1, ct[0..NS-1], cy.
// CLAMP (entropy only) raises -inf inputs to a large negative finite value
// first, so that 2^y y is 0 rather than NaN there; without it the caller must
// see to it that no -inf is in q (a NaN sum sends the chunk down the slow path).
template <int DT, int NP, bool ENT, int VPL, bool CLAMP = ENT>
__device__ __forceinline__ void sum_vecs(const uint4 (&q)[VPL], float R, float g, float &c1,
                                         float (&ct)[3], float &cy) {
    const float2 L2 = make_float2(kLog2e, kLog2e);
    const float2 nR2 = make_float2(-R, -R);
    const float2 GL2 = make_float2(g * kLog2e, g * kLog2e);
    const float2 nGR2 = make_float2(-g * R, -g * R);
    float2 a1[4], at[4][3], ay[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        a1[j] = make_float2(0.f, 0.f);
        at[j][0] = at[j][1] = at[j][2] = make_float2(0.f, 0.f);
        ay[j] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
        if constexpr (DT == PS_BF16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (ENT && CLAMP) w[j] = max_nan_bf16x2(w[j], kFloorBf16x2);
                const float2 v = make_float2(__uint_as_float(w[j] << 16),
                                             __uint_as_float(w[j] & 0xffff0000u));
                step2<NP, ENT>(v, L2, nR2, GL2, nGR2, a1[j], at[j], ay[j]);
            }
        } else {
            float f[4] = {__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]),
                          __uint_as_float(w[3])};
            if constexpr (ENT && CLAMP) {
#pragma unroll
                for (int j = 0; j < 4; ++j) f[j] = max_nan_f32(f[j], kFloorF32);
            }
            step2<NP, ENT>(make_float2(f[0], f[1]), L2, nR2, GL2, nGR2, a1[(i & 1) * 2],
                           at[(i & 1) * 2], ay[(i & 1) * 2]);
            step2<NP, ENT>(make_float2(f[2], f[3]), L2, nR2, GL2, nGR2, a1[(i & 1) * 2 + 1],
                           at[(i & 1) * 2 + 1], ay[(i & 1) * 2 + 1]);
        }
    }
    c1 = hsum4(a1);
    if constexpr (NP == 1) {
        ct[0] = c1;
    } else {
#pragma unroll
        for (int k = 0; k < n_tau_sums<NP>(); ++k) {
            const float2 t[4] = {at[0][k], at[1][k], at[2][k], at[3][k]};
            ct[k] = hsum4(t);
        }
    }
    cy = ENT ? hsum4(ay) : 0.f;
}

// Rescale factor of tau sum k when the reference moves by d (log2 units).
template <int NP>
__device__ __forceinline__ float tau_scale(float d, float g, int k) {
    if constexpr (NP == 0) return ex2(d * g);
    else if constexpr (multi_tau<NP>()) return ex2(d * (float)(2 << k));
    else return ex2(d * (float)NP);
}

// Moves the reference of `a` from a.R to Rn >= a.R.  With y' = y - D,
// D = Rn - R: sum 2^y' = 2^-D S1 and sum 2^y' y' = 2^-D (Y1 - D S1).
template <int NP, bool ENT>
__device__ __forceinline__ Acc rebase(Acc a, float Rn, float g) {
    if (a.R == -INFINITY) {            // empty so far (or only -inf): nothing to move
        a.R = Rn;
        return a;
    }
    const float d = a.R - Rn;          // <= 0
    const float f = ex2(d);
    if constexpr (ENT) a.y1 = f * fmaf(d, a.s1, a.y1);
    a.s1 *= f;
    if constexpr (NP != 1) {
#pragma unroll
        for (int k = 0; k < n_tau_sums<NP>(); ++k) a.st[k] *= tau_scale<NP>(d, g, k);
    }
    a.R = Rn;
    return a;
}

// Load one lane's VPL vectors of a stage; vectors past the chunk read as -inf
// (or, with FLOOR, as the large negative finite floor).
template <int DT, int VPL, bool FLOOR = false>
__device__ __forceinline__ void load_vecs(const uint4 *v4, int nvec, int lane,
                                          uint4 (&q)[VPL]) {
    if (nvec == VPL * 32) {                    // a full chunk: no predication
#pragma unroll
        for (int i = 0; i < VPL; ++i) q[i] = v4[lane + 32 * i];
        return;
    }
    const uint32_t ni = FLOOR ? Elem<DT>::kFloorWord : Elem<DT>::kNegInfWord;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int idx = lane + 32 * i;
        q[i] = idx < nvec ? v4[idx] : make_uint4(ni, ni, ni, ni);
    }
}

// Adds a chunk's sums to the running ones.
template <int NP, bool ENT>
__device__ __forceinline__ void add_chunk(Acc &a, float c1, const float (&ct)[3], float cy) {
    a.s1 += c1;
    if constexpr (NP != 1) {
#pragma unroll
        for (int k = 0; k < n_tau_sums<NP>(); ++k) a.st[k] += ct[k];
    }
    if constexpr (ENT) a.y1 += cy;
}

// The largest of a chunk's sums (the one that overflows first).
template <int NP>
__device__ __forceinline__ float chunk_peak(float c1, const float (&ct)[3]) {
    return fmaxf(c1, ct[n_tau_sums<NP>() - 1]);
}

// Rare path: the chunk's sums overflowed or were NaN (always the case for a
// lane's first chunk of a row, whose reference is still -inf).  Re-reads the
// lane's vectors from shared memory, raises R to their maximum (for the
// entropy variant, which calls it on all lanes at once, to the warp's
// maximum), rescales the running sums and adds the chunk.
template <int DT, int NP, bool ENT, int VPL>
__device__ __noinline__ Acc slow_chunk(const uint4 *v4, int nvec, int lane, float g, Acc a) {
    uint4 q[VPL];
    load_vecs<DT, VPL>(v4, nvec, lane, q);
    float m = -INFINITY;
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (DT == PS_BF16) {
                float lo = __uint_as_float(w[j] << 16);
                float hi = __uint_as_float(w[j] & 0xffff0000u);
                nan_seen |= (lo != lo) | (hi != hi);
                if constexpr (ENT) {          // patched entries hold the floor
                    lo = lo > kAbsentBelow ? lo : -INFINITY;
                    hi = hi > kAbsentBelow ? hi : -INFINITY;
                }
                m = fmaxf(m, fmaxf(lo, hi));
            } else {
                float v = __uint_as_float(w[j]);
                nan_seen |= (v != v);
                if constexpr (ENT) v = v > kAbsentBelow ? v : -INFINITY;
                m = fmaxf(m, v);
            }
        }
    }
    if constexpr (ENT) {
        // every lane is here (the caller votes): one reference for the warp
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    if (nan_seen) {
        const float qn = __int_as_float(0x7fc00000);
        a.s1 = a.y1 = qn;
        a.st[0] = a.st[1] = a.st[2] = qn;
        return a;
    }
    const float Rn = fmaxf(a.R, m * kLog2e);
    if (Rn == -INFINITY) return a;     // only -inf so far: nothing to add
    if (Rn > a.R) a = rebase<NP, ENT>(a, Rn, g);
    float c1, ct[3], cy;
    sum_vecs<DT, NP, ENT, VPL>(q, a.R, g, c1, ct, cy);
    add_chunk<NP, ENT>(a, c1, ct, cy);
    return a;
}

// Merge part b into a (each relative to its own reference).
template <int NP, bool ENT>
__device__ __forceinline__ Acc merge_part(Acc a, Acc b, float g) {
    const float M = fmaxf(a.R, b.R);
    if (M == -INFINITY) {              // both parts saw only -inf logits
        a.s1 += b.s1;                  // keeps a NaN poison, else 0
        a.st[0] += b.st[0];
        a.st[1] += b.st[1];
        a.st[2] += b.st[2];
        a.y1 += b.y1;
        return a;
    }
    a = rebase<NP, ENT>(a, M, g);
    b = rebase<NP, ENT>(b, M, g);
    const float z[3] = {b.st[0], b.st[1], b.st[2]};
    add_chunk<NP, ENT>(a, b.s1, z, b.y1);
    return a;
}

template <int NP, bool ENT>
__device__ __forceinline__ Acc warp_merge(Acc a, float g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Acc b;
        b.R = __shfl_xor_sync(0xffffffffu, a.R, off);
        b.s1 = __shfl_xor_sync(0xffffffffu, a.s1, off);
#pragma unroll
        for (int k = 0; k < 3; ++k)
            b.st[k] = (NP != 1 && k < n_tau_sums<NP>())
                          ? __shfl_xor_sync(0xffffffffu, a.st[k], off) : 0.f;
        b.y1 = ENT ? __shfl_xor_sync(0xffffffffu, a.y1, off) : 0.f;
        a = merge_part<NP, ENT>(a, b, g);
    }
    return a;
}

// -ln(1 + 2^a) in float64 (the value is computed in float, except for the tiny
// tail, whose magnitude is below float's range).
__device__ __forceinline__ double neg_log1p_exp2(float a) {
    if (a > 24.f) return -(double)(a * kLn2f + log1pf(exp2f(-a)));
    if (a > -120.f) return -(double)log1pf(exp2f(a));
    return -exp2((double)a);
}

// Entropy in nats from S1, Y1 (the sums without the token) and the token's
// exponent t, all relative to the same reference (the general form, for
// shifts outside the range the fast form handles).
__device__ double entropy_nats_wide(double s1, double y1, double t) {
    const bool tok = t != -INFINITY;
    const double m = fmax(tok ? t : -INFINITY, log2(s1));
    const double et = tok ? exp2(t - m) : 0.0;
    const double zs = s1 * exp2(-m) + et;
    const double ms = y1 * exp2(-m) + (tok ? t * et : 0.0);
    return 0.6931471805599453 * (m + log2(zs) - ms / zs);
}

// The same with an integer shift m >= every exponent (m = ceil(max(t,
// log2 S1))): Z = S1 2^-m + 2^(t-m) lies in (1/2, 2] and
//     D = sum_j 2^(y_j - m) (m - y_j) = m Z - (Y1 2^-m + t 2^(t-m)) >= 0,
//     H = ln 2 (log2 Z + D / Z).
// D is formed in float64, since it is a difference of nearly equal terms when
// one logit holds most of the mass; log2 Z and D / Z carry only float relative
// error, so they are taken in float.  Few float64 operations: GB300's FP64
// pipe is narrow, and this runs once per row.
__device__ double entropy_nats(float s1, float y1, float t) {
    const bool tok = t != -INFINITY;
    // no other finite logit: the token holds all the mass (its exponent is +inf
    // then, since the reference never left -inf)
    if (!(s1 > 0.f)) return tok ? 0.0 : __longlong_as_double(0x7ff8000000000000ll);
    const float m = ceilf(fmaxf(tok ? t : -INFINITY, log2f(s1)));
    if (!(fabsf(m) < 1000.f))
        return entropy_nats_wide((double)s1, (double)y1, tok ? (double)t : -INFINITY);
    const double sc = __longlong_as_double((long long)(1023 - (int)m) << 52);   // 2^-m
    const double et = tok ? (double)exp2f(t - m) : 0.0;
    const double zs = fma((double)s1, sc, et);
    const double ms = fma((double)y1, sc, tok ? (double)t * et : 0.0);
    const double d = fma((double)m, zs, -ms);
    const float zf = (float)zs;
    return 0.6931471805599453 * ((double)log2f(zf) + (double)((float)d / zf));
}

template <int NP, bool ENT>
__device__ void finalize_row(const RowsParams &p, int64_t r, Acc a, float lt, bool bad) {
    double o0, oq = 0.0, h = 0.0;
    const double qnan = __longlong_as_double(0x7ff8000000000000ll);
    if constexpr (NP == 1) a.st[0] = a.s1;
    bool nonfinite = false;
    if (bad || __float_as_uint(lt) == kAbsent) {
        o0 = oq = h = qnan;
        nonfinite = true;          // already flagged (token or row index)
        if constexpr (multi_tau<NP>())
            for (int k = 0; k < p.n_taus; ++k) p.lq_multi[(int64_t)k * p.n_rows + r] = qnan;
    } else {
        const float t = fmaf(lt, kLog2e, -a.R);
        nonfinite = (lt != lt) || (lt == INFINITY) || (a.R != a.R) || (a.s1 != a.s1) ||
                    (a.st[0] != a.st[0]) || (a.st[n_tau_sums<NP>() - 1] !=
                                             a.st[n_tau_sums<NP>() - 1]) ||
                    (a.R == INFINITY) || (t != t) || (ENT && (a.y1 != a.y1));
        if (nonfinite) {
            set_status(p.status, PS_DEV_NONFINITE);
            o0 = oq = h = qnan;
            if constexpr (multi_tau<NP>())
                for (int k = 0; k < p.n_taus; ++k) p.lq_multi[(int64_t)k * p.n_rows + r] = qnan;
        } else {
            o0 = neg_log1p_exp2(a.s1 > 0.f ? log2f(a.s1) - t : -INFINITY);
            if constexpr (NP == 1) {
                oq = o0;
            } else if constexpr (multi_tau<NP>()) {
                for (int k = 0; k < p.n_taus; ++k) {
                    const int pw = p.tau_pow[k];           // 1/tau: 1, 2, 4 or 8
                    const float sk = pw == 1 ? a.s1 : (pw == 2 ? a.st[0] : (pw == 4 ? a.st[1] : a.st[2]));
                    p.lq_multi[(int64_t)k * p.n_rows + r] =
                        neg_log1p_exp2(sk > 0.f ? log2f(sk) - t * (float)pw : -INFINITY);
                }
            } else {
                const float gt = (NP == 0) ? t * p.g : t * (float)NP;
                oq = neg_log1p_exp2(a.st[0] > 0.f ? log2f(a.st[0]) - gt : -INFINITY);
            }
            if constexpr (ENT) {
                // a token logit of -inf has no mass: t = -inf leaves it out
                h = entropy_nats(a.s1, a.y1, lt == -INFINITY ? -INFINITY : t);
            }
        }
    }
    p.lp0[r] = o0;
    if constexpr (!multi_tau<NP>()) p.lq[r] = oq;
    if constexpr (ENT) p.entropy[r] = h;
}

// WARPS warps per CTA, each with a ring of STAGES stages of SB bytes.  CF
// (entropy only): clamp -inf in the fast path too (PS_FLAG_MASKED_LOGITS).
template <int DT, int NP, bool ENT, int WARPS, int STAGES, int SB, bool CF>
__global__ void __launch_bounds__(WARPS * 32, 1) score_rows_kernel(const RowsParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kWarpsPerCta = WARPS;
    constexpr int kStages = STAGES;
    constexpr int kStageBytes = SB;
    constexpr int kVecPerLane = SB / 16 / 32;
    static_assert(SB % 512 == 0, "a stage holds a whole number of 16-byte vectors per lane");
    constexpr int kEsz = Elem<DT>::kSize;
    constexpr int kElemsPerStage = kStageBytes / kEsz;
    // With entropy, sum 2^y y cancels against S1 log2 S1 when one logit holds
    // most of the mass, so its float error grows with the distance between
    // the reference and the largest logit.  The entropy variant therefore
    // keeps one reference for the whole warp, and a chunk in which any lane's
    // sum exceeds the lane's element count (which needs an element above the
    // reference) takes the slow path on all lanes, raising the reference to
    // the chunk's maximum: the largest terms are added within log2(count) of
    // the reference.  A warp-wide reference tracks the row's running maximum,
    // so this happens on few chunks.
    constexpr float kEntLimit = (float)(kVecPerLane * 16 / kEsz);
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t W = p.n_vwarps;
    const int64_t vw = (int64_t)blockIdx.x * kWarpsPerCta + wid;
    if (vw >= W) return;
    const int64_t C = p.n_chunks;
    const int64_t cb = range_begin(vw, C, W);
    const int64_t ce = range_begin(vw + 1, C, W);
    const int32_t cpr = p.cpr;
    const float g = p.g;

    uint8_t *stage = smem + (size_t)wid * kStages * kStageBytes;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + (size_t)kWarpsPerCta * kStages * kStageBytes) +
        wid * kStages;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = l2_evict_first_policy();   // logits are read once

    // ---- issue side: next chunk to copy and a lane-parallel cache of row_index
    int64_t ic = cb;
    int64_t irow = cb / cpr;
    int32_t ik = (int32_t)(cb - irow * cpr);
    int64_t ri_base = -1;
    int64_t ri_reg = 0;
    auto src_row_of = [&](int64_t row) -> int64_t {   // warp-collective
        if (p.row_index == nullptr) return row;
        if (ri_base < 0 || row >= ri_base + 32 || row < ri_base) {
            ri_base = row;
            const int64_t rr = row + lane;
            ri_reg = rr < p.n_rows ? __ldg(p.row_index + rr) : 0;
        }
        int64_t s = __shfl_sync(0xffffffffu, ri_reg, (int)(row - ri_base));
        if (s < 0 || s >= p.n_logit_rows) s = 0;      // flagged on the consume side
        return s;
    };
    auto issue_next = [&](int s) {                    // warp-collective
        const int64_t srow = src_row_of(irow);
        if (lane == 0) {
            const uint32_t off = (uint32_t)ik * kStageBytes;
            const uint32_t bytes = min((uint32_t)kStageBytes, (uint32_t)p.row_bytes - off);
            const uint8_t *src = p.logits + srow * p.ld_bytes + off;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(stage + (size_t)s * kStageBytes, src, bytes, &bars[s], policy);
        }
        ++ic;
        if (++ik == cpr) {
            ik = 0;
            ++irow;
        }
    };
#pragma unroll
    for (int s = 0; s < kStages; ++s)
        if (ic < ce) issue_next(s);

    // ---- consume side
    int64_t row = cb / cpr;
    int32_t k = (int32_t)(cb - row * cpr);
    int64_t tb = -1;
    int32_t tok_reg = 0;
    int64_t rib_reg = 0;
    int32_t tok = 0;
    bool bad = false;
    auto row_start = [&]() {                          // warp-collective
        if (tb < 0 || row >= tb + 32) {
            tb = row;
            const int64_t rr = row + lane;
            tok_reg = rr < p.n_rows ? __ldg(p.tokens + rr) : 0;
            rib_reg = (p.row_index != nullptr && rr < p.n_rows) ? __ldg(p.row_index + rr) : 0;
        }
        tok = __shfl_sync(0xffffffffu, tok_reg, (int)(row - tb));
        const int64_t src = __shfl_sync(0xffffffffu, rib_reg, (int)(row - tb));
        const bool bad_tok = tok < 0 || tok >= p.V;
        const bool bad_src = p.row_index != nullptr && (src < 0 || src >= p.n_logit_rows);
        bad = bad_tok || bad_src;
        if (lane == 0) {
            if (bad_tok) set_status(p.status, PS_DEV_BAD_TOKEN);
            if (bad_src) set_status(p.status, PS_DEV_BAD_ROW_INDEX);
        }
    };
    row_start();

    Acc acc = acc_empty();
    float ltok = __uint_as_float(kAbsent);
    uint32_t phase = 0;
    int s = 0;                                        // stage of chunk c

    for (int64_t c = cb; c < ce; ++c, s = (s + 1 == kStages) ? 0 : s + 1) {
        if (!mbar_wait_bounded(&bars[s], (phase >> s) & 1u, kWaitLimitNs)) {
            if (lane == 0) {
                set_status(p.status, PS_DEV_TIMEOUT);
                // let this warp's copies in flight land before the warp exits
                for (int j = 0; j < kStages; ++j) {
                    if (c + j < ic) {
                        const int sj = (s + j) % kStages;
                        mbar_wait_bounded(&bars[sj], (phase >> sj) & 1u, kDrainLimitNs);
                    }
                }
            }
            __syncwarp();
            return;
        }
        phase ^= 1u << s;
        uint8_t *buf = stage + (size_t)s * kStageBytes;
        const uint32_t off = (uint32_t)k * kStageBytes;
        const uint32_t bytes = min((uint32_t)kStageBytes, (uint32_t)p.row_bytes - off);
        if (lane == 0) {
            const int64_t e0 = (int64_t)k * kElemsPerStage;
            const int64_t nel = bytes / kEsz;
            if (!bad) {
                const int64_t o = (int64_t)tok - e0;
                if (o >= 0 && o < nel) {
                    if constexpr (DT == PS_BF16) {
                        uint16_t *h = reinterpret_cast<uint16_t *>(buf) + o;
                        ltok = __uint_as_float((uint32_t)*h << 16);
                        *h = ENT ? Elem<PS_BF16>::kFloorElem : 0xff80u;
                    } else {
                        float *f = reinterpret_cast<float *>(buf) + o;
                        ltok = *f;
                        *f = ENT ? kFloorF32 : -INFINITY;
                    }
                }
            }
            if (k == cpr - 1) {
                for (int64_t j = (int64_t)p.V - e0; j < nel; ++j) {
                    if constexpr (DT == PS_BF16)
                        reinterpret_cast<uint16_t *>(buf)[j] = ENT ? Elem<PS_BF16>::kFloorElem
                                                                   : 0xff80u;
                    else
                        reinterpret_cast<float *>(buf)[j] = ENT ? kFloorF32 : -INFINITY;
                }
            }
        }
        __syncwarp();
        {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
            const int nvec = (int)(bytes >> 4);
            uint4 q[kVecPerLane];
            load_vecs<DT, kVecPerLane, ENT>(v4, nvec, lane, q);
            float c1, ct[3], cy;
            // the entropy variant's fast path skips the -inf clamp (unless the
            // batch says its logits may be masked): the row's patches hold the
            // floor, and a -inf input makes 2^y y NaN, which sends the chunk to
            // the slow path (clamped)
            sum_vecs<DT, NP, ENT, kVecPerLane, ENT && CF>(q, acc.R, g, c1, ct, cy);
            bool fast = chunk_peak<NP>(c1, ct) <= kLimit;
            if constexpr (ENT)
                fast = __all_sync(0xffffffffu, fast && c1 <= kEntLimit && cy == cy);
            if (fast) {
                add_chunk<NP, ENT>(acc, c1, ct, cy);
            } else {
                acc = slow_chunk<DT, NP, ENT, kVecPerLane>(v4, nvec, lane, g, acc);
            }
        }
        __syncwarp();
        if (ic < ce) issue_next(s);

        const bool row_end = (k == cpr - 1) || (c == ce - 1);
        if (row_end) {
            acc = warp_merge<NP, ENT>(acc, g);
            const float lt = __shfl_sync(0xffffffffu, ltok, 0);
            const int64_t rc0 = row * cpr, rc1 = rc0 + cpr;
            if (rc0 >= cb && rc1 <= ce) {
                if (lane == 0) finalize_row<NP, ENT>(p, row, acc, lt, bad);
            } else {
                const int64_t slot = (row == cb / cpr) ? 2 * vw : 2 * vw + 1;
                const int64_t owner = warp_of_chunk(rc0, C, W);
                const int64_t lastw = warp_of_chunk(rc1 - 1, C, W);
                int last = 0;
                if (lane == 0) {
                    RowPart part;
                    part.R = acc.R;
                    part.s1 = acc.s1;
                    part.st = acc.st[0];
                    part.ltok = lt;
                    part.y1 = acc.y1;
                    part.st1 = acc.st[1];
                    part.st2 = acc.st[2];
                    part.pad = 0.f;
                    p.parts[slot] = part;
                    __threadfence();
                    const int old = atomicAdd(p.counters + owner, 1);
                    last = (old == (int)(lastw - owner));
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    Acc m = acc_empty();
                    float ltm = __uint_as_float(kAbsent);
                    // lanes take the parts in warp order, then a fixed butterfly
                    for (int64_t u = owner + lane; u <= lastw; u += 32) {
                        const int64_t su =
                            (row == range_begin(u, C, W) / cpr) ? 2 * u : 2 * u + 1;
                        const float4 pv = __ldcg(reinterpret_cast<const float4 *>(p.parts + su));
                        const float4 pw =
                            __ldcg(reinterpret_cast<const float4 *>(p.parts + su) + 1);
                        m = merge_part<NP, ENT>(m, Acc{pv.x, pv.y, {pv.z, pw.y, pw.z}, pw.x}, g);
                        if (__float_as_uint(pv.w) != kAbsent) ltm = pv.w;
                    }
                    m = warp_merge<NP, ENT>(m, g);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float other = __shfl_xor_sync(0xffffffffu, ltm, o);
                        if (__float_as_uint(ltm) == kAbsent) ltm = other;
                    }
                    if (lane == 0) {
                        finalize_row<NP, ENT>(p, row, m, ltm, bad);
                        p.counters[owner] = 0;
                    }
                }
            }
            acc = acc_empty();
            ltok = __uint_as_float(kAbsent);
        }
        if (++k == cpr) {
            k = 0;
            ++row;
            if (c + 1 < ce) row_start();
        }
    }
    // the next kernel (suffix sums) may be launched once every CTA gets here;
    // it still waits for this grid to complete before it reads the per-row
    // results.  Triggering at the end rather than the start keeps its CTAs
    // from waiting on the SMs through this kernel's tail, which measured
    // slower on GB300.
    pdl_launch_dependents();
}

// The scoring kernel of the variants without entropy, with tail blocks: each
// warp reads its own range, then takes tail blocks (a counter in the
// workspace) until none is left; on batches without tail blocks it reads its
// own range only.  The entropy variants use score_rows_kernel above, whose
// body is the same without the range loop: wrapping that body in the loop
// made the heaviest of them (any other tau, with entropy) 9% slower on GB300,
// as its code at the 128-register cap was scheduled differently, while they
// gain little from tail blocks (they are bound by issue rather than by
// memory).
template <int DT, int NP, int WARPS, int STAGES, int SB>
__global__ void __launch_bounds__(WARPS * 32, 1) score_rows_tail_kernel(const RowsParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kWarpsPerCta = WARPS;
    constexpr int kStages = STAGES;
    constexpr int kStageBytes = SB;
    constexpr int kVecPerLane = SB / 16 / 32;
    static_assert(SB % 512 == 0, "a stage holds a whole number of 16-byte vectors per lane");
    constexpr int kEsz = Elem<DT>::kSize;
    constexpr int kElemsPerStage = kStageBytes / kEsz;
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t W = p.n_vwarps;
    const int64_t vw = (int64_t)blockIdx.x * kWarpsPerCta + wid;
    if (vw >= W) return;
    const int32_t cpr = p.cpr;
    const float g = p.g;

    uint8_t *stage = smem + (size_t)wid * kStages * kStageBytes;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + (size_t)kWarpsPerCta * kStages * kStageBytes) +
        wid * kStages;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = l2_evict_first_policy();   // logits are read once
    uint32_t phase = 0;                               // mbarrier parity of each stage
    int s = 0;                                        // stage of the next chunk

    // the warp's own range, then tail blocks until none is left
    for (int64_t vr = vw;;) {
        const int64_t cb = tail_range_begin(p, vr);
        const int64_t ce = tail_range_begin(p, vr + 1);

        // ---- issue side: next chunk to copy and a lane-parallel cache of row_index
        int64_t ic = cb;
        int64_t irow = cb / cpr;
        int32_t ik = (int32_t)(cb - irow * cpr);
        int64_t ri_base = -1;
        int64_t ri_reg = 0;
        auto src_row_of = [&](int64_t row) -> int64_t {   // warp-collective
            if (p.row_index == nullptr) return row;
            if (ri_base < 0 || row >= ri_base + 32 || row < ri_base) {
                ri_base = row;
                const int64_t rr = row + lane;
                ri_reg = rr < p.n_rows ? __ldg(p.row_index + rr) : 0;
            }
            int64_t sr = __shfl_sync(0xffffffffu, ri_reg, (int)(row - ri_base));
            if (sr < 0 || sr >= p.n_logit_rows) sr = 0;   // flagged on the consume side
            return sr;
        };
        auto issue_next = [&](int st) {                   // warp-collective
            const int64_t srow = src_row_of(irow);
            if (lane == 0) {
                const uint32_t off = (uint32_t)ik * kStageBytes;
                const uint32_t bytes = min((uint32_t)kStageBytes, (uint32_t)p.row_bytes - off);
                const uint8_t *src = p.logits + srow * p.ld_bytes + off;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[st], bytes);
                bulk_g2s(stage + (size_t)st * kStageBytes, src, bytes, &bars[st], policy);
            }
            ++ic;
            if (++ik == cpr) {
                ik = 0;
                ++irow;
            }
        };
#pragma unroll
        for (int j = 0; j < kStages; ++j)
            if (ic < ce) issue_next(s + j < kStages ? s + j : s + j - kStages);

        // ---- consume side
        int64_t row = cb / cpr;
        int32_t k = (int32_t)(cb - row * cpr);
        int64_t tb = -1;
        int32_t tok_reg = 0;
        int64_t rib_reg = 0;
        int32_t tok = 0;
        bool bad = false;
        auto row_start = [&]() {                          // warp-collective
            if (tb < 0 || row >= tb + 32) {
                tb = row;
                const int64_t rr = row + lane;
                tok_reg = rr < p.n_rows ? __ldg(p.tokens + rr) : 0;
                rib_reg = (p.row_index != nullptr && rr < p.n_rows) ? __ldg(p.row_index + rr) : 0;
            }
            tok = __shfl_sync(0xffffffffu, tok_reg, (int)(row - tb));
            const int64_t src = __shfl_sync(0xffffffffu, rib_reg, (int)(row - tb));
            const bool bad_tok = tok < 0 || tok >= p.V;
            const bool bad_src = p.row_index != nullptr && (src < 0 || src >= p.n_logit_rows);
            bad = bad_tok || bad_src;
            if (lane == 0) {
                if (bad_tok) set_status(p.status, PS_DEV_BAD_TOKEN);
                if (bad_src) set_status(p.status, PS_DEV_BAD_ROW_INDEX);
            }
        };
        row_start();

        Acc acc = acc_empty();
        float ltok = __uint_as_float(kAbsent);

        for (int64_t c = cb; c < ce; ++c, s = (s + 1 == kStages) ? 0 : s + 1) {
            if (!mbar_wait_bounded(&bars[s], (phase >> s) & 1u, kWaitLimitNs)) {
                if (lane == 0) {
                    set_status(p.status, PS_DEV_TIMEOUT);
                    // let this warp's copies in flight land before the warp exits
                    for (int j = 0; j < kStages; ++j) {
                        if (c + j < ic) {
                            const int sj = (s + j) % kStages;
                            mbar_wait_bounded(&bars[sj], (phase >> sj) & 1u, kDrainLimitNs);
                        }
                    }
                }
                __syncwarp();
                return;
            }
            phase ^= 1u << s;
            uint8_t *buf = stage + (size_t)s * kStageBytes;
            const uint32_t off = (uint32_t)k * kStageBytes;
            const uint32_t bytes = min((uint32_t)kStageBytes, (uint32_t)p.row_bytes - off);
            if (lane == 0) {
                const int64_t e0 = (int64_t)k * kElemsPerStage;
                const int64_t nel = bytes / kEsz;
                if (!bad) {
                    const int64_t o = (int64_t)tok - e0;
                    if (o >= 0 && o < nel) {
                        if constexpr (DT == PS_BF16) {
                            uint16_t *h = reinterpret_cast<uint16_t *>(buf) + o;
                            ltok = __uint_as_float((uint32_t)*h << 16);
                            *h = 0xff80u;
                        } else {
                            float *f = reinterpret_cast<float *>(buf) + o;
                            ltok = *f;
                            *f = -INFINITY;
                        }
                    }
                }
                if (k == cpr - 1) {
                    for (int64_t j = (int64_t)p.V - e0; j < nel; ++j) {
                        if constexpr (DT == PS_BF16)
                            reinterpret_cast<uint16_t *>(buf)[j] = 0xff80u;
                        else
                            reinterpret_cast<float *>(buf)[j] = -INFINITY;
                    }
                }
            }
            __syncwarp();
            {
                const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
                const int nvec = (int)(bytes >> 4);
                uint4 q[kVecPerLane];
                load_vecs<DT, kVecPerLane, false>(v4, nvec, lane, q);
                float c1, ct[3], cy;
                sum_vecs<DT, NP, false, kVecPerLane, false>(q, acc.R, g, c1, ct, cy);
                const bool fast = chunk_peak<NP>(c1, ct) <= kLimit;
                if (fast) {
                    add_chunk<NP, false>(acc, c1, ct, cy);
                } else {
                    acc = slow_chunk<DT, NP, false, kVecPerLane>(v4, nvec, lane, g, acc);
                }
            }
            __syncwarp();
            if (ic < ce) issue_next(s);

            const bool row_end = (k == cpr - 1) || (c == ce - 1);
            if (row_end) {
                acc = warp_merge<NP, false>(acc, g);
                const float lt = __shfl_sync(0xffffffffu, ltok, 0);
                const int64_t rc0 = row * cpr, rc1 = rc0 + cpr;
                if (rc0 >= cb && rc1 <= ce) {
                    if (lane == 0) finalize_row<NP, false>(p, row, acc, lt, bad);
                } else {
                    const int64_t slot = (row == cb / cpr) ? 2 * vr : 2 * vr + 1;
                    const int64_t owner = tail_range_of_chunk(p, rc0);
                    const int64_t lastw = tail_range_of_chunk(p, rc1 - 1);
                    int last = 0;
                    if (lane == 0) {
                        RowPart part;
                        part.R = acc.R;
                        part.s1 = acc.s1;
                        part.st = acc.st[0];
                        part.ltok = lt;
                        part.y1 = acc.y1;
                        part.st1 = acc.st[1];
                        part.st2 = acc.st[2];
                        part.pad = 0.f;
                        p.parts[slot] = part;
                        __threadfence();
                        const int old = atomicAdd(p.counters + owner, 1);
                        last = (old == (int)(lastw - owner));
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last) {
                        __threadfence();
                        Acc m = acc_empty();
                        float ltm = __uint_as_float(kAbsent);
                        // lanes take the parts in range order, then a fixed butterfly
                        for (int64_t u = owner + lane; u <= lastw; u += 32) {
                            const int64_t su =
                                (row == tail_range_begin(p, u) / cpr) ? 2 * u : 2 * u + 1;
                            const float4 *pp = reinterpret_cast<const float4 *>(p.parts + su);
                            const float4 pv = __ldcg(pp);
                            const float4 pw = __ldcg(pp + 1);
                            m = merge_part<NP, false>(m, Acc{pv.x, pv.y, {pv.z, pw.y, pw.z}, pw.x},
                                                    g);
                            if (__float_as_uint(pv.w) != kAbsent) ltm = pv.w;
                        }
                        m = warp_merge<NP, false>(m, g);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const float other = __shfl_xor_sync(0xffffffffu, ltm, o);
                            if (__float_as_uint(ltm) == kAbsent) ltm = other;
                        }
                        if (lane == 0) {
                            finalize_row<NP, false>(p, row, m, ltm, bad);
                            p.counters[owner] = 0;
                        }
                    }
                }
                acc = acc_empty();
                ltok = __uint_as_float(kAbsent);
            }
            if (++k == cpr) {
                k = 0;
                ++row;
                if (c + 1 < ce) row_start();
            }
        }
        // every copy issued for this range has been consumed; take a tail block
        if (p.n_tail == 0) break;
        int32_t b = 0;
        if (lane == 0) b = atomicAdd(p.claim, 1);
        b = __shfl_sync(0xffffffffu, b, 0);
        if (b >= p.n_tail) break;
        vr = W + b;
    }
    // the next kernel may be launched once every CTA gets here (as in
    // score_rows_kernel)
    pdl_launch_dependents();
}

template <int WARPS, int STAGES, int SB>
constexpr size_t smem_bytes_for() {
    return (size_t)WARPS * STAGES * SB + (size_t)WARPS * STAGES * 8;
}

template <typename Kernel>
cudaError_t launch_k(Kernel kern, const RowsParams &p, int n_ctas, cudaStream_t stream) {
    const size_t smem = smem_bytes_for<kWarpsPerCta, kStages, kStageBytes>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<n_ctas, kWarpsPerCta * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

// The entropy variants run score_rows_kernel, the others score_rows_tail_kernel.
template <int DT, int NP, bool ENT, bool CF>
cudaError_t launch_t(const RowsParams &p, int n_ctas, cudaStream_t stream) {
    if constexpr (ENT)
        return launch_k(score_rows_kernel<DT, NP, ENT, kWarpsPerCta, kStages, kStageBytes, CF>,
                        p, n_ctas, stream);
    else
        return launch_k(score_rows_tail_kernel<DT, NP, kWarpsPerCta, kStages, kStageBytes>, p,
                        n_ctas, stream);
}

template <int DT, bool ENT, bool CF>
cudaError_t launch_dt(const RowsParams &p, int n_ctas, cudaStream_t stream) {
    switch (p.npow) {
        case 1: return launch_t<DT, 1, ENT, CF>(p, n_ctas, stream);
        case 2: return launch_t<DT, 2, ENT, CF>(p, n_ctas, stream);
        case 4: return launch_t<DT, 4, ENT, CF>(p, n_ctas, stream);
        case 8: return launch_t<DT, 8, ENT, CF>(p, n_ctas, stream);
        case kAllPowers: return launch_t<DT, kAllPowers, ENT, CF>(p, n_ctas, stream);
        case kPowersTo4: return launch_t<DT, kPowersTo4, ENT, CF>(p, n_ctas, stream);
        default: return launch_t<DT, 0, ENT, CF>(p, n_ctas, stream);
    }
}

template <int DT>
cudaError_t launch_ent(const RowsParams &p, int n_ctas, cudaStream_t stream) {
    if (p.entropy == nullptr) return launch_dt<DT, false, false>(p, n_ctas, stream);
    if (p.flags & PS_FLAG_MASKED_LOGITS) return launch_dt<DT, true, true>(p, n_ctas, stream);
    return launch_dt<DT, true, false>(p, n_ctas, stream);
}

}  // namespace

size_t score_rows_smem_bytes() { return smem_bytes_for<kWarpsPerCta, kStages, kStageBytes>(); }

cudaError_t launch_score_rows(const RowsParams &p, int n_ctas, cudaStream_t stream) {
    if (p.dtype == PS_BF16) return launch_ent<PS_BF16>(p, n_ctas, stream);
    return launch_ent<PS_F32>(p, n_ctas, stream);
}

}  // namespace ps
