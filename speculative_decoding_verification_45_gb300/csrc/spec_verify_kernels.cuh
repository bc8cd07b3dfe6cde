// spec_verify_kernels.cuh -- device code of the verification kernels.
//
// Included by the host translation unit (spec_verify.cu) for the shared types
// and constants, and by one translation unit per (dtype, proposal form) that
// instantiates that variant's kernels (kernels_*.cu), so nvcc compiles them in
// parallel.  Everything here has internal linkage; the variant units export
// only the kernel lookup functions declared at the end.
//
// The operation is the modified rejection sampler stated in
//   "Speculative Decoding" (atonlee.tistory.com/330), ch.2-3;
//   "Speculative Decoding으로 LLM 추론 속도 높이기" (donmain.dev), section
//   "품질은 rejection sampling이 지킨다";
//   "Fast Inference from Transformers via Speculative Decoding" notes, method
//   details steps 2-3;
//   "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가", section on why the output
//   does not change;
// and is specified in full in include/spec_verify.h.
//
// Design (one kernel launch per call):
//   * One thread-block cluster of C CTAs per sequence (1 <= C <= 16, chosen
//     from B, V and the SM count).  CTA c of the cluster owns the contiguous
//     slice [c*NC/C, (c+1)*NC/C) of 16-byte chunks of every row the sequence
//     needs.  Grids longer than one wave take sequences longest-first.
//   * Pass 1 streams those slices once, in batches of eight 16-byte loads per
//     thread (the row's next batch requested into L2 first).  Target and draft
//     rows of sampled sequences (T > 0) keep an online (max, sum of 2^(a-m))
//     per thread, a = logit * log2(e)/T, with m an integer so that rescaling is
//     an exact power of two and the sum compensated; greedy rows (T = 0) keep
//     (max, lowest argmax) of the raw logits.  Partials are reduced over the
//     warp (shuffles), the CTA (shared memory) and the cluster (every CTA
//     pushes its row partials into every other CTA's shared memory, DSMEM).
//   * After one cluster barrier each CTA holds all partials, merges them in
//     rank order (identical bits in every CTA) and takes the accept decision
//     itself: one lane per draft position, a warp ballot gives the first
//     rejection.  No second barrier is needed to broadcast it.
//   * Pass 2 (sampled sequences only) sweeps the one decided row (target, plus
//     draft when a draft was rejected) and puts every sampling weight on an
//     exact 2^-60 integer grid: ids near the top of the row get an extended-
//     precision exp2 (about 2^-36 relative), the rest their float32 value, so
//     that the draw agrees with the float64 definition except within ~1e-9
//     of a boundary (see "pass 2" below).  Per-warp and per-CTA sums cross the
//     cluster over DSMEM; the CTA whose slice holds floor(u*S) recomputes one
//     warp range of it and writes the id.
//
// Kernels sharing that protocol:
//   spec_verify_stream_kernel (full sweep) 128-bit loads straight into registers,
//                             32 reducing warps per SM; element loads when rows
//                             are not 16-byte aligned; variants that read
//                             several rows per round trip for narrow slices.
//   spec_verify_early_kernel  positions in order, no row after the first
//                             rejection read; its staged form (rows in
//                             page-locked host memory, which L2 does not
//                             cache) keeps each position's slices in shared
//                             memory so pass 2 reads nothing over the link.
//   spec_tree_kernel          a walk down a tree of candidates, one row per level.
// No kernel uses global scratch memory, atomics on the data path (only the
// optional status word and counters) or waits other than hardware barriers
// that every thread of the CTA or of the cluster reaches.

#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

#include <atomic>
#include <cfloat>
#include <climits>
#include <cstdint>

#include "spec_verify.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kWarps = 8;  // warps that reduce
constexpr int kThreads = kWarps * 32;
constexpr int kMaxRows = 2 * SPEC_MAX_GAMMA + 1;
constexpr int kMaxCluster = 16;
constexpr int kUnroll = 8;         // pass 1: 16-byte loads in flight per thread
constexpr int kMaxOrdered = 1024;  // longest-first scheduling for B up to this
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2eLo = (float)(1.4426950408889634073599 - (double)kLog2e);  // log2(e) - kLog2e
constexpr float kLn2 = 0.69314718055994531f;

struct Params {
    const void *target;
    const void *draft;  // NULL: point-mass proposals (q_i is 1 at the drafted id)
    const int32_t *tokens;
    const int32_t *num_draft;  // NULL for spec_sample: every sequence has g = 0
    const float *uniforms;
    const float *temperature;
    int32_t *out_tokens;
    int32_t *out_num;  // NULL for spec_sample (no accepted count)
    uint32_t *status;
    float *p_hat;
    float *q_hat;
    float *logz_t;
    float *logz_d;
    float *resid_mass;
    int32_t *seq_status;
    int B, gmax, V;
    int num_chunks;  // 16-byte chunks per row; the last is partial on the scalar path
    int ordered;     // map clusters to sequences longest-first (small B only)
    unsigned long long *counters;  // optional: += drafted, accepted, verified sequences
    unsigned long long *hist;      // optional: [SPEC_MAX_GAMMA + 1] += 1 at the accepted count
    const int32_t *parent;         // tree kernel: [B, gmax+1] parent of each node (num_draft = node count)
    int32_t *out_path;             // tree kernel: [B, gmax+1] accepted node indices, or NULL
};

// ---------------------------------------------------------------------------
// element types: a chunk is 16 bytes = 8 bfloat16 or 4 float32 values
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
    static constexpr int W = 8;
    static constexpr uint32_t kNegInfPair = 0xFF80FF80u;
};
template <> struct Elem<float> {
    static constexpr int W = 4;
    static constexpr uint32_t kNegInfPair = 0xFF800000u;
};

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

template <typename T> __device__ __forceinline__ uint4 neg_inf_chunk()
{
    const uint32_t v = Elem<T>::kNegInfPair;
    return make_uint4(v, v, v, v);
}

// One chunk of a row.  ALIGNED: the row base is 16-byte aligned and V is a
// multiple of the chunk width.  Otherwise each element is loaded on its own and
// positions >= V read as -inf (zero weight, never an argmax).
template <typename T, bool ALIGNED>
__device__ __forceinline__ uint4 load_chunk(const T *row, int chunk, int V)
{
    if (ALIGNED)
        return ld_stream16(row + (size_t)chunk * Elem<T>::W);
    uint32_t w[4];
    const int base = chunk * Elem<T>::W;
    if (sizeof(T) == 2) {
        const unsigned short *r = reinterpret_cast<const unsigned short *>(row);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t lo = base + 2 * q < V ? __ldg(r + base + 2 * q) : 0xFF80u;
            uint32_t hi = base + 2 * q + 1 < V ? __ldg(r + base + 2 * q + 1) : 0xFF80u;
            w[q] = lo | (hi << 16);
        }
    } else {
        const uint32_t *r = reinterpret_cast<const uint32_t *>(row);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = base + q < V ? __ldg(r + base + q) : 0xFF800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int q)
{
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// Element e of a chunk, widened to float (bfloat16 is the top half of a float).
template <typename T> __device__ __forceinline__ float elem(const uint4 &v, int e)
{
    if (sizeof(T) == 2) {
        const uint32_t w = word(v, e >> 1);
        return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
    return __uint_as_float(word(v, e));
}

// Largest value of a chunk (NaN elements ignored).
template <typename T> __device__ __forceinline__ float chunk_max(const uint4 &v)
{
    if (sizeof(T) == 2) {
        __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&v.w));
        __nv_bfloat162 c = __hmax2(a, b);
        return fmaxf(__low2float(c), __high2float(c));
    }
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^d for an integer-valued d <= 0, exactly (0 below the normal range, and for
// -inf or NaN).
__device__ __forceinline__ float pow2_int(float d)
{
    if (!(d >= -126.0f))
        return 0.0f;
    return __int_as_float((127 + (int)d) << 23);
}

// Pair q of a chunk as two floats (elements 2q and 2q+1); bfloat16 is the top
// half of a float, so widening is a shift or a mask.
template <typename T> __device__ __forceinline__ float2 pair(const uint4 &v, int q)
{
    if (sizeof(T) == 2) {
        const uint32_t w = word(v, q);
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    return make_float2(__uint_as_float(word(v, 2 * q)), __uint_as_float(word(v, 2 * q + 1)));
}

// Largest value over N chunks (NaN elements ignored), packed where possible.
template <typename T, int N> __device__ __forceinline__ float chunks_max(const uint4 (&v)[N])
{
    if (sizeof(T) == 2) {
        __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162 *>(&v[0].x);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162 *>(&v[u].x));
            m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162 *>(&v[u].y));
            m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162 *>(&v[u].z));
            m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162 *>(&v[u].w));
        }
        return fmaxf(__low2float(m), __high2float(m));
    }
    float m = -INFINITY;
#pragma unroll
    for (int u = 0; u < N; ++u)
        m = fmaxf(m, chunk_max<T>(v[u]));
    return m;
}

__device__ __forceinline__ float2 ex2_pair(float2 a)
{
    return make_float2(ex2_approx(a.x), ex2_approx(a.y));
}

// ---------------------------------------------------------------------------
// per-row statistics and their merges
// ---------------------------------------------------------------------------
// Softmax rows: sum_j 2^(a_j - m) = hi + lo, m integer-valued (or -inf).
// Greedy rows:  (m, idx) = largest raw logit and its lowest index.
struct RowStat {
    float m;
    float hi;
    float lo;
    int idx;
};

__device__ __forceinline__ void compensated_add(float &hi, float &lo, float v)
{
    const float y = v + lo;
    const float t = hi + y;
    lo = y - (t - hi);
    hi = t;
}

__device__ __forceinline__ RowStat soft_merge(const RowStat &a, const RowStat &b)
{
    const float M = fmaxf(a.m, b.m);
    RowStat r;
    r.m = M;
    r.idx = 0;
    if (M == -INFINITY) {
        r.hi = 0.0f;
        r.lo = 0.0f;
        return r;
    }
    const float sa = pow2_int(a.m - M), sb = pow2_int(b.m - M);
    const float x = a.hi * sa, y = b.hi * sb;
    const float s = x + y;
    const float bb = s - x;
    const float err = (x - (s - bb)) + (y - bb);  // two-sum: s + err == x + y exactly
    r.hi = s;
    r.lo = (a.lo * sa + b.lo * sb) + err;
    return r;
}

__device__ __forceinline__ RowStat arg_merge(const RowStat &a, const RowStat &b)
{
    return (b.m > a.m || (b.m == a.m && b.idx < a.idx)) ? b : a;
}

__device__ __forceinline__ RowStat shfl_xor_stat(const RowStat &s, int mask)
{
    RowStat r;
    r.m = __shfl_xor_sync(0xffffffffu, s.m, mask);
    r.hi = __shfl_xor_sync(0xffffffffu, s.hi, mask);
    r.lo = __shfl_xor_sync(0xffffffffu, s.lo, mask);
    r.idx = __shfl_xor_sync(0xffffffffu, s.idx, mask);
    return r;
}

__device__ __forceinline__ RowStat warp_reduce(RowStat s, bool sampled)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s = sampled ? soft_merge(s, shfl_xor_stat(s, o)) : arg_merge(s, shfl_xor_stat(s, o));
    return s;
}

__device__ __forceinline__ bool soft_row_ok(const RowStat &s)
{
    const float z = s.hi + s.lo;
    return isfinite(s.m) && isfinite(z) && z > 0.0f;
}

// Running per-thread statistics of one row.
struct RowAcc {
    float m, hi, lo;  // sampled rows (greedy rows: m is the best value)
    int idx;          // greedy rows: index of the best value
    __device__ __forceinline__ void reset(int first_idx)
    {
        m = -INFINITY;
        hi = 0.0f;
        lo = 0.0f;
        idx = first_idx;
    }
    // Adds chunks v[0..N) of a softmax row: online max, exact power-of-two
    // rescale, packed FMA/add (two elements per instruction), four independent
    // partial sums, then one compensated add per batch.
    template <typename T, int N> __device__ __forceinline__ void add_soft(const uint4 (&v)[N], float k)
    {
        const float amax = chunks_max<T, N>(v) * k;
        if (amax > m) {
            const float mn = ceilf(amax);
            const float sc = pow2_int(m - mn);
            hi *= sc;
            lo *= sc;
            m = mn;
        }
        if (m == -INFINITY)
            return;
        constexpr int P = Elem<T>::W / 2;
        const float2 k2 = make_float2(k, k), nm2 = make_float2(-m, -m);
        float2 acc[P];
#pragma unroll
        for (int q = 0; q < P; ++q)
            acc[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int u = 0; u < N; ++u)
#pragma unroll
            for (int q = 0; q < P; ++q)
                acc[q] = __fadd2_rn(acc[q], ex2_pair(__ffma2_rn(pair<T>(v[u], q), k2, nm2)));
        float2 t = acc[0];
#pragma unroll
        for (int q = 1; q < P; ++q)
            t = __fadd2_rn(t, acc[q]);
        compensated_add(hi, lo, t.x + t.y);
    }
    // Adds chunks v[0..N) of a greedy row; chunk u starts at element index
    // base + u * stride.  Chunks arrive in increasing index order, so a strict
    // improvement keeps the lowest index of the maximum.
    template <typename T, int N>
    __device__ __forceinline__ void add_arg(const uint4 (&v)[N], int base, int stride)
    {
        const float bm = chunks_max<T, N>(v);
        if (bm > m) {
            int found = -1;
#pragma unroll
            for (int u = 0; u < N; ++u)
#pragma unroll
                for (int e = 0; e < Elem<T>::W; ++e)
                    if (found < 0 && elem<T>(v[u], e) == bm)
                        found = base + u * stride + e;
            m = bm;
            idx = found;
        }
    }
    __device__ __forceinline__ RowStat stat() const
    {
        RowStat s;
        s.m = m;
        s.hi = hi;
        s.lo = lo;
        s.idx = idx;
        return s;
    }
};

// floor(w * 2^(60 - sc)) for a finite w >= 0 with w * 2^(60 - sc) < 2^64, by
// integer operations only (a float-to-64-bit-integer conversion instruction
// would run on the FP64 pipe).  sc = 0: w on the 2^-60 grid itself.
__device__ __forceinline__ unsigned long long to_fixed60(float w, int sc = 0)
{
    const uint32_t bits = __float_as_uint(w);
    const int ex = (int)(bits >> 23);  // w >= 0: no sign bit
    if (ex == 0)
        return 0ull;  // zero or below 2^-126, far under the 2^-60 unit
    const unsigned long long mant = (bits & 0x7FFFFFu) | 0x800000u;
    const int sh = ex - 90 - sc;  // w = mant * 2^(ex - 150), so w * 2^(60 - sc) = mant * 2^(ex - 90 - sc)
    if (sh >= 0)
        return mant << sh;
    if (sh <= -24)
        return 0ull;
    return mant >> (-sh);
}


// ---------------------------------------------------------------------------
// pass 2: sampling weights on an exact integer grid
// ---------------------------------------------------------------------------
// The final draw is the smallest id j with u*S < C_j, so the boundary C_j/S of
// an id depends on every weight before it.  Float32 weights (about 1e-7
// relative error each, plus the float32 rounding of log2(e)/T, which tilts a
// whole row) move the boundaries of a 128k-id row by ~1e-8 each, enough to
// change about one full-row draw in a thousand against the float64
// definition; a residual max(0, p - q) of small total amplifies that by
// 1/total.  Pass 2 therefore puts every weight on a 2^-60 integer grid:
//   * a "heavy" id, with l*K above m - kHeavySpan - 1 for the row's integer
//     maximum m, gets 2^(l*K - mref) to about 2^-36 relative (exact_weight:
//     K = log2(e)/T as a float-float pair, a float-float table of 2^(i/32) and
//     a degree-4 polynomial for the rest -- the table-driven exponential of
//     P. T. P. Tang, ACM TOMS 15(2), 1989 -- with Dekker's exact product and
//     Knuth's exact sum splits);
//   * every other id keeps a float32 weight ex2.approx(l*K - mf), summed in
//     float32 per chunk in id order and rounded to the grid once per chunk
//     (an exact power-of-two rescale by 2^-sf on the way).  The fast
//     reference mf = m - kFastRef puts the heavy threshold at argument 0, so
//     the ids just below it, whose weights carry the largest absolute errors,
//     get arguments with rounding errors under 2^-24: what is left is
//     ex2.approx's own relative error (~2^-22).  The same reference at the
//     grid's mref would leave arguments near -kHeavySpan - ez, rounded to
//     2^-20.  A draw's chance to land between two versions of a boundary
//     grows with V * err * sqrt(threshold weight), so the 4x smaller error
//     lets the threshold rise 16x (span 18 -> 14) at the same bound; on the
//     V = 128256, T = 1 Zipf rows that cuts the heavy ids from 17 % to 4 %.
// Sums of grid integers are exact and order-free, so every CTA and every pass
// sees the same boundaries.  A residual max(0, p - q) = max(0, a/A - b/B) (a, b
// the target and draft weights, A, B their row totals) is sampled as the
// integer weight a*B - b*A over the set J of ids where the float32 values say
// p > q; a sum over J is then A_J*B - B_J*A, so a single sweep that keeps A_J
// and B_J per warp range and A, B per row is enough.  (An id that float32
// misplaces in J has |p - q| ~ 1e-7 p, so its contribution is negligible.)
constexpr float kHeavySpan = 14.0f;  // log2 of the heavy window below the top weight
constexpr float kFastRef = kHeavySpan + 1.0f;  // fast path: reference this far below the row's max
constexpr int kP2Unroll = 4;         // pass-2 sweep: chunks in flight per thread (one row; half each for two)
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: x + kMagic rounds x to an integer for |x| < 2^22
constexpr float kLn2Lo = -1.9046542121259336e-09f;  // ln 2 - (float)ln 2
constexpr float kC2 = 0.24022650718688965f;    // (ln 2)^2 / 2
constexpr float kC3 = 0.05550410971045494f;    // (ln 2)^3 / 6
constexpr float kC4 = 0.009618128649890423f;   // (ln 2)^4 / 24

// 2^(i/32) for i = -16..16 as float-float pairs (hi + lo), from the
// exponential series summed in double precision at compile time.
constexpr double series_exp(double x)
{
    double term = 1.0, sum = 1.0;
    for (int n = 1; n < 40; ++n) {
        term *= x / n;
        sum += term;
    }
    return sum;
}
struct Exp2Table {
    float hi[33];
    float lo[33];
};
constexpr Exp2Table make_exp2_table()
{
    Exp2Table t{};
    for (int i = 0; i < 33; ++i) {
        const double v = series_exp((i - 16) / 32.0 * 0.6931471805599453094);
        t.hi[i] = (float)v;
        t.lo[i] = (float)(v - (double)t.hi[i]);
    }
    return t;
}
__device__ const Exp2Table kExp2Table = make_exp2_table();

// One row's weight scale: weight_j = 2^(l_j * K - mref), K = khi + klo.  The
// fast path works in units 2^sf times larger, fast weight 2^(l_j * K - mf)
// with mf = mref - sf, so that the heavy threshold sits at fast argument 0.
struct ExactRow {
    float khi, klo;  // log2(e)/T as a float-float pair
    float nmf;       // -mf (integer-valued)
    int sf;          // mref - mf: grid weight = fast weight * 2^-sf
    int e60;         // 60 - mref: weight * 2^60 = 2^(n + e60) * 2^f
    float heavy;     // fast argument above this: exact weight (0, or +inf: none)
    bool wide;       // |l * K| may pass 2^12: fold the product's low part in first
    float c;         // 2^-kFastRef / Z: float32 probability = fast weight * c (the set J)
    float koff;      // keep_flag offset: 1 (heavy above fast argument 0), +inf (no heavy ids)
};

// floor((s + lo) * 2^E) for a normalised float-float pair (s in [1/2, 2),
// |lo| <= ulp(s)/2), by integer operations; E <= 62.
__device__ __forceinline__ unsigned long long fixed_pair(float s, float lo, int E)
{
    const uint32_t sb = __float_as_uint(s);
    const int es = (int)(sb >> 23) - 127;              // -1 or 0
    const uint32_t ms = (sb & 0x7FFFFFu) | 0x800000u;  // s = ms * 2^(es - 23)
    // lo * 2^(45 - es): |.| <= 2^21, rounded to an integer
    const float L = __fmaf_rn(lo, es < 0 ? 70368744177664.0f : 35184372088832.0f, kMagic);
    const long long M = ((long long)ms << 22) + (long long)(__float_as_int(L) - __float_as_int(kMagic));
    const int sh = E + es - 45;  // (s + lo) * 2^E = M * 2^sh
    if (sh >= 0)
        return (unsigned long long)M << sh;
    if (sh <= -63)
        return 0ull;
    return (unsigned long long)M >> (-sh);
}

// v * 2^(60 - sc), truncated towards zero, for a float v with |v| * 2^(60 - sc)
// < 2^63, signed, by integer operations.
__device__ __forceinline__ long long fixed60_signed(float v, int sc = 0)
{
    const uint32_t b = __float_as_uint(v);
    const int ex = (int)((b >> 23) & 0xFFu);
    if (ex == 0)
        return 0;  // zero or below 2^-126
    const unsigned long long mant = (b & 0x7FFFFFu) | 0x800000u;
    const int sh = ex - 90 - sc;  // |v| * 2^(60 - sc) = mant * 2^(ex - 90 - sc)
    const unsigned long long mag = sh >= 0 ? mant << sh : (sh <= -24 ? 0ull : mant >> (-sh));
    return (b >> 31) ? -(long long)mag : (long long)mag;
}

// 2^(l * K - mref) on the 2^-60 grid, to about 2^-36 relative, by float32
// operations only (each rounding explicit, so that every call site computes
// the same bits).  Needs |l * K| < 2^21 (the caller's 'exact' rows).
__device__ __forceinline__ unsigned long long exact_weight(float l, const ExactRow &er)
{
    const float ph = __fmul_rn(l, er.khi);
    float pl = __fmaf_rn(l, er.khi, -ph);  // l*khi = ph + pl exactly (Dekker)
    pl = __fmaf_rn(l, er.klo, pl);         // + l*klo
    const float t = __fadd_rn(ph, kMagic);
    float f = __fsub_rn(ph, __fsub_rn(t, kMagic));  // ph - rint(ph): exact, |f| <= 1/2
    int n = __float_as_int(t) - __float_as_int(kMagic);
    if (er.wide) {  // |pl| up to 2^-2: two-sum f + pl (Knuth) and split again
        const float s = __fadd_rn(f, pl);
        const float bb = __fsub_rn(s, f);
        const float e = __fadd_rn(__fsub_rn(f, __fsub_rn(s, bb)), __fsub_rn(pl, bb));
        const float t1 = __fadd_rn(s, kMagic);
        f = __fsub_rn(s, __fsub_rn(t1, kMagic));
        n += __float_as_int(t1) - __float_as_int(kMagic);
        pl = e;
    }
    // f = i/32 + r with |r| <= 1/64, r exact
    const float t2 = __fmaf_rn(f, 32.0f, kMagic);
    const int i = min(max(__float_as_int(t2) - __float_as_int(kMagic) + 16, 0), 32);  // [0, 32] already
    const float r = __fmaf_rn(__fsub_rn(t2, kMagic), -0.03125f, f);
    // 2^(r + pl) - 1 = hh + Q: first-order part as an exact pair, the rest small
    const float h = __fmul_rn(r, kLn2);
    const float he = __fmaf_rn(r, kLn2, -h);
    const float g = __fmul_rn(pl, kLn2);
    const float hh = __fadd_rn(h, g);
    const float gb = __fsub_rn(hh, h);
    const float eg = __fadd_rn(__fsub_rn(h, __fsub_rn(hh, gb)), __fsub_rn(g, gb));
    const float rs = __fadd_rn(r, pl);
    const float r2 = __fmul_rn(rs, rs);
    float q = __fmaf_rn(rs, kC4, kC3);
    q = __fmaf_rn(rs, q, kC2);
    float Q = __fmaf_rn(r2, q, he);
    Q = __fadd_rn(Q, eg);
    Q = __fmaf_rn(rs, kLn2Lo, Q);
    // 2^(i/32) * (1 + hh + Q) as a normalised float-float pair
    const float th = __ldg(&kExp2Table.hi[i]), tl = __ldg(&kExp2Table.lo[i]);
    const float u = __fmul_rn(th, hh);
    const float ue = __fmaf_rn(th, hh, -u);
    const float s0 = __fadd_rn(th, u);  // |u| < th: fast two-sum
    const float se = __fsub_rn(u, __fsub_rn(s0, th));
    float lo = __fmaf_rn(th, Q, tl);
    lo = __fmaf_rn(tl, hh, lo);
    lo = __fadd_rn(lo, ue);
    lo = __fadd_rn(lo, se);
    const float s = __fadd_rn(s0, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, s0));
    return fixed_pair(s, lo, n + er.e60);
}

// Pass-2 weights of one decided row (or of a target/draft pair).
enum P2Mode {
    kP2Full = 0,      // p (the bonus row, or a degenerate residual)
    kP2Residual = 1,  // max(0, p - q) from a target and a draft row
    kP2Zero = 2       // p without some ids (point-mass residual; a tree node's rejected candidates)
};

// Per-sequence constants of pass 2, identical in every CTA of the cluster.
struct P2Seq {
    ExactRow rt, rd;  // target row; draft row (residual)
    int mode;
    int zero_at, zero_chunk;  // kP2Zero: one removed id (-1: none) and its chunk
    const int *zset;          // kP2Zero: nz more removed ids (shared memory)
    int nz;
};

// ExactRow of a row with merged pass-1 statistics st at temperature temp:
// mref = st.m + e, 2^e >= the row's float32 normaliser, so that each weight is
// at most ~1 and a row total at most ~1 on the 2^-60 grid.
__device__ __forceinline__ ExactRow exact_row(const RowStat &st, float temp)
{
    ExactRow er;
    // K = (kLog2e + kLog2eLo) / temp as a float-float pair, by float32
    // operations only (FP64 is a slow pipe on this GPU): q = RN(kLog2e / temp)
    // leaves the exact remainder kLog2e - q * temp (one FMA).  khi is then
    // stepped one ulp down when needed so that klo > 0: l = -inf must give
    // -inf, not -inf + inf.
    const float q = __fdiv_rn(kLog2e, temp);
    const float rem = __fmaf_rn(-q, temp, kLog2e);
    const float lo = __fdiv_rn(__fadd_rn(rem, kLog2eLo), temp);  // |lo| <= ulp(q) / 2
    er.khi = lo > 0.0f ? q : __uint_as_float(__float_as_uint(q) - 1u);
    er.klo = lo > 0.0f ? lo : __fadd_rn(lo, __fsub_rn(q, er.khi));
    const float z = st.hi + st.lo;  // >= 1/2
    const int ez = (int)((__float_as_uint(z) >> 23) & 0xFFu) - 126;  // z < 2^ez
    const float mref = st.m + (float)ez;
    er.nmf = kFastRef - st.m;  // mf = m - kFastRef
    er.sf = ez + (int)kFastRef;
    er.e60 = 60 - (int)mref;
    const float am = fabsf(st.m) + 48.0f;  // bound on |l * K| over heavy ids
    er.wide = am >= 4096.0f;
    // heavy: weight above 2^-(kHeavySpan + 1) of the row's largest l * K, i.e.
    // fast argument l * K - m + kFastRef above 0
    er.heavy = am < 2097152.0f ? 0.0f : INFINITY;
    er.koff = am < 2097152.0f ? 1.0f : INFINITY;
    er.c = __fdiv_rn(1.0f / (float)(1 << (int)kFastRef), z);
    return er;
}

// Fast pass over one chunk: the float32 weights of the non-heavy ids summed in
// id order (J only and all), which ids are heavy and which are in J.  runt /
// rund receive the running J sums after each id (the owner's final search).
struct ChunkP2 {
    float jt, at, jd, ad;  // non-heavy weights: in J, all (target, draft)
    uint32_t heavy;        // bit e: target id e heavy; bit 8 + e: draft id e heavy
    uint32_t inj;          // bit e: id e in J
};

// sat(a * b + c) with subnormal inputs and results flushed to zero: with
// |b| = 2^127 it maps every finite a to exactly 0 or 1 (NaN gives 0).
__device__ __forceinline__ float fma_ftz_sat(float a, float b, float c)
{
    float d;
    asm("fma.rn.ftz.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 1 for a tail id (fast argument at most 0, a subnormal counting as 0, or any
// id of a row without exact weights, whose koff is +inf), 0 for a heavy one;
// -inf gives 1.
__device__ __forceinline__ float keep_flag(float y, const ExactRow &er)
{
    return fma_ftz_sat(y, -0x1p127f, er.koff);
}

// The low 8 bits of a float holding an integer in [0, 255].
__device__ __forceinline__ uint32_t float_bits8(float m)
{
    return __float_as_uint(__fadd_rn(m, 8388608.0f)) & 0xFFu;
}

template <typename T, bool RESID, bool FULL = false>
__device__ __forceinline__ ChunkP2 p2_chunk(const uint4 &tv, const uint4 &dv, int c, const P2Seq &ps,
                                            float (&runt)[Elem<T>::W], float (&rund)[Elem<T>::W])
{
    constexpr int W = Elem<T>::W, P = W / 2;
    if constexpr (FULL) {  // p itself (J = every id): one sum, no J flags
        const float2 kh = make_float2(ps.rt.khi, ps.rt.khi), kl = make_float2(ps.rt.klo, ps.rt.klo);
        const float2 nmt = make_float2(ps.rt.nmf, ps.rt.nmf);
        ChunkP2 o{0.0f, 0.0f, 0.0f, 0.0f, 0u, (1u << W) - 1u};
        float tm = 0.0f;  // tail ids as a bit mask held in a float (exact below 2^24)
#pragma unroll
        for (int q = 0; q < P; ++q) {
            const float2 l = pair<T>(tv, q);
            float2 y = __ffma2_rn(l, kh, nmt);
            y = __ffma2_rn(l, kl, y);
            const float2 w = ex2_pair(y);
            const float k0 = keep_flag(y.x, ps.rt), k1 = keep_flag(y.y, ps.rt);
            tm = __fmaf_rn(k0, (float)(1 << (2 * q)), tm);
            tm = __fmaf_rn(k1, (float)(2 << (2 * q)), tm);
            o.jt = __fmaf_rn(w.x, k0, o.jt);
            runt[2 * q] = o.jt;
            o.jt = __fmaf_rn(w.y, k1, o.jt);
            runt[2 * q + 1] = o.jt;
        }
        o.heavy = ~float_bits8(tm) & ((1u << W) - 1u);
        o.at = o.jt;
        return o;
    }
    const float2 kh = make_float2(ps.rt.khi, ps.rt.khi), kl = make_float2(ps.rt.klo, ps.rt.klo);
    const float2 nmt = make_float2(ps.rt.nmf, ps.rt.nmf), nmd = make_float2(ps.rd.nmf, ps.rd.nmf);
    uint32_t inj = (1u << W) - 1u;
    if (!RESID && ps.mode == kP2Zero) {
        if (c == ps.zero_chunk)
            inj &= ~(1u << (ps.zero_at - c * W));
        for (int z = 0; z < ps.nz; ++z) {
            const int d = ps.zset[z] - c * W;
            if (d >= 0 && d < W)
                inj &= ~(1u << d);
        }
    }
    ChunkP2 o{0.0f, 0.0f, 0.0f, 0.0f, 0u, 0u};
    float tm = 0.0f, dm = 0.0f, jm = 0.0f;  // tail ids (target, draft) and J, as float bit masks
    // one id at a time, in id order (the running sums are sequential)
    auto step = [&](int e, float yt, float wt, float yd, float wd) {
        const float kt = keep_flag(yt, ps.rt);
        const float a = __fmul_rn(wt, kt);
        tm = __fmaf_rn(kt, (float)(1 << e), tm);
        float jf;
        if (RESID) {
            const float kd = keep_flag(yd, ps.rd);
            const float b = __fmul_rn(wd, kd);
            dm = __fmaf_rn(kd, (float)(1 << e), dm);
            // J: p > q by the float32 probabilities, as an exact 0 or 1
            jf = fma_ftz_sat(__fmaf_rn(wt, ps.rt.c, -__fmul_rn(wd, ps.rd.c)), 0x1p127f, 0.0f);
            o.ad = __fadd_rn(o.ad, b);
            o.jd = __fmaf_rn(b, jf, o.jd);
        } else {
            jf = ((inj >> e) & 1u) ? 1.0f : 0.0f;
        }
        jm = __fmaf_rn(jf, (float)(1 << e), jm);
        o.at = __fadd_rn(o.at, a);
        o.jt = __fmaf_rn(a, jf, o.jt);
        runt[e] = o.jt;
        rund[e] = o.jd;
    };
#pragma unroll
    for (int q = 0; q < P; ++q) {
        const float2 l = pair<T>(tv, q);
        float2 y = __ffma2_rn(l, kh, nmt);
        y = __ffma2_rn(l, kl, y);
        const float2 w = ex2_pair(y);
        float2 x = make_float2(0.0f, 0.0f), v = make_float2(0.0f, 0.0f);
        if (RESID) {
            const float2 ld = pair<T>(dv, q);
            x = __ffma2_rn(ld, kh, nmd);
            x = __ffma2_rn(ld, kl, x);
            v = ex2_pair(x);
        }
        step(2 * q, y.x, w.x, x.x, v.x);
        step(2 * q + 1, y.y, w.y, x.y, v.y);
    }
    o.heavy = (~float_bits8(tm) & ((1u << W) - 1u)) | (RESID ? (~float_bits8(dm) & ((1u << W) - 1u)) << 8 : 0u);
    o.inj = float_bits8(jm);
    return o;
}

// Element e of a staged 16-byte chunk.
template <typename T> __device__ __forceinline__ float staged_elem(const uint4 *chunk, int e)
{
    if (sizeof(T) == 2)
        return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short *>(chunk)[e] << 16);
    return reinterpret_cast<const float *>(chunk)[e];
}

// Dynamic shared memory of pass 2: the chunks of one warp batch (kP2Slots
// slots: kP2Unroll chunks of one row, or half as many of two) and the queue of
// their heavy ids.
// The small-grid full sweep (2 CTAs per SM, registers and shared memory to
// spare) takes twice as many chunks per batch: fewer, longer trips where the
// few resident warps leave latency exposed.
constexpr int kP2Slots = kP2Unroll;
constexpr int kP2SlotsWide = 2 * kP2Unroll;
template <int S> struct P2SmemT {
    static_assert(S <= 8, "queue entries keep the slot in 3 bits");
    uint4 stage[kWarps][S][32];
    unsigned short queue[kWarps][S * 32 * 8];
};
using P2Smem = P2SmemT<kP2Slots>;
constexpr int kP2SmemBytes = (int)sizeof(P2Smem);
constexpr int kP2SmemBytesWide = (int)sizeof(P2SmemT<kP2SlotsWide>);

typedef __int128 i128;
typedef unsigned __int128 u128;

// Residual weight of a sum: JT*B - JD*A; the weights themselves otherwise (B = 1, JD = 0).
__device__ __forceinline__ i128 p2_value(unsigned long long jt, unsigned long long jd, unsigned long long A,
                                         unsigned long long B)
{
    return (i128)((u128)jt * B) - (i128)((u128)jd * A);
}

// floor(u * R) exactly, u a float in [0, 1), 0 <= R < 2^124.
__device__ __forceinline__ i128 scaled_floor128(float u, i128 R)
{
    const uint32_t bits = __float_as_uint(u);
    const uint32_t ex = (bits >> 23) & 0xFFu;
    if (R <= 0 || (ex == 0 && (bits & 0x7FFFFFu) == 0))
        return 0;
    const unsigned long long mant = (bits & 0x7FFFFFu) | (ex ? 0x800000u : 0u);
    const int sh = 150 - (int)(ex ? ex : 1u);  // u = mant * 2^-sh, sh >= 24
    const u128 ur = (u128)R;
    const u128 hi = (u128)mant * (unsigned long long)(ur >> 64);  // mant * R = hi * 2^64 + lo
    const u128 lo = (u128)mant * (unsigned long long)ur;
    if (sh >= 192)
        return 0;
    if (sh <= 64)
        return (i128)((hi << (64 - sh)) + (lo >> sh));
    return (i128)((hi + (lo >> 64)) >> (sh - 64));
}

// Inclusive block scan of a signed 128-bit value over the CTA; also the total.
__device__ __forceinline__ i128 block_scan_i128(i128 v, i128 &total, i128 *warp_tot)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long lo = __shfl_up_sync(0xffffffffu, (unsigned long long)v, d);
        const long long hi = __shfl_up_sync(0xffffffffu, (long long)(v >> 64), d);
        if (lane >= d)
            v += (i128)(((u128)(unsigned long long)hi << 64) | lo);
    }
    __syncthreads();
    if (lane == 31)
        warp_tot[wid] = v;
    __syncthreads();
    i128 before = 0, t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w < wid)
            before += warp_tot[w];
        t += warp_tot[w];
    }
    total = t;
    return v + before;
}

// Lowest thread of the CTA with flag set (kThreads if none); all threads call it.
__device__ __forceinline__ int block_first(bool flag, int *wmin)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    __syncthreads();
    if (lane == 0)
        wmin[wid] = b ? wid * 32 + __ffs(b) - 1 : kThreads;
    __syncthreads();
    int m = kThreads;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        m = min(m, wmin[w]);
    return m;
}

// ---------------------------------------------------------------------------
// barriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// shared state and the per-sequence protocol common to both kernels
// ---------------------------------------------------------------------------
struct SharedState {
    RowStat warp_part[kMaxRows][kWarps];
    RowStat recv[kMaxCluster][kMaxRows];  // written remotely by every CTA of the cluster
    RowStat row[kMaxRows];                // merged statistics, identical in every CTA
    unsigned long long p2w[kWarps][4];    // pass 2: sums of each warp range (J target, J draft, all target, all draft)
    unsigned long long p2recv[2][kMaxCluster][4];  // pass 2: each CTA's sums, written remotely [attempt][rank]
    i128 p2scan[kWarps];                  // pass 2: block-scan partials
    int hist[kMaxRows + 1];
    int cnt[kWarps];
    int seq;
    int seq_g;
    float seq_temp;
    int bin;
    int rank_in_bin;
    RowStat recv_pos[2][kMaxCluster][2];  // early-exit kernel: [position parity][source rank][t / d]
    int n;
    int bits;
    int stop;
    int drafted[SPEC_MAX_GAMMA];  // the sequence's drafted ids (full-sweep decision)
};

// Tree kernel: the sequence's tree and the walk's state.
constexpr int kMaxTree = SPEC_MAX_TREE_NODES;
static_assert(kMaxTree <= kThreads, "one thread per tree node");
struct TreeShared {
    int parent[kMaxTree];
    int token[kMaxTree];
    int child[kMaxTree];  // children of the current node, in index order
    int rej[kMaxTree];    // ids rejected at the current node (the final sample's zero set)
    float glog[kMaxTree]; // target logit of each child's id
    float uch[kMaxTree];  // each child's uniform
    int wcnt[kWarps];
    int next, nrej, bits;
};

struct Seq {
    int b, g, gmax, V, rank, C, c0, c1;
    bool sampled;
    bool point;   // deterministic proposals: no draft rows, q_i(x_i) = 1
    bool drafts;  // sampled with draft rows to read
    float k;      // log2(e) / T for sampled sequences (pass 1)
    float temp;   // T
    size_t rowlen;
};

// Problems that decide which rows would be read: a bad draft count or
// temperature (identical in every CTA of the cluster).  Drafted ids are checked
// here only on this error path; otherwise the decision checks them, one lane
// per position, off the critical path.
__device__ __forceinline__ uint32_t check_inputs(const Params &p, int b, int g, float temp)
{
    if (g < 0 || g > p.gmax)
        return SPEC_STATUS_BAD_NUM_DRAFT;
    if (!(isnan(temp) || isinf(temp) || temp < 0.0f || (temp > 0.0f && temp < FLT_MIN)))
        return 0;
    uint32_t bad = SPEC_STATUS_BAD_TEMPERATURE;
    for (int i = 0; i < g; ++i) {
        const int x = p.tokens[(size_t)b * p.gmax + i];
        if (x < 0 || x >= p.V)
            bad |= SPEC_STATUS_BAD_TOKEN;
    }
    return bad;
}

// Rank 0 marks the diagnostics of a sequence as "not computed" (NaN).
__device__ __forceinline__ void init_diagnostics(const Params &p, int b, int rank)
{
    const int tid = threadIdx.x, gmax = p.gmax;
    if (rank != 0 || tid > gmax)
        return;
    const float nan = __int_as_float(0x7fc00000);
    if (p.logz_t)
        p.logz_t[(size_t)b * (gmax + 1) + tid] = nan;
    if (tid < gmax) {
        if (p.p_hat)
            p.p_hat[(size_t)b * gmax + tid] = nan;
        if (p.q_hat)
            p.q_hat[(size_t)b * gmax + tid] = nan;
        if (p.logz_d)
            p.logz_d[(size_t)b * gmax + tid] = nan;
    }
    if (tid == 0 && p.resid_mass)
        p.resid_mass[b] = nan;
}

// Rank 0 writes -1 tokens and the status of an invalid sequence.
__device__ __forceinline__ void write_invalid(const Params &p, int b, int rank, uint32_t bits)
{
    if (rank != 0)
        return;
    const int tid = threadIdx.x;
    if (tid <= p.gmax)
        p.out_tokens[(size_t)b * (p.gmax + 1) + tid] = -1;
    if (tid == 0) {
        if (p.out_num)
            p.out_num[b] = 0;
        if (p.seq_status)
            p.seq_status[b] = (int32_t)bits;
        if (p.status)
            atomicOr(p.status, bits);
    }
}

// Logical row r (target i -> i, draft i -> g + 1 + i) read at sweep position
// 'step'.  Order t_g, t_{g-1}, d_{g-1}, ..., t_0, d_0: the rows most likely to
// be decided (small i) come last, so pass 2 finds them in L2.
__device__ __forceinline__ int row_at_step(int step, int g, bool sampled)
{
    if (step == 0)
        return g;
    if (!sampled)
        return g - step;
    const int i = g - 1 - (step - 1) / 2;
    return ((step - 1) & 1) ? g + 1 + i : i;
}

template <typename T> __device__ __forceinline__ const T *row_ptr(const Params &p, const Seq &s, int r)
{
    if (r <= s.g)
        return reinterpret_cast<const T *>(p.target) + ((size_t)s.b * (s.gmax + 1) + r) * s.rowlen;
    return reinterpret_cast<const T *>(p.draft) + ((size_t)s.b * s.gmax + (r - s.g - 1)) * s.rowlen;
}

// Merges the warp partials of each row, sends them to every CTA of the cluster
// and merges what arrives in rank order.  All threads of the CTA call it; the
// cluster arrive (relaxed) must have been issued at kernel start.
__device__ __forceinline__ void exchange_rows(SharedState &sh, const Seq &s, int nrows)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    __syncthreads();
    cluster_wait();  // every CTA of the cluster is running: DSMEM is addressable
    if (tid < nrows) {
        RowStat v = sh.warp_part[tid][0];
        for (int w = 1; w < kWarps; ++w)
            v = s.sampled ? soft_merge(v, sh.warp_part[tid][w]) : arg_merge(v, sh.warp_part[tid][w]);
        for (int dst = 0; dst < s.C; ++dst)
            *cluster.map_shared_rank(&sh.recv[s.rank][tid], dst) = v;
    }
    cluster_sync_all();
    if (tid < nrows) {
        RowStat v = sh.recv[0][tid];
        for (int src = 1; src < s.C; ++src)
            v = s.sampled ? soft_merge(v, sh.recv[src][tid]) : arg_merge(v, sh.recv[src][tid]);
        sh.row[tid] = v;
    }
    __syncthreads();
}

// Accept decisions (warp 0: lane i tests draft position i; a ballot finds the
// cut) and rank 0's output writes.  Returns true if the sequence goes on to
// pass 2 (sampled and valid).  All threads call it.
// Acceptance counters of a verified sequence: drafted ids, accepted ids, and
// one round (the page on vLLM exports the same two counts; their ratio is the
// acceptance rate a, and accepted / rounds + 1 the tokens per round).
__device__ __forceinline__ void count_round(unsigned long long *counters, unsigned long long *hist, int g, int n)
{
    if (hist)
        atomicAdd(&hist[n < SPEC_MAX_GAMMA ? n : SPEC_MAX_GAMMA], 1ull);
    if (!counters)
        return;
    atomicAdd(&counters[0], (unsigned long long)g);
    atomicAdd(&counters[1], (unsigned long long)n);
    atomicAdd(&counters[2], 1ull);
}

// What warp 0's lane i needs for position i's decision, loaded before pass 1
// so the loads overlap the sweep: the drafted id and (sampled) the target and
// draft logits at it.
struct Gathered {
    int x;      // drafted id
    float lt, ld;  // target and draft logits at x (sampled sequences)
    float u;    // the position's accept-test uniform (sampled sequences)
};

// Position i's drafted id and uniform (lane i of warp 0).  Issued in the
// prologue and not waited for: the values are first used at the decision.
__device__ __forceinline__ Gathered gather_ids(const Params &p, const Seq &s, int i)
{
    Gathered gt{-1, 0.0f, 0.0f, 0.0f};
    if (i < s.g) {
        gt.x = p.tokens[(size_t)s.b * s.gmax + i];
        if (s.sampled)
            gt.u = p.uniforms[(size_t)s.b * (s.gmax + 1) + i];
    }
    return gt;
}

// The logits at the drafted id, once the id has arrived: issued after pass 1,
// so they land during the cluster exchange.
template <typename T> __device__ __forceinline__ void gather_logits(const Params &p, const Seq &s, int i, Gathered &gt)
{
    if (i < s.g && s.sampled && gt.x >= 0 && gt.x < s.V) {
        const T *tr = row_ptr<T>(p, s, i);
        if (sizeof(T) == 2)
            gt.lt = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(tr)[gt.x]);
        else
            gt.lt = reinterpret_cast<const float *>(tr)[gt.x];
        if (s.drafts) {
            const T *dr = row_ptr<T>(p, s, s.g + 1 + i);
            if (sizeof(T) == 2)
                gt.ld = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(dr)[gt.x]);
            else
                gt.ld = reinterpret_cast<const float *>(dr)[gt.x];
        }
    }
}

template <typename T> __device__ __forceinline__ Gathered gather_position(const Params &p, const Seq &s, int i)
{
    Gathered gt = gather_ids(p, s, i);
    gather_logits<T>(p, s, i, gt);
    return gt;
}

template <typename T>
__device__ __forceinline__ bool decide_and_write(const Params &p, SharedState &sh, const Seq &s, const Gathered &gt)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int b = s.b, g = s.g, gmax = s.gmax;
    if (wid == 0) {
        bool ok = false, valid = true, tok_bad = false;
        float phat = 0.0f, qhat = 0.0f;
        if (lane < g) {
            const int x = gt.x;
            tok_bad = x < 0 || x >= p.V;
            if (tok_bad) {
                // an invalid id: no gather; the sequence is reported invalid below
            } else if (!s.sampled) {
                ok = x == sh.row[lane].idx;
            } else {
                const RowStat st = sh.row[lane];
                valid = soft_row_ok(st);
                phat = ex2_approx(fmaf(gt.lt, s.k, -st.m)) / (st.hi + st.lo);
                qhat = 1.0f;  // point-mass proposal
                if (s.drafts) {
                    const RowStat sd = sh.row[g + 1 + lane];
                    valid = valid && soft_row_ok(sd);
                    qhat = ex2_approx(fmaf(gt.ld, s.k, -sd.m)) / (sd.hi + sd.lo);
                }
                ok = valid && (gt.u * qhat < phat);
            }
        }
        const unsigned pass = __ballot_sync(0xffffffffu, ok);
        const unsigned fine = __ballot_sync(0xffffffffu, valid);
        const unsigned lanes = g >= 32 ? 0xffffffffu : ((1u << g) - 1u);
        const unsigned fail = ~pass & lanes;
        const int n = fail ? __ffs(fail) - 1 : g;
        uint32_t bits = 0;
        if (__ballot_sync(0xffffffffu, tok_bad))
            bits = SPEC_STATUS_BAD_TOKEN;
        else if (s.sampled && (n < g ? !((fine >> n) & 1u) : !soft_row_ok(sh.row[g])))
            bits = SPEC_STATUS_BAD_LOGITS;
        if (lane == 0) {
            sh.n = n;
            sh.bits = (int)bits;
        }
        if (lane < g)
            sh.drafted[lane] = gt.x;
        if (s.rank == 0 && s.sampled && lane < g) {
            if (p.p_hat)
                p.p_hat[(size_t)b * gmax + lane] = phat;
            if (p.q_hat)
                p.q_hat[(size_t)b * gmax + lane] = qhat;
        }
    }
    __syncthreads();
    const int n = sh.n;
    const uint32_t bits = (uint32_t)sh.bits;
    if (s.rank == 0) {
        int32_t *out = p.out_tokens + (size_t)b * (gmax + 1);
        if (s.sampled && tid <= g) {
            const RowStat st = sh.row[tid];
            if (p.logz_t)
                p.logz_t[(size_t)b * (gmax + 1) + tid] = (st.m + log2f(st.hi + st.lo)) * kLn2;
            if (tid < g && p.logz_d && s.drafts) {
                const RowStat sd = sh.row[g + 1 + tid];
                p.logz_d[(size_t)b * gmax + tid] = (sd.m + log2f(sd.hi + sd.lo)) * kLn2;
            }
        }
        if (tid <= gmax) {
            int v = -1;
            if (!bits) {
                if (tid < n)
                    v = sh.drafted[tid];
                else if (tid == n)
                    v = s.sampled ? INT_MIN : sh.row[n].idx;  // sampled: written by pass 2
            }
            if (v != INT_MIN)
                out[tid] = v;
        }
        if (tid == 0) {
            if (p.out_num)
                p.out_num[b] = bits ? 0 : n;
            if (p.seq_status)
                p.seq_status[b] = (int32_t)bits;
            if (bits && p.status)
                atomicOr(p.status, bits);
            if (!bits && (p.counters || p.hist))
                count_round(p.counters, p.hist, g, n);
        }
    }
    return s.sampled && !bits;
}


// The final uniform, clamped into [0, 1).
__device__ __forceinline__ float final_uniform(const Params &p, const Seq &s)
{
    float u = p.uniforms[(size_t)s.b * (s.gmax + 1) + s.gmax];
    if (!(u >= 0.0f))
        u = 0.0f;
    if (u >= 1.0f)
        u = __uint_as_float(0x3F7FFFFFu);
    return u;
}


// Cost of sequence i for the longest-first order: the rows it reads, g + 1
// target rows plus, when sampled, g draft rows; 0 for an invalid draft count.
// With point-mass proposals no draft row exists and a sampled sequence counts
// one row more for its final draw, which sweeps a row again: in a one-row call
// (gamma_max = 0) that puts the sampled rows before the greedy ones.
template <bool POINT>
__device__ __forceinline__ int seq_cost(const Params &p, int g, float temp)
{
    if (g < 0 || g > p.gmax)
        return 0;
    return g + 1 + (temp > 0.0f ? (POINT ? 1 : g) : 0);
}

struct SeqPick {
    int b;       // sequence index
    int g;       // its num_draft
    float temp;  // its temperature
};

// Sequence verified by cluster k.  With p.ordered, clusters take sequences in
// order of decreasing row count (ties by index), so the longest start first and
// the grid's tail is made of short ones; the block scheduler dispatches
// clusters in index order.  Every CTA of the cluster computes the same value.
// All threads of the CTA call it (blockDim.x >= kThreads).  The point-mass
// kernels, where batches of equal cost are common (one-row calls at one
// temperature), first test with one barrier whether every cost is the same.
template <bool POINT>
__device__ SeqPick seq_for_cluster(const Params &p, SharedState &sh, int k)
{
    if (!p.ordered)
        return SeqPick{k, p.num_draft ? p.num_draft[k] : 0, p.temperature[k]};
    constexpr int kPer = kMaxOrdered / kThreads;
    const int tid = threadIdx.x;
    const bool active = tid < kThreads;
    int cost[kPer], gv[kPer];
    float tv[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        const int i = tid * kPer + e;
        const bool in = active && i < p.B;
        gv[e] = (in && p.num_draft) ? p.num_draft[i] : 0;
        tv[e] = in ? p.temperature[i] : 0.0f;
        cost[e] = in ? seq_cost<POINT>(p, gv[e], tv[e]) : -1;
    }
    if (tid <= kMaxRows)
        sh.hist[tid] = 0;
    if constexpr (POINT) {
        // one cost for every sequence: cluster k takes sequence k (loads issued
        // before the barrier, used only then)
        const int gk = p.num_draft ? p.num_draft[k] : 0;
        const float tk = p.temperature[k];
        const int c0 = seq_cost<POINT>(p, p.num_draft ? p.num_draft[0] : 0, p.temperature[0]);
        bool same = true;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            same = same && (cost[e] < 0 || cost[e] == c0);
        if (__syncthreads_and(same))
            return SeqPick{k, gk, tk};
    } else {
        __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        if (cost[e] >= 0)
            atomicAdd(&sh.hist[cost[e]], 1);
    __syncthreads();
    if (tid < 32) {  // bins by decreasing cost: lane j holds bins kMaxRows - j and, for j < 2, 1 - j
        const int h0 = sh.hist[kMaxRows - tid];
        const int h1 = tid < 2 ? sh.hist[1 - tid] : 0;
        int inc0 = h0, inc1 = h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, inc0, o);
            const int y1 = __shfl_up_sync(0xffffffffu, inc1, o);
            if (tid >= o) {
                inc0 += y0;
                inc1 += y1;
            }
        }
        inc1 += __shfl_sync(0xffffffffu, inc0, 31);
        const unsigned in0 = __ballot_sync(0xffffffffu, k < inc0);
        const unsigned in1 = __ballot_sync(0xffffffffu, tid < 2 && k < inc1);
        const int j = in0 ? __ffs(in0) - 1 : 32 + __ffs(in1) - 1;  // k < B, so some bin holds it
        const int src = j & 31;
        const int inc = __shfl_sync(0xffffffffu, j < 32 ? inc0 : inc1, src);
        const int h = __shfl_sync(0xffffffffu, j < 32 ? h0 : h1, src);
        if (tid == 0) {
            sh.bin = kMaxRows - j;
            sh.rank_in_bin = k - (inc - h);
        }
    }
    __syncthreads();
    const int bin = sh.bin, want = sh.rank_in_bin;
    int mine = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        mine += cost[e] == bin;
    // exclusive prefix of 'mine' over threads in index order (contiguous ranges)
    const int lane = tid & 31, wid = tid >> 5;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (active && lane == 31)
        sh.cnt[wid] = incl;
    __syncthreads();
    int before = incl - mine;
    for (int w = 0; w < wid && w < kWarps; ++w)
        before += sh.cnt[w];
    if (active && before <= want && want < before + mine) {
        int r = want - before;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (cost[e] == bin) {
                if (r == 0) {
                    sh.seq = tid * kPer + e;
                    sh.seq_g = gv[e];
                    sh.seq_temp = tv[e];
                }
                --r;
            }
    }
    __syncthreads();
    return SeqPick{sh.seq, sh.seq_g, sh.seq_temp};
}

// POINT: point-mass proposals, a template parameter of the kernels so that the
// usual path carries none of its branches.
template <bool POINT>
__device__ __forceinline__ Seq make_seq(const Params &p, int C, int rank, int b, int g, float temp)
{
    Seq s;
    s.b = b;
    s.g = g;
    s.gmax = p.gmax;
    s.V = p.V;
    s.rank = rank;
    s.C = C;
    s.c0 = (int)((long long)p.num_chunks * rank / C);
    s.c1 = (int)((long long)p.num_chunks * (rank + 1) / C);
    s.sampled = temp > 0.0f;
    s.point = POINT;
    s.drafts = s.sampled && !s.point;
    s.k = s.sampled ? __fdiv_rn(kLog2e, temp) : 0.0f;
    s.temp = temp;
    s.rowlen = (size_t)p.V;
    return s;
}

// One row of pass 1 over this CTA's slice, reduced over the warp: online
// softmax statistics (sampled) or the lowest argmax (greedy).  Eight 16-byte
// loads per thread are issued before the batch is reduced.  When the slice
// gives a thread more than one batch of a row, the next batch is first
// requested into L2 (prefetch.global.L2: no registers held), so the row's
// bytes are in flight while a batch is reduced (B=256, V=128256: 86.2 us
// against 89.7 us without; prefetching across rows or two batches ahead was
// slower).
// STAGE: every chunk of the slice is also kept in shared memory, stage[c - c0],
// for a pass 2 that must not read the row again (rows in host memory).
template <typename T, bool ALIGNED, bool STAGE = false>
__device__ __forceinline__ RowStat sweep_row(const Seq &s, const T *row, uint4 *stage = nullptr)
{
    constexpr int W = Elem<T>::W;
    const int tid = threadIdx.x;
    RowAcc acc;
    acc.reset(s.c0 + tid < s.c1 ? (s.c0 + tid) * W : INT_MAX);
    const bool multi = ALIGNED && s.c1 - s.c0 > kUnroll * kThreads;
    for (int ch = s.c0 + tid; ch < s.c1; ch += kUnroll * kThreads) {
        if (multi) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int c = ch + (kUnroll + u) * kThreads;
                if (c < s.c1)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + (size_t)c * Elem<T>::W));
            }
        }
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = ch + u * kThreads;
            v[u] = c < s.c1 ? load_chunk<T, ALIGNED>(row, c, s.V) : neg_inf_chunk<T>();
        }
        if constexpr (STAGE) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int c = ch + u * kThreads;
                if (c < s.c1)
                    stage[c - s.c0] = v[u];
            }
        }
        if (s.sampled)
            acc.add_soft<T, kUnroll>(v, s.k);
        else
            acc.add_arg<T, kUnroll>(v, ch * W, kThreads * W);
    }
    return warp_reduce(acc.stat(), s.sampled);
}

// Chunk c of a decided row's slice for pass 2: loaded from the row, or (STAGED)
// taken from the copy pass 1 left in shared memory.
template <typename T, bool ALIGNED, bool STAGED>
__device__ __forceinline__ uint4 slice_chunk(const T *row, const uint4 *stage, int c, const Seq &s)
{
    if constexpr (STAGED)
        return stage[c - s.c0];
    else
        return load_chunk<T, ALIGNED>(row, c, s.V);
}


// Pass 1 when every thread holds at most K chunks of each row (small slices:
// small vocabularies or large clusters): the loads of U/K rows are issued
// together (U = 8 loads in flight, 16 for the two-CTAs-per-SM variant) and
// each row is reduced after they land, so a round needs about nrows*K/U
// memory round trips instead of nrows.  Same per-row results as sweep_row
// (same chunks, same order per thread).
template <typename T, bool ALIGNED, int K, int U = kUnroll>
__device__ __forceinline__ void sweep_rows_batched(const Params &p, SharedState &sh, const Seq &s, int nrows)
{
    constexpr int W = Elem<T>::W;
    constexpr int RB = U / K;  // rows per batch
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int first = s.c0 + tid < s.c1 ? (s.c0 + tid) * W : INT_MAX;
    for (int step0 = 0; step0 < nrows; step0 += RB) {
        uint4 v[RB][K];
#pragma unroll
        for (int rr = 0; rr < RB; ++rr) {
            const bool live = step0 + rr < nrows;
            const T *row = live ? row_ptr<T>(p, s, row_at_step(step0 + rr, s.g, s.drafts)) : nullptr;
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int c = s.c0 + u * kThreads + tid;
                v[rr][u] = (live && c < s.c1) ? load_chunk<T, ALIGNED>(row, c, s.V) : neg_inf_chunk<T>();
            }
        }
#pragma unroll
        for (int rr = 0; rr < RB; ++rr) {
            if (step0 + rr >= nrows)
                break;
            RowAcc acc;
            acc.reset(first);
            if (s.sampled)
                acc.add_soft<T, K>(v[rr], s.k);
            else
                acc.add_arg<T, K>(v[rr], s.c0 * W + tid * W, kThreads * W);
            const RowStat st = warp_reduce(acc.stat(), s.sampled);
            if (lane == 0)
                sh.warp_part[row_at_step(step0 + rr, s.g, s.drafts)][wid] = st;
        }
    }
}


// Warp w's contiguous range [r0, r1) of this CTA's slice.
__device__ __forceinline__ void warp_range(const Seq &s, int w, int &r0, int &r1)
{
    const long long n = s.c1 - s.c0;
    r0 = s.c0 + (int)(n * w / kWarps);
    r1 = s.c0 + (int)(n * (w + 1) / kWarps);
}

// Sums of one warp range (every lane gets them): JT = sum over J of the target
// weights, JD = of the draft weights, AT, AD = over all ids.
struct RangeSums {
    unsigned long long jt, jd, at, ad;
};

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Pass-2 sweep of this warp's range: chunks base + u*32 + lane, kP2Unroll
// chunks in flight per thread (U per row).  After the fast pass over a batch,
// its heavy ids are queued (slot, lane, id, J) and spread over the lanes, 32
// exact weights at a time, while the batch's chunks wait in shared memory.
// All threads of the warp call it.
template <typename T, bool ALIGNED, bool RESID, bool STAGED, bool FULL = false, int SLOTS = kP2Slots>
__device__ __forceinline__ RangeSums p2_sweep(const Seq &s, const T *trow, const T *drow, const uint4 *tst,
                                              const uint4 *dst, const P2Seq &ps, P2SmemT<SLOTS> &sm)
{
    constexpr int U = RESID ? SLOTS / 2 : SLOTS;  // chunks per row in a batch
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int r0, r1;
    warp_range(s, wid, r0, r1);
    unsigned long long jt = 0, jd = 0, hat = 0, had = 0;
    float ath = 0.0f, atl = 0.0f, adh = 0.0f, adl = 0.0f;
    for (int base = r0; base < r1; base += 32 * U) {
        int queued = 0;  // heavy ids of this batch (uniform over the warp)
        {
            uint4 tv[U], dv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = base + u * 32 + lane;
                tv[u] = c < r1 ? slice_chunk<T, ALIGNED, STAGED>(trow, tst, c, s) : neg_inf_chunk<T>();
                dv[u] = (RESID && c < r1) ? slice_chunk<T, ALIGNED, STAGED>(drow, dst, c, s) : neg_inf_chunk<T>();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (base + u * 32 >= r1)
                    break;  // uniform over the warp
                const int c = base + u * 32 + lane;
                float runt[Elem<T>::W], rund[Elem<T>::W];
                const ChunkP2 o = p2_chunk<T, RESID, FULL>(tv[u], dv[u], c, ps, runt, rund);
                jt += to_fixed60(o.jt, ps.rt.sf);
                compensated_add(ath, atl, o.at);
                if (RESID) {
                    jd += to_fixed60(o.jd, ps.rd.sf);
                    compensated_add(adh, adl, o.ad);
                }
                if (!__any_sync(0xffffffffu, o.heavy != 0))
                    continue;
                const int slot = RESID ? 2 * u : u;
                sm.stage[wid][slot][lane] = tv[u];
                if (RESID)
                    sm.stage[wid][slot + 1][lane] = dv[u];
                const int cnt = __popc(o.heavy);
                int incl = cnt;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d)
                        incl += y;
                }
                int off = queued + incl - cnt;
                queued += __shfl_sync(0xffffffffu, incl, 31);
                for (uint32_t hm = o.heavy; hm; hm &= hm - 1u) {
                    const int bit = __ffs(hm) - 1, e = bit & 7;
                    sm.queue[wid][off++] = (unsigned short)((slot + (bit >> 3)) | (lane << 3) | (e << 8) |
                                                            (((o.inj >> e) & 1u) << 11));
                }
            }
        }
        if (!queued)
            continue;
        __syncwarp();
        for (int k = lane; k < queued; k += 32) {
            const unsigned ent = sm.queue[wid][k];
            const int slot = ent & 7;
            const bool row = RESID && (slot & 1);
            const float l = staged_elem<T>(&sm.stage[wid][slot][(ent >> 3) & 31], (ent >> 8) & 7);
            const unsigned long long w = exact_weight(l, row ? ps.rd : ps.rt);
            const bool inj = (ent >> 11) & 1u;
            if (row) {
                had += w;
                jd += inj ? w : 0ull;
            } else {
                hat += w;
                jt += inj ? w : 0ull;
            }
        }
        __syncwarp();
    }
    RangeSums r;
    r.jt = warp_sum_u64(jt);
    r.jd = warp_sum_u64(jd);
    r.at = warp_sum_u64(hat + (unsigned long long)((long long)to_fixed60(ath, ps.rt.sf) +
                                                    fixed60_signed(atl, ps.rt.sf)));
    r.ad = warp_sum_u64(had + (unsigned long long)((long long)to_fixed60(adh, ps.rd.sf) +
                                                    fixed60_signed(adl, ps.rd.sf)));
    return r;
}

__device__ __forceinline__ i128 shfl_i128(i128 v, int src)
{
    const unsigned long long lo = __shfl_sync(0xffffffffu, (unsigned long long)v, src);
    const long long hi = __shfl_sync(0xffffffffu, (long long)(v >> 64), src);
    return (i128)(((u128)(unsigned long long)hi << 64) | lo);
}

// Inclusive scan of a signed 128-bit value over the warp's lanes.
__device__ __forceinline__ i128 warp_scan_i128(i128 v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long lo = __shfl_up_sync(0xffffffffu, (unsigned long long)v, d);
        const long long hi = __shfl_up_sync(0xffffffffu, (long long)(v >> 64), d);
        if (lane >= d)
            v += (i128)(((u128)(unsigned long long)hi << 64) | lo);
    }
    return v;
}

// Signed 128-bit value as a double (diagnostics only).
__device__ __forceinline__ double i128_to_double(i128 v)
{
    const bool neg = v < 0;
    const u128 m = neg ? (u128)(-v) : (u128)v;
    const double d = (double)(unsigned long long)(m >> 64) * 18446744073709551616.0 + (double)(unsigned long long)m;
    return neg ? -d : d;
}

// The owner CTA's search inside warp range [r0, r1) of its slice, which holds
// the draw (rel = theta - start of the range, on the exact grid).  The range is
// recomputed chunk by chunk with the sweep's arithmetic (identical bits), one
// chunk per thread and pass; the exact weights of a warp's heavy ids in J are
// queued and computed one per lane, then added to their chunks' sums with
// shared-memory atomics (integer sums: any order gives the same bits).  A
// block scan finds the chunk, and the warp holding it the id from the running
// sums in id order.  All threads of the CTA call it.
template <typename T, bool ALIGNED, bool RESID, bool STAGED, bool FULL = false, int SLOTS = kP2Slots>
__device__ __noinline__ void p2_owner(i128 *scan_tmp, int *wmin, P2SmemT<SLOTS> &sm, const Seq &s, const T *trow,
                                      const T *drow, const uint4 *tst, const uint4 *dst, const P2Seq &ps, int r0,
                                      int r1, i128 rel, unsigned long long A, unsigned long long B, int32_t *outn)
{
    constexpr int W = Elem<T>::W;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // per warp: slots 0 (target) and 1 (draft) stage the lanes' chunks, slot 2
    // holds each lane's sums of exact weights (target, draft)
    unsigned long long *hs = reinterpret_cast<unsigned long long *>(&sm.stage[wid][2][0]);
    i128 carry = 0;
    for (int base = r0; base < r1; base += kThreads) {
        const int c = base + tid;
        uint4 tv = neg_inf_chunk<T>(), dv = neg_inf_chunk<T>();
        float runt[W], rund[W];
        ChunkP2 o{0.0f, 0.0f, 0.0f, 0.0f, 0u, 0u};
        i128 v = 0;
        if (c < r1) {
            tv = slice_chunk<T, ALIGNED, STAGED>(trow, tst, c, s);
            if (RESID)
                dv = slice_chunk<T, ALIGNED, STAGED>(drow, dst, c, s);
            o = p2_chunk<T, RESID, FULL>(tv, dv, c, ps, runt, rund);
        }
        // heavy ids in J: queued (slot, lane, element) and computed one per lane
        uint32_t hj = o.heavy & (o.inj | (o.inj << 8));
        hs[2 * lane] = 0ull;
        hs[2 * lane + 1] = 0ull;
        __syncwarp();
        int queued = 0;
        if (__any_sync(0xffffffffu, hj != 0)) {
            sm.stage[wid][0][lane] = tv;
            sm.stage[wid][1][lane] = dv;
            const int cnt = __popc(hj);
            int incl = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += y;
            }
            int off = incl - cnt;
            queued = __shfl_sync(0xffffffffu, incl, 31);
            for (; hj; hj &= hj - 1u) {
                const int bit = __ffs(hj) - 1;
                sm.queue[wid][off++] = (unsigned short)((bit >> 3) | (lane << 3) | ((bit & 7) << 8));
            }
            __syncwarp();
            for (int k = lane; k < queued; k += 32) {
                const unsigned ent = sm.queue[wid][k];
                const int row = ent & 1, src = (ent >> 3) & 31;
                const float l = staged_elem<T>(&sm.stage[wid][row][src], (ent >> 8) & 7);
                atomicAdd(&hs[2 * src + row], exact_weight(l, row ? ps.rd : ps.rt));
            }
        }
        __syncwarp();
        if (c < r1) {
            const unsigned long long jt = to_fixed60(o.jt, ps.rt.sf) + hs[2 * lane];
            const unsigned long long jd = RESID ? to_fixed60(o.jd, ps.rd.sf) + hs[2 * lane + 1] : 0ull;
            v = RESID ? p2_value(jt, jd, A, B) : (i128)jt;
        }
        __syncwarp();
        i128 total;
        const i128 incl = block_scan_i128(v, total, scan_tmp);
        const int first = block_first(c < r1 && carry + incl > rel, wmin);
        if (first < kThreads) {
            // the warp holding that chunk finds the id: lane e (< W) holds id e's
            // running sums, lanes e and W + e its exact weights (if heavy, in J)
            if ((first >> 5) == (tid >> 5)) {
                const int src = first & 31, lane = tid & 31, e = lane & (W - 1), row = lane / W;
                const i128 off = rel - (carry + incl - v);  // 0 <= off < v in the source lane
                const long long off_hi = __shfl_sync(0xffffffffu, (long long)(off >> 64), src);
                const unsigned long long off_lo = __shfl_sync(0xffffffffu, (unsigned long long)off, src);
                const i128 off_s = (i128)(((u128)(unsigned long long)off_hi << 64) | off_lo);
                uint4 t2, d2;
                t2.x = __shfl_sync(0xffffffffu, tv.x, src);
                t2.y = __shfl_sync(0xffffffffu, tv.y, src);
                t2.z = __shfl_sync(0xffffffffu, tv.z, src);
                t2.w = __shfl_sync(0xffffffffu, tv.w, src);
                d2.x = __shfl_sync(0xffffffffu, dv.x, src);
                d2.y = __shfl_sync(0xffffffffu, dv.y, src);
                d2.z = __shfl_sync(0xffffffffu, dv.z, src);
                d2.w = __shfl_sync(0xffffffffu, dv.w, src);
                const uint32_t heavy = __shfl_sync(0xffffffffu, o.heavy, src);
                const uint32_t inj = __shfl_sync(0xffffffffu, o.inj, src);
                float rt_e = 0.0f, rd_e = 0.0f;
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    const float x = __shfl_sync(0xffffffffu, runt[k], src);
                    const float y = __shfl_sync(0xffffffffu, rund[k], src);
                    if (e == k) {
                        rt_e = x;
                        rd_e = y;
                    }
                }
                unsigned long long wv = 0;
                if (row < 2 && ((inj >> e) & 1u) && ((heavy >> (row * 8 + e)) & 1u))
                    wv = exact_weight(elem<T>(row ? d2 : t2, e), row ? ps.rd : ps.rt);
                // running sums of the exact weights in id order, per row (groups of W lanes)
#pragma unroll
                for (int d = 1; d < W; d <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, wv, d, W);
                    if (e >= d)
                        wv += y;
                }
                const unsigned long long pd = __shfl_sync(0xffffffffu, wv, W + e);
                const unsigned long long at = to_fixed60(rt_e, ps.rt.sf) + wv;
                const i128 cum = RESID ? p2_value(at, to_fixed60(rd_e, ps.rd.sf) + pd, A, B) : (i128)at;
                const unsigned hit = __ballot_sync(0xffffffffu, lane < W && off_s < cum);
                if (lane == 0)
                    *outn = (base + first) * W + (hit ? __ffs(hit) - 1 : W - 1);  // chunk base + first
            }
            return;
        }
        carry += total;
    }
    if (tid == 0)
        *outn = -1;  // unreachable: the range's exact total exceeds rel
}

// Pass 2 of one sequence across its cluster: the inverse-CDF draw with uniform
// u from the weights ps describes, into *outn.  Every CTA sweeps its slice
// (p2_sweep), the CTA totals cross the cluster over DSMEM, and the CTA whose
// slice holds floor(u * R) searches one warp range of it; the rank and the
// warp range are found lane-parallel (one source per lane, a warp scan and a
// ballot) in every warp alike.  A total R of 0 (a
// residual with no mass, unreachable in exact arithmetic, or p without ids
// that hold all of it) samples p instead.  mass_out (rank 0; may be NULL):
// the normalised total (residual mass, or 1 - p(removed ids)).  All threads
// of every CTA of the cluster call it.
template <typename T, bool ALIGNED, bool STAGED, bool ONE_ROW = false, int SLOTS = kP2Slots>
__device__ __noinline__ void pass2_sample(SharedState &sh, const Seq &s, const T *trow, const T *drow,
                                          const uint4 *tst, const uint4 *dst, P2Seq ps, float u, int32_t *outn,
                                          float *mass_out)
{
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    P2SmemT<SLOTS> &sm = *reinterpret_cast<P2SmemT<SLOTS> *>(dyn_smem);
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    unsigned long long A = 0, B = 1;
    i128 R = 0, vsrc = 0, isrc = 0;
    int att = 0;
    bool resid = false;
    for (;; ++att) {
        resid = ps.mode == kP2Residual;
        const RangeSums r = ONE_ROW ? p2_sweep<T, ALIGNED, false, STAGED, true, SLOTS>(s, trow, drow, tst, dst, ps, sm)
                            : resid ? p2_sweep<T, ALIGNED, true, STAGED, false, SLOTS>(s, trow, drow, tst, dst, ps, sm)
                                    : p2_sweep<T, ALIGNED, false, STAGED, false, SLOTS>(s, trow, drow, tst, dst, ps, sm);
        if (lane == 0) {
            sh.p2w[wid][0] = r.jt;
            sh.p2w[wid][1] = r.jd;
            sh.p2w[wid][2] = r.at;
            sh.p2w[wid][3] = r.ad;
        }
        __syncthreads();
        if (tid < 4) {
            unsigned long long v = 0;
            for (int w = 0; w < kWarps; ++w)
                v += sh.p2w[w][tid];
            for (int d = 0; d < s.C; ++d)
                *cluster.map_shared_rank(&sh.p2recv[att][s.rank][tid], d) = v;
        }
        cluster_sync_all();
        // lane k < C of every warp takes source rank k: row totals A, B, the
        // ranks' values and their running sums (identical in every warp)
        const bool src_lane = lane < s.C;
        A = warp_sum_u64(src_lane ? sh.p2recv[att][lane][2] : 0ull);
        B = resid ? warp_sum_u64(src_lane ? sh.p2recv[att][lane][3] : 0ull) : 1ull;
        vsrc = src_lane ? p2_value(sh.p2recv[att][lane][0], resid ? sh.p2recv[att][lane][1] : 0ull, A, B) : (i128)0;
        isrc = warp_scan_i128(vsrc);
        R = shfl_i128(isrc, 31);
        if (R > 0 || att == 1)
            break;
        ps.mode = kP2Full;  // no mass: sample p of the target row
        ps.nz = 0;
        ps.zero_at = -1;
        ps.zero_chunk = -1;
    }
    if (mass_out && s.rank == 0 && tid == 0)
        *mass_out = (float)(resid ? i128_to_double(R) / ((double)A * (double)B) : i128_to_double(R) / (double)A);
    if (R <= 0)
        return;  // nothing to draw from
    const i128 theta = scaled_floor128(u, R);  // the draw: first weight whose running sum passes theta
    // the rank whose slice holds it: the first whose running sum passes theta
    const unsigned hit_src = __ballot_sync(0xffffffffu, lane < s.C && isrc > theta);
    const int owner = hit_src ? __ffs(hit_src) - 1 : s.C - 1;
    if (owner != s.rank)
        return;
    // the warp range inside the slice, the same way over the warps' values
    const i128 rel0 = theta - shfl_i128(isrc - vsrc, owner);
    const i128 vw = lane < kWarps ? p2_value(sh.p2w[lane][0], resid ? sh.p2w[lane][1] : 0ull, A, B) : (i128)0;
    const i128 iw = warp_scan_i128(vw);
    const unsigned hit_w = __ballot_sync(0xffffffffu, lane < kWarps && iw > rel0);
    const int w = hit_w ? __ffs(hit_w) - 1 : kWarps - 1;
    const i128 rel = rel0 - shfl_i128(iw - vw, w);
    int r0, r1;
    warp_range(s, w, r0, r1);
    if (ONE_ROW)
        p2_owner<T, ALIGNED, false, STAGED, true, SLOTS>(sh.p2scan, sh.cnt, sm, s, trow, drow, tst, dst, ps, r0, r1, rel,
                                                         A, B, outn);
    else if (resid)
        p2_owner<T, ALIGNED, true, STAGED, false, SLOTS>(sh.p2scan, sh.cnt, sm, s, trow, drow, tst, dst, ps, r0, r1, rel,
                                                         A, B, outn);
    else
        p2_owner<T, ALIGNED, false, STAGED, false, SLOTS>(sh.p2scan, sh.cnt, sm, s, trow, drow, tst, dst, ps, r0, r1,
                                                          rel, A, B, outn);
}

// Pass-2 weights of a chain sequence whose cut is n (sh.row holds the merged
// statistics of rows t_n and, if n < g, d_n): the residual row after a
// rejection (max(0, p - q), or p without x_n for point-mass drafts), the
// bonus row t_g otherwise.
template <typename T>
__device__ __forceinline__ P2Seq chain_p2seq(const SharedState &sh, const Seq &s, int n)
{
    const int g = s.g;
    const bool rejected = n < g;
    const bool rows = rejected && s.drafts;
    P2Seq ps;
    ps.rt = exact_row(sh.row[n], s.temp);
    ps.rd = rows ? exact_row(sh.row[g + 1 + n], s.temp) : ps.rt;
    ps.mode = !rejected ? kP2Full : rows ? kP2Residual : kP2Zero;
    ps.zero_at = (rejected && !s.drafts) ? sh.drafted[n] : -1;
    ps.zero_chunk = ps.zero_at >= 0 ? ps.zero_at / Elem<T>::W : -1;
    ps.zset = nullptr;
    ps.nz = 0;
    return ps;
}

// Pass 2 of the chain kernels for a sampled, valid sequence whose cut is n,
// across its cluster.  STAGED: tst and dst hold this CTA's slices of rows t_n
// and d_n (early exit with rows in host memory), so pass 2 reads neither row
// again.
template <typename T, bool ALIGNED, bool POINT, bool STAGED = false, int SLOTS = kP2Slots>
__device__ __forceinline__ void chain_pass2(const Params &p, SharedState &sh, const Seq &s, int n,
                                            const uint4 *tst = nullptr, const uint4 *dst = nullptr)
{
    const int g = s.g, b = s.b;
    const bool rows = n < g && s.drafts;
    const P2Seq ps = chain_p2seq<T>(sh, s, n);
    const T *trow = row_ptr<T>(p, s, n);
    const T *drow = rows ? row_ptr<T>(p, s, g + 1 + n) : trow;
    int32_t *outn = p.out_tokens + (size_t)b * (s.gmax + 1) + n;
    float *mass = p.resid_mass ? p.resid_mass + b : nullptr;
    // Rows of one-row calls (gamma_max = 0: the sampler, which the host runs on
    // the point-mass instantiations) are always p and take a pass 2
    // specialised for it, a separate function in those instantiations only, so
    // that the verify kernels' code is unchanged (B = 256, V = 128256 sampler:
    // 53.4 against 56.9 us; folding the specialisation into the shared function
    // cost the verify kernels 1-2 us).
    if (POINT && s.gmax == 0)
        pass2_sample<T, ALIGNED, STAGED, true, SLOTS>(sh, s, trow, drow, tst, tst, ps, final_uniform(p, s), outn,
                                                      mass);
    else
        pass2_sample<T, ALIGNED, STAGED, false, SLOTS>(sh, s, trow, drow, tst, rows ? dst : tst, ps,
                                                       final_uniform(p, s), outn, mass);
}

// ===========================================================================
// Kernel 1: register loads (any alignment; the default)
// ===========================================================================
// KB = 1, 2, 4: the slice gives every thread at most KB chunks of a row, and
// pass 1 reads 8/KB rows per round trip (sweep_rows_batched); KB = 8: at most
// 8 chunks, two rows per round trip with 16 loads in flight per thread, for
// grids that fit in two CTAs per SM (small batches); KB = 0: one row at a time.
template <typename T, bool ALIGNED, bool POINT, int KB>
__global__ void __launch_bounds__(kThreads, KB == 8 ? 2 : 4) spec_verify_stream_kernel(const Params p)
{
    __shared__ SharedState sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const SeqPick pick = seq_for_cluster<POINT>(p, sh, (int)(blockIdx.x / (unsigned)C));
    const int b = pick.b, g = pick.g;
    const float temp = pick.temp;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    const uint32_t bad = check_inputs(p, b, g, temp);
    init_diagnostics(p, b, rank);
    if (bad) {  // uniform over the cluster: every CTA leaves before any barrier
        write_invalid(p, b, rank, bad);
        return;
    }
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store

    const Seq s = make_seq<POINT>(p, C, rank, b, g, temp);
    const int nrows = s.drafts ? 2 * g + 1 : g + 1;
    Gathered gt = wid == 0 ? gather_ids(p, s, lane) : Gathered{-1, 0.0f, 0.0f, 0.0f};

    // ---- pass 1: one streaming sweep of this CTA's slice of every needed row
    if constexpr (KB == 8) {
        sweep_rows_batched<T, ALIGNED, 8, 2 * kUnroll>(p, sh, s, nrows);
    } else if constexpr (KB > 0) {
        sweep_rows_batched<T, ALIGNED, KB>(p, sh, s, nrows);
    } else {
        for (int step = 0; step < nrows; ++step) {
            const int r = row_at_step(step, g, s.drafts);
            const RowStat st = sweep_row<T, ALIGNED>(s, row_ptr<T>(p, s, r));
            if (lane == 0)
                sh.warp_part[r][wid] = st;
        }
    }
    if (wid == 0)
        gather_logits<T>(p, s, lane, gt);
    exchange_rows(sh, s, nrows);
    if (!decide_and_write<T>(p, sh, s, gt))
        return;  // uniform over the cluster; no DSMEM access follows
    chain_pass2<T, ALIGNED, POINT, false, KB == 8 ? kP2SlotsWide : kP2Slots>(p, sh, s, sh.n);
}

// ===========================================================================
// Kernel 3: row-ordered early exit (register loads; variant)
// ===========================================================================
// Positions are verified in order: the rows of position i (t_i, plus d_i for a
// sampled sequence) are streamed, reduced over the cluster and tested before
// any row of position i+1 is read, and the first rejection ends the sweep.  The
// method needs no row after the cut (drafts after a rejection are discarded:
// "Speculative Decoding", ch.2), so a round reads n+1 target rows and
// min(n+1, g) draft rows instead of g+1 and g.  The outputs are those of the
// full sweep; diagnostics exist only for the rows read.
// STAGED (rows in page-locked host memory, read over the host link, where L2
// keeps no copy): each position's slices also go to shared memory, after the
// chunk sums, cap = ceil(num_chunks / C) chunks per row (t_i, then d_i), and
// pass 2 takes the decided rows from there instead of the link.
template <typename T, bool ALIGNED, bool POINT, bool STAGED = false>
__global__ void __launch_bounds__(kThreads, 4) spec_verify_early_kernel(const Params p)
{
    __shared__ SharedState sh;
    extern __shared__ __align__(16) unsigned char early_dyn[];
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const SeqPick pick = seq_for_cluster<POINT>(p, sh, (int)(blockIdx.x / (unsigned)C));
    const int b = pick.b, g = pick.g;
    const float temp = pick.temp;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    const uint32_t bad = check_inputs(p, b, g, temp);
    init_diagnostics(p, b, rank);
    if (bad) {  // uniform over the cluster: every CTA leaves before any barrier
        write_invalid(p, b, rank, bad);
        return;
    }
    if (tid == 0)
        sh.stop = 0;
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store
    const Seq s = make_seq<POINT>(p, C, rank, b, g, temp);
    const int gmax = s.gmax;
    const int cap = (p.num_chunks + C - 1) / C;
    uint4 *stage = STAGED ? reinterpret_cast<uint4 *>(early_dyn + kP2SmemBytes) : nullptr;
    // every drafted id is checked, as in the full sweep (lane-parallel)
    if (wid == 0) {
        const bool tb = lane < g && !(p.tokens[(size_t)b * gmax + lane] >= 0 &&
                                      p.tokens[(size_t)b * gmax + lane] < s.V);
        const unsigned any = __ballot_sync(0xffffffffu, tb);
        if (lane == 0)
            sh.bits = any ? (int)SPEC_STATUS_BAD_TOKEN : 0;
    }

    // Positions in order; each ends with one exchange over the cluster and a
    // decision that every CTA takes identically.  (Streaming position i+1
    // during position i's exchange was measured slower on the B=256 workload:
    // the extra position read per rejection costs more than the barrier.)
    int n = g;
    uint32_t bits = 0;
    for (int i = 0; i <= g; ++i) {
        const int nslot = (s.drafts && i < g) ? 2 : 1;
        // the decision's logits at x_i, loaded ahead of the rows
        const Gathered gt = tid == 0 ? gather_position<T>(p, s, i) : Gathered{-1, 0.0f, 0.0f, 0.0f};
        for (int slot = 0; slot < nslot; ++slot) {
            const T *row = row_ptr<T>(p, s, slot ? g + 1 + i : i);
            // greedy rows need no pass 2: only sampled sequences keep a copy
            const RowStat st = (STAGED && s.sampled)
                                   ? sweep_row<T, ALIGNED, true>(s, row, stage + (size_t)slot * cap)
                                   : sweep_row<T, ALIGNED>(s, row);
            if (lane == 0)
                sh.warp_part[slot][wid] = st;
        }
        __syncthreads();
        if (i == 0)
            cluster_wait();  // every CTA of the cluster is running: DSMEM is addressable
        if (tid < nslot) {
            RowStat v = sh.warp_part[tid][0];
            for (int w = 1; w < kWarps; ++w)
                v = s.sampled ? soft_merge(v, sh.warp_part[tid][w]) : arg_merge(v, sh.warp_part[tid][w]);
            for (int dst = 0; dst < C; ++dst)
                *cluster.map_shared_rank(&sh.recv_pos[i & 1][rank][tid], dst) = v;
        }
        cluster_sync_all();
        if (tid < nslot) {
            RowStat v = sh.recv_pos[i & 1][0][tid];
            for (int src = 1; src < C; ++src)
                v = s.sampled ? soft_merge(v, sh.recv_pos[i & 1][src][tid]) : arg_merge(v, sh.recv_pos[i & 1][src][tid]);
            sh.row[tid ? g + 1 + i : i] = v;
        }
        __syncthreads();
        if (tid == 0) {
            int stop = 0;
            uint32_t bb = (uint32_t)sh.bits;
            if (i < g)
                sh.drafted[i] = gt.x;  // pass 2 reads the rejected id from here (point mode)
            if (bb) {
                stop = 1;  // invalid drafted id
            } else if (i == g) {
                stop = 1;  // every draft accepted: the bonus row was read
                if (s.sampled && !soft_row_ok(sh.row[g]))
                    bb = SPEC_STATUS_BAD_LOGITS;
            } else if (!s.sampled) {
                stop = gt.x != sh.row[i].idx;
            } else {
                const RowStat st = sh.row[i];
                const RowStat sd = s.drafts ? sh.row[g + 1 + i] : st;
                if (!(soft_row_ok(st) && soft_row_ok(sd))) {
                    stop = 1;
                    bb = SPEC_STATUS_BAD_LOGITS;
                } else {
                    const float phat = ex2_approx(fmaf(gt.lt, s.k, -st.m)) / (st.hi + st.lo);
                    const float qhat = s.drafts ? ex2_approx(fmaf(gt.ld, s.k, -sd.m)) / (sd.hi + sd.lo) : 1.0f;
                    stop = !(p.uniforms[(size_t)b * (gmax + 1) + i] * qhat < phat);
                    if (rank == 0) {
                        if (p.p_hat)
                            p.p_hat[(size_t)b * gmax + i] = phat;
                        if (p.q_hat)
                            p.q_hat[(size_t)b * gmax + i] = qhat;
                    }
                }
            }
            sh.stop = stop;
            sh.n = i;
            sh.bits = (int)bb;
        }
        __syncthreads();
        if (sh.stop) {
            n = sh.n;
            bits = (uint32_t)sh.bits;
            break;
        }
    }

    if (rank == 0) {
        int32_t *out = p.out_tokens + (size_t)b * (gmax + 1);
        if (s.sampled && !bits && tid <= n) {
            const RowStat st = sh.row[tid];
            if (p.logz_t)
                p.logz_t[(size_t)b * (gmax + 1) + tid] = (st.m + log2f(st.hi + st.lo)) * kLn2;
            if (tid < g && p.logz_d && s.drafts) {
                const RowStat sd = sh.row[g + 1 + tid];
                p.logz_d[(size_t)b * gmax + tid] = (sd.m + log2f(sd.hi + sd.lo)) * kLn2;
            }
        }
        if (tid <= gmax) {
            int v = -1;
            if (!bits) {
                if (tid < n)
                    v = p.tokens[(size_t)b * gmax + tid];
                else if (tid == n)
                    v = s.sampled ? INT_MIN : sh.row[n].idx;  // sampled: written by pass 2
            }
            if (v != INT_MIN)
                out[tid] = v;
        }
        if (tid == 0) {
            if (p.out_num)
                p.out_num[b] = bits ? 0 : n;
            if (p.seq_status)
                p.seq_status[b] = (int32_t)bits;
            if (bits && p.status)
                atomicOr(p.status, bits);
            if (!bits && (p.counters || p.hist))
                count_round(p.counters, p.hist, g, n);
        }
    }
    if (!s.sampled || bits)
        return;  // uniform over the cluster; no DSMEM access follows
    chain_pass2<T, ALIGNED, POINT, STAGED>(p, sh, s, n, stage, STAGED ? stage + cap : nullptr);
}

// ===========================================================================
// Kernel 4: candidate-tree verification (point-mass candidates)
// ===========================================================================
// A proposer's top candidates per position form a tree that one target
// forward checks ("Speculative Decoding", ch.5: Medusa heads and tree
// attention; "Speculative Decoding으로 LLM 추론 속도 높이기", EAGLE paragraph:
// EAGLE-2 drafts a tree).  Node 0 is the root, node k >= 1 carries candidate
// tokens[b][k] under parent[b][k] < k, and target row k is the next-token
// distribution after the path to k.  The walk starts at the root; at each node
// the CTAs of the cluster sweep that one row (softmax statistics, or the argmax
// at T = 0), merge it over DSMEM and test the children in index order with
// the page's single-candidate rule for a point mass, applied to p without the
// ids already rejected there (R): child c passes iff u_c * (1 - p(R)) < p(x_c)
// ("Speculative Decoding", ch.3).  The first child to pass becomes the next
// node; when none passes, one token is sampled from p without R by the same
// exact inverse CDF as the chain kernels (pass2_sample, with R as a zero set),
// using uniforms[b][0] (the root is never tested).  T = 0 follows the child
// whose id is the argmax, and emits the argmax where none is.  Only the rows
// on the accepted path are read.
template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 4) spec_tree_kernel(const Params p)
{
    __shared__ SharedState sh;
    __shared__ TreeShared tr;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)C);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int N = p.gmax + 1;  // node slots per sequence (<= kThreads)
    const int nn = p.num_draft[b];
    const float temp = p.temperature[b];
    const size_t base = (size_t)b * N;

    // every CTA of the cluster reads the same inputs, so the verdict is uniform
    uint32_t bad = (nn >= 1 && nn <= N) ? 0u : SPEC_STATUS_BAD_NUM_DRAFT;
    if (isnan(temp) || isinf(temp) || temp < 0.0f || (temp > 0.0f && temp < FLT_MIN))
        bad |= SPEC_STATUS_BAD_TEMPERATURE;
    int pk = -1, xk = -1;
    if (!bad && tid < nn) {
        pk = p.parent[base + tid];
        xk = p.tokens[base + tid];
    }
    const bool bad_tree = tid >= 1 && tid < nn && !bad && !(pk >= 0 && pk < tid);
    const bool bad_token = tid >= 1 && tid < nn && !bad && !(xk >= 0 && xk < p.V);
    if (__syncthreads_or(bad_tree))
        bad |= SPEC_STATUS_BAD_TREE;
    if (__syncthreads_or(bad_token))
        bad |= SPEC_STATUS_BAD_TOKEN;
    if (bad) {
        write_invalid(p, b, rank, bad);
        if (rank == 0 && p.out_path && tid < N)
            p.out_path[base + tid] = -1;
        return;
    }
    if (tid < kMaxTree) {
        tr.parent[tid] = tid < nn ? pk : -1;
        tr.token[tid] = tid < nn ? xk : -1;
    }
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store

    Seq s;
    s.b = b;
    s.g = p.gmax;
    s.gmax = p.gmax;
    s.V = p.V;
    s.rank = rank;
    s.C = C;
    s.c0 = (int)((long long)p.num_chunks * rank / C);
    s.c1 = (int)((long long)p.num_chunks * (rank + 1) / C);
    s.sampled = temp > 0.0f;
    s.point = true;
    s.drafts = false;
    s.k = s.sampled ? __fdiv_rn(kLog2e, temp) : 0.0f;
    s.temp = temp;
    s.rowlen = (size_t)p.V;
    __syncthreads();

    int node = 0, n = 0, step = 0;
    uint32_t bits = 0;
    for (;;) {
        // children of the current node, in index order
        const bool is_child = tid >= 1 && tid < nn && tr.parent[tid] == node;
        const unsigned bal = __ballot_sync(0xffffffffu, is_child);
        if (lane == 0)
            tr.wcnt[wid] = __popc(bal);
        __syncthreads();
        int before = 0, m = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            before += w < wid ? tr.wcnt[w] : 0;
            m += tr.wcnt[w];
        }
        if (is_child)
            tr.child[before + __popc(bal & ((1u << lane) - 1u))] = tid;
        __syncthreads();
        // the decision's logits: loaded now, stored after the sweep
        const T *row = row_ptr<T>(p, s, node);
        float gl = 0.0f, uc = 0.0f;
        if (s.sampled && tid < m) {
            const int x = tr.token[tr.child[tid]];
            uc = p.uniforms[base + tr.child[tid]];
            if (sizeof(T) == 2)
                gl = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(row)[x]);
            else
                gl = reinterpret_cast<const float *>(row)[x];
        }
        const RowStat st = sweep_row<T, ALIGNED>(s, row);
        if (lane == 0)
            sh.warp_part[0][wid] = st;
        __syncthreads();
        if (step == 0)
            cluster_wait();  // every CTA of the cluster is running: DSMEM is addressable
        const int par = step & 1;
        if (tid < C) {
            RowStat v = sh.warp_part[0][0];
            for (int w = 1; w < kWarps; ++w)
                v = s.sampled ? soft_merge(v, sh.warp_part[0][w]) : arg_merge(v, sh.warp_part[0][w]);
            *cluster.map_shared_rank(&sh.recv_pos[par][rank][0], tid) = v;
        }
        cluster_sync_all();
        if (tid == 0) {
            RowStat v = sh.recv_pos[par][0][0];
            for (int src = 1; src < C; ++src)
                v = s.sampled ? soft_merge(v, sh.recv_pos[par][src][0]) : arg_merge(v, sh.recv_pos[par][src][0]);
            sh.row[0] = v;
        }
        if (tid < m) {
            tr.glog[tid] = gl;
            tr.uch[tid] = uc;
        }
        __syncthreads();
        if (tid == 0) {
            int next = -1, nrej = 0;
            uint32_t bb = 0;
            const RowStat rs = sh.row[0];
            if (!s.sampled) {
                for (int j = 0; j < m; ++j)
                    if (tr.token[tr.child[j]] == rs.idx) {
                        next = tr.child[j];
                        break;
                    }
            } else if (!soft_row_ok(rs)) {
                bb = SPEC_STATUS_BAD_LOGITS;
            } else {
                const float z = rs.hi + rs.lo;
                float pr = 0.0f;  // p(R): mass of the ids rejected at this node
                for (int j = 0; j < m; ++j) {
                    const int c = tr.child[j], x = tr.token[c];
                    bool dup = false;
                    for (int r = 0; r < nrej; ++r)
                        dup |= tr.rej[r] == x;
                    const float pc = dup ? 0.0f : ex2_approx(fmaf(tr.glog[j], s.k, -rs.m)) / z;
                    if (tr.uch[j] * (1.0f - pr) < pc) {
                        next = c;
                        break;
                    }
                    if (!dup) {
                        pr += pc;
                        tr.rej[nrej++] = x;
                    }
                }
            }
            tr.next = next;
            tr.nrej = nrej;
            tr.bits = (int)bb;
        }
        __syncthreads();
        if (tr.bits) {
            bits = (uint32_t)tr.bits;
            break;
        }
        const int next = tr.next;
        if (next < 0)
            break;
        if (rank == 0 && tid == 0) {
            p.out_tokens[base + n] = tr.token[next];
            if (p.out_path)
                p.out_path[base + n] = next;
        }
        ++n;
        node = next;
        ++step;
    }

    if (bits) {
        write_invalid(p, b, rank, bits);
        if (rank == 0 && p.out_path && tid < N)
            p.out_path[base + tid] = -1;
        return;  // uniform over the cluster; no DSMEM access follows
    }
    if (rank == 0) {
        if (tid > n && tid < N)
            p.out_tokens[base + tid] = -1;
        if (p.out_path && tid >= n && tid < N)
            p.out_path[base + tid] = -1;
        if (tid == 0) {
            if (!s.sampled)
                p.out_tokens[base + n] = sh.row[0].idx;
            p.out_num[b] = n;
            if (p.counters || p.hist)
                count_round(p.counters, p.hist, nn - 1, n);
        }
    }
    if (!s.sampled)
        return;
    P2Seq ps;
    ps.rt = exact_row(sh.row[0], temp);
    ps.rd = ps.rt;
    ps.mode = tr.nrej ? kP2Zero : kP2Full;
    ps.zero_at = -1;
    ps.zero_chunk = -1;
    ps.zset = tr.rej;
    ps.nz = tr.nrej;
    float u = p.uniforms[base];
    if (!(u >= 0.0f))
        u = 0.0f;
    if (u >= 1.0f)
        u = __uint_as_float(0x3F7FFFFFu);
    const T *row = row_ptr<T>(p, s, node);
    pass2_sample<T, ALIGNED, false>(sh, s, row, row, nullptr, nullptr, ps, u, p.out_tokens + base + n, nullptr);
}


// ---------------------------------------------------------------------------
// kernel variants
// ---------------------------------------------------------------------------
enum KernelKind {
    kKindScalarAligned = 0,  // full sweep, register loads, 16-byte aligned rows
    kKindScalar = 1,         // full sweep, register loads, any alignment
    kKindEarlyAligned = 2,   // early exit, 16-byte aligned rows
    kKindEarly = 3,          // early exit, any alignment
    kKindSmall1 = 4,         // full sweep, aligned, at most 1/2/4 chunks per thread and row
    kKindSmall2 = 5,
    kKindSmall4 = 6,
    kKindTreeAligned = 7,    // candidate-tree walk, 16-byte aligned rows
    kKindTree = 8,           // candidate-tree walk, any alignment
    kKindWide8 = 9,          // full sweep, aligned, at most 8 chunks per thread and row, 2 CTAs/SM
    kKindEarlyStaged = 10,   // early exit, aligned, decided rows kept in shared memory (rows in host memory)
    kKinds = 11
};

// The kernel of one variant, as the pointer the launch API takes (nullptr: no
// such variant; the tree walk has no separate point-mass form).
template <typename T, bool POINT> const void *kernel_for_t(int kind)
{
    switch (kind) {
    case kKindScalarAligned:
        return (const void *)spec_verify_stream_kernel<T, true, POINT, 0>;
    case kKindScalar:
        return (const void *)spec_verify_stream_kernel<T, false, POINT, 0>;
    case kKindSmall1:
        return (const void *)spec_verify_stream_kernel<T, true, POINT, 1>;
    case kKindSmall2:
        return (const void *)spec_verify_stream_kernel<T, true, POINT, 2>;
    case kKindSmall4:
        return (const void *)spec_verify_stream_kernel<T, true, POINT, 4>;
    case kKindWide8:
        return (const void *)spec_verify_stream_kernel<T, true, POINT, 8>;
    case kKindTreeAligned:  // candidates are point masses already: one variant
        if constexpr (POINT)
            return nullptr;
        else
            return (const void *)spec_tree_kernel<T, true>;
    case kKindTree:
        if constexpr (POINT)
            return nullptr;
        else
            return (const void *)spec_tree_kernel<T, false>;
    case kKindEarlyAligned:
        return (const void *)spec_verify_early_kernel<T, true, POINT>;
    case kKindEarlyStaged:
        return (const void *)spec_verify_early_kernel<T, true, POINT, true>;
    case kKindEarly:
        return (const void *)spec_verify_early_kernel<T, false, POINT>;
    default:
        return nullptr;
    }
}

}  // namespace

namespace specv {
// Kernel of a KernelKind for each (dtype, proposal form); defined in kernels_*.cu.
const void *kernel_f32(int kind);
const void *kernel_f32_point(int kind);
const void *kernel_bf16(int kind);
const void *kernel_bf16_point(int kind);
}  // namespace specv
