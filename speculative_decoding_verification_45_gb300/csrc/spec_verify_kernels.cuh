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
//   * Pass 2 (sampled sequences only) touches the one decided row (target,
//     plus draft when a draft was rejected): weights max(0, p - q), p, or p
//     without some ids, as unsigned 64-bit fixed point (2^-60 units), so every
//     sum is exact and order-free.  Slice sums are exchanged over DSMEM; the
//     CTA whose slice holds floor(u*S) scans its chunks and writes the id.
//
// Kernels sharing that protocol:
//   spec_verify_stream_kernel (default) 128-bit loads straight into registers,
//                             32 reducing warps per SM; element loads when rows
//                             are not 16-byte aligned; variants that read
//                             several rows per round trip for narrow slices.
//   spec_verify_early_kernel  positions in order, no row after the first
//                             rejection read; its staged form (rows in
//                             page-locked host memory, which L2 does not
//                             cache) keeps each position's slices in shared
//                             memory so pass 2 reads nothing over the link.
//   spec_tree_kernel          a walk down a tree of candidates, one row per level.
//   spec_verify_ring_kernel   16-byte-aligned rows only.  A producer warp streams
//                             the CTA's slices through an 8-stage shared-memory
//                             ring with cp.async.bulk (the bulk-copy engine)
//                             and mbarriers; eight reducing warps read shared
//                             memory.  On GB300 it is slower here: the ring's
//                             78 KB of shared memory leaves only 16 reducing
//                             warps per SM.  Kept for A/B runs.
// No kernel uses global scratch memory, atomics on the data path (only the
// optional status word and counters) or unbounded waits: mbarrier waits give up
// after a fixed number of tries or 0.2 s and report SPEC_STATUS_TIMEOUT, and
// the only other waits are hardware barriers that every thread reaches.

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

constexpr int kWarps = 8;  // warps that reduce (both kernels)
constexpr int kThreads = kWarps * 32;
constexpr int kTmaThreads = kThreads + 32;  // + one producer warp
constexpr int kMaxRows = 2 * SPEC_MAX_GAMMA + 1;
constexpr int kMaxCluster = 16;
constexpr int kUnroll = 8;       // scalar kernel: 16-byte loads in flight per thread
constexpr int kSegChunks = 512;  // ring kernel: 16-byte chunks per ring stage (8 KB)
constexpr int kChunksPerThread = kSegChunks / kThreads;
constexpr int kStages = 8;  // ring depth: 64 KB
constexpr int kRingBytes = kStages * kSegChunks * 16;
constexpr int kMaxSpin = 1 << 18;  // tries of one mbarrier wait before giving up
constexpr unsigned long long kMaxWaitNs = 200000000ull;  // ... or this much wall time (0.2 s)
constexpr int kMaxScanTiles = 48;  // register kernel: at most 48 * kThreads chunk sums (48 KB) in shared memory
constexpr int kMaxOrdered = 1024;  // longest-first scheduling for B up to this
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kFixedUnit = 8.6736173798840355e-19f;    // 2^-60: pass-2 weight unit (to_fixed60)
constexpr unsigned long long kTimeoutFlag = 1ull << 63;  // carried in exchanged slice sums

static_assert(kSegChunks % kThreads == 0, "a segment must split evenly over the reducing threads");

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
    int scan_tiles;  // register kernel: tiles of kThreads chunk sums kept in shared memory (0 = none)
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
    // add_soft that also leaves each chunk's sum of 2^(a - m) in cs[j * kThreads]
    // (j = j0 + u: the chunk's tile in the slice, for j < tiles), rescaling the
    // entries stored earlier when m rises.  Used for a row that pass 2 samples
    // from as p itself (the sampler), so that its owner needs no second sweep.
    template <typename T, int N>
    __device__ __forceinline__ void add_soft_store(const uint4 (&v)[N], float k, float *cs, int j0, int tiles)
    {
        const float amax = chunks_max<T, N>(v) * k;
        if (amax > m) {
            const float mn = ceilf(amax);
            const float sc = pow2_int(m - mn);
            hi *= sc;
            lo *= sc;
            for (int j = 0; j < j0 && j < tiles; ++j)
                cs[j * kThreads] *= sc;
            m = mn;
        }
        if (m == -INFINITY) {
#pragma unroll
            for (int u = 0; u < N; ++u)
                if (j0 + u < tiles)
                    cs[(j0 + u) * kThreads] = 0.0f;
            return;
        }
        constexpr int P = Elem<T>::W / 2;
        const float2 k2 = make_float2(k, k), nm2 = make_float2(-m, -m);
        float t = 0.0f;
#pragma unroll
        for (int u = 0; u < N; ++u) {
            float2 a = ex2_pair(__ffma2_rn(pair<T>(v[u], 0), k2, nm2));
#pragma unroll
            for (int q = 1; q < P; ++q)
                a = __fadd2_rn(a, ex2_pair(__ffma2_rn(pair<T>(v[u], q), k2, nm2)));
            const float cu = a.x + a.y;
            if (j0 + u < tiles)
                cs[(j0 + u) * kThreads] = cu;
            t += cu;
        }
        compensated_add(hi, lo, t);
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

// floor(w * 2^60) for a finite w in [0, 16), by integer operations only (a
// float-to-64-bit-integer conversion instruction would run on the FP64 pipe).
__device__ __forceinline__ unsigned long long to_fixed60(float w)
{
    const uint32_t bits = __float_as_uint(w);
    const int ex = (int)(bits >> 23);  // w >= 0: no sign bit
    if (ex == 0)
        return 0ull;  // zero or below 2^-126, far under the 2^-60 unit
    const unsigned long long mant = (bits & 0x7FFFFFu) | 0x800000u;
    const int sh = ex - 90;  // w = mant * 2^(ex - 150), so w * 2^60 = mant * 2^(ex - 90)
    if (sh >= 0)
        return mant << sh;
    if (sh <= -24)
        return 0ull;
    return mant >> (-sh);
}

// Pass-2 weights of one chunk of the decided row: max(0, p - q) (residual) or
// p, in float32.  tv/dv: the target and draft chunk.
struct WeightParams {
    float k, negmt, invzt, negmd, invzd;
    bool residual;  // max(0, p - q) with q from the draft row
    int zero_at;    // point-mass residual: p with this id removed (-1: none)
    int zero_chunk; // the chunk holding zero_at (-1: none)
    const int *zset;  // ZSET weights: p with these nz ids removed (a tree node's rejected candidates)
    int nz;
};

template <typename T, bool ZSET = false>
__device__ __forceinline__ void chunk_weights(const uint4 &tv, const uint4 &dv, const WeightParams &wp,
                                              float (&w)[Elem<T>::W], int chunk = -2)
{
    constexpr int P = Elem<T>::W / 2;
    const float2 k2 = make_float2(wp.k, wp.k);
    const float2 nmt = make_float2(wp.negmt, wp.negmt), izt = make_float2(wp.invzt, wp.invzt);
    const float2 nmd = make_float2(wp.negmd, wp.negmd), nizd = make_float2(-wp.invzd, -wp.invzd);
#pragma unroll
    for (int q = 0; q < P; ++q) {
        float2 pq = __fmul2_rn(ex2_pair(__ffma2_rn(pair<T>(tv, q), k2, nmt)), izt);
        if (wp.residual) {
            pq = __ffma2_rn(ex2_pair(__ffma2_rn(pair<T>(dv, q), k2, nmd)), nizd, pq);  // p - q
            pq.x = fmaxf(pq.x, 0.0f);
            pq.y = fmaxf(pq.y, 0.0f);
        }
        w[2 * q] = pq.x;
        w[2 * q + 1] = pq.y;
    }
    if (chunk == wp.zero_chunk) {  // point-mass residual: the rejected id has no weight
#pragma unroll
        for (int e = 0; e < Elem<T>::W; ++e)
            if (chunk * Elem<T>::W + e == wp.zero_at)
                w[e] = 0.0f;
    }
    if constexpr (ZSET) {  // several rejected ids (short list in shared memory)
        const int lo = chunk * Elem<T>::W;
        for (int z = 0; z < wp.nz; ++z) {
            const int id = wp.zset[z];
            if (id >= lo && id < lo + Elem<T>::W) {
#pragma unroll
                for (int e = 0; e < Elem<T>::W; ++e)
                    if (lo + e == id)
                        w[e] = 0.0f;
            }
        }
    }
}

// A chunk's weight: the float32 sum of its elements in a fixed tree order ...
template <typename T> __device__ __forceinline__ float chunk_sum(const float (&w)[Elem<T>::W])
{
    if (Elem<T>::W == 8)
        return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
    return (w[0] + w[1]) + (w[2] + w[3]);
}

// ... on the exact 2^-60 grid, converted once.  Prefix sums of these are exact,
// so every CTA and every pass sees the same cumulative boundaries.
template <typename T> __device__ __forceinline__ unsigned long long chunk_fixed(const float (&w)[Elem<T>::W])
{
    return to_fixed60(chunk_sum<T>(w));
}

template <typename T>
__device__ __forceinline__ unsigned long long chunk_weight_fixed(const uint4 &tv, const uint4 &dv,
                                                                 const WeightParams &wp)
{
    float w[Elem<T>::W];
    chunk_weights<T>(tv, dv, wp, w);
    return chunk_fixed<T>(w);
}

// Inside the chunk whose cumulative interval holds theta (rel = theta - chunk
// start, 0 <= rel < chunk weight): the first element whose running float sum,
// on the 2^-60 grid, passes rel; the last element with weight > 0 if rounding
// leaves none.  An element of weight 0 is never picked.
template <typename T>
__device__ __forceinline__ int pick_in_chunk(const float (&w)[Elem<T>::W], unsigned long long rel)
{
    float run = 0.0f;
    int last = 0;
#pragma unroll
    for (int e = 0; e < Elem<T>::W; ++e) {
        run += w[e];
        if (w[e] > 0.0f) {
            if (rel < to_fixed60(run))
                return e;
            last = e;
        }
    }
    return last;
}

// floor(u * S) exactly, u a float in [0, 1), S a 64-bit integer.
__device__ __forceinline__ unsigned long long scaled_floor(float u, unsigned long long S)
{
    const uint32_t bits = __float_as_uint(u);
    const uint32_t ex = (bits >> 23) & 0xFFu;
    if (ex == 0 && (bits & 0x7FFFFFu) == 0)
        return 0ull;
    const unsigned long long mant = (bits & 0x7FFFFFu) | (ex ? 0x800000u : 0u);
    const int sh = 150 - (int)(ex ? ex : 1u);  // u = mant * 2^-sh, sh >= 24
    const unsigned long long lo = mant * S;
    const unsigned long long hi = __umul64hi(mant, S);
    if (sh >= 128)
        return 0ull;
    if (sh >= 64)
        return hi >> (sh - 64);
    return (lo >> sh) | (hi << (64 - sh));
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
// Barrier of the kThreads reducing threads only (named barrier 1).
__device__ __forceinline__ void reducers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase of the given parity to complete; false after kMaxSpin
// tries or kMaxWaitNs of wall time, whichever comes first (one try may suspend
// the thread for a hardware-defined time, so the tries alone bound the count,
// not the duration).
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const unsigned long long t0 = global_ns();
    for (int i = 0; i < kMaxSpin; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done)
            return true;
        if ((i & 63) == 63 && global_ns() - t0 > kMaxWaitNs)
            break;
    }
    return false;
}
// Bulk copy (bulk-copy engine, no registers involved) of 'bytes' from global
// memory into this CTA's shared memory; completion is signalled on 'bar'.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, unsigned long long *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// ---------------------------------------------------------------------------
// shared state and the per-sequence protocol common to both kernels
// ---------------------------------------------------------------------------
struct SharedState {
    RowStat warp_part[kMaxRows][kWarps];
    RowStat recv[kMaxCluster][kMaxRows];  // written remotely by every CTA of the cluster
    RowStat row[kMaxRows];                // merged statistics, identical in every CTA
    unsigned long long recv_sum[2][kMaxCluster];
    unsigned long long warp_sum[kWarps + 1];
    unsigned long long tile_tot[kMaxScanTiles];
    int hist[kMaxRows + 1];
    int cnt[kWarps];
    int seq;
    int seq_g;
    float seq_temp;
    int bin;
    int rank_in_bin;
    int recv_flag[kMaxCluster];
    RowStat recv_pos[2][kMaxCluster][2];  // early-exit kernel: [position parity][source rank][t / d]
    int n;
    int bits;
    int timeout;
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
    float k;  // log2(e) / T for sampled sequences
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
    if (tid < s.C)
        *cluster.map_shared_rank(&sh.recv_flag[s.rank], tid) = sh.timeout;
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
        int flag = 0;
        for (int c = 0; c < s.C; ++c)
            flag |= sh.recv_flag[c];
        if (flag)
            bits = SPEC_STATUS_TIMEOUT;
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

// Pass-2 weight parameters of decided row n.  residual: the row of a
// rejection, whose weights are max(0, p - q); with point-mass proposals that
// is p with the rejected id xn removed.  Otherwise the weights are p.
__device__ __forceinline__ WeightParams weight_params(const SharedState &sh, const Seq &s, int n, bool residual,
                                                     int xn, int chunk_width)
{
    const RowStat st = sh.row[n];
    const bool rows = residual && s.drafts;
    const RowStat sd = rows ? sh.row[s.g + 1 + n] : st;
    WeightParams wp;
    wp.k = s.k;
    wp.negmt = -st.m;
    wp.invzt = 1.0f / (st.hi + st.lo);
    wp.negmd = -sd.m;
    wp.invzd = 1.0f / (sd.hi + sd.lo);
    wp.residual = rows;
    wp.zero_at = (residual && !s.drafts) ? xn : -1;
    wp.zero_chunk = wp.zero_at >= 0 ? wp.zero_at / chunk_width : -1;
    wp.zset = nullptr;
    wp.nz = 0;
    return wp;
}

// Sends this CTA's slice sum to every CTA of the cluster, then sums what
// arrives: S (total) and P (sum over the lower ranks).  All threads call it.
__device__ __forceinline__ void exchange_slice_sum(SharedState &sh, const Seq &s, int attempt,
                                                   unsigned long long mine, unsigned long long &S,
                                                   unsigned long long &P, bool &timed_out)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    if (tid < s.C)
        *cluster.map_shared_rank(&sh.recv_sum[attempt][s.rank], tid) = mine;
    cluster_sync_all();
    S = 0;
    P = 0;
    timed_out = false;
    for (int src = 0; src < s.C; ++src) {
        const unsigned long long v = sh.recv_sum[attempt][src];
        timed_out |= (v & kTimeoutFlag) != 0;
        if (src < s.rank)
            P += v & ~kTimeoutFlag;
        S += v & ~kTimeoutFlag;
    }
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

// Block-wide sum of a 64-bit value over all NW warps of the CTA (exact); every
// thread gets the total.
template <int NW>
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, SharedState &sh)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        sh.warp_sum[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w)
        t += sh.warp_sum[w];
    return t;
}

// Inclusive scan of a 64-bit value over the kThreads reducing threads (exact);
// also returns their total.  NAMED: the reducing threads are not the whole CTA
// (ring kernel), so they meet at named barrier 1 instead of __syncthreads.
template <bool NAMED>
__device__ __forceinline__ unsigned long long reducers_scan_u64(unsigned long long v, unsigned long long &total,
                                                                SharedState &sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    if (NAMED)
        reducers_sync();
    else
        __syncthreads();
    if (lane == 31)
        sh.warp_sum[wid] = v;
    if (NAMED)
        reducers_sync();
    else
        __syncthreads();
    unsigned long long before = 0, t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w < wid)
            before += sh.warp_sum[w];
        t += sh.warp_sum[w];
    }
    total = t;
    return v + before;
}

// Number of rows sequence i reads: g + 1 target rows, plus g draft rows when
// sampled; 0 for an invalid draft count.
__device__ __forceinline__ int seq_cost(const Params &p, int g, float temp)
{
    if (g < 0 || g > p.gmax)
        return 0;
    return g + 1 + (temp > 0.0f ? g : 0);
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
// All threads of the CTA call it (blockDim.x >= kThreads).
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
        cost[e] = in ? seq_cost(p, gv[e], tv[e]) : -1;
    }
    if (tid <= kMaxRows)
        sh.hist[tid] = 0;
    __syncthreads();
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
// STORE (sampled rows): each chunk's sum also goes to cs[tile * kThreads + tid],
// relative to the warp's merged maximum once the row is done.
// STAGE: every chunk of the slice is also kept in shared memory, stage[c - c0],
// for a pass 2 that must not read the row again (rows in host memory).
template <typename T, bool ALIGNED, bool STORE = false, bool STAGE = false>
__device__ __forceinline__ RowStat sweep_row(const Seq &s, const T *row, float *cs = nullptr,
                                             uint4 *stage = nullptr)
{
    constexpr int W = Elem<T>::W;
    const int tid = threadIdx.x;
    RowAcc acc;
    acc.reset(s.c0 + tid < s.c1 ? (s.c0 + tid) * W : INT_MAX);
    const bool multi = ALIGNED && s.c1 - s.c0 > kUnroll * kThreads;
    const int tiles = (s.c1 - s.c0 + kThreads - 1) / kThreads;
    for (int ch = s.c0 + tid, j0 = 0; ch < s.c1; ch += kUnroll * kThreads, j0 += kUnroll) {
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
        if (STORE && s.sampled)
            acc.add_soft_store<T, kUnroll>(v, s.k, cs + tid, j0, tiles);
        else if (s.sampled)
            acc.add_soft<T, kUnroll>(v, s.k);
        else
            acc.add_arg<T, kUnroll>(v, ch * W, kThreads * W);
    }
    const RowStat w = warp_reduce(acc.stat(), s.sampled);
    if (STORE && s.sampled) {  // this thread's entries, relative to the warp's maximum
        const float sc = pow2_int(acc.m - w.m);
        for (int j = 0; j < tiles; ++j)
            cs[j * kThreads + tid] *= sc;
    }
    return w;
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

// The owner CTA's search for theta inside its slice (rel = theta - P, the
// offset from the slice's start on the exact grid).  With 'keep', chunk_sums
// holds the slice's chunk sums ([tile][lane]); otherwise the slice is scanned
// tile by tile with reloads.  When rounding leaves rel at or beyond the slice's
// own total (only on the bonus path, where the slice mass comes from the pass-1
// partials), the last id of the slice with weight > 0 is taken.  All threads of
// the CTA call it.
template <typename T, bool ALIGNED, bool ZSET = false, bool STAGED = false>
__device__ __forceinline__ void owner_search(const Params &p, SharedState &sh, const Seq &s, const T *trow, const T *drow,
                             const WeightParams &wp, bool keep, const float *chunk_sums, unsigned long long rel,
                             int32_t *outn, const uint4 *tst = nullptr, const uint4 *dst = nullptr)
{
    constexpr int W = Elem<T>::W;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int tiles = (s.c1 - s.c0 + kThreads - 1) / kThreads;
    auto pick_at = [&](int c, unsigned long long r) {
        const uint4 tv = slice_chunk<T, ALIGNED, STAGED>(trow, tst, c, s);
        const uint4 dv = wp.residual ? slice_chunk<T, ALIGNED, STAGED>(drow, dst, c, s) : tv;
        float w[W];
        chunk_weights<T, ZSET>(tv, dv, wp, w, c);
        *outn = c * W + pick_in_chunk<T>(w, r);
    };
    if (keep) {
        for (int j = wid; j < tiles; j += kWarps) {
            unsigned long long t = 0;
            for (int i = lane; i < kThreads; i += 32)
                t += to_fixed60(chunk_sums[j * kThreads + i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                t += __shfl_xor_sync(0xffffffffu, t, o);
            if (lane == 0)
                sh.tile_tot[j] = t;
        }
        __syncthreads();
        unsigned long long before = 0;
        int jt = -1;
        for (int j = 0; j < tiles; ++j) {
            if (rel < before + sh.tile_tot[j]) {
                jt = j;
                break;
            }
            before += sh.tile_tot[j];
        }
        if (jt >= 0) {
            const unsigned long long f = to_fixed60(chunk_sums[jt * kThreads + tid]);
            unsigned long long total;
            const unsigned long long start = before + reducers_scan_u64<false>(f, total, sh) - f;
            if (start <= rel && rel < start + f)
                pick_at(s.c0 + jt * kThreads + tid, rel - start);
            return;
        }
        // rel beyond the slice's chunk total: the last chunk with weight > 0
        int last = -1;
        for (int i = tid; i < tiles * kThreads; i += kThreads)
            if (chunk_sums[i] > 0.0f)
                last = i;
        const int c_last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0)
            sh.cnt[wid] = c_last;
        __syncthreads();
        if (tid == 0) {
            int m = -1;
            for (int w = 0; w < kWarps; ++w)
                m = max(m, sh.cnt[w]);
            if (m >= 0)
                pick_at(s.c0 + m, ~0ull);  // pick_in_chunk returns the last positive element
        }
        return;
    }
    // slice too large for shared memory: tiles in order, reloaded
    unsigned long long carry = 0;
    int last = -1;
    for (int base = s.c0; base < s.c1; base += kThreads) {
        const int c = base + tid;
        float w[W];
        unsigned long long sigma = 0;
        if (c < s.c1) {
            const uint4 tv = slice_chunk<T, ALIGNED, STAGED>(trow, tst, c, s);
            const uint4 dv = wp.residual ? slice_chunk<T, ALIGNED, STAGED>(drow, dst, c, s) : tv;
            chunk_weights<T, ZSET>(tv, dv, wp, w, c);
            sigma = chunk_fixed<T>(w);
            if (chunk_sum<T>(w) > 0.0f)
                last = c;
        }
        unsigned long long total;
        const unsigned long long incl = reducers_scan_u64<false>(sigma, total, sh);
        const unsigned long long start = carry + incl - sigma;
        if (c < s.c1 && start <= rel && rel < start + sigma)
            *outn = c * W + pick_in_chunk<T>(w, rel - start);
        carry += total;
        if (rel < carry)
            return;
    }
    const int c_last = __reduce_max_sync(0xffffffffu, last);
    __syncthreads();
    if (lane == 0)
        sh.cnt[wid] = c_last;
    __syncthreads();
    if (tid == 0) {
        int m = -1;
        for (int w = 0; w < kWarps; ++w)
            m = max(m, sh.cnt[w]);
        if (m >= 0)
            pick_at(m, ~0ull);
    }
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

// Inverse-CDF sample of one decided row across the cluster (pass 2).  The
// weights are wp's: max(0, p - q) with q from drow, p, or p without some ids.
// bonus: the weights are p itself, so CTA c's slice mass is its pass-1 partial
// parts[c * stride] over the row's merged statistics tot, already known to
// every CTA; only the owner reads its slice again and nothing crosses the
// cluster.  Otherwise every CTA sums its slice's weights (pass 2a, chunk sums
// kept in shared memory), the slice sums cross the cluster, and the CTA whose
// slice holds floor(u*S) searches it.  A zero total (unreachable in exact
// arithmetic) samples p instead.  All threads of the CTA call it; the
// cluster's CTAs call it together.  mass_out (rank 0, may be NULL) receives S.
// STAGED: the slices of trow and drow are read from the shared-memory copies
// tst and dst that pass 1 made (sweep_row with STAGE), never from the rows.
template <typename T, bool ALIGNED, bool ZSET, bool STAGED = false>
__device__ __forceinline__ void sample_row(const Params &p, SharedState &sh, const Seq &s, const T *trow,
                                           const T *drow, WeightParams wp, bool bonus, const RowStat &tot,
                                           const RowStat *parts, int stride, float u, int32_t *outn,
                                           float *mass_out, const RowStat *stored = nullptr,
                                           const uint4 *tst = nullptr, const uint4 *dst = nullptr)
{
    constexpr int W = Elem<T>::W;
    const int tid = threadIdx.x;
    const int rank = s.rank;
    extern __shared__ float chunk_sums[];  // [scan_tiles][kThreads]
    const int tiles = (s.c1 - s.c0 + kThreads - 1) / kThreads;
    const bool keep = tiles <= p.scan_tiles;
    constexpr int U2 = kUnroll / 2;
    // chunk c = c0 + j*kThreads + tid is tile j, lane tid; returns the thread's fixed-point total
    auto slice_sums = [&]() {
        unsigned long long acc = 0;
        for (int j0 = 0; j0 < tiles; j0 += U2) {
            uint4 tv[U2], dv[U2];
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int c = s.c0 + (j0 + u) * kThreads + tid;
                tv[u] = c < s.c1 ? slice_chunk<T, ALIGNED, STAGED>(trow, tst, c, s) : neg_inf_chunk<T>();
                dv[u] = (wp.residual && c < s.c1) ? slice_chunk<T, ALIGNED, STAGED>(drow, dst, c, s)
                                                  : neg_inf_chunk<T>();
            }
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int c = s.c0 + (j0 + u) * kThreads + tid;
                float sum = 0.0f;
                if (c < s.c1) {
                    float w[W];
                    chunk_weights<T, ZSET>(tv[u], dv[u], wp, w, c);
                    sum = chunk_sum<T>(w);
                    acc += to_fixed60(sum);
                }
                if (keep && j0 + u < tiles)
                    chunk_sums[(j0 + u) * kThreads + tid] = sum;
            }
        }
        return acc;
    };

    if (bonus) {
        const float z = tot.hi + tot.lo;
        unsigned long long S = 0, P = 0, mine = 0;
        for (int c = 0; c < s.C; ++c) {
            const RowStat part = parts[c * stride];
            const float share = (part.hi + part.lo) * pow2_int(part.m - tot.m) / z;
            const unsigned long long f = to_fixed60(fminf(fmaxf(share, 0.0f), 8.0f));
            if (c < rank)
                P += f;
            if (c == rank)
                mine = f;
            S += f;
        }
        if (rank == 0 && tid == 0 && mass_out)
            *mass_out = (float)S * kFixedUnit;
        const unsigned long long theta = scaled_floor(u, S);
        if (S == 0 || !(P <= theta && theta < P + mine))
            return;  // another CTA owns the sample
        if (keep) {
            if (stored) {  // pass 1 kept the chunk sums: scale them to p
                const float f = pow2_int(stored[threadIdx.x >> 5].m - tot.m) / z;
                for (int j = 0; j < tiles; ++j)
                    chunk_sums[j * kThreads + tid] *= f;
            } else {
                slice_sums();
            }
            __syncthreads();
        }
        owner_search<T, ALIGNED, ZSET, STAGED>(p, sh, s, trow, drow, wp, keep, chunk_sums, theta - P, outn, tst,
                                                 dst);
        return;
    }

    unsigned long long S = 0, P = 0, mine = 0;
    bool timed_out = false;
    bool use_weights = true;
    for (int attempt = 0; attempt < 2; ++attempt) {
        mine = block_sum_u64<kWarps>(slice_sums(), sh);
        exchange_slice_sum(sh, s, attempt, mine, S, P, timed_out);
        if (S > 0 || !use_weights)
            break;
        use_weights = false;  // degenerate residual (unreachable in exact arithmetic): sample p
        wp.residual = false;
        wp.zero_at = -1;
        wp.zero_chunk = -1;
        wp.nz = 0;
    }
    if (rank == 0 && tid == 0 && mass_out)
        *mass_out = (float)S * kFixedUnit;
    const unsigned long long theta = scaled_floor(u, S);  // pick: C_{j-1} <= theta < C_j
    if (S == 0 || !(P <= theta && theta < P + mine))
        return;  // another CTA owns the sample (S == 0 only for an all-zero row)
    owner_search<T, ALIGNED, ZSET, STAGED>(p, sh, s, trow, drow, wp, keep, chunk_sums, theta - P, outn, tst,
                                                 dst);
}

// Pass 2 of the chain kernels for a sampled, valid sequence whose cut is n
// (sh.row holds the merged statistics of rows t_n and, if n < g, d_n; parts
// [c * stride] is CTA c's pass-1 partial of row t_n): the residual row after a
// rejection (max(0, p - q), or p without x_n for point-mass drafts), the bonus
// row t_g otherwise.
// stored: the row's pass-1 warp partials when pass 1 kept its chunk sums (the sampler).
// STAGED: tst and dst hold this CTA's slices of rows t_n and d_n (early exit
// with rows in host memory), so pass 2 reads neither row again.
template <typename T, bool ALIGNED, bool STAGED = false>
__device__ __forceinline__ void stream_pass2(const Params &p, SharedState &sh, const Seq &s, int n, const RowStat *parts,
                             int stride, const RowStat *stored = nullptr, const uint4 *tst = nullptr,
                             const uint4 *dst = nullptr)
{
    constexpr int W = Elem<T>::W;
    const int g = s.g, b = s.b;
    const bool residual = n < g;
    const T *trow = row_ptr<T>(p, s, n);
    const T *drow = (residual && s.drafts) ? row_ptr<T>(p, s, g + 1 + n) : trow;
    const int xn = (residual && !s.drafts) ? sh.drafted[n] : -1;  // point mode only
    const WeightParams wp = weight_params(sh, s, n, residual, xn, W);
    int32_t *outn = p.out_tokens + (size_t)b * (s.gmax + 1) + n;
    sample_row<T, ALIGNED, false, STAGED>(p, sh, s, trow, drow, wp, !residual, sh.row[n], parts, stride,
                                          final_uniform(p, s), outn, p.resid_mass ? p.resid_mass + b : nullptr,
                                          residual ? nullptr : stored, tst,
                                          (residual && s.drafts) ? dst : tst);
}

// ===========================================================================
// Kernel 1: register loads (any alignment; the default)
// ===========================================================================
// KB = 1, 2, 4: the slice gives every thread at most KB chunks of a row, and
// pass 1 reads 8/KB rows per round trip (sweep_rows_batched); KB = 8: at most
// 8 chunks, two rows per round trip with 16 loads in flight per thread, for
// grids that fit in two CTAs per SM (small batches); KB = 16: the sampler (one
// row, gamma_max = 0), whose pass 1 keeps the chunk sums for pass 2; KB = 0:
// one row at a time.
template <typename T, bool ALIGNED, bool POINT, int KB>
__global__ void __launch_bounds__(kThreads, KB == 8 ? 2 : 4) spec_verify_stream_kernel(const Params p)
{
    __shared__ SharedState sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const SeqPick pick = seq_for_cluster(p, sh, (int)(blockIdx.x / (unsigned)C));
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
        sh.timeout = 0;
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store

    const Seq s = make_seq<POINT>(p, C, rank, b, g, temp);
    const int nrows = s.drafts ? 2 * g + 1 : g + 1;
    Gathered gt = wid == 0 ? gather_ids(p, s, lane) : Gathered{-1, 0.0f, 0.0f, 0.0f};

    // ---- pass 1: one streaming sweep of this CTA's slice of every needed row
    bool stored = false;
    if constexpr (KB == 16) {
        extern __shared__ float chunk_sums[];
        stored = (s.c1 - s.c0 + kThreads - 1) / kThreads <= p.scan_tiles;  // room for every tile
        const T *row = row_ptr<T>(p, s, 0);
        const RowStat st = stored ? sweep_row<T, ALIGNED, true>(s, row, chunk_sums) : sweep_row<T, ALIGNED>(s, row);
        if (lane == 0)
            sh.warp_part[0][wid] = st;
    } else if constexpr (KB == 8) {
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
    stream_pass2<T, ALIGNED>(p, sh, s, sh.n, &sh.recv[0][sh.n], kMaxRows, stored ? sh.warp_part[0] : nullptr);
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
    const SeqPick pick = seq_for_cluster(p, sh, (int)(blockIdx.x / (unsigned)C));
    const int b = pick.b, g = pick.g;
    const float temp = pick.temp;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    const uint32_t bad = check_inputs(p, b, g, temp);
    init_diagnostics(p, b, rank);
    if (bad) {  // uniform over the cluster: every CTA leaves before any barrier
        write_invalid(p, b, rank, bad);
        return;
    }
    if (tid == 0) {
        sh.timeout = 0;
        sh.stop = 0;
    }
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store
    const Seq s = make_seq<POINT>(p, C, rank, b, g, temp);
    const int gmax = s.gmax;
    const int cap = (p.num_chunks + C - 1) / C;
    uint4 *stage = STAGED ? reinterpret_cast<uint4 *>(early_dyn + (size_t)p.scan_tiles * kThreads * 4) : nullptr;
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
                                   ? sweep_row<T, ALIGNED, false, true>(s, row, nullptr, stage + (size_t)slot * cap)
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
    stream_pass2<T, ALIGNED, STAGED>(p, sh, s, n, &sh.recv_pos[n & 1][0][0], 2, nullptr, stage,
                                     STAGED ? stage + cap : nullptr);
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
// exact inverse CDF as the chain kernels (sample_row, with R as a zero set),
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
    const RowStat rs = sh.row[0];
    WeightParams wp;
    wp.k = s.k;
    wp.negmt = -rs.m;
    wp.invzt = 1.0f / (rs.hi + rs.lo);
    wp.negmd = 0.0f;
    wp.invzd = 0.0f;
    wp.residual = false;
    wp.zero_at = -1;
    wp.zero_chunk = -1;
    wp.zset = tr.rej;
    wp.nz = tr.nrej;
    float u = p.uniforms[base];
    if (!(u >= 0.0f))
        u = 0.0f;
    if (u >= 1.0f)
        u = __uint_as_float(0x3F7FFFFFu);
    const T *row = row_ptr<T>(p, s, node);
    sample_row<T, ALIGNED, true>(p, sh, s, row, row, wp, tr.nrej == 0, rs, &sh.recv_pos[step & 1][0][0], 2, u,
                                 p.out_tokens + base + n, nullptr);
}

// ===========================================================================
// Kernel 2: bulk-copy ring (16-byte aligned rows; A/B alternative)
// ===========================================================================
// Segment k of a CTA's copy stream lands in ring stage k % kStages; both the
// producer lane and the reducing warps walk the same sequence of segments.
struct RingState {
    uint4 *ring;
    unsigned long long *full;
    unsigned long long *empty;
};

// A CTA that saw one wait run out waits no more (its results are void anyway),
// so a fault costs at most one wait's bound per CTA.
__device__ __forceinline__ bool timed_out_before(const SharedState &sh)
{
    return *reinterpret_cast<const volatile int *>(&sh.timeout) != 0;
}

// Producer: waits until stage k % kStages is free, then starts the copy of
// segment k into it.  Returns false (copy not started) if the wait ran out or
// an earlier one did.
__device__ __forceinline__ bool ring_produce(const RingState &rs, const SharedState &sh, uint32_t k,
                                             const void *src, uint32_t bytes)
{
    const uint32_t st = k % kStages, use = k / kStages;
    if (timed_out_before(sh))
        return false;
    if (use > 0 && !mbar_wait(&rs.empty[st], (use - 1) & 1u))
        return false;
    mbar_arrive_expect_tx(&rs.full[st], bytes);
    bulk_copy_g2s(rs.ring + (size_t)st * kSegChunks, src, bytes, &rs.full[st]);
    return true;
}

// Reducers: wait for segment k, then read this thread's chunks of it.
// 'contiguous' picks chunks tid*N .. tid*N+N-1 (prefix order, pass 2b) instead of
// tid, tid+kThreads, ... (conflict-free, passes 1 and 2a).
template <typename T>
__device__ __forceinline__ void ring_consume(const RingState &rs, SharedState &sh, uint32_t k, int count,
                                             bool contiguous, uint4 (&v)[kChunksPerThread])
{
    const uint32_t st = k % kStages;
    if (!timed_out_before(sh) && !mbar_wait(&rs.full[st], (k / kStages) & 1u))
        sh.timeout = 1;
    const uint4 *seg = rs.ring + (size_t)st * kSegChunks;
    const int tid = threadIdx.x;
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
        const int i = contiguous ? tid * kChunksPerThread + u : tid + u * kThreads;
        v[u] = i < count ? seg[i] : neg_inf_chunk<T>();
    }
    __syncwarp();
    if ((tid & 31) == 0)
        mbar_arrive(&rs.empty[st]);
}

template <typename T>
__global__ void __launch_bounds__(kTmaThreads, 2) spec_verify_ring_kernel(const Params p)
{
    extern __shared__ __align__(128) uint4 ring_mem[];
    __shared__ SharedState sh;
    __shared__ __align__(8) unsigned long long full_bar[kStages];
    __shared__ __align__(8) unsigned long long empty_bar[kStages];
    cg::cluster_group cluster = cg::this_cluster();
    constexpr int W = Elem<T>::W;
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const SeqPick pick = seq_for_cluster(p, sh, (int)(blockIdx.x / (unsigned)C));
    const int b = pick.b, g = pick.g;
    const float temp = pick.temp;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const bool producer = wid == kWarps;

    const uint32_t bad = check_inputs(p, b, g, temp);
    init_diagnostics(p, b, rank);
    if (bad) {  // uniform over the cluster: every CTA leaves before any barrier
        write_invalid(p, b, rank, bad);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kWarps);
        }
        sh.timeout = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store

    const Seq s = make_seq<false>(p, C, rank, b, g, temp);
    const int nrows = s.sampled ? 2 * g + 1 : g + 1;
    const int slice = s.c1 - s.c0;
    const int nseg = (slice + kSegChunks - 1) / kSegChunks;  // segments per row slice
    const RingState rs{ring_mem, full_bar, empty_bar};
    uint32_t k = 0;  // segment counter, identical on both sides
    const Gathered gt = wid == 0 ? gather_position<T>(p, s, lane) : Gathered{-1, 0.0f, 0.0f, 0.0f};

    // ---- pass 1: every needed row slice in one continuous copy stream
    if (producer) {
        if (lane == 0) {
            for (int step = 0; step < nrows; ++step) {
                const T *row = row_ptr<T>(p, s, row_at_step(step, g, s.sampled));
                for (int j = 0; j < nseg; ++j) {
                    const int start = s.c0 + j * kSegChunks;
                    const int cnt = min(kSegChunks, s.c1 - start);
                    if (!ring_produce(rs, sh, k + (uint32_t)(step * nseg + j), row + (size_t)start * W,
                                      (uint32_t)cnt * 16u))
                        sh.timeout = 1;
                }
            }
        }
        __syncwarp();
        k = (uint32_t)(nrows * nseg);
    } else {
        for (int step = 0; step < nrows; ++step) {
            const int r = row_at_step(step, g, s.sampled);
            RowAcc acc;
            acc.reset(tid < min(kSegChunks, slice) ? (s.c0 + tid) * W : INT_MAX);
            for (int j = 0; j < nseg; ++j) {
                const int start = s.c0 + j * kSegChunks;
                const int cnt = min(kSegChunks, s.c1 - start);
                uint4 v[kChunksPerThread];
                ring_consume<T>(rs, sh, k++, cnt, false, v);
                if (s.sampled) {
                    acc.add_soft<T, kChunksPerThread>(v, s.k);
                } else {
                    acc.add_arg<T, kChunksPerThread>(v, (start + tid) * W, kThreads * W);
                }
            }
            const RowStat st = warp_reduce(acc.stat(), s.sampled);
            if (lane == 0)
                sh.warp_part[r][wid] = st;
        }
    }
    exchange_rows(sh, s, nrows);
    if (!decide_and_write<T>(p, sh, s, gt))
        return;  // uniform over the cluster; every copy issued so far has been consumed

    // ---- pass 2a: slice sums of the decided row's weights (streamed again)
    const int n = sh.n;
    bool use_residual = n < g;
    const T *trow = row_ptr<T>(p, s, n);
    const T *drow = n < g ? row_ptr<T>(p, s, g + 1 + n) : trow;
    WeightParams wp = weight_params(sh, s, n, use_residual, -1, W);
    unsigned long long S = 0, P = 0, mine = 0;
    bool timed_out = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const uint32_t per = use_residual ? 2u : 1u;
        unsigned long long acc = 0;
        if (producer) {
            if (lane == 0) {
                for (int j = 0; j < nseg; ++j) {
                    const int start = s.c0 + j * kSegChunks;
                    const uint32_t bytes = (uint32_t)min(kSegChunks, s.c1 - start) * 16u;
                    if (!ring_produce(rs, sh, k + per * j, trow + (size_t)start * W, bytes))
                        sh.timeout = 1;
                    if (use_residual && !ring_produce(rs, sh, k + per * j + 1, drow + (size_t)start * W, bytes))
                        sh.timeout = 1;
                }
            }
            __syncwarp();
        } else {
            for (int j = 0; j < nseg; ++j) {
                const int start = s.c0 + j * kSegChunks;
                const int cnt = min(kSegChunks, s.c1 - start);
                uint4 tv[kChunksPerThread], dv[kChunksPerThread];
                ring_consume<T>(rs, sh, k + per * j, cnt, false, tv);
                if (use_residual)
                    ring_consume<T>(rs, sh, k + per * j + 1, cnt, false, dv);
#pragma unroll
                for (int u = 0; u < kChunksPerThread; ++u)
                    if (tid + u * kThreads < cnt)
                        acc += chunk_weight_fixed<T>(tv[u], use_residual ? dv[u] : tv[u], wp);
            }
        }
        k += per * (uint32_t)nseg;
        mine = block_sum_u64<kWarps + 1>(acc, sh);
        if (sh.timeout)
            mine |= kTimeoutFlag;
        exchange_slice_sum(sh, s, attempt, mine, S, P, timed_out);
        mine &= ~kTimeoutFlag;
        if (timed_out || S > 0 || !use_residual)
            break;
        use_residual = false;  // degenerate residual (unreachable in exact arithmetic): sample p_n
        wp = weight_params(sh, s, n, false, -1, W);
    }
    if (rank == 0 && tid == 0 && p.resid_mass)
        p.resid_mass[b] = (float)S * kFixedUnit;
    if (timed_out) {
        if (rank == 0) {
            if (tid <= s.gmax)
                p.out_tokens[(size_t)b * (s.gmax + 1) + tid] = -1;
            if (tid == 0) {
                if (p.out_num)
                    p.out_num[b] = 0;
                if (p.seq_status)
                    p.seq_status[b] = SPEC_STATUS_TIMEOUT;
                if (p.status)
                    atomicOr(p.status, SPEC_STATUS_TIMEOUT);
            }
        }
        return;
    }

    // ---- pass 2b: the CTA whose slice holds floor(u*S) finds the id
    const unsigned long long theta = scaled_floor(final_uniform(p, s), S);  // pick: C_{j-1} <= theta < C_j
    if (S == 0 || !(P <= theta && theta < P + mine))
        return;  // another CTA owns the sample (S == 0 only for an all-zero bonus row)
    const uint32_t per = use_residual ? 2u : 1u;
    if (producer) {
        if (lane == 0) {
            for (int j = 0; j < nseg; ++j) {
                const int start = s.c0 + j * kSegChunks;
                const uint32_t bytes = (uint32_t)min(kSegChunks, s.c1 - start) * 16u;
                if (!ring_produce(rs, sh, k + per * j, trow + (size_t)start * W, bytes))
                    sh.timeout = 1;
                if (use_residual && !ring_produce(rs, sh, k + per * j + 1, drow + (size_t)start * W, bytes))
                    sh.timeout = 1;
            }
        }
        __syncwarp();
        return;
    }
    unsigned long long carry = P;
    for (int j = 0; j < nseg; ++j) {
        const int start = s.c0 + j * kSegChunks;
        const int cnt = min(kSegChunks, s.c1 - start);
        uint4 tv[kChunksPerThread], dv[kChunksPerThread];
        ring_consume<T>(rs, sh, k + per * j, cnt, true, tv);
        if (use_residual)
            ring_consume<T>(rs, sh, k + per * j + 1, cnt, true, dv);
        if (theta < carry)
            continue;  // found in an earlier segment: drain the stream only (uniform)
        unsigned long long sig[kChunksPerThread];
        unsigned long long L = 0;
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            const int i = tid * kChunksPerThread + u;
            sig[u] = i < cnt ? chunk_weight_fixed<T>(tv[u], use_residual ? dv[u] : tv[u], wp) : 0ull;
            L += sig[u];
        }
        unsigned long long total;
        const unsigned long long incl = reducers_scan_u64<true>(L, total, sh);
        unsigned long long start_u = carry + incl - L;
        if (start_u <= theta && theta < start_u + L) {
#pragma unroll
            for (int u = 0; u < kChunksPerThread; ++u) {
                if (start_u <= theta && theta < start_u + sig[u]) {
                    float w[W];
                    chunk_weights<T>(tv[u], use_residual ? dv[u] : tv[u], wp, w);
                    const int c = start + tid * kChunksPerThread + u;
                    p.out_tokens[(size_t)b * (s.gmax + 1) + n] = c * W + pick_in_chunk<T>(w, theta - start_u);
                }
                start_u += sig[u];
            }
        }
        carry += total;
    }
    reducers_sync();
    if (sh.timeout && tid == 0) {
        p.out_tokens[(size_t)b * (s.gmax + 1) + n] = -1;
        if (p.status)
            atomicOr(p.status, SPEC_STATUS_TIMEOUT);
    }
}

// ---------------------------------------------------------------------------
// kernel variants
// ---------------------------------------------------------------------------
enum KernelKind {
    kKindRing = 0,
    kKindScalarAligned = 1,  // full sweep, register loads, 16-byte aligned rows
    kKindScalar = 2,         // full sweep, register loads, any alignment
    kKindEarlyAligned = 3,   // early exit, 16-byte aligned rows
    kKindEarly = 4,          // early exit, any alignment
    kKindSmall1 = 5,         // full sweep, aligned, at most 1/2/4 chunks per thread and row
    kKindSmall2 = 6,
    kKindSmall4 = 7,
    kKindTreeAligned = 8,    // candidate-tree walk, 16-byte aligned rows
    kKindTree = 9,           // candidate-tree walk, any alignment
    kKindWide8 = 10,         // full sweep, aligned, at most 8 chunks per thread and row, 2 CTAs/SM
    kKindSample = 11,        // the sampler (gamma_max = 0), aligned: pass 1 keeps the chunk sums
    kKindEarlyStaged = 12,   // early exit, aligned, decided rows kept in shared memory (rows in host memory)
    kKinds = 13
};

// The kernel of one variant, as the pointer the launch API takes (nullptr: no
// such variant; the ring kernel has no point-mass form).
template <typename T, bool POINT> const void *kernel_for_t(int kind)
{
    switch (kind) {
    case kKindRing:
        if constexpr (POINT)
            return nullptr;
        else
            return (const void *)spec_verify_ring_kernel<T>;
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
    case kKindSample:
        if constexpr (POINT)
            return nullptr;
        else
            return (const void *)spec_verify_stream_kernel<T, true, false, 16>;
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
    default:
        return (const void *)spec_verify_early_kernel<T, false, POINT>;
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
