// spec_verify.cu -- speculative-decoding verification round on GB300 (sm_103a).
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
//   * One thread-block cluster of C CTAs per sequence (C in {1,2,4,8,16},
//     chosen from B and V).  CTA c of the cluster owns the contiguous slice
//     [c*NC/C, (c+1)*NC/C) of 16-byte chunks of every row the sequence needs.
//   * Pass 1 streams those slices once with 128-bit loads.  Target and draft
//     rows of sampled sequences (T > 0) keep an online (max, sum of 2^(a-m))
//     per thread, a = logit * log2(e)/T, with m an integer so that rescaling
//     is an exact power of two and the sum compensated; greedy rows (T = 0)
//     keep (max, lowest argmax) of the raw logits.  Partials are reduced over
//     the warp (shuffles), the CTA (shared memory) and the cluster (every CTA
//     pushes its row partials into every other CTA's shared memory, DSMEM).
//   * After one cluster barrier each CTA holds all partials, merges them in
//     rank order (identical bits in every CTA) and takes the accept decision
//     itself: one lane per draft position, a warp ballot gives the first
//     rejection.  No second barrier is needed to broadcast it.
//   * Pass 2 (sampled sequences only) touches the one decided row (target,
//     plus draft when a draft was rejected): weights max(0, p - q) or p as
//     unsigned 64-bit fixed point (2^-60 units), so every sum is exact and
//     order-free.  Slice sums are exchanged over DSMEM; the CTA whose slice
//     holds floor(u*S) scans its chunks and writes the sampled id.
//   No global scratch memory, no atomics on the data path (only the optional
//   status word), no spin waits: the only waits are hardware cluster barriers
//   that every thread of the cluster reaches.

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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 2 * SPEC_MAX_GAMMA + 1;
constexpr int kMaxCluster = 16;
constexpr int kUnroll = 8;  // independent 16-byte loads in flight per thread
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kFixedScale = 1152921504606846976.0f;  // 2^60: pass-2 weight units

struct Params {
    const void *target;
    const void *draft;
    const int32_t *tokens;
    const int32_t *num_draft;
    const float *uniforms;
    const float *temperature;
    int32_t *out_tokens;
    int32_t *out_num;
    uint32_t *status;
    float *p_hat;
    float *q_hat;
    float *logz_t;
    float *logz_d;
    float *resid_mass;
    int32_t *seq_status;
    int B, gmax, V;
    int num_chunks;  // 16-byte chunks per row; the last is partial on the scalar path
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

// Sum over a chunk of 2^(x*k - m), tree order.
template <typename T> __device__ __forceinline__ float chunk_exp_sum(const uint4 &v, float k, float negm)
{
    float e[Elem<T>::W];
#pragma unroll
    for (int i = 0; i < Elem<T>::W; ++i)
        e[i] = ex2_approx(fmaf(elem<T>(v, i), k, negm));
    if (Elem<T>::W == 8)
        return ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    return (e[0] + e[1]) + (e[2] + e[3]);
}

// ---------------------------------------------------------------------------
// per-row statistics and their merges
// ---------------------------------------------------------------------------
// Softmax rows: sum_j 2^(a_j - m) = hi + lo, m integer-valued (or -inf).
// Greedy rows:  (v, i) = largest raw logit and its lowest index.
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

__device__ __forceinline__ bool soft_row_ok(const RowStat &s)
{
    const float z = s.hi + s.lo;
    return isfinite(s.m) && isfinite(z) && z > 0.0f;
}

// Pass-1 sweep of one row slice for a sampled sequence.
template <typename T, bool ALIGNED>
__device__ __forceinline__ RowStat sweep_softmax(const T *row, int c0, int c1, int V, float k)
{
    float m = -INFINITY, hi = 0.0f, lo = 0.0f;
    for (int ch = c0 + (int)threadIdx.x; ch < c1; ch += kUnroll * kThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = ch + u * kThreads;
            v[u] = c < c1 ? load_chunk<T, ALIGNED>(row, c, V) : neg_inf_chunk<T>();
        }
        float bmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            bmax = fmaxf(bmax, chunk_max<T>(v[u]));
        const float amax = bmax * k;
        if (amax > m) {
            const float mn = ceilf(amax);
            const float sc = pow2_int(m - mn);
            hi *= sc;
            lo *= sc;
            m = mn;
        }
        if (m == -INFINITY)
            continue;
        const float negm = -m;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            compensated_add(hi, lo, chunk_exp_sum<T>(v[u], k, negm));
    }
    RowStat s;
    s.m = m;
    s.hi = hi;
    s.lo = lo;
    s.idx = 0;
    return s;
}

// Pass-1 sweep of one row slice for a greedy sequence.
template <typename T, bool ALIGNED>
__device__ __forceinline__ RowStat sweep_argmax(const T *row, int c0, int c1, int V)
{
    float best = -INFINITY;
    int bidx = c0 + (int)threadIdx.x < c1 ? (c0 + (int)threadIdx.x) * Elem<T>::W : INT_MAX;
    for (int ch = c0 + (int)threadIdx.x; ch < c1; ch += kUnroll * kThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = ch + u * kThreads;
            v[u] = c < c1 ? load_chunk<T, ALIGNED>(row, c, V) : neg_inf_chunk<T>();
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float cm = chunk_max<T>(v[u]);
            if (cm > best) {  // chunks arrive in increasing index order: strict > keeps the lowest
                int first = 0;
#pragma unroll
                for (int e = Elem<T>::W - 1; e >= 0; --e)
                    if (elem<T>(v[u], e) == cm)
                        first = e;
                best = cm;
                bidx = (ch + u * kThreads) * Elem<T>::W + first;
            }
        }
    }
    RowStat s;
    s.m = best;
    s.hi = 0.0f;
    s.lo = 0.0f;
    s.idx = bidx;
    return s;
}

// Fixed-point pass-2 weights of one chunk of the decided row.
template <typename T, bool ALIGNED>
__device__ __forceinline__ void chunk_weights(const T *trow, const T *drow, int c, int V, bool residual, float k,
                                              float negmt, float invzt, float negmd, float invzd,
                                              unsigned long long (&w)[Elem<T>::W])
{
    const uint4 tv = load_chunk<T, ALIGNED>(trow, c, V);
    uint4 dv = make_uint4(0, 0, 0, 0);
    if (residual)
        dv = load_chunk<T, ALIGNED>(drow, c, V);
#pragma unroll
    for (int e = 0; e < Elem<T>::W; ++e) {
        float p = ex2_approx(fmaf(elem<T>(tv, e), k, negmt)) * invzt;
        if (residual) {
            const float q = ex2_approx(fmaf(elem<T>(dv, e), k, negmd)) * invzd;
            p = fmaxf(p - q, 0.0f);
        }
        w[e] = __float2ull_rn(p * kFixedScale);
    }
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

struct SharedState {
    RowStat warp_part[kMaxRows][kWarps];
    RowStat recv[kMaxCluster][kMaxRows];  // written remotely by every CTA of the cluster
    RowStat row[kMaxRows];                // merged statistics, identical in every CTA
    unsigned long long recv_sum[2][kMaxCluster];
    unsigned long long warp_sum[kWarps];
    int n;
    int bits;
};

// Block-wide sum of a 64-bit value (exact); every thread gets the total.
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
    for (int w = 0; w < kWarps; ++w)
        t += sh.warp_sum[w];
    return t;
}

// Block-wide inclusive scan of a 64-bit value (exact); also returns the total.
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long &total,
                                                             SharedState &sh)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    __syncthreads();
    if (lane == 31)
        sh.warp_sum[wid] = v;
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

template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) spec_verify_kernel(const Params p)
{
    __shared__ SharedState sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)C);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int gmax = p.gmax, V = p.V;
    const size_t rowlen = (size_t)V;
    int32_t *out = p.out_tokens + (size_t)b * (gmax + 1);

    // ---- inputs of this sequence; every CTA of the cluster decides the same way
    const int g = p.num_draft[b];
    const float temp = p.temperature[b];
    uint32_t bad = 0;
    if (g < 0 || g > gmax)
        bad = SPEC_STATUS_BAD_NUM_DRAFT;
    else {
        if (isnan(temp) || isinf(temp) || temp < 0.0f || (temp > 0.0f && temp < FLT_MIN))
            bad |= SPEC_STATUS_BAD_TEMPERATURE;
        for (int i = 0; i < g; ++i) {
            const int x = p.tokens[(size_t)b * gmax + i];
            if (x < 0 || x >= V)
                bad |= SPEC_STATUS_BAD_TOKEN;
        }
    }
    const bool sampled = temp > 0.0f;

    // diagnostics default to NaN (rank 0 overwrites what it computes)
    if (rank == 0 && tid <= gmax) {
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

    if (bad) {  // uniform over the cluster: every CTA leaves before any barrier
        if (rank == 0) {
            if (tid <= gmax)
                out[tid] = -1;
            if (tid == 0) {
                p.out_num[b] = 0;
                if (p.seq_status)
                    p.seq_status[b] = (int32_t)bad;
                if (p.status)
                    atomicOr(p.status, bad);
            }
        }
        return;
    }

    cluster_arrive_relaxed();  // paired with the wait before the first DSMEM store

    const T *trows = reinterpret_cast<const T *>(p.target) + (size_t)b * (gmax + 1) * rowlen;
    const T *drows = reinterpret_cast<const T *>(p.draft) + (size_t)b * gmax * rowlen;
    const int c0 = (int)((long long)p.num_chunks * rank / C);
    const int c1 = (int)((long long)p.num_chunks * (rank + 1) / C);
    const float k = sampled ? __fdiv_rn(kLog2e, temp) : 0.0f;
    const int nrows = sampled ? 2 * g + 1 : g + 1;

    // ---- pass 1: one streaming sweep of this CTA's slice of every needed row
    for (int r = 0; r < nrows; ++r) {
        const T *row = r <= g ? trows + (size_t)r * rowlen : drows + (size_t)(r - g - 1) * rowlen;
        RowStat s;
        if (sampled) {
            s = sweep_softmax<T, ALIGNED>(row, c0, c1, V, k);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                s = soft_merge(s, shfl_xor_stat(s, o));
        } else {
            s = sweep_argmax<T, ALIGNED>(row, c0, c1, V);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                s = arg_merge(s, shfl_xor_stat(s, o));
        }
        if (lane == 0)
            sh.warp_part[r][wid] = s;
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster is running: DSMEM is addressable
    if (tid < nrows) {
        RowStat s = sh.warp_part[tid][0];
        for (int w = 1; w < kWarps; ++w)
            s = sampled ? soft_merge(s, sh.warp_part[tid][w]) : arg_merge(s, sh.warp_part[tid][w]);
        for (int dst = 0; dst < C; ++dst) {
            RowStat *remote = cluster.map_shared_rank(&sh.recv[rank][tid], dst);
            *remote = s;
        }
    }
    cluster_sync_all();
    if (tid < nrows) {
        RowStat s = sh.recv[0][tid];
        for (int src = 1; src < C; ++src)
            s = sampled ? soft_merge(s, sh.recv[src][tid]) : arg_merge(s, sh.recv[src][tid]);
        sh.row[tid] = s;
    }
    __syncthreads();

    // ---- accept decisions: lane i tests draft position i; a ballot finds the cut
    if (wid == 0) {
        bool ok = false, valid = true;
        float phat = 0.0f, qhat = 0.0f;
        if (lane < g) {
            const int x = p.tokens[(size_t)b * gmax + lane];
            if (!sampled) {
                ok = x == sh.row[lane].idx;
            } else {
                const RowStat st = sh.row[lane], sd = sh.row[g + 1 + lane];
                valid = soft_row_ok(st) && soft_row_ok(sd);
                float lt, ld;
                if (sizeof(T) == 2) {
                    lt = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(trows)[(size_t)lane * rowlen + x]);
                    ld = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(drows)[(size_t)lane * rowlen + x]);
                } else {
                    lt = reinterpret_cast<const float *>(trows)[(size_t)lane * rowlen + x];
                    ld = reinterpret_cast<const float *>(drows)[(size_t)lane * rowlen + x];
                }
                phat = ex2_approx(fmaf(lt, k, -st.m)) / (st.hi + st.lo);
                qhat = ex2_approx(fmaf(ld, k, -sd.m)) / (sd.hi + sd.lo);
                ok = valid && (p.uniforms[(size_t)b * (gmax + 1) + lane] * qhat < phat);
            }
        }
        const unsigned pass = __ballot_sync(0xffffffffu, ok);
        const unsigned fine = __ballot_sync(0xffffffffu, valid);
        const unsigned lanes = g >= 32 ? 0xffffffffu : ((1u << g) - 1u);
        const unsigned fail = ~pass & lanes;
        const int n = fail ? __ffs(fail) - 1 : g;
        uint32_t bits = 0;
        if (sampled) {
            if (n < g ? !((fine >> n) & 1u) : !soft_row_ok(sh.row[g]))
                bits = SPEC_STATUS_BAD_LOGITS;
        }
        if (lane == 0) {
            sh.n = n;
            sh.bits = (int)bits;
        }
        if (rank == 0 && sampled && lane < g) {
            if (p.p_hat)
                p.p_hat[(size_t)b * gmax + lane] = phat;
            if (p.q_hat)
                p.q_hat[(size_t)b * gmax + lane] = qhat;
        }
    }
    __syncthreads();
    const int n = sh.n;
    const uint32_t bits = (uint32_t)sh.bits;

    if (rank == 0) {
        if (sampled && tid <= g && (p.logz_t || p.logz_d)) {
            const RowStat st = sh.row[tid];
            if (p.logz_t)
                p.logz_t[(size_t)b * (gmax + 1) + tid] = (st.m + log2f(st.hi + st.lo)) * kLn2;
            if (tid < g && p.logz_d) {
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
                    v = sampled ? INT_MIN : sh.row[n].idx;  // sampled: written by pass 2
            }
            if (v != INT_MIN)
                out[tid] = v;
        }
        if (tid == 0) {
            p.out_num[b] = bits ? 0 : n;
            if (p.seq_status)
                p.seq_status[b] = (int32_t)bits;
            if (bits && p.status)
                atomicOr(p.status, bits);
        }
    }
    if (!sampled || bits)
        return;  // uniform over the cluster; no DSMEM access follows

    // ---- pass 2: inverse-CDF sample from the decided row
    const bool residual = n < g;
    const RowStat st = sh.row[n];
    const RowStat sd = residual ? sh.row[g + 1 + n] : st;
    const T *trow = trows + (size_t)n * rowlen;
    const T *drow = drows + (size_t)n * rowlen;
    const float invzt = 1.0f / (st.hi + st.lo);
    const float invzd = 1.0f / (sd.hi + sd.lo);
    const float u = p.uniforms[(size_t)b * (gmax + 1) + gmax];
    constexpr int W = Elem<T>::W;

    bool use_residual = residual;
    unsigned long long S = 0, P = 0, mine = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        unsigned long long acc = 0;
        for (int c = c0 + tid; c < c1; c += kThreads) {
            unsigned long long w[W];
            chunk_weights<T, ALIGNED>(trow, drow, c, V, use_residual, k, -st.m, invzt, -sd.m, invzd, w);
#pragma unroll
            for (int e = 0; e < W; ++e)
                acc += w[e];
        }
        mine = block_sum_u64(acc, sh);
        if (tid < C) {
            unsigned long long *remote = cluster.map_shared_rank(&sh.recv_sum[attempt][rank], tid);
            *remote = mine;
        }
        cluster_sync_all();
        S = 0;
        P = 0;
        for (int src = 0; src < C; ++src) {
            const unsigned long long v = sh.recv_sum[attempt][src];
            if (src < rank)
                P += v;
            S += v;
        }
        if (S > 0 || !use_residual)
            break;
        use_residual = false;  // degenerate residual (unreachable in exact arithmetic): sample p_n
    }
    if (rank == 0 && tid == 0 && p.resid_mass)
        p.resid_mass[b] = (float)S * (1.0f / kFixedScale);

    float uu = u;
    if (!(uu >= 0.0f))
        uu = 0.0f;
    if (uu >= 1.0f)
        uu = __uint_as_float(0x3F7FFFFFu);
    const unsigned long long theta = scaled_floor(uu, S);  // pick: C_{j-1} <= theta < C_j
    if (S == 0 || !(P <= theta && theta < P + mine))
        return;  // another CTA owns the sample (S == 0 only for an all-zero bonus row)

    unsigned long long carry = P;
    for (int base = c0; base < c1; base += kThreads) {
        const int c = base + tid;
        unsigned long long w[W];
        unsigned long long sigma = 0;
        if (c < c1) {
            chunk_weights<T, ALIGNED>(trow, drow, c, V, use_residual, k, -st.m, invzt, -sd.m, invzd, w);
#pragma unroll
            for (int e = 0; e < W; ++e)
                sigma += w[e];
        }
        unsigned long long total;
        const unsigned long long incl = block_scan_u64(sigma, total, sh);
        const unsigned long long start = carry + incl - sigma;
        if (c < c1 && start <= theta && theta < start + sigma) {
            unsigned long long run = start;
            int j = c * W + W - 1;
#pragma unroll
            for (int e = 0; e < W; ++e) {
                run += w[e];
                if (theta < run) {
                    j = c * W + e;
                    break;
                }
            }
            out[n] = j;
        }
        carry += total;
        if (theta < carry)
            break;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using KernelFn = void (*)(Params);

KernelFn kernel_for(spec_dtype dt, bool aligned)
{
    if (dt == SPEC_BF16)
        return aligned ? spec_verify_kernel<__nv_bfloat16, true> : spec_verify_kernel<__nv_bfloat16, false>;
    return aligned ? spec_verify_kernel<float, true> : spec_verify_kernel<float, false>;
}

int kernel_slot(spec_dtype dt, bool aligned) { return (dt == SPEC_BF16 ? 2 : 0) + (aligned ? 1 : 0); }

constexpr int kMaxDevices = 64;
// Per-device cache: SM count, and per kernel variant and cluster size whether
// the size is launchable (0 unknown, 1 yes, 2 no).  Idempotent; safe to race.
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_cluster_ok[kMaxDevices][4][5];
std::atomic<int> g_nonportable_set[kMaxDevices][4];

int log2_cluster(int c) { return c == 1 ? 0 : c == 2 ? 1 : c == 4 ? 2 : c == 8 ? 3 : 4; }

spec_status device_sm_count(int dev, int *out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SPEC_ERR_UNSUPPORTED;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ERR_CUDA;
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return SPEC_OK;
}

// Whether clusters of C CTAs of this kernel can be resident on the device.
spec_status cluster_launchable(int dev, spec_dtype dt, bool aligned, int C, bool *ok)
{
    const int slot = kernel_slot(dt, aligned), lc = log2_cluster(C);
    int state = g_cluster_ok[dev][slot][lc].load(std::memory_order_relaxed);
    if (state == 0) {
        KernelFn fn = kernel_for(dt, aligned);
        if (C > 8 && !g_nonportable_set[dev][slot].load(std::memory_order_relaxed)) {
            if (cudaFuncSetAttribute((const void *)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
                cudaGetLastError();
                g_cluster_ok[dev][slot][lc].store(2, std::memory_order_relaxed);
                *ok = false;
                return SPEC_OK;
            }
            g_nonportable_set[dev][slot].store(1, std::memory_order_relaxed);
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)C * 4u);
        cfg.blockDim = dim3(kThreads);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, (const void *)fn, &cfg);
        if (e != cudaSuccess)
            cudaGetLastError();
        state = (e == cudaSuccess && clusters > 0) ? 1 : 2;
        g_cluster_ok[dev][slot][lc].store(state, std::memory_order_relaxed);
    }
    *ok = state == 1;
    return SPEC_OK;
}

int chunk_width(spec_dtype dt) { return dt == SPEC_BF16 ? 8 : 4; }
int elem_size(spec_dtype dt) { return dt == SPEC_BF16 ? 2 : 4; }

// Automatic cluster size: enough CTAs in flight for the streaming sweep (about
// four per SM), but at least kThreads chunks per CTA and row.
int auto_cluster(int B, int num_chunks, int sms)
{
    const long long target = 4LL * sms;
    int C = 1;
    while (C < kMaxCluster && (long long)B * C < target && num_chunks / (C * 2) >= kThreads)
        C *= 2;
    return C;
}

spec_status resolve_shape(int B, int V, spec_dtype dt, bool aligned, int requested, int *C_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    int sms = 0;
    spec_status st = device_sm_count(dev, &sms);
    if (st != SPEC_OK)
        return st;
    const int W = chunk_width(dt);
    const int num_chunks = (V + W - 1) / W;
    int C = requested > 0 ? requested : auto_cluster(B, num_chunks, sms);
    for (;;) {
        bool ok = false;
        st = cluster_launchable(dev, dt, aligned, C, &ok);
        if (st != SPEC_OK)
            return st;
        if (ok)
            break;
        if (requested > 0 || C == 1)
            return SPEC_ERR_UNSUPPORTED;
        C >>= 1;
    }
    *C_out = C;
    return SPEC_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

spec_status run(const void *target, const void *draft, const int32_t *tokens, const int32_t *num_draft,
                const float *uniforms, const float *temperature, int32_t *out_tokens, int32_t *out_num, int B,
                int gmax, int V, spec_dtype dtype, uint32_t *status, void *stream, float *p_hat, float *q_hat,
                float *logz_t, float *logz_d, float *resid_mass, int32_t *seq_status, int cluster_req)
{
    if (dtype != SPEC_F32 && dtype != SPEC_BF16)
        return SPEC_ERR_UNSUPPORTED;
    if (B < 0 || B > SPEC_MAX_BATCH || gmax < 0 || gmax > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_VOCAB)
        return SPEC_ERR_INVALID_ARG;
    if (cluster_req != 0 && cluster_req != 1 && cluster_req != 2 && cluster_req != 4 && cluster_req != 8 &&
        cluster_req != 16)
        return SPEC_ERR_INVALID_ARG;
    if (B == 0)
        return SPEC_OK;
    if (!target || !num_draft || !uniforms || !temperature || !out_tokens || !out_num)
        return SPEC_ERR_INVALID_ARG;
    if (gmax > 0 && (!draft || !tokens))
        return SPEC_ERR_INVALID_ARG;
    const uintptr_t es = (uintptr_t)elem_size(dtype);
    if (((uintptr_t)target % es) || (draft && ((uintptr_t)draft % es)))
        return SPEC_ERR_INVALID_ARG;
    const void *four[] = {tokens, num_draft, uniforms, temperature, out_tokens, out_num, status,
                          p_hat,  q_hat,     logz_t,   logz_d,      resid_mass, seq_status};
    for (const void *q : four)
        if ((uintptr_t)q & 3u)
            return SPEC_ERR_INVALID_ARG;
    const bool aligned = aligned16(target) && (gmax == 0 || aligned16(draft)) &&
                         ((size_t)V * (size_t)es) % 16 == 0;

    int C = 1;
    spec_status st = resolve_shape(B, V, dtype, aligned, cluster_req, &C);
    if (st != SPEC_OK)
        return st;

    Params prm;
    prm.target = target;
    prm.draft = draft ? draft : target;
    prm.tokens = tokens;
    prm.num_draft = num_draft;
    prm.uniforms = uniforms;
    prm.temperature = temperature;
    prm.out_tokens = out_tokens;
    prm.out_num = out_num;
    prm.status = status;
    prm.p_hat = p_hat;
    prm.q_hat = q_hat;
    prm.logz_t = logz_t;
    prm.logz_d = logz_d;
    prm.resid_mass = resid_mass;
    prm.seq_status = seq_status;
    prm.B = B;
    prm.gmax = gmax;
    prm.V = V;
    prm.num_chunks = (V + chunk_width(dtype) - 1) / chunk_width(dtype);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B * (unsigned)C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel_for(dtype, aligned), prm);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
}

}  // namespace

extern "C" {

spec_status spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                        const int32_t *num_draft, const float *uniforms, const float *temperature,
                        int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                        spec_dtype dtype, uint32_t *status, void *stream)
{
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, nullptr, nullptr, nullptr, nullptr,
               nullptr, nullptr, 0);
}

spec_status spec_verify_debug(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                              const int32_t *num_draft, const float *uniforms, const float *temperature,
                              int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                              spec_dtype dtype, uint32_t *status, void *stream, float *p_hat, float *q_hat,
                              float *logz_t, float *logz_d, float *resid_mass, int32_t *seq_status)
{
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, p_hat, q_hat, logz_t, logz_d, resid_mass,
               seq_status, 0);
}

spec_status spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                           const int32_t *num_draft, const float *uniforms, const float *temperature,
                           int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                           spec_dtype dtype, uint32_t *status, void *stream, int cluster_size)
{
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, nullptr, nullptr, nullptr, nullptr,
               nullptr, nullptr, cluster_size);
}

spec_status spec_verify_launch_shape(int B, int gamma_max, int V, spec_dtype dtype, int *cluster_size,
                                     int *num_ctas, int *threads_per_cta)
{
    if (dtype != SPEC_F32 && dtype != SPEC_BF16)
        return SPEC_ERR_UNSUPPORTED;
    if (B < 0 || B > SPEC_MAX_BATCH || gamma_max < 0 || gamma_max > SPEC_MAX_GAMMA || V < 1 ||
        V > SPEC_MAX_VOCAB)
        return SPEC_ERR_INVALID_ARG;
    const bool aligned = ((size_t)V * (size_t)elem_size(dtype)) % 16 == 0;
    int C = 1;
    spec_status st = resolve_shape(B > 0 ? B : 1, V, dtype, aligned, 0, &C);
    if (st != SPEC_OK)
        return st;
    if (cluster_size)
        *cluster_size = C;
    if (num_ctas)
        *num_ctas = B * C;
    if (threads_per_cta)
        *threads_per_cta = kThreads;
    return SPEC_OK;
}

const char *spec_status_string(spec_status s)
{
    switch (s) {
    case SPEC_OK:
        return "ok";
    case SPEC_ERR_INVALID_ARG:
        return "invalid argument";
    case SPEC_ERR_UNSUPPORTED:
        return "unsupported dtype or launch shape";
    case SPEC_ERR_CUDA:
        return "CUDA runtime error";
    }
    return "unknown status";
}

}  // extern "C"
