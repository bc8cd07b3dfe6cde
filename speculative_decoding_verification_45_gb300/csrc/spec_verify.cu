// spec_verify.cu -- host side of libspec_verify (GB300, sm_103a).
//
// Argument checks, the launch shape (cluster size and kernel variant per call,
// from B, V, the alignment and the device's SM count), the C entry points of
// include/spec_verify.h, and the prompt-lookup kernel.  The verification
// kernels and their design notes are in spec_verify_kernels.cuh; the
// operation is specified in include/spec_verify.h.

#include "spec_verify_kernels.cuh"

#include <nvtx3/nvToolsExt.h>

namespace {

// ===========================================================================
// Prompt-lookup (n-gram) proposer
// ===========================================================================
// Drafts without a model ("Speculative Decoding", ch.5: find the current suffix
// earlier in the context and propose what followed it; prompt_lookup_min/max
// in the vLLM section of "Speculative Decoding으로 LLM 추론 속도 높이기").  For
// every candidate end e in [1, L-1] the kernel measures l(e), the length of the
// longest common suffix of context[0, e) and context[0, L), capped at max_n;
// the proposal follows the end with the largest l(e) >= min_n, the latest such
// end on ties.  That is the same as trying n from max_n down to min_n and
// taking the most recent occurrence of the n-gram (an occurrence of length n
// ends at e exactly when l(e) >= n).  One CTA per sequence.
constexpr int kMaxNgram = 64;
constexpr int kNgramThreads = 256;
constexpr int kNgramTile = 8192;  // context tokens staged in shared memory per step (32 KB)

// The context is staged in shared memory a tile at a time (coalesced loads,
// plus max_n tokens of halo before the tile), so every comparison reads
// shared memory instead of a chain of dependent global loads.
__global__ void __launch_bounds__(kNgramThreads)
    spec_ngram_kernel(const int32_t *context, long long stride, const int32_t *context_len, int min_n, int max_n,
                      int gmax, int32_t *out_tokens, int32_t *out_num)
{
    __shared__ int tile[kMaxNgram + kNgramTile];  // context[t0 - kMaxNgram, t0 + kNgramTile)
    __shared__ int suffix[kMaxNgram];             // suffix[t] = context[L - 1 - t]
    __shared__ unsigned long long best_warp[kNgramThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int32_t *ctx = context + (size_t)b * (size_t)stride;
    int L = context_len[b];
    L = L < 0 ? 0 : (L > stride ? (int)stride : L);
    if (tid < max_n && tid < L)
        suffix[tid] = ctx[L - 1 - tid];
    // (l << 32) | e, larger is better; 0 = no candidate
    unsigned long long best = 0;
    for (int t0 = 0; t0 < L - 1; t0 += kNgramTile) {  // candidate ends e in [t0 + 1, t0 + kNgramTile]
        __syncthreads();  // the previous tile's readers are done (and suffix is written)
        for (int i = tid; i < kMaxNgram + kNgramTile; i += kNgramThreads) {
            const int pos = t0 - kMaxNgram + i;
            tile[i] = (pos >= 0 && pos < L) ? ctx[pos] : -1;
        }
        __syncthreads();
        const int e_hi = min(t0 + kNgramTile, L - 1);
        const int *at = tile + kMaxNgram - t0 - 1;  // at[e - l] = context[e - 1 - l]
        for (int e = t0 + 1 + tid; e <= e_hi; e += kNgramThreads) {
            int l = 0;
            while (l < max_n && l < e && at[e - l] == suffix[l])
                ++l;
            if (l >= min_n) {
                const unsigned long long key = ((unsigned long long)l << 32) | (unsigned)e;
                best = key > best ? key : best;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
        best = y > best ? y : best;
    }
    if (lane == 0)
        best_warp[wid] = best;
    __syncthreads();
    if (wid == 0) {
        unsigned long long v = lane < kNgramThreads / 32 ? best_warp[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, v, o);
            v = y > v ? y : v;
        }
        const int e = (int)(v & 0xffffffffu);
        const int k = v ? min(gmax, L - e) : 0;
        if (lane < gmax)
            out_tokens[(size_t)b * gmax + lane] = lane < k ? ctx[e + lane] : -1;
        if (lane == 0)
            out_num[b] = k;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// point: point-mass proposals.
const void *kernel_for(spec_dtype dt, int kind, bool point)
{
    if (dt == SPEC_BF16)
        return point ? specv::kernel_bf16_point(kind) : specv::kernel_bf16(kind);
    return point ? specv::kernel_f32_point(kind) : specv::kernel_f32(kind);
}

// Dynamic shared memory of the staged early-exit kernel at most: pass 2's
// staging area and its copies of the decided rows' slices (one CTA per SM).
constexpr int kStagedDynMax = 200 * 1024;
// Largest dynamic shared memory a kernel kind is launched with: the staged
// early exit, or pass 2's staging area and queue.
int kernel_dyn_smem(int kind)
{
    return kind == kKindEarlyStaged ? kStagedDynMax : kind == kKindWide8 ? kP2SmemBytesWide : kP2SmemBytes;
}
int variant_slot(spec_dtype dt, int kind, bool point)
{
    return ((dt == SPEC_BF16 ? 2 : 0) + (point ? 1 : 0)) * kKinds + kind;
}
int chunk_width(spec_dtype dt) { return dt == SPEC_BF16 ? 8 : 4; }
int elem_size(spec_dtype dt) { return dt == SPEC_BF16 ? 2 : 4; }

constexpr int kMaxDevices = 64;
// Per-device caches (idempotent, safe to race): SM count; whether the kernel
// attributes were applied; per variant and cluster size whether the size can be
// resident (0 unknown, 1 yes, 2 no).
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_attrs[kMaxDevices][4 * kKinds];
std::atomic<int> g_cluster_ok[kMaxDevices][4 * kKinds][kMaxCluster];

spec_status current_device(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    if (*dev < 0 || *dev >= kMaxDevices)
        return SPEC_ERR_UNSUPPORTED;
    return SPEC_OK;
}

spec_status device_sm_count(int dev, int *out)
{
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return SPEC_ERR_CUDA;
        }
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return SPEC_OK;
}

// Applies the kernel attributes once per device: dynamic shared memory above
// the 48 KB default (staged early exit) and clusters of 16 CTAs.
bool prepare_kernel(int dev, spec_dtype dt, int kind, bool point)
{
    const int slot = variant_slot(dt, kind, point);
    int st = g_attrs[dev][slot].load(std::memory_order_relaxed);
    if (st == 0) {
        const void *fn = kernel_for(dt, kind, point);
        bool ok = fn && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        if (ok && kernel_dyn_smem(kind) > 0)
            ok = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kernel_dyn_smem(kind)) ==
                 cudaSuccess;
        if (!ok)
            cudaGetLastError();
        st = ok ? 1 : 2;
        g_attrs[dev][slot].store(st, std::memory_order_relaxed);
    }
    return st == 1;
}

cudaLaunchConfig_t launch_config(unsigned grid, int C, size_t dyn_smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Whether clusters of C CTAs of this variant can be resident on the device.
bool cluster_launchable(int dev, spec_dtype dt, int kind, int C, bool point)
{
    const int slot = variant_slot(dt, kind, point), lc = C - 1;
    int state = g_cluster_ok[dev][slot][lc].load(std::memory_order_relaxed);
    if (state == 0) {
        state = 2;
        if (prepare_kernel(dev, dt, kind, point)) {
            cudaLaunchAttribute attr[1];
            cudaLaunchConfig_t cfg = launch_config((unsigned)C * 4u, C, (size_t)kernel_dyn_smem(kind), 0, attr);
            int clusters = 0;
            const cudaError_t e =
                cudaOccupancyMaxActiveClusters(&clusters, kernel_for(dt, kind, point), &cfg);
            if (e != cudaSuccess)
                cudaGetLastError();
            state = (e == cudaSuccess && clusters > 0) ? 1 : 2;
        }
        g_cluster_ok[dev][slot][lc].store(state, std::memory_order_relaxed);
    }
    return state == 1;
}

// Automatic cluster size.  First the smallest power of two giving about six
// CTAs per SM in the grid, at most 8 (16 for one or two sequences with long
// rows, lone_cap) and at least
// kThreads/2 chunks per CTA and row.  A thread reads its chunks of a row in
// batches of kUnroll loads, and on GB300 the sweep time follows the number of
// batches, not the bytes in the last one: when the slice leaves a second batch
// less than half full (9 to 12 chunks per thread), the smallest cluster that
// fits every row in one batch is taken instead, up to 16 CTAs, if the grid stays
// within about one wave of resident CTAs (four per SM).  Measured on GB300:
// B=256, V=128256 is best at 4; B=32 at 8; B=64, V=151936 at 10 (42 us
// against 57 us at 8).
int per_thread_chunks(int num_chunks, int C) { return ((num_chunks + C - 1) / C + kThreads - 1) / kThreads; }

// One or two sequences with long rows (at least 512 chunks per CTA at 16) take
// clusters of up to 16: B = 1, V = 128256 (config 3's rows): 22.5 us at 16
// against 23.6 at 8; V = 151936: 12.7 against 17.6.  Shorter rows stop at 8,
// where the cluster's barriers and exchanges cost more than the smaller
// slices save: B = 1, V = 32000 (config 2): 25.6 us at 8 against 27.9 at 16
// (graph replay, 10-call graphs).
int lone_cap(int B, int num_chunks) { return (B <= 2 && num_chunks >= 16 * 512) ? 16 : 8; }

int auto_cluster(int B, int num_chunks, int sms)
{
    const long long target = 6LL * sms;
    const int cap = lone_cap(B, num_chunks);
    int C = 1;
    while (C < cap && (long long)B * C < target && num_chunks / (C * 2) >= kThreads / 2)
        C *= 2;
    const int pt = per_thread_chunks(num_chunks, C);
    if (pt > kUnroll && pt <= kUnroll + kUnroll / 2) {
        for (int c = C + 1; c <= kMaxCluster; ++c) {
            if ((long long)B * c * 10 > 44LL * sms)  // more than 1.1 waves of 4 CTAs per SM
                break;
            if (per_thread_chunks(num_chunks, c) <= kUnroll)
                return c;
        }
    }
    return C;
}

// Automatic cluster size for one row per sequence (gamma_max = 0: the
// sampler).  Every cluster then does the same work, and a few long CTAs that
// are all resident at once beat a grid of several waves for the streaming:
// the largest power of two with B*C <= 2 * SMs (at most 8; 16 for one or two
// long rows, lone_cap).  But the final draw's exact weights (pass 2) cost several times the
// streaming's ALU work per byte and run on the row's own CTAs, so a long row
// (at least 4096 chunks) is split over at least 4 CTAs.  Measured on GB300,
// 10-call graphs, V = 128256 bf16, half the rows at T = 1: B = 256 takes
// 119 us at 1 CTA per row, 101 at 2, 69 at 4, 82 at 8; B = 64 and 32 are best
// at the first rule's 4 and 8.
int sampler_cluster(int B, int num_chunks, int sms)
{
    const int cap = lone_cap(B, num_chunks);
    int C = 1;
    while (C < cap && (long long)B * C * 2 <= 2LL * sms)
        C *= 2;
    if (num_chunks >= 4096 && C < 4)
        C = 4;
    return C;
}

// Whether the automatic choice is the row-ordered early exit: when the full
// sweep's grid would fill more than half of the resident slots (many
// sequences: reading only the rows up to each cut saves bandwidth and the
// final draws start earlier), or for tiny rows (at most 512 chunks: one
// round trip per position either way).  Measured on GB300, 10-call graphs:
// B = 256, V = 128256 (half greedy): 122 us early exit against 150 us full
// sweep; B = 64, V = 151936: 69 against 71; B = 32 (every sequence sampled):
// 51 against 45; B = 1, V = 32000: 45 against 33; B = 1, V = 1024: 18
// against 23.
bool auto_early_exit(int B, int num_chunks, int sms)
{
    return num_chunks <= 512 || (long long)B * auto_cluster(B, num_chunks, sms) > 2LL * sms;
}

// Automatic cluster size of a candidate-tree walk.  Each level of the walk is
// one row read and one cluster exchange, so a walk is latency-bound, and a grid
// resident in one wave (at most 4 CTAs per SM) beats a second wave as long as
// each tree keeps at least 4 CTAs: the chain rule's size, halved while that
// holds.  Measured on GB300, 20-call graphs, V = 128256: 128 trees of 16 or 32
// nodes take 34.9 / 41.2 us at 8 and 30.3 / 32.9 us at 4; 256 trees stay at 4
// (49.5 us, against 52.1 at 2); 8 to 64 trees stay at 8.
int tree_cluster(int B, int num_chunks, int sms)
{
    int C = auto_cluster(B, num_chunks, sms);
    while ((long long)B * C > 4LL * sms && C / 2 >= 4)
        C /= 2;
    return C;
}

struct Shape {
    int kind;
    int C;
    int sms;  // the device's SM count
};


// Picks the kernel and cluster size.  want_kind: -1 automatic, else a KernelKind.
// point: point-mass proposals.
spec_status resolve_shape(int B, int V, spec_dtype dt, bool aligned, int want_kind, int want_C, Shape *out,
                          bool point = false, bool one_row = false)
{
    int dev = 0, sms = 0;
    spec_status st = current_device(&dev);
    if (st != SPEC_OK)
        return st;
    st = device_sm_count(dev, &sms);
    if (st != SPEC_OK)
        return st;
    int kinds[1];
    int nk = 0;
    if (want_kind >= 0) {
        if (!aligned && (want_kind == kKindScalarAligned || want_kind == kKindEarlyAligned))
            return SPEC_ERR_UNSUPPORTED;
        kinds[nk++] = want_kind;
    } else {
        kinds[nk++] = aligned ? kKindScalarAligned : kKindScalar;
    }
    const int W = chunk_width(dt);
    const int num_chunks = (V + W - 1) / W;
    for (int i = 0; i < nk; ++i) {
        const bool walk = kinds[i] == kKindTreeAligned || kinds[i] == kKindTree;
        int C = want_C > 0 ? want_C
                : walk     ? tree_cluster(B, num_chunks, sms)
                : one_row  ? sampler_cluster(B, num_chunks, sms)
                           : auto_cluster(B, num_chunks, sms);
        for (;;) {
            if (cluster_launchable(dev, dt, kinds[i], C, point)) {
                out->kind = kinds[i];
                out->C = C;
                out->sms = sms;
                if (kinds[i] == kKindScalarAligned) {  // narrow slices: the multi-row variants
                    const int per_thread = ((num_chunks + C - 1) / C + kThreads - 1) / kThreads;
                    const bool two_per_sm = (long long)B * C <= 2LL * sms;  // resident at 2 CTAs per SM
                    const int small = per_thread <= 1                        ? kKindSmall1
                                      : per_thread <= 2                      ? kKindSmall2
                                      : per_thread <= 4                      ? kKindSmall4
                                      : (per_thread <= 8 && two_per_sm) ? kKindWide8
                                                                             : -1;
                    if (small >= 0 && cluster_launchable(dev, dt, small, C, point))
                        out->kind = small;
                }
                return SPEC_OK;
            }
            if (want_C > 0 || C == 1)
                break;
            C >>= 1;
        }
    }
    return SPEC_ERR_UNSUPPORTED;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// True when p lies in device (or managed) memory; the kernels also read
// page-locked host memory mapped into the device's address space, with
// ordinary loads.
bool device_memory(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

spec_status run(const void *target, const void *draft, const int32_t *tokens, const int32_t *num_draft,
                const float *uniforms, const float *temperature, int32_t *out_tokens, int32_t *out_num, int B,
                int gmax, int V, spec_dtype dtype, uint32_t *status, void *stream, float *p_hat, float *q_hat,
                float *logz_t, float *logz_d, float *resid_mass, int32_t *seq_status,
                const spec_verify_options *opt)
{
    if (dtype != SPEC_F32 && dtype != SPEC_BF16)
        return SPEC_ERR_UNSUPPORTED;
    if (B < 0 || B > SPEC_MAX_BATCH || gmax < 0 || gmax > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_VOCAB)
        return SPEC_ERR_INVALID_ARG;
    int want_C = 0, want_kind = -1;
    if (opt) {
        want_C = opt->cluster_size;
        if (want_C < 0 || want_C > kMaxCluster)
            return SPEC_ERR_INVALID_ARG;
        if (opt->kernel < 0 || opt->kernel > 3 || opt->kernel == 1)
            return SPEC_ERR_INVALID_ARG;
        want_kind = opt->kernel == 2 ? kKindScalarAligned : opt->kernel == 3 ? kKindEarlyAligned : -1;
    }
    if (B == 0)
        return SPEC_OK;
    if (!target || !uniforms || !temperature || !out_tokens)
        return SPEC_ERR_INVALID_ARG;
    if ((!num_draft || !out_num) && gmax != 0)
        return SPEC_ERR_INVALID_ARG;  // only the sampler (gamma_max 0) runs without them
    if (gmax > 0 && !tokens)
        return SPEC_ERR_INVALID_ARG;  // draft may be NULL: point-mass proposals
    const uintptr_t es = (uintptr_t)elem_size(dtype);
    if (((uintptr_t)target % es) || (draft && ((uintptr_t)draft % es)))
        return SPEC_ERR_INVALID_ARG;
    const void *four[] = {tokens, num_draft, uniforms, temperature, out_tokens, out_num, status,
                          p_hat,  q_hat,     logz_t,   logz_d,      resid_mass, seq_status};
    if (opt && (((uintptr_t)opt->counters & 7u) || ((uintptr_t)opt->accept_hist & 7u)))
        return SPEC_ERR_INVALID_ARG;
    for (const void *q : four)
        if ((uintptr_t)q & 3u)
            return SPEC_ERR_INVALID_ARG;
    const bool aligned = aligned16(target) && (!draft || aligned16(draft)) && ((size_t)V * (size_t)es) % 16 == 0;
    // point-mass kernels also for gamma_max = 0 (the sampler: no draft rows at
    // all), whose pass 2 is specialised for rows that are always p
    const bool point = gmax == 0 || !draft;
    // automatic: full sweep or early exit (the debug call's row diagnostics
    // need the full sweep, which reads every row)
    if (want_kind < 0 && gmax > 0 && !p_hat && !q_hat && !logz_t && !logz_d) {
        int dev = 0, sms = 0;
        if (current_device(&dev) == SPEC_OK && device_sm_count(dev, &sms) == SPEC_OK &&
            auto_early_exit(B, (V + chunk_width(dtype) - 1) / chunk_width(dtype), sms))
            want_kind = kKindEarlyAligned;
    }
    const bool host_rows = want_kind == kKindEarlyAligned && aligned &&
                           (!device_memory(target) || (draft && !device_memory(draft)));
    if (!aligned && want_kind == kKindScalarAligned)
        want_kind = kKindScalar;  // register loads work at any alignment
    if (!aligned && want_kind == kKindEarlyAligned)
        want_kind = kKindEarly;

    Shape shp;
    spec_status st = resolve_shape(B, V, dtype, aligned, want_kind, want_C, &shp, point, gmax == 0);
    if (st != SPEC_OK)
        return st;
    const int nslot = point ? 1 : 2;  // rows a position reads: t_i, and d_i unless point-mass
    if (host_rows && shp.kind == kKindEarlyAligned) {
        // Rows read over the host link reach no cache, so the early exit keeps
        // each position's slices in shared memory for pass 2: the smallest
        // cluster (from the automatic or requested one) whose slices fit.
        int dev = 0;
        if (current_device(&dev) == SPEC_OK) {
            const int chunks = (V + chunk_width(dtype) - 1) / chunk_width(dtype);
            for (int C = shp.C; C <= kMaxCluster; ++C) {
                if (want_C > 0 && C != want_C)
                    break;
                const long long cap = (chunks + C - 1) / C;
                const long long need = kP2SmemBytes + nslot * cap * 16;
                if (need <= kStagedDynMax && cluster_launchable(dev, dtype, kKindEarlyStaged, C, point)) {
                    shp.kind = kKindEarlyStaged;
                    shp.C = C;
                    break;
                }
            }
        }
    }
    Params prm;
    prm.target = target;
    prm.draft = draft;
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
    const int slice = (prm.num_chunks + shp.C - 1) / shp.C;
    // Longest-first order matters only when clusters wait for a free slot: a
    // grid that is resident at once (at most 4 CTAs per SM; 2 for the
    // two-rows-per-trip variant, 1 for the staged early exit) skips it and its
    // prologue.
    const long long slots = (long long)shp.sms * (shp.kind == kKindEarlyStaged ? 1 : shp.kind == kKindWide8 ? 2 : 4);
    // (in a one-row call the sampled rows, which draw exactly, go first)
    prm.ordered = (B <= kMaxOrdered && (long long)B * shp.C > slots) ? 1 : 0;
    prm.counters = opt ? reinterpret_cast<unsigned long long *>(opt->counters) : nullptr;
    prm.hist = opt ? reinterpret_cast<unsigned long long *>(opt->accept_hist) : nullptr;
    prm.parent = nullptr;
    prm.out_path = nullptr;
    size_t dyn = (size_t)(shp.kind == kKindWide8 ? kP2SmemBytesWide : kP2SmemBytes);
    if (shp.kind == kKindEarlyStaged)
        dyn += (size_t)nslot * (size_t)slice * 16;

    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg =
        launch_config((unsigned)B * (unsigned)shp.C, shp.C, dyn, (cudaStream_t)stream, attr);
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel_for(dtype, shp.kind, point), args);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
}

// Candidate-tree verification (spec_tree_verify): one cluster per sequence,
// the same automatic cluster size as the chain kernels.
spec_status run_tree(const void *target, const int32_t *parent, const int32_t *tokens, const int32_t *num_nodes,
                     const float *uniforms, const float *temperature, int32_t *out_tokens, int32_t *out_num,
                     int32_t *out_path, int B, int N, int V, spec_dtype dtype, uint32_t *status, void *stream,
                     const spec_verify_options *opt)
{
    if (dtype != SPEC_F32 && dtype != SPEC_BF16)
        return SPEC_ERR_UNSUPPORTED;
    if (B < 0 || B > SPEC_MAX_BATCH || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_VOCAB)
        return SPEC_ERR_INVALID_ARG;
    int want_C = 0;
    if (opt) {
        want_C = opt->cluster_size;
        if (want_C < 0 || want_C > kMaxCluster || opt->kernel != 0)
            return SPEC_ERR_INVALID_ARG;
        if (((uintptr_t)opt->counters & 7u) || ((uintptr_t)opt->accept_hist & 7u))
            return SPEC_ERR_INVALID_ARG;
    }
    if (B == 0)
        return SPEC_OK;
    if (!target || !parent || !tokens || !num_nodes || !uniforms || !temperature || !out_tokens || !out_num)
        return SPEC_ERR_INVALID_ARG;
    const uintptr_t es = (uintptr_t)elem_size(dtype);
    if ((uintptr_t)target % es)
        return SPEC_ERR_INVALID_ARG;
    const void *four[] = {parent, tokens, num_nodes, uniforms, temperature, out_tokens, out_num, out_path, status};
    for (const void *q : four)
        if ((uintptr_t)q & 3u)
            return SPEC_ERR_INVALID_ARG;
    const bool aligned = aligned16(target) && ((size_t)V * (size_t)es) % 16 == 0;
    Shape shp;
    spec_status st = resolve_shape(B, V, dtype, aligned, aligned ? kKindTreeAligned : kKindTree, want_C, &shp);
    if (st != SPEC_OK)
        return st;
    Params prm = {};
    prm.target = target;
    prm.draft = nullptr;
    prm.tokens = tokens;
    prm.num_draft = num_nodes;
    prm.uniforms = uniforms;
    prm.temperature = temperature;
    prm.out_tokens = out_tokens;
    prm.out_num = out_num;
    prm.status = status;
    prm.B = B;
    prm.gmax = N - 1;
    prm.V = V;
    prm.num_chunks = (V + chunk_width(dtype) - 1) / chunk_width(dtype);
    prm.ordered = 0;
    prm.counters = opt ? reinterpret_cast<unsigned long long *>(opt->counters) : nullptr;
    prm.hist = opt ? reinterpret_cast<unsigned long long *>(opt->accept_hist) : nullptr;
    prm.parent = parent;
    prm.out_path = out_path;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg =
        launch_config((unsigned)B * (unsigned)shp.C, shp.C, (size_t)kP2SmemBytes, (cudaStream_t)stream, attr);
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel_for(dtype, shp.kind, false), args);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
}

// An NVTX range around each entry point (launch side), so that a profiler's
// timeline names the calls; header-only NVTX, a no-op without a tool attached.
struct NvtxScope {
    explicit NvtxScope(const char *name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope &) = delete;
    NvtxScope &operator=(const NvtxScope &) = delete;
};

}  // namespace

extern "C" {

spec_status spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                        const int32_t *num_draft, const float *uniforms, const float *temperature,
                        int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                        spec_dtype dtype, uint32_t *status, void *stream)
{
    NvtxScope nvtx("spec_verify");
    if (B > 0 && (!num_draft || !out_num_accepted))
        return SPEC_ERR_INVALID_ARG;
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, nullptr, nullptr, nullptr, nullptr,
               nullptr, nullptr, nullptr);
}

spec_status spec_verify_debug(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                              const int32_t *num_draft, const float *uniforms, const float *temperature,
                              int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                              spec_dtype dtype, uint32_t *status, void *stream, float *p_hat, float *q_hat,
                              float *logz_t, float *logz_d, float *resid_mass, int32_t *seq_status,
                              const spec_verify_options *options)
{
    NvtxScope nvtx("spec_verify_debug");
    if (B > 0 && (!num_draft || !out_num_accepted))
        return SPEC_ERR_INVALID_ARG;
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, p_hat, q_hat, logz_t, logz_d, resid_mass,
               seq_status, options);
}

spec_status spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                           const int32_t *num_draft, const float *uniforms, const float *temperature,
                           int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                           spec_dtype dtype, uint32_t *status, void *stream, const spec_verify_options *options)
{
    NvtxScope nvtx("spec_verify_ex");
    if (B > 0 && (!num_draft || !out_num_accepted))
        return SPEC_ERR_INVALID_ARG;
    return run(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens,
               out_num_accepted, B, gamma_max, V, dtype, status, stream, nullptr, nullptr, nullptr, nullptr,
               nullptr, nullptr, options);
}

spec_status spec_sample(const void *logits, const float *uniforms, const float *temperature, int32_t *out_tokens,
                        int B, int V, spec_dtype dtype, uint32_t *status, void *stream,
                        const spec_verify_options *options)
{
    NvtxScope nvtx("spec_sample");
    return run(logits, nullptr, nullptr, nullptr, uniforms, temperature, out_tokens, nullptr, B, 0, V, dtype, status,
               stream, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, options);
}

spec_status spec_tree_verify(const void *target_logits, const int32_t *parent, const int32_t *tokens,
                             const int32_t *num_nodes, const float *uniforms, const float *temperature,
                             int32_t *out_tokens, int32_t *out_num_accepted, int32_t *out_path, int B,
                             int max_nodes, int V, spec_dtype dtype, uint32_t *status, void *stream,
                             const spec_verify_options *options)
{
    NvtxScope nvtx("spec_tree_verify");
    return run_tree(target_logits, parent, tokens, num_nodes, uniforms, temperature, out_tokens, out_num_accepted,
                    out_path, B, max_nodes, V, dtype, status, stream, options);
}

spec_status spec_ngram_propose(const int32_t *context, int64_t context_stride, const int32_t *context_len, int B,
                               int min_n, int max_n, int gamma_max, int32_t *draft_tokens, int32_t *num_draft,
                               void *stream)
{
    NvtxScope nvtx("spec_ngram_propose");
    if (B < 0 || B > SPEC_MAX_BATCH || gamma_max < 0 || gamma_max > SPEC_MAX_GAMMA || min_n < 1 ||
        max_n < min_n || max_n > kMaxNgram || context_stride < 1 || context_stride > (int64_t)INT_MAX)
        return SPEC_ERR_INVALID_ARG;
    if (B == 0)
        return SPEC_OK;
    if (!context || !context_len || !num_draft || (gamma_max > 0 && !draft_tokens))
        return SPEC_ERR_INVALID_ARG;
    const void *four[] = {context, context_len, draft_tokens, num_draft};
    for (const void *q : four)
        if ((uintptr_t)q & 3u)
            return SPEC_ERR_INVALID_ARG;
    spec_ngram_kernel<<<B, kNgramThreads, 0, (cudaStream_t)stream>>>(context, (long long)context_stride,
                                                                     context_len, min_n, max_n, gamma_max,
                                                                     draft_tokens, num_draft);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_verify_launch_shape(int B, int gamma_max, int V, spec_dtype dtype, int *cluster_size,
                                     int *num_ctas, int *threads_per_cta, int *kernel)
{
    if (dtype != SPEC_F32 && dtype != SPEC_BF16)
        return SPEC_ERR_UNSUPPORTED;
    if (B < 0 || B > SPEC_MAX_BATCH || gamma_max < 0 || gamma_max > SPEC_MAX_GAMMA || V < 1 ||
        V > SPEC_MAX_VOCAB)
        return SPEC_ERR_INVALID_ARG;
    const bool aligned = ((size_t)V * (size_t)elem_size(dtype)) % 16 == 0;
    int want = -1;
    if (gamma_max > 0) {
        int dev = 0, sms = 0;
        spec_status st0 = current_device(&dev);
        if (st0 == SPEC_OK)
            st0 = device_sm_count(dev, &sms);
        if (st0 != SPEC_OK)
            return st0;
        if (auto_early_exit(B > 0 ? B : 1, (V + chunk_width(dtype) - 1) / chunk_width(dtype), sms))
            want = aligned ? kKindEarlyAligned : kKindEarly;
    }
    Shape shp;
    spec_status st = resolve_shape(B > 0 ? B : 1, V, dtype, aligned, want, 0, &shp, gamma_max == 0, gamma_max == 0);
    if (st != SPEC_OK)
        return st;
    if (kernel)
        *kernel = (shp.kind == kKindEarlyAligned || shp.kind == kKindEarly) ? 3 : 2;
    if (cluster_size)
        *cluster_size = shp.C;
    if (num_ctas)
        *num_ctas = B * shp.C;
    if (threads_per_cta)
        *threads_per_cta = kThreads;
    return SPEC_OK;
}

spec_status spec_device_pointer(const void *ptr, const void **device_ptr)
{
    if (!ptr || !device_ptr)
        return SPEC_ERR_INVALID_ARG;
    int dev = 0;
    spec_status st = current_device(&dev);
    if (st != SPEC_OK)
        return st;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    if (!a.devicePointer)
        return SPEC_ERR_INVALID_ARG;  // pageable or unregistered host memory
    if ((a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device != dev)
        return SPEC_ERR_INVALID_ARG;  // another GPU's memory
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged && a.type != cudaMemoryTypeHost)
        return SPEC_ERR_INVALID_ARG;
    *device_ptr = a.devicePointer;
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
