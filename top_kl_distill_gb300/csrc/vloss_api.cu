// C ABI of libvloss: argument checks on the host, launch choice, small kernels
// (acc_add, windowed mean).  Declarations and contracts: include/vloss.h.
#include "vl_device.cuh"
#include "vl_internal.h"
#include "vloss.h"

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

namespace vl {
namespace {

thread_local std::string g_last_error;

vl_status fail(vl_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

vl_status cuda_fail(cudaError_t e, const char* where) {
    return fail(VL_ELAUNCH, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

vl_status ok() { return VL_OK; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Longest row: the kernels index a row with 32-bit ints and step through it in
// tiles of a few thousand columns, so a row stays 2^16 columns short of 2^31.
constexpr long long kMaxCols = VL_MAX_COLS;

vl_status check_rows(const void* logits, int64_t ld, int64_t ntok, int64_t V, const char* fn) {
    if (ntok < 0) return fail(VL_EINVAL, "%s: ntok < 0", fn);
    if (V < 1 || V > kMaxCols) return fail(VL_EINVAL, "%s: V must be in [1, %lld]", fn, kMaxCols);
    if (ld < V) return fail(VL_EINVAL, "%s: ld (%lld) < V (%lld)", fn, (long long)ld, (long long)V);
    if (ntok > 0 && logits == nullptr) return fail(VL_EINVAL, "%s: logits is NULL", fn);
    return ok();
}

vl_status check_window(int64_t ls, int64_t le, int64_t ntok, const char* fn) {
    if (!(0 <= ls && ls <= le && le <= ntok))
        return fail(VL_EINVAL, "%s: window [%lld, %lld) not inside [0, %lld]", fn, (long long)ls, (long long)le,
                    (long long)ntok);
    return ok();
}

vl_status check_slice(int64_t col0, int64_t ncols, int64_t V, const char* fn) {
    if (col0 < 0 || ncols < 0 || col0 + ncols > V)
        return fail(VL_EINVAL, "%s: slice [%lld, %lld) not inside [0, %lld)", fn, (long long)col0,
                    (long long)(col0 + ncols), (long long)V);
    return ok();
}

int num_sms() {
    static std::atomic<int> cache[64];
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_acquire);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_release);
    return sms;
}

// Grid of a launch.  Streaming modes: one CTA per SM (or per row when there are
// fewer rows).  Self-contained mode: a row may be split over a cluster of c CTAs;
// c is chosen from the estimated time, rows per cluster x (columns per CTA + a
// fixed per-row cost of the cluster exchange), which favours c > 1 only when
// rows are scarce.  VLOSS_CLUSTER=c overrides the choice.
struct Grid {
    int csize;
    int nclusters;
};

int l2_bytes() {
    static std::atomic<int> cache[64];
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_acquire);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_release);
    return v;
}

Grid choose_grid(int op, bool resident, long long rows, long long ncols, int dtype) {
    const int sms = num_sms();
    if (!resident) {
        long long g = rows < sms ? rows : sms;
        return Grid{1, (int)(g > 0 ? g : 1)};
    }
    // Self-contained mode re-reads a row part in pass B from L2 while the next part is
    // read: about two parts of esize ncols / c bytes per CTA are live.  Splitting a row over
    // c CTAs keeps them within 0.4 of L2 for fp32 (c = 3 at 128256 columns on a GB300: 1.46 ms
    // for 8192 rows, against 1.51 ms with c = 4 and 1.86 ms with c = 2).  bf16 rows cost
    // twice the arithmetic per byte, so the kernel is issue-bound before it is HBM-bound and a
    // cluster's per-row exchange costs more than the re-reads that spill from L2: bf16 takes
    // up to 0.6 of L2 (c = 1 at 128256 columns: 1.01 ms against 1.23 ms with c = 2).
    const double live = 2.0 * (dtype == kBf16 ? 2.0 : 4.0) * (double)ncols * (double)sms;
    const double budget = l2_bytes() > 0 ? l2_bytes() * (dtype == kBf16 ? 0.6 : 0.4) : 40e6;
    int cmin = 1;
    while (cmin < kMaxCluster && live / cmin > budget) ++cmin;
    static const int forced = [] {
        const char* e = std::getenv("VLOSS_CLUSTER");
        return e ? std::atoi(e) : 0;
    }();
    if (forced >= 1 && forced <= kMaxCluster) {
        const int n = row_max_clusters(op, resident, forced, dtype);
        if (n > 0) return Grid{forced, (int)(rows < n ? rows : n)};
    }
    const double esize = dtype == kBf16 ? 2.0 : 4.0;
    const double exchange = 61440.0;               // modelled fixed cost of a cluster exchange, in bytes
    Grid best{0, 0};
    double best_cost = 0;
    for (int c = cmin; c <= kMaxCluster; ++c) {
        const int n = row_max_clusters(op, resident, c, dtype);
        if (n <= 0) continue;
        const long long ncl = rows < n ? rows : n;
        const long long waves = (rows + ncl - 1) / ncl;
        const double cost = (double)waves * ((double)((ncols + c - 1) / c) * esize + (c > 1 ? exchange : 0.0));
        if (best.csize == 0 || cost < best_cost * 0.98) {
            best = Grid{c, (int)(ncl > 0 ? ncl : 1)};
            best_cost = cost;
        }
    }
    return best;
}

// ------------------------------------------------------------------ small kernels

__global__ void acc_add_kernel(float* a, const float* b, long long head, long long n4,
                               long long n) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    if (tid < head) a[tid] = a[tid] + b[tid];
    float4* a4 = reinterpret_cast<float4*>(a + head);
    const float4* b4 = reinterpret_cast<const float4*>(b + head);
    for (long long i = tid; i < n4; i += stride) {
        float4 x = a4[i];
        const float4 y = b4[i];
        x.x = x.x + y.x;
        x.y = x.y + y.y;
        x.z = x.z + y.z;
        x.w = x.w + y.w;
        a4[i] = x;
    }
    const long long t0 = head + 4 * n4;
    if (t0 + tid < n) a[t0 + tid] = a[t0 + tid] + b[t0 + tid];
}

__global__ void acc_add_scalar_kernel(float* a, const float* b, long long n) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) a[i] = a[i] + b[i];
}

// Error-free sum of two floats (Knuth's TwoSum): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// (hi, lo) += (h2, l2) for unevaluated float pairs (double-float addition).
__device__ __forceinline__ void ff_add(float& hi, float& lo, float h2, float l2) {
    float s, e;
    two_sum(hi, h2, s, e);
    e += lo + l2;
    two_sum(s, e, hi, lo);
}

// mean of loss[ls, le), accumulated as float pairs (about 48 significant bits) in a
// fixed order, so the result does not depend on the launch and needs no FP64 unit.
// Launched as a programmatic dependent of the loss kernel: its launch overlaps that
// kernel, griddepcontrol.wait holds it until the losses are in memory.
__global__ void __launch_bounds__(1024) mean_kernel(const float* __restrict__ loss, long long ls, long long le,
                                                    float* __restrict__ mean) {
    pdl_launch_dependents();                 // the next kernel may start its set-up
    pdl_wait_primary();
    __shared__ float2 red[32];
    float hi = 0.f, lo = 0.f;
    for (long long i = ls + threadIdx.x; i < le; i += blockDim.x) ff_add(hi, lo, loss[i], 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, off), l2 = __shfl_xor_sync(0xffffffffu, lo, off);
        ff_add(hi, lo, h2, l2);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(hi, lo);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int nw = (int)(blockDim.x >> 5);
        float2 v = (int)threadIdx.x < nw ? red[threadIdx.x] : make_float2(0.f, 0.f);
        hi = v.x;
        lo = v.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float h2 = __shfl_xor_sync(0xffffffffu, hi, off), l2 = __shfl_xor_sync(0xffffffffu, lo, off);
            ff_add(hi, lo, h2, l2);
        }
        if (threadIdx.x == 0) {
            // (hi + lo) / n: the quotient of the pair, one correction step
            const float n = (float)(le - ls);
            float q = hi / n, pe;
            const float p = q * n;
            pe = fmaf(q, n, -p);                     // q * n = p + pe exactly
            q += ((hi - p) - pe + lo) / n;
            *mean = le > ls ? q : 0.0f;
        }
    }
}

cudaError_t launch_mean(const float* loss, long long ls, long long le, float* mean, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(1024, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {(void*)&loss, (void*)&ls, (void*)&le, (void*)&mean};
    return cudaLaunchKernelExC(&cfg, (const void*)mean_kernel, args);
}

RowParams base_params(const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V) {
    RowParams P;
    std::memset(&P, 0, sizeof(P));
    P.x = const_cast<void*>(logits);
    P.dtype = dtype;
    P.ld = ld;
    P.ntok = ntok;
    P.V = V;
    P.col0 = 0;
    P.ncols = V;
    P.rbeg = 0;
    P.rend = ntok;
    P.csize = 1;
    P.wait_limit = kWaitTimeoutCycles;
    P.withhold = -1;
    return P;
}

// Test hook (vl_test_inject_wait_timeout): applies to the next row-engine launch made
// from this host thread, then clears itself.
thread_local long long g_inject_withhold = -1;
thread_local long long g_inject_wait = 0;

// Fused CE with one CTA per row leaves some CTAs a whole row more than others when the rows
// do not divide evenly (512 rows on 152 SMs: 56 CTAs take 4 rows, 96 take 3).  On 2-CTA
// clusters each CTA takes whole rows of its cluster's block and an odd block's last row is
// split over the pair (exchanged through distributed shared memory), so no CTA carries more
// than half a row above another.  Taken when that lowers the most rows a CTA carries by 10%
// or more (512 rows: 3.5 against 4, 26.7 against 28.5 us; at 2048 rows 13.5 against 14 is
// slower, 94.7 against 90.3 us) and every cluster has at least two rows.  VLOSS_MIXED=0
// turns it off.
Grid mixed_grid(int op, bool resident, long long rows, long long ncols, int dtype, const Grid& g) {
    static const int env = [] {
        const char* e = std::getenv("VLOSS_MIXED");
        return e ? std::atoi(e) : -1;
    }();
    const int nv = dtype == kBf16 ? 8 : 4;
    if (env == 0 || op != kCeFused || !resident || g.csize != 1 || ncols < 4 * nv) return Grid{0, 0};
    const int n2 = row_max_clusters(op, resident, 2, dtype);
    if (n2 <= 0 || rows < 2LL * n2) return Grid{0, 0};
    const double whole = (double)((rows + g.nclusters - 1) / g.nclusters);
    const double pair = 0.5 * (double)((rows + n2 - 1) / n2);
    if (env != 1 && pair > 0.9 * whole) return Grid{0, 0};
    return Grid{2, n2};
}

vl_status run_rows(int op, bool resident, RowParams& P, long long rows, const char* fn, cudaStream_t st) {
    Grid g = choose_grid(op, resident, rows, P.ncols, P.dtype);
    if (g.csize == 0) return fail(VL_ELAUNCH, "%s: no launch configuration fits this device", fn);
    const Grid gm = mixed_grid(op, resident, rows, P.ncols, P.dtype, g);
    P.mixed = gm.csize == 2 ? 1 : 0;
    if (P.mixed) g = gm;
    P.csize = g.csize;
    if (g_inject_wait > 0) {
        P.withhold = g_inject_withhold;
        P.wait_limit = g_inject_wait;
        g_inject_withhold = -1;
        g_inject_wait = 0;
    }
    const cudaError_t e = launch_rows(op, resident, P, g.nclusters, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
}

}  // namespace
}  // namespace vl

using namespace vl;

extern "C" {

int vl_version(void) { return 100; }

const char* vl_status_string(vl_status s) {
    switch (s) {
        case VL_OK: return "ok";
        case VL_EINVAL: return "invalid argument";
        case VL_ELAUNCH: return "CUDA launch or runtime error";
        case VL_EUNSUPPORTED: return "unsupported by this build";
    }
    return "unknown status";
}

const char* vl_last_error_string(void) { return g_last_error.c_str(); }

static vl_status ce_fwd_impl(const char* fn, const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                    int64_t loss_start, int64_t loss_end, float* loss, float* lse, float* stats, float* mean,
                    int32_t* err, void* stream) {
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (ntok > 0 && (labels == nullptr || loss == nullptr)) return fail(VL_EINVAL, "%s: labels or loss is NULL", fn);
    const cudaStream_t st = as_stream(stream);
    if (ntok > 0) {
        RowParams P = base_params(logits, dtype, ld, ntok, V);
        P.labels = labels;
        P.ls = loss_start;
        P.le = loss_end;
        P.loss = loss;
        P.lse_out = lse;
        P.stats_out = stats;
        P.err = err;
        if ((s = run_rows(kCeFwd, false, P, ntok, fn, st))) return s;
    }
    if (mean) {
        const cudaError_t e = launch_mean(loss, loss_start, loss_end, mean, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return VL_OK;
}

static vl_status ce_bwd_impl(const char* fn, const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                            const uint32_t* labels, const float* lse, const float* stats, int64_t loss_start,
                            int64_t loss_end, float scale, float* loss_part, int32_t* err, void* stream) {
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if ((s = check_slice(col0, ncols, V, fn))) return s;
    if (ntok > 0 && labels == nullptr) return fail(VL_EINVAL, "%s: labels is NULL", fn);
    if (ntok > 0 && lse == nullptr && stats == nullptr) return fail(VL_EINVAL, "%s: need lse or stats", fn);
    if (ntok == 0 || ncols == 0) return VL_OK;
    RowParams P = base_params(logits, dtype, ld, ntok, V);
    P.col0 = col0;
    P.ncols = ncols;
    P.labels = labels;
    P.lse_in = lse;
    P.stats_in = stats;
    P.ls = loss_start;
    P.le = loss_end;
    P.cg = scale;
    P.ce_coef = scale;
    P.loss = loss_part;
    P.err = err;
    return run_rows(kCeBwd, false, P, ntok, fn, as_stream(stream));
}

static vl_status ce_fused_impl(const char* fn, const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                      int64_t loss_start, int64_t loss_end, float scale, float* loss, float* lse, float* stats,
                      float* mean, int32_t* err, void* stream) {
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (ntok > 0 && (labels == nullptr || loss == nullptr)) return fail(VL_EINVAL, "%s: labels or loss is NULL", fn);
    const cudaStream_t st = as_stream(stream);
    if (ntok > 0) {
        RowParams P = base_params(logits, dtype, ld, ntok, V);
        P.labels = labels;
        P.ls = loss_start;
        P.le = loss_end;
        P.cg = scale;
        P.ce_coef = scale;
        P.loss = loss;
        P.lse_out = lse;
        P.stats_out = stats;
        P.err = err;
        if ((s = run_rows(kCeFused, true, P, ntok, fn, st))) return s;
    }
    if (mean) {
        const cudaError_t e = launch_mean(loss, loss_start, loss_end, mean, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return VL_OK;
}

static vl_status kl_impl(const char* fn, const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                             const uint32_t* tid, const float* tp, int64_t k, float coef, int64_t loss_start,
                             int64_t loss_end, const float* lse_in, const float* stats_in, const uint32_t* labels,
                             float ce_coef, float* loss, int32_t* err, void* stream) {
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if ((s = check_slice(col0, ncols, V, fn))) return s;
    if (k < 1) return fail(VL_EINVAL, "%s: k < 1", fn);
    if (k > VL_KL_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_KL_KMAX);
    if (ntok > 0 && (tid == nullptr || tp == nullptr || loss == nullptr))
        return fail(VL_EINVAL, "%s: tid, tp or loss is NULL", fn);
    const bool self = lse_in == nullptr && stats_in == nullptr;
    if (self && (col0 != 0 || ncols != V))
        return fail(VL_EINVAL, "%s: a slice needs lse_in or stats_in (the statistics of the full row)", fn);
    if (ntok == 0) return VL_OK;
    RowParams P = base_params(logits, dtype, ld, ntok, V);
    P.col0 = col0;
    P.ncols = ncols;
    P.tid = tid;
    P.tp = tp;
    P.k = (int)k;
    const bool fold = labels != nullptr && ce_coef != 0.0f;
    P.labels = fold ? labels : nullptr;
    P.ce_coef = fold ? ce_coef : 0.0f;
    P.coef = coef;
    P.cg = coef + P.ce_coef;
    P.ls = loss_start;
    P.le = loss_end;
    P.lse_in = lse_in;
    P.stats_in = stats_in;
    P.loss = loss;
    P.err = err;
    const long long rows = loss_end - loss_start;
    return run_rows(kKl, self, P, rows > 0 ? rows : 1, fn, as_stream(stream));
}

static vl_status ce_kl_impl(const char* fn, const void* logits, int dtype, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                         const uint32_t* tid, const float* tp, int64_t k, float coef, float ce_coef,
                         int64_t loss_start, int64_t loss_end, float* kl_loss, float* ce_loss, float* lse,
                         float* stats, float* ce_mean, int32_t* err, void* stream) {
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (k < 1) return fail(VL_EINVAL, "%s: k < 1", fn);
    if (k > VL_KL_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_KL_KMAX);
    if (ntok > 0 && (labels == nullptr || tid == nullptr || tp == nullptr || kl_loss == nullptr ||
                     ce_loss == nullptr))
        return fail(VL_EINVAL, "%s: labels, tid, tp, kl_loss or ce_loss is NULL", fn);
    const cudaStream_t st = as_stream(stream);
    if (ntok > 0) {
        RowParams P = base_params(logits, dtype, ld, ntok, V);
        P.tid = tid;
        P.tp = tp;
        P.k = (int)k;
        P.labels = labels;
        P.coef = coef;
        P.ce_coef = ce_coef;
        P.cg = coef + ce_coef;
        P.ls = loss_start;
        P.le = loss_end;
        P.loss = kl_loss;
        P.ce_loss = ce_loss;
        P.lse_out = lse;
        P.stats_out = stats;
        P.err = err;
        const long long rows = loss_end - loss_start;
        if ((s = run_rows(kKl, true, P, rows > 0 ? rows : 1, fn, st))) return s;
    }
    if (ce_mean) {
        const cudaError_t e = launch_mean(ce_loss, loss_start, loss_end, ce_mean, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return VL_OK;
}

vl_status vl_ce_fwd(const float* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                    int64_t loss_start, int64_t loss_end, float* loss, float* lse, float* stats, float* mean,
                    int32_t* err, void* stream) {
    return ce_fwd_impl("vl_ce_fwd", logits, kF32, ld, ntok, V, labels, loss_start, loss_end, loss, lse, stats,
                       mean, err, stream);
}

vl_status vl_ce_fwd_bf16(const uint16_t* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                    int64_t loss_start, int64_t loss_end, float* loss, float* lse, float* stats, float* mean,
                    int32_t* err, void* stream) {
    return ce_fwd_impl("vl_ce_fwd_bf16", logits, kBf16, ld, ntok, V, labels, loss_start, loss_end, loss, lse,
                       stats, mean, err, stream);
}

vl_status vl_ce_bwd_inplace(float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                            const uint32_t* labels, const float* lse, const float* stats, int64_t loss_start,
                            int64_t loss_end, float scale, float* loss_part, int32_t* err, void* stream) {
    return ce_bwd_impl("vl_ce_bwd_inplace", logits, kF32, ld, ntok, V, col0, ncols, labels, lse, stats, loss_start,
                       loss_end, scale, loss_part, err, stream);
}

vl_status vl_ce_bwd_inplace_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                            const uint32_t* labels, const float* lse, const float* stats, int64_t loss_start,
                            int64_t loss_end, float scale, float* loss_part, int32_t* err, void* stream) {
    return ce_bwd_impl("vl_ce_bwd_inplace_bf16", logits, kBf16, ld, ntok, V, col0, ncols, labels, lse, stats,
                       loss_start, loss_end, scale, loss_part, err, stream);
}

vl_status vl_ce_fused(float* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                      int64_t loss_start, int64_t loss_end, float scale, float* loss, float* lse, float* stats,
                      float* mean, int32_t* err, void* stream) {
    return ce_fused_impl("vl_ce_fused", logits, kF32, ld, ntok, V, labels, loss_start, loss_end, scale, loss, lse,
                         stats, mean, err, stream);
}

vl_status vl_ce_fused_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                      int64_t loss_start, int64_t loss_end, float scale, float* loss, float* lse, float* stats,
                      float* mean, int32_t* err, void* stream) {
    return ce_fused_impl("vl_ce_fused_bf16", logits, kBf16, ld, ntok, V, labels, loss_start, loss_end, scale, loss,
                         lse, stats, mean, err, stream);
}

vl_status vl_kl_topk_inplace(float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                             const uint32_t* tid, const float* tp, int64_t k, float coef, int64_t loss_start,
                             int64_t loss_end, const float* lse_in, const float* stats_in, const uint32_t* labels,
                             float ce_coef, float* loss, int32_t* err, void* stream) {
    return kl_impl("vl_kl_topk_inplace", logits, kF32, ld, ntok, V, col0, ncols, tid, tp, k, coef, loss_start,
                   loss_end, lse_in, stats_in, labels, ce_coef, loss, err, stream);
}

vl_status vl_kl_topk_inplace_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V, int64_t col0, int64_t ncols,
                             const uint32_t* tid, const float* tp, int64_t k, float coef, int64_t loss_start,
                             int64_t loss_end, const float* lse_in, const float* stats_in, const uint32_t* labels,
                             float ce_coef, float* loss, int32_t* err, void* stream) {
    return kl_impl("vl_kl_topk_inplace_bf16", logits, kBf16, ld, ntok, V, col0, ncols, tid, tp, k, coef,
                   loss_start, loss_end, lse_in, stats_in, labels, ce_coef, loss, err, stream);
}

vl_status vl_ce_kl_fused(float* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                         const uint32_t* tid, const float* tp, int64_t k, float coef, float ce_coef,
                         int64_t loss_start, int64_t loss_end, float* kl_loss, float* ce_loss, float* lse,
                         float* stats, float* ce_mean, int32_t* err, void* stream) {
    return ce_kl_impl("vl_ce_kl_fused", logits, kF32, ld, ntok, V, labels, tid, tp, k, coef, ce_coef, loss_start,
                      loss_end, kl_loss, ce_loss, lse, stats, ce_mean, err, stream);
}

vl_status vl_ce_kl_fused_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V, const uint32_t* labels,
                         const uint32_t* tid, const float* tp, int64_t k, float coef, float ce_coef,
                         int64_t loss_start, int64_t loss_end, float* kl_loss, float* ce_loss, float* lse,
                         float* stats, float* ce_mean, int32_t* err, void* stream) {
    return ce_kl_impl("vl_ce_kl_fused_bf16", logits, kBf16, ld, ntok, V, labels, tid, tp, k, coef, ce_coef,
                      loss_start, loss_end, kl_loss, ce_loss, lse, stats, ce_mean, err, stream);
}

// SMs of the current device; without one, 256 (more than any current GPU has).
static long long current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        cudaGetLastError();
        return 256;
    }
    return sms;
}

int64_t vl_topk_workspace_bytes(int64_t ntok, int64_t V, int64_t k) {
    if (ntok < 1 || V < 1 || V > kMaxCols || k < 1 || k > V || k > VL_TOPK_KMAX) return 0;
    if (topk_filter_spec_a(V, (int)k) == 0) return 0;
    const long long sms = current_sms();
    return topk_ws_bytes(ntok, V, (int)k, ntok < sms ? ntok : sms);
}

vl_status vl_topk_rows(const float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t k, int64_t loss_start,
                       int64_t loss_end, uint32_t* ids, float* probs, int32_t* err, void* workspace,
                       int64_t workspace_bytes, void* stream) {
    const char* fn = "vl_topk_rows";
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (k < 1 || k > V) return fail(VL_EINVAL, "%s: k = %lld outside [1, V]", fn, (long long)k);
    if (k > VL_TOPK_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_TOPK_KMAX);
    if (loss_end > loss_start && (ids == nullptr || probs == nullptr))
        return fail(VL_EINVAL, "%s: ids or probs is NULL", fn);
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return fail(VL_EINVAL, "%s: workspace not 16-byte aligned", fn);
    if (loss_end == loss_start) return VL_OK;
    cudaError_t e;
    if (workspace && topk_filter_spec_a(V, (int)k) > 0 &&
        workspace_bytes >= topk_ws_bytes(loss_end - loss_start, V, (int)k, 1))
        e = launch_topk_stream(logits, ld, V, (int)k, loss_start, loss_end, ids, probs, err, workspace,
                               workspace_bytes, kWaitTimeoutCycles, as_stream(stream));
    else
        e = launch_topk(logits, ld, ntok, V, (int)k, loss_start, loss_end, nullptr, nullptr, ids, probs, err,
                        as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return VL_OK;
}

int64_t vl_teacher_topk_workspace_bytes(int64_t rows, int64_t V, int64_t k) {
    if (rows < 1 || V < 1 || V > kMaxCols || k < 1 || k > V || k > VL_TOPK_KMAX) return 0;
    return teacher_ws_bytes(rows, V, (int)k);
}

int64_t vl_head_kl_workspace_bytes(int64_t rows, int64_t V) {
    if (rows < 1 || V < 1 || V > kMaxCols) return 0;
    return head_kl_ws_bytes(rows, V);
}

static vl_status check_head(const void* hidden, int64_t hs, const void* w, int64_t V, int64_t ntok, void* ws,
                            const char* fn) {
    if (ntok < 0 || hs < 8 || hs % 8 != 0) return fail(VL_EINVAL, "%s: need ntok >= 0 and hs a positive multiple of 8", fn);
    if (V < 1 || V > kMaxCols) return fail(VL_EINVAL, "%s: V must be in [1, %lld]", fn, kMaxCols);
    if (ntok > 0 && (hidden == nullptr || w == nullptr || ws == nullptr))
        return fail(VL_EINVAL, "%s: hidden, w or workspace is NULL", fn);
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(ws)) & 15u)
        return fail(VL_EINVAL, "%s: hidden, w and workspace must be 16-byte aligned", fn);
    return VL_OK;
}

vl_status vl_teacher_topk(const uint16_t* hidden, int64_t hs, const uint16_t* w, int64_t V, int64_t ntok, int64_t k,
                          int64_t loss_start, int64_t loss_end, uint32_t* ids, float* probs, int32_t* err,
                          void* workspace, int64_t workspace_bytes, void* stream) {
    const char* fn = "vl_teacher_topk";
    vl_status s = check_head(hidden, hs, w, V, ntok, workspace, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (k < 1 || k > V) return fail(VL_EINVAL, "%s: k = %lld outside [1, V]", fn, (long long)k);
    if (k > VL_TOPK_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_TOPK_KMAX);
    if (loss_end > loss_start && (ids == nullptr || probs == nullptr))
        return fail(VL_EINVAL, "%s: ids or probs is NULL", fn);
    if (loss_end == loss_start) return VL_OK;
    char msg[400];
    const int r = teacher_topk(hidden, hs, w, V, ntok, (int)k, loss_start, loss_end, ids, probs, err, workspace,
                               workspace_bytes, as_stream(stream), msg, sizeof(msg));
    if (r) return fail((vl_status)r, "%s: %s", fn, msg);
    return VL_OK;
}

vl_status vl_head_kl(const uint16_t* hidden, int64_t hs, const uint16_t* w, const uint16_t* wt, int64_t V, int64_t ntok,
                     const uint32_t* labels, const uint32_t* tid, const float* tp, int64_t k, float coef,
                     float ce_coef, float dx_scale, int64_t loss_start, int64_t loss_end, float* dx, float* kl_loss,
                     float* ce_loss, float* ce_mean, int32_t* err, void* workspace, int64_t workspace_bytes,
                     void* stream) {
    const char* fn = "vl_head_kl";
    vl_status s = check_head(hidden, hs, w, V, ntok, workspace, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (k < 1) return fail(VL_EINVAL, "%s: k < 1", fn);
    if (k > VL_KL_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_KL_KMAX);
    if (ntok > 0 && (labels == nullptr || tid == nullptr || tp == nullptr || dx == nullptr || kl_loss == nullptr ||
                     ce_loss == nullptr))
        return fail(VL_EINVAL, "%s: labels, tid, tp, dx, kl_loss or ce_loss is NULL", fn);
    if (reinterpret_cast<uintptr_t>(dx) & 15u) return fail(VL_EINVAL, "%s: dx must be 16-byte aligned", fn);
    if (ntok == 0) return VL_OK;
    char msg[400];
    if (wt && (reinterpret_cast<uintptr_t>(wt) & 15u)) return fail(VL_EINVAL, "%s: wt must be 16-byte aligned", fn);
    const int r = head_kl(hidden, hs, w, wt, V, ntok, labels, tid, tp, (int)k, coef, ce_coef, dx_scale, loss_start,
                          loss_end, dx, kl_loss, ce_loss, ce_mean, err, workspace, workspace_bytes,
                          as_stream(stream), msg, sizeof(msg));
    if (r) return fail((vl_status)r, "%s: %s", fn, msg);
    return VL_OK;
}

vl_status vl_gemm_bf16_tn(const uint16_t* A, const uint16_t* B, float* D, int64_t M, int64_t N, int64_t K,
                          int64_t ldd, float alpha, void* stream) {
    const char* fn = "vl_gemm_bf16_tn";
    if (M < 0 || N < 0 || K < 0) return fail(VL_EINVAL, "%s: negative size", fn);
    if (M == 0 || N == 0) return VL_OK;
    if (K < 8 || K % 8 != 0) return fail(VL_EINVAL, "%s: K must be a positive multiple of 8", fn);
    if (ldd < N) return fail(VL_EINVAL, "%s: ldd < N", fn);
    if (A == nullptr || B == nullptr || D == nullptr) return fail(VL_EINVAL, "%s: NULL pointer", fn);
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u)
        return fail(VL_EINVAL, "%s: A and B must be 16-byte aligned", fn);
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return fail(VL_EUNSUPPORTED, "%s: size above 2^30", fn);
    const cudaError_t e = tc_gemm_tn(A, B, D, M, N, K, ldd, alpha, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return VL_OK;
}

// Scratch of a stream launch over `rows` rows with its full grid on the current device.
static long long noalloc_need(long long rows, long long V, int k, long long sms) {
    return topk_ws_bytes(rows, V, k, rows < sms ? rows : sms);
}

// The most rows one call takes with the fixed array (the need grows with the rows).
static long long noalloc_max_rows(long long V, int k, long long sms) {
    long long lo = 0, hi = 1LL << 40;
    while (lo < hi) {
        const long long mid = lo + (hi - lo + 1) / 2;
        if (noalloc_need(mid, V, k, sms) <= VL_TOPK_NOALLOC_BYTES) lo = mid; else hi = mid - 1;
    }
    return lo;
}

vl_status vl_topk_rows_noalloc(const float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t k,
                               int64_t loss_start, int64_t loss_end, uint32_t* ids, float* probs, int32_t* err,
                               void* stream) {
    const char* fn = "vl_topk_rows_noalloc";
    vl_status s = check_rows(logits, ld, ntok, V, fn);
    if (s) return s;
    if ((s = check_window(loss_start, loss_end, ntok, fn))) return s;
    if (k < 1 || k > V) return fail(VL_EINVAL, "%s: k = %lld outside [1, V]", fn, (long long)k);
    if (k > VL_TOPK_KMAX) return fail(VL_EUNSUPPORTED, "%s: k = %lld > %d", fn, (long long)k, VL_TOPK_KMAX);
    if (loss_end > loss_start && (ids == nullptr || probs == nullptr))
        return fail(VL_EINVAL, "%s: ids or probs is NULL", fn);
    const long long rows = loss_end - loss_start;
    if (rows == 0) return VL_OK;
    cudaError_t e;
    if (topk_filter_spec_a(V, (int)k) > 0) {
        const long long sms = current_sms();
        const long long need = noalloc_need(rows, V, (int)k, sms);
        if (need > VL_TOPK_NOALLOC_BYTES)
            return fail(VL_EUNSUPPORTED,
                        "%s: %lld rows need %lld bytes of scratch, more than the fixed %lld; call it on at most "
                        "%lld rows at a time",
                        fn, rows, need, (long long)VL_TOPK_NOALLOC_BYTES, noalloc_max_rows(V, (int)k, sms));
        void* scratch = nullptr;
        if ((e = topk_noalloc_scratch(&scratch)) != cudaSuccess) return cuda_fail(e, fn);
        e = launch_topk_stream(logits, ld, V, (int)k, loss_start, loss_end, ids, probs, err, scratch,
                               VL_TOPK_NOALLOC_BYTES, kWaitTimeoutCycles, as_stream(stream));
    } else {
        e = launch_topk(logits, ld, ntok, V, (int)k, loss_start, loss_end, nullptr, nullptr, ids, probs, err,
                        as_stream(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return VL_OK;
}

vl_status vl_window_mean(const float* loss, int64_t ntok, int64_t loss_start, int64_t loss_end, float* mean,
                         void* stream) {
    const char* fn = "vl_window_mean";
    if (ntok < 0) return fail(VL_EINVAL, "%s: ntok < 0", fn);
    vl_status s = check_window(loss_start, loss_end, ntok, fn);
    if (s) return s;
    if (mean == nullptr) return fail(VL_EINVAL, "%s: mean is NULL", fn);
    if (loss_end > loss_start && loss == nullptr) return fail(VL_EINVAL, "%s: loss is NULL", fn);
    const cudaError_t e = launch_mean(loss, loss_start, loss_end, mean, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return VL_OK;
}

vl_status vl_acc_add(float* a, const float* b, int64_t n, void* stream) {
    const char* fn = "vl_acc_add";
    if (n < 0) return fail(VL_EINVAL, "%s: n < 0", fn);
    if (n == 0) return VL_OK;
    if (a == nullptr || b == nullptr) return fail(VL_EINVAL, "%s: NULL pointer", fn);
    if (a != b && ((a < b && a + n > b) || (b < a && b + n > a)))
        return fail(VL_EINVAL, "%s: a and b overlap", fn);
    const cudaStream_t st = as_stream(stream);
    const int sms = num_sms();
    const uintptr_t ma = reinterpret_cast<uintptr_t>(a) & 15u, mb = reinterpret_cast<uintptr_t>(b) & 15u;
    if (ma == mb && (ma & 3u) == 0) {
        long long head = (long long)((16u - ma) & 15u) / 4;
        if (head > n) head = n;
        const long long n4 = (n - head) / 4;
        long long blocks = (n4 + 255) / 256;
        const long long cap = (long long)(sms > 0 ? sms : 1) * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        acc_add_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, b, head, n4, n);
    } else {
        long long blocks = (n + 255) / 256;
        const long long cap = (long long)(sms > 0 ? sms : 1) * 8;
        if (blocks > cap) blocks = cap;
        acc_add_scalar_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, b, n);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return VL_OK;
}

vl_status vl_test_inject_wait_timeout(int64_t withhold_tile, int64_t wait_cycles) {
    if (withhold_tile < 0 || wait_cycles < 1000 || wait_cycles > kWaitTimeoutCycles)
        return fail(VL_EINVAL, "vl_test_inject_wait_timeout: need withhold_tile >= 0 and wait_cycles in [1000, %lld]",
                    (long long)kWaitTimeoutCycles);
    g_inject_withhold = withhold_tile;
    g_inject_wait = wait_cycles;
    return VL_OK;
}

int vl_watchdog_flag(int device, int clear) {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return -1;
    if (cudaSetDevice(device) != cudaSuccess) return -1;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaSetDevice(prev);
        return -1;
    }
    const unsigned int a = rows_watchdog(clear != 0), b = topk_watchdog(clear != 0),
                       c = topk_stream_watchdog(clear != 0), d = gemm_watchdog(clear != 0);
    cudaSetDevice(prev);
    if (a == 0xffffffffu || b == 0xffffffffu || c == 0xffffffffu || d == 0xffffffffu) return -1;
    return (int)((a | b | c | d) & 0x7fffffffu);
}

}  // extern "C"
