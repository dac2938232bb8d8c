// Row engine: cross-entropy (fused, forward, backward) and top-k KL over rows of
// fp32 vocabulary logits, one persistent CTA (or cluster of CTAs) per SM.
//
// Layout of one launch
//   * grid = nclusters * csize CTAs, at most one CTA per SM (the ring below takes
//     ~200 KB of shared memory).  Cluster i handles rows i, i + nclusters, ...
//   * a row slice of ncols floats is cut into a <=3-float head, a 16-byte-aligned
//     body and a <=3-float tail.  The body is split evenly (in float4 units)
//     across the csize CTAs of the cluster; CTA rank 0 also takes the head and
//     the last rank the tail.
//   * warp 0 (one lane) is the producer: it streams each CTA's body through a
//     ring of kSlots tiles of kTileF floats with 1-D bulk copies (TMA) signalled
//     on per-slot mbarriers; warps 1..16 are consumers.
//
// Modes
//   resident  (CE fused, KL without given statistics): the whole body part of a
//             row sits in the ring.  Consumers reduce (max, sum exp) over it,
//             merge across warps (shared memory) and across the cluster
//             (distributed shared memory + remote mbarrier arrive), then emit
//             the gradient from the staged tiles.  One HBM read, one HBM write.
//   streaming (CE backward, KL with given statistics): each tile is turned into
//             gradient as soon as it lands and its slot is released.
//   reduce    (CE forward): statistics only, tiles released after reduction.
//
// Sources: aprender-train wgpu_cross_entropy.rs (module doc, forward_async,
// backward: loss = lse - s[label], gradient scale * (softmax - onehot), loss
// window) and cortiq-engine train_head.rs (module doc and kl_rows: KL over the
// teacher's top-k, gradient coef * (softmax - p_T)).  The pages' kernels read a
// row three times with workgroup tree reductions; this engine reads it once.
#include "vl_device.cuh"
#include "vl_internal.h"

#include <atomic>
#include <cmath>

namespace vl {
namespace {

constexpr int NCW = 16;                 // consumer warps
constexpr int NCT = NCW * 32;           // consumer threads
constexpr int NTHREADS = NCT + 32;      // + the producer warp
constexpr int KMAX = 1024;              // teacher support per row
constexpr uint32_t kBarConsumers = 1;   // named barrier id used by consumers only

static_assert(kTileF / 4 == NCT, "one float4 of each tile per consumer thread");

__device__ unsigned int g_watchdog;

struct alignas(128) Smem {
    float ring[kSlots][kTileF];
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t xbar[2];                   // cluster exchange of (max, sum)
    uint64_t lbar[2];                   // cluster exchange of KL loss parts (rank 0)
    float2 xbuf[2][kMaxCluster];
    float lbuf[2][kMaxCluster];
    float2 wred[2][NCW];
    float wloss[2][NCW];
    unsigned long long skey[KMAX];      // (column << 32 | q) of the teacher support, unsorted
    float sp_raw[KMAX];
    uint32_t scol[KMAX];                // support sorted by (column, q)
    float sp[KMAX];
    int abort;
    uint32_t issued;
};

// Columns of one row slice handled by CTA `rank` of `c` (relative to the slice start).
struct Part {
    long long h;    // head length (first columns up to the 16-byte boundary)
    long long hn;   // head columns this CTA handles
    long long b0;   // first body column of this CTA
    long long bn;   // body columns of this CTA (a multiple of 4)
    long long t0;   // first tail column
    long long tn;   // tail columns this CTA handles
    long long lo;   // this CTA owns columns [lo, hi)
    long long hi;
};

__device__ __forceinline__ Part part_of(const float* rowp, long long n, int rank, int c) {
    Part p;
    const long long mis = (long long)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
    long long h = (4 - mis) & 3;
    if (h > n) h = n;
    const long long bt = (n - h) & ~3LL;
    const long long per = (((bt >> 2) + c - 1) / c) * 4;
    const long long s = min((long long)rank * per, bt);
    const long long e = min((long long)(rank + 1) * per, bt);
    p.h = h;
    p.hn = rank == 0 ? h : 0;
    p.b0 = h + s;
    p.bn = e - s;
    p.t0 = h + bt;
    p.tn = rank == c - 1 ? n - p.t0 : 0;
    p.lo = rank == 0 ? 0 : h + s;
    p.hi = rank == c - 1 ? n : h + e;
    return p;
}

template <int OP>
__device__ __forceinline__ bool row_loaded(const RowParams& P, long long r) {
    if (OP == kCeFused || OP == kCeFwd) return true;    // lse is produced for every row
    return r >= P.ls && r < P.le;
}

__device__ __forceinline__ float pick(const float4& v, long long d) {
    return d == 0 ? v.x : d == 1 ? v.y : d == 2 ? v.z : v.w;
}

__device__ __forceinline__ void sub_at(float4& o, long long d, float a) {
    if (d == 0) o.x -= a;
    else if (d == 1) o.y -= a;
    else if (d == 2) o.z -= a;
    else o.w -= a;
}

// softmax value from the row statistics: exp((s - m) - lnS)
__device__ __forceinline__ float soft(float s, float m, float lnS) {
    return ex2(((s - m) - lnS) * kLog2e);
}

// ---------------------------------------------------------------- producer

template <int OP>
__device__ void producer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    uint32_t g = 0;
    for (long long r = cid; r < P.ntok; r += ncl) {
        if (!row_loaded<OP>(P, r)) continue;
        const float* rowp = P.x + r * P.ld + P.col0;
        const Part pt = part_of(rowp, P.ncols, rank, P.csize);
        for (long long c0 = 0; c0 < pt.bn; c0 += kTileF) {
            const uint32_t slot = g % kSlots, use = g / kSlots;
            if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog)) {
                S.issued = g;
                return;
            }
            const uint32_t bytes = (uint32_t)min((long long)kTileF, pt.bn - c0) * 4u;
            mbar_arrive_expect_tx(&S.full[slot], bytes);
            bulk_g2s(S.ring[slot], rowp + pt.b0 + c0, bytes, &S.full[slot]);
            ++g;
        }
    }
    S.issued = g;
}

// Before the CTA exits, every bulk copy it issued must have landed.
__device__ void drain(Smem& S) {
    const uint32_t iss = S.issued;
    for (uint32_t gt = iss > (uint32_t)kSlots ? iss - kSlots : 0u; gt < iss; ++gt)
        wait_parity_drain(&S.full[gt % kSlots], (gt / kSlots) & 1u);
}

// ---------------------------------------------------------------- consumer helpers

__device__ void zero_part(float* rowp, const Part& pt, int ct) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = ct; i < (pt.bn >> 2); i += NCT) st_global_v4(rowp + pt.b0 + 4 * i, z);
    if (ct < pt.hn) rowp[ct] = 0.f;
    if (ct >= 4 && ct - 4 < pt.tn) rowp[pt.t0 + ct - 4] = 0.f;
}

// Teacher support of row r inside this CTA's columns, sorted by (column, q) into
// S.scol / S.sp.  Returns the number of entries.  Ids >= V are counted as errors.
__device__ int load_support(const RowParams& P, Smem& S, long long r, const Part& pt, int rank, int ct) {
    const int k = P.k;
    bool in[2] = {false, false};
    unsigned long long key[2] = {~0ull, ~0ull};
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
        const int q = ct + rep * NCT;
        if (q < k) {
            const uint32_t id = P.tid[r * k + q];
            const float p = P.tp[r * k + q];
            if ((long long)id >= P.V) {
                if (rank == 0 && P.err) atomicAdd(P.err, 1);
            } else {
                const long long rel = (long long)id - P.col0;
                if (rel >= pt.lo && rel < pt.hi) key[rep] = ((unsigned long long)rel << 32) | (unsigned)q;
            }
            S.skey[q] = key[rep];
            S.sp_raw[q] = p;
            in[rep] = key[rep] != ~0ull;
        }
    }
    uint32_t n = named_sync_popc(kBarConsumers, NCT, in[0]);
    if (k > NCT) n += named_sync_popc(kBarConsumers, NCT, in[1]);
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
        const int q = ct + rep * NCT;
        if (q < k && in[rep]) {
            int pos = 0;
            for (int j = 0; j < k; ++j) pos += S.skey[j] < key[rep] ? 1 : 0;
            S.scol[pos] = (uint32_t)(key[rep] >> 32);
            S.sp[pos] = S.sp_raw[q];
        }
    }
    named_sync(kBarConsumers, NCT);
    return (int)n;
}

// KL terms of the support entries [e0, e1) that fall on columns [c0, c0 + 4):
// subtract coef * p from the gradient and add p (ln p - (s - lse)) to the loss.
__device__ __forceinline__ void kl_apply4(const Smem& S, uint32_t e0, uint32_t e1, long long c0, const float4& v,
                                          float4& o, float coef, float m, float lnS, float& lacc) {
    for (uint32_t e = e0; e < e1; ++e) {
        const long long d = (long long)S.scol[e] - c0;
        if (d >= 0 && d < 4) {
            const float p = S.sp[e];
            sub_at(o, d, coef * p);
            if (p > 0.f) lacc += p * (logf(p) - ((pick(v, d) - m) - lnS));
        }
    }
}

// ---------------------------------------------------------------- consumer

template <int OP, bool RES>
__device__ void consumer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    constexpr bool kKL = OP == kKl;
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int c = P.csize;
    uint32_t g = 0, nred = 0, nloss = 0, nx = 0, nlx = 0;
    const bool has_label = (OP != kKl) || (P.labels != nullptr && P.ce_coef != 0.f);

    for (long long r = cid; r < P.ntok; r += ncl) {
        float* rowp = P.x + r * P.ld + P.col0;
        const Part pt = part_of(rowp, P.ncols, rank, c);
        const bool inwin = r >= P.ls && r < P.le;
        const uint32_t nt = (uint32_t)((pt.bn + kTileF - 1) / kTileF);
        if (RES && nt > (uint32_t)kSlots && ct == 0) {
            // the host never launches this; unwind rather than wait on a ring that cannot fill
            S.abort = 1;
            atomicOr(&g_watchdog, 2u);
        }

        if (!row_loaded<OP>(P, r)) {
            zero_part(rowp, pt, ct);
            if (ct == 0 && rank == 0 && P.loss) P.loss[r] = 0.f;
            continue;
        }

        // the label as a slice-relative column; -1 when there is none
        long long jl = -1;
        bool bad_label = false;
        if (has_label) {
            const uint32_t lab = P.labels[r];
            if ((long long)lab >= P.V) bad_label = true;
            else jl = (long long)lab - P.col0;
        }
        if (bad_label && inwin && rank == 0 && ct == 0 && P.err) atomicAdd(P.err, 1);

        int nsup = 0;
        if (kKL && inwin) nsup = load_support(P, S, r, pt, rank, ct);

        float m, lnS;
        float hv = 0.f, tv = 0.f;
        float s_label = 0.f;
        bool own_label = false;
        const bool has_head = ct < pt.hn;
        const bool has_tail = ct >= 4 && ct - 4 < pt.tn;

        if (RES || OP == kCeFwd) {
            // ---- statistics of the row: (max, sum exp) over head, body tiles and tail
            MaxSum ms = ms_empty();
            if (has_head) { hv = rowp[ct]; ms_add(ms, hv); }
            if (has_tail) { tv = rowp[pt.t0 + ct - 4]; ms_add(ms, tv); }
            for (uint32_t t = 0; t < nt; ++t) {
                const uint32_t gt = g + t, slot = gt % kSlots;
                wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog);
                const long long tc0 = pt.b0 + (long long)t * kTileF;
                const int n4 = (int)(min((long long)kTileF, pt.bn - (long long)t * kTileF) >> 2);
                if (ct < n4) {
                    const float4 v = ld_shared_v4(&S.ring[slot][ct * 4]);
                    ms_add4(ms, v);
                    if (OP == kCeFwd) {
                        const long long d = jl - (tc0 + 4 * ct);
                        if (d >= 0 && d < 4) { own_label = true; s_label = pick(v, d); }
                    }
                }
                if (OP == kCeFwd) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.empty[slot]);
                }
            }
            if (OP == kCeFwd) {
                g += nt;
                if (has_head && jl == ct) { own_label = true; s_label = hv; }
                if (has_tail && jl == pt.t0 + ct - 4) { own_label = true; s_label = tv; }
            }
            ms = ms_warp_reduce(ms);
            const uint32_t b = nred & 1u;
            ++nred;
            if (lane == 0) S.wred[b][cw] = make_float2(ms.m, ms.s);
            named_sync(kBarConsumers, NCT);
            MaxSum tot{S.wred[b][0].x, S.wred[b][0].y};
#pragma unroll
            for (int w = 1; w < NCW; ++w) tot = ms_merge(tot, MaxSum{S.wred[b][w].x, S.wred[b][w].y});
            if (c > 1) {
                const uint32_t xb = nx & 1u, xpar = (nx >> 1) & 1u;
                ++nx;
                if (ct == 0) {
                    for (int q = 0; q < c; ++q) {
                        st_cluster_f32x2(map_to_rank(&S.xbuf[xb][rank], (uint32_t)q), tot.m, tot.s);
                        mbar_arrive_remote_release(map_to_rank(&S.xbar[xb], (uint32_t)q));
                    }
                }
                wait_parity<true>(&S.xbar[xb], xpar, &S.abort, &g_watchdog);
                tot = MaxSum{S.xbuf[xb][0].x, S.xbuf[xb][0].y};
                for (int q = 1; q < c; ++q) tot = ms_merge(tot, MaxSum{S.xbuf[xb][q].x, S.xbuf[xb][q].y});
            }
            m = tot.m;
            lnS = logf(tot.s);
            if (rank == 0 && ct == 0) {
                if (P.lse_out) P.lse_out[r] = m + lnS;
                if (P.stats_out) { P.stats_out[2 * r] = m; P.stats_out[2 * r + 1] = lnS; }
            }
        } else {
            if (P.stats_in) { m = P.stats_in[2 * r]; lnS = P.stats_in[2 * r + 1]; }
            else { m = P.lse_in[r]; lnS = 0.f; }
        }

        if (OP == kCeFwd) {
            if (inwin && own_label) P.loss[r] = (m - s_label) + lnS;
            if (rank == 0 && ct == 0) {
                if (!inwin) P.loss[r] = 0.f;
                else if (bad_label) P.loss[r] = __int_as_float(0x7fc00000);
            }
            continue;
        }

        // ---- gradient, written in place from the staged tiles
        const float cg = P.cg;
        float lacc = 0.f;
        uint32_t e_lo = 0;
        if (kKL) while (e_lo < (uint32_t)nsup && (long long)S.scol[e_lo] < pt.b0) ++e_lo;
        for (uint32_t t = 0; t < nt; ++t) {
            const uint32_t gt = g + t, slot = gt % kSlots;
            if (!RES) wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog);
            const long long tc0 = pt.b0 + (long long)t * kTileF;
            const long long n = min((long long)kTileF, pt.bn - (long long)t * kTileF);
            uint32_t e_hi = e_lo;
            if (kKL) while (e_hi < (uint32_t)nsup && (long long)S.scol[e_hi] < tc0 + n) ++e_hi;
            if (ct < (int)(n >> 2)) {
                const long long c0 = tc0 + 4 * ct;
                const float4 v = ld_shared_v4(&S.ring[slot][ct * 4]);
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (inwin) {
                    o.x = cg * soft(v.x, m, lnS);
                    o.y = cg * soft(v.y, m, lnS);
                    o.z = cg * soft(v.z, m, lnS);
                    o.w = cg * soft(v.w, m, lnS);
                    const long long d = jl - c0;
                    if (d >= 0 && d < 4) {
                        sub_at(o, d, P.ce_coef);
                        own_label = true;
                        s_label = pick(v, d);
                    }
                    if (kKL && e_hi > e_lo) kl_apply4(S, e_lo, e_hi, c0, v, o, P.coef, m, lnS, lacc);
                }
                st_global_v4(rowp + c0, o);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            e_lo = e_hi;
        }
        g += nt;

        // head and tail elements (scalar)
        if (has_head || has_tail) {
            const long long j = has_head ? (long long)ct : pt.t0 + ct - 4;
            const float s = has_head ? (RES ? hv : rowp[j]) : (RES ? tv : rowp[j]);
            float o = 0.f;
            if (inwin) {
                o = cg * soft(s, m, lnS);
                if (j == jl) { o -= P.ce_coef; own_label = true; s_label = s; }
                if (kKL) {
                    for (uint32_t e = 0; e < (uint32_t)nsup; ++e) {
                        if ((long long)S.scol[e] == j) {
                            const float p = S.sp[e];
                            o -= P.coef * p;
                            if (p > 0.f) lacc += p * (logf(p) - ((s - m) - lnS));
                        }
                    }
                }
            }
            rowp[j] = o;
        }

        // ---- losses
        if (OP == kCeFused || OP == kCeBwd) {
            if (P.loss) {
                if (inwin && own_label) P.loss[r] = (m - s_label) + lnS;
                if (rank == 0 && ct == 0) {
                    if (!inwin) P.loss[r] = 0.f;
                    else if (bad_label) P.loss[r] = __int_as_float(0x7fc00000);
                    else if (jl < 0 || jl >= P.ncols) P.loss[r] = 0.f;   // label in another slice
                }
            }
        } else if (kKL) {
            lacc = warp_sum(lacc);
            const uint32_t b = nloss & 1u;
            ++nloss;
            if (lane == 0) S.wloss[b][cw] = lacc;
            named_sync(kBarConsumers, NCT);
            if (ct == 0) {
                float L = 0.f;
                for (int w = 0; w < NCW; ++w) L += S.wloss[b][w];
                if (c == 1) {
                    P.loss[r] = L;
                } else {
                    const uint32_t lb = nlx & 1u, lpar = (nlx >> 1) & 1u;
                    ++nlx;
                    st_cluster_f32(map_to_rank(&S.lbuf[lb][rank], 0u), L);
                    mbar_arrive_remote_release(map_to_rank(&S.lbar[lb], 0u));
                    if (rank == 0) {
                        wait_parity<true>(&S.lbar[lb], lpar, &S.abort, &g_watchdog);
                        float T = 0.f;
                        for (int q = 0; q < c; ++q) T += S.lbuf[lb][q];
                        P.loss[r] = T;
                    }
                }
            }
        }
    }
}

template <int OP, bool RES>
__global__ void __launch_bounds__(NTHREADS, 1) row_kernel(const __grid_constant__ RowParams P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int c = P.csize;
    const int rank = c > 1 ? (int)cluster_ctarank() : 0;
    const long long cid = c > 1 ? (long long)cluster_id_x() : (long long)blockIdx.x;
    const long long ncl = c > 1 ? (long long)ncluster_x() : (long long)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.xbar[b], (uint32_t)c);
            mbar_init(&S.lbar[b], (uint32_t)c);
        }
        S.abort = 0;
        S.issued = 0;
        fence_mbar_init_cluster();
    }
    if (c > 1) cluster_sync_all();
    else __syncthreads();
    pdl_launch_dependents();

    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer<OP>(P, S, rank, cid, ncl);
            drain(S);
        }
        __syncwarp();
    } else {
        consumer<OP, RES>(P, S, rank, cid, ncl);
    }
    // no CTA may leave while a peer can still write into its shared memory
    if (c > 1) cluster_sync_all();
}

const void* kernel_for(int op, bool res) {
    switch (op) {
        case kCeFused: return (const void*)row_kernel<kCeFused, true>;
        case kCeFwd: return (const void*)row_kernel<kCeFwd, false>;
        case kCeBwd: return (const void*)row_kernel<kCeBwd, false>;
        case kKl: return res ? (const void*)row_kernel<kKl, true> : (const void*)row_kernel<kKl, false>;
        default: return nullptr;
    }
}

constexpr int kMaxDev = 64;
std::atomic<int> g_attr_done[kMaxDev][8];

cudaError_t prepare(const void* fn, int slot) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (g_attr_done[dev][slot].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    g_attr_done[dev][slot].store(1, std::memory_order_release);
    return cudaSuccess;
}

int slot_of(int op, bool res) { return op * 2 + (res ? 1 : 0); }

}  // namespace

cudaError_t launch_rows(int op, bool resident, const RowParams& P, int nclusters, cudaStream_t st) {
    const void* fn = kernel_for(op, resident);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = prepare(fn, slot_of(op, resident));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclusters * P.csize), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (P.csize > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)P.csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    RowParams p = P;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int row_max_clusters(int op, bool resident, int c) {
    const void* fn = kernel_for(op, resident);
    if (!fn || prepare(fn, slot_of(op, resident)) != cudaSuccess) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (c <= 1) return sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(c * sms), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

unsigned int rows_watchdog(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_watchdog, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_watchdog, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}

}  // namespace vl
