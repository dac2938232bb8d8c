// Row engine: cross-entropy (fused, forward, backward) and top-k KL over rows of
// fp32 vocabulary logits, one persistent CTA (or cluster of CTAs) per SM.
//
// Layout of one launch
//   * grid = nclusters * csize CTAs, one CTA per SM (the ring below takes
//     ~200 KB of shared memory).  Cluster i handles rows i, i + nclusters, ...
//   * a row slice of ncols floats is cut into a <=3-float head, a 16-byte-aligned
//     body and a <=3-float tail.  The body is split evenly (in float4 units)
//     across the csize CTAs of the cluster; CTA rank 0 also takes the head and
//     the last rank the tail.
//   * warp 0 (one lane) is the producer: it streams each CTA's body through a
//     ring of kSlots tiles of kTileF floats with 1-D bulk copies (TMA) signalled
//     on per-slot mbarriers; warps 1..15 are consumers.  A consumer thread owns
//     float4s ct, ct + NCT, ... (kVec of them) of every tile.
//
// Modes
//   self-contained (CE fused, KL without given statistics): the producer streams
//             each row part twice.  Pass A reduces (max, sum of exponentials)
//             online per thread; partials are merged across warps (shared
//             memory) and across the cluster (distributed shared memory: st.async
//             that completes the peer's mbarrier transaction count).  Pass B
//             re-reads the part -- it was read microseconds earlier, so the bytes
//             come from L2 -- and writes the gradient tile by tile.  HBM sees one
//             read and one write per element; no row has to fit on chip.
//   streaming (CE backward, KL with given statistics): pass B only.
//   reduce    (CE forward): pass A only.
//
// Sparse columns (the label, the teacher's top-k ids).  Streaming mode gathers their
// logits from the staged tiles as they pass and rewrites their gradient after the
// bulk store of the row and a barrier.  Self-contained mode folds the label into
// pass B, gathers the support logits from global memory before pass A (the row is
// not written until after it) for the KL loss, and adds -coef * p_q at the support
// columns with reduction adds after a barrier that follows the row's pass B.
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

constexpr int NCW = kConsumerWarps;     // consumer warps
constexpr int NCT = NCW * 32;           // consumer threads
constexpr int NTHREADS = NCT + 32;      // + the producer warp
constexpr int EPT = 3;                  // teacher support entries per consumer thread
constexpr int KMAX = EPT * NCT;         // teacher support per row
constexpr int LT = NCT - 1;             // the consumer thread that handles the label
constexpr int KSELF = 1024;             // teacher support per row, self-contained mode
// A row's support is written before its pass A and scattered two rows later, after
// the barrier that follows its pass B; four buffers keep the writer of row i + 2
// behind the barrier of row i + 1, which every scatter of row i - 2 precedes.
constexpr uint32_t kSupBufs = 4;
constexpr uint32_t kBarConsumers = 1;   // named barrier id used by consumers only
// Self-contained CE hands each warp's pass A partial to the row's pass B through
// kPartBufs buffers and mbarriers, without a CTA barrier.  An mbarrier phase cannot
// come round again before every warp, the waiter included, has arrived for it.  A
// buffer's data is rewritten kPartBufs rows later; when every row has at least one
// body tile per pass, a warp that far ahead of another would hold 2 kPartBufs - 2
// tiles more than it, which the kSlots-tile ring does not allow.
constexpr uint32_t kPartBufs = 8;
static_assert(2 * kPartBufs - 2 > kSlots, "partial buffers outlast the ring");

static_assert(kTileF / 4 == NCT * kVec, "kVec float4s of each tile per consumer thread");
static_assert(KMAX >= 1024, "the C ABI promises k <= 1024");

__device__ unsigned int g_watchdog;

struct alignas(128) Smem {
    float ring[kSlots][kTileF];
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t xbar[4];                   // cluster exchange of (max, sum)
    uint64_t lbar[2];                   // cluster exchange of KL loss parts (rank 0)
    float4 xbuf[4][kMaxCluster];        // (max, sum, KL a, KL b) of each rank's part
    float lbuf[2][kMaxCluster];
    float4 wred[2][NCW];                // per warp: (max, sum, KL a, KL b)
    uint64_t abar[kPartBufs];           // self-contained CE: every warp's pass A partial is in
    float2 wpart[kPartBufs][NCW];
    float wloss[2][NCW];
    union {
        struct {                        // streaming mode: support of the current row
            alignas(16) int kcol[2][KMAX];   // column (slice-relative) per entry, -1 outside this CTA
            float kp[2][KMAX];               // probability per entry
            float ks[2][KMAX];               // the logit at that column, gathered as its tile passes
        };
        struct {                        // self-contained mode: support of the last kSupBufs rows
            int ecol[kSupBufs][KSELF];       // support column (slice-relative; -1 elsewhere)
            float ep[kSupBufs][KSELF];
        };
    };
    int abort;
    uint32_t issued;
};

static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");

// Columns of one row slice handled by CTA `rank` of `c` (relative to the slice start).
struct Part {
    int h;     // head length (first columns up to the 16-byte boundary)
    int hn;    // head columns this CTA handles
    int b0;    // first body column of this CTA
    int bn;    // body columns of this CTA (a multiple of 4)
    int t0;    // first tail column
    int tn;    // tail columns this CTA handles
    int lo;    // this CTA owns columns [lo, hi)
    int hi;
};

__device__ __forceinline__ Part part_of(const float* rowp, int n, int rank, int c) {
    Part p;
    const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
    int h = (4 - mis) & 3;
    if (h > n) h = n;
    const int bt = (n - h) & ~3;
    const int per = (((bt >> 2) + c - 1) / c) * 4;
    const int s = min(rank * per, bt);
    const int e = min((rank + 1) * per, bt);
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

// Columns of units [u0, u1) of a row slice of n floats, cut into U = ceil(n / 4) units:
// unit u is body float4 min(u, nb4) (nb4 body float4s after the head); the head goes
// with the part that starts at unit 0, the tail with the part that ends at unit U.
// The parts of any partition of [0, U) cover the row exactly once.
__device__ __forceinline__ Part part_units(const float* rowp, int n, int U, int u0, int u1) {
    Part p;
    const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
    int h = (4 - mis) & 3;
    if (h > n) h = n;
    const int nb4 = (n - h) >> 2;
    const int f0 = min(u0, nb4), f1 = min(u1, nb4);
    p.h = h;
    p.hn = u0 == 0 ? h : 0;
    p.b0 = h + 4 * f0;
    p.bn = 4 * (f1 - f0);
    p.t0 = h + 4 * nb4;
    p.tn = u1 == U ? n - p.t0 : 0;
    p.lo = u0 == 0 ? 0 : p.b0;
    p.hi = u1 == U ? n : p.b0 + p.bn;
    return p;
}

// ---------------------------------------------------------------- tail split
//
// With G CTAs and R rows, every CTA first takes q = R / G whole rows (b, b + G, ...).
// The T = R - qG rows left over are not given whole to T of the CTAs (which would leave
// the others idle for a row's time): their units, T * U in all, are cut into G equal
// ranges, CTA b taking units [b TU / G, (b + 1) TU / G).  A range is shorter than a
// row, so it touches at most two rows: the CTA's tail segments 0 and 1.  A segment's
// (max, sum) is published in the workspace; before a segment's pass B its CTA merges
// the parts of the row from every CTA that holds one, in CTA order, so that all of
// them use bit-identical row statistics.
//
// Workspace words: [0] generation, [1] ticket, then slot (b, s) at word
// 4 + 4 (2b + s) = {max, sum, sequence, -}.  A launch reads the generation g at its
// start and marks its slots with sequence g + 1; the last CTA to finish (ticket)
// advances the generation, so a launch never reads a slot left by an earlier one.

struct Item {
    long long r;     // row
    int u0, u1;      // units [u0, u1) of the row
    int which;       // -1: a whole row; 0 / 1: this CTA's first / second tail segment
    long long j;     // tail row index (which >= 0)
};

__device__ __forceinline__ bool item_at(const RowParams& P, long long i, int U, Item& it) {
    const long long G = gridDim.x, b = blockIdx.x;
    const long long q = P.ntok / G;
    if (i < q) {
        it.r = b + i * G;
        it.u0 = 0;
        it.u1 = U;
        it.which = -1;
        it.j = -1;
        return true;
    }
    const long long TU = (P.ntok - q * G) * (long long)U;
    const long long lo = b * TU / G, hi = (b + 1) * TU / G;
    if (lo >= hi) return false;
    const long long j0 = lo / U, j1 = (hi - 1) / U;
    if (i == q) {
        it.j = j0;
        it.u0 = (int)(lo - j0 * U);
        it.u1 = (int)(min(hi, (j0 + 1) * U) - j0 * U);
    } else if (i == q + 1 && j1 > j0) {
        it.j = j1;
        it.u0 = 0;
        it.u1 = (int)(hi - j1 * U);
    } else {
        return false;
    }
    it.which = (int)(i - q);
    it.r = q * G + it.j;
    return true;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned int* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int* ws_slot(const RowParams& P, long long b, int which) {
    return P.ws + kWsHeaderWords + 4 * (2 * b + which);
}

// This CTA's (max, sum) of tail segment `which`, for the other parts of its row.
__device__ __forceinline__ void publish_part(const RowParams& P, int which, MaxSum ms, uint32_t epoch) {
    unsigned int* sl = ws_slot(P, blockIdx.x, which);
    asm volatile("st.global.cg.v2.f32 [%0], {%1, %2};" :: "l"(sl), "f"(ms.m), "f"(ms.s) : "memory");
    st_release_u32(sl + 2, epoch);
}

template <int OP>
__device__ __forceinline__ bool row_loaded(const RowParams& P, long long r) {
    if (OP == kCeFused || OP == kCeFwd) return true;    // lse is produced for every row
    return r >= P.ls && r < P.le;
}

// softmax value from the row statistics: exp((s - m) - lnS)
__device__ __forceinline__ float soft(float s, float m, float lnS) {
    return ex2(((s - m) - lnS) * kLog2e);
}

__device__ __forceinline__ void sub_at(float4& o, unsigned d, float a) {
    if (d == 0) o.x -= a;
    else if (d == 1) o.y -= a;
    else if (d == 2) o.z -= a;
    else o.w -= a;
}

// (max, sum) update with kVec float4s (absent values are -inf): one max update,
// independent exponentials summed as a tree.
__device__ __forceinline__ void ms_addv(MaxSum& a, const float4 (&v)[kVec]) {
    float mx = fmaxf(fmaxf(v[0].x, v[0].y), fmaxf(v[0].z, v[0].w));
#pragma unroll
    for (int u = 1; u < kVec; ++u) mx = fmaxf(mx, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
    if (mx > a.m) {
        a.s *= ex2((a.m - mx) * kLog2e);
        a.m = mx;
    }
    float e[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u)
        e[u] = (ex2((v[u].x - a.m) * kLog2e) + ex2((v[u].y - a.m) * kLog2e)) +
               (ex2((v[u].z - a.m) * kLog2e) + ex2((v[u].w - a.m) * kLog2e));
    float t = e[0];
#pragma unroll
    for (int u = 1; u < kVec; ++u) t += e[u];
    a.s += t;
}

// ---------------------------------------------------------------- producer

// Issue the body tiles of one row part; false if a wait gave up.
__device__ __forceinline__ bool issue_body(const RowParams& P, Smem& S, const float* rowp, const Part& pt,
                                           uint32_t& g) {
    for (int c0 = 0; c0 < pt.bn; c0 += kTileF) {
        // test hook: CTA 0 stops before this tile, so the consumers' wait for it runs out
        if ((long long)g == P.withhold && blockIdx.x == 0) return false;
        const uint32_t slot = g % kSlots, use = g / kSlots;
        if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog, P.wait_limit)) return false;
        const uint32_t bytes = (uint32_t)min(kTileF, pt.bn - c0) * 4u;
        mbar_arrive_expect_tx(&S.full[slot], bytes);
        bulk_g2s(S.ring[slot], rowp + pt.b0 + c0, bytes, &S.full[slot]);
        ++g;
    }
    return true;
}

__device__ __forceinline__ bool issue_part(const RowParams& P, Smem& S, long long r, int rank, uint32_t& g) {
    const float* rowp = P.x + r * P.ld + P.col0;
    return issue_body(P, S, rowp, part_of(rowp, (int)P.ncols, rank, P.csize), g);
}

__device__ __forceinline__ bool issue_item(const RowParams& P, Smem& S, const Item& it, int U, uint32_t& g) {
    const float* rowp = P.x + it.r * P.ld + P.col0;
    return issue_body(P, S, rowp, part_units(rowp, (int)P.ncols, U, it.u0, it.u1), g);
}

// Tail split: the items (whole rows, then tail segments) in the two-pass order.
__device__ void producer_split(const RowParams& P, Smem& S) {
    const int U = (int)((P.ncols + 3) >> 2);
    uint32_t g = 0;
    Item it, prev;
    bool have_prev = false, ok = true;
    for (long long i = 0; ok && item_at(P, i, U, it); ++i) {
        ok = issue_item(P, S, it, U, g);
        if (ok && have_prev) ok = issue_item(P, S, prev, U, g);
        prev = it;
        have_prev = true;
    }
    if (ok && have_prev && !S.abort) issue_item(P, S, prev, U, g);
    S.issued = g;
}

// Tile order: one pass per row for the streaming and reduce modes; for the
// self-contained mode pass A of a row, then pass B of the row before it, so the
// reads of the next row are in flight while the current one is written.
template <int OP, bool RES>
__device__ void producer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    uint32_t g = 0;
    long long prev = -1;
    for (long long r = cid; r < P.ntok; r += ncl) {
        if (!row_loaded<OP>(P, r)) continue;
        if (!issue_part(P, S, r, rank, g)) break;
        if (RES) {
            if (prev >= 0 && !issue_part(P, S, prev, rank, g)) break;
            prev = r;
        }
    }
    if (RES && prev >= 0 && !S.abort) issue_part(P, S, prev, rank, g);
    S.issued = g;
}

// Before the CTA exits, every bulk copy it issued must have landed.
__device__ void drain(Smem& S, long long limit) {
    const uint32_t iss = S.issued;
    for (uint32_t gt = iss > (uint32_t)kSlots ? iss - kSlots : 0u; gt < iss; ++gt)
        wait_parity_drain(&S.full[gt % kSlots], (gt / kSlots) & 1u, limit);
}

// ---------------------------------------------------------------- consumer helpers

__device__ void zero_part(float* rowp, const Part& pt, int ct) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = ct; i < (pt.bn >> 2); i += NCT) st_global_v4(rowp + pt.b0 + 4 * i, z);
    if (ct < pt.hn) rowp[ct] = 0.f;
    if (ct >= 4 && ct - 4 < pt.tn) rowp[pt.t0 + ct - 4] = 0.f;
}

// A sparse column this thread looks after: where it sits in the row part, and its
// logit once the tile holding it has passed.
struct Sparse {
    int col;     // slice-relative column, -1 if none
    int rel;     // column - b0 inside this CTA's body (tile = rel / kTileF), -1 for head/tail
    float s;     // the logit
};

__device__ __forceinline__ void locate(Sparse& e, const Part& pt, const float* rowp) {
    if (e.col >= pt.b0 && e.col < pt.b0 + pt.bn) {
        e.rel = e.col - pt.b0;
    } else {
        e.rel = -1;
        e.s = rowp[e.col];     // head or tail: read before anything of the row is written
    }
}

__device__ __forceinline__ void gather(Sparse& e, int t, const float* tile) {
    if (e.rel >= 0 && (e.rel / kTileF) == t) e.s = tile[e.rel % kTileF];
}

__device__ __forceinline__ void gather_support(Smem& S, uint32_t kb, const int (&erel)[EPT], int ct, int t,
                                               const float* tile) {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
        if (erel[i] >= 0 && erel[i] / kTileF == t) S.ks[kb][ct + i * NCT] = tile[erel[i] % kTileF];
}

// (max, sum) of n partials: the max first, then the sums rescaled independently.
__device__ __forceinline__ MaxSum combine(const float2* part, int n) {
    float M = part[0].x;
    for (int i = 1; i < n; ++i) M = fmaxf(M, part[i].x);
    float T = 0.f;
    for (int i = 0; i < n; ++i) T += part[i].y * ex2((part[i].x - M) * kLog2e);
    return MaxSum{M, T};
}

// Row partials with the KL loss parts: (max, sum) combined as above, and the sums
// a = sum p (ln p - s), b = sum p over the teacher support entries the parts hold.
// KL = sum p (ln p - (s - lse)) = a + lse * b, so the loss needs no statistics until
// the parts meet.
struct Part4 {
    MaxSum ms;
    float a, b;
};

__device__ __forceinline__ Part4 combine4(const float4* part, int n) {
    float M = part[0].x;
    for (int i = 1; i < n; ++i) M = fmaxf(M, part[i].x);
    float T = 0.f, A = 0.f, B = 0.f;
    for (int i = 0; i < n; ++i) {
        T += part[i].y * ex2((part[i].x - M) * kLog2e);
        A += part[i].z;
        B += part[i].w;
    }
    return Part4{MaxSum{M, T}, A, B};
}

// ---------------------------------------------------------------- consumer

template <int OP, bool RES>
__device__ void consumer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    constexpr bool kKL = OP == kKl;
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int c = P.csize;
    const int ncols = (int)P.ncols;
    uint32_t g = 0, nred = 0, nloss = 0, nlx = 0, nrow = 0;
    const bool has_label = (OP != kKl) || (P.labels != nullptr && P.ce_coef != 0.f);
    const float cg = P.cg;
    // the label and support entry q = ct of the next row, loaded one row ahead
    uint32_t nlab = 0, nid = 0;
    float np = 0.f;
    auto prefetch = [&](long long rr) {
        if (rr >= P.ntok) return;
        if (has_label) nlab = P.labels[rr];
        if (kKL && ct < P.k) { nid = P.tid[rr * P.k + ct]; np = P.tp[rr * P.k + ct]; }
    };
    prefetch(cid);

    for (long long r = cid; r < P.ntok; r += ncl) {
        const uint32_t lab_r = nlab, id0 = nid;
        const float p0 = np;
        prefetch(r + ncl);
        float* rowp = P.x + r * P.ld + P.col0;
        const Part pt = part_of(rowp, ncols, rank, c);
        const bool inwin = r >= P.ls && r < P.le;
        const int nt = (pt.bn + kTileF - 1) / kTileF;
        if (!row_loaded<OP>(P, r)) {
            zero_part(rowp, pt, ct);
            if (ct == 0 && rank == 0 && P.loss) P.loss[r] = 0.f;
            continue;
        }
        const uint32_t kb = nrow & 1u;
        ++nrow;

        // ---- the label: its slice column jl (every thread), its logit (thread LT);
        //      the teacher support: entry q on thread q % NCT
        int jl = -1;
        bool bad_label = false;
        if (has_label) {
            const uint32_t l = lab_r;
            if ((long long)l >= P.V) bad_label = true;
            else if ((long long)l >= P.col0 && (long long)l < P.col0 + ncols) jl = (int)((long long)l - P.col0);
        }
        if (bad_label && inwin && rank == 0 && ct == LT && P.err) atomicAdd(P.err, 1);
        Sparse lab{-1, -1, 0.f};
        if (ct == LT && jl >= pt.lo && jl < pt.hi) { lab.col = jl; locate(lab, pt, rowp); }
        // support entry q = ct + i * NCT: its body offset in erel[i] (-1: head/tail or none)
        int erel[EPT] = {-1, -1, -1};
        if (kKL && inwin) {
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int q = ct + i * NCT;
                if (q < P.k) {
                    const uint32_t id = i == 0 ? id0 : P.tid[r * P.k + q];
                    int col = -1;
                    if ((long long)id >= P.V) {
                        if (rank == 0 && P.err) atomicAdd(P.err, 1);
                    } else {
                        const long long j = (long long)id - P.col0;
                        if (j >= pt.lo && j < pt.hi) col = (int)j;
                    }
                    S.kcol[kb][q] = col;
                    S.kp[kb][q] = i == 0 ? p0 : P.tp[r * P.k + q];
                    if (col >= 0) {
                        if (col >= pt.b0 && col < pt.b0 + pt.bn) erel[i] = col - pt.b0;
                        else S.ks[kb][q] = rowp[col];    // head or tail: before anything is written
                    }
                }
            }
        }

        // head and tail columns: one per thread, finished after the sparse barrier
        const bool has_ht = ct < pt.hn || (ct >= 4 && ct - 4 < pt.tn);
        const int jht = ct < pt.hn ? ct : pt.t0 + ct - 4;
        const float ht = has_ht ? rowp[jht] : 0.f;
        float m, lnS;

        if (OP == kCeFwd || RES) {
            // ---- pass A: (max, sum) online over the streamed tiles; sparse logits gathered
            MaxSum ms = ms_empty();
            if (has_ht) ms_add(ms, ht);
            for (int t = 0; t < nt; ++t) {
                const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
                wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
                const int n4 = min(kTileF, pt.bn - t * kTileF) >> 2;
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int j = u * NCT + ct;
                    if (j < n4) ms_add4(ms, ld_shared_v4(&S.ring[slot][j * 4]));
                }
                if (kKL) gather_support(S, kb, erel, ct, t, S.ring[slot]);
                if (ct == LT) gather(lab, t, S.ring[slot]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            g += (uint32_t)nt;
            ms = ms_warp_reduce(ms);
            const uint32_t b = nred & 1u;
            ++nred;
            if (lane == 0) S.wred[b][cw] = make_float4(ms.m, ms.s, 0.f, 0.f);
            named_sync(kBarConsumers, NCT);
            const MaxSum tot = combine4(S.wred[b], NCW).ms;
            m = tot.m;
            lnS = logf(tot.s);
            if (rank == 0 && ct == LT) {
                if (P.lse_out) P.lse_out[r] = m + lnS;
                if (P.stats_out) { P.stats_out[2 * r] = m; P.stats_out[2 * r + 1] = lnS; }
            }
            if (OP == kCeFwd) {
                if (ct == LT) {
                    if (!inwin) P.loss[r] = 0.f;
                    else if (bad_label) P.loss[r] = __int_as_float(0x7fc00000);
                    else if (lab.col >= 0) P.loss[r] = (m - lab.s) + lnS;
                }
                continue;
            }
        } else {
            if (P.stats_in) { m = P.stats_in[2 * r]; lnS = P.stats_in[2 * r + 1]; }
            else { m = P.lse_in[r]; lnS = 0.f; }
        }

        // ---- pass B: each tile turned into gradient as it lands (zeros outside the window)
        {
            const float c1 = inwin ? cg : 0.f;
            // c1 * exp(d - lnS) = 2^(d * log2e - K), K = lnS * log2e - log2(c1), for c1 >= 0
            const bool fold = c1 >= 0.f;
            const float K = fold ? lnS * kLog2e - log2f(c1) : 0.f;
            const uint64_t pol = l2_evict_first();
            for (int t = 0; t < nt; ++t) {
                const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
                wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
                const int n4 = min(kTileF, pt.bn - t * kTileF) >> 2;
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int j = u * NCT + ct;
                    if (j < n4) {
                        const float4 x = ld_shared_v4(&S.ring[slot][j * 4]);
                        float4 o;
                        if (fold) {
                            o = make_float4(ex2(fmaf(x.x - m, kLog2e, -K)), ex2(fmaf(x.y - m, kLog2e, -K)),
                                            ex2(fmaf(x.z - m, kLog2e, -K)), ex2(fmaf(x.w - m, kLog2e, -K)));
                        } else {
                            o = make_float4(c1 * soft(x.x, m, lnS), c1 * soft(x.y, m, lnS),
                                            c1 * soft(x.z, m, lnS), c1 * soft(x.w, m, lnS));
                        }
                        st_global_v4_hint(rowp + pt.b0 + t * kTileF + 4 * j, o, pol);
                    }
                }
                if (!RES) {
                    if (kKL) gather_support(S, kb, erel, ct, t, S.ring[slot]);
                    if (ct == LT) gather(lab, t, S.ring[slot]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            g += (uint32_t)nt;
        }

        // ---- sparse columns, once every bulk store of the row is done: the label,
        //      the support ids, and the head/tail columns with their corrections
        named_sync(kBarConsumers, NCT);
        float lacc = 0.f;
        if (has_ht) {
            float o = 0.f;
            if (inwin) {
                o = cg * soft(ht, m, lnS);
                if (kKL)
                    for (int j = 0; j < P.k; ++j)
                        if (S.kcol[kb][j] == jht) o -= P.coef * S.kp[kb][j];
                if (jht == jl) o -= P.ce_coef;
            }
            rowp[jht] = o;
        }
        if (inwin) {
            if (kKL) {
#pragma unroll
                for (int i = 0; i < EPT; ++i) {
                    const int q = ct + i * NCT;
                    if (q >= P.k) continue;
                    const int col = S.kcol[kb][q];
                    if (col < 0) continue;
                    const float pq = S.kp[kb][q], sq = S.ks[kb][q];
                    if (pq > 0.f) lacc += pq * (logf(pq) - ((sq - m) - lnS));
                    if (erel[i] < 0) continue;         // head/tail columns: finished above
                    // repeated ids: the lowest q writes the column, with every entry's p
                    bool first = true;
                    float psum = 0.f;
                    const int4* kc4 = reinterpret_cast<const int4*>(S.kcol[kb]);
                    for (int j4 = 0; j4 < (P.k + 3) >> 2; ++j4) {
                        const int4 cc = kc4[j4];
                        const int j = 4 * j4;
                        if (cc.x == col && j < P.k) { first &= j >= q; psum += S.kp[kb][j]; }
                        if (cc.y == col && j + 1 < P.k) { first &= j + 1 >= q; psum += S.kp[kb][j + 1]; }
                        if (cc.z == col && j + 2 < P.k) { first &= j + 2 >= q; psum += S.kp[kb][j + 2]; }
                        if (cc.w == col && j + 3 < P.k) { first &= j + 3 >= q; psum += S.kp[kb][j + 3]; }
                    }
                    if (first) {
                        float o = cg * soft(sq, m, lnS) - P.coef * psum;
                        if (col == jl) o -= P.ce_coef;
                        rowp[col] = o;
                    }
                }
            }
            if (ct == LT && lab.col >= 0 && lab.rel >= 0) {
                bool in_support = false;
                if (kKL)
                    for (int j = 0; j < P.k; ++j) in_support |= S.kcol[kb][j] == lab.col;
                if (!in_support) rowp[lab.col] = cg * soft(lab.s, m, lnS) - P.ce_coef;
            }
        }

        // ---- losses
        if (OP == kCeFused || OP == kCeBwd) {
            if (P.loss) {
                if (ct == LT && inwin && lab.col >= 0) P.loss[r] = (m - lab.s) + lnS;
                if (rank == 0 && ct == LT) {
                    if (!inwin) P.loss[r] = 0.f;
                    else if (bad_label) P.loss[r] = __int_as_float(0x7fc00000);
                    else if (jl < 0) P.loss[r] = 0.f;   // the label lies in another slice
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
                    if (rank == 0) mbar_arrive_expect_tx(&S.lbar[lb], 4u * (uint32_t)c);
                    st_async_f32(map_to_rank(&S.lbuf[lb][rank], 0u), L, map_to_rank(&S.lbar[lb], 0u));
                    if (rank == 0) {
                        wait_parity<true>(&S.lbar[lb], lpar, &S.abort, &g_watchdog, P.wait_limit);
                        float T = 0.f;
                        for (int q = 0; q < c; ++q) T += S.lbuf[lb][q];
                        P.loss[r] = T;
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- self-contained consumer

// A row whose pass A is done and whose pass B is still to come.
struct Pending {
    long long r;
    float* rowp;
    Part pt;
    int nt;
    bool inwin, bad;
    int jl;          // slice-relative label column, -1 when none or outside this CTA's columns
    float m, lnS;
    bool has_ht;
    int jht;
    float ht;
    uint32_t xb, xpar;   // cluster exchange buffer of its statistics and the phase to wait for
    uint32_t ab, apar;   // CE: buffer of the warps' pass A partials and the phase to wait for
    bool first;          // this part holds column 0 of the row: it writes lse, stats, out-of-window loss
    int which;           // tail split: -1 whole row, else the tail segment
    long long j;         // tail split: tail row index
};

// Pass B of a row whose statistics are known: the gradient tile by tile with the
// label's one-hot folded in.  The teacher support is left to scatter_support.
template <int OP>
__device__ __forceinline__ void pass_b(const RowParams& P, Smem& S, const Pending& w, uint32_t& g, int ct, int lane) {
    // the CE loss: the fused CE output, or beside the KL when labels come with it
    float* const ce_out = OP == kCeFused ? P.loss : OP == kKl ? P.ce_loss : nullptr;
    const float c1 = w.inwin ? P.cg : 0.f;
    // c1 * exp(d - lnS) = 2^(d * log2e - K) with K = lnS * log2e - log2(c1), for c1 >= 0
    const bool fold = c1 >= 0.f;
    // the gradient lines are done with: written back first, ahead of the logits that
    // pass B of the next row still re-reads from L2
    const uint64_t pol = l2_evict_first();
    const float K = fold ? w.lnS * kLog2e - log2f(c1) : 0.f;
    for (int t = 0; t < w.nt; ++t) {
        const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
        wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
        const int n4 = min(kTileF, w.pt.bn - t * kTileF) >> 2;
        float4 v[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int j = u * NCT + ct;
            if (j < n4) v[u] = ld_shared_v4(&S.ring[slot][j * 4]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int j = u * NCT + ct;
            if (j < n4) {
                const int c0 = w.pt.b0 + t * kTileF + 4 * j;
                const float4 x = v[u];
                float4 o;
                if (fold) {
                    o = make_float4(ex2(fmaf(x.x - w.m, kLog2e, -K)), ex2(fmaf(x.y - w.m, kLog2e, -K)),
                                    ex2(fmaf(x.z - w.m, kLog2e, -K)), ex2(fmaf(x.w - w.m, kLog2e, -K)));
                } else {
                    o = make_float4(c1 * soft(x.x, w.m, w.lnS), c1 * soft(x.y, w.m, w.lnS),
                                    c1 * soft(x.z, w.m, w.lnS), c1 * soft(x.w, w.m, w.lnS));
                }
                if (w.inwin) {
                    const unsigned d = (unsigned)(w.jl - c0);
                    if (d < 4u) {
                        const float xs = d == 0 ? x.x : d == 1 ? x.y : d == 2 ? x.z : x.w;
                        sub_at(o, d, P.ce_coef);
                        if (ce_out) ce_out[w.r] = (w.m - xs) + w.lnS;
                    }
                }
                st_global_v4_hint(w.rowp + c0, o, pol);
            }
        }
    }
    g += (uint32_t)w.nt;
    if (w.has_ht) {
        float o = c1 * soft(w.ht, w.m, w.lnS);
        if (w.inwin && w.jht == w.jl) {
            o -= P.ce_coef;
            if (ce_out) ce_out[w.r] = (w.m - w.ht) + w.lnS;
        }
        w.rowp[w.jht] = o;
    }
    if (ce_out && w.first && ct == LT) {
        if (!w.inwin) ce_out[w.r] = 0.f;
        else if (w.bad) ce_out[w.r] = __int_as_float(0x7fc00000);
    }
}

// Self-contained CE, one CTA per row: the row's statistics from the warps' partials.
__device__ __forceinline__ void collect(const RowParams& P, Smem& S, Pending& w, int ct) {
    wait_parity<false>(&S.abar[w.ab], w.apar, &S.abort, &g_watchdog, P.wait_limit);
    const MaxSum tot = combine(S.wpart[w.ab], NCW);
    w.m = tot.m;
    w.lnS = logf(tot.s);
    if (ct == LT) {
        if (P.lse_out) P.lse_out[w.r] = w.m + w.lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = w.m; P.stats_out[2 * w.r + 1] = w.lnS; }
    }
}

// Cluster mode: the row's statistics (and KL loss parts) from every rank's part, sent
// after its pass A.  Every rank combines the parts in rank order: the same bits.
template <int OP>
__device__ __forceinline__ void settle(const RowParams& P, Smem& S, Pending& w, int ct, int rank) {
    wait_parity<true>(&S.xbar[w.xb], w.xpar, &S.abort, &g_watchdog, P.wait_limit);
    const Part4 tot = combine4(S.xbuf[w.xb], P.csize);
    w.m = tot.ms.m;
    w.lnS = logf(tot.ms.s);
    if (rank == 0 && ct == LT) {
        if (P.lse_out) P.lse_out[w.r] = w.m + w.lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = w.m; P.stats_out[2 * w.r + 1] = w.lnS; }
        if (OP == kKl) P.loss[w.r] = fmaf(w.m + w.lnS, tot.b, tot.a);
    }
}

// -coef * p_q added at every support column of loaded row r (buffer sb).  Reduction
// adds, so repeated ids sum.  Runs after a barrier that follows the row's pass B:
// the barrier orders every thread's gradient store before these adds.
__device__ __forceinline__ void scatter_support(const RowParams& P, const Smem& S, long long r, uint32_t sb, int ct) {
    float* rowp = P.x + r * P.ld + P.col0;
    for (int q = ct; q < P.k; q += NCT) {
        const int col = S.ecol[sb][q];
        if (col >= 0) atomicAdd(rowp + col, -P.coef * S.ep[sb][q]);
    }
}

template <int OP>
__device__ void consumer_self(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    constexpr bool kKL = OP == kKl;
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int c = P.csize;
    const int ncols = (int)P.ncols;
    const bool has_label = (OP != kKl) || P.labels != nullptr;
    // barrier-free statistics (CE, one CTA per row, every row at least one body tile)
    const bool nobar = !kKL && c == 1 && ncols >= 8;
    uint32_t g = 0, nred = 0, nx = 0, li = 0;
    long long rk1 = -1, rk2 = -1;      // KL: the last two loaded rows (loss, support scatter owed)
    uint32_t nlab = 0, nid = 0;
    float np = 0.f;
    auto prefetch = [&](long long rr) {
        if (rr >= P.ntok) return;
        if (has_label) nlab = P.labels[rr];
        if (kKL && ct < P.k) { nid = P.tid[rr * P.k + ct]; np = P.tp[rr * P.k + ct]; }
    };
    prefetch(cid);
    Pending pend;
    pend.r = -1;

    for (long long r = cid; r < P.ntok; r += ncl) {
        const uint32_t lab_r = nlab, id0 = nid;
        const float p0 = np;
        prefetch(r + ncl);
        float* rowp = P.x + r * P.ld + P.col0;
        const Part pt = part_of(rowp, ncols, rank, c);
        const bool inwin = r >= P.ls && r < P.le;
        if (!row_loaded<OP>(P, r)) {
            zero_part(rowp, pt, ct);
            if (ct == 0 && rank == 0) {
                P.loss[r] = 0.f;
                if (P.ce_loss) P.ce_loss[r] = 0.f;
            }
            continue;
        }
        const uint32_t sb = li % kSupBufs;
        Pending cur;
        cur.r = r;
        cur.rowp = rowp;
        cur.pt = pt;
        cur.nt = (pt.bn + kTileF - 1) / kTileF;
        cur.inwin = inwin;
        cur.first = rank == 0;
        cur.which = -1;
        cur.j = -1;
        cur.jl = -1;
        cur.bad = false;
        if (has_label) {
            if ((long long)lab_r >= P.V) cur.bad = true;
            else {
                const long long j = (long long)lab_r - P.col0;
                if (j >= pt.lo && j < pt.hi) cur.jl = (int)j;
            }
        }
        if (cur.bad && inwin && rank == 0 && ct == LT && P.err) atomicAdd(P.err, 1);
        // teacher support entries q = ct + i * NCT: column and probability to shared
        // memory for the scatter, the logit gathered now -- nothing of the row is
        // written before the barrier that ends its pass A -- for the loss
        int scol[EPT];
        float sp[EPT], sx[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            scol[i] = -1;
            sp[i] = 0.f;
            sx[i] = 0.f;
        }
        if (kKL) {
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int q = ct + i * NCT;
                if (q < P.k) {
                    const uint32_t id = i == 0 ? id0 : P.tid[r * P.k + q];
                    const float p = i == 0 ? p0 : P.tp[r * P.k + q];
                    int col = -1;
                    if ((long long)id >= P.V) {
                        if (rank == 0 && P.err) atomicAdd(P.err, 1);
                    } else {
                        const long long j = (long long)id - P.col0;
                        if (j >= pt.lo && j < pt.hi) col = (int)j;
                    }
                    S.ecol[sb][q] = col;
                    S.ep[sb][q] = p;
                    scol[i] = col;
                    sp[i] = p;
                    if (col >= 0) sx[i] = rowp[col];
                }
            }
        }
        // KL loss parts of the support entries this thread holds: a = sum p (ln p - s),
        // b = sum p (the loss is a + lse * b; entries with p <= 0 add no term)
        float ka = 0.f, kb = 0.f;
        if (kKL) {
#pragma unroll
            for (int i = 0; i < EPT; ++i)
                if (scol[i] >= 0 && sp[i] > 0.f) {
                    ka += sp[i] * (logf(sp[i]) - sx[i]);
                    kb += sp[i];
                }
        }
        cur.has_ht = ct < pt.hn || (ct >= 4 && ct - 4 < pt.tn);
        cur.jht = ct < pt.hn ? ct : pt.t0 + ct - 4;
        cur.ht = cur.has_ht ? rowp[cur.jht] : 0.f;

        // ---- pass A: (max, sum) online over the streamed tiles
        MaxSum ms = ms_empty();
        if (cur.has_ht) ms_add(ms, cur.ht);
        for (int t = 0; t < cur.nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
            wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
            const int n4 = min(kTileF, pt.bn - t * kTileF) >> 2;
            float4 v[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int j = u * NCT + ct;
                v[u] = j < n4 ? ld_shared_v4(&S.ring[slot][j * 4]) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            ms_addv(ms, v);
        }
        g += (uint32_t)cur.nt;
        ms = ms_warp_reduce(ms);
        if (nobar) {
            // CE: publish this warp's partial and move on; the row's statistics are
            // collected just before its pass B, one row later, when every warp has long
            // arrived -- no CTA-wide barrier per row
            cur.ab = nred % kPartBufs;
            cur.apar = (nred / kPartBufs) & 1u;
            ++nred;
            if (lane == 0) {
                S.wpart[cur.ab][cw] = make_float2(ms.m, ms.s);
                mbar_arrive(&S.abar[cur.ab]);
            }
            if (pend.r >= 0) {
                collect(P, S, pend, ct);
                pass_b<OP>(P, S, pend, g, ct, lane);
            }
            pend = cur;
            rk2 = rk1;
            rk1 = r;
            ++li;
            continue;
        }
        const uint32_t b = nred & 1u;
        ++nred;
        if (kKL) {
            ka = warp_sum(ka);
            kb = warp_sum(kb);
        }
        if (lane == 0) S.wred[b][cw] = make_float4(ms.m, ms.s, ka, kb);
        named_sync(kBarConsumers, NCT);
        const Part4 tot = combine4(S.wred[b], NCW);
        if (c > 1) {
            // send this CTA's part to every rank; the parts are collected just before this
            // row's pass B, one row later, so the exchange overlaps the next pass A.  Four
            // buffers: a peer writes buffer i + 4 only after its own collection of row
            // i + 2, which needs this CTA's part of row i + 2, sent after row i was read.
            cur.xb = nx & 3u;
            cur.xpar = (nx >> 2) & 1u;
            ++nx;
            if (ct == 0) {
                mbar_arrive_expect_tx(&S.xbar[cur.xb], 16u * (uint32_t)c);
                const float4 mine = make_float4(tot.ms.m, tot.ms.s, tot.a, tot.b);
                for (int q = 0; q < c; ++q)
                    st_async_f32x4(map_to_rank(&S.xbuf[cur.xb][rank], (uint32_t)q), mine,
                                   map_to_rank(&S.xbar[cur.xb], (uint32_t)q));
            }
        } else {
            cur.m = tot.ms.m;
            cur.lnS = logf(tot.ms.s);
            if (ct == LT) {
                if (P.lse_out) P.lse_out[r] = cur.m + cur.lnS;
                if (P.stats_out) { P.stats_out[2 * r] = cur.m; P.stats_out[2 * r + 1] = cur.lnS; }
                if (kKL) P.loss[r] = fmaf(cur.m + cur.lnS, tot.b, tot.a);
            }
        }
        // past this row's barrier, pass B of the row two back is done: its support terms
        if (kKL && rk2 >= 0) scatter_support(P, S, rk2, (li + kSupBufs - 2u) % kSupBufs, ct);
        // ---- pass B of the previous row
        if (pend.r >= 0) {
            if (c > 1) settle<OP>(P, S, pend, ct, rank);
            pass_b<OP>(P, S, pend, g, ct, lane);
        }
        pend = cur;
        rk2 = rk1;
        rk1 = r;
        ++li;
    }
    if (pend.r >= 0) {
        if (nobar) collect(P, S, pend, ct);
        else if (c > 1) settle<OP>(P, S, pend, ct, rank);
        pass_b<OP>(P, S, pend, g, ct, lane);
    }
    if (kKL && li > 0) {
        named_sync(kBarConsumers, NCT);
        if (rk2 >= 0) scatter_support(P, S, rk2, (li - 2u) % kSupBufs, ct);
        scatter_support(P, S, rk1, (li - 1u) % kSupBufs, ct);
    }
}

// Tail split: the statistics of tail row w.j from every CTA's part of it, merged in CTA
// order.  Each warp merges on its own (lane i takes parts i, i + 32, ...; a butterfly
// leaves the same sum in every lane), so every warp of every CTA holding a part gets the
// same bits.  Waits are bounded like every other wait.
__device__ void merge_parts(const RowParams& P, Smem& S, Pending& w, int ct, int lane, int U, uint32_t epoch) {
    const long long G = gridDim.x;
    const long long TU = (P.ntok - (P.ntok / G) * G) * (long long)U;
    const long long x0 = w.j * U, x1 = (w.j + 1) * U - 1;
    const long long b0 = ((x0 + 1) * G - 1) / TU, b1 = ((x1 + 1) * G - 1) / TU;   // CTAs holding units x0, x1
    MaxSum acc = ms_empty();
    for (long long b = b0 + lane; b <= b1; b += 32) {
        const long long lo = b * TU / G;
        if (lo >= (b + 1) * TU / G) continue;       // a CTA with an empty range holds no part
        const int which = lo / U == w.j ? 0 : 1;
        const unsigned int* sl = ws_slot(P, b, which);
        const long long t0 = clock64();
        bool ok = true;
        while (ld_acquire_u32(sl + 2) != epoch) {
            if (S.abort) { ok = false; break; }
            if (clock64() - t0 > P.wait_limit) {
                S.abort = 1;
                atomicOr(&g_watchdog, 1u);
                ok = false;
                break;
            }
        }
        if (!ok) break;
        float m, sum;
        asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(m), "=f"(sum) : "l"(sl) : "memory");
        acc = ms_merge(acc, MaxSum{m, sum});
    }
    acc = ms_warp_reduce(acc);
    w.m = acc.m;
    w.lnS = logf(acc.s);
    if (w.first && ct == LT) {
        if (P.lse_out) P.lse_out[w.r] = w.m + w.lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = w.m; P.stats_out[2 * w.r + 1] = w.lnS; }
    }
}

// Self-contained CE with the tail split (one CTA per SM, no clusters): whole rows with
// the barrier-free statistics of consumer_self, then up to two tail segments whose
// statistics come from every CTA's part of their row.
template <int OP>
__device__ void consumer_split(const RowParams& P, Smem& S) {
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int ncols = (int)P.ncols;
    const int U = (ncols + 3) >> 2;
    const uint32_t epoch = ld_relaxed_u32(P.ws) + 1u;
    // barrier-free statistics need a body tile in every row (the ring then keeps the
    // warps within kPartBufs rows of each other); shorter rows take the barrier
    const bool nobar = ncols >= 8;
    uint32_t g = 0, na = 0, nb = 0;
    Pending pend;
    pend.r = -1;
    Item nxt;
    bool have = item_at(P, 0, U, nxt);
    uint32_t nlab = have ? P.labels[nxt.r] : 0u;
    for (long long i = 0; have; ++i) {
        const Item it = nxt;
        const uint32_t lab_r = nlab;
        have = item_at(P, i + 1, U, nxt);
        if (have) nlab = P.labels[nxt.r];
        float* rowp = P.x + it.r * P.ld + P.col0;
        const Part pt = part_units(rowp, ncols, U, it.u0, it.u1);
        Pending cur;
        cur.r = it.r;
        cur.rowp = rowp;
        cur.pt = pt;
        cur.nt = (pt.bn + kTileF - 1) / kTileF;
        cur.inwin = it.r >= P.ls && it.r < P.le;
        cur.first = it.u0 == 0;
        cur.which = it.which;
        cur.j = it.j;
        cur.jl = -1;
        cur.bad = (long long)lab_r >= P.V;
        if (!cur.bad) {
            const long long jj = (long long)lab_r - P.col0;
            if (jj >= pt.lo && jj < pt.hi) cur.jl = (int)jj;
        }
        if (cur.bad && cur.inwin && cur.first && ct == LT && P.err) atomicAdd(P.err, 1);
        cur.has_ht = ct < pt.hn || (ct >= 4 && ct - 4 < pt.tn);
        cur.jht = ct < pt.hn ? ct : pt.t0 + ct - 4;
        cur.ht = cur.has_ht ? rowp[cur.jht] : 0.f;

        // ---- pass A
        MaxSum ms = ms_empty();
        if (cur.has_ht) ms_add(ms, cur.ht);
        for (int t = 0; t < cur.nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
            wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
            const int n4 = min(kTileF, pt.bn - t * kTileF) >> 2;
            float4 v[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int jv = u * NCT + ct;
                v[u] = jv < n4 ? ld_shared_v4(&S.ring[slot][jv * 4]) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            ms_addv(ms, v);
        }
        g += (uint32_t)cur.nt;
        ms = ms_warp_reduce(ms);
        if (it.which < 0 && nobar) {
            // a whole row: the warps' partials go through the mbarrier buffers
            cur.ab = na % kPartBufs;
            cur.apar = (na / kPartBufs) & 1u;
            ++na;
            if (lane == 0) {
                S.wpart[cur.ab][cw] = make_float2(ms.m, ms.s);
                mbar_arrive(&S.abar[cur.ab]);
            }
        } else {
            const uint32_t b = nb & 1u;
            ++nb;
            if (lane == 0) S.wred[b][cw] = make_float4(ms.m, ms.s, 0.f, 0.f);
            named_sync(kBarConsumers, NCT);
            const MaxSum tot = combine4(S.wred[b], NCW).ms;
            if (it.which >= 0) {
                // a tail segment: this CTA's part, published at once for the row's other parts
                if (ct == 0) publish_part(P, it.which, tot, epoch);
            } else {
                cur.m = tot.m;
                cur.lnS = logf(tot.s);
                if (ct == LT) {
                    if (P.lse_out) P.lse_out[it.r] = cur.m + cur.lnS;
                    if (P.stats_out) { P.stats_out[2 * it.r] = cur.m; P.stats_out[2 * it.r + 1] = cur.lnS; }
                }
            }
        }
        if (pend.r >= 0) {
            if (pend.which >= 0) merge_parts(P, S, pend, ct, lane, U, epoch);
            else if (nobar) collect(P, S, pend, ct);
            pass_b<OP>(P, S, pend, g, ct, lane);
        }
        pend = cur;
    }
    if (pend.r >= 0) {
        if (pend.which >= 0) merge_parts(P, S, pend, ct, lane, U, epoch);
        else if (nobar) collect(P, S, pend, ct);
        pass_b<OP>(P, S, pend, g, ct, lane);
    }
}

// Tail split: the last CTA to finish advances the workspace generation (every CTA has
// read it at its start and is done with every slot by now).
__device__ __forceinline__ void take_ticket(const RowParams& P) {
    __threadfence();
    const unsigned int t = atomicAdd(P.ws + 1, 1u);
    if (t == gridDim.x - 1) {
        P.ws[1] = 0u;
        __threadfence();
        atomicAdd(P.ws, 1u);
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
        for (int b = 0; b < 4; ++b) mbar_init(&S.xbar[b], 1u);   // the local expect_tx; the peers' data completes the bytes
        for (int b = 0; b < 2; ++b) mbar_init(&S.lbar[b], 1u);
        for (int b = 0; b < kPartBufs; ++b) mbar_init(&S.abar[b], NCW);
        S.abort = 0;
        S.issued = 0;
        fence_mbar_init_cluster();
    }
    if (c > 1) cluster_sync_all();
    else __syncthreads();
    // launched as a programmatic dependent: the set-up above overlaps the tail of the
    // previous kernel on the stream; its results are visible past this wait
    pdl_wait_primary();
    pdl_launch_dependents();

    const bool split = OP == kCeFused && P.split;
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            if (split) producer_split(P, S);
            else producer<OP, RES>(P, S, rank, cid, ncl);
            drain(S, P.wait_limit);
        }
        __syncwarp();
    } else {
        if (split) consumer_split<OP>(P, S);
        else if (RES) consumer_self<OP>(P, S, rank, cid, ncl);
        else consumer<OP, false>(P, S, rank, cid, ncl);
    }
    // no CTA may leave while a peer can still write into its shared memory
    if (c > 1) cluster_sync_all();
    if (split) {
        __syncthreads();
        if (threadIdx.x == 0) take_ticket(P);
    }
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (P.csize > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)P.csize;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    RowParams p = P;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Occupancy answers per (device, kernel, cluster size), queried once: the query costs
// tens of microseconds, far more than a launch.
std::atomic<int> g_max_clusters[kMaxDev][8][kMaxCluster + 1];

int row_max_clusters(int op, bool resident, int c) {
    const void* fn = kernel_for(op, resident);
    const int slot = slot_of(op, resident);
    if (!fn || c < 1 || c > kMaxCluster || prepare(fn, slot) != cudaSuccess) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    const int cached = g_max_clusters[dev][slot][c].load(std::memory_order_acquire);
    if (cached > 0) return cached;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    int n = sms;
    if (c > 1) {
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
        n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        if (n <= 0) n = -1;         // remember "does not fit" too
    }
    g_max_clusters[dev][slot][c].store(n, std::memory_order_release);
    return n > 0 ? n : 0;
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
