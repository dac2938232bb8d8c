// Row engine: cross-entropy (fused, forward, backward) and top-k KL over rows of
// vocabulary logits, one persistent CTA (or cluster of CTAs) per SM.  The logits are
// fp32, or bf16 (read as bf16, every sum and exponential in fp32, the gradient
// rounded to bf16, nearest even, when it is written back).
//
// Layout of one launch
//   * grid = nclusters * csize CTAs, one CTA per SM (the ring below takes
//     ~200 KB of shared memory).  Cluster i handles rows i, i + nclusters, ...
//     A mixed launch (fused CE, 2-CTA clusters) gives cluster i a block of consecutive
//     rows instead: each CTA takes every other row whole, and an odd block's last row
//     is split over the pair, so that no CTA carries more than half a row above another.
//   * a row slice of ncols elements is cut into a head (the elements before the first
//     16-byte boundary: at most 3 fp32 or 7 bf16), a 16-byte-aligned body and a tail
//     of the same bound.  The body is split evenly (in 16-byte chunks) across the csize
//     CTAs of the cluster; CTA rank 0 also takes the head and the last rank the tail.
//   * warp 0 (one lane) is the producer: it streams each CTA's body through a
//     ring of kSlots tiles of kTileB bytes with 1-D bulk copies (TMA) signalled
//     on per-slot mbarriers; warps 1..15 are consumers.  A consumer thread owns
//     16-byte chunks ct, ct + NCT, ... (kVec of them) of every tile.
//
// Modes
//   self-contained (CE fused, KL without given statistics): the producer streams
//             each row part twice.  Pass A reduces (max, sum of exponentials)
//             online per thread; partials are merged across warps (shared
//             memory: for CE, and for KL rows of four tiles a pass or more, each warp
//             publishes its partial and one warp, in turn, combines them) and across
//             the cluster (distributed shared memory:
//             st.async that completes the peer's mbarrier transaction count).  Pass B
//             re-reads the part -- it was read microseconds earlier, so the bytes
//             come from L2 -- and writes the gradient tile by tile.  HBM sees one
//             read and one write per element; no row has to fit on chip.
//   streaming (CE backward, KL with given statistics): pass B only.
//   reduce    (CE forward): pass A only.
//
// Sparse columns (the label, the teacher's top-k ids).  Streaming mode gathers their
// logits from the staged tiles as they pass and rewrites their gradient after every
// gradient store of the row and a barrier.  Self-contained mode folds the label into
// pass B and gathers the support logits from global memory before pass A (the row is
// not written until after it) for the KL loss; once every warp's pass B of the row is
// done (a barrier, or an mbarrier each warp arrives on after it) it adds -coef * p_q at
// the support columns with reduction adds (fp32), or rewrites those columns with their
// whole gradient from the gathered logits (bf16, so that every element is rounded once).
//
// Sources: aprender-train wgpu_cross_entropy.rs (module doc, forward_async,
// backward: loss = lse - s[label], gradient scale * (softmax - onehot), loss
// window) and cortiq-engine train_head.rs (module doc and kl_rows: KL over the
// teacher's top-k, gradient coef * (softmax - p_T); the f16 activations beside f32
// logits).  The pages' kernels read a row three times with workgroup tree
// reductions; this engine reads it once.
#include "vl_device.cuh"
#include "vl_internal.h"

#include <cuda_bf16.h>

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

static_assert(kTileB / 16 == NCT * kVec, "kVec 16-byte chunks of each tile per consumer thread");
static_assert(KMAX >= 1024, "the C ABI promises k <= 1024");

__device__ unsigned int g_watchdog;

// ---------------------------------------------------------------- element types

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int NV = 4;        // elements per 16 bytes
    static __device__ __forceinline__ void unpack(uint4 r, float (&f)[NV]) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[NV]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    static __device__ __forceinline__ float get(const float* p) { return *p; }
    static __device__ __forceinline__ void put(float* p, float v) { *p = v; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int NV = 8;
    static __device__ __forceinline__ void unpack(uint4 r, float (&f)[NV]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);            // the element at the lower address
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    // two floats to bf16, rounded to nearest even: lo to the lower address
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
        return d;
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[NV]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
    }
    static __device__ __forceinline__ float get(const __nv_bfloat16* p) {
        return __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(p) << 16);
    }
    static __device__ __forceinline__ void put(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

template <typename T>
constexpr int kTileE = kTileB / (int)sizeof(T);    // elements per tile

__device__ __forceinline__ uint4 ld_shared_u4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ void st_global_u4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_global_u4_hint(void* p, uint4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy) : "memory");
}

// ---------------------------------------------------------------- shared memory

struct alignas(128) Smem {
    alignas(16) unsigned char ring[kSlots][kTileB];
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t xbar[4];                   // cluster exchange of (max, sum, KL a, KL b)
    float4 xbuf[4][kMaxCluster];        // (max, sum, KL a, KL b) of each rank's part
    float4 wred[2][NCW];                // per warp: (max, sum, KL a, KL b)
    uint64_t abar[kPartBufs];           // self-contained CE: every warp's pass A partial is in
    float2 wpart[kPartBufs][NCW];
    uint64_t sbar[kPartBufs];           // self-contained CE: the row's statistics are in
    float2 rstat[kPartBufs];            // (max, ln sum) of the row
    float4 wpart4[kPartBufs][NCW];      // self-contained KL without a barrier: each warp's (max, sum, a, b)
    uint64_t bdone[kSupBufs];           // ... every warp's pass B stores of the row are done
    float wloss[2][NCW];
    union {
        struct {                        // streaming mode: support of the current row
            alignas(16) int kcol[2][KMAX];   // column (slice-relative) per entry, -1 outside this CTA
            float kp[2][KMAX];               // probability per entry
            float ks[2][KMAX];               // the logit at that column, gathered as its tile passes
        };
        struct {                        // self-contained CE over a cluster: every warp's pass A partial of
                                        // the row's parts, from every rank (4 rows in flight)
            float2 xw[4][kMaxCluster][NCW];
        };
        struct {                        // self-contained mode: support of the last kSupBufs rows
            alignas(16) int ecol[kSupBufs][KSELF];   // support column (slice-relative; -1 elsewhere)
            float ep[kSupBufs][KSELF];
            unsigned short es[kSupBufs][KSELF];      // bf16: the gathered logit (exact), for the rewrite
            float erow[kSupBufs][3];                 // bf16: m, lnS and the label column of the row
        };
    };
    int abort;
    uint32_t issued;
};

static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");

// Columns of one row slice handled by CTA `rank` of `c` (relative to the slice start).
struct Part {
    int h;     // head length (elements before the first 16-byte boundary)
    int hn;    // head columns this CTA handles
    int b0;    // first body column of this CTA
    int bn;    // body columns of this CTA (a multiple of a 16-byte chunk)
    int t0;    // first tail column
    int tn;    // tail columns this CTA handles
    int lo;    // this CTA owns columns [lo, hi)
    int hi;
};

template <typename T>
__device__ __forceinline__ Part part_of(const T* rowp, int n, int rank, int c) {
    constexpr int NV = Elem<T>::NV;
    Part p;
    const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) & 15u) / sizeof(T));
    int h = (NV - mis) & (NV - 1);
    if (h > n) h = n;
    const int bt = (n - h) & ~(NV - 1);
    const int per = c == 1 ? bt : ((bt / NV + c - 1) / c) * NV;
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

// The head and tail columns: thread ct < hn takes head column ct, thread NV + i the
// tail column t0 + i.
template <typename T>
__device__ __forceinline__ bool has_ht(const Part& pt, int ct) {
    constexpr int NV = Elem<T>::NV;
    return ct < pt.hn || (ct >= NV && ct - NV < pt.tn);
}

template <typename T>
__device__ __forceinline__ int ht_col(const Part& pt, int ct) {
    constexpr int NV = Elem<T>::NV;
    return ct < pt.hn ? ct : pt.t0 + ct - NV;
}

template <int OP>
__device__ __forceinline__ bool row_loaded(const RowParams& P, long long r) {
    if (OP == kCeFused || OP == kCeFwd) return true;    // lse is produced for every row
    return r >= P.ls && r < P.le;
}

template <typename T>
__device__ __forceinline__ T* row_ptr(const RowParams& P, long long r) {
    return static_cast<T*>(P.x) + r * P.ld + P.col0;
}

// softmax value from the row statistics: exp((s - m) - lnS)
__device__ __forceinline__ float soft(float s, float m, float lnS) {
    return ex2(((s - m) - lnS) * kLog2e);
}

// (max, sum) update with a whole tile's kVec chunks of NV values: one max update (a
// tree of maxima), independent exponentials summed as a tree.
template <int NV>
__device__ __forceinline__ void ms_addv(MaxSum& a, const float (&v)[kVec][NV]) {
    constexpr int N = kVec * NV;
    static_assert((N & (N - 1)) == 0, "a power of two values a tile");
    float t[N];
#pragma unroll
    for (int u = 0; u < kVec; ++u)
#pragma unroll
        for (int i = 0; i < NV; ++i) t[u * NV + i] = v[u][i];
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
    const float mx = t[0];
    if (mx > a.m) {
        a.s *= ex2((a.m - mx) * kLog2e);
        a.m = mx;
    }
    float e[N / 2];
#pragma unroll
    for (int u = 0; u < kVec; ++u)
#pragma unroll
        for (int i = 0; i < NV / 2; ++i)
            e[u * (NV / 2) + i] = ex2((v[u][2 * i] - a.m) * kLog2e) + ex2((v[u][2 * i + 1] - a.m) * kLog2e);
#pragma unroll
    for (int w = N / 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) e[i] += e[i + w];
    a.s += e[0];
}

// The same update with one chunk.
template <int NV>
__device__ __forceinline__ void ms_add_chunk(MaxSum& a, const float (&v)[NV]) {
    float mx = v[0];
#pragma unroll
    for (int i = 1; i < NV; ++i) mx = fmaxf(mx, v[i]);
    if (mx > a.m) {
        a.s *= ex2((a.m - mx) * kLog2e);
        a.m = mx;
    }
    float e = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) e += ex2((v[i] - a.m) * kLog2e);
    a.s += e;
}

// A tile of n16 chunks: thread ct holds chunks u * NCT + ct.  A row's last tile is
// usually partial; its absent chunks are skipped rather than summed as -inf.
template <int NV>
__device__ __forceinline__ void ms_add_tile(MaxSum& a, const float (&v)[kVec][NV], int n16, int ct) {
    if (n16 >= kVec * NCT) {
        ms_addv<NV>(a, v);
        return;
    }
#pragma unroll
    for (int u = 0; u < kVec; ++u)
        if (u * NCT + ct < n16) ms_add_chunk<NV>(a, v[u]);
}

// Chunk j of tile `slot` into v (absent chunks: -inf).
template <typename T>
__device__ __forceinline__ void load_chunk(const Smem& S, uint32_t slot, int j, int n16, float (&v)[Elem<T>::NV]) {
    if (j < n16) {
        Elem<T>::unpack(ld_shared_u4(&S.ring[slot][16 * j]), v);
    } else {
#pragma unroll
        for (int i = 0; i < Elem<T>::NV; ++i) v[i] = -INFINITY;
    }
}

// ---------------------------------------------------------------- producer

// Row item i of this CTA: the row, and which part of it (part prank of pc) the CTA takes.
// Plain launches walk rows cid, cid + ncl, ... whole (pc = 1) or split over the cluster.
// Mixed launches (2-CTA clusters) give cluster cid a block of consecutive rows; an odd
// block's last row comes first and is split over the pair, then each CTA takes every other
// row of the block whole.  A CTA then carries at most half a row more than another.
struct Item {
    long long r;
    int prank, pc;
};

__device__ __forceinline__ bool row_item(const RowParams& P, int rank, long long cid, long long ncl, long long i,
                                         Item& it) {
    if (!P.mixed) {
        it.r = P.rbeg + cid + i * ncl;
        it.prank = rank;
        it.pc = P.csize;
        return it.r < P.rend;
    }
    const long long R = P.rend - P.rbeg, q = R / ncl, rm = R % ncl;
    const long long nk = q + (cid < rm ? 1 : 0);
    const long long base = P.rbeg + cid * q + (cid < rm ? cid : rm);
    const long long odd = nk & 1;
    if (odd && i == 0) {
        it.r = base + nk - 1;
        it.prank = rank;
        it.pc = 2;
        return true;
    }
    const long long j = i - odd;
    it.r = base + 2 * j + rank;
    it.prank = 0;
    it.pc = 1;
    return j < nk / 2;
}

// Issue the body tiles of one row part; false if a wait gave up.
template <typename T>
__device__ __forceinline__ bool issue_body(const RowParams& P, Smem& S, const T* rowp, const Part& pt, uint32_t& g) {
    for (int c0 = 0; c0 < pt.bn; c0 += kTileE<T>) {
        // test hook: CTA 0 stops before this tile, so the consumers' wait for it runs out
        if ((long long)g == P.withhold && blockIdx.x == 0) return false;
        const uint32_t slot = g % kSlots, use = g / kSlots;
        if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog, P.wait_limit)) return false;
        const uint32_t bytes = (uint32_t)min(kTileE<T>, pt.bn - c0) * (uint32_t)sizeof(T);
        mbar_arrive_expect_tx(&S.full[slot], bytes);
        bulk_g2s(S.ring[slot], rowp + pt.b0 + c0, bytes, &S.full[slot]);
        ++g;
    }
    return true;
}

template <typename T>
__device__ __forceinline__ bool issue_part(const RowParams& P, Smem& S, const Item& it, uint32_t& g) {
    const T* rowp = row_ptr<T>(P, it.r);
    return issue_body<T>(P, S, rowp, part_of<T>(rowp, (int)P.ncols, it.prank, it.pc), g);
}

// Tile order: one pass per row for the streaming and reduce modes; for the
// self-contained mode pass A of a row, then pass B of the row before it, so the
// reads of the next row are in flight while the current one is written.
template <typename T, int OP, bool RES>
__device__ void producer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    uint32_t g = 0;
    Item it, prev;
    prev.r = -1;
    for (long long i = 0; row_item(P, rank, cid, ncl, i, it); ++i) {
        if (!row_loaded<OP>(P, it.r)) continue;
        if (!issue_part<T>(P, S, it, g)) break;
        if (RES) {
            if (prev.r >= 0 && !issue_part<T>(P, S, prev, g)) break;
            prev = it;
        }
    }
    if (RES && prev.r >= 0 && !S.abort) issue_part<T>(P, S, prev, g);
    S.issued = g;
}

// Before the CTA exits, every bulk copy it issued must have landed.
__device__ void drain(Smem& S, long long limit) {
    const uint32_t iss = S.issued;
    for (uint32_t gt = iss > (uint32_t)kSlots ? iss - kSlots : 0u; gt < iss; ++gt)
        wait_parity_drain(&S.full[gt % kSlots], (gt / kSlots) & 1u, limit);
}

// ---------------------------------------------------------------- consumer helpers

template <typename T>
__device__ void zero_part(T* rowp, const Part& pt, int ct) {
    constexpr int NV = Elem<T>::NV;
    for (int i = ct; i < pt.bn / NV; i += NCT) st_global_u4(rowp + pt.b0 + NV * i, make_uint4(0u, 0u, 0u, 0u));
    if (has_ht<T>(pt, ct)) Elem<T>::put(rowp + ht_col<T>(pt, ct), 0.f);
}

// A sparse column this thread looks after: where it sits in the row part, and its
// logit once the tile holding it has passed.
struct Sparse {
    int col;     // slice-relative column, -1 if none
    int rel;     // column - b0 inside this CTA's body (tile = rel / tile elements), -1 for head/tail
    float s;     // the logit
};

template <typename T>
__device__ __forceinline__ void locate(Sparse& e, const Part& pt, const T* rowp) {
    if (e.col >= pt.b0 && e.col < pt.b0 + pt.bn) {
        e.rel = e.col - pt.b0;
    } else {
        e.rel = -1;
        e.s = Elem<T>::get(rowp + e.col);     // head or tail: read before anything of the row is written
    }
}

template <typename T>
__device__ __forceinline__ void gather(Sparse& e, int t, const unsigned char* tile) {
    if (e.rel >= 0 && (e.rel / kTileE<T>) == t) e.s = Elem<T>::get(reinterpret_cast<const T*>(tile) + e.rel % kTileE<T>);
}

template <typename T>
__device__ __forceinline__ void gather_support(Smem& S, uint32_t kb, const int (&erel)[EPT], int ct, int t,
                                               const unsigned char* tile) {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
        if (erel[i] >= 0 && erel[i] / kTileE<T> == t)
            S.ks[kb][ct + i * NCT] = Elem<T>::get(reinterpret_cast<const T*>(tile) + erel[i] % kTileE<T>);
}

// (max, sum) of n <= 128 partials, by one warp: lane i takes partials i, i + 32, ...; the
// max and then the rescaled sums meet in butterflies, which leave every lane (and every
// warp that runs this on the same partials) with the same bits.
__device__ __forceinline__ MaxSum combine_warp(const float2* part, int n, int lane) {
    float2 q[4];
    float M = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = lane + 32 * i;
        q[i] = j < n ? part[j] : make_float2(-FLT_MAX, 0.f);
        M = fmaxf(M, q[i].x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float T = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) T += q[i].y * ex2((q[i].x - M) * kLog2e);
    return MaxSum{M, warp_sum(T)};
}
static_assert(kMaxCluster * NCW <= 128, "combine_warp takes up to 128 partials");

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

// The gradient of a chunk: c1 * exp(x - m - lnS) per element, as 2^(x log2 e - m log2 e - K)
// with K = lnS log2 e - log2 c1 when c1 >= 0 (the scale folded into the exponent).
template <int NV>
__device__ __forceinline__ void grad_chunk(const float (&x)[NV], float (&o)[NV], bool fold, float m, float lnS, float K,
                                           float c1) {
    if (fold) {
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = ex2(fmaf(x[i] - m, kLog2e, -K));
    } else {
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = c1 * soft(x[i], m, lnS);
    }
}

// ---------------------------------------------------------------- streaming consumer

template <typename T, int OP>
__device__ void consumer(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    constexpr bool kKL = OP == kKl;
    constexpr int NV = Elem<T>::NV;
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int c = P.csize;
    const int ncols = (int)P.ncols;
    uint32_t g = 0, nred = 0, nloss = 0, nrow = 0;
    const bool has_label = (OP != kKl) || (P.labels != nullptr && P.ce_coef != 0.f);
    const float cg = P.cg;
    // the label and support entry q = ct of the next row, loaded one row ahead
    uint32_t nlab = 0, nid = 0;
    float np = 0.f;
    auto prefetch = [&](long long rr) {
        if (rr >= P.rend) return;
        if (has_label) nlab = P.labels[rr];
        if (kKL && ct < P.k) { nid = P.tid[rr * P.k + ct]; np = P.tp[rr * P.k + ct]; }
    };
    prefetch(P.rbeg + cid);

    for (long long r = P.rbeg + cid; r < P.rend; r += ncl) {
        const uint32_t lab_r = nlab, id0 = nid;
        const float p0 = np;
        prefetch(r + ncl);
        T* rowp = row_ptr<T>(P, r);
        const Part pt = part_of<T>(rowp, ncols, rank, c);
        const bool inwin = r >= P.ls && r < P.le;
        const int nt = (pt.bn + kTileE<T> - 1) / kTileE<T>;
        if (!row_loaded<OP>(P, r)) {
            zero_part<T>(rowp, pt, ct);
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
        if (ct == LT && jl >= pt.lo && jl < pt.hi) { lab.col = jl; locate<T>(lab, pt, rowp); }
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
                        else S.ks[kb][q] = Elem<T>::get(rowp + col);    // head or tail: before anything is written
                    }
                }
            }
        }

        // head and tail columns: one per thread, finished after the sparse barrier
        const bool hht = has_ht<T>(pt, ct);
        const int jht = ht_col<T>(pt, ct);
        const float ht = hht ? Elem<T>::get(rowp + jht) : 0.f;
        float m, lnS;

        if (OP == kCeFwd) {
            // ---- pass A: (max, sum) online over the streamed tiles; the label's logit gathered
            MaxSum ms = ms_empty();
            if (hht) ms_add(ms, ht);
            for (int t = 0; t < nt; ++t) {
                const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
                wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
                const int n16 = min(kTileE<T>, pt.bn - t * kTileE<T>) / NV;
                float v[kVec][NV];
#pragma unroll
                for (int u = 0; u < kVec; ++u) load_chunk<T>(S, slot, u * NCT + ct, n16, v[u]);
                if (ct == LT) gather<T>(lab, t, S.ring[slot]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
                ms_add_tile<NV>(ms, v, n16, ct);
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
            if (ct == LT) {
                if (!inwin) P.loss[r] = 0.f;
                else if (bad_label) P.loss[r] = __int_as_float(0x7fc00000);
                else if (lab.col >= 0) P.loss[r] = (m - lab.s) + lnS;
            }
            continue;
        }
        if (P.stats_in) { m = P.stats_in[2 * r]; lnS = P.stats_in[2 * r + 1]; }
        else { m = P.lse_in[r]; lnS = 0.f; }

        // ---- pass B: each tile turned into gradient as it lands (zeros outside the window)
        {
            const float c1 = inwin ? cg : 0.f;
            const bool fold = c1 >= 0.f;
            const float K = fold ? lnS * kLog2e - log2f(c1) : 0.f;
            const uint64_t pol = l2_evict_first();
            for (int t = 0; t < nt; ++t) {
                const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
                wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
                const int n16 = min(kTileE<T>, pt.bn - t * kTileE<T>) / NV;
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int j = u * NCT + ct;
                    if (j < n16) {
                        float x[NV], o[NV];
                        Elem<T>::unpack(ld_shared_u4(&S.ring[slot][16 * j]), x);
                        grad_chunk<NV>(x, o, fold, m, lnS, K, c1);
                        st_global_u4_hint(rowp + pt.b0 + t * kTileE<T> + NV * j, Elem<T>::pack(o), pol);
                    }
                }
                if (kKL) gather_support<T>(S, kb, erel, ct, t, S.ring[slot]);
                if (ct == LT) gather<T>(lab, t, S.ring[slot]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            g += (uint32_t)nt;
        }

        // ---- sparse columns, once every bulk store of the row is done: the label,
        //      the support ids, and the head/tail columns with their corrections
        named_sync(kBarConsumers, NCT);
        float lacc = 0.f;
        if (hht) {
            float o = 0.f;
            if (inwin) {
                o = cg * soft(ht, m, lnS);
                if (kKL)
                    for (int j = 0; j < P.k; ++j)
                        if (S.kcol[kb][j] == jht) o -= P.coef * S.kp[kb][j];
                if (jht == jl) o -= P.ce_coef;
            }
            Elem<T>::put(rowp + jht, o);
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
                        Elem<T>::put(rowp + col, o);
                    }
                }
            }
            if (ct == LT && lab.col >= 0 && lab.rel >= 0) {
                bool in_support = false;
                if (kKL)
                    for (int j = 0; j < P.k; ++j) in_support |= S.kcol[kb][j] == lab.col;
                if (!in_support) Elem<T>::put(rowp + lab.col, cg * soft(lab.s, m, lnS) - P.ce_coef);
            }
        }

        // ---- losses (streaming launches run one CTA per row: c == 1)
        if (OP == kCeBwd) {
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
                P.loss[r] = L;
            }
        }
    }
}

// ---------------------------------------------------------------- self-contained consumer

// A row whose pass A is done and whose pass B is still to come.  Two of these are live
// across a pass A, so the record is kept small: what can be recomputed from the row
// index (its pointer, its tile count) is, and the flags and buffer indices share a word.
struct Pending {
    long long r;
    int b0, bn;      // this CTA's body columns of the row (slice coordinates)
    int jl;          // slice-relative label column, -1 when none or outside this CTA's columns
    int jht;         // this thread's head or tail column, -1 when none
    float m, lnS;
    float ht;        // the logit at jht
    // bit 0 in the window, bit 1 bad label, bit 2 this part holds column 0 of the row (it
    // writes lse, stats and the out-of-window loss), bit 3 the row is split over the cluster;
    // bits 8-9 the cluster exchange buffer of
    // the row's statistics and bit 10 the phase to wait for; bits 16-19 the buffer of the
    // warps' pass A partials (CE; KL without a barrier) and bit 20 its phase
    uint32_t f;
    __device__ __forceinline__ bool inwin() const { return f & 1u; }
    __device__ __forceinline__ bool bad() const { return f & 2u; }
    __device__ __forceinline__ bool first() const { return f & 4u; }
    __device__ __forceinline__ bool shared() const { return f & 8u; }
    __device__ __forceinline__ uint32_t xb() const { return (f >> 8) & 3u; }
    __device__ __forceinline__ uint32_t xpar() const { return (f >> 10) & 1u; }
    __device__ __forceinline__ uint32_t ab() const { return (f >> 16) & 15u; }
    __device__ __forceinline__ uint32_t apar() const { return (f >> 20) & 1u; }
};

// Pass B of a row whose statistics are known: the gradient tile by tile with the
// label's one-hot folded in.  The teacher support is left to scatter_support.
template <typename T, int OP>
__device__ __forceinline__ void pass_b(const RowParams& P, Smem& S, const Pending& w, uint32_t& g, int ct, int lane,
                                       float l2cg) {
    constexpr int NV = Elem<T>::NV;
    T* const rowp = row_ptr<T>(P, w.r);
    const int nt = (w.bn + kTileE<T> - 1) / kTileE<T>;
    // the CE loss: the fused CE output, or beside the KL when labels come with it
    float* const ce_out = OP == kCeFused ? P.loss : OP == kKl ? P.ce_loss : nullptr;
    const float c1 = w.inwin() ? P.cg : 0.f;
    const bool fold = c1 >= 0.f;
    // the gradient lines are done with: written back first, ahead of the logits that
    // pass B of the next row still re-reads from L2
    const uint64_t pol = l2_evict_first();
    const float K = fold ? w.lnS * kLog2e - (w.inwin() ? l2cg : -INFINITY) : 0.f;
    for (int t = 0; t < nt; ++t) {
        const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
        wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
        const int n16 = min(kTileE<T>, w.bn - t * kTileE<T>) / NV;
        auto grad = [&](int u, uint4 raw) {
            const int j = u * NCT + ct;
            const int c0 = w.b0 + t * kTileE<T> + NV * j;
            float x[NV], o[NV];
            Elem<T>::unpack(raw, x);
            grad_chunk<NV>(x, o, fold, w.m, w.lnS, K, c1);
            if (w.inwin()) {
                const unsigned d = (unsigned)(w.jl - c0);
                if (d < (unsigned)NV) {
#pragma unroll
                    for (int i = 0; i < NV; ++i)
                        if ((unsigned)i == d) {
                            o[i] -= P.ce_coef;
                            if (ce_out) ce_out[w.r] = (w.m - x[i]) + w.lnS;
                        }
                }
            }
            st_global_u4_hint(rowp + c0, Elem<T>::pack(o), pol);
        };
        // half the tile's chunks turned into gradient while the other half is still in the
        // slot; the slot is released once the second half is in registers
        constexpr int H = kVec / 2;
        uint4 raw[H];
#pragma unroll
        for (int u = 0; u < H; ++u)
            if (u * NCT + ct < n16) raw[u] = ld_shared_u4(&S.ring[slot][16 * (u * NCT + ct)]);
#pragma unroll
        for (int u = 0; u < H; ++u)
            if (u * NCT + ct < n16) grad(u, raw[u]);
#pragma unroll
        for (int u = 0; u < H; ++u)
            if ((H + u) * NCT + ct < n16) raw[u] = ld_shared_u4(&S.ring[slot][16 * ((H + u) * NCT + ct)]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
#pragma unroll
        for (int u = 0; u < H; ++u)
            if ((H + u) * NCT + ct < n16) grad(H + u, raw[u]);
    }
    g += (uint32_t)nt;
    if (w.jht >= 0) {
        float o = c1 * soft(w.ht, w.m, w.lnS);
        if (w.inwin() && w.jht == w.jl) {
            o -= P.ce_coef;
            if (ce_out) ce_out[w.r] = (w.m - w.ht) + w.lnS;
        }
        Elem<T>::put(rowp + w.jht, o);
    }
    if (ce_out && w.first() && ct == LT) {
        if (!w.inwin()) ce_out[w.r] = 0.f;
        else if (w.bad()) ce_out[w.r] = __int_as_float(0x7fc00000);
    }
}

// Self-contained CE, one CTA per row: one warp (the row's collector, in turn) combines the
// warps' pass A partials once all are in and publishes the row's statistics; the other
// warps only read them, a row later, before the row's pass B.
__device__ __forceinline__ void collect_row(const RowParams& P, Smem& S, const Pending& w, int lane) {
    wait_parity<false>(&S.abar[w.ab()], w.apar(), &S.abort, &g_watchdog, P.wait_limit);
    const MaxSum tot = combine_warp(S.wpart[w.ab()], NCW, lane);
    const float lnS = logf(tot.s);
    if (lane == 0) {
        S.rstat[w.ab()] = make_float2(tot.m, lnS);
        mbar_arrive(&S.sbar[w.ab()]);
        if (P.lse_out) P.lse_out[w.r] = tot.m + lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = tot.m; P.stats_out[2 * w.r + 1] = lnS; }
    }
}

__device__ __forceinline__ void collect(const RowParams& P, Smem& S, Pending& w) {
    wait_parity<false>(&S.sbar[w.ab()], w.apar(), &S.abort, &g_watchdog, P.wait_limit);
    const float2 st = S.rstat[w.ab()];
    w.m = st.x;
    w.lnS = st.y;
}

// Self-contained CE over a cluster: the row's statistics from every warp of every rank,
// sent with st.async after each warp's pass A; every rank combines them in the same order
// (rank, then warp), so all hold the same bits.
__device__ __forceinline__ void collect_cluster(const RowParams& P, Smem& S, Pending& w, int ct, int rank) {
    wait_parity<true>(&S.xbar[w.xb()], w.xpar(), &S.abort, &g_watchdog, P.wait_limit);
    const MaxSum tot = combine_warp(&S.xw[w.xb()][0][0], P.csize * NCW, ct & 31);
    w.m = tot.m;
    w.lnS = logf(tot.s);
    if (rank == 0 && ct == LT) {
        if (P.lse_out) P.lse_out[w.r] = w.m + w.lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = w.m; P.stats_out[2 * w.r + 1] = w.lnS; }
    }
}

// Cluster mode: the row's statistics (and KL loss parts) from every rank's part, sent
// after its pass A.  Every rank combines the parts in rank order: the same bits.
template <int OP>
__device__ __forceinline__ void settle(const RowParams& P, Smem& S, Pending& w, int ct, int rank) {
    wait_parity<true>(&S.xbar[w.xb()], w.xpar(), &S.abort, &g_watchdog, P.wait_limit);
    const Part4 tot = combine4(S.xbuf[w.xb()], P.csize);
    w.m = tot.ms.m;
    w.lnS = logf(tot.ms.s);
    if (rank == 0 && ct == LT) {
        if (P.lse_out) P.lse_out[w.r] = w.m + w.lnS;
        if (P.stats_out) { P.stats_out[2 * w.r] = w.m; P.stats_out[2 * w.r + 1] = w.lnS; }
        if (OP == kKl) P.loss[w.r] = fmaf(w.m + w.lnS, tot.b, tot.a);
    }
}

// The teacher's part of the gradient at every support column of loaded row r (buffer
// sb).  Runs after a barrier that follows the row's pass B, which orders every
// thread's gradient store before it.  fp32: -coef * p_q added with reduction adds, so
// repeated ids sum.  bf16: the column's whole gradient, cg * p_S - coef * (sum of its
// entries' p) - ce_coef * [label], computed from the gathered logit and written once
// (by the column's lowest entry), so that it is rounded to bf16 once.
template <typename T>
__device__ __forceinline__ void scatter_support(const RowParams& P, const Smem& S, long long r, uint32_t sb, int ct) {
    T* rowp = row_ptr<T>(P, r);
    if constexpr (sizeof(T) == 4) {
        for (int q = ct; q < P.k; q += NCT) {
            const int col = S.ecol[sb][q];
            if (col >= 0) atomicAdd(reinterpret_cast<float*>(rowp) + col, -P.coef * S.ep[sb][q]);
        }
    } else {
        const float m = S.erow[sb][0], lnS = S.erow[sb][1];
        const int jl = __float_as_int(S.erow[sb][2]);
        for (int q = ct; q < P.k; q += NCT) {
            const int col = S.ecol[sb][q];
            if (col < 0) continue;
            bool first = true;
            float psum = 0.f;
            for (int j = 0; j < P.k; ++j)
                if (S.ecol[sb][j] == col) {
                    first &= j >= q;
                    psum += S.ep[sb][j];
                }
            if (!first) continue;
            const float s = __uint_as_float((uint32_t)S.es[sb][q] << 16);
            float o = P.cg * soft(s, m, lnS) - P.coef * psum;
            if (col == jl) o -= P.ce_coef;
            Elem<T>::put(rowp + col, o);
        }
    }
}

template <typename T, int OP>
__device__ void consumer_self(const RowParams& P, Smem& S, int rank, long long cid, long long ncl) {
    constexpr bool kKL = OP == kKl;
    constexpr int NV = Elem<T>::NV;
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int c = P.csize;
    const int ncols = (int)P.ncols;
    const bool has_label = (OP != kKl) || P.labels != nullptr;
    // barrier-free statistics (CE, one CTA per row, every row at least one body tile)
    const bool nobar = !kKL && ncols >= 2 * NV * c;   // mixed launches: c = 2 covers the whole rows too
    // KL without a CTA barrier per row, when a row part spans at least four tiles a pass (a
    // warp is then less than a row ahead of any other: the ring holds kSlots tiles).  Each
    // warp publishes its partial on an mbarrier; one warp in turn combines them; the support
    // scatter of a row waits for every warp's pass B of it on another.
    const bool kfree = kKL && ncols >= 4 * c * kTileE<T>;
    static_assert(4 * 2 > kSlots, "four tiles a pass keep the warps within a row of each other");
    const float l2cg = log2f(P.cg);   // the gradient scale folded into pass B's exponent
    uint32_t g = 0, nred = 0, nx = 0, li = 0;
    long long rk1 = -1, rk2 = -1;      // KL: the last two loaded rows (support scatter owed)
    uint32_t nlab = 0, nid = 0;
    float np = 0.f;
    auto prefetch = [&](long long rr) {
        if (rr >= P.rend) return;
        if (has_label) nlab = P.labels[rr];
        if (kKL && ct < P.k) { nid = P.tid[rr * P.k + ct]; np = P.tp[rr * P.k + ct]; }
    };
    Item it, nx_it;
    const bool any = row_item(P, rank, cid, ncl, 0, nx_it);
    if (any) prefetch(nx_it.r);
    Pending pend;
    pend.r = -1;

    for (long long ii = 0; any; ++ii) {
        it = nx_it;
        const long long r = it.r;
        const bool more = row_item(P, rank, cid, ncl, ii + 1, nx_it);
        const uint32_t lab_r = nlab, id0 = nid;
        const float p0 = np;
        if (more) prefetch(nx_it.r);
        T* rowp = row_ptr<T>(P, r);
        const Part pt = part_of<T>(rowp, ncols, it.prank, it.pc);
        const bool inwin = r >= P.ls && r < P.le;
        const bool shared = it.pc > 1;
        if (!row_loaded<OP>(P, r)) {
            zero_part<T>(rowp, pt, ct);
            if (ct == 0 && it.prank == 0) {
                P.loss[r] = 0.f;
                if (P.ce_loss) P.ce_loss[r] = 0.f;
            }
            if (more) continue;
            break;
        }
        const uint32_t sb = li % kSupBufs;
        Pending cur;
        cur.r = r;
        cur.b0 = pt.b0;
        cur.bn = pt.bn;
        const int nt = (pt.bn + kTileE<T> - 1) / kTileE<T>;
        cur.jl = -1;
        bool bad = false;
        if (has_label) {
            if ((long long)lab_r >= P.V) bad = true;
            else {
                const long long j = (long long)lab_r - P.col0;
                if (j >= pt.lo && j < pt.hi) cur.jl = (int)j;
            }
        }
        cur.f = (inwin ? 1u : 0u) | (bad ? 2u : 0u) | (it.prank == 0 ? 4u : 0u) | (shared ? 8u : 0u);
        if (bad && inwin && it.prank == 0 && ct == LT && P.err) atomicAdd(P.err, 1);
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
                        if (it.prank == 0 && P.err) atomicAdd(P.err, 1);
                    } else {
                        const long long j = (long long)id - P.col0;
                        if (j >= pt.lo && j < pt.hi) col = (int)j;
                    }
                    S.ecol[sb][q] = col;
                    S.ep[sb][q] = p;
                    scol[i] = col;
                    sp[i] = p;
                    if (col >= 0) sx[i] = Elem<T>::get(rowp + col);
                }
            }
        }
        const bool ht_here = has_ht<T>(pt, ct);
        cur.jht = ht_here ? ht_col<T>(pt, ct) : -1;
        cur.ht = ht_here ? Elem<T>::get(rowp + cur.jht) : 0.f;

        // ---- pass A: (max, sum) online over the streamed tiles
        MaxSum ms = ms_empty();
        if (ht_here) ms_add(ms, cur.ht);
        for (int t = 0; t < nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % kSlots;
            wait_parity<false>(&S.full[slot], (gt / kSlots) & 1u, &S.abort, &g_watchdog, P.wait_limit);
            const int n16 = min(kTileE<T>, pt.bn - t * kTileE<T>) / NV;
            float v[kVec][NV];
#pragma unroll
            for (int u = 0; u < kVec; ++u) load_chunk<T>(S, slot, u * NCT + ct, n16, v[u]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            ms_add_tile<NV>(ms, v, n16, ct);
        }
        g += (uint32_t)nt;
        ms = ms_warp_reduce(ms);
        if (nobar && shared) {
            // CE over a cluster: this warp's partial goes to every rank (st.async completing the
            // rank's exchange barrier, whose one local arrival carries the bytes expected); the
            // row is collected just before its pass B, one row later -- no CTA barrier per row.
            // Four buffers: a warp writes buffer i + 4 only after its own collection of row
            // i + 2, which needs every warp's partial of row i + 2, each sent after that warp's
            // collection of row i.
            cur.f |= ((nx & 3u) << 8) | (((nx >> 2) & 1u) << 10);
            ++nx;
            if (ct == 0) mbar_arrive_expect_tx(&S.xbar[cur.xb()], 8u * (uint32_t)(c * NCW));
            if (lane == 0)
                for (int q = 0; q < c; ++q)
                    st_async_f32x2(map_to_rank(&S.xw[cur.xb()][rank][cw], (uint32_t)q), ms.m, ms.s,
                                   map_to_rank(&S.xbar[cur.xb()], (uint32_t)q));
            if (pend.r >= 0) {
                if (pend.shared()) collect_cluster(P, S, pend, ct, rank);
                else collect(P, S, pend);
                pass_b<T, OP>(P, S, pend, g, ct, lane, l2cg);
            }
            pend = cur;
            ++li;
            if (more) continue;
            break;
        }
        if (nobar) {
            // CE: publish this warp's partial and move on; the row's statistics are
            // collected just before its pass B, one row later, when every warp has long
            // arrived -- no CTA-wide barrier per row
            cur.f |= ((nred % kPartBufs) << 16) | (((nred / kPartBufs) & 1u) << 20);
            if (lane == 0) {
                S.wpart[cur.ab()][cw] = make_float2(ms.m, ms.s);
                mbar_arrive(&S.abar[cur.ab()]);
            }
            if (cw == (int)(nred % NCW)) collect_row(P, S, cur, lane);
            ++nred;
            if (pend.r >= 0) {
                if (pend.shared()) collect_cluster(P, S, pend, ct, rank);
                else collect(P, S, pend);
                pass_b<T, OP>(P, S, pend, g, ct, lane, l2cg);
            }
            pend = cur;
            ++li;
            if (more) continue;
            break;
        }
        const uint32_t b = nred & 1u;
        const uint32_t ab = nred % kPartBufs, apar = (nred / kPartBufs) & 1u;
        const bool collector = cw == (int)(nred % NCW);
        ++nred;
        // KL loss parts of the support entries this thread holds: a = sum p (ln p - s),
        // b = sum p (the loss is a + lse * b; entries with p <= 0 add no term).  Formed
        // after pass A, so the gather of s overlaps the row's stream.
        float ka = 0.f, kb = 0.f;
        if (kKL) {
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                if (scol[i] >= 0 && sp[i] > 0.f) {
                    ka += sp[i] * (logf(sp[i]) - sx[i]);
                    kb += sp[i];
                }
                // bf16: the logit kept for the support rewrite (exact: it is a bf16 value)
                if (sizeof(T) == 2 && scol[i] >= 0)
                    S.es[sb][ct + i * NCT] = (unsigned short)(__float_as_uint(sx[i]) >> 16);
            }
            ka = warp_sum(ka);
            kb = warp_sum(kb);
        }
        Part4 tot{MaxSum{0.f, 0.f}, 0.f, 0.f};
        if (kfree) {
            cur.f |= (ab << 16) | (apar << 20);
            if (lane == 0) {
                S.wpart4[ab][cw] = make_float4(ms.m, ms.s, ka, kb);
                mbar_arrive(&S.abar[ab]);
            }
            if (collector) {
                wait_parity<false>(&S.abar[ab], apar, &S.abort, &g_watchdog, P.wait_limit);
                tot = combine4(S.wpart4[ab], NCW);
            }
        } else {
            if (lane == 0) S.wred[b][cw] = make_float4(ms.m, ms.s, ka, kb);
            named_sync(kBarConsumers, NCT);
            tot = combine4(S.wred[b], NCW);
        }
        if (shared) {
            // send this CTA's part to every rank; the parts are collected just before this
            // row's pass B, one row later, so the exchange overlaps the next pass A.  Four
            // buffers: a peer writes buffer i + 4 only after its own collection of row
            // i + 2, which needs this CTA's part of row i + 2, sent after row i was read.
            cur.f |= ((nx & 3u) << 8) | (((nx >> 2) & 1u) << 10);
            ++nx;
            if (kfree ? collector && lane == 0 : ct == 0) {
                mbar_arrive_expect_tx(&S.xbar[cur.xb()], 16u * (uint32_t)c);
                const float4 mine = make_float4(tot.ms.m, tot.ms.s, tot.a, tot.b);
                for (int q = 0; q < c; ++q)
                    st_async_f32x4(map_to_rank(&S.xbuf[cur.xb()][rank], (uint32_t)q), mine,
                                   map_to_rank(&S.xbar[cur.xb()], (uint32_t)q));
            }
        } else if (kfree) {
            if (collector) {
                const float lnS = logf(tot.ms.s);
                if (lane == 0) {
                    S.rstat[ab] = make_float2(tot.ms.m, lnS);
                    mbar_arrive(&S.sbar[ab]);
                    if (P.lse_out) P.lse_out[r] = tot.ms.m + lnS;
                    if (P.stats_out) { P.stats_out[2 * r] = tot.ms.m; P.stats_out[2 * r + 1] = lnS; }
                    P.loss[r] = fmaf(tot.ms.m + lnS, tot.b, tot.a);
                }
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
        // pass B of the row two back is done (past this row's barrier, or every warp has
        // arrived for it): its support terms
        if (kKL && rk2 >= 0) {
            const uint32_t l2 = li - 2u;
            if (kfree && ct < P.k)
                wait_parity<false>(&S.bdone[l2 % kSupBufs], (l2 / kSupBufs) & 1u, &S.abort, &g_watchdog, P.wait_limit);
            scatter_support<T>(P, S, rk2, l2 % kSupBufs, ct);
        }
        // bf16: the label column of this row (slice coordinates; -1 none) for its rewrite
        if (kKL && sizeof(T) == 2 && ct == LT) {
            int jfull = -1;
            if (has_label && !bad) {
                const long long j = (long long)lab_r - P.col0;
                if (j >= 0 && j < ncols) jfull = (int)j;
            }
            S.erow[sb][2] = __int_as_float(jfull);
        }
        // ---- pass B of the previous row
        if (pend.r >= 0) {
            if (pend.shared()) settle<OP>(P, S, pend, ct, rank);
            else if (kfree) collect(P, S, pend);
            if (kKL && sizeof(T) == 2 && ct == 0) {
                // bf16: the row statistics for its support rewrite, two rows on
                const uint32_t pb = (li + kSupBufs - 1u) % kSupBufs;
                S.erow[pb][0] = pend.m;
                S.erow[pb][1] = pend.lnS;
            }
            pass_b<T, OP>(P, S, pend, g, ct, lane, l2cg);
            if (kfree) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.bdone[(li - 1u) % kSupBufs]);
            }
        }
        pend = cur;
        rk2 = rk1;
        rk1 = r;
        ++li;
        if (!more) break;
    }
    if (pend.r >= 0) {
        if (nobar && pend.shared()) collect_cluster(P, S, pend, ct, rank);
        else if (nobar) collect(P, S, pend);
        else if (pend.shared()) settle<OP>(P, S, pend, ct, rank);
        else if (kfree) collect(P, S, pend);
        if (kKL && sizeof(T) == 2 && ct == 0) {
            const uint32_t pb = (li + kSupBufs - 1u) % kSupBufs;
            S.erow[pb][0] = pend.m;
            S.erow[pb][1] = pend.lnS;
        }
        pass_b<T, OP>(P, S, pend, g, ct, lane, l2cg);
    }
    if (kKL && li > 0) {
        named_sync(kBarConsumers, NCT);
        if (rk2 >= 0) scatter_support<T>(P, S, rk2, (li - 2u) % kSupBufs, ct);
        scatter_support<T>(P, S, rk1, (li - 1u) % kSupBufs, ct);
    }
}

template <typename T, int OP, bool RES>
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
        for (int b = 0; b < kPartBufs; ++b) {
            mbar_init(&S.abar[b], NCW);
            mbar_init(&S.sbar[b], 1);
        }
        for (int b = 0; b < (int)kSupBufs; ++b) mbar_init(&S.bdone[b], NCW);
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

    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer<T, OP, RES>(P, S, rank, cid, ncl);
            drain(S, P.wait_limit);
        }
        __syncwarp();
    } else {
        if (RES) consumer_self<T, OP>(P, S, rank, cid, ncl);
        else consumer<T, OP>(P, S, rank, cid, ncl);
    }
    // no CTA may leave while a peer can still write into its shared memory
    if (c > 1) cluster_sync_all();
}

template <typename T>
const void* kernel_for_t(int op, bool res) {
    switch (op) {
        case kCeFused: return (const void*)row_kernel<T, kCeFused, true>;
        case kCeFwd: return (const void*)row_kernel<T, kCeFwd, false>;
        case kCeBwd: return (const void*)row_kernel<T, kCeBwd, false>;
        case kKl: return res ? (const void*)row_kernel<T, kKl, true> : (const void*)row_kernel<T, kKl, false>;
        default: return nullptr;
    }
}

const void* kernel_for(int op, bool res, int dtype) {
    return dtype == kBf16 ? kernel_for_t<__nv_bfloat16>(op, res) : kernel_for_t<float>(op, res);
}

constexpr int kMaxDev = 64;
constexpr int kFnSlots = 16;
std::atomic<int> g_attr_done[kMaxDev][kFnSlots];

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

int slot_of(int op, bool res, int dtype) { return (dtype == kBf16 ? 8 : 0) + op * 2 + (res ? 1 : 0); }

}  // namespace

cudaError_t launch_rows(int op, bool resident, const RowParams& P, int nclusters, cudaStream_t st) {
    const void* fn = kernel_for(op, resident, P.dtype);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = prepare(fn, slot_of(op, resident, P.dtype));
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
std::atomic<int> g_max_clusters[kMaxDev][kFnSlots][kMaxCluster + 1];

int row_max_clusters(int op, bool resident, int c, int dtype) {
    const void* fn = kernel_for(op, resident, dtype);
    const int slot = slot_of(op, resident, dtype);
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
