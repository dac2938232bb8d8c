// Teacher top-k of long rows in one streaming kernel (cortiq-engine train_head.rs, topk_rows:
// the k largest logits of a row, descending, ties to the lower column, and
// exp(v_q - v_0) / sum over the k).
//
// The single-kernel select (topk.cu) orders a row's survivors on the warps that stream
// the rows, so the HBM stream of a CTA stalls while it sorts.  Here one persistent CTA per
// SM takes rows r0 + blockIdx.x + i * gridDim.x and splits its warps three ways:
//
//   warp 0        producer: the row's 30 KB tiles into a ring of shared memory (1-D bulk
//                 copies signalled on mbarriers), evict-first in L2;
//   warps 1-15    filter: every value at or above a threshold T goes to the warp's own
//                 candidate region of the row -- each warp keeps its own count, so an
//                 admission costs a ballot and a store, no atomics.  T comes from the
//                 row's first tile: each warp's a-th largest of its share, averaged over
//                 the warps, with a chosen so that at least k values pass with a margin
//                 of about 5.5 standard deviations (128256 columns: about 3.4 k values
//                 pass at k = 2048, 0.9 k at k = 256);
//   warps 16-23   finish: while the filter warps stream row i + 1 they order row i: a
//                 histogram of NB value buckets over [T, max], the bucket that holds the
//                 k-th largest, the members of that bucket and of the ones above it ranked
//                 exactly by (value desc, column asc), and the first k written with their
//                 probabilities.
//
// A row's regions (two sets per CTA, rows alternate between them) sit in the caller's
// workspace and stay in L2 from the filter's writes to the finish's reads.  The result is
// exact iff at least k values passed T (then all of the top k did), no warp overflowed its
// region and the k-th largest's bucket fits the finish's arrays; a row that misses one of
// these goes on a list that the exact kernel takes afterwards (a launch that finds the
// list empty does nothing).
#include "vl_device.cuh"
#include "vl_internal.h"
#include "vl_topk.cuh"

#include "vloss.h"

#include <atomic>
#include <cmath>
#include <mutex>

namespace vl {
namespace {

constexpr int FW = kConsumerWarps;          // filter warps
constexpr int FT = FW * 32;
constexpr int NF = 8;                       // finish warps
constexpr int NFT = NF * 32;
constexpr int STHREADS = 32 + FT + NFT;
constexpr int FVEC = 4;                     // float4s of each tile per filter thread
constexpr int FTILE = 4 * FT * FVEC;        // floats per tile (30 KB)
constexpr int NSLOT = 5;                    // ring tiles (150 KB)
constexpr int NB = 2048;                    // value buckets of the finish
constexpr int KMAX = VL_TOPK_KMAX;
constexpr int SELCAP = KMAX + 2048;         // members of the buckets at and above the k-th's
constexpr uint32_t FBAR = 1, NBAR = 2;      // named barriers: filter warps, finish warps
constexpr int RT = 17;                      // finish threads per candidate region (15 x 17 = 255)
constexpr int FB = 16;                      // candidates a finish thread loads at once
constexpr long long kMaxStreamCols = 1LL << 20;

static_assert(FTILE / 4 == FT * FVEC, "FVEC float4s of each tile per filter thread");
static_assert(NB % NFT == 0, "buckets split evenly over the finish threads");
static_assert(FW * RT <= NFT, "a group of finish threads per region");
static_assert(KMAX % NFT == 0, "output positions split evenly over the finish threads");

__device__ unsigned int g_watchdog;

struct alignas(128) KSmem {
    float ring[NSLOT][FTILE];
    uint32_t hcnt[NB];
    uint32_t hpos[NB];
    uint32_t skey[SELCAP];
    uint32_t sid[SELCAP];
    uint32_t okey[KMAX];
    uint32_t oid[KMAX];
    uint64_t full[NSLOT];
    uint64_t empty[NSLOT];
    uint64_t rowdone[2];                    // the filter warps' records of a row are in
    uint64_t areafree[2];                   // the finish has read a row's regions
    float wspec[2][FW];                     // the warps' estimates (by row parity)
    float T[2];
    uint32_t wcnt[2][FW];                   // values each warp admitted (may exceed capw)
    float wmax[2][FW];                      // the largest value each warp admitted
    int wnan[2][FW];
    uint32_t fred[NF];
    float zred[NF];
    uint32_t bstar, nsel;
    uint32_t fin_lo, fin_hi;                // the row's bucket range, as keys
    int fin_hist, fin_nan;                  // the finish's decisions, taken by one thread
    int abort;
    uint32_t issued;
};

static_assert(sizeof(KSmem) <= 227 * 1024, "shared memory of one CTA");

struct StreamParams {
    const float* x;
    long long ld;
    int V, K;
    long long r0, r1;         // rows of the launch
    uint2* cand;              // regions: ((blockIdx.x * 2 + parity) * FW + warp) * capw
    int capw;
    int* list;                // rows the exact kernel takes
    int* nlist;
    int* err;
    uint32_t* ids;
    float* probs;
    int spec_a;               // rank of a warp's estimate within its share of the first tile
    long long wait_limit;
};

__device__ __forceinline__ void row_cut(const float* rowp, int V, int& h, int& bt) {
    const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
    h = (4 - mis) & 3;
    if (h > V) h = V;
    bt = (V - h) & ~3;
}

__device__ __forceinline__ uint2* region(const StreamParams& F, uint32_t p) {
    return F.cand + ((long long)blockIdx.x * 2 + p) * FW * (long long)F.capw;
}

// ---------------------------------------------------------------- producer

__device__ void producer(const StreamParams& F, KSmem& S) {
    uint32_t g = 0;
    const uint64_t pol = l2_evict_first();           // each logit is read once
    for (long long r = F.r0 + blockIdx.x; r < F.r1; r += gridDim.x) {
        const float* rowp = F.x + r * F.ld;
        int h, bt;
        row_cut(rowp, F.V, h, bt);
        for (int c0 = 0; c0 < bt; c0 += FTILE) {
            const uint32_t slot = g % NSLOT, use = g / NSLOT;
            if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog, F.wait_limit)) {
                S.issued = g;
                return;
            }
            const uint32_t bytes = (uint32_t)min(FTILE, bt - c0) * 4u;
            mbar_arrive_expect_tx(&S.full[slot], bytes);
            bulk_g2s_hint(S.ring[slot], rowp + h + c0, bytes, &S.full[slot], pol);
            ++g;
        }
    }
    S.issued = g;
}

__device__ void producer_drain(KSmem& S, long long limit) {
    const uint32_t iss = S.issued;
    for (uint32_t gt = iss > (uint32_t)NSLOT ? iss - NSLOT : 0u; gt < iss; ++gt)
        wait_parity_drain(&S.full[gt % NSLOT], (gt / NSLOT) & 1u, limit);
}

// ---------------------------------------------------------------- filter

// Append the lanes' (v, id) with keep set to this warp's region: slots in lane order after
// the warp's count (warp-uniform), which grows by the ballot's size even past capw.
__device__ __forceinline__ void admit(uint2* out, uint32_t capw, uint32_t& wcnt, float& wmax, bool keep, float v,
                                      uint32_t id, uint64_t pol) {
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (!bal) return;
    const uint32_t pos = wcnt + (uint32_t)__popc(bal & lanemask_lt());
    if (keep) {
        wmax = fmaxf(wmax, v);
        if (pos < capw)
            asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;"
                         :: "l"(out + pos), "r"(__float_as_uint(v)), "r"(id), "l"(pol) : "memory");
    }
    wcnt += (uint32_t)__popc(bal);
}

// max with NaN propagation (max.NaN): a NaN among the operands gives NaN.
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Value q of e[16] for a lane-varying q: a four-level select tree.
__device__ __forceinline__ float pick16(const float (&e)[16], uint32_t q) {
    const bool b0 = q & 1u, b1 = q & 2u, b2 = q & 4u, b3 = q & 8u;
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = b0 ? e[2 * i + 1] : e[2 * i];
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = b1 ? t[2 * i + 1] : t[2 * i];
    const float w0 = b2 ? u[1] : u[0], w1 = b2 ? u[3] : u[2];
    return b3 ? w1 : w0;
}

// Admit this lane's 16 values of a tile (float4 u at columns cu[u] .. cu[u] + 3) that reach
// T to the warp's region, all lanes at once: the lane's keep mask and count c (0..16), one
// ballot per bit plane of c gives every lane its slot offset (the lanes below it), redux the
// warp's total; then each lane stores its kept values in column order, one loop iteration
// per kept value (the warp runs as many as its busiest lane: two or three at a few percent
// admitted).  A lane whose slots would pass capw stores nothing (the warp's count passes
// capw: the row goes to the exact kernel).
__device__ __forceinline__ void admit16(uint2* out, uint32_t capw, uint32_t& wcnt, float& wmax, bool& nan,
                                        const float4 (&v)[FVEC], const uint32_t (&cu)[FVEC], const bool (&act)[FVEC],
                                        float T, uint64_t pol) {
    static_assert(FVEC == 4, "16 values a lane: five bit planes");
    float e[16];
#pragma unroll
    for (int u = 0; u < FVEC; ++u) {
        e[4 * u] = v[u].x;
        e[4 * u + 1] = v[u].y;
        e[4 * u + 2] = v[u].z;
        e[4 * u + 3] = v[u].w;
    }
    uint32_t km = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q)
        if (act[q >> 2] && e[q] >= T) km |= 1u << q;   // slots past the row's body hold -inf, which T = -inf admits
    float mx = e[0];
#pragma unroll
    for (int q = 1; q < 16; ++q) mx = max_nan(mx, e[q]);
    nan |= mx != mx;
    if (!__any_sync(0xffffffffu, km != 0)) return;
    const uint32_t c = (uint32_t)__popc(km);
    const uint32_t lt = lanemask_lt();
    uint32_t pos = wcnt;
#pragma unroll
    for (int b = 0; b < 5; ++b) pos += (uint32_t)__popc(__ballot_sync(0xffffffffu, (c >> b) & 1u) & lt) << b;
    wcnt += __reduce_add_sync(0xffffffffu, c);
    if (km != 0) wmax = fmaxf(wmax, mx);          // mx is NaN only with a NaN here; fmaxf skips it
    if (pos + c > capw) km = 0;
    uint2* o = out + pos;
    while (km) {
        const uint32_t q = (uint32_t)(__ffs(km) - 1);
        km &= km - 1u;
        const uint32_t col = cu[0] + (q >> 2) * (uint32_t)(4 * FT) + (q & 3u);
        asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;"
                     :: "l"(o), "r"(__float_as_uint(pick16(e, q))), "r"(col), "l"(pol) : "memory");
        ++o;
    }
}

// The filter warps never leave a barrier out: a wait that gave up (the CTA's abort flag is
// then set and every later wait returns at once) is followed by the same steps on whatever
// the buffers hold, and the host reports the watchdog.
__device__ void filter_warps(const StreamParams& F, KSmem& S) {
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const uint64_t keep_pol = l2_evict_last();
    const uint32_t capw = (uint32_t)F.capw;
    uint32_t g = 0, i = 0;
    for (long long r = F.r0 + blockIdx.x; r < F.r1; r += gridDim.x, ++i) {
        const float* rowp = F.x + r * F.ld;
        int h, bt;
        row_cut(rowp, F.V, h, bt);
        const int t0 = h + bt;
        const int nt = (bt + FTILE - 1) / FTILE;
        const uint32_t p = i & 1u;
        uint2* out = region(F, p) + (long long)cw * capw;
        // the finish is done with these regions (row i - 2's)
        if (i >= 2) wait_parity<false>(&S.areafree[p], ((i >> 1) - 1u) & 1u, &S.abort, &g_watchdog, F.wait_limit);
        float T = -INFINITY, wmax = -INFINITY;
        uint32_t wcnt = 0;
        bool nan = false;
        for (int t = 0; t < nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % NSLOT;
            wait_parity<false>(&S.full[slot], (gt / NSLOT) & 1u, &S.abort, &g_watchdog, F.wait_limit);
            const int n4 = min(FTILE, bt - t * FTILE) >> 2;
            float4 v[FVEC];
#pragma unroll
            for (int u = 0; u < FVEC; ++u) {
                const int j = u * FT + ct;
                v[u] = j < n4 ? ld_shared_v4(&S.ring[slot][j * 4]) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            if (t == 0) {
                // the threshold from the first tile (every row here has at least 4 full tiles)
                const float e = warp_kth<FVEC>(v, (uint32_t)F.spec_a, lane);
                if (lane == 0) S.wspec[p][cw] = e;
                named_sync(FBAR, FT);
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < FW; ++w) sum += S.wspec[p][w];
                T = sum * (1.0f / FW);
                if (ct == 0) S.T[p] = T;
                // the head and tail columns (at most 3 + 3), now that T is known
                if (cw == 0) {
                    bool keep = false;
                    float hv = 0.f;
                    uint32_t id = 0;
                    if (lane < h) { id = (uint32_t)lane; hv = rowp[id]; keep = true; }
                    else if (lane >= 4 && lane - 4 < F.V - t0) { id = (uint32_t)(t0 + lane - 4); hv = rowp[id]; keep = true; }
                    if (keep && isnan(hv)) { keep = false; nan = true; }
                    admit(out, capw, wcnt, wmax, keep && hv >= T, hv, id, keep_pol);
                }
            }
            uint32_t cu[FVEC];
            bool act[FVEC];
#pragma unroll
            for (int u = 0; u < FVEC; ++u) {
                cu[u] = (uint32_t)(h + t * FTILE + 4 * (u * FT + ct));
                act[u] = u * FT + ct < n4;
            }
            admit16(out, capw, wcnt, wmax, nan, v, cu, act, T, keep_pol);
        }
        g += (uint32_t)nt;
        // the warp's record of the row; the arrive releases it and the region's stores
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
        const bool wnan = __any_sync(0xffffffffu, nan);
        __syncwarp();
        if (lane == 0) {
            S.wcnt[p][cw] = wcnt;
            S.wmax[p][cw] = wmax;
            S.wnan[p][cw] = wnan ? 1 : 0;
            mbar_arrive(&S.rowdone[p]);
        }
    }
}

// ---------------------------------------------------------------- finish

// Buckets of the finish: NB equal bins of [lo value, hi value] when that range is finite and
// not empty, else an 11-bit window of (key - lo).  Non-decreasing in the key either way, so
// a higher bucket never holds a smaller value.
struct Buckets {
    bool lin;
    float vmin, scale;
    uint32_t lo;
    int s2;
    __device__ Buckets(uint32_t lo_key, uint32_t hi_key) {
        lo = lo_key;
        vmin = key2f(lo_key);
        const float range = key2f(hi_key) - vmin;
        lin = range > 0.f && range < INFINITY;
        scale = lin ? (float)NB / range : 0.f;
        const uint32_t R = hi_key > lo_key ? hi_key - lo_key : 0u;
        const int nbits = R ? 32 - __clz(R) : 0;
        s2 = nbits > 11 ? nbits - 11 : 0;
    }
    __device__ __forceinline__ uint32_t operator()(uint32_t kk) const {
        if (lin) return (uint32_t)fminf((float)(NB - 1), fmaxf(0.f, (key2f(kk) - vmin) * scale));
        return min((uint32_t)(NB - 1), (kk > lo ? kk - lo : 0u) >> s2);
    }
};

__device__ void finish_warps(const StreamParams& F, KSmem& S) {
    const int ft = (int)threadIdx.x - 32 - FT;
    const int fw = ft >> 5, lane = ft & 31;
    const uint32_t K = (uint32_t)F.K, capw = (uint32_t)F.capw;
    uint32_t i = 0;
    for (long long r = F.r0 + blockIdx.x; r < F.r1; r += gridDim.x, ++i) {
        const uint32_t p = i & 1u;
        wait_parity<false>(&S.rowdone[p], (i >> 1) & 1u, &S.abort, &g_watchdog, F.wait_limit);
        // past this barrier the previous row's use of the histogram (and its clearing) is over;
        // one thread reads the warps' records and takes the row's decisions, so that the
        // branches around the barriers below are the same for every finish thread
        named_sync(NBAR, NFT);
        if (ft == 0) {
            uint32_t n = 0;
            bool over = false, nan = false;
            float vmax = -INFINITY;
#pragma unroll
            for (int w = 0; w < FW; ++w) {
                const uint32_t c = S.wcnt[p][w];
                n += c;
                over |= c > capw;
                vmax = fmaxf(vmax, S.wmax[p][w]);
                nan |= S.wnan[p][w] != 0;
            }
            S.fin_hist = !over && n >= K;
            S.fin_nan = nan;
            S.fin_lo = f2key(S.T[p]);
            S.fin_hi = f2key(vmax);
            S.nsel = 0xffffffffu;                // stays so unless the scan finds the k-th's bucket
        }
        named_sync(NBAR, NFT);
        const bool hist = S.fin_hist != 0, nan = S.fin_nan != 0;
        const Buckets bucket(S.fin_lo, S.fin_hi);
        const uint2* area = region(F, p);
        bool ok = hist;
        uint32_t bstar = 0, nsel = 0;
        // each region is read by its own group of RT threads, FB candidates a thread at a time:
        // the loads of a pass go out together, one L2 round trip while the stream loads L2
        const int rw = ft / RT, rs = ft % RT;
        const uint32_t rc = rw < FW ? min(S.wcnt[p][rw], capw) : 0u;
        const uint2* rin = area + (long long)(rw < FW ? rw : 0) * capw;
        if (hist) {
            for (uint32_t j0 = (uint32_t)rs; j0 < rc; j0 += RT * FB) {
                uint32_t x[FB];
#pragma unroll
                for (int i = 0; i < FB; ++i) {
                    const uint32_t j = j0 + (uint32_t)(i * RT);
                    if (j < rc) x[i] = rin[j].x;
                }
#pragma unroll
                for (int i = 0; i < FB; ++i)
                    if (j0 + (uint32_t)(i * RT) < rc) atomicAdd(&S.hcnt[bucket(f2key(__uint_as_float(x[i])))], 1u);
            }
            named_sync(NBAR, NFT);
            // bucket starts in descending order; thread ft owns buckets [c0, c0 + PER)
            constexpr int PER = NB / NFT;
            const int c0 = ft * PER;
            uint32_t loc = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) loc += S.hcnt[c0 + q];
            uint32_t suf = loc;                  // sum over this lane and the lanes above
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t t = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane + off < 32) suf += t;
            }
            if (lane == 0) S.fred[fw] = suf;
            named_sync(NBAR, NFT);
            uint32_t a = suf - loc;
            for (int ww = fw + 1; ww < NF; ++ww) a += S.fred[ww];
#pragma unroll
            for (int q = PER - 1; q >= 0; --q) {
                const uint32_t b = (uint32_t)(c0 + q), hb = S.hcnt[b];
                S.hpos[b] = a;
                if (a < K && a + hb >= K) {     // the bucket of the k-th largest (one, as n >= K)
                    S.bstar = b;
                    S.nsel = a + hb;
                }
                a += hb;
            }
            named_sync(NBAR, NFT);
            bstar = S.bstar;
            nsel = S.nsel;
            ok = nsel <= (uint32_t)SELCAP;
            if (ok) {
                for (uint32_t j0 = (uint32_t)rs; j0 < rc; j0 += RT * FB) {
                    uint2 e[FB];
#pragma unroll
                    for (int i = 0; i < FB; ++i) {
                        const uint32_t j = j0 + (uint32_t)(i * RT);
                        if (j < rc) e[i] = rin[j];
                    }
#pragma unroll
                    for (int i = 0; i < FB; ++i) {
                        if (j0 + (uint32_t)(i * RT) >= rc) continue;
                        const uint32_t kk = f2key(__uint_as_float(e[i].x));
                        const uint32_t b = bucket(kk);
                        if (b >= bstar) {
                            const uint32_t q = atomicAdd(&S.hpos[b], 1u);
                            if (q < (uint32_t)SELCAP) {
                                S.skey[q] = kk;
                                S.sid[q] = e[i].y;
                            }
                        }
                    }
                }
            }
        }
        // every read of the row's regions is done: hand them back to the filter warps
        named_sync(NBAR, NFT);
        if (ft == 0) {
            mbar_arrive(&S.areafree[p]);
            if (!ok) F.list[atomicAdd(F.nlist, 1)] = (int)r;
            if (nan && F.err) atomicAdd(F.err, 1);
        }
        if (ok) {
            // exact rank: the bucket's start plus the members ahead of it in (key desc, id asc)
            for (uint32_t q = (uint32_t)ft; q < nsel; q += NFT) {
                const uint32_t kk = S.skey[q], id = S.sid[q];
                const uint32_t b = bucket(kk);
                const uint32_t end = min(S.hpos[b], (uint32_t)SELCAP), hb = S.hcnt[b];
                const uint32_t beg = hb < end ? end - hb : 0u;
                const unsigned long long me = comp(kk, id);
                uint32_t rank = beg;
                for (uint32_t j = beg; j < end; ++j) rank += comp(S.skey[j], S.sid[j]) > me ? 1u : 0u;
                if (rank < K) {
                    S.okey[rank] = kk;
                    S.oid[rank] = id;
                }
            }
            named_sync(NBAR, NFT);
        }
        if (hist)
            for (int b = ft; b < NB; b += NFT) S.hcnt[b] = 0u;
        if (ok) {
            // probabilities renormalised over the k
            // (each thread keeps the exponentials of its positions for the write)
            constexpr int QPT = KMAX / NFT;
            const float v0 = key2f(S.okey[0]);
            float ez[QPT];
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < QPT; ++i) {
                const uint32_t q = (uint32_t)(ft + i * NFT);
                ez[i] = q < K ? expf(key2f(S.okey[q]) - v0) : 0.f;
                part += ez[i];
            }
            part = warp_sum(part);
            if (lane == 0) S.zred[fw] = part;
            named_sync(NBAR, NFT);
            float Z = 0.f;
#pragma unroll
            for (int w = 0; w < NF; ++w) Z += S.zred[w];
            const float rZ = 1.0f / Z;
            uint32_t* oi = F.ids + r * (long long)K;
            float* op = F.probs + r * (long long)K;
#pragma unroll
            for (int i = 0; i < QPT; ++i) {
                const uint32_t q = (uint32_t)(ft + i * NFT);
                if (q < K) {
                    oi[q] = S.oid[q];
                    op[q] = ez[i] * rZ;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(STHREADS, 1) topk_stream_kernel(const __grid_constant__ StreamParams F) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    KSmem& S = *reinterpret_cast<KSmem*>(smem_raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], FW);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&S.rowdone[q], FW);
            mbar_init(&S.areafree[q], 1);
        }
        S.abort = 0;
        S.issued = 0;
        fence_mbar_init_cluster();
    }
    for (int b = (int)threadIdx.x; b < NB; b += STHREADS) S.hcnt[b] = 0u;
    __syncthreads();
    pdl_wait_primary();
    pdl_launch_dependents();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer(F, S);
            producer_drain(S, F.wait_limit);
        }
        __syncwarp();
    } else if (threadIdx.x < 32 + FT) {
        filter_warps(F, S);
    } else {
        finish_warps(F, S);
    }
}

std::atomic<int> g_stream_attr[64];

long long list_bytes(long long rows) { return (16 + 4 * rows + 255) / 256 * 256; }

}  // namespace

// Rows qualify when they have at least 4 full tiles (the first one is a sample of the row),
// at most 2^20 columns, and the warp estimates' rank stays small.  Each warp's estimate is
// the a-th largest of its 512 values of the first tile, about a V / 512 values of the row
// pass T, and the count's relative spread is about 1 / sqrt(15 a) (the mean of 15 order
// statistics).  a is the smallest rank that keeps k at least 5.5 spreads below the mean:
// a = 14 for k = 2048 of 128256 columns (mean 3449 admitted, standard deviation 228 over
// the 4096 teacher rows, first tiles simulated), a = 4 for k = 256 (919 and 122).
int topk_filter_spec_a(long long V, int k) {
    if (V < 4LL * FTILE || V > kMaxStreamCols) return 0;
    const double share = (double)k * (double)(FTILE / FW) / (double)V;
    for (int a = 2; a <= FTILE / FW / 8; ++a)
        if ((double)a * 0.97 / share * (1.0 - 5.5 / sqrt(15.0 * a)) >= 1.0) return a;
    return 0;
}

// Slots of a warp's region: the expected admissions m = a V / (256 * 15), plus six binomial
// deviations, half of m for rows whose threshold lands low, and 32.
int topk_filter_capw(long long V, int k) {
    const int a = topk_filter_spec_a(V, k);
    if (a == 0) return 0;
    const double m = (double)a * (double)V / (double)(FTILE / FW) / (double)FW;
    const long long c = (long long)ceil(m + 6.0 * sqrt(m) + 0.5 * m + 32.0);
    return (int)((c + 31) / 32 * 32);
}

long long topk_cta_bytes(long long V, int k) { return 2LL * FW * topk_filter_capw(V, k) * (long long)sizeof(uint2); }

// Workspace: [0, 16) the list's length; the list (4 bytes a row); then, 256-byte aligned,
// two sets of FW regions of capw (value bits, column) slots for each of `ctas` CTAs.
long long topk_ws_bytes(long long rows, long long V, int k, long long ctas) {
    return list_bytes(rows) + ctas * topk_cta_bytes(V, k);
}

cudaError_t launch_topk_stream(const float* x, long long ld, long long V, int k, long long ls, long long le,
                               uint32_t* ids, float* probs, int* err, void* ws, long long ws_bytes,
                               long long wait_limit, cudaStream_t st) {
    const int a = topk_filter_spec_a(V, k);
    if (a == 0 || k > KMAX) return cudaErrorInvalidValue;
    const long long rows = le - ls;
    if (rows <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (!g_stream_attr[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute((const void*)topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(KSmem));
        if (e != cudaSuccess) return e;
        g_stream_attr[dev].store(1, std::memory_order_release);
    }
    // CTAs: one per SM, at most one per row, as many as the workspace holds regions for
    const long long cb = topk_cta_bytes(V, k);
    long long grid = rows < sms ? rows : sms;
    const long long fit = (ws_bytes - list_bytes(rows)) / cb;
    if (fit < grid) grid = fit;
    if (grid < 1) return cudaErrorInvalidValue;
    char* base = static_cast<char*>(ws);
    int* nlist = reinterpret_cast<int*>(base);
    int* list = reinterpret_cast<int*>(base + 16);
    if ((e = cudaMemsetAsync(nlist, 0, sizeof(int), st)) != cudaSuccess) return e;
    StreamParams F;
    F.x = x;
    F.ld = ld;
    F.V = (int)V;
    F.K = k;
    F.r0 = ls;
    F.r1 = le;
    F.cand = reinterpret_cast<uint2*>(base + list_bytes(rows));
    F.capw = topk_filter_capw(V, k);
    F.list = list;
    F.nlist = nlist;
    F.err = err;
    F.ids = ids;
    F.probs = probs;
    F.spec_a = a;
    F.wait_limit = wait_limit;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(STHREADS, 1, 1);
    cfg.dynamicSmemBytes = sizeof(KSmem);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, topk_stream_kernel, F)) != cudaSuccess) return e;
    // the rows the stream could not settle, exactly (NaN rows were counted already)
    return launch_topk(x, ld, le, V, k, ls, le, list, nlist, ids, probs, nullptr, st);
}

// ---------------------------------------------------------------- scratch without allocation
//
// For callers that cannot allocate device memory: the stream kernel's scratch in a fixed
// array that every device loading the library holds until the process exits.  Host code
// needs the array's device address (the symbol itself names a host-side stand-in); it is
// looked up once per device, with that device current.

static __device__ __align__(256) unsigned char g_noalloc_scratch[VL_TOPK_NOALLOC_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};
}  // namespace

cudaError_t topk_noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

unsigned int topk_stream_watchdog(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_watchdog, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_watchdog, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}

}  // namespace vl
