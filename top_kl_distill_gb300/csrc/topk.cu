// Exact teacher top-k per row with probabilities renormalised over the k
// (cortiq-engine train_head.rs, topk_rows: the k largest logits of a row,
// descending, and exp(v_q - v_0) / sum over the k).
//
// The page keeps each thread's best 8 of a strided scan and bitonic-sorts the
// 2048 survivors, which misses true top-k members when more than 8 of them
// share a residue class and breaks ties arbitrarily.  This kernel is exact, with
// ties going to the lower column:
//
//   * one persistent CTA per SM streams its rows through a ring of 15 KB tiles
//     (1-D bulk copies, producer warp + 15 consumer warps, as the row engine);
//   * each consumer warp owns a region of the shared candidate buffer and streams
//     its float4s of every tile on its own (no barrier per tile): values at or
//     above the admission threshold T are appended with one ballot per float4 group;
//   * speculation: on a long row each warp estimates, from its share of the first
//     tile, the value that about 1.4 k of the row's values reach, and T starts at the
//     warps' mean estimate.  The answer is exact when at least k values of the row
//     reach T (or a cut below proved a higher bound), which the end of the row
//     checks; otherwise the row is redone exactly, read again from global memory;
//   * cuts: a warp whose region could overflow on its next tile (or, without
//     speculation, that sees the candidate total pass a few times k) raises a
//     shared flag; every warp checks it before each tile and while waiting for one,
//     and all cut together: the candidates are counted into equal bins of their
//     value range, everything from the bin holding the k-th largest up is kept
//     (spread over the regions) and the smallest kept value becomes T, a lower bound
//     of the row's k-th largest.  Crowded or degenerate ranges fall back to an exact
//     MSD radix select over order-preserving keys (-0.0 folded into +0.0), the k-th
//     key's ties kept by lowest column;
//   * at the end of the row at most k + 1024 survivors are placed into 2048 value
//     buckets in descending order, ranked exactly by (value desc, id asc) within
//     their bucket, and the first k written with their probabilities.
#include "vl_device.cuh"
#include "vl_internal.h"
#include "vl_topk.cuh"

#include <atomic>

namespace vl {
namespace {

constexpr int NCW = kConsumerWarps;
constexpr int NCT = NCW * 32;
constexpr int NTHREADS = NCT + 32;
constexpr int kVecT = 2;                   // float4s of each tile per consumer thread
constexpr int kTileT = 4 * NCT * kVecT;    // floats per tile (15 KB)
constexpr int kSlotsT = 7;                 // ring tiles (105 KB)
constexpr int RW = 512;                    // candidate entries per consumer warp
constexpr int CB = RW * NCW;               // candidate buffer entries
constexpr int NPER = RW / 32;              // candidates per lane while cutting
constexpr int KMAXT = 2048;
constexpr int SLACK = 1024;                // survivors beyond k the final ordering takes
constexpr int KOUT = KMAXT + SLACK;
constexpr int DBC = 10;                    // digit bits of one exact cut round
constexpr int NBC = 1024;                  // linear bins of a cut
constexpr int NBK = 2048;                  // buckets of the final ordering
constexpr int PER_TILE = kTileT / NCW;     // most candidates a warp can add per tile
constexpr int LIMIT_MAX = NCW * (RW - PER_TILE - 8);   // survivors that leave each region room for a tile
constexpr uint32_t kBar = 1;

static_assert(kTileT / 4 == NCT * kVecT, "kVecT float4s of each tile per consumer thread");
static_assert(8 + PER_TILE <= RW, "the row's head and tail plus one tile fit an empty region");
static_assert(KMAXT + KMAXT / 8 <= LIMIT_MAX, "cuts keep at most LIMIT_MAX");
static_assert((1 << DBC) <= NBK && (NBK & (NBK - 1)) == 0, "histogram sizes");
static_assert(KOUT <= CB, "the final order is written over the candidate buffer");

__device__ unsigned int g_watchdog;

struct alignas(128) TSmem {
    float ring[kSlotsT][kTileT];
    uint64_t full[kSlotsT];
    uint64_t empty[kSlotsT];
    float cval[CB];                  // candidate values, region w = [w * RW, (w + 1) * RW)
    uint32_t cid[CB];
    uint32_t hcnt[NBK];              // digit histogram / bucket sizes
    uint32_t hpos[NBK];              // bucket starts in descending order
    uint32_t okey[KOUT];             // survivors in bucket order: key, id
    uint32_t oid[KOUT];
    uint32_t wtmp[2][NCW];
    uint32_t wcnt[NCW];
    uint32_t wadm[NCW];              // values each warp admitted
    float wspec[NCW];                // each warp's estimate of the speculative threshold
    float zred[NCW];
    uint32_t sel[4];
    uint32_t total;                  // candidates held, counted up as warps append
    int need;                        // a warp asks for a cut
    int nanrow;                      // a NaN was seen in the current row
    int abort;
    uint32_t issued;
};

static_assert(sizeof(TSmem) <= 227 * 1024, "shared memory of one CTA");

// ---------------------------------------------------------------- producer

// Rows of a launch: [ls, le), or the `nlist` rows of `list` (the rows a filtered launch
// could not finish).
struct Rows {
    long long ls;
    long long n;
    const int* list;
    __device__ __forceinline__ long long at(long long i) const { return list ? (long long)list[i] : ls + i; }
};

__device__ void producer(const float* x, long long ld, long long V, const Rows& R, TSmem& S) {
    uint32_t g = 0;
    for (long long i = blockIdx.x; i < R.n; i += gridDim.x) {
        const long long r = R.at(i);
        const float* rowp = x + r * ld;
        const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        int h = (4 - mis) & 3;
        if (h > V) h = (int)V;
        const int bt = ((int)V - h) & ~3;
        for (int c0 = 0; c0 < bt; c0 += kTileT) {
            const uint32_t slot = g % kSlotsT, use = g / kSlotsT;
            if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog)) {
                S.issued = g;
                return;
            }
            const uint32_t bytes = (uint32_t)min(kTileT, bt - c0) * 4u;
            mbar_arrive_expect_tx(&S.full[slot], bytes);
            bulk_g2s(S.ring[slot], rowp + h + c0, bytes, &S.full[slot]);
            ++g;
        }
    }
    S.issued = g;
}

__device__ void drain(TSmem& S) {
    const uint32_t iss = S.issued;
    for (uint32_t gt = iss > (uint32_t)kSlotsT ? iss - kSlotsT : 0u; gt < iss; ++gt)
        wait_parity_drain(&S.full[gt % kSlotsT], (gt / kSlotsT) & 1u);
}

// ---------------------------------------------------------------- block-wide helpers (consumer threads)

// Append `keep` lanes' (value, id) to this warp's region; cnt is the warp's count.
__device__ __forceinline__ void wappend(TSmem& S, int cw, uint32_t& cnt, bool keep, float v, uint32_t id) {
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (keep) {
        const uint32_t pos = (uint32_t)cw * RW + cnt + (uint32_t)__popc(bal & lanemask_lt());
        S.cval[pos] = v;
        S.cid[pos] = id;
    }
    cnt += (uint32_t)__popc(bal);
}

// Block-wide min and max of u32s.  The caller separates the next use of S.wtmp by a barrier.
__device__ __forceinline__ void block_minmax(uint32_t& lo, uint32_t& hi, TSmem& S, int ct) {
    const int cw = ct >> 5, lane = ct & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    if (lane == 0) { S.wtmp[0][cw] = lo; S.wtmp[1][cw] = hi; }
    named_sync(kBar, NCT);
    lo = S.wtmp[0][0];
    hi = S.wtmp[1][0];
#pragma unroll
    for (int w = 1; w < NCW; ++w) { lo = min(lo, S.wtmp[0][w]); hi = max(hi, S.wtmp[1][w]); }
}

// Sum of v over the consumer threads with a higher index.  The caller separates the
// next use of S.wtmp by a barrier.
__device__ __forceinline__ uint32_t block_above(uint32_t v, TSmem& S, int ct) {
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t suf = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += t;
    }
    if (lane == 0) S.wtmp[0][cw] = suf;
    named_sync(kBar, NCT);
    uint32_t a = suf - v;
    for (int w = cw + 1; w < NCW; ++w) a += S.wtmp[0][w];
    return a;
}

struct Cut {
    uint32_t tk;     // keep the keys >= tk
    uint32_t ge;     // keys >= tk
    uint32_t gt;     // keys > tk (exact cuts)
    bool exact;      // tk is the K-th largest key itself
};

// Over the keys f[j] of the slots with bit j of vmask set (K <= their count): a key
// tk with K <= #(f >= tk).  MSD digit rounds of DBC bits over the range [min, max]
// present narrow the bin holding the K-th largest key until #(f >= its lower edge)
// <= limit, or until the bin is one key (then tk is the K-th largest key, exact).
__device__ Cut select_cut(const uint32_t (&f)[NPER], uint32_t vmask, uint32_t K, uint32_t limit, TSmem& S, int ct) {
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (vmask >> j & 1u) { lo = min(lo, f[j]); hi = max(hi, f[j]); }
    block_minmax(lo, hi, S, ct);
    const uint32_t R = hi - lo;
    int shift = R ? 32 - __clz(R) : 0;
    uint32_t prefix = 0, rem = K, abv = 0;
    for (;;) {
        const int bits = shift < DBC ? shift : DBC;
        shift -= bits;
        const int nb = 1 << bits;
        for (int i = ct; i < nb; i += NCT) S.hcnt[i] = 0u;
        named_sync(kBar, NCT);
#pragma unroll
        for (int j = 0; j < NPER; ++j) {
            if (vmask >> j & 1u) {
                const uint32_t u = f[j] - lo;
                const uint32_t top = (shift + bits >= 32) ? 0u : (u >> (shift + bits));
                if (top == prefix) atomicAdd(&S.hcnt[(u >> shift) & (uint32_t)(nb - 1)], 1u);
            }
        }
        named_sync(kBar, NCT);
        // thread ct owns bins [c0, c1); the bin holding the K-th largest is found from the top
        const int per = (nb + NCT - 1) / NCT;
        const int c0 = min(nb, ct * per), c1 = min(nb, c0 + per);
        uint32_t loc = 0;
        for (int i = c0; i < c1; ++i) loc += S.hcnt[i];
        uint32_t a = block_above(loc, S, ct);
        for (int i = c1 - 1; i >= c0; --i) {
            const uint32_t c = S.hcnt[i];
            if (a < rem && rem <= a + c) { S.sel[0] = (uint32_t)i; S.sel[1] = a; S.sel[2] = c; }
            a += c;
        }
        named_sync(kBar, NCT);
        const uint32_t b = S.sel[0], ab = S.sel[1], cb = S.sel[2];
        abv += ab;
        rem -= ab;
        prefix = (prefix << bits) | b;
        const uint32_t ge = abv + cb;
        if (shift == 0) return Cut{lo + prefix, ge, abv, true};
        if (ge <= limit) return Cut{lo + (prefix << shift), ge, abv, false};
        named_sync(kBar, NCT);   // S.sel and S.hcnt are reused
    }
}

// This warp's candidates into registers: key[j], id[j] for slot lane + 32 j < cnt.
__device__ __forceinline__ uint32_t load_region(const TSmem& S, int cw, int lane, uint32_t cnt, uint32_t (&key)[NPER],
                                                uint32_t (&id)[NPER]) {
    uint32_t vmask = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const uint32_t i = (uint32_t)lane + 32u * j;
        key[j] = 0u;
        id[j] = 0u;
        if (i < cnt) {
            id[j] = S.cid[cw * RW + i];
            key[j] = f2key(S.cval[cw * RW + i]);
            vmask |= 1u << j;
        }
    }
    return vmask;
}

// Which loaded candidates survive when tot > K: keys >= a cut that keeps at most `limit`
// (and at least K); when ties at the exact K-th key exceed that, exactly K, the tied
// keys by lowest id.  *tk is the cut key.
__device__ uint32_t choose(const uint32_t (&key)[NPER], const uint32_t (&id)[NPER], uint32_t vmask, uint32_t K,
                           uint32_t limit, TSmem& S, int ct, uint32_t* tk) {
    const Cut c = select_cut(key, vmask, K, limit, S, ct);
    *tk = c.tk;
    uint32_t idmax = 0xffffffffu;
    if (c.exact && c.ge > limit) {
        uint32_t nid[NPER];
        uint32_t emask = 0;
#pragma unroll
        for (int j = 0; j < NPER; ++j) {
            nid[j] = ~id[j];
            if ((vmask >> j & 1u) && key[j] == c.tk) emask |= 1u << j;
        }
        named_sync(kBar, NCT);
        const uint32_t need = K - c.gt;
        const Cut ci = select_cut(nid, emask, need, need, S, ct);   // ids are distinct: exactly `need`
        idmax = ~ci.tk;
    }
    uint32_t keep = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool kj = (vmask >> j & 1u) && (key[j] > c.tk || (key[j] == c.tk && id[j] <= idmax));
        keep |= (uint32_t)kj << j;
    }
    return keep;
}

// A cut over linear bins of the value range: the loaded candidates (keys, vmask) fall into
// NBC equal bins of [min, max]; the bins from the one holding the K-th largest value up
// are kept when they hold at most `limit` candidates.  The bin index is a monotone
// function of the value, so the kept set holds the K largest.  Returns false (nothing
// decided) when the range is empty or not finite, or the boundary bin is too crowded.
// S.hcnt[0, NBC) must be zero on entry and is zero again on return.
__device__ bool linear_cut(const uint32_t (&key)[NPER], uint32_t vmask, uint32_t K, uint32_t limit, TSmem& S, int ct,
                           uint32_t* keep) {
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (vmask >> j & 1u) { lo = min(lo, key[j]); hi = max(hi, key[j]); }
    block_minmax(lo, hi, S, ct);
    const float vmin = key2f(lo), vmax = key2f(hi);
    const float range = vmax - vmin;
    if (!(range > 0.f) || !(range < INFINITY)) return false;    // every thread sees the same
    const float scale = (float)NBC / range;
    uint32_t bin[NPER];
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        bin[j] = min((uint32_t)(NBC - 1), (uint32_t)((key2f(key[j]) - vmin) * scale));
        if (vmask >> j & 1u) atomicAdd(&S.hcnt[bin[j]], 1u);
    }
    named_sync(kBar, NCT);
    constexpr int per = (NBC + NCT - 1) / NCT;
    const int c0 = min(NBC, ct * per), c1 = min(NBC, c0 + per);
    uint32_t hc[per];
    uint32_t loc = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        hc[i] = c0 + i < c1 ? S.hcnt[c0 + i] : 0u;
        loc += hc[i];
        if (c0 + i < c1) S.hcnt[c0 + i] = 0u;            // zero again for the next cut
    }
    uint32_t a = block_above(loc, S, ct);
#pragma unroll
    for (int i = per - 1; i >= 0; --i) {
        if (a < K && K <= a + hc[i]) { S.sel[0] = (uint32_t)(c0 + i); S.sel[1] = a + hc[i]; }
        a += hc[i];
    }
    named_sync(kBar, NCT);
    const uint32_t b = S.sel[0], ge = S.sel[1];
    if (ge > limit) return false;
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j) m |= (uint32_t)((vmask >> j & 1u) && bin[j] >= b) << j;
    *keep = m;
    return true;
}

// All consumer warps: cut the candidates of all regions (when there are more than K),
// spread the survivors evenly over the regions and raise T.  cnt: this warp's count.
// What a cut leaves a warp: its candidate count, the threshold, and the total kept.
struct CutOut {
    uint32_t cnt;
    float T;
    uint32_t total;
};

// (Returned by value rather than through references, so that the callers' row state
// stays in registers instead of local memory.)
__device__ __noinline__ CutOut compact(TSmem& S, uint32_t K, uint32_t limit, uint32_t tot, int ct, uint32_t cnt,
                                       float T) {
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t key[NPER], id[NPER];
    const uint32_t vmask = load_region(S, cw, lane, cnt, key, id);
    uint32_t keep = vmask;
    if (tot > K) {
        if (!linear_cut(key, vmask, K, limit, S, ct, &keep)) {
            named_sync(kBar, NCT);           // S.wtmp and S.sel are reused
            uint32_t tk;
            keep = choose(key, id, vmask, K, limit, S, ct, &tk);
            named_sync(kBar, NCT);
            for (int i = ct; i < NBC; i += NCT) S.hcnt[i] = 0u;
        }
    }
    // the smallest kept key: the new threshold (the K-th largest of the row is at least it)
    uint32_t kept = 0, kmin = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool kj = keep >> j & 1u;
        kept += (uint32_t)__popc(__ballot_sync(0xffffffffu, kj));
        if (kj) kmin = min(kmin, key[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
    named_sync(kBar, NCT);                 // every region has been read into registers
    if (lane == 0) { S.wcnt[cw] = kept; S.wtmp[1][cw] = kmin; }
    named_sync(kBar, NCT);
    uint32_t base = 0, total = 0;
    kmin = 0xffffffffu;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
        const uint32_t c = S.wcnt[w];
        base += w < cw ? c : 0u;
        total += c;
        kmin = min(kmin, S.wtmp[1][w]);
    }
    if (tot > K) T = key2f(kmin);
    // survivor i goes to region i % NCW, entry i / NCW
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool kj = keep >> j & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, kj);
        if (kj) {
            const uint32_t i = base + (uint32_t)__popc(bal & lanemask_lt());
            const uint32_t slot = (i % (uint32_t)NCW) * RW + i / (uint32_t)NCW;
            S.cval[slot] = key2f(key[j]);   // -0.0 comes back as +0.0: same rank, same probability
            S.cid[slot] = id[j];
        }
        base += (uint32_t)__popc(bal);
    }
    cnt = (total + (uint32_t)(NCW - 1 - cw)) / (uint32_t)NCW;
    if (ct == 0) { S.total = total; S.need = 0; }
    named_sync(kBar, NCT);                 // regions rewritten, S.wcnt and S.wtmp read, flag lowered
    return CutOut{cnt, T, total};
}

// Per-row state of a consumer thread (the same in every thread of a warp; the cut
// fields the same in every consumer thread).
struct RowState {
    uint32_t cnt;          // this warp's candidates
    float T;               // admission threshold
    uint32_t adm;          // values this warp admitted
    bool spec;             // the row runs with a speculative threshold
    bool spec_pending;     // which is set after the first tile
    uint32_t aspec;        // rank, within a warp's share of the first tile, of its estimate
    bool valid_cut;        // a cut over the row's K largest was made
    bool nan;              // this thread saw a NaN in the row
};

// Entry of every warp into a collective step.  Returns how many warps had finished the
// row; unless all had, the candidates are cut (compact) to the K largest, whose
// smallest value becomes T (a lower bound of the row's K-th largest).
__device__ __forceinline__ uint32_t collective(TSmem& S, RowState& st, uint32_t K, uint32_t limit, int ct,
                                               bool fin) {
    const int cw = ct >> 5, lane = ct & 31;
    if (lane == 0) S.wcnt[cw] = st.cnt;
    const uint32_t nfin = named_sync_popc(kBar, NCT, fin && lane == 0);
    if (nfin == (uint32_t)NCW) return nfin;
    uint32_t tot = 0;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += S.wcnt[w];
    named_sync(kBar, NCT);                 // S.wcnt is rewritten by compact
    const CutOut o = compact(S, K, limit, tot, ct, st.cnt, st.T);
    st.cnt = o.cnt;
    st.T = o.T;
    st.valid_cut |= tot > K;
    return nfin;
}

// Admission of one tile's values (absent ones -inf): those at or above T are appended
// to this warp's region with one ballot per float4 group.  A warp that sees the
// candidate total pass `trig` asks for a cut (not in a speculative row, where only a
// full region does).
__device__ __forceinline__ void admit(TSmem& S, RowState& st, const float4 (&v)[kVecT], int n4, int h, int t,
                                      int ct, uint32_t trig) {
    const int cw = ct >> 5, lane = ct & 31;
    const uint32_t before = st.cnt;
    const float T = st.T;
#pragma unroll
    for (int u = 0; u < kVecT; ++u) {
        const int j = u * NCT + ct;
        const bool active = j < n4;
        // a NaN never compares >= T, so it is never admitted; the row is flagged
        // (the sum is NaN for any NaN member, and for +inf with -inf: then look closer)
        const float s4 = (v[u].x + v[u].y) + (v[u].z + v[u].w);
        if (active && s4 != s4) st.nan |= isnan(v[u].x) || isnan(v[u].y) || isnan(v[u].z) || isnan(v[u].w);
        // most float4s hold nothing at or above the threshold: one vote per warp
        const bool any = active && fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)) >= T;
        if (__any_sync(0xffffffffu, any)) {
            const uint32_t c0 = (uint32_t)(h + t * kTileT + 4 * j);
            wappend(S, cw, st.cnt, any && v[u].x >= T, v[u].x, c0);
            wappend(S, cw, st.cnt, any && v[u].y >= T, v[u].y, c0 + 1);
            wappend(S, cw, st.cnt, any && v[u].z >= T, v[u].z, c0 + 2);
            wappend(S, cw, st.cnt, any && v[u].w >= T, v[u].w, c0 + 3);
        }
    }
    const uint32_t added = st.cnt - before;
    st.adm += added;
    if (lane == 0 && added && !st.spec) {
        const uint32_t now = atomicAdd(&S.total, added) + added;
        if (now > trig) S.need = 1;
    }
}

// The end of a row, all warps: at most K + SLACK survivors, ordered by (value desc, id asc)
// through 2048 buckets of the key range, the first K written with their probabilities.
// Returns false, doing nothing, when the row ran with a speculative threshold that
// proved too high: fewer than K values at or above it and no exact cut since.
__device__ __noinline__ bool finish_row(TSmem& S, uint32_t K, int ct, const RowState st, long long r, uint32_t* ids,
                                        float* probs, int* err) {
    const int cw = ct >> 5, lane = ct & 31;
    const uint32_t cnt = st.cnt;
    if (st.spec && !st.valid_cut) {
        uint32_t adm = 0;
#pragma unroll
        for (int w = 0; w < NCW; ++w) adm += S.wadm[w];
        if (adm < K) {
            if (ct == 0) { S.total = 0; S.need = 0; }
            named_sync(kBar, NCT);         // S.wcnt and S.wadm are read before the row is redone
            return false;
        }
    }
    uint32_t tot = 0;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += S.wcnt[w];
    uint32_t key[NPER], id[NPER];
    const uint32_t vmask = load_region(S, cw, lane, cnt, key, id);
    uint32_t keep = vmask;
    if (tot > K + (uint32_t)SLACK) {
        const bool done = linear_cut(key, vmask, K, K + (uint32_t)SLACK, S, ct, &keep);
        named_sync(kBar, NCT);             // S.sel, S.hcnt and S.wtmp are reused
        if (!done) {
            uint32_t tk;
            keep = choose(key, id, vmask, K, K + (uint32_t)SLACK, S, ct, &tk);
            named_sync(kBar, NCT);
        }
    }
    // ---- buckets: NBK equal bins of the value range when it is finite and not empty,
    //      else an 11-bit window of (key - lo); higher buckets first
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (keep >> j & 1u) { lo = min(lo, key[j]); hi = max(hi, key[j]); }
    for (int i = ct; i < NBK; i += NCT) S.hcnt[i] = 0u;
    block_minmax(lo, hi, S, ct);
    const float vmin = key2f(lo), range = key2f(hi) - vmin;
    const bool lin = range > 0.f && range < INFINITY;
    const float scale = lin ? (float)NBK / range : 0.f;
    const uint32_t R = hi - lo;
    const int nbits = R ? 32 - __clz(R) : 0;
    const int s2 = nbits > 11 ? nbits - 11 : 0;
    auto bucket = [&](uint32_t kk) -> uint32_t {
        return lin ? min((uint32_t)(NBK - 1), (uint32_t)((key2f(kk) - vmin) * scale)) : (kk - lo) >> s2;
    };
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (keep >> j & 1u) atomicAdd(&S.hcnt[bucket(key[j])], 1u);
    named_sync(kBar, NCT);
    {
        constexpr int per = (NBK + NCT - 1) / NCT;
        const int c0 = min(NBK, ct * per), c1 = min(NBK, c0 + per);
        uint32_t loc = 0;
        for (int i = c0; i < c1; ++i) loc += S.hcnt[i];
        uint32_t a = block_above(loc, S, ct);
        for (int i = c1 - 1; i >= c0; --i) {
            S.hpos[i] = a;
            a += S.hcnt[i];
        }
    }
    named_sync(kBar, NCT);
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        if (keep >> j & 1u) {
            const uint32_t p = atomicAdd(&S.hpos[bucket(key[j])], 1u);
            S.okey[p] = key[j];
            S.oid[p] = id[j];
        }
    }
    named_sync(kBar, NCT);
    // ---- exact rank: the bucket's start plus the members ahead in (key desc, id asc)
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        if (keep >> j & 1u) {
            const uint32_t bk = bucket(key[j]);
            const uint32_t end = S.hpos[bk], beg = end - S.hcnt[bk];
            const unsigned long long me = comp(key[j], id[j]);
            uint32_t rank = beg;
            for (uint32_t i = beg; i < end; ++i) rank += comp(S.okey[i], S.oid[i]) > me ? 1u : 0u;
            if (rank < K) {
                S.cval[rank] = key2f(key[j]);
                S.cid[rank] = id[j];
            }
        }
    }
    named_sync(kBar, NCT);
    // ---- probabilities renormalised over the k, summed in rank order.  A row with fewer
    //      than K values that are not NaN (NaN is never admitted) fills the rest with
    //      id 0xFFFFFFFF and probability 0.
    const uint32_t nout = tot < K ? tot : K;
    const float v0 = nout ? S.cval[0] : 0.f;
    float part = 0.f;
    for (uint32_t q = (uint32_t)ct; q < nout; q += NCT) part += expf(S.cval[q] - v0);
    part = warp_sum(part);
    if (lane == 0) S.zred[cw] = part;
    named_sync(kBar, NCT);
    float Z = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) Z += S.zred[w];
    for (uint32_t q = (uint32_t)ct; q < K; q += NCT) {
        const bool have = q < nout;
        ids[r * K + q] = have ? S.cid[q] : 0xFFFFFFFFu;
        probs[r * K + q] = have ? expf(S.cval[q] - v0) / Z : 0.f;
    }
    for (int i = ct; i < NBC; i += NCT) S.hcnt[i] = 0u;
    if (ct == 0) {
        S.total = 0;
        S.need = 0;
        if (S.nanrow) {                       // one count per row that holds a NaN
            if (err) atomicAdd(err, 1);
            S.nanrow = 0;
        }
    }
    named_sync(kBar, NCT);   // the regions, S.zred, S.total and S.nanrow are reused by the next row
    return true;
}

// ---------------------------------------------------------------- consumer

__device__ void consumer(const float* x, long long ld, long long V, int k, const Rows& R,
                         uint32_t* ids, float* probs, int* err, TSmem& S) {
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const uint32_t K = (uint32_t)k;
    const uint32_t limit = min((uint32_t)LIMIT_MAX, K + max(K / 8u, 64u));   // survivors of a cut
    const uint32_t trig = max(4u * K, 1024u);                               // total that asks for a cut
    volatile int* need = &S.need;
    uint32_t g = 0;
    for (long long i = blockIdx.x; i < R.n; i += gridDim.x) {
        const long long r = R.at(i);
        const float* rowp = x + r * ld;
        const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        int h = (4 - mis) & 3;
        if (h > V) h = (int)V;
        const int bt = ((int)V - h) & ~3;
        const int t0 = h + bt;
        const int nt = (bt + kTileT - 1) / kTileT;

        // Speculation: the first tile's values are a sample of the row, and a threshold
        // estimated from it lets about 2.5 K values of the row through.  The row's answer
        // is exact when at least K of its values reach the threshold (or a cut proved a
        // higher bound), which finish_row checks; the row is redone exactly when not.
        RowState st;
        st.cnt = 0;
        st.T = -INFINITY;
        st.adm = 0;
        st.valid_cut = false;
        st.nan = false;
        {
            // a warp's share of the first tile holds K * (kTileT / NCW) / V of the row's
            // K largest on average; its estimate is the value with 1.4 times that many (at
            // least 2) of its share at or above it, and the threshold is the mean of the
            // warps' estimates: about 1.4 K values of the row pass it (the count check
            // fails only when fewer than K do, about three standard deviations out for
            // these ranks), their regions keep room for a tile without a cut, and the
            // survivors fit the final ordering without one
            const float share = (float)K * (float)(kTileT / NCW) / (float)V;
            st.aspec = max(2u, (uint32_t)ceilf(1.4f * share));
            st.spec = nt >= 8 && st.aspec <= (uint32_t)(kTileT / NCW / 8);
            st.spec_pending = st.spec;
        }
        // head and tail columns (at most 3 + 3) go to warp 0 unconditionally
        auto head_tail = [&]() {
            if (cw == 0) {
                bool keep = false;
                float v = 0.f;
                uint32_t id = 0;
                if (ct < h) { id = (uint32_t)ct; v = rowp[id]; keep = true; }
                else if (ct >= 4 && ct - 4 < (int)V - t0) { id = (uint32_t)(t0 + ct - 4); v = rowp[id]; keep = true; }
                if (keep && isnan(v)) { keep = false; st.nan = true; }
                wappend(S, cw, st.cnt, keep, v, id);
            }
        };
        head_tail();
        for (int t = 0; t < nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % kSlotsT, par = (gt / kSlotsT) & 1u;
            // a cut first when another warp asks for one or this region has no room for a tile
            if (__shfl_sync(0xffffffffu, *need, 0) || st.cnt + PER_TILE > (uint32_t)RW) {
                if (lane == 0) *need = 1;
                collective(S, st, K, limit, ct, false);
            }
            // the tile; a cut asked for by another warp is joined while waiting
            {
                const uint32_t fb = smem_u32(&S.full[slot]);
                long long w0 = 0;
                for (uint32_t it = 0;; ++it) {
                    if (__all_sync(0xffffffffu, mbar_try_wait(fb, par))) break;
                    if (__shfl_sync(0xffffffffu, *need, 0)) {
                        collective(S, st, K, limit, ct, false);
                        continue;
                    }
                    if ((it & 255u) == 255u) {
                        if (S.abort) break;
                        const long long now = clock64();
                        if (w0 == 0) {
                            w0 = now;
                        } else if (now - w0 > kWaitTimeoutCycles) {
                            S.abort = 1;
                            atomicOr(&g_watchdog, 1u);
                            break;
                        }
                    }
                }
            }
            const int n4 = min(kTileT, bt - t * kTileT) >> 2;
            float4 v[kVecT];
#pragma unroll
            for (int u = 0; u < kVecT; ++u) {
                const int j = u * NCT + ct;
                v[u] = j < n4 ? ld_shared_v4(&S.ring[slot][j * 4]) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            if (st.spec_pending) {
                // first tile of a speculative row (every warp gets here before any cut)
                const float e = warp_kth(v, st.aspec, lane);
                if (lane == 0) S.wspec[cw] = e;
                named_sync(kBar, NCT);
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) sum += S.wspec[w];
                st.T = sum * (1.0f / NCW);
                st.spec_pending = false;
            }
            admit(S, st, v, n4, h, t, ct, trig);
        }
        g += (uint32_t)nt;
        if (lane == 0) S.wadm[cw] = st.adm;
        if (st.nan) S.nanrow = 1;
        while (collective(S, st, K, limit, ct, true) != (uint32_t)NCW) {
        }
        if (finish_row(S, K, ct, st, r, ids, probs, err)) continue;

        // ---- the speculative threshold was too high: the row again, exactly, read from
        //      global memory (the ring has moved on to the next rows)
        st.cnt = 0;
        st.T = -INFINITY;
        st.adm = 0;
        st.spec = false;
        st.spec_pending = false;
        st.valid_cut = false;
        st.nan = false;
        head_tail();
        for (int t = 0; t < nt; ++t) {
            if (__shfl_sync(0xffffffffu, *need, 0) || st.cnt + PER_TILE > (uint32_t)RW) {
                if (lane == 0) *need = 1;
                collective(S, st, K, limit, ct, false);
            }
            const int n4 = min(kTileT, bt - t * kTileT) >> 2;
            float4 v[kVecT];
#pragma unroll
            for (int u = 0; u < kVecT; ++u) {
                const int j = u * NCT + ct;
                v[u] = j < n4 ? *reinterpret_cast<const float4*>(rowp + h + t * kTileT + 4 * j)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            admit(S, st, v, n4, h, t, ct, trig);
        }
        if (st.nan) S.nanrow = 1;
        while (collective(S, st, K, limit, ct, true) != (uint32_t)NCW) {
        }
        finish_row(S, K, ct, st, r, ids, probs, err);
    }
}

__global__ void __maxnreg__(128)
topk_kernel(const float* __restrict__ x, long long ld, long long V, int k, long long ls, long long le,
            const int* list, const int* nlist, uint32_t* __restrict__ ids, float* __restrict__ probs, int* err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TSmem& S = *reinterpret_cast<TSmem*>(smem_raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlotsT; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        S.abort = 0;
        S.issued = 0;
        S.total = 0;
        S.need = 0;
        S.nanrow = 0;
        fence_mbar_init_cluster();
    }
    for (int i = (int)threadIdx.x; i < NBC; i += (int)blockDim.x) S.hcnt[i] = 0u;
    __syncthreads();
    // launched as a programmatic dependent: the set-up above overlaps the tail of the
    // previous kernel on the stream; its results are visible past this wait
    pdl_wait_primary();
    pdl_launch_dependents();
    const Rows R{ls, list ? (long long)*nlist : le - ls, list};
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer(x, ld, V, R, S);
            drain(S);
        }
        __syncwarp();
    } else {
        consumer(x, ld, V, k, R, ids, probs, err, S);
    }
}

std::atomic<int> g_attr_done[64];

}  // namespace

cudaError_t launch_topk(const float* x, long long ld, long long ntok, long long V, int k, long long ls,
                        long long le, const int* list, const int* nlist, uint32_t* ids, float* probs, int* err,
                        cudaStream_t st) {
    (void)ntok;
    if (k < 1 || k > KMAXT) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute((const void*)topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(TSmem));
        if (e != cudaSuccess) return e;
        g_attr_done[dev].store(1, std::memory_order_release);
    }
    static std::atomic<int> sm_cache[64];
    sms = sm_cache[dev].load(std::memory_order_acquire);
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sm_cache[dev].store(sms, std::memory_order_release);
    }
    const long long rows = le - ls;
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(rows < sms ? rows : sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = sizeof(TSmem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_kernel, x, ld, V, k, ls, le, list, nlist, ids, probs, err);
}

unsigned int topk_watchdog(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_watchdog, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_watchdog, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}

}  // namespace vl
