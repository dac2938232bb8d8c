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
//   * each consumer warp owns a region of the shared candidate buffer.  A value
//     enters its warp's region when it is at or above the running threshold T
//     (the k-th best value kept so far); ties with T are decided by the
//     composite order (value desc, id asc) at the next selection;
//   * when a region could overflow, an exact radix select over order-preserving
//     32-bit keys (-0.0 folded into +0.0; 8-bit digits over the key range
//     present, warp-private histograms; then over the ids of tied keys) keeps the
//     best k, spreads them evenly over the regions and raises T;
//   * at the end of the row the k survivors are ordered by (value desc, id asc)
//     and written with their probabilities.
#include "vl_device.cuh"
#include "vl_internal.h"

#include <atomic>

namespace vl {
namespace {

constexpr int NCW = kConsumerWarps;
constexpr int NCT = NCW * 32;
constexpr int NTHREADS = NCT + 32;
constexpr int kSlotsT = 7;           // ring tiles (105 KB)
constexpr int RW = 512;              // candidate entries per consumer warp
constexpr int CB = RW * NCW;         // candidate buffer entries
constexpr int NPER = RW / 32;        // candidates per lane while compacting
constexpr int KMAXT = 2048;
constexpr int DB = 8;                // radix digit bits
constexpr int NBIN = 1 << DB;
constexpr int PER_TILE = kTileF / NCW;   // most candidates a warp can add per tile
constexpr uint32_t kBar = 1;

static_assert(kTileF / 4 == NCT * kVec, "kVec float4s of each tile per consumer thread");
static_assert(((KMAXT + NCW - 1) / NCW) + 6 + PER_TILE <= RW, "survivors plus one tile fit a region");

__device__ unsigned int g_watchdog;

struct alignas(128) TSmem {
    float ring[kSlotsT][kTileF];
    uint64_t full[kSlotsT];
    uint64_t empty[kSlotsT];
    float cval[CB];                  // candidate values, region w = [w * RW, (w + 1) * RW)
    uint32_t cid[CB];
    uint32_t whist[NCW][NBIN];       // warp-private digit histograms
    uint32_t hist[NBIN];
    float okey[KMAXT];               // the k survivors, then in final order
    uint32_t oid[KMAXT];
    uint32_t wtmp[2][NCW];
    uint32_t wcnt[NCW];
    float zred[NCW];
    uint32_t sel[4];
    int abort;
    uint32_t issued;
};

static_assert(sizeof(TSmem) <= 227 * 1024, "shared memory of one CTA");

__device__ __forceinline__ uint32_t f2key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;                      // -0.0 ranks as +0.0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7fffffffu) : __uint_as_float(~k);
}

// composite order: larger value first, then lower id
__device__ __forceinline__ unsigned long long comp(float v, uint32_t id) {
    return ((unsigned long long)f2key(v) << 32) | (unsigned long long)(0xffffffffu - id);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------- producer

__device__ void producer(const float* x, long long ld, long long V, long long ls, long long le, TSmem& S) {
    uint32_t g = 0;
    for (long long r = ls + (long long)blockIdx.x; r < le; r += gridDim.x) {
        const float* rowp = x + r * ld;
        const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        int h = (4 - mis) & 3;
        if (h > V) h = (int)V;
        const int bt = ((int)V - h) & ~3;
        for (int c0 = 0; c0 < bt; c0 += kTileF) {
            const uint32_t slot = g % kSlotsT, use = g / kSlotsT;
            if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog)) {
                S.issued = g;
                return;
            }
            const uint32_t bytes = (uint32_t)min(kTileF, bt - c0) * 4u;
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

// ---------------------------------------------------------------- consumer helpers

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

// The K-th largest of f[j] over the slots with bit j of vmask set, 1 <= K <= count.
// Returns v*; *above = #{f > v*}, *eq = #{f == v*}.  Exact MSD radix select, 8-bit
// digits over the range [min, max] present, warp-private histograms.
__device__ __forceinline__ uint32_t select_kth_largest(const uint32_t (&f)[NPER], uint32_t vmask, uint32_t K,
                                                       TSmem& S, int ct, uint32_t* above, uint32_t* eq) {
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int j = 0; j < NPER; ++j)
        if (vmask >> j & 1u) { lo = min(lo, f[j]); hi = max(hi, f[j]); }
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
    const uint32_t R = hi - lo;
    int shift = R ? 32 - __clz(R) : 0;
    uint32_t prefix = 0, rem = K, abv = 0, eqc = 0;
    int bits = 0;
    do {
        bits = shift < DB ? shift : DB;
        shift -= bits;
        const uint32_t dmask = (1u << bits) - 1u;
        uint32_t* wh = S.whist[cw];
#pragma unroll
        for (int i = lane; i < NBIN; i += 32) wh[i] = 0u;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NPER; ++j) {
            if (vmask >> j & 1u) {
                const uint32_t u = f[j] - lo;
                const uint32_t top = (shift + bits >= 32) ? 0u : (u >> (shift + bits));
                if (top == prefix) atomicAdd(&wh[(u >> shift) & dmask], 1u);
            }
        }
        named_sync(kBar, NCT);
        if (ct < NBIN) {
            uint32_t s = 0;
#pragma unroll
            for (int w = 0; w < NCW; ++w) s += S.whist[w][ct];
            S.hist[ct] = s;
        }
        named_sync(kBar, NCT);
        if (cw == 0) {
            // suffix sums over the bins, lane l owns bins [8 l, 8 l + 8)
            uint32_t hs[8];
            uint32_t loc = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { hs[i] = S.hist[8 * lane + i]; loc += hs[i]; }
            uint32_t suf = loc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane + off < 32) suf += v;
            }
            uint32_t a = suf - loc;     // entries in bins above this lane's
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (a < rem && rem <= a + hs[i]) {
                    S.sel[0] = (uint32_t)(8 * lane + i);
                    S.sel[1] = a;
                    S.sel[2] = hs[i];
                }
                a += hs[i];
            }
        }
        named_sync(kBar, NCT);
        const uint32_t bin = S.sel[0], ab = S.sel[1], cnt = S.sel[2];
        rem -= ab;
        abv += ab;
        prefix = (prefix << bits) | bin;
        eqc = cnt;
        if (shift > 0) named_sync(kBar, NCT);   // S.sel and the histograms are reused
    } while (shift > 0);
    *above = abv;
    *eq = eqc;
    return lo + prefix;
}

// Keep exactly the best K candidates (value desc, id asc) of all regions (all of them
// when there are at most K) and spread them evenly over the regions, at most
// ceil(K / NCW) each.  `tot` is the number of candidates.  Returns true and the K-th
// best value in *T when a selection was made: later columns are admitted above it.
__device__ __forceinline__ bool compact(TSmem& S, uint32_t K, uint32_t tot, int ct, uint32_t& cnt, float* T) {
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t key[NPER], id[NPER];
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
    const bool sel = tot > K;
    uint32_t Tk = 0u, idmax = 0xffffffffu;
    if (sel) {
        uint32_t above, eq;
        Tk = select_kth_largest(key, vmask, K, S, ct, &above, &eq);
        const uint32_t need = K - above;
        if (eq > need) {
            uint32_t nid[NPER];
            uint32_t emask = 0;
#pragma unroll
            for (int j = 0; j < NPER; ++j) {
                nid[j] = ~id[j];
                if ((vmask >> j & 1u) && key[j] == Tk) emask |= 1u << j;
            }
            named_sync(kBar, NCT);
            uint32_t a2, e2;
            idmax = ~select_kth_largest(nid, emask, need, S, ct, &a2, &e2);
        }
    }
    uint32_t keep = 0, kept = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool kj = (vmask >> j & 1u) && (!sel || key[j] > Tk || (key[j] == Tk && id[j] <= idmax));
        keep |= (uint32_t)kj << j;
        kept += (uint32_t)__popc(__ballot_sync(0xffffffffu, kj));
    }
    named_sync(kBar, NCT);                 // every region has been read into registers
    if (lane == 0) S.wcnt[cw] = kept;
    named_sync(kBar, NCT);
    uint32_t base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
        const uint32_t c = S.wcnt[w];
        base += w < cw ? c : 0u;
        total += c;
    }
    const uint32_t per = (total + NCW - 1) / NCW;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool kj = keep >> j & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, kj);
        if (kj) {
            const uint32_t i = base + (uint32_t)__popc(bal & lanemask_lt());
            const uint32_t slot = (i / per) * RW + i % per;
            S.cval[slot] = key2f(key[j]);   // -0.0 comes back as +0.0: same rank, same probability
            S.cid[slot] = id[j];
        }
        base += (uint32_t)__popc(bal);
    }
    const int left = (int)total - cw * (int)per;
    cnt = left <= 0 ? 0u : (left < (int)per ? (uint32_t)left : per);
    named_sync(kBar, NCT);                 // regions rewritten, S.wcnt read
    if (sel) *T = key2f(Tk);
    return sel;
}

// ---------------------------------------------------------------- consumer

__device__ void consumer(const float* x, long long ld, long long V, int k, long long ls, long long le,
                         uint32_t* ids, float* probs, TSmem& S) {
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t g = 0;
    for (long long r = ls + (long long)blockIdx.x; r < le; r += gridDim.x) {
        const float* rowp = x + r * ld;
        const int mis = (int)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        int h = (4 - mis) & 3;
        if (h > V) h = (int)V;
        const int bt = ((int)V - h) & ~3;
        const int t0 = h + bt;
        const int nt = (bt + kTileF - 1) / kTileF;

        uint32_t cnt = 0;          // this warp's candidates (same in every lane)
        bool armed = false;        // a threshold exists once k candidates were kept
        float T = 0.f;
        // head and tail columns (at most 3 + 3) go to warp 0 unconditionally
        if (cw == 0) {
            bool keep = false;
            float v = 0.f;
            uint32_t id = 0;
            if (ct < h) { id = (uint32_t)ct; v = rowp[id]; keep = true; }
            else if (ct >= 4 && ct - 4 < (int)V - t0) { id = (uint32_t)(t0 + ct - 4); v = rowp[id]; keep = true; }
            wappend(S, cw, cnt, keep, v, id);
        }
        for (int t = 0; t < nt; ++t) {
            const uint32_t gt = g + (uint32_t)t, slot = gt % kSlotsT;
            wait_parity<false>(&S.full[slot], (gt / kSlotsT) & 1u, &S.abort, &g_watchdog);
            const int n4 = min(kTileF, bt - t * kTileF) >> 2;
            float4 v[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int j = u * NCT + ct;
                v[u] = j < n4 ? ld_shared_v4(&S.ring[slot][j * 4]) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int j = u * NCT + ct;
                const bool active = j < n4;
                // most float4s hold nothing at or above the threshold: one vote per warp
                const bool any = active && (!armed || fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)) >= T);
                if (__any_sync(0xffffffffu, any)) {
                    const uint32_t c0 = (uint32_t)(h + t * kTileF + 4 * j);
                    wappend(S, cw, cnt, any && (!armed || v[u].x >= T), v[u].x, c0);
                    wappend(S, cw, cnt, any && (!armed || v[u].y >= T), v[u].y, c0 + 1);
                    wappend(S, cw, cnt, any && (!armed || v[u].z >= T), v[u].z, c0 + 2);
                    wappend(S, cw, cnt, any && (!armed || v[u].w >= T), v[u].w, c0 + 3);
                }
            }
            // compact when some region could overflow on the next tile
            if (t + 1 < nt) {
                const uint32_t full = named_sync_popc(kBar, NCT, lane == 0 && cnt + PER_TILE > (uint32_t)RW);
                if (full) {
                    if (lane == 0) S.wcnt[cw] = cnt;
                    named_sync(kBar, NCT);
                    uint32_t tot = 0;
#pragma unroll
                    for (int w = 0; w < NCW; ++w) tot += S.wcnt[w];
                    named_sync(kBar, NCT);
                    armed |= compact(S, (uint32_t)k, tot, ct, cnt, &T);
                }
            }
        }
        g += (uint32_t)nt;

        // ---- exactly k survivors, gathered in one array
        if (lane == 0) S.wcnt[cw] = cnt;
        named_sync(kBar, NCT);
        uint32_t tot = 0;
#pragma unroll
        for (int w = 0; w < NCW; ++w) tot += S.wcnt[w];
        named_sync(kBar, NCT);
        if (tot > (uint32_t)k) compact(S, (uint32_t)k, tot, ct, cnt, &T);
        if (lane == 0) S.wcnt[cw] = cnt;
        named_sync(kBar, NCT);
        uint32_t base = 0;
#pragma unroll
        for (int w = 0; w < cw; ++w) base += S.wcnt[w];
        for (uint32_t i = (uint32_t)lane; i < cnt; i += 32) {
            S.okey[base + i] = S.cval[cw * RW + i];
            S.oid[base + i] = S.cid[cw * RW + i];
        }
        named_sync(kBar, NCT);

        // ---- order the k survivors by (value desc, id asc)
        const uint32_t K = (uint32_t)k;
        if (K <= (uint32_t)NCT) {
            // rank of each survivor among all k by the composite key, built once
            unsigned long long* ck = reinterpret_cast<unsigned long long*>(S.cval);
            const bool mine = (uint32_t)ct < K;
            float mv = 0.f;
            uint32_t mi = 0;
            unsigned long long mc = 0;
            if (mine) { mv = S.okey[ct]; mi = S.oid[ct]; mc = comp(mv, mi); ck[ct] = mc; }
            named_sync(kBar, NCT);
            if (mine) {
                uint32_t p0 = 0, p1 = 0, p2 = 0, p3 = 0, j = 0;
                for (; j + 4 <= K; j += 4) {
                    p0 += ck[j] > mc;
                    p1 += ck[j + 1] > mc;
                    p2 += ck[j + 2] > mc;
                    p3 += ck[j + 3] > mc;
                }
                for (; j < K; ++j) p0 += ck[j] > mc;
                const uint32_t pos = (p0 + p1) + (p2 + p3);
                S.okey[pos] = mv;      // every thread read its own entry before the barrier
                S.oid[pos] = mi;
            }
            named_sync(kBar, NCT);
        } else {
            uint32_t Kp = 1;
            while (Kp < K) Kp <<= 1;
            for (uint32_t i = K + (uint32_t)ct; i < Kp; i += NCT) { S.okey[i] = -INFINITY; S.oid[i] = 0xffffffffu; }
            named_sync(kBar, NCT);
            for (uint32_t size = 2; size <= Kp; size <<= 1) {
                for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
                    for (uint32_t i = (uint32_t)ct; i < Kp / 2; i += NCT) {
                        const uint32_t a = 2 * stride * (i / stride) + (i % stride), b = a + stride;
                        const bool down = (a & size) == 0u;
                        const unsigned long long ca = comp(S.okey[a], S.oid[a]), cb = comp(S.okey[b], S.oid[b]);
                        if (down ? (ca < cb) : (ca > cb)) {
                            const float tv = S.okey[a];
                            const uint32_t ti = S.oid[a];
                            S.okey[a] = S.okey[b]; S.oid[a] = S.oid[b];
                            S.okey[b] = tv; S.oid[b] = ti;
                        }
                    }
                    named_sync(kBar, NCT);
                }
            }
        }

        // ---- probabilities renormalised over the k, summed in rank order
        const float v0 = S.okey[0];
        float part = 0.f;
        for (uint32_t q = (uint32_t)ct; q < K; q += NCT) part += expf(S.okey[q] - v0);
        part = warp_sum(part);
        if (lane == 0) S.zred[cw] = part;
        named_sync(kBar, NCT);
        float Z = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) Z += S.zred[w];
        for (uint32_t q = (uint32_t)ct; q < K; q += NCT) {
            ids[r * k + q] = S.oid[q];
            probs[r * k + q] = expf(S.okey[q] - v0) / Z;
        }
        named_sync(kBar, NCT);   // okey, zred and the regions are reused by the next row
    }
}

__global__ void __maxnreg__(128)
topk_kernel(const float* __restrict__ x, long long ld, long long V, int k, long long ls, long long le,
            uint32_t* __restrict__ ids, float* __restrict__ probs) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TSmem& S = *reinterpret_cast<TSmem*>(smem_raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlotsT; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        S.abort = 0;
        S.issued = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer(x, ld, V, ls, le, S);
            drain(S);
        }
        __syncwarp();
    } else {
        consumer(x, ld, V, k, ls, le, ids, probs, S);
    }
}

std::atomic<int> g_attr_done[64];

}  // namespace

cudaError_t launch_topk(const float* x, long long ld, long long ntok, long long V, int k, long long ls,
                        long long le, uint32_t* ids, float* probs, int* err, cudaStream_t st) {
    (void)err;
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
    topk_kernel<<<grid, NTHREADS, sizeof(TSmem), st>>>(x, ld, V, k, ls, le, ids, probs);
    return cudaGetLastError();
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
