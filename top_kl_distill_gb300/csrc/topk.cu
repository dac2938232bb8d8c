// Exact teacher top-k per row with probabilities renormalised over the k
// (cortiq-engine train_head.rs, topk_rows: the k largest logits of a row,
// descending, and exp(v_q - v_0) / sum over the k).
//
// The page keeps each thread's best 8 of a strided scan and bitonic-sorts the
// 2048 survivors, which misses true top-k members when more than 8 of them
// share a residue class and breaks ties arbitrarily.  This kernel is exact, with
// ties going to the lower column:
//
//   * one persistent CTA per SM streams its rows through a ring of 8 KB tiles
//     (1-D bulk copies, producer warp + 16 consumer warps, as the row engine);
//   * each value x becomes an order-preserving 32-bit key (-0.0 folded into
//     +0.0); a value enters the shared-memory candidate buffer if its key is
//     above the running threshold T (the key of the current k-th best).  Columns
//     arrive in increasing order, so an equal key always loses to the candidate
//     already held and "key > T" is the exact admission test;
//   * when the buffer could overflow, an exact radix select (11-bit digits over
//     the key range actually present, then over the ids of the tied keys) keeps
//     the best k and raises T;
//   * at the end of the row the k survivors are ordered by (key desc, id asc)
//     and written with their probabilities.
#include "vl_device.cuh"
#include "vl_internal.h"

#include <atomic>

namespace vl {
namespace {

constexpr int NCW = 16;
constexpr int NCT = NCW * 32;
constexpr int NTHREADS = NCT + 32;
constexpr int kSlotsT = 16;          // ring tiles
constexpr int CB = 8192;             // candidate buffer entries
constexpr int NPER = CB / NCT;       // candidates per thread while compacting
constexpr int KMAXT = 2048;
constexpr int HB = 11;               // radix digit bits
constexpr int NBIN = 1 << HB;
constexpr uint32_t kBar = 1;

static_assert(kTileF / 4 == NCT, "one float4 of each tile per consumer thread");
static_assert(KMAXT + kTileF + 8 <= CB, "buffer holds k survivors plus one tile");

__device__ unsigned int g_watchdog;

struct alignas(128) TSmem {
    float ring[kSlotsT][kTileF];
    uint64_t full[kSlotsT];
    uint64_t empty[kSlotsT];
    uint32_t ckey[CB];
    uint32_t cid[CB];
    uint32_t hist[NBIN];
    uint32_t wtmp[2][NCW];
    float zred[NCW];
    uint32_t sel[4];
    uint32_t n;
    int abort;
    uint32_t issued;
};

__device__ __forceinline__ uint32_t f2key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;                      // -0.0 ranks as +0.0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7fffffffu) : __uint_as_float(~k);
}

// composite order: larger key first, then lower id
__device__ __forceinline__ unsigned long long comp(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - id);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------- producer

__device__ void producer(const float* x, long long ld, long long ntok, long long V, long long ls, long long le,
                         TSmem& S) {
    uint32_t g = 0;
    for (long long r = ls + (long long)blockIdx.x; r < le; r += gridDim.x) {
        const float* rowp = x + r * ld;
        const long long mis = (long long)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        long long h = (4 - mis) & 3;
        if (h > V) h = V;
        const long long bt = (V - h) & ~3LL;
        for (long long c0 = 0; c0 < bt; c0 += kTileF) {
            const uint32_t slot = g % kSlotsT, use = g / kSlotsT;
            if (use > 0 && !wait_parity<false>(&S.empty[slot], (use - 1) & 1u, &S.abort, &g_watchdog)) {
                S.issued = g;
                return;
            }
            const uint32_t bytes = (uint32_t)min((long long)kTileF, bt - c0) * 4u;
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

// ---------------------------------------------------------------- block helpers (consumers)

// Append the elements with keep = true to the candidate buffer (warp-aggregated).
__device__ __forceinline__ void append(TSmem& S, bool keep, uint32_t key, uint32_t id, int lane) {
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (bal == 0u) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&S.n, (uint32_t)__popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (keep) {
        const uint32_t pos = base + (uint32_t)__popc(bal & lanemask_lt());
        S.ckey[pos] = key;
        S.cid[pos] = id;
    }
}

// Four candidates from one float4 (columns c0 .. c0+3), one atomic per warp.
__device__ __forceinline__ void append4(TSmem& S, const float4& v, uint32_t c0, uint32_t T, bool active, int lane) {
    const uint32_t k0 = f2key(v.x), k1 = f2key(v.y), k2 = f2key(v.z), k3 = f2key(v.w);
    const bool a0 = active && k0 > T, a1 = active && k1 > T, a2 = active && k2 > T, a3 = active && k3 > T;
    const uint32_t b0 = __ballot_sync(0xffffffffu, a0), b1 = __ballot_sync(0xffffffffu, a1);
    const uint32_t b2 = __ballot_sync(0xffffffffu, a2), b3 = __ballot_sync(0xffffffffu, a3);
    const uint32_t p0 = __popc(b0), p1 = __popc(b1), p2 = __popc(b2), p3 = __popc(b3);
    const uint32_t tot = p0 + p1 + p2 + p3;
    if (tot == 0u) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&S.n, tot);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t lt = lanemask_lt();
    if (a0) { const uint32_t p = base + __popc(b0 & lt); S.ckey[p] = k0; S.cid[p] = c0; }
    base += p0;
    if (a1) { const uint32_t p = base + __popc(b1 & lt); S.ckey[p] = k1; S.cid[p] = c0 + 1; }
    base += p1;
    if (a2) { const uint32_t p = base + __popc(b2 & lt); S.ckey[p] = k2; S.cid[p] = c0 + 2; }
    base += p2;
    if (a3) { const uint32_t p = base + __popc(b3 & lt); S.ckey[p] = k3; S.cid[p] = c0 + 3; }
}

// The K-th largest of f[j] over the slots j with bit j of vmask set, 1 <= K <= count.
// Returns v*; *above = #{f > v*}, *eq = #{f == v*}.  Exact radix select over the
// range [min, max] actually present, 11 bits per pass from the top.
__device__ __forceinline__ uint32_t select_kth_largest(const uint32_t (&f)[NPER], uint32_t vmask, uint32_t K, TSmem& S,
                                       int ct, uint32_t* above, uint32_t* eq) {
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
    const int B = R ? 32 - __clz(R) : 0;
    int bits = B < HB ? B : HB;
    int shift = B - bits;
    uint32_t prefix = 0, rem = K, abv = 0, eqc = 0;
    for (;;) {
        for (int i = ct; i < NBIN; i += NCT) S.hist[i] = 0u;
        named_sync(kBar, NCT);
        const uint32_t dmask = (1u << bits) - 1u;
#pragma unroll
        for (int j = 0; j < NPER; ++j) {
            if (vmask >> j & 1u) {
                const uint32_t u = f[j] - lo;
                const uint32_t top = (bits + shift >= 32) ? 0u : (u >> (shift + bits));
                if (top == prefix) atomicAdd(&S.hist[(u >> shift) & dmask], 1u);
            }
        }
        named_sync(kBar, NCT);
        // suffix sums over bins: thread ct owns bins [4 ct, 4 ct + 4)
        const uint32_t h0 = S.hist[4 * ct], h1 = S.hist[4 * ct + 1], h2 = S.hist[4 * ct + 2], h3 = S.hist[4 * ct + 3];
        const uint32_t loc = h0 + h1 + h2 + h3;
        uint32_t suf = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t v = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf += v;
        }
        if (lane == 0) S.wtmp[0][cw] = suf;
        named_sync(kBar, NCT);
        for (int w = cw + 1; w < NCW; ++w) suf += S.wtmp[0][w];
        // bins above 4ct+3
        uint32_t a = suf - loc;
        const uint32_t hs[4] = {h0, h1, h2, h3};
#pragma unroll
        for (int i = 3; i >= 0; --i) {
            if (a < rem && rem <= a + hs[i]) {
                S.sel[0] = (uint32_t)(4 * ct + i);
                S.sel[1] = a;
                S.sel[2] = hs[i];
            }
            a += hs[i];
        }
        named_sync(kBar, NCT);
        const uint32_t bin = S.sel[0], ab = S.sel[1], cnt = S.sel[2];
        rem -= ab;
        abv += ab;
        prefix = (prefix << bits) | bin;
        if (shift == 0) { eqc = cnt; break; }
        bits = shift < HB ? shift : HB;
        shift -= bits;
        named_sync(kBar, NCT);   // everyone has read S.sel before it is rewritten
    }
    *above = abv;
    *eq = eqc;
    return lo + prefix;
}

// Keep exactly the best K candidates (key desc, id asc) of the n in the buffer.
// Returns the key of the K-th best: later columns are admitted only above it.
__device__ __forceinline__ uint32_t compact(TSmem& S, uint32_t K, int ct) {
    const int lane = ct & 31;
    const uint32_t n = S.n;
    uint32_t key[NPER], id[NPER];
    uint32_t vmask = 0;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const uint32_t i = (uint32_t)ct + (uint32_t)j * NCT;
        key[j] = 0u;
        id[j] = 0u;
        if (i < n) { key[j] = S.ckey[i]; id[j] = S.cid[i]; vmask |= 1u << j; }
    }
    uint32_t above, eq;
    const uint32_t T = select_kth_largest(key, vmask, K, S, ct, &above, &eq);
    const uint32_t need = K - above;
    bool idsel = eq > need;
    uint32_t idmax = 0xffffffffu;
    if (idsel) {
        uint32_t nid[NPER];
        uint32_t emask = 0;
#pragma unroll
        for (int j = 0; j < NPER; ++j) {
            nid[j] = ~id[j];
            if ((vmask >> j & 1u) && key[j] == T) emask |= 1u << j;
        }
        named_sync(kBar, NCT);
        uint32_t a2, e2;
        idmax = ~select_kth_largest(nid, emask, need, S, ct, &a2, &e2);
    }
    if (ct == 0) S.n = 0u;
    named_sync(kBar, NCT);
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const bool keep = (vmask >> j & 1u) && (key[j] > T || (key[j] == T && id[j] <= idmax));
        append(S, keep, key[j], id[j], lane);
    }
    named_sync(kBar, NCT);
    return T;
}

// ---------------------------------------------------------------- consumer

__device__ void consumer(const float* x, long long ld, long long ntok, long long V, int k, long long ls,
                         long long le, uint32_t* ids, float* probs, TSmem& S) {
    const int ct = (int)threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    uint32_t g = 0;
    for (long long r = ls + (long long)blockIdx.x; r < le; r += gridDim.x) {
        const float* rowp = x + r * ld;
        const long long mis = (long long)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
        long long h = (4 - mis) & 3;
        if (h > V) h = V;
        const long long bt = (V - h) & ~3LL;
        const long long t0 = h + bt;
        const uint32_t nt = (uint32_t)((bt + kTileF - 1) / kTileF);

        if (ct == 0) S.n = 0u;
        named_sync(kBar, NCT);
        uint32_t T = 0u;                     // admits every key but a NaN's
        // head and tail columns first (at most 3 + 3)
        {
            bool keep = false;
            uint32_t key = 0, id = 0;
            if (ct < h) { id = (uint32_t)ct; key = f2key(rowp[id]); keep = key > T; }
            else if (ct >= 4 && ct - 4 < V - t0) { id = (uint32_t)(t0 + ct - 4); key = f2key(rowp[id]); keep = key > T; }
            if (cw == 0) append(S, keep, key, id, lane);
        }
        named_sync(kBar, NCT);
        for (uint32_t t = 0; t < nt; ++t) {
            const uint32_t gt = g + t, slot = gt % kSlotsT;
            wait_parity<false>(&S.full[slot], (gt / kSlotsT) & 1u, &S.abort, &g_watchdog);
            const long long tc0 = h + (long long)t * kTileF;
            const int n4 = (int)(min((long long)kTileF, bt - (long long)t * kTileF) >> 2);
            const bool active = ct < n4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active) v = ld_shared_v4(&S.ring[slot][ct * 4]);
            append4(S, v, (uint32_t)(tc0 + 4 * ct), T, active, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            named_sync(kBar, NCT);
            if (S.n + (uint32_t)kTileF > (uint32_t)CB) T = compact(S, (uint32_t)k, ct);
        }
        g += nt;
        if (S.n > (uint32_t)k) T = compact(S, (uint32_t)k, ct);

        // ---- order the k survivors by (key desc, id asc)
        const uint32_t K = (uint32_t)k;
        if (K <= (uint32_t)NCT) {
            uint32_t mk = 0, mi = 0;
            unsigned long long mc = 0;
            const bool mine = (uint32_t)ct < K;
            if (mine) { mk = S.ckey[ct]; mi = S.cid[ct]; mc = comp(mk, mi); }
            uint32_t pos = 0;
            if (mine)
                for (uint32_t j = 0; j < K; ++j) pos += comp(S.ckey[j], S.cid[j]) > mc ? 1u : 0u;
            named_sync(kBar, NCT);
            if (mine) { S.ckey[pos] = mk; S.cid[pos] = mi; }
            named_sync(kBar, NCT);
        } else {
            uint32_t Kp = 1;
            while (Kp < K) Kp <<= 1;
            for (uint32_t i = K + (uint32_t)ct; i < Kp; i += NCT) { S.ckey[i] = 0u; S.cid[i] = 0xffffffffu; }
            named_sync(kBar, NCT);
            for (uint32_t size = 2; size <= Kp; size <<= 1) {
                for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
                    for (uint32_t i = (uint32_t)ct; i < Kp / 2; i += NCT) {
                        const uint32_t a = 2 * stride * (i / stride) + (i % stride), b = a + stride;
                        const bool down = (a & size) == 0u;
                        const unsigned long long ca = comp(S.ckey[a], S.cid[a]), cb = comp(S.ckey[b], S.cid[b]);
                        if (down ? (ca < cb) : (ca > cb)) {
                            const uint32_t tk = S.ckey[a], ti = S.cid[a];
                            S.ckey[a] = S.ckey[b]; S.cid[a] = S.cid[b];
                            S.ckey[b] = tk; S.cid[b] = ti;
                        }
                    }
                    named_sync(kBar, NCT);
                }
            }
        }

        // ---- probabilities renormalised over the k, summed in rank order
        const float v0 = key2f(S.ckey[0]);
        float part = 0.f;
        for (uint32_t q = (uint32_t)ct; q < K; q += NCT) part += expf(key2f(S.ckey[q]) - v0);
        part = warp_sum(part);
        if (lane == 0) S.zred[cw] = part;
        named_sync(kBar, NCT);
        float Z = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) Z += S.zred[w];
        for (uint32_t q = (uint32_t)ct; q < K; q += NCT) {
            ids[r * k + q] = S.cid[q];
            probs[r * k + q] = expf(key2f(S.ckey[q]) - v0) / Z;
        }
        named_sync(kBar, NCT);   // buffer and zred are reused by the next row
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
topk_kernel(const float* __restrict__ x, long long ld, long long ntok, long long V, int k, long long ls,
            long long le, uint32_t* __restrict__ ids, float* __restrict__ probs) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TSmem& S = *reinterpret_cast<TSmem*>(smem_raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlotsT; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        S.abort = 0;
        S.issued = 0;
        S.n = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            producer(x, ld, ntok, V, ls, le, S);
            drain(S);
        }
        __syncwarp();
    } else {
        consumer(x, ld, ntok, V, k, ls, le, ids, probs, S);
    }
}

std::atomic<int> g_attr_done[64];

}  // namespace

cudaError_t launch_topk(const float* x, long long ld, long long ntok, long long V, int k, long long ls,
                        long long le, uint32_t* ids, float* probs, int* err, cudaStream_t st) {
    (void)err;
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
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long rows = le - ls;
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(rows < sms ? rows : sms);
    topk_kernel<<<grid, NTHREADS, sizeof(TSmem), st>>>(x, ld, ntok, V, k, ls, le, ids, probs);
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
