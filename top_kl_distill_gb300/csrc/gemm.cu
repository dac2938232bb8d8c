// The head GEMM on the 5th-generation tensor cores (sm_103a): D[M][N] = alpha * A[M][K] . B[N][K]^T
// with A and B bf16, row-major (both K-major), fp32 accumulation in tensor memory, D fp32.
// Used for the vocabulary head around the losses (cortiq-engine train_head.rs: mm_cols for the
// logits, hidden . W^T; and the backward mm over the transposed weight plane wt, dlogits . wt^T).
//
// One persistent CTA per SM walks 128 x 256 tiles of D (blockIdx.x, blockIdx.x + gridDim.x, ...):
//   warp 0    TMA producer: 2-D tiled bulk copies of 128 x 64 (A) and 256 x 64 (B) bf16 boxes
//             with 128-byte swizzle into a 4-stage shared-memory ring, signalled on mbarriers,
//             the ring's position running on across tiles;
//   warp 1    allocates 512 columns of tensor memory (two 128 x 256 fp32 accumulators) and,
//             from one thread, issues tcgen05.mma (kind::f16, M = 128, N = 256, K = 16; four per
//             64-wide stage) into the accumulator of the tile's parity, once the epilogue has
//             handed it back; tcgen05.commit to the stage's empty barrier (the stage is free once
//             its MMAs have read it) and, after the tile's last stage, to the accumulator's full
//             barrier;
//   warps 2-5 the epilogue: tcgen05.ld of their 32-lane quarter of a full accumulator (row i of
//             the tile is tensor-memory lane i, column j is column j), alpha, stores to D, then
//             an arrival that hands the accumulator back -- so the stores of tile i overlap the
//             MMAs of tile i + 1.
// Rows, columns and K past the matrix edges: the TMA fills zeros, the epilogue masks stores.
// Every wait is bounded; a wait that runs out raises the watchdog word, the producer still
// waits for its copies in flight, and tensor memory is freed only after a final commit shows
// every MMA issued complete.
#include "vl_device.cuh"
#include "vl_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace vl {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB: 128 rows of 128 bytes
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int GT = 192;                     // six warps
constexpr uint32_t TMEM_COLS = 2 * BN;          // two accumulators of 128 x 256 fp32

__device__ unsigned int g_watchdog;

struct alignas(1024) GSmem {
    uint8_t a[STAGES][A_BYTES];             // each stage 1024-byte aligned (the swizzle atom)
    uint8_t b[STAGES][B_BYTES];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];                      // an accumulator's tile is complete (MMA commit)
    uint64_t tempty[2];                     // the epilogue has read an accumulator
    uint64_t done;                          // every MMA issued has completed
    uint32_t tmem_base;
    int abort;
};

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, groups of 8 rows 1024 bytes apart.  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused for this layout), stride byte
// offset >> 4 (32-45), the fixed version bits 0b001 (46-48), swizzle mode 2 = 128-byte
// (61-63).  Advancing K by 16 elements inside the 128-byte row adds 32 bytes to the start.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: D f32 (bits 4-5 = 1), A and B bf16 (7-9, 10-12 = 1),
// both K-major (15, 16 = 0), N >> 3 (17-22), M >> 4 (24-28).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive accumulator columns of this warp's 32 lanes: lane i gets row i's values.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(GT, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap ta,
                                                        const __grid_constant__ CUtensorMap tb, float* __restrict__ D,
                                                        long long ldd, int M, int N, int K, float alpha, int m_fast) {
    extern __shared__ uint8_t gsm_raw[];
    GSmem& S = *reinterpret_cast<GSmem*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (M + BM - 1) / BM, ntl = (N + BN - 1) / BN;
    const int tiles = mt * ntl;
    const int nk = (K + BK - 1) / BK;
    // tile t of this CTA's sequence blockIdx.x, blockIdx.x + gridDim.x, ...: its (m0, n0)
    auto tile_at = [&](int t, int& m0, int& n0) {
        const int a = m_fast ? t % mt : t / ntl, b = m_fast ? t / mt : t % ntl;
        m0 = a * BM;
        n0 = b * BN;
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.tfull[b], 1);
            mbar_init(&S.tempty[b], 4);      // one arrival per epilogue warp
        }
        mbar_init(&S.done, 1);
        S.abort = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&S.tmem_base)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait_primary();
    pdl_launch_dependents();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = 0, issued = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x) {
                int m0, n0;
                tile_at(t, m0, n0);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t s = g % STAGES, use = g / STAGES;
                    if (use > 0 && !wait_parity<false>(&S.empty[s], (use - 1) & 1u, &S.abort, &g_watchdog)) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(&S.full[s], A_BYTES + B_BYTES);
                    tma_load_2d(S.a[s], &ta, kb * BK, m0, &S.full[s]);
                    tma_load_2d(S.b[s], &tb, kb * BK, n0, &S.full[s]);
                    issued = g + 1;
                }
            }
            // every copy issued has landed before the CTA can leave
            for (uint32_t gg = issued > (uint32_t)STAGES ? issued - STAGES : 0u; gg < issued; ++gg)
                wait_parity_drain(&S.full[gg % STAGES], (gg / STAGES) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = 0, i = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x, ++i) {
                const uint32_t b = i & 1u, use = i >> 1;
                // the epilogue has read this accumulator's previous tile
                if (use > 0 && !wait_parity<false>(&S.tempty[b], (use - 1) & 1u, &S.abort, &g_watchdog)) break;
                tc_fence_after();
                const uint32_t acc = tmem + b * (uint32_t)BN;
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t s = g % STAGES;
                    if (!wait_parity<false>(&S.full[s], (g / STAGES) & 1u, &S.abort, &g_watchdog)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(S.a[s]), b0 = smem_u32(S.b[s]);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16(acc, sw128_desc(a0 + 32u * k), sw128_desc(b0 + 32u * k), (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&S.empty[s]);        // the stage is free once these MMAs have read it
                }
                if (!stop) mma_commit(&S.tfull[b]); // the tile's accumulator is complete
            }
            mma_commit(&S.done);                    // always: the dealloc waits for every MMA issued
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31 of the tile's accumulator
        const int q = warp & 3;
        const bool vec = (ldd & 3) == 0 && (reinterpret_cast<uintptr_t>(D) & 15u) == 0;
        uint32_t i = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const uint32_t b = i & 1u;
            if (!wait_parity<false>(&S.tfull[b], (i >> 1) & 1u, &S.abort, &g_watchdog)) break;
            tc_fence_after();
            int m0, n0;
            tile_at(t, m0, n0);
            const int row = m0 + 32 * q + lane;
            for (int c = 0; c < BN; c += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + b * (uint32_t)BN + (uint32_t)c, v);
                if (row >= M) continue;
                float* out = D + (long long)row * ldd + n0 + c;
                if (vec && n0 + c + 32 <= N) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(out + j) =
                            make_float4(alpha * v[j], alpha * v[j + 1], alpha * v[j + 2], alpha * v[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + c + j < N) out[j] = alpha * v[j];
                }
            }
            // this warp's reads of the accumulator are done (tcgen05.ld waited): hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.tempty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA issued has completed before the columns are freed
        wait_parity_drain(&S.done, 0u);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A 2-D map over a row-major bf16 matrix [rows][K] with boxes of box_rows x 64.
bool make_map(CUtensorMap* map, const void* base, long long rows, long long K, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::atomic<int> g_gemm_attr[64];

}  // namespace

size_t tc_gemm_smem() { return sizeof(GSmem) + 1024; }

// D[M][N] (fp32, ldd) = alpha * A[M][K] . B[N][K]^T; A, B bf16 row-major, 16-byte aligned,
// K a multiple of 8.  cudaErrorInvalidValue when the shapes do not qualify.
cudaError_t tc_gemm_tn(const void* A, const void* B, float* D, long long M, long long N, long long K, long long ldd,
                       float alpha, cudaStream_t st) {
    if (M < 1 || N < 1 || K < 8 || K % 8 != 0 || M > (1LL << 31) - BM || N > (1LL << 31) - BN || K > (1LL << 31))
        return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_gemm_attr[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute((const void*)tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc_gemm_smem());
        if (e != cudaSuccess) return e;
        g_gemm_attr[dev].store(1, std::memory_order_release);
    }
    CUtensorMap ta, tb;
    if (!make_map(&ta, A, M, K, BM) || !make_map(&tb, B, N, K, BN)) return cudaErrorInvalidValue;
    // Tile order: the CTAs that run together share the tiles of the larger operand, which is
    // then read from HBM about once, while the smaller one is re-read (from L2 when it fits).
    // M-tiles vary fastest when A is the smaller operand (the head's logits: a chunk of hidden
    // rows against the whole weight plane), N-tiles otherwise.  One persistent CTA per SM
    // walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... of that order.
    const long long mt = (M + BM - 1) / BM, ntl = (N + BN - 1) / BN;
    if (mt * ntl > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int m_fast = M <= N ? 1 : 0;
    static std::atomic<int> sm_cache[64];
    int sms = sm_cache[dev].load(std::memory_order_acquire);
    if (sms <= 0) {
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        sm_cache[dev].store(sms, std::memory_order_release);
    }
    const long long tiles = mt * ntl;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms), 1, 1);
    cfg.blockDim = dim3(GT, 1, 1);
    cfg.dynamicSmemBytes = tc_gemm_smem();
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, ta, tb, D, ldd, (int)M, (int)N, (int)K, alpha, m_fast);
}

unsigned int gemm_watchdog(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_watchdog, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_watchdog, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}

}  // namespace vl
