// The frozen vocabulary head around the row losses (cortiq-engine train_head.rs: the
// teacher's topk and the student's head_kl), on chunks of rows so that the [ntok][V]
// logits are never held whole:
//
//   teacher top-k  per chunk: logits = hidden . W^T (bf16 inputs, fp32 accumulation and
//                  output), then the top-k of each logits row (vl_topk_rows).  No host
//                  readback between chunks (the page downloads each chunk).
//   head KL step   per chunk: logits = hidden . W^T as above, the CE + top-k KL gradient
//                  written over them in one pass (vl_ce_kl_fused), the gradient rounded
//                  to bf16 (the page's cvt_cols), then dx = dx_scale * dlogits . wt^T with
//                  the transposed weight plane wt [hs][V] (the page's mm(wt, ..., 1/gscale)).
//
// The GEMMs run on this library's tensor-core kernel (gemm.cu: TMA, tcgen05.mma, tensor
// memory).  Without wt, or with V not a multiple of 8, the backward GEMM reads W itself
// through cuBLASLt instead, with a workspace carved from the caller's (the library
// allocates nothing).
#include "vl_device.cuh"
#include "vl_internal.h"
#include "vloss.h"

#include <cublasLt.h>
#include <cuda_bf16.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

namespace vl {
namespace {

constexpr long long kLtWorkspace = 32ll << 20;    // cuBLASLt workspace carved from the caller's

std::mutex g_lt_mu;
cublasLtHandle_t g_lt[64] = {};

cublasLtHandle_t lt_handle(int dev) {
    std::lock_guard<std::mutex> lk(g_lt_mu);
    if (!g_lt[dev] && cublasLtCreate(&g_lt[dev]) != CUBLAS_STATUS_SUCCESS) g_lt[dev] = nullptr;
    return g_lt[dev];
}

// One cached plan per (device, ops, shape, leading dimensions, types).
struct Plan {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulAlgo_t algo;
    bool ok = false;
};
using PlanKey = std::tuple<int, int, int, long long, long long, long long, long long, long long, long long, int>;
std::map<PlanKey, Plan> g_plans;

// Column-major C (m x n, ldc) = alpha * op(A) op(B), A and B bf16, C of type ctype
// (fp32 or bf16), fp32 accumulation.  0 on success, else a cuBLASLt status.
int lt_matmul(cublasOperation_t opa, cublasOperation_t opb, long long m, long long n, long long k, const void* A,
              long long lda, const void* B, long long ldb, void* C, long long ldc, cudaDataType ctype, float alpha,
              void* ws, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    cublasLtHandle_t h = lt_handle(dev);
    if (!h) return -2;
    const PlanKey key{dev, (int)opa, (int)opb, m, n, k, lda, ldb, ldc, (int)ctype};
    Plan* p;
    {
        std::lock_guard<std::mutex> lk(g_lt_mu);
        p = &g_plans[key];
        if (!p->ok) {
            if (cublasLtMatmulDescCreate(&p->op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return -3;
            cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa));
            cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb));
            const bool ta = opa == CUBLAS_OP_T, tb = opb == CUBLAS_OP_T;
            cublasLtMatrixLayoutCreate(&p->la, CUDA_R_16BF, ta ? k : m, ta ? m : k, lda);
            cublasLtMatrixLayoutCreate(&p->lb, CUDA_R_16BF, tb ? n : k, tb ? k : n, ldb);
            cublasLtMatrixLayoutCreate(&p->lc, ctype, m, n, ldc);
            cublasLtMatmulPreference_t pref;
            cublasLtMatmulPreferenceCreate(&pref);
            const size_t wsb = (size_t)kLtWorkspace;
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb));
            cublasLtMatmulHeuristicResult_t res;
            int nres = 0;
            const cublasStatus_t s =
                cublasLtMatmulAlgoGetHeuristic(h, p->op, p->la, p->lb, p->lc, p->lc, pref, 1, &res, &nres);
            cublasLtMatmulPreferenceDestroy(pref);
            if (s != CUBLAS_STATUS_SUCCESS || nres < 1) return (int)(s ? s : -4);
            p->algo = res.algo;
            p->ok = true;
        }
    }
    const float beta = 0.f;
    const cublasStatus_t s = cublasLtMatmul(h, p->op, &alpha, A, p->la, B, p->lb, &beta, C, p->lc, C, p->lc, &p->algo,
                                            ws, (size_t)kLtWorkspace, st);
    return s == CUBLAS_STATUS_SUCCESS ? 0 : (int)s;
}

// Row-major logits[rows][V] (ld V) = hidden[rows][hs] . W[V][hs]^T on the tensor cores.
int head_logits(const void* hidden, long long rows, long long hs, const void* w, long long V, float* logits,
                cudaStream_t st) {
    const cudaError_t e = tc_gemm_tn(hidden, w, logits, rows, V, hs, V, 1.0f, st);
    return e == cudaSuccess ? 0 : -(int)e;
}

// Row-major dx[rows][hs] = alpha * g[rows][V] . W[V][hs]: with the transposed plane
// wt[hs][V] a tensor-core GEMM (g . wt^T, both K-major); else cuBLASLt over W, column-major
// dx^T (hs x rows) = W^T (hs x V, the row-major W read column-major) . g^T (V x rows).
int head_dx(const void* g, long long rows, long long V, const void* w, const void* wt, long long hs, float* dx,
            float alpha, void* ws, cudaStream_t st) {
    if (wt && V % 8 == 0) {
        const cudaError_t e = tc_gemm_tn(g, wt, dx, rows, hs, V, hs, alpha, st);
        return e == cudaSuccess ? 0 : -(int)e;
    }
    return lt_matmul(CUBLAS_OP_N, CUBLAS_OP_N, hs, rows, V, w, hs, g, V, dx, hs, CUDA_R_32F, alpha, ws, st);
}

// fp32 -> bf16, nearest even (the page's cvt_cols of the gradient); both buffers
// 16-byte aligned, any n.
__global__ void cvt_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ out, long long n) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const long long n4 = n / 4;
    const float4* in4 = reinterpret_cast<const float4*>(in);
    uint2* out4 = reinterpret_cast<uint2*>(out);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        const float4 v = in4[i];
        uint32_t a, b;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(a) : "f"(v.y), "f"(v.x));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(v.w), "f"(v.z));
        out4[i] = make_uint2(a, b);
    }
    const long long t = 4 * n4 + threadIdx.x;
    if (blockIdx.x == 0 && t < n) {
        const __nv_bfloat16 h = __float2bfloat16_rn(in[t]);
        out[t] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

cudaError_t launch_cvt(const float* in, uint16_t* out, long long n, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long n4 = n / 4;
    long long blocks = (n4 + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cvt_bf16_kernel, in, out, n);
}

long long align256(long long b) { return (b + 255) / 256 * 256; }

}  // namespace

// ---------------------------------------------------------------- workspace sizes

long long teacher_ws_bytes(long long rows, long long V, int k) {
    const long long tk = vl_topk_workspace_bytes(rows, V, k);
    return kLtWorkspace + align256(4 * rows * V) + align256(tk);
}

long long head_kl_ws_bytes(long long rows, long long V) {
    return kLtWorkspace + align256(4 * rows * V) + align256(2 * rows * V);
}

// The largest chunk of rows (at most `want`) whose workspace fits `bytes`.
long long chunk_rows(long long want, long long bytes, long long (*size)(long long, long long, int), long long V,
                     int k) {
    if (want < 1 || size(1, V, k) > bytes) return 0;
    long long lo = 1, hi = want;
    while (lo < hi) {
        const long long mid = (lo + hi + 1) / 2;
        if (size(mid, V, k) <= bytes) lo = mid; else hi = mid - 1;
    }
    return lo;
}

long long head_kl_ws_bytes3(long long rows, long long V, int) { return head_kl_ws_bytes(rows, V); }

int teacher_topk(const uint16_t* hidden, long long hs, const uint16_t* w, long long V, long long ntok, int k,
                       long long ls, long long le, uint32_t* ids, float* probs, int32_t* err, void* ws,
                       long long ws_bytes, cudaStream_t st, char* msg, size_t msg_len) {
    const long long chunk = chunk_rows(le - ls, ws_bytes, teacher_ws_bytes, V, k);
    if (chunk < 1) {
        snprintf(msg, msg_len, "workspace of %lld bytes is below the %lld a row needs", ws_bytes,
                 teacher_ws_bytes(1, V, k));
        return VL_EINVAL;
    }
    char* base = static_cast<char*>(ws);
    void* lt_ws = base;
    float* logits = reinterpret_cast<float*>(base + kLtWorkspace);
    void* tk_ws = base + kLtWorkspace + align256(4 * chunk * V);
    const long long tk_bytes = ws_bytes - kLtWorkspace - align256(4 * chunk * V);
    for (long long r0 = ls; r0 < le; r0 += chunk) {
        const long long r1 = r0 + chunk < le ? r0 + chunk : le;
        const long long rows = r1 - r0;
        const int s = head_logits(hidden + r0 * hs, rows, hs, w, V, logits, st);
        if (s) {
            snprintf(msg, msg_len, "logits GEMM failed (%d)", s);
            return VL_ELAUNCH;
        }
        const vl_status v = vl_topk_rows(logits, V, rows, V, k, 0, rows, ids + r0 * k, probs + r0 * k, err, tk_ws,
                                         tk_bytes, st);
        if (v) {
            snprintf(msg, msg_len, "top-k of a chunk: %s", vl_last_error_string());
            return v;
        }
    }
    return VL_OK;
}

int head_kl(const uint16_t* hidden, long long hs, const uint16_t* w, const uint16_t* wt, long long V, long long ntok,
                  const uint32_t* labels, const uint32_t* tid, const float* tp, int k, float coef, float ce_coef,
                  float dx_scale, long long ls, long long le, float* dx, float* kl_loss, float* ce_loss,
                  float* ce_mean, int32_t* err, void* ws, long long ws_bytes, cudaStream_t st, char* msg,
                  size_t msg_len) {
    const long long chunk = chunk_rows(ntok, ws_bytes, head_kl_ws_bytes3, V, k);
    if (chunk < 1) {
        snprintf(msg, msg_len, "workspace of %lld bytes is below the %lld a row needs", ws_bytes,
                 head_kl_ws_bytes(1, V));
        return VL_EINVAL;
    }
    char* base = static_cast<char*>(ws);
    void* lt_ws = base;
    float* logits = reinterpret_cast<float*>(base + kLtWorkspace);
    uint16_t* g16 = reinterpret_cast<uint16_t*>(base + kLtWorkspace + align256(4 * chunk * V));
    for (long long r0 = 0; r0 < ntok; r0 += chunk) {
        const long long r1 = r0 + chunk < ntok ? r0 + chunk : ntok;
        const long long rows = r1 - r0;
        int s = head_logits(hidden + r0 * hs, rows, hs, w, V, logits, st);
        if (s) {
            snprintf(msg, msg_len, "logits GEMM failed (%d)", s);
            return VL_ELAUNCH;
        }
        const long long a = ls - r0 < 0 ? 0 : (ls - r0 > rows ? rows : ls - r0);
        const long long b = le - r0 < 0 ? 0 : (le - r0 > rows ? rows : le - r0);
        vl_status v = vl_ce_kl_fused(logits, V, rows, V, labels + r0, tid + r0 * k, tp + r0 * k, k, coef, ce_coef,
                                     a, b > a ? b : a, kl_loss + r0, ce_loss + r0, nullptr, nullptr, nullptr, err,
                                     st);
        if (v) {
            snprintf(msg, msg_len, "loss of a chunk: %s", vl_last_error_string());
            return v;
        }
        cudaError_t e = launch_cvt(logits, g16, rows * V, st);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "conversion kernel: %s", cudaGetErrorString(e));
            return VL_ELAUNCH;
        }
        s = head_dx(g16, rows, V, w, wt, hs, dx + r0 * hs, dx_scale, lt_ws, st);
        if (s) {
            snprintf(msg, msg_len, "dx GEMM failed (%d)", s);
            return VL_ELAUNCH;
        }
    }
    if (ce_mean) {
        const vl_status v = vl_window_mean(ce_loss, ntok, ls, le, ce_mean, st);
        if (v) {
            snprintf(msg, msg_len, "mean: %s", vl_last_error_string());
            return v;
        }
    }
    return VL_OK;
}

}  // namespace vl
