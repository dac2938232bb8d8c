// Internal interface between the C ABI (vloss_api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vl {

// Element types of the logits.
enum Dtype : int { kF32 = 0, kBf16 = 1 };

// Work of one row-engine launch.  Column indices are relative to col0.
struct RowParams {
    void* x;                  // logits (fp32 or bf16, as dtype), column 0 of row 0
    int dtype;
    long long ld, ntok, V, col0, ncols;
    long long rbeg, rend;     // rows this launch walks (a launch may take part of [0, ntok))
    const uint32_t* labels;   // CE ops; KL fold (nullable)
    const uint32_t* tid;      // KL teacher ids [ntok][k]
    const float* tp;          // KL teacher probabilities [ntok][k]
    int k;
    float cg;                 // multiplier of softmax in the gradient
    float coef;               // KL: teacher scatter coefficient
    float ce_coef;            // one-hot subtraction coefficient (0: none)
    long long ls, le;         // loss window
    const float* lse_in;      // given row statistics (stats_in wins)
    const float* stats_in;
    float* loss;              // per-row loss (CE loss / KL / CE loss part)
    float* ce_loss;           // self-contained KL with labels: the CE loss of the row as well (nullable)
    float* lse_out;
    float* stats_out;
    int* err;
    int csize;                // CTAs per row (cluster size)
    int mixed;                // fused CE on 2-CTA clusters: each CTA takes whole rows of its cluster's
                              // block, and an odd block's last row is split over the pair
    long long wait_limit;     // SM cycles after which a wait gives up (normally about 2 s)
    long long withhold;       // test hook: body tile of CTA 0 the producer never issues (-1: none)
};

enum RowOp : int { kCeFused = 0, kCeFwd = 1, kCeBwd = 2, kKl = 3 };

// Row-engine geometry limits (rows.cu).
constexpr int kConsumerWarps = 15;        // + one producer warp: 16 warps, up to 128 registers a thread
constexpr int kVec = 4;                   // row engine: 16-byte chunks of each tile per consumer thread
constexpr int kTileB = 16 * 32 * kConsumerWarps * kVec;  // bytes per pipeline tile (30 KB)
constexpr int kTileF = kTileB / 4;        // fp32 elements per tile
constexpr int kSlots = 6;                 // tiles in the shared-memory ring (180 KB)
constexpr int kMaxCluster = 8;

// Launch `op` over P; `resident` selects the self-contained mode that computes the
// row statistics itself (CE fused, KL without given statistics).  Returns a CUDA
// error code.
cudaError_t launch_rows(int op, bool resident, const RowParams& P, int nclusters, cudaStream_t st);

// Max active clusters of size c for the row kernel of `op` on the current device.
int row_max_clusters(int op, bool resident, int c, int dtype);

unsigned int rows_watchdog(bool clear);

// Top-k (topk.cu): exact, rows [ls, le), or the *nlist rows of list when list is given.
cudaError_t launch_topk(const float* x, long long ld, long long ntok, long long V, int k,
                        long long ls, long long le, const int* list, const int* nlist,
                        uint32_t* ids, float* probs, int* err, cudaStream_t st);
unsigned int topk_watchdog(bool clear);

// Top-k of long rows in one streaming kernel with filter and finish warps (topk_stream.cu).
int topk_filter_spec_a(long long V, int k);      // 0: the rows do not qualify
int topk_filter_capw(long long V, int k);        // slots of a warp's candidate region
long long topk_ws_bytes(long long rows, long long V, int k, long long ctas);
cudaError_t launch_topk_stream(const float* x, long long ld, long long V, int k, long long ls, long long le,
                               uint32_t* ids, float* probs, int* err, void* ws, long long ws_bytes,
                               long long wait_limit, cudaStream_t st);
unsigned int topk_stream_watchdog(bool clear);
// The device address of the fixed scratch array of vl_topk_rows_noalloc on the current
// device (looked up once per device).
cudaError_t topk_noalloc_scratch(void** out);

// The head GEMM on the tensor cores (gemm.cu): D[M][N] (fp32, ldd) = alpha * A[M][K] . B[N][K]^T,
// A and B bf16 row-major, 16-byte aligned, K a multiple of 8.
cudaError_t tc_gemm_tn(const void* A, const void* B, float* D, long long M, long long N, long long K, long long ldd,
                       float alpha, cudaStream_t st);
unsigned int gemm_watchdog(bool clear);

// The vocabulary head around the losses (head.cu).  Arguments as the C entry points;
// msg receives the reason of a failure.
long long teacher_ws_bytes(long long rows, long long V, int k);
long long head_kl_ws_bytes(long long rows, long long V);
int teacher_topk(const uint16_t* hidden, long long hs, const uint16_t* w, long long V, long long ntok, int k,
                 long long ls, long long le, uint32_t* ids, float* probs, int32_t* err, void* ws, long long ws_bytes,
                 cudaStream_t st, char* msg, size_t msg_len);
int head_kl(const uint16_t* hidden, long long hs, const uint16_t* w, const uint16_t* wt, long long V, long long ntok,
            const uint32_t* labels, const uint32_t* tid, const float* tp, int k, float coef, float ce_coef,
            float dx_scale, long long ls, long long le, float* dx, float* kl_loss, float* ce_loss, float* ce_mean,
            int32_t* err, void* ws, long long ws_bytes, cudaStream_t st, char* msg, size_t msg_len);
}  // namespace vl
