// Internal interface between the C ABI (vloss_api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vl {

// Work of one row-engine launch.  Column indices are relative to col0.
struct RowParams {
    float* x;                 // logits, column 0 of row 0
    long long ld, ntok, V, col0, ncols;
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
    long long wait_limit;     // SM cycles after which a wait gives up (normally about 2 s)
    long long withhold;       // test hook: body tile of CTA 0 the producer never issues (-1: none)
    unsigned int* ws;         // tail split (CE fused): exchange workspace, see rows.cu
    int split;                // 1: the rows past the last full wave are split over all CTAs
};

// Exchange workspace of the tail split: a header (generation, ticket) and one 16-byte
// slot per (CTA, tail segment).
constexpr int kWsHeaderWords = 4;
constexpr long long ws_bytes_for(long long ctas) { return 4LL * kWsHeaderWords + 32LL * ctas; }

enum RowOp : int { kCeFused = 0, kCeFwd = 1, kCeBwd = 2, kKl = 3 };

// Row-engine geometry limits (rows.cu).
constexpr int kConsumerWarps = 15;        // + one producer warp: 16 warps, up to 128 registers a thread
constexpr int kVec = 2;                   // row engine: float4s of each tile per consumer thread
constexpr int kTileF = 4 * 32 * kConsumerWarps * kVec;   // floats per pipeline tile (15 KB)
constexpr int kSlots = 12;                // tiles in the shared-memory ring (180 KB)
constexpr int kMaxCluster = 8;

// Launch `op` over P; `resident` selects the self-contained mode that computes the
// row statistics itself (CE fused, KL without given statistics).  Returns a CUDA
// error code.
cudaError_t launch_rows(int op, bool resident, const RowParams& P, int nclusters, cudaStream_t st);

// Max active clusters of size c for the row kernel of `op` on the current device.
int row_max_clusters(int op, bool resident, int c);

unsigned int rows_watchdog(bool clear);

// Top-k (topk.cu).
cudaError_t launch_topk(const float* x, long long ld, long long ntok, long long V, int k,
                        long long ls, long long le, uint32_t* ids, float* probs, int* err,
                        cudaStream_t st);
unsigned int topk_watchdog(bool clear);

}  // namespace vl
