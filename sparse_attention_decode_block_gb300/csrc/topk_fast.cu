// Exact top-k of score rows of up to 8192 columns: one block of 256
// threads per row runs block_topk (topk_block.cuh).
#include "topk_block.cuh"

namespace lsa {
namespace {

// Output index of column `col` of row `row`: the column, or for the fine
// pass of coarse-to-fine the token position it stands for.
__device__ __forceinline__ int32_t tf_out(const TopkArgs &a, int row, int col)
{
    if (!a.cand) return col;
    const int cb = a.cand[(int64_t)row * a.ncand + col / a.b];
    return cb * a.b + col % a.b;
}

template <int KPT>
__global__ void __launch_bounds__(kTfThreads) k_topk_fast(TopkArgs a)
{
    pdl_enter();
    __shared__ TopkScratch sm;
    const int row = blockIdx.x;
    int n = a.num_cols ? a.num_cols[row] : a.cols;
    n = max(0, min(n, a.cols));
    const float *srow = a.scores + (int64_t)row * a.cols;
    const bool aligned = (a.cols & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    int32_t *orow = a.idx + (int64_t)row * a.k;
    const int keff = block_topk<KPT>(srow, n, aligned, a.k, a.status, sm,
                                     [&](int pos, int col) { orow[pos] = tf_out(a, row, col); });
    for (int i = keff + (int)threadIdx.x; i < a.k; i += kTfThreads) orow[i] = -1;
}

}  // namespace
// Rows of up to kTfThreads * 32 columns; returns false (nothing launched)
// for wider rows.
bool launch_topk_fast(const TopkArgs &a, cudaStream_t s, cudaError_t *err)
{
    if (a.cols <= kTfThreads * 8) {
        *err = launch_step_kernel(k_topk_fast<8>, dim3(a.rows), dim3(kTfThreads), 0, s, a);
        if (*err != cudaSuccess) return true;
    } else if (a.cols <= kTfThreads * 32) {
        *err = launch_step_kernel(k_topk_fast<32>, dim3(a.rows), dim3(kTfThreads), 0, s, a);
        if (*err != cudaSuccess) return true;
    } else {
        return false;
    }
    *err = cudaGetLastError();
    return true;
}

}  // namespace lsa
