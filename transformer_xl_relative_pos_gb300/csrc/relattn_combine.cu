// Merge of the key-range partial results of a split attention call (the
// tensor-core and the short-segment kernels both write them): for every query
// row, out = sum_s 2^(lse_s - max) o_s / sum_s 2^(lse_s - max), the log-sum-exp
// identity of softmax over a union of disjoint key sets.
#include "kernels.h"

namespace txl {
namespace {

constexpr int DH = kTcDH;

// Merge of split-key partial results: out = sum_s w_s o_s / sum_s w_s with
// w_s = 2^(lse_s - max lse).  One warp per query row, two columns per lane.
// The splits' log-sum-exps are read one per lane (32 at a time), the weights
// handed out by shuffles, and the partial rows read eight splits at a time so
// that their loads overlap.
__global__ void relattn_combine_kernel(const float *__restrict__ part_o,
                                       const float *__restrict__ part_lse,
                                       __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                                       int n_splits, int rows)
{
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float mx = -INFINITY;
    for (int s = lane; s < n_splits; s += 32) mx = fmaxf(mx, part_lse[(size_t)s * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float wsum = 0.f, a0 = 0.f, a1 = 0.f;
    if (mx != -INFINITY) {
        for (int s0 = 0; s0 < n_splits; s0 += 32) {
            // weight of split s0 + lane (0 for a split without keys or past the end)
            const int sl = s0 + lane;
            const float l = (sl < n_splits) ? part_lse[(size_t)sl * rows + row] : -INFINITY;
            const float wl = (l == -INFINITY) ? 0.f : exp2f(l - mx);
            const int n = min(32, n_splits - s0);
            for (int e0 = 0; e0 < n; e0 += 8) {
                float2 o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s = s0 + min(e0 + e, n - 1);
                    o[e] = reinterpret_cast<const float2 *>(part_o + ((size_t)s * rows + row) * DH)[lane];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float w = __shfl_sync(0xffffffffu, wl, (e0 + e) & 31);
                    if (e0 + e >= n) w = 0.f;
                    // a split without keys has w = 0 and a zero partial row
                    if (w != 0.f) {
                        wsum += w;
                        a0 = fmaf(w, o[e].x, a0);
                        a1 = fmaf(w, o[e].y, a1);
                    }
                }
            }
        }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    reinterpret_cast<__nv_bfloat162 *>(out + (size_t)row * DH)[lane] =
        __floats2bfloat162_rn(a0 * inv, a1 * inv);
    if (lse && lane == 0)
        lse[row] = (wsum > 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

} // namespace

cudaError_t launch_relattn_combine(const float *part_o, const float *part_lse,
                                   __nv_bfloat16 *out, float *lse, int n_splits, int rows,
                                   cudaStream_t s)
{
    const int warps = 8;
    const int blocks = (rows + warps - 1) / warps;
    relattn_combine_kernel<<<blocks, warps * 32, 0, s>>>(part_o, part_lse, out, lse, n_splits,
                                                         rows);
    return cudaGetLastError();
}

} // namespace txl
