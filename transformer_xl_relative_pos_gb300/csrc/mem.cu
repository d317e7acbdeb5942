// Segment memory of one Transformer-XL layer as a ring buffer.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.2: the hidden states of earlier segments are cached (a memory of the last
// M states, possibly spanning several segments) and concatenated, under a
// stop-gradient, in front of the current segment as extended context; §3.3's
// summary writes this as h~ = [SG(m) o h].  SG is the identity in a forward pass.
//
// Both kernels are pure row copies in 16-byte units, one block per row;
// HBM-bound.
#include "kernels.h"

namespace txl {
namespace {

// One block per (row, batch); the row's 16-byte vectors spread over the threads.
// ext[b][t] = t < fill ? mem[b][(head - fill + t) mod cap] : h_new[b][t - fill]
__global__ void mem_concat_kernel(uint4 *__restrict__ ext, const uint4 *__restrict__ mem,
                                  const uint4 *__restrict__ h_new, int fill, int head, int cap,
                                  int L, int row_vec)
{
    const int t = blockIdx.x;
    const int b = blockIdx.y;
    const uint4 *src;
    if (t < fill) {
        int slot = head - fill + t;
        slot += (slot < 0) ? cap : 0;
        src = mem + ((size_t)b * cap + slot) * row_vec;
    } else {
        src = h_new + ((size_t)b * L + (t - fill)) * row_vec;
    }
    uint4 *dst = ext + ((size_t)b * (fill + L) + t) * row_vec;
    for (int c = threadIdx.x; c < row_vec; c += blockDim.x) dst[c] = src[c];
}

// mem[b][(head + l) mod cap] = h_new[b][l] for l in [first_row, L).  Each block
// copies kRowsPerBlock rows so that every thread has several loads in flight.
constexpr int kRowsPerBlock = 4;
__global__ void mem_write_kernel(uint4 *__restrict__ mem, const uint4 *__restrict__ h_new, int L,
                                 int first_row, int head, int cap, int row_vec)
{
    const int l0 = first_row + blockIdx.x * kRowsPerBlock;
    const int b = blockIdx.y;
    const int nrows = min(kRowsPerBlock, L - l0);
    for (int c = threadIdx.x; c < row_vec; c += blockDim.x) {
        uint4 v[kRowsPerBlock];
#pragma unroll
        for (int r = 0; r < kRowsPerBlock; ++r)
            if (r < nrows) v[r] = h_new[((size_t)b * L + l0 + r) * row_vec + c];
#pragma unroll
        for (int r = 0; r < kRowsPerBlock; ++r)
            if (r < nrows) {
                const int slot = (int)(((long long)head + l0 + r) % cap);
                mem[((size_t)b * cap + slot) * row_vec + c] = v[r];
            }
    }
}

int threads_for(int row_vec) { return row_vec >= 256 ? 256 : ((row_vec + 31) / 32) * 32; }

} // namespace

cudaError_t launch_mem_concat(uint4 *ext, const uint4 *mem, const uint4 *h_new, int B,
                              int fill, int head, int cap, int L, int row_vec, cudaStream_t s)
{
    const int rows = fill + L;
    if (rows == 0 || B == 0) return cudaSuccess;
    if (B > 65535) return cudaErrorInvalidValue;
    mem_concat_kernel<<<dim3(rows, B), threads_for(row_vec), 0, s>>>(ext, mem, h_new, fill, head,
                                                                     cap, L, row_vec);
    return cudaGetLastError();
}

cudaError_t launch_mem_write(uint4 *mem, const uint4 *h_new, int B, int L, int first_row,
                             int head, int cap, int row_vec, cudaStream_t s)
{
    const int rows = L - first_row;
    if (rows <= 0 || B == 0) return cudaSuccess;
    if (B > 65535) return cudaErrorInvalidValue;
    const int blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    mem_write_kernel<<<dim3(blocks, B), threads_for(row_vec), 0, s>>>(mem, h_new, L, first_row,
                                                                      head, cap, row_vec);
    return cudaGetLastError();
}

} // namespace txl
