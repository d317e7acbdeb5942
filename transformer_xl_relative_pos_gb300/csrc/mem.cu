// Segment memory of one Transformer-XL layer as a ring buffer.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.2: the hidden states of earlier segments are cached (a memory of the last
// M states, possibly spanning several segments) and concatenated, under a
// stop-gradient, in front of the current segment as extended context; §3.3's
// summary writes this as h~ = [SG(m) o h].  SG is the identity in a forward pass.
//
// Both kernels are pure row copies in 16-byte units with a grid-stride loop;
// HBM-bound.
#include "kernels.h"

namespace txl {
namespace {

// ext[b][t] = t < fill ? mem[b][(head - fill + t) mod cap] : h_new[b][t - fill]
__global__ void mem_concat_kernel(uint4 *__restrict__ ext, const uint4 *__restrict__ mem,
                                  const uint4 *__restrict__ h_new, int B, int fill, int head,
                                  int cap, int L, int row_vec)
{
    const int rows = fill + L;
    const long long total = (long long)B * rows * row_vec;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % row_vec);
        const long long br = e / row_vec;
        const int t = (int)(br % rows);
        const int b = (int)(br / rows);
        const uint4 *src;
        if (t < fill) {
            int slot = head - fill + t;
            slot += (slot < 0) ? cap : 0;
            src = mem + ((size_t)b * cap + slot) * row_vec;
        } else {
            src = h_new + ((size_t)b * L + (t - fill)) * row_vec;
        }
        ext[e] = src[c];
    }
}

// mem[b][(head + l) mod cap] = h_new[b][l] for l in [first_row, L)
__global__ void mem_write_kernel(uint4 *__restrict__ mem, const uint4 *__restrict__ h_new,
                                 int B, int L, int first_row, int head, int cap, int row_vec)
{
    const int rows = L - first_row;
    const long long total = (long long)B * rows * row_vec;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % row_vec);
        const long long br = e / row_vec;
        const int l = first_row + (int)(br % rows);
        const int b = (int)(br / rows);
        const int slot = (int)(((long long)head + l) % cap);
        mem[((size_t)b * cap + slot) * row_vec + c] = h_new[((size_t)b * L + l) * row_vec + c];
    }
}

int grid_for(long long total)
{
    long long blocks = (total + 255) / 256;
    const long long cap = 152LL * 16;  // enough blocks to fill every SM several times
    return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

} // namespace

cudaError_t launch_mem_concat(uint4 *ext, const uint4 *mem, const uint4 *h_new, int B,
                              int fill, int head, int cap, int L, int row_vec, cudaStream_t s)
{
    const long long total = (long long)B * (fill + L) * row_vec;
    if (total == 0) return cudaSuccess;
    mem_concat_kernel<<<grid_for(total), 256, 0, s>>>(ext, mem, h_new, B, fill, head, cap, L,
                                                      row_vec);
    return cudaGetLastError();
}

cudaError_t launch_mem_write(uint4 *mem, const uint4 *h_new, int B, int L, int first_row,
                             int head, int cap, int row_vec, cudaStream_t s)
{
    const long long total = (long long)B * (L - first_row) * row_vec;
    if (total == 0) return cudaSuccess;
    mem_write_kernel<<<grid_for(total), 256, 0, s>>>(mem, h_new, B, L, first_row, head, cap,
                                                     row_vec);
    return cudaGetLastError();
}

} // namespace txl
