// Segment memory of one Transformer-XL layer as a ring buffer.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.2: the hidden states of earlier segments are cached (a memory of the last
// M states, possibly spanning several segments) and concatenated, under a
// stop-gradient, in front of the current segment as extended context; §3.3's
// summary writes this as h~ = [SG(m) o h].  SG is the identity in a forward pass.
//
// Both kernels are pure copies of 16-byte vectors, flattened per batch row
// over (row, vector) so that every block moves many rows whatever the row size
// (128-byte rows of per-head projected keys as well as d_model-wide hidden
// states); each thread keeps four vectors in flight.  HBM-bound.
#include "kernels.h"

namespace txl {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;

// Row and vector of flat index i: shift = log2(row_vec) when row_vec is a power
// of two (every d_model and head size here), else -1 (one division).
__device__ __forceinline__ int row_of(int i, int row_vec, int shift)
{
    return shift >= 0 ? (i >> shift) : i / row_vec;
}

// ext[b][t] = t < fill ? mem[b][(head - fill + t) mod cap] : h_new[b][t - fill]
__global__ void __launch_bounds__(kThreads) mem_concat_kernel(uint4 *__restrict__ ext,
                                                              const uint4 *__restrict__ mem,
                                                              const uint4 *__restrict__ h_new,
                                                              int fill, int head, int cap, int L,
                                                              int row_vec, int shift,
                                                              unsigned int *status)
{
    const int rows = fill + L;
    const int total = rows * row_vec;  // vectors of this batch row
    const long long b = blockIdx.y;
    const int base = blockIdx.x * kThreads * kVecPerThread + threadIdx.x;
    uint4 v[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = base + k * kThreads;
        if (i >= total) continue;
        const int t = row_of(i, row_vec, shift);
        const int c = i - t * row_vec;
        const uint4 *src;
        TXL_CHECK(t >= 0 && t < rows && c >= 0 && c < row_vec, status);
        if (t < fill) {
            int slot = head - fill + t;
            slot += (slot < 0) ? cap : 0;
            TXL_CHECK(slot >= 0 && slot < cap, status);
            src = mem + (b * cap + slot) * row_vec + c;
        } else {
            src = h_new + (b * L + (t - fill)) * row_vec + c;
        }
        v[k] = __ldcs(src);
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = base + k * kThreads;
        if (i < total) ext[b * total + i] = v[k];
    }
}

// mem[b][(head + l) mod cap] = h_new[b][l] for l in [first_row, L).
__global__ void __launch_bounds__(kThreads) mem_write_kernel(uint4 *__restrict__ mem,
                                                             const uint4 *__restrict__ h_new,
                                                             int L, int first_row, int head,
                                                             int cap, int row_vec, int shift,
                                                             unsigned int *status)
{
    const int total = (L - first_row) * row_vec;  // vectors of this batch row
    const long long b = blockIdx.y;
    const int base = blockIdx.x * kThreads * kVecPerThread + threadIdx.x;
    uint4 v[kVecPerThread];
    long long dst[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = base + k * kThreads;
        dst[k] = -1;
        if (i >= total) continue;
        const int r = row_of(i, row_vec, shift);
        const int c = i - r * row_vec;
        const int l = first_row + r;
        TXL_CHECK(l >= 0 && l < L && (head + l) % cap < cap, status);
        v[k] = __ldcs(h_new + (b * L + l) * row_vec + c);
        dst[k] = (b * cap + (head + l) % cap) * row_vec + c;
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k)
        if (dst[k] >= 0) mem[dst[k]] = v[k];
}

// dst[p][dst_row0 + r] = src[p][src_row0 + r] for r in [0, rows), planes p
// dst_plane / src_plane vectors apart: the k / v window of a memory kept in a
// larger buffer (compaction to the buffer's front, the segment's rows behind
// the memory's).
__global__ void __launch_bounds__(kThreads) rows_copy_kernel(uint4 *__restrict__ dst,
                                                             long long dst_plane, int dst_row0,
                                                             const uint4 *__restrict__ src,
                                                             long long src_plane, int src_row0,
                                                             int rows, int row_vec, int shift,
                                                             unsigned int *status)
{
    const int total = rows * row_vec;  // vectors of this plane
    const long long pl = blockIdx.y;
    const int base = blockIdx.x * kThreads * kVecPerThread + threadIdx.x;
    uint4 v[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = base + k * kThreads;
        if (i < total) {
            const int r = row_of(i, row_vec, shift);
            // both rows inside their planes
            TXL_CHECK((long long)(src_row0 + r + 1) * row_vec <= src_plane &&
                          (long long)(dst_row0 + r + 1) * row_vec <= dst_plane,
                      status);
            v[k] = __ldcs(src + pl * src_plane + (long long)(src_row0 + r) * row_vec + (i - r * row_vec));
        }
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = base + k * kThreads;
        if (i < total) {
            const int r = row_of(i, row_vec, shift);
            dst[pl * dst_plane + (long long)(dst_row0 + r) * row_vec + (i - r * row_vec)] = v[k];
        }
    }
}

int shift_of(int row_vec)
{
    if (row_vec <= 0 || (row_vec & (row_vec - 1))) return -1;
    int sh = 0;
    while ((1 << sh) < row_vec) ++sh;
    return sh;
}

} // namespace

cudaError_t launch_mem_concat(uint4 *ext, const uint4 *mem, const uint4 *h_new, int B,
                              int fill, int head, int cap, int L, int row_vec,
                              unsigned int *status, cudaStream_t s)
{
    const long long total = (long long)(fill + L) * row_vec;
    if (total == 0 || B == 0) return cudaSuccess;
    if (B > 65535 || total > 0x7fffffffLL - kThreads * kVecPerThread) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((total + kThreads * kVecPerThread - 1) / (kThreads * kVecPerThread));
    mem_concat_kernel<<<dim3(blocks, B), kThreads, 0, s>>>(ext, mem, h_new, fill, head, cap, L,
                                                           row_vec, shift_of(row_vec), status);
    return cudaGetLastError();
}

cudaError_t launch_mem_write(uint4 *mem, const uint4 *h_new, int B, int L, int first_row,
                             int head, int cap, int row_vec, unsigned int *status, cudaStream_t s)
{
    const long long total = (long long)(L - first_row) * row_vec;
    if (total <= 0 || B == 0) return cudaSuccess;
    if (B > 65535 || total > 0x7fffffffLL - kThreads * kVecPerThread) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((total + kThreads * kVecPerThread - 1) / (kThreads * kVecPerThread));
    mem_write_kernel<<<dim3(blocks, B), kThreads, 0, s>>>(mem, h_new, L, first_row, head, cap,
                                                          row_vec, shift_of(row_vec), status);
    return cudaGetLastError();
}

cudaError_t launch_rows_copy(uint4 *dst, long long dst_plane_vec, int dst_row0, const uint4 *src,
                             long long src_plane_vec, int src_row0, int planes, int rows,
                             int row_vec, unsigned int *status, cudaStream_t s)
{
    const long long total = (long long)rows * row_vec;
    if (total <= 0 || planes == 0) return cudaSuccess;
    if (planes > 65535 || total > 0x7fffffffLL - kThreads * kVecPerThread)
        return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((total + kThreads * kVecPerThread - 1) / (kThreads * kVecPerThread));
    rows_copy_kernel<<<dim3(blocks, planes), kThreads, 0, s>>>(
        dst, dst_plane_vec, dst_row0, src, src_plane_vec, src_row0, rows, row_vec, shift_of(row_vec),
        status);
    return cudaGetLastError();
}

} // namespace txl
