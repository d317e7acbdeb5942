// Internal launch interface of the short-segment (decode) attention kernel.
// Not part of the public ABI.
#pragma once

#include "kernels.h"

namespace txl {

// Short-segment (decode) kernels: L <= kDecodeMaxL queries per (batch, head);
// the keys are split into n_splits ranges of whole 32-key chunks.  The
// CUDA-core kernel takes L <= kDecodeFmaMaxL (one query: its per-key arithmetic
// grows with L), the warp-MMA kernel the rest.
constexpr int kDecodeMaxL = 8;
constexpr int kDecodeFmaMaxL = 1;
constexpr int kDecodeMaxCluster = 8;  // portable cluster size
// Tensor maps of the tensor-core kernel: k and v [B*H planes][K][64] read in
// boxes of 32 rows, the table [H][r_rows][64] in boxes of 40 rows (the 32 + L - 1
// rows one chunk needs); bf16, 128-byte swizzle.
constexpr int kDecodeMmaKeyBox = 32;
constexpr int kDecodeMmaTableBox = 40;

struct DecodeParams {
    int B, H, M, L, K;
    int r_rows;         // table rows per head (>= K)
    int r_off;          // r_rows - K
    int n_splits;       // key ranges per (batch, head); > 1 writes partials
    long long kv_stride;  // elements between consecutive (b, h) planes of k and v
    float scale_log2;   // scale * log2(e)
    const __nv_bfloat16 *q;   // [B][H][L][64]
    const __nv_bfloat16 *k;   // [B*H planes, kv_stride apart][K][64]
    const __nv_bfloat16 *v;   // [B*H planes, kv_stride apart][K][64]
    const __nv_bfloat16 *r;   // [H][r_rows][64]
    const __nv_bfloat16 *u;   // [H][64]
    const __nv_bfloat16 *vb;  // [H][64]
    __nv_bfloat16 *out;       // [B][H][L][64]            (n_splits == 1)
    float *lse;               // [B][H][L] natural log or null
    float *part_o;            // [n_splits][B*H*L][64]   (n_splits > 1)
    float *part_lse;          // [n_splits][B*H*L], log2 domain
    int cluster;              // 1: the n_splits ranges of a head are one thread-block
                              // cluster and merge in distributed shared memory
    unsigned int *status;     // device status word
    unsigned long long wait_ns;
};

// Keys of one split of a head's K keys over n blocks: a whole number of 32-key
// chunks.  Shared by the kernel and the host's choice of splits.
__host__ __device__ inline int decode_span(int K, int n_splits)
{
    return ((K + n_splits - 1) / n_splits + 31) / 32 * 32;
}
int decode_chunk_keys();                // 32
// CUDA-core kernel (L <= kDecodeFmaMaxL): resident blocks per SM, launch.
int decode_blocks_per_sm(int L);
cudaError_t launch_relattn_decode(const DecodeParams &p, cudaStream_t s);
// Tensor-core kernel (L <= kDecodeMaxL): resident blocks per SM, launch.
int decode_mma_blocks_per_sm(int L);
cudaError_t launch_relattn_decode_mma(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_r, const DecodeParams &p,
                                      cudaStream_t s);

} // namespace txl
