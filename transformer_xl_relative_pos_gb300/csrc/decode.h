// Internal launch interface of the short-segment (decode) attention kernel.
// Not part of the public ABI.
#pragma once

#include "kernels.h"

namespace txl {

// Short-segment (decode) kernel: L <= kDecodeMaxL queries per (batch, head);
// the keys are split into n_splits ranges of whole 32-key chunks.
constexpr int kDecodeMaxL = 6;
constexpr int kDecodeMaxCluster = 8;  // portable cluster size

struct DecodeParams {
    int B, H, M, L, K;
    int r_rows;         // table rows per head (>= K)
    int r_off;          // r_rows - K
    int n_splits;       // key ranges per (batch, head); > 1 writes partials
    float scale_log2;   // scale * log2(e)
    const __nv_bfloat16 *q;   // [B][H][L][64]
    const __nv_bfloat16 *k;   // [B][H][K][64]
    const __nv_bfloat16 *v;   // [B][H][K][64]
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
int decode_blocks_per_sm(int L);        // resident decode blocks per SM for L queries

cudaError_t launch_relattn_decode(const DecodeParams &p, cudaStream_t s);

} // namespace txl
