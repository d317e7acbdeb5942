// Internal launch interface between the C-ABI layer (txl_api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

// Bits of the device status word (read and cleared by txl_device_status).
#define TXL_STATUS_TIMEOUT 1u  // a bounded barrier wait gave up
#define TXL_STATUS_INDEX 2u    // a device-side index check failed (TXL_DEBUG builds)

// Device-side index checks of the debug build (compiled with -DTXL_DEBUG): a
// failed check records TXL_STATUS_INDEX in the status word and the kernel goes
// on (no trap); release builds compile the checks away.
#ifdef TXL_DEBUG
#define TXL_CHECK(cond, status)                                                   \
    do {                                                                          \
        if (!(cond)) atomicOr((status), TXL_STATUS_INDEX);                        \
    } while (0)
#else
#define TXL_CHECK(cond, status) \
    do {                        \
    } while (0)
#endif

namespace txl {

// Tile shape of the tensor-core attention kernel.
constexpr int kTcBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kTcBN = 128;  // keys per tile
constexpr int kTcDH = 64;   // head size

struct TcParams {
    int B, H, M, L, K;
    int r_off;        // r_rows - K: row offset of the K-key table inside r
    int n_qtiles;     // ceil(L / kTcBM)
    int n_splits;     // key-range splits per query tile
    float scale_log2; // scale * log2(e)
    const __nv_bfloat16 *u;  // [H][64]
    const __nv_bfloat16 *vb; // [H][64]
    __nv_bfloat16 *out;      // [B][H][L][64]            (n_splits == 1)
    float *lse;              // [B][H][L] natural log or null
    float *part_o;           // [n_splits][B*H][L][64]   (n_splits > 1)
    float *part_lse;         // [n_splits][B*H][L], log2 domain
    unsigned int *status;    // device status word
    unsigned long long wait_ns;
};

// Dynamic shared memory the tensor-core kernel needs (bytes).
size_t tc_smem_bytes();

cudaError_t launch_relattn_tc(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const CUtensorMap &tm_r,
                              const TcParams &p, cudaStream_t s);

cudaError_t launch_relattn_combine(const float *part_o, const float *part_lse,
                                   __nv_bfloat16 *out, float *lse, int n_splits, int rows,
                                   cudaStream_t s);

struct F32Params {
    const float *q, *k, *v, *r, *u, *vb;
    float *out, *lse;
    int B, H, M, L, K, r_rows;
    long long kv_stride;  // elements between consecutive (b, h) planes of k and v
    float scale;
};

cudaError_t launch_relattn_f32(const F32Params &p, cudaStream_t s);

cudaError_t launch_rel_pos_emb(void *R, int K, int d_model, bool bf16, cudaStream_t s);

// Rows [src_row0, src_row0 + rows) of every plane of src into rows
// [dst_row0, ...) of the same plane of dst (planes rows apart by the strides,
// in 16-byte units); row_vec = row bytes / 16.  The row ranges of one plane must
// not overlap.
cudaError_t launch_rows_copy(uint4 *dst, long long dst_plane_vec, int dst_row0, const uint4 *src,
                             long long src_plane_vec, int src_row0, int planes, int rows,
                             int row_vec, unsigned int *status, cudaStream_t s);

// Row copies for the segment memory; row_vec = row bytes / 16.
cudaError_t launch_mem_concat(uint4 *ext, const uint4 *mem, const uint4 *h_new, int B,
                              int fill, int head, int cap, int L, int row_vec,
                              unsigned int *status, cudaStream_t s);
cudaError_t launch_mem_write(uint4 *mem, const uint4 *h_new, int B, int L, int first_row,
                             int head, int cap, int row_vec, unsigned int *status, cudaStream_t s);

// Projection of a segment's states h [M = B*L][K] by stacked weights [N][K]
// (N = n_out * H * 64; outputs in order, e.g. q, k, v), written per head: output
// o, head hd, batch b, segment row l goes to out[o] + ((b*H + hd) *
// plane_stride[o] + row0[o] + l) * 64; optionally mem[b][(mem_head + l) mod
// mem_cap] = h[b][l] for l >= mem_first (the memory update).
struct ProjParams {
    int M, N, K, L, B, H, n_out;
    const __nv_bfloat16 *h;
    __nv_bfloat16 *out[3];
    long long plane_stride[3];  // elements
    int row0[3];
    __nv_bfloat16 *mem;         // [B][mem_cap][K] or null
    int mem_cap, mem_head, mem_first;
    unsigned int *status;
    unsigned long long wait_ns;
};
int project_smem_bytes();
cudaError_t launch_project(const CUtensorMap &tm_h, const CUtensorMap &tm_w, const ProjParams &p,
                           cudaStream_t s);

// Backward of the relative attention (relattn_bwd.cu): bf16 inputs, fp32
// gradients.  lse2 / dsum / part point into the caller's workspace: per query
// row the log2-sum-exp of the scaled scores and D = sum_j P dP, per (b*H + h,
// 64-row query chunk) the two bias partials (64 + 64 floats).
struct BwdParams {
    const __nv_bfloat16 *q, *k, *v, *r, *u, *vb, *dout;
    float *dq, *dk, *dv, *dr, *du, *dvb;
    float *lse2, *dsum, *part;
    float *dq_part;  // segments of at most two row chunks: dq per key split
    float *g_all;    // g of every visited pair: [B*H][L][Kd], for the table gradient
    int B, H, M, L, K, r_rows;
    int Kd;          // K rounded up to a whole tile (the row stride of g_all)
    float scale, scale_log2;
    unsigned int *status;
};
constexpr int kBwdRows = 64;  // query rows (and keys, distances) per tile
constexpr int kBwdMaxSplits = 8;  // key splits of the two-chunk statistics and dq / dk / dv launches
size_t bwd_workspace_bytes(int B, int H, int L, int M);
size_t bwd_dq_part_offset(int B, int H, int L);  // where the dq partials start in the workspace
size_t bwd_g_offset(int B, int H, int L);        // where g of every pair starts
cudaError_t launch_relattn_bwd(const BwdParams &p, cudaStream_t s);

cudaError_t launch_wait_probe(unsigned int *status, unsigned long long wait_ns, cudaStream_t s);
// One thread fails one index check (a no-op in release builds).
cudaError_t launch_index_probe(unsigned int *status, cudaStream_t s);

} // namespace txl
