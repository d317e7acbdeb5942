// C-ABI entry points declared in include/txl.h: argument validation, TMA
// descriptor construction, launch configuration and the device status word.
// All arithmetic happens in the kernels (relattn_tc.cu, relattn_decode.cu,
// relattn_combine.cu, relattn_f32.cu, relpos.cu, mem.cu); this file only
// checks and dispatches.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels.h"
#include "decode.h"
#include "txl.h"

namespace {

// Kernels OR their failure bits into this word (bit 0: barrier time-out).
__device__ unsigned int g_status_word;

unsigned long long g_wait_ns = 1000000000ull;

constexpr int kMaxDevices = 64;

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return TXL_OK;
    return TXL_ERR_CUDA;
}

// Device address of g_status_word for the current device (looked up once).
unsigned int *status_word(cudaError_t *err)
{
    static std::mutex mu;
    static unsigned int *addr[kMaxDevices] = {};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_status_word);
        if (*err != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D bf16 view [outer][rows][64] with a 64 x box_rows box and 128-byte
// swizzle; planes plane_elems elements apart (rows * 64 when dense).
bool make_map(CUtensorMap *map, const void *base, long long rows, long long outer,
              unsigned box_rows = 128, long long plane_elems = 0)
{
    auto fn = encode_fn();
    if (!fn) return false;
    if (plane_elems == 0) plane_elems = rows * 64;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)outer};
    const cuuint64_t strides[2] = {64 * 2, (cuuint64_t)plane_elems * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count()
{
    static int n[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    if (!n[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 152;  // GB300
        n[dev] = v;
    }
    return n[dev];
}

size_t workspace_bytes_for(int B, int H, int L, int dh, int n_splits)
{
    if (n_splits <= 1) return 0;
    const size_t rows = (size_t)B * H * L;
    size_t o = (size_t)n_splits * rows * dh * sizeof(float);
    o = (o + 255) & ~(size_t)255;
    return o + (size_t)n_splits * rows * sizeof(float);
}

// Key-range splits when the caller lets the library choose.  One block per SM
// at a time, so a launch of units * s blocks runs in ceil(units * s / SMs)
// waves, each as long as one block's ceil(tiles / s) key tiles plus its fixed
// start and finish (about 1.5 tiles: the first copies from HBM, the first
// biases and scores, the epilogue); splitting also writes partials and adds
// the merge kernel (about one tile).  The s with the least estimated time wins
// (B=8 H=16 L=128 M=3800, 128 blocks on 152 SMs: 55.5 us unsplit against
// 69.7 us with 2 splits), keeping >= 4 key tiles per split.
double tc_wave_cost(long long units, int n_key_tiles, int s)
{
    const int sms = sm_count();
    const long long waves = (units * s + sms - 1) / sms;
    return (double)waves * ((n_key_tiles + s - 1) / s + 1.5) + (s > 1 ? 1.0 : 0.0);
}

int auto_splits(int units, int n_key_tiles)
{
    const int sms = sm_count();
    if (units >= sms) return 1;
    const int max_s = std::max(1, n_key_tiles / 4);
    int best = 1;
    double best_cost = 0.0;
    for (int s = 1; s <= max_s; ++s) {
        const double cost = tc_wave_cost(units, n_key_tiles, s);
        if (s == 1 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

// Key splits of the tensor-core kernel for one call: the caller's n_splits,
// or the automatic choice when that is 0, limited to 1 when there is no usable
// workspace (have_ws: non-NULL and 256-byte aligned) big enough for the
// partial results.
int tc_splits(int B, int H, int L, int dh, int n_qtiles, int n_key_tiles, int n_splits,
              bool have_ws, size_t workspace_bytes)
{
    int splits = n_splits;
    if (splits == 0) {
        const long long units = std::min<long long>((long long)B * H * n_qtiles, 1 << 30);
        splits = auto_splits((int)units, n_key_tiles);
        if (splits > 1 && (!have_ws || workspace_bytes < workspace_bytes_for(B, H, L, dh, splits)))
            splits = 1;
    }
    if (splits > n_key_tiles) splits = n_key_tiles;
    return splits;
}

// Which decode kernel a segment of L queries runs: the CUDA-core one for
// L <= kDecodeFmaMaxL (one query), the warp-MMA one above.  One query is the
// CUDA-core kernel's best case (eight sequences of 16 heads against M = 3800:
// 22.2 against 23.5 us); from two on the warp-MMA kernel is faster (24.3
// against 23.6 us) and its time hardly grows with L (23.6 to 24.8 us for
// L = 2..7, where the CUDA-core kernel went to 44.9 us at L = 6).
bool decode_on_mma(int L) { return L > txl::kDecodeFmaMaxL; }

int decode_blocks(int L)
{
    return decode_on_mma(L) ? txl::decode_mma_blocks_per_sm(L) : txl::decode_blocks_per_sm(L);
}

// Key ranges per (b, h) of the decode kernel: the caller's n_splits or the
// automatic choice, capped at one per 128 keys, without ranges that own no key.
int decode_splits(long long BH, long long K, int L, int n_splits)
{
    // At most one split per 128 keys (four 32-key chunks), and only splits that
    // own keys.
    const int max_splits = (int)((K + 127) / 128);
    int splits = n_splits;
    if (splits == 0) {
        // One wave of resident blocks: each block streams its key range
        // through its warps' copy rings, so long ranges amortise the first
        // copies' latency, and a second, partly filled wave would cost a full
        // block time.  At most a cluster's worth of ranges: merging in the
        // cluster beat more ranges merged through the workspace even where
        // those would fill more SMs (one sequence of 16 heads, M = 3800: 8.4 us
        // with 8 ranges, 9.0 us with 19).
        const long long slots = (long long)sm_count() * decode_blocks(L);
        splits = (int)std::max<long long>(
            1, std::min<long long>(std::min<long long>(slots / BH, max_splits),
                                   txl::kDecodeMaxCluster));
    }
    if (splits > max_splits) splits = max_splits;
    // Drop splits that would own no keys once ranges are rounded to chunks.
    while (splits > 1 && (long long)(splits - 1) * txl::decode_span((int)K, splits) >= K) --splits;
    return splits;
}

// Which bf16 kernel a call runs: the decode kernel for every segment of at
// most kDecodeMaxL queries.  Forced both ways on 48 shapes (H = 16, B = 1, 2,
// 4, L = 2, 4, 6, 8, M = 800 to 12000, graph-replayed), the decode kernel was
// the faster one on all of them, by 1.19x (one sequence, M = 8000, L = 8:
// 14.7 against 17.5 us) to 2.2x; with eight sequences against M = 3800 it
// takes 24 us for any L from 2 to 7, the tensor-core kernel 44 us (that kernel
// multiplies whole 128-row query tiles, 16x the rows of an eight-query segment).
bool use_decode(int L) { return L <= txl::kDecodeMaxL; }

// Short segments (L <= kDecodeMaxL): split-K decode kernel, on the tensor
// cores (warp MMAs) or the CUDA cores.
// Up to kDecodeMaxCluster key ranges of a head merge inside their thread-block
// cluster; more go through the workspace and the log-sum-exp merge kernel.
int relattn_decode(const void *q, const void *k, const void *v, long long kv_stride,
                   const void *r, int r_rows, const void *u, const void *v_bias, void *out,
                   float *lse, int B, int H, int M, int L, float scale, int n_splits,
                   void *workspace, size_t workspace_bytes, cudaStream_t s)
{
    const long long K = (long long)M + L;
    const long long BH = (long long)B * H;
    // Up to kDecodeMaxCluster key ranges of a head run as one thread-block
    // cluster and merge in distributed shared memory; more need the workspace
    // for their partial results and a merge kernel.
    const int splits = decode_splits(BH, K, L, n_splits);
    const bool cluster = splits >= 2 && splits <= txl::kDecodeMaxCluster;
    if (splits > 1 && !cluster) {
        if (!workspace || workspace_bytes < workspace_bytes_for(B, H, L, 64, splits))
            return TXL_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return TXL_ERR_MISALIGNED;
    }
    if (BH * splits > 0x7fffffffLL) return TXL_ERR_UNSUPPORTED;

    cudaError_t serr = cudaSuccess;
    unsigned int *status = status_word(&serr);
    if (!status) return TXL_ERR_CUDA;

    txl::DecodeParams p{};
    p.status = status;
    p.wait_ns = g_wait_ns;
    p.B = B;
    p.H = H;
    p.M = M;
    p.L = L;
    p.K = (int)K;
    p.r_rows = r_rows;
    p.r_off = r_rows - (int)K;
    p.n_splits = splits;
    p.kv_stride = kv_stride;
    p.cluster = cluster ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.r = static_cast<const __nv_bfloat16 *>(r);
    p.u = static_cast<const __nv_bfloat16 *>(u);
    p.vb = static_cast<const __nv_bfloat16 *>(v_bias);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    if (splits > 1 && !cluster) {
        const size_t rows = (size_t)BH * L;
        size_t off = (size_t)splits * rows * 64 * sizeof(float);
        off = (off + 255) & ~(size_t)255;
        p.part_o = static_cast<float *>(workspace);
        p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + off);
        p.lse = nullptr;
    }
    cudaError_t err;
    if (decode_on_mma(L)) {
        CUtensorMap tk, tv, tr;
        if (!make_map(&tk, k, K, BH, txl::kDecodeMmaKeyBox, kv_stride) ||
            !make_map(&tv, v, K, BH, txl::kDecodeMmaKeyBox, kv_stride) ||
            !make_map(&tr, r, r_rows, H, txl::kDecodeMmaTableBox))
            return TXL_ERR_CUDA;
        err = txl::launch_relattn_decode_mma(tk, tv, tr, p, s);
    } else {
        err = txl::launch_relattn_decode(p, s);
    }
    if (err != cudaSuccess) return TXL_ERR_CUDA;
    if (splits > 1 && !cluster) {
        err = txl::launch_relattn_combine(p.part_o, p.part_lse, p.out, lse, splits,
                                          (int)(BH * L), s);
        if (err != cudaSuccess) return TXL_ERR_CUDA;
    }
    return TXL_OK;
}

} // namespace

extern "C" {

const char *txl_status_string(int status)
{
    switch (status) {
    case TXL_OK: return "ok";
    case TXL_ERR_INVALID_ARG: return "invalid argument";
    case TXL_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TXL_ERR_MISALIGNED: return "misaligned pointer";
    case TXL_ERR_SHAPE: return "inconsistent sizes";
    case TXL_ERR_CUDA: return "CUDA error";
    case TXL_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case TXL_ERR_WORKSPACE: return "workspace missing or too small";
    case TXL_ERR_INDEX: return "a device-side index check failed";
    default: return "unknown status";
    }
}

int txl_version(void) { return 100; }

uint64_t txl_set_wait_limit_ns(uint64_t ns)
{
    const uint64_t old = g_wait_ns;
    g_wait_ns = ns;
    return old;
}

int txl_rel_pos_emb(void *R, int K, int d_model, int dtype, void *stream)
{
    if (!R || K < 1 || d_model < 2 || (d_model & 1)) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (!aligned(R, dtype == TXL_F32 ? 8 : 4)) return TXL_ERR_MISALIGNED;
    if (K >= (1 << 24) || d_model > 12288) return TXL_ERR_UNSUPPORTED;
    return cuda_status(txl::launch_rel_pos_emb(R, K, d_model, dtype == TXL_BF16, as_stream(stream)));
}

size_t txl_relattn_workspace_size(int B, int H, int L, int dh, int n_splits)
{
    if (B < 1 || H < 1 || L < 1 || dh < 1) return 0;
    return workspace_bytes_for(B, H, L, dh, n_splits);
}

int txl_relattn_plan(int B, int H, int M, int L, int r_rows, int dh, int dtype, int n_splits,
                     size_t workspace_bytes, int *kernel, int *splits)
{
    if (!kernel || !splits) return TXL_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || M < 0 || L < 1 || dh < 1 || n_splits < 0) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    const long long K = (long long)M + L;
    if (K > 0x7fffffffLL / 2 || r_rows < K) return TXL_ERR_SHAPE;
    if (dh != 64) return TXL_ERR_UNSUPPORTED;
    if (dtype == TXL_F32) {
        if (n_splits > 1) return TXL_ERR_UNSUPPORTED;
        *kernel = TXL_KERNEL_F32;
        *splits = 1;
        return TXL_OK;
    }
    const long long BH = (long long)B * H;
    if (BH * L > 0x7fffffffLL || BH > 0x7fffffffLL / 64) return TXL_ERR_UNSUPPORTED;
    const bool have_ws = workspace_bytes > 0;
    int n = 1;
    if (use_decode(L)) {
        n = decode_splits(BH, K, L, n_splits);
        if (n > txl::kDecodeMaxCluster && workspace_bytes < workspace_bytes_for(B, H, L, 64, n))
            return TXL_ERR_WORKSPACE;
        if (BH * n > 0x7fffffffLL) return TXL_ERR_UNSUPPORTED;
        *kernel = decode_on_mma(L) ? TXL_KERNEL_DECODE_MMA : TXL_KERNEL_DECODE;
    } else {
        const int n_qtiles = (L + txl::kTcBM - 1) / txl::kTcBM;
        const int jmax_all = (int)std::min<long long>(K - 1, (long long)M + L - 1);
        const int n_key_tiles = jmax_all / txl::kTcBN + 1;
        n = tc_splits(B, H, L, dh, n_qtiles, n_key_tiles, n_splits, have_ws, workspace_bytes);
        if (n > 1 && workspace_bytes < workspace_bytes_for(B, H, L, dh, n)) return TXL_ERR_WORKSPACE;
        if (BH * n_qtiles * n > 0x7fffffffLL) return TXL_ERR_UNSUPPORTED;
        *kernel = TXL_KERNEL_TC;
    }
    *splits = n;
    return TXL_OK;
}

} // extern "C"

namespace {

// txl_relattn_fwd with k and v planes kv_stride elements apart (0: dense).
int relattn_impl(const void *q, const void *k, const void *v, long long kv_stride,
                 const void *r, int r_rows, const void *u, const void *v_bias, void *out,
                 float *lse, int B, int H, int M, int L, int dh, float scale, int dtype,
                 int n_splits, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!q || !k || !v || !r || !u || !v_bias || !out) return TXL_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || M < 0 || L < 1 || dh < 1 || n_splits < 0) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (!(scale == scale)) return TXL_ERR_INVALID_ARG;  // NaN
    const long long K = (long long)M + L;
    if (K > 0x7fffffffLL / 2 || r_rows < K) return TXL_ERR_SHAPE;
    if (dh != 64) return TXL_ERR_UNSUPPORTED;
    if (kv_stride == 0) kv_stride = K * dh;
    if (kv_stride < K * dh) return TXL_ERR_SHAPE;
    if (kv_stride % 8 != 0) return TXL_ERR_MISALIGNED;
    cudaStream_t s = as_stream(stream);

    if (dtype == TXL_F32) {
        for (const void *p : {q, k, v, r, u, v_bias, (const void *)out})
            if (!aligned(p, 4)) return TXL_ERR_MISALIGNED;
        if (lse && !aligned(lse, 4)) return TXL_ERR_MISALIGNED;
        if (n_splits > 1) return TXL_ERR_UNSUPPORTED;
        txl::F32Params p{};
        p.q = static_cast<const float *>(q);
        p.k = static_cast<const float *>(k);
        p.v = static_cast<const float *>(v);
        p.r = static_cast<const float *>(r);
        p.u = static_cast<const float *>(u);
        p.vb = static_cast<const float *>(v_bias);
        p.out = static_cast<float *>(out);
        p.lse = lse;
        p.B = B;
        p.H = H;
        p.M = M;
        p.L = L;
        p.K = (int)K;
        p.r_rows = r_rows;
        p.kv_stride = kv_stride;
        p.scale = scale;
        return cuda_status(txl::launch_relattn_f32(p, s));
    }

    // bf16 tensor-core path
    for (const void *p : {q, k, v, r, u, v_bias, (const void *)out})
        if (!aligned(p, 16)) return TXL_ERR_MISALIGNED;
    if (lse && !aligned(lse, 4)) return TXL_ERR_MISALIGNED;
    const long long BH = (long long)B * H;
    if (BH * L > 0x7fffffffLL || BH > 0x7fffffffLL / 64) return TXL_ERR_UNSUPPORTED;
    const bool have_ws = workspace && aligned(workspace, 256);
    if (use_decode(L))
        return relattn_decode(q, k, v, kv_stride, r, r_rows, u, v_bias, out, lse, B, H, M, L,
                              scale, n_splits, workspace, workspace_bytes, s);
    const int n_qtiles = (L + txl::kTcBM - 1) / txl::kTcBM;
    const int jmax_all = (int)std::min<long long>(K - 1, (long long)M + L - 1);
    const int n_key_tiles = jmax_all / txl::kTcBN + 1;
    const int splits =
        tc_splits(B, H, L, dh, n_qtiles, n_key_tiles, n_splits, have_ws, workspace_bytes);
    if (splits > 1) {
        if (!workspace || workspace_bytes < workspace_bytes_for(B, H, L, dh, splits))
            return TXL_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return TXL_ERR_MISALIGNED;
    }
    if (BH * n_qtiles * splits > 0x7fffffffLL) return TXL_ERR_UNSUPPORTED;

    CUtensorMap tq, tk, tv, tr;
    if (!make_map(&tq, q, L, BH) || !make_map(&tk, k, K, BH, 128, kv_stride) ||
        !make_map(&tv, v, K, BH, 128, kv_stride) || !make_map(&tr, r, r_rows, H))
        return TXL_ERR_CUDA;

    cudaError_t err;
    unsigned int *status = status_word(&err);
    if (!status) return TXL_ERR_CUDA;

    txl::TcParams p{};
    p.B = B;
    p.H = H;
    p.M = M;
    p.L = L;
    p.K = (int)K;
    p.r_off = r_rows - (int)K;
    p.n_qtiles = n_qtiles;
    p.n_splits = splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.u = static_cast<const __nv_bfloat16 *>(u);
    p.vb = static_cast<const __nv_bfloat16 *>(v_bias);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.status = status;
    p.wait_ns = g_wait_ns;
    if (splits > 1) {
        const size_t rows = (size_t)BH * L;
        size_t off = (size_t)splits * rows * dh * sizeof(float);
        off = (off + 255) & ~(size_t)255;
        p.part_o = static_cast<float *>(workspace);
        p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + off);
        p.lse = nullptr;
    }
    err = txl::launch_relattn_tc(tq, tk, tv, tr, p, s);
    if (err != cudaSuccess) return TXL_ERR_CUDA;
    if (splits > 1) {
        err = txl::launch_relattn_combine(p.part_o, p.part_lse, p.out, lse, splits,
                                          (int)(BH * L), s);
        if (err != cudaSuccess) return TXL_ERR_CUDA;
    }
    return TXL_OK;
}

bool window_ok(const txl_kv_window *w)
{
    return w && w->M >= 0 && w->fill >= 0 && w->fill <= w->M && w->start >= 0 &&
           w->capacity >= 0 && (long long)w->start + w->fill <= w->capacity;
}

// 2-D bf16 view [rows][inner] (as 3-D with one plane) read in boxes of
// 64 columns x box_rows rows with 128-byte swizzle.
bool make_map_rows(CUtensorMap *map, const void *base, long long inner, long long rows,
                   unsigned box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)(inner * rows * 2)};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool mem_state_ok(const txl_mem_state *st)
{
    return st && st->capacity >= 0 && st->fill >= 0 && st->fill <= st->capacity && st->head >= 0 &&
           (st->capacity == 0 ? st->head == 0 : st->head < st->capacity);
}

} // namespace

extern "C" {

int txl_relattn_fwd(const void *q, const void *k, const void *v, const void *r, int r_rows,
                    const void *u, const void *v_bias, void *out, float *lse, int B, int H,
                    int M, int L, int dh, float scale, int dtype, int n_splits,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    return relattn_impl(q, k, v, 0, r, r_rows, u, v_bias, out, lse, B, H, M, L, dh, scale, dtype,
                        n_splits, workspace, workspace_bytes, stream);
}

int txl_relattn_fwd_strided(const void *q, const void *k, const void *v, long long kv_stride,
                            const void *r, int r_rows, const void *u, const void *v_bias,
                            void *out, float *lse, int B, int H, int M, int L, int dh,
                            float scale, int dtype, int n_splits, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    if (kv_stride < 1) return TXL_ERR_INVALID_ARG;
    return relattn_impl(q, k, v, kv_stride, r, r_rows, u, v_bias, out, lse, B, H, M, L, dh,
                        scale, dtype, n_splits, workspace, workspace_bytes, stream);
}

int txl_kv_window_append(void *buf, txl_kv_window *w, const void *seg, int planes, int L, int d,
                         int dtype, void *stream)
{
    if (!window_ok(w) || planes < 1 || L < 0 || d < 1) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if ((long long)w->capacity < 2LL * w->M + L) return TXL_ERR_SHAPE;
    if (L == 0) return TXL_OK;
    if (!buf || !seg) return TXL_ERR_INVALID_ARG;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (((size_t)d * esz) % 16 != 0) return TXL_ERR_MISALIGNED;
    if (!aligned(buf, 16) || !aligned(seg, 16)) return TXL_ERR_MISALIGNED;
    const int row_vec = (int)((size_t)d * esz / 16);
    const long long plane = (long long)w->capacity * row_vec;
    cudaStream_t s = as_stream(stream);
    cudaError_t serr;
    unsigned int *status = status_word(&serr);
    if (!status) return TXL_ERR_CUDA;
    int start = w->start;
    if ((long long)start + w->fill + L > w->capacity) {
        // Move the memory rows to the buffer's front.  With capacity >= 2M + L the
        // window starts at row >= M >= fill here, so the two ranges are disjoint.
        if (w->fill > 0) {
            cudaError_t e = txl::launch_rows_copy(static_cast<uint4 *>(buf), plane, 0,
                                                  static_cast<const uint4 *>(buf), plane, start,
                                                  planes, w->fill, row_vec, status, s);
            if (e != cudaSuccess) return TXL_ERR_CUDA;
        }
        start = 0;
    }
    cudaError_t e = txl::launch_rows_copy(static_cast<uint4 *>(buf), plane, start + w->fill,
                                          static_cast<const uint4 *>(seg), (long long)L * row_vec,
                                          0, planes, L, row_vec, status, s);
    if (e != cudaSuccess) return TXL_ERR_CUDA;
    w->start = start;
    return TXL_OK;
}

int txl_qkv_project(const void *h, const void *w, int B, int L, int d_model, int H, int dh,
                    void *q, void *kv_buf, txl_kv_window *kv_win, void *mem,
                    txl_mem_state *mem_st, void *stream)
{
    if (!h || !w || !kv_buf || !window_ok(kv_win)) return TXL_ERR_INVALID_ARG;
    if (B < 1 || L < 0 || d_model < 1 || H < 1 || dh < 1) return TXL_ERR_INVALID_ARG;
    if (mem && !mem_state_ok(mem_st)) return TXL_ERR_INVALID_ARG;
    if (dh != 64) return TXL_ERR_UNSUPPORTED;
    if ((long long)kv_win->capacity < 2LL * kv_win->M + L) return TXL_ERR_SHAPE;
    if (d_model % 8 != 0) return TXL_ERR_MISALIGNED;
    for (const void *p : {h, w, (const void *)kv_buf})
        if (!aligned(p, 16)) return TXL_ERR_MISALIGNED;
    if ((q && !aligned(q, 16)) || (mem && !aligned(mem, 16))) return TXL_ERR_MISALIGNED;
    const long long M = (long long)B * L;
    const int n_out = q ? 3 : 2;
    const long long N = (long long)n_out * H * 64;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || (long long)B * H * 2 > 0x7fffffffLL)
        return TXL_ERR_UNSUPPORTED;
    if (L == 0) return TXL_OK;
    cudaStream_t s = as_stream(stream);
    cudaError_t serr;
    unsigned int *status = status_word(&serr);
    if (!status) return TXL_ERR_CUDA;

    const long long C = kv_win->capacity;
    const int row_vec = 64 * 2 / 16;
    int start = kv_win->start;
    if ((long long)start + kv_win->fill + L > C) {
        // move the memory rows of every key and value plane to the front, as
        // txl_kv_window_append does (disjoint ranges since C >= 2M + L)
        if (kv_win->fill > 0) {
            cudaError_t e = txl::launch_rows_copy(static_cast<uint4 *>(kv_buf), C * row_vec, 0,
                                                  static_cast<const uint4 *>(kv_buf), C * row_vec,
                                                  start, 2 * B * H, kv_win->fill, row_vec, status, s);
            if (e != cudaSuccess) return TXL_ERR_CUDA;
        }
        start = 0;
    }

    txl::ProjParams p{};
    p.M = (int)M;
    p.N = (int)N;
    p.K = d_model;
    p.L = L;
    p.B = B;
    p.H = H;
    p.n_out = n_out;
    p.h = static_cast<const __nv_bfloat16 *>(h);
    auto *kv = static_cast<__nv_bfloat16 *>(kv_buf);
    int o = 0;
    if (q) {
        p.out[o] = static_cast<__nv_bfloat16 *>(q);
        p.plane_stride[o] = (long long)L * 64;
        p.row0[o] = 0;
        ++o;
    }
    for (int kv_i = 0; kv_i < 2; ++kv_i, ++o) {
        p.out[o] = kv + (size_t)kv_i * B * H * C * 64;
        p.plane_stride[o] = C * 64;
        p.row0[o] = start + kv_win->fill;
    }
    int new_head = 0, new_fill = 0;
    if (mem && mem_st->capacity > 0) {
        const int cap = mem_st->capacity;
        p.mem = static_cast<__nv_bfloat16 *>(mem);
        p.mem_cap = cap;
        p.mem_head = mem_st->head;
        p.mem_first = L > cap ? L - cap : 0;  // older rows would be overwritten anyway
        new_head = (int)(((long long)mem_st->head + L) % cap);
        new_fill = (int)std::min<long long>((long long)mem_st->fill + L, cap);
    }
    p.status = status;
    p.wait_ns = g_wait_ns;

    CUtensorMap tm_h, tm_w;
    if (!make_map_rows(&tm_h, h, d_model, M, 128) || !make_map_rows(&tm_w, w, d_model, N, 256))
        return TXL_ERR_CUDA;
    if (txl::launch_project(tm_h, tm_w, p, s) != cudaSuccess) return TXL_ERR_CUDA;
    kv_win->start = start;
    if (p.mem) {
        mem_st->head = new_head;
        mem_st->fill = new_fill;
    }
    return TXL_OK;
}

int txl_kv_window_advance(txl_kv_window *w, int L)
{
    if (!window_ok(w) || L < 0) return TXL_ERR_INVALID_ARG;
    const long long total = (long long)w->fill + L;
    if ((long long)w->start + total > w->capacity) return TXL_ERR_SHAPE;
    const int keep = (int)std::min<long long>(total, w->M);
    w->start = (int)(w->start + total - keep);
    w->fill = keep;
    return TXL_OK;
}

int txl_mem_concat(void *ext, const void *mem, const txl_mem_state *st, const void *h_new,
                   int B, int L, int d, int dtype, void *stream)
{
    if (!st || B < 1 || L < 0 || d < 1) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (st->capacity < 0 || st->fill < 0 || st->fill > st->capacity || st->head < 0 ||
        (st->capacity > 0 && st->head >= st->capacity) || (st->capacity == 0 && st->head != 0))
        return TXL_ERR_SHAPE;
    if (st->fill + L == 0) return TXL_OK;  // empty extended context
    if (!ext || (L > 0 && !h_new) || (st->fill > 0 && !mem)) return TXL_ERR_INVALID_ARG;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (((size_t)d * esz) % 16 != 0) return TXL_ERR_MISALIGNED;
    if (!aligned(ext, 16) || (h_new && !aligned(h_new, 16)) || (mem && !aligned(mem, 16)))
        return TXL_ERR_MISALIGNED;
    const int row_vec = (int)((size_t)d * esz / 16);
    cudaError_t serr;
    unsigned int *status = status_word(&serr);
    if (!status) return TXL_ERR_CUDA;
    return cuda_status(txl::launch_mem_concat(
        static_cast<uint4 *>(ext), static_cast<const uint4 *>(mem),
        static_cast<const uint4 *>(h_new), B, st->fill, st->head, st->capacity, L, row_vec,
        status, as_stream(stream)));
}

int txl_mem_update(void *mem, txl_mem_state *st, const void *h_new, int B, int L, int d,
                   int dtype, void *stream)
{
    if (!st || B < 1 || L < 0 || d < 1) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (st->capacity < 0 || st->fill < 0 || st->fill > st->capacity || st->head < 0 ||
        (st->capacity > 0 && st->head >= st->capacity) || (st->capacity == 0 && st->head != 0))
        return TXL_ERR_SHAPE;
    if (st->capacity == 0 || L == 0) return TXL_OK;  // nothing to keep or nothing new
    if (!mem || !h_new) return TXL_ERR_INVALID_ARG;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (((size_t)d * esz) % 16 != 0) return TXL_ERR_MISALIGNED;
    if (!aligned(mem, 16) || !aligned(h_new, 16)) return TXL_ERR_MISALIGNED;
    const int row_vec = (int)((size_t)d * esz / 16);
    const int cap = st->capacity;
    const int first = L > cap ? L - cap : 0;  // older rows would be overwritten anyway
    cudaError_t serr;
    unsigned int *status = status_word(&serr);
    if (!status) return TXL_ERR_CUDA;
    cudaError_t e = txl::launch_mem_write(static_cast<uint4 *>(mem),
                                          static_cast<const uint4 *>(h_new), B, L, first,
                                          st->head, cap, row_vec, status, as_stream(stream));
    if (e != cudaSuccess) return TXL_ERR_CUDA;
    st->head = (int)(((long long)st->head + L) % cap);
    st->fill = (int)std::min<long long>((long long)st->fill + L, cap);
    return TXL_OK;
}

int txl_device_status(void *stream)
{
    cudaError_t err;
    unsigned int *w = status_word(&err);
    if (!w) return TXL_ERR_CUDA;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TXL_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TXL_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return TXL_ERR_CUDA;
        return (v & TXL_STATUS_TIMEOUT) ? TXL_ERR_TIMEOUT : TXL_ERR_INDEX;
    }
    return TXL_OK;
}

int txl_debug_checks(void)
{
#ifdef TXL_DEBUG
    return 1;
#else
    return 0;
#endif
}

int txl_debug_index_probe(void *stream)
{
    cudaError_t err;
    unsigned int *w = status_word(&err);
    if (!w) return TXL_ERR_CUDA;
    err = txl::launch_index_probe(w, as_stream(stream));
    if (err != cudaSuccess) return TXL_ERR_CUDA;
    return txl_device_status(stream);
}

int txl_debug_wait_timeout(uint64_t ns, void *stream)
{
    cudaError_t err;
    unsigned int *w = status_word(&err);
    if (!w) return TXL_ERR_CUDA;
    if (ns == 0 || ns > 10000000000ull) return TXL_ERR_INVALID_ARG;  // at most 10 s
    err = txl::launch_wait_probe(w, ns, as_stream(stream));
    if (err != cudaSuccess) return TXL_ERR_CUDA;
    return txl_device_status(stream);
}

} // extern "C"

// ---------------------------------------------------------------------------
// Backward of the attention (one segment, §3.2: the memory is SG(m)).
// ---------------------------------------------------------------------------
extern "C" size_t txl_relattn_bwd_workspace_size(int B, int H, int L, int M)
{
    return txl::bwd_workspace_bytes(B, H, L, M);
}

extern "C" int txl_relattn_bwd(const void *q, const void *k, const void *v, const void *r,
                               int r_rows, const void *u, const void *v_bias, const void *dout,
                               float *dq, float *dk, float *dv, float *dr, float *du,
                               float *dv_bias, int B, int H, int M, int L, int dh, float scale,
                               int dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!q || !k || !v || !r || !u || !v_bias || !dout || !dq || !dk || !dv || !dr || !du ||
        !dv_bias)
        return TXL_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || M < 0 || L < 1 || dh < 1) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (!(scale == scale)) return TXL_ERR_INVALID_ARG;  // NaN
    const long long K = (long long)M + L;
    if (K > 0x7fffffffLL / 2 || r_rows < K) return TXL_ERR_SHAPE;
    if (dh != 64 || dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    for (const void *p : {q, k, v, r, u, v_bias, dout, (const void *)dq, (const void *)dk,
                          (const void *)dv, (const void *)dr, (const void *)du,
                          (const void *)dv_bias})
        if (!aligned(p, 16)) return TXL_ERR_MISALIGNED;
    const long long BH = (long long)B * H;
    const long long rows = txl::kBwdRows;
    if (BH > 0x7fffffffLL || (L + rows - 1) / rows > 65535 || (K + rows - 1) / rows > 65535 ||
        H > 65535)
        return TXL_ERR_UNSUPPORTED;
    const size_t need = txl::bwd_workspace_bytes(B, H, L, M);
    if (!workspace || workspace_bytes < need) return TXL_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TXL_ERR_MISALIGNED;

    cudaError_t err;
    unsigned int *status = status_word(&err);
    if (!status) return TXL_ERR_CUDA;
    txl::BwdParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.r = static_cast<const __nv_bfloat16 *>(r);
    p.u = static_cast<const __nv_bfloat16 *>(u);
    p.vb = static_cast<const __nv_bfloat16 *>(v_bias);
    p.dout = static_cast<const __nv_bfloat16 *>(dout);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dr = dr;
    p.du = du;
    p.dvb = dv_bias;
    // workspace: log2-sum-exp and D per row, the bias partials, the dq
    // partials of the key splits, g of every pair (256-byte aligned regions, as
    // txl::bwd_workspace_bytes counts them)
    const size_t row_bytes = ((size_t)BH * L * sizeof(float) + 255) & ~(size_t)255;
    char *ws = static_cast<char *>(workspace);
    p.lse2 = reinterpret_cast<float *>(ws);
    p.dsum = reinterpret_cast<float *>(ws + row_bytes);
    p.part = reinterpret_cast<float *>(ws + 2 * row_bytes);
    p.dq_part = reinterpret_cast<float *>(ws + txl::bwd_dq_part_offset(B, H, L));
    p.g_all = reinterpret_cast<float *>(ws + txl::bwd_g_offset(B, H, L));
    p.Kd = (int)((K + rows - 1) / rows * rows);
    p.B = B;
    p.H = H;
    p.M = M;
    p.L = L;
    p.K = (int)K;
    p.r_rows = r_rows;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = status;
    return cuda_status(txl::launch_relattn_bwd(p, as_stream(stream)));
}
