// Backward of the relative-position attention for one segment
// ("Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context":
// §3.3 score A_ij = (q_i + u).k_j + (q_i + v).W_kR R_{i-j}, masked softmax over
// the extended context, times v; §3.2 training backpropagates within a
// segment, the memory being SG(m)).  Gradients, per head, with A scaled:
//   D_i = sum_j P_ij dP_ij,  dP_ij = dout_i . v_j,  g_ij = scale P_ij (dP_ij - D_i)
//   dq_i = sum_j g_ij (k_j + r_{M+i-j})   dk_j = sum_i g_ij (q_i + u)
//   dv_j = sum_i P_ij dout_i              dr_d = sum_{i-j=d-M} g_ij (q_i + v)
//   du = sum g_ij k_j                     dv_bias = sum g_ij r_{M+i-j}
// (dr, du, dv_bias summed over the batch: the table and biases are shared).
//
// Launches over tiles of 64 query rows x 64 columns (keys, or distances for
// the table gradient), 512 threads = 16 warps, warp w taking rows
// 16 (w / 4) .. +15 and columns 16 (w % 4) .. +15 of every 64 x 64 product
// (and columns 32 (w % 4) .. +31 of a 64 x 128 window product):
//   stats   per 64-row chunk, over its key tiles: online log-sum-exp of the
//           scores and D (nothing from the forward call is needed); for
//           segments of at most two chunks stats2, per (batch row, head, key
//           split) over both chunks, the splits merged in order
//   dqkv    segments of at most two chunks: per (batch row, head, key split),
//           one score pass for dq, dk, dv (dq partials summed over the splits
//           in order by dq_reduce)
//   dq      longer segments: per 64-row chunk, over its key tiles: dq
//   dkv     longer segments: per 64-key tile, over the chunks that see it
//   dr      per head and 64-distance tile, over the batch and query chunks:
//           the table gradient from g, which the dq passes store
//   bias    per head: du, dv_bias from the partials, in a fixed order
// The dq / dk / dv tiles recompute their scores.  All products run on the
// tensor cores as warp-level mma.m16n8k16 (bf16 operands from shared memory by
// ldmatrix, fp32 accumulation), exactly: q, k, v, r and dout are bf16 already,
// the bias terms u.k_j and v.r_d are per-column vectors added in fp32, g and P
// (fp32) enter as a bf16 head plus the bf16 rounding of the rest (~2^-17
// relative), and the rank-one parts of dk and dr (column sums of g times u or
// v) are added in fp32.  The Appendix B shift is index arithmetic, as in the
// forward: the position term of a pair tile is row i of the product q R_w^T
// over the tile's 127-distance window, read at window column i - j + 63; dq's
// position part is a window product of g laid out by the same index, and the
// table gradient reads the stored g along the same diagonals (row i of a
// distance tile starts at key M + i - d0 - 63).  Results repeat bit for bit.
#include <cmath>

#include "kernels.h"

namespace txl {
namespace {

constexpr int DH = 64;
constexpr int T = kBwdRows;     // rows / columns of a pair tile
constexpr int W = 2 * T;        // window rows of a tile (127 used)
constexpr int THREADS = 512;
constexpr int NF = 2;   // 8-column fragments of a warp in a 64 x 64 product
constexpr int NWF = 4;  // in a 64 x 128 window product
constexpr int LDB = (DH + 8) * 2;   // bytes per bf16 row of 64 (+8 pad: conflict-free ldmatrix)
constexpr int LDZ = (W + 8) * 2;    // bytes per bf16 row of 128
constexpr int LDX = W + 8;          // floats per row of the fp32 window product (= 8 mod 32:
                                    // a half warp's paired stores hit distinct banks)

// Shared memory (bytes): bf16 operand tiles, g and P as head / rest pairs, the
// window-ordered g, the fp32 window product, per-column bias vectors and
// reduction scratch.
constexpr int OFF_Q = 0;                    // q rows of the chunk [64][72]
constexpr int OFF_D = OFF_Q + T * LDB;      // dout rows
constexpr int OFF_K = OFF_D + T * LDB;      // key tile
constexpr int OFF_V = OFF_K + T * LDB;      // value tile
constexpr int OFF_W = OFF_V + T * LDB;      // table window [128][72]
constexpr int OFF_W2 = OFF_W + W * LDB;     // the one-pass kernel's window rows 128.. and v.r vector
constexpr int OFF_GH = OFF_W2 + W * LDB;    // g head [64][72], pair (i, column)
constexpr int OFF_GL = OFF_GH + T * LDB;    // g rest
constexpr int OFF_PH = OFF_GL + T * LDB;    // P head
constexpr int OFF_PL = OFF_PH + T * LDB;    // P rest
constexpr int OFF_ZH = OFF_PL + T * LDB;    // g by window column [64][136], head
constexpr int OFF_ZL = OFF_ZH + T * LDZ;    // rest
constexpr int OFF_XS = OFF_ZL + T * LDZ;    // fp32 [64][132] window product
constexpr int OFF_BK = OFF_XS + T * LDX * 4;  // fp32 [64]: u.k_j
constexpr int OFF_BW = OFF_BK + T * 4;        // fp32 [128]: v.r_w of the window
constexpr int OFF_RED = OFF_BW + W * 4;       // fp32 [16][64] reduction scratch
constexpr int OFF_CS = OFF_RED + 16 * T * 4;   // fp32 [64]: column sums of g over the rows
// second key tile, value tile and table window: the row-chunk kernels copy
// the next key tile in while computing on the current one
constexpr int OFF_K1 = OFF_CS + T * 4;
constexpr int OFF_V1 = OFF_K1 + T * LDB;
constexpr int OFF_W1 = OFF_V1 + T * LDB;
constexpr int SMEM_BYTES = OFF_W1 + W * LDB;
static_assert(OFF_XS - OFF_ZH == T * LDX * 4, "the window-ordered g region holds a second window product");
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_W % 16 == 0 && OFF_GH % 16 == 0 && OFF_ZH % 16 == 0 && OFF_XS % 16 == 0 &&
                  OFF_K1 % 16 == 0 && OFF_W1 % 16 == 0,
              "ldmatrix rows must be 16-byte aligned");

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf(uint32_t w, int hi)
{
    return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// (head, rest) bf16 pairs of two fp32 values: x ~ head + rest to ~2^-17.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &head, uint32_t &rest)
{
    head = pack2(x0, x1);
    rest = pack2(x0 - bf(head, 0), x1 - bf(head, 1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NT>
__device__ __forceinline__ void zero(float (&c)[NT][4])
{
#pragma unroll
    for (int n = 0; n < NT; ++n) c[n][0] = c[n][1] = c[n][2] = c[n][3] = 0.f;
}

// One warp: C[16][8 NT] += A[16][kd] B^T with A stored [row][k] (a: address of
// the warp's first row) and B stored [n][k] (b: address of its first column n).
template <int NT>
__device__ __forceinline__ void warp_nt(float (&c)[NT][4], uint32_t a, int lda, uint32_t b,
                                        int ldb, int kd, int lane)
{
#pragma unroll 2
    for (int k0 = 0; k0 < kd; k0 += 16) {
        uint32_t af[4];
        ldsm_x4(af, a + (lane & 15) * lda + (k0 + (lane >> 4) * 8) * 2);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            uint32_t bfr[4];
            ldsm_x4(bfr, b + (np * 16 + (lane >> 4) * 8 + (lane & 7)) * ldb +
                             (k0 + ((lane >> 3) & 1) * 8) * 2);
            mma16816(c[2 * np], af, bfr[0], bfr[1]);
            mma16816(c[2 * np + 1], af, bfr[2], bfr[3]);
        }
    }
}

// One warp: C[16][8 NT] += (Ah + Al)[16][kd] B with B stored [k][n] (b: address
// of row k = 0 at the warp's first column n).  A stored [row][k] (a_trans
// false; ah, al: addresses of the warp's first row) or [k][row] (a_trans: the
// addresses of row k = 0 at the warp's first row index).
template <int NT>
__device__ __forceinline__ void warp_nn2(float (&c)[NT][4], uint32_t ah, uint32_t al, int lda,
                                         bool a_trans, uint32_t b, int ldb, int kd, int lane)
{
#pragma unroll 2
    for (int k0 = 0; k0 < kd; k0 += 16) {
        uint32_t fh[4], fl[4];
        if (a_trans) {
            const uint32_t off = (k0 + (lane >> 4) * 8 + (lane & 7)) * lda + ((lane >> 3) & 1) * 16;
            ldsm_x4_t(fh, ah + off);
            ldsm_x4_t(fl, al + off);
        } else {
            const uint32_t off = (lane & 15) * lda + (k0 + (lane >> 4) * 8) * 2;
            ldsm_x4(fh, ah + off);
            ldsm_x4(fl, al + off);
        }
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            uint32_t bfr[4];
            ldsm_x4_t(bfr, b + (k0 + ((lane >> 3) & 1) * 8 + (lane & 7)) * ldb +
                               (np * 16 + (lane >> 4) * 8) * 2);
            mma16816(c[2 * np], fh, bfr[0], bfr[1]);
            mma16816(c[2 * np + 1], fh, bfr[2], bfr[3]);
            mma16816(c[2 * np], fl, bfr[0], bfr[1]);
            mma16816(c[2 * np + 1], fl, bfr[2], bfr[3]);
        }
    }
}

// Rows w = 0 .. n-1 of a bf16 tile (row stride ld bytes) from rows row0 + step w
// of a [rows_total][64] bf16 matrix; rows outside [0, rows_total) are zeros.
__device__ __forceinline__ void stage(uint8_t *dst, int ld, int n, const __nv_bfloat16 *src,
                                      long long row0, int step, long long rows_total)
{
    for (int idx = threadIdx.x; idx < n * 8; idx += THREADS) {
        const int w = idx >> 3, c = idx & 7;
        const long long sr = row0 + (long long)step * w;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (sr >= 0 && sr < rows_total) x = __ldg(reinterpret_cast<const uint4 *>(src + sr * DH) + c);
        *reinterpret_cast<uint4 *>(dst + w * ld + c * 16) = x;
    }
}

// The same with asynchronous 16-byte copies (rows outside the matrix are
// zero-filled by a zero source size; their source address stays in bounds).
__device__ __forceinline__ void stage_async(uint8_t *dst, int ld, int n, const __nv_bfloat16 *src,
                                            long long row0, int step, long long rows_total)
{
    for (int idx = threadIdx.x; idx < n * 8; idx += THREADS) {
        const int w = idx >> 3, c = idx & 7;
        const long long sr = row0 + (long long)step * w;
        const bool in = sr >= 0 && sr < rows_total;
        const __nv_bfloat16 *g = src + (in ? sr * DH : 0) + c * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + w * ld + c * 16)),
                     "l"(g), "r"(in ? 16 : 0)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// out[w] = vec . row w of a staged bf16 tile (n = 64 or 128 rows), fp32; vec:
// 64 bf16 in global memory.  Four threads per row (n * 4 items and the block
// size are multiples of 32, so each warp runs an iteration with all its lanes
// or skips it whole: the shuffles stay within full warps).
__device__ __forceinline__ void row_dots(float *out, const uint8_t *tile, int ld, int n,
                                         const __nv_bfloat16 *vec)
{
    for (int idx = threadIdx.x; idx < n * 4; idx += THREADS) {
        const int w = idx >> 2, part = idx & 3;
        const uint4 *row = reinterpret_cast<const uint4 *>(tile + w * ld) + part * 2;
        const uint4 *vv = reinterpret_cast<const uint4 *>(vec) + part * 2;
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 x = row[h], y = __ldg(vv + h);
            s = fmaf(bf(x.x, 0), bf(y.x, 0), s); s = fmaf(bf(x.x, 1), bf(y.x, 1), s);
            s = fmaf(bf(x.y, 0), bf(y.y, 0), s); s = fmaf(bf(x.y, 1), bf(y.y, 1), s);
            s = fmaf(bf(x.z, 0), bf(y.z, 0), s); s = fmaf(bf(x.z, 1), bf(y.z, 1), s);
            s = fmaf(bf(x.w, 0), bf(y.w, 0), s); s = fmaf(bf(x.w, 1), bf(y.w, 1), s);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (part == 0) out[w] = s;
    }
}

// The lane's place in a 64 x 64 product: warp w holds rows 16 (w/4) + g and
// + 8, columns 16 (w%4) + 8 n + 2 t and + 1 (n = 0, 1): element q of
// fragment n is row rb + g + 8 (q / 2), column cb + 8 n + 2 t + q % 2.
struct Lane {
    int warp, lane, g, t, rb, cb;
};

__device__ __forceinline__ Lane lane_of()
{
    Lane L;
    L.warp = threadIdx.x >> 5;
    L.lane = threadIdx.x & 31;
    L.g = L.lane >> 2;
    L.t = L.lane & 3;
    L.rb = 16 * (L.warp >> 2);
    L.cb = 16 * (L.warp & 3);
    return L;
}

// The 64 x 128 window product of the warp's rows, plus a per-column vector,
// into an fp32 window buffer (columns 32 (w%4) .. +31).
__device__ __forceinline__ void window_product(uint8_t *sm, const Lane &L, int a_off, int b_off,
                                               const float *colvec, int xs_off = OFF_XS)
{
    float x[NWF][4];
    zero(x);
    warp_nt<NWF>(x, smem_u32(sm + a_off) + L.rb * LDB, LDB,
               smem_u32(sm + b_off) + 32 * (L.warp & 3) * LDB, LDB, DH, L.lane);
    float *xs = reinterpret_cast<float *>(sm + xs_off);
#pragma unroll
    for (int n = 0; n < NWF; ++n)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int col = 32 * (L.warp & 3) + 8 * n + 2 * L.t;
            const float c0 = colvec ? colvec[col] : 0.f, c1 = colvec ? colvec[col + 1] : 0.f;
            *reinterpret_cast<float2 *>(xs + (L.rb + L.g + 8 * hh) * LDX + col) =
                make_float2(x[n][2 * hh] + c0, x[n][2 * hh + 1] + c1);
        }
}

// Where the operands of the current tile sit (byte offsets): q rows, dout
// rows, keys, values, table window.
struct Bufs {
    int q, d, k, v, w;
    int bw = OFF_BW;  // the window's v.r vector (fp32)
};

// The lane's 16 log2-scaled scores (-inf where masked) of the pair tile at
// (i0, j0) from its content part sc, the column vector u.k_j and the window
// product in the buffer at xs_off (complete: after a barrier).
__device__ __forceinline__ void finish_scores(const uint8_t *sm, const BwdParams &p, const Lane &L, int i0,
                                              int j0, const float (&sc)[NF][4], float (&s)[NF][4],
                                              int xs_off)
{
    const float *bk = reinterpret_cast<const float *>(sm + OFF_BK);
    const float *xs = reinterpret_cast<const float *>(sm + xs_off);
    float b[NF][2];
#pragma unroll
    for (int n = 0; n < NF; ++n) {
        const float2 x = *reinterpret_cast<const float2 *>(bk + L.cb + 8 * n + 2 * L.t);
        b[n][0] = x.x;
        b[n][1] = x.y;
    }
    // every pair of the tile kept: rows and keys in range, the last key of
    // the tile visible from its first row (block-uniform)
    const bool interior = i0 + T <= p.L && j0 + T <= p.K && j0 + T - 1 <= p.M + i0;
#pragma unroll
    for (int n = 0; n < NF; ++n)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = L.rb + L.g + 8 * (q >> 1), j = L.cb + 8 * n + 2 * L.t + (q & 1);
            // Appendix B: distance M + i0 + i - (j0 + j) is window column i - j + 63
            const float v = (sc[n][q] + b[n][q & 1] + xs[i * LDX + i - j + T - 1]) * p.scale_log2;
            if (interior) {
                s[n][q] = v;
            } else {
                const int gi = i0 + i, gj = j0 + j;
                s[n][q] = (gi < p.L && gj < p.K && gj <= p.M + gi) ? v : -INFINITY;
            }
        }
}

// Log2-scaled scores (-inf where masked) and dP = dout . v of the lane's 16
// pairs of the key tile at j0, from the staged q, dout, keys, values, table
// window (distances M + i0 - j0 - 63 + w) and bias vectors (u.k_j, v.r_w).
// Contains a block barrier.
__device__ __forceinline__ void key_tile_scores(uint8_t *sm, const BwdParams &p, const Lane &L,
                                                int i0, int j0, float (&s)[NF][4], float (&dp)[NF][4],
                                                const Bufs &B)
{
    float sc[NF][4];
    zero(sc);
    zero(dp);
    warp_nt<NF>(sc, smem_u32(sm + B.q) + L.rb * LDB, LDB, smem_u32(sm + B.k) + L.cb * LDB, LDB,
               DH, L.lane);
    warp_nt<NF>(dp, smem_u32(sm + B.d) + L.rb * LDB, LDB, smem_u32(sm + B.v) + L.cb * LDB, LDB,
               DH, L.lane);
    window_product(sm, L, B.q, B.w, reinterpret_cast<const float *>(sm + B.bw));
    __syncthreads();
    finish_scores(sm, p, L, i0, j0, sc, s, OFF_XS);
}

__device__ __forceinline__ void stage_rows(uint8_t *sm, const BwdParams &p, long long bh, int i0)
{
    stage(sm + OFF_Q, LDB, T, p.q + bh * p.L * DH, i0, 1, p.L);
    stage(sm + OFF_D, LDB, T, p.dout + bh * p.L * DH, i0, 1, p.L);
}

// The row-chunk kernels' key tiles, double-buffered: copies of tile j0 (keys,
// values, table window of distances M + i0 - j0 - 63 + w) into buffer `buf`
// go out asynchronously; key_tile_ready waits for the older group, then
// forms u.k_j and v.r_w of that buffer.
__device__ __forceinline__ void issue_key_tile(uint8_t *sm, const BwdParams &p, long long bh, int h,
                                               int i0, int j0, int buf)
{
    stage_async(sm + (buf ? OFF_K1 : OFF_K), LDB, T, p.k + bh * p.K * DH, j0, 1, p.K);
    stage_async(sm + (buf ? OFF_V1 : OFF_V), LDB, T, p.v + bh * p.K * DH, j0, 1, p.K);
    const long long dmin = (long long)p.M + i0 - j0 - (T - 1);
    stage_async(sm + (buf ? OFF_W1 : OFF_W), LDB, W, p.r + (size_t)h * p.r_rows * DH,
                p.r_rows - 1 - dmin, -1, p.r_rows);
}

// `more`: another tile's copies were issued after this one's (3 groups each).
__device__ __forceinline__ void key_tile_ready(uint8_t *sm, const BwdParams &p, int h, int buf, bool more)
{
    if (more) async_wait<3>();
    else async_wait<0>();
    __syncthreads();
    row_dots(reinterpret_cast<float *>(sm + OFF_BK), sm + (buf ? OFF_K1 : OFF_K), LDB, T,
             p.u + (size_t)h * DH);
    row_dots(reinterpret_cast<float *>(sm + OFF_BW), sm + (buf ? OFF_W1 : OFF_W), LDB, W,
             p.vb + (size_t)h * DH);
    __syncthreads();
}

// The key-tile kernel's row chunks, double-buffered the same way: q and dout
// rows and the table window of chunk i0 into buffer `buf` (buffer 1 uses the
// second key / value regions, which that kernel does not need).
__device__ __forceinline__ Bufs chunk_bufs(int buf)
{
    return Bufs{buf ? OFF_K1 : OFF_Q, buf ? OFF_V1 : OFF_D, OFF_K, OFF_V, buf ? OFF_W1 : OFF_W};
}

__device__ __forceinline__ void issue_chunk(uint8_t *sm, const BwdParams &p, long long bh, int h,
                                            int i0, int j0, int buf)
{
    const Bufs B = chunk_bufs(buf);
    stage_async(sm + B.q, LDB, T, p.q + bh * p.L * DH, i0, 1, p.L);
    stage_async(sm + B.d, LDB, T, p.dout + bh * p.L * DH, i0, 1, p.L);
    const long long dmin = (long long)p.M + i0 - j0 - (T - 1);
    stage_async(sm + B.w, LDB, W, p.r + (size_t)h * p.r_rows * DH, p.r_rows - 1 - dmin, -1, p.r_rows);
}

// Row statistics of the lane's two rows (rb + g, rb + g + 8).
__device__ __forceinline__ void load_row_stats(const BwdParams &p, const Lane &L, long long bh,
                                               int i0, float (&ls)[2], float (&dd)[2])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int gi = i0 + L.rb + L.g + 8 * h;
        ls[h] = gi < p.L ? p.lse2[bh * p.L + gi] : 0.f;
        dd[h] = gi < p.L ? p.dsum[bh * p.L + gi] : 0.f;
    }
}

// g = scale P (dP - D) with P = 2^(s - lse2) (0 where masked); g and P as
// head / rest pairs into the [row][column] tiles (P only with with_p), and g
// also by window column i - j + 63 (with_z: the dq kernel's shifted operand).
__device__ __forceinline__ void grad_scores(uint8_t *sm, const BwdParams &p, const Lane &L,
                                            const float (&s)[NF][4], const float (&dp)[NF][4],
                                            const float (&ls)[2], const float (&dd)[2],
                                            float (&g)[NF][4], bool with_p, bool with_z = false)
{
#pragma unroll
    for (int n = 0; n < NF; ++n)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float P[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = 2 * hh + e;
                P[e] = exp2f(s[n][q] - ls[hh]);  // 0 where masked (ls is finite)
                g[n][q] = p.scale * P[e] * (dp[n][q] - dd[hh]);
            }
            const int off = (L.rb + L.g + 8 * hh) * LDB + (L.cb + 8 * n + 2 * L.t) * 2;
            uint32_t hd, rs;
            split2(g[n][2 * hh], g[n][2 * hh + 1], hd, rs);
            *reinterpret_cast<uint32_t *>(sm + OFF_GH + off) = hd;
            *reinterpret_cast<uint32_t *>(sm + OFF_GL + off) = rs;
            if (with_z) {
                // columns j, j + 1 of row i land at window columns w, w - 1
                const int i = L.rb + L.g + 8 * hh, j = L.cb + 8 * n + 2 * L.t, w = i - j + T - 1;
                uint16_t *zh = reinterpret_cast<uint16_t *>(sm + OFF_ZH) + i * (LDZ / 2) + w;
                uint16_t *zl = reinterpret_cast<uint16_t *>(sm + OFF_ZL) + i * (LDZ / 2) + w;
                zh[0] = (uint16_t)(hd & 0xffffu);
                zh[-1] = (uint16_t)(hd >> 16);
                zl[0] = (uint16_t)(rs & 0xffffu);
                zl[-1] = (uint16_t)(rs >> 16);
            }
            if (with_p) {
                split2(P[0], P[1], hd, rs);
                *reinterpret_cast<uint32_t *>(sm + OFF_PH + off) = hd;
                *reinterpret_cast<uint32_t *>(sm + OFF_PL + off) = rs;
            }
        }
}

// g of the lane's 16 pairs for the table gradient, blocked by key tile:
// g_all[bh][j / 64][i][j % 64] (fp32; a tile's rows are contiguous, 256 bytes
// each).  Pairs of a visited tile are written, masked ones as zeros; entries of
// tiles no pass visits stay unset and are never read.
__device__ __forceinline__ void store_g(const BwdParams &p, const Lane &L, long long bh, int i0, int j0,
                                        const float (&g)[NF][4])
{
    float *blk = p.g_all + (((size_t)bh * (p.Kd / T) + j0 / T) * p.L) * T;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int gi = i0 + L.rb + L.g + 8 * hh;
        if (gi >= p.L) continue;
#pragma unroll
        for (int n = 0; n < NF; ++n) {
            // an even column below K: the pair's second column is below Kd
            const int j = L.cb + 8 * n + 2 * L.t;
            if (j0 + j < p.K)
                *reinterpret_cast<float2 *>(blk + (size_t)gi * T + j) = make_float2(g[n][2 * hh], g[n][2 * hh + 1]);
        }
    }
}

// Column sums over the lane's rows of a fragment set, reduced over the warp's
// 16 rows; lanes with g == 0 store them at red[strip][column].
__device__ __forceinline__ void column_sums(float *red, int stride, const Lane &L, int col0,
                                            const float (&c)[NF][4])
{
#pragma unroll
    for (int n = 0; n < NF; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v = c[n][e] + c[n][2 + e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (L.g == 0) red[(L.warp >> 2) * stride + col0 + 8 * n + 2 * L.t + e] = v;
        }
}

// The online state of the lane's two rows over its column group (m: running
// max of the log2 scores, l: sum of 2^(s - m), w: sum of 2^(s - m) dP),
// updated with a key tile's scores and dP.
__device__ __forceinline__ void online_update(const float (&s)[NF][4], const float (&dp)[NF][4], float (&m)[2],
                                              float (&l)[2], float (&wsum)[2])
{
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float tmax = -INFINITY;
#pragma unroll
        for (int n = 0; n < NF; ++n) tmax = fmaxf(tmax, fmaxf(s[n][2 * hh], s[n][2 * hh + 1]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float mn = fmaxf(m[hh], tmax);
        float e = 0.f, ed = 0.f;
#pragma unroll
        for (int n = 0; n < NF; ++n)
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                // exp2f(-inf) = 0 for a masked pair; with mn = -inf (no kept pair
                // yet) the sums are discarded below
                const float ev = exp2f(s[n][2 * hh + x] - mn);
                e += ev;
                ed = fmaf(ev, dp[n][2 * hh + x], ed);
            }
        e += __shfl_xor_sync(0xffffffffu, e, 1);
        e += __shfl_xor_sync(0xffffffffu, e, 2);
        ed += __shfl_xor_sync(0xffffffffu, ed, 1);
        ed += __shfl_xor_sync(0xffffffffu, ed, 2);
        if (mn != -INFINITY) {
            const float alpha = (m[hh] == -INFINITY) ? 0.f : exp2f(m[hh] - mn);
            l[hh] = fmaf(l[hh], alpha, e);
            wsum[hh] = fmaf(wsum[hh], alpha, ed);
            m[hh] = mn;
        }
    }
}

// States (m, l, w) of n parts of a row, `stride` floats apart, combined in
// order: the row's max, and l and w rescaled to it.
__device__ __forceinline__ void combine_states(const float *a, int n, size_t stride, float &mx, float &lt,
                                               float &wt)
{
    mx = -INFINITY;
    for (int c = 0; c < n; ++c) mx = fmaxf(mx, a[c * stride]);
    lt = 0.f;
    wt = 0.f;
    for (int c = 0; c < n; ++c) {
        const float *x = a + c * stride;
        const float sa = (x[0] == -INFINITY) ? 0.f : exp2f(x[0] - mx);
        lt = fmaf(x[1], sa, lt);
        wt = fmaf(x[2], sa, wt);
    }
}

// ---- stats: log2-sum-exp and D per query row --------------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_stats_kernel(const BwdParams p)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), i0 = blockIdx.y * T;
    TXL_CHECK(bh < (long long)p.B * p.H && i0 < p.L, p.status);
    stage_rows(sm, p, bh, i0);
    // online state of the lane's two rows over its column group
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, wsum[2] = {0.f, 0.f};
    const int jend = min(p.K, p.M + i0 + T);  // later keys are hidden from every row
    issue_key_tile(sm, p, bh, h, i0, 0, 0);
    for (int j0 = 0, buf = 0; j0 < jend; j0 += T, buf ^= 1) {
        __syncthreads();  // the other buffer's last readers are done
        const bool more = j0 + T < jend;
        if (more) issue_key_tile(sm, p, bh, h, i0, j0 + T, buf ^ 1);
        key_tile_ready(sm, p, h, buf, more);
        float s[NF][4], dp[NF][4];
        key_tile_scores(sm, p, L, i0, j0, s, dp,
                        Bufs{OFF_Q, OFF_D, buf ? OFF_K1 : OFF_K, buf ? OFF_V1 : OFF_V, buf ? OFF_W1 : OFF_W});
        online_update(s, dp, m, l, wsum);
    }
    // the four column groups of each row: red[group][row][m, l, w]
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    __syncthreads();
    if (L.t == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float *d = red + ((L.warp & 3) * T + L.rb + L.g + 8 * hh) * 3;
            d[0] = m[hh];
            d[1] = l[hh];
            d[2] = wsum[hh];
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        const int i = threadIdx.x, gi = i0 + i;
        float mx, lt, wt;
        combine_states(red + i * 3, 4, T * 3, mx, lt, wt);
        if (gi < p.L && mx != -INFINITY) {
            p.lse2[bh * p.L + gi] = mx + log2f(lt);
            p.dsum[bh * p.L + gi] = wt / lt;
        }
    }
}

// ---- dq, and the chunk's partials of du and dv_bias ---------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_dq_kernel(const BwdParams p)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), i0 = blockIdx.y * T;
    TXL_CHECK(bh < (long long)p.B * p.H && i0 < p.L, p.status);
    stage_rows(sm, p, bh, i0);
    float ls[2], dd[2];
    load_row_stats(p, L, bh, i0, ls, dd);
    float dqc[NF][4], dqp[NF][4];  // content (k) and position (table) parts; rows i, columns t
    zero(dqc);
    zero(dqp);
    // g by window column, z[i][w] = g[i][i - w + 63]: the columns no key of a
    // tile reaches (w < i or w > i + 63) stay zero, the others are rewritten
    // by every tile
    for (int idx = threadIdx.x; idx < T * (LDZ / 4); idx += THREADS) {
        reinterpret_cast<uint32_t *>(sm + OFF_ZH)[idx] = 0u;
        reinterpret_cast<uint32_t *>(sm + OFF_ZL)[idx] = 0u;
    }
    const int jend = min(p.K, p.M + i0 + T);
    issue_key_tile(sm, p, bh, h, i0, 0, 0);
    for (int j0 = 0, buf = 0; j0 < jend; j0 += T, buf ^= 1) {
        __syncthreads();  // the other buffer's last readers are done
        const bool more = j0 + T < jend;
        if (more) issue_key_tile(sm, p, bh, h, i0, j0 + T, buf ^ 1);
        key_tile_ready(sm, p, h, buf, more);
        float s[NF][4], dp[NF][4], g[NF][4];
        key_tile_scores(sm, p, L, i0, j0, s, dp,
                        Bufs{OFF_Q, OFF_D, buf ? OFF_K1 : OFF_K, buf ? OFF_V1 : OFF_V, buf ? OFF_W1 : OFF_W});
        grad_scores(sm, p, L, s, dp, ls, dd, g, false, true);
        store_g(p, L, bh, i0, j0, g);
        __syncthreads();
        const int cbo = L.cb;  // output columns: dimensions
        warp_nn2<NF>(dqc, smem_u32(sm + OFF_GH) + L.rb * LDB, smem_u32(sm + OFF_GL) + L.rb * LDB, LDB,
                    false, smem_u32(sm + (buf ? OFF_K1 : OFF_K)) + cbo * 2, LDB, T, L.lane);
        warp_nn2<NF>(dqp, smem_u32(sm + OFF_ZH) + L.rb * LDZ, smem_u32(sm + OFF_ZL) + L.rb * LDZ, LDZ,
                    false, smem_u32(sm + (buf ? OFF_W1 : OFF_W)) + cbo * 2, LDB, W, L.lane);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int gi = i0 + L.rb + L.g + 8 * hh;
        if (gi < p.L) {
            float *dst = p.dq + (bh * p.L + gi) * DH;
#pragma unroll
            for (int n = 0; n < NF; ++n)
                *reinterpret_cast<float2 *>(dst + L.cb + 8 * n + 2 * L.t) =
                    make_float2(dqc[n][2 * hh] + dqp[n][2 * hh], dqc[n][2 * hh + 1] + dqp[n][2 * hh + 1]);
        }
    }
    // du and dv_bias partials of this chunk: column sums of the two parts over
    // its rows (rows past L hold zeros), the four row strips summed in order.
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    __syncthreads();
    column_sums(red, 2 * DH, L, L.cb, dqc);
    column_sums(red, 2 * DH, L, DH + L.cb, dqp);
    __syncthreads();
    if (threadIdx.x < 2 * DH) {
        const float acc = ((red[threadIdx.x] + red[2 * DH + threadIdx.x]) + red[4 * DH + threadIdx.x]) +
                          red[6 * DH + threadIdx.x];
        p.part[(bh * gridDim.y + blockIdx.y) * 2 * DH + threadIdx.x] = acc;
    }
}

// ---- dk, dv per 64-key tile ----------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_dkv_kernel(const BwdParams p)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), j0 = blockIdx.y * T;
    TXL_CHECK(bh < (long long)p.B * p.H && j0 < p.K, p.status);
    stage(sm + OFF_K, LDB, T, p.k + bh * p.K * DH, j0, 1, p.K);
    stage(sm + OFF_V, LDB, T, p.v + bh * p.K * DH, j0, 1, p.K);
    float *cs = reinterpret_cast<float *>(sm + OFF_CS);  // sum over rows of g, per key
    if (threadIdx.x < T) cs[threadIdx.x] = 0.f;
    __syncthreads();
    row_dots(reinterpret_cast<float *>(sm + OFF_BK), sm + OFF_K, LDB, T, p.u + (size_t)h * DH);
    float dk[NF][4], dv[NF][4];  // rows: keys; columns: dimensions
    zero(dk);
    zero(dv);
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    // the first chunk with a row that sees key j0 (distance M + i - j0 >= 0)
    const int i_first = max(0, j0 - p.M) / T * T;
    issue_chunk(sm, p, bh, h, i_first, j0, 0);
    for (int i0 = i_first, buf = 0; i0 < p.L; i0 += T, buf ^= 1) {
        __syncthreads();  // the other buffer's last readers are done
        const bool more = i0 + T < p.L;
        if (more) issue_chunk(sm, p, bh, h, i0 + T, j0, buf ^ 1);
        if (more) async_wait<3>();
        else async_wait<0>();
        __syncthreads();
        const Bufs B = chunk_bufs(buf);
        row_dots(reinterpret_cast<float *>(sm + OFF_BW), sm + B.w, LDB, W, p.vb + (size_t)h * DH);
        __syncthreads();
        float ls[2], dd[2];
        load_row_stats(p, L, bh, i0, ls, dd);
        float s[NF][4], dp[NF][4], g[NF][4];
        key_tile_scores(sm, p, L, i0, j0, s, dp, B);
        grad_scores(sm, p, L, s, dp, ls, dd, g, true);
        column_sums(red, T, L, L.cb, g);
        __syncthreads();
        if (threadIdx.x < T)
            cs[threadIdx.x] += ((red[threadIdx.x] + red[T + threadIdx.x]) + red[2 * T + threadIdx.x]) +
                               red[3 * T + threadIdx.x];
        // dv = P^T dout, dk = g^T q (+ the column sums times u, at the end)
        warp_nn2<NF>(dv, smem_u32(sm + OFF_PH) + L.rb * 2, smem_u32(sm + OFF_PL) + L.rb * 2, LDB,
                    true, smem_u32(sm + B.d) + L.cb * 2, LDB, T, L.lane);
        warp_nn2<NF>(dk, smem_u32(sm + OFF_GH) + L.rb * 2, smem_u32(sm + OFF_GL) + L.rb * 2, LDB,
                    true, smem_u32(sm + B.q) + L.cb * 2, LDB, T, L.lane);
    }
    __syncthreads();
    const __nv_bfloat16 *u = p.u + (size_t)h * DH;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int j = L.rb + L.g + 8 * hh, gj = j0 + j;
        if (gj < p.K) {
            float *ok = p.dk + (bh * p.K + gj) * DH, *ov = p.dv + (bh * p.K + gj) * DH;
#pragma unroll
            for (int n = 0; n < NF; ++n) {
                const int c = L.cb + 8 * n + 2 * L.t;
                const float u0 = __bfloat162float(u[c]), u1 = __bfloat162float(u[c + 1]);
                *reinterpret_cast<float2 *>(ok + c) =
                    make_float2(fmaf(cs[j], u0, dk[n][2 * hh]), fmaf(cs[j], u1, dk[n][2 * hh + 1]));
                *reinterpret_cast<float2 *>(ov + c) = make_float2(dv[n][2 * hh], dv[n][2 * hh + 1]);
            }
        }
    }
}

// ---- the table gradient per head and 64-distance tile ---------------------------
// Pair (row i, distance d) is key j = M + i - d; the dq passes stored g of every
// pair they visit.  Over the batch and the query chunks that reach the tile,
// in a fixed order: row i's 64 keys M + i - d0 - 63 .. M + i - d0 (copied in two
// items ahead, with the chunk's q rows, through a ring of three slots, as the
// 68-key run that starts at the 16-byte boundary below them; keys below 0 come
// in as zeros) become a bf16 head / rest pair indexed by e = 63 - (d - d0), the
// keys' own order; then on the tensor cores dr_e += sum_i g q_i and, through a
// column of ones, cs_e += sum_i g, which carries the v part:
// dr_d = sum g (q_i + v).
constexpr int LDGF = DH + 8;   // floats per staged g row (68 used)
constexpr int GRUN = DH + 4;   // keys staged per row
constexpr int DR_NS = 3;                            // items in the copy ring
constexpr int DR_GF = 0;                            // g rows [64][72] fp32, per ring slot
constexpr int DR_Q = DR_GF + DR_NS * T * LDGF * 4;  // q rows of the chunk, per ring slot
constexpr int DR_GH = DR_Q + DR_NS * T * LDB;       // g head, [row][e]
constexpr int DR_GL = DR_GH + T * LDB;              // g rest
constexpr int DR_CS = DR_GL + T * LDB;              // fp32 [64]: column sums by e
constexpr int DR_SMEM = DR_CS + T * 4;
static_assert(DR_Q % 16 == 0 && DR_GH % 16 == 0 && 2 * DR_SMEM <= 232448, "table-gradient tiles");

// Rows i0 .. i0 + 63 of the head's g into [64][LDGF]: row gi holds the GRUN
// keys from M + gi - d0 - 63 rounded down to a multiple of 4 (two's-complement
// `& ~3` floors negative keys too), 16 bytes per copy (4 keys never straddle a
// key tile); copies of keys outside [0, Kd) or rows at or past L are
// zero-filled by a zero source size (their address kept in bounds).  Thread
// (row w = tid / 8, runs tid % 8 + 8 m).  One commit group.
__device__ __forceinline__ void stage_g_rows(uint8_t *dst, const BwdParams &p, long long bh, int i0, int d0)
{
    static_assert(THREADS == 8 * T && GRUN / 4 <= 24 && T == 64, "eight threads per staged row");
    const int w = threadIdx.x >> 3, gi = i0 + w;
    const int a0 = (p.M + gi - d0 - (T - 1)) & ~3;
    const float *head = p.g_all + (size_t)bh * (p.Kd / T) * p.L * T;
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        const int c = (threadIdx.x & 7) + 8 * m;
        if (c < GRUN / 4) {
            const int a = a0 + 4 * c;
            const bool in = gi < p.L && a >= 0 && a < p.Kd;
            const float *g = in ? head + ((size_t)((unsigned)a >> 6) * p.L + gi) * T + (a & (T - 1)) : p.g_all;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                             smem_u32(dst + w * LDGF * 4 + c * 16)),
                         "l"(g), "r"(in ? 16 : 0)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// One warp, rows e = its 16 of the tile: c += (Gh + Gl)^T q over the 64 rows i
// (G stored [i][e], q stored [i][dimension]); with_cs: cs += (Gh + Gl)^T 1,
// whose B fragment (column 0 all ones, the others zero) lives in registers.
__device__ __forceinline__ void dr_mma(float (&c)[NF][4], float (&cs)[4], bool with_cs, uint32_t gh,
                                       uint32_t gl, uint32_t q, int lane)
{
    const uint32_t ones = (lane >> 2) == 0 ? 0x3f803f80u : 0u;  // bf16 1.0, 1.0 in column n = 0
#pragma unroll
    for (int k0 = 0; k0 < T; k0 += 16) {
        uint32_t fh[4], fl[4], bfr[4];
        const uint32_t off = (k0 + (lane >> 4) * 8 + (lane & 7)) * LDB + ((lane >> 3) & 1) * 16;
        ldsm_x4_t(fh, gh + off);
        ldsm_x4_t(fl, gl + off);
        ldsm_x4_t(bfr, q + (k0 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LDB + ((lane >> 4) * 8) * 2);
        mma16816(c[0], fh, bfr[0], bfr[1]);
        mma16816(c[1], fh, bfr[2], bfr[3]);
        mma16816(c[0], fl, bfr[0], bfr[1]);
        mma16816(c[1], fl, bfr[2], bfr[3]);
        if (with_cs) {
            mma16816(cs, fh, ones, ones);
            mma16816(cs, fl, ones, ones);
        }
    }
}

__global__ void __launch_bounds__(THREADS, 2) bwd_dr_kernel(const BwdParams p)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const int d0 = blockIdx.x * T, h = blockIdx.y;
    TXL_CHECK(h < p.H && d0 < p.r_rows, p.status);
    float dr[NF][4], cs[4];  // rows: e; columns: dimensions (cs: column 0)
    zero(dr);
    cs[0] = cs[1] = cs[2] = cs[3] = 0.f;
    const bool with_cs = (L.warp & 3) == 0;  // one warp per row strip sums g
    if (d0 < p.K) {
        // the chunks with a row that reaches distance d0 (M + i >= d0)
        const int i_first = max(0, d0 - p.M) / T * T;
        const int n_ch = (p.L - i_first + T - 1) / T, n_items = p.B * n_ch;
        // items in order (batch row, chunk): the next one to copy in, and the
        // current one's chunk (counters instead of divisions)
        int nb = 0, nc = 0, cc = 0;
        auto issue_next = [&](int slot) {
            const long long bh = (long long)nb * p.H + h;
            const int i0 = i_first + nc * T;
            stage_g_rows(sm + DR_GF + slot * T * LDGF * 4, p, bh, i0, d0);
            stage_async(sm + DR_Q + slot * T * LDB, LDB, T, p.q + bh * p.L * DH, i0, 1, p.L);
            if (++nc == n_ch) nc = 0, ++nb;
        };
        // this thread's conversion: row i, keys e = 8 r .. 8 r + 7 of the tile
        const int ci = threadIdx.x >> 3, cr = threadIdx.x & 7;
        issue_next(0);
        if (n_items > 1) issue_next(1);
        for (int it = 0, buf = 0; it < n_items; ++it, buf = (buf + 1 == DR_NS) ? 0 : buf + 1) {
            const int i0 = i_first + cc * T;
            if (++cc == n_ch) cc = 0;
            // two copy groups per item: this item's have landed once at most the
            // next item's are pending; the barrier also ends the last item's
            // readers of the g tiles and of the slot refilled below
            if (it + 1 < n_items) async_wait<2>();
            else async_wait<0>();
            __syncthreads();
            if (it + 2 < n_items) issue_next(buf + 2 >= DR_NS ? buf + 2 - DR_NS : buf + 2);
            {
                // key M + gi - d0 - 63 + e sits at staged column ((M + gi - d0 - 63) & 3) + e
                const float *src = reinterpret_cast<const float *>(sm + DR_GF + buf * T * LDGF * 4) +
                                   ci * LDGF + ((p.M + i0 + ci - d0 - (T - 1)) & 3) + 8 * cr;
                uint4 hd, rs;
                split2(src[0], src[1], hd.x, rs.x);
                split2(src[2], src[3], hd.y, rs.y);
                split2(src[4], src[5], hd.z, rs.z);
                split2(src[6], src[7], hd.w, rs.w);
                *reinterpret_cast<uint4 *>(sm + DR_GH + ci * LDB + 16 * cr) = hd;
                *reinterpret_cast<uint4 *>(sm + DR_GL + ci * LDB + 16 * cr) = rs;
            }
            __syncthreads();
            dr_mma(dr, cs, with_cs, smem_u32(sm + DR_GH) + L.rb * 2, smem_u32(sm + DR_GL) + L.rb * 2,
                   smem_u32(sm + DR_Q + buf * T * LDB) + L.cb * 2, L.lane);
        }
    }
    // the column sums of each row strip, from its first warp's column 0
    float *csm = reinterpret_cast<float *>(sm + DR_CS);
    if (with_cs && L.t == 0) {
        csm[L.rb + L.g] = cs[0];
        csm[L.rb + L.g + 8] = cs[2];
    }
    __syncthreads();
    const __nv_bfloat16 *vb = p.vb + (size_t)h * DH;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int e = L.rb + L.g + 8 * hh, d = d0 + (T - 1) - e;
        if (d < p.r_rows) {
            float *dst = p.dr + ((size_t)h * p.r_rows + (p.r_rows - 1 - d)) * DH;
            const float cd = (d < p.K) ? csm[e] : 0.f;
#pragma unroll
            for (int n = 0; n < NF; ++n) {
                const int col = L.cb + 8 * n + 2 * L.t;
                const float v0 = __bfloat162float(vb[col]), v1 = __bfloat162float(vb[col + 1]);
                *reinterpret_cast<float2 *>(dst + col) =
                    make_float2(fmaf(cd, v0, dr[n][2 * hh]), fmaf(cd, v1, dr[n][2 * hh + 1]));
            }
        }
    }
}

// ---- du, dv_bias: the chunks' partials summed over the batch in order -----------
__global__ void bwd_bias_kernel(const BwdParams p, int n_chunks)
{
    const int h = blockIdx.x, t = threadIdx.x;  // t < 2 * DH
    float acc = 0.f;
    for (int b = 0; b < p.B; ++b) {
        const size_t bh = (size_t)b * p.H + h;
        for (int c = 0; c < n_chunks; ++c) acc += p.part[(bh * n_chunks + c) * 2 * DH + t];
    }
    if (t < DH) p.du[(size_t)h * DH + t] = acc;
    else p.dvb[(size_t)h * DH + t - DH] = acc;
}

// ---- dq, dk, dv in one pass, for segments of at most two row chunks -----------
// Block (b*H + h, key split): every row of the segment stays staged (chunk 0 in
// the q / dout regions, chunk 1 in the second table-window region); over the
// split's key tiles (keys and values copied in one tile ahead, the 192-row
// table window of both chunks at the tile's start), per chunk: the scores,
// g and P, then dq += g k + (g by window column) r_w, and the tile's
// dk += g^T q, dv += P^T dout.  A tile's dk and dv are complete after its
// chunks, since the block holds every row; dq is summed over the key splits
// afterwards in a fixed order.  One score pass instead of the two of the dq and
// dk / dv launches.
constexpr int Q_ROWS1 = OFF_W1;             // q rows of chunk 1
constexpr int D_ROWS1 = OFF_W1 + T * LDB;   // dout rows of chunk 1
constexpr int WBW2 = OFF_W + (W + T) * LDB; // v.r of the 192-row window (in the value-window region)
static_assert(WBW2 + (W + T) * 4 <= OFF_GH, "window biases must fit the value-window region");
static_assert(2 * T * LDB <= W * LDB, "two row chunks must fit the second window region");

__global__ void __launch_bounds__(THREADS, 1) bwd_dqkv_kernel(const BwdParams p, int n_splits)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), split = blockIdx.y;
    const int n_ch = (p.L + T - 1) / T;
    const int n_kt = (p.K + T - 1) / T;
    const int per = (n_kt + n_splits - 1) / n_splits;
    const int kt0 = split * per, kt1 = min(n_kt, kt0 + per);
    TXL_CHECK(bh < (long long)p.B * p.H && n_ch <= 2 && split < n_splits, p.status);
    auto ko = [](int b) { return b ? OFF_K1 : OFF_K; };
    auto vo = [](int b) { return b ? OFF_V1 : OFF_V; };
    stage(sm + OFF_Q, LDB, T, p.q + bh * p.L * DH, 0, 1, p.L);
    stage(sm + OFF_D, LDB, T, p.dout + bh * p.L * DH, 0, 1, p.L);
    stage(sm + Q_ROWS1, LDB, T, p.q + bh * p.L * DH, T, 1, p.L);
    stage(sm + D_ROWS1, LDB, T, p.dout + bh * p.L * DH, T, 1, p.L);
    float ls[2][2], dd[2][2];
    load_row_stats(p, L, bh, 0, ls[0], dd[0]);
    load_row_stats(p, L, bh, T, ls[1], dd[1]);
    float dqc[2][NF][4], dqp[2][NF][4];
    zero(dqc[0]);
    zero(dqc[1]);
    zero(dqp[0]);
    zero(dqp[1]);
    float *cs = reinterpret_cast<float *>(sm + OFF_CS);  // per key of the tile: sum of g over the rows
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    // window-ordered g: the columns no key reaches stay zero
    for (int idx = threadIdx.x; idx < T * (LDZ / 4); idx += THREADS) {
        reinterpret_cast<uint32_t *>(sm + OFF_ZH)[idx] = 0u;
        reinterpret_cast<uint32_t *>(sm + OFF_ZL)[idx] = 0u;
    }
    auto issue_kv = [&](int kt, int b) {
        stage_async(sm + ko(b), LDB, T, p.k + bh * p.K * DH, (long long)kt * T, 1, p.K);
        stage_async(sm + vo(b), LDB, T, p.v + bh * p.K * DH, (long long)kt * T, 1, p.K);
    };
    if (kt0 < kt1) issue_kv(kt0, 0);
    for (int kt = kt0, buf = 0; kt < kt1; ++kt, buf ^= 1) {
        const int j0 = kt * T;
        __syncthreads();  // the last tile's readers of the window and of this buffer pair are done
        // window row w: the table row of distance M - j0 - 63 + w (w < 192);
        // chunk c reads rows 64 c .. 64 c + 127
        const long long dmin = (long long)p.M - j0 - (T - 1);
        stage_async(sm + OFF_W, LDB, W + T, p.r + (size_t)h * p.r_rows * DH, p.r_rows - 1 - dmin, -1,
                    p.r_rows);
        const bool more = kt + 1 < kt1;
        if (more) issue_kv(kt + 1, buf ^ 1);
        if (more) async_wait<2>();
        else async_wait<0>();
        __syncthreads();
        row_dots(reinterpret_cast<float *>(sm + OFF_BK), sm + ko(buf), LDB, T, p.u + (size_t)h * DH);
        row_dots(reinterpret_cast<float *>(sm + WBW2), sm + OFF_W, LDB, W + T, p.vb + (size_t)h * DH);
        if (threadIdx.x < T) cs[threadIdx.x] = 0.f;
        __syncthreads();
        float dk[NF][4], dv[NF][4];
        zero(dk);
        zero(dv);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (c >= n_ch) break;  // (block-uniform)
            if (j0 > p.M + c * T + T - 1) continue;  // the tile is hidden from every row of the chunk
            const Bufs B{c ? Q_ROWS1 : OFF_Q, c ? D_ROWS1 : OFF_D, ko(buf), vo(buf), OFF_W + c * T * LDB,
                         WBW2 + c * T * 4};
            float s[NF][4], dp[NF][4], g[NF][4];
            key_tile_scores(sm, p, L, c * T, j0, s, dp, B);
            grad_scores(sm, p, L, s, dp, ls[c], dd[c], g, true, true);
            store_g(p, L, bh, c * T, j0, g);
            column_sums(red, T, L, L.cb, g);
            __syncthreads();
            if (threadIdx.x < T)
                cs[threadIdx.x] += ((red[threadIdx.x] + red[T + threadIdx.x]) + red[2 * T + threadIdx.x]) +
                                   red[3 * T + threadIdx.x];
            warp_nn2<NF>(dqc[c], smem_u32(sm + OFF_GH) + L.rb * LDB, smem_u32(sm + OFF_GL) + L.rb * LDB,
                         LDB, false, smem_u32(sm + ko(buf)) + L.cb * 2, LDB, T, L.lane);
            warp_nn2<NF>(dqp[c], smem_u32(sm + OFF_ZH) + L.rb * LDZ, smem_u32(sm + OFF_ZL) + L.rb * LDZ,
                         LDZ, false, smem_u32(sm + B.w) + L.cb * 2, LDB, W, L.lane);
            warp_nn2<NF>(dv, smem_u32(sm + OFF_PH) + L.rb * 2, smem_u32(sm + OFF_PL) + L.rb * 2, LDB,
                         true, smem_u32(sm + B.d) + L.cb * 2, LDB, T, L.lane);
            warp_nn2<NF>(dk, smem_u32(sm + OFF_GH) + L.rb * 2, smem_u32(sm + OFF_GL) + L.rb * 2, LDB,
                         true, smem_u32(sm + B.q) + L.cb * 2, LDB, T, L.lane);
        }
        __syncthreads();  // the tile's column sums are complete
        const __nv_bfloat16 *u = p.u + (size_t)h * DH;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = L.rb + L.g + 8 * hh, gj = j0 + j;
            if (gj < p.K) {
                float *okp = p.dk + (bh * p.K + gj) * DH, *ovp = p.dv + (bh * p.K + gj) * DH;
#pragma unroll
                for (int n = 0; n < NF; ++n) {
                    const int cc = L.cb + 8 * n + 2 * L.t;
                    const float u0 = __bfloat162float(u[cc]), u1 = __bfloat162float(u[cc + 1]);
                    *reinterpret_cast<float2 *>(okp + cc) =
                        make_float2(fmaf(cs[j], u0, dk[n][2 * hh]), fmaf(cs[j], u1, dk[n][2 * hh + 1]));
                    *reinterpret_cast<float2 *>(ovp + cc) = make_float2(dv[n][2 * hh], dv[n][2 * hh + 1]);
                }
            }
        }
    }
    // dq of the split (the final dq when unsplit)
    float *dqdst = (n_splits == 1) ? p.dq : p.dq_part + (size_t)split * p.B * p.H * p.L * DH;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int gi = c * T + L.rb + L.g + 8 * hh;
            if (c < n_ch && gi < p.L) {
                float *dst = dqdst + (bh * p.L + gi) * DH;
#pragma unroll
                for (int n = 0; n < NF; ++n)
                    *reinterpret_cast<float2 *>(dst + L.cb + 8 * n + 2 * L.t) =
                        make_float2(dqc[c][n][2 * hh] + dqp[c][n][2 * hh],
                                    dqc[c][n][2 * hh + 1] + dqp[c][n][2 * hh + 1]);
            }
        }
    // du, dv_bias partials of the split: column sums of the two parts of dq
#pragma unroll
    for (int n = 0; n < NF; ++n)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            dqc[0][n][q] += dqc[1][n][q];
            dqp[0][n][q] += dqp[1][n][q];
        }
    __syncthreads();
    column_sums(red, 2 * DH, L, L.cb, dqc[0]);
    column_sums(red, 2 * DH, L, DH + L.cb, dqp[0]);
    __syncthreads();
    if (threadIdx.x < 2 * DH) {
        const float acc = ((red[threadIdx.x] + red[2 * DH + threadIdx.x]) + red[4 * DH + threadIdx.x]) +
                          red[6 * DH + threadIdx.x];
        p.part[(bh * n_splits + split) * 2 * DH + threadIdx.x] = acc;
    }
}

// ---- stats for segments of at most two row chunks ------------------------------
// Block (b*H + h, key split), staged as the one-pass kernel: both chunks' q and
// dout rows, the split's key tiles (keys and values copied in one tile ahead,
// the 192-row table window of both chunks at the tile's start), so each key,
// value and table tile is read once per segment.  Every row's online state over
// the split's keys; with one split that is the row's log2-sum-exp and D, with
// more the states go to `scratch` [split][row][m, l, w] for
// bwd_stats_merge_kernel.
__global__ void __launch_bounds__(THREADS, 1) bwd_stats2_kernel(const BwdParams p, int n_splits, float *scratch)
{
    extern __shared__ __align__(16) uint8_t sm[];
    const Lane L = lane_of();
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), split = blockIdx.y;
    const int n_ch = (p.L + T - 1) / T;
    const int n_kt = (p.K + T - 1) / T;
    const int per = (n_kt + n_splits - 1) / n_splits;
    const int kt0 = split * per, kt1 = min(n_kt, kt0 + per);
    TXL_CHECK(bh < (long long)p.B * p.H && n_ch <= 2 && split < n_splits, p.status);
    auto ko = [](int b) { return b ? OFF_K1 : OFF_K; };
    auto vo = [](int b) { return b ? OFF_V1 : OFF_V; };
    stage(sm + OFF_Q, LDB, T, p.q + bh * p.L * DH, 0, 1, p.L);
    stage(sm + OFF_D, LDB, T, p.dout + bh * p.L * DH, 0, 1, p.L);
    stage(sm + Q_ROWS1, LDB, T, p.q + bh * p.L * DH, T, 1, p.L);
    stage(sm + D_ROWS1, LDB, T, p.dout + bh * p.L * DH, T, 1, p.L);
    float m[2][2], l[2][2], wsum[2][2];  // [chunk][lane row]
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) m[c][hh] = -INFINITY, l[c][hh] = 0.f, wsum[c][hh] = 0.f;
    auto issue_kv = [&](int kt, int b) {
        stage_async(sm + ko(b), LDB, T, p.k + bh * p.K * DH, (long long)kt * T, 1, p.K);
        stage_async(sm + vo(b), LDB, T, p.v + bh * p.K * DH, (long long)kt * T, 1, p.K);
    };
    if (kt0 < kt1) issue_kv(kt0, 0);
    for (int kt = kt0, buf = 0; kt < kt1; ++kt, buf ^= 1) {
        const int j0 = kt * T;
        __syncthreads();  // the last tile's readers of the window and of this buffer pair are done
        // window row w: the table row of distance M - j0 - 63 + w (w < 192)
        const long long dmin = (long long)p.M - j0 - (T - 1);
        stage_async(sm + OFF_W, LDB, W + T, p.r + (size_t)h * p.r_rows * DH, p.r_rows - 1 - dmin, -1,
                    p.r_rows);
        const bool more = kt + 1 < kt1;
        if (more) issue_kv(kt + 1, buf ^ 1);
        if (more) async_wait<2>();
        else async_wait<0>();
        __syncthreads();
        row_dots(reinterpret_cast<float *>(sm + OFF_BK), sm + ko(buf), LDB, T, p.u + (size_t)h * DH);
        row_dots(reinterpret_cast<float *>(sm + WBW2), sm + OFF_W, LDB, W + T, p.vb + (size_t)h * DH);
        __syncthreads();
        if (n_ch == 2 && j0 <= p.M + T - 1) {
            // both chunks see the tile: their products back to back, chunk 1's
            // window product in the window-ordered g region (unused here), one barrier
            float sc[2][NF][4], dp[2][NF][4];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                zero(sc[c]);
                zero(dp[c]);
                warp_nt<NF>(sc[c], smem_u32(sm + (c ? Q_ROWS1 : OFF_Q)) + L.rb * LDB, LDB,
                            smem_u32(sm + ko(buf)) + L.cb * LDB, LDB, DH, L.lane);
                warp_nt<NF>(dp[c], smem_u32(sm + (c ? D_ROWS1 : OFF_D)) + L.rb * LDB, LDB,
                            smem_u32(sm + vo(buf)) + L.cb * LDB, LDB, DH, L.lane);
                window_product(sm, L, c ? Q_ROWS1 : OFF_Q, OFF_W + c * T * LDB,
                               reinterpret_cast<const float *>(sm + WBW2 + c * T * 4), c ? OFF_ZH : OFF_XS);
            }
            __syncthreads();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float s[NF][4];
                finish_scores(sm, p, L, c * T, j0, sc[c], s, c ? OFF_ZH : OFF_XS);
                online_update(s, dp[c], m[c], l[c], wsum[c]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (c >= n_ch) break;                    // (block-uniform)
                if (j0 > p.M + c * T + T - 1) continue;  // the tile is hidden from every row of the chunk
                if (c == 1) __syncthreads();             // chunk 0's readers of the window product are done
                const Bufs B{c ? Q_ROWS1 : OFF_Q, c ? D_ROWS1 : OFF_D, ko(buf), vo(buf), OFF_W + c * T * LDB,
                             WBW2 + c * T * 4};
                float s[NF][4], dp[NF][4];
                key_tile_scores(sm, p, L, c * T, j0, s, dp, B);
                online_update(s, dp, m[c], l[c], wsum[c]);
            }
        }
    }
    // the four column groups of each row: red[group][row][m, l, w] over the
    // 128 rows (in the window-product region, free now)
    float *red = reinterpret_cast<float *>(sm + OFF_XS);
    static_assert(4 * 2 * T * 3 <= T * LDX, "row states must fit the window-product region");
    __syncthreads();
    if (L.t == 0) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float *d = red + ((L.warp & 3) * 2 * T + c * T + L.rb + L.g + 8 * hh) * 3;
                d[0] = m[c][hh];
                d[1] = l[c][hh];
                d[2] = wsum[c][hh];
            }
    }
    __syncthreads();
    if (threadIdx.x < 2 * T) {
        const int gi = threadIdx.x;
        float mx, lt, wt;
        combine_states(red + gi * 3, 4, 2 * T * 3, mx, lt, wt);
        if (gi < p.L) {
            const size_t row = (size_t)bh * p.L + gi;
            if (n_splits == 1) {
                // one split holds every key, key 0 among them: the row has one
                p.lse2[row] = mx + log2f(lt);
                p.dsum[row] = wt / lt;
            } else {
                float *o = scratch + ((size_t)split * p.B * p.H * p.L + row) * 3;
                o[0] = mx;
                o[1] = lt;
                o[2] = wt;
            }
        }
    }
}

// The key splits' row states combined in split order.
__global__ void bwd_stats_merge_kernel(const BwdParams p, int n_splits, const float *scratch)
{
    const size_t rows = (size_t)p.B * p.H * p.L;
    for (size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += (size_t)gridDim.x * blockDim.x) {
        float mx, lt, wt;
        combine_states(scratch + r * 3, n_splits, rows * 3, mx, lt, wt);
        p.lse2[r] = mx + log2f(lt);
        p.dsum[r] = wt / lt;
    }
}

// dq = the key splits' partials summed in order.
__global__ void bwd_dq_reduce_kernel(const BwdParams p, int n_splits)
{
    const size_t n4 = (size_t)p.B * p.H * p.L * DH / 4;
    for (size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (size_t)gridDim.x * blockDim.x) {
        float4 acc = reinterpret_cast<const float4 *>(p.dq_part)[x];
        for (int s = 1; s < n_splits; ++s) {
            const float4 v = reinterpret_cast<const float4 *>(p.dq_part + (size_t)s * n4 * 4)[x];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        reinterpret_cast<float4 *>(p.dq)[x] = acc;
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

} // namespace

size_t bwd_dq_part_offset(int B, int H, int L)
{
    const size_t rows = (size_t)B * H * L;
    const int n_chunks = (L + T - 1) / T;
    const size_t parts = (size_t)B * H * (size_t)(n_chunks > kBwdMaxSplits ? n_chunks : kBwdMaxSplits);
    return 2 * align256(rows * sizeof(float)) + align256(parts * 2 * DH * sizeof(float));
}

size_t bwd_g_offset(int B, int H, int L)
{
    const size_t rows = (size_t)B * H * L;
    const int n_chunks = (L + T - 1) / T;
    size_t off = bwd_dq_part_offset(B, H, L);
    if (n_chunks <= 2) off += align256((size_t)kBwdMaxSplits * rows * DH * sizeof(float));
    return off;
}

size_t bwd_workspace_bytes(int B, int H, int L, int M)
{
    if (B <= 0 || H <= 0 || L <= 0 || M < 0) return 0;
    const size_t rows = (size_t)B * H * L;
    const size_t Kd = ((size_t)M + L + T - 1) / T * T;
    return bwd_g_offset(B, H, L) + align256(rows * Kd * sizeof(float));
}

cudaError_t launch_relattn_bwd(const BwdParams &p, cudaStream_t s)
{
    static bool attr_set[64] = {};  // the attributes are set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        for (const void *f : {(const void *)bwd_stats_kernel, (const void *)bwd_stats2_kernel,
                              (const void *)bwd_dq_kernel, (const void *)bwd_dkv_kernel,
                              (const void *)bwd_dqkv_kernel})
            if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          SMEM_BYTES)) != cudaSuccess)
                return e;
        if ((e = cudaFuncSetAttribute((const void *)bwd_dr_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, DR_SMEM)) != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const long long BH = (long long)p.B * p.H;
    const int n_chunks = (p.L + T - 1) / T, n_keys = (p.K + T - 1) / T;
    const int n_dist = (p.r_rows + T - 1) / T;
    if (BH > 0x7fffffffLL || n_chunks > 65535 || n_keys > 65535 || p.H > 65535)
        return cudaErrorInvalidValue;
    int n_bias = n_chunks;
    if (n_chunks <= 2) {
        // one pass for the statistics and one for dq, dk, dv over both chunks;
        // the key split that fills the SMs' waves best
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        int n_splits = 1;
        double best = 0.0;
        for (int sp = 1; sp <= kBwdMaxSplits && sp <= n_keys; ++sp) {
            const double blocks = (double)BH * sp;
            const double waves = std::ceil(blocks / sms);
            const double eff = blocks / (waves * sms);
            if (eff > best + 0.03) best = eff, n_splits = sp;  // more splits only for a clearly fuller wave
        }
        // the splits' row states go to the dq partials' region, free until the one-pass kernel
        bwd_stats2_kernel<<<dim3((unsigned)BH, n_splits), THREADS, SMEM_BYTES, s>>>(p, n_splits, p.dq_part);
        if (n_splits > 1) bwd_stats_merge_kernel<<<256, 256, 0, s>>>(p, n_splits, p.dq_part);
        bwd_dqkv_kernel<<<dim3((unsigned)BH, n_splits), THREADS, SMEM_BYTES, s>>>(p, n_splits);
        if (n_splits > 1) bwd_dq_reduce_kernel<<<1024, 256, 0, s>>>(p, n_splits);
        n_bias = n_splits;
    } else {
        bwd_stats_kernel<<<dim3((unsigned)BH, n_chunks), THREADS, SMEM_BYTES, s>>>(p);
        bwd_dq_kernel<<<dim3((unsigned)BH, n_chunks), THREADS, SMEM_BYTES, s>>>(p);
        bwd_dkv_kernel<<<dim3((unsigned)BH, n_keys), THREADS, SMEM_BYTES, s>>>(p);
    }
    bwd_dr_kernel<<<dim3((unsigned)n_dist, p.H), THREADS, DR_SMEM, s>>>(p);
    bwd_bias_kernel<<<p.H, 2 * DH, 0, s>>>(p, n_bias);
    return cudaGetLastError();
}

} // namespace txl
