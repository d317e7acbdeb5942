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
// Five launches, all fp32 on the CUDA cores, tiles of 64 query rows x 64
// columns (keys, or distances for the table gradient), 256 threads, each
// thread a 4 x 4 block of pairs (rows 4 ty + a, columns tx + 16 c):
//   stats   per 64-row chunk, over its key tiles: online log-sum-exp of the
//           scores and D (no value from the forward call is needed)
//   dq      per 64-row chunk, over its key tiles: dq, and the chunk's
//           partials of du and dv_bias
//   dkv     per 64-key tile, over the query chunks that see it: dk, dv
//   dr      per head and 64-distance tile, over the batch and query chunks:
//           the table gradient, with no atomics
//   bias    per head: du, dv_bias from the partials, in a fixed order
// Every tile recomputes its scores.  The Appendix B shift is index arithmetic,
// as in the forward: the position term of a 64 x 64 pair tile is row i of the
// dense product (q + v) R_w^T over the tile's 127-distance window, read at
// window column i - j + 63; the shifted contractions (dq's position part, and
// the content part of the distance tiles) are dense products over the window
// of the same g re-laid out by that index.  Results repeat bit for bit.
#include "kernels.h"

namespace txl {
namespace {

constexpr int DH = 64;
constexpr int T = kBwdRows;     // rows / columns of a pair tile
constexpr int W = 2 * T;        // window rows of a tile (127 used)
constexpr int THREADS = 256;
constexpr int LD = DH + 4;      // fp32 row stride of a 64-wide tile (16-byte rows, bank-spread)
constexpr int LDW = W + 4;      // row stride of a 128-wide window product

// Shared-memory regions (floats).  q + u, q + v and dout of a row chunk; a
// 64-row operand (key tile, or table tile by distance); a 128-row window
// (table rows by distance, or key rows); the 64 x 128 window product; a
// 64 x 64 transposed pair tile; and a region holding either the value tile and
// a second pair tile (key tiles) or the value window (distance tiles).
constexpr int OFF_QU = 0;
constexpr int OFF_QV = OFF_QU + T * LD;
constexpr int OFF_DO = OFF_QV + T * LD;
constexpr int OFF_A64 = OFF_DO + T * LD;
constexpr int OFF_W1 = OFF_A64 + T * LD;
constexpr int OFF_XS = OFF_W1 + W * LD;
constexpr int OFF_T1 = OFF_XS + T * LDW;
constexpr int OFF_U = OFF_T1 + T * LD;
constexpr int OFF_V64 = OFF_U;             // key tiles: value tile
constexpr int OFF_T2 = OFF_U + T * LD;     // key tiles: second pair tile
constexpr int OFF_W2 = OFF_U;              // distance tiles: value window
constexpr int SMEM_FLOATS = OFF_U + W * LD;
constexpr int SMEM_BYTES = SMEM_FLOATS * 4;
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert((LD * 4) % 16 == 0 && (LDW * 4) % 16 == 0, "rows must stay 16-byte aligned");

__device__ __forceinline__ float bf(uint32_t w, int hi)
{
    return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

// Rows w = 0 .. n-1 of dst [n][ld] (fp32) from bf16 rows src_row(w) = row0 +
// step * w of a [rows_total][64] matrix; rows outside [0, rows_total) become
// zeros.  `add` (may be null): a 64-vector added to every loaded row.
__device__ __forceinline__ void stage(float *dst, int ld, int n, const __nv_bfloat16 *src,
                                      long long row0, int step, long long rows_total,
                                      const __nv_bfloat16 *add)
{
    for (int idx = threadIdx.x; idx < n * 8; idx += THREADS) {
        const int w = idx >> 3, c = idx & 7;
        const long long sr = row0 + (long long)step * w;
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (sr >= 0 && sr < rows_total) {
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src + sr * DH) + c);
            lo = make_float4(bf(x.x, 0), bf(x.x, 1), bf(x.y, 0), bf(x.y, 1));
            hi = make_float4(bf(x.z, 0), bf(x.z, 1), bf(x.w, 0), bf(x.w, 1));
            if (add) {
                const uint4 y = __ldg(reinterpret_cast<const uint4 *>(add) + c);
                lo.x += bf(y.x, 0); lo.y += bf(y.x, 1); lo.z += bf(y.y, 0); lo.w += bf(y.y, 1);
                hi.x += bf(y.z, 0); hi.y += bf(y.z, 1); hi.z += bf(y.w, 0); hi.w += bf(y.w, 1);
            }
        }
        float4 *d = reinterpret_cast<float4 *>(dst + w * ld + c * 8);
        d[0] = lo;
        d[1] = hi;
    }
}

// acc[a][c] += sum_k A[4 ty + a][k] * B[tx + 16 c][k]   (both row-major in k)
template <int NC>
__device__ __forceinline__ void gemm_nt(float (&acc)[4][NC], const float *A, int lda,
                                        const float *B, int ldb, int kdim, int ty, int tx)
{
#pragma unroll 2
    for (int k = 0; k < kdim; k += 4) {
        float4 a[4], b[NC];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4 *>(A + (ty * 4 + r) * lda + k);
#pragma unroll
        for (int c = 0; c < NC; ++c) b[c] = *reinterpret_cast<const float4 *>(B + (tx + 16 * c) * ldb + k);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float s = acc[r][c];
                s = fmaf(a[r].x, b[c].x, s);
                s = fmaf(a[r].y, b[c].y, s);
                s = fmaf(a[r].z, b[c].z, s);
                s = fmaf(a[r].w, b[c].w, s);
                acc[r][c] = s;
            }
    }
}

// acc[a][c] += sum_k A[4 ty + a][k] * B[k][tx + 16 c]   (A row-major in k, B in n)
template <int NC>
__device__ __forceinline__ void gemm_nn(float (&acc)[4][NC], const float *A, int lda,
                                        const float *B, int ldb, int kdim, int ty, int tx)
{
#pragma unroll 2
    for (int k = 0; k < kdim; k += 4) {
        float4 a[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4 *>(A + (ty * 4 + r) * lda + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float b[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) b[c] = B[(k + kk) * ldb + tx + 16 * c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float av = kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w;
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(av, b[c], acc[r][c]);
            }
        }
    }
}

template <int R, int C>
__device__ __forceinline__ void zero(float (&a)[R][C])
{
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) a[r][c] = 0.f;
}

// ---- staging of a row chunk and of a key tile ------------------------------
// q + u, q + v and dout of rows i0 .. i0+63 of plane bh (rows past L: zeros).
__device__ __forceinline__ void stage_rows(float *sm, const BwdParams &p, long long bh, int h, int i0)
{
    const __nv_bfloat16 *q = p.q + bh * p.L * DH;
    stage(sm + OFF_QU, LD, T, q, i0, 1, p.L, p.u + (size_t)h * DH);
    stage(sm + OFF_QV, LD, T, q, i0, 1, p.L, p.vb + (size_t)h * DH);
    stage(sm + OFF_DO, LD, T, p.dout + bh * p.L * DH, i0, 1, p.L, nullptr);
}

// Window row w = the table row of distance dmin + w (row r_rows-1-distance of
// r; distances outside [0, r_rows) give zeros).
__device__ __forceinline__ void stage_table_window(float *dst, const BwdParams &p, int h, long long dmin)
{
    stage(dst, LD, W, p.r + (size_t)h * p.r_rows * DH, p.r_rows - 1 - dmin, -1, p.r_rows, nullptr);
}

// Log2-scaled scores (-inf where masked) and dP = dout . v of the thread's 16
// pairs (row i = 4 ty + a of the chunk at i0, key j = tx + 16 c of the tile at
// j0), from staged rows, keys (A64), values (V64) and the table window of
// distances M + i0 - j0 - 63 + w (W1).  Contains a block barrier.
__device__ __forceinline__ void key_tile_scores(float *sm, const BwdParams &p, int i0, int j0,
                                                int ty, int tx, float (&s)[4][4], float (&dp)[4][4])
{
    float sc[4][4], x[4][8];
    zero(sc);
    zero(x);
    zero(dp);
    gemm_nt<4>(sc, sm + OFF_QU, LD, sm + OFF_A64, LD, DH, ty, tx);
    gemm_nt<8>(x, sm + OFF_QV, LD, sm + OFF_W1, LD, DH, ty, tx);
    gemm_nt<4>(dp, sm + OFF_DO, LD, sm + OFF_V64, LD, DH, ty, tx);
    float *xs = sm + OFF_XS;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) xs[(ty * 4 + r) * LDW + tx + 16 * c] = x[r][c];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = ty * 4 + r, j = tx + 16 * c;
            const int gi = i0 + i, gj = j0 + j;
            // Appendix B: distance M + gi - gj is window column i - j + 63
            const float pos = xs[i * LDW + i - j + T - 1];
            const bool keep = gi < p.L && gj < p.K && gj <= p.M + gi;
            s[r][c] = keep ? (sc[r][c] + pos) * p.scale_log2 : -INFINITY;
        }
}

// Row statistics of the thread's rows, from the stats kernel's results.
__device__ __forceinline__ void load_row_stats(const BwdParams &p, long long bh, int i0, int ty,
                                               float (&ls)[4], float (&dd)[4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int gi = i0 + ty * 4 + r;
        ls[r] = gi < p.L ? p.lse2[bh * p.L + gi] : 0.f;
        dd[r] = gi < p.L ? p.dsum[bh * p.L + gi] : 0.f;
    }
}

// g = scale P (dP - D) with P = 2^(s - lse2) (0 where masked).
__device__ __forceinline__ void grad_scores(const BwdParams &p, const float (&s)[4][4],
                                            const float (&dp)[4][4], const float (&ls)[4],
                                            const float (&dd)[4], float (&P)[4][4],
                                            float (&g)[4][4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            P[r][c] = (s[r][c] == -INFINITY) ? 0.f : exp2f(s[r][c] - ls[r]);
            g[r][c] = p.scale * P[r][c] * (dp[r][c] - dd[r]);
        }
}

__device__ __forceinline__ float half_warp_max(float v)
{
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float half_warp_sum(float v)
{
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- stats: log2-sum-exp and D per query row --------------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_stats_kernel(const BwdParams p)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), i0 = blockIdx.y * T;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    TXL_CHECK(bh < (long long)p.B * p.H && i0 < p.L, p.status);
    stage_rows(sm, p, bh, h, i0);
    float m[4], l[4], wsum[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) m[r] = -INFINITY, l[r] = 0.f, wsum[r] = 0.f;
    // keys after M + (last row of the chunk) are hidden from every row
    const int jend = min(p.K, p.M + i0 + T);
    for (int j0 = 0; j0 < jend; j0 += T) {
        __syncthreads();
        stage(sm + OFF_A64, LD, T, p.k + bh * p.K * DH, j0, 1, p.K, nullptr);
        stage(sm + OFF_V64, LD, T, p.v + bh * p.K * DH, j0, 1, p.K, nullptr);
        stage_table_window(sm + OFF_W1, p, h, (long long)p.M + i0 - j0 - (T - 1));
        __syncthreads();
        float s[4][4], dp[4][4];
        key_tile_scores(sm, p, i0, j0, ty, tx, s, dp);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float tmax = fmaxf(fmaxf(s[r][0], s[r][1]), fmaxf(s[r][2], s[r][3]));
            tmax = half_warp_max(tmax);
            const float mn = fmaxf(m[r], tmax);
            // (every lane takes part in the sums; a row without a kept key so
            // far adds nothing)
            float e = 0.f, ed = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float x = (s[r][c] == -INFINITY) ? 0.f : exp2f(s[r][c] - mn);
                e += x;
                ed = fmaf(x, dp[r][c], ed);
            }
            e = half_warp_sum(e);
            ed = half_warp_sum(ed);
            if (mn != -INFINITY) {
                const float alpha = (m[r] == -INFINITY) ? 0.f : exp2f(m[r] - mn);
                l[r] = fmaf(l[r], alpha, e);
                wsum[r] = fmaf(wsum[r], alpha, ed);
                m[r] = mn;
            }
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int gi = i0 + ty * 4 + r;
            if (gi < p.L && l[r] > 0.f) {
                p.lse2[bh * p.L + gi] = m[r] + log2f(l[r]);
                p.dsum[bh * p.L + gi] = wsum[r] / l[r];
            }
        }
    }
}

// ---- dq, and the chunk's partials of du and dv_bias ---------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_dq_kernel(const BwdParams p)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), i0 = blockIdx.y * T;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    TXL_CHECK(bh < (long long)p.B * p.H && i0 < p.L, p.status);
    stage_rows(sm, p, bh, h, i0);
    float ls[4], dd[4];
    load_row_stats(p, bh, i0, ty, ls, dd);
    float dqc[4][4], dqp[4][4];  // content (k) and position (table) parts; rows i, columns t
    zero(dqc);
    zero(dqp);
    float *ga = sm + OFF_T1, *zw = sm + OFF_XS;
    const int jend = min(p.K, p.M + i0 + T);
    for (int j0 = 0; j0 < jend; j0 += T) {
        __syncthreads();
        stage(sm + OFF_A64, LD, T, p.k + bh * p.K * DH, j0, 1, p.K, nullptr);
        stage(sm + OFF_V64, LD, T, p.v + bh * p.K * DH, j0, 1, p.K, nullptr);
        stage_table_window(sm + OFF_W1, p, h, (long long)p.M + i0 - j0 - (T - 1));
        __syncthreads();
        float s[4][4], dp[4][4], P[4][4], g[4][4];
        key_tile_scores(sm, p, i0, j0, ty, tx, s, dp);
        grad_scores(p, s, dp, ls, dd, P, g);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) ga[(ty * 4 + r) * LD + tx + 16 * c] = g[r][c];
        __syncthreads();
        // g laid out by window column: zw[i][w] = g[i][i - w + 63] (zero where no key)
        for (int idx = threadIdx.x; idx < T * W; idx += THREADS) {
            const int i = idx / W, w = idx % W, j = i - w + T - 1;
            zw[i * LDW + w] = (j >= 0 && j < T) ? ga[i * LD + j] : 0.f;
        }
        __syncthreads();
        gemm_nn<4>(dqc, ga, LD, sm + OFF_A64, LD, T, ty, tx);
        gemm_nn<4>(dqp, zw, LDW, sm + OFF_W1, LD, W, ty, tx);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int gi = i0 + ty * 4 + r;
        if (gi < p.L) {
            float *dst = p.dq + (bh * p.L + gi) * DH;
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[tx + 16 * c] = dqc[r][c] + dqp[r][c];
        }
    }
    // du and dv_bias partials of this chunk: column sums of the two parts over
    // its rows (rows past L hold zeros), summed over ty in a fixed order.
    __syncthreads();
    float *red = sm + OFF_T1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        red[ty * 2 * DH + tx + 16 * c] = dqc[0][c] + dqc[1][c] + dqc[2][c] + dqc[3][c];
        red[ty * 2 * DH + DH + tx + 16 * c] = dqp[0][c] + dqp[1][c] + dqp[2][c] + dqp[3][c];
    }
    __syncthreads();
    if (threadIdx.x < 2 * DH) {
        float acc = 0.f;
        for (int y = 0; y < 16; ++y) acc += red[y * 2 * DH + threadIdx.x];
        p.part[(bh * gridDim.y + blockIdx.y) * 2 * DH + threadIdx.x] = acc;
    }
}

// ---- dk, dv per 64-key tile ----------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1) bwd_dkv_kernel(const BwdParams p)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const long long bh = blockIdx.x;
    const int h = (int)(bh % p.H), j0 = blockIdx.y * T;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    TXL_CHECK(bh < (long long)p.B * p.H && j0 < p.K, p.status);
    stage(sm + OFF_A64, LD, T, p.k + bh * p.K * DH, j0, 1, p.K, nullptr);
    stage(sm + OFF_V64, LD, T, p.v + bh * p.K * DH, j0, 1, p.K, nullptr);
    float dk[4][4], dv[4][4];  // rows: keys 4 ty + a; columns: dimensions
    zero(dk);
    zero(dv);
    float *pt = sm + OFF_T1, *gt = sm + OFF_T2;  // P and g transposed: [key][row]
    // the first chunk with a row that sees key j0 (distance M + i - j0 >= 0)
    const int i_first = max(0, j0 - p.M) / T * T;
    for (int i0 = i_first; i0 < p.L; i0 += T) {
        __syncthreads();
        stage_rows(sm, p, bh, h, i0);
        stage_table_window(sm + OFF_W1, p, h, (long long)p.M + i0 - j0 - (T - 1));
        __syncthreads();
        float ls[4], dd[4];
        load_row_stats(p, bh, i0, ty, ls, dd);
        float s[4][4], dp[4][4], P[4][4], g[4][4];
        key_tile_scores(sm, p, i0, j0, ty, tx, s, dp);
        grad_scores(p, s, dp, ls, dd, P, g);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                pt[(tx + 16 * c) * LD + ty * 4 + r] = P[r][c];
                gt[(tx + 16 * c) * LD + ty * 4 + r] = g[r][c];
            }
        __syncthreads();
        gemm_nn<4>(dv, pt, LD, sm + OFF_DO, LD, T, ty, tx);
        gemm_nn<4>(dk, gt, LD, sm + OFF_QU, LD, T, ty, tx);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int gj = j0 + ty * 4 + r;
        if (gj < p.K) {
            float *ok = p.dk + (bh * p.K + gj) * DH, *ov = p.dv + (bh * p.K + gj) * DH;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ok[tx + 16 * c] = dk[r][c];
                ov[tx + 16 * c] = dv[r][c];
            }
        }
    }
}

// ---- the table gradient per head and 64-distance tile ---------------------------
// Pair (row i, distance d) is key j = M + i - d.  Over the batch and the query
// chunks: position scores (q + v) . r_d directly; the content scores and dP
// through the chunk's 127-key window (key jmin + w, w = i - c + 63 for the
// tile's distance column c); then dr_d += sum_i g (q_i + v).
__global__ void __launch_bounds__(THREADS, 1) bwd_dr_kernel(const BwdParams p)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int d0 = blockIdx.x * T, h = blockIdx.y;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    TXL_CHECK(h < p.H && d0 < p.r_rows, p.status);
    float dr[4][4];  // rows: distances 4 ty + a; columns: dimensions
    zero(dr);
    if (d0 < p.K) {
        // the tile's table rows by distance: A64 row c = distance d0 + c
        stage(sm + OFF_A64, LD, T, p.r + (size_t)h * p.r_rows * DH, p.r_rows - 1 - d0, -1,
              p.r_rows, nullptr);
        float *xs = sm + OFF_XS, *gt = sm + OFF_T1;
        // chunks with a row that sees distance d0 (M + i - d0 >= 0 for its last row)
        const int i_first = max(0, d0 - p.M - (T - 1)) / T * T;
        for (int b = 0; b < p.B; ++b) {
            const long long bh = (long long)b * p.H + h;
            for (int i0 = i_first; i0 < p.L; i0 += T) {
                const long long jmin = (long long)p.M + i0 - d0 - (T - 1);
                __syncthreads();
                stage_rows(sm, p, bh, h, i0);
                stage(sm + OFF_W1, LD, W, p.k + bh * p.K * DH, jmin, 1, p.K, nullptr);
                stage(sm + OFF_W2, LD, W, p.v + bh * p.K * DH, jmin, 1, p.K, nullptr);
                __syncthreads();
                float ls[4], dd[4];
                load_row_stats(p, bh, i0, ty, ls, dd);
                float sp[4][4], sc[4][4], dp[4][4], x[4][8];
                zero(sp);
                gemm_nt<4>(sp, sm + OFF_QV, LD, sm + OFF_A64, LD, DH, ty, tx);
                zero(x);
                gemm_nt<8>(x, sm + OFF_QU, LD, sm + OFF_W1, LD, DH, ty, tx);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c) xs[(ty * 4 + r) * LDW + tx + 16 * c] = x[r][c];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int i = ty * 4 + r, cc = tx + 16 * c;
                        sc[r][c] = xs[i * LDW + i - cc + T - 1];
                    }
                __syncthreads();
                zero(x);
                gemm_nt<8>(x, sm + OFF_DO, LD, sm + OFF_W2, LD, DH, ty, tx);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c) xs[(ty * 4 + r) * LDW + tx + 16 * c] = x[r][c];
                __syncthreads();
                float s[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int i = ty * 4 + r, cc = tx + 16 * c;
                        dp[r][c] = xs[i * LDW + i - cc + T - 1];
                        const int gi = i0 + i, d = d0 + cc;
                        const int gj = p.M + gi - d;
                        const bool keep = gi < p.L && d < p.K && gj >= 0 && gj < p.K;
                        s[r][c] = keep ? (sc[r][c] + sp[r][c]) * p.scale_log2 : -INFINITY;
                    }
                float P[4][4], g[4][4];
                grad_scores(p, s, dp, ls, dd, P, g);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) gt[(tx + 16 * c) * LD + ty * 4 + r] = g[r][c];
                __syncthreads();
                gemm_nn<4>(dr, gt, LD, sm + OFF_QV, LD, T, ty, tx);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = d0 + ty * 4 + r;
        if (d < p.r_rows) {
            float *dst = p.dr + ((size_t)h * p.r_rows + (p.r_rows - 1 - d)) * DH;
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[tx + 16 * c] = dr[r][c];
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

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

} // namespace

size_t bwd_workspace_bytes(int B, int H, int L)
{
    if (B <= 0 || H <= 0 || L <= 0) return 0;
    const size_t rows = (size_t)B * H * L;
    const size_t chunks = (size_t)B * H * ((L + T - 1) / T);
    return 2 * align256(rows * sizeof(float)) + align256(chunks * 2 * DH * sizeof(float));
}

cudaError_t launch_relattn_bwd(const BwdParams &p, cudaStream_t s)
{
    static bool attr_set[64] = {};  // the attributes are set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        for (const void *f : {(const void *)bwd_stats_kernel, (const void *)bwd_dq_kernel,
                              (const void *)bwd_dkv_kernel, (const void *)bwd_dr_kernel})
            if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          SMEM_BYTES)) != cudaSuccess)
                return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const long long BH = (long long)p.B * p.H;
    const int n_chunks = (p.L + T - 1) / T, n_keys = (p.K + T - 1) / T;
    const int n_dist = (p.r_rows + T - 1) / T;
    if (BH > 0x7fffffffLL || n_chunks > 65535 || n_keys > 65535 || p.H > 65535)
        return cudaErrorInvalidValue;
    bwd_stats_kernel<<<dim3((unsigned)BH, n_chunks), THREADS, SMEM_BYTES, s>>>(p);
    bwd_dq_kernel<<<dim3((unsigned)BH, n_chunks), THREADS, SMEM_BYTES, s>>>(p);
    bwd_dkv_kernel<<<dim3((unsigned)BH, n_keys), THREADS, SMEM_BYTES, s>>>(p);
    bwd_dr_kernel<<<dim3((unsigned)n_dist, p.H), THREADS, SMEM_BYTES, s>>>(p);
    bwd_bias_kernel<<<p.H, 2 * DH, 0, s>>>(p, n_chunks);
    return cudaGetLastError();
}

} // namespace txl
