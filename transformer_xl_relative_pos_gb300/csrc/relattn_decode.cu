// Relative-position attention for short segments (L <= 3 queries) against a
// long memory: the decode pattern of generation, one or a few new tokens per
// step attending to the cached M states ("Transformer-XL: Attentive Language
// Models Beyond a Fixed-Length Context", §3.2 recurrence and evaluation with a
// long memory, §3.3 score, Appendix B reversed table).
//
// With so few query rows the work is reading K, V and the table once: the
// kernel is HBM-bound and runs on the CUDA cores in fp32.  Every warp works on
// its own: it takes 32 keys at a time, and lane l holds dimensions 2l and 2l+1
// of those keys' k and v rows and of the L + 31 table rows they need, read
// straight from global memory (one 128-byte line per row and warp).  For query
// row i and key j the score is
//   A_ij = (q_i + u).k_j + (q_i + v).r[r_off + L-1 - i + j]        (j <= M + i)
// where r is the reversed table (row K-1-d holds distance d; r_off = r_rows-K):
// the Appendix B left shift by L-1-i is the table row index.  q + u and q + v
// are formed in fp32 and never rounded.  Each lane sums its two dimensions of
// all 32 keys; a transposing butterfly over the warp leaves lane l with the
// whole score of key l.  Online softmax per row, P.V with the probabilities
// broadcast by shuffles, then the block's warps merge their partial results
// and the block writes the output, or its key range's normalised partial and
// log2-sum-exp for the merge kernel.  The per-key work grows with L while the
// bytes do not: from L = 4 on the tensor-core kernel is the faster path.
#include "kernels.h"
#include "ptx.cuh"

namespace txl {
namespace {

constexpr int DH = kTcDH;         // 64: lane l owns dimensions 2l, 2l+1
constexpr int WARPS = 4;          // warps per block
constexpr int GK = 32;            // keys per warp step
constexpr int LMAX = kDecodeMaxL;

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Lane l holds v[0..31], its share of 32 sums; afterwards lane l holds the whole
// sum number l.  Five butterfly stages: a lane keeps the half of its values
// whose index bit matches its own lane bit and sends the other half.
__device__ __forceinline__ float transpose_reduce(float (&v)[GK], int lane)
{
#pragma unroll
    for (int o = GK / 2; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < o; ++k) {
            const float keep = up ? v[k + o] : v[k];
            const float send = up ? v[k] : v[k + o];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

template <int L>
__global__ void __launch_bounds__(WARPS * 32) relattn_decode_kernel(const DecodeParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.n_splits;
    const int bh = blockIdx.x / p.n_splits;
    const int h = bh % p.H;
    const int K = p.K;
    // Key range of this block: a whole number of warp steps.
    const int span = ((K + p.n_splits - 1) / p.n_splits + WARPS * GK - 1) / (WARPS * GK) * (WARPS * GK);
    const int k_begin = split * span, k_end = min(K, k_begin + span);

    const uint32_t *kw = reinterpret_cast<const uint32_t *>(p.k) + (size_t)bh * K * (DH / 2) + lane;
    const uint32_t *vw = reinterpret_cast<const uint32_t *>(p.v) + (size_t)bh * K * (DH / 2) + lane;
    const uint32_t *rw = reinterpret_cast<const uint32_t *>(p.r) + (size_t)h * p.r_rows * (DH / 2) + lane;

    // q + u and q + v, this lane's two dimensions, every row.
    float qu0[L], qu1[L], qv0[L], qv1[L];
    {
        const uint32_t uu = reinterpret_cast<const uint32_t *>(p.u)[h * (DH / 2) + lane];
        const uint32_t vv = reinterpret_cast<const uint32_t *>(p.vb)[h * (DH / 2) + lane];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const uint32_t qq = reinterpret_cast<const uint32_t *>(p.q)[((size_t)bh * L + i) * (DH / 2) + lane];
            qu0[i] = lo_f(qq) + lo_f(uu);
            qu1[i] = hi_f(qq) + hi_f(uu);
            qv0[i] = lo_f(qq) + lo_f(vv);
            qv1[i] = hi_f(qq) + hi_f(vv);
        }
    }

    float m[L], l[L], a0[L], a1[L];  // running max (log2 units) and sum; output dims 2l, 2l+1
#pragma unroll
    for (int i = 0; i < L; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
        a0[i] = 0.f;
        a1[i] = 0.f;
    }

    for (int j0 = k_begin + warp * GK; j0 < k_end; j0 += WARPS * GK) {
        // ---- this lane's dimensions of the 32 keys and their table rows ----
        uint32_t kk[GK], vv[GK], rr[GK + L - 1];
#pragma unroll
        for (int e = 0; e < GK; ++e) {
            const int j = min(j0 + e, K - 1);  // rows past K are loaded clamped and masked
            kk[e] = __ldcs(kw + (size_t)j * (DH / 2));
            vv[e] = __ldcs(vw + (size_t)j * (DH / 2));
        }
        // table rows r_off + j0 + e, e in [0, 32 + L - 1): row for (i, j) is e = j - j0 + L-1-i
#pragma unroll
        for (int e = 0; e < GK + L - 1; ++e) {
            const int row = min(p.r_off + j0 + e, p.r_rows - 1);
            rr[e] = __ldg(rw + (size_t)row * (DH / 2));
        }

#pragma unroll
        for (int i = 0; i < L; ++i) {
            // ---- scores of row i for the 32 keys -----------------------------
            float part[GK];
#pragma unroll
            for (int e = 0; e < GK; ++e) {
                const uint32_t r2 = rr[e + (L - 1 - i)];
                part[e] = fmaf(qu0[i], lo_f(kk[e]),
                               fmaf(qu1[i], hi_f(kk[e]),
                                    fmaf(qv0[i], lo_f(r2), qv1[i] * hi_f(r2))));
            }
            float s = transpose_reduce(part, lane) * p.scale_log2;  // key j0 + lane
            const int j = j0 + lane;
            if (j >= k_end || j > p.M + i) s = -INFINITY;
            // ---- online softmax -------------------------------------------------
            float mx = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_new = fmaxf(m[i], mx);
            if (m_new == -INFINITY) continue;  // nothing visible yet (warp-uniform)
            const float sc = (m[i] == -INFINITY) ? 0.f : ex2f(m[i] - m_new);
            const float pj = (s == -INFINITY) ? 0.f : ex2f(s - m_new);
            float sum = pj;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            m[i] = m_new;
            l[i] = l[i] * sc + sum;
            float b0 = a0[i] * sc, b1 = a1[i] * sc;
            // ---- P.V: probability of key e from lane e -------------------------
#pragma unroll
            for (int e = 0; e < GK; ++e) {
                const float pe = __shfl_sync(0xffffffffu, pj, e);
                b0 = fmaf(pe, lo_f(vv[e]), b0);
                b1 = fmaf(pe, hi_f(vv[e]), b1);
            }
            a0[i] = b0;
            a1[i] = b1;
        }
    }

    // ---- merge the block's warps: w = 2^(m_w - max), out = sum w a / sum w l ----
    __shared__ float sm_m[WARPS][LMAX], sm_l[WARPS][LMAX];
    __shared__ float2 sm_a[WARPS][LMAX][32];
#pragma unroll
    for (int i = 0; i < L; ++i) {
        if (lane == 0) {
            sm_m[warp][i] = m[i];
            sm_l[warp][i] = l[i];
        }
        sm_a[warp][i][lane] = make_float2(a0[i], a1[i]);
    }
    __syncthreads();
    for (int i = warp; i < L; i += WARPS) {
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mx = fmaxf(mx, sm_m[w][i]);
        float ls = 0.f, o0 = 0.f, o1 = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float mw = sm_m[w][i];
                if (mw == -INFINITY) continue;
                const float sw = ex2f(mw - mx);
                ls += sw * sm_l[w][i];
                const float2 aw = sm_a[w][i][lane];
                o0 = fmaf(sw, aw.x, o0);
                o1 = fmaf(sw, aw.y, o1);
            }
        }
        const float inv = (ls > 0.f) ? 1.f / ls : 0.f;
        const float lse2 = (ls > 0.f) ? mx + __log2f(ls) : -INFINITY;
        const size_t row = (size_t)bh * L + i;
        if (p.n_splits == 1) {
            reinterpret_cast<__nv_bfloat162 *>(p.out + row * DH)[lane] =
                __floats2bfloat162_rn(o0 * inv, o1 * inv);
            if (p.lse && lane == 0) p.lse[row] = lse2 * 0.69314718055994531f;
        } else {
            const size_t prow = (size_t)split * p.B * p.H * L + row;
            reinterpret_cast<float2 *>(p.part_o + prow * DH)[lane] = make_float2(o0 * inv, o1 * inv);
            if (lane == 0) p.part_lse[prow] = lse2;
        }
    }
}

template <int L>
cudaError_t launch_l(const DecodeParams &p, cudaStream_t s)
{
    const long long blocks = (long long)p.B * p.H * p.n_splits;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    relattn_decode_kernel<L><<<(unsigned)blocks, WARPS * 32, 0, s>>>(p);
    return cudaGetLastError();
}

} // namespace

int decode_keys_per_block() { return WARPS * GK; }

cudaError_t launch_relattn_decode(const DecodeParams &p, cudaStream_t s)
{
    switch (p.L) {
    case 1: return launch_l<1>(p, s);
    case 2: return launch_l<2>(p, s);
    case 3: return launch_l<3>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace txl
