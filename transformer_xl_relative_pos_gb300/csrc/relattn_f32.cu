// fp32 CUDA-core forward kernel for Transformer-XL relative-position attention.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.3: A_ij = (q_i + u).k_j + (q_i + v).W_kR R_{i-j}, masked softmax over the
// extended context (memory rows first), times v.  The relative vector of pair
// (i, j) is row r_rows-1-(M+i-j) of the reversed table (Appendix B's Q), read
// by index arithmetic.
//
// This is the exact-fp32 path (FFMA, no TF32): one thread per query row, keys
// and values staged through shared memory 32 at a time, online softmax in fp32.
#include "kernels.h"

namespace txl {
namespace {

constexpr int DH = 64;
constexpr int ROWS = 64;   // query rows per block (one per thread)
constexpr int KT = 32;     // keys per shared-memory tile

__global__ void __launch_bounds__(ROWS)
    relattn_fwd_f32_kernel(const F32Params p)
{
    __shared__ float ks[KT][DH];
    __shared__ float vs[KT][DH];
    const int bh = blockIdx.x;
    const int h = bh % p.H;
    const int row0 = blockIdx.y * ROWS;
    const int i = row0 + threadIdx.x;
    const bool active = i < p.L;
    const int K = p.K;

    float qu[DH], qv[DH], o[DH];
    const float *qrow = p.q + ((size_t)bh * p.L + (active ? i : 0)) * DH;
#pragma unroll
    for (int t = 0; t < DH; ++t) {
        const float qq = active ? qrow[t] : 0.f;
        qu[t] = qq + p.u[h * DH + t];
        qv[t] = qq + p.vb[h * DH + t];
        o[t] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    // Keys visible to the last row of this block.
    const int last_row = min(p.L - 1, row0 + ROWS - 1);
    const int jend = min(K, p.M + last_row + 1);
    const float *kbase = p.k + (size_t)bh * p.kv_stride;
    const float *vbase = p.v + (size_t)bh * p.kv_stride;
    const float *rbase = p.r + (size_t)h * p.r_rows * DH;

    for (int j0 = 0; j0 < jend; j0 += KT) {
        __syncthreads();
        for (int e = threadIdx.x; e < KT * DH; e += ROWS) {
            const int jj = e / DH, t = e % DH;
            const int j = j0 + jj;
            ks[jj][t] = (j < K) ? kbase[(size_t)j * DH + t] : 0.f;
            vs[jj][t] = (j < K) ? vbase[(size_t)j * DH + t] : 0.f;
        }
        __syncthreads();
        if (!active) continue;
        for (int jj = 0; jj < KT; ++jj) {
            const int j = j0 + jj;
            const int delta = p.M + i - j;
            if (j >= K || delta < 0) break;  // keys are visited in increasing j
            const float *rr = rbase + (size_t)(p.r_rows - 1 - delta) * DH;
            float s = 0.f;
#pragma unroll
            for (int t = 0; t < DH; ++t) s = fmaf(qu[t], ks[jj][t], s);
#pragma unroll
            for (int t = 0; t < DH; ++t) s = fmaf(qv[t], __ldg(rr + t), s);
            s *= p.scale;
            if (s > m) {
                const float corr = expf(m - s);  // 0 when m is -inf
                l *= corr;
#pragma unroll
                for (int t = 0; t < DH; ++t) o[t] *= corr;
                m = s;
            }
            const float w = expf(s - m);
            l += w;
#pragma unroll
            for (int t = 0; t < DH; ++t) o[t] = fmaf(w, vs[jj][t], o[t]);
        }
    }
    if (!active) return;
    const float inv = 1.f / l;
    float *orow = p.out + ((size_t)bh * p.L + i) * DH;
#pragma unroll
    for (int t = 0; t < DH; ++t) orow[t] = o[t] * inv;
    if (p.lse) p.lse[(size_t)bh * p.L + i] = m + logf(l);
}

} // namespace

cudaError_t launch_relattn_f32(const F32Params &p, cudaStream_t s)
{
    const long long rb = (p.L + ROWS - 1) / ROWS;
    if (rb > 65535 || (long long)p.B * p.H > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid((unsigned)(p.B * p.H), (unsigned)rb);
    relattn_fwd_f32_kernel<<<grid, ROWS, 0, s>>>(p);
    return cudaGetLastError();
}

} // namespace txl
