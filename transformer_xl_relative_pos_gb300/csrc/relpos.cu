// Sinusoid relative-position table R for Transformer-XL.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.3: R is a sinusoid encoding matrix without learnable parameters whose row
// p encodes a relative distance of p; Appendix B orders the rows by decreasing
// distance (Q_k uses R_{M+L-1-k}).  Output row rho holds distance p = K-1-rho:
//   R[rho][2k] = sin(p w_k),  R[rho][2k+1] = cos(p w_k),  w_k = 10000^(-2k/d).
//
// Accuracy: the angle p*w_k reaches K radians, so it is formed in
// double-float (w_k split into two floats, computed on the host in long double),
// reduced modulo 2*pi by Cody and Waite's method (W. J. Cody, W. Waite,
// "Software Manual for the Elementary Functions", 1980) with 2*pi split into
// three floats, and only then passed to sincosf.  The split used here was
// derived from a 50-digit value of 2*pi: C1 and C2 keep 8 significant bits each
// so that n*C1 and n*C2 are exact for n < 2^16 (angles below ~4e5 rad).
#include <cmath>

#include "kernels.h"

namespace txl {
namespace {

constexpr float kTwoPiC1 = 6.28125f;                   // 0x1.92p+2
constexpr float kTwoPiC2 = 0x1.fap-10f;                // 0.00193023681640625
constexpr float kTwoPiC3 = 0x1.54442ep-18f;            // 5.0703634e-06
constexpr float kInvTwoPi = 0x1.45f306p-3f;            // 1/(2 pi) rounded to fp32
constexpr int kMaxHalf = 2048;                         // frequencies passed by value

// w_k = 10000^(-2k/d) as (hi, lo) floats, computed on the host in long double.
struct Freqs {
    float2 w[kMaxHalf];
};

__device__ __forceinline__ float2 sincos_pw(float pf, float whi, float wlo)
{
    // angle = p * (whi + wlo) as a_hi + a_lo (p exact: p < 2^24)
    const float a_hi = pf * whi;
    const float a_lo = fmaf(pf, wlo, fmaf(pf, whi, -a_hi));
    const float n = rintf(a_hi * kInvTwoPi);
    float r = fmaf(-n, kTwoPiC1, a_hi);
    r = fmaf(-n, kTwoPiC2, r);
    r += a_lo;
    r = fmaf(-n, kTwoPiC3, r);
    float sn, cs;
    sincosf(r, &sn, &cs);
    return make_float2(sn, cs);
}

__device__ __forceinline__ void store_pair(void *R, size_t pair, float2 v, int bf16)
{
    if (bf16)
        reinterpret_cast<__nv_bfloat162 *>(R)[pair] = __floats2bfloat162_rn(v.x, v.y);
    else
        reinterpret_cast<float2 *>(R)[pair] = v;
}

// Block = 64 frequency pairs x 4 rows of threads, covering 32 rows.  The
// block's 64 frequencies are staged from the parameter bank into shared memory
// once (parameter-bank reads are fast only when a warp reads one address).
constexpr int kPairsPerBlock = 64;
constexpr int kRowsPerTile = 32;
__global__ void __launch_bounds__(256)
    rel_pos_emb_kernel(void *R, int K, int half, int bf16, const __grid_constant__ Freqs f)
{
    __shared__ float2 w[kPairsPerBlock];
    const int k0 = blockIdx.x * kPairsPerBlock;
    const int tk = threadIdx.x % kPairsPerBlock;
    const int tr = threadIdx.x / kPairsPerBlock;  // 0..3
    if (threadIdx.x < kPairsPerBlock && k0 + threadIdx.x < half) w[threadIdx.x] = f.w[k0 + threadIdx.x];
    __syncthreads();
    const int k = k0 + tk;
    if (k >= half) return;
    const float2 wk = w[tk];
    const int rho0 = blockIdx.y * kRowsPerTile;
#pragma unroll 4
    for (int r = tr; r < kRowsPerTile; r += 4) {
        const int rho = rho0 + r;
        if (rho >= K) break;
        store_pair(R, (size_t)rho * half + k, sincos_pw((float)(K - 1 - rho), wk.x, wk.y), bf16);
    }
}

// Widths beyond the by-value table: each block derives the frequencies in fp64.
constexpr int kRowsPerBlock = 16;
__global__ void rel_pos_emb_wide_kernel(void *R, int K, int d, int bf16)
{
    extern __shared__ float w_split[];  // [d/2] high parts, then [d/2] low parts
    const int half = d / 2;
    float *whi = w_split;
    float *wlo = w_split + half;
    const double ln1e4 = 9.210340371976184;  // ln(10000)
    for (int k = threadIdx.x; k < half; k += blockDim.x) {
        const double w = exp(-(2.0 * k / d) * ln1e4);
        const float hi = (float)w;
        whi[k] = hi;
        wlo[k] = (float)(w - (double)hi);
    }
    __syncthreads();
    const int rho0 = blockIdx.x * kRowsPerBlock;
    const int rows = min(kRowsPerBlock, K - rho0);
    for (int e = threadIdx.x; e < rows * half; e += blockDim.x) {
        const int rho = rho0 + e / half;
        const int k = e % half;
        store_pair(R, (size_t)rho * half + k, sincos_pw((float)(K - 1 - rho), whi[k], wlo[k]),
                   bf16);
    }
}

} // namespace

cudaError_t launch_rel_pos_emb(void *R, int K, int d_model, bool bf16, cudaStream_t s)
{
    const int half = d_model / 2;
    if (half <= kMaxHalf) {
        // The table depends on d_model only; keep the last one per host thread.
        thread_local Freqs f;
        thread_local int f_d = 0;
        if (f_d != d_model) {
            for (int k = 0; k < half; ++k) {
                const long double w =
                    powl(10000.0L, -2.0L * (long double)k / (long double)d_model);
                const float hi = (float)w;
                f.w[k] = make_float2(hi, (float)(w - (long double)hi));
            }
            f_d = d_model;
        }
        const dim3 grid((half + kPairsPerBlock - 1) / kPairsPerBlock,
                        (K + kRowsPerTile - 1) / kRowsPerTile);
        if (grid.y > 65535u) return cudaErrorInvalidValue;
        rel_pos_emb_kernel<<<grid, 256, 0, s>>>(R, K, half, bf16 ? 1 : 0, f);
        return cudaGetLastError();
    }
    const int blocks = (K + kRowsPerBlock - 1) / kRowsPerBlock;
    const size_t shm = sizeof(float) * (size_t)d_model;
    if (shm > 48 * 1024) return cudaErrorInvalidValue;
    rel_pos_emb_wide_kernel<<<blocks, 256, shm, s>>>(R, K, d_model, bf16 ? 1 : 0);
    return cudaGetLastError();
}

} // namespace txl
