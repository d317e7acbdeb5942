// Device code shared by the two short-segment (decode) kernels: the
// fp32-on-CUDA-cores kernel (relattn_decode.cu) and the tensor-core kernel
// (relattn_decode_mma.cu).  Both split a head's keys into ranges of whole
// 32-key chunks, deal a block's chunks to its four warps in turn, and end the
// same way: every warp leaves its running maximum, sum and unnormalised output
// per query row in a record, the block merges its warps' records, and then
// either writes the output, or its range's normalised partial and
// log2-sum-exp for the merge kernel, or merges the ranges of its head inside
// the thread-block cluster.
#pragma once

#include "kernels.h"
#include "decode.h"
#include "ptx.cuh"

namespace txl {
namespace decode {

using namespace ptx;

constexpr int DH = kTcDH;         // 64
constexpr int WARPS = 4;          // warps per block
constexpr int GK = 32;            // keys per chunk
constexpr int LMAX = kDecodeMaxL;
constexpr int ROWB = DH * 2;      // bytes of one bf16 row

// One warp's result for the block merge, per query row: running maximum (log2
// units), sum of probabilities and the unnormalised output.
struct WarpRec {
    float m[LMAX];
    float l[LMAX];
    float a[LMAX][DH];
};

// The block's merged result per row, kept in shared memory for the cluster
// merge: normalised output and log2-sum-exp.
struct BlockRes {
    float o[LMAX][DH];
    float lse[LMAX];
};

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Thread-block cluster: the key ranges of one head run as one cluster and merge
// through distributed shared memory.
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every block of the cluster: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
                 : "memory");
    return v;
}

// Key range of block `split` of a head: [k_begin, k_end), and how many of its
// chunks warp `warp` takes (chunk c goes to warp c mod WARPS).
struct Range {
    int k_begin, k_end, n_mine;
};

__device__ __forceinline__ Range key_range(int K, int n_splits, int split, int warp)
{
    const int span = decode_span(K, n_splits);
    Range r;
    r.k_begin = split * span;
    r.k_end = min(K, r.k_begin + span);
    const int n_chunks = (r.k_end > r.k_begin) ? (r.k_end - r.k_begin + GK - 1) / GK : 0;
    r.n_mine = (n_chunks > warp) ? (n_chunks - warp + WARPS - 1) / WARPS : 0;
    return r;
}

// Every thread of the block, after each warp wrote its record (warp w's at
// rec(w)): merge the warps, out = sum_w 2^(m_w - max) a_w / sum_w 2^(m_w - max) l_w,
// then write the output, the range's partial, or (cluster launch) merge the
// head's ranges in block 0 of the cluster.  Every block reaches both cluster
// barriers: no thread leaves the kernel before this.
template <int L, typename RecOf>
__device__ __forceinline__ void finish_block(RecOf rec, BlockRes *res, const DecodeParams &p,
                                             int bh, int split, int warp, int lane)
{
    __syncthreads();
    for (int i = warp; i < L; i += WARPS) {
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mx = fmaxf(mx, rec(w)->m[i]);
        float ls = 0.f, o0 = 0.f, o1 = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float mw = rec(w)->m[i];
                if (mw == -INFINITY) continue;
                const float sw = ex2f(mw - mx);
                ls += sw * rec(w)->l[i];
                const float2 aw = reinterpret_cast<const float2 *>(rec(w)->a[i])[lane];
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
        } else if (p.cluster) {
            // this key range's normalised partial stays in shared memory
            reinterpret_cast<float2 *>(res->o[i])[lane] = make_float2(o0 * inv, o1 * inv);
            if (lane == 0) res->lse[i] = lse2;
        } else {
            const size_t prow = (size_t)split * p.B * p.H * L + row;
            reinterpret_cast<float2 *>(p.part_o + prow * DH)[lane] = make_float2(o0 * inv, o1 * inv);
            if (lane == 0) p.part_lse[prow] = lse2;
        }
    }
    if (p.cluster) {
        // The key ranges of this head are the blocks of one cluster (rank =
        // range): block 0 merges their partials through distributed shared
        // memory, out = sum_r 2^(lse_r - max) o_r / sum_r 2^(lse_r - max).
        cluster_sync();
        if (cluster_rank() == 0) {
            for (int i = warp; i < L; i += WARPS) {
                const uint32_t a_lse = smem_u32(&res->lse[i]);
                const uint32_t a_o = smem_u32(&res->o[i][2 * lane]);
                float mx = -INFINITY;
                for (int r = 0; r < p.n_splits; ++r)
                    mx = fmaxf(mx, ld_cluster_f32(cluster_addr(a_lse, (uint32_t)r)));
                float wsum = 0.f, c0 = 0.f, c1 = 0.f;
                if (mx != -INFINITY) {
                    for (int r = 0; r < p.n_splits; ++r) {
                        const float lr = ld_cluster_f32(cluster_addr(a_lse, (uint32_t)r));
                        if (lr == -INFINITY) continue;  // a range without keys
                        const float w = ex2f(lr - mx);
                        const float2 o = ld_cluster_f32x2(cluster_addr(a_o, (uint32_t)r));
                        wsum += w;
                        c0 = fmaf(w, o.x, c0);
                        c1 = fmaf(w, o.y, c1);
                    }
                }
                const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
                const size_t row = (size_t)bh * L + i;
                reinterpret_cast<__nv_bfloat162 *>(p.out + row * DH)[lane] =
                    __floats2bfloat162_rn(c0 * inv, c1 * inv);
                if (p.lse && lane == 0)
                    p.lse[row] = (wsum > 0.f) ? (mx + __log2f(wsum)) * 0.69314718055994531f
                                              : -INFINITY;
            }
        }
        cluster_sync();  // block 0 has read the others' shared memory
    }
}

} // namespace decode
} // namespace txl
