// Projection of a segment's hidden states into per-head q, k, v, written where
// the attention reads them, with the memory update in the same launch
// ("Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
// §3.3 N-layer summary: q = h W_q^T, k = h~ W_kE^T, v = h~ W_v^T; §3.2: the
// memory takes the newest states).  With the memory's keys and values cached
// in a window (only the segment's rows are projected), one layer's
// projections are a single GEMM  Y = h W^T  over the stacked weights
// W = [W_q ; W_kE ; W_v]; its epilogue scatters Y's columns by output and head
// into q [B][H][L][64] and into the rows behind the memory in the k / v
// window planes, and the first column of blocks also copies h into the
// memory ring.  This replaces a library GEMM, a head-major permutation copy, the
// window append and the ring update.
//
// GEMM: tcgen05 (bf16 in, fp32 accumulate in TMEM), 128 x 256 tiles, K in
// 64-column slices through a 4-stage ring of TMA copies (128-byte swizzle):
//   warp 0      TMA producer
//   warp 1      MMA issuer (converged warp, one elected lane issues)
//   warp 2      TMEM allocator
//   warps 4..7  ring copy of the tile's h rows while the MMAs run (first
//               column of blocks), then the epilogue: thread = row, 32
//               columns per TMEM load, bf16 rows of 64 stored per head
// Every barrier wait is bounded, as in the attention kernels.
#include "kernels.h"
#include "ptx.cuh"

namespace txl {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64, NS = 4;
constexpr int A_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_BYTES = BN * BK * 2;                 // 32 KB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int OFF_BAR = NS * STAGE;
constexpr int N_BAR = 2 * NS + 1;
constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;         // slack for the manual alignment
constexpr uint32_t TM_COLS = 256;

static_assert(A_BYTES % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");

__global__ void __launch_bounds__(256, 1)
    project_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                   const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int kb_n = (p.K + BK - 1) / BK;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *empty = full + NS;
    uint64_t *acc_full = empty + NS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint64_t wait_ns = p.wait_ns;

    if (warp == 0) {
        // ===================== TMA producer =====================================
        if (lane == 0) {
            prefetch_tensormap(&tm_h);
            prefetch_tensormap(&tm_w);
            bool ok = true;
            int issued = 0;
            for (int kb = 0; kb < kb_n; ++kb) {
                const int s = kb % NS;
                if (!(ok = mbar_wait(empty + s, ((kb / NS) & 1) ^ 1, abort_flag, wait_ns))) break;
                uint8_t *st = smem + s * STAGE;
                mbar_arrive_expect_tx(full + s, STAGE);
                tma_load_3d(st, &tm_h, full + s, kb * BK, m0, 0);
                tma_load_3d(st + A_BYTES, &tm_w, full + s, kb * BK, n0, 0);
                issued = kb + 1;
            }
            if (!ok) {
                atomicOr(p.status, TXL_STATUS_TIMEOUT);
                *abort_flag = 1;
                const int zero = 0;
                for (int kb = max(0, issued - NS); kb < issued; ++kb)
                    mbar_wait(full + kb % NS, (kb / NS) & 1, &zero, wait_ns);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =======================================
        constexpr uint32_t ID = idesc_bf16_f32(BM, BN, false);
        const uint64_t dA = sdesc_sw128(smem_u32(smem));
        const uint64_t dB = sdesc_sw128(smem_u32(smem + A_BYTES));
        auto elect = []() -> bool {
            uint32_t el;
            asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
                         : "=r"(el));
            return el != 0;
        };
        bool ok = true;
        for (int kb = 0; kb < kb_n && ok; ++kb) {
            const int s = kb % NS;
            ok = __all_sync(0xffffffffu, mbar_wait(full + s, (kb / NS) & 1, abort_flag, wait_ns));
            if (!ok) break;
            tc_fence_after_sync();
            const uint64_t off = (uint64_t)((s * STAGE) >> 4);
            if (elect()) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16_ss(tmem, dA + off + kk * 2, dB + off + kk * 2, ID,
                                (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit(empty + s);
            }
            __syncwarp();
        }
        // On success the accumulator is complete once acc_full fires; on a
        // time-out the commit still lets the issued MMAs drain before TMEM is
        // freed (the epilogue waits on it with the abort flag ignored).
        if (elect()) mma_commit(acc_full);
        __syncwarp();
        if (!ok && lane == 0) {
            atomicOr(p.status, TXL_STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp >= 4) {
        const int wq = warp - 4;               // TMEM lane quarter
        const int row = wq * 32 + lane;        // row of the tile
        const int m = m0 + row;
        // ---- the memory update, while the MMAs run --------------------------
        // mem[b][(head + l) mod cap] = h[b][l] for l >= first_row; each warp
        // copies its 32 rows, a row at a time with 16-byte vectors over the lanes.
        if (p.mem && blockIdx.y == 0) {
            const int row_vec = p.K / 8;       // 16-byte vectors of a row
            for (int r = 0; r < 32; ++r) {
                const int mr = m0 + wq * 32 + r;
                if (mr >= p.M) break;
                const int b = mr / p.L, l = mr - b * p.L;
                if (l < p.mem_first) continue;
                const long long slot = (long long)b * p.mem_cap + (p.mem_head + l) % p.mem_cap;
                TXL_CHECK(b < p.B && l < p.L && slot < (long long)p.B * p.mem_cap, p.status);
                const uint4 *src = reinterpret_cast<const uint4 *>(p.h) + (long long)mr * row_vec;
                uint4 *dst = reinterpret_cast<uint4 *>(p.mem) + slot * row_vec;
                for (int c = lane; c < row_vec; c += 32) dst[c] = __ldcs(src + c);
            }
        }
        // ---- epilogue: Y rows into q and the k / v window planes ---------------
        const int zero = 0;
        const bool got = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, &zero, wait_ns));
        if (!got) {
            if (lane == 0) atomicOr(p.status, TXL_STATUS_TIMEOUT);
        } else if (!*abort_flag) {
            tc_fence_after_sync();
            const uint32_t tq = tmem + ((uint32_t)(wq * 32) << 16);
            const int b = m / p.L, l = m - b * p.L;
            const int per_out = p.H * 64;      // columns of one output
#pragma unroll 1
            for (int g = 0; g < BN / 64; ++g) {
                const int n = n0 + g * 64;     // first column of this head's group
                if (n >= p.N) break;           // (warp-uniform)
                uint32_t r0[32], r1[32];
                tmem_ld32(tq + g * 64, r0);
                tmem_ld32(tq + g * 64 + 32, r1);
                tmem_ld_wait(r0);
                tmem_ld_wait(r1);
                if (m < p.M) {
                    const int o = n / per_out, hd = (n - o * per_out) / 64;
                    const long long plane = (long long)b * p.H + hd;
                    // element offset: the plane (plane_stride elements apart), then
                    // the row (64 elements)
                    const long long dst_off = plane * p.plane_stride[o] + (long long)(p.row0[o] + l) * 64;
                    TXL_CHECK(o < p.n_out && hd < p.H && b < p.B &&
                                  (long long)(p.row0[o] + l + 1) * 64 <= p.plane_stride[o],
                              p.status);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out[o] + dst_off);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]), __uint_as_float(r0[8 * c + 1])),
                                            pack_bf16x2(__uint_as_float(r0[8 * c + 2]), __uint_as_float(r0[8 * c + 3])),
                                            pack_bf16x2(__uint_as_float(r0[8 * c + 4]), __uint_as_float(r0[8 * c + 5])),
                                            pack_bf16x2(__uint_as_float(r0[8 * c + 6]), __uint_as_float(r0[8 * c + 7])));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[4 + c] = make_uint4(pack_bf16x2(__uint_as_float(r1[8 * c]), __uint_as_float(r1[8 * c + 1])),
                                                pack_bf16x2(__uint_as_float(r1[8 * c + 2]), __uint_as_float(r1[8 * c + 3])),
                                                pack_bf16x2(__uint_as_float(r1[8 * c + 4]), __uint_as_float(r1[8 * c + 5])),
                                                pack_bf16x2(__uint_as_float(r1[8 * c + 6]), __uint_as_float(r1[8 * c + 7])));
                }
            }
        }
        tc_fence_before_sync();
    }

    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TM_COLS);
    }
}

} // namespace

int project_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_project(const CUtensorMap &tm_h, const CUtensorMap &tm_w, const ProjParams &p,
                           cudaStream_t s)
{
    static bool attr_set[64] = {};  // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const dim3 grid((unsigned)((p.M + BM - 1) / BM), (unsigned)((p.N + BN - 1) / BN));
    project_kernel<<<grid, 256, SMEM_BYTES, s>>>(tm_h, tm_w, p);
    return cudaGetLastError();
}

} // namespace txl
