// Tensor-core (tcgen05 + TMEM + TMA) forward kernel for Transformer-XL
// relative-position attention, bf16 operands, fp32 accumulation.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context":
//   §3.3 score  A_ij = (q_i + u).k_j + (q_i + v).W_kR R_{i-j}
//   §3.3 summary: masked softmax over the extended context, times v
//   Appendix B: with the reversed table Q (row rho = W_kR R_{K-1-rho}) the
//   position term of row i is row i of q Q^T shifted left by L-1-i.
//
// One thread block handles 128 query rows of one (batch, head) and a range of
// 128-key tiles.  Everything accumulates in TMEM (fp32, lane = query row):
//   S      [128 x 128]  = q K_t^T   + 1 (u.k_j)            content term, tile t
//   Bt[c]  [128 x 128]  = q Qc^T    + 1 (v.r_rho)          position term, chunk c
// where chunk c is rows [c*128 + L-128-i0, +128) of the reversed table.  Key
// tile t needs chunks t and t+1 (a 256-column window: row il of the tile reads
// window column jj + 127 - il for key jj, the Appendix B shift), so each chunk
// is multiplied once and kept in one of two TMEM slots while two consecutive
// key tiles read it.  The shift is applied when the softmax warps read the
// window, through a per-thread shared-memory skew buffer; no L x K matrix
// exists anywhere.
//
// Key tile t and table chunk t+1 are one shared-memory pair [32 KB] whose two
// halves are multiplied by q as a single N = 256 operand: TMEM holds
// [even-chunk slot | S | odd-chunk slot], and the pair is laid out [chunk ; keys]
// when chunk t+1 is even (its slot precedes S) and [keys ; chunk] when it is odd,
// so that the 256 result columns of one MMA land on S and the chunk's slot.
//
// The bias terms u.k_j and v.r_rho are exact in fp32: q enters the MMA as
// given, and the biases come from small MMAs [K tile | table chunk] x [u ; v]^T
// whose fp32 results the softmax warps split into bf16 hi + lo pairs; a fifth
// MMA K-step multiplies a column of ones by those pairs.  The same pairs carry
// the causal mask: a hidden key (j > i + M, or j >= K) always meets a table row
// past the end of r, whose pair is (-inf, 0), so its score comes out -inf.
//
// P goes from the softmax registers to TMEM (tcgen05.st) and the PV product
// takes its A operand from there.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: q tile once, then K, V and table chunks through
//               shared-memory rings, with L2 prefetches further ahead
//   warp 1      MMA issuer: the whole warp follows the schedule (barrier
//               waits, descriptors) so that its values stay warp-uniform, and one
//               elected lane issues each group of MMAs and commits
//   warp 2      TMEM allocator
//   warps 4..7  softmax: thread = query row.  Per tile: gather S + shifted
//               window, release S, convert the next tile's biases, running
//               max (lazy rescale), exp2, P (bf16) to TMEM; finally O / l.
//
// Every barrier wait is bounded: on time-out the block records an error in the
// device status word, raises a block-wide abort flag, drains its own in-flight
// copies and MMAs, frees TMEM and returns.
#include "kernels.h"
#include "ptx.cuh"

namespace txl {
namespace {

using namespace ptx;

constexpr int BM = kTcBM, BN = kTcBN, DH = kTcDH;
constexpr int NP = 2;                  // pair stages [key tile t, table chunk t+1]
constexpr int NS = 2;                  // V ring stages
constexpr int PF = 2;                  // L2 prefetch distance (tiles)
constexpr int TILE = BM * DH * 2;      // 16384 bytes: 128 rows x 128 bytes
constexpr int EXT = 4096;              // bias-column tile: 128 rows x 16 bytes, then
                                       // 2 KB of zeros for K columns 8..15
constexpr int EXT2 = 8192;             // the same for a pair: 256 rows, then 4 KB of zeros
constexpr int PAIR = 2 * TILE;
constexpr int SKEW_STRIDE = 132;       // floats per skew row: a 4 x 32 ring + 4 pad
                                       // (stride = 4 mod 32: conflict-free both ways)

// TMEM columns
constexpr uint32_t TM_CA = 0;          // table-chunk slot of even chunks
constexpr uint32_t TM_S = 128;         // content scores
constexpr uint32_t TM_CC = 256;        // table-chunk slot of odd chunks
constexpr uint32_t TM_O = 384;         // output accumulator (64 columns)
constexpr uint32_t TM_BK = 448;        // k.u / k.v for the next key tile (16 columns)
constexpr uint32_t TM_BR = 464;        // r.u / r.v for the next table chunk
constexpr uint32_t TM_BR2 = 480;       // second table chunk of the first tile
constexpr uint32_t TM_P = 448;         // P (bf16 pairs, 64 columns); shares the bias
                                       // columns, which are read before P is written
                                       // and refilled only after PV has read P
constexpr uint32_t TM_COLS = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;
constexpr int OFF_PAIR = OFF_Q + TILE;            // NP pair stages
constexpr int OFF_V = OFF_PAIR + NP * PAIR;       // NS stages
constexpr int OFF_UB = OFF_V + NS * TILE;         // [u ; v ; 0 x 14] 16 x 128 bytes, swizzled
constexpr int OFF_AEXT = OFF_UB + 2048;           // ones column: rows [1, 1, 0 x 6]
constexpr int OFF_PEXT = OFF_AEXT + EXT;          // NP pair tiles of (hi, lo) of k.u / v.r
constexpr int OFF_R0EXT = OFF_PEXT + NP * EXT2;   // (hi, lo) of v.r of chunk 0
constexpr int OFF_SKEW = OFF_R0EXT + EXT;         // 128 rows x SKEW_STRIDE floats
// Table chunk 0 of the first tile shares the skew buffer's bytes: the MMAs that
// read it complete before s_full of the first tile, and the softmax warps write
// the skew buffer only after that.
constexpr int OFF_R0 = OFF_SKEW;
constexpr int OFF_BAR = OFF_SKEW + BM * SKEW_STRIDE * 4;
constexpr int N_BAR = 1 + 2 * NP + 2 * NS + 1 + 8;
constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;      // slack for the manual alignment

static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_UB % 1024 == 0 && OFF_R0 % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(OFF_R0 + TILE <= OFF_SKEW + BM * SKEW_STRIDE * 4, "chunk 0 must fit the skew buffer");

struct Bars {
    uint64_t *q_full;
    uint64_t *pair_full, *pair_empty, *v_full, *v_empty;
    uint64_t *r0_full;
    uint64_t *prep, *bias_full, *ext_full, *s_full, *s_free, *p_full, *o_done, *drain;
};

__device__ __forceinline__ Bars make_bars(uint8_t *smem)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    Bars x;
    x.q_full = b;
    x.pair_full = b + 1;
    x.pair_empty = x.pair_full + NP;
    x.v_full = x.pair_empty + NP;
    x.v_empty = x.v_full + NS;
    x.r0_full = x.v_empty + NS;
    x.prep = x.r0_full + 1;
    x.bias_full = x.prep + 1;
    x.ext_full = x.bias_full + 1;
    x.s_full = x.ext_full + 1;
    x.s_free = x.s_full + 1;
    x.p_full = x.s_free + 1;
    x.o_done = x.p_full + 1;
    x.drain = x.o_done + 1;
    return x;
}

__device__ __forceinline__ void fail(const TcParams &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicOr(p.status, 1u);
}

// Uses of r cannot move above an earlier asm volatile (the TMEM load wait).
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                   "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                   "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_x2(uint32_t taddr, uint32_t &a, uint32_t &b)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                 : "=r"(a), "=r"(b)
                 : "r"(taddr));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t a)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 2^x on the SFU.
__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Descriptor of a bias-column tile: K-major, no swizzle; rows 16 bytes apart,
// 8-row core matrices 128 bytes apart (stride offset), and the second
// core-matrix column (K 8..15) 2 KB further (leading offset), in the tile's own
// zero half.  Every address either offset can reach stays inside the tile and
// the shared-memory regions that follow it.
__device__ __forceinline__ uint64_t sdesc_ext(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(2048u >> 4) << 16) |
           ((uint64_t)(128u >> 4) << 32) | (1ull << 46);
}

// The same for a pair's 256 rows: the zero half (K columns 8..15) starts 4 KB
// after the tile.
__device__ __forceinline__ uint64_t sdesc_ext2(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(4096u >> 4) << 16) |
           ((uint64_t)(128u >> 4) << 32) | (1ull << 46);
}

// hi + lo bf16 pair whose sum is x to about 2^-17 relative.
__device__ __forceinline__ uint32_t split_bf16(float x)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    return (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
}

__global__ void __launch_bounds__(256, 1)
    relattn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_r, const TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work of this block: (b*H + h, query tile, key split) -----------------
    // Query tiles go last-first over the grid: later tiles see more keys (the
    // causal edge), so the longest blocks start first and the shorter ones
    // fill the last wave.
    int wid = blockIdx.x;
    const int split = wid % p.n_splits;
    wid /= p.n_splits;
    const int n_bh = p.B * p.H;
    const int qt = p.n_qtiles - 1 - wid / n_bh;
    const int bh = wid % n_bh;
    const int h = bh % p.H;
    const int i0 = qt * BM;
    const int rows_valid = min(BM, p.L - i0);
    const int jmax = min(p.K - 1, p.M + i0 + rows_valid - 1);   // last key any row sees
    const int n_tiles_all = jmax / BN + 1;
    const int per_split = (n_tiles_all + p.n_splits - 1) / p.n_splits;
    const int t_begin = split * per_split;
    const int T = min(n_tiles_all, t_begin + per_split) - t_begin;
    // (a split past the last tile is empty: T <= 0, handled below)
    TXL_CHECK(split < p.n_splits && qt >= 0 && qt < p.n_qtiles && bh < n_bh && t_begin >= 0 &&
                  T <= per_split && rows_valid > 0,
              p.status);

    if (T <= 0) {
        // An empty key split (only with n_splits > 1): contribute nothing.
        if (warp >= 4) {
            const int row = threadIdx.x - 128;
            if (row < rows_valid) {
                const size_t prow = ((size_t)split * p.B * p.H + bh) * p.L + i0 + row;
                float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * DH);
#pragma unroll
                for (int c = 0; c < DH / 4; ++c) po[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.part_lse[prow] = -INFINITY;
            }
        }
        return;
    }

    const Bars bar = make_bars(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full, 1);
        for (int s = 0; s < NP; ++s) {
            mbar_init(bar.pair_full + s, 1);
            mbar_init(bar.pair_empty + s, 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar.v_full + s, 1);
            mbar_init(bar.v_empty + s, 1);
        }
        mbar_init(bar.r0_full, 1);
        mbar_init(bar.prep, 128);
        mbar_init(bar.bias_full, 1);
        mbar_init(bar.ext_full, 128);
        mbar_init(bar.s_full, 1);
        mbar_init(bar.s_free, 128);
        mbar_init(bar.p_full, 128);
        mbar_init(bar.o_done, 1);
        mbar_init(bar.drain, 1);
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
    // First row of table chunk c (local index): the window of key tile t starts
    // at t*BN + L-1-i0-(BM-1), plus the row offset of a longer table.
    const int r_base = p.L - BM - i0 + p.r_off + t_begin * BN;

    if (warp == 0) {
        // ===================== TMA producer =====================================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_r);
            const uint64_t pol_stream = policy_evict_first();  // K, V: read once
            const uint64_t pol_keep = policy_evict_last();     // table: shared by the batch
            bool ok = true;
            int pc = 0, vc = 0;  // copies issued into the pair and V rings
            // Pair t: key tile t and table chunk t+1, [keys ; chunk] for even t.
            auto load_pair = [&](int t) -> bool {
                const int ps = t % NP;
                if (!mbar_wait(bar.pair_empty + ps, ((t / NP) & 1) ^ 1, abort_flag, wait_ns))
                    return false;
                const bool kfirst = (t & 1) == 0;
                uint8_t *st = smem + OFF_PAIR + ps * PAIR;
                mbar_arrive_expect_tx(bar.pair_full + ps, PAIR);
                tma_load_3d_hint(st + (kfirst ? 0 : TILE), &tm_k, bar.pair_full + ps, 0,
                                 (t_begin + t) * BN, bh, pol_stream);
                tma_load_3d_hint(st + (kfirst ? TILE : 0), &tm_r, bar.pair_full + ps, 0,
                                 r_base + (t + 1) * BN, h, pol_keep);
                pc = t + 1;
                return true;
            };
            auto load_v = [&](int t) -> bool {
                const int st = t % NS;
                if (!mbar_wait(bar.v_empty + st, ((t / NS) & 1) ^ 1, abort_flag, wait_ns))
                    return false;
                mbar_arrive_expect_tx(bar.v_full + st, TILE);
                tma_load_3d_hint(smem + OFF_V + st * TILE, &tm_v, bar.v_full + st, 0,
                                 (t_begin + t) * BN, bh, pol_stream);
                vc = t + 1;
                return true;
            };
            // The first biases need pair 0 and chunk 0, q only the scores after
            // them: copies in that order, then the L2 prefetches.
            ok = load_pair(0);
            mbar_arrive_expect_tx(bar.r0_full, TILE);
            tma_load_3d_hint(smem + OFF_R0, &tm_r, bar.r0_full, 0, r_base, h, pol_keep);
            mbar_arrive_expect_tx(bar.q_full, TILE);
            tma_load_3d(smem + OFF_Q, &tm_q, bar.q_full, 0, i0, bh);
            for (int c = 0; c < min(PF, T); ++c) {
                tma_prefetch_3d(&tm_k, 0, (t_begin + c) * BN, bh);
                tma_prefetch_3d(&tm_v, 0, (t_begin + c) * BN, bh);
                tma_prefetch_3d(&tm_r, 0, r_base + (c + 1) * BN, h);
            }
            for (int it = 0; it < T && ok; ++it) {
                const int t = t_begin + it;
                if (it + PF < T) {
                    tma_prefetch_3d(&tm_k, 0, (t + PF) * BN, bh);
                    tma_prefetch_3d(&tm_v, 0, (t + PF) * BN, bh);
                    tma_prefetch_3d(&tm_r, 0, r_base + (it + PF + 1) * BN, h);
                }
                if (it + 1 < T && !(ok = load_pair(it + 1))) break;
                if (!(ok = load_v(it))) break;
            }
            if (ok) {
                // The block that will most likely take this SM next (one block
                // per SM, launched in index order): pull its first q, key,
                // value tiles and table chunks into L2 so that its start does
                // not wait on HBM.
                uint32_t nsm;
                asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
                int nw = (int)blockIdx.x + (int)nsm;
                if (nw < (int)gridDim.x) {
                    const int n_split = nw % p.n_splits;
                    nw /= p.n_splits;
                    const int n_qt = p.n_qtiles - 1 - nw / n_bh;
                    const int nx_bh = nw % n_bh;
                    const int n_i0 = n_qt * BM;
                    const int n_jmax = min(p.K - 1, p.M + n_i0 + min(BM, p.L - n_i0) - 1);
                    const int n_per = (n_jmax / BN + 1 + p.n_splits - 1) / p.n_splits;
                    const int n_tb = n_split * n_per;
                    const int n_rbase = p.L - BM - n_i0 + p.r_off + n_tb * BN;
                    tma_prefetch_3d(&tm_q, 0, n_i0, nx_bh);
                    tma_prefetch_3d(&tm_k, 0, n_tb * BN, nx_bh);
                    tma_prefetch_3d(&tm_v, 0, n_tb * BN, nx_bh);
                    tma_prefetch_3d(&tm_r, 0, n_rbase, nx_bh % p.H);
                    tma_prefetch_3d(&tm_r, 0, n_rbase + BN, nx_bh % p.H);
                }
            }
            if (!ok) {
                fail(p, abort_flag);
                // Drain: let every copy this thread started land before the block
                // exits (bounded; the abort flag is deliberately not consulted).
                // The newest copy of each ring slot is the only one that can
                // still be in flight.
                const int zero = 0;
                const volatile int *nz = &zero;
                mbar_wait(bar.q_full, 0, nz, wait_ns);
                mbar_wait(bar.r0_full, 0, nz, wait_ns);
                for (int c = max(0, pc - NP); c < pc; ++c)
                    mbar_wait(bar.pair_full + c % NP, (c / NP) & 1, nz, wait_ns);
                for (int c = max(0, vc - NS); c < vc; ++c)
                    mbar_wait(bar.v_full + c % NS, (c / NS) & 1, nz, wait_ns);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =======================================
        // Descriptors are computed once as 64-bit bases; an offset of b bytes
        // adds b / 16.  Every lane waits on the barriers (votes keep the warp
        // converged) and one elected lane issues.
        {
            constexpr uint32_t ID_N128 = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t ID_N256 = idesc_bf16_f32(128, 256, false);
            constexpr uint32_t ID_N16 = idesc_bf16_f32(128, 16, false);
            constexpr uint32_t ID_O = idesc_bf16_f32(128, 64, true);
            const uint64_t dQ = sdesc_sw128(smem_u32(smem + OFF_Q));
            const uint64_t dPair = sdesc_sw128(smem_u32(smem + OFF_PAIR));
            const uint64_t dV = sdesc_sw128(smem_u32(smem + OFF_V));
            const uint64_t dR0 = sdesc_sw128(smem_u32(smem + OFF_R0));
            const uint64_t dUB = sdesc_sw128(smem_u32(smem + OFF_UB));
            const uint64_t d_aext = sdesc_ext(smem_u32(smem + OFF_AEXT));
            const uint64_t dPX = sdesc_ext2(smem_u32(smem + OFF_PEXT));
            const uint64_t dR0X = sdesc_ext(smem_u32(smem + OFF_R0EXT));
            auto elect = []() -> bool {
                uint32_t el;
                asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
                             : "=r"(el));
                return el != 0;
            };
            auto W = [&](uint64_t *bar, int par) {
                return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, wait_ns));
            };
            auto WP = [&](uint64_t *bar, int par) {
                return __all_sync(0xffffffffu, mbar_wait_poll(bar, par, abort_flag, wait_ns));
            };
            // descriptor offsets are added in 16-byte units
            auto bias_mma = [&](uint32_t tcol, uint64_t a_tile) {
                if (elect()) {
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        mma_bf16_ss(tmem + tcol, a_tile + kk * 2, dUB + kk * 2, ID_N16, kk);
                }
                __syncwarp();
            };
            auto pair_k = [&](int t) { return dPair + (uint64_t)(((t % NP) * PAIR + ((t & 1) ? TILE : 0)) >> 4); };
            auto pair_r = [&](int t) { return dPair + (uint64_t)(((t % NP) * PAIR + ((t & 1) ? 0 : TILE)) >> 4); };
            auto score_pair = [&](int t) {
                const uint32_t dcol = (t & 1) ? TM_CA : TM_S;
                const uint64_t bb = dPair + (uint64_t)(((t % NP) * PAIR) >> 4);
                if (elect()) {
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        mma_bf16_ss(tmem + dcol, dQ + kk * 2, bb + kk * 2, ID_N256, kk);
                }
                __syncwarp();
            };
            auto score_pair_ext = [&](int t) {
                const uint32_t dcol = (t & 1) ? TM_CA : TM_S;
                const uint64_t bx = dPX + (uint64_t)(((t % NP) * EXT2) >> 4);
                if (elect()) {
                    mma_bf16_ss(tmem + dcol, d_aext, bx, ID_N256, 1);
                    mma_commit(bar.s_full);
                    mma_commit(bar.pair_empty + t % NP);
                }
                __syncwarp();
            };
            auto commit1 = [&](uint64_t *b1) {
                if (elect()) mma_commit(b1);
                __syncwarp();
            };
            auto wait_pair = [&](int t) { return W(bar.pair_full + t % NP, (t / NP) & 1); };

            bool ok = W(bar.prep, 0);
            if (ok) ok = wait_pair(0) && W(bar.r0_full, 0);
            if (ok) {
                tc_fence_after_sync();
                bias_mma(TM_BK, pair_k(0));
                bias_mma(TM_BR, pair_r(0));
                bias_mma(TM_BR2, dR0);
                commit1(bar.bias_full);
            }
            if (ok) ok = W(bar.q_full, 0);
            if (ok) {
                tc_fence_after_sync();
                score_pair(0);
                if (elect()) {
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        mma_bf16_ss(tmem + TM_CA, dQ + kk * 2, dR0 + kk * 2, ID_N128, kk);
                }
                __syncwarp();
                ok = W(bar.ext_full, 0);
            }
            if (ok) {
                tc_fence_after_sync();
                if (elect()) {
                    mma_bf16_ss(tmem + TM_S, d_aext, dPX, ID_N256, 1);
                    mma_bf16_ss(tmem + TM_CA, d_aext, dR0X, ID_N128, 1);
                    mma_commit(bar.s_full);
                    mma_commit(bar.pair_empty);
                }
                __syncwarp();
            }
            if (ok && T > 1) {
                ok = wait_pair(1);
                if (ok) {
                    tc_fence_after_sync();
                    bias_mma(TM_BK, pair_k(1));
                    bias_mma(TM_BR, pair_r(1));
                    commit1(bar.bias_full);
                }
            }
            for (int it = 0; it < T && ok; ++it) {
                if (!(ok = WP(bar.s_free, it & 1))) break;
                if (it + 1 < T) {
                    tc_fence_after_sync();
                    score_pair(it + 1);
                    if (!(ok = WP(bar.ext_full, (it + 1) & 1))) break;
                    tc_fence_after_sync();
                    score_pair_ext(it + 1);
                }
                if (!(ok = WP(bar.p_full, it & 1))) break;
                const int st = it % NS;
                if (!(ok = W(bar.v_full + st, (it / NS) & 1))) break;
                tc_fence_after_sync();
                const uint64_t vb = dV + (uint64_t)((st * TILE) >> 4);
                if (elect()) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_bf16_ts(tmem + TM_O, tmem + TM_P + 8 * kk, vb + kk * (2048 >> 4), ID_O,
                                    (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar.o_done);
                    mma_commit(bar.v_empty + st);
                }
                __syncwarp();
                if (it + 2 < T) {
                    if (!(ok = W(bar.o_done, it & 1))) break;
                    if (!(ok = wait_pair(it + 2))) break;
                    tc_fence_after_sync();
                    bias_mma(TM_BK, pair_k(it + 2));
                    bias_mma(TM_BR, pair_r(it + 2));
                    commit1(bar.bias_full);
                }
            }
            commit1(bar.drain);
            const int zero = 0;
            mbar_wait(bar.drain, 0, &zero, wait_ns);
            if (!ok && lane == 0) fail(p, abort_flag);
        }
    } else if (warp >= 4) {
        // ===================== softmax warps ====================================
        const int wq = warp - 4;          // TMEM lane quarter of this warp
        const int row = wq * 32 + lane;   // query row within the tile (also the key /
                                          // table row for the bias conversions)
        const int i = i0 + row;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + TM_S;
        const uint32_t tB = tmem + lane_off;
        const uint32_t tO = tmem + lane_off + TM_O;
        const uint32_t skew = smem_u32(smem + OFF_SKEW) + (uint32_t)row * SKEW_STRIDE * 4;
        // Key y of a 32-key piece sits at column (31 - lane + y) of the two
        // staged window chunks.
        const uint32_t skew_rd = skew + (uint32_t)(31 - lane) * 4;
        const uint32_t sPX = smem_u32(smem + OFF_PEXT);
        // bias rows of pair t: keys first for even t, the chunk first for odd t
        auto pext_k = [&](int t) { return sPX + (t % NP) * EXT2 + ((t & 1) ? BM * 16 : 0); };
        auto pext_r = [&](int t) { return sPX + (t % NP) * EXT2 + ((t & 1) ? 0 : BM * 16); };

        // ---- one-time operands: [u ; v] tile, ones column, zeroed ext tiles ----
        {
            uint8_t *ub = smem + OFF_UB;
            if (row < 16) {
                const uint4 *src = (row == 0) ? reinterpret_cast<const uint4 *>(p.u + h * DH)
                                 : (row == 1) ? reinterpret_cast<const uint4 *>(p.vb + h * DH)
                                              : nullptr;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 val = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(ub + row * 128 + ((c ^ (row & 7)) * 16)) = val;
                }
            }
            // Ones column: row i = [1, 1, 0, 0, 0, 0, 0, 0] (bf16 1.0 = 0x3f80); then
            // zero the second half of that tile and all of the bias tiles.
            *reinterpret_cast<uint4 *>(smem + OFF_AEXT + row * 16) =
                make_uint4(0x3f803f80u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(smem + OFF_AEXT + 2048 + row * 16) = make_uint4(0, 0, 0, 0);
            for (int o = row * 16; o < NP * EXT2 + EXT; o += 128 * 16)
                *reinterpret_cast<uint4 *>(smem + OFF_PEXT + o) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            mbar_arrive(bar.prep);
        }

        // The causal mask lives in the table biases.  A key j is hidden from
        // query i exactly when its distance M + i - j is negative (j > i + M, and
        // every key past K), i.e. when the window reads a table row past the end
        // of r.  TMA fills those rows with zeros, and their bias becomes
        // (hi, lo) = (-inf, 0), so the score MMA writes -inf there and the
        // softmax needs no mask of its own.  Table row of this thread in
        // chunk c, relative to the end of r: rmask + c*BN (masked when >= 0).
        const int rmask = r_base + row - (p.K + p.r_off);
        auto r_bias = [&](uint32_t rv, int c) {
            return (rmask + c * BN >= 0) ? 0x0000FF80u : split_bf16(__uint_as_float(rv));
        };
        // Second half of a bias conversion: (hi, lo) pairs of already loaded
        // fp32 k.u and v.r values (table chunk c) into the ext tiles.
        auto convert_store = [&](uint32_t ku, uint32_t rv, int c, uint32_t kext, uint32_t rext) {
            st_shared_b32(kext + row * 16, split_bf16(__uint_as_float(ku)));
            st_shared_b32(rext + row * 16, r_bias(rv, c));
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(bar.ext_full);
        };
        // Bias conversion: fp32 k.u (key row) and v.r (table row) from TMEM into
        // (hi, lo) bf16 pairs in the ext tiles.
        auto convert = [&](int phase, uint32_t kext, uint32_t rext, uint32_t rext2) -> bool {
            const bool got = __all_sync(0xffffffffu,
                                        mbar_wait(bar.bias_full, phase & 1, abort_flag, wait_ns));
            if (!got) return false;
            tc_fence_after_sync();
            uint32_t ku, kv, ru, rv, r2u = 0, r2v = 0;
            tmem_ld_x2(tmem + lane_off + TM_BK, ku, kv);
            tmem_ld_x2(tmem + lane_off + TM_BR, ru, rv);
            if (rext2) tmem_ld_x2(tmem + lane_off + TM_BR2, r2u, r2v);
            asm volatile("tcgen05.wait::ld.sync.aligned;"
                         : "+r"(ku), "+r"(kv), "+r"(ru), "+r"(rv), "+r"(r2u), "+r"(r2v)::"memory");
            st_shared_b32(kext + row * 16, split_bf16(__uint_as_float(ku)));
            st_shared_b32(rext + row * 16, r_bias(rv, 1));
            if (rext2) st_shared_b32(rext2 + row * 16, r_bias(r2v, 0));
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(bar.ext_full);
            return true;
        };

        bool ok = convert(0, pext_k(0), pext_r(0), smem_u32(smem + OFF_R0EXT));

        const uint64_t sl2x2 = pack2(p.scale_log2, p.scale_log2);
        float m_ref = -INFINITY;  // running max (scaled, log2 units), lazily updated
        float l_sum = 0.f;
        const uint32_t tP = tmem + lane_off + TM_P;

        for (int it = 0; it < T && ok; ++it) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar.s_full, it & 1, abort_flag, wait_ns));
            if (!ok) break;
            tc_fence_after_sync();

            // ---- gather: x[jj] = S[row][jj] + window[row][jj + 127 - row] -------
            // Window columns of this warp: [96-32wq, 96-32wq+160) of the virtual
            // 256-column window (five 32-column chunks); table chunk it sits in
            // the even- or odd-chunk TMEM slot by its parity, chunk it+1 in the
            // other.  Each window chunk c goes
            // once through a 4-slot shared-memory ring (slot c % 4); key y of
            // piece pc is ring column (32*pc + 31 - lane + y), which for pc = 3
            // wraps from slot 3 to slot 0 when y > lane.  Chunk 4 of a tile is
            // chunk 0 of the next (the same 32 columns of table chunk it+1), and
            // it lands in slot 0: only a block's first tile loads chunk 0.
            // window column w of this tile in TMEM: chunk it (w < 128) or it+1
            const uint32_t slot0 = (it & 1) ? TM_CC : TM_CA, slot1 = (it & 1) ? TM_CA : TM_CC;
            const uint32_t wbase = (uint32_t)(96 - 32 * wq);
            auto wcol = [&](uint32_t w) { return w < 128u ? slot0 + w : slot1 + (w - 128u); };
            uint32_t bku = 0, bkv = 0, bru = 0, brv = 0;  // next tile's bias values
            float x[BN];
            float mx[8];  // 8 independent running-max chains over the gathered scores
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
            uint32_t wa[32], wb[32], s[32];
            if (it == 0) {
                tmem_ld32(tB + wcol(wbase), wa);
                tmem_wait_ld();
                reg_fence(wa);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(skew + c * 16, wa[4 * c], wa[4 * c + 1], wa[4 * c + 2],
                                 wa[4 * c + 3]);
            }
            tmem_ld32(tB + wcol(wbase + 32u), wb);
            tmem_ld32(tS, s);
            tmem_wait_ld();
            reg_fence(wb);
            reg_fence(s);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(skew + 128 + c * 16, wb[4 * c], wb[4 * c + 1], wb[4 * c + 2],
                             wb[4 * c + 3]);
#pragma unroll
            for (int pc = 0; pc < BN / 32; ++pc) {
                // Next window chunk and next S piece are loaded while this piece
                // is read from the ring.
                if (pc + 1 < BN / 32) {
                    tmem_ld32(tB + wcol(wbase + 32u * (pc + 2)), wa);
                    tmem_ld32(tS + 32 * (pc + 1), wb);
                }
                const uint32_t rd = skew_rd + (uint32_t)(pc * 128);
                // every skewed read stays inside this row's 4 x 32-float ring
                TXL_CHECK(pc == 3 ? (rd + 4u * (lane + 1) - 512u >= skew || lane == 31) &&
                                        rd + 4u * lane < skew + 512u
                                  : rd + 124u < skew + 512u,
                          p.status);
                float wv[32];
                if (pc == 3) {
#pragma unroll
                    for (int y = 0; y < 32; ++y)
                        wv[y] = ld_shared_f32(rd + y * 4 - ((y > lane) ? 512u : 0u));
                } else {
#pragma unroll
                    for (int y = 0; y < 32; ++y) wv[y] = ld_shared_f32(rd + y * 4);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    unpack2(add2(pack2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])),
                                 pack2(wv[2 * k], wv[2 * k + 1])),
                            x[32 * pc + 2 * k], x[32 * pc + 2 * k + 1]);
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    mx[a] = max3f(mx[a], x[32 * pc + 4 * a], x[32 * pc + 4 * a + 1]);
                    mx[a] = max3f(mx[a], x[32 * pc + 4 * a + 2], x[32 * pc + 4 * a + 3]);
                }
                if (pc + 1 < BN / 32) {
                    tmem_wait_ld();
                    reg_fence(wa);
                    reg_fence(wb);
                    // chunk pc+2 into slot (pc+2) % 4: empty, or (chunk 4) the slot of
                    // chunk 0, which no later piece of this tile reads
                    const uint32_t slot = skew + (uint32_t)(((pc + 2) % 4) * 128);
                    TXL_CHECK(wcol(wbase + 32u * (pc + 2)) + 32u <= TM_O, p.status);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(slot + c * 16, wa[4 * c], wa[4 * c + 1], wa[4 * c + 2],
                                     wa[4 * c + 3]);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[e] = wb[e];
                }
            }
            tc_fence_before_sync();
            mbar_arrive(bar.s_free);

            // ---- biases of the next tile (key tile it+1, table chunk it+2) -------
            // Read before this tile's P overwrites their columns; by now the MMA
            // warp has computed them (after the previous tile's PV), so the wait
            // is rarely a wait.
            if (it + 1 < T) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar.bias_full, (it + 1) & 1, abort_flag,
                                                       wait_ns));
                if (!ok) break;
                tc_fence_after_sync();
                tmem_ld_x2(tmem + lane_off + TM_BK, bku, bkv);
                tmem_ld_x2(tmem + lane_off + TM_BR, bru, brv);
                asm volatile("tcgen05.wait::ld.sync.aligned;"
                             : "+r"(bku), "+r"(bkv), "+r"(bru), "+r"(brv)::"memory");
                convert_store(bku, brv, it + 2, pext_k(it + 1), pext_r(it + 1));
            }

            // ---- tile max (masked keys hold -inf) ----------------------------------
            float mt = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
            mt *= p.scale_log2;  // scores scale by a positive constant

            // Lazy rescale: move the reference max only when the tile max exceeds
            // it by more than 8 (a factor 256); exact after the final division.
            float alpha = 1.f;
            const bool resc = mt > m_ref + 8.f;
            if (resc) {
                alpha = ex2f(m_ref - mt);  // 0 when m_ref is -inf
                l_sum *= alpha;
                m_ref = mt;
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;

            // PV of the previous tile must be done: it reads P and writes O.  Before
            // any tile but the last this is already known: the MMA warp issues the
            // next tile's bias products only after that PV has completed, and their
            // commit (bias_full, waited for above) covers every earlier MMA.
            if (it > 0) {
                if (it + 1 == T) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar.o_done, (it - 1) & 1, abort_flag, wait_ns));
                    if (!ok) break;
                    tc_fence_after_sync();
                }
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * half, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + 32 * half, o);
                    }
                    tmem_st_wait();
                }
            }

            // ---- exponentiate, row sum, P (bf16 pairs) into TMEM -----------------
            const uint64_t nmu = pack2(-mu, -mu);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int jj = 64 * half + 2 * e;
                    const uint64_t a = fma2(pack2(x[jj], x[jj + 1]), sl2x2, nmu);
                    float a0, a1;
                    unpack2(a, a0, a1);
                    const float p0 = ex2f(a0), p1 = ex2f(a1);
                    acc[e & 3] = add2(acc[e & 3], pack2(p0, p1));
                    pk[e] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tP + 32 * half, pk);
            }
            {
                const uint64_t s01 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
                float a0, a1;
                unpack2(s01, a0, a1);
                l_sum += a0 + a1;
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(bar.p_full);
        }

        // ---- epilogue ----------------------------------------------------------
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar.o_done, (T - 1) & 1, abort_flag, wait_ns));
        }
        if (ok) {
            tc_fence_after_sync();
            uint32_t o0[32], o1[32];
            tmem_ld32(tO, o0);
            tmem_ld32(tO + 32, o1);
            tmem_wait_ld();
            reg_fence(o0);
            reg_fence(o1);
            const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
            const float lse2 = (l_sum > 0.f) ? m_ref + __log2f(l_sum) : -INFINITY;
            if (row < rows_valid) {
                const size_t orow = (size_t)bh * p.L + i;
                TXL_CHECK(i < p.L && orow < (size_t)p.B * p.H * p.L, p.status);
                if (p.n_splits == 1) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * DH);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t *src = (c < 4) ? &o0[8 * c] : &o1[8 * (c - 4)];
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(src[2 * e]) * inv,
                                               __uint_as_float(src[2 * e + 1]) * inv);
                        dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (p.lse) p.lse[orow] = lse2 * 0.69314718055994531f;
                } else {
                    const size_t prow = (size_t)split * p.B * p.H * p.L + orow;
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * DH);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint32_t *src = (c < 8) ? &o0[4 * c] : &o1[4 * (c - 8)];
                        dst[c] = make_float4(__uint_as_float(src[0]) * inv,
                                             __uint_as_float(src[1]) * inv,
                                             __uint_as_float(src[2]) * inv,
                                             __uint_as_float(src[3]) * inv);
                    }
                    p.part_lse[prow] = lse2;
                }
            }
        }
        if (!ok && lane == 0) fail(p, abort_flag);
        tc_fence_before_sync();
    }

    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// One thread fails one index check: tests that the debug build reports it (a
// no-op in release builds, where the checks compile away).
__global__ void index_probe_kernel(unsigned int *status)
{
    if (threadIdx.x == 0) TXL_CHECK(status == nullptr, status);
}

// Waits on a barrier nothing will complete; the bounded wait must give up and
// record the time-out.  Used to test that path without hanging the device.
__global__ void wait_probe_kernel(unsigned int *status, unsigned long long wait_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(&bar, 0, reinterpret_cast<volatile int *>(&abort_flag), wait_ns))
            atomicOr(status, 1u);
    }
}

} // namespace

size_t tc_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_relattn_tc(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const CUtensorMap &tm_r,
                              const TcParams &p, cudaStream_t s)
{
    static bool attr_set[64] = {};  // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(relattn_fwd_tc_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const long long blocks = (long long)p.B * p.H * p.n_qtiles * p.n_splits;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    relattn_fwd_tc_kernel<<<(unsigned)blocks, 256, SMEM_BYTES, s>>>(tm_q, tm_k, tm_v, tm_r, p);
    return cudaGetLastError();
}

cudaError_t launch_index_probe(unsigned int *status, cudaStream_t s)
{
    index_probe_kernel<<<1, 32, 0, s>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(unsigned int *status, unsigned long long wait_ns, cudaStream_t s)
{
    wait_probe_kernel<<<1, 32, 0, s>>>(status, wait_ns);
    return cudaGetLastError();
}

} // namespace txl
