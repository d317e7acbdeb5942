// Tensor-core (tcgen05 + TMEM + TMA) forward kernel for Transformer-XL
// relative-position attention, bf16 operands, fp32 accumulation.
//
// "Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context":
//   §3.3 score  A_ij = (q_i + u).k_j + (q_i + v).W_kR R_{i-j}   (terms (a)+(c), (b)+(d))
//   §3.3 summary: masked softmax over the extended context, times v
//   Appendix B: with the reversed table Q (row rho = W_kR R_{K-1-rho}), row i of
//   the position term is row i of q Q^T shifted left by L-1-i.
//
// One thread block handles 128 query rows of one (batch, head) and a range of
// 128-key tiles.  Per key tile, in TMEM (fp32, lane = query row):
//   S  [128 x 128]  = (q + u) K^T                            content term
//   W  [128 x 256]  = (q + v) Qwin^T                         position window
// where Qwin is the 255 (+1) consecutive rows of the reversed table that any
// (row, key) pair of the tile can index.  Row il of the tile needs window
// column jj + 127 - il for key jj: the Appendix B shift, applied by index
// arithmetic when the softmax warps read W (through a small per-thread
// shared-memory skew buffer), so no L x K matrix exists anywhere.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: q tile once, then K, V and 128-row chunks of the
//               reversed table through shared-memory rings (mbarrier handshakes)
//   warp 1      MMA issuer (one thread): S and W for tile t+1 as soon as the
//               softmax has read tile t's S and W, then O += P V for tile t
//   warp 2      TMEM allocator
//   warps 4..7  softmax: thread = query row; forms q+u and q+v once, then per
//               tile gathers S + shifted W, masks (key after query), keeps a
//               running max with lazy rescaling, exponentiates (ex2), writes P
//               (bf16, 128-byte swizzled) to shared memory; finally O / l.
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
constexpr int NS = 2;                  // K / V ring stages
constexpr int NR = NS + 1;             // reversed-table chunk slots
constexpr int TILE = BM * DH * 2;      // 16384 bytes: 128 rows x 128 bytes
constexpr int SKEW_STRIDE = 68;        // floats per skew row (bank-conflict free)
constexpr uint32_t TM_S = 0, TM_W = 128, TM_O = 384, TM_COLS = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;                        // q + u (written over the raw q tile)
constexpr int OFF_QV = OFF_Q + TILE;            // q + v
constexpr int OFF_K = OFF_QV + TILE;            // NS stages
constexpr int OFF_V = OFF_K + NS * TILE;        // NS stages
constexpr int OFF_R = OFF_V + NS * TILE;        // NR chunks
constexpr int OFF_P = OFF_R + NR * TILE;        // keys 0-63, keys 64-127
constexpr int OFF_SKEW = OFF_P + 2 * TILE;      // 128 rows x SKEW_STRIDE floats
constexpr int OFF_BAR = OFF_SKEW + BM * SKEW_STRIDE * 4;
constexpr int N_BAR = 2 + 4 * NS + 2 * NR + 5;
constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;    // slack for the manual alignment

static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_BAR % 8 == 0, "barrier alignment");

struct Bars {
    uint64_t *q_full, *q_ready;
    uint64_t *k_full, *k_empty, *v_full, *v_empty;
    uint64_t *r_full, *r_empty;
    uint64_t *s_full, *s_free, *p_full, *o_done, *drain;
};

__device__ __forceinline__ Bars make_bars(uint8_t *smem)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    Bars x;
    x.q_full = b;
    x.q_ready = b + 1;
    x.k_full = b + 2;
    x.k_empty = x.k_full + NS;
    x.v_full = x.k_empty + NS;
    x.v_empty = x.v_full + NS;
    x.r_full = x.v_empty + NS;
    x.r_empty = x.r_full + NR;
    x.s_full = x.r_empty + NR;
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

// Empty registers "fence": uses of r cannot move above an earlier asm volatile.
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

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
    int wid = blockIdx.x;
    const int split = wid % p.n_splits;
    wid /= p.n_splits;
    const int qt = wid % p.n_qtiles;
    const int bh = wid / p.n_qtiles;
    const int h = bh % p.H;
    const int i0 = qt * BM;
    const int rows_valid = min(BM, p.L - i0);
    const int jmax = min(p.K - 1, p.M + i0 + rows_valid - 1);   // last key any row sees
    const int n_tiles_all = jmax / BN + 1;
    const int per_split = (n_tiles_all + p.n_splits - 1) / p.n_splits;
    const int t_begin = split * per_split;
    const int T = min(n_tiles_all, t_begin + per_split) - t_begin;

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
        mbar_init(bar.q_ready, 128);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar.k_full + s, 1);
            mbar_init(bar.k_empty + s, 1);
            mbar_init(bar.v_full + s, 1);
            mbar_init(bar.v_empty + s, 1);
        }
        for (int s = 0; s < NR; ++s) {
            mbar_init(bar.r_full + s, 1);
            mbar_init(bar.r_empty + s, 1);
        }
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

    if (warp == 0) {
        // ===================== TMA producer =====================================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_r);
            const uint64_t pol_stream = policy_evict_first();  // K, V: read once
            const uint64_t pol_keep = policy_evict_last();     // table: shared by the batch
            // Row of the reversed table at which chunk c starts: the window of key
            // tile t begins at t*BN + L-1-i0-(BM-1), plus the table's row offset.
            const int r_base = p.L - BM - i0 + p.r_off;
            bool ok = true;
            int kc = 0, vc = 0, rc = 0;  // copies issued into the K, V and table rings

            mbar_arrive_expect_tx(bar.q_full, TILE);
            tma_load_3d(smem + OFF_Q, &tm_q, bar.q_full, 0, i0, bh);
            mbar_arrive_expect_tx(bar.r_full + 0, TILE);
            tma_load_3d_hint(smem + OFF_R, &tm_r, bar.r_full + 0, 0, t_begin * BN + r_base, h,
                             pol_keep);
            rc = 1;

            for (int it = 0; it < T; ++it) {
                const int t = t_begin + it;
                const int st = it % NS;
                const uint32_t ph = (it / NS) & 1;
                if (!(ok = mbar_wait(bar.k_empty + st, ph ^ 1, abort_flag, wait_ns))) break;
                mbar_arrive_expect_tx(bar.k_full + st, TILE);
                tma_load_3d_hint(smem + OFF_K + st * TILE, &tm_k, bar.k_full + st, 0, t * BN, bh,
                                 pol_stream);
                kc = it + 1;

                const int lc = it + 1;  // table chunk used as the second half of tile it
                const int rs = lc % NR;
                if (!(ok = mbar_wait(bar.r_empty + rs, ((lc / NR) & 1) ^ 1, abort_flag, wait_ns)))
                    break;
                mbar_arrive_expect_tx(bar.r_full + rs, TILE);
                tma_load_3d_hint(smem + OFF_R + rs * TILE, &tm_r, bar.r_full + rs, 0,
                                 (t + 1) * BN + r_base, h, pol_keep);
                rc = lc + 1;

                if (!(ok = mbar_wait(bar.v_empty + st, ph ^ 1, abort_flag, wait_ns))) break;
                mbar_arrive_expect_tx(bar.v_full + st, TILE);
                tma_load_3d_hint(smem + OFF_V + st * TILE, &tm_v, bar.v_full + st, 0, t * BN, bh,
                                 pol_stream);
                vc = it + 1;
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
                for (int c = max(0, kc - NS); c < kc; ++c)
                    mbar_wait(bar.k_full + c % NS, (c / NS) & 1, nz, wait_ns);
                for (int c = max(0, vc - NS); c < vc; ++c)
                    mbar_wait(bar.v_full + c % NS, (c / NS) & 1, nz, wait_ns);
                for (int c = max(0, rc - NR); c < rc; ++c)
                    mbar_wait(bar.r_full + c % NR, (c / NR) & 1, nz, wait_ns);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =======================================
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t ID_O = idesc_bf16_f32(128, 64, true);
            const uint32_t sQ = smem_u32(smem + OFF_Q);
            const uint32_t sQV = smem_u32(smem + OFF_QV);
            const uint32_t sK = smem_u32(smem + OFF_K);
            const uint32_t sV = smem_u32(smem + OFF_V);
            const uint32_t sR = smem_u32(smem + OFF_R);
            const uint32_t sP = smem_u32(smem + OFF_P);

            auto issue_scores = [&](int it) -> bool {
                const int st = it % NS;
                if (!mbar_wait(bar.k_full + st, (it / NS) & 1, abort_flag, wait_ns)) return false;
                const int c0 = it, c1 = it + 1;
                if (!mbar_wait(bar.r_full + c0 % NR, (c0 / NR) & 1, abort_flag, wait_ns))
                    return false;
                if (!mbar_wait(bar.r_full + c1 % NR, (c1 / NR) & 1, abort_flag, wait_ns))
                    return false;
                tc_fence_after_sync();
                const uint32_t kb = sK + st * TILE;
                const uint32_t r0 = sR + (c0 % NR) * TILE;
                const uint32_t r1 = sR + (c1 % NR) * TILE;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_bf16_ss(tmem + TM_S, sdesc_sw128(sQ + kk * 32), sdesc_sw128(kb + kk * 32),
                                ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_bf16_ss(tmem + TM_W, sdesc_sw128(sQV + kk * 32),
                                sdesc_sw128(r0 + kk * 32), ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_bf16_ss(tmem + TM_W + 128, sdesc_sw128(sQV + kk * 32),
                                sdesc_sw128(r1 + kk * 32), ID_S, kk);
                mma_commit(bar.s_full);
                mma_commit(bar.k_empty + st);
                mma_commit(bar.r_empty + c0 % NR);
                return true;
            };

            bool ok = mbar_wait(bar.q_ready, 0, abort_flag, wait_ns);
            if (ok) {
                tc_fence_after_sync();
                ok = issue_scores(0);
            }
            for (int it = 0; it < T && ok; ++it) {
                if (!(ok = mbar_wait(bar.s_free, it & 1, abort_flag, wait_ns))) break;
                tc_fence_after_sync();
                if (it + 1 < T && !(ok = issue_scores(it + 1))) break;
                if (!(ok = mbar_wait(bar.p_full, it & 1, abort_flag, wait_ns))) break;
                const int st = it % NS;
                if (!(ok = mbar_wait(bar.v_full + st, (it / NS) & 1, abort_flag, wait_ns))) break;
                tc_fence_after_sync();
                const uint32_t vb = sV + st * TILE;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t a = sP + (kk >> 2) * TILE + (kk & 3) * 32;
                    mma_bf16_ss(tmem + TM_O, sdesc_sw128(a), sdesc_sw128(vb + kk * 2048), ID_O,
                                (it > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar.o_done);
                mma_commit(bar.v_empty + st);
            }
            // Every MMA issued above completes before TMEM is released.
            mma_commit(bar.drain);
            const int zero = 0;
            mbar_wait(bar.drain, 0, &zero, wait_ns);
            if (!ok) fail(p, abort_flag);
        }
    } else if (warp >= 4) {
        // ===================== softmax warps ====================================
        const int wq = warp - 4;          // TMEM lane quarter of this warp
        const int row = wq * 32 + lane;   // query row within the tile
        const int i = i0 + row;           // query index within the segment
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + TM_S;
        // This warp's rows need window columns [96-32wq, 96-32wq+160).
        const uint32_t tW = tmem + lane_off + TM_W + (uint32_t)(96 - 32 * wq);
        const uint32_t tO = tmem + lane_off + TM_O;
        const uint32_t skew = smem_u32(smem + OFF_SKEW) + (uint32_t)row * SKEW_STRIDE * 4;
        // Reading key y of a 32-key piece: column (31 - lane + y) of the two staged
        // window chunks.
        const uint32_t skew_rd = skew + (uint32_t)(31 - lane) * 4;

        bool ok = mbar_wait(bar.q_full, 0, abort_flag, wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            // q + u (in place) and q + v, rounded once to bf16.
            uint8_t *qrow = smem + OFF_Q + row * 128;
            uint8_t *qvrow = smem + OFF_QV + row * 128;
            const uint4 *uh = reinterpret_cast<const uint4 *>(p.u + h * DH);
            const uint4 *vh = reinterpret_cast<const uint4 *>(p.vb + h * DH);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int phys = c ^ (row & 7);
                const uint4 qq = *reinterpret_cast<const uint4 *>(qrow + phys * 16);
                const uint4 uu = __ldg(uh + c);
                const uint4 vv = __ldg(vh + c);
                const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
                const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
                const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                uint32_t ou[4], ov[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float ql = bf16lo(qw[e]), qh = bf16hi(qw[e]);
                    ou[e] = pack_bf16x2(ql + bf16lo(uw[e]), qh + bf16hi(uw[e]));
                    ov[e] = pack_bf16x2(ql + bf16lo(vw[e]), qh + bf16hi(vw[e]));
                }
                *reinterpret_cast<uint4 *>(qrow + phys * 16) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                *reinterpret_cast<uint4 *>(qvrow + phys * 16) =
                    make_uint4(ov[0], ov[1], ov[2], ov[3]);
            }
            fence_proxy_async_smem();
        }
        mbar_arrive(bar.q_ready);

        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;  // running max (log2 units), lazily updated
        float l_sum = 0.f;
        const uint32_t p_row = smem_u32(smem + OFF_P) + (uint32_t)row * 128;

        for (int it = 0; it < T && ok; ++it) {
            const int j0 = (t_begin + it) * BN;
            ok = __all_sync(0xffffffffu, mbar_wait(bar.s_full, it & 1, abort_flag, wait_ns));
            if (!ok) break;
            tc_fence_after_sync();

            // ---- gather: x[jj] = S[row][jj] + W[row][jj + 127 - row] ------------
            float x[BN];
#pragma unroll
            for (int pc = 0; pc < BN / 32; ++pc) {
                uint32_t wa[32], wb[32];
                tmem_ld32(tW + 32 * pc, wa);
                tmem_ld32(tW + 32 * (pc + 1), wb);
                tmem_wait_ld();
                reg_fence(wa);
                reg_fence(wb);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(skew + c * 16, wa[4 * c], wa[4 * c + 1], wa[4 * c + 2],
                                 wa[4 * c + 3]);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(skew + 128 + c * 16, wb[4 * c], wb[4 * c + 1], wb[4 * c + 2],
                                 wb[4 * c + 3]);
                uint32_t s[32];
                tmem_ld32(tS + 32 * pc, s);
                tmem_wait_ld();
                reg_fence(s);
#pragma unroll
                for (int y = 0; y < 32; ++y)
                    x[32 * pc + y] = __uint_as_float(s[y]) + ld_shared_f32(skew_rd + y * 4);
            }
            tc_fence_before_sync();
            mbar_arrive(bar.s_free);

            // ---- scale, mask, tile max ------------------------------------------
            const bool need_mask = (j0 + BN - 1 > i0 + p.M) || (j0 + BN > p.K);
            float mt = -INFINITY;
            if (need_mask) {
                const int jlim = min(i + p.M, p.K - 1) - j0;  // last visible key (tile-local)
#pragma unroll
                for (int jj = 0; jj < BN; ++jj) {
                    x[jj] = (jj <= jlim) ? x[jj] * sl2 : -INFINITY;
                    mt = fmaxf(mt, x[jj]);
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < BN; ++jj) {
                    x[jj] *= sl2;
                    mt = fmaxf(mt, x[jj]);
                }
            }
            // Lazy rescale: move the reference max only when the tile max exceeds
            // it by more than 8 (a factor 256); exact after the final division.
            float alpha = 1.f;
            const bool resc = mt > m_ref + 8.f;
            if (resc) {
                alpha = ex2(m_ref - mt);  // 0 when m_ref is -inf
                l_sum *= alpha;
                m_ref = mt;
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;

            // PV of the previous tile must be done: it reads P and writes O.
            if (it > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar.o_done, (it - 1) & 1, abort_flag, wait_ns));
                if (!ok) break;
                tc_fence_after_sync();
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

            // ---- exponentiate, row sum, P (bf16, 128-byte swizzled K-major) -----
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < BN / 8; ++c) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2(x[8 * c + 2 * e] - mu);
                    const float p1 = ex2(x[8 * c + 2 * e + 1] - mu);
                    rs += p0 + p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                const int half = c >> 3;
                const int phys = (c & 7) ^ (row & 7);
                st_shared_v4(p_row + half * TILE + phys * 16, pk[0], pk[1], pk[2], pk[3]);
            }
            l_sum += rs;
            fence_proxy_async_smem();
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

// Merge of split-key partial results: out = sum_s w_s o_s / sum_s w_s with
// w_s = 2^(lse_s - max lse).  One warp per query row, two columns per lane.
__global__ void relattn_combine_kernel(const float *__restrict__ part_o,
                                       const float *__restrict__ part_lse,
                                       __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                                       int n_splits, int rows)
{
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float mx = -INFINITY;
    for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, part_lse[(size_t)s * rows + row]);
    float wsum = 0.f, a0 = 0.f, a1 = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float l = part_lse[(size_t)s * rows + row];
        if (l == -INFINITY) continue;
        const float w = exp2f(l - mx);
        const float2 o = reinterpret_cast<const float2 *>(part_o + ((size_t)s * rows + row) * DH)[lane];
        wsum += w;
        a0 += w * o.x;
        a1 += w * o.y;
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    reinterpret_cast<__nv_bfloat162 *>(out + (size_t)row * DH)[lane] =
        __floats2bfloat162_rn(a0 * inv, a1 * inv);
    if (lse && lane == 0)
        lse[row] = (wsum > 0.f) ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
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

cudaError_t launch_wait_probe(unsigned int *status, unsigned long long wait_ns, cudaStream_t s)
{
    wait_probe_kernel<<<1, 32, 0, s>>>(status, wait_ns);
    return cudaGetLastError();
}

cudaError_t launch_relattn_combine(const float *part_o, const float *part_lse,
                                   __nv_bfloat16 *out, float *lse, int n_splits, int rows,
                                   cudaStream_t s)
{
    const int warps = 8;
    const int blocks = (rows + warps - 1) / warps;
    relattn_combine_kernel<<<blocks, warps * 32, 0, s>>>(part_o, part_lse, out, lse, n_splits,
                                                         rows);
    return cudaGetLastError();
}

} // namespace txl
