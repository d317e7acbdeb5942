// Relative-position attention for short segments (L <= 8 queries) against a
// long memory on the tensor cores ("Transformer-XL: Attentive Language Models
// Beyond a Fixed-Length Context", §3.2 evaluation with a long memory, §3.3
// score, Appendix B reversed table).
//
// The work is reading k, v and the table once; what limits the CUDA-core
// decode kernel from three queries on is its per-key arithmetic, which grows
// with L.  Here each 32-key chunk costs the same 52 warp-level MMAs
// (mma.sync m16n8k16, bf16 in, fp32 accumulate) for every L up to 8, so the
// kernel stays bound by the copies.  (These are the sm_80-form warp MMAs, not
// tcgen05: a tcgen05 tile is 64 or 128 rows, 90 % padding at L <= 8, and its
// accumulator lives in TMEM, while the online softmax here wants the scores in
// registers in exactly the layout of the next MMA's A operand.)
//
// Layout of one warp's MMAs.  The 16 rows of the A operand are the queries:
// row i (< L) holds the bf16 rounding of q_i + u (content) or q_i + v
// (position), formed in fp32, and row i + 8 the bf16 rounding of what that
// left over, so rows i and i + 8 of a product sum to the fp32 q + u to about
// 2^-17 relative; the two rows land in the same lane of the accumulator
// fragment.  Per chunk:
//   content  (q_i + u).k_j       4 key tiles x 4 dimension steps   16 MMAs
//   position (q_i + v).r_t       5 tiles of table rows t (40) x 4   20 MMAs
// The Appendix B shift: key j of row i takes table row j + L-1-i of the
// chunk's window; the position products go through a small shared-memory
// scratch (8 rows x 40 fp32) and are read back shifted by row.  The score
// fragment is then the A operand of P.V: probabilities rounded to bf16 in rows
// i, their residual in rows i + 8 (again summed in the output), V^T via
// transposing shared-memory matrix loads:
//   P.V      2 key steps x 8 tiles of output dimensions             16 MMAs
// Online softmax per row in fp32: the four lanes of a quad hold row i.
//
// Copies: per warp a ring of two stages, each filled by three TMA tensor
// copies (k and v boxes of 32 rows, the table's 40) completing on one
// mbarrier; 128-byte swizzle, so the matrix loads are bank-conflict free.
// Rows past the tensors' ends arrive as zeros.  The merge of the block's warps
// and of split key ranges is the one the CUDA-core decode kernel uses.
#include "decode_common.cuh"

#include <utility>

namespace txl {
namespace {

using namespace ptx;
using namespace decode;

constexpr int NSTG = 2;                                   // ring stages per warp
constexpr int TROWS = kDecodeMmaTableBox;                 // 40 table rows per chunk
constexpr int ST_K = 0;                                   // stage: 32 k rows,
constexpr int ST_V = ST_K + kDecodeMmaKeyBox * ROWB;      // 32 v rows,
constexpr int ST_R = ST_V + kDecodeMmaKeyBox * ROWB;      // 40 table rows
constexpr int STAGE = ST_R + TROWS * ROWB;                // 13312 bytes
constexpr int RING = NSTG * STAGE;                        // per warp
constexpr int OFF_BAR = WARPS * RING;
constexpr int OFF_RES = OFF_BAR + WARPS * NSTG * 8;       // BlockRes
constexpr int OFF_FLAG = OFF_RES + (int)sizeof(BlockRes);
constexpr int SMEM_USED = OFF_FLAG + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;              // slack for the manual alignment
constexpr int SCR_LD = 40;                                // scratch row stride (floats)

static_assert(GK == kDecodeMmaKeyBox, "one key box per chunk");
static_assert(GK + kDecodeMaxL - 1 <= TROWS, "the table box covers the shifted window");
static_assert(ST_V % 1024 == 0 && ST_R % 1024 == 0 && STAGE % 1024 == 0,
              "128-byte swizzled boxes need 1024-byte aligned destinations");
static_assert((int)sizeof(WarpRec) <= STAGE, "a warp's record fits in its ring");
static_assert(8 * SCR_LD * 4 <= TROWS * ROWB, "the shift scratch fits in the table box");

// m16n8k16 bf16 MMA, fp32 accumulators in place.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 bf16 matrices; lanes 8m .. 8m+7 give the row addresses of matrix m.
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

// Byte offset of 16-byte piece c of row `row` in a box written with the
// 128-byte swizzle (pieces of a row permuted by the row's index mod 8).
__device__ __forceinline__ uint32_t swz(int row, int c)
{
    return (uint32_t)(row * ROWB + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A bf16 pair as the (head, residual) split of two fp32 values: returns the
// rounded pair, `res` the rounding of what it left over.
__device__ __forceinline__ uint32_t split_bf16x2(float x0, float x1, uint32_t &res)
{
    const uint32_t hi = pack_bf16x2(x0, x1);
    res = pack_bf16x2(x0 - bf_lo(hi), x1 - bf_hi(hi));
    return hi;
}

// Two blocks per SM (shared memory allows two): with that bound the compiler
// keeps ~200 registers per thread instead of capping them at 128.
template <int L>
__global__ void __launch_bounds__(WARPS * 32, 2)
    relattn_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_r, const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;   // accumulator row (query) and column pair
    const int split = blockIdx.x % p.n_splits;
    const int bh = blockIdx.x / p.n_splits;
    const int h = bh % p.H;
    const Range rg = key_range(p.K, p.n_splits, split, warp);
    TXL_CHECK(rg.k_begin >= 0 && rg.k_end <= p.K && bh < p.B * p.H && split < p.n_splits, p.status);

    uint8_t *ring = smem + warp * RING;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR) + warp * NSTG;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0) {
        for (int s = 0; s < NSTG; ++s) mbar_init(bars + s, 1);
        fence_barrier_init();
    }
    __syncthreads();

    const uint64_t pol_stream = policy_evict_first();  // k, v: read once
    const uint64_t pol_keep = policy_evict_last();     // table: shared by the batch
    // Copies of this warp's chunk n into stage n % NSTG (lane 0): keys j0 ..
    // j0 + 31 of plane bh, table rows r_off + j0 .. + 39 of head h.  Boxes are
    // always complete (rows past a tensor's end are zero-filled), so the
    // transaction count is the stage size.
    auto issue = [&](int n) {
        const int j0 = rg.k_begin + (warp + WARPS * n) * GK;
        uint8_t *stg = ring + (n % NSTG) * STAGE;
        uint64_t *bar = bars + n % NSTG;
        TXL_CHECK(j0 >= rg.k_begin && j0 < rg.k_end && p.r_off + j0 < p.r_rows, p.status);
        mbar_arrive_expect_tx(bar, (uint32_t)STAGE);
        tma_load_3d_hint(stg + ST_K, &tm_k, bar, 0, j0, bh, pol_stream);
        tma_load_3d_hint(stg + ST_V, &tm_v, bar, 0, j0, bh, pol_stream);
        tma_load_3d_hint(stg + ST_R, &tm_r, bar, 0, p.r_off + j0, h, pol_keep);
    };
    int issued = 0;
    if (lane == 0)
        for (; issued < min(NSTG, rg.n_mine); ++issued) issue(issued);
    issued = __shfl_sync(0xffffffffu, issued, 0);

    // A operands, constant over the keys: per 16-dimension step ks, rows g and
    // g + 8 of (q_g + u) and of (q_g + v) as head and residual, dimensions
    // 16 ks + 2t, +1 (registers 0, 1) and 16 ks + 8 + 2t, +1 (registers 2, 3).
    uint32_t a_u[4][4], a_v[4][4];
    {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + ((size_t)bh * L + g) * DH);
        const uint32_t *urow = reinterpret_cast<const uint32_t *>(p.u + (size_t)h * DH);
        const uint32_t *vrow = reinterpret_cast<const uint32_t *>(p.vb + (size_t)h * DH);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int w = (16 * ks + 8 * half + 2 * t) / 2;  // bf16-pair index
                uint32_t hu = 0, ru = 0, hv = 0, rv = 0;
                if (g < L) {
                    const uint32_t qw = qrow[w], uw = urow[w], vw = vrow[w];
                    hu = split_bf16x2(bf_lo(qw) + bf_lo(uw), bf_hi(qw) + bf_hi(uw), ru);
                    hv = split_bf16x2(bf_lo(qw) + bf_lo(vw), bf_hi(qw) + bf_hi(vw), rv);
                }
                a_u[ks][2 * half] = hu;
                a_u[ks][2 * half + 1] = ru;
                a_v[ks][2 * half] = hv;
                a_v[ks][2 * half + 1] = rv;
            }
        }
    }

    // Running maximum (log2 units) and this lane's part of the sum for row g;
    // output accumulators of dimensions 8 nd + 2t, +1 (rows g and g + 8).
    float m_run = -INFINITY, l_run = 0.f;
    float acc[8][4];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nd][e] = 0.f;
    const int lr = lane & 7, lm = lane >> 3;  // matrix-load roles: row, matrix
    const int shift = (g < L) ? L - 1 - g : 0;

    bool ok = true;
    for (int n = 0; n < rg.n_mine; ++n) {
        const int j0 = rg.k_begin + (warp + WARPS * n) * GK;
        ok = __all_sync(0xffffffffu, mbar_wait(bars + n % NSTG, (n / NSTG) & 1, abort_flag, p.wait_ns));
        if (!ok) break;
        uint8_t *stg = ring + (n % NSTG) * STAGE;
        const uint32_t sk = smem_u32(stg + ST_K), sv = smem_u32(stg + ST_V), sr = smem_u32(stg + ST_R);

        // ---- content: (q + u).k for keys 8 nt + 2t, +1 --------------------------
        float sc[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const int row = 8 * nt + lr;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t b[4];
                ldsm_x4(b, sk + swz(row, 4 * h2 + lm));
                mma16816(c, a_u[2 * h2], b[0], b[1]);
                mma16816(c, a_u[2 * h2 + 1], b[2], b[3]);
            }
            sc[nt][0] = c[0] + c[2];
            sc[nt][1] = c[1] + c[3];
        }
        // ---- position: (q + v).r for the chunk's 40 table rows ------------------
        float ps[5][2];
#pragma unroll
        for (int nt = 0; nt < 5; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const int row = 8 * nt + lr;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t b[4];
                ldsm_x4(b, sr + swz(row, 4 * h2 + lm));
                mma16816(c, a_v[2 * h2], b[0], b[1]);
                mma16816(c, a_v[2 * h2 + 1], b[2], b[3]);
            }
            ps[nt][0] = c[0] + c[2];
            ps[nt][1] = c[1] + c[3];
        }
        // ---- Appendix B shift through the scratch (over the read table box) ---
        float *scr = reinterpret_cast<float *>(stg + ST_R);
        __syncwarp();  // every lane's table reads are done
#pragma unroll
        for (int nt = 0; nt < 5; ++nt)
            *reinterpret_cast<float2 *>(scr + g * SCR_LD + 8 * nt + 2 * t) = make_float2(ps[nt][0], ps[nt][1]);
        __syncwarp();
        float s[4][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * t + e;
                TXL_CHECK(g * SCR_LD + j + shift < 8 * SCR_LD && j + shift < TROWS, p.status);
                float x = (sc[nt][e] + scr[g * SCR_LD + j + shift]) * p.scale_log2;
                const int jg = j0 + j;
                if (jg >= rg.k_end || jg > p.M + g) x = -INFINITY;
                s[nt][e] = x;
                mx = fmaxf(mx, x);
            }
        }
        // ---- online softmax of row g over the quad ------------------------------
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        // No branch for a row that has seen no visible key yet (m_new = -inf):
        // the selects give scale 0 and probabilities 0.
        const float rescale = (m_run == -INFINITY) ? 0.f : ex2f(m_run - m_new);
        m_run = m_new;
        float psum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = (s[nt][e] == -INFINITY) ? 0.f : ex2f(s[nt][e] - m_new);
                psum += s[nt][e];
            }
        l_run = l_run * rescale + psum;
#pragma unroll
        for (int nd = 0; nd < 8; ++nd)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nd][e] *= rescale;

        // ---- P.V: keys 16 kk .. 16 kk + 15, probabilities as head + residual ---
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t a[4];
            a[0] = split_bf16x2(s[2 * kk][0], s[2 * kk][1], a[1]);
            a[2] = split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], a[3]);
            const int row = 16 * kk + (lm & 1) * 8 + lr;
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, sv + swz(row, 2 * np + (lm >> 1)));
                mma16816(acc[2 * np], a, b[0], b[1]);
                mma16816(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
        // The stage is read (and the scratch used): order this lane's accesses
        // before the copy that refills it.
        fence_proxy_async_smem();
        __syncwarp();
        if (n + NSTG < rg.n_mine) {
            if (lane == 0) issue(n + NSTG);
            ++issued;
        }
    }
    if (!ok) {
        // Time-out: record it, and let this warp's copies still in flight land
        // before the block's shared memory is reused or released (bounded waits).
        if (lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, TXL_STATUS_TIMEOUT);
            const int zero = 0;
            for (int n = max(0, issued - NSTG); n < issued; ++n)
                mbar_wait(bars + n % NSTG, (n / NSTG) & 1, &zero, p.wait_ns);
        }
        __syncwarp();
    }

    // ---- this warp's record, in its own ring (its copies have all landed) ------
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    WarpRec *mine = reinterpret_cast<WarpRec *>(ring);
    if (g < L) {
        if (t == 0) {
            mine->m[g] = m_run;
            mine->l[g] = l_run;
        }
#pragma unroll
        for (int nd = 0; nd < 8; ++nd)
            *reinterpret_cast<float2 *>(&mine->a[g][8 * nd + 2 * t]) =
                make_float2(acc[nd][0] + acc[nd][2], acc[nd][1] + acc[nd][3]);
    }
    const auto rec = [smem](int w) { return reinterpret_cast<const WarpRec *>(smem + w * RING); };
    finish_block<L>(rec, reinterpret_cast<BlockRes *>(smem + OFF_RES), p, bh, split, warp, lane);
}

template <int L>
cudaError_t set_smem_l()
{
    return cudaFuncSetAttribute(relattn_decode_mma_kernel<L>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

template <int L>
int blocks_per_sm_l()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, relattn_decode_mma_kernel<L>, WARPS * 32,
                                                      SMEM_BYTES) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

template <int L>
cudaError_t launch_l(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tr,
                     const DecodeParams &p, cudaStream_t s)
{
    const long long blocks = (long long)p.B * p.H * p.n_splits;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (!p.cluster) {
        relattn_decode_mma_kernel<L><<<(unsigned)blocks, WARPS * 32, SMEM_BYTES, s>>>(tk, tv, tr, p);
        return cudaGetLastError();
    }
    // one cluster of n_splits blocks per (batch, head)
    if (p.n_splits < 2 || p.n_splits > kDecodeMaxCluster) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(WARPS * 32, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.n_splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, relattn_decode_mma_kernel<L>, tk, tv, tr, p);
}

// Instances L = 1 .. kDecodeMaxL, indexed by L - 1.
template <int... I>
struct Table {
    static constexpr cudaError_t (*set_smem[])() = {set_smem_l<I + 1>...};
    static constexpr int (*blocks[])() = {blocks_per_sm_l<I + 1>...};
    static constexpr cudaError_t (*launch[])(const CUtensorMap &, const CUtensorMap &,
                                             const CUtensorMap &, const DecodeParams &,
                                             cudaStream_t) = {launch_l<I + 1>...};
};
template <int... I>
Table<I...> make_table(std::integer_sequence<int, I...>);
using Inst = decltype(make_table(std::make_integer_sequence<int, kDecodeMaxL>{}));

// The dynamic shared-memory attribute of every instance, once per device.
cudaError_t ensure_smem_attr()
{
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    for (int l = 0; l < kDecodeMaxL; ++l)
        if ((e = Inst::set_smem[l]()) != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
    return cudaSuccess;
}

} // namespace

int decode_mma_blocks_per_sm(int L)
{
    static int cache[kDecodeMaxL + 1] = {};  // per query count; one device per process
    if (L < 1 || L > kDecodeMaxL) return 1;
    if (!cache[L]) cache[L] = (ensure_smem_attr() == cudaSuccess) ? Inst::blocks[L - 1]() : 1;
    return cache[L];
}

cudaError_t launch_relattn_decode_mma(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_r, const DecodeParams &p,
                                      cudaStream_t s)
{
    if (p.L < 1 || p.L > kDecodeMaxL) return cudaErrorInvalidValue;
    const cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    return Inst::launch[p.L - 1](tm_k, tm_v, tm_r, p, s);
}

} // namespace txl
