// Relative-position attention for one new query (L = 1; the kernel is written
// for any small L) against a long memory: the decode pattern of generation,
// one new token per step attending to the cached M states ("Transformer-XL: Attentive Language
// Models Beyond a Fixed-Length Context", §3.2 recurrence and evaluation with a
// long memory, §3.3 score, Appendix B reversed table).
//
// With so few query rows the work is reading K, V and the table once: the
// kernel is HBM-bound and runs on the CUDA cores in fp32.  Every warp works on
// its own: it takes 32 keys at a time (a chunk) and streams each chunk's k and
// v rows and the L + 31 table rows they need into a ring of shared-memory
// stages with contiguous bulk copies (cp.async.bulk, one mbarrier per stage),
// so that the next chunk's bytes are in flight while the current one is
// computed and no registers are held by loads.  The warp's lanes form four
// groups of eight; group g takes keys 8g..8g+7 of the chunk and lane s of a
// group dimensions 8s..8s+7 (16-byte shared-memory reads).  For query row i
// and key j the score is
//   A_ij = (q_i + u).k_j + (q_i + v).r[r_off + L-1 - i + j]        (j <= M + i)
// where r is the reversed table (row K-1-d holds distance d; r_off = r_rows-K):
// the Appendix B left shift by L-1-i is the table row index.  q + u and q + v
// are formed in fp32 and never rounded (packed f32x2 FMAs).  Each lane sums its
// eight dimensions of its group's eight keys; a transposing butterfly over the
// group leaves lane l with the whole score of key l.  Online softmax per row
// over the warp, P.V with each group's probabilities broadcast by shuffles
// into per-group partial outputs (summed over the groups at the end), then the
// block's warps merge their partial results
// and the block writes the output, or its key range's normalised partial and
// log2-sum-exp for the merge kernel.  The per-key work grows with L while the
// bytes do not: from L = 2 on the warp-MMA kernel (relattn_decode_mma.cu) is
// the faster path, so only L = 1 is instantiated.
#include "decode_common.cuh"

#include <utility>

namespace txl {
namespace {

using namespace ptx;
using namespace decode;

constexpr int FMAX = kDecodeFmaMaxL;  // longest segment this kernel takes
constexpr int NSTG = 2;           // ring stages per warp
constexpr int RROWS = GK + FMAX - 1;
constexpr int ST_K = 0;                         // stage layout: 32 k rows,
constexpr int ST_V = ST_K + GK * ROWB;          // 32 v rows,
constexpr int ST_R = ST_V + GK * ROWB;          // up to 37 table rows
constexpr int STAGE = ST_R + RROWS * ROWB;      // 12928 bytes
constexpr int RING = NSTG * STAGE;              // per warp
constexpr int OFF_BAR = WARPS * RING;
constexpr int OFF_MERGE = OFF_BAR + WARPS * NSTG * 8;   // WarpRec per warp
constexpr int OFF_RES = OFF_MERGE + WARPS * (int)sizeof(WarpRec);   // BlockRes
constexpr int OFF_FLAG = OFF_RES + (int)sizeof(BlockRes);
constexpr int SMEM_BYTES = OFF_FLAG + 16;

static_assert(STAGE % 16 == 0 && RING % 16 == 0, "bulk copies need 16-byte aligned stages");

// Maximum of v over the warp in one instruction (sm_100 family).
__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed pairs of fp32 (f32x2 arithmetic).
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

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// bf16 pair (dims 2c, 2c+1) as an fp32 pair.
__device__ __forceinline__ uint64_t widen(uint32_t w) { return pack2(lo_f(w), hi_f(w)); }

__device__ __forceinline__ uint32_t word(const uint4 &v, int c)
{
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// The lanes of an 8-lane group hold v[0..7], their shares of 8 sums; afterwards
// lane s of the group holds the whole sum number s.  Three butterfly stages: a
// lane keeps the half of its values whose index bit matches its own lane bit
// and sends the other half.
__device__ __forceinline__ float transpose_reduce8(float (&v)[8], int sub)
{
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) {
        const bool up = (sub & o) != 0;
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
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.n_splits;
    const int bh = blockIdx.x / p.n_splits;
    const int h = bh % p.H;
    const int K = p.K;
    // Key range of this block: a whole number of 32-key chunks, dealt to the
    // block's warps in turn (chunk c to warp c mod 4).
    const int span = decode_span(K, p.n_splits);
    const int k_begin = split * span, k_end = min(K, k_begin + span);
    const int n_chunks = (k_end > k_begin) ? (k_end - k_begin + GK - 1) / GK : 0;
    const int n_mine = (n_chunks > warp) ? (n_chunks - warp + WARPS - 1) / WARPS : 0;
    TXL_CHECK(k_begin >= 0 && k_end <= K && bh < p.B * p.H && split < p.n_splits, p.status);

    const uint8_t *kg = reinterpret_cast<const uint8_t *>(p.k) + (size_t)bh * p.kv_stride * 2;
    const uint8_t *vg = reinterpret_cast<const uint8_t *>(p.v) + (size_t)bh * p.kv_stride * 2;
    const uint8_t *rg = reinterpret_cast<const uint8_t *>(p.r) + ((size_t)h * p.r_rows + p.r_off) * ROWB;
    uint8_t *ring = smem + warp * RING;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR) + warp * NSTG;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);

    // Zero this warp's ring once: rows a chunk does not copy (past the key
    // range) are then finite, so their zero probabilities give exact zeros.
    for (int o = lane * 16; o < RING; o += 32 * 16)
        *reinterpret_cast<uint4 *>(ring + o) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0) {
        for (int s = 0; s < NSTG; ++s) mbar_init(bars + s, 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();  // the zeros before the copies that overwrite them
    __syncthreads();

    const uint64_t pol_stream = policy_evict_first();  // k, v: read once
    const uint64_t pol_keep = policy_evict_last();     // table: shared by the batch
    // Copies of this warp's chunk n into stage n % NSTG (lane 0).  Only rows of
    // the block's range and of the table are copied.
    auto issue = [&](int n) {
        const int j0 = k_begin + (warp + WARPS * n) * GK;
        uint8_t *stg = ring + (n % NSTG) * STAGE;
        const int rows = min(GK, k_end - j0);
        const int rrows = min(min(GK + L - 1, K - j0), k_end - j0 + L - 1);
        // key rows of this block's range; table rows inside the table
        TXL_CHECK(j0 >= k_begin && rows > 0 && j0 + rows <= k_end && rrows >= rows &&
                      rrows <= GK + L - 1 && p.r_off + j0 + rrows <= p.r_rows,
                  p.status);
        mbar_arrive_expect_tx(bars + n % NSTG, (uint32_t)(2 * rows + rrows) * ROWB);
        bulk_load_hint(stg + ST_K, kg + (size_t)j0 * ROWB, rows * ROWB, bars + n % NSTG, pol_stream);
        bulk_load_hint(stg + ST_V, vg + (size_t)j0 * ROWB, rows * ROWB, bars + n % NSTG, pol_stream);
        bulk_load_hint(stg + ST_R, rg + (size_t)j0 * ROWB, rrows * ROWB, bars + n % NSTG, pol_keep);
    };
    int issued = 0;
    if (lane == 0)
        for (; issued < min(NSTG, n_mine); ++issued) issue(issued);
    issued = __shfl_sync(0xffffffffu, issued, 0);

    // q + u and q + v of this lane's eight dimensions (four fp32 pairs), every row.
    const int g = lane >> 3, sub = lane & 7;
    uint64_t qu[L][4], qv[L][4];
    {
        const uint4 uu = reinterpret_cast<const uint4 *>(p.u)[h * (DH / 8) + sub];
        const uint4 vb = reinterpret_cast<const uint4 *>(p.vb)[h * (DH / 8) + sub];
#pragma unroll
        for (int i = 0; i < L; ++i) {
            const uint4 qq = reinterpret_cast<const uint4 *>(p.q)[((size_t)bh * L + i) * (DH / 8) + sub];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t w = word(qq, c), wu = word(uu, c), wv = word(vb, c);
                qu[i][c] = pack2(lo_f(w) + lo_f(wu), hi_f(w) + hi_f(wu));
                qv[i][c] = pack2(lo_f(w) + lo_f(wv), hi_f(w) + hi_f(wv));
            }
        }
    }

    // running max (log2 units, warp-uniform) and this lane's part of the sum per
    // row (summed over the warp once, after the keys); this group's partial
    // output of dimensions 8 sub .. 8 sub + 7 (four pairs) per row
    float m[L], l[L];
    uint64_t acc[L][4];
#pragma unroll
    for (int i = 0; i < L; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0;  // +0.0f pairs
    }

    bool ok = true;
    for (int n = 0; n < n_mine; ++n) {
        const int j0 = k_begin + (warp + WARPS * n) * GK;
        ok = __all_sync(0xffffffffu, mbar_wait(bars + n % NSTG, (n / NSTG) & 1, abort_flag, p.wait_ns));
        if (!ok) break;
        // this lane's 16 bytes of row 8g + s of each block of the stage
        const uint32_t stg = smem_u32(ring + (n % NSTG) * STAGE) + (uint32_t)(8 * g * ROWB + 16 * sub);

        // ---- scores: this lane's words of its group's k and table rows --------
        float sc_row[L];
        {
            uint4 kq[8], rq[8 + L - 1];
#pragma unroll
            for (int e = 0; e < 8; ++e) kq[e] = ld_shared_v4(stg + ST_K + e * ROWB);
            // table row for (i, key 8g + e) is 8g + e + L-1-i
#pragma unroll
            for (int e = 0; e < 8 + L - 1; ++e) rq[e] = ld_shared_v4(stg + ST_R + e * ROWB);
#pragma unroll
            for (int i = 0; i < L; ++i) {
                float part[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    uint64_t a = 0;
#pragma unroll
                    for (int c = 0; c < 4; ++c) a = fma2(widen(word(kq[e], c)), qu[i][c], a);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        a = fma2(widen(word(rq[e + L - 1 - i], c)), qv[i][c], a);
                    float x0, x1;
                    unpack2(a, x0, x1);
                    part[e] = x0 + x1;
                }
                sc_row[i] = transpose_reduce8(part, sub) * p.scale_log2;  // key j0 + lane
            }
        }
        // ---- the group's v rows (after the scores: fewer live registers) ------
        uint4 vq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) vq[e] = ld_shared_v4(stg + ST_V + e * ROWB);
        // The stage is read: order the reads before the copy that refills it.
        fence_proxy_async_smem();
        __syncwarp();
        if (n + NSTG < n_mine) {
            if (lane == 0) issue(n + NSTG);
            ++issued;
        }

#pragma unroll
        for (int i = 0; i < L; ++i) {
            float s = sc_row[i];
            const int j = j0 + lane;
            if (j >= k_end || j > p.M + i) s = -INFINITY;
            // ---- online softmax over the warp's 32 keys --------------------------
            const float mx = warp_max(s);
            // No branch for a query that has seen no visible key yet (m_new = -inf):
            // the selects below then give sc = 0 and pj = 0, which leave l and acc at
            // zero, and without control flow the L queries' chains interleave.
            const float m_new = fmaxf(m[i], mx);
            const float sc = (m[i] == -INFINITY) ? 0.f : ex2f(m[i] - m_new);
            const float pj = (s == -INFINITY) ? 0.f : ex2f(s - m_new);
            m[i] = m_new;
            l[i] = l[i] * sc + pj;
            const uint64_t sc2 = pack2(sc, sc);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[i][c] = mul2(acc[i][c], sc2);
            // ---- P.V: probability of key 8g + e from lane 8g + e ----------------
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float pe = __shfl_sync(0xffffffffu, pj, (lane & 24) + e);
                const uint64_t pe2 = pack2(pe, pe);
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i][c] = fma2(widen(word(vq[e], c)), pe2, acc[i][c]);
            }
        }
    }
    if (!ok) {
        // Time-out: record it, and let this warp's copies still in flight land
        // before the block's shared memory is released (bounded waits).
        if (lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, 1u);
            const int zero = 0;
            for (int n = max(0, issued - NSTG); n < issued; ++n)
                mbar_wait(bars + n % NSTG, (n / NSTG) & 1, &zero, p.wait_ns);
        }
        __syncwarp();
    }

    // ---- sum the four groups' partial outputs (same running max) -------------
    float o8[L][8];
#pragma unroll
    for (int i = 0; i < L; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], o);
#pragma unroll
        for (int c = 0; c < 4; ++c) unpack2(acc[i][c], o8[i][2 * c], o8[i][2 * c + 1]);
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            o8[i][d] += __shfl_xor_sync(0xffffffffu, o8[i][d], 8);
            o8[i][d] += __shfl_xor_sync(0xffffffffu, o8[i][d], 16);
        }
    }

    // ---- this warp's record for the block merge ---------------------------------
    WarpRec *mine = reinterpret_cast<WarpRec *>(smem + OFF_MERGE) + warp;
#pragma unroll
    for (int i = 0; i < L; ++i) {
        if (lane == 0) {
            mine->m[i] = m[i];
            mine->l[i] = l[i];
        }
        if (g == 0) {
            float4 *dst = reinterpret_cast<float4 *>(mine->a[i] + 8 * sub);
            dst[0] = make_float4(o8[i][0], o8[i][1], o8[i][2], o8[i][3]);
            dst[1] = make_float4(o8[i][4], o8[i][5], o8[i][6], o8[i][7]);
        }
    }
    const uint8_t *const merge = smem + OFF_MERGE;
    const auto rec = [merge](int w) { return reinterpret_cast<const WarpRec *>(merge) + w; };
    finish_block<L>(rec, reinterpret_cast<BlockRes *>(smem + OFF_RES), p, bh, split, warp, lane);
}

template <int L>
cudaError_t set_smem_l()
{
    return cudaFuncSetAttribute(relattn_decode_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_BYTES);
}

template <int L>
int blocks_per_sm_l()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, relattn_decode_kernel<L>, WARPS * 32,
                                                      SMEM_BYTES) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

template <int L>
cudaError_t launch_l(const DecodeParams &p, cudaStream_t s)
{
    const long long blocks = (long long)p.B * p.H * p.n_splits;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (!p.cluster) {
        relattn_decode_kernel<L><<<(unsigned)blocks, WARPS * 32, SMEM_BYTES, s>>>(p);
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
    return cudaLaunchKernelEx(&cfg, relattn_decode_kernel<L>, p);
}

// Instances L = 1 .. FMAX, indexed by L - 1.
template <int... I>
struct Table {
    static constexpr cudaError_t (*set_smem[])() = {set_smem_l<I + 1>...};
    static constexpr int (*blocks[])() = {blocks_per_sm_l<I + 1>...};
    static constexpr cudaError_t (*launch[])(const DecodeParams &, cudaStream_t) = {launch_l<I + 1>...};
};
template <int... I>
Table<I...> make_table(std::integer_sequence<int, I...>);
using Inst = decltype(make_table(std::make_integer_sequence<int, FMAX>{}));

// The dynamic shared-memory attribute of every instance, once per device.
cudaError_t ensure_smem_attr()
{
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    for (int l = 0; l < FMAX; ++l)
        if ((e = Inst::set_smem[l]()) != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
    return cudaSuccess;
}

} // namespace

int decode_chunk_keys() { return GK; }

int decode_blocks_per_sm(int L)
{
    static int cache[FMAX + 1] = {};  // per query count; one device per process
    if (L < 1 || L > FMAX) return 1;
    if (!cache[L]) cache[L] = (ensure_smem_attr() == cudaSuccess) ? Inst::blocks[L - 1]() : 1;
    return cache[L];
}

cudaError_t launch_relattn_decode(const DecodeParams &p, cudaStream_t s)
{
    if (p.L < 1 || p.L > FMAX) return cudaErrorInvalidValue;
    const cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    return Inst::launch[p.L - 1](p, s);
}

} // namespace txl
