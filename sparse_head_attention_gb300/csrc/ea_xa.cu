// ea_xa.cu - XA block-mask estimation for EA_BLOCK heads: antidiagonal scores
// of 16 x 16 cells on the tensor cores, then per-row threshold selection of
// 128 x 128 key blocks.
//
// "Paper Reading - Elastic Attention: Test-time Adaptive Sparsity Ratios"
// names XA as XAttention, a training-free block-sparse attention that picks key
// blocks by antidiagonal scoring (Glossary "XA"), with stride 16 and threshold
// 0.9 (§07 Table 8).  The scoring is not written out there; this computes the
// reading stated in ea.h (ea_xa_estimate):
//   A[a][c]   = (scale / 16) * sum_{u<16} q[16a+u] . k[16c+15-u]
//   P[a][c]   = softmax over cells c <= a of A[a][c]
//   W[qb][kb] = sum of P over the cells of block (qb, kb) and over the query
//               heads of the KV head
// then, per query-block row, the fewest blocks holding `threshold` of the row's
// W, highest first, plus the diagonal.
//
// Launches (one stream, no host synchronisation):
//   xa_setup_kernel   one warp: lists the (b, h) units whose mode is EA_BLOCK
//                     and re-arms the work queue.
//   xa_scores_kernel  persistent, one CTA per SM.  An item is one causal tile
//                     of 128 cell rows x 256 cell columns for one unit and pair
//                     of query heads, taken from an atomic queue; all items
//                     cost the same.  The MMA warp accumulates S_t = Q'_t K'^T
//                     in TMEM (M 128, N 256, K = 16 offsets x 128 dims, in 32
//                     chunks of 64): a cell row of Q' is one query offset u of
//                     its 16 tokens, a cell row of K' the key offset 15 - u,
//                     both fetched by TMA boxes over (dim, head, offset, cell,
//                     batch).  One warpgroup per head reduces the tile to, per
//                     cell row, its max m over the tile (log2 units), the sums
//                     over each 8-cell key block of exp2(A - m), and their
//                     total, and stores them.  The scores are computed once;
//                     the tiles' partial results are combined afterwards,
//                     which needs no second pass.
//   xa_select_kernel  one CTA per (unit, query block): each cell row's log2
//                     LSE from its tiles' (max, total) pairs, W[qb][kb] from
//                     the stored sums times exp2(m - lse), the row total, and
//                     the threshold selection by bisection over float bit
//                     patterns, equal scores taken in key-block order.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ea_device.cuh"
#include "ea_internal.h"

namespace ea {

constexpr int kXs = EA_XA_STRIDE;                 // tokens per cell edge
constexpr int kXRows = 128;                       // cell rows per item (MMA M)
constexpr int kXCols = 256;                       // cell columns per key tile (MMA N)
constexpr int kXCellsPerBlock = EA_TILE / kXs;    // 8 cells per 128-token block
constexpr int kXBlocksPerTile = kXCols / kXCellsPerBlock;   // 32 key blocks per key tile
constexpr int kXChunks = kXs * (EA_HEAD_DIM / 64);          // (offset, half of d): 32
constexpr int kXQBox = kXRows * 128;              // 128 rows x 64 bf16
constexpr int kXKBox = kXCols * 128;              // 256 rows x 64 bf16
constexpr int kXStages = 3;
constexpr int kXProducerWarp = 8;
constexpr int kXMmaWarp = 9;
constexpr int kXThreads = 320;
constexpr uint32_t kXTmemCols = 512;              // S of two heads, 256 columns each
constexpr uint32_t kIdescXa = idesc_bf16_f32(128, 256, false, false);
static_assert(kXBlocksPerTile == 32, "one keep word per key tile chunk");

struct __align__(1024) XaSmem {
    uint8_t q[kXStages][2][kXQBox];
    uint8_t k[kXStages][kXKBox];
    uint64_t full[kXStages], empty[kXStages];
    uint64_t s_full[2], s_free[2];
    uint64_t item_full[2], item_empty[2];
    int item[2];
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kXaSmemBytes = sizeof(XaSmem) + 1024;

struct XaArgs {
    const uint8_t *m;
    ea_ws_header *hdr;
    int32_t *units;
    float *tsum, *rmax, *esum;
    uint8_t *block_mask;
    float *block_scores;
    int B, Hkv, g, npairs, max_units;
    int nA, nct, nB, nRT;
    int tiles;         // causal tiles of one (unit, pair): tile_off(nRT)
    int64_t tri;
    float c2;          // scale * log2(e) / stride: cell sums -> log2-domain scores
    float threshold;
};

// First stored sum of cell row a: rows hold 32 * (a / 256 + 1) sums each.
__device__ __forceinline__ int64_t xa_row_off(int64_t a)
{
    const int64_t grp = a >> 8, r = a & 255;
    return 32 * (256 * grp * (grp + 1) / 2 + r * (grp + 1));
}

__device__ __forceinline__ uint32_t xa_low_bits(int n)
{
    return n <= 0 ? 0u : n >= 32 ? 0xffffffffu : (1u << n) - 1u;
}

// Row tile rt reaches key tiles 0 .. rt / 2; tile_off(rt) counts the causal
// tiles of the row tiles before it: k (k + 1) for rt = 2k, (k + 1)^2 for 2k + 1.
__host__ __device__ __forceinline__ int64_t xa_tile_off(int64_t rt)
{
    const int64_t k = rt >> 1;
    return (rt & 1) ? (k + 1) * (k + 1) : k * (k + 1);
}

struct XaItem {
    int rt, ct, unit, b, h, qi0, nh;
};

// Items: (unit, pair) outermost, then row tile, then key tile.
__device__ __forceinline__ XaItem xa_decode(const XaArgs &a, int item)
{
    XaItem x;
    const int up = item / a.tiles;
    const int j = item % a.tiles;
    int lo = 0, hi = a.nRT;                 // tile_off(lo) <= j < tile_off(hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (xa_tile_off(mid) <= j)
            lo = mid;
        else
            hi = mid;
    }
    x.rt = lo;
    x.ct = j - static_cast<int>(xa_tile_off(lo));
    x.unit = up / a.npairs;
    const int pair = up % a.npairs;
    const int u = a.units[x.unit];
    x.b = u >> 16;
    x.h = u & 0xffff;
    x.qi0 = 2 * pair;
    x.nh = min(2, a.g - x.qi0);
    return x;
}

// ------------------------------------------------------------ setup
__global__ void xa_setup_kernel(XaArgs a)
{
    const int lane = threadIdx.x;
    const int n = a.B * a.Hkv;
    int count = 0;
    bool bad = false;
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const int mode = i < n ? a.m[i] : EA_FULL;
        bad |= mode > EA_BLOCK;
        const bool blk = mode == EA_BLOCK;
        const uint32_t bal = __ballot_sync(0xffffffffu, blk);
        const int pos = count + __popc(bal & ((1u << lane) - 1u));
        if (blk && pos < a.max_units)
            a.units[pos] = (i / a.Hkv) << 16 | (i % a.Hkv);
        count += __popc(bal);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        const int used = count < a.max_units ? count : a.max_units;
        if (bad || count > a.max_units)
            raise_error(&a.hdr->error, EA_DEVERR_CHECK);
        a.hdr->n_items = static_cast<uint32_t>(used) * a.npairs * a.tiles;
        a.hdr->reserved[0] = static_cast<uint32_t>(used);
        a.hdr->work_counter = 0;
        a.hdr->drained = 0;
    }
}

// ------------------------------------------------------------ score pass
__device__ __forceinline__ void xa_producer(const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                            const XaArgs &a, XaSmem &sm, int lane)
{
    uint32_t *err = &a.hdr->error;
    const uint32_t n_items = a.hdr->n_items;
    uint32_t kit = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&sm.item_empty[slot], ((it >> 1) & 1) ^ 1, &sm.abort, err))
            break;
        int item = -1;
        if (lane == 0) {
            const uint32_t x = atomicAdd(&a.hdr->work_counter, 1u);
            item = x < n_items ? static_cast<int>(x) : -1;
            sm.item[slot] = item;
            mbar_arrive(&sm.item_full[slot]);
        }
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item < 0)
            break;
        const XaItem x = xa_decode(a, item);
        const uint32_t bytes = x.nh * kXQBox + kXKBox;
        for (int j = 0; j < kXChunks; ++j) {
            const int st = kit % kXStages;
            if (!mbar_wait(&sm.empty[st], ((kit / kXStages) & 1) ^ 1, &sm.abort, err)) {
                ok = false;
                break;
            }
            ++kit;
            if (lane == 0) {
                const int u = j >> 1, dc = (j & 1) * 64;
                mbar_arrive_expect_tx(&sm.full[st], bytes);
                for (int t = 0; t < x.nh; ++t)
                    tma_load_5d(sm.q[st][t], tm_q, dc, x.h * a.g + x.qi0 + t, u, x.rt * kXRows,
                                x.b, &sm.full[st]);
                tma_load_5d(sm.k[st], tm_k, dc, x.h, kXs - 1 - u, x.ct * kXCols, x.b,
                            &sm.full[st]);
            }
            __syncwarp();
        }
    }
    // Before leaving on an abort, let the copies already issued land.
    if (sm.abort) {
        for (uint32_t k = kit > kXStages ? kit - kXStages : 0; k < kit; ++k) {
            volatile int no_abort = 0;
            mbar_wait(&sm.full[k % kXStages], (k / kXStages) & 1, &no_abort, nullptr);
        }
    }
}

__device__ __forceinline__ void xa_mma(const XaArgs &a, XaSmem &sm, uint32_t tmem, int lane)
{
    uint32_t *err = &a.hdr->error;
    uint32_t kit = 0, sf_cnt0 = 0, sf_cnt1 = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&sm.item_full[slot], (it >> 1) & 1, &sm.abort, err))
            break;
        const int item = sm.item[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.item_empty[slot]);
        if (item < 0)
            break;
        const XaItem x = xa_decode(a, item);
        // S_t is free once its softmax warpgroup has read the previous tile
        if (sf_cnt0 > 0 && !mbar_wait(&sm.s_free[0], (sf_cnt0 - 1) & 1, &sm.abort, err))
            break;
        ++sf_cnt0;
        if (x.nh > 1) {
            if (sf_cnt1 > 0 && !mbar_wait(&sm.s_free[1], (sf_cnt1 - 1) & 1, &sm.abort, err))
                break;
            ++sf_cnt1;
        }
        tc_fence_after();
        for (int j = 0; j < kXChunks; ++j) {
            const int st = kit % kXStages;
            if (!mbar_wait(&sm.full[st], (kit / kXStages) & 1, &sm.abort, err)) {
                ok = false;
                break;
            }
            ++kit;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kaddr = smem_u32(sm.k[st]);
                for (int t = 0; t < x.nh; ++t) {
                    const uint32_t qaddr = smem_u32(sm.q[st][t]);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma(tmem + t * 256, sdesc_sw128(qaddr + k * 32, 16, 1024),
                               sdesc_sw128(kaddr + k * 32, 16, 1024), kIdescXa,
                               (j > 0 || k > 0) ? 1u : 0u);
                    if (j == kXChunks - 1)
                        tc_commit(&sm.s_full[t]);
                }
                tc_commit(&sm.empty[st]);
            }
            __syncwarp();
        }
    }
}

// One warpgroup per head of the pair; thread r owns cell row r of the tile.
__device__ __forceinline__ void xa_softmax(const XaArgs &a, XaSmem &sm, uint32_t tmem, int warp)
{
    uint32_t *err = &a.hdr->error;
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t tS = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + t * 256;
    const float NEG_INF = -__int_as_float(0x7f800000);
    uint32_t s_cnt = 0;
    for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&sm.item_full[slot], (it >> 1) & 1, &sm.abort, err))
            break;
        const int item = sm.item[slot];
        mbar_arrive(&sm.item_empty[slot]);
        if (item < 0)
            break;
        const XaItem x = xa_decode(a, item);
        if (t >= x.nh)
            continue;
        const int row = x.rt * kXRows + r;         // cell row
        const bool valid = row < a.nA;
        const int64_t slot_q = static_cast<int64_t>(x.unit) * a.g + x.qi0 + t;
        if (!mbar_wait(&sm.s_full[t], s_cnt & 1, &sm.abort, err))
            break;
        ++s_cnt;
        tc_fence_after();
        // causal cells: column ct * 256 + c is kept iff it is <= row; only the
        // row tile's last key tile reaches past its rows
        const bool edge = x.ct == x.rt / 2;
        const int hi = row - x.ct * kXCols;
        uint32_t v[32];
        float mx = NEG_INF;
#pragma unroll
        for (int q = 0; q < kXCols / 32; ++q) {
            tmem_ld32(tS + 32 * q, v);
            tmem_wait_ld();
            const uint32_t w = edge ? xa_low_bits(hi + 1 - 32 * q) : 0xffffffffu;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if ((w >> c) & 1u)
                    mx = fmaxf(mx, __uint_as_float(v[c]));
        }
        const float m_t = mx * a.c2;     // the tile's row max, log2 units (finite: column 0 is kept)
        // per 8-cell key block: sum of exp2(score - m_t) over kept cells,
        // stored four blocks at a time as they are made
        float4 *dst = reinterpret_cast<float4 *>(
            a.esum + slot_q * a.tri + (valid ? xa_row_off(row) : 0) + kXBlocksPerTile * x.ct);
        float tile_sum = 0.f;
#pragma unroll
        for (int q = 0; q < kXCols / 32; ++q) {
            tmem_ld32(tS + 32 * q, v);
            tmem_wait_ld();
            const uint32_t w = edge ? xa_low_bits(hi + 1 - 32 * q) : 0xffffffffu;
            float gsum[4];
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                float sum = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int idx = gq * 8 + c;
                    const float p = ex2(fmaf(__uint_as_float(v[idx]), a.c2, -m_t));
                    sum += ((w >> idx) & 1u) ? p : 0.f;
                }
                gsum[gq] = sum;
                tile_sum += sum;
            }
            if (valid && in_bounds(slot_q * a.tri + xa_row_off(row) + kXBlocksPerTile * x.ct + 4 * q + 3,
                                   static_cast<int64_t>(a.max_units) * a.g * a.tri, err))
                dst[q] = make_float4(gsum[0], gsum[1], gsum[2], gsum[3]);
        }
        tc_fence_before();
        mbar_arrive(&sm.s_free[t]);
        if (valid) {
            const int64_t k = (slot_q * a.nA + row) * a.nct + x.ct;
            if (in_bounds(k, static_cast<int64_t>(a.max_units) * a.g * a.nA * a.nct, err)) {
                a.rmax[k] = m_t;
                a.tsum[k] = tile_sum;
            }
        }
    }
}

__global__ void __launch_bounds__(kXThreads, 1)
    xa_scores_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const XaArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    XaSmem &sm = *reinterpret_cast<XaSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.s_free[t], 128);
            mbar_init(&sm.item_full[t], 1);
            mbar_init(&sm.item_empty[t], 1 + 256);
        }
        sm.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kXMmaWarp) {
        tmem_alloc(&sm.tmem_base, kXTmemCols);
        tmem_relinquish();
    }
    if (warp == kXProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kXProducerWarp)
        xa_producer(&tm_q, &tm_k, a, sm, lane);
    else if (warp == kXMmaWarp)
        xa_mma(a, sm, tmem, lane);
    else
        xa_softmax(a, sm, tmem, warp);

    tc_fence_before();
    __syncthreads();
    if (warp == kXMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kXTmemCols);
    }
}

// ------------------------------------------------------------ selection
constexpr int kSelThreads = 256;

// Deterministic block sum (fixed order: per thread, then warps, then lanes).
__device__ __forceinline__ float xa_block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    __syncthreads();
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w)
        s += red[w];
    return s;
}

__global__ void __launch_bounds__(kSelThreads) xa_select_kernel(XaArgs a)
{
    extern __shared__ float dyn[];
    float *w = dyn;                  // [nB]: block scores of this row (kb <= qb used)
    float *lse_s = dyn + a.nB;       // [g * 8]: log2 LSE of (query head, cell row)
    __shared__ float red[kSelThreads / 32];
    __shared__ int tie_lim;
    const int qb = blockIdx.x, unit = blockIdx.y;
    if (unit >= static_cast<int>(a.hdr->reserved[0]))
        return;
    const int u = a.units[unit];
    const int b = u >> 16, h = u & 0xffff;
    const int a0 = qb * kXCellsPerBlock;
    const int a1 = min(a0 + kXCellsPerBlock, a.nA);
    const int n = qb + 1;

    // log2 LSE of every (query head, cell row) of the block from its tiles'
    // (max, total) pairs: eight threads per pair, each over every eighth tile,
    // then a fixed-order reduction across the eight
    const int nrow = a1 - a0;
    const int nct_row = qb / kXBlocksPerTile + 1;     // key tiles of these rows
    for (int p0 = 0; p0 < a.g * nrow; p0 += kSelThreads / 8) {
        const int p = p0 + threadIdx.x / 8, sub = threadIdx.x % 8;
        const bool live = p < a.g * nrow;
        int64_t base = 0;
        if (live) {
            const int qi = p / nrow, row = a0 + p % nrow;
            base = ((static_cast<int64_t>(unit) * a.g + qi) * a.nA + row) * a.nct;
        }
        float mx = -__int_as_float(0x7f800000);
        for (int ct = sub; live && ct < nct_row; ct += 8)
            mx = fmaxf(mx, a.rmax[base + ct]);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int ct = sub; live && ct < nct_row; ct += 8)
            l += a.tsum[base + ct] * ex2(a.rmax[base + ct] - mx);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
            l += __shfl_xor_sync(0xffffffffu, l, o);
        if (live && sub == 0) {
            const int qi = p / nrow, r = p % nrow;
            lse_s[qi * kXCellsPerBlock + r] = mx + __log2f(l);
        }
    }
    __syncthreads();

    // W[qb][kb] = sum over heads and cell rows of the stored block sums times
    // exp2(tile max - row LSE), heads outer, rows inner.  Each thread takes
    // four consecutive key blocks (one 16-byte load per row; rows are 128-byte
    // aligned and padded to whole key tiles, so the loads stay inside them).
    int64_t roff[kXCellsPerBlock];
#pragma unroll
    for (int r = 0; r < kXCellsPerBlock; ++r)
        roff[r] = a0 + r < a1 ? xa_row_off(a0 + r) : 0;
    for (int kb0 = 4 * threadIdx.x; kb0 < n; kb0 += 4 * kSelThreads) {
        const int ct = kb0 / kXBlocksPerTile;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int qi = 0; qi < a.g; ++qi) {
            const int64_t slot_q = static_cast<int64_t>(unit) * a.g + qi;
            const float *e = a.esum + slot_q * a.tri + kb0;
            const float *mxp = a.rmax + (slot_q * a.nA + a0) * a.nct + ct;
            float4 ev[kXCellsPerBlock];
            float mv[kXCellsPerBlock];
#pragma unroll
            for (int r = 0; r < kXCellsPerBlock; ++r) {
                const bool in = a0 + r < a1;
                ev[r] = in && in_bounds(slot_q * a.tri + roff[r] + kb0 + 3,
                                        static_cast<int64_t>(a.max_units) * a.g * a.tri,
                                        &a.hdr->error)
                            ? *reinterpret_cast<const float4 *>(e + roff[r])
                            : make_float4(0.f, 0.f, 0.f, 0.f);
                mv[r] = in ? mxp[static_cast<int64_t>(r) * a.nct] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < kXCellsPerBlock; ++r)
                if (a0 + r < a1) {
                    const float f = ex2(mv[r] - lse_s[qi * kXCellsPerBlock + r]);
                    acc[0] = fmaf(ev[r].x, f, acc[0]);
                    acc[1] = fmaf(ev[r].y, f, acc[1]);
                    acc[2] = fmaf(ev[r].z, f, acc[2]);
                    acc[3] = fmaf(ev[r].w, f, acc[3]);
                }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (kb0 + k < n)
                w[kb0 + k] = acc[k];
    }
    __syncthreads();

    float part = 0.f;
    for (int kb = threadIdx.x; kb < n; kb += kSelThreads)
        part += w[kb];
    const float total = xa_block_sum(part, red);
    const float target = a.threshold * total;

    // mass(v) = sum of the scores >= v: non-increasing in v, also as computed
    // (adding a non-negative term never lowers a rounded sum).  The kept
    // scores are those above v*, the largest v with mass(v) >= target, plus
    // the blocks scoring exactly v*, in key-block order, until the target is
    // reached.
    auto mass_ge = [&](float v) {
        float p = 0.f;
        for (int kb = threadIdx.x; kb < n; kb += kSelThreads)
            p += w[kb] >= v ? w[kb] : 0.f;
        return xa_block_sum(p, red);
    };
    int mode;          // 0: none but the diagonal, 1: threshold, 2: every positive score
    float vstar = 0.f;
    if (!(target > 0.f)) {
        mode = 0;
    } else if (mass_ge(0.f) < target) {
        mode = 2;
    } else {
        mode = 1;
        uint32_t lo = 0u, hi = 0x7f800000u;      // mass(lo) >= target > mass(hi)
        while (hi - lo > 1u) {
            const uint32_t mid = lo + (hi - lo) / 2u;
            if (mass_ge(__uint_as_float(mid)) >= target)
                lo = mid;
            else
                hi = mid;
        }
        vstar = __uint_as_float(lo);
        float pa = 0.f, pt = 0.f;
        for (int kb = threadIdx.x; kb < n; kb += kSelThreads) {
            pa += w[kb] > vstar ? w[kb] : 0.f;
            pt += w[kb] == vstar ? 1.f : 0.f;
        }
        const float above = xa_block_sum(pa, red);
        const float ties = xa_block_sum(pt, red);
        if (threadIdx.x == 0) {
            int lim = n - 1;
            if (ties > 1.f) {
                float run = above;
                lim = -1;
                for (int kb = 0; kb < n && run < target; ++kb)
                    if (w[kb] == vstar) {
                        run += vstar;
                        lim = kb;
                    }
            }
            tie_lim = lim;
        }
        __syncthreads();
    }

    const int64_t row_base = ((static_cast<int64_t>(b) * a.Hkv + h) * a.nB + qb) * a.nB;
    for (int kb = threadIdx.x; kb < a.nB; kb += kSelThreads) {
        uint8_t keep = 0;
        float score = 0.f;
        if (kb <= qb) {
            score = w[kb];
            if (kb == qb)
                keep = 1;
            else if (mode == 1)
                keep = score > vstar || (score == vstar && kb <= tie_lim);
            else if (mode == 2)
                keep = score > 0.f;
        }
        if (!in_bounds(row_base + kb, static_cast<int64_t>(a.B) * a.Hkv * a.nB * a.nB, &a.hdr->error))
            continue;
        a.block_mask[row_base + kb] = keep;
        if (a.block_scores)
            a.block_scores[row_base + kb] = score;
    }
}

} // namespace ea

using namespace ea;

static bool g_xa_attr_done[64];

static ea_status xa_ensure_attributes(size_t sel_smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return EA_ERR_CUDA;
    if (dev < 64 && g_xa_attr_done[dev])
        return EA_OK;
    if (cudaFuncSetAttribute(xa_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kXaSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(xa_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(float) * (EA_MAX_SEQ / EA_TILE + 8 * 64))) !=
            cudaSuccess)
        return EA_ERR_CUDA;
    (void)sel_smem;
    if (dev < 64)
        g_xa_attr_done[dev] = true;
    return EA_OK;
}

static bool xa_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" ea_status ea_xa_estimate(const void *Q, const void *K, const int64_t q_str[4],
                                    const int64_t k_str[4], int B, int S, int Hq, int Hkv, int d,
                                    float scale, const uint8_t *m, int stride, float threshold,
                                    int block_size, int max_units, uint8_t *block_mask,
                                    float *block_scores, void *workspace, size_t ws_bytes,
                                    void *stream)
{
    if (!Q || !K || !q_str || !k_str || !m || !block_mask || !(scale > 0.f) ||
        !(threshold >= 0.f) || !(threshold <= 3.0e38f))
        return EA_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || block_size != EA_TILE ||
        max_units < 1 || static_cast<int64_t>(max_units) > static_cast<int64_t>(B) * Hkv)
        return EA_ERR_INVALID_ARG;
    if (d != EA_HEAD_DIM || stride != EA_XA_STRIDE || S % stride != 0 || S > EA_MAX_SEQ ||
        B > 65535 || Hkv > 65535 || Hq / Hkv > 64)
        return EA_ERR_UNSUPPORTED;
    if (q_str[3] != 1 || k_str[3] != 1)
        return EA_ERR_INVALID_ARG;
    for (int k = 0; k < 3; ++k)
        if (q_str[k] <= 0 || k_str[k] <= 0 || q_str[k] % 8 || k_str[k] % 8)
            return EA_ERR_INVALID_ARG;
    if (!xa_aligned16(Q) || !xa_aligned16(K))
        return EA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return EA_ERR_WORKSPACE;
    const XaWs L = xa_ws_layout(B, S, Hq, Hkv, max_units);
    if (ws_bytes < L.total)
        return EA_ERR_WORKSPACE;

    XaArgs a{};
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.m = m;
    a.hdr = reinterpret_cast<ea_ws_header *>(ws);
    a.units = reinterpret_cast<int32_t *>(ws + L.units);
    a.tsum = reinterpret_cast<float *>(ws + L.tsum);
    a.rmax = reinterpret_cast<float *>(ws + L.rmax);
    a.esum = reinterpret_cast<float *>(ws + L.esum);
    a.block_mask = block_mask;
    a.block_scores = block_scores;
    a.B = B;
    a.Hkv = Hkv;
    a.g = Hq / Hkv;
    a.npairs = static_cast<int>(ceil_div(a.g, 2));
    a.max_units = max_units;
    a.nA = static_cast<int>(L.nA);
    a.nct = static_cast<int>(L.nct);
    a.nB = static_cast<int>(ceil_div(S, EA_TILE));
    a.nRT = static_cast<int>(ceil_div(L.nA, kXRows));
    a.tiles = static_cast<int>(xa_tile_off(a.nRT));
    a.tri = L.tri;
    a.c2 = scale * 1.4426950408889634f / static_cast<float>(stride);
    a.threshold = threshold;

    alignas(64) CUtensorMap tq, tk;
    if (!encode_tmap_bf16_cells(&tq, Q, d, Hq, stride, a.nA, B, q_str, kXRows) ||
        !encode_tmap_bf16_cells(&tk, K, d, Hkv, stride, a.nA, B, k_str, kXCols))
        return EA_ERR_INVALID_ARG;
    ea_status s;
    if ((s = xa_ensure_attributes(0)) != EA_OK)
        return s;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return EA_ERR_CUDA;
    const int sms = num_sms(dev);
    if (sms <= 0)
        return EA_ERR_CUDA;
    const int64_t max_items = static_cast<int64_t>(max_units) * a.npairs * a.tiles;
    if (max_items >= (int64_t{1} << 31))
        return EA_ERR_UNSUPPORTED;
    const unsigned grid = static_cast<unsigned>(max_items < sms ? max_items : sms);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    xa_setup_kernel<<<1, 32, 0, st>>>(a);
    xa_scores_kernel<<<grid, kXThreads, kXaSmemBytes, st>>>(tq, tk, a);
    xa_select_kernel<<<dim3(static_cast<unsigned>(a.nB), static_cast<unsigned>(max_units)),
                       kSelThreads, sizeof(float) * (a.nB + a.g * kXCellsPerBlock), st>>>(a);
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}
