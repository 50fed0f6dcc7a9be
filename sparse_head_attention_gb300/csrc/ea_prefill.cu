// ea_prefill.cu - fused hybrid-head attention prefill for sm_103a.
//
// What it computes ("Paper Reading - Elastic Attention" (English notes), §02
// eqs. (1)-(3); §04 Deployment, Algorithm 1(b)): every query head runs either
// full causal attention (FA) or sparse attention (SA) over its KV head's kept
// keys, in one launch, with each head writing its own slice of the output (the
// eq. 3 concatenation).  The routing decision arrives as per-KV-head metadata
// m (EA_FULL / EA_SSA / EA_BLOCK) that each work item branches on.
//
// How (GB300 design, not the A100/H100 Block-Sparse-Attention kernel the pages
// name as their implementation):
//   1. plan_costs: visited key tiles per (b, KV head, 128-query block).
//   2. plan_sort : one CTA, counting sort of those rows, longest first, into
//                  a work queue of (row, head pair) items.
//   3. hybrid_prefill_kernel: persistent, one cluster of two CTAs (two SMs)
//      per work item at a time, items taken from an atomic queue head.  An item
//      is two query heads of one GQA group over one 128-query block, one head
//      per CTA; every MMA is a 2-SM tcgen05 instruction (M = 256) whose K/V
//      operand is split between the two CTAs, so each SM loads half of every
//      K/V tile.
//        warps 0-7  two softmax warpgroups, each half of the 128 columns of
//                   every S row: online softmax in fp32 (exp2 domain, lazy
//                   rescale of O when the max grows by more than 2^8), P (bf16)
//                   written back into TMEM over S; finally O / l and LSE.
//        warp 8     TMA producer: this CTA's Q tile and K/V halves; rank 0's
//                   also takes items from the queue and publishes each item's
//                   metadata (visited tiles, mode, row fields) to both CTAs
//        warp 9     rank 0: tcgen05 issuer of S = Q K^T (smem x smem)
//        warp 10    rank 0: tcgen05 issuer of O += P V (P from TMEM, V from
//                   smem), with a second product of P's bf16 remainder on
//                   items whose rows keep few keys
//      TMEM (each CTA): O (128 columns) + three S/P buffers (3 x 128), so the
//      next tiles' S = Q K^T products run while the softmax works.
//      Shared memory (each CTA): Q (2 x 32 KB, two items in flight), a 3-slot
//      K ring and a 4-slot V ring of 16 KB halves, and the O tile on its way
//      out (32 KB).
//   Batches are either B sequences of one length S ([B][S][heads][d] tensors)
//   or sequences of different lengths packed back to back (cu_seqlens), and a
//   launch may hold up to 48 layers of one shape; the attention kernel is
//   compiled for each of these, so that the fixed-length single-layer one
//   carries none of the others' row decoding.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "ea_device.cuh"
#include "ea_internal.h"
#ifdef EA_CHECKS
#include "ea_checked.h"
#endif

namespace ea {

constexpr int T = EA_TILE;
constexpr int D = EA_HEAD_DIM;
constexpr int kTileBytes = T * D * 2;        // one 128 x 128 bf16 tile
constexpr int kHalfBytes = kTileBytes / 2;   // one 64-column swizzled TMA box of 128 rows

// Layers of one launch (a multi-layer prefill: every layer has the same shapes
// and strides; its rows are numbered layer by layer).
constexpr int kMaxLayers = EA_MAX_PREFILL_LAYERS;

struct PrefillArgs {
    __nv_bfloat16 *O[kMaxLayers];
    const uint8_t *m[kMaxLayers];
    const uint8_t *block_mask[kMaxLayers];
    float *LSE[kMaxLayers];
    int n_layers;
    uint32_t rows_per_layer;     // rows of one layer (B * Hkv * nB for fixed-length batches)
    int sort_group;              // planner: 0 longest first; 1 layer by layer, 2 sequence by sequence
    int n_sort_groups;           // groups of that order (1 for sort_group 0)
    int64_t o_sb, o_ss, o_sh;
    int64_t lse_sb, lse_sh;      // LSE[b * lse_sb + qh * lse_sh + token]
    int64_t lse_elems;           // LSE elements (bounds-checked builds)
    int64_t mask_elems;          // block-mask bytes, -1: mask_off[B] (bounds-checked builds)
    int64_t visited_bits;        // bits of the visited bitmap (bounds-checked builds)
    int o_v8;                    // every O row starts 32-byte aligned: 256-bit stores
    uint32_t *visited;
    int32_t *costs;
    uint32_t *items;
    ea_ws_header *hdr;
    int B, S, Hq, Hkv, g, npairs, nB, sink, window;
    int qb_begin, qb_end;        // query blocks this plan covers
    uint32_t n_rows, n_items;    // rows to scan, items at most (the plan counts the real ones)
    float scale_log2;
    // variable-length batch (cu_seqlens != NULL): sequence b is tokens
    // [cu_seqlens[b], cu_seqlens[b + 1]) of one packed [tokens][heads][d]
    // tensor; its rows start at row_off[b] and its block mask at mask_off[b]
    const int32_t *cu_seqlens;
    int32_t *row_off;
    int64_t *mask_off;
    int2 *row_desc;              // per planned row: {b, h << 16 | qb}, written by the planner
    int max_seqlen, total_tokens;
    uint64_t wait_timeout_ns;    // bounded device waits give up after this long
    int64_t test_skip_load;      // bounds-checked builds' tests: a K/V load left out (-1: none)
};

// One (b, KV head, query block) row of the plan.  tok0 is the sequence's first
// token in the tensors' token dimension, tma_b its batch coordinate, mask_row
// the offset of the row's block-mask entries.
struct RowInfo {
    int layer, b, h, qb, tok0, S, nB, tma_b;
    int64_t mask_row;
};

// Block-mask bytes the kernels may read (bounds-checked builds).
__device__ __forceinline__ int64_t mask_limit(const PrefillArgs &a)
{
    return a.mask_elems >= 0 ? a.mask_elems : a.mask_off[a.B];
}

// Fields of a variable-length row once b, h and qb are known.
__device__ __forceinline__ void varlen_row_fields(const PrefillArgs &a, RowInfo &x)
{
    x.layer = 0;
    x.tok0 = a.cu_seqlens[x.b];
    x.S = a.cu_seqlens[x.b + 1] - x.tok0;
    x.nB = (x.S + T - 1) / T;
    x.tma_b = 0;
    x.mask_row = a.mask_off[x.b] + (static_cast<int64_t>(x.h) * x.nB + x.qb) * x.nB;
}

// A row of a fixed-length batch: rows are [layer][b][h][qb] (the layer part
// only when the launch may hold several).
template <bool kMulti = true>
__device__ __forceinline__ void decode_row_dense(int row, const PrefillArgs &a, RowInfo &x)
{
    x.layer = 0;
    if (kMulti && a.n_layers > 1) {
        x.layer = static_cast<int>(static_cast<uint32_t>(row) / a.rows_per_layer);
        row -= x.layer * static_cast<int>(a.rows_per_layer);
    }
    x.qb = row % a.nB;
    const int bh = row / a.nB;
    x.h = bh % a.Hkv;
    x.b = bh / a.Hkv;
    x.tok0 = 0;
    x.S = a.S;
    x.nB = a.nB;
    x.tma_b = x.b;
    x.mask_row = (static_cast<int64_t>(bh) * a.nB + x.qb) * a.nB;
}

// Planner side: find the row's sequence (variable-length batches search the
// per-sequence row offsets) and record it for the attention kernel.
__device__ __forceinline__ bool decode_row_search(int row, const PrefillArgs &a, RowInfo &x)
{
    if (!a.cu_seqlens) {
        decode_row_dense(row, a, x);
        return true;
    }
    if (row >= a.row_off[a.B])
        return false;
    // the last sequence whose first row is <= row (it is never empty)
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.row_off[mid] <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    x.b = lo;
    const int S = a.cu_seqlens[lo + 1] - a.cu_seqlens[lo];
    const int nB = (S + T - 1) / T;
    const int local = row - a.row_off[lo];
    x.h = local / nB;
    x.qb = local - x.h * nB;
    varlen_row_fields(a, x);
    return true;
}

// Kernel side: a planned row (variable-length rows through the planner's
// record, which keeps the search out of the warps' register budgets).  The
// attention kernel is compiled separately for fixed- and variable-length
// batches, so that the fixed-length one carries none of this.
template <bool kVarlen, int kL>
__device__ __forceinline__ void decode_row(int row, const PrefillArgs &a, RowInfo &x)
{
    if (!kVarlen) {
        decode_row_dense<(kL > 1)>(row, a, x);
        return;
    }
    const int2 d = in_bounds(row, a.n_rows, &a.hdr->error) ? a.row_desc[row] : make_int2(0, 0);
    x.b = d.x;
    x.h = static_cast<int>(static_cast<uint32_t>(d.y) >> 16);
    x.qb = d.y & 0xFFFF;
    varlen_row_fields(a, x);
}

// ------------------------------------------------------------ tile sequences
// SSA key tiles of query block qb: the sink tiles [0, n_sink) below the window,
// then the window tiles [kb_lo, qb].  A tile is visited iff it holds at least
// one kept (query, key) pair: a sink key (kb*T < sink), a key within the window
// of the block's first query ((qb-kb-1)*T + 1 < window), or the diagonal.
__device__ __forceinline__ void ssa_tiles(int qb, int sink, int window, int &n_sink, int &kb_lo)
{
    const int w_tiles = (window - 1 + T - 1) / T;    // ceil((window-1)/T)
    kb_lo = qb - w_tiles > 0 ? qb - w_tiles : 0;
    const int s_tiles = (sink + T - 1) / T;          // ceil(sink/T)
    n_sink = s_tiles < kb_lo ? s_tiles : kb_lo;
}

// Key tile of the n-th visited tile for FULL / SSA heads.
__device__ __forceinline__ int seq_kb(int mode, int n, int n_sink, int kb_lo)
{
    if (mode == EA_FULL)
        return n;
    return n < n_sink ? n : kb_lo + (n - n_sink);
}

// Word with the low n bits set (n clamped to 0..32).
__device__ __forceinline__ uint32_t low_bits(int n)
{
    return n <= 0 ? 0u : n >= 32 ? 0xffffffffu : (1u << n) - 1u;
}

// Does every (query, key) pair of tile (qb, kb) pass the head's mask?  Only
// tiles that fail this need per-element masking.
__device__ __forceinline__ bool tile_is_full(int mode, int qb, int kb, int sink, int window)
{
    if (kb >= qb)
        return false;
    if (mode == EA_SSA)
        return (kb + 1) * T <= sink || (qb - kb) * T + T - 1 < window;
    return true;
}

// Keys kept by the first (fewest-keys) query row of block qb, for a row with
// N visited tiles: FULL keeps i + 1, SSA the sink keys up to i plus the keys of
// the window not already counted, BLOCK whole kept tiles plus i + 1 - kb*T of
// the diagonal.  Every later row of the block keeps at least as many.
__device__ __forceinline__ int first_row_keys(int mode, int qb, int sink, int window, int N,
                                              bool diag_kept)
{
    const int i = qb * T;
    if (mode == EA_FULL)
        return i + 1;
    if (mode == EA_SSA) {
        const int n_sk = i + 1 < sink ? i + 1 : sink;
        const int w_lo = i - window + 1 > sink ? i - window + 1 : sink;
        return n_sk + (i + 1 - w_lo > 0 ? i + 1 - w_lo : 0);
    }
    return diag_kept ? (N - 1) * T + 1 : N * T;
}

// Rows that keep at most this many keys take the P V product in two bf16 parts
// (P's rounding and the remainder), see pair_softmax.  A row whose weight sits
// on a few keys carries each probability's 2^-9 rounding error almost whole
// into O; with V of a large common offset (|v| in [2.2, 3.8), one sign per
// dimension) query blocks whose first row keeps 129-512 keys still put elements
// up to 1.4e-3 above a flat 1e-2 when only rows of at most 128 keys were split
// (24 of 150 random configurations).  At 512 keys none did; the 32K layer's cost is nil (its
// rows keep more keys past the first query blocks), a batch of 128 sequences
// of 256-8192 tokens pays about 1 %.
constexpr int kSplitMaxKeys = 4 * T;

// ------------------------------------------------------------ planner
// One warp per (b, KV head, q block) row: number of visited key tiles, or -1
// for a row outside the planned query blocks.
__global__ void plan_costs_kernel(PrefillArgs a)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
    if (warp >= static_cast<int>(a.n_rows))
        return;
    RowInfo x;
    if (!decode_row_search(warp, a, x) || x.qb < a.qb_begin || x.qb >= a.qb_end) {
        if (lane == 0)
            a.costs[warp] = -1;
        return;
    }
    if (a.cu_seqlens && lane == 0)
        a.row_desc[warp] = make_int2(x.b, (x.h << 16) | x.qb);
    const int qb = x.qb;
    const int mode = a.m[x.layer][x.b * a.Hkv + x.h];
    const uint8_t *bmask = a.block_mask[x.layer];
    int n = 0;
    if (mode == EA_FULL) {
        n = qb + 1;
    } else if (mode == EA_SSA) {
        int n_sink, kb_lo;
        ssa_tiles(qb, a.sink, a.window, n_sink, kb_lo);
        n = n_sink + (qb - kb_lo + 1);
    } else if (mode == EA_BLOCK && bmask) {
        const uint8_t *row = bmask + x.mask_row;
        for (int kb = lane; kb <= qb; kb += 32)
            if (in_bounds(x.mask_row + kb, mask_limit(a), &a.hdr->error))
                n += row[kb] != 0;
        for (int o = 16; o > 0; o >>= 1)
            n += __shfl_xor_sync(0xffffffffu, n, o);
    } else {
        if (lane == 0)
            raise_error(&a.hdr->error, EA_DEVERR_CHECK);  // bad mode, or BLOCK without a mask
        n = 0;
    }
    if (lane == 0)
        a.costs[warp] = n;
}

// Sort key of a planned row: longest first, and for a multi-layer launch or a
// variable-length batch in layer or sequence order first (key
// group * (nB + 1) + nB - cost), so that one group's K/V tiles stay in L2 while
// its items run and the next group's longest items follow without a drain.
// Keys of rows outside the plan: -1.
__device__ __forceinline__ int plan_key(uint32_t r, int cost, const PrefillArgs &a)
{
    if (cost < 0)
        return -1;
    int group = 0;
    if (a.sort_group == 1)
        group = static_cast<int>(r / a.rows_per_layer);
    else if (a.sort_group == 2)
        group = a.row_desc[r].x;
    return group * (a.nB + 1) + (a.nB - cost);
}

// One CTA: counting sort of the planned rows (cost >= 0) by key, ascending;
// each row contributes its npairs items back to back.  The order among rows of
// equal key is unspecified (every item is computed the same way whatever the
// order, so results do not depend on it).  Also resets the work queue head.
__global__ void __launch_bounds__(1024) plan_sort_kernel(PrefillArgs a)
{
    extern __shared__ int hist[];  // [nbins + 1]
    __shared__ int scan_tmp[1024];
    const int nbins = a.n_sort_groups * (a.nB + 1);
    const int tid = threadIdx.x;
    for (int c = tid; c < nbins; c += blockDim.x)
        hist[c] = 0;
    __syncthreads();
    __shared__ int n_planned;
    if (tid == 0)
        n_planned = 0;
    __syncthreads();
    int mine = 0;
    for (uint32_t r = tid; r < a.n_rows; r += blockDim.x) {
        const int k = plan_key(r, a.costs[r], a);
        if (k >= 0) {
            atomicAdd(&hist[k], 1);
            ++mine;
        }
    }
    atomicAdd(&n_planned, mine);
    __syncthreads();
    // Exclusive scan over the keys: start[k] = #rows with a smaller key; each
    // thread scans a segment of bins.
    const int per = (nbins + blockDim.x - 1) / blockDim.x;
    const int lo = tid * per, hi = min(lo + per, nbins);
    int local = 0;
    for (int p = lo; p < hi; ++p)
        local += hist[p];
    scan_tmp[tid] = local;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        int v = tid >= off ? scan_tmp[tid - off] : 0;
        __syncthreads();
        scan_tmp[tid] += v;
        __syncthreads();
    }
    int run = scan_tmp[tid] - local;
    for (int p = lo; p < hi; ++p) {
        const int cnt = hist[p];
        hist[p] = run;
        run += cnt;
    }
    __syncthreads();
    // Scatter by every warp, 32 rows at a time: the lanes of a warp with the
    // same key take consecutive slots, their first lane claims them for the
    // group with one shared-memory atomic.
    {
        const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
        const unsigned lt = (1u << lane) - 1u;
        for (uint32_t base = warp * 32u; base < a.n_rows; base += 32u * nwarps) {
            const uint32_t r = base + lane;
            const int k = r < a.n_rows ? plan_key(r, a.costs[r], a) : -1;
            const bool valid = k >= 0;
            const unsigned active = __ballot_sync(0xffffffffu, valid);
            const unsigned peers = __match_any_sync(0xffffffffu, k) & active;
            const int leader = peers ? __ffs(peers) - 1 : 0;
            int start = 0;
            if (valid && lane == leader)
                start = atomicAdd(&hist[k], __popc(peers));
            start = __shfl_sync(0xffffffffu, start, leader);
            if (valid) {
                const int pos = start + __popc(peers & lt);
                for (int p = 0; p < a.npairs; ++p)
                    if (in_bounds(static_cast<int64_t>(pos) * a.npairs + p, a.n_items, &a.hdr->error))
                        a.items[static_cast<uint64_t>(pos) * a.npairs + p] = r * a.npairs + p;
            }
        }
    }
    if (tid == 0) {
        a.hdr->work_counter = 0;
        a.hdr->drained = 0;
        a.hdr->n_items = static_cast<uint32_t>(n_planned) * static_cast<uint32_t>(a.npairs);
    }
}

// One CTA: per-sequence row and block-mask offsets of a variable-length batch.
// A sequence with a bad length (negative, beyond max_seqlen, or ending past
// total_tokens) is reported and planned with no rows.
__global__ void __launch_bounds__(1024) varlen_setup_kernel(PrefillArgs a)
{
    __shared__ long long scan_r[1024], scan_m[1024];
    const int tid = threadIdx.x;
    const int per = (a.B + blockDim.x - 1) / blockDim.x;
    const int lo = tid * per, hi = min(lo + per, a.B);
    long long rows = 0, bytes = 0;
    for (int b = lo; b < hi; ++b) {
        const int c0 = a.cu_seqlens[b], c1 = a.cu_seqlens[b + 1];
        int S = c1 - c0;
        if (c0 < 0 || S < 0 || S > a.max_seqlen || c1 > a.total_tokens) {
            raise_error(&a.hdr->error, EA_DEVERR_CHECK);
            S = 0;
        }
        const long long nB = (S + T - 1) / T;
        rows += a.Hkv * nB;
        bytes += a.Hkv * nB * nB;
    }
    scan_r[tid] = rows;
    scan_m[tid] = bytes;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const long long vr = tid >= off ? scan_r[tid - off] : 0;
        const long long vm = tid >= off ? scan_m[tid - off] : 0;
        __syncthreads();
        scan_r[tid] += vr;
        scan_m[tid] += vm;
        __syncthreads();
    }
    long long run_r = scan_r[tid] - rows, run_m = scan_m[tid] - bytes;
    for (int b = lo; b < hi; ++b) {
        a.row_off[b] = static_cast<int32_t>(run_r);
        a.mask_off[b] = run_m;
        const int c0 = a.cu_seqlens[b], c1 = a.cu_seqlens[b + 1];
        int S = c1 - c0;
        if (c0 < 0 || S < 0 || S > a.max_seqlen || c1 > a.total_tokens)
            S = 0;
        const long long nB = (S + T - 1) / T;
        run_r += a.Hkv * nB;
        run_m += a.Hkv * nB * nB;
    }
    if (tid == 1023) {
        a.row_off[a.B] = static_cast<int32_t>(scan_r[1023]);
        a.mask_off[a.B] = scan_m[1023];
    }
}

// ------------------------------------------------------------ attention
//
// CTA pairs.  A cluster of two CTAs on two SMs computes one work item, rank r
// holding query head 2 * pair + r of the item's GQA group, and every MMA is
// one 2-SM tcgen05 instruction (cta_group::2, M = 256 = each CTA's 128 query
// rows) issued by rank 0:
//   S = Q K^T : A = Q (each CTA its own head), B = the key tile split by keys
//               (rank r holds keys 64r .. 64r + 63 of the tile);
//   O += P V  : A = P read from each CTA's tensor memory, B = the value tile
//               split by head dim (rank r holds dims 64r .. 64r + 63).
// Each SM therefore loads half of every K/V tile, and its 512 TMEM columns
// hold O (128) and three S/P buffers (3 x 128): S of tile j + 2 is computed
// while the softmax works on tile j.  A buffer is written again only after the
// P V product that read its P has completed (an mbarrier wait): no ordering
// between MMAs into different accumulators is assumed.
//
// Roles (352 threads per CTA):
//   warps 0-7  softmax.  Warpgroup w handles columns 64w .. 64w + 63 of every
//              S row (one query row per thread); the two threads of a row
//              exchange their partial row maxima through shared memory and a
//              named barrier of their two warps.  P (bf16 pairs) is written
//              over the warpgroup's own S columns.  Epilogue: O / l of the
//              warpgroup's 64 head dims, stored by TMA (in a variable-length
//              batch the warp whose rows cross the sequence's end stores them
//              directly), and LSE.
//   warp 8     TMA producer (both CTAs): this CTA's Q and its halves of the
//              K/V tiles, tile by tile, into a 3-slot K ring and a 4-slot V
//              ring; completion is reported to rank 0's barriers.  Rank 0's
//              producer also takes items from the work queue and publishes
//              each item's metadata to both CTAs.
//   warps 9, 10  rank 0, one thread each: the S = Q K^T issuer and the
//              O += P V issuer; warp 9 of both ranks: the pair's TMEM allocation.
// A tcgen05.mma holds its issuing thread for about its own execution time, so
// whatever an issuer does between MMAs (barrier waits, commits) leaves the
// tensor pipe idle unless another thread is issuing meanwhile: hence two
// issuers, each waiting on two barriers and committing once per tile.
constexpr int kKSlots = 3;                    // K ring: slot of tile j is j % 3 (as its S/P buffer)
constexpr int kVSlots = 4;                    // V ring: slot of tile j is j % 4
constexpr int kHalf = 64 * D * 2;             // 16 KB: half a K tile or half a V tile
constexpr int kPThreads = 352;
constexpr int kPProducerWarp = 8;
constexpr int kPMmaWarp = 9;                  // QK issuer (and TMEM allocation)
constexpr int kPPvWarp = 10;                  // PV issuer
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                 // O: columns 0..127
constexpr uint32_t kColS = 128;               // S/P buffer b: columns 128 + 128 b
constexpr uint32_t kIdescQK2 = idesc_bf16_f32(256, 128, false, false);  // Q, K both K-major
constexpr uint32_t kIdescPV2 = idesc_bf16_f32(256, 128, false, true);   // V is MN-major
constexpr uint16_t kBothCtas = 3;             // multicast mask: both CTAs of the pair
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale when max grows > 2^8

// A queued item as rank 0's producer publishes it to both CTAs: the queue
// entry and, read once from global memory there, what the consumers need of it.
struct ItemMeta {
    int item;        // queue entry (row * npairs + pair), or -1: the queue is drained
    int info;        // visited tiles N | mode << 20 | diagonal kept << 22 | two-part P V << 23
    int b, hq;       // batch row or sequence; KV head << 16 | query block
    int tok0, len;   // the sequence's first token and length
    int lp;          // layer << 16 | head pair
    int row;         // planned row (item / npairs)
};
__device__ __forceinline__ int meta_n(int info) { return info & 0xFFFFF; }
__device__ __forceinline__ int meta_mode(int info) { return (info >> 20) & 3; }
__device__ __forceinline__ bool meta_diag(int info) { return (info >> 22) & 1; }
__device__ __forceinline__ bool meta_split(int info) { return (info >> 23) & 1; }

struct __align__(1024) PairSmem {
    uint8_t q[2][kTileBytes];      // this CTA's query tile, two items in flight
    uint8_t k[kKSlots][kHalf];     // this CTA's halves of the key tiles (64 keys)
    uint8_t v[kVSlots][kHalf];     // this CTA's halves of the value tiles (64 dims)
    uint8_t ostage[kTileBytes];    // O on its way out: 8 warps x (32 rows x 64 columns)
    uint64_t kv_full[kVSlots];     // tile j's K and V halves of both CTAs landed
    uint64_t v_empty[kVSlots];     // P V of tile j done: V slot free, O updated
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[3], p_ready[3];   // S ready (and the K slot free); P written
    uint64_t o_done;
    uint64_t item_full[2], item_empty[2];
    uint64_t teardown;
    uint64_t pv_issued;            // the PV issuer has issued an item's last product
    float red_max[2][2][T];        // [tile parity][warpgroup][row]
    float red_l[2][2][T];          // [item parity][warpgroup][row]
    float red_dl[2][2][T];         // the same for the normaliser's correction (see pair_softmax)
    ItemMeta meta[2];
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kPairSmemBytes = sizeof(PairSmem) + 1024;  // + alignment slack
static_assert(kPairSmemBytes <= 227 * 1024, "prefill shared memory exceeds 227 KB");

struct ItemInfo : RowInfo {
    int pair, row;
};

template <bool kVarlen, int kL>
__device__ __forceinline__ ItemInfo decode_item(int item, const PrefillArgs &a)
{
    ItemInfo x;
    x.pair = item % a.npairs;
    x.row = item / a.npairs;
    decode_row<kVarlen, kL>(x.row, a, x);
    if (kL == 1)
        x.layer = 0;
    return x;
}

// The item's metadata, read from global memory (rank 0's producer, once per item).
template <bool kVarlen, int kL>
__device__ __forceinline__ ItemMeta make_meta(int item, const PrefillArgs &a, uint32_t *err)
{
    ItemMeta mt = {};
    mt.item = item;
    if (item < 0)
        return mt;
    const ItemInfo x = decode_item<kVarlen, kL>(item, a);
    const int cost = in_bounds(x.row, a.n_rows, err) ? a.costs[x.row] : 0;
    const int N = cost > 0 ? cost : 0;
    const int mode = a.m[x.layer][x.b * a.Hkv + x.h];
    bool diag_kept = false;
    if (mode == EA_BLOCK && N > 0)
        diag_kept = in_bounds(x.mask_row + x.qb, mask_limit(a), err) &&
                    a.block_mask[x.layer][x.mask_row + x.qb] != 0;
    // Rows that keep few keys (the first query blocks, small sink and window, a
    // lone diagonal block) take P V in two bf16 parts: with a handful of keys
    // one probability's 2^-9 rounding error reaches O undiluted, and would add
    // up to 2^-9 |O| to the output's own rounding.
    const bool split = N > 0 && first_row_keys(mode, x.qb, a.sink, a.window, N, diag_kept) <= kSplitMaxKeys;
    mt.info = N | ((mode & 3) << 20) | (diag_kept ? 1 << 22 : 0) | (split ? 1 << 23 : 0);
    mt.b = x.b;
    mt.hq = (x.h << 16) | x.qb;
    mt.tok0 = x.tok0;
    mt.len = x.S;
    mt.lp = (x.layer << 16) | x.pair;
    mt.row = x.row;
    return mt;
}

// An item's row from its metadata (no global memory, no division).  mask_row
// is left for the producer to fill in where it needs it.
template <bool kVarlen, int kL>
__device__ __forceinline__ ItemInfo meta_item(const ItemMeta &mt, const PrefillArgs &a)
{
    ItemInfo x;
    x.pair = mt.lp & 0xFFFF;
    x.row = mt.row;
    x.layer = kL == 1 ? 0 : static_cast<int>(static_cast<uint32_t>(mt.lp) >> 16);
    x.b = mt.b;
    x.h = static_cast<int>(static_cast<uint32_t>(mt.hq) >> 16);
    x.qb = mt.hq & 0xFFFF;
    x.tok0 = mt.tok0;
    x.S = mt.len;
    x.nB = kVarlen ? (x.S + T - 1) / T : a.nB;
    x.tma_b = kVarlen ? 0 : x.b;
    x.mask_row = 0;
    return x;
}

// Query head of rank t of an item; an odd group size pairs its last head with
// itself (second copy computed but not stored).
__device__ __forceinline__ int item_head(const ItemInfo &x, int t, const PrefillArgs &a, bool &store)
{
    const int j = 2 * x.pair + t;
    store = j < a.g;
    return x.h * a.g + (store ? j : 2 * x.pair);
}

// Warp-uniform generator of the kept key tiles of a BLOCK row, in ascending
// order: each lane tests 16 mask bytes of a 512-byte window per refill.
struct BlockScan {
    const uint8_t *row;
    int64_t avail;  // mask bytes from row on (bounds-checked builds)
    uint32_t *err;
    int limit;      // qb + 1
    int base;       // first key tile of the current window
    int cur_lane;
    uint32_t bits;  // remaining kept tiles of cur_lane
    uint32_t mine;  // this lane's 16-bit mask of the current window

    __device__ void refill(int lane)
    {
        mine = 0;
        const int k0 = base + lane * 16;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (k0 + j < limit && in_bounds(k0 + j, avail, err) && row[k0 + j] != 0)
                mine |= 1u << j;
        cur_lane = 0;
        bits = __shfl_sync(0xffffffffu, mine, 0);
    }
    __device__ void init(const uint8_t *r, int64_t av, uint32_t *e, int lim, int lane)
    {
        row = r;
        avail = av;
        err = e;
        limit = lim;
        base = 0;
        refill(lane);
    }
    // Next kept key tile, or -1.
    __device__ int next(int lane)
    {
        while (true) {
            if (bits) {
                const int kb = base + cur_lane * 16 + (__ffs(bits) - 1);
                bits &= bits - 1;
                return kb;
            }
            if (++cur_lane < 32) {
                bits = __shfl_sync(0xffffffffu, mine, cur_lane);
                continue;
            }
            base += 512;
            if (base >= limit)
                return -1;
            refill(lane);
        }
    }
};

// What every role of a CTA of the pair needs to wait and to abort.
struct PairCtx {
    uint32_t rank;           // 0: issues the MMAs and takes items from the queue
    uint32_t peer_abort;     // shared::cluster address of the other CTA's abort flag
    volatile int *abort;     // this CTA's abort flag
    uint32_t *err;           // workspace error word
    uint64_t timeout_ns;
};

// shared::cluster address of a barrier of rank 0 (this CTA's own on rank 0).
__device__ __forceinline__ uint32_t lead_bar(const uint64_t *bar)
{
    return mapa_shared(smem_u32(bar), 0);
}

// Bounded wait of the pair kernel, called by every lane of a warp; the result
// is the same in all lanes.  It fails at once when the CTA is aborting (the
// flag is read with the barrier's first test, so that no role passes another
// wait after an abort, and neither read waits for the other) and after the
// timeout (raising EA_DEVERR_TIMEOUT and aborting both CTAs).
// Acquire at CTA scope, or at cluster scope (`cl`) for the item hand-off from
// the other CTA.
__device__ __forceinline__ bool pwait(uint64_t *bar, uint32_t parity, const PairCtx &c,
                                      bool cl = false)
{
    const int aborting = *c.abort;
    const uint32_t a = smem_u32(bar);
    bool ok = cl ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity);
    ok = ok && !aborting;
    if (!aborting) {
        if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            while (true) {
                bool done = false;
                for (int i = 0; i < 32 && !done; ++i)
                    done = cl ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity);
                if (done) {
                    ok = true;
                    break;
                }
                if (*c.abort)
                    break;
                if (globaltimer_ns() - t0 > c.timeout_ns) {
                    raise_error(c.err, EA_DEVERR_TIMEOUT);
                    *c.abort = 1;
                    red_or_cluster(c.peer_abort, 1u);
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// The same for one thread (the MMA issuer).
__device__ __forceinline__ bool pwait1(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    const int aborting = *c.abort;
    const uint32_t a = smem_u32(bar);
    const bool done = mbar_try_wait(a, parity);
    if (aborting)
        return false;
    if (done)
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity))
                return true;
        if (*c.abort)
            return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) {
            raise_error(c.err, EA_DEVERR_TIMEOUT);
            *c.abort = 1;
            red_or_cluster(c.peer_abort, 1u);
            return false;
        }
    }
}

// The TMA tensor maps of the launch's layers (one entry for single-layer
// launches).
template <int kL>
struct TmapTable {
    CUtensorMap q[kL], k[kL], v[kL], o[kL];
};

template <bool kVarlen, int kL>
__device__ __forceinline__ void pair_producer(const TmapTable<kL> &tm, const PrefillArgs &a,
                                              PairSmem &sm, const PairCtx &c, int lane)
{
    uint32_t *err = c.err;
    const bool lead = c.rank == 0;
    const uint32_t n_items = a.hdr->n_items;   // written by the planner
    const uint32_t n_clusters = gridDim.x / 2;
    uint32_t jt = 0, q_it = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        const uint32_t par = (it >> 1) & 1;
        if (lead) {
            if (!pwait(&sm.item_empty[slot], par ^ 1, c))
                break;
            if (lane == 0) {
                const uint32_t x = atomicAdd(&a.hdr->work_counter, 1u);
                const int item = x < n_items ? static_cast<int>(a.items[x]) : -1;
                // Every pair sees the empty queue exactly once; the last one
                // resets the head so the same plan can feed another launch.
                if (item < 0 && atomicAdd(&a.hdr->drained, 1u) == n_clusters - 1) {
                    a.hdr->work_counter = 0;
                    a.hdr->drained = 0;
                }
                // the item and its metadata into both CTAs' slots
                const ItemMeta mt = make_meta<kVarlen, kL>(item, a, err);
                sm.meta[slot] = mt;
                const int *w = reinterpret_cast<const int *>(&mt);
                const uint32_t peer = mapa_shared(smem_u32(&sm.meta[slot]), 1);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_cluster_u32(peer + 4 * k, static_cast<uint32_t>(w[k]));
                mbar_arrive(&sm.item_full[slot]);
                mbar_arrive_cluster(mapa_shared(smem_u32(&sm.item_full[slot]), 1));
            }
            __syncwarp();
        } else {
            if (!pwait(&sm.item_full[slot], par, c, true))
                break;
        }
        const ItemMeta mt = sm.meta[slot];
        if (!lead) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote(lead_bar(&sm.item_empty[slot]));
        }
        if (mt.item < 0)
            break;
        const int N = meta_n(mt.info);
        if (N == 0)
            continue;
        const int mode = meta_mode(mt.info);
        ItemInfo x = meta_item<kVarlen, kL>(mt, a);
        if (mode == EA_BLOCK)
            x.mask_row = (kVarlen ? a.mask_off[x.b] : static_cast<int64_t>(x.b) * a.Hkv * a.nB * a.nB) +
                         (static_cast<int64_t>(x.h) * x.nB + x.qb) * x.nB;
        const CUtensorMap *tm_q = &tm.q[kL == 1 ? 0 : x.layer];
        const CUtensorMap *tm_k = &tm.k[kL == 1 ? 0 : x.layer];
        const CUtensorMap *tm_v = &tm.v[kL == 1 ? 0 : x.layer];
        // this CTA's query tile
        const int qbuf = q_it & 1;
        if (!pwait(&sm.q_empty[qbuf], ((q_it >> 1) & 1) ^ 1, c))
            break;
        ++q_it;
        if (lane == 0) {
            const uint32_t qbar = lead_bar(&sm.q_full[qbuf]);
            if (lead)
                mbar_arrive_expect_tx(&sm.q_full[qbuf], 2 * kTileBytes);
            bool st;
            const int qh = item_head(x, static_cast<int>(c.rank), a, st);
            const int row0 = x.tok0 + x.qb * T;
            tma_load_4d_pair(sm.q[qbuf], tm_q, 0, qh, row0, x.tma_b, qbar);
            tma_load_4d_pair(sm.q[qbuf] + kHalfBytes, tm_q, 64, qh, row0, x.tma_b, qbar);
        }
        __syncwarp();
        // K and V halves of every tile, in tile order; tile jt (counted over
        // this CTA's items) goes to K slot jt % 3, freed by QK(jt - 3) (its
        // s_full commit), and V slot jt % 4, freed by PV(jt - 4)
        int n_sink = 0, kb_lo = 0;
        if (mode == EA_SSA)
            ssa_tiles(x.qb, a.sink, a.window, n_sink, kb_lo);
        BlockScan scan;
        if (mode == EA_BLOCK)
            scan.init(a.block_mask[x.layer] + x.mask_row, mask_limit(a) - x.mask_row, err, x.qb + 1, lane);
        for (int n = 0; n < N && ok; ++n, ++jt) {
            const int kb = mode == EA_BLOCK ? scan.next(lane) : seq_kb(mode, n, n_sink, kb_lo);
            const uint32_t ks = jt % kKSlots, vs = jt % kVSlots;
            if (jt >= kKSlots && !pwait(&sm.s_full[ks], ((jt / kKSlots) & 1) ^ 1, c)) {
                ok = false;
                break;
            }
            if (jt >= kVSlots && !pwait(&sm.v_empty[vs], ((jt / kVSlots) & 1) ^ 1, c)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t fbar = lead_bar(&sm.kv_full[vs]);
                if (lead)
                    mbar_arrive_expect_tx(&sm.kv_full[vs], 4 * kHalf);
                bool issue = true;
#ifdef EA_CHECKS
                // fault injection of the bounds-checked build's tests: one
                // tile's loads left out, so that a consumer's bounded wait runs out
                issue = !(lead && static_cast<int64_t>(jt) == a.test_skip_load);
#endif
                const int key0 = x.tok0 + kb * T;
                const int r64 = 64 * static_cast<int>(c.rank);
                if (issue) {
                    tma_load_4d_pair(sm.k[ks], tm_k, 0, x.h, key0 + r64, x.tma_b, fbar);
                    tma_load_4d_pair(sm.k[ks] + kHalf / 2, tm_k, 64, x.h, key0 + r64, x.tma_b, fbar);
                    tma_load_4d_pair(sm.v[vs], tm_v, r64, x.h, key0, x.tma_b, fbar);
                }
                if (lead && a.visited) {
                    const uint64_t bit = static_cast<uint64_t>(x.row) * a.nB + static_cast<uint64_t>(kb);
                    if (in_bounds(static_cast<int64_t>(bit), a.visited_bits, err))
                        atomicOr(&a.visited[bit >> 5], 1u << (bit & 31));
                }
            }
            __syncwarp();
        }
    }
    // Before leaving on an abort, let the copies already issued land (they
    // target this CTA's shared memory and rank 0's barriers); none takes
    // anywhere near this long.
    if (*c.abort) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
}

// Rank 0's MMA issuers: two threads in two warps, one for the S = Q K^T
// products and one for the O += P V products, so that each one's barrier waits
// and commits overlap the other's MMAs (a tcgen05.mma holds its issuing
// thread for about its execution time).  Every ordering the products need is
// carried by a barrier: QK(j) into S/P buffer j % 3 waits for PV(j - 3), the
// last reader of that buffer (v_empty); PV(j) waits for P(j) (p_ready) and
// for its V half (kv_full, long complete).  Tile j: K slot and S/P buffer
// j % 3, V slot j % 4; j counts the tiles of this pair's items.
template <bool kIsQK>
__device__ __forceinline__ void pair_mma(const PrefillArgs &a, PairSmem &sm, uint32_t tmem,
                                         const PairCtx &c)
{
    uint32_t q_it = 0, j = 0;
    bool ok = true;
    const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        if (!pwait1(&sm.item_full[slot], (it >> 1) & 1, c))
            break;
        const int item = sm.meta[slot].item, info = sm.meta[slot].info;
        mbar_arrive(&sm.item_empty[slot]);
        if (item < 0)
            break;
        const int N = meta_n(info);
        if (N == 0)
            continue;
        if (kIsQK) {
            // The previous item's last P V product is issued before this item's
            // first Q K^T, so that it is not queued behind up to three S tiles
            // of this item: the softmax waits for it before its epilogue.
            // (q_it counts the items with tiles; the PV issuer completes phase
            // q of pv_issued with item q's last product, and cannot complete
            // phase q + 1 before this item's S exists.)
            if (q_it > 0 && !pwait1(&sm.pv_issued, (q_it - 1) & 1, c))
                break;
            const int qbuf = q_it & 1;
            if (!pwait1(&sm.q_full[qbuf], (q_it >> 1) & 1, c))
                break;
            ++q_it;
            tc_fence_after();
            const uint32_t qaddr = q_addr[qbuf];
            for (int n = 0; n < N && ok; ++n) {
                const uint32_t jj = j + n, b = jj % 3, vs = jj % kVSlots;
                // the S/P buffer's last reader, and the tile's K/V halves
                if ((jj >= 3 && !pwait1(&sm.v_empty[(jj - 3) % kVSlots], ((jj - 3) / kVSlots) & 1, c)) ||
                    !pwait1(&sm.kv_full[vs], (jj / kVSlots) & 1, c)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sm.k[b]);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k & 3) * 32;
                    tc_mma_pair(tmem + kColS + 128 * b,
                                sdesc_sw128(qaddr + (k >> 2) * kHalfBytes + off, 16, 1024),
                                sdesc_sw128(kaddr + (k >> 2) * (kHalf / 2) + off, 16, 1024),
                                kIdescQK2, k > 0);
                }
                tc_commit_pair(&sm.s_full[b], kBothCtas);
                if (n == N - 1)
                    tc_commit_pair(&sm.q_empty[qbuf], kBothCtas);
            }
        } else {
            // the tile loop, compiled twice: with the remainder products and without
            auto tiles = [&](auto split_tag) {
                constexpr bool kSplit = decltype(split_tag)::value;
                for (int n = 0; n < N && ok; ++n) {
                    const uint32_t jj = j + n, b = jj % 3, vs = jj % kVSlots;
                    if (!pwait1(&sm.p_ready[b], (jj / 3) & 1, c) ||
                        !pwait1(&sm.kv_full[vs], (jj / kVSlots) & 1, c)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vaddr = smem_u32(sm.v[vs]);
                    const uint32_t tp = tmem + kColS + 128 * b;
#pragma unroll
                    for (int k = 0; k < T / 16; ++k)
                        tc_mma_ts_pair(tmem + kColO, tp + (k < 4 ? 8 * k : 64 + 8 * (k - 4)),
                                       sdesc_sw128(vaddr + k * 2048, kHalf, 1024), kIdescPV2,
                                       (n > 0 || k > 0) ? 1u : 0u);
                    // few-key rows: the remainder P - bf16(P), 32 columns further on
                    if constexpr (kSplit) {
#pragma unroll
                        for (int k = 0; k < T / 16; ++k)
                            tc_mma_ts_pair(tmem + kColO, tp + (k < 4 ? 32 + 8 * k : 96 + 8 * (k - 4)),
                                           sdesc_sw128(vaddr + k * 2048, kHalf, 1024), kIdescPV2, 1u);
                    }
                    tc_commit_pair(&sm.v_empty[vs], kBothCtas);
                    if (n == N - 1) {
                        tc_commit_pair(&sm.o_done, kBothCtas);
                        mbar_arrive(&sm.pv_issued);
                    }
                }
            };
            if (meta_split(info))
                tiles(std::true_type{});
            else
                tiles(std::false_type{});
        }
        j += N;
    }
    // All of this thread's MMAs must have completed before TMEM is released.
    tc_commit_pair(&sm.teardown, 1);
}

// Softmax warps: warpgroup wg, thread = query row r, columns 64 wg .. +63 of
// every S tile of this CTA's head.
template <bool kVarlen, int kL>
__device__ __forceinline__ void pair_softmax(const PrefillArgs &a, PairSmem &sm, uint32_t tmem,
                                             int warp, const TmapTable<kL> &tm, const PairCtx &c)
{
    uint32_t *err = c.err;
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int lane = threadIdx.x & 31;
    const int r = quad * 32 + lane;                       // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t bar_id = 1 + quad;                     // this row quad's two warps
    const uint32_t tO = tmem + lane_base + kColO + 64 * wg;
    const float NEG_INF = -__int_as_float(0x7f800000);
    uint32_t j = 0, o_cnt = 0;

    for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!pwait(&sm.item_full[slot], (it >> 1) & 1, c, c.rank != 0))
            break;
        const ItemMeta mt = sm.meta[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive_remote(lead_bar(&sm.item_empty[slot]));
        if (mt.item < 0)
            break;
        const ItemInfo x = meta_item<kVarlen, kL>(mt, a);
        bool store;
        const int qh = item_head(x, static_cast<int>(c.rank), a, store);
        const int N = meta_n(mt.info);
        const int mode = meta_mode(mt.info);
        int n_sink = 0, kb_lo = 0;
        if (mode == EA_SSA)
            ssa_tiles(x.qb, a.sink, a.window, n_sink, kb_lo);
        const bool diag_kept = meta_diag(mt.info);
        const bool split = meta_split(mt.info);   // P V in two bf16 parts (few kept keys)
        const int i = x.qb * T + r;
        float m_run = NEG_INF, l_run = 0.f, dl_run = 0.f;
        bool ok = true;

        // the tile loop, compiled twice: with P's remainder (rare items) and without
        auto tiles = [&](auto split_tag) {
            constexpr bool kSplit = decltype(split_tag)::value;
            for (int n = 0; n < N; ++n) {
                const uint32_t jj = j + n;
                const uint32_t b = jj % 3;
                int kb;
                if (mode == EA_BLOCK)
                    kb = (n == N - 1 && diag_kept) ? x.qb : -1;  // only the diagonal needs its index
                else
                    kb = seq_kb(mode, n, n_sink, kb_lo);
                if (!pwait(&sm.s_full[b], (jj / 3) & 1, c)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tS = tmem + lane_base + kColS + 128 * b + 64 * wg;
                uint32_t s[64];
                tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_wait_ld();

                // mask edge tiles only: key j0 + c is kept when c <= hi (causal)
                // and, for SSA, when c < sk (sink) or c > lo (inside the window);
                // one keep word per 32 columns, built from three prefix masks
                const bool edge = kb >= 0 && !tile_is_full(mode, x.qb, kb, a.sink, a.window);
                if (edge) {
                    const int j0 = kb * T;
                    const int hi = i - j0;
                    int sk = -1, lo = -1;
                    if (mode == EA_SSA) {
                        sk = a.sink - j0;
                        lo = i - a.window - j0;
                    }
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int co = 64 * wg + 32 * q;
                        const uint32_t w = low_bits(hi + 1 - co) & (low_bits(sk - co) | ~low_bits(lo + 1 - co));
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            if (!((w >> cc) & 1u))
                                s[32 * q + cc] = __float_as_uint(NEG_INF);
                    }
                }
                // partial row max over this warpgroup's 64 columns (eight 3-input
                // chains), then the row's max with the other warpgroup's
                float mxa[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mxa[k] = max3f(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]), NEG_INF);
#pragma unroll
                for (int cc = 16; cc < 64; cc += 16)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mxa[k] = max3f(mxa[k], __uint_as_float(s[cc + 2 * k]), __uint_as_float(s[cc + 2 * k + 1]));
                const float pm = max3f(max3f(mxa[0], mxa[1], mxa[2]), max3f(mxa[3], mxa[4], mxa[5]),
                                       fmaxf(mxa[6], mxa[7]));
                sm.red_max[jj & 1][wg][r] = pm;
                named_bar_sync(bar_id, 64);
                float mx = fmaxf(pm, sm.red_max[jj & 1][wg ^ 1][r]);
                mx *= a.scale_log2;
                const float m_new = fmaxf(m_run, mx);
                float factor = 1.f;
                bool rescale_o = false;
                if (m_new > m_run + kRescaleThreshold) {
                    if (m_run > NEG_INF) {
                        factor = ex2(m_run - m_new);
                        l_run *= factor;
                        dl_run *= factor;
                        rescale_o = n > 0;
                    }
                    m_run = m_new;
                }
                const float mb = m_run > NEG_INF ? m_run : 0.f;
                if constexpr (!kSplit) {
                    // The largest probability of this thread's columns enters O
                    // rounded to bf16, and it is not 1 (exact) unless the lazy
                    // running maximum is this tile's.  Its rounding error joins
                    // the normaliser of O, so that a dominant key's weight stays
                    // exact; the LSE keeps the unrounded sum.  (Same operations as
                    // the loop below, so the same value.)
                    const float pmx = ex2(fmaf(pm, a.scale_log2, -mb));
                    dl_run += __uint_as_float(pack_bf16x2(pmx, 0.f) << 16) - pmx;
                }
                // p = 2^(s * scale_log2 - mb): the affine part two lanes at a time,
                // the row sum in four packed accumulators, P packed to bf16 pairs
                // in place (s[c/2] once s[c], s[c+1] are consumed).  Rows that
                // keep few keys also take P's remainder P - bf16(P), rounded to
                // bf16, which a second P V product reads 32 columns further on
                // (an error of 2^-9 of the remainder, 2^-17 of P, is left); it
                // goes to TMEM 16 columns at a time, over S already read.
                const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
                const uint64_t nm2 = f2_pack(-mb, -mb);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t rem[16];
#pragma unroll
                for (int cc = 0; cc < 64; cc += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[cc]), __uint_as_float(s[cc + 1])), sc2, nm2),
                              x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    acc[(cc >> 1) & 3] = f2_add(acc[(cc >> 1) & 3], f2_pack(p0, p1));
                    const uint32_t hi = pack_bf16x2(p0, p1);
                    s[cc >> 1] = hi;
                    if constexpr (kSplit) {
                        rem[(cc >> 1) & 15] = pack_bf16x2(p0 - __uint_as_float(hi << 16),
                                                          p1 - __uint_as_float(hi & 0xffff0000u));
                        if (((cc >> 1) & 15) == 15)
                            tmem_st16(tS + 32 + ((cc >> 1) & ~15), rem);
                    }
                }
                float l0, l1, l2, l3;
                f2_unpack(f2_add(acc[0], acc[1]), l0, l1);
                f2_unpack(f2_add(acc[2], acc[3]), l2, l3);
                l_run += (l0 + l1) + (l2 + l3);

                // O rescale: PV of the previous tile must have completed
                if (__any_sync(0xffffffffu, rescale_o)) {
                    if (!pwait(&sm.v_empty[(jj - 1) % kVSlots], ((jj - 1) / kVSlots) & 1, c)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            o[cc] = __float_as_uint(__uint_as_float(o[cc]) * factor);
                        tmem_st32(tO + ch * 32, o);
                    }
                }
                // P (bf16 pairs) over the first 32 of this warpgroup's S columns
                tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(lead_bar(&sm.p_ready[b]));
            }
        };
        if (split)
            tiles(std::true_type{});
        else
            tiles(std::false_type{});
        if (!ok)
            break;
        j += N;

        // epilogue: O / l -> bf16, LSE = ln(2^m * l).  What needs no O (the
        // row-sum exchange, the stage's release by the previous item's store)
        // comes first, while the item's last P V product completes.
        sm.red_l[it & 1][wg][r] = l_run;
        sm.red_dl[it & 1][wg][r] = dl_run;
        named_bar_sync(bar_id, 64);
        const float l_tot = l_run + sm.red_l[it & 1][wg ^ 1][r];
        // O's normaliser: the sum of the probabilities as O received them
        const float ln_tot = l_tot + (dl_run + sm.red_dl[it & 1][wg ^ 1][r]);
        const int row0 = x.qb * T + quad * 32;   // the warp's first row in its sequence
        const bool staged = store && (!kVarlen || row0 + 32 <= x.S);
        if (staged) {
            if (lane == 0)
                bulk_wait_read_all();     // the previous item's store has read the stage
            __syncwarp();
        }
        if (N > 0) {
            if (!pwait(&sm.o_done, o_cnt & 1, c))
                break;
            ++o_cnt;
            tc_fence_after();
        }
        const RowInfo &e = x;   // the row's layer, sequence, length and offsets
        const bool row_ok = store && i < e.S &&
                            in_bounds(e.tok0 + i, kVarlen ? a.total_tokens : a.S, err) &&
                            in_bounds(qh, a.Hq, err);
        const float inv_l = ln_tot > 0.f ? 1.f / ln_tot : 0.f;
        __nv_bfloat16 *orow = a.O[e.layer] + e.b * a.o_sb + static_cast<int64_t>(e.tok0 + i) * a.o_ss +
                              qh * a.o_sh + 64 * wg;
        // A warp stages its 32 rows x 64 columns in shared memory (128-byte
        // swizzle, as the tensor map expects) and its lane 0 stores them with
        // TMA, which skips rows past S in a fixed-length batch.  In a variable-
        // length batch the warp over a sequence's end stores its rows directly:
        // the rows past the end belong to the next sequence.
        const int wrow = r & 31;
        uint8_t *wstage = sm.ostage + warp * (kTileBytes / 8);
        // both halves of this warp's O columns in one round trip to TMEM
        uint32_t oo[2][32];
        if (N > 0) {
            tmem_ld32(tO, oo[0]);
            tmem_ld32(tO + 32, oo[1]);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
                oo[0][cc] = oo[1][cc] = 0u;
        }
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const uint32_t (&o)[32] = oo[ch];
            uint32_t w[16];
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
                w[cc] = pack_bf16x2(__uint_as_float(o[2 * cc]) * inv_l,
                                    __uint_as_float(o[2 * cc + 1]) * inv_l);
            if (staged) {
                // columns ch*32 .. +31 of the warp's 64: 16-byte chunks ch*4 .. +3
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int c16 = ch * 4 + q4;
                    *reinterpret_cast<uint4 *>(wstage + wrow * 128 + ((c16 ^ (wrow & 7)) << 4)) =
                        make_uint4(w[q4 * 4], w[q4 * 4 + 1], w[q4 * 4 + 2], w[q4 * 4 + 3]);
                }
            } else if (row_ok) {
                if (a.o_v8) {
                    // whole 32-byte sectors: half the store instructions
#pragma unroll
                    for (int q8 = 0; q8 < 2; ++q8)
                        st_global_v8(orow + ch * 32 + q8 * 16, &w[q8 * 8]);
                } else {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4 *>(orow + ch * 32 + q4 * 8) =
                            make_uint4(w[q4 * 4], w[q4 * 4 + 1], w[q4 * 4 + 2], w[q4 * 4 + 3]);
                }
            }
        }
        if (staged) {
            fence_proxy_async_smem();     // the stage's writes -> the TMA unit
            __syncwarp();
            if (lane == 0) {
                tma_store_4d(&tm.o[kL == 1 ? 0 : e.layer], wstage, 64 * wg, qh, (kVarlen ? e.tok0 : 0) + row0, e.tma_b);
                bulk_commit_group();
            }
        }
        if (wg == 0 && row_ok && a.LSE[e.layer] &&
            in_bounds(e.b * a.lse_sb + qh * a.lse_sh + e.tok0 + i, a.lse_elems, err))
            a.LSE[e.layer][e.b * a.lse_sb + qh * a.lse_sh + e.tok0 + i] =
                l_tot > 0.f ? (m_run + __log2f(l_tot)) * 0.69314718055994531f : NEG_INF;
        tc_fence_before();
    }
    // On an abort this thread may have left its row partner waiting at their
    // named barrier: one arrival releases it (its next wait then fails too).
    if (*c.abort)
        named_bar_arrive(bar_id, 64);
    // the last stores must be complete before the CTA (and its shared memory) goes
    if (lane == 0)
        bulk_wait_all();
}

template <bool kVarlen, int kL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    hybrid_prefill_kernel(const __grid_constant__ TmapTable<kL> tm, const PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    PairSmem &sm = *reinterpret_cast<PairSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(&sm.kv_full[s], 1);      // rank 0's producer; bytes from both CTAs
            mbar_init(&sm.v_empty[s], 1);      // MMA commit (multicast)
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sm.q_full[t], 1);
            mbar_init(&sm.q_empty[t], 1);
            mbar_init(&sm.item_full[t], 1);
            // rank 0: its two MMA issuers and 8 softmax warps, rank 1's producer and 8 softmax warps
            mbar_init(&sm.item_empty[t], 19);
        }
        for (int t = 0; t < 3; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_ready[t], 16);     // 8 softmax warps of each CTA
        }
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.teardown, 2);            // one commit from each MMA issuer
        mbar_init(&sm.pv_issued, 1);           // the PV issuer, once per item with tiles
        sm.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kPMmaWarp) {
        tmem_alloc_pair(&sm.tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == kPProducerWarp && lane == 0 && kL == 1) {
        tma_prefetch_desc(&tm.q[0]);
        tma_prefetch_desc(&tm.k[0]);
        tma_prefetch_desc(&tm.v[0]);
        tma_prefetch_desc(&tm.o[0]);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // both CTAs' barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    PairCtx c;
    c.rank = rank;
    c.peer_abort = mapa_shared(smem_u32(&sm.abort), rank ^ 1u);
    c.abort = &sm.abort;
    c.err = &a.hdr->error;
    c.timeout_ns = a.wait_timeout_ns;

    if (warp < 8)
        pair_softmax<kVarlen, kL>(a, sm, tmem, warp, tm, c);
    else if (warp == kPProducerWarp)
        pair_producer<kVarlen, kL>(tm, a, sm, c, lane);
    else if (warp == kPMmaWarp && rank == 0 && lane == 0)
        pair_mma<true>(a, sm, tmem, c);
    else if (warp == kPPvWarp && rank == 0 && lane == 0)
        pair_mma<false>(a, sm, tmem, c);
    // every MMA has completed before TMEM is released
    if (rank == 0 && (warp == kPMmaWarp || warp == kPPvWarp) && lane == 0) {
        volatile int no_abort = 0;
        mbar_wait(&sm.teardown, 0, &no_abort, c.err);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // no remote arrival or MMA into this CTA is still to come
    if (warp == kPMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

} // namespace ea

using namespace ea;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by the planner and the attention launch; fills the kernel
// arguments that do not depend on the tensors.
static ea_status prefill_common(int B, int S, int Hq, int Hkv, int d, const uint8_t *m, int sink,
                                int window, const uint8_t *block_mask, int block_size,
                                void *workspace, size_t ws_bytes, PrefillArgs &a,
                                int qb_begin = 0, int qb_end = -1)
{
    if (!m)
        return EA_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || sink < 0 || window < 1 ||
        block_size != EA_TILE)
        return EA_ERR_INVALID_ARG;
    if (d != EA_HEAD_DIM || S > EA_MAX_SEQ || B > 65535)
        return EA_ERR_UNSUPPORTED;
    const PrefillWs L = prefill_ws_layout(B, S, Hq, Hkv);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < L.total)
        return EA_ERR_WORKSPACE;
    const int64_t nB = ceil_div(S, T);
    const int64_t n_rows = static_cast<int64_t>(B) * Hkv * nB;
    const int g = Hq / Hkv;
    const int npairs = (g + 1) / 2;
    if (n_rows * npairs >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a = PrefillArgs{};
    a.m[0] = m;
    a.block_mask[0] = block_mask;
    a.n_layers = 1;
    a.n_sort_groups = 1;
    a.costs = reinterpret_cast<int32_t *>(ws + L.costs);
    a.items = reinterpret_cast<uint32_t *>(ws + L.items);
    a.hdr = reinterpret_cast<ea_ws_header *>(ws);
    a.B = B;
    a.S = S;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = g;
    a.npairs = npairs;
    a.nB = static_cast<int>(nB);
    a.sink = sink < S ? sink : S;        // sink or window beyond S keep the same pairs
    a.window = window < S ? window : S;
    if (qb_end < 0)
        qb_end = static_cast<int>(nB);
    if (qb_begin < 0 || qb_begin >= qb_end || qb_end > nB)
        return EA_ERR_INVALID_ARG;
    a.qb_begin = qb_begin;
    a.qb_end = qb_end;
    a.lse_sb = static_cast<int64_t>(Hq) * S;
    a.lse_sh = S;
    a.lse_elems = static_cast<int64_t>(B) * Hq * S;
    a.mask_elems = block_mask ? static_cast<int64_t>(B) * Hkv * nB * nB : 0;
    a.visited_bits = static_cast<int64_t>(B) * Hkv * nB * nB;
    a.n_rows = static_cast<uint32_t>(n_rows);
    a.rows_per_layer = static_cast<uint32_t>(n_rows);
    a.n_items = static_cast<uint32_t>(static_cast<int64_t>(B) * Hkv * (qb_end - qb_begin) * npairs);
    a.wait_timeout_ns = EA_WAIT_TIMEOUT_NS;
    a.test_skip_load = -1;
    return EA_OK;
}

// Histogram bins the planner's sort may use (shared memory): a whole
// single-layer plan at the longest length, or a multi-layer plan sorted by
// layer while it fits (longer multi-layer plans are sorted by cost alone).
constexpr int kMaxSortBins = 48 * 1024;
static_assert(kMaxSortBins >= EA_MAX_SEQ / T + 2, "sort histogram");

static bool g_attr_done[64] = {};
static int g_max_clusters[64] = {};   // co-resident CTA pairs of the attention kernel, per device

static ea_status ensure_attributes()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return EA_ERR_CUDA;
    if (dev < 64 && g_attr_done[dev])
        return EA_OK;
    if (cudaFuncSetAttribute(hybrid_prefill_kernel<false, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPairSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(hybrid_prefill_kernel<true, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPairSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(hybrid_prefill_kernel<false, kMaxLayers>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPairSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(plan_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(int) * kMaxSortBins)) != cudaSuccess)
        return EA_ERR_CUDA;
    // How many CTA pairs fit on the device at once (one CTA per SM; an odd SM
    // count or pair placement rules can leave SMs out).
    int clusters = 0;
    {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        cfg.blockDim = dim3(kPThreads, 1, 1);
        cfg.dynamicSmemBytes = kPairSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, hybrid_prefill_kernel<false, 1>, &cfg) !=
                cudaSuccess ||
            clusters < 1)
            return EA_ERR_CUDA;
    }
    if (dev < 64) {
        g_max_clusters[dev] = clusters;
        g_attr_done[dev] = true;
    }
    return EA_OK;
}

#ifdef EA_CHECKS
// Fault injection of the bounds-checked build's tests: the next attention
// launch leaves out one K/V load and uses a short wait limit.
static int64_t g_test_skip_load = -1;
static uint64_t g_test_timeout_ns = 0;

extern "C" ea_status ea_checked_inject_prefill_timeout(int64_t skip_load, uint64_t timeout_ns)
{
    if (skip_load < 0 || timeout_ns == 0)
        return EA_ERR_INVALID_ARG;
    g_test_skip_load = skip_load;
    g_test_timeout_ns = timeout_ns;
    return EA_OK;
}
#endif

namespace ea {

ea_status prefill_plan_range(int B, int S, int Hq, int Hkv, int d, const uint8_t *m, int sink,
                             int window, const uint8_t *block_mask, int block_size, void *workspace,
                             size_t ws_bytes, int qb_begin, int qb_end, void *stream)
{
    PrefillArgs a;
    ea_status s = prefill_common(B, S, Hq, Hkv, d, m, sink, window, block_mask, block_size,
                                 workspace, ws_bytes, a, qb_begin, qb_end);
    if (s != EA_OK)
        return s;
    if ((s = ensure_attributes()) != EA_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int warps_per_cta = 8;
    const unsigned cost_blocks = static_cast<unsigned>(ceil_div(a.n_rows, warps_per_cta));
    plan_costs_kernel<<<cost_blocks, warps_per_cta * 32, 0, st>>>(a);
    plan_sort_kernel<<<1, 1024, sizeof(int) * (a.nB + 2), st>>>(a);
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}

template <int kL>
static ea_status launch_attend(const TmapTable<kL> &tm, const PrefillArgs &a, void *stream);

ea_status prefill_attend_range(const void *Q, const void *K, const void *V, void *O, float *LSE,
                               const int64_t q_str[4], const int64_t kv_str[4],
                               const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                               float scale, const uint8_t *m, int sink, int window,
                               const uint8_t *block_mask, int block_size, void *workspace,
                               size_t ws_bytes, uint32_t *visited_bitmap, int qb_begin, int qb_end,
                               void *stream)
{
    if (!Q || !K || !V || !O || !q_str || !kv_str || !o_str || !(scale > 0.f))
        return EA_ERR_INVALID_ARG;
    PrefillArgs a;
    ea_status s = prefill_common(B, S, Hq, Hkv, d, m, sink, window, block_mask, block_size,
                                 workspace, ws_bytes, a, qb_begin, qb_end);
    if (s != EA_OK)
        return s;
    if (q_str[3] != 1 || kv_str[3] != 1 || o_str[3] != 1)
        return EA_ERR_INVALID_ARG;
    for (int k = 0; k < 3; ++k)
        if (q_str[k] <= 0 || kv_str[k] <= 0 || o_str[k] <= 0 || q_str[k] % 8 || kv_str[k] % 8 ||
            o_str[k] % 8)
            return EA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return EA_ERR_INVALID_ARG;
    TmapTable<1> tm;
    if (!encode_tmap_bf16_4d(&tm.q[0], Q, d, Hq, S, B, q_str, 64, T, true) ||
        !encode_tmap_bf16_4d(&tm.k[0], K, d, Hkv, S, B, kv_str, 64, T / 2, true) ||
        !encode_tmap_bf16_4d(&tm.v[0], V, d, Hkv, S, B, kv_str, 64, T, true) ||
        !encode_tmap_bf16_4d(&tm.o[0], O, d, Hq, S, B, o_str, 64, 32, true))
        return EA_ERR_INVALID_ARG;
    a.O[0] = static_cast<__nv_bfloat16 *>(O);
    a.o_sb = o_str[0];
    a.o_ss = o_str[1];
    a.o_sh = o_str[2];
    a.o_v8 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0 && o_str[0] % 16 == 0 && o_str[1] % 16 == 0 &&
             o_str[2] % 16 == 0;
    a.LSE[0] = LSE;
    a.visited = visited_bitmap;
    a.scale_log2 = scale * 1.4426950408889634f;
    return launch_attend(tm, a, stream);
}

// The persistent attention launch over a plan made with the same arguments:
// as many CTA pairs as fit on the device (or as there are items).
template <int kL>
static ea_status launch_attend(const TmapTable<kL> &tm, const PrefillArgs &a_in, void *stream)
{
    ea_status s;
    if ((s = ensure_attributes()) != EA_OK)
        return s;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return EA_ERR_CUDA;
    PrefillArgs a = a_in;
#ifdef EA_CHECKS
    if (g_test_skip_load >= 0) {
        a.test_skip_load = g_test_skip_load;
        a.wait_timeout_ns = g_test_timeout_ns;
        g_test_skip_load = -1;
    }
#endif
    const uint32_t clusters = static_cast<uint32_t>(g_max_clusters[dev]);
    const unsigned grid = 2u * (a.n_items < clusters ? (a.n_items > 0 ? a.n_items : 1u) : clusters);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if constexpr (kL == 1) {
        if (a.cu_seqlens)
            hybrid_prefill_kernel<true, 1><<<grid, kPThreads, kPairSmemBytes, st>>>(tm, a);
        else
            hybrid_prefill_kernel<false, 1><<<grid, kPThreads, kPairSmemBytes, st>>>(tm, a);
    } else {
        hybrid_prefill_kernel<false, kL><<<grid, kPThreads, kPairSmemBytes, st>>>(tm, a);
    }
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}

} // namespace ea

extern "C" ea_status ea_hybrid_attn_prefill_varlen(
    const void *Q, const void *K, const void *V, void *O, float *LSE, const int64_t q_str[3],
    const int64_t kv_str[3], const int64_t o_str[3], const int32_t *cu_seqlens, int B,
    int total_tokens, int max_seqlen, int Hq, int Hkv, int d, float scale, const uint8_t *m,
    int sink, int window, const uint8_t *block_mask, int block_size, void *workspace,
    size_t ws_bytes, void *stream)
{
    if (!Q || !K || !V || !O || !q_str || !kv_str || !o_str || !cu_seqlens || !m ||
        !(scale > 0.f))
        return EA_ERR_INVALID_ARG;
    if (B < 1 || total_tokens < 1 || max_seqlen < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
        sink < 0 || window < 1 || block_size != EA_TILE)
        return EA_ERR_INVALID_ARG;
    if (d != EA_HEAD_DIM || max_seqlen > EA_MAX_SEQ || Hkv > 65535)
        return EA_ERR_UNSUPPORTED;
    if (q_str[2] != 1 || kv_str[2] != 1 || o_str[2] != 1)
        return EA_ERR_INVALID_ARG;
    for (int k = 0; k < 2; ++k)
        if (q_str[k] <= 0 || kv_str[k] <= 0 || o_str[k] <= 0 || q_str[k] % 8 || kv_str[k] % 8 ||
            o_str[k] % 8)
            return EA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return EA_ERR_INVALID_ARG;
    const PrefillVarlenWs L = prefill_varlen_ws_layout(B, total_tokens, Hq, Hkv);
    const int g = Hq / Hkv;
    const int npairs = (g + 1) / 2;
    if (L.rows * npairs >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < L.total)
        return EA_ERR_WORKSPACE;
    // one packed sequence of total_tokens rows, batch extent 1
    const int64_t q4[4] = {static_cast<int64_t>(total_tokens) * q_str[0], q_str[0], q_str[1], 1};
    const int64_t kv4[4] = {static_cast<int64_t>(total_tokens) * kv_str[0], kv_str[0], kv_str[1], 1};
    const int64_t o4[4] = {static_cast<int64_t>(total_tokens) * o_str[0], o_str[0], o_str[1], 1};
    TmapTable<1> tm;
    if (!encode_tmap_bf16_4d(&tm.q[0], Q, d, Hq, total_tokens, 1, q4, 64, T, true) ||
        !encode_tmap_bf16_4d(&tm.k[0], K, d, Hkv, total_tokens, 1, kv4, 64, T / 2, true) ||
        !encode_tmap_bf16_4d(&tm.v[0], V, d, Hkv, total_tokens, 1, kv4, 64, T, true) ||
        !encode_tmap_bf16_4d(&tm.o[0], O, d, Hq, total_tokens, 1, o4, 64, 32, true))
        return EA_ERR_INVALID_ARG;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    PrefillArgs a{};
    a.m[0] = m;
    a.block_mask[0] = block_mask;
    a.n_layers = 1;
    a.n_sort_groups = 1;
    a.costs = reinterpret_cast<int32_t *>(ws + L.costs);
    a.items = reinterpret_cast<uint32_t *>(ws + L.items);
    a.hdr = reinterpret_cast<ea_ws_header *>(ws);
    a.B = B;
    a.S = max_seqlen;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = g;
    a.npairs = npairs;
    a.nB = static_cast<int>(ceil_div(max_seqlen, T));
    a.sink = sink < max_seqlen ? sink : max_seqlen;
    a.window = window < max_seqlen ? window : max_seqlen;
    a.qb_begin = 0;
    a.qb_end = a.nB;
    a.n_rows = static_cast<uint32_t>(L.rows);
    a.rows_per_layer = static_cast<uint32_t>(L.rows);
    a.n_items = static_cast<uint32_t>(L.rows * npairs);
    a.O[0] = static_cast<__nv_bfloat16 *>(O);
    a.o_sb = 0;
    a.o_ss = o_str[0];
    a.o_sh = o_str[1];
    a.o_v8 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0 && o_str[0] % 16 == 0 && o_str[1] % 16 == 0;
    a.LSE[0] = LSE;
    a.lse_sb = 0;
    a.lse_sh = total_tokens;
    a.lse_elems = static_cast<int64_t>(Hq) * total_tokens;
    a.mask_elems = block_mask ? -1 : 0;   // the masks' total is mask_off[B], known on the device
    a.visited_bits = 0;
    a.visited = nullptr;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.cu_seqlens = cu_seqlens;
    a.row_off = reinterpret_cast<int32_t *>(ws + L.row_off);
    a.mask_off = reinterpret_cast<int64_t *>(ws + L.mask_off);
    a.row_desc = reinterpret_cast<int2 *>(ws + L.row_desc);
    a.max_seqlen = max_seqlen;
    a.total_tokens = total_tokens;
    a.wait_timeout_ns = EA_WAIT_TIMEOUT_NS;
    a.test_skip_load = -1;
    // the queue sequence by sequence when the planner's histogram holds it
    if (static_cast<int64_t>(B) * (a.nB + 1) + 1 <= kMaxSortBins) {
        a.sort_group = 2;
        a.n_sort_groups = B;
    }

    ea_status s;
    if ((s = ensure_attributes()) != EA_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int warps_per_cta = 8;
    varlen_setup_kernel<<<1, 1024, 0, st>>>(a);
    plan_costs_kernel<<<static_cast<unsigned>(ceil_div(a.n_rows, warps_per_cta)),
                        warps_per_cta * 32, 0, st>>>(a);
    plan_sort_kernel<<<1, 1024, sizeof(int) * (a.n_sort_groups * (a.nB + 1) + 1), st>>>(a);
    if (cudaGetLastError() != cudaSuccess)
        return EA_ERR_CUDA;
    return launch_attend(tm, a, stream);
}

extern "C" ea_status ea_prefill_plan(int B, int S, int Hq, int Hkv, int d, const uint8_t *m,
                                     int sink, int window, const uint8_t *block_mask,
                                     int block_size, void *workspace, size_t ws_bytes, void *stream)
{
    return prefill_plan_range(B, S, Hq, Hkv, d, m, sink, window, block_mask, block_size, workspace,
                              ws_bytes, 0, -1, stream);
}

extern "C" ea_status ea_prefill_attend(const void *Q, const void *K, const void *V, void *O,
                                       float *LSE, const int64_t q_str[4], const int64_t kv_str[4],
                                       const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                                       float scale, const uint8_t *m, int sink, int window,
                                       const uint8_t *block_mask, int block_size, void *workspace,
                                       size_t ws_bytes, uint32_t *visited_bitmap, void *stream)
{
    return prefill_attend_range(Q, K, V, O, LSE, q_str, kv_str, o_str, B, S, Hq, Hkv, d, scale, m,
                                sink, window, block_mask, block_size, workspace, ws_bytes,
                                visited_bitmap, 0, -1, stream);
}

// Every host-side check of a fixed-length prefill call (tensors included),
// so that a rejected call enqueues nothing.
static ea_status prefill_validate(const void *Q, const void *K, const void *V, void *O,
                                  const int64_t q_str[4], const int64_t kv_str[4],
                                  const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                                  float scale, const uint8_t *m, int sink, int window,
                                  const uint8_t *block_mask, int block_size, void *workspace,
                                  size_t ws_bytes)
{
    if (!Q || !K || !V || !O || !q_str || !kv_str || !o_str || !(scale > 0.f))
        return EA_ERR_INVALID_ARG;
    PrefillArgs a;
    ea_status s = prefill_common(B, S, Hq, Hkv, d, m, sink, window, block_mask, block_size,
                                 workspace, ws_bytes, a);
    if (s != EA_OK)
        return s;
    if (q_str[3] != 1 || kv_str[3] != 1 || o_str[3] != 1)
        return EA_ERR_INVALID_ARG;
    for (int k = 0; k < 3; ++k)
        if (q_str[k] <= 0 || kv_str[k] <= 0 || o_str[k] <= 0 || q_str[k] % 8 || kv_str[k] % 8 ||
            o_str[k] % 8)
            return EA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return EA_ERR_INVALID_ARG;
    return EA_OK;
}

extern "C" ea_status ea_hybrid_attn_prefill(const void *Q, const void *K, const void *V, void *O,
                                            float *LSE, const int64_t q_str[4],
                                            const int64_t kv_str[4], const int64_t o_str[4], int B,
                                            int S, int Hq, int Hkv, int d, float scale,
                                            const uint8_t *m, int sink, int window,
                                            const uint8_t *block_mask, int block_size,
                                            void *workspace, size_t ws_bytes,
                                            uint32_t *visited_bitmap, void *stream)
{
    // Validate everything (tensors included) before enqueueing the planner.
    ea_status s = prefill_validate(Q, K, V, O, q_str, kv_str, o_str, B, S, Hq, Hkv, d, scale, m,
                                   sink, window, block_mask, block_size, workspace, ws_bytes);
    if (s != EA_OK)
        return s;
    s = ea_prefill_plan(B, S, Hq, Hkv, d, m, sink, window, block_mask, block_size, workspace,
                        ws_bytes, stream);
    if (s != EA_OK)
        return s;
    return ea_prefill_attend(Q, K, V, O, LSE, q_str, kv_str, o_str, B, S, Hq, Hkv, d, scale, m,
                             sink, window, block_mask, block_size, workspace, ws_bytes,
                             visited_bitmap, stream);
}

extern "C" size_t ea_prefill_layers_workspace_size(int n_layers, int B, int S, int Hq, int Hkv, int d)
{
    if (n_layers < 1 || n_layers > EA_MAX_PREFILL_LAYERS || B < 1 ||
        static_cast<int64_t>(B) * n_layers > 65535)
        return 0;
    return ea_prefill_workspace_size(B * n_layers, S, Hq, Hkv, d);
}

extern "C" ea_status ea_hybrid_attn_prefill_layers(const ea_prefill_layer *layers, int n_layers,
                                                   const int64_t q_str[4], const int64_t kv_str[4],
                                                   const int64_t o_str[4], int B, int S, int Hq,
                                                   int Hkv, int d, float scale, int sink, int window,
                                                   int block_size, void *workspace, size_t ws_bytes,
                                                   void *stream)
{
    if (!layers || n_layers < 1)
        return EA_ERR_INVALID_ARG;
    if (n_layers > EA_MAX_PREFILL_LAYERS)
        return EA_ERR_UNSUPPORTED;
    // every layer's arguments, as a single-layer call checks them
    for (int l = 0; l < n_layers; ++l) {
        const ea_prefill_layer &ly = layers[l];
        const ea_status s = prefill_validate(ly.Q, ly.K, ly.V, ly.O, q_str, kv_str, o_str, B, S, Hq,
                                             Hkv, d, scale, ly.m, sink, window, ly.block_mask,
                                             block_size, workspace, ws_bytes);
        if (s != EA_OK)
            return s;
    }
    const size_t need = ea_prefill_layers_workspace_size(n_layers, B, S, Hq, Hkv, d);
    if (need == 0)
        return EA_ERR_UNSUPPORTED;
    if (ws_bytes < need)
        return EA_ERR_WORKSPACE;
    PrefillArgs a;
    ea_status s = prefill_common(B, S, Hq, Hkv, d, layers[0].m, sink, window, layers[0].block_mask,
                                 block_size, workspace, ws_bytes, a);
    if (s != EA_OK)
        return s;
    // rows of every layer, numbered layer by layer
    const PrefillWs WL = prefill_ws_layout(B * n_layers, S, Hq, Hkv);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.costs = reinterpret_cast<int32_t *>(ws + WL.costs);
    a.items = reinterpret_cast<uint32_t *>(ws + WL.items);
    a.n_layers = n_layers;
    a.rows_per_layer = static_cast<uint32_t>(static_cast<int64_t>(B) * Hkv * a.nB);
    const int64_t rows = static_cast<int64_t>(n_layers) * a.rows_per_layer;
    if (rows * a.npairs >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    a.n_rows = static_cast<uint32_t>(rows);
    a.n_items = static_cast<uint32_t>(rows * a.npairs);
    if (static_cast<int64_t>(n_layers) * (a.nB + 1) + 1 <= kMaxSortBins) {
        a.sort_group = 1;
        a.n_sort_groups = n_layers;
    }
    a.visited = nullptr;
    a.visited_bits = 0;
    bool any_mask = false, v8 = o_str[0] % 16 == 0 && o_str[1] % 16 == 0 && o_str[2] % 16 == 0;
    static thread_local TmapTable<kMaxLayers> tm;   // 24.5 KB: kept off the stack
    for (int l = 0; l < n_layers; ++l) {
        const ea_prefill_layer &ly = layers[l];
        a.m[l] = ly.m;
        a.block_mask[l] = ly.block_mask;
        a.O[l] = static_cast<__nv_bfloat16 *>(ly.O);
        a.LSE[l] = ly.LSE;
        any_mask |= ly.block_mask != nullptr;
        v8 = v8 && (reinterpret_cast<uintptr_t>(ly.O) & 31u) == 0;
        if (!encode_tmap_bf16_4d(&tm.q[l], ly.Q, d, Hq, S, B, q_str, 64, T, true) ||
            !encode_tmap_bf16_4d(&tm.k[l], ly.K, d, Hkv, S, B, kv_str, 64, T / 2, true) ||
            !encode_tmap_bf16_4d(&tm.v[l], ly.V, d, Hkv, S, B, kv_str, 64, T, true) ||
            !encode_tmap_bf16_4d(&tm.o[l], ly.O, d, Hq, S, B, o_str, 64, 32, true))
            return EA_ERR_INVALID_ARG;
    }
    a.mask_elems = any_mask ? static_cast<int64_t>(B) * Hkv * a.nB * a.nB : 0;
    a.o_sb = o_str[0];
    a.o_ss = o_str[1];
    a.o_sh = o_str[2];
    a.o_v8 = v8;
    a.scale_log2 = scale * 1.4426950408889634f;
    if ((s = ensure_attributes()) != EA_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int warps_per_cta = 8;
    plan_costs_kernel<<<static_cast<unsigned>(ceil_div(a.n_rows, warps_per_cta)), warps_per_cta * 32, 0,
                        st>>>(a);
    plan_sort_kernel<<<1, 1024, sizeof(int) * (a.n_sort_groups * (a.nB + 1) + 1), st>>>(a);
    if (cudaGetLastError() != cudaSuccess)
        return EA_ERR_CUDA;
    return launch_attend(tm, a, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free prefill.  Some callers cannot hand the library a workspace:
// an engine whose device memory is owned end to end by its own allocator and
// that forbids allocations after start-up, or a latency-critical path that
// cannot afford cudaMalloc's implicit device synchronisation.  This entry point
// keeps the planner's scratch (work queue and per-block tile counts) in a
// file-scope device array instead, so the caller passes only inputs and
// outputs.  The array is EA_NOALLOC_PREFILL_SCRATCH_BYTES long and lives on
// every device that loads the library until the process exits.
#define EA_NOALLOC_PREFILL_SCRATCH_BYTES (4u << 20)

static __device__ __align__(256) uint8_t g_noalloc_prefill_scratch[EA_NOALLOC_PREFILL_SCRATCH_BYTES];

// Device address of the array, resolved once per process and device (host
// code only sees a host-side stand-in under that name).  A device reset
// (cudaDeviceReset) between calls would leave it stale and is not supported.
static void *g_noalloc_scratch_ptr[64] = {};
static std::mutex g_noalloc_mutex;

extern "C" ea_status ea_hybrid_attn_prefill_noalloc(const void *Q, const void *K, const void *V,
                                                    void *O, float *LSE, const int64_t q_str[4],
                                                    const int64_t kv_str[4],
                                                    const int64_t o_str[4], int B, int S, int Hq,
                                                    int Hkv, int d, float scale, const uint8_t *m,
                                                    int sink, int window,
                                                    const uint8_t *block_mask, int block_size,
                                                    uint32_t *visited_bitmap, void *stream)
{
    const size_t need = ea_prefill_workspace_size(B, S, Hq, Hkv, d);
    if (need == 0)
        return (d != EA_HEAD_DIM || S > EA_MAX_SEQ) ? EA_ERR_UNSUPPORTED : EA_ERR_INVALID_ARG;
    if (need > EA_NOALLOC_PREFILL_SCRATCH_BYTES)
        return EA_ERR_UNSUPPORTED;  // plan would not fit the fixed scratch array
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return EA_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_scratch_ptr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_prefill_scratch) != cudaSuccess || !p)
                return EA_ERR_CUDA;
            g_noalloc_scratch_ptr[dev] = p;
        }
        scratch = g_noalloc_scratch_ptr[dev];
    }
    // Every argument check first, so that a rejected call enqueues nothing.
    const ea_status s = prefill_validate(Q, K, V, O, q_str, kv_str, o_str, B, S, Hq, Hkv, d, scale,
                                         m, sink, window, block_mask, block_size, scratch,
                                         EA_NOALLOC_PREFILL_SCRATCH_BYTES);
    if (s != EA_OK)
        return s;
    // The array keeps the previous call's contents: clear the header (error
    // word and queue counters) before planning.
    if (cudaMemsetAsync(scratch, 0, sizeof(ea_ws_header), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return EA_ERR_CUDA;
    return ea_hybrid_attn_prefill(Q, K, V, O, LSE, q_str, kv_str, o_str, B, S, Hq, Hkv, d, scale,
                                  m, sink, window, block_mask, block_size, scratch,
                                  EA_NOALLOC_PREFILL_SCRATCH_BYTES, visited_bitmap, stream);
}
