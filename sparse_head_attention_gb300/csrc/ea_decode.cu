// ea_decode.cu - one decode step of hybrid-head attention with the routing
// decision fixed at prefill ("Paper Reading - Elastic Attention" (English
// notes), §08 Commentary, stated limit ③: routing is decided once per request,
// at the prefill stage).
//
// A decode step reads every kept cache entry once, so it is bound by HBM
// bandwidth.  The design reads each (b, KV head)'s kept keys exactly once and
// shares every K/V row among the query heads of the GQA group:
//   decode_blocks_kernel (only when a block mask is given): one CTA per
//     unit; for EA_BLOCK units the list of key blocks kept in the mask row of
//     the query's block ((L - 1) / 128), ascending.
//   decode_plan_kernel: per (b, KV head) unit the number of kept keys (FULL:
//     [0, L); SSA: the sink [0, sink) and the window [L - window, L); BLOCK:
//     the kept blocks' keys below L, walked as 64-key tiles), its
//     chunk count (chunks of 2048 to 8192 kept keys, sized so that the step
//     has about four per SM, unless the caller fixes the count), and the list
//     of chunks.  Short SSA units get few chunks, long FA units many, so no
//     CTA is spent on a handful of keys.
//   decode_split_kernel: persistent, one CTA per SM taking chunks from a queue.
//     Each chunk's keys stream through a 6-stage shared-memory ring filled by
//     TMA (64 keys x 256 B per K or V box); the group's query heads share each
//     K/V row; fp32 online softmax per head.  Output: a partial (O / l, LSE)
//     per (chunk, q head).
//   decode_merge_kernel: combines the partials of each (b, q head) by
//     log-sum-exp weights and writes bf16 O and fp32 LSE.
// A paged cache (fixed-size pages of rows, a block table per sequence) runs
// through the same kernels: its tiles are 64-key aligned so that no tile
// straddles two pages (pages hold a multiple of 64 rows), each key of a tile
// is tested against the kept ranges, and the producer looks up each tile's
// page in the block table before issuing its copies.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "ea_device.cuh"
#include "ea_internal.h"

namespace ea {

constexpr int kDecKeys = 64;                           // keys per tile
constexpr int kDecSplitMaxKeys = 512;                  // units up to this many keys: P V in two parts
constexpr int kDecStages = 6;
constexpr int kDecHalfBytes = kDecKeys * 128;          // one 64-dim swizzled box: 8 KB
constexpr int kDecTileBytes = 2 * kDecHalfBytes;       // K or V of one tile: 16 KB
constexpr int kDecWarps = 4;                           // compute warps: 16 keys each per tile
constexpr int kDecThreads = (kDecWarps + 1) * 32;      // + one producer warp
constexpr int kSplitBits = 11;                         // chunk code: unit << 11 | split

struct DecodeArgs {
    const __nv_bfloat16 *q;
    int64_t q_sb, q_sh;
    const int32_t *seqlens;
    const uint8_t *m;
    int32_t *unit_first;
    int32_t *unit_splits;
    int32_t *chunks;
    float *part_o;
    float *part_lse;
    ea_ws_header *hdr;
    __nv_bfloat16 *O;
    int64_t o_sb, o_sh;
    float *LSE;
    int B, Hq, Hkv, g, Lmax, sink, window, num_splits, max_splits, num_sms;
    float scale_log2;
    // block-sparse heads: mask [B][Hkv][nBm][nBm] (NULL when no head may be
    // EA_BLOCK) and, per unit, the kept blocks of its decode row
    const uint8_t *block_mask;
    int nBm;
    int32_t *blk_count;
    uint16_t *blk_list;
    // paged cache (page_size == 0: one contiguous [B][Lmax] cache)
    const int32_t *block_table;
    int64_t bt_stride;
    int page_size, num_pages;
    // a single sequence (B * Hkv <= kSelfPlanUnits): every split CTA plans the
    // step itself and takes chunks blockIdx.x + k * gridDim.x, with no planner
    // launch and no queue
    int self_plan;
};

// Up to this many units a step is planned inside the split kernel.  Measured
// per step against the planner launch: B = 1 x 8 KV heads 36.9 -> 35.3 us; at
// B = 4 and 8 the fixed chunk assignment balances worse than the queue (+1.4 %,
// +4.6 %), so larger batches keep the planner.
constexpr int kSelfPlanUnits = 8;

struct __align__(1024) DecSmem {
    uint8_t k[kDecStages][kDecTileBytes];
    uint8_t v[kDecStages][kDecTileBytes];
    float red_o[kDecWarps][8][EA_HEAD_DIM];
    float red_m[kDecWarps][8];
    float red_l[kDecWarps][8];
    uint64_t full[kDecStages];
    uint64_t empty[kDecStages];
    uint64_t chunk_full[2], chunk_empty[2];
    int chunk[2];  // chunk index handed from the producer to the compute warps (-1: none left)
    int abort;     // set by a timed-out wait; every warp then leaves without further barriers
    int plan_first[kSelfPlanUnits], plan_ns[kSelfPlanUnits], plan_total;   // self-planned steps
};

// Kept keys of one (b, KV head) unit as at most two contiguous ranges:
// visited index v < n0 is key v, v >= n0 is key w0 + (v - n0).  A BLOCK unit
// (blk >= 0 kept blocks) is walked as 64-key tiles instead: two per kept
// block, the last block cut at L (see block_tiles).
struct KeySegs {
    int n;
    int n0;
    int w0;
    int blk;      // kept blocks of a BLOCK unit, -1 otherwise
    int L;
};

__device__ __forceinline__ bool unit_keys(const DecodeArgs &a, int b, int h, KeySegs &ks)
{
    int L = a.seqlens[b];
    const int mode = a.m[b * a.Hkv + h];
    bool ok = true;
    if (L < 0 || L > a.Lmax || mode > EA_BLOCK || (mode == EA_BLOCK && !a.block_mask)) {
        ok = false;
        L = 0;
    }
    ks.L = L;
    ks.blk = -1;
    if (mode == EA_BLOCK && ok) {
        ks.blk = a.blk_count[b * a.Hkv + h];
        ks.n0 = ks.w0 = ks.n = 0;
        return true;
    }
    if (mode == EA_SSA) {
        const int ns = a.sink < L ? a.sink : L;
        const int ws = (L - a.window) > ns ? (L - a.window) : ns;
        ks.n0 = ns;
        ks.w0 = ws;
        ks.n = ns + (L - ws);
    } else {
        ks.n0 = L;
        ks.w0 = L;
        ks.n = L;
    }
    return ok;
}

// Paged cache: the unit's 64-key-aligned tiles are [0, TA) (covering the
// sink) followed by [TB, TL) (covering the window, from the first tile not
// already visited), TL = ceil(L / 64).  Returns the tile count.
__device__ __forceinline__ int paged_tiles(const KeySegs &ks, int &TA, int &TB)
{
    const int L = ks.w0 + (ks.n - ks.n0);
    TA = (ks.n0 + kDecKeys - 1) / kDecKeys;
    const int TL = (L + kDecKeys - 1) / kDecKeys;
    TB = max(ks.w0 / kDecKeys, TA);
    return TA + max(TL - TB, 0);
}

// 64-key tiles of a BLOCK unit: two per kept block, except that the query's
// own block (kept or not, the last one listed when kept) only reaches L.
__device__ __forceinline__ int block_tiles(const DecodeArgs &a, int u, const KeySegs &ks)
{
    if (ks.blk <= 0)
        return 0;
    const int last = a.blk_list[static_cast<int64_t>(u) * a.nBm + ks.blk - 1];
    const int tail = ks.L - last * EA_TILE;          // keys of the last block below L
    return 2 * (ks.blk - 1) + (tail >= EA_TILE ? 2 : (tail + kDecKeys - 1) / kDecKeys);
}

// Kept keys of a unit as the split kernel walks them (whole tiles for a paged
// cache or a BLOCK unit).
__device__ __forceinline__ int unit_work(const DecodeArgs &a, int u, bool &ok)
{
    KeySegs ks;
    ok = unit_keys(a, u / a.Hkv, u % a.Hkv, ks);
    if (ks.blk >= 0)
        return block_tiles(a, u, ks) * kDecKeys;
    int TA, TB;
    return a.page_size ? paged_tiles(ks, TA, TB) * kDecKeys : ks.n;
}

// One CTA per unit: the key blocks kept in the unit's decode row of the block
// mask (row (L - 1) / 128, blocks 0 .. (L - 1) / 128), ascending.  Each pass
// covers 1024 blocks: thread t tests blocks 4t .. 4t + 3 (independent loads),
// and a block-wide exclusive scan of the counts places them.
constexpr int kBlkThreads = 256;

__global__ void __launch_bounds__(kBlkThreads) decode_blocks_kernel(DecodeArgs a)
{
    __shared__ int warp_tot[kBlkThreads / 32];
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int b = u / a.Hkv, h = u % a.Hkv;
    const int L = a.seqlens[b];
    int count = 0;
    if (a.m[u] == EA_BLOCK && L > 0 && L <= a.Lmax) {
        const int qb = (L - 1) / EA_TILE;
        const uint8_t *row = a.block_mask + ((static_cast<int64_t>(b) * a.Hkv + h) * a.nBm + qb) * a.nBm;
        uint16_t *list = a.blk_list + static_cast<int64_t>(u) * a.nBm;
        for (int k0 = 0; k0 <= qb; k0 += 4 * kBlkThreads) {
            uint32_t bits = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kb = k0 + 4 * tid + j;
                bits |= (kb <= qb && in_bounds(kb, a.nBm, &a.hdr->error) && row[kb] != 0) ? (1u << j)
                                                                                         : 0u;
            }
            const int mine = __popc(bits);
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (lane == 31)
                warp_tot[warp] = incl;
            __syncthreads();
            int before = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kBlkThreads / 32; ++w) {
                before += w < warp ? warp_tot[w] : 0;
                total += warp_tot[w];
            }
            int pos = count + before + incl - mine;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (((bits >> j) & 1u) && in_bounds(pos, a.nBm, &a.hdr->error))
                    list[pos++] = static_cast<uint16_t>(k0 + 4 * tid + j);
            count += total;
            __syncthreads();   // warp_tot is rewritten by the next pass
        }
    }
    if (tid == 0)
        a.blk_count[u] = count;
}

// One CTA: per-unit chunk counts, their prefix sum, and the chunk list.  The
// automatic chunk size aims at about four chunks per SM over the whole step
// (fewer, longer chunks mean fewer partial results to write and merge), between
// EA_DECODE_AUTO_CHUNK and EA_DECODE_MAX_CHUNK kept keys, so that a small
// batch still spreads over every SM.
constexpr int kPlanThreads = 256;

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(DecodeArgs a)
{
    __shared__ long long red_work[kPlanThreads / 32];
    __shared__ int red_chunks[kPlanThreads / 32];
    griddep_launch_dependents();   // the split kernel may start its prologue
    const int units = a.B * a.Hkv;
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int per = (units + kPlanThreads - 1) / kPlanThreads;
    const int lo = min(tid * per, units), hi = min(lo + per, units);
    // each unit's work, kept in unit_splits until its split count replaces it
    long long mine = 0;
    bool bad = false;
    for (int u = lo; u < hi; ++u) {
        bool ok;
        const int work = unit_work(a, u, ok);
        bad |= !ok;
        a.unit_splits[u] = work;
        mine += work;
    }
    if (bad)
        raise_error(&a.hdr->error, EA_DEVERR_CHECK);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mine += __shfl_down_sync(0xffffffffu, mine, o);
    if (lane == 0)
        red_work[warp] = mine;
    __syncthreads();
    long long total_work = 0;
#pragma unroll
    for (int w = 0; w < kPlanThreads / 32; ++w)
        total_work += red_work[w];
    const long long target = 4ll * (a.num_sms > 0 ? a.num_sms : 1);
    long long chunk = (total_work + target - 1) / target;
    chunk = chunk < EA_DECODE_AUTO_CHUNK ? EA_DECODE_AUTO_CHUNK
                                         : (chunk > EA_DECODE_MAX_CHUNK ? EA_DECODE_MAX_CHUNK : chunk);
    int local = 0;
    for (int u = lo; u < hi; ++u) {
        const int work = a.unit_splits[u];
        int ns = a.num_splits > 0 ? a.num_splits : static_cast<int>((work + chunk - 1) / chunk);
        ns = ns < 1 ? 1 : (ns > a.max_splits ? a.max_splits : ns);
        a.unit_splits[u] = ns;
        local += ns;
    }
    // exclusive scan of the per-thread chunk counts: lanes, then warps
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        red_chunks[warp] = incl;
    __syncthreads();
    int base = 0, grand = 0;
#pragma unroll
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        base += w < warp ? red_chunks[w] : 0;
        grand += red_chunks[w];
    }
    int run = base + incl - local;
    for (int u = lo; u < hi; ++u) {
        a.unit_first[u] = run;
        const int ns = a.unit_splits[u];
        for (int sp = 0; sp < ns; ++sp)
            if (in_bounds(static_cast<int64_t>(run) + sp,
                          static_cast<int64_t>(units) * a.max_splits, &a.hdr->error))
                a.chunks[run + sp] = (u << kSplitBits) | sp;
        run += ns;
    }
    if (tid == 0) {
        a.hdr->n_items = static_cast<uint32_t>(grand);
        a.hdr->work_counter = 0;   // the split kernel's chunk queue
    }
}

// Position of chunk c in the key stream.  Contiguous cache: visited keys
// [v_begin, v_end) in tiles that start at any key.  Paged cache: the unit's
// aligned tiles [v_begin, v_end) (tile indices), tile v at key
// 64 * (v < TA ? v : TB + v - TA).  BLOCK unit (either cache): aligned tiles
// [v_begin, v_end), tile v at key 128 * list[v / 2] + 64 * (v % 2).
struct ChunkInfo {
    int b, h, v_begin, v_end;
    int kept;                 // the unit's kept keys (whole tiles of a BLOCK unit)
    KeySegs ks;
    int a_tiles, b_begin, n_tiles;
    int TA, TB;
    const uint16_t *list;     // BLOCK unit: its kept blocks (NULL otherwise)
};

__device__ __forceinline__ ChunkInfo chunk_info(const DecodeArgs &a, int c, const DecSmem &sm)
{
    ChunkInfo ci;
    int u, sp, ns;
    if (a.self_plan) {
        // the last unit whose first chunk is <= c (every unit has one chunk at least)
        int lo = 0, hi = a.B * a.Hkv - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.plan_first[mid] <= c)
                lo = mid;
            else
                hi = mid - 1;
        }
        u = lo;
        sp = c - sm.plan_first[u];
        ns = sm.plan_ns[u];
    } else {
        const int code = a.chunks[c];
        u = code >> kSplitBits;
        sp = code & ((1 << kSplitBits) - 1);
        ns = a.unit_splits[u];
    }
    ci.b = u / a.Hkv;
    ci.h = u % a.Hkv;
    unit_keys(a, ci.b, ci.h, ci.ks);
    ci.list = nullptr;
    ci.kept = ci.ks.n;
    if (ci.ks.blk >= 0) {
        ci.list = a.blk_list + static_cast<int64_t>(u) * a.nBm;
        const int nt = block_tiles(a, u, ci.ks);
        ci.kept = nt * kDecKeys;
        const int len = (nt + ns - 1) / ns;
        ci.v_begin = min(sp * len, nt);
        ci.v_end = min(ci.v_begin + len, nt);
        ci.n_tiles = ci.v_end - ci.v_begin;
        ci.a_tiles = ci.b_begin = ci.TA = ci.TB = 0;
        return ci;
    }
    if (a.page_size) {
        const int nt = paged_tiles(ci.ks, ci.TA, ci.TB);
        const int len = (nt + ns - 1) / ns;
        ci.v_begin = min(sp * len, nt);
        ci.v_end = min(ci.v_begin + len, nt);
        ci.n_tiles = ci.v_end - ci.v_begin;
        ci.a_tiles = 0;
        ci.b_begin = 0;
        return ci;
    }
    ci.TA = ci.TB = 0;
    const int len = (ci.ks.n + ns - 1) / ns;
    ci.v_begin = min(sp * len, ci.ks.n);
    ci.v_end = min(ci.v_begin + len, ci.ks.n);
    const int a_end = min(ci.v_end, ci.ks.n0);
    ci.a_tiles = ci.v_begin < a_end ? (a_end - ci.v_begin + kDecKeys - 1) / kDecKeys : 0;
    ci.b_begin = max(ci.v_begin, ci.ks.n0);
    ci.n_tiles = ci.a_tiles + (ci.b_begin < ci.v_end ? (ci.v_end - ci.b_begin + kDecKeys - 1) / kDecKeys : 0);
    return ci;
}

// First key and number of leading keys that may be valid of tile t of a chunk
// (contiguous cache: a tile never straddles the sink and window ranges, and
// all nvalid keys are kept; paged cache: an aligned tile of 64 keys, each
// tested against the kept ranges by the caller).
__device__ __forceinline__ void tile_rows(const DecodeArgs &a, const ChunkInfo &ci, int t,
                                          int &key0, int &nvalid)
{
    if (ci.list) {
        const int v = ci.v_begin + t;
        key0 = EA_TILE * ci.list[v >> 1] + kDecKeys * (v & 1);
        nvalid = min(kDecKeys, ci.ks.L - key0);
        return;
    }
    if (a.page_size) {
        const int v = ci.v_begin + t;
        key0 = kDecKeys * (v < ci.TA ? v : ci.TB + (v - ci.TA));
        nvalid = kDecKeys;
        return;
    }
    if (t < ci.a_tiles) {
        const int v = ci.v_begin + t * kDecKeys;
        key0 = v;
        nvalid = min(kDecKeys, min(ci.v_end, ci.ks.n0) - v);
    } else {
        const int v = ci.b_begin + (t - ci.a_tiles) * kDecKeys;
        key0 = ci.ks.w0 + (v - ci.ks.n0);
        nvalid = min(kDecKeys, ci.v_end - v);
    }
}

// ---------------------------------------------------------------- mma.sync
// m16n8k16 bf16 -> fp32.  Fragment layouts (lane = 4 * row_in_group + quad):
//   A 16x16: a0 = (r, 2q..2q+1), a1 = (r + 8, ..), a2 = (r, 2q + 8..), a3 = (r + 8, 2q + 8..)
//   B 16x8 : b0 = (k = 2q..2q+1, n = r), b1 = (k = 2q + 8.., n = r)
//   C 16x8 : c0, c1 = (r, 2q..2q+1), c2, c3 = (r + 8, ..)
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Barrier over the compute warps only (named barrier 1).
__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
}

// Byte offset of the 16-byte chunk holding (row, 8-element column block cb)
// of a [64 rows][128 dims] tile stored as two 128-byte-swizzled 64-dim boxes.
__device__ __forceinline__ uint32_t sw_off(int row, int cb)
{
    return (cb >> 3) * kDecHalfBytes + row * 128 + (((cb & 7) ^ (row & 7)) << 4);
}

// A self-planned step (B * Hkv <= kSelfPlanUnits): warp 0 of every split CTA
// computes the plan decode_plan_kernel would (the same chunk size, split
// counts and chunk order, unit by unit), lane l taking units 2l and 2l + 1, into
// shared memory; CTA 0 also stores each unit's first chunk and split count for
// the merge kernel.
__device__ __forceinline__ void self_plan(const DecodeArgs &a, DecSmem &sm, int lane)
{
    const int units = a.B * a.Hkv;
    int w[2] = {0, 0};
    bool bad = false;
    long long mine = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int u = 2 * lane + k;
        if (u < units) {
            bool ok;
            w[k] = unit_work(a, u, ok);
            bad |= !ok;
            mine += w[k];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mine += __shfl_xor_sync(0xffffffffu, mine, o);
    const long long target = 4ll * (a.num_sms > 0 ? a.num_sms : 1);
    long long chunk = (mine + target - 1) / target;
    chunk = chunk < EA_DECODE_AUTO_CHUNK ? EA_DECODE_AUTO_CHUNK
                                         : (chunk > EA_DECODE_MAX_CHUNK ? EA_DECODE_MAX_CHUNK : chunk);
    int ns[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 2; ++k)
        if (2 * lane + k < units) {
            int n = a.num_splits > 0 ? a.num_splits : static_cast<int>((w[k] + chunk - 1) / chunk);
            ns[k] = n < 1 ? 1 : (n > a.max_splits ? a.max_splits : n);
        }
    const int local = ns[0] + ns[1];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    int first = incl - local;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int u = 2 * lane + k;
        if (u < units) {
            sm.plan_first[u] = first;
            sm.plan_ns[u] = ns[k];
            if (blockIdx.x == 0) {
                a.unit_first[u] = first;
                a.unit_splits[u] = ns[k];
            }
        }
        first += ns[k];
    }
    if (lane == 31)
        sm.plan_total = incl;
    if (bad && blockIdx.x == 0)
        raise_error(&a.hdr->error, EA_DEVERR_CHECK);
}

// Persistent: each CTA takes chunks from a queue (an atomic counter that the
// planner resets), so CTAs that drew short chunks take more of them.
// Warp w (of 4) owns keys [16w, 16w + 16) of every 64-key tile; the query
// heads of the GQA group are the rows of the MMA (padded to 16 with zeros):
//   S (16 x 16 keys) = Q K^T : 2 key blocks x 8 head-dim steps
//   O (16 x 128)    += P V   : P straight from the S fragments, 16 dim blocks
// The producer warp keeps kDecStages tiles in flight across chunk boundaries;
// each compute warp releases a stage through its arrival on `empty`.
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    DecSmem &sm = *reinterpret_cast<DecSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int r = lane >> 2, qd = lane & 3;   // fragment row / quad position
    const float NEG_INF = -__int_as_float(0x7f800000);
    volatile int *abort = &sm.abort;

    if (tid == 0) {
        sm.abort = 0;
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kDecWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.chunk_full[s], 1);
            mbar_init(&sm.chunk_empty[s], kDecWarps);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (a.self_plan) {
        if (warp == 0)
            self_plan(a, sm, lane);
        __syncthreads();
    }
    // The chunk list comes from the planner launched just before (a self-planned
    // step is launched without overlap); every CTA is resident (one per SM)
    // before the merge kernel may be scheduled.
    griddep_wait();
    griddep_launch_dependents();
    const int total = a.self_plan ? sm.plan_total : static_cast<int>(a.hdr->n_items);

    if (warp == kDecWarps) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the tile sequence (converged waits); lane 0
        // issues the copies.  It takes part in no block-wide barrier: the
        // compute warps synchronise among themselves with a named barrier.
        // Paged cache: lane j holds the page of the chunk's tile 32 * k + j,
        // looked up a group of 32 tiles ahead of the copies that need it.
        uint32_t issued = 0;
        for (int it = 0;; ++it) {
            // next chunk from the queue, handed to the compute warps in slot it % 2
            const int slot = it & 1;
            if (!mbar_wait(&sm.chunk_empty[slot], ((it >> 1) & 1) ^ 1, abort, &a.hdr->error))
                return;
            int c = -1;
            if (lane == 0) {
                const uint32_t x = a.self_plan ? blockIdx.x + static_cast<uint32_t>(it) * gridDim.x
                                               : atomicAdd(&a.hdr->work_counter, 1u);
                c = x < static_cast<uint32_t>(total) ? static_cast<int>(x) : -1;
                sm.chunk[slot] = c;
                mbar_arrive(&sm.chunk_full[slot]);
            }
            c = __shfl_sync(0xffffffffu, c, 0);
            if (c < 0)
                break;
            const ChunkInfo ci = chunk_info(a, c, sm);
            int my_page = 0;
            for (int t = 0; t < ci.n_tiles; ++t) {
                if (a.page_size && (t & 31) == 0) {
                    my_page = 0;
                    if (t + lane < ci.n_tiles) {
                        int k0, nv;
                        tile_rows(a, ci, t + lane, k0, nv);
                        if (in_bounds(k0 / a.page_size, a.Lmax / a.page_size, &a.hdr->error))
                            my_page = a.block_table[ci.b * a.bt_stride + k0 / a.page_size];
                    }
                }
                const int page = a.page_size ? __shfl_sync(0xffffffffu, my_page, t & 31) : 0;
                const int s = issued % kDecStages;
                if (!mbar_wait(&sm.empty[s], ((issued / kDecStages) & 1) ^ 1, abort, &a.hdr->error))
                    return;
                if (lane == 0) {
                    int key0, nv;
                    tile_rows(a, ci, t, key0, nv);
                    int row = key0, outer = ci.b;
                    if (a.page_size) {
                        // a page outside the cache is reported; its copy reads
                        // the fill value (a box outside the tensor is zero-filled)
                        if (page < 0 || page >= a.num_pages)
                            raise_error(&a.hdr->error, EA_DEVERR_CHECK);
                        row = key0 % a.page_size;
                        outer = page;
                    }
                    mbar_arrive_expect_tx(&sm.full[s], 2 * kDecTileBytes);
                    tma_load_4d(sm.k[s], &tm_k, 0, ci.h, row, outer, &sm.full[s]);
                    tma_load_4d(sm.k[s] + kDecHalfBytes, &tm_k, 64, ci.h, row, outer, &sm.full[s]);
                    tma_load_4d(sm.v[s], &tm_v, 0, ci.h, row, outer, &sm.full[s]);
                    tma_load_4d(sm.v[s] + kDecHalfBytes, &tm_v, 64, ci.h, row, outer, &sm.full[s]);
                }
                __syncwarp();
                ++issued;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- compute
    uint32_t consumed = 0;
    for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&sm.chunk_full[slot], (it >> 1) & 1, abort, &a.hdr->error))
            return;
        const int c = sm.chunk[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.chunk_empty[slot]);
        if (c < 0)
            break;
        const ChunkInfo ci = chunk_info(a, c, sm);
        // A unit that keeps few keys takes P V in two bf16 parts: with a handful
        // of keys one probability's 2^-9 rounding error would reach O undiluted.
        const bool split = ci.kept <= kDecSplitMaxKeys;
        // Q as the A operand: rows r < g are query heads, the rest zero
        uint32_t qa[8][2];   // per head-dim step j: (r, 16j + 2q..), (r, 16j + 8 + 2q..)
        {
            const bool real = r < a.g;
            const __nv_bfloat16 *qrow = a.q + ci.b * a.q_sb + (ci.h * a.g + (real ? r : 0)) * a.q_sh;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t *p0 = reinterpret_cast<const uint32_t *>(qrow + 16 * j + 2 * qd);
                const uint32_t *p1 = reinterpret_cast<const uint32_t *>(qrow + 16 * j + 8 + 2 * qd);
                qa[j][0] = real ? *p0 : 0u;
                qa[j][1] = real ? *p1 : 0u;
            }
        }
        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[n][e] = 0.f;
        float m_run = NEG_INF, l_part = 0.f;   // row r statistics (l summed over the quad at the end)

        // the tile loop, compiled twice: with P's remainder (rare units) and without
        auto tiles = [&](auto split_tag) -> bool {
            constexpr bool kSplit = decltype(split_tag)::value;
            for (int t = 0; t < ci.n_tiles; ++t) {
                const int s = consumed % kDecStages;
                if (!mbar_wait(&sm.full[s], (consumed / kDecStages) & 1, abort, &a.hdr->error))
                    return false;  // timed out (error word set) or another warp did
                ++consumed;
                int key0, nv;
                tile_rows(a, ci, t, key0, nv);
                const uint32_t kb = smem_u32(sm.k[s]), vb = smem_u32(sm.v[s]);
                const int kw = warp * 16;   // this warp's first key in the tile

                // S = Q K^T for keys kw..kw+15 (two 8-key blocks)
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int krow = kw + (lane >> 4) * 8 + (lane & 7);   // key this lane addresses
                    const int csel = (lane >> 3) & 1;                      // 0: first 8 dims, 1: next 8
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t b00, b01, b10, b11;
                        ldsm_x4(kb + sw_off(krow, 2 * j + csel), b00, b01, b10, b11);
                        mma_bf16(sc[0], qa[j][0], 0u, qa[j][1], 0u, b00, b01);
                        mma_bf16(sc[1], qa[j][0], 0u, qa[j][1], 0u, b10, b11);
                    }
                }
                // online softmax over this warp's 16 keys, row r
                float x[4] = {sc[0][0] * a.scale_log2, sc[0][1] * a.scale_log2,
                              sc[1][0] * a.scale_log2, sc[1][1] * a.scale_log2};
                const int kcol[4] = {kw + 2 * qd, kw + 2 * qd + 1, kw + 8 + 2 * qd, kw + 9 + 2 * qd};
                if (a.page_size && !ci.list) {
                    // aligned tile: keep key k iff (k < sink end or k >= window
                    // start) and k < L
                    const int L = ci.ks.w0 + (ci.ks.n - ci.ks.n0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = key0 + kcol[e];
                        if (!((k < ci.ks.n0 || k >= ci.ks.w0) && k < L))
                            x[e] = NEG_INF;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (kcol[e] >= nv)
                            x[e] = NEG_INF;
                }
                float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run, mx);
                if (m_new > m_run) {
                    const float f = m_run == NEG_INF ? 0.f : ex2(m_run - m_new);
                    l_part *= f;
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        o[n][0] *= f;
                        o[n][1] *= f;
                    }
                    m_run = m_new;
                }
                const float mb = m_run == NEG_INF ? 0.f : m_run;
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    p[e] = ex2(x[e] - mb);
                    l_part += p[e];
                }
                const uint32_t pa0 = pack_bf16x2(p[0], p[1]);   // (r, keys 2q..)
                const uint32_t pa2 = pack_bf16x2(p[2], p[3]);   // (r, keys 8 + 2q..)
                uint32_t pr0 = 0u, pr2 = 0u;                     // P - bf16(P), rounded to bf16
                if constexpr (kSplit) {
                    pr0 = pack_bf16x2(p[0] - __uint_as_float(pa0 << 16), p[1] - __uint_as_float(pa0 & 0xffff0000u));
                    pr2 = pack_bf16x2(p[2] - __uint_as_float(pa2 << 16), p[3] - __uint_as_float(pa2 & 0xffff0000u));
                }

                // O += P V: 16 head-dim blocks of 8, two per ldmatrix
                {
                    const int vrow = kw + ((lane >> 3) & 1) * 8 + (lane & 7);
                    const int cadd = lane >> 4;
#pragma unroll
                    for (int n = 0; n < 16; n += 2) {
                        uint32_t b00, b01, b10, b11;
                        ldsm_x4_t(vb + sw_off(vrow, n + cadd), b00, b01, b10, b11);
                        mma_bf16(o[n], pa0, 0u, pa2, 0u, b00, b01);
                        mma_bf16(o[n + 1], pa0, 0u, pa2, 0u, b10, b11);
                        if constexpr (kSplit) {
                            mma_bf16(o[n], pr0, 0u, pr2, 0u, b00, b01);
                            mma_bf16(o[n + 1], pr0, 0u, pr2, 0u, b10, b11);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm.empty[s]);
            }
            return true;
        };
        if (!(split ? tiles(std::true_type{}) : tiles(std::false_type{})))
            return;

        // per-warp results of the rows r < g -> shared memory, then merge warps
        l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
        l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
        if (r < a.g) {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                sm.red_o[warp][r][8 * n + 2 * qd] = o[n][0];
                sm.red_o[warp][r][8 * n + 2 * qd + 1] = o[n][1];
            }
            if (qd == 0) {
                sm.red_m[warp][r] = m_run;
                sm.red_l[warp][r] = l_part;
            }
        }
        if (*abort)
            return;
        compute_sync();
        for (int idx = tid; idx < a.g * EA_HEAD_DIM; idx += kDecWarps * 32) {
            const int hh = idx / EA_HEAD_DIM, dd = idx % EA_HEAD_DIM;
            float M = NEG_INF;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w)
                M = fmaxf(M, sm.red_m[w][hh]);
            float lsum = 0.f, osum = 0.f;
            if (M > NEG_INF)
#pragma unroll
                for (int w = 0; w < kDecWarps; ++w) {
                    const float f = ex2(sm.red_m[w][hh] - M);
                    lsum += sm.red_l[w][hh] * f;
                    osum += sm.red_o[w][hh][dd] * f;
                }
            const int64_t pidx = static_cast<int64_t>(c) * a.g + hh;
            if (!in_bounds(pidx, static_cast<int64_t>(a.B) * a.Hkv * a.max_splits * a.g,
                           &a.hdr->error))
                continue;
            a.part_o[pidx * EA_HEAD_DIM + dd] = lsum > 0.f ? osum / lsum : 0.f;
            if (dd == 0)
                a.part_lse[pidx] = lsum > 0.f ? (M + __log2f(lsum)) * 0.69314718055994531f : NEG_INF;
        }
        if (*abort)
            return;
        compute_sync();  // the reduction buffers are reused by the next chunk
    }
}

// One CTA per (q head, b): log-sum-exp merge of the unit's chunks.  Four
// groups of 128 threads (one thread per head dimension) each take a quarter of
// the chunks in one pass: a batch of partial LSEs and outputs is loaded at
// once, the running maximum moves to the batch's maximum (one rescale per
// batch) and the batch's weights exp(lse - max) are added to the running sum
// and the weighted output.  The four groups' states are combined in a fixed
// order.  (A separate pass for the maximum would put one more round trip to
// memory on this short kernel's path.)
constexpr int kMergeGroups = 4;

template <int K>
__device__ __forceinline__ void merge_batch(const float (&l)[K], const float (&o)[K], float &m,
                                            float &w, float &osum)
{
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float LOG2E = 1.4426950408889634f;
    float mb = l[0];
#pragma unroll
    for (int k = 1; k < K; ++k)
        mb = fmaxf(mb, l[k]);
    if (mb == NEG_INF)
        return;                       // no kept key in any of these chunks
    if (mb > m) {
        if (m > NEG_INF) {
            const float f = ex2((m - mb) * LOG2E);
            w *= f;
            osum *= f;
        }
        m = mb;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float e = ex2((l[k] - m) * LOG2E);   // 0 for an empty chunk (lse = -inf, o = 0)
        w += e;
        osum += e * o[k];
    }
}

// (two CTAs per SM: a large batch has thousands of these short CTAs)
__global__ void __launch_bounds__(kMergeGroups * EA_HEAD_DIM, 2) decode_merge_kernel(const DecodeArgs a)
{
    __shared__ float gm[kMergeGroups], gw[kMergeGroups];
    __shared__ float go[kMergeGroups][EA_HEAD_DIM];
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float LOG2E = 1.4426950408889634f;
    const int qh = blockIdx.x, b = blockIdx.y;
    const int dd = threadIdx.x % EA_HEAD_DIM, grp = threadIdx.x / EA_HEAD_DIM;
    griddep_wait();   // the partials of the split kernel launched just before
    const int u = b * a.Hkv + qh / a.g, hh = qh % a.g;
    const int first = a.unit_first[u];
    int ns = a.unit_splits[u];
    if (!in_bounds(static_cast<int64_t>(first) + ns - 1,
                   static_cast<int64_t>(a.B) * a.Hkv * a.max_splits, &a.hdr->error))
        ns = 0;
    const int64_t base = static_cast<int64_t>(first) * a.g + hh;
    const int groups = blockDim.x / EA_HEAD_DIM;   // 1 for many (b, head) rows, else kMergeGroups
    const int per = (ns + groups - 1) / groups;
    const int s0 = min(grp * per, ns), s1 = min(s0 + per, ns);
    float m = NEG_INF, w = 0.f, osum = 0.f;
    int s = s0;
    for (; s + 8 <= s1; s += 8) {
        float l[8], o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t pidx = base + static_cast<int64_t>(s + k) * a.g;
            l[k] = a.part_lse[pidx];
            o[k] = a.part_o[pidx * EA_HEAD_DIM + dd];
        }
        merge_batch(l, o, m, w, osum);
    }
    for (; s + 4 <= s1; s += 4) {
        float l[4], o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t pidx = base + static_cast<int64_t>(s + k) * a.g;
            l[k] = a.part_lse[pidx];
            o[k] = a.part_o[pidx * EA_HEAD_DIM + dd];
        }
        merge_batch(l, o, m, w, osum);
    }
    for (; s < s1; ++s) {
        const int64_t pidx = base + static_cast<int64_t>(s) * a.g;
        const float l[1] = {a.part_lse[pidx]}, o[1] = {a.part_o[pidx * EA_HEAD_DIM + dd]};
        merge_batch(l, o, m, w, osum);
    }
    if (dd == 0) {
        gm[grp] = m;
        gw[grp] = w;
    }
    go[grp][dd] = osum;
    __syncthreads();
    if (grp == 0) {
        float M = NEG_INF;
#pragma unroll
        for (int k = 0; k < kMergeGroups; ++k)
            if (k < groups)
                M = fmaxf(M, gm[k]);
        float wsum = 0.f, o = 0.f;
        if (M > NEG_INF)
#pragma unroll
            for (int k = 0; k < kMergeGroups; ++k)
                if (k < groups && gm[k] > NEG_INF) {
                    const float f = ex2((gm[k] - M) * LOG2E);
                    wsum += gw[k] * f;
                    o += go[k][dd] * f;
                }
        a.O[b * a.o_sb + qh * a.o_sh + dd] = __float2bfloat16_rn(wsum > 0.f ? o / wsum : 0.f);
        if (dd == 0 && a.LSE)
            a.LSE[static_cast<int64_t>(b) * a.Hq + qh] = wsum > 0.f ? M + __logf(wsum) : NEG_INF;
    }
}

static cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                                 int grid, cudaStream_t st, bool overlap)
{
    const size_t smem = sizeof(DecSmem) + 1024;
    static bool attr_done[64] = {};   // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_split_kernel, tk, tv, a);
}

// The merge kernel, launched so that its CTAs may be scheduled while the split
// kernel finishes (it waits for the split kernel before reading anything).
// With more (b, head) rows than two per SM, one group of 128 threads per row
// (the rows fill the GPU, and a row's chunks are few); otherwise four groups
// share a row's chunks.
static cudaError_t launch_merge(const DecodeArgs &a, int Hq, int B, cudaStream_t st)
{
    const int groups = static_cast<int64_t>(B) * Hq >= 2ll * a.num_sms ? 1 : kMergeGroups;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(Hq, B);
    cfg.blockDim = dim3(groups * EA_HEAD_DIM);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
}

} // namespace ea

using namespace ea;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared by the contiguous and the paged entry points.  Contiguous: Kc/Vc
// [B][Lmax][Hkv][d] with strides kv_str; paged (page_size > 0): Kc/Vc
// [num_pages][page_size][Hkv][d], Lmax = max_pages * page_size.
static ea_status decode_launch(const void *q, const void *Kc, const void *Vc, void *O, float *LSE,
                               const int64_t q_str[3], const int64_t kv_str[4],
                               const int64_t o_str[3], const int32_t *seqlens, int B, int Hq,
                               int Hkv, int d, int Lmax, float scale, const uint8_t *m, int sink,
                               int window, const uint8_t *block_mask, int block_size,
                               int num_splits, void *workspace, size_t ws_bytes,
                               const int32_t *block_table, int64_t bt_stride, int page_size,
                               int num_pages, void *stream)
{
    if (!q || !Kc || !Vc || !O || !q_str || !kv_str || !o_str || !seqlens || !m)
        return EA_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lmax < 1 || sink < 0 || window < 1 ||
        !(scale > 0.f) || num_splits < 0 || num_splits > 1024 || block_size != EA_TILE)
        return EA_ERR_INVALID_ARG;
    const int64_t nBm = ceil_div(Lmax, EA_TILE);
    if (block_mask && nBm > 65535)
        return EA_ERR_UNSUPPORTED;
    if (d != EA_HEAD_DIM || Hq / Hkv > 8 || B > 65535 || Hkv > 65535)
        return EA_ERR_UNSUPPORTED;
    if (q_str[2] != 1 || kv_str[3] != 1 || o_str[2] != 1)
        return EA_ERR_INVALID_ARG;
    if (q_str[0] <= 0 || q_str[1] <= 0 || o_str[0] <= 0 || o_str[1] <= 0 || q_str[0] % 8 ||
        q_str[1] % 8)
        return EA_ERR_INVALID_ARG;
    for (int k = 0; k < 3; ++k)
        if (kv_str[k] <= 0 || kv_str[k] % 8)
            return EA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(O))
        return EA_ERR_INVALID_ARG;
    const int max_splits = decode_max_splits(Lmax, num_splits);
    if (static_cast<int64_t>(B) * Hkv >= (int64_t(1) << (31 - kSplitBits)) ||
        static_cast<int64_t>(B) * Hkv * max_splits >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    const DecodeWs L = decode_ws_layout(B, Hq, Hkv, max_splits, Lmax);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < L.total)
        return EA_ERR_WORKSPACE;

    alignas(64) CUtensorMap tk, tv;
    const int rows = page_size ? page_size : Lmax;
    const int outer = page_size ? num_pages : B;
    if (!encode_tmap_bf16_4d(&tk, Kc, d, Hkv, rows, outer, kv_str, 64, kDecKeys, true) ||
        !encode_tmap_bf16_4d(&tv, Vc, d, Hkv, rows, outer, kv_str, 64, kDecKeys, true))
        return EA_ERR_INVALID_ARG;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    DecodeArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.q_sb = q_str[0];
    a.q_sh = q_str[1];
    a.seqlens = seqlens;
    a.m = m;
    a.unit_first = reinterpret_cast<int32_t *>(ws + L.unit_first);
    a.unit_splits = reinterpret_cast<int32_t *>(ws + L.unit_splits);
    a.chunks = reinterpret_cast<int32_t *>(ws + L.chunks);
    a.part_o = reinterpret_cast<float *>(ws + L.partial_o);
    a.part_lse = reinterpret_cast<float *>(ws + L.partial_lse);
    a.hdr = reinterpret_cast<ea_ws_header *>(ws);
    a.O = static_cast<__nv_bfloat16 *>(O);
    a.o_sb = o_str[0];
    a.o_sh = o_str[1];
    a.LSE = LSE;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = Hq / Hkv;
    a.Lmax = Lmax;
    a.sink = sink < Lmax ? sink : Lmax;
    a.window = window < Lmax ? window : Lmax;
    a.num_splits = num_splits;
    a.max_splits = max_splits;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_sms = 0;   // set below
    a.block_mask = block_mask;
    a.nBm = static_cast<int>(nBm);
    a.blk_count = reinterpret_cast<int32_t *>(ws + L.blk_count);
    a.blk_list = reinterpret_cast<uint16_t *>(ws + L.blk_list);
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.page_size = page_size;
    a.num_pages = num_pages;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return EA_ERR_CUDA;
    const int sms = num_sms(dev);
    if (sms <= 0)
        return EA_ERR_CUDA;
    a.num_sms = sms;
    const int64_t max_chunks = static_cast<int64_t>(B) * Hkv * max_splits;
    const int grid = static_cast<int>(max_chunks < sms ? max_chunks : sms);
    // Small batches plan inside the split kernel: no planner launch on their
    // short critical path.  That launch then may not overlap its predecessor
    // (the previous step's merge still reads the partials it overwrites).
    a.self_plan = static_cast<int64_t>(B) * Hkv <= kSelfPlanUnits ? 1 : 0;
    if (block_mask)
        decode_blocks_kernel<<<static_cast<unsigned>(static_cast<int64_t>(B) * Hkv), kBlkThreads, 0, st>>>(a);
    if (!a.self_plan)
        decode_plan_kernel<<<1, kPlanThreads, 0, st>>>(a);
    const cudaError_t e = launch_decode(tk, tv, a, grid, st, !a.self_plan);
    if (e != cudaSuccess)
        return EA_ERR_CUDA;
    if (launch_merge(a, Hq, B, st) != cudaSuccess)
        return EA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}

extern "C" ea_status ea_hybrid_attn_decode(const void *q, const void *Kc, const void *Vc, void *O,
                                           float *LSE, const int64_t q_str[3],
                                           const int64_t kv_str[4], const int64_t o_str[3],
                                           const int32_t *seqlens, int B, int Hq, int Hkv, int d,
                                           int Lmax, float scale, const uint8_t *m, int sink,
                                           int window, const uint8_t *block_mask, int block_size,
                                           int num_splits, void *workspace, size_t ws_bytes,
                                           void *stream)
{
    return decode_launch(q, Kc, Vc, O, LSE, q_str, kv_str, o_str, seqlens, B, Hq, Hkv, d, Lmax,
                         scale, m, sink, window, block_mask, block_size, num_splits, workspace,
                         ws_bytes, nullptr, 0, 0, 0, stream);
}

extern "C" ea_status ea_hybrid_attn_decode_paged(const void *q, const void *K_pages,
                                                 const void *V_pages, void *O, float *LSE,
                                                 const int64_t q_str[3], const int64_t kv_str[4],
                                                 const int64_t o_str[3], const int32_t *block_table,
                                                 int64_t bt_stride, int max_pages, int page_size,
                                                 int num_pages, const int32_t *seqlens, int B,
                                                 int Hq, int Hkv, int d, float scale,
                                                 const uint8_t *m, int sink, int window,
                                                 const uint8_t *block_mask, int block_size,
                                                 int num_splits, void *workspace, size_t ws_bytes,
                                                 void *stream)
{
    if (!block_table || max_pages < 1 || num_pages < 1 || bt_stride < max_pages)
        return EA_ERR_INVALID_ARG;
    if (page_size < kDecKeys || page_size % kDecKeys != 0)
        return EA_ERR_UNSUPPORTED;
    const int64_t Lmax = static_cast<int64_t>(max_pages) * page_size;
    if (Lmax >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    return decode_launch(q, K_pages, V_pages, O, LSE, q_str, kv_str, o_str, seqlens, B, Hq, Hkv,
                         d, static_cast<int>(Lmax), scale, m, sink, window, block_mask, block_size,
                         num_splits, workspace, ws_bytes, block_table, bt_stride, page_size,
                         num_pages, stream);
}
