// ea_internal.h - definitions shared by the library's translation units (host
// and device): workspace layout, device error bits, tile sizes, host helpers.
#pragma once

#include <cstddef>
#include <cstdint>

#include "ea.h"

// Tile edge (query rows per tile, keys per tile, block-mask block) and head dim.
#define EA_TILE 128
#define EA_HEAD_DIM 128

// Device error bits in the workspace error word.
#define EA_DEVERR_CHECK 1u    // invalid mode / missing block mask / bad seqlen
#define EA_DEVERR_TIMEOUT 2u  // a bounded wait ran out
#define EA_DEVERR_BOUNDS 4u   // bounds-checked builds (-DEA_CHECKS): an index out of range

// A bounded device wait gives up after this long (ns).
#define EA_WAIT_TIMEOUT_NS 2000000000ull

// Every workspace starts with this 256-byte header.
struct ea_ws_header {
    uint32_t error;         // EA_DEVERR_* bits
    uint32_t work_counter;  // persistent-kernel work queue head
    uint32_t n_items;       // number of work items in the queue
    uint32_t drained;       // CTAs that found the queue empty (last one resets it)
    uint32_t reserved[60];
};
static_assert(sizeof(ea_ws_header) == 256, "workspace header must be 256 bytes");

// Largest supported prefill length: the planner's histogram lives in shared
// memory (one int per possible tile count).
#define EA_MAX_SEQ (1 << 21)

namespace ea {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets of the prefill workspace regions.
struct PrefillWs {
    size_t costs;   // int32 [B*Hkv*nB]: visited tiles per (b, KV head, q block)
    size_t items;   // uint32 [n_items]: work items, longest first
    size_t total;
};
PrefillWs prefill_ws_layout(int B, int S, int Hq, int Hkv);

// Workspace of a variable-length prefill: rows are bounded by
// Hkv * (ceil(total_tokens / 128) + B) (each sequence rounds up once).
struct PrefillVarlenWs {
    int64_t rows;   // upper bound on planned rows
    size_t costs;   // int32 [rows]
    size_t items;   // uint32 [rows * pairs]
    size_t row_off; // int32 [B + 1]: first row of each sequence
    size_t mask_off;// int64 [B + 1]: first block-mask byte of each sequence
    size_t row_desc;// int2 [rows]: {b, h << 16 | qb} of each planned row
    size_t total;
};
PrefillVarlenWs prefill_varlen_ws_layout(int B, int total_tokens, int Hq, int Hkv);

// Byte offsets of the decode workspace regions.  A chunk is one split of one
// (b, KV head) unit; every unit has at most max_splits chunks.
struct DecodeWs {
    size_t unit_first;   // int32 [B*Hkv]: index of the unit's first chunk
    size_t unit_splits;  // int32 [B*Hkv]: number of chunks of the unit
    size_t chunks;       // int32 [B*Hkv*max_splits]: unit << 11 | split
    size_t partial_o;    // float [B*Hkv*max_splits][g][128]
    size_t partial_lse;  // float [B*Hkv*max_splits][g]
    size_t blk_count;    // int32 [B*Hkv]: kept key blocks of a BLOCK unit's decode row
    size_t blk_list;     // uint16 [B*Hkv][ceil(Lmax / 128)]: those blocks, ascending
    size_t total;
};
DecodeWs decode_ws_layout(int B, int Hq, int Hkv, int max_splits, int Lmax);
// Keys per chunk when the split count is automatic.
#define EA_DECODE_AUTO_CHUNK 2048
// Largest automatic decode chunk (kept keys); the planner picks a size between
// the two from the step's total kept keys.
#define EA_DECODE_MAX_CHUNK 8192
int decode_max_splits(int Lmax, int num_splits);

// Encodes a 4-D bf16 TMA tensor map (dims innermost first: head dim, heads,
// sequence, batch; strides in elements) with a 64 x 1 x box_rows x 1 box and
// 128-byte swizzle (swizzle128) or none.  Returns false if the driver rejects it.
bool encode_tmap_bf16_4d(void *tmap_out, const void *base, int d, int H, int S, int B,
                         const int64_t strides_elems[4], int box_inner, int box_rows,
                         bool swizzle128);

// Encodes a 5-D bf16 TMA tensor map that reads tokens as cells of `stride`
// consecutive tokens: dims (head dim, heads, offset u in the cell, cell a,
// batch), token a * stride + u; the sequence length must be nA * stride.  Box:
// 64 x 1 x 1 x box_rows x 1 with 128-byte swizzle (box_rows cells at one
// offset u).
bool encode_tmap_bf16_cells(void *tmap_out, const void *base, int d, int H, int stride, int nA,
                            int B, const int64_t strides_elems[4], int box_rows);

// XA estimation workspace (one slot per BLOCK (b, KV head) unit, at most
// max_units): per slot and query head of the group, and per cell row and
// 256-cell key tile, the row's max over the tile (log2 units) and the total of
// exp2(score - max) over the tile; and the per-row sums of exp2(score - tile
// max) over each key block (row a holds 32 * (a / 256 + 1) of them, rows packed
// back to back).
#define EA_XA_STRIDE 16
struct XaWs {
    int64_t nA;      // cell rows (S / stride)
    int64_t nct;     // 256-cell key tiles (ceil(nA / 256))
    int64_t tri;     // floats of one (unit, query head) row-sum block
    size_t units;    // int32 [max_units]: b << 16 | h of each BLOCK unit
    size_t tsum;     // float [max_units][g][nA][nct]
    size_t rmax;     // float [max_units][g][nA][nct]
    size_t esum;     // float [max_units][g][tri]
    size_t total;
};
XaWs xa_ws_layout(int B, int S, int Hq, int Hkv, int max_units);

int num_sms(int device);

// Planner and attention launch restricted to query blocks [qb_begin, qb_end)
// (qb_end = -1: up to the last block).  A plan and the launch that consumes it
// must name the same range.  The exported ea_prefill_plan / ea_prefill_attend
// are these over every block.
ea_status prefill_plan_range(int B, int S, int Hq, int Hkv, int d, const uint8_t *m, int sink,
                             int window, const uint8_t *block_mask, int block_size, void *workspace,
                             size_t ws_bytes, int qb_begin, int qb_end, void *stream);
ea_status prefill_attend_range(const void *Q, const void *K, const void *V, void *O, float *LSE,
                               const int64_t q_str[4], const int64_t kv_str[4],
                               const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                               float scale, const uint8_t *m, int sink, int window,
                               const uint8_t *block_mask, int block_size, void *workspace,
                               size_t ws_bytes, uint32_t *visited_bitmap, int qb_begin, int qb_end,
                               void *stream);

} // namespace ea
