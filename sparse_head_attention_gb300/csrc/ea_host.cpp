// ea_host.cpp - host-side parts of the library: status strings, workspace
// layouts, TMA tensor-map encoding, the device error word read-back, and the
// sparsity ratios (a pure host computation).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "ea_internal.h"

namespace ea {

PrefillWs prefill_ws_layout(int B, int S, int Hq, int Hkv)
{
    PrefillWs w{};
    const int64_t nB = ceil_div(S, EA_TILE);
    const int64_t rows = static_cast<int64_t>(B) * Hkv * nB;
    const int64_t pairs = ceil_div(Hq / Hkv, 2);
    size_t off = sizeof(ea_ws_header);
    w.costs = off;
    off = align_up(off + sizeof(int32_t) * rows, 256);
    w.items = off;
    off = align_up(off + sizeof(uint32_t) * rows * pairs, 256);
    w.total = off;
    return w;
}

PrefillVarlenWs prefill_varlen_ws_layout(int B, int total_tokens, int Hq, int Hkv)
{
    PrefillVarlenWs w{};
    w.rows = static_cast<int64_t>(Hkv) * (ceil_div(total_tokens, EA_TILE) + B);
    const int64_t pairs = ceil_div(Hq / Hkv, 2);
    size_t off = sizeof(ea_ws_header);
    w.costs = off;
    off = align_up(off + sizeof(int32_t) * w.rows, 256);
    w.items = off;
    off = align_up(off + sizeof(uint32_t) * w.rows * pairs, 256);
    w.row_off = off;
    off = align_up(off + sizeof(int32_t) * (static_cast<size_t>(B) + 1), 256);
    w.mask_off = off;
    off = align_up(off + sizeof(int64_t) * (static_cast<size_t>(B) + 1), 256);
    w.row_desc = off;
    off = align_up(off + 8 * static_cast<size_t>(w.rows), 256);
    w.total = off;
    return w;
}

DecodeWs decode_ws_layout(int B, int Hq, int Hkv, int max_splits, int Lmax)
{
    DecodeWs w{};
    const size_t units = static_cast<size_t>(B) * Hkv;
    const size_t chunks = units * max_splits;
    const size_t g = Hq / Hkv;
    size_t off = sizeof(ea_ws_header);
    w.unit_first = off;
    off = align_up(off + sizeof(int32_t) * units, 256);
    w.unit_splits = off;
    off = align_up(off + sizeof(int32_t) * units, 256);
    w.chunks = off;
    off = align_up(off + sizeof(int32_t) * chunks, 256);
    w.partial_o = off;
    off = align_up(off + sizeof(float) * chunks * g * EA_HEAD_DIM, 256);
    w.partial_lse = off;
    off = align_up(off + sizeof(float) * chunks * g, 256);
    w.blk_count = off;
    off = align_up(off + sizeof(int32_t) * units, 256);
    w.blk_list = off;
    off = align_up(off + sizeof(uint16_t) * units * static_cast<size_t>(ceil_div(Lmax, EA_TILE)), 256);
    w.total = off;
    return w;
}

XaWs xa_ws_layout(int B, int S, int Hq, int Hkv, int max_units)
{
    (void)B;
    XaWs w{};
    const size_t g = Hq / Hkv;
    const size_t u = static_cast<size_t>(max_units);
    w.nA = S / EA_XA_STRIDE;
    w.nct = ceil_div(w.nA, 256);
    // rows a < nA hold 32 * (a / 256 + 1) sums each
    const int64_t G = w.nA / 256, r = w.nA % 256;
    w.tri = 32 * (256 * G * (G + 1) / 2 + r * (G + 1));
    size_t off = sizeof(ea_ws_header);
    w.units = off;
    off = align_up(off + sizeof(int32_t) * u, 256);
    w.tsum = off;
    off = align_up(off + sizeof(float) * u * g * w.nA * w.nct, 256);
    w.rmax = off;
    off = align_up(off + sizeof(float) * u * g * w.nA * w.nct, 256);
    w.esum = off;
    off = align_up(off + sizeof(float) * u * g * w.tri, 256);
    w.total = off;
    return w;
}

// Chunks per unit: the caller's count, or one per EA_DECODE_AUTO_CHUNK keys of
// the longest possible sequence.
int decode_max_splits(int Lmax, int num_splits)
{
    if (num_splits > 0)
        return num_splits;
    int64_t s = ceil_div(Lmax, EA_DECODE_AUTO_CHUNK);
    return static_cast<int>(s < 1 ? 1 : (s > 1024 ? 1024 : s));
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_tmap_bf16_4d(void *tmap_out, const void *base, int d, int H, int S, int B,
                         const int64_t strides_elems[4], int box_inner, int box_rows,
                         bool swizzle128)
{
    auto fn = get_encode_fn();
    if (!fn)
        return false;
    // strides_elems: (b, s, h, dim) outermost first
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(strides_elems[2]) * 2,
                             static_cast<cuuint64_t>(strides_elems[1]) * 2,
                             static_cast<cuuint64_t>(strides_elems[0]) * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), 1u, static_cast<cuuint32_t>(box_rows),
                         1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = fn(reinterpret_cast<CUtensorMap *>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tmap_bf16_cells(void *tmap_out, const void *base, int d, int H, int stride, int nA,
                            int B, const int64_t strides_elems[4], int box_rows)
{
    auto fn = get_encode_fn();
    if (!fn)
        return false;
    // token t = a * stride + u: dims (dim, head, u, a, b) innermost first
    cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(stride), static_cast<cuuint64_t>(nA),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[4] = {static_cast<cuuint64_t>(strides_elems[2]) * 2,
                             static_cast<cuuint64_t>(strides_elems[1]) * 2,
                             static_cast<cuuint64_t>(strides_elems[1]) * 2 * stride,
                             static_cast<cuuint64_t>(strides_elems[0]) * 2};
    cuuint32_t box[5] = {64u, 1u, 1u, static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    CUresult r = fn(reinterpret_cast<CUtensorMap *>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int num_sms(int device)
{
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return 0;
    return n;
}

} // namespace ea

using namespace ea;

extern "C" const char *ea_status_string(ea_status s)
{
    switch (s) {
    case EA_OK: return "ok";
    case EA_ERR_INVALID_ARG: return "invalid argument";
    case EA_ERR_UNSUPPORTED: return "unsupported configuration";
    case EA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case EA_ERR_CUDA: return "CUDA error";
    case EA_ERR_TIMEOUT: return "device wait timed out";
    case EA_ERR_DEVICE_CHECK: return "device-side argument check failed";
    }
    return "unknown status";
}

extern "C" size_t ea_prefill_workspace_size(int B, int S, int Hq, int Hkv, int d)
{
    if (B < 1 || S < 1 || S > EA_MAX_SEQ || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d != EA_HEAD_DIM)
        return 0;
    return prefill_ws_layout(B, S, Hq, Hkv).total;
}

extern "C" size_t ea_xa_workspace_size(int B, int S, int Hq, int Hkv, int d, int stride,
                                       int max_units)
{
    if (B < 1 || S < 1 || S > EA_MAX_SEQ || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
        d != EA_HEAD_DIM || stride != EA_XA_STRIDE || S % stride != 0 || max_units < 1 ||
        static_cast<int64_t>(max_units) > static_cast<int64_t>(B) * Hkv)
        return 0;
    return xa_ws_layout(B, S, Hq, Hkv, max_units).total;
}

extern "C" size_t ea_prefill_varlen_workspace_size(int B, int total_tokens, int max_seqlen, int Hq,
                                                   int Hkv, int d)
{
    if (B < 1 || total_tokens < 1 || max_seqlen < 1 || max_seqlen > EA_MAX_SEQ || Hq < 1 ||
        Hkv < 1 || Hq % Hkv != 0 || d != EA_HEAD_DIM)
        return 0;
    return prefill_varlen_ws_layout(B, total_tokens, Hq, Hkv).total;
}

extern "C" size_t ea_decode_workspace_size(int B, int Hq, int Hkv, int d, int Lmax, int num_splits)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d != EA_HEAD_DIM || Lmax < 1 ||
        num_splits < 0 || num_splits > 1024)
        return 0;
    return decode_ws_layout(B, Hq, Hkv, decode_max_splits(Lmax, num_splits), Lmax).total;
}

extern "C" ea_status ea_check_errors(void *workspace, void *stream)
{
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return EA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return EA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return EA_ERR_CUDA;
    if (word && cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess)
        return EA_ERR_CUDA;
    if (word & EA_DEVERR_TIMEOUT)
        return EA_ERR_TIMEOUT;
    if (word & (EA_DEVERR_CHECK | EA_DEVERR_BOUNDS))
        return EA_ERR_DEVICE_CHECK;
    return EA_OK;
}

// Kept causal (query, key) pairs of one KV head over S queries.
//   FULL : every causal pair.
//   SSA  : query i keeps min(i+1, window) window keys plus the sink keys below
//          the window, max(0, min(sink, i+1-window)).
//   BLOCK: a kept block strictly below the diagonal contributes all its
//          (rows x 128) pairs; a kept diagonal block its causal triangle.
static int64_t kept_pairs(int mode, int64_t S, int64_t sink, int64_t window, const uint8_t *bm)
{
    if (mode == EA_FULL)
        return S * (S + 1) / 2;
    if (mode == EA_SSA) {
        int64_t k = 0;
        for (int64_t i = 0; i < S; ++i) {
            const int64_t w = (i + 1 < window) ? i + 1 : window;
            int64_t s = i + 1 - window;
            if (s > sink)
                s = sink;
            if (s < 0)
                s = 0;
            k += w + s;
        }
        return k;
    }
    const int64_t T = EA_TILE, nB = ceil_div(S, T);
    int64_t k = 0;
    for (int64_t qb = 0; qb < nB; ++qb) {
        const int64_t r0 = qb * T, r1 = (qb + 1) * T < S ? (qb + 1) * T : S;
        const int64_t rows = r1 - r0;
        for (int64_t kb = 0; kb < qb; ++kb)
            if (bm[qb * nB + kb])
                k += rows * T;
        if (bm[qb * nB + qb])
            k += rows * (rows + 1) / 2;  // row r0 + t keeps t + 1 keys of its own block
    }
    return k;
}

extern "C" ea_status ea_sparsity_ratios(const uint8_t *r, const uint8_t *m, int L, int Hkv, int S,
                                        int sink, int window, const uint8_t *const *block_masks,
                                        int block_size, double *omega_msr, double *omega_esr)
{
    if (!r || !m || !omega_msr || !omega_esr || L < 1 || Hkv < 1 || S < 1 || sink < 0 || window < 1)
        return EA_ERR_INVALID_ARG;
    const int64_t causal = static_cast<int64_t>(S) * (S + 1) / 2;
    const int64_t nB = ceil_div(S, EA_TILE);
    int64_t n_sa = 0, pruned = 0;
    for (int l = 0; l < L; ++l)
        for (int h = 0; h < Hkv; ++h) {
            const uint8_t rv = r[l * Hkv + h], mv = m[l * Hkv + h];
            if (rv > 1 || mv > EA_BLOCK)
                return EA_ERR_INVALID_ARG;
            n_sa += rv;
            const uint8_t *bm = nullptr;
            if (mv == EA_BLOCK) {
                if (!block_masks || !block_masks[l] || block_size != EA_TILE)
                    return EA_ERR_INVALID_ARG;
                bm = block_masks[l] + static_cast<int64_t>(h) * nB * nB;
            }
            pruned += causal - kept_pairs(mv, S, sink, window, bm);
        }
    *omega_msr = static_cast<double>(n_sa) / (static_cast<double>(L) * static_cast<double>(Hkv));
    *omega_esr = static_cast<double>(pruned) /
                 (static_cast<double>(L) * static_cast<double>(Hkv) * static_cast<double>(causal));
    return EA_OK;
}
