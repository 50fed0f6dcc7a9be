// ea_decode.cu - one decode step of hybrid-head attention with the routing
// decision fixed at prefill ("Paper Reading - Elastic Attention" (English
// notes), §08 Commentary, stated limit ③: routing is decided once per request,
// at the prefill stage).
//
// A decode step reads every kept cache entry once, so it is bound by HBM
// bandwidth.  The design reads each (b, KV head)'s kept keys exactly once and
// shares every K/V row among the query heads of the GQA group:
//   decode_plan_kernel: per (b, KV head) unit the number of kept keys (FULL:
//     [0, L); SSA: the sink [0, sink) and the window [L - window, L)), its
//     chunk count (about 2048 keys each unless the caller fixes the count),
//     and the list of chunks.  Short SSA units get few chunks, long FA units
//     many, so no CTA is spent on a handful of keys.
//   decode_split_kernel: persistent, one CTA per SM walking the chunk list.
//     Each chunk's keys stream through a 4-stage shared-memory ring filled by
//     TMA (64 keys x 256 B per K or V box); the group's query heads share each
//     K/V row; fp32 online softmax per head.  Output: a partial (O / l, LSE)
//     per (chunk, q head).
//   decode_merge_kernel: combines the partials of each (b, q head) by
//     log-sum-exp weights and writes bf16 O and fp32 LSE.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ea_device.cuh"
#include "ea_internal.h"

namespace ea {

constexpr int kDecKeys = 64;                           // keys per TMA box
constexpr int kDecStages = 4;
constexpr int kDecRowBytes = EA_HEAD_DIM * 2;          // 256
constexpr int kDecBoxBytes = kDecKeys * kDecRowBytes;  // 16 KB
constexpr int kDecThreads = 256;                       // 8 warps x 4 groups of 8 lanes
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
    int B, Hq, Hkv, g, Lmax, sink, window, num_splits, max_splits;
    float scale_log2;
};

template <int G>
struct DecSmem {
    uint8_t kv[kDecStages][2][kDecBoxBytes];
    float red_o[8][G][EA_HEAD_DIM];
    float red_m[8][G];
    float red_l[8][G];
    uint64_t full[kDecStages];
};

// Kept keys of one (b, KV head) unit as at most two contiguous ranges:
// visited index v < n0 is key v, v >= n0 is key w0 + (v - n0).
struct KeySegs {
    int n;
    int n0;
    int w0;
};

__device__ __forceinline__ bool unit_keys(const DecodeArgs &a, int b, int h, KeySegs &ks)
{
    int L = a.seqlens[b];
    const int mode = a.m[b * a.Hkv + h];
    bool ok = true;
    if (L < 0 || L > a.Lmax || mode > EA_SSA) {  // BLOCK has no decode reading
        ok = false;
        L = 0;
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

// One CTA: per-unit chunk counts (automatic: one chunk per
// EA_DECODE_AUTO_CHUNK kept keys), their prefix sum, and the chunk list.
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeArgs a)
{
    __shared__ int scan_tmp[1024];
    const int units = a.B * a.Hkv;
    const int tid = threadIdx.x;
    const int per = (units + blockDim.x - 1) / blockDim.x;
    const int lo = tid * per, hi = min(lo + per, units);
    int local = 0;
    for (int u = lo; u < hi; ++u) {
        KeySegs ks;
        if (!unit_keys(a, u / a.Hkv, u % a.Hkv, ks))
            raise_error(&a.hdr->error, EA_DEVERR_CHECK);
        int ns = a.num_splits > 0 ? a.num_splits
                                  : (ks.n + EA_DECODE_AUTO_CHUNK - 1) / EA_DECODE_AUTO_CHUNK;
        ns = ns < 1 ? 1 : (ns > a.max_splits ? a.max_splits : ns);
        a.unit_splits[u] = ns;
        local += ns;
    }
    scan_tmp[tid] = local;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int v = tid >= off ? scan_tmp[tid - off] : 0;
        __syncthreads();
        scan_tmp[tid] += v;
        __syncthreads();
    }
    int run = scan_tmp[tid] - local;
    for (int u = lo; u < hi; ++u) {
        a.unit_first[u] = run;
        const int ns = a.unit_splits[u];
        for (int sp = 0; sp < ns; ++sp)
            a.chunks[run + sp] = (u << kSplitBits) | sp;
        run += ns;
    }
    if (tid == 1023)
        a.hdr->n_items = static_cast<uint32_t>(scan_tmp[1023]);
}

// Position of chunk c in the key stream.
struct ChunkInfo {
    int b, h, v_begin, v_end;
    KeySegs ks;
    int a_tiles, b_begin, n_tiles;
};

__device__ __forceinline__ ChunkInfo chunk_info(const DecodeArgs &a, int c)
{
    ChunkInfo ci;
    const int code = a.chunks[c];
    const int u = code >> kSplitBits, sp = code & ((1 << kSplitBits) - 1);
    ci.b = u / a.Hkv;
    ci.h = u % a.Hkv;
    unit_keys(a, ci.b, ci.h, ci.ks);
    const int ns = a.unit_splits[u];
    const int len = (ci.ks.n + ns - 1) / ns;
    ci.v_begin = min(sp * len, ci.ks.n);
    ci.v_end = min(ci.v_begin + len, ci.ks.n);
    const int a_end = min(ci.v_end, ci.ks.n0);
    ci.a_tiles = ci.v_begin < a_end ? (a_end - ci.v_begin + kDecKeys - 1) / kDecKeys : 0;
    ci.b_begin = max(ci.v_begin, ci.ks.n0);
    ci.n_tiles = ci.a_tiles + (ci.b_begin < ci.v_end ? (ci.v_end - ci.b_begin + kDecKeys - 1) / kDecKeys : 0);
    return ci;
}

// First cache row and number of valid keys of tile t of a chunk (a tile never
// straddles the sink and window ranges).
__device__ __forceinline__ void tile_rows(const ChunkInfo &ci, int t, int &key0, int &nvalid)
{
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

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ void unpack16(const uint4 &u0, const uint4 &u1, float (&f)[16])
{
    f[0] = bf_lo(u0.x); f[1] = bf_hi(u0.x); f[2] = bf_lo(u0.y); f[3] = bf_hi(u0.y);
    f[4] = bf_lo(u0.z); f[5] = bf_hi(u0.z); f[6] = bf_lo(u0.w); f[7] = bf_hi(u0.w);
    f[8] = bf_lo(u1.x); f[9] = bf_hi(u1.x); f[10] = bf_lo(u1.y); f[11] = bf_hi(u1.y);
    f[12] = bf_lo(u1.z); f[13] = bf_hi(u1.z); f[14] = bf_lo(u1.w); f[15] = bf_hi(u1.w);
}

// Persistent: CTA x handles chunks x, x + grid, x + 2 grid, ...  Thread 0
// keeps kDecStages K/V tile pairs in flight, running ahead across chunk
// boundaries, so a chunk's epilogue overlaps the next chunk's loads.
template <int G>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    DecSmem<G> &sm = *reinterpret_cast<DecSmem<G> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int grp = lane >> 3, j = lane & 7;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int total = static_cast<int>(a.hdr->n_items);

    if (tid == 0) {
        for (int s = 0; s < kDecStages; ++s)
            mbar_init(&sm.full[s], 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    // producer cursor (thread 0 only)
    int pc = blockIdx.x, pt = 0;
    ChunkInfo pci;
    if (tid == 0 && pc < total)
        pci = chunk_info(a, pc);
    uint32_t issued = 0;
    auto issue_next = [&]() {
        while (pc < total && pt >= pci.n_tiles) {
            pc += gridDim.x;
            pt = 0;
            if (pc < total)
                pci = chunk_info(a, pc);
        }
        if (pc >= total)
            return;
        int key0, nv;
        tile_rows(pci, pt, key0, nv);
        const int s = issued % kDecStages;
        mbar_arrive_expect_tx(&sm.full[s], 2 * kDecBoxBytes);
        tma_load_4d(sm.kv[s][0], &tm_k, 0, pci.h, key0, pci.b, &sm.full[s]);
        tma_load_4d(sm.kv[s][1], &tm_v, 0, pci.h, key0, pci.b, &sm.full[s]);
        ++issued;
        ++pt;
    };
    if (tid == 0)
        for (int k = 0; k < kDecStages; ++k)
            issue_next();

    volatile int no_abort = 0;
    uint32_t consumed = 0;
    for (int c = blockIdx.x; c < total; c += gridDim.x) {
        const ChunkInfo ci = chunk_info(a, c);
        // query slices of this lane: d in {8j..8j+7} and {64+8j..64+8j+7}
        float q[G][16];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const int qh = ci.h * a.g + (hh < a.g ? hh : 0);
            const uint4 *qp = reinterpret_cast<const uint4 *>(a.q + ci.b * a.q_sb + qh * a.q_sh);
            unpack16(qp[j], qp[8 + j], q[hh]);
        }
        float m_run[G], l_run[G], o[G][16];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            m_run[hh] = NEG_INF;
            l_run[hh] = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                o[hh][e] = 0.f;
        }
        for (int t = 0; t < ci.n_tiles; ++t) {
            const int s = consumed % kDecStages;
            if (!mbar_wait(&sm.full[s], (consumed / kDecStages) & 1, &no_abort, &a.hdr->error))
                return;  // timed out: the error word is set
            ++consumed;
            int key0, nv;
            tile_rows(ci, t, key0, nv);
            const uint8_t *kt = sm.kv[s][0];
            const uint8_t *vt = sm.kv[s][1];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int key = warp * 8 + grp * 2 + kk;
                const uint4 *kr = reinterpret_cast<const uint4 *>(kt + key * kDecRowBytes);
                float kf[16];
                unpack16(kr[j], kr[8 + j], kf);
                float sc[G];
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        acc = fmaf(q[hh][e], kf[e], acc);
                    sc[hh] = acc;
                }
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 1);
                    sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 2);
                    sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 4);
                }
                if (key < nv) {
                    const uint4 *vr = reinterpret_cast<const uint4 *>(vt + key * kDecRowBytes);
                    float vf[16];
                    unpack16(vr[j], vr[8 + j], vf);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float x = sc[hh] * a.scale_log2;
                        if (x > m_run[hh]) {
                            const float f = ex2(m_run[hh] - x);
                            l_run[hh] *= f;
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                o[hh][e] *= f;
                            m_run[hh] = x;
                        }
                        const float p = ex2(x - m_run[hh]);
                        l_run[hh] += p;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[hh][e] = fmaf(p, vf[e], o[hh][e]);
                    }
                }
            }
            __syncthreads();  // every warp is done with stage s: refill it
            if (tid == 0)
                issue_next();
        }

        // combine the 4 groups of each warp (lanes j, j+8, j+16, j+24 hold the same d)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
#pragma unroll
            for (int off = 8; off <= 16; off <<= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, m_run[hh], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l_run[hh], off);
                const float mn = fmaxf(m_run[hh], mo);
                const float fa = mn == NEG_INF ? 0.f : ex2(m_run[hh] - mn);
                const float fb = mn == NEG_INF ? 0.f : ex2(mo - mn);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float oo = __shfl_xor_sync(0xffffffffu, o[hh][e], off);
                    o[hh][e] = o[hh][e] * fa + oo * fb;
                }
                l_run[hh] = l_run[hh] * fa + lo * fb;
                m_run[hh] = mn;
            }
        }
        // combine the 8 warps through shared memory
        if (grp == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int dd = e < 8 ? 8 * j + e : 64 + 8 * j + (e - 8);
                    sm.red_o[warp][hh][dd] = o[hh][e];
                }
                if (j == 0) {
                    sm.red_m[warp][hh] = m_run[hh];
                    sm.red_l[warp][hh] = l_run[hh];
                }
            }
        }
        __syncthreads();
        for (int idx = tid; idx < G * EA_HEAD_DIM; idx += kDecThreads) {
            const int hh = idx / EA_HEAD_DIM, dd = idx % EA_HEAD_DIM;
            if (hh >= a.g)
                continue;
            float M = NEG_INF;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                M = fmaxf(M, sm.red_m[w][hh]);
            float lsum = 0.f, osum = 0.f;
            if (M > NEG_INF)
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float f = ex2(sm.red_m[w][hh] - M);
                    lsum += sm.red_l[w][hh] * f;
                    osum += sm.red_o[w][hh][dd] * f;
                }
            const int64_t pidx = static_cast<int64_t>(c) * a.g + hh;
            a.part_o[pidx * EA_HEAD_DIM + dd] = lsum > 0.f ? osum / lsum : 0.f;
            if (dd == 0)
                a.part_lse[pidx] = lsum > 0.f ? (M + __log2f(lsum)) * 0.69314718055994531f : NEG_INF;
        }
        __syncthreads();  // the reduction buffers are reused by the next chunk
    }
}

// One CTA of 128 threads per (q head, b): log-sum-exp merge of the unit's chunks.
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a)
{
    const int qh = blockIdx.x, b = blockIdx.y, dd = threadIdx.x;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int u = b * a.Hkv + qh / a.g, hh = qh % a.g;
    const int first = a.unit_first[u], ns = a.unit_splits[u];
    float M = NEG_INF;
    for (int s = 0; s < ns; ++s)
        M = fmaxf(M, a.part_lse[static_cast<int64_t>(first + s) * a.g + hh]);
    float wsum = 0.f, osum = 0.f;
    if (M > NEG_INF)
        for (int s = 0; s < ns; ++s) {
            const int64_t pidx = static_cast<int64_t>(first + s) * a.g + hh;
            const float w = __expf(a.part_lse[pidx] - M);
            wsum += w;
            osum += w * a.part_o[pidx * EA_HEAD_DIM + dd];
        }
    const float out = wsum > 0.f ? osum / wsum : 0.f;
    a.O[b * a.o_sb + qh * a.o_sh + dd] = __float2bfloat16_rn(out);
    if (dd == 0 && a.LSE)
        a.LSE[static_cast<int64_t>(b) * a.Hq + qh] = wsum > 0.f ? M + __logf(wsum) : NEG_INF;
}

template <int G>
static cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                                 int grid, cudaStream_t st)
{
    const size_t smem = sizeof(DecSmem<G>) + 128;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    decode_split_kernel<G><<<grid, kDecThreads, smem, st>>>(tk, tv, a);
    return cudaGetLastError();
}

} // namespace ea

using namespace ea;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" ea_status ea_hybrid_attn_decode(const void *q, const void *Kc, const void *Vc, void *O,
                                           float *LSE, const int64_t q_str[3],
                                           const int64_t kv_str[4], const int64_t o_str[3],
                                           const int32_t *seqlens, int B, int Hq, int Hkv, int d,
                                           int Lmax, float scale, const uint8_t *m, int sink,
                                           int window, int num_splits, void *workspace,
                                           size_t ws_bytes, void *stream)
{
    if (!q || !Kc || !Vc || !O || !q_str || !kv_str || !o_str || !seqlens || !m)
        return EA_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lmax < 1 || sink < 0 || window < 1 ||
        !(scale > 0.f) || num_splits < 0 || num_splits > 1024)
        return EA_ERR_INVALID_ARG;
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
    const DecodeWs L = decode_ws_layout(B, Hq, Hkv, max_splits);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < L.total)
        return EA_ERR_WORKSPACE;

    alignas(64) CUtensorMap tk, tv;
    if (!encode_tmap_bf16_4d(&tk, Kc, d, Hkv, Lmax, B, kv_str, EA_HEAD_DIM, kDecKeys, false) ||
        !encode_tmap_bf16_4d(&tv, Vc, d, Hkv, Lmax, B, kv_str, EA_HEAD_DIM, kDecKeys, false))
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

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return EA_ERR_CUDA;
    const int sms = num_sms(dev);
    if (sms <= 0)
        return EA_ERR_CUDA;
    const int64_t max_chunks = static_cast<int64_t>(B) * Hkv * max_splits;
    const int grid = static_cast<int>(max_chunks < sms ? max_chunks : sms);
    decode_plan_kernel<<<1, 1024, 0, st>>>(a);
    cudaError_t e;
    if (a.g == 1)
        e = launch_decode<1>(tk, tv, a, grid, st);
    else if (a.g == 2)
        e = launch_decode<2>(tk, tv, a, grid, st);
    else if (a.g <= 4)
        e = launch_decode<4>(tk, tv, a, grid, st);
    else
        e = launch_decode<8>(tk, tv, a, grid, st);
    if (e != cudaSuccess)
        return EA_ERR_CUDA;
    decode_merge_kernel<<<dim3(Hq, B), EA_HEAD_DIM, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}
