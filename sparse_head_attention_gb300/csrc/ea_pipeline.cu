// ea_pipeline.cpp - the prefill on host-resident tensors, with copies and
// attention overlapped (ea_hybrid_attn_prefill_host).
//
// Under a causal mask (FA, SSA and block-sparse alike, "Paper Reading -
// Elastic Attention" (English notes), §02 eqs. (1)-(3)) query block qb reads
// key/value rows below (qb + 1) * 128 only.  So the sequence is cut into
// chunks of whole query blocks and run as a three-stage pipeline:
//
//   up stream       Q/K/V rows of chunk c                  -> event in[c]
//   (chunks shrink toward the end of the sequence, see chunk_bounds)
//   compute stream  wait in[c]; plan + attention over chunk c's query blocks
//                                                          -> event out[c]
//   down stream     wait out[c]; O / LSE rows of chunk c back to the host
//
// Chunk c's attention overlaps chunk c+1's upload and chunk c-1's download.
// Even chunks run on the caller's stream and odd chunks on a second compute
// stream, each with a planner workspace of its own, so that the next chunk's
// persistent CTAs take over SMs as soon as the current chunk's CTAs drain
// (a chunk ends with a few long query blocks).  Concurrent chunks write
// disjoint rows of O / LSE and only read Q/K/V.  Nothing here waits on the
// host: ordering is by events only.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "ea_internal.h"

namespace ea {

constexpr int kMaxChunks = 64;
constexpr int kAutoChunks = 10;

// Query-block boundaries of the chunks: chunk c ends near
// nB * (1 - (1 - (c + 1) / n)^1.25), so that the chunks shrink toward the end.
// Under a causal mask the last query blocks carry the most work, and what
// remains after the last upload is the last chunk's attention and download:
// the smaller that chunk, the shorter the tail.  (32K Llama-shaped layer,
// median step: 8 equal chunks 3.02 ms, 10 equal 3.00 ms; 10 shrinking with
// exponent 1.2 / 1.25-1.3 / 1.4: 2.92 / 2.92 / 2.94 ms; 12 with 1.2: 2.92 ms.)
// Every chunk holds at least one query block.
static void chunk_bounds(int nB, int n, int *qb)
{
    qb[0] = 0;
    for (int c = 1; c < n; ++c) {
        int v = static_cast<int>(nB * (1.0 - std::pow(1.0 - static_cast<double>(c) / n, 1.25)));
        v = v > qb[c - 1] + 1 ? v : qb[c - 1] + 1;
        v = v < nB - (n - c) ? v : nB - (n - c);
        qb[c] = v;
    }
    qb[n] = nB;
}

// Device buffer layout (every part 256-byte aligned): the two planner
// workspaces first.
struct HostBufLayout {
    size_t ws, ws2, ws_bytes, m, bm, q, k, v, o, lse, total;
};

static HostBufLayout host_buf_layout(int B, int S, int Hq, int Hkv, bool with_bm)
{
    HostBufLayout L{};
    const size_t nB = static_cast<size_t>(ceil_div(S, EA_TILE));
    const size_t row_q = static_cast<size_t>(Hq) * EA_HEAD_DIM * 2;
    const size_t row_kv = static_cast<size_t>(Hkv) * EA_HEAD_DIM * 2;
    const size_t BS = static_cast<size_t>(B) * S;
    size_t off = 0;
    L.ws_bytes = align_up(prefill_ws_layout(B, S, Hq, Hkv).total, 256);
    L.ws = off;
    off += L.ws_bytes;
    L.ws2 = off;
    off += L.ws_bytes;
    L.m = off;
    off = align_up(off + static_cast<size_t>(B) * Hkv, 256);
    L.bm = off;
    off = align_up(off + (with_bm ? static_cast<size_t>(B) * Hkv * nB * nB : 0), 256);
    L.q = off;
    off = align_up(off + BS * row_q, 256);
    L.k = off;
    off = align_up(off + BS * row_kv, 256);
    L.v = off;
    off = align_up(off + BS * row_kv, 256);
    L.o = off;
    off = align_up(off + BS * row_q, 256);
    L.lse = off;
    off = align_up(off + static_cast<size_t>(B) * Hq * S * sizeof(float), 256);
    L.total = off;
    return L;
}

// Per-device copy streams and events, created on first use and kept for the
// life of the process.  The mutex serialises the enqueue sequence of calls on
// one device; an event may be re-recorded once the waits on its previous
// record have been enqueued, which holds under the lock.
struct PipeResources {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr, comp = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kMaxChunks] = {}, out[kMaxChunks] = {};
};

static PipeResources g_pipe[64];
static std::mutex g_pipe_mutex[64];

static cudaError_t pipe_init(PipeResources &r)
{
    if (r.ready)
        return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&r.up, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&r.down, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&r.comp, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&r.start, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&r.done, cudaEventDisableTiming);
    for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
        e = cudaEventCreateWithFlags(&r.in[c], cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&r.out[c], cudaEventDisableTiming);
    }
    if (e == cudaSuccess)
        r.ready = true;
    return e;
}

// Rows [r0, r1) of every batch entry of a [B][S][row_bytes] tensor.
static cudaError_t copy_rows(void *dst, const void *src, size_t row_bytes, int B, int S, int r0,
                             int r1, cudaMemcpyKind kind, cudaStream_t st)
{
    const size_t pitch = row_bytes * S;
    const size_t off = row_bytes * r0;
    return cudaMemcpy2DAsync(static_cast<char *>(dst) + off, pitch,
                             static_cast<const char *>(src) + off, pitch,
                             row_bytes * (r1 - r0), B, kind, st);
}

// Fold the second workspace's device error word into the first, so that one
// ea_check_errors on the buffer reports both.
__global__ void merge_error_words(ea_ws_header *a, ea_ws_header *b)
{
    if (b->error) {
        a->error |= b->error;
        b->error = 0;
    }
}

} // namespace ea

using namespace ea;

extern "C" size_t ea_prefill_host_buffer_size(int B, int S, int Hq, int Hkv, int d,
                                              int with_block_mask)
{
    if (ea_prefill_workspace_size(B, S, Hq, Hkv, d) == 0)
        return 0;
    return host_buf_layout(B, S, Hq, Hkv, with_block_mask != 0).total;
}

extern "C" ea_status ea_hybrid_attn_prefill_host(const void *Q_host, const void *K_host,
                                                 const void *V_host, void *O_host, float *LSE_host,
                                                 int B, int S, int Hq, int Hkv, int d, float scale,
                                                 const uint8_t *m_host, int sink, int window,
                                                 const uint8_t *block_mask_host, int block_size,
                                                 void *device_buffer, size_t buffer_bytes,
                                                 int n_chunks, void *stream)
{
    // every check happens before the first enqueue
    if (!Q_host || !K_host || !V_host || !O_host || !m_host || !(scale > 0.f))
        return EA_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || sink < 0 || window < 1 ||
        block_size != EA_TILE || B > 65535)
        return EA_ERR_INVALID_ARG;
    if (d != EA_HEAD_DIM || S > EA_MAX_SEQ)
        return EA_ERR_UNSUPPORTED;
    const int nB = static_cast<int>(ceil_div(S, EA_TILE));
    if (static_cast<int64_t>(B) * Hkv * nB * ((Hq / Hkv + 1) / 2) >= (int64_t(1) << 31))
        return EA_ERR_UNSUPPORTED;
    if (n_chunks < 0 || n_chunks > kMaxChunks || n_chunks > nB)
        return EA_ERR_INVALID_ARG;
    if (n_chunks == 0)
        n_chunks = nB < kAutoChunks ? nB : kAutoChunks;
    const bool with_bm = block_mask_host != nullptr;
    const HostBufLayout L = host_buf_layout(B, S, Hq, Hkv, with_bm);
    if (!device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) ||
        buffer_bytes < L.total)
        return EA_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64)
        return EA_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    PipeResources &R = g_pipe[dev];
    if (pipe_init(R) != cudaSuccess)
        return EA_ERR_CUDA;

    uint8_t *buf = static_cast<uint8_t *>(device_buffer);
    void *ws_of[2] = {buf + L.ws, buf + L.ws2};
    uint8_t *dm = buf + L.m;
    uint8_t *dbm = with_bm ? buf + L.bm : nullptr;
    void *dQ = buf + L.q, *dK = buf + L.k, *dV = buf + L.v, *dO = buf + L.o;
    float *dL = LSE_host ? reinterpret_cast<float *>(buf + L.lse) : nullptr;
    const size_t row_q = static_cast<size_t>(Hq) * EA_HEAD_DIM * 2;
    const size_t row_kv = static_cast<size_t>(Hkv) * EA_HEAD_DIM * 2;
    const int64_t q_str[4] = {static_cast<int64_t>(S) * Hq * EA_HEAD_DIM,
                              static_cast<int64_t>(Hq) * EA_HEAD_DIM, EA_HEAD_DIM, 1};
    const int64_t kv_str[4] = {static_cast<int64_t>(S) * Hkv * EA_HEAD_DIM,
                               static_cast<int64_t>(Hkv) * EA_HEAD_DIM, EA_HEAD_DIM, 1};
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // the copy streams start after the caller's earlier work (which may still
    // use this device buffer)
    if (cudaEventRecord(R.start, st) != cudaSuccess ||
        cudaStreamWaitEvent(R.up, R.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(R.down, R.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(R.comp, R.start, 0) != cudaSuccess)
        return EA_ERR_CUDA;
    cudaStream_t comp_of[2] = {st, R.comp};
    // On a failure after this point the caller's stream is still made to wait
    // for whatever the copy streams already hold, so that freeing the buffers
    // after synchronising `stream` stays safe.
    auto fail = [&](ea_status s) {
        for (cudaStream_t x : {R.up, R.comp, R.down})
            if (cudaEventRecord(R.done, x) == cudaSuccess)
                cudaStreamWaitEvent(st, R.done, 0);
        return s;
    };
    if (cudaMemcpyAsync(dm, m_host, static_cast<size_t>(B) * Hkv, cudaMemcpyHostToDevice, R.up) !=
        cudaSuccess)
        return fail(EA_ERR_CUDA);
    if (with_bm &&
        cudaMemcpyAsync(dbm, block_mask_host, static_cast<size_t>(B) * Hkv * nB * nB,
                        cudaMemcpyHostToDevice, R.up) != cudaSuccess)
        return fail(EA_ERR_CUDA);

    int bounds[kMaxChunks + 1];
    chunk_bounds(nB, n_chunks, bounds);
    for (int c = 0; c < n_chunks; ++c) {
        const int qb0 = bounds[c];
        const int qb1 = bounds[c + 1];
        const int r0 = qb0 * EA_TILE;
        const int r1 = qb1 * EA_TILE < S ? qb1 * EA_TILE : S;
        if (copy_rows(dQ, Q_host, row_q, B, S, r0, r1, cudaMemcpyHostToDevice, R.up) ||
            copy_rows(dK, K_host, row_kv, B, S, r0, r1, cudaMemcpyHostToDevice, R.up) ||
            copy_rows(dV, V_host, row_kv, B, S, r0, r1, cudaMemcpyHostToDevice, R.up))
            return fail(EA_ERR_CUDA);
        cudaStream_t cs = comp_of[c & 1];
        void *ws = ws_of[c & 1];
        if (cudaEventRecord(R.in[c], R.up) || cudaStreamWaitEvent(cs, R.in[c], 0))
            return fail(EA_ERR_CUDA);
        ea_status s = prefill_plan_range(B, S, Hq, Hkv, d, dm, sink, window, dbm, block_size, ws,
                                         L.ws_bytes, qb0, qb1, cs);
        if (s == EA_OK)
            s = prefill_attend_range(dQ, dK, dV, dO, dL, q_str, kv_str, q_str, B, S, Hq, Hkv, d,
                                     scale, dm, sink, window, dbm, block_size, ws, L.ws_bytes,
                                     nullptr, qb0, qb1, cs);
        if (s != EA_OK)
            return fail(s);
        if (cudaEventRecord(R.out[c], cs) || cudaStreamWaitEvent(R.down, R.out[c], 0) ||
            copy_rows(O_host, dO, row_q, B, S, r0, r1, cudaMemcpyDeviceToHost, R.down))
            return fail(EA_ERR_CUDA);
        // LSE [B][Hq][S]: rows r0..r1 of each (b, head) line
        if (LSE_host &&
            cudaMemcpy2DAsync(LSE_host + r0, sizeof(float) * S, dL + r0, sizeof(float) * S,
                              sizeof(float) * (r1 - r0), static_cast<size_t>(B) * Hq,
                              cudaMemcpyDeviceToHost, R.down) != cudaSuccess)
            return fail(EA_ERR_CUDA);
    }
    // later work on the caller's stream sees the copies back as well (the
    // down stream has waited for every chunk of both compute streams)
    if (cudaEventRecord(R.done, R.down) != cudaSuccess ||
        cudaStreamWaitEvent(st, R.done, 0) != cudaSuccess)
        return fail(EA_ERR_CUDA);
    merge_error_words<<<1, 1, 0, st>>>(static_cast<ea_ws_header *>(ws_of[0]),
                                       static_cast<ea_ws_header *>(ws_of[1]));
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}
