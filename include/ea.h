/*
 * ea.h - C ABI of the Elastic Attention hybrid-head attention library (sm_103a).
 *
 * Elastic Attention gives every KV head of every layer a per-input routing
 * decision r in {0 = FA, 1 = SA} from a small Attention Router, maps r to
 * kernel metadata m, and runs all heads of a layer, whatever their mode, in one
 * fused launch whose output is the plain concatenation of the per-head outputs.
 *
 * Sources (page titles as printed):
 *   [EN] "Paper Reading - Elastic Attention: Test-time Adaptive Sparsity Ratios"
 *        (English reading notes of arXiv 2601.17367)
 *   [ZH] "论文精读 - Elastic Attention" (Chinese reading notes; eqs. 4-5)
 *
 * Conventions shared by every entry point
 *   - Tensors are caller-owned device memory unless marked "host".  The library
 *     never allocates or frees device memory at run time; scratch space is the
 *     caller's workspace buffer.  State kept between calls, besides what lives
 *     in that workspace: per device, the fixed scratch array of
 *     ea_hybrid_attn_prefill_noalloc, the copy streams and events that
 *     ea_hybrid_attn_prefill_host creates on first use, and which kernels have
 *     had their shared-memory limits raised.
 *   - Element strides are given in ELEMENTS (not bytes), outermost first.  The
 *     innermost (head-dim) stride must be 1.
 *   - bf16 tensors are passed as void* to raw 16-bit bf16 storage.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *     entry points only enqueue work on it and return without synchronising.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     rejected call returns an error and enqueues nothing.  Conditions that
 *     only the device can see (a mode value read from device memory, a wait
 *     that ran out) set an error word in the workspace, which
 *     ea_check_errors() reads back.
 *   - Every function returns an ea_status; no exception or abort crosses the ABI.
 *   - ea_route, ea_hybrid_attn_prefill, ea_hybrid_attn_prefill_varlen,
 *     ea_hybrid_attn_decode and ea_xa_estimate enqueue kernels only (no
 *     allocation, no host synchronisation): after one call on the device
 *     (which raises the kernels' shared-memory limits), a call can be captured
 *     into a CUDA graph and replayed with new contents in the same buffers.
 */
#ifndef EA_H
#define EA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EA_OK = 0,
    EA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment      */
    EA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head dim != 128)  */
    EA_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned        */
    EA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                 */
    EA_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out                */
    EA_ERR_DEVICE_CHECK = 6   /* the device met an invalid mode / missing mask     */
} ea_status;

/* Per-KV-head kernel metadata m ([EN] §04 Deployment, Algorithm 1(b): the
 * routing decision r becomes metadata that each thread block branches on). */
typedef enum {
    EA_FULL = 0,   /* full causal attention, [EN] §02 eq. (1)                       */
    EA_SSA = 1,    /* streaming sparse attention: key j < sink or i - j < window,   */
                   /* [EN] §02 eq. (2), Glossary "SSA"                              */
    EA_BLOCK = 2   /* block-sparse attention over a caller-given 128x128 block mask */
                   /* (the compute half of XAttention), [EN] Glossary "XA"          */
} ea_mode;

/* How a routing decision maps to a mode: m = r ? sa_impl : fa_impl.
 * "FA-SSA" = {EA_FULL, EA_SSA}; "XA-SSA" = {EA_BLOCK, EA_SSA}
 * ([EN] §05 Experiments, "{retrieval}-{sparse}"). */
typedef struct {
    uint8_t fa_impl;
    uint8_t sa_impl;
} ea_policy;

/* Router MLP: n_layers dense layers, dims[0] = head dim ... dims[n_layers] = 2,
 * ReLU between layers (not after the last).  W[l] is a DEVICE pointer to a
 * row-major float32 [dims[l+1]][dims[l]] matrix, b[l] a DEVICE float32
 * [dims[l+1]] vector.  The struct and the dims/W/b pointer arrays are host
 * memory.  Limits: 1 <= n_layers <= 4, every dims[l] <= 1024. */
typedef struct {
    int n_layers;
    const int *dims;
    const float *const *W;
    const float *const *b;
} ea_mlp;

/* Human-readable name of a status code (static storage). */
const char *ea_status_string(ea_status s);

/*
 * ea_route - Attention Router pre-pass ([EN] §03 Method, "Method: the Attention
 * Router" and eq. 6; [ZH] §04 Method, "Router 怎么工作").
 *
 * For every (b, KV head h): mean-pool K over the first pool_head and last
 * pool_tail tokens (100 + 100 on the pages; a token in both ranges counts
 * once), run the MLP in fp64, take r = argmax of the two logits (ties -> 0 = FA)
 * and m = r ? policy.sa_impl : policy.fa_impl.
 *
 *   K          device bf16 [B][S][Hkv][d], element strides k_strides[4]
 *   r_out      device uint8 [B][Hkv]   routing decision (0 = FA, 1 = SA)
 *   m_out      device uint8 [B][Hkv]   kernel metadata (an ea_mode)
 *   logits_out device double [B][Hkv][2] or NULL
 *
 * Constraints: d == dims[0] <= 1024, pool_head + pool_tail >= 1, S >= 1.
 * Errors: EA_ERR_INVALID_ARG / EA_ERR_UNSUPPORTED on the host, EA_ERR_CUDA if
 * the launch fails.
 */
ea_status ea_route(const void *K, const int64_t k_strides[4], int B, int S, int Hkv, int d,
                   int pool_head, int pool_tail, const ea_mlp *mlp, ea_policy policy,
                   uint8_t *r_out, uint8_t *m_out, double *logits_out, void *stream);

/*
 * ea_route_layers - ea_route for L layers in one launch (all layers' routing
 * decisions of one input at once; the router reads only the boundary tokens,
 * so the whole pre-pass of a model is one short kernel).
 *
 *   K_layers   host array of L device pointers, layer l's K as in ea_route
 *              (all layers share k_strides, B, S, Hkv, d)
 *   mlps       host array of L ea_mlp (per-layer weights; same shapes rules)
 *   r_out, m_out  device uint8 [L][B][Hkv]; logits_out device double
 *              [L][B][Hkv][2] or NULL
 * Up to 64 layers take one kernel launch (more take one per 64 layers).
 * Limits: 1 <= L <= 1024.  Errors as for ea_route; every layer's arguments
 * are checked before anything is enqueued, so an error launches nothing.
 */
ea_status ea_route_layers(const void *const *K_layers, int L, const int64_t k_strides[4], int B,
                          int S, int Hkv, int d, int pool_head, int pool_tail, const ea_mlp *mlps,
                          ea_policy policy, uint8_t *r_out, uint8_t *m_out, double *logits_out,
                          void *stream);

/* Bytes of device workspace ea_hybrid_attn_prefill needs for these sizes
 * (0 on invalid sizes).  The workspace must be 256-byte aligned. */
size_t ea_prefill_workspace_size(int B, int S, int Hq, int Hkv, int d);

/*
 * ea_hybrid_attn_prefill - fused hybrid-head attention prefill of one layer
 * ([EN] §02 eqs. (1)-(3); §04 Deployment, Algorithm 1(b) and Figure 4).
 *
 * Query head qh uses KV head h = qh / (Hq / Hkv) and that head's mode m[b][h]:
 *   EA_FULL : key j kept for query i iff j <= i
 *   EA_SSA  : j <= i and (j < sink or i - j < window)
 *   EA_BLOCK: j <= i and block_mask[b][h][i / 128][j / 128] != 0
 * O[b][i][qh][:] = softmax over kept keys of scale * q_i . k_j, times V;
 * LSE[b][qh][i] = ln sum_kept exp(scale * q_i . k_j) (natural log).
 * A query with no kept key gets O = 0 and LSE = -inf.
 * All heads run in one persistent launch; each head's output is written in
 * place into its slice of O (eq. 3 concatenation, no copy).
 *
 *   Q            device bf16 [B][S][Hq][d],  element strides q_str[4]
 *   K, V         device bf16 [B][S][Hkv][d], element strides kv_str[4] (shared)
 *   O            device bf16 [B][S][Hq][d],  element strides o_str[4]
 *   LSE          device float [B][Hq][S] contiguous, or NULL
 *   m            device uint8 [B][Hkv] (ea_mode values)
 *   block_mask   device uint8 [B][Hkv][nB][nB], nB = ceil(S/128), row-major;
 *                entries above the diagonal are ignored.  May be NULL only if
 *                no head is EA_BLOCK (checked on the device).
 *   block_size   must be 128
 *   workspace    device, >= ea_prefill_workspace_size(...) bytes, 256-aligned;
 *                overwritten by the call.  Calls that share a workspace must
 *                be ordered on one stream.
 *   visited_bitmap  device uint32 or NULL.  When non-NULL, one bit per tile
 *                (b, h, qb, kb) at bit index ((b*Hkv + h)*nB + qb)*nB + kb is
 *                OR-ed in for every key tile the kernel visits; the caller
 *                zeroes it first.  A debugging aid for tile-skipping parity.
 *
 * Constraints: d == 128; Hq % Hkv == 0; 1 <= S <= 2^21;
 * sink >= 0; window >= 1; base pointers 16-byte aligned; q/kv/o strides of the
 * b, s and h dimensions multiples of 8 elements; head-dim stride 1.
 * Errors: EA_ERR_INVALID_ARG, EA_ERR_UNSUPPORTED, EA_ERR_WORKSPACE on the host;
 * EA_ERR_CUDA on a failed launch; device-side problems (mode value > 2,
 * BLOCK head with NULL block_mask, a bounded wait that ran out) are reported
 * by ea_check_errors(workspace).
 */
ea_status ea_hybrid_attn_prefill(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                 const int64_t q_str[4], const int64_t kv_str[4],
                                 const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                                 float scale, const uint8_t *m, int sink, int window,
                                 const uint8_t *block_mask, int block_size, void *workspace,
                                 size_t ws_bytes, uint32_t *visited_bitmap, void *stream);

/*
 * The two halves of ea_hybrid_attn_prefill, for callers that reuse one plan
 * (same m, block mask and sizes) across several launches, or that time the
 * attention kernel on its own.  ea_hybrid_attn_prefill == ea_prefill_plan
 * followed by ea_prefill_attend with the same arguments and workspace.
 *
 * ea_prefill_plan enqueues the planner: per (b, KV head, 128-query block) the
 * number of key tiles that hold at least one kept pair, then a longest-first
 * work queue of (block, query-head pair) items (rows of equal cost in no set
 * order; results do not depend on it), written to the workspace.  ea_prefill_attend enqueues the persistent attention kernel that
 * consumes that queue; it must follow a plan made with the same m,
 * block_mask, sink, window and sizes, on the same stream; one plan may feed
 * any number of ea_prefill_attend launches (the kernel re-arms the queue when
 * it has drained it).  Arguments,
 * constraints and errors are those of ea_hybrid_attn_prefill.
 */
ea_status ea_prefill_plan(int B, int S, int Hq, int Hkv, int d, const uint8_t *m, int sink,
                          int window, const uint8_t *block_mask, int block_size, void *workspace,
                          size_t ws_bytes, void *stream);

ea_status ea_prefill_attend(const void *Q, const void *K, const void *V, void *O, float *LSE,
                            const int64_t q_str[4], const int64_t kv_str[4],
                            const int64_t o_str[4], int B, int S, int Hq, int Hkv, int d,
                            float scale, const uint8_t *m, int sink, int window,
                            const uint8_t *block_mask, int block_size, void *workspace,
                            size_t ws_bytes, uint32_t *visited_bitmap, void *stream);

/* Bytes of device workspace ea_hybrid_attn_prefill_varlen needs (0 on
 * invalid sizes); 256-byte aligned like every workspace. */
size_t ea_prefill_varlen_workspace_size(int B, int total_tokens, int max_seqlen, int Hq, int Hkv,
                                        int d);

/*
 * ea_hybrid_attn_prefill_varlen - ea_hybrid_attn_prefill over a batch of
 * sequences of different lengths packed back to back (the layout of a serving
 * engine's prefill batch), in one launch.  Same attention and masks per
 * sequence as ea_hybrid_attn_prefill ([EN] §02 eqs. (1)-(3); §04 Deployment,
 * Algorithm 1(b)); no sequence attends to another.
 *
 *   Q, O         device bf16 [total_tokens][Hq][d], element strides q_str[3] /
 *                o_str[3] (token, head, dim)
 *   K, V         device bf16 [total_tokens][Hkv][d], strides kv_str[3]
 *   LSE          device float [Hq][total_tokens] contiguous, or NULL
 *   cu_seqlens   device int32 [B + 1]: sequence b is tokens
 *                [cu_seqlens[b], cu_seqlens[b + 1]) (cu_seqlens[0] >= 0,
 *                non-decreasing, cu_seqlens[B] <= total_tokens); a sequence of
 *                length 0 has no output
 *   max_seqlen   an upper bound on every sequence's length (<= 2^21)
 *   m            device uint8 [B][Hkv]
 *   block_mask   device uint8, per sequence b an [Hkv][nB_b][nB_b] block
 *                (nB_b = ceil(len_b / 128)), blocks of consecutive sequences
 *                back to back; NULL if no head is EA_BLOCK
 *   workspace    ea_prefill_varlen_workspace_size(...) bytes, 256-aligned
 * A sequence whose length is negative, above max_seqlen or runs past
 * total_tokens is skipped (no output) and reported by ea_check_errors, as are
 * the conditions ea_hybrid_attn_prefill reports there.  Other constraints and
 * host-side errors as ea_hybrid_attn_prefill.
 */
ea_status ea_hybrid_attn_prefill_varlen(const void *Q, const void *K, const void *V, void *O,
                                        float *LSE, const int64_t q_str[3],
                                        const int64_t kv_str[3], const int64_t o_str[3],
                                        const int32_t *cu_seqlens, int B, int total_tokens,
                                        int max_seqlen, int Hq, int Hkv, int d, float scale,
                                        const uint8_t *m, int sink, int window,
                                        const uint8_t *block_mask, int block_size,
                                        void *workspace, size_t ws_bytes, void *stream);

/*
 * Several layers in one launch.  The pages' single launch ([EN] §04
 * Deployment, Algorithm 1(b): the per-head routing metadata drives one kernel
 * whose grid is left intact, instead of the per-group launches of Algorithm
 * 1(a)) taken across layers: one planner over the rows of every layer, one
 * longest-first work queue mixing the layers, one persistent launch.  Per
 * layer the result is exactly ea_hybrid_attn_prefill's on that layer (the same
 * items, computed the same way; bit for bit).  Every layer has the same B, S,
 * head counts and strides (a transformer's layers).
 *
 * ea_prefill_layer describes one layer; every pointer is device memory laid
 * out as for ea_hybrid_attn_prefill (Q, K, V, O with the shared strides q_str,
 * kv_str, o_str; LSE [B][Hq][S] or NULL; m [B][Hkv]; block_mask
 * [B][Hkv][nB][nB] or NULL).  `layers` itself is a host array of n_layers
 * entries, read during the call.  n_layers is 1 .. EA_MAX_PREFILL_LAYERS
 * (more: EA_ERR_UNSUPPORTED); the workspace is
 * ea_prefill_layers_workspace_size(...) bytes (0: invalid sizes, or
 * B * n_layers above 65535).  Every layer is checked as ea_hybrid_attn_prefill
 * checks its arguments before anything is enqueued; device-side conditions
 * are reported by ea_check_errors(workspace).
 */
#define EA_MAX_PREFILL_LAYERS 48

typedef struct {
    const void *Q;
    const void *K;
    const void *V;
    void *O;
    float *LSE;
    const uint8_t *m;
    const uint8_t *block_mask;
} ea_prefill_layer;

size_t ea_prefill_layers_workspace_size(int n_layers, int B, int S, int Hq, int Hkv, int d);

ea_status ea_hybrid_attn_prefill_layers(const ea_prefill_layer *layers, int n_layers,
                                        const int64_t q_str[4], const int64_t kv_str[4],
                                        const int64_t o_str[4], int B, int S, int Hq, int Hkv,
                                        int d, float scale, int sink, int window, int block_size,
                                        void *workspace, size_t ws_bytes, void *stream);

/*
 * ea_hybrid_attn_prefill_noalloc - ea_hybrid_attn_prefill for callers that
 * cannot provide a workspace, e.g. an engine whose device memory is owned by
 * its own allocator and that forbids allocations once it is running, or a
 * latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation.  The pages have no counterpart of this entry point; it is
 * an interface convenience of this library.
 *
 * Same arguments, results and constraints as ea_hybrid_attn_prefill, minus the
 * workspace.  The planner's scratch lives in a fixed 4 MiB device array
 * inside the library (one per device that loads it, kept until the process
 * exits).  It holds the plan of any problem with
 * ea_prefill_workspace_size(B, S, Hq, Hkv, d) <= 4 MiB, i.e. about
 * B * Hkv * ceil(S / 128) * (4 + 4 * ceil(Hq / Hkv / 2)) bytes: with 32 query
 * heads over 8 KV heads, every length up to the 2^21 limit at B = 1 (1.6 MB),
 * and up to about 349K (b, KV head, 128-query block) rows in all (B = 2 at
 * S = 2^21 fits, B = 3 does not).  Larger problems, and every other invalid
 * argument, return an error without enqueueing anything.  Nothing is
 * allocated.
 *
 * The first call on a device looks up that array's device address (with the
 * device current) and caches it for the rest of the process; make that first
 * call before any stream capture.  A device reset between calls leaves the
 * cached address stale and is not supported.  Every call reuses the same array and clears its header first, so
 * calls whose executions overlap on the GPU (different streams, or different
 * host threads without ordering) race and must be serialised by the caller.
 * Device-side checks (invalid mode, missing block mask, a timed-out wait)
 * leave their error word in that internal array, which no entry point reads
 * back; diagnose such inputs with ea_hybrid_attn_prefill and a workspace.
 */
ea_status ea_hybrid_attn_prefill_noalloc(const void *Q, const void *K, const void *V, void *O,
                                         float *LSE, const int64_t q_str[4],
                                         const int64_t kv_str[4], const int64_t o_str[4], int B,
                                         int S, int Hq, int Hkv, int d, float scale,
                                         const uint8_t *m, int sink, int window,
                                         const uint8_t *block_mask, int block_size,
                                         uint32_t *visited_bitmap, void *stream);

/*
 * ea_prefill_host_buffer_size - bytes of device memory ea_hybrid_attn_prefill_host
 * needs for these sizes (0 on invalid sizes): room for Q, K, V, O, LSE, m, the
 * block mask when with_block_mask != 0, and the planner workspace.
 */
size_t ea_prefill_host_buffer_size(int B, int S, int Hq, int Hkv, int d, int with_block_mask);

/*
 * ea_hybrid_attn_prefill_host - ea_hybrid_attn_prefill on tensors in HOST
 * memory, with the host->device copies, the attention and the device->host
 * copies overlapped (same attention as [EN] §02 eqs. (1)-(3) and §04
 * Deployment, Algorithm 1(b)).
 *
 * Causal masks let query rows [q0, q1) start once the K/V rows below q1 are on
 * the device, under all three modes.  The call therefore cuts the sequence
 * into n_chunks runs of whole 128-query blocks.  Chunk c's Q/K/V rows are
 * copied up on an internal stream; its planner and attention run as soon as
 * they have arrived (even chunks on `stream`, odd chunks on an internal
 * compute stream, so that consecutive chunks overlap on the SMs); its O and
 * LSE rows are copied back on another internal stream while later chunks
 * compute.  The results equal
 * ea_hybrid_attn_prefill's bit for bit (each query block is computed by the
 * same kernel with the same key tiles in the same order).
 *
 *   Q_host       host bf16 [B][S][Hq][d] contiguous
 *   K_host, V_host  host bf16 [B][S][Hkv][d] contiguous
 *   O_host       host bf16 [B][S][Hq][d] contiguous (written)
 *   LSE_host     host float [B][Hq][S] contiguous (written), or NULL
 *   m_host       host uint8 [B][Hkv] (ea_mode values)
 *   block_mask_host  host uint8 [B][Hkv][nB][nB] as for ea_hybrid_attn_prefill,
 *                or NULL (then no head may be EA_BLOCK)
 *   device_buffer  device memory of ea_prefill_host_buffer_size(...) bytes
 *                (with_block_mask = block_mask_host != NULL), 256-byte
 *                aligned, owned by the caller; the call uses it as scratch
 *                and folds every device error word into the workspace at its
 *                start, so ea_check_errors(device_buffer, stream) reads them
 *                afterwards.
 *   n_chunks     0 = automatic (10, at most nB); otherwise 1 <= n_chunks <= 64.
 *                The chunks shrink toward the end of the sequence (chunk c ends
 *                near nB * (1 - (1 - (c + 1) / n_chunks)^1.25) query blocks),
 *                each holding at least one query block
 *                and <= nB.
 *   stream       the call's work is ordered after earlier work on `stream`,
 *                and later work on `stream` is ordered after all of it
 *                (including the last copy back).
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap the attention; pageable memory gives the same results
 * without the overlap.  The call is asynchronous: O_host and LSE_host hold the
 * results once `stream` has passed the call's work; the host buffers must stay
 * valid until then.  Calls that share a device_buffer must be ordered on one
 * stream.  Constraints and errors otherwise as ea_hybrid_attn_prefill (plus
 * EA_ERR_WORKSPACE for a missing, misaligned or short device_buffer); every
 * argument is checked before anything is enqueued.
 */
ea_status ea_hybrid_attn_prefill_host(const void *Q_host, const void *K_host, const void *V_host,
                                      void *O_host, float *LSE_host, int B, int S, int Hq, int Hkv,
                                      int d, float scale, const uint8_t *m_host, int sink,
                                      int window, const uint8_t *block_mask_host, int block_size,
                                      void *device_buffer, size_t buffer_bytes, int n_chunks,
                                      void *stream);

/* Bytes of device workspace ea_hybrid_attn_decode needs (0 on invalid sizes).
 * num_splits = 0 means the automatic choice; the same value must be passed to
 * ea_hybrid_attn_decode. */
size_t ea_decode_workspace_size(int B, int Hq, int Hkv, int d, int Lmax, int num_splits);

/*
 * ea_hybrid_attn_decode - one decode step of hybrid-head attention with the
 * routing decision fixed at prefill ([EN] §08 Commentary, stated limit ③:
 * routing happens once per request at the prefill stage).
 *
 * For sequence b with L = seqlens[b] cached tokens (the cache already holds
 * the current token) and query head qh (KV head h = qh / (Hq/Hkv)):
 *   EA_FULL : keys j in [0, L)
 *   EA_SSA  : keys j in [0, L) with j < sink or (L - 1) - j < window
 *   EA_BLOCK: keys j in [0, L) with block_mask[b][h][(L - 1) / 128][j / 128] != 0
 * i.e. exactly the keys the prefill's row L - 1 keeps under the same mode and
 * mask (the block mask chosen at prefill is reused across decode steps; the
 * pages give no other decode reading of it).
 * O[b][qh][:] = softmax(scale * q . k_j) V over those keys; LSE[b][qh] its
 * natural log-sum-exp.  L = 0, or no kept key, gives O = 0, LSE = -inf.  Work
 * is split along the key axis and merged by log-sum-exp.
 *
 *   q        device bf16 [B][Hq][d], element strides q_str[3]
 *   Kc, Vc   device bf16 [B][Lmax][Hkv][d], element strides kv_str[4] (shared)
 *   O        device bf16 [B][Hq][d], element strides o_str[3]
 *   LSE      device float [B][Hq] contiguous, or NULL
 *   seqlens  device int32 [B], each in [0, Lmax] (checked on the device)
 *   m        device uint8 [B][Hkv] (ea_mode values)
 *   block_mask  device uint8 [B][Hkv][nB][nB], nB = ceil(Lmax / 128), or NULL
 *            if no head is EA_BLOCK (a BLOCK head without a mask is reported
 *            by ea_check_errors); nB must not exceed 65535
 *   block_size  must be 128
 *   num_splits  0 = automatic, else 1..1024 key-axis splits per (b, KV head)
 *   workspace   device, >= ea_decode_workspace_size(...) bytes, 256-aligned
 *
 * Constraints: d == 128; Hq % Hkv == 0 and Hq / Hkv <= 8; sink >= 0;
 * window >= 1; 16-byte aligned base pointers; cache strides of b, position and
 * head dimensions multiples of 8 elements; head-dim strides 1.
 * Errors: as for the prefill.
 */
ea_status ea_hybrid_attn_decode(const void *q, const void *Kc, const void *Vc, void *O, float *LSE,
                                const int64_t q_str[3], const int64_t kv_str[4],
                                const int64_t o_str[3], const int32_t *seqlens, int B, int Hq,
                                int Hkv, int d, int Lmax, float scale, const uint8_t *m, int sink,
                                int window, const uint8_t *block_mask, int block_size,
                                int num_splits, void *workspace, size_t ws_bytes, void *stream);

/*
 * ea_hybrid_attn_decode_paged - ea_hybrid_attn_decode on a paged KV cache: the
 * cache rows live in fixed-size pages, and each sequence lists its pages in a
 * block table (the layout serving engines use to grow caches without copies).
 * Same attention, routing and results as ea_hybrid_attn_decode on the cache
 * the pages spell out; the pages have no counterpart of this entry point (it
 * is the decode of the same method over another cache layout).
 *
 *   K_pages, V_pages  device bf16 [num_pages][page_size][Hkv][d], element
 *                strides kv_str[4] (page, row, head, dim)
 *   block_table  device int32 [B][bt_stride]: key k of sequence b is row
 *                k % page_size of page block_table[b][k / page_size]; only the
 *                first ceil(seqlens[b] / page_size) entries of a row are read
 *   max_pages    pages per sequence at most (seqlens[b] <= max_pages * page_size)
 *   page_size    rows per page, a multiple of 64
 *   num_pages    pages in K_pages / V_pages; a table entry outside
 *                [0, num_pages) is reported by ea_check_errors and reads zeros
 *   block_mask   as for ea_hybrid_attn_decode with Lmax = max_pages * page_size
 *   workspace    ea_decode_workspace_size(B, Hq, Hkv, d, max_pages * page_size,
 *                num_splits) bytes
 * Other arguments, constraints and errors as ea_hybrid_attn_decode; invalid
 * table sizes return EA_ERR_INVALID_ARG, a page size that is not a positive
 * multiple of 64 EA_ERR_UNSUPPORTED.
 */
ea_status ea_hybrid_attn_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                                      void *O, float *LSE, const int64_t q_str[3],
                                      const int64_t kv_str[4], const int64_t o_str[3],
                                      const int32_t *block_table, int64_t bt_stride, int max_pages,
                                      int page_size, int num_pages, const int32_t *seqlens, int B,
                                      int Hq, int Hkv, int d, float scale, const uint8_t *m,
                                      int sink, int window, const uint8_t *block_mask,
                                      int block_size, int num_splits, void *workspace,
                                      size_t ws_bytes, void *stream);

/*
 * ea_xa_estimate - XA block-mask estimation for the EA_BLOCK heads: scores each
 * 128 x 128 block of every BLOCK head by antidiagonal scoring and keeps the
 * smallest set of blocks per query-block row that holds `threshold` of the
 * row's score.  The pages name XAttention's antidiagonal scoring as XA's way of
 * choosing key blocks ([EN] Glossary "XA"; [ZH] glossary "XA") with stride 16
 * and threshold 0.9 ([EN] §07 Table 8, "stride/threshold 16/0.9"), without
 * writing the scoring out; this computes the following reading of it.
 *
 * With s = stride, cell (a, c) holds queries a*s .. a*s+s-1 and keys
 * c*s .. c*s+s-1, and for every query head qh of the KV head h:
 *   A[a][c]   = (scale / s) * sum_{u<s} q[a*s+u] . k[c*s+s-1-u]    (antidiagonal mean)
 *   P[a][c]   = softmax over cells c <= a of A[a][c]
 *   W[qb][kb] = sum over the group's query heads and the cells of block
 *               (qb, kb) (cell rows a*s in qb, cell columns c*s in kb) of P
 * Row qb of the mask keeps the fewest key blocks kb <= qb, highest W first
 * (equal W: lower kb first), whose W add up to at least threshold times the
 * row's total (all blocks with W > 0 if rounding leaves every run short), plus
 * the diagonal block; every other entry is 0.  Rows of heads whose mode is not
 * EA_BLOCK are not written.
 *
 *   Q            device bf16 [B][S][Hq][d],  element strides q_str[4]
 *   K            device bf16 [B][S][Hkv][d], element strides k_str[4]
 *   m            device uint8 [B][Hkv] (ea_mode values)
 *   stride       must be 16;  S must be a multiple of it
 *   threshold    in [0, 1] (the pages' value is 0.9)
 *   block_size   must be 128 (the fused prefill's mask granularity)
 *   max_units    upper bound on the number of (b, h) with m == EA_BLOCK; more
 *                raise EA_DEVERR_CHECK (ea_check_errors) and the extra heads'
 *                rows are not written
 *   block_mask   device uint8 [B][Hkv][nB][nB] (output), nB = S / 128 rounded up
 *   block_scores device float [B][Hkv][nB][nB] (output, W; 0 above the
 *                diagonal), or NULL
 *   workspace    device, >= ea_xa_workspace_size(...) bytes, 256-aligned
 *
 * Three stream-ordered launches (unit list, antidiagonal score pass on the
 * tensor cores, selection); no host synchronisation.  Results do not depend on
 * which CTA ran which work item.
 * Constraints: d == 128; Hq % Hkv == 0 and Hq / Hkv <= 64; 16 <= S <= 2^21;
 * base pointers 16-byte aligned; strides of the b, s and h dimensions multiples
 * of 8 elements, head-dim stride 1.
 * Errors: EA_ERR_INVALID_ARG, EA_ERR_UNSUPPORTED, EA_ERR_WORKSPACE on the host;
 * EA_ERR_CUDA on a failed launch; device-side problems via ea_check_errors.
 */
size_t ea_xa_workspace_size(int B, int S, int Hq, int Hkv, int d, int stride, int max_units);
ea_status ea_xa_estimate(const void *Q, const void *K, const int64_t q_str[4],
                         const int64_t k_str[4], int B, int S, int Hq, int Hkv, int d, float scale,
                         const uint8_t *m, int stride, float threshold, int block_size,
                         int max_units, uint8_t *block_mask, float *block_scores, void *workspace,
                         size_t ws_bytes, void *stream);

/*
 * ea_sparsity_ratios - model sparsity ratio and effective sparsity ratio of one
 * input over L layers ([ZH] §02 Background, eqs. (4)-(5); [EN] §02).  HOST
 * function; all pointers are host memory; nothing touches the GPU.
 *
 *   Omega_MSR = (1/(L Hkv)) sum_{l,h} [r[l][h] == 1]
 *   Omega_ESR = (1/(L Hkv)) sum_{l,h} rho(l,h)
 * where rho is the share of the S(S+1)/2 causal (query, key) pairs that the
 * head's executed mode m[l][h] prunes (0 for EA_FULL, and e.g. 0.9 when 10%
 * are kept).  Since all heads share the causal count, the result is computed
 * as one division of exact integer pair counts, i.e. correctly rounded.
 *
 *   r, m         host uint8 [L][Hkv]
 *   block_masks  host array of L pointers, each to uint8 [Hkv][nB][nB], or
 *                NULL; required for layers holding EA_BLOCK heads
 *   block_size   must be 128 when a mask is read
 * Errors: EA_ERR_INVALID_ARG (null output, r > 1, m > 2, BLOCK without mask,
 * S < 1).
 */
ea_status ea_sparsity_ratios(const uint8_t *r, const uint8_t *m, int L, int Hkv, int S, int sink,
                             int window, const uint8_t *const *block_masks, int block_size,
                             double *omega_msr, double *omega_esr);

/*
 * ea_check_errors - synchronise `stream`, then read and clear the device error
 * word at the start of a prefill, decode or XA workspace.  Returns EA_OK,
 * EA_ERR_DEVICE_CHECK (an invalid device-side argument, or, in the
 * bounds-checked build of the library, an index found out of range and not
 * used), EA_ERR_TIMEOUT, or EA_ERR_CUDA.  This is the only entry point that
 * blocks the host.
 */
ea_status ea_check_errors(void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EA_H */
