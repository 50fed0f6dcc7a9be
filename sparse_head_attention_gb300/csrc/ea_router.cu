// ea_router.cu - Attention Router pre-pass: boundary mean pooling of K per KV
// head, a small dense MLP, and hard routing by argmax.
//
// "Paper Reading - Elastic Attention" (English notes), §03 Method, "Method: the
// Attention Router" and eq. 6; "论文精读 - Elastic Attention" (Chinese notes),
// §04 Method, "Router 怎么工作": the router pools the key states over the first
// and last 100 tokens of the sequence, runs a Task MLP and a Router MLP to get
// two logits per KV head, and takes the arg max (0 = FA, 1 = SA).
//
// One CTA per (b, KV head).  The pooling reads only the boundary tokens, so the
// cost does not grow with the sequence length.  Pooling and the MLP run in
// fp64 with every multiply and add rounded separately (no fused multiply-add)
// and in index order, so the decision is reproducible and its margin can be
// checked on the host.
#include <cuda_runtime.h>

#include "ea_device.cuh"
#include "ea_internal.h"

namespace ea {

constexpr int kRouterMaxLayers = 4;
constexpr int kRouterMaxDim = 1024;
constexpr int kRouterThreads = 512;
// Dynamic shared memory: the bf16 boundary rows while pooling, then the fp64
// products of one MLP layer (72 KB holds 200 x 128 rows, or 141 x 64 products).
constexpr int kRouterStageBytes = 72 * 1024;
constexpr int kStageElems = kRouterStageBytes / 2;
constexpr int kStageDoubles = kRouterStageBytes / 8;
// Channels one thread carries through the pooling when d > blockDim.
constexpr int kChansPerThread = kRouterMaxDim / kRouterThreads;

struct RouterMlp {
    int n_layers;
    int dims[kRouterMaxLayers + 1];
    const float *W[kRouterMaxLayers];
    const float *b[kRouterMaxLayers];
};

// Model layers routed by one launch of router_layers_kernel.  The layers'
// pointers and MLPs travel as kernel parameters (about 6 KB for 64 layers,
// inside the 32 KB parameter space of sm_70 and later), so one launch needs
// no device-side table; deeper models take one more launch per 64 layers.
constexpr int kRouterLayersPerLaunch = 64;

struct RouterLayers {
    const __nv_bfloat16 *K[kRouterLayersPerLaunch];
    RouterMlp mlp[kRouterLayersPerLaunch];
};
static_assert(sizeof(RouterLayers) < 16 * 1024, "router kernel parameters");

struct RouterSmem {
    double x[kRouterMaxDim];
    double y[kRouterMaxDim];
    long long red_acc[kRouterThreads];      // per (row group, channel)
    int red_min[kRouterThreads];
    int red_max[kRouterThreads];
    int red_special[kRouterThreads];
    int ch_emin[kRouterMaxDim];             // per channel: smallest exponent
    int ch_exact[kRouterMaxDim];            // per channel: 1 = integer sum is exact
};

// fp64 arithmetic is slow on this part: a dependent add costs about 64 cycles
// and an SM retires under two fp64 operations per cycle.  The router keeps the
// fp64 rounding of a plain sequential evaluation (so logits are reproducible
// bit for bit) but moves every step that has an exact cheaper form off the
// fp64 pipe.
//
// Pooling.  A finite bf16 value is sig * 2^e with an integer sig < 256
// (sig = 128 + mantissa, e = E - 134 for E > 0; sig = mantissa, e = -133 for
// subnormals).  Over one channel's pooled values let emin and emax be the
// smallest and largest e of a nonzero value.  Every term is an integer
// multiple of 2^emin below 2^(8 + emax - emin) * 2^emin, so if
// ceil(log2(count)) + 8 + (emax - emin) <= 53, every partial sum, in any
// order, is an integer multiple of 2^emin below 2^53 * 2^emin in magnitude
// and is exact in fp64.  The sequential fp64 sum then equals the exact integer
// sum, which the integer pipe adds in any order.  Channels outside that
// bound, or holding an infinity or NaN, are summed in sequential fp64.
__device__ __forceinline__ int bf16_exponent(uint32_t u)   // e of a nonzero finite value
{
    const int E = static_cast<int>((u >> 7) & 0xFFu);
    return (E ? E : 1) - 134;
}

// float -> double by assembling the bits (exact for normal numbers) on the
// integer pipe; zero, subnormal, infinite and NaN inputs take the conversion
// instruction.
__device__ __forceinline__ double f32_to_f64(float w)
{
    const uint32_t u = __float_as_uint(w);
    const uint32_t E = (u >> 23) & 0xFFu;
    if (E == 0u || E == 0xFFu)
        return static_cast<double>(w);
    const unsigned long long bits = (static_cast<unsigned long long>(u >> 31) << 63) |
                                    (static_cast<unsigned long long>(E + 896u) << 52) |
                                    (static_cast<unsigned long long>(u & 0x7FFFFFu) << 29);
    return __longlong_as_double(static_cast<long long>(bits));
}

// Copy pooled positions [p0, p0 + rows) of one (b, head) into the stage.
__device__ __forceinline__ void stage_rows(const __nv_bfloat16 *__restrict__ base, int64_t ss, int d,
                                           bool vec, int p0, int rows, int head_end,
                                           int tail_begin, __nv_bfloat16 *stage)
{
    if (vec) {
        const int per_row = d / 8;
        const int n = rows * per_row;
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int pr = i / per_row, c8 = i - pr * per_row;
            const int p = p0 + pr;
            const int t = p < head_end ? p : tail_begin + (p - head_end);
            reinterpret_cast<uint4 *>(stage)[i] =
                __ldg(reinterpret_cast<const uint4 *>(base + t * ss) + c8);
        }
    } else {
        const int n = rows * d;
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int pr = i / d, c = i - pr * d;
            const int p = p0 + pr;
            const int t = p < head_end ? p : tail_begin + (p - head_end);
            stage[i] = base[t * ss + c];
        }
    }
}

// Pool, MLP and argmax of one (b, KV head); the whole CTA takes part.
__device__ __forceinline__ void route_one(const __nv_bfloat16 *__restrict__ K, int64_t sb, int64_t ss,
                                          int64_t sh, int S, int Hkv, int d, int pool_head,
                                          int pool_tail, const RouterMlp &mlp, uint8_t fa_impl,
                                          uint8_t sa_impl, int b, int h, uint8_t *__restrict__ r_out,
                                          uint8_t *__restrict__ m_out, double *__restrict__ logits_out,
                                          RouterSmem &sm, unsigned char *dyn)
{
    const int head_end = pool_head < S ? pool_head : S;
    const int tail_begin = (S - pool_tail) > head_end ? (S - pool_tail) : head_end;
    const int count = head_end + (S - tail_begin);
    const int tid = static_cast<int>(threadIdx.x), nthr = static_cast<int>(blockDim.x);

    // 1. boundary mean pooling over pooled positions p = 0 .. count-1 (the
    //    head tokens, then the tail tokens).  Thread (part, c) takes channel c
    //    of rows part, part + parts, ... of each staged pass.
    __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(dyn);
    const uint16_t *stage16 = reinterpret_cast<const uint16_t *>(dyn);
    const __nv_bfloat16 *base = K + b * sb + h * sh;
    const bool vec = (d % 8) == 0 && (ss % 8) == 0 &&
                     (reinterpret_cast<uintptr_t>(base) & 15u) == 0;
    const int rows_per_pass = kStageElems / d;
    const int n_pass = (count + rows_per_pass - 1) / rows_per_pass;
    const int parts = d < nthr ? nthr / d : 1;
    const int part = tid / d;                    // 0 for every thread when parts == 1
    const int c_first = parts > 1 ? tid - part * d : tid;
    const int n_ch = parts > 1 ? 1 : kChansPerThread;
    const bool active = part < parts;

    // pass A: exponent range and infinities / NaNs per channel
    int emin[kChansPerThread], emax[kChansPerThread], special[kChansPerThread];
#pragma unroll
    for (int j = 0; j < kChansPerThread; ++j) {
        emin[j] = 1 << 20;
        emax[j] = -(1 << 20);
        special[j] = 0;
    }
    for (int q = 0; q < n_pass; ++q) {
        const int p0 = q * rows_per_pass;
        const int rows = count - p0 < rows_per_pass ? count - p0 : rows_per_pass;
        stage_rows(base, ss, d, vec, p0, rows, head_end, tail_begin, stage);
        __syncthreads();
        if (active) {
#pragma unroll
            for (int j = 0; j < kChansPerThread; ++j) {
                const int c = c_first + j * nthr;
                if (j >= n_ch || c >= d)
                    continue;
#pragma unroll 4
                for (int r = part; r < rows; r += parts) {
                    const uint32_t u = stage16[r * d + c];
                    const bool nz = (u & 0x7FFFu) != 0;
                    const int e = bf16_exponent(u);
                    emin[j] = nz ? min(emin[j], e) : emin[j];
                    emax[j] = nz ? max(emax[j], e) : emax[j];
                    special[j] |= ((u >> 7) & 0xFFu) == 0xFFu;
                }
            }
        }
        if (n_pass > 1)
            __syncthreads();              // the stage is refilled next pass
    }
    const int lg_count = count > 1 ? 32 - __clz(count - 1) : 0;
    if (parts > 1) {
        if (active) {
            sm.red_min[tid] = emin[0];
            sm.red_max[tid] = emax[0];
            sm.red_special[tid] = special[0];
        }
        __syncthreads();
        if (tid < d) {
            int mn = sm.red_min[tid], mx = sm.red_max[tid], sp = sm.red_special[tid];
            for (int q = 1; q < parts; ++q) {
                mn = min(mn, sm.red_min[q * d + tid]);
                mx = max(mx, sm.red_max[q * d + tid]);
                sp |= sm.red_special[q * d + tid];
            }
            sm.ch_emin[tid] = mn;
            sm.ch_exact[tid] = !sp && (mx < mn || lg_count + 8 + (mx - mn) <= 53);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kChansPerThread; ++j) {
            const int c = tid + j * nthr;
            if (c < d) {
                sm.ch_emin[c] = emin[j];
                sm.ch_exact[c] = !special[j] &&
                                 (emax[j] < emin[j] || lg_count + 8 + (emax[j] - emin[j]) <= 53);
            }
        }
    }
    __syncthreads();

    // pass B: integer sums of the exact channels
    long long acc[kChansPerThread];
    int cmin[kChansPerThread];
    bool cexact[kChansPerThread];
#pragma unroll
    for (int j = 0; j < kChansPerThread; ++j) {
        acc[j] = 0;
        const int c = c_first + j * nthr;
        const bool ok = active && j < n_ch && c < d;
        cmin[j] = ok ? sm.ch_emin[c] : 0;
        cexact[j] = ok && sm.ch_exact[c];
    }
    for (int q = 0; q < n_pass; ++q) {
        const int p0 = q * rows_per_pass;
        const int rows = count - p0 < rows_per_pass ? count - p0 : rows_per_pass;
        if (n_pass > 1) {
            stage_rows(base, ss, d, vec, p0, rows, head_end, tail_begin, stage);
            __syncthreads();
        }
#pragma unroll
        for (int j = 0; j < kChansPerThread; ++j) {
            if (!cexact[j])
                continue;
            const int c = c_first + j * nthr;
#pragma unroll 4
            for (int r = part; r < rows; r += parts) {
                const uint32_t u = stage16[r * d + c];
                const uint32_t E = (u >> 7) & 0xFFu;
                const unsigned long long sig = E ? ((u & 0x7Fu) | 0x80u) : (u & 0x7Fu);
                const int shl = sig ? bf16_exponent(u) - cmin[j] : 0;
                const long long term = static_cast<long long>(sig << shl);
                acc[j] += (u & 0x8000u) ? -term : term;
            }
        }
        if (n_pass > 1)
            __syncthreads();
    }
    if (parts > 1) {
        if (active)
            sm.red_acc[tid] = acc[0];
        __syncthreads();
        if (tid < d)
            for (int q = 1; q < parts; ++q)
                acc[0] += sm.red_acc[q * d + tid];
    }
#pragma unroll
    for (int j = 0; j < kChansPerThread; ++j) {
        const int c = tid + j * nthr;                  // owner: part 0
        if (c >= d || (parts > 1 && j > 0))
            continue;
        double sum;
        if (sm.ch_exact[c]) {
            // |acc| < 2^53 converts exactly; a nonzero sum has emin >= -133,
            // so 2^emin is a normal double and the scaling is exact
            sum = acc[j] == 0 ? 0.0
                              : __dmul_rn(__ll2double_rn(acc[j]),
                                          __longlong_as_double(
                                              static_cast<long long>(sm.ch_emin[c] + 1023) << 52));
        } else {
            sum = 0.0;
            for (int p = 0; p < count; ++p) {
                const int t = p < head_end ? p : tail_begin + (p - head_end);
                sum = __dadd_rn(sum, static_cast<double>(__bfloat162float(base[t * ss + c])));
            }
        }
        sm.x[c] = __ddiv_rn(sum, static_cast<double>(count));
    }
    __syncthreads();

    // 2. dense layers with ReLU between them.  All threads form the products
    //    W[o][c] * x[c] in shared memory (spreading the fp64 multiplies over
    //    every warp); the owner of output o then adds them to its bias in
    //    input order.  Products of a pass are stored [c][o] with a row stride
    //    of nout + 1, so that both the writes and the owners' reads avoid bank
    //    conflicts.  Owners sit one per warp when the layer is narrow.
    double *prod = reinterpret_cast<double *>(dyn);
    double *x = sm.x, *y = sm.y;
    for (int l = 0; l < mlp.n_layers; ++l) {
        const int nin = mlp.dims[l], nout = mlp.dims[l + 1];
        const float *__restrict__ W = mlp.W[l];
        const float *__restrict__ bias = mlp.b[l];
        const int cols = kStageDoubles / (nout + 1) < nin ? kStageDoubles / (nout + 1) : nin;
        const bool spread = nout * 32 <= nthr;         // one owner per warp
        for (int c0 = 0; c0 < nin; c0 += cols) {
            const int nc = nin - c0 < cols ? nin - c0 : cols;
            const int n = nc * nout;
            for (int i = tid; i < n; i += nthr) {
                const int o = i / nc, cc = i - o * nc;
                prod[cc * (nout + 1) + o] =
                    __dmul_rn(f32_to_f64(__ldg(W + static_cast<int64_t>(o) * nin + c0 + cc)), x[c0 + cc]);
            }
            __syncthreads();
            for (int o = spread ? (tid % 32 == 0 ? tid / 32 : nout) : tid; o < nout;
                 o += spread ? nout : nthr) {
                double a = c0 == 0 ? static_cast<double>(__ldg(bias + o)) : y[o];
#pragma unroll 8
                for (int cc = 0; cc < nc; ++cc)
                    a = __dadd_rn(a, prod[cc * (nout + 1) + o]);
                if (c0 + nc == nin && l + 1 < mlp.n_layers && !(a > 0.0))
                    a = 0.0;
                y[o] = a;
            }
            __syncthreads();
        }
        double *t = x;
        x = y;
        y = t;
    }

    // 3. hard routing: first maximum wins a tie (0 = FA)
    if (tid == 0) {
        const int u = b * Hkv + h;
        const int dec = x[1] > x[0] ? 1 : 0;
        r_out[u] = static_cast<uint8_t>(dec);
        m_out[u] = dec ? sa_impl : fa_impl;
        if (logits_out) {
            logits_out[2 * u + 0] = x[0];
            logits_out[2 * u + 1] = x[1];
        }
    }
}

__global__ void __launch_bounds__(kRouterThreads)
    router_kernel(const __nv_bfloat16 *__restrict__ K, int64_t sb, int64_t ss, int64_t sh, int S,
                  int Hkv, int d, int pool_head, int pool_tail, RouterMlp mlp, uint8_t fa_impl,
                  uint8_t sa_impl, uint8_t *__restrict__ r_out, uint8_t *__restrict__ m_out,
                  double *__restrict__ logits_out)
{
    __shared__ RouterSmem sm;
    extern __shared__ __align__(16) unsigned char dyn[];
    route_one(K, sb, ss, sh, S, Hkv, d, pool_head, pool_tail, mlp, fa_impl, sa_impl, blockIdx.y,
              blockIdx.x, r_out, m_out, logits_out, sm, dyn);
}

// grid (Hkv, B, layers of this launch); layer z writes its [B][Hkv] block.
__global__ void __launch_bounds__(kRouterThreads)
    router_layers_kernel(const RouterLayers layers, int64_t sb, int64_t ss, int64_t sh, int S,
                         int B, int Hkv, int d, int pool_head, int pool_tail, uint8_t fa_impl,
                         uint8_t sa_impl, uint8_t *__restrict__ r_out, uint8_t *__restrict__ m_out,
                         double *__restrict__ logits_out)
{
    __shared__ RouterSmem sm;
    extern __shared__ __align__(16) unsigned char dyn[];
    const int z = blockIdx.z;
    const int64_t off = static_cast<int64_t>(z) * B * Hkv;
    route_one(layers.K[z], sb, ss, sh, S, Hkv, d, pool_head, pool_tail, layers.mlp[z], fa_impl,
              sa_impl, blockIdx.y, blockIdx.x, r_out + off, m_out + off,
              logits_out ? logits_out + 2 * off : nullptr, sm, dyn);
}

// Both router kernels take kRouterStageBytes of dynamic shared memory (set
// once per device).
static cudaError_t router_prepare()
{
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kRouterStageBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(router_layers_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterStageBytes);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            attr_done[dev] = true;
    }
    return cudaSuccess;
}

} // namespace ea

using namespace ea;

// Host checks shared by ea_route and ea_route_layers; fills the by-value MLP.
static ea_status check_mlp(const ea_mlp *mlp, int d, RouterMlp &p)
{
    if (!mlp || !mlp->dims || !mlp->W || !mlp->b)
        return EA_ERR_INVALID_ARG;
    if (mlp->n_layers < 1 || mlp->n_layers > kRouterMaxLayers || d > kRouterMaxDim)
        return EA_ERR_UNSUPPORTED;
    p = RouterMlp{};
    p.n_layers = mlp->n_layers;
    for (int l = 0; l <= mlp->n_layers; ++l) {
        p.dims[l] = mlp->dims[l];
        if (p.dims[l] < 1 || p.dims[l] > kRouterMaxDim)
            return EA_ERR_UNSUPPORTED;
    }
    if (p.dims[0] != d || p.dims[mlp->n_layers] != 2)
        return EA_ERR_INVALID_ARG;
    for (int l = 0; l < mlp->n_layers; ++l) {
        if (!mlp->W[l] || !mlp->b[l])
            return EA_ERR_INVALID_ARG;
        p.W[l] = mlp->W[l];
        p.b[l] = mlp->b[l];
    }
    return EA_OK;
}

extern "C" ea_status ea_route_layers(const void *const *K_layers, int L, const int64_t k_strides[4],
                                     int B, int S, int Hkv, int d, int pool_head, int pool_tail,
                                     const ea_mlp *mlps, ea_policy policy, uint8_t *r_out,
                                     uint8_t *m_out, double *logits_out, void *stream)
{
    if (!K_layers || !k_strides || !mlps || !r_out || !m_out || L < 1 || L > 1024)
        return EA_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || Hkv < 1 || d < 1 || pool_head < 0 || pool_tail < 0 ||
        pool_head + pool_tail < 1 || B > 65535 || Hkv > 65535)
        return EA_ERR_INVALID_ARG;
    if (k_strides[3] != 1 || policy.fa_impl > EA_BLOCK || policy.sa_impl > EA_BLOCK)
        return EA_ERR_INVALID_ARG;
    // every layer is checked before the first launch, so a bad argument
    // enqueues nothing
    for (int l = 0; l < L; ++l) {
        if (!K_layers[l])
            return EA_ERR_INVALID_ARG;
        RouterMlp p;
        const ea_status e = check_mlp(&mlps[l], d, p);
        if (e != EA_OK)
            return e;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (router_prepare() != cudaSuccess)
        return EA_ERR_CUDA;
    for (int l0 = 0; l0 < L; l0 += kRouterLayersPerLaunch) {
        const int n = L - l0 < kRouterLayersPerLaunch ? L - l0 : kRouterLayersPerLaunch;
        RouterLayers layers{};
        for (int z = 0; z < n; ++z) {
            check_mlp(&mlps[l0 + z], d, layers.mlp[z]);
            layers.K[z] = static_cast<const __nv_bfloat16 *>(K_layers[l0 + z]);
        }
        const int64_t off = static_cast<int64_t>(l0) * B * Hkv;
        router_layers_kernel<<<dim3(Hkv, B, n), kRouterThreads, kRouterStageBytes, st>>>(
            layers, k_strides[0], k_strides[1], k_strides[2], S, B, Hkv, d, pool_head, pool_tail,
            policy.fa_impl, policy.sa_impl, r_out + off, m_out + off,
            logits_out ? logits_out + 2 * off : nullptr);
        if (cudaGetLastError() != cudaSuccess)
            return EA_ERR_CUDA;
    }
    return EA_OK;
}

extern "C" ea_status ea_route(const void *K, const int64_t k_strides[4], int B, int S, int Hkv, int d,
                              int pool_head, int pool_tail, const ea_mlp *mlp, ea_policy policy,
                              uint8_t *r_out, uint8_t *m_out, double *logits_out, void *stream)
{
    if (!K || !k_strides || !mlp || !r_out || !m_out)
        return EA_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || Hkv < 1 || d < 1 || pool_head < 0 || pool_tail < 0 ||
        pool_head + pool_tail < 1)
        return EA_ERR_INVALID_ARG;
    if (k_strides[3] != 1 || policy.fa_impl > EA_BLOCK || policy.sa_impl > EA_BLOCK)
        return EA_ERR_INVALID_ARG;
    RouterMlp p{};
    const ea_status e = check_mlp(mlp, d, p);
    if (e != EA_OK)
        return e;
    if (router_prepare() != cudaSuccess)
        return EA_ERR_CUDA;
    dim3 grid(Hkv, B);
    router_kernel<<<grid, kRouterThreads, kRouterStageBytes, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(K), k_strides[0], k_strides[1], k_strides[2], S, Hkv, d,
        pool_head, pool_tail, p, policy.fa_impl, policy.sa_impl, r_out, m_out, logits_out);
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}
