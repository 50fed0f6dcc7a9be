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
constexpr int kRouterThreads = 256;

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

// Pool, MLP and argmax of one (b, KV head); the whole CTA takes part.
__device__ __forceinline__ void route_one(const __nv_bfloat16 *__restrict__ K, int64_t sb, int64_t ss,
                                          int64_t sh, int S, int Hkv, int d, int pool_head,
                                          int pool_tail, const RouterMlp &mlp, uint8_t fa_impl,
                                          uint8_t sa_impl, int b, int h, uint8_t *__restrict__ r_out,
                                          uint8_t *__restrict__ m_out, double *__restrict__ logits_out,
                                          double *xbuf, double *ybuf)
{
    const int head_end = pool_head < S ? pool_head : S;
    const int tail_begin = (S - pool_tail) > head_end ? (S - pool_tail) : head_end;
    const int count = head_end + (S - tail_begin);

    // 1. boundary mean pooling; a sum of bf16 values in fp64 is exact here, so
    //    the token order does not matter.
    const __nv_bfloat16 *base = K + b * sb + h * sh;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        double acc = 0.0;
        for (int t = 0; t < head_end; ++t)
            acc = __dadd_rn(acc, static_cast<double>(__bfloat162float(base[t * ss + c])));
        for (int t = tail_begin; t < S; ++t)
            acc = __dadd_rn(acc, static_cast<double>(__bfloat162float(base[t * ss + c])));
        xbuf[c] = __ddiv_rn(acc, static_cast<double>(count));
    }
    __syncthreads();

    // 2. dense layers with ReLU between them
    double *x = xbuf, *y = ybuf;
    for (int l = 0; l < mlp.n_layers; ++l) {
        const int nin = mlp.dims[l], nout = mlp.dims[l + 1];
        const float *W = mlp.W[l];
        for (int o = threadIdx.x; o < nout; o += blockDim.x) {
            double acc = static_cast<double>(mlp.b[l][o]);
            for (int c = 0; c < nin; ++c)
                acc = __dadd_rn(acc, __dmul_rn(static_cast<double>(W[o * nin + c]), x[c]));
            if (l + 1 < mlp.n_layers && !(acc > 0.0))
                acc = 0.0;
            y[o] = acc;
        }
        __syncthreads();
        double *t = x;
        x = y;
        y = t;
    }

    // 3. hard routing: first maximum wins a tie (0 = FA)
    if (threadIdx.x == 0) {
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
    __shared__ double xbuf[kRouterMaxDim];
    __shared__ double ybuf[kRouterMaxDim];
    route_one(K, sb, ss, sh, S, Hkv, d, pool_head, pool_tail, mlp, fa_impl, sa_impl, blockIdx.y,
              blockIdx.x, r_out, m_out, logits_out, xbuf, ybuf);
}

// grid (Hkv, B, layers of this launch); layer z writes its [B][Hkv] block.
__global__ void __launch_bounds__(kRouterThreads)
    router_layers_kernel(const RouterLayers layers, int64_t sb, int64_t ss, int64_t sh, int S,
                         int B, int Hkv, int d, int pool_head, int pool_tail, uint8_t fa_impl,
                         uint8_t sa_impl, uint8_t *__restrict__ r_out, uint8_t *__restrict__ m_out,
                         double *__restrict__ logits_out)
{
    __shared__ double xbuf[kRouterMaxDim];
    __shared__ double ybuf[kRouterMaxDim];
    const int z = blockIdx.z;
    const int64_t off = static_cast<int64_t>(z) * B * Hkv;
    route_one(layers.K[z], sb, ss, sh, S, Hkv, d, pool_head, pool_tail, layers.mlp[z], fa_impl,
              sa_impl, blockIdx.y, blockIdx.x, r_out + off, m_out + off,
              logits_out ? logits_out + 2 * off : nullptr, xbuf, ybuf);
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
    for (int l0 = 0; l0 < L; l0 += kRouterLayersPerLaunch) {
        const int n = L - l0 < kRouterLayersPerLaunch ? L - l0 : kRouterLayersPerLaunch;
        RouterLayers layers{};
        for (int z = 0; z < n; ++z) {
            check_mlp(&mlps[l0 + z], d, layers.mlp[z]);
            layers.K[z] = static_cast<const __nv_bfloat16 *>(K_layers[l0 + z]);
        }
        const int64_t off = static_cast<int64_t>(l0) * B * Hkv;
        router_layers_kernel<<<dim3(Hkv, B, n), kRouterThreads, 0, st>>>(
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
    dim3 grid(Hkv, B);
    router_kernel<<<grid, kRouterThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(K), k_strides[0], k_strides[1], k_strides[2], S, Hkv, d,
        pool_head, pool_tail, p, policy.fa_impl, policy.sa_impl, r_out, m_out, logits_out);
    return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}
