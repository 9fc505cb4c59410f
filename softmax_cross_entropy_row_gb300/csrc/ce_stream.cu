// Streaming path for rows too large for a cluster's shared memory.
//
// Pass A: CTA (k, b) holds chunk k of row b in registers (16 elements per
// thread, coalesced loads) and writes the chunk's (M_k, S_k) -- Steps 1 and 2
// of Pass 1 of rumus 0.1.1's cross_entropy.wgsl over the chunk -- plus the
// target logit if the chunk holds it.
// Pass B: every CTA of row b combines the row's chunk partials in the same
// fixed order (the running-max / rescaled-sum recurrence of the rumus
// FlashAttention milestone), reloads its chunk and writes the gradient
// (Step 4); chunk 0 writes the row loss (Step 3); the last CTA sums the row
// losses in a fixed order (Pass 2).  The logits cross HBM twice on this path.
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

constexpr int NT = kStreamThreads;
constexpr int PT = kStreamPerThread;

__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    return m;
}

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = red[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) s += red[w];
    __syncthreads();
    return s;
}

template <typename T, typename P>
__global__ void __launch_bounds__(NT) stream_partials_kernel(P p, long long chunks) {
    using E = Elem<T>;
    __shared__ float red[NT / 32];
    const long long b = blockIdx.x / chunks;
    const long long k = blockIdx.x % chunks;
    const long long C = p.C;
    const long long cbeg = k * kStreamChunk;
    const unsigned char *row = p.logits + (size_t)(b * C) * E::kBytes;
    float z[PT];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < PT; ++i) {
        const long long c = cbeg + i * NT + threadIdx.x;
        z[i] = c < C ? E::load_global(row + c * E::kBytes) : -INFINITY;
        mx = fmaxf(mx, z[i]);
    }
    const float M = block_max(mx, red) * kLog2e;
    const long long t = target_at(p, b);
    float s = 0.f;  // without the target's term
#pragma unroll
    for (int i = 0; i < PT; ++i) {
        const long long c = cbeg + i * NT + threadIdx.x;
        if (c < C && c != t) s += ex2(fmaf(z[i], kLog2e, -M));
    }
    const float S = block_sum(s, red);
    if (threadIdx.x == 0) p.parts[b * chunks + k] = make_float2(M, S);
    if (t >= cbeg && t < cbeg + kStreamChunk && t < C && threadIdx.x == 0)
        p.zt[b] = E::load_global(row + t * E::kBytes);
}

template <typename T, typename P>
__global__ void __launch_bounds__(NT) stream_grad_kernel(P p, long long chunks) {
    using E = Elem<T>;
    __shared__ float red[NT / 32];
    __shared__ float2 tail_scratch[kTailThreads / 32];
    __shared__ int tail_flag;
    const long long b = blockIdx.x / chunks;
    const long long k = blockIdx.x % chunks;
    const long long C = p.C;
    const long long cbeg = k * kStreamChunk;
    const float2 *part = p.parts + b * chunks;

    // Combine the row's partials: thread i takes chunks i, i+NT, ... in order,
    // then a fixed tree; every CTA of the row computes the same bits.
    float mloc = -INFINITY;
    for (long long q = threadIdx.x; q < chunks; q += NT) mloc = fmaxf(mloc, __ldcg(&part[q].x));
    const float M = block_max(mloc, red);
    float sloc = 0.f;
    for (long long q = threadIdx.x; q < chunks; q += NT) {
        const float2 pq = __ldcg(&part[q]);
        sloc += pq.y * ex2(pq.x - M);
    }
    const float s_rest = block_sum(sloc, red);  // the row's sum without the target's term

    const long long t = target_at(p, b);
    const bool has_t = t >= 0 && t < C;
    const float zt = has_t ? __ldcg(p.zt + b) : 0.f;
    const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
    const float S = s_rest + e_t;
    // (p_t - 1) / B without cancellation, times the upstream gradient
    const float scale = fast_rcp(S) * row_grad_factor(p, scalar_grad_scale(p), b);
    const float g_t = -s_rest * scale;
    if (writes_grad(p)) {  // else loss only
        const unsigned char *row = p.logits + (size_t)(b * C) * E::kBytes;
        unsigned char *grow = p.grad + (size_t)(b * C) * E::kBytes;
#pragma unroll
        for (int i = 0; i < PT; ++i) {
            const long long c = cbeg + i * NT + threadIdx.x;
            if (c < C) {
                const float ev = ex2(fmaf(E::load_global(row + c * E::kBytes), kLog2e, -M));
                E::store(grow + c * E::kBytes, c == t ? g_t : ev * scale);
            }
        }
    }
    if (k == 0 && threadIdx.x == 0 && !is_softmax(p)) {
        float l;
        if (has_t) {
            l = row_loss(s_rest, e_t, S, zt, M);
        } else {
            l = NAN;
            atomicAdd(&p.err[kErrBadTarget], 1);
        }
        p.loss_rows[b] = l;
    }
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T>
cudaError_t launch_t(const ParamsEx &p, long long chunks, cudaStream_t s) {
    const long long blocks = p.B * chunks;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const Params &pp = p;
    if (is_plain(p))
        stream_partials_kernel<T, Params><<<(unsigned)blocks, NT, 0, s>>>(pp, chunks);
    else
        stream_partials_kernel<T, ParamsEx><<<(unsigned)blocks, NT, 0, s>>>(p, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (is_plain(p))
        stream_grad_kernel<T, Params><<<(unsigned)blocks, NT, 0, s>>>(pp, chunks);
    else
        stream_grad_kernel<T, ParamsEx><<<(unsigned)blocks, NT, 0, s>>>(p, chunks);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream(const ParamsEx &p, int dtype, long long chunks, cudaStream_t s) {
    if (dtype == 0) return launch_t<float>(p, chunks, s);
    if (dtype == 2) return launch_t<__half>(p, chunks, s);
    return launch_t<__nv_bfloat16>(p, chunks, s);
}

}  // namespace ce
