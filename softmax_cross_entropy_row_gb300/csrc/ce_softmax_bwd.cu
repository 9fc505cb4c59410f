// Row-wise softmax backward: dx_b = p_b * (dy_b - sum_c p_bc dy_bc) for
// probabilities p [B][C] and upstream gradient dy [B][C]: the row-wise
// softmax backward of the rumus project page (milestone M8c, row-wise
// softmax with forward and backward kernels).  One
// dot product per row, then one pass of fused multiply-adds; HBM traffic is
// two reads and one write per element.
//
// Three kernels:
//   softmax_bwd_warp_kernel  rows of at most 4 KB (32 lanes x 8 vectors) whose
//                            every row starts 16-byte aligned: one warp per
//                            row, the row's vectors of p and dy in registers,
//                            a butterfly sum (the same bits in every lane), no
//                            barrier; many rows in flight per SM;
//   softmax_bwd_vec_kernel   rows of at most kVecThreads x kVecPerThread 16-byte
//                            vectors whose every row starts 16-byte aligned in
//                            all three tensors: 128 threads per row up to 16 KB
//                            (the CTA's 512 threads take 4 rows at a time),
//                            512 beyond, each thread's
//                            vectors of p and dy in registers (all loads in
//                            flight before the first use), one reduction over
//                            the row's threads, the row written from the
//                            registers;
//   softmax_bwd_any_kernel   any row: pass 1 accumulates the dot product over
//                            the row, pass 2 reads p and dy again and writes dx
//                            (p and dy cross HBM twice).
// Both are persistent over rows (CTA b takes rows b, b + grid, ...); the dot
// product is summed in a fixed order (per-thread partials in element order,
// then a fixed tree), so results are bitwise reproducible.
#include <map>
#include <mutex>

#include "ce_launch.h"

namespace ce {
namespace {

constexpr int kVecThreads = 512;
constexpr int kVecPerThread = 8;  // 64 KB rows of each tensor at most
constexpr size_t kPrefetchPiece = 16384;  // bytes per L2 prefetch request (4 cover a row)
constexpr int kAnyThreads = 512;
constexpr int kWarpCtaThreads = 256;
constexpr int kWarpMaxVpl = 8;  // 4 KB rows of each tensor at most

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) from global
// memory into L2; nothing is written to shared memory and nothing waits.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <int NT>
__device__ __forceinline__ float block_sum_fixed(float v, float *red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < NT / 32 ? red[lane] : 0.f;
    t = warp_sum(t);
    __syncthreads();  // red is reused by the next row
    return t;
}

// Sum over the TPR threads of row group g (warps [g * TPR / 32, ...)): warp
// sums, then the group's warps through `red` and named barrier 1 + g (barrier
// 0 is __syncthreads).  Every thread of the group gets the same bits.
template <int TPR>
__device__ __forceinline__ float group_sum_fixed(float v, float *red, int g) {
    constexpr int GW = TPR / 32;
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, wg = (threadIdx.x >> 5) % GW;
    if (lane == 0) red[g * GW + wg] = v;
    if (TPR == 32) return v;
    named_sync(1 + g, TPR);
    float t = lane < GW ? red[g * GW + lane] : 0.f;
    t = warp_sum(t);
    named_sync(1 + g, TPR);  // red is reused by the group's next row
    return t;
}

// TPR threads per row (128 or 512), kVecThreads / TPR rows of the CTA at a
// time: rows of at most TPR x kVecPerThread 16-byte vectors.
template <typename T, int TPR>
__global__ void __launch_bounds__(kVecThreads, 1)
    softmax_bwd_vec_kernel(const unsigned char *P, const unsigned char *DY, unsigned char *DX,
                           long long B, long long C) {
    using E = Elem<T>;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr int RPC = kVecThreads / TPR;  // rows per CTA at a time
    __shared__ float red[kVecThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int g = threadIdx.x / TPR;    // the thread's row group
    const int tid = threadIdx.x % TPR;  // its place in the group
    const long long nvec = C / W;  // whole vectors per row (C * es is a multiple of 16)
    const size_t row_bytes = (size_t)C * E::kBytes;
    const long long first = (long long)blockIdx.x * RPC + g;
    const long long step = (long long)gridDim.x * RPC;
    // A group's rows are first, first + step, ...; the next row's reads
    // overlap the current row.  fp32: a thread's vectors of the next row are
    // loaded into its registers as soon as it has written the same vectors of
    // the current row.  16-bit (whose unpacked pairs leave no registers for
    // that): the next row of p and dy is prefetched into L2 in 16 KB bulk
    // requests when the current row starts, so its loads are served by L2.
    constexpr bool kRegPipe = sizeof(T) == 4;
    uint4 pv[kVecPerThread], dv[kVecPerThread];
    auto load_vec = [&](long long b, int k) {
        const long long v = tid + (long long)k * TPR;
        pv[k] = make_uint4(0u, 0u, 0u, 0u);
        dv[k] = make_uint4(0u, 0u, 0u, 0u);
        if (b < B && v < nvec) {
            pv[k] = __ldcs(reinterpret_cast<const uint4 *>(P + (size_t)b * row_bytes) + v);
            dv[k] = __ldcs(reinterpret_cast<const uint4 *>(DY + (size_t)b * row_bytes) + v);
        }
    };
    if (kRegPipe) {
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) load_vec(first, k);
    }
    // each group loops over its own rows and meets only its own barrier
    for (long long b = first; b < B; b += step) {
        uint4 *xrow = reinterpret_cast<uint4 *>(DX + (size_t)b * row_bytes);
        if (!kRegPipe) {
            // 16 KB pieces of the next row of p (threads 0-3) and dy (4-7)
            const long long bn = b + step;
            const size_t off = (size_t)(tid & 3) * kPrefetchPiece;
            if (tid < 8 && bn < B && off < row_bytes) {
                const unsigned char *src = (tid < 4 ? P : DY) + (size_t)bn * row_bytes + off;
                const size_t left = row_bytes - off;
                bulk_prefetch_l2(src, (uint32_t)(left < kPrefetchPiece ? left : kPrefetchPiece));
            }
#pragma unroll
            for (int k = 0; k < kVecPerThread; ++k) load_vec(b, k);
        }
        unsigned long long acc = 0ull;
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) {
            unsigned long long p2[W2], d2[W2];
            E::unpack2(pv[k], p2);
            E::unpack2(dv[k], d2);
#pragma unroll
            for (int i = 0; i < W2; ++i) acc = f2_fma(p2[i], d2[i], acc);
        }
        float sa, sb;
        f2_unpack(acc, sa, sb);
        const float dot = group_sum_fixed<TPR>(sa + sb, red, g);
        const unsigned long long nd2 = f2_pack(-dot, -dot);
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) {
            const long long v = tid + (long long)k * TPR;
            if (v < nvec) {
                unsigned long long p2[W2], d2[W2];
                E::unpack2(pv[k], p2);
                E::unpack2(dv[k], d2);
#pragma unroll
                for (int i = 0; i < W2; ++i) p2[i] = f2_mul(p2[i], f2_add(d2[i], nd2));
                __stcs(xrow + v, E::pack2(p2));
            }
            if (kRegPipe) load_vec(b + step, k);
        }
    }
}

// One warp per row; VPL vectors per lane (32 x VPL >= the row's vectors).
template <typename T, int VPL>
__global__ void __launch_bounds__(kWarpCtaThreads, 2)
    softmax_bwd_warp_kernel(const unsigned char *P, const unsigned char *DY, unsigned char *DX,
                            long long B, long long C) {
    using E = Elem<T>;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long nvec = C / W;
    const long long warps = (long long)gridDim.x * (kWarpCtaThreads / 32);
    for (long long b = (long long)blockIdx.x * (kWarpCtaThreads / 32) + (threadIdx.x >> 5); b < B;
         b += warps) {
        const uint4 *prow = reinterpret_cast<const uint4 *>(P + (size_t)b * C * E::kBytes);
        const uint4 *drow = reinterpret_cast<const uint4 *>(DY + (size_t)b * C * E::kBytes);
        uint4 *xrow = reinterpret_cast<uint4 *>(DX + (size_t)b * C * E::kBytes);
        uint4 pv[VPL], dv[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            pv[k] = make_uint4(0u, 0u, 0u, 0u);
            dv[k] = make_uint4(0u, 0u, 0u, 0u);
            if (v < nvec) {
                pv[k] = __ldcs(prow + v);
                dv[k] = __ldcs(drow + v);
            }
        }
        unsigned long long acc = 0ull;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            unsigned long long p2[W2], d2[W2];
            E::unpack2(pv[k], p2);
            E::unpack2(dv[k], d2);
#pragma unroll
            for (int i = 0; i < W2; ++i) acc = f2_fma(p2[i], d2[i], acc);
        }
        float sa, sb;
        f2_unpack(acc, sa, sb);
        const float dot = warp_sum(sa + sb);
        const unsigned long long nd2 = f2_pack(-dot, -dot);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            if (v < nvec) {
                unsigned long long p2[W2], d2[W2];
                E::unpack2(pv[k], p2);
                E::unpack2(dv[k], d2);
#pragma unroll
                for (int i = 0; i < W2; ++i) p2[i] = f2_mul(p2[i], f2_add(d2[i], nd2));
                __stcs(xrow + v, E::pack2(p2));
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kAnyThreads)
    softmax_bwd_any_kernel(const unsigned char *P, const unsigned char *DY, unsigned char *DX,
                           long long B, long long C) {
    using E = Elem<T>;
    constexpr int ES = E::kBytes;
    __shared__ float red[kAnyThreads / 32];
    pdl_trigger();
    pdl_wait();
    for (long long b = blockIdx.x; b < B; b += gridDim.x) {
        const unsigned char *prow = P + (size_t)b * C * ES;
        const unsigned char *drow = DY + (size_t)b * C * ES;
        unsigned char *xrow = DX + (size_t)b * C * ES;
        float acc = 0.f;
        for (long long c = threadIdx.x; c < C; c += kAnyThreads)
            acc = fmaf(E::load_global(prow + c * ES), E::load_global(drow + c * ES), acc);
        const float dot = block_sum_fixed<kAnyThreads>(acc, red);
        for (long long c = threadIdx.x; c < C; c += kAnyThreads) {
            const float pc = E::load_global(prow + c * ES);
            const float dc = E::load_global(drow + c * ES);
            E::store(xrow + c * ES, pc * (dc - dot));
        }
    }
}

// CTAs per SM that the kernel can keep resident (cached per device and kernel).
int resident_ctas(const void *kern, int threads) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, kern});
    if (it != cache.end()) return it->second;
    int n = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    cache[{dev, kern}] = n;
    return n;
}

// Launch `kern` persistent over rows: at most the resident CTAs of every SM,
// `rows_per_cta` rows to a CTA per sweep.
template <typename K>
cudaError_t launch_rows(K kern, int threads, long long rows_per_cta, const void *p, const void *dy,
                        void *dx, long long B, long long C, int sms, cudaStream_t s) {
    const long long cap = (long long)sms * resident_ctas(reinterpret_cast<const void *>(kern), threads);
    const long long want = (B + rows_per_cta - 1) / rows_per_cta;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(want < cap ? want : cap), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const unsigned char *>(p),
                              static_cast<const unsigned char *>(dy),
                              static_cast<unsigned char *>(dx), B, C);
}

template <typename T>
cudaError_t launch_t(const void *p, const void *dy, void *dx, long long B, long long C, bool vec,
                     int sms, cudaStream_t s) {
    if (!vec) return launch_rows(softmax_bwd_any_kernel<T>, kAnyThreads, 1, p, dy, dx, B, C, sms, s);
    const long long nvec = C / Elem<T>::kVec;
    constexpr int kRowsPerWarpCta = kWarpCtaThreads / 32;
    if (nvec <= 32)
        return launch_rows(softmax_bwd_warp_kernel<T, 1>, kWarpCtaThreads, kRowsPerWarpCta, p, dy,
                           dx, B, C, sms, s);
    if (nvec <= 64)
        return launch_rows(softmax_bwd_warp_kernel<T, 2>, kWarpCtaThreads, kRowsPerWarpCta, p, dy,
                           dx, B, C, sms, s);
    if (nvec <= 128)
        return launch_rows(softmax_bwd_warp_kernel<T, 4>, kWarpCtaThreads, kRowsPerWarpCta, p, dy,
                           dx, B, C, sms, s);
    if (nvec <= 32 * kWarpMaxVpl)
        return launch_rows(softmax_bwd_warp_kernel<T, kWarpMaxVpl>, kWarpCtaThreads,
                           kRowsPerWarpCta, p, dy, dx, B, C, sms, s);
    // rows of up to 16 KB: 128 threads each, four rows of the CTA at once
    // (measured on GB300: 16 KB rows 183 -> 132 us bf16, 186 -> 118 us fp32,
    // 16384 rows); longer rows: 512 threads (two 256-thread groups were
    // slower on 32 KB bf16 rows, 134 against 124 us)
    if (nvec <= 128 * kVecPerThread)
        return launch_rows(softmax_bwd_vec_kernel<T, 128>, kVecThreads, kVecThreads / 128, p, dy,
                           dx, B, C, sms, s);
    return launch_rows(softmax_bwd_vec_kernel<T, 512>, kVecThreads, 1, p, dy, dx, B, C, sms, s);
}

}  // namespace

bool softmax_bwd_vec_ok(long long C, int es, uintptr_t p, uintptr_t dy, uintptr_t dx) {
    return (C * es) % 16 == 0 && C * es <= (long long)kVecThreads * kVecPerThread * 16 &&
           p % 16 == 0 && dy % 16 == 0 && dx % 16 == 0;
}

cudaError_t launch_softmax_bwd(const void *p, const void *dy, void *dx, long long B, long long C,
                               int dtype, bool vec, int sms, cudaStream_t s) {
    if (dtype == 0) return launch_t<float>(p, dy, dx, B, C, vec, sms, s);
    if (dtype == 2) return launch_t<__half>(p, dy, dx, B, C, vec, sms, s);
    return launch_t<__nv_bfloat16>(p, dy, dx, B, C, vec, sms, s);
}

}  // namespace ce
