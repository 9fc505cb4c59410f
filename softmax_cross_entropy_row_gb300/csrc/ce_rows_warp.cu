// Warp-per-row kernel for rows of at most a few KB (classifier heads).
//
// Each warp owns a private ring of `slots` shared-memory tiles; a tile is
// `rows_per_tile` consecutive rows of the logits, staged by one TMA bulk copy.
// Warps act as their own producers, so no CTA-wide barrier is needed until
// the fused batch-loss tail.  Per row the warp computes Steps 1-4 of Pass 1 of
// rumus 0.1.1's cross_entropy.wgsl (max, sum of exponentials, row loss,
// gradient) from the staged copy, with warp-shuffle reductions; the last CTA
// to finish performs Pass 2 (the fixed-order batch-loss sum).
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

template <typename T>
__global__ void __launch_bounds__(kWarpKernelWarps * 32)
    rows_warp_kernel(Params p, int slots, int rows_per_tile, int slot_bytes) {
    using E = Elem<T>;
    constexpr int NW = kWarpKernelWarps;
    constexpr int ES = E::kBytes;

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[NW * kMaxWarpSlots];
    __shared__ float2 tail_scratch[kTailThreads / 32];
    __shared__ int tail_flag;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long B = p.B;
    const long long C = p.C;
    const long long R = rows_per_tile;
    const long long ntiles = (B + R - 1) / R;
    const long long gw = (long long)blockIdx.x * NW + warp;
    const long long TW = (long long)gridDim.x * NW;
    const long long ntl = ntiles > gw ? (ntiles - gw + TW - 1) / TW : 0;
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    unsigned char *my_slots = smem + (size_t)warp * slots * slot_bytes;
    uint64_t *my_full = full + warp * kMaxWarpSlots;

    auto span = [&](long long tile, long long &r0, long long &r1, uint64_t &gs, uint64_t &ge,
                    uint64_t &g0, uint64_t &lo, uint64_t &hi) {
        r0 = tile * R;
        r1 = min(r0 + R, B);
        gs = lbase + (uint64_t)(r0 * C) * ES;
        ge = lbase + (uint64_t)(r1 * C) * ES;
        g0 = gs & ~15ull;
        lo = g0 > p.lo_clip ? g0 : p.lo_clip;
        const uint64_t ghi = (ge + 15) & ~15ull;
        hi = ghi < p.hi_clip ? ghi : p.hi_clip;
    };
    auto issue = [&](long long i) {
        const int s = (int)(i % slots);
        long long r0, r1;
        uint64_t gs, ge, g0, lo, hi;
        span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);
        unsigned char *slot = my_slots + (size_t)s * slot_bytes;
        if (hi > lo) {
            mbar_arrive_expect_tx(&my_full[s], (uint32_t)(hi - lo));
            bulk_g2s(slot + (lo - g0), reinterpret_cast<const void *>(lo), (uint32_t)(hi - lo),
                     &my_full[s]);
        } else {
            mbar_arrive(&my_full[s]);
        }
    };

    if (lane == 0) {
        for (int s = 0; s < slots; ++s) mbar_init(&my_full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    long long issued = 0;
    if (lane == 0) {
        for (; issued < ntl && issued < slots; ++issued) issue(issued);
    }

    bool failed = false;
    long long consumed = 0;
    const float inv_b = p.inv_b;

    for (long long i = 0; i < ntl; ++i) {
        const int s = (int)(i % slots);
        const uint32_t parity = (uint32_t)((i / slots) & 1);
        unsigned char *slot = my_slots + (size_t)s * slot_bytes;
        long long r0, r1;
        uint64_t gs, ge, g0, lo, hi;
        span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);

        if (!failed) {
            if (mbar_wait(&my_full[s], parity)) {
                consumed = i + 1;
            } else {
                failed = true;
                if (lane == 0) atomicAdd(&p.err[kErrTimeout], 1);
            }
        }
        failed = __any_sync(0xffffffffu, failed);
        if (failed) continue;

        // Elements of an unaligned tensor's first/last 16 bytes: plain loads.
        if (g0 < p.lo_clip || ((ge + 15) & ~15ull) > p.hi_clip) {
            if (lane < 16) {
                const long long n = (long long)((ge - gs) / ES);
                const long long e = lane < 8 ? lane : n - 16 + lane;
                if (e >= 0 && e < n) {
                    const uint64_t a = gs + (uint64_t)e * ES;
                    if (a < lo || a + ES > hi) {
                        if (ES == 4)
                            *reinterpret_cast<uint32_t *>(slot + (a - g0)) =
                                __ldg(reinterpret_cast<const unsigned int *>(a));
                        else
                            *reinterpret_cast<uint16_t *>(slot + (a - g0)) =
                                __ldg(reinterpret_cast<const unsigned short *>(a));
                    }
                }
            }
            __syncwarp();
        }

        for (long long r = r0; r < r1; ++r) {
            const unsigned char *row = slot + (gs - g0) + (size_t)((r - r0) * C) * ES;
            const long long t = __ldg(p.targets + r);
            // Step 1: max
            float m = -INFINITY;
            for (long long c = lane; c < C; c += 32) m = fmaxf(m, E::load(row + c * ES));
            m = warp_max(m);
            const float M = m * kLog2e;
            // Step 2: sum of exponentials without the target's term (added
            // back below, so that 1 - p_t keeps its relative precision)
            float sa = 0.f, sb = 0.f;
            long long c = lane;
            for (; c + 32 < C; c += 64) {
                const float ea = ex2(fmaf(E::load(row + c * ES), kLog2e, -M));
                const float eb = ex2(fmaf(E::load(row + (c + 32) * ES), kLog2e, -M));
                sa += c == t ? 0.f : ea;
                sb += c + 32 == t ? 0.f : eb;
            }
            if (c < C && c != t) sa += ex2(fmaf(E::load(row + c * ES), kLog2e, -M));
            const float s_rest = warp_sum(sa + sb);
            const bool has_t = t >= 0 && t < C;
            const float zt = has_t ? E::load(row + t * ES) : 0.f;
            const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
            const float S = s_rest + e_t;
            // Step 4: gradient; (p_t - 1) / B = -S_rest / (S B)
            const float scale = (1.0f / S) * inv_b;
            const float g_t = -s_rest * scale;
            unsigned char *grow = p.grad + (size_t)(r * C) * ES;
            for (long long k = lane; k < C; k += 32) {
                const float ev = ex2(fmaf(E::load(row + k * ES), kLog2e, -M));
                E::store(grow + k * ES, k == t ? g_t : ev * scale);
            }
            // Step 3: loss of the row, log(S / e_t)
            if (lane == 0) {
                float l;
                if (has_t) {
                    l = s_rest < e_t ? log1pf(s_rest / e_t)
                                     : kLn2 * (log2f(S) - fmaf(zt, kLog2e, -M));
                } else {
                    l = NAN;
                    atomicAdd(&p.err[kErrBadTarget], 1);
                }
                p.loss_rows[r] = l;
            }
        }
        __syncwarp();
        if (lane == 0 && issued < ntl) {
            fence_proxy_async();
            issue(issued);
            ++issued;
        }
    }

    if (lane == 0 && failed) {
        for (long long i = consumed; i < issued; ++i) {
            if (!mbar_wait(&my_full[i % slots], (uint32_t)((i / slots) & 1))) break;
        }
    }
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T>
cudaError_t launch_t(const Params &p, int ctas, int slots, int rows_per_tile, int slot_bytes,
                     int smem, cudaStream_t s) {
    auto kern = rows_warp_kernel<T>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kWarpKernelWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kern, p, slots, rows_per_tile, slot_bytes);
}

template <typename T>
cudaError_t occ_t(int smem, int *ctas) {
    auto kern = rows_warp_kernel<T>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, kWarpKernelWarps * 32, smem);
}

}  // namespace

cudaError_t launch_rows_warp(const Params &p, int dtype, int ctas, int slots, int rows_per_tile,
                             int slot_bytes, int smem, cudaStream_t s) {
    if (dtype == 0) return launch_t<float>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    return launch_t<__nv_bfloat16>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
}

cudaError_t rows_warp_max_ctas_per_sm(int dtype, int smem, int *ctas) {
    if (dtype == 0) return occ_t<float>(smem, ctas);
    return occ_t<__nv_bfloat16>(smem, ctas);
}

}  // namespace ce
