// Loss-only warp-per-row kernel (ce_forward, ce_fwd_bwd_ex without a
// gradient), for rows of any length.
//
// With no gradient to write, a row is needed only once: Steps 1-3 of Pass 1
// of rumus 0.1.1's cross_entropy.wgsl (max, sum of exponentials, row loss)
// can be formed in a single read when the sum is rescaled whenever the
// running max grows (sum_c e^(z_c - m) = e^(m' - m) sum_c e^(z_c - m'): the
// online-softmax recurrence of the rumus project page's FlashAttention
// milestone, M17).  Each warp owns whole rows and streams
// them from global memory in 16-byte loads, V vectors per lane per step; each
// lane keeps its own running max m and sum s of 2^(z*log2e - M), M =
// fp32(m*log2e), without the target's term.  At the row's end the lanes'
// sums are brought to the row's max (the lanes' maxima and the target logit)
// and added; the row loss follows from that sum and the target's term exactly
// as in the other kernels.  No shared memory, no barrier, no copy to wait
// for: many independent warps per SM keep the loads in flight.  The CTA that
// finishes last performs Pass 2 (the fixed-order batch-loss sum).
#include <math.h>

#include "ce_rows_online.h"

namespace ce {
namespace {

// 16 bytes of the logits, read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4 *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

// The builds: vectors per lane per step, whether the next step's loads are
// issued before the current step is reduced, and CTAs per SM that the
// register budget is set for.
constexpr int kBuildVecs[kOnlineBuilds] = {8, 4, 8, 16, 4};
constexpr bool kBuildAhead[kOnlineBuilds] = {false, true, true, false, false};
constexpr int kBuildMinBlocks[kOnlineBuilds] = {4, 3, 2, 2, 5};

template <typename T, int BUILD>
__global__ void __launch_bounds__(kOnlineWarps * 32, kBuildMinBlocks[BUILD])
    rows_online_kernel(ParamsEx p) {
    using E = Elem<T>;
    constexpr int ES = E::kBytes;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr int V = kBuildVecs[BUILD];
    constexpr long long STEP = 32LL * V;  // vectors a warp reads per step

    __shared__ int tail_flag;
    __shared__ float2 tail_scratch[kTailWarps];

    const int lane = threadIdx.x & 31;
    const long long B = p.B;
    const long long C = p.C;
    const long long gw = (long long)blockIdx.x * kOnlineWarps + (threadIdx.x >> 5);
    const long long TW = (long long)gridDim.x * kOnlineWarps;
    const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);
    const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);

    pdl_trigger();
    pdl_wait();  // nothing above touched global memory

    int t_next = gw < B ? target_at(p, gw) : 0;
    for (long long r = gw; r < B; r += TW) {
        const int t = t_next;
        if (r + TW < B) t_next = target_at(p, r + TW);
        const bool has_t = t >= 0 && t < C;
        const unsigned char *row = p.logits + (size_t)(r * C) * ES;
        const float zt = has_t ? E::load_global(row + (size_t)t * ES) : 0.f;

        // Row layout: nh head elements up to the first 16-byte boundary, nvec
        // whole vectors, nt tail elements.
        const uint32_t ph = (uint32_t)reinterpret_cast<uintptr_t>(row) & 15u;
        const long long nh = ph ? min((long long)((16u - ph) / ES), C) : 0LL;
        const long long nvec = (C - nh) / W;
        const long long nt = C - nh - nvec * W;
        const unsigned char *vrow = row + nh * ES;
        const uint4 *vp = reinterpret_cast<const uint4 *>(vrow);
        const long long tr = has_t ? t - nh : -1;                       // target from vector 0
        const long long v_t = tr >= 0 && tr < nvec * W ? tr / W : -1;   // its vector
        const int d_t = (int)(tr - v_t * W);                            // its place there

        // Head and tail elements (the target's read as -inf), then the lane's
        // running max and sum start from them.
        float hz = -INFINITY, tz = -INFINITY;
        if (lane < nh && lane != t) hz = E::load_global(row + lane * ES);
        if (lane < nt && nh + nvec * W + lane != t)
            tz = E::load_global(vrow + (nvec * W + lane) * ES);
        float m = fmaxf(hz, tz);
        float M = m * kLog2e;
        float s = m == -INFINITY ? 0.f : ex2(fmaf(hz, kLog2e, -M)) + ex2(fmaf(tz, kLog2e, -M));

        auto load = [&](uint4 (&x)[V], long long v0) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const long long v = v0 + 32 * k + lane;
                x[k] = v < nvec ? ld_stream(vp + v) : kNeg;
            }
        };
        // One step: the target's element set to -inf, the step's max, the sum
        // rescaled if the max grew, then the step's exponentials added.
        auto consume = [&](uint4 (&x)[V], long long v0) {
#pragma unroll
            for (int k = 0; k < V; ++k)
                if (v0 + 32 * k + lane == v_t) x[k] = with_neg_inf<E>(x[k], d_t);
            typename E::MaxAcc macc = E::max_init();
#pragma unroll
            for (int k = 0; k < V; ++k) E::max_step(macc, x[k]);
            const float cm = E::max_value(macc);
            if (cm > m) {
                const float Mn = cm * kLog2e;
                s *= ex2(M - Mn);  // 0 while m was -inf (s is 0 then)
                m = cm;
                M = Mn;
            }
            if (m != -INFINITY) {
                const unsigned long long nM2 = f2_pack(-M, -M);
                unsigned long long acc = 0ull;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    unsigned long long e2[W2];
                    E::unpack2(x[k], e2);
#pragma unroll
                    for (int j = 0; j < W2; ++j) {
                        float a, b;
                        f2_unpack(f2_fma(e2[j], kL2E2, nM2), a, b);
                        e2[j] = f2_pack(ex2(a), ex2(b));
                    }
                    const unsigned long long vs =
                        W2 == 4 ? f2_add(f2_add(e2[0], e2[1]), f2_add(e2[W2 - 2], e2[W2 - 1]))
                                : f2_add(e2[0], e2[W2 - 1]);
                    acc = f2_add(acc, vs);
                }
                float sa, sb;
                f2_unpack(acc, sa, sb);
                s += sa + sb;
            }
        };

        if constexpr (!kBuildAhead[BUILD]) {
            for (long long v0 = 0; v0 < nvec; v0 += STEP) {
                uint4 x[V];
                load(x, v0);
                consume(x, v0);
            }
        } else {
            // two register sets: the next step's loads are in flight while
            // the current step is reduced
            uint4 x[V], y[V];
            if (nvec > 0) load(x, 0);
            for (long long v0 = 0; v0 < nvec; v0 += 2 * STEP) {
                const bool second = v0 + STEP < nvec;
                if (second) load(y, v0 + STEP);
                consume(x, v0);
                if (!second) break;
                if (v0 + 2 * STEP < nvec) load(x, v0 + 2 * STEP);
                consume(y, v0 + STEP);
            }
        }

        // The row: every lane's sum brought to the row max (the target logit
        // included), then added.
        const float mr = fmaxf(warp_max(m), has_t ? zt : -INFINITY);
        const float Mr = mr * kLog2e;
        const float s_rest = warp_sum(m == -INFINITY ? 0.f : s * ex2(M - Mr));
        if (lane == 0) {
            float l;
            if (has_t) {
                const float e_t = ex2(fmaf(zt, kLog2e, -Mr));
                l = row_loss(s_rest, e_t, s_rest + e_t, zt, Mr);
            } else {
                l = NAN;
                atomicAdd(&p.err[kErrBadTarget], 1);
            }
            p.loss_rows[r] = l;
        }
    }
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, int BUILD>
cudaError_t launch_b(const ParamsEx &p, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kOnlineWarps * 32, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rows_online_kernel<T, BUILD>, p);
}

template <typename T, int BUILD>
cudaError_t occ_b(int *ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, rows_online_kernel<T, BUILD>,
                                                         kOnlineWarps * 32, 0);
}

template <typename T>
cudaError_t launch_t(const ParamsEx &p, int build, int ctas, cudaStream_t s) {
    switch (build) {
        case 0: return launch_b<T, 0>(p, ctas, s);
        case 1: return launch_b<T, 1>(p, ctas, s);
        case 2: return launch_b<T, 2>(p, ctas, s);
        case 3: return launch_b<T, 3>(p, ctas, s);
        default: return launch_b<T, 4>(p, ctas, s);
    }
}

template <typename T>
cudaError_t occ_t(int build, int *ctas) {
    switch (build) {
        case 0: return occ_b<T, 0>(ctas);
        case 1: return occ_b<T, 1>(ctas);
        case 2: return occ_b<T, 2>(ctas);
        case 3: return occ_b<T, 3>(ctas);
        default: return occ_b<T, 4>(ctas);
    }
}

}  // namespace

cudaError_t launch_rows_online(const ParamsEx &p, int dtype, int build, int ctas, cudaStream_t s) {
    if (build < 0 || build >= kOnlineBuilds) return cudaErrorInvalidValue;
    if (dtype == 0) return launch_t<float>(p, build, ctas, s);
    if (dtype == 2) return launch_t<__half>(p, build, ctas, s);
    return launch_t<__nv_bfloat16>(p, build, ctas, s);
}

cudaError_t rows_online_max_ctas_per_sm(int dtype, int build, int *ctas) {
    if (build < 0 || build >= kOnlineBuilds) return cudaErrorInvalidValue;
    if (dtype == 0) return occ_t<float>(build, ctas);
    if (dtype == 2) return occ_t<__half>(build, ctas);
    return occ_t<__nv_bfloat16>(build, ctas);
}

}  // namespace ce
