// Split-row kernel: each row of the logits crosses HBM exactly once.
//
// A cluster of K CTAs (K = 1, 2, 4 or 8) owns a row at a time; CTA `rank`
// holds the slice [rank*SE, (rank+1)*SE) of the row's classes in its shared
// memory, staged by one TMA bulk copy.  Each CTA keeps a ring of `nslots`
// staged slices so the copies of the next rows are in flight while it
// computes the current one (a persistent grid: cluster c takes rows c,
// c + nclusters, ...).  From the staged copy it computes, per row,
//
//   Step 1  m_r = max over the slice                       (block max)
//   Step 2  S_r = sum 2^(z*log2e - M_r), M_r = m_r*log2e   (block sum)
//   combine M = max_r M_r,  S = sum_r S_r * 2^(M_r - M)    (over DSMEM, K > 1)
//   Step 4  grad = (2^(z*log2e - M) / S - [c == t]) / B     (16-byte stores)
//   Step 3  l_b = ln2 * (log2 S - (z_t*log2e - M))          (rank 0)
//
// which are Steps 1-4 of Pass 1 of rumus 0.1.1's cross_entropy.wgsl, with the
// split-row combine being the running-max / rescaled-sum recurrence the rumus
// project page describes for its FlashAttention milestone (M17), applied to
// the cross-entropy row.  The last CTA to finish sums the row losses in a
// fixed order (Pass 2, fused into the same launch).
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

template <typename T, int K, int NT>
__global__ void __launch_bounds__(NT, 1)
    row_split_kernel(Params p, int nslots, int slot_bytes, long long SE) {
    using E = Elem<T>;
    constexpr int NW = NT / 32;
    constexpr int W = E::kVec;
    constexpr int ES = E::kBytes;
    constexpr int kNoTarget = -0x40000000;

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kMaxSplitSlots];
    __shared__ float red_a[NW];
    __shared__ float red_b[NW];
    __shared__ float4 part[2];
    __shared__ float4 comb;
    __shared__ float2 tail_scratch[kTailThreads / 32];
    __shared__ int tail_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = (K > 1) ? cluster_rank() : 0u;
    const long long cid = (K > 1) ? (long long)cluster_id_x() : (long long)blockIdx.x;
    const long long ncl = (K > 1) ? (long long)cluster_count_x() : (long long)gridDim.x;
    const long long C = p.C;
    const long long c0 = min((long long)rank * SE, C);
    const long long c1 = min(c0 + SE, C);
    const int slice_n = (int)(c1 - c0);
    const long long nrows = cid < p.B ? (p.B - cid + ncl - 1) / ncl : 0;
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    const bool vec_store = p.grad_vec_ok != 0;

    // Byte range [gs, ge) of this CTA's slice of row `row`, and the aligned
    // span that the TMA copy can cover inside the tensor.
    auto span = [&](long long row, uint64_t &gs, uint64_t &ge, uint64_t &g0, uint64_t &lo,
                    uint64_t &hi) {
        gs = lbase + (uint64_t)(row * C + c0) * ES;
        ge = gs + (uint64_t)slice_n * ES;
        g0 = gs & ~15ull;
        lo = g0 > p.lo_clip ? g0 : p.lo_clip;
        const uint64_t ghi = (ge + 15) & ~15ull;
        hi = ghi < p.hi_clip ? ghi : p.hi_clip;
    };
    auto issue = [&](long long j) {
        const int s = (int)(j % nslots);
        uint64_t gs, ge, g0, lo, hi;
        span(cid + j * ncl, gs, ge, g0, lo, hi);
        unsigned char *slot = smem + (size_t)s * slot_bytes;
        if (hi > lo) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(hi - lo));
            bulk_g2s(slot + (lo - g0), reinterpret_cast<const void *>(lo), (uint32_t)(hi - lo),
                     &full[s]);
        } else {
            mbar_arrive(&full[s]);
        }
    };

    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    long long issued = 0;
    if (tid == 0) {
        for (; issued < nrows && issued < nslots; ++issued) issue(issued);
    }

    bool failed = false;
    long long consumed = 0;
    int t_next = nrows > 0 ? __ldg(p.targets + cid) : 0;

    for (long long j = 0; j < nrows; ++j) {
        const long long row = cid + j * ncl;
        const int s = (int)(j % nslots);
        const uint32_t parity = (uint32_t)((j / nslots) & 1);
        unsigned char *slot = smem + (size_t)s * slot_bytes;
        const long long t = t_next;
        if (j + 1 < nrows) t_next = __ldg(p.targets + row + ncl);

        if (!failed) {
            if (mbar_wait(&full[s], parity)) {
                consumed = j + 1;
            } else {
                failed = true;
                atomicAdd(&p.err[kErrTimeout], 1);
            }
        }
        failed = __syncthreads_or(failed);

        uint64_t gs, ge, g0, lo, hi;
        span(row, gs, ge, g0, lo, hi);
        // Vector v of the slot holds the slice's local elements v*W - head ..
        // v*W - head + W - 1; local element l is valid for 0 <= l < slice_n.
        const int head = (int)((gs - g0) / ES);
        const int nv = (int)((((ge + 15) & ~15ull) - g0) >> 4);
        const bool head_part = head != 0;
        const bool tail_part = (ge & 15ull) != 0;
        const int vb = head_part ? 1 : 0;
        const int ve = nv - (tail_part ? 1 : 0);
        const int rv0 = head_part ? 0 : -1;
        const int rv1 = (tail_part && nv - 1 != rv0) ? nv - 1 : -1;
        bool has_t = t >= c0 && t < c1;
        const int tl = has_t ? (int)(t - c0) + head : kNoTarget;  // target, vector-0 based

        // Elements whose bytes the copy could not cover (only at the very
        // beginning or end of an unaligned tensor): plain loads.
        if (!failed && (g0 < p.lo_clip || ((ge + 15) & ~15ull) > p.hi_clip)) {
            if (tid < 16) {
                const int l = tid < 8 ? tid : slice_n - 16 + tid;
                if (l >= 0 && l < slice_n) {
                    const uint64_t a = gs + (uint64_t)l * ES;
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
            __syncthreads();
        }
        const bool ragged = (tid == 0 && rv0 >= 0) || (tid == NT - 1 && rv1 >= 0);
        const int rv = tid == 0 ? rv0 : rv1;

        // ---- Step 1: slice max
        float mx = -INFINITY;
        if (!failed) {
#pragma unroll 4
            for (int v = vb + tid; v < ve; v += NT) mx = fmaxf(mx, E::vmax(lds128(slot + 16 * v)));
            if (ragged) {
                float z[W];
                E::unpack(lds128(slot + 16 * rv), z);
#pragma unroll
                for (int k = 0; k < W; ++k)
                    if ((unsigned)(rv * W + k - head) < (unsigned)slice_n) mx = fmaxf(mx, z[k]);
            }
        }
        mx = warp_max(mx);
        if (lane == 0) red_a[warp] = mx;
        __syncthreads();
        float m = red_a[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) m = fmaxf(m, red_a[w]);
        float M = m * kLog2e;

        // ---- Step 2: slice sum of exponentials, the target's term left out
        // (it is added back after the combine, so that 1 - p_t keeps its
        // relative precision when the target dominates the row)
        float sa = 0.f, sb = 0.f;
        if (!failed) {
#pragma unroll 2
            for (int v = vb + tid; v < ve; v += NT) {
                float z[W];
                E::unpack(lds128(slot + 16 * v), z);
                const int d = tl - v * W;
                if ((unsigned)d < (unsigned)W) {
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        if (k != d) sa += ex2(fmaf(z[k], kLog2e, -M));
                } else {
#pragma unroll
                    for (int k = 0; k < W; k += 2) {
                        sa += ex2(fmaf(z[k], kLog2e, -M));
                        sb += ex2(fmaf(z[k + 1], kLog2e, -M));
                    }
                }
            }
            if (ragged) {
                float z[W];
                E::unpack(lds128(slot + 16 * rv), z);
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    const int e = rv * W + k;
                    if ((unsigned)(e - head) < (unsigned)slice_n && e != tl)
                        sa += ex2(fmaf(z[k], kLog2e, -M));
                }
            }
        }
        float ssum = warp_sum(sa + sb);
        if (lane == 0) red_b[warp] = ssum;
        __syncthreads();
        float S = red_b[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) S += red_b[w];

        float zt = 0.f;
        if (has_t && !failed) zt = E::load(slot + (size_t)tl * ES);

        if (K > 1) {
            // Combine the K slices' (M_r, S_r) in rank order; every CTA of the
            // cluster computes the same bits.  Only warp 0 publishes, so only
            // warp 0 arrives with release semantics.
            if (tid == 0) part[j & 1] = make_float4(M, S, zt, has_t ? 1.f : 0.f);
            if (warp == 0)
                cluster_arrive_release();
            else
                cluster_arrive_relaxed();
            cluster_wait();
            if (warp == 0) {
                float4 q = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                if (lane < K) q = ld_dsmem_f4(&part[j & 1], (uint32_t)lane);
                float Mg = -INFINITY;
#pragma unroll
                for (int r = 0; r < K; ++r) Mg = fmaxf(Mg, __shfl_sync(0xffffffffu, q.x, r));
                float Sg = 0.f, ztg = 0.f, hg = 0.f;
#pragma unroll
                for (int r = 0; r < K; ++r) {
                    const float Mr = __shfl_sync(0xffffffffu, q.x, r);
                    const float Sr = __shfl_sync(0xffffffffu, q.y, r);
                    const float zr = __shfl_sync(0xffffffffu, q.z, r);
                    const float hr = __shfl_sync(0xffffffffu, q.w, r);
                    Sg += Sr * ex2(Mr - Mg);
                    if (hr != 0.f) {
                        ztg = zr;
                        hg = 1.f;
                    }
                }
                if (lane == 0) comb = make_float4(Mg, Sg, ztg, hg);
            }
            __syncthreads();
            const float4 cb = comb;
            M = cb.x;
            S = cb.y;
            zt = cb.z;
            has_t = cb.w != 0.f;
        }
        // S holds the sum without the target's term: S_rest = S * (1 - p_t).
        const float s_rest = S;
        const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
        S = s_rest + e_t;

        // ---- Step 4: gradient of the slice
        const float scale = (1.0f / S) * p.inv_b;
        // (p_t - 1) / B = -S_rest / (S B): no cancellation when p_t is near 1
        const float g_t = -s_rest * scale;
        if (!failed) {
            unsigned char *gbase = p.grad + (g0 - lbase);  // grad byte of vector 0
#pragma unroll 2
            for (int v = vb + tid; v < ve; v += NT) {
                float z[W];
                E::unpack(lds128(slot + 16 * v), z);
                float g[W];
#pragma unroll
                for (int k = 0; k < W; ++k) g[k] = ex2(fmaf(z[k], kLog2e, -M)) * scale;
                const int d = tl - v * W;
                if ((unsigned)d < (unsigned)W) {
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        if (k == d) g[k] = g_t;
                }
                if (vec_store) {
                    *reinterpret_cast<uint4 *>(gbase + 16 * v) = E::pack(g);
                } else {
#pragma unroll
                    for (int k = 0; k < W; ++k) E::store(gbase + 16 * v + k * ES, g[k]);
                }
            }
            if (ragged) {
                float z[W];
                E::unpack(lds128(slot + 16 * rv), z);
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    const int e = rv * W + k;
                    if ((unsigned)(e - head) < (unsigned)slice_n) {
                        const float gv = e == tl ? g_t : ex2(fmaf(z[k], kLog2e, -M)) * scale;
                        E::store(gbase + 16 * rv + k * ES, gv);
                    }
                }
            }
        }

        // ---- Step 3: the row's loss (one writer per row)
        if (rank == 0 && tid == 0 && !failed) {
            float l;
            if (has_t) {
                // l = log(S / e_t) = log1p(S_rest / e_t): the second form keeps
                // its precision when the target dominates (then e_t > S / 2).
                l = s_rest < e_t ? log1pf(s_rest / e_t)
                                 : kLn2 * (log2f(S) - fmaf(zt, kLog2e, -M));
            } else {
                l = NAN;
                atomicAdd(&p.err[kErrBadTarget], 1);
            }
            p.loss_rows[row] = l;
        }

        __syncthreads();  // every thread is done with this slot
        if (tid == 0 && !failed && issued < nrows) {
            fence_proxy_async();
            issue(issued);
            ++issued;
        }
    }

    // A CTA that gave up still owns copies in flight: wait for them (bounded)
    // before its shared memory is released.
    if (tid == 0 && failed) {
        for (long long j = consumed; j < issued; ++j) {
            if (!mbar_wait(&full[j % nslots], (uint32_t)((j / nslots) & 1))) break;
        }
    }
    if (K > 1) cluster_sync();  // peers may still read this CTA's partials
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, int K, int NT>
cudaError_t launch_k(const Params &p, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, cudaStream_t s) {
    auto kern = row_split_kernel<T, K, NT>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (K > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = K;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, p, nslots, slot_bytes, se);
}

template <typename T, int K, int NT>
cudaError_t max_clusters_k(int smem, int *clusters) {
    auto kern = row_split_kernel<T, K, NT>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    if (K == 1) {
        int dev = 0, sms = 0, per_sm = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
        if (e != cudaSuccess) return e;
        *clusters = sms * per_sm;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(K, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = K;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

template <typename T, int NT>
cudaError_t launch_n(const Params &p, int K, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, cudaStream_t s) {
    switch (K) {
        case 1: return launch_k<T, 1, NT>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 2: return launch_k<T, 2, NT>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 4: return launch_k<T, 4, NT>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 8: return launch_k<T, 8, NT>(p, ctas, nslots, slot_bytes, se, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int NT>
cudaError_t max_clusters_n(int K, int smem, int *clusters) {
    switch (K) {
        case 1: return max_clusters_k<T, 1, NT>(smem, clusters);
        case 2: return max_clusters_k<T, 2, NT>(smem, clusters);
        case 4: return max_clusters_k<T, 4, NT>(smem, clusters);
        case 8: return max_clusters_k<T, 8, NT>(smem, clusters);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_t(const Params &p, int K, int threads, int ctas, int nslots, int slot_bytes,
                     long long se, int smem, cudaStream_t s) {
    if (threads == 1024) return launch_n<T, 1024>(p, K, ctas, nslots, slot_bytes, se, smem, s);
    if (threads == 512) return launch_n<T, 512>(p, K, ctas, nslots, slot_bytes, se, smem, s);
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t max_clusters_t(int K, int threads, int smem, int *clusters) {
    if (threads == 1024) return max_clusters_n<T, 1024>(K, smem, clusters);
    if (threads == 512) return max_clusters_n<T, 512>(K, smem, clusters);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_split(const Params &p, int dtype, int K, int threads, int ctas, int nslots,
                         int slot_bytes, long long slice_elems, int smem, cudaStream_t s) {
    if (dtype == 0)
        return launch_t<float>(p, K, threads, ctas, nslots, slot_bytes, slice_elems, smem, s);
    return launch_t<__nv_bfloat16>(p, K, threads, ctas, nslots, slot_bytes, slice_elems, smem, s);
}

cudaError_t split_max_clusters(int dtype, int K, int threads, int smem, int *clusters) {
    if (dtype == 0) return max_clusters_t<float>(K, threads, smem, clusters);
    return max_clusters_t<__nv_bfloat16>(K, threads, smem, clusters);
}

}  // namespace ce
