// Pipelined split-row kernel: rows of K slices, one slice per CTA of a
// cluster, with the cluster exchange of row j overlapped with the work of the
// next row.
//
// The arithmetic is that of the split-row kernel (ce_row_split.cu): per slice
// Steps 1-2 of Pass 1 of rumus 0.1.1's cross_entropy.wgsl (slice max, the
// exponentials and their sum without the target's term), the running-max /
// rescaled-sum combine of the rumus project page's FlashAttention milestone
// (M17) over the K slices, then Steps 4 and 3 (gradient, row loss) and the
// fused Pass 2 in the last CTA.  Only the schedule differs.  Iteration j of a
// CTA does
//
//   A(j)    wait for the slice of row j (TMA), read it into registers, slice
//           max and sum; one lane per peer pushes (M_r, S_r, z_t, has_t) into
//           every CTA of the cluster with st.async, which completes
//           transaction bytes on that CTA's exchange mbarrier for row j;
//   B(j-1)  wait for the K partials of row j-1 on the local exchange mbarrier
//           (they were pushed one iteration earlier), combine them, write the
//           gradient of row j-1 from the registers kept since A(j-1), and its
//           loss.
//
// So no cluster-wide barrier sits between a slice's sum and its gradient: the
// exchange latency and the skew between the K CTAs hide behind A(j).  The
// registers hold two slices (the current one and the previous one), so this
// kernel takes slices of at most kSplitThreads x 8 16-byte vectors (64 KB).
//
// Exchange buffers: NB = 4 slots of K float4 and one mbarrier each, slot
// j % NB for row j.  A CTA pushes row i only after its own B(i-2), which
// waited for every peer's row i-2, which each peer pushed only after
// finishing its iteration i-3 (and so reading row i-4's slot).  Hence when row
// i lands in a peer, rows up to i-4 have been read there and rows i-3 .. i
// occupy four distinct slots.  The mbarrier of slot (i % NB) is re-armed for
// row i (expect K x 16 bytes, one local arrival) in iteration i-2, after the
// first block barrier, i.e. once every local thread has passed its wait for
// row i-4 and before this CTA pushes row i-2 (which precedes any peer's push
// of row i).
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

constexpr int kExchangeSlots = 4;

template <typename T, int K, int NT, int VPT>
__global__ void __launch_bounds__(NT, 1)
    row_pipe_kernel(Params p, int nslots, int slot_bytes, long long SE) {
    using E = Elem<T>;
    constexpr int NW = NT / 32;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr int ES = E::kBytes;
    constexpr int NB = kExchangeSlots;
    constexpr int kNoTarget = -0x40000000;
    constexpr bool kKeepExp = sizeof(T) == 4;
    static_assert(K > 1 && K <= 32, "the pipelined kernel exchanges partials between 2..32 CTAs");

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kMaxSplitSlots];
    __shared__ uint64_t xbar[NB];
    __shared__ __align__(16) float4 xbuf[NB][K];  // [row slot][source rank]
    __shared__ float red_max[2][NW];
    __shared__ float red_sum[2][NW];
    __shared__ float zt_sh[2];
    __shared__ unsigned int warps_summed[2];
    __shared__ float2 tail_scratch[kTailWarps];
    __shared__ int tail_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    const long long cid = (long long)cluster_id_x();
    const long long ncl = (long long)cluster_count_x();
    const long long C = p.C;
    const long long c0 = min((long long)rank * SE, C);
    const long long c1 = min(c0 + SE, C);
    const int slice_n = (int)(c1 - c0);
    const long long nrows = cid < p.B ? (p.B - cid + ncl - 1) / ncl : 0;
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    const bool vec_store = p.grad_vec_ok != 0;
    const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);
    const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                  E::kNegInfWord);

    // Where this CTA's slice of row `row` sits: bytes [gs, ge), the 16-byte
    // aligned span from g0, and the part [lo, hi) a TMA copy may cover.
    struct Geom {
        uint64_t gs, ge, g0, lo, hi;
        int head, nv, vf0, vf1;
        bool head_partial, tail_partial;
    };
    auto geom = [&](long long row) {
        Geom g;
        g.gs = lbase + (uint64_t)(row * C + c0) * ES;
        g.ge = g.gs + (uint64_t)slice_n * ES;
        g.g0 = g.gs & ~15ull;
        g.lo = g.g0 > p.lo_clip ? g.g0 : p.lo_clip;
        const uint64_t ghi = (g.ge + 15) & ~15ull;
        g.hi = ghi < p.hi_clip ? ghi : p.hi_clip;
        // vector v of the slot holds local elements v*W - head .. v*W - head + W - 1
        g.head = (int)((g.gs - g.g0) / ES);
        g.nv = (int)((ghi - g.g0) >> 4);
        g.vf0 = g.head != 0 ? 1 : 0;  // whole vectors: [vf0, vf1)
        g.vf1 = (g.ge & 15ull) != 0 ? g.nv - 1 : g.nv;
        g.head_partial = g.vf0 == 1;
        g.tail_partial = g.vf1 == g.nv - 1 && g.nv - 1 >= g.vf0;
        return g;
    };
    auto issue = [&](long long j) {
        const int s = (int)(j % nslots);
        const Geom g = geom(cid + j * ncl);
        unsigned char *slot = smem + (size_t)s * slot_bytes;
        if (g.hi > g.lo) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(g.hi - g.lo));
            bulk_g2s(slot + (g.lo - g.g0), reinterpret_cast<const void *>(g.lo),
                     (uint32_t)(g.hi - g.lo), &full[s]);
        } else {
            mbar_arrive(&full[s]);
        }
    };

    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) mbar_init(&full[s], 1);
        for (int b = 0; b < NB; ++b) mbar_init(&xbar[b], 1);
        fence_mbar_init();
        warps_summed[0] = warps_summed[1] = 0u;
    }
    pdl_trigger();
    pdl_wait();  // nothing above touched global memory
    // every CTA's exchange mbarriers exist before any peer pushes into them
    cluster_sync();
    long long issued = 0;
    if (tid == 0) {
        for (int b = 0; b < NB && b < nrows; ++b)
            mbar_arrive_expect_tx(&xbar[b], (uint32_t)(K * sizeof(float4)));
        for (; issued < nrows && issued < nslots; ++issued) issue(issued);
    }

    bool failed = false;   // a copy or an exchange never completed: results are void
    bool xfailed = false;  // an exchange wait gave up: skip the later ones
    long long consumed = 0;
    int t_next = nrows > 0 ? __ldg(p.targets + cid) : 0;

    uint4 xp[VPT];       // previous row's slice: exponentials (fp32) or logits (bf16)
    long long t_prev = 0;
    float moff_prev = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) xp[k] = kNeg;

    for (long long j = 0; j <= nrows; ++j) {
        uint4 xc[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) xc[k] = kNeg;
        long long t_cur = 0;
        float moff_cur = 0.f;
        // ================================================= A(j): slice partials
        if (j < nrows) {
            const long long row = cid + j * ncl;
            const int s = (int)(j % nslots);
            const int par = (int)(j & 1);
            const uint32_t parity = (uint32_t)((j / nslots) & 1);
            unsigned char *slot = smem + (size_t)s * slot_bytes;
            const long long t = t_next;
            t_cur = t;
            if (j + 1 < nrows) t_next = __ldg(p.targets + row + ncl);
            const Geom g = geom(row);
            const bool has_t = t >= c0 && t < c1;
            const int tl = has_t ? (int)(t - c0) + g.head : kNoTarget;
            const int v_t = has_t ? tl / W : -1;

            if (!failed) {
                if (mbar_wait(&full[s], parity)) {
                    consumed = j + 1;
                } else {
                    failed = true;
                    atomicAdd(&p.err[kErrTimeout], 1);
                }
            }
            // elements the copy could not cover (only at the very beginning or
            // end of an unaligned tensor): plain loads, then a barrier
            if (g.g0 < p.lo_clip || ((g.ge + 15) & ~15ull) > p.hi_clip) {
                if (tid < 16 && !failed) {
                    const int l = tid < 8 ? tid : slice_n - 16 + tid;
                    if (l >= 0 && l < slice_n) {
                        const uint64_t a = g.gs + (uint64_t)l * ES;
                        if (a < g.lo || a + ES > g.hi) {
                            if (ES == 4)
                                *reinterpret_cast<uint32_t *>(slot + (a - g.g0)) =
                                    __ldg(reinterpret_cast<const unsigned int *>(a));
                            else
                                *reinterpret_cast<uint16_t *>(slot + (a - g.g0)) =
                                    __ldg(reinterpret_cast<const unsigned short *>(a));
                        }
                    }
                }
                __syncthreads();
            }

            // the slice into registers; -inf past it and outside it in the
            // (at most two) partial vectors
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                if (v < g.nv) xc[k] = lds128(slot + 16 * v);
            }
            if ((g.head_partial || g.tail_partial) && (tid == 0 || tid == (g.nv - 1) % NT)) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if ((v == 0 && g.head_partial) || (v == g.nv - 1 && g.tail_partial)) {
                        float z[W];
                        E::unpack(xc[k], z);
                        const int l0 = v * W - g.head;
#pragma unroll
                        for (int i = 0; i < W; ++i)
                            if ((unsigned)(l0 + i) >= (unsigned)slice_n) z[i] = -INFINITY;
                        xc[k] = E::pack(z);
                    }
                }
            }
            uint4 xt = kNeg;  // thread 0: the target's vector, masked likewise
            if (tid == 0 && has_t) {
                xt = lds128(slot + 16 * v_t);
                float z[W];
                E::unpack(xt, z);
                const int l0 = v_t * W - g.head;
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if ((unsigned)(l0 + i) >= (unsigned)slice_n) z[i] = -INFINITY;
                xt = E::pack(z);
                zt_sh[par] = E::load(slot + (size_t)tl * ES);
            }

            // Step 1: slice max
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < VPT; ++k) mx = fmaxf(mx, E::vmax(xc[k]));
            mx = warp_max(mx);
            if (lane == 0) red_max[par][warp] = mx;
            failed = __syncthreads_or(failed);  // the slot is free again
            if (tid == 0) {
                if (!failed && issued < nrows) {
                    fence_proxy_async();
                    issue(issued);
                    ++issued;
                }
                // every thread has passed its wait for row j-2: re-arm that
                // exchange slot for row j-2+NB
                if (j >= 2 && j - 2 + NB < nrows)
                    mbar_arrive_expect_tx(&xbar[(j - 2) % NB], (uint32_t)(K * sizeof(float4)));
            }
            float m = lane < NW ? red_max[par][lane] : -INFINITY;
            m = warp_max(m);
            const float M_loc = m * kLog2e;
            const float M_off = m == -INFINITY ? 0.f : M_loc;  // empty slice: any finite offset
            moff_cur = M_off;

            // Step 2: exponentials (fp32: in place) and their sum without the
            // target's vector; thread 0 adds that vector's other elements
            const unsigned long long nM2 = f2_pack(-M_off, -M_off);
            unsigned long long acc = 0ull;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                unsigned long long e2[W2];
                E::unpack2(xc[k], e2);
#pragma unroll
                for (int i = 0; i < W2; ++i) {
                    float a, b;
                    f2_unpack(f2_fma(e2[i], kL2E2, nM2), a, b);
                    e2[i] = f2_pack(ex2(a), ex2(b));
                }
                if (kKeepExp) xc[k] = E::pack2(e2);
                unsigned long long vs =
                    W2 == 4 ? f2_add(f2_add(e2[0], e2[1]), f2_add(e2[W2 - 2], e2[W2 - 1]))
                            : f2_add(e2[0], e2[W2 - 1]);
                if (v != v_t) acc = f2_add(acc, vs);
            }
            float sa, sb;
            f2_unpack(acc, sa, sb);
            if (tid == 0 && has_t) {
                float z[W];
                E::unpack(xt, z);
                const int d = tl - v_t * W;
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (i != d) sa += ex2(fmaf(z[i], kLog2e, -M_off));
            }
            const float ssum = warp_sum(sa + sb);

            // The last warp to finish (a shared-memory ticket) forms the CTA's
            // sum; its lane r pushes (M_r, S_r, z_t, has_t) to CTA r.
            unsigned int last = 0;
            if (lane == 0) {
                red_sum[par][warp] = ssum;
                __threadfence_block();
                last = atomicAdd(&warps_summed[par], 1u) == NW - 1u;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                float v = lane < NW ? *reinterpret_cast<volatile float *>(&red_sum[par][lane]) : 0.f;
                v = warp_sum(v);
                const float zt = has_t ? *reinterpret_cast<volatile float *>(&zt_sh[par]) : 0.f;
                if (lane == 0) warps_summed[par] = 0u;
                if (lane < K) {
                    const int b = (int)(j % NB);
                    st_async_f4(mapa(&xbuf[b][rank], (uint32_t)lane),
                                make_float4(M_loc, v, zt, has_t ? 1.f : 0.f),
                                mapa(&xbar[b], (uint32_t)lane));
                }
            }
        }

        // ============================================ B(j-1): gradient, loss
        if (j > 0) {
            const long long jp = j - 1;
            const long long row = cid + jp * ncl;
            const Geom g = geom(row);
            const long long t = t_prev;
            const bool has_loc = t >= c0 && t < c1;
            const int tl = has_loc ? (int)(t - c0) + g.head : kNoTarget;
            const int v_t = has_loc ? tl / W : -1;
            const int b = (int)(jp % NB);
            if (!xfailed) {
                if (!mbar_wait_cluster(&xbar[b], (uint32_t)((jp / NB) & 1))) {
                    xfailed = true;
                    failed = true;
                    atomicAdd(&p.err[kErrTimeout], 1);
                }
            }
            // combine the K partials in rank order (the same bits in every
            // warp of every CTA of the cluster)
            float4 q = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            if (lane < K) q = xbuf[b][lane];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < K; ++r) M = fmaxf(M, __shfl_sync(0xffffffffu, q.x, r));
            float S = 0.f, zt = 0.f;
            bool has_t = false;
#pragma unroll
            for (int r = 0; r < K; ++r) {
                const float Mr = __shfl_sync(0xffffffffu, q.x, r);
                const float Sr = __shfl_sync(0xffffffffu, q.y, r);
                const float zr = __shfl_sync(0xffffffffu, q.z, r);
                const float hr = __shfl_sync(0xffffffffu, q.w, r);
                if (Sr != 0.f) S += Sr * ex2(Mr - M);
                if (hr != 0.f) {
                    zt = zr;
                    has_t = true;
                }
            }
            const float s_rest = S;  // the row's sum without the target's term
            const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
            S = s_rest + e_t;

            // Step 4: gradient of the slice
            const float scale = (1.0f / S) * p.inv_b;
            const float escale = scale * ex2(moff_prev - M);
            const unsigned long long esc2 = f2_pack(escale, escale);
            const unsigned long long nM2 = f2_pack(-moff_prev, -moff_prev);
            const float g_t = -s_rest * scale;
            unsigned char *gbase = p.grad + (g.g0 - lbase);
            auto exps = [&](const uint4 &xv, unsigned long long (&e2)[W2]) {
                E::unpack2(xv, e2);
                if (!kKeepExp) {
#pragma unroll
                    for (int i = 0; i < W2; ++i) {
                        float a, bb;
                        f2_unpack(f2_fma(e2[i], kL2E2, nM2), a, bb);
                        e2[i] = f2_pack(ex2(a), ex2(bb));
                    }
                }
            };
            if (!failed) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if (v >= g.vf0 && v < g.vf1) {
                        unsigned long long g2[W2];
                        exps(xp[k], g2);
#pragma unroll
                        for (int i = 0; i < W2; ++i) g2[i] = f2_mul(g2[i], esc2);
                        if (vec_store) {
                            *reinterpret_cast<uint4 *>(gbase + 16 * v) = E::pack2(g2);
                        } else {
#pragma unroll
                            for (int i = 0; i < W2; ++i) {
                                float a, bb;
                                f2_unpack(g2[i], a, bb);
                                E::store(gbase + 16 * v + (2 * i) * ES, a);
                                E::store(gbase + 16 * v + (2 * i + 1) * ES, bb);
                            }
                        }
                        if (v == v_t) E::store(gbase + (size_t)tl * ES, g_t);
                    }
                }
                if ((g.head_partial || g.tail_partial) && (tid == 0 || tid == (g.nv - 1) % NT)) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        const int v = tid + k * NT;
                        if ((v == 0 && g.head_partial) || (v == g.nv - 1 && g.tail_partial)) {
                            const int l0 = v * W - g.head;
                            unsigned long long e2[W2];
                            exps(xp[k], e2);
#pragma unroll
                            for (int i = 0; i < W2; ++i) {
                                float a, bb;
                                f2_unpack(f2_mul(e2[i], esc2), a, bb);
                                if ((unsigned)(l0 + 2 * i) < (unsigned)slice_n)
                                    E::store(gbase + 16 * v + (2 * i) * ES,
                                             v * W + 2 * i == tl ? g_t : a);
                                if ((unsigned)(l0 + 2 * i + 1) < (unsigned)slice_n)
                                    E::store(gbase + 16 * v + (2 * i + 1) * ES,
                                             v * W + 2 * i + 1 == tl ? g_t : bb);
                            }
                        }
                    }
                }
            }
            // Step 3: the row's loss, by one thread of rank 0
            if (rank == 0 && tid == 0 && !failed) {
                float l;
                if (has_t) {
                    l = s_rest < e_t ? log1pf(s_rest / e_t)
                                     : kLn2 * (log2f(S) - fmaf(zt, kLog2e, -M));
                } else {
                    l = NAN;
                    atomicAdd(&p.err[kErrBadTarget], 1);
                }
                p.loss_rows[row] = l;
            }
        }

        // the current slice becomes the previous one
#pragma unroll
        for (int k = 0; k < VPT; ++k) xp[k] = xc[k];
        t_prev = t_cur;
        moff_prev = moff_cur;
    }

    // A CTA that gave up still owns copies in flight: wait for them (bounded)
    // before its shared memory is released.
    if (tid == 0 && failed) {
        for (long long j = consumed; j < issued; ++j) {
            if (!mbar_wait(&full[j % nslots], (uint32_t)((j / nslots) & 1))) break;
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still push into it
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, int K>
cudaError_t launch_k(const Params &p, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, cudaStream_t s) {
    auto kern = row_pipe_kernel<T, K, kSplitThreads, kPipeVecs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = K;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p, nslots, slot_bytes, se);
}

template <typename T, int K>
cudaError_t max_clusters_k(int smem, int *clusters) {
    auto kern = row_pipe_kernel<T, K, kSplitThreads, kPipeVecs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(K, 1, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
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

template <typename T>
cudaError_t launch_t(const Params &p, int K, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, cudaStream_t s) {
    switch (K) {
        case 2: return launch_k<T, 2>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 3: return launch_k<T, 3>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 4: return launch_k<T, 4>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 6: return launch_k<T, 6>(p, ctas, nslots, slot_bytes, se, smem, s);
        case 8: return launch_k<T, 8>(p, ctas, nslots, slot_bytes, se, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t max_clusters_t(int K, int smem, int *clusters) {
    switch (K) {
        case 2: return max_clusters_k<T, 2>(smem, clusters);
        case 3: return max_clusters_k<T, 3>(smem, clusters);
        case 4: return max_clusters_k<T, 4>(smem, clusters);
        case 6: return max_clusters_k<T, 6>(smem, clusters);
        case 8: return max_clusters_k<T, 8>(smem, clusters);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_split_pipe(const Params &p, int dtype, int K, int ctas, int nslots,
                              int slot_bytes, long long slice_elems, int smem, cudaStream_t s) {
    if (dtype == 0) return launch_t<float>(p, K, ctas, nslots, slot_bytes, slice_elems, smem, s);
    return launch_t<__nv_bfloat16>(p, K, ctas, nslots, slot_bytes, slice_elems, smem, s);
}

cudaError_t split_pipe_max_clusters(int dtype, int K, int smem, int *clusters) {
    if (dtype == 0) return max_clusters_t<float>(K, smem, clusters);
    return max_clusters_t<__nv_bfloat16>(K, smem, clusters);
}

}  // namespace ce
