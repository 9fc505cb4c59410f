// Pipelined split-row kernel: rows of K slices (K = 2, 3, 4, 6 or 8), one
// slice per CTA of a cluster of K, each slice of at most kSplitThreads x 8
// 16-byte vectors (64 KB), with no CTA-wide barrier per row.
//
// The row arithmetic is Pass 1 of rumus 0.1.1's cross_entropy.wgsl (Steps
// 1-4: max, sum of exponentials, loss, gradient) with the max and the sum
// taken in one pass by the running-max / rescaled-sum recurrence the rumus
// project page describes for its FlashAttention milestone (M17):
//
//   thread   m_t = max of its elements;  S_t = sum 2^(z*log2e - M_t),
//            M_t = m_t*log2e, the target's term left out;
//   warp     M_w = max M_t;  S_w = sum S_t 2^(M_t - M_w)   (shuffles)
//   CTA      M_r = max M_w;  S_r = sum S_w 2^(M_w - M_r)   (one publishing warp)
//   cluster  M = max M_r;    S = sum S_r 2^(M_r - M)       (every warp, rank order)
//   grad     e * 2^(M_t - M) / (S B), the target's element -S_rest / (S B)
//   loss     log(S / e_t)
//
// all sums in fixed orders.  The last CTA to finish sums the row losses (Pass
// 2, fused into the same launch).
//
// Schedule.  Iteration j of a CTA does
//
//   A(j)    wait for the slice of row j (TMA), read it into registers, M_t and
//           S_t, the warp's (M_w, S_w) into shared memory, then a non-blocking
//           arrive on a named barrier; the publishing warp alone waits there,
//           forms (M_r, S_r), pushes (M_r, S_r, z_t, has_t) into every CTA of
//           the cluster with st.async (completing transaction bytes on that
//           CTA's exchange mbarrier for row j) and hands the slot back to the
//           copy engine;
//   B(j-1)  wait for the K partials of row j-1 on the local exchange mbarrier
//           (pushed one iteration earlier), combine them, write the gradient
//           of row j-1 from the registers kept since A(j-1), and its loss.
//
// Warps only ever wait for data (a copy, or the partials of the row before),
// so the exchange latency and the skew between warps and CTAs hide behind
// A(j).  The registers hold two slices (the current and the previous row),
// hence 8 vectors per thread at most.
//
// Exchange buffers: NB = 4 slots of K float4 and one mbarrier each, slot
// j % NB for row j.  A CTA pushes row i only after its own B(i-2), which
// waited for every peer's row i-2, which each peer pushed only after
// finishing its iteration i-3 (and so reading row i-4's slot): when row i
// lands in a peer, rows up to i-4 have been read there and rows i-3 .. i
// occupy four distinct slots.  The mbarrier of slot (i % NB) is re-armed for
// row i (expect K x 16 bytes, one local arrival) by the publishing warp in
// A(i-2), once every warp has arrived for row i-2 (so every thread has passed
// its wait for row i-4, in B(i-4)) and before this CTA pushes row i-2 (which
// precedes any peer's push of row i).  The named barriers alternate by row
// parity: a warp cannot arrive for row j+2 before B(j), which needs the
// publisher's push of row j, which follows its wait for row j.
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

constexpr int kExchangeSlots = 4;

// A vector's exponentials as fp32 pairs: the vector itself when it already
// holds them (fp32 rows), else 2^(z*log2e - M_t) from its logits.
template <typename E, bool kHeld, int W2>
__device__ __forceinline__ void exps_of(const uint4 &xv, unsigned long long (&e2)[W2],
                                        unsigned long long l2e2, unsigned long long nm2) {
    E::unpack2(xv, e2);
    if (!kHeld) {
#pragma unroll
        for (int i = 0; i < W2; ++i) {
            float a, b;
            f2_unpack(f2_fma(e2[i], l2e2, nm2), a, b);
            e2[i] = f2_pack(ex2(a), ex2(b));
        }
    }
}

template <typename T, int K, int NT, int VPT, typename P>
__global__ void __launch_bounds__(NT, 1)
    row_pipe_kernel(P p, int nslots, int slot_bytes, long long SE) {
    using E = Elem<T>;
    constexpr int NW = NT / 32;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr int ES = E::kBytes;
    constexpr int NB = kExchangeSlots;
    constexpr int kPub = NW - 1;       // the publishing warp
    constexpr int kLossWarp = NW / 2;  // its lane 0 (in rank 0) writes the row losses
    constexpr int kNoTarget = -0x40000000;
    constexpr bool kKeepExp = sizeof(T) == 4;  // fp32: exponentials overwrite the logits
    static_assert(K >= 2 && K <= 32 && NW >= 2, "shape");

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kMaxSplitSlots];
    __shared__ uint64_t xbar[NB];
    __shared__ __align__(16) float4 xbuf[NB][K];  // [row slot][source rank]
    __shared__ float2 red[2][NW];                 // (M_w, S_w) by row parity
    __shared__ float zt_sh[2];
    __shared__ int cta_failed;
    __shared__ float2 tail_scratch[kTailWarps];
    __shared__ int tail_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    // rows, classes and targets fit in int (B, C < 2^31); only element
    // offsets (row * C) need 64 bits
    const int cid = (int)cluster_id_x();
    const int ncl = (int)cluster_count_x();
    const long long C = p.C;
    const int c0 = (int)min((long long)rank * SE, C);
    const int c1 = (int)min((long long)c0 + SE, C);
    const int slice_n = c1 - c0;
    const int nrows = cid < p.B ? (int)((p.B - cid + ncl - 1) / ncl) : 0;
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    const bool vec_store = p.grad_vec_ok != 0;
    const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);
    const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                  E::kNegInfWord);

    // Where this CTA's slice of a row sits.  e0 = the row's first element of
    // the slice; vector v of the slot holds local elements v*W - head ..
    // v*W - head + W - 1 (16-byte aligned in global memory); whole vectors
    // are [vf0, vf1); the others are partial.
    struct Geom {
        long long e0;
        int head, nv, vf0, vf1;
        bool head_partial, tail_partial;
    };
    auto geom = [&](int row) {
        Geom g;
        g.e0 = (long long)row * C + c0;
        const uint32_t b0 = ((uint32_t)lbase + (uint32_t)g.e0 * ES) & 15u;  // gs mod 16
        g.head = (int)(b0 / ES);
        const uint32_t end = b0 + (uint32_t)slice_n * ES;  // ge - g0
        g.nv = (int)((end + 15u) >> 4);
        g.vf0 = g.head != 0 ? 1 : 0;
        g.vf1 = (end & 15u) != 0 ? g.nv - 1 : g.nv;
        g.head_partial = g.vf0 == 1;
        g.tail_partial = g.vf1 == g.nv - 1 && g.nv - 1 >= g.vf0;
        return g;
    };
    auto issue = [&](int j, int s) {  // row j of this cluster into slot s
        if (skips_copy(p, cid + j * ncl, cid + j * ncl + 1)) return;  // test hook
        const Geom g = geom(cid + j * ncl);
        const uint64_t g0 = lbase + (uint64_t)g.e0 * ES - (uint64_t)g.head * ES;
        const uint64_t lo = g0 > p.lo_clip ? g0 : p.lo_clip;
        const uint64_t ghi = g0 + 16ull * (uint64_t)g.nv;
        const uint64_t hi = ghi < p.hi_clip ? ghi : p.hi_clip;
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
        for (int b = 0; b < NB; ++b) mbar_init(&xbar[b], 1);
        fence_mbar_init();
        cta_failed = 0;
    }
    pdl_trigger();
    pdl_wait();  // nothing above touched global memory
    const float gsc = scalar_grad_scale(p);
    // every CTA's exchange mbarriers exist before any peer pushes into them
    cluster_sync();

    const bool issuer = warp == kPub && lane == 0;
    int issued = 0;        // issuer: rows whose copy was issued
    int s_issue = 0;       // issuer: slot of the next copy
    if (issuer) {
        for (int b = 0; b < NB && b < nrows; ++b)
            mbar_arrive_expect_tx(&xbar[b], (uint32_t)(K * sizeof(float4)));
        for (; issued < nrows && issued < nslots; ++issued) issue(issued, (int)issued);
        s_issue = issued % nslots;
    }

    bool failed = false;   // this thread saw a wait give up
    int consumed = 0;
    int s_cur = 0;         // slot and phase parity of the next row to consume
    uint32_t ph_cur = 0;
    int t_next = nrows > 0 ? target_at(p, cid) : 0;

    auto fail = [&]() {  // one timeout counted per CTA
        failed = true;
        if (atomicExch(&cta_failed, 1) == 0) atomicAdd(&p.err[kErrTimeout], 1);
    };

    // ---------------------------------------------------------------- A(j)
    auto stage_a = [&](int j, uint4 (&x)[VPT], float &off, bool &hv, int &t_out) {
        const int row = cid + j * ncl;
        const int par = j & 1;
        const int t = t_next;
        t_out = t;
        if (j + 1 < nrows) t_next = target_at(p, row + ncl);
        const Geom g = geom(row);
        const bool has_t = t >= c0 && t < c1;
        const int tl = has_t ? t - c0 + g.head : kNoTarget;  // target, vector-0 based
        const int v_t = has_t ? tl / W : -1;
        unsigned char *slot = smem + (size_t)s_cur * slot_bytes;

        if (!failed) {
            if (mbar_wait(&full[s_cur], ph_cur, copy_wait_limit(p)))
                consumed = j + 1;
            else
                fail();
        }
        if (++s_cur == nslots) {
            s_cur = 0;
            ph_cur ^= 1u;
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * NT;
            x[k] = v < g.nv ? lds128(slot + 16 * v) : kNeg;
        }
        // Owners of the partial vectors: -inf outside the slice; at the very
        // beginning or end of an unaligned tensor, the elements the copy could
        // not cover come from plain loads.
        if ((g.head_partial || g.tail_partial) && (tid == 0 || tid == (g.nv - 1) % NT)) {
            const uint64_t g0 = lbase + (uint64_t)g.e0 * ES - (uint64_t)g.head * ES;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                if ((v == 0 && g.head_partial) || (v == g.nv - 1 && g.tail_partial)) {
                    float z[W];
                    E::unpack(x[k], z);
                    const int l0 = v * W - g.head;
#pragma unroll
                    for (int i = 0; i < W; ++i) {
                        if ((unsigned)(l0 + i) >= (unsigned)slice_n) {
                            z[i] = -INFINITY;
                        } else {
                            const uint64_t a = g0 + 16ull * v + (uint64_t)i * ES;
                            if (a < p.lo_clip || a + ES > p.hi_clip)
                                z[i] = E::load_global(reinterpret_cast<const unsigned char *>(a));
                        }
                    }
                    x[k] = E::pack(z);
                }
            }
        }

        // Step 1 (per thread): m_t.  Vectors past the slice hold -inf and
        // are skipped here and below (they would only add zeros), so a short
        // slice costs only its own vectors.
        typename E::MaxAcc macc = E::max_init();
#pragma unroll
        for (int k = 0; k < VPT; ++k)
            if (tid + k * NT < g.nv) E::max_step(macc, x[k]);
        const float mx = E::max_value(macc);
        const float Mx = mx * kLog2e;  // -inf when the thread holds no element
        hv = mx != -INFINITY;
        off = hv ? Mx : 0.f;
        const unsigned long long nM2 = f2_pack(-off, -off);

        // Step 2 (per thread): exponentials and their sum without the
        // target's term; the owner of the target's vector sums its other
        // elements and records z_t.
        unsigned long long acc = 0ull;
        float s_t = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * NT;
            if (v >= g.nv) continue;
            unsigned long long e2[W2];
            E::unpack2(x[k], e2);
            if (v == v_t) zt_sh[par] = element_of<E>(x[k], tl - v * W);
#pragma unroll
            for (int i = 0; i < W2; ++i) {
                float a, b;
                f2_unpack(f2_fma(e2[i], kL2E2, nM2), a, b);
                e2[i] = f2_pack(ex2(a), ex2(b));
            }
            if (kKeepExp) x[k] = E::pack2(e2);
            if (v != v_t) {
                const unsigned long long vs =
                    W2 == 4 ? f2_add(f2_add(e2[0], e2[1]), f2_add(e2[W2 - 2], e2[W2 - 1]))
                            : f2_add(e2[0], e2[W2 - 1]);
                acc = f2_add(acc, vs);
            } else {
                const int d = tl - v * W;
#pragma unroll
                for (int i = 0; i < W2; ++i) {
                    float a, b;
                    f2_unpack(e2[i], a, b);
                    if (2 * i != d) s_t += a;
                    if (2 * i + 1 != d) s_t += b;
                }
            }
        }
        {
            float sa, sb;
            f2_unpack(acc, sa, sb);
            s_t += sa + sb;
        }

        // warp partial (M_w, S_w)
        const float Mw = warp_max(Mx);
        float sw = s_t != 0.f ? s_t * ex2(off - Mw) : 0.f;
        sw = warp_sum(sw);
        if (lane == 0) red[par][warp] = make_float2(Mw, sw);
        if (warp != kPub) {
            named_arrive(1 + par, NT);
        } else {
            named_sync(1 + par, NT);  // every warp is done with the slot and has its partial in
            const float2 q = lane < NW ? red[par][lane] : make_float2(-INFINITY, 0.f);
            const float Mc = warp_max(q.x);
            float sc = q.y != 0.f ? q.y * ex2(q.x - Mc) : 0.f;
            sc = warp_sum(sc);
            // a CTA that gave up publishes a NaN sum: every CTA of the cluster
            // then computes NaN rows (loss and gradient) from here on
            if (*reinterpret_cast<volatile int *>(&cta_failed)) sc = NAN;
            const float zt = has_t ? zt_sh[par] : 0.f;
            // re-arm the exchange slot of row j-2 for row j-2+NB before this
            // CTA's push of row j (which any peer's push of row j-2+NB follows)
            if (lane == 0 && j >= 2 && j - 2 + NB < nrows)
                mbar_arrive_expect_tx(&xbar[(j - 2) & (NB - 1)], (uint32_t)(K * sizeof(float4)));
            __syncwarp();
            if (lane < K) {
                const int b = j & (NB - 1);
                st_async_f4(mapa(&xbuf[b][rank], (uint32_t)lane),
                            make_float4(Mc, sc, zt, has_t ? 1.f : 0.f),
                            mapa(&xbar[b], (uint32_t)lane));
            }
            if (lane == 0 && !cta_failed && issued < nrows) {
                fence_proxy_async();  // the slot was read through the generic proxy
                issue(issued, s_issue);
                ++issued;
                if (++s_issue == nslots) s_issue = 0;
            }
        }
    };

    // -------------------------------------------------------------- B(j-1)
    auto stage_b = [&](int jp, const uint4 (&x)[VPT], float off, bool hv, int t) {
        const int row = cid + jp * ncl;
        const Geom g = geom(row);
        const bool has_loc = t >= c0 && t < c1;
        const int tl = has_loc ? t - c0 + g.head : kNoTarget;
        const int v_t = has_loc ? tl / W : -1;
        const int b = jp & (NB - 1);
        if (!failed && !mbar_wait_cluster(&xbar[b], (uint32_t)((jp >> 2) & 1))) fail();
        // combine the K partials in rank order (the same bits in every warp
        // of every CTA of the cluster)
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
        const float scale = fast_rcp(S) * row_grad_factor(p, gsc, row);
        // a thread without elements has nothing to scale (and M_t = 0 is not
        // an upper bound of anything)
        const float escale = hv ? scale * ex2(off - M) : 0.f;
        const unsigned long long esc2 = f2_pack(escale, escale);
        const unsigned long long nM2 = f2_pack(-off, -off);
        const float g_t = -s_rest * scale;
        unsigned char *gbase = p.grad + ((uint64_t)g.e0 - (uint64_t)g.head) * ES;
        const bool skip = failed || *reinterpret_cast<volatile int *>(&cta_failed) != 0;
        if (!skip && writes_grad(p)) {  // else loss only
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                if (v >= g.vf0 && v < g.vf1) {
                    unsigned long long g2[W2];
                    exps_of<E, kKeepExp>(x[k], g2, kL2E2, nM2);
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
            // test hook: the whole vectors' fp32 values, before their rounding
            // (recomputed here so that the loop above carries none of it)
            if (grad_f32_of(p)) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if (v >= g.vf0 && v < g.vf1) {
                        unsigned long long g2[W2];
                        exps_of<E, kKeepExp>(x[k], g2, kL2E2, nM2);
#pragma unroll
                        for (int i = 0; i < W2; ++i) {
                            float a, bb;
                            f2_unpack(f2_mul(g2[i], esc2), a, bb);
                            grad_f32_store<ES>(p, gbase + 16 * v + (2 * i) * ES, a);
                            grad_f32_store<ES>(p, gbase + 16 * v + (2 * i + 1) * ES, bb);
                        }
                        if (v == v_t) grad_f32_store<ES>(p, gbase + (size_t)tl * ES, g_t);
                    }
                }
            }
            if ((g.head_partial || g.tail_partial) && (tid == 0 || tid == (g.nv - 1) % NT)) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if ((v == 0 && g.head_partial) || (v == g.nv - 1 && g.tail_partial)) {
                        const int l0 = v * W - g.head;
                        unsigned long long e2[W2];
                        exps_of<E, kKeepExp>(x[k], e2, kL2E2, nM2);
#pragma unroll
                        for (int i = 0; i < W2; ++i) {
                            float a, bb;
                            f2_unpack(f2_mul(e2[i], esc2), a, bb);
                            if (v * W + 2 * i == tl) a = g_t;
                            if (v * W + 2 * i + 1 == tl) bb = g_t;
                            if ((unsigned)(l0 + 2 * i) < (unsigned)slice_n) {
                                E::store(gbase + 16 * v + (2 * i) * ES, a);
                                grad_f32_store<ES>(p, gbase + 16 * v + (2 * i) * ES, a);
                            }
                            if ((unsigned)(l0 + 2 * i + 1) < (unsigned)slice_n) {
                                E::store(gbase + 16 * v + (2 * i + 1) * ES, bb);
                                grad_f32_store<ES>(p, gbase + 16 * v + (2 * i + 1) * ES, bb);
                            }
                        }
                    }
                }
            }
        }
        // Step 3: the row's loss, by one thread of rank 0 (NaN for a row this
        // CTA did not compute)
        if (rank == 0 && warp == kLossWarp && lane == 0 && !is_softmax(p)) {
            float l;
            if (skip) {
                l = NAN;
            } else if (has_t) {
                l = row_loss(s_rest, e_t, S, zt, M);
            } else {
                l = NAN;
                atomicAdd(&p.err[kErrBadTarget], 1);
            }
            p.loss_rows[row] = l;
        }
    };

    // A(j) fills one register set while B(j-1) drains the other; one copy of
    // each stage's code (the instruction cache holds the loop)
    uint4 xp[VPT];
    float offp = 0.f;
    bool hvp = false;
    int tp = 0;
#pragma unroll
    for (int k = 0; k < VPT; ++k) xp[k] = kNeg;
    for (int j = 0; j <= nrows; ++j) {
        uint4 xc[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) xc[k] = kNeg;
        float offc = 0.f;
        bool hvc = false;
        int tc = 0;
        if (j < nrows) stage_a(j, xc, offc, hvc, tc);
        if (j > 0) stage_b(j - 1, xp, offp, hvp, tp);
#pragma unroll
        for (int k = 0; k < VPT; ++k) xp[k] = xc[k];
        offp = offc;
        hvp = hvc;
        tp = tc;
    }

    // A CTA that gave up still owns copies in flight: the issuer waits for
    // them (each for up to the full limit) before its shared memory is
    // released.  A copy that has not landed after that never will; the CTA
    // then leaves rather than hang.
    if (issuer && (failed || cta_failed)) {
        for (int j = consumed; j < issued; ++j) {
            if (skips_copy(p, cid + j * ncl, cid + j * ncl + 1)) continue;  // never issued
            if (!mbar_wait(&full[j % nslots], (uint32_t)((j / nslots) & 1))) break;
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still push into it
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, int K, typename P>
cudaError_t launch_kp(const P &p, int ctas, int nslots, int slot_bytes, long long se,
                      int smem, cudaStream_t s) {
    auto kern = row_pipe_kernel<T, K, kSplitThreads, kPipeVecs, P>;
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

// The plain call runs the Params build, any other the ParamsEx build.
template <typename T, int K>
cudaError_t launch_k(const ParamsEx &p, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, cudaStream_t s) {
    if (is_plain(p))
        return launch_kp<T, K, Params>(static_cast<const Params &>(p), ctas, nslots, slot_bytes,
                                       se, smem, s);
    return launch_kp<T, K, ParamsEx>(p, ctas, nslots, slot_bytes, se, smem, s);
}

template <typename T, int K>
cudaError_t max_clusters_k(int smem, int *clusters) {
    auto kern = row_pipe_kernel<T, K, kSplitThreads, kPipeVecs, Params>;
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
cudaError_t launch_t(const ParamsEx &p, int K, int ctas, int nslots, int slot_bytes, long long se,
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

cudaError_t launch_split_pipe(const ParamsEx &p, int dtype, int K, int ctas, int nslots,
                              int slot_bytes, long long slice_elems, int smem, cudaStream_t s) {
    if (dtype == 0) return launch_t<float>(p, K, ctas, nslots, slot_bytes, slice_elems, smem, s);
    if (dtype == 2) return launch_t<__half>(p, K, ctas, nslots, slot_bytes, slice_elems, smem, s);
    return launch_t<__nv_bfloat16>(p, K, ctas, nslots, slot_bytes, slice_elems, smem, s);
}

cudaError_t split_pipe_max_clusters(int dtype, int K, int smem, int *clusters) {
    if (dtype == 0) return max_clusters_t<float>(K, smem, clusters);
    if (dtype == 2) return max_clusters_t<__half>(K, smem, clusters);
    return max_clusters_t<__nv_bfloat16>(K, smem, clusters);
}

}  // namespace ce
