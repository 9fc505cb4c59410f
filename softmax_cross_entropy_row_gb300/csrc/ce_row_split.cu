// Split-row kernel: each row of the logits crosses HBM exactly once.
//
// A cluster of K CTAs (K = 1, 2, 3, 4, 6 or 8) owns a row at a time; CTA `rank`
// holds the slice [rank*SE, (rank+1)*SE) of the row's classes.  Each CTA keeps
// a ring of `nslots` shared-memory slots filled by TMA bulk copies, so the
// copies of the next rows are in flight while it computes the current one (a
// persistent grid: cluster c takes rows c, c + nclusters, ...).
//
// A slice is read from shared memory once, into registers (VPT 16-byte
// vectors per thread); its slot is handed back to the copy engine right after
// the first block reduction.  fp32 exponentials then replace the logits in
// those registers; bf16 rows keep their logits and evaluate each exponential
// again for the gradient.  From the registers each CTA computes
//
//   Step 1  m_r = max over the slice                         (block max)
//   Step 2  e = 2^(z*log2e - M_r), M_r = m_r*log2e;
//           S_r = sum of e over the slice, the target left out (block sum)
//   combine M = max_r M_r,  S = sum_r S_r * 2^(M_r - M)      (over DSMEM, K > 1)
//   Step 4  grad = e * 2^(M_r - M) / (S B), target: -S_rest / (S B)
//   Step 3  l_b = log(S / e_t)                                (rank 0)
//
// which are Steps 1-4 of Pass 1 of rumus 0.1.1's cross_entropy.wgsl, with the
// split-row combine being the running-max / rescaled-sum recurrence the rumus
// project page describes for its FlashAttention milestone (M17), applied to
// the cross-entropy row.  The last CTA to finish sums the row losses in a
// fixed order (Pass 2, fused into the same launch).
#include <math.h>

#include <type_traits>

#include "ce_launch.h"

namespace ce {
namespace {

template <typename T, int K, int NT, int VPT, typename P>
__global__ void __launch_bounds__(NT, 1)
    row_split_kernel(P p, int nslots, int slot_bytes, long long SE, int staged) {
    using E = Elem<T>;
    constexpr int NW = NT / 32;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;  // fp32 pairs per vector
    constexpr int ES = E::kBytes;
    constexpr int kNoTarget = -0x40000000;
    constexpr bool kKeepExp = sizeof(T) == 4;  // fp32: exponentials overwrite the logits in registers

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kMaxSplitSlots];
    __shared__ float red_max[2][NW];   // per warp, by row parity
    __shared__ float red_sum[2][NW];
    __shared__ float zt_sh[2];
    __shared__ float4 part[2];         // this CTA's (M, S, z_t, has_t) for the cluster
    __shared__ unsigned int warps_summed[2];
    __shared__ float2 tail_scratch[kTailWarps];
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
    // Staged gradient: each thread writes its whole vectors' gradient over
    // their logits in the slot, and the row leaves in one TMA bulk store; the
    // slot is handed back to the copy engine one row later, once read out.
    const bool write_grad = writes_grad(p);  // false: loss only
    const bool stage = staged != 0 && vec_store && write_grad;
    const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);

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
    auto issue = [&](long long j, int s) {  // row j of this cluster into slot s
        uint64_t gs, ge, g0, lo, hi;
        if (skips_copy(p, cid + j * ncl, cid + j * ncl + 1)) return;  // test hook
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
        warps_summed[0] = warps_summed[1] = 0u;
    }
    pdl_trigger();
    pdl_wait();  // nothing above touched global memory
    const float gsc = scalar_grad_scale(p);
    __syncthreads();
    long long issued = 0;
    int s_iss = 0;  // slot of the next copy
    if (tid == 0) {
        for (; issued < nrows && issued < nslots; ++issued) issue(issued, (int)issued);
        s_iss = issued == nslots ? 0 : (int)issued;
    }
    int s = 0;            // slot and phase parity of the next row
    uint32_t parity = 0;

    bool failed = false;      // this thread saw a copy wait give up
    bool failed_cta = false;  // some thread of the CTA did (uniform)
    long long consumed = 0;
    int t_next = nrows > 0 ? target_at(p, cid) : 0;

    for (long long j = 0; j < nrows; ++j) {
        const long long row = cid + j * ncl;
        const int par = (int)(j & 1);
        unsigned char *slot = smem + (size_t)s * slot_bytes;
        uint64_t *slot_full = &full[s];
        const uint32_t slot_parity = parity;
        if (++s == nslots) {
            s = 0;
            parity ^= 1u;
        }
        const long long t = t_next;
        if (j + 1 < nrows) t_next = target_at(p, row + ncl);

        uint64_t gs, ge, g0, lo, hi;
        span(row, gs, ge, g0, lo, hi);
        // Vector v of the slot holds the slice's local elements v*W - head ..
        // v*W - head + W - 1; local element l is valid for 0 <= l < slice_n.
        const int head = (int)((gs - g0) / ES);
        const int nv = (int)((((ge + 15) & ~15ull) - g0) >> 4);
        const int vf0 = head != 0 ? 1 : 0;                     // whole vectors: [vf0, vf1)
        const int vf1 = (ge & 15ull) != 0 ? nv - 1 : nv;
        const bool head_partial = vf0 == 1;
        const bool tail_partial = vf1 == nv - 1 && nv - 1 >= vf0;
        bool has_t = t >= c0 && t < c1;
        const int tl = has_t ? (int)(t - c0) + head : kNoTarget;  // target, vector-0 based
        const int v_t = has_t ? tl / W : -1;                       // the target's vector

        if (!failed) {
            if (mbar_wait(slot_full, slot_parity, copy_wait_limit(p)))
                consumed = j + 1;
            else
                failed = true;  // made CTA-wide (and counted) at the next barrier
        }
        // Elements the copy could not cover (only at the very beginning or end
        // of an unaligned tensor): plain loads, then a barrier before use.
        if (g0 < p.lo_clip || ((ge + 15) & ~15ull) > p.hi_clip) {
            if (tid < 16 && !failed) {
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

        // ---- the slice into registers; vectors past it and the elements of
        // the (at most two) partial vectors outside it read as -inf
        const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                      E::kNegInfWord);
        uint4 x[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * NT;
            x[k] = kNeg;
            if (v < nv) x[k] = lds128(slot + 16 * v);
        }
        if ((head_partial || tail_partial) && (tid == 0 || tid == (nv - 1) % NT)) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                if ((v == 0 && head_partial) || (v == nv - 1 && tail_partial)) {
                    float z[W];
                    E::unpack(x[k], z);
                    const int l0 = v * W - head;
#pragma unroll
                    for (int i = 0; i < W; ++i)
                        if ((unsigned)(l0 + i) >= (unsigned)slice_n) z[i] = -INFINITY;
                    x[k] = E::pack(z);
                }
            }
        }
        // thread 0 also takes the target's vector (masked the same way)
        uint4 xt = kNeg;
        if (tid == 0 && has_t) {
            xt = lds128(slot + 16 * v_t);
            float z[W];
            E::unpack(xt, z);
            const int l0 = v_t * W - head;
#pragma unroll
            for (int i = 0; i < W; ++i)
                if ((unsigned)(l0 + i) >= (unsigned)slice_n) z[i] = -INFINITY;
            xt = E::pack(z);
            zt_sh[par] = E::load(slot + (size_t)tl * ES);
        }

        // ---- Step 1: slice max
        typename E::MaxAcc macc = E::max_init();
#pragma unroll
        for (int k = 0; k < VPT; ++k) E::max_step(macc, x[k]);
        float mx = E::max_value(macc);
        mx = warp_max(mx);
        if (lane == 0) red_max[par][warp] = mx;
        {
            const bool was = failed_cta;
            failed = failed_cta = __syncthreads_or(failed);
            if (failed && !was && tid == 0) atomicAdd(&p.err[kErrTimeout], 1);
        }
        if (tid == 0 && !failed && issued < nrows) {
            if (stage) {
                // the slot of row j-1 comes back once its gradient has been
                // read out by the copy engine
                if (j > 0) {
                    bulk_wait_read_all();
                    fence_proxy_async();
                    issue(issued, s_iss);
                    ++issued;
                    if (++s_iss == nslots) s_iss = 0;
                }
            } else {
                // the slot is no longer read: back to the copy engine
                fence_proxy_async();
                issue(issued, s_iss);
                ++issued;
                if (++s_iss == nslots) s_iss = 0;
            }
        }
        float m = lane < NW ? red_max[par][lane] : -INFINITY;
        m = warp_max(m);
        // An empty slice (C < K*SE) has m = -inf: it publishes M = -inf, S = 0
        // and takes a finite offset for its (absent) exponentials.
        const float M_loc = m * kLog2e;
        const float M_off = m == -INFINITY ? 0.f : M_loc;
        float zt = has_t ? zt_sh[par] : 0.f;

        // ---- Step 2: exponentials kept in registers (fp32 pairs); their sum
        // without the target's term (added back after the combine, so that
        // 1 - p_t keeps its relative precision when the target dominates the
        // row).  The target's vector is left out whole; thread 0 adds its other
        // elements.
        const unsigned long long nM2 = f2_pack(-M_off, -M_off);
        unsigned long long acc = 0ull;  // (0.f, 0.f)
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * NT;
            unsigned long long e2[W2];
            E::unpack2(x[k], e2);
#pragma unroll
            for (int i = 0; i < W2; ++i) {
                float a, b;
                f2_unpack(f2_fma(e2[i], kL2E2, nM2), a, b);
                e2[i] = f2_pack(ex2(a), ex2(b));
            }
            if (kKeepExp) x[k] = E::pack2(e2);  // fp32: the exponentials replace the logits
            unsigned long long vs = W2 == 4 ? f2_add(f2_add(e2[0], e2[1]), f2_add(e2[W2 - 2], e2[W2 - 1]))
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

        float M = M_loc;
        float S;
        if (K == 1) {
            if (lane == 0) red_sum[par][warp] = ssum;
            if (!write_grad && !is_softmax(p)) {
                // the loss alone: only warp 0 (the loss's writer) needs the
                // row's sum, so the other warps arrive without waiting and go
                // on to the next row (whose first barrier warp 0 reaches only
                // once this row's loss is written)
                if (warp != 0) {
                    named_arrive(1, NT);
                    continue;
                }
                named_sync(1, NT);
            } else {
                __syncthreads();
            }
            S = lane < NW ? red_sum[par][lane] : 0.f;
            S = warp_sum(S);
        } else {
            // The last warp of the CTA to finish its sum (a shared-memory
            // ticket) forms the CTA's total and publishes (M_r, S_r, z_t) to the
            // cluster; it alone arrives with release semantics.  After one
            // cluster barrier every warp combines the K ranks in rank order
            // (the same bits in every warp of every CTA).
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
                if (lane == 0) {
                    // a CTA that gave up publishes a NaN sum: every CTA of the
                    // cluster then computes a NaN row (loss and gradient)
                    part[par] = make_float4(M_loc, failed ? NAN : v, zt, has_t ? 1.f : 0.f);
                    warps_summed[par] = 0u;
                }
                __syncwarp();
                cluster_arrive_release();
            } else {
                cluster_arrive_relaxed();
            }
            cluster_wait();
            float4 q = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            if (lane < K) q = ld_dsmem_f4(&part[par], (uint32_t)lane);
            float Mg = -INFINITY;
#pragma unroll
            for (int r = 0; r < K; ++r) Mg = fmaxf(Mg, __shfl_sync(0xffffffffu, q.x, r));
            float Sg = 0.f, ztg = 0.f;
            bool hg = false;
#pragma unroll
            for (int r = 0; r < K; ++r) {
                const float Mr = __shfl_sync(0xffffffffu, q.x, r);
                const float Sr = __shfl_sync(0xffffffffu, q.y, r);
                const float zr = __shfl_sync(0xffffffffu, q.z, r);
                const float hr = __shfl_sync(0xffffffffu, q.w, r);
                if (Sr != 0.f) Sg += Sr * ex2(Mr - Mg);
                if (hr != 0.f) {
                    ztg = zr;
                    hg = true;
                }
            }
            M = Mg;
            S = Sg;
            zt = ztg;
            has_t = hg;
        }
        // S holds the row's sum without the target's term: S_rest = S (1 - p_t).
        const float s_rest = S;
        const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
        S = s_rest + e_t;

        // ---- Step 4: gradient of the slice
        const float scale = fast_rcp(S) * row_grad_factor(p, gsc, row);
        const float escale = K > 1 ? scale * ex2(M_off - M) : scale;
        const unsigned long long esc2 = f2_pack(escale, escale);
        // (p_t - 1) / B = -S_rest / (S B): no cancellation when p_t is near 1
        const float g_t = -s_rest * scale;
        unsigned char *gbase = p.grad + (g0 - lbase);  // grad byte of vector 0
        // The slice's exponentials as fp32 pairs: held in x for fp32 rows,
        // evaluated again from the raw bf16 logits otherwise.  Nothing is
        // written when only the loss is wanted.
        auto exps = [&](const uint4 &xv, unsigned long long (&e2)[W2]) {
            E::unpack2(xv, e2);
            if (!kKeepExp) {
#pragma unroll
                for (int i = 0; i < W2; ++i) {
                    float a, b;
                    f2_unpack(f2_fma(e2[i], kL2E2, nM2), a, b);
                    e2[i] = f2_pack(ex2(a), ex2(b));
                }
            }
        };
        if (!failed && write_grad) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = tid + k * NT;
                if (v >= vf0 && v < vf1) {
                    unsigned long long g2[W2];
                    exps(x[k], g2);
#pragma unroll
                    for (int i = 0; i < W2; ++i) g2[i] = f2_mul(g2[i], esc2);
                    if (stage) {
                        // in place of the vector's logits, which this thread alone read
                        *reinterpret_cast<uint4 *>(slot + 16 * v) = E::pack2(g2);
                        if (v == v_t) E::store(slot + (size_t)tl * ES, g_t);
                    } else if (vec_store) {
                        *reinterpret_cast<uint4 *>(gbase + 16 * v) = E::pack2(g2);
                    } else {
#pragma unroll
                        for (int i = 0; i < W2; ++i) {
                            float a, b;
                            f2_unpack(g2[i], a, b);
                            E::store(gbase + 16 * v + (2 * i) * ES, a);
                            E::store(gbase + 16 * v + (2 * i + 1) * ES, b);
                        }
                    }
                    // the owner of the target's vector overwrites the target
                    if (!stage && v == v_t) E::store(gbase + (size_t)tl * ES, g_t);
                }
            }
            // test hook: the whole vectors' fp32 values, before their rounding
            // (recomputed here so that the loop above carries none of it)
            if (grad_f32_of(p)) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if (v >= vf0 && v < vf1) {
                        unsigned long long g2[W2];
                        exps(x[k], g2);
#pragma unroll
                        for (int i = 0; i < W2; ++i) {
                            float a, b;
                            f2_unpack(f2_mul(g2[i], esc2), a, b);
                            grad_f32_store<ES>(p, gbase + 16 * v + (2 * i) * ES, a);
                            grad_f32_store<ES>(p, gbase + 16 * v + (2 * i + 1) * ES, b);
                        }
                        if (v == v_t) grad_f32_store<ES>(p, gbase + (size_t)tl * ES, g_t);
                    }
                }
            }
            // the partial vectors: element by element, by their owners
            if ((head_partial || tail_partial) && (tid == 0 || tid == (nv - 1) % NT)) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = tid + k * NT;
                    if ((v == 0 && head_partial) || (v == nv - 1 && tail_partial)) {
                        const int l0 = v * W - head;
                        unsigned long long e2[W2];
                        exps(x[k], e2);
#pragma unroll
                        for (int i = 0; i < W2; ++i) {
                            float a, b;
                            f2_unpack(f2_mul(e2[i], esc2), a, b);
                            if (v * W + 2 * i == tl) a = g_t;
                            if (v * W + 2 * i + 1 == tl) b = g_t;
                            if ((unsigned)(l0 + 2 * i) < (unsigned)slice_n) {
                                E::store(gbase + 16 * v + (2 * i) * ES, a);
                                grad_f32_store<ES>(p, gbase + 16 * v + (2 * i) * ES, a);
                            }
                            if ((unsigned)(l0 + 2 * i + 1) < (unsigned)slice_n) {
                                E::store(gbase + 16 * v + (2 * i + 1) * ES, b);
                                grad_f32_store<ES>(p, gbase + 16 * v + (2 * i + 1) * ES, b);
                            }
                        }
                    }
                }
            }
        }

        if (stage) {
            // the whole vectors leave in one bulk store once every thread's
            // writes are visible to the copy engine
            fence_proxy_async();
            failed = __syncthreads_or(failed);
            if (tid == 0 && !failed && vf1 > vf0) {
                bulk_s2g(gbase + 16 * vf0, slot + 16 * vf0, (uint32_t)(16 * (vf1 - vf0)));
                bulk_commit();
            }
        }

        // ---- Step 3: the row's loss (one writer per row); NaN for a row
        // this CTA did not compute (a copy wait gave up)
        if (rank == 0 && tid == 0 && !is_softmax(p)) {
            float l;
            if (failed) {
                l = NAN;
            } else if (has_t) {
                l = row_loss(s_rest, e_t, S, zt, M);
            } else {
                l = NAN;
                atomicAdd(&p.err[kErrBadTarget], 1);
            }
            p.loss_rows[row] = l;
        }
    }

    if (stage && tid == 0) bulk_wait_all();  // the last gradient stores have landed
    // A CTA that gave up still owns copies in flight: it waits for them
    // (each for up to the full limit) before its shared memory is released.
    // A copy that has not landed after that never will; the CTA then leaves
    // rather than hang.
    if (tid == 0 && failed) {
        for (long long j = consumed; j < issued; ++j) {
            if (skips_copy(p, cid + j * ncl, cid + j * ncl + 1)) continue;  // never issued
            if (!mbar_wait(&full[j % nslots], (uint32_t)((j / nslots) & 1))) break;
        }
    }
    if (K > 1) cluster_sync();  // peers may still read this CTA's partials
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, int K, int NT, int VPT, typename P>
cudaError_t launch_kp(const P &p, int ctas, int nslots, int slot_bytes, long long se,
                      int smem, int staged, cudaStream_t s) {
    auto kern = row_split_kernel<T, K, NT, VPT, P>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (K > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = K;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, p, nslots, slot_bytes, se, staged);
}

// The plain call runs the Params build, any other the ParamsEx build.
template <typename T, int K, int NT, int VPT>
cudaError_t launch_k(const ParamsEx &p, int ctas, int nslots, int slot_bytes, long long se,
                     int smem, int staged, cudaStream_t s) {
    if (is_plain(p))
        return launch_kp<T, K, NT, VPT, Params>(static_cast<const Params &>(p), ctas, nslots,
                                                slot_bytes, se, smem, staged, s);
    return launch_kp<T, K, NT, VPT, ParamsEx>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
}

template <typename T, int K, int NT, int VPT>
cudaError_t max_clusters_k(int smem, int *clusters) {
    auto kern = row_split_kernel<T, K, NT, VPT, Params>;
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

// At K = 1 the CTA may be narrower than kSplitThreads (nt = 128: rows of
// 128 x V vectors, several CTAs per SM); clusters keep kSplitThreads.
template <typename T, int V>
cudaError_t launch_v(const ParamsEx &p, int K, int nt, int ctas, int nslots, int slot_bytes,
                     long long se, int smem, int staged, cudaStream_t s) {
    constexpr int NT = kSplitThreads;
    if (K == 1 && nt == 128)
        return launch_k<T, 1, 128, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
    if (nt != NT) return cudaErrorInvalidValue;
    switch (K) {
        case 1: return launch_k<T, 1, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        case 2: return launch_k<T, 2, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        case 3: return launch_k<T, 3, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        case 4: return launch_k<T, 4, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        case 6: return launch_k<T, 6, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        case 8: return launch_k<T, 8, NT, V>(p, ctas, nslots, slot_bytes, se, smem, staged, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int V>
cudaError_t max_clusters_v(int K, int nt, int smem, int *clusters) {
    constexpr int NT = kSplitThreads;
    if (K == 1 && nt == 128) return max_clusters_k<T, 1, 128, V>(smem, clusters);
    if (nt != NT) return cudaErrorInvalidValue;
    switch (K) {
        case 1: return max_clusters_k<T, 1, NT, V>(smem, clusters);
        case 2: return max_clusters_k<T, 2, NT, V>(smem, clusters);
        case 3: return max_clusters_k<T, 3, NT, V>(smem, clusters);
        case 4: return max_clusters_k<T, 4, NT, V>(smem, clusters);
        case 6: return max_clusters_k<T, 6, NT, V>(smem, clusters);
        case 8: return max_clusters_k<T, 8, NT, V>(smem, clusters);
        default: return cudaErrorInvalidValue;
    }
}

// f16 rows are built for slices of 8 vectors per thread only (the planner
// keeps 16-bit rows there, as for bf16).
template <typename T>
cudaError_t launch_t(const ParamsEx &p, int K, int nt, int vecs, int ctas, int nslots,
                     int slot_bytes, long long se, int smem, int staged, cudaStream_t s) {
    if constexpr (std::is_same<T, __half>::value) {
        if (vecs != 8) return cudaErrorInvalidValue;
        return launch_v<T, 8>(p, K, nt, ctas, nslots, slot_bytes, se, smem, staged, s);
    } else {
        if (vecs == 16)
            return launch_v<T, 16>(p, K, nt, ctas, nslots, slot_bytes, se, smem, staged, s);
        if (vecs == 12)
            return launch_v<T, 12>(p, K, nt, ctas, nslots, slot_bytes, se, smem, staged, s);
        if (vecs == 8)
            return launch_v<T, 8>(p, K, nt, ctas, nslots, slot_bytes, se, smem, staged, s);
        return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t max_clusters_t(int K, int nt, int vecs, int smem, int *clusters) {
    if constexpr (std::is_same<T, __half>::value) {
        if (vecs != 8) return cudaErrorInvalidValue;
        return max_clusters_v<T, 8>(K, nt, smem, clusters);
    } else {
        if (vecs == 16) return max_clusters_v<T, 16>(K, nt, smem, clusters);
        if (vecs == 12) return max_clusters_v<T, 12>(K, nt, smem, clusters);
        if (vecs == 8) return max_clusters_v<T, 8>(K, nt, smem, clusters);
        return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_split(const ParamsEx &p, int dtype, int K, int nt, int vecs, int ctas,
                         int nslots, int slot_bytes, long long slice_elems, int smem, int staged,
                         cudaStream_t s) {
    if (dtype == 0)
        return launch_t<float>(p, K, nt, vecs, ctas, nslots, slot_bytes, slice_elems, smem,
                               staged, s);
    if (dtype == 2)
        return launch_t<__half>(p, K, nt, vecs, ctas, nslots, slot_bytes, slice_elems, smem,
                                staged, s);
    return launch_t<__nv_bfloat16>(p, K, nt, vecs, ctas, nslots, slot_bytes, slice_elems, smem,
                                   staged, s);
}

cudaError_t split_max_clusters(int dtype, int K, int nt, int vecs, int smem, int *clusters) {
    if (dtype == 0) return max_clusters_t<float>(K, nt, vecs, smem, clusters);
    if (dtype == 2) return max_clusters_t<__half>(K, nt, vecs, smem, clusters);
    return max_clusters_t<__nv_bfloat16>(K, nt, vecs, smem, clusters);
}

}  // namespace ce
