// Warp-per-row kernel for rows of at most 8 KB (classifier heads), and, swept
// in shared memory instead of held in registers, rows of up to 48 KB.
//
// Each warp owns a private ring of `slots` shared-memory tiles; a tile is
// `rows_per_tile` consecutive rows of the logits, staged by one TMA bulk copy.
// Warps act as their own producers, so no CTA-wide barrier is needed until
// the fused batch-loss tail.  A warp reads its staged row from shared memory
// once, into registers (at most MAXV 16-byte vectors per lane; vectors past
// the row read as -inf), and computes Steps 1-4 of Pass 1 of rumus 0.1.1's
// cross_entropy.wgsl (max, sum of exponentials, row loss, gradient) from
// there with warp-shuffle reductions and packed fp32 pair arithmetic.  fp32
// rows keep their exponentials in registers, so every element is
// exponentiated once.  The last CTA to finish performs Pass 2 (the
// fixed-order batch-loss sum).
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {

// MAXV > 0: the row in registers (at most MAXV vectors per lane).  MAXV = 0:
// the row swept in its slot, kWarpChunkVecs vectors per lane at a time (rows
// longer than a warp's registers hold; NWK warps, one CTA per SM).
template <typename T, int MAXV, int MINB, typename P, int NWK = warp_kernel_warps(MINB)>
__global__ void __launch_bounds__(NWK * 32, MINB)
    rows_warp_kernel(P p, int slots, int rows_per_tile, int slot_bytes) {
    using E = Elem<T>;
    constexpr int NW = NWK;
    constexpr int ES = E::kBytes;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr bool kKeepExp = sizeof(T) == 4;  // fp32: exponentials replace the logits in place

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[NW * kMaxWarpSlots];
    __shared__ float2 tail_scratch[kTailWarps];
    __shared__ unsigned int warps_done;  // warps whose last row loss is stored
    __shared__ int tail_flag;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long B = p.B;
    const int C = (int)p.C;  // rows of at most kWarpChunkRowMax bytes on this path
    // tiles and warps in 32 bits (B < 2^31, rows_per_tile <= 2048)
    const unsigned R = (unsigned)rows_per_tile;
    const unsigned ntiles = ((unsigned)B + R - 1u) / R;
    const unsigned gw = blockIdx.x * NW + warp;
    const unsigned TW = gridDim.x * NW;
    const unsigned ntl = ntiles > gw ? (ntiles - gw + TW - 1u) / TW : 0u;
    // The batch loss (mean, sum): each warp, once its last row's loss is
    // stored and before that row's gradient, counts itself done; the CTA's
    // last warp takes the grid's ticket, so the ticket's release covers the
    // row losses and not the gradient stores, and the last CTA's sum overlaps
    // the other CTAs' gradient stores.
    const bool needs_tail = reduction_of(p) != kReduceNone && !is_softmax(p);
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    unsigned char *my_slots = smem + (size_t)warp * slots * slot_bytes;
    uint64_t *my_full = full + warp * kMaxWarpSlots;
    const bool vec_store = p.grad_vec_ok != 0;
    const bool write_grad = writes_grad(p);  // false: loss only
    const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);

    auto span = [&](unsigned tile, long long &r0, long long &r1, uint64_t &gs, uint64_t &ge,
                    uint64_t &g0, uint64_t &lo, uint64_t &hi) {
        r0 = (long long)tile * R;
        r1 = min(r0 + (long long)R, B);
        gs = lbase + (uint64_t)(r0 * C) * ES;
        ge = lbase + (uint64_t)(r1 * C) * ES;
        g0 = gs & ~15ull;
        lo = g0 > p.lo_clip ? g0 : p.lo_clip;
        const uint64_t ghi = (ge + 15) & ~15ull;
        hi = ghi < p.hi_clip ? ghi : p.hi_clip;
    };
    auto issue = [&](unsigned i, int s) {  // tile i of this warp into slot s
        long long r0, r1;
        uint64_t gs, ge, g0, lo, hi;
        span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);
        if (skips_copy(p, r0, r1)) return;  // test hook: this tile's wait must give up
        unsigned char *slot = my_slots + (size_t)s * slot_bytes;
        if (hi > lo) {
            mbar_arrive_expect_tx(&my_full[s], (uint32_t)(hi - lo));
            bulk_g2s(slot + (lo - g0), reinterpret_cast<const void *>(lo), (uint32_t)(hi - lo),
                     &my_full[s]);
        } else {
            mbar_arrive(&my_full[s]);
        }
    };

    // The warp's count toward the batch loss (once per warp, by lane 0; the
    // row losses it covers were stored by lane 0).
    auto warp_done = [&]() {
        if (!needs_tail) return;
        __syncwarp();
        if (lane == 0) {
            unsigned int c;
            asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                         : "=r"(c)
                         : "r"(smem_addr(&warps_done))
                         : "memory");
            if (c == NW - 1u) {
                unsigned int prev;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                             : "=r"(prev)
                             : "l"(p.ticket)
                             : "memory");
                tail_flag = prev == gridDim.x - 1u;
            }
        }
    };

    if (lane == 0) {
        for (int s = 0; s < slots; ++s) mbar_init(&my_full[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        warps_done = 0u;
        tail_flag = 0;
    }
    pdl_trigger();
    pdl_wait();  // nothing above touched global memory
    const float gsc = scalar_grad_scale(p);
    __syncthreads();
    unsigned issued = 0;
    int s_iss = 0;  // slot of the next copy
    if (lane == 0) {
        for (; issued < ntl && issued < (unsigned)slots; ++issued) issue(issued, (int)issued);
        s_iss = (int)issued == slots ? 0 : (int)issued;
    }
    if (ntl == 0) warp_done();

    unsigned failed_at = ntl;  // the first tile whose copy wait gave up (ntl: none)
    int s = 0;                 // slot and phase parity of the next tile
    uint32_t parity = 0;

    for (unsigned i = 0; i < ntl; ++i) {
        unsigned char *slot = my_slots + (size_t)s * slot_bytes;
        long long r0, r1;
        uint64_t gs, ge, g0, lo, hi;
        span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);
        // the tile's first targets, in flight while the copy lands
        int tchunk = r0 + lane < r1 ? target_at(p, r0 + lane) : 0;

        // the warp goes on only if every lane saw the copy land
        if (!__all_sync(0xffffffffu, mbar_wait(&my_full[s], parity, copy_wait_limit(p)))) {
            failed_at = i;
            if (lane == 0) atomicAdd(&p.err[kErrTimeout], 1);
            break;
        }
        if (++s == slots) {
            s = 0;
            parity ^= 1u;
        }

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
            const int q = (int)(r - r0);
            if (q > 0 && (q & 31) == 0) tchunk = r + lane < r1 ? target_at(p, r + lane) : 0;
            const int t = __shfl_sync(0xffffffffu, tchunk, q & 31);
            const bool has_t = t >= 0 && t < C;

            // Row layout in shared memory: nh head elements up to the first
            // 16-byte boundary, nvec whole vectors, nt tail elements.
            const unsigned char *row = slot + (gs - g0) + (size_t)q * C * ES;
            const uint32_t ph = smem_addr(row) & 15u;
            const int nh = ph ? min((int)((16u - ph) / ES), C) : 0;
            const int nvec = (C - nh) / W;
            const int nt = C - nh - nvec * W;
            const unsigned char *vrow = row + nh * ES;
            const int tv = has_t ? t - nh : -0x40000000;  // target relative to vector 0
            const int v_t = has_t && tv >= 0 && tv < nvec * W ? tv / W : -1;  // its vector

            if constexpr (MAXV > 0) {
                const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                              E::kNegInfWord);
                uint4 x[MAXV];
#pragma unroll
                for (int k = 0; k < MAXV; ++k) {
                    const int v = lane + 32 * k;
                    x[k] = kNeg;
                    if (v < nvec) x[k] = lds128(vrow + 16 * v);
                }
                // head and tail elements exist only for rows that do not start and
                // end on a 16-byte boundary (the same in every lane)
                const bool ragged = (nh | nt) != 0;
                float hz = -INFINITY, tz = -INFINITY;
                if (ragged) {
                    if (lane < nh) hz = E::load(row + lane * ES);
                    if (lane < nt) tz = E::load(vrow + (nvec * W + lane) * ES);
                }
                const float zt = has_t ? E::load(row + t * ES) : 0.f;
                // lane 0 also takes the target's vector
                const uint4 xt = lane == 0 && v_t >= 0 ? lds128(vrow + 16 * v_t) : kNeg;

                // Step 1: max
                float m = fmaxf(hz, tz);
                typename E::MaxAcc macc = E::max_init();
#pragma unroll
                for (int k = 0; k < MAXV; ++k) E::max_step(macc, x[k]);
                m = fmaxf(m, E::max_value(macc));
                m = warp_max(m);
                const float M = m * kLog2e;
                const unsigned long long nM2 = f2_pack(-M, -M);

                // Step 2: sum of exponentials without the target's term.  The
                // target's vector is left out whole; lane 0 adds its other elements.
                unsigned long long acc = 0ull;
#pragma unroll
                for (int k = 0; k < MAXV; ++k) {
                    const int v = lane + 32 * k;
                    unsigned long long e2[W2];
                    E::unpack2(x[k], e2);
#pragma unroll
                    for (int j = 0; j < W2; ++j) {
                        float a, b;
                        f2_unpack(f2_fma(e2[j], kL2E2, nM2), a, b);
                        e2[j] = f2_pack(ex2(a), ex2(b));
                    }
                    if (kKeepExp) x[k] = E::pack2(e2);
                    unsigned long long vs = W2 == 4 ? f2_add(f2_add(e2[0], e2[1]),
                                                             f2_add(e2[W2 - 2], e2[W2 - 1]))
                                                    : f2_add(e2[0], e2[W2 - 1]);
                    if (v != v_t) acc = f2_add(acc, vs);
                }
                float sa, sb;
                f2_unpack(acc, sa, sb);
                if (lane == 0 && v_t >= 0) {
                    float z[W];
                    E::unpack(xt, z);
                    const int d = tv - v_t * W;
#pragma unroll
                    for (int j = 0; j < W; ++j)
                        if (j != d) sa += ex2(fmaf(z[j], kLog2e, -M));
                }
                float eh = 0.f, et = 0.f;
                if (ragged) {
                    if (lane < nh) eh = ex2(fmaf(hz, kLog2e, -M));
                    if (lane < nt) et = ex2(fmaf(tz, kLog2e, -M));
                    if (lane != t) sa += eh;
                    if (nh + nvec * W + lane != t) sb += et;
                }
                const float s_rest = warp_sum(sa + sb);
                const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
                const float S = s_rest + e_t;

                // Step 4: gradient; (p_t - 1) / B = -S_rest / (S B), times the
                // upstream gradient (1/B becomes 1 for the sum and per-row losses)
                const float scale = fast_rcp(S) * row_grad_factor(p, gsc, r);
                const unsigned long long sc2 = f2_pack(scale, scale);
                const float g_t = -s_rest * scale;

                // Step 3: loss of the row, log(S / e_t) -- before the gradient, so
                // that the warp's last row can count it done first
                if (lane == 0 && !is_softmax(p)) {
                    float l;
                    if (has_t) {
                        l = row_loss(s_rest, e_t, S, zt, M);
                    } else {
                        l = NAN;
                        atomicAdd(&p.err[kErrBadTarget], 1);
                    }
                    p.loss_rows[r] = l;
                }
                if (i + 1 == ntl && r + 1 == r1) warp_done();

                if (write_grad) {
                    unsigned char *grow = p.grad + (size_t)r * C * ES;
                    unsigned char *gvec = grow + nh * ES;
                    auto grad2 = [&](const uint4 &xv, unsigned long long (&g2)[W2]) {
                        E::unpack2(xv, g2);
#pragma unroll
                        for (int j = 0; j < W2; ++j) {
                            if (!kKeepExp) {
                                float a, b;
                                f2_unpack(f2_fma(g2[j], kL2E2, nM2), a, b);
                                g2[j] = f2_pack(ex2(a), ex2(b));
                            }
                            g2[j] = f2_mul(g2[j], sc2);
                        }
                    };
                    if (vec_store) {
#pragma unroll
                        for (int k = 0; k < MAXV; ++k) {
                            const int v = lane + 32 * k;
                            if (v < nvec) {
                                unsigned long long g2[W2];
                                grad2(x[k], g2);
                                *reinterpret_cast<uint4 *>(gvec + 16 * v) = E::pack2(g2);
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < MAXV; ++k) {
                            const int v = lane + 32 * k;
                            if (v < nvec) {
                                unsigned long long g2[W2];
                                grad2(x[k], g2);
#pragma unroll
                                for (int j = 0; j < W2; ++j) {
                                    float a, b;
                                    f2_unpack(g2[j], a, b);
                                    E::store(gvec + (v * W + 2 * j) * ES, a);
                                    E::store(gvec + (v * W + 2 * j + 1) * ES, b);
                                }
                            }
                        }
                    }
                    // the owner of the target's vector overwrites the target,
                    // after its vector's store
                    if (v_t >= 0 && lane == (v_t & 31)) E::store(grow + (size_t)t * ES, g_t);
                    // test hook: the whole vectors' fp32 values, before their
                    // rounding (recomputed so that the loop above carries none of it)
                    if (grad_f32_of(p)) {
#pragma unroll
                        for (int k = 0; k < MAXV; ++k) {
                            const int v = lane + 32 * k;
                            if (v < nvec) {
                                unsigned long long g2[W2];
                                E::unpack2(x[k], g2);
#pragma unroll
                                for (int j = 0; j < W2; ++j) {
                                    if (!kKeepExp) {
                                        float a, b;
                                        f2_unpack(f2_fma(g2[j], kL2E2, nM2), a, b);
                                        g2[j] = f2_pack(ex2(a), ex2(b));
                                    }
                                    float a, b;
                                    f2_unpack(f2_mul(g2[j], sc2), a, b);
                                    grad_f32_store<ES>(p, gvec + (v * W + 2 * j) * ES, a);
                                    grad_f32_store<ES>(p, gvec + (v * W + 2 * j + 1) * ES, b);
                                }
                                if (v == v_t) grad_f32_store<ES>(p, grow + (size_t)t * ES, g_t);
                            }
                        }
                    }
                    if (ragged) {
                        if (lane < nh) {
                            const float gh = lane == t ? g_t : eh * scale;
                            E::store(grow + lane * ES, gh);
                            grad_f32_store<ES>(p, grow + lane * ES, gh);
                        }
                        if (lane < nt) {
                            const int c = nh + nvec * W + lane;
                            const float gc = c == t ? g_t : et * scale;
                            E::store(grow + c * ES, gc);
                            grad_f32_store<ES>(p, grow + c * ES, gc);
                        }
                    }
                }
            } else {
                // The row stays in its slot and is swept there three times, CH
                // vectors per lane at a time: the max, the sum of exponentials
                // without the target's term, the gradient -- the register
                // build's per-element arithmetic.
                constexpr int CH = kWarpChunkVecs;
                const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                              E::kNegInfWord);
                auto load_chunk = [&](int base, uint4 (&x)[CH]) {
#pragma unroll
                    for (int k = 0; k < CH; ++k) {
                        const int v = base + lane + 32 * k;
                        x[k] = v < nvec ? lds128(vrow + 16 * v) : kNeg;
                    }
                };
                const bool ragged = (nh | nt) != 0;
                float hz = -INFINITY, tz = -INFINITY;
                if (ragged) {
                    if (lane < nh) hz = E::load(row + lane * ES);
                    if (lane < nt) tz = E::load(vrow + (nvec * W + lane) * ES);
                }
                const float zt = has_t ? E::load(row + t * ES) : 0.f;

                // Step 1: max
                float m = fmaxf(hz, tz);
                {
                    typename E::MaxAcc macc = E::max_init();
                    for (int base = 0; base < nvec; base += 32 * CH) {
                        uint4 x[CH];
                        load_chunk(base, x);
#pragma unroll
                        for (int k = 0; k < CH; ++k) E::max_step(macc, x[k]);
                    }
                    m = fmaxf(m, E::max_value(macc));
                }
                m = warp_max(m);
                const float M = m * kLog2e;
                const unsigned long long nM2 = f2_pack(-M, -M);

                // Step 2: sum of exponentials without the target's term (the
                // lane holding the target's vector adds its other elements)
                unsigned long long acc = 0ull;
                float sa = 0.f;
                for (int base = 0; base < nvec; base += 32 * CH) {
                    uint4 x[CH];
                    load_chunk(base, x);
#pragma unroll
                    for (int k = 0; k < CH; ++k) {
                        const int v = base + lane + 32 * k;
                        if (v == v_t) {
                            float z[W];
                            E::unpack(x[k], z);
                            const int d = tv - v_t * W;
#pragma unroll
                            for (int j = 0; j < W; ++j)
                                if (j != d) sa += ex2(fmaf(z[j], kLog2e, -M));
                            continue;
                        }
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
                }
                float pa, pb;
                f2_unpack(acc, pa, pb);
                float eh = 0.f, et = 0.f;
                if (ragged) {
                    if (lane < nh) eh = ex2(fmaf(hz, kLog2e, -M));
                    if (lane < nt) et = ex2(fmaf(tz, kLog2e, -M));
                    if (lane != t) sa += eh;
                    if (nh + nvec * W + lane != t) pb += et;
                }
                const float s_rest = warp_sum(sa + pa + pb);
                const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
                const float S = s_rest + e_t;
                const float scale = fast_rcp(S) * row_grad_factor(p, gsc, r);
                const unsigned long long sc2 = f2_pack(scale, scale);
                const float g_t = -s_rest * scale;

                // Step 3: loss of the row, before the gradient
                if (lane == 0 && !is_softmax(p)) {
                    float l;
                    if (has_t) {
                        l = row_loss(s_rest, e_t, S, zt, M);
                    } else {
                        l = NAN;
                        atomicAdd(&p.err[kErrBadTarget], 1);
                    }
                    p.loss_rows[r] = l;
                }
                if (i + 1 == ntl && r + 1 == r1) warp_done();

                // Step 4: gradient, a third sweep of the slot; the owner of the
                // target's vector overwrites the target after its vector
                if (write_grad) {
                    unsigned char *grow = p.grad + (size_t)r * C * ES;
                    unsigned char *gvec = grow + nh * ES;
                    for (int base = 0; base < nvec; base += 32 * CH) {
                        uint4 x[CH];
                        load_chunk(base, x);
#pragma unroll
                        for (int k = 0; k < CH; ++k) {
                            const int v = base + lane + 32 * k;
                            if (v < nvec) {
                                unsigned long long g2[W2];
                                E::unpack2(x[k], g2);
#pragma unroll
                                for (int j = 0; j < W2; ++j) {
                                    float a, b;
                                    f2_unpack(f2_fma(g2[j], kL2E2, nM2), a, b);
                                    g2[j] = f2_mul(f2_pack(ex2(a), ex2(b)), sc2);
                                }
                                if (vec_store) {
                                    *reinterpret_cast<uint4 *>(gvec + 16 * v) = E::pack2(g2);
                                } else {
#pragma unroll
                                    for (int j = 0; j < W2; ++j) {
                                        float a, b;
                                        f2_unpack(g2[j], a, b);
                                        E::store(gvec + (v * W + 2 * j) * ES, a);
                                        E::store(gvec + (v * W + 2 * j + 1) * ES, b);
                                    }
                                }
                                if (grad_f32_of(p)) {  // test hook: the values before rounding
#pragma unroll
                                    for (int j = 0; j < W2; ++j) {
                                        float a, b;
                                        f2_unpack(g2[j], a, b);
                                        grad_f32_store<ES>(p, gvec + (v * W + 2 * j) * ES, a);
                                        grad_f32_store<ES>(p, gvec + (v * W + 2 * j + 1) * ES, b);
                                    }
                                }
                                if (v == v_t) {
                                    E::store(grow + (size_t)t * ES, g_t);
                                    grad_f32_store<ES>(p, grow + (size_t)t * ES, g_t);
                                }
                            }
                        }
                    }
                    if (ragged) {
                        if (lane < nh) {
                            const float gh = lane == t ? g_t : eh * scale;
                            E::store(grow + lane * ES, gh);
                            grad_f32_store<ES>(p, grow + lane * ES, gh);
                        }
                        if (lane < nt) {
                            const int c = nh + nvec * W + lane;
                            const float gc = c == t ? g_t : et * scale;
                            E::store(grow + c * ES, gc);
                            grad_f32_store<ES>(p, grow + c * ES, gc);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && issued < ntl) {
            fence_proxy_async();
            issue(issued, s_iss);
            ++issued;
            if (++s_iss == slots) s_iss = 0;
        }
    }

    if (failed_at < ntl) {
        // The tiles from the one whose wait gave up on were not computed:
        // their rows' losses are NaN, so the batch loss shows the failure
        // (their gradient is not written).
        for (unsigned i = failed_at; i < ntl; ++i) {
            long long r0, r1;
            uint64_t gs, ge, g0, lo, hi;
            span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);
            if (!is_softmax(p))
                for (long long r = r0 + lane; r < r1; r += 32) p.loss_rows[r] = NAN;
        }
        warp_done();  // (lane 0 stored NaN rows too; the others before the warp's sync)
        // The warp still owns copies in flight: it waits for them (each for
        // up to the full limit) before the CTA's shared memory is released.
        // A copy that has not landed after that never will; the warp then
        // leaves rather than hang.
        if (lane == 0) {
            for (unsigned i = failed_at; i < issued; ++i) {
                long long r0, r1;
                uint64_t gs, ge, g0, lo, hi;
                span(gw + i * TW, r0, r1, gs, ge, g0, lo, hi);
                if (skips_copy(p, r0, r1)) continue;  // never issued
                if (!mbar_wait(&my_full[i % slots], (i / slots) & 1u)) break;
            }
        }
    }
    // the batch loss, in the CTA that took the grid's last ticket
    if (needs_tail) {
        __syncthreads();
        if (tail_flag) batch_tail(p, tail_scratch);
    }
}

template <typename T, int MAXV, int MINB, typename P, int NWK = warp_kernel_warps(MINB)>
cudaError_t launch_p(const P &p, int ctas, int slots, int rows_per_tile, int slot_bytes,
                     int smem, cudaStream_t s) {
    auto kern = rows_warp_kernel<T, MAXV, MINB, P, NWK>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(NWK * 32, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, slots, rows_per_tile, slot_bytes);
}

// The plain call runs the Params build, any other the ParamsEx build.
template <typename T, int MAXV, int MINB>
cudaError_t launch_v(const ParamsEx &p, int ctas, int slots, int rows_per_tile, int slot_bytes,
                     int smem, cudaStream_t s) {
    if (is_plain(p))
        return launch_p<T, MAXV, MINB, Params>(static_cast<const Params &>(p), ctas, slots,
                                               rows_per_tile, slot_bytes, smem, s);
    return launch_p<T, MAXV, MINB, ParamsEx>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
}

template <typename T, int MAXV, int MINB>
cudaError_t occ_v(int smem, int *ctas) {
    auto kern = rows_warp_kernel<T, MAXV, MINB, Params>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, warp_kernel_warps(MINB) * 32,
                                                         smem);
}

// Vectors per lane: a row of C elements holds at most C*ES/16 whole vectors.
int vectors_per_lane(long long C, int es) {
    const long long nvec = C * es / 16;
    const long long per_lane = (nvec + 31) / 32;
    return per_lane <= 2 ? 2 : per_lane <= 4 ? 4 : per_lane <= 8 ? 8 : 16;
}

template <typename T, int MINB>
cudaError_t launch_m(const ParamsEx &p, int ctas, int slots, int rows_per_tile, int slot_bytes,
                     int smem, cudaStream_t s) {
    switch (vectors_per_lane(p.C, sizeof(T))) {
        case 2: return launch_v<T, 2, MINB>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
        case 4: return launch_v<T, 4, MINB>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
        case 8: return launch_v<T, 8, MINB>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
        default: return launch_v<T, 16, MINB>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    }
}

template <typename T, int MINB>
cudaError_t occ_m(long long C, int smem, int *ctas) {
    switch (vectors_per_lane(C, sizeof(T))) {
        case 2: return occ_v<T, 2, MINB>(smem, ctas);
        case 4: return occ_v<T, 4, MINB>(smem, ctas);
        case 8: return occ_v<T, 8, MINB>(smem, ctas);
        default: return occ_v<T, 16, MINB>(smem, ctas);
    }
}

template <typename T>
cudaError_t launch_t(const ParamsEx &p, int per_sm, int ctas, int slots, int rows_per_tile,
                     int slot_bytes, int smem, cudaStream_t s) {
    if (per_sm >= 3) return launch_m<T, 3>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    if (per_sm == 2) return launch_m<T, 2>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    return launch_m<T, 1>(p, ctas, slots, rows_per_tile, slot_bytes, smem, s);
}

// The swept build (rows longer than the registers hold): NWK warps, one tile
// of one row per slot.
template <typename T, int NWK>
cudaError_t launch_c(const ParamsEx &p, int ctas, int slots, int slot_bytes, int smem,
                     cudaStream_t s) {
    if (is_plain(p))
        return launch_p<T, 0, 1, Params, NWK>(static_cast<const Params &>(p), ctas, slots, 1,
                                              slot_bytes, smem, s);
    return launch_p<T, 0, 1, ParamsEx, NWK>(p, ctas, slots, 1, slot_bytes, smem, s);
}
template <typename T, int NWK>
cudaError_t occ_c(int smem, int *ctas) {
    auto kern = rows_warp_kernel<T, 0, 1, Params, NWK>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, NWK * 32, smem);
}
template <typename T>
cudaError_t launch_ct(const ParamsEx &p, int nw, int ctas, int slots, int slot_bytes, int smem,
                      cudaStream_t s) {
    if (nw == 16) return launch_c<T, 16>(p, ctas, slots, slot_bytes, smem, s);
    if (nw == 8) return launch_c<T, 8>(p, ctas, slots, slot_bytes, smem, s);
    if (nw == 4) return launch_c<T, 4>(p, ctas, slots, slot_bytes, smem, s);
    return cudaErrorInvalidValue;
}
template <typename T>
cudaError_t occ_ct(int nw, int smem, int *ctas) {
    if (nw == 16) return occ_c<T, 16>(smem, ctas);
    if (nw == 8) return occ_c<T, 8>(smem, ctas);
    if (nw == 4) return occ_c<T, 4>(smem, ctas);
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t occ_t(int per_sm, long long C, int smem, int *ctas) {
    if (per_sm >= 3) return occ_m<T, 3>(C, smem, ctas);
    if (per_sm == 2) return occ_m<T, 2>(C, smem, ctas);
    return occ_m<T, 1>(C, smem, ctas);
}

}  // namespace

cudaError_t launch_rows_warp(const ParamsEx &p, int dtype, int per_sm, int ctas, int slots,
                             int rows_per_tile, int slot_bytes, int smem, cudaStream_t s) {
    if (dtype == 0)
        return launch_t<float>(p, per_sm, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    if (dtype == 2)
        return launch_t<__half>(p, per_sm, ctas, slots, rows_per_tile, slot_bytes, smem, s);
    return launch_t<__nv_bfloat16>(p, per_sm, ctas, slots, rows_per_tile, slot_bytes, smem, s);
}

cudaError_t rows_warp_max_ctas_per_sm(int dtype, int per_sm, long long C, int smem, int *ctas) {
    if (dtype == 0) return occ_t<float>(per_sm, C, smem, ctas);
    if (dtype == 2) return occ_t<__half>(per_sm, C, smem, ctas);
    return occ_t<__nv_bfloat16>(per_sm, C, smem, ctas);
}

cudaError_t launch_rows_warp_swept(const ParamsEx &p, int dtype, int nw, int ctas, int slots,
                                   int slot_bytes, int smem, cudaStream_t s) {
    if (dtype == 0) return launch_ct<float>(p, nw, ctas, slots, slot_bytes, smem, s);
    if (dtype == 2) return launch_ct<__half>(p, nw, ctas, slots, slot_bytes, smem, s);
    return launch_ct<__nv_bfloat16>(p, nw, ctas, slots, slot_bytes, smem, s);
}

cudaError_t rows_warp_swept_max_ctas_per_sm(int dtype, int nw, int smem, int *ctas) {
    if (dtype == 0) return occ_ct<float>(nw, smem, ctas);
    if (dtype == 2) return occ_ct<__half>(nw, smem, ctas);
    return occ_ct<__nv_bfloat16>(nw, smem, ctas);
}

}  // namespace ce
