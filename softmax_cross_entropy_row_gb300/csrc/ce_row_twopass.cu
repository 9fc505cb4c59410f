// Two-pass row kernel: one CTA per row at a time, rows of any length.
//
// A row streams through a ring of small shared-memory chunks twice.  One
// producer lane issues TMA bulk copies in the order the consumers use them
// (row j's chunks for the first pass, the same chunks again for the second
// pass, then row j+1's ...); consumer warps wait for a chunk, read it into
// registers and hand the slot back at once, so the copies of the next chunks
// are always in flight.
//
//   pass 1  every consumer thread keeps a running maximum M_t (log2 domain)
//           and a sum S_t of 2^(z*log2e - M_t) over its elements, rescaled
//           whenever M_t grows (the running-max / rescaled-sum recurrence of
//           the rumus FlashAttention milestone, M17), the target's term left
//           out; warp partials, one barrier among the consumer warps, and
//           every warp combines the partials in the same fixed order:
//           M = max M_w, S_rest = sum S_w 2^(M_w - M)            (Steps 1, 2)
//           l_b = log(S / e_t), S = S_rest + e_t                (Step 3)
//   pass 2  grad = 2^(z*log2e - M) / (S B), the target's element
//           -S_rest / (S B)                                      (Step 4)
//
// which are Pass 1 of rumus 0.1.1's cross_entropy.wgsl with the max and the
// sum taken in one sweep.  The second pass reads the row again, but the row
// was read a few microseconds before and is still in L2, so HBM sees the
// logits once: the first pass's copies ask L2 to keep their lines, the second
// pass's to drop them first.  Nothing is exchanged between CTAs, and the CTA
// needs no more shared memory for a long row than for a short one.  The
// last CTA to finish sums the row losses in the fixed order of the other
// paths (Pass 2).
#include <math.h>

#include "ce_launch.h"

namespace ce {
namespace {


// The 16-byte aligned span that covers row `row`: vector v holds the row's
// elements v*W - head .. v*W - head + W - 1 (those in [0, C) belong to it).
struct RowGeom {
    uint64_t A;   // address of vector 0
    int head;     // elements of vector 0 before the row
    int nv;       // vectors
    int nch;      // chunks
    bool head_partial, tail_partial;
};

template <int ES, int CHV>
__device__ __forceinline__ RowGeom row_geom(uint64_t lbase, long long row, long long C) {
    RowGeom g;
    const uint64_t gs = lbase + (uint64_t)row * (uint64_t)C * ES;
    const uint64_t ge = gs + (uint64_t)C * ES;
    g.A = gs & ~15ull;
    g.head = (int)((gs - g.A) / ES);
    g.nv = (int)((((ge + 15) & ~15ull) - g.A) >> 4);
    g.nch = (g.nv + CHV - 1) / CHV;
    g.head_partial = g.head != 0;
    g.tail_partial = (ge & 15ull) != 0;
    return g;
}

// Vector v of a row whose elements are not all the row's own (the first and
// last vector of an unaligned row): elements outside the row read as -inf;
// elements the copy could not reach (the first or last 16 bytes of an
// unaligned tensor) are loaded from global memory.
template <typename E, typename P>
__device__ __noinline__ uint4 fix_partial(const P &p, uint4 x, const RowGeom &g, int v,
                                          long long C) {
    constexpr int W = E::kVec;
    constexpr int ES = E::kBytes;
    float z[W];
    E::unpack(x, z);
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const long long l = (long long)v * W + i - g.head;
        if (l < 0 || l >= C) {
            z[i] = -INFINITY;
        } else {
            const uint64_t a = g.A + 16ull * v + (uint64_t)i * ES;
            if (a < p.lo_clip || a + ES > p.hi_clip)
                z[i] = E::load_global(reinterpret_cast<const unsigned char *>(a));
        }
    }
    return E::pack(z);
}

constexpr int NCW = kTwoPassConsumerWarps;
constexpr int VPC = kTwoPassVecs;  // 16-byte vectors per consumer thread per chunk
constexpr int NCT = NCW * 32;      // consumer threads
constexpr int NTT = NCT + 32;      // and the producer warp
constexpr int CHV = NCT * VPC;     // vectors per chunk
constexpr int CHB = CHV * 16;      // bytes per chunk
static_assert(CHB == kTwoPassChunkBytes, "chunk size");

template <typename T, typename P>
__global__ void __launch_bounds__(NTT, 1) row_twopass_kernel(P p, int nslots, int hint) {
    using E = Elem<T>;
    constexpr int W = E::kVec;
    constexpr int W2 = W / 2;
    constexpr int ES = E::kBytes;

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kTwoPassMaxSlots];
    __shared__ uint64_t empty[kTwoPassMaxSlots];
    __shared__ float2 red[2][NCW];  // warp partials (M_w, S_w) by row parity
    __shared__ float zt_sh[2];
    __shared__ int cta_failed;
    __shared__ float2 tail_scratch[kTailWarps];
    __shared__ int tail_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const long long C = p.C;
    const long long nrows =
        (long long)blockIdx.x < p.B ? (p.B - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint64_t lbase = reinterpret_cast<uint64_t>(p.logits);
    const int passes = writes_grad(p) ? 2 : 1;  // the loss alone needs one

    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        fence_mbar_init();
        cta_failed = 0;
    }
    pdl_trigger();
    pdl_wait();  // nothing above touched global memory
    const float gsc = scalar_grad_scale(p);
    __syncthreads();

    // producer state (lane 0 of the last warp)
    long long issued = 0;    // chunks issued (or left out by the test hook)
    long long skipped = -1;  // the chunk the test hook left out

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t keep = l2_policy_evict_last();
            const uint64_t drop = l2_policy_evict_first();
            bool stop = false;
            int s = 0;             // slot of the next copy
            uint32_t round = 0;    // how many times the ring has been filled (its parity)
            bool wrapped = false;  // slot s has been used before
            for (long long i = 0; i < nrows && !stop; ++i) {
                const long long row = blockIdx.x + i * gridDim.x;
                const RowGeom g = row_geom<ES, CHV>(lbase, row, C);
                const uint64_t end = g.A + 16ull * (uint64_t)g.nv;
                for (int pass = 0; pass < passes && !stop; ++pass) {
                    for (int k = 0; k < g.nch; ++k) {
                        // use `round` of slot s waits for the consumers' release
                        // of its use round - 1
                        if (wrapped && mbar_wait_or_flag(&empty[s], (round - 1) & 1u, &cta_failed,
                                                         kWaitLimitCycles) <= 0) {
                            stop = true;
                            break;
                        }
                        if (*reinterpret_cast<volatile int *>(&cta_failed)) {
                            stop = true;
                            break;
                        }
                        if (wrapped) fence_proxy_async();  // the slot was read through the generic proxy
                        const int slot_now = s;
                        if (++s == nslots) {
                            s = 0;
                            ++round;
                            wrapped = true;
                        }
                        if (pass == 0 && k == 0 && skips_copy(p, row, row + 1)) {
                            skipped = issued++;  // test hook: never issued
                            continue;
                        }
                        const uint64_t c0 = g.A + (uint64_t)k * CHB;
                        const uint64_t c1 = c0 + CHB < end ? c0 + CHB : end;
                        const uint64_t lo = c0 > p.lo_clip ? c0 : p.lo_clip;
                        const uint64_t hi = c1 < p.hi_clip ? c1 : p.hi_clip;
                        unsigned char *slot = smem + (size_t)slot_now * CHB;
                        uint64_t *bar = &full[slot_now];
                        if (hi > lo) {
                            mbar_arrive_expect_tx(bar, (uint32_t)(hi - lo));
                            if (hint)
                                bulk_g2s_hint(slot + (lo - c0), reinterpret_cast<const void *>(lo),
                                              (uint32_t)(hi - lo), bar, pass ? drop : keep);
                            else
                                bulk_g2s(slot + (lo - c0), reinterpret_cast<const void *>(lo),
                                         (uint32_t)(hi - lo), bar);
                        } else {
                            mbar_arrive(bar);
                        }
                        ++issued;
                    }
                }
            }
        }
    } else {
        // ----------------------------------------------------------- consumers
        // Thread ct reads vectors u*NCT + ct (u < VPC) of every chunk: a warp
        // reads 512 contiguous bytes per vector, without bank conflicts.
        const int ct = tid;
        const unsigned long long kL2E2 = f2_pack(kLog2e, kLog2e);
        const uint4 kNeg = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord,
                                      E::kNegInfWord);
        const bool vec_store = p.grad_vec_ok != 0;
        int cs = 0;           // slot of the next chunk, in the producer's order
        uint32_t cph = 0;     // the phase parity of its copy
        bool failed = false;  // this warp gave up (uniform in the warp)
        int t_next = nrows > 0 ? target_at(p, blockIdx.x) : 0;

        // Wait for the next chunk (slot s); false once this warp has given up.
        auto wait_next = [&](int &s) -> bool {
            s = cs;
            const uint32_t parity = cph;
            if (++cs == nslots) {
                cs = 0;
                cph ^= 1u;
            }
            if (failed) return false;
            const int w = mbar_wait_or_flag(&full[s], parity, &cta_failed, copy_wait_limit(p));
            if (w < 0 && atomicExch(&cta_failed, 1) == 0) atomicAdd(&p.err[kErrTimeout], 1);
            if (!__all_sync(0xffffffffu, w > 0)) {
                failed = true;
                if (lane == 0) atomicExch(&cta_failed, 1);
                return false;
            }
            return true;
        };
        // Read this thread's vectors of chunk k from slot s and hand the slot
        // back.  An edge chunk (the first of an unaligned row, or the last)
        // may end before its last vector or hold a partial vector.
        auto read = [&](int s, const RowGeom &g, int k, bool edge, uint4 (&x)[VPC]) {
            const unsigned char *slot = smem + (size_t)s * CHB;
            if (!edge) {
#pragma unroll
                for (int u = 0; u < VPC; ++u) x[u] = lds128(slot + 16 * (u * NCT + ct));
            } else {
#pragma unroll
                for (int u = 0; u < VPC; ++u) {
                    const int lv = u * NCT + ct;
                    x[u] = k * CHV + lv < g.nv ? lds128(slot + 16 * lv) : kNeg;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (edge) {
#pragma unroll
                for (int u = 0; u < VPC; ++u) {
                    const int v = k * CHV + u * NCT + ct;
                    if ((v == 0 && g.head_partial) || (v == g.nv - 1 && g.tail_partial))
                        x[u] = fix_partial<E>(p, x[u], g, v, C);
                }
            }
        };

        for (long long i = 0; i < nrows; ++i) {
            const long long row = blockIdx.x + i * gridDim.x;
            const int par = (int)(i & 1);
            const int t = t_next;
            if (i + 1 < nrows) t_next = target_at(p, row + gridDim.x);
            const RowGeom g = row_geom<ES, CHV>(lbase, row, C);
            const bool has_t = t >= 0 && t < C;
            const int vt = has_t ? (int)(((long long)g.head + t) / W) : -1;  // the target's vector
            const int dt = has_t ? (int)(((long long)g.head + t) % W) : 0;   // its element there
            const int kt = has_t ? vt / CHV : -1;                            // its chunk
            const int lt = vt - kt * CHV;                                    // its place there

            // ---- pass 1: running max and rescaled sum, the target left out
            float Mt = -INFINITY;
            unsigned long long acc = 0ull;  // (0.f, 0.f)
            for (int k = 0; k < g.nch; ++k) {
                int s;
                if (!wait_next(s)) continue;
                const bool edge = (k == 0 && g.head_partial) || k == g.nch - 1;
                uint4 x[VPC];
                read(s, g, k, edge, x);
                typename E::MaxAcc macc = E::max_init();
#pragma unroll
                for (int u = 0; u < VPC; ++u) E::max_step(macc, x[u]);
                const float CM = E::max_value(macc) * kLog2e;
                if (CM > Mt) {
                    const float r = ex2(Mt - CM);  // 0 while Mt = -inf (acc is 0 then)
                    acc = f2_mul(acc, f2_pack(r, r));
                    Mt = CM;
                }
                if (k == kt) {
                    // the target's owner records z_t and takes the target out
                    // of the sum (it counted in the maximum)
#pragma unroll
                    for (int u = 0; u < VPC; ++u) {
                        if (u * NCT + ct == lt) {
                            zt_sh[par] = element_of<E>(x[u], dt);
                            x[u] = with_neg_inf<E>(x[u], dt);
                        }
                    }
                }
                if (Mt == -INFINITY) continue;  // nothing but -inf so far
                const unsigned long long nM2 = f2_pack(-Mt, -Mt);
#pragma unroll
                for (int u = 0; u < VPC; ++u) {
                    unsigned long long e2[W2];
                    E::unpack2(x[u], e2);
#pragma unroll
                    for (int j = 0; j < W2; ++j) {
                        float a, b;
                        f2_unpack(f2_fma(e2[j], kL2E2, nM2), a, b);
                        e2[j] = f2_pack(ex2(a), ex2(b));
                    }
                    const unsigned long long vs =
                        W2 == 4 ? f2_add(f2_add(e2[0], e2[1]), f2_add(e2[2], e2[3]))
                                : f2_add(e2[0], e2[W2 - 1]);
                    acc = f2_add(acc, vs);
                }
            }

            // ---- combine: warp partials, one barrier, every warp the same sum
            float sa, sb;
            f2_unpack(acc, sa, sb);
            const float st = sa + sb;
            const float Mw = warp_max(Mt);
            float sw = st != 0.f ? st * ex2(Mt - Mw) : 0.f;
            sw = warp_sum(sw);
            if (lane == 0) red[par][warp] = make_float2(Mw, sw);
            named_sync(1, NCT);
            const float2 r = lane < NCW ? red[par][lane] : make_float2(-INFINITY, 0.f);
            const float M = warp_max(r.x);
            const float s_rest = warp_sum(r.y != 0.f ? r.y * ex2(r.x - M) : 0.f);
            const float zt = has_t ? zt_sh[par] : 0.f;
            const float e_t = has_t ? ex2(fmaf(zt, kLog2e, -M)) : 0.f;
            const float S = s_rest + e_t;
            const float scale = fast_rcp(S) * row_grad_factor(p, gsc, row);
            const float g_t = -s_rest * scale;

            // ---- Step 3: the row's loss (rows of a CTA that gave up are
            // rewritten as NaN at the end)
            if (ct == 0 && !is_softmax(p)) {
                float l;
                if (has_t) {
                    l = row_loss(s_rest, e_t, S, zt, M);
                } else {
                    l = NAN;
                    if (!failed) atomicAdd(&p.err[kErrBadTarget], 1);
                }
                p.loss_rows[row] = l;
            }
            if (passes == 1) continue;

            // ---- pass 2: the gradient
            const unsigned long long nM2 = f2_pack(-M, -M);
            const unsigned long long esc2 = f2_pack(scale, scale);
            unsigned char *gA = p.grad + (long long)(g.A - lbase);  // grad byte of vector 0
            for (int k = 0; k < g.nch; ++k) {
                int s;
                if (!wait_next(s)) continue;
                const bool edge = (k == 0 && g.head_partial) || k == g.nch - 1;
                uint4 x[VPC];
                read(s, g, k, edge, x);
                if (!edge && k != kt && vec_store && !grad_f32_of(p)) {
                    // whole vectors of the row, no target: one store each
#pragma unroll
                    for (int u = 0; u < VPC; ++u) {
                        unsigned long long g2[W2];
                        E::unpack2(x[u], g2);
#pragma unroll
                        for (int j = 0; j < W2; ++j) {
                            float a, b;
                            f2_unpack(f2_fma(g2[j], kL2E2, nM2), a, b);
                            g2[j] = f2_mul(f2_pack(ex2(a), ex2(b)), esc2);
                        }
                        __stcs(reinterpret_cast<uint4 *>(gA + 16ll * (k * CHV + u * NCT + ct)),
                               E::pack2(g2));
                    }
                    continue;
                }
#pragma unroll
                for (int u = 0; u < VPC; ++u) {
                    const int v = k * CHV + u * NCT + ct;
                    if (v >= g.nv) continue;
                    unsigned long long g2[W2];
                    E::unpack2(x[u], g2);
#pragma unroll
                    for (int j = 0; j < W2; ++j) {
                        float a, b;
                        f2_unpack(f2_fma(g2[j], kL2E2, nM2), a, b);
                        g2[j] = f2_mul(f2_pack(ex2(a), ex2(b)), esc2);
                    }
                    unsigned char *gv = gA + 16ll * v;
                    const bool whole = !((v == 0 && g.head_partial) ||
                                         (v == g.nv - 1 && g.tail_partial));
                    if (grad_f32_of(p)) {
#pragma unroll
                        for (int j = 0; j < W2; ++j) {
                            float a, b;
                            f2_unpack(g2[j], a, b);
                            if (v == vt && 2 * j == dt) a = g_t;
                            if (v == vt && 2 * j + 1 == dt) b = g_t;
                            const long long l = (long long)v * W + 2 * j - g.head;
                            if (l >= 0 && l < C) grad_f32_store<ES>(p, gv + 2 * j * ES, a);
                            if (l + 1 >= 0 && l + 1 < C)
                                grad_f32_store<ES>(p, gv + (2 * j + 1) * ES, b);
                        }
                    }
                    if (whole && vec_store) {
                        __stcs(reinterpret_cast<uint4 *>(gv), E::pack2(g2));
                        if (v == vt) E::store(gv + dt * ES, g_t);
                    } else {
#pragma unroll
                        for (int j = 0; j < W2; ++j) {
                            float a, b;
                            f2_unpack(g2[j], a, b);
                            if (v == vt && 2 * j == dt) a = g_t;
                            if (v == vt && 2 * j + 1 == dt) b = g_t;
                            const long long l = (long long)v * W + 2 * j - g.head;
                            if (l >= 0 && l < C) E::store(gv + 2 * j * ES, a);
                            if (l + 1 >= 0 && l + 1 < C) E::store(gv + (2 * j + 1) * ES, b);
                        }
                    }
                }
            }
        }
    }

    __syncthreads();  // every consumer is done: cta_failed is final
    // A CTA that gave up still owns copies in flight: the producer waits for
    // the last copy of every slot (each for up to the full limit) before the
    // shared memory is released.  A copy that has not landed after that never
    // will; the CTA then leaves rather than hang.
    if (warp == NCW && lane == 0 && cta_failed) {
        for (long long r = issued > nslots ? issued - nslots : 0; r < issued; ++r) {
            if (r == skipped) continue;
            if (!mbar_wait(&full[r % nslots], (uint32_t)((r / nslots) & 1))) break;
        }
    }
    // and its rows' losses are NaN, so the batch loss shows the failure
    if (cta_failed && !is_softmax(p))
        for (long long i = tid; i < nrows; i += NTT) p.loss_rows[blockIdx.x + i * gridDim.x] = NAN;
    finish_cta(p, &tail_flag, tail_scratch);
}

template <typename T, typename P>
cudaError_t launch_p(const P &p, int ctas, int nslots, int smem, int hint, cudaStream_t s) {
    auto kern = row_twopass_kernel<T, P>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(NTT, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, nslots, hint);
}

template <typename T>
cudaError_t launch_t(const ParamsEx &p, int ctas, int nslots, int smem, int hint, cudaStream_t s) {
    if (is_plain(p))
        return launch_p<T, Params>(static_cast<const Params &>(p), ctas, nslots, smem, hint, s);
    return launch_p<T, ParamsEx>(p, ctas, nslots, smem, hint, s);
}

template <typename T>
cudaError_t occ_t(int smem, int *ctas) {
    auto kern = row_twopass_kernel<T, Params>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, NTT, smem);
}

}  // namespace

cudaError_t launch_twopass(const ParamsEx &p, int dtype, int ctas, int nslots, int smem, int hint,
                           cudaStream_t s) {
    if (nslots < 1 || nslots > kTwoPassMaxSlots) return cudaErrorInvalidValue;
    if (dtype == 0) return launch_t<float>(p, ctas, nslots, smem, hint, s);
    if (dtype == 2) return launch_t<__half>(p, ctas, nslots, smem, hint, s);
    return launch_t<__nv_bfloat16>(p, ctas, nslots, smem, hint, s);
}

cudaError_t twopass_max_ctas_per_sm(int dtype, int smem, int *ctas) {
    if (dtype == 0) return occ_t<float>(smem, ctas);
    if (dtype == 2) return occ_t<__half>(smem, ctas);
    return occ_t<__nv_bfloat16>(smem, ctas);
}

}  // namespace ce
