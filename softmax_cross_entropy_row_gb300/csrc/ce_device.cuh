// Device-side building blocks of the softmax cross-entropy kernels (sm_103a):
// PTX wrappers for TMA bulk copies, mbarriers and thread-block clusters, the
// element-type traits, block reductions and the fixed-order batch-loss tail.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ce {

// log2(e) and ln(2) as fp32.  The kernels evaluate e^(z - m) as
// 2^(z*log2e - M) with M = fp32(m*log2e): one FFMA per element and one
// ex2.approx.  M is the same for every element of a row, so its rounding is a
// common factor that cancels in softmax = e/S; the row loss uses the same M.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Bounded waits: a wait gives up after this many SM clock cycles (about a
// second at 2 GHz), records a timeout in the device error word and the kernel
// skips the rest of its work instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;
// Upper bound on one suspended try_wait (ns); the thread wakes as soon as the
// phase completes, so this only limits how often a waiting warp re-polls.
constexpr uint32_t kSuspendHintNs = 20000u;

// Device error word layout (two int32 counters in the workspace).
constexpr int kErrBadTarget = 0;
constexpr int kErrTimeout = 1;

// Kernel parameters shared by every path.
struct Params {
    const unsigned char *logits;  // [B][C] elements, byte pointer
    const int32_t *targets;       // [B]
    unsigned char *grad;          // [B][C] elements, byte pointer
    float *loss_out;              // one fp32
    float *loss_rows;             // workspace: [B] per-row losses
    unsigned int *ticket;         // workspace: CTA completion counter (self-resetting)
    int *err;                     // workspace: error counters
    float2 *parts;                // workspace of the streaming path: [B][chunks] (M, S)
    float *zt;                    // workspace of the streaming path: [B] target logits
    long long B;
    long long C;
    float inv_b;                  // fp32(1/B)
    uint64_t lo_clip;             // TMA-safe byte range of the logits:
    uint64_t hi_clip;             //   [round_up16(begin), round_down16(end))
    int grad_vec_ok;              // grad and logits share their address mod 16
};

// The general call's parameters: a reduction, an upstream gradient, or the
// loss alone.  The kernels are built for Params (the plain call: the mean,
// no upstream gradient, a gradient to write) and for ParamsEx; the plain
// build carries none of the general case's work.
struct ParamsEx : Params {
    int reduction;                // kReduceMean, kReduceSum or kReduceNone
    float grad_base;              // the gradient's row factor: 1/B (mean) or 1 (sum, none)
    const float *grad_scale;      // nullptr (1), one fp32, or [B] fp32 (scale_per_row)
    int scale_per_row;
    int softmax;                  // 1: row softmax forward (no targets, no loss; grad = probabilities)
    // Test hooks (the library's test entry point sets them; the defaults
    // leave every kernel as it is):
    long long copy_wait_limit = kWaitLimitCycles;  // limit of the waits for row copies
    long long skip_copy_row = -1;  // the copy holding this row is never issued
    float *grad_f32 = nullptr;     // [B][C] fp32: the gradient before its rounding
};

constexpr int kReduceMean = 0;
constexpr int kReduceSum = 1;
constexpr int kReduceNone = 2;  // the row losses are the output (loss_rows = loss_out)

__host__ __device__ __forceinline__ constexpr int reduction_of(const Params &) {
    return kReduceMean;
}
__host__ __device__ __forceinline__ int reduction_of(const ParamsEx &p) { return p.reduction; }

// Row softmax forward: no target (no one-hot term, nothing left out of the
// sum), no loss; the "gradient" written is softmax(z_b) itself.
__host__ __device__ __forceinline__ constexpr bool is_softmax(const Params &) { return false; }
__host__ __device__ __forceinline__ bool is_softmax(const ParamsEx &p) { return p.softmax != 0; }

// The target of row b (-1, no target, for the softmax forward).
__device__ __forceinline__ int target_at(const Params &p, long long b) {
    return __ldg(p.targets + b);
}
__device__ __forceinline__ int target_at(const ParamsEx &p, long long b) {
    return p.softmax ? -1 : __ldg(p.targets + b);
}

// false: the loss alone (no gradient computed or written)
__host__ __device__ __forceinline__ constexpr bool writes_grad(const Params &) { return true; }
__host__ __device__ __forceinline__ bool writes_grad(const ParamsEx &p) {
    return p.grad != nullptr;
}

// The upstream gradient when it is one scalar (1 when absent or per row).
__device__ __forceinline__ float scalar_grad_scale(const Params &) { return 1.f; }
__device__ __forceinline__ float scalar_grad_scale(const ParamsEx &p) {
    return (p.grad_scale != nullptr && !p.scale_per_row) ? __ldg(p.grad_scale) : 1.f;
}

// The gradient's factor for row `row`: 1/B (mean) or 1, times the upstream
// gradient (the scalar `scalar` from scalar_grad_scale, or row's own).
__device__ __forceinline__ float row_grad_factor(const Params &p, float, long long) {
    return p.inv_b;
}
__device__ __forceinline__ float row_grad_factor(const ParamsEx &p, float scalar, long long row) {
    return p.grad_base * (p.scale_per_row ? __ldg(p.grad_scale + row) : scalar);
}

// The plain call, which runs the Params build of the kernels.
inline bool is_plain(const ParamsEx &p) {
    return p.reduction == kReduceMean && p.grad_scale == nullptr && p.grad != nullptr &&
           !p.softmax && p.copy_wait_limit == kWaitLimitCycles && p.skip_copy_row < 0 &&
           p.grad_f32 == nullptr;
}

// Test hooks; the plain build has none.
__host__ __device__ __forceinline__ constexpr long long copy_wait_limit(const Params &) {
    return kWaitLimitCycles;
}
__host__ __device__ __forceinline__ long long copy_wait_limit(const ParamsEx &p) {
    return p.copy_wait_limit;
}
// Whether the copy of rows [r0, r1) is left out (its wait can only give up).
__host__ __device__ __forceinline__ constexpr bool skips_copy(const Params &, long long,
                                                              long long) {
    return false;
}
__host__ __device__ __forceinline__ bool skips_copy(const ParamsEx &p, long long r0,
                                                    long long r1) {
    return p.skip_copy_row >= r0 && p.skip_copy_row < r1;
}
__host__ __device__ __forceinline__ constexpr float *grad_f32_of(const Params &) {
    return nullptr;
}
__host__ __device__ __forceinline__ float *grad_f32_of(const ParamsEx &p) { return p.grad_f32; }

// Records the fp32 gradient value v of the element whose gradient lives at
// byte `g` of p.grad (before it is rounded to the logits' type).
template <int ES, typename P>
__device__ __forceinline__ void grad_f32_store(const P &p, const unsigned char *g, float v) {
    if (float *d = grad_f32_of(p)) d[(g - p.grad) / ES] = v;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic: each half is rounded exactly
// as the scalar instruction would round it).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ------------------------------------------------------------ element types

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte vector
    static constexpr uint32_t kNegInfWord = 0xff800000u;  // -inf in every element of a word
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return *reinterpret_cast<const float *>(p);
    }
    __device__ __forceinline__ static float load_global(const unsigned char *p) {
        return __ldg(reinterpret_cast<const float *>(p));
    }
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[4]) {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&v)[4]) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                          __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
    // The vector as fp32 pairs (elements 2i, 2i+1 in pair i).
    __device__ __forceinline__ static void unpack2(const uint4 &w, unsigned long long (&v)[2]) {
        v[0] = (unsigned long long)w.x | ((unsigned long long)w.y << 32);
        v[1] = (unsigned long long)w.z | ((unsigned long long)w.w << 32);
    }
    __device__ __forceinline__ static uint4 pack2(const unsigned long long (&v)[2]) {
        return make_uint4((uint32_t)v[0], (uint32_t)(v[0] >> 32), (uint32_t)v[1],
                          (uint32_t)(v[1] >> 32));
    }
    __device__ __forceinline__ static void store(unsigned char *p, float v) {
        *reinterpret_cast<float *>(p) = v;
    }
    // Running max over 16-byte vectors (exact): accumulator, step, value.
    using MaxAcc = float;
    __device__ __forceinline__ static MaxAcc max_init() { return -INFINITY; }
    __device__ __forceinline__ static void max_step(MaxAcc &m, const uint4 &w) {
        m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                           fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
    }
    __device__ __forceinline__ static float max_value(MaxAcc m) { return m; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    static constexpr uint32_t kNegInfWord = 0xff80ff80u;
    __device__ __forceinline__ static float widen(uint16_t b) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return widen(*reinterpret_cast<const uint16_t *>(p));
    }
    __device__ __forceinline__ static float load_global(const unsigned char *p) {
        return widen(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[8]) {
        v[0] = __uint_as_float(w.x << 16);
        v[1] = __uint_as_float(w.x & 0xffff0000u);
        v[2] = __uint_as_float(w.y << 16);
        v[3] = __uint_as_float(w.y & 0xffff0000u);
        v[4] = __uint_as_float(w.z << 16);
        v[5] = __uint_as_float(w.z & 0xffff0000u);
        v[6] = __uint_as_float(w.w << 16);
        v[7] = __uint_as_float(w.w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float (&v)[8]) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]),
                          pack2(v[6], v[7]));
    }
    // The vector as fp32 pairs (elements 2i, 2i+1 in pair i).
    __device__ __forceinline__ static void unpack2(const uint4 &w, unsigned long long (&v)[4]) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = (unsigned long long)(q[i] << 16) | ((unsigned long long)(q[i] & 0xffff0000u) << 32);
    }
    __device__ __forceinline__ static uint32_t pack_pair(unsigned long long v) {
        float lo, hi;
        f2_unpack(v, lo, hi);
        return pack2(lo, hi);
    }
    __device__ __forceinline__ static uint4 pack2(const unsigned long long (&v)[4]) {
        return make_uint4(pack_pair(v[0]), pack_pair(v[1]), pack_pair(v[2]), pack_pair(v[3]));
    }
    __device__ __forceinline__ static void store(unsigned char *p, float v) {
        *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
    }
    // Running max over 16-byte vectors, kept as a packed bf16 pair (exact:
    // the widening to fp32 is monotonic); one max.bf16x2 per 4 elements.
    using MaxAcc = uint32_t;
    __device__ __forceinline__ static uint32_t max2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ __forceinline__ static MaxAcc max_init() { return kNegInfWord; }
    __device__ __forceinline__ static void max_step(MaxAcc &m, const uint4 &w) {
        m = max2(m, max2(max2(w.x, w.y), max2(w.z, w.w)));
    }
    __device__ __forceinline__ static float max_value(MaxAcc m) {
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

template <>
struct Elem<__half> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    static constexpr uint32_t kNegInfWord = 0xfc00fc00u;
    __device__ __forceinline__ static float widen(uint16_t h) {
        return __half2float(__ushort_as_half(h));
    }
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return widen(*reinterpret_cast<const uint16_t *>(p));
    }
    __device__ __forceinline__ static float load_global(const unsigned char *p) {
        return widen(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ __forceinline__ static float2 widen2(uint32_t w) {
        __half2 h;
        *reinterpret_cast<uint32_t *>(&h) = w;
        return __half22float2(h);  // exact
    }
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[8]) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = widen2(q[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float (&v)[8]) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]),
                          pack2(v[6], v[7]));
    }
    // The vector as fp32 pairs (elements 2i, 2i+1 in pair i).
    __device__ __forceinline__ static void unpack2(const uint4 &w, unsigned long long (&v)[4]) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = widen2(q[i]);
            v[i] = f2_pack(f.x, f.y);
        }
    }
    __device__ __forceinline__ static uint32_t pack_pair(unsigned long long v) {
        float lo, hi;
        f2_unpack(v, lo, hi);
        return pack2(lo, hi);
    }
    __device__ __forceinline__ static uint4 pack2(const unsigned long long (&v)[4]) {
        return make_uint4(pack_pair(v[0]), pack_pair(v[1]), pack_pair(v[2]), pack_pair(v[3]));
    }
    __device__ __forceinline__ static void store(unsigned char *p, float v) {
        *reinterpret_cast<__half *>(p) = __float2half_rn(v);
    }
    // Running max over 16-byte vectors on packed f16 pairs (exact: the
    // widening is monotonic); one max.f16x2 per 4 elements.
    using MaxAcc = uint32_t;
    __device__ __forceinline__ static uint32_t max2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ __forceinline__ static MaxAcc max_init() { return kNegInfWord; }
    __device__ __forceinline__ static void max_step(MaxAcc &m, const uint4 &w) {
        m = max2(m, max2(max2(w.x, w.y), max2(w.z, w.w)));
    }
    __device__ __forceinline__ static float max_value(MaxAcc m) {
        const float2 f = widen2(m);
        return fmaxf(f.x, f.y);
    }
};

// Element d of a 16-byte vector of type E, widened to fp32 (selects, no
// indexing).
template <typename E>
__device__ __forceinline__ float element_of(const uint4 &w, int d) {
    if constexpr (E::kVec == 4) {
        const uint32_t q = (d & 2) ? ((d & 1) ? w.w : w.z) : ((d & 1) ? w.y : w.x);
        return __uint_as_float(q);
    } else {
        const uint32_t q = (d & 4) ? ((d & 2) ? w.w : w.z) : ((d & 2) ? w.y : w.x);
        return E::widen((uint16_t)((d & 1) ? (q >> 16) : (q & 0xffffu)));
    }
}

// The vector w with its element d set to -inf.
template <typename E>
__device__ __forceinline__ uint4 with_neg_inf(uint4 w, int d) {
    if constexpr (E::kVec == 4) {
        if (d == 0) w.x = E::kNegInfWord;
        if (d == 1) w.y = E::kNegInfWord;
        if (d == 2) w.z = E::kNegInfWord;
        if (d == 3) w.w = E::kNegInfWord;
    } else {
        const uint32_t mask = (d & 1) ? 0xffff0000u : 0x0000ffffu;
        const uint32_t ninf = E::kNegInfWord & mask;
        const int q = d >> 1;
        if (q == 0) w.x = (w.x & ~mask) | ninf;
        if (q == 1) w.y = (w.y & ~mask) | ninf;
        if (q == 2) w.z = (w.z & ~mask) | ninf;
        if (q == 3) w.w = (w.w & ~mask) | ninf;
    }
    return w;
}

// ---------------------------------------------------------------- arithmetic

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Warp-wide max in one instruction (NaN inputs are ignored, as fmaxf does);
// every lane gets the same value.
// 1/x by the hardware approximation (rcp.approx.ftz, within 1 ulp); used for
// 1/S, where S >= 1 (the row maximum's own term is 1).
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) by the hardware approximation (lg2.approx.ftz).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The row loss l = log(S / e_t) (Step 3), from S_rest = S - e_t, e_t > 0, S
// and the target logit z_t, with e_t = 2^(z_t*log2e - M):
//   log1p(S_rest / e_t)          when the target dominates (S_rest < e_t, so
//                                l < ln 2 and only this form keeps l's
//                                relative precision);
//   ln2 * (log2(S) - (z_t*log2e - M))   otherwise (l >= ln 2).
__device__ __forceinline__ float row_loss(float s_rest, float e_t, float S, float zt, float M) {
    return s_rest < e_t ? log1pf(s_rest / e_t) : kLn2 * (fast_log2(S) - fmaf(zt, kLog2e, -M));
}

__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Programmatic dependent launch: the next kernel on the stream may start its
// prologue once every CTA of this one has called pdl_trigger(); pdl_wait()
// returns once the previous grid has completed and its memory is visible, so
// a kernel calls it before its first access to global memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// Butterfly sum: every lane ends with the same bits.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------ shared memory

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return done != 0;
}

// Polls between two reads of the clock in the bounded waits: a poll is one
// try_wait and a branch, so a waiting warp takes few issue slots from the
// warps that compute.
constexpr int kPollsPerClockRead = 8;

// Wait for phase `parity` of an mbarrier, for at most `limit` cycles (plus at
// most kPollsPerClockRead suspended polls).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll
        for (int i = 0; i < kPollsPerClockRead; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}

// Wait for phase `parity` of an mbarrier unless the shared flag `*flag`
// becomes non-zero first: 1 when the phase completed, 0 when the flag was
// seen, -1 after `limit` cycles.
__device__ __forceinline__ int mbar_wait_or_flag(uint64_t *bar, uint32_t parity,
                                                 const int *flag, long long limit) {
    if (mbar_try_wait(bar, parity)) return 1;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll
        for (int i = 0; i < kPollsPerClockRead; ++i)
            if (mbar_try_wait(bar, parity)) return 1;
        if (*reinterpret_cast<const volatile int *>(flag) != 0) return 0;
        if (clock64() - t0 > limit) return -1;
    }
}

// One TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 eviction policy (a createpolicy value) for the
// lines it reads.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 eviction policies covering every access made with them: lines to keep
// (read again soon) and lines to drop first (read for the last time).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One TMA bulk copy of this CTA's shared memory to global memory, in the
// calling thread's bulk group (then bulk_commit).  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until every committed bulk store of this thread has read its shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(const unsigned char *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// Named barriers (ids 1..15; id 0 is __syncthreads): a non-blocking arrival
// and a waiting arrival, `threads` counting both.
__device__ __forceinline__ void named_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Read a float4 from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float4 ld_dsmem_f4(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)),
                 "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// Read a float from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float ld_dsmem_f32(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)),
                 "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Shared::cluster address of `local`'s counterpart in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)),
                 "r"(rank));
    return remote;
}

// Store 16 bytes into the shared memory of a CTA of the cluster (`dst`, a
// shared::cluster address) and complete 16 bytes of the transaction count of
// that CTA's mbarrier `bar` (also a shared::cluster address).  The completion
// releases the data at cluster scope; nothing waits for it here.
__device__ __forceinline__ void st_async_f4(uint32_t dst, float4 v, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(dst),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
        : "memory");
}

// try_wait with acquire at cluster scope: for phases completed by other CTAs'
// st.async transactions.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll
        for (int i = 0; i < kPollsPerClockRead; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
}

// ---------------------------------------------------------- batch-loss tail

// Error-free sum of two floats (Knuth's TwoSum): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// The batch loss L = (1/B) * sum_b loss_rows[b] is summed in one fixed order
// that depends only on B, with compensated (float, float) accumulators:
//   virtual lane i (of 256) sums rows 4i..4i+3, 4i+1024..4i+1027, ... in order;
//   virtual warp w (lanes 32w..32w+31) combines its lanes in a shuffle-down tree;
//   the 8 virtual warps are added in order.
// Any number of real warps may evaluate it: the bits are the same.
constexpr int kTailThreads = 256;
constexpr int kTailWarps = kTailThreads / 32;

// Total of virtual warp `vw`, valid in lane 0 of the calling warp.  The
// lane's row losses are fetched kTailDepth float4s at a time, all loads in
// flight before the ordered additions.
constexpr int kTailDepth = 4;
__device__ __forceinline__ float2 tail_virtual_warp(const Params &p, int vw, int lane) {
    const int vl = vw * 32 + lane;
    const long long B = p.B;
    float hi = 0.f, lo = 0.f;
    for (long long base0 = 4LL * vl; base0 < B; base0 += 4LL * kTailThreads * kTailDepth) {
        float4 q[kTailDepth];
#pragma unroll
        for (int m = 0; m < kTailDepth; ++m) {
            const long long base = base0 + 4LL * kTailThreads * m;
            if (base + 3 < B) {
                q[m] = __ldcg(reinterpret_cast<const float4 *>(p.loss_rows + base));
            } else {
                q[m].x = base + 0 < B ? __ldcg(p.loss_rows + base + 0) : 0.f;
                q[m].y = base + 1 < B ? __ldcg(p.loss_rows + base + 1) : 0.f;
                q[m].z = base + 2 < B ? __ldcg(p.loss_rows + base + 2) : 0.f;
                q[m].w = 0.f;
            }
        }
#pragma unroll
        for (int m = 0; m < kTailDepth; ++m) {
            if (base0 + 4LL * kTailThreads * m < B) {
                const float x[4] = {q[m].x, q[m].y, q[m].z, q[m].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float s, e;
                    two_sum(hi, x[k], s, e);
                    hi = s;
                    lo += e;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_down_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_down_sync(0xffffffffu, lo, o);
        float s, e;
        two_sum(hi, h2, s, e);
        hi = s;
        lo += l2 + e;
    }
    return make_float2(hi, lo);
}

// Adds the 8 virtual-warp totals in order, writes L and re-arms the ticket.
// The sum h + l is the loss of the sum reduction; for the mean, (h + l) / B
// is formed in fp32 with one correction step (no fp64: its division is a long
// dependent sequence on this part):
//   q0 = h * fp32(1/B),  r = (h - q0 B) + l  (the fma is exact up to one
//   rounding),  L = q0 + r * fp32(1/B).
template <typename P>
__device__ __forceinline__ void tail_write(const P &p, const float2 *vw_totals) {
    float h = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kTailWarps; ++w) {
        float s, e;
        two_sum(h, vw_totals[w].x, s, e);
        h = s;
        l += vw_totals[w].y + e;
    }
    if (reduction_of(p) == kReduceSum) {
        *p.loss_out = h + l;
    } else {
        const float q0 = h * p.inv_b;
        const float r = fmaf(-q0, static_cast<float>(p.B), h) + l;
        *p.loss_out = fmaf(r, p.inv_b, q0);
    }
    *p.ticket = 0u;  // ready for the next launch on this workspace
}

// CTA-wide publication of the row losses: called by every thread once the
// CTA's row losses are stored; returns true (in every thread) in the CTA that
// finishes last.  `flag` lives in shared memory.
__device__ __forceinline__ bool publish_rows(const Params &p, int *flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        // acquire-release at GPU scope: publishes this CTA's row losses (the
        // barrier above orders the other threads' stores before it) and, in
        // the last CTA, makes every other CTA's visible to the loads of the
        // batch tail (the barrier after it extends that to the other threads)
        const unsigned int total = gridDim.x * gridDim.y * gridDim.z;
        unsigned int prev;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(p.ticket)
                     : "memory");
        *flag = (prev == total - 1u);
    }
    __syncthreads();
    return *flag != 0;
}

// The batch loss, evaluated by every thread of the last CTA (one virtual warp
// per real warp).  `scratch` ([8]) lives in shared memory.
template <typename P>
__device__ __forceinline__ void batch_tail(const P &p, float2 *scratch) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int vw = warp; vw < kTailWarps; vw += blockDim.x >> 5) {
        const float2 v = tail_virtual_warp(p, vw, lane);
        if (lane == 0) scratch[vw] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) tail_write(p, scratch);
}

// publish_rows, then the batch tail in the last CTA (nothing to do when the
// row losses are themselves the output).
template <typename P>
__device__ __forceinline__ void finish_cta(const P &p, int *flag, float2 *scratch) {
    if (reduction_of(p) == kReduceNone || is_softmax(p)) return;
    if (publish_rows(p, flag)) batch_tail(p, scratch);
}

}  // namespace ce
