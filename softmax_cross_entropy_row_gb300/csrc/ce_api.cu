// C-ABI of the fused softmax cross-entropy forward + gradient (include/ce.h):
// argument checks, the per-stream workspace, the choice of kernel path and the
// launch.  Nothing here computes on the host; every step runs in the kernels.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "../../include/ce.h"
#include "../../include/ce_testing.h"
#include "ce_launch.h"
#include "ce_rows_online.h"

namespace {

using ce::Params;
using ce::ParamsEx;

thread_local char g_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
    const char *s = cudaGetErrorString(e);
    strncpy(g_cuda_error, s ? s : "unknown CUDA error", sizeof g_cuda_error - 1);
    g_cuda_error[sizeof g_cuda_error - 1] = '\0';
    return CE_ERR_CUDA;
}

// ----------------------------------------------------------- device facts

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;  // max dynamic shared memory per CTA
    int pageable = 0;    // device can access pageable host memory
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

int device_info(int dev, DeviceInfo *out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
        *out = it->second;
        return CE_OK;
    }
    DeviceInfo d;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&d.pageable, cudaDevAttrPageableMemoryAccess, dev)) !=
        cudaSuccess)
        return cuda_fail(e);
    g_dev[dev] = d;
    *out = d;
    return CE_OK;
}

// ---------------------------------------------------------------- plans

// Occupancy answers per (device, dtype, path, split, smem), so that a call made
// during stream capture repeats no occupancy query of an earlier call.
std::mutex g_occ_mu;
std::map<std::tuple<int, int, int, int, int>, int> g_occ;

template <typename F>
int cached_occupancy(int dtype, int path, int split, int smem, F query, int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const auto key = std::make_tuple(dev, dtype, path, split, smem);
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            *out = it->second;
            return CE_OK;
        }
    }
    int v = 0;
    if ((e = query(&v)) != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = v;
    *out = v;
    return CE_OK;
}

struct Plan {
    int path = 0;
    int split = 0;        // CTAs per row (split path) / classes per chunk (stream)
    int ctas = 0;         // CTAs of the (main) launch
    int threads = 0;
    int smem = 0;         // dynamic shared memory per CTA
    int launches = 1;
    int nslots = 0;       // staged slices (split) or tiles per warp (warp path)
    int slot_bytes = 0;
    long long slice = 0;  // classes per slice (split path)
    int rows_per_tile = 0;
    int per_sm = 1;       // warp path: the build for 1, 2 or 3 resident CTAs per SM
    int swept_nw = 0;     // warp path, rows swept in shared memory: warps per CTA (else 0)
    int vecs = 8;         // split path: 16-byte vectors per thread (8, 12 or 16)
    bool pipe = false;    // split path: the pipelined kernel (slices of at most 8 vectors)
    int split_threads = ce::kSplitThreads;  // split path at K = 1: threads per CTA
    long long chunks = 0; // stream path
    int online_build = 0; // loss-only warp-per-row path: the kernel build
};

constexpr int kStaticSmemReserve = 2048;       // static __shared__ of the kernels
constexpr long long kWarpRowMax = 8192;        // bytes: warp-per-row path up to here
constexpr long long kWarpTileTarget = 2048;    // bytes of rows per warp tile
constexpr long long kOnlineMinRowsPerSm = 8;   // loss-only warp-per-row path from here

int round_up(long long v, long long a) { return (int)((v + a - 1) / a * a); }

// Tuning knob: CE_WARP_PER_SM=1, 2 or 3 forces the warp path's CTAs per SM
// (0 or unset: chosen from the shape).  Read once.
int warp_per_sm_override() {
    static const int n = [] {
        const char *e = getenv("CE_WARP_PER_SM");
        return e ? atoi(e) : 0;
    }();
    return n;
}

// Tuning knob: CE_SPLIT_PIPE=0 keeps split rows on the barrier-per-row
// kernel even where the pipelined one applies.  Read once.
bool split_pipe_enabled() {
    static const bool on = [] {
        const char *e = getenv("CE_SPLIT_PIPE");
        return !(e && atoi(e) == 0);
    }();
    return on;
}

// Tuning knob: CE_SPLIT_STAGE=0 makes the barrier-per-row split kernel store
// its gradient directly instead of through the row's slot.  Read once.
bool split_stage_enabled() {
    static const bool on = [] {
        const char *e = getenv("CE_SPLIT_STAGE");
        return !(e && atoi(e) == 0);
    }();
    return on;
}

int plan_warp(long long B, long long C, int es, const DeviceInfo &d, int dtype, Plan *pl) {
    const long long row_bytes = C * es;
    if (row_bytes > kWarpRowMax) return CE_ERR_PATH;
    long long R = kWarpTileTarget / row_bytes;
    if (R < 1) R = 1;
    if (R > B) R = B;
    const int slot_bytes = round_up(R * row_bytes + 32, 128);
    const long long ntiles = (B + R - 1) / R;
    // Two or three CTAs per SM with one staged tile per warp when every tile
    // then has a warp of its own (all copies in flight at once): 2 x 16 or
    // 3 x 9 warps, whichever leaves fewer tiles on the busiest SM (2 x 16 on a
    // tie); otherwise one CTA per SM with a ring of up to four tiles per warp.
    // The multi-CTA builds hold four 16-byte vectors per lane without
    // spilling; fp32 rows of up to eight (a few spilled registers) still ran
    // faster there than with one CTA per SM (4096 x 1000 fp32: 10.6 vs 11.3 us).
    int want = 1;
    int slots = 1;
    const int force = warp_per_sm_override();
    const bool light = (C * es / 16 + 31) / 32 <= (es == 4 ? 8 : 4);
    auto fits = [&](int per_sm) {
        return (long long)slot_bytes * ce::warp_kernel_warps(per_sm) <=
               d.smem_optin / per_sm - kStaticSmemReserve;
    };
    auto busiest = [&](int per_sm) {  // tiles on the busiest SM, all CTAs resident
        const long long nw = ce::warp_kernel_warps(per_sm);
        const long long ctas = (ntiles + nw - 1) / nw;
        if (!fits(per_sm) || ctas > (long long)per_sm * d.sms) return LLONG_MAX;
        return (ctas + d.sms - 1) / d.sms * nw;
    };
    if (force == 2 || force == 3) {
        if (fits(force)) want = force;
    } else if (force != 1 && light) {
        const long long b2 = busiest(2), b3 = busiest(3);
        if (b2 != LLONG_MAX || b3 != LLONG_MAX) want = b3 < b2 ? 3 : 2;
    }
    const int NW = ce::warp_kernel_warps(want);
    if (want == 1) {
        const int budget = d.smem_optin - kStaticSmemReserve;
        slots = ce::kMaxWarpSlots;
        while (slots > 1 && (long long)slots * slot_bytes * NW > budget) --slots;
        if ((long long)slots * slot_bytes * NW > budget) return CE_ERR_PATH;
    }
    const int smem = slots * slot_bytes * NW;
    int per_sm = 1;
    int rc = cached_occupancy(
        dtype, CE_PATH_ROWS_WARP, (int)C * 4 + want, smem,
        [&](int *v) { return ce::rows_warp_max_ctas_per_sm(dtype, want, C, smem, v); }, &per_sm);
    if (rc != CE_OK) return rc;
    if (per_sm < 1) return CE_ERR_PATH;
    if (per_sm > want) per_sm = want;
    long long ctas = (ntiles + NW - 1) / NW;
    const long long cap = (long long)d.sms * per_sm;
    if (ctas > cap) ctas = cap;
    pl->path = CE_PATH_ROWS_WARP;
    pl->split = 1;
    pl->ctas = (int)ctas;
    pl->threads = NW * 32;
    pl->smem = smem;
    pl->launches = 1;
    pl->nslots = slots;
    pl->slot_bytes = slot_bytes;
    pl->rows_per_tile = (int)R;
    pl->per_sm = want;
    return CE_OK;
}

// Tuning knobs: CE_SWEPT_WARPS=16, 8 or 4 and CE_SWEPT_SLOTS=1..4 force the
// swept warp path's warps per CTA and slots per warp (0 or unset: chosen
// from the row's bytes).  Read once.
int env_int_once(const char *name, int *cache) {
    if (*cache < 0) {
        const char *e = getenv(name);
        *cache = e ? atoi(e) : 0;
    }
    return *cache;
}
int swept_warps_override() {
    static int v = -1;
    return env_int_once("CE_SWEPT_WARPS", &v);
}
int swept_slots_override() {
    static int v = -1;
    return env_int_once("CE_SWEPT_SLOTS", &v);
}
// Tuning knob: CE_SPLIT_THREADS=512 keeps the split kernel at K = 1 in CTAs
// of kSplitThreads threads for rows a 128-thread CTA holds (0 or unset: 128
// threads there).  Read once.
int split_threads_override() {
    static int v = -1;
    return env_int_once("CE_SPLIT_THREADS", &v);
}

// Warp path for rows longer than a warp's registers hold (8 KB .. 48 KB):
// one row per tile, swept in its slot.  What the time depends on is the
// warps resident per SM (each sweeps its row with little parallelism of its
// own): measured on GB300 (16384 rows), one slot per warp and the most
// resident warps won -- 12 KB rows 0.77-0.78 of peak with 16 warps per SM,
// 16 KB bf16 rows 0.81 with three 4-warp CTAs per SM against 0.49 with one
// CTA of four warps and three slots each, 24 KB rows 0.76-0.88 with 8 warps
// -- and with 4 warps per SM (31 KB rows) the two-pass kernel is faster.  So
// the build (16, 8 or 4 warps per CTA) with the most resident warps per SM
// is taken, one slot per warp (ties: the larger CTA); the planner's own
// choice requires 8 resident warps per SM, a forced warp path takes
// whatever fits.
int plan_warp_swept(long long B, long long C, int es, const DeviceInfo &d, int dtype, bool forced,
                    Plan *pl) {
    const long long row_bytes = C * es;
    if (row_bytes > ce::kWarpChunkRowMax) return CE_ERR_PATH;
    const int budget = d.smem_optin - kStaticSmemReserve;
    const int slot_bytes = round_up(row_bytes + 32, 128);
    auto resident = [&](int nw, int slots, int *per_sm) {
        const int smem = slots * slot_bytes * nw;
        return cached_occupancy(
            dtype, CE_PATH_ROWS_WARP, -nw - 100 * slots, smem,
            [&](int *v) { return ce::rows_warp_swept_max_ctas_per_sm(dtype, nw, smem, v); },
            per_sm);
    };
    int nw = 0, slots = 1, per_sm = 0;
    const int fw = swept_warps_override(), fs = swept_slots_override();
    for (int w : {16, 8, 4}) {
        if (fw && w != fw) continue;
        const int sl = fs >= 1 && fs <= ce::kMaxWarpSlots ? fs : 1;
        if ((long long)sl * w * slot_bytes > budget) continue;
        int n = 0;
        const int rc = resident(w, sl, &n);
        if (rc != CE_OK) return rc;
        if (n >= 1 && w * n > nw * per_sm) {
            nw = w;
            slots = sl;
            per_sm = n;
        }
    }
    if (nw == 0) return CE_ERR_PATH;
    if (!forced && nw * per_sm < 8) return CE_ERR_PATH;
    long long ctas = (B + nw - 1) / nw;
    const long long cap = (long long)d.sms * per_sm;
    if (ctas > cap) ctas = cap;
    pl->path = CE_PATH_ROWS_WARP;
    pl->split = 1;
    pl->ctas = (int)ctas;
    pl->threads = nw * 32;
    pl->smem = slots * slot_bytes * nw;
    pl->launches = 1;
    pl->nslots = slots;
    pl->slot_bytes = slot_bytes;
    pl->rows_per_tile = 1;
    pl->per_sm = 1;
    pl->swept_nw = nw;
    return CE_OK;
}

// Split-row path: K CTAs per row (a cluster when K > 1), each holding a
// slice of SE classes in registers (at most kSplitThreads x 16 vectors, i.e.
// 128 KB) with a ring of at least two shared-memory slots.  The smallest such
// K is chosen: fewer CTAs per row means fewer exchanges per byte.  For K > 1,
// slices of at most 8 vectors per thread run on the pipelined kernel (no
// CTA-wide barrier per row); the rest on the barrier-per-row kernel.
int plan_split(long long B, long long C, int es, const DeviceInfo &d, int dtype, int K_forced,
               Plan *pl) {
    const int budget = d.smem_optin - kStaticSmemReserve;
    const long long per_vec_cap = (long long)ce::kSplitThreads * 16;  // bytes per vector slot
    auto slice_of = [&](int K) {
        long long se = (C + K - 1) / K;
        return (se + 7) / 8 * 8;  // slices start 16-byte aligned relative to the row
    };
    // vectors per thread for a slice (its bytes plus the two partial vectors)
    auto vecs_of = [&](long long se) {
        const long long need = se * es + 32;
        return need <= 8 * per_vec_cap ? 8 : need <= 12 * per_vec_cap ? 12
                                           : need <= 16 * per_vec_cap ? 16 : 0;
    };
    auto slot_of = [&](long long se) { return (long long)round_up(se * es + 32, 128); };
    auto nslots_of = [&](long long se) {
        long long n = budget / slot_of(se);
        return (int)(n > ce::kMaxSplitSlots ? ce::kMaxSplitSlots : n);
    };
    // 16-bit slices re-evaluate their exponentials for the gradient, so their
    // per-thread work grows twice as fast with the slice: on 128k-class bf16
    // rows, 4 CTAs of 64 KB ran faster than 3 of 96 KB, so bf16 and f16 stop
    // at 8.
    const int auto_max_vecs = es == 2 ? 8 : 16;
    int K = K_forced;
    if (K == 0) {
        for (int k : {1, 2, 3, 4, 6, 8}) {
            const long long se = slice_of(k);
            const int v = vecs_of(se);
            if (v && v <= auto_max_vecs && nslots_of(se) >= 2) {
                K = k;
                break;
            }
        }
        if (K == 0) return CE_ERR_PATH;
    }
    if (K != 1 && K != 2 && K != 3 && K != 4 && K != 6 && K != 8) return CE_ERR_PATH;
    const long long se = slice_of(K);
    int vecs = vecs_of(se);
    int nslots = nslots_of(se);
    // K = 1 rows of at most 32 KB (16 vectors per thread): 128-thread CTAs,
    // two slots each, several CTAs per SM.  Measured on GB300 (8192 rows):
    // 31 KB rows 0.80 of peak bf16 / 0.92 fp32, against 0.54 / 0.68 in one
    // 512-thread CTA per SM, which pays ~2.3 us per row; 192- and 256-thread
    // CTAs ran slower than 512 on 32-48 KB rows (one CTA per SM by registers).
    // f16 is built for 8 vectors per thread only.
    int nt = ce::kSplitThreads;
    if (K == 1 && split_threads_override() != ce::kSplitThreads) {
        const long long need = se * es + 32, cap = 128LL * 16;
        const int v128 = need <= 8 * cap ? 8 : need <= 12 * cap ? 12 : need <= 16 * cap ? 16 : 0;
        if (v128 && !(dtype == CE_F16 && v128 > 8)) {
            nt = 128;
            vecs = v128;
            if (nslots > 2) nslots = 2;
        }
    }
    if (vecs == 0 || nslots < 1) return CE_ERR_PATH;
    if (dtype == CE_F16 && vecs > 8) return CE_ERR_PATH;  // f16 is built for 8 vectors only
    const long long slot_bytes = slot_of(se);
    const int smem = nslots * (int)slot_bytes;
    // K > 1 with slices of at most 8 vectors per thread: the pipelined kernel
    // (for K = 1 the barrier-per-row kernel measured faster)
    const bool pipe = K > 1 && vecs <= ce::kPipeVecs && split_pipe_enabled();
    int clusters = 0;
    int rc = cached_occupancy(
        dtype, CE_PATH_ROW_SPLIT, K * 64 + vecs + (pipe ? 32 : 0) + nt * 1000, smem,
        [&](int *v) {
            return pipe ? ce::split_pipe_max_clusters(dtype, K, smem, v)
                        : ce::split_max_clusters(dtype, K, nt, vecs, smem, v);
        },
        &clusters);
    if (rc != CE_OK) return rc;
    if (clusters < 1) return CE_ERR_PATH;
    if ((long long)clusters > B) clusters = (int)B;
    pl->path = CE_PATH_ROW_SPLIT;
    pl->split = K;
    pl->ctas = clusters * K;
    pl->threads = nt;
    pl->split_threads = nt;
    pl->vecs = vecs;
    pl->pipe = pipe;
    pl->smem = smem;
    pl->launches = 1;
    pl->nslots = nslots;
    pl->slot_bytes = (int)slot_bytes;
    pl->slice = se;
    return CE_OK;
}

// Tuning knob: CE_TWOPASS_HINT=0 leaves the L2 eviction hints off the
// two-pass path's copies (to measure what they are worth).  Read once.
int twopass_hint() {
    static const int h = [] {
        const char *e = getenv("CE_TWOPASS_HINT");
        return (e && atoi(e) == 0) ? 0 : 1;
    }();
    return h;
}

// Two-pass path: one CTA per SM, a row at a time, with a ring of chunks as
// deep as shared memory allows (7 x 32 KB on GB300: deeper than one pass over
// a 200 KB row, so the next row's first pass is read from HBM while the
// current row's second pass is served by L2); any row length.
int plan_twopass(long long B, const DeviceInfo &d, int dtype, Plan *pl) {
    const int chb = ce::kTwoPassChunkBytes;
    int nslots = (d.smem_optin - kStaticSmemReserve) / chb;
    if (nslots > ce::kTwoPassMaxSlots) nslots = ce::kTwoPassMaxSlots;
    if (nslots < 2) return CE_ERR_PATH;
    const int smem = nslots * chb;
    int per_sm = 0;
    int rc = cached_occupancy(
        dtype, CE_PATH_ROW_TWOPASS, 0, smem,
        [&](int *v) { return ce::twopass_max_ctas_per_sm(dtype, smem, v); }, &per_sm);
    if (rc != CE_OK) return rc;
    if (per_sm < 1) return CE_ERR_PATH;
    long long ctas = (long long)d.sms;
    if (ctas > B) ctas = B;
    pl->path = CE_PATH_ROW_TWOPASS;
    pl->split = 1;
    pl->ctas = (int)ctas;
    pl->threads = ce::kTwoPassThreads;
    pl->smem = smem;
    pl->launches = 1;
    pl->nslots = nslots;
    pl->slot_bytes = chb;
    pl->per_sm = 1;
    return CE_OK;
}

// Loss-only warp-per-row path: a warp streams each row once from global
// memory (no staging), so its time is set by how many loads the resident
// warps keep in flight.  Measured on GB300 (loss alone, mean): the build of
// 16 vectors per lane per step (8 KB per warp) and two 8-warp CTAs per SM is
// the fastest or within 1% of it on rows of 16 KB to 256 KB (8192 x 32000
// bf16 107 -> 81 us against the split kernel, 4096 x 128256 bf16 169 -> 151
// against the two-pass kernel, 16384 x 16000 bf16 123 -> 80 against the
// swept warp kernel), but a row that leaves its last step mostly empty wastes
// that step's issue slots: 12 KB fp32 and 18 KB bf16 rows ran 8% faster on
// the build of 4 vectors per lane (2 KB per step, five CTAs per SM).  So the
// 8 KB build is taken when the row fills at least 90% of its steps, else the
// 2 KB one.  Rows are dealt to warps round-robin; the grid has just enough
// warps that each takes the same number of rows, ceil(B / w) with w the
// resident warps, so no warp has a row more than the others.
// `build_forced`: 0 = choose, else build_forced - 1.
int online_build_for(long long row_bytes) {
    constexpr long long kStepBytes = 32LL * 16 * 16;  // build 3: 16 vectors per lane
    const long long steps = (row_bytes + kStepBytes - 1) / kStepBytes;
    return row_bytes * 10 >= steps * kStepBytes * 9 ? 3 : 4;
}

int plan_online(long long B, long long row_bytes, const DeviceInfo &d, int dtype, int build_forced,
                Plan *pl) {
    const int build = build_forced > 0 ? build_forced - 1 : online_build_for(row_bytes);
    if (build >= ce::kOnlineBuilds) return CE_ERR_PATH;
    int per_sm = 0;
    int rc = cached_occupancy(
        dtype, CE_PATH_ROWS_ONLINE, build, 0,
        [&](int *v) { return ce::rows_online_max_ctas_per_sm(dtype, build, v); }, &per_sm);
    if (rc != CE_OK) return rc;
    if (per_sm < 1) return CE_ERR_PATH;
    const long long resident = (long long)per_sm * d.sms * ce::kOnlineWarps;
    const long long rows_per_warp = (B + resident - 1) / resident;
    const long long warps = (B + rows_per_warp - 1) / rows_per_warp;
    pl->path = CE_PATH_ROWS_ONLINE;
    pl->split = build + 1;
    pl->ctas = (int)((warps + ce::kOnlineWarps - 1) / ce::kOnlineWarps);
    pl->threads = ce::kOnlineWarps * 32;
    pl->smem = 0;
    pl->launches = 1;
    pl->online_build = build;
    return CE_OK;
}

int plan_stream(long long B, long long C, Plan *pl) {
    const long long chunks = (C + ce::kStreamChunk - 1) / ce::kStreamChunk;
    if (B * chunks > 0x7fffffffLL) return CE_ERR_SHAPE;
    pl->path = CE_PATH_STREAM;
    pl->split = ce::kStreamChunk;
    pl->ctas = (int)(B * chunks);
    pl->threads = ce::kStreamThreads;
    pl->smem = 0;
    pl->launches = 2;
    pl->chunks = chunks;
    return CE_OK;
}

cudaError_t launch_split_plan(const ce::ParamsEx &p, int dtype, const Plan &pl, cudaStream_t s) {
    if (pl.pipe)
        return ce::launch_split_pipe(p, dtype, pl.split, pl.ctas, pl.nslots, pl.slot_bytes,
                                     pl.slice, pl.smem, s);
    // staging hands a slot back one row late, so it needs a second slot (with
    // one, the next row's copy would wait for a slot that never comes back)
    const int staged = split_stage_enabled() && pl.nslots >= 2 ? 1 : 0;
    return ce::launch_split(p, dtype, pl.split, pl.split_threads, pl.vecs, pl.ctas, pl.nslots,
                            pl.slot_bytes, pl.slice, pl.smem, staged, s);
}

cudaError_t launch_plan(const ce::ParamsEx &p, int dtype, const Plan &pl, cudaStream_t s) {
    switch (pl.path) {
        case CE_PATH_ROWS_WARP:
            if (pl.swept_nw)
                return ce::launch_rows_warp_swept(p, dtype, pl.swept_nw, pl.ctas, pl.nslots,
                                                  pl.slot_bytes, pl.smem, s);
            return ce::launch_rows_warp(p, dtype, pl.per_sm, pl.ctas, pl.nslots, pl.rows_per_tile,
                                        pl.slot_bytes, pl.smem, s);
        case CE_PATH_ROW_SPLIT:
            return launch_split_plan(p, dtype, pl, s);
        case CE_PATH_ROW_TWOPASS:
            return ce::launch_twopass(p, dtype, pl.ctas, pl.nslots, pl.smem, twopass_hint(), s);
        case CE_PATH_ROWS_ONLINE:
            return ce::launch_rows_online(p, dtype, pl.online_build, pl.ctas, s);
        default:
            return ce::launch_stream(p, dtype, pl.chunks, s);
    }
}

// loss_only: no gradient and no softmax output is written (the call's
// grad_out is NULL).
int make_plan(long long B, long long C, int dtype, int path, int split, Plan *pl,
              bool loss_only = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    int rc = device_info(dev, &d);
    if (rc != CE_OK) return rc;
    const int es = dtype == CE_F32 ? 4 : 2;
    const long long row_bytes = C * es;
    switch (path) {
        case CE_PATH_AUTO:
            // rows of at most 8 KB: a warp each, held in registers; rows for
            // which 8 warps per SM fit: a warp each, swept in shared memory;
            // rows one CTA holds in registers: the split kernel at K = 1;
            // longer rows: two passes through one CTA (measured faster on
            // GB300 than splitting a row across a cluster or the streaming
            // path); the loss alone, on rows past 8 KB in batches of at least
            // 8 rows per SM: a warp per row, read once (at 4 rows per SM the
            // other kernels were faster: 11.0 against 13.5 us on 32000 bf16)
            if (row_bytes <= kWarpRowMax) return plan_warp(B, C, es, d, dtype, pl);
            if (loss_only && B >= kOnlineMinRowsPerSm * (long long)d.sms) {
                rc = plan_online(B, row_bytes, d, dtype, 0, pl);
                if (rc != CE_ERR_PATH) return rc;
            }
            rc = plan_warp_swept(B, C, es, d, dtype, false, pl);
            if (rc != CE_ERR_PATH) return rc;
            rc = plan_split(B, C, es, d, dtype, 0, pl);
            if (rc == CE_OK && pl->split == 1) return rc;
            if (rc != CE_OK && rc != CE_ERR_PATH) return rc;
            return plan_twopass(B, d, dtype, pl);
        case CE_PATH_ROWS_WARP:
            if (row_bytes <= kWarpRowMax) return plan_warp(B, C, es, d, dtype, pl);
            return plan_warp_swept(B, C, es, d, dtype, true, pl);
        case CE_PATH_ROW_SPLIT: return plan_split(B, C, es, d, dtype, split, pl);
        case CE_PATH_STREAM:
            if (split != 0 && split != ce::kStreamChunk) return CE_ERR_PATH;
            return plan_stream(B, C, pl);
        case CE_PATH_ROW_TWOPASS: return plan_twopass(B, d, dtype, pl);
        case CE_PATH_ROWS_ONLINE:
            if (!loss_only) return CE_ERR_PATH;
            return plan_online(B, row_bytes, d, dtype, split, pl);
        default: return CE_ERR_PATH;
    }
}

// -------------------------------------------------------------- workspace

// Per (device, stream): [ticket u32 | bad-target i32 | timeout i32 | pad] in
// the first 256 bytes, then B (rounded up) fp32 row losses, then the
// streaming path's partials.  Kernels leave the ticket at zero when they end.
struct Workspace {
    unsigned char *base = nullptr;
    size_t bytes = 0;
};

std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;
// Outgrown workspaces (device, base): a CUDA graph captured with a call that
// used one still holds its address, so it stays allocated until
// ce_release_workspaces.
std::vector<std::pair<int, unsigned char *>> g_ws_retired;

// Host-buffer entry points: per (device, stream) staging buffers (two chunks
// of logits, two of gradient, the targets), two helper streams for the copies
// in and out, and the events that order the three streams.  Guarded by
// g_ws_mu.
struct HostPipe {
    unsigned char *z[2] = {nullptr, nullptr};  // logits chunks
    unsigned char *g[2] = {nullptr, nullptr};  // gradient chunks (gradient to the host)
    size_t chunk_bytes = 0;                    // bytes of each z / g buffer
    size_t g_bytes = 0;                        // bytes of each g buffer allocated (0: none)
    unsigned char *t = nullptr;                // targets
    size_t tbytes = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr};   // chunk copied in
    cudaEvent_t ev_k[2] = {nullptr, nullptr};    // chunk's kernel done
    cudaEvent_t ev_out[2] = {nullptr, nullptr};  // chunk's gradient copied out
};
std::map<std::pair<int, uintptr_t>, HostPipe> g_hs;

constexpr size_t kHeaderBytes = 256;
constexpr size_t kLossSlot = 64;  // header bytes holding the host entry's device copy of L

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int get_workspace(int dev, cudaStream_t s, size_t need, Workspace *out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace &w = g_ws[{dev, reinterpret_cast<uintptr_t>(s)}];
    if (w.bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(s, &cs);
        if (e != cudaSuccess) return cuda_fail(e);
        if (cs != cudaStreamCaptureStatusNone) return CE_ERR_CAPTURE;
        if (w.base) {
            // not freed: kernels in flight and graphs captured earlier on this
            // stream may still use it
            g_ws_retired.push_back({dev, w.base});
            w.base = nullptr;
            w.bytes = 0;
        }
        size_t bytes = align_up(need, 1 << 16);
        void *p = nullptr;
        if ((e = cudaMalloc(&p, bytes)) != cudaSuccess) return cuda_fail(e);
        // Ordered before this call's kernel on the same stream.
        if ((e = cudaMemsetAsync(p, 0, kHeaderBytes, s)) != cudaSuccess) {
            cudaFree(p);
            return cuda_fail(e);
        }
        w.base = static_cast<unsigned char *>(p);
        w.bytes = bytes;
    }
    *out = w;
    return CE_OK;
}

// ------------------------------------------------------------- validation

bool ranges_overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
    return a < b + nb && b < a + na;
}

int check_pointer(const void *p, const DeviceInfo &d) {
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CE_ERR_POINTER;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return CE_OK;
    if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) return CE_OK;
    if (at.type == cudaMemoryTypeUnregistered && d.pageable) return CE_OK;
    return CE_ERR_POINTER;
}

// grad_out == nullptr: loss only.  grad_scale: nullptr, one fp32 (mean,
// sum) or [B] fp32 (none).  loss_out: one fp32 (mean, sum) or [B] (none).
// softmax: the row softmax forward -- no targets and no loss; grad_out
// receives softmax(z_b).
// hooks: the test entry point's (NULL for every other call).
int run(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
        int reduction, const float *grad_scale, float *loss_out, void *grad_out, void *stream,
        int path, int split, bool softmax = false, const ce_test_hooks *hooks = nullptr) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_DTYPE;
    if (softmax) {
        if (!logits || !grad_out) return CE_ERR_NULL;
        targets = nullptr;
        loss_out = nullptr;
        grad_scale = nullptr;
        reduction = CE_REDUCE_NONE;
    }
    if (reduction != CE_REDUCE_MEAN && reduction != CE_REDUCE_SUM && reduction != CE_REDUCE_NONE)
        return CE_ERR_REDUCTION;
    if (!softmax && (!logits || !targets || !loss_out)) return CE_ERR_NULL;
    if (B < 1 || C < 1 || B > 0x7fffffffLL || C > 0x7fffffffLL) return CE_ERR_SHAPE;
    const int es = dtype == CE_F32 ? 4 : 2;
    if ((unsigned long long)B * (unsigned long long)C > (1ull << 61) / (unsigned)es)
        return CE_ERR_SHAPE;
    const uintptr_t lz = reinterpret_cast<uintptr_t>(logits);
    const uintptr_t gz = reinterpret_cast<uintptr_t>(grad_out);
    const uintptr_t tz = reinterpret_cast<uintptr_t>(targets);
    const uintptr_t oz = reinterpret_cast<uintptr_t>(loss_out);
    const uintptr_t sz = reinterpret_cast<uintptr_t>(grad_scale);
    if (lz % es || gz % es || tz % 4 || oz % 4 || sz % 4) return CE_ERR_ALIGN;
    const size_t nbytes = (size_t)B * (size_t)C * es;
    const size_t per_row = reduction == CE_REDUCE_NONE ? (size_t)B * 4 : 4;  // loss_out, grad_scale
    if (softmax) {
        if (ranges_overlap(gz, nbytes, lz, nbytes)) return CE_ERR_OVERLAP;
    } else {
        if (grad_out && (ranges_overlap(gz, nbytes, lz, nbytes) ||
                         ranges_overlap(gz, nbytes, tz, (size_t)B * 4) ||
                         ranges_overlap(gz, nbytes, oz, per_row) ||
                         (grad_scale && ranges_overlap(gz, nbytes, sz, per_row))))
            return CE_ERR_OVERLAP;
        if (ranges_overlap(oz, per_row, lz, nbytes) || ranges_overlap(oz, per_row, tz, (size_t)B * 4) ||
            (grad_scale && ranges_overlap(oz, per_row, sz, per_row)))
            return CE_ERR_OVERLAP;
    }

    float *grad_f32 = hooks ? hooks->grad_f32_out : nullptr;
    if (grad_f32) {
        const uintptr_t fz = reinterpret_cast<uintptr_t>(grad_f32);
        const size_t fbytes = (size_t)B * (size_t)C * 4;
        if (fz % 4) return CE_ERR_ALIGN;
        if (ranges_overlap(fz, fbytes, lz, nbytes) || ranges_overlap(fz, fbytes, tz, (size_t)B * 4) ||
            (grad_out && ranges_overlap(fz, fbytes, gz, nbytes)) ||
            (loss_out && ranges_overlap(fz, fbytes, oz, per_row)))
            return CE_ERR_OVERLAP;
    }

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    int rc = device_info(dev, &d);
    if (rc != CE_OK) return rc;
    for (const void *ptr : {logits, (const void *)targets, (const void *)loss_out,
                            (const void *)grad_out, (const void *)grad_scale,
                            (const void *)grad_f32}) {
        if (ptr && (rc = check_pointer(ptr, d)) != CE_OK) return rc;
    }

    Plan pl;
    if ((rc = make_plan(B, C, dtype, path, split, &pl, !softmax && !grad_out)) != CE_OK) return rc;
    const bool hooked = hooks && (hooks->skip_copy_row >= 0 || hooks->wait_limit_cycles > 0 ||
                                  hooks->grad_f32_out);
    if (hooked && (pl.path == CE_PATH_STREAM || pl.path == CE_PATH_ROWS_ONLINE))
        return CE_ERR_PATH;  // stage nothing

    const size_t rows_bytes = align_up((size_t)B, 1024) * sizeof(float);
    size_t need = kHeaderBytes + rows_bytes;
    size_t parts_off = 0, zt_off = 0;
    if (pl.path == CE_PATH_STREAM) {
        parts_off = need;
        need += align_up((size_t)B * (size_t)pl.chunks * sizeof(float2), 256);
        zt_off = need;
        need += align_up((size_t)B * sizeof(float), 256);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Workspace ws;
    if ((rc = get_workspace(dev, s, need, &ws)) != CE_OK) return rc;

    ParamsEx p;
    p.logits = static_cast<const unsigned char *>(logits);
    p.targets = targets;
    p.grad = static_cast<unsigned char *>(grad_out);
    p.loss_out = loss_out;
    p.ticket = reinterpret_cast<unsigned int *>(ws.base);
    p.err = reinterpret_cast<int *>(ws.base + 4);
    // per-row losses as the output: written where the caller wants them
    p.loss_rows = reduction == CE_REDUCE_NONE ? loss_out
                                              : reinterpret_cast<float *>(ws.base + kHeaderBytes);
    p.parts = pl.path == CE_PATH_STREAM ? reinterpret_cast<float2 *>(ws.base + parts_off) : nullptr;
    p.zt = pl.path == CE_PATH_STREAM ? reinterpret_cast<float *>(ws.base + zt_off) : nullptr;
    p.B = B;
    p.C = C;
    p.inv_b = (float)(1.0 / (double)B);
    p.lo_clip = (uint64_t)((lz + 15) & ~(uintptr_t)15);
    p.hi_clip = (uint64_t)((lz + nbytes) & ~(uintptr_t)15);
    if (p.hi_clip < p.lo_clip) p.hi_clip = p.lo_clip;
    p.grad_vec_ok = grad_out != nullptr && ((gz - lz) % 16) == 0;
    p.reduction = reduction;
    p.grad_base = reduction == CE_REDUCE_MEAN ? p.inv_b : 1.f;
    p.grad_scale = grad_scale;
    p.scale_per_row = grad_scale != nullptr && reduction == CE_REDUCE_NONE;
    p.softmax = softmax ? 1 : 0;
    if (hooks) {
        if (hooks->wait_limit_cycles > 0) p.copy_wait_limit = hooks->wait_limit_cycles;
        p.skip_copy_row = hooks->skip_copy_row >= 0 ? hooks->skip_copy_row : -1;
        p.grad_f32 = grad_f32;
    }

    if ((e = launch_plan(p, dtype, pl, s)) != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return CE_OK;
}

// ------------------------------------------------- allocation-free entry point
//
// ce_fwd_bwd_noalloc keeps its scratch (the CTA ticket, the error counters
// and one fp32 loss per row) in a statically sized device array of this
// file instead of a cudaMalloc'd per-stream workspace.  Every device that
// loads the library holds the array until the process exits.

constexpr long long kNoAllocMaxRows = 262144;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + (size_t)kNoAllocMaxRows * sizeof(float);

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
std::map<int, unsigned char *> g_noalloc_base;  // device -> address of g_noalloc_scratch

// The device address of the static scratch on device `dev` (which must be
// current), looked up once per device.  In host code the array's name is only
// a stand-in, so the address has to come from cudaGetSymbolAddress.
int noalloc_scratch(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    auto it = g_noalloc_base.find(dev);
    if (it != g_noalloc_base.end()) {
        *out = it->second;
        return CE_OK;
    }
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_noalloc_base[dev] = static_cast<unsigned char *>(ptr);
    *out = static_cast<unsigned char *>(ptr);
    return CE_OK;
}

int run_noalloc(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                float *loss_out, void *grad_out, void *stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_DTYPE;
    if (!logits || !targets || !loss_out || !grad_out) return CE_ERR_NULL;
    if (B < 1 || C < 1 || B > 0x7fffffffLL || C > 0x7fffffffLL) return CE_ERR_SHAPE;
    if (B > kNoAllocMaxRows) return CE_ERR_SCRATCH;
    const int es = dtype == CE_F32 ? 4 : 2;
    if ((unsigned long long)B * (unsigned long long)C > (1ull << 61) / (unsigned)es)
        return CE_ERR_SHAPE;
    const uintptr_t lz = reinterpret_cast<uintptr_t>(logits);
    const uintptr_t gz = reinterpret_cast<uintptr_t>(grad_out);
    const uintptr_t tz = reinterpret_cast<uintptr_t>(targets);
    const uintptr_t oz = reinterpret_cast<uintptr_t>(loss_out);
    if (lz % es || gz % es || tz % 4 || oz % 4) return CE_ERR_ALIGN;
    const size_t nbytes = (size_t)B * (size_t)C * es;
    if (ranges_overlap(gz, nbytes, lz, nbytes) || ranges_overlap(gz, nbytes, tz, (size_t)B * 4) ||
        ranges_overlap(gz, nbytes, oz, 4) || ranges_overlap(oz, 4, lz, nbytes) ||
        ranges_overlap(oz, 4, tz, (size_t)B * 4))
        return CE_ERR_OVERLAP;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    int rc = device_info(dev, &d);
    if (rc != CE_OK) return rc;
    for (const void *ptr : {logits, (const void *)targets, (const void *)loss_out,
                            (const void *)grad_out}) {
        if ((rc = check_pointer(ptr, d)) != CE_OK) return rc;
    }
    // Every plan the planner makes for itself (warp, split at K = 1, two-pass)
    // needs no scratch beyond the ticket, the counters and the row losses.
    Plan pl;
    if ((rc = make_plan(B, C, dtype, CE_PATH_AUTO, 0, &pl)) != CE_OK) return rc;

    unsigned char *base = nullptr;
    if ((rc = noalloc_scratch(dev, &base)) != CE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the last call's contents: the ticket and the error
    // counters must start at zero, the row losses are all rewritten.
    if ((e = cudaMemsetAsync(base, 0, kHeaderBytes, s)) != cudaSuccess) return cuda_fail(e);

    ParamsEx p;
    p.logits = static_cast<const unsigned char *>(logits);
    p.targets = targets;
    p.grad = static_cast<unsigned char *>(grad_out);
    p.loss_out = loss_out;
    p.ticket = reinterpret_cast<unsigned int *>(base);
    p.err = reinterpret_cast<int *>(base + 4);
    p.loss_rows = reinterpret_cast<float *>(base + kHeaderBytes);
    p.parts = nullptr;
    p.zt = nullptr;
    p.B = B;
    p.C = C;
    p.inv_b = (float)(1.0 / (double)B);
    p.lo_clip = (uint64_t)((lz + 15) & ~(uintptr_t)15);
    p.hi_clip = (uint64_t)((lz + nbytes) & ~(uintptr_t)15);
    if (p.hi_clip < p.lo_clip) p.hi_clip = p.lo_clip;
    p.grad_vec_ok = ((gz - lz) % 16) == 0;
    p.reduction = CE_REDUCE_MEAN;
    p.grad_base = p.inv_b;
    p.grad_scale = nullptr;
    p.scale_per_row = 0;
    p.softmax = 0;

    e = launch_plan(p, dtype, pl, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return CE_OK;
}

}  // namespace

namespace ce {

cudaError_t ensure_smem_attr(const void *func, int smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    int &have = done[{dev, func}];
    if (have >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) have = smem;
    return e;
}

}  // namespace ce

namespace {

int run_softmax_bwd(const void *probs, const void *dy, int64_t B, int64_t C, int dtype,
                    void *dx_out, void *stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_DTYPE;
    if (!probs || !dy || !dx_out) return CE_ERR_NULL;
    if (B < 1 || C < 1 || B > 0x7fffffffLL || C > 0x7fffffffLL) return CE_ERR_SHAPE;
    const int es = dtype == CE_F32 ? 4 : 2;
    if ((unsigned long long)B * (unsigned long long)C > (1ull << 61) / (unsigned)es)
        return CE_ERR_SHAPE;
    const uintptr_t pz = reinterpret_cast<uintptr_t>(probs);
    const uintptr_t dz = reinterpret_cast<uintptr_t>(dy);
    const uintptr_t xz = reinterpret_cast<uintptr_t>(dx_out);
    if (pz % es || dz % es || xz % es) return CE_ERR_ALIGN;
    const size_t nbytes = (size_t)B * (size_t)C * es;
    // dx may not overlap p or dy unless it is one of them exactly (each element
    // is read by the thread that then writes it, after the row's dot product)
    if ((xz != pz && ranges_overlap(xz, nbytes, pz, nbytes)) ||
        (xz != dz && ranges_overlap(xz, nbytes, dz, nbytes)))
        return CE_ERR_OVERLAP;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    int rc = device_info(dev, &d);
    if (rc != CE_OK) return rc;
    for (const void *ptr : {probs, dy, (const void *)dx_out})
        if ((rc = check_pointer(ptr, d)) != CE_OK) return rc;
    const bool vec = ce::softmax_bwd_vec_ok(C, es, pz, dz, xz);
    e = ce::launch_softmax_bwd(probs, dy, dx_out, B, C, dtype, vec, d.sms,
                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return CE_OK;
}

// ------------------------------------------------------ host-buffer entry
//
// ce_fwd_bwd_host and ce_fwd_bwd_host_grad: the batch goes through in chunks
// of rows.  A chunk's logits are copied in on one helper stream, its kernel
// runs on the caller's stream, and (for ce_fwd_bwd_host_grad) its gradient is
// copied out on the other helper stream, so the copies of one chunk overlap
// the kernels and copies of its neighbours; a copy engine moves ~210 GB/s
// each way from page-locked memory on GB300, ~340 GB/s both ways at once.
// Each chunk's kernel writes its rows' losses; one last launch sums them in
// the fixed order of the fused kernels, so the loss has the bits of
// ce_fwd_bwd.  A chunk holds a multiple of 16 rows, so every row keeps the
// alignment it has in a 16-byte aligned tensor, and with it the gradient's
// bits.

// Logits bytes per chunk, at most.  Measured on GB300 (16384 x 50257 fp32,
// gradient to the host): 64 MiB chunks keep the copies in and out running at
// once (20 ms, ~330 GB/s both ways); 128 and 256 MiB chunks ran the two
// directions one after the other (31-33 ms); 32 MiB chunks leave the host
// issuing more calls than the copies take.
constexpr size_t kHostChunkBytes = 64u << 20;
constexpr size_t kHostChunkMin = 4u << 20;

// Tuning knob: CE_HOST_CHUNK_MB sets the chunk's logits bytes (MiB).  Read once.
size_t host_chunk_bytes() {
    static const size_t b = [] {
        const char *e = getenv("CE_HOST_CHUNK_MB");
        const long v = e ? atol(e) : 0;
        return v > 0 ? (size_t)v << 20 : kHostChunkBytes;
    }();
    return b;
}

int host_pipe(int dev, cudaStream_t s, size_t chunk_bytes, bool grad_host, size_t tbytes,
              HostPipe **out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    HostPipe &h = g_hs[{dev, reinterpret_cast<uintptr_t>(s)}];
    cudaError_t e;
    if (!h.s_in) {
        if ((e = cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e);
        cudaEvent_t *evs[] = {&h.ev_start, &h.ev_end, &h.ev_in[0], &h.ev_in[1],
                              &h.ev_k[0],  &h.ev_k[1], &h.ev_out[0], &h.ev_out[1]};
        for (cudaEvent_t *ev : evs)
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
    }
    // A new buffer for *b; the outgrown one may still be read by queued work,
    // so it is retired, not freed.
    auto replace = [&](unsigned char **b, size_t bytes) -> int {
        if (*b) g_ws_retired.push_back({dev, *b});
        *b = nullptr;
        void *p = nullptr;
        cudaError_t err = cudaMalloc(&p, bytes);
        if (err != cudaSuccess) return cuda_fail(err);
        *b = static_cast<unsigned char *>(p);
        return CE_OK;
    };
    int rc;
    if (h.chunk_bytes < chunk_bytes) {
        const size_t bytes = align_up(chunk_bytes, 1 << 20);
        for (int b = 0; b < 2; ++b)
            if ((rc = replace(&h.z[b], bytes)) != CE_OK) return rc;
        h.chunk_bytes = bytes;
    }
    if (grad_host && h.g_bytes < h.chunk_bytes) {
        for (int b = 0; b < 2; ++b)
            if ((rc = replace(&h.g[b], h.chunk_bytes)) != CE_OK) return rc;
        h.g_bytes = h.chunk_bytes;
    }
    if (h.tbytes < tbytes) {
        const size_t bytes = align_up(tbytes, 1 << 16);
        if ((rc = replace(&h.t, bytes)) != CE_OK) return rc;
        h.tbytes = bytes;
    }
    *out = &h;  // map nodes are stable; entries are erased only by ce_release_workspaces
    return CE_OK;
}

// grad_dev: device gradient (ce_fwd_bwd_host); grad_host: host gradient
// (ce_fwd_bwd_host_grad).  Exactly one is set.
int run_host(const void *logits_host, const int32_t *targets_host, int64_t B, int64_t C,
             int dtype, float *loss_host, void *grad_dev, void *grad_host, void *stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_DTYPE;
    if (!logits_host || !targets_host || !loss_host || !(grad_dev || grad_host))
        return CE_ERR_NULL;
    if (B < 1 || C < 1 || B > 0x7fffffffLL || C > 0x7fffffffLL) return CE_ERR_SHAPE;
    const int es = dtype == CE_F32 ? 4 : 2;
    if ((unsigned long long)B * (unsigned long long)C > (1ull << 61) / (unsigned)es)
        return CE_ERR_SHAPE;
    const uintptr_t lz = reinterpret_cast<uintptr_t>(logits_host);
    const uintptr_t gz = reinterpret_cast<uintptr_t>(grad_dev ? grad_dev : grad_host);
    const uintptr_t tz = reinterpret_cast<uintptr_t>(targets_host);
    const uintptr_t oz = reinterpret_cast<uintptr_t>(loss_host);
    if (lz % es || gz % es || tz % 4 || oz % 4) return CE_ERR_ALIGN;
    const size_t nbytes = (size_t)B * (size_t)C * es;
    if (ranges_overlap(gz, nbytes, lz, nbytes)) return CE_ERR_OVERLAP;
    if (grad_host && (ranges_overlap(gz, nbytes, tz, (size_t)B * 4) ||
                      ranges_overlap(gz, nbytes, oz, 4) || ranges_overlap(oz, 4, lz, nbytes) ||
                      ranges_overlap(oz, 4, tz, (size_t)B * 4)))
        return CE_ERR_OVERLAP;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    int rc = device_info(dev, &d);
    if (rc != CE_OK) return rc;
    if (grad_dev && (rc = check_pointer(grad_dev, d)) != CE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return cuda_fail(e);
    if (cs != cudaStreamCaptureStatusNone) return CE_ERR_CAPTURE;

    // chunks: a multiple of 16 rows, at most kHostChunkBytes of logits and
    // (so that a small batch's copies overlap too) about a quarter of the
    // batch when that is at least kHostChunkMin; at least 16 rows
    const size_t row_bytes = (size_t)C * es;
    size_t want = nbytes / 4 > kHostChunkMin ? nbytes / 4 : kHostChunkMin;
    if (want > host_chunk_bytes()) want = host_chunk_bytes();
    long long chunk_rows = (long long)(want / row_bytes) / 16 * 16;
    if (chunk_rows < 16) chunk_rows = 16;
    if (chunk_rows > B) chunk_rows = B;
    Plan pl;
    if ((rc = make_plan(chunk_rows, C, dtype, CE_PATH_AUTO, 0, &pl)) != CE_OK) return rc;
    if (pl.path == CE_PATH_STREAM) return CE_ERR_PATH;  // never planned (needs partials per chunk)
    Workspace ws;
    if ((rc = get_workspace(dev, s, kHeaderBytes + align_up((size_t)B, 1024) * sizeof(float),
                            &ws)) != CE_OK)
        return rc;
    HostPipe *h = nullptr;
    if ((rc = host_pipe(dev, s, (size_t)chunk_rows * row_bytes, grad_host != nullptr,
                        (size_t)B * 4, &h)) != CE_OK)
        return rc;

    float *rows = reinterpret_cast<float *>(ws.base + kHeaderBytes);
    float *dloss = reinterpret_cast<float *>(ws.base + kLossSlot);
    const float inv_b = (float)(1.0 / (double)B);
    auto fail = [&](cudaError_t err) { return cuda_fail(err); };
    if ((e = cudaEventRecord(h->ev_start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h->s_in, h->ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h->s_out, h->ev_start, 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h->t, targets_host, (size_t)B * 4, cudaMemcpyDefault, h->s_in)) !=
            cudaSuccess)
        return fail(e);
    const long long nchunks = (B + chunk_rows - 1) / chunk_rows;
    for (long long i = 0; i < nchunks; ++i) {
        const int b = (int)(i & 1);
        const long long r0 = i * chunk_rows;
        const long long nr = r0 + chunk_rows <= B ? chunk_rows : B - r0;
        const size_t off = (size_t)r0 * row_bytes, cb = (size_t)nr * row_bytes;
        // copy in once the kernel two chunks back has read this buffer
        if ((i >= 2 && (e = cudaStreamWaitEvent(h->s_in, h->ev_k[b], 0)) != cudaSuccess) ||
            (e = cudaMemcpyAsync(h->z[b], static_cast<const unsigned char *>(logits_host) + off,
                                 cb, cudaMemcpyDefault, h->s_in)) != cudaSuccess ||
            (e = cudaEventRecord(h->ev_in[b], h->s_in)) != cudaSuccess)
            return fail(e);
        // the chunk's kernel, once its logits are in and (gradient to the
        // host) the copy out two chunks back has read its gradient buffer
        if ((e = cudaStreamWaitEvent(s, h->ev_in[b], 0)) != cudaSuccess ||
            (grad_host && i >= 2 && (e = cudaStreamWaitEvent(s, h->ev_out[b], 0)) != cudaSuccess))
            return fail(e);
        unsigned char *gdst = grad_host ? h->g[b] : static_cast<unsigned char *>(grad_dev) + off;
        const uintptr_t zz = reinterpret_cast<uintptr_t>(h->z[b]);
        ce::ParamsEx p;
        p.logits = h->z[b];
        p.targets = reinterpret_cast<const int32_t *>(h->t) + r0;
        p.grad = gdst;
        p.loss_out = rows + r0;
        p.loss_rows = rows + r0;  // the chunk's row losses, summed at the end
        p.ticket = reinterpret_cast<unsigned int *>(ws.base);
        p.err = reinterpret_cast<int *>(ws.base + 4);
        p.parts = nullptr;
        p.zt = nullptr;
        p.B = nr;
        p.C = C;
        p.inv_b = inv_b;
        p.lo_clip = (uint64_t)((zz + 15) & ~(uintptr_t)15);
        p.hi_clip = (uint64_t)((zz + cb) & ~(uintptr_t)15);
        if (p.hi_clip < p.lo_clip) p.hi_clip = p.lo_clip;
        p.grad_vec_ok = ((reinterpret_cast<uintptr_t>(gdst) - zz) % 16) == 0;
        p.reduction = CE_REDUCE_NONE;
        p.grad_base = inv_b;  // the gradient of the mean over all B rows
        p.grad_scale = nullptr;
        p.scale_per_row = 0;
        p.softmax = 0;
        Plan cp = pl;
        if (nr != chunk_rows && (rc = make_plan(nr, C, dtype, CE_PATH_AUTO, 0, &cp)) != CE_OK)
            return rc;
        if ((e = launch_plan(p, dtype, cp, s)) != cudaSuccess ||
            (e = cudaEventRecord(h->ev_k[b], s)) != cudaSuccess)
            return fail(e);
        if (grad_host &&
            ((e = cudaStreamWaitEvent(h->s_out, h->ev_k[b], 0)) != cudaSuccess ||
             (e = cudaMemcpyAsync(static_cast<unsigned char *>(grad_host) + off, h->g[b], cb,
                                  cudaMemcpyDefault, h->s_out)) != cudaSuccess ||
             (e = cudaEventRecord(h->ev_out[b], h->s_out)) != cudaSuccess))
            return fail(e);
    }
    // the batch loss over all rows, in the fused kernels' order, and its copy
    // back; the call ends on `stream` once the last gradient chunk is out
    ce::Params tp;
    tp.loss_rows = rows;
    tp.loss_out = dloss;
    tp.ticket = reinterpret_cast<unsigned int *>(ws.base);
    tp.B = B;
    tp.inv_b = inv_b;
    if ((e = ce::launch_batch_loss(tp, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(loss_host, dloss, sizeof(float), cudaMemcpyDefault, s)) !=
            cudaSuccess ||
        (e = cudaEventRecord(h->ev_end, h->s_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, h->ev_end, 0)) != cudaSuccess)
        return fail(e);
    e = cudaGetLastError();
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int ce_softmax_fwd(const void *logits, int64_t B, int64_t C, int dtype, void *probs_out,
                   void *stream) {
    return run(logits, nullptr, B, C, dtype, CE_REDUCE_NONE, nullptr, nullptr, probs_out, stream,
               CE_PATH_AUTO, 0, true);
}

int ce_softmax_fwd_path(const void *logits, int64_t B, int64_t C, int dtype, void *probs_out,
                        void *stream, int path, int split) {
    return run(logits, nullptr, B, C, dtype, CE_REDUCE_NONE, nullptr, nullptr, probs_out, stream,
               path, split, true);
}

int ce_fwd_bwd_host(const void *logits_host, const int32_t *targets_host, int64_t B, int64_t C,
                    int dtype, float *loss_host, void *grad_out, void *stream) {
    if (!grad_out) return CE_ERR_NULL;
    return run_host(logits_host, targets_host, B, C, dtype, loss_host, grad_out, nullptr, stream);
}

int ce_fwd_bwd_host_grad(const void *logits_host, const int32_t *targets_host, int64_t B,
                         int64_t C, int dtype, float *loss_host, void *grad_host, void *stream) {
    if (!grad_host) return CE_ERR_NULL;
    return run_host(logits_host, targets_host, B, C, dtype, loss_host, nullptr, grad_host, stream);
}

int ce_softmax_bwd(const void *probs, const void *dy, int64_t B, int64_t C, int dtype,
                   void *dx_out, void *stream) {
    return run_softmax_bwd(probs, dy, B, C, dtype, dx_out, stream);
}

int ce_fwd_bwd(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
               float *loss_out, void *grad_out, void *stream) {
    if (!grad_out) return CE_ERR_NULL;
    return run(logits, targets, B, C, dtype, CE_REDUCE_MEAN, nullptr, loss_out, grad_out, stream,
               CE_PATH_AUTO, 0);
}

int ce_fwd_bwd_path(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                    float *loss_out, void *grad_out, void *stream, int path, int split) {
    if (!grad_out) return CE_ERR_NULL;
    return run(logits, targets, B, C, dtype, CE_REDUCE_MEAN, nullptr, loss_out, grad_out, stream,
               path, split);
}

int ce_fwd_bwd_ex(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                  int reduction, const float *grad_scale, float *loss_out, void *grad_out,
                  void *stream) {
    return run(logits, targets, B, C, dtype, reduction, grad_scale, loss_out, grad_out, stream,
               CE_PATH_AUTO, 0);
}

int ce_fwd_bwd_ex_path(const void *logits, const int32_t *targets, int64_t B, int64_t C,
                       int dtype, int reduction, const float *grad_scale, float *loss_out,
                       void *grad_out, void *stream, int path, int split) {
    return run(logits, targets, B, C, dtype, reduction, grad_scale, loss_out, grad_out, stream,
               path, split);
}

int ce_forward(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
               int reduction, float *loss_out, void *stream) {
    return run(logits, targets, B, C, dtype, reduction, nullptr, loss_out, nullptr, stream,
               CE_PATH_AUTO, 0);
}

int ce_fwd_bwd_test(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                    float *loss_out, void *grad_out, void *stream, int path, int split,
                    const ce_test_hooks *hooks) {
    if (!grad_out) return CE_ERR_NULL;
    return run(logits, targets, B, C, dtype, CE_REDUCE_MEAN, nullptr, loss_out, grad_out, stream,
               path, split, false, hooks);
}

int ce_query_plan(int64_t B, int64_t C, int dtype, int *path, int *split, int *ctas,
                  int *threads, int *smem_bytes, int *launches) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_DTYPE;
    if (B < 1 || C < 1 || B > 0x7fffffffLL || C > 0x7fffffffLL) return CE_ERR_SHAPE;
    Plan pl;
    int rc = make_plan(B, C, dtype, CE_PATH_AUTO, 0, &pl);
    if (rc != CE_OK) return rc;
    if (path) *path = pl.path;
    if (split) *split = pl.split;
    if (ctas) *ctas = pl.ctas;
    if (threads) *threads = pl.threads;
    if (smem_bytes) *smem_bytes = pl.smem;
    if (launches) *launches = pl.launches;
    return CE_OK;
}

int ce_get_device_errors(void *stream, int32_t *bad_targets, int32_t *timeouts) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find({dev, reinterpret_cast<uintptr_t>(s)});
        if (it != g_ws.end()) base = it->second.base;
    }
    int32_t h[2] = {0, 0};
    if (base) {
        if ((e = cudaMemcpyAsync(h, base + 4, sizeof h, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaMemsetAsync(base + 4, 0, sizeof h, s)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    }
    if (bad_targets) *bad_targets = h[0];
    if (timeouts) *timeouts = h[1];
    return CE_OK;
}

int ce_release_workspaces(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int rc = CE_OK;
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &kv : g_ws) {
        if (!kv.second.base) continue;
        cudaSetDevice(kv.first.first);
        cudaError_t e = cudaFree(kv.second.base);
        if (e != cudaSuccess) rc = cuda_fail(e);
    }
    for (auto &kv : g_hs) {
        HostPipe &h = kv.second;
        cudaSetDevice(kv.first.first);
        for (void *b : {(void *)h.z[0], (void *)h.z[1], (void *)h.g[0], (void *)h.g[1],
                        (void *)h.t})
            if (b) {
                cudaError_t e = cudaFree(b);
                if (e != cudaSuccess) rc = cuda_fail(e);
            }
        for (cudaStream_t st : {h.s_in, h.s_out})
            if (st) cudaStreamDestroy(st);
        for (cudaEvent_t ev : {h.ev_start, h.ev_end, h.ev_in[0], h.ev_in[1], h.ev_k[0], h.ev_k[1],
                               h.ev_out[0], h.ev_out[1]})
            if (ev) cudaEventDestroy(ev);
    }
    for (auto &r : g_ws_retired) {
        cudaSetDevice(r.first);
        cudaError_t e = cudaFree(r.second);
        if (e != cudaSuccess) rc = cuda_fail(e);
    }
    g_ws.clear();
    g_hs.clear();
    g_ws_retired.clear();
    cudaSetDevice(cur);
    return rc;
}

const char *ce_status_string(int status) {
    switch (status) {
        case CE_OK: return "ok";
        case CE_ERR_NULL: return "a required pointer is NULL";
        case CE_ERR_SHAPE: return "invalid shape (B and C must be in [1, 2^31-1])";
        case CE_ERR_DTYPE: return "unknown dtype";
        case CE_ERR_ALIGN: return "pointer not aligned to its element size";
        case CE_ERR_CUDA: return "CUDA runtime error";
        case CE_ERR_OVERLAP: return "an output overlaps an input or the other output";
        case CE_ERR_POINTER: return "pointer not accessible from the current device";
        case CE_ERR_CAPTURE: return "workspace must grow while the stream is being captured";
        case CE_ERR_PATH: return "the forced path cannot run this shape";
        case CE_ERR_SCRATCH:
            return "more rows than the static scratch of ce_fwd_bwd_noalloc holds (B <= 262144)";
        case CE_ERR_REDUCTION: return "reduction is not a ce_reduction";
        default: return "unknown status";
    }
}

const char *ce_last_cuda_error(void) { return g_cuda_error; }

int ce_fwd_bwd_noalloc(const void *logits, const int32_t *targets, int64_t B, int64_t C,
                       int dtype, float *loss_out, void *grad_out, void *stream) {
    return run_noalloc(logits, targets, B, C, dtype, loss_out, grad_out, stream);
}

}  // extern "C"
