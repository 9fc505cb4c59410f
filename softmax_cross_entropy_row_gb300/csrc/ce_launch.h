// Host-side interface between the C-ABI layer (ce_api.cu) and the kernel
// translation units.  Internal to the library.
#pragma once

#include <cuda_runtime.h>

#include "ce_device.cuh"

namespace ce {

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, kernel)
// and size: later launches (including ones made during stream capture) skip it.
cudaError_t ensure_smem_attr(const void *func, int smem);

// Threads per CTA of each path.
constexpr int kSplitThreads = 512;
constexpr int kSplitMaxVecs = 16;  // 16-byte vectors per thread: slices of at most 128 KB
constexpr int kWarpKernelWarps = 16;
// The warp path's build for three resident CTAs per SM has 9 warps each (27
// per SM), so a batch of up to 27 rows per SM spreads evenly over the SMs.
constexpr int kWarpKernelWarps3 = 9;
__host__ __device__ constexpr int warp_kernel_warps(int per_sm) {
    return per_sm >= 3 ? kWarpKernelWarps3 : kWarpKernelWarps;
}
constexpr int kStreamThreads = 256;
constexpr int kStreamPerThread = 16;  // elements each thread keeps in registers
constexpr int kStreamChunk = kStreamThreads * kStreamPerThread;

// Upper bounds of the shared-memory ring sizes (slots of staged rows).
constexpr int kMaxSplitSlots = 8;
constexpr int kMaxWarpSlots = 4;  // per warp

// Split-row path: one row (K = 1) or one slice of a row per CTA of a cluster
// of K CTAs; `nslots` staged slices of `slot_bytes` each per CTA.
// K CTAs per row (1, 2, 3, 4, 6 or 8), each holding a slice of at most
// nt * vecs 16-byte vectors (vecs = 8, 12 or 16) in registers; nt threads per
// CTA: kSplitThreads, or at K = 1 also 128 (narrower CTAs, several per SM).  `staged` = 1: gradients of whole vectors go out through the row's own
// slot by one TMA bulk store (needs grad and logits equally aligned mod 16).
cudaError_t launch_split(const ParamsEx &p, int dtype, int K, int nt, int vecs, int ctas,
                         int nslots, int slot_bytes, long long slice_elems, int smem, int staged,
                         cudaStream_t s);
// Largest number of co-resident clusters of K CTAs of nt threads with `smem`
// dynamic bytes.
cudaError_t split_max_clusters(int dtype, int K, int nt, int vecs, int smem, int *clusters);

// The pipelined split-row kernel (ce_row_pipe.cu): K = 2..8 CTAs per row,
// slices of at most kSplitThreads * kPipeVecs vectors, no CTA-wide barrier per
// row; the partials of one row are exchanged while the next row is reduced.
constexpr int kPipeVecs = 8;
cudaError_t launch_split_pipe(const ParamsEx &p, int dtype, int K, int ctas, int nslots,
                              int slot_bytes, long long slice_elems, int smem, cudaStream_t s);
cudaError_t split_pipe_max_clusters(int dtype, int K, int smem, int *clusters);

// Warp-per-row path: tiles of `rows_per_tile` consecutive rows, `slots` tiles
// staged per warp; `per_sm` (1, 2 or 3) selects the build made for that many
// resident CTAs per SM (16 warps each for 1 and 2, 9 for 3).
cudaError_t launch_rows_warp(const ParamsEx &p, int dtype, int per_sm, int ctas, int slots,
                             int rows_per_tile, int slot_bytes, int smem, cudaStream_t s);
cudaError_t rows_warp_max_ctas_per_sm(int dtype, int per_sm, long long C, int smem, int *ctas);
// The same kernel for rows longer than a warp's registers hold: each row is
// swept in its shared-memory slot (max, sum, gradient) kWarpChunkVecs vectors
// per lane at a time; nw (16, 8 or 4) warps per CTA, one CTA per SM, one row
// per tile.
constexpr int kWarpChunkVecs = 8;
constexpr long long kWarpChunkRowMax = 49152;  // bytes
cudaError_t launch_rows_warp_swept(const ParamsEx &p, int dtype, int nw, int ctas, int slots,
                                   int slot_bytes, int smem, cudaStream_t s);
cudaError_t rows_warp_swept_max_ctas_per_sm(int dtype, int nw, int smem, int *ctas);

// Two-pass row path (ce_row_twopass.cu): one CTA per SM, a row at a time,
// rows of any length streamed twice through a ring of `nslots` chunks of
// kTwoPassChunkBytes (the second pass served by L2); kTwoPassConsumerWarps
// consumer warps and one producer warp.  `hint` = 1: L2 eviction hints on the
// copies (keep for the first pass, drop first for the second).
constexpr int kTwoPassConsumerWarps = 16;
constexpr int kTwoPassVecs = 4;  // 16-byte vectors per consumer thread per chunk
constexpr int kTwoPassChunkBytes = kTwoPassConsumerWarps * 32 * kTwoPassVecs * 16;
constexpr int kTwoPassThreads = (kTwoPassConsumerWarps + 1) * 32;
constexpr int kTwoPassMaxSlots = 16;
cudaError_t launch_twopass(const ParamsEx &p, int dtype, int ctas, int nslots, int smem, int hint,
                           cudaStream_t s);
cudaError_t twopass_max_ctas_per_sm(int dtype, int smem, int *ctas);

// The batch loss (mean or sum, as p's reduction says) of p.B row losses at
// p.loss_rows written by earlier launches, in the fused kernels' fixed order:
// one CTA of kTailThreads threads (ce_batch_loss.cu).
cudaError_t launch_batch_loss(const Params &p, cudaStream_t s);

// Streaming path: pass A (chunk partials) and pass B (combine, gradient, loss).
cudaError_t launch_stream(const ParamsEx &p, int dtype, long long chunks, cudaStream_t s);

// Row softmax backward (ce_softmax_bwd.cu): dx = p * (dy - sum p dy) per row.
// The vector kernel needs rows of at most 64 KB whose starts are 16-byte
// aligned in all three tensors (softmax_bwd_vec_ok); the other reads p and dy
// twice.
bool softmax_bwd_vec_ok(long long C, int es, uintptr_t p, uintptr_t dy, uintptr_t dx);
cudaError_t launch_softmax_bwd(const void *p, const void *dy, void *dx, long long B, long long C,
                               int dtype, bool vec, int sms, cudaStream_t s);

}  // namespace ce
