// Launchers shared between the library's translation units (host side).
#pragma once
#include "common.cuh"

namespace lora {

// Shrink output layout: s_parts float32 arrays [n, r_max] (original token order); the shrink
// value of token t is scale_s * x[t] A_s^T = sum over parts p of s[p][t][:].  Rows of
// base-only tokens are not written.

// CUDA-core shrink.  Small batches of 16-bit data: one CTA per (sorted token, 8 adapter rows,
// 1024 input features), *s_parts = ceil(h_in / 1024).  tiled: one CTA per (segment, 64 tokens)
// through shared memory, *s_parts = 1.  float32: one warp per (token, rows), *s_parts = 1.
// xready: nonzero for the small-batch kernels ahead of a fused decode GEMM launched with the
// same value (GroupView::xready).
int launch_shrink(const PoolView& pv, const SegView& sv, const void* x, float* s_out, cudaStream_t st, bool tiled,
                  int* s_parts, int xready = 0);
int shrink_parts(const PoolView& pv, int n, bool tiled);
// Whether the small-batch shrink of 16-bit data takes the segmented kernel (A rows read once per
// work item) rather than the per-token one.
int shrink_segmented(const PoolView& pv, int n);
// The same for the slices of a group (16-bit data, not tiled): slice q's output starts at
// s_out + q * grp.s_stride.  One launch covers every slice.
int launch_shrink_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                        cudaStream_t st, bool tiled, int* s_parts);

// Whether the fused tensor-core decode GEMM (n <= 256) holds every adapter's B rows a CTA can
// need in shared memory during its main loop (the variant policy keys on this).
int decode_fused_fits(const PoolView& pv, int n);

// y[t, :] += s[t, :] B_s^T (separate variant's residual kernel).
int launch_expand(const PoolView& pv, const SegView& sv, const float* s_in, int s_parts, void* y, cudaStream_t st);
// The same for the slices of a group (16-bit data): y has row stride grp.ldy, slice q owns
// columns [grp.col[q], grp.col[q + 1]).  One launch covers every slice.
int launch_expand_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const float* s_in, int s_parts,
                        void* y, cudaStream_t st);

// CUDA-core base GEMM y = x W^T (+ fused expand when fuse).
int launch_gemm_simt(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in,
                     int s_parts, void* y, bool fuse, cudaStream_t st);

// Tensor-core (tcgen05) base GEMM with optional fused expand.
//   decode path  (n <= 256): W tiles on the MMA M side, tokens on N, split-K across the CTAs
//                 of a thread-block cluster, reduced through distributed shared memory.
//   prefill path (n > 256):  token tiles on M (128), outputs on N (256), persistent CTAs.
int tc_supported(const PoolView& pv, int n);
// prefetch/prefetch_bytes: optional device range the decode kernel streams into L2 after its
// own loads (ignored by the prefill kernel).
// grp: output slices of a group (nullptr: the single linear of pv).  pv.h_out is then the
// concatenated width; y has row stride grp->ldy.  The prefill kernel applies every slice's
// LoRA term; the decode kernel takes one slice with fuse, or several without the LoRA term
// (a single slice may also be a column range of a wider y: pv.h_out < grp->ldy).
// xready: nonzero when the shrink kernel just before this fused decode GEMM was launched with
// the same value: the GEMM then streams its weight from its start and reads x once the shrink
// has published the value.
int launch_gemm_tc(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in, int s_parts,
                   void* y, bool fuse, cudaStream_t st, const void* prefetch = nullptr, size_t prefetch_bytes = 0,
                   const GroupView* grp = nullptr, int xready = 0);

// The launch sequence of one LoRA-augmented linear (lora_linear_fwd and its variants), after the
// caller's arguments were checked; s_buf receives the shrink output.
int linear_fwd_impl(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev, const lora_segments* seg,
                    int variant, float* s_buf, const void* prefetch_dev, size_t prefetch_bytes, cudaStream_t st);

// Base GEMM y = x W^T (no LoRA term) with 256 W rows per CTA, two M=128 MMAs sharing each x
// tile, full K per CTA (batches of up to 256 tokens); y has row stride ldy.
int launch_gemm_tall(const PoolView& pv, const SegView& sv, const void* W, const void* x, void* y, int ldy,
                     cudaStream_t st);

// Grouped tcgen05 shrink for batches of more than 256 tokens (one CTA per 128-token tile).
int shrink_tc_supported(const PoolView& pv);
int launch_shrink_tc(const PoolView& pv, const SegView& sv, const void* x, float* s_out, cudaStream_t st);
// The same for the slices of a group in one launch (count * r_max <= 256): slice q's output
// starts at s_out + q * grp.s_stride.
int shrink_tc_group_supported(const PoolView& pv, int count);
int launch_shrink_tc_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                           cudaStream_t st);

int num_sms();

}  // namespace lora
