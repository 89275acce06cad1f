// Internal definitions shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/lora.h"

// Host handle of one pool (opaque to callers of the C ABI).
struct lora_pool {
    lora_pool_desc desc;
    char* base;
    size_t bytes;
    void* table;  // lora::SlotEntry[n_slots]
    void* A;
    void* B;
    std::vector<uint8_t> mounted;  // host mirror of the slot states this handle enqueued
    std::vector<int> ranks;        // true rank of each mounted slot (host mirror)
    int device = -1;               // CUDA device that holds the pool's memory
    bool top_dirty = true;         // top_chunks needs recomputing
    int top_chunks[33] = {};       // see PoolView::top_chunks
};

namespace lora {

// Slot table entry as stored in device memory (16 bytes).
struct SlotEntry {
    int32_t rank;   // true rank of the mounted adapter (0 when empty)
    int32_t state;  // kSlotEmpty / kSlotReady
    float scale;    // alpha / rank
    int32_t reserved;
};
static_assert(sizeof(SlotEntry) == 16, "slot entry layout");

constexpr int32_t kSlotEmpty = 0;
constexpr int32_t kSlotReady = 1;
constexpr int kMaxSlots = 2048;
constexpr int kMaxRank = 256;

// Everything a compute kernel needs to know about one pool.
struct PoolView {
    const SlotEntry* table;
    const void* A;  // [S, R, h_in]
    const void* B;  // [S, h_out, R]
    int h_in, h_out, R, S;
    int dtype;      // lora_dtype
    // top_chunks[k]: the largest number of 8-column chunks k slots can need at their true ranks
    // (ceil(rank / 8); empty slots count as r_max / 8, the worst a later mount can bring).  Sizes
    // the decode GEMM's staging of B tiles; the kernel re-checks the room it was given.
    int top_chunks[33];
};

// Segments as the kernels see them (device pointers).
// Words of the segment workspace's nseg array after the segment and item counts: the x-ready
// word a decode shrink publishes for the GEMM after it, and the count of that GEMM's CTAs that
// have read it.
constexpr int kXreadyWord = 2;
constexpr int kXreadyCount = 3;

struct SegView {
    const int32_t* perm;
    const int32_t* seg_start;
    const int32_t* seg_slot;
    const int32_t* nseg;
    int32_t* status;
    const int32_t* idx;
    const int32_t* items;  // [n][8] {slot, count, token[4]}; nseg[1] = number of items
    int n;
};

inline SegView seg_view(const lora_segments* s) {
    SegView v;
    v.perm = s->perm_dev;
    v.seg_start = s->seg_start_dev;
    v.seg_slot = s->seg_slot_dev;
    v.nseg = s->nseg_dev;
    v.status = s->status_dev;
    v.idx = s->idx_dev;
    v.items = s->items_dev;
    v.n = s->n_tokens;
    return v;
}

// Projections that read the same x and the same segments (q, k and v of an attention block;
// gate and up of an MLP) run as one linear over their row-concatenated base weight.  Slice q
// owns output columns [col[q], col[q + 1]) of y, whose row stride is ldy = col[count], and
// has its own adapter pool (same h_in, r_max, slot count and dtype as the others).  A single
// linear is the one-slice case.
constexpr int kMaxGroup = 4;
struct GroupView {
    int count;
    int ldy;
    int col[kMaxGroup + 1];
    int blk[kMaxGroup + 1];  // first expand block of each slice (set by the expand launcher)
    const SlotEntry* table[kMaxGroup];
    const void* A[kMaxGroup];
    const void* B[kMaxGroup];
    long long s_stride;  // floats between the shrink outputs of consecutive slices
    int rank_aware;      // some mounted slot holds a rank below r_max: kernels may skip its padding
    unsigned long long* stamp;  // benchmark instrumentation of the launch (nullptr: off)
    // Nonzero: the shrink kernel releases the fused decode GEMM after it at its start, and
    // writes this value to the segments' x-ready word once its own dependency wait has
    // returned (every kernel before it complete); the GEMM reads x after seeing that value.
    int xready;
};

// Whether some slot of the pool (empty slots count at r_max) holds fewer 8-column chunks than
// r_max: then skipping a slot's padding saves reads.
inline int has_padded_slots(const PoolView& pv) {
    const int k = pv.S < 32 ? pv.S : 32;
    return pv.top_chunks[k] < k * ((pv.R + 7) / 8) ? 1 : 0;
}

inline GroupView single_group(const PoolView& pv) {
    GroupView g;
    memset(&g, 0, sizeof(g));
    g.count = 1;
    g.ldy = pv.h_out;
    g.col[1] = pv.h_out;
    g.blk[1] = (pv.h_out + 255) / 256;
    g.table[0] = pv.table;
    g.A[0] = pv.A;
    g.B[0] = pv.B;
    g.rank_aware = has_padded_slots(pv);
    return g;
}

// One slice of a group, selected with compile-time indices (no local-memory copy of the
// parameter block).
struct SliceRef {
    const SlotEntry* table;
    const void* A;
    const void* B;
    int col, h_out;
    long long s_off;
};

__device__ __forceinline__ SliceRef group_slice(const GroupView& g, int q) {
    SliceRef r{g.table[0], g.A[0], g.B[0], g.col[0], g.col[1] - g.col[0], 0};
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (i == q) r = SliceRef{g.table[i], g.A[i], g.B[i], g.col[i], g.col[i + 1] - g.col[i], i * g.s_stride};
    return r;
}

// Slice owning output column c (columns of one slice are contiguous).
__device__ __forceinline__ int group_slice_of_col(const GroupView& g, int c) {
    int q = 0;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (i < g.count && c >= g.col[i]) q = i;
    return q;
}

inline size_t dtype_size(int dt) { return dt == LORA_F32 ? 4 : 2; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PoolView pool_view(const lora_pool_t p);

// Host-side error reporting (thread-local message), defined in api.cu.
int set_error(int code, const char* fmt, ...);
void count_launch(int n = 1);

// Launch helper attributes: every kernel of the hot path is launched with programmatic
// stream serialisation so that its prologue overlaps the tail of the previous kernel;
// each kernel waits (griddepcontrol.wait) before touching data an earlier kernel wrote.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

// ---- device helpers -----------------------------------------------------------------------

// Benchmark instrumentation (off unless lora_set_kernel_stamps is set): a launch records the
// %globaltimer of its first CTA's start and of its last CTA's end into a pair the host handed
// out.  Two atomics per CTA, no serialisation of neighbouring launches.
unsigned long long* take_kernel_stamp();
__device__ __forceinline__ unsigned long long stamp_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void stamp_start(unsigned long long* st) {
    if (st != nullptr && threadIdx.x == 0) atomicMin(st, stamp_clock());
}
__device__ __forceinline__ void stamp_end(unsigned long long* st) {
    if (st != nullptr && threadIdx.x == 0) atomicMax(st + 1, stamp_clock());
}
// The shrink / expand kernels' stamps (lora_set_aux_stamps): a triple {first CTA start, first
// return from the grid-dependency wait, last CTA end}, the end taken when thread 0 leaves.
unsigned long long* take_aux_stamp();
struct AuxStamp {
    unsigned long long* p;
    __device__ explicit AuxStamp(unsigned long long* q) : p(q) {
        if (p != nullptr && threadIdx.x == 0) atomicMin(p, stamp_clock());
    }
    __device__ void waited() const {
        if (p != nullptr && threadIdx.x == 0) atomicMin(p + 1, stamp_clock());
    }
    __device__ ~AuxStamp() {
        if (p != nullptr && threadIdx.x == 0) atomicMax(p + 2, stamp_clock());
    }
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Store with release semantics at GPU scope (a flag other CTAs or grids acquire).
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Unpack 8 16-bit values held in a uint4 to floats.
template <typename T> __device__ __forceinline__ void unpack8(const uint4& v, float* f);
template <> __device__ __forceinline__ void unpack8<__half>(const uint4& v, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 p = __half22float2(h[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}
template <> __device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4& v, float* f) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

}  // namespace lora

#define LORA_CUDA_TRY(expr)                                                                 \
    do {                                                                                    \
        cudaError_t _e = (expr);                                                            \
        if (_e != cudaSuccess)                                                              \
            return ::lora::set_error(LORA_ECUDA, "%s: %s", #expr, cudaGetErrorString(_e));  \
    } while (0)
