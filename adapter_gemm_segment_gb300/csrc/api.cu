// C ABI of the LoRA-augmented linear: workspace sizing, argument checks, variant policy and
// the launch sequence shrink -> base GEMM (+ fused expand) [-> separate expand].
//
// Variant policy: the blog.lonae.com page ("LLM 多 LoRA 推理服务工程 2026") reports that on
// A100/H100 the fused kernel wins from batch 8 up and the separate kernel at batch 1, and
// asks for the fused/separate threshold to be tuned per GPU model.  The threshold below is the
// one measured on GB300 (see the policy sweep of the benchmark).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace lora {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static unsigned long long* g_stamps = nullptr;
static int g_stamp_pairs = 0;
static int g_stamp_next = 0;

static unsigned long long* g_aux = nullptr;
static int g_aux_triples = 0;
static int g_aux_next = 0;

unsigned long long* take_aux_stamp() {
    if (!g_aux || g_aux_triples <= 0) return nullptr;
    unsigned long long* p = g_aux + 3 * (size_t)g_aux_next;
    g_aux_next = (g_aux_next + 1) % g_aux_triples;
    return p;
}

unsigned long long* take_kernel_stamp() {
    if (!g_stamps || g_stamp_pairs <= 0) return nullptr;
    unsigned long long* p = g_stamps + 2 * (size_t)g_stamp_next;
    g_stamp_next = (g_stamp_next + 1) % g_stamp_pairs;
    return p;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e == cudaSuccess) count_launch();
    return e;
}

int num_sms() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
    }
    return sms;
}

// Benchmark instrumentation: events recorded around the kernels of lora_linear_fwd.
static cudaEvent_t g_ev_before_shrink = nullptr, g_ev_before_gemm = nullptr, g_ev_after_gemm = nullptr;

static void record_if(cudaEvent_t e, cudaStream_t st) {
    if (!e) return;
    // Under stream capture a plain record only tracks dependencies; an external record node
    // is what re-records the event at every graph replay.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}

// Fused expand from this many tokens up; below it the separate residual kernel.
constexpr int kFusedMinTokens = 1;
constexpr int kVariantCudaCore = LORA_VARIANT_CUDA_CORE;

// Linear workspace: the shrink output, up to ceil(h_in/1024) K-parts of float32 [n, r_max]
// (alpha/r folded in).
struct LinWsLayout {
    size_t s_off, total;
};

static LinWsLayout lin_layout(const PoolView& pv, int n) {
    LinWsLayout L;
    L.s_off = 0;
    const int parts = shrink_parts(pv, n, false);
    L.total = align256(sizeof(float) * (size_t)(n > 0 ? n : 1) * pv.R * (size_t)parts);
    return L;
}

}  // namespace lora

using namespace lora;

extern "C" {

const char* lora_last_error(void) { return g_err; }

uint64_t lora_kernel_launch_count(void) { return g_launches.load(); }

int lora_set_aux_stamps(void* stamps_dev, int triples) {
    if (stamps_dev && triples <= 0) return set_error(LORA_EINVAL, "triples must be > 0");
    if (reinterpret_cast<uintptr_t>(stamps_dev) % 8) return set_error(LORA_EINVAL, "stamps must be 8-byte aligned");
    g_aux = static_cast<unsigned long long*>(stamps_dev);
    g_aux_triples = stamps_dev ? triples : 0;
    g_aux_next = 0;
    return LORA_OK;
}

int lora_set_kernel_stamps(void* stamps_dev, int pairs) {
    if (stamps_dev && pairs <= 0) return set_error(LORA_EINVAL, "pairs must be > 0");
    if (reinterpret_cast<uintptr_t>(stamps_dev) % 8) return set_error(LORA_EINVAL, "stamps must be 8-byte aligned");
    g_stamps = static_cast<unsigned long long*>(stamps_dev);
    g_stamp_pairs = stamps_dev ? pairs : 0;
    g_stamp_next = 0;
    return LORA_OK;
}

int lora_set_timing_events(void* before_shrink, void* before_gemm, void* after_gemm) {
    g_ev_before_shrink = static_cast<cudaEvent_t>(before_shrink);
    g_ev_before_gemm = static_cast<cudaEvent_t>(before_gemm);
    g_ev_after_gemm = static_cast<cudaEvent_t>(after_gemm);
    return LORA_OK;
}

int lora_linear_workspace_bytes(lora_pool_t pool, int n_tokens, size_t* bytes) {
    if (!pool || !bytes) return set_error(LORA_EINVAL, "pool/bytes is NULL");
    if (n_tokens < 0) return set_error(LORA_EINVAL, "n_tokens < 0");
    *bytes = lin_layout(pool_view(pool), n_tokens).total;
    return LORA_OK;
}

int lora_linear_policy(lora_pool_t pool, int n_tokens, int* variant) {
    if (!pool || !variant) return set_error(LORA_EINVAL, "pool/variant is NULL");
    // Measured on GB300 (32 chained linears per step): fused wins from one token up as long
    // as the decode GEMM stages every adapter its CTAs meet; past that the separate variant
    // (base GEMM + segmented expand) is faster.  Prefill batches (> 256 tokens) are fused.
    const PoolView pv = pool_view(pool);
    if (n_tokens < kFusedMinTokens) *variant = LORA_VARIANT_SEPARATE;
    else if (n_tokens <= 256 && tc_supported(pv, n_tokens) && !decode_fused_fits(pv, n_tokens))
        *variant = LORA_VARIANT_SEPARATE;
    else
        *variant = LORA_VARIANT_FUSED;
    return LORA_OK;
}

int lora_linear_fwd(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev, const lora_segments* seg,
                    int variant, void* ws_dev, size_t ws_bytes, void* stream) {
    return lora_linear_fwd_ex(pool, W_dev, x_dev, y_dev, seg, variant, ws_dev, ws_bytes, nullptr, 0, stream);
}

int lora_linear_fwd_ex(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev, const lora_segments* seg,
                       int variant, void* ws_dev, size_t ws_bytes, const void* prefetch_dev, size_t prefetch_bytes,
                       void* stream) {
    if (!pool || !seg) return set_error(LORA_EINVAL, "pool/seg is NULL");
    const PoolView pv = pool_view(pool);
    const int n = seg->n_tokens;
    if (seg->n_slots != pv.S)
        return set_error(LORA_EINVAL, "segments were built for %d slots, pool has %d", seg->n_slots, pv.S);
    if (variant < LORA_VARIANT_AUTO || variant > kVariantCudaCore) return set_error(LORA_EINVAL, "bad variant %d", variant);
    if (n == 0) return LORA_OK;
    if (!W_dev || !x_dev || !y_dev || !ws_dev) return set_error(LORA_EINVAL, "W/x/y/ws is NULL");
    if (prefetch_dev && (reinterpret_cast<uintptr_t>(prefetch_dev) % 16))
        return set_error(LORA_EINVAL, "prefetch range must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(ws_dev) % 256) return set_error(LORA_EINVAL, "ws must be 256-byte aligned");
    if (pv.dtype != LORA_F32) {
        if ((reinterpret_cast<uintptr_t>(W_dev) | reinterpret_cast<uintptr_t>(x_dev) |
             reinterpret_cast<uintptr_t>(y_dev)) % 16)
            return set_error(LORA_EINVAL, "W/x/y must be 16-byte aligned");
    } else if ((reinterpret_cast<uintptr_t>(W_dev) | reinterpret_cast<uintptr_t>(x_dev) |
                reinterpret_cast<uintptr_t>(y_dev)) % 4) {
        return set_error(LORA_EINVAL, "W/x/y must be 4-byte aligned");
    }
    const LinWsLayout L = lin_layout(pv, n);
    if (ws_bytes < L.total) return set_error(LORA_ENOSPACE, "linear workspace needs %zu bytes, got %zu", L.total, ws_bytes);
    char* w = static_cast<char*>(ws_dev);
    float* s_buf = reinterpret_cast<float*>(w + L.s_off);
    return linear_fwd_impl(pool, W_dev, x_dev, y_dev, seg, variant, s_buf, prefetch_dev, prefetch_bytes,
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace lora {

// Values of the x-ready hand-off: distinct for the shrink/GEMM pairs launched one after another
// over the same segments (never 0, which means off).
static int next_xready_value() {
    static std::atomic<unsigned> seq{0};
    return static_cast<int>((seq.fetch_add(1, std::memory_order_relaxed) & 0x3fffffffu) + 1u);
}

// The launch sequence of one LoRA-augmented linear, after its arguments were checked; s_buf
// receives the shrink output (float32 [parts][n][r_max]).
int linear_fwd_impl(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev, const lora_segments* seg,
                    int variant, float* s_buf, const void* prefetch_dev, size_t prefetch_bytes, cudaStream_t st) {
    const PoolView pv = pool_view(pool);
    const int n = seg->n_tokens;
    if (variant == LORA_VARIANT_AUTO) lora_linear_policy(pool, n, &variant);
    const SegView sv = seg_view(seg);

    const bool tc = variant != kVariantCudaCore && tc_supported(pv, n);
    const bool fused = variant != LORA_VARIANT_SEPARATE;
    // A fused decode GEMM after the per-token shrink kernel follows it through the x-ready
    // hand-off: the shrink releases it at once and publishes a value unique to this pair once
    // every earlier kernel is complete, so the GEMM's weight stream and its B staging overlap
    // the previous linear's tail.  Measured on GB300 (32 chained 4096 x 4096 fp16 linears, us
    // per linear with / without): r_max 8 at 16, 32, 64 tokens 13.44 / 14.09, 13.68 / 14.61,
    // 13.58 / 15.17; r_max 64 at 16 tokens 16.49 / 16.67.  Behind the segmented shrink (r_max 64
    // at 64 tokens: many more CTAs, a longer shrink) it lost: 19.44 / 18.83.  At 1-8 tokens it
    // also beat a shrink computed inside the GEMM's own grid (11.7-11.9 against 12.2-13.2).
    const int xready = (tc && fused && n <= 256 && !shrink_segmented(pv, n)) ? next_xready_value() : 0;
    record_if(g_ev_before_shrink, st);
    int rc = LORA_OK;
    int s_parts = 1;
    if (tc && n > 256 && shrink_tc_supported(pv))
        rc = launch_shrink_tc(pv, sv, x_dev, s_buf, st);
    else
        rc = launch_shrink(pv, sv, x_dev, s_buf, st, /*tiled=*/n > 256, &s_parts, xready);
    if (rc) return rc;
    record_if(g_ev_before_gemm, st);
    if (tc) {
        rc = launch_gemm_tc(pv, sv, W_dev, x_dev, s_buf, s_parts, y_dev, fused, st, prefetch_dev, prefetch_bytes,
                            nullptr, xready);
    } else {
        rc = launch_gemm_simt(pv, sv, W_dev, x_dev, s_buf, s_parts, y_dev, fused, st);
    }
    if (rc) return rc;
    record_if(g_ev_after_gemm, st);
    if (!fused) {
        rc = launch_expand(pv, sv, s_buf, s_parts, y_dev, st);
        if (rc) return rc;
    }
    return LORA_OK;
}

}  // namespace lora

// ---- grouped projections ------------------------------------------------------------------

namespace lora {

// Checks the pools of a group and builds the pool views and the slice table (s_stride left 0).
static int group_setup(int count, const lora_pool_t* pools, PoolView* pvs, GroupView* grp) {
    if (count < 1 || count > kMaxGroup) return set_error(LORA_EINVAL, "group of %d slices (1..%d)", count, kMaxGroup);
    if (!pools) return set_error(LORA_EINVAL, "pools is NULL");
    for (int q = 0; q < count; ++q) {
        if (!pools[q]) return set_error(LORA_EINVAL, "pools[%d] is NULL", q);
        pvs[q] = pool_view(pools[q]);
    }
    const PoolView& p0 = pvs[0];
    if (p0.dtype != LORA_F16 && p0.dtype != LORA_BF16)
        return set_error(LORA_EUNSUP, "grouped projections need fp16 or bf16 pools");
    memset(grp, 0, sizeof(*grp));
    grp->count = count;
    for (int q = 0; q < count; ++q) {
        const PoolView& p = pvs[q];
        if (p.h_in != p0.h_in || p.R != p0.R || p.S != p0.S || p.dtype != p0.dtype)
            return set_error(LORA_EINVAL, "pool %d differs from pool 0 in h_in, r_max, n_slots or dtype", q);
        if (count > 1 && p.h_out % 16)
            return set_error(LORA_EINVAL, "pool %d: h_out %d is not a multiple of 16", q, p.h_out);
        if (pools[q]->mounted != pools[0]->mounted)
            return set_error(LORA_EINVAL, "pool %d does not hold the same slots as pool 0", q);
        grp->table[q] = p.table;
        grp->A[q] = p.A;
        grp->B[q] = p.B;
        grp->rank_aware |= has_padded_slots(p);
        grp->col[q + 1] = grp->col[q] + p.h_out;
        grp->blk[q + 1] = grp->blk[q] + (p.h_out + 255) / 256;
    }
    grp->ldy = grp->col[count];
    return LORA_OK;
}

}  // namespace lora

using namespace lora;

extern "C" {

int lora_linear_group_workspace_bytes(int count, const lora_pool_t* pools, int n_tokens, size_t* bytes) {
    if (!bytes) return set_error(LORA_EINVAL, "bytes is NULL");
    if (n_tokens < 0) return set_error(LORA_EINVAL, "n_tokens < 0");
    PoolView pvs[kMaxGroup];
    GroupView grp;
    const int rc = group_setup(count, pools, pvs, &grp);
    if (rc) return rc;
    *bytes = (size_t)count * lin_layout(pvs[0], n_tokens).total;
    return LORA_OK;
}

int lora_linear_group_policy(int count, const lora_pool_t* pools, int n_tokens, int* variant) {
    if (!variant) return set_error(LORA_EINVAL, "variant is NULL");
    PoolView pvs[kMaxGroup];
    GroupView grp;
    const int rc = group_setup(count, pools, pvs, &grp);
    if (rc) return rc;
    // A group of one is a single linear: its policy.  Otherwise, measured on GB300 (7B-shaped
    // layers, 64 and 256 tokens, bf16, r_max 16): the base GEMM over the concatenated weight
    // plus one segmented expand beat per-slice fused GEMMs at decode sizes; prefill batches
    // keep the fused epilogue.
    if (count == 1) return lora_linear_policy(pools[0], n_tokens, variant);
    *variant = n_tokens <= 256 ? LORA_VARIANT_SEPARATE : LORA_VARIANT_FUSED;
    return LORA_OK;
}

int lora_linear_fwd_group(int count, const lora_pool_t* pools, const void* W_dev, const void* x_dev, void* y_dev,
                          const lora_segments* seg, int variant, void* ws_dev, size_t ws_bytes, void* stream) {
    if (!seg) return set_error(LORA_EINVAL, "seg is NULL");
    PoolView pvs[kMaxGroup];
    GroupView grp;
    int rc = group_setup(count, pools, pvs, &grp);
    if (rc) return rc;
    const PoolView& p0 = pvs[0];
    const int n = seg->n_tokens;
    if (seg->n_slots != p0.S)
        return set_error(LORA_EINVAL, "segments were built for %d slots, pools have %d", seg->n_slots, p0.S);
    if (variant != LORA_VARIANT_AUTO && variant != LORA_VARIANT_FUSED && variant != LORA_VARIANT_SEPARATE)
        return set_error(variant == kVariantCudaCore ? LORA_EUNSUP : LORA_EINVAL, "variant %d for a group", variant);
    if (n == 0) return LORA_OK;
    if (!W_dev || !x_dev || !y_dev || !ws_dev) return set_error(LORA_EINVAL, "W/x/y/ws is NULL");
    if ((reinterpret_cast<uintptr_t>(W_dev) | reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev)) %
        16)
        return set_error(LORA_EINVAL, "W/x/y must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(ws_dev) % 256) return set_error(LORA_EINVAL, "ws must be 256-byte aligned");
    const size_t slice_ws = lin_layout(p0, n).total;
    if (ws_bytes < (size_t)count * slice_ws)
        return set_error(LORA_ENOSPACE, "group workspace needs %zu bytes, got %zu", (size_t)count * slice_ws, ws_bytes);
    grp.s_stride = (long long)(slice_ws / sizeof(float));
    PoolView pcat = p0;  // the concatenated linear: [sum of h_out, h_in]
    pcat.h_out = grp.ldy;
    if (!tc_supported(pcat, n)) return set_error(LORA_EUNSUP, "no tensor-core plan for this group and batch");
    if (variant == LORA_VARIANT_AUTO) lora_linear_group_policy(count, pools, n, &variant);
    if (count == 1)  // one slice: exactly the single linear's launch sequence
        return linear_fwd_impl(pools[0], W_dev, x_dev, y_dev, seg, variant,
                               reinterpret_cast<float*>(static_cast<char*>(ws_dev) + lin_layout(p0, n).s_off), nullptr, 0,
                               static_cast<cudaStream_t>(stream));
    const bool fused = variant == LORA_VARIANT_FUSED;
    const bool decode = n <= 256;
    if (decode && fused)
        for (int q = 0; q < count; ++q)
            if (!tc_supported(pvs[q], n)) return set_error(LORA_EUNSUP, "no fused tensor-core plan for slice %d", q);
    const SegView sv = seg_view(seg);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* s_buf = static_cast<float*>(ws_dev);
    const size_t elt = dtype_size(p0.dtype);

    record_if(g_ev_before_shrink, st);
    int s_parts = 1;
    if (decode) {
        rc = launch_shrink_group(p0, grp, sv, x_dev, s_buf, st, /*tiled=*/false, &s_parts);  // every slice, one launch
        if (rc) return rc;
    } else if (shrink_tc_group_supported(p0, count)) {
        rc = launch_shrink_tc_group(p0, grp, sv, x_dev, s_buf, st);  // every slice, one launch
        if (rc) return rc;
    } else {
        for (int q = 0; q < count; ++q) {
            float* s_q = s_buf + (size_t)q * grp.s_stride;
            rc = shrink_tc_supported(pvs[q]) ? launch_shrink_tc(pvs[q], sv, x_dev, s_q, st)
                                             : launch_shrink(pvs[q], sv, x_dev, s_q, st, /*tiled=*/true, &s_parts);
            if (rc) return rc;
        }
    }
    record_if(g_ev_before_gemm, st);
    if (decode && fused) {
        // the decode kernel's fused epilogue serves one pool: one launch per slice, each writing
        // its column range of y
        for (int q = 0; q < count; ++q) {
            GroupView gq;
            memset(&gq, 0, sizeof(gq));
            gq.count = 1;
            gq.ldy = grp.ldy;
            gq.col[1] = pvs[q].h_out;
            gq.blk[1] = (pvs[q].h_out + 255) / 256;
            gq.table[0] = pvs[q].table;
            gq.A[0] = pvs[q].A;
            gq.B[0] = pvs[q].B;
            gq.rank_aware = has_padded_slots(pvs[q]);
            const char* Wq = static_cast<const char*>(W_dev) + (size_t)grp.col[q] * p0.h_in * elt;
            char* yq = static_cast<char*>(y_dev) + (size_t)grp.col[q] * elt;
            rc = launch_gemm_tc(pvs[q], sv, Wq, x_dev, s_buf + (size_t)q * grp.s_stride, s_parts, yq, true, st, nullptr,
                                0, &gq);
            if (rc) return rc;
        }
    } else if (decode && !fused && count > 1 && n > 64) {
        // x is as large as the W tiles here: 256-row tiles halve its re-reads
        rc = launch_gemm_tall(pcat, sv, W_dev, x_dev, y_dev, grp.ldy, st);
        if (rc) return rc;
    } else {
        // one base GEMM over the concatenated weight; the prefill kernel applies each slice's
        // LoRA term in its epilogue
        rc = launch_gemm_tc(pcat, sv, W_dev, x_dev, s_buf, s_parts, y_dev, fused && !decode, st, nullptr, 0, &grp);
        if (rc) return rc;
    }
    record_if(g_ev_after_gemm, st);
    if (!fused) {
        rc = launch_expand_group(p0, grp, sv, s_buf, s_parts, y_dev, st);
        if (rc) return rc;
    }
    return LORA_OK;
}

}  // extern "C"
