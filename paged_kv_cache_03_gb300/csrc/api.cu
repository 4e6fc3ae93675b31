// api.cu -- the extern "C" entry points of paged_attn.h: argument checks on
// the host, schedule choice (the shape dispatch that "Week 3 Day 5: Paged
// FlashAttention" puts inside the extension), and the launches.
#include <cfloat>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace pa {

pa_status current_device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    if (dev >= 64) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = cache[dev];
    if (d.device != dev) {
        DeviceInfo n;
        n.device = dev;
        if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&n.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        d = n;
    }
    *out = d;
    return PA_OK;
}

namespace {

pa_status check_shape(const pa_shape* s) {
    if (!s) return PA_ERR_INVALID_ARG;
    if (s->B < 1 || s->H_q < 1 || s->H_kv < 1 || s->L < 1 || s->D < 1 || s->num_pages < 1 ||
        s->page_size < 1 || s->max_pages_per_seq < 1)
        return PA_ERR_INVALID_ARG;
    if (s->H_q % s->H_kv != 0) return PA_ERR_INVALID_ARG;
    if (s->dtype != PA_BF16 && s->dtype != PA_F32) return PA_ERR_INVALID_ARG;
    if (s->D != kHeadDim) return PA_ERR_UNSUPPORTED;
    // row indices of the pool and key positions stay inside int32
    if (static_cast<long long>(s->num_pages) * s->H_kv * s->page_size >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(s->max_pages_per_seq) * s->page_size >= (1ll << 30))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(s->H_q) * s->L >= (1ll << 30)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// `scale` is the softmax temperature 1/sqrt(D) of standard attention: finite
// and >= 0.  (The tile kernel takes a row's max over the raw scores and scales
// it once, which is the max of the scaled scores only for scale >= 0.)  NaN,
// negative and infinite values are rejected.
bool scale_ok(float scale) { return scale >= 0.f && scale <= FLT_MAX; }

int choose(const pa_shape& s) {
    if (s.dtype != PA_BF16 || !prefill_supported(s)) return PA_SCHED_DECODE;
    const long long rows = static_cast<long long>(s.H_q / s.H_kv) * s.L;
    // Measured crossover (operator sweep, G in {1, 4}, L in {1, 2, 4},
    // contexts 256 to 16384, B in {1, 2, 4, 8, 64}, H_kv = 8): with more than
    // 4 query rows per kv head the tensor-core tiles win everywhere (1.5x at 8
    // rows and B = 8 over 16384 keys, 2-3x beyond).  With at most 4 rows the
    // page walk wins over a real batch; the tiles, which cut the keys of few
    // (sequence, kv head) pairs into chunks on SMs of their own, win (1) on
    // calls so small that their lower fixed cost decides: B * H_kv * context
    // capacity up to 64K token rows and a capacity of at most 1024 keys,
    // (2) with at most 8 pairs at any context (B = 1 over 16384 keys: 29-33
    // against 41-42 us), (3) with at most 32 pairs over at most 4096 keys
    // (B = 4: 27 against 31-32 us; over 16384 keys the page walk, 60 against
    // 69 us; B = 8 over 4096 keys: page walk 41 against 44 us).
    if (rows > kMixedDecodeRows) return PA_SCHED_PREFILL;
    const long long cap = static_cast<long long>(s.max_pages_per_seq) * s.page_size;
    const long long pairs = static_cast<long long>(s.B) * s.H_kv;
    if (pairs * cap <= 65536 && cap <= 1024) return PA_SCHED_PREFILL;
    if (pairs <= 8 || (pairs <= 32 && cap <= 4096)) return PA_SCHED_PREFILL;
    return PA_SCHED_DECODE;
}

}  // namespace

pa_status check_call_args(const pa_shape* shape, const void* query, const void* key_pages,
                          const void* value_pages, const int32_t* block_table,
                          const int32_t* context_lens, float scale, const void* out) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(key_pages, 16) || !aligned(value_pages, 16) ||
        !aligned(out, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!scale_ok(scale)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

namespace {

pa_status run(const pa_shape* shape, const void* query, const void* key_pages,
              const void* value_pages, const int32_t* block_table, const int32_t* context_lens,
              float scale, int causal, void* out, void* workspace, size_t workspace_bytes,
              void* cuda_stream, int schedule, void* ev_before = nullptr,
              void* ev_after = nullptr, const float* mask = nullptr, long long mask_S = 0) {
    pa_status st = check_call_args(shape, query, key_pages, value_pages, block_table,
                                   context_lens, scale, out);
    if (st != PA_OK) return st;
    if (!workspace || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    if (schedule == PA_SCHED_AUTO) schedule = choose(*shape);
    if (schedule != PA_SCHED_DECODE && schedule != PA_SCHED_PREFILL) return PA_ERR_INVALID_ARG;
    if (schedule == PA_SCHED_PREFILL && !prefill_supported(*shape)) return PA_ERR_UNSUPPORTED;

    Call c;
    c.sh = *shape;
    c.q = query;
    c.kp = key_pages;
    c.vp = value_pages;
    c.bt = block_table;
    c.ctx = context_lens;
    c.scale = scale;
    c.causal = causal ? 1 : 0;
    c.out = out;
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.stream = static_cast<cudaStream_t>(cuda_stream);
    c.ev_before = static_cast<cudaEvent_t>(ev_before);
    c.ev_after = static_cast<cudaEvent_t>(ev_after);
    c.mask = mask;
    c.mask_S = mask_S;
    st = current_device_info(&c.dev);
    if (st != PA_OK) return st;
    if (c.dev.cc_major != 10 || c.dev.cc_minor != 3) return PA_ERR_UNSUPPORTED;
    if (workspace_bytes < kFlagBytes) return PA_ERR_WORKSPACE;
    return schedule == PA_SCHED_DECODE ? decode_launch(c) : prefill_launch(c);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_workspace_bytes(const pa_shape* shape) {
    if (check_shape(shape) != PA_OK) return 0;
    DeviceInfo dev;
    if (current_device_info(&dev) != PA_OK) return 0;
    return workspace_bytes_total(*shape, dev.sm_count);
}

pa_status pa_paged_attention(const pa_shape* shape, const void* query, const void* key_pages,
                             const void* value_pages, const int32_t* block_table,
                             const int32_t* context_lens, float scale, int causal, void* out,
                             void* workspace, size_t workspace_bytes, void* cuda_stream) {
    return run(shape, query, key_pages, value_pages, block_table, context_lens, scale, causal,
               out, workspace, workspace_bytes, cuda_stream, PA_SCHED_AUTO);
}

pa_status pa_paged_attention_sched(const pa_shape* shape, const void* query,
                                   const void* key_pages, const void* value_pages,
                                   const int32_t* block_table, const int32_t* context_lens,
                                   float scale, int causal, void* out, void* workspace,
                                   size_t workspace_bytes, void* cuda_stream, int schedule) {
    return run(shape, query, key_pages, value_pages, block_table, context_lens, scale, causal,
               out, workspace, workspace_bytes, cuda_stream, schedule);
}

pa_status pa_paged_attention_profiled(const pa_shape* shape, const void* query,
                                      const void* key_pages, const void* value_pages,
                                      const int32_t* block_table, const int32_t* context_lens,
                                      float scale, int causal, void* out, void* workspace,
                                      size_t workspace_bytes, void* cuda_stream, int schedule,
                                      void* event_before, void* event_after) {
    return run(shape, query, key_pages, value_pages, block_table, context_lens, scale, causal,
               out, workspace, workspace_bytes, cuda_stream, schedule, event_before, event_after);
}

pa_status pa_paged_attention_masked(const pa_shape* shape, const void* query,
                                    const void* key_pages, const void* value_pages,
                                    const int32_t* block_table, const int32_t* context_lens,
                                    float scale, int causal, const float* mask,
                                    long long mask_S, void* out, void* workspace,
                                    size_t workspace_bytes, void* cuda_stream, int schedule) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!mask || !aligned(mask, 16)) return PA_ERR_INVALID_ARG;
    const long long cap = static_cast<long long>(shape->max_pages_per_seq) * shape->page_size;
    if (mask_S < cap || mask_S % 4 != 0) return PA_ERR_INVALID_ARG;
    return run(shape, query, key_pages, value_pages, block_table, context_lens, scale, causal,
               out, workspace, workspace_bytes, cuda_stream, schedule, nullptr, nullptr, mask,
               mask_S);
}

pa_status pa_paged_attention_varlen(const pa_shape* shape, const void* query,
                                    const void* key_pages, const void* value_pages,
                                    const int32_t* block_table, const int32_t* context_lens,
                                    const int32_t* cu_q, int total_q, float scale, int causal,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* cuda_stream, int schedule) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    const pa_shape& sh = *shape;
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !cu_q || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(key_pages, 16) || !aligned(value_pages, 16) ||
        !aligned(out, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4) ||
        !aligned(cu_q, 4))
        return PA_ERR_INVALID_ARG;
    if (total_q < 0 || !scale_ok(scale)) return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(total_q) * sh.H_q >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    if (schedule != PA_SCHED_AUTO && schedule != PA_SCHED_DECODE && schedule != PA_SCHED_PREFILL)
        return PA_ERR_INVALID_ARG;

    Call c;
    c.sh = sh;
    c.q = query;
    c.kp = key_pages;
    c.vp = value_pages;
    c.bt = block_table;
    c.ctx = context_lens;
    c.scale = scale;
    c.causal = causal ? 1 : 0;
    c.out = out;
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.stream = static_cast<cudaStream_t>(cuda_stream);
    c.cu_q = cu_q;
    c.total_q = total_q;
    st = current_device_info(&c.dev);
    if (st != PA_OK) return st;
    if (c.dev.cc_major != 10 || c.dev.cc_minor != 3) return PA_ERR_UNSUPPORTED;
    c.plan_off = varlen_plan_offset(sh, c.dev.sm_count);
    if (workspace_bytes < workspace_bytes_total(sh, c.dev.sm_count)) return PA_ERR_WORKSPACE;
    if (total_q == 0) return PA_OK;  // no query rows

    // Which sequences each schedule takes: a forced schedule takes all; AUTO
    // gives sequences with at most kMixedDecodeRows query rows per kv head to
    // the page walk and the rest to the tensor-core tiles, both in this call.
    const int G = sh.H_q / sh.H_kv;
    const bool tiles_ok = sh.dtype == PA_BF16 && prefill_supported(sh);
    bool run_decode = false, run_tiles = false;
    int dec_L = sh.L;
    if (schedule == PA_SCHED_DECODE || (schedule == PA_SCHED_AUTO && !tiles_ok)) {
        run_decode = true;
    } else if (schedule == PA_SCHED_PREFILL) {
        if (!tiles_ok) return PA_ERR_UNSUPPORTED;
        run_tiles = true;
        c.tiles_min_L = 0;
    } else {  // AUTO, mixed
        dec_L = kMixedDecodeRows / G < sh.L ? kMixedDecodeRows / G : sh.L;
        run_decode = dec_L > 0;
        run_tiles = dec_L < sh.L;
        c.tiles_min_L = dec_L;
        c.route_mixed = run_tiles ? 1 : 0;
    }
    if (run_tiles) {
        st = prefill_launch(c);
        if (st != PA_OK) return st;
    }
    if (run_decode) {
        Call d = c;
        d.sh.L = dec_L;  // the largest L_b the page walk takes
        d.overlap_prev = run_tiles;  // the two touch disjoint rows: run side by side
        st = decode_launch(d);
    }
    return st;
}

pa_status pa_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                   unsigned timeout_us, void* cuda_stream) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < kFlagBytes)
        return PA_ERR_WORKSPACE;
    if (timeout_us > kWaitTimeoutNs / 1000) return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    const pa_status st = current_device_info(&dev);
    if (st != PA_OK) return st;
    return wait_timeout_launch(static_cast<uint32_t*>(workspace), 1000ull * timeout_us,
                               static_cast<cudaStream_t>(cuda_stream));
}

pa_status pa_gather_debug(const pa_shape* shape, const void* key_pages, const void* value_pages,
                          const int32_t* block_table, const int32_t* context_lens, int max_S,
                          void* k_dense, void* v_dense, void* workspace, void* cuda_stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!key_pages || !value_pages || !block_table || !context_lens || !k_dense || !v_dense ||
        max_S < 1)
        return PA_ERR_INVALID_ARG;
    if (!aligned(key_pages, 16) || !aligned(value_pages, 16) || !aligned(k_dense, 16) ||
        !aligned(v_dense, 16))
        return PA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 4)) return PA_ERR_WORKSPACE;
    return gather_launch(*shape, key_pages, value_pages, block_table, context_lens, max_S,
                         k_dense, v_dense, static_cast<uint32_t*>(workspace),
                         static_cast<cudaStream_t>(cuda_stream));
}

pa_status pa_append_kv(const pa_shape* shape, const void* k_new, const void* v_new,
                       void* key_pages, void* value_pages, const int32_t* block_table,
                       const int32_t* context_lens, void* workspace, size_t workspace_bytes,
                       void* cuda_stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!k_new || !v_new || !key_pages || !value_pages || !block_table || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(key_pages, 16) ||
        !aligned(value_pages, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 4) || workspace_bytes < kFlagBytes)
        return PA_ERR_WORKSPACE;
    const int es = shape->dtype == PA_BF16 ? 2 : 4;
    const long long chunks = static_cast<long long>(shape->B) * shape->H_kv * shape->L *
                             (shape->D * es / 16);
    if (chunks >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    DeviceInfo dev;
    st = current_device_info(&dev);
    if (st != PA_OK) return st;
    return append_launch(*shape, k_new, v_new, key_pages, value_pages, block_table, context_lens,
                         static_cast<uint32_t*>(workspace), dev.sm_count,
                         static_cast<cudaStream_t>(cuda_stream));
}

pa_status pa_check_device_flag(void* workspace, uint32_t* flag_out, int clear, void* cuda_stream) {
    if (!workspace) return PA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    uint32_t f = 0;
    if (cudaMemcpyAsync(&f, workspace, sizeof f, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    if (clear && f) {
        if (cudaMemsetAsync(workspace, 0, sizeof f, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }
    if (flag_out) *flag_out = f;
    return f ? PA_ERR_DEVICE_FLAG : PA_OK;
}

pa_status pa_validate_metadata(const pa_shape* shape, const int32_t* block_table,
                               const int32_t* context_lens, int causal, void* cuda_stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!block_table || !context_lens) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    std::vector<int32_t> ctx(shape->B);
    std::vector<int32_t> bt(static_cast<size_t>(shape->B) * shape->max_pages_per_seq);
    if (cudaMemcpyAsync(ctx.data(), context_lens, ctx.size() * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(bt.data(), block_table, bt.size() * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    const long long cap = static_cast<long long>(shape->max_pages_per_seq) * shape->page_size;
    for (int b = 0; b < shape->B; ++b) {
        const int S = ctx[b];
        if (S < 1 || S > cap || (causal && S < shape->L)) return PA_ERR_INVALID_ARG;
        const int npg = (S + shape->page_size - 1) / shape->page_size;
        for (int i = 0; i < npg; ++i) {
            const int32_t pp = bt[static_cast<size_t>(b) * shape->max_pages_per_seq + i];
            if (pp < 0 || pp >= shape->num_pages) return PA_ERR_BAD_BLOCK_TABLE;
        }
    }
    return PA_OK;
}

pa_status pa_validate_metadata_varlen(const pa_shape* shape, const int32_t* block_table,
                                      const int32_t* context_lens, const int32_t* cu_q,
                                      int total_q, int causal, void* cuda_stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!block_table || !context_lens || !cu_q || total_q < 0) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    std::vector<int32_t> ctx(shape->B), cu(static_cast<size_t>(shape->B) + 1);
    std::vector<int32_t> bt(static_cast<size_t>(shape->B) * shape->max_pages_per_seq);
    if (cudaMemcpyAsync(ctx.data(), context_lens, ctx.size() * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(cu.data(), cu_q, cu.size() * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(bt.data(), block_table, bt.size() * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    if (cu[0] != 0 || cu[shape->B] != total_q) return PA_ERR_INVALID_ARG;
    const long long cap = static_cast<long long>(shape->max_pages_per_seq) * shape->page_size;
    for (int b = 0; b < shape->B; ++b) {
        const int Lb = cu[b + 1] - cu[b];
        if (Lb < 0 || Lb > shape->L) return PA_ERR_INVALID_ARG;
        if (Lb == 0) continue;  // not read
        const int S = ctx[b];
        if (S < 1 || S > cap || (causal && S < Lb)) return PA_ERR_INVALID_ARG;
        const int npg = (S + shape->page_size - 1) / shape->page_size;
        for (int i = 0; i < npg; ++i) {
            const int32_t pp = bt[static_cast<size_t>(b) * shape->max_pages_per_seq + i];
            if (pp < 0 || pp >= shape->num_pages) return PA_ERR_BAD_BLOCK_TABLE;
        }
    }
    return PA_OK;
}

int pa_choose_schedule(const pa_shape* shape) {
    if (check_shape(shape) != PA_OK) return -1;
    return choose(*shape);
}

int pa_launch_count(const pa_shape* shape, int schedule) {
    if (check_shape(shape) != PA_OK) return -1;
    if (schedule == PA_SCHED_AUTO) schedule = choose(*shape);
    if (schedule == PA_SCHED_DECODE) return 2;
    DeviceInfo dev;
    if (current_device_info(&dev) != PA_OK) return -1;
    // tiles (+ the merge of key chunks or of the last tile's rows)
    return (tile_nsplit(*shape, dev.sm_count) > 1 || tile_remainder_rows(*shape) > 0) ? 2 : 1;
}

const char* pa_status_str(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_BAD_BLOCK_TABLE: return "block table entry out of range";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_DEVICE_FLAG: return "kernel recorded an error in the device flag";
    }
    return "unknown status";
}

}  // extern "C"
