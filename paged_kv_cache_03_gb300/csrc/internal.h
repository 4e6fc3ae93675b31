// internal.h -- declarations shared by the host dispatcher and the kernel
// translation units (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "paged_attn.h"

namespace pa {

constexpr int kHeadDim = 128;
// Workspace: [0, kFlagBytes) holds the sticky flag word (offset 0) and the
// decode schedule's chunk counters, all zero between calls.
constexpr size_t kFlagBytes = 256;
constexpr size_t kChunkCounterOffset = 64;
constexpr size_t kDoneCounterOffset = 128;
// the tile schedule's work-item counter and its CTAs-done counter (2 ints)
constexpr size_t kTileCounterOffset = 192;

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};

// Properties of the current device (cached per device).
pa_status current_device_info(DeviceInfo* out);

// Host-side checks of one attention call that need no device: the shape,
// null and misaligned pointers, and the scale (finite, >= 0).
pa_status check_call_args(const pa_shape* shape, const void* query, const void* key_pages,
                          const void* value_pages, const int32_t* block_table,
                          const int32_t* context_lens, float scale, const void* out);

struct Call {
    pa_shape sh;
    const void* q;
    const void* kp;
    const void* vp;
    const int32_t* bt;
    const int32_t* ctx;
    float scale;
    int causal;
    void* out;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
    cudaEvent_t ev_before = nullptr;  // recorded around the dominant kernel
    cudaEvent_t ev_after = nullptr;
    // optional additive mask [B * H_q, L, mask_S] (fp32), mask_S >= the table's
    // capacity and a multiple of 4
    const float* mask = nullptr;
    long long mask_S = 0;
    // ragged batch: query / output packed by token [total_q, H_q, D], sequence
    // b owns tokens cu_q[b] .. cu_q[b + 1] - 1 (null: [B, H_q, L, D]); sh.L
    // bounds every L_b
    const int32_t* cu_q = nullptr;
    int total_q = 0;
    int route_mixed = 0;   // decode: sequences with L_b > sh.L belong to the tiles
    int tiles_min_L = 0;   // tiles: only sequences with L_b > tiles_min_L
    size_t plan_off = 0;   // workspace offset of the tile schedule's pair plan
    bool overlap_prev = false;  // decode: launch as the tile kernel's programmatic dependent
    DeviceInfo dev;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- decode schedule (split-S page walk on CUDA cores + combine) ----------
// Rows of one (b, kv_head) handled together by one pass over its keys.
int decode_rows_per_chunk(const pa_shape& sh);
size_t decode_workspace_bytes(const pa_shape& sh, int sm_count);
// Ragged batches: the tile schedule's pair plan (B + 1 ints) follows the
// decode schedule's workspace.
size_t varlen_plan_offset(const pa_shape& sh, int sm_count);
size_t workspace_bytes_total(const pa_shape& sh, int sm_count);
// In a mixed ragged batch the page walk takes the sequences with at most this
// many query rows per kv head (G * L_b), the tiles the rest.
constexpr int kMixedDecodeRows = 4;
int decode_grid(const pa_shape& sh, int sm_count);
pa_status decode_launch(const Call& c);

// ---- prefill schedule (tcgen05 tensor cores) ------------------------------
bool prefill_supported(const pa_shape& sh);
// Key chunks per query-tile pair ([B, H_q, L, D] layout, no mask): more than 1
// when at least two chunks per pair still give every item an SM of its own;
// their partials follow the ragged batch's plan in the workspace.
int tile_nsplit(const pa_shape& sh, int sm_count);
// Rows of a last query tile of at most 8 rows that the tile schedule gives to
// the warp-level tensor cores of the last full pair's CTA (0: none).
int tile_remainder_rows(const pa_shape& sh);
size_t tile_partial_bytes(const pa_shape& sh, int sm_count);
size_t tile_partials_offset(const pa_shape& sh, int sm_count);
// 2-D TMA map over a bf16 row-major [rows, 128] matrix (the K or V pool seen
// as rows (page * H_kv + kv_head) * page_size + slot), boxes of 64 dims x
// box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, long long rows, int box_rows);
pa_status prefill_launch(const Call& c);

// ---- K/V append -----------------------------------------------------------
pa_status append_launch(const pa_shape& sh, const void* k_new, const void* v_new, void* kp,
                        void* vp, const int32_t* bt, const int32_t* ctx, uint32_t* flag,
                        int sm_count, cudaStream_t stream);

// ---- self-test of the bounded waits ---------------------------------------
pa_status wait_timeout_launch(uint32_t* flag, unsigned long long limit_ns, cudaStream_t stream);

// ---- debug gather ---------------------------------------------------------
pa_status gather_launch(const pa_shape& sh, const void* kp, const void* vp, const int32_t* bt,
                        const int32_t* ctx, int max_S, void* kd, void* vd, uint32_t* flag,
                        cudaStream_t stream);

}  // namespace pa
