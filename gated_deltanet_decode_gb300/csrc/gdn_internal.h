// Host-side interface between the C ABI (gdn_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_decode.h"

struct gdn_pool {
    float *data;
    int num_slots;
    gdn_dims dims;
    bool owned;
    int work_index; // this pool's pair of work counters in the library's table
    unsigned int *qk_count; // in-place counters [num_slots][qk_stride], or NULL
    int qk_stride;          // counters a slot: hk rounded up to a multiple of 4
    bool owns_qk_count;     // allocated with the pool (create), else caller memory
};

struct conv_pool {
    void *data;
    int num_slots;
    int channels;
    int width;
    int dtype;
    bool owned;
};

namespace gdn {

// Everything one launch of the state kernels needs.  Pointers are device
// pointers; layouts as in gdn_decode.h.
struct StepArgs {
    // gdn_decode_step inputs (unused by the fused layer)
    const void *q, *k, *v;
    // shared
    const void *a, *b;
    const float *A_log, *dt_bias;
    float *pool;
    int num_slots;
    const int32_t *read_slot, *write_slot;
    int in_place;
    void *out;
    int rows, hk, hv, dk, dv;
    int *err;
    unsigned int *work; // the pool's two work counters (claim, producers done), zero between launches
    int commit;         // twin only: swap read_slot and write_slot once every producer has read them
    const int32_t *n_live; // device count or NULL: rows at or past *n_live are left alone (outputs zero)
    unsigned int *qk_count; // fused layer, in place: the pool's counters [slot][qk_stride], or NULL
    int qk_stride;
    // fused layer only
    const void *x;
    void *conv;        // conv pool data
    const void *w;     // [C][W]
    const void *bias;  // [C] or null
    int silu;
    int width;
    int channels;
};

struct ConvArgs {
    const void *x;
    int x_stride;
    void *conv;
    int num_slots;
    const int32_t *read_slot, *write_slot;
    const void *w, *bias;
    int silu;
    void *out;
    int rows, channels, width;
    int *err;
};

// Many tokens a sequence (prefill, verification).  Sequence r holds tokens
// [cu_seqlens[r], cu_seqlens[r+1]) of the packed token-major inputs.
struct PrefillArgs {
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    float *pool;
    int num_slots;
    const int32_t *cu_seqlens, *read_slot;
    const int32_t *write_slot; // NULL: in place
    const int32_t *token_slot; // non-NULL: the state after each token goes to token_slot[t]
    void *out;
    int nseq, total_tokens, hk, hv, dk, dv;
    int *err;
    void *work;                // gdn_prefill_chunked, bf16: the chunk prep workspace
};

struct ConvPrefillArgs {
    const void *x; // [T][C]
    void *conv;
    int num_slots;
    const int32_t *cu_seqlens, *read_slot, *write_slot, *token_slot;
    const void *w, *bias;
    int silu;
    void *out;
    int nseq, total_tokens, channels, width;
    int *err;
};

// Launchers return cudaSuccess or the launch error.  Shapes were validated by
// the caller.
cudaError_t launch_gdn_step(const StepArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_gdn_layer(const StepArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_conv(const ConvArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_gdn_prefill(const PrefillArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_conv_prefill(const ConvPrefillArgs &a, int dtype, cudaStream_t s);
// The chunked (tensor-core) form of launch_gdn_prefill: in place or twin, no token slots.
// bf16 activations run the tcgen05 kernel (gdn_chunked_tc.cu), fp32 the mma.sync one.
cudaError_t launch_gdn_prefill_chunked(const PrefillArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_gdn_prefill_chunked_tc(const PrefillArgs &a, cudaStream_t s);
// Bytes of the workspace the bf16 chunked prefill needs (0 for no sequence).
size_t prefill_chunked_workspace_bytes(int nseq, int total_tokens, int hv);

// True when the state kernels are built for (dk, dv).
bool step_shape_supported(int dk, int dv);
// True when the chunked prefill is built for (dk, dv).
bool chunked_shape_supported(int dk, int dv);
// True when the fused layer can run this shape.
bool layer_shape_supported(int dk, int dv, int group, bool in_place);

} // namespace gdn
